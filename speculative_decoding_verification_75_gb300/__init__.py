"""GB300-native speculative-decoding verification (vectorised rejection sampler).

``verify`` runs one verification step of a batch on the GPU through the C ABI
of ``lib/libspecverify.so`` (declared in ``include/spec_verify.h``);
``verify_host`` does the same from host tensors, copies included.
"""
from .api import (SpecVerifyError, last_error, load_library, verify,  # noqa: F401
                  verify_host, workspace_bytes)
