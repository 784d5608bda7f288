"""GB300-native speculative-decoding verification (vectorised rejection sampler).

``verify`` runs one verification step of a batch on the GPU through the C ABI
of ``lib/libspecverify.so`` (declared in ``include/spec_verify.h``);
``bind`` fixes the tensors of a loop once and re-runs the step cheaply;
``verify_host`` does the same from host tensors, copies included.
"""
from .api import (BoundVerify, SpecVerifyError, bind, last_error,  # noqa: F401
                  load_library, verify, verify_host, workspace_bytes)
