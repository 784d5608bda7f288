"""The C-ABI library: it builds, loads without a GPU, exports every symbol
include/spec_verify.h declares, and rejects bad host arguments before any
CUDA call (CPU only: nothing here launches a kernel)."""
import ctypes
import re
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADERS = sorted((ROOT / "include").glob("*.h"))

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None
                                and not Path("/usr/local/cuda/bin/nvcc").exists(),
                                reason="needs nvcc to build the library")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_75_gb300 import api, build
    build.build()
    return api.load_library()


def declared_symbols():
    names = set()
    for h in HEADERS:
        text = h.read_text()
        names |= set(re.findall(r"^SV_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M))
    return names


def test_header_declares_the_boundary():
    names = declared_symbols()
    assert {"spec_verify", "spec_verify_diag", "sv_workspace_bytes",
            "sv_last_error", "sv_status_string"} <= names


def test_every_declared_symbol_is_exported(lib):
    from speculative_decoding_verification_75_gb300 import api
    names = declared_symbols()
    assert names == set(api.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", str(api.library_path())],
                         capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in names:
        assert n in exported, n
        assert getattr(lib, n) is not None


def test_status_strings(lib):
    for code in range(7):
        s = lib.sv_status_string(code).decode()
        assert s.startswith("SV_")
    assert lib.sv_status_string(99).decode() == "unknown sv_status"


def test_workspace_bytes(lib):
    a = lib.sv_workspace_bytes(128, 5, 151936)
    assert a > 0 and a % 256 == 0
    assert lib.sv_workspace_bytes(256, 5, 151936) > a
    assert lib.sv_workspace_bytes(128, 7, 151936) > a
    assert lib.sv_workspace_bytes(-1, 5, 10) == 0
    assert lib.sv_workspace_bytes(1, -1, 10) == 0
    assert lib.sv_workspace_bytes(1, 5, 0) == 0
    assert lib.sv_workspace_bytes(0, 0, 1) > 0


def _call(lib, **over):
    fake = ctypes.c_void_p(0x10000)        # never dereferenced: checks fail first
    args = dict(logits=fake, dtype=1, ids=fake, q=None, ua=fake, us=fake, t=fake,
                lens=None, B=4, g=3, V=100, tok=fake, nacc=fake, ws=fake,
                wsb=1 << 30, stream=None)
    args.update(over)
    return lib.spec_verify(*args.values())


def test_host_argument_errors_need_no_gpu(lib):
    from speculative_decoding_verification_75_gb300 import api
    assert _call(lib, dtype=7) == api.SV_ERR_UNSUPPORTED_DTYPE
    assert _call(lib, B=-1) == api.SV_ERR_INVALID_ARG
    assert _call(lib, g=-1) == api.SV_ERR_INVALID_ARG
    assert _call(lib, V=0) == api.SV_ERR_INVALID_ARG
    assert _call(lib, logits=None) == api.SV_ERR_INVALID_ARG
    assert _call(lib, ids=None) == api.SV_ERR_INVALID_ARG
    assert _call(lib, us=None) == api.SV_ERR_INVALID_ARG
    assert _call(lib, tok=None) == api.SV_ERR_INVALID_ARG
    assert _call(lib, ws=ctypes.c_void_p(0x10010)) == api.SV_ERR_INVALID_ARG
    assert _call(lib, logits=ctypes.c_void_p(0x10001)) == api.SV_ERR_INVALID_ARG
    assert _call(lib, wsb=16) == api.SV_ERR_WORKSPACE_TOO_SMALL
    assert _call(lib, B=0) == api.SV_OK            # empty batch: nothing to do
    assert _call(lib, g=0, ids=None, ua=None, B=0) == api.SV_OK
    assert lib.sv_last_error(None, None, None) == api.SV_ERR_INVALID_ARG


def test_selftest_argument_errors_need_no_gpu(lib):
    from speculative_decoding_verification_75_gb300 import api
    p = ctypes.c_void_p(0x10000)  # never dereferenced: the call returns before any launch
    assert lib.sv_selftest_wait_timeout(None, p, 1000, None) == api.SV_ERR_INVALID_ARG
    assert lib.sv_selftest_wait_timeout(p, None, 1000, None) == api.SV_ERR_INVALID_ARG
    assert lib.sv_selftest_wait_timeout(p, p, 0, None) == api.SV_ERR_INVALID_ARG
    assert lib.sv_selftest_wait_timeout(p, p, 2_000_000, None) == api.SV_ERR_INVALID_ARG
