"""The allocation-free entry point (spec_verify_noalloc) against spec_verify.

spec_verify_noalloc is for callers that cannot allocate device memory (an
allocation-free serving loop, a plugin without an allocator): it runs the same
kernels on a scratch array the library keeps in device memory instead of a
caller-provided workspace.  Called through the C ABI, it must give exactly the
outputs of spec_verify with a workspace, on two calls in a row (the second
reuses the scratch array left behind by the first).

This file is collected last on purpose; it must pass alone in a fresh process
and after the other GPU tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verification_75_gb300 import api, verify, workloads

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
_P = ctypes.c_void_p
_I = ctypes.c_int


def _noalloc_fn():
    fn = api.load_library().spec_verify_noalloc
    fn.restype = _I
    fn.argtypes = [_P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P]
    return fn


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(fn, case):
    lg = case["logits"]
    B, R, V = lg.shape
    tok = torch.full((B, R), -7, dtype=torch.int32, device=DEV)
    nacc = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    dt = api.SV_BF16 if lg.dtype == torch.bfloat16 else api.SV_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    rc = fn(_ptr(lg), dt, _ptr(case["draft_ids"]), _ptr(case["draft_probs"]),
            _ptr(case["u_accept"]), _ptr(case["u_sample"]), _ptr(case["temperature"]),
            _ptr(case["draft_lens"]), B, R - 1, V, _ptr(tok), _ptr(nacc), stream)
    assert rc == api.SV_OK, api.status_string(rc)
    torch.cuda.synchronize(DEV)
    return tok.cpu().numpy(), nacc.cpu().numpy()


@pytest.mark.parametrize("key,B", [("c3", 64), ("c5", 64), ("c3", 128), ("c5", 256)])
def test_noalloc_matches_spec_verify_twice(key, B):
    """B = 256 with gamma_max = 7 and V = 151936 (workload c5 at full size) is
    the size the header quotes as fitting the scratch array."""
    fn = _noalloc_fn()
    w = workloads.workload(key, B=B)
    for seed in (101, 202):  # two calls in a row on the shared scratch array
        case = workloads.make_case(w, device=DEV, seed=seed)
        ref_tok, ref_nacc = verify(case["logits"], case["draft_ids"], case["draft_probs"],
                                   case["u_accept"], case["u_sample"], case["temperature"],
                                   case["draft_lens"])
        torch.cuda.synchronize(DEV)
        tok, nacc = _call_noalloc(fn, case)
        # Same kernels on the same inputs: integer outputs agree exactly.
        assert np.array_equal(nacc, ref_nacc.cpu().numpy())
        assert np.array_equal(tok, ref_tok.cpu().numpy())


def test_noalloc_rejects_sizes_beyond_the_scratch_array():
    fn = _noalloc_fn()
    lib = api.load_library()
    big_B, g, V = 4096, 7, 151936
    assert lib.sv_workspace_bytes(big_B, g, V) > (4 << 20)
    dummy = torch.empty(16, dtype=torch.int32, device=DEV)
    p = _ptr(dummy)
    rc = fn(p, api.SV_BF16, p, p, p, p, p, None, big_B, g, V, p, p, None)
    assert rc == api.SV_ERR_WORKSPACE_TOO_SMALL
