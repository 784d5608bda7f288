"""Python binding of libspecverify.so (argument marshalling only).

Every step of the verification runs in the library's CUDA kernels; this
module checks tensor shapes and dtypes, allocates outputs and a workspace
with PyTorch, and passes raw device pointers plus the current CUDA stream to
the C ABI declared in ``include/spec_verify.h``.  There is no fallback: if
the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
from pathlib import Path
from typing import Optional

import torch

from . import build as _build

SV_OK = 0
SV_ERR_INVALID_ARG = 1
SV_ERR_UNSUPPORTED_DTYPE = 2
SV_ERR_WORKSPACE_TOO_SMALL = 3
SV_ERR_CUDA = 4
SV_ERR_TIMEOUT = 5
SV_ERR_BAD_INPUT_DATA = 6

SV_F32 = 0
SV_BF16 = 1

SV_BAD_DRAFT_LEN = 0x1
SV_BAD_TEMPERATURE = 0x2
SV_BAD_TOKEN = 0x4
SV_BAD_U_ACCEPT = 0x8
SV_BAD_U_SAMPLE = 0x10
SV_BAD_NORMALISER = 0x20
SV_FAULT_TIMEOUT = 0x10000

# Every symbol include/spec_verify.h declares.
EXPORTS = ("sv_workspace_bytes", "spec_verify", "spec_verify_diag",
           "sv_last_error", "sv_status_string", "spec_verify_noalloc", "sv_kv_rollback",
           "sv_selftest_wait_timeout", "sv_set_small_batch_path")

# Bits of the status word of sv_kv_rollback (include/spec_verify.h).
SV_KV_FREE_LIST_FULL = 0x1
SV_KV_MISSING_BLOCK = 0x2
SV_KV_BAD_LENGTH = 0x4
SV_KV_TABLE_SHORT = 0x8

_P = ctypes.c_void_p
_I = ctypes.c_int


class SvDiag(ctypes.Structure):
    """Mirror of ``sv_diag``: device pointers, any may be NULL."""
    _fields_ = [("p_tok", _P), ("q_tok", _P), ("accept_prob", _P),
                ("flags", _P), ("row_max", _P), ("row_sum", _P),
                ("row_argmax", _P), ("resid_mass", _P), ("accept_hist", _P)]


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, lib):
        self.status = status
        super().__init__(lib.sv_status_string(status).decode())


_lib = None


def library_path() -> Path:
    return _build.LIB


def load_library():
    """Load libspecverify.so (it must have been built); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not path.exists():
        raise RuntimeError(
            f"{path} is not built: run `python -m "
            "speculative_decoding_verification_75_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(str(path))
    lib.sv_workspace_bytes.restype = ctypes.c_size_t
    lib.sv_workspace_bytes.argtypes = [_I, _I, _I]
    common = [_P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P,
              ctypes.c_size_t, _P]
    lib.spec_verify.restype = _I
    lib.spec_verify.argtypes = common
    lib.spec_verify_diag.restype = _I
    lib.spec_verify_diag.argtypes = common + [ctypes.POINTER(SvDiag)]
    lib.sv_last_error.restype = _I
    lib.sv_last_error.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_uint32)]
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.sv_status_string.argtypes = [_I]
    lib.sv_set_small_batch_path.restype = _I
    lib.sv_set_small_batch_path.argtypes = [_I]
    lib.sv_selftest_wait_timeout.restype = _I
    lib.sv_selftest_wait_timeout.argtypes = [_P, _P, ctypes.c_uint, _P]
    lib.sv_kv_rollback.restype = _I
    lib.sv_kv_rollback.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _P]
    _lib = lib
    return lib


def workspace_bytes(B: int, gamma_max: int, V: int) -> int:
    return int(load_library().sv_workspace_bytes(B, gamma_max, V))


def set_small_batch_path(enabled: bool) -> bool:
    """Route small batches to the cluster kernel (True, the default) or send
    every batch to the persistent kernel (False), process-wide.  Returns the
    previous setting."""
    return bool(load_library().sv_set_small_batch_path(1 if enabled else 0))


def status_string(status: int) -> str:
    return load_library().sv_status_string(status).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream: Optional[torch.cuda.Stream], device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


_ws_cache: dict = {}


def get_workspace(B: int, gamma_max: int, V: int, device,
                  stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """A cached uint8 device buffer of at least sv_workspace_bytes() bytes,
    one per (device, stream): calls that share a workspace must be ordered on
    one stream, so calls on different streams get different workspaces and
    may run concurrently.  ``stream`` defaults to the device's current
    stream."""
    need = workspace_bytes(B, gamma_max, V)
    dev = torch.device(device)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    key = (dev, s.cuda_stream)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        _ws_cache[key] = ws
    return ws


def _check(t: Optional[torch.Tensor], name, dtype, shape, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def verify(target_logits: torch.Tensor, draft_token_ids: torch.Tensor,
           draft_probs: Optional[torch.Tensor], uniforms_accept: torch.Tensor,
           uniforms_sample: torch.Tensor, temperature: torch.Tensor,
           draft_lens: Optional[torch.Tensor] = None, *,
           out_tokens: Optional[torch.Tensor] = None,
           out_num_accepted: Optional[torch.Tensor] = None,
           workspace: Optional[torch.Tensor] = None, diag: bool = False,
           stream: Optional[torch.cuda.Stream] = None):
    """One speculative-decoding verification step on CUDA tensors.

    target_logits [B, g+1, V] bf16/fp32, draft_token_ids [B, g] int32,
    draft_probs [B, g, V] fp32 or None (deterministic drafts),
    uniforms_accept [B, g] fp32, uniforms_sample [B] fp32,
    temperature [B] fp32, draft_lens [B] int32 or None.

    Returns (out_tokens [B, g+1] int32, out_num_accepted [B] int32), plus a
    dict of diagnostic tensors when ``diag`` is true.  Asynchronous on the
    current (or given) stream.
    """
    lib = load_library()
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, gamma_max+1, V]")
    B, R, V = target_logits.shape
    g = R - 1
    dev = target_logits.device
    if dev.type != "cuda":
        raise ValueError("verify() takes CUDA tensors; see verify_host()")
    if target_logits.dtype == torch.bfloat16:
        dt = SV_BF16
    elif target_logits.dtype == torch.float32:
        dt = SV_F32
    else:
        raise TypeError(f"unsupported logits dtype {target_logits.dtype}")
    _check(target_logits, "target_logits", target_logits.dtype, (B, R, V), dev)
    _check(draft_token_ids, "draft_token_ids", torch.int32, (B, g), dev)
    _check(draft_probs, "draft_probs", torch.float32, (B, g, V), dev)
    _check(uniforms_accept, "uniforms_accept", torch.float32, (B, g), dev)
    _check(uniforms_sample, "uniforms_sample", torch.float32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    _check(draft_lens, "draft_lens", torch.int32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty(B, R, dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    _check(out_tokens, "out_tokens", torch.int32, (B, R), dev)
    _check(out_num_accepted, "out_num_accepted", torch.int32, (B,), dev)
    if workspace is None:
        workspace = get_workspace(B, g, V, dev, stream)
    args = [_ptr(target_logits), dt, _ptr(draft_token_ids), _ptr(draft_probs),
            _ptr(uniforms_accept), _ptr(uniforms_sample), _ptr(temperature),
            _ptr(draft_lens), B, g, V, _ptr(out_tokens), _ptr(out_num_accepted),
            _ptr(workspace), workspace.numel(), _stream_handle(stream, dev)]
    d = None
    if diag:
        f32 = dict(dtype=torch.float32, device=dev)
        d = {"p_tok": torch.empty(B, g, **f32), "q_tok": torch.empty(B, g, **f32),
             "accept_prob": torch.empty(B, g, **f32),
             "flags": torch.empty(B, g, dtype=torch.uint8, device=dev),
             "row_max": torch.empty(B, R, **f32), "row_sum": torch.empty(B, R, **f32),
             "row_argmax": torch.empty(B, R, dtype=torch.int32, device=dev),
             "resid_mass": torch.empty(B, **f32),
             "accept_hist": torch.empty(g + 2, dtype=torch.int32, device=dev)}
        sd = SvDiag(**{k: v.data_ptr() for k, v in d.items()})
        rc = lib.spec_verify_diag(*args, ctypes.byref(sd))
    else:
        rc = lib.spec_verify(*args)
    if rc != SV_OK:
        raise SpecVerifyError(rc, lib)
    if diag:
        return out_tokens, out_num_accepted, d
    return out_tokens, out_num_accepted


class BoundVerify:
    """``spec_verify`` bound to fixed tensors: every call re-runs the step on
    the tensors' current contents with the arguments marshalled once (about
    5 us of host time per call instead of ~19 us for ``verify``), for loops
    that reuse their buffers (a serving loop, a benchmark).  The tensors must
    stay alive and keep their storage while the object is used; calls are
    asynchronous on the bound stream."""

    def __init__(self, target_logits, draft_token_ids, draft_probs, uniforms_accept,
                 uniforms_sample, temperature, draft_lens=None, *, out_tokens=None,
                 out_num_accepted=None, workspace=None, stream=None):
        lib = load_library()
        B, R, V = target_logits.shape
        dev = target_logits.device
        # verify() checks every shape and dtype once; its outputs and
        # workspace are then reused by every call.
        self.out_tokens, self.out_num_accepted = verify(
            target_logits, draft_token_ids, draft_probs, uniforms_accept, uniforms_sample,
            temperature, draft_lens, out_tokens=out_tokens, out_num_accepted=out_num_accepted,
            workspace=workspace, stream=stream)
        if workspace is None:
            workspace = get_workspace(B, R - 1, V, dev, stream)
        self._keep = (target_logits, draft_token_ids, draft_probs, uniforms_accept,
                      uniforms_sample, temperature, draft_lens, workspace)
        dt = SV_BF16 if target_logits.dtype == torch.bfloat16 else SV_F32
        self._fn = lib.spec_verify
        self._lib = lib
        self._args = [_ptr(target_logits), dt, _ptr(draft_token_ids), _ptr(draft_probs),
                      _ptr(uniforms_accept), _ptr(uniforms_sample), _ptr(temperature),
                      _ptr(draft_lens), B, R - 1, V, _ptr(self.out_tokens),
                      _ptr(self.out_num_accepted), _ptr(workspace), workspace.numel(),
                      _stream_handle(stream, dev)]

    def __call__(self):
        rc = self._fn(*self._args)
        if rc != SV_OK:
            raise SpecVerifyError(rc, self._lib)
        return self.out_tokens, self.out_num_accepted


def bind(*args, **kwargs) -> BoundVerify:
    """``BoundVerify`` for the given tensors (same arguments as ``verify``)."""
    return BoundVerify(*args, **kwargs)


def kv_rollback(num_accepted: torch.Tensor, seq_lens: torch.Tensor,
                block_tables: torch.Tensor, block_size: int, free_list: torch.Tensor,
                free_count: torch.Tensor, draft_lens: Optional[torch.Tensor] = None, *,
                gamma_max: Optional[int] = None, status: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """KV rollback after verification, in place, through ``sv_kv_rollback``.

    num_accepted [B] int32 (from ``verify``), seq_lens [B] int32 (committed
    tokens before the drafts; updated to L + k), block_tables [B, max_blocks]
    int32 (-1 = no block; freed entries become -1), free_list [capacity]
    int32 and free_count [1] int32 (freed block ids are appended), draft_lens
    [B] int32 or None (then gamma_max drafts each), status [1] int32/uint32
    or None (receives SV_KV_* bits; the caller zeroes it).  All CUDA tensors
    on one device; asynchronous on the current (or given) stream."""
    lib = load_library()
    B = seq_lens.shape[0] if seq_lens.dim() == 1 else -1
    if B < 0 or block_tables.dim() != 2 or block_tables.shape[0] != B:
        raise ValueError("seq_lens must be [B] and block_tables [B, max_blocks]")
    dev = seq_lens.device
    if gamma_max is None:
        if draft_lens is None:
            raise ValueError("gamma_max is needed when draft_lens is None")
        gamma_max = int(draft_lens.max().item()) if B else 0
    _check(num_accepted, "num_accepted", torch.int32, (B,), dev)
    _check(seq_lens, "seq_lens", torch.int32, (B,), dev)
    _check(block_tables, "block_tables", torch.int32, tuple(block_tables.shape), dev)
    _check(draft_lens, "draft_lens", torch.int32, (B,), dev)
    _check(free_list, "free_list", torch.int32, (free_list.numel(),), dev)
    _check(free_count, "free_count", torch.int32, (1,), dev)
    if status is not None and (status.device != dev or status.numel() != 1
                               or status.dtype not in (torch.int32, torch.uint32)):
        raise ValueError("status must be a 1-element int32/uint32 tensor on the same device")
    rc = lib.sv_kv_rollback(_ptr(num_accepted), _ptr(draft_lens), _ptr(seq_lens),
                            _ptr(block_tables), B, int(gamma_max), block_tables.shape[1],
                            int(block_size), _ptr(free_list), _ptr(free_count),
                            free_list.numel(), _ptr(status), _stream_handle(stream, dev))
    if rc != SV_OK:
        raise SpecVerifyError(rc, lib)


def selftest_wait_timeout(limit_us: int = 1000, device="cuda") -> int:
    """Run the bounded-wait self-test (``sv_selftest_wait_timeout``) and
    return the status word it sets (synchronises)."""
    lib = load_library()
    dev = torch.device(device)
    word = torch.zeros(1, dtype=torch.int32, device=dev)
    never = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = lib.sv_selftest_wait_timeout(_ptr(word), _ptr(never), int(limit_us),
                                      _stream_handle(None, dev))
    if rc != SV_OK:
        raise SpecVerifyError(rc, lib)
    torch.cuda.synchronize(dev)
    return int(word.item()) & 0xFFFFFFFF


def acceptance_stats(accept_hist) -> dict:
    """Acceptance statistics of one batch from ``accept_hist`` (the
    ``sv_diag`` histogram, [gamma_max + 2]: requests per number of accepted
    drafts, then requests with invalid data).  Host arithmetic only.

    Returns n_valid, n_bad, accepted_at[i] (requests whose draft i was
    accepted), reached[i] (requests that tested draft i and every earlier one
    was accepted -- with uniform draft lengths, the requests whose draft i
    was tested), the conditional acceptance rate accepted_at / reached per
    position, and the mean number of emitted tokens (num_accepted + 1,
    P3 §3.3)."""
    h = [int(v) for v in (accept_hist.tolist() if hasattr(accept_hist, "tolist") else accept_hist)]
    g = len(h) - 2
    if g < 0:
        raise ValueError("accept_hist must have gamma_max + 2 entries")
    counts, n_bad = h[:g + 1], h[g + 1]
    n_valid = sum(counts)
    accepted_at = [sum(counts[j] for j in range(i + 1, g + 1)) for i in range(g)]
    reached = [sum(counts[j] for j in range(i, g + 1)) for i in range(g)]
    rate = [a / r if r else float("nan") for a, r in zip(accepted_at, reached)]
    mean_emitted = (sum((j + 1) * c for j, c in enumerate(counts)) / n_valid
                    if n_valid else float("nan"))
    return {"n_valid": n_valid, "n_bad": n_bad, "accepted_at": accepted_at,
            "reached": reached, "rate": rate, "mean_emitted": mean_emitted}


def verify_host(target_logits: torch.Tensor, draft_token_ids: torch.Tensor,
                draft_probs: Optional[torch.Tensor], uniforms_accept: torch.Tensor,
                uniforms_sample: torch.Tensor, temperature: torch.Tensor,
                draft_lens: Optional[torch.Tensor] = None, *, device="cuda",
                stream: Optional[torch.cuda.Stream] = None):
    """``verify`` for host tensors (pinned for asynchronous copies): copies
    the inputs to ``device``, runs the step there and copies the two outputs
    back.  Returns host (out_tokens, out_num_accepted) once they are ready."""
    dev = torch.device(device)

    def up(t):
        return None if t is None else t.to(dev, non_blocking=True)

    with torch.cuda.stream(stream) if stream is not None else _nullctx():
        tok, nacc = verify(up(target_logits), up(draft_token_ids), up(draft_probs),
                           up(uniforms_accept), up(uniforms_sample), up(temperature),
                           up(draft_lens), stream=stream)
        tok_h = torch.empty(tok.shape, dtype=tok.dtype, pin_memory=True)
        nacc_h = torch.empty(nacc.shape, dtype=nacc.dtype, pin_memory=True)
        tok_h.copy_(tok, non_blocking=True)
        nacc_h.copy_(nacc, non_blocking=True)
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        s.synchronize()
    return tok_h, nacc_h


class _nullctx:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def last_error(workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None):
    """(status, error word) of the last call that used ``workspace``."""
    lib = load_library()
    word = ctypes.c_uint32(0)
    rc = lib.sv_last_error(_ptr(workspace), _stream_handle(stream, workspace.device),
                           ctypes.byref(word))
    return rc, word.value
