"""fp64 CPU oracle of the speculative-decoding verification step.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain definition of what the
verification step computes, written from the speculative-decoding tutorial
page at dpshk.com/news/5598276 ("P3"; §3.1-§3.2, §4, §5.2-§5.3).  It shares no
code with the CUDA path; only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it.

``verify`` takes host numpy arrays with the same layout as the CUDA library's
``spec_verify`` and returns every intermediate the parity tests compare,
including the decision margins that mark borderline cases.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from .build import build_oracle

# Bits of the per-request bad-input word (the oracle's own definitions).
BAD_DRAFT_LEN = 1
BAD_TEMP = 2
BAD_TOKEN = 4
BAD_U_ACCEPT = 8
BAD_U_SAMPLE = 16
BAD_NORMALISER = 32

_P = ctypes.c_void_p


class _Outputs(ctypes.Structure):
    _fields_ = [(name, _P) for name in (
        "tokens", "num_accepted", "bad", "resid_mass", "sample_margin",
        "sample_fallback", "p_tok", "q_tok", "accept_prob", "flags",
        "accept_margin", "row_max", "row_sum", "row_argmax")]


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_P)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def logits_to_numpy(logits):
    """Return (array, is_bf16) for a torch tensor or numpy array of logits.

    bf16 tensors become their uint16 bit patterns, fp32 stays fp32."""
    try:
        import torch
        if isinstance(logits, torch.Tensor):
            t = logits.detach().to("cpu").contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16), True
            return t.to(torch.float32).numpy(), False
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(logits)
    if a.dtype == np.uint16:
        return a, True
    return a.astype(np.float32, copy=False), False


class Oracle:
    """ctypes handle on one build of the oracle library.

    The default instance wraps ``liboracle.so``; the mutation tests build
    altered copies of ``oracle.c`` and wrap them the same way."""

    def __init__(self, lib_path=None):
        lib = ctypes.CDLL(str(lib_path or build_oracle()))
        lib.orc_verify.restype = ctypes.c_int
        lib.orc_verify.argtypes = [_P, ctypes.c_int, _P, _P, _P, _P, _P, _P,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(_Outputs)]
        self.has_mt = hasattr(lib, "orc_verify_mt")
        if self.has_mt:
            lib.orc_verify_mt.restype = ctypes.c_int
            lib.orc_verify_mt.argtypes = lib.orc_verify.argtypes + [ctypes.c_int]
        lib.orc_row_stats.restype = None
        lib.orc_row_stats.argtypes = [_P, ctypes.c_int, ctypes.c_size_t,
                                      ctypes.c_int, ctypes.c_double, _P, _P, _P]
        lib.orc_draw_cdf.restype = ctypes.c_int
        lib.orc_draw_cdf.argtypes = [_P, ctypes.c_int, _P, _P, _P, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, _P]
        lib.orc_draw_weights.restype = ctypes.c_int
        lib.orc_draw_weights.argtypes = lib.orc_draw_cdf.argtypes
        lib.orc_inverse_cdf.restype = ctypes.c_int
        lib.orc_inverse_cdf.argtypes = [_P, ctypes.c_int, ctypes.c_double, _P]
        self.lib = lib

    def verify(self, logits, draft_ids, draft_probs, u_acc, u_samp,
               temperature, draft_lens=None, *, is_bf16: Optional[bool] = None,
               nthreads: int = 1):
        """Run the oracle.  Shapes: logits [B, g+1, V] (uint16 bf16 bits or
        fp32), draft_ids [B, g], draft_probs [B, g, V] or None, u_acc [B, g],
        u_samp [B], temperature [B], draft_lens [B] or None.  nthreads > 1
        splits the requests over that many host threads (same arithmetic,
        same results)."""
        if is_bf16 is None:
            logits, is_bf16 = logits_to_numpy(logits)
        else:
            logits = np.ascontiguousarray(logits)
        B, rows, V = logits.shape
        g = rows - 1
        draft_ids = _c(_np(draft_ids).reshape(B, g), np.int32)
        draft_probs = (None if draft_probs is None
                       else _c(_np(draft_probs).reshape(B, g, V), np.float32))
        u_acc = _c(_np(u_acc).reshape(B, g), np.float32)
        u_samp = _c(_np(u_samp).reshape(B), np.float32)
        temperature = _c(_np(temperature).reshape(B), np.float32)
        draft_lens = (None if draft_lens is None
                      else _c(_np(draft_lens).reshape(B), np.int32))

        res = {
            "tokens": np.empty((B, g + 1), np.int32),
            "num_accepted": np.empty(B, np.int32),
            "bad": np.empty(B, np.int32),
            "resid_mass": np.empty(B, np.float64),
            "sample_margin": np.empty(B, np.float64),
            "sample_fallback": np.empty(B, np.int32),
            "p_tok": np.empty((B, g), np.float64),
            "q_tok": np.empty((B, g), np.float64),
            "accept_prob": np.empty((B, g), np.float64),
            "flags": np.empty((B, g), np.uint8),
            "accept_margin": np.empty((B, g), np.float64),
            "row_max": np.empty((B, g + 1), np.float64),
            "row_sum": np.empty((B, g + 1), np.float64),
            "row_argmax": np.empty((B, g + 1), np.int32),
        }
        outs = _Outputs(**{k: _ptr(v) for k, v in res.items()})
        args = [_ptr(logits), int(bool(is_bf16)), _ptr(draft_ids), _ptr(draft_probs),
                _ptr(u_acc), _ptr(u_samp), _ptr(temperature), _ptr(draft_lens), B, g, V,
                ctypes.byref(outs)]
        if nthreads > 1 and self.has_mt:
            rc = self.lib.orc_verify_mt(*args, int(nthreads))
        else:
            rc = self.lib.orc_verify(*args)
        if rc != 0:
            raise MemoryError("oracle scratch allocation failed")
        return res

    def draw_cdf(self, logits, draft_ids, draft_probs, temperature, b: int, k: int, g: int):
        """Inclusive prefix sums (fp64, [V]) of the weights of the draw at
        position k of request b (g its draft length), as the oracle walks
        them; None for a greedy request."""
        return self._draw(self.lib.orc_draw_cdf, logits, draft_ids, draft_probs, temperature,
                          b, k, g)

    def draw_weights(self, logits, draft_ids, draft_probs, temperature, b: int, k: int,
                     g: int):
        """The weights themselves (fp64, [V]) of that draw; None for a greedy
        request."""
        return self._draw(self.lib.orc_draw_weights, logits, draft_ids, draft_probs,
                          temperature, b, k, g)

    def _draw(self, fn, logits, draft_ids, draft_probs, temperature, b, k, g):
        arr, is_bf16 = logits_to_numpy(logits)
        arr = np.ascontiguousarray(arr)
        B, rows, V = arr.shape
        gmax = rows - 1
        ids = _c(_np(draft_ids).reshape(B, gmax), np.int32)
        q = None if draft_probs is None else _c(_np(draft_probs).reshape(B, gmax, V), np.float32)
        T = _c(_np(temperature).reshape(B), np.float32)
        out = np.empty(V, np.float64)
        rc = fn(_ptr(arr), int(bool(is_bf16)), _ptr(ids), _ptr(q), _ptr(T),
                int(b), int(k), int(g), gmax, V, _ptr(out))
        return None if rc != 0 else out

    def row_stats(self, row, temperature: float):
        """(max, normaliser, argmax) of the softmax of row / T for one row."""
        arr, is_bf16 = logits_to_numpy(row)
        arr = np.ascontiguousarray(arr.reshape(-1))
        m = ctypes.c_double()
        s = ctypes.c_double()
        a = ctypes.c_int()
        self.lib.orc_row_stats(_ptr(arr), int(is_bf16), 0, arr.size,
                               float(temperature), ctypes.byref(m),
                               ctypes.byref(s), ctypes.byref(a))
        return m.value, s.value, a.value

    def inverse_cdf(self, weights, u: float):
        """(token, margin) of the oracle's inverse-CDF draw on raw weights."""
        w = np.ascontiguousarray(weights, dtype=np.float64)
        margin = ctypes.c_double()
        tok = self.lib.orc_inverse_cdf(_ptr(w), w.size, float(u),
                                       ctypes.byref(margin))
        return tok, margin.value


def _np(a):
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return a.detach().to("cpu").numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(a)


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def verify(*args, **kwargs):
    return default().verify(*args, **kwargs)


def row_stats(row, temperature: float):
    return default().row_stats(row, temperature)


def inverse_cdf(weights, u: float):
    return default().inverse_cdf(weights, u)
