"""fp64 CPU oracle for the batch-invariant forward kernels.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library never loads it and shares no code with it.

Each function evaluates the plain definition of one operation in double
precision (see ``bi_oracle.c`` for the formulas and the passages they follow)
and returns float64 numpy arrays; ``round_bf16`` turns them into the bf16 bit
patterns those values round to (nearest-even, one rounding from fp64).

Inputs are bf16 tensors given as uint16 bit patterns (numpy) or torch bf16 CPU
tensors; both are accepted.

Pins (checked by ``tests/test_oracle.py`` without reference to this code):
  round_bf16 .......... brute-force nearest search over all 65536 patterns,
                        agreement with IEEE float32->bf16 on float32 inputs
  rmsnorm ............. constant row, one-hot row, zero row, eps-dominated row
                        (closed forms), power-of-two scale invariance
  gemm ................ exact rational brute force (fractions.Fraction) on
                        4x8x8 and non-square shapes; identity weight
  decode_attention .... one key returns v0; equal keys return mean(V);
                        two keys give the closed-form sigmoid weights that fix
                        the 1/sqrt(D) scale; GQA head mapping; dense
                        scipy-softmax evaluation of gathered pages
  decode_attention_chunked ... equals the unchunked definition; chunk plan
                        1000 -> 256, 256, 256, 232 from the pages
  logprobs ............ uniform row (-log V), two-level row closed form,
                        scipy logsumexp, probabilities summing to 1
No function is left "parity unpinned".
"""
from __future__ import annotations

import ctypes
import math

import numpy as np

from .build import build_oracle

_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build_oracle())
    lib.oracle_round_bf16.argtypes = [_f64p, _u16p, ctypes.c_int64]
    lib.oracle_round_bf16.restype = None
    lib.oracle_bf16_to_double.argtypes = [_u16p, _f64p, ctypes.c_int64]
    lib.oracle_bf16_to_double.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_rmsnorm.argtypes = [_u16p, _u16p, ctypes.c_int64, ctypes.c_int32,
                                   ctypes.c_double, _f64p]
    lib.oracle_rmsnorm.restype = ctypes.c_int
    lib.oracle_gemm.argtypes = [_u16p, _u16p, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int32, _f64p]
    lib.oracle_gemm.restype = ctypes.c_int
    lib.oracle_gemm_entries.argtypes = [_u16p, _u16p, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, _i32p, _i32p, ctypes.c_int64,
                                        _f64p]
    lib.oracle_gemm_entries.restype = ctypes.c_int
    attn_common = [_u16p, _u16p, _u16p, _i32p, ctypes.c_int32, _i32p,
                   ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                   ctypes.c_int32, ctypes.c_double]
    lib.oracle_decode_attention.argtypes = attn_common + [_f64p]
    lib.oracle_decode_attention.restype = ctypes.c_int
    lib.oracle_decode_attention_chunked.argtypes = attn_common + [
        ctypes.c_int32, ctypes.c_int32, _f64p, _f64p]
    lib.oracle_decode_attention_chunked.restype = ctypes.c_int
    lib.oracle_logprobs.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int32, _i32p, _f64p, _f64p]
    lib.oracle_logprobs.restype = ctypes.c_int
    _lib = lib
    return lib


def num_threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(_load().oracle_num_threads())


def _bits(a) -> np.ndarray:
    """bf16 input -> contiguous uint16 numpy array of its bit patterns."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        a = a.detach().to("cpu").contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns (uint16), got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    if hasattr(a, "numpy"):
        a = a.detach().to("cpu").numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def round_bf16(values) -> np.ndarray:
    """fp64 values -> uint16 bf16 bit patterns, round to nearest, ties to even."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_round_bf16(_p(v, _f64p), _p(out, _u16p), v.size)
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """uint16 bf16 bit patterns -> exact fp64 values."""
    b = _bits(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_bf16_to_double(_p(b, _u16p), _p(out, _f64p), b.size)
    return out


def rmsnorm(x, w, eps: float) -> np.ndarray:
    """y = x * w / sqrt(mean(x^2) + eps) per row, fp64.  x [rows, H], w [H]."""
    xb, wb = _bits(x), _bits(w)
    if xb.ndim != 2 or wb.ndim != 1 or xb.shape[1] != wb.shape[0]:
        raise ValueError("rmsnorm: x [rows, H] and w [H] expected")
    rows, H = xb.shape
    y = np.empty((rows, H), dtype=np.float64)
    rc = _load().oracle_rmsnorm(_p(xb, _u16p), _p(wb, _u16p), rows, H, float(eps),
                                _p(y, _f64p))
    if rc != 0:
        raise ValueError(f"oracle_rmsnorm failed ({rc})")
    return y


def gemm(x, W) -> np.ndarray:
    """y = x @ W^T in fp64.  x [M, K], W [N, K]."""
    xb, Wb = _bits(x), _bits(W)
    if xb.ndim != 2 or Wb.ndim != 2 or xb.shape[1] != Wb.shape[1]:
        raise ValueError("gemm: x [M, K] and W [N, K] expected")
    M, K = xb.shape
    N = Wb.shape[0]
    y = np.empty((M, N), dtype=np.float64)
    rc = _load().oracle_gemm(_p(xb, _u16p), _p(Wb, _u16p), M, N, K, _p(y, _f64p))
    if rc != 0:
        raise ValueError(f"oracle_gemm failed ({rc})")
    return y


def gemm_entries(x, W, ms, ns) -> np.ndarray:
    """y[i] = sum_k x[ms[i], k] * W[ns[i], k] in fp64, for sampled positions."""
    xb, Wb = _bits(x), _bits(W)
    M, K = xb.shape
    N = Wb.shape[0]
    ms, ns = _i32(ms).ravel(), _i32(ns).ravel()
    if ms.shape != ns.shape:
        raise ValueError("gemm_entries: ms and ns differ in length")
    y = np.empty(ms.shape, dtype=np.float64)
    _load().oracle_gemm_entries(_p(xb, _u16p), _p(Wb, _u16p), M, N, K,
                                _p(ms, _i32p), _p(ns, _i32p), ms.size, _p(y, _f64p))
    if np.isnan(y).any():
        raise ValueError("gemm_entries: position out of range")
    return y


def _attn_args(q, k_cache, v_cache, block_table, seq_lens):
    qb, kb, vb = _bits(q), _bits(k_cache), _bits(v_cache)
    bt, sl = _i32(block_table), _i32(seq_lens)
    if qb.ndim != 3 or kb.ndim != 4 or kb.shape != vb.shape or bt.ndim != 2:
        raise ValueError("decode_attention: q [B,Hq,D], caches [P,Hkv,page,D], "
                         "block_table [B,max_pages] expected")
    B, Hq, D = qb.shape
    _, Hkv, page, D2 = kb.shape
    if D2 != D or bt.shape[0] != B or sl.shape != (B,):
        raise ValueError("decode_attention: inconsistent shapes")
    return qb, kb, vb, bt, sl, B, Hq, Hkv, D, page


def decode_attention(q, k_cache, v_cache, block_table, seq_lens,
                     scale: float | None = None) -> np.ndarray:
    """Unchunked softmax(q k^T * scale) v over each sequence's cached tokens."""
    qb, kb, vb, bt, sl, B, Hq, Hkv, D, page = _attn_args(
        q, k_cache, v_cache, block_table, seq_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.empty((B, Hq, D), dtype=np.float64)
    rc = _load().oracle_decode_attention(
        _p(qb, _u16p), _p(kb, _u16p), _p(vb, _u16p), _p(bt, _i32p), bt.shape[1],
        _p(sl, _i32p), B, Hq, Hkv, D, page, float(scale), _p(out, _f64p))
    if rc != 0:
        raise ValueError(f"oracle_decode_attention failed ({rc})")
    return out


def decode_attention_chunked(q, k_cache, v_cache, block_table, seq_lens,
                             chunk: int = 256, scale: float | None = None,
                             max_chunks: int | None = None,
                             want_partials: bool = False):
    """Fixed split-size attention in fp64: chunks of `chunk` tokens, partials
    folded in ascending order by the log-sum-exp rule.  Returns out, or
    (out, partials[B, Hq, max_chunks, D + 2]) with (m, l, a[0..D-1])."""
    qb, kb, vb, bt, sl, B, Hq, Hkv, D, page = _attn_args(
        q, k_cache, v_cache, block_table, seq_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if max_chunks is None:
        max_chunks = int(max(1, -(-int(sl.max()) // chunk))) if B else 1
    out = np.empty((B, Hq, D), dtype=np.float64)
    part = (np.full((B, Hq, max_chunks, D + 2), np.nan, dtype=np.float64)
            if want_partials else None)
    rc = _load().oracle_decode_attention_chunked(
        _p(qb, _u16p), _p(kb, _u16p), _p(vb, _u16p), _p(bt, _i32p), bt.shape[1],
        _p(sl, _i32p), B, Hq, Hkv, D, page, float(scale), int(chunk),
        int(max_chunks), _p(out, _f64p),
        _p(part, _f64p) if part is not None else None)
    if rc != 0:
        raise ValueError(f"oracle_decode_attention_chunked failed ({rc})")
    return (out, part) if want_partials else out


def logprobs(logits, targets=None):
    """(logprob of targets [rows], lse [rows]) of bf16 logits [rows, vocab], fp64."""
    lb = _bits(logits)
    rows, vocab = lb.shape
    lse = np.empty(rows, dtype=np.float64)
    lp = np.empty(rows, dtype=np.float64)
    t = _i32(targets).ravel() if targets is not None else None
    rc = _load().oracle_logprobs(_p(lb, _u16p), rows, vocab,
                                 _p(t, _i32p) if t is not None else None,
                                 _p(lp, _f64p) if t is not None else None, _p(lse, _f64p))
    if rc != 0:
        raise ValueError(f"oracle_logprobs failed ({rc})")
    return (lp if t is not None else None), lse
