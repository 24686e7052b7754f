"""Batch-invariant forward kernels for LLM inference on GB300 (sm_103a).

Thin Python binding over libbi.so (C ABI: include/bi.h).  Each function only
checks and marshals its torch arguments (device pointers, sizes, leading
dimensions, the current CUDA stream) and calls the library; every step of the
computation runs in the library's CUDA kernels.  There is no CPU fallback:
tensors must live on a CUDA device, and a missing library raises.

    rmsnorm(x, w, eps)                    y = x * rsqrt(mean(x^2) + eps) * w, per row
    add_rmsnorm(x, residual, w, eps)      residual += x, then rmsnorm(residual)
    gemm(x, W)                            y = x @ W.T  (W in nn.Linear [N, K] layout)
    gemm_swiglu(x, interleave_gate_up(W)) silu(x @ W_gate.T) * (x @ W_up.T), fused
    decode_attention(q, k_cache, v_cache, block_table, seq_lens, max_seq_len)
                                          paged decode attention, 256-token splits
    prefill_attention(...)                causal attention for many rows per sequence,
                                          bit-identical per row to decode_attention
    qk_norm_rope_append(...), silu_mul(gate_up), logprobs(logits, targets)

Every output row's bits depend only on that row's own inputs (batch
invariance); see include/bi.h for the exact contract of each call.
"""
from __future__ import annotations

import math

import torch

from . import _lib
from ._lib import DECODE_CHUNK, DECODE_COUNTER_BYTES, PAGE_SIZE

__all__ = ["BiError", "rmsnorm", "gemm", "gemm_swiglu", "interleave_gate_up",
           "decode_attention", "decode_attention_fixed_splits",
           "prefill_attention", "prefill_attention_workspace_size", "add_rmsnorm",
           "qk_norm_rope_append", "silu_mul", "logprobs",
           "decode_attention_workspace_size", "selftest_wait_timeout",
           "decode_num_chunks", "decode_chunk_len", "get_device_error", "abi_version",
           "status_string", "PAGE_SIZE", "DECODE_CHUNK"]


class BiError(RuntimeError):
    """A libbi.so call returned a status other than BI_OK."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def status_string(status: int) -> str:
    return _lib.load().bi_status_string(int(status)).decode()


def abi_version() -> int:
    return int(_lib.load().bi_abi_version())


def _check(status: int, where: str) -> None:
    if status != _lib.BI_OK:
        raise BiError(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _cuda_bf16(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16, got {t.dtype}")


def _row_major_2d(t: torch.Tensor, name: str) -> int:
    """Leading dimension (elements) of a 2-D tensor with unit inner stride."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    return int(t.stride(0)) if t.shape[0] > 1 else int(t.shape[1])


def get_device_error(stream=None) -> None:
    """Synchronise `stream` and raise BiError if a kernel recorded a
    device-side problem (a barrier wait past its limit, or an out-of-range
    seq_lens / block_table entry).  Clears the record."""
    _check(_lib.load().bi_get_device_error(_stream(stream)), "bi_get_device_error")


# ------------------------------------------------------------- RMSNorm ------
def rmsnorm(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, out: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """Batch-invariant RMSNorm over the last dimension of x [rows, hidden]."""
    _cuda_bf16(x, "x")
    _cuda_bf16(w, "w")
    if x.dim() != 2 or w.dim() != 1 or w.shape[0] != x.shape[1] or not w.is_contiguous():
        raise ValueError("rmsnorm: x [rows, hidden] and contiguous w [hidden] expected")
    rows, hidden = x.shape
    if out is None:
        out = torch.empty((rows, hidden), dtype=torch.bfloat16, device=x.device)
    _cuda_bf16(out, "out")
    if tuple(out.shape) != (rows, hidden):
        raise ValueError("rmsnorm: out has the wrong shape")
    ld_x = _row_major_2d(x, "x")
    ld_y = _row_major_2d(out, "out")
    _check(_lib.load().bi_rmsnorm(x.data_ptr(), w.data_ptr(), out.data_ptr(), rows, hidden,
                                  ld_x, ld_y, float(eps), _stream(stream)), "bi_rmsnorm")
    return out


def add_rmsnorm(x: torch.Tensor, residual: torch.Tensor, w: torch.Tensor, eps: float = 1e-6,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """residual += x (bf16, in place), then RMSNorm(residual) * w -> out."""
    for t, n in ((x, "x"), (residual, "residual"), (w, "w")):
        _cuda_bf16(t, n)
    if x.shape != residual.shape or x.dim() != 2 or w.dim() != 1 or w.shape[0] != x.shape[1]:
        raise ValueError("add_rmsnorm: x, residual [rows, hidden] and w [hidden] expected")
    rows, hidden = x.shape
    if out is None:
        out = torch.empty((rows, hidden), dtype=torch.bfloat16, device=x.device)
    _cuda_bf16(out, "out")
    _check(_lib.load().bi_add_rmsnorm(x.data_ptr(), residual.data_ptr(), w.data_ptr(),
                                      out.data_ptr(), rows, hidden, _row_major_2d(x, "x"),
                                      _row_major_2d(residual, "residual"),
                                      _row_major_2d(out, "out"), float(eps), _stream(stream)),
           "bi_add_rmsnorm")
    return out


def qk_norm_rope_append(qkv: torch.Tensor, Hq: int, Hkv: int, positions: torch.Tensor,
                        slots: torch.Tensor, rope: torch.Tensor, q_norm_w, k_norm_w,
                        k_cache: torch.Tensor, v_cache: torch.Tensor, eps: float = 1e-6,
                        q_out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per-head q/k RMSNorm + RoPE; q -> q_out [T, Hq, 128]; k, v -> cache slots."""
    _cuda_bf16(qkv, "qkv")
    T = qkv.shape[0]
    D = 128
    if q_out is None:
        q_out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=qkv.device)
    for t, n in ((positions, "positions"), (slots, "slots")):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous() or t.shape[0] != T:
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor of length T")
    if not rope.is_cuda or rope.dtype != torch.float32 or not rope.is_contiguous():
        raise ValueError("rope must be a contiguous float32 CUDA tensor")
    num_pages, Hkv2, page, D2 = k_cache.shape
    if Hkv2 != Hkv or D2 != D:
        raise ValueError("qk_norm_rope_append: cache shape mismatch")
    _check(_lib.load().bi_qk_norm_rope_append(
        qkv.data_ptr(), _row_major_2d(qkv, "qkv"), T, Hq, Hkv, D, positions.data_ptr(),
        slots.data_ptr(), rope.data_ptr(), rope.shape[0],
        q_norm_w.data_ptr() if q_norm_w is not None else None,
        k_norm_w.data_ptr() if k_norm_w is not None else None, float(eps), q_out.data_ptr(),
        k_cache.data_ptr(), v_cache.data_ptr(), num_pages, page, _stream(stream)),
        "bi_qk_norm_rope_append")
    return q_out


def silu_mul(gate_up: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """SwiGLU: out = silu(gate_up[:, :F]) * gate_up[:, F:]."""
    _cuda_bf16(gate_up, "gate_up")
    T, F2 = gate_up.shape
    F = F2 // 2
    if out is None:
        out = torch.empty((T, F), dtype=torch.bfloat16, device=gate_up.device)
    _check(_lib.load().bi_silu_mul(gate_up.data_ptr(), _row_major_2d(gate_up, "gate_up"), T, F,
                                   out.data_ptr(), _row_major_2d(out, "out"), _stream(stream)),
           "bi_silu_mul")
    return out


def logprobs(logits: torch.Tensor, targets: torch.Tensor | None = None, stream=None):
    """(logprob of targets [rows] fp32 or None, lse [rows] fp32) of bf16 logits
    [rows, vocab], batch-invariant per row."""
    _cuda_bf16(logits, "logits")
    rows, vocab = logits.shape
    lse = torch.empty(rows, dtype=torch.float32, device=logits.device)
    lp = None
    if targets is not None:
        if not targets.is_cuda or targets.dtype != torch.int32 or not targets.is_contiguous():
            raise ValueError("targets must be a contiguous int32 CUDA tensor")
        lp = torch.empty(rows, dtype=torch.float32, device=logits.device)
    _check(_lib.load().bi_logprobs(logits.data_ptr(), rows, vocab, _row_major_2d(logits, "logits"),
                                   targets.data_ptr() if targets is not None else None,
                                   lp.data_ptr() if lp is not None else None, lse.data_ptr(),
                                   _stream(stream)), "bi_logprobs")
    return lp, lse


# ---------------------------------------------------------------- GEMM ------
def gemm(x: torch.Tensor, W: torch.Tensor, out: torch.Tensor | None = None,
         stream=None) -> torch.Tensor:
    """Batch-invariant y = x @ W.T with x [M, K] and W [N, K] (nn.Linear layout)."""
    _cuda_bf16(x, "x")
    _cuda_bf16(W, "W")
    if x.dim() != 2 or W.dim() != 2 or x.shape[1] != W.shape[1]:
        raise ValueError("gemm: x [M, K] and W [N, K] expected")
    M, K = x.shape
    N = W.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _cuda_bf16(out, "out")
    if tuple(out.shape) != (M, N):
        raise ValueError("gemm: out has the wrong shape")
    _check(_lib.load().bi_gemm(x.data_ptr(), W.data_ptr(), out.data_ptr(), M, N, K,
                               _row_major_2d(x, "x"), _row_major_2d(W, "W"),
                               _row_major_2d(out, "out"), _stream(stream)), "bi_gemm")
    return out


def interleave_gate_up(W_gate_up: torch.Tensor) -> torch.Tensor:
    """[2F, K] weight with the gate rows first and the up rows after them ->
    the [2F, K] layout bi_gemm_swiglu reads: groups of 8 gate rows, each
    followed by the 8 matching up rows."""
    F2, K = W_gate_up.shape
    if F2 % 16:
        raise ValueError("interleave_gate_up: 2F must be a multiple of 16")
    F = F2 // 2
    g = W_gate_up[:F].reshape(F // 8, 8, K)
    u = W_gate_up[F:].reshape(F // 8, 8, K)
    return torch.cat([g, u], dim=1).reshape(F2, K).contiguous()


def gemm_swiglu(x: torch.Tensor, W_gu: torch.Tensor, out: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """Batch-invariant h = silu(x @ W_gate.T) * (x @ W_up.T), bit-identical to
    silu_mul(gemm(x, W_gate_up)); W_gu is interleave_gate_up(W_gate_up)."""
    _cuda_bf16(x, "x")
    _cuda_bf16(W_gu, "W_gu")
    if x.dim() != 2 or W_gu.dim() != 2 or x.shape[1] != W_gu.shape[1]:
        raise ValueError("gemm_swiglu: x [M, K] and W_gu [2F, K] expected")
    M, K = x.shape
    if W_gu.shape[0] % 16:
        raise ValueError("gemm_swiglu: W_gu must have 2F rows, F a multiple of 8")
    F = W_gu.shape[0] // 2
    if out is None:
        out = torch.empty((M, F), dtype=torch.bfloat16, device=x.device)
    _cuda_bf16(out, "out")
    if tuple(out.shape) != (M, F):
        raise ValueError("gemm_swiglu: out has the wrong shape")
    _check(_lib.load().bi_gemm_swiglu(x.data_ptr(), W_gu.data_ptr(), out.data_ptr(), M, F, K,
                                      _row_major_2d(x, "x"), _row_major_2d(W_gu, "W_gu"),
                                      _row_major_2d(out, "out"), _stream(stream)),
           "bi_gemm_swiglu")
    return out


# ----------------------------------------------------------- attention ------
def decode_attention_workspace_size(B: int, Hq: int, D: int, max_seq_len: int) -> int:
    return int(_lib.load().bi_decode_attention_workspace_size(B, Hq, D, max_seq_len))


def decode_num_chunks(seq_len: int) -> int:
    return int(_lib.load().bi_decode_num_chunks(seq_len))


def decode_chunk_len(seq_len: int, c: int) -> int:
    return int(_lib.load().bi_decode_chunk_len(seq_len, c))


def selftest_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the device timeout self-test (a bounded wait that must run out);
    read its outcome with get_device_error()."""
    _check(_lib.load().bi_selftest_wait_timeout(int(limit_us), _stream(stream)),
           "bi_selftest_wait_timeout")


def _attention_args(q, k_cache, v_cache, block_table, seq_lens):
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _cuda_bf16(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for t, n in ((block_table, "block_table"), (seq_lens, "seq_lens")):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    if q.dim() != 3 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("decode_attention: q [B,Hq,D] and caches [P,Hkv,page,D] expected")
    B, Hq, D = q.shape
    num_pages, Hkv, page, D2 = k_cache.shape
    if D2 != D or block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("decode_attention: inconsistent shapes")
    return B, Hq, D, num_pages, Hkv, page


def decode_attention_fixed_splits(q, k_cache, v_cache, block_table, seq_lens, max_seq_len: int,
                                  num_splits: int, scale: float | None = None, out=None,
                                  workspace=None, stream=None) -> torch.Tensor:
    """Fixed split-COUNT attention: NOT batch- or growth-invariant.  The
    comparison variant (negative control and cost reference) only."""
    B, Hq, D, num_pages, Hkv, page = _attention_args(q, k_cache, v_cache, block_table, seq_lens)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    need = decode_attention_workspace_size(B, Hq, D, int(num_splits) * DECODE_CHUNK)
    if workspace is None and need > 0:
        # the leading arrival counters must start at zero (every call leaves
        # them zero, so a caller-kept workspace is cleared only once)
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.load().bi_decode_attention_fixed_splits(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
        block_table.shape[1], seq_lens.data_ptr(), B, Hq, Hkv, D, page, num_pages,
        int(max_seq_len), float(scale), int(num_splits), out.data_ptr(), ws_ptr, ws_bytes,
        _stream(stream)), "bi_decode_attention_fixed_splits")
    return out


def prefill_attention_workspace_size(T: int, Hq: int, D: int, max_seq_len: int) -> int:
    return int(_lib.load().bi_prefill_attention_workspace_size(T, Hq, D, max_seq_len))


def prefill_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_table: torch.Tensor, seq_lens: torch.Tensor, q_indptr: torch.Tensor,
                      max_q_len: int, max_seq_len: int, scale: float | None = None,
                      out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """Causal attention for the last n_i tokens of each sequence at once.

    q [T, Hq, D]; q_indptr [S + 1] int32 (sequence i owns q rows
    q_indptr[i] .. q_indptr[i+1]-1); seq_lens [S] int32 (cached tokens,
    including the query rows); block_table [S, max_pages_per_seq] int32.
    Bit-identical per row to decode_attention with the row's own length."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _cuda_bf16(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for t, n in ((block_table, "block_table"), (seq_lens, "seq_lens"), (q_indptr, "q_indptr")):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    if q.dim() != 3 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("prefill_attention: q [T,Hq,D] and caches [P,Hkv,page,D] expected")
    T, Hq, D = q.shape
    num_pages, Hkv, page, D2 = k_cache.shape
    S = seq_lens.shape[0]
    if (D2 != D or block_table.dim() != 2 or block_table.shape[0] != S
            or tuple(q_indptr.shape) != (S + 1,)):
        raise ValueError("prefill_attention: inconsistent shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=q.device)
    _cuda_bf16(out, "out")
    if tuple(out.shape) != (T, Hq, D) or not out.is_contiguous():
        raise ValueError("prefill_attention: out must be a contiguous [T, Hq, D] tensor")
    need = prefill_attention_workspace_size(T, Hq, D, int(max_seq_len))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.load().bi_prefill_attention(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
        block_table.shape[1], seq_lens.data_ptr(), q_indptr.data_ptr(), S, T, Hq, Hkv, D, page,
        num_pages, int(max_q_len), int(max_seq_len), float(scale), out.data_ptr(), ws_ptr,
        ws_bytes, _stream(stream)), "bi_prefill_attention")
    return out


def decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                     block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                     scale: float | None = None, out: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Batch-invariant paged decode attention.

    q [B, Hq, D]; k_cache, v_cache [num_pages, Hkv, 16, D]; block_table
    [B, max_pages_per_seq] int32; seq_lens [B] int32 (1 .. max_seq_len).
    `max_seq_len` is a host-side bound on seq_lens that sizes the launch (it
    is not read from the device, so no synchronisation happens)."""
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _cuda_bf16(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    for t, n in ((block_table, "block_table"), (seq_lens, "seq_lens")):
        if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    if q.dim() != 3 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("decode_attention: q [B,Hq,D] and caches [P,Hkv,page,D] expected")
    B, Hq, D = q.shape
    num_pages, Hkv, page, D2 = k_cache.shape
    if D2 != D or block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
        raise ValueError("decode_attention: inconsistent shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    _cuda_bf16(out, "out")
    if tuple(out.shape) != (B, Hq, D) or not out.is_contiguous():
        raise ValueError("decode_attention: out must be a contiguous [B, Hq, D] tensor")
    need = decode_attention_workspace_size(B, Hq, D, max_seq_len)
    if workspace is None and need > 0:
        # the leading arrival counters must start at zero (every call leaves
        # them zero, so a caller-kept workspace is cleared only once)
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib.load().bi_decode_attention(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_table.data_ptr(),
        block_table.shape[1], seq_lens.data_ptr(), B, Hq, Hkv, D, page, num_pages,
        int(max_seq_len), float(scale), out.data_ptr(), ws_ptr, ws_bytes, _stream(stream)),
        "bi_decode_attention")
    return out
