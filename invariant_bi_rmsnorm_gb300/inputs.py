"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module draws random numbers and lays them out; it holds none of the
arithmetic of the kernels or of the oracle.  By default everything is generated on
the CPU with ``torch.Generator``, so the same seed gives the same bits on any
machine.  Multi-gigabyte inputs (the benchmark's KV caches and weights) can be
drawn on a CUDA device instead (``device="cuda"``): torch's seeded Philox
generator, deterministic for a given seed on a given GPU; whatever checks them
against the oracle copies the drawn tensors to the host.

Shapes and distributions follow the Qwen3-8B-shaped workloads the kernels are
measured on:
  * GEMM:       weights W ~ N(0, 0.02) stored [N, K]; activations ~ N(0, 1).
  * RMSNorm:    rows ~ N(0, 1) with each element independently (p = 0.01)
                multiplied by 100 before rounding to bf16; weight ~ N(1, 0.1).
  * Attention:  q, k, v ~ N(0, 1); sequence lengths uniform on [1, max_len];
                KV pages handed out by a seeded random permutation, so
                sequences own scattered, non-contiguous pages.
"""
from __future__ import annotations

import torch

PAGE_SIZE = 16  # tokens per KV page


def _gen(seed: int, device=None) -> torch.Generator:
    g = torch.Generator(device=torch.device(device or "cpu"))
    g.manual_seed(int(seed))
    return g


def _dev(device):
    return torch.device(device or "cpu")


def normal_bf16(shape, seed: int, mean: float = 0.0, std: float = 1.0,
                device=None) -> torch.Tensor:
    """bf16 tensor of N(mean, std) draws (drawn in fp32, rounded once to bf16)."""
    t = torch.randn(*shape, generator=_gen(seed, device), dtype=torch.float32,
                    device=_dev(device))
    return (t * std + mean).to(torch.bfloat16)


# ---------------------------------------------------------------- GEMM ------
def gemm_weight(N: int, K: int, seed: int = 1, device=None) -> torch.Tensor:
    """nn.Linear-layout weight [N, K] ~ N(0, 0.02)."""
    return normal_bf16((N, K), seed, std=0.02, device=device)


def gemm_rows(M: int, K: int, seed: int = 2, device=None) -> torch.Tensor:
    """Activation rows [M, K] ~ N(0, 1), drawn as one block.  Tests that need
    the same row in batches of different sizes slice one pool of rows."""
    return normal_bf16((M, K), seed, device=device)


# ------------------------------------------------------------- RMSNorm ------
def rmsnorm_rows(B: int, H: int, seed: int = 3, outlier_p: float = 0.01,
                 outlier_scale: float = 100.0, device=None) -> torch.Tensor:
    """Rows [B, H] ~ N(0, 1), each element independently scaled by
    `outlier_scale` with probability `outlier_p` (scaled in fp32, then rounded)."""
    g = _gen(seed, device)
    x = torch.randn(B, H, generator=g, dtype=torch.float32, device=_dev(device))
    mask = torch.rand(B, H, generator=g, dtype=torch.float32, device=_dev(device)) < outlier_p
    x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def rmsnorm_weight(H: int, seed: int = 4, device=None) -> torch.Tensor:
    """Norm weight [H] ~ N(1, 0.1)."""
    return normal_bf16((H,), seed, mean=1.0, std=0.1, device=device)


# ----------------------------------------------------------- attention ------
def seq_lens_uniform(B: int, max_len: int, seed: int = 5, min_len: int = 1) -> torch.Tensor:
    """Per-sequence KV lengths, int32, uniform on [min_len, max_len]."""
    return torch.randint(min_len, max_len + 1, (B,), generator=_gen(seed),
                         dtype=torch.int64).to(torch.int32)


def paged_layout(seq_lens: torch.Tensor, seed: int = 6, page_size: int = PAGE_SIZE,
                 spare_pages: int = 0, max_pages_per_seq: int | None = None):
    """Assign pages to sequences by a seeded random permutation.

    Returns (block_table [B, max_pages_per_seq] int32, num_pages).  Entries
    past a sequence's last page are -1 (never read).  `spare_pages` extra
    pages belong to nobody, so stray reads of them would show up."""
    lens = [int(v) for v in seq_lens.tolist()]
    need = [(L + page_size - 1) // page_size for L in lens]
    total = sum(need)
    if max_pages_per_seq is None:
        max_pages_per_seq = max(need) if need else 1
    num_pages = total + spare_pages
    perm = torch.randperm(num_pages, generator=_gen(seed)).to(torch.int32)
    bt = torch.full((len(lens), max(1, max_pages_per_seq)), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[off:off + n]
        off += n
    return bt, max(num_pages, 1)


def kv_cache(num_pages: int, Hkv: int, D: int, seed: int = 7,
             page_size: int = PAGE_SIZE, device=None):
    """K and V caches [num_pages, Hkv, page_size, D] bf16, ~ N(0, 1)."""
    shape = (num_pages, Hkv, page_size, D)
    return (normal_bf16(shape, seed, device=device),
            normal_bf16(shape, seed + 1_000_003, device=device))


def decode_queries(B: int, Hq: int, D: int, seed: int = 8, device=None) -> torch.Tensor:
    """One query row per sequence, [B, Hq, D] bf16 ~ N(0, 1)."""
    return normal_bf16((B, Hq, D), seed, device=device)


def decode_problem(B: int, Hq: int = 32, Hkv: int = 8, D: int = 128,
                   max_len: int = 8192, seed: int = 11, seq_lens=None,
                   spare_pages: int = 0, page_size: int = PAGE_SIZE, device=None):
    """A whole paged-decode input set.  Returns a dict with q, k_cache,
    v_cache, block_table, seq_lens.  Lengths and the page table are always
    drawn on the CPU; q and the caches on `device` (default CPU)."""
    if seq_lens is None:
        seq_lens = seq_lens_uniform(B, max_len, seed=seed + 1)
        width = (max_len + page_size - 1) // page_size  # room for any length <= max_len
    else:
        seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32)
        width = None
    bt, num_pages = paged_layout(seq_lens, seed=seed + 2, page_size=page_size,
                                 spare_pages=spare_pages, max_pages_per_seq=width)
    k, v = kv_cache(num_pages, Hkv, D, seed=seed + 3, page_size=page_size, device=device)
    q = decode_queries(len(seq_lens), Hq, D, seed=seed + 4, device=device)
    return {"q": q, "k_cache": k, "v_cache": v, "block_table": bt,
            "seq_lens": seq_lens}
