"""Seeded random shapes and batch compositions for every reduction kernel.

Each case draws its sizes from a fixed seed, then checks two things. First,
parity with the fp64 oracle, at the tolerances the kernel-specific tests use.
Second, that rows computed alone, or inside a different batch, are
bit-identical to the same rows in the full batch. The shapes cover sizes the
hand-picked tests do not: odd row counts, non-multiple-of-tile N and K,
lengths on and off page and chunk edges, and every GQA group size."""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import inputs
from tests._util import bits, f64, ulp_distance

pytestmark = pytest.mark.gpu


def _rng(seed):
    return np.random.default_rng(seed)


@pytest.mark.parametrize("seed", range(8))
def test_gemm_random_shapes(seed):
    r = _rng(1000 + seed)
    M = int(r.integers(1, 700))
    N = 8 * int(r.integers(1, 150))
    K = 8 * int(r.integers(1, 100))
    W = inputs.gemm_weight(N, K, seed=2000 + seed)
    x = inputs.gemm_rows(M, K, seed=3000 + seed)
    Wd, xd = W.cuda(), x.cuda()
    y = bi.gemm(xd, Wd)
    ref = oracle.gemm(x, W)
    absdot = oracle.gemm(x.abs(), W.abs())
    err = np.abs(f64(y) - ref)
    assert (err <= 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -22 * absdot + 1e-30).all(), (M, N, K)
    # a random subset of rows, alone and as a smaller batch, in shuffled order
    pick = r.choice(M, size=min(M, int(r.integers(1, 9))), replace=False)
    sub = bi.gemm(xd[torch.as_tensor(pick)].contiguous(), Wd)
    assert torch.equal(sub, y[torch.as_tensor(pick)]), (M, N, K, pick)
    one = bi.gemm(xd[int(pick[0]):int(pick[0]) + 1].contiguous(), Wd)
    assert torch.equal(one[0], y[int(pick[0])])
    bi.get_device_error()


@pytest.mark.parametrize("seed", range(6))
def test_rmsnorm_random_shapes(seed):
    r = _rng(4000 + seed)
    H = 8 * int(r.integers(1, 1024))
    B = int(r.integers(1, 300))
    x = inputs.rmsnorm_rows(B, H, seed=5000 + seed)
    w = inputs.rmsnorm_weight(H, seed=6000 + seed)
    xd, wd = x.cuda(), w.cuda()
    y = bi.rmsnorm(xd, wd, 1e-6)
    ref = oracle.round_bf16(oracle.rmsnorm(x, w, 1e-6))
    assert ulp_distance(bits(y), ref).max() <= 2, (B, H)
    pick = r.choice(B, size=min(B, 5), replace=False)
    sub = bi.rmsnorm(xd[torch.as_tensor(pick)].contiguous(), wd, 1e-6)
    assert torch.equal(sub, y[torch.as_tensor(pick)]), (B, H)
    bi.get_device_error()


def _check_attention(out, ref):
    err = np.abs(f64(out) - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()
    assert (err.max(axis=-1) <= 2.0 ** -6 * np.abs(ref).max(axis=-1) + 2.0 ** -12).all()


EDGES = [1, 15, 16, 17, 255, 256, 257, 4096, 4097]


@pytest.mark.parametrize("seed", range(6))
def test_decode_attention_random_batches(seed):
    r = _rng(7000 + seed)
    Hkv = int(r.choice([1, 2, 4, 8]))
    G = int(r.choice([1, 2, 4, 8]))
    B = int(r.integers(1, 24))
    lens = [int(r.choice(EDGES)) if r.random() < 0.4 else int(r.integers(1, 3000))
            for _ in range(B)]
    p = inputs.decode_problem(B, Hq=Hkv * G, Hkv=Hkv, seq_lens=lens, seed=8000 + seed,
                              spare_pages=2)
    d = {k: v.cuda() for k, v in p.items()}
    mx = max(lens)

    def run(idx):
        i = torch.as_tensor(idx, dtype=torch.long, device="cuda")
        return bi.decode_attention(d["q"][i].contiguous(), d["k_cache"], d["v_cache"],
                                   d["block_table"][i].contiguous(), d["seq_lens"][i].contiguous(),
                                   max_seq_len=mx)
    full = run(list(range(B)))
    _check_attention(full, oracle.decode_attention(p["q"], p["k_cache"], p["v_cache"],
                                                   p["block_table"], p["seq_lens"]))
    for _ in range(3):
        idx = list(r.permutation(B)[:int(r.integers(1, B + 1))])
        sub = run(idx)
        assert torch.equal(sub, full[torch.as_tensor(idx, device="cuda")]), (seed, idx)
    bi.get_device_error()


@pytest.mark.parametrize("seed", range(4))
def test_prefill_random_chunkings_equal_decode(seed):
    r = _rng(9000 + seed)
    S = int(r.integers(1, 5))
    lens = [int(r.integers(1, 700)) for _ in range(S)]
    Hq, Hkv = 32, 8
    p = inputs.decode_problem(S, Hq=Hq, Hkv=Hkv, seq_lens=lens, seed=9500 + seed)
    T = sum(lens)
    q = inputs.decode_queries(T, Hq, 128, seed=9600 + seed)
    d = {k: v.cuda() for k, v in p.items() if k != "q"}
    qd = q.cuda()
    # each prompt's rows as decode rows of their own causal lengths
    rows = [(s, j + 1) for s, L in enumerate(lens) for j in range(L)]
    sidx = torch.tensor([s for s, _ in rows], dtype=torch.long, device="cuda")
    dlens = torch.tensor([L for _, L in rows], dtype=torch.int32, device="cuda")
    dec = bi.decode_attention(qd, d["k_cache"], d["v_cache"], d["block_table"][sidx].contiguous(),
                              dlens, max_seq_len=max(lens))
    # the last part of each prompt (a random chunk) as prefill rows
    nq = [int(r.integers(1, L + 1)) for L in lens]
    starts = np.cumsum([0] + lens)
    take = torch.cat([torch.arange(int(starts[s] + lens[s] - nq[s]), int(starts[s] + lens[s]))
                      for s in range(S)]).cuda()
    indptr = torch.tensor([0] + list(np.cumsum(nq)), dtype=torch.int32, device="cuda")
    pre = bi.prefill_attention(qd[take].contiguous(), d["k_cache"], d["v_cache"],
                               d["block_table"], d["seq_lens"], indptr, max_q_len=max(nq),
                               max_seq_len=max(lens))
    assert torch.equal(pre, dec[take]), (lens, nq)
    bi.get_device_error()
