"""Row counts far past the bench's: the index arithmetic, grids and schedules
at sizes where each kernel walks many waves (and, for the GEMM, many tiles per
CTA pair and several M-tile groups), checked on sampled rows against the fp64
oracle and by the same rows computed alone.

- GEMM: M = 100003 rows of K = 1024 into N = 1032 (391 M-tiles, a ragged last
  one; 5 N-tiles, a ragged last one).
- RMSNorm: 1,000,003 rows of hidden 128 (one CTA per row: a million CTAs).
- Decode attention: 8192 sequences of 1 to 64 tokens (one CTA row of the grid
  per sequence), and 2048 sequences of 1 to 700 tokens (up to three chunks).
"""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import inputs
from tests._util import bits, f64, ulp_distance

pytestmark = pytest.mark.gpu


def test_gemm_hundred_thousand_rows():
    M, N, K = 100003, 1032, 1024
    W = inputs.gemm_weight(N, K, seed=41)
    x = inputs.gemm_rows(M, K, seed=42)
    Wd, xd = W.cuda(), x.cuda()
    y = bi.gemm(xd, Wd)
    rows = np.array([0, 1, 255, 256, 50000, 65535, 65536, 99840, 100002])
    ref = oracle.gemm(x[torch.as_tensor(rows)], W)
    absdot = oracle.gemm(x[torch.as_tensor(rows)].abs(), W.abs())
    err = np.abs(f64(y[torch.as_tensor(rows, device="cuda")]) - ref)
    # bf16 output rounding (2^-8 relative) plus fp32 accumulation over K terms
    assert (err <= 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -22 * absdot + 1e-30).all()
    for r in (0, 65536, 100002):
        one = bi.gemm(xd[r:r + 1].contiguous(), Wd)
        assert torch.equal(one[0], y[r]), r
    bi.get_device_error()


def test_rmsnorm_million_rows():
    B, H = 1_000_003, 128
    x = inputs.rmsnorm_rows(B, H, seed=43)
    w = inputs.rmsnorm_weight(H, seed=44)
    xd, wd = x.cuda(), w.cuda()
    y = bi.rmsnorm(xd, wd, 1e-6)
    rows = torch.as_tensor(np.r_[0:64, 524288:524352, B - 64:B])
    ref = oracle.round_bf16(oracle.rmsnorm(x[rows], w, 1e-6))
    assert ulp_distance(bits(y[rows.cuda()]), ref).max() <= 2
    for r in (0, 777777, B - 1):
        one = bi.rmsnorm(xd[r:r + 1], wd, 1e-6)
        assert torch.equal(one[0], y[r]), r
    bi.get_device_error()


def _check_attention(out, ref):
    err = np.abs(f64(out) - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()


@pytest.mark.parametrize("B,max_len", [(8192, 64), (2048, 700)])
def test_decode_attention_many_sequences(B, max_len):
    g = torch.Generator().manual_seed(45 + B)
    lens = torch.randint(1, max_len + 1, (B,), generator=g, dtype=torch.int32)
    # caches drawn on the device (a few GB), copied to the host for the oracle
    d = inputs.decode_problem(B, seq_lens=lens, seed=46 + B, device="cuda")
    d = {k: v.cuda() for k, v in d.items()}
    p = {k: v.cpu() for k, v in d.items()}
    out = bi.decode_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                              d["seq_lens"], max_seq_len=max_len)
    pick = sorted({0, 1, B // 2, B - 2, B - 1} | set(range(0, B, B // 16)))
    i = torch.as_tensor(pick)
    ref = oracle.decode_attention(p["q"][i], p["k_cache"], p["v_cache"], p["block_table"][i],
                                  p["seq_lens"][i])
    _check_attention(out[i.cuda()], ref)
    for r in (0, B // 2, B - 1):
        one = bi.decode_attention(d["q"][r:r + 1], d["k_cache"], d["v_cache"],
                                  d["block_table"][r:r + 1].contiguous(), d["seq_lens"][r:r + 1],
                                  max_seq_len=max_len)
        assert torch.equal(one[0], out[r]), r
    bi.get_device_error()
