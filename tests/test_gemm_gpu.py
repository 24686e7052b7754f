"""bi_gemm on the GPU: parity with the fp64 oracle and bitwise batch invariance.

Tolerances: the stated one, max|gpu - ref| <= 1e-2 * max|ref| per call, and a
tighter per-element bound derived from the arithmetic (one bf16 rounding of
the output plus fp32 accumulation over K terms):
    |gpu - ref| <= 2^-8 * |ref| + K * 2^-22 * sum_k |x_k w_k|
which a dropped or doubled K block, a wrong tile row, or a transposed operand
would all exceed.
"""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import inputs
from tests._util import bits, f64

pytestmark = pytest.mark.gpu


def _check_parity(y_gpu, x, W, ref=None):
    if ref is None:
        ref = oracle.gemm(x, W)
    absdot = oracle.gemm(x.abs(), W.abs())
    err = np.abs(f64(y_gpu) - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max(), f"max err {err.max()} vs max|ref| {np.abs(ref).max()}"
    K = x.shape[1]
    bound = 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -22 * absdot + 1e-30
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} elements beyond the derived bound; first at {np.argwhere(bad)[0]}"


# ------------------------------------------- C1: K = N = 1024, M in {1, 32} ---
def test_c1_row_alone_and_embedded_bit_identical():
    K = N = 1024
    W = inputs.gemm_weight(N, K, seed=1)
    pool = inputs.gemm_rows(64, K, seed=2)
    r = pool[0:1]
    Wd = W.cuda()
    alone = bi.gemm(r.cuda(), Wd)
    _check_parity(alone, r, W)
    for pos in (0, 7, 31):
        others = pool[32:64].clone()
        others[pos] = r[0]
        y = bi.gemm(others.cuda(), Wd)
        assert np.array_equal(bits(y[pos]), bits(alone[0])), f"position {pos} differs"
        _check_parity(y, others, W)


def test_run_to_run_deterministic():
    W = inputs.gemm_weight(1024, 1024, seed=1).cuda()
    x = inputs.gemm_rows(300, 1024, seed=5).cuda()
    assert np.array_equal(bits(bi.gemm(x, W)), bits(bi.gemm(x, W)))


# --------------------------------------------- ragged shapes and edge cases ---
@pytest.mark.parametrize("M,N,K", [
    (1, 8, 8), (5, 24, 72), (127, 256, 64), (128, 256, 128), (129, 264, 200),
    (300, 1000, 1000), (257, 512, 4104), (64, 2056, 520)])
def test_ragged_shapes_against_oracle(M, N, K):
    x = inputs.gemm_rows(M, K, seed=M + 7)
    W = inputs.gemm_weight(N, K, seed=N + 11)
    _check_parity(bi.gemm(x.cuda(), W.cuda()), x, W)


def test_strided_operands():
    x = inputs.gemm_rows(40, 512 + 24, seed=31)
    W = inputs.gemm_weight(96, 512 + 8, seed=32)
    out = torch.zeros(40, 96 + 16, dtype=torch.bfloat16, device="cuda")
    y = bi.gemm(x.cuda()[:, :512], W.cuda()[:, :512], out=out[:, :96])
    _check_parity(y, x[:, :512].contiguous(), W[:, :512].contiguous())
    assert not out[:, 96:].any()  # nothing written past N


def test_identity_weight_returns_x_exactly():
    K = 256
    x = inputs.gemm_rows(33, K, seed=33)
    I = torch.eye(K, dtype=torch.bfloat16)
    assert np.array_equal(bits(bi.gemm(x.cuda(), I.cuda())), bits(x))


def test_empty_m_is_a_no_op():
    W = inputs.gemm_weight(64, 64).cuda()
    y = bi.gemm(torch.empty(0, 64, dtype=torch.bfloat16, device="cuda"), W)
    assert y.shape == (0, 64)
    bi.get_device_error()


# --------------------------- C3: Qwen3-8B-shaped layers, invariance over M ---
C3 = {"qkv": (6144, 4096), "o": (4096, 4096), "gate_up": (24576, 4096), "down": (4096, 12288)}


@pytest.mark.parametrize("name", list(C3))
def test_c3_rows_invariant_across_m_and_full_parity(name):
    N, K = C3[name]
    W = inputs.gemm_weight(N, K, seed=40)
    Wd = W.cuda()
    pool = inputs.gemm_rows(4096, K, seed=41)
    xd = pool.cuda()
    big = bi.gemm(xd, Wd)
    bb = bits(big)
    for M in (1, 8, 64, 256, 1024):
        ym = bits(bi.gemm(xd[:M].contiguous(), Wd))
        assert np.array_equal(ym, bb[:M]), f"{name}: rows of M={M} differ from M=4096"
    perm = torch.randperm(4096, generator=torch.Generator().manual_seed(3))
    yp = bits(bi.gemm(xd[perm.cuda()].contiguous(), Wd))
    assert np.array_equal(yp, bb[perm.numpy()]), f"{name}: permuted batch differs"
    # every entry of the full-size layer against the fp64 oracle
    ref = oracle.gemm(pool, W)
    err = np.abs(f64(big) - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()
    # fp32 accumulation over K plus the bf16 output rounding; sum_k |x||W| is
    # only a bound factor, so numpy's fp32 product (with a small margin) serves
    absdot = np.abs(pool.float().numpy()) @ np.abs(W.float().numpy()).T
    bound = 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -22 * (1.0 + 2.0 ** -10) * absdot + 1e-30
    bad = np.count_nonzero(err > bound)
    assert bad == 0, f"{name}: {bad} of {err.size} entries outside the bound"


# ------------------------------- fused gate|up GEMM + SwiGLU (decoder MLP) ---
@pytest.mark.parametrize("M,F,K", [(1, 12288, 4096), (300, 12288, 4096), (37, 200, 192),
                                   (513, 8, 64)])
def test_gemm_swiglu_equals_gemm_then_silu_mul_bitwise(M, F, K):
    """The fused epilogue rounds gate and up to bf16 as bi_gemm stores them and
    applies bi_silu_mul's arithmetic, so the two paths agree bit for bit --
    across ragged N tiles (2F = 400 and 16 leave a partial last tile) and M."""
    W = inputs.gemm_weight(2 * F, K, seed=70).cuda()
    x = inputs.gemm_rows(M, K, seed=71).cuda()
    unfused = bi.silu_mul(bi.gemm(x, W))
    fused = bi.gemm_swiglu(x, bi.interleave_gate_up(W))
    assert torch.equal(fused, unfused)
    bi.get_device_error()


def test_gemm_swiglu_rows_invariant_and_against_oracle():
    """Rows alone vs in a batch of 512, bitwise; and the fused result against
    the oracle's GEMM rounded to bf16 with SwiGLU in fp64."""
    from oracle import decoder as odec
    F, K = 200, 256
    W = inputs.gemm_weight(2 * F, K, seed=72)
    x = inputs.gemm_rows(512, K, seed=73)
    Wi = bi.interleave_gate_up(W.cuda())
    full = bi.gemm_swiglu(x.cuda(), Wi)
    for r in (0, 255, 511):
        assert torch.equal(bi.gemm_swiglu(x[r:r + 1].cuda(), Wi)[0], full[r])
    gu = oracle.bf16_to_f64(oracle.round_bf16(oracle.gemm(x, W)))
    g, u = gu[:, :F], gu[:, F:]
    ref = odec.silu_mul(g, u)
    err = np.abs(f64(full) - ref)
    # g and u may each sit one bf16 step (<= 2^-7 relative) from the oracle's
    # rounding of the exact sum (fp32 accumulation can cross a rounding
    # boundary); propagate that through silu(g) * u, plus the output rounding
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    bound = (2.0 ** -8 * np.abs(ref) + np.abs(dsilu * u) * 2.0 ** -7 * np.abs(g)
             + np.abs(g * sig) * 2.0 ** -7 * np.abs(u) + 1e-30)
    assert (err <= bound).all(), (err / bound).max()
    bi.get_device_error()
