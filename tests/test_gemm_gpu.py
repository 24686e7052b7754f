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
def test_c3_rows_invariant_across_m_and_sampled_parity(name):
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
    # sampled parity at the full size: every output tile row/col class covered
    rng = np.random.default_rng(4)
    ms = np.concatenate([rng.integers(0, 4096, 600), [0, 127, 128, 4095]])
    ns = np.concatenate([rng.integers(0, N, 600), [0, 255, 256, N - 1]])
    ref = oracle.gemm_entries(pool, W, ms, ns)
    got = f64(big)[ms, ns]
    err = np.abs(got - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()
    absdot = oracle.gemm_entries(pool.abs(), W.abs(), ms, ns)
    assert (err <= 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -22 * absdot + 1e-30).all()
