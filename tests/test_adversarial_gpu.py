"""Adversarial inputs against the oracle: peaked and flat softmaxes, heavy
cancellation in long dot products, extreme and subnormal RMSNorm rows, huge
and tied logits.  Each keeps the kernel-specific tolerances (stated in the
other test files) and the bitwise alone-vs-batched property."""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import inputs
from tests._util import bits, f64, ulp_distance

pytestmark = pytest.mark.gpu


def _attn(p, **kw):
    d = {k: v.cuda() for k, v in p.items()}
    return bi.decode_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                               d["seq_lens"], max_seq_len=int(p["seq_lens"].max()), **kw)


def _check_attn(out, ref):
    err = np.abs(f64(out) - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()
    assert (err.max(axis=-1) <= 2.0 ** -6 * np.abs(ref).max(axis=-1) + 2.0 ** -12).all()


@pytest.mark.parametrize("qscale", [0.0, 8.0, 40.0])
def test_attention_flat_and_peaked_softmax(qscale):
    """q = 0 makes every score equal (the output is the mean of V over the
    sequence, across chunk boundaries); a large q makes the softmax nearly
    one-hot, so one token's V dominates and the LSE merge must keep it."""
    lens = [1, 255, 256, 257, 1000, 3000]
    p = inputs.decode_problem(len(lens), seq_lens=lens, seed=1200)
    p["q"] = (p["q"].float() * qscale).to(torch.bfloat16)
    out = _attn(p)
    _check_attn(out, oracle.decode_attention(**p))
    if qscale == 0.0:
        # flat: the mean of each sequence's V rows, per kv head
        for s, L in enumerate(lens):
            pages = p["block_table"][s][: (L + 15) // 16].long()
            v = p["v_cache"][pages].double()              # [pages, Hkv, 16, 128]
            v = v.permute(1, 0, 2, 3).reshape(8, -1, 128)[:, :L]
            mean = v.mean(dim=1).repeat_interleave(4, dim=0).numpy()
            assert np.abs(f64(out[s]) - mean).max() <= 2.0 ** -7 * np.abs(mean).max() + 2.0 ** -12
    for s in (0, 4):
        one = _attn({k: (v[s:s + 1] if k in ("q", "block_table", "seq_lens") else v)
                     for k, v in p.items()})
        assert torch.equal(one[0], out[s])
    bi.get_device_error()


def test_attention_large_value_magnitudes():
    """K and V entries of magnitude ~1e3 (scores ~1e5 before scaling): the
    online max subtraction keeps exp2 in range."""
    lens = [17, 600]
    p = inputs.decode_problem(len(lens), seq_lens=lens, seed=1201)
    p["k_cache"] = (p["k_cache"].float() * 30.0).to(torch.bfloat16)
    p["v_cache"] = (p["v_cache"].float() * 1000.0).to(torch.bfloat16)
    out = _attn(p)
    assert torch.isfinite(out.float()).all()
    _check_attn(out, oracle.decode_attention(**p))
    bi.get_device_error()


def test_gemm_heavy_cancellation():
    """Rows whose products cancel to a small fraction of sum |x w|: the
    derived per-element bound (2^-8 |ref| + K 2^-22 sum|x w|) still holds and
    rows stay bit-identical alone vs batched."""
    K, N, M = 12288, 512, 40
    g = torch.Generator().manual_seed(1202)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    base = torch.randn(M, K // 2, generator=g)
    x = torch.cat([base, -base], dim=1)             # x . w cancels up to the W difference
    x = (x + torch.randn(M, K, generator=g) * 1e-3).to(torch.bfloat16)
    y = bi.gemm(x.cuda(), W.cuda())
    ref = oracle.gemm(x, W)
    absdot = oracle.gemm(x.abs(), W.abs())
    err = np.abs(f64(y) - ref)
    assert (err <= 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -22 * absdot + 1e-30).all()
    assert torch.equal(bi.gemm(x[7:8].cuda(), W.cuda())[0], y[7])
    bi.get_device_error()


def test_rmsnorm_extreme_rows():
    """Rows of huge (1e15), tiny (subnormal bf16) and mixed magnitudes."""
    H = 4096
    g = torch.Generator().manual_seed(1203)
    rows = torch.randn(6, H, generator=g)
    rows[0] *= 1e15
    rows[1] *= 1e-38                                  # bf16 subnormals; eps dominates
    rows[2, : H // 2] *= 1e10                         # half huge, half O(1)
    rows[3] = 0.0
    rows[3, 17] = 3.0e4                               # one-hot
    rows[4] *= 1e-20
    x = rows.to(torch.bfloat16)
    w = inputs.rmsnorm_weight(H, seed=1204)
    y = bi.rmsnorm(x.cuda(), w.cuda(), 1e-6)
    ref = oracle.round_bf16(oracle.rmsnorm(x, w, 1e-6))
    assert ulp_distance(bits(y), ref).max() <= 2
    for r in (0, 1, 3):
        assert torch.equal(bi.rmsnorm(x[r:r + 1].cuda(), w.cuda(), 1e-6)[0], y[r])
    bi.get_device_error()


def test_logprobs_huge_and_tied_logits():
    """Logits around 1e4 (exp overflows without the max shift), a row of all
    equal values (lse = x + log V exactly up to rounding), and ties at the max."""
    V = 151936
    x = inputs.normal_bf16((4, V), seed=1205, std=2.0)
    x[0] = (x[0].float() + 1.0e4).to(torch.bfloat16)
    x[1] = 7.0
    x[2, 5] = 50.0
    x[2, 100000] = 50.0
    t = torch.tensor([3, 9, 100000, 11], dtype=torch.int32)
    lp, lse = bi.logprobs(x.cuda(), t.cuda())
    lp_ref, lse_ref = oracle.logprobs(x, t.numpy())
    # lse is an fp32 number: near 1e4 its spacing is 2^-10, and the log-prob
    # x_t - lse inherits that absolute error, so the bound scales with |lse|
    bound = 1e-4 + 2.0 ** -22 * np.abs(lse_ref)
    for got, ref in ((lp, lp_ref), (lse, lse_ref)):
        g_ = got.cpu().double().numpy()
        assert np.isfinite(g_).all()
        assert (np.abs(g_ - ref) <= bound).all(), np.abs(g_ - ref).max()
    bi.get_device_error()
