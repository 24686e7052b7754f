"""The decoder-layer helper kernels against the fp64 oracle.

bi_add_rmsnorm must equal an elementwise bf16 add followed by bi_rmsnorm bit
for bit; bi_silu_mul and bi_qk_norm_rope_append are checked against the
oracle's fp64 silu and rotate-half RoPE (after the per-head RMSNorm, rounded
to bf16 as the kernel does).  Tolerances: 2 bf16 ulp for SwiGLU; for RoPE
2^-6 of each rotated pair's length: the normed inputs may already differ from
the oracle's by one bf16 ulp (up to 2^-7 relative, as RMSNorm's 2-ulp bound
allows), the rotation carries that into both outputs of the pair, and the
output is rounded once more -- and since a rotation can cancel, the bound is
on the pair's length rather than on each element.
"""

import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import inputs, qwen3
from oracle import decoder as odec
from tests._util import bits, f64, ulp_distance

pytestmark = pytest.mark.gpu


def test_add_rmsnorm_equals_add_then_rmsnorm_bitwise():
    x = inputs.rmsnorm_rows(300, 4096, seed=700)
    r = inputs.rmsnorm_rows(300, 4096, seed=701)
    w = inputs.rmsnorm_weight(4096, seed=702)
    xd, rd, wd = x.cuda(), r.cuda(), w.cuda()
    summed = (rd.float() + xd.float()).to(torch.bfloat16)  # one fp32 add, one rounding
    ref = bi.rmsnorm(summed, wd, 1e-6)
    res = rd.clone()
    y = bi.add_rmsnorm(xd, res, wd, 1e-6)
    assert np.array_equal(bits(res), bits(summed))
    assert np.array_equal(bits(y), bits(ref))
    # and row 17 alone gives the same bits
    res1 = rd[17:18].clone()
    y1 = bi.add_rmsnorm(xd[17:18], res1, wd, 1e-6)
    assert np.array_equal(bits(y1[0]), bits(y[17]))


def test_silu_mul_against_oracle():
    gu = inputs.normal_bf16((65, 2 * 1536), seed=710, std=3.0)
    out = bits(bi.silu_mul(gu.cuda()))
    g = gu[:, :1536].double().numpy()
    u = gu[:, 1536:].double().numpy()
    ref = oracle.round_bf16(odec.silu_mul(g, u))
    assert ulp_distance(out, ref).max() <= 2


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (3, 1), (12, 3), (5, 5), (64, 8)])
def test_qk_norm_rope_append_against_oracle(Hq, Hkv):
    # a warp works on two heads at once: odd head counts leave a pair with
    # one head, and pairs straddle the q/k and k/v boundaries
    T, D = 37, 128
    qkv = inputs.normal_bf16((T, (Hq + 2 * Hkv) * D), seed=720, std=1.5)
    qn = inputs.rmsnorm_weight(D, seed=721)
    kn = inputs.rmsnorm_weight(D, seed=722)
    pos = torch.randint(0, 4000, (T,), generator=torch.Generator().manual_seed(723)).to(torch.int32)
    num_pages = 8
    perm = torch.randperm(num_pages * 16, generator=torch.Generator().manual_seed(724))[:T]
    slots = perm.to(torch.int32)
    kc = torch.zeros(num_pages, Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    rope = qwen3.rope_table(4096, 1e6, D, device="cuda")
    q = bi.qk_norm_rope_append(qkv.cuda(), Hq, Hkv, pos.cuda(), slots.cuda(), rope, qn.cuda(),
                               kn.cuda(), kc, vc, 1e-6)
    x = qkv.double().numpy().reshape(T, Hq + 2 * Hkv, D)
    qb = oracle.round_bf16(x[:, :Hq].reshape(-1, D))
    kb = oracle.round_bf16(x[:, Hq:Hq + Hkv].reshape(-1, D))
    qn_ = oracle.bf16_to_f64(oracle.round_bf16(oracle.rmsnorm(qb, qn, 1e-6))).reshape(T, Hq, D)
    kn_ = oracle.bf16_to_f64(oracle.round_bf16(oracle.rmsnorm(kb, kn, 1e-6))).reshape(T, Hkv, D)
    pn = pos.numpy()
    q_ref = odec.rope(qn_.transpose(1, 0, 2), pn, 1e6).transpose(1, 0, 2)
    k_ref = odec.rope(kn_.transpose(1, 0, 2), pn, 1e6).transpose(1, 0, 2)

    def close(got, ref):
        pair = np.hypot(ref[..., :64], ref[..., 64:])
        tol = 2.0 ** -6 * np.concatenate([pair, pair], axis=-1) + 1e-30
        assert (np.abs(got - ref) <= tol).all(), np.abs(got - ref).max()

    close(f64(q), q_ref)
    kcc, vcc = kc.cpu(), vc.cpu()
    for t in range(T):
        s = int(slots[t])
        close(kcc[s // 16, :, s % 16].double().numpy(), k_ref[t])
        assert torch.equal(vcc[s // 16, :, s % 16], qkv[t, (Hq + Hkv) * D:].view(Hkv, D))
    # untouched slots stay zero
    used = torch.zeros(num_pages * 16, dtype=torch.bool)
    used[slots.long()] = True
    assert not kcc.permute(0, 2, 1, 3).reshape(num_pages * 16, -1)[~used].any()
