"""The premise of the tcgen05 prefill: on this GPU, tcgen05.mma and the
mma.sync steps decode uses give the same fp32 bits for the same 16-deep
products (operand roles swapped), both for the page scores S = Q . K^T and
for the output update O0 + P . V.  "3. Batch-Invariant Attention" warns that
different tensor-core instructions may reduce in different orders, so this is
checked element by element -- the fp32 accumulators, before any rounding to
bf16 could hide a difference -- on random data and on inputs built to expose
a different internal order or precision: products spread over a wide
exponent range, exact cancellation, tiny (subnormal-range) products, signed
zeros, accumulators that dominate the products, and a zero accumulator
(the first page of every chunk starts from zero).
"""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
from invariant_bi_rmsnorm_gb300 import _lib

pytestmark = pytest.mark.gpu


def _run(q, k, v, p, o0):
    lib = _lib.load()
    dev = torch.device("cuda")
    q, k, v, p = (t.to(dev, torch.bfloat16).contiguous() for t in (q, k, v, p))
    o0 = o0.to(dev, torch.float32).contiguous()
    s_tc = torch.full((128, 16), float("nan"), device=dev)
    s_mma = torch.full_like(s_tc, float("nan"))
    o_tc = torch.full((128, 128), float("nan"), device=dev)
    o_mma = torch.full_like(o_tc, float("nan"))
    st = torch.cuda.current_stream().cuda_stream
    assert lib.bi_selftest_tcgen05_vs_mma_sync(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), p.data_ptr(), o0.data_ptr(), s_tc.data_ptr(),
        s_mma.data_ptr(), o_tc.data_ptr(), o_mma.data_ptr(), st) == _lib.BI_OK
    bi.get_device_error()
    return [t.cpu().numpy().view(np.uint32) for t in (s_tc, s_mma, o_tc, o_mma)]


def _assert_same(name, a, b):
    diff = np.count_nonzero(a != b)
    assert diff == 0, f"{name}: {diff} of {a.size} fp32 results differ between tcgen05 and mma.sync"


def _case(kind, seed):
    g = torch.Generator().manual_seed(seed)
    n = lambda *s: torch.randn(*s, generator=g)  # noqa: E731
    q, k, v = n(128, 128), n(16, 128), n(16, 128)
    p = torch.rand(128, 16, generator=g)
    o0 = n(128, 128)
    if kind == "scaled":
        q, k, v, o0 = q * 30, k * 30, v * 300, o0 * 1e4
    elif kind == "wide_exponents":
        # each 16-deep step mixes products from 2^-40 to 2^40
        e = torch.randint(-20, 21, (128, 128), generator=g).float()
        q = q * torch.exp2(e)
        k = k * torch.exp2(torch.randint(-20, 21, (16, 128), generator=g).float())
        v = v * torch.exp2(torch.randint(-20, 21, (16, 128), generator=g).float())
        p = p * torch.exp2(torch.randint(-30, 1, (128, 16), generator=g).float())
    elif kind == "cancellation":
        # pairs of dims / tokens whose products cancel exactly, plus a small rest
        q[:, 1::2] = q[:, 0::2]
        k[:, 1::2] = -k[:, 0::2]
        k[:, 0] += 1e-3
        v[1::2] = -v[0::2]
        p[:, 1::2] = p[:, 0::2]
        o0 = o0 * 1e-3
    elif kind == "tiny":
        # products near and below the fp32 normal range
        q, k = q * 2.0 ** -62, k * 2.0 ** -62
        v, p = v * 2.0 ** -70, p * 2.0 ** -60
        o0 = o0 * 2.0 ** -126
    elif kind == "signed_zeros":
        q[:, :64] = -0.0
        k[:8] = 0.0
        v[:, ::3] = -0.0
        p[::2] = 0.0
        o0[::3] = -0.0
    elif kind == "dominant_accumulator":
        o0 = o0 * 2.0 ** 24
    elif kind == "zero_accumulator":
        # products onto a zero accumulator (weights with exact zeros and
        # products of both signs, so zero sums of either sign occur)
        o0 = torch.zeros_like(o0)
        p[:, ::2] = 0.0
        v[3] = -0.0
    return q, k, v, p, o0


@pytest.mark.parametrize("kind", ["random", "scaled", "wide_exponents", "cancellation", "tiny",
                                  "signed_zeros", "dominant_accumulator", "zero_accumulator"])
def test_tcgen05_and_mma_sync_accumulate_identically(kind):
    for seed in range(3):
        s_tc, s_mma, o_tc, o_mma = _run(*_case(kind, 700 + seed))
        assert not np.isnan(s_tc.view(np.float32)).any() and not np.isnan(o_tc.view(np.float32)).any()
        _assert_same(f"{kind} S", s_tc, s_mma)
        _assert_same(f"{kind} O", o_tc, o_mma)
