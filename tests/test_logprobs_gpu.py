"""bi_logprobs on the GPU: parity with the fp64 oracle and bitwise row
invariance across batches.  Tolerance, derived from fp32 arithmetic: the sum
of exp over V terms carries a relative error of about V * 2^-24 at worst,
which log turns into an absolute error; |gpu - ref| <= 1e-4 + 1e-6 |ref|
covers V = 151936 with margin, and is far below what a wrong max, a dropped
term or an off-by-one target would cause."""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu

V = 151936


def test_logprobs_match_oracle_and_are_row_invariant():
    x = inputs.normal_bf16((64, V), seed=91, std=2.0)
    x[5, 123] = 40.0  # a dominant entry
    t = torch.randint(0, V, (64,), generator=torch.Generator().manual_seed(92)).to(torch.int32)
    t[5] = 123
    xd, td = x.cuda(), t.cuda()
    lp, lse = bi.logprobs(xd, td)
    lp_ref, lse_ref = oracle.logprobs(x, t.numpy())
    for got, ref in ((lp, lp_ref), (lse, lse_ref)):
        g = got.cpu().double().numpy()
        assert (np.abs(g - ref) <= 1e-4 + 1e-6 * np.abs(ref)).all(), np.abs(g - ref).max()
    for r in (0, 5, 63):
        lp1, lse1 = bi.logprobs(xd[r:r + 1], td[r:r + 1])
        assert torch.equal(lp1.cpu(), lp[r:r + 1].cpu()) and torch.equal(lse1.cpu(), lse[r:r + 1].cpu())
    bi.get_device_error()


def test_bad_target_reported_without_fault():
    x = inputs.normal_bf16((2, 1024), seed=93).cuda()
    bi.get_device_error()
    lp, _ = bi.logprobs(x, torch.tensor([3, 5000], dtype=torch.int32, device="cuda"))
    with pytest.raises(bi.BiError, match="BAD_INPUT"):
        bi.get_device_error()
    assert torch.isnan(lp[1]) and not torch.isnan(lp[0])


def test_masked_vocabulary_entries():
    """-inf logits (a masked vocabulary) contribute nothing: rows with 90% of
    entries masked, a row with one visible entry (lse = that entry, its
    log-probability 0, up to fp32 rounding), and a row masked except its last
    vector."""
    x = inputs.normal_bf16((6, V), seed=94, std=3.0)
    g = torch.Generator().manual_seed(95)
    mask = torch.rand((6, V), generator=g) < 0.9
    x[mask] = float("-inf")
    x[3] = float("-inf")
    x[3, 77777] = 1.5
    x[4, :V - 8] = float("-inf")
    x[5, :1000] = float("-inf")
    t = torch.tensor([int(torch.nonzero(~mask[0])[0]), int(torch.nonzero(~mask[1])[0]),
                      int(torch.nonzero(~mask[2])[0]), 77777, V - 3,
                      1000 + int(torch.nonzero(~mask[5, 1000:])[0])], dtype=torch.int32)
    xd, td = x.cuda(), t.cuda()
    lp, lse = bi.logprobs(xd, td)
    lp_ref, lse_ref = oracle.logprobs(x, t.numpy())
    for got, ref in ((lp, lp_ref), (lse, lse_ref)):
        g_ = got.cpu().double().numpy()
        assert np.isfinite(g_).all()
        assert (np.abs(g_ - ref) <= 1e-4 + 1e-6 * np.abs(ref)).all(), np.abs(g_ - ref).max()
    assert abs(lse[3].item() - 1.5) <= 1e-6 and abs(lp[3].item()) <= 1e-6
    bi.get_device_error()


def test_terms_below_the_fp32_normal_range():
    """Each term is one ex2.approx.ftz, which flushes results below 2^-126 to
    zero.  Rows built so that many terms land there -- every other entry
    about 100 below the row's maximum (terms near e^-100 = 2^-144), with the
    maximum first, last, or alone among -inf entries -- must still give the
    oracle's lse and log-probabilities: a flushed term is far below half an
    ulp of the sum, which holds the maximum's own term (about 1)."""
    rows = torch.full((4, V), -100.0)
    rows[0, 0] = 0.0                       # maximum in the first vector
    rows[1, V - 1] = 0.0                   # maximum in the last vector, after every tiny term
    rows[2, 4000:4008] = torch.tensor([-100.0, -99.0, 0.0, -101.0, -98.5, -100.0, -30.0, -97.0])
    rows[3] = float("-inf")
    rows[3, 77] = 5.0
    rows[3, 78] = -95.0                    # one tiny term beside the maximum
    x = rows.to(torch.bfloat16)
    t = torch.tensor([0, 5, 4006, 78], dtype=torch.int32)
    lp, lse = bi.logprobs(x.cuda(), t.cuda())
    lp_ref, lse_ref = oracle.logprobs(x, t.numpy())
    for got, ref in ((lp, lp_ref), (lse, lse_ref)):
        g = got.cpu().double().numpy()
        assert (np.abs(g - ref) <= 1e-4 + 1e-6 * np.abs(ref)).all(), (g, ref)
    bi.get_device_error()
