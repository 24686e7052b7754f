"""bi_decode_attention on the GPU: parity with the fp64 oracle and bitwise
invariance to batch composition, position and KV-cache growth.

Tolerances: the stated one, max|gpu - ref| <= 1e-2 * max|ref| per call, and a
tighter per-row one, max over d of |gpu - ref| <= 2^-6 * max_d |ref| + 2^-12,
derived from the arithmetic (bf16-rounded softmax weights, relative error
2^-9 each, averaged over the row; one bf16 rounding of the output).  A
dropped, repeated or mis-masked token moves a short row far beyond it.

Workload (GQA 32 query / 8 kv heads, head_dim 128, bf16 cache, 16-token pages,
q/k/v ~ N(0, 1), lengths uniform on [1, 8192], pages scattered by a seeded
permutation).
"""
import math

import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import inputs
from tests._util import bits, f64

pytestmark = pytest.mark.gpu


def _to_dev(p):
    return {k: v.cuda() for k, v in p.items()}


def _run(p, max_seq_len=None, **kw):
    d = _to_dev(p)
    if max_seq_len is None:
        max_seq_len = int(p["seq_lens"].max())
    return bi.decode_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                               d["seq_lens"], max_seq_len=max_seq_len, **kw)


def _check(out, ref):
    got = f64(out)
    err = np.abs(got - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max(), f"call tolerance: {err.max()}"
    row_tol = 2.0 ** -6 * np.abs(ref).max(axis=-1) + 2.0 ** -12
    row_err = err.max(axis=-1)
    bad = row_err > row_tol
    assert not bad.any(), f"{bad.sum()} rows beyond tolerance, first {np.argwhere(bad)[0]}"


def _host_subset(p, pick):
    """Sequences `pick` of a problem, with only their pages copied to the host."""
    bt = p["block_table"][pick].cpu()
    used = bt[bt >= 0].unique()
    remap = torch.full((p["k_cache"].shape[0],), -1, dtype=torch.int32)
    remap[used.long()] = torch.arange(used.numel(), dtype=torch.int32)
    nbt = torch.where(bt >= 0, remap[bt.clamp(min=0).long()], bt).contiguous()
    idx = used.long().to(p["k_cache"].device)
    return {"q": p["q"][pick].cpu(), "k_cache": p["k_cache"][idx].cpu(),
            "v_cache": p["v_cache"][idx].cpu(), "block_table": nbt,
            "seq_lens": p["seq_lens"][pick].cpu()}


EDGE_LENS = [1, 2, 15, 16, 17, 31, 255, 256, 257, 511, 512, 513, 1000, 4097, 8192]


def test_edge_lengths_against_oracle():
    p = inputs.decode_problem(len(EDGE_LENS), seq_lens=EDGE_LENS, seed=200, spare_pages=7)
    _check(_run(p), oracle.decode_attention(**p))


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 8), (24, 8), (16, 4), (32, 8), (40, 8),
                                    (48, 8), (56, 8), (64, 8)])
def test_gqa_group_sizes(Hq, Hkv):
    # group sizes 1 .. 8; the 3000- and 9000-token sequences span several
    # CTAs, so the last-arriving CTA folds them (9000 tokens: 36 chunks, more
    # than one scan block or staging batch for every group size)
    lens = [3, 300, 1000, 3000, 9000]
    p = inputs.decode_problem(len(lens), Hq=Hq, Hkv=Hkv, seq_lens=lens, seed=210 + Hq)
    _check(_run(p), oracle.decode_attention(**p))


@pytest.mark.parametrize("G", [1, 2, 3, 5, 8])
def test_last_cta_fold_equals_in_cta_fold_for_every_group_size(G):
    # In a batch of 256 each sequence (up to 32 chunks) is walked and folded
    # by one CTA; alone it runs on the small-batch kernel (each chunk's pages
    # shared by a score warp and an update warp), spread over up to 16 CTAs
    # and folded by the last to arrive.  Same operations in the same order:
    # same bits.
    B, Hkv = 256, 8
    p = inputs.decode_problem(B, Hq=G * Hkv, Hkv=Hkv, max_len=8192, seed=400 + G, device="cuda")
    lib = bi._lib.load()
    full = bits(_run(p, max_seq_len=8192))
    lens = p["seq_lens"]
    pick = [int(i) for i in torch.argsort(lens, descending=True)[:3]] + [int(torch.argmin(lens))]
    for s in pick:
        one = {k: (v[s:s + 1] if k in ("q", "block_table", "seq_lens") else v) for k, v in p.items()}
        assert np.array_equal(bits(_run(one, max_seq_len=8192))[0], full[s]), f"sequence {s}"
    assert lib.bi_decode_attention_launches(1, Hkv, 8192) == 1
    sub = _host_subset(p, np.array(pick))
    rows = torch.from_numpy(full[pick].view(np.int16)).view(torch.bfloat16)
    _check(rows, oracle.decode_attention(**sub))


@pytest.mark.parametrize("G", [4, 7])
def test_small_batch_kernel_equals_split_kernel(G):
    # One or two sequences take the small-batch kernel (a warp pair per
    # chunk); the same sequences inside a batch of 64 take the split kernel
    # (a warp per chunk).  Lengths of one chunk, of two chunks (one CTA, both
    # pairs), and of many chunks (several CTAs and the last-CTA fold).
    Hkv = 8
    g = torch.Generator().manual_seed(G)
    lens = [100, 300, 5000, 8192] + torch.randint(1, 8193, (60,), generator=g).tolist()
    p = inputs.decode_problem(len(lens), Hq=G * Hkv, Hkv=Hkv, seq_lens=lens, seed=450 + G,
                              spare_pages=3)
    full = bits(_run(p, max_seq_len=8192))
    for idx in ([0], [1], [2], [3], [1, 2]):
        sel = torch.tensor(idx)
        few = {k: (v[sel].contiguous() if k in ("q", "block_table", "seq_lens") else v)
               for k, v in p.items()}
        got = bits(_run(few, max_seq_len=8192))
        assert np.array_equal(got, full[idx]), f"sequences {idx}"
    bi.get_device_error()


def test_custom_scale():
    p = inputs.decode_problem(4, seq_lens=[5, 70, 600, 2000], seed=220)
    _check(_run(p, scale=0.03), oracle.decode_attention(**p, scale=0.03))


def test_garbage_past_sequence_end_is_ignored():
    # tokens past seq_len inside the last page hold NaN/inf: never read into
    # the result (masked scores, zeroed V rows)
    lens = [1, 17, 250, 1000]
    p = inputs.decode_problem(4, seq_lens=lens, seed=230)
    ref = oracle.decode_attention(**p)
    clean = bits(_run(p))
    bt = p["block_table"]
    for s, L in enumerate(lens):
        last = int(bt[s, (L - 1) // 16])
        if L % 16:
            p["k_cache"][last, :, L % 16:] = float("nan")
            p["v_cache"][last, :, L % 16:] = float("inf")
    dirty = _run(p)
    assert np.array_equal(bits(dirty), clean)
    _check(dirty, ref)


def test_single_sequence_bit_identical_in_any_batch():
    B = 128
    p = inputs.decode_problem(B, max_len=8192, seed=240)
    full = bits(_run(p, max_seq_len=8192))  # block tables have room for 8192
    for s in (0, 5, 77, 127):
        one = {k: (v[s:s + 1] if k in ("q", "block_table", "seq_lens") else v) for k, v in p.items()}
        alone = bits(_run(one, max_seq_len=8192))
        assert np.array_equal(alone[0], full[s]), f"sequence {s} alone differs from batched"
        # a launch sized for a smaller bound (fewer grid chunks) gives the same bits
        alone2 = bits(_run(one))
        assert np.array_equal(alone2[0], full[s])
    # permutation of the batch
    perm = torch.randperm(B, generator=torch.Generator().manual_seed(5))
    pp = dict(p)
    for k in ("q", "block_table", "seq_lens"):
        pp[k] = p[k][perm].contiguous()
    assert np.array_equal(bits(_run(pp, max_seq_len=8192)), full[perm.numpy()])


def test_growth_from_100_to_1000_tokens():
    # One sequence grows from 100 to 1000 tokens: before each call the caller
    # appends the new tokens' K/V into their page slots, and the batch
    # partners change every step.  The outputs for two fixed queries taken at
    # L = 100 and L = 512 are recorded when first computed, then recomputed
    # once the cache holds all 1000 tokens (seq_len set back): same bits.
    Hq, D = 32, 128
    g = torch.Generator().manual_seed(250)
    grown = inputs.decode_problem(1, seq_lens=[1000], seed=251)
    partners = inputs.decode_problem(64, max_len=2000, seed=252)
    num_pages_a = grown["k_cache"].shape[0]
    k_true = torch.cat([grown["k_cache"], partners["k_cache"]])
    v_true = torch.cat([grown["v_cache"], partners["v_cache"]])
    pbt = partners["block_table"].clone()
    pbt[pbt >= 0] += num_pages_a
    width = 125  # room for 2000 tokens
    gbt = grown["block_table"][0]

    def table(rows):
        t = torch.full((len(rows), width), -1, dtype=torch.int32)
        for i, r in enumerate(rows):
            t[i, :r.shape[0]] = r
        return t

    kd, vd = k_true.cuda(), v_true.cuda()
    kd[:num_pages_a] = 0  # the growing sequence's pages start empty
    vd[:num_pages_a] = 0

    def append(t0, t1):  # write tokens [t0, t1) of the growing sequence
        for t in range(t0, t1):
            pg, slot = int(gbt[t // 16]), t % 16
            kd[pg, :, slot] = k_true[pg, :, slot].cuda()
            vd[pg, :, slot] = v_true[pg, :, slot].cuda()

    q_fixed = {L: inputs.decode_queries(1, Hq, D, seed=1000 + L)[0] for L in (100, 512)}
    recorded = {}
    have = 0
    for L in list(range(100, 1001, 4)):
        append(have, L)
        have = L
        nb = int(torch.randint(0, 9, (1,), generator=g))
        pick = torch.randperm(64, generator=g)[:nb].tolist()
        pos = int(torch.randint(0, nb + 1, (1,), generator=g))
        rows = [pbt[i] for i in pick]
        lens = [int(partners["seq_lens"][i]) for i in pick]
        qs = [partners["q"][i] for i in pick]
        rows.insert(pos, gbt)
        lens.insert(pos, L)
        qs.insert(pos, q_fixed.get(L, inputs.decode_queries(1, Hq, D, seed=2000 + L)[0]))
        out = bi.decode_attention(torch.stack(qs).cuda(), kd, vd, table(rows).cuda(),
                                  torch.tensor(lens, dtype=torch.int32).cuda(), max_seq_len=2000)
        if L in q_fixed:
            recorded[L] = bits(out[pos])
    assert have == 1000
    for L, want in recorded.items():
        out = bi.decode_attention(q_fixed[L][None].cuda(), kd, vd, table([gbt]).cuda(),
                                  torch.tensor([L], dtype=torch.int32).cuda(), max_seq_len=1000)
        assert np.array_equal(bits(out[0]), want), f"output at L={L} changed after growth"
        one = {"q": q_fixed[L][None], "k_cache": k_true, "v_cache": v_true,
               "block_table": table([gbt]), "seq_lens": torch.tensor([L], dtype=torch.int32)}
        _check(out, oracle.decode_attention(**one))


def test_complete_chunk_partials_stable_as_cache_grows():
    # the workspace holds each chunk's (m, l, O) partial; a complete chunk's
    # partial must not change when the sequence grows past it
    Hq, D = 32, 128
    base = inputs.decode_problem(1, seq_lens=[2048], seed=260)
    max_chunks = 8
    ws = torch.zeros(bi.decode_attention_workspace_size(1, Hq, D, 2048), dtype=torch.uint8,
                     device="cuda")
    acc_elems = 1 * Hq * max_chunks * D

    def partial_acc(L):
        p = dict(base)
        p["seq_lens"] = torch.tensor([L], dtype=torch.int32)
        ws.zero_()
        _run(p, max_seq_len=2048, workspace=ws)
        f = ws[bi.DECODE_COUNTER_BYTES:].view(torch.float32)  # after the arrival counters
        return (f[:acc_elems].view(Hq, max_chunks, D).cpu().numpy().copy(),
                f[acc_elems:].view(Hq, max_chunks, 2).cpu().numpy().copy())

    # (a sequence whose chunks all fall to one CTA is folded there and writes
    # no partials; with one sequence a CTA walks at most 4 chunks, so both
    # lengths here leave their partials in the workspace)
    a1, m1 = partial_acc(1100)  # chunks 0..3 complete; chunk 4 partial
    a2, m2 = partial_acc(2048)  # all 8 complete
    assert np.isfinite(a1[:, :5]).all() and (m1[:, :5, 1] > 0).all(), "partials not written"
    assert np.array_equal(a1[:, :4].view(np.uint32), a2[:, :4].view(np.uint32))
    assert np.array_equal(m1[:, :4].view(np.uint32), m2[:, :4].view(np.uint32))
    # and they agree with the oracle's fp64 chunk partials: m is kept in log2
    # units, so l and O are scaled by 2^(m) / e^(m_oracle)
    _, part = oracle.decode_attention_chunked(**base, chunk=256, max_chunks=max_chunks,
                                              want_partials=True)
    for c in range(8):
        mo, lo, ao = part[0, :, c, 0], part[0, :, c, 1], part[0, :, c, 2:]
        factor = np.exp(mo - m2[:, c, 0].astype(np.float64) * math.log(2.0))
        np.testing.assert_allclose(m2[:, c, 1], lo * factor, rtol=2 ** -7)
        o_gpu = a2[:, c] / m2[:, c, 1:2]
        o_ref = ao / lo[:, None]
        assert (np.abs(o_gpu - o_ref).max(axis=-1) <= 2 ** -6 * np.abs(o_ref).max(axis=-1) + 2 ** -12).all()


def test_c4_full_size_parity():
    # batch 1 .. 256, lengths U[1, 8192]: every row of every sequence against
    # the oracle (the multi-gigabyte caches are drawn on the device by torch's
    # seeded generator, then copied to the host for the oracle)
    for B in (1, 16, 128, 256):
        p = inputs.decode_problem(B, max_len=8192, seed=270 + B, device="cuda")
        out = _run(p, max_seq_len=8192)
        sub = _host_subset(p, np.arange(B))
        _check(out, oracle.decode_attention(**sub))
        del p, sub


def test_one_launch_folds_in_the_last_cta_and_leaves_counters_zero():
    # A sequence spread over several CTAs is folded by the last of them to
    # arrive, in the same launch: one kernel for every C4 batch.  The
    # workspace's arrival counters are back at zero after each call, so the
    # same workspace serves the next call (same bits), and the result matches
    # the oracle.
    lib = bi._lib.load()
    for B in (1, 16, 128, 256):
        assert lib.bi_decode_attention_launches(B, 8, 8192) == 1
    B = 16
    p = inputs.decode_problem(B, max_len=8192, seed=330)
    d = _to_dev(p)
    ws = torch.zeros(bi.decode_attention_workspace_size(B, 32, 128, 8192), dtype=torch.uint8,
                     device="cuda")
    counters = ws[:bi.DECODE_COUNTER_BYTES].view(torch.int32)
    outs = []
    for _ in range(3):
        outs.append(bits(bi.decode_attention(d["q"], d["k_cache"], d["v_cache"],
                                             d["block_table"], d["seq_lens"], max_seq_len=8192,
                                             workspace=ws)))
        assert int(counters.count_nonzero()) == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
    # the long sequences really were spread over several CTAs (partials written)
    assert int(ws[bi.DECODE_COUNTER_BYTES:].count_nonzero()) > 0
    pick = np.arange(0, B, 3)
    out = torch.from_numpy(outs[0][pick].view(np.int16)).view(torch.bfloat16)
    _check(out, oracle.decode_attention(**_host_subset(p, pick)))
    # a sequence alone (more CTAs per sequence) gives the batched bits
    for s in (0, 7):
        sl = slice(s, s + 1)
        alone = bits(bi.decode_attention(d["q"][sl], d["k_cache"], d["v_cache"],
                                         d["block_table"][sl], d["seq_lens"][sl],
                                         max_seq_len=8192, workspace=ws))
        assert np.array_equal(alone[0], outs[0][s])
        assert int(counters.count_nonzero()) == 0


def test_more_sequence_heads_than_counters_fall_back_to_the_merge_kernel():
    # 2049 sequences x 32 kv-heads is more (sequence, kv-head) pairs than the
    # workspace has arrival counters: sequences spread over several CTAs are
    # then folded by the separate merge kernel, with the same fold -- the bits
    # equal those of the same sequences run alone (one launch, counters).
    lib = bi._lib.load()
    B, Hq, Hkv, msl = 2049, 32, 32, 8448  # 33 chunks: more than one CTA walks
    assert B * Hkv > bi.DECODE_COUNTER_BYTES // 4
    assert lib.bi_decode_attention_launches(B, Hkv, msl) == 2
    assert lib.bi_decode_attention_launches(1, Hkv, msl) == 1
    special = {0: 8448, 1000: 5000, 2048: 300}
    base = inputs.decode_problem(3, Hq=Hq, Hkv=Hkv, seq_lens=list(special.values()), seed=340)
    width = msl // 16
    bt = torch.zeros(B, width, dtype=torch.int32)
    lens = torch.ones(B, dtype=torch.int32)
    bt[:] = base["block_table"][2, 0]  # length-1 rows read one page of the short sequence
    for j, (s, L) in enumerate(special.items()):
        n = -(-L // 16)
        bt[s, :n] = base["block_table"][j, :n]
        lens[s] = L
    q = inputs.decode_queries(B, Hq, 128, seed=341)
    kc, vc = base["k_cache"].cuda(), base["v_cache"].cuda()
    qd, btd, ld = q.cuda(), bt.cuda(), lens.cuda()
    big = bits(bi.decode_attention(qd, kc, vc, btd, ld, max_seq_len=msl))
    for j, s in enumerate(special):
        sl = slice(s, s + 1)
        alone = bi.decode_attention(qd[sl], kc, vc, btd[sl], ld[sl], max_seq_len=msl)
        assert np.array_equal(bits(alone)[0], big[s]), f"sequence {s}"
        one = {"q": q[sl], "k_cache": base["k_cache"], "v_cache": base["v_cache"],
               "block_table": bt[sl], "seq_lens": lens[sl]}
        _check(alone, oracle.decode_attention(**one))


def test_device_side_bad_inputs_reported_without_fault():
    p = inputs.decode_problem(3, seq_lens=[10, 20, 30], seed=280)
    d = _to_dev(p)
    bi.get_device_error()
    bad_lens = torch.tensor([10, 0, 30], dtype=torch.int32, device="cuda")
    bi.decode_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"], bad_lens, max_seq_len=30)
    with pytest.raises(bi.BiError, match="BAD_INPUT"):
        bi.get_device_error()
    bad_bt = d["block_table"].clone()
    bad_bt[2, 0] = 10 ** 6
    bi.decode_attention(d["q"], d["k_cache"], d["v_cache"], bad_bt, d["seq_lens"], max_seq_len=30)
    with pytest.raises(bi.BiError, match="BAD_INPUT"):
        bi.get_device_error()
    # a bad page in one CTA of a sequence spread over several CTAs: reported,
    # and the arrival counter still goes back to zero for the next call
    q = inputs.decode_problem(2, seq_lens=[3000, 2000], seed=281)
    dq = _to_dev(q)
    ws = torch.zeros(bi.decode_attention_workspace_size(2, 32, 128, 3000), dtype=torch.uint8,
                     device="cuda")
    bad_bt = dq["block_table"].clone()
    bad_bt[0, 100] = -5  # a page in chunk 6 (CTA 1 of 3)
    bi.decode_attention(dq["q"], dq["k_cache"], dq["v_cache"], bad_bt, dq["seq_lens"],
                        max_seq_len=3000, workspace=ws)
    with pytest.raises(bi.BiError, match="BAD_INPUT"):
        bi.get_device_error()
    assert int(ws[:bi.DECODE_COUNTER_BYTES].count_nonzero()) == 0
    good = bi.decode_attention(dq["q"], dq["k_cache"], dq["v_cache"], dq["block_table"],
                               dq["seq_lens"], max_seq_len=3000, workspace=ws)
    _check(good, oracle.decode_attention(**q))
    # the context is still usable and later calls are clean
    _check(_run(p), oracle.decode_attention(**p))
    bi.get_device_error()


def test_empty_batch_is_a_no_op():
    p = inputs.decode_problem(1, seq_lens=[5], seed=290)
    d = _to_dev(p)
    out = bi.decode_attention(d["q"][:0], d["k_cache"], d["v_cache"], d["block_table"][:0],
                              d["seq_lens"][:0], max_seq_len=5)
    assert out.shape == (0, 32, 128)


# ------------------------------------- fixed split COUNT: negative control ---
def _flashdecoding_splits(B, Hkv=8, sms=152):
    """A split count chosen to fill the GPU, as split-KV kernels commonly do:
    more splits when fewer sequences are in flight."""
    return max(1, min(32, -(-2 * sms // (B * Hkv))))


def test_fixed_split_count_matches_oracle():
    p = inputs.decode_problem(5, seq_lens=[1, 100, 1000, 3000, 8192], seed=310)
    d = _to_dev(p)
    ref = oracle.decode_attention(**p)
    for ns in (1, 3, 16):
        out = bi.decode_attention_fixed_splits(d["q"], d["k_cache"], d["v_cache"],
                                               d["block_table"], d["seq_lens"], max_seq_len=8192,
                                               num_splits=ns)
        _check(out, ref)


def test_fixed_split_count_breaks_invariance_where_fixed_size_does_not():
    # The same sequences run alone (B = 1) and in a batch of 128: with the
    # split count following the batch size the bits change; with the fixed
    # 256-token split size they never do.  The first half is the negative
    # control that shows the invariance checks can fail.
    B = 128
    p = inputs.decode_problem(B, max_len=8192, seed=320)
    d = _to_dev(p)
    ns_batch, ns_alone = _flashdecoding_splits(B), _flashdecoding_splits(1)
    assert ns_batch != ns_alone
    batched_fc = bits(bi.decode_attention_fixed_splits(
        d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"], 8192, ns_batch))
    batched_fs = bits(bi.decode_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                          d["seq_lens"], 8192))
    changed = 0
    for s in range(0, B, 8):
        sl = slice(s, s + 1)
        alone_fc = bits(bi.decode_attention_fixed_splits(
            d["q"][sl], d["k_cache"], d["v_cache"], d["block_table"][sl], d["seq_lens"][sl],
            8192, ns_alone))
        alone_fs = bits(bi.decode_attention(d["q"][sl], d["k_cache"], d["v_cache"],
                                            d["block_table"][sl], d["seq_lens"][sl], 8192))
        changed += int(not np.array_equal(alone_fc[0], batched_fc[s]))
        assert np.array_equal(alone_fs[0], batched_fs[s])
    assert changed > 0, "the fixed-count control never changed: the comparison would have no teeth"
