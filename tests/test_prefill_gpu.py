"""bi_prefill_attention on the GPU.

A prefilled token must get the same bits as the same token computed by
bi_decode_attention, and the same bits whatever chunking of the prompt
produced it -- the prefill / chunked-prefill invariance "3. Batch-Invariant
Attention" asks for.  Parity is checked against the fp64 oracle, with each
query row expanded into a decode row of its own causal length.
"""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import inputs
from tests._util import bits, f64

pytestmark = pytest.mark.gpu


def _check(out, ref):
    got = f64(out)
    err = np.abs(got - ref)
    assert err.max() <= 1e-2 * np.abs(ref).max()
    row_tol = 2.0 ** -6 * np.abs(ref).max(axis=-1) + 2.0 ** -12
    assert (err.max(axis=-1) <= row_tol).all()


def _prompts(lens, Hq=32, Hkv=8, seed=400, spare=3):
    """Sequences of the given lengths with their K/V in the cache, plus one
    query per prompt token."""
    p = inputs.decode_problem(len(lens), Hq=Hq, Hkv=Hkv, seq_lens=lens, seed=seed,
                              spare_pages=spare)
    T = sum(lens)
    q = inputs.decode_queries(T, Hq, 128, seed=seed + 50)
    return p, q


def _expanded(p, q, rows_of):
    """Decode-shaped problem with one row per query: (block-table row, length)."""
    seq_idx = torch.tensor([i for i, _ in rows_of], dtype=torch.long)
    lens = torch.tensor([L for _, L in rows_of], dtype=torch.int32)
    return {"q": q, "k_cache": p["k_cache"], "v_cache": p["v_cache"],
            "block_table": p["block_table"][seq_idx].contiguous(), "seq_lens": lens}


def _prefill(p, q, nq, lens=None, max_seq_len=None):
    lens = p["seq_lens"] if lens is None else torch.as_tensor(lens, dtype=torch.int32)
    indptr = torch.zeros(len(nq) + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(torch.as_tensor(nq, dtype=torch.int32), 0)
    return bi.prefill_attention(q.cuda(), p["k_cache"].cuda(), p["v_cache"].cuda(),
                                p["block_table"].cuda(), lens.cuda(), indptr.cuda(),
                                max_q_len=int(max(nq)), max_seq_len=int(max_seq_len or lens.max()))


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 8), (24, 8), (40, 8), (64, 8)])
def test_full_prompt_matches_oracle_and_decode_bitwise(Hq, Hkv):
    lens = [1, 37, 300, 700]
    p, q = _prompts(lens, Hq=Hq, Hkv=Hkv, seed=400 + Hq)
    out = _prefill(p, q, lens)
    rows = [(i, r + 1) for i, L in enumerate(lens) for r in range(L)]
    e = _expanded(p, q, rows)
    dec = bi.decode_attention(e["q"].cuda(), e["k_cache"].cuda(), e["v_cache"].cuda(),
                              e["block_table"].cuda(), e["seq_lens"].cuda(), max_seq_len=max(lens))
    ob, db = bits(out), bits(dec)
    same = (ob == db).all(axis=(1, 2))
    assert same.all(), f"{(~same).sum()} of {len(rows)} rows differ from decode; first {np.argmin(same)}"
    _check(out, oracle.decode_attention(**e))


def test_long_prompts_many_chunks_match_decode_bitwise():
    # 2100 and 4100 tokens: 9 and 17 chunks, so every row past the first 256
    # folds several chunk partials, and tile pairs of every length run
    lens = [2100, 4100]
    p, q = _prompts(lens, seed=410)
    out = _prefill(p, q, lens)
    rows = [(i, r + 1) for i, L in enumerate(lens) for r in range(L)]
    e = _expanded(p, q, rows)
    dec = bi.decode_attention(e["q"].cuda(), e["k_cache"].cuda(), e["v_cache"].cuda(),
                              e["block_table"].cuda(), e["seq_lens"].cuda(), max_seq_len=max(lens))
    same = (bits(out) == bits(dec)).all(axis=(1, 2))
    assert same.all(), f"{(~same).sum()} of {len(rows)} rows differ from decode; first {np.argmin(same)}"
    pick = np.r_[0:40, 250:270, 2090:2110, 4000:4040, 6160:6200]
    sub = _expanded(p, q[torch.from_numpy(pick)], [rows[i] for i in pick])
    _check(out[torch.from_numpy(pick).cuda()], oracle.decode_attention(**sub))


def test_chunked_prefill_matches_whole_prompt_bitwise():
    L = 900
    p, q = _prompts([L], seed=420)
    whole = bits(_prefill(p, q, [L]))
    for cuts in ([0, 100, 250, 900], [0, 1, 2, 511, 512, 513, 900], [0, 256, 512, 768, 900]):
        got = np.empty_like(whole)
        for a, b in zip(cuts[:-1], cuts[1:]):
            # the cache holds tokens < b when rows [a, b) are computed
            out = _prefill(p, q[a:b].contiguous(), [b - a], lens=[b], max_seq_len=L)
            got[a:b] = bits(out)
        assert np.array_equal(got, whole), f"chunking {cuts} changed bits"


def test_mixed_batch_rows_equal_individual_calls():
    # a decode row (n = 1) next to prompts of several lengths, in one launch
    lens = [513, 40, 1000, 7]
    nq = [1, 40, 300, 7]  # sequence 2 has its first 700 tokens cached already
    p, _ = _prompts(lens, seed=430)
    q = inputs.decode_queries(sum(nq), 32, 128, seed=431)
    batched = bits(_prefill(p, q, nq))
    off = 0
    for i, n in enumerate(nq):
        one = {k: (v[i:i + 1] if k in ("block_table",) else v) for k, v in p.items()}
        alone = bits(_prefill(one, q[off:off + n].contiguous(), [n], lens=[lens[i]]))
        assert np.array_equal(alone, batched[off:off + n]), f"sequence {i} differs"
        off += n
    rows = [(i, lens[i] - n + 1 + r) for i, n in enumerate(nq) for r in range(n)]
    _check(torch.from_numpy(batched.view(np.int16)).view(torch.bfloat16),
           oracle.decode_attention(**_expanded(p, q, rows)))


def test_garbage_past_the_last_query_token_is_ignored():
    lens = [45]
    p, q = _prompts(lens, seed=440, spare=0)
    clean = bits(_prefill(p, q, lens))
    pg = int(p["block_table"][0, 2])  # tokens 32..47: 45..47 are past the sequence
    p["k_cache"][pg, :, 13:] = float("nan")
    p["v_cache"][pg, :, 13:] = float("inf")
    assert np.array_equal(bits(_prefill(p, q, lens)), clean)


def test_inconsistent_indptr_reported_without_fault():
    p, q = _prompts([20, 30], seed=450)
    d = {k: v.cuda() for k, v in p.items()}
    bi.get_device_error()
    # sequence 1 claims 40 query rows but has 30 tokens (and q has only 50 rows)
    indptr = torch.tensor([0, 20, 60], dtype=torch.int32, device="cuda")
    bi.prefill_attention(q.cuda(), d["k_cache"], d["v_cache"], d["block_table"], d["seq_lens"],
                         indptr, max_q_len=30, max_seq_len=30)
    with pytest.raises(bi.BiError, match="BAD_INPUT"):
        bi.get_device_error()
    bi.get_device_error()


def test_page_outside_the_cache_reported_and_only_its_readers_skipped():
    # a 100-token prompt in tiles of 32 rows: rows 0-31 read pages 0-1,
    # rows 96-99 read pages 0-6.  Page 6 (tokens 96-99) points past the
    # cache: the tile that reads it is reported and not written (its loads
    # read zeros there, no fault); every other tile keeps its clean bits.
    lens = [100]
    p, q = _prompts(lens, seed=460)
    clean = bits(_prefill(p, q, lens))
    bad = {k: v.clone() for k, v in p.items()}
    bad["block_table"][0, 6] = int(p["k_cache"].shape[0]) + 5
    bi.get_device_error()
    sentinel = torch.full((100, 32, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    d = {k: v.cuda() for k, v in bad.items()}
    indptr = torch.tensor([0, 100], dtype=torch.int32, device="cuda")
    out = bi.prefill_attention(q.cuda(), d["k_cache"], d["v_cache"], d["block_table"],
                               d["seq_lens"], indptr, max_q_len=100, max_seq_len=100,
                               out=sentinel)
    with pytest.raises(bi.BiError, match="BAD_INPUT"):
        bi.get_device_error()
    bi.get_device_error()
    got = bits(out)
    assert np.array_equal(got[:96], clean[:96])
    assert (got[96:] == bits(torch.full((4, 32, 128), 7.0, dtype=torch.bfloat16))).all()


def test_bench_workload_every_row_equals_decode():
    # the launch the bench times: 29 prompts of U[32, 512] tokens (8048 rows,
    # 3712 CTAs, most tile classes and the empty ones); every row against
    # decode bit for bit, a sample against the oracle
    lens_all = inputs.seq_lens_uniform(64, 512, seed=610, min_len=32).tolist()
    lens, tot = [], 0
    for L in lens_all:
        if tot + L > 8192:
            break
        lens.append(L)
        tot += L
    p = inputs.decode_problem(len(lens), Hq=32, Hkv=8, D=128, seq_lens=lens, seed=611)
    q = inputs.normal_bf16((tot, 32, 128), 612)
    out = _prefill(p, q, lens)
    rows = [(i, r + 1) for i, L in enumerate(lens) for r in range(L)]
    e = _expanded(p, q, rows)
    dec = bi.decode_attention(e["q"].cuda(), e["k_cache"].cuda(), e["v_cache"].cuda(),
                              e["block_table"].cuda(), e["seq_lens"].cuda(), max_seq_len=max(lens))
    same = (bits(out) == bits(dec)).all(axis=(1, 2))
    assert same.all(), f"{(~same).sum()} of {len(rows)} rows differ from decode; first {np.argmin(same)}"
    pick = np.unique(np.r_[0:8, np.linspace(0, tot - 1, 56).astype(int)])
    sub = _expanded(p, q[torch.from_numpy(pick)], [rows[i] for i in pick])
    _check(out[torch.from_numpy(pick).cuda()], oracle.decode_attention(**sub))


@pytest.mark.parametrize("kind", ["flat", "peaked", "ramp"])
def test_adversarial_scores_match_decode_bitwise(kind):
    # flat: q = 0, every score equal; peaked: q x 40, a nearly one-hot
    # softmax; ramp: page j of each prompt holds K x (1 + j), so the scores
    # grow along the prompt and the reference maximum keeps moving past its
    # slack -- the path that rescales O in TMEM, which seeded N(0, 1) data
    # almost never takes
    lens = [300, 700]
    p, q = _prompts(lens, seed=470)
    if kind == "flat":
        q = torch.zeros_like(q)
    elif kind == "peaked":
        q = (q.float() * 40.0).to(torch.bfloat16)
    else:
        for s, L in enumerate(lens):
            for j in range((L + 15) // 16):
                pg = int(p["block_table"][s, j])
                p["k_cache"][pg] = (p["k_cache"][pg].float() * (1.0 + j)).to(torch.bfloat16)
    out = _prefill(p, q, lens)
    rows = [(i, r + 1) for i, L in enumerate(lens) for r in range(L)]
    e = _expanded(p, q, rows)
    dec = bi.decode_attention(e["q"].cuda(), e["k_cache"].cuda(), e["v_cache"].cuda(),
                              e["block_table"].cuda(), e["seq_lens"].cuda(), max_seq_len=max(lens))
    same = (bits(out) == bits(dec)).all(axis=(1, 2))
    assert same.all(), f"{(~same).sum()} of {len(rows)} rows differ from decode; first {np.argmin(same)}"
    _check(out, oracle.decode_attention(**e))
