"""The random-init Qwen3-8B-shaped decoder on the batch-invariant kernels.

1. Parity: a 2-layer truncation of the model (full Qwen3-8B widths, vocab
   151936), teacher-forced, against the fp64 oracle decoder -- logits within
   1e-2 * max|ref| at every generated position.
2. Batch invariance end to end: sequences served in a continuously batched
   run (changing partners, prompts split across steps by a small token budget)
   produce bit-identical logits at every step to the same sequences run alone.
"""
import numpy as np
import pytest
import torch

from invariant_bi_rmsnorm_gb300 import qwen3
from oracle import decoder as odec
from tests._util import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def two_layer():
    cfg = qwen3.Qwen3Config(layers=2, max_pos=1024)
    w = qwen3.Qwen3Weights(cfg, seed=2000)
    return cfg, w


def test_two_layer_logits_match_oracle(two_layer):
    cfg, w = two_layer
    eng = qwen3.Engine(w, num_pages=64, max_tokens_per_step=512)
    g = torch.Generator().manual_seed(5)
    seqs = []
    for i, L in enumerate((12, 20, 7)):
        prompt = torch.randint(0, cfg.vocab, (L,), generator=g).tolist()
        forced = torch.randint(0, cfg.vocab, (4,), generator=g).tolist()
        seqs.append(qwen3.Sequence(sid=i, prompt=prompt, max_new=4, forced=forced))
    logs = eng.generate(seqs, record={0, 1, 2})
    host = w.host_bits(2)
    for s in seqs:
        toks = np.array(s.prompt + s.forced[:3])
        L = len(s.prompt)
        ref = odec.forward_logits(host, toks, 2, positions=[L - 1, L, L + 1, L + 2])
        got = torch.stack(logs[s.sid]).double().numpy()
        err = np.abs(got - ref)
        assert err.max() <= 1e-2 * np.abs(ref).max(), (s.sid, err.max(), np.abs(ref).max())


def test_logits_bit_identical_alone_and_batched(two_layer):
    cfg, w = two_layer
    reqs = qwen3.random_requests(24, cfg.vocab, 32, 160, max_new=6, seed=11)
    track = {0, 5, 13, 23}
    eng = qwen3.Engine(w, num_pages=24 * 12, max_tokens_per_step=300)
    batched = eng.generate(reqs, record=track)
    batched_lp = dict(eng.logprobs)
    assert eng.steps > 10  # prompts were split and mixed over many steps
    for sid in sorted(track):
        r = reqs[sid]
        eng.reset()
        alone_req = qwen3.Sequence(sid=sid, prompt=list(r.prompt), max_new=6)
        lp_batched = list(batched_lp[sid])
        alone = eng.generate([alone_req], record={sid})
        assert alone_req.generated == r.generated, f"sequence {sid}: tokens differ"
        for step, (a, b) in enumerate(zip(alone[sid], batched[sid])):
            assert np.array_equal(bits(a), bits(b)), f"sequence {sid}: logits differ at step {step}"
        # the sampler's log-probabilities of its own tokens agree bit for bit too
        assert all(torch.equal(a, b) for a, b in zip(eng.logprobs[sid], lp_batched))


def test_cuda_graph_decode_steps_bit_identical(two_layer):
    """Decode-only steps replayed from captured CUDA graphs (padded to their
    batch bucket with rows on a reserved page) give the same tokens and the
    same logit bits as eager launches, across changing batch sizes."""
    cfg, w = two_layer
    track = set(range(10))
    runs = []
    for graphs in (False, True):
        reqs = qwen3.random_requests(10, cfg.vocab, 16, 64, max_new=8, seed=21)
        eng = qwen3.Engine(w, num_pages=10 * 6 + 1, max_tokens_per_step=96, cuda_graphs=graphs)
        logs = eng.generate(reqs, record=track)
        runs.append((reqs, logs, eng.graph_steps, len(eng._graphs)))
    (r0, l0, g0, _), (r1, l1, g1, nb) = runs
    assert g0 == 0 and g1 > 0 and nb >= 2  # several buckets were captured and replayed
    for sid in sorted(track):
        assert r0[sid].generated == r1[sid].generated, f"sequence {sid}: tokens differ"
        for step, (a, b) in enumerate(zip(l0[sid], l1[sid])):
            assert np.array_equal(bits(a), bits(b)), f"sequence {sid}: logits differ at step {step}"


def test_tiny_requests_and_staggered_finishes(two_layer):
    """One-token prompts, one-token generations and requests finishing at
    different steps, with a budget that splits the longest prompt: the same
    tokens and logits alone as batched, eager and graphed."""
    cfg, w = two_layer
    g = torch.Generator().manual_seed(77)
    spec = [(1, 1), (1, 5), (2, 3), (40, 2), (130, 4)]   # (prompt length, new tokens)

    def make():
        out = []
        for i, (L, n) in enumerate(spec):
            prompt = torch.randint(0, cfg.vocab, (L,), generator=torch.Generator().manual_seed(500 + i)).tolist()
            out.append(qwen3.Sequence(sid=i, prompt=prompt, max_new=n))
        return out
    results = []
    for graphs in (False, True):
        eng = qwen3.Engine(w, num_pages=40, max_tokens_per_step=64, cuda_graphs=graphs)
        reqs = make()
        logs = eng.generate(reqs, record=set(range(len(spec))))
        assert all(len(r.generated) == n for r, (_, n) in zip(reqs, spec))
        results.append((reqs, logs))
        for i in (0, 4):
            eng.reset()
            one = make()[i]
            alone = eng.generate([one], record={i})
            assert one.generated == reqs[i].generated
            assert all(np.array_equal(bits(a), bits(b)) for a, b in zip(alone[i], logs[i]))
    (r0, l0), (r1, l1) = results
    for i in range(len(spec)):
        assert r0[i].generated == r1[i].generated
        assert all(np.array_equal(bits(a), bits(b)) for a, b in zip(l0[i], l1[i]))
