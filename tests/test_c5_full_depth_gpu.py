"""The random-init Qwen3-8B-shaped decoder at its full depth (36 layers,
hidden 4096, FFN 12288, 32/8 heads of 128, vocab 151936, RoPE theta 1e6),
served with continuous batching: requests' logits are bit-identical whether
they run in the batch or alone -- the end-to-end property of "Defeating
Nondeterminism in LLM Inference: The Core Role of Batch Invariance"
("Experimental Validation and Future Prospects"), here on random weights.

64 requests with prompts of U[32, 512] random tokens generate 8 greedy tokens
each under an 8192-token step budget (prompts split across steps and mixed
with decode rows).  Four tracked requests are re-run alone; their tokens and
every logit row must match the batched run bit for bit, with eager launches
and with CUDA-graph decode steps.  The same engine with torch/cuBLAS GEMMs and
torch RMSNorms (the non-invariant comparison) must show differing rows: the
check has teeth.

Parity against the fp64 oracle is pinned on a 2-layer truncation
(tests/test_qwen3_gpu.py); at 36 layers the pin is the bitwise property.
"""
import numpy as np
import pytest
import torch

from invariant_bi_rmsnorm_gb300 import qwen3
from tests._util import bits

pytestmark = pytest.mark.gpu

N_REQ, NEW, BUDGET = 64, 8, 8192
TRACK = (0, 21, 42, 63)


@pytest.fixture(scope="module")
def model():
    cfg = qwen3.Qwen3Config()
    assert cfg.layers == 36
    w = qwen3.Qwen3Weights(cfg, seed=1000)
    yield w
    del w
    torch.cuda.empty_cache()


def _requests(cfg):
    return qwen3.random_requests(N_REQ, cfg.vocab, 32, 512, NEW, seed=7)


def _serve(w, ops, graphs):
    """Batched run of every request, then each tracked request alone."""
    reqs = _requests(w.cfg)
    pages = sum(-(-(len(r.prompt) + NEW) // 16) for r in reqs) + 64
    eng = qwen3.Engine(w, num_pages=pages, max_tokens_per_step=BUDGET, ops=ops, cuda_graphs=graphs)
    logs = eng.generate(reqs, record=set(TRACK))
    info = {"steps": eng.steps, "graph_steps": eng.graph_steps}
    alone = {}
    for sid in TRACK:
        eng.reset()
        one = qwen3.Sequence(sid=sid, prompt=list(reqs[sid].prompt), max_new=NEW)
        rows = eng.generate([one], record={sid})[sid]
        alone[sid] = (one.generated, rows)
    del eng
    torch.cuda.empty_cache()
    return reqs, logs, alone, info


def test_36_layers_bitwise_alone_vs_batched_eager_and_graphed(model):
    runs = {}
    for graphs in (False, True):
        reqs, logs, alone, info = _serve(model, "bi", graphs)
        assert info["steps"] > NEW  # prompts were spread over several steps
        assert (info["graph_steps"] > 0) == graphs
        for sid in TRACK:
            toks, rows = alone[sid]
            assert toks == reqs[sid].generated, f"graphs={graphs} request {sid}: tokens differ"
            assert len(rows) == NEW == len(logs[sid])
            for step, (a, b) in enumerate(zip(rows, logs[sid])):
                assert np.array_equal(bits(a), bits(b)), \
                    f"graphs={graphs} request {sid}: logits differ at step {step}"
        runs[graphs] = (reqs, logs)
    # eager and graphed batched runs agree too
    (r0, l0), (r1, l1) = runs[False], runs[True]
    for sid in TRACK:
        assert r0[sid].generated == r1[sid].generated
        assert all(np.array_equal(bits(a), bits(b)) for a, b in zip(l0[sid], l1[sid]))


def test_36_layers_torch_ops_control_differs(model):
    reqs, logs, alone, _ = _serve(model, "torch", False)
    differing = sum(int(not np.array_equal(bits(a), bits(b)))
                    for sid in TRACK for a, b in zip(alone[sid][1], logs[sid]))
    assert differing > 0, "cuBLAS / F.rms_norm gave identical rows: the control has no teeth"
