"""bi_decode_attention_noalloc: the attention entry point for callers that
cannot allocate device memory at call time (a plugin given only its input and
output buffers, a serving loop whose memory a caching allocator reserved up
front).  It keeps its arrival counters and chunk partials in a fixed scratch
array inside the library instead of a caller workspace.

This file is collected last on purpose: a failure here comes after every
other test has run.  It must pass alone in a fresh process and after the rest.

Checks, through the C ABI:
  - two calls in a row, each bit-identical to bi_decode_attention (caller
    workspace) on the same inputs, and the first one within the attention
    tolerance of the fp64 oracle (max |gpu - ref| <= 1e-2 * max |ref|);
  - a call whose partials reach the very end of the scratch array;
  - a call that needs no scratch at all (every sequence within one chunk) is
    accepted at any batch size;
  - the call allocates nothing: device memory in use is unchanged;
  - the size limit, rejected before any launch.
"""
import ctypes

import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
import oracle
from invariant_bi_rmsnorm_gb300 import _lib, inputs
from tests._util import bits, f64

pytestmark = pytest.mark.gpu

CAPACITY = 65536  # chunk partials the scratch array holds


def _problem(seed, lens, device="cuda"):
    p = inputs.decode_problem(len(lens), seq_lens=lens, seed=seed, device=device)
    return p, {k: v.cuda() for k, v in p.items()}


def _call_noalloc(lib, d, max_seq_len, out):
    B, Hq, D = d["q"].shape
    num_pages, Hkv, page, _ = d["k_cache"].shape
    return lib.bi_decode_attention_noalloc(
        d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
        d["block_table"].data_ptr(), d["block_table"].shape[1], d["seq_lens"].data_ptr(),
        B, Hq, Hkv, D, page, num_pages, max_seq_len, ctypes.c_float(1.0 / np.sqrt(D)),
        out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _with_workspace(d, msl):
    return bi.decode_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                               d["seq_lens"], max_seq_len=msl)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    lib = _lib.load()
    # two different problems, back to back, so the second call runs over what
    # the first one left in the shared scratch
    for k, (seed, lens) in enumerate(((300, [1, 256, 257, 1000, 4097, 60]),
                                      (301, [8192, 3, 700, 2048]))):
        p, d = _problem(seed, lens)
        msl = int(max(lens))
        ref = _with_workspace(d, msl)
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(lib, d, msl, out) == _lib.BI_OK
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), bits(ref))
        if k == 0:
            want = oracle.decode_attention(**p)
            err = np.abs(f64(out) - want)
            assert err.max() <= 1e-2 * np.abs(want).max()
    bi.get_device_error()


def test_noalloc_fills_the_scratch_to_its_last_partial():
    # 8 sequences x 32 heads x 256 chunks = 65536 partials, the capacity; the
    # 65536-token sequence is the last one, so its partials end at the top of
    # the array (and its (m, l) pairs at the top of their section)
    lib = _lib.load()
    lens = [1, 200, 300, 1000, 5, 4000, 2, 65536]
    assert len(lens) * 32 * (65536 // 256) == CAPACITY
    _, d = _problem(305, lens)
    ref = _with_workspace(d, 65536)
    out = torch.full_like(ref, float("nan"))
    assert _call_noalloc(lib, d, 65536, out) == _lib.BI_OK
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(ref))
    bi.get_device_error()


def test_noalloc_needs_no_scratch_for_single_chunk_sequences():
    # every sequence within one 256-token chunk: nothing goes to the scratch,
    # so a batch far beyond its partial capacity is accepted
    lib = _lib.load()
    B = 4096
    assert B * 32 > CAPACITY
    g = torch.Generator().manual_seed(306)
    lens = torch.randint(1, 257, (B,), generator=g).tolist()
    _, d = _problem(306, lens)
    ref = _with_workspace(d, 256)
    out = torch.full_like(ref, float("nan"))
    assert _call_noalloc(lib, d, 256, out) == _lib.BI_OK
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(ref))
    bi.get_device_error()


def test_noalloc_allocates_no_device_memory():
    lib = _lib.load()
    _, d = _problem(307, [3000, 17, 900])
    out = torch.empty(3, 32, 128, dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(lib, d, 3000, out) == _lib.BI_OK  # warm-up: module and symbol ready
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    torch0 = torch.cuda.memory_allocated()
    for _ in range(3):
        assert _call_noalloc(lib, d, 3000, out) == _lib.BI_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == torch0
    assert free1 == free0
    bi.get_device_error()


def test_noalloc_rejects_calls_beyond_its_scratch():
    lib = _lib.load()
    _, d = _problem(302, [5, 6])
    out = torch.empty(2, 32, 128, dtype=torch.bfloat16, device="cuda")
    # 2 sequences x 32 heads x 1025 chunks > 65536 partials: refused, nothing launched
    bt = torch.zeros(2, 16400, dtype=torch.int32, device="cuda")
    bt[:, :1] = d["block_table"][:, :1]
    d2 = dict(d, block_table=bt)
    assert _call_noalloc(lib, d2, 1025 * 256, out) == _lib.BI_ERR_WORKSPACE_TOO_SMALL
    # at the limit it runs
    assert _call_noalloc(lib, d2, 1024 * 256, out) == _lib.BI_OK
    torch.cuda.synchronize()
    bi.get_device_error()
