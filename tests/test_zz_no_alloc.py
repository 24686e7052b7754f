"""bi_decode_attention_noalloc: the attention entry point for callers that
cannot allocate device memory at call time (a plugin given only its input and
output buffers, a serving loop whose memory a caching allocator reserved up
front).  It keeps its chunk partials in a fixed scratch array inside the
library instead of a caller workspace.

This file is collected last on purpose: a failure here comes after every
other test has run.  It must pass alone in a fresh process and after the rest.

Checks, through the C ABI: two calls in a row, each compared with
bi_decode_attention on the same inputs (bit-identical, and within the
attention tolerance of the oracle tests); and the size limit, rejected before
any launch.
"""
import ctypes

import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_gb300 as bi
from invariant_bi_rmsnorm_gb300 import _lib, inputs
from tests._util import bits, f64

pytestmark = pytest.mark.gpu


def _problem(seed, lens):
    p = inputs.decode_problem(len(lens), seq_lens=lens, seed=seed)
    return {k: v.cuda() for k, v in p.items()}


def _call_noalloc(lib, d, max_seq_len, out):
    B, Hq, D = d["q"].shape
    num_pages, Hkv, page, _ = d["k_cache"].shape
    return lib.bi_decode_attention_noalloc(
        d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
        d["block_table"].data_ptr(), d["block_table"].shape[1], d["seq_lens"].data_ptr(),
        B, Hq, Hkv, D, page, num_pages, max_seq_len, ctypes.c_float(1.0 / np.sqrt(D)),
        out.data_ptr(), torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    lib = _lib.load()
    # two different problems, back to back, so the second call runs over the
    # partials the first one left in the shared scratch
    for seed, lens in ((300, [1, 256, 257, 1000, 4097, 60]), (301, [8192, 3, 700, 2048])):
        d = _problem(seed, lens)
        msl = int(max(lens))
        ref = bi.decode_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                  d["seq_lens"], max_seq_len=msl)
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(lib, d, msl, out) == _lib.BI_OK
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), bits(ref))
        err = np.abs(f64(out) - f64(ref))
        assert err.max() <= 1e-2 * np.abs(f64(ref)).max()
    bi.get_device_error()


def test_noalloc_rejects_calls_beyond_its_scratch():
    lib = _lib.load()
    d = _problem(302, [5, 6])
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
