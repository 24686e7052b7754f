"""Host-side checks of libbi.so that need no GPU: the library loads, exports
every entry point include/bi.h declares, and rejects invalid arguments before
touching the device.  No call here launches a kernel (the pointers passed are
never dereferenced: validation fails first)."""
import os
import re

import pytest

from invariant_bi_rmsnorm_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_entry_points():
    src = open(os.path.join(ROOT, "include", "bi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return _lib.load()


def test_library_exports_every_declared_entry_point(lib):
    declared = _declared_entry_points()
    assert declared, "no declarations parsed"
    assert set(declared) == set(_lib.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_abi_version_and_status_strings(lib):
    assert lib.bi_abi_version() == 2
    for code, name in [(0, "BI_OK"), (1, "BI_ERR_INVALID_ARG"), (2, "BI_ERR_UNSUPPORTED_SHAPE"),
                       (3, "BI_ERR_MISALIGNED"), (4, "BI_ERR_WORKSPACE_TOO_SMALL"),
                       (5, "BI_ERR_CUDA"), (6, "BI_ERR_DEVICE_TIMEOUT"),
                       (7, "BI_ERR_DEVICE_BAD_INPUT")]:
        assert lib.bi_status_string(code).decode() == name


def _golden_plans():
    out = []
    for line in open(os.path.join(ROOT, "tests", "golden", "chunk_plan.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            head, tail = line.split(":")
            L, chunk = (int(t) for t in head.split())
            out.append((L, chunk, [int(t) for t in tail.split()]))
    return out


@pytest.mark.parametrize("L,chunk,plan", _golden_plans())
def test_chunk_plan_matches_pages_example(lib, L, chunk, plan):
    assert chunk == _lib.DECODE_CHUNK
    n = lib.bi_decode_num_chunks(L)
    assert [lib.bi_decode_chunk_len(L, c) for c in range(n)] == plan


@pytest.mark.parametrize("L", [1, 2, 255, 256, 257, 511, 512, 513, 4097, 8192])
def test_chunk_plan_properties(lib, L):
    n = lib.bi_decode_num_chunks(L)
    lens = [lib.bi_decode_chunk_len(L, c) for c in range(n)]
    assert sum(lens) == L
    assert all(x == 256 for x in lens[:-1]) and 1 <= lens[-1] <= 256
    assert lib.bi_decode_chunk_len(L, n) == 0 and lib.bi_decode_chunk_len(L, -1) == 0
    # a length-L plan is a prefix of every longer sequence's plan, chunk for
    # chunk, up to its last (partial) chunk: the growth-invariance property
    longer = [lib.bi_decode_chunk_len(L + 300, c) for c in range(lib.bi_decode_num_chunks(L + 300))]
    assert longer[:n - 1] == lens[:n - 1]


def test_workspace_size(lib):
    ctr = _lib.DECODE_COUNTER_BYTES  # arrival counters ahead of the partials
    assert ctr == 262144
    assert lib.bi_decode_attention_workspace_size(256, 32, 128, 8192) == ctr + 256 * 32 * 32 * 130 * 4
    assert lib.bi_decode_attention_workspace_size(4, 32, 128, 256) == 0  # single chunk
    assert lib.bi_decode_attention_workspace_size(4, 32, 128, 257) == ctr + 4 * 32 * 2 * 130 * 4
    assert lib.bi_decode_attention_workspace_size(-1, 32, 128, 1000) == 0


FAKE = 0x10000  # 16-byte aligned, never dereferenced


def test_rmsnorm_argument_validation(lib):
    f = lib.bi_rmsnorm
    assert f(FAKE, FAKE, FAKE, 4, 4100, 4100, 4100, 1e-6, None) == _lib.BI_ERR_UNSUPPORTED_SHAPE
    assert f(FAKE, FAKE, FAKE, 4, 40000, 40000, 40000, 1e-6, None) == _lib.BI_ERR_UNSUPPORTED_SHAPE
    assert f(FAKE, FAKE, FAKE, 4, 4096, 4000, 4096, 1e-6, None) == _lib.BI_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 4, 4096, 4100, 4096, 1e-6, None) == _lib.BI_ERR_MISALIGNED
    assert f(FAKE, FAKE, FAKE, -1, 4096, 4096, 4096, 1e-6, None) == _lib.BI_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 4, 4096, 4096, 4096, -1.0, None) == _lib.BI_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, 4, 4096, 4096, 4096, float("nan"), None) == _lib.BI_ERR_INVALID_ARG
    assert f(None, FAKE, FAKE, 4, 4096, 4096, 4096, 1e-6, None) == _lib.BI_ERR_INVALID_ARG
    assert f(FAKE + 2, FAKE, FAKE, 4, 4096, 4096, 4096, 1e-6, None) == _lib.BI_ERR_MISALIGNED
    assert f(None, None, None, 0, 4096, 4096, 4096, 1e-6, None) == _lib.BI_OK  # empty: no launch


def test_gemm_argument_validation(lib):
    f = lib.bi_gemm
    assert f(FAKE, FAKE, FAKE, 4, 12, 64, 64, 64, 12, None) == _lib.BI_ERR_UNSUPPORTED_SHAPE  # N % 8
    assert f(FAKE, FAKE, FAKE, 4, 16, 60, 60, 60, 16, None) == _lib.BI_ERR_UNSUPPORTED_SHAPE  # K % 8
    assert f(FAKE, FAKE, FAKE, 4, 16, 64, 32, 64, 16, None) == _lib.BI_ERR_INVALID_ARG  # ld_x < K
    assert f(FAKE, FAKE, FAKE, 4, 16, 64, 68, 64, 16, None) == _lib.BI_ERR_MISALIGNED
    assert f(FAKE, FAKE, FAKE, -4, 16, 64, 64, 64, 16, None) == _lib.BI_ERR_INVALID_ARG
    assert f(FAKE + 8, FAKE, FAKE, 4, 16, 64, 64, 64, 16, None) == _lib.BI_ERR_MISALIGNED
    assert f(None, None, None, 0, 16, 64, 64, 64, 16, None) == _lib.BI_OK


def test_decode_attention_argument_validation(lib):
    f = lib.bi_decode_attention
    # (q, k, v, bt, max_pages, lens, B, Hq, Hkv, D, page, num_pages, max_seq_len, scale, out, ws, ws_bytes, stream)
    ok = dict(q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mp=64, lens=FAKE, B=4, Hq=32, Hkv=8, D=128,
              page=16, np_=256, msl=1000, scale=0.088, out=FAKE, ws=FAKE, wsb=10 ** 9, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["v"], a["bt"], a["mp"], a["lens"], a["B"], a["Hq"], a["Hkv"],
                 a["D"], a["page"], a["np_"], a["msl"], a["scale"], a["out"], a["ws"], a["wsb"],
                 a["s"])
    assert call(D=64) == _lib.BI_ERR_UNSUPPORTED_SHAPE
    assert call(page=32) == _lib.BI_ERR_UNSUPPORTED_SHAPE
    assert call(Hq=30) == _lib.BI_ERR_UNSUPPORTED_SHAPE       # Hq % Hkv
    assert call(Hq=80, Hkv=8) == _lib.BI_ERR_UNSUPPORTED_SHAPE  # group 10 > 8
    assert call(msl=64 * 16 + 1) == _lib.BI_ERR_INVALID_ARG   # beyond the block table
    assert call(scale=0.0) == _lib.BI_ERR_INVALID_ARG
    assert call(wsb=100) == _lib.BI_ERR_WORKSPACE_TOO_SMALL
    assert call(ws=None) == _lib.BI_ERR_WORKSPACE_TOO_SMALL
    assert call(q=FAKE + 4) == _lib.BI_ERR_MISALIGNED
    assert call(bt=FAKE + 2) == _lib.BI_ERR_MISALIGNED
    assert call(lens=None) == _lib.BI_ERR_INVALID_ARG
    assert call(np_=2 ** 27) == _lib.BI_ERR_UNSUPPORTED_SHAPE  # rows overflow int32
    assert call(B=0) == _lib.BI_OK


def test_selftest_and_fixed_splits_validation(lib):
    assert lib.bi_selftest_wait_timeout(0, None) == _lib.BI_ERR_INVALID_ARG
    assert lib.bi_selftest_wait_timeout(2000001, None) == _lib.BI_ERR_INVALID_ARG
    f = lib.bi_decode_attention_fixed_splits
    args = [FAKE, FAKE, FAKE, FAKE, 64, FAKE, 4, 32, 8, 128, 16, 256, 1000, 0.088]
    assert f(*args, 0, FAKE, FAKE, 10 ** 9, None) == _lib.BI_ERR_INVALID_ARG      # no splits
    assert f(*args, 4, FAKE, FAKE, 100, None) == _lib.BI_ERR_WORKSPACE_TOO_SMALL
    big = [FAKE, FAKE, FAKE, FAKE, 1024, FAKE, 4, 32, 8, 128, 16, 256, 16384, 0.088]
    assert f(*big, 1, FAKE, FAKE, 10 ** 9, None) == _lib.BI_ERR_UNSUPPORTED_SHAPE  # 1024 pages per split


def test_binding_refuses_cpu_tensors():
    import torch
    import invariant_bi_rmsnorm_gb300 as bi
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        bi.rmsnorm(x, torch.ones(64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA"):
        bi.gemm(x, x)


def test_noalloc_size_limit_is_checked_on_the_host(lib):
    f = lib.bi_decode_attention_noalloc
    # (q, k, v, bt, max_pages, lens, B, Hq, Hkv, D, page, num_pages, max_seq_len, scale, out, stream)
    # 2 x 32 x 1025 chunk partials > 65536: refused before any device work
    assert f(FAKE, FAKE, FAKE, FAKE, 16400, FAKE, 2, 32, 8, 128, 16, 256, 1025 * 256, 0.088,
             FAKE, None) == _lib.BI_ERR_WORKSPACE_TOO_SMALL
    assert f(FAKE, FAKE, FAKE, FAKE, 64, FAKE, -1, 32, 8, 128, 16, 256, 1000, 0.088,
             FAKE, None) == _lib.BI_ERR_INVALID_ARG
