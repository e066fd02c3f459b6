"""csa_index_topk_noalloc: the indexer + top-k entry point for callers that
cannot allocate device memory themselves (they are handed their buffers by a
host framework that owns every allocation).  Its scratch is a fixed array in
the library's device memory; these checks compare it, through the C ABI,
with csa_index_topk run on a workspace of its own, over two calls in a row
(the array keeps the previous call's contents between calls), and read its
status word back through csa_index_topk_noalloc_status.

This file is named so that pytest collects it last."""
import ctypes

import pytest
import torch

from long_context_sparse_21_b300 import abi, synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True, scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    abi.lib()


def _bf16_case(seed, ctx):
    B = len(ctx)
    s = synth.Synth(seed, DEV)
    nk = max(c + 1 for c in ctx) // 4
    keys = s.normal("keys", (B, nk, 128))
    pool = abi.make_pool(abi.FMT_INDEX_POOL_BF16, B, nk, 128, page_entries=256, device=DEV, shuffle_seed=seed)
    abi.csa_cache_write(keys, pool)
    q = s.normal("q_idx", (B, 64, 128), dtype=torch.bfloat16)
    w = s.uniform("w", (B, 64))
    pos = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    return pool, q, w, pos


def _f32_case(seed, n=2048, nk=512):
    s = synth.Synth(seed, DEV)
    q = s.normal("q_idx", (n, 4, 64))
    w = s.uniform("w", (4,))
    keys = s.normal("keys", (1, nk, 64))
    pos = torch.arange(n, dtype=torch.int32, device=DEV)
    seq = torch.zeros(n, dtype=torch.int32, device=DEV)
    return q, w, keys, pos, seq


def _noalloc(call: abi.IndexCall):
    """Run the no-allocation entry point with the same parameters as `call`,
    into fresh idx / cnt buffers; returns them."""
    idx = torch.full_like(call.idx, -7)
    cnt = torch.full_like(call.cnt, -7)
    p = abi.CIndexParams()
    ctypes.pointer(p)[0] = call.p
    p.idx, p.cnt = idx.data_ptr(), cnt.data_ptr()
    st = abi.lib().csa_index_topk_noalloc(ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == abi.OK, abi.status_string(st)
    return idx, cnt


@pytest.mark.parametrize("score_dtype", [abi.F32, abi.BF16])
def test_noalloc_matches_workspace_call_bf16_tensor_core(score_dtype):
    # decode-shaped: 64 heads x 128 BF16 indexer, ragged contexts, one shorter than k
    pool, q, w, pos = _bf16_case(21, [65535, 4095, 16391, 515])
    call = abi.IndexCall(q, w, pos, pool, 512, 4, int(pos.max()), 4, score_dtype=score_dtype)
    want_idx, want_cnt = call()
    torch.cuda.synchronize()
    assert call.status() == abi.OK
    for _ in range(2):
        idx, cnt = _noalloc(call)
        torch.cuda.synchronize()
        assert torch.equal(cnt, want_cnt)
        assert torch.equal(idx, want_idx)


def test_noalloc_matches_workspace_call_f32_then_reuse():
    # the canonical float32 path (bit-exact), then a different problem on the
    # same array: the second problem must not see the first one's scores
    q, w, keys, pos, seq = _f32_case(22)
    call = abi.IndexCall(q, w, pos, abi.dense_store(keys), 64, 4, 2047, 1, seq=seq, w_shared=True)
    want_idx, want_cnt = call()
    pool, q2, w2, pos2 = _bf16_case(23, [8191, 300])
    call2 = abi.IndexCall(q2, w2, pos2, pool, 256, 4, int(pos2.max()), 2)
    want2_idx, want2_cnt = call2()
    torch.cuda.synchronize()
    for c, wi, wc in [(call, want_idx, want_cnt), (call2, want2_idx, want2_cnt), (call, want_idx, want_cnt)]:
        idx, cnt = _noalloc(c)
        torch.cuda.synchronize()
        assert torch.equal(cnt, wc)
        assert torch.equal(idx, wi)


def test_noalloc_status_reports_a_nan_score_then_resets():
    """NaN head weights for one query row give NaN index scores: the selector
    records CSA_ERR_INVALID_ARG in the array's status word, which the status
    reader returns.  The next call starts from CSA_OK again."""
    pool, q, w, pos = _bf16_case(25, [8191, 4095])
    w_bad = w.clone()
    w_bad[1] = float("nan")
    call = abi.IndexCall(q, w_bad, pos, pool, 128, 4, int(pos.max()), 2)
    _noalloc(call)
    assert abi.csa_index_topk_noalloc_status() == abi.ERR_INVALID_ARG
    good = abi.IndexCall(q, w, pos, pool, 128, 4, int(pos.max()), 2)
    want_idx, want_cnt = good()
    idx, cnt = _noalloc(good)
    assert abi.csa_index_topk_noalloc_status() == abi.OK
    assert torch.equal(idx, want_idx) and torch.equal(cnt, want_cnt)


def test_noalloc_rejects_oversized_problem():
    # 8 MiB of scratch: 20,000 queries x 128 float32 score slots (10.24 MB) do not fit
    T = 20000
    s = synth.Synth(24, DEV)
    q = s.normal("q", (T, 1, 4))
    w = s.uniform("w", (1,))
    keys = s.normal("keys", (1, 128, 4))
    pos = torch.full((T,), 511, dtype=torch.int32, device=DEV)
    seq = torch.zeros(T, dtype=torch.int32, device=DEV)
    p = abi.CIndexParams(struct_size=ctypes.sizeof(abi.CIndexParams), num_queries=T, batch=1, heads=1, dim=4, m=4,
                         max_pos=511, q=q.data_ptr(), q_dtype=abi.F32, w=w.data_ptr(), w_shared=1,
                         pos=pos.data_ptr(), seq=seq.data_ptr(), keys=abi.dense_store(keys).c(), top_k=8,
                         score_dtype=abi.F32)
    idx = torch.empty((T, 8), dtype=torch.int32, device=DEV)
    cnt = torch.empty((T,), dtype=torch.int32, device=DEV)
    p.idx, p.cnt = idx.data_ptr(), cnt.data_ptr()
    assert abi.lib().csa_index_topk_workspace_size(ctypes.byref(p)) > 8 << 20
    st = abi.lib().csa_index_topk_noalloc(ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == abi.ERR_WORKSPACE
