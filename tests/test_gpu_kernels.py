"""Parity of every C-ABI kernel against the CPU oracle, on the same seeded
inputs, at sizes that span several tiles and a ragged tail.

Bars: bit-exact for codes, layouts and index sets of the float32 path;
max-abs-rel 1e-4 for float32 attention, 2e-2 for the BF16/FP8 path; selection
sets of the tensor-core indexer checked for validity within the score error."""
import math

import numpy as np
import pytest
import torch

from long_context_sparse_21_b300 import abi, synth
from oracle import codecs, csa

from helpers import (f64, max_abs_rel, read_index_bf16_pool, read_index_fp4_pool, read_kv_pool,
                     score_error_bound, selection_valid)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True, scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    abi.lib()


def sync():
    torch.cuda.synchronize()


# ------------------------------------------------------------------ cache writer

def _entries(B, n, D, seed):
    s = synth.Synth(seed, DEV)
    x = s.normal("entries", (B, n, D))
    x[0, 3] = 0.0                         # amax 0 -> scale 1
    x[0, 5] *= 1e3                        # large
    x[1, 7] *= 1e-30                      # subnormal e4m3 region after scaling
    x[1, 9, :16] = 0.0                    # an all-zero FP4 block
    x[1, 11] *= 1e-6
    return x


def test_cache_write_kv_fp8_bit_exact():
    B, n = 2, 300
    x = _entries(B, n, 576, 1)
    pool = abi.make_pool(abi.FMT_KV_POOL_FP8, B, n, 576, page_entries=128, device=DEV, shuffle_seed=3)
    abi.csa_cache_write(x, pool)
    sync()
    xc = x.cpu().numpy()
    for b in range(B):
        codes, scale, rope = read_kv_pool(pool, b, n)
        wc, ws, wr = codecs.kv_entry_encode(xc[b])
        assert np.array_equal(scale.view(np.uint32), ws.view(np.uint32))
        assert np.array_equal(codes, wc)
        assert np.array_equal(rope, wr)


def test_cache_write_index_bf16_layout_bit_exact():
    B, n = 2, 300
    x = _entries(B, n, 128, 2)
    pool = abi.make_pool(abi.FMT_INDEX_POOL_BF16, B, n, 128, page_entries=256, device=DEV, shuffle_seed=4)
    abi.csa_cache_write(x, pool, first=0)
    sync()
    for b in range(B):
        assert np.array_equal(read_index_bf16_pool(pool, b, n), codecs.bf16_encode(x[b].cpu().numpy()))


def test_cache_write_index_fp4_bit_exact():
    B, n = 2, 300
    x = _entries(B, n, 128, 5) * 3
    pool = abi.make_pool(abi.FMT_INDEX_POOL_E2M1, B, n, 128, page_entries=128, device=DEV, shuffle_seed=6)
    abi.csa_cache_write(x, pool)
    sync()
    for b in range(B):
        codes, scales = read_index_fp4_pool(pool, b, n)
        wc, ws = codecs.fp4_block_encode(x[b].cpu().numpy())
        assert np.array_equal(scales, ws)
        assert np.array_equal(codes, wc)


# ------------------------------------------------------------------ compressor

@pytest.mark.parametrize("m,D,n,dtype", [(4, 192, 2048, torch.float32), (4, 64, 2048, torch.float32),
                                         (128, 576, 3 * 128 + 5, torch.bfloat16), (1, 32, 40, torch.float32)])
def test_compress_dense(m, D, n, dtype):
    s = synth.Synth(7, DEV)
    B = 2
    k = s.normal("k", (B, n, D), dtype=dtype)
    g = s.normal("g", (B, n, D), dtype=dtype)
    bias = s.normal("bias", (m, D), 0.1)
    out = torch.full((B, n // m + 1, D), float("nan"), device=DEV)
    abi.csa_compress(abi.dense_store(out), bias, m, k=k, g=g)
    sync()
    for b in range(B):
        want = csa.compress(f64(k[b]), f64(g[b]), f64(bias), m)
        got = f64(out[b, : n // m])
        assert np.abs(got - want).max() <= 2e-6 * np.abs(want).max()
    assert torch.isnan(out[:, n // m]).all()  # the partial block is not emitted


def test_compress_dense_into_kv_pool():
    m, D, n, B = 4, 576, 1024 + 3, 2
    s = synth.Synth(8, DEV)
    k = s.normal("k", (B, n, D), dtype=torch.bfloat16)
    g = s.normal("g", (B, n, D), dtype=torch.bfloat16)
    bias = s.normal("bias", (m, D), 0.1)
    pool = abi.make_pool(abi.FMT_KV_POOL_FP8, B, n // m, D, page_entries=128, device=DEV)
    abi.csa_compress(pool, bias, m, k=k, g=g)
    sync()
    for b in range(B):
        want = csa.compress(f64(k[b]), f64(g[b]), f64(bias), m)
        got = codecs.kv_entry_decode(*read_kv_pool(pool, b, n // m))
        amax = np.abs(want[:, :512]).max(1, keepdims=True)
        # one e4m3 rounding of the content (<= 2^-4 relative + subnormal step), bf16 for RoPE dims
        assert np.all(np.abs(got[:, :512] - want[:, :512]) <= 2.0 ** -4 * np.abs(want[:, :512]) + amax / 448 * 2.0 ** -9 * 1.01 + 1e-6 * amax)
        assert np.all(np.abs(got[:, 512:] - want[:, 512:]) <= 2.0 ** -8 * np.abs(want[:, 512:]) + 1e-6)


@pytest.mark.parametrize("m", [4, 128])
def test_compress_append(m):
    D, B, R = 576, 3, 128
    s = synth.Synth(9, DEV)
    # lengths before the append: the first and last complete a block, the middle one does not
    L = [131, 140, 139] if m == 4 else [383, 389, 511]
    ring = s.normal("ring", (B, R, D), dtype=torch.bfloat16)
    tail = s.normal("tail", (B, m, D))
    bias = s.normal("bias", (m, D), 0.1)
    k_new = s.normal("k_new", (B, D), dtype=torch.bfloat16)
    g_new = s.normal("g_new", (B, D))
    cap = max(L) // m + 1
    out = torch.full((B, cap, D), float("nan"), device=DEV)
    ring0, tail0 = ring.clone(), tail.clone()
    seq_len = torch.tensor(L, dtype=torch.int32, device=DEV)
    for rep in range(2):  # idempotent: the same call twice gives the same state
        abi.csa_compress(abi.dense_store(out), bias, m, seq_len=seq_len, k_new=k_new, g_new=g_new, ring=ring,
                         tail_gate=tail)
    sync()
    for b in range(B):
        Lb = L[b]
        assert torch.equal(ring[b, Lb % R], k_new[b])
        assert torch.equal(tail[b, Lb % m], g_new[b])
        others = [i for i in range(R) if i != Lb % R]
        assert torch.equal(ring[b, others], ring0[b, others])
        j = (Lb + 1) // m - 1
        if (Lb + 1) % m == 0:
            p = np.arange(Lb + 1 - m, Lb + 1)
            kb = f64(ring0[b])[p % R]
            kb[-1] = f64(k_new[b])
            gb = f64(tail0[b])[p % m]
            gb[-1] = f64(g_new[b])
            want = csa.compress(kb, gb, f64(bias), m)[0]
            got = f64(out[b, j])
            assert np.abs(got - want).max() <= 2e-6 * np.abs(want).max()
        else:
            assert torch.isnan(out[b]).all()


# ------------------------------------------------------------------ indexer + top-k

def _f32_index_inputs(seed, n=2048, nk=512, H=4, dI=64, dup=False):
    s = synth.Synth(seed, DEV)
    q = s.normal("q_idx", (n, H, dI))
    w = s.uniform("w", (H,))
    keys = s.normal("keys", (1, nk, dI))
    if dup:  # repeated keys -> exactly tied scores
        keys[0, 1::3] = keys[0, 0:-1:3][: keys[0, 1::3].shape[0]]
    return q, w, keys


@pytest.mark.parametrize("score_dtype,dup", [(abi.F32, False), (abi.F32, True), (abi.BF16, False)])
def test_index_topk_f32_bit_exact(score_dtype, dup):
    n, m, k = 2048, 4, 64
    q, w, keys = _f32_index_inputs(11, n=n, dup=dup)
    pos = torch.arange(n, dtype=torch.int32, device=DEV)
    seq = torch.zeros(n, dtype=torch.int32, device=DEV)
    scores_out = torch.full((n, 512), float("nan"), device=DEV)
    call = abi.IndexCall(q, w, pos, abi.dense_store(keys), k, m, n - 1, 1, seq=seq, score_dtype=score_dtype,
                         w_shared=True, scores_out=scores_out)
    idx, cnt = call()
    sync()
    assert call.status() == 0
    idx, cnt, sc = idx.cpu().numpy(), cnt.cpu().numpy(), scores_out.cpu().numpy()
    qn, wn, kn = q.cpu().numpy(), w.cpu().numpy(), keys[0].cpu().numpy()
    for t in range(n):
        nc = (t + 1) // m
        s32 = csa.index_scores_f32(qn[t], wn, kn[:nc])
        if score_dtype == abi.BF16:
            s32 = csa.bf16_score(s32).astype(np.float32)
        assert np.array_equal(sc[t, :nc].view(np.uint32), s32.view(np.uint32)), t
        want, wc = csa.topk(s32, nc, k)
        assert cnt[t] == wc and np.array_equal(idx[t], want), t


@pytest.mark.parametrize("score_dtype", [abi.F32, abi.BF16])
@pytest.mark.parametrize("rows", [(262144, 100000, 5000, 1000), (400000, 300000), (700000, 2000), (1100000, 5000),
                                  (262144,) * 8])
def test_topk_long_rows_with_ties(score_dtype, rows):
    """The selector alone on long rows with many exact ties, bit-exact against
    the oracle's stable top-k.  One query head of dim 4 with q = e0 and w = 1
    makes each score exactly ReLU(key[0]) (canonical float32), so the scores
    are chosen directly: multiples of 1/8 (ties everywhere, and ~half the
    blocks at exactly 0).  A few rows take clusters of 16 CTAs (8 where 16
    would not all fit at once): the first two sets stage their chunks (up to
    25,000 blocks) in shared memory; 700,000-block rows (chunks of 43,750) are
    read from global memory, and 1,100,000-block rows (chunks of 68,750) give
    each thread a run of more than 64 blocks in the compaction.  Eight rows of
    262,144 ask for eight clusters of 16, which the occupancy check admits or
    turns into clusters of 8 depending on the GPU: either way the result is
    checked."""
    n_max, k = rows[0], 1024
    s = synth.Synth(31 + len(rows), DEV)
    keys = torch.zeros((1, n_max, 4), device=DEV)
    keys[0, :, 0] = torch.floor(s.normal("v", (n_max,)) * 8) / 8
    T = len(rows)
    q = torch.zeros((T, 1, 4), device=DEV)
    q[:, 0, 0] = 1.0
    w = torch.ones((1,), device=DEV)
    pos = torch.tensor([r - 1 for r in rows], dtype=torch.int32, device=DEV)
    seq = torch.zeros(T, dtype=torch.int32, device=DEV)
    call = abi.IndexCall(q, w, pos, abi.dense_store(keys), k, 1, n_max - 1, 1, seq=seq, score_dtype=score_dtype,
                         w_shared=True)
    idx, cnt = call()
    sync()
    assert call.status() == 0
    v = np.maximum(keys[0, :, 0].cpu().numpy(), 0).astype(np.float32)
    if score_dtype == abi.BF16:
        v = csa.bf16_score(v).astype(np.float32)
    for r, n in enumerate(rows):
        want, wc = csa.topk(v[:n], n, k)
        assert int(cnt[r]) == wc, r
        assert np.array_equal(idx[r].cpu().numpy(), want), r


def _bf16_index_setup(seed, ctx, fmt=abi.FMT_INDEX_POOL_BF16, P=2048):
    B = len(ctx)
    s = synth.Synth(seed, DEV)
    nk = max(c + 1 for c in ctx) // 4
    keys = s.normal("keys", (B, nk, 128))
    pool = abi.make_pool(fmt, B, nk, 128, page_entries=P, device=DEV, shuffle_seed=seed)
    abi.csa_cache_write(keys, pool)
    q = s.normal("q_idx", (B, 64, 128), dtype=torch.bfloat16)
    w = s.uniform("w", (B, 64))
    pos = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    return keys, pool, q, w, pos


@pytest.mark.parametrize("score_dtype", [abi.F32, abi.BF16])
def test_index_topk_bf16_tensor_core(score_dtype):
    ctx = [3999, 16391, 1199, 65535, 515]  # ragged tiles; the last has fewer blocks than k
    k = 512
    keys, pool, q, w, pos = _bf16_index_setup(12, ctx, P=256)
    nk = keys.shape[1]
    scores_out = torch.full((len(ctx), nk), float("nan"), device=DEV)
    call = abi.IndexCall(q, w, pos, pool, k, 4, max(ctx), len(ctx), score_dtype=score_dtype, scores_out=scores_out)
    idx, cnt = call()
    sync()
    assert call.status() == 0
    kb = codecs.bf16_round(keys.cpu().numpy())
    for b, t in enumerate(ctx):
        nc = (t + 1) // 4
        want = csa.index_scores(f64(q[b]), f64(w[b]), kb[b, :nc])
        got = f64(scores_out[b, :nc])
        tol = score_error_bound(f64(q[b]), f64(w[b]), kb[b, :nc], bf16_scores=score_dtype == abi.BF16)
        assert np.all(np.abs(got - want) <= tol), b
        ok, why = selection_valid(idx[b].cpu().numpy(), int(cnt[b]), want, k, tol)
        assert ok, (b, why)


def test_index_topk_fp4():
    ctx = [8191, 2999]
    k = 512
    keys, pool, _, w, pos = _bf16_index_setup(13, ctx, fmt=abi.FMT_INDEX_POOL_E2M1, P=128)
    s = synth.Synth(13, DEV)
    q = s.normal("q_idx32", (len(ctx), 64, 128))
    nk = keys.shape[1]
    scores_out = torch.full((len(ctx), nk), float("nan"), device=DEV)
    call = abi.IndexCall(q, w, pos, pool, k, 4, max(ctx), len(ctx), scores_out=scores_out)
    idx, cnt = call()
    sync()
    recalls = []
    for b, t in enumerate(ctx):
        nc = (t + 1) // 4
        kc, ks = codecs.fp4_block_encode(keys[b, :nc].cpu().numpy())
        qc, qsc = codecs.fp4_block_encode(q[b].cpu().numpy())
        qd, kd = codecs.fp4_block_decode(qc, qsc), codecs.fp4_block_decode(kc, ks)
        want = csa.index_scores(qd, f64(w[b]), kd)
        got = f64(scores_out[b, :nc])
        tol = score_error_bound(qd, f64(w[b]), kd, bf16_scores=False)
        assert np.all(np.abs(got - want) <= tol)
        ok, why = selection_valid(idx[b].cpu().numpy(), int(cnt[b]), want, k, tol)
        assert ok, why
        ref = csa.index_scores(f64(q[b]), f64(w[b]), f64(keys[b, :nc]))
        ridx, rc = csa.topk(ref, nc, k)
        recalls.append(len(np.intersect1d(ridx[:rc], idx[b, : int(cnt[b])].cpu().numpy())) / rc)
    print("FP4 indexer recall vs float32 oracle:", recalls)
    assert min(recalls) > 0.5


# ------------------------------------------------------------------ attention

def _idx_for(s, name, pos, m, k):
    rows = []
    cnts = []
    gen = np.random.Generator(np.random.Philox(synth._key(s.seed, name)))
    for t in pos:
        nc = (t + 1) // m
        kk = min(k, nc)
        r = np.full(k, -1, np.int32)
        r[:kk] = np.sort(gen.choice(nc, size=kk, replace=False)) if kk else []
        rows.append(r)
        cnts.append(kk)
    return (torch.tensor(np.array(rows), dtype=torch.int32, device=DEV),
            torch.tensor(cnts, dtype=torch.int32, device=DEV))


@pytest.mark.parametrize("sparse,sink,W,nq", [(True, False, 128, 300), (False, False, 128, 300), (True, True, 128, 300),
                                              (True, False, 0, 9), (False, False, 128, 2)])
def test_attend_f32(sparse, sink, W, nq):
    n, D, H, m, k = 300, 192, 16, 4, 64
    s = synth.Synth(21, DEV)
    comp = s.normal("comp", (1, n // m, D))
    raw = s.normal("raw", (1, n, D))
    pos_l = list(range(n))[:nq] if nq > 2 else [n - 1, 150]
    pos = torch.tensor(pos_l, dtype=torch.int32, device=DEV)
    seq = torch.zeros(len(pos_l), dtype=torch.int32, device=DEV)
    q = s.normal("q", (len(pos_l), H, D))
    idx, cnt = _idx_for(s, "idx", pos_l, m, k)
    sk = s.normal("sink", (H,)) if sink else None
    call = abi.AttendCall(sparse, q, pos, abi.dense_store(comp), W, raw, 1 / math.sqrt(D), m, n - 1, 1,
                          idx=idx, cnt=cnt, seq=seq, sink=sk)
    o, lse = call()
    sync()
    assert call.status() == 0
    qn, cn, rn = f64(q), f64(comp[0]), f64(raw[0])
    skn = None if sk is None else f64(sk)
    want_o, want_l = [], []
    for r, t in enumerate(pos_l):
        if sparse:
            wo, wl = csa.csa_attend(qn[r], t, idx[r].cpu().numpy(), int(cnt[r]), cn, rn, W, 1 / math.sqrt(D), skn)
        else:
            wo, wl = csa.hca_attend(qn[r], t, m, cn, rn, W, 1 / math.sqrt(D), skn)
        want_o.append(wo)
        want_l.append(wl)
    want_o, want_l = np.array(want_o), np.array(want_l)
    got_o, got_l = f64(o), f64(lse)
    empty = np.isneginf(want_l)
    assert np.all(got_o[empty] == 0) and np.all(np.isneginf(got_l[empty]))
    nz = ~empty.all(axis=1)
    assert max_abs_rel(got_o[nz], want_o[nz]) <= 1e-4
    assert np.allclose(got_l[~empty], want_l[~empty], rtol=0, atol=1e-4)


def _fp8_attend_setup(seed, ctx, m, k):
    B = len(ctx)
    s = synth.Synth(seed, DEV)
    nk = max(c + 1 for c in ctx) // m
    ent = s.normal("entries", (B, nk, 576))
    pool = abi.make_pool(abi.FMT_KV_POOL_FP8, B, nk, 576, page_entries=128, device=DEV, shuffle_seed=seed)
    abi.csa_cache_write(ent, pool)
    ring = s.normal("ring", (B, 128, 576), dtype=torch.bfloat16)
    q = s.normal("q", (B, 64, 576), dtype=torch.bfloat16)
    pos = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    idx, cnt = _idx_for(s, "idx", ctx, m, k)
    return ent, pool, ring, q, pos, idx, cnt


@pytest.mark.parametrize("sparse,out_dtype,ctx,sink", [
    (False, torch.bfloat16, [2800, 1203, 130], False),
    (True, torch.float32, [2800, 1203, 130], False),
    (True, torch.bfloat16, list(range(150, 150 + 7 * 190, 7)), False),   # many queries: no split
    (False, torch.float32, [64, 2, 0], False),                              # tiny and single-token windows
    (True, torch.float32, [2800, 1203, 130], True),                         # attention sink (report §2.3.3)
    (False, torch.bfloat16, [5000, 64, 0], True),                           # sink with split-K and an empty set
    (False, torch.bfloat16, [20000, 9000], False),                          # 41 splits: partials merged by the combine kernel
    (True, torch.float32, [20000, 9000], True),                             # 4-5 splits merged in a cluster, with a sink
])
def test_attend_fp8_tensor_core(sparse, out_dtype, ctx, sink):
    m, k = 4, 512
    ent, pool, ring, q, pos, idx, cnt = _fp8_attend_setup(31, ctx, m, k)
    scale = 1 / 24
    # sink logits around the typical logit range, so they take a visible share of the mass
    sk = synth.Synth(32, DEV).normal("sink", (64,)) * 2 + 1 if sink else None
    call = abi.AttendCall(sparse, q, pos, pool, 128, ring, scale, m, max(ctx), len(ctx), idx=idx, cnt=cnt,
                          out_dtype=out_dtype, sink=sk)
    o, lse = call()
    sync()
    assert call.status() == 0
    print("splits, merge:", call.plan())
    entn = ent.cpu().numpy()
    ringn = f64(ring)
    skn = None if sk is None else f64(sk)
    worst = 0.0
    for b, t in enumerate(ctx):
        nc = (t + 1) // m
        rows = idx[b, : int(cnt[b])].cpu().numpy() if sparse else np.arange(nc)
        X = codecs.kv_entry_decode(*codecs.kv_entry_encode(entn[b, rows])) if len(rows) else np.zeros((0, 576))
        wp = csa.window_positions(t, 128)
        wo, wl = csa.attend_one(f64(q[b]), X, ringn[b, wp % 128], scale, skn)
        worst = max(worst, max_abs_rel(f64(o[b]), wo))
        assert np.allclose(f64(lse[b]), wl, atol=2e-2)
    print("max-abs-rel", worst)
    assert worst <= 2e-2


# ------------------------------------------------------------------ device-side checks of page ids and sequences

def test_page_ids_outside_the_pool_are_reported_not_read():
    """Page ids are device data: a page table entry outside [0, num_pages)
    must be skipped by every kernel that reads or writes pages, with
    CSA_ERR_INVALID_ARG in the call's status word (the pages' layout is the
    state cache of report §3.5.1; the ids here are planted by the test)."""
    ctx = [4000, 3000]
    ent, pool, ring, q, pos, idx, cnt = _fp8_attend_setup(41, ctx, 4, 64)
    bad = pool.page_table.clone()
    pool.page_table[0, 1] = pool.num_pages        # one past the pool
    pool.page_table[1, 0] = -1
    call = abi.AttendCall(False, q, pos, pool, 128, ring, 1 / 24, 4, max(ctx), len(ctx))
    call()
    sync()
    assert call.status() == abi.ERR_INVALID_ARG
    # the indexer's bulk-copy producer
    keys, ipool, qi, w, ipos = _bf16_index_setup(42, ctx, P=256)
    ipool.page_table[1, 2] = ipool.num_pages + 7
    icall = abi.IndexCall(qi, w, ipos, ipool, 64, 4, max(ctx), len(ctx))
    icall()
    sync()
    assert icall.status() == abi.ERR_INVALID_ARG
    # the FP4 indexer's copy warp (a tensor-map load of the codes, a bulk copy of the scales)
    _, fpool, _, fw, fpos = _bf16_index_setup(44, ctx, fmt=abi.FMT_INDEX_POOL_E2M1, P=128)
    fpool.page_table[0, 3] = fpool.num_pages
    fq = synth.Synth(44, DEV).normal("q_idx32", (len(ctx), 64, 128))
    fcall = abi.IndexCall(fq, fw, fpos, fpool, 64, 4, max(ctx), len(ctx))
    fcall()
    sync()
    assert fcall.status() == abi.ERR_INVALID_ARG
    # the cache writer drops the write
    ws = abi.alloc_workspace(1024)
    ws.zero_()
    abi.csa_cache_write(ent[:, :300].contiguous(), pool, status=ws)
    sync()
    assert abi.workspace_status(ws) == abi.ERR_INVALID_ARG
    pool.page_table.copy_(bad)
    ws.zero_()
    abi.csa_cache_write(ent[:, :300].contiguous(), pool, status=ws)
    sync()
    assert abi.workspace_status(ws) == abi.OK


def test_sequence_index_outside_the_batch_is_reported():
    ctx = [900, 800]
    ent, pool, ring, q, pos, idx, cnt = _fp8_attend_setup(43, ctx, 4, 64)
    seq = torch.tensor([0, 2], dtype=torch.int32, device=DEV)  # batch is 2: sequence 2 does not exist
    call = abi.AttendCall(True, q, pos, pool, 128, ring, 1 / 24, 4, max(ctx), 2, idx=idx, cnt=cnt, seq=seq)
    o, _ = call()
    sync()
    assert call.status() == abi.ERR_INVALID_ARG
    assert torch.all(o[1] == 0)  # the query's item list is empty


# ------------------------------------------------------------------ query / KV RMSNorm and partial RoPE (report §2.3.3)

NORM_EPS, ROPE_BASE = 1e-6, 10000.0


@pytest.mark.parametrize("m,n", [(4, 1024 + 3), (128, 3 * 128 + 5)])
def test_compress_dense_norm_rope_into_kv_pool(m, n):
    D, B = 576, 2
    s = synth.Synth(61, DEV)
    k = s.normal("k", (B, n, D), dtype=torch.bfloat16)
    g = s.normal("g", (B, n, D), dtype=torch.bfloat16)
    bias = s.normal("bias", (m, D), 0.1)
    gain = s.uniform("gain", (D,), 0.5, 1.5)
    pool = abi.make_pool(abi.FMT_KV_POOL_FP8, B, n // m, D, page_entries=128, device=DEV)
    abi.csa_compress(pool, bias, m, k=k, g=g, norm=gain, norm_eps=NORM_EPS, rope_base=ROPE_BASE)
    sync()
    for b in range(B):
        want = csa.prep_entries(csa.compress(f64(k[b]), f64(g[b]), f64(bias), m), m, f64(gain), NORM_EPS, ROPE_BASE)
        got = codecs.kv_entry_decode(*read_kv_pool(pool, b, n // m))
        amax = np.abs(want[:, :512]).max(1, keepdims=True)
        assert np.all(np.abs(got[:, :512] - want[:, :512]) <= 2.0 ** -4 * np.abs(want[:, :512]) + amax * 2e-5)
        rmax = np.abs(want[:, 512:]).max(1, keepdims=True)
        assert np.all(np.abs(got[:, 512:] - want[:, 512:]) <= 2.0 ** -8 * np.abs(want[:, 512:]) + 2e-5 * rmax)


@pytest.mark.parametrize("m", [4, 128])
def test_compress_append_norm_rope(m):
    D, B, R = 576, 3, 128
    s = synth.Synth(62, DEV)
    L = [131, 139, 140] if m == 4 else [383, 511, 389]  # the first two complete a block
    ring = s.normal("ring", (B, R, D), dtype=torch.bfloat16)
    tail = s.normal("tail", (B, m, D))
    bias = s.normal("bias", (m, D), 0.1)
    gain = s.uniform("gain", (D,), 0.5, 1.5)
    k_new = s.normal("k_new", (B, D), dtype=torch.bfloat16)
    g_new = s.normal("g_new", (B, D))
    cap = max(L) // m + 1
    out = torch.full((B, cap, D), float("nan"), device=DEV)
    ring0, tail0 = ring.clone(), tail.clone()
    seq_len = torch.tensor(L, dtype=torch.int32, device=DEV)
    abi.csa_compress(abi.dense_store(out), bias, m, seq_len=seq_len, k_new=k_new, g_new=g_new, ring=ring,
                     tail_gate=tail, norm=gain, norm_eps=NORM_EPS, rope_base=ROPE_BASE)
    sync()
    for b in range(B):
        Lb = L[b]
        j = (Lb + 1) // m - 1
        if (Lb + 1) % m != 0:
            assert torch.isnan(out[b]).all()
            continue
        p = np.arange(Lb + 1 - m, Lb + 1)
        kb = f64(ring0[b])[p % R]
        kb[-1] = f64(k_new[b])
        gb = f64(tail0[b])[p % m]
        gb[-1] = f64(g_new[b])
        want = csa.prep_entries(csa.compress(kb, gb, f64(bias), m), m, f64(gain), NORM_EPS, ROPE_BASE, first=j)[0]
        got = f64(out[b, j])
        assert np.abs(got - want).max() <= 1e-5 * np.abs(want).max(), b


@pytest.mark.parametrize("sparse,ctx,out_dtype,sink,qn,wn", [
    (True, [2800, 1203, 130], torch.float32, False, True, True),      # cluster merge (4-5 splits)
    (False, [20000, 9000], torch.bfloat16, True, True, True),         # 41 splits: combine kernel
    (True, list(range(150, 150 + 7 * 190, 7)), torch.bfloat16, False, True, True),  # one split per query
    (False, [2800, 64, 0], torch.float32, False, False, False),       # RoPE alone
    (True, [1048576 + 77, 70000], torch.float32, False, True, True),  # positions past 1M
])
def test_attend_norm_rope_tensor_core(sparse, ctx, out_dtype, sink, qn, wn):
    m, k = 4, 512
    if max(ctx) > 100000:
        # sparse queries past 1M: the selected blocks sit in the first pages of a
        # small pool, and the page table is widened (to page 0) to cover 1M positions
        ent, pool, ring, q, pos, idx, cnt = _fp8_attend_setup(71, [4000] * len(ctx), m, k)
        pos = torch.tensor(ctx, dtype=torch.int32, device=DEV)
        wide = torch.zeros((len(ctx), (max(ctx) + 1) // m // 128 + 1), dtype=torch.int32, device=DEV)
        wide[:, : pool.page_table.shape[1]] = pool.page_table
        pool.page_table = wide
    else:
        ent, pool, ring, q, pos, idx, cnt = _fp8_attend_setup(71, ctx, m, k)
    s = synth.Synth(72, DEV)
    qg = s.uniform("qg", (576,), 0.5, 1.5) if qn else None
    wg = s.uniform("wg", (576,), 0.5, 1.5) if wn else None
    sk = s.normal("sink", (64,)) * 2 + 1 if sink else None
    call = abi.AttendCall(sparse, q, pos, pool, 128, ring, 1 / 24, m, int(pos.max()), len(ctx), idx=idx, cnt=cnt,
                          out_dtype=out_dtype, sink=sk, q_norm=qg, win_norm=wg, norm_eps=NORM_EPS,
                          rope_base=ROPE_BASE)
    o, lse = call()
    sync()
    assert call.status() == 0
    entn = ent.cpu().numpy()
    ringn = f64(ring)
    worst = 0.0
    for b, t in enumerate(ctx):
        nc = min((t + 1) // m, ent.shape[1])
        rows = idx[b, : int(cnt[b])].cpu().numpy() if sparse else np.arange(nc)
        X = codecs.kv_entry_decode(*codecs.kv_entry_encode(entn[b, rows])) if len(rows) else np.zeros((0, 576))
        wp = csa.window_positions(t, 128)
        wo, wl = csa.attend_one_rope(f64(q[b]), t, X, None, ringn[b, wp % 128], wp, 1 / 24,
                                     None if qg is None else f64(qg), None if wg is None else f64(wg), NORM_EPS,
                                     ROPE_BASE, None if sk is None else f64(sk))
        worst = max(worst, max_abs_rel(f64(o[b]), wo))
        assert np.allclose(f64(lse[b]), wl, atol=2e-2)
    print("max-abs-rel", worst)
    assert worst <= 2e-2


def test_attend_plans_cover_every_merge():
    """The attention cases above run every way of merging a query's splits:
    one split (many queries), a cluster merge inside the kernel (a few
    queries, a short item list), and the combine kernel (few queries, long
    dense lists: more splits than a cluster holds)."""
    cases = {0: (True, list(range(150, 150 + 7 * 190, 7))), 1: (True, [2800, 1203, 130]), 2: (False, [20000, 9000])}
    for merge, (sparse, ctx) in cases.items():
        ent, pool, ring, q, pos, idx, cnt = _fp8_attend_setup(31, ctx, 4, 512)
        call = abi.AttendCall(sparse, q, pos, pool, 128, ring, 1 / 24, 4, max(ctx), len(ctx), idx=idx, cnt=cnt)
        assert call.plan()[1] == merge, (merge, call.plan())
