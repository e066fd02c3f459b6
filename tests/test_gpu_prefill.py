"""The float32 CSA prefill chain (batch 1, 2048 tokens, m = 4, top-k 64,
window 128, 16 query heads of dim 192, indexer 4 heads x 64): compressor on
both streams -> lightning indexer -> top-k -> attention, every step through the
C ABI, against the oracle's whole-chain restatement on the same inputs.

The chain's top-k is compared as sets.  The compressor's float32 exp may move
a compressed key by an ulp relative to the float64 oracle, which can swap
blocks whose scores tie to within that ulp, so a row whose set differs is
checked for being a valid top-k of the oracle's scores, and its attention is
compared against the oracle's attention over the kernel's selection."""
import math

import numpy as np
import pytest
import torch

from long_context_sparse_21_b300 import abi, synth
from oracle import csa

from helpers import f64, max_abs_rel, score_error_bound, selection_valid

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    abi.lib()


def test_csa_prefill_f32_chain():
    n, m, D, dI, k, W = 2048, 4, 192, 64, 64, 128
    scale = 1.0 / math.sqrt(D)
    x = synth.csa_prefill_f32(seed=3, device="cuda")
    comp = torch.full((1, n // m, D), float("nan"), device="cuda")
    kI = torch.full((1, n // m, dI), float("nan"), device="cuda")
    abi.csa_compress(abi.dense_store(comp), x["bias"], m, k=x["k"][None], g=x["g"][None])
    abi.csa_compress(abi.dense_store(kI), x["bias_idx"], m, k=x["k_idx"][None], g=x["g_idx"][None])
    pos = torch.arange(n, dtype=torch.int32, device="cuda")
    seq = torch.zeros(n, dtype=torch.int32, device="cuda")
    index = abi.IndexCall(x["q_idx"], x["w"], pos, abi.dense_store(kI), k, m, n - 1, 1, seq=seq, w_shared=True)
    idx, cnt = index()
    attend = abi.AttendCall(True, x["q"], pos, abi.dense_store(comp), W, x["k"][None], scale, m, n - 1, 1,
                            idx=idx, cnt=cnt, seq=seq)
    out, lse = attend()
    torch.cuda.synchronize()
    assert index.status() == abi.OK and attend.status() == abi.OK

    h = {key: f64(v) for key, v in x.items()}
    ref = csa.csa_prefill(h["k"], h["g"], h["bias"], h["k_idx"], h["g_idx"], h["bias_idx"], h["q_idx"], h["w"],
                          h["q"], m, k, W, scale, score="f32")
    # compressor outputs
    for got, want in [(f64(comp[0]), ref["comp"]), (f64(kI[0]), ref["kI"])]:
        assert np.abs(got - want).max() <= 2e-6 * np.abs(want).max()
    idx_h, cnt_h, o = idx.cpu().numpy(), cnt.cpu().numpy(), f64(out)
    kI32 = ref["kI"].astype(np.float32)
    same_rows, worst = 0, 0.0
    for t in range(n):
        nc = (t + 1) // m
        assert cnt_h[t] == ref["cnt"][t]
        if np.array_equal(idx_h[t], ref["idx"][t]):
            same_rows += 1
            want = ref["o"][t]
        else:
            s = csa.index_scores_f32(np.asarray(h["q_idx"][t], np.float32), np.asarray(h["w"], np.float32), kI32[:nc])
            ok, why = selection_valid(idx_h[t], int(cnt_h[t]), s.astype(np.float64), k,
                                      1e-6 * float(np.abs(s).max()))
            assert ok, (t, why)
            want, _ = csa.csa_attend(h["q"][t], t, idx_h[t], int(cnt_h[t]), ref["comp"], h["k"], W, scale)
        err = max_abs_rel(o[t], want)
        worst = max(worst, err)
        assert err <= 1e-4, (t, err)
    print(f"rows with the oracle's exact top-k set: {same_rows}/{n}; worst max-abs-rel {worst:.2e}")
    assert same_rows >= n - 16


# ------------------------------------------------------------------ BF16 / FP8 prefill (tensor-core path)

def _check_prefill(pf, rows):
    """Oracle restatement for sampled query rows of a CsaPrefill run.

    1. Compressor: every stored entry (FP8 content + scale + BF16 RoPE) and
       every stored indexer key (BF16) equals the oracle's float64 pooling up
       to one rounding of the storage format.  (The kernel pools in float32,
       so near a rounding boundary it may pick the neighbouring code.)
    2. Indexer + top-k: scores of the stored keys; the kernel's selection is a
       valid top-k within the BF16-score rounding.
    3. Attention over that selection, on the stored entries (the cache's
       dequantized values, so the comparison measures the attention kernel)."""
    from oracle import codecs
    from helpers import read_index_bf16_pool, read_kv_pool
    n_ent = pf.n // pf.m
    k = f64(pf.k)
    if pf.overlap_ab:
        comp = csa.compress_overlap(k, f64(pf.g), f64(pf.bias), f64(pf.k_b), f64(pf.g_b), f64(pf.bias_b), pf.m)
    else:
        comp = csa.compress(k, f64(pf.g), f64(pf.bias), pf.m)
    comp_st = codecs.kv_entry_decode(*read_kv_pool(pf.kv, 0, n_ent))
    amax = np.abs(comp[:, :512]).max(1, keepdims=True)
    assert np.all(np.abs(comp_st[:, :512] - comp[:, :512]) <= 2.0 ** -3 * np.abs(comp[:, :512]) + amax / 448 * 2.0 ** -8)
    rmax = np.abs(comp[:, 512:]).max(1, keepdims=True)  # float32 pooling: cancellation near zero
    assert np.all(np.abs(comp_st[:, 512:] - comp[:, 512:]) <= 2.0 ** -7 * np.abs(comp[:, 512:]) + 1e-5 * rmax)
    if pf.overlap_ab:
        kI = csa.compress_overlap(f64(pf.k_idx), f64(pf.g_idx), f64(pf.bias_idx), f64(pf.k_idx_b),
                                  f64(pf.g_idx_b), f64(pf.bias_idx_b), pf.m)
    else:
        kI = csa.compress(f64(pf.k_idx), f64(pf.g_idx), f64(pf.bias_idx), pf.m)
    kI_st = codecs.bf16_decode(read_index_bf16_pool(pf.ki, 0, n_ent)).astype(np.float64)
    assert np.all(np.abs(kI_st - kI) <= 2.0 ** -7 * np.abs(kI) + 1e-5 * np.abs(kI).max(1, keepdims=True))
    idx, cnt, out = pf.idx.cpu().numpy(), pf.cnt.cpu().numpy(), pf.out
    same, worst = 0, 0.0
    for t in rows:
        nc = (t + 1) // pf.m
        s = csa.index_scores(f64(pf.q_idx[t]), f64(pf.w[t]), kI_st[:nc])
        s_err = score_error_bound(f64(pf.q_idx[t]), f64(pf.w[t]), kI_st[:nc], bf16_scores=True)
        ok, why = selection_valid(idx[t], int(cnt[t]), s, pf.top_k, s_err)
        assert ok, (t, why)
        want_idx, wc = csa.topk(s, nc, pf.top_k)
        same += int(wc == cnt[t] and np.array_equal(idx[t][:wc], want_idx[:wc]))
        o, _ = csa.csa_attend(f64(pf.q[t]), t, idx[t], int(cnt[t]), comp_st, k, pf.W, pf.scale)
        err = max_abs_rel(f64(out[t]), o)
        worst = max(worst, err)
        assert err <= 2e-2, (t, err)
    print(f"rows with the oracle's exact top-k set: {same}/{len(rows)}; worst max-abs-rel {worst:.2e}")


def test_csa_prefill_bf16_16k():
    """16,384 tokens (4096 compressed entries) in chunks of 4096 queries, top-k
    1024 (selection active from t = 4099 on), the tensor-core indexer with four
    queries per CTA, BF16 index scores, FP8 KV cache, dense window source."""
    from long_context_sparse_21_b300 import prefill
    pf = prefill.CsaPrefill(n=16384, seed=4, chunk=4096)
    pf.run()
    torch.cuda.synchronize()
    assert pf.status() == abi.OK
    rng = np.random.default_rng(0)
    rows = sorted(set([0, 2, 3, 4, 127, 128, 4095, 4096, 4099, 4100, 8191, 8192, 12287, 16383] +
                      rng.integers(0, 16384, 12).tolist()))
    _check_prefill(pf, rows)


def test_csa_prefill_bf16_overlapping_compression():
    """The 16,384-token prefill with overlapping compression (report §2.3.1)
    in both compressors: entry j pools the a stream over block j and the b
    stream over block j - 1."""
    from long_context_sparse_21_b300 import prefill
    pf = prefill.CsaPrefill(n=16384, seed=8, chunk=4096, overlap_ab=True)
    pf.run()
    torch.cuda.synchronize()
    assert pf.status() == abi.OK
    _check_prefill(pf, [0, 3, 4, 7, 4099, 8191, 12000, 16383])


def test_csa_prefill_bf16_full_size_sampled():
    """The full workload: 131,072 tokens (32,768 entries), chunks of 4096, top-k
    1024, 1% outlier tokens x8, as benchmarked; sampled rows of every region."""
    from long_context_sparse_21_b300 import prefill
    pf = prefill.CsaPrefill(n=131072, seed=5, chunk=4096)
    pf.run()
    torch.cuda.synchronize()
    assert pf.status() == abi.OK
    rows = [5, 4096, 65535, 65536, 100000, 126975, 126976, 131071]
    _check_prefill(pf, rows)
