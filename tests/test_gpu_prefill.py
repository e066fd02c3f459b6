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

from helpers import f64, max_abs_rel, selection_valid

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
