"""The 8-layer hybrid decode stack at 1,048,576 tokens of context, batch 4:
layers 0-1 HCA (m' = 128), then CSA (m = 4, top-k 1024, FP4 indexer) and HCA
alternating, replayed from one CUDA graph as benchmarked.  Sampled sequences
are recomputed layer by layer by the oracle from the same synthetic state.

The tails are chosen so that, in this step, sequence 0 completes an HCA block
and a CSA block, and sequence 3 completes a CSA block.
"""
import numpy as np
import pytest
import torch

from long_context_sparse_21_b300 import abi, decode
from oracle import codecs

from helpers import (f64, max_abs_rel, oracle_decode_step, read_kv_pool, recall_vs_f32, score_error_bound,
                     selection_valid)

pytestmark = pytest.mark.gpu

CTX = [1048576 + t for t in (127, 37, 74, 3)]
SAMPLES = [0, 3]


@pytest.fixture(scope="module")
def stack():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    abi.lib()
    st = decode.HybridStack(4, CTX, seed=5, keep_sources=SAMPLES)
    st.capture()
    st.replay()
    torch.cuda.synchronize()
    return st


def test_layer_order(stack):
    assert stack.kinds == ["hca", "hca", "csa", "hca", "csa", "hca", "csa", "hca"]
    assert [layer.m for layer in stack.layers] == [128, 128, 4, 128, 4, 128, 4, 128]
    assert all(layer.index_fmt == abi.FMT_INDEX_POOL_E2M1 for layer in stack.layers if layer.kind == "csa")


@pytest.mark.parametrize("li", range(8))
def test_layer_matches_oracle(stack, li):
    layer = stack.layers[li]
    assert layer.attend.status() == abi.OK
    if layer.kind == "csa":
        assert layer.index.status() == abi.OK
    for b in SAMPLES:
        ref = oracle_decode_step(layer, b)
        L = layer.ctx[b]
        same = True
        if layer.kind == "csa":
            sel = layer.index.idx[b].cpu().numpy()
            cnt = int(layer.index.cnt[b])
            s = ref["scores"]
            err = score_error_bound(ref["q_idx"], f64(layer.inputs["w"][b]), ref["keys"],
                                    bf16_scores=layer.score_dtype == abi.BF16)
            ok, why = selection_valid(sel, cnt, s, layer.top_k, err)
            assert ok, (li, b, why)
            same = cnt == ref["cnt"] and np.array_equal(sel[:cnt], ref["idx"][:cnt])
            if not same:  # a valid selection that differs near a tie: attend over it
                ref = oracle_decode_step(layer, b, selection=sel[:cnt])
                same = True
            rec = recall_vs_f32(layer, b, ref, sel, cnt)
            print(f"layer {li} seq {b}: FP4-indexer recall vs float32 selection {rec:.4f}")
            # measured 0.80-0.83 on these keys: the gate sits just below, so a regression shows
            assert rec > 0.75
        if ref["comp_new"] is not None:
            j = (L + 1) // layer.m - 1
            got = codecs.kv_entry_decode(*[x[j:j + 1] for x in read_kv_pool(layer.kv, b, j + 1)])[0]
            want = ref["comp_new"]
            amax = np.abs(want[:512]).max()
            assert np.all(np.abs(got[:512] - want[:512]) <= 2.0 ** -4 * np.abs(want[:512]) + amax * 1e-5)
        if same:
            err = max_abs_rel(f64(layer.attend.out[b]), ref["o"])
            print(f"layer {li} seq {b}: max-abs-rel {err:.2e}")
            assert err <= 2e-2, (li, b, err)
