"""A decode step through the Flash model's 43 attention layers (report §4.2.1:
the first two layers pure sliding-window attention, then CSA and HCA
alternating; CSA m = 4 with top-k 512 and an FP4 lightning indexer, HCA
m' = 128; 64 query heads, 512 + 64 dims; window 128), with query / KV RMSNorm
and partial RoPE (report §2.3.3), replayed from one CUDA graph.  Contexts of
64K + tails keep the oracle's work small; sequence 0 completes an HCA block
and a CSA block in the step.  Layers of every kind are recomputed by the
oracle on the sampled sequences."""
import numpy as np
import pytest
import torch

from long_context_sparse_21_b300 import abi, decode

from helpers import f64, max_abs_rel, oracle_decode_step, score_error_bound, selection_valid

pytestmark = pytest.mark.gpu

CTX = [65536 + t for t in (127, 37)]
SAMPLES = [0, 1]
CHECK = [0, 1, 2, 3, 40, 41, 42]


@pytest.fixture(scope="module")
def stack():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    abi.lib()
    st = decode.HybridStack(2, CTX, seed=9, kinds=decode.FLASH_43, top_k=512, keep_sources=SAMPLES, norm_rope=True)
    st.capture()
    st.replay()
    torch.cuda.synchronize()
    return st


def test_layer_plan(stack):
    kinds = stack.kinds
    assert len(kinds) == 43 and kinds[:2] == ["swa", "swa"]
    assert kinds[2::2] == ["csa"] * 21 and kinds[3::2] == ["hca"] * 20
    assert all(layer.top_k == 512 for layer in stack.layers if layer.kind == "csa")


@pytest.mark.parametrize("li", CHECK)
def test_flash_layer_matches_oracle(stack, li):
    layer = stack.layers[li]
    assert layer.attend.status() == abi.OK
    for b in SAMPLES:
        ref = oracle_decode_step(layer, b)
        if layer.kind == "csa":
            assert layer.index.status() == abi.OK
            sel = layer.index.idx[b].cpu().numpy()
            cnt = int(layer.index.cnt[b])
            err = score_error_bound(ref["q_idx"], f64(layer.inputs["w"][b]), ref["keys"],
                                    bf16_scores=layer.score_dtype == abi.BF16)
            ok, why = selection_valid(sel, cnt, ref["scores"], layer.top_k, err)
            assert ok, (li, b, why)
            if not (cnt == ref["cnt"] and np.array_equal(sel[:cnt], ref["idx"][:cnt])):
                ref = oracle_decode_step(layer, b, selection=sel[:cnt])
        e = max_abs_rel(f64(layer.attend.out[b]), ref["o"])
        print(f"layer {li} ({layer.kind}) seq {b}: max-abs-rel {e:.2e}")
        assert e <= 2e-2, (li, b, e)
