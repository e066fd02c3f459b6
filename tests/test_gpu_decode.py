"""Whole decode steps (compress-append -> index -> top-k -> attention) against
the oracle: small cases that exercise block completion, and the full-size
workloads in the launch configuration the benchmark times (CUDA graph), on
sampled sequences the oracle recomputes one by one."""
import numpy as np
import pytest
import torch

from long_context_sparse_21_b300 import abi, decode
from oracle import codecs

from helpers import (f64, max_abs_rel, oracle_decode_step, read_index_bf16_pool, read_kv_pool, recall_vs_f32,
                     score_error_bound, selection_valid)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    abi.lib()


def check_layer(layer, samples, graph=False, tol=2e-2):
    if graph:
        layer.capture()
        out = layer.replay()
    else:
        out = layer.step()
    torch.cuda.synchronize()
    assert layer.attend.status() == 0
    if layer.kind == "csa":
        assert layer.index.status() == 0
    worst = 0.0
    for b in samples:
        ref = oracle_decode_step(layer, b)
        L = layer.ctx[b]
        if layer.kind == "csa":
            sel = layer.index.idx[b].cpu().numpy()
            cnt = int(layer.index.cnt[b])
            rec = recall_vs_f32(layer, b, ref, sel, cnt)
            print(f"seq {b}: indexer recall vs float32 selection {rec:.4f}")
            # measured 0.98-1.000 with BF16 keys (report section 5.2.1 reports 99.7%);
            # the gate sits below that, so a regression of the selector shows
            assert rec >= 0.95, (b, rec)
            s = ref["scores"]
            err = score_error_bound(ref["q_idx"], f64(layer.inputs["w"][b]), ref["keys"],
                                    bf16_scores=layer.score_dtype == abi.BF16)
            ok, why = selection_valid(sel, cnt, s, layer.top_k, err)
            assert ok, (b, why)
            same = cnt == ref["cnt"] and np.array_equal(sel[:cnt], ref["idx"][:cnt])
            if not same:  # a valid selection that differs near a tie: attend over it
                ref = oracle_decode_step(layer, b, selection=sel[:cnt])
                same = True
        else:
            same = True
        if ref["comp_new"] is not None:
            j = (L + 1) // layer.m - 1
            got = codecs.kv_entry_decode(*[x[j:j + 1] for x in read_kv_pool(layer.kv, b, j + 1)])[0]
            want = ref["comp_new"]
            amax = np.abs(want[:512]).max()
            assert np.all(np.abs(got[:512] - want[:512]) <= 2.0 ** -4 * np.abs(want[:512]) + amax * 1e-5)
            rmax = np.abs(want[512:]).max()
            assert np.all(np.abs(got[512:] - want[512:]) <= 2.0 ** -8 * np.abs(want[512:]) + rmax * 1e-5)
            if layer.kind == "csa":
                gi = codecs.bf16_decode(read_index_bf16_pool(layer.ki, b, j + 1)[j])
                assert np.all(np.abs(gi - ref["kI_new"]) <= 2.0 ** -8 * np.abs(ref["kI_new"]) + 1e-6)
        if same:
            err = max_abs_rel(f64(out[b]), ref["o"])
            worst = max(worst, err)
            assert err <= tol, (b, err)
    return worst


def test_csa_decode_step_small_with_block_completion():
    layer = decode.DecodeLayer("csa", 3, [1023, 2001, 4095], seed=41, top_k=64, page_entries=128,
                               keep_sources=range(3))
    print("worst max-abs-rel", check_layer(layer, range(3)))


def test_hca_decode_step_small_with_block_completion():
    layer = decode.DecodeLayer("hca", 3, [128 * 9 - 1, 128 * 20 + 5, 300], seed=42, page_entries=128,
                               keep_sources=range(3))
    print("worst max-abs-rel", check_layer(layer, range(3)))


@pytest.mark.parametrize("score_dtype", [abi.F32, abi.BF16])
def test_csa_decode_full_size_graph(score_dtype):
    """CSA decode: batch 32, contexts 65535 + (b mod 4) raw tokens (16384
    visible compressed entries) per sequence as benchmarked, so sequence 0
    completes a block in the step; top-k 512, BF16 indexer, float32 or BF16
    index scores (the benchmark uses BF16 scores), replayed from a graph."""
    samples = [0, 13, 31]
    ctx = [65535 + (b % 4) for b in range(32)]
    layer = decode.DecodeLayer("csa", 32, ctx, seed=1, top_k=512, keep_sources=samples, score_dtype=score_dtype)
    print("worst max-abs-rel", check_layer(layer, samples, graph=True))


def test_hca_decode_full_size_graph():
    """HCA decode: batch 16, 1,048,576 + tail raw tokens (8192 entries), one
    sequence completing a block in the step."""
    tails = list(np.random.Generator(np.random.Philox(7)).integers(0, 128, 16))
    tails[5] = 127
    ctx = [1048576 + int(t) for t in tails]
    samples = [0, 5, 15]
    layer = decode.DecodeLayer("hca", 16, ctx, seed=2, keep_sources=samples)
    print("worst max-abs-rel", check_layer(layer, samples, graph=True))


def test_csa_decode_norm_rope_full_size_graph():
    """The CSA decode workload with query / KV RMSNorm and partial RoPE (report
    §2.3.3) fused in: the append normalizes and rotates the completed entry
    before storing it (sequence 0 completes one), the attention normalizes and
    rotates the query and the window rows and turns the output back."""
    samples = [0, 13, 31]
    ctx = [65535 + (b % 4) for b in range(32)]
    layer = decode.DecodeLayer("csa", 32, ctx, seed=6, top_k=512, keep_sources=samples, score_dtype=abi.BF16,
                               norm_rope=True)
    print("worst max-abs-rel", check_layer(layer, samples, graph=True))


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_decode_small_norm_rope(kind):
    ctx = [1023, 2001, 4095] if kind == "csa" else [128 * 9 - 1, 128 * 20 + 5, 300]
    layer = decode.DecodeLayer(kind, 3, ctx, seed=43, top_k=64, page_entries=128, keep_sources=range(3),
                               norm_rope=True)
    print("worst max-abs-rel", check_layer(layer, range(3)))


@pytest.mark.parametrize("norm_rope", [False, True])
def test_csa_decode_overlapping_compression_small(norm_rope):
    """Overlapping compression (report §2.3.1) in the decode append of both
    compressors: a completed entry also pools the b stream over the block
    before it, read from the two-block b tail; sequence 3 completes block 0,
    which has no previous block."""
    layer = decode.DecodeLayer("csa", 4, [1023, 2001, 4095, 3], seed=44, top_k=64, page_entries=128,
                               keep_sources=range(4), norm_rope=norm_rope, overlap_ab=True)
    print("worst max-abs-rel", check_layer(layer, range(4)))


def test_csa_decode_overlapping_compression_full_size_graph():
    samples = [0, 4, 13, 31]
    ctx = [65535 + (b % 4) for b in range(32)]
    layer = decode.DecodeLayer("csa", 32, ctx, seed=7, top_k=512, keep_sources=samples, score_dtype=abi.BF16,
                               overlap_ab=True)
    print("worst max-abs-rel", check_layer(layer, samples, graph=True))


@pytest.mark.parametrize("norm_rope", [False, True])
def test_window_only_decode_small(norm_rope):
    """Pure sliding-window layers (report §4.2.1): the window append and the
    window-only attention, including contexts shorter than the window."""
    layer = decode.DecodeLayer("swa", 4, [0, 5, 127, 3000], seed=44, keep_sources=range(4), norm_rope=norm_rope)
    assert layer.kv is None
    print("worst max-abs-rel", check_layer(layer, range(4)))
