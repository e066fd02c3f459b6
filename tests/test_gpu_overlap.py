"""Overlapping compression (CSA's form, DeepSeek-V4 report §2.3.1: two KV sets
C_a, C_b with weights Z_a, Z_b; §2.3.2: HCA compresses without overlap)
through the C ABI, against the oracle's compress_overlap: the dense mode over
whole sequences with a ragged tail, and the decode append driven token by
token from an empty state, which must store the same entries as the dense
pooling of the whole sequence.  Bar: max-abs error <= 2e-6 x max |entry| for
the float32 store (float32 softmax vs float64), one FP8/BF16 rounding for the
KV pool."""
import numpy as np
import pytest
import torch

from long_context_sparse_21_b300 import abi, synth
from oracle import codecs, csa

from helpers import f64, read_kv_pool

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True, scope="module")
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    abi.lib()


def _streams(s, B, n, m, D, dtype):
    return (s.normal("ka", (B, n, D), dtype=dtype), s.normal("ga", (B, n, D), 2.0, dtype=dtype),
            s.normal("ba", (m, D), 0.1), s.normal("kb", (B, n, D), dtype=dtype),
            s.normal("gb", (B, n, D), 2.0, dtype=dtype), s.normal("bb", (m, D), 0.1))


@pytest.mark.parametrize("m,D,n,dtype", [(4, 576, 1024 + 3, torch.bfloat16), (4, 192, 2048 + 1, torch.float32),
                                         (16, 128, 512 + 15, torch.float32), (1, 64, 33, torch.float32)])
def test_compress_dense_ab(m, D, n, dtype):
    B = 2
    s = synth.Synth(71, DEV)
    ka, ga, ba, kb, gb, bb = _streams(s, B, n, m, D, dtype)
    out = torch.full((B, n // m, D), float("nan"), device=DEV)
    abi.csa_compress(abi.dense_store(out), ba, m, k=ka, g=ga, bias_b=bb, k_b=kb, g_b=gb)
    torch.cuda.synchronize()
    for b in range(B):
        want = csa.compress_overlap(f64(ka[b]), f64(ga[b]), f64(ba), f64(kb[b]), f64(gb[b]), f64(bb), m)
        got = f64(out[b])
        assert np.abs(got - want).max() <= 2e-6 * np.abs(want).max(), b


def test_compress_dense_ab_into_kv_pool():
    m, D, n, B = 4, 576, 4 * 300 + 2, 2
    s = synth.Synth(72, DEV)
    ka, ga, ba, kb, gb, bb = _streams(s, B, n, m, D, torch.bfloat16)
    pool = abi.make_pool(abi.FMT_KV_POOL_FP8, B, n // m + 1, 576, page_entries=128, device=DEV)
    abi.csa_compress(pool, ba, m, k=ka, g=ga, bias_b=bb, k_b=kb, g_b=gb)
    torch.cuda.synchronize()
    for b in range(B):
        want = csa.compress_overlap(f64(ka[b]), f64(ga[b]), f64(ba), f64(kb[b]), f64(gb[b]), f64(bb), m)
        got = codecs.kv_entry_decode(*read_kv_pool(pool, b, n // m))
        amax = np.abs(want[:, :512]).max(1, keepdims=True)
        assert np.all(np.abs(got[:, :512] - want[:, :512]) <= 2.0 ** -3 * np.abs(want[:, :512]) + amax / 448 * 2.0 ** -8)
        rmax = np.abs(want[:, 512:]).max(1, keepdims=True)
        assert np.all(np.abs(got[:, 512:] - want[:, 512:]) <= 2.0 ** -7 * np.abs(want[:, 512:]) + 1e-5 * rmax)


@pytest.mark.parametrize("m,n", [(4, 4 * 17 + 3), (16, 16 * 5 + 7)])
def test_compress_append_ab_token_by_token(m, n):
    """From an empty state, append every token of three sequences (the a
    stream's raw keys go to the window ring, the b stream's to its two-block
    tail); the stored entries equal the dense overlapping pooling of the whole
    sequences, and a partial block leaves its entry unwritten."""
    B, D, R = 3, 576, 2 * m
    s = synth.Synth(73, DEV)
    ka, ga, ba, kb, gb, bb = _streams(s, B, n, m, D, torch.bfloat16)
    ga, gb = ga.float(), gb.float()
    ring = torch.zeros((B, R, D), dtype=torch.bfloat16, device=DEV)
    tail = torch.zeros((B, m, D), device=DEV)
    # the tails start as NaN: nothing the first entry pools may come from them
    tail_b = torch.full((B, 2 * m, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    tail_gate_b = torch.full((B, 2 * m, D), float("nan"), device=DEV)
    out = torch.full((B, n // m + 1, D), float("nan"), device=DEV)
    seq_len = torch.zeros(B, dtype=torch.int32, device=DEV)
    ws = abi.compress_workspace(B, D, DEV)
    for L in range(n):
        seq_len.fill_(L)
        abi.csa_compress(abi.dense_store(out), ba, m, seq_len=seq_len, k_new=ka[:, L].contiguous(),
                         g_new=ga[:, L].contiguous(), ring=ring, tail_gate=tail, workspace=ws, bias_b=bb,
                         k_new_b=kb[:, L].contiguous(), g_new_b=gb[:, L].contiguous(), tail_b=tail_b,
                         tail_gate_b=tail_gate_b)
    torch.cuda.synchronize()
    assert abi.workspace_status(ws) == abi.OK
    for b in range(B):
        want = csa.compress_overlap(f64(ka[b]), f64(ga[b]), f64(ba), f64(kb[b]), f64(gb[b]), f64(bb), m)
        got = f64(out[b, : n // m])
        assert np.abs(got - want).max() <= 2e-6 * np.abs(want).max(), b
        assert torch.isnan(out[b, n // m]).all()
        # the b tails hold the last 2m tokens of the b stream at slot p % 2m
        p = np.arange(n - 2 * m, n)
        assert torch.equal(tail_b[b, p % (2 * m)], kb[b, p])
        assert torch.equal(tail_gate_b[b, p % (2 * m)], gb[b, p])
