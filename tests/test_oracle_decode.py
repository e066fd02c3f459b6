"""Pins for the oracle's decode step (``oracle/decode.py``): one step of a
layer, driven by the state cache (window ring, tail gates, indexer-key ring),
must give what the whole-sequence definitions of ``oracle/csa.py`` give at
position t = L on the same raw sequence.  Those definitions are pinned on
their own in ``test_oracle.py``; this file pins the step's bookkeeping: which
raw positions the window holds, which tail slot holds which gate, when a block
completes, and that the completed block's indexer key joins the scored keys.

Each case builds a raw sequence of L + 1 tokens (KV stream and indexer-key
stream, with gate logits), derives the state a cache would hold before the
step, and compares:
  * comp_new with csa.compress over the raw tokens L + 1 - m .. L;
  * kI_new with csa.compress over the indexer stream likewise;
  * scores / idx / cnt with csa.index_scores and csa.topk over every visible
    compressed key, rounded to its storage format (BF16, or FP4 for key and
    query);
  * o and lse with csa.csa_attend / csa.hca_attend at t = L, over the stored
    (FP8 content + BF16 RoPE) entries and the raw window.
The last tests plant a mistake in the step's bookkeeping and check that these
comparisons catch it.  CPU only."""
import numpy as np
import pytest

from oracle import codecs, csa
from oracle import decode as odec

D, DI, H, HI = 576, 128, 3, 4


def _fp4(x):
    c, s = codecs.fp4_block_encode(np.asarray(x, np.float32))
    return codecs.fp4_block_decode(c, s)


def _stored(x):
    """Entries after storage: FP8 content with the per-entry scale, BF16 RoPE."""
    return codecs.kv_entry_decode(*codecs.kv_entry_encode(np.asarray(x, np.float32)))


PREP = dict(q_gain=np.random.default_rng(5).random(D) + 0.5, kv_gain=np.random.default_rng(6).random(D) + 0.5,
            eps=1e-6, rope_base=1e4)
NO_PREP = dict(q_gain=None, kv_gain=None, eps=0.0, rope_base=0.0)


def _case(seed, L, m, W, prep=NO_PREP, ab=False):
    """Raw sequence of L + 1 tokens and the state a cache holds before the
    step that appends token L.  Slots of the state buffers that hold no live
    position are filled with junk, so that reading a wrong slot shows.  With
    query / KV normalization and RoPE the stored entries are the prepared
    ones (csa.prep_entries)."""
    rng = np.random.default_rng(seed)
    n = L + 1
    k = rng.standard_normal((n, D))
    g = rng.standard_normal((n, D)) * 2
    b = rng.standard_normal((m, D)) * 0.1
    ki = rng.standard_normal((n, DI))
    gi = rng.standard_normal((n, DI)) * 2
    bi = rng.standard_normal((m, DI)) * 0.1
    q = rng.standard_normal((H, D))
    qi = rng.standard_normal((HI, DI))
    w = rng.random(HI)
    n_old = L // m
    tail = range(n_old * m, L)  # positions of the uncompressed tail before the step
    junk = lambda shape: rng.standard_normal(shape) * 50  # noqa: E731
    window = junk((W, D))
    for i in range(W):
        p = L - W + i
        if p >= 0:
            window[i] = k[p]
    tail_gate, ring_idx, tail_gate_idx = junk((m, D)), junk((m, DI)), junk((m, DI))
    for p in tail:
        tail_gate[p % m] = g[p]
        ring_idx[p % m] = ki[p]
        tail_gate_idx[p % m] = gi[p]
    overlap = None
    if ab:  # overlapping compression: b streams of both compressors, tails of 2m slots
        kb, gb, bb = rng.standard_normal((n, D)), rng.standard_normal((n, D)) * 2, rng.standard_normal((m, D)) * 0.1
        kib, gib = rng.standard_normal((n, DI)), rng.standard_normal((n, DI)) * 2
        bib = rng.standard_normal((m, DI)) * 0.1
        tb, tgb, tib, tgib = junk((2 * m, D)), junk((2 * m, D)), junk((2 * m, DI)), junk((2 * m, DI))
        for p in range(max(0, n_old * m - m), L):  # the previous block and the current tail
            tb[p % (2 * m)], tgb[p % (2 * m)] = kb[p], gb[p]
            tib[p % (2 * m)], tgib[p % (2 * m)] = kib[p], gib[p]
        overlap = {"kv": (tb, tgb, bb), "idx": (tib, tgib, bib)}
        pooled = csa.compress_overlap(k, g, b, kb, gb, bb, m)
        ki_all = csa.compress_overlap(ki, gi, bi, kib, gib, bib, m)
    else:
        pooled = csa.compress(k, g, b, m)
        ki_all = csa.compress(ki, gi, bi, m)
    comp_all = csa.prep_entries(pooled, m, prep["kv_gain"], prep["eps"], prep["rope_base"])
    entries = np.vstack([comp_all[:n_old], junk((2, D))]).astype(np.float32)  # slots past n_old: junk
    keys_idx = np.vstack([ki_all[:n_old], junk((2, DI))]).astype(np.float32)
    state = dict(entries=entries, window=window, tail_gate=tail_gate, bias=b, q=q, k_new=k[L], g_new=g[L],
                 keys_idx=keys_idx, ring_idx=ring_idx, tail_gate_idx=tail_gate_idx, bias_idx=bi, q_idx=qi, w=w,
                 k_idx_new=ki[L], g_idx_new=gi[L])
    if overlap is not None:
        state["overlap"] = overlap
    seq = dict(k=k, comp_all=comp_all, ki_all=ki_all, q=q, qi=qi, w=w)
    return state, seq


def _check(kind, m, W, L, top_k, fmt, seed=0, prep=NO_PREP, ab=False):
    """Runs the step and returns the list of mismatches against the
    whole-sequence definitions (empty when the step is right)."""
    state, seq = _case(seed, L, m, W, prep, ab)
    if kind == "hca":
        for key in ("keys_idx", "ring_idx", "tail_gate_idx", "bias_idx", "q_idx", "w", "k_idx_new", "g_idx_new"):
            state.pop(key)
    scale = 1 / 24
    got = odec.decode_step(kind, m, W, L, top_k, scale, index_fmt=fmt, **state, **prep)
    bad = []
    nvis = (L + 1) // m
    if (L + 1) % m == 0:
        if got["comp_new"] is None or not np.allclose(got["comp_new"], seq["comp_all"][nvis - 1], rtol=0, atol=1e-12):
            bad.append("comp_new")
    elif got["comp_new"] is not None:
        bad.append("comp_new on a step that completes no block")
    comp = _stored(seq["comp_all"])
    if kind == "csa":
        if (L + 1) % m == 0 and (got["kI_new"] is None or
                                 not np.allclose(got["kI_new"], seq["ki_all"][nvis - 1], rtol=0, atol=1e-12)):
            bad.append("kI_new")
        keys32 = seq["ki_all"][:nvis].astype(np.float32)
        if fmt == "bf16":
            keys, qq = codecs.bf16_round(keys32), seq["qi"]
        else:
            keys, qq = _fp4(keys32), _fp4(seq["qi"])
        s = csa.index_scores(qq, seq["w"], keys)
        idx, cnt = csa.topk(s, nvis, top_k)
        if got["scores"] is None or len(got["scores"]) != nvis or not np.allclose(got["scores"], s, rtol=1e-12,
                                                                                   atol=1e-12):
            bad.append("scores")
        if got["cnt"] != cnt or not np.array_equal(got["idx"], idx):
            bad.append("idx")
        sel = idx[:cnt]
    else:
        sel = np.arange(nvis)
    wpos = csa.window_positions(L, W)
    o, lse = csa.attend_one_rope(seq["q"], L, comp[sel], None, seq["k"][wpos], wpos, scale, prep["q_gain"],
                                 prep["kv_gain"], prep["eps"], prep["rope_base"])
    if prep is NO_PREP:  # the plain path is also the textbook CSA / HCA attention of csa.py
        plain = csa.csa_attend(seq["q"], L, idx, cnt, comp, seq["k"], W, scale) if kind == "csa" else \
            csa.hca_attend(seq["q"], L, m, comp, seq["k"], W, scale)
        assert np.allclose(plain[0], o, atol=1e-12)
    if not (np.allclose(got["o"], o, rtol=0, atol=1e-10) and np.allclose(got["lse"], lse, rtol=0, atol=1e-10)):
        bad.append("attention")
    return bad


CASES = [
    # kind, m, W, L, top_k, fmt.  The window ring also holds the tail's raw
    # tokens (the cache's ring has W = 128 >= m rows), so W >= m - 1.
    ("csa", 4, 16, 39, 3, "bf16"),    # (L+1) % m == 0: completes block 9
    ("csa", 4, 16, 41, 3, "bf16"),    # no completion
    ("csa", 4, 16, 43, 64, "bf16"),   # k >= visible blocks: every block kept
    ("csa", 4, 16, 7, 2, "bf16"),     # L < W, completes block 1
    ("csa", 4, 16, 2, 2, "bf16"),     # L < W, no visible block yet
    ("csa", 4, 16, 47, 4, "fp4"),     # FP4 keys and query, completes
    ("csa", 4, 16, 45, 4, "fp4"),     # FP4, no completion
    ("csa", 4, 128, 130, 5, "bf16"),  # the window of the workloads (W = 128) crossing its ring
    ("hca", 128, 128, 255, 0, "bf16"),  # m = 128: completes block 1
    ("hca", 128, 128, 300, 0, "bf16"),  # m = 128: tail of 44 tokens
    ("hca", 128, 128, 127, 0, "bf16"),  # the first block completes with L < W
    ("hca", 128, 128, 60, 0, "bf16"),  # no visible block: window only
]


@pytest.mark.parametrize("kind,m,W,L,top_k,fmt", CASES)
def test_decode_step_matches_whole_sequence_definitions(kind, m, W, L, top_k, fmt):
    assert _check(kind, m, W, L, top_k, fmt) == []


@pytest.mark.parametrize("kind,m,W,L,top_k,fmt", [CASES[0], CASES[1], CASES[5], CASES[7], CASES[8], CASES[9]])
def test_decode_step_with_norm_and_rope(kind, m, W, L, top_k, fmt):
    """The same pins with query / KV RMSNorm and partial RoPE (report
    §2.3.3): the completed entry is prepared before storage and the step's
    attention equals csa.attend_one_rope over the prepared entries."""
    assert _check(kind, m, W, L, top_k, fmt, prep=PREP) == []


@pytest.mark.parametrize("kind,m", [("csa", 4), ("hca", 128)])
def test_first_token_window_of_one(kind, m):
    """L = 0: no compressed entry is visible and the window holds only the new
    token, so every head's output is that token exactly and lse is its scaled
    logit."""
    rng = np.random.default_rng(7)
    W = 128
    k0 = rng.standard_normal(D)
    q = rng.standard_normal((H, D))
    kw = dict(entries=np.zeros((1, D), np.float32), window=rng.standard_normal((W, D)) * 50,
              tail_gate=rng.standard_normal((m, D)), bias=np.zeros((m, D)), q=q, k_new=k0, g_new=np.zeros(D))
    if kind == "csa":
        kw.update(keys_idx=np.zeros((1, DI), np.float32), ring_idx=np.zeros((m, DI)), tail_gate_idx=np.zeros((m, DI)),
                  bias_idx=np.zeros((m, DI)), q_idx=rng.standard_normal((HI, DI)), w=rng.random(HI),
                  k_idx_new=np.zeros(DI), g_idx_new=np.zeros(DI))
    got = odec.decode_step(kind, m, W, 0, 4, 0.5, **kw)
    assert np.array_equal(got["o"], np.tile(k0, (H, 1)))
    assert np.allclose(got["lse"], 0.5 * q @ k0, rtol=0, atol=1e-12)
    if kind == "csa":
        assert got["cnt"] == 0 and np.all(got["idx"] == -1)


def test_sink_passes_through():
    """A sink logit at -inf leaves the step's output unchanged; a large one
    takes the attention mass (report §2.3.3)."""
    state, _ = _case(3, 39, 4, 16)
    base = odec.decode_step("csa", 4, 16, 39, 3, 1 / 24, **state)
    same = odec.decode_step("csa", 4, 16, 39, 3, 1 / 24, sink=np.full(H, -np.inf), **state)
    assert np.allclose(base["o"], same["o"], atol=1e-14)
    big = odec.decode_step("csa", 4, 16, 39, 3, 1 / 24, sink=np.full(H, 300.0), **state)
    assert np.all(np.abs(big["o"]) < 1e-60)


# overlapping compression (report §2.3.1; CSA only): the completed entry also
# pools the b stream over the block before it, from the two-block b tail
AB_CASES = [
    ("csa", 4, 16, 39, 3, "bf16"),    # completes block 9: pools block 8 of the b stream
    ("csa", 4, 16, 3, 2, "bf16"),     # completes block 0: no previous block
    ("csa", 4, 16, 7, 2, "bf16"),     # completes block 1: previous block 0
    ("csa", 4, 16, 41, 3, "bf16"),    # no completion
    ("csa", 4, 16, 47, 4, "fp4"),
    ("csa", 16, 128, 16 * 9 - 1, 4, "bf16"),
]


@pytest.mark.parametrize("kind,m,W,L,top_k,fmt", AB_CASES)
def test_decode_step_with_overlapping_compression(kind, m, W, L, top_k, fmt):
    assert _check(kind, m, W, L, top_k, fmt, ab=True) == []
    assert _check(kind, m, W, L, top_k, fmt, prep=PREP, ab=True) == []


AB_MUTATIONS = {
    "b slot p mod m": ("b_slot", lambda p, m: p % m),
    "b slot one block late": ("b_slot", lambda p, m: (p + m) % (2 * m)),
    "previous block dropped": ("previous_block", lambda L, m, kb, gb: None),
}


@pytest.mark.parametrize("name", sorted(AB_MUTATIONS))
def test_planted_overlap_mistakes_are_caught(monkeypatch, name):
    attr, bad_fn = AB_MUTATIONS[name]
    monkeypatch.setattr(odec, attr, bad_fn)
    found = []
    for case in AB_CASES:
        try:
            found += _check(*case, ab=True)
        except Exception:
            found.append("crash")
    assert found, f"mutation '{name}' passed every pin"


# ------------------------------------------------------------------ planted mistakes

MUTATIONS = {
    "window shifted by one position": (
        "window_tokens",
        lambda L, W, window, k_new: {**{L - W + 1 + i: np.asarray(window[i], np.float64) for i in range(W)},
                                     L: np.asarray(k_new, np.float64)}),
    "tail slot (p + 1) mod m": ("tail_slot", lambda p, m: (p + 1) % m),
    "new indexer key not appended": ("append_key", lambda keys, new: keys),
    "completion one token late": ("block_completes", lambda L, m: L % m == 0 and L > 0),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(monkeypatch, name):
    attr, bad_fn = MUTATIONS[name]
    monkeypatch.setattr(odec, attr, bad_fn)
    found = []
    for case in CASES:
        try:
            found += _check(*case)
        except Exception:  # a crash also exposes the mistake
            found.append("crash")
    assert found, f"mutation '{name}' passed every pin"


@pytest.mark.parametrize("L", [0, 5, 127, 128, 300])
def test_window_only_layer(L):
    """A layer without a compressed branch (pure sliding-window attention,
    report §4.2.1): the step attends over the window alone, whatever the
    stored entries, and compresses nothing."""
    W, m = 128, 4
    state, seq = _case(11, L, m, W)
    got = odec.decode_step("swa", 1, W, L, 0, 1 / 24, entries=state["entries"], window=state["window"],
                           q=state["q"], k_new=state["k_new"])
    wpos = csa.window_positions(L, W)
    o, lse = csa.attend_one(seq["q"], np.zeros((0, D)), seq["k"][wpos], 1 / 24)
    assert got["comp_new"] is None
    assert np.allclose(got["o"], o, atol=1e-12) and np.allclose(got["lse"], lse, atol=1e-12)
