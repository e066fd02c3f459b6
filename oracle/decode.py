"""The oracle's view of one decode step of a CSA or HCA layer.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

DeepSeek-V4 report (cnblogs translation) §3.5.1: a decode step appends the new
raw token to the state cache (window + uncompressed tail); when the tail fills
a block of m tokens, the block is compressed into a new entry of the classical
cache.  Then (CSA) the lightning indexer scores every visible compressed key,
the top-k selector keeps k blocks, and the core attention runs over them plus
the window; (HCA) the core attention runs over every visible entry plus the
window.  Positions and stored values are taken as plain arrays; no cache
layout is modelled here.

The bookkeeping of the state cache (which raw position sits in which window or
tail slot, when a block completes, where the new indexer key goes) is kept in
the small functions below, so that a test can check each of them against the
whole-sequence definitions of ``csa`` and can plant a mistake in one of them.
"""
from __future__ import annotations

import numpy as np

from . import codecs, csa


def _fp4_roundtrip(x):
    """Values of x after storage in the FP4 indexer format (e2m1 with one e4m3
    scale per 16 elements, report §5.2.1 / the workload's NVFP4-style format)."""
    x = np.asarray(x, dtype=np.float32)
    shape = x.shape
    codes, s_code = codecs.fp4_block_encode(x.reshape(-1, shape[-1]))
    return codecs.fp4_block_decode(codes, s_code).reshape(shape)


def tail_slot(p: int, m: int) -> int:
    """Slot of raw position p in a per-sequence buffer of m rows (the tail
    gates, the indexer stream's raw keys): p mod m (report §3.5.1, state cache
    of the uncompressed tail)."""
    return p % m


def window_tokens(L: int, W: int, window, k_new) -> dict:
    """Raw tokens the step can see, by position: the W stored tokens at
    positions L - W .. L - 1 (oldest first) and the new token at L."""
    raw = {L - W + i: np.asarray(window[i], dtype=np.float64) for i in range(W)}
    raw[L] = np.asarray(k_new, dtype=np.float64)
    return raw


def block_completes(L: int, m: int) -> bool:
    """The token at position L closes block (L + 1) / m - 1 when L + 1 is a
    multiple of m (the block covers positions L + 1 - m .. L)."""
    return (L + 1) % m == 0


def b_slot(p: int, m: int) -> int:
    """Slot of raw position p in the b stream's tail of overlapping
    compression, which keeps two blocks (the one being filled and the one
    before it, which the next entry pools): p mod 2m."""
    return p % (2 * m)


def previous_block(L: int, m: int, keys_b, gates_b):
    """The b stream's tokens of the block before the one that position L
    completes (positions L + 1 - 2m .. L - m, from their tail slots), or None
    when that block is the first."""
    p0 = L + 1 - 2 * m
    if p0 < 0:
        return None
    rows = [b_slot(p, m) for p in range(p0, p0 + m)]
    return np.asarray(keys_b, dtype=np.float64)[rows], np.asarray(gates_b, dtype=np.float64)[rows]


def pool_entry(kblk, gblk, bias, m: int, prev=None):
    """The entry of one completed block: the plain compressor, or (prev =
    (keys, gates, bias) of the b stream's previous block) overlapping
    compression, evaluated as entry 1 of csa.compress_overlap over the two
    blocks."""
    if prev is None:
        return csa.compress(kblk, gblk, bias, m)[0]
    kb, gb, bias_b = prev
    z = np.zeros_like(np.asarray(kblk, dtype=np.float64))
    return csa.compress_overlap(np.vstack([z, kblk]), np.vstack([z, gblk]), bias, np.vstack([kb, z]),
                                np.vstack([gb, z]), bias_b, m)[1]


def append_key(keys, new_key):
    """Indexer keys after the step: the stored keys followed by the key of
    the block the step completed."""
    return np.vstack([keys, new_key])


def decode_step(kind, m, W, L, top_k, scale, *, entries, window, q, k_new, tail_gate=None, bias=None, g_new=None,
                keys_idx=None, ring_idx=None, tail_gate_idx=None, bias_idx=None, q_idx=None, w=None,
                k_idx_new=None, g_idx_new=None, index_fmt="bf16", selection=None, sink=None,
                q_gain=None, kv_gain=None, eps=0.0, rope_base=0.0, overlap=None):
    """One sequence with L raw tokens before the step (the new token sits at L).
    kind: "csa", "hca", or "swa" (window only: no compressed branch).

    entries   float32 [>= L // m, 576]: compressed entries before the step,
              stored as FP8 content + scale + BF16 RoPE (codecs.kv_entry_*).
    window    [W, D]: raw tokens at positions L-W .. L-1 (bf16 values).  The
              same ring holds the raw tokens of the uncompressed tail, so
              W >= m - 1 (the cache's ring has 128 rows, m <= 128).
    tail_gate [m, D]: gate logits by slot p % m of the tail positions.
    keys_idx  float32 [>= L // m, 128]: compressed indexer keys, stored BF16
              (index_fmt "bf16") or FP4 (index_fmt "fp4"; the query is then
              quantized to the same FP4 format before scoring).
    ring_idx  [m, 128]: raw indexer keys by slot p % m; tail_gate_idx likewise.
    selection: optional kept block indices to attend over instead of the
    oracle's own top-k (to check the attention given another valid selection).
    sink      optional [H] attention-sink logits (report §2.3.3).
    q_gain, kv_gain, eps, rope_base: query / KV RMSNorm and partial RoPE
              (report §2.3.3; csa.attend_one_rope): the completed entry is
              prepared (csa.prep_entries) before it is stored, the stored
              entries are taken as prepared already, and the query and the
              window are normalized and rotated by the attention.
    overlap   optional dict for overlapping compression (report §2.3.1):
              "kv" = (keys_b [2m, D], gates_b [2m, D], bias_b [m, D]) and,
              for CSA, "idx" likewise for the indexer stream: the b stream's
              tail by slot p % 2m; a completed block's entry then also pools
              the b stream over the block before it (csa.compress_overlap).
    Returns dict(o [H, D], lse [H], idx, cnt, scores, comp_new, kI_new,
    keys, q_idx, keys_f32): keys and q_idx are the scored values (after their
    storage rounding); keys_f32 are the unquantized float32 keys of the
    visible blocks (for recall against a float32 selection).
    """
    f = lambda x: np.asarray(x, dtype=np.float64)  # noqa: E731
    n_old = L // m
    nvis = (L + 1) // m
    raw = window_tokens(L, W, window, k_new)
    out = {"comp_new": None, "kI_new": None, "idx": None, "cnt": None, "scores": None}
    # a window-only layer (kind "swa", report §4.2.1) has no compressed branch
    completes = kind != "swa" and block_completes(L, m)
    if completes:
        p0 = L + 1 - m
        kblk = np.stack([raw[p] for p in range(p0, L + 1)])
        gblk = np.stack([f(tail_gate[tail_slot(p, m)]) if p < L else f(g_new) for p in range(p0, L + 1)])
        prev = None
        if overlap is not None:
            kb, gb, bb = overlap["kv"]
            pb = previous_block(L, m, kb, gb)
            prev = None if pb is None else (pb[0], pb[1], f(bb))
        out["comp_new"] = csa.prep_entries(pool_entry(kblk, gblk, f(bias), m, prev)[None], m, kv_gain, eps,
                                           rope_base, first=nvis - 1)[0]
    entries = np.asarray(entries, dtype=np.float32)

    def comp_rows(rows):
        rows = np.asarray(rows, dtype=np.int64)
        vals = np.empty((len(rows), entries.shape[1]), np.float32)
        old = rows < n_old
        vals[old] = entries[rows[old]]
        if (~old).any():
            vals[~old] = out["comp_new"].astype(np.float32)
        return codecs.kv_entry_decode(*codecs.kv_entry_encode(vals))

    if kind == "csa":
        store = codecs.bf16_round if index_fmt == "bf16" else _fp4_roundtrip
        raw_keys = np.asarray(keys_idx[:n_old], dtype=np.float32)
        keys = store(raw_keys)
        if completes:
            ring_i = f(ring_idx).copy()
            ring_i[tail_slot(L, m)] = f(k_idx_new)
            gates_i = f(tail_gate_idx).copy()
            gates_i[tail_slot(L, m)] = f(g_idx_new)
            # rows of the ring in position order L + 1 - m .. L
            order = [tail_slot(p, m) for p in range(L + 1 - m, L + 1)]
            prev = None
            if overlap is not None:
                kb, gb, bb = overlap["idx"]
                pb = previous_block(L, m, kb, gb)
                prev = None if pb is None else (pb[0], pb[1], f(bb))
            out["kI_new"] = pool_entry(ring_i[order], gates_i[order], f(bias_idx), m, prev)
            new32 = out["kI_new"].astype(np.float32)[None]
            keys = append_key(keys, store(new32))
            raw_keys = append_key(raw_keys, new32)
        out["keys_f32"] = raw_keys[:nvis]
        qq = f(q_idx) if index_fmt == "bf16" else _fp4_roundtrip(np.asarray(q_idx, dtype=np.float32))
        s = csa.index_scores(qq, f(w), keys[:nvis])
        idx, cnt = csa.topk(s, nvis, top_k)
        out.update(scores=s, idx=idx, cnt=cnt, keys=keys[:nvis], q_idx=qq)
        sel = idx[:cnt] if selection is None else np.asarray(selection, dtype=np.int64)
    elif kind == "hca":
        sel = np.arange(nvis)
    else:
        sel = np.arange(0)
    X = comp_rows(sel) if len(sel) else np.zeros((0, entries.shape[1]))
    wpos = csa.window_positions(L, W)
    Wx = np.stack([raw[p] for p in wpos])
    o, lse = csa.attend_one_rope(f(q), L, X, None, Wx, wpos, scale, q_gain, kv_gain, eps, rope_base, sink)
    out.update(o=o, lse=lse)
    return out
