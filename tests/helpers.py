"""Shared test helpers: error metrics, readers of the documented pool layouts,
and the oracle's view of one decode step.  The oracle side here only uses
``oracle/`` and the seeded synthetic inputs, never a CUDA output."""
from __future__ import annotations

import numpy as np
import torch

from oracle import codecs, csa


def max_abs_rel(x, y) -> float:
    """Per output row: max_i |x_i - y_i| / max_i |y_i|; the max over rows."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    num = np.abs(x - y).max(axis=-1)
    den = np.abs(y).max(axis=-1)
    return float(np.max(num / np.maximum(den, 1e-300)))


def f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


# ------------------------------------------------------------------ pool readers (layouts of include/csa.h)

_TABLES = {}


def _page_bytes(store, b, e):
    P = store.page_entries
    key = id(store.page_table)
    if key not in _TABLES or _TABLES[key][0] is not store.page_table:
        _TABLES[key] = (store.page_table, store.page_table.cpu().numpy())
    pg = int(_TABLES[key][1][b, e // P])
    return pg, e % P


def read_kv_pool(store, b, n):
    """-> (codes u8 [n,512], scale f32 [n], rope u16 [n,64]) of entries 0..n-1."""
    raw = store.tensor[store.offset:].cpu().numpy()
    P = store.page_entries
    pb = 644 * P
    codes = np.empty((n, 512), np.uint8)
    scale = np.empty(n, np.float32)
    rope = np.empty((n, 64), np.uint16)
    for e in range(n):
        pg, s = _page_bytes(store, b, e)
        base = pg * pb
        codes[e] = raw[base + s * 512: base + s * 512 + 512]
        rope[e] = raw[base + 512 * P + s * 128: base + 512 * P + s * 128 + 128].view(np.uint16)
        scale[e] = raw[base + 640 * P + s * 4: base + 640 * P + s * 4 + 4].view(np.float32)[0]
    return codes, scale, rope


def read_index_bf16_pool(store, b, n):
    """-> bf16 bits u16 [n, 128], undoing the 128-byte swizzle."""
    raw = store.tensor[store.offset:].cpu().numpy()
    P = store.page_entries
    out = np.empty((n, 128), np.uint16)
    d = np.arange(128)
    for e in range(n):
        pg, s = _page_bytes(store, b, e)
        r = s % 128
        off = (s // 128) * 32768 + (d // 64) * 16384 + r * 128 + ((((d % 64) // 8) ^ (r % 8)) * 16) + (d % 8) * 2
        off = pg * 256 * P + off
        lo = raw[off].astype(np.uint16)
        hi = raw[off + 1].astype(np.uint16)
        out[e] = lo | (hi << 8)
    return out


def read_index_fp4_pool(store, b, n):
    """-> (codes u8 [n,128] one per element, scale codes u8 [n, 8])."""
    raw = store.tensor[store.offset:].cpu().numpy()
    P = store.page_entries
    codes = np.empty((n, 128), np.uint8)
    scales = np.empty((n, 8), np.uint8)
    for e in range(n):
        pg, s = _page_bytes(store, b, e)
        base = pg * 72 * P
        codes[e] = codecs.unpack_nibbles(raw[base + s * 64: base + s * 64 + 64])
        scales[e] = raw[base + 64 * P + s * 8: base + 64 * P + s * 8 + 8]
    return codes, scales


# ------------------------------------------------------------------ selection checks

def score_error_bound(q, w, keys, bf16_scores: bool):
    """Per-key bound on |kernel score - exact score| for a tensor-core index
    score s_j = sum_h w_h ReLU(q_h . k_j) of exactly representable operands
    (the stored keys, the query as the kernel reads it).

    Float32 accumulation: the dot products (d_I terms) and the head sum (H_I
    terms) change the result by at most (d_I + H_I) u_32 times the score's
    absolute magnitude sum_h |w_h| sum_d |q_hd k_jd| (u_32 = 2^-24), doubled as a
    margin for the tensor core's accumulation order.  A BF16 score is then
    rounded to nearest, which moves it by at most half a unit in its last of 8
    significant bits: 2^-8 of its magnitude."""
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64).reshape(-1, q.shape[1])
    mag = (np.abs(keys) @ np.abs(q).T) @ np.abs(np.asarray(w, dtype=np.float64))
    acc = 2.0 * (q.shape[1] + q.shape[0]) * 2.0 ** -24 * mag
    if not bf16_scores:
        return acc
    s = csa.index_scores(q, w, keys)
    return acc + 2.0 ** -8 * (np.abs(s) + acc)


def selection_valid(sel, cnt, scores, k, err):
    """The kept set is a valid top-k of `scores` (float64, visible blocks
    only) given per-block score errors `err` (an array, or one number for
    every block): right size, ascending, unique, -1 padded, and every kept
    block a may rank above every dropped block b, i.e.
    scores[a] + err[a] >= scores[b] - err[b]."""
    n = len(scores)
    want = min(k, n)
    if cnt != want:
        return False, f"cnt {cnt} != {want}"
    s = np.asarray(sel[:cnt])
    if np.any(np.diff(s) <= 0) or (cnt and (s[0] < 0 or s[-1] >= n)):
        return False, "not ascending / out of range"
    if np.any(np.asarray(sel[cnt:]) != -1):
        return False, "padding"
    if cnt == n:
        return True, ""
    e = np.broadcast_to(np.asarray(err, dtype=np.float64), (n,))
    mask = np.zeros(n, bool)
    mask[s] = True
    lo_kept = (scores + e)[mask].min()
    hi_dropped = (scores - e)[~mask].max()
    if lo_kept < hi_dropped:
        a = np.flatnonzero(mask)[np.argmin((scores + e)[mask])]
        b = np.flatnonzero(~mask)[np.argmax((scores - e)[~mask])]
        return False, f"kept {a} ({scores[a]} +- {e[a]}) below dropped {b} ({scores[b]} +- {e[b]})"
    return True, ""


# ------------------------------------------------------------------ oracle view of a decode step

def oracle_decode_step(layer, b, selection=None):
    """What the oracle computes for sequence b of a DecodeLayer step, from the
    synthetic state and step inputs only.  `selection` (optional) replaces the
    oracle's own top-k for the attention step: a selection the caller has
    checked to be a valid top-k of the oracle's scores."""
    from oracle import decode as odec
    src = layer.sources[b]
    sh = layer.shared_sources
    qs = {k: f64(v[b]) for k, v in layer.inputs.items()}
    kw = dict(entries=src["entries"].numpy(), window=f64(src["window"]), tail_gate=f64(src["tail_gate"]),
              bias=f64(sh["bias"]), q=qs["q"], k_new=qs["k_new"], g_new=qs["g_new"])
    if layer.kind == "csa":
        kw.update(keys_idx=src["keys_idx"].numpy(), ring_idx=f64(src["ring_idx"]),
                  tail_gate_idx=f64(src["tail_gate_idx"]), bias_idx=f64(sh["bias_idx"]), q_idx=qs["q_idx"],
                  w=qs["w"], k_idx_new=qs["k_idx_new"], g_idx_new=qs["g_idx_new"])
        kw["index_fmt"] = "fp4" if layer.index_fmt == 4 else "bf16"  # abi.FMT_INDEX_POOL_E2M1
        kw["selection"] = selection
    if getattr(layer, "overlap_ab", False):
        kw["overlap"] = {"kv": (f64(src["tail_b"]), f64(src["tail_gate_b"]), f64(sh["bias_b"])),
                         "idx": (f64(src["tail_idx_b"]), f64(src["tail_gate_idx_b"]), f64(sh["bias_idx_b"]))}
    if getattr(layer, "norm_rope", False):
        kw.update(q_gain=f64(layer.q_gain), kv_gain=f64(layer.kv_gain), eps=layer.norm_eps,
                  rope_base=layer.rope_base)
    return odec.decode_step(layer.kind, layer.m, layer.W, layer.ctx[b], layer.top_k, layer.scale, **kw)


def recall_vs_f32(layer, b, ref, sel, cnt):
    """|S_path & S_f32| / |S_f32|: S_f32 is the top-k of the canonical float32
    score of the unquantized keys and query (report §5.2.1 measures the
    selector's KV-entry recall this way)."""
    q32 = np.asarray(layer.inputs["q_idx"][b].float().cpu().numpy(), np.float32)
    w32 = np.asarray(layer.inputs["w"][b].float().cpu().numpy(), np.float32)
    keys = ref["keys_f32"]
    s32 = csa.index_scores_f32(q32, w32, keys)
    want, wc = csa.topk(s32, len(keys), layer.top_k)
    got = set(int(x) for x in sel[:cnt])
    return len(got & set(int(x) for x in want[:wc])) / max(wc, 1)
