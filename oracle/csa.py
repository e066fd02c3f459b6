"""The CSA / HCA hot path, restated step by step in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources (the pages are Chinese translations; their formulas are prose):

* "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
  (cnblogs translation of the report), §2.3.1 compressed sparse attention,
  §2.3.2 heavily compressed attention, §2.3.3 other details, §3.5.1 KV cache
  layout, §4.2.1 model settings, §5.2.1 FP4 QAT.  Cited below as "report".
* "DeepSeek-V4: million-token context usable by agents" (translation of the
  Hugging Face blog post ``deepseekv4``), section "Hybrid attention: CSA and
  HCA" with Fig. 3 and Fig. 4.  Cited below as "HF blog".

Where the pages leave a step open, the reading taken is written beside it.

Notation: m is the compression ratio, t a 0-based query position,
N_c(t) = floor((t + 1) / m) the number of compressed blocks whose last raw
token is at or before t, W the sliding-window size.
"""
from __future__ import annotations

import numpy as np

from . import canon

# ------------------------------------------------------------------ step 1: compressor


def pooling_weights(g_block: np.ndarray, bias: np.ndarray) -> np.ndarray:
    """Softmax-gated pooling weights of one block.

    report §2.3.1 ("compressed key-value entries"): every m entries are folded
    into one using compression weights and a learnable position bias; HF blog,
    "Hybrid attention": the compressor is softmax-gated pooling with a
    learnable position bias.  Reading: the softmax runs over the m positions of
    the block, separately for every channel, on the logit g_i + b_{i mod m}.

    g_block: [m, D] gate logits; bias: [m, D].  Returns [m, D], columns sum to 1.
    """
    a = np.asarray(g_block, dtype=np.float64) + np.asarray(bias, dtype=np.float64)
    a = a - a.max(axis=0, keepdims=True)
    e = np.exp(a)
    return e / e.sum(axis=0, keepdims=True)


def compress(k: np.ndarray, g: np.ndarray, bias: np.ndarray, m: int) -> np.ndarray:
    """c_j[d] = sum_{i in block j} softmax_i(g_i[d] + b[i - j m][d]) * k_i[d].

    report §2.3.1 (CSA, m = 4) and §2.3.2 (HCA, m' = 128, no overlap).
    Blocks start at token 0; a trailing partial block is not emitted (it stays
    in the uncompressed tail, report §3.5.1).  k, g: [n, D] -> [n // m, D].
    """
    k = np.asarray(k, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    n, D = k.shape
    nb = n // m
    out = np.zeros((nb, D))
    for j in range(nb):
        w = pooling_weights(g[j * m:(j + 1) * m], bias)
        out[j] = (w * k[j * m:(j + 1) * m]).sum(axis=0)
    return out


def compress_overlap(ka, ga, ba, kb, gb, bb, m: int) -> np.ndarray:
    """Overlapping compression of CSA.

    report §2.3.1: the hidden states give two sets of KV entries C_a, C_b
    with compression weights Z_a, Z_b, and every m entries are folded into one
    with those weights and learnable position biases; §2.3.2 says HCA does
    *not* compress with overlap, so CSA's blocks overlap.  Reading: entry j
    pools C_a over its own block j (positions j m .. (j + 1) m - 1) and C_b
    over the previous block j - 1, with one softmax per channel over all 2 m
    logits (Z_a + B_a[i - j m] for the first, Z_b + B_b[i - (j - 1) m] for the
    second); entry 0 has no previous block and pools C_a alone.  The entry
    still ends at token (j + 1) m - 1, so visibility is unchanged.

    ka, ga, kb, gb: [n, D]; ba, bb: [m, D] -> [n // m, D]."""
    ka, ga, kb, gb = (np.asarray(x, dtype=np.float64) for x in (ka, ga, kb, gb))
    ba, bb = np.asarray(ba, dtype=np.float64), np.asarray(bb, dtype=np.float64)
    n, D = ka.shape
    out = np.zeros((n // m, D))
    for j in range(n // m):
        cur = slice(j * m, (j + 1) * m)
        logits = [ga[cur] + ba]
        vals = [ka[cur]]
        if j > 0:
            prev = slice((j - 1) * m, j * m)
            logits.append(gb[prev] + bb)
            vals.append(kb[prev])
        a = np.concatenate(logits, axis=0)  # [m or 2 m, D]
        a = a - a.max(axis=0, keepdims=True)
        e = np.exp(a)
        w = e / e.sum(axis=0, keepdims=True)
        out[j] = (w * np.concatenate(vals, axis=0)).sum(axis=0)
    return out


def n_visible(t, m: int):
    """Number of compressed blocks visible to query t: block j ends at raw
    token (j + 1) m - 1, which must be <= t (no block that ends after t)."""
    return (np.asarray(t) + 1) // m


# ------------------------------------------------------------------ step 2: lightning indexer


def index_scores(q_idx: np.ndarray, w: np.ndarray, k_idx: np.ndarray) -> np.ndarray:
    """s[j] = sum_h w[h] * ReLU(q_h . kI_j) in float64.

    report §2.3.1 ("lightning indexer"), HF blog "Hybrid attention" (ReLU-scored
    multi-head dot product).  q_idx: [H_I, d_I]; w: [H_I]; k_idx: [N, d_I].
    The inputs are taken as exact values (already decoded from their storage
    format by the caller).
    """
    q = np.asarray(q_idx, dtype=np.float64)
    kk = np.asarray(k_idx, dtype=np.float64)
    logits = kk @ q.T  # [N, H_I]
    return np.maximum(logits, 0.0) @ np.asarray(w, dtype=np.float64)


def index_scores_f32(q_idx: np.ndarray, w: np.ndarray, k_idx: np.ndarray) -> np.ndarray:
    """The float32 index score in the canonical order (see ``canon``)."""
    return canon.index_scores_f32(q_idx, w, k_idx)


def bf16_score(s) -> np.ndarray:
    """BF16 index score (report §5.2.1: index scores quantized FP32 -> BF16):
    round to float32, then round-to-nearest-even to bf16."""
    from .codecs import bf16_round
    return bf16_round(np.asarray(s, dtype=np.float64).astype(np.float32))


# ------------------------------------------------------------------ step 3: top-k selector


def topk(scores: np.ndarray, n_cand: int, k: int):
    """Keep the best k of the first ``n_cand`` blocks.

    report §2.3.1: a top-k selector keeps a subset of compressed entries for
    the core attention.  Order: score descending, ties to the lower block index;
    -0 counts as +0.  The kept indices are returned ascending, padded with -1
    to length k, plus the count min(k, n_cand).
    """
    s = np.asarray(scores, dtype=np.float64)[:n_cand] + 0.0  # -0 -> +0
    j = np.arange(n_cand)
    order = np.lexsort((j, -s))  # primary key -score, then j
    keep = np.sort(np.asarray(order[:min(k, n_cand)], dtype=np.int64))
    out = np.full(k, -1, dtype=np.int64)
    out[:len(keep)] = keep
    return out, len(keep)


# ------------------------------------------------------------------ steps 4/5: core attention


def attend_one(q: np.ndarray, entries: np.ndarray, window: np.ndarray, scale: float,
               sink=None):
    """Shared-KV MQA for one query token over compressed entries + window.

    report §2.3.1 ("shared key-value MQA": every compressed entry is both key
    and value) and §2.3.3 (the sliding-window branch adds n_win uncompressed
    entries; attention sink logits let a head's weights sum to less than one).
    One softmax over the union, so the two branches merge as online softmax
    would.  q: [H, D]; entries: [S, D]; window: [Wn, D] -> (o [H, D], lse [H]).
    Empty union: o = 0, lse = -inf.
    """
    X = np.concatenate([np.asarray(entries, dtype=np.float64).reshape(-1, q.shape[1]),
                        np.asarray(window, dtype=np.float64).reshape(-1, q.shape[1])], axis=0)
    H = q.shape[0]
    if X.shape[0] == 0:
        return np.zeros_like(q, dtype=np.float64), np.full(H, -np.inf)
    logits = scale * (np.asarray(q, dtype=np.float64) @ X.T)  # [H, S+Wn]
    mx = logits.max(axis=1, keepdims=True)
    if sink is not None:
        mx = np.maximum(mx, np.asarray(sink, dtype=np.float64)[:, None])
    e = np.exp(logits - mx)
    den = e.sum(axis=1, keepdims=True)
    if sink is not None:
        den = den + np.exp(np.asarray(sink, dtype=np.float64)[:, None] - mx)
    p = e / den
    return p @ X, (mx + np.log(den))[:, 0]


def window_positions(t: int, W: int) -> np.ndarray:
    """Raw positions of the sliding window of query t: max(0, t - W + 1) .. t
    (reading: the current token is inside its own window)."""
    return np.arange(max(0, t - W + 1), t + 1)


def csa_attend(q, t, idx, cnt, comp, raw, W, scale, sink=None):
    """CSA core attention for one query at position t.

    comp: [N, D] compressed entries (decoded), raw: indexable by raw position
    -> [D] raw tokens, idx/cnt: the selected blocks.  No de-duplication between
    a selected block and window tokens it covers (the window branch is an
    additional set of entries, report §2.3.3)."""
    sel = np.asarray(idx[:cnt], dtype=np.int64)
    return attend_one(q, comp[sel], raw[window_positions(t, W)], scale, sink)


def hca_attend(q, t, m, comp, raw, W, scale, sink=None):
    """HCA core attention: dense over every visible compressed entry + window
    (report §2.3.2: no sparse selection)."""
    nc = int(n_visible(t, m))
    return attend_one(q, comp[:nc], raw[window_positions(t, W)], scale, sink)


# ------------------------------------------------------------------ query / KV normalization and partial RoPE


def rms_norm(x, gain, eps: float) -> np.ndarray:
    """RMSNorm of the last axis: x / sqrt(mean(x^2) + eps) * gain.

    report §2.3.3 ("other details"): each head's query and the compressed KV
    entries are RMS-normalized before the core attention (and §2.4: this,
    not QK-Clip, keeps the logits bounded).  Reading: one learnable gain per
    dimension of the 576-d vector, eps added inside the root; the same norm
    (with the KV gain) is applied to every KV entry the core attention sees,
    compressed or from the sliding window."""
    x = np.asarray(x, dtype=np.float64)
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / r * np.asarray(gain, dtype=np.float64)


ROPE_DIMS = 64


def rope(x, pos, base: float, dims: int = ROPE_DIMS) -> np.ndarray:
    """Rotary position embedding on the last ``dims`` dimensions of x.

    report §2.3.3: RoPE is applied to the last 64 dims of every query and
    KV entry vector.  Reading (the rotary embedding of Su et al., RoFormer):
    consecutive pairs (x_{2i}, x_{2i+1}) of those dims turn by the angle
    pos * base^(-2i / dims); the other dims are unchanged.  pos may be an
    array broadcasting against x's leading axes."""
    x = np.array(x, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.float64)
    i = np.arange(dims // 2)
    ang = pos[..., None] * base ** (-2.0 * i / dims)  # [..., dims / 2]
    c, s = np.cos(ang), np.sin(ang)
    r = x[..., -dims:]
    a, b = r[..., 0::2].copy(), r[..., 1::2].copy()
    r[..., 0::2] = a * c - b * s
    r[..., 1::2] = a * s + b * c
    x[..., -dims:] = r
    return x


def entry_position(j, m: int):
    """Raw position at which compressed entry j is rotated: its block's first
    token, j * m (reading: the pages rotate "KV entries" without saying where
    a pooled entry sits; the first token of its block keeps query-entry
    offsets in raw-token units, like the window's)."""
    return np.asarray(j) * m


def prep_entries(comp, m: int, gain, eps: float, base: float, first: int = 0):
    """Compressed entries first, first + 1, .. as the core attention sees
    them: RMSNorm with the KV gain (None: no norm), then RoPE at
    entry_position (base 0: no RoPE) (report §2.3.3)."""
    x = np.asarray(comp, dtype=np.float64)
    if gain is not None:
        x = rms_norm(x, gain, eps)
    if base > 0:
        x = rope(x, entry_position(first + np.arange(x.shape[0]), m), base)
    return x


def attend_one_rope(q, t, entries, entry_pos, window, window_pos, scale, q_gain, kv_gain, eps, base, sink=None):
    """Core attention of one query at position t with query / KV RMSNorm and
    partial RoPE (report §2.3.3): the query is normalized (q_gain) and rotated
    by t; window tokens are normalized (kv_gain) and rotated by their own
    positions; the compressed entries are taken as already prepared
    (prep_entries: they are stored that way).  The output's last 64 dims are
    rotated back by t, so they carry the position of each value relative to
    the query ("RoPE on the core attention output").  A gain of None skips
    that norm; base 0 skips every rotation.  Returns (o, lse)."""
    qn = np.asarray(q, dtype=np.float64)
    wn = np.asarray(window, dtype=np.float64).reshape(-1, qn.shape[1])
    if q_gain is not None:
        qn = rms_norm(qn, q_gain, eps)
    if kv_gain is not None and len(wn):
        wn = rms_norm(wn, kv_gain, eps)
    if base > 0:
        qn = rope(qn, np.full(qn.shape[0], t), base)
        if len(wn):
            wn = rope(wn, np.asarray(window_pos), base)
    o, lse = attend_one(qn, entries, wn, scale, sink)
    if base > 0:
        o = rope(o, np.full(o.shape[0], -t), base)
    return o, lse


# ------------------------------------------------------------------ whole chains


def csa_prefill(k, g, bias, k_idx_raw, g_idx, bias_idx, q_idx, w, q, m, top_k, W, scale,
                score="f32", sink=None, rows=None):
    """compress -> index -> top-k -> attention for every (or the given) query
    rows of one sequence.  Returns dict with idx, cnt, o, lse for those rows.

    score="f32": the canonical float32 score (bit-exact selection target);
    score="f64": float64 scores."""
    comp = compress(k, g, bias, m)
    kI = compress(k_idx_raw, g_idx, bias_idx, m)
    n = k.shape[0]
    rows = range(n) if rows is None else rows
    res = {"idx": [], "cnt": [], "o": [], "lse": [], "comp": comp, "kI": kI}
    for t in rows:
        nc = int(n_visible(t, m))
        wt = w if np.ndim(w) == 1 else w[t]
        if score == "f32":
            s = index_scores_f32(np.asarray(q_idx[t], np.float32), np.asarray(wt, np.float32),
                                 kI[:nc].astype(np.float32))
        else:
            s = index_scores(q_idx[t], wt, kI[:nc])
        idx, cnt = topk(s, nc, top_k)
        o, lse = csa_attend(q[t], t, idx, cnt, comp, k, W, scale, sink)
        res["idx"].append(idx)
        res["cnt"].append(cnt)
        res["o"].append(o)
        res["lse"].append(lse)
    for key in ("idx", "cnt", "o", "lse"):
        res[key] = np.asarray(res[key])
    return res
