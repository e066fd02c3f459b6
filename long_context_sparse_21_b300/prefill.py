"""Causal CSA prefill of one sequence over the C ABI.

DeepSeek-V4 report (cnblogs translation) §2.3.1: the compressor folds every
m = 4 raw KV entries into one; the lightning indexer scores every compressed
block each query may see and a top-k selector keeps k of them; the core
attention runs over the kept entries plus the sliding window (§2.3.3).  For a
prompt this is, per query position t:

    compress (KV stream and indexer-key stream, whole sequence)
    -> for each chunk of queries: indexer + top-k -> sparse attention

Queries are processed in chunks (a chunk's scores live in one workspace that
the next chunk reuses).  Everything runs in libcsa's kernels; this module
allocates memory and sequences the calls.
"""
from __future__ import annotations

import math

import torch

from . import abi, synth


class CsaPrefill:
    """One sequence of n raw tokens.

    Synthetic inputs (synth): raw KV tokens and gate logits N(0,1) BF16 [n, 576]
    and an indexer-key stream N(0,1) BF16 [n, 128] with its own gates, the same
    seeded fraction `outliers` of positions scaled by 8 in both raw streams;
    position biases N(0, 0.1); queries N(0,1) BF16 [n, 64, 576]; indexer
    queries N(0,1) BF16 [n, 64, 128]; head weights U(0,1) [n, 64].
    """

    def __init__(self, n: int = 131072, seed: int = 0, chunk: int = 4096, top_k: int = 1024, W: int = 128,
                 m: int = 4, page_entries: int = 2048, score_dtype: int = abi.BF16, outliers: float = 0.01,
                 device: str = "cuda", overlap_ab: bool = False):
        self.n, self.chunk, self.top_k, self.W, self.m = n, chunk, top_k, W, m
        self.H, self.D, self.H_idx, self.d_idx = 64, 576, 64, 128
        self.scale = 1.0 / math.sqrt(self.D)
        s = synth.Synth(seed, device)
        k = s.normal("k", (n, self.D))
        k_idx = s.normal("k_idx", (n, self.d_idx))
        if outliers > 0:
            mask = s.outlier_mask("outliers", n, outliers)
            k[mask] *= 8.0
            k_idx[mask] *= 8.0
        self.k = k.to(torch.bfloat16).contiguous()
        self.k_idx = k_idx.to(torch.bfloat16).contiguous()
        del k, k_idx
        self.g = s.normal("g", (n, self.D), dtype=torch.bfloat16)
        self.g_idx = s.normal("g_idx", (n, self.d_idx), dtype=torch.bfloat16)
        self.bias = s.normal("bias", (m, self.D), 0.1)
        self.bias_idx = s.normal("bias_idx", (m, self.d_idx), 0.1)
        # overlapping compression (report §2.3.1): a b stream per compressor,
        # drawn like the a stream's tokens and gates (no outliers)
        self.overlap_ab = overlap_ab
        if overlap_ab:
            self.k_b = s.normal("k_b", (n, self.D), dtype=torch.bfloat16)
            self.g_b = s.normal("g_b", (n, self.D), dtype=torch.bfloat16)
            self.k_idx_b = s.normal("k_idx_b", (n, self.d_idx), dtype=torch.bfloat16)
            self.g_idx_b = s.normal("g_idx_b", (n, self.d_idx), dtype=torch.bfloat16)
            self.bias_b = s.normal("bias_b", (m, self.D), 0.1)
            self.bias_idx_b = s.normal("bias_idx_b", (m, self.d_idx), 0.1)
        self.q = s.normal("q", (n, self.H, self.D), dtype=torch.bfloat16)
        self.q_idx = s.normal("q_idx", (n, self.H_idx, self.d_idx), dtype=torch.bfloat16)
        self.w = s.uniform("w", (n, self.H_idx))
        self.pos = torch.arange(n, dtype=torch.int32, device=device)
        self.seq = torch.zeros(n, dtype=torch.int32, device=device)

        n_ent = n // m
        self.kv = abi.make_pool(abi.FMT_KV_POOL_FP8, 1, n_ent, self.D, page_entries, device, shuffle_seed=seed)
        self.ki = abi.make_pool(abi.FMT_INDEX_POOL_BF16, 1, n_ent, self.d_idx, page_entries, device,
                                shuffle_seed=seed + 1)
        self.out = torch.empty((n, self.H, self.D), dtype=torch.bfloat16, device=device)
        self.idx = torch.empty((n, top_k), dtype=torch.int32, device=device)
        self.cnt = torch.empty((n,), dtype=torch.int32, device=device)

        # one indexer workspace, sized for the last (longest) chunk, shared by all chunks
        ws_bytes = abi.IndexCall.workspace_bytes(chunk, self.H_idx, self.d_idx, m, n - 1, self.ki, score_dtype)
        self.ws = abi.alloc_workspace(max(ws_bytes, 1024), device)
        self.calls = []
        for c0 in range(0, n, chunk):
            c1 = min(n, c0 + chunk)
            # every kernel before these calls is this library's (compressor,
            # indexer, attention of the previous chunk): none writes the
            # queries, so the calls may start early
            index = abi.IndexCall(self.q_idx[c0:c1], self.w[c0:c1], self.pos[c0:c1], self.ki, top_k, m, c1 - 1, 1,
                                  seq=self.seq[c0:c1], score_dtype=score_dtype, ws=self.ws, idx=self.idx[c0:c1],
                                  cnt=self.cnt[c0:c1], overlap=True)
            attend = abi.AttendCall(True, self.q[c0:c1], self.pos[c0:c1], self.kv, W, self.k[None], self.scale, m,
                                    c1 - 1, 1, idx=self.idx[c0:c1], cnt=self.cnt[c0:c1], seq=self.seq[c0:c1],
                                    out=self.out[c0:c1], with_lse=False, overlap=True)
            self.calls.append((c0, c1, index, attend))

    def stages(self) -> list[str]:
        return ["compress", "index_score", "index_select", "attend"]

    def run(self, stream=None, marks=None) -> dict:
        """The whole prefill.  marks: optional dict stage -> [(start, end)
        event pairs] to time each kernel group (events recorded on `stream`)."""
        st = stream if stream is not None else torch.cuda.current_stream()

        def timed(name, fn):
            if marks is None:
                fn()
                return
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            fn()
            b.record(st)
            marks.setdefault(name, []).append((a, b))

        def compress():
            ab_kv, ab_idx = {}, {}
            if self.overlap_ab:
                ab_kv = dict(bias_b=self.bias_b, k_b=self.k_b[None], g_b=self.g_b[None])
                ab_idx = dict(bias_b=self.bias_idx_b, k_b=self.k_idx_b[None], g_b=self.g_idx_b[None])
            abi.csa_compress(self.kv, self.bias, self.m, k=self.k[None], g=self.g[None], stream=stream, **ab_kv)
            abi.csa_compress(self.ki, self.bias_idx, self.m, k=self.k_idx[None], g=self.g_idx[None], stream=stream,
                             **ab_idx)

        timed("compress", compress)
        for c0, c1, index, attend in self.calls:
            timed("index_score", lambda: index.score(stream))
            timed("index_select", lambda: index.select(stream))
            timed("attend", lambda: attend(stream))
        return {"out": self.out, "idx": self.idx, "cnt": self.cnt}

    def launches(self) -> int:
        return 2 + sum(2 + a.launches() for _, _, _, a in self.calls)

    def status(self) -> int:
        for _, _, index, attend in self.calls:
            for st in (index.status(), attend.status()):
                if st != 0:
                    return st
        return 0

    def flops(self) -> dict:
        """Algorithmic FLOPs: the indexer over every causal block of every query
        (64 heads x 128 dims, multiply-add = 2), attention over the kept entries
        plus the window (QK^T and PV over 64 heads x 576 dims)."""
        import numpy as np
        u = np.arange(1, self.n + 1, dtype=np.int64)  # t + 1
        nc = u // self.m
        idx_flops = int(nc.sum()) * self.H_idx * self.d_idx * 2
        items = int((np.minimum(self.top_k, nc) + np.minimum(self.W, u)).sum())
        att_flops = items * self.H * self.D * 2 * 2
        return {"index": idx_flops, "attend": att_flops}
