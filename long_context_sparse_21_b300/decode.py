"""Decode-step orchestration over the C ABI: one CSA or HCA attention layer of a
batch of sequences, with its paged compressed cache and its state cache.

DeepSeek-V4 report (cnblogs translation) §3.5.1: the KV cache has a classical
paged part for compressed entries and a state part (sliding-window tokens plus
the uncompressed tail).  A decode step of one layer is:

    CSA: compress-append (KV stream) -> compress-append (indexer-key stream)
         -> lightning indexer + top-k -> sparse attention
    HCA: compress-append (KV stream) -> dense attention

This module only allocates memory and sequences C-ABI calls; all arithmetic
runs in libcsa's kernels.  `Layer.step()` performs the whole step; the calls
are prepared once so a step allocates nothing and can be captured into a CUDA
graph.
"""
from __future__ import annotations

import math

import torch

from . import abi, synth


class DecodeLayer:
    """State + prepared calls of one layer for B sequences.

    ctx: raw tokens already in each sequence before the step (int, or a list
    of per-sequence lengths).  The new token of the step sits at position
    L_b = ctx_b.  Synthetic state (synth.decode_context): compressed entries
    for blocks j < L_b // m, the last W raw tokens in the window ring, gate
    logits of the uncompressed tail; per-step inputs from synth.decode_queries.
    """

    def __init__(self, kind: str, B: int, ctx, seed: int = 0, *, m: int | None = None, top_k: int = 512,
                 W: int = 128, H: int = 64, D: int = 576, H_idx: int = 64, d_idx: int = 128,
                 page_entries: int = 2048, index_fmt: int = abi.FMT_INDEX_POOL_BF16, score_dtype: int = abi.F32,
                 device: str = "cuda", tag: str = "", keep_sources=(), norm_rope: bool = False,
                 batch_invariant: bool = False, overlap_ab: bool = False):
        assert kind in ("csa", "hca", "swa")
        assert not overlap_ab or kind == "csa", "overlapping compression is CSA's"
        self.kind, self.B, self.W, self.H, self.D = kind, B, W, H, D
        # swa: a layer without a compressed branch (window only); its m is unused
        self.m = m if m is not None else {"csa": 4, "hca": 128, "swa": 1}[kind]
        self.top_k = top_k
        self.index_fmt = index_fmt
        self.score_dtype = score_dtype
        self.device = device
        ctx = [ctx] * B if isinstance(ctx, int) else list(ctx)
        self.ctx = ctx
        n_entries = max(c // self.m for c in ctx) if kind != "swa" else 0
        self.capacity = max(c + 1 for c in ctx) // self.m if kind != "swa" else 0
        s = synth.Synth(seed, device)
        st = synth.decode_context(seed, B, n_entries, W=W, m=self.m, D=D, d_idx=d_idx, device=device, tag=tag,
                                  with_index=(kind == "csa"))
        qs = synth.decode_queries(seed, B, H=H, D=D, H_idx=H_idx, d_idx=d_idx, device=device, tag=tag)
        self.inputs = qs
        self.scale = 1.0 / math.sqrt(D)
        # query / KV RMSNorm gains and partial RoPE (report §2.3.3): seeded
        # U(0.5, 1.5) gains, eps 1e-6, RoPE base 10000
        self.norm_rope = norm_rope
        self.q_gain = s.uniform(tag + "q_gain", (D,), 0.5, 1.5) if norm_rope else None
        self.kv_gain = s.uniform(tag + "kv_gain", (D,), 0.5, 1.5) if norm_rope else None
        self.norm_eps, self.rope_base = (1e-6, 10000.0) if norm_rope else (0.0, 0.0)
        self.seq_len = torch.tensor(ctx, dtype=torch.int32, device=device)
        self.pos = self.seq_len.clone()  # the new token's position
        self.max_pos = max(ctx)

        # classical cache: FP8 content + scale + BF16 RoPE entries (none in a window-only layer)
        self.kv = None
        if kind != "swa":
            self.kv = abi.make_pool(abi.FMT_KV_POOL_FP8, B, self.capacity, D, page_entries, device,
                                    shuffle_seed=seed)
            abi.csa_cache_write(st["entries"].contiguous(), self.kv)
        # state cache: window ring (slot = position % W) and tail gates (slot = position % m)
        self.ring = torch.empty((B, W, D), dtype=torch.bfloat16, device=device)
        for b, L in enumerate(ctx):
            slots = (torch.arange(L - W, L, device=device) % W).long()
            self.ring[b, slots] = st["window"][b]
        self.tail_gate = st["tail_gate"].contiguous()
        self.bias = st["bias"].contiguous()
        self.ws_kv = abi.compress_workspace(B, D, device)
        if kind == "csa":
            self.ki = abi.make_pool(index_fmt, B, self.capacity, d_idx, page_entries, device,
                                    shuffle_seed=seed + 1)
            abi.csa_cache_write(st["keys_idx"].contiguous(), self.ki)
            self.ring_idx = st["ring_idx"].contiguous()  # ring of size m: slot = position % m
            self.tail_gate_idx = st["tail_gate_idx"].contiguous()
            self.bias_idx = st["bias_idx"].contiguous()
            self.ws_idx = abi.compress_workspace(B, d_idx, device)
        # overlapping compression (report §2.3.1): a b stream per compressor, its
        # tail of two blocks (slot = position % 2m), seeded like the a stream
        self.overlap_ab = overlap_ab
        if overlap_ab:
            m2 = 2 * self.m
            ab = dict(tail_b=s.normal(tag + "tail_b", (B, m2, D), dtype=torch.bfloat16),
                      tail_gate_b=s.normal(tag + "tail_gate_b", (B, m2, D)),
                      tail_idx_b=s.normal(tag + "tail_idx_b", (B, m2, d_idx), dtype=torch.bfloat16),
                      tail_gate_idx_b=s.normal(tag + "tail_gate_idx_b", (B, m2, d_idx)))
            self.tail_b, self.tail_gate_b = ab["tail_b"], ab["tail_gate_b"]
            self.tail_idx_b, self.tail_gate_idx_b = ab["tail_idx_b"], ab["tail_gate_idx_b"]
            self.bias_b = s.normal(tag + "bias_b", (self.m, D), 0.1)
            self.bias_idx_b = s.normal(tag + "bias_idx_b", (self.m, d_idx), 0.1)
            qs.update(k_new_b=s.normal(tag + "k_new_b", (B, D), dtype=torch.bfloat16),
                      g_new_b=s.normal(tag + "g_new_b", (B, D)),
                      k_idx_new_b=s.normal(tag + "k_idx_new_b", (B, d_idx), dtype=torch.bfloat16),
                      g_idx_new_b=s.normal(tag + "g_idx_new_b", (B, d_idx)))
            st.update(ab)
            st.update(bias_b=self.bias_b, bias_idx_b=self.bias_idx_b)
        # host copies of the synthetic state of the listed sequences (for checks)
        keep = list(keep_sources)
        self.sources = {b: {k: v[b].detach().cpu() for k, v in st.items() if v.dim() >= 3 and v.shape[0] == B}
                        for b in keep}
        self.shared_sources = {k: v.detach().cpu() for k, v in st.items()
                               if k in ("bias", "bias_idx", "bias_b", "bias_idx_b")}
        del st

        # prepared calls
        if kind == "csa":
            q_idx = qs["q_idx"] if index_fmt == abi.FMT_INDEX_POOL_BF16 else qs["q_idx"].float()
            self._q_idx = q_idx
            # the kernels before the indexer and the attention in a step are this
            # library's (the appends, the indexer): they never write the step's
            # queries, so those calls may start early
            self.index = abi.IndexCall(q_idx, qs["w"], self.pos, self.ki, top_k, self.m, self.max_pos, B,
                                       score_dtype=score_dtype, overlap=True, after_append=True)
        prep = dict(q_norm=self.q_gain, win_norm=self.kv_gain, norm_eps=self.norm_eps, rope_base=self.rope_base,
                    batch_invariant=batch_invariant, overlap=True)
        if kind == "csa":
            self.attend = abi.AttendCall(True, qs["q"], self.pos, self.kv, W, self.ring, self.scale, self.m,
                                         self.max_pos, B, idx=self.index.idx, cnt=self.index.cnt, **prep)
        else:
            self.attend = abi.AttendCall(False, qs["q"], self.pos, self.kv, W, self.ring, self.scale, self.m,
                                         self.max_pos, B, window_only=(kind == "swa"), **prep)
        self.graph = None

    # ------------------------------------------------------------------ the step
    def launches_per_step(self) -> int:
        """Kernels one step launches: compress-append per stream, the score and
        top-k kernels (CSA), the attention kernel and, when its splits are
        merged by a second kernel, that kernel."""
        n = 2 + 2 if self.kind == "csa" else 1
        return n + self.attend.launches()

    def stages(self) -> list[str]:
        """Names of the kernel groups of one step, in launch order."""
        return ["compress", "index_score", "index_select", "attend"] if self.kind == "csa" else \
            ["compress", "attend"]

    def step(self, stream=None, marks=None):
        """One decode step.  marks: optional list of len(stages()) + 1 CUDA
        events recorded before the first and after every kernel group."""
        qs = self.inputs
        st = stream if stream is not None else torch.cuda.current_stream()
        mark = (lambda i: marks[i].record(st)) if marks is not None else (lambda i: None)  # noqa: E731
        mark(0)
        if self.kind == "swa":
            abi.csa_window_append(self.seq_len, qs["k_new"], self.ring, stream=stream)
        else:
            ab = {}
            if self.overlap_ab:
                ab = dict(bias_b=self.bias_b, k_new_b=qs["k_new_b"], g_new_b=qs["g_new_b"], tail_b=self.tail_b,
                          tail_gate_b=self.tail_gate_b)
            abi.csa_compress(self.kv, self.bias, self.m, seq_len=self.seq_len, k_new=qs["k_new"],
                             g_new=qs["g_new"], ring=self.ring, tail_gate=self.tail_gate, workspace=self.ws_kv,
                             stream=stream, norm=self.kv_gain, norm_eps=self.norm_eps, rope_base=self.rope_base, **ab)
        if self.kind == "csa":
            # the indexer-key append touches none of the KV append's buffers: it
            # runs alongside it
            ab = {}
            if self.overlap_ab:
                ab = dict(bias_b=self.bias_idx_b, k_new_b=qs["k_idx_new_b"], g_new_b=qs["g_idx_new_b"],
                          tail_b=self.tail_idx_b, tail_gate_b=self.tail_gate_idx_b)
            abi.csa_compress(self.ki, self.bias_idx, self.m, seq_len=self.seq_len, k_new=qs["k_idx_new"],
                             g_new=qs["g_idx_new"], ring=self.ring_idx, tail_gate=self.tail_gate_idx,
                             workspace=self.ws_idx, stream=stream, overlap=True, **ab)
            mark(1)
            self.index.score(stream)
            mark(2)
            self.index.select(stream)
            mark(3)
        else:
            mark(1)
        out, _ = self.attend(stream)
        mark(len(self.stages()))
        return out

    def capture(self, timed: bool = False):
        """Capture step() into a CUDA graph (after one eager warm-up step).
        With timed=True a second graph also records one CUDA event before the
        step and after each kernel group (stage_ms() reads them after
        replay_timed()).  The events sit between kernels, which breaks the
        early start of the next kernel, so the untimed graph is the one that
        gives the step's time."""
        self.step()
        torch.cuda.synchronize()
        self.graph = _capture(lambda s, marks: self.step(stream=s, marks=marks), None)
        self.marks = None
        self.graph_timed = None
        if timed:
            self.marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(self.stages()) + 1)]
            self.graph_timed = _capture(lambda s, marks: self.step(stream=s, marks=marks), self.marks)
        return self.graph

    def stage_ms(self) -> dict:
        """Device time of each kernel group in the last replay_timed()."""
        return {name: self.marks[i].elapsed_time(self.marks[i + 1]) for i, name in enumerate(self.stages())}

    def replay(self):
        if self.graph is None:
            return self.step()
        self.graph.replay()
        return self.attend.out

    def replay_timed(self):
        self.graph_timed.replay()
        return self.attend.out

    def step_inputs(self) -> dict:
        """The per-step input tensors the kernels read (new token, its gates,
        the queries and head weights)."""
        qs = self.inputs
        out = {"q": qs["q"], "k_new": qs["k_new"], "g_new": qs["g_new"]}
        if self.kind == "csa":
            out.update(q_idx=self._q_idx, w=qs["w"], k_idx_new=qs["k_idx_new"], g_idx_new=qs["g_idx_new"])
        if self.overlap_ab:
            out.update({k: qs[k] for k in ("k_new_b", "g_new_b", "k_idx_new_b", "g_idx_new_b")})
        return out

    def outputs(self) -> list:
        return [self.attend.out]

    # ------------------------------------------------------------------ bytes moved (algorithmic)
    def algorithmic_bytes(self) -> dict:
        """Bytes the method must move per step, by kernel (entries of 644 B,
        BF16 indexer keys 256 B or FP4 keys 72 B, window and query/output rows)."""
        B, D, H = self.B, self.D, self.H
        entry = 644
        nvis = [(c + 1) // self.m for c in self.ctx]
        win = sum(min(self.W, c + 1) for c in self.ctx)
        qo = B * H * D * 2 * 2
        out = {}
        if self.kind == "csa":
            kb = 256 if self.index_fmt == abi.FMT_INDEX_POOL_BF16 else 72
            out["index"] = sum(nvis) * kb + B * 64 * 128 * 2
            sel = sum(min(self.top_k, n) for n in nvis)
            out["attend"] = sel * entry + win * D * 2 + qo
        elif self.kind == "hca":
            out["attend"] = sum(nvis) * entry + win * D * 2 + qo
        else:  # window only
            out["attend"] = win * D * 2 + qo
        return out


def _capture(step, marks):
    """A CUDA graph of step(stream, marks) captured on a side stream."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step(s, marks)
    torch.cuda.current_stream().wait_stream(s)
    return g


# Hybrid interleave of the layers (report §4.2.1 / HF blog "Hybrid attention"):
# the first two layers are HCA, after which CSA and HCA alternate.
HYBRID_8 = ["hca", "hca", "csa", "hca", "csa", "hca", "csa", "hca"]
# The Flash model's 43 attention layers (report §4.2.1): the first two pure
# sliding-window attention, then CSA and HCA alternating from CSA.
FLASH_43 = ["swa", "swa"] + ["csa", "hca"] * 20 + ["csa"]


class HybridStack:
    """One decode step through a stack of CSA / HCA layers, each with its own
    paged caches, state cache and seeded per-layer inputs (no projections
    between layers: each layer's query is an independent input).

    CSA layers use top-k `top_k` over an indexer pool of format `index_fmt`
    (FP4 e2m1 with per-16 e4m3 scales by default, report §5.2.1)."""

    def __init__(self, B: int, ctx, seed: int = 0, kinds=tuple(HYBRID_8), top_k: int = 1024,
                 index_fmt: int = abi.FMT_INDEX_POOL_E2M1, score_dtype: int = abi.BF16, device: str = "cuda",
                 keep_sources=(), norm_rope: bool = False):
        self.kinds = list(kinds)
        self.B = B
        self.layers = []
        for i, kind in enumerate(self.kinds):
            self.layers.append(DecodeLayer(kind, B, ctx, seed=seed * 1000 + i, top_k=top_k, index_fmt=index_fmt,
                                           score_dtype=score_dtype, device=device, tag=f"layer{i}:",
                                           keep_sources=keep_sources, norm_rope=norm_rope))
            torch.cuda.synchronize()
        self.graph = None

    def stages(self) -> list[str]:
        out = []
        for i, layer in enumerate(self.layers):
            out += [f"L{i}.{name}" for name in layer.stages()]
        return out

    def launches_per_step(self) -> int:
        return sum(layer.launches_per_step() for layer in self.layers)

    def step(self, stream=None, marks=None):
        k = 0
        out = None
        for layer in self.layers:
            n = len(layer.stages())
            out = layer.step(stream, marks=None if marks is None else marks[k:k + n + 1])
            k += n
        return out

    def capture(self, timed: bool = False):
        """As DecodeLayer.capture, for the whole stack."""
        self.step()
        torch.cuda.synchronize()
        self.graph = _capture(lambda s, marks: self.step(stream=s, marks=marks), None)
        self.marks = None
        self.graph_timed = None
        if timed:
            self.marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(self.stages()) + 1)]
            self.graph_timed = _capture(lambda s, marks: self.step(stream=s, marks=marks), self.marks)
        return self.graph

    def replay(self):
        if self.graph is None:
            return self.step()
        self.graph.replay()
        return self.layers[-1].attend.out

    def replay_timed(self):
        self.graph_timed.replay()
        return self.layers[-1].attend.out

    def stage_ms(self) -> dict:
        return {name: self.marks[i].elapsed_time(self.marks[i + 1]) for i, name in enumerate(self.stages())}

    def algorithmic_bytes(self) -> dict:
        out = {}
        for i, layer in enumerate(self.layers):
            for k, v in layer.algorithmic_bytes().items():
                out[f"L{i}.{k}"] = v
        return out

    def step_inputs(self) -> dict:
        return {f"L{i}.{k}": v for i, layer in enumerate(self.layers) for k, v in layer.step_inputs().items()}

    def outputs(self) -> list:
        return [layer.attend.out for layer in self.layers]
