"""Seeded synthetic inputs for the CSA / HCA workloads.

This module only draws random numbers and arranges them in the shapes of the
workloads; it holds none of the method's arithmetic (no pooling, scoring,
selection, attention or quantization).  Both the CUDA path and the CPU oracle
take their inputs from here, so the two sides always see the same values.

Every named draw gets its own generator, seeded from (seed, name), so a draw
does not depend on the order of the calls.  On the CPU the generator is
numpy's counter-based Philox; on a CUDA device it is torch's Philox.  The two
give different numbers for the same seed; a run uses one device throughout
and hands the oracle host copies of exactly the tensors the kernels got.

Workload shapes follow the model settings of the DeepSeek-V4 report (cnblogs
translation, §4.2.1): m = 4, m' = 128, 64 indexer heads of dim 128, 64 query
heads, head dim 512 + 64 RoPE, n_win = 128.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np
import torch


def _key(seed: int, name: str) -> int:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


@dataclass
class Synth:
    seed: int = 0
    device: str = "cpu"

    def _gen(self, name):
        k = _key(self.seed, name)
        if self.device == "cpu":
            return np.random.Generator(np.random.Philox(k))
        g = torch.Generator(device=self.device)
        g.manual_seed(k)
        return g

    def normal(self, name, shape, std=1.0, dtype=torch.float32):
        g = self._gen(name)
        if self.device == "cpu":
            x = torch.from_numpy(g.standard_normal(size=shape, dtype=np.float32))
        else:
            x = torch.randn(shape, generator=g, device=self.device, dtype=torch.float32)
        if std != 1.0:
            x = x * std
        return x.to(dtype)

    def uniform(self, name, shape, lo=0.0, hi=1.0):
        g = self._gen(name)
        if self.device == "cpu":
            x = torch.from_numpy(g.random(size=shape, dtype=np.float32))
        else:
            x = torch.rand(shape, generator=g, device=self.device, dtype=torch.float32)
        return x * (hi - lo) + lo

    def integers(self, name, lo, hi, shape):
        """Uniform integers in [lo, hi)."""
        g = self._gen(name)
        if self.device == "cpu":
            return torch.from_numpy(g.integers(lo, hi, size=shape).astype(np.int64))
        return torch.randint(lo, hi, shape, generator=g, device=self.device)

    def subset_sorted(self, name, n, k, rows):
        """``rows`` independent sorted random subsets of size min(k, n) of
        range(n), padded with -1 to width k (int32)."""
        out = torch.full((rows, k), -1, dtype=torch.int32)
        kk = min(k, n)
        gen = np.random.Generator(np.random.Philox(_key(self.seed, name)))
        for r in range(rows):
            out[r, :kk] = torch.from_numpy(np.sort(gen.choice(n, size=kk, replace=False)).astype(np.int32))
        return out.to(self.device)

    def outlier_mask(self, name, n, frac=0.01):
        """Boolean [n] with round(frac * n) positions set, chosen at random."""
        gen = np.random.Generator(np.random.Philox(_key(self.seed, name)))
        cnt = int(round(frac * n))
        mask = np.zeros(n, dtype=bool)
        mask[gen.choice(n, size=cnt, replace=False)] = True
        return torch.from_numpy(mask).to(self.device)


# ------------------------------------------------------------------ workload recipes


def csa_prefill_f32(seed=0, n=2048, D=192, d_idx=64, H_idx=4, H=16, m=4, device="cpu"):
    """Single-layer CSA prefill, float32 throughout.

    Raw KV tokens and gate logits N(0,1) [n, D]; position bias N(0, 0.1) [m, D];
    the indexer-key stream the same way with dim d_idx; indexer queries N(0,1)
    [n, H_idx, d_idx]; one head-weight vector U(0,1) [H_idx] shared by all
    queries; attention queries N(0,1) [n, H, D]."""
    s = Synth(seed, device)
    return dict(
        k=s.normal("k", (n, D)), g=s.normal("g", (n, D)), bias=s.normal("bias", (m, D), 0.1),
        k_idx=s.normal("k_idx", (n, d_idx)), g_idx=s.normal("g_idx", (n, d_idx)),
        bias_idx=s.normal("bias_idx", (m, d_idx), 0.1),
        q_idx=s.normal("q_idx", (n, H_idx, d_idx)), w=s.uniform("w", (H_idx,)),
        q=s.normal("q", (n, H, D)),
    )


def decode_queries(seed, B, H=64, D=576, H_idx=64, d_idx=128, device="cpu", tag=""):
    """One new query token per sequence: attention query bf16 [B, H, D],
    indexer query bf16 [B, H_idx, d_idx], head weights U(0,1) [B, H_idx],
    and the new raw token with its gate logits (bf16 / f32 [B, D]) for the KV
    stream and the indexer stream."""
    s = Synth(seed, device)
    return dict(
        q=s.normal(tag + "q", (B, H, D), dtype=torch.bfloat16),
        q_idx=s.normal(tag + "q_idx", (B, H_idx, d_idx), dtype=torch.bfloat16),
        w=s.uniform(tag + "w", (B, H_idx)),
        k_new=s.normal(tag + "k_new", (B, D), dtype=torch.bfloat16),
        g_new=s.normal(tag + "g_new", (B, D)),
        k_idx_new=s.normal(tag + "k_idx_new", (B, d_idx), dtype=torch.bfloat16),
        g_idx_new=s.normal(tag + "g_idx_new", (B, d_idx)),
    )


def decode_context(seed, B, n_entries, W=128, m=4, D=576, d_idx=128, device="cpu", tag="",
                   with_index=True, entries_dtype=torch.float32):
    """State of B sequences before a decode step.

    Compressed entries N(0,1) [B, n_entries, D] as float32 values (the cache
    writer stores them as FP8 content + per-entry scale + BF16 RoPE dims);
    compressed indexer keys N(0,1) [B, n_entries, d_idx]; the last W raw tokens
    bf16 [B, W, D] in position order (oldest first); the gate logits of the
    uncompressed tail f32 [B, m, D]; the indexer stream's last m raw keys and
    tail gates; and per-stream position biases N(0, 0.1)."""
    s = Synth(seed, device)
    out = dict(
        entries=s.normal(tag + "entries", (B, n_entries, D), dtype=entries_dtype),
        window=s.normal(tag + "window", (B, W, D), dtype=torch.bfloat16),
        tail_gate=s.normal(tag + "tail_gate", (B, m, D)),
        bias=s.normal(tag + "bias", (m, D), 0.1),
    )
    if with_index:
        out.update(
            keys_idx=s.normal(tag + "keys_idx", (B, n_entries, d_idx)),
            ring_idx=s.normal(tag + "ring_idx", (B, m, d_idx), dtype=torch.bfloat16),
            tail_gate_idx=s.normal(tag + "tail_gate_idx", (B, m, d_idx)),
            bias_idx=s.normal(tag + "bias_idx", (m, d_idx), 0.1),
        )
    return out
