"""Seeded synthetic workloads for the WeDLM window decode step.

This module is the only code shared by the CUDA path's tests/benchmark and
the CPU oracle.  It draws random numbers and lays them out; it holds none of
the step's arithmetic (no norm, no RoPE, no attention, no softmax, no
selection).  Every generator is seeded; the same seed gives the same arrays.

Shapes follow the workloads of the WeDLM pages ("WeDLM: Reconciling Diffusion
Language Models with Standard Causal Attention for Fast Inference", Method
section): a Qwen3-8B-shaped backbone with a paged prefix KV cache and a
fixed-size decoding window of W slots.  Weights are random-initialised
N(0, 0.02); norm gains are 1; cached prefix K/V pages are N(0, 1).

KV pool format (the interface both sides implement on their own): one pool
per layer, an array of `num_pages` pages, each page holding
`[2 (K, V)][n_kv_heads][page_block tokens][head_dim]` values.  Inside one
(page, K|V, kv head) block of `page_block * head_dim` values, element
(token t, dim d) sits at

    ((t // 8) * (head_dim // 8) + d // 8) * 64 + (t % 8) * 8 + d % 8

i.e. 8x8 tiles, tiles ordered token-group-major.  This module only fills
pools with random numbers, so it never needs that formula.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

__all__ = [
    "Shape", "Workload", "TINY", "QWEN3_8B", "WORKLOADS", "qwen3_layers",
    "make_weights_np", "make_weights_torch", "make_state_np",
    "make_pool_np", "make_pool_torch", "plant_targets", "plant_bias_for",
]


@dataclass(frozen=True)
class Shape:
    """Backbone shape.  `mask_id` defaults to vocab-1."""
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    qk_norm: bool
    rope_theta: float
    rms_eps: float = 1e-6
    dtype: str = "bf16"          # storage/arithmetic type of the CUDA path
    page_block: int = 16
    mask_id_: Optional[int] = None

    @property
    def mask_id(self) -> int:
        return self.vocab - 1 if self.mask_id_ is None else self.mask_id_

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def replace(self, **kw) -> "Shape":
        return dataclasses.replace(self, **kw)


# tiny single-layer parity shape: hidden 256, 4 q / 2 kv heads, head_dim 64,
# fp32, RoPE theta 1e4, vocab 1024; FFN 3x hidden (same ratio as Qwen3-8B).
TINY = Shape(n_layers=1, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
             ffn=768, vocab=1024, qk_norm=False, rope_theta=1e4, dtype="fp32")

# Qwen3-8B-shaped stack (random init): 36 layers, hidden 4096, 32 q / 8 kv
# heads of 128, FFN 12288, vocab 151936, QK-norm, RoPE theta 1e6, bf16.
QWEN3_8B = Shape(n_layers=36, hidden=4096, n_q_heads=32, n_kv_heads=8,
                 head_dim=128, ffn=12288, vocab=151936, qk_norm=True,
                 rope_theta=1e6, dtype="bf16")


def qwen3_layers(n: int) -> Shape:
    return QWEN3_8B.replace(n_layers=n)


@dataclass(frozen=True)
class Workload:
    """One synthetic decode-step workload.

    prefix: fixed cached prefix length, or (lo, hi) for per-sequence
    uniform lengths in [lo, hi].  masked: (lo, hi) inclusive range of the
    number of masked slots per sequence (drawn uniformly), or an int.
    """
    name: str
    shape: Shape
    batch: int
    window: int
    prefix: object
    masked: object
    shuffled_pages: bool = False
    all_masked_start: bool = False
    plant: bool = False
    steps: int = 1
    alpha: float = 0.01
    tau: float = 1.0
    seed: int = 0
    prefix_from_prefill: bool = False
    extra_pages: int = 0          # page-table headroom beyond prefix+window

    def describe(self) -> str:
        s = self.shape
        return (f"{self.name}: L={s.n_layers} H={s.hidden} nq={s.n_q_heads} "
                f"nkv={s.n_kv_heads} hd={s.head_dim} F={s.ffn} V={s.vocab} "
                f"{s.dtype} B={self.batch} W={self.window} prefix={self.prefix}")


WORKLOADS = {
    # tiny fp32 single layer, prefix 128 built by prefill, W=8 with 3 observed
    "tiny": Workload("tiny", TINY, batch=1, window=8, prefix=128, masked=5,
                     prefix_from_prefill=True, seed=0),
    # one Qwen3-8B-shaped layer, B=1, prefix 2048, W=16, 25-75% masked
    "one_layer": Workload("one_layer", qwen3_layers(1), batch=1, window=16,
                          prefix=2048, masked=(4, 12), seed=0),
    # ragged batch of 32, prefixes U[512, 8192], shuffled page tables
    "ragged": Workload("ragged", qwen3_layers(1), batch=32, window=16,
                       prefix=(512, 8192), masked=(4, 12),
                       shuffled_pages=True, seed=0),
    # full 36-layer stack, prefix 4096, W=16, batch 8, start all-masked,
    # 256 streaming steps
    "full_stack": Workload("full_stack", QWEN3_8B, batch=8, window=16,
                           prefix=4096, masked=16, all_masked_start=True,
                           steps=256, seed=0, extra_pages=256),
    # the full_stack shapes with 2 layers: small enough (about 3.5 GB on the
    # device) for profiler captures of the same kernels
    "two_layer": Workload("two_layer", qwen3_layers(2), batch=8, window=16,
                          prefix=4096, masked=16, all_masked_start=True,
                          steps=256, seed=0, extra_pages=256),
    # the low_entropy shapes with 2 layers, for profiler captures
    "two_layer_long": Workload("two_layer_long", qwen3_layers(2), batch=8, window=32,
                               prefix=32768, masked=32, all_masked_start=True,
                               plant=True, steps=256, tau=2.0, seed=0, extra_pages=512),
    # the low_entropy shapes with 1 layer (about 4 GB on the device), for
    # full-section profiler captures of single kernels
    "one_layer_long": Workload("one_layer_long", qwen3_layers(1), batch=8, window=32,
                               prefix=32768, masked=32, all_masked_start=True,
                               plant=True, steps=256, tau=2.0, seed=0, extra_pages=512),
    # low-entropy long context: prefix 32768, W=32, batch 8, planted
    # peaked next-token bias on a seeded counting sequence
    "low_entropy": Workload("low_entropy", QWEN3_8B, batch=8, window=32,
                            prefix=32768, masked=32, all_masked_start=True,
                            plant=True, steps=256, tau=2.0, seed=0,
                            extra_pages=512),
}


# --------------------------------------------------------------------------
# weights
# --------------------------------------------------------------------------
_WEIGHT_NAMES = ("w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down")


def _layer_shapes(s: Shape):
    return {
        "attn_norm": (s.hidden,),
        "w_q": (s.n_q_heads * s.head_dim, s.hidden),
        "w_k": (s.n_kv_heads * s.head_dim, s.hidden),
        "w_v": (s.n_kv_heads * s.head_dim, s.hidden),
        "q_norm": (s.head_dim,),
        "k_norm": (s.head_dim,),
        "w_o": (s.hidden, s.n_q_heads * s.head_dim),
        "ffn_norm": (s.hidden,),
        "w_gate": (s.ffn, s.hidden),
        "w_up": (s.ffn, s.hidden),
        "w_down": (s.hidden, s.ffn),
    }


def make_weights_np(s: Shape, seed: int = 0, std: float = 0.02,
                    norm_jitter: float = 0.0):
    """Random weights as float32 numpy arrays (small shapes only).

    Linear weights are [out_features][in_features] (nn.Linear order).
    Norm gains are 1 (+ optional uniform jitter so tests can see them).
    """
    rng = np.random.Generator(np.random.PCG64(seed))

    def lin(shape):
        return (rng.standard_normal(shape) * std).astype(np.float32)

    def gain(n):
        g = np.ones(n, np.float32)
        if norm_jitter:
            g += rng.uniform(-norm_jitter, norm_jitter, n).astype(np.float32)
        return g

    w = {"embed": lin((s.vocab, s.hidden)), "layers": []}
    for _ in range(s.n_layers):
        lw = {}
        for name, shp in _layer_shapes(s).items():
            lw[name] = gain(shp[0]) if len(shp) == 1 else lin(shp)
        w["layers"].append(lw)
    w["final_norm"] = gain(s.hidden)
    w["lm_head"] = lin((s.vocab, s.hidden))
    return w


def make_weights_torch(s: Shape, seed: int = 0, device="cuda", std=0.02,
                       norm_jitter: float = 0.0):
    """Random weights as torch tensors on `device` in the shape's dtype.

    Drawn with a seeded torch.Generator on that device (large shapes: the
    36-layer stack is 15 GB in bf16).
    """
    import torch
    dt = torch.bfloat16 if s.dtype == "bf16" else torch.float32
    g = torch.Generator(device=device)
    g.manual_seed(seed)

    def lin(shape):
        t = torch.empty(shape, dtype=dt, device=device)
        # draw in chunks of rows to bound the fp32 temporary
        rows = shape[0]
        step = max(1, (1 << 26) // max(1, shape[1]))
        for r0 in range(0, rows, step):
            r1 = min(rows, r0 + step)
            t[r0:r1] = (torch.randn((r1 - r0, shape[1]), generator=g,
                                    device=device) * std).to(dt)
        return t

    def gain(n):
        t = torch.ones(n, dtype=dt, device=device)
        if norm_jitter:
            t += ((torch.rand(n, generator=g, device=device) * 2 - 1)
                  * norm_jitter).to(dt)
        return t

    w = {"embed": lin((s.vocab, s.hidden)), "layers": []}
    for _ in range(s.n_layers):
        lw = {}
        for name, shp in _layer_shapes(s).items():
            lw[name] = gain(shp[0]) if len(shp) == 1 else lin(shp)
        w["layers"].append(lw)
    w["final_norm"] = gain(s.hidden)
    w["lm_head"] = lin((s.vocab, s.hidden))
    return w


# --------------------------------------------------------------------------
# decoder state: window, lengths, page tables
# --------------------------------------------------------------------------
def make_state_np(wl: Workload, seed: Optional[int] = None,
                  prefix_override=None):
    """Window arrays, prefix lengths and page tables for a workload.

    Returns dict with int32 tokens[B][W], int32 pos[B][W], uint8 obs[B][W],
    int32 seq_len[B], int32 page_table[B][max_pages], int num_pages.
    The window of sequence b covers logical positions seq_len[b] ..
    seq_len[b]+W-1; masked slots hold mask_id.
    """
    s = wl.shape
    rng = np.random.Generator(np.random.PCG64(wl.seed if seed is None else seed))
    B, W, blk = wl.batch, wl.window, s.page_block
    if prefix_override is not None:
        lens = np.asarray(prefix_override, np.int64).reshape(-1)
        assert lens.size == B
    elif isinstance(wl.prefix, tuple):
        lens = rng.integers(wl.prefix[0], wl.prefix[1] + 1, size=B)
    else:
        lens = np.full(B, int(wl.prefix))
    lens = lens.astype(np.int32)

    tokens = np.empty((B, W), np.int32)
    pos = np.empty((B, W), np.int32)
    obs = np.zeros((B, W), np.uint8)
    for b in range(B):
        pos[b] = lens[b] + np.arange(W)
        if wl.all_masked_start:
            n_masked = W
        elif isinstance(wl.masked, tuple):
            n_masked = int(rng.integers(wl.masked[0], wl.masked[1] + 1))
        else:
            n_masked = int(wl.masked)
        masked_slots = rng.choice(W, size=n_masked, replace=False)
        obs[b] = 1
        obs[b, masked_slots] = 0
        # observed tokens avoid the mask id
        tokens[b] = rng.integers(0, s.vocab - 1, size=W)
        tokens[b, obs[b] == 0] = s.mask_id

    max_pages = int(math.ceil((int(lens.max()) + W) / blk)) + wl.extra_pages
    pages_needed = [int(math.ceil((int(lens[b]) + W) / blk)) + wl.extra_pages
                    for b in range(B)]
    num_pages = int(sum(pages_needed))
    ids = np.arange(num_pages, dtype=np.int32)
    if wl.shuffled_pages:
        ids = rng.permutation(num_pages).astype(np.int32)
    page_table = np.full((B, max_pages), -1, np.int32)
    o = 0
    for b in range(B):
        n = pages_needed[b]
        page_table[b, :n] = ids[o:o + n]
        o += n
    return {"tokens": tokens, "pos": pos, "obs": obs, "seq_len": lens,
            "page_table": page_table, "num_pages": num_pages,
            "max_pages": max_pages}


def make_pool_np(s: Shape, num_pages: int, seed: int, layer: int = 0):
    """One layer's KV pool filled with N(0, 1) float32 (small shapes)."""
    rng = np.random.Generator(np.random.PCG64([seed, 7919, layer]))
    n = num_pages * 2 * s.n_kv_heads * s.page_block * s.head_dim
    return rng.standard_normal(n).astype(np.float32)


def make_pool_torch(s: Shape, num_pages: int, seed: int, layer: int = 0,
                    device="cuda"):
    """One layer's KV pool filled with N(0, 1) in the shape's dtype."""
    import torch
    dt = torch.bfloat16 if s.dtype == "bf16" else torch.float32
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000003 + 7919 * (layer + 1))
    n = num_pages * 2 * s.n_kv_heads * s.page_block * s.head_dim
    out = torch.empty(n, dtype=dt, device=device)
    step = 1 << 27
    for i in range(0, n, step):
        j = min(n, i + step)
        out[i:j] = torch.randn(j - i, generator=g, device=device).to(dt)
    return out


# --------------------------------------------------------------------------
# low-entropy regime: a planted counting sequence
# --------------------------------------------------------------------------
def plant_targets(pos: np.ndarray, s0: int) -> np.ndarray:
    """Target token of the seeded counting sequence at each logical position:
    (s0 + pos) mod 200 + 1000."""
    return ((s0 + np.asarray(pos, np.int64)) % 200 + 1000).astype(np.int32)


def plant_bias_for(vocab: int) -> float:
    """Bias that gives p_top = 0.95 over otherwise-equal logits:
    e^b / (e^b + V - 1) = 0.95  <=>  b = ln(19 (V - 1))."""
    return float(math.log(19.0 * (vocab - 1)))
