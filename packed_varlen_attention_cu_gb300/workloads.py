"""Seeded synthetic inputs for packed document-masked attention.

This module only draws inputs: document lengths, cu_seqlens and bf16 Q/K/V
tensors.  It holds none of the method's arithmetic (no masks, no pair counts,
no softmax), so both the CUDA path and the CPU oracle can take their inputs
from it without sharing any computation.

Document-length recipe (used for every lognormal workload): draw
``round(lognormal(mu, sigma))`` from ``numpy.random.default_rng(seed)``, clip
to ``[lo, hi]``, and keep drawing until the running total reaches the pack
length; the last document is shortened to fill the pack exactly (it may end up
below the clip floor).  Values are ``torch.randn`` (fp32, seeded generator)
times a scale, rounded to bf16 (round-to-nearest-even).

Workloads follow the long-context load-balancing pages
("03 · 长文负载均衡", §1.1: the Libra 40K-vs-ten-4K example and the
median-644 production corpus; §1.2: sliding-window and shared-question masks;
§4.2-4.3: zigzag context parallelism).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

# Mask kinds.  The integer values are the interface agreement shared by the
# C header, the binding and the oracle (each side keeps its own copy).
MASK_CAUSAL = 0
MASK_SLIDING_WINDOW = 1
MASK_SHARED_QUESTION = 2
MASK_ZIGZAG_PAIR = 3
MASK_SLICES = 4
MASK_ZIGZAG_STEP = 5


def lognormal_doc_lengths(total: int, mu: float, sigma: float, lo: int, hi: int,
                          seed: int) -> List[int]:
    """Document lengths of one pack of ``total`` tokens (recipe in the module doc)."""
    rng = np.random.default_rng(seed)
    out: List[int] = []
    acc = 0
    while acc < total:
        ell = int(np.clip(round(rng.lognormal(mu, sigma)), lo, hi))
        if acc + ell >= total:
            ell = total - acc
        out.append(ell)
        acc += ell
    return out


def cu_seqlens_of(lengths: Sequence[int]) -> np.ndarray:
    """Exclusive prefix offsets [0, l0, l0+l1, ...] as int32."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    assert cu[-1] < 2**31
    return cu.astype(np.int32)


@dataclasses.dataclass
class Workload:
    """A named packed-attention workload: lengths, heads, dims and mask."""
    name: str
    lengths: List[int]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    mask_kind: int = MASK_CAUSAL
    window: int = 0
    num_prefix_docs: int = 0
    cp: int = 0
    value_scale: float = 1.0
    seed: int = 0

    @property
    def total_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def cu_seqlens(self) -> np.ndarray:
        return cu_seqlens_of(self.lengths)

    @property
    def num_docs(self) -> int:
        return len(self.lengths)


def tiny_pack(seed: int = 0) -> Workload:
    """2048-token pack, lognormal(5, 1) lengths clipped to [16, 1024], 4 heads, d=64."""
    return Workload("tiny pack T=2048 H=4/4 d=64",
                    lognormal_doc_lengths(2048, 5.0, 1.0, 16, 1024, seed),
                    4, 4, 64, seed=seed)


def libra_pair() -> Workload:
    """Pack A (one 40960-token doc) followed by pack B (ten 4096-token docs)."""
    return Workload("libra pair 1x40960 + 10x4096 H=16/16 d=128",
                    [40960] + [4096] * 10, 16, 16, 128, value_scale=0.5)


def long_tail_gqa(num_packs: int = 8) -> Workload:
    """``num_packs`` packs of 32768 tokens (seeds 0..n-1), median 644, sigma 1.6, GQA 14:2, d=64."""
    lengths: List[int] = []
    for s in range(num_packs):
        lengths += lognormal_doc_lengths(32768, math.log(644.0), 1.6, 32, 32768, s)
    return Workload(f"long-tail GQA {num_packs}x32768 H=14/2 d=64", lengths, 14, 2, 64)


def zigzag_pack(seed: int = 0) -> Workload:
    """131072-token pack, median 2048, sigma 1.5, clip [1, 65536], 32 q / 8 kv heads, d=128, cp=8."""
    return Workload("128K causal pack H=32/8 d=128",
                    lognormal_doc_lengths(131072, math.log(2048.0), 1.5, 1, 65536, seed),
                    32, 8, 128, cp=8, seed=seed)


def shared_question() -> Workload:
    """One 4096-token question followed by eight 2048-token answers, 16 q / 4 kv heads, d=128."""
    return Workload("shared question 4096+8x2048 H=16/4 d=128", [4096] + [2048] * 8,
                    16, 4, 128, mask_kind=MASK_SHARED_QUESTION, num_prefix_docs=1)


def sliding_window() -> Workload:
    """Four documents (131072, 65536, 49152, 16384) under a causal window of 4096."""
    return Workload("sliding window 4 docs T=262144 w=4096 H=16/4 d=128",
                    [131072, 65536, 49152, 16384], 16, 4, 128,
                    mask_kind=MASK_SLIDING_WINDOW, window=4096)


def short_docs(seed: int = 0) -> Workload:
    """131072-token pack of short documents (lognormal median 64, sigma 0.75, clip [8, 512]),
    32 q / 8 kv heads, d=128: many documents shorter than a 128-row tile."""
    return Workload("short-document pack T=131072 H=32/8 d=128",
                    lognormal_doc_lengths(131072, math.log(64.0), 0.75, 8, 512, seed),
                    32, 8, 128, seed=seed)


def make_qkv(total_q: int, total_k: int, hq: int, hkv: int, d: int, seed: int,
             scale: float = 1.0, device: str = "cpu"):
    """bf16 Q [Tq,Hq,d], K and V [Tk,Hkv,d] drawn N(0,1)*scale from a seeded generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    q = torch.randn((total_q, hq, d), generator=g, device=device, dtype=torch.float32)
    k = torch.randn((total_k, hkv, d), generator=g, device=device, dtype=torch.float32)
    v = torch.randn((total_k, hkv, d), generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        q *= scale
        k *= scale
        v *= scale
    return (q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16))


def workload_qkv(w: Workload, device: str = "cpu"):
    """Q, K, V for a workload (same seed on any device gives the same draw per device type)."""
    t = w.total_tokens
    return make_qkv(t, t, w.num_q_heads, w.num_kv_heads, w.head_dim, w.seed,
                    w.value_scale, device)


def random_rows(total: int, heads: int, count: int, seed: int,
                must_include: Optional[Sequence[int]] = None) -> np.ndarray:
    """Seeded sample of (row, head) pairs, int32 [n, 2], for sampled parity checks."""
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, total, size=count)
    hs = rng.integers(0, heads, size=count)
    out = np.stack([rows, hs], axis=1)
    if must_include:
        extra = np.array([[r % total, i % heads] for i, r in enumerate(must_include)])
        out = np.concatenate([out, extra], axis=0)
    return out.astype(np.int32)
