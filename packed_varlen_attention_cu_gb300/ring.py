"""Zigzag context parallelism emulated on one GPU (host orchestration only).

The ring loop of "长序列训练与上下文并行": cp ranks each hold a zigzag shard
("03 · 长文负载均衡" §4.2-4.3: chunks r and 2cp-1-r of every document); at
ring step t rank r computes attention of its Q shard against the K/V shard of
rank (r - t) mod cp, and the step's partial (O, LSE) is merged into the
running result by online softmax.  Here the cp ranks are virtual and share
one GPU, so no K/V moves; every step of the path runs in libpva's kernels and
this module only sequences the calls on one stream.

Two launch schemes:
- per pair: one worklist build and one attention launch per (rank, step)
  pair (PVA_MASK_ZIGZAG_PAIR), one merge per rank and step;
- per step: Q, K and V in ring order (pva_zigzag_ring_map), one worklist
  build and one attention launch per ring step covering every rank
  (PVA_MASK_ZIGZAG_STEP), one merge per step over all rows.
Either scheme can merge in the attention epilogue instead of writing partials
(fused: pva_attn_fwd_accumulate).
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import api
from .workloads import MASK_ZIGZAG_PAIR, MASK_ZIGZAG_STEP


class ZigzagRing:
    """Buffers and calls of the emulated ring for one pack.

    step(q, k, v) runs the whole ring (shard maps, gathers, cp x cp partial
    attentions or cp ring-step attentions, merges) and leaves the merged
    fp32 result in rank-local order; outputs() gives it with the pack row of
    every local row."""

    def __init__(self, cu_np: np.ndarray, cp: int, hq: int, hkv: int, d: int,
                 c_tile: int = 0, dispatch: int = api.DISPATCH_DYNAMIC,
                 per_step: bool = True, fused: bool = False, device=None):
        dev = device or torch.device("cuda")
        self.cp, self.hq, self.hkv, self.d = cp, hq, hkv, d
        self.per_step, self.fused = per_step, fused
        self.dev = dev
        self.cu_np = np.ascontiguousarray(cu_np, dtype=np.int32)
        self.cu = torch.from_numpy(self.cu_np).to(dev)
        self.nd = self.cu_np.shape[0] - 1
        self.T = int(self.cu_np[-1])
        self.params = api.make_params(hq, hkv, num_ctas=0, c_tile=c_tile, dispatch=dispatch)
        self.lens = [api.zigzag_shard_len(self.cu_np, cp, r) for r in range(cp)]
        T, bf16, f32 = self.T, torch.bfloat16, torch.float32
        if per_step:
            self.ring_map = torch.empty((max(T, 1),), dtype=torch.int32, device=dev)
            self.q = torch.empty((T, hq, d), dtype=bf16, device=dev)
            self.k = torch.empty((T, hkv, d), dtype=bf16, device=dev)
            self.v = torch.empty((T, hkv, d), dtype=bf16, device=dev)
            self.acc_o = torch.empty((T, hq, d), dtype=f32, device=dev)
            self.acc_l = torch.empty((hq, T), dtype=f32, device=dev)
            self.masks = [api.make_mask(MASK_ZIGZAG_STEP, T, T, cp=cp, ring_step=t)
                          for t in range(cp)]
            self.wls = [api.alloc_worklist(self.nd, m, self.params, dev) for m in self.masks]
            if not fused:
                self.part_o = torch.empty_like(self.acc_o)
                self.part_l = torch.empty_like(self.acc_l)
        else:
            n = self.lens
            self.maps = [torch.empty((max(x, 1),), dtype=torch.int32, device=dev) for x in n]
            self.qs = [torch.empty((x, hq, d), dtype=bf16, device=dev) for x in n]
            self.ks = [torch.empty((x, hkv, d), dtype=bf16, device=dev) for x in n]
            self.vs = [torch.empty((x, hkv, d), dtype=bf16, device=dev) for x in n]
            self.acc_o = [torch.empty((x, hq, d), dtype=f32, device=dev) for x in n]
            self.acc_l = [torch.empty((hq, x), dtype=f32, device=dev) for x in n]
            self.masks = {(r, s): api.make_mask(MASK_ZIGZAG_PAIR, n[r], n[s], cp=cp, q_rank=r,
                                                k_rank=s)
                          for r in range(cp) for s in range(cp)}
            self.wls = {key: api.alloc_worklist(self.nd, m, self.params, dev)
                        for key, m in self.masks.items()}
            if not fused:
                nmax = max(n) if n else 1
                self.part_o = torch.empty((nmax, hq, d), dtype=f32, device=dev)
                self.part_l = torch.empty((hq * nmax,), dtype=f32, device=dev)

    # ------------------------------------------------------------ launches
    def launches_per_step(self) -> int:
        """Library kernels one step() launches."""
        cp, nb = self.cp, api.worklist_build_kernels(self.params)
        merges = 0 if self.fused else cp - 1
        if self.per_step:
            return 1 + 3 + cp * (nb + 1) + merges
        return cp * 4 + cp * cp * (nb + 1) + cp * merges

    def merge_rows_per_step(self) -> int:
        """(token, head) rows one step's merges read and write (0 when fused)."""
        if self.fused:
            return 0
        return (self.cp - 1) * self.T * self.hq

    def step(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, stream=None,
             merge_events: Optional[list] = None) -> None:
        """One pass of the ring over the pack (q, k, v in the pack's row order)."""
        st = stream or torch.cuda.current_stream()
        if self.per_step:
            self._step_ring_order(q, k, v, st, merge_events)
        else:
            self._step_pairs(q, k, v, st, merge_events)

    def _merge(self, acc_o, acc_l, po, pl, st, merge_events, rows):
        ev = None
        if merge_events is not None:
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record(st)
        api.merge_partials(acc_o, acc_l, po, pl, acc_o, acc_l, st)
        if ev is not None:
            ev[1].record(st)
            merge_events.append((ev[0], ev[1], rows))

    def _step_ring_order(self, q, k, v, st, merge_events):
        api.zigzag_ring_map(self.cu, self.cp, self.ring_map, st)
        api.gather_rows(q, self.ring_map, self.q, stream=st)
        api.gather_rows(k, self.ring_map, self.k, stream=st)
        api.gather_rows(v, self.ring_map, self.v, stream=st)
        for t in range(self.cp):
            m, wl = self.masks[t], self.wls[t]
            api.build_worklist(self.cu, m, self.params, wl, st)
            if t == 0:
                api.attn_fwd(self.q, self.k, self.v, self.cu, m, self.params, wl, self.acc_o,
                             self.acc_l, 0.0, None, st)
            elif self.fused:
                api.attn_fwd_accumulate(self.q, self.k, self.v, self.cu, m, self.params, wl,
                                        self.acc_o, self.acc_l, 0.0, None, st)
            else:
                api.attn_fwd(self.q, self.k, self.v, self.cu, m, self.params, wl, self.part_o,
                             self.part_l, 0.0, None, st)
                self._merge(self.acc_o, self.acc_l, self.part_o, self.part_l, st, merge_events,
                            self.T)

    def _step_pairs(self, q, k, v, st, merge_events):
        cp = self.cp
        for r in range(cp):
            # the map buffer has at least one entry; a rank may own no rows at all
            mp = self.maps[r][: self.lens[r]]
            api.zigzag_shard(self.cu, cp, r, self.maps[r], None, st)
            api.gather_rows(q, mp, self.qs[r], stream=st)
            api.gather_rows(k, mp, self.ks[r], stream=st)
            api.gather_rows(v, mp, self.vs[r], stream=st)
        for r in range(cp):
            n = self.lens[r]
            for t in range(cp):
                s = (r - t) % cp
                m, wl = self.masks[(r, s)], self.wls[(r, s)]
                api.build_worklist(self.cu, m, self.params, wl, st)
                if t == 0:
                    api.attn_fwd(self.qs[r], self.ks[s], self.vs[s], self.cu, m, self.params, wl,
                                 self.acc_o[r], self.acc_l[r], 0.0, None, st)
                elif self.fused:
                    api.attn_fwd_accumulate(self.qs[r], self.ks[s], self.vs[s], self.cu, m,
                                            self.params, wl, self.acc_o[r], self.acc_l[r], 0.0,
                                            None, st)
                else:
                    po = self.part_o[:n]
                    pl = self.part_l[: self.hq * n].view(self.hq, n)
                    api.attn_fwd(self.qs[r], self.ks[s], self.vs[s], self.cu, m, self.params, wl,
                                 po, pl, 0.0, None, st)
                    self._merge(self.acc_o[r], self.acc_l[r], po, pl, st, merge_events, n)

    def worklists(self):
        return list(self.wls.values()) if isinstance(self.wls, dict) else list(self.wls)

    # ------------------------------------------------------------ results
    def outputs(self):
        """The merged result in rank-local order: a list of (map, O, LSE) blocks,
        map[i] the pack row of block row i, O [n, Hq, d] and LSE [Hq, n] fp32
        (one block in ring order, or one per rank)."""
        if self.per_step:
            return [(self.ring_map[: self.T], self.acc_o, self.acc_l)]
        return [(self.maps[r][: self.lens[r]], self.acc_o[r], self.acc_l[r])
                for r in range(self.cp) if self.lens[r] > 0]
