"""One decode step on the GPU through the C ABI: device buffers for a case, plan, append, attention.

Holds the device-resident state of a synthetic step (pools, page tables,
indirection, queries, new token rows) and calls the binding. Used by the tests,
the benchmark and ``__graft_entry__.smoke()``.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np
import torch

from . import bsp
from .synth import Case


class DeviceStep:
    def __init__(self, case: Case, device="cuda", max_tail: int = bsp.MAX_TAIL,
                 workspace: Optional[bsp.Workspace] = None):
        wl = case.workload
        self.case = case
        self.device = torch.device(device)
        dev = self.device
        self.geo = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, case.num_pages,
                                wl.dtype)
        self.max_tail = max_tail
        self.q = case.q.to(dev)
        self.k_pool = case.k_pool.to(dev)
        self.v_pool = case.v_pool.to(dev)
        R = wl.batch * wl.beam_width
        n, row = case.k_new.shape[0], wl.num_kv_heads * wl.head_dim
        self.k_new = case.k_new.to(dev).reshape(n, row)
        self.v_new = case.v_new.to(dev).reshape(n, row)
        self.out_cache_loc = torch.from_numpy(case.out_cache_loc).to(dev)
        self.beam_pages = torch.from_numpy(case.beam_pages).to(dev)
        self.cache_indirection = torch.from_numpy(case.cache_indirection).to(dev)
        self.o = torch.empty((R, wl.num_q_heads, wl.head_dim), dtype=self.q.dtype, device=dev)
        self.lse = torch.empty((R, wl.num_q_heads), dtype=torch.float32, device=dev)
        self.scale = 1.0 / math.sqrt(wl.head_dim)
        self.ws = workspace or bsp.Workspace(self.geo, max(1, wl.batch), wl.beam_width,
                                             case.prefix_pages.shape[1], device=dev)
        self.plan = None

    def make_plan(self, stream=None):
        c = self.case
        wl = c.workload
        self.plan = self.ws.plan(self.geo, wl.batch, wl.beam_width, c.prefix_len, c.tail_len, c.prefix_pages,
                                 self.max_tail, stream=stream)
        return self.plan

    def update_tails(self, tail_len, stream=None):
        """Per-step update of the current plan: new tail lengths, same prompts and pages."""
        bsp.plan_update_tails(self.plan, tail_len, stream=stream)
        return self.plan

    def fused_requests(self) -> np.ndarray:
        """Which requests the prompt kernel finishes, from a host-only plan of the same inputs."""
        c = self.case
        wl = c.workload
        plan, img = bsp.plan_build(self.geo, wl.batch, wl.beam_width, c.prefix_len, c.tail_len, c.prefix_pages,
                                   self.max_tail, self.plan.num_sms)
        return bsp.plan_requests(plan, img)[:, 5] != 0

    def append(self, events=None, stream=None):
        bsp.append_kv(self.plan, self.k_new, self.v_new, self.out_cache_loc, self.k_pool, self.v_pool,
                      events=events, stream=stream)

    def attend(self, flags: int = 0, events=None, stream=None):
        bsp.decode_attn(self.plan, self.q, self.k_pool, self.v_pool, self.beam_pages, self.cache_indirection,
                        self.scale, self.o, self.lse, flags=flags, events=events, stream=stream)

    def run(self, flags: int = 0, stream=None):
        """plan + append (full steps) + attention, then the device status (syncs)."""
        self.make_plan(stream)
        if self.case.full_step:
            self.append(stream=stream)
        self.attend(flags, stream=stream)
        return bsp.read_device_status(self.plan, clear=True, stream=stream)


def algorithmic_bytes(case: Case, fused: Optional[np.ndarray] = None) -> dict:
    """Bytes each kernel must move at least once, from the drawn lengths.

    fused[b]: request b is finished by the prompt kernel (default: none is).
    prefix: valid K+V prompt rows once per (request, kv head) + Q; per request either the fp32
            partial O/LSE write or, when fused, its beams' K+V tail rows + the final O/LSE write;
    tail:   for the other requests, gathered K+V tail rows per (beam, kv head) + Q + partial
            read + O/LSE write;
    append: read + write of the new K and V rows.
    """
    wl = case.workload
    e = 2
    D, Hq, Hkv, W = wl.head_dim, wl.num_q_heads, wl.num_kv_heads, wl.beam_width
    P = case.prefix_len.astype(np.int64)
    T = case.tail_len.astype(np.int64)
    B = wl.batch
    fz = np.zeros(B, bool) if fused is None else np.asarray(fused, bool)
    active = P > 0
    row_kv = Hkv * D * e * 2              # K + V of one position, every kv head
    row_q = Hq * D * e                    # one beam row's queries
    row_part = Hq * (D + 1) * 4           # one beam row's fp32 partial O and LSE
    row_out = Hq * (D * e + 4)            # one beam row's final O and LSE
    prefix_kv = int(np.sum(P)) * row_kv
    pa = active & ~fz
    prefix = (prefix_kv + int(np.sum(active)) * W * row_q + int(np.sum(pa)) * W * row_part
              + int(np.sum(T[fz])) * W * row_kv + int(np.sum(fz)) * W * row_out)
    tl = ~fz
    tail = (int(np.sum(T[tl])) * W * row_kv + int(np.sum(tl)) * W * (row_q + row_out)
            + int(np.sum(pa)) * W * row_part)
    n = int(case.out_cache_loc.shape[0])
    append = n * Hkv * D * e * 2 * 2
    flops = (int(np.sum(P)) + int(np.sum(T[fz]))) * W * Hq * D * 4
    return {"prefix": prefix, "tail": tail, "append": append, "prefix_flops": flops,
            "prefix_kv": prefix_kv}


class PrefillStep:
    """Device buffers of one synthetic prefill (synth.PrefillCase), its plan, append and attention."""

    def __init__(self, case, device="cuda"):
        wl = case.workload
        self.case = case
        dev = torch.device(device)
        self.geo = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, case.num_pages,
                                wl.dtype)
        self.q = case.q.to(dev)
        self.k_pool = case.k_pool.to(dev)
        self.v_pool = case.v_pool.to(dev)
        R, row = case.rows, wl.num_kv_heads * wl.head_dim
        self.k_new = case.k_new.to(dev).reshape(R, row)
        self.v_new = case.v_new.to(dev).reshape(R, row)
        self.out_cache_loc = torch.from_numpy(case.out_cache_loc).to(dev)
        self.o = torch.empty((R, wl.num_q_heads, wl.head_dim), dtype=self.q.dtype, device=dev)
        self.lse = torch.empty((R, wl.num_q_heads), dtype=torch.float32, device=dev)
        self.scale = 1.0 / math.sqrt(wl.head_dim)
        self.ws = bsp.Workspace(self.geo, max(1, wl.batch), max(1, int(case.prompt_len.max(initial=0))),
                                case.pages.shape[1], device=dev)
        self.plan = None

    def make_plan(self, stream=None):
        c = self.case
        self.plan = bsp.plan_prefill(self.geo, c.workload.batch, c.cached_len, c.prompt_len, c.pages,
                                     c.workload.causal, self.ws, stream=stream)
        return self.plan

    def append(self, stream=None):
        bsp.append_kv(self.plan, self.k_new, self.v_new, self.out_cache_loc, self.k_pool, self.v_pool, stream=stream)

    def attend(self, flags: int = 0, events=None, stream=None):
        bsp.prefill_attn(self.plan, self.q, self.k_pool, self.v_pool, self.scale, self.o, self.lse, flags=flags,
                         events=events, stream=stream)

    def run(self, flags: int = 0, stream=None):
        """plan + append of the prompt's K/V + attention, then the device status (syncs)."""
        self.make_plan(stream)
        self.append(stream)
        self.attend(flags, stream=stream)
        return bsp.read_device_status(self.plan, clear=True, stream=stream)


def prefill_work(case) -> dict:
    """Algorithmic bytes and flops of a prefill attention (the prompt kernel): each (request, kv head)
    reads its keys' K and V once, plus Q and O/LSE; the flops count
    only the (row, key) pairs the mask keeps (Q*K^T and P*V, 2 flops per multiply-add)."""
    wl = case.workload
    e = 2
    D, Hq, Hkv = wl.head_dim, wl.num_q_heads, wl.num_kv_heads
    C = case.cached_len.astype(np.int64)
    S = case.prompt_len.astype(np.int64)
    if wl.causal:
        pairs = int(np.sum(C * S + S * (S + 1) // 2))
    else:
        pairs = int(np.sum(S * (C + S)))
    kv_bytes = int(np.sum(np.where(S > 0, C + S, 0))) * Hkv * D * e * 2   # each key once per kv head
    io_bytes = int(S.sum()) * Hq * (D * e * 2 + 4)                         # Q in, O and LSE out
    return {"bytes": kv_bytes + io_bytes, "flops": pairs * Hq * D * 4, "pairs": pairs}
