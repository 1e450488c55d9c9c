"""bsp_decode_attn_noalloc against bsp_decode_attn, through the C ABI.

The no-allocation entry point serves callers that cannot call cudaMalloc on
the decode path (engines that give the whole GPU to their KV pools at start-up,
plugins whose host runtime owns all device memory). It plans the step itself
and keeps its scratch in a fixed device array compiled into the library. This
file is collected last; it passes on its own in a fresh process and after the
other tests.
"""
import math

import numpy as np
import pytest
import torch

from beam_search_shared_gb300 import bsp, synth
from beam_search_shared_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3   # the tolerance the parity tests use


def _noalloc(step: DeviceStep, o, lse):
    c, wl = step.case, step.case.workload
    bsp.decode_attn_noalloc(step.geo, wl.batch, wl.beam_width, c.prefix_len, c.tail_len, c.prefix_pages,
                            step.max_tail, step.q, step.k_pool, step.v_pool, step.beam_pages, step.cache_indirection,
                            step.scale, o, lse, flags=bsp.FLAG_CHECK)


def _close(o, lse, o_ref, lse_ref):
    a, r = o.double(), o_ref.double()
    assert torch.all((a - r).abs() <= ATOL + RTOL * r.abs())
    both_inf = torch.isneginf(lse) & torch.isneginf(lse_ref)
    d = torch.where(both_inf, torch.zeros_like(lse), (lse - lse_ref).abs())
    assert torch.all(d <= LSE_TOL)


@pytest.mark.parametrize("name,batch,beams,seed", [("qwen3_0p6b_b64_w30", 8, 30, 1), ("qwen3_4b_fp16_d256", 3, 8, 2),
                                                   ("bucketed_prefix_p10000", 1, 1, 3)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(name, batch, beams, seed):
    wl = synth.WORKLOADS[name]
    if wl.batch > 1:
        wl = wl.scaled(batch).with_(beam_width=beams)
    outs = []
    for call in range(2):        # two calls in a row share (and overwrite) the scratch array
        case = synth.make_case(wl, 900 + 10 * seed + call, full_step=False, device="cuda")
        step = DeviceStep(case)
        step.make_plan()
        step.attend(flags=bsp.FLAG_CHECK)
        o = torch.full_like(step.o, float("nan"))
        lse = torch.full_like(step.lse, float("nan"))
        _noalloc(step, o, lse)
        torch.cuda.synchronize()
        _close(o, lse, step.o, step.lse)
        outs.append(o)
    assert not torch.equal(outs[0], outs[1])


def test_noalloc_rejects_steps_beyond_its_scratch():
    B = 64
    wl = synth.WORKLOADS["wide_beam_b128_w96"].scaled(B)      # ~50 MB of prompt partials > the fixed array
    P = np.full(B, 2900, np.int32)
    g = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, 2000, wl.dtype)
    pages = np.zeros((B, math.ceil(2900 / wl.page_size)), np.int32)
    R = B * wl.beam_width
    q = torch.zeros((R, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((8, wl.num_kv_heads, wl.page_size, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros((R, wl.num_q_heads), dtype=torch.float32, device="cuda")
    with pytest.raises(bsp.BspError, match="CAPACITY"):
        bsp.decode_attn_noalloc(g, B, wl.beam_width, P, np.zeros(B, np.int32), pages, 8, q, pool, pool,
                                None, None, 1 / math.sqrt(wl.head_dim), o, lse)
    assert torch.all(o == 0)
