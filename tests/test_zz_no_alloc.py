"""bsp_decode_attn_noalloc through the C ABI: against the workspace entry point and the oracle.

The no-allocation entry point serves callers that cannot call cudaMalloc on
the decode path (engines that give the whole GPU to their KV pools at start-up,
plugins whose host runtime owns all device memory). It plans the step itself
and keeps its scratch in a fixed device array compiled into the library. This
file is collected last; it passes on its own in a fresh process and after the
other tests.
"""
import math
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import oracle
from beam_search_shared_gb300 import bsp, synth
from beam_search_shared_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3   # the tolerance the parity tests use
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _noalloc(step: DeviceStep, o, lse, stream=None):
    c, wl = step.case, step.case.workload
    bsp.decode_attn_noalloc(step.geo, wl.batch, wl.beam_width, c.prefix_len, c.tail_len, c.prefix_pages,
                            step.max_tail, step.q, step.k_pool, step.v_pool, step.beam_pages, step.cache_indirection,
                            step.scale, o, lse, flags=bsp.FLAG_CHECK, stream=stream)


def _close(o, lse, o_ref, lse_ref):
    a, r = o.double(), o_ref.double()
    assert torch.all((a - r).abs() <= ATOL + RTOL * r.abs())
    both_inf = torch.isneginf(lse) & torch.isneginf(lse_ref)
    d = torch.where(both_inf, torch.zeros_like(lse), (lse - lse_ref).abs())
    assert torch.all(d <= LSE_TOL)


def _oracle(case):
    wl = case.workload
    return oracle.decode_attn(
        dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
        ps=wl.page_size, num_pages=case.num_pages, prefix_len=case.prefix_len, tail_len=case.tail_len,
        prefix_pages=case.prefix_pages, beam_pages=case.beam_pages, cache_indirection=case.cache_indirection,
        q_bits=synth.bits(case.q), k_pool_bits=synth.bits(case.k_pool), v_pool_bits=synth.bits(case.v_pool),
        scale=1 / math.sqrt(wl.head_dim))


@pytest.mark.parametrize("name,batch,beams,seed", [("qwen3_0p6b_b64_w30", 8, 30, 1), ("qwen3_4b_fp16_d256", 3, 8, 2),
                                                   ("bucketed_prefix_p10000", 1, 1, 3)])
def test_noalloc_matches_workspace_entry_point_and_oracle_on_two_calls(name, batch, beams, seed):
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
        _close(o, lse, step.o, step.lse)            # the workspace entry point, same tolerance
        O, L = _oracle(case)                         # and the fp64 oracle
        _close(o, lse, torch.from_numpy(O).to(o.device), torch.from_numpy(L).to(lse.device).float())
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


def test_noalloc_refuses_a_capturing_stream():
    """Each call copies its plan from one shared host array, so a call on a capturing stream is refused
    before anything is enqueued (the capture itself stays valid)."""
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(2)
    case = synth.make_case(wl, 931, full_step=False, device="cuda")
    step = DeviceStep(case)
    o = torch.zeros_like(step.o)
    lse = torch.zeros_like(step.lse)
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    refused = None
    with torch.cuda.graph(g, stream=side):
        o.add_(1.0)  # one captured op, so the graph is not empty
        try:
            _noalloc(step, o, lse, stream=side)
        except bsp.BspError as e:
            refused = e
    assert refused is not None and "INVALID_ARG" in str(refused)
    g.replay()
    torch.cuda.synchronize()
    assert torch.all(o == 1.0)                     # only the captured op ran
    # outside capture the same call works
    _noalloc(step, o, lse)
    torch.cuda.synchronize()
    O, L = _oracle(case)
    _close(o, lse, torch.from_numpy(O).to(o.device), torch.from_numpy(L).to(lse.device).float())


_MEMCHECK = textwrap.dedent("""
    import json, math, sys
    sys.path.insert(0, {root!r})
    import torch
    from beam_search_shared_gb300 import bsp, synth
    from beam_search_shared_gb300.step import DeviceStep
    torch.cuda.set_device(0)
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(4)
    case = synth.make_case(wl, 77, full_step=False, device="cuda")
    step = DeviceStep(case)
    o = torch.zeros_like(step.o)
    lse = torch.zeros_like(step.lse)
    def call():
        c = step.case
        bsp.decode_attn_noalloc(step.geo, wl.batch, wl.beam_width, c.prefix_len, c.tail_len, c.prefix_pages,
                                step.max_tail, step.q, step.k_pool, step.v_pool, step.beam_pages,
                                step.cache_indirection, step.scale, o, lse, flags=bsp.FLAG_CHECK)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    free = [torch.cuda.mem_get_info()[0]]
    # the documented set-up call: batch 0 only looks the scratch array up
    bsp.decode_attn_noalloc(step.geo, 0, wl.beam_width, [], [], [], step.max_tail, step.q, step.k_pool,
                            step.v_pool, None, None, step.scale, o, lse)
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
    call()   # first launches load the kernels' code
    free.append(torch.cuda.mem_get_info()[0])
    call()
    free.append(torch.cuda.mem_get_info()[0])
    call()
    free.append(torch.cuda.mem_get_info()[0])
    print(json.dumps({{"free": free, "torch_allocated": torch.cuda.memory_allocated()}}))
""")


def test_noalloc_allocates_nothing_after_setup():
    """In a fresh process: after the set-up call (batch 0) and one warm call, further calls leave the
    device's free memory unchanged."""
    r = subprocess.run([sys.executable, "-c", _MEMCHECK.format(root=ROOT)], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    import json
    d = json.loads(r.stdout.strip().splitlines()[-1])
    free = d["free"]
    # the set-up call is where the lazily loaded array lands on the device (nothing is freed by it)
    assert free[1] <= free[0]
    assert free[3] == free[2] and free[4] == free[2], free
