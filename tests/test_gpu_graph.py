"""CUDA-graph mode (BSP_FLAG_GRAPH): the attention launches are captured once and replayed after new
plans of the same shape, each replay checked against the oracle; a plan of another shape is refused on
the device (nothing written, BSP_DEVFLAG_GRAPH)."""
import math

import numpy as np
import pytest
import torch

import oracle
from beam_search_shared_gb300 import bsp, synth
from beam_search_shared_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3


def oracle_attn(case, P, T):
    wl = case.workload
    return oracle.decode_attn(
        dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
        ps=wl.page_size, num_pages=case.num_pages, prefix_len=P, tail_len=T, prefix_pages=case.prefix_pages,
        beam_pages=case.beam_pages, cache_indirection=case.cache_indirection, q_bits=synth.bits(case.q),
        k_pool_bits=synth.bits(case.k_pool), v_pool_bits=synth.bits(case.v_pool), scale=1 / math.sqrt(wl.head_dim))


@pytest.mark.parametrize("name,batch", [("qwen3_4b_fp16_d128", 4), ("qwen3_0p6b_b64_w30", 16), ("tiny_b1_w4_d64", 1),
                                        ("wide_beam_b128_w96", 2)])
def test_graph_replay_after_new_plans(name, batch):
    wl = synth.WORKLOADS[name].scaled(batch)
    case = synth.make_case(wl, 77 + batch, full_step=False, device="cuda")
    st = DeviceStep(case)
    P0, T0 = case.prefix_len.copy(), case.tail_len.copy()
    rng = np.random.default_rng(batch)
    st.plan = st.ws.plan(st.geo, wl.batch, wl.beam_width, P0, T0, case.prefix_pages, bsp.MAX_TAIL)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bsp.decode_attn(st.plan, st.q, st.k_pool, st.v_pool, st.beam_pages, st.cache_indirection, st.scale, st.o,
                        st.lse, flags=bsp.FLAG_GRAPH)
    trials = [(P0, T0), (P0 // 3, np.minimum(T0 + 3, bsp.MAX_TAIL)), (np.zeros_like(P0), T0),
              (P0, np.zeros_like(T0)), (rng.integers(0, P0 + 1).astype(np.int32), rng.integers(0, bsp.MAX_TAIL + 1, P0.shape).astype(np.int32))]
    for P, T in trials:
        P = np.asarray(P, np.int32)
        # tail positions stay inside the case's tables (cache_indirection is drawn for positions < P0 + T0)
        T = np.minimum(np.asarray(T, np.int32), P0 + T0 - P).astype(np.int32)
        st.ws.plan(st.geo, wl.batch, wl.beam_width, P, T, case.prefix_pages, bsp.MAX_TAIL)   # outside the graph
        st.o.fill_(float("nan"))
        g.replay()
        assert bsp.read_device_status(st.plan) == (0, 0)
        O, L = oracle_attn(case, P, T)
        o = st.o.double().cpu().numpy()
        lse = st.lse.double().cpu().numpy()
        assert np.isfinite(o).all()
        err = np.abs(o - O)
        assert (err <= ATOL + RTOL * np.abs(O)).all(), (P.tolist(), T.tolist(), err.max())
        both = np.isneginf(lse) & np.isneginf(L)
        np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(L))
        assert (np.abs(lse[~both] - L[~both]) <= LSE_TOL).all()


def test_graph_replay_refuses_another_shape():
    wl = synth.WORKLOADS["qwen3_4b_fp16_d128"].scaled(4)
    case = synth.make_case(wl, 5, full_step=False, device="cuda")
    st = DeviceStep(case)
    st.plan = st.ws.plan(st.geo, wl.batch, wl.beam_width, case.prefix_len, case.tail_len, case.prefix_pages,
                         bsp.MAX_TAIL)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bsp.decode_attn(st.plan, st.q, st.k_pool, st.v_pool, st.beam_pages, st.cache_indirection, st.scale, st.o,
                        st.lse, flags=bsp.FLAG_GRAPH)
    # a plan of three requests on the same workspace: the captured launches are for four
    st.ws.plan(st.geo, 3, wl.beam_width, case.prefix_len[:3], case.tail_len[:3], case.prefix_pages[:3], bsp.MAX_TAIL)
    st.o.fill_(7.0)
    g.replay()
    stt, flags = bsp.read_device_status(st.plan)
    assert flags & bsp.DEVFLAG_GRAPH and bsp.STATUS_NAMES[stt] == "BSP_ERR_STALE_PLAN"
    assert bool((st.o == 7.0).all())
    # flags that do not go with graph mode
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        plan = st.ws.plan(st.geo, wl.batch, wl.beam_width, case.prefix_len, case.tail_len, case.prefix_pages,
                          bsp.MAX_TAIL)
        bsp.decode_attn(plan, st.q, st.k_pool, st.v_pool, st.beam_pages, st.cache_indirection, st.scale, st.o,
                        st.lse, flags=bsp.FLAG_GRAPH | bsp.FLAG_CHECK)
