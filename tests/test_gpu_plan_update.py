"""Per-step plan update (bsp_plan_update_tails): a plan dealt once for a batch's prompts, then new tail
lengths each step. The updated plan's request records and outputs equal those of a fresh plan of the same
step bit for bit (the work units depend on the prompts only), and both match the oracle; graph replays
follow the updates; the error paths leave the plan as it was."""
import math

import numpy as np
import pytest
import torch

import oracle
from beam_search_shared_gb300 import bsp, synth
from beam_search_shared_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3
REQ_BYTES = 12 * 4


def oracle_attn(case, P, T):
    wl = case.workload
    return oracle.decode_attn(
        dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
        ps=wl.page_size, num_pages=case.num_pages, prefix_len=P, tail_len=T, prefix_pages=case.prefix_pages,
        beam_pages=case.beam_pages, cache_indirection=case.cache_indirection, q_bits=synth.bits(case.q),
        k_pool_bits=synth.bits(case.k_pool), v_pool_bits=synth.bits(case.v_pool), scale=1 / math.sqrt(wl.head_dim))


def check_oracle(st, P, T):
    O, L = oracle_attn(st.case, P, T)
    o = st.o.double().cpu().numpy()
    lse = st.lse.double().cpu().numpy()
    assert np.isfinite(o).all()
    err = np.abs(o - O)
    assert (err <= ATOL + RTOL * np.abs(O)).all(), (T.tolist(), err.max())
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(L))
    both = np.isneginf(lse) & np.isneginf(L)
    assert (np.abs(lse[~both] - L[~both]) <= LSE_TOL).all()


def req_records(plan, ws):
    lo = plan.off_req
    return ws.device[lo:lo + plan.batch * REQ_BYTES].cpu().numpy().view(np.int32).reshape(plan.batch, 12)


def tail_trials(T_case, rng):
    """Tail lengths of successive steps: the beam-search pattern (+1 per step up to the case's tails), all
    zero, the case's own, and random ones within the case's tables."""
    out = [np.minimum(T_case, k).astype(np.int32) for k in range(0, 9, 2)]
    out += [np.zeros_like(T_case), T_case.copy(), rng.integers(0, T_case + 1).astype(np.int32)]
    return out


@pytest.mark.parametrize("name,batch", [("qwen3_0p6b_b64_w30", 16), ("wide_beam_b128_w96", 3),
                                        ("qwen3_4b_fp16_d128", 6), ("qwen3_4b_fp16_d64", 4),
                                        ("qwen3_4b_fp16_d256", 4), ("tiny_b1_w4_d64", 1)])
def test_update_matches_a_fresh_plan_bit_for_bit_and_the_oracle(name, batch):
    wl = synth.WORKLOADS[name].scaled(batch)
    rng = np.random.default_rng(batch)
    T_case = rng.integers(0, bsp.MAX_TAIL + 1, batch).astype(np.int32)
    T_case[0] = bsp.MAX_TAIL
    case = synth.make_case(wl, 300 + batch, full_step=False, device="cuda", tail_lengths=T_case)
    st = DeviceStep(case)
    fresh = bsp.Workspace(st.geo, batch, wl.beam_width, case.prefix_pages.shape[1])
    P = case.prefix_len.astype(np.int32)
    T0 = np.zeros(batch, np.int32)
    st.plan = st.ws.plan(st.geo, batch, wl.beam_width, P, T0, case.prefix_pages, bsp.MAX_TAIL)
    units0 = st.plan.num_units
    layouts = set()
    for T in tail_trials(T_case, rng):
        st.update_tails(T)
        up = (st.plan.tail_requests, st.plan.max_tail_len, st.plan.max_total_len, st.plan.num_units)
        st.o.fill_(float("nan"))
        st.attend()
        assert bsp.read_device_status(st.plan) == (0, 0)
        o_u, lse_u = st.o.clone(), st.lse.clone()
        rec_u = req_records(st.plan, st.ws)
        check_oracle(st, P, T)
        # the same step from a fresh plan on a second workspace
        pf = fresh.plan(st.geo, batch, wl.beam_width, P, T, case.prefix_pages, bsp.MAX_TAIL)
        layouts.add(pf.layout)
        assert up == (pf.tail_requests, pf.max_tail_len, pf.max_total_len, units0)
        assert pf.num_units == units0
        bsp.decode_attn(pf, st.q, st.k_pool, st.v_pool, st.beam_pages, st.cache_indirection, st.scale, st.o, st.lse)
        assert bsp.read_device_status(pf) == (0, 0)
        np.testing.assert_array_equal(rec_u, req_records(pf, fresh))
        assert torch.equal(o_u, st.o) and torch.equal(lse_u, st.lse)
    assert len(layouts) == 1


def test_graph_replays_follow_updates():
    wl = synth.WORKLOADS["qwen3_4b_fp16_d128"].scaled(5)
    T_case = np.array([8, 3, 0, 6, 8], np.int32)
    case = synth.make_case(wl, 41, full_step=False, device="cuda", tail_lengths=T_case)
    st = DeviceStep(case)
    P = case.prefix_len.astype(np.int32)
    st.plan = st.ws.plan(st.geo, wl.batch, wl.beam_width, P, np.zeros(5, np.int32), case.prefix_pages, bsp.MAX_TAIL)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bsp.decode_attn(st.plan, st.q, st.k_pool, st.v_pool, st.beam_pages, st.cache_indirection, st.scale, st.o,
                        st.lse, flags=bsp.FLAG_GRAPH)
    for T in tail_trials(T_case, np.random.default_rng(3)):
        st.update_tails(T)                        # outside the graph, on the replay's stream
        st.o.fill_(float("nan"))
        g.replay()
        assert bsp.read_device_status(st.plan) == (0, 0)
        check_oracle(st, P, T)


def test_update_errors_leave_the_plan_unchanged():
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(3)
    case = synth.make_case(wl, 8, full_step=False, device="cuda", tail_lengths=[2, 2, 2])
    st = DeviceStep(case, max_tail=4)
    st.make_plan()
    before = bytes(st.plan)
    with pytest.raises(bsp.BspError, match="CAPACITY"):
        st.update_tails([1, 5, 0])                # above the plan's max_tail
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        st.update_tails([1, -1, 0])
    with pytest.raises(ValueError):
        st.update_tails([1, 1])
    assert bytes(st.plan) == before
    st.update_tails([1, 2, 3])
    stale = bsp.Plan.from_buffer_copy(before)     # the plan before the update is now stale
    with pytest.raises(bsp.BspError, match="STALE_PLAN"):
        bsp.plan_update_tails(stale, [0, 0, 0])
    with pytest.raises(bsp.BspError, match="STALE_PLAN"):
        bsp.decode_attn(stale, st.q, st.k_pool, st.v_pool, st.beam_pages, st.cache_indirection, st.scale, st.o,
                        st.lse)
    torch.cuda.synchronize()
    # a prefill plan has no tails to update
    pwl = synth.PREFILL_WORKLOADS["prefill_tiny_d64"]
    pcase = synth.make_prefill_case(pwl, 3, device="cuda")
    from beam_search_shared_gb300.step import PrefillStep
    ps = PrefillStep(pcase)
    ps.make_plan()
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.plan_update_tails(ps.plan, np.zeros(ps.plan.batch, np.int32))
