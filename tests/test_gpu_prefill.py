"""GPU parity of the prefill over the cached prefix: the CUDA path through the C ABI against the fp64
oracle, element by element (|O - O_ref| <= 2e-2 + 1e-2 |O_ref|, |LSE - LSE_ref| <= 1e-3)."""
import math

import numpy as np
import pytest
import torch

import oracle
from beam_search_shared_gb300 import bsp, synth
from beam_search_shared_gb300.step import PrefillStep

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3


def oracle_prefill(case):
    wl = case.workload
    kp, vp = synth.bits(case.k_pool).copy(), synth.bits(case.v_pool).copy()
    oracle.append_kv(Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages,
                     out_cache_loc=case.out_cache_loc, k_new_bits=synth.bits(case.k_new),
                     v_new_bits=synth.bits(case.v_new), k_pool_bits=kp, v_pool_bits=vp)
    O, L = oracle.prefill_attn(dtype=wl.dtype, B=wl.batch, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
                               ps=wl.page_size, num_pages=case.num_pages, cached_len=case.cached_len,
                               prompt_len=case.prompt_len, pages=case.pages, causal=wl.causal,
                               q_bits=synth.bits(case.q), k_pool_bits=kp, v_pool_bits=vp,
                               scale=1 / math.sqrt(wl.head_dim))
    return O, L, kp, vp


def run_and_check(case):
    step = PrefillStep(case)
    st, flags = step.run()
    assert st == 0 and flags == 0, (st, flags)
    O, L, kp, vp = oracle_prefill(case)
    o = step.o.float().double().cpu().numpy()
    lse = step.lse.double().cpu().numpy()
    assert np.isfinite(o).all()
    err = np.abs(o - O)
    bad = err > ATOL + RTOL * np.abs(O)
    assert not bad.any(), f"{bad.sum()} O elements out of tolerance, worst {err.max():.3g}"
    assert np.abs(lse - L).max() <= LSE_TOL
    np.testing.assert_array_equal(synth.bits(step.k_pool), kp)
    np.testing.assert_array_equal(synth.bits(step.v_pool), vp)
    return step


CASES = [
    ("prefill_tiny_d64", dict()),
    ("prefill_tiny_d64", dict(causal=False)),
    ("prefill_text_b8", dict(batch=3, cached=(0, 700), prompt=(1, 150))),
    ("prefill_text_b8", dict(batch=3, cached=(0, 700), prompt=(1, 150), causal=False)),
    ("prefill_text_b8", dict(batch=2, head_dim=64, dtype="bf16", prompt=(40, 90), cached=(0, 200))),
    ("prefill_text_b8", dict(batch=2, head_dim=256, prompt=(20, 70), cached=(0, 150))),
    ("prefill_text_b8", dict(batch=2, num_q_heads=8, num_kv_heads=8, page_size=8, prompt=(100, 180),
                             cached=(0, 90))),   # MHA: blocks of 128 tokens
    ("prefill_text_b8", dict(batch=2, num_q_heads=24, num_kv_heads=4, prompt=(5, 60), cached=(3, 60))),  # G 6
    ("prefill_text_b8", dict(batch=3, num_q_heads=24, num_kv_heads=8, prompt=(30, 200), cached=(0, 400))),  # G 3
    ("prefill_text_b8", dict(batch=2, num_q_heads=40, num_kv_heads=8, prompt=(50, 130), cached=(0, 100),
                             causal=False)),     # G 5: blocks of 24 tokens, 30 rows per TMEM lane quadrant
    ("prefill_text_b8", dict(batch=2, num_q_heads=8, num_kv_heads=8, head_dim=64, dtype="bf16", prompt=(250, 300),
                             cached=(0, 64))),   # MHA at head_dim 64: units of 256 tokens
]


@pytest.mark.parametrize("name,kw", CASES)
def test_prefill_parity(name, kw):
    wl = synth.PREFILL_WORKLOADS[name].with_(**kw)
    run_and_check(synth.make_prefill_case(wl, 11))


def test_prefill_empty_requests_and_empty_cache():
    wl = synth.PREFILL_WORKLOADS["prefill_text_b8"].with_(batch=4)
    case = synth.make_prefill_case(wl, 12, cached_lengths=[0, 50, 300, 0], prompt_lengths=[33, 0, 1, 64])
    run_and_check(case)


@pytest.mark.parametrize("Hq,D", [(32, 128), (24, 64), (8, 128)])
def test_prefill_two_block_unit_edges(Hq, D):
    """Units of two row blocks (head_dim <= 128): prompts ending at a block's end, one token past it, at
    the unit's end and one past it (the next unit's second block empty), cached rows ending inside a key
    tile; the causal mask of each row follows its own position."""
    wl = synth.PREFILL_WORKLOADS["prefill_text_b8"].with_(batch=6, num_q_heads=Hq, num_kv_heads=8, head_dim=D,
                                                          dtype="bf16" if D == 64 else "fp16")
    G = Hq // 8
    wblk = 4 * (32 // G)
    S = [wblk, wblk + 1, 2 * wblk, 2 * wblk + 1, 1, 3 * wblk + 5]
    case = synth.make_prefill_case(wl, 15, cached_lengths=[0, 10, 130, 64, 0, 500], prompt_lengths=S)
    step = run_and_check(case)
    assert step.plan.layout == 2 and step.plan.beams_per_block == wblk


@pytest.mark.parametrize("kw", [
    dict(),                                   # head_dim 128: the two-block kernel writes the partial states
    dict(causal=False),
    dict(head_dim=64, dtype="bf16"),
    dict(head_dim=256, num_q_heads=16),       # the one-set kernel
])
def test_prefill_key_splits_of_long_caches(kw):
    """Requests with long cached prefixes and short prompts: the planner cuts their cached keys into
    ranges (partial states merged by the tail kernel), the others stay whole."""
    wl = synth.PREFILL_WORKLOADS["prefill_text_b8"].with_(batch=4, **kw)
    case = synth.make_prefill_case(wl, 16, cached_lengths=[3000, 2500, 40, 1900], prompt_lengths=[20, 57, 300, 1])
    step = run_and_check(case)
    assert step.plan.tail_requests > 0
    assert step.plan.beam_width == 300            # partial-state rows: the longest prompt


def test_prefill_without_room_for_partials_is_planned_whole():
    """A workspace sized for one row per partial slot cannot hold the split requests' partial states: the
    plan keeps every request whole (no tail kernel) and stays correct."""
    wl = synth.PREFILL_WORKLOADS["prefill_text_b8"].with_(batch=4)
    case = synth.make_prefill_case(wl, 17, cached_lengths=[3000, 2500, 40, 1900], prompt_lengths=[20, 57, 300, 1])
    step = PrefillStep(case)
    step.ws = bsp.Workspace(step.geo, wl.batch, 1, case.pages.shape[1])
    st, flags = step.run()
    assert st == 0 and flags == 0
    assert step.plan.tail_requests == 0
    O, L, _, _ = oracle_prefill(case)
    o = step.o.float().double().cpu().numpy()
    assert (np.abs(o - O) <= ATOL + RTOL * np.abs(O)).all()
    assert np.abs(step.lse.double().cpu().numpy() - L).max() <= LSE_TOL


def test_prefill_image_prompt_from_empty_cache():
    """Image tokens prefilled with nothing cached (the case the page measures), 2 x 512 tokens."""
    wl = synth.PREFILL_WORKLOADS["prefill_image_b4_s1024"].with_(batch=2, prompt=(512, 512))
    run_and_check(synth.make_prefill_case(wl, 13))


def test_plan_kinds_are_not_mixed():
    wl = synth.PREFILL_WORKLOADS["prefill_tiny_d64"]
    step = PrefillStep(synth.make_prefill_case(wl, 14))
    step.make_plan()
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.decode_attn(step.plan, step.q, step.k_pool, step.v_pool, None, None, step.scale, step.o, step.lse)
