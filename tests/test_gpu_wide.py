"""GPU parity of the wide layout: all W*G query rows (129-256) of a (request, kv head) in one unit as two
128-row tensor-core blocks sharing every K/V tile, against the fp64 oracle element by element.

Covers the fused path (no key splits: the unit gathers up to four tiles of the beams' tail keys and
writes the final O and LSE), the split path (partial states merged by the tail kernel), tails too long
for the fused path, head_dim 64, odd beam counts, group sizes 2-4, page sizes 16-64 and fp16."""
import math

import numpy as np
import pytest
import torch

import oracle
from beam_search_shared_gb300 import bsp, synth
from beam_search_shared_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3
WIDE = synth.WORKLOADS["wide_beam_b128_w96"]


def oracle_after_append(case, rows=None):
    wl = case.workload
    kp, vp = synth.bits(case.k_pool).copy(), synth.bits(case.v_pool).copy()
    if case.full_step and case.out_cache_loc.size:
        oracle.append_kv(Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages,
                         out_cache_loc=case.out_cache_loc, k_new_bits=synth.bits(case.k_new),
                         v_new_bits=synth.bits(case.v_new), k_pool_bits=kp, v_pool_bits=vp)
    return oracle.decode_attn(
        dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
        ps=wl.page_size, num_pages=case.num_pages, prefix_len=case.prefix_len, tail_len=case.tail_len,
        prefix_pages=case.prefix_pages, beam_pages=case.beam_pages, cache_indirection=case.cache_indirection,
        q_bits=synth.bits(case.q), k_pool_bits=kp, v_pool_bits=vp, scale=1 / math.sqrt(wl.head_dim), rows=rows)


def check(step, rows=None):
    O, L = oracle_after_append(step.case, rows)
    o = (step.o if rows is None else step.o[torch.from_numpy(rows).long().to(step.o.device)]).double().cpu().numpy()
    lse = (step.lse if rows is None else step.lse[torch.from_numpy(rows).long().to(step.o.device)]).double().cpu().numpy()
    assert np.isfinite(o).all()
    err = np.abs(o - O)
    bad = err > ATOL + RTOL * np.abs(O)
    assert not bad.any(), (int(bad.sum()), float(err.max()), np.argwhere(bad)[:5].tolist())
    both = np.isneginf(lse) & np.isneginf(L)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(L))
    assert (np.abs(lse[~both] - L[~both]) <= LSE_TOL).all(), float(np.abs(lse[~both] - L[~both]).max())


def run(wl, seed, full_step=True, **kw):
    case = synth.make_case(wl, seed, full_step=full_step, device="cuda", **kw)
    step = DeviceStep(case)
    st, flags = step.run()
    assert (st, flags) == (0, 0)
    assert step.plan.mma_blocks == 2, "expected the wide layout"
    return step


def test_wide_fused_tail_tiles():
    """40 requests x 8 kv heads fill the GPU without key splits: every request (tails of 0-5 tokens:
    up to 4 tiles of 96 beams' tail keys) is finished by the prompt kernel, no tail launch."""
    wl = WIDE.scaled(40).with_(prompt=(100, 400), tail=(0, 5))
    step = run(wl, 11)
    assert step.plan.tail_requests == 0 and step.plan.num_parts == 40
    check(step)
    np.testing.assert_array_equal(synth.bits(step.k_pool), oracle_pools(step.case)[0])


def oracle_pools(case):
    wl = case.workload
    kp, vp = synth.bits(case.k_pool).copy(), synth.bits(case.v_pool).copy()
    oracle.append_kv(Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages,
                     out_cache_loc=case.out_cache_loc, k_new_bits=synth.bits(case.k_new),
                     v_new_bits=synth.bits(case.v_new), k_pool_bits=kp, v_pool_bits=vp)
    return kp, vp


def test_wide_long_tails_go_to_the_tail_kernel():
    """Tails of 6-8 tokens need 5-6 tiles of 96 beams' keys: those requests' prompt partials are merged
    with their tails by the tail kernel, in the same batch as fused ones."""
    wl = WIDE.scaled(40).with_(prompt=(60, 300), tail=(0, 8))
    T = np.array([8, 6, 7, 0, 5, 1] + [3] * 34, np.int32)
    step = run(wl, 12, tail_lengths=T)
    assert step.plan.tail_requests == 3
    check(step)


def test_wide_split_prompts_and_empty_requests():
    """Few requests: prompts are split over key ranges (partial states, tail kernel), one request has
    no prompt, one a prompt shorter than a page."""
    wl = WIDE.scaled(3)
    step = run(wl, 13, prompt_lengths=[3000, 0, 17], tail_lengths=[2, 3, 1])
    assert step.plan.num_parts > 2
    check(step)


@pytest.mark.parametrize("kw,batch", [
    (dict(beam_width=70, page_size=16), 40),                                  # odd beams: 35 + 35, 9 per quadrant
    (dict(beam_width=64, num_q_heads=32, num_kv_heads=8, dtype="fp16"), 40),  # G = 4: 256 rows, full quadrants
    (dict(beam_width=50, num_q_heads=6, num_kv_heads=2, page_size=64), 160),  # G = 3, 150 rows
    (dict(beam_width=96, head_dim=64), 40),                                   # head_dim 64
    (dict(beam_width=65, head_dim=64, dtype="fp16", page_size=8), 3),         # 130 rows, split prompts
])
def test_wide_shapes(kw, batch):
    wl = WIDE.scaled(batch).with_(prompt=(40, 500), tail=(0, 4), **kw)
    step = run(wl, 14 + batch)
    R = wl.batch * wl.beam_width
    rng = np.random.default_rng(batch)
    rows = np.unique(np.concatenate([rng.integers(0, R, 300), [0, R - 1]])).astype(np.int32)
    check(step, rows)


def test_wide_full_size_all_rows_of_some_requests():
    """The full wide-beam workload (128 requests, 96 beams, ~3000-key prompts): every row of three
    requests (the first, one in the middle, the last) against the oracle."""
    case = synth.make_case(WIDE, 1001, full_step=True, device="cuda")
    step = DeviceStep(case)
    assert step.run() == (0, 0)
    assert step.plan.mma_blocks == 2 and step.plan.tail_requests == 0
    W = WIDE.beam_width
    rows = np.concatenate([np.arange(b * W, (b + 1) * W) for b in (0, 63, 127)]).astype(np.int32)
    check(step, rows)
