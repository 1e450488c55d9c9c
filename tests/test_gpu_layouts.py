"""GPU parity of the decode prompt kernels chosen by shape, against the fp64 oracle element by element.

Layout 2 (two MMA blocks per CTA): a (request, kv head) with 129-256 query rows keeps all of them in one
CTA, so its prompt is read once. Layout 1 (alternating-tile kernel): two softmax warp sets take a unit's
key tiles alternately, each with its own score buffer and output accumulator, and merge at the unit's
end; the row blocks of a (request, kv head) with more than 128 rows run on neighbouring CTAs.

Covers, for both: the fused path (no key splits: the unit gathers up to four tiles of its beams' tail
keys and writes the final O and LSE), the split path (partial states merged by the tail kernel), tails
too long for the fused path, units of one tile (set B without a tile) and units whose second tile is a
tail tile, head_dim 64 and 128, odd beam counts, group sizes 1-8, page sizes 8-64, bf16 and fp16."""
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
FOURB = synth.WORKLOADS["qwen3_4b_fp16_d128"]


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
    sel = slice(None) if rows is None else torch.from_numpy(rows).long().to(step.o.device)
    o = step.o[sel].double().cpu().numpy()
    lse = step.lse[sel].double().cpu().numpy()
    assert np.isfinite(o).all()
    err = np.abs(o - O)
    bad = err > ATOL + RTOL * np.abs(O)
    assert not bad.any(), (int(bad.sum()), float(err.max()), np.argwhere(bad)[:5].tolist())
    both = np.isneginf(lse) & np.isneginf(L)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(L))
    assert (np.abs(lse[~both] - L[~both]) <= LSE_TOL).all(), float(np.abs(lse[~both] - L[~both]).max())


def run(wl, seed, layout, full_step=True, **kw):
    case = synth.make_case(wl, seed, full_step=full_step, device="cuda", **kw)
    step = DeviceStep(case)
    st, flags = step.run()
    assert (st, flags) == (0, 0)
    assert step.plan.layout == layout
    return step


def sample_rows(wl, seed, n=300):
    R = wl.batch * wl.beam_width
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.integers(0, R, n), [0, R - 1]])).astype(np.int32)


# ------------------------------------------------------------------ layout 2: two MMA blocks per CTA
def test_wide_fused_tail_tiles():
    """40 requests x 8 kv heads fill the GPU without key splits: every request (tails of 0-5 tokens: up
    to 4 tiles of 96 beams' tail keys) is finished by the prompt kernel, no tail launch."""
    wl = WIDE.scaled(40).with_(prompt=(100, 400), tail=(0, 5))
    step = run(wl, 11, 2)
    assert step.plan.tail_requests == 0 and step.plan.num_parts == 40
    check(step)


def test_wide_long_tails_go_to_the_tail_kernel():
    """Tails of 6-8 tokens need 5-6 tiles of 96 beams' keys: those requests' prompt partials are merged
    with their tails by the tail kernel, in the same batch as fused ones."""
    wl = WIDE.scaled(40).with_(prompt=(60, 300), tail=(0, 8))
    T = np.array([8, 6, 7, 0, 5, 1] + [3] * 34, np.int32)
    step = run(wl, 12, 2, tail_lengths=T)
    assert step.plan.tail_requests == 3
    check(step)


def test_wide_split_prompts_and_empty_requests():
    """Few requests: prompts are split over key ranges (partial states, tail kernel), one request has no
    prompt, one a prompt shorter than a page."""
    step = run(WIDE.scaled(3), 13, 2, prompt_lengths=[3000, 0, 17], tail_lengths=[2, 3, 1])
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
    step = run(wl, 14 + batch, 2)
    check(step, sample_rows(wl, batch))


def test_wide_full_size_all_rows_of_some_requests():
    """The full wide-beam workload (128 requests, 96 beams, ~3000-key prompts): every row of three
    requests (the first, one in the middle, the last) against the oracle."""
    case = synth.make_case(WIDE, 1001, full_step=True, device="cuda")
    step = DeviceStep(case)
    assert step.run() == (0, 0)
    assert step.plan.layout == 2 and step.plan.tail_requests == 0
    W = WIDE.beam_width
    check(step, np.concatenate([np.arange(b * W, (b + 1) * W) for b in (0, 63, 127)]).astype(np.int32))


# ------------------------------------------------------------------ layout 1: alternating-tile kernel
@pytest.mark.parametrize("head_dim", [128, 64])
def test_alt_fused_tails_up_to_eight_tokens(head_dim):
    """The 4B-shaped layer (30 beams x 4 heads = 120 rows, fp16, page 16): 40 requests fill the GPU
    without key splits and tails of up to 8 tokens (2 tiles of 240 keys) finish in the prompt kernel,
    including requests with no tail and tails crossing a page."""
    wl = FOURB.scaled(40).with_(head_dim=head_dim, prompt=(200, 700))
    step = run(wl, 21 + head_dim, 1)
    assert step.plan.tail_requests == 0
    check(step)


def test_alt_short_units_and_tail_tile_second():
    """Units of a single tile (prompts of at most 128 keys, no tail: set B takes no tile) next to units
    whose second tile is already a tail tile (set B's first tile holds only other beams' keys for most of
    its rows), with longer ones between."""
    wl = FOURB.scaled(40).with_(prompt=(1, 128))
    rng = np.random.default_rng(5)
    P = rng.integers(1, 129, 40).astype(np.int32)
    P[::5] = rng.integers(300, 900, 8)
    T = rng.integers(0, 9, 40).astype(np.int32)
    T[1::4] = 0
    step = run(wl, 22, 1, prompt_lengths=P, tail_lengths=T)
    check(step)


def test_alt_row_block_groups_and_long_tails():
    """96 beams x 4 heads = 384 rows: three row blocks per (request, kv head) on neighbouring CTAs;
    and 128 beams of one head each with tails of 5-8 tokens (5-8 tiles of a block's tail keys), which
    the tail kernel finishes."""
    wl = WIDE.scaled(16).with_(num_q_heads=32, num_kv_heads=8, prompt=(100, 900), tail=(0, 3))
    step = run(wl, 23, 1)
    assert step.plan.row_blocks == 3
    check(step, sample_rows(wl, 23, 600))
    wl = WIDE.scaled(40).with_(beam_width=128, num_q_heads=8, num_kv_heads=8, prompt=(60, 300), tail=(0, 8))
    T = np.array([8, 6, 5, 0, 4, 1] + [3] * 34, np.int32)
    step = run(wl, 24, 1, tail_lengths=T)
    assert step.plan.tail_requests == 3
    check(step, sample_rows(wl, 24, 600))


@pytest.mark.parametrize("kw,batch", [
    (dict(beam_width=16, num_q_heads=64, num_kv_heads=8), 40),                # G = 8, 4 beams per quadrant
    (dict(beam_width=30, num_q_heads=24, num_kv_heads=8, page_size=64), 40),  # G = 3, 90 rows
    (dict(beam_width=30, page_size=8, dtype="bf16"), 3),                      # split prompts
])
def test_alt_shapes(kw, batch):
    wl = FOURB.scaled(batch).with_(prompt=(40, 1500), **kw)
    step = run(wl, 25 + batch, 1)
    check(step, sample_rows(wl, batch))


# ------------------------------------------------------------------ layout 0: one softmax set
@pytest.mark.parametrize("kw,batch", [
    (dict(head_dim=64, page_size=16), 96),   # half-row layout at head_dim 64: K ring 6 deep, V ring 7
    (dict(head_dim=64, page_size=8), 64),
    (dict(), 96),                            # head_dim 128, half-row
])
def test_one_set_kernel_many_short_units_with_tail_tiles(kw, batch):
    """Prompts of one key tile and fused tails in every unit: the producer runs several tail tiles ahead
    of the epilogue warps that gather them (deep rings, short units), and the hand-over must follow."""
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(batch).with_(**kw)
    rng = np.random.default_rng(batch)
    P = rng.integers(1, 129, batch).astype(np.int32)
    T = rng.integers(1, 5, batch).astype(np.int32)
    step = run(wl, 31 + batch, 0, prompt_lengths=P, tail_lengths=T)
    assert step.plan.tail_requests == 0 and step.plan.num_units == batch * wl.num_kv_heads
    check(step)


@pytest.mark.parametrize("name,kw,batch", [
    ("qwen3_4b_fp16_d256", dict(), 8),                          # 64-key tiles: 30 x 8 tail keys in 4 tiles
    ("qwen3_0p6b_b64_w30", dict(), 16),                         # half-row: 30 x 8 in 2 tiles of 128
    ("qwen3_0p6b_b64_w30", dict(head_dim=64, page_size=16), 16),
    ("qwen3_4b_fp16_d256", dict(beam_width=21), 6),             # a partial last tail tile, odd beams
])
def test_one_set_kernel_several_tail_tiles(name, kw, batch):
    """Fused units ending with up to four tail tiles (tails of up to 8 tokens), short and long prompts in
    one batch; the request whose prompt is split over partial states goes to the tail kernel."""
    wl = synth.WORKLOADS[name].scaled(batch).with_(**kw)
    rng = np.random.default_rng(batch + len(kw))
    P = rng.integers(1, 700, batch).astype(np.int32)
    T = rng.integers(0, bsp.MAX_TAIL + 1, batch).astype(np.int32)
    T[0], T[1] = bsp.MAX_TAIL, 5
    step = run(wl, 61 + batch, 0, prompt_lengths=P, tail_lengths=T)
    wblk = step.plan.beams_per_block
    tile = 64 if wl.head_dim == 256 else 128
    assert max(-(-int(t) * wblk // tile) for t in T) >= 2     # some unit has several tail tiles
    check(step)
