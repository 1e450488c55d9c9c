"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element by element.

Bar: append and gathers bit-exact; attention |O - O_ref| <= 2e-2 + 1e-2 |O_ref| elementwise and
|LSE - LSE_ref| <= 1e-3 (natural log), for bf16/fp16 inputs with fp32 accumulation.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from beam_search_shared_gb300 import bsp, synth
from beam_search_shared_gb300.step import DeviceStep

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3


def oracle_after_append(case, rows=None):
    """Oracle pools after the step's append (full steps), then unsplit attention."""
    wl = case.workload
    kp, vp = synth.bits(case.k_pool).copy(), synth.bits(case.v_pool).copy()
    if case.full_step and case.out_cache_loc.size:
        oracle.append_kv(Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages,
                         out_cache_loc=case.out_cache_loc, k_new_bits=synth.bits(case.k_new),
                         v_new_bits=synth.bits(case.v_new), k_pool_bits=kp, v_pool_bits=vp)
    O, L = oracle.decode_attn(
        dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
        ps=wl.page_size, num_pages=case.num_pages, prefix_len=case.prefix_len, tail_len=case.tail_len,
        prefix_pages=case.prefix_pages, beam_pages=case.beam_pages, cache_indirection=case.cache_indirection,
        q_bits=synth.bits(case.q), k_pool_bits=kp, v_pool_bits=vp, scale=1 / math.sqrt(wl.head_dim), rows=rows)
    return O, L, kp, vp


def assert_attn_close(o_gpu, lse_gpu, O, L, what=""):
    o = o_gpu.float().double().cpu().numpy()
    lse = lse_gpu.double().cpu().numpy()
    assert np.isfinite(o).all(), f"{what}: non-finite O"
    err = np.abs(o - O)
    bound = ATOL + RTOL * np.abs(O)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} O elements out of tolerance, worst {err.max():.3g} "
                           f"at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    both_inf = np.isneginf(lse) & np.isneginf(L)
    dl = np.where(both_inf, 0.0, np.abs(lse - L))
    assert (dl <= LSE_TOL).all(), f"{what}: LSE worst {dl.max():.3g}"


def run_and_check(case, flags=0):
    step = DeviceStep(case)
    st, dev_flags = step.run(flags=flags)
    assert st == 0 and dev_flags == 0, (st, dev_flags)
    O, L, kp, vp = oracle_after_append(case)
    assert_attn_close(step.o, step.lse, O, L, case.workload.name)
    if case.full_step:
        np.testing.assert_array_equal(synth.bits(step.k_pool), kp)
        np.testing.assert_array_equal(synth.bits(step.v_pool), vp)
    return step


# ------------------------------------------------------------------ append
@pytest.mark.parametrize("name,batch", [("tiny_b1_w4_d64", 1), ("qwen3_0p6b_b64_w30", 64),
                                        ("qwen3_4b_fp16_d256", 4)])
def test_append_bit_exact(name, batch):
    case = synth.make_case(synth.WORKLOADS[name].scaled(batch), 100 + batch, full_step=True, device="cuda")
    step = DeviceStep(case)
    step.make_plan()
    step.append()
    assert bsp.read_device_status(step.plan) == (0, 0)
    kp, vp = synth.bits(case.k_pool).copy(), synth.bits(case.v_pool).copy()
    wl = case.workload
    oracle.append_kv(Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages,
                     out_cache_loc=case.out_cache_loc, k_new_bits=synth.bits(case.k_new),
                     v_new_bits=synth.bits(case.v_new), k_pool_bits=kp, v_pool_bits=vp)
    np.testing.assert_array_equal(synth.bits(step.k_pool), kp)
    np.testing.assert_array_equal(synth.bits(step.v_pool), vp)


def test_append_strided_source_empty_and_bad_slot():
    case = synth.make_case(synth.WORKLOADS["tiny_b1_w4_d64"], 5, full_step=True, device="cuda")
    step = DeviceStep(case)
    step.make_plan()
    wl = case.workload
    n, row = case.k_new.shape[0], wl.num_kv_heads * wl.head_dim
    fused = torch.randn((n, 3 * row + 8), device="cuda").to(step.q.dtype)   # a wider projection output
    fused[:, :row] = step.k_new
    fused[:, row:2 * row] = step.v_new
    bsp.append_kv(step.plan, fused[:, :row], fused[:, row:2 * row], step.out_cache_loc, step.k_pool, step.v_pool,
                  src_row_stride=fused.stride(0))
    assert bsp.read_device_status(step.plan) == (0, 0)
    kp, vp = synth.bits(case.k_pool).copy(), synth.bits(case.v_pool).copy()
    oracle.append_kv(Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages,
                     out_cache_loc=case.out_cache_loc, k_new_bits=synth.bits(case.k_new),
                     v_new_bits=synth.bits(case.v_new), k_pool_bits=kp, v_pool_bits=vp)
    np.testing.assert_array_equal(synth.bits(step.k_pool), kp)
    np.testing.assert_array_equal(synth.bits(step.v_pool), vp)
    # n == 0 is a no-op
    before = step.k_pool.clone()
    bsp.append_kv(step.plan, step.k_new[:0], step.v_new[:0], step.out_cache_loc[:0], step.k_pool, step.v_pool)
    assert torch.equal(before, step.k_pool)
    # an out-of-range slot is skipped and flagged; the valid ones are written
    loc = step.out_cache_loc.clone()
    loc[1] = case.num_pages * wl.page_size
    fresh_k = torch.randn_like(step.k_new.float()).to(step.q.dtype)
    bsp.append_kv(step.plan, fresh_k, step.v_new, loc, step.k_pool, step.v_pool)
    st, flags = bsp.read_device_status(step.plan)
    assert flags == bsp.DEVFLAG_PAGE_INDEX and bsp.STATUS_NAMES[st] == "BSP_ERR_PAGE_INDEX"
    p0, o0 = divmod(int(loc[0]), wl.page_size)
    assert torch.equal(step.k_pool[p0, :, o0].reshape(-1), fresh_k[0])
    # host pointers are rejected before anything is launched
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.append_kv(step.plan, step.k_new.cpu(), step.v_new, step.out_cache_loc, step.k_pool, step.v_pool)


# ------------------------------------------------------------------ attention parity, small cases
SMALL = [
    ("tiny_b1_w4_d64", 1, dict()),
    ("qwen3_0p6b_b64_w30", 3, dict()),
    ("wide_beam_b128_w96", 2, dict()),              # 192 query rows per kv head -> two row blocks
    ("qwen3_4b_fp16_d128", 3, dict()),
    ("qwen3_4b_fp16_d64", 3, dict()),
    ("qwen3_4b_fp16_d256", 3, dict()),
    ("qwen3_0p6b_b64_w30", 2, dict(num_q_heads=6, num_kv_heads=2)),     # group 3
    ("qwen3_0p6b_b64_w30", 2, dict(num_q_heads=12, num_kv_heads=2, dtype="fp16")),  # group 6
    ("qwen3_0p6b_b64_w30", 2, dict(num_q_heads=8, num_kv_heads=8, page_size=8)),   # MHA, small pages
    ("qwen3_0p6b_b64_w30", 2, dict(num_q_heads=16, num_kv_heads=2, page_size=64)),  # group 8
    ("qwen3_0p6b_b64_w30", 2, dict(page_size=128, beam_width=7)),
]


@pytest.mark.parametrize("name,batch,kw", SMALL)
@pytest.mark.parametrize("full_step", [False, True])
def test_decode_parity_small(name, batch, kw, full_step):
    wl = synth.WORKLOADS[name].scaled(batch).with_(**kw)
    case = synth.make_case(wl, 7 + batch, full_step=full_step, device="cuda")
    run_and_check(case)


@pytest.mark.parametrize("P", [0, 5, 40, 2047, 10000])
@pytest.mark.parametrize("T", [0, 1])
def test_bucketed_prefix_parity(P, T):
    """Single-allocation decode: garbage beyond the valid prefix must stay hidden."""
    if P == 0 and T == 0:
        pytest.skip("empty sequence covered by test_empty_sequences")
    wl = synth.WORKLOADS[f"bucketed_prefix_p{P}"]
    case = synth.make_case(wl, 40 + P, full_step=T > 0, device="cuda", tail_lengths=[T])
    run_and_check(case)


def test_tail_lengths_mixed_and_boundary_crossing():
    wl = synth.WORKLOADS["qwen3_4b_fp16_d128"].scaled(6)
    case = synth.make_case(wl, 77, full_step=True, device="cuda",
                           prompt_lengths=[16, 29, 1, 0, 64, 131], tail_lengths=[8, 8, 3, 5, 0, 1])
    run_and_check(case)


@pytest.mark.parametrize("name", ["qwen3_0p6b_b64_w30", "qwen3_4b_fp16_d64", "qwen3_4b_fp16_d128",
                                  "qwen3_4b_fp16_d256"])
def test_prompt_kernel_finishes_short_requests(name):
    """Requests with one prompt partial state and few tail keys per row block are finished by the
    prompt kernel (tail keys gathered as up to four extra key tiles: 5 x 30 tail keys take two 128-key
    tiles, or three 64-key tiles at head_dim 256); the other, in the same batch, by the tail kernel: the
    3000-key prompt split over partial states."""
    wl = synth.WORKLOADS[name].scaled(6)
    case = synth.make_case(wl, 84, full_step=True, device="cuda", prompt_lengths=[100, 128, 60, 3000, 31, 7],
                           tail_lengths=[2, 0, 5, 2, 2, 1])
    step = run_and_check(case)
    assert step.plan.tail_requests == 1


def test_empty_sequences():
    """P = 0 and T = 0 rows give O = 0 and LSE = -inf; other rows are unaffected."""
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(3).with_(beam_width=4)
    case = synth.make_case(wl, 78, full_step=False, device="cuda", prompt_lengths=[0, 70, 0],
                           tail_lengths=[0, 0, 2])
    step = run_and_check(case)
    assert torch.all(step.o[:4] == 0)
    assert torch.all(torch.isneginf(step.lse[:4]))


def test_poisoned_garbage_rows_stay_hidden():
    wl = synth.WORKLOADS["qwen3_4b_fp16_d128"].scaled(3)
    case = synth.make_case(wl, 79, full_step=True, device="cuda", poison=True)
    assert torch.isnan(case.k_pool.float()).any()
    run_and_check(case)
    wl5 = synth.WORKLOADS["bucketed_prefix_p2047"]
    run_and_check(synth.make_case(wl5, 80, full_step=True, device="cuda", poison=True))


def test_lse_base2_flag():
    case = synth.make_case(synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(2), 81, full_step=False, device="cuda")
    step = DeviceStep(case)
    step.make_plan()
    step.attend(flags=bsp.FLAG_LSE_BASE2 | bsp.FLAG_CHECK)
    O, L, _, _ = oracle_after_append(case)
    assert_attn_close(step.o, step.lse / math.log2(math.e), O, L)


# ------------------------------------------------------------------ plan life cycle and device-side indices
def test_stale_plan_and_replanning_without_sync():
    case = synth.make_case(synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(2), 82, full_step=False, device="cuda")
    step = DeviceStep(case)
    first = step.make_plan()
    for _ in range(6):           # more generations than staging slots: exercises the echo wait
        step.make_plan()
        step.attend()
    with pytest.raises(bsp.BspError, match="STALE_PLAN"):
        bsp.decode_attn(first, step.q, step.k_pool, step.v_pool, step.beam_pages, step.cache_indirection,
                        step.scale, step.o, step.lse)
    assert bsp.read_device_status(step.plan) == (0, 0)
    O, L, _, _ = oracle_after_append(case)
    assert_attn_close(step.o, step.lse, O, L)


def test_bad_device_indices_are_flagged_not_faulted():
    case = synth.make_case(synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(2).with_(beam_width=4), 83,
                           full_step=False, device="cuda", tail_lengths=[2, 2])
    step = DeviceStep(case)
    step.make_plan()
    P0 = int(case.prefix_len[0])
    step.cache_indirection[0, 1, P0] = 99           # indirection beyond the beam width
    step.attend()
    st, flags = bsp.read_device_status(step.plan)
    assert flags & bsp.DEVFLAG_PAGE_INDEX
    step.cache_indirection.copy_(torch.from_numpy(case.cache_indirection))
    src = int(case.cache_indirection[1, 2, int(case.prefix_len[1]) + 1])
    step.beam_pages[1 * 4 + src, (int(case.prefix_len[1]) + 1) // case.workload.page_size] = case.num_pages + 5
    step.attend()
    st, flags = bsp.read_device_status(step.plan)
    assert flags & bsp.DEVFLAG_PAGE_INDEX
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.decode_attn(step.plan, step.q.cpu(), step.k_pool, step.v_pool, step.beam_pages,
                        step.cache_indirection, step.scale, step.o, step.lse)


# ------------------------------------------------------------------ full sizes, sampled rows
FULL = ["qwen3_0p6b_b64_w30", "wide_beam_b128_w96", "qwen3_4b_fp16_d128", "qwen3_4b_fp16_d64",
        "qwen3_4b_fp16_d256"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_parity(name):
    wl = synth.WORKLOADS[name]
    case = synth.make_case(wl, 1000 + FULL.index(name), full_step=True, device="cuda")
    step = DeviceStep(case)
    st, flags = step.run()
    assert (st, flags) == (0, 0)
    R = wl.batch * wl.beam_width
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([rng.integers(0, R, 48), [0, R - 1, wl.beam_width - 1]])).astype(np.int32)
    O, L, kp, vp = oracle_after_append(case, rows=rows)
    assert_attn_close(step.o[rows], step.lse[rows], O, L, name)
    # the append is checked bit-exact on every slot it wrote
    loc = case.out_cache_loc
    pg, off = loc // wl.page_size, loc % wl.page_size
    np.testing.assert_array_equal(synth.bits(step.k_pool[pg, :, off]), kp[pg, :, off])
    np.testing.assert_array_equal(synth.bits(step.v_pool[pg, :, off]), vp[pg, :, off])


def test_one_request_with_more_key_splits_than_the_unrolled_merge():
    """Nine requests without a prompt and one of 73 595 keys on one kv head: the planner gives the long
    one 72 key splits (its bound is batch + 64 in all), more than the tail kernel's unrolled partial-LSE
    loads cover; the merge must still take every split into its maximum."""
    wl = synth.Workload("one_long_request_b10", 10, 1, 8, 1, 128, 32, "bf16", (0, 0), (1, 1))
    P = [0] * 10
    P[3] = 1150 * 64 - 5
    case = synth.make_case(wl, 99, full_step=True, device="cuda", prompt_lengths=P, tail_lengths=[1] * 10)
    step = DeviceStep(case)
    step.make_plan()
    plan, img = bsp.plan_build(step.geo, wl.batch, wl.beam_width, case.prefix_len, case.tail_len,
                               case.prefix_pages, bsp.MAX_TAIL, step.plan.num_sms)
    assert bsp.plan_requests(plan, img)[3, 2] > 65
    run_and_check(case)
