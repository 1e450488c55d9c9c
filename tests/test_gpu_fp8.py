"""GPU parity of the append into FP8 E4M3 pools (bsp_append_kv_fp8) against the oracle: bit-exact (the
quantised code is decided on both sides from the same fp32 product, rounded to nearest even with
saturation)."""
import numpy as np
import pytest
import torch

import oracle
from beam_search_shared_gb300 import bsp, synth

pytestmark = pytest.mark.gpu

TDT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def make_plan(Hq, Hkv, D, ps, num_pages, dtype, n):
    geo = bsp.geometry(Hq, Hkv, D, ps, num_pages, dtype)
    ws = bsp.Workspace(geo, 1, n, 1, device="cuda")
    plan = ws.plan(geo, 1, n, [ps], [1], np.zeros((1, 1), np.int32), max_tail=1)
    return plan, ws


def u8(t):
    return t.view(torch.uint8).cpu().numpy() if t.dtype != torch.uint8 else t.cpu().numpy()


@pytest.mark.parametrize("dtype,Hkv,D,n,k_mul,v_mul", [
    ("bf16", 8, 128, 61, 1.0, 1.0),
    ("fp16", 8, 128, 33, 0.05, 7.5),     # K saturates in places, V uses the subnormal range
    ("bf16", 2, 64, 17, 3.0, 0.25),
    ("fp16", 4, 256, 9, 1.0, 1.0),
])
def test_fp8_append_bit_exact(dtype, Hkv, D, n, k_mul, v_mul):
    ps, num_pages = 16, 48
    g = torch.Generator().manual_seed(n + D)
    plan, ws = make_plan(4 * Hkv, Hkv, D, ps, num_pages, dtype, n)
    # a wider projection output: rows of K, V and more, K and V as column slices
    row = Hkv * D
    fused = (torch.randn((n, 3 * row + 16), generator=g) * torch.tensor(200.0)).to(TDT[dtype])
    fused[:, row:2 * row] = (torch.randn((n, row), generator=g) * 0.01).to(TDT[dtype])
    fused = fused.cuda()
    k_new, v_new = fused[:, :row], fused[:, row:2 * row]
    loc = torch.randperm(num_pages * ps, generator=g)[:n].to(torch.int32)
    k_pool = torch.randint(0, 256, (num_pages, Hkv, ps, D), generator=g, dtype=torch.uint8).cuda()
    v_pool = torch.randint(0, 256, (num_pages, Hkv, ps, D), generator=g, dtype=torch.uint8).cuda()
    kp, vp = k_pool.cpu().numpy().copy(), v_pool.cpu().numpy().copy()
    bsp.append_kv_fp8(plan, k_new, v_new, loc.cuda(), k_pool, v_pool, k_mul=k_mul, v_mul=v_mul)
    assert bsp.read_device_status(plan) == (0, 0)
    kb = synth.bits(k_new.contiguous()).reshape(n, -1)
    vb = synth.bits(v_new.contiguous()).reshape(n, -1)
    oracle.append_kv_fp8(src_dtype=dtype, Hkv=Hkv, D=D, ps=ps, num_pages=num_pages, out_cache_loc=loc.numpy(),
                         k_new_bits=kb, v_new_bits=vb, k_pool_bits=kp, v_pool_bits=vp, k_mul=k_mul, v_mul=v_mul)
    np.testing.assert_array_equal(k_pool.cpu().numpy(), kp)
    np.testing.assert_array_equal(v_pool.cpu().numpy(), vp)
    if k_new.float().abs().max().item() * k_mul > 464:
        assert ((kp & 0x7F) == 0x7E).any()   # products past the range saturate at +-448


def test_fp8_source_copied_bad_slot_and_arguments():
    dtype, Hkv, D, ps, num_pages, n = "bf16", 4, 128, 16, 16, 11
    plan, ws = make_plan(16, Hkv, D, ps, num_pages, dtype, n)
    g = torch.Generator().manual_seed(5)
    k8 = torch.randint(0, 256, (n, Hkv * D), generator=g, dtype=torch.uint8)
    k8[k8 == 0x7F] = 0          # keep NaN patterns out of the view below
    v8 = torch.randint(0, 256, (n, Hkv * D), generator=g, dtype=torch.uint8)
    loc = torch.randperm(num_pages * ps, generator=g)[:n].to(torch.int32)
    k_pool = torch.zeros((num_pages, Hkv, ps, D), dtype=torch.uint8, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    bsp.append_kv_fp8(plan, k8.cuda().view(torch.float8_e4m3fn), v8.cuda(), loc.cuda(), k_pool, v_pool)
    assert bsp.read_device_status(plan) == (0, 0)
    kp, vp = np.zeros((num_pages, Hkv, ps, D), np.uint8), np.zeros((num_pages, Hkv, ps, D), np.uint8)
    oracle.append_kv_fp8(src_dtype="e4m3", Hkv=Hkv, D=D, ps=ps, num_pages=num_pages, out_cache_loc=loc.numpy(),
                         k_new_bits=k8.numpy(), v_new_bits=v8.numpy(), k_pool_bits=kp, v_pool_bits=vp)
    np.testing.assert_array_equal(k_pool.cpu().numpy(), kp)
    np.testing.assert_array_equal(v_pool.cpu().numpy(), vp)
    # a bad slot: that token is skipped and flagged, the others written
    k16 = torch.randn((n, Hkv * D), generator=g).to(torch.bfloat16).cuda()
    l2 = loc.clone()
    l2[4] = num_pages * ps
    k_pool.zero_()
    v_pool.zero_()
    bsp.append_kv_fp8(plan, k16, k16, l2.cuda(), k_pool, v_pool)
    st, flags = bsp.read_device_status(plan)
    assert flags == bsp.DEVFLAG_PAGE_INDEX and bsp.STATUS_NAMES[st] == "BSP_ERR_PAGE_INDEX"
    s0 = int(loc[0])
    assert k_pool[s0 // ps, :, s0 % ps].any()
    # host-checkable errors: nothing launched
    for kw in (dict(k_mul=0.0), dict(v_mul=float("inf")), dict(k_mul=-1.0)):
        with pytest.raises(bsp.BspError, match="INVALID_ARG"):
            bsp.append_kv_fp8(plan, k16, k16, loc.cuda(), k_pool, v_pool, **kw)
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):   # a host pool
        bsp.append_kv_fp8(plan, k16, k16, loc.cuda(), k_pool.cpu(), v_pool)
    before = k_pool.clone()
    bsp.append_kv_fp8(plan, k16[:0], k16[:0], loc[:0].cuda(), k_pool, v_pool)   # n == 0: no-op
    assert torch.equal(before, k_pool)


def test_fp8_append_decode_workload_full_size():
    """The new tokens of the benchmark's decode step, quantised into E4M3 pools, bit for bit."""
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"]
    case = synth.make_case(wl, 1000, full_step=True, device="cuda")
    n = case.out_cache_loc.size
    geo = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, case.num_pages, wl.dtype)
    ws = bsp.Workspace(geo, wl.batch, wl.beam_width, case.prefix_pages.shape[1], device="cuda")
    plan = ws.plan(geo, wl.batch, wl.beam_width, case.prefix_len, case.tail_len, case.prefix_pages)
    shape = (case.num_pages, wl.num_kv_heads, wl.page_size, wl.head_dim)
    k_pool = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    v_pool = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    bsp.append_kv_fp8(plan, case.k_new.reshape(n, -1), case.v_new.reshape(n, -1),
                      torch.from_numpy(case.out_cache_loc).cuda(), k_pool, v_pool, k_mul=2.0, v_mul=2.0)
    assert bsp.read_device_status(plan) == (0, 0)
    kp, vp = np.zeros(shape, np.uint8), np.zeros(shape, np.uint8)
    oracle.append_kv_fp8(src_dtype=wl.dtype, Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size,
                         num_pages=case.num_pages, out_cache_loc=case.out_cache_loc,
                         k_new_bits=synth.bits(case.k_new).reshape(n, -1), v_new_bits=synth.bits(case.v_new).reshape(n, -1),
                         k_pool_bits=kp, v_pool_bits=vp, k_mul=2.0, v_mul=2.0)
    np.testing.assert_array_equal(k_pool.cpu().numpy(), kp)
    np.testing.assert_array_equal(v_pool.cpu().numpy(), vp)
