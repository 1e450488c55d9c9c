"""GPU parity of RoPE on the paged append (bsp_rope_cos_sin, bsp_rope_append_kv) against the fp64 oracle.

Bar: V rows, unrotated dims and untouched pool rows bit-exact. A rotated element is the kernel's fp32
result (fp32 table, one product and one fused multiply-add) rounded to nearest even, so it must be the
rounding of a value within delta = 2^-21 (|x| + |y|) of the exact fp64 rotation of its pair (x, y):
between round(v - delta) and round(v + delta). The table's fp32 entries must be within half an fp32
unit (2^-25 for |value| <= 1) of the exact cos / sin.
"""
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


def pair_bounds(x, rot, interleaved):
    """|x| + |y| of the pair of every element of rows x [.., D] (0 past rot)."""
    a = np.abs(x)
    partner = a.copy()
    if interleaved:
        partner[..., 0:rot:2], partner[..., 1:rot:2] = a[..., 1:rot:2], a[..., 0:rot:2]
    else:
        h = rot // 2
        partner[..., :h], partner[..., h:rot] = a[..., h:rot], a[..., :h]
    s = a + partner
    s[..., rot:] = 0
    return s


def assert_rotated(got_bits, x_bits, pos, dtype, rot, interleaved, base, what):
    """got_bits / x_bits uint16 [rows, D]; pos [rows]."""
    x = decode(x_bits, dtype)
    v = oracle.rope_rotate_rows(x, pos, rot=rot, interleaved=interleaved, base=base)
    delta = 2.0 ** -21 * pair_bounds(x, rot, interleaved)
    lo = decode(oracle.round_half_array(v - delta, dtype), dtype)
    hi = decode(oracle.round_half_array(v + delta, dtype), dtype)
    g = decode(got_bits, dtype)
    bad = ~((g >= lo) & (g <= hi))
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside the rounding bound, first at {np.argwhere(bad)[:3]}"
    np.testing.assert_array_equal(got_bits[:, rot:], x_bits[:, rot:])
    return float((got_bits == oracle.round_half_array(v, dtype)).mean())


def decode(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(TDT[dtype])
    return t.double().numpy()


def test_cos_sin_table_against_oracle():
    for max_pos, rot, base in ((4096, 128, 1e6), (300, 64, 10000.0), (17, 96, 5e5)):
        r = bsp.Rope(max_pos, rot, base)
        torch.cuda.synchronize()
        got = r.cos_sin.double().cpu().numpy()
        want = oracle.rope_cos_sin(max_pos, rot, base)
        err = np.abs(got - want)
        assert err.max() <= 2.0 ** -25 + 1e-13, err.max()


CASES = [
    # dtype, Hq, Hkv, D, rot, interleaved, with q, n
    ("bf16", 16, 8, 128, 128, False, True, 61),
    ("fp16", 32, 8, 128, 128, False, True, 33),
    ("bf16", 4, 2, 64, 32, False, True, 45),      # partial rotation, partner lookup over 2 chunks
    ("fp16", 8, 2, 64, 64, True, False, 19),
    ("bf16", 8, 4, 256, 128, True, True, 23),     # a head row on the whole warp, half rotated
    ("fp16", 8, 1, 256, 96, False, True, 7),      # rot/2 = 48: partner 6 chunks away
    ("bf16", 16, 8, 128, 16, False, False, 5),
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,rot,inter,with_q,n", CASES)
def test_rope_append_parity(dtype, Hq, Hkv, D, rot, inter, with_q, n):
    ps, num_pages, max_pos, base = 16, 64, 20000, 1e6 if D >= 128 else 10000.0
    g = torch.Generator().manual_seed(n * 31 + D + rot)
    plan, ws = make_plan(Hq, Hkv, D, ps, num_pages, dtype, n)
    rope = bsp.Rope(max_pos, rot, base, interleaved=inter)
    tdt = TDT[dtype]
    k_new = (torch.randn((n, Hkv * D), generator=g) * 4).to(tdt).cuda()
    v_new = torch.randn((n, Hkv * D), generator=g).to(tdt).cuda()
    q = (torch.randn((n, Hq * D), generator=g) * 2).to(tdt).cuda() if with_q else None
    loc = torch.randperm(num_pages * ps, generator=g)[:n].to(torch.int32)
    pos = torch.randint(0, max_pos, (n,), generator=g).to(torch.int32)
    pos[0] = 0
    pos[-1] = max_pos - 1
    k_pool = torch.randn((num_pages, Hkv, ps, D), generator=g).to(tdt).cuda()
    v_pool = torch.randn((num_pages, Hkv, ps, D), generator=g).to(tdt).cuda()
    kp0, vp0 = synth.bits(k_pool).copy(), synth.bits(v_pool).copy()
    q0 = None if q is None else synth.bits(q).copy()
    bsp.rope_append_kv(plan, rope, pos.cuda(), q, k_new, v_new, loc.cuda(), k_pool, v_pool)
    assert bsp.read_device_status(plan) == (0, 0)
    kp, vp = synth.bits(k_pool), synth.bits(v_pool)
    locn, posn = loc.numpy(), pos.numpy()
    page, off = locn // ps, locn % ps
    kb, vb = synth.bits(k_new).reshape(n, Hkv, D), synth.bits(v_new).reshape(n, Hkv, D)
    # V rows copied, other slots untouched
    np.testing.assert_array_equal(vp[page, :, off], vb)
    touched = np.zeros((num_pages, ps), bool)
    touched[page, off] = True
    np.testing.assert_array_equal(kp.transpose(0, 2, 1, 3)[~touched], kp0.transpose(0, 2, 1, 3)[~touched])
    np.testing.assert_array_equal(vp.transpose(0, 2, 1, 3)[~touched], vp0.transpose(0, 2, 1, 3)[~touched])
    # K rows rotated
    exact = assert_rotated(kp[page, :, off].reshape(n * Hkv, D), kb.reshape(n * Hkv, D), np.repeat(posn, Hkv),
                           dtype, rot, inter, base, "K")
    assert exact > 0.99
    np.testing.assert_array_equal(kp[page[0], :, off[0]], kb[0])   # position 0: a copy
    if with_q:
        qb = synth.bits(q).reshape(n * Hq, D)
        assert_rotated(qb, q0.reshape(n * Hq, D), np.repeat(posn, Hq), dtype, rot, inter, base, "q")
    # the oracle's own rounded append agrees except where its fp64 value is within delta of a tie
    q_o = None if q0 is None else q0.copy()
    kp_o, vp_o = kp0.copy(), vp0.copy()
    oracle.rope_append_kv(dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, rot=rot, interleaved=inter, base=base, max_pos=max_pos,
                          ps=ps, num_pages=num_pages, positions=posn, out_cache_loc=locn, q_bits=q_o,
                          k_new_bits=kb.reshape(n, -1), v_new_bits=vb.reshape(n, -1), k_pool_bits=kp_o,
                          v_pool_bits=vp_o)
    np.testing.assert_array_equal(vp, vp_o)
    assert (kp == kp_o).mean() > 0.999


def test_rope_append_decode_workload_full_size():
    """The decode step of the benchmark workload: every beam's new token at P_b + T_b - 1, q rotated."""
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"]
    case = synth.make_case(wl, 1000, full_step=True, device="cuda")
    n = case.out_cache_loc.size
    geo = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, case.num_pages, wl.dtype)
    ws = bsp.Workspace(geo, wl.batch, wl.beam_width, case.prefix_pages.shape[1], device="cuda")
    plan = ws.plan(geo, wl.batch, wl.beam_width, case.prefix_len, case.tail_len, case.prefix_pages)
    rope = bsp.Rope(40960, wl.head_dim, 1e6)
    pos = synth.token_positions(case)
    q = case.q[torch.from_numpy(case.new_rows).long().cuda()].reshape(n, -1).contiguous()
    q0 = synth.bits(q).copy()
    k_new, v_new = case.k_new.reshape(n, -1), case.v_new.reshape(n, -1)
    k_pool, v_pool = case.k_pool.clone(), case.v_pool.clone()
    bsp.rope_append_kv(plan, rope, torch.from_numpy(pos).cuda(), q, k_new, v_new,
                       torch.from_numpy(case.out_cache_loc).cuda(), k_pool, v_pool)
    assert bsp.read_device_status(plan) == (0, 0)
    ps, D, Hkv = wl.page_size, wl.head_dim, wl.num_kv_heads
    page, off = case.out_cache_loc // ps, case.out_cache_loc % ps
    kp = synth.bits(k_pool)
    np.testing.assert_array_equal(synth.bits(v_pool)[page, :, off], synth.bits(case.v_new))
    assert_rotated(kp[page, :, off].reshape(-1, D), synth.bits(case.k_new).reshape(-1, D), np.repeat(pos, Hkv),
                   wl.dtype, D, False, 1e6, "K")
    rows = np.random.default_rng(0).choice(n, 64, replace=False)
    assert_rotated(synth.bits(q).reshape(n, -1, D)[rows].reshape(-1, D), q0.reshape(n, -1, D)[rows].reshape(-1, D),
                   np.repeat(pos[rows], wl.num_q_heads), wl.dtype, D, False, 1e6, "q")


def test_rope_append_bad_position_or_slot_skips_the_token():
    dtype, Hq, Hkv, D, ps, num_pages, n, max_pos = "bf16", 8, 2, 128, 16, 32, 9, 1000
    plan, ws = make_plan(Hq, Hkv, D, ps, num_pages, dtype, n)
    rope = bsp.Rope(max_pos, D, 1e4)
    g = torch.Generator().manual_seed(3)
    k_new = torch.randn((n, Hkv * D), generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn((n, Hkv * D), generator=g).to(torch.bfloat16).cuda()
    q = torch.randn((n, Hq * D), generator=g).to(torch.bfloat16).cuda()
    loc = torch.randperm(num_pages * ps, generator=g)[:n].to(torch.int32)
    pos = torch.randint(0, max_pos, (n,), generator=g).to(torch.int32)
    pos[3] = 7
    k_pool = torch.zeros((num_pages, Hkv, ps, D), dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    for bad, flag in ((lambda p, l: p.__setitem__(2, max_pos), bsp.DEVFLAG_POSITION),
                      (lambda p, l: p.__setitem__(2, -5), bsp.DEVFLAG_POSITION),
                      (lambda p, l: l.__setitem__(2, num_pages * ps), bsp.DEVFLAG_PAGE_INDEX)):
        p2, l2 = pos.clone(), loc.clone()
        bad(p2, l2)
        k_pool.zero_()
        v_pool.zero_()
        q2 = q.clone()
        bsp.rope_append_kv(plan, rope, p2.cuda(), q2, k_new, v_new, l2.cuda(), k_pool, v_pool)
        st, flags = bsp.read_device_status(plan, clear=True)
        assert flags == flag and bsp.STATUS_NAMES[st] == "BSP_ERR_PAGE_INDEX"
        assert torch.equal(q2[2], q[2])                       # the bad token's q rows untouched
        assert not torch.equal(q2[3], q[3])                   # the others rotated
        slot = int(loc[2])
        if flag == bsp.DEVFLAG_POSITION:
            assert not k_pool[slot // ps, :, slot % ps].any()    # nothing written for it
        for t in (0, 1, 3):
            s_ = int(l2[t])
            assert torch.equal(v_pool[s_ // ps, :, s_ % ps].reshape(-1), v_new[t])


def test_rope_append_argument_checks():
    dtype, Hq, Hkv, D, ps, num_pages, n = "fp16", 4, 2, 64, 16, 8, 3
    plan, ws = make_plan(Hq, Hkv, D, ps, num_pages, dtype, n)
    k = torch.zeros((n, Hkv * D), dtype=torch.float16, device="cuda")
    loc = torch.arange(n, dtype=torch.int32, device="cuda")
    pos = torch.zeros(n, dtype=torch.int32, device="cuda")
    pool = torch.zeros((num_pages, Hkv, ps, D), dtype=torch.float16, device="cuda")
    for rot, inter in ((24, False), (80, False), (0, False), (64, 2)):
        r = bsp.Rope(10, 64, 1e4)
        r.config.rotary_dim, r.config.interleaved = rot, inter
        with pytest.raises(bsp.BspError, match="INVALID_ARG"):
            bsp.rope_append_kv(plan, r, pos, None, k, k, loc, pool, pool)
    r = bsp.Rope(10, 64, 1e4)
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):    # positions on the host
        bsp.rope_append_kv(plan, r, pos.cpu(), None, k, k, loc, pool, pool)
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):    # q row stride below Hq * D
        bsp.rope_append_kv(plan, r, pos, k, k, k, loc, pool, pool)
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):    # a table base that is not > 1
        bsp.Rope(10, 64, 1.0)
    before = pool.clone()
    bsp.rope_append_kv(plan, r, pos[:0], None, k[:0], k[:0], loc[:0], pool, pool)   # n == 0: no-op
    assert torch.equal(before, pool)


E4M3 = np.array([oracle.e4m3_to_double(b) for b in range(256)])


@pytest.mark.parametrize("dtype,Hkv,D,rot,inter,k_mul,v_mul", [
    ("bf16", 8, 128, 128, False, 1.0, 1.0),
    ("fp16", 2, 64, 32, False, 4.0, 0.5),       # partial rotation; large K products saturate
    ("bf16", 4, 256, 128, True, 0.02, 3.0),
])
def test_rope_append_fp8_parity(dtype, Hkv, D, rot, inter, k_mul, v_mul):
    """K rotated in fp32 and quantised: its E4M3 code lies between the codes of the exact rotation times
    the multiplier, moved down and up by the fp32 error bound; V bit-exact; q as the 16-bit append."""
    n, ps, num_pages, max_pos, base = 37, 16, 48, 20000, 1e6
    Hq = 2 * Hkv
    g = torch.Generator().manual_seed(D + rot)
    plan, ws = make_plan(Hq, Hkv, D, ps, num_pages, dtype, n)
    rope = bsp.Rope(max_pos, rot, base, interleaved=inter)
    tdt = TDT[dtype]
    k_new = (torch.randn((n, Hkv * D), generator=g) * 30).to(tdt).cuda()
    v_new = torch.randn((n, Hkv * D), generator=g).to(tdt).cuda()
    q = torch.randn((n, Hq * D), generator=g).to(tdt).cuda()
    q0 = synth.bits(q).copy()
    loc = torch.randperm(num_pages * ps, generator=g)[:n].to(torch.int32)
    pos = torch.randint(0, max_pos, (n,), generator=g).to(torch.int32)
    kp = torch.zeros((num_pages, Hkv, ps, D), dtype=torch.uint8, device="cuda")
    vp = torch.zeros_like(kp)
    bsp.rope_append_kv_fp8(plan, rope, pos.cuda(), q, k_new, v_new, loc.cuda(), kp, vp, k_mul=k_mul, v_mul=v_mul)
    assert bsp.read_device_status(plan) == (0, 0)
    locn, posn = loc.numpy(), pos.numpy()
    page, off = locn // ps, locn % ps
    kb, vb = synth.bits(k_new).reshape(n, -1), synth.bits(v_new).reshape(n, -1)
    kp_o, vp_o = np.zeros(kp.shape, np.uint8), np.zeros(vp.shape, np.uint8)
    q_o = q0.copy()
    oracle.rope_append_kv_fp8(dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, rot=rot, interleaved=inter, base=base,
                              max_pos=max_pos, ps=ps, num_pages=num_pages, positions=posn, out_cache_loc=locn,
                              q_bits=q_o, k_new_bits=kb, v_new_bits=vb, k_pool_bits=kp_o, v_pool_bits=vp_o,
                              k_mul=k_mul, v_mul=v_mul)
    np.testing.assert_array_equal(vp.cpu().numpy(), vp_o)
    got = kp.cpu().numpy()[page, :, off].reshape(n * Hkv, D)
    x = decode(kb.reshape(n * Hkv, D), dtype)
    v = oracle.rope_rotate_rows(x, np.repeat(posn, Hkv), rot=rot, interleaved=inter, base=base)
    m = float(np.float32(k_mul))
    dk = 2.0 ** -21 * pair_bounds(x, rot, inter) * m * 1.001 + np.abs(v * m) * 2.0 ** -23
    lo = np.vectorize(lambda t: E4M3[oracle.round_e4m3(float(t))])(v * m - dk)
    hi = np.vectorize(lambda t: E4M3[oracle.round_e4m3(float(t))])(v * m + dk)
    gv = E4M3[got]
    assert ((gv >= lo) & (gv <= hi)).all()
    assert (got == kp_o[page, :, off].reshape(n * Hkv, D)).mean() > 0.99
    assert_rotated(synth.bits(q).reshape(n * Hq, D), q0.reshape(n * Hq, D), np.repeat(posn, Hq), dtype, rot, inter,
                   base, "q")
