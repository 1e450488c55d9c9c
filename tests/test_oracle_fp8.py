"""Pins of the oracle's FP8 (E4M3) KV write: the format's decoding and round-to-nearest-even with
saturation against the format definition and torch's own float -> float8_e4m3fn conversion, and the
quantising paged append against a numpy/torch restatement.

The pages ask that an fp8 source can be written to an fp8 cache and that the write converts between the
fused KV write (TensorRT-LLM PR #18614, the review follow-up commit on the fused KV write and
the review of msa_scatter.py); the quantisation multiplier and the saturation are the plain readings
(a per-tensor scale, CUDA's satfinite conversion)."""
import math

import numpy as np
import pytest
import torch

import oracle


def test_every_pattern_decodes_and_round_trips():
    for b in range(256):
        v = oracle.e4m3_to_double(b)
        if b & 0x7F == 0x7F:
            assert math.isnan(v)
            continue
        assert oracle.round_e4m3(v) == b, hex(b)
    # the format's landmarks
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_to_double(0x38) == 1.0
    # decoding agrees with torch's float8_e4m3fn
    bits = torch.arange(256, dtype=torch.uint8)
    t = bits.view(torch.float8_e4m3fn).double().numpy()
    o = np.array([oracle.e4m3_to_double(b) for b in range(256)])
    np.testing.assert_array_equal(np.isnan(t), np.isnan(o))
    np.testing.assert_array_equal(t[~np.isnan(t)], o[~np.isnan(o)])


def test_midpoints_go_to_even_and_saturation():
    for b in range(0, 0x7D):
        lo, hi = oracle.e4m3_to_double(b), oracle.e4m3_to_double(b + 1)
        mid = (lo + hi) / 2
        even = b if b % 2 == 0 else b + 1
        assert oracle.round_e4m3(mid) == even
        assert oracle.round_e4m3(-mid) == even | 0x80
        assert oracle.round_e4m3(math.nextafter(mid, 0.0)) == b
        assert oracle.round_e4m3(math.nextafter(mid, math.inf)) == b + 1
    for v in (448.0, 449.0, 463.9, 464.0, 1e6, math.inf):
        assert oracle.round_e4m3(v) == 0x7E
        assert oracle.round_e4m3(-v) == 0xFE
    assert oracle.round_e4m3(math.nan) == 0x7F
    assert oracle.round_e4m3(2.0 ** -10) == 0x00          # half the smallest subnormal: ties to even (zero)
    assert oracle.round_e4m3(math.nextafter(2.0 ** -10, 1.0)) == 0x01


def test_rounding_matches_torch_inside_the_range():
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(5000) * np.exp2(rng.integers(-12, 9, 5000))).astype(np.float32)
    x = x[np.abs(x) < 464]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.round_e4m3(float(v)) for v in x], np.uint8)
    np.testing.assert_array_equal(got, want)


def _restated(x_bits, dtype, mul):
    """fp32 product with the multiplier, clamped to +-448 (satfinite), torch's RNE conversion."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    x = torch.from_numpy(x_bits.view(np.int16)).view(tdt).float()
    y = x * torch.tensor(mul, dtype=torch.float32)
    return y.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_fp8_append_matches_restatement(dtype):
    rng = np.random.default_rng(22)
    n, Hkv, D, ps, npg = 7, 2, 64, 4, 6
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    kn = (torch.randn(n, Hkv * D, generator=torch.Generator().manual_seed(1)) * 40).to(tdt)
    vn = (torch.randn(n, Hkv * D, generator=torch.Generator().manual_seed(2)) * 3).to(tdt)
    kb, vb = kn.view(torch.int16).numpy().view(np.uint16), vn.view(torch.int16).numpy().view(np.uint16)
    loc = rng.choice(npg * ps, n, replace=False).astype(np.int32)
    kp = rng.integers(0, 256, (npg, Hkv, ps, D)).astype(np.uint8)
    vp = rng.integers(0, 256, (npg, Hkv, ps, D)).astype(np.uint8)
    kp0, vp0 = kp.copy(), vp.copy()
    k_mul, v_mul = 0.37, 11.0          # K saturates in places (|x| * 0.37 up to ~60; * 40 -> some > 448)
    oracle.append_kv_fp8(src_dtype=dtype, Hkv=Hkv, D=D, ps=ps, num_pages=npg, out_cache_loc=loc, k_new_bits=kb,
                         v_new_bits=vb, k_pool_bits=kp, v_pool_bits=vp, k_mul=k_mul * 40, v_mul=v_mul)
    wk = _restated(kb, dtype, np.float32(k_mul * 40)).reshape(n, Hkv, D)
    wv = _restated(vb, dtype, np.float32(v_mul)).reshape(n, Hkv, D)
    assert (wk == 0x7E).any() or (wk == 0xFE).any()     # the saturating branch is exercised
    for i in range(n):
        pg, off = loc[i] // ps, loc[i] % ps
        np.testing.assert_array_equal(kp[pg, :, off], wk[i])
        np.testing.assert_array_equal(vp[pg, :, off], wv[i])
    touched = np.zeros((npg, ps), bool)
    touched[loc // ps, loc % ps] = True
    np.testing.assert_array_equal(kp.transpose(0, 2, 1, 3)[~touched], kp0.transpose(0, 2, 1, 3)[~touched])


def test_fp8_source_is_copied_and_bad_slot_writes_nothing():
    rng = np.random.default_rng(23)
    n, Hkv, D, ps, npg = 5, 2, 32, 4, 4
    kb = rng.integers(0, 256, (n, Hkv * D)).astype(np.uint8)
    vb = rng.integers(0, 256, (n, Hkv * D)).astype(np.uint8)
    loc = rng.choice(npg * ps, n, replace=False).astype(np.int32)
    kp = np.zeros((npg, Hkv, ps, D), np.uint8)
    vp = np.zeros_like(kp)
    oracle.append_kv_fp8(src_dtype="e4m3", Hkv=Hkv, D=D, ps=ps, num_pages=npg, out_cache_loc=loc, k_new_bits=kb,
                         v_new_bits=vb, k_pool_bits=kp, v_pool_bits=vp, k_mul=3.0, v_mul=3.0)
    for i in range(n):
        pg, off = loc[i] // ps, loc[i] % ps
        np.testing.assert_array_equal(kp[pg, :, off].reshape(-1), kb[i])
        np.testing.assert_array_equal(vp[pg, :, off].reshape(-1), vb[i])
    bad = loc.copy()
    bad[2] = npg * ps
    kp2, vp2 = kp.copy(), vp.copy()
    with pytest.raises(ValueError):
        oracle.append_kv_fp8(src_dtype="e4m3", Hkv=Hkv, D=D, ps=ps, num_pages=npg, out_cache_loc=bad, k_new_bits=kb,
                             v_new_bits=vb, k_pool_bits=kp2, v_pool_bits=vp2)
    np.testing.assert_array_equal(kp2, kp)
    np.testing.assert_array_equal(vp2, vp)


@pytest.mark.parametrize("dtype,inter", [("bf16", False), ("fp16", True)])
def test_rope_fp8_append_is_the_composition_of_its_pinned_parts(dtype, inter):
    """K: the exact rotation (oracle.rope_rotate, pinned) times the multiplier, rounded by round_e4m3
    (pinned); V: the quantising append (pinned); q: the 16-bit RoPE append (pinned)."""
    rng = np.random.default_rng(31)
    n, Hq, Hkv, D, ps, npg, rot = 5, 4, 2, 32, 4, 6, 16
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    kb = (torch.randn(n, Hkv * D) * 30).to(tdt).view(torch.int16).numpy().view(np.uint16)
    vb = torch.randn(n, Hkv * D).to(tdt).view(torch.int16).numpy().view(np.uint16)
    qb = torch.randn(n, Hq * D).to(tdt).view(torch.int16).numpy().view(np.uint16)
    loc = rng.choice(npg * ps, n, replace=False).astype(np.int32)
    pos = rng.integers(0, 3000, n).astype(np.int32)
    kp = np.zeros((npg, Hkv, ps, D), np.uint8)
    vp = np.zeros_like(kp)
    q1 = qb.copy()
    k_mul, v_mul = 2.5, 0.75
    oracle.rope_append_kv_fp8(dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, rot=rot, interleaved=inter, base=1e4, max_pos=3000,
                              ps=ps, num_pages=npg, positions=pos, out_cache_loc=loc, q_bits=q1, k_new_bits=kb,
                              v_new_bits=vb, k_pool_bits=kp, v_pool_bits=vp, k_mul=k_mul, v_mul=v_mul)
    vp2 = np.zeros_like(vp)
    oracle.append_kv_fp8(src_dtype=dtype, Hkv=Hkv, D=D, ps=ps, num_pages=npg, out_cache_loc=loc, k_new_bits=kb,
                         v_new_bits=vb, k_pool_bits=np.zeros_like(kp), v_pool_bits=vp2, k_mul=1.0, v_mul=v_mul)
    np.testing.assert_array_equal(vp, vp2)
    q2 = qb.copy()
    oracle.rope_append_kv(dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, rot=rot, interleaved=inter, base=1e4, max_pos=3000, ps=ps,
                          num_pages=npg, positions=pos, out_cache_loc=loc, q_bits=q2, k_new_bits=kb, v_new_bits=vb,
                          k_pool_bits=np.zeros((npg, Hkv, ps, D), np.uint16), v_pool_bits=np.zeros((npg, Hkv, ps, D), np.uint16))
    np.testing.assert_array_equal(q1, q2)
    for i in range(n):
        for h in range(Hkv):
            x = np.array([oracle.half_to_double(int(b), dtype) for b in kb[i, h * D:(h + 1) * D]])
            y = oracle.rope_rotate(x, rot=rot, interleaved=inter, base=1e4, pos=int(pos[i]))
            want = [oracle.round_e4m3(float(v) * float(np.float32(k_mul))) for v in y]
            np.testing.assert_array_equal(kp[loc[i] // ps, h, loc[i] % ps], np.array(want, np.uint8))


def test_e4m3_values_are_exact_in_both_16bit_formats():
    for dtype in ("bf16", "fp16"):
        bits = oracle.e4m3_to_half_bits(np.arange(256, dtype=np.uint8), dtype)
        for b in range(256):
            v = oracle.e4m3_to_double(b)
            h = oracle.half_to_double(int(bits[b]), dtype)
            assert (math.isnan(v) and math.isnan(h)) or v == h, (dtype, b)
    # the field decoder of the brute force agrees with the oracle's decoder
    from oracle import brute
    for b in range(256):
        v, w = oracle.e4m3_to_double(b), brute.e4m3_bits_to_float(b)
        assert (math.isnan(v) and math.isnan(w)) or v == w


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_decode_attention_over_e4m3_pools_matches_brute_force(dtype):
    """The C oracle through exact 16-bit carriers against the nested-list restatement that scales each
    decoded key and value itself; tiny paged cases with prompts, tails and the indirection."""
    from oracle import brute
    from beam_search_shared_gb300 import synth
    rng = np.random.default_rng(41)
    for seed, (k_scale, v_scale) in enumerate([(1.0, 1.0), (0.0625, 3.0), (0.3, 0.02)]):
        wl = synth.WORKLOADS["tiny_b1_w4_d64"].with_(batch=2, prompt=(5, 40), tail=(0, 3), page_size=8,
                                                       num_q_heads=4, num_kv_heads=2, head_dim=16, dtype=dtype)
        case = synth.make_case(wl, 300 + seed, full_step=False, device="cpu")
        k8 = rng.integers(0, 256, case.k_pool.shape).astype(np.uint8)
        v8 = rng.integers(0, 256, case.v_pool.shape).astype(np.uint8)
        k8[(k8 & 0x7F) == 0x7F] = 0x38     # no NaN patterns
        v8[(v8 & 0x7F) == 0x7F] = 0x38
        kw = dict(dtype=dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
                  ps=wl.page_size, prefix_len=case.prefix_len, tail_len=case.tail_len, prefix_pages=case.prefix_pages,
                  beam_pages=case.beam_pages, cache_indirection=case.cache_indirection, scale=0.25)
        q = synth.bits(case.q)
        O, L = oracle.decode_attn_fp8(num_pages=case.num_pages, q_bits=q, k_pool_bits=k8, v_pool_bits=v8,
                                      k_scale=k_scale, v_scale=v_scale, **kw)
        Ob, Lb = brute.decode_attn_fp8(q_bits=q.tolist(), k_pool_bits=k8.tolist(), v_pool_bits=v8.tolist(),
                                       k_scale=k_scale, v_scale=v_scale, **kw)
        np.testing.assert_allclose(O, np.array(Ob), rtol=1e-9, atol=1e-12)
        Lb = np.array(Lb)
        np.testing.assert_array_equal(np.isneginf(L), np.isneginf(Lb))
        fin = ~np.isneginf(L)
        np.testing.assert_allclose(L[fin], Lb[fin], rtol=1e-9, atol=1e-9)
