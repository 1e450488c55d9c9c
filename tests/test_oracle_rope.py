"""Pins of the oracle's rounding to 16-bit floats and of its RoPE (rotary position embedding) on the
paged append, against the formats' definitions, numpy's own double -> half conversion, brute-force
search, closed forms of rotations and the brute-force restatement in ``oracle.brute``.

The pages name RoPE on the KV write (TensorRT-LLM PR #21738, the review of flash_attn4_kernels.py:
rope_write_kv_paged and its partial-RoPE partner lookup) without defining it; the definition pinned
here is the published one (RoFormer, section 3.2)."""
import math

import numpy as np
import pytest

import oracle
from oracle import brute

DT = ("bf16", "fp16")


# ---------------------------------------------------------------- rounding to the 16-bit formats
@pytest.mark.parametrize("dtype", DT)
def test_round_half_roundtrips_every_finite_pattern(dtype):
    for b in range(0x10000):
        v = oracle.half_to_double(b, dtype)
        if math.isnan(v):
            continue
        assert oracle.round_half(v, dtype) == b, hex(b)


@pytest.mark.parametrize("dtype", DT)
def test_round_half_midpoints_go_to_even(dtype):
    rng = np.random.default_rng(5)
    top = 0x7F7F if dtype == "bf16" else 0x7BFF
    for b in rng.integers(0, top, 400):
        lo, hi = oracle.half_to_double(int(b), dtype), oracle.half_to_double(int(b) + 1, dtype)
        mid = (lo + hi) / 2                      # exact in double
        even = int(b) if int(b) % 2 == 0 else int(b) + 1
        assert oracle.round_half(mid, dtype) == even
        assert oracle.round_half(-mid, dtype) == even | 0x8000
        assert oracle.round_half(math.nextafter(mid, 0.0), dtype) == int(b)
        assert oracle.round_half(math.nextafter(mid, math.inf), dtype) == int(b) + 1


def test_round_half_fp16_matches_numpy_conversion():
    """numpy converts float64 to float16 directly, rounding to nearest even."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal(4000) * np.exp2(rng.integers(-30, 17, 4000))
    x = np.concatenate([x, [65504.0, 65519.999, 65520.0, 1e6, -1e6, 2.0 ** -25, 2.0 ** -26, 0.0, -0.0]])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    got = oracle.round_half_array(x, "fp16")
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("dtype", DT)
def test_round_half_matches_brute_nearest(dtype):
    rng = np.random.default_rng(7)
    lo_e, hi_e = (-135, 128) if dtype == "bf16" else (-26, 16)
    x = rng.standard_normal(600) * np.exp2(rng.integers(lo_e, hi_e, 600).astype(np.float64))
    for v in x:
        assert oracle.round_half(float(v), dtype) == brute.nearest_half_bits(float(v), dtype), v


def test_round_half_special_values():
    assert oracle.round_half(math.nan, "bf16") == 0x7FC0
    assert oracle.round_half(math.nan, "fp16") == 0x7E00
    assert oracle.round_half(math.inf, "fp16") == 0x7C00
    assert oracle.round_half(-math.inf, "bf16") == 0xFF80
    # largest finite binary16 is 65504, spacing 32 there: 65520 ties to even (the infinity pattern)
    assert oracle.round_half(65519.99, "fp16") == 0x7BFF
    assert oracle.round_half(65520.0, "fp16") == 0x7C00
    # bf16: largest finite 0x7F7F = (2 - 2^-7) * 2^127
    top = (2 - 2.0 ** -7) * 2.0 ** 127
    assert oracle.round_half(top, "bf16") == 0x7F7F
    assert oracle.round_half(top + 2.0 ** 119, "bf16") == 0x7F80
    assert oracle.round_half(-0.0, "fp16") == 0x8000
    assert oracle.round_half(1e-40, "fp16") == 0


# ---------------------------------------------------------------- RoPE
def test_rope_frequencies_form_the_geometric_sequence():
    """At position 1 each pair turns by theta_j: theta_0 = 1 and theta_{j+1} / theta_j = base^(-2/rot)."""
    for rot, base in ((8, 10000.0), (128, 1e6), (64, 500000.0)):
        cs = oracle.rope_cos_sin(2, rot, base)
        np.testing.assert_array_equal(cs[0], np.r_[np.ones(rot // 2), np.zeros(rot // 2)])
        theta = np.arctan2(cs[1, rot // 2:], cs[1, :rot // 2])   # all theta_j <= 1 < pi
        assert theta[0] == pytest.approx(1.0, abs=1e-15)
        np.testing.assert_allclose(theta[1:] / theta[:-1], base ** (-2.0 / rot), rtol=1e-12)


def test_rope_rotation_is_the_complex_product():
    """Interleaved pairs as complex numbers: each is multiplied by e^{i p theta_j} (numpy complex exp)."""
    rng = np.random.default_rng(8)
    rot, base, D = 16, 10000.0, 24
    cs = oracle.rope_cos_sin(1000, rot, base)
    theta = np.arctan2(oracle.rope_cos_sin(2, rot, base)[1, rot // 2:], oracle.rope_cos_sin(2, rot, base)[1, :rot // 2])
    for p in (0, 1, 7, 999):
        x = rng.standard_normal(D)
        y = oracle.rope_rotate(x, rot=rot, interleaved=True, base=base, pos=p)
        z = (x[0:rot:2] + 1j * x[1:rot:2]) * np.exp(1j * p * theta)
        np.testing.assert_allclose(y[0:rot:2], z.real, atol=1e-12)
        np.testing.assert_allclose(y[1:rot:2], z.imag, atol=1e-12)
        np.testing.assert_array_equal(y[rot:], x[rot:])                  # partial: the rest passes
        np.testing.assert_allclose(cs[p, :rot // 2] + 1j * cs[p, rot // 2:], np.exp(1j * p * theta), atol=1e-12)


def test_rope_position_zero_is_identity_and_layouts_are_a_permutation():
    rng = np.random.default_rng(9)
    rot, D = 32, 64
    x = rng.standard_normal(D)
    for inter in (False, True):
        np.testing.assert_array_equal(oracle.rope_rotate(x, rot=rot, interleaved=inter, base=1e4, pos=0), x)
    # rotate-half pair j is (j, j + rot/2); interleaved pair j is (2j, 2j + 1)
    perm = np.arange(D)
    perm[:rot:2] = np.arange(rot // 2)
    perm[1:rot:2] = np.arange(rot // 2) + rot // 2
    for p in (3, 4000):
        y_half = oracle.rope_rotate(x, rot=rot, interleaved=False, base=1e4, pos=p)
        y_int = oracle.rope_rotate(x[perm], rot=rot, interleaved=True, base=1e4, pos=p)
        np.testing.assert_array_equal(y_int, y_half[perm])


def test_rope_is_a_rotation_group_and_encodes_relative_position():
    rng = np.random.default_rng(10)
    rot, D, base = 64, 64, 1e6
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    R = lambda v, p: oracle.rope_rotate(v, rot=rot, interleaved=False, base=base, pos=p)
    for m, n in ((5, 2), (1000, 999), (4096, 17)):
        # norm of every pair kept
        y = R(q, m)
        np.testing.assert_allclose(y[:32] ** 2 + y[32:] ** 2, q[:32] ** 2 + q[32:] ** 2, rtol=1e-12)
        # R(m) R(n) = R(m + n)
        np.testing.assert_allclose(R(R(q, m), n), R(q, m + n), atol=1e-9)
        # <R(m) q, R(n) k> depends on m - n only
        assert float(R(q, m) @ R(k, n)) == pytest.approx(float(R(q, m - n) @ k), abs=1e-9)


def _tiny_case(dtype, rng, n=5, Hq=4, Hkv=2, D=32, ps=4, num_pages=6):
    k_new = rng.standard_normal((n, Hkv, D)) * 3
    v_new = rng.standard_normal((n, Hkv, D))
    q = rng.standard_normal((n, Hq, D)) * 2
    bits = lambda a: oracle.round_half_array(a, dtype)
    loc = rng.choice(num_pages * ps, n, replace=False).astype(np.int32)
    pos = rng.integers(0, 5000, n).astype(np.int32)
    kp = rng.integers(0, 0x3000, (num_pages, Hkv, ps, D)).astype(np.uint16)
    vp = rng.integers(0, 0x3000, (num_pages, Hkv, ps, D)).astype(np.uint16)
    return bits(q), bits(k_new), bits(v_new), kp, vp, loc, pos


@pytest.mark.parametrize("dtype", DT)
@pytest.mark.parametrize("rot,inter", [(32, False), (16, False), (16, True), (32, True)])
def test_rope_append_matches_brute(dtype, rot, inter):
    rng = np.random.default_rng(11 + rot + inter)
    n, Hq, Hkv, D, ps, npg = 5, 4, 2, 32, 4, 6
    q, kn, vn, kp, vp, loc, pos = _tiny_case(dtype, rng)
    q_o, kp_o, vp_o = q.copy(), kp.copy(), vp.copy()
    oracle.rope_append_kv(dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, rot=rot, interleaved=inter, base=10000.0, max_pos=5000,
                          ps=ps, num_pages=npg, positions=pos, out_cache_loc=loc, q_bits=q_o,
                          k_new_bits=kn.reshape(n, -1), v_new_bits=vn.reshape(n, -1), k_pool_bits=kp_o,
                          v_pool_bits=vp_o)
    q_b, kp_b, vp_b = q.tolist(), kp.tolist(), vp.tolist()
    brute.rope_append_kv(dtype=dtype, Hq=Hq, Hkv=Hkv, D=D, rot=rot, interleaved=inter, base=10000.0, ps=ps,
                         positions=pos.tolist(), out_cache_loc=loc.tolist(), q_bits=q_b, k_new_bits=kn.tolist(),
                         v_new_bits=vn.tolist(), k_pool_bits=kp_b, v_pool_bits=vp_b)
    np.testing.assert_array_equal(q_o, np.array(q_b, np.uint16))
    np.testing.assert_array_equal(kp_o, np.array(kp_b, np.uint16))
    np.testing.assert_array_equal(vp_o, np.array(vp_b, np.uint16))
    # V rows and position-0 K rows are copies; untouched slots keep their bits
    for i in range(n):
        pg, off = loc[i] // ps, loc[i] % ps
        np.testing.assert_array_equal(vp_o[pg, :, off], vn[i])
    touched = np.zeros((npg, ps), bool)
    touched[loc // ps, loc % ps] = True
    np.testing.assert_array_equal(kp_o.transpose(0, 2, 1, 3)[~touched], kp.transpose(0, 2, 1, 3)[~touched])


def test_rope_append_rejects_bad_slot_or_position_without_writing():
    rng = np.random.default_rng(12)
    n, Hq, Hkv, D, ps, npg = 5, 4, 2, 32, 4, 6
    q, kn, vn, kp, vp, loc, pos = _tiny_case("bf16", rng)
    kw = dict(dtype="bf16", Hq=Hq, Hkv=Hkv, D=D, rot=32, interleaved=False, base=1e4, ps=ps, num_pages=npg,
              k_new_bits=kn.reshape(n, -1), v_new_bits=vn.reshape(n, -1))
    for bad_loc, bad_pos, max_pos in ((True, False, 5000), (False, True, 5000), (False, False, int(pos.max()))):
        l2, p2 = loc.copy(), pos.copy()
        if bad_loc:
            l2[3] = npg * ps
        if bad_pos:
            p2[1] = -1
        q_o, kp_o, vp_o = q.copy(), kp.copy(), vp.copy()
        with pytest.raises(ValueError):
            oracle.rope_append_kv(max_pos=max_pos, positions=p2, out_cache_loc=l2, q_bits=q_o, k_pool_bits=kp_o,
                                  v_pool_bits=vp_o, **kw)
        np.testing.assert_array_equal(q_o, q)
        np.testing.assert_array_equal(kp_o, kp)
        np.testing.assert_array_equal(vp_o, vp)


def test_rope_append_position_zero_and_no_q():
    rng = np.random.default_rng(13)
    n, Hq, Hkv, D, ps, npg = 5, 4, 2, 32, 4, 6
    q, kn, vn, kp, vp, loc, pos = _tiny_case("fp16", rng)
    kp_o, vp_o = kp.copy(), vp.copy()
    oracle.rope_append_kv(dtype="fp16", Hq=Hq, Hkv=Hkv, D=D, rot=32, interleaved=False, base=1e4, max_pos=5000,
                          ps=ps, num_pages=npg, positions=np.zeros(n, np.int32), out_cache_loc=loc, q_bits=None,
                          k_new_bits=kn.reshape(n, -1), v_new_bits=vn.reshape(n, -1), k_pool_bits=kp_o,
                          v_pool_bits=vp_o)
    for i in range(n):
        pg, off = loc[i] // ps, loc[i] % ps
        np.testing.assert_array_equal(kp_o[pg, :, off], kn[i])


def test_array_forms_equal_the_scalar_routines():
    rng = np.random.default_rng(14)
    x = rng.standard_normal(300) * np.exp2(rng.integers(-20, 20, 300))
    for dtype in DT:
        np.testing.assert_array_equal(oracle.round_half_array(x, dtype),
                                      np.array([oracle.round_half(v, dtype) for v in x], np.uint16))
    rows = rng.standard_normal((7, 32))
    pos = rng.integers(0, 9000, 7)
    y = oracle.rope_rotate_rows(rows, pos, rot=16, interleaved=True, base=5e5)
    for i in range(7):
        np.testing.assert_array_equal(y[i], oracle.rope_rotate(rows[i], rot=16, interleaved=True, base=5e5, pos=pos[i]))
