"""Pins for the fp64 oracle, against what the definitions and the mathematics fix.

Each test would fail on a plausible slip in the oracle: a wrong half-float
decode, a dropped max-subtraction or normaliser, a wrong log base, a wrong
scale, a transposed operand, a wrong page / slot / indirection index, a read of
a row beyond the valid length, or a bad append slot.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from beam_search_shared_gb300 import synth

RNG = np.random.default_rng(20261202)


# ---------------------------------------------------------------- half decode
def test_half_decode_matches_numpy_and_bit_shift_for_every_pattern():
    pats = np.arange(65536, dtype=np.uint32)
    f16 = pats.astype(np.uint16).view(np.float16).astype(np.float64)
    bf16 = (pats << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    lib = oracle._load()
    got16 = np.array([lib.orc_half_to_double(int(p), 1) for p in pats])
    gotbf = np.array([lib.orc_half_to_double(int(p), 0) for p in pats])
    np.testing.assert_array_equal(np.isnan(got16), np.isnan(f16))
    np.testing.assert_array_equal(got16[~np.isnan(f16)], f16[~np.isnan(f16)])
    np.testing.assert_array_equal(np.isnan(gotbf), np.isnan(bf16))
    np.testing.assert_array_equal(gotbf[~np.isnan(bf16)], bf16[~np.isnan(bf16)])
    # and the brute force's struct-based decode agrees on a sample
    for p in RNG.integers(0, 65536, 200):
        for dt, ref in (("fp16", f16), ("bf16", bf16)):
            v = brute.half_bits_to_float(int(p), dt)
            assert (math.isnan(v) and math.isnan(ref[p])) or v == ref[p]


# ---------------------------------------------------------------- attend closed forms
def test_attend_single_key_returns_its_value_and_score():
    D = 16
    q, k, v = RNG.normal(size=D), RNG.normal(size=(1, D)), RNG.normal(size=(1, D))
    o, lse = oracle.attend(q, k, v, 0.25)
    np.testing.assert_allclose(o, v[0], rtol=0, atol=1e-15)
    assert lse == pytest.approx(0.25 * float(q @ k[0]), abs=1e-14)


def test_attend_zero_query_is_mean_and_log_n():
    D, n = 8, 37
    K, V = RNG.normal(size=(n, D)), RNG.normal(size=(n, D))
    o, lse = oracle.attend(np.zeros(D), K, V, 0.3)
    np.testing.assert_allclose(o, V.mean(axis=0), rtol=1e-13, atol=1e-14)
    assert lse == pytest.approx(math.log(n), abs=1e-13)


def test_attend_two_keys_sigmoid_weights():
    D = 4
    q, K, V = RNG.normal(size=D), RNG.normal(size=(2, D)), RNG.normal(size=(2, D))
    scale = 1 / math.sqrt(D)
    s0, s1 = scale * q @ K[0], scale * q @ K[1]
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    o, lse = oracle.attend(q, K, V, scale)
    np.testing.assert_allclose(o, w0 * V[0] + (1 - w0) * V[1], rtol=1e-13, atol=1e-14)
    assert lse == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))), abs=1e-13)


def test_attend_equal_values_and_empty_and_huge_scores():
    D, n = 8, 9
    v = RNG.normal(size=D)
    o, _ = oracle.attend(RNG.normal(size=D), RNG.normal(size=(n, D)), np.tile(v, (n, 1)), 1.0)
    np.testing.assert_allclose(o, v, rtol=1e-13, atol=1e-14)
    o, lse = oracle.attend(np.ones(D), np.zeros((0, D)), np.zeros((0, D)), 1.0)
    assert lse == -math.inf and np.all(o == 0)
    # scores of ~1e4 must not overflow: the max is subtracted
    K = np.stack([np.full(D, 1000.0), np.full(D, 999.0)])
    o, lse = oracle.attend(np.ones(D), K, np.eye(2, D), 1.0)
    s0, s1 = 8000.0, 7992.0
    assert lse == pytest.approx(s0 + math.log1p(math.exp(s1 - s0)), rel=1e-15)
    assert o[0] == pytest.approx(1 / (1 + math.exp(s1 - s0)), rel=1e-13)


def test_attend_matches_torch_sdpa_and_logsumexp():
    for D, n in ((64, 1), (64, 130), (128, 257), (256, 31)):
        q, K, V = RNG.normal(size=D), RNG.normal(size=(n, D)), RNG.normal(size=(n, D))
        scale = 1 / math.sqrt(D)
        o, lse = oracle.attend(q, K, V, scale)
        tq = torch.from_numpy(q)[None, None, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, torch.from_numpy(K)[None, None], torch.from_numpy(V)[None, None], scale=scale)
        np.testing.assert_allclose(o, ref.reshape(-1).numpy(), rtol=1e-12, atol=1e-13)
        ref_lse = torch.logsumexp(torch.from_numpy(K) @ torch.from_numpy(q) * scale, 0).item()
        assert lse == pytest.approx(ref_lse, abs=1e-12)


# ---------------------------------------------------------------- merge
def test_merge_of_any_split_equals_unsplit():
    D = 32
    for n in (1, 2, 7, 40):
        q, K, V = RNG.normal(size=D), RNG.normal(size=(n, D)) * 2, RNG.normal(size=(n, D))
        o_all, l_all = oracle.attend(q, K, V, 0.2)
        for k in range(n + 1):
            o1, l1 = oracle.attend(q, K[:k], V[:k], 0.2)
            o2, l2 = oracle.attend(q, K[k:], V[k:], 0.2)
            o, lse = oracle.merge(np.stack([o1, o2]), [l1, l2])
            np.testing.assert_allclose(o, o_all, rtol=1e-12, atol=1e-13)
            assert lse == pytest.approx(l_all, abs=1e-12)
        # a three-way split
        a, b = n // 3, 2 * n // 3
        parts = [oracle.attend(q, K[x:y], V[x:y], 0.2) for x, y in ((0, a), (a, b), (b, n))]
        o, lse = oracle.merge(np.stack([p[0] for p in parts]), [p[1] for p in parts])
        np.testing.assert_allclose(o, o_all, rtol=1e-12, atol=1e-13)
        assert lse == pytest.approx(l_all, abs=1e-12)


def test_merge_closed_forms_and_empty_states():
    D = 4
    o1, o2 = RNG.normal(size=D), RNG.normal(size=D)
    o, lse = oracle.merge(np.stack([o1, o2]), [0.7, 0.7])
    np.testing.assert_allclose(o, (o1 + o2) / 2, rtol=1e-14)
    assert lse == pytest.approx(0.7 + math.log(2), abs=1e-14)
    o, lse = oracle.merge(np.stack([o1, np.zeros(D)]), [1.5, -math.inf])
    np.testing.assert_allclose(o, o1, rtol=0, atol=0)
    assert lse == 1.5
    o, lse = oracle.merge(np.zeros((2, D)), [-math.inf, -math.inf])
    assert lse == -math.inf and np.all(o == 0)


# ---------------------------------------------------------------- paged decode attention
def _tiny(Hq=4, Hkv=2, D=8, ps=4, B=2, W=3, prompt=(0, 13), tail=(0, 3), dtype="bf16"):
    return synth.Workload("t", B, W, Hq, Hkv, D, ps, dtype, prompt, tail)


def _oracle(case, rows=None, prefix_pages=None):
    wl = case.workload
    return oracle.decode_attn(
        dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads,
        D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages, prefix_len=case.prefix_len,
        tail_len=case.tail_len,
        prefix_pages=case.prefix_pages if prefix_pages is None else prefix_pages,
        beam_pages=case.beam_pages, cache_indirection=case.cache_indirection,
        q_bits=synth.bits(case.q), k_pool_bits=synth.bits(case.k_pool),
        v_pool_bits=synth.bits(case.v_pool), scale=1 / math.sqrt(wl.head_dim), rows=rows)


@pytest.mark.parametrize("kw,seed", [
    (dict(), 1), (dict(dtype="fp16"), 2), (dict(Hq=6, Hkv=2, D=16, ps=8), 3),
    (dict(Hq=3, Hkv=1, ps=2, W=4, prompt=(4, 4), tail=(2, 2)), 4),   # prompt fills its last page
    (dict(B=3, prompt=(0, 0), tail=(1, 3)), 5),                    # empty prefixes
    (dict(B=3, prompt=(5, 9), tail=(0, 0)), 6),                    # prefix only
    (dict(Hq=8, Hkv=8, D=4, ps=16, prompt=(1, 40), tail=(0, 8)), 7),
])
def test_paged_oracle_matches_brute_force(kw, seed):
    for full_step in (False, True):
        case = synth.make_case(_tiny(**kw), seed, full_step=full_step)
        wl = case.workload
        O, L = _oracle(case)
        bo, bl = brute.decode_attn(
            dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads,
            D=wl.head_dim, ps=wl.page_size, prefix_len=case.prefix_len, tail_len=case.tail_len,
            prefix_pages=case.prefix_pages.tolist(), beam_pages=case.beam_pages.tolist(),
            cache_indirection=case.cache_indirection.tolist(), q_bits=synth.bits(case.q).tolist(),
            k_pool_bits=synth.bits(case.k_pool).tolist(), v_pool_bits=synth.bits(case.v_pool).tolist(),
            scale=1 / math.sqrt(wl.head_dim))
        np.testing.assert_allclose(O, np.array(bo), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(L, np.array(bl), rtol=1e-12, atol=1e-12)


def _dense_gather(case, r, g):
    """Dense K, V [n, D] of row r, kv head g, gathered with numpy fancy indexing."""
    wl = case.workload
    W, ps = wl.beam_width, wl.page_size
    b, w = divmod(r, W)
    P, T = int(case.prefix_len[b]), int(case.tail_len[b])
    pos = np.arange(P + T)
    src = np.where(pos < P, 0, case.cache_indirection[b, w, pos])
    pages = np.where(pos < P, case.prefix_pages[b, np.minimum(pos // ps, case.prefix_pages.shape[1] - 1)],
                     case.beam_pages[b * W + src, pos // ps])
    k = case.k_pool.float().double().numpy()[pages, g, pos % ps]
    v = case.v_pool.float().double().numpy()[pages, g, pos % ps]
    return k, v


def test_tiny_workload_matches_sdpa_over_dense_gather():
    case = synth.make_case(synth.WORKLOADS["tiny_b1_w4_d64"], 1, full_step=False)
    wl = case.workload
    O, L = _oracle(case)
    G = wl.num_q_heads // wl.num_kv_heads
    scale = 1 / math.sqrt(wl.head_dim)
    for r in range(case.rows):
        for h in range(wl.num_q_heads):
            k, v = _dense_gather(case, r, h // G)
            q = case.q[r, h].double()
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[None, None, None], torch.from_numpy(k)[None, None], torch.from_numpy(v)[None, None],
                scale=scale).reshape(-1)
            np.testing.assert_allclose(O[r, h], ref.numpy(), rtol=1e-12, atol=1e-12)
            assert L[r, h] == pytest.approx(
                torch.logsumexp(torch.from_numpy(k) @ q * scale, 0).item(), abs=1e-12)


def test_cascade_split_of_paged_oracle_is_exact():
    """merge(prefix-only state, tail-only state) equals the unsplit oracle."""
    case = synth.make_case(_tiny(B=3, W=4, prompt=(3, 17), tail=(1, 3)), 11, full_step=False)
    wl = case.workload
    O, L = _oracle(case)
    T0 = np.zeros_like(case.tail_len)
    Op, Lp = oracle.decode_attn(
        dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads,
        D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages, prefix_len=case.prefix_len,
        tail_len=T0, prefix_pages=case.prefix_pages, beam_pages=case.beam_pages,
        cache_indirection=case.cache_indirection, q_bits=synth.bits(case.q),
        k_pool_bits=synth.bits(case.k_pool), v_pool_bits=synth.bits(case.v_pool),
        scale=1 / math.sqrt(wl.head_dim))
    G = wl.num_q_heads // wl.num_kv_heads
    for r in range(case.rows):
        b = r // wl.beam_width
        P = int(case.prefix_len[b])
        for h in range(wl.num_q_heads):
            k, v = _dense_gather(case, r, h // G)
            ot, lt = oracle.attend(case.q[r, h].double().numpy(), k[P:], v[P:], 1 / math.sqrt(wl.head_dim))
            o, lse = oracle.merge(np.stack([Op[r, h], ot]), [Lp[r, h], lt])
            np.testing.assert_allclose(o, O[r, h], rtol=1e-12, atol=1e-12)
            assert lse == pytest.approx(L[r, h], abs=1e-12)


def test_tail_zero_equals_prefix_only_attention():
    case = synth.make_case(_tiny(B=2, W=2, prompt=(9, 9), tail=(0, 0)), 12, full_step=False)
    wl = case.workload
    O, L = _oracle(case)
    for r in range(case.rows):
        for h in range(wl.num_q_heads):
            k, v = _dense_gather(case, r, h // (wl.num_q_heads // wl.num_kv_heads))
            assert k.shape[0] == 9
            o, lse = oracle.attend(case.q[r, h].double().numpy(), k, v, 1 / math.sqrt(wl.head_dim))
            np.testing.assert_array_equal(O[r, h], o)
            assert L[r, h] == lse


def test_rows_beyond_valid_lengths_are_never_read():
    """Poisoning every invalid row with NaN leaves the output bit-identical."""
    wl = _tiny(B=3, W=3, Hq=4, Hkv=2, D=16, ps=8, prompt=(1, 30), tail=(0, 5))
    clean = synth.make_case(wl, 21, full_step=True)
    poisoned = synth.make_case(wl, 21, full_step=True, poison=True)
    assert torch.isnan(poisoned.k_pool.float()).any()
    a = _oracle(clean)
    b = _oracle(poisoned)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert np.isfinite(b[0]).all()


def test_rows_subset_equals_full_rows():
    case = synth.make_case(_tiny(B=3, W=4), 22, full_step=False)
    O, L = _oracle(case)
    rows = np.array([11, 0, 5], np.int32)
    Os, Ls = _oracle(case, rows=rows)
    np.testing.assert_array_equal(Os, O[rows])
    np.testing.assert_array_equal(Ls, L[rows])


def test_bad_indices_are_rejected():
    case = synth.make_case(_tiny(B=2, W=2, prompt=(5, 9), tail=(2, 2)), 23, full_step=False)
    bad = case.prefix_pages.copy()
    bad[0, 0] = case.num_pages
    with pytest.raises(ValueError, match="index"):
        _oracle(case, prefix_pages=bad)
    ci = case.cache_indirection.copy()
    b, w = 1, 1
    ci[b, w, case.prefix_len[b]] = case.workload.beam_width
    case.cache_indirection = ci
    with pytest.raises(ValueError, match="index"):
        _oracle(case)


# ---------------------------------------------------------------- bucket
def test_bucket_rows_table():
    cap = 10368
    table = {0: 1, 1: 256, 5: 256, 40: 256, 255: 256, 256: 256, 257: 512, 2047: 2048,
             2048: 2048, 10000: 10240, 10240: 10240, 10241: 10368, 10368: 10368}
    for valid, rows in table.items():
        assert oracle.bucket_rows(valid, cap) == rows, valid
    assert oracle.bucket_rows(5, 64) == 64


@pytest.mark.parametrize("P", [0, 5, 40, 2047, 10000])
def test_bound_bucket_equals_full_allocation(P):
    """Binding bucket(P) rows or the whole 10368-row allocation gives identical output."""
    wl = synth.WORKLOADS[f"bucketed_prefix_p{P}"]
    case = synth.make_case(wl, 30 + P, full_step=False)
    ps = wl.page_size
    full = np.arange(wl.identity_rows // ps, dtype=np.int32)[None, :]
    bucket_pages = -(-oracle.bucket_rows(P, wl.identity_rows) // ps)
    bound = np.full_like(full, -1)
    bound[0, :bucket_pages] = full[0, :bucket_pages]
    a = _oracle(case, prefix_pages=full)
    b = _oracle(case, prefix_pages=bound)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    assert np.isfinite(a[0]).all()


# ---------------------------------------------------------------- append
def test_append_matches_numpy_scatter_bit_exact():
    for wl_name, seed in (("tiny_b1_w4_d64", 3),):
        case = synth.make_case(synth.WORKLOADS[wl_name], seed, full_step=True)
        wl = case.workload
        kp, vp = synth.bits(case.k_pool).copy(), synth.bits(case.v_pool).copy()
        kn, vn = synth.bits(case.k_new), synth.bits(case.v_new)
        loc = case.out_cache_loc
        oracle.append_kv(Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages,
                         out_cache_loc=loc, k_new_bits=kn, v_new_bits=vn, k_pool_bits=kp, v_pool_bits=vp)
        rk, rv = synth.bits(case.k_pool).copy(), synth.bits(case.v_pool).copy()
        rk[loc // wl.page_size, :, loc % wl.page_size, :] = kn
        rv[loc // wl.page_size, :, loc % wl.page_size, :] = vn
        np.testing.assert_array_equal(kp, rk)
        np.testing.assert_array_equal(vp, rv)


def test_append_strided_source_bad_slot_and_empty():
    Hkv, D, ps, npg, n = 2, 8, 4, 5, 3
    kp = RNG.integers(0, 65536, (npg, Hkv, ps, D)).astype(np.uint16)
    vp = RNG.integers(0, 65536, (npg, Hkv, ps, D)).astype(np.uint16)
    stride = Hkv * D + 8           # a row view of a wider fused projection
    src_k = RNG.integers(0, 65536, (n, stride)).astype(np.uint16)
    src_v = RNG.integers(0, 65536, (n, stride)).astype(np.uint16)
    loc = np.array([19, 0, 7], np.int32)
    k0, v0 = kp.copy(), vp.copy()
    oracle.append_kv(Hkv=Hkv, D=D, ps=ps, num_pages=npg, out_cache_loc=loc, k_new_bits=src_k,
                     v_new_bits=src_v, k_pool_bits=kp, v_pool_bits=vp, row_stride=stride)
    k0[loc // ps, :, loc % ps, :] = src_k[:, :Hkv * D].reshape(n, Hkv, D)
    v0[loc // ps, :, loc % ps, :] = src_v[:, :Hkv * D].reshape(n, Hkv, D)
    np.testing.assert_array_equal(kp, k0)
    np.testing.assert_array_equal(vp, v0)
    before = kp.copy(), vp.copy()
    with pytest.raises(ValueError):
        oracle.append_kv(Hkv=Hkv, D=D, ps=ps, num_pages=npg, out_cache_loc=np.array([3, npg * ps], np.int32),
                         k_new_bits=src_k, v_new_bits=src_v, k_pool_bits=kp, v_pool_bits=vp, row_stride=stride)
    np.testing.assert_array_equal(kp, before[0])
    np.testing.assert_array_equal(vp, before[1])
    oracle.append_kv(Hkv=Hkv, D=D, ps=ps, num_pages=npg, out_cache_loc=np.zeros(0, np.int32),
                     k_new_bits=src_k[:0], v_new_bits=src_v[:0], k_pool_bits=kp, v_pool_bits=vp)
    np.testing.assert_array_equal(kp, before[0])


# ------------------------------------------------------------------ prefill over the cached prefix
def _prefill_oracle(case, causal, k_pool=None, v_pool=None):
    wl = case.workload
    kp = synth.bits(case.k_pool).copy() if k_pool is None else k_pool
    vp = synth.bits(case.v_pool).copy() if v_pool is None else v_pool
    if k_pool is None:
        oracle.append_kv(Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size, num_pages=case.num_pages,
                         out_cache_loc=case.out_cache_loc, k_new_bits=synth.bits(case.k_new),
                         v_new_bits=synth.bits(case.v_new), k_pool_bits=kp, v_pool_bits=vp)
    O, L = oracle.prefill_attn(dtype=wl.dtype, B=wl.batch, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
                               ps=wl.page_size, num_pages=case.num_pages, cached_len=case.cached_len,
                               prompt_len=case.prompt_len, pages=case.pages, causal=causal,
                               q_bits=synth.bits(case.q), k_pool_bits=kp, v_pool_bits=vp,
                               scale=1 / math.sqrt(wl.head_dim))
    return O, L, kp, vp


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed", [1, 2])
def test_prefill_oracle_matches_brute_force(causal, seed):
    wl = synth.PREFILL_WORKLOADS["prefill_tiny_d64"].with_(head_dim=8, page_size=4, cached=(0, 9), prompt=(1, 5))
    case = synth.make_prefill_case(wl, seed)
    O, L, kp, vp = _prefill_oracle(case, causal)
    Ob, Lb = brute.prefill_attn(dtype=wl.dtype, B=wl.batch, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
                                ps=wl.page_size, cached_len=case.cached_len, prompt_len=case.prompt_len,
                                pages=case.pages, causal=causal, q_bits=synth.bits(case.q).tolist(),
                                k_pool_bits=kp.tolist(), v_pool_bits=vp.tolist(), scale=1 / math.sqrt(wl.head_dim))
    np.testing.assert_allclose(O, np.asarray(Ob), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(L, np.asarray(Lb), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_rows_equal_decode_of_a_single_beam(causal):
    """Prompt token i (causal) sees exactly the keys a one-beam decode step sees with a prompt of
    C + i + 1 rows and no tail (C + S rows when not causal): the two oracle functions agree."""
    wl = synth.PREFILL_WORKLOADS["prefill_tiny_d64"].with_(cached=(3, 30), prompt=(2, 9))
    case = synth.make_prefill_case(wl, 7)
    O, L, kp, vp = _prefill_oracle(case, causal)
    qb = synth.bits(case.q)
    r = 0
    for b in range(wl.batch):
        C, S = int(case.cached_len[b]), int(case.prompt_len[b])
        for i in range(S):
            n = C + i + 1 if causal else C + S
            Od, Ld = oracle.decode_attn(
                dtype=wl.dtype, B=1, W=1, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim, ps=wl.page_size,
                num_pages=case.num_pages, prefix_len=[n], tail_len=[0], prefix_pages=case.pages[b:b + 1],
                beam_pages=case.pages[b:b + 1], cache_indirection=np.zeros((1, 1, max(1, n)), np.int32),
                q_bits=qb[r:r + 1], k_pool_bits=kp, v_pool_bits=vp, scale=1 / math.sqrt(wl.head_dim))
            np.testing.assert_array_equal(O[r], Od[0])
            np.testing.assert_array_equal(L[r], Ld[0])
            r += 1


def test_prefill_first_token_of_empty_cache_sees_only_itself():
    """Causal, no cached rows: token 0's only key is its own, so O = v_0 and LSE = scale * q.k_0."""
    wl = synth.PREFILL_WORKLOADS["prefill_tiny_d64"]
    case = synth.make_prefill_case(wl, 3, cached_lengths=[0, 0], prompt_lengths=[3, 1])
    O, L, kp, vp = _prefill_oracle(case, True)
    G = wl.num_q_heads // wl.num_kv_heads
    r = 0
    for b in range(wl.batch):
        for h in range(wl.num_q_heads):
            kb = synth.bits(case.k_new)[r, h // G]
            vb = synth.bits(case.v_new)[r, h // G]
            v0 = np.array([oracle.half_to_double(x, wl.dtype) for x in vb])
            k0 = np.array([oracle.half_to_double(x, wl.dtype) for x in kb])
            q0 = np.array([oracle.half_to_double(x, wl.dtype) for x in synth.bits(case.q)[r, h]])
            np.testing.assert_array_equal(O[r, h], v0)
            assert L[r, h] == pytest.approx(float(q0 @ k0) / math.sqrt(wl.head_dim), rel=1e-12, abs=1e-12)
        r += int(case.prompt_len[b])


def test_prefill_never_reads_rows_past_the_prompt():
    """Rows of the allocation past C + S (and, causally, past each token) hold garbage the
    result must not depend on: poisoning them with NaN changes nothing."""
    wl = synth.PREFILL_WORKLOADS["prefill_tiny_d64"].with_(alloc_rows=96)
    case = synth.make_prefill_case(wl, 5)
    O, L, kp, vp = _prefill_oracle(case, True)
    kp2, vp2 = kp.copy(), vp.copy()
    nan = np.uint16(0x7FC0)
    for b in range(wl.batch):
        end = int(case.cached_len[b] + case.prompt_len[b])
        for pos in range(end, (case.pages.shape[1]) * wl.page_size):
            pg = int(case.pages[b, pos // wl.page_size])
            if pg >= 0:
                kp2[pg, :, pos % wl.page_size] = nan
                vp2[pg, :, pos % wl.page_size] = nan
    O2, L2, _, _ = _prefill_oracle(case, True, k_pool=kp2, v_pool=vp2)
    np.testing.assert_array_equal(O, O2)
    np.testing.assert_array_equal(L, L2)
