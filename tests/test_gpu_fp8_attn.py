"""Decode attention over FP8 E4M3 pools (bsp_decode_attn_fp8) against the oracle (oracle.decode_attn_fp8:
the pools' codes decoded exactly, keys scaled by k_scale, values by v_scale), at the parity tests'
tolerance: the E4M3 tiles are widened exactly to the q dtype, so the arithmetic is that of the 16-bit path.
The pools are random E4M3 bit patterns (synth.e4m3_codes) in the layout of the case's 16-bit pools."""
import math

import numpy as np
import pytest
import torch

import oracle
from beam_search_shared_gb300 import bsp, synth

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3


class Fp8Step:
    """Device buffers of a case with E4M3 pools, a plan of an E4M3 geometry, and the E4M3 attention."""

    def __init__(self, case, seed, k_scale, v_scale):
        wl = case.workload
        g = torch.Generator().manual_seed(seed)
        self.case = case
        self.k8 = synth.e4m3_codes(tuple(case.k_pool.shape), g)
        self.v8 = synth.e4m3_codes(tuple(case.v_pool.shape), g)
        self.k_scale, self.v_scale = k_scale, v_scale
        self.geo = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, case.num_pages,
                                wl.dtype, kv_dtype=bsp.KV_DTYPE_E4M3)
        self.q = case.q.cuda()
        self.kd, self.vd = self.k8.cuda(), self.v8.cuda()
        self.beam_pages = torch.from_numpy(case.beam_pages).cuda()
        self.ci = torch.from_numpy(case.cache_indirection).cuda()
        R = wl.batch * wl.beam_width
        self.o = torch.full((R, wl.num_q_heads, wl.head_dim), float("nan"), dtype=self.q.dtype, device="cuda")
        self.lse = torch.full((R, wl.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
        self.scale = 1.0 / math.sqrt(wl.head_dim)
        self.ws = bsp.Workspace(self.geo, max(1, wl.batch), wl.beam_width, case.prefix_pages.shape[1])
        self.plan = self.ws.plan(self.geo, wl.batch, wl.beam_width, case.prefix_len, case.tail_len,
                                 case.prefix_pages, bsp.MAX_TAIL)

    def attend(self, flags=0):
        bsp.decode_attn_fp8(self.plan, self.q, self.kd, self.vd, self.beam_pages, self.ci, self.scale, self.k_scale,
                            self.v_scale, self.o, self.lse, flags=flags)

    def oracle(self, rows=None):
        c, wl = self.case, self.case.workload
        return oracle.decode_attn_fp8(
            dtype=wl.dtype, B=wl.batch, W=wl.beam_width, Hq=wl.num_q_heads, Hkv=wl.num_kv_heads, D=wl.head_dim,
            ps=wl.page_size, num_pages=c.num_pages, prefix_len=c.prefix_len, tail_len=c.tail_len,
            prefix_pages=c.prefix_pages, beam_pages=c.beam_pages, cache_indirection=c.cache_indirection,
            q_bits=synth.bits(c.q), k_pool_bits=self.k8.numpy(), v_pool_bits=self.v8.numpy(), scale=self.scale,
            k_scale=self.k_scale, v_scale=self.v_scale, rows=rows)


def assert_close(o, lse, O, L):
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    assert np.isfinite(o).all()
    err = np.abs(o - O)
    assert (err <= ATOL + RTOL * np.abs(O)).all(), err.max()
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(L))
    both = np.isneginf(lse) & np.isneginf(L)
    assert (np.abs(lse[~both] - L[~both]) <= LSE_TOL).all()


@pytest.mark.parametrize("name,batch,k_scale,v_scale,layout", [
    ("qwen3_0p6b_b64_w30", 6, 1.0, 1.0, 1),      # the 0.6B-shaped layer: alternating-tile kernel
    ("wide_beam_b128_w96", 2, 0.25, 2.0, 2),     # the wide-beam layer: wide kernel, the prompt read once
    ("qwen3_4b_fp16_d128", 5, 0.5, 0.75, 1),     # fp16 queries, tails up to 8 tokens
    ("qwen3_4b_fp16_d64", 4, 1.0, 0.125, 1),     # head_dim 64: the whole-tile widening
    ("tiny_b1_w4_d64", 1, 2.0, 1.0, 1),
])
def test_fp8_attention_matches_oracle(name, batch, k_scale, v_scale, layout):
    wl = synth.WORKLOADS[name].scaled(batch)
    case = synth.make_case(wl, 500 + batch, full_step=False, device="cpu")
    st = Fp8Step(case, 600 + batch, k_scale, v_scale)
    assert st.plan.layout == layout
    st.attend(flags=bsp.FLAG_CHECK)
    O, L = st.oracle()
    assert_close(st.o, st.lse, O, L)


@pytest.mark.parametrize("kw,batch", [
    (dict(num_q_heads=24, num_kv_heads=8, beam_width=42), 3),   # G = 3: row blocks of at most 40 beams
    (dict(num_q_heads=24, num_kv_heads=8, beam_width=50), 2),   # G = 3, 150 rows: the wide kernel
    (dict(num_q_heads=64, num_kv_heads=8, beam_width=12), 2),   # G = 8: 96 rows in one alternating-tile block
    (dict(num_q_heads=64, num_kv_heads=8, beam_width=20), 2),   # G = 8, 160 rows: the wide kernel
    (dict(page_size=16, beam_width=7), 4),
    (dict(page_size=128), 3),
    (dict(head_dim=64, num_q_heads=32, num_kv_heads=8, beam_width=40), 3),   # head_dim 64, 160 rows: wide
    (dict(head_dim=64, num_q_heads=16, num_kv_heads=8, beam_width=96, dtype="fp16"), 2),  # D 64, fp16, 192 rows
    (dict(head_dim=64, beam_width=30), 3),                                    # head_dim 64, 60 rows: alternating
])
def test_fp8_attention_shapes(kw, batch):
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(batch).with_(**kw)
    case = synth.make_case(wl, 700 + batch, full_step=False, device="cpu")
    st = Fp8Step(case, 800 + batch, 0.5, 1.5)
    assert st.plan.layout in (1, 2)
    G = wl.num_q_heads // wl.num_kv_heads
    if wl.head_dim == 64:  # the intended kernel: two blocks above 128 rows per (request, kv head)
        assert st.plan.layout == (2 if wl.beam_width * G > 128 else 1)
    st.attend(flags=bsp.FLAG_CHECK)
    O, L = st.oracle()
    assert_close(st.o, st.lse, O, L)


def test_fp8_attention_split_prompts_long_tails_and_empty_requests():
    """Key splits (few units), tails that the tail kernel finishes, a request without a prompt and one
    without anything, prompts ending inside a page and inside a tile."""
    wl = synth.WORKLOADS["qwen3_4b_fp16_d128"].scaled(6)
    case = synth.make_case(wl, 901, full_step=False, device="cpu",
                           prompt_lengths=[3000, 129, 0, 0, 1, 517], tail_lengths=[8, 5, 3, 0, 8, 1])
    st = Fp8Step(case, 902, 0.75, 0.5)
    assert st.plan.tail_requests > 0
    st.attend(flags=bsp.FLAG_CHECK)
    O, L = st.oracle()
    assert_close(st.o, st.lse, O, L)


def test_fp8_attention_full_size_wide_beam_sampled():
    """The wide-beam workload at full size (batch 128, beam 96): every output row computed, sampled rows
    checked against the oracle."""
    wl = synth.WORKLOADS["wide_beam_b128_w96"]
    case = synth.make_case(wl, 1000, full_step=False, device="cpu")
    st = Fp8Step(case, 1001, 0.5, 0.5)
    assert st.plan.layout == 2
    st.attend(flags=bsp.FLAG_CHECK)
    R = wl.batch * wl.beam_width
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([rng.integers(0, R, 32), [0, R - 1]])).astype(np.int32)
    O, L = st.oracle(rows=rows)
    assert_close(st.o[rows], st.lse[rows], O, L)
    assert torch.isfinite(st.o).all()


def test_fp8_entry_points_refuse_the_other_pool_type():
    wl = synth.WORKLOADS["qwen3_0p6b_b64_w30"].scaled(2)
    case = synth.make_case(wl, 11, full_step=True, device="cpu")
    st = Fp8Step(case, 12, 1.0, 1.0)
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):    # a 16-bit entry point, an E4M3 plan
        bsp.decode_attn(st.plan, st.q, st.kd, st.vd, st.beam_pages, st.ci, st.scale, st.o, st.lse)
    n = case.out_cache_loc.shape[0]
    kn = case.k_new.reshape(n, -1).cuda()
    vn = case.v_new.reshape(n, -1).cuda()
    loc = torch.from_numpy(case.out_cache_loc).cuda()
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.append_kv(st.plan, kn, vn, loc, st.kd, st.vd)
    for ks, vs in ((0.0, 1.0), (1.0, float("inf")), (-1.0, 1.0)):
        with pytest.raises(bsp.BspError, match="INVALID_ARG"):
            bsp.decode_attn_fp8(st.plan, st.q, st.kd, st.vd, st.beam_pages, st.ci, st.scale, ks, vs, st.o, st.lse)
    # the E4M3 write accepts the E4M3 plan, and the attention then reads the written rows
    bsp.append_kv_fp8(st.plan, kn, vn, loc, st.kd, st.vd)
    st.attend(flags=bsp.FLAG_CHECK)
    assert torch.isfinite(st.o).all()
    # the E4M3 entry point refuses a plan of 16-bit pools
    geo16 = bsp.geometry(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, case.num_pages, wl.dtype)
    ws16 = bsp.Workspace(geo16, wl.batch, wl.beam_width, case.prefix_pages.shape[1])
    p16 = ws16.plan(geo16, wl.batch, wl.beam_width, case.prefix_len, case.tail_len, case.prefix_pages)
    with pytest.raises(bsp.BspError, match="INVALID_ARG"):
        bsp.decode_attn_fp8(p16, st.q, st.kd, st.vd, st.beam_pages, st.ci, st.scale, 1.0, 1.0, st.o, st.lse)
    # and the no-allocation entry point has 16-bit pools only
    with pytest.raises(bsp.BspError, match="UNSUPPORTED"):
        bsp.decode_attn_noalloc(st.geo, wl.batch, wl.beam_width, case.prefix_len, case.tail_len, case.prefix_pages,
                                bsp.MAX_TAIL, st.q, st.kd, st.vd, st.beam_pages, st.ci, st.scale, st.o, st.lse)
