"""Host-side tests of libbsp.so: exports, status codes, bucket rule and planning.

No CUDA device is needed: only entry points that stay on the host are called.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from beam_search_shared_gb300 import bsp, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STATUS_OFFSET = 256  # device status words precede the plan image


@pytest.fixture(scope="module")
def lib():
    build.build()
    return bsp.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "bsp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsp_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(bsp.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n
    # nothing else leaks out of the library (symbols are hidden by default)
    out = os.popen(f"nm -D --defined-only {build.LIB}").read()
    exported = sorted(set(re.findall(r" T (bsp_\w+)", out)))
    assert exported == names


def test_status_strings(lib):
    for code, name in bsp.STATUS_NAMES.items():
        assert bsp.status_string(code)
    assert bsp.status_string(99) == "unknown status"


def test_bucket_rows_matches_oracle_rule(lib):
    for cap in (1, 64, 300, 10368):
        for valid in list(range(0, 600)) + [2047, 2048, 10000, 10240, 10241, 10368, 20000]:
            assert bsp.bucket_rows(valid, cap) == oracle.bucket_rows(valid, cap), (valid, cap)
    assert bsp.bucket_rows(5, 0) == -1


def geo(Hq=16, Hkv=8, D=128, ps=32, npages=1000, dtype="bf16"):
    return bsp.geometry(Hq, Hkv, D, ps, npages, dtype)


def test_workspace_size_grows_with_limits(lib):
    d1, h1 = bsp.workspace_size(geo(), 64, 30, 32)
    d2, h2 = bsp.workspace_size(geo(), 128, 96, 128)
    assert 0 < d1 < d2 and 0 < h1 < h2
    with pytest.raises(bsp.BspError, match="UNSUPPORTED"):
        bsp.workspace_size(geo(D=96), 1, 1, 1)


def _err(fn, *a, **k):
    with pytest.raises(bsp.BspError) as e:
        fn(*a, **k)
    return bsp.STATUS_NAMES[e.value.status]


def test_plan_build_validation(lib):
    P, T = [100, 40], [2, 0]
    pages = np.arange(8, dtype=np.int32).reshape(2, 4)
    ok = lambda **kw: bsp.plan_build(kw.pop("g", geo()), kw.pop("B", 2), kw.pop("W", 4), kw.pop("P", P),
                                     kw.pop("T", T), kw.pop("pages", pages), kw.pop("max_tail", 8),
                                     kw.pop("sms", 152))
    ok()
    assert _err(ok, g=geo(dtype="bf16", D=80)) == "BSP_ERR_UNSUPPORTED"
    assert _err(ok, g=geo(Hq=18, Hkv=2)) == "BSP_ERR_UNSUPPORTED"     # group 9 > 8
    assert _err(ok, g=geo(Hq=12, Hkv=8)) == "BSP_ERR_UNSUPPORTED"     # not a multiple
    assert _err(ok, g=geo(ps=24)) == "BSP_ERR_UNSUPPORTED"
    assert _err(ok, g=geo(ps=256)) == "BSP_ERR_UNSUPPORTED"
    assert _err(ok, g=geo(npages=0)) == "BSP_ERR_INVALID_ARG"
    assert _err(ok, T=[9, 0]) == "BSP_ERR_CAPACITY"                  # tail above max_tail
    assert _err(ok, T=[3, 0], max_tail=2) == "BSP_ERR_CAPACITY"
    assert _err(ok, max_tail=9) == "BSP_ERR_UNSUPPORTED"
    assert _err(ok, P=[-1, 4]) == "BSP_ERR_INVALID_ARG"
    assert _err(ok, W=0) == "BSP_ERR_INVALID_ARG"
    assert _err(ok, sms=0) == "BSP_ERR_INVALID_ARG"
    bad = pages.copy()
    bad[1, 1] = 1000                                                  # second prompt page of request 1
    assert _err(ok, P=[100, 40], pages=bad) == "BSP_ERR_PAGE_INDEX"
    bad[1, 1] = -1
    assert _err(ok, pages=bad) == "BSP_ERR_PAGE_INDEX"
    # entries past ceil(P/ps) are never read
    bad = pages.copy()
    bad[1, 2:] = -7
    ok(pages=bad)
    # a page table narrower than the longest prompt
    assert _err(ok, P=[200, 40]) == "BSP_ERR_INVALID_ARG"


def decode_image(plan, img, with_cta=False):
    i32 = img.view(np.int32)
    base = STATUS_OFFSET
    req = i32[(plan.off_req - base) // 4:(plan.off_units - base) // 4].reshape(plan.batch, 12)
    u0 = (plan.off_units - base) // 4
    units = i32[u0:u0 + plan.num_units * 8].reshape(plan.num_units, 8)
    cta_off = i32[(plan.off_cta - base) // 4:(plan.off_pages - base) // 4]
    pages = i32[(plan.off_pages - base) // 4:]
    if with_cta:
        return req, units, pages, cta_off
    return req, units, pages


def row_blocks(W, G):
    """Query-row blocks of a (request, kv head): whole beams, at most 128 rows each, balanced."""
    wmax = max(1, 128 // G)
    nrb = -(-W // wmax)
    return nrb, -(-W // nrb)


def prompt_layout(D, W, G):
    """The prompt kernel of a decode plan: 0 (one softmax set) at head_dim 256 or when a row block fits 16
    rows per TMEM lane quadrant (half-row softmax); 2 (two MMA blocks per CTA) for 129-256 query rows per
    (request, kv head) spread over the quadrants; 1 (alternating-tile sets) when a row block's beams
    spread over the four 32-lane quadrants; else 0."""
    _, wblk = row_blocks(W, G)
    if D > 128 or -(-wblk // 4) * G <= 16:
        return 0
    if 128 < W * G <= 256 and -(-(-(-W // 2)) // 4) * G <= 32:
        return 2
    return 1 if -(-wblk // 4) * G <= 32 else 0


def check_fused(plan, req, T, head_dim=128):
    """A request is finished by the prompt kernel iff it has one prompt partial state and its tail keys
    fit the kernel's tail tiles: a unit's beams' (a row block's, or all W for the two-block kernel) in at
    most 4 tiles of 128 keys (layouts 1 and 2), else in at most 4 prompt-kernel tiles (128 keys up to
    head_dim 128, 64 at 256)."""
    T = np.asarray(T)
    tile = 128 if plan.layout in (1, 2) or head_dim <= 128 else 64
    want = (req[:, 2] == 1) & (-(-T * plan.beams_per_block // tile) <= 4)
    np.testing.assert_array_equal(req[:, 5], want.astype(np.int32))
    assert plan.tail_requests == int((~want).sum())


def check_units_cover(plan, req, units, P, tile=64):
    """Every (request, kv head, row block) covers its prompt tiles exactly once."""
    B, Hkv, nrb = plan.batch, plan.geo.num_kv_heads, plan.row_blocks
    cover = {}
    for b_, g_, rb_, t0, t1, part, _, _ in units:
        assert 0 <= t0 < t1
        key = (b_, g_, rb_)
        cover.setdefault(key, []).append((t0, t1, part))
    for b in range(B):
        ntile = -(-P[b] // tile)
        for g in range(Hkv):
            for rb in range(nrb):
                spans = sorted(cover.get((b, g, rb), []))
                if ntile == 0:
                    assert not spans
                    continue
                assert spans[0][0] == 0 and spans[-1][1] == ntile
                for (a0, a1, _), (c0, c1, _) in zip(spans, spans[1:]):
                    assert a1 == c0
                parts = [s[2] for s in spans]
                assert parts == list(range(req[b][3], req[b][3] + req[b][2]))
    assert len(cover) == sum(1 for b in range(B) if P[b] > 0) * Hkv * nrb


def test_plan_image_wide_batch_needs_no_split(lib):
    rng = np.random.default_rng(3)
    B, W, ps = 64, 30, 32
    P = rng.integers(400, 601, B)
    T = rng.integers(0, 5, B)
    maxp = -(-P.max() // ps)
    pages = rng.integers(0, 5000, (B, maxp)).astype(np.int32)
    plan, img = bsp.plan_build(geo(npages=5000), B, W, P, T, pages, 8, 152)
    req, units, pl, cta_off = decode_image(plan, img, with_cta=True)
    assert plan.row_blocks == 1 and plan.beams_per_block == 30
    assert plan.num_units == B * 8 and plan.num_parts == B
    assert plan.max_tail_len == T.max() and plan.max_total_len == (P + T).max()
    np.testing.assert_array_equal(req[:, 0], P)
    np.testing.assert_array_equal(req[:, 1], T)
    np.testing.assert_array_equal(req[:, 2], 1)
    # rows per request, no causal limit, first row b * W
    np.testing.assert_array_equal(req[:, 8:11], np.stack([np.full(B, W), np.full(B, -1), np.arange(B) * W], 1))
    assert plan.total_rows == B * W and plan.kind == 0
    check_units_cover(plan, req, units, P)
    check_fused(plan, req, T)
    assert plan.tail_requests == 0                          # 30 beams x <= 4 tail keys fit one tile
    assert plan.prefix_ctas == 152 and len(cta_off) == 153
    assert cta_off[0] == 0 and cta_off[-1] == plan.num_units and np.all(np.diff(cta_off) >= 1)
    # dealing cost: eighths of a 128-key tile, for the unit's key tiles, its tail tile and half a tile
    keys = np.minimum(units[:, 4] * 64, P[units[:, 0]]) - units[:, 3] * 64
    want = 8 * (-(-keys // 128) + (T[units[:, 0]] > 0)) + 4
    np.testing.assert_array_equal(units[:, 6], want)
    cost = units[:, 6]
    per_cta = np.array([cost[cta_off[c]:cta_off[c + 1]].sum() for c in range(152)])
    assert per_cta.max() <= per_cta.mean() + cost.max()    # greedy dealing balances the persistent CTAs
    # no worse than dealing each unit, longest first, to the least-loaded CTA
    lpt = np.zeros(152, np.int64)
    for x in sorted(cost.tolist(), reverse=True):
        lpt[np.argmin(lpt)] += x
    assert per_cta.max() <= lpt.max()
    for b in range(B):
        n = -(-P[b] // ps)
        np.testing.assert_array_equal(pl[req[b][4]:req[b][4] + n], pages[b, :n])


def check_groups(plan, units, cta):
    """The row blocks of a (request, kv head, key split) sit on neighbouring CTAs at the same place of
    their lists (CTA c * nrb + rb holds row block rb)."""
    nrb = plan.row_blocks if plan.layout == 1 else 1
    if nrb == 1:
        return
    ctas = len(cta) - 1
    used = [c for c in range(ctas) if cta[c + 1] > cta[c]]
    assert len(used) % nrb == 0 and used == list(range(len(used)))
    for g0 in range(0, len(used), nrb):
        lists = [units[cta[c]:cta[c + 1]] for c in range(g0, g0 + nrb)]
        for rb, l in enumerate(lists):
            assert len(l) == len(lists[0])
            np.testing.assert_array_equal(l[:, 2], rb)
            np.testing.assert_array_equal(np.delete(l, 2, axis=1), np.delete(lists[0], 2, axis=1))


def test_plan_image_wide_beam_one_unit_per_kv_head(lib):
    """192 query rows per (request, kv head) at head_dim 128: one unit holds both 96-row blocks (the
    two-block kernel), so the prompt is read once; up to 4 tiles of 128 tail keys (96 beams x T <= 512)
    finish in the prompt kernel."""
    B, W = 3, 96
    P = [3000, 2900, 0]                       # 16 units on 8 SMs: no key splits
    T = [1, 0, 3]
    pages = np.tile(np.arange(94, dtype=np.int32), (B, 1))
    plan, img = bsp.plan_build(geo(npages=200), B, W, P, T, pages, 8, 8)
    req, units, _ = decode_image(plan, img)
    assert plan.layout == 2 and plan.row_blocks == 1 and plan.beams_per_block == 96
    check_units_cover(plan, req, units, P)
    assert req[2][2] == 0                                            # empty prompt: no split, no unit
    check_fused(plan, req, T)
    assert list(req[:, 5]) == [1, 1, 0] and plan.tail_requests == 1
    # dealing cost: the prompt tiles, ceil(96 T / 128) tail tiles and one tile for the unit's ends
    keys = np.minimum(units[:, 4] * 64, np.asarray(P)[units[:, 0]]) - units[:, 3] * 64
    want = 8 * (-(-keys // 128) + -(-np.asarray(T)[units[:, 0]] * 96 // 128)) + 8
    np.testing.assert_array_equal(units[:, 6], want)
    plan, img = bsp.plan_build(geo(npages=200), B, W, P, [5, 6, 1], pages, 8, 8)
    req, _, _ = decode_image(plan, img)
    check_fused(plan, req, [5, 6, 1])                                # 96 x 6 tail keys exceed 4 tiles
    assert list(req[:, 5]) == [1, 0, 0]
    # head_dim 256 keeps two row blocks on the one-set kernel
    plan, img = bsp.plan_build(geo(D=256, npages=200), B, W, P, T, pages, 8, 152)
    req, units, _ = decode_image(plan, img)
    assert plan.layout == 0 and plan.row_blocks == 2 and plan.beams_per_block == 48
    check_units_cover(plan, req, units, P)
    check_fused(plan, req, T, head_dim=256)


def test_plan_image_row_block_groups_on_neighbouring_ctas(lib):
    """384 query rows per (request, kv head) (96 beams x 4 heads): three 128-row blocks on the
    alternating-tile kernel, dealt to three neighbouring CTAs in the same order; a block's tail keys
    (32 beams x T) finish in the prompt kernel up to 4 tiles of 128 keys."""
    B, W = 3, 96
    P = [3000, 2900, 0]                       # 48 units on 24 SMs: no key splits
    T = [1, 0, 3]
    pages = np.tile(np.arange(94, dtype=np.int32), (B, 1))
    g4 = geo(Hq=32, Hkv=8, npages=200)
    plan, img = bsp.plan_build(g4, B, W, P, T, pages, 8, 24)
    req, units, _, cta = decode_image(plan, img, with_cta=True)
    assert plan.layout == 1 and plan.row_blocks == 3 and plan.beams_per_block == 32
    check_units_cover(plan, req, units, P)
    check_groups(plan, units, cta)
    check_fused(plan, req, T)
    assert list(req[:, 5]) == [1, 1, 0] and plan.tail_requests == 1
    keys = np.minimum(units[:, 4] * 64, np.asarray(P)[units[:, 0]]) - units[:, 3] * 64
    want = 8 * (-(-keys // 128) + -(-np.asarray(T)[units[:, 0]] * 32 // 128)) + 4
    np.testing.assert_array_equal(units[:, 6], want)
    # the tail kernel finishes a block's tail beyond 4 tiles (128 beams x 5 keys, one row per beam)
    g1 = geo(Hq=8, Hkv=8, npages=200)
    plan, img = bsp.plan_build(g1, B, 128, P, [5, 4, 1], pages, 8, 8)
    req, _, _ = decode_image(plan, img)
    assert plan.layout == 1 and plan.beams_per_block == 128
    check_fused(plan, req, [5, 4, 1])
    assert list(req[:, 5]) == [0, 1, 0]


def test_plan_image_single_long_request_is_split(lib):
    """One request with 8 kv heads is split along its keys to fill the GPU."""
    P = [10000]
    pages = np.arange(324, dtype=np.int32)[None]
    plan, img = bsp.plan_build(geo(Hq=32, Hkv=8, npages=324, dtype="fp16"), 1, 1, P, [1], pages, 8, 152)
    req, units, _ = decode_image(plan, img)
    assert plan.num_parts == req[0][2] > 8
    assert plan.num_parts <= 1 + 64
    assert plan.num_units == plan.num_parts * 8
    check_units_cover(plan, req, units, P)
    lens = units[:, 4] - units[:, 3]
    assert lens.max() - lens.min() <= 1
    check_fused(plan, req, [1])
    assert plan.tail_requests == 1                                   # split prompt: merged by the tail kernel


def test_plan_image_empty_batch_and_empty_prompts(lib):
    plan, img = bsp.plan_build(geo(), 0, 4, [], [], np.zeros((0, 1), np.int32), 8, 152)
    assert plan.num_units == 0 and plan.batch == 0
    plan, img = bsp.plan_build(geo(), 2, 4, [0, 0], [1, 3], np.zeros((2, 1), np.int32), 8, 152)
    assert plan.num_units == 0 and plan.num_parts == 0 and plan.max_tail_len == 3
    assert plan.tail_requests == 2


def test_plan_struct_layout_matches_header(lib):
    """The ctypes mirror has the field order and sizes of bsp_plan_t."""
    text = open(os.path.join(ROOT, "include", "bsp.h")).read()
    body = text[text.index("typedef struct bsp_plan_t"):text.index("} bsp_plan_t;")]
    fields = re.findall(r"^\s+(?:int32_t|uint64_t|void\*|bsp_geometry)\s+(\w+)", body, flags=re.M)
    names = [f[0] for f in bsp.Plan._fields_]
    assert fields == names
    assert ctypes.sizeof(bsp.Plan) % 8 == 0


def test_geometry_struct_layout_matches_header(lib):
    text = open(os.path.join(ROOT, "include", "bsp.h")).read()
    body = text[text.index("typedef struct bsp_geometry"):text.index("} bsp_geometry;")]
    fields = re.findall(r"^\s+int32_t\s+(\w+);", body, flags=re.M)
    assert fields == [f[0] for f in bsp.Geometry._fields_]


def test_e4m3_pool_plans(lib):
    """Plans over E4M3 pools use the kernels that widen E4M3 tiles: the wide kernel for 129-256 query rows
    per (request, kv head), else alternating-tile row blocks of at most 4 * floor(32 / G) beams; head_dim
    256, prefill and an unknown pool type are unsupported."""
    def plan8(Hq, Hkv, W, D=128, B=3, T=2):
        g = bsp.geometry(Hq, Hkv, D, 32, 5000, "bf16", kv_dtype=bsp.KV_DTYPE_E4M3)
        P = [700, 90, 1]
        pages = np.arange(B * 32, dtype=np.int32).reshape(B, 32)
        return bsp.plan_build(g, B, W, P[:B], [T] * B, pages[:B], 8, 152)
    for Hq, Hkv, W, layout, rb, wblk in [(16, 8, 30, 1, 1, 30), (16, 8, 96, 2, 1, 96), (24, 8, 42, 1, 2, 21),
                                         (24, 8, 50, 2, 1, 50), (64, 8, 12, 1, 1, 12), (64, 8, 20, 2, 1, 20),
                                         (8, 8, 128, 1, 1, 128), (64, 8, 40, 1, 3, 14)]:
        plan, img = plan8(Hq, Hkv, W)
        G = Hq // Hkv
        # the workspace sized for this shape holds the plan
        dev_bytes, host_bytes = bsp.workspace_size(
            bsp.geometry(Hq, Hkv, 128, 32, 5000, "bf16", kv_dtype=bsp.KV_DTYPE_E4M3), 3, W, 32)
        assert plan.device_bytes_used <= dev_bytes and 256 + 2 * plan.image_bytes <= host_bytes
        assert (plan.layout, plan.row_blocks, plan.beams_per_block) == (layout, rb, wblk), (Hq, Hkv, W)
        if layout == 1:
            assert -(-wblk // 4) * G <= 32 and wblk * G <= 128
        req, units, _ = decode_image(plan, img)
        check_fused(plan, req, np.array([2, 2, 2]))
        # the 16-bit plan of the same shape may pick another kernel, with the same request records' lengths
        p16, img16 = bsp.plan_build(geo(Hq=Hq, Hkv=Hkv), 3, W, [700, 90, 1], [2, 2, 2],
                                    np.arange(96, dtype=np.int32).reshape(3, 32), 8, 152)
        np.testing.assert_array_equal(decode_image(p16, img16)[0][:, :2], req[:, :2])
    with pytest.raises(bsp.BspError) as e:
        plan8(16, 8, 30, D=256)
    assert bsp.STATUS_NAMES[e.value.status] == "BSP_ERR_UNSUPPORTED"
    g = bsp.geometry(16, 8, 128, 32, 5000, "bf16", kv_dtype=2)
    assert _err(bsp.plan_build, g, 1, 4, [10], [1], np.zeros((1, 1), np.int32), 8, 152) == "BSP_ERR_UNSUPPORTED"
    g = bsp.geometry(16, 8, 128, 32, 5000, "bf16", kv_dtype=bsp.KV_DTYPE_E4M3)
    assert _err(bsp.plan_prefill_build, g, 1, [0], [20], np.zeros((1, 1), np.int32), True, 152) == \
        "BSP_ERR_UNSUPPORTED"


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("Hq,D", [(32, 128), (24, 64), (32, 256), (24, 256)])
def test_prefill_plan_units_and_records(lib, causal, Hq, D):
    """A prefill plan: the prompt tokens are the rows, keys are the cached rows and the prompt, no tail
    and no key splits; a causal unit reads keys only up to its last token (rounded up to a 64-key plan
    tile). At head_dim <= 128 a unit is a pair of row blocks of 4 * floor(32 / G) tokens on the two-block
    kernel (layout 2), at head_dim 256 one block of floor(128 / G) tokens on the one-set kernel."""
    C = np.array([0, 300, 5, 40])
    S = np.array([1000, 7, 0, 200])
    ps = 32
    maxp = -(-(C + S).max() // ps)
    rng = np.random.default_rng(4)
    pages = rng.integers(0, 400, (4, maxp)).astype(np.int32)
    G = Hq // 8
    g = geo(Hq=Hq, Hkv=8, D=D, npages=400)
    plan, img = bsp.plan_prefill_build(g, 4, C, S, pages, causal, 152)
    req, units, pl = decode_image(plan, img)
    wblk = 4 * (32 // G) if D <= 128 else 128 // G
    urows = 2 * wblk if D <= 128 else wblk
    assert plan.kind == 1 and plan.total_rows == S.sum() and plan.tail_requests == 0
    assert plan.beams_per_block == wblk and plan.max_tail_len == 0
    assert plan.layout == (2 if D <= 128 else 0)
    np.testing.assert_array_equal(req[:, 0], np.where(S > 0, C + S, 0))
    np.testing.assert_array_equal(req[:, 1], 0)
    np.testing.assert_array_equal(req[:, 8], S)
    np.testing.assert_array_equal(req[:, 9], C if causal else -1)
    np.testing.assert_array_equal(req[:, 10], np.concatenate([[0], np.cumsum(S)[:-1]]))
    np.testing.assert_array_equal(req[:, 5], (S > 0).astype(np.int32))
    np.testing.assert_array_equal(req[:, 2], (S > 0).astype(np.int32))
    want = set()
    for b in range(4):
        for gg in range(8):
            for rb in range(-(-S[b] // urows)):
                last = min(S[b], (rb + 1) * urows)
                end = -(-(C[b] + last) // 64) if causal else -(-(C[b] + S[b]) // 64)
                want.add((b, gg, rb, 0, end))
    got = set(tuple(int(x) for x in u[:5]) for u in units)
    assert got == want
    for b in range(4):
        n = -(-(C[b] + S[b]) // ps) if S[b] else 0
        np.testing.assert_array_equal(pl[req[b][4]:req[b][4] + n], pages[b, :n])


def test_plan_requests_reads_whole_records(lib):
    """bsp.plan_requests returns the 12-field request records in order (the fused flag of a mixed
    batch at head_dim 256: request 1 has more tail keys per row block than four 64-key tiles hold)."""
    g = geo(Hq=8, Hkv=8, D=256, ps=16, npages=4000, dtype="fp16")
    B, W = 3, 64
    P = np.array([300, 500, 700], np.int32)
    T = np.array([2, 8, 0], np.int32)
    pages = np.arange(B * 64, dtype=np.int32).reshape(B, 64)
    plan, img = bsp.plan_build(g, B, W, P, T, pages, 8, 8)    # 24 units fill 8 SMs: no key splits
    req = bsp.plan_requests(plan, img)
    assert req.shape == (B, 12)
    np.testing.assert_array_equal(req[:, 2], 1)
    np.testing.assert_array_equal(req[:, 0], P)
    np.testing.assert_array_equal(req[:, 1], T)
    np.testing.assert_array_equal(req[:, 5], [1, 0, 1])       # 64 x 2 = 128 <= 4 x 64 < 64 x 8 = 512
    np.testing.assert_array_equal(req[:, 10], np.arange(B) * W)


def test_decode_plan_layout_is_fixed_by_its_shape(lib):
    """Graph mode relies on it: decode plans of one shape (batch, beam width, SM count, page-table
    stride) put every image section at the same offsets whatever the lengths, and the CTA table has
    num_sms + 1 non-decreasing entries ending at the unit count."""
    g = geo(Hq=32, Hkv=8, D=128, ps=16, npages=20000, dtype="fp16")
    B, W, sms, stride = 6, 30, 152, 200
    rng = np.random.default_rng(3)
    pages = rng.integers(0, 20000, (B, stride)).astype(np.int32)
    seen = set()
    for trial in range(8):
        P = rng.integers(0, stride * 16 + 1, B).astype(np.int32)
        if trial == 1:
            P[:] = 0
        T = rng.integers(0, 9, B).astype(np.int32)
        plan, img = bsp.plan_build(g, B, W, P, T, pages, 8, sms)
        seen.add((plan.off_req, plan.off_units, plan.off_cta, plan.off_pages, plan.off_part_lse, plan.off_part_o,
                  plan.image_bytes))
        req, units, pg, cta = decode_image(plan, img, with_cta=True)
        assert len(cta) == sms + 1 and cta[0] == 0 and cta[-1] == plan.num_units
        assert (np.diff(cta) >= 0).all()
    assert len(seen) == 1, seen
    # a prefill plan is packed: its sections follow the unit count
    pf1, _ = bsp.plan_prefill_build(g, 2, [0, 0], [10, 300], pages[:2], True, sms)
    pf2, _ = bsp.plan_prefill_build(g, 2, [0, 0], [600, 900], pages[:2], True, sms)
    assert pf1.off_cta != pf2.off_cta


def test_write_side_entry_points_reject_bad_arguments_without_a_launch(lib):
    """Host checks of the RoPE table, the RoPE append, the E4M3 append and the graph flag, before any
    launch (no GPU needed: every call below fails on its arguments or on a plan that was never staged)."""
    import ctypes
    c = ctypes
    name = lambda rc: bsp.STATUS_NAMES.get(rc, rc)
    buf = np.zeros(1024, np.float32)
    # bsp_rope_cos_sin: positions, rotary dim, base, and a host pointer
    for args in ((0, 64, 1e4), (16, 63, 1e4), (16, 0, 1e4), (16, 64, 1.0), (16, 64, float("inf")), (16, 64, 1e4)):
        rc = lib.bsp_rope_cos_sin(args[0], args[1], c.c_double(args[2]), buf.ctypes.data_as(c.c_void_p), None)
        assert name(rc) == "BSP_ERR_INVALID_ARG", args
    # an unstaged plan (built on the host only) is refused by every launch entry point
    g = geo()
    plan, _ = bsp.plan_build(g, 1, 4, [64], [1], np.zeros((1, 4), np.int32), 8, 152)
    rope = bsp.RopeConfig(None, 16, 64, 0, 0)
    rc = lib.bsp_rope_append_kv(c.byref(plan), c.byref(rope), None, None, 0, None, None, 1024, None, 1, None, None,
                                None, None)
    assert name(rc) != "BSP_OK"
    rc = lib.bsp_append_kv_fp8(c.byref(plan), None, None, 1024, 0, c.c_float(1.0), c.c_float(1.0), None, 1, None, None,
                               None, None)
    assert name(rc) != "BSP_OK"
    rc = lib.bsp_rope_append_kv_fp8(c.byref(plan), c.byref(rope), None, None, 0, None, None, 1024, c.c_float(1.0),
                                    c.c_float(1.0), None, 1, None, None, None, None)
    assert name(rc) != "BSP_OK"
    rc = lib.bsp_decode_attn(c.byref(plan), None, None, None, None, 0, None, 0, c.c_float(0.1), bsp.FLAG_GRAPH, None,
                             None, None, None)
    assert name(rc) != "BSP_OK"


def test_planner_random_sweep(lib):
    """Random shapes and lengths: every plan covers each (request, kv head, row block)'s prompt tiles once,
    its CTA table is a monotone partition of the units over at most num_sms CTAs, the fused flags follow
    the rule, each CTA's units are longest first, and no CTA's dealt cost exceeds the LPT bound of the
    same units (the dealing only improves on LPT)."""
    rng = np.random.default_rng(2024)
    for trial in range(120):
        D = int(rng.choice([64, 128, 256]))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 4, 8]))
        ps = int(rng.choice([8, 16, 32, 64]))
        B = int(rng.integers(1, 40))
        W = int(rng.integers(1, 100))
        sms = int(rng.choice([8, 37, 148, 152]))
        P = rng.integers(0, 3000, B)
        P[rng.random(B) < 0.2] = 0
        T = rng.integers(0, 9, B)
        maxp = max(1, int(-(-P.max() // ps)))
        pages = rng.integers(0, 100000, (B, maxp)).astype(np.int32)
        g = bsp.geometry(G * Hkv, Hkv, D, ps, 100000, "bf16")
        plan, img = bsp.plan_build(g, B, W, P, T, pages, 8, sms)
        req, units, pl, cta = decode_image(plan, img, with_cta=True)
        assert plan.layout == prompt_layout(D, W, G)
        check_units_cover(plan, req, units, P)
        check_groups(plan, units, cta)
        check_fused(plan, req, T, head_dim=D)
        assert len(cta) == sms + 1 and cta[0] == 0 and cta[-1] == plan.num_units and (np.diff(cta) >= 0).all()
        assert plan.prefix_ctas <= sms
        cost = units[:, 6].astype(np.int64)
        loads = [int(cost[cta[c]:cta[c + 1]].sum()) for c in range(sms)]
        for c in range(sms):
            seg = cost[cta[c]:cta[c + 1]]
            assert (np.diff(seg) <= 0).all()                   # longest first within a CTA
        # LPT on the same costs (longest first, each to the least-loaded CTA) bounds the largest load; the
        # row blocks of a group are dealt together, to the CTA groups
        grp = plan.row_blocks if plan.layout == 1 else 1
        gcost = units[units[:, 2] == 0][:, 6].astype(np.int64) if grp > 1 else cost
        heap = [0] * min(len(gcost), sms // grp)
        for x in sorted(gcost, reverse=True):
            i = int(np.argmin(heap))
            heap[i] += int(x)
        if len(cost):
            assert max(loads) <= max(heap), (trial, max(loads), max(heap))


def check_prefill_units(plan, req, units, B, Hkv, C, S, causal, urows, trial=None):
    """A prefill plan's units: for every (request, kv head, run of urows tokens) their key ranges tile
    [0, end) in 64-key plan tiles (end: the run's last visible key, or the prompt's end); a request's
    ranges are the same for all its units but the last one's end, every cut lies inside the cached
    rows (so each row has keys in each range), range s writes partial slot part_off + s, and a request
    with more than one range is the tail kernel's (not fused)."""
    by = {}
    for u in units:
        b, g, rb, t0, t1, part = (int(x) for x in u[:6])
        by.setdefault((b, g, rb), []).append((t0, t1, part))
    want_keys = set()
    tail = 0
    for b in range(B):
        nsplit, part_off, fused = int(req[b][2]), int(req[b][3]), int(req[b][5])
        if S[b] == 0:
            assert nsplit == 0
            continue
        assert nsplit >= 1 and fused == (nsplit == 1), (trial, b)
        tail += nsplit > 1
        cuts = None
        for g in range(Hkv):
            for rb in range(-(-int(S[b]) // urows)):
                want_keys.add((b, g, rb))
                last = min(int(S[b]), (rb + 1) * urows)
                end = -(-(int(C[b]) + last) // 64) if causal else -(-(int(C[b]) + int(S[b])) // 64)
                r = sorted(by.get((b, g, rb), []))
                assert len(r) == nsplit and r[0][0] == 0 and r[-1][1] == end, (trial, b, g, rb, r, end)
                assert all(r[i][1] == r[i + 1][0] for i in range(nsplit - 1)), (trial, r)
                assert [x[2] for x in r] == list(range(part_off, part_off + nsplit)), (trial, r)
                c = [x[0] for x in r[1:]]
                assert cuts is None or c == cuts
                cuts = c
                assert all(x * 64 <= C[b] for x in c), (trial, b, c, C[b])
    assert set(by) == want_keys, trial
    assert plan.tail_requests == tail and plan.num_parts <= B + 64


@pytest.mark.parametrize("causal", [True, False])
def test_prefill_key_splits_of_a_long_cache(lib, causal):
    """One request with a long cached prefix among short ones: its cached keys are cut into ranges (cuts
    inside the cached rows), the others stay whole; without long caches nothing is split."""
    C = np.array([20000, 500, 300, 800, 100, 600, 700, 200])
    S = np.array([100, 200, 150, 250, 90, 300, 120, 60])
    ps = 32
    maxp = -(-(C + S).max() // ps)
    pages = np.arange(8 * maxp, dtype=np.int32).reshape(8, maxp) % 4000
    g = geo(Hq=32, Hkv=8, npages=4000)
    plan, img = bsp.plan_prefill_build(g, 8, C, S, pages, causal, 152)
    req, units, _ = decode_image(plan, img)
    assert plan.tail_requests == 1 and req[0][2] > 1 and (req[1:, 2] == 1).all()
    assert plan.beam_width == S.max() and plan.num_parts == 8 + req[0][2] - 1
    check_prefill_units(plan, req, units, 8, 8, C, S, causal, 64)
    # the same batch with short caches: whole requests, no partial slots
    plan2, img2 = bsp.plan_prefill_build(g, 8, np.minimum(C, 800), S, pages, causal, 152)
    req2, units2, _ = decode_image(plan2, img2)
    assert plan2.tail_requests == 0 and (req2[:, 2] == 1).all() and plan2.beam_width == 1
    check_prefill_units(plan2, req2, units2, 8, 8, np.minimum(C, 800), S, causal, 64)


def test_prefill_planner_random_sweep(lib):
    """Random prefill batches: one unit per (request, kv head, run of prompt tokens: two blocks of
    4 * floor(32 / G) at head_dim <= 128, one block of floor(128 / G) at head_dim 256) reading plan tiles
    [0, end) with end the unit's last visible key (causal) or the prompt's end, the request records'
    rows / row offsets / causal bases, and a CTA table partitioning the units."""
    rng = np.random.default_rng(77)
    for trial in range(60):
        Hkv = int(rng.choice([1, 2, 8]))
        G = int(rng.choice([1, 2, 4, 8]))
        ps = int(rng.choice([16, 32, 64]))
        B = int(rng.integers(1, 12))
        causal = bool(rng.integers(0, 2))
        C = rng.integers(0, 2000, B)
        S = rng.integers(0, 700, B)
        S[rng.random(B) < 0.2] = 0
        maxp = max(1, int(-(-(C + S).max() // ps)))
        pages = rng.integers(0, 50000, (B, maxp)).astype(np.int32)
        D = int(rng.choice([64, 128, 256]))
        g = bsp.geometry(G * Hkv, Hkv, D, ps, 50000, "bf16")
        sms = int(rng.choice([16, 152]))
        plan, img = bsp.plan_prefill_build(g, B, C, S, pages, causal, sms)
        req, units, pl, cta = decode_image(plan, img, with_cta=True)
        wblk = 4 * (32 // G) if D <= 128 else 128 // G
        urows = 2 * wblk if D <= 128 else wblk
        assert plan.kind == 1 and plan.total_rows == S.sum() and plan.beams_per_block == wblk
        assert plan.layout == (2 if D <= 128 else 0)
        np.testing.assert_array_equal(req[:, 8], S)
        np.testing.assert_array_equal(req[:, 9], C if causal else -1)
        np.testing.assert_array_equal(req[:, 10], np.concatenate([[0], np.cumsum(S)[:-1]]))
        check_prefill_units(plan, req, units, B, Hkv, C, S, causal, urows, trial)
        assert cta[0] == 0 and cta[-1] == plan.num_units and (np.diff(cta) >= 0).all()
        # a workspace sized for the batch with the longest prompt as beam width holds the plan, key
        # splits' partial states included
        dev_bytes, host_bytes = bsp.workspace_size(g, B, max(1, int(S.max())), maxp)
        assert plan.device_bytes_used <= dev_bytes and 256 + 2 * plan.image_bytes <= host_bytes, trial
