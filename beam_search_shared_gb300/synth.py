"""Seeded synthetic paged KV caches shaped like the beam-search decode workloads.

This module only builds inputs: lengths, page tables, cache_indirection, the
paged pools and the new token's rows. It holds none of the attention
arithmetic. Both the CUDA path's tests/benchmark and the fp64 oracle are fed
from it, with identical bits.

Recipe (per workload, ``seed`` drives a CPU ``torch.Generator`` for every
structural draw and a generator on ``device`` for the bulk values):

* prompt length P_b and tail length T_b per request, uniform in the workload's
  ranges (T_b counts generated positions whose K/V is in the cache, the current
  token included);
* pages: each request's full prompt pages are shared by all beams; the page
  holding the prompt's partial last rows and every page of the tail are private
  to each beam (the prompt rows of that page are copied to every beam); the
  physical page ids are a random permutation of the pool, with ~5% spare pages
  that nothing references (identity pages for the single-allocation workload);
* prefix_pages[b] is beam 0's prompt page list; beam_pages[r] is beam r's full
  list; unused entries are -1;
* cache_indirection[b][w][pos] is a uniform source beam for every position
  (prefix positions are never read); with ``full_step`` the current position
  P+T-1 points at the beam itself, since the append writes it there;
* values: valid rows ~ N(0, 1), rows beyond every valid length are garbage,
  uniform in [-1000, 1000] (or NaN with ``poison``), all rounded to the dtype;
* with ``full_step``, each row with T_b >= 1 gets a new K/V row (N(0, 1)) and the
  flat slot (page * page_size + offset) of its current position.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape recipe of one synthetic decode step."""
    name: str
    batch: int
    beam_width: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: str
    prompt: Sequence[int]          # (lo, hi) inclusive uniform range
    tail: Sequence[int]            # (lo, hi) inclusive uniform range
    identity_rows: int = 0         # >0: one contiguous allocation of this many rows
    force_tail_patterns: bool = False  # >=1 request with T=0 and >=1 tail crossing a page

    def scaled(self, batch: int) -> "Workload":
        return dataclasses.replace(self, batch=batch, name=f"{self.name}@B{batch}")

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The workloads: a tiny case, a Qwen3-0.6B-shaped layer, a wide-beam recommendation
# shape, a 4B-shaped fp16 layer (head_dim 128 / 64 / 256) and bucketed cached-prefix
# decode over one 10368-row allocation.
WORKLOADS = {
    "tiny_b1_w4_d64": Workload("tiny_b1_w4_d64", 1, 4, 4, 2, 64, 32, "bf16", (128, 128), (3, 3)),
    "qwen3_0p6b_b64_w30": Workload("qwen3_0p6b_b64_w30", 64, 30, 16, 8, 128, 32, "bf16",
                                   (400, 600), (0, 4)),
    "wide_beam_b128_w96": Workload("wide_beam_b128_w96", 128, 96, 16, 8, 128, 32, "bf16",
                                   (2800, 3200), (0, 3)),
    "qwen3_4b_fp16_d128": Workload("qwen3_4b_fp16_d128", 64, 30, 32, 8, 128, 16, "fp16",
                                   (1600, 2400), (0, 8), force_tail_patterns=True),
    "qwen3_4b_fp16_d64": Workload("qwen3_4b_fp16_d64", 64, 30, 32, 8, 64, 16, "fp16",
                                  (1600, 2400), (0, 8), force_tail_patterns=True),
    "qwen3_4b_fp16_d256": Workload("qwen3_4b_fp16_d256", 64, 30, 32, 8, 256, 16, "fp16",
                                   (1600, 2400), (0, 8), force_tail_patterns=True),
}
for _p in (0, 5, 40, 2047, 10000):
    WORKLOADS[f"bucketed_prefix_p{_p}"] = Workload(
        f"bucketed_prefix_p{_p}", 1, 1, 32, 8, 128, 32, "fp16", (_p, _p), (1, 1), identity_rows=10368)


@dataclasses.dataclass
class Case:
    """One synthetic decode step. Index arrays are numpy int32; values are torch tensors."""
    workload: Workload
    seed: int
    full_step: bool
    num_pages: int
    prefix_len: np.ndarray        # [B]
    tail_len: np.ndarray          # [B]
    prefix_pages: np.ndarray      # [B, maxp_prefix], beam 0's prompt pages, -1 padded
    beam_pages: np.ndarray        # [B*W, maxp], -1 padded
    cache_indirection: np.ndarray  # [B, W, max_seq]
    q: torch.Tensor               # [B*W, Hq, D]
    k_pool: torch.Tensor          # [num_pages, Hkv, ps, D] (before the append)
    v_pool: torch.Tensor
    k_new: torch.Tensor           # [n, Hkv, D]
    v_new: torch.Tensor
    out_cache_loc: np.ndarray     # [n]
    new_rows: np.ndarray          # [n] row r of each new token

    @property
    def rows(self) -> int:
        return self.workload.batch * self.workload.beam_width

    @property
    def max_seq(self) -> int:
        return int(self.cache_indirection.shape[2])


def e4m3_codes(shape, generator: torch.Generator, exp_mean: float = 7.0, exp_sd: float = 1.5,
               zero_frac: float = 0.02, device="cpu") -> torch.Tensor:
    """Random E4M3 codes (uint8) for synthetic 8-bit pools, drawn as bit patterns: a random sign and
    3-bit fraction, the 4-bit exponent field drawn around exp_mean (bias 7: magnitudes near 1) and
    clipped to [0, 15] (0: the subnormal codes), a fraction zero_frac of +-0 codes, and the two NaN
    codes (exponent 15, fraction 7) replaced by the largest finite ones. Drawn in chunks of 2^24 codes
    (the same codes for the same generator state) on `device`, the generator's device."""
    out = torch.empty(int(np.prod(shape)), dtype=torch.uint8, device=device)
    chunk = 1 << 24
    for lo in range(0, out.numel(), chunk):
        n = min(chunk, out.numel() - lo)
        sign = torch.randint(0, 2, (n,), generator=generator, dtype=torch.int32, device=device)
        frac = torch.randint(0, 8, (n,), generator=generator, dtype=torch.int32, device=device)
        expo = torch.round(torch.randn((n,), generator=generator, device=device) * exp_sd + exp_mean)
        expo = expo.clamp(0, 15).to(torch.int32)
        frac = torch.where((expo == 15) & (frac == 7), torch.full_like(frac, 6), frac)
        code = (sign << 7) | (expo << 3) | frac
        zero = torch.rand((n,), generator=generator, device=device) < zero_frac
        out[lo:lo + n] = torch.where(zero, sign << 7, code).to(torch.uint8)
    return out.reshape(tuple(shape))


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a 16-bit float tensor, on the host."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def make_case(wl: Workload, seed: int, *, full_step: bool = True, device="cpu",
              poison: bool = False, prompt_lengths: Optional[Sequence[int]] = None,
              tail_lengths: Optional[Sequence[int]] = None, spare_fraction: float = 0.05) -> Case:
    B, W, Hq, Hkv, D, ps = (wl.batch, wl.beam_width, wl.num_q_heads, wl.num_kv_heads,
                            wl.head_dim, wl.page_size)
    R = B * W
    tdt = TORCH_DTYPES[wl.dtype]
    g = torch.Generator().manual_seed(seed)

    # ---- lengths
    if prompt_lengths is not None:
        P = np.asarray(prompt_lengths, np.int64)
    else:
        P = torch.randint(wl.prompt[0], wl.prompt[1] + 1, (B,), generator=g).numpy().astype(np.int64)
    if tail_lengths is not None:
        T = np.asarray(tail_lengths, np.int64)
    else:
        T = torch.randint(wl.tail[0], wl.tail[1] + 1, (B,), generator=g).numpy().astype(np.int64)
    if wl.force_tail_patterns and B >= 2 and prompt_lengths is None and tail_lengths is None:
        T[0] = 0
        P[1] = max(ps, P[1] - P[1] % ps + ps - 3)   # P % ps = ps-3 >= 9 for ps = 16
        T[1] = wl.tail[1]                            # the tail crosses a page boundary
    assert P.shape == (B,) and T.shape == (B,)

    # ---- pages
    if wl.identity_rows:
        assert B == 1 and W == 1 and wl.identity_rows % ps == 0
        num_pages = wl.identity_rows // ps
        assert P[0] + T[0] <= wl.identity_rows
        maxp = num_pages
        beam_pages = np.arange(num_pages, dtype=np.int32)[None, :].copy()
        nfull = P // ps
        row_valid = np.zeros((num_pages, ps), bool)
        flat = np.arange(num_pages * ps).reshape(num_pages, ps)
        row_valid[flat < P[0] + T[0]] = True
        priv_first = np.full((B, W), -1, np.int64)
    else:
        nfull = P // ps
        npriv = np.array([_ceil_div(int(P[b] + T[b]), ps) - int(nfull[b]) for b in range(B)], np.int64)
        needed = int(np.sum(nfull + W * npriv))
        spare = max(2, int(math.ceil(needed * spare_fraction)))
        num_pages = needed + spare
        perm = torch.randperm(num_pages, generator=g).numpy().astype(np.int64)
        maxp = max(1, int(np.max(nfull + npriv)) if B else 1)
        beam_pages = np.full((R, maxp), -1, np.int64)
        row_valid = np.zeros((num_pages, ps), bool)
        priv_first = np.full((B, W), -1, np.int64)
        cur = 0
        for b in range(B):
            shared = perm[cur:cur + nfull[b]]
            cur += int(nfull[b])
            row_valid[shared] = True
            for w in range(W):
                r = b * W + w
                beam_pages[r, :nfull[b]] = shared
                priv = perm[cur:cur + npriv[b]]
                cur += int(npriv[b])
                beam_pages[r, nfull[b]:nfull[b] + npriv[b]] = priv
                if npriv[b]:
                    priv_first[b, w] = priv[0]
                for k, pg in enumerate(priv):
                    first_pos = (int(nfull[b]) + k) * ps
                    nvalid = min(ps, int(P[b] + T[b]) - first_pos)
                    row_valid[pg, :max(0, nvalid)] = True
        assert cur == needed
    maxp_prefix = max(1, max((_ceil_div(int(P[b]), ps) for b in range(B)), default=1))
    prefix_pages = np.full((B, maxp_prefix), -1, np.int64)
    for b in range(B):
        n = _ceil_div(int(P[b]), ps)
        prefix_pages[b, :n] = beam_pages[b * W, :n]

    # ---- cache_indirection
    max_seq = max(1, int(np.max(P + T)) if B else 1)
    ci = torch.randint(0, W, (B, W, max_seq), generator=g).numpy().astype(np.int64)
    pos = np.arange(max_seq)[None, None, :]
    ci = np.where(pos < (P + T)[:, None, None], ci, -1)
    if full_step:
        for b in range(B):
            if T[b] >= 1:
                ci[b, :, P[b] + T[b] - 1] = np.arange(W)

    # ---- values
    dev = torch.device(device)
    gd = torch.Generator(device=dev).manual_seed(seed + 7919)
    k_pool = torch.empty((num_pages, Hkv, ps, D), dtype=tdt, device=dev)
    v_pool = torch.empty_like(k_pool)
    valid_t = torch.from_numpy(row_valid).to(dev)
    chunk = max(1, (1 << 26) // max(1, Hkv * ps * D))   # bounded temporaries
    for pool in (k_pool, v_pool):
        for p0 in range(0, num_pages, chunk):
            p1 = min(num_pages, p0 + chunk)
            shape = (p1 - p0, Hkv, ps, D)
            # drawn even when poisoned, so valid rows get the same values either way
            garbage = torch.rand(shape, generator=gd, device=dev) * 2000.0 - 1000.0
            if poison:
                garbage.fill_(float("nan"))
            normal = torch.randn(shape, generator=gd, device=dev)
            m = valid_t[p0:p1][:, None, :, None]
            pool[p0:p1] = torch.where(m, normal, garbage).to(tdt)
    # the partial prompt page's rows are the same for every beam of a request
    if not wl.identity_rows:
        for b in range(B):
            m = int(P[b] % ps)
            if m and W > 1:
                src = int(priv_first[b, 0])
                dst = torch.from_numpy(priv_first[b, 1:].copy()).to(dev)
                for pool in (k_pool, v_pool):
                    pool[dst, :, :m] = pool[src, :, :m].unsqueeze(0)
    q = torch.randn((R, Hq, D), generator=gd, device=dev).to(tdt)

    # ---- the new token of each row (full step only)
    new_rows, loc = [], []
    if full_step:
        for b in range(B):
            if T[b] < 1:
                continue
            cur_pos = int(P[b] + T[b] - 1)
            for w in range(W):
                r = b * W + w
                new_rows.append(r)
                loc.append(int(beam_pages[r, cur_pos // ps]) * ps + cur_pos % ps)
    n = len(new_rows)
    k_new = torch.randn((n, Hkv, D), generator=gd, device=dev).to(tdt)
    v_new = torch.randn((n, Hkv, D), generator=gd, device=dev).to(tdt)

    return Case(workload=wl, seed=seed, full_step=full_step, num_pages=num_pages,
                prefix_len=P.astype(np.int32), tail_len=T.astype(np.int32),
                prefix_pages=prefix_pages.astype(np.int32), beam_pages=beam_pages.astype(np.int32),
                cache_indirection=ci.astype(np.int32), q=q, k_pool=k_pool, v_pool=v_pool,
                k_new=k_new, v_new=v_new, out_cache_loc=np.asarray(loc, np.int32),
                new_rows=np.asarray(new_rows, np.int32))


def token_positions(case) -> np.ndarray:
    """Logical position of each new token of a full decode step (the model's position ids): the
    current token of every beam of request b sits at P_b + T_b - 1."""
    W = case.workload.beam_width
    b = case.new_rows // W
    return (case.prefix_len[b] + case.tail_len[b] - 1).astype(np.int32)


# ---------------------------------------------------------------- prefill over the cached prefix
@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    """Shape recipe of one synthetic prefill: per request, C cached rows and S prompt tokens."""
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    dtype: str
    cached: Sequence[int]   # (lo, hi) inclusive uniform range of valid cached rows C
    prompt: Sequence[int]   # (lo, hi) inclusive uniform range of prompt tokens S
    causal: bool = True
    alloc_rows: int = 0     # > 0: every request owns this many rows of pages (garbage past C + S)

    def with_(self, **kw) -> "PrefillWorkload":
        return dataclasses.replace(self, **kw)


# The phi4-multimodal shapes of the bucketed-prefix page: a 10368-row allocation per request, an image
# prompt prefilled with nothing cached, or text after a cached prefix; the 4B-shaped heads of the decode
# workloads (32 q heads, 8 kv heads, head_dim 128, fp16).
PREFILL_WORKLOADS = {
    "prefill_tiny_d64": PrefillWorkload("prefill_tiny_d64", 2, 4, 2, 64, 16, "bf16", (0, 40), (1, 20)),
    "prefill_image_b4_s1024": PrefillWorkload("prefill_image_b4_s1024", 4, 32, 8, 128, 32, "fp16", (0, 0),
                                              (1024, 1024), alloc_rows=10368),
    "prefill_text_b8": PrefillWorkload("prefill_text_b8", 8, 32, 8, 128, 32, "fp16", (0, 3000), (16, 300),
                                       alloc_rows=10368),
}


@dataclasses.dataclass
class PrefillCase:
    """One synthetic prefill. Index arrays are numpy int32; values are torch tensors."""
    workload: PrefillWorkload
    seed: int
    num_pages: int
    cached_len: np.ndarray    # [B]
    prompt_len: np.ndarray    # [B]
    pages: np.ndarray         # [B, maxp] the request's page table over its allocation
    q: torch.Tensor           # [R, Hq, D], R = sum S
    k_pool: torch.Tensor      # [num_pages, Hkv, ps, D] (before the prompt's K/V are written)
    v_pool: torch.Tensor
    k_new: torch.Tensor       # [R, Hkv, D] the prompt tokens' K/V
    v_new: torch.Tensor
    out_cache_loc: np.ndarray  # [R] slot of prompt token i of request b: position C_b + i

    @property
    def rows(self) -> int:
        return int(self.prompt_len.sum())


def make_prefill_case(wl: PrefillWorkload, seed: int, *, device="cpu", cached_lengths=None,
                      prompt_lengths=None) -> PrefillCase:
    B, Hq, Hkv, D, ps = wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size
    tdt = TORCH_DTYPES[wl.dtype]
    g = torch.Generator().manual_seed(seed)
    if cached_lengths is not None:
        C = np.asarray(cached_lengths, np.int64)
    else:
        C = torch.randint(wl.cached[0], wl.cached[1] + 1, (B,), generator=g).numpy().astype(np.int64)
    if prompt_lengths is not None:
        S = np.asarray(prompt_lengths, np.int64)
    else:
        S = torch.randint(wl.prompt[0], wl.prompt[1] + 1, (B,), generator=g).numpy().astype(np.int64)
    assert C.shape == (B,) and S.shape == (B,)
    rows_each = [max(int(wl.alloc_rows), int(C[b] + S[b])) for b in range(B)]
    npg = [_ceil_div(r, ps) for r in rows_each]
    num_pages = max(1, sum(npg)) + 2
    perm = torch.randperm(num_pages, generator=g).numpy().astype(np.int64)
    maxp = max([1] + npg)
    pages = np.full((B, maxp), -1, np.int64)
    cur = 0
    row_valid = np.zeros((num_pages, ps), bool)
    for b in range(B):
        pages[b, :npg[b]] = perm[cur:cur + npg[b]]
        cur += npg[b]
        flat = np.arange(npg[b] * ps)
        vr = flat < C[b]                       # cached rows; prompt rows are written by the append
        for k_, pg in enumerate(pages[b, :npg[b]]):
            row_valid[pg] = vr[k_ * ps:(k_ + 1) * ps]
    dev = torch.device(device)
    gd = torch.Generator(device=dev).manual_seed(seed + 7919)
    k_pool = torch.empty((num_pages, Hkv, ps, D), dtype=tdt, device=dev)
    v_pool = torch.empty_like(k_pool)
    valid_t = torch.from_numpy(row_valid).to(dev)
    chunk = max(1, (1 << 26) // max(1, Hkv * ps * D))
    for pool in (k_pool, v_pool):
        for p0 in range(0, num_pages, chunk):
            p1 = min(num_pages, p0 + chunk)
            shape = (p1 - p0, Hkv, ps, D)
            garbage = torch.rand(shape, generator=gd, device=dev) * 2000.0 - 1000.0
            normal = torch.randn(shape, generator=gd, device=dev)
            pool[p0:p1] = torch.where(valid_t[p0:p1][:, None, :, None], normal, garbage).to(tdt)
    R = int(S.sum())
    q = torch.randn((R, Hq, D), generator=gd, device=dev).to(tdt)
    k_new = torch.randn((R, Hkv, D), generator=gd, device=dev).to(tdt)
    v_new = torch.randn((R, Hkv, D), generator=gd, device=dev).to(tdt)
    loc = []
    for b in range(B):
        for i in range(int(S[b])):
            pos = int(C[b]) + i
            loc.append(int(pages[b, pos // ps]) * ps + pos % ps)
    return PrefillCase(workload=wl, seed=seed, num_pages=num_pages, cached_len=C.astype(np.int32),
                       prompt_len=S.astype(np.int32), pages=pages.astype(np.int32), q=q, k_pool=k_pool,
                       v_pool=v_pool, k_new=k_new, v_new=v_new, out_cache_loc=np.asarray(loc, np.int32))
