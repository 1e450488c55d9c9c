"""Pure-Python brute force of cascade beam decode attention, for tiny inputs.

TEST INFRASTRUCTURE ONLY. An independent restatement of the same definition as
``bsp_oracle.c`` (different language, different code): it materialises each
beam's logical K/V sequence densely, one position at a time, and applies the
textbook softmax-weighted average with Python floats. It pins the C oracle's
paged gather and attention arithmetic on small cases.

Definition followed: TensorRT-LLM PR #21738 ("Add opt-in cascade attention for
wide beam search on KVCM V2"), description: the prompt is read through beam 0's
page table and each beam's tail through cache_indirection, and the split
prefix/tail states merge exactly to unsplit attention.
"""
from __future__ import annotations

import math
import struct


def half_bits_to_float(bits: int, dtype: str) -> float:
    """Decode one 16-bit pattern with the struct module (IEEE half or bf16)."""
    bits &= 0xFFFF
    if dtype == "fp16":
        return struct.unpack("<e", struct.pack("<H", bits))[0]
    return struct.unpack("<f", struct.pack("<I", bits << 16))[0]


def logical_sequence(b, w, *, W, ps, prefix_len, tail_len, prefix_pages, beam_pages, ci):
    """List of (page, slot) for each logical position of beam w of request b."""
    seq = []
    P, T = int(prefix_len[b]), int(tail_len[b])
    for pos in range(P + T):
        if pos < P:
            page = int(prefix_pages[b][pos // ps])
        else:
            src = int(ci[b][w][pos])
            page = int(beam_pages[b * W + src][pos // ps])
        seq.append((page, pos % ps))
    return seq


def attend(q, keys, values, scale):
    """softmax(scale * q.k_j) weighted mean of values; (O, LSE) in Python floats."""
    if not keys:
        return [0.0] * len(q), -math.inf
    scores = [scale * math.fsum(a * c for a, c in zip(q, k)) for k in keys]
    top = max(scores)
    weights = [math.exp(s - top) for s in scores]
    total = math.fsum(weights)
    out = [math.fsum(wt * v[d] for wt, v in zip(weights, values)) / total for d in range(len(q))]
    return out, top + math.log(total)


def decode_attn(*, dtype, B, W, Hq, Hkv, D, ps, prefix_len, tail_len, prefix_pages, beam_pages,
                cache_indirection, q_bits, k_pool_bits, v_pool_bits, scale):
    """Nested lists O[r][h][d], LSE[r][h] for every row r = b*W + w."""
    G = Hq // Hkv
    O, L = [], []
    for b in range(B):
        for w in range(W):
            r = b * W + w
            seq = logical_sequence(b, w, W=W, ps=ps, prefix_len=prefix_len, tail_len=tail_len,
                                   prefix_pages=prefix_pages, beam_pages=beam_pages,
                                   ci=cache_indirection)
            row_o, row_l = [], []
            for h in range(Hq):
                g = h // G
                q = [half_bits_to_float(x, dtype) for x in q_bits[r][h]]
                keys = [[half_bits_to_float(x, dtype) for x in k_pool_bits[p][g][s]] for p, s in seq]
                vals = [[half_bits_to_float(x, dtype) for x in v_pool_bits[p][g][s]] for p, s in seq]
                o, lse = attend(q, keys, vals, scale)
                row_o.append(o)
                row_l.append(lse)
            O.append(row_o)
            L.append(row_l)
    return O, L


def prefill_attn(*, dtype, B, Hq, Hkv, D, ps, cached_len, prompt_len, pages, causal, q_bits, k_pool_bits,
                 v_pool_bits, scale):
    """Nested lists O[r][h][d], LSE[r][h] for every prompt row r (requests in order, tokens in order).

    Prefill over the cached prefix (TensorRT-Model-Connect PR #2202, Implementation): prompt token i of
    request b sees the request's cached rows and its prompt rows up to itself (all of them when not
    causal), every position read through the request's page table."""
    G = Hq // Hkv
    O, L = [], []
    r = 0
    for b in range(B):
        C, S = int(cached_len[b]), int(prompt_len[b])
        for i in range(S):
            n = C + i + 1 if causal else C + S
            seq = [(int(pages[b][pos // ps]), pos % ps) for pos in range(n)]
            row_o, row_l = [], []
            for h in range(Hq):
                g = h // G
                q = [half_bits_to_float(x, dtype) for x in q_bits[r][h]]
                keys = [[half_bits_to_float(x, dtype) for x in k_pool_bits[p][g][s]] for p, s in seq]
                vals = [[half_bits_to_float(x, dtype) for x in v_pool_bits[p][g][s]] for p, s in seq]
                o, lse = attend(q, keys, vals, scale)
                row_o.append(o)
                row_l.append(lse)
            O.append(row_o)
            L.append(row_l)
            r += 1
    return O, L


def nearest_half_bits(x: float, dtype: str) -> int:
    """Nearest 16-bit pattern of a Python float by search over every finite pattern of the format
    (ties to the pattern with the even fraction; past the largest finite value by half its spacing or
    more: infinity). Slow and obvious; for small inputs."""
    global _FINITE
    if math.isnan(x):
        return 0x7FC0 if dtype == "bf16" else 0x7E00
    key = dtype
    if key not in _FINITE:
        vals = []
        for b in range(0x8000):
            v = half_bits_to_float(b, dtype)
            if math.isfinite(v):
                vals.append((v, b))
        vals.sort()
        _FINITE[key] = vals
    vals = _FINITE[key]
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    top, top_bits = vals[-1]
    step = top - vals[-2][0]
    if a >= top + step / 2:
        return sign | (top_bits + 1)          # the infinity pattern follows the largest finite one
    lo, hi = 0, len(vals) - 1
    while lo < hi:                             # first value >= a
        mid = (lo + hi) // 2
        if vals[mid][0] < a:
            lo = mid + 1
        else:
            hi = mid
    if vals[lo][0] == a or lo == 0:
        return sign | vals[lo][1]
    below, above = vals[lo - 1], vals[lo]
    if a - below[0] < above[0] - a:
        return sign | below[1]
    if a - below[0] > above[0] - a:
        return sign | above[1]
    return sign | (below[1] if below[1] % 2 == 0 else above[1])


_FINITE: dict = {}


def rope_rotate(x, *, rot, interleaved, base, pos):
    """RoPE of one head row as complex multiplication (RoFormer, the complex form of section 3.2):
    pair j is the complex number x_a + i x_b, multiplied by e^{i pos theta_j}, theta_j = base^(-2j/rot)."""
    half = rot // 2
    y = list(x)
    for j in range(half):
        a, b = (2 * j, 2 * j + 1) if interleaved else (j, j + half)
        theta = base ** (-2.0 * j / rot)
        z = complex(x[a], x[b]) * complex(math.cos(pos * theta), math.sin(pos * theta))
        y[a], y[b] = z.real, z.imag
    return y


def rope_append_kv(*, dtype, Hq, Hkv, D, rot, interleaved, base, ps, positions, out_cache_loc, q_bits,
                   k_new_bits, v_new_bits, k_pool_bits, v_pool_bits):
    """Nested-list restatement of the RoPE paged append (in place on the nested lists): rotated K and
    plain V of token i, head h at pool[loc // ps][h][loc % ps]; q rows of token i rotated in place."""
    for i, (p, loc) in enumerate(zip(positions, out_cache_loc)):
        page, off = loc // ps, loc % ps
        for h in range(Hkv):
            k = [half_bits_to_float(v, dtype) for v in k_new_bits[i][h]]
            k_pool_bits[page][h][off] = [nearest_half_bits(v, dtype)
                                         for v in rope_rotate(k, rot=rot, interleaved=interleaved, base=base, pos=p)]
            v_pool_bits[page][h][off] = list(v_new_bits[i][h])
        if q_bits is not None:
            for h in range(Hq):
                qv = [half_bits_to_float(v, dtype) for v in q_bits[i][h]]
                q_bits[i][h] = [nearest_half_bits(v, dtype)
                                for v in rope_rotate(qv, rot=rot, interleaved=interleaved, base=base, pos=p)]


def e4m3_bits_to_float(bits: int) -> float:
    """Decode one E4M3 byte from its fields: sign, 4 exponent bits (bias 7), 3 fraction bits; exponent 0
    is subnormal (fraction x 2^-9), the all-ones pattern of exponent and fraction is NaN."""
    bits &= 0xFF
    sign = -1.0 if bits & 0x80 else 1.0
    e, m = (bits >> 3) & 15, bits & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1 + m / 8) * 2.0 ** (e - 7)


def decode_attn_fp8(*, dtype, B, W, Hq, Hkv, D, ps, prefix_len, tail_len, prefix_pages, beam_pages,
                    cache_indirection, q_bits, k_pool_bits, v_pool_bits, scale, k_scale, v_scale):
    """Decode attention over E4M3 pools: every key is its E4M3 value times k_scale and every value row
    its E4M3 values times v_scale (the dequantisation of a per-tensor-scaled fp8 cache); q in dtype."""
    G = Hq // Hkv
    O, L = [], []
    for b in range(B):
        for w in range(W):
            r = b * W + w
            seq = logical_sequence(b, w, W=W, ps=ps, prefix_len=prefix_len, tail_len=tail_len,
                                   prefix_pages=prefix_pages, beam_pages=beam_pages, ci=cache_indirection)
            row_o, row_l = [], []
            for h in range(Hq):
                g = h // G
                q = [half_bits_to_float(x, dtype) for x in q_bits[r][h]]
                keys = [[e4m3_bits_to_float(x) * k_scale for x in k_pool_bits[p][g][s]] for p, s in seq]
                vals = [[e4m3_bits_to_float(x) * v_scale for x in v_pool_bits[p][g][s]] for p, s in seq]
                o, lse = attend(q, keys, vals, scale)
                row_o.append(o)
                row_l.append(lse)
            O.append(row_o)
            L.append(row_l)
    return O, L
