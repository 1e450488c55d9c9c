"""fp64 CPU oracle for shared-prefix (cascade) beam decode attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by ``bench.py``'s CPU-baseline leg, never by the product package.

The C source (``bsp_oracle.c``) holds the plain definitions; this module builds
it with gcc (``build()``) and wraps it with numpy arrays. ``brute`` holds an
independent pure-Python restatement used to pin the C code on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsp_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liborc.so")

DTYPES = {"bf16": 0, "fp16": 1}
ERRORS = {0: "ok", 1: "bad argument", 2: "index out of range", 3: "out of memory"}

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP) into ``oracle/_build/liborc.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    p = ctypes.c_void_p
    i32 = ctypes.c_int32
    lib.orc_half_to_double.restype = ctypes.c_double
    lib.orc_half_to_double.argtypes = [ctypes.c_uint16, ctypes.c_int]
    lib.orc_bucket_rows.restype = i32
    lib.orc_bucket_rows.argtypes = [i32, i32]
    lib.orc_attend.restype = None
    lib.orc_attend.argtypes = [ctypes.c_int, ctypes.c_int, p, p, p, ctypes.c_double, p, p, p]
    lib.orc_merge.restype = None
    lib.orc_merge.argtypes = [ctypes.c_int, ctypes.c_int, p, p, p, p]
    lib.orc_decode_attn.restype = ctypes.c_int
    lib.orc_decode_attn.argtypes = [ctypes.c_int] * 8 + [p, p, p, ctypes.c_int, p, ctypes.c_int, p,
                                                       ctypes.c_int, p, p, p, ctypes.c_double, p,
                                                       ctypes.c_int, p, p]
    lib.orc_prefill_attn.restype = ctypes.c_int
    lib.orc_prefill_attn.argtypes = [ctypes.c_int] * 7 + [p, p, p, ctypes.c_int, ctypes.c_int, p, p, p,
                                                       ctypes.c_double, p, p]
    lib.orc_append_kv.restype = ctypes.c_int
    lib.orc_append_kv.argtypes = [ctypes.c_int] * 5 + [p, p, p, ctypes.c_int64, p, p]
    lib.orc_round_half.restype = ctypes.c_uint16
    lib.orc_round_half.argtypes = [ctypes.c_double, ctypes.c_int]
    lib.orc_rope_cos_sin.restype = None
    lib.orc_rope_cos_sin.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, p]
    lib.orc_rope_rotate.restype = None
    lib.orc_rope_rotate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, p, p]
    lib.orc_round_half_array.restype = None
    lib.orc_round_half_array.argtypes = [ctypes.c_int64, p, p, ctypes.c_int]
    lib.orc_rope_rotate_rows.restype = None
    lib.orc_rope_rotate_rows.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, p,
                                         p, p]
    lib.orc_e4m3_to_double.restype = ctypes.c_double
    lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.orc_round_e4m3.restype = ctypes.c_uint8
    lib.orc_round_e4m3.argtypes = [ctypes.c_double]
    lib.orc_append_kv_fp8.restype = ctypes.c_int
    lib.orc_append_kv_fp8.argtypes = [ctypes.c_int] * 6 + [p, p, p, ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                                                          p, p]
    lib.orc_rope_append_kv_fp8.restype = ctypes.c_int
    lib.orc_rope_append_kv_fp8.argtypes = ([ctypes.c_int] * 6 + [ctypes.c_double] + [ctypes.c_int] * 4 +
                                           [p, p, p, ctypes.c_int64, p, p, ctypes.c_int64, ctypes.c_float,
                                            ctypes.c_float, p, p])
    lib.orc_rope_append_kv.restype = ctypes.c_int
    lib.orc_rope_append_kv.argtypes = ([ctypes.c_int] * 6 + [ctypes.c_double] + [ctypes.c_int] * 4 +
                                       [p, p, p, ctypes.c_int64, p, p, ctypes.c_int64, p, p])
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def half_to_double(bits: int, dtype: str) -> float:
    return _load().orc_half_to_double(int(bits) & 0xFFFF, DTYPES[dtype])


def bucket_rows(valid: int, capacity: int) -> int:
    return int(_load().orc_bucket_rows(int(valid), int(capacity)))


def attend(q, K, V, scale):
    """One fp64 query against explicit keys: returns (O [D], LSE)."""
    q = _c(q, np.float64)
    K = _c(K, np.float64).reshape(-1, q.shape[0])
    V = _c(V, np.float64).reshape(-1, q.shape[0])
    n, D = K.shape
    s = np.empty(max(n, 1), np.float64)
    o = np.empty(D, np.float64)
    lse = np.empty(1, np.float64)
    _load().orc_attend(D, n, _ptr(q), _ptr(K), _ptr(V), float(scale), _ptr(s), _ptr(o), _ptr(lse))
    return o, float(lse[0])


def merge(Os, Ls):
    """Log-sum-exp merge of k partial states: Os [k][D], Ls [k] -> (O [D], LSE)."""
    Os = _c(Os, np.float64)
    Ls = _c(Ls, np.float64).reshape(-1)
    k, D = Os.shape
    o = np.empty(D, np.float64)
    lse = np.empty(1, np.float64)
    _load().orc_merge(D, k, _ptr(Os), _ptr(Ls), _ptr(o), _ptr(lse))
    return o, float(lse[0])


def decode_attn(*, dtype, B, W, Hq, Hkv, D, ps, num_pages, prefix_len, tail_len, prefix_pages,
                beam_pages, cache_indirection, q_bits, k_pool_bits, v_pool_bits, scale, rows=None):
    """Unsplit fp64 decode attention over each beam's logical sequence.

    q_bits [R,Hq,D], pools [num_pages,Hkv,ps,D] as uint16 bit patterns.
    Returns (O [nrows,Hq,D] float64, LSE [nrows,Hq] float64) for ``rows``
    (all B*W rows when None).
    """
    prefix_len = _c(prefix_len, np.int32)
    tail_len = _c(tail_len, np.int32)
    prefix_pages = _c(prefix_pages, np.int32).reshape(B, -1)
    beam_pages = _c(beam_pages, np.int32).reshape(B * W, -1)
    ci = _c(cache_indirection, np.int32).reshape(B, W, -1)
    q_bits = _c(q_bits, np.uint16)
    k_pool_bits = _c(k_pool_bits, np.uint16)
    v_pool_bits = _c(v_pool_bits, np.uint16)
    if rows is None:
        nrows = B * W
        rows_arr = None
    else:
        rows_arr = _c(rows, np.int32)
        nrows = rows_arr.shape[0]
    O = np.empty((nrows, Hq, D), np.float64)
    L = np.empty((nrows, Hq), np.float64)
    rc = _load().orc_decode_attn(
        DTYPES[dtype], B, W, Hq, Hkv, D, ps, num_pages,
        _ptr(prefix_len), _ptr(tail_len), _ptr(prefix_pages), prefix_pages.shape[1],
        _ptr(beam_pages), beam_pages.shape[1], _ptr(ci), ci.shape[2],
        _ptr(q_bits), _ptr(k_pool_bits), _ptr(v_pool_bits), float(scale),
        None if rows_arr is None else _ptr(rows_arr), nrows, _ptr(O), _ptr(L))
    if rc != 0:
        raise ValueError(f"oracle decode_attn: {ERRORS.get(rc, rc)}")
    return O, L


def prefill_attn(*, dtype, B, Hq, Hkv, D, ps, num_pages, cached_len, prompt_len, pages, causal, q_bits,
                 k_pool_bits, v_pool_bits, scale):
    """fp64 prefill over the cached prefix: prompt token i of request b attends positions
    0 .. C_b + i (causal) or 0 .. C_b + S_b - 1, read through pages[b]. q_bits [R,Hq,D] with
    R = sum S_b (requests in order). Returns (O [R,Hq,D], LSE [R,Hq]) in float64."""
    cached_len = _c(cached_len, np.int32)
    prompt_len = _c(prompt_len, np.int32)
    pages = _c(pages, np.int32).reshape(B, -1)
    q_bits = _c(q_bits, np.uint16)
    k_pool_bits = _c(k_pool_bits, np.uint16)
    v_pool_bits = _c(v_pool_bits, np.uint16)
    R = int(prompt_len.sum())
    O = np.empty((R, Hq, D), np.float64)
    L = np.empty((R, Hq), np.float64)
    rc = _load().orc_prefill_attn(
        DTYPES[dtype], B, Hq, Hkv, D, ps, num_pages, _ptr(cached_len), _ptr(prompt_len), _ptr(pages),
        pages.shape[1], 1 if causal else 0, _ptr(q_bits), _ptr(k_pool_bits), _ptr(v_pool_bits), float(scale),
        _ptr(O), _ptr(L))
    if rc != 0:
        raise ValueError(f"oracle prefill_attn: {ERRORS.get(rc, rc)}")
    return O, L


def append_kv(*, Hkv, D, ps, num_pages, out_cache_loc, k_new_bits, v_new_bits, k_pool_bits,
              v_pool_bits, row_stride=None):
    """Paged KV append in place on uint16 pools; raises on a bad slot (pools unchanged)."""
    loc = _c(out_cache_loc, np.int32)
    kn = _c(k_new_bits, np.uint16)
    vn = _c(v_new_bits, np.uint16)
    assert k_pool_bits.flags.c_contiguous and v_pool_bits.flags.c_contiguous
    assert k_pool_bits.dtype == np.uint16 and v_pool_bits.dtype == np.uint16
    n = loc.shape[0]
    if row_stride is None:
        row_stride = Hkv * D
    rc = _load().orc_append_kv(Hkv, D, ps, num_pages, n, _ptr(loc), _ptr(kn), _ptr(vn),
                               int(row_stride), _ptr(k_pool_bits), _ptr(v_pool_bits))
    if rc != 0:
        raise ValueError(f"oracle append_kv: {ERRORS.get(rc, rc)}")


def round_half(x: float, dtype: str) -> int:
    """Nearest bf16 / binary16 bit pattern of a double, ties to even."""
    return int(_load().orc_round_half(float(x), DTYPES[dtype]))


def round_half_array(x, dtype: str) -> np.ndarray:
    """round_half over an array."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_round_half_array(x.size, _ptr(x), _ptr(out), DTYPES[dtype])
    return out


def rope_cos_sin(max_pos: int, rot: int, base: float) -> np.ndarray:
    """fp64 [max_pos][rot]: cos(p*theta_j) for j < rot/2, then sin(p*theta_j)."""
    cs = np.empty((max_pos, rot), np.float64)
    _load().orc_rope_cos_sin(int(max_pos), int(rot), float(base), _ptr(cs))
    return cs


def rope_rotate(x, *, rot: int, interleaved: bool, base: float, pos: int) -> np.ndarray:
    """One head row (fp64 [D]) rotated by position ``pos``, unrounded."""
    x = _c(x, np.float64)
    y = np.empty_like(x)
    _load().orc_rope_rotate(x.shape[0], int(rot), 1 if interleaved else 0, float(base), int(pos), _ptr(x), _ptr(y))
    return y


def rope_rotate_rows(x, positions, *, rot: int, interleaved: bool, base: float) -> np.ndarray:
    """rope_rotate over rows: x fp64 [rows][D], row i by positions[i]; unrounded."""
    x = _c(x, np.float64)
    rows, D = x.shape
    pos = _c(positions, np.int32).reshape(rows)
    y = np.empty_like(x)
    _load().orc_rope_rotate_rows(rows, D, int(rot), 1 if interleaved else 0, float(base), _ptr(pos), _ptr(x), _ptr(y))
    return y


def rope_append_kv(*, dtype, Hq, Hkv, D, rot, interleaved, base, max_pos, ps, num_pages, positions,
                   out_cache_loc, q_bits, k_new_bits, v_new_bits, k_pool_bits, v_pool_bits,
                   q_row_stride=None, row_stride=None):
    """RoPE on the paged append, in place on uint16 arrays: rotated K and plain V rows into the pools,
    the query rows (``q_bits`` [n][..], may be None) rotated in place. Raises on a bad slot or
    position (nothing written)."""
    pos = _c(positions, np.int32)
    loc = _c(out_cache_loc, np.int32)
    n = loc.shape[0]
    for a in (k_pool_bits, v_pool_bits) + (() if q_bits is None else (q_bits,)):
        assert a.dtype == np.uint16 and a.flags.c_contiguous
    kn = _c(k_new_bits, np.uint16).reshape(n, -1) if n else np.zeros((0, Hkv * D), np.uint16)
    vn = _c(v_new_bits, np.uint16).reshape(n, -1) if n else np.zeros((0, Hkv * D), np.uint16)
    rs = kn.shape[1] if row_stride is None else int(row_stride)
    qrs = 0 if q_bits is None else (q_bits.size // max(n, 1) if q_row_stride is None else int(q_row_stride))
    rc = _load().orc_rope_append_kv(
        DTYPES[dtype], Hq, Hkv, D, int(rot), 1 if interleaved else 0, float(base), int(max_pos), ps, num_pages, n,
        _ptr(pos), _ptr(loc), None if q_bits is None else _ptr(q_bits), qrs, _ptr(kn), _ptr(vn), rs,
        _ptr(k_pool_bits), _ptr(v_pool_bits))
    if rc != 0:
        raise ValueError(f"oracle rope_append_kv: {ERRORS.get(rc, rc)}")


def e4m3_to_double(bits: int) -> float:
    return float(_load().orc_e4m3_to_double(int(bits) & 0xFF))


def round_e4m3(x: float) -> int:
    """Nearest E4M3 pattern, ties to even, saturating at +-448."""
    return int(_load().orc_round_e4m3(float(x)))


FP8_SRC = {"bf16": 0, "fp16": 1, "e4m3": 2}


def append_kv_fp8(*, src_dtype, Hkv, D, ps, num_pages, out_cache_loc, k_new_bits, v_new_bits, k_pool_bits,
                  v_pool_bits, k_mul=1.0, v_mul=1.0, row_stride=None):
    """Paged append into uint8 E4M3 pools, in place: 16-bit sources quantised (fp32 product with the
    multiplier, then round_e4m3), E4M3 sources copied. Raises on a bad slot (pools unchanged)."""
    loc = _c(out_cache_loc, np.int32)
    n = loc.shape[0]
    et = np.uint8 if src_dtype == "e4m3" else np.uint16
    kn = _c(k_new_bits, et).reshape(n, -1) if n else np.zeros((0, Hkv * D), et)
    vn = _c(v_new_bits, et).reshape(n, -1) if n else np.zeros((0, Hkv * D), et)
    for a in (k_pool_bits, v_pool_bits):
        assert a.dtype == np.uint8 and a.flags.c_contiguous
    rs = kn.shape[1] if row_stride is None else int(row_stride)
    rc = _load().orc_append_kv_fp8(FP8_SRC[src_dtype], Hkv, D, ps, num_pages, n, _ptr(loc), _ptr(kn), _ptr(vn), rs,
                                   float(np.float32(k_mul)), float(np.float32(v_mul)), _ptr(k_pool_bits),
                                   _ptr(v_pool_bits))
    if rc != 0:
        raise ValueError(f"oracle append_kv_fp8: {ERRORS.get(rc, rc)}")


def rope_append_kv_fp8(*, dtype, Hq, Hkv, D, rot, interleaved, base, max_pos, ps, num_pages, positions,
                       out_cache_loc, q_bits, k_new_bits, v_new_bits, k_pool_bits, v_pool_bits, k_mul=1.0, v_mul=1.0,
                       q_row_stride=None, row_stride=None):
    """RoPE on the append into uint8 E4M3 pools, in place (q rows, 16-bit, rotated in place when given)."""
    pos = _c(positions, np.int32)
    loc = _c(out_cache_loc, np.int32)
    n = loc.shape[0]
    for a in (k_pool_bits, v_pool_bits):
        assert a.dtype == np.uint8 and a.flags.c_contiguous
    if q_bits is not None:
        assert q_bits.dtype == np.uint16 and q_bits.flags.c_contiguous
    kn = _c(k_new_bits, np.uint16).reshape(n, -1) if n else np.zeros((0, Hkv * D), np.uint16)
    vn = _c(v_new_bits, np.uint16).reshape(n, -1) if n else np.zeros((0, Hkv * D), np.uint16)
    rs = kn.shape[1] if row_stride is None else int(row_stride)
    qrs = 0 if q_bits is None else (q_bits.size // max(n, 1) if q_row_stride is None else int(q_row_stride))
    rc = _load().orc_rope_append_kv_fp8(
        DTYPES[dtype], Hq, Hkv, D, int(rot), 1 if interleaved else 0, float(base), int(max_pos), ps, num_pages, n,
        _ptr(pos), _ptr(loc), None if q_bits is None else _ptr(q_bits), qrs, _ptr(kn), _ptr(vn), rs,
        float(np.float32(k_mul)), float(np.float32(v_mul)), _ptr(k_pool_bits), _ptr(v_pool_bits))
    if rc != 0:
        raise ValueError(f"oracle rope_append_kv_fp8: {ERRORS.get(rc, rc)}")


def e4m3_to_half_bits(pool_bits: np.ndarray, dtype: str) -> np.ndarray:
    """E4M3 bytes as bits of the 16-bit dtype with the same value: every E4M3 value (3 fraction bits,
    2^-9 .. 448) is exact in bf16 and in binary16."""
    table = np.array([round_half(e4m3_to_double(b), dtype) for b in range(256)], np.uint16)
    return table[np.asarray(pool_bits, np.uint8)]


def decode_attn_fp8(*, dtype, B, W, Hq, Hkv, D, ps, num_pages, prefix_len, tail_len, prefix_pages, beam_pages,
                    cache_indirection, q_bits, k_pool_bits, v_pool_bits, scale, k_scale=1.0, v_scale=1.0, rows=None):
    """Decode attention over uint8 E4M3 pools dequantised by per-tensor scales (key = E4M3 value x
    k_scale, value = E4M3 value x v_scale): the unsplit attention over the same keys with the scores
    scaled by scale x k_scale and O by v_scale (LSE unchanged), the pools carried exactly in the q dtype.
    Returns (O, LSE) as decode_attn."""
    kp = e4m3_to_half_bits(k_pool_bits, dtype)
    vp = e4m3_to_half_bits(v_pool_bits, dtype)
    O, L = decode_attn(dtype=dtype, B=B, W=W, Hq=Hq, Hkv=Hkv, D=D, ps=ps, num_pages=num_pages,
                       prefix_len=prefix_len, tail_len=tail_len, prefix_pages=prefix_pages, beam_pages=beam_pages,
                       cache_indirection=cache_indirection, q_bits=q_bits, k_pool_bits=kp, v_pool_bits=vp,
                       scale=float(scale) * float(k_scale), rows=rows)
    return O * float(v_scale), L
