"""Thin ctypes binding of libbsp.so (include/bsp.h): argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels. The functions
mirror the C entry points by name; torch tensors supply device memory, pinned
host staging and the current CUDA stream. If the native library is missing or
fails to load, every call raises ``NativeLibraryError``: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

from . import build as _build

BSP_OK = 0
STATUS_NAMES = {0: "BSP_OK", 1: "BSP_ERR_INVALID_ARG", 2: "BSP_ERR_UNSUPPORTED", 3: "BSP_ERR_PAGE_INDEX",
                4: "BSP_ERR_CAPACITY", 5: "BSP_ERR_STALE_PLAN", 6: "BSP_ERR_CUDA", 7: "BSP_ERR_DEVICE_TIMEOUT"}
DTYPES = {"bf16": 0, "fp16": 1, torch.bfloat16: 0, torch.float16: 1}
FLAG_LSE_BASE2 = 1
FLAG_CHECK = 2
FLAG_GRAPH = 4
MAX_TAIL = 8
MAX_GROUP = 8
STATUS_BYTES = 256  # device status words ahead of the plan image in the workspace
DEVFLAG_PAGE_INDEX = 1
DEVFLAG_TIMEOUT = 2
DEVFLAG_POSITION = 4
DEVFLAG_GRAPH = 8


class NativeLibraryError(RuntimeError):
    pass


class BspError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class Geometry(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32)]


class Plan(ctypes.Structure):
    _fields_ = [("geo", Geometry)] + [(n, ctypes.c_int32) for n in (
        "batch", "beam_width", "max_tail", "prefix_pages_stride", "num_units", "num_parts", "row_blocks",
        "beams_per_block", "tile_keys", "max_prefix_len", "max_total_len", "num_sms", "max_tail_len",
        "prefix_ctas")] + [
        ("generation", ctypes.c_uint64), ("ws_device", ctypes.c_void_p), ("ws_device_bytes", ctypes.c_uint64),
        ("ws_host", ctypes.c_void_p), ("image_bytes", ctypes.c_uint64), ("off_req", ctypes.c_uint64),
        ("off_units", ctypes.c_uint64), ("off_pages", ctypes.c_uint64), ("off_part_lse", ctypes.c_uint64),
        ("off_part_o", ctypes.c_uint64), ("device_bytes_used", ctypes.c_uint64),
        ("tail_requests", ctypes.c_int32), ("total_rows", ctypes.c_int32), ("kind", ctypes.c_int32),
        ("layout", ctypes.c_int32), ("off_cta", ctypes.c_uint64), ("reserved", ctypes.c_uint64)]


class RopeConfig(ctypes.Structure):
    _fields_ = [("cos_sin", ctypes.c_void_p), ("max_position", ctypes.c_int32), ("rotary_dim", ctypes.c_int32),
                ("interleaved", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lib = None
EXPORTS = ["bsp_status_string", "bsp_bucket_rows", "bsp_workspace_size", "bsp_plan_build", "bsp_plan",
           "bsp_append_kv", "bsp_decode_attn", "bsp_read_device_status", "bsp_decode_attn_noalloc",
           "bsp_plan_prefill_build", "bsp_plan_prefill", "bsp_prefill_attn", "bsp_rope_cos_sin",
           "bsp_rope_append_kv", "bsp_append_kv_fp8", "bsp_rope_append_kv_fp8", "bsp_plan_update_tails",
           "bsp_decode_attn_fp8"]
NOALLOC_SCRATCH_MIB = 32


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> ctypes.CDLL:
    """Load libbsp.so (building it first only when asked)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise NativeLibraryError(
            f"{_build.LIB} is missing: build it with beam_search_shared_gb300.build.build() "
            "(there is no fallback path)")
    try:
        lib = ctypes.CDLL(_build.LIB)
    except OSError as e:  # pragma: no cover - depends on the box
        raise NativeLibraryError(f"cannot load {_build.LIB}: {e}") from e
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    P = ctypes.POINTER
    lib.bsp_status_string.restype = ctypes.c_char_p
    lib.bsp_status_string.argtypes = [i32]
    lib.bsp_bucket_rows.restype = i32
    lib.bsp_bucket_rows.argtypes = [i32, i32]
    lib.bsp_workspace_size.restype = i32
    lib.bsp_workspace_size.argtypes = [P(Geometry), i32, i32, i32, P(sz), P(sz)]
    lib.bsp_plan_build.restype = i32
    lib.bsp_plan_build.argtypes = [P(Geometry), i32, i32, vp, vp, vp, i32, i32, i32, vp, sz, P(Plan)]
    lib.bsp_plan.restype = i32
    lib.bsp_plan.argtypes = [P(Geometry), i32, i32, vp, vp, vp, i32, i32, vp, sz, vp, sz, vp, P(Plan)]
    lib.bsp_plan_update_tails.restype = i32
    lib.bsp_plan_update_tails.argtypes = [P(Plan), vp, vp]
    lib.bsp_append_kv.restype = i32
    lib.bsp_append_kv.argtypes = [P(Plan), vp, vp, i64, vp, i32, vp, vp, vp, vp]
    lib.bsp_decode_attn.restype = i32
    lib.bsp_decode_attn.argtypes = [P(Plan), vp, vp, vp, vp, i32, vp, i32, ctypes.c_float, i32, vp, vp, vp, vp]
    f32 = ctypes.c_float
    lib.bsp_decode_attn_fp8.restype = i32
    lib.bsp_decode_attn_fp8.argtypes = [P(Plan), vp, vp, vp, vp, i32, vp, i32, f32, f32, f32, i32, vp, vp, vp, vp]
    lib.bsp_plan_prefill_build.restype = i32
    lib.bsp_plan_prefill_build.argtypes = [P(Geometry), i32, vp, vp, vp, i32, i32, i32, vp, sz, P(Plan)]
    lib.bsp_plan_prefill.restype = i32
    lib.bsp_plan_prefill.argtypes = [P(Geometry), i32, vp, vp, vp, i32, i32, vp, sz, vp, sz, vp, P(Plan)]
    lib.bsp_prefill_attn.restype = i32
    lib.bsp_prefill_attn.argtypes = [P(Plan), vp, vp, vp, ctypes.c_float, i32, vp, vp, vp, vp]
    lib.bsp_rope_cos_sin.restype = i32
    lib.bsp_rope_cos_sin.argtypes = [i32, i32, ctypes.c_double, vp, vp]
    lib.bsp_rope_append_kv.restype = i32
    lib.bsp_rope_append_kv.argtypes = [P(Plan), P(RopeConfig), vp, vp, i64, vp, vp, i64, vp, i32, vp, vp, vp, vp]
    lib.bsp_rope_append_kv_fp8.restype = i32
    lib.bsp_rope_append_kv_fp8.argtypes = [P(Plan), P(RopeConfig), vp, vp, i64, vp, vp, i64, ctypes.c_float,
                                           ctypes.c_float, vp, i32, vp, vp, vp, vp]
    lib.bsp_append_kv_fp8.restype = i32
    lib.bsp_append_kv_fp8.argtypes = [P(Plan), vp, vp, i64, i32, ctypes.c_float, ctypes.c_float, vp, i32, vp, vp, vp, vp]
    lib.bsp_read_device_status.restype = i32
    lib.bsp_read_device_status.argtypes = [P(Plan), vp, i32, P(i32)]
    lib.bsp_decode_attn_noalloc.restype = i32
    lib.bsp_decode_attn_noalloc.argtypes = [P(Geometry), i32, i32, vp, vp, vp, i32, i32, vp, vp, vp, vp, i32, vp, i32,
                                            ctypes.c_float, i32, vp, vp, vp]
    _lib = lib
    return lib


def _check(fn: str, st: int):
    if st != BSP_OK:
        raise BspError(fn, st)


def status_string(status: int) -> str:
    return load().bsp_status_string(int(status)).decode()


KV_DTYPE_SAME, KV_DTYPE_E4M3 = 0, 1


def geometry(num_q_heads, num_kv_heads, head_dim, page_size, num_pages, dtype, kv_dtype: int = KV_DTYPE_SAME) -> Geometry:
    """kv_dtype: KV_DTYPE_SAME (the pools hold `dtype`) or KV_DTYPE_E4M3 (one-byte E4M3 pools)."""
    return Geometry(int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size), int(num_pages),
                    DTYPES[dtype], int(kv_dtype))


def bucket_rows(valid_rows: int, capacity: int) -> int:
    return int(load().bsp_bucket_rows(int(valid_rows), int(capacity)))


def workspace_size(geo: Geometry, max_batch: int, max_beam: int, max_prefix_pages: int):
    d, h = ctypes.c_size_t(), ctypes.c_size_t()
    _check("bsp_workspace_size", load().bsp_workspace_size(ctypes.byref(geo), int(max_batch), int(max_beam),
                                                           int(max_prefix_pages), ctypes.byref(d), ctypes.byref(h)))
    return d.value, h.value


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def plan_build(geo: Geometry, batch, beam_width, prefix_len, tail_len, prefix_pages, max_tail, num_sms,
               image_bytes: int = 1 << 24):
    """Host-only planning. Returns (Plan, image bytes as a numpy uint8 array)."""
    pl, tl = _i32(prefix_len), _i32(tail_len)
    pp = _i32(prefix_pages).reshape(int(batch), -1) if int(batch) else np.zeros((0, 1), np.int32)
    img = np.zeros(int(image_bytes), np.uint8)
    plan = Plan()
    _check("bsp_plan_build", load().bsp_plan_build(
        ctypes.byref(geo), int(batch), int(beam_width), _ptr(pl), _ptr(tl), _ptr(pp), pp.shape[1], int(max_tail),
        int(num_sms), _ptr(img), img.nbytes, ctypes.byref(plan)))
    return plan, img[:plan.image_bytes]


REQ_FIELDS = 12  # int32 per request record of a plan image


def plan_requests(plan_: Plan, img: np.ndarray) -> np.ndarray:
    """Per-request records of a host plan image (``plan_build``), int32 [batch, 12]: prompt length,
    tail length, prompt partial states, first partial slot, first page entry, finished by the
    prompt kernel (1) or by the tail kernel (0), two unused, query rows per head, causal base (-1:
    none), first query row, one unused."""
    lo = plan_.off_req - STATUS_BYTES
    return img[lo:lo + plan_.batch * REQ_FIELDS * 4].view(np.int32).reshape(plan_.batch, REQ_FIELDS)


def plan_prefill_build(geo: Geometry, batch, cached_len, prompt_len, pages, causal, num_sms,
                       image_bytes: int = 1 << 24):
    """Host-only prefill planning. Returns (Plan, image bytes as a numpy uint8 array)."""
    cl, pl = _i32(cached_len), _i32(prompt_len)
    pg = _i32(pages).reshape(int(batch), -1) if int(batch) else np.zeros((0, 1), np.int32)
    img = np.zeros(int(image_bytes), np.uint8)
    plan = Plan()
    _check("bsp_plan_prefill_build", load().bsp_plan_prefill_build(
        ctypes.byref(geo), int(batch), _ptr(cl), _ptr(pl), _ptr(pg), pg.shape[1], 1 if causal else 0,
        int(num_sms), _ptr(img), img.nbytes, ctypes.byref(plan)))
    return plan, img[:plan.image_bytes]


def plan_prefill(geo: Geometry, batch, cached_len, prompt_len, pages, causal, ws: "Workspace",
                 stream=None) -> Plan:
    """bsp_plan_prefill: host arrays in, plan staged into ``ws`` on ``stream`` (no sync)."""
    cl, pl = _i32(cached_len), _i32(prompt_len)
    pg = _i32(pages).reshape(int(batch), -1) if int(batch) else np.zeros((0, 1), np.int32)
    out = Plan()
    _check("bsp_plan_prefill", load().bsp_plan_prefill(
        ctypes.byref(geo), int(batch), _ptr(cl), _ptr(pl), _ptr(pg), pg.shape[1], 1 if causal else 0,
        _dptr(ws.device), ws.device.numel(), _dptr(ws.host), ws.host.numel(), _stream(stream), ctypes.byref(out)))
    return out


def prefill_attn(plan_: Plan, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, softmax_scale: float,
                 o: torch.Tensor, lse: torch.Tensor, flags: int = 0, events=None, stream=None):
    """bsp_prefill_attn: writes o [total_rows,Hq,D] and lse [total_rows,Hq] (fp32)."""
    _check("bsp_prefill_attn", load().bsp_prefill_attn(
        ctypes.byref(plan_), _dptr(q), _dptr(k_pool), _dptr(v_pool), float(softmax_scale), int(flags), _dptr(o),
        _dptr(lse), _events(events, 3), _stream(stream)))


class Workspace:
    """A device workspace and its pinned host staging buffer, sized by bsp_workspace_size."""

    def __init__(self, geo: Geometry, max_batch: int, max_beam: int, max_prefix_pages: int, device=None):
        dev_bytes, host_bytes = workspace_size(geo, max_batch, max_beam, max_prefix_pages)
        device = torch.device("cuda") if device is None else torch.device(device)
        self.device = torch.empty(dev_bytes, dtype=torch.uint8, device=device)
        self.device.zero_()
        self.host = torch.empty(host_bytes, dtype=torch.uint8, pin_memory=True)
        self.host.zero_()

    def plan(self, geo: Geometry, batch, beam_width, prefix_len, tail_len, prefix_pages, max_tail=MAX_TAIL,
             stream=None) -> Plan:
        return plan(geo, batch, beam_width, prefix_len, tail_len, prefix_pages, max_tail, self, stream)


def plan(geo: Geometry, batch, beam_width, prefix_len, tail_len, prefix_pages, max_tail, ws: Workspace,
         stream=None) -> Plan:
    """bsp_plan: host arrays in, plan staged into ``ws`` on ``stream`` (no sync)."""
    pl, tl = _i32(prefix_len), _i32(tail_len)
    pp = _i32(prefix_pages).reshape(int(batch), -1) if int(batch) else np.zeros((0, 1), np.int32)
    out = Plan()
    _check("bsp_plan", load().bsp_plan(
        ctypes.byref(geo), int(batch), int(beam_width), _ptr(pl), _ptr(tl), _ptr(pp), pp.shape[1], int(max_tail),
        _dptr(ws.device), ws.device.numel(), _dptr(ws.host), ws.host.numel(), _stream(stream), ctypes.byref(out)))
    return out


def plan_update_tails(plan_: Plan, tail_len, stream=None) -> Plan:
    """bsp_plan_update_tails: new tail lengths for a current decode plan, in place (no sync)."""
    tl = _i32(tail_len)
    if tl.shape[0] != plan_.batch:
        raise ValueError(f"tail_len has {tl.shape[0]} entries for a batch of {plan_.batch}")
    _check("bsp_plan_update_tails", load().bsp_plan_update_tails(ctypes.byref(plan_), _ptr(tl), _stream(stream)))
    return plan_


def _events(events, n):
    if events is None:
        return None
    assert len(events) == n
    for e in events:
        if e.cuda_event == 0:
            e.record()  # materialise the underlying cudaEvent_t
    return (ctypes.c_void_p * n)(*[e.cuda_event for e in events])


def append_kv(plan_: Plan, k_new: torch.Tensor, v_new: torch.Tensor, out_cache_loc: torch.Tensor,
              k_pool: torch.Tensor, v_pool: torch.Tensor, src_row_stride: Optional[int] = None, events=None,
              stream=None):
    """bsp_append_kv: k_new/v_new rows [n, Hkv*D] (row stride in elements), out_cache_loc int32 [n].

    ``events``: optional 2 timing events recorded before and after the append kernel.
    """
    n = int(out_cache_loc.numel())
    if src_row_stride is None:
        src_row_stride = int(k_new.stride(0)) if k_new.dim() >= 1 and n else plan_.geo.num_kv_heads * plan_.geo.head_dim
    _check("bsp_append_kv", load().bsp_append_kv(
        ctypes.byref(plan_), _dptr(k_new), _dptr(v_new), int(src_row_stride), _dptr(out_cache_loc), n,
        _dptr(k_pool), _dptr(v_pool), _events(events, 2), _stream(stream)))


FP8_SRC_16BIT, FP8_SRC_E4M3 = 0, 1


def append_kv_fp8(plan_: Plan, k_new: torch.Tensor, v_new: torch.Tensor, out_cache_loc: torch.Tensor,
                  k_pool: torch.Tensor, v_pool: torch.Tensor, k_mul: float = 1.0, v_mul: float = 1.0,
                  src_row_stride: Optional[int] = None, events=None, stream=None):
    """bsp_append_kv_fp8: uint8 (E4M3) pools; k_new/v_new rows [n, Hkv*D] of the geometry's 16-bit dtype
    (quantised with the multipliers) or of E4M3 bytes (torch.float8_e4m3fn or uint8, copied)."""
    n = int(out_cache_loc.numel())
    src = FP8_SRC_E4M3 if k_new.dtype in (torch.uint8, torch.float8_e4m3fn) else FP8_SRC_16BIT
    if src_row_stride is None:
        src_row_stride = int(k_new.stride(0)) if k_new.dim() >= 1 and n else plan_.geo.num_kv_heads * plan_.geo.head_dim
    _check("bsp_append_kv_fp8", load().bsp_append_kv_fp8(
        ctypes.byref(plan_), _dptr(k_new), _dptr(v_new), int(src_row_stride), src, float(k_mul), float(v_mul),
        _dptr(out_cache_loc), n, _dptr(k_pool), _dptr(v_pool), _events(events, 2), _stream(stream)))


class Rope:
    """A RoPE table (device fp32 [max_position][rotary_dim], filled by bsp_rope_cos_sin) and its layout."""

    def __init__(self, max_position: int, rotary_dim: int, base: float, interleaved: bool = False, device="cuda",
                 stream=None):
        self.cos_sin = torch.empty((int(max_position), int(rotary_dim)), dtype=torch.float32, device=device)
        self.base = float(base)
        _check("bsp_rope_cos_sin", load().bsp_rope_cos_sin(int(max_position), int(rotary_dim), self.base,
                                                            _dptr(self.cos_sin), _stream(stream)))
        self.config = RopeConfig(self.cos_sin.data_ptr(), int(max_position), int(rotary_dim), 1 if interleaved else 0, 0)

    @property
    def rotary_dim(self) -> int:
        return int(self.config.rotary_dim)

    @property
    def interleaved(self) -> bool:
        return bool(self.config.interleaved)

    @property
    def max_position(self) -> int:
        return int(self.config.max_position)


def rope_append_kv(plan_: Plan, rope: Rope, positions: torch.Tensor, q: Optional[torch.Tensor], k_new: torch.Tensor,
                   v_new: torch.Tensor, out_cache_loc: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                   src_row_stride: Optional[int] = None, q_row_stride: Optional[int] = None, events=None,
                   stream=None):
    """bsp_rope_append_kv: rotated K and plain V rows into the pools, q [n, Hq*D] rotated in place (or None).
    positions, out_cache_loc: int32 [n] on the device."""
    n = int(out_cache_loc.numel())
    row = plan_.geo.num_kv_heads * plan_.geo.head_dim
    if src_row_stride is None:
        src_row_stride = int(k_new.stride(0)) if k_new.dim() >= 1 and n else row
    if q is not None and q_row_stride is None:
        q_row_stride = int(q.stride(0)) if q.dim() >= 1 and n else plan_.geo.num_q_heads * plan_.geo.head_dim
    _check("bsp_rope_append_kv", load().bsp_rope_append_kv(
        ctypes.byref(plan_), ctypes.byref(rope.config), _dptr(positions), _dptr(q), int(q_row_stride or 0),
        _dptr(k_new), _dptr(v_new), int(src_row_stride), _dptr(out_cache_loc), n, _dptr(k_pool), _dptr(v_pool),
        _events(events, 2), _stream(stream)))


def rope_append_kv_fp8(plan_: Plan, rope: Rope, positions: torch.Tensor, q: Optional[torch.Tensor],
                       k_new: torch.Tensor, v_new: torch.Tensor, out_cache_loc: torch.Tensor, k_pool: torch.Tensor,
                       v_pool: torch.Tensor, k_mul: float = 1.0, v_mul: float = 1.0,
                       src_row_stride: Optional[int] = None, q_row_stride: Optional[int] = None, events=None,
                       stream=None):
    """bsp_rope_append_kv_fp8: rotated K and V quantised into uint8 (E4M3) pools, q rotated in place."""
    n = int(out_cache_loc.numel())
    row = plan_.geo.num_kv_heads * plan_.geo.head_dim
    if src_row_stride is None:
        src_row_stride = int(k_new.stride(0)) if k_new.dim() >= 1 and n else row
    if q is not None and q_row_stride is None:
        q_row_stride = int(q.stride(0)) if q.dim() >= 1 and n else plan_.geo.num_q_heads * plan_.geo.head_dim
    _check("bsp_rope_append_kv_fp8", load().bsp_rope_append_kv_fp8(
        ctypes.byref(plan_), ctypes.byref(rope.config), _dptr(positions), _dptr(q), int(q_row_stride or 0),
        _dptr(k_new), _dptr(v_new), int(src_row_stride), float(k_mul), float(v_mul), _dptr(out_cache_loc), n,
        _dptr(k_pool), _dptr(v_pool), _events(events, 2), _stream(stream)))


def decode_attn(plan_: Plan, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                beam_pages: Optional[torch.Tensor], cache_indirection: Optional[torch.Tensor], softmax_scale: float,
                o: torch.Tensor, lse: torch.Tensor, flags: int = 0, events=None, stream=None):
    """bsp_decode_attn: writes o [R,Hq,D] and lse [R,Hq] (fp32).

    ``events``: optional 3 torch.cuda.Event(enable_timing=True) recorded around the prompt and tail kernels.
    """
    bps = int(beam_pages.shape[-1]) if beam_pages is not None else 0
    max_seq = int(cache_indirection.shape[-1]) if cache_indirection is not None else 0
    ev = _events(events, 3)
    _check("bsp_decode_attn", load().bsp_decode_attn(
        ctypes.byref(plan_), _dptr(q), _dptr(k_pool), _dptr(v_pool), _dptr(beam_pages), bps,
        _dptr(cache_indirection), max_seq, float(softmax_scale), int(flags), _dptr(o), _dptr(lse), ev,
        _stream(stream)))


def read_device_status(plan_: Plan, clear: bool = True, stream=None):
    """Synchronises the stream; returns (status, device flag bits)."""
    flags = ctypes.c_int32(0)
    st = load().bsp_read_device_status(ctypes.byref(plan_), _stream(stream), int(bool(clear)), ctypes.byref(flags))
    return int(st), int(flags.value)


def decode_attn_fp8(plan_: Plan, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                    beam_pages: Optional[torch.Tensor], cache_indirection: Optional[torch.Tensor], softmax_scale: float,
                    k_scale: float, v_scale: float, o: torch.Tensor, lse: torch.Tensor, flags: int = 0, events=None,
                    stream=None):
    """bsp_decode_attn_fp8: decode attention over uint8 E4M3 pools (key = code x k_scale, value = code x
    v_scale); writes o [R,Hq,D] in the q dtype and lse [R,Hq] (fp32)."""
    bps = int(beam_pages.shape[-1]) if beam_pages is not None else 0
    max_seq = int(cache_indirection.shape[-1]) if cache_indirection is not None else 0
    ev = _events(events, 3)
    _check("bsp_decode_attn_fp8", load().bsp_decode_attn_fp8(
        ctypes.byref(plan_), _dptr(q), _dptr(k_pool), _dptr(v_pool), _dptr(beam_pages), bps,
        _dptr(cache_indirection), max_seq, float(softmax_scale), float(k_scale), float(v_scale), int(flags),
        _dptr(o), _dptr(lse), ev, _stream(stream)))


def decode_attn_noalloc(geo: Geometry, batch, beam_width, prefix_len, tail_len, prefix_pages, max_tail,
                        q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                        beam_pages: Optional[torch.Tensor], cache_indirection: Optional[torch.Tensor],
                        softmax_scale: float, o: torch.Tensor, lse: torch.Tensor, flags: int = 0, stream=None):
    """bsp_decode_attn_noalloc: plan + cascade attention with the library's fixed device scratch.

    For callers that cannot allocate device memory: no workspace is passed and nothing is allocated.
    Calls share one scratch array per GPU; calls whose GPU work overlaps race on it.
    """
    pl, tl = _i32(prefix_len), _i32(tail_len)
    pp = _i32(prefix_pages).reshape(int(batch), -1) if int(batch) else np.zeros((0, 1), np.int32)
    bps = int(beam_pages.shape[-1]) if beam_pages is not None else 0
    max_seq = int(cache_indirection.shape[-1]) if cache_indirection is not None else 0
    _check("bsp_decode_attn_noalloc", load().bsp_decode_attn_noalloc(
        ctypes.byref(geo), int(batch), int(beam_width), _ptr(pl), _ptr(tl), _ptr(pp), pp.shape[1], int(max_tail),
        _dptr(q), _dptr(k_pool), _dptr(v_pool), _dptr(beam_pages), bps, _dptr(cache_indirection), max_seq,
        float(softmax_scale), int(flags), _dptr(o), _dptr(lse), _stream(stream)))
