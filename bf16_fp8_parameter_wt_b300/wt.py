"""Thin Python binding of libwt.so (include/wt.h): argument marshalling only.

Every step of the preparation runs in the library's CUDA kernels; this
module only turns Python descriptors and integer device pointers into the
C structures and calls the entry points of the same names. There is no
fallback: if libwt.so is missing the import of the library fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwt.so")

WT_OK = 0
STATUS_NAMES = ["WT_OK", "WT_ERR_INVALID_ARGUMENT", "WT_ERR_SHAPE", "WT_ERR_LAYOUT_OVERLAP",
                "WT_ERR_POOL_TOO_SMALL", "WT_ERR_ALIGNMENT", "WT_ERR_OUT_OF_MEMORY",
                "WT_ERR_CUDA", "WT_ERR_TIMEOUT", "WT_ERR_INTERNAL"]
WT_OUT_BF16 = 0
WT_OUT_FP8_E4M3_B128 = 1
WT_OFFSET_AUTO = 2**64 - 1
WT_FLAG_FORCE_NARROW = 0x1
WT_FLAG_DEBUG_CHECKS = 0x2
WT_FLAG_SHARD_LOCAL = 0x4
WT_FLAG_SHARD_HALO = 0x8

# every entry point include/wt.h declares
EXPORTS = ["wt_plan_create", "wt_plan_pool_bytes", "wt_plan_output_layout",
           "wt_plan_shard_host_offset", "wt_plan_shard_rows_read", "wt_plan_get_stats", "wt_prepare", "wt_prepare_offload",
           "wt_plan_check", "wt_debug_fail_offload_chunk", "wt_debug_stall_unit", "wt_plan_destroy",
           "wt_prepare_noalloc", "wt_noalloc_check", "wt_debug_noalloc_stall_unit", "wt_quantize_tokens", "wt_tokens_check",
           "wt_debug_tokens_stall_group", "wt_plan_set_counters",
           "wt_plan_expected_count", "wt_wait_counters", "wt_debug_e4m3_encode",
           "wt_status_string", "wt_last_error"]


class WTError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{self.name}: {detail}")


class wt_param_desc(C.Structure):
    _fields_ = [("name", C.c_char_p), ("rows", C.c_int64), ("cols", C.c_int64),
                ("num_shards", C.c_int32), ("shard_rows", C.POINTER(C.c_int64))]


class wt_slice_desc(C.Structure):
    _fields_ = [("dim", C.c_int32), ("num_ranges", C.c_int32),
                ("begin", C.POINTER(C.c_int64)), ("length", C.POINTER(C.c_int64))]


class wt_output_desc(C.Structure):
    _fields_ = [("name", C.c_char_p), ("num_parts", C.c_int32),
                ("part_params", C.POINTER(C.c_int32)), ("format", C.c_int32),
                ("num_dsts", C.c_int32), ("dst_ranks", C.POINTER(C.c_int32)),
                ("dst_data_off", C.POINTER(C.c_uint64)), ("dst_scale_off", C.POINTER(C.c_uint64)),
                ("dst_slices", C.POINTER(wt_slice_desc))]


class wt_plan_desc(C.Structure):
    _fields_ = [("num_params", C.c_int32), ("params", C.POINTER(wt_param_desc)),
                ("num_outputs", C.c_int32), ("outputs", C.POINTER(wt_output_desc)),
                ("num_ranks", C.c_int32), ("pool_capacity", C.POINTER(C.c_uint64)),
                ("offload_chunk_bytes", C.c_uint64), ("flags", C.c_uint32),
                ("local_shard", C.c_int32)]


class wt_plan_stats(C.Structure):
    _fields_ = [("num_units", C.c_int64), ("num_params_total", C.c_int64),
                ("bytes_read", C.c_uint64), ("bytes_written", C.c_uint64),
                ("host_bytes", C.c_uint64), ("num_chunks", C.c_int32), ("num_slots", C.c_int32)]


_lib = None


def lib() -> C.CDLL:
    """Load libwt.so (built in-tree by bf16_fp8_parameter_wt_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m bf16_fp8_parameter_wt_b300.build`")
        L = C.CDLL(LIB_PATH)
        P = C.c_void_p
        L.wt_plan_create.argtypes = [C.POINTER(wt_plan_desc), C.c_int, C.POINTER(P)]
        L.wt_plan_pool_bytes.argtypes = [P, C.c_int32, C.POINTER(C.c_uint64)]
        L.wt_plan_output_layout.argtypes = [P, C.c_int32, C.c_int32, C.POINTER(C.c_int32),
                                            C.POINTER(C.c_uint64), C.POINTER(C.c_uint64)]
        L.wt_plan_shard_host_offset.argtypes = [P, C.c_int32, C.c_int32, C.POINTER(C.c_uint64)]
        L.wt_plan_shard_rows_read.argtypes = [P, C.c_int32, C.c_int32, C.POINTER(C.c_int64)]
        L.wt_plan_get_stats.argtypes = [P, C.POINTER(wt_plan_stats)]
        L.wt_prepare.argtypes = [P, P, P, P]
        L.wt_prepare_offload.argtypes = [P, P, P, P, P]
        L.wt_prepare_noalloc.argtypes = [C.POINTER(wt_plan_desc), P, P, P]
        L.wt_noalloc_check.argtypes = [P]
        L.wt_debug_noalloc_stall_unit.argtypes = [C.c_int64, C.c_uint64]
        L.wt_plan_check.argtypes = [P, P]
        L.wt_debug_fail_offload_chunk.argtypes = [P, C.c_int32]
        L.wt_debug_stall_unit.argtypes = [P, C.c_int64, C.c_uint64]
        L.wt_quantize_tokens.argtypes = [P, C.c_int64, C.c_int64, C.c_int64, P, P, P, P]
        L.wt_tokens_check.argtypes = [P]
        L.wt_debug_tokens_stall_group.argtypes = [C.c_int64, C.c_uint64]
        L.wt_plan_set_counters.argtypes = [P, P, C.c_uint32]
        L.wt_plan_expected_count.argtypes = [P, C.c_int32, C.POINTER(C.c_uint64)]
        L.wt_wait_counters.argtypes = [P, C.c_int32, P, C.c_uint64, P, P]
        L.wt_debug_e4m3_encode.argtypes = [C.c_uint32, C.c_uint64, P, P]
        L.wt_plan_destroy.argtypes = [P]
        L.wt_status_string.restype = C.c_char_p
        L.wt_status_string.argtypes = [C.c_int]
        L.wt_last_error.restype = C.c_char_p
        L.wt_last_error.argtypes = []
        for f in EXPORTS:
            if f not in ("wt_status_string", "wt_last_error"):
                getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def _check(status: int) -> None:
    if status != WT_OK:
        raise WTError(status, lib().wt_last_error().decode(errors="replace"))


def _ptr_array(ptrs):
    """A C array of device pointers; an array that is already one (see
    Plan.bind) is passed through without copying."""
    if isinstance(ptrs, C.Array):
        return ptrs
    arr = (C.c_void_p * max(1, len(ptrs)))()
    for i, p in enumerate(ptrs):
        arr[i] = int(p) if p else None
    return arr


class PlanDesc:
    """A wt_plan_desc built from a workload-like object: .params (name,
    rows, cols, shard_rows), .outputs (name, parts, fp8, dst_ranks,
    data_off, scale_off; None offsets = automatic; slices: None or per
    destination None / (dim, ((begin, length), ...))) and .num_ranks.
    local_shard >= 0 builds a shard-local plan (sets WT_FLAG_SHARD_LOCAL;
    halo=True also sets WT_FLAG_SHARD_HALO)."""

    def __init__(self, w, pool_capacity: Optional[Sequence[int]] = None,
                 offload_chunk_bytes: int = 0, flags: int = 0, local_shard: int = -1,
                 halo: bool = False):
        if local_shard >= 0:
            flags |= WT_FLAG_SHARD_LOCAL | (WT_FLAG_SHARD_HALO if halo else 0)
        keep = []
        params = (wt_param_desc * max(1, len(w.params)))()
        for i, p in enumerate(w.params):
            sr = (C.c_int64 * max(1, len(p.shard_rows)))(*p.shard_rows)
            name = p.name.encode()
            keep += [sr, name]
            params[i] = wt_param_desc(name, p.rows, p.cols, len(p.shard_rows), sr)
        outs = (wt_output_desc * max(1, len(w.outputs)))()
        for i, o in enumerate(w.outputs):
            parts = (C.c_int32 * max(1, len(o.parts)))(*o.parts)
            ranks = (C.c_int32 * max(1, len(o.dst_ranks)))(*o.dst_ranks)
            name = o.name.encode()
            keep += [parts, ranks, name]
            doff = soff = None
            if getattr(o, "data_off", None) is not None:
                doff = (C.c_uint64 * len(o.data_off))(
                    *[WT_OFFSET_AUTO if v is None else v for v in o.data_off])
                keep.append(doff)
            if getattr(o, "scale_off", None) is not None:
                soff = (C.c_uint64 * len(o.scale_off))(
                    *[WT_OFFSET_AUTO if v is None else v for v in o.scale_off])
                keep.append(soff)
            slices = None
            if getattr(o, "slices", None) is not None:
                slices = (wt_slice_desc * max(1, len(o.slices)))()
                for d, sl in enumerate(o.slices):
                    if sl is None:
                        slices[d] = wt_slice_desc(0, 0, None, None)
                        continue
                    dim, ranges = sl
                    b = (C.c_int64 * max(1, len(ranges)))(*[r[0] for r in ranges])
                    n = (C.c_int64 * max(1, len(ranges)))(*[r[1] for r in ranges])
                    keep += [b, n]
                    slices[d] = wt_slice_desc(dim, len(ranges), b, n)
                keep.append(slices)
            fmt = WT_OUT_FP8_E4M3_B128 if o.fp8 else WT_OUT_BF16
            outs[i] = wt_output_desc(name, len(o.parts), parts, fmt, len(o.dst_ranks), ranks,
                                     doff, soff, slices)
        cap = None
        if pool_capacity is not None:
            cap = (C.c_uint64 * max(1, len(pool_capacity)))(*pool_capacity)
            keep.append(cap)
        self._keep = (keep, params, outs)
        self.c = wt_plan_desc(len(w.params), params, len(w.outputs), outs, w.num_ranks, cap,
                              offload_chunk_bytes, flags, max(local_shard, 0))


# ---- entry points, same names as the C ABI ---------------------------------

def wt_plan_create(desc: PlanDesc, device: int) -> int:
    h = C.c_void_p()
    _check(lib().wt_plan_create(C.byref(desc.c), device, C.byref(h)))
    return h.value


def wt_plan_pool_bytes(plan: int, rank: int) -> int:
    v = C.c_uint64()
    _check(lib().wt_plan_pool_bytes(plan, rank, C.byref(v)))
    return v.value


def wt_plan_output_layout(plan: int, out: int, dst: int):
    r, d, s = C.c_int32(), C.c_uint64(), C.c_uint64()
    _check(lib().wt_plan_output_layout(plan, out, dst, C.byref(r), C.byref(d), C.byref(s)))
    return r.value, d.value, s.value


def wt_plan_shard_rows_read(plan: int, param: int, shard: int) -> int:
    v = C.c_int64()
    _check(lib().wt_plan_shard_rows_read(plan, param, shard, C.byref(v)))
    return v.value


def wt_plan_shard_host_offset(plan: int, param: int, shard: int) -> int:
    v = C.c_uint64()
    _check(lib().wt_plan_shard_host_offset(plan, param, shard, C.byref(v)))
    return v.value


def wt_plan_get_stats(plan: int) -> dict:
    st = wt_plan_stats()
    _check(lib().wt_plan_get_stats(plan, C.byref(st)))
    return {k: getattr(st, k) for k, _ in wt_plan_stats._fields_}


def wt_prepare(plan: int, shard_ptrs: Sequence[int], pools: Sequence[int], stream: int = 0) -> None:
    _check(lib().wt_prepare(plan, _ptr_array(shard_ptrs), _ptr_array(pools), stream or None))


def wt_prepare_offload(plan: int, host_image: int, pools: Sequence[int], copy_stream: int,
                       compute_stream: int) -> None:
    _check(lib().wt_prepare_offload(plan, host_image or None, _ptr_array(pools),
                                    copy_stream or None, compute_stream or None))


def wt_prepare_noalloc(desc: "PlanDesc", shard_ptrs: Sequence[int], pools: Sequence[int],
                       stream: int = 0) -> None:
    """One step without any device allocation (see include/wt.h): the
    schedule of `desc` is rebuilt on every call into the library's fixed
    scratch array. Calls overlapping on the GPU share that array and race."""
    _check(lib().wt_prepare_noalloc(C.byref(desc.c), _ptr_array(shard_ptrs), _ptr_array(pools),
                                    stream or None))


def wt_noalloc_check(stream: int = 0) -> None:
    """Synchronise `stream` and report (then clear) a wait that gave up in an
    earlier wt_prepare_noalloc kernel on the current device."""
    _check(lib().wt_noalloc_check(stream or None))


def wt_debug_noalloc_stall_unit(unit: int, wait_limit_ns: int = 0) -> None:
    _check(lib().wt_debug_noalloc_stall_unit(unit, wait_limit_ns))


def wt_plan_check(plan: int, stream: int = 0) -> None:
    _check(lib().wt_plan_check(plan, stream or None))


def wt_debug_fail_offload_chunk(plan: int, chunk: int) -> None:
    _check(lib().wt_debug_fail_offload_chunk(plan, chunk))


def wt_quantize_tokens(x: int, tokens: int, hidden: int, x_ld: int, codes: int, scales: int,
                       stream: int = 0, ticket: int = 0) -> None:
    """The 1 x 128 activation codec on device buffers (see include/wt.h);
    `ticket`: the address of two zeroed uint32 device words, or 0."""
    _check(lib().wt_quantize_tokens(x or None, tokens, hidden, x_ld, codes or None, scales or None,
                                    ticket or None, stream or None))


def wt_tokens_check(stream: int = 0) -> None:
    """Synchronise `stream` and report (then clear) a wait that gave up in an
    earlier wt_quantize_tokens kernel on the current device."""
    _check(lib().wt_tokens_check(stream or None))


def wt_debug_tokens_stall_group(group: int, wait_limit_ns: int = 0) -> None:
    _check(lib().wt_debug_tokens_stall_group(group, wait_limit_ns))


WT_COUNT_PER_LAUNCH = 0
WT_COUNT_PER_RANK = 1


def wt_plan_set_counters(plan: int, counters: int, mode: int = WT_COUNT_PER_LAUNCH) -> None:
    _check(lib().wt_plan_set_counters(plan, counters or None, mode))


def wt_plan_expected_count(plan: int, rank: int) -> int:
    v = C.c_uint64()
    _check(lib().wt_plan_expected_count(plan, rank, C.byref(v)))
    return v.value


def wt_wait_counters(counters: int, targets: Sequence[int], limit_ns: int, status: int,
                     stream: int = 0) -> None:
    """Queue a bounded wait until counters[i] >= targets[i] (modulo 2^32)."""
    t = (C.c_uint32 * max(1, len(targets)))(*[int(v) & 0xFFFFFFFF for v in targets])
    _check(lib().wt_wait_counters(counters or None, len(targets), t, limit_ns, status or None,
                                  stream or None))


def wt_debug_e4m3_encode(first_bits: int, n: int, codes: int, stream: int = 0) -> None:
    """The library's e4m3 convert applied to n consecutive fp32 bit patterns
    (testing hook, see include/wt.h)."""
    _check(lib().wt_debug_e4m3_encode(first_bits, n, codes or None, stream or None))


def wt_debug_stall_unit(plan: int, unit: int, wait_limit_ns: int = 0) -> None:
    _check(lib().wt_debug_stall_unit(plan, unit, wait_limit_ns))


def wt_plan_destroy(plan: int) -> None:
    _check(lib().wt_plan_destroy(plan))


def wt_status_string(status: int) -> str:
    return lib().wt_status_string(status).decode()


def wt_last_error() -> str:
    return lib().wt_last_error().decode(errors="replace")


class Plan:
    """Owning handle over a compiled plan (calls the entry points above)."""

    def __init__(self, w, device: int = 0, pool_capacity=None, offload_chunk_bytes: int = 0,
                 flags: int = 0, local_shard: int = -1, halo: bool = False):
        self.desc = PlanDesc(w, pool_capacity, offload_chunk_bytes, flags, local_shard, halo)
        self.handle = wt_plan_create(self.desc, device)
        self.num_ranks = w.num_ranks
        self.num_outputs = len(w.outputs)

    def pool_bytes(self, rank: int) -> int:
        return wt_plan_pool_bytes(self.handle, rank)

    def output_layout(self, out: int, dst: int):
        return wt_plan_output_layout(self.handle, out, dst)

    def shard_rows_read(self, param: int, shard: int) -> int:
        return wt_plan_shard_rows_read(self.handle, param, shard)

    def shard_host_offset(self, param: int, shard: int) -> int:
        return wt_plan_shard_host_offset(self.handle, param, shard)

    @property
    def stats(self) -> dict:
        return wt_plan_get_stats(self.handle)

    def bind(self, shard_ptrs, pools) -> tuple:
        """The pointer arrays of one set of buffers, built once: passing the
        result to prepare (as prepare(*plan.bind(...), stream)) skips the
        per-call conversion of thousands of Python integers."""
        return _ptr_array(shard_ptrs), _ptr_array(pools)

    def prepare(self, shard_ptrs, pools, stream: int = 0) -> None:
        wt_prepare(self.handle, shard_ptrs, pools, stream)

    def prepare_offload(self, host_image: int, pools, copy_stream: int, compute_stream: int):
        wt_prepare_offload(self.handle, host_image, pools, copy_stream, compute_stream)

    def check(self, stream: int = 0) -> None:
        wt_plan_check(self.handle, stream)

    def set_counters(self, counters: int, mode: int = WT_COUNT_PER_LAUNCH) -> None:
        wt_plan_set_counters(self.handle, counters, mode)

    def expected_count(self, rank: int) -> int:
        return wt_plan_expected_count(self.handle, rank)

    def close(self) -> None:
        if self.handle:
            h, self.handle = self.handle, None
            wt_plan_destroy(h)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
