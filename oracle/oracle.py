"""ctypes wrapper around the C oracle (wt_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use it; the product library never does. The oracle takes
the same workload descriptor as the library but lays it out, reassembles,
fuses and quantizes with its own code.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wt_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")

OFFSET_AUTO = 2**64 - 1


def build(force: bool = False) -> str:
    """Compile the oracle with plain IEEE arithmetic (no contraction, no
    fast-math) into oracle/liboracle.so."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "wt_oracle.h"))):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off",
                               "-fno-fast-math", "-fPIC", "-shared", "-pthread", "-o", tmp,
                               _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class _Param(C.Structure):
    _fields_ = [("rows", C.c_int64), ("cols", C.c_int64), ("num_shards", C.c_int32),
                ("shard_rows", C.POINTER(C.c_int64))]


class _Slice(C.Structure):
    _fields_ = [("dim", C.c_int32), ("num_ranges", C.c_int32),
                ("begin", C.POINTER(C.c_int64)), ("length", C.POINTER(C.c_int64))]


class _Output(C.Structure):
    _fields_ = [("num_parts", C.c_int32), ("parts", C.POINTER(C.c_int32)),
                ("fp8", C.c_int32), ("num_dsts", C.c_int32),
                ("dst_rank", C.POINTER(C.c_int32)),
                ("data_off", C.POINTER(C.c_uint64)), ("scale_off", C.POINTER(C.c_uint64)),
                ("dst_slice", C.POINTER(_Slice))]


class _Model(C.Structure):
    _fields_ = [("num_params", C.c_int32), ("params", C.POINTER(_Param)),
                ("num_outputs", C.c_int32), ("outputs", C.POINTER(_Output)),
                ("num_ranks", C.c_int32)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        L.wo_e4m3_encode.restype = C.c_uint8
        L.wo_e4m3_encode.argtypes = [C.c_float]
        L.wo_e4m3_decode.restype = C.c_double
        L.wo_e4m3_decode.argtypes = [C.c_uint8]
        L.wo_e4m3_encode_array.argtypes = [C.c_void_p, C.c_void_p, C.c_int64]
        L.wo_e4m3_encode_bits_range.argtypes = [C.c_uint32, C.c_int64, C.c_void_p]
        L.wo_bf16_value.restype = C.c_float
        L.wo_bf16_value.argtypes = [C.c_uint16]
        L.wo_tile_scale.restype = C.c_float
        L.wo_tile_scale.argtypes = [C.c_float]
        L.wo_quantize_element.restype = C.c_uint8
        L.wo_quantize_element.argtypes = [C.c_uint16, C.c_float]
        L.wo_output_shape.argtypes = [C.POINTER(_Model), C.c_int32, C.POINTER(C.c_int64),
                                      C.POINTER(C.c_int64)]
        L.wo_dst_shape.argtypes = [C.POINTER(_Model), C.c_int32, C.c_int32,
                                   C.POINTER(C.c_int64), C.POINTER(C.c_int64)]
        L.wo_layout.argtypes = [C.POINTER(_Model), C.c_void_p, C.c_void_p, C.c_void_p]
        L.wo_prepare_output.argtypes = [C.POINTER(_Model), C.c_int32, C.c_void_p, C.c_void_p,
                                        C.c_void_p]
        L.wo_prepare.argtypes = [C.POINTER(_Model), C.c_void_p, C.c_void_p, C.c_void_p,
                                 C.c_void_p, C.c_int32]
        L.wo_quantize_tokens.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_int64,
                                         C.c_void_p, C.c_void_p]
        L.wo_expected_blocks.restype = C.c_int64
        L.wo_expected_blocks.argtypes = [C.POINTER(_Model), C.c_int32]
        _lib = L
    return _lib


# --------------------------------------------------------------------------
# element-level entry points
# --------------------------------------------------------------------------

def e4m3_encode(y) -> np.ndarray:
    y = np.ascontiguousarray(np.asarray(y, dtype=np.float32))
    out = np.empty(y.shape, dtype=np.uint8)
    lib().wo_e4m3_encode_array(y.ctypes.data, out.ctypes.data, y.size)
    return out


def e4m3_encode_bits_range(first: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint8)
    lib().wo_e4m3_encode_bits_range(first, n, out.ctypes.data)
    return out


def e4m3_decode(code: int) -> float:
    return lib().wo_e4m3_decode(code)


def tile_scale(amax: float) -> np.float32:
    return np.float32(lib().wo_tile_scale(float(amax)))


def quantize_element(x_bits: int, s) -> int:
    return lib().wo_quantize_element(int(x_bits), float(np.float32(s)))


def quantize_tokens(x_bits: np.ndarray, hidden: int = None):
    """(codes, scales) of the 1 x 128 activation codec for a 2-D uint16 BF16
    array (rows are tokens; a strided view is honoured through its row
    stride)."""
    assert x_bits.dtype == np.uint16 and x_bits.ndim == 2 and x_bits.strides[1] == 2
    tokens, h = x_bits.shape
    hidden = h if hidden is None else hidden
    ld = x_bits.strides[0] // 2
    codes = np.empty((tokens, hidden), np.uint8)
    scales = np.empty((tokens, -(-hidden // 128)), np.float32)
    lib().wo_quantize_tokens(x_bits.ctypes.data, tokens, hidden, ld, codes.ctypes.data,
                             scales.ctypes.data)
    return codes, scales


# --------------------------------------------------------------------------
# model-level entry points
# --------------------------------------------------------------------------

class Model:
    """The oracle's own C descriptor built from a workloads.Workload."""

    def __init__(self, w):
        self.w = w
        self._keep = []
        params = (_Param * max(1, len(w.params)))()
        for i, p in enumerate(w.params):
            sr = (C.c_int64 * max(1, len(p.shard_rows)))(*p.shard_rows)
            self._keep.append(sr)
            params[i] = _Param(p.rows, p.cols, len(p.shard_rows), sr)
        outs = (_Output * max(1, len(w.outputs)))()
        for i, o in enumerate(w.outputs):
            parts = (C.c_int32 * len(o.parts))(*o.parts)
            ranks = (C.c_int32 * max(1, len(o.dst_ranks)))(*o.dst_ranks)
            self._keep += [parts, ranks]
            doff = soff = None
            if o.data_off is not None:
                doff = (C.c_uint64 * len(o.dst_ranks))(
                    *[OFFSET_AUTO if v is None else v for v in o.data_off])
                self._keep.append(doff)
            if o.scale_off is not None:
                soff = (C.c_uint64 * len(o.dst_ranks))(
                    *[OFFSET_AUTO if v is None else v for v in o.scale_off])
                self._keep.append(soff)
            slices = None
            if getattr(o, "slices", None) is not None:
                slices = (_Slice * len(o.dst_ranks))()
                for d, sl in enumerate(o.slices):
                    if sl is None:
                        slices[d] = _Slice(0, 0, None, None)
                        continue
                    dim, ranges = sl
                    b = (C.c_int64 * len(ranges))(*[r[0] for r in ranges])
                    n = (C.c_int64 * len(ranges))(*[r[1] for r in ranges])
                    self._keep += [b, n]
                    slices[d] = _Slice(dim, len(ranges), b, n)
                self._keep.append(slices)
            outs[i] = _Output(len(o.parts), parts, int(bool(o.fp8)), len(o.dst_ranks), ranks,
                              doff, soff, slices)
        self._params, self._outs = params, outs
        self.c = _Model(len(w.params), params, len(w.outputs), outs, w.num_ranks)
        self.num_dsts = sum(len(o.dst_ranks) for o in w.outputs)

    def dst_shape(self, o: int, d: int) -> tuple:
        """(rows, cols) that destination d of output o holds."""
        r, c = C.c_int64(), C.c_int64()
        if lib().wo_dst_shape(C.byref(self.c), o, d, C.byref(r), C.byref(c)):
            raise ValueError("oracle: invalid slice")
        return r.value, c.value

    def expected_blocks(self, rank: int) -> int:
        """Blocks landing at `rank` per step (its completion counter's step)."""
        v = lib().wo_expected_blocks(C.byref(self.c), rank)
        if v < 0:
            raise ValueError("oracle: invalid model")
        return int(v)

    def layout(self):
        """(data_off, scale_off) as lists per output of per-destination
        offsets, and the per-rank pool sizes."""
        n = max(1, self.num_dsts)
        doff = np.zeros(n, np.uint64)
        soff = np.zeros(n, np.uint64)
        pools = np.zeros(max(1, self.w.num_ranks), np.uint64)
        if lib().wo_layout(C.byref(self.c), doff.ctypes.data, soff.ctypes.data,
                           pools.ctypes.data):
            raise ValueError("oracle: invalid model")
        d, s, k = [], [], 0
        for o in self.w.outputs:
            d.append([int(v) for v in doff[k:k + len(o.dst_ranks)]])
            s.append([int(v) for v in soff[k:k + len(o.dst_ranks)]])
            k += len(o.dst_ranks)
        return d, s, [int(v) for v in pools[:self.w.num_ranks]]

    def _shard_table(self, flat_shards):
        tbl = (C.c_void_p * max(1, len(flat_shards)))()
        for i, a in enumerate(flat_shards):
            if a is not None:
                assert a.dtype == np.uint16 and a.flags.c_contiguous
                tbl[i] = a.ctypes.data
        return tbl

    def prepare_output(self, o: int, flat_shards):
        """(data bytes, scales) of output o; flat_shards is param-major,
        then shard (None for params output o does not use)."""
        m, n = self.w.output_shape(o)
        fp8 = self.w.outputs[o].fp8
        data = np.empty(m * n * (1 if fp8 else 2), np.uint8)
        scales = np.empty(max(1, (-(-m // 128)) * (-(-n // 128))) if fp8 else 1, np.float32)
        tbl = self._shard_table(flat_shards)
        if lib().wo_prepare_output(C.byref(self.c), o, tbl, data.ctypes.data,
                                   scales.ctypes.data):
            raise RuntimeError("oracle: prepare_output failed")
        return data, (scales if fp8 else None)

    def prepare(self, flat_shards, nthreads: int = 1, fill: int = 0):
        """Every destination pool as a host uint8 array (pool bytes, padding
        filled with `fill`)."""
        d, s, pool_bytes = self.layout()
        doff = np.array([v for per in d for v in per] or [0], np.uint64)
        soff = np.array([v for per in s for v in per] or [0], np.uint64)
        pools = [np.full(max(1, b), fill, np.uint8) for b in pool_bytes]
        ptbl = (C.c_void_p * max(1, len(pools)))(*[p.ctypes.data for p in pools])
        tbl = self._shard_table(flat_shards)
        if lib().wo_prepare(C.byref(self.c), doff.ctypes.data, soff.ctypes.data, tbl, ptbl,
                            nthreads):
            raise RuntimeError("oracle: prepare failed")
        return [p[:b] for p, b in zip(pools, pool_bytes)]
