// The preparation kernel: one pass over the static schedule's 128x128 work
// units. Each unit reassembles one block of a fused output from its FSDP
// shards (row gather), and either quantises it to e4m3 with one fp32 scale
// (block amax / 448) or passes the BF16 bytes through, then stores it at
// every destination of that output.
//
// Method: "Weight transfer for RL post-training in under 2 seconds",
// section "Task pipeline" (rebuild with full_tensor(), projection fusion,
// quantize if needed) and section "DeviceMesh and mesh groups" (dim-0 FSDP
// shards). FP8 = e4m3 "fn", RNE, saturating; scale = amax / 448 as an IEEE
// binary32 division, 1.0 for an all-zero block; code = e4m3(fl32(x / scale)).
//
// Mapping. A CTA of 256 threads owns one unit at a time (persistent grid,
// units strided by gridDim.x). Thread t owns the 16-byte column chunk
// t % 16 of the rows t / 16 + 16 i, i = 0..7, so a warp reads two full
// 256-byte block rows per load instruction and the block stays in
// registers between the amax and the quantisation (one HBM read per byte).
//
// Pipelining. Warp 0 fetches the 32-byte descriptor of the unit two steps
// ahead and the source / destination addresses of the unit one step ahead,
// and publishes them in a shared-memory ring before the per-unit barrier,
// so no thread waits on a dependent metadata load. The data loads of the
// next unit are issued as soon as the current unit's codes are computed,
// so they are in flight while the current unit is being stored.
//
// Division. The code of x must be E(fl32(x / s)). Dividing every element
// is an ALU-heavy sequence, so the kernel brackets the quotient instead:
// with r = RN(1/s), rlo = RN(r (1 - 2^-21)) and rhi = RN(r (1 + 2^-21)),
// ylo = RN(x rlo) and yhi = RN(x rhi) satisfy |ylo| < |fl32(x/s)| < |yhi|
// whenever the values are normal (each RN adds a relative error of at
// most 2^-24, five of them stay below the 2^-21 margin), and all three
// share the sign of x. E is monotone in |y|, so when E(ylo) == E(yhi) that
// code is E(fl32(x/s)). Otherwise (a rounding boundary of E lies inside
// the bracket, about once per 2^17 elements, or exactly on a tie) the
// chunk is recomputed with the IEEE division. Subnormal results are far
// below the smallest e4m3 step and encode to a signed zero on every path.
// Blocks whose scale or reciprocal would be subnormal use the IEEE
// division throughout.
#include <cuda_fp8.h>

#include "plan.h"

namespace wt {
namespace {

constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerThread = kTile * kTile / 8 / kThreads;   // 8
constexpr int kMetaSlots = 4;
constexpr unsigned kFull = 0xFFFFFFFFu;

// Shared-memory metadata slot (16 words):
//   0..7   the unit's DevUnit
//   8, 9   source address of its block row (one-shard rows)
//   10..13 data and scale addresses of its first destination
constexpr int kMetaWords = 16;

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_meta_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// max(|a|, |b|) per bf16 half; the sign bits of the result are meaningless
// (xorsign), only magnitudes are kept.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two e4m3 codes (first value in the low byte), RNE, satfinite.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// 8 BF16 elements (one 16-byte chunk) -> 8 codes with the IEEE division.
__device__ __noinline__ uint2 quant_chunk_exact(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    c[k] = e4m3x2(__fdiv_rn(bf16_lo(w[k]), s), __fdiv_rn(bf16_hi(w[k]), s));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// The bracketed version; returns false if any of the 8 codes is uncertain.
__device__ __forceinline__ bool quant_chunk_bracket(const uint4& v, float rlo, float rhi, uint2& out) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4], diff = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float x0 = bf16_lo(w[k]), x1 = bf16_hi(w[k]);
    const uint32_t clo = e4m3x2(x0 * rlo, x1 * rlo);
    const uint32_t chi = e4m3x2(x0 * rhi, x1 * rhi);
    diff |= clo ^ chi;
    c[k] = clo;
  }
  out = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  return diff == 0;
}

// Per-thread view of one unit's metadata (read from the shared ring).
struct Meta {
  uint32_t bi, bj, N, shape, num_dsts, dst_begin, gtr;
  const uint16_t* src;
  uint8_t* dst0;
  float* scale0;
  __device__ __forceinline__ int nrows() const { return (int)(shape & 0xFFu) + 1; }
  __device__ __forceinline__ int ncols() const { return (int)((shape >> 8) & 0xFFu) + 1; }
  __device__ __forceinline__ uint32_t flags() const { return shape >> 16; }
};

__device__ __forceinline__ Meta read_meta(const uint32_t* s) {
  const uint4 a = *reinterpret_cast<const uint4*>(s);
  const uint4 b = *reinterpret_cast<const uint4*>(s + 4);
  const uint4 c = *reinterpret_cast<const uint4*>(s + 8);
  const uint4 d = *reinterpret_cast<const uint4*>(s + 12);
  Meta m;
  m.gtr = a.y;
  m.bi = a.z;
  m.bj = a.w;
  m.N = b.x;
  m.shape = b.y;
  m.num_dsts = b.z;
  m.dst_begin = b.w;
  m.src = reinterpret_cast<const uint16_t*>(((uint64_t)c.y << 32) | c.x);
  m.dst0 = reinterpret_cast<uint8_t*>(((uint64_t)c.w << 32) | c.z);
  m.scale0 = reinterpret_cast<float*>(((uint64_t)d.y << 32) | d.x);
  return m;
}

// Warp 0, lanes 0..7: word `lane` of the descriptor of unit u (0 past the end).
__device__ __forceinline__ uint32_t fetch_unit_word(const PrepArgs& a, int64_t u, int lane) {
  if (lane >= 8 || u >= a.unit_end) return 0;
  return ld_meta_u32(reinterpret_cast<const uint32_t*>(a.units + u) + lane);
}

// Warp 0, lanes 8..13: the dynamic words of the unit whose descriptor words
// lanes 0..7 hold in w.
__device__ __forceinline__ uint32_t fetch_dyn_word(const PrepArgs& a, uint32_t w, int lane, bool valid) {
  const uint32_t gtr = __shfl_sync(kFull, w, 1);
  const uint32_t dst_begin = __shfl_sync(kFull, w, 7);
  if (!valid) return 0;
  if (lane == 8 || lane == 9)
    return ld_meta_u32(reinterpret_cast<const uint32_t*>(a.trow_src + gtr) + (lane - 8));
  if (lane >= 10 && lane < 14)
    return ld_meta_u32(reinterpret_cast<const uint32_t*>(a.dst_ptrs + dst_begin) + (lane - 10));
  return 0;
}

template <bool kDebug>
__device__ __forceinline__ bool store_ok(const PrepArgs& a, const Meta& m, int d, const void* p, uint64_t n) {
  if (!kDebug) return true;
  const DevDstPtr& dp = a.dst_ptrs[m.dst_begin + d];
  const uint8_t* q = static_cast<const uint8_t*>(p);
  if (q >= dp.pool_begin && q + n <= dp.pool_end) return true;
  atomicExch(a.error_word, 1);
  return false;
}

// Issue the loads of a unit's block into v. Blocks whose rows span several
// shards first resolve each row's address into shared memory (barrier).
__device__ __forceinline__ void load_unit(const PrepArgs& a, const Meta& m, uint4 (&v)[kRowsPerThread],
                                          const uint16_t** s_rowptr, int tid, int cc, int rsub) {
  const int nrows = m.nrows(), ncols = m.ncols();
  const uint32_t f = m.flags();
  const int64_t N = m.N;
  const bool vec = f & kUnitVec;
  if (f & kUnitMulti) {
    // row gather over several runs (the full_tensor() stand-in)
    if (tid < kTile) {
      const uint16_t* ptr = nullptr;
      if (tid < nrows) {
        const int64_t fr = (int64_t)m.bi * kTile + tid;
        int k = a.trow_first_run[m.gtr];
        while (fr >= a.runs[k].row0 + a.runs[k].rows) ++k;
        const DevRun run = a.runs[k];
        ptr = a.shard_ptrs[run.slot] + (fr - run.row0) * N;
      }
      s_rowptr[tid] = ptr;
    }
    __syncthreads();
  }
  const int64_t col = (int64_t)m.bj * kTile + cc * 8;
  const uint16_t* base = m.src + (int64_t)rsub * N + col;
  const int64_t rstep = 16 * N;
  if (vec) {
    const bool col_ok = cc * 8 < ncols;
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int r = rsub + 16 * i;
      v[i] = make_uint4(0, 0, 0, 0);
      if (r < nrows && col_ok) {
        const uint16_t* p = (f & kUnitMulti) ? s_rowptr[r] + col : base + i * rstep;
        v[i] = ld_stream_v4(p);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
      const int r = rsub + 16 * i;
      uint16_t e[8];
      const uint16_t* p = nullptr;
      if (r < nrows) p = (f & kUnitMulti) ? s_rowptr[r] + col : base + i * rstep;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        e[j] = 0;
        if (r < nrows && cc * 8 + j < ncols) e[j] = ld_stream_u16(p + j);
      }
      v[i] = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16),
                        e[4] | ((uint32_t)e[5] << 16), e[6] | ((uint32_t)e[7] << 16));
    }
  }
}

template <bool kDebug>
__device__ __forceinline__ void store_fp8(const PrepArgs& a, const Meta& m,
                                          const uint2 (&q)[kRowsPerThread], float s, int tid,
                                          int cc, int rsub) {
  const int nrows = m.nrows(), ncols = m.ncols();
  const int64_t N = m.N;
  const bool vec = m.flags() & kUnitVec;
  const int64_t off0 = ((int64_t)m.bi * kTile + rsub) * N + (int64_t)m.bj * kTile + cc * 8;
  const int64_t rstep = 16 * N;
  const uint32_t tiles_n = (m.N + kTile - 1) / kTile;
  for (int d = 0; d < (int)m.num_dsts; ++d) {
    uint8_t* data = m.dst0;
    float* scale = m.scale0;
    if (d > 0) {
      const DevDstPtr dp = a.dst_ptrs[m.dst_begin + d];
      data = dp.data;
      scale = dp.scale;
    }
    if (tid == 0) {
      float* sp = scale + (uint64_t)m.bi * tiles_n + m.bj;
      if (store_ok<kDebug>(a, m, d, sp, 4)) *sp = s;
    }
    uint8_t* row = data + off0;
    if (vec) {
      const bool col_ok = cc * 8 < ncols;
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        uint8_t* p = row + i * rstep;
        if (rsub + 16 * i < nrows && col_ok && store_ok<kDebug>(a, m, d, p, 8))
          *reinterpret_cast<uint2*>(p) = q[i];
      }
    } else {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const uint32_t wds[2] = {q[i].x, q[i].y};
        uint8_t* p = row + i * rstep;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (rsub + 16 * i < nrows && cc * 8 + j < ncols && store_ok<kDebug>(a, m, d, p + j, 1))
            p[j] = (uint8_t)(wds[j >> 2] >> (8 * (j & 3)));
      }
    }
  }
}

template <bool kDebug>
__device__ __forceinline__ void store_bf16(const PrepArgs& a, const Meta& m,
                                           const uint4 (&v)[kRowsPerThread], int cc, int rsub) {
  const int nrows = m.nrows(), ncols = m.ncols();
  const int64_t N = m.N;
  const bool vec = m.flags() & kUnitVec;
  const int64_t off0 = 2 * (((int64_t)m.bi * kTile + rsub) * N + (int64_t)m.bj * kTile + cc * 8);
  const int64_t rstep = 32 * N;
  for (int d = 0; d < (int)m.num_dsts; ++d) {
    uint8_t* data = d == 0 ? m.dst0 : a.dst_ptrs[m.dst_begin + d].data;
    uint8_t* row = data + off0;
    if (vec) {
      const bool col_ok = cc * 8 < ncols;
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        uint8_t* p = row + i * rstep;
        if (rsub + 16 * i < nrows && col_ok && store_ok<kDebug>(a, m, d, p, 16))
          *reinterpret_cast<uint4*>(p) = v[i];
      }
    } else {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const uint32_t wds[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint8_t* p = row + i * rstep;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (rsub + 16 * i < nrows && cc * 8 + j < ncols && store_ok<kDebug>(a, m, d, p + 2 * j, 2))
            *reinterpret_cast<uint16_t*>(p + 2 * j) = (uint16_t)(wds[j >> 1] >> (16 * (j & 1)));
      }
    }
  }
}

template <bool kDebug>
__global__ void __launch_bounds__(kThreads, 3) prep_kernel(const PrepArgs a) {
  __shared__ __align__(16) uint32_t s_meta[kMetaSlots][kMetaWords];
  __shared__ const uint16_t* s_rowptr[kTile];
  __shared__ float s_wmax[2][kWarps];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int cc = tid & 15;            // 16-byte column chunk within the block
  const int rsub = tid >> 4;          // first row within the block
  const int64_t G = gridDim.x;

  int64_t u = a.unit_begin + blockIdx.x;
  if (u >= a.unit_end) return;
  // descriptor words (lanes 0..7 of warp 0) of the units one and two ahead
  uint32_t wa = 0, wb = 0;
  if (warp == 0) {
    const uint32_t w0 = fetch_unit_word(a, u, lane);
    const uint32_t d0 = fetch_dyn_word(a, w0, lane, true);
    if (lane < 14) s_meta[0][lane] = lane < 8 ? w0 : d0;
    wa = fetch_unit_word(a, u + G, lane);
    wb = fetch_unit_word(a, u + 2 * G, lane);
  }
  __syncthreads();
  uint4 v[kRowsPerThread];
  load_unit(a, read_meta(s_meta[0]), v, s_rowptr, tid, cc, rsub);

  for (int n = 0;; ++n) {
    const int slot = n & (kMetaSlots - 1), nslot = (n + 1) & (kMetaSlots - 1);
    const int buf = n & 1;
    const int64_t un = u + G;
    const bool has_next = un < a.unit_end;
    uint32_t dn = 0;
    if (warp == 0) dn = fetch_dyn_word(a, wa, lane, has_next);
    const uint32_t flags = s_meta[slot][5] >> 16;
    if (flags & kUnitFp8) {
      // block amax: per thread, then warp shuffle, then across warps
      uint32_t m2 = 0;
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        m2 = absmax_bf16x2(m2, v[i].x);
        m2 = absmax_bf16x2(m2, v[i].y);
        m2 = absmax_bf16x2(m2, v[i].z);
        m2 = absmax_bf16x2(m2, v[i].w);
      }
      m2 &= 0x7FFF7FFFu;
      float mx = fmaxf(bf16_lo(m2), bf16_hi(m2));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
      if (warp == 0) {
        if (lane < 14) s_meta[nslot][lane] = lane < 8 ? wa : dn;
        wa = wb;
        wb = fetch_unit_word(a, un + 2 * G, lane);
      }
      if (lane == 0) s_wmax[buf][warp] = mx;
      __syncthreads();
      float amax = s_wmax[buf][0];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, s_wmax[buf][w]);
      const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
      const uint32_t se = (__float_as_uint(s) >> 23) & 0xFFu;
      uint2 q[kRowsPerThread];
      if (se >= 1u && se <= 252u) {           // s and 1/s normal: bracketed path
        const float r = __frcp_rn(s);
        const float rlo = r * (1.0f - 0x1p-21f), rhi = r * (1.0f + 0x1p-21f);
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i)
          if (!quant_chunk_bracket(v[i], rlo, rhi, q[i])) q[i] = quant_chunk_exact(v[i], s);
      } else {
#pragma unroll
        for (int i = 0; i < kRowsPerThread; ++i) q[i] = quant_chunk_exact(v[i], s);
      }
      if (has_next) load_unit(a, read_meta(s_meta[nslot]), v, s_rowptr, tid, cc, rsub);
      store_fp8<kDebug>(a, read_meta(s_meta[slot]), q, s, tid, cc, rsub);
    } else {
      if (warp == 0) {
        if (lane < 14) s_meta[nslot][lane] = lane < 8 ? wa : dn;
        wa = wb;
        wb = fetch_unit_word(a, un + 2 * G, lane);
      }
      __syncthreads();
      store_bf16<kDebug>(a, read_meta(s_meta[slot]), v, cc, rsub);
      if (has_next) load_unit(a, read_meta(s_meta[nslot]), v, s_rowptr, tid, cc, rsub);
    }
    if (!has_next) break;
    u = un;
  }
}

}  // namespace

int prep_blocks_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, prep_kernel<false>, kThreads, 0) != cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

cudaError_t launch_prepare(const PrepArgs& a, int grid, cudaStream_t s, bool debug) {
  if (a.unit_end <= a.unit_begin) return cudaSuccess;
  if (debug)
    prep_kernel<true><<<grid, kThreads, 0, s>>>(a);
  else
    prep_kernel<false><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace wt
