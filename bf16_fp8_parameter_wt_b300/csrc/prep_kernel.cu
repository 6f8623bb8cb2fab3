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
// binary32 division, 1.0 for an all-zero block; code = e4m3(x / scale)
// with an IEEE binary32 division per element.
//
// Mapping: a CTA of 256 threads owns one unit at a time (persistent grid,
// units strided by gridDim.x). Thread t owns the 16-byte column chunk
// t % 16 of the rows t / 16 + 16 i, i = 0..7, so a warp reads two full
// 256-byte block rows per load instruction and the block stays in
// registers between the amax and the quantisation (one HBM read per byte).
#include <cuda_fp8.h>

#include "plan.h"

namespace wt {
namespace {

constexpr int kRowsPerThread = kTile * kTile / 8 / kThreads;   // 8

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

// max(|a|, |b|) per bf16 half; the sign bits of the result are meaningless
// (xorsign), only magnitudes are kept.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two BF16 elements (low half first) -> two e4m3 codes (low byte first).
__device__ __forceinline__ uint32_t quant_pair(uint32_t w, float s) {
  const float y0 = __fdiv_rn(bf16_lo(w), s);
  const float y1 = __fdiv_rn(bf16_hi(w), s);
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
}

// 8 BF16 elements (one 16-byte chunk) -> 8 codes.
__device__ __forceinline__ uint2 quant_chunk(const uint4& v, float s) {
  uint2 r;
  r.x = quant_pair(v.x, s) | (quant_pair(v.y, s) << 16);
  r.y = quant_pair(v.z, s) | (quant_pair(v.w, s) << 16);
  return r;
}

template <bool kDebug>
__device__ __forceinline__ bool store_ok(const PrepArgs& a, int rank, uint64_t off, uint64_t n) {
  if (!kDebug) return true;
  if (off + n <= a.pool_bytes[rank]) return true;
  atomicExch(a.error_word, 1);
  return false;
}

template <bool kDebug>
__global__ void __launch_bounds__(kThreads, 3) prep_kernel(const PrepArgs a) {
  __shared__ const uint16_t* s_rowptr[2][kTile];
  __shared__ float s_wmax[2][kThreads / 32];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int cc = tid & 15;            // 16-byte column chunk within the block
  const int rsub = tid >> 4;          // first row within the block
  int buf = 0;

  for (int64_t u = a.unit_begin + blockIdx.x; u < a.unit_end; u += gridDim.x, buf ^= 1) {
    const uint32_t o = a.unit_out[u];
    const DevOutput out = a.outs[o];
    const int64_t t = u - out.unit_begin;
    const int64_t bi = t / out.tiles_n, bj = t - bi * out.tiles_n;
    const int64_t r0 = bi * kTile, c0 = bj * kTile;
    const int nrows = (int)(out.rows - r0 < kTile ? out.rows - r0 : kTile);
    const int ncols = (int)(out.cols - c0 < kTile ? out.cols - c0 : kTile);
    const int64_t N = out.cols;

    // row gather: the source address of each of the block's rows
    if (tid < kTile) {
      const uint16_t* ptr = nullptr;
      if (tid < nrows) {
        const int64_t row = r0 + tid;
        int k = a.trow_first_run[out.trow_begin + bi];
        while (row >= a.runs[k].row0 + a.runs[k].rows) ++k;
        const DevRun run = a.runs[k];
        ptr = a.shard_ptrs[run.slot] + (row - run.row0) * N + c0;
      }
      s_rowptr[buf][tid] = ptr;
    }
    __syncthreads();

    // load the block: 8 rows x 16 bytes per thread
    uint4 v[kRowsPerThread];
    const bool col_ok = cc * 8 < ncols;
    if (out.vec) {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int r = rsub + 16 * i;
        v[i] = make_uint4(0, 0, 0, 0);
        if (r < nrows && col_ok) v[i] = ld_stream_v4(s_rowptr[buf][r] + cc * 8);
      }
    } else {
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) {
        const int r = rsub + 16 * i;
        uint16_t e[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          e[j] = 0;
          if (r < nrows && cc * 8 + j < ncols) e[j] = ld_stream_u16(s_rowptr[buf][r] + cc * 8 + j);
        }
        v[i].x = e[0] | ((uint32_t)e[1] << 16);
        v[i].y = e[2] | ((uint32_t)e[3] << 16);
        v[i].z = e[4] | ((uint32_t)e[5] << 16);
        v[i].w = e[6] | ((uint32_t)e[7] << 16);
      }
    }

    const DevDst* dsts = a.dsts + out.dst_begin;
    if (out.fp8) {
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
      float m = fmaxf(bf16_lo(m2), bf16_hi(m2));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
      if (lane == 0) s_wmax[buf][warp] = m;
      __syncthreads();
      float amax = s_wmax[buf][0];
#pragma unroll
      for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, s_wmax[buf][w]);
      const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);

      uint2 q[kRowsPerThread];
#pragma unroll
      for (int i = 0; i < kRowsPerThread; ++i) q[i] = quant_chunk(v[i], s);

      for (int d = 0; d < out.num_dsts; ++d) {
        const DevDst ds = dsts[d];
        uint8_t* pool = a.pool_ptrs[ds.rank];
        if (tid == 0) {
          const uint64_t so = ds.scale_off + (uint64_t)(bi * out.tiles_n + bj) * 4u;
          if (store_ok<kDebug>(a, ds.rank, so, 4)) *reinterpret_cast<float*>(pool + so) = s;
        }
        if (out.vec) {
#pragma unroll
          for (int i = 0; i < kRowsPerThread; ++i) {
            const int r = rsub + 16 * i;
            if (r < nrows && col_ok) {
              const uint64_t off = ds.data_off + (uint64_t)((r0 + r) * N + c0 + cc * 8);
              if (store_ok<kDebug>(a, ds.rank, off, 8)) *reinterpret_cast<uint2*>(pool + off) = q[i];
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < kRowsPerThread; ++i) {
            const int r = rsub + 16 * i;
            const uint32_t wds[2] = {q[i].x, q[i].y};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (r < nrows && cc * 8 + j < ncols) {
                const uint64_t off = ds.data_off + (uint64_t)((r0 + r) * N + c0 + cc * 8 + j);
                if (store_ok<kDebug>(a, ds.rank, off, 1)) pool[off] = (uint8_t)(wds[j >> 2] >> (8 * (j & 3)));
              }
            }
          }
        }
      }
    } else {
      // BF16 pass-through
      for (int d = 0; d < out.num_dsts; ++d) {
        const DevDst ds = dsts[d];
        uint8_t* pool = a.pool_ptrs[ds.rank];
        if (out.vec) {
#pragma unroll
          for (int i = 0; i < kRowsPerThread; ++i) {
            const int r = rsub + 16 * i;
            if (r < nrows && col_ok) {
              const uint64_t off = ds.data_off + 2u * (uint64_t)((r0 + r) * N + c0 + cc * 8);
              if (store_ok<kDebug>(a, ds.rank, off, 16)) *reinterpret_cast<uint4*>(pool + off) = v[i];
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < kRowsPerThread; ++i) {
            const int r = rsub + 16 * i;
            const uint32_t wds[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (r < nrows && cc * 8 + j < ncols) {
                const uint64_t off = ds.data_off + 2u * (uint64_t)((r0 + r) * N + c0 + cc * 8 + j);
                if (store_ok<kDebug>(a, ds.rank, off, 2))
                  *reinterpret_cast<uint16_t*>(pool + off) = (uint16_t)(wds[j >> 1] >> (16 * (j & 1)));
              }
            }
          }
        }
      }
    }
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
