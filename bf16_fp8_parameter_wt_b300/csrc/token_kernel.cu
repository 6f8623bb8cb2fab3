// The activation codec of the MoE dispatch: tokens x hidden BF16 ->
// e4m3 codes with one fp32 scale per token per group of 128 channels
// ("Enabling trillion-parameter models on AWS EFA", section on the
// dispatch/combine kernels: block-scaled FP8 dispatch at hidden 7168), with
// the weight path's scale and code (codec.cuh).
//
// Two kernels, one arithmetic. In both, four lanes own one group of 128
// channels, each lane four 16-byte chunks of it; the group's amax is a
// two-step shuffle, and its scale and reciprocal are computed once per 32
// elements of a lane.
//
// Large batches of 16-byte-aligned rows with hidden a multiple of 128 go
// through a TMA ring: the batch's groups, in token order, are cut into
// stages of 128 groups (32 KiB; the last may be shorter), each copied with
// one bulk copy when rows are contiguous (x_ld == hidden), else one per
// token row it touches (rows of at least 32 groups). A producer warp per
// CTA (one CTA per SM) copies stages into a ring of shared-memory slots
// with cp.async.bulk and tells the consumers which stage each slot holds;
// two consumer groups of twelve warps take alternate slots, quantise from
// shared memory and store codes and scales straight to global memory. With
// a caller's ticket counter the producers of a contiguous batch take
// stages from it one at a time, each ticket a stage ahead (SMs that are
// served faster take more; the last CTA resets it), six slots deep;
// otherwise CTA b takes stages b, b + gridDim.x, ..., four slots deep (a
// deeper ring measured slower with the fixed hand-out). Lane l of group j
// reads chunk 4 ((c + j) mod 4) + l % 4 at step c, so that the two groups
// in each 8-lane phase of a 16-byte shared load fall in different bank
// halves. Every wait is bounded; the role that gives up records
// kErrTimeout in the codec's error word (wt_tokens_check).
//
// Smaller batches, and all other shapes (hidden not a multiple of 128,
// short strided rows, unaligned x), use a register-streaming kernel, which
// starts faster than the ring fills: each lane loads its chunks of four
// groups straight into registers (chunk c of lane l is chunk 4c + l % 4 of
// the group, so each load instruction reads whole 64-byte runs and each
// store writes whole 32-byte sectors); contiguous batches index groups as
// one flat sequence (no division), and rows that are not 16-byte aligned
// are read and written element by element. Loops are warp-uniform so the
// shuffles never see an exited lane.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>

#include "codec.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace wt {
namespace {

constexpr int kTokLanes = 4;                         // lanes per group
constexpr int kTokChunks = kTile / 8 / kTokLanes;    // 16-byte chunks per lane and group
constexpr int kTokGroupsPerWarp = 32 / kTokLanes;

// Scale of one group whose 128 channels four lanes hold (v: this lane's
// chunks; lanes outside the group's valid range hold zeros): the group's
// amax over the four lanes, divided by 448; 1.0 for an all-zero group.
__device__ __forceinline__ float group_scale(const uint4 (&v)[kTokChunks]) {
  uint32_t m2 = 0;
#pragma unroll
  for (int c = 0; c < kTokChunks; ++c)
    m2 = absmax_bf16x2(absmax_bf16x2(m2, absmax_bf16x2(v[c].x, v[c].y)), absmax_bf16x2(v[c].z, v[c].w));
  m2 &= 0x7FFF7FFFu;
  float amax = fmaxf(bf16_lo(m2), bf16_hi(m2));
#pragma unroll
  for (int off = kTokLanes / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// ------------------------------------------------- large batches: TMA ring ---
constexpr int kRingGroupWarps = 12;                  // warps per consumer group
constexpr int kRingGroups = 2;                       // consumer groups: ring entry i -> group i % 2
constexpr int kRingSlots = 6;                        // shared-memory slots (the deepest ring used)
constexpr int kRingDepthTicket = 6;                  // ring depth with a ticket counter
constexpr int kRingDepthFixed = 4;                   // ring depth with the fixed hand-out
constexpr int kRingStageGroups = 128;                // channel groups per stage (the last may be fewer)
constexpr int kRingStageBytes = kRingStageGroups * kTile * 2;
constexpr int kRingConsumerWarps = kRingGroupWarps * kRingGroups;
constexpr int kRingThreads = 32 * (kRingConsumerWarps + 1);
constexpr uint32_t kStageEnd = 0xFFFFFFFFu;          // a ring entry that ends a consumer group
// A parity wait is meaningful only for a waiter that saw the previous
// phase of the same barrier complete; a group takes its entries in order,
// so each slot must belong to one group.
static_assert(kRingDepthTicket % kRingGroups == 0 && kRingDepthFixed % kRingGroups == 0,
              "every slot must belong to one consumer group");
static_assert(kRingDepthTicket <= kRingSlots && kRingDepthFixed <= kRingSlots, "slots");
static_assert(kRingThreads <= 1024, "threads per CTA");

struct RingCtl {
  uint64_t full[kRingSlots];
  uint64_t empty[kRingSlots];
  uint32_t stage_of[kRingSlots];     // the stage a slot holds, or kStageEnd
  int abort_flag;
};
constexpr size_t kRingSmemBytes = 128 + (size_t)kRingSlots * kRingStageBytes + sizeof(RingCtl);
static_assert(kRingSmemBytes <= 227 * 1024, "shared memory");

struct RingArgs {
  const uint16_t* x;
  int64_t ld;                // row stride of x, elements (a multiple of 8)
  uint32_t groups_per_token; // hidden / 128
  uint8_t* codes;
  float* scales;
  uint32_t* ticket;          // {next stage, CTAs done}, zero between launches; NULL: fixed hand-out
  uint32_t num_groups;       // tokens x hidden / 128
  uint32_t num_stages;       // ceil(num_groups / kRingStageGroups)
  uint32_t depth;            // ring depth: kRingDepthTicket or kRingDepthFixed
  int64_t stall_stage;       // testing hook: a stage that is never copied (-1: none)
  uint64_t limit_ns;         // bound of every wait
  int* error_word;
};

__device__ __forceinline__ void ring_give_up(const RingArgs& a, RingCtl& sm) {
  *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
  atomicOr(a.error_word, kErrTimeout);
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// One lane of the producer warp: ring entries 0, 1, ... are the CTA's
// stages in the order it takes them, then one end marker per consumer
// group. With a ticket counter each stage's ticket is taken one stage
// ahead, so that the atomic's round trip overlaps the wait for a slot.
__device__ void ring_producer(const RingArgs& a, RingCtl& sm, uint8_t* stages) {
  const uint64_t pol = load_policy();
  const volatile int* abort_flag = &sm.abort_flag;
  const uint32_t depth = a.depth;
  uint32_t i = 0;                                    // ring entries filled so far
  int ends = 0;
  bool failed = false;
  uint32_t next = a.ticket ? atomicAdd(a.ticket, 1u) : blockIdx.x;   // the first stage
  while (ends < kRingGroups) {
    const uint32_t slot = i % depth;
    if (i >= depth && !wait_bounded(smem_u32(&sm.empty[slot]), (i / depth - 1) & 1u, a.limit_ns, abort_flag)) {
      ring_give_up(a, sm);
      failed = true;
      break;
    }
    uint32_t s = kStageEnd;
    if (!ends) {
      s = next;
      if (s >= a.num_stages) s = kStageEnd;
      else next = a.ticket ? atomicAdd(a.ticket, 1u) : s + gridDim.x;
    }
    sm.stage_of[slot] = s;                           // published by the arrive below
    ++i;
    if (s == kStageEnd) {
      ++ends;
      mbar_arrive(smem_u32(&sm.full[slot]));
      continue;
    }
    if ((int64_t)s == a.stall_stage) continue;       // never armed: its consumers' wait runs out
    const uint32_t g0 = s * kRingStageGroups;
    const uint32_t n = min((uint32_t)kRingStageGroups, a.num_groups - g0);
    const uint32_t dst = smem_u32(stages + (size_t)slot * kRingStageBytes);
    mbar_arrive_tx(smem_u32(&sm.full[slot]), n * (uint32_t)(kTile * 2));
    if (a.ld == (int64_t)a.groups_per_token * kTile) {
      // contiguous rows: the stage is one run of bytes
      bulk_load(dst, a.x + (size_t)g0 * kTile, n * (uint32_t)(kTile * 2), smem_u32(&sm.full[slot]), pol);
    } else {
      // one copy per token row the stage touches
      for (uint32_t g = g0; g < g0 + n;) {
        const uint32_t t = g / a.groups_per_token, gin = g - t * a.groups_per_token;
        const uint32_t len = min(a.groups_per_token - gin, g0 + n - g);
        bulk_load(dst + (g - g0) * (uint32_t)(kTile * 2), a.x + (int64_t)t * a.ld + (int64_t)gin * kTile,
                  len * (uint32_t)(kTile * 2), smem_u32(&sm.full[slot]), pol);
        g += len;
      }
    }
  }
  // the CTA must not leave with copies in flight: wait (bounded) for the
  // last entry filled on each slot
  for (uint32_t j = 0; j < depth && j < i; ++j) {
    const uint32_t k = i - 1 - j;
    wait_bounded(smem_u32(&sm.full[k % depth]), (k / depth) & 1u, a.limit_ns, nullptr);
  }
  if (!a.ticket) return;
  // a CTA that gave up takes the tickets left, so that every CTA ends and
  // the counter is reset; every ticket taken has landed (its value is used)
  // before the CTA counts itself done, and the last CTA to do so resets it
  if (failed)
    while (next < a.num_stages) next = atomicAdd(a.ticket, 1u);
  asm volatile("" ::"r"(next) : "memory");
  __threadfence();
  if (atomicAdd(a.ticket + 1, 1u) == gridDim.x - 1) {
    *reinterpret_cast<volatile uint32_t*>(a.ticket) = 0u;
    *reinterpret_cast<volatile uint32_t*>(a.ticket + 1) = 0u;
    __threadfence();
  }
}

// Warp w of consumer group `grp`: in each of the group's ring entries,
// groups 8 w + lane / 4, + 8 kRingGroupWarps, ... of the stage it holds.
__device__ void ring_consumer(const RingArgs& a, RingCtl& sm, const uint8_t* stages, int grp, int w, int lane) {
  const volatile int* abort_flag = &sm.abort_flag;
  const uint32_t depth = a.depth;
  const int sub = lane % kTokLanes, gl = lane / kTokLanes;
  for (uint32_t i = (uint32_t)grp;; i += kRingGroups) {
    const uint32_t slot = i % depth;
    if (!__all_sync(kFull, wait_bounded(smem_u32(&sm.full[slot]), (i / depth) & 1u, a.limit_ns, abort_flag))) {
      if (lane == 0) ring_give_up(a, sm);
      return;
    }
    const uint32_t s = sm.stage_of[slot];
    if (s == kStageEnd) return;
    const uint32_t g0 = s * kRingStageGroups;
    const int n = (int)min((uint32_t)kRingStageGroups, a.num_groups - g0);
    const uint32_t base = smem_u32(stages + (size_t)slot * kRingStageBytes);
    for (int jb = w * kTokGroupsPerWarp; jb < n; jb += kRingGroupWarps * kTokGroupsPerWarp) {
      const int j = jb + gl;
      const bool valid = j < n;
      uint4 v[kTokChunks];
#pragma unroll
      for (int c = 0; c < kTokChunks; ++c) {
        const int q = kTokLanes * ((c + j) % kTokChunks) + sub;
        v[c] = valid ? lds_v4(base + (uint32_t)(j * kTile * 2 + q * 16)) : make_uint4(0, 0, 0, 0);
      }
      const float sc = group_scale(v);
      const bool corr = scale_in_range(sc);
      const float r = corr ? __frcp_rn(sc) : 0.0f;
      if (valid) {
        uint8_t* dst = a.codes + (size_t)(g0 + j) * kTile;
#pragma unroll
        for (int c = 0; c < kTokChunks; ++c) {
          const int q = kTokLanes * ((c + j) % kTokChunks) + sub;
          *reinterpret_cast<uint2*>(dst + q * 8) = corr ? quant_chunk(v[c], sc, r) : quant_exact(v[c], sc);
        }
        if (sub == 0) a.scales[g0 + j] = sc;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm.empty[slot]));
  }
}

__global__ void __launch_bounds__(kRingThreads, 1) token_ring_kernel(const __grid_constant__ RingArgs a) {
  extern __shared__ unsigned char smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  RingCtl& sm = *reinterpret_cast<RingCtl*>(stages + (size_t)kRingSlots * kRingStageBytes);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kRingGroupWarps);
    }
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (warp == kRingConsumerWarps) {
    if (lane == 0) ring_producer(a, sm, stages);
    return;
  }
  ring_consumer(a, sm, stages, warp / kRingGroupWarps, warp % kRingGroupWarps, lane);
}

// ------------------------------------------- other shapes: register stream ---
constexpr int kTokThreads = 256;
constexpr int kTokSlots = 4;        // groups in flight per lane

struct TokArgs {
  const uint16_t* x;
  uint8_t* codes;
  float* scales;
  int64_t hidden, ld;
  uint32_t groups_per_token;
  uint32_t num_groups;
};

enum TokMode { kTokFlat = 0, kTokVec = 1, kTokElem = 2 };

// kTokFlat: contiguous rows, hidden a multiple of 128 (groups are one flat
// sequence); kTokVec: 16-byte-aligned rows (vector loads, 8-byte code
// stores); kTokElem: element by element.
template <int kMode>
__global__ void __launch_bounds__(kTokThreads) token_kernel(const __grid_constant__ TokArgs a) {
  const int lane = threadIdx.x & 31, sub = lane % kTokLanes;
  const uint32_t gw = (uint32_t)(lane / kTokLanes);
  const uint32_t warp = (blockIdx.x * kTokThreads + threadIdx.x) >> 5;
  const uint32_t nwarps = (gridDim.x * kTokThreads) >> 5;
  for (uint32_t p = warp; kTokGroupsPerWarp * p < a.num_groups; p += kTokSlots * nwarps) {
    uint4 v[kTokSlots][kTokChunks];
    int64_t xoff[kTokSlots], coff[kTokSlots];
    int64_t cols[kTokSlots];                      // valid channels of the group
    uint32_t g[kTokSlots];
#pragma unroll
    for (int k = 0; k < kTokSlots; ++k) {
      g[k] = kTokGroupsPerWarp * (p + (uint32_t)k * nwarps) + gw;
      cols[k] = 0;
      xoff[k] = coff[k] = 0;
      if (g[k] < a.num_groups) {
        if (kMode == kTokFlat) {
          xoff[k] = coff[k] = (int64_t)g[k] * kTile;
          cols[k] = kTile;
        } else {
          const uint32_t t = g[k] / a.groups_per_token;
          const int64_t c0 = (int64_t)(g[k] - t * a.groups_per_token) * kTile;
          cols[k] = min((int64_t)kTile, a.hidden - c0);
          xoff[k] = (int64_t)t * a.ld + c0;
          coff[k] = (int64_t)t * a.hidden + c0;
        }
      }
#pragma unroll
      for (int c = 0; c < kTokChunks; ++c) {
        const int col = (c * kTokLanes + sub) * 8;
        v[k][c] = make_uint4(0, 0, 0, 0);
        if (kMode != kTokElem) {
          if (col < cols[k]) v[k][c] = ld_nc_v4(a.x + xoff[k] + col);
        } else {
          uint16_t e[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) e[j] = col + j < cols[k] ? ld_nc_u16(a.x + xoff[k] + col + j) : (uint16_t)0;
          v[k][c] = make_uint4(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16),
                               e[4] | ((uint32_t)e[5] << 16), e[6] | ((uint32_t)e[7] << 16));
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kTokSlots; ++k) {
      const float s = group_scale(v[k]);
      const bool corr = scale_in_range(s);
      const float r = corr ? __frcp_rn(s) : 0.0f;
#pragma unroll
      for (int c = 0; c < kTokChunks; ++c) {
        const int col = (c * kTokLanes + sub) * 8;
        if (col >= cols[k]) continue;
        const uint2 q = corr ? quant_chunk(v[k][c], s, r) : quant_exact(v[k][c], s);
        uint8_t* dst = a.codes + coff[k] + col;
        if (kMode != kTokElem) {
          *reinterpret_cast<uint2*>(dst) = q;
        } else {
          const uint32_t wds[2] = {q.x, q.y};
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (col + j < cols[k]) dst[j] = (uint8_t)(wds[j >> 2] >> (8 * (j & 3)));
        }
      }
      if (sub == 0 && g[k] < a.num_groups) a.scales[g[k]] = s;
    }
  }
}

// The codec's error word: one per device (a module variable), set by a ring
// wait that gave up, read and cleared by wt_tokens_check.
__device__ int g_token_error;

// The ring takes a batch from this many stages per SM on (contiguous with
// a ticket counter, else any): below, the register kernel, which needs no
// ring to fill, measured faster on B300.
constexpr int kRingMinStagesPerSmTicket = 16;
constexpr int kRingMinStagesPerSmFixed = 32;
// Strided rows (x_ld > hidden) take one copy per row segment of a stage;
// the ring takes them when rows are at least this many groups long (at
// most five copies per stage), the register kernel otherwise.
constexpr int64_t kRingMinGroupsPerStridedRow = 32;
constexpr int kMaxDevices = 64;
struct DeviceInfo {
  int sm_count = 0;
  int ctas[3] = {1, 1, 1};                 // resident register-kernel CTAs per SM, per mode
  int* error_word = nullptr;
};
DeviceInfo g_dev[kMaxDevices];               // filled once per device, under g_mu
std::mutex g_mu;
std::atomic<int64_t> g_stall_group{-1};     // testing hook (wt_debug_tokens_stall_group)
std::atomic<uint64_t> g_wait_limit_ns{0};

cudaError_t device_info(int dev, DeviceInfo* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.sm_count) {
    DeviceInfo n;
    void* word = nullptr;
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&n.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n.ctas[kTokFlat], token_kernel<kTokFlat>, kTokThreads,
                                                           0)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n.ctas[kTokVec], token_kernel<kTokVec>, kTokThreads,
                                                           0)) != cudaSuccess ||
        (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n.ctas[kTokElem], token_kernel<kTokElem>, kTokThreads,
                                                           0)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(token_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kRingSmemBytes)) != cudaSuccess ||
        (e = cudaGetSymbolAddress(&word, g_token_error)) != cudaSuccess)
      return e;
    for (int& c : n.ctas) c = std::max(1, c);
    n.error_word = static_cast<int*>(word);
    d = n;
  }
  *out = d;
  return cudaSuccess;
}

wt_status fail_tok(wt_status st, const std::string& msg) {
  set_error(msg);
  return st;
}

}  // namespace
}  // namespace wt

using namespace wt;

extern "C" wt_status wt_quantize_tokens(const void* x, int64_t tokens, int64_t hidden, int64_t x_ld,
                                        void* codes, float* scales, uint32_t* ticket, void* stream) {
  if (tokens < 0 || hidden < 1 || x_ld < hidden)
    return fail_tok(WT_ERR_INVALID_ARGUMENT, "wt_quantize_tokens: need tokens >= 0, hidden >= 1 and x_ld >= hidden");
  if (tokens == 0) return WT_OK;
  if (!x || !codes || !scales)
    return fail_tok(WT_ERR_INVALID_ARGUMENT, "wt_quantize_tokens: x, codes and scales must not be NULL");
  const int64_t gpt = (hidden + kTile - 1) / kTile;
  if (tokens * gpt >= (int64_t(1) << 31))
    return fail_tok(WT_ERR_INVALID_ARGUMENT,
                    "wt_quantize_tokens: more than 2^31 - 1 groups of 128 channels in one call");
  if (reinterpret_cast<uintptr_t>(x) % 2 || reinterpret_cast<uintptr_t>(scales) % 4 ||
      reinterpret_cast<uintptr_t>(ticket) % 4)
    return fail_tok(WT_ERR_ALIGNMENT, "wt_quantize_tokens: x must be 2-byte, scales and ticket 4-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail_tok(WT_ERR_CUDA, std::string("wt_quantize_tokens: cudaGetDevice: ") + cudaGetErrorString(e));
  DeviceInfo info;
  const DeviceInfo* di = &info;
  if ((e = device_info(dev, &info)) != cudaSuccess)
    return fail_tok(WT_ERR_CUDA, std::string("wt_quantize_tokens: device set-up: ") + cudaGetErrorString(e));
  const uint32_t num_groups = (uint32_t)(tokens * gpt);
  const bool vec = hidden % 8 == 0 && x_ld % 8 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(codes) % 8 == 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool flat = vec && hidden % kTile == 0 && x_ld == hidden;
  // strided rows go through the ring when a stage touches few of them
  const bool ring_ok = flat || (vec && hidden % kTile == 0 && gpt >= kRingMinGroupsPerStridedRow);
  const uint32_t num_stages = (num_groups + kRingStageGroups - 1) / kRingStageGroups;
  const uint32_t sms = (uint32_t)di->sm_count;
  // strided rows measured slower with the ticket counter than with the
  // fixed hand-out (0.484 against 0.443 ms for 131072 x 7168 rows 7296
  // apart), so they take the fixed hand-out
  const bool use_ticket = flat && ticket && num_stages >= kRingMinStagesPerSmTicket * sms;
  if (use_ticket || (ring_ok && num_stages >= kRingMinStagesPerSmFixed * sms)) {
    RingArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.ld = x_ld;
    a.groups_per_token = (uint32_t)gpt;
    a.codes = static_cast<uint8_t*>(codes);
    a.scales = scales;
    a.ticket = use_ticket ? ticket : nullptr;
    a.num_groups = num_groups;
    a.num_stages = num_stages;
    a.depth = use_ticket ? kRingDepthTicket : kRingDepthFixed;
    const int64_t stall = g_stall_group.load();
    a.stall_stage = stall >= 0 ? stall / kRingStageGroups : -1;
    const uint64_t lim = g_wait_limit_ns.load();
    a.limit_ns = lim ? lim : kDefaultTimeoutNs;
    a.error_word = di->error_word;
    token_ring_kernel<<<(int)sms, kRingThreads, kRingSmemBytes, s>>>(a);
  } else {
    TokArgs a;
    a.x = static_cast<const uint16_t*>(x);
    a.codes = static_cast<uint8_t*>(codes);
    a.scales = scales;
    a.hidden = hidden;
    a.ld = x_ld;
    a.groups_per_token = (uint32_t)gpt;
    a.num_groups = num_groups;
    // eight groups per warp per slot; one wave of resident CTAs at most
    const int mode = flat ? kTokFlat : vec ? kTokVec : kTokElem;
    const int64_t warps = (a.num_groups + kTokGroupsPerWarp - 1) / kTokGroupsPerWarp;
    const int64_t want = (warps + (kTokThreads / 32) - 1) / (kTokThreads / 32);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sms * di->ctas[mode]));
    if (mode == kTokFlat)
      token_kernel<kTokFlat><<<grid, kTokThreads, 0, s>>>(a);
    else if (mode == kTokVec)
      token_kernel<kTokVec><<<grid, kTokThreads, 0, s>>>(a);
    else
      token_kernel<kTokElem><<<grid, kTokThreads, 0, s>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_tok(WT_ERR_CUDA, std::string("wt_quantize_tokens: launch: ") + cudaGetErrorString(e));
  return WT_OK;
}

extern "C" wt_status wt_tokens_check(void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail_tok(WT_ERR_CUDA, std::string("wt_tokens_check: cudaGetDevice: ") + cudaGetErrorString(e));
  if ((e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return fail_tok(WT_ERR_CUDA, std::string("wt_tokens_check: cudaStreamSynchronize: ") + cudaGetErrorString(e));
  int* word;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    word = g_dev[dev].error_word;
  }
  if (!word) return WT_OK;                 // no call has run on this device
  int v = 0;
  if ((e = cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return fail_tok(WT_ERR_CUDA, std::string("wt_tokens_check: reading the error word: ") + cudaGetErrorString(e));
  if (!v) return WT_OK;
  const int zero = 0;
  if ((e = cudaMemcpy(word, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
    return fail_tok(WT_ERR_CUDA, std::string("wt_tokens_check: clearing the error word: ") + cudaGetErrorString(e));
  return fail_tok(WT_ERR_TIMEOUT,
                  "wt_tokens_check: a wait inside wt_quantize_tokens gave up; that call's codes and scales are "
                  "incomplete");
}

extern "C" wt_status wt_debug_tokens_stall_group(int64_t group, uint64_t wait_limit_ns) {
  if (group < -1) return fail_tok(WT_ERR_INVALID_ARGUMENT, "wt_debug_tokens_stall_group: group must be >= -1");
  g_wait_limit_ns.store(group < 0 ? 0 : wait_limit_ns);
  g_stall_group.store(group);
  return WT_OK;
}
