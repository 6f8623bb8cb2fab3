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
// Structure (one persistent CTA per SM):
//   - units (128x128 blocks) come in batches of four consecutive units of
//     the schedule, taken from a per-launch ticket counter, so that SMs
//     that run faster take more of them and every SM finishes within about
//     one batch of the others; the last CTA to finish resets the counter.
//   - a producer warp moves each unit's BF16 block into a ring of four
//     34 KiB shared-memory stages with the tensor memory accelerator: one
//     2-D tensor copy when all 128 rows come from one shard and are 16-byte
//     aligned; for rows that are not, k tensor copies through the shard's
//     view map (k shard rows per view row, see tmap.cpp). The full_tensor()
//     row gather across shards of 16-byte rows, and blocks of rows at most
//     8 elements wide, take no copy: the producer publishes each row's
//     address in the stage and the consumers load their chunks themselves
//     (128 small bulk copies cost about 5 us per block). The rest (wider
//     unaligned rows from several shards or without a view map) take one
//     1-D bulk copy per row. Full/empty mbarriers order the ring; the
//     producer runs up to four units ahead, so HBM reads stay in flight
//     while the consumers compute.
//   - two consumer groups of four warps take alternate units. Thread t of a
//     group owns the 16-byte column chunk t % 16 of the rows t / 16 + 8 j,
//     j = 0..15: it loads them from shared memory (conflict-free, two full
//     256-byte rows per warp instruction; unaligned rows are read out of
//     their slots), reduces |x| with packed bf16x2 abs-max, a warp shuffle
//     and one named barrier, quantises from registers, releases the stage
//     and stores its chunks. Each HBM byte is read once. That straight-line
//     path covers whole blocks of 16-byte rows and blocks of unaligned rows
//     with one destination; partial blocks of 16-byte rows, several
//     destinations, extreme scales and debug checks go through general
//     routines that re-read the thread's rows from the stage before
//     releasing it, so their code stays out of the hot path's registers.
// Division: each code is E(fl32(x / s)), computed from r = RN(1/s) with
// one exact correction step (codec.cuh).
//
// Waits. Every mbarrier wait gives up after PrepArgs::timeout_ns; the role
// that gives up sets kErrTimeout in the error word and an abort flag in
// shared memory, the others notice it and leave, and the producer first
// waits (bounded) for its copies in flight to land.
#include "codec.cuh"
#include "plan.h"
#include "ptx.cuh"

namespace wt {
namespace {

constexpr int kGroups = 2;                          // consumer groups
constexpr int kGroupWarps = 4;
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kStages = 4;                          // ring depth
// Unit k uses stage k % kStages and group k % kGroups. Each stage must
// belong to one group: a parity wait on an mbarrier is only meaningful
// when the waiter has already seen the previous phase complete, which a
// group guarantees for its own stages by taking their units in order.
static_assert(kStages % kGroups == 0, "every stage must belong to one consumer group");
constexpr int kStageBytes = kTile * kTile * 2;      // one BF16 block
constexpr int kRowBytes = kTile * 2;                // one block row in a stage
// A row that is not 16-byte aligned is copied as the 16-byte-aligned span
// around it (at most 16 + 256 bytes) into a slot of its own, and the
// consumers move it into place; a stage holds 128 such slots.
constexpr int kSlotBytes = kRowBytes + 16;
constexpr int kStageStride = kTile * kSlotBytes;
// A block whose rows the consumers load themselves (kUnitDirect) leaves the
// stage empty; the producer publishes the row addresses in the stage's
// tail, past the 256-byte rows that the general store routines write back.
constexpr int kRowPtrOffset = kStageBytes;
static_assert(kRowPtrOffset + kTile * 8 <= kStageStride, "row addresses fit in the stage's tail");
// units per descriptor batch (one 32-byte descriptor per 8 lanes)
constexpr int kBatch = 4;
constexpr int kConsumerThreads = kGroups * kGroupThreads;
constexpr int kCtaThreads = kConsumerThreads + 32;
constexpr int kRowStride = kGroupThreads / 16;      // rows between a thread's rows
constexpr int kRows = kTile / kRowStride;           // rows per consumer thread


struct SmemCtl {
  DevUnit meta[kStages];                 // the unit in each stage
  uint64_t full[kStages];                // producer -> consumers
  uint64_t empty[kStages];               // consumers -> producer
  float wmax[kGroups][2][kGroupWarps];   // per-warp block amax, double-buffered
  int abort_flag;
  uint16_t roff[kStages][kTile];         // unaligned rows: byte offset of each row in the stage
};
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageStride + sizeof(SmemCtl);
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

// --------------------------------------------------------- waits, abort ---
__device__ __forceinline__ void give_up(const PrepArgs& a, SmemCtl& sm) {
  *reinterpret_cast<volatile int*>(&sm.abort_flag) = 1;
  atomicOr(a.error_word, kErrTimeout);
}

// --------------------------------------------------------------- producer ---
// Units come in batches of kBatch consecutive units of the schedule. With a
// ticket counter (PrepArgs::ticket) every CTA takes the next free batch when
// it needs one, so SMs that run faster take more batches and the launch ends
// evenly; without one, CTA b takes units b, b + grid, b + 2 grid, ...
struct Batch {
  uint32_t word;   // lane l: word l % 8 of the batch's unit l / 8
  int64_t first;   // the batch's first unit (static: its CTA-local index)
  int n;           // units in the batch, 0 once the CTA's units are done
};

// Lane 0 takes the next ticket. The value is broadcast only when its batch
// is loaded, a batch later, so the atomic's latency does not stall the warp.
__device__ __forceinline__ uint32_t take_ticket(const PrepArgs& a, int lane) {
  return lane == 0 ? atomicAdd(a.ticket, 1u) : 0u;
}

// Global unit index of unit j of a batch.
__device__ __forceinline__ int64_t batch_unit(bool dyn, const Batch& bt, int j, int64_t first) {
  return dyn ? bt.first + j : first + (bt.first + j) * (int64_t)gridDim.x;
}

__device__ __forceinline__ Batch load_batch(const PrepArgs& a, bool dyn, int64_t first, int64_t n_local,
                                            int64_t index, int lane) {
  Batch bt;
  if (dyn) {
    index = __shfl_sync(kFull, (uint32_t)index, 0);      // lane 0's ticket
    bt.first = a.unit_begin + (int64_t)kBatch * index;
    bt.n = (int)(a.unit_end <= bt.first ? 0 : a.unit_end - bt.first >= kBatch ? kBatch : a.unit_end - bt.first);
  } else {
    bt.first = (int64_t)kBatch * index;                   // CTA-local units
    bt.n = (int)(n_local <= bt.first ? 0 : n_local - bt.first >= kBatch ? kBatch : n_local - bt.first);
  }
  bt.word = 0;
  if ((lane >> 3) < bt.n)
    bt.word = ld_nc_u32(reinterpret_cast<const uint32_t*>(a.units + batch_unit(dyn, bt, lane >> 3, first)) +
                        (lane & 7));
  return bt;
}

// Rows that are not 16-byte aligned (or treated as such under
// WT_FLAG_FORCE_NARROW), wider than 8 elements, from several shards or
// without a view map: one bulk copy per row. Each row is copied as the
// 16-byte-aligned span that holds it into its 272-byte slot, at offset
// address % 16 (the span starts at most 15 bytes before the row and ends
// at most 15 after it; both ends lie in the 16-byte granules of the row's
// own first and last bytes, so no page that the row does not touch is
// read), and the consumers move it into place. Blocks of 16-byte rows take
// tensor copies or direct loads, so the branch below that would copy such
// a row straight to its place in the stage serves no current unit.
__device__ __forceinline__ void load_rows(const PrepArgs& a, SmemCtl& sm, const uint32_t (&w)[8], int st,
                                          uint32_t dst, uint32_t full, uint64_t pol, int lane) {
  const int nrows = (int)(w[5] & 0xFFu) + 1;
  const uint32_t row_bytes = (((w[5] >> 8) & 0xFFu) + 1u) * 2u;
  const bool narrow = !((w[5] >> 16) & kUnitVec);
  const int64_t N = w[4];
  int run = (int)w[0];
  uintptr_t src[kTile / 32];
  uint32_t len[kTile / 32];
  uint32_t total = 0;
#pragma unroll
  for (int i = 0; i < kTile / 32; ++i) {
    const int r = lane + 32 * i;
    src[i] = 0;
    len[i] = 0;
    if (r < nrows) {
      const int64_t fr = (int64_t)w[1] + r;
      while (fr >= a.runs[run].row0 + a.runs[run].rows) ++run;
      const DevRun rn = a.runs[run];
      const uintptr_t p = reinterpret_cast<uintptr_t>(a.shard_ptrs[rn.slot] + (fr - rn.row0) * N +
                                                      (int64_t)w[3] * kTile);
      if (narrow) {
        src[i] = p & ~(uintptr_t)15;
        len[i] = (uint32_t)(((p + row_bytes + 15) & ~(uintptr_t)15) - src[i]);
        sm.roff[st][r] = (uint16_t)(r * kSlotBytes + (p & 15));
      } else {
        src[i] = p;
        len[i] = row_bytes;
      }
      total += len[i];
    }
  }
  total = __reduce_add_sync(kFull, total);
  __syncwarp();                 // the row offsets are written before the stage's arrival
  if (lane == 0) mbar_arrive_tx(full, total);
  __syncwarp();
  const uint32_t stride = narrow ? (uint32_t)kSlotBytes : (uint32_t)kRowBytes;
#pragma unroll
  for (int i = 0; i < kTile / 32; ++i)
    if (len[i]) bulk_load(dst + (uint32_t)(lane + 32 * i) * stride, reinterpret_cast<const void*>(src[i]),
                          len[i], full, pol);
}

// Rows that are not 16-byte aligned, all from one shard that has a view map
// (see tmap.cpp): the block's rows fall into k residue classes, each one
// box of 128 / k view rows by 136 columns, copied by one tensor copy into
// consecutive 272-byte slots of the stage; the producer records where each
// block row starts (slot and offset 0..7 elements) for the consumers.
__device__ __forceinline__ void load_view(const PrepArgs& a, SmemCtl& sm, const uint32_t (&w)[8], const DevRun& rn,
                                          int st, uint32_t dst, uint32_t full, uint64_t pol, int lane) {
  const int64_t N = w[4];
  const int k = (N & 1) ? 8 : (N & 2) ? 4 : (N & 4) ? 2 : 1;
  const int per_box = kTile / k;
  const int64_t s0 = (int64_t)w[1] - rn.row0;   // the block's first row in the shard
  const int64_t col0 = (int64_t)w[3] * kTile;
#pragma unroll
  for (int i = 0; i < kTile / 32; ++i) {
    const int r = lane + 32 * i;
    const int j = r % k;
    const int64_t x = ((s0 + j) % k) * N + col0;
    sm.roff[st][r] = (uint16_t)(((j * per_box) + r / k) * kSlotBytes + 2 * (int)(x & 7));
  }
  __syncwarp();                 // the row offsets are written before the stage's arrival
  if (lane == 0) mbar_arrive_tx(full, (uint32_t)(kTile * kSlotBytes));
  __syncwarp();
  if (lane < k) {
    const unsigned char* map = a.tmaps + (size_t)rn.slot * kTmapBytes;
    const int64_t x = ((s0 + lane) % k) * N + col0;
    tma_load_2d(dst + (uint32_t)(lane * per_box * kSlotBytes), map, (int)(x & ~(int64_t)7), (int)((s0 + lane) / k),
                full, pol);
  }
}

// Rows the consumers load themselves (kUnitDirect): the address of each
// block row's first element, resolved through the row runs like load_rows,
// published with the stage's arrival instead of a copy.
__device__ __forceinline__ void publish_rows(const PrepArgs& a, const uint32_t (&w)[8], uint8_t* sp, uint32_t full,
                                             int lane) {
  const uint16_t** rowp = reinterpret_cast<const uint16_t**>(sp + kRowPtrOffset);
  const int nrows = (int)(w[5] & 0xFFu) + 1;
  const int64_t N = w[4];
  int run = (int)w[0];
#pragma unroll
  for (int i = 0; i < kTile / 32; ++i) {
    const int r = lane + 32 * i;
    if (r < nrows) {
      const int64_t fr = (int64_t)w[1] + r;
      while (fr >= a.runs[run].row0 + a.runs[run].rows) ++run;
      const DevRun rn = a.runs[run];
      rowp[r] = a.shard_ptrs[rn.slot] + (fr - rn.row0) * N + (int64_t)w[3] * kTile;
    }
  }
  fence_proxy_async_smem();     // the stage is refilled by copies later
  __syncwarp();                 // the row addresses are written before the stage's arrival
  if (lane == 0) mbar_arrive(full);
}

// dyn: units come from the ticket counter, else the static sequence.
__device__ void producer(const PrepArgs& a, bool dyn, SmemCtl& sm, uint8_t* stages, int64_t first,
                         int64_t n_local, int lane) {
  const uint32_t stage0 = smem_u32(stages);
  const uint64_t pol = load_policy();
  // descriptors of a batch are loaded two batches ahead; with tickets, the
  // ticket of a batch is taken one batch before its descriptors
  int64_t idx[3] = {0, 1, 2};
  if (dyn) {
    idx[0] = take_ticket(a, lane);
    idx[1] = take_ticket(a, lane);
    idx[2] = take_ticket(a, lane);
  }
  Batch cur = load_batch(a, dyn, first, n_local, idx[0], lane);
  Batch nxt = load_batch(a, dyn, first, n_local, idx[1], lane);
  int64_t next_idx = idx[2];
  int64_t last_slot = -1;
  int64_t k = 0;                // CTA-local sequence of stage uses
  bool ok = true;
  // wait until stage k % kStages is free; false (and give up) if the wait ran out
  auto claim = [&](int st) {
    bool got = true;
    if (lane == 0) got = wait_bounded(smem_u32(&sm.empty[st]), (uint32_t)((k / kStages) & 1) ^ 1u,
                                      a.timeout_ns, &sm.abort_flag);
    if (!__shfl_sync(kFull, (int)got, 0)) {
      if (lane == 0) give_up(a, sm);
      return false;
    }
    return true;
  };
  while (ok && cur.n > 0) {
    const Batch nn = load_batch(a, dyn, first, n_local, next_idx, lane);
    if (dyn && nn.n > 0) next_idx = take_ticket(a, lane);
    else next_idx += dyn ? 0 : 1;
    for (int j = 0; j < cur.n; ++j, ++k) {
      uint32_t w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = __shfl_sync(kFull, cur.word, 8 * j + i);
      const int st = (int)(k % kStages);
      const uint32_t full = smem_u32(&sm.full[st]);
      if (!claim(st)) {
        ok = false;
        break;
      }
      // testing hook: leave this unit's stage unfilled, so that its
      // consumers' wait runs out
      if (batch_unit(dyn, cur, j, first) == a.stall_unit) continue;
      const uint32_t flags = w[5] >> 16;
      const uint32_t dst = stage0 + (uint32_t)st * kStageStride;
      if (lane == 0) {
        uint4* m = reinterpret_cast<uint4*>(&sm.meta[st]);
        m[0] = make_uint4(w[0], w[1], w[2], w[3]);
        m[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      if (flags & kUnitDirect) {
        publish_rows(a, w, stages + (size_t)st * kStageStride, full, lane);
      } else if ((flags & kUnitVec) && !(flags & kUnitMulti)) {
        if (lane == 0) {
          const unsigned char* map = a.tmaps + (size_t)w[0] * kTmapBytes;
          if (a.tmap_fence && (int64_t)w[0] != last_slot) tmap_acquire(map);
          last_slot = w[0];
          mbar_arrive_tx(full, kStageBytes);
          tma_load_2d(dst, map, (int)(w[3] * kTile), (int)w[1], full, pol);
        }
      } else if (flags & kUnitView) {
        const DevRun rn = a.runs[w[0]];
        if (a.view_ok[rn.slot]) {
          if (lane == 0 && a.tmap_fence && (int64_t)rn.slot != last_slot)
            tmap_acquire(a.tmaps + (size_t)rn.slot * kTmapBytes);
          last_slot = rn.slot;
          load_view(a, sm, w, rn, st, dst, full, pol, lane);
        } else {
          load_rows(a, sm, w, st, dst, full, pol, lane);
        }
      } else {
        load_rows(a, sm, w, st, dst, full, pol, lane);
      }
    }
    cur = nxt;
    nxt = nn;
  }
  // a ticket taken but not used (after an abort) must still have landed
  // before this CTA counts itself done: wait for the atomic's return value
  if (dyn) asm volatile("" ::"r"((uint32_t)next_idx) : "memory");
  // this CTA takes no more units: a launch queued after this one as a
  // programmatic dependent may start once every CTA has said so
  if (lane == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // one end marker per consumer group: an arrival with no copy
  for (int e = 0; ok && e < kGroups; ++e, ++k) {
    const int st = (int)(k % kStages);
    if (!claim(st)) {
      ok = false;
      break;
    }
    if (lane == 0) {
      sm.meta[st].shape = kUnitEnd << 16;
      mbar_arrive(smem_u32(&sm.full[st]));
    }
  }
  // no copy may still be landing in this CTA's shared memory when it exits:
  // wait for the last fill of every stage (completed fills return at once)
  if (lane == 0) {
    for (int st = 0; st < kStages && st < k; ++st) {
      const int64_t last = st + ((k - 1 - st) / kStages) * kStages;
      if (!wait_bounded(smem_u32(&sm.full[st]), (uint32_t)((last / kStages) & 1), a.timeout_ns, nullptr))
        give_up(a, sm);
    }
  }
  __syncwarp();
}

// -------------------------------------------------------------- consumers ---
template <bool kDebug>
__device__ __forceinline__ bool store_ok(const PrepArgs& a, const DevDstPtr& dp, const void* p, uint64_t n) {
  if (!kDebug) return true;
  const uint8_t* q = static_cast<const uint8_t*>(p);
  if (q >= dp.pool_begin && q + n <= dp.pool_end) return true;
  atomicOr(a.error_word, kErrBadStore);
  return false;
}

template <bool kDebug>
__device__ __forceinline__ DevDstPtr load_dst(const PrepArgs& a, uint32_t i) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(a.dst_ptrs + i);
  DevDstPtr d;
  d.data = reinterpret_cast<uint8_t*>(((uint64_t)ld_nc_u32(p + 1) << 32) | ld_nc_u32(p));
  d.scale = reinterpret_cast<float*>(((uint64_t)ld_nc_u32(p + 3) << 32) | ld_nc_u32(p + 2));
  d.pool_begin = d.pool_end = nullptr;
  if (kDebug) {
    d.pool_begin = reinterpret_cast<const uint8_t*>(((uint64_t)ld_nc_u32(p + 5) << 32) | ld_nc_u32(p + 4));
    d.pool_end = reinterpret_cast<const uint8_t*>(((uint64_t)ld_nc_u32(p + 7) << 32) | ld_nc_u32(p + 6));
  }
  return d;
}

// Where block (bi, bj) lands in one destination: the element offset of the
// thread's first row chunk, the element step between its rows, the index
// of the block's scale, and whether the destination holds the block at all
// (a tensor-parallel slice holds only some block rows or block columns).
struct Place {
  int64_t off, step;
  uint32_t sidx;
  bool held;
};

__device__ __forceinline__ Place place(const PrepArgs& a, const DevUnit& m, uint32_t entry, int r0, int cc) {
  const uint32_t bi = m.bi, bj = m.bj;
  // dim, map_off, ld, sld; an output without slices needs no table
  const uint4 g = ((m.shape >> 16) & kUnitSliced)
                      ? ld_nc_v4(a.geom + entry)
                      : make_uint4(0xFFFFFFFFu, 0u, m.cols, (m.cols + kTile - 1) / kTile);
  int32_t di = (int32_t)bi, dj = (int32_t)bj;
  if ((int32_t)g.x == 0) di = (int32_t)ld_nc_u32(a.blockmap + (int32_t)g.y + bi);
  else if ((int32_t)g.x == 1) dj = (int32_t)ld_nc_u32(a.blockmap + (int32_t)g.y + bj);
  Place pl;
  pl.held = di >= 0 && dj >= 0;
  pl.off = ((int64_t)di * kTile + r0) * (int64_t)g.z + (int64_t)dj * kTile + cc * 8;
  pl.step = kRowStride * (int64_t)g.z;
  pl.sidx = (uint32_t)di * g.w + (uint32_t)dj;
  return pl;
}

// The 16 bytes at stage offset `off` (even: rows are 2-byte aligned): four
// 4-byte loads, or five and a 16-bit funnel shift when they start 2 bytes
// past a word.
__device__ __forceinline__ uint4 ld_skewed(const uint8_t* sp, int off) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(sp + (off & ~3));
  if ((off & 2) == 0) return make_uint4(w[0], w[1], w[2], w[3]);
  const uint32_t w4 = w[4];
  return make_uint4(__funnelshift_r(w[0], w[1], 16), __funnelshift_r(w[1], w[2], 16),
                    __funnelshift_r(w[2], w[3], 16), __funnelshift_r(w[3], w4, 16));
}

// Zero the BF16 values of a chunk at and after index `valid` (0..8).
__device__ __forceinline__ uint4 keep_first(uint4 v, int valid) {
  if (valid >= 8) return v;
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k)
    w[k] &= (2 * k < valid ? 0x0000FFFFu : 0u) | (2 * k + 1 < valid ? 0xFFFF0000u : 0u);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Rows that are not 16-byte aligned arrive in slots (see load_rows and
// load_view): the thread's chunks, read from them, with what lies outside
// the block zeroed.
__device__ __forceinline__ void read_slots(const SmemCtl& sm, int st, const uint8_t* sp, int nrows, int ncols,
                                           int r0, int cc, uint4 (&v)[kRows]) {
  const int valid = ncols - 8 * cc;
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    const int r = r0 + kRowStride * j;
    v[j] = make_uint4(0, 0, 0, 0);
    if (r < nrows && valid > 0) v[j] = keep_first(ld_skewed(sp, sm.roff[st][r] + 16 * cc), valid);
  }
}

// kUnitDirect: the thread's chunks loaded from the row addresses the
// producer published, 16 bytes at a time for 16-byte rows, element by
// element for rows narrower than one chunk; zero outside the block. The
// element loads are predicated rather than branched around and are not
// volatile, so that a thread's rows are in flight together (measured: a
// 1-column block 0.7 us faster than with branched volatile loads; for the
// 16-byte loads the volatile form measured faster).
__device__ __forceinline__ void load_direct(const uint8_t* sp, bool vec, int nrows, int ncols, int r0, int cc,
                                            uint4 (&v)[kRows]) {
  const uint16_t* const* rowp = reinterpret_cast<const uint16_t* const*>(sp + kRowPtrOffset);
  const int valid = ncols - 8 * cc;
#pragma unroll
  for (int j = 0; j < kRows; ++j) {
    const int r = r0 + kRowStride * j;
    const bool ok = r < nrows && valid > 0;
    const uint16_t* p = ok ? rowp[r] + 8 * cc : nullptr;
    if (vec) {
      v[j] = make_uint4(0, 0, 0, 0);
      if (ok) v[j] = ld_nc_v4(p);
    } else {
      uint32_t e[4];
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        const uint32_t lo = ok && k < valid ? (uint32_t)__ldg(p + k) : 0u;
        const uint32_t hi = ok && k + 1 < valid ? (uint32_t)__ldg(p + k + 1) : 0u;
        e[k >> 1] = lo | (hi << 16);
      }
      v[j] = make_uint4(e[0], e[1], e[2], e[3]);
    }
  }
}

// The thread's chunks written back at their aligned places in the stage
// (256-byte rows) for the general routines, once the whole group has read
// the slots they overlap.
__device__ __forceinline__ void write_back(uint8_t* sp, int r0, int cc, const uint4 (&v)[kRows]) {
#pragma unroll
  for (int j = 0; j < kRows; ++j)
    *reinterpret_cast<uint4*>(sp + (r0 + kRowStride * j) * kRowBytes + cc * 16) = v[j];
  fence_proxy_async_smem();          // the stage is refilled by copies later
}

// Codes of one row chunk where rows are not 8-byte aligned; `valid` bytes
// of the 8 are inside the block. A whole chunk goes out in the widest
// stores its address allows (rows of an even length are 2-byte aligned,
// every fourth one 8-byte aligned), a partial one byte by byte.
template <bool kDebug>
__device__ __forceinline__ void store_codes_bytes(const PrepArgs& a, const DevDstPtr& dp, uint8_t* p, uint2 q,
                                                  bool row_ok, int valid) {
  if (!row_ok) return;
  const uint32_t wds[2] = {q.x, q.y};
  const uintptr_t al = reinterpret_cast<uintptr_t>(p);
  if (valid >= 8 && (al & 1u) == 0) {
    if (!store_ok<kDebug>(a, dp, p, 8)) return;
    if ((al & 7u) == 0) {
      *reinterpret_cast<uint2*>(p) = q;
    } else if ((al & 3u) == 0) {
      reinterpret_cast<uint32_t*>(p)[0] = q.x;
      reinterpret_cast<uint32_t*>(p)[1] = q.y;
    } else {
#pragma unroll
      for (int h = 0; h < 4; ++h) reinterpret_cast<uint16_t*>(p)[h] = (uint16_t)(wds[h >> 1] >> (16 * (h & 1)));
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (e < valid && store_ok<kDebug>(a, dp, p + e, 1)) p[e] = (uint8_t)(wds[e >> 2] >> (8 * (e & 3)));
}

// Eight BF16 values of one row chunk where rows are not 16-byte aligned
// (always 2-byte aligned): the widest stores the address allows for a
// whole chunk, element by element for a partial one.
template <bool kDebug>
__device__ __forceinline__ void store_bf16_chunk(const PrepArgs& a, const DevDstPtr& dp, uint8_t* p, uint4 v,
                                                 int valid) {
  const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
  const uintptr_t al = reinterpret_cast<uintptr_t>(p);
  if (valid >= 8) {
    if (!store_ok<kDebug>(a, dp, p, 16)) return;
    if ((al & 15u) == 0) {
      *reinterpret_cast<uint4*>(p) = v;
    } else if ((al & 7u) == 0) {
      reinterpret_cast<uint2*>(p)[0] = make_uint2(v.x, v.y);
      reinterpret_cast<uint2*>(p)[1] = make_uint2(v.z, v.w);
    } else if ((al & 3u) == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) reinterpret_cast<uint32_t*>(p)[k] = wds[k];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) reinterpret_cast<uint16_t*>(p)[e] = (uint16_t)(wds[e >> 1] >> (16 * (e & 1)));
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (e < valid && store_ok<kDebug>(a, dp, p + 2 * e, 2))
      *reinterpret_cast<uint16_t*>(p + 2 * e) = (uint16_t)(wds[e >> 1] >> (16 * (e & 1)));
}

// The general FP8 path (partial blocks, rows that are not 16-byte aligned,
// several destinations, a scale outside the correction step's range, debug
// checks): the thread's rows again from the stage, one row at a time, to
// every destination.
template <bool kDebug>
__device__ __noinline__ void store_fp8_general(const PrepArgs& a, const DevUnit m, const DevDstPtr dp0,
                                               const uint8_t* tp, float s, int t, int r0, int cc) {
  const int nrows = (int)(m.shape & 0xFFu) + 1, ncols = (int)((m.shape >> 8) & 0xFFu) + 1;
  const bool vec = (m.shape >> 16) & kUnitVec;
  const uint32_t se = (__float_as_uint(s) >> 23) & 0xFFu;
  const bool corr = se >= kMinScaleExp && se <= kMaxScaleExp;
  const float r = corr ? __frcp_rn(s) : 0.0f;
  for (uint32_t d = 0; d < m.num_dsts; ++d) {
    const Place pl = place(a, m, m.dst_begin + d, r0, cc);
    if (!pl.held) continue;
    const DevDstPtr dp = d == 0 ? dp0 : load_dst<kDebug>(a, m.dst_begin + d);
    if (t == 0) {
      float* sp4 = dp.scale + pl.sidx;
      if (store_ok<kDebug>(a, dp, sp4, 4)) *sp4 = s;
    }
    if (cc * 8 >= ncols) continue;
    uint8_t* row = dp.data + pl.off;
    const int64_t row_step = pl.step;
#pragma unroll 1
    for (int j = 0; j < kRows && r0 + kRowStride * j < nrows; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(tp + j * kRowStride * kRowBytes);
      const uint2 q = corr ? quant_chunk(v, s, r) : quant_exact(v, s);
      uint8_t* p = row + j * row_step;
      if (vec) {
        if (store_ok<kDebug>(a, dp, p, 8)) *reinterpret_cast<uint2*>(p) = q;
      } else {
        store_codes_bytes<kDebug>(a, dp, p, q, true, ncols - cc * 8);
      }
    }
  }
}

// The general BF16 pass-through path, same cases.
template <bool kDebug>
__device__ __noinline__ void store_bf16_general(const PrepArgs& a, const DevUnit m, const DevDstPtr dp0,
                                                const uint8_t* tp, int r0, int cc) {
  const int nrows = (int)(m.shape & 0xFFu) + 1, ncols = (int)((m.shape >> 8) & 0xFFu) + 1;
  const bool vec = (m.shape >> 16) & kUnitVec;
  if (cc * 8 >= ncols) return;
  for (uint32_t d = 0; d < m.num_dsts; ++d) {
    const Place pl = place(a, m, m.dst_begin + d, r0, cc);
    if (!pl.held) continue;
    const DevDstPtr dp = d == 0 ? dp0 : load_dst<kDebug>(a, m.dst_begin + d);
    uint8_t* row = dp.data + 2 * pl.off;
    const int64_t row_step = pl.step;
#pragma unroll 1
    for (int j = 0; j < kRows && r0 + kRowStride * j < nrows; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(tp + j * kRowStride * kRowBytes);
      uint8_t* p = row + 2 * j * row_step;
      if (vec) {
        if (store_ok<kDebug>(a, dp, p, 16)) *reinterpret_cast<uint4*>(p) = v;
      } else {
        store_bf16_chunk<kDebug>(a, dp, p, v, ncols - cc * 8);
      }
    }
  }
}

template <bool kDebug>
__device__ void consumer(const PrepArgs& a, SmemCtl& sm, uint8_t* stages, int g, int t) {
  const int lane = t & 31, wg = t >> 5;
  const int cc = t & 15;       // 16-byte column chunk
  const int r0 = t >> 4;       // first row; rows r0 + kRowStride j
  const int bar_id = 1 + g;
  int it = 0;
  for (int64_t k = g;; k += kGroups, ++it) {
    const int st = (int)(k % kStages);
    const bool ok = wait_bounded(smem_u32(&sm.full[st]), (uint32_t)((k / kStages) & 1), a.timeout_ns,
                                 &sm.abort_flag);
    if (!ok) give_up(a, sm);
    if (bar_red_or(bar_id, kGroupThreads, !ok)) return;
    DevUnit m;
    {
      const uint4 m0 = reinterpret_cast<const uint4*>(&sm.meta[st])[0];
      const uint4 m1 = reinterpret_cast<const uint4*>(&sm.meta[st])[1];
      m = DevUnit{m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    }
    const uint32_t flags = m.shape >> 16;
    if (flags & kUnitEnd) return;       // the producer has no more units
    const DevDstPtr dp0 = load_dst<kDebug>(a, m.dst_begin);
    const Place pl0 = place(a, m, m.dst_begin, r0, cc);
    const int nrows = (int)(m.shape & 0xFFu) + 1, ncols = (int)((m.shape >> 8) & 0xFFu) + 1;
    const bool whole = (m.shape & 0xFFFFu) == 0x7F7Fu;
    const bool vec = flags & kUnitVec;
    uint8_t* sp = stages + (size_t)st * kStageStride;
    uint4 v[kRows];
    const uint8_t* tp = sp + r0 * kRowBytes + cc * 16;
    const bool direct = flags & kUnitDirect;
    if (direct) {
      load_direct(sp, vec, nrows, ncols, r0, cc, v);
    } else if (!vec) {
      read_slots(sm, st, sp, nrows, ncols, r0, cc, v);
    } else if (whole) {
#pragma unroll
      for (int j = 0; j < kRows; ++j) v[j] = *reinterpret_cast<const uint4*>(tp + j * kRowStride * kRowBytes);
    } else {
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        v[j] = make_uint4(0, 0, 0, 0);
        if (r0 + kRowStride * j < nrows && cc * 8 < ncols)
          v[j] = *reinterpret_cast<const uint4*>(tp + j * kRowStride * kRowBytes);
      }
    }
    // the common case runs straight through: a whole block of 16-byte rows
    // with one destination; rows that are not 16-byte aligned with one
    // destination also store from registers, chunk by chunk with the widest
    // stores their addresses allow; everything else takes the general routines
    const bool fast = !kDebug && whole && vec && m.num_dsts == 1 && pl0.held;
    const bool narrow_fast = !kDebug && !vec && m.num_dsts == 1 && pl0.held;
    const uint32_t empty = smem_u32(&sm.empty[st]);

    if (flags & kUnitFp8) {
      // block amax: per thread, across the warp, across the group's warps
      uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
      for (int j = 0; j < kRows; ++j) {
        a0 = absmax_bf16x2(a0, v[j].x);
        a1 = absmax_bf16x2(a1, v[j].y);
        a2 = absmax_bf16x2(a2, v[j].z);
        a3 = absmax_bf16x2(a3, v[j].w);
      }
      const uint32_t m2 = absmax_bf16x2(absmax_bf16x2(a0, a1), absmax_bf16x2(a2, a3)) & 0x7FFF7FFFu;
      float mx = fmaxf(bf16_lo(m2), bf16_hi(m2));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
      if (lane == 0) sm.wmax[g][it & 1][wg] = mx;
      bar_sync(bar_id, kGroupThreads);
      const float* wm = sm.wmax[g][it & 1];
      float amax = wm[0];
#pragma unroll
      for (int w = 1; w < kGroupWarps; ++w) amax = fmaxf(amax, wm[w]);
      const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
      const uint32_t se = (__float_as_uint(s) >> 23) & 0xFFu;
      if (fast && se >= kMinScaleExp && se <= kMaxScaleExp) {
        const float r = __frcp_rn(s);
        uint2 q[kRows];
#pragma unroll
        for (int j = 0; j < kRows; ++j) q[j] = quant_chunk(v[j], s, r);
        mbar_arrive(empty);                       // the codes are in registers
        if (t == 0) dp0.scale[pl0.sidx] = s;
        uint8_t* row = dp0.data + pl0.off;
#pragma unroll
        for (int j = 0; j < kRows; ++j) __stcs(reinterpret_cast<uint2*>(row + j * pl0.step), q[j]);
      } else if (narrow_fast && se >= kMinScaleExp && se <= kMaxScaleExp) {
        const float r = __frcp_rn(s);
        uint2 q[kRows];
#pragma unroll
        for (int j = 0; j < kRows; ++j) q[j] = quant_chunk(v[j], s, r);
        mbar_arrive(empty);                       // the codes are in registers
        if (t == 0) dp0.scale[pl0.sidx] = s;
        uint8_t* row = dp0.data + pl0.off;
        const int valid = ncols - cc * 8;
        if (valid > 0)
#pragma unroll
          for (int j = 0; j < kRows; ++j)
            store_codes_bytes<false>(a, dp0, row + j * pl0.step, q[j], r0 + kRowStride * j < nrows, valid);
      } else {
        // the slots were read before the amax barrier; rows loaded directly
        // were never in the stage
        if (!vec || direct) write_back(sp, r0, cc, v);
        store_fp8_general<kDebug>(a, m, dp0, tp, s, t, r0, cc);
        mbar_arrive(empty);
      }
    } else if (fast) {
      mbar_arrive(empty);                         // the block is in registers
      uint8_t* row = dp0.data + 2 * pl0.off;
#pragma unroll
      for (int j = 0; j < kRows; ++j) __stcs(reinterpret_cast<uint4*>(row + 2 * j * pl0.step), v[j]);
    } else if (narrow_fast) {
      mbar_arrive(empty);                         // the block is in registers
      uint8_t* row = dp0.data + 2 * pl0.off;
      const int valid = ncols - cc * 8;
      if (valid > 0)
#pragma unroll
        for (int j = 0; j < kRows; ++j)
          if (r0 + kRowStride * j < nrows) store_bf16_chunk<false>(a, dp0, row + 2 * j * pl0.step, v[j], valid);
    } else {
      if (!vec || direct) {
        bar_sync(bar_id, kGroupThreads);          // every thread has read its slots
        write_back(sp, r0, cc, v);
      }
      store_bf16_general<kDebug>(a, m, dp0, tp, r0, cc);
      mbar_arrive(empty);
    }
  }
}

template <bool kDebug>
__global__ void __launch_bounds__(kCtaThreads, 1) prep_kernel(const __grid_constant__ PrepArgs a) {
  extern __shared__ unsigned char smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  SmemCtl& sm = *reinterpret_cast<SmemCtl*>(stages + (size_t)kStages * kStageStride);
  const int tid = threadIdx.x;
  // without a ticket counter, CTA b takes units first, first + grid, ...
  const int64_t first = a.unit_begin + blockIdx.x;
  const int64_t n_local = first < a.unit_end ? (a.unit_end - first + gridDim.x - 1) / gridDim.x : 0;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), kGroupThreads);
    }
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid >= kConsumerThreads)
    producer(a, a.ticket != nullptr, sm, stages, first, n_local, tid & 31);
  else
    consumer<kDebug>(a, sm, stages, tid / kGroupThreads, tid % kGroupThreads);
  if (!a.ticket) return;
  // the last CTA to finish resets the ticket counter for the next launch:
  // every CTA takes its last ticket before it counts itself done
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.ticket + 1, 1u) == gridDim.x - 1) {
      *reinterpret_cast<volatile uint32_t*>(a.ticket) = 0u;
      *reinterpret_cast<volatile uint32_t*>(a.ticket + 1) = 0u;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t prep_kernel_setup() {
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(prep_kernel<false>, attr, (int)kSmemBytes)) != cudaSuccess) return e;
  return cudaFuncSetAttribute(prep_kernel<true>, attr, (int)kSmemBytes);
}

cudaError_t launch_prepare(const PrepArgs& a, int grid, cudaStream_t s, bool debug, bool pdl) {
  if (a.unit_end <= a.unit_begin) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kCtaThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return debug ? cudaLaunchKernelEx(&cfg, prep_kernel<true>, a) : cudaLaunchKernelEx(&cfg, prep_kernel<false>, a);
}

}  // namespace wt
