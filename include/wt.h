/*
 * wt.h -- C ABI of the B300 parameter-preparation library.
 *
 * The stage this library runs is "parameter preparation" from the page
 * "Weight transfer for RL post-training in under 2 seconds" (Perplexity):
 *   - section "Task pipeline": per parameter, rebuild the full weight from
 *     its shards (full_tensor()), apply projection fusion, quantize if the
 *     destination needs it;
 *   - section "DeviceMesh and mesh groups": parameters are FSDP-sharded
 *     along dim 0;
 *   - section "High-level workflow" and "Why it is fast and simple /
 *     static schedule": the controller computes a static transfer schedule
 *     once at start-up and every step only replays it;
 *   - section "RDMA WRITE: one-sided transfers": a write is addressed by a
 *     destination memory region and an offset in it.
 * The inference side stores FP8 (page intro). Here FP8 means e4m3 ("fn":
 * bias 7, no infinities, largest finite 448) with one fp32 scale per
 * 128x128 block: scale = amax/448 (1.0 for an all-zero block), each code =
 * e4m3_rne_satfinite(x / scale) with an IEEE binary32 division.
 *
 * Destination "memory regions" are caller-owned device buffers ("pools"),
 * one per destination rank, on the plan's device. The remote RDMA write of
 * the pages is out of scope: the library's coalesced stores into the pools
 * stand in for it.
 *
 * Conventions for every call:
 *   - Every call returns wt_status. Out-parameters are written only on
 *     WT_OK. wt_last_error() gives a human-readable detail for the calling
 *     thread's last failure.
 *   - Device pointers are plain addresses on the plan's device. Streams are
 *     cudaStream_t values passed as void* (NULL = the legacy default
 *     stream).
 *   - Nothing here synchronises the device unless documented.
 */
#ifndef WT_H
#define WT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WT_OK = 0,
  WT_ERR_INVALID_ARGUMENT = 1, /* null/out-of-range argument, bad index      */
  WT_ERR_SHAPE = 2,            /* shard rows do not sum, fused cols differ   */
  WT_ERR_LAYOUT_OVERLAP = 3,   /* destination ranges intersect               */
  WT_ERR_POOL_TOO_SMALL = 4,   /* layout exceeds a given pool capacity       */
  WT_ERR_ALIGNMENT = 5,        /* pointer/offset not aligned as required     */
  WT_ERR_OUT_OF_MEMORY = 6,    /* device or pinned allocation failed         */
  WT_ERR_CUDA = 7,             /* a CUDA runtime call failed                 */
  WT_ERR_TIMEOUT = 8,          /* a bounded wait gave up                     */
  WT_ERR_INTERNAL = 9          /* a debug check in a kernel fired            */
} wt_status;

typedef enum {
  WT_OUT_BF16 = 0,          /* pass-through: the fused BF16 bytes           */
  WT_OUT_FP8_E4M3_B128 = 1  /* e4m3 codes + fp32 scale per 128x128 block    */
} wt_out_format;

/* An offset that the plan chooses (auto-pack). */
#define WT_OFFSET_AUTO UINT64_MAX

/* Plan flags. */
/* Testing: treat every output's rows as not 16-byte aligned and copy them
 * one row at a time (no tensor or view maps), the path that rows from
 * several shards and unaligned shards take. */
#define WT_FLAG_FORCE_NARROW 0x1u
#define WT_FLAG_DEBUG_CHECKS 0x2u /* bounds-check every store; see wt_plan_check   */
/* Shard-local plan (FSDP rank `local_shard` prepares the blocks its own
 * shards hold, with no exchange): see wt_plan_desc.local_shard. */
#define WT_FLAG_SHARD_LOCAL 0x4u
/* With WT_FLAG_SHARD_LOCAL: shard boundaries may lie off the 128-row grid.
 * A block row then belongs to the shard holding its first row, and the
 * rank also reads the leading rows of the following shards that the block
 * spans (its halo, at most 127 rows per boundary, never a whole gather);
 * wt_plan_shard_rows_read says how many rows of each shard. */
#define WT_FLAG_SHARD_HALO 0x8u

/* One source parameter: a rows x cols BF16 row-major tensor split along
 * dim 0 into num_shards contiguous shards of shard_rows[i] rows each
 * (FSDP placement; a shard may hold 0 rows). A 1-D tensor is cols = 1. */
typedef struct {
  const char* name;         /* optional, for messages; may be NULL */
  int64_t rows, cols;
  int32_t num_shards;
  const int64_t* shard_rows;
} wt_param_desc;

/* The part of an output that one destination takes, for tensor-parallel
 * inference layouts (the pages map 256 training GPUs onto 128 inference
 * GPUs, each holding its shard of every layer): the listed row ranges
 * (dim 0: column-parallel layers such as qkv or gate_up, one range per
 * fusion part) or column ranges (dim 1: row-parallel layers such as o or
 * down) of the fused tensor, concatenated in order. The destination holds
 * that tensor (row-major, no padding) and, for FP8, the matching block rows
 * or block columns of the scale grid. Every range starts at a multiple of
 * 128 and is a multiple of 128 long, except that the last range may end at
 * the tensor's edge; ranges do not overlap. num_ranges == 0: the whole
 * tensor. */
typedef struct {
  int32_t dim;              /* 0: rows, 1: columns */
  int32_t num_ranges;
  const int64_t* begin;     /* first row / column of each range */
  const int64_t* length;    /* rows / columns of each range */
} wt_slice_desc;

/* One output tensor: the row concatenation of part_params in that order
 * (projection fusion: q,k,v -> qkv; gate,up -> gate_up), written in
 * `format` to each of num_dsts destinations (rank, data offset, scale
 * offset). dst_data_off / dst_scale_off may be NULL (all automatic) or hold
 * WT_OFFSET_AUTO entries. Explicit data offsets must be multiples of 16,
 * explicit scale offsets multiples of 4.
 *
 * dst_slices may be NULL (every destination takes the whole tensor) or hold
 * one wt_slice_desc per destination.
 *
 * Destination layout of an output (or slice) of M x N:
 *   FP8 : M*N code bytes, row-major, no padding inside the tensor, at
 *         data_off; ceil(M/128) x ceil(N/128) fp32 scales, row-major,
 *         little-endian, at scale_off. Blocks are aligned to the fused
 *         tensor's origin; edge blocks cover only the valid elements.
 *   BF16: M*N*2 bytes, row-major, at data_off (scale_off unused).
 * Automatic offsets: per rank, outputs in plan order, each destination on
 * that rank gets its data at the next 256-byte boundary, then (FP8) its
 * scales at the next 256-byte boundary, all after the end of any
 * explicitly placed range on that rank. */
typedef struct {
  const char* name;
  int32_t num_parts;
  const int32_t* part_params;
  int32_t format;           /* wt_out_format */
  int32_t num_dsts;
  const int32_t* dst_ranks;
  const uint64_t* dst_data_off;
  const uint64_t* dst_scale_off;
  const wt_slice_desc* dst_slices;
} wt_output_desc;

/* The whole static schedule. Every param must be used by exactly one
 * output. pool_capacity (NULL = unchecked) bounds each rank's pool size.
 * offload_chunk_bytes > 0 enables wt_prepare_offload: the plan then owns two
 * device staging buffers of the largest chunk's size (the GPU-memory
 * watermark of the page's section "GPU memory usage control"). */
typedef struct {
  int32_t num_params;
  const wt_param_desc* params;
  int32_t num_outputs;
  const wt_output_desc* outputs;
  int32_t num_ranks;
  const uint64_t* pool_capacity;
  uint64_t offload_chunk_bytes;
  uint32_t flags;
  /* With WT_FLAG_SHARD_LOCAL (ignored otherwise): the shard index this plan
   * reads. The plan then holds only the 128-row block rows of each output
   * that lie wholly in shard `local_shard` of their part, so that FSDP rank
   * r, holding shard r of every param, quantizes its own rows without
   * gathering the others' (the 128x128 scale never mixes rows of two
   * shards). Plans for local_shard = 0 .. S-1 together write exactly what
   * the full plan writes, each block once. Needs every shard boundary of
   * every part on a multiple of 128 rows of its output (else
   * WT_ERR_SHAPE) unless WT_FLAG_SHARD_HALO is set, in which case a block
   * row belongs to the shard of its first row and the plan reads halo rows
   * of the next shards; excludes offload_chunk_bytes. Layout, pool sizes and
   * host offsets are those of the full plan; stats, expected counts and
   * the units run are the local ones; shard pointers of other indices may
   * be NULL (see wt_plan_shard_rows_read). WT_ERR_INVALID_ARGUMENT for a
   * negative local_shard, for offload_chunk_bytes > 0, or for
   * WT_FLAG_SHARD_HALO without WT_FLAG_SHARD_LOCAL; a local_shard past a
   * parameter's last shard simply selects none of its rows. */
  int32_t local_shard;
} wt_plan_desc;

typedef struct wt_plan wt_plan;

/* Plan statistics (algorithmic sizes of one wt_prepare). */
typedef struct {
  int64_t num_units;          /* 128x128 tiles this plan runs                 */
  int64_t num_params_total;   /* elements those tiles read                    */
  uint64_t bytes_read;        /* BF16 source bytes per pass                   */
  uint64_t bytes_written;     /* destination bytes per pass (all dsts)        */
  uint64_t host_bytes;        /* size of the packed pinned image (offload)    */
  int32_t num_chunks;         /* offload chunks (0 if offload is disabled)    */
  int32_t num_slots;          /* total shards = length of shard_ptrs          */
} wt_plan_stats;

/* Compile the static schedule (the page's "schedule computed once at
 * initialization"). Validates the descriptor, resolves fusion groups and
 * destination offsets, proves destination ranges disjoint, enumerates the
 * 128x128 work units, and (device >= 0) uploads the tables to that device.
 * device = -1 builds a host-only plan: layout queries work, wt_prepare*
 * return WT_ERR_INVALID_ARGUMENT. The descriptor is deep-copied; the caller
 * may free it on return. Errors: WT_ERR_INVALID_ARGUMENT, WT_ERR_SHAPE,
 * WT_ERR_LAYOUT_OVERLAP, WT_ERR_POOL_TOO_SMALL, WT_ERR_ALIGNMENT,
 * WT_ERR_OUT_OF_MEMORY, WT_ERR_CUDA. */
wt_status wt_plan_create(const wt_plan_desc* desc, int device, wt_plan** out);

/* Bytes the pool of `rank` must hold (0 for a rank with no destination).
 * The pool is the destination memory region of "Weight transfer for RL
 * post-training in under 2 seconds", section "RDMA WRITE: one-sided
 * transfers" (the inference side registers it once; every write lands at
 * an offset in it). Errors: WT_ERR_INVALID_ARGUMENT (NULL plan or out
 * pointer, rank out of range). */
wt_status wt_plan_pool_bytes(const wt_plan* p, int32_t rank, uint64_t* bytes);

/* Resolved destination `dst` of output `out`: the rank whose pool holds it
 * and the byte offsets of its data and (FP8) its scale grid in that pool --
 * the (memory region, offset) pair that addresses a one-sided write in
 * "Weight transfer for RL post-training in under 2 seconds", section "RDMA
 * WRITE: one-sided transfers". scale_off is 0 for a BF16 output. Errors:
 * WT_ERR_INVALID_ARGUMENT (NULL argument, index out of range). */
wt_status wt_plan_output_layout(const wt_plan* p, int32_t out, int32_t dst,
                                int32_t* rank, uint64_t* data_off,
                                uint64_t* scale_off);

/* Byte offset of (param, shard) inside the packed pinned-host image used
 * by wt_prepare_offload (the "host-to-device memcpy if FSDP offloads to
 * CPU" stage, "Weight transfer for RL post-training in under 2 seconds",
 * section "Task pipeline"). The image holds the params in the order their
 * outputs appear (parts in fusion order), each param's shards in order,
 * every shard starting at a 256-byte boundary. Errors:
 * WT_ERR_INVALID_ARGUMENT (NULL argument, index out of range). */
wt_status wt_plan_shard_host_offset(const wt_plan* p, int32_t param,
                                    int32_t shard, uint64_t* off);

/* How many leading rows of (param, shard) one step of this plan reads:
 * every row for a full plan; for a shard-local plan (the FSDP placement of
 * "Weight transfer for RL post-training in under 2 seconds", section
 * "DeviceMesh and mesh groups"), every row of the shards of its own index,
 * the halo rows of the shards its blocks span into (WT_FLAG_SHARD_HALO),
 * 0 otherwise. A shard with 0 rows read may be NULL in wt_prepare; one
 * with r < shard_rows rows read needs only its first r rows valid at the
 * pointer passed (a halo buffer received from the rank that holds the
 * shard). Errors: WT_ERR_INVALID_ARGUMENT (NULL argument, index out of
 * range). */
wt_status wt_plan_shard_rows_read(const wt_plan* p, int32_t param, int32_t shard,
                                  int64_t* rows);

/* Algorithmic sizes of one step of this plan (what a roofline divides by).
 * No counterpart on the pages. Errors: WT_ERR_INVALID_ARGUMENT (NULL
 * argument). */
wt_status wt_plan_get_stats(const wt_plan* p, wt_plan_stats* stats);

/* One step: run the preparation of every output on `stream` -- the
 * page's per-step work ("Weight transfer for RL post-training in under 2
 * seconds", section "Task pipeline": rebuild each weight from its FSDP
 * shards, fuse projections, quantize where the destination wants FP8),
 * replaying the schedule compiled once by wt_plan_create (same page,
 * sections "High-level workflow" and "Why it is fast and simple" / static
 * schedule), with every write addressed by (pool, offset) as in its
 * section "RDMA WRITE: one-sided transfers".
 * shard_ptrs: num_slots device pointers, param-major then shard (the order
 *   of wt_plan_desc.params and their shard_rows); each shard is a
 *   contiguous shard_rows x cols BF16 row-major block. A shard with 0 rows,
 *   or one that a shard-local plan does not read, may be NULL; of a halo
 *   shard only the rows read need be valid (wt_plan_shard_rows_read).
 *   Shards of outputs whose cols are a multiple of 8 must be 16-byte
 *   aligned, the others 2-byte aligned (a 16-byte-aligned one is read
 *   through tensor copies, any other row by row).
 * pools: num_ranks device pointers, each 16-byte aligned, holding at least
 *   wt_plan_pool_bytes bytes (NULL allowed for a 0-byte pool).
 * Shards and pools are borrowed: they must stay valid until the stream
 * work completes. Asynchronous: no allocation, no device synchronisation.
 * The plan keeps the device tables of the last four distinct (shard_ptrs,
 * pools) sets it was given; a call with a known set uploads nothing, a new
 * set replaces the least recently used one with one stream-ordered copy
 * (and tensor maps encoded on the host for the shards that changed). A
 * caller alternating between up to four buffer sets therefore never waits;
 * the only host wait is for the upload of the replaced set, four new sets
 * back. Calls on one plan must be ordered on one stream.
 * CUDA graphs: a call may be captured once an uncaptured call has staged
 * the same shard and pool pointers (a captured call with new pointers
 * returns WT_ERR_INVALID_ARGUMENT). A set that a capture used is kept for
 * the plan's lifetime, so its graph stays valid however many other sets
 * are used later; once all four sets are held by captures, new pointers
 * return WT_ERR_INVALID_ARGUMENT. Finish a graph's replays before
 * destroying the plan.
 * Errors: WT_ERR_INVALID_ARGUMENT (null pointer where data is needed,
 * host-only plan), WT_ERR_ALIGNMENT, WT_ERR_CUDA (a launch or copy failed,
 * including an earlier asynchronous error). */
wt_status wt_prepare(wt_plan* p, const void* const* shard_ptrs,
                     void* const* pools, void* stream);

/* One step for FSDP CPU offload (the page's "host-to-device memcpy if FSDP
 * offloads to CPU" stage, pipelined with preparation): the packed pinned
 * host image (see wt_plan_shard_host_offset) is copied chunk by chunk into
 * the plan's two staging buffers on copy_stream while the preparation of
 * the previous chunk runs on compute_stream. Chunks are greedy runs of whole
 * outputs in plan order, each at most offload_chunk_bytes of image (an
 * output larger than that is a chunk of its own). When the call returns,
 * all work is queued; compute_stream's completion implies the copies'.
 * host_image must be pinned (cudaHostAlloc / cudaHostRegister) and stay
 * untouched until then. Errors: as wt_prepare; WT_ERR_INVALID_ARGUMENT when
 * the plan was built without offload_chunk_bytes. If queueing fails midway
 * the call waits for what it queued and returns the error; the plan stays
 * usable. It cannot be captured into a CUDA graph (WT_ERR_INVALID_ARGUMENT). */
wt_status wt_prepare_offload(wt_plan* p, const void* host_image,
                             void* const* pools, void* copy_stream,
                             void* compute_stream);

/* One step that allocates no device memory. The pages have no counterpart:
 * this exists for callers that cannot call cudaMalloc -- code running
 * inside a memory pool or arena it does not own, or next to an engine that
 * has reserved all device memory up front. Instead of a plan's cudaMalloc'd
 * tables, every call compiles `desc` on the host and copies its schedule
 * tables into one fixed 4 MiB array inside the library image (each device
 * that loads the library holds it until the process exits), then runs the
 * same kernel as wt_prepare on the current device. Arguments and results
 * are those of wt_plan_create(desc) + wt_prepare(shard_ptrs, pools, stream).
 * The first call on a device looks up the array's device address there.
 * Every call shares the array, so calls whose work overlaps on the GPU
 * (different streams) race: order them on one stream. Calls from several
 * host threads onto one stream are safe: a library lock keeps each call's
 * table upload and kernel adjacent. A wait that gives up inside the kernel
 * is recorded outside the tables and kept until wt_noalloc_check reads it.
 * Errors: as wt_plan_create and wt_prepare; WT_ERR_INVALID_ARGUMENT when
 * the tables need more than the array's 4 MiB less 256 bytes (roughly 120k
 * 128x128 blocks), when offload_chunk_bytes is set, with
 * WT_FLAG_DEBUG_CHECKS, or when `stream` is being captured into a CUDA
 * graph (the upload reads a host buffer that lives only for the call).
 * Never calls cudaMalloc or cudaFree. */
wt_status wt_prepare_noalloc(const wt_plan_desc* desc, const void* const* shard_ptrs,
                             void* const* pools, void* stream);

/* The check of wt_prepare_noalloc, allocating nothing either: synchronise
 * `stream`, then read and clear the error word that the kernels of earlier
 * wt_prepare_noalloc calls on the current device share. WT_ERR_TIMEOUT if a
 * wait inside one of them gave up (that step's pools are incomplete),
 * WT_OK otherwise (also before any call on this device). No counterpart on
 * the pages. Errors: WT_ERR_CUDA. */
wt_status wt_noalloc_check(void* stream);

/* Testing hook of wt_prepare_noalloc's bounded waits, like
 * wt_debug_stall_unit for every later wt_prepare_noalloc call of the
 * process: `unit` is never filled and every wait gives up after
 * wait_limit_ns (0 = the default 2 s); unit = -1 restores normal
 * operation. Errors: WT_ERR_INVALID_ARGUMENT (unit < -1). */
wt_status wt_debug_noalloc_stall_unit(int64_t unit, uint64_t wait_limit_ns);

/* The activation codec of the MoE dispatch: the same e4m3 arithmetic at
 * 1 x 128 granularity ("Enabling trillion-parameter models on AWS EFA",
 * dispatch/combine kernels: tokens are sent as block-scaled FP8 at hidden
 * 7168). x: tokens x hidden BF16 on the current device, row stride x_ld
 * elements (x_ld >= hidden). For each token and each group of 128
 * consecutive channels (the last group may be shorter): scale = amax / 448
 * (1.0 for an all-zero group), code = e4m3_rne_satfinite(x / scale) with an
 * IEEE binary32 quotient. codes: tokens x hidden bytes, row-major;
 * scales: tokens x ceil(hidden / 128) fp32, row-major; both caller-owned on
 * the same device. x 2-byte and scales 4-byte aligned; 16-byte-aligned x
 * with hidden and x_ld multiples of 8 (and 8-byte-aligned codes) take the
 * vector path, and of those a large batch with hidden a multiple of 128
 * (contiguous, or rows of at least 4096 channels x_ld apart) is streamed
 * through shared memory by bulk copies, whose waits are bounded: one that
 * gives up leaves that call's output incomplete and is reported by
 * wt_tokens_check.
 * ticket: NULL, or two uint32 words of device memory (4-byte aligned) that
 * are zero before the first call that uses them. Large contiguous batches
 * then hand their shared-memory stages to the SMs one at a time from this
 * counter, so that SMs that are served faster take more (about 3 % faster
 * on a 131072 x 7168 batch); every call leaves the words zero again, also
 * when a wait gives up. Calls that share a ticket must not run at the same
 * time (order them on one stream); NULL gives each SM a fixed share and
 * has no such rule. Other shapes and small batches ignore it.
 * Asynchronous on `stream`, allocates nothing, no plan needed.
 * Errors: WT_ERR_INVALID_ARGUMENT (hidden < 1, x_ld < hidden, NULL buffers,
 * more than 2^31 - 1 groups), WT_ERR_ALIGNMENT, WT_ERR_CUDA. */
wt_status wt_quantize_tokens(const void* x, int64_t tokens, int64_t hidden, int64_t x_ld,
                             void* codes, float* scales, uint32_t* ticket, void* stream);

/* Synchronise `stream`, then read and clear the error word that the
 * kernels of earlier wt_quantize_tokens calls on the current device share:
 * WT_ERR_TIMEOUT if a wait inside one of them gave up (that call's codes
 * and scales are incomplete), WT_OK otherwise (also before any call on this
 * device). No counterpart on the pages. Errors: WT_ERR_CUDA. */
wt_status wt_tokens_check(void* stream);

/* Testing hook of wt_quantize_tokens' bounded waits, for every later call
 * of the process: the shared-memory stage that holds channel group `group`
 * (token t's group g is t * ceil(hidden / 128) + g) is never copied, and
 * every wait gives up after wait_limit_ns (0 = the default 2 s), so the
 * kernel returns with WT_ERR_TIMEOUT recorded; group = -1 restores normal
 * operation. Calls that are not streamed through shared memory ignore it.
 * Errors: WT_ERR_INVALID_ARGUMENT (group < -1). */
wt_status wt_debug_tokens_stall_group(int64_t group, uint64_t wait_limit_ns);

/* Synchronise `stream`, then report what the kernels of earlier
 * wt_prepare* calls recorded, and clear it: WT_ERR_TIMEOUT if a wait inside
 * the kernel gave up (every wait is bounded; the step's output is then
 * incomplete), else, with WT_FLAG_DEBUG_CHECKS, WT_ERR_INTERNAL if a store
 * fell outside its destination range (the offending store is skipped,
 * never performed). WT_OK otherwise. */
wt_status wt_plan_check(wt_plan* p, void* stream);

/* Testing hook: make chunk `chunk` of the next wt_prepare_offload calls
 * fail on the host before it is queued (-1 disables). Exercises the
 * drain-and-report path without touching the GPU. */
wt_status wt_debug_fail_offload_chunk(wt_plan* p, int32_t chunk);

/* Completion counters, the receiving side of the transfer stage: with
 * counters set (a device array of num_ranks uint32, caller-owned and
 * caller-zeroed, on the plan's device; NULL turns counting off), every
 * later wt_prepare / wt_prepare_offload adds, for each 128 x 128 block and
 * each destination holding it, one to counters[rank] once that block's
 * stores to rank are visible device-wide (release at device scope). One
 * step adds wt_plan_expected_count(rank) to each counter; a consumer that
 * waits until counter >= base + expected (modulo 2^32) with an acquire
 * load sees the rank's whole step. The pages' transfer engine counts the
 * immediates of one-sided writes the same way ("RDMA point-to-point
 * communication for LLM systems", ImmCounter). Counts are added by a small
 * stream-ordered kernel after a preparation launch has ended, so the
 * stores they announce are complete; the modes differ in how a step is cut
 * into launches:
 *   WT_COUNT_PER_LAUNCH: wt_prepare runs one launch and adds the whole
 *     step's counts after it.
 *   WT_COUNT_PER_RANK: wt_prepare runs one launch per rank group -- the
 *     blocks whose lowest holding rank is g, for g = 0, 1, ... -- each
 *     followed by its counts, so rank g's counter is complete when group g
 *     ends, before the step does, and the ranks finish one after another
 *     (a sender can start on rank 0 while later ranks are prepared).
 * wt_prepare_offload adds counts after each chunk's launch in both modes.
 * After a launch whose waits gave up (WT_ERR_TIMEOUT), nothing more is
 * counted until wt_plan_check has reported and cleared the error.
 * Errors: WT_ERR_INVALID_ARGUMENT (NULL plan, host-only plan, unknown
 * mode), WT_ERR_ALIGNMENT. */
#define WT_COUNT_PER_LAUNCH 0u
#define WT_COUNT_PER_RANK 1u
wt_status wt_plan_set_counters(wt_plan* p, uint32_t* counters, uint32_t mode);

/* Blocks that `rank` receives per step: the amount one step adds to its
 * completion counter. */
wt_status wt_plan_expected_count(const wt_plan* p, int32_t rank, uint64_t* count);

/* A bounded device-side wait for a consumer: queues on `stream` a kernel
 * that waits until (int32)(counters[i] - targets[i]) >= 0 for every i < n
 * (n <= 1000; targets is a host array, copied at the call), or until
 * limit_ns nanoseconds have passed, and then writes 0 or WT_ERR_TIMEOUT to
 * *status (device memory). Work queued after it on `stream` sees the
 * counted stores. It must not be the only thing that can make the
 * counters advance on a device that cannot run both at once: queue it after
 * the preparation on the same stream, or give it a limit. Errors:
 * WT_ERR_INVALID_ARGUMENT, WT_ERR_ALIGNMENT, WT_ERR_CUDA. */
wt_status wt_wait_counters(const uint32_t* counters, int32_t n, const uint32_t* targets,
                           uint64_t limit_ns, int32_t* status, void* stream);

/* Testing hook for the kernel's bounded waits: the next wt_prepare* calls
 * on this plan never fill the shared-memory stage of work unit `unit`
 * (a 128x128 block, numbered over all outputs in plan order), and every
 * wait inside the kernel gives up after wait_limit_ns (0 = the default of
 * 2 s). The consumers of that stage then stop waiting, the kernel records
 * the timeout, waits (bounded) for its copies in flight, and returns; the
 * next wt_plan_check reports WT_ERR_TIMEOUT and the pools hold an
 * incomplete step. Nothing faults or hangs, and the plan stays usable.
 * unit = -1 restores normal operation. Errors: WT_ERR_INVALID_ARGUMENT. */
wt_status wt_debug_stall_unit(wt_plan* p, int64_t unit, uint64_t wait_limit_ns);

/* Testing hook for the e4m3 convert that every code of the library goes
 * through (round to nearest even, saturating to +-448): it is applied on
 * the current device, on `stream`, to the n fp32 values whose bit patterns
 * are first_bits, first_bits + 1, ..., writing one code per value to
 * `codes` (n bytes of device memory), so that a test can compare it with
 * the CPU definition of the format over every fp32 value. No counterpart
 * on the pages. Errors: WT_ERR_INVALID_ARGUMENT (codes NULL with n > 0,
 * first_bits + n > 2^32), WT_ERR_CUDA. */
wt_status wt_debug_e4m3_encode(uint32_t first_bits, uint64_t n, uint8_t* codes, void* stream);

/* Synchronise the plan's device with the last stream it ran on, then free
 * the plan and everything it owns. NULL is accepted. The pages have no
 * counterpart (their schedule lives as long as the training job). Errors:
 * WT_ERR_CUDA if waiting for the last step failed (the plan is freed
 * anyway). */
wt_status wt_plan_destroy(wt_plan* p);

/* Name of a status code ("WT_OK", "WT_ERR_SHAPE", ...); "WT_ERR_UNKNOWN"
 * for a value outside the enum. A static string. No counterpart on the
 * pages. */
const char* wt_status_string(wt_status s);
/* Detail of the calling thread's last failure (thread-local; valid until
 * that thread's next failing call). No counterpart on the pages. */
const char* wt_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* WT_H */
