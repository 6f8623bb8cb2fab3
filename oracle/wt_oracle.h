/*
 * CPU oracle for the parameter-preparation stage of a train-to-inference
 * weight transfer.
 *
 * TEST INFRASTRUCTURE ONLY. This file and wt_oracle.c are the plain, slow,
 * obviously-correct definition that the CUDA library is checked against.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it. The product library shares no code with it.
 *
 * What it computes follows the stage described on the page
 * "Weight transfer for RL post-training in under 2 seconds" (Perplexity),
 * section "Task pipeline": rebuild each full weight from its FSDP dim-0
 * shards (the full_tensor() step), apply projection fusion, then quantize
 * where the destination wants FP8. The FP8 format (e4m3 "fn"), the 128x128
 * block size and the fp32 scale come from the statement of the stage this
 * code serves; the readings taken where the page is silent are listed in
 * wt_oracle.c next to the code that takes them.
 *
 * Parity status per function (what pins each one in the tests):
 *   wo_e4m3_encode / wo_e4m3_decode : closed-form code table, a brute-force
 *       nearest-code search, exhaustive comparison with torch's e4m3fn cast
 *       over the whole non-saturating fp32 range, and with an independent
 *       nearest-code search over all 2^32 fp32 bit patterns.
 *   wo_tile_scale, wo_quantize_element : numpy float32 division, the
 *       dequantisation error bound, exact-rational brute force.
 *   wo_layout, wo_dst_shape : closed-form pool sizes, disjointness, explicit
 *       offsets; slices against numpy slicing of the whole output.
 *   wo_prepare_output / wo_prepare : torch.cat of the shards (reassembly and
 *       fusion), numpy amax, exact-rational brute force on tiny tensors.
 *   wo_expected_blocks : closed-form counts (round-robin experts, TP
 *       partitions), sums over ranks.
 *   wo_quantize_tokens : exact-rational brute force per group, the
 *       dequantisation error bound, power-of-two scaling invariance.
 */
#ifndef WT_ORACLE_H
#define WT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define WO_OFFSET_AUTO UINT64_MAX

/* One source parameter: rows x cols BF16, split along dim 0 into shards. */
typedef struct {
  int64_t rows, cols;
  int32_t num_shards;
  const int64_t* shard_rows;
} wo_param;

/* The part of an output one destination takes: the listed row ranges
 * (dim 0) or column ranges (dim 1) of the fused tensor, concatenated in
 * order, with the matching block rows / columns of the scale grid.
 * num_ranges == 0 means the whole tensor. Each range starts at a multiple
 * of 128 and is a multiple of 128 long, except that the last range may end
 * at the tensor's edge; ranges do not overlap. */
typedef struct {
  int32_t dim;
  int32_t num_ranges;
  const int64_t* begin;
  const int64_t* length;
} wo_slice;

/* One output tensor: the row concatenation of its parts, written as BF16
 * bytes (fp8 == 0) or as e4m3 codes plus a 128x128 fp32 scale grid
 * (fp8 == 1), once per destination. data_off / scale_off may be NULL or
 * hold WO_OFFSET_AUTO entries, which the layout packs. dst_slice may be
 * NULL (every destination takes the whole tensor) or hold one slice per
 * destination. */
typedef struct {
  int32_t num_parts;
  const int32_t* parts;
  int32_t fp8;
  int32_t num_dsts;
  const int32_t* dst_rank;
  const uint64_t* data_off;
  const uint64_t* scale_off;
  const wo_slice* dst_slice;
} wo_output;

typedef struct {
  int32_t num_params;
  const wo_param* params;
  int32_t num_outputs;
  const wo_output* outputs;
  int32_t num_ranks;
} wo_model;

/* e4m3 "fn": sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinity,
 * 0x7F/0xFF are NaN, largest finite 448. Round to nearest, ties to even,
 * saturating to +-448. */
uint8_t wo_e4m3_encode(float y);
double wo_e4m3_decode(uint8_t code);
void wo_e4m3_encode_array(const float* y, uint8_t* out, int64_t n);
/* Encode every fp32 whose bit pattern lies in [first, first + n). */
void wo_e4m3_encode_bits_range(uint32_t first, int64_t n, uint8_t* out);

/* Exact fp32 value of a BF16 bit pattern. */
float wo_bf16_value(uint16_t bits);
/* Block scale: amax / 448 rounded once to binary32; 1.0 for an all-zero block. */
float wo_tile_scale(float amax);
/* Code of one element: E(fl32(x / s)). */
uint8_t wo_quantize_element(uint16_t x_bits, float s);

/* Output shape after fusion. Returns 0, or -1 if the parts disagree. */
int wo_output_shape(const wo_model* m, int32_t o, int64_t* rows, int64_t* cols);

/* Shape of what destination d of output o holds (its slice, or the whole
 * tensor). Returns 0, or -1 if the slice breaks the rules above. */
int wo_dst_shape(const wo_model* m, int32_t o, int32_t d, int64_t* rows, int64_t* cols);

/* Destination offsets (flat over outputs, then destinations) and pool sizes.
 * Returns 0 or -1 on an invalid model. */
int wo_layout(const wo_model* m, uint64_t* data_off, uint64_t* scale_off,
              uint64_t* pool_bytes);

/* One output, destination independent. shards: flat array over all params
 * of the model (param-major, then shard), NULL allowed for params not used
 * by output o. data_out: rows*cols bytes (FP8) or rows*cols*2 bytes (BF16).
 * scale_out: ceil(rows/128)*ceil(cols/128) floats (FP8 only). */
int wo_prepare_output(const wo_model* m, int32_t o,
                      const uint16_t* const* shards, uint8_t* data_out,
                      float* scale_out);

/* Blocks (128 x 128 units) that rank receives per step: for every
 * destination on that rank, the blocks of the fused tensor it holds (all
 * of them, or the block rows / block columns of its slice). This is what a
 * per-rank completion counter advances by in one step. */
int64_t wo_expected_blocks(const wo_model* m, int32_t rank);

/* The activation codec of the MoE dispatch (the same e4m3 arithmetic at
 * 1 x 128 granularity): x is tokens x hidden BF16 with a row stride of ld
 * elements; for each token and each group of 128 consecutive channels (the
 * last group may be shorter), scale = amax / 448 (1.0 for an all-zero
 * group) and code = E(fl32(x / scale)). codes: tokens x hidden bytes,
 * row-major; scales: tokens x ceil(hidden / 128) floats, row-major. */
void wo_quantize_tokens(const uint16_t* x, int64_t tokens, int64_t hidden, int64_t ld,
                        uint8_t* codes, float* scales);

/* The whole stage into host pools at the given (resolved) offsets, using
 * nthreads worker threads over outputs. */
int wo_prepare(const wo_model* m, const uint64_t* data_off,
               const uint64_t* scale_off, const uint16_t* const* shards,
               uint8_t* const* pools, int32_t nthreads);

#ifdef __cplusplus
}
#endif

#endif
