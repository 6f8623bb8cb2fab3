/*
 * CPU oracle for the parameter-preparation stage. TEST INFRASTRUCTURE ONLY:
 * loaded by the tests, the smoke check and the benchmark's CPU-baseline leg,
 * never by the product library. See wt_oracle.h for what pins each function.
 *
 * Source of the method: "Weight transfer for RL post-training in under 2
 * seconds" (Perplexity), section "Task pipeline" (parameter preparation =
 * rebuild with full_tensor(), projection fusion, quantize if needed) and
 * section "DeviceMesh and mesh groups" (parameters are FSDP-placed; the full
 * tensor is rebuilt from its shards). The intro of the same page fixes the
 * direction: BF16 on the training side, FP8 on the inference side.
 *
 * Readings taken where the page is silent (each marked READING below):
 *   R1  FP8 = e4m3 "fn" with one fp32 scale per 128x128 block.
 *   R2  Quantize after fusion; blocks are aligned to the fused tensor.
 *   R3  scale = amax / 448 in binary32 round-to-nearest; stored as is;
 *       dequantised value = code * scale.
 *   R4  element = E(fl32(x / scale)): a true division, not a reciprocal.
 *   R5  an all-zero block gets scale 1.0.
 *   R6  E rounds to nearest, ties to even, saturates to +-448, keeps the
 *       sign of zero, and maps NaN to 0x7F with the sign bit kept.
 *   R7  edge blocks: amax over the valid elements only, nothing padded.
 *   R8  fusion order = the order of the parts in the descriptor.
 *   R9  destinations are auto-packed per rank at 256-byte boundaries in
 *       output order (data, then scales), after any explicit ranges.
 *
 * Floating point: every value is formed in double (binary64) and rounded
 * once to binary32 where the method stores a binary32. For a quotient of
 * two binary32 numbers this double rounding gives the correctly rounded
 * binary32 quotient, because 53 >= 2*24 + 2 (Figueroa, "When is double
 * rounding innocuous?", SIGNUM 1995). Build with -ffp-contract=off and
 * without fast-math.
 */
#include "wt_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define TILE 128

/* ------------------------------------------------------------------------ */
/* e4m3 "fn" (READING R1, R6)                                               */
/* ------------------------------------------------------------------------ */

double wo_e4m3_decode(uint8_t code) {
  int sign = code >> 7;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);                 /* subnormal: m * 2^-9 */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);          /* normal: 1.m * 2^(e-7) */
  return sign ? -v : v;
}

/* Round a double that is exactly representable to the nearest integer,
 * ties to even (the default IEEE rounding direction). */
static double rne_int(double v) {
  return nearbyint(v);
}

uint8_t wo_e4m3_encode(float yf) {
  uint32_t bits;
  memcpy(&bits, &yf, sizeof bits);
  uint8_t sign = (bits >> 31) ? 0x80 : 0x00;
  if (isnan(yf)) return (uint8_t)(0x7F | sign);
  double a = fabs((double)yf);
  if (a >= 448.0) return (uint8_t)(0x7E | sign);          /* satfinite */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: code = RNE(a / 2^-9); 8 is exactly 0x08 = 2^-6 */
    double m = rne_int(a * 512.0);
    return (uint8_t)((int)m | sign);
  }
  int ex;
  frexp(a, &ex);                    /* a = f * 2^ex, f in [0.5, 1) */
  int e = ex - 1;                   /* floor(log2 a), in [-6, 8] */
  double frac = a / ldexp(1.0, e) - 1.0;   /* exact, in [0, 1) */
  double m = rne_int(frac * 8.0);
  if (m == 8.0) {
    e += 1;
    m = 0.0;
  }
  /* a < 448 keeps e <= 8 and the code below 0x7F */
  return (uint8_t)((((e + 7) << 3) | (int)m) | sign);
}

void wo_e4m3_encode_array(const float* y, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = wo_e4m3_encode(y[i]);
}

void wo_e4m3_encode_bits_range(uint32_t first, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    uint32_t b = first + (uint32_t)i;
    float y;
    memcpy(&y, &b, sizeof y);
    out[i] = wo_e4m3_encode(y);
  }
}

/* ------------------------------------------------------------------------ */
/* BF16, scale, element code (READING R3, R4, R5)                           */
/* ------------------------------------------------------------------------ */

float wo_bf16_value(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return f;
}

float wo_tile_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  return (float)((double)amax / 448.0);
}

uint8_t wo_quantize_element(uint16_t x_bits, float s) {
  double x = (double)wo_bf16_value(x_bits);
  float y = (float)(x / (double)s);
  return wo_e4m3_encode(y);
}

/* ------------------------------------------------------------------------ */
/* Shapes and layout (READING R8, R9)                                       */
/* ------------------------------------------------------------------------ */

static int64_t shard_base_index(const wo_model* m, int32_t p) {
  int64_t k = 0;
  for (int32_t q = 0; q < p; ++q) k += m->params[q].num_shards;
  return k;
}

int wo_output_shape(const wo_model* m, int32_t o, int64_t* rows,
                    int64_t* cols) {
  const wo_output* out = &m->outputs[o];
  int64_t r = 0, c = -1;
  for (int32_t i = 0; i < out->num_parts; ++i) {
    const wo_param* p = &m->params[out->parts[i]];
    if (c < 0) c = p->cols;
    if (p->cols != c) return -1;
    r += p->rows;
  }
  if (c < 0) return -1;
  *rows = r;
  *cols = c;
  return 0;
}

static uint64_t align256(uint64_t v) { return (v + 255u) & ~(uint64_t)255u; }

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

static uint64_t data_bytes(const wo_output* out, int64_t r, int64_t c) {
  return (uint64_t)(r * c) * (out->fp8 ? 1u : 2u);
}

static uint64_t scale_bytes(const wo_output* out, int64_t r, int64_t c) {
  return out->fp8 ? (uint64_t)(ceil_div(r, TILE) * ceil_div(c, TILE)) * 4u : 0u;
}

/* The slice of destination d, or NULL for the whole tensor. */
static const wo_slice* dst_slice(const wo_output* out, int32_t d) {
  if (!out->dst_slice || out->dst_slice[d].num_ranges == 0) return NULL;
  return &out->dst_slice[d];
}

/* READING (tensor-parallel destinations): a destination may take 128-aligned
 * row ranges (column-parallel layers) or column ranges (row-parallel layers)
 * of the fused tensor; it holds their concatenation. */
int wo_dst_shape(const wo_model* m, int32_t o, int32_t d, int64_t* rows, int64_t* cols) {
  int64_t r, c;
  if (wo_output_shape(m, o, &r, &c)) return -1;
  const wo_slice* sl = dst_slice(&m->outputs[o], d);
  if (!sl) {
    *rows = r;
    *cols = c;
    return 0;
  }
  if (sl->dim != 0 && sl->dim != 1) return -1;
  const int64_t extent = sl->dim == 0 ? r : c;
  int64_t total = 0;
  for (int32_t k = 0; k < sl->num_ranges; ++k) {
    const int64_t b = sl->begin[k], n = sl->length[k];
    if (b < 0 || n < 1 || b % TILE || b + n > extent) return -1;
    if (n % TILE && !(b + n == extent && k == sl->num_ranges - 1)) return -1;
    for (int32_t q = 0; q < k; ++q)   /* no overlap with an earlier range */
      if (b < sl->begin[q] + sl->length[q] && sl->begin[q] < b + n) return -1;
    total += n;
  }
  *rows = sl->dim == 0 ? total : r;
  *cols = sl->dim == 0 ? c : total;
  return 0;
}

int wo_layout(const wo_model* m, uint64_t* data_off, uint64_t* scale_off,
              uint64_t* pool_bytes) {
  for (int32_t rank = 0; rank < m->num_ranks; ++rank) {
    /* first: the end of every explicitly placed range on this rank */
    uint64_t explicit_end = 0;
    for (int32_t o = 0; o < m->num_outputs; ++o) {
      const wo_output* out = &m->outputs[o];
      for (int32_t d = 0; d < out->num_dsts; ++d) {
        int64_t r, c;
        if (wo_dst_shape(m, o, d, &r, &c)) return -1;
        if (out->dst_rank[d] != rank) continue;
        if (out->data_off && out->data_off[d] != WO_OFFSET_AUTO) {
          uint64_t e = out->data_off[d] + data_bytes(out, r, c);
          if (e > explicit_end) explicit_end = e;
        }
        if (out->fp8 && out->scale_off && out->scale_off[d] != WO_OFFSET_AUTO) {
          uint64_t e = out->scale_off[d] + scale_bytes(out, r, c);
          if (e > explicit_end) explicit_end = e;
        }
      }
    }
    /* then: pack the automatic ranges in output order after them */
    uint64_t cursor = explicit_end;
    uint64_t end = explicit_end;
    int64_t flat = 0;
    for (int32_t o = 0; o < m->num_outputs; ++o) {
      const wo_output* out = &m->outputs[o];
      for (int32_t d = 0; d < out->num_dsts; ++d, ++flat) {
        if (out->dst_rank[d] != rank) continue;
        int64_t r, c;
        wo_dst_shape(m, o, d, &r, &c);
        uint64_t doff, soff = 0;
        if (out->data_off && out->data_off[d] != WO_OFFSET_AUTO) {
          doff = out->data_off[d];
        } else {
          doff = align256(cursor);
          cursor = doff + data_bytes(out, r, c);
        }
        if (out->fp8) {
          if (out->scale_off && out->scale_off[d] != WO_OFFSET_AUTO) {
            soff = out->scale_off[d];
          } else {
            soff = align256(cursor);
            cursor = soff + scale_bytes(out, r, c);
          }
        }
        data_off[flat] = doff;
        scale_off[flat] = soff;
        if (doff + data_bytes(out, r, c) > end) end = doff + data_bytes(out, r, c);
        if (out->fp8 && soff + scale_bytes(out, r, c) > end)
          end = soff + scale_bytes(out, r, c);
      }
    }
    pool_bytes[rank] = end ? align256(end) : 0;
  }
  return 0;
}

/* ------------------------------------------------------------------------ */
/* The stage                                                                */
/* ------------------------------------------------------------------------ */

/* Step 1 and 2 of the task pipeline's preparation: rebuild each part from
 * its dim-0 shards (row r of the part is row r - offset(s) of shard s,
 * offset(s) = rows of the shards before s), then stack the parts in order
 * (READING R8). Returns a freshly allocated rows x cols BF16 array. */
static uint16_t* reassemble_and_fuse(const wo_model* m, int32_t o,
                                     const uint16_t* const* shards,
                                     int64_t* rows_out, int64_t* cols_out) {
  int64_t rows, cols;
  if (wo_output_shape(m, o, &rows, &cols)) return NULL;
  uint16_t* t = (uint16_t*)malloc((size_t)(rows * cols) * sizeof(uint16_t) + 1);
  if (!t) return NULL;
  const wo_output* out = &m->outputs[o];
  int64_t row = 0;
  for (int32_t i = 0; i < out->num_parts; ++i) {
    int32_t p = out->parts[i];
    const wo_param* par = &m->params[p];
    int64_t base = shard_base_index(m, p);
    for (int32_t s = 0; s < par->num_shards; ++s) {
      int64_t n = par->shard_rows[s];
      if (n > 0)
        memcpy(t + row * cols, shards[base + s],
               (size_t)(n * cols) * sizeof(uint16_t));
      row += n;
    }
  }
  *rows_out = rows;
  *cols_out = cols;
  return t;
}

int wo_prepare_output(const wo_model* m, int32_t o,
                      const uint16_t* const* shards, uint8_t* data_out,
                      float* scale_out) {
  int64_t rows, cols;
  uint16_t* t = reassemble_and_fuse(m, o, shards, &rows, &cols);
  if (!t) return -1;
  const wo_output* out = &m->outputs[o];
  if (!out->fp8) {
    /* BF16 pass-through: the bytes of the fused tensor, row-major */
    memcpy(data_out, t, (size_t)(rows * cols) * sizeof(uint16_t));
    free(t);
    return 0;
  }
  int64_t tiles_n = ceil_div(cols, TILE);
  for (int64_t bi = 0; bi * TILE < rows; ++bi) {
    for (int64_t bj = 0; bj * TILE < cols; ++bj) {
      int64_t r0 = bi * TILE, r1 = r0 + TILE < rows ? r0 + TILE : rows;
      int64_t c0 = bj * TILE, c1 = c0 + TILE < cols ? c0 + TILE : cols;
      /* amax over the valid elements of the block (READING R7) */
      float amax = 0.0f;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c1; ++c) {
          float a = fabsf(wo_bf16_value(t[r * cols + c]));
          if (a > amax) amax = a;
        }
      float s = wo_tile_scale(amax);
      scale_out[bi * tiles_n + bj] = s;
      for (int64_t r = r0; r < r1; ++r)
        for (int64_t c = c0; c < c1; ++c)
          data_out[r * cols + c] = wo_quantize_element(t[r * cols + c], s);
    }
  }
  free(t);
  return 0;
}

/* Copy the slice sl of a prepared output (data: rows x cols elements of
 * esize bytes; scales: its block grid) into a destination: the ranges'
 * rows or columns, concatenated in order, and the same ranges of block
 * rows or block columns of the grid. */
static void copy_slice(const wo_output* out, const wo_slice* sl, int64_t rows, int64_t cols,
                       const uint8_t* data, const float* scales, uint8_t* dst_data,
                       float* dst_scales) {
  const int64_t es = out->fp8 ? 1 : 2;
  const int64_t tiles_n = ceil_div(cols, TILE), tiles_m = ceil_div(rows, TILE);
  if (sl->dim == 0) {
    int64_t at = 0, sat = 0;
    for (int32_t k = 0; k < sl->num_ranges; ++k) {
      const int64_t b = sl->begin[k], n = sl->length[k];
      memcpy(dst_data + at * cols * es, data + b * cols * es, (size_t)(n * cols * es));
      at += n;
      if (dst_scales) {
        const int64_t nb = ceil_div(n, TILE);
        memcpy(dst_scales + sat * tiles_n, scales + (b / TILE) * tiles_n,
               (size_t)(nb * tiles_n) * sizeof(float));
        sat += nb;
      }
    }
  } else {
    int64_t width = 0, swidth = 0;
    for (int32_t k = 0; k < sl->num_ranges; ++k) {
      width += sl->length[k];
      swidth += ceil_div(sl->length[k], TILE);
    }
    for (int64_t r = 0; r < rows; ++r) {
      int64_t at = 0;
      for (int32_t k = 0; k < sl->num_ranges; ++k) {
        const int64_t b = sl->begin[k], n = sl->length[k];
        memcpy(dst_data + (r * width + at) * es, data + (r * cols + b) * es, (size_t)(n * es));
        at += n;
      }
    }
    if (dst_scales)
      for (int64_t bi = 0; bi < tiles_m; ++bi) {
        int64_t at = 0;
        for (int32_t k = 0; k < sl->num_ranges; ++k) {
          const int64_t nb = ceil_div(sl->length[k], TILE);
          memcpy(dst_scales + bi * swidth + at, scales + bi * tiles_n + sl->begin[k] / TILE,
                 (size_t)nb * sizeof(float));
          at += nb;
        }
      }
  }
}

/* READING (completion counters, the receiver-side immediate counter of the
 * transfer engine page): one count per block landing at a destination. */
int64_t wo_expected_blocks(const wo_model* m, int32_t rank) {
  int64_t total = 0;
  for (int32_t o = 0; o < m->num_outputs; ++o) {
    const wo_output* out = &m->outputs[o];
    int64_t r, c;
    if (wo_output_shape(m, o, &r, &c)) return -1;
    for (int32_t d = 0; d < out->num_dsts; ++d) {
      if (out->dst_rank[d] != rank) continue;
      int64_t bm = ceil_div(r, TILE), bn = ceil_div(c, TILE);
      const wo_slice* sl = dst_slice(out, d);
      if (sl) {
        int64_t nb = 0;
        for (int32_t k = 0; k < sl->num_ranges; ++k) nb += ceil_div(sl->length[k], TILE);
        if (sl->dim == 0) bm = nb; else bn = nb;
      }
      total += bm * bn;
    }
  }
  return total;
}

/* READING (activation codec): the dispatch kernels quantise each token's
 * hidden vector in groups of 128 channels ("block-scaled fp8 dispatch",
 * hidden 7168); the scale and code are those of the weight blocks. */
void wo_quantize_tokens(const uint16_t* x, int64_t tokens, int64_t hidden, int64_t ld,
                        uint8_t* codes, float* scales) {
  const int64_t groups = ceil_div(hidden, TILE);
  for (int64_t t = 0; t < tokens; ++t)
    for (int64_t g = 0; g < groups; ++g) {
      const int64_t c0 = g * TILE, c1 = c0 + TILE < hidden ? c0 + TILE : hidden;
      float amax = 0.0f;
      for (int64_t c = c0; c < c1; ++c) {
        float a = fabsf(wo_bf16_value(x[t * ld + c]));
        if (a > amax) amax = a;
      }
      const float s = wo_tile_scale(amax);
      scales[t * groups + g] = s;
      for (int64_t c = c0; c < c1; ++c) codes[t * hidden + c] = wo_quantize_element(x[t * ld + c], s);
    }
}

typedef struct {
  const wo_model* m;
  const uint64_t* data_off;
  const uint64_t* scale_off;
  const uint16_t* const* shards;
  uint8_t* const* pools;
  int32_t nthreads, tid;
  int status;
} worker_arg;

static void* worker(void* argp) {
  worker_arg* a = (worker_arg*)argp;
  const wo_model* m = a->m;
  for (int32_t o = a->tid; o < m->num_outputs; o += a->nthreads) {
    const wo_output* out = &m->outputs[o];
    int64_t rows, cols;
    if (wo_output_shape(m, o, &rows, &cols)) { a->status = -1; return NULL; }
    uint64_t db = data_bytes(out, rows, cols), sb = scale_bytes(out, rows, cols);
    uint8_t* data = (uint8_t*)malloc(db + 1);
    float* scales = (float*)malloc(sb + 4);
    if (!data || !scales || wo_prepare_output(m, o, a->shards, data, scales)) {
      free(data); free(scales);
      a->status = -1;
      return NULL;
    }
    int64_t flat = 0;
    for (int32_t q = 0; q < o; ++q) flat += m->outputs[q].num_dsts;
    for (int32_t d = 0; d < out->num_dsts; ++d) {
      uint8_t* pool = a->pools[out->dst_rank[d]];
      const wo_slice* sl = dst_slice(out, d);
      if (!sl) {
        memcpy(pool + a->data_off[flat + d], data, db);
        if (out->fp8) memcpy(pool + a->scale_off[flat + d], scales, sb);
      } else {
        copy_slice(out, sl, rows, cols, data, scales, pool + a->data_off[flat + d],
                   out->fp8 ? (float*)(pool + a->scale_off[flat + d]) : NULL);
      }
    }
    free(data);
    free(scales);
  }
  return NULL;
}

int wo_prepare(const wo_model* m, const uint64_t* data_off,
               const uint64_t* scale_off, const uint16_t* const* shards,
               uint8_t* const* pools, int32_t nthreads) {
  if (nthreads < 1) nthreads = 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  worker_arg* args = (worker_arg*)malloc(sizeof(worker_arg) * (size_t)nthreads);
  if (!th || !args) { free(th); free(args); return -1; }
  for (int32_t i = 0; i < nthreads; ++i) {
    worker_arg w = {m, data_off, scale_off, shards, pools, nthreads, i, 0};
    args[i] = w;
    pthread_create(&th[i], NULL, worker, &args[i]);
  }
  int status = 0;
  for (int32_t i = 0; i < nthreads; ++i) {
    pthread_join(th[i], NULL);
    if (args[i].status) status = args[i].status;
  }
  free(th);
  free(args);
  return status;
}
