/*
 * dsa_oracle.c — plain, slow, fp64 CPU oracle for the DSA decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link, load or call this file.  Only
 * the test-suite, the smoke check and the benchmark's CPU-baseline leg use
 * it.  It shares no code, header, table or constant with the CUDA path: the
 * number formats are decoded here from their published definitions, and the
 * paged-cache layout is read from the descriptor values the caller passes.
 *
 * Sources (cited by page title and section):
 *   [K31]  "vLLM 为 Kimi K3.1 Pro 提供 Day-0 支持" (vLLM Day-0 support for
 *          Kimi K3.1 Pro), sections "K3.1 Pro 中的稀疏注意力" (sparse
 *          attention), "为三类状态服务的 KV 缓存" (the packed KV cache),
 *          "量化：原生 MXFP4 索引器" (MXFP4 indexer, AMD section).
 *   [SUM]  "vLLM 对 Kimi K3.1 Pro 的 Day-0 支持：稀疏注意力、DCP 与零失配强化学习"
 *          (agentlens summary), architecture table (32 heads x 128 dims,
 *          FP8 keys, top-2048, NoPE) and the per-token KV byte table.
 *   Formats: OCP 8-bit floating point (E4M3, "fn" variant without infinities)
 *   and the OCP Microscaling (MX) specification (E2M1 elements, E8M0 scales).
 *
 * What is computed (all arithmetic in double precision):
 *   index score   s[t] = sum_h w[h] * max(0, scale_t * (q_h . k_t))
 *                 32 heads x 128 dims; FP8 key + fp32 scale = 132 B per token
 *                 ([K31] sparse-attention section; [SUM] architecture table).
 *                 The ReLU/weighted-head form is DeepSeek-V3.2's lightning
 *                 indexer, which [K31] names as the origin of DSA; the AMD
 *                 section confirms FP32 accumulation and a weighted reduction
 *                 across heads.
 *   MXFP4 keys    k[d] = 2^(E[d/32]-127) * e2m1(code[d]), 128 elements +
 *                 4 E8M0 scales = 68 B per token, no per-token fp32 scale
 *                 ([K31] MXFP4 indexer section: 132 B -> 68 B).
 *   native FP4    MXFP4 keys scored against an MXFP4 query ([K31] MXFP4
 *                 indexer section: scoring uses native FP4 matrix
 *                 instructions; fused-decode section: the front end quantises
 *                 the query to FP8 or MXFP4): q[h][d] = 2^(Q[h][d/32]-127) *
 *                 e2m1(qcode[h][d]).  The query buffer is then codes
 *                 [rows][32][64] (two per byte, low nibble first) followed by
 *                 the E8M0 scales [rows][32][4]; the head weights are used as
 *                 given (the block scales stay with the codes).
 *   top-k         keep the k highest-scoring visible tokens (k = 2048 in the
 *                 model, [K31]); ties go to the lower token index; output in
 *                 ascending token order, padded with -1.
 *   sparse MLA    exact softmax attention of 96 heads over the selected
 *                 tokens' 576-wide latents (absorbed MLA: keys are the full
 *                 576 columns, values the first 512) ([K31]: the attention
 *                 is exact, restricted to the selected tokens).
 *
 * NVFP4 latents ([K31] packed-cache section: 352 B per token instead of 576;
 *                 the layout within the record is a reading of that size):
 *                 dims 0..511 as E2M1 codes with one E4M3 scale per 16 dims
 *                 (256 B + 32 B), dims 512..575 as E4M3 codes (64 B);
 *                 value = latent_scale * e4m3(scale) * e2m1(code), resp.
 *                 latent_scale * e4m3(code).
 *
 * Paged cache ([K31] packed-cache section): a pool of block rows; a block row
 * holds, at caller-given byte offsets, the latent page (64 tokens x 576 B
 * e4m3, or 64 x 352 B NVFP4 records) and the index-key page.  The FP8 index page stores the 64 codes
 * rows (64 x 128 B) followed by the 64 fp32 scales; the MXFP4 page stores
 * 64 x 64 B of packed E2M1 codes followed by 64 x 4 E8M0 scales.  Token t of
 * sequence b lives in block row block_table[b][t / 64], slot t % 64.
 *
 * Visibility: a sequence with nq query rows (speculative-verify draft) and
 * context length L: query row j (0 <= j < nq) sees the first L - (nq-1) + j
 * tokens (causal within the draft; nq = 1 gives L).
 *
 * Pins (tests/test_oracle_pins.py) tie every function here to something other
 * than itself: library decoders, exact integer dot products, closed forms,
 * brute-force selection, and a library softmax on the gathered rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_BLOCK 64          /* tokens per page */
#define ORACLE_IDX_HEADS 32      /* light indexer heads */
#define ORACLE_IDX_DIM 128       /* indexer head dimension */
#define ORACLE_MLA_HEADS 96      /* MLA attention heads */
#define ORACLE_LATENT 576        /* latent width (keys) */
#define ORACLE_VALUE 512         /* value width (first 512 latent columns) */
#define ORACLE_NVFP4_RECORD 352  /* bytes per token of an NVFP4 latent record */

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_BAD_BLOCK = 3 };

/* ------------------------------------------------------------------ */
/* Number formats, decoded from their definitions.                     */
/* ------------------------------------------------------------------ */

/* OCP E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite 448. */
double oracle_e4m3_to_double(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* OCP MX E2M1: 1 sign, 2 exponent (bias 1), 1 mantissa bit; no NaN/inf.
 * Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}. Only the low 4 bits are used. */
double oracle_e2m1_to_double(uint8_t c) {
  int s = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  double v;
  if (e == 0) v = 0.5 * m;
  else v = ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

/* OCP MX E8M0 scale: 2^(E-127); 0xFF is NaN. */
double oracle_e8m0_to_double(uint8_t c) {
  if (c == 0xFF) return NAN;
  return ldexp(1.0, (int)c - 127);
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static float load_f32(const uint8_t* p) {
  float f;
  memcpy(&f, p, 4);
  return f;
}

/* Visible length of query row j of a sequence with context L and nq rows. */
static int64_t visible_len(int64_t L, int nq, int j) {
  int64_t v = L - (nq - 1) + j;
  return v < 0 ? 0 : v;
}

/* Address of the block row holding token t of sequence b, or NULL if the
 * block table entry is outside the pool. */
static const uint8_t* block_row(const uint8_t* pool, int64_t row_stride, int32_t num_blocks,
                                const int32_t* block_table, int32_t max_blocks, int b, int64_t t) {
  int64_t j = t / ORACLE_BLOCK;
  if (j >= max_blocks) return NULL;
  int32_t r = block_table[(int64_t)b * max_blocks + j];
  if (r < 0 || r >= num_blocks) return NULL;
  return pool + (int64_t)r * row_stride;
}

/* ------------------------------------------------------------------ */
/* Lightning indexer scores.                                           */
/* ------------------------------------------------------------------ */

/* The query head (row, h) as 128 doubles.  key_format 0 and 1: E4M3 codes
 * [rows][32][128]; key_format 2 (native FP4): E2M1 codes [rows][32][64]
 * followed by E8M0 scales [rows][32][4]. */
static void query_head(const uint8_t* q_codes, int64_t rows, int32_t key_format, int64_t row, int h,
                       double qv[ORACLE_IDX_DIM]) {
  const int64_t rh = row * ORACLE_IDX_HEADS + h;
  if (key_format != 2) {
    for (int d = 0; d < ORACLE_IDX_DIM; ++d) qv[d] = oracle_e4m3_to_double(q_codes[rh * ORACLE_IDX_DIM + d]);
    return;
  }
  const uint8_t* packed = q_codes + rh * (ORACLE_IDX_DIM / 2);
  const uint8_t* e8 = q_codes + rows * ORACLE_IDX_HEADS * (ORACLE_IDX_DIM / 2) + rh * 4;
  for (int d = 0; d < ORACLE_IDX_DIM; ++d) {
    const uint8_t nib = (d % 2 == 0) ? (packed[d / 2] & 0xF) : (packed[d / 2] >> 4);
    qv[d] = oracle_e8m0_to_double(e8[d / 32]) * oracle_e2m1_to_double(nib);
  }
}

/* raw[h] = q_h . k_t for an MXFP4 key against a native-FP4 query (the
 * products are exact in double; the sum over the four blocks, whose scales
 * may differ widely, is rounded once per addition in double). */
static void raw_dots_native(const uint8_t* q_codes, int64_t rows, int64_t row, const uint8_t* packed,
                            const uint8_t* e8m0, double raw[ORACLE_IDX_HEADS]) {
  double k[ORACLE_IDX_DIM];
  for (int d = 0; d < ORACLE_IDX_DIM; ++d) {
    const uint8_t nib = (d % 2 == 0) ? (packed[d / 2] & 0xF) : (packed[d / 2] >> 4);
    k[d] = oracle_e8m0_to_double(e8m0[d / 32]) * oracle_e2m1_to_double(nib);
  }
  for (int h = 0; h < ORACLE_IDX_HEADS; ++h) {
    double qv[ORACLE_IDX_DIM], acc = 0.0;
    query_head(q_codes, rows, 2, row, h, qv);
    for (int d = 0; d < ORACLE_IDX_DIM; ++d) acc += qv[d] * k[d];
    raw[h] = acc;
  }
}

/* raw[h] = q_h . k_t  for the FP8 key of token t (exact in double: every
 * e4m3 value is a multiple of 2^-9 below 2^9, so each product is a multiple
 * of 2^-18 below 2^18 and a 128-term sum stays far inside 53 bits). */
static void raw_dots_fp8(const uint8_t* q /*[32][128] codes*/, const uint8_t* key /*[128]*/,
                         double raw[ORACLE_IDX_HEADS]) {
  double k[ORACLE_IDX_DIM];
  for (int d = 0; d < ORACLE_IDX_DIM; ++d) k[d] = oracle_e4m3_to_double(key[d]);
  for (int h = 0; h < ORACLE_IDX_HEADS; ++h) {
    double acc = 0.0;
    for (int d = 0; d < ORACLE_IDX_DIM; ++d)
      acc += oracle_e4m3_to_double(q[h * ORACLE_IDX_DIM + d]) * k[d];
    raw[h] = acc;
  }
}

/* raw[h] = q_h . k_t for an MXFP4 key: 128 E2M1 codes packed two per byte
 * (element 2i in the low nibble of byte i, element 2i+1 in the high nibble)
 * and one E8M0 scale per 32 consecutive elements. */
static void raw_dots_mxfp4(const uint8_t* q, const uint8_t* packed /*[64]*/,
                           const uint8_t* e8m0 /*[4]*/, double raw[ORACLE_IDX_HEADS]) {
  double k[ORACLE_IDX_DIM];
  for (int d = 0; d < ORACLE_IDX_DIM; ++d) {
    uint8_t byte = packed[d / 2];
    uint8_t nib = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    k[d] = oracle_e8m0_to_double(e8m0[d / 32]) * oracle_e2m1_to_double(nib);
  }
  for (int h = 0; h < ORACLE_IDX_HEADS; ++h) {
    double acc = 0.0;
    for (int d = 0; d < ORACLE_IDX_DIM; ++d)
      acc += oracle_e4m3_to_double(q[h * ORACLE_IDX_DIM + d]) * k[d];
    raw[h] = acc;
  }
}

/* Scores of every visible token for every query row.
 *   key_format 0: FP8 page = 64 x 128 B codes, then 64 fp32 scales.
 *   key_format 1: MXFP4 page = 64 x 64 B packed codes, then 64 x 4 E8M0.
 *   key_format 2: the MXFP4 page against a native-FP4 query (query_head).
 * scores[row * ld + t] is written for t < visible length; other entries are
 * left untouched.  Returns ORACLE_BAD_BLOCK if a visible token's block-table
 * entry is outside the pool. */
int oracle_index_scores(const uint8_t* pool, int64_t row_stride, int64_t index_off, int32_t num_blocks,
                        int32_t key_format, const int32_t* block_table, int32_t max_blocks,
                        const int32_t* seq_lens, int32_t batch, int32_t nq,
                        const uint8_t* q_codes /*[batch*nq][32][128]*/, const float* head_w /*[batch*nq][32]*/,
                        double* scores, int64_t ld) {
  if (!pool || !block_table || !seq_lens || !q_codes || !head_w || !scores || nq < 1 || batch < 0)
    return ORACLE_BAD_ARG;
  if (key_format < 0 || key_format > 2) return ORACLE_BAD_ARG;
  int bad = 0;
  int64_t rows = (int64_t)batch * nq;
  for (int64_t row = 0; row < rows; ++row) {
    int b = (int)(row / nq), j = (int)(row % nq);
    int64_t vis = visible_len(seq_lens[b], nq, j);
    if (vis > ld) return ORACLE_BAD_ARG;
    const uint8_t* q = q_codes + (key_format == 2 ? 0 : row * ORACLE_IDX_HEADS * ORACLE_IDX_DIM);
    const float* w = head_w + row * ORACLE_IDX_HEADS;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t t = 0; t < vis; ++t) {
      const uint8_t* rowp = block_row(pool, row_stride, num_blocks, block_table, max_blocks, b, t);
      if (!rowp) { bad = 1; continue; }
      const uint8_t* page = rowp + index_off;
      int slot = (int)(t % ORACLE_BLOCK);
      double raw[ORACLE_IDX_HEADS];
      double scale;
      if (key_format == 0) {
        raw_dots_fp8(q, page + slot * ORACLE_IDX_DIM, raw);
        scale = (double)load_f32(page + ORACLE_BLOCK * ORACLE_IDX_DIM + slot * 4);
      } else if (key_format == 2) {
        raw_dots_native(q_codes, rows, row, page + slot * (ORACLE_IDX_DIM / 2),
                        page + ORACLE_BLOCK * (ORACLE_IDX_DIM / 2) + slot * 4, raw);
        scale = 1.0;
      } else {
        raw_dots_mxfp4(q, page + slot * (ORACLE_IDX_DIM / 2),
                       page + ORACLE_BLOCK * (ORACLE_IDX_DIM / 2) + slot * 4, raw);
        scale = 1.0;
      }
      double s = 0.0;
      for (int h = 0; h < ORACLE_IDX_HEADS; ++h) {
        double x = scale * raw[h];
        s += (double)w[h] * (x > 0.0 ? x : 0.0);
      }
      scores[row * ld + t] = s;
    }
  }
  return bad ? ORACLE_BAD_BLOCK : ORACLE_OK;
}

/* Per-token magnitude bound A_t = sum_h |w_h| * |scale_t| * sum_d |q_hd * k_td|
 * (the scale of the rounding error of any evaluation order of the score). */
int oracle_index_score_bounds(const uint8_t* pool, int64_t row_stride, int64_t index_off, int32_t num_blocks,
                              int32_t key_format, const int32_t* block_table, int32_t max_blocks,
                              const int32_t* seq_lens, int32_t batch, int32_t nq,
                              const uint8_t* q_codes, const float* head_w, double* bounds, int64_t ld) {
  if (!pool || !block_table || !seq_lens || !q_codes || !head_w || !bounds || nq < 1) return ORACLE_BAD_ARG;
  if (key_format < 0 || key_format > 2) return ORACLE_BAD_ARG;
  int bad = 0;
  int64_t rows = (int64_t)batch * nq;
  for (int64_t row = 0; row < rows; ++row) {
    int b = (int)(row / nq), j = (int)(row % nq);
    int64_t vis = visible_len(seq_lens[b], nq, j);
    if (vis > ld) return ORACLE_BAD_ARG;
    const float* w = head_w + row * ORACLE_IDX_HEADS;
    double qv[ORACLE_IDX_HEADS][ORACLE_IDX_DIM];
    for (int h = 0; h < ORACLE_IDX_HEADS; ++h) query_head(q_codes, rows, key_format, row, h, qv[h]);
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t t = 0; t < vis; ++t) {
      const uint8_t* rowp = block_row(pool, row_stride, num_blocks, block_table, max_blocks, b, t);
      if (!rowp) { bad = 1; continue; }
      const uint8_t* page = rowp + index_off;
      int slot = (int)(t % ORACLE_BLOCK);
      double k[ORACLE_IDX_DIM], scale;
      if (key_format == 0) {
        for (int d = 0; d < ORACLE_IDX_DIM; ++d) k[d] = oracle_e4m3_to_double(page[slot * ORACLE_IDX_DIM + d]);
        scale = (double)load_f32(page + ORACLE_BLOCK * ORACLE_IDX_DIM + slot * 4);
      } else {
        const uint8_t* packed = page + slot * (ORACLE_IDX_DIM / 2);
        const uint8_t* e8 = page + ORACLE_BLOCK * (ORACLE_IDX_DIM / 2) + slot * 4;
        for (int d = 0; d < ORACLE_IDX_DIM; ++d) {
          uint8_t nib = (d % 2 == 0) ? (packed[d / 2] & 0xF) : (packed[d / 2] >> 4);
          k[d] = oracle_e8m0_to_double(e8[d / 32]) * oracle_e2m1_to_double(nib);
        }
        scale = 1.0;
      }
      double a = 0.0;
      for (int h = 0; h < ORACLE_IDX_HEADS; ++h) {
        double acc = 0.0;
        for (int d = 0; d < ORACLE_IDX_DIM; ++d) acc += fabs(qv[h][d] * k[d]);
        a += fabs((double)w[h]) * fabs(scale) * acc;
      }
      bounds[row * ld + t] = a;
    }
  }
  return bad ? ORACLE_BAD_BLOCK : ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Top-k selection.                                                    */
/* ------------------------------------------------------------------ */

typedef struct { double s; int32_t t; } scored_t;

/* Order: higher score first; NaN ranks below every number; -0 equals +0;
 * equal scores: lower token index first. */
static int by_score_then_index(const void* pa, const void* pb) {
  const scored_t* a = (const scored_t*)pa;
  const scored_t* b = (const scored_t*)pb;
  int an = isnan(a->s), bn = isnan(b->s);
  if (an != bn) return an ? 1 : -1;
  if (!an) {
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
  }
  return (a->t < b->t) ? -1 : (a->t > b->t);
}

static int by_index(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

/* For each row: the min(k, len) best tokens among t < row_lens[row], in
 * ascending token order, then -1 up to k entries. Scores are doubles; fp32
 * scores converted to double keep their exact values and order. */
int oracle_topk(const double* scores, int64_t ld, const int32_t* row_lens, int32_t rows, int32_t k,
                int32_t* idx_out /*[rows][k]*/) {
  if (!scores || !row_lens || !idx_out || k < 1 || rows < 0) return ORACLE_BAD_ARG;
  int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
  for (int32_t row = 0; row < rows; ++row) {
    int64_t len = row_lens[row];
    if (len < 0 || len > ld) { bad = 1; continue; }
    scored_t* all = (scored_t*)malloc(sizeof(scored_t) * (size_t)(len > 0 ? len : 1));
    for (int64_t t = 0; t < len; ++t) { all[t].s = scores[(int64_t)row * ld + t]; all[t].t = (int32_t)t; }
    qsort(all, (size_t)len, sizeof(scored_t), by_score_then_index);
    int64_t n = len < k ? len : k;
    int32_t* out = idx_out + (int64_t)row * k;
    for (int64_t i = 0; i < n; ++i) out[i] = all[i].t;
    qsort(out, (size_t)n, sizeof(int32_t), by_index);
    for (int64_t i = n; i < k; ++i) out[i] = -1;
    free(all);
  }
  return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Decode context parallelism: the exact top-k merge across W shards.  */
/* ------------------------------------------------------------------ */

/* [K31] decode-context-parallelism section.  Shard r of W holds the tokens t
 * with t mod W = r (local position t div W).  Each shard sends its best
 * ceil(1.5 k / W) candidates, chosen on bf16 scores, each packed with its
 * score into one 32-bit word; every shard then selects the same global top-k
 * from the gathered words.  A shard all of whose sent words were selected,
 * and which holds more tokens, may hold more of the top-k than it sent: it
 * resends its full local top-k (min(k, its tokens) words) for that row and
 * the selection runs again (a shard that has sent its full local top-k
 * cannot hold more of a top-k of k tokens).
 * Readings: the word is the 16-bit order key of the bf16-rounded score
 * (round to nearest even) in the upper half and the local position in the
 * lower half, so a shard holds at most 65,536 tokens of a row.  Keys order
 * as the fp32 top-k does (higher first, NaN below every number, -0 = +0) and
 * equal keys go to the lower global token index.  The result is therefore
 * the top-k of the bf16-rounded scores. */
static uint16_t bf16_order_key(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0; /* NaN: below every number */
  uint32_t b = (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16; /* round to nearest even */
  if (b == 0x8000u) b = 0;                            /* -0 = +0 */
  return (uint16_t)((b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u));
}

typedef struct { uint32_t key; int32_t t; } dcp_cand_t;  /* t: global token index */

/* Higher key first; equal keys: lower global index first. */
static int dcp_order(const void* pa, const void* pb) {
  const dcp_cand_t* a = (const dcp_cand_t*)pa;
  const dcp_cand_t* b = (const dcp_cand_t*)pb;
  if (a->key != b->key) return a->key > b->key ? -1 : 1;
  return (a->t < b->t) ? -1 : (a->t > b->t);
}

int oracle_dcp_topk(const float* scores, int64_t ld, const int32_t* row_lens, int32_t rows, int32_t k,
                    int32_t shards, int32_t* idx_out /*[rows][k]*/, int64_t* stats /*[rows][3] or NULL*/) {
  if (!scores || !row_lens || !idx_out || k < 1 || rows < 0 || shards < 1 || shards > 64) return ORACLE_BAD_ARG;
  const int32_t c = (int32_t)((3LL * k + 2LL * shards - 1) / (2LL * shards)); /* ceil(1.5 k / W) */
  int bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(| : bad)
  for (int32_t row = 0; row < rows; ++row) {
    const int64_t len = row_lens[row];
    if (len < 0 || len > ld || (len + shards - 1) / shards > 65536) { bad = 1; continue; }
    const float* srow = scores + (int64_t)row * ld;
    /* every shard's tokens in its own order: (key desc, local asc) */
    dcp_cand_t** local = (dcp_cand_t**)calloc((size_t)shards, sizeof(dcp_cand_t*));
    int64_t* n = (int64_t*)calloc((size_t)shards, sizeof(int64_t));
    int64_t* sent = (int64_t*)calloc((size_t)shards, sizeof(int64_t));
    int64_t* taken = (int64_t*)calloc((size_t)shards, sizeof(int64_t));
    for (int32_t r = 0; r < shards; ++r) {
      n[r] = len > r ? (len - r + shards - 1) / shards : 0;
      local[r] = (dcp_cand_t*)malloc(sizeof(dcp_cand_t) * (size_t)(n[r] > 0 ? n[r] : 1));
      for (int64_t l = 0; l < n[r]; ++l) {
        const int64_t t = l * shards + r;
        /* the word a shard sends: key above, local position below */
        const uint32_t word = ((uint32_t)bf16_order_key(srow[t]) << 16) | (uint32_t)l;
        local[r][l].key = word >> 16;
        local[r][l].t = (int32_t)t;
      }
      qsort(local[r], (size_t)n[r], sizeof(dcp_cand_t), dcp_order);
      sent[r] = n[r] < c ? n[r] : c;
    }
    int64_t words = 0, resent_shards = 0, resent_words = 0;
    for (int32_t r = 0; r < shards; ++r) words += sent[r];
    dcp_cand_t* pool = (dcp_cand_t*)malloc(sizeof(dcp_cand_t) * (size_t)(len > 0 ? len : 1));
    int64_t m = 0, sel = 0;
    for (int round = 0; round < 2; ++round) {
      /* gather every shard's sent words and select the global top-k */
      m = 0;
      for (int32_t r = 0; r < shards; ++r)
        for (int64_t i = 0; i < sent[r]; ++i) pool[m++] = local[r][i];
      qsort(pool, (size_t)m, sizeof(dcp_cand_t), dcp_order);
      sel = m < k ? m : k;
      for (int32_t r = 0; r < shards; ++r) taken[r] = 0;
      for (int64_t i = 0; i < sel; ++i) taken[pool[i].t % shards]++;
      /* a shard whose sent words were all taken, and which sent fewer than its
       * full local top-k, may hold more of the global top-k: it resends */
      int again = 0;
      for (int32_t r = 0; r < shards; ++r)
        if (taken[r] == sent[r] && sent[r] < (n[r] < k ? n[r] : k)) {
          if (round == 1) { bad = 1; }
          const int64_t full = n[r] < k ? n[r] : k;
          resent_shards++;
          resent_words += full;
          sent[r] = full;
          again = 1;
        }
      if (!again) break;
    }
    int32_t* out = idx_out + (int64_t)row * k;
    for (int64_t i = 0; i < sel; ++i) out[i] = pool[i].t;
    qsort(out, (size_t)sel, sizeof(int32_t), by_index);
    for (int64_t i = sel; i < k; ++i) out[i] = -1;
    if (stats) {
      stats[3 * (int64_t)row] = words;
      stats[3 * (int64_t)row + 1] = resent_shards;
      stats[3 * (int64_t)row + 2] = resent_words;
    }
    for (int32_t r = 0; r < shards; ++r) free(local[r]);
    free(local); free(n); free(sent); free(taken); free(pool);
  }
  return bad ? ORACLE_BAD_ARG : ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Exact sparse MLA attention over the selected tokens.                */
/* ------------------------------------------------------------------ */

/* Latent column d of a record, before the per-layer scale: e4m3 for FP8
 * records; for NVFP4 records, dims 0..511 are e4m3(block scale d/16) times
 * e2m1(nibble d: the low nibble of byte d/2 for even d), dims 512..575
 * e4m3 codes after the 256 code bytes and 32 scale bytes. */
static double latent_code_value(const uint8_t* rec, int32_t latent_format, int d) {
  if (latent_format == 0) return oracle_e4m3_to_double(rec[d]);
  if (d < ORACLE_VALUE) {
    const uint8_t nib = (uint8_t)((rec[d / 2] >> (4 * (d & 1))) & 0xF);
    return oracle_e4m3_to_double(rec[ORACLE_VALUE / 2 + d / 16]) * oracle_e2m1_to_double(nib);
  }
  return oracle_e4m3_to_double(rec[ORACLE_VALUE / 2 + ORACLE_VALUE / 16 + (d - ORACLE_VALUE)]);
}

/* For query row `row` (sequence row / nq), head h:
 *   c_i      = latent_scale * value(latent record of t_i)  (576 values; e4m3, or NVFP4)
 *   l_i      = sm_scale * sum_d q[h][d] * c_i[d]
 *   out[h][d]= sum_i softmax(l)_i * c_i[d]   for d < 512
 *   lse[h]   = ln sum_i exp(l_i)             (natural log, scaled logits)
 * over the entries of idx[row] that are >= 0.  With no valid entry the
 * output row is 0 and lse is -inf.  An index that is not a visible token of
 * its sequence, or whose block is outside the pool, is an error. */
int oracle_sparse_mla(const uint8_t* pool, int64_t row_stride, int64_t latent_off, int32_t num_blocks,
                      double latent_scale, const int32_t* block_table, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t batch, int32_t nq,
                      const uint16_t* q_bf16 /*[rows][96][576]*/, const int32_t* idx /*[rows][k]*/, int32_t k,
                      double sm_scale, double* out /*[rows][96][512]*/, double* lse /*[rows][96]*/,
                      int32_t latent_format) {
  if (!pool || !block_table || !seq_lens || !q_bf16 || !idx || !out || !lse || k < 1 || nq < 1 ||
      (latent_format != 0 && latent_format != 1))
    return ORACLE_BAD_ARG;
  const int64_t rec_bytes = latent_format == 0 ? ORACLE_LATENT : ORACLE_NVFP4_RECORD;
  int64_t rows = (int64_t)batch * nq;
  int bad = 0;
#pragma omp parallel for schedule(dynamic) collapse(2) reduction(| : bad)
  for (int64_t row = 0; row < rows; ++row) {
    for (int h = 0; h < ORACLE_MLA_HEADS; ++h) {
      int b = (int)(row / nq), j = (int)(row % nq);
      int64_t vis = visible_len(seq_lens[b], nq, j);
      const int32_t* sel = idx + row * k;
      double q[ORACLE_LATENT];
      for (int d = 0; d < ORACLE_LATENT; ++d)
        q[d] = oracle_bf16_to_double(q_bf16[(row * ORACLE_MLA_HEADS + h) * ORACLE_LATENT + d]);
      double* lg = (double*)malloc(sizeof(double) * (size_t)k);
      const uint8_t** lat = (const uint8_t**)malloc(sizeof(uint8_t*) * (size_t)k);
      int n = 0;
      double m = -INFINITY;
      for (int i = 0; i < k; ++i) {
        int32_t t = sel[i];
        if (t < 0) continue;
        const uint8_t* rowp = (t < vis) ? block_row(pool, row_stride, num_blocks, block_table, max_blocks, b, t) : NULL;
        if (!rowp) { bad = 1; continue; }
        const uint8_t* c = rowp + latent_off + (int64_t)(t % ORACLE_BLOCK) * rec_bytes;
        double dot = 0.0;
        for (int d = 0; d < ORACLE_LATENT; ++d) dot += q[d] * (latent_scale * latent_code_value(c, latent_format, d));
        lg[n] = sm_scale * dot;
        lat[n] = c;
        if (lg[n] > m) m = lg[n];
        ++n;
      }
      double* o = out + (row * ORACLE_MLA_HEADS + h) * ORACLE_VALUE;
      for (int d = 0; d < ORACLE_VALUE; ++d) o[d] = 0.0;
      if (n == 0) {
        lse[row * ORACLE_MLA_HEADS + h] = -INFINITY;
      } else {
        double z = 0.0;
        for (int i = 0; i < n; ++i) z += exp(lg[i] - m);
        for (int i = 0; i < n; ++i) {
          double p = exp(lg[i] - m) / z;
          for (int d = 0; d < ORACLE_VALUE; ++d) o[d] += p * (latent_scale * latent_code_value(lat[i], latent_format, d));
        }
        lse[row * ORACLE_MLA_HEADS + h] = m + log(z);
      }
      free(lg);
      free((void*)lat);
    }
  }
  return bad ? ORACLE_BAD_BLOCK : ORACLE_OK;
}

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif

/* ------------------------------------------------------------------ */
/* New-token cache write and indexer-query quantisation.               */
/* ------------------------------------------------------------------ */
/*
 * The fused decode path of [K31] ("低延迟解码：融合的 DSA 解码路径": the
 * new token's index key and latent are written into the paged cache each
 * step, and the indexer's query is FP8 with its scale folded into the head
 * weights, "为三类状态服务的 KV 缓存" for the packed pages).  Encodings follow
 * their definitions: round to the nearest representable value, ties to the
 * even code, finite inputs beyond the largest magnitude saturate to it, the
 * sign (of zero too) is kept.  Scales are computed in single precision, as
 * the cache stores them: amax / 448 for an FP8 key or query head, and for an
 * MXFP4 block the OCP MX shared exponent floor(log2 amax) - 2 (E8M0 byte
 * exponent + 127; an all-zero block takes byte 0).
 */

/* nearest code by search over the non-negative codes, ties to the even code */
static uint8_t nearest_code(double a, double (*decode)(uint8_t), int ncodes, double maxmag) {
  if (a >= maxmag) {
    for (int c = ncodes - 1; c >= 0; --c)
      if (decode((uint8_t)c) == maxmag) return (uint8_t)c;
  }
  int best = 0;
  double bd = fabs(a - decode(0));
  for (int c = 1; c < ncodes; ++c) {
    const double v = decode((uint8_t)c);
    if (isnan(v)) continue;
    const double d = fabs(a - v);
    if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bd = d;
    }
  }
  return (uint8_t)best;
}

/* OCP E4M3 ("fn") encode; NaN -> 0x7F. */
uint8_t oracle_e4m3_encode(double x) {
  if (isnan(x)) return 0x7F;
  const uint8_t mag = nearest_code(fabs(x), oracle_e4m3_to_double, 0x7F, 448.0);
  return (uint8_t)(mag | (signbit(x) ? 0x80 : 0));
}

/* OCP MX E2M1 encode (4 bits). */
uint8_t oracle_e2m1_encode(double x) {
  const uint8_t mag = nearest_code(fabs(x), oracle_e2m1_to_double, 8, 6.0);
  return (uint8_t)(mag | (signbit(x) ? 0x8 : 0));
}

/* One OCP MX block of 32 values: the shared exponent E = floor(log2 amax) - 2
 * (E2M1's largest exponent is 2) clamped to [-127, 127], -127 for an all-zero
 * block; codes e2m1(x * 2^-E) (exact scaling), two per byte, low nibble
 * first; the scale byte E + 127. */
static void mx_block_encode(const float* x /*[32]*/, uint8_t* packed /*[16]*/, uint8_t* e8) {
  double amax = 0.0;
  for (int d = 0; d < 32; ++d) amax = fmax(amax, fabs((double)x[d]));
  int e = -127;
  if (amax > 0.0) {
    int ex;
    frexp(amax, &ex);  /* amax = m * 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1 */
    e = ex - 1 - 2;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
  }
  uint8_t codes[32];
  for (int d = 0; d < 32; ++d) codes[d] = oracle_e2m1_encode(ldexp((double)x[d], -e));
  for (int d = 0; d < 32; d += 2) packed[d / 2] = (uint8_t)(codes[d] | (codes[d + 1] << 4));
  *e8 = (uint8_t)(e + 127);
}

/* float amax / 448 in single precision; 1 for an all-zero vector */
static float fp8_scale(const float* x, int n) {
  float amax = 0.f;
  for (int i = 0; i < n; ++i) {
    const float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  return amax > 0.f ? amax / 448.0f : 1.0f;
}

/*
 * Writes the nq new tokens of every sequence (context L includes them: token
 * L - nq + j is new row j) into the pool: latent codes e4m3(x / latent_scale)
 * and the index key (FP8: codes e4m3(x / s) with s = amax/448 stored as fp32;
 * MXFP4: per 32 elements E = floor(log2 amax) - 2 clamped to [-127, 127],
 * codes e2m1(x * 2^-E), byte E + 127).  Inputs are bf16 bits:
 * new_latent [batch*nq][576], new_key [batch*nq][128].  Returns 3 for a
 * block-table entry outside the pool.
 * NVFP4 latents (latent_format 1; the scale rule is a reading, the pages give
 * only the record size): per 16 dims of 0..511 the block scale code is
 * e4m3(amax / (6 * latent_scale)) (fp32 quotient; the block's largest
 * magnitude maps to E2M1's largest, 6), the codes are
 * e2m1(x / (latent_scale * e4m3(scale code))) (fp32 product, fp32 quotient),
 * and a block whose scale decodes to 0 gets zero codes; dims 512..575 are
 * e4m3(x / latent_scale) as for FP8 latents.
 */
int oracle_cache_append(uint8_t* pool, int64_t row_stride, int64_t latent_off, int64_t index_off,
                        int32_t num_blocks, int32_t key_format, float latent_scale, const int32_t* block_table,
                        int32_t max_blocks, const int32_t* seq_lens, int32_t batch, int32_t nq,
                        const uint16_t* new_latent, const uint16_t* new_key, int32_t latent_format) {
  if (latent_format != 0 && latent_format != 1) return ORACLE_BAD_ARG;
  for (int b = 0; b < batch; ++b) {
    for (int j = 0; j < nq; ++j) {
      const int64_t t = (int64_t)seq_lens[b] - nq + j;
      if (t < 0) continue;
      const int32_t r = block_table[(int64_t)b * max_blocks + t / ORACLE_BLOCK];
      if (r < 0 || r >= num_blocks) return ORACLE_BAD_BLOCK;
      const int slot = (int)(t % ORACLE_BLOCK);
      uint8_t* row = pool + (int64_t)r * row_stride;
      const int64_t nr = (int64_t)b * nq + j;
      const uint16_t* lat = new_latent + nr * ORACLE_LATENT;
      if (latent_format == 0) {
        for (int d = 0; d < ORACLE_LATENT; ++d) {
          const float x = (float)oracle_bf16_to_double(lat[d]);
          row[latent_off + (int64_t)slot * ORACLE_LATENT + d] = oracle_e4m3_encode((double)(x / latent_scale));
        }
      } else {
        uint8_t* rec = row + latent_off + (int64_t)slot * ORACLE_NVFP4_RECORD;
        for (int blk = 0; blk < ORACLE_VALUE / 16; ++blk) {
          float x[16], amax = 0.f;
          for (int d = 0; d < 16; ++d) {
            x[d] = (float)oracle_bf16_to_double(lat[16 * blk + d]);
            if (fabsf(x[d]) > amax) amax = fabsf(x[d]);
          }
          const uint8_t sc = oracle_e4m3_encode((double)(amax / (6.0f * latent_scale)));
          const float sdec = (float)oracle_e4m3_to_double(sc);
          const float step = latent_scale * sdec;
          uint8_t codes[16];
          for (int d = 0; d < 16; ++d) codes[d] = sdec > 0.f ? oracle_e2m1_encode((double)(x[d] / step)) : 0;
          for (int d = 0; d < 16; d += 2) rec[8 * blk + d / 2] = (uint8_t)(codes[d] | (codes[d + 1] << 4));
          rec[ORACLE_VALUE / 2 + blk] = sc;
        }
        for (int d = ORACLE_VALUE; d < ORACLE_LATENT; ++d) {
          const float x = (float)oracle_bf16_to_double(lat[d]);
          rec[ORACLE_VALUE / 2 + ORACLE_VALUE / 16 + (d - ORACLE_VALUE)] = oracle_e4m3_encode((double)(x / latent_scale));
        }
      }
      float k[ORACLE_IDX_DIM];
      for (int d = 0; d < ORACLE_IDX_DIM; ++d) k[d] = (float)oracle_bf16_to_double(new_key[nr * ORACLE_IDX_DIM + d]);
      uint8_t* page = row + index_off;
      if (key_format == 0) {
        const float s = fp8_scale(k, ORACLE_IDX_DIM);
        for (int d = 0; d < ORACLE_IDX_DIM; ++d)
          page[(int64_t)slot * ORACLE_IDX_DIM + d] = oracle_e4m3_encode((double)(k[d] / s));
        memcpy(page + ORACLE_BLOCK * ORACLE_IDX_DIM + 4 * slot, &s, 4);
      } else {  /* MXFP4 keys (key_format 1 and 2) */
        for (int blk = 0; blk < ORACLE_IDX_DIM / 32; ++blk)
          mx_block_encode(k + 32 * blk, page + (int64_t)slot * (ORACLE_IDX_DIM / 2) + 16 * blk,
                          page + ORACLE_BLOCK * (ORACLE_IDX_DIM / 2) + 4 * slot + blk);
      }
    }
  }
  return ORACLE_OK;
}

/*
 * Indexer query in FP8 per (row, head): s = amax/448 (fp32), codes
 * e4m3(q / s), and the scale folded into the head weight, w_out = w * s
 * (ReLU is positively homogeneous: w max(0, t q.k) = w s max(0, t (q/s).k)).
 */
int oracle_quantize_query(const uint16_t* q, const float* w, int32_t rows, uint8_t* codes, float* w_out) {
  for (int64_t rh = 0; rh < (int64_t)rows * ORACLE_IDX_HEADS; ++rh) {
    float x[ORACLE_IDX_DIM];
    for (int d = 0; d < ORACLE_IDX_DIM; ++d) x[d] = (float)oracle_bf16_to_double(q[rh * ORACLE_IDX_DIM + d]);
    const float s = fp8_scale(x, ORACLE_IDX_DIM);
    for (int d = 0; d < ORACLE_IDX_DIM; ++d) codes[rh * ORACLE_IDX_DIM + d] = oracle_e4m3_encode((double)(x[d] / s));
    w_out[rh] = w[rh] * s;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Fused indexer front end.                                             */
/* ------------------------------------------------------------------ */
/*
 * [K31] "低延迟解码：融合的 DSA 解码路径", second bullet: one kernel does the
 * query norm, the indexer's query projection, its FP8 quantisation with the
 * scale folded into the head weights, and the new token's index key.  The
 * pages name the steps, not their formulas.  Readings:
 *   norm        RMSNorm of the row's compressed query c (width D) with a
 *               learned weight gamma:  xn[i] = c[i] / sqrt(mean_j c[j]^2 + eps)
 *               * gamma[i], rounded to bf16 (the projection's operand type);
 *   projection  q[o] = sum_i W[o][i] * xn[i] for the 32 x 128 outputs
 *               o = h * 128 + d (W: bf16, row-major [4096][D]);
 *   quantise    per (row, head) as oracle_quantize_query, from the fp32 value
 *               of q (the projection's accumulator type): s = amax/448,
 *               codes e4m3(q / s), w_out = w * s, all in single precision;
 *   index key   written with the new latent by oracle_cache_append.
 * Norm and projection are in double precision.
 */

/* fp64 -> nearest bf16 (ties to even), as bf16 bits; values here are far
   from the bf16 range's end (no overflow handling). */
static uint16_t bf16_bits_rne(double x) {
  double r = x;
  if (isfinite(x) && x != 0.0) {
    int e;
    frexp(x, &e);                       /* |x| = m 2^e, m in [0.5, 1) */
    int qe = e - 8;                     /* bf16 keeps 8 significant bits */
    if (qe < -133) qe = -133;           /* subnormal spacing 2^-133 */
    r = rint(ldexp(x, -qe));            /* exact scaling, round half to even */
    r = ldexp(r, qe);
  }
  const float f = (float)r;            /* exact: r is a bf16 value */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

int oracle_rms_norm_bf16(const uint16_t* c, const uint16_t* gamma, int32_t rows, int32_t dim, double eps,
                         uint16_t* xn) {
  if (!c || !gamma || !xn || rows < 0 || dim < 1 || !(eps >= 0.0)) return ORACLE_BAD_ARG;
  for (int64_t r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int i = 0; i < dim; ++i) {
      const double v = oracle_bf16_to_double(c[r * dim + i]);
      ss += v * v;
    }
    const double inv = 1.0 / sqrt(ss / dim + eps);
    for (int i = 0; i < dim; ++i)
      xn[r * dim + i] = bf16_bits_rne(oracle_bf16_to_double(c[r * dim + i]) * inv * oracle_bf16_to_double(gamma[i]));
  }
  return ORACLE_OK;
}

int oracle_index_query_proj(const uint16_t* xn, const uint16_t* w, int32_t rows, int32_t dim, int32_t outs,
                            double* q) {
  if (!xn || !w || !q || rows < 0 || dim < 1 || outs < 1) return ORACLE_BAD_ARG;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t o = 0; o < outs; ++o) {
      double acc = 0.0;
      for (int i = 0; i < dim; ++i)
        acc += oracle_bf16_to_double(w[o * dim + i]) * oracle_bf16_to_double(xn[r * dim + i]);
      q[r * outs + o] = acc;
    }
  return ORACLE_OK;
}

/* oracle_quantize_query on fp32 query values */
int oracle_quantize_query_f32(const float* q, const float* w, int32_t rows, uint8_t* codes, float* w_out) {
  if (!q || !w || !codes || !w_out || rows < 0) return ORACLE_BAD_ARG;
  for (int64_t rh = 0; rh < (int64_t)rows * ORACLE_IDX_HEADS; ++rh) {
    const float* x = q + rh * ORACLE_IDX_DIM;
    const float s = fp8_scale(x, ORACLE_IDX_DIM);
    for (int d = 0; d < ORACLE_IDX_DIM; ++d) codes[rh * ORACLE_IDX_DIM + d] = oracle_e4m3_encode((double)(x[d] / s));
    w_out[rh] = w[rh] * s;
  }
  return ORACLE_OK;
}

/*
 * The indexer query in native FP4 ([K31] fused-decode section: the front end
 * quantises the query to FP8 or MXFP4; MXFP4 indexer section: native FP4
 * scoring), from fp32 values q [rows][32][128]: per (row, head) and 32-dim
 * block the OCP MX encoding of mx_block_encode, as the MXFP4 keys are
 * written.  out: codes [rows][32][64], then E8M0 scales [rows][32][4].  The
 * block scales stay with the codes (the block-scaled product applies them), so
 * the head weights pass through unchanged: w_out = w.
 */
int oracle_quantize_query_mxfp4(const float* q, const float* w, int32_t rows, uint8_t* out, float* w_out) {
  if (!q || !w || !out || !w_out || rows < 0) return ORACLE_BAD_ARG;
  const int64_t heads = (int64_t)rows * ORACLE_IDX_HEADS;
  for (int64_t rh = 0; rh < heads; ++rh) {
    for (int blk = 0; blk < ORACLE_IDX_DIM / 32; ++blk)
      mx_block_encode(q + rh * ORACLE_IDX_DIM + 32 * blk, out + rh * (ORACLE_IDX_DIM / 2) + 16 * blk,
                      out + heads * (ORACLE_IDX_DIM / 2) + rh * 4 + blk);
    w_out[rh] = w[rh];
  }
  return ORACLE_OK;
}

/*
 * Physical KV rows of selected tokens ([K31] "低延迟解码：融合的 DSA 解码路径",
 * fourth bullet: the fused indexer outputs the physical KV rows that the
 * attention reads; "为三类状态服务的 KV 缓存": a block table maps each
 * sequence's logical blocks to pool rows).  Row r belongs to sequence r / nq;
 * token t of it lives in pool row block_table[b][t / 64], slot t % 64, read as
 * the physical row number block_row * 64 + slot.  -1 stays -1.  Returns 3 for
 * a table entry outside 0..num_blocks-1 (that output is -1).
 */
int oracle_phys_rows(const int32_t* block_table, int32_t max_blocks, int32_t num_blocks, int32_t nq,
                     const int32_t* idx, int32_t rows, int32_t k, int32_t* phys) {
  if (!block_table || !idx || !phys || nq < 1 || rows < 0 || k < 1) return ORACLE_BAD_ARG;
  int bad = 0;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t p = 0; p < k; ++p) {
      const int32_t t = idx[r * k + p];
      int32_t v = -1;
      if (t >= 0) {
        if (t / ORACLE_BLOCK >= max_blocks) {
          bad = 1;
        } else {
          const int32_t row = block_table[(r / nq) * max_blocks + t / ORACLE_BLOCK];
          if (row < 0 || row >= num_blocks)
            bad = 1;
          else
            v = row * ORACLE_BLOCK + t % ORACLE_BLOCK;
        }
      }
      phys[r * k + p] = v;
    }
  return bad ? ORACLE_BAD_BLOCK : ORACLE_OK;
}
