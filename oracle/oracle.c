/*
 * oracle.c -- plain, slow, fp64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the package's smoke() check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library: it has its own dtype codes, its own
 * element decoders and its own E4M3 encoder.
 *
 * Sources (web pages; cited by title and section):
 *   [ENG26]  "The engineering truth of long-context inference 2026: PagedAttention,
 *            Ring Attention and KV-cache offload from 128K to 1M context"
 *            (blog.lonae.com) -- section 1.1 (KV bytes per token), section 2.2
 *            (block-table pseudocode: pool [num_blocks, 2, L, H, block_size, D],
 *            block_id = token_idx // block_size, offset = token_idx % block_size),
 *            section 3.1 (online softmax: running max m, running sum l,
 *            rescale by exp(m - m_new)).
 *   [UNLOCK] "Unlocking long context: engineering practice for million-token LLM
 *            inference" (ybb.press) -- section 3.1 (physical block pool and
 *            per-sequence block table), section 3.2 (per-tensor FP8 E4M3 KV),
 *            section 4.1 (naive attention softmax(q k^T / sqrt(d)) v).
 *   [MHPN]   long-context article at mhpn.cn (news 2466452) -- section 1.1
 *            (decode: one new query against all n cached K/V), section 3.1
 *            (KV size = 2 x layers x kv_heads x head_dim x seq_len x bytes),
 *            section 3.2 (GQA: a group of query heads shares one KV head).
 *   [SEQPAR] "Sequence-parallel engineering for long-context LLM inference: Ring
 *            Attention and distributed KV cache" (ybb.press) -- section
 *            "numerically stable incremental softmax" (log-sum-exp correction
 *            when merging partial results), "communication cost analysis".
 *   [OFP8]   OCP 8-bit floating point specification (E4M3: bias 7, no
 *            infinities, S.1111.111 is NaN, max finite 448, subnormals m*2^-9).
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - the softmax scale is an explicit argument (the pages use 1/sqrt(d));
 *   - exp is the natural exponential;
 *   - FP8 encode: y = x / scale in IEEE single precision, then round to nearest
 *     E4M3 with ties to even, saturating finite overflow and +-Inf to +-448,
 *     NaN -> 0x7F, -0 keeps its sign;
 *   - a sequence of length 0 (or an empty token range) attends to nothing:
 *     output 0 and log-sum-exp -inf, and it has weight 0 in a merge.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_F32 0
#define OR_F16 1
#define OR_BF16 2
#define OR_E4M3 3

static int or_elem_bytes(int dtype) {
  switch (dtype) {
    case OR_F32: return 4;
    case OR_F16: return 2;
    case OR_BF16: return 2;
    case OR_E4M3: return 1;
    default: return 0;
  }
}

int or_dtype_bytes(int dtype) { return or_elem_bytes(dtype); }

int or_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---- element decoders: each is the format's definition, written out ---- */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double or_f16_to_f64(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, f = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp(1.0 + f / 1024.0, e - 15);
  return s ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double or_bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* [OFP8] E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; S.1111.111 = NaN. */
double or_e4m3_to_f64(uint8_t c) {
  int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);                  /* subnormal: m * 2^-9 */
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

static double or_load(const void* base, size_t idx, int dtype) {
  switch (dtype) {
    case OR_F32: return (double)((const float*)base)[idx];
    case OR_F16: return or_f16_to_f64(((const uint16_t*)base)[idx]);
    case OR_BF16: return or_bf16_to_f64(((const uint16_t*)base)[idx]);
    case OR_E4M3: return or_e4m3_to_f64(((const uint8_t*)base)[idx]);
    default: return NAN;
  }
}

/* ---- [UNLOCK 3.2] per-tensor FP8 E4M3 encode, with the reading above ---- */
uint8_t or_e4m3_encode(float x, float scale) {
  float y = x / scale;                 /* IEEE binary32 division, round to nearest */
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a > 448.0) return sign | 0x7E;   /* saturate, including +-Inf */
  /* spacing of representable values around a */
  double quantum;
  if (a < ldexp(1.0, -6)) {
    quantum = ldexp(1.0, -9);          /* subnormal range (and zero) */
  } else {
    int k;
    frexp(a, &k);                      /* a = f * 2^k, f in [0.5, 1) */
    quantum = ldexp(1.0, (k - 1) - 3); /* 3 mantissa bits below the leading one */
  }
  double r = nearbyint(a / quantum);   /* exact quotient; round half to even */
  double v = r * quantum;
  if (v > 448.0) v = 448.0;
  if (v == 0.0) return sign;
  if (v < ldexp(1.0, -6)) {
    int m = (int)(v / ldexp(1.0, -9));
    return sign | (uint8_t)m;
  }
  int k;
  double f = frexp(v, &k);             /* v = f * 2^k, f in [0.5, 1) */
  int e = (k - 1) + 7;                 /* biased exponent */
  int m = (int)((f * 2.0 - 1.0) * 8.0 + 0.5);
  return sign | (uint8_t)(e << 3) | (uint8_t)m;
}

float or_fp8_scale(double amax);

/* ---- [MHPN 3.1] / [ENG26 1.1] KV bytes: 2 x layers x kv_heads x head_dim x tokens x bytes ---- */
uint64_t or_kv_bytes(uint64_t layers, uint64_t kv_heads, uint64_t head_dim, uint64_t tokens,
                     uint64_t elem_bytes) {
  return 2ull * layers * kv_heads * head_dim * tokens * elem_bytes;
}

/* ---- pool addressing: [ENG26 2.2] pool shape [num_blocks, 2, L, H_kv, block_size, D] ---- */
static size_t or_pool_index(int blk, int kv, int layer, int h, int t, int d,
                            int L, int Hkv, int bs, int D) {
  return (((((size_t)blk * 2 + kv) * L + layer) * Hkv + h) * bs + t) * (size_t)D + d;
}

/* Scale of the E4M3 tile (blk, kv, layer, h): from the block-scale array
 * [NB, 2, L, Hkv] when one is given ([UNLOCK 3.2] block-wise scaling), else the
 * per-tensor scale. */
static float or_tile_scale(const float* block_scales, float tensor_scale, int blk, int kv,
                           int layer, int h, int L, int Hkv) {
  if (!block_scales) return tensor_scale;
  return block_scales[(((size_t)blk * 2 + kv) * L + layer) * Hkv + h];
}

/* Store one token's k or v row [Hkv, D] (dtype in_dtype) into slot (blk, t). */
static void or_store_token(void* pool, int kv_dtype, int L, int Hkv, int bs, int D,
                           int layer, int kv, int blk, int t, const void* src, size_t src_row,
                           int in_dtype, float fp8_scale, const float* block_scales) {
  int eb = or_elem_bytes(kv_dtype);
  for (int h = 0; h < Hkv; ++h) {
    float sc = or_tile_scale(block_scales, fp8_scale, blk, kv, layer, h, L, Hkv);
    for (int d = 0; d < D; ++d) {
      size_t di = or_pool_index(blk, kv, layer, h, t, d, L, Hkv, bs, D);
      size_t si = (src_row * Hkv + h) * (size_t)D + d;
      if (kv_dtype == OR_E4M3) {
        float x = (float)or_load(src, si, in_dtype);   /* f32/f16/bf16 -> f32 is exact */
        ((uint8_t*)pool)[di] = or_e4m3_encode(x, sc);
      } else {
        memcpy((char*)pool + di * eb, (const char*)src + si * eb, (size_t)eb);
      }
    }
  }
}

/*
 * [ENG26 2.2] append_token: for each sequence s, position pos = positions[s],
 * block_id = pos // bs, offset = pos % bs, and
 * pool[table[s][block_id], 0/1, layer, :, offset, :] = k[s], v[s].
 * Block allocation is the caller's job (the table must already hold the block).
 * A negative position means the sequence has no token to append (skipped).
 * Returns 0, or -1 on an invalid dtype pair, -2 on an out-of-range position or block id.
 */
int or_append(void* pool, int kv_dtype, int NB, int L, int Hkv, int bs, int D, int layer,
              const void* k, const void* v, int in_dtype, const int32_t* tables, int max_blocks,
              const int32_t* positions, int B, float k_scale, float v_scale,
              const float* block_scales) {
  if (kv_dtype != OR_E4M3 && in_dtype != kv_dtype) return -1;
  for (int s = 0; s < B; ++s) {
    int pos = positions[s];
    if (pos < 0) continue;
    if (pos / bs >= max_blocks) return -2;
    int blk = tables[(size_t)s * max_blocks + pos / bs];
    if (blk < 0 || blk >= NB) return -2;
    or_store_token(pool, kv_dtype, L, Hkv, bs, D, layer, 0, blk, pos % bs, k, (size_t)s, in_dtype, k_scale, block_scales);
    or_store_token(pool, kv_dtype, L, Hkv, bs, D, layer, 1, blk, pos % bs, v, (size_t)s, in_dtype, v_scale, block_scales);
  }
  return 0;
}

/*
 * Bulk form of the same store for n tokens: token i belongs to sequence
 * seq_ids[i] at position positions[i]; block_id = pos // bs through that
 * sequence's table, offset = pos % bs.  Returns 0, -1 (dtype pair) or -2
 * (sequence, position or block id out of range).
 */
int or_append_tokens(void* pool, int kv_dtype, int NB, int L, int Hkv, int bs, int D, int layer,
                     const void* k, const void* v, int in_dtype, const int32_t* tables,
                     int max_blocks, int B, const int32_t* seq_ids, const int32_t* positions,
                     long long n, float k_scale, float v_scale, const float* block_scales) {
  if (kv_dtype != OR_E4M3 && in_dtype != kv_dtype) return -1;
  for (long long i = 0; i < n; ++i) {
    int s = seq_ids[i], pos = positions[i];
    if (pos < 0) continue;
    if (s < 0 || s >= B || pos / bs >= max_blocks) return -2;
    int blk = tables[(size_t)s * max_blocks + pos / bs];
    if (blk < 0 || blk >= NB) return -2;
    or_store_token(pool, kv_dtype, L, Hkv, bs, D, layer, 0, blk, pos % bs, k, (size_t)i, in_dtype, k_scale, block_scales);
    or_store_token(pool, kv_dtype, L, Hkv, bs, D, layer, 1, blk, pos % bs, v, (size_t)i, in_dtype, v_scale, block_scales);
  }
  return 0;
}

/*
 * [UNLOCK 3.2] block-wise scaling: one fp32 scale per group of group_tokens
 * consecutive token positions of a sequence (the page: one scale per 64-128
 * tokens), per K / V, layer and KV head.  group_tokens is a multiple of bs (0
 * means bs: one scale per block).  A paged pool scatters a group's blocks, so
 * the group's scale is stored in the scale slot of every one of its blocks
 * ([NB, 2, L, Hkv] fp32, the same layout as per-block scales).
 * For every group that the n tokens land in: scale = fp32(amax over those
 * tokens' finite elements) / 448 in IEEE single precision (amax 0 -> 1),
 * written to every block of the group present in the table.  A group is named
 * by its first block (entry pos / group_tokens * group_tokens / bs of the
 * table); groups of several sequences with the same first block (a shared
 * prefix) are one group.  Slots of other blocks are left unchanged.
 * Returns 0, -1 (group size) or -2 (a token, or its group's first block, out of range).
 */
int or_block_scales(float* scales, int NB, int L, int Hkv, int bs, int D, int layer,
                    const void* k, const void* v, int in_dtype, const int32_t* tables,
                    int max_blocks, int B, const int32_t* seq_ids, const int32_t* positions,
                    long long n, int group_tokens) {
  const int S = group_tokens == 0 ? bs : group_tokens;
  if (S < bs || S % bs != 0) return -1;
  const int per = S / bs;                            /* blocks per group */
  size_t tiles = (size_t)NB * 2 * L * Hkv;
  double* amax = (double*)calloc(tiles, sizeof(double));
  char* touched = (char*)calloc(tiles, 1);
  if (!amax || !touched) { free(amax); free(touched); return -3; }
  /* amax per group, kept in the tile of the group's first block */
  for (long long i = 0; i < n; ++i) {
    int s = seq_ids[i], pos = positions[i];
    if (pos < 0) continue;
    if (s < 0 || s >= B || pos / bs >= max_blocks) { free(amax); free(touched); return -2; }
    int blk = tables[(size_t)s * max_blocks + pos / bs];
    int lead = tables[(size_t)s * max_blocks + (pos / S) * per];
    if (blk < 0 || blk >= NB || lead < 0 || lead >= NB) { free(amax); free(touched); return -2; }
    for (int kv = 0; kv < 2; ++kv)
      for (int h = 0; h < Hkv; ++h) {
        size_t tile = (((size_t)lead * 2 + kv) * L + layer) * Hkv + h;
        touched[tile] = 1;
        for (int d = 0; d < D; ++d) {
          double x = fabs(or_load(kv ? v : k, ((size_t)i * Hkv + h) * D + d, in_dtype));
          if (isfinite(x) && x > amax[tile]) amax[tile] = x;   /* NaN, +-Inf left out */
        }
      }
  }
  /* the group's scale into the slot of every block of the group */
  for (long long i = 0; i < n; ++i) {
    int s = seq_ids[i], pos = positions[i];
    if (pos < 0) continue;
    int e0 = (pos / S) * per;
    int lead = tables[(size_t)s * max_blocks + e0];
    for (int e = e0; e < e0 + per && e < max_blocks; ++e) {
      int blk = tables[(size_t)s * max_blocks + e];
      if (blk < 0 || blk >= NB) continue;
      for (int kv = 0; kv < 2; ++kv)
        for (int h = 0; h < Hkv; ++h) {
          size_t lt = (((size_t)lead * 2 + kv) * L + layer) * Hkv + h;
          scales[(((size_t)blk * 2 + kv) * L + layer) * Hkv + h] = or_fp8_scale(amax[lt]);
        }
    }
  }
  free(amax);
  free(touched);
  return 0;
}

/*
 * Decode attention for one (sequence s, query head hq), tokens [tb, te):
 *   [MHPN 3.2]   GQA: kv head = hq / (Hq / Hkv)
 *   [ENG26 2.2]  token j lives at pool[table[s][j / bs], kv, layer, h, j % bs, :]
 *   [UNLOCK 3.2] FP8 elements are decoded and multiplied by the per-tensor scale
 *   [UNLOCK 4.1] s_j = scale * q . k_j ;  w = softmax(s) ;  o = sum_j w_j v_j
 * The softmax is computed with the maximum subtracted, in fp64.  Writes o[D],
 * returns the natural log-sum-exp of the scores (-inf when the range is empty).
 * mutant != 0 plants a deliberate mistake (used only by the tests that show
 * the pins catch such mistakes).
 */
static double or_head(double* o, double* wsum_out, const void* q, int q_dtype, size_t qrow,
                      const void* pool, int kv_dtype, int L, int Hkv, int bs, int D, int Hq,
                      int layer, const int32_t* table_row, int hq, int tb, int te, double scale,
                      double k_scale, double v_scale, const float* block_scales, double* sbuf,
                      int mutant) {
  int G = Hq / Hkv;
  int h = (mutant == 1) ? (hq % Hkv) : (hq / G);
  const int fp8 = kv_dtype == OR_E4M3;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (wsum_out) *wsum_out = 0.0;
  if (te <= tb) return -INFINITY;
  qrow *= (size_t)D;   /* element offset of the query row */
  double m = -INFINITY;
  for (int j = tb; j < te; ++j) {
    int jj = (mutant == 2) ? (j + 1) % (te > tb ? te : 1) : j;
    int blk = table_row[jj / bs];
    int t = jj % bs;
    double ks = fp8 ? or_tile_scale(block_scales, (float)k_scale, blk, 0, layer, h, L, Hkv) : 1.0;
    double acc = 0.0;
    for (int d = 0; d < D; ++d) {
      int dk = (mutant == 3) ? (D - 1 - d) : d;
      acc += or_load(q, qrow + d, q_dtype) *
             (or_load(pool, or_pool_index(blk, 0, layer, h, t, dk, L, Hkv, bs, D), kv_dtype) * ks);
    }
    double sc = (mutant == 4) ? acc : scale * acc;
    sbuf[j - tb] = sc;
    if (sc > m) m = sc;
  }
  double l = 0.0;
  for (int j = tb; j < te; ++j) {
    double w = (mutant == 5) ? exp(m - sbuf[j - tb]) : exp(sbuf[j - tb] - m);
    sbuf[j - tb] = w;
    l += w;
  }
  for (int j = tb; j < te; ++j) {
    double w = sbuf[j - tb] / l;
    if (wsum_out) *wsum_out += w;
    int blk = table_row[j / bs];
    int t = j % bs;
    int kv = (mutant == 6) ? 0 : 1;
    double vs = fp8 ? or_tile_scale(block_scales, (float)v_scale, blk, 1, layer, h, L, Hkv) : 1.0;
    for (int d = 0; d < D; ++d)
      o[d] += w * (or_load(pool, or_pool_index(blk, kv, layer, h, t, d, L, Hkv, bs, D), kv_dtype) * vs);
  }
  return m + log(l);
}

/*
 * Decode attention over a paged pool, fp64.
 *   out   [B, Hq, D] fp64 (rows not in `rows` are left untouched)
 *   lse   [B, Hq] fp64 natural log-sum-exp, or NULL
 *   wsum  [B, Hq] fp64 sum of the softmax weights (an invariant: 1), or NULL
 *   q     [B, Hq, D] in q_dtype
 *   pool  [NB, 2, L, Hkv, bs, D] in kv_dtype
 *   tables [B, max_blocks] int32 ; seq_lens [B] int32
 *   tok_begin / tok_end: per-sequence token range [tb, te) to attend over
 *     (NULL: [0, seq_len)) -- used for split partitions.
 *   rows / n_rows: which flattened (s * Hq + hq) rows to compute (NULL: all).
 * Parallel over rows with OpenMP.  Returns 0, or -1 on invalid geometry,
 * -2 on an out-of-range block id.
 */
int or_decode(double* out, double* lse, double* wsum, const void* q, int q_dtype,
              const void* pool, int kv_dtype, int NB, int L, int Hkv, int bs, int D, int Hq,
              int layer, const int32_t* tables, int max_blocks, const int32_t* seq_lens, int B,
              double scale, double k_scale, double v_scale, const int32_t* tok_begin,
              const int32_t* tok_end, const int32_t* rows, int n_rows, int mutant,
              const float* block_scales) {
  if (Hkv <= 0 || Hq % Hkv != 0 || bs <= 0 || D <= 0 || layer < 0 || layer >= L) return -1;
  long long total = rows ? n_rows : (long long)B * Hq;
  int max_len = 0;
  for (int s = 0; s < B; ++s) {
    int te = tok_end ? tok_end[s] : seq_lens[s];
    if (te > max_len) max_len = te;
    int nblk = (te + bs - 1) / bs;
    if (nblk > max_blocks) return -1;
    for (int i = 0; i < nblk; ++i) {
      int blk = tables[(size_t)s * max_blocks + i];
      if (blk < 0 || blk >= NB) return -2;
    }
  }
  int bad = 0;
#pragma omp parallel
  {
    double* sbuf = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
    if (!sbuf || !o) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (long long r = 0; r < total; ++r) {
        long long row = rows ? rows[r] : r;
        int s = (int)(row / Hq), hq = (int)(row % Hq);
        int tb = tok_begin ? tok_begin[s] : 0;
        int te = tok_end ? tok_end[s] : seq_lens[s];
        double ws = 0.0;
        double l = or_head(o, &ws, q, q_dtype, (size_t)s * Hq + hq, pool, kv_dtype, L, Hkv, bs,
                           D, Hq, layer, tables + (size_t)s * max_blocks, hq, tb, te, scale,
                           k_scale, v_scale, block_scales, sbuf, mutant);
        memcpy(out + (size_t)row * D, o, sizeof(double) * (size_t)D);
        if (lse) lse[row] = l;
        if (wsum) wsum[row] = ws;
      }
    }
    free(sbuf);
    free(o);
  }
  return bad ? -3 : 0;
}

/*
 * Multi-token decode ([UNLOCK 5.2] chunked prefill interleaved with decode,
 * read for a chunk of q_len new tokens): sequence s holds n = seq_lens[s]
 * tokens whose last q_len are the chunk's queries.  Query token i (position
 * n - q_len + i) attends causally over tokens [0, n - q_len + i] -- the plain
 * definition of causal attention, computed per row exactly like or_decode.
 *   q   [B, q_len, Hq, D] ;  out [B, q_len, Hq, D] fp64 ;  lse [B, q_len, Hq] or NULL
 * A query whose position is negative (n < q_len - i) attends to nothing: out 0,
 * lse -inf.  Returns 0, -1 (geometry), -2 (block id out of range).
 */
int or_decode_mq(double* out, double* lse, const void* q, int q_dtype, const void* pool,
                 int kv_dtype, int NB, int L, int Hkv, int bs, int D, int Hq, int layer,
                 const int32_t* tables, int max_blocks, const int32_t* seq_lens, int B, int q_len,
                 double scale, double k_scale, double v_scale, const float* block_scales) {
  if (q_len < 1 || Hkv <= 0 || Hq % Hkv != 0 || layer < 0 || layer >= L) return -1;
  int max_len = 0;
  for (int s = 0; s < B; ++s) {
    int n = seq_lens[s];
    if (n > max_len) max_len = n;
    int nblk = (n + bs - 1) / bs;
    if (nblk > max_blocks) return -1;
    for (int i = 0; i < nblk; ++i) {
      int blk = tables[(size_t)s * max_blocks + i];
      if (blk < 0 || blk >= NB) return -2;
    }
  }
  long long total = (long long)B * q_len * Hq;
  int bad = 0;
#pragma omp parallel
  {
    double* sbuf = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)D);
    if (!sbuf || !o) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (long long r = 0; r < total; ++r) {
        int s = (int)(r / ((long long)q_len * Hq));
        int i = (int)((r / Hq) % q_len);
        int hq = (int)(r % Hq);
        int te = seq_lens[s] - q_len + i + 1;        /* keys 0 .. position of query i */
        if (te < 0) te = 0;
        double l = or_head(o, NULL, q, q_dtype, ((size_t)s * q_len + i) * Hq + hq, pool,
                           kv_dtype, L, Hkv, bs, D, Hq, layer, tables + (size_t)s * max_blocks,
                           hq, 0, te, scale, k_scale, v_scale, block_scales, sbuf, 0);
        memcpy(out + (size_t)r * D, o, sizeof(double) * (size_t)D);
        if (lse) lse[r] = l;
      }
    }
    free(sbuf);
    free(o);
  }
  return bad ? -3 : 0;
}

/*
 * [SEQPAR "numerically stable incremental softmax"] / [ENG26 3.1] merge of
 * partial results over disjoint key ranges.  Partial p of a row carries the
 * normalised output O_p and its natural log-sum-exp lse_p.  With
 * M = max_p lse_p and w_p = exp(lse_p - M):  out = sum_p w_p O_p / sum_p w_p,
 * lse = M + log(sum_p w_p).  A partial with lse = -inf has weight 0; a row
 * whose partials are all -inf gets out = 0, lse = -inf.
 *   part_o [rows, S, D], part_lse [rows, S], out [rows, D], out_lse [rows] or NULL.
 */
void or_merge(double* out, double* out_lse, const double* part_o, const double* part_lse,
              long long rows, int S, int D) {
#pragma omp parallel for schedule(static)
  for (long long r = 0; r < rows; ++r) {
    double M = -INFINITY;
    for (int p = 0; p < S; ++p)
      if (part_lse[r * S + p] > M) M = part_lse[r * S + p];
    double* o = out + r * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (M == -INFINITY) {
      if (out_lse) out_lse[r] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int p = 0; p < S; ++p) {
      double w = exp(part_lse[r * S + p] - M);
      wsum += w;
      for (int d = 0; d < D; ++d) o[d] += w * part_o[(r * S + p) * D + d];
    }
    for (int d = 0; d < D; ++d) o[d] /= wsum;
    if (out_lse) out_lse[r] = M + log(wsum);
  }
}

/* Largest |x| over the n elements' finite values ([UNLOCK 3.2] per-tensor FP8:
 * the scale comes from the tensor's absolute maximum).  NaN and +-Inf are left
 * out: the encoder already maps them to 0x7F and +-448, and a scale must be
 * finite.  0 when no element is finite and nonzero. */
double or_absmax(const void* x, int dtype, long long n) {
  double m = 0.0;
  for (long long i = 0; i < n; ++i) {
    double a = fabs(or_load(x, (size_t)i, dtype));
    if (isfinite(a) && a > m) m = a;
  }
  return m;
}

/* [UNLOCK 3.2] per-tensor FP8 scale from the absolute maximum: amax / 448 (448 is
 * the largest finite E4M3 value, [OFP8]) in IEEE single precision, so that the
 * largest element is stored as +-448; amax = 0 (an all-zero tensor) gives 1. */
float or_fp8_scale(double amax) {
  if (!(amax > 0.0)) return 1.0f;
  float a = (float)amax;                 /* exact: amax is an f32/f16/bf16 value */
  return a / 448.0f;
}

/* Decode an array of elements to fp64 (used by the tests to read pools). */
void or_to_f64(double* out, const void* x, int dtype, long long n, double scale) {
  for (long long i = 0; i < n; ++i) out[i] = or_load(x, (size_t)i, dtype) * scale;
}

/* Vector form of the encoder (the tests run it over every bf16 value). */
void or_e4m3_encode_n(uint8_t* out, const float* x, long long n, float scale) {
  for (long long i = 0; i < n; ++i) out[i] = or_e4m3_encode(x[i], scale);
}
