/*
 * oracle.c — plain, slow, fp64 CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library. It shares no code, header, table
 * or constant with the CUDA path.
 *
 * What it computes (each function below names the passage it follows):
 *  - attention as its defining formula: scores, an exact softmax
 *    (max-subtracted, one pass over the whole context), the weighted sum of
 *    V, the log-sum-exp; no online softmax, no tiling, no reordering beyond
 *    the plain loops. The serving pages name the operation ("flash attention
 *    decode (online softmax, paged KV, GQA)", rvLLM: High-performance LLM
 *    inference in Rust, Kernel Compiler Stack); the online softmax is a way
 *    to compute exactly this result, so the oracle writes the result out.
 *  - K/V reached through the block table (Welcome to vLLM, feature list,
 *    "PagedAttention"; Litellama, Architecture tree, attention_metadata.py).
 *  - the split-KV variant and its log-sum-exp merge (rvLLM, FA3 v3 Attention
 *    Kernel, "split-KV for long context"; rapid_llm README, feature table,
 *    "Decode context parallelism ... merges partial attention by
 *    log-sum-exp"), used to pin that the merge reproduces the unsplit result.
 *  - the causal chunked prefill (Litellama, Features, "Chunked Prefill").
 *  - the rotary position embedding of the new tokens' queries and keys fused
 *    with their cache write (rvLLM, Kernel Compiler Stack, "RoPE + KV cache
 *    write -- fused, no intermediate alloc"; the rotation itself is the
 *    RoFormer rotary embedding: each pair of dims turned by the angle its
 *    cos/sin table row gives for the token's position).
 *  - the cache write with the FP8 E4M3 encode (Litellama, Features, "FP8 KV
 *    Cache"; rvLLM, Kernel Compiler Stack, "RoPE + KV cache write"). The
 *    E4M3 format follows the OCP 8-bit floating point specification (OFP8):
 *    bias 7, no infinities, S.1111.111 is NaN, largest finite 448.
 *
 * Every floating-point value is decoded from its bits by the IEEE-754
 * binary16 / bfloat16 / OFP8 definitions and carried in double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { O_F16 = 0, O_BF16 = 1, O_E4M3 = 2 };

/* ---- number formats -------------------------------------------------- */

/* IEEE-754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double pkvo_f16_value(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)f, -24);               /* f * 2^-14 / 2^10 */
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp((double)(1024 + f), e - 25);          /* (1 + f/2^10) 2^(e-15) */
  return s ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double pkvo_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* OFP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent field 0
 * is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity. */
double pkvo_e4m3_value(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xf, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp((double)(8 + m), e - 10);             /* (1 + m/8) 2^(e-7) */
  return s ? -v : v;
}

/* Round a binary32 value to the nearest E4M3 value, ties to the even code,
 * clamping magnitudes above the largest finite value (448) to 448. The E4M3
 * magnitudes are k * 2^-9 for codes k = 0..8 (subnormals, then 2^-6) and
 * (8 + m) * 2^(x-3) for binade x = -6..8, so one rounding of |y| on the grid
 * of its binade gives the code directly. NaN maps to the NaN code 0x7F. */
uint8_t pkvo_e4m3_encode(float y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    double k = nearbyint(a * 512.0);                   /* grid step 2^-9 */
    return sign | (uint8_t)k;                          /* k <= 8: 8 is 2^-6 */
  }
  int ex;
  frexp(a, &ex);                                       /* a = f 2^ex, f in [.5,1) */
  int x = ex - 1;                                      /* 2^x <= a < 2^(x+1) */
  double k = nearbyint(ldexp(a, 3 - x));               /* grid step 2^(x-3) */
  if (k >= 16.0) { k = 8.0; x += 1; }
  return sign | (uint8_t)(((x + 7) << 3) | ((int)k - 8));
}

/* Round a double to a 16-bit binary format with p significand bits (hidden
 * bit included) and `ebits` exponent bits: bias and largest exponent
 * emax = 2^(ebits-1) - 1, smallest normal exponent emin = 1 - emax. The
 * result is the nearest value, ties to the even significand; magnitudes past
 * the largest finite value round to infinity as IEEE-754 round-to-nearest
 * prescribes; subnormals keep the quantum 2^(emin - p + 1) of the smallest
 * binade. Returns the bit pattern (sign in bit 15). */
static uint16_t round_to_binary16(double v, int p, int ebits) {
  const int fbits = p - 1, emax = (1 << (ebits - 1)) - 1, emin = 1 - emax;
  const uint16_t sign = signbit(v) ? 0x8000u : 0u;
  const uint16_t inf = (uint16_t)(((1u << ebits) - 1u) << fbits);
  if (isnan(v)) return (uint16_t)(inf | (1u << (fbits - 1)));
  double a = fabs(v);
  if (isinf(a)) return sign | inf;
  if (a < ldexp(1.0, emin)) {                          /* subnormal binade */
    double k = nearbyint(ldexp(a, fbits - emin));      /* grid step 2^(emin-fbits) */
    return sign | (uint16_t)k;                         /* k = 2^fbits: smallest normal */
  }
  int ex;
  frexp(a, &ex);
  int x = ex - 1;                                      /* 2^x <= a < 2^(x+1) */
  double k = nearbyint(ldexp(a, fbits - x));           /* k in [2^fbits, 2^p] */
  if (k >= ldexp(1.0, p)) { k = ldexp(1.0, fbits); x += 1; }
  if (x > emax) return sign | inf;
  return sign | (uint16_t)(((unsigned)(x + emax) << fbits) | ((unsigned)k - (1u << fbits)));
}

/* IEEE binary16: 11 significand bits, 5 exponent bits. */
uint16_t pkvo_f16_encode(double v) { return round_to_binary16(v, 11, 5); }

/* bfloat16: 8 significand bits, the 8 exponent bits of binary32. */
uint16_t pkvo_bf16_encode(double v) { return round_to_binary16(v, 8, 8); }

static uint16_t encode16(double v, int dtype) {
  return dtype == O_F16 ? pkvo_f16_encode(v) : pkvo_bf16_encode(v);
}

static double elem(const void* base, int dtype, int64_t i) {
  switch (dtype) {
    case O_F16: return pkvo_f16_value(((const uint16_t*)base)[i]);
    case O_BF16: return pkvo_bf16_value(((const uint16_t*)base)[i]);
    default: return pkvo_e4m3_value(((const uint8_t*)base)[i]);
  }
}

static float elem_f32(const void* base, int dtype, int64_t i) {
  return (float)elem(base, dtype, i);                  /* exact: 16-bit -> fp32 */
}

/* The one accessor of the cache layout [num_blocks, Hkv, BS, D]. */
static int64_t cache_index(int64_t block, int kvh, int off, int d, int Hkv, int BS, int D) {
  return ((block * Hkv + kvh) * (int64_t)BS + off) * D + d;
}

#ifdef _OPENMP
void pkvo_set_threads(int n) { omp_set_num_threads(n > 0 ? n : omp_get_num_procs()); }
int pkvo_get_threads(void) { return omp_get_max_threads(); }
#else
void pkvo_set_threads(int n) { (void)n; }
int pkvo_get_threads(void) { return 1; }
#endif

/* ---- cache write ------------------------------------------------------ */

/* For each token t with slot s >= 0 and each KV head h: the D values go to
 * block s / BS, offset s % BS of head h; a copy of the bits when the cache
 * has the source dtype, else E4M3(x / scale[h]) with x and the quotient in
 * binary32. Returns 0, or -1 if a slot is outside the pool (nothing written
 * for that token). */
int pkvo_reshape_and_cache(const void* key, const void* value, int src_dtype,
                           void* k_cache, void* v_cache, int kv_dtype,
                           const int64_t* slots, int T, int Hkv, int D, int BS,
                           int num_blocks, const float* k_scales, const float* v_scales) {
  int bad = 0;
  for (int t = 0; t < T; ++t) {
    int64_t s = slots[t];
    if (s < 0) continue;
    if (s >= (int64_t)num_blocks * BS) { bad = 1; continue; }
    int64_t blk = s / BS;
    int off = (int)(s % BS);
    for (int h = 0; h < Hkv; ++h) {
      for (int d = 0; d < D; ++d) {
        int64_t src = ((int64_t)t * Hkv + h) * D + d;
        int64_t dst = cache_index(blk, h, off, d, Hkv, BS, D);
        if (kv_dtype == src_dtype) {
          ((uint16_t*)k_cache)[dst] = ((const uint16_t*)key)[src];
          ((uint16_t*)v_cache)[dst] = ((const uint16_t*)value)[src];
        } else {
          float xk = elem_f32(key, src_dtype, src);
          float xv = elem_f32(value, src_dtype, src);
          float yk = xk / k_scales[h];
          float yv = xv / v_scales[h];
          ((uint8_t*)k_cache)[dst] = pkvo_e4m3_encode(yk);
          ((uint8_t*)v_cache)[dst] = pkvo_e4m3_encode(yv);
        }
      }
    }
  }
  return bad ? -1 : 0;
}

/* ---- rotary position embedding ---------------------------------------- */

/* Rotates rows x [T, H, D] (16-bit dtype) by their tokens' positions into
 * out (same shape and dtype). Row cos_sin[pos] holds rot/2 cosines, then
 * rot/2 sines. Pair i (i < rot/2) is dims (i, i + rot/2) when neox is set
 * (the rotate-half convention) and dims (2i, 2i+1) otherwise (interleaved);
 * for pair (x1, x2) with c, s of row pos:
 *   y1 = x1 c - x2 s,   y2 = x2 c + x1 s,
 * both products exact in double (a 16-bit value times a binary32 value needs
 * at most 35 significand bits), one rounding for the sum, then one rounding
 * to the row dtype. Dims from rot on are copied. A token whose position is
 * outside [0, max_pos) is copied unrotated and sets bit 2 of the result. */
int pkvo_rope(const void* x, int dtype, int T, int H, int D, const int64_t* pos,
              const float* cos_sin, int64_t max_pos, int rot, int neox, void* out) {
  int bad = 0;
  const uint16_t* xs = (const uint16_t*)x;
  uint16_t* ys = (uint16_t*)out;
  const int half = rot / 2;
  for (int t = 0; t < T; ++t) {
    const int64_t p = pos[t];
    const int ok = p >= 0 && p < max_pos;
    if (!ok) bad = 2;
    for (int h = 0; h < H; ++h) {
      const int64_t row = ((int64_t)t * H + h) * D;
      for (int d = 0; d < D; ++d) ys[row + d] = xs[row + d];
      if (!ok) continue;
      const float* cs = cos_sin + p * rot;
      for (int i = 0; i < half; ++i) {
        const int d1 = neox ? i : 2 * i;
        const int d2 = neox ? i + half : 2 * i + 1;
        const double x1 = elem(x, dtype, row + d1), x2 = elem(x, dtype, row + d2);
        const double c = (double)cs[i], sn = (double)cs[half + i];
        const double y1 = x1 * c - x2 * sn;
        const double y2 = x2 * c + x1 * sn;
        ys[row + d1] = encode16(y1, dtype);
        ys[row + d2] = encode16(y2, dtype);
      }
    }
  }
  return bad;
}

/* The fused step: rotate the queries (into q_out) and the keys, then write
 * the rotated keys, rounded to the source dtype, and the values into their
 * slots exactly as pkvo_reshape_and_cache does. Tokens with a position
 * outside [0, max_pos) keep their query unrotated and write nothing.
 * Returns a bit set: 1 = some slot outside the pool, 2 = some position
 * outside the table. */
int pkvo_rope_reshape_and_cache(const void* q, const void* key, const void* value, int src_dtype,
                                void* k_cache, void* v_cache, int kv_dtype,
                                const int64_t* slots, const int64_t* pos, const float* cos_sin,
                                int64_t max_pos, int rot, int neox, int T, int Hq, int Hkv,
                                int D, int BS, int num_blocks, const float* k_scales,
                                const float* v_scales, void* q_out) {
  int flags = pkvo_rope(q, src_dtype, T, Hq, D, pos, cos_sin, max_pos, rot, neox, q_out);
  uint16_t* krot = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)T * Hkv * D + 1);
  int64_t* sl = (int64_t*)malloc(sizeof(int64_t) * (size_t)T + 1);
  if (krot == NULL || sl == NULL) { free(krot); free(sl); return -1; }
  flags |= pkvo_rope(key, src_dtype, T, Hkv, D, pos, cos_sin, max_pos, rot, neox, krot);
  for (int t = 0; t < T; ++t) sl[t] = (pos[t] >= 0 && pos[t] < max_pos) ? slots[t] : -1;
  if (pkvo_reshape_and_cache(krot, value, src_dtype, k_cache, v_cache, kv_dtype, sl, T, Hkv, D,
                             BS, num_blocks, k_scales, v_scales) != 0)
    flags |= 1;
  free(krot);
  free(sl);
  return flags;
}

/* ---- attention over one sequence and head ----------------------------- */

typedef struct {
  const void* k_cache; const void* v_cache; int kv_dtype;
  int Hkv, BS, D;
  int64_t num_blocks;
  double k_scale, v_scale;
} kvview;

/* Exact softmax attention of one query vector q[D] (fp64) over logical keys
 * [j0, j1) of the sequence whose block-table row is `table`. Writes the
 * normalised output o[D] and returns the natural-log log-sum-exp of the
 * scores (-inf and o = 0 for an empty range). Sets *bad on an out-of-pool
 * block id. */
static double attend(const kvview* kv, const int32_t* table, int kvh,
                     const double* q, double scale, int j0, int j1,
                     double* o, double* s, int* bad) {
  int D = kv->D, BS = kv->BS;
  for (int d = 0; d < D; ++d) o[d] = 0.0;
  if (j1 <= j0) return -INFINITY;
  double m = -INFINITY;
  for (int j = j0; j < j1; ++j) {
    int64_t blk = table[j / BS];
    if (blk < 0 || blk >= kv->num_blocks) { *bad = 1; s[j - j0] = -INFINITY; continue; }
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += q[d] * elem(kv->k_cache, kv->kv_dtype, cache_index(blk, kvh, j % BS, d, kv->Hkv, BS, D));
    s[j - j0] = scale * kv->k_scale * dot;
    if (s[j - j0] > m) m = s[j - j0];
  }
  double z = 0.0;
  for (int j = j0; j < j1; ++j) {
    int64_t blk = table[j / BS];
    if (blk < 0 || blk >= kv->num_blocks) continue;
    double w = exp(s[j - j0] - m);
    z += w;
    for (int d = 0; d < D; ++d)
      o[d] += w * elem(kv->v_cache, kv->kv_dtype, cache_index(blk, kvh, j % BS, d, kv->Hkv, BS, D));
  }
  for (int d = 0; d < D; ++d) o[d] = kv->v_scale * o[d] / z;
  return m + log(z);
}

static void load_q(double* qd, const void* q, int q_dtype, int64_t row, int D) {
  for (int d = 0; d < D; ++d) qd[d] = elem(q, q_dtype, row * D + d);
}

/*
 * Decode: for each selected sequence b (sel[i], or i when sel is NULL) and
 * query head h, attention of q[b, h] over keys 0 .. seq_lens[b]-1 of KV head
 * h / (Hq / Hkv). out: [nsel, Hq, D] fp64; lse: [nsel, Hq] (may be NULL).
 * part_tokens > 0 computes each partition [p*part, (p+1)*part) on its own
 * and merges the partitions by log-sum-exp:
 *   LSE = log sum_p exp(lse_p),  out = sum_p exp(lse_p - LSE) o_p,
 * with empty partitions (lse_p = -inf) weighted 0. part_tokens = 0 is the
 * unsplit definition. Only query heads h_lo .. h_hi-1 are computed (out is
 * then [nsel, h_hi - h_lo, D]); pass 0 and Hq for all heads. Returns 0, or
 * -1 on an out-of-pool block id.
 */
int pkvo_decode(double* out, double* lse, const void* q, int q_dtype,
                const void* k_cache, const void* v_cache, int kv_dtype,
                const int32_t* block_tables, const int32_t* seq_lens,
                int B, int Hq, int Hkv, int D, int BS, int max_blocks,
                int64_t num_blocks, double scale, const float* k_scales,
                const float* v_scales, const int32_t* sel, int nsel,
                int part_tokens, int h_lo, int h_hi) {
  (void)B;
  int G = Hq / Hkv;
  int bad = 0;
  int nh = h_hi - h_lo;
  int64_t total = (int64_t)nsel * nh;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t w = 0; w < total; ++w) {
    int i = (int)(w / nh), h = h_lo + (int)(w % nh);
    int b = sel ? sel[i] : i;
    int g = h / G;
    int n = seq_lens[b];
    kvview kv = {k_cache, v_cache, kv_dtype, Hkv, BS, D, num_blocks,
                 k_scales ? (double)k_scales[g] : 1.0, v_scales ? (double)v_scales[g] : 1.0};
    double* qd = (double*)malloc(sizeof(double) * D);
    double* s = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
    double* o = out + w * D;
    const int32_t* table = block_tables + (int64_t)b * max_blocks;
    load_q(qd, q, q_dtype, (int64_t)b * Hq + h, D);
    double l;
    if (part_tokens <= 0) {
      l = attend(&kv, table, g, qd, scale, 0, n, o, s, &bad);
    } else {
      int np = (n + part_tokens - 1) / part_tokens;
      double* op = (double*)malloc(sizeof(double) * D * (np > 0 ? np : 1));
      double* lp = (double*)malloc(sizeof(double) * (np > 0 ? np : 1));
      double M = -INFINITY;
      for (int p = 0; p < np; ++p) {
        int j0 = p * part_tokens, j1 = j0 + part_tokens < n ? j0 + part_tokens : n;
        lp[p] = attend(&kv, table, g, qd, scale, j0, j1, op + (int64_t)p * D, s, &bad);
        if (lp[p] > M) M = lp[p];
      }
      double z = 0.0;
      for (int p = 0; p < np; ++p) z += (lp[p] == -INFINITY) ? 0.0 : exp(lp[p] - M);
      l = (np == 0) ? -INFINITY : M + log(z);
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (int p = 0; p < np; ++p) {
        double wp = (lp[p] == -INFINITY) ? 0.0 : exp(lp[p] - l);
        for (int d = 0; d < D; ++d) o[d] += wp * op[(int64_t)p * D + d];
      }
      free(op);
      free(lp);
    }
    if (lse) lse[w] = l;
    free(qd);
    free(s);
  }
  return bad ? -1 : 0;
}

/*
 * Chunked prefill: sequence n has query rows cu_q_lens[n] .. cu_q_lens[n+1]-1
 * (L_n rows) and context seq_lens[n] including the chunk, so P_n =
 * seq_lens[n] - L_n keys precede it. Query row i (0 <= i < L_n) attends keys
 * 0 .. P_n + i. out: [total_q, Hq, D] fp64, lse: [total_q, Hq] (may be
 * NULL). Returns 0, -1 on an out-of-pool block id, -2 if L_n > seq_lens[n].
 */
int pkvo_prefill_chunk(double* out, double* lse, const void* q, int q_dtype,
                       const void* k_cache, const void* v_cache, int kv_dtype,
                       const int32_t* block_tables, const int32_t* seq_lens,
                       const int32_t* cu_q_lens, int num_seqs, int Hq, int Hkv,
                       int D, int BS, int max_blocks, int64_t num_blocks,
                       double scale, const float* k_scales, const float* v_scales) {
  int G = Hq / Hkv;
  int bad = 0;
  int64_t total_q = cu_q_lens[num_seqs];
  for (int n = 0; n < num_seqs; ++n)
    if (cu_q_lens[n + 1] - cu_q_lens[n] > seq_lens[n]) return -2;
  int64_t total = total_q * Hq;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : bad)
  for (int64_t w = 0; w < total; ++w) {
    int64_t row = w / Hq;
    int h = (int)(w % Hq);
    int n = 0;
    while (cu_q_lens[n + 1] <= row) ++n;
    int L = cu_q_lens[n + 1] - cu_q_lens[n];
    int P = seq_lens[n] - L;
    int i = (int)(row - cu_q_lens[n]);
    int g = h / G;
    kvview kv = {k_cache, v_cache, kv_dtype, Hkv, BS, D, num_blocks,
                 k_scales ? (double)k_scales[g] : 1.0, v_scales ? (double)v_scales[g] : 1.0};
    double* qd = (double*)malloc(sizeof(double) * D);
    double* s = (double*)malloc(sizeof(double) * (P + i + 1));
    load_q(qd, q, q_dtype, row * Hq + h, D);
    double l = attend(&kv, block_tables + (int64_t)n * max_blocks, g, qd, scale, 0,
                      P + i + 1, out + w * D, s, &bad);
    if (lse) lse[w] = l;
    free(qd);
    free(s);
  }
  return bad ? -1 : 0;
}
