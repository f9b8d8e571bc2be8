/*
 * i8kv_oracle.c -- plain, slow CPU oracle for INT8 KV-cache paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  The product path (the
 * CUDA library under int8_kv_cache_token_gb300/) never links, loads or calls
 * this file, and this file shares no code, header, table or helper with it.
 *
 * Sources (cited by short key throughout):
 *   [KV] "gfx936 DCU上实现INT8 KV与INT8 MMAC Attention推理优化"
 *        (series part 1: producer, quantization formula, cache layouts, routing)
 *   [PV] "gfx936 DCU上实现INT8 PV MMAC：V Scale融合、概率量化与Fragment分组"
 *        (series part 3: V-scale folding, online softmax, decode partitions,
 *        32-token probability groups)
 *
 * Precision policy.  The pages compute the producer scale, the dequantized
 * score and the probability-side quantization in fp32 ([PV] §3 listing: `float
 * w[32]`, `amax / 127.0f`; [KV] §3.3 listing: `float score = float(qk) *
 * q_scale * k_scale[token] * softmax_scale`).  With `fp32_decisions` set the
 * oracle rounds to fp32 exactly at those steps (every value is held in a double
 * and rounded with R(); a double product/quotient of two floats rounded once to
 * float equals the IEEE fp32 operation, since 53 >= 2*24+2).  Everything the
 * pages do not fix -- the softmax sums l, the output accumulators o, the
 * partition merge -- is accumulated in fp64.  With `fp32_decisions` clear the
 * whole computation is fp64; the tests use that mode to check partition- and
 * tile-invariance without fp32 rounding noise.
 *
 * Readings of points the pages leave open:
 *   - "round" is round-half-to-even ([KV] §2.1 writes round(x/scale)).
 *   - amax == 0 gives scale 0 and an all-zero vector ([KV] §2.1 asks for a
 *     safe scale or all-zero output).
 *   - A probability group is 32 consecutive tokens aligned to absolute token
 *     position 0; a partition or key tile is a multiple of 32 tokens, so no
 *     group straddles two of them ([PV] §1 and §4: the group is the set of 32
 *     tokens one INT8 MMA consumes; the CPU reference uses the same groups).
 *   - Each query row (q-head, query token) has its own sW per group.
 *   - GQA: query head h reads KV head h / (Hq / Hkv).
 *   - The decode history of a sequence is every cached token, 0 .. L-1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_BAD_ARG 1

/* Round a double to fp32 precision when fp32 is requested. */
static inline double R(double x, int fp32) { return fp32 ? (double)(float)x : x; }

/* bf16 bit pattern -> exact fp32 value (bf16 is the top half of an fp32). */
static inline float bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round-half-to-even of a value already rounded to the working precision. */
static inline double rne(double x) { return nearbyint(x); }

/* ------------------------------------------------------------------------- */
/* Paged cache addressing ([KV] §2.3).                                        */
/*   K cache  [blocks, Hkv, D/16, bs, 16] int8 (16 head-dims per chunk)        */
/*   V cache  [blocks, Hkv, D, bs]        int8 (tokens inner-most)             */
/*   scales   [blocks, bs, Hkv]           fp32, one tensor each for K and V     */
/* ------------------------------------------------------------------------- */
static inline size_t k_index(int blk, int h, int d, int off, int Hkv, int D, int bs) {
  return ((((size_t)blk * Hkv + h) * (D / 16) + d / 16) * bs + off) * 16 + (d % 16);
}
static inline size_t v_index(int blk, int h, int d, int off, int Hkv, int D, int bs) {
  return (((size_t)blk * Hkv + h) * D + d) * bs + off;
}
static inline size_t s_index(int blk, int h, int off, int Hkv, int bs) {
  return ((size_t)blk * bs + off) * Hkv + h;
}

/* ------------------------------------------------------------------------- */
/* Symmetric per-vector absmax quantization ([KV] §2.1):                      */
/*   amax = max|x|, scale = amax/127, q = clamp(round(x/scale), -127, 127).   */
/* The producer's arithmetic is fp32 (bit-exact target), whatever the mode.  */
/* ------------------------------------------------------------------------- */
static void quantize_f32(const float* x, int n, int8_t* q, float* scale) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) {
    double a = fabs((double)x[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0) {
    *scale = 0.0f;
    for (int i = 0; i < n; ++i) q[i] = 0;
    return;
  }
  double s = R(amax / 127.0, 1);
  *scale = (float)s;
  for (int i = 0; i < n; ++i) {
    double r = rne(R((double)x[i] / s, 1));
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    q[i] = (int8_t)r;
  }
}

void orc_quantize_vector(const uint16_t* x, int n, int8_t* q, float* scale) {
  float* f = (float*)malloc((size_t)n * sizeof(float));
  for (int i = 0; i < n; ++i) f[i] = bf16_to_f32(x[i]);
  quantize_f32(f, n, q, scale);
  free(f);
}

/* KV producer ([KV] §2.2 steps 3-6, without RoPE): quantize K and V of every
 * token and KV head, scatter them to slot_mapping[t] = block * bs + offset,
 * write the two scales; optionally quantize Q per (token, q-head) ([KV] §2.2:
 * the query is quantized once and reused).  slot < 0 skips the token. */
int orc_kv_quant_write(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping, int T, int Hkv, int D,
                       int bs, int8_t* k_cache, int8_t* v_cache, float* k_scale, float* v_scale, const uint16_t* q,
                       int Hq, int8_t* q_i8, float* q_scale) {
  if (D % 16 != 0 || bs <= 0 || Hkv <= 0) return ORC_BAD_ARG;
  int8_t* tmp = (int8_t*)malloc((size_t)D);
  for (int t = 0; t < T; ++t) {
    int slot = slot_mapping[t];
    if (slot < 0) continue;
    int blk = slot / bs, off = slot % bs;
    for (int h = 0; h < Hkv; ++h) {
      float s;
      orc_quantize_vector(k + ((size_t)t * Hkv + h) * D, D, tmp, &s);
      for (int d = 0; d < D; ++d) k_cache[k_index(blk, h, d, off, Hkv, D, bs)] = tmp[d];
      k_scale[s_index(blk, h, off, Hkv, bs)] = s;
      orc_quantize_vector(v + ((size_t)t * Hkv + h) * D, D, tmp, &s);
      for (int d = 0; d < D; ++d) v_cache[v_index(blk, h, d, off, Hkv, D, bs)] = tmp[d];
      v_scale[s_index(blk, h, off, Hkv, bs)] = s;
    }
  }
  if (q != NULL) {
    for (int t = 0; t < T; ++t)
      for (int h = 0; h < Hq; ++h)
        orc_quantize_vector(q + ((size_t)t * Hq + h) * D, D, q_i8 + ((size_t)t * Hq + h) * D,
                            q_scale + (size_t)t * Hq + h);
  }
  free(tmp);
  return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Fused producer with Q/K RMSNorm and RoPE.  [KV] §2.2 lists RoPE on Q and K  */
/* as the producer's second step, before the absmax, scale and quantization;  */
/* [KV] §5.3 notes that the served model applies a per-head RMSNorm to Q and  */
/* K before RoPE.  The pages give neither formula, so the plain readings:     */
/*   RMSNorm   y_i = (x_i * (1 / sqrt(mean_j x_j^2 + eps))) * w_i             */
/*   RoPE      rotate-half on the first rd dims with h = rd/2 and a table     */
/*             row cs = cos_sin[position] = (cos_0..cos_{h-1}, sin_0..sin_{h-1}):*/
/*             y_i = a c_i - b s_i,  y_{i+h} = b c_i + a s_i,  a = x_i, b = x_{i+h}*/
/*   then the quantization rule of [KV] §2.1 on the fp32 result.              */
/* Every step is one correctly rounded fp32 operation in the order written    */
/* (the file is built without FP contraction): the sum of squares is a        */
/* balanced binary tree in index order, mean = sum * (1/D) (exact, D a power  */
/* of two), then sqrt, the reciprocal, and the two products.  No bf16         */
/* rounding happens between the steps; the optional bf16 copies (q_out,       */
/* k_out) are the fp32 result rounded to nearest even.                        */
/* ------------------------------------------------------------------------- */
#define ORC_BAD_POSITION 2

/* Sum of x_i^2 over n = 2^k elements: each half summed the same way, then added. */
static float sum_sq_tree(const float* x, int n) {
  if (n == 1) return x[0] * x[0];
  float lo = sum_sq_tree(x, n / 2);
  float hi = sum_sq_tree(x + n / 2, n / 2);
  return lo + hi;
}

static void rms_norm_f32(float* x, int D, const uint16_t* w, float eps) {
  float ss = sum_sq_tree(x, D);
  float mean = ss * (1.0f / (float)D);
  float var = mean + eps;
  float rms = sqrtf(var);
  float inv = 1.0f / rms;
  for (int i = 0; i < D; ++i) {
    float t = x[i] * inv;
    x[i] = t * bf16_to_f32(w[i]);
  }
}

static void rope_rotate_half(float* x, int rd, const float* cs) {
  int h = rd / 2;
  for (int i = 0; i < h; ++i) {
    float c = cs[i], s = cs[h + i];
    float a = x[i], b = x[i + h];
    float ac = a * c, bsn = b * s, bc = b * c, asn = a * s;
    x[i] = ac - bsn;
    x[i + h] = bc + asn;
  }
}

/* fp32 -> bf16 bits, round to nearest even (finite values). */
static uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static int is_pow2(int n) { return n > 0 && (n & (n - 1)) == 0; }

/* One Q or K head vector: bf16 -> fp32, optional RMSNorm, optional RoPE. */
static void qk_transform(const uint16_t* src, int D, const uint16_t* norm_w, float eps, const float* cs, int rd,
                         float* x) {
  for (int i = 0; i < D; ++i) x[i] = bf16_to_f32(src[i]);
  if (norm_w) rms_norm_f32(x, D, norm_w, eps);
  if (rd > 0) rope_rotate_half(x, rd, cs);
}

/* Per-channel K smoothing (the accuracy variant for stable channel outliers in
 * K that [KV] §2.1 points to, KIVI's observation): with factors s [Hkv, D]
 * (fp32, > 0), after RMSNorm and RoPE the K vector of KV head h becomes
 * k_d * RN(1/s[h][d]) and the Q vector of query head hq becomes
 * q_d * s[hq / G][d] (G = Hq / Hkv), each product rounded once.  q.k is
 * unchanged in exact arithmetic, the same folding the PV page applies to sV,
 * and the per-token scales no longer see K's channel outliers.  The bf16 copies
 * q_out / k_out are taken before the smoothing. */
static void smooth_vec(float* x, int D, const float* f, int invert) {
  for (int d = 0; d < D; ++d) {
    float m = invert ? 1.0f / f[d] : f[d];
    x[d] = x[d] * m;
  }
}

/* The fused producer.  positions [T] and cos_sin [max_position, rd] fp32 are
 * needed when rd > 0 (rd even, <= D); rd = 0 rotates nothing.  A null norm
 * weight skips that RMSNorm.  K/V go to the cache for slot >= 0 exactly as in
 * orc_kv_quant_write; q (nullable) is transformed and, when q_i8 is given,
 * quantized into q_i8 / q_scale.  q_out / k_out (nullable) receive the
 * transformed Q / K in bf16 for every token, whatever its slot.  A token whose
 * position lies outside [0, max_position) is skipped entirely (nothing of it
 * is written) and the call returns ORC_BAD_POSITION after the other tokens. */
int orc_kv_rope_quant_write(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping, int T, int Hkv, int D,
                            int bs, int8_t* k_cache, int8_t* v_cache, float* k_scale, float* v_scale,
                            const uint16_t* q, int Hq, int8_t* q_i8, float* q_scale, const int32_t* positions,
                            const float* cos_sin, int max_position, int rd, const uint16_t* q_norm_w,
                            const uint16_t* k_norm_w, float eps, uint16_t* q_out, uint16_t* k_out,
                            const float* k_smooth) {
  if (D % 16 != 0 || bs <= 0 || Hkv <= 0 || rd < 0 || rd % 2 != 0 || rd > D) return ORC_BAD_ARG;
  if (k_smooth && q != NULL && (Hq <= 0 || Hq % Hkv != 0)) return ORC_BAD_ARG;
  if ((q_norm_w || k_norm_w) && !is_pow2(D)) return ORC_BAD_ARG;
  if (rd > 0 && (positions == NULL || cos_sin == NULL || max_position <= 0)) return ORC_BAD_ARG;
  int bad = 0;
  float* x = (float*)malloc((size_t)D * sizeof(float));
  int8_t* tmp = (int8_t*)malloc((size_t)D);
  for (int t = 0; t < T; ++t) {
    const float* cs = NULL;
    if (rd > 0) {
      int p = positions[t];
      if (p < 0 || p >= max_position) {
        bad = 1;
        continue;
      }
      cs = cos_sin + (size_t)p * rd;
    }
    int slot = slot_mapping[t];
    int blk = slot >= 0 ? slot / bs : 0, off = slot >= 0 ? slot % bs : 0;
    for (int h = 0; h < Hkv; ++h) {
      size_t row = ((size_t)t * Hkv + h) * D;
      float s;
      qk_transform(k + row, D, k_norm_w, eps, cs, rd, x);
      if (k_out)
        for (int d = 0; d < D; ++d) k_out[row + d] = f32_to_bf16(x[d]);
      if (slot < 0) continue;
      if (k_smooth) smooth_vec(x, D, k_smooth + (size_t)h * D, 1);
      quantize_f32(x, D, tmp, &s);
      for (int d = 0; d < D; ++d) k_cache[k_index(blk, h, d, off, Hkv, D, bs)] = tmp[d];
      k_scale[s_index(blk, h, off, Hkv, bs)] = s;
      orc_quantize_vector(v + row, D, tmp, &s);
      for (int d = 0; d < D; ++d) v_cache[v_index(blk, h, d, off, Hkv, D, bs)] = tmp[d];
      v_scale[s_index(blk, h, off, Hkv, bs)] = s;
    }
    if (q == NULL) continue;
    for (int h = 0; h < Hq; ++h) {
      size_t row = ((size_t)t * Hq + h) * D;
      qk_transform(q + row, D, q_norm_w, eps, cs, rd, x);
      if (q_out)
        for (int d = 0; d < D; ++d) q_out[row + d] = f32_to_bf16(x[d]);
      if (k_smooth) smooth_vec(x, D, k_smooth + (size_t)(h / (Hq / Hkv)) * D, 0);
      if (q_i8) quantize_f32(x, D, q_i8 + row, q_scale + (size_t)t * Hq + h);
    }
  }
  free(tmp);
  free(x);
  return bad ? ORC_BAD_POSITION : ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* INT8 QK: acc_t = sum_d Qi8[d] * Ki8_t[d], exact in int32 ([PV] §2).        */
/* ------------------------------------------------------------------------- */
static int32_t qk_acc(const int8_t* qv, const int8_t* k_cache, int blk, int kvh, int off, int Hkv, int D, int bs) {
  int32_t acc = 0;
  for (int d = 0; d < D; ++d) acc += (int32_t)qv[d] * (int32_t)k_cache[k_index(blk, kvh, d, off, Hkv, D, bs)];
  return acc;
}

/* Raw int32 accumulators for every (sequence, q-head, token); tokens past a
 * sequence's length are written as 0.  acc is [B, Hq, max_len]. */
int orc_qk_i32(int32_t* acc, const int8_t* q_i8, const int8_t* k_cache, const int32_t* block_tables,
               const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int bs, int max_blocks, int max_len) {
  if (Hq % Hkv != 0) return ORC_BAD_ARG;
  int G = Hq / Hkv;
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) {
      int kvh = h / G;
      const int8_t* qv = q_i8 + ((size_t)b * Hq + h) * D;
      for (int t = 0; t < max_len; ++t) {
        int32_t a = 0;
        if (t < seq_lens[b]) {
          int blk = block_tables[(size_t)b * max_blocks + t / bs];
          a = qk_acc(qv, k_cache, blk, kvh, t % bs, Hkv, D, bs);
        }
        acc[((size_t)b * Hq + h) * max_len + t] = a;
      }
    }
  return ORC_OK;
}

/* Dequantized score ([PV] §2, [KV] §3.3): score = acc * sQ * sK_t / sqrt(d),
 * evaluated left to right. */
static inline double score_of(int32_t acc, float sq, float sk, double c, int fp32) {
  double s = R((double)acc * (double)sq, fp32);
  s = R(s * (double)sk, fp32);
  return R(s * c, fp32);
}

/* One 32-token probability group ([PV] §1, §2.2, §3):
 *   A = max W over the group, sW = A / pmax, Wq = round(W / sW),
 *   o[d] += sW * sum_t Wq_t * Vq_t[d]   (integer contraction, rescaled to float).
 * W >= 0 here, so Wq lies in [0, pmax].  A == 0 gives Wq = 0.  pmax = 127 is
 * the pages' signed INT8 probability code; pmax = 255 is the UINT8 code that
 * [PV] §6 weighs (probabilities are non-negative, so 0..255 gains one bit)
 * and leaves unbuilt for want of a mixed-sign MMA. */
static void pv_group(const double* W, int n, const int8_t* const* vrows, int D, int fp32, double weight, double* o,
                     int16_t* trace_wq, double* trace_sw, int pmax) {
  double A = 0.0;
  for (int i = 0; i < n; ++i)
    if (W[i] > A) A = W[i];
  double sW = R(A / (double)pmax, fp32);
  int wq[64];
  for (int i = 0; i < n; ++i) {
    double r = (A > 0.0) ? rne(R(W[i] / sW, fp32)) : 0.0;
    if (r > (double)pmax) r = (double)pmax;
    if (r < 0.0) r = 0.0;
    wq[i] = (int)r;
    if (trace_wq) trace_wq[i] = (int16_t)wq[i];
    if (trace_sw) trace_sw[i] = sW;
  }
  for (int d = 0; d < D; ++d) {
    int64_t acc = 0;
    for (int i = 0; i < n; ++i) acc += (int64_t)wq[i] * (int64_t)vrows[i][d];
    o[d] += weight * sW * (double)acc;
  }
}

/* Gather the token-major int8 V row of token t (from the token-inner layout). */
static void gather_v(int8_t* dst, const int8_t* v_cache, int blk, int kvh, int off, int Hkv, int D, int bs) {
  for (int d = 0; d < D; ++d) dst[d] = v_cache[v_index(blk, kvh, d, off, Hkv, D, bs)];
}

/* ------------------------------------------------------------------------- */
/* Decode attention, literal form ([PV] §2.2, [KV] §3.3).                     */
/* History [0, L) is split into partitions of `partition` tokens.  Partition  */
/* g: m_g = max score, l_g = sum exp(score - m_g), P = exp(score - m_g) / l_g, */
/* W = P * sV; 32-token groups quantize W and run the INT8 W x Vq contraction. */
/* Partitions are merged by log-sum-exp: M = max m_g, w_g = l_g exp(m_g - M), */
/* O = sum_g w_g o_g / sum_g w_g.  An empty sequence gives O = 0.             */
/* out is [B, Hq, D] fp64.                                                    */
/* Optional trace of one (trace_b, trace_h): per history token, the fp value  */
/* W, the code Wq, the group scale sW and the token's partition merge weight */
/* c_g = w_g / sum w (so the global probability is c_g * P).                 */
/* ------------------------------------------------------------------------- */
int orc_decode_attn(double* out, const int8_t* q_i8, const float* q_scale, const int8_t* k_cache,
                    const int8_t* v_cache, const float* k_scale, const float* v_scale, const int32_t* block_tables,
                    const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int bs, int max_blocks,
                    float softmax_scale, int partition, int group, int fp32_decisions, int nthreads, int trace_b,
                    int trace_h, double* tr_W, int16_t* tr_Wq, double* tr_sW, double* tr_c, int pmax) {
  if (Hq % Hkv != 0 || D % 16 != 0 || group <= 0 || group > 64 || partition <= 0 || partition % group != 0 ||
      (pmax != 127 && pmax != 255))
    return ORC_BAD_ARG;
  const int G = Hq / Hkv;
  const int fp32 = fp32_decisions;
  const double c = R((double)softmax_scale, 1);
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) {
      const int L = seq_lens[b];
      const int kvh = h / G;
      double* O = out + ((size_t)b * Hq + h) * D;
      for (int d = 0; d < D; ++d) O[d] = 0.0;
      if (L <= 0) continue;
      const int8_t* qv = q_i8 + ((size_t)b * Hq + h) * D;
      const float sq = q_scale[(size_t)b * Hq + h];
      const int32_t* bt = block_tables + (size_t)b * max_blocks;
      const int tracing = (b == trace_b && h == trace_h);

      double* s = (double*)malloc(sizeof(double) * L);
      for (int t = 0; t < L; ++t) {
        int blk = bt[t / bs], off = t % bs;
        s[t] = score_of(qk_acc(qv, k_cache, blk, kvh, off, Hkv, D, bs), sq, k_scale[s_index(blk, kvh, off, Hkv, bs)],
                        c, fp32);
      }
      const int NP = (L + partition - 1) / partition;
      double* m_g = (double*)malloc(sizeof(double) * NP);
      double* l_g = (double*)malloc(sizeof(double) * NP);
      double* o_g = (double*)calloc((size_t)NP * D, sizeof(double));
      double* W = (double*)malloc(sizeof(double) * partition);
      int8_t* vbuf = (int8_t*)malloc((size_t)group * D);
      const int8_t* vrows[64];
      for (int g = 0; g < NP; ++g) {
        int t0 = g * partition, t1 = t0 + partition < L ? t0 + partition : L;
        double m = -INFINITY;
        for (int t = t0; t < t1; ++t)
          if (s[t] > m) m = s[t];
        double l = 0.0;
        for (int t = t0; t < t1; ++t) {
          double p = R(exp(R(s[t] - m, fp32)), fp32);
          W[t - t0] = p;
          l += p;
        }
        for (int t = t0; t < t1; ++t) {
          int blk = bt[t / bs], off = t % bs;
          double P = R(W[t - t0] / l, fp32);
          W[t - t0] = R(P * (double)v_scale[s_index(blk, kvh, off, Hkv, bs)], fp32);
        }
        m_g[g] = m;
        l_g[g] = l;
        for (int j0 = t0; j0 < t1; j0 += group) {
          int n = (j0 + group < t1 ? j0 + group : t1) - j0;
          for (int i = 0; i < n; ++i) {
            int t = j0 + i;
            gather_v(vbuf + (size_t)i * D, v_cache, bt[t / bs], kvh, t % bs, Hkv, D, bs);
            vrows[i] = vbuf + (size_t)i * D;
          }
          pv_group(W + (j0 - t0), n, vrows, D, fp32, 1.0, o_g + (size_t)g * D, tracing ? tr_Wq + j0 : NULL,
                   tracing ? tr_sW + j0 : NULL, pmax);
          if (tracing)
            for (int i = 0; i < n; ++i) tr_W[j0 + i] = W[j0 - t0 + i];
        }
      }
      double M = -INFINITY;
      for (int g = 0; g < NP; ++g)
        if (m_g[g] > M) M = m_g[g];
      double wsum = 0.0;
      for (int g = 0; g < NP; ++g) wsum += l_g[g] * exp(m_g[g] - M);
      for (int g = 0; g < NP; ++g) {
        double w = l_g[g] * exp(m_g[g] - M);
        for (int d = 0; d < D; ++d) O[d] += w * o_g[(size_t)g * D + d];
        if (tracing) {
          int t0 = g * partition, t1 = t0 + partition < L ? t0 + partition : L;
          for (int t = t0; t < t1; ++t) tr_c[t] = w / wsum;
        }
      }
      for (int d = 0; d < D; ++d) O[d] /= wsum;
      free(s);
      free(m_g);
      free(l_g);
      free(o_g);
      free(W);
      free(vbuf);
    }
  return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Prefix-prefill chunk, literal single online softmax ([PV] §2.1, [KV] §3.2). */
/* Chunk query j sits at absolute position H + j and sees keys 0 .. H + j of  */
/* the cache (history then the chunk itself, causal).  Keys are visited in    */
/* tiles of `key_tile` tokens; per tile with the running state (m, l, o):     */
/*   m' = max(m, max score), alpha = exp(m - m'), p~ = exp(score - m'),       */
/*   W = p~ * sV (unnormalized), o = alpha o + sum_groups sW * (Wq x Vq),     */
/*   l = alpha l + sum p~;  finally O = o / l.                                 */
/* rows (nullable) selects chunk rows; out is [nrows, Hq, D] fp64.            */
/* ------------------------------------------------------------------------- */
int orc_prefix_attn(double* out, const int8_t* q_i8, const float* q_scale, const int8_t* k_cache,
                    const int8_t* v_cache, const float* k_scale, const float* v_scale, const int32_t* block_table,
                    int history_len, int chunk_len, int Hq, int Hkv, int D, int bs, float softmax_scale, int key_tile,
                    int group, const int32_t* rows, int nrows, int fp32_decisions, int nthreads) {
  if (Hq % Hkv != 0 || D % 16 != 0 || group <= 0 || group > 64 || key_tile <= 0 || key_tile % group != 0)
    return ORC_BAD_ARG;
  if (rows == NULL) nrows = chunk_len;
  const int G = Hq / Hkv;
  const int fp32 = fp32_decisions;
  const double c = R((double)softmax_scale, 1);
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int r = 0; r < nrows; ++r)
    for (int h = 0; h < Hq; ++h) {
      const int j = rows ? rows[r] : r;
      const int n_keys = history_len + j + 1;
      const int kvh = h / G;
      const int8_t* qv = q_i8 + ((size_t)j * Hq + h) * D;
      const float sq = q_scale[(size_t)j * Hq + h];
      double* O = out + ((size_t)r * Hq + h) * D;
      double* o = (double*)calloc((size_t)D, sizeof(double));
      double* s = (double*)malloc(sizeof(double) * key_tile);
      double* W = (double*)malloc(sizeof(double) * key_tile);
      int8_t* vbuf = (int8_t*)malloc((size_t)group * D);
      const int8_t* vrows[64];
      double m = -INFINITY, l = 0.0;
      for (int k0 = 0; k0 < n_keys; k0 += key_tile) {
        int k1 = k0 + key_tile < n_keys ? k0 + key_tile : n_keys;
        double m_new = m;
        for (int t = k0; t < k1; ++t) {
          int blk = block_table[t / bs], off = t % bs;
          s[t - k0] = score_of(qk_acc(qv, k_cache, blk, kvh, off, Hkv, D, bs), sq,
                               k_scale[s_index(blk, kvh, off, Hkv, bs)], c, fp32);
          if (s[t - k0] > m_new) m_new = s[t - k0];
        }
        double alpha = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        for (int d = 0; d < D; ++d) o[d] *= alpha;
        l *= alpha;
        for (int t = k0; t < k1; ++t) {
          int blk = block_table[t / bs], off = t % bs;
          double p = R(exp(R(s[t - k0] - m_new, fp32)), fp32);
          l += p;
          W[t - k0] = R(p * (double)v_scale[s_index(blk, kvh, off, Hkv, bs)], fp32);
        }
        for (int j0 = k0; j0 < k1; j0 += group) {
          int n = (j0 + group < k1 ? j0 + group : k1) - j0;
          for (int i = 0; i < n; ++i) {
            int t = j0 + i;
            gather_v(vbuf + (size_t)i * D, v_cache, block_table[t / bs], kvh, t % bs, Hkv, D, bs);
            vrows[i] = vbuf + (size_t)i * D;
          }
          pv_group(W + (j0 - k0), n, vrows, D, fp32, 1.0, o, NULL, NULL, 127);
        }
        m = m_new;
      }
      for (int d = 0; d < D; ++d) O[d] = o[d] / l;
      free(o);
      free(s);
      free(W);
      free(vbuf);
    }
  return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* BF16-KV comparison cache: the same paging with bf16 elements.             */
/*   K cache [blocks, Hkv, D/8, bs, 8] bf16 (16-byte chunks of 8 head-dims)   */
/*   V cache [blocks, Hkv, D, bs]      bf16                                    */
/* ------------------------------------------------------------------------- */
static inline size_t kb_index(int blk, int h, int d, int off, int Hkv, int D, int bs) {
  return ((((size_t)blk * Hkv + h) * (D / 8) + d / 8) * bs + off) * 8 + (d % 8);
}

int orc_bf16_kv_write(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping, int T, int Hkv, int D, int bs,
                      uint16_t* k_cache, uint16_t* v_cache) {
  if (D % 8 != 0) return ORC_BAD_ARG;
  for (int t = 0; t < T; ++t) {
    int slot = slot_mapping[t];
    if (slot < 0) continue;
    int blk = slot / bs, off = slot % bs;
    for (int h = 0; h < Hkv; ++h)
      for (int d = 0; d < D; ++d) {
        k_cache[kb_index(blk, h, d, off, Hkv, D, bs)] = k[((size_t)t * Hkv + h) * D + d];
        v_cache[v_index(blk, h, d, off, Hkv, D, bs)] = v[((size_t)t * Hkv + h) * D + d];
      }
  }
  return ORC_OK;
}

/* Plain softmax attention in fp64 over the bf16 paged cache, for a bf16 query
 * [B, Hq, D]: O = sum_t softmax(q.k_t * scale) v_t.  out is [B, Hq, D]. */
/* High-precision chunk attention, the first-chunk path of [KV] §3.1 (the
 * first prefill chunk keeps a high-precision attention while the producer
 * writes its K/V to the INT8 cache) and of the routing in [KV] §4 (chunks
 * whose history is below the INT8 threshold stay high-precision).  Query row
 * j of the chunk (position history_len + j) attends to keys 0 .. history_len
 * + j: a history key t < history_len is read back from the INT8 cache as
 * code * scale (the only copy the cache keeps), a chunk key from the bf16
 * inputs k_chunk / v_chunk [chunk_len, Hkv, D].  Plain softmax attention in
 * fp64: out = sum_t e^(s_t - m) V_t / sum_t e^(s_t - m), s_t = scale q.K_t.
 * rows (nullable) selects chunk rows; out is [nrows, Hq, D]. */
int orc_bf16_prefix_attn(double* out, const uint16_t* q, const uint16_t* k_chunk, const uint16_t* v_chunk,
                         const int8_t* k_cache, const int8_t* v_cache, const float* k_scale, const float* v_scale,
                         const int32_t* block_table, int history_len, int chunk_len, int Hq, int Hkv, int D, int bs,
                         double softmax_scale, const int32_t* rows, int nrows, int nthreads) {
  if (Hq % Hkv != 0 || D % 16 != 0 || history_len < 0 || chunk_len < 0) return ORC_BAD_ARG;
  if (rows == NULL) nrows = chunk_len;
  const int G = Hq / Hkv;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int r = 0; r < nrows; ++r)
    for (int h = 0; h < Hq; ++h) {
      const int j = rows ? rows[r] : r;
      const int n_keys = history_len + j + 1;
      const int kvh = h / G;
      const uint16_t* qv = q + ((size_t)j * Hq + h) * D;
      double* O = out + ((size_t)r * Hq + h) * D;
      double* s = (double*)malloc(sizeof(double) * (size_t)n_keys);
      double* kx = (double*)malloc(sizeof(double) * (size_t)D);
      double m = -INFINITY;
      for (int t = 0; t < n_keys; ++t) {
        if (t < history_len) {
          const int blk = block_table[t / bs], off = t % bs;
          const double sc = (double)k_scale[s_index(blk, kvh, off, Hkv, bs)];
          for (int d = 0; d < D; ++d) kx[d] = (double)k_cache[k_index(blk, kvh, d, off, Hkv, D, bs)] * sc;
        } else {
          const uint16_t* kr = k_chunk + ((size_t)(t - history_len) * Hkv + kvh) * D;
          for (int d = 0; d < D; ++d) kx[d] = (double)bf16_to_f32(kr[d]);
        }
        double a = 0.0;
        for (int d = 0; d < D; ++d) a += (double)bf16_to_f32(qv[d]) * kx[d];
        s[t] = a * softmax_scale;
        if (s[t] > m) m = s[t];
      }
      double l = 0.0;
      for (int d = 0; d < D; ++d) O[d] = 0.0;
      for (int t = 0; t < n_keys; ++t) {
        const double p = exp(s[t] - m);
        l += p;
        if (t < history_len) {
          const int blk = block_table[t / bs], off = t % bs;
          const double sc = (double)v_scale[s_index(blk, kvh, off, Hkv, bs)];
          for (int d = 0; d < D; ++d) O[d] += p * (double)v_cache[v_index(blk, kvh, d, off, Hkv, D, bs)] * sc;
        } else {
          const uint16_t* vr = v_chunk + ((size_t)(t - history_len) * Hkv + kvh) * D;
          for (int d = 0; d < D; ++d) O[d] += p * (double)bf16_to_f32(vr[d]);
        }
      }
      for (int d = 0; d < D; ++d) O[d] /= l;
      free(kx);
      free(s);
    }
  return ORC_OK;
}

int orc_bf16_decode_attn(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                         const int32_t* block_tables, const int32_t* seq_lens, int B, int Hq, int Hkv, int D, int bs,
                         int max_blocks, double softmax_scale, int nthreads) {
  if (Hq % Hkv != 0 || D % 8 != 0) return ORC_BAD_ARG;
  const int G = Hq / Hkv;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) {
      const int L = seq_lens[b];
      const int kvh = h / G;
      double* O = out + ((size_t)b * Hq + h) * D;
      for (int d = 0; d < D; ++d) O[d] = 0.0;
      if (L <= 0) continue;
      const uint16_t* qv = q + ((size_t)b * Hq + h) * D;
      const int32_t* bt = block_tables + (size_t)b * max_blocks;
      double* s = (double*)malloc(sizeof(double) * L);
      double m = -INFINITY;
      for (int t = 0; t < L; ++t) {
        int blk = bt[t / bs], off = t % bs;
        double a = 0.0;
        for (int d = 0; d < D; ++d)
          a += (double)bf16_to_f32(qv[d]) * (double)bf16_to_f32(k_cache[kb_index(blk, kvh, d, off, Hkv, D, bs)]);
        s[t] = a * softmax_scale;
        if (s[t] > m) m = s[t];
      }
      double l = 0.0;
      for (int t = 0; t < L; ++t) {
        int blk = bt[t / bs], off = t % bs;
        double p = exp(s[t] - m);
        l += p;
        for (int d = 0; d < D; ++d) O[d] += p * (double)bf16_to_f32(v_cache[v_index(blk, kvh, d, off, Hkv, D, bs)]);
      }
      for (int d = 0; d < D; ++d) O[d] /= l;
      free(s);
    }
  return ORC_OK;
}

/* The BF16-KV comparison of the prefix chunk (the BF16 control of [KV] §4.2,
 * where BF16 and INT8 attention are compared on prefill chunks by history):
 * chunk row j (position history_len + j) of the bf16 query [chunk_len, Hq, D]
 * attends, causally, to keys 0 .. history_len + j of one sequence, every key
 * (history and the chunk's own) read from the bf16 paged cache through
 * block_table.  Plain softmax attention in fp64 on the bf16 values.  rows
 * (nullable) selects chunk rows; out is [nrows, Hq, D]. */
int orc_bf16_kv_prefix_attn(double* out, const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                            const int32_t* block_table, int history_len, int chunk_len, int Hq, int Hkv, int D, int bs,
                            double softmax_scale, const int32_t* rows, int nrows, int nthreads) {
  if (Hq % Hkv != 0 || D % 8 != 0 || history_len < 0 || chunk_len < 0) return ORC_BAD_ARG;
  if (rows == NULL) nrows = chunk_len;
  const int G = Hq / Hkv;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int r = 0; r < nrows; ++r)
    for (int h = 0; h < Hq; ++h) {
      const int j = rows ? rows[r] : r;
      const int kv_head = h / G;
      const int visible = history_len + j + 1; /* keys 0 .. history_len + j */
      const uint16_t* qv = q + ((size_t)j * Hq + h) * D;
      double* O = out + ((size_t)r * Hq + h) * D;
      double* s = (double*)malloc(sizeof(double) * (size_t)visible);
      double m = -INFINITY;
      for (int t = 0; t < visible; ++t) {
        const int blk = block_table[t / bs], off = t % bs;
        double a = 0.0;
        for (int d = 0; d < D; ++d)
          a += (double)bf16_to_f32(qv[d]) * (double)bf16_to_f32(k_cache[kb_index(blk, kv_head, d, off, Hkv, D, bs)]);
        s[t] = a * softmax_scale;
        if (s[t] > m) m = s[t];
      }
      double l = 0.0;
      for (int d = 0; d < D; ++d) O[d] = 0.0;
      for (int t = 0; t < visible; ++t) {
        const int blk = block_table[t / bs], off = t % bs;
        const double p = exp(s[t] - m);
        l += p;
        for (int d = 0; d < D; ++d)
          O[d] += p * (double)bf16_to_f32(v_cache[v_index(blk, kv_head, d, off, Hkv, D, bs)]);
      }
      for (int d = 0; d < D; ++d) O[d] /= l;
      free(s);
    }
  return ORC_OK;
}

/* Threads the OpenMP runtime would use by default (1 without OpenMP). */
int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
