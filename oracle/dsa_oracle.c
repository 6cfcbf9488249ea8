/*
 * Oracle for the DSA indexer Q/K prepare-and-store.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU statement of what the GPU path computes.  Only the test suite, the smoke
 * check and the bench's CPU-baseline leg may load it; the product library never
 * links, calls or falls back to it, and it shares no code, header or table with
 * the CUDA sources.
 *
 * Sources (page title, section):
 *   [FUSE-QK]  sglang PR "[AMD] [GLM5] Fuse the DSA indexer Q/K rope + quant +
 *              K-cache write": Motivation (rope on q and k, LayerNorm on k, an
 *              fp8 quant of each, the head-gate scale, the index-K cache write),
 *              Modifications (fp32 k_norm params, separate cos/sin rows of
 *              rope_dim/2, the sliced out_cache_loc, the k-only store),
 *              Accuracy (note on the two K-cache writers: fp32 -> fp8 in one
 *              step, ue8m0 scales).
 *   [FUSE-Q]   vllm PR "[ROCm][Perf] Enable fused indexer-Q RoPE+quant kernel
 *              for DeepSeek/GLM sparse attention": Summary (RoPE + FP8
 *              quantization + weight-scale fold), Kernel-level evidence table
 *              ("q -> FP8 (ue8m0) quant", "weights scale-fold").
 *   [OFP8]     OCP 8-bit Floating Point Specification (OFP8) rev. 1.0, E4M3:
 *              bias 7, no infinities, S.1111.111 is NaN, max normal 448.
 *
 * Readings where the pages are silent (each is a stated choice, not a pin):
 *   - k: LayerNorm over all 128 dims first, then RoPE on dims [0, rope_dim).
 *   - The rope slice is the first rope_dim dims; NeoX pairs (i, i + r/2),
 *     GPT-J pairs (2i, 2i + 1); both use frequency index i.
 *   - RoPE in fp32 in the fused form a' = fma(a, c, -(b*s)),
 *     b' = fma(b, c, a*s), each product rounded to fp32 first.
 *   - LayerNorm in double, biased variance, eps inside the square root,
 *     result rounded once to fp32.
 *   - ue8m0 scale 2^e with e the smallest integer such that
 *     max(amax, 1e-4) <= 448 * 2^e  (the 1e-4 floor: parity unpinned).
 *   - fp32 -> e4m3 round-to-nearest-even, saturating at 448, never NaN.
 *   - weights = w * 2^e_q * softmax_scale * H^-0.5, in double, rounded once
 *     (the constants of the fold: parity unpinned).
 *   - index-K cache page p holds page_size*128 code bytes, then page_size
 *     fp32 scales; slot s lives in page s / page_size at offset s % page_size
 *     (the other layout: 132 bytes per slot, codes then scale).
 *   - The Hadamard variant (the rotation [FUSE-QK] Modifications says the
 *     fused path leaves out): after RoPE, each q head and k is multiplied by
 *     the Sylvester matrix H_128 divided by sqrt(128); computed as fp32
 *     butterflies over index bits 0..6 in that order, then one multiply by
 *     fp32(128^-0.5), so every rounding is fixed.
 *
 * Build: plain C99, -O2 -ffp-contract=off (no fused multiply-add except the
 * explicit fmaf calls the RoPE form asks for).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define DSA_D 128

/* ---------------------------------------------------------------- formats */

/* bf16 bit pattern -> fp32: a bf16 is the upper half of an fp32. */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* fp32 -> bf16, round to nearest, ties to even (finite inputs). */
static float round_to_bf16(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u = (u + 0x7FFFu + lsb) & 0xFFFF0000u;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* [OFP8] E4M3 encode with round-to-nearest-even, saturating to +-448. */
uint8_t oracle_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double m = fabs((double)v);
  if (isnan(v)) return (uint8_t)(sign | 0x7F);
  if (m >= 448.0) return (uint8_t)(sign | 0x7E);
  if (m < ldexp(1.0, -6)) {
    /* subnormal range: step 2^-9, codes 0..7; q == 8 is the min normal 0x08 */
    double q = nearbyint(m * 512.0);
    return (uint8_t)(sign | (uint8_t)q);
  }
  int x;
  (void)frexp(m, &x); /* m = f * 2^x, f in [0.5, 1) */
  int E = x - 1;      /* m in [2^E, 2^(E+1)) */
  double q = nearbyint(ldexp(m, 3 - E)); /* 8 .. 16 */
  if (q == 16.0) {
    E += 1;
    q = 8.0;
  }
  if (E > 8 || (E == 8 && q > 14.0)) return (uint8_t)(sign | 0x7E);
  return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | ((int)q - 8)));
}

/* [OFP8] E4M3 decode. */
float oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return (float)(s ? -v : v);
}

/* [FUSE-Q] ue8m0: the smallest e with max(amax, 1e-4) <= 448 * 2^e. */
int oracle_ue8m0_exponent(float amax) {
  double a = (double)fmaxf(amax, 1e-4f);
  int x;
  double f = frexp(a / 448.0, &x); /* a/448 = f * 2^x, f in [0.5, 1) */
  int e = (f == 0.5) ? x - 1 : x;
  /* the quotient above is rounded; settle e with exact comparisons */
  while (ldexp(448.0, e - 1) >= a) e -= 1;
  while (ldexp(448.0, e) < a) e += 1;
  return e;
}

/* ----------------------------------------------------------- the steps */

/* [FUSE-QK] Motivation / Modifications: LayerNorm on k with fp32 gamma/beta.
 * y_j = (x_j - mean) / sqrt(var + eps) * gamma_j + beta_j, biased variance. */
void oracle_layernorm(const float* x, const float* gamma, const float* beta,
                      float eps, float* y) {
  double mean = 0.0, var = 0.0;
  for (int j = 0; j < DSA_D; ++j) mean += (double)x[j];
  mean /= DSA_D;
  for (int j = 0; j < DSA_D; ++j) {
    double d = (double)x[j] - mean;
    var += d * d;
  }
  var /= DSA_D;
  double rstd = 1.0 / sqrt(var + (double)eps);
  for (int j = 0; j < DSA_D; ++j)
    y[j] = (float)(((double)x[j] - mean) * rstd * (double)gamma[j] +
                   (double)beta[j]);
}

/* [FUSE-QK] Motivation ("rope on q and k"), Modifications (cos and sin kept
 * apart, rope_dim/2 per position).  Rotates each pair (a, b) of the first
 * rope_dim dims by the angle whose cos/sin are cos_row[i], sin_row[i]:
 *   a' = a*c - b*s,  b' = b*c + a*s.
 * style 0 = NeoX: pair i is (i, i + rope_dim/2); style 1 = GPT-J: (2i, 2i+1). */
void oracle_rope(float* x, const float* cos_row, const float* sin_row,
                 int rope_dim, int style) {
  int half = rope_dim / 2;
  for (int i = 0; i < half; ++i) {
    int ia = style == 0 ? i : 2 * i;
    int ib = style == 0 ? i + half : 2 * i + 1;
    float a = x[ia], b = x[ib], c = cos_row[i], s = sin_row[i];
    float bs = b * s;
    float as = a * s;
    x[ia] = fmaf(a, c, -bs);
    x[ib] = fmaf(b, c, as);
  }
}

/* The Hadamard rotation that [FUSE-QK] Modifications says the fused path
 * assumes absent ("the no-Hadamard invariant"): x <- H_128 x / sqrt(128), the
 * normalised Walsh-Hadamard transform, applied after RoPE and before the
 * quantiser.  Written as the radix-2 butterfly network in fp32, stage by stage
 * over index bits 0, 1, ..., 6 -- each stage replaces (a, b) = (x[i], x[i+h])
 * by (a + b, a - b) for every i with bit h clear -- and then one multiply by
 * the fp32 value of 128^-0.5; that fixes every rounding. */
void oracle_hadamard(float* x) {
  for (int h = 1; h < DSA_D; h <<= 1)
    for (int i = 0; i < DSA_D; ++i)
      if ((i & h) == 0) {
        float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
  const float s = (float)(1.0 / sqrt((double)DSA_D));
  for (int i = 0; i < DSA_D; ++i) x[i] = x[i] * s;
}

/* [FUSE-Q] "q -> FP8 (ue8m0) quant"; [FUSE-QK] Accuracy (fp32 -> fp8 in one
 * step): one power-of-two scale per 128-vector, codes = e4m3(z / scale).
 * Returns the scale exponent e. */
int oracle_quantize_vector(const float* z, uint8_t* codes) {
  float amax = 0.0f;
  for (int j = 0; j < DSA_D; ++j) amax = fmaxf(amax, fabsf(z[j]));
  int e = oracle_ue8m0_exponent(amax);
  float inv_scale = (float)ldexp(1.0, -e);
  for (int j = 0; j < DSA_D; ++j) codes[j] = oracle_e4m3_encode(z[j] * inv_scale);
  return e;
}

/* [FUSE-QK] Motivation ("the index-K cache write") and Modifications (the
 * sliced out_cache_loc): store the codes and the fp32 scale of one k vector
 * into its slot of the paged index-K cache.  Checklist ("both paged
 * layouts"): token_major == 0 is the page-blocked layout (a page's codes,
 * then its scales); token_major == 1 gives each slot 132 consecutive bytes,
 * its codes then its scale. */
static void store_index_k(uint8_t* cache, int64_t slot, int32_t page_size,
                          const uint8_t* codes, int e, int token_major) {
  float scale = (float)ldexp(1.0, e);
  if (token_major) {
    uint8_t* row = cache + slot * (DSA_D + 4);
    memcpy(row, codes, DSA_D);
    memcpy(row + DSA_D, &scale, 4);
    return;
  }
  int64_t page = slot / page_size, off = slot % page_size;
  uint8_t* page_base = cache + page * (int64_t)page_size * (DSA_D + 4);
  memcpy(page_base + off * DSA_D, codes, DSA_D);
  memcpy(page_base + (int64_t)page_size * DSA_D + off * 4, &scale, 4);
}

/* The k side of one token: bf16 -> fp32, LayerNorm, RoPE, quantise.
 * bf16_intermediate = 1: the rotated vector is rounded to bf16 just before it
 * is quantised -- the unfused writer of [FUSE-QK] Accuracy (note on the two
 * writers), which "rounds to bf16 before quantizing"; one rounding there can
 * move a code by at most one step, which is what that note reports.
 * bf16_intermediate = 2: the four-launch chain of [FUSE-QK] Profile (rope,
 * LayerNorm, act_quant, k quant + cache as separate kernels), which hands bf16
 * tensors from launch to launch: the LayerNorm output and the rotated vector
 * are both rounded to bf16. */
static int prepare_k(const uint16_t* krow, const float* cos_row,
                     const float* sin_row, const float* gamma,
                     const float* beta, float eps, int rope_dim, int style,
                     int bf16_intermediate, int hadamard, uint8_t* codes) {
  float x[DSA_D], y[DSA_D];
  for (int j = 0; j < DSA_D; ++j) x[j] = bf16_to_f32(krow[j]);
  oracle_layernorm(x, gamma, beta, eps, y);
  if (bf16_intermediate == 2)
    for (int j = 0; j < DSA_D; ++j) y[j] = round_to_bf16(y[j]);
  oracle_rope(y, cos_row, sin_row, rope_dim, style);
  if (hadamard) oracle_hadamard(y);
  if (bf16_intermediate)
    for (int j = 0; j < DSA_D; ++j) y[j] = round_to_bf16(y[j]);
  return oracle_quantize_vector(y, codes);
}

/* k-only prepare-and-store ([FUSE-QK] Modifications: the k-only store reached
 * by the dense decode fast path).  Strides are in elements.  Returns the
 * error bits: 1 = a position outside [0, max_position) (token skipped),
 * 2 = a slot outside [0, num_pages * page_size) (cache write skipped).
 * k_scale_exp, if not NULL, receives each token's scale exponent. */
static int k_prepare_store(int64_t T, const uint16_t* k, int64_t k_stride_t,
                           const int64_t* positions, const int64_t* slots,
                           const float* cos_t, const float* sin_t,
                           int64_t cs_stride, int64_t max_position,
                           const float* gamma, const float* beta, float eps,
                           uint8_t* cache, int64_t num_pages, int32_t page_size,
                           int32_t rope_dim, int32_t style,
                           int32_t bf16_intermediate, int32_t* k_scale_exp,
                           int32_t token_major, int32_t hadamard) {
  int err = 0;
  for (int64_t t = 0; t < T; ++t) {
    int64_t pos = positions[t];
    if (pos < 0 || pos >= max_position) {
      err |= 1;
      continue;
    }
    uint8_t codes[DSA_D];
    int e = prepare_k(k + t * k_stride_t, cos_t + pos * cs_stride,
                      sin_t + pos * cs_stride, gamma, beta, eps, rope_dim,
                      style, bf16_intermediate, hadamard, codes);
    if (k_scale_exp) k_scale_exp[t] = e;
    int64_t slot = slots[t];
    if (slot < 0 || slot >= num_pages * (int64_t)page_size) {
      err |= 2;
      continue;
    }
    store_index_k(cache, slot, page_size, codes, e, token_major);
  }
  return err;
}

int oracle_k_prepare_store(int64_t T, const uint16_t* k, int64_t k_stride_t,
                           const int64_t* positions, const int64_t* slots,
                           const float* cos_t, const float* sin_t,
                           int64_t cs_stride, int64_t max_position,
                           const float* gamma, const float* beta, float eps,
                           uint8_t* cache, int64_t num_pages, int32_t page_size,
                           int32_t rope_dim, int32_t style,
                           int32_t bf16_intermediate, int32_t* k_scale_exp,
                           int32_t token_major) {
  return k_prepare_store(T, k, k_stride_t, positions, slots, cos_t, sin_t, cs_stride,
                         max_position, gamma, beta, eps, cache, num_pages, page_size,
                         rope_dim, style, bf16_intermediate, k_scale_exp, token_major, 0);
}

/* Both Q/K writers; chain != 0 rounds the tensors the four-launch chain
 * hands between launches to bf16 (see prepare_k); hadamard != 0 rotates
 * every rotated q head and k by oracle_hadamard before quantising. */
static int qk_prepare_store(
    int64_t T, int32_t H, const uint16_t* q, int64_t q_stride_t,
    int64_t q_stride_h, const uint16_t* k, int64_t k_stride_t,
    const uint16_t* w, int64_t w_stride_t, const int64_t* positions,
    const int64_t* slots, const float* cos_t, const float* sin_t,
    int64_t cs_stride, int64_t max_position, const float* gamma,
    const float* beta, float eps, float softmax_scale, uint8_t* q_fp8,
    float* weights, uint8_t* cache, int64_t num_pages, int32_t page_size,
    int32_t rope_dim, int32_t style, int32_t* q_scale_exp,
    int32_t* k_scale_exp, int chain, int32_t token_major, int hadamard) {
  int err = 0;
  double head_factor = 1.0 / sqrt((double)H);
  for (int64_t t = 0; t < T; ++t) {
    int64_t pos = positions[t];
    if (pos < 0 || pos >= max_position) {
      err |= 1;
      continue;
    }
    const float* cos_row = cos_t + pos * cs_stride;
    const float* sin_row = sin_t + pos * cs_stride;
    for (int32_t h = 0; h < H; ++h) {
      const uint16_t* qrow = q + t * q_stride_t + h * q_stride_h;
      float z[DSA_D];
      for (int j = 0; j < DSA_D; ++j) z[j] = bf16_to_f32(qrow[j]);
      oracle_rope(z, cos_row, sin_row, rope_dim, style);
      if (hadamard) oracle_hadamard(z);
      if (chain)
        for (int j = 0; j < DSA_D; ++j) z[j] = round_to_bf16(z[j]);
      int e = oracle_quantize_vector(z, q_fp8 + (t * H + h) * DSA_D);
      if (q_scale_exp) q_scale_exp[t * H + h] = e;
      double wv = (double)bf16_to_f32(w[t * w_stride_t + h]);
      weights[t * H + h] =
          (float)(wv * ldexp(1.0, e) * (double)softmax_scale * head_factor);
    }
    err |= k_prepare_store(1, k + t * k_stride_t, k_stride_t,
                           positions + t, slots + t, cos_t, sin_t,
                           cs_stride, max_position, gamma, beta, eps,
                           cache, num_pages, page_size, rope_dim, style,
                           chain ? 2 : 0, k_scale_exp ? k_scale_exp + t : NULL,
                           token_major, hadamard);
  }
  return err;
}

/* The fused Q/K prepare-and-store ([FUSE-QK] Motivation and Modifications:
 * one call returns (q_fp8, weights) and writes the index-K cache; [FUSE-Q]
 * Summary: RoPE + FP8 quantization + weight-scale fold on the q side).
 * q_fp8 is [T, H, 128] e4m3 codes, weights is [T, H] fp32:
 *   weights[t, h] = w[t, h] * 2^e_q[t, h] * softmax_scale * H^-0.5. */
int oracle_qk_prepare_store(
    int64_t T, int32_t H, const uint16_t* q, int64_t q_stride_t,
    int64_t q_stride_h, const uint16_t* k, int64_t k_stride_t,
    const uint16_t* w, int64_t w_stride_t, const int64_t* positions,
    const int64_t* slots, const float* cos_t, const float* sin_t,
    int64_t cs_stride, int64_t max_position, const float* gamma,
    const float* beta, float eps, float softmax_scale, uint8_t* q_fp8,
    float* weights, uint8_t* cache, int64_t num_pages, int32_t page_size,
    int32_t rope_dim, int32_t style, int32_t* q_scale_exp,
    int32_t* k_scale_exp, int32_t token_major) {
  return qk_prepare_store(T, H, q, q_stride_t, q_stride_h, k, k_stride_t, w,
                          w_stride_t, positions, slots, cos_t, sin_t, cs_stride,
                          max_position, gamma, beta, eps, softmax_scale, q_fp8,
                          weights, cache, num_pages, page_size, rope_dim, style,
                          q_scale_exp, k_scale_exp, 0, token_major, 0);
}

/* The same outputs as written by the four-launch chain of [FUSE-QK] Profile,
 * whose launches pass bf16 tensors: the key's LayerNorm output and every
 * rotated vector (q and k) are rounded to bf16 before the next step. */
int oracle_qk_prepare_store_chain(
    int64_t T, int32_t H, const uint16_t* q, int64_t q_stride_t,
    int64_t q_stride_h, const uint16_t* k, int64_t k_stride_t,
    const uint16_t* w, int64_t w_stride_t, const int64_t* positions,
    const int64_t* slots, const float* cos_t, const float* sin_t,
    int64_t cs_stride, int64_t max_position, const float* gamma,
    const float* beta, float eps, float softmax_scale, uint8_t* q_fp8,
    float* weights, uint8_t* cache, int64_t num_pages, int32_t page_size,
    int32_t rope_dim, int32_t style, int32_t* q_scale_exp,
    int32_t* k_scale_exp, int32_t token_major) {
  return qk_prepare_store(T, H, q, q_stride_t, q_stride_h, k, k_stride_t, w,
                          w_stride_t, positions, slots, cos_t, sin_t, cs_stride,
                          max_position, gamma, beta, eps, softmax_scale, q_fp8,
                          weights, cache, num_pages, page_size, rope_dim, style,
                          q_scale_exp, k_scale_exp, 1, token_major, 0);
}

/* The Q/K writer with the Hadamard rotation (see oracle_hadamard): every
 * rotated q head and the normalised, rotated k pass through H_128 / sqrt(128)
 * before they are quantised. */
int oracle_qk_prepare_store_hadamard(
    int64_t T, int32_t H, const uint16_t* q, int64_t q_stride_t,
    int64_t q_stride_h, const uint16_t* k, int64_t k_stride_t,
    const uint16_t* w, int64_t w_stride_t, const int64_t* positions,
    const int64_t* slots, const float* cos_t, const float* sin_t,
    int64_t cs_stride, int64_t max_position, const float* gamma,
    const float* beta, float eps, float softmax_scale, uint8_t* q_fp8,
    float* weights, uint8_t* cache, int64_t num_pages, int32_t page_size,
    int32_t rope_dim, int32_t style, int32_t* q_scale_exp,
    int32_t* k_scale_exp, int32_t token_major) {
  return qk_prepare_store(T, H, q, q_stride_t, q_stride_h, k, k_stride_t, w,
                          w_stride_t, positions, slots, cos_t, sin_t, cs_stride,
                          max_position, gamma, beta, eps, softmax_scale, q_fp8,
                          weights, cache, num_pages, page_size, rope_dim, style,
                          q_scale_exp, k_scale_exp, 0, token_major, 1);
}

/* ------------------------------------------------------------ the consumer */

/* The indexer's fp8 paged MQA logits, the kernel that reads this path's
 * outputs ([FUSE-Q] Kernel-level evidence lists it after the index-K store as
 * "_gluon_deepgemm_fp8_paged_mqa_logits"; the pages give no formula).  It is
 * read from the DeepSeek sparse-attention indexer: a score per (query token,
 * key) is the gate-weighted sum over heads of the ReLU'd dot product,
 *   logits[t, j] = k_scale[j] * sum_h weights[t, h] * max(q[t, h] . k[j], 0)
 * with q and k the decoded e4m3 codes; weights already hold the q scales, and
 * since every scale is a positive power of two it moves through the ReLU.
 * Key j of token t sits in page block_table[t][j / page_size], row
 * j % page_size of the page-blocked index-K cache.  Columns j >= context_lens[t]
 * (up to max_context) are -inf.  Computed in double, rounded once.  Returns 2
 * if a block-table entry is out of range (that key's logit is then NaN). */
int oracle_mqa_logits(int32_t T, int32_t H, const uint8_t* q_fp8,
                      const float* weights, const uint8_t* cache,
                      int64_t num_pages, int32_t page_size,
                      const int32_t* block_table, int64_t bt_stride,
                      const int32_t* context_lens, float* logits,
                      int64_t logits_stride, int32_t max_context) {
  int err = 0;
  double dec[256];
  for (int c = 0; c < 256; ++c) dec[c] = (double)oracle_e4m3_decode((uint8_t)c);
  for (int32_t t = 0; t < T; ++t) {
    for (int32_t j = 0; j < max_context; ++j) {
      float* out = logits + (int64_t)t * logits_stride + j;
      if (j >= context_lens[t]) {
        *out = -INFINITY;
        continue;
      }
      int64_t page = block_table[(int64_t)t * bt_stride + j / page_size];
      if (page < 0 || page >= num_pages) {
        err |= 2;
        *out = NAN;
        continue;
      }
      const uint8_t* base = cache + page * (int64_t)page_size * (DSA_D + 4);
      const uint8_t* kc = base + (int64_t)(j % page_size) * DSA_D;
      float kscale;
      memcpy(&kscale, base + (int64_t)page_size * DSA_D + 4 * (j % page_size), 4);
      double acc = 0.0;
      for (int32_t h = 0; h < H; ++h) {
        const uint8_t* qc = q_fp8 + ((int64_t)t * H + h) * DSA_D;
        double dot = 0.0;
        for (int d = 0; d < DSA_D; ++d) dot += dec[qc[d]] * dec[kc[d]];
        acc += (double)weights[(int64_t)t * H + h] * (dot > 0.0 ? dot : 0.0);
      }
      *out = (float)(acc * (double)kscale);
    }
  }
  return err;
}
