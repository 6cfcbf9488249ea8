// DSA indexer Q/K prepare-and-store for GB300 (sm_103a): kernels, launcher
// and the C ABI declared in include/dsa_prep.h.
//
// The work is one streaming pass (HBM-bound, ~1 flop per byte): per token,
// H query heads and one key of 128 bf16 each are rotated, quantised to e4m3
// with a power-of-two scale and written out; the key is LayerNorm'd first and
// scattered into the paged index-K cache; the gate weights absorb the query
// scales.  (sglang PR "[AMD] [GLM5] Fuse the DSA indexer Q/K rope + quant +
// K-cache write", Motivation and Modifications; vllm PR "[ROCm][Perf] Enable
// fused indexer-Q RoPE+quant kernel for DeepSeek/GLM sparse attention",
// Summary.)
//
// Mapping: a 128-vector belongs to one half-warp; lane l16 holds elements
// 8*l16 .. 8*l16+7 (one 16-byte load of bf16, one 8-byte store of codes).
// A warp works on two vectors of the same kind at a time:
//   * q work item = one token and G consecutive heads (G loads in flight per
//     lane, one cos/sin read shared by the G heads);
//   * k work item = one token's key (LayerNorm, RoPE, quantise, cache store).
// Warp units [0, q_units) are q items (two per warp), the rest k items (two
// per warp), so no warp mixes the two code paths and every shuffle runs with
// the whole warp converged.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "dsa_prep.h"

namespace {

constexpr int kD = DSA_HEAD_DIM;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr int64_t kMaxBlocks = 1 << 20;

struct Params {
  const uint16_t* q;
  int64_t sq_t, sq_h;
  const uint16_t* k;
  int64_t sk_t;
  const uint16_t* w;
  int64_t sw_t;
  const int64_t* pos;
  const int64_t* loc;
  const float* cos_t;
  const float* sin_t;
  int64_t cs_stride;
  int64_t max_pos;
  const float* gamma;
  const float* beta;
  float eps;
  float fold;  // softmax_scale * H^-0.5, rounded once to fp32
  uint8_t* q_out;
  float* w_out;
  uint8_t* cache;
  int64_t num_slots;
  int64_t page_bytes;  // page_size * 132
  int32_t page_size;
  int32_t T;
  int32_t H;
  int32_t rope_dim;
  int32_t n_groups;  // ceil(H / G)
  int64_t q_units;   // warps of q work
  int64_t k_units;   // warps of k work
  int32_t* err;
};

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_stream8(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y)
               : "memory");
}

__device__ __forceinline__ void unpack_bf16x8(uint4 r, float (&x)[8]) {
  x[0] = __uint_as_float(r.x << 16);
  x[1] = __uint_as_float(r.x & 0xffff0000u);
  x[2] = __uint_as_float(r.y << 16);
  x[3] = __uint_as_float(r.y & 0xffff0000u);
  x[4] = __uint_as_float(r.z << 16);
  x[5] = __uint_as_float(r.z & 0xffff0000u);
  x[6] = __uint_as_float(r.w << 16);
  x[7] = __uint_as_float(r.w & 0xffff0000u);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// cos/sin values this lane needs for its slice of the rope dims.
//   NeoX: lanes [0, r/16) hold the first members of pairs 8*l16 .. 8*l16+7 and
//         lanes [r/16, r/8) the second members of the same pairs.
//   GPT-J: lane l16 < r/8 holds pairs 4*l16 .. 4*l16+3 inside its own 8 values.
template <int STYLE>
__device__ __forceinline__ void load_cos_sin(const Params& p, int64_t row, int l16,
                                             float (&c)[8], float (&s)[8]) {
  const int rl = p.rope_dim >> 4;
  if (STYLE == DSA_ROPE_NEOX) {
    if (l16 < 2 * rl) {
      const int base = 8 * (l16 < rl ? l16 : l16 - rl);
      const float4* cp = reinterpret_cast<const float4*>(p.cos_t + row * p.cs_stride + base);
      const float4* sp = reinterpret_cast<const float4*>(p.sin_t + row * p.cs_stride + base);
      float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
      c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
      c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
      s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
      s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
    }
  } else {
    if (l16 < 2 * rl) {
      float4 c0 = __ldg(reinterpret_cast<const float4*>(p.cos_t + row * p.cs_stride + 4 * l16));
      float4 s0 = __ldg(reinterpret_cast<const float4*>(p.sin_t + row * p.cs_stride + 4 * l16));
      c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
      s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
    }
  }
}

// RoPE on this lane's 8 values: (a, b) -> (fma(a, c, -(b*s)), fma(b, c, a*s)),
// products rounded to fp32 (no contraction).  Every lane of the warp must call
// it (NeoX exchanges values with the partner lane r/16 away).
template <int STYLE>
__device__ __forceinline__ void rope_apply(float (&x)[8], int l16, int rope_dim,
                                           const float (&c)[8], const float (&s)[8]) {
  const int rl = rope_dim >> 4;
  if (STYLE == DSA_ROPE_NEOX) {
    const bool first = l16 < rl;
    const bool rot = l16 < 2 * rl;
    const int partner = first ? l16 + rl : (rot ? l16 - rl : l16);
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __shfl_sync(kFull, x[j], partner, 16);
    if (rot) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float ps = __fmul_rn(o[j], s[j]);
        x[j] = __fmaf_rn(x[j], c[j], first ? -ps : ps);
      }
    }
  } else {
    if (l16 < 2 * rl) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = x[2 * j], b = x[2 * j + 1];
        x[2 * j] = __fmaf_rn(a, c[j], -__fmul_rn(b, s[j]));
        x[2 * j + 1] = __fmaf_rn(b, c[j], __fmul_rn(a, s[j]));
      }
    }
  }
}

// Half-warp reductions (xor offsets 8..1 never leave the 16-lane group).
__device__ __forceinline__ float halfwarp_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 8));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 4));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 2));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 1));
  return v;
}

__device__ __forceinline__ float halfwarp_sum(float v) {
  v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 8));
  v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 4));
  v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 2));
  v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 1));
  return v;
}

// ue8m0 exponent of the vector: the smallest e with max(amax, 1e-4) <= 448*2^e.
// With A = max(amax, 1e-4) = 1.f * 2^E (normal), 448 * 2^e = 1.75 * 2^(e+8), so
// e = E - 8 when the fraction is <= 0.75 (bits <= 0x600000) and E - 7 above:
// read straight off the exponent and fraction bits, no division or log.
__device__ __forceinline__ int ue8m0_exponent(const float (&x)[8]) {
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(x[j]));
  m = fmaxf(halfwarp_max(m), 1e-4f);
  const uint32_t b = __float_as_uint(m);
  return static_cast<int>(b >> 23) - 127 - 8 + ((b & 0x7fffffu) > 0x600000u ? 1 : 0);
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// codes = e4m3_rne(x * 2^-e): the multiply by a power of two is exact.
__device__ __forceinline__ uint2 quantize8(const float (&x)[8], int e) {
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  const uint32_t p0 = cvt_e4m3x2(__fmul_rn(x[0], inv), __fmul_rn(x[1], inv));
  const uint32_t p1 = cvt_e4m3x2(__fmul_rn(x[2], inv), __fmul_rn(x[3], inv));
  const uint32_t p2 = cvt_e4m3x2(__fmul_rn(x[4], inv), __fmul_rn(x[5], inv));
  const uint32_t p3 = cvt_e4m3x2(__fmul_rn(x[6], inv), __fmul_rn(x[7], inv));
  return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
}

// ---------------------------------------------------------------- q side

template <int STYLE, int G>
__device__ __forceinline__ void q_item(const Params& p, int64_t item, int l16) {
  const int64_t n_items = static_cast<int64_t>(p.T) * p.n_groups;
  const bool valid = item < n_items;
  const int64_t t = valid ? item / p.n_groups : 0;
  const int h0 = valid ? static_cast<int>(item - t * p.n_groups) * G : 0;

  const int64_t pos = valid ? __ldg(p.pos + t) : 0;
  uint4 raw[G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    raw[j] = make_uint4(0, 0, 0, 0);
    if (valid && h0 + j < p.H)
      raw[j] = ld_stream16(p.q + t * p.sq_t + static_cast<int64_t>(h0 + j) * p.sq_h + 8 * l16);
  }
  float wv = 0.0f;
  if (valid && l16 < G && h0 + l16 < p.H) wv = bf16_to_f32(__ldg(p.w + t * p.sw_t + h0 + l16));

  const bool pos_ok = pos >= 0 && pos < p.max_pos;
  float c[8] = {}, s[8] = {};
  load_cos_sin<STYLE>(p, (valid && pos_ok) ? pos : 0, l16, c, s);

  const bool store = valid && pos_ok;
  int es[G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    float x[8];
    unpack_bf16x8(raw[j], x);
    rope_apply<STYLE>(x, l16, p.rope_dim, c, s);
    const int e = ue8m0_exponent(x);
    es[j] = e;
    const uint2 codes = quantize8(x, e);
    if (store && h0 + j < p.H)
      st_stream8(p.q_out + ((t * p.H + h0 + j) * kD + 8 * l16), codes);
  }
  // gate fold: lane j of the half-warp writes head h0 + j
  if (store && l16 < G && h0 + l16 < p.H) {
    int e = es[0];
#pragma unroll
    for (int j = 1; j < G; ++j)
      if (l16 == j) e = es[j];
    const float scale = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    __stcs(p.w_out + t * p.H + h0 + l16, __fmul_rn(__fmul_rn(wv, scale), p.fold));
  }
}

// ---------------------------------------------------------------- k side

template <int STYLE>
__device__ __forceinline__ void k_item(const Params& p, int64_t t, int l16) {
  const bool valid = t < p.T;
  const int64_t tt = valid ? t : 0;
  const int64_t pos = valid ? __ldg(p.pos + tt) : 0;
  const int64_t slot = valid ? __ldg(p.loc + tt) : 0;
  const uint4 raw = valid ? ld_stream16(p.k + tt * p.sk_t + 8 * l16) : make_uint4(0, 0, 0, 0);
  const float4* g4 = reinterpret_cast<const float4*>(p.gamma + 8 * l16);
  const float4* b4 = reinterpret_cast<const float4*>(p.beta + 8 * l16);
  const float4 g0 = __ldg(g4), g1 = __ldg(g4 + 1), b0 = __ldg(b4), b1 = __ldg(b4 + 1);
  const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  const float bt[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};

  const bool pos_ok = pos >= 0 && pos < p.max_pos;
  float c[8] = {}, s[8] = {};
  load_cos_sin<STYLE>(p, (valid && pos_ok) ? pos : 0, l16, c, s);

  // LayerNorm over the 128 values: mean, biased variance, eps inside the root
  float x[8];
  unpack_bf16x8(raw, x);
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) sum = __fadd_rn(sum, x[j]);
  const float mean = __fmul_rn(halfwarp_sum(sum), 1.0f / kD);
  float sq = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    x[j] = __fsub_rn(x[j], mean);
    sq = __fmaf_rn(x[j], x[j], sq);
  }
  const float var = __fmul_rn(halfwarp_sum(sq), 1.0f / kD);
  const float rstd = __frsqrt_rn(__fadd_rn(var, p.eps));
#pragma unroll
  for (int j = 0; j < 8; ++j) x[j] = __fmaf_rn(__fmul_rn(x[j], rstd), g[j], bt[j]);

  rope_apply<STYLE>(x, l16, p.rope_dim, c, s);
  const int e = ue8m0_exponent(x);
  const uint2 codes = quantize8(x, e);

  if (!valid) return;
  if (!pos_ok) {
    if (l16 == 0 && p.err) atomicOr(p.err, DSA_DEVERR_POSITION);
    return;
  }
  if (slot < 0 || slot >= p.num_slots) {
    if (l16 == 0 && p.err) atomicOr(p.err, DSA_DEVERR_SLOT);
    return;
  }
  const int64_t page = slot / p.page_size;
  const int64_t off = slot - page * p.page_size;
  uint8_t* base = p.cache + page * p.page_bytes;
  *reinterpret_cast<uint2*>(base + off * kD + 8 * l16) = codes;
  if (l16 == 0)
    *reinterpret_cast<float*>(base + static_cast<int64_t>(p.page_size) * kD + 4 * off) =
        __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// ---------------------------------------------------------------- kernel

template <int STYLE, int G>
__global__ void __launch_bounds__(kThreads) dsa_prepare_store_kernel(const Params p) {
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int hw = lane >> 4;
  const int l16 = lane & 15;
  const int64_t total = p.q_units + p.k_units;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * kWarps + warp; u < total;
       u += static_cast<int64_t>(gridDim.x) * kWarps) {
    if (u < p.q_units)
      q_item<STYLE, G>(p, 2 * u + hw, l16);
    else
      k_item<STYLE>(p, 2 * (u - p.q_units) + hw, l16);
  }
}

// ---------------------------------------------------------------- host side

bool misaligned(const void* ptr, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
}

// Heads per q work item: more loads in flight per lane for large calls, more
// independent items (spread over more SMs) for small ones.
int choose_group(int64_t T, int32_t H) {
  const int64_t vecs = T * static_cast<int64_t>(H);
  if (vecs >= 65536) return 4;
  if (vecs >= 16384) return 2;
  return 1;
}

template <int STYLE, int G>
cudaError_t launch_typed(const Params& p, cudaStream_t stream) {
  const int64_t total = p.q_units + p.k_units;
  int64_t blocks = (total + kWarps - 1) / kWarps;
  if (blocks > kMaxBlocks) blocks = kMaxBlocks;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, dsa_prepare_store_kernel<STYLE, G>, p);
}

template <int STYLE>
cudaError_t launch_style(const Params& p, int G, cudaStream_t stream) {
  switch (G) {
    case 4: return launch_typed<STYLE, 4>(p, stream);
    case 2: return launch_typed<STYLE, 2>(p, stream);
    default: return launch_typed<STYLE, 1>(p, stream);
  }
}

dsa_status check_k_side(const void* k, int64_t k_stride_t, const int64_t* positions,
                        const int64_t* out_cache_loc, const float* cos_cache,
                        const float* sin_cache, int64_t cs_stride, int64_t max_position,
                        const float* ln_gamma, const float* ln_beta, float ln_eps,
                        const void* index_k_cache, int64_t num_pages, int32_t page_size,
                        int32_t T, int32_t head_dim, int32_t rope_dim, int32_t rope_style) {
  if (T < 0) return DSA_ERR_SHAPE;
  if (head_dim != kD) return DSA_ERR_UNSUPPORTED;
  if (rope_dim < 0 || rope_dim > kD || rope_dim % 16 != 0) return DSA_ERR_UNSUPPORTED;
  if (rope_style != DSA_ROPE_NEOX && rope_style != DSA_ROPE_GPTJ) return DSA_ERR_UNSUPPORTED;
  if (!(ln_eps >= 0.0f) || !std::isfinite(ln_eps)) return DSA_ERR_UNSUPPORTED;
  if (page_size < 1 || num_pages < 1 || max_position < 1) return DSA_ERR_SHAPE;
  if (num_pages > INT64_MAX / (static_cast<int64_t>(page_size) * (kD + 4)))
    return DSA_ERR_SHAPE;
  if (k_stride_t < 0 || cs_stride < 0) return DSA_ERR_SHAPE;
  if (T == 0) return DSA_OK;
  if (!k || !positions || !out_cache_loc || !ln_gamma || !ln_beta || !index_k_cache)
    return DSA_ERR_NULL;
  if (rope_dim > 0 && (!cos_cache || !sin_cache)) return DSA_ERR_NULL;
  if (rope_dim > 0 && cs_stride < rope_dim / 2) return DSA_ERR_SHAPE;
  if (page_size % 4 != 0) return DSA_ERR_ALIGN;
  if (misaligned(k, 16) || k_stride_t % 8 != 0) return DSA_ERR_ALIGN;
  if (misaligned(positions, 8) || misaligned(out_cache_loc, 8)) return DSA_ERR_ALIGN;
  if (misaligned(ln_gamma, 16) || misaligned(ln_beta, 16)) return DSA_ERR_ALIGN;
  if (misaligned(index_k_cache, 16)) return DSA_ERR_ALIGN;
  if (rope_dim > 0 && (misaligned(cos_cache, 16) || misaligned(sin_cache, 16) ||
                       cs_stride % 4 != 0))
    return DSA_ERR_ALIGN;
  return DSA_OK;
}

void fill_k_side(Params& p, const void* k, int64_t k_stride_t, const int64_t* positions,
                 const int64_t* out_cache_loc, const float* cos_cache, const float* sin_cache,
                 int64_t cs_stride, int64_t max_position, const float* ln_gamma,
                 const float* ln_beta, float ln_eps, void* index_k_cache, int64_t num_pages,
                 int32_t page_size, int32_t T, int32_t rope_dim, int32_t* err_flags) {
  p.k = static_cast<const uint16_t*>(k);
  p.sk_t = k_stride_t;
  p.pos = positions;
  p.loc = out_cache_loc;
  p.cos_t = cos_cache;
  p.sin_t = sin_cache;
  p.cs_stride = cs_stride;
  p.max_pos = max_position;
  p.gamma = ln_gamma;
  p.beta = ln_beta;
  p.eps = ln_eps;
  p.cache = static_cast<uint8_t*>(index_k_cache);
  p.num_slots = num_pages * page_size;
  p.page_size = page_size;
  p.page_bytes = static_cast<int64_t>(page_size) * (kD + 4);
  p.T = T;
  p.rope_dim = rope_dim;
  p.k_units = (static_cast<int64_t>(T) + 1) / 2;
  p.err = err_flags;
}

}  // namespace

extern "C" {

dsa_status dsa_indexer_qk_prepare_store(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k, int64_t k_stride_t,
    const void* w, int64_t w_stride_t, const int64_t* positions, const int64_t* out_cache_loc,
    const float* cos_cache, const float* sin_cache, int64_t cs_stride, int64_t max_position,
    const float* ln_gamma, const float* ln_beta, float ln_eps, float softmax_scale,
    void* q_fp8_out, float* weights_out, void* index_k_cache, int64_t num_pages,
    int32_t page_size, int32_t T, int32_t H, int32_t head_dim, int32_t rope_dim,
    int32_t rope_style, int32_t* err_flags, void* stream) {
  dsa_status st = check_k_side(k, k_stride_t, positions, out_cache_loc, cos_cache, sin_cache,
                               cs_stride, max_position, ln_gamma, ln_beta, ln_eps,
                               index_k_cache, num_pages, page_size, T, head_dim, rope_dim,
                               rope_style);
  if (st != DSA_OK) return st;
  if (H < 1 || H > 4096) return DSA_ERR_SHAPE;
  if (q_stride_t < 0 || q_stride_h < 0 || w_stride_t < H) return DSA_ERR_SHAPE;
  if (!std::isfinite(softmax_scale)) return DSA_ERR_UNSUPPORTED;
  if (T == 0) return DSA_OK;
  if (!q || !w || !q_fp8_out || !weights_out) return DSA_ERR_NULL;
  if (misaligned(q, 16) || q_stride_t % 8 != 0 || q_stride_h % 8 != 0) return DSA_ERR_ALIGN;
  if (misaligned(w, 2)) return DSA_ERR_ALIGN;
  if (misaligned(q_fp8_out, 16) || misaligned(weights_out, 4)) return DSA_ERR_ALIGN;

  Params p = {};
  fill_k_side(p, k, k_stride_t, positions, out_cache_loc, cos_cache, sin_cache, cs_stride,
              max_position, ln_gamma, ln_beta, ln_eps, index_k_cache, num_pages, page_size, T,
              rope_dim, err_flags);
  const int G = choose_group(T, H);
  p.q = static_cast<const uint16_t*>(q);
  p.sq_t = q_stride_t;
  p.sq_h = q_stride_h;
  p.w = static_cast<const uint16_t*>(w);
  p.sw_t = w_stride_t;
  p.fold = static_cast<float>(static_cast<double>(softmax_scale) / std::sqrt(static_cast<double>(H)));
  p.q_out = static_cast<uint8_t*>(q_fp8_out);
  p.w_out = weights_out;
  p.H = H;
  p.n_groups = (H + G - 1) / G;
  p.q_units = (static_cast<int64_t>(T) * p.n_groups + 1) / 2;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = rope_style == DSA_ROPE_NEOX ? launch_style<DSA_ROPE_NEOX>(p, G, s)
                                              : launch_style<DSA_ROPE_GPTJ>(p, G, s);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_LAUNCH;
}

dsa_status dsa_indexer_k_prepare_store(
    const void* k, int64_t k_stride_t, const int64_t* positions, const int64_t* out_cache_loc,
    const float* cos_cache, const float* sin_cache, int64_t cs_stride, int64_t max_position,
    const float* ln_gamma, const float* ln_beta, float ln_eps, void* index_k_cache,
    int64_t num_pages, int32_t page_size, int32_t T, int32_t head_dim, int32_t rope_dim,
    int32_t rope_style, int32_t* err_flags, void* stream) {
  dsa_status st = check_k_side(k, k_stride_t, positions, out_cache_loc, cos_cache, sin_cache,
                               cs_stride, max_position, ln_gamma, ln_beta, ln_eps,
                               index_k_cache, num_pages, page_size, T, head_dim, rope_dim,
                               rope_style);
  if (st != DSA_OK || T == 0) return st;
  Params p = {};
  fill_k_side(p, k, k_stride_t, positions, out_cache_loc, cos_cache, sin_cache, cs_stride,
              max_position, ln_gamma, ln_beta, ln_eps, index_k_cache, num_pages, page_size, T,
              rope_dim, err_flags);
  p.n_groups = 1;
  p.q_units = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = rope_style == DSA_ROPE_NEOX ? launch_typed<DSA_ROPE_NEOX, 1>(p, s)
                                              : launch_typed<DSA_ROPE_GPTJ, 1>(p, s);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_LAUNCH;
}

const char* dsa_status_string(dsa_status status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_NULL: return "a required pointer is NULL";
    case DSA_ERR_ALIGN: return "a pointer or stride breaks an alignment rule";
    case DSA_ERR_SHAPE: return "a negative or inconsistent size or stride";
    case DSA_ERR_UNSUPPORTED: return "unsupported head_dim, rope_dim, rope_style or scalar";
    case DSA_ERR_LAUNCH: return "the CUDA kernel launch failed";
  }
  return "unknown status";
}

int32_t dsa_prep_version(void) { return (1 << 16) | 0; }

}  // extern "C"
