// The unfused DSA indexer prologue: the same steps as the fused kernels,
// split into the four launches per full-indexer layer and decode step that the
// sglang PR "[AMD] [GLM5] Fuse the DSA indexer Q/K rope + quant + K-cache
// write" lists in its Profile section -- rope on q and k, LayerNorm on k, the
// q activation quant (here with the head-gate fold), and the k quant + index-K
// cache store -- with bf16 tensors handed from launch to launch through a
// workspace.  It is the baseline the fusion is measured against (4 launches
// and ~2.3x the HBM bytes of the fused call), re-created for sm_103a.
//
// Order: LayerNorm(k) -> RoPE(q, k) -> quant(q) + fold -> quant(k) + store.
// Workspace (bf16, 256-byte aligned segments): k_ln [T,128], q_rot [T,H,128],
// k_rot [T,128].  Every kernel is a quarter-warp per 128-row streaming pass.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "dsa_common.cuh"
#include "dsa_prep.h"

namespace {

using namespace dsa_dev;

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = kThreads / 8;  // one row per quarter-warp

struct UParams {
  const uint16_t* q;
  long long sq_t, sq_h;
  const uint16_t* k;
  long long sk_t;
  const uint16_t* w;
  long long sw_t;
  const long long* pos;
  const long long* loc;
  const float* cos_t;
  const float* sin_t;
  long long cs_stride;
  long long max_pos;
  const float* gamma;
  const float* beta;
  float eps;
  float fold;  // softmax_scale * H^-0.5, rounded once to fp32
  uint8_t* q_out;
  float* w_out;
  CacheGeom cg;
  int T;
  int H;
  int rope_dim;
  uint16_t* k_ln;   // [T, 128]
  uint16_t* q_rot;  // [T, H, 128]
  uint16_t* k_rot;  // [T, 128]
  int* err;
};

// The row index of this quarter-warp; rows beyond n do nothing but still run
// the shuffles with their warp.
__device__ __forceinline__ long long row_of_quarter() {
  return static_cast<long long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 3);
}

__device__ __forceinline__ bool position_ok(const UParams& p, long long t, long long& pos) {
  pos = __ldg(p.pos + t);
  return pos >= 0 && pos < p.max_pos;
}

// 16 fp32 values of a contiguous slice -> 16 bf16 (RNE) -> 32 bytes at dst.
__device__ __forceinline__ void store_bf16x16(uint16_t* dst, const float (&x)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
  store_codes<32, 16, false>(reinterpret_cast<uint8_t*>(dst), w);
}

// bf16 of a balanced slice (chunk layout of Slice<STYLE, RP>) back to its row.
template <int STYLE, int RP>
__device__ __forceinline__ void store_bf16_slice(uint16_t* row, int l, const float (&x)[16]) {
  using S = Slice<STYLE, RP>;
  uint8_t* b = reinterpret_cast<uint8_t*>(row);
  if constexpr (RP > 0) {
    if constexpr (S::NEOX) {
      uint32_t wa[4], wb[4];
#pragma unroll
      for (int j = 0; j < RP; j += 2) {
        wa[j / 2] = pack_bf16x2(x[j], RP > 1 ? x[j + 1] : 0.0f);
        wb[j / 2] = pack_bf16x2(x[RP + j], RP > 1 ? x[RP + j + 1] : 0.0f);
      }
      store_codes<2 * RP, S::ALIGN_A_BF16, false>(b + 2 * RP * l, wa);
      store_codes<2 * RP, S::ALIGN_B_BF16, false>(b + 2 * (S::B_BASE + RP * l), wb);
    } else {
      uint32_t wr[8];
#pragma unroll
      for (int j = 0; j < RP; ++j) wr[j] = pack_bf16x2(x[j], x[RP + j]);
      store_codes<4 * RP, S::ALIGN_A_BF16, false>(b + 4 * RP * l, wr);
    }
  }
  if constexpr (S::NP > 0) {
    uint32_t wp[8];
#pragma unroll
    for (int j = 0; j < S::NP; j += 2) wp[j / 2] = pack_bf16x2(x[2 * RP + j], x[2 * RP + j + 1]);
    store_codes<2 * S::NP, S::ALIGN_P_BF16, false>(b + 2 * (S::P_BASE + S::NP * l), wp);
  }
}

// ---------------------------------------------------------------- launch 1
// LayerNorm of every key row (mean, biased variance, eps inside the root,
// fp32 gamma / beta), written as bf16.
__global__ void __launch_bounds__(kThreads) unfused_layernorm_kernel(const UParams p) {
  grid_launch_dependents();
  grid_dependency_wait();
  const long long t = row_of_quarter();
  const int l = threadIdx.x & 7;
  const bool real = t < p.T;
  float x[16] = {};
  if (real)
    load_slice<0, 0, GlobalMem>(reinterpret_cast<const unsigned char*>(p.k + t * p.sk_t), l, x);
  // two-pass sums (the fused kernels merge per-lane statistics instead; the
  // chain is a baseline, not a latency path)
  float sum = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) sum = __fadd_rn(sum, x[j]);
  const float mean = __fmul_rn(quad_sum(sum), 1.0f / kD);
  float sq = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    x[j] = __fsub_rn(x[j], mean);
    sq = __fmaf_rn(x[j], x[j], sq);
  }
  const float rstd = __frsqrt_rn(__fadd_rn(__fmul_rn(quad_sum(sq), 1.0f / kD), p.eps));
  affine_slice<0, 0>(p.gamma, p.beta, l, x, rstd);
  if (real) store_bf16x16(p.k_ln + t * kD + 16 * l, x);
}

// ---------------------------------------------------------------- launch 2
// RoPE on every query row and every normalised key row, written as bf16.
// Rows [0, T*H) are queries (t = row / H), rows [T*H, T*H + T) keys.
template <int STYLE, int RP>
__global__ void __launch_bounds__(kThreads) unfused_rope_kernel(const UParams p) {
  grid_launch_dependents();
  grid_dependency_wait();
  const long long row = row_of_quarter();
  const int l = threadIdx.x & 7;
  const long long nq = static_cast<long long>(p.T) * p.H;
  const bool real = row < nq + p.T;
  const bool is_q = row < nq;
  const long long t = !real ? 0 : (is_q ? row / p.H : row - nq);
  float x[16] = {};
  uint16_t* dst = nullptr;
  if (real) {
    const uint16_t* src;
    if (is_q) {
      const long long h = row - t * p.H;
      src = p.q + t * p.sq_t + h * p.sq_h;
      dst = p.q_rot + row * kD;
    } else {
      src = p.k_ln + t * kD;
      dst = p.k_rot + t * kD;
    }
    load_slice<STYLE, RP, GlobalMem>(reinterpret_cast<const unsigned char*>(src), l, x);
  }
  long long pos = 0;
  const bool pos_ok = position_ok(p, t, pos);
  if constexpr (RP > 0) {
    Rot<RP> r;
    const long long prow = pos_ok ? pos : 0;
    load_f32_global<RP, Slice<0, RP>::ALIGN_CS>(p.cos_t + prow * p.cs_stride + RP * l, r.c);
    load_f32_global<RP, Slice<0, RP>::ALIGN_CS>(p.sin_t + prow * p.cs_stride + RP * l, r.s);
    finish_rot<RP>(r);
    rope_slice<RP>(x, r);
  }
  if (real) store_bf16_slice<STYLE, RP>(dst, l, x);
}

// ---------------------------------------------------------------- launch 3
// Quantise every rotated query row to e4m3 with its ue8m0 scale and fold the
// scale into the gate weight.
__global__ void __launch_bounds__(kThreads) unfused_q_quant_kernel(const UParams p) {
  grid_launch_dependents();
  grid_dependency_wait();
  const long long row = row_of_quarter();
  const int l = threadIdx.x & 7;
  const long long nq = static_cast<long long>(p.T) * p.H;
  const bool real = row < nq;
  const long long t = real ? row / p.H : 0;
  float x[16] = {};
  if (real)
    load_slice<0, 0, GlobalMem>(reinterpret_cast<const unsigned char*>(p.q_rot + row * kD), l, x);
  long long pos = 0;
  const bool pos_ok = position_ok(p, t, pos);
  const int e = ue8m0_exponent(x);
  uint32_t wa[4], wb[4], wp[4];
  quantize_slice<0, 0>(x, e, wa, wb, wp);
  if (real && pos_ok) {
    store_slice<0, 0>(p.q_out + row * kD, l, wa, wb, wp);
    if (l == 0) {
      const long long h = row - t * p.H;
      const float wv = __uint_as_float(static_cast<uint32_t>(__ldg(p.w + t * p.sw_t + h)) << 16);
      __stcs(p.w_out + row, __fmul_rn(__fmul_rn(wv, pow2f(e)), p.fold));
    }
  }
}

// ---------------------------------------------------------------- launch 4
// Quantise every rotated key row and store codes and scale into its slot.
__global__ void __launch_bounds__(kThreads) unfused_k_quant_store_kernel(const UParams p) {
  grid_launch_dependents();
  grid_dependency_wait();
  const long long t = row_of_quarter();
  const int l = threadIdx.x & 7;
  const bool real = t < p.T;
  const long long tt = real ? t : 0;
  float x[16] = {};
  if (real)
    load_slice<0, 0, GlobalMem>(reinterpret_cast<const unsigned char*>(p.k_rot + t * kD), l, x);
  long long pos = 0;
  const bool pos_ok = position_ok(p, tt, pos);
  const long long slot = __ldg(p.loc + tt);
  const int e = ue8m0_exponent(x);
  uint32_t wa[4], wb[4], wp[4];
  quantize_slice<0, 0>(x, e, wa, wb, wp);
  if (!real) return;
  if (!pos_ok) {
    if (l == 0 && p.err) atomicOr(p.err, DSA_DEVERR_POSITION);
    return;
  }
  if (slot < 0 || slot >= p.cg.num_slots) {
    if (l == 0 && p.err) atomicOr(p.err, DSA_DEVERR_SLOT);
    return;
  }
  store_index_k<0, 0>(p.cg, slot, l, wa, wb, wp, e);
}

// ---------------------------------------------------------------- host side

using RopeFn = void (*)(UParams);
template <int STYLE, int RP>
constexpr RopeFn rope_fn() { return unfused_rope_kernel<STYLE, RP>; }
const RopeFn kRope[2][5] = {
    {rope_fn<0, 0>(), rope_fn<0, 1>(), rope_fn<0, 2>(), rope_fn<0, 4>(), rope_fn<0, 8>()},
    {rope_fn<1, 0>(), rope_fn<1, 1>(), rope_fn<1, 2>(), rope_fn<1, 4>(), rope_fn<1, 8>()}};

int rope_index(int rope_dim) {
  switch (rope_dim) {
    case 0: return 0;
    case 16: return 1;
    case 32: return 2;
    case 64: return 3;
    case 128: return 4;
  }
  return -1;
}

bool misaligned(const void* ptr, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

cudaError_t launch_one(void (*fn)(UParams), long long rows, const UParams& p, bool pdl,
                       cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock));
  cfg.blockDim = dim3(kThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace

extern "C" {

size_t dsa_unfused_workspace_bytes(int32_t T, int32_t H) {
  if (T < 0 || H < 1 || H > 4096) return 0;
  const size_t t = static_cast<size_t>(T);
  return 2 * round256(t * kD * 2) + round256(t * static_cast<size_t>(H) * kD * 2);
}

dsa_status dsa_indexer_qk_prepare_store_unfused(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k, int64_t k_stride_t,
    const void* w, int64_t w_stride_t, const int64_t* positions, const int64_t* out_cache_loc,
    const float* cos_cache, const float* sin_cache, int64_t cs_stride, int64_t max_position,
    const float* ln_gamma, const float* ln_beta, float ln_eps, float softmax_scale,
    void* q_fp8_out, float* weights_out, void* index_k_cache, int64_t num_pages,
    int32_t page_size, int32_t T, int32_t H, int32_t head_dim, int32_t rope_dim,
    int32_t rope_style, uint32_t flags, void* workspace, size_t workspace_bytes,
    int32_t* err_flags, void* stream) {
  if (T < 0 || H < 1 || H > 4096) return DSA_ERR_SHAPE;
  if (head_dim != kD || rope_index(rope_dim) < 0) return DSA_ERR_UNSUPPORTED;
  if (rope_style != DSA_ROPE_NEOX && rope_style != DSA_ROPE_GPTJ) return DSA_ERR_UNSUPPORTED;
  if (flags & ~static_cast<uint32_t>(DSA_FLAG_PDL | DSA_FLAG_CACHE_TOKEN_MAJOR))
    return DSA_ERR_UNSUPPORTED;
  if (!(ln_eps >= 0.0f) || !std::isfinite(ln_eps) || !std::isfinite(softmax_scale))
    return DSA_ERR_UNSUPPORTED;
  if (page_size < 1 || num_pages < 1 || max_position < 1) return DSA_ERR_SHAPE;
  if (num_pages > INT64_MAX / (static_cast<int64_t>(page_size) * (kD + 4))) return DSA_ERR_SHAPE;
  if (q_stride_t < 0 || q_stride_h < 0 || k_stride_t < 0 || cs_stride < 0 || w_stride_t < H)
    return DSA_ERR_SHAPE;
  if (T == 0) return DSA_OK;
  if (!q || !k || !w || !positions || !out_cache_loc || !ln_gamma || !ln_beta || !q_fp8_out ||
      !weights_out || !index_k_cache || !workspace)
    return DSA_ERR_NULL;
  if (rope_dim > 0 && (!cos_cache || !sin_cache)) return DSA_ERR_NULL;
  if (rope_dim > 0 && cs_stride < rope_dim / 2) return DSA_ERR_SHAPE;
  if (workspace_bytes < dsa_unfused_workspace_bytes(T, H)) return DSA_ERR_SHAPE;
  if (page_size % 4 != 0 && !(flags & DSA_FLAG_CACHE_TOKEN_MAJOR)) return DSA_ERR_ALIGN;
  if (misaligned(q, 16) || q_stride_t % 8 != 0 || q_stride_h % 8 != 0) return DSA_ERR_ALIGN;
  if (misaligned(k, 16) || k_stride_t % 8 != 0 || misaligned(w, 2)) return DSA_ERR_ALIGN;
  if (misaligned(positions, 8) || misaligned(out_cache_loc, 8)) return DSA_ERR_ALIGN;
  if (misaligned(ln_gamma, 16) || misaligned(ln_beta, 16) || misaligned(index_k_cache, 16))
    return DSA_ERR_ALIGN;
  if (misaligned(q_fp8_out, 16) || misaligned(weights_out, 4) || misaligned(workspace, 256))
    return DSA_ERR_ALIGN;
  if (rope_dim > 0 && (misaligned(cos_cache, 16) || misaligned(sin_cache, 16) ||
                       cs_stride % 4 != 0))
    return DSA_ERR_ALIGN;

  UParams p = {};
  p.q = static_cast<const uint16_t*>(q);
  p.sq_t = q_stride_t;
  p.sq_h = q_stride_h;
  p.k = static_cast<const uint16_t*>(k);
  p.sk_t = k_stride_t;
  p.w = static_cast<const uint16_t*>(w);
  p.sw_t = w_stride_t;
  p.pos = reinterpret_cast<const long long*>(positions);
  p.loc = reinterpret_cast<const long long*>(out_cache_loc);
  p.cos_t = cos_cache;
  p.sin_t = sin_cache;
  p.cs_stride = cs_stride;
  p.max_pos = max_position;
  p.gamma = ln_gamma;
  p.beta = ln_beta;
  p.eps = ln_eps;
  p.fold = static_cast<float>(static_cast<double>(softmax_scale) / std::sqrt(static_cast<double>(H)));
  p.q_out = static_cast<uint8_t*>(q_fp8_out);
  p.w_out = weights_out;
  p.cg.cache = static_cast<uint8_t*>(index_k_cache);
  p.cg.num_slots = num_pages * page_size;
  p.cg.page_bytes = static_cast<long long>(page_size) * (kD + 4);
  p.cg.page_size = page_size;
  p.cg.page_shift = page_shift_of(page_size);
  p.cg.token_major = (flags & DSA_FLAG_CACHE_TOKEN_MAJOR) ? 1 : 0;
  p.T = T;
  p.H = H;
  p.rope_dim = rope_dim;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t kbytes = round256(static_cast<size_t>(T) * kD * 2);
  p.k_ln = reinterpret_cast<uint16_t*>(ws);
  p.k_rot = reinterpret_cast<uint16_t*>(ws + kbytes);
  p.q_rot = reinterpret_cast<uint16_t*>(ws + 2 * kbytes);
  p.err = err_flags;

  const bool pdl = (flags & DSA_FLAG_PDL) != 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long nq = static_cast<long long>(T) * H;
  cudaError_t e = launch_one(unfused_layernorm_kernel, T, p, pdl, s);
  if (e == cudaSuccess) e = launch_one(kRope[rope_style][rope_index(rope_dim)], nq + T, p, pdl, s);
  if (e == cudaSuccess) e = launch_one(unfused_q_quant_kernel, nq, p, pdl, s);
  if (e == cudaSuccess) e = launch_one(unfused_k_quant_store_kernel, T, p, pdl, s);
  return e == cudaSuccess ? DSA_OK : DSA_ERR_LAUNCH;
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation variant
//
// Some callers cannot allocate device memory at the moment they run this
// chain: an engine that hands the whole GPU to its own pool at start-up and
// forbids any other allocation, a plugin host that only passes the plugin
// pointers to its inputs and outputs, or code running where a cudaMalloc
// would synchronise the device or fail (inside a region that is being
// captured, for example).  For them the chain can use a scratch buffer that
// lives inside the library itself: a fixed array in device global memory,
// created when the library's device code is loaded on a GPU and kept until
// the process exits.  Its size caps the call: T * (H + 2) * 256 bytes of
// intermediates must fit in it.

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per GPU

// Device memory; on the host this name is only a stand-in for the symbol, so
// the kernels get the address that cudaGetSymbolAddress returns below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxScratchDevices = 64;
void* g_noalloc_ptr[kMaxScratchDevices] = {};
std::mutex g_noalloc_mu;

// The scratch array's device address on the current device, looked up once
// per device (the first call on a device does it, with that device current).
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

dsa_status dsa_indexer_qk_prepare_store_unfused_noalloc(
    const void* q, int64_t q_stride_t, int64_t q_stride_h, const void* k, int64_t k_stride_t,
    const void* w, int64_t w_stride_t, const int64_t* positions, const int64_t* out_cache_loc,
    const float* cos_cache, const float* sin_cache, int64_t cs_stride, int64_t max_position,
    const float* ln_gamma, const float* ln_beta, float ln_eps, float softmax_scale,
    void* q_fp8_out, float* weights_out, void* index_k_cache, int64_t num_pages,
    int32_t page_size, int32_t T, int32_t H, int32_t head_dim, int32_t rope_dim,
    int32_t rope_style, uint32_t flags, int32_t* err_flags, void* stream) {
  const size_t need = dsa_unfused_workspace_bytes(T, H);
  if (T > 0 && need > kNoAllocScratchBytes) return DSA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  if (T > 0 && need > 0 && noalloc_scratch(&scratch) != cudaSuccess) return DSA_ERR_LAUNCH;
  // Every intermediate the chain reads was written earlier in the same call,
  // so the buffer's previous contents never matter and nothing is cleared.
  return dsa_indexer_qk_prepare_store_unfused(
      q, q_stride_t, q_stride_h, k, k_stride_t, w, w_stride_t, positions, out_cache_loc,
      cos_cache, sin_cache, cs_stride, max_position, ln_gamma, ln_beta, ln_eps, softmax_scale,
      q_fp8_out, weights_out, index_k_cache, num_pages, page_size, T, H, head_dim, rope_dim,
      rope_style, flags, scratch, kNoAllocScratchBytes, err_flags, stream);
}

}  // extern "C"
