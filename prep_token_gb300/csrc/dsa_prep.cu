// DSA indexer Q/K prepare-and-store for GB300 (sm_103a): launcher and the C
// ABI declared in include/dsa_prep.h.  The kernels and their lane layouts
// are described in dsa_prep_kernels.cuh.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "dsa_prep_kernels.cuh"

namespace {

using namespace dsa_dev;
using namespace dsa_prep_impl;

// ---------------------------------------------------------------- host side

bool misaligned(const void* ptr, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
}

// rope_dim / 16 in {0, 1, 2, 4, 8} -> table index
int rp_index(int rope_dim) {
  switch (rope_dim) {
    case 0: return 0;
    case 16: return 1;
    case 32: return 2;
    case 64: return 3;
    case 128: return 4;
  }
  return -1;
}

const KernelFn kPipeline[2][5] = {
    {pipeline_fn<false, 0, 0>(), pipeline_fn<false, 0, 1>(), pipeline_fn<false, 0, 2>(),
     pipeline_fn<false, 0, 4>(), pipeline_fn<false, 0, 8>()},
    {pipeline_fn<false, 1, 0>(), pipeline_fn<false, 1, 1>(), pipeline_fn<false, 1, 2>(),
     pipeline_fn<false, 1, 4>(), pipeline_fn<false, 1, 8>()}};
const KernelFn kPipelineMulti[2][5] = {
    {pipeline_fn<false, 0, 0, true>(), pipeline_fn<false, 0, 1, true>(), pipeline_fn<false, 0, 2, true>(),
     pipeline_fn<false, 0, 4, true>(), pipeline_fn<false, 0, 8, true>()},
    {pipeline_fn<false, 1, 0, true>(), pipeline_fn<false, 1, 1, true>(), pipeline_fn<false, 1, 2, true>(),
     pipeline_fn<false, 1, 4, true>(), pipeline_fn<false, 1, 8, true>()}};
const KernelFn kDirect[2][5] = {
    {direct_fn<false, 0, 0>(), direct_fn<false, 0, 1>(), direct_fn<false, 0, 2>(),
     direct_fn<false, 0, 4>(), direct_fn<false, 0, 8>()},
    {direct_fn<false, 1, 0>(), direct_fn<false, 1, 1>(), direct_fn<false, 1, 2>(),
     direct_fn<false, 1, 4>(), direct_fn<false, 1, 8>()}};

const KernelFn kStream[2][5] = {
    {kstream_fn<false, 0, 0>(), kstream_fn<false, 0, 1>(), kstream_fn<false, 0, 2>(),
     kstream_fn<false, 0, 4>(), kstream_fn<false, 0, 8>()},
    {kstream_fn<false, 1, 0>(), kstream_fn<false, 1, 1>(), kstream_fn<false, 1, 2>(),
     kstream_fn<false, 1, 4>(), kstream_fn<false, 1, 8>()}};

// dynamic shared memory of the k-stream kernels, by rope_dim / 16 index
const int kStreamSmem[5] = {kstream_smem<0>(), kstream_smem<1>(), kstream_smem<2>(),
                            kstream_smem<4>(), kstream_smem<8>()};

int max_pipeline_smem() { return kBarrierBytes + kStages * kMaxStageBytes; }

// Per-device facts looked up once: the SM count, and whether the pipeline
// kernels' dynamic shared-memory limit has been raised on that device.
struct DeviceInfo {
  int sms = 0;
  int smem_per_sm = 0;  // shared memory of one SM, bytes
  bool ready = false;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

cudaError_t device_info(int* sms, int* smem_per_sm = nullptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return e;
    for (int s = 0; s < 2; ++s)
      for (int r = 0; r < 5; ++r) {
        for (const KernelFn fn : {kPipeline[s][r], kPipelineHad[s][r], kPipelineMulti[s][r],
                                  kPipelineMultiHad[s][r]}) {
          e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   max_pipeline_smem());
          if (e != cudaSuccess) return e;
        }
        for (const KernelFn fn : {kStream[s][r], kStreamHad[s][r]}) {
          e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kStreamSmem[r]);
          if (e != cudaSuccess) return e;
        }
      }
    d.ready = true;
  }
  *sms = d.sms;
  if (smem_per_sm) *smem_per_sm = d.smem_per_sm;
  return cudaSuccess;
}

// Calls up to this many query vectors (T * H) take the direct kernel.
constexpr long long kDirectMaxVectors = 16384;
// k-only calls with more keys than this take the k-stream kernel.
constexpr long long kStreamMinKeys = 8192;

// Pipeline units.  With few heads (H <= 32) and tokens enough to fill the
// machine, a unit is 2 (H <= 32) or 4 (H <= 16) whole tokens, so a unit
// still carries up to 64 query rows: one bulk copy when the rows are
// contiguous, and all eight consumer warps busy (8 / TPU per token).  Otherwise a unit is one
// token: all its heads (up to 64) when there are tokens enough, else heads
// split into chunks of >= 8 until the units cover the SMs.  Chunks hold a
// multiple of 8 heads when H >= 8, so each chunk's weights start on a 16-byte
// boundary and can ride the bulk copies.
void choose_units(Params& p, int sms, bool w_rows_aligned) {
  p.TPU = 1;
  if (p.H == 0) {
    p.HC = 0;
    p.NC = 1;
  } else {
    if (p.H <= 32) {
      const int tpu = p.H <= 16 ? 4 : 2;  // 64 / H tokens, rounded down to 1, 2 or 4
      if (static_cast<long long>(p.T) >= static_cast<long long>(tpu) * 2 * kPipeCtas * sms) p.TPU = tpu;
    }
    if (p.TPU > 1) {
      p.HC = p.H;
      p.NC = 1;
    } else {
      int nc = (p.H + kHCMax - 1) / kHCMax;
      const long long target = 3LL * sms;
      while (static_cast<long long>(p.T) * nc * 2 <= target && (p.H + 2 * nc - 1) / (2 * nc) >= 8)
        nc *= 2;
      int hc = (p.H + nc - 1) / nc;
      if (hc > 8) hc = (hc + 7) / 8 * 8;
      p.HC = hc;
      p.NC = (p.H + hc - 1) / hc;
    }
  }
  p.tpu_shift = p.TPU == 4 ? 2 : p.TPU == 2 ? 1 : 0;
  // fused k|w rows (w = k + 128 elements, one stride, rows of at most 512 B):
  // one copy per unit brings keys and weights
  const long long kw_row_b = 2 * p.sk_t;
  p.kw_fused = (p.TPU > 1 && p.w == p.k + kD && p.sw_t == p.sk_t && kw_row_b % 16 == 0 &&
                kw_row_b <= 512 && p.H % 8 == 0 && w_rows_aligned) ? 1 : 0;
  p.kw_row_b = p.kw_fused ? static_cast<int>(kw_row_b) : 256;
  p.cs_contig = (p.cs_stride == p.rope_dim / 2) ? 1 : 0;
  p.units = (static_cast<long long>(p.T) + p.TPU - 1) / p.TPU * p.NC;
  p.w_bulk = (w_rows_aligned && p.H % 8 == 0 && p.HC % 8 == 0) ? 1 : 0;
  // stage layout: headers (32 B a token), key rows, cos rows, sin rows,
  // weights, query rows (from a 128-byte boundary); one-token units keep
  // the fixed layout kOff*
  if (p.TPU == 1) {  // the fixed layout of one-token units
    p.off_k = kOffK;
    p.off_cos = kOffCos;
    p.off_sin = kOffSin;
    p.off_w = kOffW;
    p.off_q = kOffQ;
  } else {
    p.off_k = 32 * p.TPU;
    p.off_cos = p.off_k + p.kw_row_b * p.TPU;
    p.off_sin = p.off_cos + p.cs_bytes * p.TPU;
    p.off_w = p.off_sin + p.cs_bytes * p.TPU;
    p.off_q = (p.off_w + 2 * p.HC * p.TPU + 127) / 128 * 128;
  }
  p.stage_bytes = p.off_q + 256 * p.HC * p.TPU;
}

cudaError_t launch(Params& p, int rope_style, uint32_t flags, bool w_rows_aligned,
                   cudaStream_t stream) {
  int sms = 0, smem_per_sm = 0;
  cudaError_t e = device_info(&sms, &smem_per_sm);
  if (e != cudaSuccess) return e;
  const int ri = rp_index(p.rope_dim);
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (flags & DSA_FLAG_PDL) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  p.early_rope = (flags & DSA_FLAG_PDL_EARLY_ROPE) ? 1 : 0;
  p.test_withhold = (flags & DSA_FLAG_TEST_WITHHOLD_UNIT) ? 1 : 0;
  p.cg.token_major = (flags & DSA_FLAG_CACHE_TOKEN_MAJOR) ? 1 : 0;
  const bool had = (flags & DSA_FLAG_HADAMARD) != 0;
  if (p.H == 0) {
    // k-only: the direct kernel up to kStreamMinKeys keys (least latency),
    // the k-stream kernel above (DSA_FLAG_PIPELINE forces it).
    const bool stream_k =
        !(flags & DSA_FLAG_DIRECT) && ((flags & DSA_FLAG_PIPELINE) || p.T > kStreamMinKeys);
    if (stream_k) {
      const long long steps = (static_cast<long long>(p.T) + kStreamKeys - 1) / kStreamKeys;
      // as many CTAs as are resident at once (one per SM at rope_dim 128,
      // whose ring takes more than half of an SM's shared memory)
      int per_sm = kStreamCtas;
      while (per_sm > 1 && per_sm * (kStreamSmem[ri] + 1024) > smem_per_sm) --per_sm;
      long long blocks = static_cast<long long>(sms) * per_sm;
      const long long need = (steps + kStreamWarps - 1) / kStreamWarps;
      if (blocks > need) blocks = need;
      cfg.gridDim = dim3(static_cast<unsigned>(blocks));
      cfg.blockDim = dim3(kStreamThreads);
      cfg.dynamicSmemBytes = static_cast<size_t>(kStreamSmem[ri]);
      return cudaLaunchKernelEx(&cfg, had ? kStreamHad[rope_style][ri] : kStream[rope_style][ri], p);
    }
  }
  const long long vecs = static_cast<long long>(p.T) * p.H;
  bool direct = p.H == 0 || vecs <= kDirectMaxVectors;
  if (flags & DSA_FLAG_PIPELINE) direct = false;
  if (flags & DSA_FLAG_DIRECT) direct = true;
  if (direct) {
    p.NQ = (p.H + 3) / 4;
    p.q_warps = static_cast<long long>(p.T) * p.NQ;
    p.k_warps = (static_cast<long long>(p.T) + 3) / 4;
    const long long warps = p.q_warps + p.k_warps;
    // L2 hints before the PDL wait, in a launch of at most one wave
    p.l2_hints = (flags & DSA_FLAG_PDL) && warps <= static_cast<long long>(sms) * kDirectWarps;
    // Spread the warps over the SMs: as few per CTA as fill them once (a
    // small call gets one warp per SM, so no two warps share an SM's issue
    // slots), at most kDirectWarps.
    long long wpc = (warps + sms - 1) / sms;
    if (wpc < 1) wpc = 1;
    if (wpc > kDirectWarps) wpc = kDirectWarps;
    cfg.gridDim = dim3(static_cast<unsigned>((warps + wpc - 1) / wpc));
    cfg.blockDim = dim3(static_cast<unsigned>(32 * wpc));
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, had ? kDirectHad[rope_style][ri] : kDirect[rope_style][ri], p);
  }
  choose_units(p, sms, w_rows_aligned);
  // one wave of persistent CTAs: as many as are resident at once (the
  // kernel's register budget, or fewer if the ring's shared memory says so)
  const int smem = kBarrierBytes + kStages * p.stage_bytes;
  int per_sm = had ? kPipeCtasHad : kPipeCtas;
  while (per_sm > 1 && per_sm * (smem + 1024) > smem_per_sm) --per_sm;
  long long blocks = static_cast<long long>(sms) * per_sm;
  if (blocks > p.units) blocks = p.units;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kPipeThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  const KernelFn fn = p.TPU > 1 ? (had ? kPipelineMultiHad : kPipelineMulti)[rope_style][ri]
                                 : (had ? kPipelineHad : kPipeline)[rope_style][ri];
  return cudaLaunchKernelEx(&cfg, fn, p);
}

dsa_status check_k_side(const void* k, int64_t k_stride_t, const int64_t* positions,
                        const int64_t* out_cache_loc, const float* cos_cache,
                        const float* sin_cache, int64_t cs_stride, int64_t max_position,
                        const float* ln_gamma, const float* ln_beta, float ln_eps,
                        const void* index_k_cache, int64_t num_pages, int32_t page_size,
                        int32_t T, int32_t head_dim, int32_t rope_dim, int32_t rope_style,
                        uint32_t flags) {
  if (T < 0) return DSA_ERR_SHAPE;
  if (head_dim != kD) return DSA_ERR_UNSUPPORTED;
  if (rp_index(rope_dim) < 0) return DSA_ERR_UNSUPPORTED;
  if (rope_style != DSA_ROPE_NEOX && rope_style != DSA_ROPE_GPTJ) return DSA_ERR_UNSUPPORTED;
  if (flags & ~static_cast<uint32_t>(DSA_FLAG_PDL | DSA_FLAG_PIPELINE | DSA_FLAG_DIRECT |
                                     DSA_FLAG_PDL_EARLY_ROPE | DSA_FLAG_CACHE_TOKEN_MAJOR |
                                     DSA_FLAG_HADAMARD | DSA_FLAG_TEST_WITHHOLD_UNIT))
    return DSA_ERR_UNSUPPORTED;
  if ((flags & DSA_FLAG_TEST_WITHHOLD_UNIT) && !(flags & DSA_FLAG_PIPELINE))
    return DSA_ERR_UNSUPPORTED;
  if ((flags & DSA_FLAG_PDL_EARLY_ROPE) && !(flags & DSA_FLAG_PDL)) return DSA_ERR_UNSUPPORTED;
  if ((flags & DSA_FLAG_PIPELINE) && (flags & DSA_FLAG_DIRECT)) return DSA_ERR_UNSUPPORTED;
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
  if (page_size % 4 != 0 && !(flags & DSA_FLAG_CACHE_TOKEN_MAJOR)) return DSA_ERR_ALIGN;
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
  p.pos = reinterpret_cast<const long long*>(positions);
  p.loc = reinterpret_cast<const long long*>(out_cache_loc);
  p.cos_t = cos_cache;
  p.sin_t = sin_cache;
  p.cs_stride = cs_stride;
  p.max_pos = max_position;
  p.gamma = ln_gamma;
  p.beta = ln_beta;
  p.eps = ln_eps;
  p.cg.cache = static_cast<uint8_t*>(index_k_cache);
  p.cg.num_slots = num_pages * page_size;
  p.cg.page_size = page_size;
  p.cg.page_shift = page_shift_of(page_size);
  p.cg.page_bytes = static_cast<long long>(page_size) * (kD + 4);
  p.T = T;
  p.rope_dim = rope_dim;
  p.cs_bytes = rope_dim * 2;
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
    int32_t rope_style, uint32_t flags, int32_t* err_flags, void* stream) {
  dsa_status st = check_k_side(k, k_stride_t, positions, out_cache_loc, cos_cache, sin_cache,
                               cs_stride, max_position, ln_gamma, ln_beta, ln_eps,
                               index_k_cache, num_pages, page_size, T, head_dim, rope_dim,
                               rope_style, flags);
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
  p.q = static_cast<const uint16_t*>(q);
  p.sq_t = q_stride_t;
  p.sq_h = q_stride_h;
  p.w = static_cast<const uint16_t*>(w);
  p.sw_t = w_stride_t;
  p.fold = static_cast<float>(static_cast<double>(softmax_scale) / std::sqrt(static_cast<double>(H)));
  p.q_out = static_cast<uint8_t*>(q_fp8_out);
  p.w_out = weights_out;
  p.H = H;
  const bool w_rows_aligned = !misaligned(w, 16) && w_stride_t % 8 == 0;
  cudaError_t e = launch(p, rope_style, flags, w_rows_aligned, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_LAUNCH;
}

dsa_status dsa_indexer_k_prepare_store(
    const void* k, int64_t k_stride_t, const int64_t* positions, const int64_t* out_cache_loc,
    const float* cos_cache, const float* sin_cache, int64_t cs_stride, int64_t max_position,
    const float* ln_gamma, const float* ln_beta, float ln_eps, void* index_k_cache,
    int64_t num_pages, int32_t page_size, int32_t T, int32_t head_dim, int32_t rope_dim,
    int32_t rope_style, uint32_t flags, int32_t* err_flags, void* stream) {
  dsa_status st = check_k_side(k, k_stride_t, positions, out_cache_loc, cos_cache, sin_cache,
                               cs_stride, max_position, ln_gamma, ln_beta, ln_eps,
                               index_k_cache, num_pages, page_size, T, head_dim, rope_dim,
                               rope_style, flags);
  if (st != DSA_OK || T == 0) return st;
  if (flags & DSA_FLAG_TEST_WITHHOLD_UNIT) return DSA_ERR_UNSUPPORTED;  // no producer warp here
  Params p = {};
  fill_k_side(p, k, k_stride_t, positions, out_cache_loc, cos_cache, sin_cache, cs_stride,
              max_position, ln_gamma, ln_beta, ln_eps, index_k_cache, num_pages, page_size, T,
              rope_dim, err_flags);
  p.H = 0;
  cudaError_t e = launch(p, rope_style, flags, false, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DSA_OK : DSA_ERR_LAUNCH;
}

const char* dsa_status_string(dsa_status status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_NULL: return "a required pointer is NULL";
    case DSA_ERR_ALIGN: return "a pointer or stride breaks an alignment rule";
    case DSA_ERR_SHAPE: return "a negative or inconsistent size or stride";
    case DSA_ERR_UNSUPPORTED: return "unsupported head_dim, rope_dim, rope_style, flag or scalar";
    case DSA_ERR_LAUNCH: return "the CUDA kernel launch failed";
    case DSA_ERR_SCRATCH_LIMIT:
      return "the call needs more scratch than the library's built-in 32 MiB buffer";
  }
  return "unknown status";
}

int32_t dsa_prep_version(void) { return (3 << 16) | 1; }

}  // extern "C"
