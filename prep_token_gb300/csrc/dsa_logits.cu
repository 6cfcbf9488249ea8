// fp8 paged MQA logits -- the indexer kernel that consumes this path's
// outputs (q_fp8, folded gate weights, the page-blocked index-K cache) -- on
// the 5th-generation tensor cores.  The vllm PR "[ROCm][Perf] Enable fused
// indexer-Q RoPE+quant kernel for DeepSeek/GLM sparse attention" lists it
// (Kernel-level evidence) right after the index-K store; its formula follows
// the DeepSeek sparse-attention indexer:
//   logits[t, j] = k_scale[j] * sum_h weights[t, h] * max(q[t, h] . k[j], 0),
// j < context_lens[t]; -inf up to max_context after that.
//
// One CTA works on one query token t and a strided set of 128-key tiles
// (two 64-key pages each).  Per tile:
//   * warp 0 (one lane) issues two 3-D TMA loads (128B swizzle) of the pages'
//     code blocks straight from the paged cache into a 4-stage ring, and a
//     bulk copy of each page's 256-byte scale block beside them;
//   * warp 1 (one lane) issues four tcgen05.mma.kind::f8f6f4 (M = 128 keys,
//     N = H heads, K = 32 each) into one of two TMEM accumulators, and commits
//     them to the "stage free" and "accumulator full" mbarriers;
//   * warps 2..5 read their 32 TMEM lanes (one key per thread, H fp32 per key)
//     with tcgen05.ld, release the accumulator, and reduce over heads with
//     ReLU and the gate weights, times the key's scale (from shared memory;
//     the stage is refilled only after all four warps have read it).
// Every wait is bounded in time; TMEM is always released before exit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "dsa_common.cuh"
#include "dsa_prep.h"

namespace {

using namespace dsa_dev;

constexpr int kTileKeys = 128;                  // MMA M: keys per tile
constexpr int kPageKeys = 64;                   // keys per cache page
constexpr int kKStages = 4;                     // key-tile ring depth
constexpr int kBatch = 8;                       // block-table entries fetched ahead, in tiles
constexpr int kLThreads = 6 * 32;               // producer, MMA, 4 epilogue warps
constexpr int kTileBytes = kTileKeys * kD;      // 16 KiB of e4m3 codes
constexpr int kPageBytes = kPageKeys * kD;      // 8 KiB
constexpr int kPageStride = kPageKeys * (kD + 4);  // bytes per cache page

struct LParams {
  const float* weights;
  const uint8_t* cache;
  long long num_pages;
  const int* block_table;
  long long bt_stride;
  const int* context_lens;
  float* logits;
  long long logits_stride;
  int max_context;
  int tiles_max;  // ceil(max_context / 128)
  int T;
  int early_index;  // read context_lens / block_table before the PDL wait
                    // (also every launch without PDL: nothing runs before it)
  int* err;
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major tile whose rows are 128 bytes,
// written by TMA with the 128-byte swizzle: 8-row groups of 1024 bytes
// (stride-dimension offset), leading offset unused, descriptor version 1,
// layout SWIZZLE_128B.  Stepping K by 32 bytes adds 2 to the address field.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t smem_addr) {
  uint64_t d = static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;    // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;            // version
  d |= static_cast<uint64_t>(2) << 61;            // 128-byte swizzle
  return d;
}

// Instruction descriptor: D fp32, A and B e4m3, both K-major, M x N.
__host__ __device__ constexpr uint32_t mma_idesc(int m, int n) {
  return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- the kernel

template <int NH>
struct LSmem {
  static constexpr int kQBytes = NH * kD;                       // B operand
  static constexpr int kOffQ = 0;                               // 1024-aligned
  static constexpr int kOffK = ((kQBytes + 1023) / 1024) * 1024;  // A stages
  static constexpr int kOffS = kOffK + kKStages * kTileBytes;    // key scales, 128 per stage
  static constexpr int kOffW = kOffS + kKStages * kTileKeys * 4;  // weights[NH]
  static constexpr int kOffBar = kOffW + NH * 4;
  // barriers: full[S], empty[S], qfull, accfull[2], accempty[2], drain
  static constexpr int kBars = 2 * kKStages + 6;
  static constexpr int kOffTmem = kOffBar + 8 * kBars;
  static constexpr int kOffAbort = kOffTmem + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kTmemCols = 2 * NH < 32 ? 32 : 2 * NH;   // two accumulators
};

template <int NH>
__global__ void __launch_bounds__(kLThreads, 1)
    dsa_mqa_logits_kernel(const __grid_constant__ CUtensorMap tq,
                          const __grid_constant__ CUtensorMap tk, const LParams p) {
  using L = LSmem<NH>;
  extern __shared__ __align__(1024) unsigned char smem[];
  // The 128-byte-swizzled tiles need a 1024-byte aligned base.  The dynamic
  // shared window of a kernel without static shared memory starts on such a
  // boundary; should it ever not, report it and leave before taking anything.
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0 && p.err) atomicOr(p.err, DSA_DEVERR_INTERNAL);
    return;
  }
  const uint32_t bar0 = sbase + L::kOffBar;
  auto full = [&](int s) { return bar0 + 8 * s; };
  auto empty = [&](int s) { return bar0 + 8 * (kKStages + s); };
  const uint32_t qfull = bar0 + 8 * (2 * kKStages);
  auto accfull = [&](int b) { return bar0 + 8 * (2 * kKStages + 1 + b); };
  auto accempty = [&](int b) { return bar0 + 8 * (2 * kKStages + 3 + b); };
  const uint32_t drain = bar0 + 8 * (2 * kKStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);
  float* wsm = reinterpret_cast<float*>(smem + L::kOffW);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.y;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1 + 4);  // the MMA commit and the four epilogue warps
    }
    mbar_init(qfull, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(accfull(b), 1);
      mbar_init(accempty(b), 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {  // whole warp: allocate the two accumulators
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(sbase + L::kOffTmem), "r"(L::kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kOffTmem);

  // Page indices come from the block table a batch of kBatch tiles at a
  // time (the producer keeps the next batch's loads in flight while it
  // issues this one), so the table's latency is not paid per tile.
  const int* bt = p.block_table + t * p.bt_stride;
  const int step = static_cast<int>(gridDim.x);
  auto load_batch = [&](int i0, int ntiles, int len, int (&pg)[2 * kBatch]) {
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = i0 + k * step;
      pg[2 * k] = i < ntiles ? __ldg(bt + 2 * i) : 0;
      pg[2 * k + 1] = (i < ntiles && (2 * i + 1) * kPageKeys < len) ? __ldg(bt + 2 * i + 1) : 0;
    }
  };
  auto tiles_of = [](int len) { return len > 0 ? (len + kTileKeys - 1) / kTileKeys : 0; };
  // keys past max_context have no column: the context is clamped to it
  auto context_of = [&](int t) { return max(0, min(__ldg(p.context_lens + t), p.max_context)); };
  int cur[2 * kBatch];
  int len = 0;
  if (p.early_index) {
    // DSA_FLAG_PDL_EARLY_INDEX (or no PDL): the context length and the block
    // table are not written by the previous kernel.  The first batch of the
    // table is read without waiting for the length (bounded by max_context,
    // which the table covers), and the producer starts its first pages on
    // their way into L2 (a hint, coherent with any write the previous kernel
    // makes to them) while that kernel finishes.
    if (warp == 0 && lane == 0)
      load_batch(static_cast<int>(blockIdx.x), p.tiles_max, p.max_context, cur);
    len = context_of(t);
    if (warp == 0 && lane == 0) {
      const int nt = tiles_of(len);
#pragma unroll
      for (int k = 0; k < kKStages; ++k) {
        const int i = static_cast<int>(blockIdx.x) + k * step;
        if (i < nt) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const long long pg = cur[2 * k + h];
            if ((h == 0 || (2 * i + 1) * kPageKeys < len) && pg >= 0 && pg < p.num_pages)
              prefetch_l2_bulk(p.cache + pg * kPageStride, kPageStride);
          }
        }
      }
    }
  }

  grid_dependency_wait();
  grid_launch_dependents();

  // The query tile does not depend on the context length: its copy goes out
  // first, overlapping the length's read (every CTA waits for it before exit).
  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(qfull, L::kQBytes);
    tma_load_2d(sbase + L::kOffQ, &tq, 0, t * NH, qfull);
  }
  if (!p.early_index) len = context_of(t);
  const int ntiles = tiles_of(len);

  if (warp == 0) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      int m = 0;
      bool ok = true;
      int nxt[2 * kBatch];
      if (!p.early_index) load_batch(static_cast<int>(blockIdx.x), ntiles, len, cur);
      for (int i0 = blockIdx.x; ok && i0 < ntiles; i0 += kBatch * step) {
        load_batch(i0 + kBatch * step, ntiles, len, nxt);
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int i = i0 + k * step;
          if (!ok || i >= ntiles) break;
          const int s = m % kKStages;
          if (m >= kKStages && !mbar_wait(empty(s), ((m / kKStages) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const bool has1 = (2 * i + 1) * kPageKeys < len;
          const uint32_t dst = sbase + L::kOffK + s * kTileBytes;
          const uint32_t sdst = sbase + L::kOffS + s * kTileKeys * 4;
          // A page outside [0, num_pages) sets the error bit; its keys' logits
          // are NaN, as the oracle defines them: the MMA still takes page 0's
          // codes, but the stage gets NaN scales, stored before the arrival
          // below publishes them, instead of a copy.
          const long long pg0 = cur[2 * k], pg1 = cur[2 * k + 1];
          const bool bad0 = pg0 < 0 || pg0 >= p.num_pages;
          const bool bad1 = has1 && (pg1 < 0 || pg1 >= p.num_pages);
          if (bad0 || bad1) {
            if (p.err) atomicOr(p.err, DSA_DEVERR_SLOT);
            for (int h = 0; h < 2; ++h)
              if (h == 0 ? bad0 : bad1)
                for (int q = 0; q < kPageKeys; q += 4)
                  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};"
                               ::"r"(sdst + 4 * (h * kPageKeys + q)), "r"(0x7fc00000) : "memory");
          }
          const int scales = (bad0 ? 0 : 1) + (has1 && !bad1 ? 1 : 0);
          mbar_arrive_expect_tx(full(s), (has1 ? 2 : 1) * kPageBytes + scales * kPageKeys * 4);
          auto load_page = [&](int h, long long pg, bool bad) {
            tma_load_3d(dst + h * kPageBytes, &tk, 0, 0, bad ? 0 : static_cast<int>(pg), full(s));
            if (!bad)
              bulk_g2s(sdst + h * kPageKeys * 4, p.cache + pg * kPageStride + kPageBytes,
                       kPageKeys * 4, full(s));
          };
          load_page(0, pg0, bad0);
          if (has1) load_page(1, pg1, bad1);
          ++m;
        }
#pragma unroll
        for (int k = 0; k < 2 * kBatch; ++k) cur[k] = nxt[k];
      }
      if (!ok) {
        *abort_flag = 1;
        if (p.err) atomicOr(p.err, DSA_DEVERR_TIMEOUT);
      }
      // stay until every load issued has landed
      volatile int never = 0;
      for (int d = (m > kKStages ? m - kKStages : 0); d < m; ++d)
        mbar_wait(full(d % kKStages), (d / kKStages) & 1, &never);
      mbar_wait(qfull, 0, &never);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = mma_idesc(kTileKeys, NH);
      const uint64_t bdesc = sw128_desc(sbase + L::kOffQ);
      bool ok = ntiles <= static_cast<int>(blockIdx.x) || mbar_wait(qfull, 0, abort_flag);
      int m = 0;
      for (int i = blockIdx.x; ok && i < ntiles; i += gridDim.x, ++m) {
        const int s = m % kKStages;
        const int b = m & 1;
        if (!mbar_wait(full(s), (m / kKStages) & 1, abort_flag)) {
          ok = false;
          break;
        }
        if (m >= 2 && !mbar_wait(accempty(b), ((m >> 1) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t adesc = sw128_desc(sbase + L::kOffK + s * kTileBytes);
        const uint32_t d = tmem + static_cast<uint32_t>(b * NH);
#pragma unroll
        for (int k = 0; k < kD / 32; ++k)
          mma_f8(d, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0 ? 1u : 0u);
        mma_commit(empty(s));
        mma_commit(accfull(b));
      }
      if (!ok) {
        *abort_flag = 1;
        if (p.err) atomicOr(p.err, DSA_DEVERR_TIMEOUT);
        // every MMA issued must finish before TMEM is released
        mma_commit(drain);
        volatile int never = 0;
        mbar_wait(drain, 0, &never);
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2..5)
    const int e = threadIdx.x - 64;
    for (int h = e; h < NH; h += 128) wsm[h] = __ldg(p.weights + static_cast<long long>(t) * NH + h);
    named_barrier(1, 128);
    const int sub = warp & 3;               // the TMEM lanes this warp may read
    const int row = 32 * sub + lane;        // key within the tile
    float* out = p.logits + static_cast<long long>(t) * p.logits_stride;
    const float* ssm = reinterpret_cast<const float*>(smem + L::kOffS);
    int m = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < p.tiles_max; i += gridDim.x) {
      const int j = i * kTileKeys + row;
      if (i < ntiles && ok) {
        const int b = m & 1;
        const int s = m % kKStages;
        // the stage's scale block landed with its codes; the stage cannot be
        // refilled before this warp arrives on its "empty" barrier below
        const bool got = mbar_wait(accfull(b), (m >> 1) & 1, abort_flag) &&
                         mbar_wait(full(s), (m / kKStages) & 1, abort_flag);
        if (!__all_sync(kFull, got)) {
          ok = false;
          if (lane == 0) {
            *abort_flag = 1;
            if (p.err) atomicOr(p.err, DSA_DEVERR_TIMEOUT);
          }
          continue;
        }
        tc_fence_after();
        const float ks = ssm[s * kTileKeys + row];
        __syncwarp();
        if (lane == 0) mbar_arrive(empty(s));
        float acc = 0.0f;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * sub) << 16) +
                               static_cast<uint32_t>(b * NH);
#pragma unroll
        for (int c = 0; c < NH / 16; ++c) {
          float v[16];
          tmem_ld16(taddr + 16 * c, v);
#pragma unroll
          for (int q = 0; q < 16; ++q) acc = __fmaf_rn(wsm[16 * c + q], fmaxf(v[q], 0.0f), acc);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(accempty(b));
        ++m;
        if (j < p.max_context) out[j] = j < len ? __fmul_rn(acc, ks) : -INFINITY;
      } else if (j < p.max_context) {
        out[j] = j < len ? __int_as_float(0x7fc00000) : -INFINITY;  // NaN only on abort
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 ::"r"(tmem), "r"(L::kTmemCols) : "memory");
}

// ---------------------------------------------------------------- host side

bool misaligned(const void* ptr, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

using LogitsFn = void (*)(CUtensorMap, CUtensorMap, LParams);

struct LDevice {
  int sms = 0;
  int occ[4] = {1, 1, 1, 1};  // resident CTAs per SM for H = 16, 32, 64, 128
  bool ready = false;
};
constexpr int kMaxLDevices = 64;
LDevice g_ldev[kMaxLDevices];
std::mutex g_ldev_mu;

// Resident CTAs per SM, from the limits that bind here: shared memory (with
// the per-block reservation), registers and threads.
template <int NH>
cudaError_t prepare_kernel(int dev, int* occ) {
  const int smem = LSmem<NH>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(dsa_mqa_logits_kernel<NH>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(dsa_mqa_logits_kernel<NH>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  cudaFuncAttributes fa;
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, dsa_mqa_logits_kernel<NH>);
  int sm_smem = 0, reserved = 0, sm_regs = 0, sm_threads = 0;
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_regs, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&sm_threads, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
  if (e != cudaSuccess) return e;
  int n = sm_smem / (smem + reserved);
  const int by_regs = sm_regs / (kLThreads * (fa.numRegs > 0 ? fa.numRegs : 1));
  const int by_threads = sm_threads / kLThreads;
  if (by_regs < n) n = by_regs;
  if (by_threads < n) n = by_threads;
  *occ = n < 1 ? 1 : n;
  return cudaSuccess;
}

cudaError_t logits_device(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxLDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_ldev_mu);
  LDevice& d = g_ldev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = prepare_kernel<16>(dev, &d.occ[0]);
    if (e == cudaSuccess) e = prepare_kernel<32>(dev, &d.occ[1]);
    if (e == cudaSuccess) e = prepare_kernel<64>(dev, &d.occ[2]);
    if (e == cudaSuccess) e = prepare_kernel<128>(dev, &d.occ[3]);
    if (e != cudaSuccess) return e;
    d.ready = true;
  }
  *sms = d.sms;
  return cudaSuccess;
}

int resident_ctas(int H) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxLDevices) return 1;
  const int i = H == 16 ? 0 : H == 32 ? 1 : H == 64 ? 2 : 3;
  return g_ldev[dev].sms * g_ldev[dev].occ[i];
}

template <int NH>
cudaError_t launch_logits(const CUtensorMap& tq, const CUtensorMap& tk, const LParams& p,
                          dim3 grid, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kLThreads);
  cfg.dynamicSmemBytes = LSmem<NH>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, dsa_mqa_logits_kernel<NH>, tq, tk, p);
}

}  // namespace

extern "C" {

dsa_status dsa_indexer_mqa_logits(const void* q_fp8, const float* weights,
                                  const void* index_k_cache, int64_t num_pages,
                                  int32_t page_size, const int32_t* block_table,
                                  int64_t bt_stride, const int32_t* context_lens,
                                  float* logits, int64_t logits_stride, int32_t max_context,
                                  int32_t T, int32_t H, uint32_t flags, int32_t* err_flags,
                                  void* stream) {
  if (T < 0 || T > 65535 || max_context < 0 || num_pages < 1 || bt_stride < 0)
    return DSA_ERR_SHAPE;
  if (H != 16 && H != 32 && H != 64 && H != 128) return DSA_ERR_UNSUPPORTED;
  if (page_size != kPageKeys) return DSA_ERR_UNSUPPORTED;
  if (flags & ~static_cast<uint32_t>(DSA_FLAG_PDL | DSA_FLAG_PDL_EARLY_INDEX))
    return DSA_ERR_UNSUPPORTED;
  if ((flags & DSA_FLAG_PDL_EARLY_INDEX) && !(flags & DSA_FLAG_PDL)) return DSA_ERR_UNSUPPORTED;
  if (num_pages > 0x7fffffffLL || static_cast<long long>(T) * H > 0x7fffffffLL)
    return DSA_ERR_SHAPE;
  if (logits_stride < max_context) return DSA_ERR_SHAPE;
  // every row of the table covers max_context keys (the kernel may read a
  // row's first blocks before it knows the token's context length)
  if (bt_stride < (static_cast<long long>(max_context) + kPageKeys - 1) / kPageKeys)
    return DSA_ERR_SHAPE;
  if (T == 0 || max_context == 0) return DSA_OK;
  if (!q_fp8 || !weights || !index_k_cache || !block_table || !context_lens || !logits)
    return DSA_ERR_NULL;
  if (misaligned(q_fp8, 16) || misaligned(index_k_cache, 16)) return DSA_ERR_ALIGN;
  if (misaligned(weights, 4) || misaligned(block_table, 4) || misaligned(context_lens, 4) ||
      misaligned(logits, 4))
    return DSA_ERR_ALIGN;

  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return DSA_ERR_LAUNCH;
  int sms = 0;
  if (logits_device(&sms) != cudaSuccess) return DSA_ERR_LAUNCH;

  // q codes: [T*H rows of 128 bytes]; one box = the H rows of a token
  alignas(64) CUtensorMap tq;
  {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(T) * H};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(H)};
    cuuint32_t estr[2] = {1, 1};
    if (encode(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(q_fp8), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return DSA_ERR_LAUNCH;
  }
  // key codes: [pages][64 rows][128 bytes] inside the page-blocked cache
  alignas(64) CUtensorMap tk;
  {
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(kPageKeys),
                          static_cast<cuuint64_t>(num_pages)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(kPageStride)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kD), static_cast<cuuint32_t>(kPageKeys), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(index_k_cache), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return DSA_ERR_LAUNCH;
  }

  LParams p = {};
  p.weights = weights;
  p.cache = static_cast<const uint8_t*>(index_k_cache);
  p.num_pages = num_pages;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.context_lens = context_lens;
  p.logits = logits;
  p.logits_stride = logits_stride;
  p.max_context = max_context;
  p.tiles_max = (max_context + kTileKeys - 1) / kTileKeys;
  p.T = T;
  // A launch without PDL starts once the previous kernel has finished, so
  // it may read the lengths and the table at once, as the early mode does.
  p.early_index = ((flags & DSA_FLAG_PDL_EARLY_INDEX) || !(flags & DSA_FLAG_PDL)) ? 1 : 0;
  p.err = err_flags;
  // split each token's tiles over as many CTAs as fit on the GPU at once
  // (all resident: no second wave), at least one per token
  int gx = resident_ctas(H) / T;
  if (gx > p.tiles_max) gx = p.tiles_max;
  if (gx < 1) gx = 1;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(T));
  const bool pdl = (flags & DSA_FLAG_PDL) != 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (H) {
    case 16: e = launch_logits<16>(tq, tk, p, grid, pdl, s); break;
    case 32: e = launch_logits<32>(tq, tk, p, grid, pdl, s); break;
    case 64: e = launch_logits<64>(tq, tk, p, grid, pdl, s); break;
    default: e = launch_logits<128>(tq, tk, p, grid, pdl, s); break;
  }
  return e == cudaSuccess ? DSA_OK : DSA_ERR_LAUNCH;
}

}  // extern "C"
