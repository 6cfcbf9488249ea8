// DSA indexer Q/K prepare-and-store for GB300 (sm_103a): kernel, launcher
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
// Kernel shape (persistent, warp-specialised):
//   * a unit of work is one token and a chunk of HC <= 64 of its heads (the
//     chunk starting at head 0 also carries the token's key);
//   * warp 0 is the producer: its lane 0 moves each unit's bytes -- the HC
//     query rows, the key row, the cos/sin rows of the token's position and the
//     gate weights -- from HBM into a 4-stage shared-memory ring with bulk
//     asynchronous copies (cp.async.bulk, completion counted on an mbarrier);
//     the other lanes prefetch positions and slots 32 units ahead;
//   * warps 1..NCW are consumers: each reads a stage, runs RoPE (+ LayerNorm
//     for the key), the amax / ue8m0 / e4m3 quantisation and the gate fold in
//     registers, stores the results straight to global memory, and releases
//     the stage on its "empty" mbarrier.
// Bytes in flight are set by the ring depth (up to ~200 KB per SM), not by
// registers or occupancy.  Every mbarrier wait is bounded in time; on expiry
// the CTA raises DSA_DEVERR_TIMEOUT, drains its own copies (bounded too) and
// exits, so a fault can never hang the device.
//
// Lane layout inside a consumer: a half-warp owns one 128-vector, lane l16
// holds elements 8*l16 .. 8*l16+7 (one 16-byte shared-memory load, one 8-byte
// global store of codes).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "dsa_prep.h"

namespace {

constexpr int kD = DSA_HEAD_DIM;
constexpr int kHCMax = 64;        // heads per unit at most
constexpr int kStages = 4;        // shared-memory ring depth
constexpr int kConsumers = 8;     // consumer warps per CTA
constexpr int kThreads = 32 * (1 + kConsumers);
constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// stage layout (byte offsets from the stage base)
constexpr int kOffHdr = 0;     // StageHeader
constexpr int kOffK = 64;      // key row, 256 B
constexpr int kOffCos = 320;   // cos row, rope_dim/2 floats (<= 256 B)
constexpr int kOffSin = 576;   // sin row
constexpr int kOffW = 832;     // gate weights of the chunk, HC bf16 (<= 128 B)
constexpr int kOffQ = 1024;    // HC query rows of 256 B
constexpr int kBarrierBytes = 128;  // full[kStages], empty[kStages], abort flag

struct StageHeader {
  long long pos;
  long long slot;
  int pos_ok;
};

struct Params {
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
  uint8_t* cache;
  long long num_slots;
  long long page_bytes;  // page_size * 132
  int page_size;
  int T;
  int H;
  int rope_dim;
  int cs_bytes;   // rope_dim / 2 * 4
  int HC;         // heads per unit
  int NC;         // units per token
  long long units;
  int stage_bytes;
  int w_bulk;     // the chunk's weights can be bulk-copied (16-byte aligned)
  int* err;
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete.  Returns false when
// the CTA was told to abort or after kWaitLimitNs.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// Global -> shared bulk copy; completion is counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Programmatic dependent launch: no-ops unless the launch carries the attribute.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 ld_shared16(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}

__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 r;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "r"(addr));
  return r;
}

__device__ __forceinline__ void st_stream8(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
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

__device__ __forceinline__ float pow2f(int e) {
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// ---------------------------------------------------------------- the math

// Per-unit rotation operands of this lane.
//   NeoX: lanes [0, r/16) hold the first members a of pairs 8*l16 .. 8*l16+7,
//         lanes [r/16, r/8) the second members b of the same pairs.  Every lane
//         computes own' = fma(own, c, partner * s'), with s' = -s for the
//         first members (so partner * s' = -(b*s) exactly) and s' = s for the
//         second ones -- the fused forms a' = fma(a, c, -(b*s)) and
//         b' = fma(b, c, a*s) with the products rounded to fp32.
//   GPT-J: lane l16 < r/8 holds pairs 4*l16 .. 4*l16+3 inside its 8 values.
struct Rot {
  float c[8];
  float s[8];
  bool rot;
  bool first;
  int partner;
};

template <int STYLE>
__device__ __forceinline__ void load_rot(Rot& R, uint32_t st, int l16, int rope_dim) {
  const int rl = rope_dim >> 4;
#pragma unroll
  for (int j = 0; j < 8; ++j) R.c[j] = 1.0f, R.s[j] = 0.0f;
  R.rot = l16 < 2 * rl;
  R.first = l16 < rl;
  R.partner = R.first ? l16 + rl : (R.rot ? l16 - rl : l16);
  if (!R.rot) return;
  if (STYLE == DSA_ROPE_NEOX) {
    const int base = 4 * 8 * (R.first ? l16 : l16 - rl);
    const float4 c0 = ld_shared_f4(st + kOffCos + base), c1 = ld_shared_f4(st + kOffCos + base + 16);
    const float4 s0 = ld_shared_f4(st + kOffSin + base), s1 = ld_shared_f4(st + kOffSin + base + 16);
    R.c[0] = c0.x; R.c[1] = c0.y; R.c[2] = c0.z; R.c[3] = c0.w;
    R.c[4] = c1.x; R.c[5] = c1.y; R.c[6] = c1.z; R.c[7] = c1.w;
    R.s[0] = s0.x; R.s[1] = s0.y; R.s[2] = s0.z; R.s[3] = s0.w;
    R.s[4] = s1.x; R.s[5] = s1.y; R.s[6] = s1.z; R.s[7] = s1.w;
    if (R.first) {
#pragma unroll
      for (int j = 0; j < 8; ++j) R.s[j] = -R.s[j];
    }
  } else {
    const float4 c0 = ld_shared_f4(st + kOffCos + 16 * l16);
    const float4 s0 = ld_shared_f4(st + kOffSin + 16 * l16);
    R.c[0] = c0.x; R.c[1] = c0.y; R.c[2] = c0.z; R.c[3] = c0.w;
    R.s[0] = s0.x; R.s[1] = s0.y; R.s[2] = s0.z; R.s[3] = s0.w;
  }
}

// RoPE on this lane's 8 values.  Every lane of the warp must call it (NeoX
// exchanges values with the lane r/16 away).
template <int STYLE>
__device__ __forceinline__ void rope_apply(float (&x)[8], const Rot& R) {
  if (STYLE == DSA_ROPE_NEOX) {
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = __shfl_sync(kFull, x[j], R.partner, 16);
    if (R.rot) {
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const float2 ps = __fmul2_rn(make_float2(o[j], o[j + 1]), make_float2(R.s[j], R.s[j + 1]));
        const float2 r = __ffma2_rn(make_float2(x[j], x[j + 1]), make_float2(R.c[j], R.c[j + 1]), ps);
        x[j] = r.x;
        x[j + 1] = r.y;
      }
    }
  } else {
    if (R.rot) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = x[2 * j], b = x[2 * j + 1];
        x[2 * j] = __fmaf_rn(a, R.c[j], -__fmul_rn(b, R.s[j]));
        x[2 * j + 1] = __fmaf_rn(b, R.c[j], __fmul_rn(a, R.s[j]));
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
  float m01, m23;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m01) : "f"(fabsf(x[0])), "f"(fabsf(x[1])), "f"(fabsf(x[2])));
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m23) : "f"(fabsf(x[3])), "f"(fabsf(x[4])), "f"(fabsf(x[5])));
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(m01), "f"(m23), "f"(fabsf(x[6])));
  m = fmaxf(m, fabsf(x[7]));
  m = fmaxf(halfwarp_max(m), 1e-4f);
  const uint32_t b = __float_as_uint(m);
  return static_cast<int>(b >> 23) - 135 + ((b & 0x7fffffu) > 0x600000u ? 1 : 0);
}

// codes = e4m3_rne(x * 2^-e): the multiply by a power of two is exact.
__device__ __forceinline__ uint2 quantize8(const float (&x)[8], int e) {
  const float inv = pow2f(-e);
  const float2 i2 = make_float2(inv, inv);
  const float2 v0 = __fmul2_rn(make_float2(x[0], x[1]), i2);
  const float2 v1 = __fmul2_rn(make_float2(x[2], x[3]), i2);
  const float2 v2 = __fmul2_rn(make_float2(x[4], x[5]), i2);
  const float2 v3 = __fmul2_rn(make_float2(x[6], x[7]), i2);
  const uint32_t p0 = cvt_e4m3x2(v0.x, v0.y), p1 = cvt_e4m3x2(v1.x, v1.y);
  const uint32_t p2 = cvt_e4m3x2(v2.x, v2.y), p3 = cvt_e4m3x2(v3.x, v3.y);
  return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
}

// ---------------------------------------------------------------- roles

__device__ __forceinline__ void raise_error(const Params& p, int bit) {
  if (p.err) atomicOr(p.err, bit);
}

// Producer warp: lane 0 fills the ring; all lanes prefetch (position, slot)
// for the next 32 units of this CTA.
__device__ void producer(const Params& p, unsigned char* ring, uint32_t full0, uint32_t empty0,
                         volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  long long my_pos = 0, my_slot = 0;
  int i = 0;
  for (long long u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
    const int j = i & 31;
    if (j == 0) {
      const long long uu = u + static_cast<long long>(lane) * gridDim.x;
      my_pos = 0;
      my_slot = 0;
      if (uu < p.units) {
        const long long tt = uu / p.NC;
        my_pos = __ldg(p.pos + tt);
        if (uu - tt * p.NC == 0) my_slot = __ldg(p.loc + tt);
      }
    }
    const long long pos = __shfl_sync(kFull, my_pos, j);
    const long long slot = __shfl_sync(kFull, my_slot, j);
    int stop = 0;
    if (lane == 0) {
      const int s = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      const uint32_t full = full0 + 8 * s, empty = empty0 + 8 * s;
      unsigned char* st = ring + static_cast<size_t>(s) * p.stage_bytes;
      const uint32_t sts = smem_u32(st);
      if (i >= kStages && !mbar_wait(empty, ph ^ 1, abort_flag)) {
        stop = 1;
      } else {
        const long long t = u / p.NC;
        const int c = static_cast<int>(u - t * p.NC);
        const int h0 = c * p.HC;
        const int n = min(p.HC, p.H - h0);
        const bool pos_ok = pos >= 0 && pos < p.max_pos;
        const long long row = pos_ok ? pos : 0;
        StageHeader* hd = reinterpret_cast<StageHeader*>(st + kOffHdr);
        hd->pos = pos;
        hd->slot = slot;
        hd->pos_ok = pos_ok ? 1 : 0;
        const uint32_t bytes = static_cast<uint32_t>(n) * 256u + (c == 0 ? 256u : 0u) +
                               (p.rope_dim ? 2u * p.cs_bytes : 0u) +
                               (p.w_bulk ? 2u * n : 0u);
        mbar_arrive_expect_tx(full, bytes);
        if (n > 0) {
          const uint16_t* qsrc = p.q + t * p.sq_t + static_cast<long long>(h0) * p.sq_h;
          if (p.sq_h == kD) {
            bulk_g2s(sts + kOffQ, qsrc, static_cast<uint32_t>(n) * 256u, full);
          } else {
            for (int h = 0; h < n; ++h) bulk_g2s(sts + kOffQ + 256 * h, qsrc + h * p.sq_h, 256u, full);
          }
          if (p.w_bulk) bulk_g2s(sts + kOffW, p.w + t * p.sw_t + h0, 2u * n, full);
        }
        if (c == 0) bulk_g2s(sts + kOffK, p.k + t * p.sk_t, 256u, full);
        if (p.rope_dim) {
          bulk_g2s(sts + kOffCos, p.cos_t + row * p.cs_stride, p.cs_bytes, full);
          bulk_g2s(sts + kOffSin, p.sin_t + row * p.cs_stride, p.cs_bytes, full);
        }
      }
    }
    stop = __shfl_sync(kFull, stop, 0);
    if (stop) {
      if (lane == 0) {
        *abort_flag = 1;
        raise_error(p, DSA_DEVERR_TIMEOUT);
      }
      break;
    }
  }
  // Stay until the copies of the last (up to kStages) units have landed, so
  // the CTA never exits with a bulk copy still writing its shared memory.
  if (lane == 0) {
    volatile int never = 0;
    for (int d = (i > kStages ? i - kStages : 0); d < i; ++d)
      mbar_wait(full0 + 8 * (d % kStages), (d / kStages) & 1, &never);
  }
}

// One q vector (half-warp) -> codes, returns the scale exponent.
template <int STYLE>
__device__ __forceinline__ int q_vector(uint4 raw, const Rot& R, uint2& codes) {
  float x[8];
  unpack_bf16x8(raw, x);
  rope_apply<STYLE>(x, R);
  const int e = ue8m0_exponent(x);
  codes = quantize8(x, e);
  return e;
}

// The key of one token (half-warp): LayerNorm, RoPE, quantise, cache store.
template <int STYLE>
__device__ __forceinline__ void k_vector(const Params& p, uint32_t sts, const StageHeader& hd,
                                         const Rot& R, bool real, int l16) {
  const uint4 raw = ld_shared16(sts + kOffK + 16 * l16);
  const float4* g4 = reinterpret_cast<const float4*>(p.gamma + 8 * l16);
  const float4* b4 = reinterpret_cast<const float4*>(p.beta + 8 * l16);
  const float4 g0 = __ldg(g4), g1 = __ldg(g4 + 1), b0 = __ldg(b4), b1 = __ldg(b4 + 1);
  const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
  const float bt[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};

  // LayerNorm: mean, biased variance, eps inside the root
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

  rope_apply<STYLE>(x, R);
  const int e = ue8m0_exponent(x);
  const uint2 codes = quantize8(x, e);

  if (!real) return;
  if (!hd.pos_ok) {
    if (l16 == 0) raise_error(p, DSA_DEVERR_POSITION);
    return;
  }
  const long long slot = hd.slot;
  if (slot < 0 || slot >= p.num_slots) {
    if (l16 == 0) raise_error(p, DSA_DEVERR_SLOT);
    return;
  }
  const long long page = slot / p.page_size;
  const long long off = slot - page * p.page_size;
  uint8_t* base = p.cache + page * p.page_bytes;
  *reinterpret_cast<uint2*>(base + off * kD + 8 * l16) = codes;
  if (l16 == 0)
    *reinterpret_cast<float*>(base + static_cast<long long>(p.page_size) * kD + 4 * off) = pow2f(e);
}

template <int STYLE>
__device__ void consumer(const Params& p, int cw, unsigned char* ring, uint32_t full0,
                         uint32_t empty0, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const int hw = lane >> 4;
  const int l16 = lane & 15;
  int i = 0;
  for (long long u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
    const int s = i % kStages;
    const uint32_t ph = (i / kStages) & 1;
    unsigned char* st = ring + static_cast<size_t>(s) * p.stage_bytes;
    const uint32_t sts = smem_u32(st);
    const bool ok = mbar_wait(full0 + 8 * s, ph, abort_flag);
    if (!__all_sync(kFull, ok)) {
      if (lane == 0) {
        *abort_flag = 1;
        raise_error(p, DSA_DEVERR_TIMEOUT);
      }
      return;
    }
    const StageHeader hd = *reinterpret_cast<const StageHeader*>(st + kOffHdr);
    const long long t = u / p.NC;
    const int c = static_cast<int>(u - t * p.NC);
    const int h0 = c * p.HC;
    const int n = min(p.HC, p.H - h0);

    Rot R;
    load_rot<STYLE>(R, sts, l16, p.rope_dim);

    // query heads: warp cw takes head pairs cw, cw + kConsumers, ...
    for (int pr = cw; 2 * pr < n; pr += kConsumers) {
      const int v = 2 * pr + hw;
      const bool valid = v < n;
      float wv = 0.0f;
      if (valid && l16 == 0)
        wv = p.w_bulk ? bf16_to_f32(*reinterpret_cast<const uint16_t*>(st + kOffW + 2 * v))
                      : bf16_to_f32(__ldg(p.w + t * p.sw_t + h0 + v));
      const uint4 raw = valid ? ld_shared16(sts + kOffQ + 256 * v + 16 * l16) : make_uint4(0, 0, 0, 0);
      uint2 codes;
      const int e = q_vector<STYLE>(raw, R, codes);
      if (valid && hd.pos_ok) {
        const long long row = t * p.H + h0 + v;
        st_stream8(p.q_out + row * kD + 8 * l16, codes);
        if (l16 == 0) __stcs(p.w_out + row, __fmul_rn(__fmul_rn(wv, pow2f(e)), p.fold));
      }
    }
    // the key rides with chunk 0; the warp that takes it rotates per unit
    if (c == 0 && cw == i % kConsumers) k_vector<STYLE>(p, sts, hd, R, hw == 0, l16);

    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
}

template <int STYLE>
__global__ void __launch_bounds__(kThreads) dsa_prepare_store_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
  unsigned char* ring = smem + kBarrierBytes;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + kStages);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kConsumers);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // inputs may be written by the kernel before this one in the stream (PDL)
  grid_dependency_wait();
  grid_launch_dependents();

  const int warp = threadIdx.x >> 5;
  if (warp == 0)
    producer(p, ring, full0, empty0, abort_flag);
  else
    consumer<STYLE>(p, warp - 1, ring, full0, empty0, abort_flag);
}

// ---------------------------------------------------------------- host side

bool misaligned(const void* ptr, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) != 0;
}

// Per-device facts looked up once: SM count, and whether the kernels' dynamic
// shared-memory limit has been raised on that device.
struct DeviceInfo {
  int sms = 0;
  bool smem_set = false;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

int max_smem_bytes() { return kBarrierBytes + kStages * (kOffQ + kHCMax * 256); }

cudaError_t device_info(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.smem_set) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dsa_prepare_store_kernel<DSA_ROPE_NEOX>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_bytes());
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dsa_prepare_store_kernel<DSA_ROPE_GPTJ>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_bytes());
    if (e != cudaSuccess) return e;
    d.smem_set = true;
  }
  *sms = d.sms;
  return cudaSuccess;
}

// Heads per unit: whole tokens (HC = H, up to 64) when there are enough tokens
// to fill the machine; for small T the heads are split (down to 8 per unit)
// until the units cover the SMs.
// Chunks hold a multiple of 8 heads when H >= 8, so every chunk's weights start
// on a 16-byte boundary and can ride the bulk copies (when w itself allows).
void choose_units(Params& p, int sms, bool w_rows_aligned) {
  if (p.H == 0) {
    p.HC = 0;
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
  p.units = static_cast<long long>(p.T) * p.NC;
  p.stage_bytes = kOffQ + p.HC * 256;
  p.w_bulk = (w_rows_aligned && p.H % 8 == 0 && p.HC % 8 == 0) ? 1 : 0;
}

cudaError_t launch(Params& p, int rope_style, uint32_t flags, bool w_rows_aligned,
                   cudaStream_t stream) {
  int sms = 0;
  cudaError_t e = device_info(&sms);
  if (e != cudaSuccess) return e;
  choose_units(p, sms, w_rows_aligned);
  const int smem = kBarrierBytes + kStages * p.stage_bytes;
  const int per_sm = p.HC >= 32 ? 3 : 6;
  long long blocks = static_cast<long long>(sms) * per_sm;
  if (blocks > p.units) blocks = p.units;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (flags & DSA_FLAG_PDL) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return rope_style == DSA_ROPE_NEOX
             ? cudaLaunchKernelEx(&cfg, dsa_prepare_store_kernel<DSA_ROPE_NEOX>, p)
             : cudaLaunchKernelEx(&cfg, dsa_prepare_store_kernel<DSA_ROPE_GPTJ>, p);
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
  if (rope_dim < 0 || rope_dim > kD || rope_dim % 16 != 0) return DSA_ERR_UNSUPPORTED;
  if (rope_style != DSA_ROPE_NEOX && rope_style != DSA_ROPE_GPTJ) return DSA_ERR_UNSUPPORTED;
  if (flags & ~static_cast<uint32_t>(DSA_FLAG_PDL)) return DSA_ERR_UNSUPPORTED;
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
  p.pos = reinterpret_cast<const long long*>(positions);
  p.loc = reinterpret_cast<const long long*>(out_cache_loc);
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
  p.page_bytes = static_cast<long long>(page_size) * (kD + 4);
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
  }
  return "unknown status";
}

int32_t dsa_prep_version(void) { return (2 << 16) | 0; }

}  // extern "C"
