// Device-side building blocks shared by the fused kernels (dsa_prep.cu) and
// the unfused chain (dsa_unfused.cu): PTX wrappers, typed loads and stores,
// the balanced lane slice of a 128-vector, RoPE, the ue8m0 exponent and the
// e4m3 packing.  Header-only; every function is inline.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "dsa_prep.h"

namespace dsa_dev {

constexpr int kD = DSA_HEAD_DIM;
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One bounded probe: the thread may sleep up to ~1 ms inside it, waking as soon
// as the phase completes, so waiting warps do not spin on issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(bar), "r"(parity), "r"(1000000) : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// Wait for the phase with the given parity to complete.  Returns false when
// the CTA was told to abort or after kWaitLimitNs.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity,
                                            volatile int* abort_flag) {
  const unsigned long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag);
}

// Global -> shared bulk copy; completion is counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// Hint: bring `bytes` (a multiple of 16, 16-byte aligned) at global p into L2.
// L2 is the GPU's point of coherence, so a line prefetched before another
// kernel writes it is updated by that write; nothing is cached nearer.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// cp.async (LDGSTS): a thread copies 16 or 8 bytes from global to shared
// memory without holding a register for them; completion is tracked per
// thread in commit groups, so a later wait on an older group does not wait
// for the copies of a newer one.  .cg streams through L2 only (16 bytes);
// .ca (4, 8 or 16 bytes) may also keep the line in L1, for data many warps
// read, such as gamma and beta.
__device__ __forceinline__ void cp_async16_cg(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16_ca(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's most recent groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Programmatic dependent launch: no-ops unless the launch carries the attribute.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float pow2f(int e) {
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ---------------------------------------------------------------- memory spaces

// Loads of 2/4/8/16 bytes at a byte address, from global (read-only path,
// streaming) or from shared memory.
struct GlobalMem {
  using Addr = const unsigned char*;
  __device__ __forceinline__ static uint4 ld16(Addr a) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(a));
    return r;
  }
  __device__ __forceinline__ static uint2 ld8(Addr a) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(a));
    return r;
  }
  __device__ __forceinline__ static uint32_t ld4(Addr a) {
    uint32_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(a));
    return r;
  }
  __device__ __forceinline__ static uint32_t ld2(Addr a) {
    uint16_t r;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(a));
    return r;
  }
};

struct SharedMem {
  using Addr = uint32_t;
  __device__ __forceinline__ static uint4 ld16(Addr a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
  }
  __device__ __forceinline__ static uint2 ld8(Addr a) {
    uint2 r;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
  }
  __device__ __forceinline__ static uint32_t ld4(Addr a) {
    uint32_t r;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(r) : "r"(a));
    return r;
  }
  __device__ __forceinline__ static uint32_t ld2(Addr a) {
    uint16_t r;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(a));
    return r;
  }
};

__host__ __device__ constexpr int pow2_floor(int x) { return x >= 16 ? 16 : x >= 8 ? 8 : x >= 4 ? 4 : x >= 2 ? 2 : 1; }
__host__ __device__ constexpr int gcd_pow2(int x) { return x == 0 ? 16 : (x & -x) > 16 ? 16 : (x & -x); }

// `BYTES` bytes at `a` (aligned to ALIGN) as 32-bit words w[]; 2-byte pieces
// land in the low half of a word.
template <class M, int BYTES, int ALIGN>
__device__ __forceinline__ void load_words(typename M::Addr a, uint32_t* w) {
  constexpr int W = pow2_floor(ALIGN < BYTES ? ALIGN : BYTES);
#pragma unroll
  for (int b = 0; b < BYTES; b += W) {
    if constexpr (W == 16) {
      const uint4 v = M::ld16(a + b);
      w[b / 4] = v.x; w[b / 4 + 1] = v.y; w[b / 4 + 2] = v.z; w[b / 4 + 3] = v.w;
    } else if constexpr (W == 8) {
      const uint2 v = M::ld8(a + b);
      w[b / 4] = v.x; w[b / 4 + 1] = v.y;
    } else if constexpr (W == 4) {
      w[b / 4] = M::ld4(a + b);
    } else {
      w[b / 4] = M::ld2(a + b);
    }
  }
}

// N bf16 elements -> fp32 x[0..N)
template <class M, int N, int ALIGN>
__device__ __forceinline__ void load_bf16(typename M::Addr a, float* x) {
  uint32_t w[(2 * N + 3) / 4];
  load_words<M, 2 * N, ALIGN>(a, w);
#pragma unroll
  for (int j = 0; j < N; ++j) x[j] = (j & 1) ? bf16_hi(w[j / 2]) : bf16_lo(w[j / 2]);
}

// N fp32 values from global (gamma / beta / cos / sin rows), read-only cached.
template <int N, int ALIGN>
__device__ __forceinline__ void load_f32_global(const float* p, float* x) {
  constexpr int W = pow2_floor(ALIGN < 4 * N ? ALIGN : 4 * N);
#pragma unroll
  for (int b = 0; b < 4 * N; b += W) {
    if constexpr (W == 16) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(p + b / 4));
      x[b / 4] = v.x; x[b / 4 + 1] = v.y; x[b / 4 + 2] = v.z; x[b / 4 + 3] = v.w;
    } else if constexpr (W == 8) {
      const float2 v = __ldg(reinterpret_cast<const float2*>(p + b / 4));
      x[b / 4] = v.x; x[b / 4 + 1] = v.y;
    } else {
      x[b / 4] = __ldg(p + b / 4);
    }
  }
}

template <int N, int ALIGN>
__device__ __forceinline__ void load_f32_shared(uint32_t a, float* x) {
  uint32_t w[N];
  load_words<SharedMem, 4 * N, ALIGN>(a, w);
#pragma unroll
  for (int j = 0; j < N; ++j) x[j] = __uint_as_float(w[j]);
}

// N fp32 values at element offset `off` of an fp32 row held in global memory
// (read-only cached) or in shared memory (byte address).
template <int N, int ALIGN>
__device__ __forceinline__ void load_f32_at(const float* row, int off, float* x) {
  load_f32_global<N, ALIGN>(row + off, x);
}
template <int N, int ALIGN>
__device__ __forceinline__ void load_f32_at(uint32_t row, int off, float* x) {
  load_f32_shared<N, ALIGN>(row + 4 * off, x);
}

// Store `BYTES` bytes (packed little-endian in w[]) at global p when `pred`
// holds.  The predicate goes on the store instructions themselves, so a
// quarter-warp that skips its store costs no branch.  STREAM selects the
// evict-first cache hint for data this pass will not read again.
#define DSA_ST_PRED(OP, ...)                                                            \
  asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n @q " OP "\n}" ::__VA_ARGS__ \
               : "memory")
template <int BYTES, int ALIGN, bool STREAM = true>
__device__ __forceinline__ void store_codes(uint8_t* p, const uint32_t* w, bool pred = true) {
  constexpr int W = pow2_floor(ALIGN < BYTES ? ALIGN : BYTES);
  const uint32_t q = pred ? 1u : 0u;
#pragma unroll
  for (int b = 0; b < BYTES; b += W) {
    if constexpr (W == 16) {
      if constexpr (STREAM)
        DSA_ST_PRED("st.global.cs.v4.u32 [%1], {%2,%3,%4,%5};", "r"(q), "l"(p + b), "r"(w[b / 4]),
                    "r"(w[b / 4 + 1]), "r"(w[b / 4 + 2]), "r"(w[b / 4 + 3]));
      else
        DSA_ST_PRED("st.global.v4.u32 [%1], {%2,%3,%4,%5};", "r"(q), "l"(p + b), "r"(w[b / 4]),
                    "r"(w[b / 4 + 1]), "r"(w[b / 4 + 2]), "r"(w[b / 4 + 3]));
    } else if constexpr (W == 8) {
      if constexpr (STREAM)
        DSA_ST_PRED("st.global.cs.v2.u32 [%1], {%2,%3};", "r"(q), "l"(p + b), "r"(w[b / 4]),
                    "r"(w[b / 4 + 1]));
      else
        DSA_ST_PRED("st.global.v2.u32 [%1], {%2,%3};", "r"(q), "l"(p + b), "r"(w[b / 4]),
                    "r"(w[b / 4 + 1]));
    } else if constexpr (W == 4) {
      if constexpr (STREAM)
        DSA_ST_PRED("st.global.cs.u32 [%1], %2;", "r"(q), "l"(p + b), "r"(w[b / 4]));
      else
        DSA_ST_PRED("st.global.u32 [%1], %2;", "r"(q), "l"(p + b), "r"(w[b / 4]));
    } else if constexpr (W == 2) {
      const uint16_t v = static_cast<uint16_t>(w[b / 4] >> (8 * (b & 3)));
      if constexpr (STREAM)
        DSA_ST_PRED("st.global.cs.u16 [%1], %2;", "r"(q), "l"(p + b), "h"(v));
      else
        DSA_ST_PRED("st.global.u16 [%1], %2;", "r"(q), "l"(p + b), "h"(v));
    } else {
      const uint16_t v = static_cast<uint16_t>((w[b / 4] >> (8 * (b & 3))) & 0xff);
      if constexpr (STREAM)
        DSA_ST_PRED("st.global.cs.u8 [%1], %2;", "r"(q), "l"(p + b), "h"(v));
      else
        DSA_ST_PRED("st.global.u8 [%1], %2;", "r"(q), "l"(p + b), "h"(v));
    }
  }
}

// One fp32 at global p when `pred` holds (evict-first), without a branch.
__device__ __forceinline__ void store_f32_cs(float* p, float v, bool pred) {
  DSA_ST_PRED("st.global.cs.f32 [%1], %2;", "r"(pred ? 1u : 0u), "l"(p), "f"(v));
}

// The same with the default cache policy.
__device__ __forceinline__ void store_f32(float* p, float v, bool pred) {
  DSA_ST_PRED("st.global.f32 [%1], %2;", "r"(pred ? 1u : 0u), "l"(p), "f"(v));
}

// ---------------------------------------------------------------- the slice

// Where a lane's 16 elements live (element offsets inside the 128-vector and
// their alignment in bytes for bf16 / e4m3 / fp32 rows).
template <int STYLE, int RP>
struct Slice {
  static constexpr int R = 16 * RP;      // rope_dim
  static constexpr int NR = 2 * RP;      // rotated elements per lane
  static constexpr int NP = 16 - NR;     // pass-through elements per lane
  static constexpr bool NEOX = STYLE == DSA_ROPE_NEOX;
  // element offset of each chunk for lane l: base + stride * l
  static constexpr int A_STRIDE = NEOX ? RP : 2 * RP;  // NeoX a-chunk / GPT-J pair chunk
  static constexpr int B_BASE = R / 2;                  // NeoX b-chunk
  static constexpr int P_BASE = R;
  // alignments (bytes) of the per-lane chunk starts
  static constexpr int ALIGN_A_BF16 = gcd_pow2(2 * A_STRIDE);
  static constexpr int ALIGN_B_BF16 = gcd_pow2(2 * RP) < gcd_pow2(2 * B_BASE) ? gcd_pow2(2 * RP)
                                                                               : gcd_pow2(2 * B_BASE);
  static constexpr int ALIGN_P_BF16 = gcd_pow2(2 * NP) < gcd_pow2(2 * P_BASE) ? gcd_pow2(2 * NP)
                                                                               : gcd_pow2(2 * P_BASE);
  static constexpr int ALIGN_A_U8 = gcd_pow2(A_STRIDE);
  static constexpr int ALIGN_B_U8 = gcd_pow2(RP) < gcd_pow2(B_BASE) ? gcd_pow2(RP) : gcd_pow2(B_BASE);
  static constexpr int ALIGN_P_U8 = gcd_pow2(NP) < gcd_pow2(P_BASE) ? gcd_pow2(NP) : gcd_pow2(P_BASE);
  static constexpr int ALIGN_A_F32 = gcd_pow2(4 * A_STRIDE);
  static constexpr int ALIGN_B_F32 = gcd_pow2(4 * RP) < gcd_pow2(4 * B_BASE) ? gcd_pow2(4 * RP)
                                                                               : gcd_pow2(4 * B_BASE);
  static constexpr int ALIGN_P_F32 = gcd_pow2(4 * NP) < gcd_pow2(4 * P_BASE) ? gcd_pow2(4 * NP)
                                                                               : gcd_pow2(4 * P_BASE);
  static constexpr int ALIGN_CS = gcd_pow2(4 * RP);
};

// Load the lane's 16 bf16 values of a row into x[]: x[0..RP) the a-members,
// x[RP..2RP) the b-members, x[2RP..16) the pass-through values.
template <int STYLE, int RP, class M>
__device__ __forceinline__ void load_slice(typename M::Addr row, int l, float (&x)[16]) {
  using S = Slice<STYLE, RP>;
  if constexpr (RP > 0) {
    if constexpr (S::NEOX) {
      load_bf16<M, RP, S::ALIGN_A_BF16>(row + 2 * RP * l, x);
      load_bf16<M, RP, S::ALIGN_B_BF16>(row + 2 * (S::B_BASE + RP * l), x + RP);
    } else {
      float t[2 * RP];
      load_bf16<M, 2 * RP, S::ALIGN_A_BF16>(row + 4 * RP * l, t);
#pragma unroll
      for (int j = 0; j < RP; ++j) x[j] = t[2 * j], x[RP + j] = t[2 * j + 1];
    }
  }
  if constexpr (S::NP > 0) load_bf16<M, S::NP, S::ALIGN_P_BF16>(row + 2 * (S::P_BASE + S::NP * l), x + 2 * RP);
}

// Rotation operands of the lane: frequencies RP*l .. RP*l + RP - 1.
template <int RP>
struct Rot {
  float c[RP > 0 ? RP : 1];
  float s[RP > 0 ? RP : 1];
  float ns[RP > 0 ? RP : 1];
};

template <int RP>
__device__ __forceinline__ void finish_rot(Rot<RP>& r) {
#pragma unroll
  for (int j = 0; j < RP; ++j) r.ns[j] = -r.s[j];
}

// RoPE on the lane's pairs (a_j, b_j):
//   a' = fma(a, c, b * (-s)) = fma(a, c, -(b*s)),  b' = fma(b, c, a * s),
// products rounded to fp32 (no contraction), two pairs per packed instruction.
template <int RP>
__device__ __forceinline__ void rope_slice(float (&x)[16], const Rot<RP>& r) {
  if constexpr (RP == 1) {
    const float a = x[0], b = x[1];
    x[0] = __fmaf_rn(a, r.c[0], __fmul_rn(b, r.ns[0]));
    x[1] = __fmaf_rn(b, r.c[0], __fmul_rn(a, r.s[0]));
  } else {
#pragma unroll
    for (int j = 0; j < RP; j += 2) {
      const float2 a = make_float2(x[j], x[j + 1]);
      const float2 b = make_float2(x[RP + j], x[RP + j + 1]);
      const float2 c = make_float2(r.c[j], r.c[j + 1]);
      const float2 pa = __fmul2_rn(b, make_float2(r.ns[j], r.ns[j + 1]));
      const float2 pb = __fmul2_rn(a, make_float2(r.s[j], r.s[j + 1]));
      const float2 na = __ffma2_rn(a, c, pa);
      const float2 nb = __ffma2_rn(b, c, pb);
      x[j] = na.x; x[j + 1] = na.y;
      x[RP + j] = nb.x; x[RP + j + 1] = nb.y;
    }
  }
}

// Quarter-warp reductions (xor offsets 4, 2, 1 stay inside the 8-lane group).
// (The single-instruction f32 max reduction over a lane mask measured slower
// here than these three shuffles, in latency and in throughput.)
__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 4));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 2));
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 1));
  return v;
}

__device__ __forceinline__ float quad_sum(float v) {
  v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 4));
  v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 2));
  v = __fadd_rn(v, __shfl_xor_sync(kFull, v, 1));
  return v;
}

// LayerNorm statistics of the quarter-warp's 128-vector (16 values in each of
// its 8 lanes): the mean and M2, the sum of squared deviations from it.  Each
// lane takes the mean and M2 of its own 16 values (pairwise sums, two at a
// time in packed f32x2 instructions), then three merges with the xor
// partners 4, 2 and 1 combine two sets a and b of n values each as
//   mean = (mean_a + mean_b) / 2,   M2 = M2_a + M2_b + d^2 * n / 2,
// d = mean_b - mean_a (the pairwise update of Chan, Golub and LeVeque,
// "Algorithms for computing the sample variance", 1983).  Every step is
// symmetric in a and b, so the 8 lanes end with bit-identical results; three
// shuffle rounds instead of the six of a two-pass sum.
__device__ __forceinline__ float2 f2(const float (&x)[16], int j) {
  return make_float2(x[2 * j], x[2 * j + 1]);
}

__device__ __forceinline__ void ln_stats(const float (&x)[16], float& mean, float& m2) {
  // sum: (x0 + x2 + ..., x1 + x3 + ...) as a tree of packed adds
  float2 a[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) a[j] = __fadd2_rn(f2(x, 2 * j), f2(x, 2 * j + 1));
  a[0] = __fadd2_rn(a[0], a[1]);
  a[2] = __fadd2_rn(a[2], a[3]);
  a[0] = __fadd2_rn(a[0], a[2]);
  float m = __fmul_rn(__fadd_rn(a[0].x, a[0].y), 1.0f / 16.0f);
  // M2 of the lane's values about its own mean
  const float2 nm = make_float2(-m, -m);
  float2 q[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 d0 = __fadd2_rn(f2(x, 2 * j), nm);
    const float2 d1 = __fadd2_rn(f2(x, 2 * j + 1), nm);
    q[j] = __ffma2_rn(d1, d1, __fmul2_rn(d0, d0));
  }
  q[0] = __fadd2_rn(q[0], q[1]);
  q[2] = __fadd2_rn(q[2], q[3]);
  q[0] = __fadd2_rn(q[0], q[2]);
  float v = __fadd_rn(q[0].x, q[0].y);
  float half_n = 8.0f;  // n / 2, n = values per merged set
#pragma unroll
  for (int off = 4; off >= 1; off >>= 1) {
    const float mo = __shfl_xor_sync(kFull, m, off);
    const float vo = __shfl_xor_sync(kFull, v, off);
    const float d = __fsub_rn(mo, m);
    v = __fmaf_rn(d, __fmul_rn(d, half_n), __fadd_rn(v, vo));
    m = __fmul_rn(__fadd_rn(m, mo), 0.5f);
    half_n *= 2.0f;
  }
  mean = m;
  m2 = v;
}

// rstd of the LayerNorm (biased variance, eps inside the root) from M2, and
// x - mean in place.
__device__ __forceinline__ float ln_center(float (&x)[16], float eps) {
  float mean, m2;
  ln_stats(x, mean, m2);
  const float2 nm = make_float2(-mean, -mean);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 d = __fadd2_rn(f2(x, j), nm);
    x[2 * j] = d.x;
    x[2 * j + 1] = d.y;
  }
  return __frsqrt_rn(__fadd_rn(__fmul_rn(m2, 1.0f / kD), eps));
}

// ue8m0 exponent of the vector: the smallest e with max(amax, 1e-4) <= 448*2^e.
// With A = max(amax, 1e-4) = 1.f * 2^E (normal), 448 * 2^e = 1.75 * 2^(e+8), so
// e = E - 8 when the fraction is <= 0.75 (bits <= 0x600000) and E - 7 above:
// read straight off the exponent and fraction bits, no division or log.  The
// compare rides a carry: fraction > 0x600000 exactly when fraction + 0x1fffff
// reaches 2^23 and bumps the exponent field.
__device__ __forceinline__ float lane_amax(const float (&x)[16]) {
  float m = max3f(fabsf(x[0]), fabsf(x[1]), fabsf(x[2]));
#pragma unroll
  for (int j = 3; j < 15; j += 2) m = max3f(m, fabsf(x[j]), fabsf(x[j + 1]));
  return fmaxf(m, fabsf(x[15]));
}

__device__ __forceinline__ float vector_amax(const float (&x)[16]) { return quad_max(lane_amax(x)); }

__device__ __forceinline__ int exponent_of_amax(float amax) {
  const uint32_t b = __float_as_uint(fmaxf(amax, 1e-4f));
  return static_cast<int>((b + 0x1fffffu) >> 23) - 135;
}

__device__ __forceinline__ int ue8m0_exponent(const float (&x)[16]) {
  return exponent_of_amax(vector_amax(x));
}

// e4m3 codes of x * 2^-e (the multiply by a power of two is exact), packed in
// element order of each chunk: words wa (a-chunk or GPT-J pair chunk), wb
// (NeoX b-chunk), wp (pass-through chunk).
template <int STYLE, int RP>
__device__ __forceinline__ void quantize_slice(const float (&x)[16], int e, uint32_t* wa,
                                               uint32_t* wb, uint32_t* wp) {
  using S = Slice<STYLE, RP>;
  const float inv = pow2f(-e);
  const float2 i2 = make_float2(inv, inv);
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const float2 t = __fmul2_rn(make_float2(x[j], x[j + 1]), i2);
    v[j] = t.x;
    v[j + 1] = t.y;
  }
  if constexpr (RP > 0) {
    if constexpr (S::NEOX) {
      // a-chunk: v[0..RP), b-chunk: v[RP..2RP); RP = 1 packs a lone code
#pragma unroll
      for (int j = 0; j < RP; j += 2) {
        const uint32_t ca = cvt_e4m3x2(v[j], RP > 1 ? v[j + 1] : 0.0f);
        const uint32_t cb = cvt_e4m3x2(v[RP + j], RP > 1 ? v[RP + j + 1] : 0.0f);
        if ((j & 2) == 0) wa[j / 4] = ca, wb[j / 4] = cb;
        else wa[j / 4] |= ca << 16, wb[j / 4] |= cb << 16;
      }
    } else {
      // pair chunk in element order: a_0 b_0 a_1 b_1 ...
#pragma unroll
      for (int j = 0; j < RP; ++j) {
        const uint32_t c = cvt_e4m3x2(v[j], v[RP + j]);
        if ((j & 1) == 0) wa[j / 2] = c;
        else wa[j / 2] |= c << 16;
      }
    }
  }
#pragma unroll
  for (int j = 0; j < S::NP; j += 2) {
    const uint32_t c = cvt_e4m3x2(v[2 * RP + j], v[2 * RP + j + 1]);
    if ((j & 2) == 0) wp[j / 4] = c;
    else wp[j / 4] |= c << 16;
  }
}

// Store the lane's codes to a 128-byte row whose start is ROW_ALIGN-aligned.
template <int STYLE, int RP, int ROW_ALIGN = 16>
__device__ __forceinline__ void store_slice(uint8_t* row, int l, const uint32_t* wa,
                                            const uint32_t* wb, const uint32_t* wp,
                                            bool pred = true) {
  using S = Slice<STYLE, RP>;
  constexpr int AA = S::ALIGN_A_U8 < ROW_ALIGN ? S::ALIGN_A_U8 : ROW_ALIGN;
  constexpr int AB = S::ALIGN_B_U8 < ROW_ALIGN ? S::ALIGN_B_U8 : ROW_ALIGN;
  constexpr int AP = S::ALIGN_P_U8 < ROW_ALIGN ? S::ALIGN_P_U8 : ROW_ALIGN;
  if constexpr (RP > 0) {
    if constexpr (S::NEOX) {
      store_codes<RP, AA>(row + RP * l, wa, pred);
      store_codes<RP, AB>(row + S::B_BASE + RP * l, wb, pred);
    } else {
      store_codes<2 * RP, AA>(row + 2 * RP * l, wa, pred);
    }
  }
  if constexpr (S::NP > 0) store_codes<S::NP, AP>(row + S::P_BASE + S::NP * l, wp, pred);
}

// Index-K cache geometry and the store of one key's codes and scale into it.
//   page-blocked (default): page p holds page_size rows of 128 codes, then
//     page_size fp32 scales; slot s = row s % page_size of page s / page_size;
//   token-major (DSA_FLAG_CACHE_TOKEN_MAJOR): slot s owns bytes
//     [132 s, 132 s + 132): 128 codes, then its fp32 scale.
struct CacheGeom {
  uint8_t* cache;
  long long num_slots;
  long long page_bytes;  // page_size * 132
  int page_size;
  int page_shift;  // log2(page_size) when it is a power of two, else -1
  int token_major;
};

// log2(page_size) for a power of two, else -1 (set by the host).
inline int page_shift_of(int page_size) {
  for (int s = 0; s < 31; ++s)
    if ((1 << s) == page_size) return s;
  return -1;
}

// (page, row in page) of a valid slot: a shift and a mask for a power-of-two
// page size, else a 32-bit division while the slot fits (a 64-bit one is a
// long instruction sequence).
__device__ __forceinline__ void slot_page(const CacheGeom& g, long long slot, long long& page,
                                          long long& off) {
  if (g.page_shift >= 0) {
    page = slot >> g.page_shift;
    off = slot & (g.page_size - 1);
  } else if (slot <= 0xffffffffLL) {
    const uint32_t pg = static_cast<uint32_t>(slot) / static_cast<uint32_t>(g.page_size);
    page = pg;
    off = slot - static_cast<long long>(pg) * g.page_size;
  } else {
    page = slot / g.page_size;
    off = slot - page * g.page_size;
  }
}

// Store one key's codes and scale into slot `slot` (a valid slot) when
// `pred` holds; the predicate rides on the store instructions.
template <int STYLE, int RP>
__device__ __forceinline__ void store_index_k(const CacheGeom& g, long long slot, int l,
                                              const uint32_t* wa, const uint32_t* wb,
                                              const uint32_t* wp, int e, bool pred = true) {
  if (g.token_major) {
    uint8_t* row = g.cache + slot * (kD + 4);
    store_slice<STYLE, RP, 4>(row, l, wa, wb, wp, pred);
    store_f32(reinterpret_cast<float*>(row + kD), pow2f(e), pred && l == 0);
  } else {
    long long page, off;
    slot_page(g, slot, page, off);
    uint8_t* base = g.cache + page * g.page_bytes;
    store_slice<STYLE, RP>(base + off * kD, l, wa, wb, wp, pred);
    store_f32(reinterpret_cast<float*>(base + static_cast<long long>(g.page_size) * kD + 4 * off),
              pow2f(e), pred && l == 0);
  }
}

// y = x * rstd * gamma + beta on N values (at offset `at` of each of M
// vectors) whose gamma/beta start at `row` (fp32 [128] rows), one aligned
// piece at a time to keep few registers live; the piece is loaded once for
// all M vectors.
template <int N, int ALIGN, int M>
__device__ __forceinline__ void affine_piece(const float* g_row, const float* b_row,
                                             float (&x)[M][16], int at, const float (&rstd)[M]) {
  float g[N], b[N];
  load_f32_global<N, ALIGN>(g_row, g);
  load_f32_global<N, ALIGN>(b_row, b);
#pragma unroll
  for (int m = 0; m < M; ++m) {
    if (N % 2 == 0 && at % 2 == 0) {  // two elements per packed instruction
      const float2 r2 = make_float2(rstd[m], rstd[m]);
#pragma unroll
      for (int j = 0; j < N; j += 2) {
        const float2 y = __ffma2_rn(__fmul2_rn(make_float2(x[m][at + j], x[m][at + j + 1]), r2),
                                    make_float2(g[j], g[j + 1]), make_float2(b[j], b[j + 1]));
        x[m][at + j] = y.x;
        x[m][at + j + 1] = y.y;
      }
    } else {
#pragma unroll
      for (int j = 0; j < N; ++j)
        x[m][at + j] = __fmaf_rn(__fmul_rn(x[m][at + j], rstd[m]), g[j], b[j]);
    }
  }
}

template <int STYLE, int RP, int M>
__device__ __forceinline__ void affine_slice(const float* gamma, const float* beta, int l,
                                             float (&x)[M][16], const float (&rstd)[M]) {
  using S = Slice<STYLE, RP>;
  if constexpr (RP > 0) {
    if constexpr (S::NEOX) {
      affine_piece<RP, S::ALIGN_A_F32>(gamma + RP * l, beta + RP * l, x, 0, rstd);
      affine_piece<RP, S::ALIGN_B_F32>(gamma + S::B_BASE + RP * l, beta + S::B_BASE + RP * l,
                                       x, RP, rstd);
    } else {
      float g[2 * RP], b[2 * RP];
      load_f32_global<2 * RP, S::ALIGN_A_F32>(gamma + 2 * RP * l, g);
      load_f32_global<2 * RP, S::ALIGN_A_F32>(beta + 2 * RP * l, b);
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int j = 0; j < RP; ++j) {
          x[m][j] = __fmaf_rn(__fmul_rn(x[m][j], rstd[m]), g[2 * j], b[2 * j]);
          x[m][RP + j] = __fmaf_rn(__fmul_rn(x[m][RP + j], rstd[m]), g[2 * j + 1], b[2 * j + 1]);
        }
    }
  }
  constexpr int NP = S::NP;
  if constexpr (NP > 0) {
    // pieces of 4, 2 or 1 values, whichever divides the chunk (14 values at
    // rope_dim 16)
    constexpr int PIECE = NP % 4 == 0 ? 4 : NP % 2 == 0 ? 2 : 1;
#pragma unroll
    for (int j = 0; j < NP; j += PIECE) {
      constexpr int A = S::ALIGN_P_F32 < 4 * PIECE ? S::ALIGN_P_F32 : 4 * PIECE;
      affine_piece<PIECE, A>(gamma + S::P_BASE + NP * l + j, beta + S::P_BASE + NP * l + j, x,
                             2 * RP + j, rstd);
    }
  }
}

template <int STYLE, int RP>
__device__ __forceinline__ void affine_slice(const float* gamma, const float* beta, int l,
                                             float (&x)[16], float rstd) {
  const float r1[1] = {rstd};
  affine_slice<STYLE, RP, 1>(gamma, beta, l, reinterpret_cast<float (&)[1][16]>(x), r1);
}


// ---------------------------------------------------------------- Hadamard layout
//
// The variant that rotates q and k by the normalised Walsh-Hadamard matrix
// H_128 / sqrt(128) after RoPE (the rotation the fused path of sglang PR
// "[AMD] [GLM5] Fuse the DSA indexer Q/K rope + quant + K-cache write",
// Modifications, states it does without).  Its butterflies pair elements
// whose indices differ in one bit, so the lane layout must make every index
// bit either a register bit or a lane bit: each lane holds chunks of W
// consecutive elements dealt round-robin over the 8 lanes,
//   element (c * 8W + W * l + i)  of chunk c, offset i  ->  lane l,
// with W = rope_dim/16 (NeoX: chunk 0 the a-members, chunk 1 the b-members),
// 2 * rope_dim/16 (GPT-J: chunk 0 the interleaved pairs) or 16 (no RoPE).
// The rotated chunks are exactly those of Slice, so the RoPE operands and
// rope_slice carry over; only the pass-through elements are spread.  Index
// bits below log2(W) and from log2(8W) up are register bits; the three in
// between are the lane bits.  With GPT-J every chunk keeps its even elements
// in its first W/2 registers and its odd ones in the rest (chunk 0: the a-
// and b-members), so registers 2m and 2m+1 -- the operands of one packed
// f32x2 instruction -- differ in the same index bit in every chunk.
template <int STYLE, int RP>
struct HSlice {
  static constexpr bool NEOX = STYLE == DSA_ROPE_NEOX;
  static constexpr bool PAIRED = !NEOX && RP > 0;  // GPT-J: chunks hold pairs
  static constexpr int W = RP == 0 ? 16 : (NEOX ? RP : 2 * RP);
  static constexpr int NCH = 16 / W;
  static constexpr int STRIDE = 8 * W;  // elements from one of a lane's chunks to the next
  // register holding element i of chunk c (x[0..RP) a-members, x[RP..2RP) b-members)
  __host__ __device__ static constexpr int reg(int c, int i) {
    return c * W + (PAIRED ? ((i & 1) ? W / 2 + i / 2 : i / 2) : i);
  }
  // element index, less the lane's W * l, of register j
  __host__ __device__ static constexpr int off(int j) {
    return (j / W) * STRIDE +
           (PAIRED ? (j % W < W / 2 ? 2 * (j % W) : 2 * (j % W - W / 2) + 1) : j % W);
  }
  __host__ __device__ static constexpr int reg_at(int o) {
    for (int j = 0; j < 16; ++j)
      if (off(j) == o) return j;
    return -1;
  }
  // the k-th register (in increasing order) whose element has bit B clear
  __host__ __device__ static constexpr int low_reg(int B, int k) {
    for (int j = 0; j < 16; ++j)
      if ((off(j) & B) == 0 && k-- == 0) return j;
    return -1;
  }
};

// 2^-3.5 = 128^-0.5 rounded to fp32.
constexpr float kHadamardScale = 0.0883883461356163f;

template <int STYLE, int RP, class M>
__device__ __forceinline__ void load_hslice(typename M::Addr row, int l, float (&x)[16]) {
  using S = HSlice<STYLE, RP>;
#pragma unroll
  for (int c = 0; c < S::NCH; ++c) {
    float t[S::W];
    load_bf16<M, S::W, gcd_pow2(2 * S::W)>(row + 2 * (c * S::STRIDE + S::W * l), t);
#pragma unroll
    for (int i = 0; i < S::W; ++i) x[S::reg(c, i)] = t[i];
  }
}

template <int STYLE, int RP, int M>
__device__ __forceinline__ void affine_hslice(const float* gamma, const float* beta, int l,
                                              float (&x)[M][16], const float (&rstd)[M]) {
  using S = HSlice<STYLE, RP>;
  constexpr int PIECE = S::W < 4 ? S::W : 4;
#pragma unroll
  for (int c = 0; c < S::NCH; ++c)
#pragma unroll
    for (int i0 = 0; i0 < S::W; i0 += PIECE) {
      const int o = c * S::STRIDE + S::W * l + i0;
      float g[PIECE], b[PIECE];
      load_f32_global<PIECE, 4 * PIECE>(gamma + o, g);
      load_f32_global<PIECE, 4 * PIECE>(beta + o, b);
#pragma unroll
      for (int m = 0; m < M; ++m)
#pragma unroll
        for (int i = 0; i < PIECE; ++i) {
          float& v = x[m][S::reg(c, i0 + i)];
          v = __fmaf_rn(__fmul_rn(v, rstd[m]), g[i], b[i]);
        }
    }
}

template <int STYLE, int RP>
__device__ __forceinline__ void affine_hslice(const float* gamma, const float* beta, int l,
                                              float (&x)[16], float rstd) {
  const float r1[1] = {rstd};
  affine_hslice<STYLE, RP, 1>(gamma, beta, l, reinterpret_cast<float (&)[1][16]>(x), r1);
}

// Butterflies on index bit log2(B) between two pairs of registers of the lane:
// (a, b) -> (a + b, a - b), a the element with the bit clear.  Packed into
// f32x2 instructions when both operand pairs are register pairs (2m, 2m+1).
template <int STYLE, int RP, int B, int K>
__device__ __forceinline__ void fwht_local_pairs(float (&x)[16]) {
  using S = HSlice<STYLE, RP>;
  constexpr int j0 = S::low_reg(B, K), j1 = S::low_reg(B, K + 1);
  constexpr int p0 = S::reg_at(S::off(j0) + B), p1 = S::reg_at(S::off(j1) + B);
  static_assert(j0 >= 0 && j1 >= 0 && p0 >= 0 && p1 >= 0, "Hadamard pair outside the lane");
  if constexpr (j0 % 2 == 0 && j1 == j0 + 1 && p0 % 2 == 0 && p1 == p0 + 1) {
    const float2 a = make_float2(x[j0], x[j1]);
    const float2 b = make_float2(x[p0], x[p1]);
    const float2 sum = __fadd2_rn(a, b);
    const float2 dif = __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);  // a - b, one rounding
    x[j0] = sum.x; x[j1] = sum.y;
    x[p0] = dif.x; x[p1] = dif.y;
  } else {
    const float a0 = x[j0], b0 = x[p0], a1 = x[j1], b1 = x[p1];
    x[j0] = __fadd_rn(a0, b0); x[p0] = __fsub_rn(a0, b0);
    x[j1] = __fadd_rn(a1, b1); x[p1] = __fsub_rn(a1, b1);
  }
}

// One butterfly stage over index bit H.  A lane bit pairs register j of lane
// l with register j of lane l ^ m: the lane with the bit clear keeps x + y,
// the other y - x, each one fp32 rounding of the same sum as the oracle's.
template <int STYLE, int RP, int H>
__device__ __forceinline__ void fwht_stage(float (&x)[16], int l) {
  using S = HSlice<STYLE, RP>;
  constexpr int B = 1 << H;
  if constexpr (B >= S::W && B < S::STRIDE) {
    constexpr int m = B / S::W;
    const float sg = (l & m) ? -1.0f : 1.0f;
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const float2 y = make_float2(__shfl_xor_sync(kFull, x[j], m),
                                   __shfl_xor_sync(kFull, x[j + 1], m));
      const float2 r = __ffma2_rn(sg2, make_float2(x[j], x[j + 1]), y);
      x[j] = r.x;
      x[j + 1] = r.y;
    }
  } else {
    fwht_local_pairs<STYLE, RP, B, 0>(x);
    fwht_local_pairs<STYLE, RP, B, 2>(x);
    fwht_local_pairs<STYLE, RP, B, 4>(x);
    fwht_local_pairs<STYLE, RP, B, 6>(x);
  }
}

// H_128 x (unnormalised): stages over index bits 0, 1, ..., 6 in that order.
// The 1/sqrt(128) is applied by the quantiser.
template <int STYLE, int RP>
__device__ __forceinline__ void fwht_hslice(float (&x)[16], int l) {
  fwht_stage<STYLE, RP, 0>(x, l);
  fwht_stage<STYLE, RP, 1>(x, l);
  fwht_stage<STYLE, RP, 2>(x, l);
  fwht_stage<STYLE, RP, 3>(x, l);
  fwht_stage<STYLE, RP, 4>(x, l);
  fwht_stage<STYLE, RP, 5>(x, l);
  fwht_stage<STYLE, RP, 6>(x, l);
}

// Scale exponent of the normalised vector y = fp32(x * 128^-0.5): rounding is
// monotonic, so max|y| = fp32(max|x| * 128^-0.5).
__device__ __forceinline__ int hadamard_exponent(const float (&x)[16]) {
  return exponent_of_amax(__fmul_rn(vector_amax(x), kHadamardScale));
}

// e4m3 codes of fp32(x * 128^-0.5) * 2^-e, as fp32(x * (128^-0.5 * 2^-e)):
// the factor is exact and scaling by a power of two commutes with rounding
// (values small enough for that to fail give code 0 either way).  Codes
// are packed chunk after chunk, element order inside each: byte c*W + i.
template <int STYLE, int RP>
__device__ __forceinline__ void quantize_hslice(const float (&x)[16], int e, uint32_t (&w)[4]) {
  using S = HSlice<STYLE, RP>;
  const float f = __fmul_rn(kHadamardScale, pow2f(-e));
  const float2 f2 = make_float2(f, f);
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; j += 2) {  // register order: packed multiplies
    const float2 t = __fmul2_rn(make_float2(x[j], x[j + 1]), f2);
    v[j] = t.x;
    v[j + 1] = t.y;
  }
#pragma unroll
  for (int n = 0; n < 16; n += 2) {  // n = c * W + i: byte n of the packed codes
    const int c0 = n / S::W, i0 = n % S::W, c1 = (n + 1) / S::W, i1 = (n + 1) % S::W;
    const uint32_t code = cvt_e4m3x2(v[S::reg(c0, i0)], v[S::reg(c1, i1)]);
    if ((n & 2) == 0) w[n / 4] = code;
    else w[n / 4] |= code << 16;
  }
}

// Store the packed codes to a 128-byte row whose start is ROW_ALIGN-aligned.
template <int STYLE, int RP, int ROW_ALIGN = 16>
__device__ __forceinline__ void store_hslice(uint8_t* row, int l, const uint32_t (&w)[4],
                                             bool pred = true) {
  using S = HSlice<STYLE, RP>;
  constexpr int A = gcd_pow2(S::W) < ROW_ALIGN ? gcd_pow2(S::W) : ROW_ALIGN;
#pragma unroll
  for (int c = 0; c < S::NCH; ++c) {
    uint8_t* p = row + c * S::STRIDE + S::W * l;
    if constexpr (S::W >= 4) {
      store_codes<S::W, A>(p, w + c * S::W / 4, pred);
    } else {
      const uint32_t v = w[(c * S::W) / 4] >> (8 * ((c * S::W) & 3));
      store_codes<S::W, A>(p, &v, pred);
    }
  }
}

template <int STYLE, int RP>
__device__ __forceinline__ void store_index_k_h(const CacheGeom& g, long long slot, int l,
                                                const uint32_t (&w)[4], int e, bool pred = true) {
  if (g.token_major) {
    uint8_t* row = g.cache + slot * (kD + 4);
    store_hslice<STYLE, RP, 4>(row, l, w, pred);
    store_f32(reinterpret_cast<float*>(row + kD), pow2f(e), pred && l == 0);
  } else {
    long long page, off;
    slot_page(g, slot, page, off);
    uint8_t* base = g.cache + page * g.page_bytes;
    store_hslice<STYLE, RP>(base + off * kD, l, w, pred);
    store_f32(reinterpret_cast<float*>(base + static_cast<long long>(g.page_size) * kD + 4 * off),
              pow2f(e), pred && l == 0);
  }
}

// gamma and beta of the lane's 16 elements, in register order, loaded all at
// once (for latency-bound callers: the loads overlap the LayerNorm sums).
// The rows are fp32 [128] in global memory (const float*) or staged in shared
// memory (a byte address).
template <int STYLE, int RP, class A>
__device__ __forceinline__ void load_affine_slice(A gamma, A beta, int l, float (&g)[16],
                                                  float (&b)[16]) {
  using S = Slice<STYLE, RP>;
  if constexpr (RP > 0) {
    if constexpr (S::NEOX) {
      load_f32_at<RP, S::ALIGN_A_F32>(gamma, RP * l, g);
      load_f32_at<RP, S::ALIGN_A_F32>(beta, RP * l, b);
      load_f32_at<RP, S::ALIGN_B_F32>(gamma, S::B_BASE + RP * l, g + RP);
      load_f32_at<RP, S::ALIGN_B_F32>(beta, S::B_BASE + RP * l, b + RP);
    } else {
      float tg[2 * RP], tb[2 * RP];
      load_f32_at<2 * RP, S::ALIGN_A_F32>(gamma, 2 * RP * l, tg);
      load_f32_at<2 * RP, S::ALIGN_A_F32>(beta, 2 * RP * l, tb);
#pragma unroll
      for (int j = 0; j < RP; ++j) {
        g[j] = tg[2 * j], g[RP + j] = tg[2 * j + 1];
        b[j] = tb[2 * j], b[RP + j] = tb[2 * j + 1];
      }
    }
  }
  if constexpr (S::NP > 0) {
    load_f32_at<S::NP, S::ALIGN_P_F32>(gamma, S::P_BASE + S::NP * l, g + 2 * RP);
    load_f32_at<S::NP, S::ALIGN_P_F32>(beta, S::P_BASE + S::NP * l, b + 2 * RP);
  }
}

template <int STYLE, int RP, class A>
__device__ __forceinline__ void load_affine_hslice(A gamma, A beta, int l, float (&g)[16],
                                                   float (&b)[16]) {
  using S = HSlice<STYLE, RP>;
  constexpr int PIECE = S::W < 4 ? S::W : 4;
#pragma unroll
  for (int c = 0; c < S::NCH; ++c)
#pragma unroll
    for (int i0 = 0; i0 < S::W; i0 += PIECE) {
      const int o = c * S::STRIDE + S::W * l + i0;
      float tg[PIECE], tb[PIECE];
      load_f32_at<PIECE, 4 * PIECE>(gamma, o, tg);
      load_f32_at<PIECE, 4 * PIECE>(beta, o, tb);
#pragma unroll
      for (int i = 0; i < PIECE; ++i) g[S::reg(c, i0 + i)] = tg[i], b[S::reg(c, i0 + i)] = tb[i];
    }
}

// y = x * rstd * gamma + beta with gamma and beta already in registers, two
// elements per packed instruction (each half rounds as the scalar form).
__device__ __forceinline__ void apply_affine(float (&x)[16], float rstd, const float (&g)[16],
                                             const float (&b)[16]) {
  const float2 r2 = make_float2(rstd, rstd);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 y = __ffma2_rn(__fmul2_rn(f2(x, j), r2), f2(g, j), f2(b, j));
    x[2 * j] = y.x;
    x[2 * j + 1] = y.y;
  }
}

// bf16 of x, round to nearest even (two at a time): lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------- staged LayerNorm parameters
//
// Element index of register r of lane l: the balanced slice, or the
// Hadamard layout.
template <bool HAD, int STYLE, int RP>
__device__ __forceinline__ int slice_elem(int l, int r) {
  if constexpr (HAD) {
    using S = HSlice<STYLE, RP>;
    return S::off(r) + S::W * l;
  } else {
    using S = Slice<STYLE, RP>;
    if (r >= 2 * RP) return S::P_BASE + S::NP * l + (r - 2 * RP);
    if (S::NEOX) return r < RP ? RP * l + r : S::B_BASE + RP * l + (r - RP);
    return 2 * RP * l + (r < RP ? 2 * r : 2 * (r - RP) + 1);
  }
}

// gamma and beta staged in shared memory in the lanes' register order, so
// that the affine step reads four registers' worth at once and runs packed in
// every layout: gamma's registers 4k .. 4k+3 of lane l at byte 16 (8k + l)
// (a quarter-warp's eight lanes read 128 contiguous bytes), beta 512 bytes on.
constexpr int kStagedGbBytes = 2 * 4 * kD;

// Thread `i` (0 .. 255) of a block stages value i of the layout above.
template <bool HAD, int STYLE, int RP>
__device__ __forceinline__ void stage_gb(float* dst, const float* gamma, const float* beta, int i) {
  const int j = i & 127;
  const int r = 4 * (j >> 5) + (j & 3);
  const int l = (j >> 2) & 7;
  dst[i] = __ldg((i < 128 ? gamma : beta) + slice_elem<HAD, STYLE, RP>(l, r));
}

// y = x * rstd * gamma + beta for M vectors of lane l, from the staged rows
// at shared byte address gb; each piece is read once for all M.
template <int M>
__device__ __forceinline__ void affine_staged(uint32_t gb, int l, float (&x)[M][16],
                                              const float (&rstd)[M]) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float g[4], b[4];
    load_f32_shared<4, 16>(gb + 16 * (8 * k + l), g);
    load_f32_shared<4, 16>(gb + 4 * kD + 16 * (8 * k + l), b);
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float2 r2 = make_float2(rstd[m], rstd[m]);
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        const float2 y = __ffma2_rn(__fmul2_rn(make_float2(x[m][4 * k + i], x[m][4 * k + i + 1]), r2),
                                    make_float2(g[i], g[i + 1]), make_float2(b[i], b[i + 1]));
        x[m][4 * k + i] = y.x;
        x[m][4 * k + i + 1] = y.y;
      }
    }
  }
}

// ---------------------------------------------------------------- four-lane Hadamard layout
//
// The Hadamard variant's query path in the prefill kernel gives each vector
// to four consecutive lanes: lane j of a group holds the HSlice slices of
// lanes 2j and 2j + 1 of the eight-lane layout as two halves x0 and x1, in
// those lanes' register order.  The butterfly stage on the eight-lane lane bit
// 0 pairs the two halves inside the lane, the stages on lane bits 1 and 2 are
// shuffles with the group's partners xor 1 and 2, the rest are register
// stages: the same operations on the same values in the same stage order, so
// the codes are those of the eight-lane layout, with a third fewer shuffles
// and half the per-vector scalar work per lane.

// The pair's bf16 row chunks (lane j of the group): eight-lane lanes 2j and
// 2j + 1 own neighbouring W-element pieces of every chunk.
template <int STYLE, int RP, class M>
__device__ __forceinline__ void load_hslice_pair(typename M::Addr row, int j, float (&x0)[16],
                                                 float (&x1)[16]) {
  using S = HSlice<STYLE, RP>;
#pragma unroll
  for (int c = 0; c < S::NCH; ++c) {
    float t[2 * S::W];
    load_bf16<M, 2 * S::W, gcd_pow2(4 * S::W)>(row + 2 * (c * S::STRIDE + 2 * S::W * j), t);
#pragma unroll
    for (int i = 0; i < S::W; ++i) x0[S::reg(c, i)] = t[i], x1[S::reg(c, i)] = t[S::W + i];
  }
}

// fwht_stage for the pair: B == W is the eight-lane lane bit 0 (the halves),
// 2W and 4W the group partners xor 1 and 2.
template <int STYLE, int RP, int H>
__device__ __forceinline__ void fwht_stage_pair(float (&x0)[16], float (&x1)[16], int j) {
  using S = HSlice<STYLE, RP>;
  constexpr int B = 1 << H;
  if constexpr (B == S::W) {
#pragma unroll
    for (int r = 0; r < 16; r += 2) {
      const float2 a = make_float2(x0[r], x0[r + 1]);
      const float2 b = make_float2(x1[r], x1[r + 1]);
      const float2 sum = __fadd2_rn(a, b);
      const float2 dif = __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);  // a - b, one rounding
      x0[r] = sum.x, x0[r + 1] = sum.y;
      x1[r] = dif.x, x1[r + 1] = dif.y;
    }
  } else if constexpr (B > S::W && B < S::STRIDE) {
    constexpr int m = B / S::W / 2;
    const float sg = (j & m) ? -1.0f : 1.0f;
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float (&x)[16] = h ? x1 : x0;
#pragma unroll
      for (int r = 0; r < 16; r += 2) {
        const float2 y = make_float2(__shfl_xor_sync(kFull, x[r], m),
                                     __shfl_xor_sync(kFull, x[r + 1], m));
        const float2 t = __ffma2_rn(sg2, make_float2(x[r], x[r + 1]), y);
        x[r] = t.x;
        x[r + 1] = t.y;
      }
    }
  } else {
    fwht_local_pairs<STYLE, RP, B, 0>(x0);
    fwht_local_pairs<STYLE, RP, B, 2>(x0);
    fwht_local_pairs<STYLE, RP, B, 4>(x0);
    fwht_local_pairs<STYLE, RP, B, 6>(x0);
    fwht_local_pairs<STYLE, RP, B, 0>(x1);
    fwht_local_pairs<STYLE, RP, B, 2>(x1);
    fwht_local_pairs<STYLE, RP, B, 4>(x1);
    fwht_local_pairs<STYLE, RP, B, 6>(x1);
  }
}

template <int STYLE, int RP>
__device__ __forceinline__ void fwht_pair(float (&x0)[16], float (&x1)[16], int j) {
  fwht_stage_pair<STYLE, RP, 0>(x0, x1, j);
  fwht_stage_pair<STYLE, RP, 1>(x0, x1, j);
  fwht_stage_pair<STYLE, RP, 2>(x0, x1, j);
  fwht_stage_pair<STYLE, RP, 3>(x0, x1, j);
  fwht_stage_pair<STYLE, RP, 4>(x0, x1, j);
  fwht_stage_pair<STYLE, RP, 5>(x0, x1, j);
  fwht_stage_pair<STYLE, RP, 6>(x0, x1, j);
}

// amax of the pair's vector over the group of four lanes.
__device__ __forceinline__ float pair_amax(const float (&x0)[16], const float (&x1)[16]) {
  float m = fmaxf(lane_amax(x0), lane_amax(x1));
  m = fmaxf(m, __shfl_xor_sync(kFull, m, 1));
  return fmaxf(m, __shfl_xor_sync(kFull, m, 2));
}

// Store the pair's codes (quantize_hslice's words of each half) to a
// 16-byte aligned 128-byte row: chunk c's two W-byte pieces are neighbours.
template <int STYLE, int RP>
__device__ __forceinline__ void store_hslice_pair(uint8_t* row, int j, const uint32_t (&w0)[4],
                                                  const uint32_t (&w1)[4], bool pred) {
  using S = HSlice<STYLE, RP>;
  constexpr int A = gcd_pow2(2 * S::W);
  uint32_t v[8];
  if constexpr (S::W % 4 == 0) {
#pragma unroll
    for (int c = 0; c < S::NCH; ++c) {
#pragma unroll
      for (int i = 0; i < S::W / 4; ++i)
        v[i] = w0[c * S::W / 4 + i], v[S::W / 4 + i] = w1[c * S::W / 4 + i];
      store_codes<2 * S::W, A>(row + c * S::STRIDE + 2 * S::W * j, v, pred);
    }
  } else {
    static_assert(S::W <= 2, "chunks of 1 or 2 codes");
    constexpr uint32_t mask = (1u << (8 * S::W)) - 1u;
#pragma unroll
    for (int c = 0; c < S::NCH; ++c) {
      const int sh = 8 * ((c * S::W) & 3);
      v[0] = ((w0[(c * S::W) / 4] >> sh) & mask) | (((w1[(c * S::W) / 4] >> sh) & mask) << (8 * S::W));
      store_codes<2 * S::W, A>(row + c * S::STRIDE + 2 * S::W * j, v, pred);
    }
  }
}

}  // namespace dsa_dev
