// DSA indexer Q/K prepare-and-store for GB300 (sm_103a): the fused kernels.
// The launcher and the C ABI are in dsa_prep.cu; the Hadamard variant's
// instantiations in dsa_hadamard.cu.
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
// Lane layout ("balanced slices").  A quarter-warp (8 lanes) owns one
// 128-vector; lane l holds 16 of its elements chosen so that every RoPE pair
// sits inside one lane and every lane rotates the same number of pairs.  With
// RP = rope_dim / 16 pairs per lane:
//   NeoX   a-members  RP elements at  RP*l           (pair partner i + r/2)
//          b-members  RP elements at  r/2 + RP*l
//   GPT-J  pairs      2*RP elements at 2*RP*l        (pairs (2i, 2i+1))
//   both   pass-through 16 - 2*RP elements at r + (16 - 2*RP)*l
// so the lane's frequencies are RP*l .. RP*l + RP - 1 in both styles, RoPE
// needs no shuffles, and it runs as packed f32x2 FMUL2/FFMA2.  A warp
// handles four vectors per instruction stream.
//
// Three kernels share that math:
//   * dsa_pipeline_kernel (large calls): persistent, warp-specialised.  Warp 0
//     moves each unit -- one token and up to 64 of its heads, plus the key on
//     the first chunk, or several whole tokens when they have few heads --
//     from HBM into a 4-stage shared-memory ring with cp.async.bulk copies
//     counted on mbarriers; 8 consumer warps compute from shared memory and
//     store to HBM.  Bytes in flight are set by the ring (up to ~200 KB per
//     SM), not by registers.
//   * dsa_direct_kernel (small calls, decode): one warp per four vectors,
//     every input in flight at once in two cp.async groups (the position and
//     slot first, so the cos/sin loads go out while the rows still travel),
//     warps spread over the SMs; the least latency per call.
//   * dsa_kstream_kernel (large k-only calls): persistent warps over
//     contiguous key ranges, two keys per quarter-warp, a cp.async ring per
//     warp one step ahead of the math.
// All come in a Hadamard variant (HAD = true) that rotates every vector by
// H_128 / sqrt(128) after RoPE; it uses the HSlice lane layout.
// Every mbarrier wait is bounded in time (DSA_DEVERR_TIMEOUT); nothing traps.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "dsa_common.cuh"
#include "dsa_prep.h"

namespace dsa_prep_impl {

using namespace dsa_dev;

// ---------------------------------------------------------------- parameters

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
  CacheGeom cg;
  int T;
  int H;
  int rope_dim;
  int cs_bytes;  // rope_dim / 2 * 4
  // pipeline kernel
  int HC;         // heads per unit
  int NC;         // units per token
  int TPU;        // tokens per unit: 1, 2 or 4 (more than 1 only when NC is 1)
  int tpu_shift;  // log2(TPU)
  long long units;
  int stage_bytes;
  int w_bulk;     // the chunk's weights can be bulk-copied (16-byte aligned)
  // stage layout (byte offsets): per-token headers at 0, then key rows,
  // cos rows, sin rows, gate weights, query rows
  int off_k, off_cos, off_sin, off_w, off_q;
  // multi-token units: k and w are the fused k|w projection (w = k + 128,
  // one row stride), so one copy brings a unit's key rows with their
  // weights; kw_row_b is the rows' stride in the stage (256 when not fused)
  int kw_fused;
  int kw_row_b;
  int cs_contig;  // cos/sin rows are packed (cs_stride == rope_dim / 2)
  // direct kernel
  int NQ;            // quads of heads per token
  long long q_warps;  // warps doing q quads
  long long k_warps;  // warps doing keys (four per warp)
  int early_rope;     // read positions and cos/sin before the PDL wait
  int l2_hints;       // prefetch the input rows into L2 before the PDL wait
  int test_withhold;  // DSA_FLAG_TEST_WITHHOLD_UNIT
  int* err;
};

// A bf16 row into the lane's 16 registers: the balanced slice, or the
// Hadamard layout (HSlice) when the variant rotates by H_128.
template <bool HAD, int STYLE, int RP, class M>
__device__ __forceinline__ void load_vec(typename M::Addr row, int l, float (&x)[16]) {
  if constexpr (HAD)
    load_hslice<STYLE, RP, M>(row, l, x);
  else
    load_slice<STYLE, RP, M>(row, l, x);
}

// Query vector: rotate (RoPE, then H_128 / sqrt(128) in the Hadamard
// variant), quantise, store codes; returns the scale exponent.
template <bool HAD, int STYLE, int RP>
__device__ __forceinline__ int q_slice(float (&x)[16], const Rot<RP>& r, uint8_t* out_row,
                                       int l, bool store) {
  if constexpr (RP > 0) rope_slice<RP>(x, r);
  if constexpr (HAD) {
    fwht_hslice<STYLE, RP>(x, l);
    const int e = hadamard_exponent(x);
    uint32_t w[4];
    quantize_hslice<STYLE, RP>(x, e, w);
    store_hslice<STYLE, RP>(out_row, l, w, store);
    return e;
  } else {
    const int e = ue8m0_exponent(x);
    uint32_t wa[4], wb[4], wp[4];
    quantize_slice<STYLE, RP>(x, e, wa, wb, wp);
    store_slice<STYLE, RP>(out_row, l, wa, wb, wp, store);
    return e;
  }
}

__device__ __forceinline__ void raise_error(const Params& p, int bit) {
  if (p.err) atomicOr(p.err, bit);
}

// Key vector: LayerNorm (mean, biased variance, eps inside the root), RoPE
// (then H_128 / sqrt(128) in the Hadamard variant), quantise, and store the
// codes and the scale into slot `slot` of the cache.  STAGED_AFFINE reads
// the lane's gamma and beta from shared memory (gamma at byte address
// gb_smem, beta 512 bytes on), all before the sums (for the latency-bound
// decode kernel, which stages them with its input row); otherwise they are
// loaded from global memory piece by piece after the sums, which keeps fewer
// registers live.
template <bool HAD, int STYLE, int RP, bool STAGED_AFFINE = false>
__device__ __forceinline__ void k_slice(const Params& p, float (&x)[16], const Rot<RP>& r,
                                        int l, bool real, bool pos_ok, long long slot,
                                        uint32_t gb_smem = 0) {
  float ga[16], be[16];  // used only with STAGED_AFFINE
  if constexpr (STAGED_AFFINE) {
    if constexpr (HAD)
      load_affine_hslice<STYLE, RP>(gb_smem, gb_smem + 4 * kD, l, ga, be);
    else
      load_affine_slice<STYLE, RP>(gb_smem, gb_smem + 4 * kD, l, ga, be);
  }
  const float rstd = ln_center(x, p.eps);
  if constexpr (STAGED_AFFINE)
    apply_affine(x, rstd, ga, be);
  else if constexpr (HAD)
    affine_hslice<STYLE, RP>(p.gamma, p.beta, l, x, rstd);
  else
    affine_slice<STYLE, RP>(p.gamma, p.beta, l, x, rstd);
  if constexpr (RP > 0) rope_slice<RP>(x, r);
  int e;
  uint32_t wa[4], wb[4], wp[4];
  if constexpr (HAD) {
    fwht_hslice<STYLE, RP>(x, l);
    e = hadamard_exponent(x);
    quantize_hslice<STYLE, RP>(x, e, wa);
  } else {
    e = ue8m0_exponent(x);
    quantize_slice<STYLE, RP>(x, e, wa, wb, wp);
  }

  // A key with a bad position or slot sets its error bit (the rare path)
  // and stores nothing; the stores carry their predicate, not a branch.
  const bool slot_ok = slot >= 0 && slot < p.cg.num_slots;
  if (real && l == 0 && !(pos_ok && slot_ok))
    raise_error(p, pos_ok ? DSA_DEVERR_SLOT : DSA_DEVERR_POSITION);
  const bool store = real && pos_ok && slot_ok;
  if constexpr (HAD)
    store_index_k_h<STYLE, RP>(p.cg, store ? slot : 0, l, wa, e, store);
  else
    store_index_k<STYLE, RP>(p.cg, store ? slot : 0, l, wa, wb, wp, e, store);
}

// Several keys at once, N per quarter-warp: the steps of k_slice with gamma
// and beta read from their staged copy in shared memory (stage_gb), each
// phase run for all N keys before the next so their dependent chains
// interleave, and each gamma/beta piece loaded once for all N.  Per key the
// arithmetic is k_slice's, so the bytes written are the same.  The caller
// has resolved each key's slot: `code` and `scale` are where its 128 codes
// and its scale go, `store` whether they are written, and `err` the error
// bit it raises (0 for none).
template <bool HAD, int STYLE, int RP, int N>
__device__ __forceinline__ void k_multi(const Params& p, float (&x)[N][16], const Rot<RP> (&r)[N],
                                        int l, uint8_t* const (&code)[N], float* const (&scale)[N],
                                        const bool (&store)[N], const int (&err)[N], uint32_t gb) {
  float rstd[N];
#pragma unroll
  for (int n = 0; n < N; ++n) rstd[n] = ln_center(x[n], p.eps);
  affine_staged<N>(gb, l, x, rstd);
  int e[N];
  uint32_t wa[N][4], wb[N][4], wp[N][4];
#pragma unroll
  for (int n = 0; n < N; ++n) {
    if constexpr (RP > 0) rope_slice<RP>(x[n], r[n]);
    if constexpr (HAD) {
      fwht_hslice<STYLE, RP>(x[n], l);
      e[n] = hadamard_exponent(x[n]);
      quantize_hslice<STYLE, RP>(x[n], e[n], wa[n]);
    } else {
      e[n] = ue8m0_exponent(x[n]);
      quantize_slice<STYLE, RP>(x[n], e[n], wa[n], wb[n], wp[n]);
    }
  }
#pragma unroll
  for (int n = 0; n < N; ++n) {
    if (err[n] && l == 0) raise_error(p, err[n]);
    // paged rows start on 16 bytes, token-major ones (132 bytes apart) on 4
    if (p.cg.token_major) {
      if constexpr (HAD)
        store_hslice<STYLE, RP, 4>(code[n], l, wa[n], store[n]);
      else
        store_slice<STYLE, RP, 4>(code[n], l, wa[n], wb[n], wp[n], store[n]);
    } else {
      if constexpr (HAD)
        store_hslice<STYLE, RP>(code[n], l, wa[n], store[n]);
      else
        store_slice<STYLE, RP>(code[n], l, wa[n], wb[n], wp[n], store[n]);
    }
    store_f32(scale[n], pow2f(e[n]), store[n] && l == 0);
  }
}

// ================================================================ direct kernel

constexpr int kDirectThreads = 256;
constexpr int kDirectWarps = kDirectThreads / 32;

// cos/sin of the lane's frequencies at row `row`, from global memory.
template <int RP>
__device__ __forceinline__ void load_rot_global(const Params& p, long long row, int l, Rot<RP>& r) {
  if constexpr (RP > 0) {
    load_f32_global<RP, Slice<0, RP>::ALIGN_CS>(p.cos_t + row * p.cs_stride + RP * l, r.c);
    load_f32_global<RP, Slice<0, RP>::ALIGN_CS>(p.sin_t + row * p.cs_stride + RP * l, r.s);
    finish_rot<RP>(r);
  }
}

// Position-dependent prologue of a token: its position, whether it is in
// range, and the lane's cos/sin values.
template <int RP>
__device__ __forceinline__ bool token_rot(const Params& p, long long t, int l, long long& pos,
                                          Rot<RP>& r) {
  pos = __ldg(p.pos + t);
  const bool pos_ok = pos >= 0 && pos < p.max_pos;
  load_rot_global<RP>(p, pos_ok ? pos : 0, l, r);
  return pos_ok;
}

// Direct kernel: one warp per four vectors (a quarter-warp each) -- four
// heads of one token, or four keys.  Key warps come first: the LayerNorm
// makes theirs the longest chain.  Latency rules here, so every
// input is in flight at once, in two cp.async groups per thread:
//   group 1: the token's position (and the key's slot), 8 bytes each;
//   group 2: the 256-byte input row (lane l copies bytes 16l and 128 + 16l)
//            and, for key warps, gamma and beta (1 KB, the whole warp).
// Waiting for group 1 alone, the quarter-warp reads the position and issues
// the cos/sin loads while the rows are still on their way; then it waits for
// group 2 and reads its slice from shared memory.
template <bool HAD, int STYLE, int RP>
__global__ void __launch_bounds__(kDirectThreads) dsa_direct_kernel(const Params p) {
  __shared__ __align__(16) unsigned char s_rows[kDirectWarps][4][2 * kD];
  __shared__ __align__(16) float s_gb[kDirectWarps][2][kD];
  __shared__ __align__(16) long long s_idx[kDirectWarps][4][2];
  const int lane = threadIdx.x & 31;
  const int wi = threadIdx.x >> 5;
  const int qtr = lane >> 3;
  const int l = lane & 7;
  // Work items are numbered down the columns of the grid (warp wi of CTA b is
  // item wi * gridDim + b), so the key warps, items 0 .. k_warps - 1, land on
  // different SMs; the launcher sizes CTAs so that small calls get one warp
  // per SM.
  const long long u = static_cast<long long>(wi) * gridDim.x + blockIdx.x;
  const bool is_q = u >= p.k_warps;
  const long long uq = u - p.k_warps;
  // q warp: four heads of one token; k warp: four keys, one per quarter-warp
  const long long t = is_q ? uq / p.NQ : 4 * u + qtr;
  const bool real = is_q || t < p.T;
  const long long tt = real ? t : 0;
  long long pos = 0;
  bool pos_ok = false;
  Rot<RP> r;
  // Let the next kernel of the stream get its CTAs resident now: it waits for
  // this grid's completion on its own griddepcontrol.wait.
  grid_launch_dependents();
  if (u >= p.q_warps + p.k_warps) return;  // warp-uniform
  const int v = is_q ? static_cast<int>(uq - t * p.NQ) * 4 + qtr : 0;
  const bool valid = v < p.H;
  // a quarter-warp past the last head re-reads head H-1 and stores nothing
  const int vl = valid ? v : p.H - 1;
  const unsigned char* row = reinterpret_cast<const unsigned char*>(
      is_q ? p.q + t * p.sq_t + static_cast<long long>(vl) * p.sq_h : p.k + tt * p.sk_t);
  // Under PDL what follows, up to the wait, runs while the previous kernel of
  // the stream finishes.  In a launch of one wave the quarter-warp's input
  // row (and, for keys, the LayerNorm parameters) start on their way into L2
  // (a hint, safe whoever writes them; see prefetch_l2_bulk).  The hints go
  // through the bulk-copy engine, which takes small requests slowly, so a
  // larger launch, or one without PDL, issues none.  With DSA_FLAG_PDL_EARLY_ROPE the
  // caller guarantees that positions, slots and the cos/sin cache are not
  // written by the previous kernel, so their two dependent round trips
  // overlap its tail as well.
  if (p.l2_hints && l == 0) {
    prefetch_l2_bulk(row, 2 * kD);
    if (is_q) {
      prefetch_l2(p.w + t * p.sw_t + vl);
    } else if (qtr == 0) {
      prefetch_l2_bulk(p.gamma, 4 * kD);
      prefetch_l2_bulk(p.beta, 4 * kD);
    }
  }
  if (p.early_rope) pos_ok = token_rot<RP>(p, tt, l, pos, r);
  grid_dependency_wait();

  const uint32_t s_idx_q = smem_u32(&s_idx[wi][qtr][0]);
  if (l == 0) {
    cp_async8(s_idx_q, p.pos + tt);
    if (!is_q) cp_async8(s_idx_q + 8, p.loc + tt);
  }
  cp_async_commit();
  const uint32_t s_row = smem_u32(&s_rows[wi][qtr][0]);
  cp_async16_cg(s_row + 16 * l, row + 16 * l);
  cp_async16_cg(s_row + 128 + 16 * l, row + 128 + 16 * l);
  const uint32_t s_gbw = smem_u32(&s_gb[wi][0][0]);
  if (!is_q) {
    cp_async16_ca(s_gbw + 16 * lane, p.gamma + 4 * lane);
    cp_async16_ca(s_gbw + 4 * kD + 16 * lane, p.beta + 4 * lane);
  }
  cp_async_commit();
  const float wv =
      is_q ? __uint_as_float(static_cast<uint32_t>(__ldg(p.w + t * p.sw_t + vl)) << 16) : 0.0f;
  cp_async_wait<1>();
  __syncwarp();
  if (!p.early_rope) {
    pos = s_idx[wi][qtr][0];
    pos_ok = pos >= 0 && pos < p.max_pos;
    load_rot_global<RP>(p, pos_ok ? pos : 0, l, r);
  }
  const long long slot = s_idx[wi][qtr][1];
  cp_async_wait<0>();
  __syncwarp();
  float x[16];
  load_vec<HAD, STYLE, RP, SharedMem>(s_row, l, x);
  if (is_q) {
    const long long orow = t * p.H + v;
    const int e = q_slice<HAD, STYLE, RP>(x, r, p.q_out + orow * kD, l, valid && pos_ok);
    store_f32_cs(p.w_out + orow, __fmul_rn(__fmul_rn(wv, pow2f(e)), p.fold),
                 valid && pos_ok && l == 0);
  } else {
    k_slice<HAD, STYLE, RP, true>(p, x, r, l, real, pos_ok, slot, s_gbw);
  }
}

// ================================================================ k-stream kernel

// Large k-only calls (the decode fast path's key store at prefill size):
// persistent CTAs whose warps each own a contiguous range of keys, walked in
// steps of kStreamKeys keys -- kStreamKPQ per quarter-warp, computed together
// by k_multi.  Keys come in batches of 32: when a batch becomes current, lane
// L resolves key L -- its position and slot, the offset of its cos/sin row,
// the cache bytes of its codes and its scale, and whether it is in range --
// into a per-warp table in shared memory (two batches deep), so no lane
// repeats that scalar work for its key.  Every input of a step -- the key
// rows and their cos/sin row slices -- is copied by cp.async into a stage of
// the warp's shared-memory ring kStreamStages - 1 steps ahead of the math;
// gamma and beta are staged once per CTA, in the lanes' register order
// (stage_gb), so the affine step runs packed in every layout.  Per key the
// arithmetic is that of the other kernels, so every kernel writes the same
// bytes.
constexpr int kStreamKPQ = 2;                 // keys per quarter-warp per step
constexpr int kStreamKeys = 4 * kStreamKPQ;   // keys per warp per step
constexpr int kStreamWarps = 8;
constexpr int kStreamThreads = 32 * kStreamWarps;
static_assert(kStreamThreads == 2 * kD, "stage_gb: one gamma or beta value a thread");
constexpr int kStreamStages = 2;              // the step computed and the one in flight
constexpr int kStreamCtas = 2;                // resident CTAs per SM the grid is sized for

// A key resolved for the k-stream kernel (one per lane of a batch).
struct StreamKey {
  long long cs_off;     // element offset of its cos/sin row
  long long code_off;   // cache byte offset of its 128 codes
  long long scale_off;  // cache byte offset of its scale
  int store;            // position and slot in range
  int err;              // the error bit it raises, or 0
};

// Stage layout (bytes): kStreamKeys key rows ROW bytes apart, then the cos
// and the sin slices of those keys (32 * RP bytes each: lane l's RP values at
// 4 * RP * l).  Key u of a step sits in quarter-warp u % 4.  ROW = 256 + 64
// puts the rows of quarter-warps 0 and 1 (and 2 and 3) in different banks, so
// an 8-byte slice load of the whole warp takes two shared-memory wavefronts,
// not four.
template <int RP>
struct StreamStage {
  static constexpr int ROW = 2 * kD + 64;
  static constexpr int CS = 32 * RP;  // cos (or sin) bytes of one key
  static constexpr int COS = kStreamKeys * ROW;
  static constexpr int SIN = COS + kStreamKeys * CS;
  static constexpr int BYTES = SIN + kStreamKeys * CS;
};

// per warp: the ring, then two batches of resolved keys
template <int RP>
__host__ __device__ constexpr int kstream_warp_bytes() {
  return kStreamStages * StreamStage<RP>::BYTES + 2 * 32 * static_cast<int>(sizeof(StreamKey));
}

template <int RP>
__host__ __device__ constexpr int kstream_smem() {
  return kStagedGbBytes + kStreamWarps * kstream_warp_bytes<RP>();
}

// cp.async of the lane's RP fp32 values (4 * RP bytes, aligned to that or 16).
template <int RP>
__device__ __forceinline__ void cp_async_rot(uint32_t dst, const float* src) {
  if constexpr (RP == 8) {
    cp_async16_ca(dst, src);
    cp_async16_ca(dst + 16, src + 4);
  } else if constexpr (RP == 4) {
    cp_async16_ca(dst, src);
  } else if constexpr (RP == 2) {
    cp_async8(dst, src);
  } else if constexpr (RP == 1) {
    cp_async4(dst, src);
  }
}

template <bool HAD, int STYLE, int RP>
__global__ void __launch_bounds__(kStreamThreads, kStreamCtas) dsa_kstream_kernel(const Params p) {
  using SS = StreamStage<RP>;
  constexpr int SPB = 32 / kStreamKeys;  // steps per batch of 32 keys
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int wi = threadIdx.x >> 5;
  const int qtr = lane >> 3;
  const int l = lane & 7;
  // this warp's keys: [k0, k1), steps [w G / W, (w + 1) G / W) of the G
  // steps, so the W warps' shares differ by one step at most
  const long long nw = static_cast<long long>(gridDim.x) * kStreamWarps;
  const long long steps = (static_cast<long long>(p.T) + kStreamKeys - 1) / kStreamKeys;
  const long long w = static_cast<long long>(blockIdx.x) * kStreamWarps + wi;
  long long s0, s1;  // (32-bit divisions while the products fit: shorter)
  if ((w + 1) * steps <= 0xffffffffLL) {
    s0 = static_cast<uint32_t>(w * steps) / static_cast<uint32_t>(nw);
    s1 = static_cast<uint32_t>((w + 1) * steps) / static_cast<uint32_t>(nw);
  } else {
    s0 = w * steps / nw;
    s1 = (w + 1) * steps / nw;
  }
  const long long k0 = kStreamKeys * s0;
  const long long k1 = min(static_cast<long long>(p.T), kStreamKeys * s1);
  const int n = k0 < k1 ? static_cast<int>((k1 - k0 + kStreamKeys - 1) / kStreamKeys) : 0;
  grid_launch_dependents();
  if (!p.early_rope) grid_dependency_wait();
  unsigned char* const wbase = smem + kStagedGbBytes + wi * kstream_warp_bytes<RP>();
  const uint32_t ring = smem_u32(wbase);
  StreamKey* const keys = reinterpret_cast<StreamKey*>(wbase + kStreamStages * SS::BYTES);

  // position and slot of key k0 + 32 b + lane (clamped into the range)
  auto batch = [&](int b, long long& pos, long long& slot) {
    long long t = k0 + 32LL * b + lane;
    t = t < k1 ? t : k1 - 1;
    pos = __ldg(p.pos + t);
    slot = __ldg(p.loc + t);
  };
  // Lane L resolves key L of batch b into the table (slot b % 2).
  auto resolve = [&](int b, long long pos, long long slot) {
    StreamKey kk;
    const bool pos_ok = pos >= 0 && pos < p.max_pos;
    const bool slot_ok = slot >= 0 && slot < p.cg.num_slots;
    kk.cs_off = (pos_ok ? pos : 0) * p.cs_stride;
    const long long sl = slot_ok ? slot : 0;
    if (p.cg.token_major) {
      kk.code_off = sl * (kD + 4);
      kk.scale_off = kk.code_off + kD;
    } else {
      long long page, off;
      slot_page(p.cg, sl, page, off);
      kk.code_off = page * p.cg.page_bytes + off * kD;
      kk.scale_off = page * p.cg.page_bytes + static_cast<long long>(p.cg.page_size) * kD + 4 * off;
    }
    const bool real = k0 + 32LL * b + lane < k1;
    kk.store = real && pos_ok && slot_ok;
    kk.err = !real || (pos_ok && slot_ok) ? 0 : pos_ok ? DSA_DEVERR_SLOT : DSA_DEVERR_POSITION;
    keys[32 * (b & 1) + lane] = kk;
  };
  long long pos0 = 0, slot0 = 0, nb_pos = 0, nb_slot = 0;
  if (n > 0) {  // the loads go out now; resolving batch 0 waits for them
    batch(0, pos0, slot0);
    batch(1, nb_pos, nb_slot);
  }
  // Copy step j into its stage, as two cp.async groups (empty past the warp's
  // last step).  Rows: for each of the step's keys u = 4h + q, lane l of
  // quarter-warp q copies bytes 16l and 128 + 16l of the key row.  Rotation:
  // each lane copies its own cos/sin values of the key.  The rows need no
  // position, so the first step's rows go out before the first batch of
  // positions has arrived.
  auto issue_rows = [&](int j) {
    if (j < n) {
      const uint32_t st = ring + (j % kStreamStages) * SS::BYTES;
#pragma unroll
      for (int h = 0; h < kStreamKPQ; ++h) {
        const int u = 4 * h + qtr;
        long long t = k0 + static_cast<long long>(kStreamKeys) * j + u;
        t = t < k1 ? t : k1 - 1;
        const unsigned char* row = reinterpret_cast<const unsigned char*>(p.k + t * p.sk_t);
        cp_async16_cg(st + SS::ROW * u + 16 * l, row + 16 * l);
        cp_async16_cg(st + SS::ROW * u + 128 + 16 * l, row + 128 + 16 * l);
      }
    }
    cp_async_commit();
  };
  auto issue_rot = [&](int j) {
    if (j < n) {
      if (j > 0 && j % SPB == 0) {  // the next batch of 32 keys becomes current
        resolve(j / SPB, nb_pos, nb_slot);
        __syncwarp();
        batch(j / SPB + 1, nb_pos, nb_slot);
      }
      if constexpr (RP > 0) {
        const uint32_t st = ring + (j % kStreamStages) * SS::BYTES;
        const StreamKey* kb = keys + 32 * ((j / SPB) & 1) + kStreamKeys * (j % SPB);
#pragma unroll
        for (int h = 0; h < kStreamKPQ; ++h) {
          const int u = 4 * h + qtr;
          const long long crow = kb[u].cs_off + RP * l;
          cp_async_rot<RP>(st + SS::COS + SS::CS * u + 4 * RP * l, p.cos_t + crow);
          cp_async_rot<RP>(st + SS::SIN + SS::CS * u + 4 * RP * l, p.sin_t + crow);
        }
      }
    }
    cp_async_commit();
  };

  // Groups in commit order: rows(0) and rot(0) (either first), rows(1),
  // rot(1), ...; with step j + 1 in flight, step j has landed once at most two
  // groups are pending.  (Issuing rows(1) before the first positions have
  // arrived measured slower: it delays the chain to the first cos/sin rows.)
  static_assert(kStreamStages == 2, "the wait counts below assume two stages");
  if (p.early_rope) {
    // DSA_FLAG_PDL_EARLY_ROPE: positions, slots and the cos/sin cache are not
    // the previous kernel's outputs, so the first cos/sin rows are on their
    // way before the wait; only the key rows wait for it.
    if (n > 0) {
      resolve(0, pos0, slot0);
      __syncwarp();
    }
    issue_rot(0);
    grid_dependency_wait();
    issue_rows(0);
  } else {
    issue_rows(0);  // before the first positions are needed
    if (n > 0) {
      resolve(0, pos0, slot0);
      __syncwarp();
    }
    issue_rot(0);
  }
  // gamma and beta, once per CTA, in the lanes' register order
  stage_gb<HAD, STYLE, RP>(reinterpret_cast<float*>(smem), p.gamma, p.beta, threadIdx.x);
  __syncthreads();
  for (int j = 0; j < n; ++j) {
    // refill the stage freed by step j - 1, then wait for step j
    issue_rows(j + 1);
    issue_rot(j + 1);
    cp_async_wait<2>();
    __syncwarp();
    const uint32_t st = ring + (j % kStreamStages) * SS::BYTES;
    const StreamKey* kb = keys + 32 * ((j / SPB) & 1) + kStreamKeys * (j % SPB);
    float x[kStreamKPQ][16];
    Rot<RP> r[kStreamKPQ];
    uint8_t* code[kStreamKPQ];
    float* scale[kStreamKPQ];
    bool store[kStreamKPQ];
    int err[kStreamKPQ];
#pragma unroll
    for (int h = 0; h < kStreamKPQ; ++h) {
      const int u = 4 * h + qtr;
      code[h] = p.cg.cache + kb[u].code_off;
      scale[h] = reinterpret_cast<float*>(p.cg.cache + kb[u].scale_off);
      store[h] = kb[u].store != 0;
      err[h] = kb[u].err;
      load_vec<HAD, STYLE, RP, SharedMem>(st + SS::ROW * u, l, x[h]);
      if constexpr (RP > 0) {
        load_f32_shared<RP, Slice<0, RP>::ALIGN_CS>(st + SS::COS + SS::CS * u + 4 * RP * l, r[h].c);
        load_f32_shared<RP, Slice<0, RP>::ALIGN_CS>(st + SS::SIN + SS::CS * u + 4 * RP * l, r[h].s);
        finish_rot<RP>(r[h]);
      }
    }
    k_multi<HAD, STYLE, RP, kStreamKPQ>(p, x, r, l, code, scale, store, err, smem_u32(smem));
    __syncwarp();  // every lane is done with this stage before it is refilled
  }
}

// ================================================================ pipeline kernel

constexpr int kHCMax = 64;        // heads per unit at most
constexpr int kTPUMax = 4;        // tokens per unit at most
constexpr int kStages = 4;        // shared-memory ring depth
constexpr int kConsumers = 8;     // consumer warps per CTA
constexpr int kPipeThreads = 32 * (1 + kConsumers);
// Resident CTAs per SM the pipeline kernels are compiled for (registers per
// thread <= 65536 / (kPipeThreads * this)); the launcher sizes grids to match.
constexpr int kPipeCtas = 3;
// The Hadamard variant's four-lane query path holds two slices a lane: it
// runs spill-free at 2 CTAs per SM (up to 113 registers), which measured
// faster than 3 with spills (48.5 against 53.3 us at T=8192, H=64).
constexpr int kPipeCtasHad = 2;
constexpr int kBarrierBytes = 128;  // full[kStages], empty[kStages], abort flag
// stage layout of one-token units (byte offsets from the stage base)
constexpr int kOffK = 64;      // key row, 256 B (after the StageHeader)
constexpr int kOffCos = 320;   // cos row, rope_dim/2 floats (<= 256 B)
constexpr int kOffSin = 576;   // sin row
constexpr int kOffW = 832;     // gate weights of the chunk, HC bf16 (<= 128 B)
constexpr int kOffQ = 1024;    // HC query rows of 256 B
// the largest stage: headers, key rows (<= 512 B each with fused weights),
// cos and sin rows (<= 256 B each) and
// weights of kTPUMax tokens, then query rows of at most kHCMax heads in all
constexpr int kMaxStageBytes = 32 * kTPUMax + 512 * kTPUMax + 2 * 256 * kTPUMax + 128 + 256 * kHCMax;

// Per-token header of a stage.
struct StageHeader {
  long long pos;
  long long slot;
  int pos_ok;
  int pad[3];
};

// Producer warp for units of one token (the layout kOff*): lane 0 fills the
// ring; all lanes prefetch (position, slot) for the next 32 units of this CTA.  The position-independent copies (query
// rows, key row, weights) go out before the position is known.
static __device__ void producer_single(const Params& p, unsigned char* ring, uint32_t full0, uint32_t empty0,
                         volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  long long my_pos = 0, my_slot = 0;
  // (token, chunk) of unit u, advanced incrementally as u steps by gridDim.x
  const int dt = static_cast<int>(gridDim.x) / p.NC;
  const int dc = static_cast<int>(gridDim.x) - dt * p.NC;
  int t = static_cast<int>(blockIdx.x) / p.NC;
  int c = static_cast<int>(blockIdx.x) - t * p.NC;
  int i = 0;
  for (long long u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
    if (i > 0) {
      t += dt;
      c += dc;
      if (c >= p.NC) c -= p.NC, ++t;
    }
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
    int stop = 0;
    const int s = i % kStages;
    const uint32_t full = full0 + 8 * s;
    unsigned char* st = ring + static_cast<size_t>(s) * p.stage_bytes;
    const uint32_t sts = smem_u32(st);
    // test hook: CTA 0 never fills its first stage (see DSA_FLAG_TEST_WITHHOLD_UNIT)
    const bool withhold = p.test_withhold && blockIdx.x == 0 && i == 0;
    if (lane == 0) {
      const uint32_t ph = (i / kStages) & 1;
      if (i >= kStages && !mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag)) {
        stop = 1;
      } else if (!withhold) {
        const int h0 = c * p.HC;
        const int n = min(p.HC, p.H - h0);
        const uint32_t early = static_cast<uint32_t>(n) * 256u + (c == 0 ? 256u : 0u) +
                               (p.w_bulk ? 2u * n : 0u);
        if (early) mbar_expect_tx(full, early);
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
    const long long pos = __shfl_sync(kFull, my_pos, j);
    const long long slot = __shfl_sync(kFull, my_slot, j);
    if (lane == 0 && !withhold) {
      const bool pos_ok = pos >= 0 && pos < p.max_pos;
      const long long row = pos_ok ? pos : 0;
      StageHeader* hd = reinterpret_cast<StageHeader*>(st);
      hd->pos = pos;
      hd->slot = slot;
      hd->pos_ok = pos_ok ? 1 : 0;
      if (p.rope_dim) {
        mbar_arrive_expect_tx(full, 2u * p.cs_bytes);
        bulk_g2s(sts + kOffCos, p.cos_t + row * p.cs_stride, p.cs_bytes, full);
        bulk_g2s(sts + kOffSin, p.sin_t + row * p.cs_stride, p.cs_bytes, full);
      } else {
        mbar_arrive(full);
      }
    }
    __syncwarp();
  }
  // Stay until the copies of the last (up to kStages) units have landed, so
  // the CTA never exits with a bulk copy still writing its shared memory.
  if (lane == 0) {
    volatile int never = 0;
    for (int d = (i > kStages ? i - kStages : 0); d < i; ++d)
      mbar_wait(full0 + 8 * (d % kStages), (d / kStages) & 1, &never);
  }
}

// Producer warp for units of TPU > 1 tokens (the layout p.off_*).  A unit is
// TPU tokens (t0, t0 + 1, ...) and heads
// [h0, h0 + n) of each; lane 0 fills the ring, and all lanes prefetch the
// (position, slot) of the tokens of this CTA's next 32 / TPU units (lane L:
// token L % TPU of the (L / TPU)-th unit on).  The position-independent copies
// (query rows, key rows, weights) go out before the positions are known.
static __device__ void producer_multi(const Params& p, unsigned char* ring, uint32_t full0, uint32_t empty0,
                         volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const int ub_mask = (32 >> p.tpu_shift) - 1;  // units per prefetch batch, less one
  long long my_pos = 0, my_slot = 0;
  // (token unit, chunk) of unit u, advanced incrementally as u steps by gridDim.x
  const int dt = static_cast<int>(gridDim.x) / p.NC;
  const int dc = static_cast<int>(gridDim.x) - dt * p.NC;
  int t = static_cast<int>(blockIdx.x) / p.NC;
  int c = static_cast<int>(blockIdx.x) - t * p.NC;
  int i = 0;
  for (long long u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
    if (i > 0) {
      t += dt;
      c += dc;
      if (c >= p.NC) c -= p.NC, ++t;
    }
    const int j = i & ub_mask;
    if (j == 0) {
      const long long uu = u + static_cast<long long>(lane >> p.tpu_shift) * gridDim.x;
      my_pos = 0;
      my_slot = 0;
      if (uu < p.units) {
        const long long tu = uu / p.NC;
        const long long tt = (tu << p.tpu_shift) + (lane & (p.TPU - 1));
        if (tt < p.T) {
          my_pos = __ldg(p.pos + tt);
          if (uu - tu * p.NC == 0) my_slot = __ldg(p.loc + tt);
        }
      }
    }
    const long long t0 = static_cast<long long>(t) << p.tpu_shift;
    const int nt = static_cast<int>(min(static_cast<long long>(p.TPU), p.T - t0));
    int stop = 0;
    const int s = i % kStages;
    const uint32_t full = full0 + 8 * s;
    unsigned char* st = ring + static_cast<size_t>(s) * p.stage_bytes;
    const uint32_t sts = smem_u32(st);
    // test hook: CTA 0 never fills its first stage (see DSA_FLAG_TEST_WITHHOLD_UNIT)
    const bool withhold = p.test_withhold && blockIdx.x == 0 && i == 0;
    if (lane == 0) {
      const uint32_t ph = (i / kStages) & 1;
      if (i >= kStages && !mbar_wait(empty0 + 8 * s, ph ^ 1, abort_flag)) {
        stop = 1;
      } else if (!withhold) {
        const int h0 = c * p.HC;
        const int n = min(p.HC, p.H - h0);
        // query rows; key rows (with their weights when fused); weights
        const uint32_t kw_bytes = p.kw_fused ? static_cast<uint32_t>((nt - 1) * p.kw_row_b + 256 + 2 * n)
                                             : 256u * nt + (p.w_bulk ? 2u * n * nt : 0u);
        const uint32_t early = static_cast<uint32_t>(nt * n) * 256u + (c == 0 ? kw_bytes : 0u);
        if (early) mbar_expect_tx(full, early);
        if (n > 0) {
          const uint16_t* qsrc = p.q + t0 * p.sq_t + static_cast<long long>(h0) * p.sq_h;
          if (p.sq_h == kD && (nt == 1 || p.sq_t == static_cast<long long>(n) * kD)) {
            bulk_g2s(sts + p.off_q, qsrc, static_cast<uint32_t>(nt * n) * 256u, full);
          } else if (p.sq_h == kD) {
            for (int k = 0; k < nt; ++k)
              bulk_g2s(sts + p.off_q + 256 * n * k, qsrc + k * p.sq_t,
                       static_cast<uint32_t>(n) * 256u, full);
          } else {
            for (int k = 0; k < nt; ++k)
              for (int h = 0; h < n; ++h)
                bulk_g2s(sts + p.off_q + 256 * (n * k + h), qsrc + k * p.sq_t + h * p.sq_h, 256u,
                         full);
          }
          if (p.w_bulk && !p.kw_fused) {
            const uint16_t* wsrc = p.w + t0 * p.sw_t + h0;
            if (nt == 1 || p.sw_t == n)
              bulk_g2s(sts + p.off_w, wsrc, static_cast<uint32_t>(nt * n) * 2u, full);
            else
              for (int k = 0; k < nt; ++k)
                bulk_g2s(sts + p.off_w + 2 * n * k, wsrc + k * p.sw_t, 2u * n, full);
          }
        }
        if (c == 0) {
          if (p.kw_fused)  // rows t0.. of the k|w buffer: keys, weights and what lies between
            bulk_g2s(sts + p.off_k, p.k + t0 * p.sk_t, kw_bytes, full);
          else if (nt == 1 || p.sk_t == kD)
            bulk_g2s(sts + p.off_k, p.k + t0 * p.sk_t, static_cast<uint32_t>(nt) * 256u, full);
          else
            for (int k = 0; k < nt; ++k)
              bulk_g2s(sts + p.off_k + 256 * k, p.k + (t0 + k) * p.sk_t, 256u, full);
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
    long long pos[kTPUMax], slot[kTPUMax];
#pragma unroll
    for (int k = 0; k < kTPUMax; ++k) {
      if (k < p.TPU) {  // uniform across the warp
        const int src = (j << p.tpu_shift) + k;
        pos[k] = __shfl_sync(kFull, my_pos, src);
        slot[k] = __shfl_sync(kFull, my_slot, src);
      }
    }
    if (lane == 0 && !withhold) {
      if (p.rope_dim)
        mbar_arrive_expect_tx(full, 2u * p.cs_bytes * nt);
      // consecutive in-range positions over packed rows: one copy each of
      // the unit's cos rows and sin rows (prefill), else one per token
      bool consec = p.cs_contig != 0;
#pragma unroll
      for (int k = 0; k < kTPUMax; ++k) {
        if (k < nt) {
          const bool pos_ok = pos[k] >= 0 && pos[k] < p.max_pos;
          consec = consec && pos_ok && pos[k] == pos[0] + k;
          StageHeader* hd = reinterpret_cast<StageHeader*>(st) + k;
          hd->pos = pos[k];
          hd->slot = slot[k];
          hd->pos_ok = pos_ok ? 1 : 0;
        }
      }
      if (p.rope_dim) {
        if (consec) {
          const uint32_t bytes = static_cast<uint32_t>(p.cs_bytes * nt);
          bulk_g2s(sts + p.off_cos, p.cos_t + pos[0] * p.cs_stride, bytes, full);
          bulk_g2s(sts + p.off_sin, p.sin_t + pos[0] * p.cs_stride, bytes, full);
        } else {
#pragma unroll
          for (int k = 0; k < kTPUMax; ++k) {
            if (k < nt) {
              const long long row = (pos[k] >= 0 && pos[k] < p.max_pos) ? pos[k] : 0;
              bulk_g2s(sts + p.off_cos + p.cs_bytes * k, p.cos_t + row * p.cs_stride, p.cs_bytes, full);
              bulk_g2s(sts + p.off_sin + p.cs_bytes * k, p.sin_t + row * p.cs_stride, p.cs_bytes, full);
            }
          }
        }
      } else {
        mbar_arrive(full);
      }
    }
    __syncwarp();
  }
  // Stay until the copies of the last (up to kStages) units have landed, so
  // the CTA never exits with a bulk copy still writing its shared memory.
  if (lane == 0) {
    volatile int never = 0;
    for (int d = (i > kStages ? i - kStages : 0); d < i; ++d)
      mbar_wait(full0 + 8 * (d % kStages), (d / kStages) & 1, &never);
  }
}

// Consumer warp for units of one token (the layout kOff*).
template <bool HAD, int STYLE, int RP>
__device__ void consumer_single(const Params& p, int cw, unsigned char* ring, uint32_t full0,
                         uint32_t empty0, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const int qtr = lane >> 3;
  const int l = lane & 7;
  const int dt = static_cast<int>(gridDim.x) / p.NC;
  const int dc = static_cast<int>(gridDim.x) - dt * p.NC;
  int t = static_cast<int>(blockIdx.x) / p.NC;
  int c = static_cast<int>(blockIdx.x) - t * p.NC;
  int i = 0;
  for (long long u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
    if (i > 0) {
      t += dt;
      c += dc;
      if (c >= p.NC) c -= p.NC, ++t;
    }
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
    const StageHeader* hd = reinterpret_cast<const StageHeader*>(st);
    const bool pos_ok = hd->pos_ok != 0;
    const int h0 = c * p.HC;
    const int n = min(p.HC, p.H - h0);

    // the eight-lane rotation operands (the Hadamard variant's queries use
    // their own, and its key loads these when it has one)
    Rot<RP> r;
    auto load_rot8 = [&]() {
      if constexpr (RP > 0) {
        load_f32_shared<RP, Slice<0, RP>::ALIGN_CS>(sts + kOffCos + 4 * RP * l, r.c);
        load_f32_shared<RP, Slice<0, RP>::ALIGN_CS>(sts + kOffSin + 4 * RP * l, r.s);
        finish_rot<RP>(r);
      }
    };
    if constexpr (!HAD) load_rot8();
    // Per-unit bases, so a head costs a few 32-bit offsets: its output rows,
    // and its gate weights -- in the stage when they rode the bulk copy, else
    // in global memory; one generic pointer serves both.
    const long long orow0 = t * p.H + h0;
    uint8_t* const q_out = p.q_out + orow0 * kD;
    float* const w_out = p.w_out + orow0;
    const uint16_t* const w_src =
        p.w_bulk ? reinterpret_cast<const uint16_t*>(st + kOffW) : p.w + t * p.sw_t + h0;
    const bool w_lane = pos_ok && l == 0;
    // One query head of the chunk for this quarter-warp: head v (a quarter-
    // warp past the chunk's last head re-reads it and stores nothing).
    auto q_head = [&](int v, float (&x)[16]) {
      const bool valid = v < n;
      const int vl = valid ? v : n - 1;
      load_vec<HAD, STYLE, RP, SharedMem>(sts + kOffQ + 256 * vl, l, x);
      const float wv = __uint_as_float(static_cast<uint32_t>(w_src[vl]) << 16);
      const int e = q_slice<HAD, STYLE, RP>(x, r, q_out + v * kD, l, valid && pos_ok);
      store_f32_cs(w_out + v, __fmul_rn(__fmul_rn(wv, pow2f(e)), p.fold), valid && w_lane);
    };
    if constexpr (HAD) {
      // query heads in the four-lane layout: lanes 4g .. 4g + 3 take head
      // 8 qd + g, warp cw the head octets cw, cw + kConsumers, ...
      const int g = lane >> 2, jj = lane & 3;
      Rot<RP> r0, r1;  // frequencies 2 RP jj .. 2 RP jj + 2 RP - 1
      if constexpr (RP > 0) {
        float cs[2 * RP], sn[2 * RP];
        load_f32_shared<2 * RP, gcd_pow2(8 * RP)>(sts + kOffCos + 8 * RP * jj, cs);
        load_f32_shared<2 * RP, gcd_pow2(8 * RP)>(sts + kOffSin + 8 * RP * jj, sn);
#pragma unroll
        for (int i = 0; i < RP; ++i) {
          r0.c[i] = cs[i], r1.c[i] = cs[RP + i];
          r0.s[i] = sn[i], r1.s[i] = sn[RP + i];
        }
        finish_rot<RP>(r0);
        finish_rot<RP>(r1);
      }
      for (int qd = cw; 8 * qd < n; qd += kConsumers) {
        const int v = 8 * qd + g;
        const bool valid = v < n;
        const int vl = valid ? v : n - 1;
        float x0[16], x1[16];
        load_hslice_pair<STYLE, RP, SharedMem>(sts + kOffQ + 256 * vl, jj, x0, x1);
        const float wv = __uint_as_float(static_cast<uint32_t>(w_src[vl]) << 16);
        if constexpr (RP > 0) {
          rope_slice<RP>(x0, r0);
          rope_slice<RP>(x1, r1);
        }
        fwht_pair<STYLE, RP>(x0, x1, jj);
        const int e = exponent_of_amax(__fmul_rn(pair_amax(x0, x1), kHadamardScale));
        uint32_t w0[4], w1[4];
        quantize_hslice<STYLE, RP>(x0, e, w0);
        quantize_hslice<STYLE, RP>(x1, e, w1);
        store_hslice_pair<STYLE, RP>(q_out + v * kD, jj, w0, w1, valid && pos_ok);
        store_f32_cs(w_out + v, __fmul_rn(__fmul_rn(wv, pow2f(e)), p.fold),
                     valid && pos_ok && jj == 0);
      }
    } else {
      // query heads: warp cw takes head quads cw, cw + kConsumers, ...
      for (int qd = cw; 4 * qd < n; qd += kConsumers) {
        float x[16];
        q_head(4 * qd + qtr, x);
      }
    }
    // the key rides with chunk 0; the warp that takes it rotates per unit
    if (c == 0 && cw == i % kConsumers) {
      if constexpr (HAD) load_rot8();
      float x[16];
      load_vec<HAD, STYLE, RP, SharedMem>(sts + kOffK, l, x);
      k_slice<HAD, STYLE, RP>(p, x, r, l, qtr == 0, pos_ok, hd->slot);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
}

// The rotation operands of token k of a stage.
template <int RP>
__device__ __forceinline__ void stage_rot(const Params& p, uint32_t sts, int k, int l, Rot<RP>& r) {
  if constexpr (RP > 0) {
    load_f32_shared<RP, Slice<0, RP>::ALIGN_CS>(sts + p.off_cos + p.cs_bytes * k + 4 * RP * l, r.c);
    load_f32_shared<RP, Slice<0, RP>::ALIGN_CS>(sts + p.off_sin + p.cs_bytes * k + 4 * RP * l, r.s);
    finish_rot<RP>(r);
  }
}

template <bool HAD, int STYLE, int RP>
__device__ void consumer_multi(const Params& p, int cw, unsigned char* ring, uint32_t full0,
                         uint32_t empty0, volatile int* abort_flag) {
  const int lane = threadIdx.x & 31;
  const int qtr = lane >> 3;
  const int l = lane & 7;
  const int dt = static_cast<int>(gridDim.x) / p.NC;
  const int dc = static_cast<int>(gridDim.x) - dt * p.NC;
  int t = static_cast<int>(blockIdx.x) / p.NC;
  int c = static_cast<int>(blockIdx.x) - t * p.NC;
  int i = 0;
  for (long long u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
    if (i > 0) {
      t += dt;
      c += dc;
      if (c >= p.NC) c -= p.NC, ++t;
    }
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
    const StageHeader* hd = reinterpret_cast<const StageHeader*>(st);
    const long long t0 = static_cast<long long>(t) << p.tpu_shift;
    const int nt = static_cast<int>(min(static_cast<long long>(p.TPU), p.T - t0));
    const int h0 = c * p.HC;
    const int n = min(p.HC, p.H - h0);
    const int nq = (n + 3) >> 2;  // head quads per token

    // One query head for this quarter-warp: head v of a token whose output
    // rows start at q_out / w_out, whose query rows start at q_sts in the
    // stage and whose gate weights start at w_src -- in the stage when they
    // rode the bulk copy, else in global memory; one generic pointer serves
    // both.  A quarter-warp past the chunk's last head re-reads it and stores
    // nothing.
    auto q_head = [&](int v, uint32_t q_sts, const uint16_t* w_src, uint8_t* q_out, float* w_out,
                      const Rot<RP>& r, bool pos_ok) {
      const bool valid = v < n;
      const int vl = valid ? v : n - 1;
      float x[16];
      load_vec<HAD, STYLE, RP, SharedMem>(q_sts + 256 * vl, l, x);
      const float wv = __uint_as_float(static_cast<uint32_t>(w_src[vl]) << 16);
      const int e = q_slice<HAD, STYLE, RP>(x, r, q_out + v * kD, l, valid && pos_ok);
      store_f32_cs(w_out + v, __fmul_rn(__fmul_rn(wv, pow2f(e)), p.fold),
                   valid && pos_ok && l == 0);
    };
    // token k's weights: beside its key row (fused k|w), in the weights
    // region, or in global memory
    auto w_base = [&](int k) {
      return p.kw_fused ? reinterpret_cast<const uint16_t*>(st + p.off_k + p.kw_row_b * k + 2 * kD)
             : p.w_bulk ? reinterpret_cast<const uint16_t*>(st + p.off_w) + n * k
                        : p.w + (t0 + k) * p.sw_t + h0;
    };
    if (nt == 1) {
      // one token: its rotation and bases once for the whole unit
      Rot<RP> r;
      stage_rot<RP>(p, sts, 0, l, r);
      const bool pos_ok = hd[0].pos_ok != 0;
      const long long orow0 = t0 * p.H + h0;
      uint8_t* const q_out = p.q_out + orow0 * kD;
      float* const w_out = p.w_out + orow0;
      const uint16_t* const w_src = w_base(0);
      const uint32_t q_sts = sts + p.off_q;
      // query heads: warp cw takes head quads cw, cw + kConsumers, ...
      for (int qd = cw; qd < nq; qd += kConsumers)
        q_head(4 * qd + qtr, q_sts, w_src, q_out, w_out, r, pos_ok);
      // the key rides with chunk 0; the warp that takes it rotates per unit
      if (c == 0 && cw == i % kConsumers) {
        float x[16];
        load_vec<HAD, STYLE, RP, SharedMem>(sts + p.off_k, l, x);
        k_slice<HAD, STYLE, RP>(p, x, r, l, qtr == 0, pos_ok, hd[0].slot);
      }
    } else {
      // several tokens: warp cw takes token cw % TPU and its head quads
      // cw / TPU, cw / TPU + 8 / TPU, ...; the token's rotation and bases once
      const int k = cw & (p.TPU - 1);
      if (k < nt) {
        Rot<RP> r;
        stage_rot<RP>(p, sts, k, l, r);
        const bool pos_ok = hd[k].pos_ok != 0;
        const long long orow0 = (t0 + k) * p.H + h0;
        uint8_t* const q_out = p.q_out + orow0 * kD;
        float* const w_out = p.w_out + orow0;
        const uint16_t* const w_src = w_base(k);
        const uint32_t q_sts = sts + p.off_q + 256 * n * k;
        for (int qd = cw >> p.tpu_shift; qd < nq; qd += kConsumers >> p.tpu_shift)
          q_head(4 * qd + qtr, q_sts, w_src, q_out, w_out, r, pos_ok);
      }
      // the unit's keys (chunk 0 only): quarter-warp k of one warp takes key k
      if (c == 0 && cw == i % kConsumers) {
        const int k = min(qtr, nt - 1);
        Rot<RP> r;
        stage_rot<RP>(p, sts, k, l, r);
        float x[16];
        load_vec<HAD, STYLE, RP, SharedMem>(sts + p.off_k + p.kw_row_b * k, l, x);
        k_slice<HAD, STYLE, RP>(p, x, r, l, qtr < nt, hd[k].pos_ok != 0, hd[k].slot);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }
}

// MULTI: units of several tokens (Params::TPU > 1), else of one token; the
// two are separate kernels so each gets its own register allocation.
template <bool HAD, int STYLE, int RP, bool MULTI>
__global__ void __launch_bounds__(kPipeThreads, HAD ? kPipeCtasHad : kPipeCtas)
    dsa_pipeline_kernel(const Params p) {
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

  // one-token units keep their own lean loops (fixed layout, no token
  // bookkeeping); units of several tokens take the general ones
  const int warp = threadIdx.x >> 5;
  if constexpr (!MULTI) {
    if (warp == 0)
      producer_single(p, ring, full0, empty0, abort_flag);
    else
      consumer_single<HAD, STYLE, RP>(p, warp - 1, ring, full0, empty0, abort_flag);
  } else {
    if (warp == 0)
      producer_multi(p, ring, full0, empty0, abort_flag);
    else
      consumer_multi<HAD, STYLE, RP>(p, warp - 1, ring, full0, empty0, abort_flag);
  }
}

// ---------------------------------------------------------------- kernel tables

using KernelFn = void (*)(Params);

template <bool HAD, int STYLE, int RP, bool MULTI = false>
constexpr KernelFn pipeline_fn() { return dsa_pipeline_kernel<HAD, STYLE, RP, MULTI>; }
template <bool HAD, int STYLE, int RP>
constexpr KernelFn direct_fn() { return dsa_direct_kernel<HAD, STYLE, RP>; }
template <bool HAD, int STYLE, int RP>
constexpr KernelFn kstream_fn() { return dsa_kstream_kernel<HAD, STYLE, RP>; }

// The Hadamard variant's kernels, [rope_style][rope_dim / 16 -> 0, 1, 2, 4, 8];
// instantiated in their own translation unit.
extern const KernelFn kPipelineHad[2][5];
extern const KernelFn kPipelineMultiHad[2][5];
extern const KernelFn kDirectHad[2][5];
extern const KernelFn kStreamHad[2][5];

}  // namespace dsa_prep_impl
