/*
 * dsa_prep.h -- C ABI of the DSA indexer Q/K prepare-and-store for GB300
 * (sm_103a).
 *
 * What the calls compute (page title, section):
 *   sglang PR "[AMD] [GLM5] Fuse the DSA indexer Q/K rope + quant + K-cache
 *   write", Motivation: per layer and step the indexer applies rope to q and
 *   k, LayerNorm to k, an fp8 quant to each, the head-gate scale, and writes
 *   the index-K cache, all of which one fused launch does.  Modifications: the
 *   fused call returns the (q_fp8, weights) contract, honours the token count
 *   and the sliced out_cache_loc of the graph split-op, needs fp32 LayerNorm
 *   parameters, reads cos and sin as separate [max_position, rope_dim/2]
 *   rows, and a k-only prepare-and-store serves the dense decode fast path.
 *   Accuracy (note on the two K-cache writers): fp32 goes to fp8 in one step,
 *   with ue8m0 (power-of-two) scales.
 *   vllm PR "[ROCm][Perf] Enable fused indexer-Q RoPE+quant kernel for
 *   DeepSeek/GLM sparse attention", Summary and Kernel-level evidence: on the
 *   query side RoPE, FP8 (ue8m0) quantisation and the weight-scale fold are one
 *   launch.
 *
 * Per token t (D = 128, r = rope_dim):
 *   k:  y = LayerNorm(k[t]) with fp32 gamma/beta (biased variance, eps inside
 *       the root); RoPE on y[0:r); e_k = the smallest integer with
 *       max(amax(y), 1e-4) <= 448 * 2^e_k; codes = e4m3_rne(y * 2^-e_k);
 *       the 128 codes and the fp32 scale 2^e_k go to slot out_cache_loc[t].
 *   q:  for every head h: RoPE on q[t,h,0:r); e_q and codes as above
 *       (no LayerNorm) -> q_fp8[t,h,:];
 *       weights[t,h] = w[t,h] * 2^e_q[t,h] * softmax_scale * H^-0.5.
 *   RoPE pairs: DSA_ROPE_NEOX (i, i + r/2), DSA_ROPE_GPTJ (2i, 2i + 1), both
 *   with frequency index i; a' = a*c - b*s, b' = b*c + a*s with c, s the
 *   fp32 cos/sin at (position, i), evaluated as fma(a, c, -(b*s)) and
 *   fma(b, c, a*s) with the products rounded to fp32.  Dims >= r pass through.
 *   fp32 -> e4m3 is round-to-nearest-even, saturating at +-448.
 *
 * Index-K cache layout: num_pages pages of page_size * 132 bytes; page p
 * holds page_size rows of 128 e4m3 codes, then page_size fp32 scales.  Slot s
 * is row s % page_size of page s / page_size.  DSA_FLAG_CACHE_TOKEN_MAJOR
 * selects the other layout, 132 bytes per slot (codes, then scale).
 *
 * Conventions shared by every call:
 *   - Pointers are DEVICE pointers owned by the caller; the library allocates
 *     nothing, keeps no state between calls and caches no pointer or table
 *     contents (a replaced cos/sin cache is read afresh on the next call).
 *   - A call acts on the current CUDA device: the stream and every pointer
 *     must belong to it (the SM count and kernel attributes are that
 *     device's).
 *   - Strides are in elements.  The innermost dimension of q, k and w is
 *     contiguous.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  No call synchronises the host, so every call can be
 *     captured into a CUDA graph.  One kernel launch per call (the unfused
 *     comparison chain: four).  The first call
 *     on a device raises the kernel's dynamic shared-memory limit there (a
 *     per-device, once-only setting); make it before capturing a graph.
 *   - Host-side checks: a bad argument returns a status other than DSA_OK and
 *     launches nothing.  T == 0 returns DSA_OK and launches nothing.
 *   - Device-side checks: a position outside [0, max_position) sets bit
 *     DSA_DEVERR_POSITION of *err_flags and that token writes nothing (no
 *     q_fp8 rows, weights or cache slot); a slot outside
 *     [0, num_pages * page_size) sets DSA_DEVERR_SLOT and skips that token's
 *     cache write.  err_flags may be NULL (then nothing is reported).  The
 *     kernel never traps and every internal wait is bounded: a wait that
 *     gives up (never expected) sets DSA_DEVERR_TIMEOUT.  The caller clears
 *     *err_flags.
 *   - Slots within one call must be distinct (two tokens writing one slot
 *     race).  Inputs must not overlap outputs.
 *   - Non-finite inputs give unspecified codes and scales.
 */
#ifndef DSA_PREP_H
#define DSA_PREP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DSA_OK = 0,
  DSA_ERR_NULL = 1,        /* a required pointer is NULL */
  DSA_ERR_ALIGN = 2,       /* a pointer or stride breaks an alignment rule */
  DSA_ERR_SHAPE = 3,       /* a negative or inconsistent size or stride */
  DSA_ERR_UNSUPPORTED = 4, /* head_dim != 128, bad rope_dim, style or flag */
  DSA_ERR_LAUNCH = 5,      /* the CUDA launch itself failed */
  DSA_ERR_SCRATCH_LIMIT = 6 /* the call needs more than the library's built-in
                               scratch buffer holds (the _noalloc entry point) */
} dsa_status;

typedef enum { DSA_ROPE_NEOX = 0, DSA_ROPE_GPTJ = 1 } dsa_rope_style;

#define DSA_HEAD_DIM 128

/* Bits of the device error word. */
#define DSA_DEVERR_POSITION 1 /* a position outside [0, max_position) */
#define DSA_DEVERR_SLOT 2     /* a slot outside [0, num_pages * page_size) */
#define DSA_DEVERR_TIMEOUT 4  /* an internal wait gave up (never expected) */
#define DSA_DEVERR_INTERNAL 8 /* an internal precondition failed: the logits
                                 kernel's shared-memory base was not 1024-byte
                                 aligned (never expected); nothing was written */

/* Launch flags. */
#define DSA_FLAG_PDL 1u /* programmatic dependent launch: the kernel may start
                           while the previous kernel in the stream finishes; it
                           waits for that kernel's memory before reading
                           anything */
/* Kernel choice.  By default calls with T * H <= 16384 query vectors take the
 * direct kernel (every input in flight at once: least latency, for decode)
 * and larger ones the pipeline kernel (bulk copies through a shared-memory
 * ring: most bandwidth, for prefill).  k-only calls take the direct kernel up
 * to 8192 keys and the k-stream kernel (persistent warps over key ranges,
 * cp.async rings) above; for them DSA_FLAG_PIPELINE selects the k-stream
 * kernel.  These flags force one; all give the same bytes.  Setting both is
 * an error. */
#define DSA_FLAG_PIPELINE 2u
#define DSA_FLAG_DIRECT 4u
/* With DSA_FLAG_PDL only: the caller promises that positions, out_cache_loc
 * and the cos/sin cache are NOT written by the kernel that precedes this call
 * in the stream (true in a decode step, where they are set up before the
 * layers run).  The kernel then reads them -- and fetches the cos/sin rows
 * they select -- before it waits for that kernel, overlapping two dependent
 * memory round trips with its tail.  q, k and w are still read only after the
 * wait.  Without DSA_FLAG_PDL this flag is an error. */
#define DSA_FLAG_PDL_EARLY_ROPE 8u
/* Index-K cache layout.  Default (page-blocked): page p holds page_size rows
 * of 128 e4m3 codes, then page_size fp32 scales; slot s is row s % page_size
 * of page s / page_size, and page_size must be a multiple of 4.  With this
 * flag (token-major): slot s owns bytes [132*s, 132*s + 132) -- its 128 codes,
 * then its fp32 scale -- and page_size only sets the slot count
 * num_pages * page_size.  Same buffer size either way. */
#define DSA_FLAG_CACHE_TOKEN_MAJOR 16u
/* Hadamard-rotated variant.  After RoPE (and, for k, LayerNorm then RoPE)
 * every q head and k is multiplied by H_128 / sqrt(128), H_128 the Sylvester
 * Walsh-Hadamard matrix, before its scale and codes are taken -- the rotation
 * that the fused path of sglang PR "[AMD] [GLM5] Fuse the DSA indexer Q/K
 * rope + quant + K-cache write" (Modifications, "no-Hadamard invariant")
 * leaves out.  The product is computed as fp32 butterflies over index bits
 * 0, 1, ..., 6 in that order, (a, b) -> (a + b, a - b), then one multiply by
 * fp32(128^-0.5): the rounding is fixed, so the codes are reproducible.
 * Scores are unchanged up to quantisation, since H_128 / sqrt(128) is
 * orthogonal.  Accepted by dsa_indexer_qk_prepare_store and
 * dsa_indexer_k_prepare_store; the unfused chain rejects it. */
#define DSA_FLAG_HADAMARD 32u
/* dsa_indexer_mqa_logits, with DSA_FLAG_PDL only: the caller promises that
 * block_table and context_lens are NOT written by the kernel that precedes
 * the call in the stream (true in a decode step, where only q_fp8, the
 * weights and one cache slot per sequence are).  The kernel then reads them,
 * and starts its first key pages on their way into L2, before it waits for
 * that kernel.  The fused prepare-and-store calls reject this flag. */
#define DSA_FLAG_PDL_EARLY_INDEX 64u
/* TEST ONLY, with DSA_FLAG_PIPELINE: the producer warp of the pipeline
 * kernel's first CTA withholds the copies of its first unit and never marks
 * that stage full.  That CTA's consumers then give up their bounded waits
 * (2 s each), the CTA stops, and the call sets DSA_DEVERR_TIMEOUT in
 * *err_flags; the outputs of that CTA's units are unspecified and every other
 * CTA completes normally.  It exists so the timeout path can be tested
 * without a fault; the context stays usable.  Without DSA_FLAG_PIPELINE this
 * flag is an error. */
#define DSA_FLAG_TEST_WITHHOLD_UNIT (1u << 30)

/*
 * Fused Q/K prepare-and-store: returns the (q_fp8, weights) contract and
 * writes k's codes and scale into the index-K cache, in one launch.
 *
 *   q              bf16 [T, H, 128]; row strides q_stride_t, q_stride_h.
 *                  16-byte aligned; both strides multiples of 8.
 *   k              bf16 [T, 128]; row stride k_stride_t (multiple of 8);
 *                  16-byte aligned.  May be a column slice of the fused
 *                  k/weights projection output.
 *   w              bf16 [T, H] gate weights; row stride w_stride_t >= H;
 *                  2-byte aligned.
 *   positions      int64 [T], 8-byte aligned.
 *   out_cache_loc  int64 [T] cache slots (the live, possibly sliced, view).
 *   cos_cache,     fp32 [max_position, >= rope_dim/2] each, row stride
 *   sin_cache      cs_stride (multiple of 4); 16-byte aligned.  May be NULL
 *                  when rope_dim == 0.
 *   ln_gamma,      fp32 [128], 16-byte aligned; ln_eps finite and >= 0 (it
 *   ln_beta        sits inside the square root).
 *   softmax_scale  the caller's attention scale (DeepSeek-style indexers pass
 *                  128^-0.5); H^-0.5 is applied here.
 *   q_fp8_out      e4m3 bytes [T, H, 128], contiguous, 16-byte aligned.
 *   weights_out    fp32 [T, H], contiguous, 4-byte aligned.
 *   index_k_cache  num_pages * page_size * 132 bytes, 16-byte aligned;
 *                  page_size a multiple of 4 (page-blocked layout only).
 *   T >= 0, 1 <= H <= 4096, head_dim == 128, rope_dim in {0, 16, 32, 64, 128},
 *   rope_style a dsa_rope_style, flags a set of DSA_FLAG_* bits.
 */
dsa_status dsa_indexer_qk_prepare_store(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    const void* k, int64_t k_stride_t,
    const void* w, int64_t w_stride_t,
    const int64_t* positions, const int64_t* out_cache_loc,
    const float* cos_cache, const float* sin_cache, int64_t cs_stride,
    int64_t max_position,
    const float* ln_gamma, const float* ln_beta, float ln_eps,
    float softmax_scale,
    void* q_fp8_out, float* weights_out,
    void* index_k_cache, int64_t num_pages, int32_t page_size,
    int32_t T, int32_t H, int32_t head_dim, int32_t rope_dim,
    int32_t rope_style, uint32_t flags, int32_t* err_flags, void* stream);

/*
 * k-only prepare-and-store (the decode fast path of sglang PR "[AMD] [GLM5]
 * Fuse the DSA indexer Q/K rope + quant + K-cache write", Modifications):
 * the k side of dsa_indexer_qk_prepare_store alone, same arguments, same
 * rules, same cache bytes.
 */
dsa_status dsa_indexer_k_prepare_store(
    const void* k, int64_t k_stride_t,
    const int64_t* positions, const int64_t* out_cache_loc,
    const float* cos_cache, const float* sin_cache, int64_t cs_stride,
    int64_t max_position,
    const float* ln_gamma, const float* ln_beta, float ln_eps,
    void* index_k_cache, int64_t num_pages, int32_t page_size,
    int32_t T, int32_t head_dim, int32_t rope_dim, int32_t rope_style,
    uint32_t flags, int32_t* err_flags, void* stream);

/*
 * The unfused chain: the same computation as dsa_indexer_qk_prepare_store,
 * as the four launches per layer that the sglang PR "[AMD] [GLM5] Fuse the
 * DSA indexer Q/K rope + quant + K-cache write" profiles before fusing
 * (Profile section: rope q+k, LayerNorm, act_quant, k quant + cache; the gate
 * fold rides with the q quant here).  Launch order: LayerNorm(k) -> RoPE(q, k)
 * -> quant(q) + fold -> quant(k) + cache store.  The tensors between launches
 * are bf16, kept in `workspace` (device memory owned by the caller, 256-byte
 * aligned, at least dsa_unfused_workspace_bytes(T, H) bytes, contents
 * scratch).  Because LayerNorm and RoPE outputs are rounded to bf16, its codes
 * can differ from the fused call's by one step near rounding boundaries; its
 * scales and slots follow the same rules.  Arguments and checks are those of
 * dsa_indexer_qk_prepare_store; flags may hold DSA_FLAG_PDL and
 * DSA_FLAG_CACHE_TOKEN_MAJOR only.  Kept as the
 * baseline the fused call is measured against.
 */
size_t dsa_unfused_workspace_bytes(int32_t T, int32_t H);

dsa_status dsa_indexer_qk_prepare_store_unfused(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    const void* k, int64_t k_stride_t,
    const void* w, int64_t w_stride_t,
    const int64_t* positions, const int64_t* out_cache_loc,
    const float* cos_cache, const float* sin_cache, int64_t cs_stride,
    int64_t max_position,
    const float* ln_gamma, const float* ln_beta, float ln_eps,
    float softmax_scale,
    void* q_fp8_out, float* weights_out,
    void* index_k_cache, int64_t num_pages, int32_t page_size,
    int32_t T, int32_t H, int32_t head_dim, int32_t rope_dim,
    int32_t rope_style, uint32_t flags, void* workspace, size_t workspace_bytes,
    int32_t* err_flags, void* stream);

/*
 * The unfused chain without a caller workspace, for callers that cannot
 * allocate device memory when they run it: an engine that gives the whole GPU
 * to its own memory pool at start-up and forbids other allocations, a plugin
 * host that only hands over pointers to inputs and outputs, or code in a
 * place where cudaMalloc would synchronise or is not allowed.  The paper has
 * no counterpart to this entry point; it is an interface convenience.
 *
 * The bf16 intermediates go to a 32 MiB buffer compiled into the library (a
 * fixed array in device global memory, present on every GPU that loads the
 * library until the process exits).  A call therefore needs
 * dsa_unfused_workspace_bytes(T, H) <= 32 MiB, i.e. T * (H + 2) <= 131072;
 * larger calls return DSA_ERR_SCRATCH_LIMIT and launch nothing.
 *
 * The caller still passes all inputs and outputs; the call allocates nothing
 * (no cudaMalloc or cudaFree).  The first call on each device looks the
 * buffer's device address up once, with that device current -- make that
 * first call outside any stream capture.  The address is kept for the life
 * of the process: after a cudaDeviceReset of a device this entry point has
 * run on, the kept address is stale, so do not call it on that device again.
 *
 * All calls on a device share the one buffer: two calls that may run on the
 * GPU at the same time (different streams without ordering between them)
 * race and corrupt each other's results.  Order them (one stream, or events).
 * The buffer keeps whatever the last call left in it; the chain writes every
 * intermediate before reading it, so nothing needs clearing between calls.
 * Arguments, checks and results are otherwise those of
 * dsa_indexer_qk_prepare_store_unfused.
 */
dsa_status dsa_indexer_qk_prepare_store_unfused_noalloc(
    const void* q, int64_t q_stride_t, int64_t q_stride_h,
    const void* k, int64_t k_stride_t,
    const void* w, int64_t w_stride_t,
    const int64_t* positions, const int64_t* out_cache_loc,
    const float* cos_cache, const float* sin_cache, int64_t cs_stride,
    int64_t max_position,
    const float* ln_gamma, const float* ln_beta, float ln_eps,
    float softmax_scale,
    void* q_fp8_out, float* weights_out,
    void* index_k_cache, int64_t num_pages, int32_t page_size,
    int32_t T, int32_t H, int32_t head_dim, int32_t rope_dim,
    int32_t rope_style, uint32_t flags, int32_t* err_flags, void* stream);

/*
 * fp8 paged MQA logits: the indexer kernel that reads what the calls above
 * write.  The vllm PR "[ROCm][Perf] Enable fused indexer-Q RoPE+quant kernel
 * for DeepSeek/GLM sparse attention" lists it (Kernel-level evidence,
 * "_gluon_deepgemm_fp8_paged_mqa_logits") right after the index-K store and
 * gives no formula; the one here is the DeepSeek sparse-attention indexer's:
 *   logits[t, j] = k_scale[j] * sum_h weights[t, h] * max(q[t, h] . k[j], 0)
 * for j < context_lens[t], with q and k the e4m3 codes (weights already hold
 * the q scales); columns context_lens[t] <= j < max_context get -inf.
 *
 *   q_fp8          e4m3 [T, H, 128] contiguous, 16-byte aligned.
 *   weights        fp32 [T, H] contiguous.
 *   index_k_cache  page-blocked layout, page_size == 64, 16-byte aligned.
 *   block_table    int32 [T, bt_stride], bt_stride >= ceil(max_context / 64)
 *                  (else DSA_ERR_SHAPE): the physical page of each 64-key
 *                  block.  A row's entries past its token's context are read
 *                  and ignored, so they may hold anything.
 *   context_lens   int32 [T], keys of token t; only the first max_context
 *                  of them have a column (a longer context is clamped).
 *   logits         fp32 [T, logits_stride >= max_context].
 *   T <= 65535; H in {16, 32, 64, 128}; flags may hold DSA_FLAG_PDL and,
 *   with it, DSA_FLAG_PDL_EARLY_INDEX.
 * Runs on the tensor cores (tcgen05, fp32 accumulation in TMEM); the first
 * call on a device raises its shared-memory limit there.  A block-table entry
 * (within the context) outside [0, num_pages) sets DSA_DEVERR_SLOT, and its
 * keys' logits are NaN.
 */
dsa_status dsa_indexer_mqa_logits(
    const void* q_fp8, const float* weights,
    const void* index_k_cache, int64_t num_pages, int32_t page_size,
    const int32_t* block_table, int64_t bt_stride, const int32_t* context_lens,
    float* logits, int64_t logits_stride, int32_t max_context,
    int32_t T, int32_t H, uint32_t flags, int32_t* err_flags, void* stream);

/* A static, NUL-terminated description of a status code. */
const char* dsa_status_string(dsa_status status);

/* Library version, (major << 16) | minor. */
int32_t dsa_prep_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DSA_PREP_H */
