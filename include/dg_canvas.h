/*
 * dg_canvas.h -- C ABI of libdgcanvas, the GB300 (sm_103a) hot path of one
 * uniform-state text-diffusion denoising step over a fixed-size canvas.
 *
 * Source of each operation: the DiffusionGemma explainer ("Understanding
 * DiffusionGemma", ai.google.dev/gemma/docs/diffusiongemma/explained):
 *   dg_canvas_attn   -- "Architecture: incremental prefill and denoising",
 *                       denoising mode: every canvas query attends to every
 *                       canvas token and to the KV cache (bidirectional).
 *   dg_vocab_step    -- "2. Uniform-state diffusion" (a token's probability
 *                       against a threshold) and "Self-conditioning" (the
 *                       probability matrix times the token-embedding table).
 *   dg_renoise       -- "2. Uniform-state diffusion": a token whose
 *                       probability falls below the threshold is replaced by
 *                       a random vocabulary token.
 *   dg_canvas_init   -- "The problem with autoregressive models": the canvas
 *                       starts as random tokens drawn from the vocabulary.
 *   dg_kv_append     -- "Architecture..." prefill mode and "Multi-canvas
 *                       sampling": each finalised canvas is appended to the
 *                       KV cache with causal attention.
 * Further calls, each documented in its section below: dg_vocab_step_renoise
 * (the vocabulary step with the re-noise fused in), dg_vocab_step_plan,
 * dg_canvas_attn_noalloc, the calls next to the step (dg_selfcond_input,
 * dg_token_prob, dg_unmask, dg_canvas_fill, dg_count_flags), the device-side
 * cache length variants (*_devlen, *_devpos) and the test hook
 * dg_debug_inject.
 *
 * Conventions shared by every call
 *   - Pointers named as tensors are DEVICE pointers owned by the caller, in
 *     the layout stated beside them (row-major, densely packed). `stream` is
 *     a cudaStream_t (NULL = the legacy default stream). Calls are
 *     asynchronous on `stream`.
 *   - Host-side validation runs first. On any error no kernel is launched and
 *     no output is touched; the call returns the error.
 *   - A launch failure returns DG_ERR_CUDA. Faults a kernel detects itself
 *     (a bounded wait that ran out, an index out of range) are latched into a
 *     library-owned device status word, read and cleared by dg_device_status.
 *     Kernels never trap.
 *   - The library allocates nothing per call. Scratch memory is the caller's
 *     workspace, sized by the *_workspace_size queries (0 is a valid size).
 *     A workspace must be 256-byte aligned and must not be shared by calls
 *     that can run concurrently.
 *   - dtype DG_BF16: bf16 tensors, fp32 accumulation and softmax; this is the
 *     tensor-core (tcgen05) path. dtype DG_F32: fp32 tensors, a CUDA-core
 *     path meant for small shapes.
 */
#ifndef DG_CANVAS_H
#define DG_CANVAS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DG_API __attribute__((visibility("default")))
#else
#define DG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, bad size, len+C > cap ... */
  DG_ERR_UNSUPPORTED = -2,   /* shape or dtype the library does not implement     */
  DG_ERR_WORKSPACE = -3,     /* workspace smaller than the size query returned    */
  DG_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed              */
  DG_ERR_TIMEOUT = -5,       /* (device status) a bounded wait ran out            */
  DG_ERR_DEVICE_BOUNDS = -6  /* (device status) a kernel saw an index out of range */
} dg_status;

typedef enum { DG_BF16 = 0, DG_F32 = 1 } dg_dtype;

typedef enum {
  DG_MASK_BIDIR = 0,        /* denoising: no mask                                      */
  DG_MASK_CAUSAL_BLOCK = 1  /* prefill: query i (absolute position P+i) sees keys 0..P+i */
} dg_mask;

/* Human-readable name of a status code. Never NULL. */
DG_API const char* dg_status_string(int status);

/* Synchronises `stream`, then returns the device status word (DG_OK or the
 * first DG_ERR_TIMEOUT / DG_ERR_DEVICE_BOUNDS latched since the last call)
 * and clears it. Returns DG_ERR_CUDA if the synchronisation itself fails. */
DG_API int dg_device_status(void* stream);

/* ---------------------------------------------------------------- attention
 * Canvas attention (denoising mode), grouped-query:
 *   for query head h (KV head g = h / (Hq/Hkv)) and canvas position i,
 *   keys/values = [cache rows 0..P-1 of head g ; canvas rows 0..C-1 of head g]
 *   out[i][h]  = softmax_j(q[i][h] . k_j * scale) . v
 *   lse[h][i]  = natural-log log-sum-exp of the scaled scores
 *
 *   q         [C][Hq][hd]        k_cache, v_cache [Hkv][cap][hd] (rows [0,P) read)
 *   k_canvas  [Hkv][C][hd]       v_canvas [Hkv][C][hd]
 *   out       [C][Hq][hd] (dtype)   lse [Hq][C] fp32, or NULL
 *   scale <= 0 selects 1/sqrt(hd). mask = dg_mask.
 * Requirements: Hq % Hkv == 0; hd in {32, 64, 128}; 0 <= P <= cap; C >= 1;
 * every pointer 16-byte aligned. Workspace: split-KV partials.
 * At hd = 128 with key splits the call launches a one-CTA kernel that zeroes
 * the workspace's arrival counters, then the attention kernel as its
 * programmatic dependent: at most one CTA per SM, all resident at once, with
 * bounded waits between the splits of a row block (a wait that expires,
 * after about two seconds, sets DG_ERR_TIMEOUT and the outputs are not
 * valid). DG_ATTN_COOP=1 in the environment replaces the reset kernel by a
 * memset and makes the attention launch cooperative, which the driver
 * co-schedules next to other work.
 */
DG_API size_t dg_canvas_attn_workspace_size(int C, int Hq, int Hkv, int hd, int64_t prefix_len, int dtype);
DG_API int dg_canvas_attn(const void* q, const void* k_cache, const void* v_cache, int64_t cap, int64_t prefix_len,
                   const void* k_canvas, const void* v_canvas, void* out, float* lse,
                   int C, int Hq, int Hkv, int hd, float scale, int dtype, int mask,
                   void* workspace, size_t workspace_bytes, void* stream);

/* Canvas attention for callers that cannot allocate device memory (hosts that
 * own every device allocation, plugins given no scratch buffer, loops where an
 * allocation could synchronise the device). The explainer pages have no counterpart:
 * this is a deployment variant of dg_canvas_attn, same arguments and results
 * minus the workspace. Its split-KV scratch is a fixed array inside the
 * library's device image (dg_canvas_attn_noalloc_max_scratch() bytes, 32 MiB),
 * reserved on every GPU that loads the library until the process exits.
 *   - Returns DG_ERR_WORKSPACE if the shape needs more scratch than that.
 *   - The first call on a device looks up the array's device address with the
 *     device current; make that first call before any stream capture.
 *   - All calls share the array: calls that may overlap on the GPU race on it.
 *   - Allocates nothing (no cudaMalloc, no library allocator). */
DG_API int dg_canvas_attn_noalloc(const void* q, const void* k_cache, const void* v_cache, int64_t cap,
                                  int64_t prefix_len, const void* k_canvas, const void* v_canvas, void* out,
                                  float* lse, int C, int Hq, int Hkv, int hd, float scale, int dtype, int mask,
                                  void* stream);
DG_API size_t dg_canvas_attn_noalloc_max_scratch(void);

/* ---------------------------------------------------------------- vocabulary step
 * For each canvas position i (row of h):
 *   logits l_i = h_i . emb^T            (emb is the tied token-embedding table)
 *   argmax[i]  = lowest vocabulary id attaining max_v l_iv
 *   conf[i]    = softmax(l_i)[argmax[i]] = 1 / sum_v exp(l_iv - max l_i)
 *   lse[i]     = log-sum-exp of l_i (natural log)
 *   selfcond[i]= softmax(l_i) . emb     (the self-conditioning vector)
 * One pass over vocabulary tiles of 256 ids. The fp32 logits never reach
 * memory; the softmax numerators exp(l - R) (R a per-row reference) go to
 * the workspace in bf16 (V x 512 bytes, read back through L2) for the
 * self-conditioning product. E is streamed from HBM once for the logits;
 * the self-conditioning product reads each E tile again shortly after, from
 * L2 where most of it is still resident (measured at V = 262144, d = 2816:
 * 1.71 GB of DRAM reads per call for a 1.48 GB table).
 * The step runs one CTA on every SM, all resident at once, with bounded
 * waits between them: run it when other kernels do not hold SMs for long
 * (a wait that expires, after about two seconds, sets DG_ERR_TIMEOUT in the
 * device status word and the call's outputs are not valid). A one-CTA
 * kernel first zeroes the workspace's flags; the main kernel is launched as
 * its programmatic dependent, and the combine kernel as the main kernel's.
 * Setting DG_VOCAB_COOP=1 in the environment zeroes the flags with a memset
 * and makes the main launch cooperative, which the driver co-schedules next
 * to other work (Nsight Compute cannot replay that form).
 *
 *   h        [C][d] (dtype)     emb [V][d] (dtype)
 *   argmax   [C] int32          conf [C] fp32      lse [C] fp32 or NULL
 *   selfcond [C][d] (dtype) or NULL
 * Requirements (DG_BF16): 1 <= C <= 256, d % 64 == 0, 64 <= d <= 8192, V >= 1.
 * (DG_F32): C >= 1, 1 <= V <= 16384, 1 <= d <= 1024.
 */
DG_API size_t dg_vocab_step_workspace_size(int C, int V, int d, int dtype);
DG_API int dg_vocab_step(const void* h, const void* emb, int C, int V, int d, int dtype,
                  int32_t* argmax, float* conf, float* lse, void* selfcond,
                  void* workspace, size_t workspace_bytes, void* stream);

/* dg_vocab_step followed by dg_renoise on its argmax/conf, with the re-noise
 * done inside the vocabulary step's last kernel (one launch fewer per step).
 * Arguments and results are those of the two calls; tokens/renoised as in
 * dg_renoise (step, seed, abs_pos0 key the Philox draw). */
DG_API int dg_vocab_step_renoise(const void* h, const void* emb, int C, int V, int d, int dtype,
                                 int32_t* argmax, float* conf, float* lse, void* selfcond,
                                 int32_t* tokens, float threshold, uint64_t seed, uint32_t step, int64_t abs_pos0,
                                 uint8_t* renoised, void* workspace, size_t workspace_bytes, void* stream);

/* Launch plan of the bf16 vocabulary step on the current device (host-only
 * query, no kernel): plan[0] producer CTAs, [1] consumer CTAs, [2] vocabulary
 * residue classes of the consumers, [3] 1 if the kernel runs on CTA pairs
 * (clusters of two CTAs sharing each MMA; 0: one CTA per role unit, where such
 * clusters cannot be placed), [4] CTAs launched, [5] vocabulary tiles of 256
 * ids. The query needs no device: without one it plans for 152 SMs. */
DG_API int dg_vocab_step_plan(int C, int V, int d, int dtype, int32_t* plan /* [6] */);

/* ---------------------------------------------------------------- re-noise
 * tokens[i] = conf[i] < threshold ? U(seed, step, abs_pos0 + i) : argmax[i]
 * renoised[i] = (conf[i] < threshold)            (renoised may be NULL)
 * U is a uniform vocabulary id: Philox4x64-10 with key (seed, 0) and counter
 * (absolute position, step, 0, 0); output word 0, mapped to [0, V) as
 * ((word >> 32) * V) >> 32. The comparison is in fp32 and strict.
 *   tokens [C] int32 (out; may alias nothing else)   argmax [C] int32   conf [C] fp32
 * Requirements: C >= 1, 1 <= V <= 2^31 - 1. An argmax outside [0, V) is copied
 * as is and latches DG_ERR_DEVICE_BOUNDS.
 */
DG_API int dg_renoise(int32_t* tokens, const int32_t* argmax, const float* conf, int C, int V, float threshold,
               uint64_t seed, uint32_t step, int64_t abs_pos0, uint8_t* renoised, void* stream);

/* Fresh canvas: tokens[i] = U_init(seed, abs_pos0 + i): the same Philox draw
 * with counter (absolute position, 0, 1, 0). */
DG_API int dg_canvas_init(int32_t* tokens, int C, int V, uint64_t seed, int64_t abs_pos0, void* stream);

/* ---------------------------------------------------------------- KV append
 * Incremental causal prefill of one finalised canvas:
 *   k_cache[g][*len + i] = k_new[g][i], v_cache likewise, for i < C, all g;
 *   then *len += C (host-side; advanced only when the call returns DG_OK).
 * If q_new is not NULL, also computes the block's causal attention over the
 * updated cache (query i at absolute position P+i sees keys 0..P+i):
 *   out [C][Hq][hd] (dtype), lse [Hq][C] fp32 or NULL.
 *   k_cache, v_cache [Hkv][cap][hd]   k_new, v_new [Hkv][C][hd]   q_new [C][Hq][hd]
 * Requirements: *len + C <= cap; rows outside [*len, *len + C) are not written.
 * Workspace: as dg_canvas_attn for (C, Hq, Hkv, hd, *len) when q_new != NULL.
 */
DG_API int dg_kv_append(void* k_cache, void* v_cache, int64_t cap, int64_t* len,
                 const void* k_new, const void* v_new, int C, int Hkv, int hd, int dtype,
                 const void* q_new, int Hq, void* out, float* lse,
                 void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- next to the step
 * Self-conditioning input. DiffusionGemma explainer, "Self-conditioning": the
 * probabilities times the embedding table (selfcond, from dg_vocab_step) are
 * handed to the next step. The backbone layer that takes them is outside this
 * library; this is the stand-in input it would read:
 *   x[i][:] = emb[tokens[i]][:] + selfcond[i][:]    (selfcond NULL: emb rows alone)
 * summed in fp32 and rounded once to dtype.
 *   tokens [C] int32   emb [V][d] (dtype)   selfcond [C][d] (dtype) or NULL
 *   x [C][d] (dtype, out; must not alias the inputs)
 * Requirements: C >= 1, V >= 1, d >= 1 with d % 8 == 0 (DG_BF16) or d % 4 == 0
 * (DG_F32); every pointer 16-byte aligned. A token outside [0, V) gives a zero
 * row and latches DG_ERR_DEVICE_BOUNDS.
 */
DG_API int dg_selfcond_input(const int32_t* tokens, const void* emb, const void* selfcond, void* x, int C, int V,
                             int d, int dtype, void* stream);

/* Probability of the token now on the canvas. DiffusionGemma explainer,
 * "2. Uniform-state diffusion", with "a token's probability" read as the
 * probability of the current token rather than of the prediction:
 *   prob[i] = exp(h[i] . emb[tokens[i]] - lse[i])
 * where lse is the natural-log log-sum-exp dg_vocab_step returned for row i
 * (fp32 dot product). Passing prob to dg_renoise as conf re-noises by this
 * reading.
 *   h [C][d] (dtype)   emb [V][d] (dtype)   tokens [C] int32   lse [C] fp32
 *   prob [C] fp32 (out)
 * Requirements: as dg_selfcond_input. A token outside [0, V) gives prob 0 and
 * latches DG_ERR_DEVICE_BOUNDS.
 */
DG_API int dg_token_prob(const void* h, const void* emb, const int32_t* tokens, const float* lse, float* prob, int C,
                         int V, int d, int dtype, void* stream);

/* Masked diffusion with lock-in. DiffusionGemma explainer, "1. Masked
 * diffusion": positions start as a [MASK] id; once the model is confident a
 * [MASK] becomes a word, and a replaced token is never changed again:
 *   if tokens[i] == mask_id and conf[i] >= threshold (fp32):
 *        tokens[i] = argmax[i], unmasked[i] = 1
 *   else tokens[i] unchanged,   unmasked[i] = 0          (unmasked may be NULL)
 */
DG_API int dg_unmask(int32_t* tokens, const int32_t* argmax, const float* conf, int C, int32_t mask_id,
                     float threshold, uint8_t* unmasked, void* stream);

/* tokens[i] = value for i < C (e.g. a fully masked canvas for dg_unmask). */
DG_API int dg_canvas_fill(int32_t* tokens, int C, int32_t value, void* stream);

/* *count = number of i < C with flags[i] != 0, written on the device (early
 * stop: a step whose renoised flags are all zero finishes the canvas). */
DG_API int dg_count_flags(const uint8_t* flags, int C, int32_t* count, void* stream);

/* ---------------------------------------------------------------- device-side cache length
 * Block diffusion (DiffusionGemma explainer, "Multi-canvas sampling (block
 * diffusion)") appends every finished canvas to the cache, so the prefix
 * grows by C per canvas. These variants read the prefix length / position
 * offset from device memory instead of a host argument, so one captured CUDA
 * graph of a canvas (init, steps, append) can be replayed for every block.
 * Results are those of the host-length calls with the same values.
 *
 * dg_canvas_attn_devlen: dg_canvas_attn with P = *prefix_len_dev, which must
 * lie in [0, prefix_max] (prefix_max <= cap; outside: clamped, and
 * DG_ERR_DEVICE_BOUNDS latched). The kernel is planned for prefix_max, so the
 * workspace is dg_canvas_attn_workspace_size(C, Hq, Hkv, hd, prefix_max, dtype).
 * The key tiles follow the device-side P: no tile past P is read, except the
 * rows past P inside the last, partly filled 128-row cache tile, which are
 * read and masked out; they must hold finite values (zero-initialise the
 * cache once). DG_BF16 and hd == 128 only.
 */
DG_API int dg_canvas_attn_devlen(const void* q, const void* k_cache, const void* v_cache, int64_t cap,
                                 const int64_t* prefix_len_dev, int64_t prefix_max, const void* k_canvas,
                                 const void* v_canvas, void* out, float* lse, int C, int Hq, int Hkv, int hd,
                                 float scale, int dtype, int mask, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* dg_canvas_init with abs_pos0 = *abs_pos0_dev. */
DG_API int dg_canvas_init_devpos(int32_t* tokens, int C, int V, uint64_t seed, const int64_t* abs_pos0_dev,
                                 void* stream);

/* dg_vocab_step_renoise with abs_pos0 = *abs_pos0_dev (DG_BF16 only). */
DG_API int dg_vocab_step_renoise_devpos(const void* h, const void* emb, int C, int V, int d, int dtype,
                                        int32_t* argmax, float* conf, float* lse, void* selfcond, int32_t* tokens,
                                        float threshold, uint64_t seed, uint32_t step, const int64_t* abs_pos0_dev,
                                        uint8_t* renoised, void* workspace, size_t workspace_bytes, void* stream);

/* dg_kv_append without the attention, at P = *len_dev on the device, then
 * *len_dev += C on the device. If P < 0 or P + C > cap nothing is written,
 * *len_dev is unchanged and DG_ERR_DEVICE_BOUNDS is latched. */
DG_API int dg_kv_append_devlen(void* k_cache, void* v_cache, int64_t cap, int64_t* len_dev, const void* k_new,
                               const void* v_new, int C, int Hkv, int hd, int dtype, void* stream);

/* ---------------------------------------------------------------- failure injection (tests)
 * Not part of the method (the explainer pages have no counterpart): a test
 * hook that makes the NEXT launch of one kernel fail its cross-CTA handshake
 * without any fault, so that the bounded waits, DG_ERR_TIMEOUT and the
 * recovery of the context can be exercised on a GPU.
 *   kind 0: clear a pending injection
 *   kind 1: dg_canvas_attn (head_dim 128, more than one key split): key split
 *           0 of every group withholds its arrival on the merge counter
 *   kind 2: dg_vocab_step / dg_vocab_step_renoise (bf16): the P tile 0 ready
 *           flag is never released
 * wait_ms bounds every wait of that launch (0: the default, about 2 s; at
 * most 10000). The launch then latches DG_ERR_TIMEOUT in the device status
 * word, its outputs are undefined, and every CTA returns; later launches run
 * normally. Host-side state, one pending injection per process.
 */
DG_API int dg_debug_inject(int kind, int wait_ms);

#ifdef __cplusplus
}
#endif
#endif /* DG_CANVAS_H */
