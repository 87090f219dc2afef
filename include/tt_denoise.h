/*
 * tt_denoise.h -- C ABI of the TwoTower denoise-step library (libtt_denoise.so).
 *
 * One denoiser step of block-wise diffusion decoding on one GPU:
 *   tt_denoise_attn  two-segment attention of the S block queries of one layer
 *   tt_context_block_attn  the same attention with a causal view inside the
 *                    block: the context tower taking in a committed block
 *   tt_unmask        confidence unmasking of the block over the vocabulary logits
 *   tt_kv_append     commit of a finished block's KV into the context caches
 *   tt_block_step    all attention layers of one step followed by the unmasking
 * and, on the training side of the same method:
 *   tt_linear_schedule_mask  corruption of clean blocks under the linear schedule
 *   tt_masked_nll    the masked-diffusion loss over the vocabulary logits
 *
 * Sources.  The method is described by the pages on "Nemotron-TwoTower:
 * Diffusion Language Modeling with Pretrained Autoregressive Context":
 *   [ARCH]  gist.science summary (German), "Technisches Resuemee -- Architektur":
 *           the frozen context tower produces layer-aligned KV caches; the
 *           denoiser uses bidirectional attention inside the noisy block and
 *           causal cross-attention to the same layer of the context tower.
 *   [GEN]   same page, "Generierungsprozess" (Algorithm 1): a block of S masked
 *           tokens is refined over T steps; at every step the denoiser attends to
 *           the context tower's KV cache of past blocks and to its own
 *           bidirectional KV of the current block; a finished block is committed
 *           and the context tower extends its state with the clean tokens.
 *   [SAMP]  same page, "Training und Konditionierung -- Sampling" (Algorithm 2)
 *           and "Der Konfidenz-Trick": all masked tokens are predicted in
 *           parallel, those whose confidence exceeds a threshold are committed
 *           and locked, the rest stay masked for the next step.
 *   [T]     same page, "Training und Konditionierung -- Maskierte Diffusion": clean
 *           blocks are corrupted by replacing tokens with [MASK] under a linear
 *           schedule, and the denoiser minimises the negative log-likelihood of the
 *           original tokens at the masked positions.
 *   [NEWS]  dgnews.ru article, "How the architecture actually works": inside the
 *           block every masked position attends to every other block position,
 *           towards earlier blocks and the prompt attention stays causal, and each
 *           denoiser layer reads the matching context-tower layer.
 *
 * Conventions (every entry point):
 *   - Asynchronous on the caller's stream (`tt_stream_t`, binary-compatible with
 *     cudaStream_t; NULL is the legacy default stream).  Only
 *     tt_get_device_error synchronises.
 *   - Every pointer argument marked "device" is device memory owned by the
 *     caller.  The library never allocates or frees memory and keeps no state
 *     between calls; it is safe to call from several host threads.  The one
 *     exception is tt_unmask_noalloc: it keeps its scratch in a device array of
 *     the library's own (shared by all its calls, which therefore must not
 *     overlap on the GPU) and caches that array's address per device; its own
 *     comment below gives the rules.
 *   - Workspace: each call that needs scratch takes (ws, ws_bytes); the size
 *     comes from the matching *_workspace_size function.  The workspace must be
 *     zero-filled before its first use; the kernels leave their counters at zero
 *     when they finish, so it can be reused by later calls on the same stream
 *     without clearing.  After a device error (see below) clear it again.  Two
 *     calls that run concurrently on different streams need separate
 *     workspaces.
 *   - Host-detectable argument errors return an error code before anything is
 *     launched.  Errors that only the device can see (a page id outside the
 *     pool, a context longer than its pages, a bounded wait that gave up) are
 *     written to the caller's device word `dev_err` (first error wins; the
 *     value is a tt_status) and the affected work is skipped; read it with
 *     tt_get_device_error.  `dev_err` may be NULL only if the caller accepts
 *     that such errors go unreported.
 *   - No C++ exception crosses this interface.
 *
 * Layouts (row-major, innermost last):
 *   q        [B, S, Hq, D]             block queries (already position-encoded)
 *   k_blk    [B, S, Hkv, D]            the block's own keys / values
 *   out      [B, S, Hq, D]             attention output, same dtype as q
 *   lse      [B, Hq, S] fp32           natural-log sum of exp(scores), optional
 *   k_pool   [num_pages, Hkv, page_size, D]   context keys / values of one layer
 *   page_table [B, max_pages_per_seq] int32   logical page i of sequence b lives in
 *                                      physical page page_table[b][i]
 *   ctx_len  [B] int32                 context positions per sequence
 *   logits   [B, S, V]                 denoiser logits of one step
 *   masked   [B, S] uint8              1 = position still [MASK]
 *   tokens   [B, S] int32              committed token ids (untouched while masked)
 * Query head h reads KV head h / (Hq / Hkv) (contiguous GQA groups).
 */
#ifndef TT_DENOISE_H
#define TT_DENOISE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TT_API __attribute__((visibility("default")))
#else
#define TT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *tt_stream_t; /* same type as cudaStream_t */

typedef enum {
    TT_OK = 0,
    TT_ERR_INVALID_ARG = 1,     /* NULL pointer, negative size, inconsistent arguments */
    TT_ERR_UNSUPPORTED = 2,     /* valid but not implemented (a shape, a dtype, alignment) */
    TT_ERR_CAPACITY = 3,        /* workspace too small, or a block does not fit its pages */
    TT_ERR_CUDA = 4,            /* a CUDA runtime / driver call failed */
    TT_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait gave up (device word only) */
    TT_ERR_BOUNDS = 6           /* a page id or a context length out of range (device word only) */
} tt_status;

typedef enum {
    TT_BF16 = 0,   /* bfloat16 storage, fp32 arithmetic */
    TT_FP32 = 1    /* float32 storage, fp32 arithmetic (parity mode) */
} tt_dtype;

/* One attention layer's paged context KV cache, as produced by the frozen
 * context tower ([ARCH]: layer-aligned KV caches reused across blocks).
 * All pointers are device pointers owned by the caller. */
typedef struct {
    void *k_pool;                /* [num_pages, n_kv_heads, page_size, head_dim] */
    void *v_pool;                /* same shape as k_pool */
    const int32_t *page_table;   /* [B, max_pages_per_seq] */
    int32_t *ctx_len;            /* [B]; read by attention, advanced by tt_kv_append */
    int32_t num_pages;
    int32_t max_pages_per_seq;   /* max_pages_per_seq * page_size <= 2^30 tokens, else
                                    every call returns TT_ERR_UNSUPPORTED */
    int32_t page_size;           /* tokens per page; 64 on the tensor-core path */
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t dtype;               /* tt_dtype; must equal the dtype of q / k_blk / out */
} tt_kv_cache;

/* Text of a status code (static storage, never NULL). */
TT_API const char *tt_status_string(tt_status s);

/* Library version as major*10000 + minor*100 + patch. */
TT_API int tt_version(void);

/* Bytes of workspace tt_denoise_attn needs for this shape (0 is possible).
 * Pure host arithmetic; no device is touched. */
TT_API tt_status tt_denoise_attn_workspace_size(int B, int S, int Hq, int Hkv, int D, tt_dtype dtype,
                                         size_t *bytes);

/* Two-segment attention of one denoiser layer ([ARCH], [GEN], [NEWS]).
 *
 * For every sequence b, block position i and query head h (KV head g = h / G):
 *   keys   = the L = ctx_len[b] context keys of layer ctx (logical order through
 *            the page table), followed by the S block keys k_blk[b, :, g];
 *   s_j    = sm_scale * <q[b,i,h], k_j>;   p = softmax(s) over all L + S keys;
 *   out[b,i,h] = sum_j p_j v_j;   lse[b,h,i] = log(sum_j exp(s_j)).
 * Every context position precedes the block, so the causal cross-attention
 * admits all L context keys to every block query; inside the block there is no
 * mask (bidirectional).  L may be 0 (attention within the block only).  Page
 * slots at or beyond L are never read into the result (they may hold any bits).
 *
 * ctx      host pointer to one tt_kv_cache (the struct is read on the host; the
 *          buffers it names are device memory)
 * q, k_blk, v_blk, out   device, layouts above, dtype ctx->dtype
 * lse      device [B, Hq, S] fp32 or NULL
 * sm_scale softmax scale (1/sqrt(D) is the usual choice)
 * max_ctas 0 = one persistent CTA per SM; k > 0 caps the number of CTAs that
 *          share the work (1 = no split of any sequence's context)
 * ws, ws_bytes  device workspace of at least tt_denoise_attn_workspace_size bytes
 *
 * S = 1 is one step of autoregressive decoding from the same cache (the token's
 * own key and value are the "block" keys): the baseline the pages compare the
 * block-wise diffusion against (dgnews.ru, "What the tests actually show").
 *
 * Supported: S >= 1, Hq % Hkv == 0, D in {32, 64, 128}.  With bf16, D = 128,
 * page_size = 64 and sm_scale > 0, two tensor-core kernels serve: S a multiple
 * of 16 up to 128 with (Hq/Hkv)*S a multiple of 128 up to 2048 (the block
 * kernel), and S = 1 with Hq/Hkv = 16 (the decode kernel; its workspace is sized
 * by the same function for S = 1).  Every other supported shape (and all of
 * fp32) runs on the CUDA-core kernel.  Other shapes return TT_ERR_UNSUPPORTED. */
TT_API tt_status tt_denoise_attn(const tt_kv_cache *ctx, const void *q, const void *k_blk,
                          const void *v_blk, void *out, float *lse, int B, int S, int Hq,
                          float sm_scale, int max_ctas, void *ws, size_t ws_bytes,
                          uint32_t *dev_err, tt_stream_t stream);

/* Attention of the frozen context tower over a committed block ([ARCH]: that
 * tower is a causal autoregressive model over the prompt and the committed
 * tokens; [GEN]: once a block is committed, the tower extends its state with
 * the clean block).
 *
 * Identical to tt_denoise_attn -- arguments, layouts, workspace (sized by
 * tt_denoise_attn_workspace_size), supported shapes, kernels and errors --
 * except for the view inside the block, which is causal:
 *   keys of block query i = the L = ctx_len[b] context keys, then the block
 *                           keys 0..i (L + i + 1 keys in all);
 *   p = softmax(s) over those keys;  out and lse as in tt_denoise_attn.
 * q, k_blk and v_blk are the context tower's projections of the block's clean
 * tokens for this layer; the k_blk and v_blk it attends to are the rows that
 * tt_kv_append then stores in the cache. */
TT_API tt_status tt_context_block_attn(const tt_kv_cache *ctx, const void *q, const void *k_blk,
                                const void *v_blk, void *out, float *lse, int B, int S, int Hq,
                                float sm_scale, int max_ctas, void *ws, size_t ws_bytes,
                                uint32_t *dev_err, tt_stream_t stream);

/* Bytes of workspace tt_unmask needs (pure host arithmetic). */
TT_API tt_status tt_unmask_workspace_size(int B, int S, int V, tt_dtype dtype, size_t *bytes);

/* Confidence unmasking of one denoise step ([SAMP]).
 *
 * For every sequence b and position p with masked[b,p] != 0 (locked positions
 * are skipped; their logits are never read):
 *   m = max_v logits[b,p,v];  Z = sum_v exp(logits[b,p,v] - m);
 *   conf[b,p] = 1 / Z  (the largest softmax probability);
 *   a = the lowest v with logits[b,p,v] == m.
 * Commit set C = { p masked : conf >= tau }.  If C is empty and a position is
 * masked, C = { the most confident masked position } (lowest p on ties).  If
 * step >= T, C = every masked position.  For p in C: tokens[b,p] = a,
 * masked[b,p] = 0, committed_now[b,p] = 1; every other position keeps its
 * token and mask and gets committed_now = 0.  n_masked[b] = masked positions
 * left.  conf[b,p] is NaN for positions that were already locked.
 *
 * logits   device [B, S, V], dtype bf16 or fp32 (finite, |value| < 2^127)
 * step     1-based step index; T >= 1 the step budget of a block
 * masked, tokens         device, in/out
 * committed_now          device [B,S] uint8 out (may be NULL)
 * conf                   device [B,S] fp32 out (may be NULL)
 * n_masked               device [B] int32 out (may be NULL)
 * Arithmetic: fp32; the maximum and argmax are exact, conf has a relative error
 * of a few 1e-7. */
TT_API tt_status tt_unmask(const void *logits, tt_dtype dtype, int B, int S, int V, float tau, int step,
                    int T, uint8_t *masked, int32_t *tokens, uint8_t *committed_now, float *conf,
                    int32_t *n_masked, void *ws, size_t ws_bytes, uint32_t *dev_err,
                    tt_stream_t stream);

/* Largest scratch, in bytes, that tt_unmask_noalloc can use (its file-scope device array). */
#define TT_UNMASK_NOALLOC_SCRATCH_BYTES (256u * 1024u)

/* tt_unmask for callers that cannot allocate device memory.  (The pages have no
 * counterpart of this call; it exists for deployment.)
 *
 * Some callers cannot call cudaMalloc or any allocator: code that runs while a
 * stream is being captured into a CUDA graph (allocation is not a capturable
 * operation), plugins and callbacks inside a serving framework that owns every
 * byte of device memory through its own pool, and real-time loops whose memory
 * is fixed at start-up.  This call takes no workspace: its scratch (the
 * per-chunk partials and the per-sequence counters) lives in one file-scope
 * device array of TT_UNMASK_NOALLOC_SCRATCH_BYTES, which every GPU that loads
 * the library holds until the process exits.  The caller still owns logits,
 * masked, tokens and the outputs.  Arguments and results are exactly those of
 * tt_unmask.
 *
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current); make that first call before any stream
 *    capture.  If that lookup fails the call returns TT_ERR_CUDA and the next
 *    call on the device tries again (nothing is latched on failure).
 *  - A shape whose scratch would exceed the array returns TT_ERR_CAPACITY before
 *    anything is launched (tt_unmask_workspace_size gives the need; about 82 KB
 *    for 32 sequences x 16 positions x 131072 bf16 logits).
 *  - Every call shares the one array and it keeps the last call's contents; the
 *    counters that must start at zero are cleared on the stream before each
 *    launch.  Calls that overlap on the GPU (different streams, or several host
 *    threads) race on the array and give wrong results: serialise them. */
TT_API tt_status tt_unmask_noalloc(const void *logits, tt_dtype dtype, int B, int S, int V, float tau,
                                   int step, int T, uint8_t *masked, int32_t *tokens,
                                   uint8_t *committed_now, float *conf, int32_t *n_masked,
                                   uint32_t *dev_err, tt_stream_t stream);

/* Corruption of clean blocks for the masked-diffusion objective ([T]: clean blocks
 * are corrupted by replacing tokens with [MASK] under a linear schedule).
 *
 * For every sequence b and position p: masked[b,p] = (u[b,p] < t[b]) -- each
 * position is masked independently with probability t[b] when u is uniform on
 * [0, 1) -- and, if noisy is not NULL, noisy[b,p] = mask_id where masked and
 * clean[b,p] elsewhere.  The uniform draws are the caller's (no random numbers are
 * drawn here).
 *
 * clean    device [B, S] int32 clean tokens (may be NULL when noisy is NULL)
 * u        device [B, S] fp32 uniform draws
 * t        device [B] fp32 diffusion times in [0, 1]; a sequence whose t lies
 *          outside (or is NaN) sets TT_ERR_BOUNDS in dev_err and its outputs are
 *          left untouched
 * noisy    device [B, S] int32 out or NULL;  masked  device [B, S] uint8 out */
TT_API tt_status tt_linear_schedule_mask(const int32_t *clean, const float *u, const float *t, int B, int S,
                                         int32_t mask_id, int32_t *noisy, uint8_t *masked, uint32_t *dev_err,
                                         tt_stream_t stream);

/* Bytes of workspace tt_masked_nll needs (pure host arithmetic). */
TT_API tt_status tt_masked_nll_workspace_size(int B, int S, int V, tt_dtype dtype, size_t *bytes);

/* Masked-diffusion loss of the denoiser's logits ([T]: the negative
 * log-likelihood of the original tokens at the masked positions).
 *
 * For every sequence b and position p with masked[b,p] != 0 and clean token
 * x = targets[b,p]:
 *   nll[b,p] = log sum_v exp(logits[b,p,v]) - logits[b,p,x]
 *            = (m - logits[b,p,x]) + log sum_v exp(logits[b,p,v] - m),  m = max_v;
 * nll_sum[b] = the sum of nll over the masked positions of b (no weighting; a
 * caller may weight per sequence), count[b] = their number.  Positions that are
 * not masked get nll = NaN and their logits are never read.
 *
 * logits   device [B, S, V], bf16 or fp32, finite with |value| < 2^127; the rows
 *          must be 16-byte aligned (base address and V * element size a multiple
 *          of 16), else TT_ERR_UNSUPPORTED
 * targets  device [B, S] int32; a masked position whose target lies outside
 *          [0, V) gets NaN and sets TT_ERR_BOUNDS in dev_err
 * masked   device [B, S] uint8 (as written by tt_linear_schedule_mask)
 * nll      device [B, S] fp32 out or NULL;  nll_sum  device [B] fp32 out or NULL;
 * count    device [B] int32 out or NULL
 * ws, ws_bytes  device workspace of at least tt_masked_nll_workspace_size bytes,
 *          zero-filled before its first use (left zeroed by every call)
 * Arithmetic: fp32; |nll - exact| <= 1e-5 * max(1, |nll|). */
TT_API tt_status tt_masked_nll(const void *logits, tt_dtype dtype, int B, int S, int V, const int32_t *targets,
                               const uint8_t *masked, float *nll, float *nll_sum, int32_t *count, void *ws,
                               size_t ws_bytes, uint32_t *dev_err, tt_stream_t stream);

/* Commit of a finished block into the context caches of n_layers layers ([GEN]:
 * the context tower extends its state with the clean tokens).
 *
 * For every sequence b with seq_active[b] != 0 (all, if seq_active is NULL) and
 * every layer l: context position L_b + s (s < S, L_b = ctx_len[b]) receives
 * k_new[l][b, s] / v_new[l][b, s] (page page_table[b][(L_b+s)/page_size], slot
 * (L_b+s) % page_size; the block may straddle pages); then ctx_len[b] += S, once.
 * All layers in one call must share the same ctx_len array (they hold the same
 * tokens) and the same shape; each layer has its own pools and may have its own
 * page table.  A block that does not fit max_pages_per_seq pages sets
 * TT_ERR_CAPACITY in dev_err and leaves that sequence untouched.
 *
 * layers   host array of n_layers tt_kv_cache structs (1 <= n_layers <= 16;
 *          more return TT_ERR_UNSUPPORTED, as do S > 1024 and rows of D
 *          elements that are not a multiple of 16 bytes)
 * k_new, v_new  host arrays of n_layers device pointers, each [B, S, Hkv, D],
 *          16-byte aligned like the pools
 * seq_active    device [B] uint8 or NULL */
TT_API tt_status tt_kv_append(const tt_kv_cache *layers, int n_layers, const void *const *k_new,
                       const void *const *v_new, const uint8_t *seq_active, int B, int S,
                       uint32_t *dev_err, tt_stream_t stream);

/* Bytes of workspace tt_block_step needs (attention + unmasking). */
TT_API tt_status tt_block_step_workspace_size(int B, int S, int Hq, int Hkv, int D, int V, tt_dtype dtype,
                                       size_t *bytes);

/* One denoiser step ([GEN]): tt_denoise_attn for each of the n_layers layers
 * (layer l reads q[l], k_blk[l], v_blk[l], ctx[l] and writes out[l]), then
 * tt_unmask on the step's logits.  All arrays of pointers are host arrays of
 * device pointers; arguments mean what they mean in the two calls above.  The
 * logits are an input: producing them needs the denoiser's weights, which are
 * outside this library. */
TT_API tt_status tt_block_step(const tt_kv_cache *ctx, int n_layers, const void *const *q,
                        const void *const *k_blk, const void *const *v_blk, void *const *out,
                        const void *logits, int B, int S, int Hq, int V, float tau, int step,
                        int T, float sm_scale, uint8_t *masked, int32_t *tokens,
                        uint8_t *committed_now, float *conf, int32_t *n_masked, void *ws,
                        size_t ws_bytes, uint32_t *dev_err, tt_stream_t stream);

/* Copy the device error word to *host_code after the stream's prior work has
 * finished (synchronises the stream).  The word is not cleared. */
TT_API tt_status tt_get_device_error(const uint32_t *dev_err, tt_stream_t stream, uint32_t *host_code);

/* Self-check of the failure path every kernel uses (the pages have no counterpart;
 * it exists so that a caller can see, without faulting or hanging a GPU, that a
 * wait that can never finish gives up and reports).  Launches one warp that waits
 * on a shared-memory mbarrier which nothing arrives at, polling it at most
 * `polls` times (1 <= polls <= 2^24) with the same bounded wait the kernels use,
 * then records TT_ERR_DEVICE_TIMEOUT in dev_err (device word, required) and
 * exits; the context stays usable.  Returns TT_ERR_INVALID_ARG for a bad
 * argument, TT_ERR_CUDA if the launch fails. */
TT_API tt_status tt_check_wait_timeout(uint32_t polls, uint32_t *dev_err, tt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TT_DENOISE_H */
