// Internal launchers shared by the C-ABI layer and the kernel files (host side).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/tt_denoise.h"

namespace tt {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- unmasking
struct UnmaskPartial {   // one (row, chunk) of the vocabulary
    float m;             // chunk maximum
    float z;             // sum of exp(x - m) over the chunk
    int32_t arg;         // lowest index of the maximum
    int32_t pad;
};

int unmask_chunk_elems(tt_dtype dtype);
size_t unmask_ws_bytes(int B, int S, int V, tt_dtype dtype);
tt_status launch_unmask(const void *logits, tt_dtype dtype, int B, int S, int V, float tau,
                        int step, int T, uint8_t *masked, int32_t *tokens, uint8_t *committed_now,
                        float *conf, int32_t *n_masked, void *ws, uint32_t *dev_err,
                        cudaStream_t stream);

tt_status launch_unmask_noalloc(const void *logits, tt_dtype dtype, int B, int S, int V, float tau,
                                int step, int T, uint8_t *masked, int32_t *tokens,
                                uint8_t *committed_now, float *conf, int32_t *n_masked,
                                uint32_t *dev_err, cudaStream_t stream);

// ---------------------------------------------------------------- masked-diffusion loss
size_t masked_nll_ws_bytes(int B, int S, int V, tt_dtype dtype);
tt_status launch_masked_nll(const void *logits, tt_dtype dtype, int B, int S, int V, const int32_t *targets,
                            const uint8_t *masked, float *nll, float *nll_sum, int32_t *count, void *ws,
                            uint32_t *dev_err, cudaStream_t stream);
tt_status launch_linear_schedule(const int32_t *clean, const float *u, const float *t, int B, int S,
                                 int32_t mask_id, int32_t *noisy, uint8_t *masked, uint32_t *dev_err,
                                 cudaStream_t stream);

// ---------------------------------------------------------------- append
tt_status launch_kv_append(const tt_kv_cache *layers, int n_layers, const void *const *k_new,
                           const void *const *v_new, const uint8_t *seq_active, int B, int S,
                           uint32_t *dev_err, cudaStream_t stream);

// ---------------------------------------------------------------- attention
struct AttnArgs {
    const tt_kv_cache *ctx;
    const void *q, *k_blk, *v_blk;
    void *out;
    float *lse;
    int B, S, Hq, Hkv, D;
    float sm_scale;
    bool causal_block;   // block query i sees block keys 0..i only (else all S)
    int max_ctas;
    void *ws;
    size_t ws_bytes;
    uint32_t *dev_err;
    cudaStream_t stream;
};

tt_status launch_attn_simt(const AttnArgs &a);

bool attn_tc_supported(int S, int Hq, int Hkv, int D, int page_size, tt_dtype dtype);
size_t attn_tc_ws_bytes(int B, int S, int Hq, int Hkv, int D);
tt_status launch_attn_tc(const AttnArgs &a);

// Single-position queries (S = 1) with 16 query heads per KV head: the decode kernel.
bool attn_decode_supported(int S, int Hq, int Hkv, int D, int page_size, tt_dtype dtype);
size_t attn_decode_ws_bytes(int B, int Hkv);
tt_status launch_attn_decode(const AttnArgs &a);

// One warp waits (bounded) on an mbarrier nothing arrives at and reports the timeout.
tt_status launch_wait_check(uint32_t polls, uint32_t *dev_err, cudaStream_t stream);

}  // namespace tt
