// C-ABI entry points: argument validation, workspace sizing and dispatch.
// Declarations and the meaning of every argument: include/tt_denoise.h.

#include <cmath>
#include <cstring>

#include "tt_internal.h"

using namespace tt;

namespace {

constexpr int kMaxS = 1024;
// Context capacity per sequence: keeps every length sum in the kernels (a length plus a
// block, a length rounded up to a tile) inside 32-bit integers.
constexpr long long kMaxCtxTokens = 1LL << 30;

bool dtype_ok(int d) { return d == TT_BF16 || d == TT_FP32; }
bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

tt_status check_cache(const tt_kv_cache *c) {
    if (c == nullptr) return TT_ERR_INVALID_ARG;
    if (!dtype_ok(c->dtype)) return TT_ERR_INVALID_ARG;
    if (c->page_size < 1 || c->n_kv_heads < 1 || c->head_dim < 1 || c->num_pages < 0 ||
        c->max_pages_per_seq < 1)
        return TT_ERR_INVALID_ARG;
    if (c->page_table == nullptr || c->ctx_len == nullptr) return TT_ERR_INVALID_ARG;
    if (c->num_pages > 0 && (c->k_pool == nullptr || c->v_pool == nullptr)) return TT_ERR_INVALID_ARG;
    if ((long long)c->max_pages_per_seq * c->page_size > kMaxCtxTokens) return TT_ERR_UNSUPPORTED;
    if (c->num_pages > 0 && (!aligned16(c->k_pool) || !aligned16(c->v_pool))) return TT_ERR_UNSUPPORTED;
    return TT_OK;
}

tt_status attn_shape(int B, int S, int Hq, int Hkv, int D, int dtype) {
    if (B < 0 || S < 1 || Hq < 1 || Hkv < 1 || D < 1 || !dtype_ok(dtype)) return TT_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return TT_ERR_INVALID_ARG;
    if (S > kMaxS) return TT_ERR_UNSUPPORTED;
    if (D != 32 && D != 64 && D != 128) return TT_ERR_UNSUPPORTED;
    return TT_OK;
}

}  // namespace

extern "C" {

const char *tt_status_string(tt_status s) {
    switch (s) {
        case TT_OK: return "ok";
        case TT_ERR_INVALID_ARG: return "invalid argument";
        case TT_ERR_UNSUPPORTED: return "unsupported shape, dtype or alignment";
        case TT_ERR_CAPACITY: return "insufficient capacity (workspace or pages)";
        case TT_ERR_CUDA: return "CUDA call failed";
        case TT_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case TT_ERR_BOUNDS: return "page id or context length out of range";
    }
    return "unknown status";
}

int tt_version(void) { return 1 * 10000 + 0 * 100 + 0; }

tt_status tt_denoise_attn_workspace_size(int B, int S, int Hq, int Hkv, int D, tt_dtype dtype,
                                         size_t *bytes) {
    if (bytes == nullptr) return TT_ERR_INVALID_ARG;
    *bytes = 0;
    const tt_status st = attn_shape(B, S, Hq, Hkv, D, dtype);
    if (st != TT_OK) return st;
    // The tensor-core kernels need split partials; page size is checked at call time,
    // so size for them whenever the rest of the shape qualifies.
    if (attn_tc_supported(S, Hq, Hkv, D, 64, dtype)) *bytes = attn_tc_ws_bytes(B, S, Hq, Hkv, D);
    if (attn_decode_supported(S, Hq, Hkv, D, 64, dtype)) *bytes = attn_decode_ws_bytes(B, Hkv);
    return TT_OK;
}

}  // extern "C"

namespace {

// The two attention entry points differ only in the view inside the block.
tt_status attention(const tt_kv_cache *ctx, const void *q, const void *k_blk, const void *v_blk,
                    void *out, float *lse, int B, int S, int Hq, float sm_scale, int max_ctas,
                    void *ws, size_t ws_bytes, uint32_t *dev_err, tt_stream_t stream,
                    bool causal_block) {
    tt_status st = check_cache(ctx);
    if (st != TT_OK) return st;
    st = attn_shape(B, S, Hq, ctx->n_kv_heads, ctx->head_dim, ctx->dtype);
    if (st != TT_OK) return st;
    if (!std::isfinite(sm_scale) || max_ctas < 0) return TT_ERR_INVALID_ARG;
    if (B == 0) return TT_OK;
    if (q == nullptr || k_blk == nullptr || v_blk == nullptr || out == nullptr) return TT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(out)) return TT_ERR_UNSUPPORTED;
    AttnArgs a;
    a.ctx = ctx; a.q = q; a.k_blk = k_blk; a.v_blk = v_blk; a.out = out; a.lse = lse;
    a.B = B; a.S = S; a.Hq = Hq; a.Hkv = ctx->n_kv_heads; a.D = ctx->head_dim;
    a.sm_scale = sm_scale; a.causal_block = causal_block;
    a.max_ctas = max_ctas; a.ws = ws; a.ws_bytes = ws_bytes;
    a.dev_err = dev_err; a.stream = reinterpret_cast<cudaStream_t>(stream);
    if (attn_tc_supported(S, Hq, a.Hkv, a.D, ctx->page_size, (tt_dtype)ctx->dtype) && sm_scale > 0.f) {
        const size_t need = attn_tc_ws_bytes(B, S, Hq, a.Hkv, a.D);
        if (need > 0 && (ws == nullptr || ws_bytes < need)) return TT_ERR_CAPACITY;
        if (need > 0 && reinterpret_cast<uintptr_t>(ws) % 256 != 0) return TT_ERR_UNSUPPORTED;
        return launch_attn_tc(a);
    }
    if (attn_decode_supported(S, Hq, a.Hkv, a.D, ctx->page_size, (tt_dtype)ctx->dtype) && sm_scale > 0.f) {
        const size_t need = attn_decode_ws_bytes(B, a.Hkv);
        if (ws == nullptr || ws_bytes < need) return TT_ERR_CAPACITY;
        if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return TT_ERR_UNSUPPORTED;
        return launch_attn_decode(a);
    }
    return launch_attn_simt(a);
}

}  // namespace

extern "C" {

tt_status tt_denoise_attn(const tt_kv_cache *ctx, const void *q, const void *k_blk,
                          const void *v_blk, void *out, float *lse, int B, int S, int Hq,
                          float sm_scale, int max_ctas, void *ws, size_t ws_bytes,
                          uint32_t *dev_err, tt_stream_t stream) {
    return attention(ctx, q, k_blk, v_blk, out, lse, B, S, Hq, sm_scale, max_ctas, ws, ws_bytes,
                     dev_err, stream, false);
}

tt_status tt_context_block_attn(const tt_kv_cache *ctx, const void *q, const void *k_blk,
                                const void *v_blk, void *out, float *lse, int B, int S, int Hq,
                                float sm_scale, int max_ctas, void *ws, size_t ws_bytes,
                                uint32_t *dev_err, tt_stream_t stream) {
    return attention(ctx, q, k_blk, v_blk, out, lse, B, S, Hq, sm_scale, max_ctas, ws, ws_bytes,
                     dev_err, stream, true);
}

tt_status tt_unmask_workspace_size(int B, int S, int V, tt_dtype dtype, size_t *bytes) {
    if (bytes == nullptr) return TT_ERR_INVALID_ARG;
    *bytes = 0;
    if (B < 0 || S < 1 || V < 1 || !dtype_ok(dtype)) return TT_ERR_INVALID_ARG;
    if (S > kMaxS) return TT_ERR_UNSUPPORTED;
    *bytes = unmask_ws_bytes(B, S, V, dtype);
    return TT_OK;
}

tt_status tt_unmask(const void *logits, tt_dtype dtype, int B, int S, int V, float tau, int step,
                    int T, uint8_t *masked, int32_t *tokens, uint8_t *committed_now, float *conf,
                    int32_t *n_masked, void *ws, size_t ws_bytes, uint32_t *dev_err,
                    tt_stream_t stream) {
    if (B < 0 || S < 1 || V < 1 || !dtype_ok(dtype) || step < 1 || T < 1 || std::isnan(tau))
        return TT_ERR_INVALID_ARG;
    if (S > kMaxS) return TT_ERR_UNSUPPORTED;
    if (B == 0) return TT_OK;
    if (logits == nullptr || masked == nullptr || tokens == nullptr) return TT_ERR_INVALID_ARG;
    const size_t need = unmask_ws_bytes(B, S, V, dtype);
    if (ws == nullptr || ws_bytes < need) return TT_ERR_CAPACITY;
    if (reinterpret_cast<uintptr_t>(ws) % 16 != 0) return TT_ERR_UNSUPPORTED;
    if (B > 65535) return TT_ERR_UNSUPPORTED;   // the chunked kernel's grid limit
    return launch_unmask(logits, dtype, B, S, V, tau, step, T, masked, tokens, committed_now, conf,
                         n_masked, ws, dev_err, reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_unmask_noalloc(const void *logits, tt_dtype dtype, int B, int S, int V, float tau, int step,
                            int T, uint8_t *masked, int32_t *tokens, uint8_t *committed_now, float *conf,
                            int32_t *n_masked, uint32_t *dev_err, tt_stream_t stream) {
    if (B < 0 || S < 1 || V < 1 || !dtype_ok(dtype) || step < 1 || T < 1 || std::isnan(tau))
        return TT_ERR_INVALID_ARG;
    if (S > kMaxS) return TT_ERR_UNSUPPORTED;
    if (B == 0) return TT_OK;
    if (logits == nullptr || masked == nullptr || tokens == nullptr) return TT_ERR_INVALID_ARG;
    if (B > 65535) return TT_ERR_UNSUPPORTED;
    return launch_unmask_noalloc(logits, dtype, B, S, V, tau, step, T, masked, tokens, committed_now, conf,
                                 n_masked, dev_err, reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_linear_schedule_mask(const int32_t *clean, const float *u, const float *t, int B, int S,
                                  int32_t mask_id, int32_t *noisy, uint8_t *masked, uint32_t *dev_err,
                                  tt_stream_t stream) {
    if (B < 0 || S < 1) return TT_ERR_INVALID_ARG;
    if (B == 0) return TT_OK;
    if (u == nullptr || t == nullptr || masked == nullptr || (noisy != nullptr && clean == nullptr))
        return TT_ERR_INVALID_ARG;
    return launch_linear_schedule(clean, u, t, B, S, mask_id, noisy, masked, dev_err,
                                  reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_masked_nll_workspace_size(int B, int S, int V, tt_dtype dtype, size_t *bytes) {
    if (bytes == nullptr) return TT_ERR_INVALID_ARG;
    *bytes = 0;
    if (B < 0 || S < 1 || V < 1 || !dtype_ok(dtype)) return TT_ERR_INVALID_ARG;
    if (S > kMaxS) return TT_ERR_UNSUPPORTED;
    *bytes = masked_nll_ws_bytes(B, S, V, dtype);
    return TT_OK;
}

tt_status tt_masked_nll(const void *logits, tt_dtype dtype, int B, int S, int V, const int32_t *targets,
                        const uint8_t *masked, float *nll, float *nll_sum, int32_t *count, void *ws,
                        size_t ws_bytes, uint32_t *dev_err, tt_stream_t stream) {
    if (B < 0 || S < 1 || V < 1 || !dtype_ok(dtype)) return TT_ERR_INVALID_ARG;
    if (S > kMaxS) return TT_ERR_UNSUPPORTED;
    if (B == 0) return TT_OK;
    if (logits == nullptr || targets == nullptr || masked == nullptr) return TT_ERR_INVALID_ARG;
    const size_t need = masked_nll_ws_bytes(B, S, V, dtype);
    if (ws == nullptr || ws_bytes < need) return TT_ERR_CAPACITY;
    if (reinterpret_cast<uintptr_t>(ws) % 16 != 0) return TT_ERR_UNSUPPORTED;
    return launch_masked_nll(logits, dtype, B, S, V, targets, masked, nll, nll_sum, count, ws, dev_err,
                             reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_kv_append(const tt_kv_cache *layers, int n_layers, const void *const *k_new,
                       const void *const *v_new, const uint8_t *seq_active, int B, int S,
                       uint32_t *dev_err, tt_stream_t stream) {
    if (layers == nullptr || n_layers < 1 || k_new == nullptr || v_new == nullptr || B < 0 || S < 1)
        return TT_ERR_INVALID_ARG;
    if (S > kMaxS) return TT_ERR_UNSUPPORTED;
    for (int l = 0; l < n_layers; ++l) {
        const tt_status st = check_cache(&layers[l]);
        if (st != TT_OK) return st;
        const tt_kv_cache &a = layers[0], &c = layers[l];
        if (c.ctx_len != a.ctx_len || c.dtype != a.dtype || c.page_size != a.page_size ||
            c.n_kv_heads != a.n_kv_heads || c.head_dim != a.head_dim ||
            c.num_pages != a.num_pages || c.max_pages_per_seq != a.max_pages_per_seq)
            return TT_ERR_INVALID_ARG;
        if (B > 0 && (k_new[l] == nullptr || v_new[l] == nullptr || c.num_pages == 0))
            return TT_ERR_INVALID_ARG;
    }
    if (B == 0) return TT_OK;
    return launch_kv_append(layers, n_layers, k_new, v_new, seq_active, B, S, dev_err,
                            reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_block_step_workspace_size(int B, int S, int Hq, int Hkv, int D, int V, tt_dtype dtype,
                                       size_t *bytes) {
    if (bytes == nullptr) return TT_ERR_INVALID_ARG;
    *bytes = 0;
    size_t a = 0, u = 0;
    tt_status st = tt_denoise_attn_workspace_size(B, S, Hq, Hkv, D, dtype, &a);
    if (st != TT_OK) return st;
    st = tt_unmask_workspace_size(B, S, V, dtype, &u);
    if (st != TT_OK) return st;
    *bytes = align_up(a, 256) + u;
    return TT_OK;
}

tt_status tt_block_step(const tt_kv_cache *ctx, int n_layers, const void *const *q,
                        const void *const *k_blk, const void *const *v_blk, void *const *out,
                        const void *logits, int B, int S, int Hq, int V, float tau, int step,
                        int T, float sm_scale, uint8_t *masked, int32_t *tokens,
                        uint8_t *committed_now, float *conf, int32_t *n_masked, void *ws,
                        size_t ws_bytes, uint32_t *dev_err, tt_stream_t stream) {
    if (ctx == nullptr || n_layers < 1 || q == nullptr || k_blk == nullptr || v_blk == nullptr ||
        out == nullptr)
        return TT_ERR_INVALID_ARG;
    const tt_kv_cache &c0 = ctx[0];
    tt_status st = check_cache(&c0);
    if (st != TT_OK) return st;
    size_t attn_ws = 0, total = 0;
    st = tt_denoise_attn_workspace_size(B, S, Hq, c0.n_kv_heads, c0.head_dim, (tt_dtype)c0.dtype,
                                        &attn_ws);
    if (st != TT_OK) return st;
    st = tt_block_step_workspace_size(B, S, Hq, c0.n_kv_heads, c0.head_dim, V, (tt_dtype)c0.dtype,
                                      &total);
    if (st != TT_OK) return st;
    if (B > 0 && (ws == nullptr || ws_bytes < total)) return TT_ERR_CAPACITY;
    // Validate the unmasking arguments before launching any attention layer.
    if (step < 1 || T < 1 || std::isnan(tau) || V < 1) return TT_ERR_INVALID_ARG;
    if (B > 0 && (logits == nullptr || masked == nullptr || tokens == nullptr)) return TT_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l) {
        st = check_cache(&ctx[l]);
        if (st != TT_OK) return st;
        if (ctx[l].dtype != c0.dtype || ctx[l].head_dim != c0.head_dim ||
            ctx[l].n_kv_heads != c0.n_kv_heads)
            return TT_ERR_INVALID_ARG;
    }
    const size_t attn_region = align_up(attn_ws, 256);
    for (int l = 0; l < n_layers; ++l) {
        st = tt_denoise_attn(&ctx[l], q[l], k_blk[l], v_blk[l], out[l], nullptr, B, S, Hq, sm_scale,
                             0, ws, attn_ws, dev_err, stream);
        if (st != TT_OK) return st;
    }
    void *uws = static_cast<char *>(ws) + attn_region;
    return tt_unmask(logits, (tt_dtype)c0.dtype, B, S, V, tau, step, T, masked, tokens,
                     committed_now, conf, n_masked, uws, ws_bytes - attn_region, dev_err, stream);
}

tt_status tt_check_wait_timeout(uint32_t polls, uint32_t *dev_err, tt_stream_t stream) {
    if (dev_err == nullptr || polls < 1 || polls > (1u << 24)) return TT_ERR_INVALID_ARG;
    return tt::launch_wait_check(polls, dev_err, reinterpret_cast<cudaStream_t>(stream));
}

tt_status tt_get_device_error(const uint32_t *dev_err, tt_stream_t stream, uint32_t *host_code) {
    if (dev_err == nullptr || host_code == nullptr) return TT_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_code, dev_err, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return TT_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return TT_ERR_CUDA;
    return TT_OK;
}

}  // extern "C"
