// Commit of a finished block into the paged context caches (tt_kv_append).
//
// TwoTower summary on gist.science, "Generierungsprozess": once a block is
// committed the context tower updates its state with the clean tokens.  Here
// that update is the append of the block's per-layer keys and values at context
// positions L_b .. L_b + S - 1 (the KV themselves come from the context tower,
// which is outside this library).
//
// One CTA per sequence copies the block of every layer with 16-byte loads and
// stores (each (position, head) row of D elements is contiguous in both the
// source and the page), then advances the shared length once.  Positions are
// resolved through the page table, so a block may straddle a page boundary.

#include "tt_common.cuh"
#include "tt_internal.h"

namespace tt {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxLayers = 16;

struct AppendLayer {
    char *k_pool, *v_pool;
    const int32_t *page_table;
    const char *k_new, *v_new;
};

struct AppendParams {
    AppendLayer layer[kMaxLayers];
    int n_layers;
    int32_t *ctx_len;
    const uint8_t *seq_active;
    int B, S, Hkv, page_size, max_pages, num_pages;
    int row_vecs;        // 16-byte vectors per (position, head) row
    uint32_t *dev_err;
};

__global__ void __launch_bounds__(kThreads) kv_append_kernel(const __grid_constant__ AppendParams p) {
    const int b = blockIdx.x;
    if (p.seq_active != nullptr && p.seq_active[b] == 0) return;
    const int L = p.ctx_len[b];
    if (L < 0 || (long long)L + p.S > (long long)p.max_pages * p.page_size) {
        if (threadIdx.x == 0) report_error(p.dev_err, L < 0 ? TT_ERR_BOUNDS : TT_ERR_CAPACITY);
        return;
    }
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    // Validate every page the block touches before writing anything.
    for (int l = 0; l < p.n_layers; ++l) {
        for (int s = threadIdx.x; s < p.S; s += kThreads) {
            const int pg = p.layer[l].page_table[(size_t)b * p.max_pages + (L + s) / p.page_size];
            if (pg < 0 || pg >= p.num_pages) s_bad = 1;
        }
    }
    __syncthreads();
    if (s_bad) {
        if (threadIdx.x == 0) report_error(p.dev_err, TT_ERR_BOUNDS);
        return;
    }
    const int per_layer = p.S * p.Hkv * p.row_vecs;   // vectors of K (and of V) per layer
    for (int l = 0; l < p.n_layers; ++l) {
        const AppendLayer &ly = p.layer[l];
        for (int i = threadIdx.x; i < per_layer; i += kThreads) {
            const int v = i % p.row_vecs;
            const int h = (i / p.row_vecs) % p.Hkv;
            const int s = i / (p.row_vecs * p.Hkv);
            const int j = L + s;
            const int pg = ly.page_table[(size_t)b * p.max_pages + j / p.page_size];
            const size_t src = (((size_t)b * p.S + s) * p.Hkv + h) * p.row_vecs + v;
            const size_t dst = (((size_t)pg * p.Hkv + h) * p.page_size + j % p.page_size) * p.row_vecs + v;
            const uint4 kv = __ldg(reinterpret_cast<const uint4 *>(ly.k_new) + src);
            const uint4 vv = __ldg(reinterpret_cast<const uint4 *>(ly.v_new) + src);
            reinterpret_cast<uint4 *>(ly.k_pool)[dst] = kv;
            reinterpret_cast<uint4 *>(ly.v_pool)[dst] = vv;
        }
    }
    __syncthreads();   // every thread has read L before it changes
    if (threadIdx.x == 0) p.ctx_len[b] = L + p.S;
}

}  // namespace

tt_status launch_kv_append(const tt_kv_cache *layers, int n_layers, const void *const *k_new,
                           const void *const *v_new, const uint8_t *seq_active, int B, int S,
                           uint32_t *dev_err, cudaStream_t stream) {
    if (n_layers > kMaxLayers) return TT_ERR_UNSUPPORTED;
    const tt_kv_cache &c0 = layers[0];
    const size_t elem = c0.dtype == TT_BF16 ? 2 : 4;
    const size_t row_bytes = (size_t)c0.head_dim * elem;
    if (row_bytes % 16 != 0) return TT_ERR_UNSUPPORTED;
    AppendParams p = {};
    for (int l = 0; l < n_layers; ++l) {
        p.layer[l].k_pool = static_cast<char *>(layers[l].k_pool);
        p.layer[l].v_pool = static_cast<char *>(layers[l].v_pool);
        p.layer[l].page_table = layers[l].page_table;
        p.layer[l].k_new = static_cast<const char *>(k_new[l]);
        p.layer[l].v_new = static_cast<const char *>(v_new[l]);
        const uintptr_t al = reinterpret_cast<uintptr_t>(layers[l].k_pool) |
                             reinterpret_cast<uintptr_t>(layers[l].v_pool) |
                             reinterpret_cast<uintptr_t>(k_new[l]) |
                             reinterpret_cast<uintptr_t>(v_new[l]);
        if (al % 16 != 0) return TT_ERR_UNSUPPORTED;
    }
    p.n_layers = n_layers;
    p.ctx_len = c0.ctx_len;
    p.seq_active = seq_active;
    p.B = B; p.S = S; p.Hkv = c0.n_kv_heads; p.page_size = c0.page_size;
    p.max_pages = c0.max_pages_per_seq; p.num_pages = c0.num_pages;
    p.row_vecs = (int)(row_bytes / 16);
    p.dev_err = dev_err;
    kv_append_kernel<<<B, kThreads, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace tt
