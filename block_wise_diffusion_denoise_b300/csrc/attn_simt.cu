// Two-segment denoise attention on CUDA cores (fp32 parity mode, and every
// shape the tensor-core kernel does not take).
//
// Visibility (TwoTower summary on gist.science, "Technisches Resuemee --
// Architektur"; dgnews.ru, "How the architecture actually works"): a block
// query attends to every key the context tower holds for its layer (all of them
// precede the block, so the causal cross-attention admits them all) and,
// without a mask, to every key of its own block.  In the context tower's view of
// a committed block (causal_block; the same summary: that tower is causal over
// the committed tokens) block query i reads the block keys 0..i only.
//
// One warp owns one (sequence, block position, query head) row.  Each lane
// holds D/32 consecutive dimensions, so a key or value row is one coalesced
// warp load.  Keys are taken four at a time through the page table (context)
// and then from the block; scores are reduced across the warp and folded into
// an online softmax in fp32 with full-precision expf, which keeps the fp32 mode
// within a few 1e-7 of the exact result.

#include <cmath>

#include "tt_common.cuh"
#include "tt_internal.h"

namespace tt {
namespace {

constexpr int kWarpsPerCta = 8;

struct SimtParams {
    const void *k_pool, *v_pool;
    const int32_t *page_table;
    const int32_t *ctx_len;
    int num_pages, max_pages, page_size;
    const void *q, *k_blk, *v_blk;
    void *out;
    float *lse;
    int B, S, Hq, Hkv, G;
    float sm_scale;
    int causal_block;
    uint32_t *dev_err;
};

template <typename T, int DPL> struct RowIO;

template <int DPL> struct RowIO<float, DPL> {
    static __device__ __forceinline__ void load(const float *p, float *x) {
        if constexpr (DPL == 4) {
            const float4 v = *reinterpret_cast<const float4 *>(p);
            x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
        } else if constexpr (DPL == 2) {
            const float2 v = *reinterpret_cast<const float2 *>(p);
            x[0] = v.x; x[1] = v.y;
        } else {
            x[0] = *p;
        }
    }
    static __device__ __forceinline__ void store(float *p, const float *x) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) p[i] = x[i];
    }
};

template <int DPL> struct RowIO<uint16_t, DPL> {
    static __device__ __forceinline__ void load(const uint16_t *p, float *x) {
        if constexpr (DPL == 4) {
            const uint2 v = *reinterpret_cast<const uint2 *>(p);
            x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        } else if constexpr (DPL == 2) {
            const uint32_t v = *reinterpret_cast<const uint32_t *>(p);
            x[0] = bf16_lo(v); x[1] = bf16_hi(v);
        } else {
            x[0] = bf16_bits_to_f32(*p);
        }
    }
    static __device__ __forceinline__ void store(uint16_t *p, const float *x) {
#pragma unroll
        for (int i = 0; i < DPL; ++i) p[i] = (uint16_t)f32_to_bf16_bits(x[i]);
    }
};

template <typename T, int DPL>
__global__ void __launch_bounds__(kWarpsPerCta * 32) attn_simt_kernel(const SimtParams p) {
    constexpr int D = DPL * 32;
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    const long long rows = (long long)p.B * p.S * p.Hq;
    if (gw >= rows) return;
    const int h = (int)(gw % p.Hq);
    const int i = (int)((gw / p.Hq) % p.S);
    const int b = (int)(gw / ((long long)p.Hq * p.S));
    const int g = h / p.G;

    int L = p.ctx_len[b];
    if (L < 0 || L > p.max_pages * p.page_size) {
        if (lane == 0) report_error(p.dev_err, TT_ERR_BOUNDS);
        L = 0;
    }
    const T *kp = static_cast<const T *>(p.k_pool);
    const T *vp = static_cast<const T *>(p.v_pool);
    const T *kb = static_cast<const T *>(p.k_blk);
    const T *vb = static_cast<const T *>(p.v_blk);

    float q[DPL];
    RowIO<T, DPL>::load(static_cast<const T *>(p.q) + (((size_t)b * p.S + i) * p.Hq + h) * D + lane * DPL, q);
#pragma unroll
    for (int d = 0; d < DPL; ++d) q[d] *= p.sm_scale;

    // Address of key / value row j of this sequence and KV head (context first, then block).
    auto row_off = [&](int j, bool &ok) -> size_t {
        if (j < L) {
            const int pg = p.page_table[(size_t)b * p.max_pages + j / p.page_size];
            ok = (pg >= 0 && pg < p.num_pages);
            return (((size_t)(ok ? pg : 0) * p.Hkv + g) * p.page_size + j % p.page_size) * D;
        }
        ok = true;
        return (((size_t)b * p.S + (j - L)) * p.Hkv + g) * D;
    };

    float m = -INFINITY, l = 0.f;
    float o[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[d] = 0.f;
    bool bad = false;
    const int n_keys = L + (p.causal_block ? i + 1 : p.S);
    for (int j0 = 0; j0 < n_keys; j0 += 4) {
        float s[4];
        float v[4][DPL];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = j0 + u;
            s[u] = -INFINITY;
#pragma unroll
            for (int d = 0; d < DPL; ++d) v[u][d] = 0.f;
            if (j < n_keys) {
                bool ok;
                const size_t off = row_off(j, ok);
                bad |= !ok;
                float k[DPL];
#pragma unroll
                for (int d = 0; d < DPL; ++d) k[d] = 0.f;
                if (ok) {   // a page id outside the pool is never dereferenced
                    RowIO<T, DPL>::load((j < L ? kp : kb) + off + lane * DPL, k);
                    RowIO<T, DPL>::load((j < L ? vp : vb) + off + lane * DPL, v[u]);
                }
                float acc = 0.f;
#pragma unroll
                for (int d = 0; d < DPL; ++d) acc = fmaf(q[d], k[d], acc);
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2);
                s[u] = ok ? acc : -INFINITY;
            }
        }
        const float mn = fmaxf(fmaxf(m, fmaxf(s[0], s[1])), fmaxf(s[2], s[3]));
        const float alpha = (m == -INFINITY) ? 0.f : expf(m - mn);
        float pw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) pw[u] = (s[u] == -INFINITY) ? 0.f : expf(s[u] - mn);
        l = l * alpha + ((pw[0] + pw[1]) + (pw[2] + pw[3]));
#pragma unroll
        for (int d = 0; d < DPL; ++d) {
            float acc = o[d] * alpha;
#pragma unroll
            for (int u = 0; u < 4; ++u) acc = fmaf(pw[u], v[u][d], acc);
            o[d] = acc;
        }
        m = mn;
    }
    if (bad && lane == 0) report_error(p.dev_err, TT_ERR_BOUNDS);
    const float inv = 1.f / l;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[d] *= inv;
    RowIO<T, DPL>::store(static_cast<T *>(p.out) + (((size_t)b * p.S + i) * p.Hq + h) * D + lane * DPL, o);
    if (p.lse != nullptr && lane == 0) p.lse[((size_t)b * p.Hq + h) * p.S + i] = m + logf(l);
}

template <typename T>
tt_status launch_typed(const SimtParams &p, int D, cudaStream_t stream) {
    const long long rows = (long long)p.B * p.S * p.Hq;
    const long long ctas = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
    if (ctas > 0x7fffffffLL) return TT_ERR_UNSUPPORTED;
    const dim3 grid((unsigned)ctas), block(kWarpsPerCta * 32);
    switch (D) {
        case 32: attn_simt_kernel<T, 1><<<grid, block, 0, stream>>>(p); break;
        case 64: attn_simt_kernel<T, 2><<<grid, block, 0, stream>>>(p); break;
        case 128: attn_simt_kernel<T, 4><<<grid, block, 0, stream>>>(p); break;
        default: return TT_ERR_UNSUPPORTED;
    }
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace

tt_status launch_attn_simt(const AttnArgs &a) {
    SimtParams p;
    p.k_pool = a.ctx->k_pool; p.v_pool = a.ctx->v_pool;
    p.page_table = a.ctx->page_table; p.ctx_len = a.ctx->ctx_len;
    p.num_pages = a.ctx->num_pages; p.max_pages = a.ctx->max_pages_per_seq;
    p.page_size = a.ctx->page_size;
    p.q = a.q; p.k_blk = a.k_blk; p.v_blk = a.v_blk; p.out = a.out; p.lse = a.lse;
    p.B = a.B; p.S = a.S; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = a.Hq / a.Hkv;
    p.sm_scale = a.sm_scale;
    p.causal_block = a.causal_block ? 1 : 0;
    p.dev_err = a.dev_err;
    if (p.B == 0) return TT_OK;
    return a.ctx->dtype == TT_BF16 ? launch_typed<uint16_t>(p, a.D, a.stream)
                                   : launch_typed<float>(p, a.D, a.stream);
}

}  // namespace tt
