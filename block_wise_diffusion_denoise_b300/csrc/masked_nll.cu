// The masked-diffusion objective of the denoiser (tt_linear_schedule_mask, tt_masked_nll).
//
// TwoTower summary on gist.science, "Training und Konditionierung -- Maskierte
// Diffusion": clean blocks are corrupted by replacing tokens with [MASK] under a
// linear schedule, and the denoiser is trained to minimise the negative
// log-likelihood of the original tokens at the masked positions.
//
//  * Corruption: at diffusion time t (one per sequence) each position is masked
//    independently with probability t; the uniform draws u are inputs, and a
//    position is masked exactly when u < t.  One thread per position.
//  * Loss: for every masked position p with clean token x_p,
//        nll_p = log sum_v exp(l_{p,v}) - l_{p,x_p} = (m - l_{p,x_p}) + log Z,
//    with m the row maximum and Z = sum_v exp(l_{p,v} - m).  (m, Z) come from the
//    streaming pass over the vocabulary shared with the unmasking (vocab_stream.cuh,
//    the argmax is simply not used); its Finish policy below gathers the target
//    logit, forms nll_p and the per-sequence sum (a fixed-order reduction) and count.

#include <cmath>

#include "tt_common.cuh"
#include "tt_internal.h"
#include "vocab_stream.cuh"

namespace tt {
namespace {

struct NllFin {
    struct Params {
        const int32_t *targets;    // [B, S] clean tokens
        float *nll;                // [B, S] or NULL
        float *nll_sum;            // [B] or NULL
        int32_t *count;            // [B] or NULL
        int bf16;                  // logits are bf16 (else fp32)
    };

    // mk: the sequence's masked flags (a copy in shared memory, or the array itself)
    static __device__ void finish(const vs::Common &c, const Params &f, int b, const uint8_t *mk) {
        const int lane = threadIdx.x & 31;
        float sum = 0.f;
        int cnt = 0;
        for (int p = lane; p < c.S; p += 32) {
            const size_t rr = (size_t)b * c.S + p;
            if (mk[p] == 0) {   // not masked: not in the loss, its logits are not read
                if (f.nll) f.nll[rr] = NAN;
                continue;
            }
            const int t = f.targets[rr];
            float lt = NAN;
            if (t >= 0 && t < c.V) {
                const size_t off = rr * (size_t)c.V + (size_t)t;
                lt = f.bf16 ? bf16_bits_to_f32(static_cast<const uint16_t *>(c.logits)[off])
                            : static_cast<const float *>(c.logits)[off];
            } else {
                report_error(c.dev_err, TT_ERR_BOUNDS);
            }
            float m, z;
            int a;
            vs::row_state(c, (long long)rr, m, z, a);
            // the exact value is never below 0 (log sum exp >= every logit); fp32 rounding of a
            // sum that is 1 to within an ulp must not turn that into a negative loss
            // (a NaN from an out-of-range target stays NaN)
            const float raw = (m - lt) + logf(z);
            const float v = raw < 0.f ? 0.f : raw;
            if (f.nll) f.nll[rr] = v;
            sum += v;
            ++cnt;
        }
        // fixed-order reduction over the lanes
        for (int o = 16; o > 0; o >>= 1) {
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
            cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
        }
        if (lane == 0) {
            if (f.nll_sum) f.nll_sum[b] = sum;
            if (f.count) f.count[b] = cnt;
        }
    }
};

__global__ void __launch_bounds__(256) linear_schedule_kernel(const int32_t *clean, const float *u, const float *t,
                                                              int B, int S, int32_t mask_id, int32_t *noisy,
                                                              uint8_t *masked, uint32_t *dev_err) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)B * S) return;
    const float tb = t[i / S];
    if (!(tb >= 0.f && tb <= 1.f)) {   // a diffusion time outside [0, 1] (or NaN)
        report_error(dev_err, TT_ERR_BOUNDS);
        return;
    }
    const bool m = u[i] < tb;
    masked[i] = m ? 1 : 0;
    if (noisy) noisy[i] = m ? mask_id : clean[i];
}

}  // namespace

size_t masked_nll_ws_bytes(int B, int S, int V, tt_dtype dtype) {
    const size_t part = align_up((size_t)vs::blocks_of(B, S, V, dtype) * sizeof(UnmaskPartial), 256);
    return part + align_up((size_t)(B + 1) * sizeof(unsigned), 256);   // tickets, block counter
}

tt_status launch_masked_nll(const void *logits, tt_dtype dtype, int B, int S, int V, const int32_t *targets,
                            const uint8_t *masked, float *nll, float *nll_sum, int32_t *count, void *ws,
                            uint32_t *dev_err, cudaStream_t stream) {
    if (!vs::rows_aligned(logits, V, dtype)) return TT_ERR_UNSUPPORTED;
    const size_t part_bytes = align_up((size_t)vs::blocks_of(B, S, V, dtype) * sizeof(UnmaskPartial), 256);
    char *w = static_cast<char *>(ws);
    NllFin::Params f;
    f.targets = targets;
    f.nll = nll;
    f.nll_sum = nll_sum;
    f.count = count;
    f.bf16 = dtype == TT_BF16 ? 1 : 0;
    return vs::launch<NllFin>(f, logits, dtype, B, S, V, masked, reinterpret_cast<UnmaskPartial *>(w),
                              reinterpret_cast<unsigned *>(w + part_bytes), dev_err, stream);
}

tt_status launch_linear_schedule(const int32_t *clean, const float *u, const float *t, int B, int S,
                                 int32_t mask_id, int32_t *noisy, uint8_t *masked, uint32_t *dev_err,
                                 cudaStream_t stream) {
    const long long n = (long long)B * S;
    const long long ctas = (n + 255) / 256;
    if (ctas > 0x7fffffffLL) return TT_ERR_UNSUPPORTED;
    linear_schedule_kernel<<<(unsigned)ctas, 256, 0, stream>>>(clean, u, t, B, S, mask_id, noisy, masked, dev_err);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace tt
