// Confidence unmasking of one denoise step (tt_unmask).
//
// Rule (TwoTower summary on gist.science, "Training und Konditionierung --
// Sampling" and "Der Konfidenz-Trick"): every still-masked position of the
// block is predicted in parallel; positions whose confidence (largest softmax
// probability) reaches the threshold are committed and locked, the others stay
// masked.  Completed by two rules that keep a block finite: if nothing reaches
// the threshold the single most confident masked position is committed, and at
// the last step every masked position is committed.
//
// Two kernels compute it.  Rows that are 16-byte aligned (every workload here) take the
// streaming pass over the vocabulary of vocab_stream.cuh, with the commit rule below as
// its Finish.  Unaligned rows (a base address or a row length that is not a multiple of
// 16 bytes) take the chunked kernel: the grid is (vocabulary chunk, position,
// sequence); each CTA reads one 32 KB chunk of one row (bulk copies when the chunk is
// aligned, plain loads otherwise), reduces it to (max, sum of exponentials, first
// argmax) and writes one partial; the last CTA of a sequence to finish (atomic ticket,
// no waiting) merges the partials of the sequence's rows and applies the commit rules.
// Locked rows are never read.

#include <cfloat>
#include <climits>
#include <mutex>

#include "sm100_ptx.cuh"
#include "tt_common.cuh"
#include "tt_internal.h"
#include "vocab_stream.cuh"

namespace tt {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kChunkBytes = 32768;   // one CTA's share of a row
constexpr int kPieces = 4;           // bulk copies (and mbarriers) per chunk
constexpr int kPieceBytes = kChunkBytes / kPieces;
constexpr uint32_t kWaitLimit = 1u << 20;

struct UnmaskParams {
    const void *logits;
    int B, S, V, nchunk;
    float tau;
    int step, T;
    uint8_t *masked;
    int32_t *tokens;
    uint8_t *committed_now;
    float *conf;
    int32_t *n_masked;
    UnmaskPartial *part;
    unsigned *tickets;
    uint32_t *dev_err;
};

template <typename T> struct Vec;
template <> struct Vec<uint16_t> { static constexpr int kElems = 8; };
template <> struct Vec<float> { static constexpr int kElems = 4; };

template <typename T>
__device__ __forceinline__ void unpack(const uint4 &u, float *x);
template <>
__device__ __forceinline__ void unpack<uint16_t>(const uint4 &u, float *x) {
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x);
    x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z);
    x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}
template <>
__device__ __forceinline__ void unpack<float>(const uint4 &u, float *x) {
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
}

template <typename T> __device__ __forceinline__ float load_scalar(const T *p);
template <> __device__ __forceinline__ float load_scalar<uint16_t>(const uint16_t *p) {
    return bf16_bits_to_f32(*p);
}
template <> __device__ __forceinline__ float load_scalar<float>(const float *p) { return *p; }

// Merge two (max, sum-exp relative to max, first argmax) triples.
__device__ __forceinline__ void merge(float &m, float &z, int &a, float m2, float z2, int a2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; z = z2; a = a2; return; }
    const float M = fmaxf(m, m2);
    z = z * fast_exp2((m - M) * kLog2e) + z2 * fast_exp2((m2 - M) * kLog2e);
    a = (m > m2) ? a : (m2 > m) ? a2 : min(a, a2);
    m = M;
}

// Warp-wide merge; both lanes of every pair merge (lower lane, upper lane) in that
// order, so all lanes end with the same, order-fixed result.
__device__ __forceinline__ void warp_merge(float &m, float &z, int &a) {
    const int lane = threadIdx.x & 31;
    for (int o = 1; o < 32; o <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
        const int a2 = __shfl_xor_sync(0xffffffffu, a, o);
        if (lane & o) {
            const float tm = m, tz = z;
            const int ta = a;
            m = m2; z = z2; a = a2;
            merge(m, z, a, tm, tz, ta);
        } else {
            merge(m, z, a, m2, z2, a2);
        }
    }
}

// Fold EPV consecutive elements starting at index e0 into the running state.
// A new maximum must be strictly larger, so the first index of a repeated
// maximum is kept.
template <int EPV>
__device__ __forceinline__ void fold(const float *x, int e0, float &m, float &z, int &a) {
    float gm = x[0];
#pragma unroll
    for (int j = 1; j < EPV; ++j) gm = fmaxf(gm, x[j]);
    if (gm > m) {
        z = (m == -INFINITY) ? 0.f : z * fast_exp2((m - gm) * kLog2e);
        m = gm;
        int j0 = EPV - 1;
#pragma unroll
        for (int j = EPV - 1; j >= 0; --j) j0 = (x[j] == gm) ? j : j0;
        a = e0 + j0;
    }
#pragma unroll
    for (int j = 0; j < EPV; ++j) z += fast_exp2((x[j] - m) * kLog2e);
}

// Largest element of one 16-byte vector.  bf16: a packed pairwise maximum (exact in
// bf16) and one scalar compare; fp32: a compare tree.
template <typename T> __device__ __forceinline__ float vec_max(const uint4 &u);
template <> __device__ __forceinline__ float vec_max<uint16_t>(const uint4 &u) {
    uint32_t a, b, c;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(u.x), "r"(u.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(u.z), "r"(u.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(a), "r"(b));
    return fmaxf(bf16_lo(c), bf16_hi(c));
}
template <> __device__ __forceinline__ float vec_max<float>(const uint4 &u) {
    return fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)),
                 fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
}

// Sum of 2^((x - m)*log2e) over one vector, in two independent partial sums (the
// difference before the scale: see vocab_stream.cuh).
template <typename T>
__device__ __forceinline__ void vec_expsum(const uint4 &u, float m, float &z0, float &z1) {
    constexpr int EPV = Vec<T>::kElems;
    float x[EPV];
    unpack<T>(u, x);
#pragma unroll
    for (int j = 0; j < EPV; j += 2) {
        z0 += fast_exp2((x[j] - m) * kLog2e);
        z1 += fast_exp2((x[j + 1] - m) * kLog2e);
    }
}

// First position in the vector holding the value mx (which it holds).
template <typename T>
__device__ __forceinline__ int vec_first(const uint4 &u, float mx) {
    constexpr int EPV = Vec<T>::kElems;
    float x[EPV];
    unpack<T>(u, x);
    int j0 = EPV - 1;
#pragma unroll
    for (int j = EPV - 1; j >= 0; --j) j0 = (x[j] == mx) ? j : j0;
    return j0;
}

template <typename T, bool kVec>
__global__ void __launch_bounds__(kThreads) unmask_kernel(const UnmaskParams p) {
    constexpr int EPV = Vec<T>::kElems;               // elements per 16-byte vector
    constexpr int CE = kChunkBytes / (int)sizeof(T);  // elements per chunk
    __shared__ __align__(128) uint4 buf[kVec ? kChunkBytes / 16 : 1];
    __shared__ uint64_t bars[kPieces];
    __shared__ float s_m[kWarps], s_z[kWarps];
    __shared__ int s_a[kWarps];
    __shared__ int s_last;

    const int chunk = blockIdx.x, pos = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const size_t row = (size_t)b * p.S + pos;
    const T *rowp = static_cast<const T *>(p.logits) + row * (size_t)p.V;

    if (p.masked[row] != 0) {
        const int c0 = chunk * CE;
        const int n = min(CE, p.V - c0);                 // elements of this chunk
        float m = -INFINITY, z = 0.f;
        int a = INT_MAX;
        if constexpr (kVec) {
            const int bytes = n * (int)sizeof(T);        // a multiple of 16 on this path
            if (tid == 0) {
                for (int k = 0; k < kPieces; ++k) sm100::mbar_init(&bars[k], 1);
                sm100::fence_mbar_init();
                for (int k = 0; k < kPieces; ++k) {
                    const int pb = min(kPieceBytes, bytes - k * kPieceBytes);
                    if (pb <= 0) break;
                    sm100::mbar_arrive_expect_tx(&bars[k], (uint32_t)pb);
                    sm100::bulk_load(reinterpret_cast<char *>(buf) + k * kPieceBytes,
                                     reinterpret_cast<const char *>(rowp + c0) + k * kPieceBytes, (uint32_t)pb,
                                     &bars[k]);
                }
            }
            __syncthreads();
            bool timed_out = false;
            for (int k = 0; k < kPieces; ++k) {
                const int pb = min(kPieceBytes, bytes - k * kPieceBytes);
                if (pb <= 0) break;
                if (!sm100::mbar_wait(&bars[k], 0, kWaitLimit)) {
                    timed_out = true;
                    break;
                }
                // Two passes over the piece in shared memory: this thread's maximum and
                // the first of its vectors that holds it, then the sum of exponentials
                // relative to that maximum; merged into the running state.
                const int nv = pb / 16;
                const uint4 *pv = buf + k * (kPieceBytes / 16);
                float pm = -INFINITY;
                int pvi = -1;
                for (int v = tid; v < nv; v += kThreads) {
                    const float vm = vec_max<T>(pv[v]);
                    if (vm > pm) { pm = vm; pvi = v; }
                }
                if (pvi >= 0) {
                    float z0 = 0.f, z1 = 0.f;
                    for (int v = tid; v < nv; v += kThreads) vec_expsum<T>(pv[v], pm, z0, z1);
                    const int pa = c0 + (k * (kPieceBytes / 16) + pvi) * EPV + vec_first<T>(pv[pvi], pm);
                    merge(m, z, a, pm, z0 + z1, pa);
                }
            }
            if (timed_out) {
                if (tid == 0) report_error(p.dev_err, TT_ERR_DEVICE_TIMEOUT);
                // give the copies a second bounded chance to land before the CTA leaves
                for (int k = 0; k < kPieces; ++k)
                    if (min(kPieceBytes, bytes - k * kPieceBytes) > 0) sm100::mbar_wait(&bars[k], 0, kWaitLimit);
            }
        } else {
            for (int e = tid; e < n; e += kThreads) {
                const float x = load_scalar<T>(rowp + c0 + e);
                fold<1>(&x, c0 + e, m, z, a);
            }
        }
        warp_merge(m, z, a);
        const int w = tid >> 5;
        if ((tid & 31) == 0) { s_m[w] = m; s_z[w] = z; s_a[w] = a; }
        __syncthreads();
        if (tid == 0) {
            float M = s_m[0], Z = s_z[0];
            int A = s_a[0];
            for (int k = 1; k < kWarps; ++k) merge(M, Z, A, s_m[k], s_z[k], s_a[k]);
            UnmaskPartial q;
            q.m = M; q.z = Z; q.arg = A; q.pad = 0;
            p.part[row * p.nchunk + chunk] = q;
        }
    }

    // Ticket: the last CTA of this sequence applies the commit rules.
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned t = atomicAdd(&p.tickets[b], 1u);
        s_last = (t == (unsigned)(p.S * p.nchunk - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    extern __shared__ unsigned char dyn[];
    float *s_conf = reinterpret_cast<float *>(dyn);
    int *s_arg = reinterpret_cast<int *>(s_conf + p.S);
    int *s_commit = s_arg + p.S;
    const int warp = tid >> 5, lane = tid & 31;
    for (int r = warp; r < p.S; r += kWarps) {
        const size_t rr = (size_t)b * p.S + r;
        if (p.masked[rr] == 0) {
            if (lane == 0) { s_conf[r] = NAN; s_arg[r] = -1; }
            continue;
        }
        float m = -INFINITY, zz = 0.f;
        int a = INT_MAX;
        for (int c = lane; c < p.nchunk; c += 32) {
            const UnmaskPartial *qp = p.part + rr * p.nchunk + c;
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(qp));
            merge(m, zz, a, v.x, v.y, __float_as_int(v.z));
        }
        warp_merge(m, zz, a);
        if (lane == 0) { s_conf[r] = 1.0f / zz; s_arg[r] = a; }
    }
    __syncthreads();
    if (tid == 0) {
        const bool last_step = p.step >= p.T;
        int n_commit = 0, best = -1;
        float best_conf = -1.f;
        for (int r = 0; r < p.S; ++r) {
            const bool m = p.masked[(size_t)b * p.S + r] != 0;
            const bool c = m && (last_step || s_conf[r] >= p.tau);
            s_commit[r] = c;
            n_commit += c;
            if (m && s_conf[r] > best_conf) { best_conf = s_conf[r]; best = r; }
        }
        if (n_commit == 0 && best >= 0) s_commit[best] = 1;
    }
    __syncthreads();
    int left = 0;
    for (int r = tid; r < p.S; r += kThreads) {
        const size_t rr = (size_t)b * p.S + r;
        const bool m = p.masked[rr] != 0;
        const bool c = s_commit[r] != 0;
        if (c) { p.tokens[rr] = s_arg[r]; p.masked[rr] = 0; }
        if (p.committed_now) p.committed_now[rr] = c ? 1 : 0;
        if (p.conf) p.conf[rr] = s_conf[r];
        left += (m && !c) ? 1 : 0;
    }
    // count of positions left masked
    for (int o = 16; o > 0; o >>= 1) left += __shfl_xor_sync(0xffffffffu, left, o);
    __syncthreads();
    if (lane == 0) s_a[warp] = left;
    __syncthreads();
    if (tid == 0) {
        int tot = 0;
        for (int w = 0; w < kWarps; ++w) tot += s_a[w];
        if (p.n_masked) p.n_masked[b] = tot;
        p.tickets[b] = 0;   // leave the workspace ready for the next call
    }
}

// ---------------------------------------------------------------- streaming pass
//
// Aligned rows take the shared streaming pass over the vocabulary (vocab_stream.cuh);
// this is its Finish: the commit rule of one sequence, run by one warp once every block
// of the sequence is in.

struct UnmaskFin {
    struct Params {
        float tau;
        int step, T;
        uint8_t *masked;             // in/out (the pass reads it before this Finish runs)
        int32_t *tokens;
        uint8_t *committed_now;
        float *conf;
        int32_t *n_masked;
    };

    // mk: the sequence's masked flags as they were when the launch began (a copy in shared
    // memory, or the array itself); the commits go to f.masked.
    static __device__ void finish(const vs::Common &c, const Params &f, int b, const uint8_t *mk) {
        const int lane = threadIdx.x & 31;
        const bool last_step = f.step >= f.T;
        int n_commit = 0, n_m = 0;
        float best_conf = -1.f;
        int best_pos = INT_MAX, best_arg = 0;
        for (int p = lane; p < c.S; p += 32) {
            const size_t rr = (size_t)b * c.S + p;
            if (mk[p] == 0) {   // locked: nothing read, nothing committed, no confidence
                if (f.committed_now) f.committed_now[rr] = 0;
                if (f.conf) f.conf[rr] = NAN;
                continue;
            }
            float m, z;
            int a;
            vs::row_state(c, (long long)rr, m, z, a);
            const float cf = 1.0f / z;
            if (f.conf) f.conf[rr] = cf;
            const bool com = last_step || cf >= f.tau;
            ++n_m;
            n_commit += com ? 1 : 0;
            if (cf > best_conf || (cf == best_conf && p < best_pos)) { best_conf = cf; best_pos = p; best_arg = a; }
            if (com) { f.tokens[rr] = a; f.masked[rr] = 0; }
            if (f.committed_now) f.committed_now[rr] = com ? 1 : 0;
        }
        // the warp's totals and its most confident masked position (lowest position on ties)
        for (int o = 16; o > 0; o >>= 1) {
            n_commit += __shfl_xor_sync(0xffffffffu, n_commit, o);
            n_m += __shfl_xor_sync(0xffffffffu, n_m, o);
            const float oc = __shfl_xor_sync(0xffffffffu, best_conf, o);
            const int op = __shfl_xor_sync(0xffffffffu, best_pos, o);
            const int oa = __shfl_xor_sync(0xffffffffu, best_arg, o);
            if (oc > best_conf || (oc == best_conf && op < best_pos)) { best_conf = oc; best_pos = op; best_arg = oa; }
        }
        int fallback = 0;
        if (n_commit == 0 && n_m > 0) {
            // nothing reached the threshold: commit the single most confident masked position
            fallback = 1;
            if (lane == 0) {
                const size_t rr = (size_t)b * c.S + best_pos;
                f.tokens[rr] = best_arg;
                f.masked[rr] = 0;
                if (f.committed_now) f.committed_now[rr] = 1;
            }
        }
        if (lane == 0 && f.n_masked) f.n_masked[b] = n_m - n_commit - fallback;
    }
};

}  // namespace

int unmask_chunk_elems(tt_dtype dtype) { return kChunkBytes / (dtype == TT_BF16 ? 2 : 4); }

// Workspace: partial slots at offset 0 (one per (row, 32 KB chunk) for the chunked kernel,
// one per block for the streaming pass; the larger count is reserved), then the
// per-sequence tickets and the streaming pass's block counter.
size_t unmask_tickets_off(int B, int S, int V, tt_dtype dtype) {
    const size_t nchunk = (size_t)((V + unmask_chunk_elems(dtype) - 1) / unmask_chunk_elems(dtype));
    const size_t chunked = (size_t)B * S * nchunk;
    const size_t streamed = (size_t)vs::blocks_of(B, S, V, dtype);
    return align_up((chunked > streamed ? chunked : streamed) * sizeof(UnmaskPartial), 256);
}

size_t unmask_ws_bytes(int B, int S, int V, tt_dtype dtype) {
    return unmask_tickets_off(B, S, V, dtype) + align_up((size_t)(B + 1) * sizeof(unsigned), 256);
}

tt_status launch_unmask(const void *logits, tt_dtype dtype, int B, int S, int V, float tau,
                        int step, int T, uint8_t *masked, int32_t *tokens, uint8_t *committed_now,
                        float *conf, int32_t *n_masked, void *ws, uint32_t *dev_err,
                        cudaStream_t stream) {
    UnmaskPartial *part = static_cast<UnmaskPartial *>(ws);
    unsigned *tickets = reinterpret_cast<unsigned *>(static_cast<char *>(ws) + unmask_tickets_off(B, S, V, dtype));
    if (vs::rows_aligned(logits, V, dtype)) {
        UnmaskFin::Params f;
        f.tau = tau; f.step = step; f.T = T;
        f.masked = masked; f.tokens = tokens; f.committed_now = committed_now; f.conf = conf;
        f.n_masked = n_masked;
        return vs::launch<UnmaskFin>(f, logits, dtype, B, S, V, masked, part, tickets, dev_err, stream);
    }
    UnmaskParams p;
    p.logits = logits;
    p.B = B; p.S = S; p.V = V;
    p.nchunk = (V + unmask_chunk_elems(dtype) - 1) / unmask_chunk_elems(dtype);
    p.tau = tau; p.step = step; p.T = T;
    p.masked = masked; p.tokens = tokens; p.committed_now = committed_now; p.conf = conf;
    p.n_masked = n_masked;
    p.part = part;
    p.tickets = tickets;
    p.dev_err = dev_err;
    const bool vec = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) &&
                     (V % (dtype == TT_BF16 ? 8 : 4) == 0);
    const dim3 grid(p.nchunk, S, B);
    const size_t smem = (size_t)S * 3 * sizeof(float);
    if (dtype == TT_BF16) {
        if (vec) unmask_kernel<uint16_t, true><<<grid, kThreads, smem, stream>>>(p);
        else unmask_kernel<uint16_t, false><<<grid, kThreads, smem, stream>>>(p);
    } else {
        if (vec) unmask_kernel<float, true><<<grid, kThreads, smem, stream>>>(p);
        else unmask_kernel<float, false><<<grid, kThreads, smem, stream>>>(p);
    }
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

// ---------------------------------------------------------------- scratch-free variant
//
// For callers that cannot allocate device memory (graph capture, pool-owning
// frameworks, fixed-memory real-time loops): the same kernel, with its scratch in
// this file-scope device array instead of a caller workspace.  The array is held
// by every GPU that loads the library until the process exits; all calls share it.

static __device__ __align__(256) unsigned char g_unmask_scratch[TT_UNMASK_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices];   // set only by a lookup that succeeded

// Device address of the scratch array on device `dev` (current), looked up on the first
// call that succeeds; a failed lookup is not remembered, so a later call tries again.
void *scratch_address(int dev) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_unmask_scratch) != cudaSuccess) {
            cudaGetLastError();   // take back the error it recorded, so no later check sees it
            return nullptr;
        }
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

tt_status launch_unmask_noalloc(const void *logits, tt_dtype dtype, int B, int S, int V, float tau,
                                int step, int T, uint8_t *masked, int32_t *tokens,
                                uint8_t *committed_now, float *conf, int32_t *n_masked,
                                uint32_t *dev_err, cudaStream_t stream) {
    const size_t need = unmask_ws_bytes(B, S, V, dtype);
    if (need > TT_UNMASK_NOALLOC_SCRATCH_BYTES) return TT_ERR_CAPACITY;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TT_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TT_ERR_UNSUPPORTED;
    // Host code only holds a stand-in for the array; its device address comes from
    // the runtime, once per device, with that device current.
    void *ws = scratch_address(dev);
    if (ws == nullptr) return TT_ERR_CUDA;
    // The per-sequence counters must start at zero, whatever an earlier call left (they
    // lie at the end of the workspace layout).
    const size_t tick_off = unmask_tickets_off(B, S, V, dtype);
    if (cudaMemsetAsync(static_cast<char *>(ws) + tick_off, 0, unmask_ws_bytes(B, S, V, dtype) - tick_off,
                        stream) != cudaSuccess)
        return TT_ERR_CUDA;
    return launch_unmask(logits, dtype, B, S, V, tau, step, T, masked, tokens, committed_now, conf, n_masked,
                         ws, dev_err, stream);
}

}  // namespace tt
