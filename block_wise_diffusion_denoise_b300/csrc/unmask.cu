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
// Design: HBM-bound single pass over the masked rows' logits.  The grid is
// (vocabulary chunk, position, sequence); each CTA brings one 32 KB chunk of one
// row into shared memory with four bulk copies (cp.async.bulk, one mbarrier per
// 8 KB piece) issued before any arithmetic, so up to six CTAs per SM keep about
// 190 KB in flight with few registers.  Each thread makes two passes over its
// vectors of a piece in shared memory -- the maximum (packed bf16 pairs, exact)
// with the first vector holding it, then the sum of exponentials relative to
// that maximum -- and merges the piece into a running (max, sum, first argmax)
// state; the CTA merges the threads' states in a fixed order and writes one
// partial.  The last CTA of a sequence to
// finish (atomic ticket, no waiting) merges the partials of the sequence's rows
// and applies the commit rules.  Locked rows cost one byte read.

#include <cfloat>
#include <climits>
#include <mutex>

#include "sm100_ptx.cuh"
#include "tt_common.cuh"
#include "tt_internal.h"

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
    const float mc = m * kLog2e;
#pragma unroll
    for (int j = 0; j < EPV; ++j) z += fast_exp2(fmaf(x[j], kLog2e, -mc));
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

// Sum of 2^(x*log2e - mc) over one vector, in two independent partial sums.
template <typename T>
__device__ __forceinline__ void vec_expsum(const uint4 &u, float mc, float &z0, float &z1) {
    constexpr int EPV = Vec<T>::kElems;
    float x[EPV];
    unpack<T>(u, x);
#pragma unroll
    for (int j = 0; j < EPV; j += 2) {
        z0 += fast_exp2(fmaf(x[j], kLog2e, -mc));
        z1 += fast_exp2(fmaf(x[j + 1], kLog2e, -mc));
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
                    const float mc = pm * kLog2e;
                    float z0 = 0.f, z1 = 0.f;
                    for (int v = tid; v < nv; v += kThreads) vec_expsum<T>(pv[v], mc, z0, z1);
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

// ---------------------------------------------------------------- streaming kernel
//
// Persistent variant for batches whose masked-row list fits in shared memory: one CTA
// per SM, sixteen warps, and every warp streams its own contiguous share of the
// (masked row, 6 KB chunk) units through a private two-stage ring of bulk copies,
// so that the copies stay in flight across the whole launch instead of stopping at
// every CTA boundary.  A warp folds consecutive chunks of one row into a running
// state and publishes one partial per row it touches (slot = warp + row ordinal);
// the warp that completes a sequence's count of units merges that sequence's
// partials and applies the commit rules.

constexpr int kSWarps = 16;
constexpr int kSThreads = 32 * kSWarps;
constexpr int kSStages = 2;
constexpr int kSChunkBytes = 6144;
constexpr int kSRowsMax = 4096;           // masked-row list held in shared memory
constexpr int kSCtasMax = 296;            // grid cap (sizes the workspace)
constexpr int kSMinUnits = 4;             // a warp's share is at least this many units
constexpr int kSSmemBytes = kSWarps * kSStages * kSChunkBytes;

struct StreamParams {
    const void *logits;
    int B, S, V, nc;                      // nc: chunks per row
    float tau;
    int step, T;
    uint8_t *masked;
    int32_t *tokens;
    uint8_t *committed_now;
    float *conf;
    int32_t *n_masked;
    UnmaskPartial *part;                  // kSCtasMax * kSWarps + B * S slots
    unsigned *tickets;                    // [B] units done per sequence
    uint32_t *dev_err;
};

// Running maximum of vectors, kept as four independent words (packed bf16 pairs, or
// fp32): exact, and free of a dependency chain across words.
template <typename T> struct PackedMax;
template <> struct PackedMax<uint16_t> {
    uint32_t w[4] = {0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u};   // (-inf, -inf)
    __device__ __forceinline__ void add(const uint4 &u) {
        asm("max.bf16x2 %0, %0, %1;" : "+r"(w[0]) : "r"(u.x));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(w[1]) : "r"(u.y));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(w[2]) : "r"(u.z));
        asm("max.bf16x2 %0, %0, %1;" : "+r"(w[3]) : "r"(u.w));
    }
    __device__ __forceinline__ float result() const {
        return vec_max<uint16_t>(make_uint4(w[0], w[1], w[2], w[3]));
    }
};
template <> struct PackedMax<float> {
    float w[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    __device__ __forceinline__ void add(const uint4 &u) {
        w[0] = fmaxf(w[0], __uint_as_float(u.x)); w[1] = fmaxf(w[1], __uint_as_float(u.y));
        w[2] = fmaxf(w[2], __uint_as_float(u.z)); w[3] = fmaxf(w[3], __uint_as_float(u.w));
    }
    __device__ __forceinline__ float result() const { return fmaxf(fmaxf(w[0], w[1]), fmaxf(w[2], w[3])); }
};

__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

// acc += (2^(lo*l2 - mc), 2^(hi*l2 - mc)) with one paired FMA and one paired add.
__device__ __forceinline__ void expsum_pair(float lo, float hi, uint64_t l2x2, uint64_t nmc2, uint64_t &acc) {
    uint64_t y;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(y) : "l"(f32x2(lo, hi)), "l"(l2x2), "l"(nmc2));
    float y0, y1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(y0), "=f"(y1) : "l"(y));
    asm("add.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(f32x2(fast_exp2(y0), fast_exp2(y1))));
}

// Exponential sums of one vector into two paired accumulators.
template <typename T>
__device__ __forceinline__ void vec_expsum2(const uint4 &u, uint64_t l2x2, uint64_t nmc2, uint64_t &za, uint64_t &zb);
template <>
__device__ __forceinline__ void vec_expsum2<uint16_t>(const uint4 &u, uint64_t l2x2, uint64_t nmc2, uint64_t &za,
                                                      uint64_t &zb) {
    expsum_pair(bf16_lo(u.x), bf16_hi(u.x), l2x2, nmc2, za);
    expsum_pair(bf16_lo(u.y), bf16_hi(u.y), l2x2, nmc2, zb);
    expsum_pair(bf16_lo(u.z), bf16_hi(u.z), l2x2, nmc2, za);
    expsum_pair(bf16_lo(u.w), bf16_hi(u.w), l2x2, nmc2, zb);
}
template <>
__device__ __forceinline__ void vec_expsum2<float>(const uint4 &u, uint64_t l2x2, uint64_t nmc2, uint64_t &za,
                                                   uint64_t &zb) {
    expsum_pair(__uint_as_float(u.x), __uint_as_float(u.y), l2x2, nmc2, za);
    expsum_pair(__uint_as_float(u.z), __uint_as_float(u.w), l2x2, nmc2, zb);
}

// The warp whose unit range [w*NU/NW, (w+1)*NU/NW) holds unit u.
__device__ __forceinline__ int unit_owner(long long u, long long NU, int NW) {
    long long w = u * NW / NU;
    while (w + 1 < NW && (w + 1) * NU / NW <= u) ++w;
    while (w > 0 && w * NU / NW > u) --w;
    return (int)w;
}

// First index in the sorted list rows[0, n) holding a value >= x.
__device__ __forceinline__ int lower_bound_rows(const int *rows, int n, int x) {
    int a = 0, z = n;
    while (a < z) {
        const int mid = (a + z) >> 1;
        if (rows[mid] < x) a = mid + 1; else z = mid;
    }
    return a;
}

// Commit rules of sequence b, by one warp, after every partial of its masked rows is in.
__device__ void stream_rules(const StreamParams &p, const int *rows, int R, int b, int NW, long long NU) {
    const int lane = threadIdx.x & 31;
    const int k0 = lower_bound_rows(rows, R, b * p.S), k1 = lower_bound_rows(rows, R, (b + 1) * p.S);
    const bool last_step = p.step >= p.T;
    // per masked row: merge its partials (group order) into (conf, argmax)
    int n_commit = 0;
    float best_conf = -1.f;
    int best_pos = INT_MAX, best_arg = 0;
    for (int k = k0 + lane; k < k1; k += 32) {
        const int w0 = unit_owner((long long)k * p.nc, NU, NW);
        const int w1 = unit_owner((long long)(k + 1) * p.nc - 1, NU, NW);
        float m = -INFINITY, z = 0.f;
        int a = INT_MAX;
        for (int w = w0; w <= w1; ++w) {
            // a warp whose share is empty (fewer units than warps) wrote no partial
            if ((long long)(w + 1) * NU / NW == (long long)w * NU / NW) continue;
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.part + w + k));
            merge(m, z, a, v.x, v.y, __float_as_int(v.z));
        }
        const float cf = 1.0f / z;
        const int pos = rows[k] - b * p.S;
        const size_t rr = (size_t)rows[k];
        if (p.conf) p.conf[rr] = cf;
        const bool c = last_step || cf >= p.tau;
        n_commit += c ? 1 : 0;
        if (cf > best_conf || (cf == best_conf && pos < best_pos)) { best_conf = cf; best_pos = pos; best_arg = a; }
        if (c) { p.tokens[rr] = a; p.masked[rr] = 0; }
        if (p.committed_now) p.committed_now[rr] = c ? 1 : 0;
    }
    // warp totals: commits and the most confident masked position (lowest position on ties)
    for (int o = 16; o > 0; o >>= 1) {
        n_commit += __shfl_xor_sync(0xffffffffu, n_commit, o);
        const float oc = __shfl_xor_sync(0xffffffffu, best_conf, o);
        const int op = __shfl_xor_sync(0xffffffffu, best_pos, o);
        const int oa = __shfl_xor_sync(0xffffffffu, best_arg, o);
        if (oc > best_conf || (oc == best_conf && op < best_pos)) { best_conf = oc; best_pos = op; best_arg = oa; }
    }
    const int n_m = k1 - k0;
    int fallback = 0;
    if (n_commit == 0 && n_m > 0) {
        // nothing reached the threshold: commit the single most confident masked position
        // (its argmax travelled with it through the reduction)
        fallback = 1;
        if (lane == 0) {
            const size_t rr = (size_t)b * p.S + best_pos;
            p.tokens[rr] = best_arg;
            p.masked[rr] = 0;
            if (p.committed_now) p.committed_now[rr] = 1;
        }
    }
    // positions that were not masked: nothing committed, no confidence
    for (int pos = lane; pos < p.S; pos += 32) {
        const size_t rr = (size_t)b * p.S + pos;
        const int k = lower_bound_rows(rows + k0, n_m, (int)rr) + k0;
        if (k < k1 && rows[k] == (int)rr) continue;
        if (p.committed_now) p.committed_now[rr] = 0;
        if (p.conf) p.conf[rr] = NAN;
    }
    if (lane == 0) {
        if (p.n_masked) p.n_masked[b] = n_m - n_commit - fallback;
        p.tickets[b] = 0;   // leave the workspace ready for the next call
    }
}

template <typename T>
__global__ void __launch_bounds__(kSThreads, 1) unmask_stream_kernel(const StreamParams p) {
    constexpr int EPV = Vec<T>::kElems;
    constexpr int CE = kSChunkBytes / (int)sizeof(T);
    extern __shared__ __align__(128) unsigned char ring_raw[];
    __shared__ uint64_t bars[kSWarps][kSStages];
    __shared__ int s_rows[kSRowsMax];
    __shared__ int s_wsum[kSWarps];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int BS = p.B * p.S;

    // ---- the masked rows in (sequence, position) order
    int R = 0;
    for (int base = 0; base < BS; base += kSThreads) {
        const int row = base + tid;
        const bool m = row < BS && p.masked[row] != 0;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        if (lane == 0) s_wsum[warp] = __popc(bal);
        __syncthreads();
        int before = 0, total = 0;
        for (int w = 0; w < kSWarps; ++w) {
            before += (w < warp) ? s_wsum[w] : 0;
            total += s_wsum[w];
        }
        if (m) s_rows[R + before + __popc(bal & ((1u << lane) - 1u))] = row;
        R += total;
        __syncthreads();
    }
    if (lane == 0)
        for (int k = 0; k < kSStages; ++k) sm100::mbar_init(&bars[warp][k], 1);
    sm100::fence_mbar_init();
    __syncthreads();

    // ---- sequences without a masked position: nothing to read, nothing committed
    for (int b = blockIdx.x * kSWarps + warp; b < p.B; b += gridDim.x * kSWarps) {
        const int k = lower_bound_rows(s_rows, R, b * p.S);
        if (k < R && s_rows[k] < (b + 1) * p.S) continue;
        for (int pos = lane; pos < p.S; pos += 32) {
            const size_t rr = (size_t)b * p.S + pos;
            if (p.committed_now) p.committed_now[rr] = 0;
            if (p.conf) p.conf[rr] = NAN;
        }
        if (lane == 0 && p.n_masked) p.n_masked[b] = 0;
    }

    // ---- this warp's units: the shares go to at most NU / kSMinUnits warps, so that a
    // small batch is not spread over warps of one unit each (every share is a partial
    // the rule stage must read)
    const long long NU = (long long)R * p.nc;
    const int NWall = gridDim.x * kSWarps, w = blockIdx.x * kSWarps + warp;
    const int NW = (int)(NU / kSMinUnits < 1 ? 1 : (NU / kSMinUnits < NWall ? NU / kSMinUnits : NWall));
    if (w >= NW) return;
    const long long u0 = (long long)w * NU / NW, u1 = (long long)(w + 1) * NU / NW;
    const int n = (int)(u1 - u0);
    if (n <= 0) return;
    unsigned char *ring = ring_raw + (size_t)warp * kSStages * kSChunkBytes;
    const T *logits = static_cast<const T *>(p.logits);

    // (row ordinal, chunk) of the next unit to load, advanced one unit per copy
    int ik = (int)(u0 / p.nc), ic = (int)(u0 % p.nc);
    auto issue = [&](int i) {   // lane 0: bring unit u0 + i (= (ik, ic)) into stage i % kSStages
        const int e0 = ic * CE, ne = min(CE, p.V - e0);
        uint64_t *bar = &bars[warp][i % kSStages];
        sm100::mbar_arrive_expect_tx(bar, (uint32_t)(ne * sizeof(T)));
        sm100::bulk_load(ring + (i % kSStages) * kSChunkBytes, logits + (size_t)s_rows[ik] * p.V + e0,
                         (uint32_t)(ne * sizeof(T)), bar);
        if (++ic == p.nc) { ic = 0; ++ik; }
    };
    if (lane == 0)
        for (int i = 0; i < kSStages && i < n; ++i) issue(i);

    float m = -INFINITY, z = 0.f;
    int a = INT_MAX, seg = 0;
    int k = (int)(u0 / p.nc), c = (int)(u0 % p.nc);   // the unit being consumed
    const uint64_t l2x2 = f32x2(kLog2e, kLog2e);
    for (int i = 0; i < n; ++i) {
        const int e0 = c * CE, nv = min(CE, p.V - e0) / EPV;
        if (!sm100::mbar_wait(&bars[warp][i % kSStages], (uint32_t)(i / kSStages) & 1, kWaitLimit)) {
            if (lane == 0) report_error(p.dev_err, TT_ERR_DEVICE_TIMEOUT);
            // let the copies still in flight land before the warp leaves
            for (int j = i; j < n && j < i + kSStages; ++j)
                sm100::mbar_wait(&bars[warp][j % kSStages], (uint32_t)(j / kSStages) & 1, kWaitLimit);
            return;
        }
        // two passes over the chunk: this lane's maximum with its first vector, then the
        // sum of exponentials relative to it
        const uint4 *pv = reinterpret_cast<const uint4 *>(ring + (i % kSStages) * kSChunkBytes);
        if (lane < nv) {
            // this lane's maximum (four independent packed accumulators), the first of its
            // vectors holding it, then the sum of exponentials relative to it
            PackedMax<T> acc;
#pragma unroll 4
            for (int v = lane; v < nv; v += 32) acc.add(pv[v]);
            const float pm = acc.result();
            int pvi = lane;
            while (pvi + 32 < nv && vec_max<T>(pv[pvi]) != pm) pvi += 32;
            const uint64_t nmc2 = f32x2(-pm * kLog2e, -pm * kLog2e);
            uint64_t za = 0, zb = 0;
#pragma unroll 4
            for (int v = lane; v < nv; v += 32) vec_expsum2<T>(pv[v], l2x2, nmc2, za, zb);
            asm("add.f32x2 %0, %0, %1;" : "+l"(za) : "l"(zb));
            float z0, z1;
            asm("mov.b64 {%0, %1}, %2;" : "=f"(z0), "=f"(z1) : "l"(za));
            merge(m, z, a, pm, z0 + z1, e0 + pvi * EPV + vec_first<T>(pv[pvi], pm));
        }
        // the stage is consumed: refill it with the unit kSStages ahead
        __syncwarp();
        sm100::fence_proxy_async_smem();
        if (lane == 0 && i + kSStages < n) issue(i + kSStages);
        ++seg;
        const bool row_end = (c + 1 == p.nc);
        if (i == n - 1 || row_end) {
            // end of this warp's part of row k: publish it and count it for the sequence
            warp_merge(m, z, a);
            const int row = s_rows[k], b = row / p.S;
            unsigned last = 0;
            if (lane == 0) {
                UnmaskPartial q;
                q.m = m; q.z = z; q.arg = a; q.pad = 0;
                p.part[w + k] = q;
                const int nm = lower_bound_rows(s_rows, R, (b + 1) * p.S) - lower_bound_rows(s_rows, R, b * p.S);
                const unsigned done = sm100::atom_add_acq_rel_gpu(&p.tickets[b], (unsigned)seg);
                last = (done + (unsigned)seg == (unsigned)(nm * p.nc)) ? 1u : 0u;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence();
                stream_rules(p, s_rows, R, b, NW, NU);
            }
            m = -INFINITY; z = 0.f; a = INT_MAX; seg = 0;
        }
        if (row_end) { c = 0; ++k; } else { ++c; }
    }
}

}  // namespace

int unmask_chunk_elems(tt_dtype dtype) { return kChunkBytes / (dtype == TT_BF16 ? 2 : 4); }

namespace {

// Partial slots of either kernel: one per (row, 32 KB chunk) for the chunked kernel, one
// per (warp, row ordinal) pair for the streaming kernel.
size_t unmask_part_slots(int B, int S, int V, tt_dtype dtype) {
    const size_t nchunk = (size_t)((V + unmask_chunk_elems(dtype) - 1) / unmask_chunk_elems(dtype));
    const size_t chunked = (size_t)B * S * nchunk;
    const size_t streamed = (size_t)kSCtasMax * kSWarps + (size_t)B * S;
    return chunked > streamed ? chunked : streamed;
}

size_t unmask_tickets_off(int B, int S, int V, tt_dtype dtype) {
    return align_up(unmask_part_slots(B, S, V, dtype) * sizeof(UnmaskPartial), 256);
}

}  // namespace

size_t unmask_ws_bytes(int B, int S, int V, tt_dtype dtype) {
    return unmask_tickets_off(B, S, V, dtype) + align_up((size_t)B * sizeof(unsigned), 256);
}

tt_status launch_unmask(const void *logits, tt_dtype dtype, int B, int S, int V, float tau,
                        int step, int T, uint8_t *masked, int32_t *tokens, uint8_t *committed_now,
                        float *conf, int32_t *n_masked, void *ws, uint32_t *dev_err,
                        cudaStream_t stream) {
    UnmaskParams p;
    p.logits = logits;
    p.B = B; p.S = S; p.V = V;
    p.nchunk = (V + unmask_chunk_elems(dtype) - 1) / unmask_chunk_elems(dtype);
    p.tau = tau; p.step = step; p.T = T;
    p.masked = masked; p.tokens = tokens; p.committed_now = committed_now; p.conf = conf;
    p.n_masked = n_masked;
    p.part = static_cast<UnmaskPartial *>(ws);
    p.tickets = reinterpret_cast<unsigned *>(static_cast<char *>(ws) + unmask_tickets_off(B, S, V, dtype));
    p.dev_err = dev_err;
    const bool vec = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) &&
                     (V % (dtype == TT_BF16 ? 8 : 4) == 0);
    if (vec && (size_t)B * S <= (size_t)kSRowsMax) {
        // streaming kernel: one CTA per SM
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return TT_ERR_CUDA;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TT_ERR_CUDA;
        const int grid = sms < kSCtasMax ? sms : kSCtasMax;
        StreamParams q;
        q.logits = logits;
        q.B = B; q.S = S; q.V = V;
        q.nc = (V + kSChunkBytes / (dtype == TT_BF16 ? 2 : 4) - 1) / (kSChunkBytes / (dtype == TT_BF16 ? 2 : 4));
        q.tau = tau; q.step = step; q.T = T;
        q.masked = masked; q.tokens = tokens; q.committed_now = committed_now; q.conf = conf;
        q.n_masked = n_masked; q.part = p.part; q.tickets = p.tickets; q.dev_err = dev_err;
        if (dtype == TT_BF16) {
            if (cudaFuncSetAttribute(unmask_stream_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSSmemBytes) != cudaSuccess)
                return TT_ERR_CUDA;
            unmask_stream_kernel<uint16_t><<<grid, kSThreads, kSSmemBytes, stream>>>(q);
        } else {
            if (cudaFuncSetAttribute(unmask_stream_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSSmemBytes) != cudaSuccess)
                return TT_ERR_CUDA;
            unmask_stream_kernel<float><<<grid, kSThreads, kSSmemBytes, stream>>>(q);
        }
        return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
    }
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
    // The per-sequence counters must start at zero, whatever an earlier call left.
    const size_t tick_off = unmask_tickets_off(B, S, V, dtype);
    if (cudaMemsetAsync(static_cast<char *>(ws) + tick_off, 0, (size_t)B * sizeof(unsigned), stream) !=
        cudaSuccess)
        return TT_ERR_CUDA;
    return launch_unmask(logits, dtype, B, S, V, tau, step, T, masked, tokens, committed_now, conf, n_masked,
                         ws, dev_err, stream);
}

}  // namespace tt
