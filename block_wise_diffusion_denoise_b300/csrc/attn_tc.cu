// Two-segment denoise attention on the 5th-generation tensor cores (bf16, D = 128,
// 64-token pages).
//
// What it computes (TwoTower summary on gist.science, "Technisches Resuemee --
// Architektur" and "Generierungsprozess"; dgnews.ru, "How the architecture
// actually works"): the S block queries of every query head attend, in one
// softmax, to all L context keys the frozen context tower holds for this layer
// and to the S keys of their own block, without a mask inside the block.
//
// Design for sm_103a:
//  * Rows.  The G = Hq/Hkv query heads of one KV head share every key, so the
//    G*S (s, head) rows of one (sequence, KV head) segment form the M side of
//    the MMA: one or two 128-row tiles, each key tile is read from HBM once for
//    all of them (256 flop per key byte at G*S = 256).
//  * Tiles.  A key tile is one 64-token page of the paged cache (or the block's
//    own S keys).  A producer warp moves K and V pages with TMA (128-byte
//    swizzle) into separate rings (4 K stages, freed as soon as QK has read them;
//    6 V stages, freed after PV), fetching page ids 32 at a time; Q of the
//    segment is loaded once.  S = Q K^T goes to a double-buffered TMEM tile,
//    then O += P V with P read from TMEM.  Each issuing thread waits about a
//    hundred cycles per tcgen05.mma while the tensor pipe accepts several
//    streams, so the QK product of each M tile and the PV product have their own
//    issuing warps (one elected lane of a converged warp issues).
//  * Softmax.  One thread per row (two warpgroups for two M tiles) reads its S
//    row from TMEM, keeps the running maximum in the log2 domain and only
//    rescales O (in TMEM) when the maximum grows by more than 2^8, and writes P
//    back over its S row as packed bf16 (the A operand of the PV product).
//    Columns past the valid keys of a partial page are masked, and the matching
//    V rows are zeroed before the PV product, so slots past L never matter.
//  * Work split.  The whole batch is a list of segments (b, g), each a run of
//    page tiles plus one block tile; cost 4 per page and 1 per block tile.  A
//    persistent grid of one CTA per SM cuts the list into equal cost ranges
//    (stream-K style): a CTA that owns a whole segment writes the final output;
//    pieces of a shared segment go to fp32 partial slots and the last CTA to
//    finish the segment (atomic ticket, no waiting) merges them with log-sum-exp
//    weights.  Ragged and long contexts balance without host knowledge of the
//    lengths, which live on the device.
//  * Every mbarrier wait is bounded; a wait that gives up records
//    TT_ERR_DEVICE_TIMEOUT, the CTA drains its copies and MMAs and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "sm100_ptx.cuh"
#include "tt_common.cuh"
#include "tt_internal.h"

namespace tt {
namespace {

using namespace sm100;

constexpr int kD = 128;                  // head dim
constexpr int kPage = 64;                // tokens per page = keys per tile
constexpr int kKStages = 4;              // K ring depth (a stage is free once QK has read it)
constexpr int kVStages = 6;              // V ring depth (a stage is free once PV has read it)
constexpr int kMaxCtas = 296;            // upper bound of the persistent grid (sizes the workspace)
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr float kRescaleThreshold = 8.0f;   // log2 units

// Shared memory (offsets from a 1024-byte aligned base).  Every tile is stored as two
// 128-byte-swizzled halves of 64 columns (d 0..63 and d 64..127).
constexpr int kHalf = 8192;              // 64 rows x 128 bytes
constexpr int kTile = 2 * kHalf;         // one K or V page
constexpr int kQTile = 16384;            // 128 rows x 128 bytes
constexpr int kOffQ = 0;                 // Q[mt][d-half], 16 KB each
constexpr int kOffK = 4 * kQTile;
constexpr int kOffV = kOffK + kKStages * kTile;
constexpr int kSmemBytes = kOffV + kVStages * kTile + 1024;

// TMEM columns.
constexpr int kTmemCols = 512;
constexpr int kColO = 0;                 // O[mt]: 128 columns each
constexpr int kColS = 256;               // S[buf][mt]: 64 fp32 columns; P overwrites the first 32 as bf16 pairs

struct TcParams {
    const int32_t *page_table;
    const int32_t *ctx_len;
    int num_pages, max_pages;
    uint16_t *out;
    float *lse;
    int B, S, Hq, Hkv, G, rows, NT;
    float scale_log2;
    int n_ctas;
    unsigned *tickets;
    float *part;
    long long slot_floats;
    uint32_t *dev_err;
};

struct Bars {
    uint64_t q_full, q_empty;
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2][2];   // [buffer][M tile]: S of the tile is in TMEM
    uint64_t s_free[2][2];   // the PV product that read P from this buffer has completed
    uint64_t p_full[2][2];   // the M tile's four softmax warps wrote P; one per buffer so a warp
                             // already on tile t+1 cannot complete tile t's phase
    uint64_t o_full[2], o_empty[2];
    uint64_t grp;            // softmax warps among themselves (bounded, unlike bar.sync)
    uint64_t done[3];        // last MMA of each issuer has completed
};

struct Shared {
    Bars bar;
    uint32_t tmem_base;
    int abort;
    int last;
};

// ------------------------------------------------------------------ work partition

__device__ __forceinline__ int clamp_len(const TcParams &p, int b) {
    const int L = p.ctx_len[b];
    return (L < 0 || L > p.max_pages * kPage) ? 0 : L;
}

struct Piece {
    int b, g, sg;          // sequence, KV head, segment index b * Hkv + g
    int L, ntc;            // context length and its page tiles (tile ntc is the block tile)
    int first, last;       // tiles [first, last) of this segment belong to this CTA
    long long X;           // start unit of the segment
    bool whole;
};

struct WorkIter {
    long long U, lo, hi, X;
    int b, g, L, ntc, C;
    int B, Hkv;

    __device__ void init(const TcParams &p, int cta) {
        B = p.B; Hkv = p.Hkv;
        U = 0;
        for (int i = 0; i < B; ++i) U += (long long)Hkv * (4 * ((clamp_len(p, i) + kPage - 1) / kPage) + 1);
        lo = (long long)cta * U / p.n_ctas;
        hi = (long long)(cta + 1) * U / p.n_ctas;
        X = 0; b = 0; g = 0;
        load(p);
        // skip whole sequences that end before lo
        while (b < B && X + (long long)Hkv * C <= lo) {
            X += (long long)Hkv * C;
            ++b;
            if (b < B) load(p);
        }
    }
    __device__ void load(const TcParams &p) {
        if (b < B) {
            L = clamp_len(p, b);
            ntc = (L + kPage - 1) / kPage;
            C = 4 * ntc + 1;
        }
    }
    // Next piece owned by this CTA; false when the range is exhausted.
    __device__ bool next(const TcParams &p, Piece &pc) {
        while (b < B && X < hi) {
            const long long first = (lo > X) ? (lo - X + 3) / 4 : 0;
            long long last = (hi - X + 3) / 4;
            if (last > ntc + 1) last = ntc + 1;
            const bool have = first < last;
            if (have) {
                pc.b = b; pc.g = g; pc.sg = b * Hkv + g; pc.L = L; pc.ntc = ntc;
                pc.first = (int)first; pc.last = (int)last; pc.X = X;
                pc.whole = (first == 0 && last == ntc + 1);
            }
            X += C;
            if (++g == Hkv) { g = 0; ++b; load(p); }
            if (have) return true;
        }
        return false;
    }
};

__device__ __forceinline__ long long range_lo(long long c, long long U, int n) { return c * U / n; }

// The CTA whose range holds unit u.
__device__ __forceinline__ int owner(long long u, long long U, int n) {
    long long c = u * n / U;
    while (c + 1 < n && range_lo(c + 1, U, n) <= u) ++c;
    while (c > 0 && range_lo(c, U, n) > u) --c;
    return (int)c;
}

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ bool wait_bar(Shared &sh, uint64_t *bar, uint32_t parity, uint32_t *dev_err) {
    if (*(volatile int *)&sh.abort) return false;
    if (mbar_wait(bar, parity, kWaitLimit)) return true;
    *(volatile int *)&sh.abort = 1;
    report_error(dev_err, TT_ERR_DEVICE_TIMEOUT);
    return false;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// All softmax warps meet (k-th meeting of this CTA); false if a warp never came.
__device__ __forceinline__ bool group_sync(Shared &sh, int &k, uint32_t *dev_err) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.bar.grp);
    const bool ok = wait_bar(sh, &sh.bar.grp, (uint32_t)k & 1, dev_err);
    ++k;
    return ok;
}

__device__ __forceinline__ int tile_valid(const Piece &pc, int i, int S) {
    return i < pc.ntc ? min(kPage, pc.L - kPage * i) : S;
}

// One elected lane of a converged warp issues each MMA, so the operands stay warp-uniform.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
    return pred != 0;
}

// Does CTA c own at least one tile of the segment starting at unit X with ntc page tiles?
__device__ __forceinline__ bool owns_tile(int c, long long X, int ntc, long long U, int n) {
    const long long lo_c = range_lo(c, U, n), hi_c = range_lo(c + 1, U, n);
    const long long i0 = (lo_c > X) ? (lo_c - X + 3) / 4 : 0;
    return i0 <= ntc && X + 4 * i0 < hi_c;
}

// exp2 of 32 scores of a row -> 16 packed bf16 pairs; columns at or past `valid` give 0.
template <bool kMasked>
__device__ __forceinline__ float softmax_half(const uint32_t (&sv)[32], int col0, int valid, float c2, float m,
                                              uint32_t (&pw)[16]) {
    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        float a = fast_exp2(fmaf(__uint_as_float(sv[2 * k]), c2, -m));
        float b = fast_exp2(fmaf(__uint_as_float(sv[2 * k + 1]), c2, -m));
        if (kMasked) {
            a = (col0 + 2 * k < valid) ? a : 0.f;
            b = (col0 + 2 * k + 1 < valid) ? b : 0.f;
        }
        sum0 += a;
        sum1 += b;
        pw[k] = pack_bf16(a, b);
    }
    return sum0 + sum1;
}

// ------------------------------------------------------------------ the kernel
//
// Warps: 0 TMA producer; 1 and 2 issue QK for M tile 0 and 1; 3 issues PV for every M
// tile; 4.. softmax, four warps per M tile.  The tensor pipe accepts MMAs from several
// issuing threads at once, while each issuing thread waits about a hundred cycles per
// MMA, so QK and PV run on separate issuers.

__global__ void __launch_bounds__(384, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kb,
               const __grid_constant__ CUtensorMap tm_vb, const TcParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ Shared sh;
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = p.NT;
    Bars &bar = sh.bar;

    if (threadIdx.x == 0) {
        mbar_init(&bar.q_full, 1);
        mbar_init(&bar.q_empty, NT);
        for (int s = 0; s < kKStages; ++s) { mbar_init(&bar.k_full[s], 1); mbar_init(&bar.k_empty[s], NT); }
        for (int s = 0; s < kVStages; ++s) { mbar_init(&bar.v_full[s], 1); mbar_init(&bar.v_empty[s], 1); }
        for (int s = 0; s < 2; ++s)
            for (int m = 0; m < 2; ++m) {
                mbar_init(&bar.s_full[s][m], 1);
                mbar_init(&bar.s_free[s][m], 1);
                mbar_init(&bar.p_full[s][m], 4);
            }
        for (int m = 0; m < 2; ++m) { mbar_init(&bar.o_full[m], 1); mbar_init(&bar.o_empty[m], 4); }
        mbar_init(&bar.grp, 4 * NT);
        for (int i = 0; i < 3; ++i) mbar_init(&bar.done[i], 1);
        fence_mbar_init();
        sh.abort = 0;
        prefetch_tmap(&tm_q); prefetch_tmap(&tm_k); prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_kb); prefetch_tmap(&tm_vb);
        for (int i = 0; i < p.B; ++i) {
            const int L = p.ctx_len[i];
            if (L < 0 || L > p.max_pages * kPage) { report_error(p.dev_err, TT_ERR_BOUNDS); break; }
        }
    }
    if (warp == 1) { tmem_alloc(&sh.tmem_base, kTmemCols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    WorkIter it;
    it.init(p, blockIdx.x);
    const int S = p.S, G = p.G;

    if (warp == 0) {
        // ================================================================ TMA producer
        // The whole warp walks the work (page ids are fetched 32 at a time, one per lane);
        // lane 0 issues the copies.
        Piece pc;
        int qi = 0, t = 0;
        bool issued = false;
        while (it.next(p, pc)) {
            if (!wait_bar(sh, &bar.q_empty, (qi & 1) ^ 1, p.dev_err)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(&bar.q_full, (uint32_t)(NT * 2 * kQTile));
                for (int mt = 0; mt < NT; ++mt)
                    for (int dh = 0; dh < 2; ++dh)
                        tma_load_3d(sm + kOffQ + (2 * mt + dh) * kQTile, &tm_q, &bar.q_full, 64 * dh, pc.g * G,
                                    pc.b * S + mt * (128 / G));
            }
            issued = true;
            bool ok = true;
            int my_page = 0;
            for (int i = pc.first; i < pc.last; ++i, ++t) {
                const int rel = i - pc.first;
                if ((rel & 31) == 0) {
                    const int ii = i + lane;
                    my_page = 0;
                    if (ii < pc.last && ii < pc.ntc) {
                        my_page = p.page_table[(size_t)pc.b * p.max_pages + ii];
                        if (my_page < 0 || my_page >= p.num_pages) {
                            report_error(p.dev_err, TT_ERR_BOUNDS);
                            my_page = 0;
                        }
                    }
                }
                const int page = __shfl_sync(0xffffffffu, my_page, rel & 31);
                const int kst = t % kKStages, vst = t % kVStages;
                if (!wait_bar(sh, &bar.k_empty[kst], ((uint32_t)(t / kKStages) & 1) ^ 1, p.dev_err)) { ok = false; break; }
                unsigned char *kd = sm + kOffK + kst * kTile;
                unsigned char *vd = sm + kOffV + vst * kTile;
                if (lane == 0) {
                    if (i < pc.ntc) {
                        mbar_arrive_expect_tx(&bar.k_full[kst], kTile);
                        tma_load_4d(kd, &tm_k, &bar.k_full[kst], 0, 0, pc.g, page);
                        tma_load_4d(kd + kHalf, &tm_k, &bar.k_full[kst], 64, 0, pc.g, page);
                    } else {
                        mbar_arrive_expect_tx(&bar.k_full[kst], (uint32_t)(2 * S * 128));
                        tma_load_3d(kd, &tm_kb, &bar.k_full[kst], 0, pc.g, pc.b * S);
                        tma_load_3d(kd + kHalf, &tm_kb, &bar.k_full[kst], 64, pc.g, pc.b * S);
                    }
                }
                if (!wait_bar(sh, &bar.v_empty[vst], ((uint32_t)(t / kVStages) & 1) ^ 1, p.dev_err)) {
                    ok = false;
                    ++t;   // the K copy of this tile is in flight: count it for the drain
                    break;
                }
                if (lane == 0) {
                    if (i < pc.ntc) {
                        mbar_arrive_expect_tx(&bar.v_full[vst], kTile);
                        tma_load_4d(vd, &tm_v, &bar.v_full[vst], 0, 0, pc.g, page);
                        tma_load_4d(vd + kHalf, &tm_v, &bar.v_full[vst], 64, 0, pc.g, page);
                    } else {
                        mbar_arrive_expect_tx(&bar.v_full[vst], (uint32_t)(2 * S * 128));
                        tma_load_3d(vd, &tm_vb, &bar.v_full[vst], 0, pc.g, pc.b * S);
                        tma_load_3d(vd + kHalf, &tm_vb, &bar.v_full[vst], 64, pc.g, pc.b * S);
                    }
                }
            }
            ++qi;
            if (!ok) break;
        }
        // Drain: every copy issued must land before the CTA may exit.  The last copy into
        // a stage completes that stage's latest phase.
        if (issued) mbar_wait(&bar.q_full, (uint32_t)(qi - 1) & 1, kWaitLimit);
        for (int k = 1; k <= kKStages && t - k >= 0; ++k)
            mbar_wait(&bar.k_full[(t - k) % kKStages], (uint32_t)((t - k) / kKStages) & 1, kWaitLimit);
        for (int k = 1; k <= kVStages && t - k >= 0; ++k)
            mbar_wait(&bar.v_full[(t - k) % kVStages], (uint32_t)((t - k) / kVStages) & 1, kWaitLimit);
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        // ================================================================ QK issuer of M tile mt
        const int mt = warp - 1;
        if (mt < NT) {
            Piece pc;
            int qi = 0, t = 0;
            bool ok = true;
            const uint32_t qa = smem_u32(sm + kOffQ + 2 * mt * kQTile);
            while (ok && it.next(p, pc)) {
                if (!wait_bar(sh, &bar.q_full, qi & 1, p.dev_err)) break;
                tc_fence_after();
                const int ntiles = pc.last - pc.first;
                for (int j = 0; j < ntiles; ++j, ++t) {
                    const int i = pc.first + j;
                    const int kst = t % kKStages, sb = t & 1;
                    const int valid = tile_valid(pc, i, S);
                    const int nk = (valid + 15) & ~15;
                    if (!wait_bar(sh, &bar.k_full[kst], (uint32_t)(t / kKStages) & 1, p.dev_err)) { ok = false; break; }
                    if (!wait_bar(sh, &bar.s_free[sb][mt], (((uint32_t)t >> 1) & 1) ^ 1, p.dev_err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t idesc = idesc_bf16_f32(128, nk, false, false);
                    const uint32_t kb = smem_u32(sm + kOffK + kst * kTile);
                    const uint32_t dcol = tmem + kColS + 64 * (2 * sb + mt);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t da = sdesc_sw128(qa + (kk >> 2) * (uint32_t)kQTile + (kk & 3) * 32, 16, 1024);
                        const uint64_t db = sdesc_sw128(kb + (kk >> 2) * (uint32_t)kHalf + (kk & 3) * 32, 16, 1024);
                        if (elect_one()) mma_bf16_ss(dcol, da, db, idesc, kk > 0);
                        __syncwarp();
                    }
                    if (elect_one()) {
                        mma_commit(&bar.s_full[sb][mt]);
                        mma_commit(&bar.k_empty[kst]);
                        if (j == ntiles - 1) mma_commit(&bar.q_empty);
                    }
                    __syncwarp();
                }
                ++qi;
            }
            if (elect_one()) mma_commit(&bar.done[mt]);
            __syncwarp();
        }
    } else if (warp == 3) {
        // ================================================================ PV issuer
        Piece pc;
        int t = 0, pi = 0;
        bool ok = true;
        const uint32_t idesc_pv = idesc_bf16_f32(128, kD, false, true);
        while (ok && it.next(p, pc)) {
            const int ntiles = pc.last - pc.first;
            for (int j = 0; j < ntiles && ok; ++j, ++t) {
                const int i = pc.first + j;
                const int vst = t % kVStages, sb = t & 1;
                const int valid = tile_valid(pc, i, S);
                const int nk = (valid + 15) & ~15;
                if (!wait_bar(sh, &bar.v_full[vst], (uint32_t)(t / kVStages) & 1, p.dev_err)) { ok = false; break; }
                unsigned char *v0 = sm + kOffV + vst * kTile;
                if (valid < nk) {
                    // rows [valid, nk) of this page are past the context: zero them in both halves
                    const int words = (nk - valid) * 8;   // 16-byte words per half
                    for (int w = lane; w < 2 * words; w += 32) {
                        const int h = w / words, r = valid + (w % words) / 8, c = w % 8;
                        *reinterpret_cast<uint4 *>(v0 + h * kHalf + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                for (int mt = 0; mt < NT; ++mt) {
                    if (!wait_bar(sh, &bar.p_full[sb][mt], ((uint32_t)t >> 1) & 1, p.dev_err)) { ok = false; break; }
                    if (j == 0 && !wait_bar(sh, &bar.o_empty[mt], (pi & 1) ^ 1, p.dev_err)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t pcol = tmem + kColS + 64 * (2 * sb + mt);
                    for (int kk = 0; kk < nk / 16; ++kk) {
                        const uint64_t dv = sdesc_sw128(smem_u32(v0) + kk * 2048, kHalf, 1024);
                        if (elect_one()) mma_bf16_ts(tmem + kColO + 128 * mt, pcol + 8 * kk, dv, idesc_pv, !(j == 0 && kk == 0));
                        __syncwarp();
                    }
                    if (elect_one()) {
                        mma_commit(&bar.s_free[sb][mt]);
                        if (j == ntiles - 1) mma_commit(&bar.o_full[mt]);
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (elect_one()) mma_commit(&bar.v_empty[vst]);
                __syncwarp();
            }
            ++pi;
        }
        if (elect_one()) mma_commit(&bar.done[2]);
        __syncwarp();
    } else if (warp >= 4 && warp < 4 + 4 * NT) {
        // ================================================================ softmax / epilogue
        const int mt = (warp - 4) >> 2, wq = warp & 3;
        const int r = 128 * mt + 32 * wq + lane;         // row of the segment: r = s * G + hh
        const int s_pos = r / G, hh = r % G;
        const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
        const float c2 = p.scale_log2;
        Piece pc;
        int t = 0, pi = 0, k_grp = 0;
        bool ok = true;
        while (ok && it.next(p, pc)) {
            float m_used = -INFINITY, l = 0.f;
            const int ntiles = pc.last - pc.first;
            for (int j = 0; j < ntiles; ++j, ++t) {
                const int i = pc.first + j;
                const int sb = t & 1;
                const int valid = tile_valid(pc, i, S);
                if (!wait_bar(sh, &bar.s_full[sb][mt], ((uint32_t)t >> 1) & 1, p.dev_err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t scol = tmem + lane_off + kColS + 64 * (2 * sb + mt);
                uint32_t sa[32], sc[32];
                tmem_ld32(scol, sa);
                if (valid > 32) tmem_ld32(scol + 32, sc);
                tmem_wait_ld();
                float mx0 = -INFINITY, mx1 = -INFINITY;
                if (valid == kPage) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        mx0 = fmaxf(mx0, __uint_as_float(sa[k]));
                        mx1 = fmaxf(mx1, __uint_as_float(sc[k]));
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        if (k < valid) mx0 = fmaxf(mx0, __uint_as_float(sa[k]));
                        if (k + 32 < valid) mx1 = fmaxf(mx1, __uint_as_float(sc[k]));
                    }
                }
                const float mt2 = fmaxf(mx0, mx1) * c2;
                const bool resc = mt2 > m_used + kRescaleThreshold;
                float alpha = 1.f;
                if (resc) {
                    alpha = (m_used == -INFINITY) ? 0.f : fast_exp2(m_used - mt2);
                    m_used = mt2;
                }
                // O rescale (rare: the row maximum grew by more than 2^8) once PV(t-1) is done;
                // warp-uniform because tcgen05.ld/st are warp-collective.
                if (j > 0 && __any_sync(0xffffffffu, resc)) {
                    if (!wait_bar(sh, &bar.s_free[(t - 1) & 1][mt], ((uint32_t)(t - 1) >> 1) & 1, p.dev_err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int ch = 0; ch < 4; ++ch) {
                        uint32_t o[32];
                        const uint32_t ocol = tmem + lane_off + kColO + 128 * mt + 32 * ch;
                        tmem_ld32(ocol, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st32(ocol, o);
                        tmem_wait_st();   // o is reused by the next chunk
                    }
                }
                // tcgen05.st reads its source registers asynchronously: each half has its own
                // registers, and nothing reuses them before tcgen05.wait::st.
                uint32_t pw0[16], pw1[16];
                float psum;
                if (valid == kPage) {
                    psum = softmax_half<false>(sa, 0, valid, c2, m_used, pw0);
                    psum += softmax_half<false>(sc, 32, valid, c2, m_used, pw1);
                    tmem_st16(scol, pw0);
                    tmem_st16(scol + 16, pw1);
                } else {
                    psum = softmax_half<true>(sa, 0, valid, c2, m_used, pw0);
                    tmem_st16(scol, pw0);
                    if (valid > 32) {
                        psum += softmax_half<true>(sc, 32, valid, c2, m_used, pw1);
                        tmem_st16(scol + 16, pw1);
                    }
                }
                tmem_wait_st();
                l = l * alpha + psum;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.p_full[sb][mt]);
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue of the piece
            if (!wait_bar(sh, &bar.o_full[mt], pi & 1, p.dev_err)) { ok = false; break; }
            tc_fence_after();
            const int hq = pc.g * G + hh;
            if (pc.whole) {
                const float inv = 1.f / l;
                uint16_t *orow = p.out + (((size_t)pc.b * S + s_pos) * p.Hq + hq) * kD;
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + kColO + 128 * mt + 32 * ch, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint4 w;
                        w.x = pack_bf16(__uint_as_float(o[8 * k + 0]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
                        w.y = pack_bf16(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
                        w.z = pack_bf16(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
                        w.w = pack_bf16(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
                        *reinterpret_cast<uint4 *>(orow + 32 * ch + 8 * k) = w;
                    }
                }
                if (p.lse) p.lse[((size_t)pc.b * p.Hq + hq) * S + s_pos] = (m_used + __log2f(l)) * kLn2;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.o_empty[mt]);
            } else {
                // partial: unnormalised O, the row maximum used (log2 units) and the row sum
                float *slot = p.part + (long long)(blockIdx.x + pc.sg) * p.slot_floats;
                float *orow = slot + (size_t)r * kD;
                for (int ch = 0; ch < 4; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + kColO + 128 * mt + 32 * ch, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        __stcg(reinterpret_cast<float4 *>(orow + 32 * ch + 4 * k),
                               make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                           __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3])));
                }
                __stcg(slot + (size_t)p.rows * kD + r, m_used);
                __stcg(slot + (size_t)p.rows * kD + p.rows + r, l);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.o_empty[mt]);
                __threadfence();
                if (!group_sync(sh, k_grp, p.dev_err)) { ok = false; break; }
                if (threadIdx.x == 128) {
                    const unsigned n_here = (unsigned)(pc.last - pc.first);
                    const unsigned before = atomicAdd(&p.tickets[pc.sg], n_here);
                    sh.last = (before + n_here == (unsigned)(pc.ntc + 1));
                }
                if (!group_sync(sh, k_grp, p.dev_err)) { ok = false; break; }
                if (sh.last) {
                    __threadfence();
                    // merge every piece of this segment, in CTA order
                    const long long U = it.U;
                    const int n = p.n_ctas;
                    const int c_first = owner(pc.X, U, n);
                    const int c_last = owner(pc.X + 4LL * pc.ntc, U, n);
                    float M = -INFINITY;
                    for (int c = c_first; c <= c_last; ++c) {
                        if (!owns_tile(c, pc.X, pc.ntc, U, n)) continue;
                        const float *sl = p.part + (long long)(c + pc.sg) * p.slot_floats;
                        M = fmaxf(M, __ldcg(sl + (size_t)p.rows * kD + r));
                    }
                    float Lsum = 0.f;
                    for (int c = c_first; c <= c_last; ++c) {
                        if (!owns_tile(c, pc.X, pc.ntc, U, n)) continue;
                        const float *sl = p.part + (long long)(c + pc.sg) * p.slot_floats;
                        Lsum += fast_exp2(__ldcg(sl + (size_t)p.rows * kD + r) - M) *
                                __ldcg(sl + (size_t)p.rows * kD + p.rows + r);
                    }
                    const float inv = 1.f / Lsum;
                    uint16_t *orow_out = p.out + (((size_t)pc.b * S + s_pos) * p.Hq + hq) * kD;
                    for (int ch = 0; ch < 4; ++ch) {
                        float acc[32];
#pragma unroll
                        for (int d = 0; d < 32; ++d) acc[d] = 0.f;
                        for (int c = c_first; c <= c_last; ++c) {
                            if (!owns_tile(c, pc.X, pc.ntc, U, n)) continue;
                            const float *sl = p.part + (long long)(c + pc.sg) * p.slot_floats;
                            const float w = fast_exp2(__ldcg(sl + (size_t)p.rows * kD + r) - M);
                            const float4 *orw = reinterpret_cast<const float4 *>(sl + (size_t)r * kD + 32 * ch);
#pragma unroll
                            for (int d4 = 0; d4 < 8; ++d4) {
                                const float4 v = __ldcg(orw + d4);
                                acc[4 * d4] += w * v.x; acc[4 * d4 + 1] += w * v.y;
                                acc[4 * d4 + 2] += w * v.z; acc[4 * d4 + 3] += w * v.w;
                            }
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint4 w;
                            w.x = pack_bf16(acc[8 * k + 0] * inv, acc[8 * k + 1] * inv);
                            w.y = pack_bf16(acc[8 * k + 2] * inv, acc[8 * k + 3] * inv);
                            w.z = pack_bf16(acc[8 * k + 4] * inv, acc[8 * k + 5] * inv);
                            w.w = pack_bf16(acc[8 * k + 6] * inv, acc[8 * k + 7] * inv);
                            *reinterpret_cast<uint4 *>(orow_out + 32 * ch + 8 * k) = w;
                        }
                    }
                    if (p.lse) p.lse[((size_t)pc.b * p.Hq + hq) * S + s_pos] = (M + __log2f(Lsum)) * kLn2;
                    if (threadIdx.x == 128) p.tickets[pc.sg] = 0;   // ready for the next launch
                }
            }
            ++pi;
        }
    }

    // ------------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        // every MMA of this CTA has completed (each issuer committed its last one)
        for (int i = 0; i < NT; ++i) mbar_wait(&bar.done[i], 0, kWaitLimit);
        mbar_wait(&bar.done[2], 0, kWaitLimit);
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

bool make_map(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims, const uint64_t *strides,
              const uint32_t *box) {
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; e[i] = 1; }
    for (int i = 0; i < rank - 1; ++i) s[i] = strides[i];
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(ptr), d, s, b, e,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int rows_of(int S, int Hq, int Hkv) { return (Hq / Hkv) * S; }

}  // namespace

bool attn_tc_supported(int S, int Hq, int Hkv, int D, int page_size, tt_dtype dtype) {
    // (a positive softmax scale is also required; the caller checks it)
    if (dtype != TT_BF16 || D != kD || page_size != kPage || Hkv < 1 || Hq % Hkv != 0) return false;
    const int G = Hq / Hkv;
    const int rows = G * S;
    return (S % 16 == 0) && S <= kPage && (rows == 128 || rows == 256) && (128 % G == 0);
}

size_t attn_tc_ws_bytes(int B, int S, int Hq, int Hkv, int D) {
    const size_t rows = (size_t)rows_of(S, Hq, Hkv);
    const size_t slot = (rows * D + 2 * rows) * sizeof(float);
    const size_t nseg = (size_t)B * Hkv;
    return align_up(nseg * sizeof(unsigned), 256) + (kMaxCtas + nseg) * slot;
}

tt_status launch_attn_tc(const AttnArgs &a) {
    const tt_kv_cache &c = *a.ctx;
    if (c.num_pages < 1) return launch_attn_simt(a);      // no pool to map: nothing paged to read
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TT_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TT_ERR_CUDA;
    const int G = a.Hq / a.Hkv;
    const int rows = G * a.S;
    const int NT = rows / 128;
    CUtensorMap mq, mk, mv, mkb, mvb;
    {
        const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.Hq, (uint64_t)a.B * a.S};
        const uint64_t str[2] = {(uint64_t)kD * 2, (uint64_t)a.Hq * kD * 2};
        const uint32_t box[3] = {64, (uint32_t)G, (uint32_t)(128 / G)};
        if (!make_map(&mq, a.q, 3, dims, str, box)) return TT_ERR_CUDA;
    }
    {
        const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)kPage, (uint64_t)a.Hkv, (uint64_t)c.num_pages};
        const uint64_t str[3] = {(uint64_t)kD * 2, (uint64_t)kPage * kD * 2, (uint64_t)a.Hkv * kPage * kD * 2};
        const uint32_t box[4] = {64, (uint32_t)kPage, 1, 1};
        if (!make_map(&mk, c.k_pool, 4, dims, str, box)) return TT_ERR_CUDA;
        if (!make_map(&mv, c.v_pool, 4, dims, str, box)) return TT_ERR_CUDA;
    }
    {
        const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.Hkv, (uint64_t)a.B * a.S};
        const uint64_t str[2] = {(uint64_t)kD * 2, (uint64_t)a.Hkv * kD * 2};
        const uint32_t box[3] = {64, 1, (uint32_t)a.S};
        if (!make_map(&mkb, a.k_blk, 3, dims, str, box)) return TT_ERR_CUDA;
        if (!make_map(&mvb, a.v_blk, 3, dims, str, box)) return TT_ERR_CUDA;
    }
    TcParams p;
    p.page_table = c.page_table;
    p.ctx_len = c.ctx_len;
    p.num_pages = c.num_pages;
    p.max_pages = c.max_pages_per_seq;
    p.out = static_cast<uint16_t *>(a.out);
    p.lse = a.lse;
    p.B = a.B; p.S = a.S; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.rows = rows; p.NT = NT;
    p.scale_log2 = a.sm_scale * kLog2e;
    int n = a.max_ctas > 0 ? a.max_ctas : sms;
    if (n > kMaxCtas) n = kMaxCtas;
    p.n_ctas = n;
    const size_t nseg = (size_t)a.B * a.Hkv;
    p.tickets = static_cast<unsigned *>(a.ws);
    p.part = reinterpret_cast<float *>(static_cast<char *>(a.ws) + align_up(nseg * sizeof(unsigned), 256));
    p.slot_floats = (long long)rows * kD + 2LL * rows;
    p.dev_err = a.dev_err;
    if (cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
        return TT_ERR_CUDA;
    attn_tc_kernel<<<n, 128 + 128 * NT, kSmemBytes, a.stream>>>(mq, mk, mv, mkb, mvb, p);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace tt
