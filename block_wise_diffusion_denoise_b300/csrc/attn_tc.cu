// Two-segment denoise attention on the 5th-generation tensor cores (bf16, D = 128,
// 64-token pages).
//
// What it computes (TwoTower summary on gist.science, "Technisches Resuemee --
// Architektur" and "Generierungsprozess"; dgnews.ru, "How the architecture
// actually works"): the S block queries of every query head attend, in one
// softmax, to all L context keys the frozen context tower holds for this layer
// and to the S keys of their own block, without a mask inside the block.  In the
// context tower's view of a committed block (the same summary makes that tower
// causal over the committed tokens) block query i reads block keys 0..i only:
// a second instance of the kernel (kCausal) that masks the block tile per row,
// so the denoise instance carries no code for it.
//
// Design for sm_103a:
//  * Rows.  The G = Hq/Hkv query heads of one KV head share every key, so the
//    G*S (s, head) rows of one (sequence, KV head) segment form the M side of
//    the MMAs.  Each CTA owns one 128-row M tile; when G*S is a larger
//    multiple of 128, neighbouring CTAs of the persistent grid (a group) take
//    the M tiles of the same rows and walk the same pages at the same time, so
//    the later reads of every page are served by L2 and HBM sees each byte once.
//  * Tensor memory (512 columns): O (128 fp32 columns), S (128, one tile, given
//    back as soon as the softmax has read it), P (two buffers of 64 columns of
//    packed bf16 pairs) and Q (64 columns of packed bf16 pairs).  Q lives in
//    tensor memory as the A operand of the QK product, which frees its 32 KB of
//    shared memory for a third V stage.
//  * Tiles.  A key tile is two 64-token pages of the paged cache (or the block's
//    own S keys).  Two producer warps move them with TMA (128-byte swizzle) into
//    separate three-stage K and V rings (a K stage is free once QK has read it,
//    a V stage once PV has), each fetching page ids 32 at a time; the K
//    producer also starts each tile's V pages towards L2.  Q is written into
//    tensor memory by the softmax warps once per piece.
//  * MMAs.  One warp issues S = Q K^T (M 128, N 128 keys, A from tensor
//    memory), another issues O += P V (M 128, N 128 = D, K 128 keys, A from
//    tensor memory); one elected lane of a converged warp issues a tile's eight
//    MMAs and their commits in one go (electing a lane per MMA, with a warp
//    barrier after each, measured 2-3 % slower).
//  * Softmax.  Two warps share each TMEM lane quarter and take alternate tiles,
//    one thread per row: the row's 128 scores come into registers at once and
//    S goes back to the QK issuer immediately; the running maximum (log2
//    domain) is taken over from the partner's previous tile and only raised --
//    with a rescale of O in TMEM -- when the tile exceeds it by more than 2^8; P
//    is written as packed bf16 into its own double-buffered TMEM tile.  The
//    exponent phase of one tile overlaps the next QK product and the score
//    phase of the partner's tile.  A register split (setmaxnreg) gives the
//    softmax warpgroups 208 registers per thread and the role warps 80.
//    Columns past the valid keys of a partial tile are masked, and the matching
//    V rows are zeroed before the PV product, so slots past L never matter.
//  * Work split.  The batch is a list of segments (b, g), each a run of
//    two-page tiles plus one block tile, counted in work units (a boundary
//    charge per segment, then a tile, then the block tile).  When every group
//    can take a whole segment and splitting would not pay, group i takes
//    segment i; otherwise the persistent grid cuts the list into equal unit
//    ranges, one per CTA group (stream-K style): a group that owns a whole
//    segment writes the final output; pieces of a shared segment go to fp32
//    partial slots and the last CTA to finish the segment's M tile (atomic
//    ticket, no waiting) merges them with log-sum-exp weights.  Ragged and long
//    contexts balance without host knowledge of the lengths, which live on the
//    device.
//  * Every mbarrier wait is bounded; a wait that gives up records
//    TT_ERR_DEVICE_TIMEOUT, the CTA drains its copies and MMAs and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "sm100_ptx.cuh"
#include "tt_common.cuh"
#include "tt_internal.h"
#include "attn_work.cuh"

namespace tt {
namespace {

using namespace sm100;

constexpr int kD = 128;                  // head dim
constexpr int kKStages = 3;              // K ring depth (K is needed first: QK starts a tile)
constexpr int kVStages = 3;              // V ring depth (a V stage is held until PV completes)
constexpr int kMaxCtas = 296;            // upper bound of the persistent grid (sizes the workspace)
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// Shared memory (offsets from a 1024-byte aligned base).  Every 128-row operand is
// stored as two 128-byte-swizzled halves of 64 columns (d 0..63 and d 64..127).
constexpr int kHalf = 16384;             // 128 rows x 128 bytes
constexpr int kStage = 2 * kHalf;        // one K or V tile (128 keys x 128 d)
constexpr int kOffK = 0;
constexpr int kOffV = kOffK + kKStages * kStage;
// Per-sequence table of one launch: clamped context lengths and the prefix sums of the
// sequences' work units (at most kSeqMax sequences per launch; the host splits larger
// batches into several launches).
constexpr int kSeqMax = 1024;
constexpr int kOffSeqPre = kOffV + kVStages * kStage;               // long long [kSeqMax + 1]
constexpr int kOffSeqLen = kOffSeqPre + 8 * (kSeqMax + 1);          // int [kSeqMax]
constexpr int kSmemBytes = kOffSeqLen + 4 * kSeqMax + 1024;

// TMEM columns (one M tile per CTA).
constexpr int kTmemCols = 512;
constexpr int kColO = 0;                 // O: 128 fp32 columns
constexpr int kColS = 128;               // S: 128 fp32 columns (released as soon as it is read)
constexpr int kColP = 256;               // P[buf]: 64 columns of packed bf16 pairs each
constexpr int kColQ = 384;               // Q: 64 columns of packed bf16 pairs (the A operand of QK)

struct TcParams {
    const uint16_t *q;            // [B, S, Hq, D] block queries (read into TMEM per piece)
    const int32_t *page_table;
    const int32_t *ctx_len;
    int num_pages, max_pages;
    uint16_t *out;
    float *lse;
    int B, S, Hq, Hkv, G, rows;
    int cps;                             // CTAs per segment (M tiles): 1 or 2
    float scale_log2;
    int n_groups;
    unsigned *tickets;                   // [segment][M tile]
    float *part;
    long long slot_floats;
    uint32_t *dev_err;
};

struct Bars {
    uint64_t q_full, q_empty;
    uint64_t k_full[kKStages], k_empty[kKStages];
    uint64_t v_full[kVStages], v_empty[kVStages];
    uint64_t s_full[2];    // [tile parity] S of the tile is in TMEM (QK committed).  One barrier
                           // per parity, so each is waited by one warp set in phase order (a
                           // shared one could be passed a phase early by the other set).
    uint64_t s_empty;      // the tile's four softmax warps have read S (waited by QK only)
    uint64_t p_full[2];    // the tile's four softmax warps wrote P
    uint64_t p_free[2];    // the PV product that read P has completed
    uint64_t pub[2][4];    // [tile parity][lane quarter]: the running maximum after the tile is published
    uint64_t o_full, o_empty;
    uint64_t grp;          // softmax warps among themselves (bounded, unlike bar.sync)
    uint64_t done[2];      // last MMA of each issuer has completed
};

struct Shared {
    Bars bar;
    float mpub[2][128];    // [tile parity][row]: running maximum after the tile (log2 units)
    float lsum[2][128];    // [warp half][row]: row sums at the end of a piece
    float lmax[2][128];    // [warp half][row]: the maximum each row sum is scaled by
    uint32_t tmem_base;
    int abort;
    int last;
    int max_len;           // longest context of the launch
};

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ bool wait_bar(Shared &sh, uint64_t *bar, uint32_t parity, uint32_t *dev_err) {
    if (*(volatile int *)&sh.abort) return false;
    if (mbar_wait(bar, parity, kWaitLimit)) return true;
    *(volatile int *)&sh.abort = 1;
    report_error(dev_err, TT_ERR_DEVICE_TIMEOUT);
    return false;
}

// All softmax warps meet (k-th meeting of this CTA); false if a warp never came.
__device__ __forceinline__ bool group_sync(Shared &sh, int &k, uint32_t *dev_err) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.bar.grp);
    const bool ok = wait_bar(sh, &sh.bar.grp, (uint32_t)k & 1, dev_err);
    ++k;
    return ok;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Register split between warpgroups: the launch gives 384 x 168 registers; the role
// warpgroup (warps 0-3) drops to 80 each and the two softmax warpgroups rise to 208
// each (128 x 80 + 256 x 208 = 63488 <= 64512).  Measured against 64 / 216: the
// attention 1.4 % and its causal-block view 2 % faster.
__device__ __forceinline__ void regs_release() { asm volatile("setmaxnreg.dec.sync.aligned.u32 80;"); }
__device__ __forceinline__ void regs_acquire() { asm volatile("setmaxnreg.inc.sync.aligned.u32 208;"); }

// Scores at columns at or past `valid` become -inf (only the last context tile of a
// segment and the block tile are partial), so one code path serves every tile.
__device__ __forceinline__ void mask_scores(uint32_t (&sv)[32], int col0, int valid) {
#pragma unroll
    for (int k = 0; k < 32; ++k)
        if (col0 + k >= valid) sv[k] = 0xff800000u;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Largest of 32 scores (two independent three-input chains).
__device__ __forceinline__ float chunk_max(const uint32_t (&sv)[32]) {
    float m0 = max3f(__uint_as_float(sv[0]), __uint_as_float(sv[1]), __uint_as_float(sv[2]));
    float m1 = max3f(__uint_as_float(sv[3]), __uint_as_float(sv[4]), __uint_as_float(sv[5]));
#pragma unroll
    for (int k = 6; k < 30; k += 4) {
        m0 = max3f(m0, __uint_as_float(sv[k]), __uint_as_float(sv[k + 1]));
        m1 = max3f(m1, __uint_as_float(sv[k + 2]), __uint_as_float(sv[k + 3]));
    }
    return max3f(m0, m1, fmaxf(__uint_as_float(sv[30]), __uint_as_float(sv[31])));
}

__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

// exp2(s * c - m) of 32 scores -> 16 packed bf16 pairs and their sum; the scale and the
// subtraction run as paired fp32 FMAs, the sums as paired adds.  cx2 = (c, c), nmx2 = (-m, -m).
__device__ __forceinline__ float softmax_chunk(const uint32_t (&sv)[32], uint64_t cx2, uint64_t nmx2,
                                               uint32_t (&pw)[16]) {
    uint64_t acc0 = 0, acc1 = 0;   // (+0, +0)
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        uint64_t y;
        asm("fma.rn.f32x2 %0, %1, %2, %3;"
            : "=l"(y)
            : "l"(f32x2(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1]))), "l"(cx2), "l"(nmx2));
        float y0, y1;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(y0), "=f"(y1) : "l"(y));
        const float a = fast_exp2(y0), b = fast_exp2(y1);
        if (k & 1) asm("add.f32x2 %0, %0, %1;" : "+l"(acc1) : "l"(f32x2(a, b)));
        else asm("add.f32x2 %0, %0, %1;" : "+l"(acc0) : "l"(f32x2(a, b)));
        pw[k] = pack_bf16(a, b);
    }
    asm("add.f32x2 %0, %0, %1;" : "+l"(acc0) : "l"(acc1));
    float s0, s1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(acc0));
    return s0 + s1;
}

// ------------------------------------------------------------------ the kernel
//
// Warps: 0 TMA producer of K; 1 QK issuer; 2 PV issuer; 3 TMA producer of V;
// 4..11 softmax and epilogue
// (two warps per TMEM lane quarter taking alternate tiles; at the end of a piece each
// writes half of the O columns).

template <bool kCausal>
__global__ void __launch_bounds__(384, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kb,
               const __grid_constant__ CUtensorMap tm_vb, const TcParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ Shared sh;
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = blockIdx.x / p.cps, mt = blockIdx.x % p.cps;
    Bars &bar = sh.bar;

    if (threadIdx.x == 0) {
        mbar_init(&bar.q_full, 4);
        mbar_init(&bar.q_empty, 1);
        for (int s = 0; s < kKStages; ++s) { mbar_init(&bar.k_full[s], 1); mbar_init(&bar.k_empty[s], 1); }
        for (int s = 0; s < kVStages; ++s) { mbar_init(&bar.v_full[s], 1); mbar_init(&bar.v_empty[s], 1); }
        for (int s = 0; s < 2; ++s) {

            mbar_init(&bar.p_full[s], 4);
            mbar_init(&bar.p_free[s], 1);
            for (int q = 0; q < 4; ++q) mbar_init(&bar.pub[s][q], 1);
        }
        mbar_init(&bar.s_full[0], 1);
        mbar_init(&bar.s_full[1], 1);
        mbar_init(&bar.s_empty, 4);
        mbar_init(&bar.o_full, 1);
        mbar_init(&bar.o_empty, 8);
        mbar_init(&bar.grp, 8);
        for (int i = 0; i < 2; ++i) mbar_init(&bar.done[i], 1);
        fence_mbar_init();
        sh.abort = 0;
        prefetch_tmap(&tm_k); prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_kb); prefetch_tmap(&tm_vb);
    }
    // the sequence table: lengths loaded by all threads at once, prefix sums by warp 2
    long long *seq_pre = reinterpret_cast<long long *>(sm + kOffSeqPre);
    int *seq_len = reinterpret_cast<int *>(sm + kOffSeqLen);
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        int L = p.ctx_len[i];
        if (L < 0 || L > p.max_pages * kPage) {
            report_error(p.dev_err, TT_ERR_BOUNDS);
            L = 0;
        }
        seq_len[i] = L;
    }
    if (warp == 1) { tmem_alloc(&sh.tmem_base, kTmemCols); tmem_relinquish(); }
    __syncthreads();
    if (warp == 2) {
        long long carry = 0;
        int mlen = 0;
        if (lane == 0) seq_pre[0] = 0;
        for (int base = 0; base < p.B; base += 32) {
            const int i = base + lane;
            long long v = (i < p.B) ? (long long)seq_cost<TcCosts>(seq_len[i], p.Hkv) : 0;
            if (i < p.B) mlen = max(mlen, seq_len[i]);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (i < p.B) seq_pre[i + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
        mlen = __reduce_max_sync(0xffffffffu, mlen);
        if (lane == 0) sh.max_len = mlen;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    WorkIter<TcCosts> it;
    it.init(p, group, seq_pre, seq_len, sh.max_len);
    const int S = p.S, G = p.G;

    if (warp == 0 || warp == 3) {
        regs_release();
        // ================================================================ TMA producers
        // Warp 0 loads K, warp 3 loads V, so that a K copy never waits behind the
        // release of a V stage (they are freed by different products).  Each whole warp
        // walks the work (page ids are fetched 32 at a time, one per lane); lane 0 issues
        // the copies.
        const bool is_v = warp == 3;
        const CUtensorMap *tm_pool = is_v ? &tm_v : &tm_k;
        const CUtensorMap *tm_blk = is_v ? &tm_vb : &tm_kb;
        const int nst = is_v ? kVStages : kKStages;
        uint64_t *full = is_v ? bar.v_full : bar.k_full;
        uint64_t *empty = is_v ? bar.v_empty : bar.k_empty;
        unsigned char *ring = sm + (is_v ? kOffV : kOffK);
        Piece pc;
        int t = 0;
        while (it.next(p, pc)) {
            bool ok = true;
            int my_page = 0;
            for (int i = pc.first; i < pc.last; ++i, ++t) {
                // page ids of tiles [i, i + 16): lane l holds page 2i + l of the sequence
                const int rel = i - pc.first;
                if ((rel & 15) == 0) my_page = page_id(p, pc, 2 * i + lane);
                const int page0 = __shfl_sync(0xffffffffu, my_page, (2 * rel) & 31);
                const int page1 = __shfl_sync(0xffffffffu, my_page, (2 * rel + 1) & 31);
                const int valid = tile_valid(pc, i, S);
                const bool ctx = i < pc.ntc;
                const bool two = ctx && valid > kPage;
                const int st = t % nst;
                if (!wait_bar(sh, &empty[st], ((uint32_t)(t / nst) & 1) ^ 1, p.dev_err)) { ok = false; break; }
                unsigned char *dst = ring + st * kStage;
                if (lane == 0) {
                    if (ctx && !is_v) {
                        // The same tile's V pages are needed two tile periods later than its
                        // K, behind a shallower ring: start them towards L2 now.
                        tma_prefetch_4d(&tm_v, 0, 0, pc.g, page0);
                        tma_prefetch_4d(&tm_v, 64, 0, pc.g, page0);
                        if (two) {
                            tma_prefetch_4d(&tm_v, 0, 0, pc.g, page1);
                            tma_prefetch_4d(&tm_v, 64, 0, pc.g, page1);
                        }
                    }
                    if (ctx) {
                        mbar_arrive_expect_tx(&full[st], two ? 4 * 8192u : 2 * 8192u);
                        tma_load_4d(dst, tm_pool, &full[st], 0, 0, pc.g, page0);
                        tma_load_4d(dst + kHalf, tm_pool, &full[st], 64, 0, pc.g, page0);
                        if (two) {
                            tma_load_4d(dst + 8192, tm_pool, &full[st], 0, 0, pc.g, page1);
                            tma_load_4d(dst + kHalf + 8192, tm_pool, &full[st], 64, 0, pc.g, page1);
                        }
                    } else {
                        mbar_arrive_expect_tx(&full[st], (uint32_t)(2 * S * 128));
                        tma_load_3d(dst, tm_blk, &full[st], 0, pc.g, pc.b * S);
                        tma_load_3d(dst + kHalf, tm_blk, &full[st], 64, pc.g, pc.b * S);
                    }
                }
            }
            if (!ok) break;
        }
        // Drain: every copy issued must land before the CTA may exit.  The last copy into
        // a stage completes that stage's latest phase.
        for (int k = 1; k <= nst && t - k >= 0; ++k)
            mbar_wait(&full[(t - k) % nst], (uint32_t)((t - k) / nst) & 1, kWaitLimit);
        __syncwarp();
    } else if (warp == 1) {
        regs_release();
        // ================================================================ QK issuer
        Piece pc;
        int qi = 0, t = 0;
        bool ok = true;
        while (ok && it.next(p, pc)) {
            if (!wait_bar(sh, &bar.q_full, qi & 1, p.dev_err)) break;
            tc_fence_after();
            const int ntiles = pc.last - pc.first;
            for (int j = 0; j < ntiles; ++j, ++t) {
                const int kst = t % kKStages;
                const int valid = tile_valid(pc, pc.first + j, S);
                const int nk = (valid + 15) & ~15;
                if (!wait_bar(sh, &bar.k_full[kst], (uint32_t)(t / kKStages) & 1, p.dev_err)) { ok = false; break; }
                // S is single-buffered: the previous tile's scores must have been read
                if (t > 0 && !wait_bar(sh, &bar.s_empty, (uint32_t)(t - 1) & 1, p.dev_err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(128, nk, false, false);
                const uint32_t kb = smem_u32(sm + kOffK + kst * kStage);
                const uint32_t dcol = tmem + kColS;
                if (elect_one()) {   // one lane issues the tile's MMAs and their commits
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {   // 16 head dimensions per step; Q from TMEM
                        const uint64_t db = sdesc_sw128(kb + (kk >> 2) * (uint32_t)kHalf + (kk & 3) * 32, 16, 1024);
                        mma_bf16_ts(dcol, tmem + kColQ + 8 * kk, db, idesc, kk > 0);
                    }
                    mma_commit(&bar.s_full[t & 1]);
                    mma_commit(&bar.k_empty[kst]);
                    if (j == ntiles - 1) mma_commit(&bar.q_empty);
                }
                __syncwarp();
            }
            ++qi;
        }
        if (elect_one()) mma_commit(&bar.done[0]);
        __syncwarp();
    } else if (warp == 2) {
        regs_release();
        // ================================================================ PV issuer
        Piece pc;
        int t = 0, pi = 0;
        bool ok = true;
        const uint32_t idesc_pv = idesc_bf16_f32(128, kD, false, true);
        while (ok && it.next(p, pc)) {
            const int ntiles = pc.last - pc.first;
            for (int j = 0; j < ntiles; ++j, ++t) {
                const int vst = t % kVStages, sb = t & 1;
                const int valid = tile_valid(pc, pc.first + j, S);
                const int nk = (valid + 15) & ~15;
                if (!wait_bar(sh, &bar.v_full[vst], (uint32_t)(t / kVStages) & 1, p.dev_err)) { ok = false; break; }
                unsigned char *vp = sm + kOffV + vst * kStage;
                if (valid < nk) {
                    // rows [valid, nk) of this tile are past the context: zero them in both halves
                    const int words = (nk - valid) * 8;   // 16-byte words per half
                    for (int w = lane; w < 2 * words; w += 32) {
                        const int h = w / words, r = valid + (w % words) / 8, c = w % 8;
                        *reinterpret_cast<uint4 *>(vp + h * kHalf + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (!wait_bar(sh, &bar.p_full[sb], ((uint32_t)t >> 1) & 1, p.dev_err)) { ok = false; break; }
                if (j == 0 && !wait_bar(sh, &bar.o_empty, (pi & 1) ^ 1, p.dev_err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t v0 = smem_u32(vp);
                const uint32_t pcol = tmem + kColP + 64 * sb;
                if (elect_one()) {   // one lane issues the tile's MMAs and their commits
                    for (int kk = 0; kk < nk / 16; ++kk) {
                        const uint64_t dv = sdesc_sw128(v0 + kk * 2048, kHalf, 1024);
                        mma_bf16_ts(tmem + kColO, pcol + 8 * kk, dv, idesc_pv, !(j == 0 && kk == 0));
                    }
                    mma_commit(&bar.p_free[sb]);
                    mma_commit(&bar.v_empty[vst]);
                    if (j == ntiles - 1) mma_commit(&bar.o_full);
                }
                __syncwarp();
            }
            ++pi;
        }
        if (elect_one()) mma_commit(&bar.done[1]);
        __syncwarp();
    } else {
        regs_acquire();
        // ================================================================ softmax / epilogue
        // Warps 4 + q and 8 + q both read TMEM lanes 32q..32q+31 (rows of quarter q) and
        // take alternate tiles (half h = t & 1), so the exponent phase of tile t overlaps
        // the score phase of tile t+1.  Only the running maximum passes from one to the
        // next (one-directional, through shared memory); each keeps its own row sum in
        // the scale of the last maximum it used.
        const int wq = warp & 3, h = (warp - 4) >> 2;
        const int rl = 32 * wq + lane;                   // row within the M tile
        const int r = 128 * mt + rl;                     // row of the segment: r = s * G + hh
        const int s_pos = r / G, hh = r % G;
        const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
        const float c2 = p.scale_log2;
        // Q of a piece into TMEM (the A operand of QK): the h = 0 warps write their rows,
        // once the QK products of the previous piece are done with the old Q.
        int qn = 0;
        auto load_q = [&](const Piece &qc) -> bool {
            if (qn > 0 && !wait_bar(sh, &bar.q_empty, (uint32_t)(qn - 1) & 1, p.dev_err)) return false;
            const uint4 *src = reinterpret_cast<const uint4 *>(
                p.q + (((size_t)qc.b * S + s_pos) * p.Hq + qc.g * G + hh) * kD);
            tc_fence_after();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t w[32];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 v = __ldg(src + 8 * half + k);
                    w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
                }
                tmem_st32(tmem + lane_off + kColQ + 32 * half, w);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.q_full);
            ++qn;
            return true;
        };
        Piece pc, npc;
        int t = 0, pi = 0, k_grp = 0;
        bool ok = true;
        bool have = it.next(p, pc);
        if (have && h == 0) ok = load_q(pc);
        while (ok && have) {
            float m_l = -INFINITY, l = 0.f;              // my row sum and the maximum it is scaled by
            float m_last = -INFINITY;                    // maximum after my latest tile
            const int ntiles = pc.last - pc.first;
            for (int j = 0; j < ntiles; ++j, ++t) {
                if ((t & 1) != h) continue;              // the partner's tile
                const int sb = h;                        // P buffer of this tile
                int valid = tile_valid(pc, pc.first + j, S);
                if constexpr (kCausal) {
                    if (pc.first + j == pc.ntc) valid = s_pos + 1;   // block keys 0..s_pos
                }
                if (!wait_bar(sh, &bar.s_full[h], ((uint32_t)t >> 1) & 1, p.dev_err)) { ok = false; break; }
                tc_fence_after();
                const uint32_t scol = tmem + lane_off + kColS;
                // ---- the row's 128 scores into registers (all loads in flight at once), its
                // maximum, and S released to the next QK product right away
                uint32_t a0[32], a1[32], a2[32], a3[32];
                tmem_ld32(scol, a0);
                tmem_ld32(scol + 32, a1);
                tmem_ld32(scol + 64, a2);
                tmem_ld32(scol + 96, a3);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.s_empty);
                if (valid < kTileKeys) {   // warp-uniform (per row on a causal block tile)
                    mask_scores(a0, 0, valid);
                    mask_scores(a1, 32, valid);
                    mask_scores(a2, 64, valid);
                    mask_scores(a3, 96, valid);
                }
                const float mx = fmaxf(fmaxf(chunk_max(a0), chunk_max(a1)), fmaxf(chunk_max(a2), chunk_max(a3)));
                // ---- the running maximum: the previous tile's (from the partner), raised when
                // this tile's maximum exceeds it by more than 2^8
                float m_prev = -INFINITY;
                if (j > 0) {
                    if (!wait_bar(sh, &bar.pub[(t - 1) & 1][wq], ((uint32_t)(t - 1) >> 1) & 1, p.dev_err)) {
                        ok = false;
                        break;
                    }
                    m_prev = sh.mpub[(t - 1) & 1][rl];
                }
                const float mt2 = mx * c2;
                const float m_t = (mt2 > m_prev + kRescaleThreshold) ? mt2 : m_prev;
                sh.mpub[t & 1][rl] = m_t;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.pub[t & 1][wq]);
                // P buffer sb is free once the PV product of tile t-2 has completed.
                if (!wait_bar(sh, &bar.p_free[sb], (((uint32_t)t >> 1) & 1) ^ 1, p.dev_err)) { ok = false; break; }
                // O rescale (rare: the maximum moved at this tile) between PV(t-1) and PV(t);
                // warp-uniform because tcgen05.ld/st are warp-collective.
                const bool moved = j > 0 && m_t != m_prev;
                if (__any_sync(0xffffffffu, moved)) {
                    if (!wait_bar(sh, &bar.p_free[sb ^ 1], ((uint32_t)(t - 1) >> 1) & 1, p.dev_err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float alpha = moved ? fast_exp2(m_prev - m_t) : 1.f;
                    // 16 columns at a time: the tile's scores are live in registers meanwhile
                    for (int ch = 0; ch < 8; ++ch) {
                        uint32_t o[16];
                        const uint32_t ocol = tmem + lane_off + kColO + 16 * ch;
                        tmem_ld16(ocol, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
                        tmem_st16(ocol, o);
                        tmem_wait_st();   // o is reused by the next chunk
                    }
                }
                tc_fence_after();
                if (m_l != -INFINITY && m_l != m_t) l *= fast_exp2(m_l - m_t);
                m_l = m_t;
                m_last = m_t;
                // ---- P = 2^(s*c - m_t) as packed bf16 into TMEM (tcgen05.st takes its source
                // registers at issue; tcgen05.wait::st below orders the TMEM writes before the PV
                // product)
                const uint32_t pcolt = tmem + lane_off + kColP + 64 * sb;
                const uint64_t cx2 = f32x2(c2, c2), nmx2 = f32x2(-m_t, -m_t);
                uint32_t pw[16];
                float psum = softmax_chunk(a0, cx2, nmx2, pw);
                tmem_st16(pcolt, pw);
                psum += softmax_chunk(a1, cx2, nmx2, pw);
                tmem_st16(pcolt + 16, pw);
                psum += softmax_chunk(a2, cx2, nmx2, pw);
                tmem_st16(pcolt + 32, pw);
                psum += softmax_chunk(a3, cx2, nmx2, pw);
                tmem_st16(pcolt + 48, pw);
                tmem_wait_st();
                l += psum;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.p_full[sb]);
            }
            if (!ok) break;
            // the next piece's Q, ahead of this piece's epilogue so that its QK can start
            const bool have_next = it.next(p, npc);
            if (have_next && h == 0 && !load_q(npc)) { ok = false; break; }
            // ---------------------------------------------------------- epilogue of the piece
            if (!wait_bar(sh, &bar.o_full, pi & 1, p.dev_err)) { ok = false; break; }
            tc_fence_after();
            // merge the two row sums in the scale of the final maximum (the larger of the two)
            sh.lsum[h][rl] = l;
            sh.lmax[h][rl] = m_last;
            if (!group_sync(sh, k_grp, p.dev_err)) { ok = false; break; }
            {
                const float l2 = sh.lsum[h ^ 1][rl], m2 = sh.lmax[h ^ 1][rl];
                const float mf = fmaxf(m_last, m2);
                l = (m_last == -INFINITY ? 0.f : l * fast_exp2(m_last - mf)) +
                    (m2 == -INFINITY ? 0.f : l2 * fast_exp2(m2 - mf));
                m_last = mf;
            }
            const float m_used = m_last;
            const int hq = pc.g * G + hh;
            if (pc.whole) {
                const float inv = 1.f / l;
                uint16_t *orow = p.out + (((size_t)pc.b * S + s_pos) * p.Hq + hq) * kD + 64 * h;
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + kColO + 64 * h + 32 * ch, o);
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
                if (p.lse && h == 0) p.lse[((size_t)pc.b * p.Hq + hq) * S + s_pos] = (m_used + __log2f(l)) * kLn2;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.o_empty);
            } else {
                // partial: unnormalised O, the row maximum used (log2 units) and the row sum.
                // O is stored as [column / 4][row][4] so that the lanes (consecutive rows)
                // write, and later read, consecutive 16-byte pieces.
                float *slot = p.part + (long long)(group + pc.sg) * p.slot_floats;
                float4 *ocol4 = reinterpret_cast<float4 *>(slot) + r;
                for (int ch = 0; ch < 2; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_off + kColO + 64 * h + 32 * ch, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        __stcg(ocol4 + (size_t)(16 * h + 8 * ch + k) * p.rows,
                               make_float4(__uint_as_float(o[4 * k]), __uint_as_float(o[4 * k + 1]),
                                           __uint_as_float(o[4 * k + 2]), __uint_as_float(o[4 * k + 3])));
                }
                if (h == 0) {
                    __stcg(slot + (size_t)p.rows * kD + r, m_used);
                    __stcg(slot + (size_t)p.rows * kD + p.rows + r, l);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.o_empty);
                // One thread publishes the whole group's partial: the group barrier orders
                // every thread's stores before its release, the acquire half orders the
                // merge's loads (of the other pieces) after it.
                if (!group_sync(sh, k_grp, p.dev_err)) { ok = false; break; }
                unsigned *ticket = p.tickets + (size_t)pc.sg * p.cps + mt;
                if (threadIdx.x == 128) {
                    const unsigned n_here = (unsigned)(pc.last - pc.first);
                    const unsigned before = atom_add_acq_rel_gpu(ticket, n_here);
                    sh.last = (before + n_here == (unsigned)(pc.ntc + 1));
                }
                if (!group_sync(sh, k_grp, p.dev_err)) { ok = false; break; }
                if (sh.last) {
                    // Merge every piece of this segment's M tile in group order: an online
                    // rescale, so each piece costs one round trip (its maximum, sum and 64
                    // output values are loaded together).
                    const long long U = it.U;
                    const int n = it.NG;
                    const int c_first = first_owner<TcCosts>(pc.X, U, n);
                    const int c_last = last_owner<TcCosts>(pc.X, pc.ntc, U, n);
                    float M = -INFINITY, Lsum = 0.f;
                    float acc[64];
#pragma unroll
                    for (int d = 0; d < 64; ++d) acc[d] = 0.f;
                    for (int c = c_first; c <= c_last; ++c) {
                        if (!owns_tile<TcCosts>(c, pc.X, pc.ntc, U, n)) continue;
                        const float *sl = p.part + (long long)(c + pc.sg) * p.slot_floats;
                        const float4 *orw = reinterpret_cast<const float4 *>(sl) + (size_t)16 * h * p.rows + r;
                        float4 v[16];
#pragma unroll
                        for (int d4 = 0; d4 < 16; ++d4) v[d4] = __ldcg(orw + (size_t)d4 * p.rows);
                        const float mc = __ldcg(sl + (size_t)p.rows * kD + r);
                        const float lc = __ldcg(sl + (size_t)p.rows * kD + p.rows + r);
                        const float Mn = fmaxf(M, mc);
                        const float a = fast_exp2(M - Mn), w = fast_exp2(mc - Mn);
                        Lsum = Lsum * a + lc * w;
#pragma unroll
                        for (int d4 = 0; d4 < 16; ++d4) {
                            acc[4 * d4] = acc[4 * d4] * a + w * v[d4].x;
                            acc[4 * d4 + 1] = acc[4 * d4 + 1] * a + w * v[d4].y;
                            acc[4 * d4 + 2] = acc[4 * d4 + 2] * a + w * v[d4].z;
                            acc[4 * d4 + 3] = acc[4 * d4 + 3] * a + w * v[d4].w;
                        }
                        M = Mn;
                    }
                    const float inv = 1.f / Lsum;
                    uint16_t *orow_out = p.out + (((size_t)pc.b * S + s_pos) * p.Hq + hq) * kD + 64 * h;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        uint4 w;
                        w.x = pack_bf16(acc[8 * k + 0] * inv, acc[8 * k + 1] * inv);
                        w.y = pack_bf16(acc[8 * k + 2] * inv, acc[8 * k + 3] * inv);
                        w.z = pack_bf16(acc[8 * k + 4] * inv, acc[8 * k + 5] * inv);
                        w.w = pack_bf16(acc[8 * k + 6] * inv, acc[8 * k + 7] * inv);
                        *reinterpret_cast<uint4 *>(orow_out + 8 * k) = w;
                    }
                    if (p.lse && h == 0)
                        p.lse[((size_t)pc.b * p.Hq + hq) * S + s_pos] = (M + __log2f(Lsum)) * kLn2;
                    if (threadIdx.x == 128) *ticket = 0;   // ready for the next launch
                }
            }
            ++pi;
            pc = npc;
            have = have_next;
        }
    }

    // ------------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        // every MMA of this CTA has completed (each issuer committed its last one)
        mbar_wait(&bar.done[0], 0, kWaitLimit);
        mbar_wait(&bar.done[1], 0, kWaitLimit);
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side

int rows_of(int S, int Hq, int Hkv) { return (Hq / Hkv) * S; }

}  // namespace

bool attn_tc_supported(int S, int Hq, int Hkv, int D, int page_size, tt_dtype dtype) {
    // (a positive softmax scale is also required; the caller checks it)
    if (dtype != TT_BF16 || D != kD || page_size != kPage || Hkv < 1 || Hq % Hkv != 0) return false;
    const int G = Hq / Hkv;
    const int rows = G * S;
    // whole 128-row M tiles, one CTA each, at most 16 CTAs per segment
    return (S % 16 == 0) && S <= kTileKeys && rows % 128 == 0 && rows <= 16 * 128;
}

size_t attn_tc_ws_bytes(int B, int S, int Hq, int Hkv, int D) {
    const size_t rows = (size_t)rows_of(S, Hq, Hkv);
    const size_t slot = (rows * D + 2 * rows) * sizeof(float);
    const size_t nseg = (size_t)(B < kSeqMax ? B : kSeqMax) * Hkv;   // one launch's segments
    return align_up(rows / 128 * nseg * sizeof(unsigned), 256) + (kMaxCtas + nseg) * slot;
}

namespace {

// One launch over sequences [b0, b0 + nb) (nb <= kSeqMax): every per-sequence pointer is
// offset to b0, the pools are shared.
tt_status launch_chunk(const AttnArgs &a, int b0, int nb, int sms) {
    const tt_kv_cache &c = *a.ctx;
    const size_t qrow = (size_t)a.Hq * kD, kvrow = (size_t)a.Hkv * kD;
    const uint16_t *q = static_cast<const uint16_t *>(a.q) + (size_t)b0 * a.S * qrow;
    const uint16_t *k_blk = static_cast<const uint16_t *>(a.k_blk) + (size_t)b0 * a.S * kvrow;
    const uint16_t *v_blk = static_cast<const uint16_t *>(a.v_blk) + (size_t)b0 * a.S * kvrow;
    const int G = a.Hq / a.Hkv;
    const int rows = G * a.S;
    const int cps = rows / 128;   // CTAs per segment, one per 128-row M tile
    CUtensorMap mk, mv, mkb, mvb;
    if (!make_pool_maps(c, a.Hkv, &mk, &mv)) return TT_ERR_CUDA;
    {
        const uint64_t dims[3] = {(uint64_t)kD, (uint64_t)a.Hkv, (uint64_t)nb * a.S};
        const uint64_t str[2] = {(uint64_t)kD * 2, (uint64_t)a.Hkv * kD * 2};
        const uint32_t box[3] = {64, 1, (uint32_t)a.S};
        if (!make_map(&mkb, k_blk, 3, dims, str, box)) return TT_ERR_CUDA;
        if (!make_map(&mvb, v_blk, 3, dims, str, box)) return TT_ERR_CUDA;
    }
    TcParams p;
    p.q = q;
    p.page_table = c.page_table + (size_t)b0 * c.max_pages_per_seq;
    p.ctx_len = c.ctx_len + b0;
    p.num_pages = c.num_pages;
    p.max_pages = c.max_pages_per_seq;
    p.out = static_cast<uint16_t *>(a.out) + (size_t)b0 * a.S * qrow;
    p.lse = a.lse ? a.lse + (size_t)b0 * a.Hq * a.S : nullptr;
    p.B = nb; p.S = a.S; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.rows = rows; p.cps = cps;
    p.scale_log2 = a.sm_scale * kLog2e;
    int n = a.max_ctas > 0 ? a.max_ctas : sms;
    if (n > kMaxCtas) n = kMaxCtas;
    const int n_groups = n / cps > 0 ? n / cps : 1;
    p.n_groups = n_groups;
    const size_t nseg = (size_t)nb * a.Hkv;
    p.tickets = static_cast<unsigned *>(a.ws);
    p.part = reinterpret_cast<float *>(static_cast<char *>(a.ws) + align_up((size_t)cps * nseg * sizeof(unsigned), 256));
    p.slot_floats = (long long)rows * kD + 2LL * rows;
    p.dev_err = a.dev_err;
    auto kernel = a.causal_block ? attn_tc_kernel<true> : attn_tc_kernel<false>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
        return TT_ERR_CUDA;
    kernel<<<n_groups * cps, 384, kSmemBytes, a.stream>>>(mk, mv, mkb, mvb, p);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace

// Batches above the kernel's sequence table run as consecutive launches on the stream;
// they share the workspace, which each launch leaves as it found it (tickets zero).
tt_status launch_attn_tc(const AttnArgs &a) {
    if (a.ctx->num_pages < 1) return launch_attn_simt(a);   // no pool to map: nothing paged to read
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TT_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TT_ERR_CUDA;
    for (int b0 = 0; b0 < a.B; b0 += kSeqMax) {
        const tt_status st = launch_chunk(a, b0, a.B - b0 < kSeqMax ? a.B - b0 : kSeqMax, sms);
        if (st != TT_OK) return st;
    }
    return TT_OK;
}

}  // namespace tt
