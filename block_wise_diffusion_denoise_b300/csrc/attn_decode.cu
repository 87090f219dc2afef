// Decode attention on the 5th-generation tensor cores: a block of one position (S = 1),
// G = 16 query heads per KV head, bf16, D = 128, 64-token pages.
//
// What it computes is the two-segment attention of the denoise step (TwoTower summary on
// gist.science, "Technisches Resuemee -- Architektur"; dgnews.ru, "How the architecture
// actually works") for a block of one token: each query head attends, in one softmax, to
// the L context keys of its KV head and to the token's own key.  That is one step of
// autoregressive decoding, the baseline the pages measure the block-wise diffusion
// against (dgnews.ru, "What the tests actually show": generation throughput relative to
// AR decoding), served here from the same paged cache.
//
// Design for sm_103a.  The 16 query heads of a KV head read the same keys, so every K and
// V byte is brought in once for all of them.  The products are transposed so that the 128
// keys of a tile, not the 16 heads, fill the M side of the MMA:
//   S^T [128 keys x 16 heads]  = K_tile [128 x 128 d] . Q^T         (M 128, N 16, K 128 d)
//   O^T [128 d x 16 heads]    += V_tile^T [128 d x keys] . P^T      (M 128, N 16, K keys)
// K is the A operand as staged (K-major, 128-byte swizzle); V^T is the same staged V tile
// read M-major; Q and P^T are 16-row K-major tiles in shared memory.  Accumulators live in
// tensor memory: two S^T buffers and O^T, 16 columns each.
//  * Warps: 0 and 6 move K and V tiles by TMA into two 3-stage rings (0 also each piece's
//    16 query rows); 1 issues the QK products and 7 the PV products;
//    2-5 (one per TMEM lane quarter) run the softmax, one key per thread: the 16 scores of
//    the key come from tensor memory, each head's maximum over the tile by a warp
//    reduction and an exchange between the four warps in shared memory; the running
//    maximum of a head is raised only when the tile exceeds it by more than 2^8 (a lazy
//    rescale of O^T, exact because the final normalisation uses the same maximum), and
//    P = 2^(s*c - m) goes as bf16 into a double-buffered P^T tile.  At the end of a piece
//    thread r holds d lane r of O^T for the 16 heads and finishes their outputs.
//  * Work split: the device-side split of the 128-row kernel (attn_work.cuh) with one CTA
//    per group and a cost model of its own: whole segments, or stream-K pieces whose fp32
//    partials (O^T, m, l) are merged with log-sum-exp weights by the CTA that completes
//    the segment's ticket, after its own tiles.  Page ids are loaded a batch ahead of
//    their use and Q is double-buffered, so that the producers never stall at a batch or
//    piece boundary.
//  * Every mbarrier wait is bounded; a wait that gives up records TT_ERR_DEVICE_TIMEOUT,
//    and the CTA drains its copies and MMAs and exits.

#include <cuda.h>
#include <cudaTypedefs.h>

#include "sm100_ptx.cuh"
#include "tt_common.cuh"
#include "tt_internal.h"
#include "attn_work.cuh"

namespace tt {
namespace {

using namespace sm100;

constexpr int kDD = 128;                   // head dim
constexpr int kG = 16;                     // query heads per KV head: the N of both products
constexpr int kRingK = 3;                  // K ring depth (a K stage is free once QK has read it)
constexpr int kRingV = 3;                  // V ring depth (a V stage is held until PV completes)
constexpr int kTileHalf = 16384;           // one 64-column half of a 128-key tile (128 rows x 128 B)
constexpr int kTile = 2 * kTileHalf;
constexpr int kSmallHalf = kG * 128;       // one 64-column half of a 16-row tile (Q, P^T)
constexpr int kSmall = 2 * kSmallHalf;
constexpr int kSeqMaxD = 1024;             // sequences per launch (the host splits larger batches)
constexpr int kMaxCtasD = 296;             // upper bound of the persistent grid
constexpr int kOffKd = 0;
constexpr int kOffVd = kOffKd + kRingK * kTile;
constexpr int kOffQd = kOffVd + kRingV * kTile;
constexpr int kOffPd = kOffQd + 2 * kSmall;                      // Q [2 buffers], then P^T [2 buffers]
constexpr int kOffPre = kOffPd + 2 * kSmall;                     // long long [kSeqMaxD + 1]
constexpr int kOffLen = kOffPre + 8 * (kSeqMaxD + 1);            // int [kSeqMaxD]
constexpr int kOffRange = kOffLen + 4 * kSeqMaxD;                // long long [kMaxCtasD + 1]
constexpr int kSmemD = kOffRange + 8 * (kMaxCtasD + 1) + 1024;
constexpr int kTmemColsD = 64;
constexpr int kColSd = 0;                  // S^T[buf]: 16 fp32 columns each
constexpr int kColOd = 32;                 // O^T: 16 fp32 columns
constexpr uint32_t kWaitLimitD = 1u << 20;
constexpr float kRescaleD = 8.0f;          // log2 units
constexpr int kSlotFloats = kG * kDD + 2 * kG;   // O^T as [16 heads][128 d], then m[16], l[16]

// Work units of the split (attn_work.cuh): the token's own K/V tile is a full softmax
// step but a 256-byte load, and a piece boundary costs little more than a tile: Q is a
// 4 KB copy behind the K ring, and the epilogue of 16 heads x 128 d overlaps the next
// piece's loads.
struct DecCosts {
    static constexpr int tile = 8, block = 6, seg = 8, split = 80, min_group = 64;
};

struct DecParams {
    const int32_t *page_table;
    const int32_t *ctx_len;
    int num_pages, max_pages;
    uint16_t *out;             // [B, 1, Hq, D]
    float *lse;                // [B, Hq, 1] or null
    int B, Hq, Hkv, n_groups;
    float scale_log2;
    unsigned *tickets;         // [segment]
    float *part;               // slots of kSlotFloats
    uint32_t *dev_err;
};

struct DBars {
    uint64_t q_full[2], q_empty[2];   // [piece parity]
    uint64_t k_full[kRingK], k_empty[kRingK], v_full[kRingV], v_empty[kRingV];
    uint64_t s_full[2], s_empty[2];   // [tile parity]
    uint64_t p_full[2], p_free[2];    // [tile parity]
    uint64_t o_full, o_empty;
    uint64_t grp;                     // the four softmax warps among themselves
    uint64_t done[2];                 // each issuer's last MMA has completed
};

struct alignas(16) DShared {
    DBars bar;
    alignas(16) float red[2][kG][4];  // [meeting parity][head][warp]: read as float4
    uint32_t tmem_base;
    int abort;
    int last;
    int max_len;
};

__device__ __forceinline__ bool dwait(DShared &sh, uint64_t *bar, uint32_t parity, uint32_t *dev_err) {
    if (*(volatile int *)&sh.abort) return false;
    if (mbar_wait(bar, parity, kWaitLimitD)) return true;
    *(volatile int *)&sh.abort = 1;
    report_error(dev_err, TT_ERR_DEVICE_TIMEOUT);
    return false;
}

// The four softmax warps meet (k-th meeting); false if one never came.  Values exchanged
// through red[k & 1] are written before meeting k and read right after it, so a warp that
// runs ahead writes the other buffer, and can only come back to this one after meeting
// k + 1, which every warp reaches after its reads.
__device__ __forceinline__ bool dgroup_sync(DShared &sh, int &k, uint32_t *dev_err) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.bar.grp);
    const bool ok = dwait(sh, &sh.bar.grp, (uint32_t)k & 1, dev_err);
    ++k;
    return ok;
}

// Order-preserving map of fp32 onto int32 (for the integer max reduction), and back.
__device__ __forceinline__ int fkey(float x) {
    const int i = __float_as_int(x);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float keyf(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

__device__ __forceinline__ uint16_t to_bf16(float x) {
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return h;
}

// a[i] for a register array and a runtime index (no local-memory copy of the array).
__device__ __forceinline__ float pick(const float (&a)[kG], int i) {
    float v = a[0];
#pragma unroll
    for (int k = 1; k < kG; ++k) v = (i == k) ? a[k] : v;
    return v;
}

__global__ void __launch_bounds__(256, 1)
attn_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_kb, const __grid_constant__ CUtensorMap tm_vb,
                   const __grid_constant__ CUtensorMap tm_q, const DecParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ DShared sh;
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = blockIdx.x;
    DBars &bar = sh.bar;
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) { mbar_init(&bar.q_full[s], 1); mbar_init(&bar.q_empty[s], 1); }
        for (int s = 0; s < kRingK; ++s) { mbar_init(&bar.k_full[s], 1); mbar_init(&bar.k_empty[s], 1); }
        for (int s = 0; s < kRingV; ++s) { mbar_init(&bar.v_full[s], 1); mbar_init(&bar.v_empty[s], 1); }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar.s_full[s], 1); mbar_init(&bar.s_empty[s], 4);
            mbar_init(&bar.p_full[s], 4); mbar_init(&bar.p_free[s], 1);
        }
        mbar_init(&bar.o_full, 1);
        mbar_init(&bar.o_empty, 4);
        mbar_init(&bar.grp, 4);
        mbar_init(&bar.done[0], 1);
        mbar_init(&bar.done[1], 1);
        fence_mbar_init();
        sh.abort = 0;
        prefetch_tmap(&tm_k); prefetch_tmap(&tm_v); prefetch_tmap(&tm_kb); prefetch_tmap(&tm_vb);
        prefetch_tmap(&tm_q);
    }
    // the sequence table: clamped lengths, then the prefix sums of the sequences' work units
    long long *seq_pre = reinterpret_cast<long long *>(sm + kOffPre);
    int *seq_len = reinterpret_cast<int *>(sm + kOffLen);
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        int L = p.ctx_len[i];
        if (L < 0 || L > p.max_pages * kPage) {
            report_error(p.dev_err, TT_ERR_BOUNDS);
            L = 0;
        }
        seq_len[i] = L;
    }
    if (warp == 1) { tmem_alloc(&sh.tmem_base, kTmemColsD); tmem_relinquish(); }
    __syncthreads();
    if (warp == 2) {
        long long carry = 0;
        int mlen = 0;
        if (lane == 0) seq_pre[0] = 0;
        for (int base = 0; base < p.B; base += 32) {
            const int i = base + lane;
            long long v = (i < p.B) ? (long long)seq_cost<DecCosts>(seq_len[i], p.Hkv) : 0;
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
    WorkIter<DecCosts> it;
    it.init(p, group, seq_pre, seq_len, sh.max_len);

    if (warp == 0 || warp == 6) {
        // ================================================================ TMA producers
        // Warp 0 loads K (and each piece's 16 query rows), warp 6 loads V, so that a K copy
        // never waits behind the release of a V stage (V is held until its PV product has
        // completed, K only until QK has read it).  Each whole warp walks the work (page
        // ids are fetched 32 at a time, one per lane); lane 0 issues the copies: the two
        // pages of a context tile, or the token's own key / value for the block tile.
        const bool is_v = warp == 6;
        const int nst = is_v ? kRingV : kRingK;
        uint64_t *full = is_v ? bar.v_full : bar.k_full;
        uint64_t *empty = is_v ? bar.v_empty : bar.k_empty;
        const CUtensorMap *pool = is_v ? &tm_v : &tm_k;
        const CUtensorMap *blk = is_v ? &tm_vb : &tm_kb;
        unsigned char *ring = sm + (is_v ? kOffVd : kOffKd);
        const uint64_t pol = policy_evict_first();
        // Page ids are loaded one batch (16 tiles, one page per lane) ahead of their use --
        // the next batch of the piece, or the first of the next piece, which a second
        // iterator running one piece ahead names -- so that no copy waits on a page-table
        // load.
        WorkIter<DecCosts> ahead = it;
        Piece pc, pn;
        bool have = ahead.next(p, pc);
        bool have_n = have && ahead.next(p, pn);
        int cur = have ? page_id(p, pc, 2 * pc.first + lane) : 0, nxt = 0;
        int t = 0, qi = 0;
        bool ok = true;
        while (ok && have) {
            if (!is_v) {
                // Q of the piece into its buffer (two buffers: the next piece's Q does not
                // wait for the last QK product of this one)
                const int qb = qi & 1;
                if (!dwait(sh, &bar.q_empty[qb], (((uint32_t)qi >> 1) & 1) ^ 1, p.dev_err)) break;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bar.q_full[qb], kSmall);
                    const int row = pc.b * p.Hq + pc.g * kG;
                    tma_load_3d(sm + kOffQd + qb * kSmall, &tm_q, &bar.q_full[qb], 0, row, 0);
                    tma_load_3d(sm + kOffQd + qb * kSmall + kSmallHalf, &tm_q, &bar.q_full[qb], 64, row, 0);
                }
                ++qi;
            }
            for (int i = pc.first; i < pc.last; ++i, ++t) {
                const int rel = i - pc.first;
                if ((rel & 15) == 0) {
                    if (rel > 0) cur = nxt;
                    if (i + 16 < pc.last) nxt = page_id(p, pc, 2 * (i + 16) + lane);
                    else if (have_n) nxt = page_id(p, pn, 2 * pn.first + lane);
                }
                const int page0 = __shfl_sync(0xffffffffu, cur, (2 * rel) & 31);
                const int page1 = __shfl_sync(0xffffffffu, cur, (2 * rel + 1) & 31);
                const bool ctx = i < pc.ntc;
                const bool two = ctx && tile_valid(pc, i, 1) > kPage;
                const int st = t % nst;
                if (!dwait(sh, &empty[st], ((uint32_t)(t / nst) & 1) ^ 1, p.dev_err)) { ok = false; break; }
                unsigned char *dst = ring + st * kTile;
                if (lane == 0) {
                    if (ctx) {
                        // the pages are read once per launch: first out of L2
                        mbar_arrive_expect_tx(&full[st], two ? 4 * 8192u : 2 * 8192u);
                        tma_load_4d_hint(dst, pool, &full[st], 0, 0, pc.g, page0, pol);
                        tma_load_4d_hint(dst + kTileHalf, pool, &full[st], 64, 0, pc.g, page0, pol);
                        if (two) {
                            tma_load_4d_hint(dst + 8192, pool, &full[st], 0, 0, pc.g, page1, pol);
                            tma_load_4d_hint(dst + kTileHalf + 8192, pool, &full[st], 64, 0, pc.g, page1, pol);
                        }
                    } else {
                        mbar_arrive_expect_tx(&full[st], 2 * 128u);
                        tma_load_3d(dst, blk, &full[st], 0, pc.g, pc.b);
                        tma_load_3d(dst + kTileHalf, blk, &full[st], 64, pc.g, pc.b);
                    }
                }
                __syncwarp();
            }
            // the last batch of a piece always prefetched the first batch of the next one
            cur = nxt;
            pc = pn;
            have = have_n;
            have_n = have && ahead.next(p, pn);
        }
        // Drain: every copy issued must land before the CTA may exit.  The last copy into a
        // stage completes that stage's latest phase.
        for (int k = 1; k <= nst && t - k >= 0; ++k)
            mbar_wait(&full[(t - k) % nst], (uint32_t)((t - k) / nst) & 1, kWaitLimitD);
        __syncwarp();
    } else if (warp == 1 || warp == 7) {
        // ================================================================ MMA issuers
        // Warp 1 issues the QK products, warp 7 the PV products.  A commit tracks the MMAs
        // of the thread that issued them, so a V stage (and the P^T buffer) is released as
        // soon as its own PV product has completed, whatever QK products are queued.
        const uint32_t idesc_qk = idesc_bf16_f32(128, kG, false, false);
        const uint32_t idesc_pv = idesc_bf16_f32(128, kG, true, false);
        Piece pc;
        int t0 = 0, qi = 0, pi = 0;
        bool ok = true;
        // S^T[tt & 1] = K_tile . Q^T for tile tt, with the piece's Q in buffer qbuf
        auto issue_qk = [&](int tt, int qbuf, bool last) -> bool {
            const int st = tt % kRingK;
            if (!dwait(sh, &bar.k_full[st], (uint32_t)(tt / kRingK) & 1, p.dev_err)) return false;
            if (!dwait(sh, &bar.s_empty[tt & 1], (((uint32_t)tt >> 1) & 1) ^ 1, p.dev_err)) return false;
            tc_fence_after();
            const uint32_t kbase = smem_u32(sm + kOffKd + st * kTile);
            const uint32_t qb = smem_u32(sm + kOffQd + qbuf * kSmall);
            const uint32_t dcol = tmem + kColSd + 16 * (tt & 1);
            if (elect_one()) {   // one lane issues the tile's MMAs and their commits
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {   // 16 head dimensions per step
                    const uint64_t da = sdesc_sw128(kbase + (kk >> 2) * (uint32_t)kTileHalf + (kk & 3) * 32, 16, 1024);
                    const uint64_t db = sdesc_sw128(qb + (kk >> 2) * (uint32_t)kSmallHalf + (kk & 3) * 32, 16, 1024);
                    mma_bf16_ss(dcol, da, db, idesc_qk, kk > 0);
                }
                mma_commit(&bar.s_full[tt & 1]);
                mma_commit(&bar.k_empty[st]);
                if (last) mma_commit(&bar.q_empty[qbuf]);
            }
            __syncwarp();
            return true;
        };
        // O^T += V_tile^T . P^T for tile tt (j-th of its piece); rows of the V tile past the
        // valid keys are zeroed first (their P is 0, but stale bits could hold a NaN)
        auto issue_pv = [&](int tt, int j, int valid, bool last) -> bool {
            const int st = tt % kRingV;
            const int nk = (valid + 15) & ~15;
            if (!dwait(sh, &bar.v_full[st], (uint32_t)(tt / kRingV) & 1, p.dev_err)) return false;
            unsigned char *vp = sm + kOffVd + st * kTile;
            if (valid < nk) {
                const int words = (nk - valid) * 8;   // 16-byte words per half
                for (int w = lane; w < 2 * words; w += 32) {
                    const int h = w / words, r = valid + (w % words) / 8, c = w % 8;
                    *reinterpret_cast<uint4 *>(vp + h * kTileHalf + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (!dwait(sh, &bar.p_full[tt & 1], ((uint32_t)tt >> 1) & 1, p.dev_err)) return false;
            if (j == 0 && !dwait(sh, &bar.o_empty, ((uint32_t)pi & 1) ^ 1, p.dev_err)) return false;
            tc_fence_after();
            const uint32_t vbase = smem_u32(vp);
            const uint32_t pb = smem_u32(sm + kOffPd + (tt & 1) * kSmall);
            if (elect_one()) {   // one lane issues the tile's MMAs and their commits
                for (int kk = 0; kk < nk / 16; ++kk) {   // 16 keys per step
                    const uint64_t da = sdesc_sw128(vbase + kk * 2048, kTileHalf, 1024);
                    const uint64_t db = sdesc_sw128(pb + (kk >> 2) * (uint32_t)kSmallHalf + (kk & 3) * 32, 16, 1024);
                    mma_bf16_ss(tmem + kColOd, da, db, idesc_pv, !(j == 0 && kk == 0));
                }
                mma_commit(&bar.p_free[tt & 1]);
                mma_commit(&bar.v_empty[st]);
                if (last) mma_commit(&bar.o_full);
            }
            __syncwarp();
            return true;
        };
        while (ok && it.next(p, pc)) {
            const int ntiles = pc.last - pc.first;
            if (warp == 1) {
                const int qbuf = qi & 1;
                if (!dwait(sh, &bar.q_full[qbuf], ((uint32_t)qi >> 1) & 1, p.dev_err)) break;
                ++qi;
                for (int j = 0; ok && j < ntiles; ++j) ok = issue_qk(t0 + j, qbuf, j + 1 == ntiles);
            } else {
                for (int j = 0; ok && j < ntiles; ++j)
                    ok = issue_pv(t0 + j, j, tile_valid(pc, pc.first + j, 1), j + 1 == ntiles);
            }
            t0 += ntiles;
            ++pi;
        }
        if (elect_one()) mma_commit(&bar.done[warp == 1 ? 0 : 1]);
        __syncwarp();
    } else {
        // ================================================================ softmax / epilogue
        // Thread r (TMEM lane r) owns key r of every tile and, at the end of a piece, d lane
        // r of O^T.  Warp w reads the TMEM lane quarter w % 4.
        const int wq = warp & 3;
        const int r = 32 * wq + lane;
        const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
        const float c2 = p.scale_log2;
        const int pt_half = r >> 6, pt_chunk = (r & 63) >> 3, pt_within = (r & 7) * 2;
        // Merge every piece of a split segment in group order (d lane r of each head) and
        // leave its ticket at zero for the next launch.
        // lo[c] of every group (for the merges), filled while the first tiles load
        long long *range_tab = reinterpret_cast<long long *>(sm + kOffRange);
        for (int c = r; c <= it.NG; c += 128) range_tab[c] = range_lo(c, it.U, it.NG);
        auto merge = [&](const Piece &q) {
            const int n = it.NG;
            const int c_first = owner_tab(q.X + DecCosts::seg, range_tab, n);
            const int c_last = owner_tab(q.X + DecCosts::seg + (long long)DecCosts::tile * q.ntc, range_tab, n);
            float M[kG], Ls[kG], acc[kG];
#pragma unroll
            for (int h = 0; h < kG; ++h) { M[h] = -INFINITY; Ls[h] = 0.f; acc[h] = 0.f; }
            // up to four pieces per round, every load of a round in flight at once: lane L
            // loads the maximum (L < 16) or the sum (L >= 16) of head L % 16, and every thread
            // its d lane of the 16 heads
            for (int c0 = c_first; c0 <= c_last; c0 += 4) {
                bool u[4];
                float ml[4], o[4][kG];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    u[k] = c0 + k <= c_last && owns_tile_tab<DecCosts>(c0 + k, q.X, q.ntc, range_tab);
                    const float *sl = p.part + (long long)(c0 + k + q.sg) * kSlotFloats;
                    ml[k] = u[k] ? __ldcg(sl + kG * kDD + lane) : (lane < kG ? -INFINITY : 0.f);
#pragma unroll
                    for (int h = 0; h < kG; ++h) o[k][h] = u[k] ? __ldcg(sl + h * kDD + r) : 0.f;
                }
#pragma unroll
                for (int h = 0; h < kG; ++h) {
                    float mk[4], lk[4];
                    float Mn = M[h];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        mk[k] = __shfl_sync(0xffffffffu, ml[k], h);
                        lk[k] = __shfl_sync(0xffffffffu, ml[k], kG + h);
                        Mn = fmaxf(Mn, mk[k]);
                    }
                    if (Mn == -INFINITY) continue;   // no piece yet for this head
                    const float a = fast_exp2(M[h] - Mn);
                    float ls = Ls[h] * a, ac = acc[h] * a;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float w = fast_exp2(mk[k] - Mn);
                        ls += lk[k] * w;
                        ac += o[k][h] * w;
                    }
                    Ls[h] = ls;
                    acc[h] = ac;
                    M[h] = Mn;
                }
            }
            const int hq0 = q.g * kG;
            uint16_t *out = p.out + ((size_t)q.b * p.Hq + hq0) * kDD + r;
#pragma unroll
            for (int h = 0; h < kG; ++h) out[h * kDD] = to_bf16(acc[h] / Ls[h]);
            if (p.lse && r < kG)
                p.lse[(size_t)q.b * p.Hq + hq0 + r] = (pick(M, r) + __log2f(pick(Ls, r))) * kLn2;
            if (r == 0) p.tickets[q.sg] = 0;
        };
        Piece pc, pend0, pend1;           // the split pieces of this CTA (at most two)
        int npend = 0, last0 = 0, last1 = 0;  // (last*: thread r == 0 only)
        int t = 0, pi = 0, k_grp = 0;
        bool ok = true;
        while (ok && it.next(p, pc)) {
            float m[kG], l[kG];
#pragma unroll
            for (int h = 0; h < kG; ++h) { m[h] = -INFINITY; l[h] = 0.f; }
            const int ntiles = pc.last - pc.first;
            for (int j = 0; j < ntiles; ++j, ++t) {
                const int sb = t & 1;
                const int valid = tile_valid(pc, pc.first + j, 1);
                if (!dwait(sh, &bar.s_full[sb], ((uint32_t)t >> 1) & 1, p.dev_err)) { ok = false; break; }
                tc_fence_after();
                uint32_t sv[16];
                tmem_ld16(tmem + lane_off + kColSd + 16 * sb, sv);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.s_empty[sb]);
                float x[kG];
#pragma unroll
                for (int h = 0; h < kG; ++h) x[h] = (r < valid) ? __uint_as_float(sv[h]) * c2 : -INFINITY;
                // each head's maximum over the tile: within the warp, then across the four warps
                float (*red)[4] = sh.red[k_grp & 1];
#pragma unroll
                for (int h = 0; h < kG; ++h) {
                    const int mk = __reduce_max_sync(0xffffffffu, fkey(x[h]));
                    if (lane == h) red[h][wq] = keyf(mk);
                }
                if (!dgroup_sync(sh, k_grp, p.dev_err)) { ok = false; break; }
                float mn[kG];
                bool moved = false;
#pragma unroll
                for (int h = 0; h < kG; ++h) {
                    const float4 v = *reinterpret_cast<const float4 *>(&red[h][0]);
                    const float tm = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
                    mn[h] = (tm > m[h] + kRescaleD) ? tm : m[h];
                    moved |= (j > 0 && mn[h] != m[h]);
                }
                if (moved) {
                    // (the same in every thread) a head's maximum rose: once the PV product of
                    // the previous tile has completed, rescale its O^T column (this thread's d
                    // lane) and its sums
                    if (!dwait(sh, &bar.p_free[sb ^ 1], ((uint32_t)(t - 1) >> 1) & 1, p.dev_err)) { ok = false; break; }
                    tc_fence_after();
                    uint32_t o[16];
                    tmem_ld16(tmem + lane_off + kColOd, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < kG; ++h) {
                        const float a = (mn[h] != m[h]) ? fast_exp2(m[h] - mn[h]) : 1.f;
                        o[h] = __float_as_uint(__uint_as_float(o[h]) * a);
                        l[h] *= a;
                    }
                    tmem_st16(tmem + lane_off + kColOd, o);
                    tmem_wait_st();
                }
#pragma unroll
                for (int h = 0; h < kG; ++h) m[h] = mn[h];
                // P^T buffer sb is free once the PV product of tile t-2 has completed
                if (!dwait(sh, &bar.p_free[sb], (((uint32_t)t >> 1) & 1) ^ 1, p.dev_err)) { ok = false; break; }
                // P = 2^(x - m) into P^T[h][r]: K-major with 128-byte swizzle, so the 16-byte
                // chunk of key r in row h sits at chunk ((r % 64) / 8) XOR (h % 8)
                unsigned char *pt = sm + kOffPd + sb * kSmall + pt_half * kSmallHalf + pt_within;
#pragma unroll
                for (int h = 0; h < kG; ++h) {
                    const float pv = (r < valid) ? fast_exp2(x[h] - m[h]) : 0.f;
                    l[h] += pv;
                    *reinterpret_cast<uint16_t *>(pt + h * 128 + ((pt_chunk ^ (h & 7)) << 4)) = to_bf16(pv);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar.p_full[sb]);
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue of the piece
            // each head's sum over the 128 keys: within the warp, then across the four warps
            {
                float (*red)[4] = sh.red[k_grp & 1];
#pragma unroll
                for (int h = 0; h < kG; ++h) {
                    float v = l[h];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane == h) red[h][wq] = v;
                }
                if (!dgroup_sync(sh, k_grp, p.dev_err)) { ok = false; break; }
#pragma unroll
                for (int h = 0; h < kG; ++h) {
                    const float4 v = *reinterpret_cast<const float4 *>(&red[h][0]);
                    l[h] = (v.x + v.y) + (v.z + v.w);
                }
            }
            if (!dwait(sh, &bar.o_full, (uint32_t)pi & 1, p.dev_err)) { ok = false; break; }
            tc_fence_after();
            uint32_t o[16];
            tmem_ld16(tmem + lane_off + kColOd, o);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar.o_empty);
            const int hq0 = pc.g * kG;
            uint16_t *out = p.out + ((size_t)pc.b * p.Hq + hq0) * kDD + r;
            if (pc.whole) {
#pragma unroll
                for (int h = 0; h < kG; ++h) out[h * kDD] = to_bf16(__uint_as_float(o[h]) / l[h]);
                if (p.lse && r < kG)
                    p.lse[(size_t)pc.b * p.Hq + hq0 + r] = (pick(m, r) + __log2f(pick(l, r))) * kLn2;
            } else {
                // partial: unnormalised O^T, the maxima (log2 units) and the sums
                float *slot = p.part + (long long)(group + pc.sg) * kSlotFloats;
#pragma unroll
                for (int h = 0; h < kG; ++h) __stcg(slot + h * kDD + r, __uint_as_float(o[h]));
                if (r < kG) {
                    __stcg(slot + kG * kDD + r, pick(m, r));
                    __stcg(slot + kG * kDD + kG + r, pick(l, r));
                }
                // One thread publishes the piece: the meeting orders every thread's stores
                // before its release.  The add returns at once (release only), so the
                // pipeline does not wait for it; whether this piece completed the segment is
                // read at the end, where the last one acquires (fence) and merges -- after
                // this CTA's own tiles (at most two split pieces: only the first and the last
                // piece of a CTA's range can be split).
                if (!dgroup_sync(sh, k_grp, p.dev_err)) { ok = false; break; }
                if (r == 0) {
                    const unsigned n_here = (unsigned)(pc.last - pc.first);
                    const unsigned before = atom_add_release_gpu(p.tickets + pc.sg, n_here);
                    const int done = (before + n_here == (unsigned)(pc.ntc + 1)) ? 1 : 0;
                    if (npend == 0) last0 = done; else last1 = done;
                }
                if (npend == 0) pend0 = pc; else pend1 = pc;
                ++npend;
            }
            ++pi;
        }
        if (ok && npend > 0) {
            if (r == 0) {
                if (last0 | last1) fence_acq_rel_gpu();
                sh.last = last0 | (last1 << 1);
            }
            if (dgroup_sync(sh, k_grp, p.dev_err)) {
                const int f = sh.last;
                if (f & 1) merge(pend0);
                if (npend > 1 && (f & 2)) merge(pend1);
            }
        }
    }

    // ------------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        mbar_wait(&bar.done[0], 0, kWaitLimitD);
        mbar_wait(&bar.done[1], 0, kWaitLimitD);
        tmem_dealloc(tmem, kTmemColsD);
    }
}

}  // namespace

bool attn_decode_supported(int S, int Hq, int Hkv, int D, int page_size, tt_dtype dtype) {
    return dtype == TT_BF16 && S == 1 && D == kDD && page_size == kPage && Hkv >= 1 && Hq == kG * Hkv;
}

size_t attn_decode_ws_bytes(int B, int Hkv) {
    const size_t nseg = (size_t)(B < kSeqMaxD ? B : kSeqMaxD) * Hkv;   // one launch's segments
    return align_up(nseg * sizeof(unsigned), 256) + (kMaxCtasD + nseg) * kSlotFloats * sizeof(float);
}

// Batches above the kernel's sequence table run as consecutive launches on the stream;
// they share the workspace, which each launch leaves as it found it (tickets zero).
tt_status launch_attn_decode(const AttnArgs &a) {
    const tt_kv_cache &c = *a.ctx;
    if (c.num_pages < 1) return launch_attn_simt(a);   // no pool to map: nothing paged to read
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TT_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TT_ERR_CUDA;
    CUtensorMap mk, mv;
    if (!make_pool_maps(c, a.Hkv, &mk, &mv)) return TT_ERR_CUDA;
    if (cudaFuncSetAttribute(attn_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemD) !=
        cudaSuccess)
        return TT_ERR_CUDA;
    for (int b0 = 0; b0 < a.B; b0 += kSeqMaxD) {
        const int nb = a.B - b0 < kSeqMaxD ? a.B - b0 : kSeqMaxD;
        const uint16_t *q = static_cast<const uint16_t *>(a.q) + (size_t)b0 * a.Hq * kDD;
        const uint16_t *k_blk = static_cast<const uint16_t *>(a.k_blk) + (size_t)b0 * a.Hkv * kDD;
        const uint16_t *v_blk = static_cast<const uint16_t *>(a.v_blk) + (size_t)b0 * a.Hkv * kDD;
        CUtensorMap mkb, mvb, mq;
        {
            // the token's own keys and values, [nb][Hkv][D]
            const uint64_t dims[3] = {(uint64_t)kDD, (uint64_t)a.Hkv, (uint64_t)nb};
            const uint64_t str[2] = {(uint64_t)kDD * 2, (uint64_t)a.Hkv * kDD * 2};
            const uint32_t box[3] = {64, 1, 1};
            if (!make_map(&mkb, k_blk, 3, dims, str, box)) return TT_ERR_CUDA;
            if (!make_map(&mvb, v_blk, 3, dims, str, box)) return TT_ERR_CUDA;
        }
        {
            // the queries as [nb * Hq rows][D]; a box is the 16 rows of one KV head, 64 columns
            const uint64_t dims[3] = {(uint64_t)kDD, (uint64_t)nb * a.Hq, 1};
            const uint64_t str[2] = {(uint64_t)kDD * 2, (uint64_t)nb * a.Hq * kDD * 2};
            const uint32_t box[3] = {64, (uint32_t)kG, 1};
            if (!make_map(&mq, q, 3, dims, str, box)) return TT_ERR_CUDA;
        }
        DecParams p;
        p.page_table = c.page_table + (size_t)b0 * c.max_pages_per_seq;
        p.ctx_len = c.ctx_len + b0;
        p.num_pages = c.num_pages;
        p.max_pages = c.max_pages_per_seq;
        p.out = static_cast<uint16_t *>(a.out) + (size_t)b0 * a.Hq * kDD;
        p.lse = a.lse ? a.lse + (size_t)b0 * a.Hq : nullptr;
        p.B = nb; p.Hq = a.Hq; p.Hkv = a.Hkv;
        int n = a.max_ctas > 0 ? a.max_ctas : sms;
        if (n > kMaxCtasD) n = kMaxCtasD;
        p.n_groups = n;
        p.scale_log2 = a.sm_scale * kLog2e;
        const size_t nseg = (size_t)nb * a.Hkv;
        p.tickets = static_cast<unsigned *>(a.ws);
        p.part = reinterpret_cast<float *>(static_cast<char *>(a.ws) + align_up(nseg * sizeof(unsigned), 256));
        p.dev_err = a.dev_err;
        attn_decode_kernel<<<n, 256, kSmemD, a.stream>>>(mk, mv, mkb, mvb, mq, p);
        if (cudaGetLastError() != cudaSuccess) return TT_ERR_CUDA;
    }
    return TT_OK;
}

}  // namespace tt
