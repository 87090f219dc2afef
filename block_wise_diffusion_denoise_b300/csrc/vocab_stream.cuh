// One streaming pass over the vocabulary logits of the masked block positions:
// for every masked row, its maximum m, the sum Z of exp(l - m) and the lowest index
// holding m.  Two steps of the method are built on it: the confidence unmasking of a
// denoise step (conf = 1/Z, token = argmax; TwoTower summary on gist.science,
// "Training und Konditionierung -- Sampling") and the masked-diffusion loss of
// training (NLL = m + log Z - l_target; same page, "Maskierte Diffusion").  Each
// supplies a Finish policy that turns a sequence's rows into its outputs.
//
// Design (HBM-bound; every masked logit is read once):
//  * Work.  A row of V logits is cut into units of 64 KB; up to kUnitsPerBlock
//    consecutive units of one row form a block, the grain of the partial results.
//    The blocks of masked rows are ranked in row order (from a copy of the flags in
//    shared memory); CTA c takes rank c, then one rank after another from a counter in
//    the workspace, so the CTAs that the memory system serves faster take more blocks
//    and all of them run dry together (a static share left the last CTAs about 4 us
//    behind the first).  Batches too large for the copy of the flags keep a static
//    share: CTA c takes blocks c, c + grid, ...  The grid walks the blocks in row order
//    together, so sequences complete one after another during the launch and their
//    finishing work overlaps the streaming of later ones.
//  * Pipeline.  One producer warp moves units into a CTA-wide ring of kStages
//    shared-memory stages with plain bulk copies (cp.async.bulk, completion as
//    transaction bytes on the stage's mbarrier); sixteen consumer warps share every
//    stage (each thread takes eight 16-byte vectors), so the warps of a CTA move in
//    step.  A stage is given back as soon as all sixteen warps have loaded it into
//    registers, before any arithmetic, so that the next copy into it starts early.  The
//    bulk copies carry an L2 evict-first policy: every logit is read once.
//  * Arithmetic.  Per thread, in two passes over the unit's vectors in registers: the
//    maximum (one value per vector by packed bf16 maxima, exact, then three-input fp32
//    maxima), the first index holding it (only when it rises), then sum
//    2^(x*log2e - mc) over eight scalar accumulators, two values per paired FMA and
//    paired add, with mc = m*log2e rounded to fp32.  Every term then
//    carries the same factor 2^delta, delta = m*log2e - mc, which one FMA gives exactly
//    and one exponential removes at the end of the block (below 2^-3 in magnitude while
//    |m| < 2^20; for larger logits the terms take the difference first, (x - m)*log2e,
//    and delta = 0).  Without that correction the confidence 1/Z would be off by a
//    relative 1e-6 at m = 40, and without bound for huge logits.  A rise of the maximum
//    rescales the sums by one exponential.  At the end of a block each warp reduces its
//    32 states (integer max reduction, one rescale per lane, a fixed butterfly sum, a
//    min reduction for the index) and hands the result to the publisher.
//  * Completion.  A consumer warp hands its state at the end of a block to a publisher
//    warp through a small ring in shared memory and moves on; the publisher merges the
//    sixteen states of a block, writes its partial and adds one to the sequence's ticket
//    (acquire-release; a batch of blocks from its lanes at once).  While the copies
//    stream, a publisher's batch (merge, release, add) takes several microseconds,
//    longer than the consumers take for a block, so two publisher warps take alternate
//    ring entries and their round trips overlap.  The add that brings the
//    ticket to (masked rows of the sequence) x (blocks per row) runs the Finish policy for
//    that sequence, which merges each masked row's partials in block order -- so the
//    result does not depend on which CTA processed which block -- and resets the ticket.
//    Sequences with no masked row are finished at the start.  A sequence's `masked`
//    entries are read only before its own Finish, the one place that may change them.
//  * A waiting warp polls its mbarrier with short naps in between (__nanosleep), so it
//    takes few issue slots from the arithmetic yet wakes within a fraction of a
//    microsecond.  Every wait is bounded (1 s of wall time); a wait that gives up records
//    TT_ERR_DEVICE_TIMEOUT and the CTA stops.  After such an error the workspace
//    must be cleared before the next call.
#pragma once

#include <climits>
#include <cstdint>

#include "sm100_ptx.cuh"
#include "tt_common.cuh"
#include "tt_internal.h"

namespace tt {
namespace vs {

constexpr int kConsumerWarps = 16;                  // four per SM sub-partition
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kProducerWarp = kConsumerWarps;       // moves the data
constexpr int kPublisherWarp = kConsumerWarps + 1;  // the first of the warps that publish finished blocks
constexpr int kPublishers = 2;                      // publisher p takes ring entries p, p + 2, ...
constexpr int kThreads = kConsumers + 32 + 32 * kPublishers;
constexpr int kRed = 16;                            // finished blocks awaiting the publishers
static_assert(kRed % kPublishers == 0, "each ring slot belongs to one publisher");
constexpr int kUnitBytes = 65536;
constexpr int kVecPerThread = kUnitBytes / 16 / kConsumers;   // 8
constexpr int kStages = 3;
constexpr int kUnitsPerBlock = 2;
constexpr int kMaskSnap = 16384;                    // masked flags copied to shared memory (B*S <= this)
constexpr int kSmemBytes = kStages * kUnitBytes + kMaskSnap;   // dynamic: the ring, then the flags
constexpr uint32_t kWaitLimit = 1u << 22;           // polls of a single-thread drain wait
constexpr uint64_t kWaitNs = 1000000000ull;         // a warp wait gives up after 1 s

// Arguments every pass shares (the Finish policy brings its own).
struct Common {
    const void *logits;        // [B, S, V]
    int B, S, V;
    int nc;                    // units per row
    int bpr;                   // blocks per row
    long long nblocks;         // B * S * bpr
    const uint8_t *masked;     // [B, S]: rows to read (read before a sequence's Finish runs)
    UnmaskPartial *part;       // [nblocks]
    unsigned *tickets;         // [B]: blocks done per sequence
    uint32_t *dev_err;
};

template <typename T> struct Elem;
template <> struct Elem<uint16_t> { static constexpr int kPerVec = 8; };
template <> struct Elem<float> { static constexpr int kPerVec = 4; };

// Merge two (max, sum of exp(x - max), first argmax) triples; the sums are exact (no
// pending factor).  The lower index wins a tie of the maxima.
__device__ __forceinline__ void merge_state(float &m, float &z, int &a, float m2, float z2, int a2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; z = z2; a = a2; return; }
    // the sum under the larger maximum keeps its scale; one exponential rescales the other
    if (m >= m2) {
        z = fmaf(z2, fast_exp2((m2 - m) * kLog2e), z);
        if (m2 == m) a = min(a, a2);
    } else {
        z = fmaf(z, fast_exp2((m - m2) * kLog2e), z2);
        m = m2;
        a = a2;
    }
}

// Order-preserving map of fp32 onto int32 (for the integer warp-max reduction) and back.
__device__ __forceinline__ int f2key(float x) {
    const int i = __float_as_int(x);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float key2f(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

// Warp-wide (max, exact sum, first argmax) in three steps: the maximum M by one integer
// reduction, every lane's sum rescaled to M (one exponential) and added up by a fixed
// butterfly, and the lowest index among the lanes whose maximum equals M.  Every lane ends
// with the same result, whatever the timing.
__device__ __forceinline__ void warp_reduce_state(float &m, float &z, int &a) {
    const float M = key2f(__reduce_max_sync(0xffffffffu, f2key(m)));
    float zt = (m == -INFINITY) ? 0.f : z * fast_exp2((m - M) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zt += __shfl_xor_sync(0xffffffffu, zt, o);
    const int A = (int)__reduce_min_sync(0xffffffffu, (unsigned)((M != -INFINITY && m == M) ? a : INT_MAX));
    m = M;
    z = zt;
    a = A;
}

// Largest element of a 16-byte vector (bf16: packed pairwise maxima, exact).
template <typename T> __device__ __forceinline__ uint32_t vmax_bits(const uint4 &u);
template <> __device__ __forceinline__ uint32_t vmax_bits<uint16_t>(const uint4 &u) {
    uint32_t a, b, c;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(u.x), "r"(u.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(u.z), "r"(u.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(a), "r"(b));
    return c;
}
template <typename T> __device__ __forceinline__ float vec_max(const uint4 &u);
template <> __device__ __forceinline__ float vec_max<uint16_t>(const uint4 &u) {
    const uint32_t c = vmax_bits<uint16_t>(u);
    return fmaxf(bf16_lo(c), bf16_hi(c));
}
template <> __device__ __forceinline__ float vec_max<float>(const uint4 &u) {
    return fmaxf(fmaxf(__uint_as_float(u.x), __uint_as_float(u.y)),
                 fmaxf(__uint_as_float(u.z), __uint_as_float(u.w)));
}

// Position of the first element equal to mx in the vector (mx is one of its elements).
template <typename T> __device__ __forceinline__ int vec_first(const uint4 &u, float mx);
template <> __device__ __forceinline__ int vec_first<uint16_t>(const uint4 &u, float mx) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    int j0 = 7;
#pragma unroll
    for (int j = 3; j >= 0; --j) {
        j0 = (bf16_hi(w[j]) == mx) ? 2 * j + 1 : j0;
        j0 = (bf16_lo(w[j]) == mx) ? 2 * j : j0;
    }
    return j0;
}
template <> __device__ __forceinline__ int vec_first<float>(const uint4 &u, float mx) {
    return (__uint_as_float(u.x) == mx) ? 0 : (__uint_as_float(u.y) == mx) ? 1 : (__uint_as_float(u.z) == mx) ? 2 : 3;
}

// What the producer tells the consumers about the unit in a stage.
struct StageDesc {
    int blk;        // block index, or -1: no more work
    int elem0;      // index of the unit's first element within its row
    int nvec;       // valid 16-byte vectors in the stage
    int last;       // 1: the last unit of its block
};

struct Shared {
    uint64_t full[kStages], empty[kStages];
    uint64_t red_full[kRed], red_empty[kRed];   // ring of finished blocks: consumers -> publisher
    StageDesc desc[kStages];
    float red_m[kRed][kConsumerWarps], red_z[kRed][kConsumerWarps];
    int red_a[kRed][kConsumerWarps];
    int red_blk[kRed];                           // block id, or -1: no more blocks
    int warp_masked[kThreads / 32];              // masked rows each warp found in the snapshot
    int abort;
};

// Bounded wait by a whole warp; the result is the same in every lane.  A wait that gives up
// raises the CTA's abort flag (every later wait then fails at once) and reports the timeout.
__device__ __forceinline__ bool wait_or_abort(Shared &sh, uint64_t *bar, uint32_t parity, uint32_t *dev_err,
                                              uint32_t nap_ns = 64) {
    if (__any_sync(0xffffffffu, *(volatile int *)&sh.abort != 0)) return false;
    if (sm100::mbar_wait_warp_nap(bar, parity, nap_ns, kWaitNs)) return true;
    if ((threadIdx.x & 31) == 0) {
        *(volatile int *)&sh.abort = 1;
        report_error(dev_err, TT_ERR_DEVICE_TIMEOUT);
    }
    return false;
}

// Merged (max, exact sum, first argmax) of one row from its block partials, in block order.
__device__ __forceinline__ void row_state(const Common &c, long long row, float &m, float &z, int &a) {
    m = -INFINITY; z = 0.f; a = INT_MAX;
    const UnmaskPartial *pp = c.part + row * c.bpr;
    int g = 0;
    for (; g + 4 <= c.bpr; g += 4) {   // four independent loads in flight
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = __ldcg(reinterpret_cast<const float4 *>(pp + g + k));
#pragma unroll
        for (int k = 0; k < 4; ++k) merge_state(m, z, a, v[k].x, v[k].y, __float_as_int(v[k].z));
    }
    if (g < c.bpr) {   // the last one to three, also loaded together (merged in block order)
        float4 v[3];
#pragma unroll
        for (int k = 0; k < 3; ++k)
            if (g + k < c.bpr) v[k] = __ldcg(reinterpret_cast<const float4 *>(pp + g + k));
#pragma unroll
        for (int k = 0; k < 3; ++k)
            if (g + k < c.bpr) merge_state(m, z, a, v[k].x, v[k].y, __float_as_int(v[k].z));
    }
}

// Masked rows of sequence b (read before its Finish, the one place that may change them).
__device__ __forceinline__ int masked_rows(const Common &c, const uint8_t *snap, bool use_snap, int b) {
    int n = 0;
    const uint8_t *mk = use_snap ? snap + (size_t)b * c.S : c.masked + (size_t)b * c.S;
    for (int p = 0; p < c.S; ++p) n += mk[p] != 0;
    return n;
}

// The EPV values of one 16-byte vector as fp32 (bf16: one shift or mask per value, exact).
template <typename T> __device__ __forceinline__ void unpack_vec(const uint4 &u, float *x);
template <> __device__ __forceinline__ void unpack_vec<uint16_t>(const uint4 &u, float *x) {
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}
template <> __device__ __forceinline__ void unpack_vec<float>(const uint4 &u, float *x) {
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y);
    x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
}

// Two fp32 values as one 64-bit operand of the paired instructions, and back.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// acc[j] += 2^(x[j] * log2e - mc) for the EPV values of one vector, two at a time with the
// paired fp32 FMA and add (each lane an ordinary round-to-nearest fma / add: the same
// results as the scalar form, in half the instructions).
template <int EPV>
__device__ __forceinline__ void exps_fma2(const float *x, uint64_t l2, uint64_t nm, float *acc) {
#pragma unroll
    for (int j = 0; j < EPV; j += 2) {
        uint64_t y;
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(y) : "l"(pk2(x[j], x[j + 1])), "l"(l2), "l"(nm));
        float y0, y1;
        upk2(y, y0, y1);
        uint64_t a2 = pk2(acc[j], acc[j + 1]);
        asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a2) : "l"(pk2(fast_exp2(y0), fast_exp2(y1))));
        upk2(a2, acc[j], acc[j + 1]);
    }
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// One unit of a block, by one consumer thread: its vectors are loaded into registers and
// the stage is given back at once; then two passes over the registers:
//  1. the maximum: one value per vector (packed bf16 maxima), then over the vectors; if it
//     rises above the running maximum, the first vector holding it gives the first index,
//     and the sums are rescaled;
//  2. every value is unpacked once into its exponential term.
// kFull: every vector of the unit is valid (no checks).
template <typename T, bool kFull>
__device__ __forceinline__ void consume_unit(const uint4 *pv, const StageDesc &d, int s, Shared &sh, float &m,
                                             float &mc, float &delta, int &a, float (&acc)[8]) {
    constexpr int EPV = Elem<T>::kPerVec;
    constexpr float kFastLimit = 1048576.f;
    const int tid = threadIdx.x, lane = tid & 31;
    uint4 u[kVecPerThread];
    bool okv[kVecPerThread];
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) {
        const int v = tid + kConsumers * q;
        okv[q] = kFull || v < d.nvec;
        u[q] = okv[q] ? pv[v] : make_uint4(0, 0, 0, 0);
    }
    // The unit is in registers: give the stage back before any arithmetic, so that it is
    // held only for the loads and the next copy into it starts as early as possible.
    __syncwarp();
    if (lane == 0) sm100::mbar_arrive(&sh.empty[s]);
    float vm[kVecPerThread];
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) vm[q] = okv[q] ? vec_max<T>(u[q]) : -INFINITY;
    float cm = fmax3(vm[0], vm[1], vm[2]);
#pragma unroll
    for (int q = 3; q + 1 < kVecPerThread; q += 2) cm = fmax3(cm, vm[q], vm[q + 1]);
    if ((kVecPerThread - 3) % 2) cm = fmaxf(cm, vm[kVecPerThread - 1]);
    if (cm > m) {
        // a new maximum: the first vector holding it, its first position there, and the sums
        // moved to it
        int q0 = kVecPerThread - 1;
#pragma unroll
        for (int q = kVecPerThread - 1; q >= 0; --q) q0 = (vm[q] == cm) ? q : q0;
        const int v0 = tid + kConsumers * q0;
        uint4 w = u[0];
#pragma unroll
        for (int q = 1; q < kVecPerThread; ++q) w = (q == q0) ? u[q] : w;
        a = d.elem0 + v0 * EPV + vec_first<T>(w, cm);
        const bool fast = fabsf(cm) < kFastLimit;
        const float mcn = fast ? cm * kLog2e : 0.f;
        const float dn = fast ? fmaf(cm, kLog2e, -mcn) : 0.f;
        if (m != -INFINITY) {
            // sums times 2^delta_old relative to m, to times 2^delta_new relative to cm
            const float r = fast_exp2(fmaf(m - cm, kLog2e, dn - delta));
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] *= r;
        }
        m = cm;
        mc = mcn;
        delta = dn;
    }
    if (m == -INFINITY) return;
    if (fabsf(m) < kFastLimit) {
        const uint64_t l2 = pk2(kLog2e, kLog2e), nm = pk2(-mc, -mc);
#pragma unroll
        for (int q = 0; q < kVecPerThread; ++q)
            if (okv[q]) {
                float x[EPV];
                unpack_vec<T>(u[q], x);
                exps_fma2<EPV>(x, l2, nm, acc);
            }
    } else {
#pragma unroll
        for (int q = 0; q < kVecPerThread; ++q)
            if (okv[q]) {
                float x[EPV];
                unpack_vec<T>(u[q], x);
#pragma unroll
                for (int j = 0; j < EPV; ++j) acc[j] += fast_exp2((x[j] - m) * kLog2e);
            }
    }
}

template <typename T, class Fin>
__global__ void __launch_bounds__(kThreads, 1) vocab_stream_kernel(const Common c, const typename Fin::Params f) {
    constexpr int EPV = Elem<T>::kPerVec;
    constexpr int UE = kUnitBytes / (int)sizeof(T);    // elements per unit
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ Shared sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            sm100::mbar_init(&sh.full[s], 1);
            sm100::mbar_init(&sh.empty[s], kConsumerWarps);
        }
        for (int r = 0; r < kRed; ++r) {
            sm100::mbar_init(&sh.red_full[r], kConsumerWarps);
            sm100::mbar_init(&sh.red_empty[r], 1);
        }
        sh.abort = 0;
        sm100::fence_mbar_init();
    }
    // The masked flags, copied once: the producer decides from them whether a block is read
    // (a global load per block would sit on its critical path), the publisher counts a
    // sequence's masked rows from them.  A flag changes only in its own sequence's Finish,
    // which runs after every block of that sequence -- this CTA's included -- is done, so
    // for every sequence this CTA still has a block of, the copy equals the live array.
    uint8_t *snap = ring + (size_t)kStages * kUnitBytes;
    const long long rows = (long long)c.B * c.S;
    const bool use_snap = rows <= kMaskSnap;
    int my_masked = 0;
    if (use_snap)
        for (long long r = tid; r < rows; r += kThreads) {
            const uint8_t v = c.masked[r];
            snap[r] = v;
            my_masked += v != 0 ? 1 : 0;
        }
    my_masked = (int)__reduce_add_sync(0xffffffffu, (unsigned)my_masked);
    if (lane == 0) sh.warp_masked[warp] = my_masked;
    __syncthreads();

    if (warp >= kPublisherWarp) {
        // ================================================================ publishers
        // Publisher p takes the ring entries p, p + kPublishers, ... (every slot of the ring
        // belongs to one publisher): the finished blocks in the order the consumers finish
        // them, up to kRed / kPublishers at a time.  The sixteen warp states of a block are
        // merged by a half-warp, one state per lane, the way a consumer warp reduces its
        // lanes (every lane of the half ends with the same bits); lane j then holds entry
        // j's result, writes the block's partial and adds it
        // to its sequence's ticket with an acquire-release atomic, so a batch costs one
        // round trip; a lane whose add completes a sequence has the warp run that sequence's
        // Finish.  No consumer waits on this.
        const int pw = warp - kPublisherWarp;
        int k = pw;                                  // next finished block of this CTA for this warp
        bool more = true;
        while (more) {
            if (!wait_or_abort(sh, &sh.red_full[k % kRed], (uint32_t)(k / kRed) & 1, c.dev_err)) break;
            // the ready prefix of entries k, k+P, k+2P, ... (entry k is ready)
            const int e = k + kPublishers * lane;
            const bool ready = lane < kRed / kPublishers &&
                               (lane == 0 || sm100::mbar_test_wait(&sh.red_full[e % kRed], (uint32_t)(e / kRed) & 1));
            const unsigned rb = __ballot_sync(0xffffffffu, ready);
            const int n = __ffs(~rb) - 1;            // n >= 1 of this warp's entries are ready
            // entries j0 and j0 + 1 by the two half-warps at a time; lane j keeps entry j's state
            float pm = -INFINITY, pz = 0.f;
            int pa = INT_MAX, pblk = -1;
            bool ended = false;
            for (int j0 = 0; j0 < n; j0 += 2) {
                const int j = j0 + (lane >> 4);
                const int r = (k + kPublishers * j) % kRed;
                const int blk = j < n ? sh.red_blk[r] : -1;
                float M = -INFINITY, Z = 0.f;
                int A = INT_MAX;
                if (blk >= 0) { M = sh.red_m[r][lane & 15]; Z = sh.red_z[r][lane & 15]; A = sh.red_a[r][lane & 15]; }
                // as a consumer warp reduces its lanes: the half's maximum, one rescale per
                // lane, a butterfly sum (the same bits in every lane) and the lowest index
                int key = f2key(M);
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
                const float Mb = key2f(key);
                float zt = (M == -INFINITY) ? 0.f : Z * fast_exp2((M - Mb) * kLog2e);
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) zt += __shfl_xor_sync(0xffffffffu, zt, o);
                int at = (Mb != -INFINITY && M == Mb) ? A : INT_MAX;
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) at = min(at, __shfl_xor_sync(0xffffffffu, at, o));
                M = Mb;
                Z = zt;
                A = at;
                // every lane of the half has read the entry (the shuffles above): reusable
                if ((lane & 15) == 0 && blk >= 0) sm100::mbar_arrive(&sh.red_empty[r]);
                ended = ended || (j < n && blk < 0);
                const int from = lane == j0 + 1 ? 16 : 0;
                const float sm_ = __shfl_sync(0xffffffffu, M, from), sz = __shfl_sync(0xffffffffu, Z, from);
                const int sa = __shfl_sync(0xffffffffu, A, from), sb = __shfl_sync(0xffffffffu, blk, from);
                if (lane == j0 || (lane == j0 + 1 && j0 + 1 < n)) { pm = sm_; pz = sz; pa = sa; pblk = sb; }
            }
            int b = -1;
            unsigned last = 0;
            if (lane < n && pblk >= 0) {
                UnmaskPartial q;
                q.m = pm; q.z = pz; q.arg = pa; q.pad = 0;
                c.part[pblk] = q;
                b = pblk / c.bpr / c.S;
                const unsigned target = (unsigned)masked_rows(c, snap, use_snap, b) * (unsigned)c.bpr;
                last = (sm100::atom_add_acq_rel_gpu(&c.tickets[b], 1u) + 1u == target) ? 1u : 0u;
            }
            more = !__any_sync(0xffffffffu, ended);   // the end marker stops the loop
            // Finish every sequence this batch completed, one at a time with the whole warp
            // (the completing lane's acquire-release add acquired every block's partial; the
            // warp barrier orders the other lanes' reads after it)
            unsigned todo = __ballot_sync(0xffffffffu, last != 0);
            __syncwarp();
            while (todo) {
                const int src = __ffs(todo) - 1;
                todo &= todo - 1;
                const int bs = __shfl_sync(0xffffffffu, b, src);
                Fin::finish(c, f, bs, use_snap ? snap + (size_t)bs * c.S : c.masked + (size_t)bs * c.S);
                __syncwarp();
                if (lane == 0) c.tickets[bs] = 0;   // ready for the next launch
            }
            k += kPublishers * n;
        }
        return;
    }

    if (warp == kProducerWarp) {
        // ================================================================ producer (one warp)
        // With the flags in shared memory, the blocks of masked rows are handed out in row
        // order by rank: CTA c takes rank c first, then each next rank from a counter in the
        // workspace (one atomic per block, issued when the block before starts, so its round
        // trip hides behind the copies); CTAs that get more bandwidth take more blocks and
        // all of them run out of work together.  A rank is turned into its row by a forward
        // scan of the flags (ranks only grow within a CTA).  Every block takes exactly one
        // atomic, so the one that returns the last value resets the counter for the next
        // launch.  Without the copy of the flags (very large batches), CTA c takes blocks c,
        // c + grid, c + 2 grid, ... and skips those of rows that are not masked.  Lane 0
        // issues the copies.
        const T *logits = static_cast<const T *>(c.logits);
        const uint64_t pol = sm100::policy_evict_first();   // each logit is read once
        int i = 0;                                       // units issued (stage = i % kStages)
        bool ok = true;
        // the copies of block j (row j / bpr, its units u0 .. u1 - 1); after the first one,
        // lane 0 takes the CTA's next rank from the counter (when one is given)
        unsigned *counter = c.tickets + c.B;
        unsigned nxt = 0;
        auto issue = [&](long long j, bool grab) {
            const long long row = j / c.bpr;
            const int g = (int)(j % c.bpr);
            const int u0 = g * kUnitsPerBlock, u1 = min(c.nc, u0 + kUnitsPerBlock);
            const T *rowp = logits + row * (long long)c.V;
            for (int u = u0; u < u1; ++u, ++i) {
                const int s = i % kStages;
                if (!wait_or_abort(sh, &sh.empty[s], ((uint32_t)(i / kStages) & 1) ^ 1, c.dev_err)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int e0 = u * UE, ne = min(UE, c.V - e0);
                    sh.desc[s] = StageDesc{(int)j, e0, ne / EPV, u == u1 - 1 ? 1 : 0};
                    const uint32_t bytes = (uint32_t)(ne * (int)sizeof(T));
                    sm100::mbar_arrive_expect_tx(&sh.full[s], bytes);
                    sm100::bulk_load_hint(ring + (size_t)s * kUnitBytes, rowp + e0, bytes, &sh.full[s], pol);
                    if (grab && u == u0) nxt = atomicAdd(counter, 1u);   // in flight during the block
                }
                __syncwarp();
            }
        };
        if (use_snap) {
            const int nmr = (int)__reduce_add_sync(0xffffffffu, lane < kThreads / 32 ? (unsigned)sh.warp_masked[lane] : 0u);
            const long long total = (long long)nmr * c.bpr;   // blocks of masked rows
            const int nrows = (int)rows;
            int cur_row = 0, cur_cnt = 0;                     // rows [0, cur_row) hold cur_cnt masked rows
            long long r = blockIdx.x;                         // rank among the blocks of masked rows
            while (ok && r < total) {
                const long long q = r / c.bpr;                 // the q-th masked row
                int row = -1;
                while (cur_row < nrows) {
                    const int rr = cur_row + lane;
                    const bool mk = rr < nrows && snap[rr] != 0;
                    const unsigned bal = __ballot_sync(0xffffffffu, mk);
                    const int cnt = __popc(bal);
                    if (q < cur_cnt + cnt) {
                        const bool hit = mk && __popc(bal & ((1u << lane) - 1u)) == (int)(q - cur_cnt);
                        row = cur_row + __ffs(__ballot_sync(0xffffffffu, hit)) - 1;
                        break;
                    }
                    cur_cnt += cnt;
                    cur_row += 32;
                }
                if (row < 0) {   // cannot happen: the ranks are below the count of the same flags
                    if (lane == 0) report_error(c.dev_err, TT_ERR_BOUNDS);
                    ok = false;
                    break;
                }
                issue((long long)row * c.bpr + r % c.bpr, true);
                if (!ok) break;   // the grab may not have happened: the counter is left to the error
                const unsigned v = __shfl_sync(0xffffffffu, nxt, 0);
                if (lane == 0 && (long long)v == total - 1) *counter = 0u;   // the launch's last atomic
                r = (long long)gridDim.x + v;
            }
        } else {
            for (long long j = blockIdx.x; ok && j < c.nblocks; j += gridDim.x) {
                if (c.masked[j / c.bpr] == 0) continue;   // nothing to read
                issue(j, false);
            }
        }
        // end of the work: a stage without data
        const int s = i % kStages;
        if (ok && wait_or_abort(sh, &sh.empty[s], ((uint32_t)(i / kStages) & 1) ^ 1, c.dev_err)) {
            if (lane == 0) {
                sh.desc[s].blk = -1;
                sm100::mbar_arrive(&sh.full[s]);
            }
        } else if (lane == 0) {
            // the consumers stop on the abort flag; let the copies in flight land first
            for (int k = 1; k <= kStages && i - k >= 0; ++k)
                sm100::mbar_wait(&sh.full[(i - k) % kStages], (uint32_t)((i - k) / kStages) & 1, kWaitLimit);
        }
        return;
    }

    // ==================================================================== consumers
    // sequences with no masked position have no block to wait for: finish them now (each by
    // one warp of one CTA; nothing else in this launch touches them)
    for (int b = blockIdx.x * kConsumerWarps + warp; b < c.B; b += gridDim.x * kConsumerWarps)
        if (masked_rows(c, snap, use_snap, b) == 0)
            Fin::finish(c, f, b, use_snap ? snap + (size_t)b * c.S : c.masked + (size_t)b * c.S);
    // Per thread, over the units of the current block: the running maximum m, the first
    // index a holding it, and the sums (eight scalar accumulators) in the form of
    // vec_exps8_fma / vec_exps8_diff: exp(x - m) times 2^delta.
    float m = -INFINITY, mc = 0.f, delta = 0.f;
    int a = INT_MAX;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int kb = 0;                                      // blocks this warp has finished
    for (int i = 0;; ++i) {
        const int s = i % kStages;
        if (!wait_or_abort(sh, &sh.full[s], (uint32_t)(i / kStages) & 1, c.dev_err)) break;
        const StageDesc d = sh.desc[s];
        if (d.blk < 0) {
            // no more work: hand every publisher an end marker (the next entry of each)
            for (int e = kb; e < kb + kPublishers; ++e) {
                const int r = e % kRed;
                if (!wait_or_abort(sh, &sh.red_empty[r], ((uint32_t)(e / kRed) & 1) ^ 1, c.dev_err)) break;
                if (lane == 0) {
                    if (warp == 0) sh.red_blk[r] = -1;
                    sm100::mbar_arrive(&sh.red_full[r]);
                }
            }
            break;
        }
        const uint4 *pv = reinterpret_cast<const uint4 *>(ring + (size_t)s * kUnitBytes);
        if (d.nvec == kConsumers * kVecPerThread)
            consume_unit<T, true>(pv, d, s, sh, m, mc, delta, a, acc);
        else
            consume_unit<T, false>(pv, d, s, sh, m, mc, delta, a, acc);
        if (d.last) {
            // end of the block: my exact sum, the warp's state, handed to the publisher
            float z = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            if (m != -INFINITY) z *= fast_exp2(-delta);      // remove the 2^delta factor
            warp_reduce_state(m, z, a);
            const int r = kb % kRed;
            if (!wait_or_abort(sh, &sh.red_empty[r], ((uint32_t)(kb / kRed) & 1) ^ 1, c.dev_err)) break;
            if (lane == 0) {
                sh.red_m[r][warp] = m;
                sh.red_z[r][warp] = z;
                sh.red_a[r][warp] = a;
                if (warp == 0) sh.red_blk[r] = d.blk;
                sm100::mbar_arrive(&sh.red_full[r]);
            }
            ++kb;
            m = -INFINITY;
            mc = delta = 0.f;
            a = INT_MAX;
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = 0.f;
        }
    }
}


// ------------------------------------------------------------------ host side

inline int unit_elems(tt_dtype dtype) { return kUnitBytes / (dtype == TT_BF16 ? 2 : 4); }

// Blocks of a batch: B * S rows of ceil(V / unit) units, kUnitsPerBlock units per block.
inline long long blocks_of(int B, int S, int V, tt_dtype dtype) {
    const long long nc = (V + unit_elems(dtype) - 1) / unit_elems(dtype);
    return (long long)B * S * ((nc + kUnitsPerBlock - 1) / kUnitsPerBlock);
}

// Bulk copies need 16-byte aligned rows: an aligned base and a row length in bytes that
// is a multiple of 16.
inline bool rows_aligned(const void *logits, int V, tt_dtype dtype) {
    return reinterpret_cast<uintptr_t>(logits) % 16 == 0 && ((size_t)V * (dtype == TT_BF16 ? 2 : 4)) % 16 == 0;
}

// One launch of the pass with the Finish policy Fin; the workspace pieces are the caller's
// (part: blocks_of() slots; tickets: B + 1 words, the sequences' tickets and then the
// block counter, zero before the first launch and left zero by every launch that
// completes).
template <class Fin>
tt_status launch(const typename Fin::Params &f, const void *logits, tt_dtype dtype, int B, int S, int V,
                 const uint8_t *masked, UnmaskPartial *part, unsigned *tickets, uint32_t *dev_err,
                 cudaStream_t stream) {
    Common c;
    c.logits = logits;
    c.B = B; c.S = S; c.V = V;
    c.nc = (V + unit_elems(dtype) - 1) / unit_elems(dtype);
    c.bpr = (c.nc + kUnitsPerBlock - 1) / kUnitsPerBlock;
    c.nblocks = blocks_of(B, S, V, dtype);
    if (c.nblocks >= (1LL << 31)) return TT_ERR_UNSUPPORTED;   // block ids are 32-bit
    c.masked = masked;
    c.part = part;
    c.tickets = tickets;
    c.dev_err = dev_err;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TT_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TT_ERR_CUDA;
    const int grid = (int)(c.nblocks < sms ? (c.nblocks > 0 ? c.nblocks : 1) : sms);
    auto kernel = dtype == TT_BF16 ? vocab_stream_kernel<uint16_t, Fin> : vocab_stream_kernel<float, Fin>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
        return TT_ERR_CUDA;
    kernel<<<grid, kThreads, kSmemBytes, stream>>>(c, f);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

}  // namespace vs
}  // namespace tt
