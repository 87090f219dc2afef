// Work partition and paged-cache helpers shared by the attention kernels (the 128-row
// tensor-core kernel of the denoise step and the decode kernel of single-position queries).
//
// A segment is one (sequence b, KV head g): the query rows that share every key of that
// head.  Its keys are ceil(L_b / kTileKeys) context tiles of two pages each, then one tile
// of the block's own keys.  Work is counted in units -- a charge per segment for what a
// piece boundary costs, one per context tile, one for the block tile (a cost model per
// kernel) -- and cut into one range per CTA group: whole segments when every group can
// take one and splitting would not pay, otherwise equal unit ranges (stream-K), so ragged
// and long contexts balance with the lengths known only on the device.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "tt_common.cuh"

namespace tt {
namespace {

constexpr int kPage = 64;                // tokens per page
constexpr int kTileKeys = 128;           // keys per context tile (two pages)

// Work units of the stream-K split, one cost model per kernel: a context tile costs
// `tile`, the block tile `block`, and every segment carries `seg` up front for what a
// piece boundary costs (Q load, pipeline refill, epilogue and, for split segments, the
// merge).  When every group can take a whole segment and the longest one is within
// `split` units of the even share (splitting would cost about that much more than it
// saves: a second boundary, the partial write and the merge), each group takes one whole
// segment; a stream-K group gets at least `min_group` units.
//
// The 128-row kernel: its block tile's MMAs are short but its softmax is a full tile's,
// and a boundary costs about three tiles (the Q load into tensor memory and the epilogue
// of 128 rows x 128 columns).
struct TcCosts {
    static constexpr int tile = 8, block = 6, seg = 24, split = 80, min_group = 64;
};

// ------------------------------------------------------------------ work partition

template <class C>
__device__ __forceinline__ int seq_cost(int L, int Hkv) {
    return Hkv * (C::seg + C::tile * ((L + kTileKeys - 1) / kTileKeys) + C::block);
}

struct Piece {
    int b, g, sg;          // sequence, KV head, segment index b * Hkv + g
    int L, ntc;            // context length and its tiles (tile ntc is the block tile)
    int first, last;       // tiles [first, last) of this segment belong to this group
    long long X;           // start unit of the segment
    bool whole;
};

// Walks the pieces of one CTA group's cost range [lo, hi).  Tile i of a segment that
// starts at unit X starts at unit X + C::seg + C::tile * i (the block tile is i = ntc).
template <class C>
struct WorkIter {
    long long U, lo, hi, X;
    int NG;                 // groups that share the work (the stream-K split's divisor)
    int b, g, L, ntc, cost;
    int B, Hkv;
    const long long *pre;   // shared: prefix sums of the sequences' work units
    const int *lens;        // shared: clamped context lengths

    template <class P>
    __device__ void init(const P &p, int group, const long long *pre_, const int *lens_, int max_len) {
        B = p.B; Hkv = p.Hkv; pre = pre_; lens = lens_;
        U = pre[B];
        const long long nseg = (long long)B * Hkv;
        const long long max_seg = seq_cost<C>(max_len, 1);
        NG = p.n_groups;
        if (nseg <= p.n_groups && max_seg <= U / p.n_groups + C::split) {
            // one whole segment per group: the range of segment `group` exactly
            if (group < nseg) {
                const int sb = (int)(group / Hkv), sg = (int)(group % Hkv);
                lo = pre[sb] + (long long)sg * seq_cost<C>(lens[sb], 1);
                hi = lo + seq_cost<C>(lens[sb], 1);
            } else {
                lo = hi = U;
            }
        } else {
            // stream-K over at most U / C::min_group groups, so that a small batch is not
            // cut into one-tile pieces whose merges would cost more than the tiles
            const long long ng = U / C::min_group;
            NG = (int)(ng < 1 ? 1 : (ng < p.n_groups ? ng : p.n_groups));
            if (group < NG) {
                lo = (long long)group * U / NG;
                hi = (long long)(group + 1) * U / NG;
            } else {
                lo = hi = U;
            }
        }
        // the first sequence that ends after lo
        int a = 0, z = B;
        while (a < z) {
            const int mid = (a + z) >> 1;
            if (pre[mid + 1] > lo) z = mid; else a = mid + 1;
        }
        b = a; g = 0;
        X = (b < B) ? pre[b] : U;
        load();
    }
    __device__ void load() {
        if (b < B) {
            L = lens[b];
            ntc = (L + kTileKeys - 1) / kTileKeys;
            cost = C::seg + C::tile * ntc + C::block;
        }
    }
    template <class P>
    __device__ bool next(const P &, Piece &pc) {
        while (b < B && X < hi) {
            const long long T0 = X + C::seg;   // unit of tile 0
            const long long first = (lo > T0) ? (lo - T0 + C::tile - 1) / C::tile : 0;
            long long last = (hi > T0) ? (hi - T0 + C::tile - 1) / C::tile : 0;
            if (last > ntc + 1) last = ntc + 1;
            const bool have = first < last;
            if (have) {
                pc.b = b; pc.g = g; pc.sg = b * Hkv + g; pc.L = L; pc.ntc = ntc;
                pc.first = (int)first; pc.last = (int)last; pc.X = X;
                pc.whole = (first == 0 && last == ntc + 1);
            }
            X += cost;
            if (++g == Hkv) { g = 0; ++b; load(); }
            if (have) return true;
        }
        return false;
    }
};

__device__ __forceinline__ long long range_lo(long long c, long long U, int n) { return c * U / n; }

// The group whose range holds unit u.
__device__ __forceinline__ int owner(long long u, long long U, int n) {
    long long c = u * n / U;
    while (c + 1 < n && range_lo(c + 1, U, n) <= u) ++c;
    while (c > 0 && range_lo(c, U, n) > u) --c;
    return (int)c;
}

// Does group c own at least one tile of the segment starting at unit X with ntc context tiles?
template <class C>
__device__ __forceinline__ bool owns_tile(int c, long long X, int ntc, long long U, int n) {
    const long long lo_c = range_lo(c, U, n), hi_c = range_lo(c + 1, U, n);
    const long long T0 = X + C::seg;
    const long long i0 = (lo_c > T0) ? (lo_c - T0 + C::tile - 1) / C::tile : 0;
    return i0 <= ntc && T0 + C::tile * i0 < hi_c;
}

// The same questions answered from a table lo[c] = range_lo(c) for c = 0..n (filled once
// per launch), without 64-bit divisions.
__device__ __forceinline__ int owner_tab(long long u, const long long *lo, int n) {
    int a = 0, z = n - 1;   // the last c with lo[c] <= u
    while (a < z) {
        const int mid = (a + z + 1) >> 1;
        if (lo[mid] <= u) a = mid; else z = mid - 1;
    }
    return a;
}
template <class C>
__device__ __forceinline__ bool owns_tile_tab(int c, long long X, int ntc, const long long *lo) {
    const long long lo_c = lo[c], hi_c = lo[c + 1];
    const long long T0 = X + C::seg;
    const long long i0 = (lo_c > T0) ? (lo_c - T0 + C::tile - 1) / C::tile : 0;
    return i0 <= ntc && T0 + C::tile * i0 < hi_c;
}

// The groups that own the first and the last tile of the segment starting at unit X.
template <class C>
__device__ __forceinline__ int first_owner(long long X, long long U, int n) { return owner(X + C::seg, U, n); }
template <class C>
__device__ __forceinline__ int last_owner(long long X, int ntc, long long U, int n) {
    return owner(X + C::seg + (long long)C::tile * ntc, U, n);
}

// Physical page of logical page pg of the piece's sequence (0 past the context; an id
// outside the pool is reported and replaced by 0 so that no copy leaves the pool).
template <class P>
__device__ __forceinline__ int page_id(const P &p, const Piece &pc, int pg) {
    if (pg * kPage >= pc.L) return 0;
    const int id = p.page_table[(size_t)pc.b * p.max_pages + pg];
    if (id < 0 || id >= p.num_pages) {
        report_error(p.dev_err, TT_ERR_BOUNDS);
        return 0;
    }
    return id;
}

__device__ __forceinline__ int tile_valid(const Piece &pc, int i, int S) {
    return i < pc.ntc ? min(kTileKeys, pc.L - kTileKeys * i) : S;
}

// ------------------------------------------------------------------ host: tensor maps

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// A bf16 tensor map with 128-byte swizzle (dims, strides in bytes, box: innermost first).
inline bool make_map(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims, const uint64_t *strides,
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

// The K and V pools of a paged cache as [num_pages][Hkv][64 tokens][D = 128] maps with a
// box of one 64-column half of one page of one KV head.
inline bool make_pool_maps(const tt_kv_cache &c, int Hkv, CUtensorMap *mk, CUtensorMap *mv) {
    const uint64_t dims[4] = {128, (uint64_t)kPage, (uint64_t)Hkv, (uint64_t)c.num_pages};
    const uint64_t str[3] = {128 * 2, (uint64_t)kPage * 128 * 2, (uint64_t)Hkv * kPage * 128 * 2};
    const uint32_t box[4] = {64, (uint32_t)kPage, 1, 1};
    return make_map(mk, c.k_pool, 4, dims, str, box) && make_map(mv, c.v_pool, 4, dims, str, box);
}

}  // namespace
}  // namespace tt
