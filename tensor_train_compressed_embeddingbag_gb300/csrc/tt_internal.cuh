// tt_internal.cuh -- shared definitions of the TT-EmbeddingBag CUDA library (sm_103a).
//
// Forward pass of one call, in stream order:
//   k_decode_small | k_decode_hist   decode i -> (i1,i2,i3), bag id and pooling
//                   scale per lookup; mark the touched (i1, i2) pairs
//   grouping for the backward pass (stable counting sorts), either
//     nnz <= kSmallMaxNnz: per-chunk ranks in k_decode_small, scans by extra
//                   blocks of k_fwd_T, scatter by extra blocks of k_pool -> pi1 by (i1, pos),
//                   pi3 by (i3, pos), pi21 by (i2, pos), tiles
//     larger nnz:   per-chunk histograms in k_decode_hist, segmented scans
//                   (k_scan_sums, k_scan_apply), k_scatter13, the same scans of
//                   the i2 histogram (the last block cuts the tiles), k_scatter2
//                   -> pi1, pi3, pi21 by (i2, i1, pos) (pairs contiguous), tiles
//   k_fwd_T         per (table, i2): T = G1[i1] G2[i2] for every touched pair
//   k_pool          per bag: row = T G3[i3], pooled in registers -> out
// and the backward pass:
//   k_tile_bwd      per tile (x column split), sorted in shared memory by
//                   (i1, i3, pos): summed upstream gradient per row,
//                   dG3 partial per row, dT per pair, dG1 partial per pair, dG2
//                   of the group (reduced over the group's tiles by its last
//                   tile, which applies the G2 update)
//   k_reduce13      per i1 / i3 slice: sum of the partials in sorted-segment
//                   order, G1 / G3 update
//   k_cache_gmax, k_cache_acc, k_cache_apply (trainable cache rows only): the
//                   hits' gradient per cached value as a 64-bit fixed-point sum,
//                   then its optimizer step
// Every floating-point sum runs in an order fixed by the sort keys, so results are
// bitwise reproducible; no floating-point atomics are used (the trainable rows'
// sums are integer).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/tt_emb.h"

namespace ttemb {

constexpr int kChunk = 2048;        // lookups per counting-sort chunk
constexpr int kSortThreads = 256;   // 8 warps; each warp owns kChunk/8 consecutive lookups
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kWarpSpan = kChunk / kSortWarps;
constexpr int kScanThreads = 1024;
constexpr int kScanPer = 16;                       // histogram elements per thread and round of a scan
constexpr int kScanSeg = kScanThreads * kScanPer;  // histogram elements per block of the scans
constexpr int kTileThreads = 256;
constexpr int kMaxBinsPerDigit = 6144;  // per-warp rank tables: 8 x bins x 4 B of shared memory
constexpr int kFieldBits = 20;          // bits per field of the in-tile sort key
constexpr int kSmallMaxNnz = 12288;     // small path: lookups
constexpr int kSmallMaxBins = 1024;     // small path: bins per digit
constexpr int kSmallChunk = 256;        // small path: lookups per decode block (8 warps)
constexpr int kDecodeOffs = 1024;       // bag offsets staged per decode block
constexpr int kMaxD = 256;              // largest q1 q2 q3

enum ErrBits { kErrIndex = 1, kErrOffsets = 2, kErrTimeout = 4, kErrBounds = 8 };

// Debug build (compiled with -DTTEMB_DEBUG): every index below that is derived from
// data (decoded slices, bag ids, positions in the sorted orders, tile ranges, partial
// slots) is checked against its bound where it is used; an index outside [0, bound)
// records kErrBounds (tt_emb_get_last_error: TT_ERR_BOUNDS) and is clamped into range,
// so the access stays inside its buffer.  The release build compiles the checks away.
#ifdef TTEMB_DEBUG
template <class I>
__device__ __forceinline__ I dcheck(int* err, I v, int64_t bound) {
    if (v < 0 || (int64_t)v >= bound) {
        atomicOr(err, kErrBounds);
        return (I)(v < 0 ? 0 : (bound > 0 ? bound - 1 : 0));
    }
    return v;
}
#define TT_DCHECK(P, v, bound) ::ttemb::dcheck((P).err, (v), (int64_t)(bound))
#else
#define TT_DCHECK(P, v, bound) (v)
#endif

constexpr unsigned kTcWaitPolls = 1u << 24;  // default polls of a bounded mbarrier wait

struct TableDev {
    int64_t E;
    int p1, p2, p3;
    int q1, q2, q3;
    int r1, r2;
    int D;
    float* G1;
    float* G2;
    float* G3;
    int64_t tbase;  // float offset of this table's dense (i2, i1) block in Tbuf
    int64_t fbase;  // offset of this table's dense (i2, i1) touched-flag block
    int base1, base2, base3;  // first global bin of each digit
    int dclass;     // compiled dimension class (tt_dims.cuh)
    int idx32;      // p1 p2 p3 < 2^31: rows decode with 32-bit arithmetic
    float* aux[3];  // per core: Adagrad state or gradient buffer (tt_emb_set_optimizer), else null
};

struct Params {
    // handle constants
    const TableDev* tables;
    int ntab;
    int n1, n2, n3;                 // bins per digit (sum over tables of p1, p2, p3)
    const int* bin1_tab;            // bin -> table, per digit
    const int* bin2_tab;
    const int* bin3_tab;
    int D;
    int qs_max;                     // max q1 r1  (dG1 partial stride)
    int ps_max;                     // max r2 q3  (dG3 partial stride)
    int s2_max;                     // max r1 q2 r2 (dG2 partial stride)
    int tile_cap;                   // max lookups per tile (power of two, <= kTileThreads)
    int r1_max, N_max, q1N_max;     // max r1, q2 r2 and q1 q2 r2 over the tables
    int fwd_tc_floats;              // k_fwd_T tensor-core operand tiles (max over the tables that use them)
    int p1_max;
    int split;                      // column splits of r2 in k_tile_bwd (1 or 2)
    int small;                      // 1: chunk-rank path (nnz <= kSmallMaxNnz); pi21 is then ordered by (i2, pos)
    int dclass_all;                 // dimension class shared by every table, or -1 (mixed)
    int fwd_split;                  // k_fwd_T blocks per (table, i2) group (1 or 2)
    int sms;                        // multiprocessors of the handle's device (grid sizes)
    unsigned wait_polls;            // polls before a bounded mbarrier wait gives up (tt_emb_set_wait_limit)
    int bwd_tc;                     // 1: k_tile_bwd_tc (tensor cores) takes the backward tiles
    int g1s_floats, dts_floats;     // k_tile_bwd batch buffers (max over tables, this call's split)
    int g2s_floats;                 // k_tile_bwd G2 columns of one split, padded rows (max over tables)
    // call arguments
    const int64_t* idx;
    const int64_t* off;
    const float* w;
    int mean;
    int64_t nnz;
    int64_t nbags;
    int64_t bags_per_table;
    float* out;
    const float* grad_out;
    float lr;
    int opt;                        // tt_optim of the backward: what happens to each core gradient
    float eps;                      // Adagrad denominator term
    int nch;                        // chunks of kChunk lookups
    int max_tiles;
    // workspace
    int* lk_i1;
    int* lk_i2;
    int* lk_i3;
    int* lk_bag;
    float* lk_s;
    uint16_t* lr1;                  // small path: rank of the lookup in its chunk among equal i1 / i2 / i3
    uint16_t* lr2;
    uint16_t* lr3;
    int* H1;                        // [n1][nch]
    int* H3;                        // [n3][nch]
    int* H2;                        // [n2][nch]
    int* pi1;
    int* pi3;
    int* pi21;
    // the lookups' (i1, i3, bag, scale) in the (table, i2)-grouped order of pi21,
    // written by the grouping scatter so that k_tile_bwd reads a tile in one pass
    int* g_i1;
    int* g_i3;
    int* g_bag;
    float* g_s;
    int* g_p1;                      // grouped order: the lookup's position in pi1
    int* g_p3;                      // grouped order: the lookup's position in pi3
    int* inv3;                      // [nnz] position of lookup n in pi3 (multi-CTA grouping)
    int* sigma;
    int4* tiles;                    // {start, len, group bin, tile index in group}
    int* tile_order;                // small path with the tensor-core backward: tile ids in launch
                                    // order, longest first (else the identity)
    int* tflag;                     // dense touched-pair flags, == *epoch when touched by this call
    int* epoch;                     // device counter: advanced by k_pool at the end of every forward pass
    int* ntiles;
    int* grp_first;                 // [n2]
    int* grp_ntiles;                // [n2]
    int* grp_done;                  // [n2], zero between calls
    int* multi_groups;              // [n2]: the (table, i2) groups of several tiles, in group order
    int* multi_count;               // their number (written by the tile cut)
    int* dec_done;                  // [kDecDoneSlots]: small-path decode block c stores the pass's
                                    // epoch once the touched flags of its lookups are written
    float* Tbuf;
    int* rep1;                      // [nnz] by position in pi1: partial slot of the tile-pair starting at that lookup, or -1
    int* rep3;                      // [nnz] by position in pi3: partial slot of the tile-row starting at that lookup, or -1
                                    // (slot = position of that lookup in pi21)
    float* Qbuf;                    // [nnz][qs_max]
    float* Pbuf;                    // [nnz][ps_max]
    float* dG2part;                 // [max_tiles][s2_max]
    int* nincl;                     // lookups in the sorted orders (all but the trainable cache hits)
    int* segsum;                    // segment totals of the multi-block histogram scans
    int* scan_done;                 // blocks of the H2 scan that have finished (0 between passes)
    int* err;
    // hot-row cache (single table)
    const int64_t* cache_rows;      // row id per slot (-1 = empty way)
    const longlong2* cache_hidx;    // explicit rows: open-addressing index, (row id or -1, slot)
    int cache_hmask;                //   entries - 1 (a power of two minus one)
    int cache_hprobe;               //   longest probe sequence of the index
    int64_t cache_n;
    float* cache_vals;              // [cache_n][D]
    int* cache_stamp;               // [cache_n] *dstep when the row was computed
    int* cache_claim;               // [cache_n] epoch of the pass whose decode chose the row's refresher
    int* slice_stamp;               // [p1 + p2 + p3] *dstep + 1 of the backward that last changed the slice
    int* dstep;                     // device counter: advanced by the decode kernel of every forward pass
    // FBTT README, "Software Cache": access-frequency table (open addressing, linear
    // probing) updated by every forward pass, and the set-associative layout of the
    // cache (cache_sets > 0: slot = set * kLfuWays + way; 0: cache_rows sorted)
    unsigned long long* freq_keys;  // [freq_mask + 1], ~0 = empty
    unsigned* freq_counts;          // [freq_mask + 1]
    int freq_mask;
    int cache_sets;
    // trainable cache rows (FBTT README, "Parameters": sparse, the gradient w.r.t. the
    // cache): a hit reads the cached value and its gradient goes to that value
    int cache_train;
    int* lk_hit;                    // [nnz] cache slot of the lookup, or -1
    float* lk_sh;                   // [nnz] pooling scale of a hit (its TT scale is 0)
    unsigned long long* cache_acc;  // [cache_n][D] fixed-point gradient sums
    float* cache_state;             // [cache_n][D] Adagrad accumulators of the cached values
    float* cache_grad;              // [cache_n][D] last gradient of the cached values (sparse=False)
    unsigned* cache_gmax;           // [4]: max|grad_out| (float bits), shift S, touched slots, max|hit scale|
    int* cache_touch;               // [cache_n] 1 once a hit of this step touched the slot
    int* cache_list;                // [cache_n] the touched slots of the step
};

// ---------------------------------------------------------------- helpers

// Programmatic dependent launch: let the next kernel of the stream launch now
// (its blocks then wait in pdl_wait), and wait until the previous kernel of the
// stream has completed and its writes are visible.  Both are no-ops for a
// kernel launched without the programmatic-serialization attribute.  Every
// kernel calls this before its first global memory access.
// The one write of core element i (of the slice at G, aux) with its gradient g,
// after every gradient of the step has been taken (FBTT README, "Parameters":
// sparse, optimizer, learning_rate, eps):
//   TT_OPT_SGD      G -= lr g
//   TT_OPT_ADAGRAD  s += g^2;  G -= lr g / (sqrt(s) + eps)      (s = aux, per element)
//   TT_OPT_GRAD     aux = g, G unchanged                         (sparse = False)
__device__ __forceinline__ void core_update(const Params& P, float* G, float* aux, int64_t i, float g) {
    if (P.opt == TT_OPT_SGD) {
        G[i] = fmaf(-P.lr, g, G[i]);
    } else if (P.opt == TT_OPT_ADAGRAD) {
        const float st = fmaf(g, g, aux[i]);
        aux[i] = st;
        G[i] -= P.lr * g / (sqrtf(st) + P.eps);
    } else {
        aux[i] = g;
    }
}

// core_update of n elements, every load issued before the first store (the
// elements are distinct, so the order of the writes does not matter).
template <int N>
__device__ __forceinline__ void core_update_n(const Params& P, float* G, float* aux, const int* idx, const float* g) {
    if (P.opt == TT_OPT_GRAD) {
#pragma unroll
        for (int i = 0; i < N; ++i) aux[idx[i]] = g[i];
        return;
    }
    float w[N], st[N];
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = G[idx[i]];
    if (P.opt == TT_OPT_ADAGRAD) {
#pragma unroll
        for (int i = 0; i < N; ++i) st[i] = fmaf(g[i], g[i], aux[idx[i]]);
#pragma unroll
        for (int i = 0; i < N; ++i) {
            aux[idx[i]] = st[i];
            G[idx[i]] = w[i] - P.lr * g[i] / (sqrtf(st[i]) + P.eps);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) G[idx[i]] = fmaf(-P.lr, g[i], w[i]);
    }
}

// sum[u] = the sum over tiles tt < nt, in tile order, of part[tt * stride + e[u]] for NE
// elements (e[u] < 0: none); four tiles' loads of every element in flight at once.
template <int NE>
__device__ __forceinline__ void sum_partials(const float* part, int64_t stride, int nt, const int* e, float* sum) {
#pragma unroll
    for (int u = 0; u < NE; ++u) sum[u] = 0.f;
    int tt = 0;
    for (; tt + 4 <= nt; tt += 4) {
        float x[NE][4];
#pragma unroll
        for (int u = 0; u < NE; ++u)
#pragma unroll
            for (int k = 0; k < 4; ++k) x[u][k] = e[u] >= 0 ? __ldcg(part + (int64_t)(tt + k) * stride + e[u]) : 0.f;
#pragma unroll
        for (int u = 0; u < NE; ++u)
#pragma unroll
            for (int k = 0; k < 4; ++k) sum[u] += x[u][k];
    }
    for (; tt < nt; ++tt)
#pragma unroll
        for (int u = 0; u < NE; ++u)
            if (e[u] >= 0) sum[u] += __ldcg(part + (int64_t)tt * stride + e[u]);
}

// core_update_n where idx[i] < 0 marks an unused slot.
template <int N>
__device__ __forceinline__ void core_update_nm(const Params& P, float* G, float* aux, const int* idx, const float* g) {
    if (P.opt == TT_OPT_GRAD) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (idx[i] >= 0) aux[idx[i]] = g[i];
        return;
    }
    float w[N], st[N];
#pragma unroll
    for (int i = 0; i < N; ++i) w[i] = idx[i] >= 0 ? G[idx[i]] : 0.f;
    if (P.opt == TT_OPT_ADAGRAD) {
#pragma unroll
        for (int i = 0; i < N; ++i) st[i] = idx[i] >= 0 ? fmaf(g[i], g[i], aux[idx[i]]) : 0.f;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            if (idx[i] < 0) continue;
            aux[idx[i]] = st[i];
            G[idx[i]] = w[i] - P.lr * g[i] / (sqrtf(st[i]) + P.eps);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (idx[i] >= 0) G[idx[i]] = fmaf(-P.lr, g[i], w[i]);
    }
}

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_entry() {
    pdl_launch_dependents();
    pdl_wait();
}

constexpr int kDecDoneSlots = 64;        // >= the small path's decode blocks
constexpr int kDecodeFlagPolls = 256;    // polls of the decode stamps before the grid wait

// Small path: the k_fwd_T blocks of the (table, i2) groups read only the touched flags
// of the decode kernel just before them, not its histograms.  They wait for every decode
// block's epoch stamp (bounded polls; then the whole-grid wait) instead of the grid's end.
__device__ __forceinline__ void wait_decode_flags(const Params& P) {
    const int epoch = *P.epoch;
    bool ok = false;
    for (int it = 0; it < kDecodeFlagPolls && !ok; ++it) {
        const bool mine = (int)threadIdx.x >= P.nch || *(volatile const int*)(P.dec_done + threadIdx.x) == epoch;
        ok = __syncthreads_and(mine);
        if (!ok) __nanosleep(64);
    }
    if (!ok) pdl_wait();
    __threadfence();
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan of one int per thread across the block; sh needs 33 ints.
__device__ __forceinline__ int block_scan_excl(int x, int* sh, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sh[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int v = lane < nw ? sh[lane] : 0;
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += y;
        }
        if (lane < nw) sh[lane] = inc - v;
        if (lane == 31) sh[32] = inc;
    }
    __syncthreads();
    int res = sh[wid] + incl - x;
    *total = sh[32];
    __syncthreads();
    return res;
}

// Block-wide copy of n floats from global to shared memory with U loads in
// flight per thread (a plain strided loop would wait for each load in turn).
template <int U = 8>
__device__ __forceinline__ void stage_f32(float* dst, const float* src, int n) {
    for (int base = 0; base < n; base += U * blockDim.x) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * blockDim.x + threadIdx.x;
            v[u] = i < n ? __ldg(src + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = base + u * blockDim.x + threadIdx.x;
            if (i < n) dst[i] = v[u];
        }
    }
}

__device__ __forceinline__ int table_of_bag(const Params& P, int bag) {
    return P.ntab == 1 ? 0 : (int)(bag / P.bags_per_table);
}

// Largest g in [0, nbags) with off[g] <= n (the bag of lookup n when offsets are valid).
__device__ __forceinline__ int64_t bag_of(const Params& P, int64_t n) {
    int64_t a = 0, b = P.nbags;
    while (b - a > 1) {
        const int64_t m = (a + b) >> 1;
        if (P.off[m] <= n) a = m; else b = m;
    }
    return a;
}

// Decode lookup n of bag `bag`: slice indices, pooling scale, touched-pair flag.
// SplitMix64 output function (Steele, Lea and Flood, "Fast splittable pseudorandom
// number generators", OOPSLA 2014): the first output of a generator seeded with x.
// Hashes row ids for the frequency table (low bits) and the cache sets (high bits).
__host__ __device__ __forceinline__ uint64_t mix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

constexpr int kLfuWays = 32;      // cache associativity
constexpr int kLfuMaxProbe = 64;  // frequency-table probes before a lookup goes uncounted

__host__ __device__ __forceinline__ int64_t lfu_set_of(int64_t row, int sets) {
    return (int64_t)((mix64((uint64_t)row) >> 32) % (uint64_t)sets);
}

// Count one access of `row` in the frequency table (integer atomics: the final
// counts do not depend on the order of the lookups while the table has room).
__device__ __forceinline__ void lfu_count(const Params& P, int64_t row) {
    unsigned slot = (unsigned)mix64((uint64_t)row) & (unsigned)P.freq_mask;
    for (int probe = 0; probe < kLfuMaxProbe; ++probe) {
        unsigned long long k = P.freq_keys[slot];
        if (k == ~0ull) k = atomicCAS(P.freq_keys + slot, ~0ull, (unsigned long long)row);
        if (k == ~0ull || k == (unsigned long long)row) {
            atomicAdd(P.freq_counts + slot, 1u);
            return;
        }
        slot = (slot + 1) & (unsigned)P.freq_mask;
    }
}

// Lookup n with its index `row` and weight `w` (loaded by the caller, so that the
// loads can be issued early).
// Cache slot of `row` (table 0) or -1.  Set-associative cache: the kLfuWays ways of
// the row's set, all loaded at once (16-byte loads of a 256-byte aligned set).
// Explicit rows: linear probing in the open-addressing index from entry
// mix64(row) mod size, at most the index's longest probe sequence; with has_pre,
// `pre` is that first entry, already loaded.
__device__ __forceinline__ int cache_find(const Params& P, int64_t row, bool has_pre = false,
                                          longlong2 pre = longlong2{-1, 0}) {
    if (P.cache_sets > 0) {
        const longlong2* set = reinterpret_cast<const longlong2*>(P.cache_rows + lfu_set_of(row, P.cache_sets) * kLfuWays);
        long long w[kLfuWays];
#pragma unroll
        for (int v = 0; v < kLfuWays / 2; ++v) {
            const longlong2 x = __ldg(set + v);
            w[2 * v] = x.x;
            w[2 * v + 1] = x.y;
        }
        int found = -1;
#pragma unroll
        for (int v = 0; v < kLfuWays; ++v) found = (w[v] == row) ? v : found;
        return found < 0 ? -1 : (int)(lfu_set_of(row, P.cache_sets) * kLfuWays) + found;
    }
    unsigned e = (unsigned)mix64((uint64_t)row) & (unsigned)P.cache_hmask;
    for (int k = 0; k < P.cache_hprobe; ++k) {
        const longlong2 x = (k == 0 && has_pre) ? pre : __ldg(P.cache_hidx + e);
        if (x.x == row) return (int)x.y;
        if (x.x < 0) return -1;
        e = (e + 1) & (unsigned)P.cache_hmask;
    }
    return -1;
}

// Returns false for a lookup that stays out of the TT path and its grouping (a
// trainable cache hit), true otherwise.  CACHE: the handle has a hot-row cache.
template <bool CACHE>
__device__ __forceinline__ bool decode_lookup(const Params& P, int64_t n, int bag, int64_t row, float w, int& t,
                                              int& i1, int& i2, int& i3, int epoch, bool has_pre = false,
                                              longlong2 pre = longlong2{-1, 0}) {
    t = table_of_bag(P, bag);
    const TableDev& T = P.tables[t];
    float s = w;
    const bool valid = row >= 0 && row < T.E;
    if (!valid) {
        atomicOr(P.err, kErrIndex);
        row = 0;
        s = 0.0f;
    } else if (P.freq_keys) {  // FBTT README, "Software Cache": every forward counts its rows
        lfu_count(P, row);
    }
    if (P.mean) {
        const int64_t L = P.off[bag + 1] - P.off[bag];
        s = s / (float)(L > 0 ? L : 1);
    }
    if (T.idx32) {
        const unsigned r = (unsigned)row, p3 = (unsigned)T.p3, q = r / p3;
        i3 = (int)(r - q * p3);
        i2 = (int)(q % (unsigned)T.p2);
        i1 = (int)(q / (unsigned)T.p2);
    } else {
        const int64_t p23 = (int64_t)T.p2 * T.p3;
        i1 = (int)(row / p23);
        i2 = (int)((row / T.p3) % T.p2);
        i3 = (int)(row % T.p3);
    }
    // cache: lk_hit = slot for a lookup that reads its cached value (the pool gives its
    // TT path scale 0), -2 - slot for the one lookup of a pass that refreshes a stale
    // exact copy, -1 otherwise.  A trainable hit takes no part in the cores' gradient
    // (lk_s = 0); an exact-copy hit keeps it.
    if constexpr (CACHE) {
        int slot = valid ? cache_find(P, row, has_pre, pre) : -1;
        if (slot >= 0) {
            if (P.cache_train) {
                P.lk_sh[n] = s;
                s = 0.0f;
            } else {
                const int need = max(max(P.slice_stamp[i1], P.slice_stamp[T.p1 + i2]), P.slice_stamp[T.p1 + T.p2 + i3]);
                if (P.cache_stamp[slot] >= need)
                    P.lk_sh[n] = s;
                else
                    slot = atomicExch(P.cache_claim + slot, epoch) != epoch ? -2 - slot : -1;
            }
        }
        P.lk_hit[n] = slot;
    }
    i1 = TT_DCHECK(P, i1, T.p1);
    i2 = TT_DCHECK(P, i2, T.p2);
    i3 = TT_DCHECK(P, i3, T.p3);
    P.lk_i1[n] = i1;
    P.lk_i2[n] = i2;
    P.lk_i3[n] = i3;
    P.lk_bag[n] = TT_DCHECK(P, bag, P.nbags);
    P.lk_s[n] = s;
    if (CACHE && P.cache_train && P.lk_hit[n] >= 0) return false;
    P.tflag[T.fbase + (int64_t)i2 * T.p1 + i1] = epoch;
    return true;
}

// The lookup stays out of the sorted orders (a trainable cache hit).
__device__ __forceinline__ bool excluded(const Params& P, int64_t n) {
    return P.cache_train && P.lk_hit[n] >= 0;
}

// Small path, part `part` (of kSmallChunk / blockDim) of chunk c: position =
// scanned base of (digit, chunk) + rank in chunk; a thread per lookup.
__device__ __forceinline__ void scatter_chunk(const Params& P, int c, int part) {
    const int64_t lo = (int64_t)c * kSmallChunk + (int64_t)part * blockDim.x;
    const int64_t cend = (int64_t)(c + 1) * kSmallChunk;
    const int64_t hi = (cend < P.nnz) ? cend : P.nnz;
    for (int64_t n = lo + threadIdx.x; n < hi && n < lo + blockDim.x; n += blockDim.x) {
        if (excluded(P, n)) continue;
        const TableDev& T = P.tables[table_of_bag(P, P.lk_bag[n])];
        const int d1 = T.base1 + P.lk_i1[n], d2 = T.base2 + P.lk_i2[n], d3 = T.base3 + P.lk_i3[n];
        const int p1 = TT_DCHECK(P, P.H1[(int64_t)d1 * P.nch + c] + P.lr1[n], P.nnz);
        const int p3 = TT_DCHECK(P, P.H3[(int64_t)d3 * P.nch + c] + P.lr3[n], P.nnz);
        const int pos = TT_DCHECK(P, P.H2[(int64_t)d2 * P.nch + c] + P.lr2[n], P.nnz);
        P.pi1[p1] = (int)n;
        P.pi3[p3] = (int)n;
        P.pi21[pos] = (int)n;
        P.g_i1[pos] = P.lk_i1[n];
        P.g_i3[pos] = P.lk_i3[n];
        P.g_bag[pos] = P.lk_bag[n];
        P.g_s[pos] = P.lk_s[n];
        P.g_p1[pos] = p1;
        P.g_p3[pos] = p3;
    }
}

// Small path: exclusive scan of digit k's [bin][chunk] histogram (k = 0: i1,
// 1: i2, 2: i3) by one block, in place in global memory.  Rounds of blockDim
// bins: the round's rows (contiguous) are copied to shared memory with coalesced
// int4 loads, eight in flight per thread; a thread per bin sums its row, the
// block scans the bin totals, the thread rewrites its row as running prefixes,
// and the rows go back with coalesced stores.  The i2 block then cuts every
// (table, i2) group into tiles of <= tile_cap lookups.  sm: kScanSmemInts ints.
constexpr int kMaxTcTileCap = 64;  // the tensor-core backward's tile cap
constexpr int kScanChunkMax = 48;  // >= kSmallMaxNnz / kSmallChunk
constexpr int kScanBlock = 256;    // threads of the scanning block
constexpr int kScanSmemInts = 64 + kScanBlock * kScanChunkMax;
__device__ __forceinline__ void scan_digit_block(const Params& P, int k, int* sm) {
    int* sh = sm;
    int* hs = sm + 64;  // 16-byte aligned when sm is
    const int nb = k == 0 ? P.n1 : (k == 1 ? P.n2 : P.n3);
    int* H = k == 0 ? P.H1 : (k == 1 ? P.H2 : P.H3);
    const int nch = P.nch;  // <= kScanChunkMax on this path
    int carry = 0, tcarry = 0, mcarry = 0;
    for (int b0 = 0; b0 < nb; b0 += kScanBlock) {
        const int nbr = min(kScanBlock, nb - b0);
        const int n = nbr * nch, n4 = n >> 2;
        int* src = H + (int64_t)b0 * nch;  // 16-byte aligned: H is, and b0 nch is a multiple of 256
        for (int base = 0; base < n4; base += 8 * kScanBlock) {
            int4 v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = base + q * kScanBlock + threadIdx.x;
                if (e < n4) v[q] = reinterpret_cast<const int4*>(src)[e];
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = base + q * kScanBlock + threadIdx.x;
                if (e < n4) reinterpret_cast<int4*>(hs)[e] = v[q];
            }
        }
        for (int e = 4 * n4 + threadIdx.x; e < n; e += kScanBlock) hs[e] = src[e];
        __syncthreads();
        const int bl = threadIdx.x, b = b0 + bl;
        int tot = 0;
        if (bl < nbr)
            for (int c = 0; c < nch; ++c) tot += hs[bl * nch + c];
        int total;
        const int start = carry + block_scan_excl(tot, sh, &total);
        if (bl < nbr) {
            int run = start;
            for (int c = 0; c < nch; ++c) {
                const int x = hs[bl * nch + c];
                hs[bl * nch + c] = run;
                run += x;
            }
        }
        carry += total;
        if (k == 1) {  // tiles of the (table, i2) groups of this round of bins
            const int cap = P.tile_cap;
            const int nt = bl < nbr ? (tot + cap - 1) / cap : 0;
            int ttot, mtot;
            const int first = tcarry + block_scan_excl(nt, sh, &ttot);
            __syncthreads();
            const int mpos = mcarry + block_scan_excl(nt > 1 ? 1 : 0, sh, &mtot);
            if (bl < nbr) {
                P.grp_first[b] = first;
                P.grp_ntiles[b] = nt;
                for (int t = 0; t < nt; ++t)
                    P.tiles[first + t] = make_int4(start + t * cap, min(cap, tot - t * cap), b, t);
                if (nt > 1) P.multi_groups[mpos] = b;
            }
            tcarry += ttot;
            mcarry += mtot;
        }
        __syncthreads();
        for (int e = threadIdx.x; e < n4; e += kScanBlock) reinterpret_cast<int4*>(src)[e] = reinterpret_cast<const int4*>(hs)[e];
        for (int e = 4 * n4 + threadIdx.x; e < n; e += kScanBlock) src[e] = hs[e];
        __syncthreads();  // the next round reuses hs
    }
    if (k == 1 && threadIdx.x == 0) {
        *P.ntiles = tcarry;
        *P.multi_count = mcarry;
    }
    if (k == 1 && P.bwd_tc) {
        // launch order of the tensor-core backward's tiles: longest first (a counting sort
        // by length; the order within a length does not matter), so that the longest
        // tiles are placed first, one to an SM
        static_assert(kMaxTcTileCap + 1 <= kScanBlock, "a tile length per thread");
        __syncthreads();
        int* bucket = hs;  // [tile_cap + 1], the histogram rows are written back
        const int cap = P.tile_cap;
        for (int b = threadIdx.x; b <= cap; b += kScanBlock) bucket[b] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < tcarry; i += kScanBlock) atomicAdd(&bucket[__ldcg(&P.tiles[i].y)], 1);
        __syncthreads();
        const int len = cap - (int)threadIdx.x;  // thread t: length cap - t
        const int cnt = len >= 0 ? bucket[len] : 0;
        int total;
        const int pos0 = block_scan_excl(cnt, sh, &total);
        __syncthreads();
        if (len >= 0) bucket[len] = pos0;
        __syncthreads();
        for (int i = threadIdx.x; i < tcarry; i += kScanBlock) P.tile_order[atomicAdd(&bucket[__ldcg(&P.tiles[i].y)], 1)] = i;
    }
    if (k == 0 && threadIdx.x == 0) *P.nincl = carry;
}

// ---------------------------------------------------------------- launchers
// Each returns the cudaError_t of its launch.

extern bool g_use_pdl;  // programmatic dependent launch between the library's kernels

// Allow a kernel the largest dynamic shared memory the device permits next to
// its static shared memory, and ask for the largest shared-memory carve-out.
// The carve-out matters for the overlap of consecutive kernels: an SM whose
// L1/shared split was chosen for a kernel with little shared memory cannot take
// a block that needs more until it has drained, so every kernel of the library
// asks for the same (maximal) split and the blocks of the next kernel can move
// in next to those of the previous one.
inline cudaError_t allow_max_dynamic_smem(const void* kernel, int max_smem) {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, kernel);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem - (int)a.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}

// Launch with the programmatic-stream-serialization attribute (see pdl_entry).
template <class... Args>
inline cudaError_t launch_pdl(void (*kernel)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              const Params& P) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = g_use_pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, P);
}
cudaError_t launch_decode_small(const Params& P, cudaStream_t s);
cudaError_t launch_decode_hist(const Params& P, cudaStream_t s);
cudaError_t launch_scan13(const Params& P, cudaStream_t s);
cudaError_t launch_scan_sums13(const Params& P, cudaStream_t s);
cudaError_t launch_scan_sums2(const Params& P, cudaStream_t s);
// Blocks of the histogram scans: W = 0 the H1 and H3 segments (*s1 = H1's), W = 1 H2's.
int scan_segments(const Params& P, int W, int* s1 = nullptr);
cudaError_t launch_scatter13(const Params& P, cudaStream_t s);
cudaError_t launch_scan2_tiles(const Params& P, cudaStream_t s);
cudaError_t launch_scatter2(const Params& P, cudaStream_t s);
cudaError_t launch_fwd_T(const Params& P, cudaStream_t s);
int fwd_tc_floats_of(int dclass, int r1, int N);
cudaError_t launch_pool(const Params& P, cudaStream_t s);
cudaError_t launch_tile_bwd(const Params& P, cudaStream_t s);
cudaError_t launch_tile_bwd_tc(const Params& P, cudaStream_t s);
bool bwd_tc_eligible(int dclass_all);  // the backward pair contractions run on the tensor cores
int bwd_tc_cap();                      // lookups per tile of the tensor-core backward
cudaError_t set_bwd_tc_attributes(int max_smem);
cudaError_t launch_reduce13(const Params& P, cudaStream_t s);
cudaError_t launch_cache_fill(const Params& P, cudaStream_t s);
cudaError_t launch_cache_gmax(const Params& P, cudaStream_t s);
cudaError_t launch_cache_acc(const Params& P, cudaStream_t s);
cudaError_t launch_cache_apply(const Params& P, cudaStream_t s);
cudaError_t launch_full_weight(const TableDev* tables, int t, int64_t row0, int64_t nrows, float* out, cudaStream_t s);

// Update of the cores from summed gradients (tt_emb_apply_gradients): up to
// kApplySegs cores per launch; segment sg has n[sg] elements, float4 groups
// start[sg] .. start[sg + 1].
constexpr int kApplySegs = 48;
struct ApplyArgs {
    int nseg;
    int opt;
    float lr, eps;
    float* G[kApplySegs];
    const float* g[kApplySegs];
    float* s[kApplySegs];
    int* stamp[kApplySegs];        // slice stamps of an exact-copy cache (table 0), else null
    int64_t slice_elems[kApplySegs];
    int64_t n[kApplySegs];
    int64_t start[kApplySegs + 1];
    const int* dstep;
};
cudaError_t launch_apply_grads(const ApplyArgs& a, int sms, cudaStream_t s);

size_t tile_bwd_smem(const Params& P);
cudaError_t set_sort_attributes(int max_smem);
cudaError_t set_fwd_attributes(int max_smem);
cudaError_t set_bwd_attributes(int max_smem);
int bwd_batch_pairs(int q1, int Ns, int r1);
int dim_class_of(int q1, int q2, int q3, int r1, int r2);

}  // namespace ttemb
