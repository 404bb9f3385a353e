// tt_internal.cuh -- shared definitions of the TT-EmbeddingBag CUDA library (sm_103a).
//
// The forward pass of one call runs these kernels, in stream order:
//   k_decode_hist   decode i -> (i1,i2,i3), bag id and pooling scale per lookup,
//                   per-chunk histograms of the i1 and i3 digits
//   k_scan13        exclusive scans of those histograms (bin-major)
//   k_scatter13     stable counting-sort scatter by i1 (pi1) and by i3 (pi3);
//                   per-chunk histogram of i2 over pi1 order
//   k_scan2_tiles   exclusive scan of the i2 histogram; tiles of <= tile_cap
//                   lookups inside each (table, i2) group
//   k_scatter2      stable scatter of pi1 by i2: pi21, ordered by (table, i2, i1, position)
//   k_tile_fwd      per tile: local sort by (i1, i3, position) -> sigma; partial
//                   products T = G1[i1] G2[i2] once per (i1, i2) pair -> Tbuf
//   k_pool          per bag: row = T G3[i3], pooled in registers -> out
// and the backward pass:
//   k_tile_bwd      per tile: summed upstream gradient per row, dG3 partial per
//                   row, dT per pair, dG1 partial per pair, dG2 of the group
//                   (reduced across the group's tiles by the last tile, which
//                   applies the G2 update)
//   k_reduce13      per i1 / i3 slice: sum of the partials in sorted segment
//                   order, G1 / G3 update
// Every sum runs in an order fixed by the sort keys, so results are
// bitwise reproducible; no floating-point atomics are used.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ttemb {

constexpr int kChunk = 2048;        // lookups per counting-sort chunk
constexpr int kSortThreads = 256;   // 8 warps; each warp owns kChunk/8 consecutive lookups
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kWarpSpan = kChunk / kSortWarps;
constexpr int kScanThreads = 1024;
constexpr int kTileThreads = 256;
constexpr int kMaxBinsPerDigit = 6144;  // per-warp rank tables: 8 x bins x 4 B of shared memory
constexpr int kFieldBits = 20;          // bits per field of the in-tile sort key

enum ErrBits { kErrIndex = 1, kErrOffsets = 2, kErrTimeout = 4 };

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
    int base1, base2, base3;  // first global bin of each digit
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
    int nch;                        // chunks of kChunk lookups
    int max_tiles;
    // workspace
    int* lk_i1;
    int* lk_i2;
    int* lk_i3;
    int* lk_bag;
    float* lk_s;
    int* H1;                        // [n1][nch]
    int* H3;                        // [n3][nch]
    int* H2;                        // [n2][nch]
    int* pi1;
    int* pi3;
    int* pi21;
    int* sigma;
    int4* tiles;                    // {start, len, group bin, tile index in group}
    int* ntiles;
    int* grp_first;                 // [n2]
    int* grp_ntiles;                // [n2]
    int* grp_done;                  // [n2], zero between calls
    float* Tbuf;
    int* rep_pair;                  // [nnz] slot of the tile-pair starting at this lookup, or -1
    int* rep_row;                   // [nnz] slot of the tile-row starting at this lookup, or -1
    float* Qbuf;                    // [nnz][qs_max]
    float* Pbuf;                    // [nnz][ps_max]
    float* dG2part;                 // [max_tiles][s2_max]
    int* counters;                  // [0] tile-row slots, [1] tile-pair slots
    int* err;
    // hot-row cache (single table)
    const int64_t* cache_rows;      // sorted row ids, or null
    int64_t cache_n;
    float* cache_vals;              // [cache_n][D]
    int* cache_stamp;               // [cache_n] step at which the row was computed
    int* slice_stamp;               // [p1 + p2 + p3] step at which each slice last changed
    int step;
};

// ---------------------------------------------------------------- helpers

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

// Ascending bitonic sort of n (power of two) keys in shared memory.
__device__ __forceinline__ void block_bitonic_sort(unsigned long long* keys, int n) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            __syncthreads();
            for (int i = threadIdx.x; i < (n >> 1); i += blockDim.x) {
                int lo = 2 * i - (i & (stride - 1));
                int hi = lo + stride;
                bool asc = (lo & size) == 0;
                unsigned long long a = keys[lo], b = keys[hi];
                if ((a > b) == asc) {
                    keys[lo] = b;
                    keys[hi] = a;
                }
            }
        }
    }
    __syncthreads();
}

__device__ __forceinline__ int table_of_bag(const Params& P, int bag) {
    return P.ntab == 1 ? 0 : (int)(bag / P.bags_per_table);
}

// ---------------------------------------------------------------- launchers
// Each returns the cudaError_t of its launch.
cudaError_t launch_decode_hist(const Params& P, cudaStream_t s);
cudaError_t launch_scan13(const Params& P, cudaStream_t s);
cudaError_t launch_scatter13(const Params& P, cudaStream_t s);
cudaError_t launch_scan2_tiles(const Params& P, cudaStream_t s);
cudaError_t launch_scatter2(const Params& P, cudaStream_t s);
cudaError_t launch_tile_fwd(const Params& P, cudaStream_t s);
cudaError_t launch_pool(const Params& P, cudaStream_t s);
cudaError_t launch_tile_bwd(const Params& P, cudaStream_t s);
cudaError_t launch_reduce13(const Params& P, cudaStream_t s);
cudaError_t launch_cache_fill(const Params& P, cudaStream_t s);

size_t tile_fwd_smem(const Params& P);
size_t tile_bwd_smem(const Params& P);

}  // namespace ttemb
