// tt_sort.cu -- decode and grouping of the lookups (sm_103a).
//
// Lookups are grouped so that those sharing core slices are adjacent (the
// tensorflow/addons EmbeddingBag issue: the gradient is formed by sorting by
// key, so that no two threads write the same entry).  Three stable counting
// sorts are built from one decode pass:
//   pi1  by (table, i1, position)   -> segments for the dG1 reduction
//   pi3  by (table, i3, position)   -> segments for the dG3 reduction
//   pi21 by (table, i2, i1, position), an LSD pass by i2 over pi1 order
// A counting sort over a chunk of kChunk lookups computes each lookup's rank
// among the chunk's lookups with the same digit with warp match masks and a
// per-warp count table, so the scatter is stable without atomics on the
// output positions.
#include "tt_internal.cuh"

namespace ttemb {

// ------------------------------------------------------------------ decode

__global__ void __launch_bounds__(kSortThreads) k_decode_hist(const __grid_constant__ Params P) {
    extern __shared__ int sm[];
    int* h1 = sm;           // [n1]
    int* h3 = sm + P.n1;    // [n3]
    const int c = blockIdx.x;
    for (int b = threadIdx.x; b < P.n1 + P.n3; b += blockDim.x) sm[b] = 0;
    // H2 is filled with atomics by k_scatter13; clear it here.
    {
        const int64_t total = (int64_t)P.n2 * P.nch;
        for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
             e += (int64_t)gridDim.x * blockDim.x)
            P.H2[e] = 0;
    }
    if (c == 0 && threadIdx.x == 0) {
        P.counters[0] = 0;
        P.counters[1] = 0;
        if (P.off[0] != 0 || P.off[P.nbags] != P.nnz) atomicOr(P.err, kErrOffsets);
    }
    // offsets must be non-decreasing: each block checks a slice of them
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < P.nbags;
         g += (int64_t)gridDim.x * blockDim.x)
        if (P.off[g] > P.off[g + 1]) atomicOr(P.err, kErrOffsets);
    __syncthreads();

    const int64_t lo = (int64_t)c * kChunk;
    const int64_t hi = (lo + kChunk < P.nnz) ? lo + kChunk : P.nnz;
    for (int64_t n = lo + threadIdx.x; n < hi; n += blockDim.x) {
        // bag = largest g with off[g] <= n
        int64_t a = 0, b = P.nbags;  // invariant: off[a] <= n (if offsets are valid), answer in [a, b)
        while (b - a > 1) {
            int64_t m = (a + b) >> 1;
            if (P.off[m] <= n) a = m; else b = m;
        }
        const int bag = (int)a;
        const int t = table_of_bag(P, bag);
        const TableDev& T = P.tables[t];
        int64_t row = P.idx[n];
        float s = P.w ? P.w[n] : 1.0f;
        if (row < 0 || row >= T.E) {
            atomicOr(P.err, kErrIndex);
            row = 0;
            s = 0.0f;
        }
        if (P.mean) {
            const int64_t L = P.off[bag + 1] - P.off[bag];
            s = s / (float)(L > 0 ? L : 1);
        }
        const int64_t p23 = (int64_t)T.p2 * T.p3;
        const int i1 = (int)(row / p23);
        const int i2 = (int)((row / T.p3) % T.p2);
        const int i3 = (int)(row % T.p3);
        P.lk_i1[n] = i1;
        P.lk_i2[n] = i2;
        P.lk_i3[n] = i3;
        P.lk_bag[n] = bag;
        P.lk_s[n] = s;
        atomicAdd(&h1[T.base1 + i1], 1);
        atomicAdd(&h3[T.base3 + i3], 1);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < P.n1; b += blockDim.x) P.H1[(int64_t)b * P.nch + c] = h1[b];
    for (int b = threadIdx.x; b < P.n3; b += blockDim.x) P.H3[(int64_t)b * P.nch + c] = h3[b];
}

// ------------------------------------------------------------------ scans

__device__ void scan_inplace(int* a, int64_t L, int* sh) {
    int carry = 0;
    for (int64_t base = 0; base < L; base += blockDim.x) {
        const int64_t i = base + threadIdx.x;
        const int v = i < L ? a[i] : 0;
        int total;
        const int ex = block_scan_excl(v, sh, &total);
        if (i < L) a[i] = carry + ex;
        carry += total;
    }
}

__global__ void __launch_bounds__(kScanThreads) k_scan13(const __grid_constant__ Params P) {
    __shared__ int sh[33];
    scan_inplace(P.H1, (int64_t)P.n1 * P.nch, sh);
    scan_inplace(P.H3, (int64_t)P.n3 * P.nch, sh);
}

// Exclusive scan of H2, then the tiles: each (table, i2) group of `cnt`
// lookups (contiguous in pi21) is cut into ceil(cnt / tile_cap) tiles.
__global__ void __launch_bounds__(kScanThreads) k_scan2_tiles(const __grid_constant__ Params P) {
    __shared__ int sh[33];
    scan_inplace(P.H2, (int64_t)P.n2 * P.nch, sh);
    __syncthreads();
    int carry = 0;
    for (int base = 0; base < P.n2; base += blockDim.x) {
        const int g = base + threadIdx.x;
        int start = 0, cnt = 0, nt = 0;
        if (g < P.n2) {
            start = P.H2[(int64_t)g * P.nch];
            const int end = (g + 1 < P.n2) ? P.H2[(int64_t)(g + 1) * P.nch] : (int)P.nnz;
            cnt = end - start;
            nt = (cnt + P.tile_cap - 1) / P.tile_cap;
        }
        int total;
        const int first = carry + block_scan_excl(nt, sh, &total);
        if (g < P.n2) {
            P.grp_first[g] = first;
            P.grp_ntiles[g] = nt;
            for (int k = 0; k < nt; ++k)
                P.tiles[first + k] = make_int4(start + k * P.tile_cap, min(P.tile_cap, cnt - k * P.tile_cap), g, k);
        }
        carry += total;
    }
    if (threadIdx.x == 0) *P.ntiles = carry;
}

// ------------------------------------------------------------------ scatters

// Stable rank of every lookup of this chunk among the chunk's lookups with the
// same digit; calls emit(n, digit, rank) for each.  cnt is [kSortWarps][nb].
template <class DigitFn, class EmitFn>
__device__ void chunk_stable_ranks(int c, int64_t count, int nb, int* cnt, DigitFn digit_of, EmitFn emit) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int e = threadIdx.x; e < kSortWarps * nb; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    int* mine = cnt + w * nb;
    const int64_t lo = (int64_t)c * kChunk + (int64_t)w * kWarpSpan;
    const int64_t hi = (lo + kWarpSpan < count) ? lo + kWarpSpan : count;
    // pass 1: per-warp counts
    for (int64_t s = lo; s < hi; s += 32) {
        const int64_t k = s + lane;
        const int d = k < hi ? digit_of(k) : -1;
        const unsigned m = __match_any_sync(0xffffffffu, d);
        if (d >= 0 && lane == __ffs(m) - 1) mine[d] += __popc(m);
    }
    __syncthreads();
    // exclusive prefix over warps, per bin
    for (int b = threadIdx.x; b < nb; b += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int ww = 0; ww < kSortWarps; ++ww) {
            const int v = cnt[ww * nb + b];
            cnt[ww * nb + b] = run;
            run += v;
        }
    }
    __syncthreads();
    // pass 2: ranks
    for (int64_t s = lo; s < hi; s += 32) {
        const int64_t k = s + lane;
        const int d = k < hi ? digit_of(k) : -1;
        const unsigned m = __match_any_sync(0xffffffffu, d);
        const int leader = __ffs(m) - 1;
        int base = 0;
        if (d >= 0 && lane == leader) {
            base = mine[d];
            mine[d] = base + __popc(m);
        }
        base = __shfl_sync(0xffffffffu, base, leader);
        if (d >= 0) emit(k, d, base + __popc(m & lanemask_lt()));
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kSortThreads) k_scatter13(const __grid_constant__ Params P) {
    extern __shared__ int cnt[];
    const int c = blockIdx.x;
    // by i1 -> pi1, and the i2 histogram of pi1 chunks
    chunk_stable_ranks(
        c, P.nnz, P.n1, cnt,
        [&](int64_t n) { return P.tables[table_of_bag(P, P.lk_bag[n])].base1 + P.lk_i1[n]; },
        [&](int64_t n, int d, int rank) {
            const int pos = P.H1[(int64_t)d * P.nch + c] + rank;
            P.pi1[pos] = (int)n;
            const int d2 = P.tables[table_of_bag(P, P.lk_bag[n])].base2 + P.lk_i2[n];
            atomicAdd(&P.H2[(int64_t)d2 * P.nch + pos / kChunk], 1);
        });
    // by i3 -> pi3
    chunk_stable_ranks(
        c, P.nnz, P.n3, cnt,
        [&](int64_t n) { return P.tables[table_of_bag(P, P.lk_bag[n])].base3 + P.lk_i3[n]; },
        [&](int64_t n, int d, int rank) { P.pi3[P.H3[(int64_t)d * P.nch + c] + rank] = (int)n; });
}

__global__ void __launch_bounds__(kSortThreads) k_scatter2(const __grid_constant__ Params P) {
    extern __shared__ int cnt[];
    const int c = blockIdx.x;
    chunk_stable_ranks(
        c, P.nnz, P.n2, cnt,
        [&](int64_t k) {
            const int n = P.pi1[k];
            return P.tables[table_of_bag(P, P.lk_bag[n])].base2 + P.lk_i2[n];
        },
        [&](int64_t k, int d, int rank) { P.pi21[P.H2[(int64_t)d * P.nch + c] + rank] = P.pi1[k]; });
}

// ------------------------------------------------------------------ launchers

cudaError_t launch_decode_hist(const Params& P, cudaStream_t s) {
    const size_t smem = sizeof(int) * (size_t)(P.n1 + P.n3);
    cudaError_t e = cudaFuncSetAttribute(k_decode_hist, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_decode_hist<<<P.nch, kSortThreads, smem, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_scan13(const Params& P, cudaStream_t s) {
    k_scan13<<<1, kScanThreads, 0, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_scatter13(const Params& P, cudaStream_t s) {
    const size_t smem = sizeof(int) * kSortWarps * (size_t)max(P.n1, P.n3);
    cudaError_t e = cudaFuncSetAttribute(k_scatter13, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_scatter13<<<P.nch, kSortThreads, smem, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_scan2_tiles(const Params& P, cudaStream_t s) {
    k_scan2_tiles<<<1, kScanThreads, 0, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_scatter2(const Params& P, cudaStream_t s) {
    const size_t smem = sizeof(int) * kSortWarps * (size_t)P.n2;
    cudaError_t e = cudaFuncSetAttribute(k_scatter2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_scatter2<<<P.nch, kSortThreads, smem, s>>>(P);
    return cudaGetLastError();
}

}  // namespace ttemb
