// tt_tile.cuh -- the backward tile's lookups, shared by the FFMA and the
// tensor-core backward kernels.
//
// A tile is a run of at most tile_cap lookups of one (table, i2) group in the
// grouped order.  Sorted in shared memory by (i1, i3, position), its maximal
// runs of equal (i1, i3) are the tile's rows and its maximal runs of equal i1
// its pairs (tensorflow/addons EmbeddingBag issue: gradients are formed after
// sorting by key, so that no two threads write one entry).
#pragma once

#include "tt_internal.cuh"

namespace ttemb {

// The tile's lookups come grouped by (table, i2) (ordered by (i1, pos) on the
// multi-CTA path, by pos on the small path); sort them by (i1, i3, position) in
// shared memory.  Bag and scale of each lookup are read in the same pass (from
// the grouped-order copies the scatter wrote) and follow the sort.
__device__ __forceinline__ void load_and_sort_tile(const Params& P, int start, int len, unsigned long long* keys, int* sp1,
                                   int* sp3, int* si1, int* si3, int* sbag, float* ss) {
    // len <= blockDim: thread k holds lookup k of the tile.  The keys (i1, i3, k) are
    // distinct, so a key's rank is the number of smaller keys: every thread counts its
    // own with broadcast shared-memory reads and writes its lookup at that rank.
    const int k = threadIdx.x;
    unsigned long long key = ~0ull;
    int p1 = 0, p3 = 0, i1 = 0, i3 = 0, bag = 0;
    float sc = 0.f;
    if (k < len) {  // grouped-order copies: one coalesced pass, no dependent loads
        const int64_t at = TT_DCHECK(P, (int64_t)start + k, P.nnz);
        p1 = TT_DCHECK(P, P.g_p1[at], P.nnz);
        p3 = TT_DCHECK(P, P.g_p3[at], P.nnz);
        i1 = P.g_i1[at];
        i3 = P.g_i3[at];
        bag = TT_DCHECK(P, P.g_bag[at], P.nbags);
        sc = P.g_s[at];
        key = ((unsigned long long)i1 << (2 * kFieldBits)) | ((unsigned long long)i3 << kFieldBits) | (unsigned long long)k;
        keys[k] = key;
    }
    __syncthreads();
    if (k < len) {
        int r = 0;
        for (int j = 0; j < len; ++j) r += keys[j] < key ? 1 : 0;
        sp1[r] = p1;
        sp3[r] = p3;
        si1[r] = i1;
        si3[r] = i3;
        sbag[r] = bag;
        ss[r] = sc;
    }
    __syncthreads();
}

// Summed upstream gradient of every tile-row: gs[row] = sum over the row's lookups k
// (a run of the sorted tile) of s_k grad_out[bag_k], D floats (D % 4 == 0).  First
// every lookup's scaled gradient row goes to gs at the lookup's position (all loads in
// flight at once: a hot row of many lookups is not a chain of dependent loads), then
// each row's run is summed from shared memory, blockDim items (row, 4 columns) a
// round, and written at the row's position.  A row's position is at most that of its
// first lookup, so a round overwrites only positions that no later round reads.
// Ends with the block synchronised; gs holds nrows rows.
__device__ __forceinline__ void tile_gs(const Params& P, int len, int nrows, const int* sbag, const float* ss,
                                        const int* rowbeg, float* gs, int D) {
    const int D4 = D >> 2;
    float4* g4 = reinterpret_cast<float4*>(gs);
    const int n1 = len * D4;
    for (int e0 = threadIdx.x; e0 < n1; e0 += 4 * blockDim.x) {
        float4 x[4];
        float sc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * blockDim.x;
            x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            sc[u] = 0.f;
            if (e < n1) {
                const int k = e / D4, q = e - k * D4;
                sc[u] = ss[k];
                x[u] = __ldg(reinterpret_cast<const float4*>(P.grad_out + (int64_t)sbag[k] * D) + q);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * blockDim.x;
            if (e < n1) g4[e] = make_float4(sc[u] * x[u].x, sc[u] * x[u].y, sc[u] * x[u].z, sc[u] * x[u].w);
        }
    }
    __syncthreads();
    const int n2 = nrows * D4;
    for (int base = 0; base < n2; base += blockDim.x) {  // uniform trip count
        const int e = base + threadIdx.x;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < n2) {
            const int row = e / D4, q = e - row * D4;
            const int kb = rowbeg[row], ke = rowbeg[row + 1];
            a = g4[kb * D4 + q];
            for (int k = kb + 1; k < ke; ++k) {
                const float4 y = g4[k * D4 + q];
                a.x += y.x; a.y += y.y; a.z += y.z; a.w += y.w;
            }
        }
        __syncthreads();
        if (e < n2) g4[e] = a;
    }
    __syncthreads();
}

// tile_gs in two halves for tiles whose len D / 4 float4 items fit four a thread: the
// loads of every lookup's gradient row are issued early (right after the tile sort) and
// land while the block does other work; tile_gs_rows then stores and sums them.
struct GsLoads {
    float4 x[4];
    float sc[4];
};
__device__ __forceinline__ void tile_gs_issue(const Params& P, int len, const int* sbag, const float* ss, int D,
                                              GsLoads& g) {
    const int D4 = D >> 2, n1 = len * D4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = threadIdx.x + u * blockDim.x;
        g.x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        g.sc[u] = 0.f;
        if (e < n1) {
            const int k = e / D4, q = e - k * D4;
            g.sc[u] = ss[k];
            g.x[u] = __ldg(reinterpret_cast<const float4*>(P.grad_out + (int64_t)sbag[k] * D) + q);
        }
    }
}
__device__ __forceinline__ void tile_gs_rows(const GsLoads& g, int len, int nrows, const int* rowbeg, float* gs, int D) {
    const int D4 = D >> 2, n1 = len * D4;
    float4* g4 = reinterpret_cast<float4*>(gs);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = threadIdx.x + u * blockDim.x;
        if (e < n1) g4[e] = make_float4(g.sc[u] * g.x[u].x, g.sc[u] * g.x[u].y, g.sc[u] * g.x[u].z, g.sc[u] * g.x[u].w);
    }
    __syncthreads();
    const int n2 = nrows * D4;
    for (int base = 0; base < n2; base += blockDim.x) {  // uniform trip count
        const int e = base + threadIdx.x;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < n2) {
            const int row = e / D4, q = e - row * D4;
            const int kb = rowbeg[row], ke = rowbeg[row + 1];
            a = g4[kb * D4 + q];
            for (int k = kb + 1; k < ke; ++k) {
                const float4 y = g4[k * D4 + q];
                a.x += y.x; a.y += y.y; a.z += y.z; a.w += y.w;
            }
        }
        __syncthreads();
        if (e < n2) g4[e] = a;
    }
    __syncthreads();
}

}  // namespace ttemb
