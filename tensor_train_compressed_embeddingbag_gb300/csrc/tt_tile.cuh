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
        p1 = P.g_p1[start + k];
        p3 = P.g_p3[start + k];
        i1 = P.g_i1[start + k];
        i3 = P.g_i3[start + k];
        bag = P.g_bag[start + k];
        sc = P.g_s[start + k];
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

}  // namespace ttemb
