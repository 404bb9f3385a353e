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
#include <algorithm>

#include "tt_internal.cuh"

namespace ttemb {

// ------------------------------------------------------------------ decode

// Bag offsets covering lookups lo .. hi-1 into soff: all of them when they
// fit, else offsets b0 .. b1 + 1 of the bags of lo and hi - 1.  Returns the
// number staged (sb[0] = b0), or 0 when the range does not fit (the caller
// then searches global memory).
__device__ int stage_bag_offsets(const Params& P, int64_t lo, int64_t hi, int64_t* soff, int64_t* sb, int cap) {
    if (P.nbags + 1 <= cap) {
        const int nst = (int)(P.nbags + 1);
        for (int base = 0; base < nst; base += 4 * blockDim.x) {  // 4 loads in flight per thread
            int64_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = base + u * blockDim.x + threadIdx.x;
                v[u] = i < nst ? P.off[i] : 0;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = base + u * blockDim.x + threadIdx.x;
                if (i < nst) soff[i] = v[u];
            }
        }
        if (threadIdx.x == 0) sb[0] = 0;
        __syncthreads();
        return (int)(P.nbags + 1);
    }
    if (threadIdx.x == 0) sb[0] = bag_of(P, lo);
    if (threadIdx.x == 32) sb[1] = bag_of(P, hi - 1);
    __syncthreads();
    const int64_t b0 = sb[0], nst = sb[1] - b0 + 2;
    const bool ok = nst >= 2 && nst <= cap;
    if (ok)
        for (int i = threadIdx.x; i < nst; i += blockDim.x) soff[i] = P.off[b0 + i];
    __syncthreads();
    return ok ? (int)nst : 0;
}

__device__ __forceinline__ int64_t staged_bag(const int64_t* soff, int64_t b0, int nst, int64_t n) {
    int a = 0, b = nst - 1;  // largest a < nst - 1 with soff[a] <= n
    while (b - a > 1) {
        const int m = (a + b) >> 1;
        if (soff[m] <= n) a = m; else b = m;
    }
    return b0 + a;
}


template <bool CACHE>
__global__ void __launch_bounds__(kSortThreads, 1) k_decode_hist(const __grid_constant__ Params P) {
    pdl_entry();
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(P.dstep, 1);  // the pass's cache stamp
    extern __shared__ int sm[];
    __shared__ int64_t soff[kChunk + 2];
    __shared__ int64_t sb[2];
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
        if (P.off[0] != 0 || P.off[P.nbags] != P.nnz) atomicOr(P.err, kErrOffsets);
    }
    // offsets must be non-decreasing: each block checks a slice of them
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < P.nbags;
         g += (int64_t)gridDim.x * blockDim.x)
        if (P.off[g] > P.off[g + 1]) atomicOr(P.err, kErrOffsets);
    __syncthreads();

    const int64_t lo = (int64_t)c * kChunk;
    const int64_t hi = (lo + kChunk < P.nnz) ? lo + kChunk : P.nnz;
    // this thread's indices and weights, all in flight while the chunk's bag offsets
    // are staged in shared memory (bag search there rather than in global memory)
    constexpr int kPer = kChunk / kSortThreads;
    int64_t rows[kPer];
    float wts[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int64_t n = lo + threadIdx.x + (int64_t)u * kSortThreads;
        rows[u] = n < hi ? P.idx[n] : 0;
        wts[u] = (n < hi && P.w) ? P.w[n] : 1.0f;
    }
    const int epoch = *P.epoch;
    // explicit cache rows: the first index entry of every row in flight too
    longlong2 hx[CACHE ? kPer : 1];
    const bool pre = CACHE && P.cache_sets == 0;
    if constexpr (CACHE) {
#pragma unroll
        for (int u = 0; u < kPer; ++u)
            hx[u] = pre ? __ldg(P.cache_hidx + ((unsigned)mix64((uint64_t)rows[u]) & (unsigned)P.cache_hmask))
                        : longlong2{-1, 0};
    }
    const int nst = stage_bag_offsets(P, lo, hi, soff, sb, kChunk + 2);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int64_t n = lo + threadIdx.x + (int64_t)u * kSortThreads;
        if (n >= hi) break;
        const int64_t bag = nst ? staged_bag(soff, sb[0], nst, n) : bag_of(P, n);
        int t, i1, i2, i3;
        if (!decode_lookup<CACHE>(P, n, (int)bag, rows[u], wts[u], t, i1, i2, i3, epoch, pre, hx[CACHE ? u : 0]))
            continue;
        const TableDev& T = P.tables[t];
        atomicAdd(&h1[T.base1 + i1], 1);
        atomicAdd(&h3[T.base3 + i3], 1);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < P.n1; b += blockDim.x) P.H1[(int64_t)b * P.nch + c] = h1[b];
    for (int b = threadIdx.x; b < P.n3; b += blockDim.x) P.H3[(int64_t)b * P.nch + c] = h3[b];
}

// ------------------------------------------------------------------ scans

// Exclusive scan of a[0, L) in place by one block, starting from `carry`; returns
// carry + the total.  Each thread takes kScanPer consecutive elements per round (int4
// loads; `a` is 16-byte aligned), so one block scan covers blockDim * kScanPer elements.
__device__ int scan_inplace(int* a, int64_t L, int* sh, int carry) {
    for (int64_t base = 0; base < L; base += (int64_t)blockDim.x * kScanPer) {
        const int64_t i0 = base + (int64_t)threadIdx.x * kScanPer;
        int v[kScanPer];
        if (i0 + kScanPer <= L) {
#pragma unroll
            for (int q = 0; q < kScanPer / 4; ++q) {
                const int4 x = reinterpret_cast<const int4*>(a + i0)[q];
                v[4 * q] = x.x; v[4 * q + 1] = x.y; v[4 * q + 2] = x.z; v[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < kScanPer; ++e) v[e] = i0 + e < L ? a[i0 + e] : 0;
        }
        int tot = 0;
#pragma unroll
        for (int e = 0; e < kScanPer; ++e) {
            const int x = v[e];
            v[e] = tot;
            tot += x;
        }
        int total;
        const int ex = carry + block_scan_excl(tot, sh, &total);
        if (i0 + kScanPer <= L) {
#pragma unroll
            for (int q = 0; q < kScanPer / 4; ++q)
                reinterpret_cast<int4*>(a + i0)[q] = make_int4(ex + v[4 * q], ex + v[4 * q + 1], ex + v[4 * q + 2], ex + v[4 * q + 3]);
        } else {
#pragma unroll
            for (int e = 0; e < kScanPer; ++e)
                if (i0 + e < L) a[i0 + e] = ex + v[e];
        }
        carry += total;
        __syncthreads();  // sh is reused by the next round's block scan
    }
    return carry;
}

// The [digit][chunk] histograms are scanned in segments of kScanSeg elements, a block
// per segment: W = 0 covers H1 then H3 (the sorts by i1 and i3), W = 1 covers H2.
// Block b's array, its length, the segment's index in it and the index of the
// array's first segment.
int scan_segments(const Params& P, int W, int* s1) {
    const auto segs = [](int64_t L) { return (int)std::max<int64_t>(1, (L + kScanSeg - 1) / kScanSeg); };
    const int a = segs((int64_t)(W == 0 ? P.n1 : P.n2) * P.nch);
    if (s1) *s1 = a;
    return W == 0 ? a + segs((int64_t)P.n3 * P.nch) : a;
}

template <int W>
__device__ __forceinline__ void scan_segment_of(const Params& P, int b, int*& a, int64_t& L, int& seg, int& base) {
    const int64_t L1 = (int64_t)(W == 0 ? P.n1 : P.n2) * P.nch;
    const int s1 = (int)((L1 + kScanSeg - 1) / kScanSeg);
    if (W == 1 || b < (s1 > 0 ? s1 : 1)) {
        a = W == 0 ? P.H1 : P.H2;
        L = L1;
        seg = b;
        base = 0;
    } else {
        a = P.H3;
        L = (int64_t)P.n3 * P.nch;
        seg = b - (s1 > 0 ? s1 : 1);
        base = s1 > 0 ? s1 : 1;
    }
}

// Pass 1 (only when some array has several segments): each block's segment total
// into segsum.
template <int W>
__global__ void __launch_bounds__(kScanThreads) k_scan_sums(const __grid_constant__ Params P) {
    pdl_entry();
    __shared__ int sh[33];
    int* a;
    int64_t L;
    int seg, base;
    scan_segment_of<W>(P, blockIdx.x, a, L, seg, base);
    const int64_t lo = (int64_t)seg * kScanSeg, hi = lo + kScanSeg < L ? lo + kScanSeg : L;
    int sum = 0;
    for (int64_t i = lo + threadIdx.x; i < hi; i += blockDim.x) sum += a[i];
    int total;
    block_scan_excl(sum, sh, &total);
    if (threadIdx.x == 0) P.segsum[blockIdx.x] = total;
}

// Pass 2: each block scans its segment from the sum of the earlier segments of its
// array.  W = 0: the block with H1's last segment stores the count of lookups in the
// sorted orders.  W = 1: the last block to finish (a counter, no waiting) cuts each
// (table, i2) group of `cnt` lookups (contiguous in pi21) into ceil(cnt / tile_cap)
// tiles.
template <int W>
__global__ void __launch_bounds__(kScanThreads) k_scan_apply(const __grid_constant__ Params P) {
    pdl_entry();
    __shared__ int sh[33];
    __shared__ int last;
    int* a;
    int64_t L;
    int seg, base;
    scan_segment_of<W>(P, blockIdx.x, a, L, seg, base);
    int part = 0;
    for (int k = threadIdx.x; k < seg; k += blockDim.x) part += P.segsum[base + k];
    int offset;
    block_scan_excl(part, sh, &offset);
    __syncthreads();
    const int64_t lo = (int64_t)seg * kScanSeg;
    const int64_t n = lo < L ? (lo + kScanSeg < L ? kScanSeg : L - lo) : 0;
    const int end = scan_inplace(a + lo, n, sh, offset);
    if (W == 0) {
        if (a == P.H1 && lo + kScanSeg >= L && threadIdx.x == 0) *P.nincl = end;
        return;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        last = atomicAdd(P.scan_done, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    int carry = 0, mcarry = 0;
    for (int gb = 0; gb < P.n2; gb += blockDim.x) {
        const int g = gb + threadIdx.x;
        int start = 0, cnt = 0, nt = 0;
        if (g < P.n2) {
            start = __ldcg(P.H2 + (int64_t)g * P.nch);
            const int e = (g + 1 < P.n2) ? __ldcg(P.H2 + (int64_t)(g + 1) * P.nch) : *P.nincl;
            cnt = e - start;
            nt = (cnt + P.tile_cap - 1) / P.tile_cap;
        }
        int total, mtot;
        const int first = carry + block_scan_excl(nt, sh, &total);
        __syncthreads();
        const int mpos = mcarry + block_scan_excl(nt > 1 ? 1 : 0, sh, &mtot);
        if (g < P.n2) {
            P.grp_first[g] = first;
            P.grp_ntiles[g] = nt;
            for (int k = 0; k < nt; ++k)
                P.tiles[first + k] = make_int4(start + k * P.tile_cap, min(P.tile_cap, cnt - k * P.tile_cap), g, k);
            if (nt > 1) P.multi_groups[mpos] = g;
        }
        carry += total;
        mcarry += mtot;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *P.ntiles = carry;
        *P.multi_count = mcarry;
        *P.scan_done = 0;  // ready for the next pass
    }
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

__global__ void __launch_bounds__(kSortThreads, 1) k_scatter13(const __grid_constant__ Params P) {
    pdl_entry();
    extern __shared__ int cnt[];
    const int c = blockIdx.x;
    // by i1 -> pi1, and the i2 histogram of pi1 chunks
    chunk_stable_ranks(
        c, P.nnz, P.n1, cnt,
        [&](int64_t n) { return excluded(P, n) ? -1 : P.tables[table_of_bag(P, P.lk_bag[n])].base1 + P.lk_i1[n]; },
        [&](int64_t n, int d, int rank) {
            const int pos = TT_DCHECK(P, P.H1[(int64_t)d * P.nch + c] + rank, P.nnz);
            P.pi1[pos] = (int)n;
            const int d2 = P.tables[table_of_bag(P, P.lk_bag[n])].base2 + P.lk_i2[n];
            atomicAdd(&P.H2[(int64_t)d2 * P.nch + pos / kChunk], 1);
        });
    // by i3 -> pi3
    chunk_stable_ranks(
        c, P.nnz, P.n3, cnt,
        [&](int64_t n) { return excluded(P, n) ? -1 : P.tables[table_of_bag(P, P.lk_bag[n])].base3 + P.lk_i3[n]; },
        [&](int64_t n, int d, int rank) {
            const int pos = TT_DCHECK(P, P.H3[(int64_t)d * P.nch + c] + rank, P.nnz);
            P.pi3[pos] = (int)n;
            P.inv3[n] = pos;
        });
}

__global__ void __launch_bounds__(kSortThreads, 1) k_scatter2(const __grid_constant__ Params P) {
    pdl_entry();
    extern __shared__ int cnt[];
    const int c = blockIdx.x;
    const int nincl = *P.nincl;  // positions of the i1 order in use
    chunk_stable_ranks(
        c, P.nnz, P.n2, cnt,
        [&](int64_t k) {
            if (k >= nincl) return -1;
            const int n = P.pi1[k];
            return P.tables[table_of_bag(P, P.lk_bag[n])].base2 + P.lk_i2[n];
        },
        [&](int64_t k, int d, int rank) {
            const int n = TT_DCHECK(P, P.pi1[k], P.nnz), pos = TT_DCHECK(P, P.H2[(int64_t)d * P.nch + c] + rank, P.nnz);
            P.pi21[pos] = n;
            P.g_i1[pos] = P.lk_i1[n];
            P.g_i3[pos] = P.lk_i3[n];
            P.g_bag[pos] = P.lk_bag[n];
            P.g_s[pos] = P.lk_s[n];
            P.g_p1[pos] = (int)k;
            P.g_p3[pos] = P.inv3[n];
        });
}

// ------------------------------------------------------------------ small path
//
// For nnz <= kSmallMaxNnz the three stable counting sorts (by i1, i2 and i3,
// each over original order) run with chunks of kSmallChunk lookups:
//   k_decode_small  one block per chunk: decode, and for every digit the
//                   chunk histogram and each lookup's stable rank among the
//                   chunk's lookups with the same digit
//   scan_digit_block  one block per digit: exclusive scan of [bin][chunk]; the
//                   i2 block also cuts the (table, i2) groups into tiles (run by
//                   three extra blocks of the k_fwd_T launch)
//   scatter_chunk   position = scanned base + rank (run by extra blocks of the
//                   k_pool launch)

template <bool CACHE>
__global__ void __launch_bounds__(kSmallChunk) k_decode_small(const __grid_constant__ Params P) {
    pdl_entry();
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(P.dstep, 1);  // the pass's cache stamp
    __shared__ int64_t soff[kDecodeOffs];
    __shared__ int64_t sb[2];
    __shared__ int cnt[kSmallChunk / 32][kSmallMaxBins];
    const int c = blockIdx.x;
    const int64_t lo = (int64_t)c * kSmallChunk;
    const int64_t hi = (lo + kSmallChunk < P.nnz) ? lo + kSmallChunk : P.nnz;
    // this thread's index, weight and the epoch: in flight while the offsets are checked and staged
    const int64_t n = lo + threadIdx.x;
    const int64_t row = n < hi ? P.idx[n] : 0;
    const float wv = (n < hi && P.w) ? P.w[n] : 1.0f;
    const int epoch = *P.epoch;
    if (threadIdx.x == 0) asm volatile("prefetch.global.L1 [%0];" ::"l"(P.tables));  // the decode reads it next
    const int nst = stage_bag_offsets(P, lo, hi, soff, sb, kDecodeOffs);
    if (nst == P.nbags + 1) {  // every offset staged: block 0 checks them in shared memory
        if (c == 0) {
            if (threadIdx.x == 64 && (soff[0] != 0 || soff[P.nbags] != P.nnz)) atomicOr(P.err, kErrOffsets);
            for (int64_t g = threadIdx.x; g < P.nbags; g += blockDim.x)
                if (soff[g] > soff[g + 1]) atomicOr(P.err, kErrOffsets);
        }
    } else {
        if (c == 0 && threadIdx.x == 64 && (P.off[0] != 0 || P.off[P.nbags] != P.nnz)) atomicOr(P.err, kErrOffsets);
        for (int64_t g = (int64_t)c * blockDim.x + threadIdx.x; g < P.nbags; g += (int64_t)gridDim.x * blockDim.x)
            if (P.off[g] > P.off[g + 1]) atomicOr(P.err, kErrOffsets);
    }
    int d[3] = {-1, -1, -1};
    if (n < hi) {
        const int64_t bag = nst ? staged_bag(soff, sb[0], nst, n) : bag_of(P, n);
        int t, i1, i2, i3;
        if (decode_lookup<CACHE>(P, n, (int)bag, row, wv, t, i1, i2, i3, epoch)) {
            const TableDev& T = P.tables[t];
            d[0] = T.base1 + i1;
            d[1] = T.base2 + i2;
            d[2] = T.base3 + i3;
        }
    }
    // the touched flags of this block's lookups are stored: stamp the pass's epoch for the
    // k_fwd_T blocks waiting on them
    static_assert(kScanChunkMax <= kDecDoneSlots, "a decode stamp per block");
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) atomicExch(P.dec_done + c, epoch);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nbs[3] = {P.n1, P.n2, P.n3};
    int* Hs[3] = {P.H1, P.H2, P.H3};
    uint16_t* lrs[3] = {P.lr1, P.lr2, P.lr3};
#pragma unroll
    for (int k = 0; k < 3; ++k) {
        const int nb = nbs[k];
        for (int e = threadIdx.x; e < (kSmallChunk / 32) * nb; e += blockDim.x) cnt[e / nb][e % nb] = 0;
        __syncthreads();
        const unsigned m = __match_any_sync(0xffffffffu, d[k]);
        if (d[k] >= 0 && lane == __ffs(m) - 1) cnt[w][d[k]] = __popc(m);
        __syncthreads();
        for (int b = threadIdx.x; b < nb; b += blockDim.x) {
            int run = 0;
#pragma unroll
            for (int ww = 0; ww < kSmallChunk / 32; ++ww) {
                const int v = cnt[ww][b];
                cnt[ww][b] = run;
                run += v;
            }
            Hs[k][(int64_t)b * P.nch + c] = run;
        }
        __syncthreads();
        if (d[k] >= 0) lrs[k][n] = (uint16_t)(cnt[w][d[k]] + __popc(m & lanemask_lt()));
        __syncthreads();
    }
}

// ------------------------------------------------------------------ launchers

cudaError_t launch_decode_small(const Params& P, cudaStream_t s) {
    cudaError_t le = P.cache_n > 0 ? launch_pdl(k_decode_small<true>, dim3((unsigned)P.nch), dim3(kSmallChunk), 0, s, P)
                                   : launch_pdl(k_decode_small<false>, dim3((unsigned)P.nch), dim3(kSmallChunk), 0, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t launch_decode_hist(const Params& P, cudaStream_t s) {
    const size_t smem = sizeof(int) * (size_t)(P.n1 + P.n3);
    cudaError_t le = P.cache_n > 0 ? launch_pdl(k_decode_hist<true>, dim3(P.nch), dim3(kSortThreads), smem, s, P)
                                   : launch_pdl(k_decode_hist<false>, dim3(P.nch), dim3(kSortThreads), smem, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t launch_scan_sums13(const Params& P, cudaStream_t s) {
    cudaError_t le = launch_pdl(k_scan_sums<0>, dim3(scan_segments(P, 0)), dim3(kScanThreads), 0, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t launch_scan13(const Params& P, cudaStream_t s) {
    cudaError_t le = launch_pdl(k_scan_apply<0>, dim3(scan_segments(P, 0)), dim3(kScanThreads), 0, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t launch_scan_sums2(const Params& P, cudaStream_t s) {
    cudaError_t le = launch_pdl(k_scan_sums<1>, dim3(scan_segments(P, 1)), dim3(kScanThreads), 0, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t launch_scatter13(const Params& P, cudaStream_t s) {
    const size_t smem = sizeof(int) * kSortWarps * (size_t)max(P.n1, P.n3);
    cudaError_t le = launch_pdl(k_scatter13, dim3(P.nch), dim3(kSortThreads), smem, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t launch_scan2_tiles(const Params& P, cudaStream_t s) {
    cudaError_t le = launch_pdl(k_scan_apply<1>, dim3(scan_segments(P, 1)), dim3(kScanThreads), 0, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t launch_scatter2(const Params& P, cudaStream_t s) {
    const size_t smem = sizeof(int) * kSortWarps * (size_t)P.n2;
    cudaError_t le = launch_pdl(k_scatter2, dim3(P.nch), dim3(kSortThreads), smem, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t set_sort_attributes(int max_smem) {
    const void* ks[] = {(const void*)k_decode_hist<false>, (const void*)k_decode_hist<true>,
                        (const void*)k_scatter13, (const void*)k_scatter2,
                        (const void*)k_decode_small<false>, (const void*)k_decode_small<true>, (const void*)k_scan_sums<0>, (const void*)k_scan_sums<1>,
                        (const void*)k_scan_apply<0>, (const void*)k_scan_apply<1>};
    for (const void* k : ks) {
        cudaError_t e = allow_max_dynamic_smem(k, max_smem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace ttemb
