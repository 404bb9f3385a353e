// tt_compute.cu -- contractions, pooling and the fused SGD update (sm_103a).
//
// Notation (TT-Rec / FBTT-Embedding pages, FBTT README "Software Cache": a row
// is two consecutive small matrix products, and the core gradients are a chain
// of products in reversed order):
//   T  = G1[i1] (q1 x r1) . G2[i2] (r1 x q2 r2)            per (i1, i2) pair
//   row = T (q1 q2 x r2) . G3[i3] (r2 x q3)                per lookup
//   g   = s_n grad_out[bag]           (q1 q2 x q3)         per lookup
//   gs  = sum of g over the lookups of one row (i1, i2, i3) inside a tile
//   dG3[i3] += T^T gs                 (r2 x q3)            per tile-row
//   dT      = sum_rows gs . G3[i3]^T  (q1 x q2 r2)         per tile-pair
//   dG1[i1] += dT . G2[i2]^T          (q1 x r1)            per tile-pair
//   dG2[i2] += G1[i1]^T . dT          (r1 x q2 r2)         per tile-pair
// N = q2 r2 is the width of one G2 slice row.
#include "tt_internal.cuh"

namespace ttemb {

constexpr int kMaxAcc2 = 64;   // dG2 accumulators per thread: r1 q2 r2 <= 64 * 256
constexpr int kMaxAcc13 = 32;  // dG1 / dG3 accumulators per thread: slice <= 32 * 256
constexpr int kPoolWarps = 8;
constexpr int kMaxDPerLane = 8;  // D <= 256

struct TileSmem {
    // offsets in bytes into dynamic shared memory
    size_t keys, sn, si1, si3, rowid, pairid, rowbeg, pairbeg, flag, gs, g2s, dts, total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

__host__ __device__ inline int pairs_per_batch(int q1N) {
    int pb = 8192 / q1N;
    return pb < 1 ? 1 : (pb > 32 ? 32 : pb);
}

// Shared-memory layout of the tile kernels for the largest table of a handle.
__host__ __device__ inline TileSmem tile_layout(int cap, int D, int r1max, int Nmax, int q1Nmax) {
    TileSmem L;
    size_t o = 0;
    L.keys = o;    o = align16(o + sizeof(unsigned long long) * cap);
    L.sn = o;      o = align16(o + sizeof(int) * cap);
    L.si1 = o;     o = align16(o + sizeof(int) * cap);
    L.si3 = o;     o = align16(o + sizeof(int) * cap);
    L.rowid = o;   o = align16(o + sizeof(int) * cap);
    L.pairid = o;  o = align16(o + sizeof(int) * cap);
    L.rowbeg = o;  o = align16(o + sizeof(int) * (cap + 1));
    L.pairbeg = o; o = align16(o + sizeof(int) * (cap + 1));
    L.flag = o;    o = align16(o + sizeof(int) * 40);
    L.gs = o;      o = align16(o + sizeof(float) * (size_t)cap * D);
    L.g2s = o;     o = align16(o + sizeof(float) * (size_t)r1max * (Nmax + 1));
    // a batch of pairs_per_batch(x) pairs of x floats never exceeds max(8192, x) floats
    L.dts = o;     o = align16(o + sizeof(float) * (size_t)(q1Nmax > 8192 ? q1Nmax : 8192));
    L.total = o;
    return L;
}

// Stage G2[i2] into shared memory with a padded row stride N + 1.
__device__ __forceinline__ void stage_g2(const TableDev& T, int i2, float* g2s) {
    const int N = T.q2 * T.r2;
    const int S = T.r1 * N;
    const float* src = T.G2 + (int64_t)i2 * S;
    for (int e = threadIdx.x; e < S; e += blockDim.x) g2s[(e / N) * (N + 1) + (e % N)] = src[e];
}

__device__ __forceinline__ const float* t_of_pair(const Params& P, const TableDev& T, int i2, int i1) {
    return P.Tbuf + T.tbase + ((int64_t)i2 * T.p1 + i1) * (int64_t)(T.q1 * T.q2 * T.r2);
}

// Load the tile's lookups (already grouped by (table, i2), ordered by (i1, pos))
// and sort them by (i1, i3, pos).  Fills keys/sn/si1/si3 of the sorted order.
__device__ void load_and_sort_tile(const Params& P, int start, int len, unsigned long long* keys, int* sn,
                                   int* si1, int* si3) {
    int npow = 1;
    while (npow < len) npow <<= 1;
    for (int k = threadIdx.x; k < npow; k += blockDim.x) {
        unsigned long long key = ~0ull;
        if (k < len) {
            const int n = P.pi21[start + k];
            key = ((unsigned long long)P.lk_i1[n] << (2 * kFieldBits)) |
                  ((unsigned long long)P.lk_i3[n] << kFieldBits) | (unsigned long long)k;
        }
        keys[k] = key;
    }
    block_bitonic_sort(keys, npow);
    const unsigned long long fmask = (1ull << kFieldBits) - 1;
    for (int k = threadIdx.x; k < len; k += blockDim.x) {
        const unsigned long long key = keys[k];
        sn[k] = P.pi21[start + (int)(key & fmask)];
        si1[k] = (int)(key >> (2 * kFieldBits));
        si3[k] = (int)((key >> kFieldBits) & fmask);
    }
    __syncthreads();
}

// ------------------------------------------------------------------ forward

__global__ void __launch_bounds__(kTileThreads) k_tile_fwd(const __grid_constant__ Params P) {
    if ((int)blockIdx.x >= *P.ntiles) return;
    extern __shared__ __align__(16) unsigned char smraw[];
    const TileSmem L = tile_layout(P.tile_cap, P.D, P.r1_max, P.N_max, P.q1N_max);
    unsigned long long* keys = (unsigned long long*)(smraw + L.keys);
    int* sn = (int*)(smraw + L.sn);
    int* si1 = (int*)(smraw + L.si1);
    int* si3 = (int*)(smraw + L.si3);
    int* ulist = (int*)(smraw + L.pairid);
    int* sh = (int*)(smraw + L.flag);
    float* g2s = (float*)(smraw + L.g2s);

    const int4 tl = P.tiles[blockIdx.x];
    const int start = tl.x, len = tl.y, g = tl.z, kin = tl.w;
    const int t = P.bin2_tab[g];
    const TableDev& T = P.tables[t];
    const int i2 = g - T.base2;
    const int q1 = T.q1, r1 = T.r1, N = T.q2 * T.r2;

    load_and_sort_tile(P, start, len, keys, sn, si1, si3);
    for (int k = threadIdx.x; k < len; k += blockDim.x) P.sigma[start + k] = sn[k];

    // pairs whose first lookup lies in this tile compute T here
    int prev_i1 = -1;
    if (kin > 0) prev_i1 = P.lk_i1[P.pi21[start - 1]];
    const int k = threadIdx.x;  // tile_cap <= blockDim
    int f = 0;
    if (k < len) f = (k == 0) ? (si1[0] != prev_i1) : (si1[k] != si1[k - 1]);
    int nU;
    const int slot = block_scan_excl(f, sh, &nU);
    if (f) ulist[slot] = si1[k];
    stage_g2(T, i2, g2s);
    __syncthreads();

    const int64_t total = (int64_t)nU * N;
    for (int64_t e = threadIdx.x; e < total; e += blockDim.x) {
        const int u = (int)(e / N), jc = (int)(e % N);
        const int i1 = ulist[u];
        const float* g1 = T.G1 + (int64_t)i1 * q1 * r1;
        float* dst = P.Tbuf + T.tbase + ((int64_t)i2 * T.p1 + i1) * (int64_t)(q1 * N);
        for (int j1 = 0; j1 < q1; ++j1) {
            float acc = 0.f;
            for (int a = 0; a < r1; ++a) acc = fmaf(g1[j1 * r1 + a], g2s[a * (N + 1) + jc], acc);
            dst[j1 * N + jc] = acc;
        }
    }
}

// Row of one lookup straight from T and G3, for the lanes' columns.
__device__ __forceinline__ void row_from_t(const TableDev& T, const float* Tp, int i3, int lane, float* v) {
    const int q3 = T.q3, r2 = T.r2, D = T.D;
    const float* g3 = T.G3 + (int64_t)i3 * r2 * q3;
#pragma unroll
    for (int m = 0; m < kMaxDPerLane; ++m) {
        const int j = lane + 32 * m;
        float acc = 0.f;
        if (j < D) {
            const int j12 = j / q3, j3 = j - j12 * q3;
            const float* tr = Tp + j12 * r2;
            for (int c = 0; c < r2; ++c) acc = fmaf(tr[c], g3[c * q3 + j3], acc);
        }
        v[m] = acc;
    }
}

// Cache slot of `row` (table 0) or -1.
__device__ __forceinline__ int64_t cache_find(const Params& P, int64_t row) {
    int64_t a = 0, b = P.cache_n;
    while (a < b) {
        const int64_t m = (a + b) >> 1;
        const int64_t v = P.cache_rows[m];
        if (v < row) a = m + 1; else b = m;
    }
    return (a < P.cache_n && P.cache_rows[a] == row) ? a : -1;
}

__global__ void __launch_bounds__(kPoolWarps * 32) k_pool(const __grid_constant__ Params P) {
    const int lane = threadIdx.x & 31;
    const int64_t bag = (int64_t)blockIdx.x * kPoolWarps + (threadIdx.x >> 5);
    if (bag >= P.nbags) return;
    const int t = table_of_bag(P, (int)bag);
    const TableDev& T = P.tables[t];
    const int D = T.D;
    float acc[kMaxDPerLane];
#pragma unroll
    for (int m = 0; m < kMaxDPerLane; ++m) acc[m] = 0.f;
    int64_t lo = P.off[bag], hi = P.off[bag + 1];
    lo = lo < 0 ? 0 : (lo > P.nnz ? P.nnz : lo);
    hi = hi < lo ? lo : (hi > P.nnz ? P.nnz : hi);
    for (int64_t n = lo; n < hi; ++n) {
        const int i1 = P.lk_i1[n], i2 = P.lk_i2[n], i3 = P.lk_i3[n];
        const float s = P.lk_s[n];
        float v[kMaxDPerLane];
        int64_t slot = -1;
        bool fresh = false;
        if (P.cache_n > 0) {
            const int64_t row = ((int64_t)i1 * T.p2 + i2) * T.p3 + i3;
            slot = cache_find(P, row);
            if (slot >= 0) {
                const int need = max(max(P.slice_stamp[i1], P.slice_stamp[T.p1 + i2]), P.slice_stamp[T.p1 + T.p2 + i3]);
                fresh = *(volatile const int*)(P.cache_stamp + slot) >= need;
                __threadfence();  // a refreshed stamp is seen only after its values
            }
        }
        if (fresh) {
            const float* cv = P.cache_vals + slot * D;
#pragma unroll
            for (int m = 0; m < kMaxDPerLane; ++m) {
                const int j = lane + 32 * m;
                v[m] = j < D ? __ldcg(cv + j) : 0.f;
            }
        } else {
            row_from_t(T, t_of_pair(P, T, i2, i1), i3, lane, v);
            if (slot >= 0) {
                // refresh a stale cached row; every writer stores the same values
                float* cv = P.cache_vals + slot * D;
#pragma unroll
                for (int m = 0; m < kMaxDPerLane; ++m) {
                    const int j = lane + 32 * m;
                    if (j < D) __stcg(cv + j, v[m]);
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicExch(P.cache_stamp + slot, P.step);
            }
        }
#pragma unroll
        for (int m = 0; m < kMaxDPerLane; ++m) acc[m] = fmaf(s, v[m], acc[m]);
    }
    float* o = P.out + bag * D;
#pragma unroll
    for (int m = 0; m < kMaxDPerLane; ++m) {
        const int j = lane + 32 * m;
        if (j < D) o[j] = acc[m];
    }
}

// Decompress the cached rows of table 0 (chain product, fp32).
__global__ void k_cache_fill(const __grid_constant__ Params P) {
    const int lane = threadIdx.x & 31;
    const int64_t slot = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (slot >= P.cache_n) return;
    const TableDev& T = P.tables[0];
    const int64_t row = P.cache_rows[slot];
    const int64_t p23 = (int64_t)T.p2 * T.p3;
    const int i1 = (int)(row / p23), i2 = (int)((row / T.p3) % T.p2), i3 = (int)(row % T.p3);
    const int q2 = T.q2, q3 = T.q3, r1 = T.r1, r2 = T.r2, D = T.D;
    const float* g1 = T.G1 + (int64_t)i1 * T.q1 * r1;
    const float* g2 = T.G2 + (int64_t)i2 * r1 * q2 * r2;
    const float* g3 = T.G3 + (int64_t)i3 * r2 * q3;
    for (int j = lane; j < D; j += 32) {
        const int j3 = j % q3, j12 = j / q3, j2 = j12 % q2, j1 = j12 / q2;
        float acc = 0.f;
        for (int c = 0; c < r2; ++c) {
            float tv = 0.f;
            for (int a = 0; a < r1; ++a) tv = fmaf(g1[j1 * r1 + a], g2[(a * q2 + j2) * r2 + c], tv);
            acc = fmaf(tv, g3[c * q3 + j3], acc);
        }
        P.cache_vals[slot * D + j] = acc;
    }
    if (lane == 0) P.cache_stamp[slot] = P.step;
}

// ------------------------------------------------------------------ backward

__global__ void __launch_bounds__(kTileThreads) k_tile_bwd(const __grid_constant__ Params P) {
    if (*P.err) return;  // a device error was recorded: leave every core unchanged
    if ((int)blockIdx.x >= *P.ntiles) return;
    extern __shared__ __align__(16) unsigned char smraw[];
    const TileSmem L = tile_layout(P.tile_cap, P.D, P.r1_max, P.N_max, P.q1N_max);
    int* sn = (int*)(smraw + L.sn);
    int* si1 = (int*)(smraw + L.si1);
    int* si3 = (int*)(smraw + L.si3);
    int* rowid = (int*)(smraw + L.rowid);
    int* pairid = (int*)(smraw + L.pairid);
    int* rowbeg = (int*)(smraw + L.rowbeg);
    int* pairbeg = (int*)(smraw + L.pairbeg);
    int* sh = (int*)(smraw + L.flag);
    float* gs = (float*)(smraw + L.gs);
    float* g2s = (float*)(smraw + L.g2s);
    float* dts = (float*)(smraw + L.dts);

    const int4 tl = P.tiles[blockIdx.x];
    const int start = tl.x, len = tl.y, g = tl.z;
    const int t = P.bin2_tab[g];
    const TableDev& T = P.tables[t];
    const int i2 = g - T.base2;
    const int q1 = T.q1, q2 = T.q2, q3 = T.q3, r1 = T.r1, r2 = T.r2, D = T.D;
    const int N = q2 * r2, q12 = q1 * q2;
    const int S2 = r1 * N;

    // sorted lookups of the tile (order fixed by the forward pass)
    const int k = threadIdx.x;  // tile_cap <= blockDim
    if (k < len) {
        const int n = P.sigma[start + k];
        sn[k] = n;
        si1[k] = P.lk_i1[n];
        si3[k] = P.lk_i3[n];
    }
    __syncthreads();
    int fr = 0, fp = 0;
    if (k < len) {
        fp = (k == 0) || (si1[k] != si1[k - 1]);
        fr = fp || (si3[k] != si3[k - 1]);
    }
    int nrows, npairs;
    const int rex = block_scan_excl(fr, sh, &nrows);
    const int pex = block_scan_excl(fp, sh, &npairs);
    if (k < len) {
        rowid[k] = rex + fr - 1;
        pairid[k] = pex + fp - 1;
        if (fr) rowbeg[rex] = k;
        if (fp) pairbeg[pex] = k;
    }
    if (k == 0) {
        rowbeg[nrows] = len;
        pairbeg[npairs] = len;
        sh[34] = atomicAdd(&P.counters[0], nrows);
        sh[35] = atomicAdd(&P.counters[1], npairs);
    }
    __syncthreads();
    const int slotR = sh[34], slotP = sh[35];
    if (k < len) {
        const int n = sn[k];
        P.rep_row[n] = fr ? slotR + rowid[k] : -1;
        P.rep_pair[n] = fp ? slotP + pairid[k] : -1;
    }
    stage_g2(T, i2, g2s);

    // gs: summed upstream gradient of each tile-row
    for (int e = threadIdx.x; e < nrows * D; e += blockDim.x) {
        const int row = e / D, j = e - row * D;
        float acc = 0.f;
        for (int kk = rowbeg[row]; kk < rowbeg[row + 1]; ++kk) {
            const int n = sn[kk];
            acc = fmaf(P.lk_s[n], P.grad_out[(int64_t)P.lk_bag[n] * D + j], acc);
        }
        gs[row * D + j] = acc;
    }
    __syncthreads();

    // dG3 partial per tile-row: P3[c][j3] = sum_j12 T[j12][c] gs[j12 q3 + j3]
    const int PS = r2 * q3;
    for (int e = threadIdx.x; e < nrows * PS; e += blockDim.x) {
        const int row = e / PS, cj = e - row * PS;
        const int c = cj / q3, j3 = cj - c * q3;
        const int kk = rowbeg[row];
        const float* Tp = t_of_pair(P, T, i2, si1[kk]);
        const float* gr = gs + row * D;
        float acc = 0.f;
        for (int j12 = 0; j12 < q12; ++j12) acc = fmaf(Tp[j12 * r2 + c], gr[j12 * q3 + j3], acc);
        P.Pbuf[(int64_t)(slotR + row) * P.ps_max + cj] = acc;
    }

    // pairs in batches: dT, dG1 partial, dG2 accumulation
    float acc2[kMaxAcc2];
#pragma unroll
    for (int m = 0; m < kMaxAcc2; ++m) acc2[m] = 0.f;
    const int PB = pairs_per_batch(q1 * N);
    const int TS = q1 * N;  // dT size = q1 q2 r2
    for (int u0 = 0; u0 < npairs; u0 += PB) {
        const int nb = min(PB, npairs - u0);
        __syncthreads();
        // dT[u][j12][c] = sum_{rows of u} sum_j3 gs[row][j12 q3 + j3] G3[i3_row][c][j3]
        for (int e = threadIdx.x; e < nb * TS; e += blockDim.x) {
            const int u = e / TS, jc = e - u * TS;
            const int j12 = jc / r2, c = jc - j12 * r2;
            const int kb = pairbeg[u0 + u], ke = pairbeg[u0 + u + 1];
            float acc = 0.f;
            for (int kk = kb; kk < ke; ++kk) {
                if (kk != kb && rowid[kk] == rowid[kk - 1]) continue;  // once per tile-row
                const float* g3 = T.G3 + (int64_t)si3[kk] * r2 * q3 + c * q3;
                const float* gr = gs + rowid[kk] * D + j12 * q3;
                for (int j3 = 0; j3 < q3; ++j3) acc = fmaf(gr[j3], g3[j3], acc);
            }
            dts[u * TS + jc] = acc;
        }
        __syncthreads();
        // dG1 partial: Q[j1][a] = sum_jc dT[j1][jc] G2[a][jc]
        for (int e = threadIdx.x; e < nb * q1 * r1; e += blockDim.x) {
            const int u = e / (q1 * r1), ja = e - u * (q1 * r1);
            const int j1 = ja / r1, a = ja - j1 * r1;
            const float* dt = dts + u * TS + j1 * N;
            const float* g2 = g2s + a * (N + 1);
            float acc = 0.f;
            for (int jc = 0; jc < N; ++jc) acc = fmaf(dt[jc], g2[jc], acc);
            P.Qbuf[(int64_t)(slotP + u0 + u) * P.qs_max + ja] = acc;
        }
        // dG2 += G1[i1]^T dT
#pragma unroll
        for (int m = 0; m < kMaxAcc2; ++m) {
            const int e = threadIdx.x + m * kTileThreads;
            if (e < S2) {
                const int a = e / N, jc = e - a * N;
                float acc = acc2[m];
                for (int u = 0; u < nb; ++u) {
                    const float* g1 = T.G1 + (int64_t)si1[pairbeg[u0 + u]] * q1 * r1 + a;
                    const float* dt = dts + u * TS + jc;
                    for (int j1 = 0; j1 < q1; ++j1) acc = fmaf(g1[j1 * r1], dt[j1 * N], acc);
                }
                acc2[m] = acc;
            }
        }
    }

    // dG2 of the group: direct update, or partials reduced by the group's last tile
    const int nt = P.grp_ntiles[g];
    float* G2p = T.G2 + (int64_t)i2 * S2;
    if (nt == 1) {
#pragma unroll
        for (int m = 0; m < kMaxAcc2; ++m) {
            const int e = threadIdx.x + m * kTileThreads;
            if (e < S2) G2p[e] = fmaf(-P.lr, acc2[m], G2p[e]);
        }
        if (P.slice_stamp && threadIdx.x == 0 && t == 0) P.slice_stamp[T.p1 + i2] = P.step + 1;
        return;
    }
    float* mine = P.dG2part + (int64_t)blockIdx.x * P.s2_max;
#pragma unroll
    for (int m = 0; m < kMaxAcc2; ++m) {
        const int e = threadIdx.x + m * kTileThreads;
        if (e < S2) mine[e] = acc2[m];
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) sh[36] = (atomicAdd(&P.grp_done[g], 1) == nt - 1);
    __syncthreads();
    if (!sh[36]) return;
    __threadfence();
    const int first = P.grp_first[g];
    for (int e = threadIdx.x; e < S2; e += blockDim.x) {
        float sum = 0.f;
        for (int tt = 0; tt < nt; ++tt) sum += __ldcg(P.dG2part + (int64_t)(first + tt) * P.s2_max + e);
        G2p[e] = fmaf(-P.lr, sum, G2p[e]);
    }
    if (threadIdx.x == 0) {
        P.grp_done[g] = 0;
        if (P.slice_stamp && t == 0) P.slice_stamp[T.p1 + i2] = P.step + 1;
    }
}

// Sum the dG1 (per tile-pair) and dG3 (per tile-row) partials of one slice in
// sorted-segment order, then apply the SGD update to that slice.
__global__ void __launch_bounds__(kTileThreads) k_reduce13(const __grid_constant__ Params P) {
    if (*P.err) return;
    __shared__ int reps[kTileThreads];
    int b = blockIdx.x;
    const bool first_core = b < P.n1;
    if (!first_core) b -= P.n1;
    const int nb = first_core ? P.n1 : P.n3;
    const int* H = first_core ? P.H1 : P.H3;
    const int* pi = first_core ? P.pi1 : P.pi3;
    const int* rep = first_core ? P.rep_pair : P.rep_row;
    const float* buf = first_core ? P.Qbuf : P.Pbuf;
    const int stride = first_core ? P.qs_max : P.ps_max;
    const int start = H[(int64_t)b * P.nch];
    const int end = (b + 1 < nb) ? H[(int64_t)(b + 1) * P.nch] : (int)P.nnz;
    if (start >= end) return;
    const int t = first_core ? P.bin1_tab[b] : P.bin3_tab[b];
    const TableDev& T = P.tables[t];
    const int slice = b - (first_core ? T.base1 : T.base3);
    const int S = first_core ? T.q1 * T.r1 : T.r2 * T.q3;
    float acc[kMaxAcc13];
#pragma unroll
    for (int m = 0; m < kMaxAcc13; ++m) acc[m] = 0.f;
    for (int base = start; base < end; base += blockDim.x) {
        const int kk = base + threadIdx.x;
        reps[threadIdx.x] = kk < end ? rep[pi[kk]] : -1;
        __syncthreads();
        const int cnt = min((int)blockDim.x, end - base);
        for (int j = 0; j < cnt; ++j) {
            const int r = reps[j];
            if (r < 0) continue;
            const float* src = buf + (int64_t)r * stride;
#pragma unroll
            for (int m = 0; m < kMaxAcc13; ++m) {
                const int e = threadIdx.x + m * kTileThreads;
                if (e < S) acc[m] += src[e];
            }
        }
        __syncthreads();
    }
    float* G = (first_core ? T.G1 : T.G3) + (int64_t)slice * S;
#pragma unroll
    for (int m = 0; m < kMaxAcc13; ++m) {
        const int e = threadIdx.x + m * kTileThreads;
        if (e < S) G[e] = fmaf(-P.lr, acc[m], G[e]);
    }
    if (P.slice_stamp && threadIdx.x == 0 && t == 0)
        P.slice_stamp[first_core ? slice : T.p1 + T.p2 + slice] = P.step + 1;
}

// ------------------------------------------------------------------ launchers

size_t tile_fwd_smem(const Params& P) { return tile_layout(P.tile_cap, P.D, P.r1_max, P.N_max, P.q1N_max).total; }
size_t tile_bwd_smem(const Params& P) { return tile_layout(P.tile_cap, P.D, P.r1_max, P.N_max, P.q1N_max).total; }

cudaError_t launch_tile_fwd(const Params& P, cudaStream_t s) {
    const size_t smem = tile_fwd_smem(P);
    cudaError_t e = cudaFuncSetAttribute(k_tile_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_tile_fwd<<<P.max_tiles, kTileThreads, smem, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_pool(const Params& P, cudaStream_t s) {
    const int64_t blocks = (P.nbags + kPoolWarps - 1) / kPoolWarps;
    k_pool<<<(unsigned)blocks, kPoolWarps * 32, 0, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_cache_fill(const Params& P, cudaStream_t s) {
    const int64_t blocks = (P.cache_n + 7) / 8;
    k_cache_fill<<<(unsigned)blocks, 256, 0, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_tile_bwd(const Params& P, cudaStream_t s) {
    const size_t smem = tile_bwd_smem(P);
    cudaError_t e = cudaFuncSetAttribute(k_tile_bwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_tile_bwd<<<P.max_tiles, kTileThreads, smem, s>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_reduce13(const Params& P, cudaStream_t s) {
    k_reduce13<<<P.n1 + P.n3, kTileThreads, 0, s>>>(P);
    return cudaGetLastError();
}

}  // namespace ttemb
