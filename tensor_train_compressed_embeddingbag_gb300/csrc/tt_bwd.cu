// tt_bwd.cu -- backward contractions, sorted-segment reductions and the fused
// SGD update (sm_103a, FP32 FFMA).
//
// FBTT README, "Software Cache" (the core gradients are a chain of products in
// reversed order) and "Fused Kernel" (the update is applied inside the
// backward pass); tensorflow/addons EmbeddingBag issue (gradients are formed
// after sorting by key so that no two threads write the same entry).
// Per tile of lookups that share (table, i2), with rows (i1, i2, i3) and pairs
// (i1, i2) as maximal runs of the sorted tile:
//   gs  = sum over the row's lookups of s_n grad_out[bag]  (q1 q2 x q3)
//   P3  = T^T gs                       (r2 x q3)   dG3 partial per row
//   dT  = sum_rows gs . G3[i3]^T       (q1 x q2 r2) per pair
//   Q   = dT . G2[i2]^T                (q1 x r1)   dG1 partial per pair
//   dG2 += G1[i1]^T . dT               (r1 x q2 r2)
// A column split (SPLIT = 2) gives each of two blocks the columns c of one
// half of r2: P3, dT and dG2 columns are disjoint, Q is summed over the two
// halves when its G1 slice is reduced.  k_reduce13 then reduces every G1 / G3
// slice in sorted-segment order, one block per slice.
#include <algorithm>

#include "tt_dims.cuh"
#include "tt_tile.cuh"

namespace ttemb {

constexpr int kBwdThreads = 256;
constexpr int kMaxAcc2 = 64;   // generic path: dG2 accumulators per thread (r1 q2 r2 <= 64 * 256)
constexpr int kGsUnroll = 4;     // independent gradient rows per thread in flight
constexpr int kDtUnroll = 4;     // independent dT items per thread in flight

__host__ __device__ inline size_t al16(size_t x) { return (x + 15) & ~(size_t)15; }

// Pairs per batch: dT batch <= 8192 floats, G1 batch <= 8192 floats, and at
// most 256 threads for the Q register tiles.
__host__ __device__ inline int bwd_pairs_per_batch(int q1, int Ns, int r1) {
    int pb = 16;
    if (pb * q1 * Ns > 8192) pb = 8192 / (q1 * Ns);
    if (pb * q1 * r1 > 8192) pb = 8192 / (q1 * r1);
    if (pb * (r1 / 4 > 0 ? r1 / 4 : 1) > 256) pb = 256 / (r1 / 4 > 0 ? r1 / 4 : 1);
    return pb < 1 ? 1 : pb;
}

struct BwdLayout {
    size_t keys, sp1, sp3, si1, si3, sbag, ss, rowid, pairid, rowbeg, pairbeg, sh, gs, g2t, g1s, dts, total;
};

__host__ __device__ inline BwdLayout bwd_layout(int cap, int D, int g2f, int g1f, int dtf) {
    BwdLayout L;
    size_t o = 0;
    L.keys = o;    o = al16(o + sizeof(unsigned long long) * cap);
    L.sp1 = o;     o = al16(o + sizeof(int) * cap);
    L.sp3 = o;     o = al16(o + sizeof(int) * cap);
    L.si1 = o;     o = al16(o + sizeof(int) * cap);
    L.si3 = o;     o = al16(o + sizeof(int) * cap);
    L.sbag = o;    o = al16(o + sizeof(int) * cap);
    L.ss = o;      o = al16(o + sizeof(float) * cap);
    L.rowid = o;   o = al16(o + sizeof(int) * cap);
    L.pairid = o;  o = al16(o + sizeof(int) * cap);
    L.rowbeg = o;  o = al16(o + sizeof(int) * (cap + 1));
    L.pairbeg = o; o = al16(o + sizeof(int) * (cap + 1));
    L.sh = o;      o = al16(o + sizeof(int) * 64);
    L.gs = o;      o = al16(o + sizeof(float) * (size_t)cap * D);
    L.g2t = o;     o = al16(o + sizeof(float) * (size_t)g2f);  // G2 columns of the split, padded rows
    L.g1s = o;     o = al16(o + sizeof(float) * (size_t)g1f);
    L.dts = o;     o = al16(o + sizeof(float) * (size_t)dtf);
    L.total = o;
    return L;
}

// Sum the dG1 (per tile-pair, over the column splits) or dG3 (per tile-row)
// partials of one slice in sorted-segment order, then apply the SGD update to
// the slice (one block per slice, after every tile block).  The slots of the slice are compacted in segment order; thread
// (lane group r, element e) loads slots j = r, r + R, ... kReducePer at a time
// and sums them in order, then the R partial sums are added in r order.
constexpr int kReduceSlots = 1024;   // slots gathered per round
constexpr int kReducePer = 32;       // loads in flight per thread (scalar columns)
constexpr int kReducePer4 = 16;      // float4 loads in flight per thread
constexpr int kP3Items = 3;          // P3 items per thread whose T loads are in flight together

__device__ void reduce_slice(const Params& P, int bglob, int* slots, int* sh, float* sacc) {
    const bool first_core = bglob < P.n1;
    const int b = first_core ? bglob : bglob - P.n1;
    const int nb = first_core ? P.n1 : P.n3;
    const int* H = first_core ? P.H1 : P.H3;
    const int* rep = first_core ? P.rep1 : P.rep3;  // indexed by position in the i1 / i3 order
    const int start = H[(int64_t)b * P.nch];
    const int end = (b + 1 < nb) ? H[(int64_t)(b + 1) * P.nch] : *P.nincl;
    const int t = first_core ? P.bin1_tab[b] : P.bin3_tab[b];
    const TableDev& T = P.tables[t];
    const int slice = b - (first_core ? T.base1 : T.base3);
    const int S = first_core ? T.q1 * T.r1 : T.r2 * T.q3;
    const int nsub = first_core ? P.split : 1;  // dG1 partials: one per column split
    const int stride = first_core ? P.qs_max : P.ps_max;
    const float* buf = first_core ? P.Qbuf : P.Pbuf;
    float* G = (first_core ? T.G1 : T.G3) + (int64_t)slice * S;
    float* A = (first_core ? T.aux[0] : T.aux[2]);
    if (A) A += (int64_t)slice * S;
    // Lanes: groups of W threads; thread (r, e) sums element column e (float4 when S % 4 == 0:
    // four elements per thread, every slot row read in 16-byte words) over the slots
    // j = r, r + R, ..., kReducePer loads in flight; the R group sums are added in group order.
    const bool v4 = (S & 3) == 0;  // slot strides are whole 16-byte words (rounded on the host)
    const int SE = v4 ? S >> 2 : S;  // element columns (float4 or float)
    const int W = SE >= kBwdThreads ? kBwdThreads : SE;
    const int R = kBwdThreads / W;
    const int r = threadIdx.x / W;
    const int nacc = R * S > S ? R * S : S;  // group sums, or S when one group walks every column
    for (int e = threadIdx.x; e < nacc; e += blockDim.x) sacc[e] = 0.f;
    __syncthreads();
    for (int base = start; base < end;) {
        int nslot = 0;
        while (base < end && nslot + (int)blockDim.x * nsub <= kReduceSlots) {
            const int kk = base + threadIdx.x;
            const int rv = kk < end ? rep[kk] : -1;
#ifdef TTEMB_DEBUG
            if (rv >= 0) TT_DCHECK(P, rv, P.nnz);
#endif
            int tot;
            const int ex = block_scan_excl(rv >= 0 ? 1 : 0, sh, &tot);
            if (rv >= 0)
                for (int q = 0; q < nsub; ++q) slots[nslot + ex * nsub + q] = rv * nsub + q;
            nslot += tot * nsub;
            base += blockDim.x;
        }
        __syncthreads();
        if (r < R) {
            const int e0 = threadIdx.x - r * W;
#pragma unroll 1
            for (int e = e0; e < SE; e += W) {
                if (v4) {
                    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
                    for (int j0 = r; j0 < nslot; j0 += R * kReducePer4) {
                        float4 v[kReducePer4];
#pragma unroll
                        for (int u = 0; u < kReducePer4; ++u) {
                            const int j = j0 + u * R;
                            v[u] = j < nslot ? __ldg(reinterpret_cast<const float4*>(buf + (int64_t)slots[j] * stride) + e)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int u = 0; u < kReducePer4; ++u) {
                            a.x += v[u].x; a.y += v[u].y; a.z += v[u].z; a.w += v[u].w;
                        }
                    }
                    float* dst = sacc + (R > 1 ? r * S : 0) + 4 * e;
                    dst[0] += a.x; dst[1] += a.y; dst[2] += a.z; dst[3] += a.w;
                } else {
                    float a = 0.f;
#pragma unroll 1
                    for (int j0 = r; j0 < nslot; j0 += R * kReducePer) {
                        float v[kReducePer];
#pragma unroll
                        for (int u = 0; u < kReducePer; ++u) {
                            const int j = j0 + u * R;
                            v[u] = j < nslot ? __ldg(buf + (int64_t)slots[j] * stride + e) : 0.f;
                        }
#pragma unroll
                        for (int u = 0; u < kReducePer; ++u) a += v[u];
                    }
                    sacc[(R > 1 ? r * S : 0) + e] += a;
                }
            }
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < S; e += blockDim.x) {
        float sum = 0.f;  // the R lane groups' sums in group order
        for (int rr = 0; rr < R; ++rr) sum += sacc[(R > 1 ? rr * S : 0) + e];
        core_update(P, G, A, e, sum);
    }
    if (P.slice_stamp && P.opt != TT_OPT_GRAD && threadIdx.x == 0 && t == 0)
        P.slice_stamp[first_core ? slice : T.p1 + T.p2 + slice] = *P.dstep + 1;
    __syncthreads();
}

// Register tiling of the batch loop for the compiled classes (q1 = 4, r1 % 16 == 0).
//   Q   = dT . G2^T : thread (kh, a4, u) owns a 4 (j1) x 4 (a) tile summed over the columns
//                     jc = kh mod KH; a warp spans KH x AL x UL threads, so one shared load
//                     touches at most 8 distinct 16-byte words (dT pairs US floats apart,
//                     G2 rows GS floats apart, both strides chosen to spread the banks);
//   dG2 = G1^T . dT : thread owns a = ag + A4 i, jc = jg + JG c (i, c < 4); a warp spans
//                     AG x JL such tiles (AG consecutive G1 words, JL consecutive dT words);
//                     the pairs are split over KS warp groups when one group covers all tiles.
template <class Dm, int SPLIT>
struct BwdTiling {
    static constexpr int R1 = Dm::r1(), Q2 = Dm::q2(), Q3 = Dm::q3(), R2 = Dm::r2();
    static constexpr int R2S = R2 / SPLIT, NS = Q2 * R2S, D = 4 * Q2 * Q3;
    static constexpr int PBc = (16 * 4 * NS > 8192) ? 8192 / (4 * NS) : ((16 * 4 * R1 > 8192) ? 8192 / (4 * R1) : 16);
    static constexpr int PBS = (PBc * (R1 / 4) > 256) ? 256 / (R1 / 4) : PBc;
    static constexpr int A4 = R1 / 4;
    static constexpr int KH = 256 / (PBS * A4) >= 1 ? 256 / (PBS * A4) : 1;
    static constexpr int AL = (KH == 1 ? 8 : 4) < A4 ? (KH == 1 ? 8 : 4) : A4;
    static constexpr int UL = 32 / (KH * AL);
    static constexpr int US = 4 * NS + 4 * KH;  // dts pair stride (floats)
    static constexpr int GS = KH == 1 ? R1 + 4 : R1 + (((4 * AL - R1) % 32) + 32) % 32;  // g2t row stride
    static constexpr int JG = NS / 4;
    static constexpr int AG = A4 < 8 ? A4 : 8;
    static constexpr int JL = 32 / AG;
    static constexpr int WT = (A4 / AG) * (JG / JL);  // warps that cover every dG2 tile once
    static constexpr int NT = WT >= 8 ? WT / 8 : 1;   // tile sets per warp
    static constexpr int KS = WT >= 8 ? 1 : 8 / WT;   // warp groups splitting the pairs
    static_assert(kBwdThreads == 256, "tiling assumes 8 warps");
    static_assert(KH >= 1 && KH <= 4 && (KH & (KH - 1)) == 0 && KH * AL * UL == 32, "Q lanes");
    static_assert(A4 % AL == 0 && PBS % UL == 0 && (A4 / AL) * (PBS / UL) == 8, "Q warps");
    static_assert(PBS <= 16 && US <= 4 * NS + 16 && GS <= R1 + 32, "padding within the host sizes");
    static_assert(A4 % AG == 0 && JG % JL == 0 && (NT * 8 == WT || KS * WT == 8), "dG2 tiles");
    static_assert(KS == 1 || D * (4096 / D) >= 4096, "cross-warp dG2 sums fit in gs");
};

template <class Dm, int SPLIT>
__device__ void tile_bwd_body(const Params& P, const TableDev& T, const Dm dm, unsigned char* smraw) {
    const BwdLayout L = bwd_layout(P.tile_cap, P.D, P.g2s_floats, P.g1s_floats, P.dts_floats);
    unsigned long long* keys = (unsigned long long*)(smraw + L.keys);
    int* sp1 = (int*)(smraw + L.sp1);
    int* sp3 = (int*)(smraw + L.sp3);
    int* si1 = (int*)(smraw + L.si1);
    int* si3 = (int*)(smraw + L.si3);
    int* sbag = (int*)(smraw + L.sbag);
    float* ss = (float*)(smraw + L.ss);
    int* rowid = (int*)(smraw + L.rowid);
    int* pairid = (int*)(smraw + L.pairid);
    int* rowbeg = (int*)(smraw + L.rowbeg);
    int* pairbeg = (int*)(smraw + L.pairbeg);
    int* sh = (int*)(smraw + L.sh);
    float* gs = (float*)(smraw + L.gs);
    float* g2t = (float*)(smraw + L.g2t);
    float* g1s = (float*)(smraw + L.g1s);
    float* dts = (float*)(smraw + L.dts);

    const int tile = blockIdx.x / SPLIT, sp = blockIdx.x % SPLIT;
    const int4 tl = P.tiles[tile];
    const int start = tl.x, len = tl.y, g = tl.z;
    const int i2 = g - T.base2;
    const int q1 = dm.q1(), q2 = dm.q2(), q3 = dm.q3(), r1 = dm.r1(), r2 = dm.r2();
    const int D = q1 * q2 * q3, q12 = q1 * q2;
    const int r2s = r2 / SPLIT, c0 = sp * r2s, Ns = q2 * r2s;
    const int t = P.bin2_tab[g];

    // ---- the first 8 G2 values of this thread (the G2 slice depends only on i2): their
    // loads are in flight while the tile's lookups are read and sorted
    const float* g2src = T.G2 + (int64_t)i2 * r1 * q2 * r2;
    const int g2n = r1 * Ns;
    float g2v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int e = q * kBwdThreads + threadIdx.x;
        g2v[q] = 0.f;
        if (e < g2n) {
            const int a = e / Ns, jc = e - a * Ns;
            const int j2 = jc / r2s, c = jc - j2 * r2s;
            g2v[q] = __ldg(g2src + (a * q2 + j2) * r2 + c0 + c);
        }
    }

    // ---- lookups of the tile, sorted by (i1, i3, position)
    load_and_sort_tile(P, start, len, keys, sp1, sp3, si1, si3, sbag, ss);
#ifdef TTEMB_DEBUG
    if ((int)threadIdx.x < len) {  // the tile's slices within the table, its group within the bins
        si1[threadIdx.x] = TT_DCHECK(P, si1[threadIdx.x], T.p1);
        si3[threadIdx.x] = TT_DCHECK(P, si3[threadIdx.x], T.p3);
    }
    if (threadIdx.x == 0) TT_DCHECK(P, i2, T.p2);
    __syncthreads();
#endif
    const int k = threadIdx.x;  // tile_cap <= blockDim
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
    }
    __syncthreads();
    // partial slots are numbered by the position of the run's first lookup in the
    // grouped order, so every run of every tile owns one slot, with no atomics
    if (sp == 0 && k < len) {
        P.rep3[sp3[k]] = fr ? start + k : -1;
        P.rep1[sp1[k]] = fp ? start + k : -1;
    }

    // ---- G2 columns of this split, transposed: g2t[jc'][a], jc' = j2 r2s + c' (8 loads in flight;
    // the first round was loaded before the sort)
    {
        const float* src = g2src;
        const int n = g2n;
        int gstride = r1 + 4;
        if constexpr (Dm::kStatic) gstride = BwdTiling<Dm, SPLIT>::GS;
        for (int base = 0; base < n; base += 8 * kBwdThreads) {
            float v[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = base + q * kBwdThreads + threadIdx.x;
                v[q] = 0.f;
                if (base == 0) {
                    v[q] = g2v[q];
                } else if (e < n) {
                    const int a = e / Ns, jc = e - a * Ns;
                    const int j2 = jc / r2s, c = jc - j2 * r2s;
                    v[q] = __ldg(src + (a * q2 + j2) * r2 + c0 + c);
                }
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = base + q * kBwdThreads + threadIdx.x;
                if (e < n) {
                    const int a = e / Ns, jc = e - a * Ns;
                    g2t[jc * gstride + a] = v[q];
                }
            }
        }
    }
    // ---- gs: summed upstream gradient of every tile-row
    if ((D & 3) == 0) {  // every compiled class and every D % 4 == 0 table
        tile_gs(P, len, nrows, sbag, ss, rowbeg, gs, D);
    } else {
        __syncthreads();
        for (int e = threadIdx.x; e < nrows * D; e += blockDim.x) {
            const int row = e / D, j = e - row * D;
            float acc = 0.f;
            for (int kk = rowbeg[row]; kk < rowbeg[row + 1]; ++kk)
                acc = fmaf(ss[kk], __ldg(P.grad_out + (int64_t)sbag[kk] * D + j), acc);
            gs[row * D + j] = acc;
        }
        __syncthreads();
    }

    // ---- dG3 partial per tile-row, columns c of this split: P3[c][j3] = sum_j12 T[j12][c] gs[j12 q3 + j3]
    if constexpr (Dm::kStatic) {
        // kP3Items items per thread: the T columns of all are loaded before any is summed
        constexpr int Q3 = Dm::q3(), Q12 = Dm::q1() * Dm::q2(), R2 = Dm::r2();
        const int items = nrows * r2s;
        for (int e0 = threadIdx.x; e0 < items; e0 += kP3Items * kBwdThreads) {
            float tv[kP3Items][Q12];
            int rowv[kP3Items], cv[kP3Items];
#pragma unroll
            for (int v = 0; v < kP3Items; ++v) {
                const int e = e0 + v * kBwdThreads;
                rowv[v] = e < items ? e / r2s : -1;
                cv[v] = e < items ? c0 + (e - rowv[v] * r2s) : 0;
                const int kk = rowv[v] >= 0 ? rowbeg[rowv[v]] : 0;
                const float* Tp = P.Tbuf + T.tbase + ((int64_t)i2 * T.p1 + si1[kk]) * (int64_t)(Q12 * R2) + cv[v];
#pragma unroll
                for (int j12 = 0; j12 < Q12; ++j12) tv[v][j12] = rowv[v] >= 0 ? __ldg(Tp + j12 * R2) : 0.f;
            }
#pragma unroll
            for (int v = 0; v < kP3Items; ++v) {
                if (rowv[v] < 0) continue;
                const float* gr = gs + rowv[v] * D;
                float acc[Q3];
#pragma unroll
                for (int j3 = 0; j3 < Q3; ++j3) acc[j3] = 0.f;
#pragma unroll
                for (int j12 = 0; j12 < Q12; ++j12) {
#pragma unroll
                    for (int j3 = 0; j3 < Q3; j3 += 4) {
                        const float4 x = *reinterpret_cast<const float4*>(gr + j12 * Q3 + j3);
                        acc[j3] = fmaf(tv[v][j12], x.x, acc[j3]);
                        acc[j3 + 1] = fmaf(tv[v][j12], x.y, acc[j3 + 1]);
                        acc[j3 + 2] = fmaf(tv[v][j12], x.z, acc[j3 + 2]);
                        acc[j3 + 3] = fmaf(tv[v][j12], x.w, acc[j3 + 3]);
                    }
                }
                float* dst = P.Pbuf + (int64_t)(start + rowbeg[rowv[v]]) * P.ps_max + cv[v] * Q3;
                if constexpr (Q3 % 4 == 0) {  // whole 16-byte words: lanes of consecutive c fill whole sectors
#pragma unroll
                    for (int j3 = 0; j3 < Q3; j3 += 4)
                        *reinterpret_cast<float4*>(dst + j3) = make_float4(acc[j3], acc[j3 + 1], acc[j3 + 2], acc[j3 + 3]);
                } else {
#pragma unroll
                    for (int j3 = 0; j3 < Q3; ++j3) dst[j3] = acc[j3];
                }
            }
        }
    } else {
        for (int e = threadIdx.x; e < nrows * r2s; e += blockDim.x) {
            const int row = e / r2s, c = c0 + (e - row * r2s);
            const int kk = rowbeg[row];
            const float* Tp = P.Tbuf + T.tbase + ((int64_t)i2 * T.p1 + si1[kk]) * (int64_t)(q12 * r2) + c;
            const float* gr = gs + row * D;
            float* dst = P.Pbuf + (int64_t)(start + kk) * P.ps_max + c * q3;
            for (int j3 = 0; j3 < q3; ++j3) {
                float acc = 0.f;
                for (int j12 = 0; j12 < q12; ++j12) acc = fmaf(Tp[j12 * r2], gr[j12 * q3 + j3], acc);
                dst[j3] = acc;
            }
        }
    }

    // ---- pairs in batches: dT, dG1 partial (Q), dG2 accumulation
    const int PB = bwd_pairs_per_batch(q1, Ns, r1);
    float* G2p = T.G2 + (int64_t)i2 * r1 * q2 * r2;
    float* A2p = T.aux[1] ? T.aux[1] + (int64_t)i2 * r1 * q2 * r2 : nullptr;

    if constexpr (Dm::kStatic) {
        using BT = BwdTiling<Dm, SPLIT>;
        constexpr int R1 = BT::R1, Q2 = BT::Q2, Q3 = BT::Q3, R2 = BT::R2;
        constexpr int R2S = BT::R2S, NS = BT::NS, D_ = BT::D, PBS = BT::PBS, A4 = BT::A4;
        constexpr int KH = BT::KH, AL = BT::AL, UL = BT::UL, US = BT::US, GS = BT::GS;
        constexpr int JG = BT::JG, AG = BT::AG, JL = BT::JL, WT = BT::WT, NT = BT::NT, KS = BT::KS;
        const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
        float acc2[NT][4][4];
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc2[i][a][c] = 0.f;
        // dG2 tile of this thread (tile set i adds 8 i to the warp's tile index)
        const int ks = KS > 1 ? w / WT : 0, wt0 = KS > 1 ? w % WT : w;
        // g1s[u][a][j1] of a batch: GPT values per thread (every compiled class: PBS R1 4 <= 16 kBwdThreads);
        // the next batch's values are loaded into registers while this batch computes
        constexpr int GPT = (PBS * R1 * 4 + kBwdThreads - 1) / kBwdThreads;
        static_assert(GPT <= 16, "G1 prefetch registers");
        float g1n[GPT];
        auto load_g1 = [&](int ub) {
            const int nbb = min(PBS, npairs - ub);
#pragma unroll
            for (int q = 0; q < GPT; ++q) {
                const int e = q * kBwdThreads + threadIdx.x;
                g1n[q] = 0.f;
                if (e < nbb * R1 * 4) {
                    const int u = e / (R1 * 4), rem = e - u * (R1 * 4);
                    g1n[q] = __ldg(T.G1 + (int64_t)si1[pairbeg[ub + u]] * (4 * R1) + (rem & 3) * R1 + (rem >> 2));
                }
            }
        };
        if (npairs > 0) load_g1(0);
        for (int u0 = 0; u0 < npairs; u0 += PBS) {
            const int nb = min(PBS, npairs - u0);
            __syncthreads();
#pragma unroll
            for (int q = 0; q < GPT; ++q) {
                const int e = q * kBwdThreads + threadIdx.x;
                if (e < nb * R1 * 4) g1s[e] = g1n[q];
            }
            if (u0 + PBS < npairs) load_g1(u0 + PBS);
            // dts[u][jc'][j1] = sum_rows sum_j3 gs[row][(j1 q2 + j2) q3 + j3] G3[i3][c][j3];
            // kDtUnroll items per thread load the G3 row of their pair's first row together
            for (int e0 = threadIdx.x; e0 < nb * NS; e0 += kDtUnroll * kBwdThreads) {
                float g3v[kDtUnroll][Q3];
                int uu[kDtUnroll], jj[kDtUnroll];
#pragma unroll
                for (int v = 0; v < kDtUnroll; ++v) {
                    const int e = e0 + v * kBwdThreads;
                    uu[v] = e < nb * NS ? e / NS : -1;
                    jj[v] = e < nb * NS ? e - uu[v] * NS : 0;
                    const int j2 = jj[v] / R2S, c = c0 + (jj[v] - j2 * R2S);
                    const int kb = uu[v] >= 0 ? pairbeg[u0 + uu[v]] : 0;
                    const float* g3 = T.G3 + (int64_t)si3[kb] * (R2 * Q3) + c * Q3;
#pragma unroll
                    for (int j3 = 0; j3 < Q3; j3 += 4) {
                        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (uu[v] >= 0) x = __ldg(reinterpret_cast<const float4*>(g3 + j3));
                        g3v[v][j3] = x.x; g3v[v][j3 + 1] = x.y; g3v[v][j3 + 2] = x.z; g3v[v][j3 + 3] = x.w;
                    }
                }
#pragma unroll
                for (int v = 0; v < kDtUnroll; ++v) {
                    if (uu[v] < 0) continue;
                    const int u = uu[v], jc = jj[v];
                    const int j2 = jc / R2S, c = c0 + (jc - j2 * R2S);
                    const int kb = pairbeg[u0 + u], ke = pairbeg[u0 + u + 1];
                    float a4v[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int kk = kb; kk < ke; ++kk) {
                        if (kk != kb && rowid[kk] == rowid[kk - 1]) continue;  // once per tile-row
                        float g3r[Q3];
                        if (kk == kb) {
#pragma unroll
                            for (int j3 = 0; j3 < Q3; ++j3) g3r[j3] = g3v[v][j3];
                        } else {
                            const float* g3 = T.G3 + (int64_t)si3[kk] * (R2 * Q3) + c * Q3;
#pragma unroll
                            for (int j3 = 0; j3 < Q3; j3 += 4) {
                                const float4 x = __ldg(reinterpret_cast<const float4*>(g3 + j3));
                                g3r[j3] = x.x; g3r[j3 + 1] = x.y; g3r[j3 + 2] = x.z; g3r[j3 + 3] = x.w;
                            }
                        }
                        const float* gr = gs + rowid[kk] * D_ + j2 * Q3;
#pragma unroll
                        for (int j1 = 0; j1 < 4; ++j1) {
#pragma unroll
                            for (int j3 = 0; j3 < Q3; j3 += 4) {
                                const float4 x = *reinterpret_cast<const float4*>(gr + j1 * Q2 * Q3 + j3);
                                a4v[j1] = fmaf(x.x, g3r[j3], a4v[j1]);
                                a4v[j1] = fmaf(x.y, g3r[j3 + 1], a4v[j1]);
                                a4v[j1] = fmaf(x.z, g3r[j3 + 2], a4v[j1]);
                                a4v[j1] = fmaf(x.w, g3r[j3 + 3], a4v[j1]);
                            }
                        }
                    }
                    *reinterpret_cast<float4*>(dts + u * US + jc * 4) = make_float4(a4v[0], a4v[1], a4v[2], a4v[3]);
                }
            }
            __syncthreads();
            // Q[u][j1][a] = sum_jc' dts[u][jc'][j1] g2t[jc'][a]: thread (kh, a4, u)
            if ((w / (A4 / AL)) * UL < nb) {  // warps whose pairs all lie past the batch skip it
                const int kh = lane % KH, al = (lane / KH) % AL, ul = lane / (KH * AL);
                const int a4 = (w % (A4 / AL)) * AL + al, u = (w / (A4 / AL)) * UL + ul;
                float q[4][4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int a = 0; a < 4; ++a) q[j][a] = 0.f;
                const float* dt = dts + u * US;
                const float* gt = g2t + a4 * 4;
#pragma unroll 4
                for (int jc = kh; jc < NS; jc += KH) {
                    const float4 x = *reinterpret_cast<const float4*>(dt + jc * 4);
                    const float4 y = *reinterpret_cast<const float4*>(gt + jc * GS);
                    const float xv[4] = {x.x, x.y, x.z, x.w};
                    const float yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int a = 0; a < 4; ++a) q[j][a] = fmaf(xv[j], yv[a], q[j][a]);
                }
#pragma unroll
                for (int o = KH / 2; o >= 1; o >>= 1)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int a = 0; a < 4; ++a) q[j][a] += __shfl_xor_sync(0xffffffffu, q[j][a], o);
                if (kh == 0 && u < nb) {
                    float* dst = P.Qbuf + ((int64_t)(start + pairbeg[u0 + u]) * SPLIT + sp) * P.qs_max + a4 * 4;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        *reinterpret_cast<float4*>(dst + j * R1) = make_float4(q[j][0], q[j][1], q[j][2], q[j][3]);
                }
            }
            // dG2[a][jc'] += sum_u sum_j1 g1s[u][a][j1] dts[u][jc'][j1] over the pairs u = ks mod KS
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                const int wt = wt0 + 8 * i;
                const int ag = (wt % (A4 / AG)) * AG + lane % AG, jg = (wt / (A4 / AG)) * JL + lane / AG;
                for (int u = ks; u < nb; u += KS) {
                    float gv[4][4], dv[4][4];
#pragma unroll
                    for (int a = 0; a < 4; ++a) {
                        const float4 x = *reinterpret_cast<const float4*>(g1s + (u * R1 + ag + A4 * a) * 4);
                        gv[a][0] = x.x; gv[a][1] = x.y; gv[a][2] = x.z; gv[a][3] = x.w;
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const float4 x = *reinterpret_cast<const float4*>(dts + u * US + (jg + JG * c) * 4);
                        dv[c][0] = x.x; dv[c][1] = x.y; dv[c][2] = x.z; dv[c][3] = x.w;
                    }
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int j = 0; j < 4; ++j) acc2[i][a][c] = fmaf(gv[a][j], dv[c][j], acc2[i][a][c]);
                }
            }
        }
        // add the KS warp groups' sums in group order (gs is free after the last batch)
        if constexpr (KS > 1) {
            __syncthreads();
            float* red = gs;
            if (ks > 0) {
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int c = 0; c < 4; ++c) red[(((ks - 1) * WT + wt0) * 16 + a * 4 + c) * 32 + lane] = acc2[0][a][c];
            }
            __syncthreads();
            if (ks == 0) {
                for (int k2 = 1; k2 < KS; ++k2)
#pragma unroll
                    for (int a = 0; a < 4; ++a)
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc2[0][a][c] += red[(((k2 - 1) * WT + wt0) * 16 + a * 4 + c) * 32 + lane];
            }
        }
        // dG2 of this split: direct update, or partial + the group's last tile
        const int nt = P.grp_ntiles[g];
        float* part = P.dG2part + ((int64_t)tile * SPLIT + sp) * P.s2_max;
        if (ks == 0) {
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                const int wt = wt0 + 8 * i;
                const int ag = (wt % (A4 / AG)) * AG + lane % AG, jg = (wt / (A4 / AG)) * JL + lane / AG;
#pragma unroll
                for (int ah = 0; ah < 4; ah += 2) {  // two halves of 8 elements (register pressure)
                    int gidx[8];
                    float gv[8];
#pragma unroll
                    for (int a = ah; a < ah + 2; ++a)
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const int aa = ag + A4 * a, jc = jg + JG * c, j2 = jc / R2S, cc = c0 + (jc - j2 * R2S);
                            gidx[(a - ah) * 4 + c] = nt == 1 ? (aa * Q2 + j2) * R2 + cc : aa * NS + jc;
                            gv[(a - ah) * 4 + c] = acc2[i][a][c];
                        }
                    if (nt == 1) {
                        core_update_n<8>(P, G2p, A2p, gidx, gv);  // 8 loads in flight, then the stores
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) part[gidx[e]] = gv[e];
                    }
                }
            }
        }
        if (nt == 1 && P.slice_stamp && P.opt != TT_OPT_GRAD && threadIdx.x == 0 && t == 0) P.slice_stamp[T.p1 + i2] = *P.dstep + 1;
    } else {
        // generic dimensions
        float acc2[kMaxAcc2];
#pragma unroll
        for (int m = 0; m < kMaxAcc2; ++m) acc2[m] = 0.f;
        const int S2 = r1 * Ns;
        for (int u0 = 0; u0 < npairs; u0 += PB) {
            const int nb = min(PB, npairs - u0);
            __syncthreads();
            for (int e = threadIdx.x; e < nb * r1 * q1; e += blockDim.x) {
                const int u = e / (r1 * q1), rem = e - u * (r1 * q1);
                const int a = rem / q1, j1 = rem - a * q1;
                g1s[e] = T.G1[(int64_t)si1[pairbeg[u0 + u]] * (q1 * r1) + j1 * r1 + a];
            }
            for (int e = threadIdx.x; e < nb * Ns * q1; e += blockDim.x) {
                const int u = e / (Ns * q1), rem = e - u * (Ns * q1);
                const int jc = rem / q1, j1 = rem - jc * q1;
                const int j2 = jc / r2s, c = c0 + (jc - j2 * r2s);
                const int kb = pairbeg[u0 + u], ke = pairbeg[u0 + u + 1];
                float acc = 0.f;
                for (int kk = kb; kk < ke; ++kk) {
                    if (kk != kb && rowid[kk] == rowid[kk - 1]) continue;
                    const float* g3 = T.G3 + (int64_t)si3[kk] * (r2 * q3) + c * q3;
                    const float* gr = gs + rowid[kk] * D + (j1 * q2 + j2) * q3;
                    for (int j3 = 0; j3 < q3; ++j3) acc = fmaf(gr[j3], g3[j3], acc);
                }
                dts[(u * Ns + jc) * q1 + j1] = acc;
            }
            __syncthreads();
            for (int e = threadIdx.x; e < nb * q1 * r1; e += blockDim.x) {
                const int u = e / (q1 * r1), ja = e - u * (q1 * r1);
                const int j1 = ja / r1, a = ja - j1 * r1;
                float acc = 0.f;
                for (int jc = 0; jc < Ns; ++jc) acc = fmaf(dts[(u * Ns + jc) * q1 + j1], g2t[jc * (r1 + 4) + a], acc);
                P.Qbuf[((int64_t)(start + pairbeg[u0 + u]) * SPLIT + sp) * P.qs_max + ja] = acc;
            }
#pragma unroll
            for (int m = 0; m < kMaxAcc2; ++m) {
                const int e = threadIdx.x + m * kBwdThreads;
                if (e < S2) {
                    const int a = e / Ns, jc = e - a * Ns;
                    float acc = acc2[m];
                    for (int u = 0; u < nb; ++u)
                        for (int j1 = 0; j1 < q1; ++j1)
                            acc = fmaf(g1s[(u * r1 + a) * q1 + j1], dts[(u * Ns + jc) * q1 + j1], acc);
                    acc2[m] = acc;
                }
            }
        }
        const int nt = P.grp_ntiles[g];
        float* part = P.dG2part + ((int64_t)tile * SPLIT + sp) * P.s2_max;
#pragma unroll
        for (int m = 0; m < kMaxAcc2; ++m) {
            const int e = threadIdx.x + m * kBwdThreads;
            if (e < S2) {
                const int a = e / Ns, jc = e - a * Ns;
                const int j2 = jc / r2s, c = c0 + (jc - j2 * r2s);
                const int ga = (a * q2 + j2) * r2 + c;
                if (nt == 1) core_update(P, G2p, A2p, ga, acc2[m]);
                else part[e] = acc2[m];
            }
        }
        if (nt == 1 && P.slice_stamp && P.opt != TT_OPT_GRAD && threadIdx.x == 0 && t == 0) P.slice_stamp[T.p1 + i2] = *P.dstep + 1;
    }

    // a group of several tiles: k_reduce13 sums its dG2 partials in tile order (a block
    // per group and column half, so that a hot group's sum is not one tile's tail)
}

// Column-split kernels: three blocks per SM for the rank-16/32 classes (registers capped at 80), two otherwise.
template <int DC, int SPLIT>
__global__ void __launch_bounds__(kBwdThreads, SPLIT == 2 ? ((DC == kQ444R32 || DC == kQ444R16) ? 3 : 2) : 1) k_tile_bwd(const __grid_constant__ Params P) {
    pdl_entry();
    if (*P.err) return;  // a device error was recorded: leave every core unchanged
    if ((int)(blockIdx.x / SPLIT) >= *P.ntiles) return;
    extern __shared__ __align__(16) unsigned char smraw[];
    const int g = P.tiles[blockIdx.x / SPLIT].z;
    const TableDev& T = P.tables[P.bin2_tab[g]];
    switch (DC >= 0 ? DC : T.dclass) {
        case kQ444R32: tile_bwd_body<SDims<4, 4, 4, 32, 32>, SPLIT>(P, T, {}, smraw); break;
        case kQ444R16: tile_bwd_body<SDims<4, 4, 4, 16, 16>, SPLIT>(P, T, {}, smraw); break;
        case kQ444R64: tile_bwd_body<SDims<4, 4, 4, 64, 64>, SPLIT>(P, T, {}, smraw); break;
        case kQ448R64: tile_bwd_body<SDims<4, 4, 8, 64, 64>, SPLIT>(P, T, {}, smraw); break;
        default: tile_bwd_body<DDims, SPLIT>(P, T, DDims{T.q1, T.q2, T.q3, T.r1, T.r2}, smraw); break;
    }
}

// Three blocks per SM (the slice count of the workloads fits one wave); without a minimum
// the register target is so low that the partial loads of a thread no longer overlap.
// FFMA backward: dG2 of the (table, i2) groups of several tiles, as work items of
// kGrpChunk elements (group, column half, chunk): the sum of the group's per-tile
// partials in tile order, then the update.  k_reduce13's first blocks (before those of
// the G1 / G3 slices) take the items in turn, so that a hot group (thousands of tiles)
// is spread over many blocks.
constexpr int kGrpChunk = 4 * kBwdThreads;
__device__ void reduce_group_items(const Params& P, int b0, int nblocks) {
    const int SPLIT = P.split;
    const int chunks = (P.s2_max / SPLIT + kGrpChunk - 1) / kGrpChunk;
    const int items = *P.multi_count * SPLIT * chunks;
    for (int item = b0; item < items; item += nblocks) {
        const int gi = item / (SPLIT * chunks), rem = item - gi * (SPLIT * chunks);
        const int sp = rem / chunks, ch = rem - sp * chunks;
        const int g = P.multi_groups[gi];
        const int nt = P.grp_ntiles[g];
        const int t = P.ntab == 1 ? 0 : P.bin2_tab[g];
        const TableDev& T = P.tables[t];
        const int i2 = g - T.base2;
        const int r1 = T.r1, q2 = T.q2, r2 = T.r2;
        const int r2s = r2 / SPLIT, c0 = sp * r2s, Ns = q2 * r2s, n = r1 * Ns;
        float* G2p = T.G2 + (int64_t)i2 * r1 * q2 * r2;
        float* A2p = T.aux[1] ? T.aux[1] + (int64_t)i2 * r1 * q2 * r2 : nullptr;
        int ee[4], gidx[4];
        float sum[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = ch * kGrpChunk + u * blockDim.x + threadIdx.x;
            ee[u] = e < n ? e : -1;
            gidx[u] = -1;
            if (e < n) {
                const int a = e / Ns, jc = e - a * Ns;
                const int j2 = jc / r2s, c = c0 + (jc - j2 * r2s);
                gidx[u] = (a * q2 + j2) * r2 + c;
            }
        }
        sum_partials<4>(P.dG2part + ((int64_t)P.grp_first[g] * SPLIT + sp) * P.s2_max, (int64_t)SPLIT * P.s2_max, nt, ee,
                        sum);
        core_update_nm<4>(P, G2p, A2p, gidx, sum);  // then the four updates' loads together
        if (sp == 0 && ch == 0 && threadIdx.x == 0 && P.slice_stamp && P.opt != TT_OPT_GRAD && t == 0)
            P.slice_stamp[T.p1 + i2] = *P.dstep + 1;
    }
}

__global__ void __launch_bounds__(kBwdThreads, 3) k_reduce13(const __grid_constant__ Params P) {
    pdl_entry();
    if (*P.err) return;  // a device error was recorded: leave every core unchanged
    __shared__ int slots[kReduceSlots];
    __shared__ int sh[40];
    extern __shared__ float sacc[];
    // the group blocks come first, so that they run beside the slice blocks
    const int ngb = (int)gridDim.x - (P.n1 + P.n3);
    if ((int)blockIdx.x < ngb) {
        reduce_group_items(P, blockIdx.x, ngb);
        return;
    }
    const int b = blockIdx.x - ngb;
    const int nb = b < P.n1 ? P.n1 : P.n3;
    const int bb = b < P.n1 ? b : b - P.n1;
    const int* H = b < P.n1 ? P.H1 : P.H3;
    const int start = H[(int64_t)bb * P.nch];
    const int end = (bb + 1 < nb) ? H[(int64_t)(bb + 1) * P.nch] : *P.nincl;
    if (start >= end) return;
    reduce_slice(P, b, slots, sh, sacc);
}

// ------------------------------------------------------------------ summed-gradient update

// Data-parallel step: ranks that hold disjoint shares of the bags and the same
// cores sum their gradients (an all-reduce outside the library); every rank then
// applies the same update here.  An element whose summed gradient is exactly 0 is
// left alone (bit-identical to an element of an untouched slice); the others take
// the optimizer step of core_update.  Four elements per thread (float4 where the
// four lie inside the segment; every segment starts 16-byte aligned).
__global__ void __launch_bounds__(256) k_apply_grads(const __grid_constant__ ApplyArgs a) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
    for (int64_t q = tid; q < a.start[a.nseg]; q += nthreads) {
        int sg = 0;
        while (q >= a.start[sg + 1]) ++sg;
        const int64_t e0 = (q - a.start[sg]) * 4;
        const int64_t n = a.n[sg];
        float* G = a.G[sg];
        const float* g = a.g[sg];
        float* st = a.s[sg];
        bool any = false;
        if (e0 + 4 <= n) {
            const float4 gv = *reinterpret_cast<const float4*>(g + e0);
            const float gg[4] = {gv.x, gv.y, gv.z, gv.w};
            any = gv.x != 0.f || gv.y != 0.f || gv.z != 0.f || gv.w != 0.f;
            if (any) {
                float4 w = *reinterpret_cast<const float4*>(G + e0);
                float ww[4] = {w.x, w.y, w.z, w.w};
                if (a.opt == TT_OPT_ADAGRAD) {
                    float4 sv = *reinterpret_cast<const float4*>(st + e0);
                    float ss[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (gg[i] != 0.f) {
                            ss[i] = fmaf(gg[i], gg[i], ss[i]);
                            ww[i] -= a.lr * gg[i] / (sqrtf(ss[i]) + a.eps);
                        }
                    *reinterpret_cast<float4*>(st + e0) = make_float4(ss[0], ss[1], ss[2], ss[3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (gg[i] != 0.f) ww[i] = fmaf(-a.lr, gg[i], ww[i]);
                }
                *reinterpret_cast<float4*>(G + e0) = make_float4(ww[0], ww[1], ww[2], ww[3]);
            }
        } else {
            for (int64_t e = e0; e < n; ++e) {
                const float gi = g[e];
                if (gi == 0.f) continue;
                any = true;
                if (a.opt == TT_OPT_ADAGRAD) {
                    const float t = fmaf(gi, gi, st[e]);
                    st[e] = t;
                    G[e] -= a.lr * gi / (sqrtf(t) + a.eps);
                } else {
                    G[e] = fmaf(-a.lr, gi, G[e]);
                }
            }
        }
        // exact-copy hot-row cache: the slices changed here are stale from the next pass on
        if (any && a.stamp[sg]) {
            const int64_t s_lo = e0 / a.slice_elems[sg];
            const int64_t s_hi = (e0 + 3 < n ? e0 + 3 : n - 1) / a.slice_elems[sg];
            for (int64_t sl = s_lo; sl <= s_hi; ++sl) a.stamp[sg][sl] = *a.dstep + 1;
        }
    }
}

cudaError_t launch_apply_grads(const ApplyArgs& a, int sms, cudaStream_t s) {
    if (a.nseg == 0 || a.start[a.nseg] == 0) return cudaSuccess;
    const int64_t want = (a.start[a.nseg] + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;
    const unsigned blocks = (unsigned)(want < cap ? want : cap);
    k_apply_grads<<<blocks, 256, 0, s>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ launchers

size_t tile_bwd_smem(const Params& P) {
    return bwd_layout(P.tile_cap, P.D, P.g2s_floats, P.g1s_floats, P.dts_floats).total;
}

int bwd_batch_pairs(int q1, int Ns, int r1) { return bwd_pairs_per_batch(q1, Ns, r1); }

template <int DC, int SPLIT>
static cudaError_t launch_tile_bwd_dc(const Params& P, cudaStream_t s) {
    const size_t smem = tile_bwd_smem(P);
    cudaError_t le = launch_pdl(k_tile_bwd<DC, SPLIT>, dim3((unsigned)P.max_tiles * SPLIT), dim3(kBwdThreads), smem, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

template <int SPLIT>
static cudaError_t launch_tile_bwd_split(const Params& P, cudaStream_t s) {
    switch (P.dclass_all) {
        case kQ444R32: return launch_tile_bwd_dc<kQ444R32, SPLIT>(P, s);
        case kQ444R16: return launch_tile_bwd_dc<kQ444R16, SPLIT>(P, s);
        case kQ444R64: return launch_tile_bwd_dc<kQ444R64, SPLIT>(P, s);
        case kQ448R64: return launch_tile_bwd_dc<kQ448R64, SPLIT>(P, s);
        case kDynamic: return launch_tile_bwd_dc<kDynamic, SPLIT>(P, s);
        default: return launch_tile_bwd_dc<-1, SPLIT>(P, s);
    }
}

cudaError_t launch_tile_bwd(const Params& P, cudaStream_t s) {
    if (P.bwd_tc) return launch_tile_bwd_tc(P, s);
    return P.split == 2 ? launch_tile_bwd_split<2>(P, s) : launch_tile_bwd_split<1>(P, s);
}


template <int SPLIT>
static cudaError_t set_tile_attrs(int max_smem) {
    const void* ks[] = {(const void*)k_tile_bwd<kQ444R32, SPLIT>, (const void*)k_tile_bwd<kQ444R16, SPLIT>,
                        (const void*)k_tile_bwd<kQ444R64, SPLIT>, (const void*)k_tile_bwd<kQ448R64, SPLIT>,
                        (const void*)k_tile_bwd<kDynamic, SPLIT>, (const void*)k_tile_bwd<-1, SPLIT>};
    for (const void* k : ks) {
        cudaError_t e = allow_max_dynamic_smem(k, max_smem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_reduce13(const Params& P, cudaStream_t s) {
    // per-group sums: R S <= 4 kBwdThreads floats while one group's columns fit the block, else S
    const size_t smem = sizeof(float) * std::max<size_t>(4 * kBwdThreads, (size_t)std::max(P.qs_max, P.ps_max));
    // the FFMA backward leaves the dG2 sums of its multi-tile groups to blocks of this launch
    const int groups = P.bwd_tc ? 0 : 2 * P.sms;
    cudaError_t le = launch_pdl(k_reduce13, dim3(P.n1 + P.n3 + groups), dim3(kBwdThreads), smem, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t set_bwd_attributes(int max_smem) {
    cudaError_t e = set_tile_attrs<1>(max_smem);
    if (e == cudaSuccess) e = set_tile_attrs<2>(max_smem);
    if (e == cudaSuccess) e = allow_max_dynamic_smem((const void*)k_reduce13, max_smem);
    if (e == cudaSuccess) e = set_bwd_tc_attributes(max_smem);
    return e;
}

}  // namespace ttemb
