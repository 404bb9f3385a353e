// tt_fwd.cu -- forward contractions and pooling (sm_103a, FP32 FFMA).
//
// FBTT README, "Software Cache": a row is computed from the cores by two
// consecutive small matrix products; the TT-Rec abstract batches them.  Here
//   T[i1,i2] = G1[i1] (q1 x r1) . G2[i2] (r1 x q2 r2)   once per touched pair,
// batched per (table, i2) with the G2 slice in shared memory, and
//   row = T (q1 q2 x r2) . G3[i3] (r2 x q3)            per lookup, pooled per bag
// in registers (tensorflow/addons EmbeddingBag issue: the pre-pool rows are
// never materialised).
#include "tt_dims.cuh"
#include "tt_tc.cuh"

namespace ttemb {

constexpr int kFwdThreads = 256;
constexpr int kListCap = 1024;      // touched i1 handled per round
constexpr int kPoolWarps = 4;       // warps per bag
constexpr int kPoolPer = 3;         // lookups of a warp whose T and G3 loads are in flight together
constexpr int kPoolWarpBag = 4;     // average bag length up to which a warp takes a whole bag
constexpr int kMaxDPerLane = 8;     // generic pool path: D <= 256
constexpr int kScatterParts = kSmallChunk / (kPoolWarps * 32);  // grouping-scatter blocks per chunk
static_assert(kScatterParts * kPoolWarps * 32 == kSmallChunk, "scatter parts cover a chunk");

// ------------------------------------------------------------------ T per pair

struct FwdSmem {
    int* ulist;
    int* sh;
    float* g2s;
    float* g1s;
    unsigned char* tc;  // tensor-core path: operand tiles, mbarrier, tensor-memory address
};

constexpr int kG1Floats = 8192;     // G1 rows gathered at once (pairs x q1 r1 floats)
constexpr size_t kFwdTcBase = 5120;  // byte offset of the tensor-core region (after ulist + sh)
constexpr int kTcTiles = 2;          // 128-row tensor-core tiles per batch (64 pairs)

// Dimension classes whose T = G1 G2 runs on the tensor cores (3xTF32): q1 = 4,
// r1 <= 32, q2 r2 <= 128 (one MMA covers every column; operand tiles fit three
// blocks per SM).
__host__ __device__ constexpr bool fwd_tc_class(int dclass) { return dclass == kQ444R32 || dclass == kQ444R16; }

// fp32 words of the operand tiles: A (kTcTiles x 128 rows x r1) and B (N rows x r1), hi and lo.
int fwd_tc_floats_of(int dclass, int r1, int N) { return fwd_tc_class(dclass) ? 2 * r1 * (kTcTiles * kTcM + N) : 0; }

constexpr size_t kFwdTcCtl = 128;  // mbarrier, tensor-memory address and flag ahead of the tiles

__host__ __device__ inline size_t fwd_smem_bytes(int r1max, int Nmax, int tc_floats) {
    // ulist + sh, G2 slice, G1 rows of up to kG1Floats / (q1 r1) pairs; or the tensor-core tiles
    const size_t ffma = sizeof(int) * (kListCap + 64) + sizeof(float) * (size_t)(r1max + 4) * Nmax + sizeof(float) * kG1Floats;
    const size_t tc = tc_floats > 0 ? kFwdTcBase + kFwdTcCtl + sizeof(float) * (size_t)tc_floats : 0;
    const size_t scan = sizeof(int) * (size_t)kScanSmemInts;  // the small path's histogram-scan blocks
    const size_t m = ffma > tc ? ffma : tc;
    return m > scan ? m : scan;
}

// Tensor-memory columns a tensor-core k_fwd_T block holds: kTcTiles accumulators of q2 r2 columns.
__host__ __device__ constexpr uint32_t fwd_tc_cols(int dclass) {
    return dclass == kQ444R32 ? kTcTiles * 128u : (dclass == kQ444R16 ? kTcTiles * 64u : 0u);
}

// Touched i1 of pair block [i2][base .. base + kListCap) into ulist; returns the count.
__device__ __forceinline__ int touched_list(const Params& P, const TableDev& T, int i2, int base, int* ulist,
                                            int* sh) {
    const int* fl = P.tflag + T.fbase + (int64_t)i2 * T.p1;
    const int end = min(T.p1, base + kListCap);
    const int epoch = *P.epoch;
    int m = 0;
    for (int b = base; b < end; b += blockDim.x) {
        const int i1 = b + threadIdx.x;
        const int f = (i1 < end) && (__ldcg(fl + i1) == epoch);
        int tot;
        const int ex = block_scan_excl(f, sh, &tot);
        if (f) ulist[m + ex] = i1;
        m += tot;
    }
    return m;
}

// g1s[u][0 .. 4 R1) = G1 slice of pair u (contiguous [j1][a]), float4 loads, 4 in flight.
// Pair u starts at u (4 R1 + 4) floats: the pairs read together by one warp fall in
// distinct banks.
template <int R1>
__device__ __forceinline__ void stage_g1_rows(float* g1s, const float* G1, const int* ulist, int gn) {
    constexpr int F4 = R1;  // float4 per slice (4 R1 floats)
    const int n4 = gn * F4;
    for (int base = 0; base < n4; base += 4 * kFwdThreads) {
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = base + q * kFwdThreads + threadIdx.x;
            if (e < n4) v[q] = __ldg(reinterpret_cast<const float4*>(G1 + (int64_t)ulist[e / F4] * (4 * R1)) + e % F4);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = base + q * kFwdThreads + threadIdx.x;
            if (e < n4) reinterpret_cast<float4*>(g1s)[(e / F4) * (F4 + 1) + e % F4] = v[q];
        }
    }
}

// T = G1 G2 for the touched pairs of (table, i2) on the tensor cores.  Batches of
// up to kTcTiles x 32 pairs: A = their G1 slices as rows (u, j1) x r1 (128 rows per
// tile), B = G2^T (q2 r2 rows x r1), D_t = A_t . B^T = 32 T blocks per tile in
// tensor memory (columns [t N, t N + N)); three TF32 MMAs per K step (hi.hi +
// hi.lo + lo.hi).  The G2 slice's bulk copy is issued before the touched-pair scan
// so that the two latencies overlap.
// The block's tensor memory (fwd_tc_cols columns) is allocated at kernel entry.
template <int R1, int NN>
__device__ void fwd_T_group_tc(const Params& P, const TableDev& T, int i2, int half, FwdSmem S) {
    static_assert(R1 % 8 == 0 && R1 <= 32 && NN % 32 == 0 && NN <= 128, "tensor-core tile shapes");
    static_assert(2 * kTcTiles * kTcM * R1 >= (kFwdThreads / 32) * 1024, "write-out buffers fit in the A tiles (hi and lo)");
    constexpr uint32_t kIdesc = tc_idesc_tf32(kTcM, NN);
    constexpr uint32_t kLbo = 128, kSbo = R1 * 32;  // K core matrices / 8-row groups, bytes
    constexpr int kBQ = (R1 / 4) * NN;              // float4 quads of B
    constexpr int kBPer = (kBQ + kFwdThreads - 1) / kFwdThreads;
    constexpr int kPairs = kTcTiles * kTcM / 4;     // pairs per batch
    uint64_t* bar = reinterpret_cast<uint64_t*>(S.tc);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
    int* okflag = reinterpret_cast<int*>(tslot + 1);
    float* Ah = reinterpret_cast<float*>(S.tc + kFwdTcCtl);
    float* Al = Ah + kTcTiles * kTcM * R1;
    float* Bh = Al + kTcTiles * kTcM * R1;
    float* Bl = Bh + NN * R1;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;

    // G2 of this i2 ([a][jc], contiguous) comes by one bulk copy into the A-lo tile, which
    // is free until the first batch; the copy is in flight during the touched-pair scan.
    // Element (jc, a) of B is G2[i2][a][jc].
    uint64_t* gbar = reinterpret_cast<uint64_t*>(S.tc + 16);
    const float* g2raw = Al;
    if (threadIdx.x == 0) {
        mbar_init(gbar, 1);
        bulk_copy_g2s(Al, T.G2 + (int64_t)i2 * R1 * NN, (uint32_t)(R1 * NN * sizeof(float)), gbar);
    }
    bool staged = false, failed = false;
    int nbatch = 0;
    int* list0 = S.ulist;
    for (int base = 0; base < T.p1; base += kListCap) {
        int m = touched_list(P, T, i2, base, list0, S.sh);
        if (P.fwd_split == 2) {
            const int m2 = (m + 1) / 2;
            S.ulist = list0 + half * m2;
            m = half ? m - m2 : m2;
        }
        if (m == 0) continue;
        if (!staged) {
            if (threadIdx.x == 0 && !mbar_wait(gbar, 0, P.wait_polls)) {
                atomicOr(P.err, kErrTimeout);
                mbar_wait(gbar, 0, kTcWaitLimit);  // the copy writes shared memory: let it finish
            }
            __syncthreads();
#pragma unroll
            for (int q = 0; q < kBPer; ++q) {
                const int e = threadIdx.x + q * kFwdThreads;
                if (e < kBQ) {
                    const int jc = e % NN, a4 = e / NN;
                    float x[4], hi[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x[i] = g2raw[(4 * a4 + i) * NN + jc];
                        hi[i] = tf32_round(x[i]);
                    }
                    const int o = tc_off(jc, 4 * a4, R1);
                    *reinterpret_cast<float4*>(Bh + o) = make_float4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<float4*>(Bl + o) =
                        make_float4(x[0] - hi[0], x[1] - hi[1], x[2] - hi[2], x[3] - hi[3]);
                }
            }
            if (threadIdx.x == 32) mbar_init(bar, 1);
            staged = true;
        }
        for (int g0 = 0; g0 < m; g0 += kPairs) {
            const int gn = min(kPairs, m - g0);
            const int ntl = (gn + kTcM / 4 - 1) / (kTcM / 4);  // tiles of this batch
            tc_fence_before();
            __syncthreads();  // the previous batch's tensor-memory reads and A reads are done
            // A: row (u, j1) = G1[i1_u][j1][0 .. r1) (tile u / 32); lanes take 8 rows x 4
            // column quads (rows counted up to a multiple of 8; rows past 4 gn are skipped)
            // (every load of the batch is issued before the first store)
            const int rows8 = (4 * gn + 7) & ~7;
            constexpr int kAPer = kTcTiles * kTcM * (R1 / 4) / kFwdThreads;
            float4 xa[kAPer];
            int oa[kAPer];
#pragma unroll
            for (int q = 0; q < kAPer; ++q) {
                const int e4 = threadIdx.x + q * kFwdThreads;
                const int rl = e4 & 7, a4 = (e4 >> 3) % (R1 / 4), rh = (e4 >> 3) / (R1 / 4);
                const int row = rh * 8 + rl;
                oa[q] = -1;
                xa[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (e4 < rows8 * (R1 / 4) && row < 4 * gn) {
                    const int u = row >> 2, j1 = row & 3;
                    xa[q] = __ldg(reinterpret_cast<const float4*>(T.G1 + (int64_t)S.ulist[g0 + u] * (4 * R1) + j1 * R1) + a4);
                    oa[q] = (row / kTcM) * (kTcM * R1) + tc_off(row % kTcM, 4 * a4, R1);
                }
            }
#pragma unroll
            for (int q = 0; q < kAPer; ++q) {
                if (oa[q] < 0) continue;
                const float4 x = xa[q];
                const float4 hi = make_float4(tf32_round(x.x), tf32_round(x.y), tf32_round(x.z), tf32_round(x.w));
                *reinterpret_cast<float4*>(Ah + oa[q]) = hi;
                *reinterpret_cast<float4*>(Al + oa[q]) = make_float4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
            }
            tc_fence_smem();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (threadIdx.x == 0) {
                const uint32_t bh = smem_addr(Bh), bl = smem_addr(Bl);
                for (int t = 0; t < ntl; ++t) {
                    const uint32_t d = *tslot + (uint32_t)(t * NN);
                    const uint32_t ah = smem_addr(Ah + t * kTcM * R1), al = smem_addr(Al + t * kTcM * R1);
#pragma unroll
                    for (int ks = 0; ks < R1 / 8; ++ks) {
                        const uint32_t ko = ks * 256;
                        tc_mma_tf32(d, tc_desc(ah + ko, kLbo, kSbo), tc_desc(bh + ko, kLbo, kSbo), kIdesc, ks > 0);
                        tc_mma_tf32(d, tc_desc(ah + ko, kLbo, kSbo), tc_desc(bl + ko, kLbo, kSbo), kIdesc, true);
                        tc_mma_tf32(d, tc_desc(al + ko, kLbo, kSbo), tc_desc(bh + ko, kLbo, kSbo), kIdesc, true);
                    }
                }
                tc_commit(bar);
                *okflag = mbar_wait(bar, nbatch & 1, P.wait_polls) ? 1 : 0;
                if (!*okflag) atomicOr(P.err, kErrTimeout);
            }
            __syncthreads();
            tc_fence_after();
            if (!*okflag) {  // gave up: no further MMA, no operand rewrite (uniform: shared flag)
                failed = true;
                break;
            }
            // warp w reads tile w / 4, lanes 32 (w % 4) .. + 31 (its 32 rows), all N columns, 32 at
            // a time; each 32 x 32 block goes through a private shared buffer (the A tiles are free
            // now; float4 chunk q of row r sits at chunk q ^ (r & 7), so neither side has bank
            // conflicts) and leaves as four full 128-byte row segments per store instruction.
            const int t = w >> 2;
            if (*okflag && t < ntl) {
                const int rbase = 32 * (w & 3);  // first row (tensor-memory lane) of this warp in tile t
                const uint32_t taddr = *tslot + ((uint32_t)rbase << 16) + (uint32_t)(t * NN);
                float* buf = Ah + w * 1024;
                const int q = lane & 7;
#pragma unroll 1
                for (int c0 = 0; c0 < NN; c0 += 32) {
                    float v[32];
                    tc_ld32(taddr + c0, v);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<float4*>(buf + lane * 32 + ((k ^ (lane & 7)) << 2)) =
                            make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int r = 4 * i + (lane >> 3);
                        const int row = rbase + r, u = t * (kTcM / 4) + (row >> 2), j1 = row & 3;
                        const float4 x = *reinterpret_cast<const float4*>(buf + r * 32 + ((q ^ (r & 7)) << 2));
                        if (u < gn)
                            *reinterpret_cast<float4*>(P.Tbuf + T.tbase +
                                                       (((int64_t)i2 * T.p1 + S.ulist[g0 + u]) * 4 + j1) * NN + c0 +
                                                       4 * q) = x;
                    }
                    __syncwarp();
                }
            }
            ++nbatch;
        }
        if (failed) break;
    }
    // after a give-up the MMAs of that batch may still run: wait for them (full
    // limit) before the tensor memory is freed
    if (failed && threadIdx.x == 0) mbar_wait(bar, nbatch & 1, kTcWaitLimit);
    // no touched pair: the G2 copy was never waited for; it must land before the block ends
    if (!staged && threadIdx.x == 0 && !mbar_wait(gbar, 0, kTcWaitLimit)) atomicOr(P.err, kErrTimeout);
    tc_fence_before();
    __syncthreads();
    if (w == 0) tc_dealloc(*tslot, kTcTiles * NN);
}

template <class Dm>
__device__ void fwd_T_group(const Params& P, const TableDev& T, const Dm dm, int i2, int half, FwdSmem S) {
    if constexpr (Dm::kStatic) {
        if constexpr (Dm::r1() <= 32 && Dm::q2() * Dm::r2() <= 128) {
            fwd_T_group_tc<Dm::r1(), Dm::q2() * Dm::r2()>(P, T, i2, half, S);
            return;
        }
    }
    const int q1 = dm.q1(), r1 = dm.r1(), N = dm.q2() * dm.r2();
    bool staged = false;
    int* list0 = S.ulist;
    for (int base = 0; base < T.p1; base += kListCap) {
        int m = touched_list(P, T, i2, base, list0, S.sh);
        if (P.fwd_split == 2) {  // this block takes one half of the touched pairs
            const int m2 = (m + 1) / 2;
            S.ulist = list0 + half * m2;
            m = half ? m - m2 : m2;
        }
        if (m == 0) continue;
        if (!staged) {
            const float* src = T.G2 + (int64_t)i2 * r1 * N;
            if constexpr (Dm::kStatic) {
                // transposed: g2t[jc][a] with row stride r1 + 4 (8 loads in flight per thread)
                for (int base = 0; base < r1 * N; base += 8 * kFwdThreads) {
                    float v[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int e = base + q * kFwdThreads + threadIdx.x;
                        v[q] = e < r1 * N ? __ldg(src + e) : 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int e = base + q * kFwdThreads + threadIdx.x;
                        if (e < r1 * N) S.g2s[(e % N) * (r1 + 4) + e / N] = v[q];
                    }
                }
            } else {
                stage_f32<8>(S.g2s, src, r1 * N);
            }
            staged = true;
        }
        if constexpr (Dm::kStatic) {
            // every compiled class has q1 = 4 and q2 r2 % 4 == 0.  Register tile: 4 rows (j1) x 4
            // columns jc = cg + CG c per thread, PS pairs per pass.  A warp covers CL column
            // groups x PL pairs, so each of its shared loads touches at most 8 distinct 16-byte
            // words (G2 rows of stride r1 + 4 and G1 slices of stride 4 r1 + 4 hit distinct
            // banks): one wavefront per load.  Paired FFMA over a: even / odd partial sums.
            constexpr int R1 = Dm::r1(), NN = Dm::q2() * Dm::r2();
            constexpr int CG = NN / 4;
            constexpr int PS = kFwdThreads / CG;
            constexpr int CL = CG < 8 ? CG : 8, PL = 32 / CL, WC = CG / CL;  // lanes: CL x PL; warps: WC per pair block
            static_assert(CG % CL == 0 && (kFwdThreads / 32) % WC == 0 && PS == (kFwdThreads / 32 / WC) * PL, "fwd_T tiles");
            constexpr int GS = R1 + 4;      // g2t row stride
            constexpr int US = 4 * R1 + 4;  // g1s pair stride
            const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
            const int cg = (w % WC) * CL + lane % CL, ps = (w / WC) * PL + lane / CL;
            constexpr int GB = kG1Floats / US;  // pairs gathered at once
            for (int g0 = 0; g0 < m; g0 += GB) {
                const int gn = min(GB, m - g0);
                __syncthreads();
                // g1s[u][j1][a] = G1[i1_u][j1][a]: the pair's contiguous slice, 4 float4 loads in flight
                stage_g1_rows<R1>(S.g1s, T.G1, S.ulist + g0, gn);
                __syncthreads();
                for (int u0 = 0; u0 < gn; u0 += PS) {
                    const int u = u0 + ps;
                    if (u < gn) {
                        float2 acc[4][4];
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int c = 0; c < 4; ++c) acc[j][c] = make_float2(0.f, 0.f);
                        const float* g1 = S.g1s + u * US;
                        const float* g2 = S.g2s + cg * GS;
#pragma unroll 2
                        for (int a = 0; a < R1; a += 4) {
                            float4 x[4], y[4];
#pragma unroll
                            for (int j = 0; j < 4; ++j) x[j] = *reinterpret_cast<const float4*>(g1 + j * R1 + a);
#pragma unroll
                            for (int c = 0; c < 4; ++c) y[c] = *reinterpret_cast<const float4*>(g2 + c * CG * GS + a);
#pragma unroll
                            for (int j = 0; j < 4; ++j)
#pragma unroll
                                for (int c = 0; c < 4; ++c) {
                                    acc[j][c] = __ffma2_rn(make_float2(x[j].x, x[j].y), make_float2(y[c].x, y[c].y), acc[j][c]);
                                    acc[j][c] = __ffma2_rn(make_float2(x[j].z, x[j].w), make_float2(y[c].z, y[c].w), acc[j][c]);
                                }
                        }
                        float* dst = P.Tbuf + T.tbase + ((int64_t)i2 * T.p1 + S.ulist[g0 + u]) * (4 * NN) + cg;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int c = 0; c < 4; ++c) dst[j * NN + c * CG] = acc[j][c].x + acc[j][c].y;
                    }
                }
            }
            __syncthreads();
        } else {
            __syncthreads();
            const int64_t total = (int64_t)m * N;
            for (int64_t e = threadIdx.x; e < total; e += blockDim.x) {
                const int u = (int)(e / N), jc = (int)(e % N);
                const int i1 = S.ulist[u];
                const float* g1 = T.G1 + (int64_t)i1 * q1 * r1;
                float* dst = P.Tbuf + T.tbase + ((int64_t)i2 * T.p1 + i1) * (int64_t)(q1 * N);
                for (int j1 = 0; j1 < q1; ++j1) {
                    float acc = 0.f;
                    for (int a = 0; a < r1; ++a) acc = fmaf(g1[j1 * r1 + a], S.g2s[a * N + jc], acc);
                    dst[j1 * N + jc] = acc;
                }
            }
            __syncthreads();
        }
    }
}

template <int DC>
__global__ void __launch_bounds__(kFwdThreads, 2) k_fwd_T(const __grid_constant__ Params P) {
    extern __shared__ __align__(16) unsigned char smraw[];
    // small path: the first three blocks scan the grouping histograms (first, so
    // that they are resident from the start; they are the longest blocks)
    const int nscan = P.small ? 3 : 0;
    if ((int)blockIdx.x < nscan) {
        pdl_entry();
        scan_digit_block(P, blockIdx.x, (int*)smraw);
        return;
    }
    // the handle's constant tables may be read before the previous kernel completes
    const int g = (blockIdx.x - nscan) / P.fwd_split, half = (blockIdx.x - nscan) % P.fwd_split;
    const TableDev& T = P.tables[P.bin2_tab[g]];
    const int i2 = g - T.base2;
    // Tensor memory first: while a block holds its allocation permit, no further
    // block of a tensor-memory kernel is placed on the SM, so the permit is
    // released at once.  (The previous kernels of the library hold no tensor memory.)
    const uint32_t tcols = fwd_tc_cols(DC >= 0 ? DC : T.dclass);
    if (tcols != 0 && threadIdx.x < 32) tc_alloc(reinterpret_cast<uint32_t*>(smraw + kFwdTcBase + 8), tcols);
    if (P.small) {  // the decode blocks' touched flags, not the end of the decode grid
        pdl_launch_dependents();
        wait_decode_flags(P);
    } else {
        pdl_entry();
    }
    FwdSmem S;
    S.ulist = (int*)smraw;
    S.sh = S.ulist + kListCap;
    S.g2s = (float*)(S.sh + 64);
    S.g1s = S.g2s + (size_t)(P.r1_max + 4) * P.N_max;
    S.tc = smraw + kFwdTcBase;
    switch (DC >= 0 ? DC : T.dclass) {
        case kQ444R32: fwd_T_group(P, T, SDims<4, 4, 4, 32, 32>{}, i2, half, S); break;
        case kQ444R16: fwd_T_group(P, T, SDims<4, 4, 4, 16, 16>{}, i2, half, S); break;
        case kQ444R64: fwd_T_group(P, T, SDims<4, 4, 4, 64, 64>{}, i2, half, S); break;
        case kQ448R64: fwd_T_group(P, T, SDims<4, 4, 8, 64, 64>{}, i2, half, S); break;
        default: fwd_T_group(P, T, DDims{T.q1, T.q2, T.q3, T.r1, T.r2}, i2, half, S); break;
    }
}

// ------------------------------------------------------------------ pooling

__device__ __forceinline__ const float* t_of_pair(const Params& P, const TableDev& T, int i2, int i1) {
    i2 = TT_DCHECK(P, i2, T.p2);
    i1 = TT_DCHECK(P, i1, T.p1);
    return P.Tbuf + T.tbase + ((int64_t)i2 * T.p1 + i1) * (int64_t)(T.q1 * T.q2 * T.r2);
}

// Exact-copy cache: the lookups that the decode chose to refresh a stale cached row
// (one per row and pass, lk_hit = -2 - slot) recompute the row from T and G3 and
// write it back with the pass's stamp.  A warp per lookup, lanes over columns.
// first / step: the warp's share of the bag's lookups.
__device__ void cache_refresh_rows(const Params& P, const TableDev& T, int64_t first, int64_t hi, int step) {
    const int lane = threadIdx.x & 31;
    const int q3 = T.q3, r2 = T.r2, D = T.D;
    for (int64_t n = first; n < hi; n += step) {
        const int code = P.lk_hit[n];
        if (code > -2) continue;
        const int64_t slot = -2 - (int64_t)code;
        const float* Tp = t_of_pair(P, T, P.lk_i2[n], P.lk_i1[n]);
        const float* g3 = T.G3 + (int64_t)P.lk_i3[n] * r2 * q3;
        for (int j = lane; j < D; j += 32) {
            const int j12 = j / q3, j3 = j - j12 * q3;
            float a = 0.f;
            for (int c = 0; c < r2; ++c) a = fmaf(Tp[j12 * r2 + c], g3[c * q3 + j3], a);
            __stcg(P.cache_vals + slot * D + j, a);
        }
        if (lane == 0) P.cache_stamp[slot] = *P.dstep;
    }
}

// Static fast path: lanes = 2 output halves (lj) x 16 contraction lanes (lc);
// lane (lj, lc) sums c = lc, lc + 16, ... for the outputs j = lj * D/2 + v.
// After the bag, a reduce-scatter over the 16 lc lanes leaves V = D/32 sums
// per lane.  WARP: one warp takes the whole bag and stores its row (short bags);
// else the block's kPoolWarps warps share the bag and sum through `red`.
template <class Dm, bool WARP, bool CACHE>
__device__ void pool_bag_static(const Params& P, const TableDev& T, int64_t bag, int64_t lo, int64_t hi,
                                float* red) {
    constexpr int Q3 = Dm::q3(), R2 = Dm::r2(), Q12 = Dm::q1() * Dm::q2();
    constexpr int D = Q12 * Q3, H = D / 2, J12H = Q12 / 2, NC = R2 / 16;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int lc = lane & 15, lj = lane >> 4;
    float acc[H];
#pragma unroll
    for (int v = 0; v < H; ++v) acc[v] = 0.f;
    {
        // warp w takes lookups lo + w + kPoolWarps l; lane l first loads the indices of the
        // warp's l-th lookup of a round (one pass), then the warp walks them PP at a time
        constexpr int NW = WARP ? 1 : kPoolWarps;  // warps sharing the bag
        // lookups in flight per warp: short bags (WARP) get one, and more warps per SM
        constexpr int PP = WARP ? 1 : kPoolPer;
        const int wb = WARP ? 0 : w;                // this warp's rank among them
        for (int64_t nb0 = lo; nb0 < hi; nb0 += 32 * NW) {
            const int64_t nl = nb0 + wb + (int64_t)NW * lane;
            int i1l = 0, i2l = 0, i3l = 0;
            float sl = 0.f;
            if (nl < hi) {
                i1l = P.lk_i1[nl];
                i2l = P.lk_i2[nl];
                i3l = P.lk_i3[nl];
                sl = P.lk_s[nl];
                if (CACHE && P.lk_hit[nl] >= 0) sl = 0.f;  // read from the cache below
            }
            const int64_t left = hi - nb0 - wb;  // this warp's lookups nb0 + wb + NW l < hi
            const int64_t c64 = left <= 0 ? 0 : (left + NW - 1) / NW;
            const int cnt = c64 > 32 ? 32 : (int)c64;
            for (int l = 0; l < cnt; l += PP) {
                // PP lookups of this warp: their T and G3 values are all in flight together
                int li[PP];
                float sv[PP];
                const float* Tp[PP];
                const float* g3p[PP];
#pragma unroll
                for (int q = 0; q < PP; ++q) {
                    const bool valid = l + q < cnt;
                    li[q] = valid ? l + q : l;
                    const int i1q = __shfl_sync(0xffffffffu, i1l, li[q]), i2q = __shfl_sync(0xffffffffu, i2l, li[q]);
                    const int i3q = __shfl_sync(0xffffffffu, i3l, li[q]);
                    const float sq = __shfl_sync(0xffffffffu, sl, li[q]);
                    sv[q] = valid ? sq : 0.f;
                    Tp[q] = t_of_pair(P, T, i2q, i1q) + lj * J12H * R2;
                    g3p[q] = T.G3 + (int64_t)i3q * R2 * Q3;
                }
                float tv[PP][J12H][NC], gv[PP][NC][Q3];
#pragma unroll
                for (int q = 0; q < PP; ++q)
#pragma unroll
                    for (int k = 0; k < NC; ++k) {
                        const int c = lc + 16 * k;
#pragma unroll
                        for (int j = 0; j < J12H; ++j) tv[q][j][k] = __ldg(Tp[q] + j * R2 + c);
#pragma unroll
                        for (int j3 = 0; j3 < Q3; j3 += 4) {
                            const float4 x = __ldg(reinterpret_cast<const float4*>(g3p[q] + c * Q3 + j3));
                            gv[q][k][j3] = x.x; gv[q][k][j3 + 1] = x.y; gv[q][k][j3 + 2] = x.z; gv[q][k][j3 + 3] = x.w;
                        }
                    }
#pragma unroll
                for (int j = 0; j < J12H; ++j)
#pragma unroll
                    for (int j3 = 0; j3 < Q3; ++j3) {
                        float a = acc[j * Q3 + j3];
#pragma unroll
                        for (int q = 0; q < PP; ++q) {
                            float x = 0.f;
#pragma unroll
                            for (int k = 0; k < NC; ++k) x = fmaf(tv[q][j][k], gv[q][k][j3], x);
                            a = fmaf(sv[q], x, a);
                        }
                        acc[j * Q3 + j3] = a;
                    }
            }
        }
    }
    // reduce-scatter over the 16 lc lanes: each stage halves the vector
#pragma unroll
    for (int o = 8, len = H; o >= 1; o >>= 1, len >>= 1) {
        const bool up = (lc & o) != 0;
#pragma unroll
        for (int v = 0; v < len / 2; ++v) {
            const float send = up ? acc[v] : acc[v + len / 2];
            const float keep = up ? acc[v + len / 2] : acc[v];
            acc[v] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    constexpr int V = H / 16;
    const int64_t first = lo + (WARP ? 0 : w);
    const int step = WARP ? 1 : kPoolWarps;
    if (CACHE) {  // cache hits: s times the cached value, V columns a lane
        for (int64_t n = first; n < hi; n += step) {
            const int slot = P.lk_hit[n];
            if (slot < 0) continue;
            const float sh = P.lk_sh[n];
            const float* cv = P.cache_vals + (int64_t)slot * D + lj * H + lc * V;
#pragma unroll
            for (int v = 0; v < V; ++v) acc[v] = fmaf(sh, __ldcg(cv + v), acc[v]);
        }
    }
    if (CACHE && !P.cache_train) cache_refresh_rows(P, T, first, hi, step);
    if constexpr (WARP) {
        float* o = P.out + bag * D + lj * H + lc * V;
#pragma unroll
        for (int v = 0; v < V; ++v) o[v] = acc[v];
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v) red[w * D + lj * H + lc * V + v] = acc[v];
        __syncthreads();
        for (int j = threadIdx.x; j < D; j += blockDim.x) {
            float sum = 0.f;
#pragma unroll
            for (int ww = 0; ww < kPoolWarps; ++ww) sum += red[ww * D + j];
            P.out[bag * D + j] = sum;
        }
    }
}

// Generic path: lanes over output columns, loop over c.  WARP as for the static path.
template <bool WARP, bool CACHE>
__device__ void pool_bag_generic(const Params& P, const TableDev& T, int64_t bag, int64_t lo, int64_t hi,
                                 float* red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int q3 = T.q3, r2 = T.r2, D = T.D;
    const int64_t first = lo + (WARP ? 0 : w);
    const int step = WARP ? 1 : kPoolWarps;
    float acc[kMaxDPerLane];
#pragma unroll
    for (int m = 0; m < kMaxDPerLane; ++m) acc[m] = 0.f;
    for (int64_t n = first; n < hi; n += step) {
        const int i1 = P.lk_i1[n], i2 = P.lk_i2[n], i3 = P.lk_i3[n];
        const float s = (CACHE && P.lk_hit[n] >= 0) ? 0.f : P.lk_s[n];  // a hit reads the cache below
        const float* Tp = t_of_pair(P, T, i2, i1);
        const float* g3 = T.G3 + (int64_t)i3 * r2 * q3;
#pragma unroll
        for (int m = 0; m < kMaxDPerLane; ++m) {
            const int j = lane + 32 * m;
            float a = 0.f;
            if (j < D) {
                const int j12 = j / q3, j3 = j - j12 * q3;
                for (int c = 0; c < r2; ++c) a = fmaf(Tp[j12 * r2 + c], g3[c * q3 + j3], a);
            }
            acc[m] = fmaf(s, a, acc[m]);
        }
        if (CACHE) {  // a cache hit: s times the cached value
            const int slot2 = P.lk_hit[n];
            if (slot2 >= 0) {
                const float sh = P.lk_sh[n];
#pragma unroll
                for (int m = 0; m < kMaxDPerLane; ++m) {
                    const int j = lane + 32 * m;
                    if (j < D) acc[m] = fmaf(sh, __ldcg(P.cache_vals + (int64_t)slot2 * D + j), acc[m]);
                }
            }
        }
    }
    if (CACHE && !P.cache_train) cache_refresh_rows(P, T, first, hi, step);
    if constexpr (WARP) {
#pragma unroll
        for (int m = 0; m < kMaxDPerLane; ++m) {
            const int j = lane + 32 * m;
            if (j < D) P.out[bag * D + j] = acc[m];
        }
    } else {
#pragma unroll
        for (int m = 0; m < kMaxDPerLane; ++m) {
            const int j = lane + 32 * m;
            if (j < D) red[w * D + j] = acc[m];
        }
        __syncthreads();
        for (int j = threadIdx.x; j < D; j += blockDim.x) {
            float sum = 0.f;
            for (int ww = 0; ww < kPoolWarps; ++ww) sum += red[ww * D + j];
            P.out[bag * D + j] = sum;
        }
    }
}

template <int DC, bool WARP, bool CACHE>
__device__ __forceinline__ void pool_one_bag(const Params& P, int64_t bag, float* red) {
    const TableDev& T = P.tables[table_of_bag(P, (int)bag)];
    int64_t lo = P.off[bag], hi = P.off[bag + 1];
    lo = lo < 0 ? 0 : (lo > P.nnz ? P.nnz : lo);
    hi = hi < lo ? lo : (hi > P.nnz ? P.nnz : hi);
    // DC = -1: mixed classes of width 64 (no q3 = 8 class); -2: mixed, another width
    const int dc = DC >= 0 ? DC : T.dclass;
    switch (dc) {
        case kQ444R32: if constexpr (DC != -2) pool_bag_static<SDims<4, 4, 4, 32, 32>, WARP, CACHE>(P, T, bag, lo, hi, red); break;
        case kQ444R16: if constexpr (DC != -2) pool_bag_static<SDims<4, 4, 4, 16, 16>, WARP, CACHE>(P, T, bag, lo, hi, red); break;
        case kQ444R64: if constexpr (DC != -2) pool_bag_static<SDims<4, 4, 4, 64, 64>, WARP, CACHE>(P, T, bag, lo, hi, red); break;
        case kQ448R64: if constexpr (DC != -1) pool_bag_static<SDims<4, 4, 8, 64, 64>, WARP, CACHE>(P, T, bag, lo, hi, red); break;
        default: pool_bag_generic<WARP, CACHE>(P, T, bag, lo, hi, red); break;
    }
}

// MODE & 1 (short bags, on average at most kPoolWarpBag lookups): one warp per bag;
// else one block of kPoolWarps warps per bag, the warps share the bag's lookups.
// MODE & 2: the handle has a hot-row cache.  Blocks past the bags' run the grouping
// scatter of the small path.  DC >= 0: every table of the handle has dimension class
// DC; DC < 0: per table.
template <int DC, int MODE>
__global__ void __launch_bounds__(kPoolWarps * 32) k_pool(const __grid_constant__ Params P) {
    pdl_entry();
    __shared__ float red[kPoolWarps * kMaxD];
    constexpr bool WARP = (MODE & 1) != 0, CACHE = (MODE & 2) != 0;
    const int64_t nbb = WARP ? (P.nbags + kPoolWarps - 1) / kPoolWarps : P.nbags;  // bag blocks
    if ((int64_t)blockIdx.x >= nbb) {  // small path: extra blocks scatter the lookups of part of a chunk
        const int e = (int)(blockIdx.x - nbb);
        scatter_chunk(P, e / kScatterParts, e % kScatterParts);
        return;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(P.epoch, 1);  // k_fwd_T has finished reading it
    if constexpr (WARP) {
        const int64_t bag = (int64_t)blockIdx.x * kPoolWarps + (threadIdx.x >> 5);
        if (bag < P.nbags) pool_one_bag<DC, true, CACHE>(P, bag, red);
    } else {
        pool_one_bag<DC, false, CACHE>(P, blockIdx.x, red);
    }
}

// Decompress the cached rows of table 0 (chain product, fp32).
__global__ void k_cache_fill(const __grid_constant__ Params P) {
    pdl_entry();
    const int lane = threadIdx.x & 31;
    const int64_t slot = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (slot >= P.cache_n) return;
    const TableDev& T = P.tables[0];
    const int64_t row = P.cache_rows[slot];
    if (row < 0) return;  // empty way of a set-associative cache
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
    if (lane == 0) P.cache_stamp[slot] = *P.dstep;
}

// ------------------------------------------------------------------ launchers

int dim_class_of(int q1, int q2, int q3, int r1, int r2) { return dim_class(q1, q2, q3, r1, r2); }


template <int DC>
static cudaError_t launch_fwd_T_dc(const Params& P, cudaStream_t s) {
    const size_t smem = fwd_smem_bytes(P.r1_max, P.N_max, P.fwd_tc_floats);
    cudaError_t le = launch_pdl(k_fwd_T<DC>, dim3(P.n2 * P.fwd_split + (P.small ? 3 : 0)), dim3(kFwdThreads), smem, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t launch_fwd_T(const Params& P, cudaStream_t s) {
    switch (P.dclass_all) {
        case kQ444R32: return launch_fwd_T_dc<kQ444R32>(P, s);
        case kQ444R16: return launch_fwd_T_dc<kQ444R16>(P, s);
        case kQ444R64: return launch_fwd_T_dc<kQ444R64>(P, s);
        case kQ448R64: return launch_fwd_T_dc<kQ448R64>(P, s);
        case kDynamic: return launch_fwd_T_dc<kDynamic>(P, s);
        default: return launch_fwd_T_dc<-1>(P, s);
    }
}

template <int DC, int MODE>
static cudaError_t launch_pool_mode(const Params& P, cudaStream_t s) {
    const int64_t nbb = (MODE & 1) ? (P.nbags + kPoolWarps - 1) / kPoolWarps : P.nbags;
    cudaError_t le = launch_pdl(k_pool<DC, MODE>, dim3((unsigned)(nbb + (P.small ? (int64_t)P.nch * kScatterParts : 0))),
                                dim3(kPoolWarps * 32), 0, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

// The hot-row cache exists on single-table handles only: no cached variant of the
// mixed-class kernels.
template <int DC>
static cudaError_t launch_pool_dc(const Params& P, cudaStream_t s) {
    const int warp = P.nnz <= (int64_t)kPoolWarpBag * P.nbags ? 1 : 0;
    if constexpr (DC >= 0) {
        if (P.cache_n > 0) return warp ? launch_pool_mode<DC, 3>(P, s) : launch_pool_mode<DC, 2>(P, s);
    }
    return warp ? launch_pool_mode<DC, 1>(P, s) : launch_pool_mode<DC, 0>(P, s);
}

cudaError_t launch_pool(const Params& P, cudaStream_t s) {
    switch (P.dclass_all) {
        case kQ444R32: return launch_pool_dc<kQ444R32>(P, s);
        case kQ444R16: return launch_pool_dc<kQ444R16>(P, s);
        case kQ444R64: return launch_pool_dc<kQ444R64>(P, s);
        case kQ448R64: return launch_pool_dc<kQ448R64>(P, s);
        case kDynamic: return launch_pool_dc<kDynamic>(P, s);
        default: return P.D == 64 ? launch_pool_dc<-1>(P, s) : launch_pool_dc<-2>(P, s);
    }
}

// Rows [row0, row0 + nrows) of one table as dense rows (warp per row, chain
// product G1[i1] G2[i2] G3[i3], fp32); rows are independent.
__global__ void k_full_weight(const TableDev* __restrict__ tables, int t, int64_t row0, int64_t nrows,
                              float* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t k = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (k >= nrows) return;
    const TableDev& T = tables[t];
    const int64_t row = row0 + k;
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
        out[k * D + j] = acc;
    }
}

cudaError_t launch_full_weight(const TableDev* tables, int t, int64_t row0, int64_t nrows, float* out,
                               cudaStream_t s) {
    const int64_t blocks = (nrows + 7) / 8;
    k_full_weight<<<dim3((unsigned)blocks), dim3(256), 0, s>>>(tables, t, row0, nrows, out);
    return cudaGetLastError();
}

// Trainable cache rows, backward (FBTT README, "Parameters": sparse, the gradient
// w.r.t. the cache).  The gradient of cached value [slot][j] is the sum, over the hits n
// of the slot, of sh_n * grad_out[bag_n][j].  The sum is taken in 64-bit fixed point with
// integer atomics, so it does not depend on the order of the hits: each term (the fp32
// product) is rounded to a multiple of 2^-S.  With every |term| <= 2^e and at most 2^k
// terms, S = 61 - e - k keeps every partial sum within 2^61.

// 2^x as a float (x within the normal exponent range).
__device__ __forceinline__ float pow2f(int x) { return __int_as_float((x + 127) << 23); }

// v * 2^x, exact for the ranges used here: two power-of-two factors within the
// normal exponent range, so neither product overflows while |v * 2^x| < 2^62.
__device__ __forceinline__ float scale2(float v, int x) {
    const int a = x / 2;
    return v * pow2f(a) * pow2f(x - a);
}

// S of the step, or INT_MIN when a bound is not finite.  Every hit term satisfies
// |sh * g| <= max|sh| * max|g| < 2^(eS + eG) (the exponents of the two maxima); fp32
// terms are 0 or >= 2^-149, so e = max(eS + eG, -149) and S = 61 - e - k, nnz <= 2^k.
__device__ __forceinline__ int cache_fixed_shift(const Params& P) {
    const int EG = (int)((P.cache_gmax[0] >> 23) & 255u), ES = (int)((P.cache_gmax[3] >> 23) & 255u);
    if (EG == 255 || ES == 255) return INT_MIN;
    int e = ((EG == 0 ? 1 : EG) - 126) + ((ES == 0 ? 1 : ES) - 126);
    e = e < -149 ? -149 : e;
    int k = 0;
    while (((int64_t)1 << k) < P.nnz) ++k;
    return 61 - e - k;
}

// max|grad_out| into cache_gmax[0] and max|sh| over the hits into cache_gmax[3]
// (a non-finite value counts as infinity; both words were left at 0 by the previous
// step's k_cache_apply); the touched-slot list starts empty.
__global__ void __launch_bounds__(256) k_cache_gmax(const __grid_constant__ Params P) {
    pdl_entry();
    __shared__ float wm[2][8];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (int64_t)gridDim.x * blockDim.x;
    if (gt == 0) P.cache_gmax[2] = 0u;
    const float inf = __int_as_float(0x7f800000);
    float mg = 0.f, ms = 0.f;
    const int64_t ng = (int64_t)P.nbags * P.D;
    for (int64_t i = gt; i < ng; i += stride) {
        const float a = fabsf(__ldg(P.grad_out + i));
        mg = fmaxf(mg, a <= 3.402823466e38f ? a : inf);
    }
    for (int64_t n = gt; n < P.nnz; n += stride) {
        const float a = P.lk_hit[n] >= 0 ? fabsf(P.lk_sh[n]) : 0.f;
        ms = fmaxf(ms, a <= 3.402823466e38f ? a : inf);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, o));
        ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, o));
    }
    if (lane == 0) {
        wm[0][w] = mg;
        wm[1][w] = ms;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int v = 1; v < (int)(blockDim.x >> 5); ++v) {
            mg = fmaxf(mg, wm[0][v]);
            ms = fmaxf(ms, wm[1][v]);
        }
        if (mg > 0.f) atomicMax(P.cache_gmax, __float_as_uint(mg));
        if (ms > 0.f) atomicMax(P.cache_gmax + 3, __float_as_uint(ms));
    }
}

// Fixed-point sums of the hit terms into cache_acc.  A block takes kCacheChunk
// consecutive lookups and sorts its hits by slot in shared memory; a warp sums each
// slot's run in registers (term = round(fl(sh * g) * 2^S), four hits' loads in
// flight at a time) and adds it with one integer atomic per column, so a hot row
// costs one atomic per block and column.  The first block to touch a slot appends it
// to the touched list (one list reservation per block).  Block 0 passes S on in
// cache_gmax[1].  DPL = columns per lane (D <= 32 DPL).
constexpr int kCacheChunk = 256;

template <int DPL>
__global__ void __launch_bounds__(kCacheChunk) k_cache_acc(const __grid_constant__ Params P) {
    pdl_entry();
    __shared__ unsigned long long key[kCacheChunk];  // (slot << 32) | position in the chunk
    __shared__ float shs[kCacheChunk];
    __shared__ int bags[kCacheChunk];
    __shared__ int heads[kCacheChunk];
    __shared__ int fresh[kCacheChunk];  // slots this block touched first
    __shared__ int wcnt[2][kCacheChunk / 32];
    __shared__ int nhead, nhit, nfresh, fbase;
    const int S = cache_fixed_shift(P);
    if (blockIdx.x == 0 && threadIdx.x == 0) P.cache_gmax[1] = (unsigned)S;
    const bool finite = S != INT_MIN;  // else the touched slots get NaN from k_cache_apply
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, D = P.D;
    for (int64_t c0 = (int64_t)blockIdx.x * kCacheChunk; c0 < P.nnz; c0 += (int64_t)gridDim.x * kCacheChunk) {
        const int64_t n = c0 + tid;
        const int slot = n < P.nnz ? P.lk_hit[n] : -1;
        if (slot >= 0) {
            shs[tid] = P.lk_sh[n];
            bags[tid] = P.lk_bag[n];
        }
        key[tid] = ((unsigned long long)(slot >= 0 ? (unsigned)slot : 0xffffffffu) << 32) | (unsigned)tid;
        if (tid == 0) nfresh = 0;
        __syncthreads();
        // bitonic sort of the chunk's keys, ascending: hits first, runs of equal slots
        for (int k = 2; k <= kCacheChunk; k <<= 1)
            for (int j = k >> 1; j > 0; j >>= 1) {
                const int o = tid ^ j;
                if (o > tid) {
                    const unsigned long long a = key[tid], b = key[o];
                    if (((tid & k) == 0) == (a > b)) {
                        key[tid] = b;
                        key[o] = a;
                    }
                }
                __syncthreads();
            }
        // run heads in sorted order (ballot + prefix over the warps)
        const unsigned ks = (unsigned)(key[tid] >> 32);
        const bool hit = ks != 0xffffffffu;
        const bool head = hit && (tid == 0 || (unsigned)(key[tid - 1] >> 32) != ks);
        const unsigned hb = __ballot_sync(0xffffffffu, head), xb = __ballot_sync(0xffffffffu, hit);
        if (lane == 0) {
            wcnt[0][w] = __popc(hb);
            wcnt[1][w] = __popc(xb);
        }
        __syncthreads();
        int off = 0;
        for (int v = 0; v < w; ++v) off += wcnt[0][v];
        if (head) heads[off + __popc(hb & lanemask_lt())] = tid;
        if (tid == 0) {
            int a = 0, b = 0;
            for (int v = 0; v < kCacheChunk / 32; ++v) {
                a += wcnt[0][v];
                b += wcnt[1][v];
            }
            nhead = a;
            nhit = b;
        }
        __syncthreads();
        for (int h = w; h < nhead; h += kCacheChunk / 32) {
            const int i0 = heads[h], i1 = h + 1 < nhead ? heads[h + 1] : nhit;
            const unsigned sl = (unsigned)(key[i0] >> 32);
            long long acc[DPL];
#pragma unroll
            for (int m = 0; m < DPL; ++m) acc[m] = 0;
            int i = i0;
            if (finite) {
                for (; i + 4 <= i1; i += 4) {
                    float gv[4][DPL], sv[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int t = (int)(key[i + q] & 0xffffffffu);
                        sv[q] = shs[t];
                        const float* g = P.grad_out + (int64_t)bags[t] * D;
#pragma unroll
                        for (int m = 0; m < DPL; ++m) gv[q][m] = lane + 32 * m < D ? g[lane + 32 * m] : 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int m = 0; m < DPL; ++m) acc[m] += __float2ll_rn(scale2(sv[q] * gv[q][m], S));
                }
                for (; i < i1; ++i) {
                    const int t = (int)(key[i] & 0xffffffffu);
                    const float sh = shs[t];
                    const float* g = P.grad_out + (int64_t)bags[t] * D;
#pragma unroll
                    for (int m = 0; m < DPL; ++m)
                        if (lane + 32 * m < D) acc[m] += __float2ll_rn(scale2(sh * g[lane + 32 * m], S));
                }
            }
            unsigned long long* dst = P.cache_acc + (int64_t)sl * D;
#pragma unroll
            for (int m = 0; m < DPL; ++m)
                if (lane + 32 * m < D) atomicAdd(dst + lane + 32 * m, (unsigned long long)acc[m]);
        }
        // touched-slot bookkeeping, a thread per run
        if (tid < nhead) {
            const int sl = (int)(key[heads[tid]] >> 32);
            if (P.cache_touch[sl] == 0 && atomicExch(P.cache_touch + sl, 1) == 0) fresh[atomicAdd(&nfresh, 1)] = sl;
        }
        __syncthreads();
        if (tid == 0 && nfresh > 0) fbase = (int)atomicAdd(P.cache_gmax + 2, (unsigned)nfresh);
        __syncthreads();
        if (tid < nfresh) P.cache_list[fbase + tid] = fresh[tid];
        __syncthreads();
    }
}

// The optimizer step of the touched cached values (SGD, Adagrad, or the gradient kept
// for reading): a warp per listed slot, lanes over columns, two slots' loads in flight;
// the accumulators, touch flags and the two bound words return to zero.  DPL =
// columns per lane (D <= 32 DPL).
template <int DPL>
__device__ __forceinline__ void cache_apply_slot(const Params& P, int slot, int S, const unsigned long long* a,
                                                 const float* v, const float* st) {
    const int lane = threadIdx.x & 31, D = P.D;
#pragma unroll
    for (int m = 0; m < DPL; ++m) {
        const int j = lane + 32 * m;
        if (j >= D) continue;
        const int64_t e = (int64_t)slot * D + j;
        const float g = S == INT_MIN ? __int_as_float(0x7fffffff) : scale2(__ll2float_rn((long long)a[m]), -S);
        P.cache_acc[e] = 0ull;
        if (P.opt == TT_OPT_SGD) {
            P.cache_vals[e] = fmaf(-P.lr, g, v[m]);
        } else if (P.opt == TT_OPT_ADAGRAD) {
            const float t = fmaf(g, g, st[m]);
            P.cache_state[e] = t;
            P.cache_vals[e] = v[m] - P.lr * g / (sqrtf(t) + P.eps);
        } else {
            P.cache_grad[e] = g;
        }
    }
    if (lane == 0) P.cache_touch[slot] = 0;
}

template <int DPL>
__global__ void __launch_bounds__(256) k_cache_apply(const __grid_constant__ Params P) {
    pdl_entry();
    const int S = (int)P.cache_gmax[1];
    const int cnt = (int)P.cache_gmax[2];
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        P.cache_gmax[0] = 0u;
        P.cache_gmax[3] = 0u;
    }
    const int lane = threadIdx.x & 31, D = P.D;
    const int nw = gridDim.x * (blockDim.x >> 5);
    const bool adagrad = P.opt == TT_OPT_ADAGRAD, update = P.opt != TT_OPT_GRAD;
    for (int i = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < cnt; i += 2 * nw) {
        const int s0 = P.cache_list[i];
        const int s1 = i + nw < cnt ? P.cache_list[i + nw] : -1;
        unsigned long long a0[DPL], a1[DPL];
        float v0[DPL], v1[DPL], t0[DPL], t1[DPL];
#pragma unroll
        for (int m = 0; m < DPL; ++m) {
            const int j = lane + 32 * m;
            const bool in = j < D;
            const int64_t e0 = (int64_t)s0 * D + j, e1 = (int64_t)s1 * D + j;
            a0[m] = in ? P.cache_acc[e0] : 0ull;
            v0[m] = in && update ? P.cache_vals[e0] : 0.f;
            t0[m] = in && adagrad ? P.cache_state[e0] : 0.f;
            a1[m] = in && s1 >= 0 ? P.cache_acc[e1] : 0ull;
            v1[m] = in && s1 >= 0 && update ? P.cache_vals[e1] : 0.f;
            t1[m] = in && s1 >= 0 && adagrad ? P.cache_state[e1] : 0.f;
        }
        cache_apply_slot<DPL>(P, s0, S, a0, v0, t0);
        if (s1 >= 0) cache_apply_slot<DPL>(P, s1, S, a1, v1, t1);
    }
}

cudaError_t launch_cache_fill(const Params& P, cudaStream_t s) {
    const int64_t blocks = (P.cache_n + 7) / 8;
    cudaError_t le = launch_pdl(k_cache_fill, dim3((unsigned)blocks), dim3(256), 0, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

static int64_t grid_for(int64_t units, int per_block, int64_t cap) {
    const int64_t b = (units + per_block - 1) / per_block;
    return b < 1 ? 1 : (b > cap ? cap : b);
}

cudaError_t launch_cache_gmax(const Params& P, cudaStream_t s) {
    const int64_t b = grid_for(std::max<int64_t>(P.nnz, (int64_t)P.nbags * P.D), 256 * 4, (int64_t)P.sms * 2);
    cudaError_t le = launch_pdl(k_cache_gmax, dim3((unsigned)b), dim3(256), 0, s, P);
    return le != cudaSuccess ? le : cudaGetLastError();
}

cudaError_t launch_cache_acc(const Params& P, cudaStream_t s) {
    const int64_t b = grid_for(P.nnz, kCacheChunk, (int64_t)P.sms * 8);
    cudaError_t le = P.D <= 64 ? launch_pdl(k_cache_acc<2>, dim3((unsigned)b), dim3(kCacheChunk), 0, s, P)
                   : P.D <= 128 ? launch_pdl(k_cache_acc<4>, dim3((unsigned)b), dim3(kCacheChunk), 0, s, P)
                                : launch_pdl(k_cache_acc<8>, dim3((unsigned)b), dim3(kCacheChunk), 0, s, P);
    return le != cudaSuccess ? le : cudaGetLastError();
}

cudaError_t launch_cache_apply(const Params& P, cudaStream_t s) {
    const int64_t b = grid_for(P.cache_n, 8, (int64_t)P.sms * 8);
    cudaError_t le = P.D <= 64 ? launch_pdl(k_cache_apply<2>, dim3((unsigned)b), dim3(256), 0, s, P)
                   : P.D <= 128 ? launch_pdl(k_cache_apply<4>, dim3((unsigned)b), dim3(256), 0, s, P)
                                : launch_pdl(k_cache_apply<8>, dim3((unsigned)b), dim3(256), 0, s, P);
    return le != cudaSuccess ? le : cudaGetLastError();
}

cudaError_t set_fwd_attributes(int max_smem) {
    const void* ks[] = {(const void*)k_fwd_T<kQ444R32>, (const void*)k_fwd_T<kQ444R16>,
                        (const void*)k_fwd_T<kQ444R64>, (const void*)k_fwd_T<kQ448R64>,
                        (const void*)k_fwd_T<kDynamic>, (const void*)k_fwd_T<-1>,
#define TT_POOL4(DC) (const void*)k_pool<DC, 0>, (const void*)k_pool<DC, 1>, (const void*)k_pool<DC, 2>, (const void*)k_pool<DC, 3>
                        TT_POOL4(kQ444R32), TT_POOL4(kQ444R16), TT_POOL4(kQ444R64), TT_POOL4(kQ448R64), TT_POOL4(kDynamic),
#undef TT_POOL4
                        (const void*)k_pool<-1, 0>, (const void*)k_pool<-1, 1>, (const void*)k_pool<-2, 0>,
                        (const void*)k_pool<-2, 1>, (const void*)k_cache_fill, (const void*)k_cache_gmax,
                        (const void*)k_cache_acc<2>, (const void*)k_cache_acc<4>, (const void*)k_cache_acc<8>,
                        (const void*)k_cache_apply<2>, (const void*)k_cache_apply<4>, (const void*)k_cache_apply<8>};
    for (const void* k : ks) {
        cudaError_t e = allow_max_dynamic_smem(k, max_smem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace ttemb
