// tt_bwd_tc.cu -- the backward pair contractions on the 5th-generation tensor
// cores (tcgen05, sm_103a) for the dimension classes q = [4, 4, 4], r1 = r2 = R
// with R in {16, 32}.
//
// FBTT README, "Software Cache" (the gradient of each core is a chain of
// products in reversed order) and "Fused Kernel" (the update is applied inside
// the backward pass); TT-Rec review, abstract (the TT products as batched
// GEMMs); tensorflow/addons EmbeddingBag issue (gradients formed after sorting
// by key, no two threads writing one entry).  Per tile of lookups that share
// (table, i2), rows (i1, i3) and pairs (i1) being the runs of the sorted tile:
//   gs  = sum over the row's lookups of s_n grad_out[bag]   (FFMA, shared memory)
//   P3  = T^T gs per row: dG3 partial                         (FFMA, T of the forward pass)
//   dT  = sum over the pair's rows of gs G3[i3]^T            (FFMA, 16 pairs per batch)
//   Q   = dT G2[i2]^T per pair: dG1 partial                   (tcgen05, M = 64 = 16 pairs x q1)
//   dG2^T += dT^T G1 over all the tile's pairs               (tcgen05, M = q2 R, accumulated
//                                                              in tensor memory across batches)
// then the G2 update (or a partial for the group's last tile) as in the FFMA path.
//
// Precision.  Every fp32 operand x is held as three bf16 pieces x = x1 + x2 + x3
// (x1 the bf16 rounding of x, x2 of x - x1, x3 of x - x1 - x2; each difference is
// exact in fp32) and a product as x1 y1 + x1 y2 + x2 y1 + x1 y3 + x2 y2 + x3 y1,
// six kind::f16 MMAs with fp32 accumulation in tensor memory.  The dropped terms
// and the residue of x are below 2^-26 |x y|, finer than fp32 rounding.  With
// 16-bit pieces the tensor core also reads a transposed (MN-major) operand, so one
// copy of dT serves both products: K-major rows (pair, j1) for Q, MN-major rows jc
// for dG2^T.
//
// Shared-memory operand layout (no swizzle): 8-row x 16-byte core matrices of 8
// bf16.  K-major: element (row, k) of a [rows][K] tile at
//   (row / 8) (8 K) + (k / 8) 64 + (row % 8) 8 + k % 8     (bf16 elements),
// leading (K) byte offset 128, stride (8-row) byte offset 16 K.  The same bytes
// read MN-major, element (m = k, kk = row): leading (K) byte offset 16 K, stride
// (MN) byte offset 128.  dT's 8-row groups are 16 K + 16 bytes apart instead, which
// puts the eight rows that one quarter-warp stores in distinct banks.
// Accumulators: M = 128 puts row r in tensor-memory lane r; M = 64 puts row r in
// lane 32 (r / 16) + r % 16.  The three pieces of the B operand (R rows each) lie
// one after another with the same 8-row stride, so [y1 | y2 | y3] and [y1 | y2] are
// themselves B operands of N = 3R and 2R rows: one MMA x1 [y1 | y2 | y3] gives x1 y1,
// x1 y2 and x1 y3 in three R-column accumulators, x2 [y1 | y2] adds x2 y1 and x2 y2
// to the first two, and x3 y1 adds to the first.  Three MMAs per K step instead of
// six, and each A piece (the large operand: dT) is read from shared memory once per
// K step; the tensor core of these skinny products is bound by its shared-memory
// operand reads.  The column blocks are summed when read out (small terms first).
// Q runs as two chains (x1 [..] and x2 [..] + x3 y1, separate accumulators) and
// dG2^T as one, each issued by its own thread (lane 0 of warps 0, 1, 2).
#include "tt_dims.cuh"
#include "tt_tc.cuh"
#include "tt_tile.cuh"

namespace ttemb {

constexpr int kTcBwdThreads = 256;
constexpr int kTcBwdCap = 64;    // lookups per tile
constexpr int kTcBwdPairs = 16;  // pairs per batch: Q has M = 16 x q1 = 64 rows
constexpr int kTcBwdG3Rows = 16;  // G3 slices staged in shared memory per batch (its first rows)
constexpr uint32_t kTcBwdCols = 256;  // tensor-memory columns (tc_cols_q1, tc_cols_q2, tc_cols_g below)
constexpr int kTcBwdIssuers = 3;      // accumulator chains per batch, one commit each

__host__ __device__ constexpr bool bwd_tc_class(int dclass) { return dclass == kQ444R32 || dclass == kQ444R16; }

__host__ __device__ constexpr size_t al128(size_t x) { return (x + 127) & ~(size_t)127; }

// Tensor-memory column of each accumulator (multiples of 32): Q's x1 chain (3R
// columns), Q's x2 / x3 chain (2R), dG2^T (3R).
__host__ __device__ constexpr uint32_t tc_cols_q2(int R) { return (3u * R + 31u) & ~31u; }
__host__ __device__ constexpr uint32_t tc_cols_g(int R) { return tc_cols_q2(R) + ((2u * R + 31u) & ~31u); }
static_assert(tc_cols_g(32) + 96 <= kTcBwdCols && tc_cols_g(16) + 48 <= kTcBwdCols, "accumulators fit");

template <int R>
struct TcBwdLayout {
    static constexpr int N2 = 4 * R;                                 // q2 r2: columns jc of dT and G2
    static constexpr int kRows = 4 * kTcBwdPairs;                    // rows (pair, j1) of a batch
    static constexpr size_t ctl = 0;                                 // mbarrier, tensor-memory address, flag
    static constexpr size_t keys = 64;
    static constexpr size_t ints = keys + 8 * kTcBwdCap;            // sp1 sp3 si1 si3 sbag ss rowid pairid
    static constexpr size_t begs = ints + 8 * 4 * kTcBwdCap;        // rowbeg, pairbeg
    static constexpr size_t sh = begs + 2 * 4 * (kTcBwdCap + 4);
    static constexpr size_t gs = al128(sh + 4 * 64);                 // [rows][64] fp32
    static constexpr size_t g2 = al128(gs + 4 * kTcBwdCap * 64);     // 3 pieces of [R][N2] bf16, K-major
    static constexpr uint32_t g2sbo = 16 * N2 + 16;                   //   8-row group stride (bytes, padded)
    static constexpr size_t g2p = (size_t)(R / 8) * g2sbo;          //   bytes per piece
    static constexpr size_t g1 = al128(g2 + 3 * g2p);                // 3 pieces of [R][kRows] bf16, K-major
    static constexpr uint32_t g1sbo = 16 * kRows + 16;                //   8-row group stride (bytes, padded)
    static constexpr size_t g1p = (size_t)(R / 8) * g1sbo;
    static constexpr size_t dt = al128(g1 + 3 * g1p);                // 3 pieces of [kRows][N2] bf16, K-major
    static constexpr uint32_t dts = 16 * N2 + 16;                     //   8-row group stride (bytes, padded)
    static constexpr size_t dtp = (size_t)(kRows / 8) * dts;
    static constexpr size_t g3 = dt + 3 * dtp;                       // G3 slices of a batch's first rows (fp32,
                                                                     //   R + 1 float4 a row: a gap between the halves)
    static constexpr size_t total = g3 + 4 * (size_t)kTcBwdG3Rows * (R * 4 + 4);
    static_assert(g2p % 16 == 0 && g1p % 16 == 0 && dtp % 16 == 0, "pieces 16-byte aligned");
    // two blocks per SM: 228 KB of shared memory per SM, 1 KB of it reserved per block
    static_assert(2 * (total + 1024) <= 228 * 1024, "two blocks per SM");
};

// K-major bf16 element offset of (row, k) in a tile whose K extent is K, its 8-row
// groups padded by 16 bytes (8 K + 8 elements apart).
__device__ __forceinline__ int kmaj16(int row, int k, int K) {
    return (row >> 3) * (K * 8 + 8) + (k >> 3) * 64 + (row & 7) * 8 + (k & 7);
}

// Byte offset of dT element (row, jc) in a piece: padded 8-row groups.
template <int R>
__device__ __forceinline__ int dt_off(int row, int jc) {
    return (row >> 3) * (int)TcBwdLayout<R>::dts + (jc >> 3) * 128 + (row & 7) * 16 + (jc & 7) * 2;
}

// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulator; ta: A MN-major.
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N, int ta) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)ta << 15) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}


// 16 consecutive fp32 columns of this warp's 32 lanes (lane i gets lane base + i).
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float* v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 columns of a product's column blocks, summed last block first into v (t:
// scratch): c[0] the block holding x1 y1, the others smaller terms.
template <int NB>
__device__ __forceinline__ void tc_sumx16(uint32_t lanebase, const uint32_t (&c)[NB], float* v, float* t) {
    tc_ld16(lanebase + c[NB - 1], t);
#pragma unroll
    for (int b = NB - 2; b >= 0; --b) {
        tc_ld16(lanebase + c[b], v);
#pragma unroll
        for (int a = 0; a < 16; ++a) t[a] += v[a];
    }
#pragma unroll
    for (int a = 0; a < 16; ++a) v[a] = t[a];
}

// x rounded to a bf16 value (8-bit significand, ties away from zero), kept in fp32
// bits: add half of the dropped part to the magnitude, then clear it.  Integer
// operations only (the float-to-bf16 conversions run at a fraction of the ALU rate).
__device__ __forceinline__ uint32_t bf16_round_bits(uint32_t b) { return (b + 0x8000u) & 0xFFFF0000u; }

// x = x1 + x2 + x3 in bf16 pieces, returned as fp32 bit patterns whose low 16 bits
// are 0 (x1 = x rounded, x2 = (x - x1) rounded, x3 = (x - x1 - x2) rounded; each
// difference is exact in fp32).
__device__ __forceinline__ void split3(float x, uint32_t& a, uint32_t& b, uint32_t& c) {
    a = bf16_round_bits(__float_as_uint(x));
    const float r1 = x - __uint_as_float(a);
    b = bf16_round_bits(__float_as_uint(r1));
    c = bf16_round_bits(__float_as_uint(r1 - __uint_as_float(b)));
}

// Two pieces (high halves of fp32 bit patterns) as one bf16x2 word, lo first.
__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) { return __byte_perm(lo, hi, 0x7632); }

// Eight consecutive fp32 values as three 16-byte piece chunks at byte offset `boff`
// of the three piece regions (`stride` bytes apart).
__device__ __forceinline__ void store_pieces8b(unsigned char* base, size_t stride, int boff, const float* v) {
    uint32_t w[3][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t a0, b0, c0, a1, b1, c1;
        split3(v[2 * i], a0, b0, c0);
        split3(v[2 * i + 1], a1, b1, c1);
        w[0][i] = pack2(a0, a1);
        w[1][i] = pack2(b0, b1);
        w[2][i] = pack2(c0, c1);
    }
#pragma unroll
    for (int p = 0; p < 3; ++p)
        *reinterpret_cast<uint4*>(base + p * stride + boff) = make_uint4(w[p][0], w[p][1], w[p][2], w[p][3]);
}

// The same at bf16 element offset `off`.
__device__ __forceinline__ void store_pieces8(unsigned char* base, size_t stride, int off, const float* v) {
    uint32_t w[3][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t a0, b0, c0, a1, b1, c1;
        split3(v[2 * i], a0, b0, c0);
        split3(v[2 * i + 1], a1, b1, c1);
        w[0][i] = pack2(a0, a1);
        w[1][i] = pack2(b0, b1);
        w[2][i] = pack2(c0, c1);
    }
#pragma unroll
    for (int p = 0; p < 3; ++p)
        *reinterpret_cast<uint4*>(base + p * stride + 2 * (size_t)off) = make_uint4(w[p][0], w[p][1], w[p][2], w[p][3]);
}

// 16 bytes from shared memory at a shared-window address (an explicit shared load).
__device__ __forceinline__ float4 lds128(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}

// Asynchronous 16-byte global-to-shared copies (completion: cp_async_wait_all).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Start copying the G3 slices of tile-rows [r0, r0 + kTcBwdG3Rows) (clipped at nrows) into g3s:
// slice r at float4 r (R + 1), its second half one float4 further (the dT lanes of a
// quarter-warp read both halves at once, now from different banks).
template <int R>
__device__ __forceinline__ void stage_g3(const TableDev& T, const int* rowbeg, const int* si3, float* g3s, int r0,
                                         int nrows) {
    constexpr int CH = R;  // 16-byte chunks per slice (R x q3 floats)
    const int n = min(kTcBwdG3Rows, nrows - r0) * CH;
    for (int e = threadIdx.x; e < n; e += kTcBwdThreads) {
        const int r = e / CH, c = e - r * CH;
        cp_async16(g3s + (r * (CH + 1) + c + (c >= CH / 2 ? 1 : 0)) * 4, T.G3 + (int64_t)si3[rowbeg[r0 + r]] * (R * 4) + c * 4);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// dG3 partial per tile-row, items [i0, i1) of nrows x R/4 (a row and four columns c):
// P3[c][j3] = sum_j12 T[j12][c] gs[j12 q3 + j3], T of the pair from the forward pass
// (sixteen float4 loads of T in flight per item).  Items go to the highest threads
// first: the low warps issue the MMAs and start late.
template <int R>
__device__ __forceinline__ void tile_p3(const Params& P, const TableDev& T, int i2, int start, const int* rowbeg,
                                        const int* si1, const float* gs, int i0, int i1) {
    constexpr int D = 64, C4 = R / 4;
    for (int e = i0 + (kTcBwdThreads - 1 - (int)threadIdx.x); e < i1; e += kTcBwdThreads) {
        const int row = e / C4, c4 = e - row * C4;
        const int kk = rowbeg[row];
        const float4* Tp = reinterpret_cast<const float4*>(
                               P.Tbuf + T.tbase + ((int64_t)i2 * T.p1 + si1[kk]) * (int64_t)(16 * R)) + c4;
        float4 tv[16];
#pragma unroll
        for (int j12 = 0; j12 < 16; ++j12) tv[j12] = __ldg(Tp + j12 * C4);
        const float* gr = gs + row * D;
        float acc[4][4] = {};
#pragma unroll
        for (int j12 = 0; j12 < 16; ++j12) {
            const float4 x = *reinterpret_cast<const float4*>(gr + j12 * 4);
            const float t4[4] = {tv[j12].x, tv[j12].y, tv[j12].z, tv[j12].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                acc[c][0] = fmaf(t4[c], x.x, acc[c][0]);
                acc[c][1] = fmaf(t4[c], x.y, acc[c][1]);
                acc[c][2] = fmaf(t4[c], x.z, acc[c][2]);
                acc[c][3] = fmaf(t4[c], x.w, acc[c][3]);
            }
        }
        float4* dst = reinterpret_cast<float4*>(P.Pbuf + (int64_t)(start + kk) * P.ps_max + c4 * 16);
#pragma unroll
        for (int c = 0; c < 4; ++c) dst[c] = make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
    }
}

template <int R>
__device__ void tile_bwd_tc_body(const Params& P, const TableDev& T, unsigned char* sm, int tile) {
    using L = TcBwdLayout<R>;
    constexpr int N2 = L::N2, D = 64, KR = L::kRows;
    constexpr int G2I = R * (N2 / 8);                      // G2 items: (a, 8 columns)
    uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::ctl);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + L::ctl + 8);
    int* flag = reinterpret_cast<int*>(sm + L::ctl + 12);
    uint64_t* gbar = reinterpret_cast<uint64_t*>(sm + L::ctl + 16);  // the G2 slice's bulk copy
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(sm + L::keys);
    int* sp1 = reinterpret_cast<int*>(sm + L::ints);
    int* sp3 = sp1 + kTcBwdCap;
    int* si1 = sp3 + kTcBwdCap;
    int* si3 = si1 + kTcBwdCap;
    int* sbag = si3 + kTcBwdCap;
    float* ss = reinterpret_cast<float*>(sbag + kTcBwdCap);
    int* rowid = reinterpret_cast<int*>(ss + kTcBwdCap);
    int* pairid = rowid + kTcBwdCap;
    int* rowbeg = reinterpret_cast<int*>(sm + L::begs);
    int* pairbeg = rowbeg + kTcBwdCap + 4;
    int* sh = reinterpret_cast<int*>(sm + L::sh);
    float* gs = reinterpret_cast<float*>(sm + L::gs);
    unsigned char* g2s = sm + L::g2;
    unsigned char* g1s = sm + L::g1;
    unsigned char* dts = sm + L::dt;
    float* g3s = reinterpret_cast<float*>(sm + L::g3);

    const int4 tl = P.tiles[tile];
    const int start = tl.x, len = tl.y, g = tl.z;
    const int i2 = g - T.base2;
    const int t = P.ntab == 1 ? 0 : P.bin2_tab[g];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;

    // The G2 slice (it depends only on i2) comes by bulk copies, one a row a, into the dT
    // piece region (free until the first batch), rows N2 + 4 floats apart so that the
    // eight rows one quarter-warp reads below lie in different banks; the copies are in
    // flight during the tile sort.
    const float* g2src = T.G2 + (int64_t)i2 * R * N2;
    float* g2raw = reinterpret_cast<float*>(sm + L::dt);
    static_assert(R * (N2 + 4) * 4 <= 3 * L::dtp, "raw G2 rows fit the dT region");
    if (threadIdx.x < 32) {
        if (threadIdx.x == 0) {
            mbar_init(gbar, 1);
            bulk_expect(gbar, (uint32_t)(R * N2 * sizeof(float)));
        }
        __syncwarp();
        if ((int)threadIdx.x < R)
            bulk_copy(g2raw + threadIdx.x * (N2 + 4), g2src + threadIdx.x * N2, (uint32_t)(N2 * sizeof(float)), gbar);
    }

    // ---- lookups of the tile, sorted by (i1, i3, position); rows and pairs
    load_and_sort_tile(P, start, len, keys, sp1, sp3, si1, si3, sbag, ss);
#ifdef TTEMB_DEBUG
    if ((int)threadIdx.x < len) {  // the tile's slices within the table, its group within the bins
        si1[threadIdx.x] = TT_DCHECK(P, si1[threadIdx.x], T.p1);
        si3[threadIdx.x] = TT_DCHECK(P, si3[threadIdx.x], T.p3);
    }
    if (threadIdx.x == 0) TT_DCHECK(P, i2, T.p2);
    __syncthreads();
#endif
    // every lookup's gradient row: loads in flight during the scans and the G2 staging
    static_assert(kTcBwdCap * 16 <= 4 * kTcBwdThreads, "gradient rows of a tile: four float4 a thread");
    GsLoads gl;
    tile_gs_issue(P, len, sbag, ss, D, gl);
    const int k = threadIdx.x;
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
    // partial slots by the position of the run's first lookup in the grouped order
    if (k < len) {
        P.rep3[sp3[k]] = fr ? start + k : -1;
        P.rep1[sp1[k]] = fp ? start + k : -1;
    }

    __syncthreads();  // rowbeg / pairbeg complete
    stage_g3<R>(T, rowbeg, si3, g3s, 0, nrows);  // the first batch's G3 slices
    // G1 item of this thread (row a, eight K positions (pair, j1)); the next batch's values
    // are loaded while the MMAs of the current one run
    const bool g1item = (int)threadIdx.x < R * (KR / 8);
    const int g1a = (threadIdx.x & 7) + 8 * (threadIdx.x / (8 * (KR / 8))), g1k8 = (threadIdx.x >> 3) % (KR / 8);
    float g1v[8];
    auto load_g1 = [&](int ub) {
        const int nbb = min(kTcBwdPairs, npairs - ub);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int u = 2 * g1k8 + (i >> 2), j1 = i & 3;
            g1v[i] = (g1item && u < nbb) ? __ldg(T.G1 + (int64_t)si1[pairbeg[ub + u]] * (4 * R) + j1 * R + g1a) : 0.f;
        }
    };
    load_g1(0);
    // ---- G2 as the B operand of Q: rows a, K = jc, three pieces (from the bulk copy)
    if (threadIdx.x == 0 && !mbar_wait(gbar, 0, P.wait_polls)) {
        atomicOr(P.err, kErrTimeout);
        mbar_wait(gbar, 0, kTcWaitLimit);  // the copy writes shared memory: let it finish
    }
    __syncthreads();
    for (int e = threadIdx.x; e < G2I; e += kTcBwdThreads) {
        const int a = (e & 7) + 8 * (e / (8 * (N2 / 8))), jc8 = (e >> 3) % (N2 / 8);
        const float4* src = reinterpret_cast<const float4*>(g2raw + a * (N2 + 4) + jc8 * 8);
        const float4 x = src[0], y = src[1];
        const float v[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
        store_pieces8(g2s, L::g2p, kmaj16(a, jc8 * 8, N2), v);
    }
    if (threadIdx.x == 32) mbar_init(bar, kTcBwdIssuers);  // one commit per accumulator chain
    __syncthreads();  // rowid / pairid / rowbeg / pairbeg complete

    // ---- gs: summed upstream gradient of every tile-row
    tile_gs_rows(gl, len, nrows, rowbeg, gs, D);

    // ---- batches of kTcBwdPairs pairs: dT and the G1 rows as pieces, then the MMAs
    constexpr uint32_t kIdescQ3 = tc_idesc_bf16(64, 3 * R, 0), kIdescQ2 = tc_idesc_bf16(64, 2 * R, 0),
                       kIdescQ1 = tc_idesc_bf16(64, R, 0);
    constexpr uint32_t kIdescG3 = tc_idesc_bf16(N2, 3 * R, 1), kIdescG2 = tc_idesc_bf16(N2, 2 * R, 1),
                       kIdescG1 = tc_idesc_bf16(N2, R, 1);
    constexpr uint32_t DTS = L::dts;
    const uint32_t tq1 = *tslot, tq2 = *tslot + tc_cols_q2(R), tg = *tslot + tc_cols_g(R);
    bool failed = false;
    int nbatch = 0;
    for (int u0 = 0; u0 < npairs; u0 += kTcBwdPairs, ++nbatch) {
        const int nb = min(kTcBwdPairs, npairs - u0);
        // G1 as the B operand of dG2^T: rows a, K = (pair, j1); zero past the batch's pairs
        if (g1item) store_pieces8(g1s, L::g1p, kmaj16(g1a, g1k8 * 8, KR), g1v);
        cp_async_wait_all();  // this batch's G3 slices have landed (every thread's copies) ...
        __syncthreads();      // ... and are visible to the block
        // dT rows of the batch: warp w takes pairs w and w + 8; lane (j2, j1, h) the columns
        // c of one half of r2 for (j1, j2): per row of the pair the G3 slice is read as
        // broadcasts and the gs row without bank conflicts, and a quarter-warp's piece
        // stores cover four rows.  Zero past the batch's pairs.
        {
            constexpr int CH = R / 2;  // columns c per lane
            const int j2 = lane >> 3, j1 = (lane >> 1) & 3, c0 = (lane & 1) * CH;
#pragma unroll 1
            for (int u = w; u < kTcBwdPairs; u += kTcBwdThreads / 32) {
                float acc[CH];
#pragma unroll
                for (int i = 0; i < CH; ++i) acc[i] = 0.f;
                if (u < nb) {
                    const int kb = pairbeg[u0 + u], ke = pairbeg[u0 + u + 1];
                    for (int kk = kb; kk < ke; ++kk) {
                        if (kk != kb && rowid[kk] == rowid[kk - 1]) continue;  // once per tile-row
                        const float4 gv = *reinterpret_cast<const float4*>(gs + rowid[kk] * D + (j1 * 4 + j2) * 4);
                        const int rs = rowid[kk] - rowid[pairbeg[u0]];  // staged position of this row
                        // the G3 slice from shared memory (staged rows) or global memory, each
                        // path with its own load form: a pointer that may be either would turn
                        // every load into a slow generic one
                        float4 y[CH];
                        if (rs < kTcBwdG3Rows) {
                            const uint32_t a0 = smem_addr(g3s + (rs * (R + 1) + c0 + (c0 ? 1 : 0)) * 4);
#pragma unroll
                            for (int i = 0; i < CH; ++i) y[i] = lds128(a0 + 16 * i);
                        } else {
                            const float4* g3 = reinterpret_cast<const float4*>(T.G3 + (int64_t)si3[kk] * (R * 4)) + c0;
#pragma unroll
                            for (int i = 0; i < CH; ++i) y[i] = __ldg(g3 + i);
                        }
#pragma unroll
                        for (int i = 0; i < CH; ++i) {
                            float a = acc[i];
                            a = fmaf(gv.x, y[i].x, a);
                            a = fmaf(gv.y, y[i].y, a);
                            a = fmaf(gv.z, y[i].z, a);
                            acc[i] = fmaf(gv.w, y[i].w, a);
                        }
                    }
                }
#pragma unroll
                for (int h8 = 0; h8 < CH; h8 += 8)
                    store_pieces8b(dts, L::dtp, dt_off<R>(4 * u + j1, j2 * R + c0 + h8), acc + h8);
            }
        }
        tc_fence_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (lane == 0 && w < kTcBwdIssuers) {
            // Q = dT G2^T (A = dT K-major rows (u, j1), B = G2 K-major rows a, K = jc) and
            // dG2^T += dT^T G1 (A = dT read MN-major rows jc, B = G1 K-major rows a, K = (u, j1)).
            // Warp 0: Q's x1 [y1 | y2 | y3]; warp 1: Q's x2 [y1 | y2] + x3 y1; warp 2: dG2^T's
            // three MMAs per K step.  Each chain commits once.
            const uint32_t d0 = smem_addr(dts), g1b = smem_addr(g1s), g2a = smem_addr(g2s);
            if (w < 2) {
#pragma unroll
                for (int ks = 0; ks < N2 / 16; ++ks) {
                    const uint64_t a0 = tc_desc(d0 + ks * 256, 128, DTS);
                    const uint64_t b0 = tc_desc(g2a + ks * 256, 128, L::g2sbo);
                    const uint64_t a1 = a0 + (L::dtp >> 4), a2 = a0 + 2 * (L::dtp >> 4);
                    const bool acc = ks > 0;
                    if (w == 0) {
                        tc_mma_f16(tq1, a0, b0, kIdescQ3, acc);
                    } else {
                        tc_mma_f16(tq2, a1, b0, kIdescQ2, acc);
                        tc_mma_f16(tq2, a2, b0, kIdescQ1, true);
                    }
                }
            } else {
                const int NG = (4 * nb + 15) / 16;
#pragma unroll
                for (int ks = 0; ks < KR / 16; ++ks) {
                    if (ks < NG) {
                        const uint64_t a0 = tc_desc(d0 + ks * 2 * DTS, DTS, 128);
                        const uint64_t b0 = tc_desc(g1b + ks * 256, 128, L::g1sbo);
                        const uint64_t a1 = a0 + (L::dtp >> 4), a2 = a0 + 2 * (L::dtp >> 4);
                        tc_mma_f16(tg, a0, b0, kIdescG3, nbatch > 0 || ks > 0);
                        tc_mma_f16(tg, a1, b0, kIdescG2, true);
                        tc_mma_f16(tg, a2, b0, kIdescG1, true);
                    }
                }
            }
            tc_commit(bar);
        }
        if (u0 + kTcBwdPairs < npairs) {  // the next batch's G1 values and G3 slices, in flight during the MMAs
            load_g1(u0 + kTcBwdPairs);
            stage_g3<R>(T, rowbeg, si3, g3s, rowid[pairbeg[u0 + kTcBwdPairs]], nrows);
        }
        {   // this batch's share of the dG3 partials, computed while the MMAs run
            const int nbt = (npairs + kTcBwdPairs - 1) / kTcBwdPairs, items = nrows * (R / 4);
            const int per = (items + nbt - 1) / nbt;
            tile_p3<R>(P, T, i2, start, rowbeg, si1, gs, nbatch * per, min(items, (nbatch + 1) * per));
        }
        if (threadIdx.x == 0) {
            *flag = mbar_wait(bar, nbatch & 1, P.wait_polls) ? 1 : 0;
            if (!*flag) atomicOr(P.err, kErrTimeout);
        }
        __syncthreads();
        tc_fence_after();
        if (!*flag) {  // gave up: no further MMA, no operand rewrite (uniform: shared flag)
            failed = true;
            break;
        }
        // Q rows (u, j1): M = 64 puts row r in lane 32 (r / 16) + r % 16
        // warp w reads lane quarter w % 4 (the only lanes it may access) and, at R = 32, the
        // 16-column half w / 4: every warp takes one 16-column chunk
        if (R == 32 || w < 4) {
            const int qw = w & 3, c0 = R == 32 ? 16 * (w >> 2) : 0;
            const int r = 16 * qw + lane, u = r >> 2, j1 = r & 3;
            const bool live = lane < 16 && u < nb;
            float* dst = P.Qbuf + (int64_t)(start + (live ? pairbeg[u0 + u] : 0)) * P.qs_max + j1 * R;
            float q[16], e[16];
            const uint32_t cq[5] = {tq1 + c0, tq2 + c0, tq1 + R + c0, tq2 + R + c0, tq1 + 2 * R + c0};
            tc_sumx16<5>((uint32_t)(32 * qw) << 16, cq, q, e);
            if (live) {
#pragma unroll
                for (int a = 0; a < 16; a += 4)
                    *reinterpret_cast<float4*>(dst + c0 + a) = make_float4(q[a], q[a + 1], q[a + 2], q[a + 3]);
            }
        }
        tc_fence_before();
        __syncthreads();  // Q read out and the operand tiles free before the next batch
        tc_fence_after();
    }

    if (failed) {
        // the MMAs of the batch that gave up may still run: wait for them (full bound)
        if (threadIdx.x == 0) mbar_wait(bar, nbatch & 1, kTcWaitLimit);
        tc_fence_before();
        __syncthreads();
        if (w == 0) tc_dealloc(*tslot, kTcBwdCols);
        return;
    }

    // ---- dG2 of the tile: rows jc of dG2^T (M = N2 lanes), direct update or partial
    float* G2p = T.G2 + (int64_t)i2 * R * N2;
    float* A2p = T.aux[1] ? T.aux[1] + (int64_t)i2 * R * N2 : nullptr;
    const int nt = P.grp_ntiles[g];
    float* part = P.dG2part + (int64_t)tile * P.s2_max;
    if (R == 32 || w < 4) {  // as for Q: warp w takes lane quarter w % 4 and one 16-column chunk
        const int qw = w & 3, c0 = R == 32 ? 16 * (w >> 2) : 0;
        const int jc = N2 == 128 ? 32 * qw + lane : 16 * qw + lane;
        const bool live = N2 == 128 || lane < 16;
        float gv[16], ge[16];
        const uint32_t cg[3] = {tg + c0, tg + R + c0, tg + 2 * R + c0};
        tc_sumx16<3>((uint32_t)(32 * qw) << 16, cg, gv, ge);
        if (live) {
            if (nt == 1) {  // sixteen loads in flight, then the stores
                int idx[16];
#pragma unroll
                for (int a = 0; a < 16; ++a) idx[a] = (c0 + a) * N2 + jc;
                core_update_n<16>(P, G2p, A2p, idx, gv);
            } else {
#pragma unroll
                for (int a = 0; a < 16; ++a) part[(c0 + a) * N2 + jc] = gv[a];
            }
        }
    }
    if (nt == 1 && P.slice_stamp && P.opt != TT_OPT_GRAD && threadIdx.x == 0 && t == 0)
        P.slice_stamp[T.p1 + i2] = *P.dstep + 1;

    // every partial of this block is written: publish them before any arrival count
    __threadfence();
    tc_fence_before();
    __syncthreads();
    if (w == 0) tc_dealloc(*tslot, kTcBwdCols);
    if (nt > 1) {
        if (threadIdx.x == 0) sh[42] = (atomicAdd(&P.grp_done[g], 1) == nt - 1);
        __syncthreads();
        if (sh[42]) {  // the group's last tile sums the dG2 partials in tile order
            __threadfence();
            const int first = P.grp_first[g];
            for (int e0 = threadIdx.x; e0 < R * N2; e0 += 8 * kTcBwdThreads) {  // eight elements a round
                int idx[8];
                float sum[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) idx[u] = e0 + u * kTcBwdThreads < R * N2 ? e0 + u * kTcBwdThreads : -1;
                sum_partials<8>(P.dG2part + (int64_t)first * P.s2_max, P.s2_max, nt, idx, sum);
                core_update_nm<8>(P, G2p, A2p, idx, sum);  // then the eight updates' loads together
            }
            if (threadIdx.x == 0) {
                P.grp_done[g] = 0;
                if (P.slice_stamp && P.opt != TT_OPT_GRAD && t == 0) P.slice_stamp[T.p1 + i2] = *P.dstep + 1;
            }
        }
    }
}

// One tile per block, two blocks per SM (about 104 KB of shared memory each).
template <int DC>
__global__ void __launch_bounds__(kTcBwdThreads, 2) k_tile_bwd_tc(const __grid_constant__ Params P) {
    pdl_entry();
    if (*P.err) return;  // a device error was recorded: leave every core unchanged
    if ((int)blockIdx.x >= *P.ntiles) return;
    const int tile = P.small ? P.tile_order[blockIdx.x] : (int)blockIdx.x;  // longest tiles first
    extern __shared__ __align__(128) unsigned char smraw[];
    // tensor memory first, and the allocation permit released at once
    if (threadIdx.x < 32) tc_alloc(reinterpret_cast<uint32_t*>(smraw + 8), kTcBwdCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const TableDev& T = P.tables[P.ntab == 1 ? 0 : P.bin2_tab[P.tiles[tile].z]];
    if constexpr (DC == kQ444R32) tile_bwd_tc_body<32>(P, T, smraw, tile);
    else tile_bwd_tc_body<16>(P, T, smraw, tile);
}

// ------------------------------------------------------------------ launchers

bool bwd_tc_eligible(int dclass_all) { return bwd_tc_class(dclass_all); }
int bwd_tc_cap() { return kTcBwdCap; }
static_assert(kTcBwdCap <= kMaxTcTileCap, "the tile order's length buckets");

static size_t tc_smem(int dclass) { return dclass == kQ444R32 ? TcBwdLayout<32>::total : TcBwdLayout<16>::total; }

cudaError_t launch_tile_bwd_tc(const Params& P, cudaStream_t s) {
    const size_t smem = tc_smem(P.dclass_all);
    cudaError_t le = P.dclass_all == kQ444R32
                         ? launch_pdl(k_tile_bwd_tc<kQ444R32>, dim3((unsigned)P.max_tiles), dim3(kTcBwdThreads), smem, s, P)
                         : launch_pdl(k_tile_bwd_tc<kQ444R16>, dim3((unsigned)P.max_tiles), dim3(kTcBwdThreads), smem, s, P);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
}

cudaError_t set_bwd_tc_attributes(int max_smem) {
    const void* ks[] = {(const void*)k_tile_bwd_tc<kQ444R32>, (const void*)k_tile_bwd_tc<kQ444R16>};
    for (const void* kf : ks) {
        cudaError_t e = allow_max_dynamic_smem(kf, max_smem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace ttemb
