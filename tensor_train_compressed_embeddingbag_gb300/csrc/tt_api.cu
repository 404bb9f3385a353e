// tt_api.cu -- the C ABI of libttemb.so (declarations and contracts in include/tt_emb.h).
//
// Host side only: argument validation, the handle's device tables, the
// workspace, and the order of the kernel launches of one forward or backward
// call.  Every step of the computation runs in the kernels of tt_sort.cu and
// tt_compute.cu.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/tt_emb.h"
#include "tt_internal.cuh"

using namespace ttemb;

namespace ttemb {
bool g_use_pdl = true;
}

namespace {

constexpr int kMaxStages = 16;

struct Arena {
    char* base = nullptr;
    size_t used = 0;
    size_t cap = 0;
    template <class T>
    T* take(size_t count) {
        size_t off = (used + 255) & ~(size_t)255;
        used = off + sizeof(T) * count;
        return base ? reinterpret_cast<T*>(base + off) : nullptr;
    }
};

}  // namespace

struct tt_emb {
    int device = 0;
    int ntab = 0;
    std::vector<TableDev> tabs;  // host copy
    TableDev* d_tables = nullptr;
    int* d_bins = nullptr;       // bin -> table for the three digits
    int* d_fixed = nullptr;      // err, (spare x2), ntiles, epoch, dstep, nincl, scan_done, grp_done[2 n2], dec_done, multi_count
    float* d_tbuf = nullptr;
    int64_t tbuf_floats = 0;
    int* d_tflag = nullptr;      // dense touched-pair flags
    int split_small = 1;         // column split of k_tile_bwd on the single-CTA-sort path
    int cap_small = 64, cap_large = 128;
    Params P{};                  // constants + workspace pointers
    // workspace
    void* d_ws = nullptr;
    size_t ws_bytes = 0;
    int64_t cap_nnz = -1, cap_bags = -1;
    // forward state
    bool has_fwd = false;
    cudaStream_t last_stream = nullptr;
    // stage timing
    bool timing = false;
    cudaEvent_t ev[2][kMaxStages + 1] = {};
    const char* names[2][kMaxStages] = {};
    int nstage[2] = {0, 0};
    int launches[2] = {0, 0};
    // cache
    int64_t* d_cache_rows = nullptr;
    float* d_cache_vals = nullptr;
    int* d_cache_stamp = nullptr;
    int* d_slice_stamp = nullptr;
    // trainable cache rows (tt_emb_cache_set_trainable)
    bool cache_train = false;
    unsigned long long* d_cache_acc = nullptr;
    float* d_cache_state = nullptr;
    float* d_cache_grad = nullptr;
    unsigned* d_cache_gmax = nullptr;
    int* d_cache_touch = nullptr;
    int* d_cache_list = nullptr;
    // explicit rows (tt_emb_cache_populate): open-addressing index row -> slot
    longlong2* d_cache_hidx = nullptr;
    int* d_cache_claim = nullptr;
    // LFU policy (tt_emb_lfu_enable)
    unsigned long long* d_freq_keys = nullptr;
    unsigned* d_freq_counts = nullptr;
    int64_t freq_size = 0;
    int64_t lfu_slots = 0;  // cache rows (a multiple of kLfuWays)
    int64_t cache_n = 0;
};

namespace {

tt_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TT_OK : TT_ERR_CUDA; }

int pow2_floor(int x) {
    int p = 1;
    while (p * 2 <= x) p *= 2;
    return p;
}

bool use_small_path(const tt_emb* h, int64_t nnz) {
    const Params& P = h->P;
    return nnz <= kSmallMaxNnz && P.n1 <= kSmallMaxBins && P.n2 <= kSmallMaxBins && P.n3 <= kSmallMaxBins;
}

// Tiles of a call: each (table, i2) group of c lookups gives ceil(c / cap) tiles.
int max_tiles_for(const tt_emb* h, int64_t nnz, int cap) {
    return (int)((std::max<int64_t>(nnz, 1) + cap - 1) / cap) + h->P.n2;
}

// Workspace carve-up for up to `nnz` lookups; base == nullptr only measures.
size_t carve(tt_emb* h, void* base, int64_t nnz, bool assign) {
    Arena A;
    A.base = static_cast<char*>(base);
    Params& P = h->P;
    const int64_t N = std::max<int64_t>(nnz, 1);
    const int64_t Ns = std::min<int64_t>(N, kSmallMaxNnz);
    const int nch = std::max((int)((N + kChunk - 1) / kChunk), (int)((Ns + kSmallChunk - 1) / kSmallChunk));
    const int tiles_small = max_tiles_for(h, Ns, h->cap_small);
    const int tiles_large = max_tiles_for(h, N, h->cap_large);
    const int max_tiles = std::max(tiles_small, tiles_large);
    const size_t part_floats = std::max((size_t)tiles_small * h->split_small, (size_t)tiles_large) * P.s2_max;
    const size_t qslots = std::max<size_t>((size_t)N, (size_t)Ns * h->split_small);
    int* lk_i1 = A.take<int>(N);
    int* lk_i2 = A.take<int>(N);
    int* lk_i3 = A.take<int>(N);
    int* lk_bag = A.take<int>(N);
    float* lk_s = A.take<float>(N);
    int* lk_hit = A.take<int>(N);
    float* lk_sh = A.take<float>(N);
    uint16_t* lr1 = A.take<uint16_t>(Ns);
    uint16_t* lr2 = A.take<uint16_t>(Ns);
    uint16_t* lr3 = A.take<uint16_t>(Ns);
    int* H1 = A.take<int>((size_t)P.n1 * nch);
    int* H3 = A.take<int>((size_t)P.n3 * nch);
    int* H2 = A.take<int>((size_t)P.n2 * nch);
    int* pi1 = A.take<int>(N);
    int* pi3 = A.take<int>(N);
    int* pi21 = A.take<int>(N);
    int* g_i1 = A.take<int>(N);
    int* g_i3 = A.take<int>(N);
    int* g_bag = A.take<int>(N);
    float* g_s = A.take<float>(N);
    int* sigma = A.take<int>(N);
    int4* tiles = A.take<int4>(max_tiles);
    int* tile_order = A.take<int>(max_tiles);
    int* grp_first = A.take<int>(P.n2);
    int* grp_ntiles = A.take<int>(P.n2);
    int* multi_groups = A.take<int>(P.n2);
    int* rep1 = A.take<int>(N);
    int* rep3 = A.take<int>(N);
    int* g_p1 = A.take<int>(N);
    int* g_p3 = A.take<int>(N);
    int* inv3 = A.take<int>(N);
    int* segsum = A.take<int>((size_t)(((int64_t)(P.n1 + P.n2 + P.n3) * nch) / kScanSeg + 4));
    float* Qbuf = A.take<float>(qslots * P.qs_max);
    float* Pbuf = A.take<float>((size_t)N * P.ps_max);
    float* dG2part = A.take<float>(part_floats);
    if (assign) {
        P.lk_i1 = lk_i1; P.lk_i2 = lk_i2; P.lk_i3 = lk_i3; P.lk_bag = lk_bag; P.lk_s = lk_s;
        P.lk_hit = lk_hit; P.lk_sh = lk_sh;
        P.lr1 = lr1; P.lr2 = lr2; P.lr3 = lr3;
        P.H1 = H1; P.H3 = H3; P.H2 = H2;
        P.pi1 = pi1; P.pi3 = pi3; P.pi21 = pi21; P.sigma = sigma;
        P.g_i1 = g_i1; P.g_i3 = g_i3; P.g_bag = g_bag; P.g_s = g_s;
        P.tiles = tiles; P.tile_order = tile_order; P.grp_first = grp_first; P.grp_ntiles = grp_ntiles;
        P.multi_groups = multi_groups;
        P.rep1 = rep1; P.rep3 = rep3; P.g_p1 = g_p1; P.g_p3 = g_p3; P.inv3 = inv3; P.segsum = segsum;
        P.Qbuf = Qbuf; P.Pbuf = Pbuf; P.dG2part = dG2part;
    }
    return A.used + 256;
}

tt_status ensure_workspace(tt_emb* h, int64_t nnz, int64_t nbags) {
    if (nnz <= h->cap_nnz && nbags <= h->cap_bags && h->d_ws) {
        carve(h, h->d_ws, h->cap_nnz, true);
        return TT_OK;
    }
    const int64_t cap = std::max<int64_t>({nnz, h->cap_nnz, 1});
    const size_t bytes = carve(h, nullptr, cap, false);
    if (h->d_ws) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return TT_ERR_CUDA;
        cudaFree(h->d_ws);
        h->d_ws = nullptr;
    }
    if (cudaMalloc(&h->d_ws, bytes) != cudaSuccess) {
        cudaGetLastError();
        h->d_ws = nullptr;
        h->cap_nnz = h->cap_bags = -1;
        return TT_ERR_NOMEM;
    }
    h->ws_bytes = bytes;
    h->cap_nnz = cap;
    h->cap_bags = std::max<int64_t>(nbags, h->cap_bags);
    carve(h, h->d_ws, cap, true);
    return TT_OK;
}

tt_status validate_table(int64_t E, const int64_t p[3], const int32_t q[3], const int32_t r[2]) {
    if (E <= 0) return TT_ERR_SHAPE;
    double prod = 1.0;
    for (int k = 0; k < 3; ++k) {
        if (p[k] <= 0 || p[k] > TT_MAX_P) return TT_ERR_SHAPE;
        if (q[k] <= 0 || q[k] > TT_MAX_Q) return TT_ERR_SHAPE;
        prod *= (double)p[k];
    }
    if (prod < (double)E) return TT_ERR_SHAPE;
    if (p[0] * p[1] * p[2] < E) return TT_ERR_SHAPE;
    for (int k = 0; k < 2; ++k)
        if (r[k] <= 0 || r[k] > TT_MAX_RANK) return TT_ERR_SHAPE;
    const int64_t D = (int64_t)q[0] * q[1] * q[2];
    if (D > TT_MAX_D) return TT_ERR_SHAPE;
    // per-thread accumulator limits of the tile and reduce kernels
    if ((int64_t)r[0] * q[1] * r[1] > 64 * kTileThreads) return TT_ERR_SHAPE;
    if ((int64_t)q[0] * r[0] > 32 * kTileThreads || (int64_t)r[1] * q[2] > 32 * kTileThreads) return TT_ERR_SHAPE;
    if ((int64_t)q[0] * q[1] * r[1] > 8192) return TT_ERR_SHAPE;  // one partial product T
    if ((int64_t)p[0] * p[1] > (int64_t)1 << 30) return TT_ERR_SHAPE;
    return TT_OK;
}

tt_status build_handle(tt_emb* h, int ntab, const tt_table_desc* d) {
    {
        const char* e = getenv("TTEMB_PDL");
        g_use_pdl = !(e && e[0] == '0');
    }
    // every host-side check comes before the first CUDA call
    for (int t = 0; t < ntab; ++t) {
        tt_status st = validate_table(d[t].num_embeddings, d[t].p, d[t].q, d[t].ranks);
        if (st != TT_OK) return st;
        if (d[t].q[0] * d[t].q[1] * d[t].q[2] != d[0].q[0] * d[0].q[1] * d[0].q[2]) return TT_ERR_SHAPE;
        for (int k = 0; k < 3; ++k)  // the kernels read the cores as float4
            if (!d[t].cores_dev[k] || ((uintptr_t)d[t].cores_dev[k] & 15u) != 0) return TT_ERR_ARG;
    }
    {
        int64_t s1 = 0, s2 = 0, s3 = 0;
        for (int t = 0; t < ntab; ++t) { s1 += d[t].p[0]; s2 += d[t].p[1]; s3 += d[t].p[2]; }
        if (s1 > kMaxBinsPerDigit || s2 > kMaxBinsPerDigit || s3 > kMaxBinsPerDigit) return TT_ERR_SHAPE;
    }
    if (cudaGetDevice(&h->device) != cudaSuccess) return TT_ERR_CUDA;
    {
        // kernel attributes are set once per device, never during a launch sequence
        static std::mutex mu;
        static std::vector<int> done;
        std::lock_guard<std::mutex> lock(mu);
        if (std::find(done.begin(), done.end(), h->device) == done.end()) {
            int max_smem = 0;
            if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess ||
                set_sort_attributes(max_smem) != cudaSuccess || set_fwd_attributes(max_smem) != cudaSuccess ||
                set_bwd_attributes(max_smem) != cudaSuccess)
                return TT_ERR_CUDA;
            done.push_back(h->device);
        }
    }
    h->ntab = ntab;
    const int D = d[0].q[0] * d[0].q[1] * d[0].q[2];
    int n1 = 0, n2 = 0, n3 = 0, qs = 1, ps = 1, s2 = 1, r1m = 1, Nm = 1, q1Nm = 1, tcf = 0;
    int64_t tb = 0, fb = 0;
    for (int t = 0; t < ntab; ++t) {
        TableDev T{};
        T.E = d[t].num_embeddings;
        T.p1 = (int)d[t].p[0]; T.p2 = (int)d[t].p[1]; T.p3 = (int)d[t].p[2];
        T.q1 = d[t].q[0]; T.q2 = d[t].q[1]; T.q3 = d[t].q[2];
        T.r1 = d[t].ranks[0]; T.r2 = d[t].ranks[1];
        T.D = D;
        T.G1 = d[t].cores_dev[0]; T.G2 = d[t].cores_dev[1]; T.G3 = d[t].cores_dev[2];
        T.tbase = tb;
        tb += (int64_t)T.p1 * T.p2 * T.q1 * T.q2 * T.r2;
        T.fbase = fb;
        fb += (int64_t)T.p1 * T.p2;
        T.dclass = dim_class_of(T.q1, T.q2, T.q3, T.r1, T.r2);
        T.idx32 = (int64_t)T.p1 * T.p2 * T.p3 < ((int64_t)1 << 31) ? 1 : 0;
        T.base1 = n1; T.base2 = n2; T.base3 = n3;
        n1 += T.p1; n2 += T.p2; n3 += T.p3;
        qs = std::max(qs, T.q1 * T.r1);
        ps = std::max(ps, T.r2 * T.q3);
        s2 = std::max(s2, T.r1 * T.q2 * T.r2);
        r1m = std::max(r1m, T.r1);
        Nm = std::max(Nm, T.q2 * T.r2);
        q1Nm = std::max(q1Nm, T.q1 * T.q2 * T.r2);
        tcf = std::max(tcf, fwd_tc_floats_of(T.dclass, T.r1, T.q2 * T.r2));
        h->tabs.push_back(T);
    }
    if (n1 > kMaxBinsPerDigit || n2 > kMaxBinsPerDigit || n3 > kMaxBinsPerDigit) return TT_ERR_SHAPE;
    Params& P = h->P;
    P.ntab = ntab;
    P.n1 = n1; P.n2 = n2; P.n3 = n3;
    P.D = D;
    // slot strides in whole 16-byte words: the kernels store the Q and P3 partials as float4
    P.qs_max = (qs + 3) & ~3; P.ps_max = (ps + 3) & ~3; P.s2_max = s2;
    P.r1_max = r1m; P.N_max = Nm; P.q1N_max = q1Nm; P.fwd_tc_floats = tcf;
    // tile caps: the summed upstream gradient of a tile (cap x D floats) stays <= 16 KB on the
    // single-CTA-sort path (many small tiles) and <= 64 KB on the multi-CTA path
    h->cap_small = pow2_floor(std::min(kTileThreads, 4096 / D));
    h->cap_large = pow2_floor(std::min(kTileThreads, 16384 / D));
    P.tile_cap = h->cap_large;
    int common = h->tabs[0].dclass, p1m = 1;
    bool can_split = true;
    for (const TableDev& T : h->tabs) {
        if (T.dclass != common) common = -1;
        p1m = std::max(p1m, T.p1);
        can_split = can_split && T.r2 % 8 == 0 && T.r2 >= 16;
    }
    P.dclass_all = common;
    {
        int sms = 0;  // few i2 groups: two k_fwd_T blocks share each group's pairs
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) return TT_ERR_CUDA;
        P.sms = sms;
        P.wait_polls = kTcWaitPolls;
        // the tensor-core T path takes a whole (table, i2) group per block
        bool all_tc = true;
        for (const TableDev& T : h->tabs) all_tc = all_tc && fwd_tc_floats_of(T.dclass, T.r1, T.q2 * T.r2) > 0;
        P.fwd_split = (!all_tc && n2 < 2 * sms) ? 2 : 1;
    }
    P.p1_max = p1m;
    h->split_small = can_split ? 2 : 1;
    {
        // the backward pair contractions on the tensor cores: one block per tile of at most
        // bwd_tc_cap() lookups, no column split (TTEMB_BWD_FFMA=1 keeps the FFMA kernel)
        const char* e = getenv("TTEMB_BWD_FFMA");
        P.bwd_tc = (bwd_tc_eligible(P.dclass_all) && !(e && e[0] == '1')) ? 1 : 0;
        if (P.bwd_tc) {
            h->split_small = 1;
            h->cap_small = h->cap_large = bwd_tc_cap();
            P.tile_cap = h->cap_large;
        }
    }
    // device tables
    std::vector<int> bins(n1 + n2 + n3);
    for (int t = 0; t < ntab; ++t) {
        const TableDev& T = h->tabs[t];
        for (int i = 0; i < T.p1; ++i) bins[T.base1 + i] = t;
        for (int i = 0; i < T.p2; ++i) bins[n1 + T.base2 + i] = t;
        for (int i = 0; i < T.p3; ++i) bins[n1 + n2 + T.base3 + i] = t;
    }
    if (cudaMalloc(&h->d_tables, sizeof(TableDev) * ntab) != cudaSuccess) return TT_ERR_NOMEM;
    if (cudaMalloc(&h->d_bins, sizeof(int) * bins.size()) != cudaSuccess) return TT_ERR_NOMEM;
    const int nfixed = 8 + 2 * n2 + kDecDoneSlots + 1;
    if (cudaMalloc(&h->d_fixed, sizeof(int) * nfixed) != cudaSuccess) return TT_ERR_NOMEM;
    if (cudaMalloc(&h->d_tbuf, sizeof(float) * std::max<int64_t>(tb, 1)) != cudaSuccess) return TT_ERR_NOMEM;
    if (cudaMalloc(&h->d_tflag, sizeof(int) * std::max<int64_t>(fb, 1)) != cudaSuccess) return TT_ERR_NOMEM;
    if (cudaMemset(h->d_tflag, 0, sizeof(int) * std::max<int64_t>(fb, 1)) != cudaSuccess) return TT_ERR_CUDA;
    // T of a pair that no lookup of a pass touched is read (times 0) by the trainable
    // cache hits of that pass: the buffer must hold finite values from the start
    if (cudaMemset(h->d_tbuf, 0, sizeof(float) * std::max<int64_t>(tb, 1)) != cudaSuccess) return TT_ERR_CUDA;
    h->tbuf_floats = tb;
    if (cudaMemcpy(h->d_tables, h->tabs.data(), sizeof(TableDev) * ntab, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(h->d_bins, bins.data(), sizeof(int) * bins.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(h->d_fixed, 0, sizeof(int) * nfixed) != cudaSuccess)
        return TT_ERR_CUDA;
    {
        const int one = 1;  // touched flags start at 0: the first epoch is 1
        if (cudaMemcpy(h->d_fixed + 4, &one, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return TT_ERR_CUDA;
    }
    P.tables = h->d_tables;
    P.bin1_tab = h->d_bins;
    P.bin2_tab = h->d_bins + n1;
    P.bin3_tab = h->d_bins + n1 + n2;
    P.err = h->d_fixed;
    P.ntiles = h->d_fixed + 3;
    P.epoch = h->d_fixed + 4;
    P.dstep = h->d_fixed + 5;
    P.nincl = h->d_fixed + 6;
    P.scan_done = h->d_fixed + 7;
    P.grp_done = h->d_fixed + 8;
    P.dec_done = h->d_fixed + 8 + 2 * n2;
    P.multi_count = h->d_fixed + 8 + 2 * n2 + kDecDoneSlots;
    P.Tbuf = h->d_tbuf;
    P.tflag = h->d_tflag;
    return TT_OK;
}

void free_handle(tt_emb* h) {
    if (!h) return;
    cudaFree(h->d_tables);
    cudaFree(h->d_bins);
    cudaFree(h->d_fixed);
    cudaFree(h->d_tbuf);
    cudaFree(h->d_tflag);
    cudaFree(h->d_ws);
    cudaFree(h->d_cache_rows);
    cudaFree(h->d_cache_vals);
    cudaFree(h->d_cache_stamp);
    cudaFree(h->d_slice_stamp);
    cudaFree(h->d_cache_acc);
    cudaFree(h->d_cache_state);
    cudaFree(h->d_cache_grad);
    cudaFree(h->d_cache_gmax);
    cudaFree(h->d_cache_touch);
    cudaFree(h->d_cache_list);
    cudaFree(h->d_cache_hidx);
    cudaFree(h->d_cache_claim);
    cudaFree(h->d_freq_keys);
    cudaFree(h->d_freq_counts);
    for (int w = 0; w < 2; ++w)
        for (int i = 0; i <= kMaxStages; ++i)
            if (h->ev[w][i]) cudaEventDestroy(h->ev[w][i]);
    delete h;
}

// Event record that also works during stream capture (as an event node of the graph).
cudaError_t record_stage(cudaEvent_t ev, cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return cudaErrorUnknown;
    return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                               : cudaEventRecord(ev, s);
}

// Launch sequence helper: records stage events when timing is on.
struct Seq {
    tt_emb* h;
    int which;
    cudaStream_t s;
    int n = 0;
    tt_status st = TT_OK;
    Seq(tt_emb* hh, int w, cudaStream_t ss) : h(hh), which(w), s(ss) {
        if (h->timing) {
            if (!h->ev[w][0] && cudaEventCreate(&h->ev[w][0]) != cudaSuccess) st = TT_ERR_CUDA;
            else if (record_stage(h->ev[w][0], s) != cudaSuccess) st = TT_ERR_CUDA;
        }
    }
    void run(const char* name, cudaError_t (*fn)(const Params&, cudaStream_t)) {
        if (st != TT_OK) return;
        cudaError_t e = fn(h->P, s);
        if (e != cudaSuccess) { st = TT_ERR_CUDA; return; }
        if (h->timing && n < kMaxStages) {
            cudaEvent_t& ev = h->ev[which][n + 1];
            if (!ev && cudaEventCreate(&ev) != cudaSuccess) { st = TT_ERR_CUDA; return; }
            if (record_stage(ev, s) != cudaSuccess) { st = TT_ERR_CUDA; return; }
            h->names[which][n] = name;
        }
        ++n;
    }
    tt_status finish() {
        h->launches[which] = n;
        h->nstage[which] = h->timing ? std::min(n, kMaxStages) : 0;
        return st;
    }
};

}  // namespace

extern "C" {

const char* tt_emb_status_string(tt_status s) {
    switch (s) {
        case TT_OK: return "ok";
        case TT_ERR_ARG: return "invalid argument";
        case TT_ERR_SHAPE: return "invalid or unsupported TT shape";
        case TT_ERR_INDEX: return "index outside [0, num_embeddings)";
        case TT_ERR_CUDA: return "CUDA runtime error";
        case TT_ERR_STATE: return "call out of order";
        case TT_ERR_TIMEOUT: return "bounded device wait gave up";
        case TT_ERR_NOMEM: return "device memory allocation failed";
        case TT_ERR_BOUNDS: return "internal index out of bounds (debug build check)";
    }
    return "unknown status";
}

tt_status tt_emb_create(int64_t num_embeddings, const int64_t p[3], const int32_t q[3], const int32_t ranks[2],
                        float* const cores_dev[3], tt_emb** out) {
    if (!out || !p || !q || !ranks || !cores_dev) return TT_ERR_ARG;
    *out = nullptr;
    tt_table_desc d{};
    d.num_embeddings = num_embeddings;
    for (int k = 0; k < 3; ++k) {
        d.p[k] = p[k];
        d.q[k] = q[k];
        d.cores_dev[k] = cores_dev[k];
    }
    d.ranks[0] = ranks[0];
    d.ranks[1] = ranks[1];
    return tt_emb_batch_create(1, &d, out);
}

tt_status tt_emb_batch_create(int32_t num_tables, const tt_table_desc* descs, tt_emb** out) {
    if (!out || !descs || num_tables <= 0) return TT_ERR_ARG;
    *out = nullptr;
    tt_emb* h = new (std::nothrow) tt_emb();
    if (!h) return TT_ERR_NOMEM;
    tt_status st = build_handle(h, num_tables, descs);
    if (st != TT_OK) {
        free_handle(h);
        return st;
    }
    *out = h;
    return TT_OK;
}

void tt_emb_destroy(tt_emb* h) {
    if (!h) return;
    cudaDeviceSynchronize();
    free_handle(h);
}

tt_status tt_emb_reserve(tt_emb* h, int64_t max_nnz, int64_t max_bags) {
    if (!h || max_nnz < 0 || max_bags < 0) return TT_ERR_ARG;
    return ensure_workspace(h, max_nnz, max_bags);
}

tt_status tt_emb_forward(tt_emb* h, const int64_t* indices, int64_t nnz, const int64_t* offsets, int64_t num_bags,
                         const float* weights, tt_pool mode, float* out, tt_stream stream) {
    if (!h || nnz < 0 || num_bags < 0) return TT_ERR_ARG;
    if (mode != TT_POOL_SUM && mode != TT_POOL_MEAN) return TT_ERR_ARG;
    if (num_bags % h->ntab) return TT_ERR_ARG;
    if (nnz > 0 && (!indices || !offsets)) return TT_ERR_ARG;
    if (num_bags > 0 && (!offsets || !out)) return TT_ERR_ARG;
    if (num_bags == 0 && nnz > 0) return TT_ERR_ARG;
    if (nnz >= ((int64_t)1 << 31) - kChunk) return TT_ERR_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    tt_status st = ensure_workspace(h, nnz, num_bags);
    if (st != TT_OK) return st;
    Params& P = h->P;
    P.idx = indices;
    P.off = offsets;
    P.w = weights;
    P.mean = mode == TT_POOL_MEAN;
    P.nnz = nnz;
    P.nbags = num_bags;
    P.bags_per_table = num_bags / h->ntab;
    P.out = out;
    const bool small = use_small_path(h, nnz);
    P.small = small ? 1 : 0;
    P.split = small ? h->split_small : 1;
    P.tile_cap = small ? h->cap_small : h->cap_large;
    P.nch = (int)((std::max<int64_t>(nnz, 1) + (small ? kSmallChunk : kChunk) - 1) / (small ? kSmallChunk : kChunk));
    P.max_tiles = max_tiles_for(h, nnz, P.tile_cap);
    {
        // k_tile_bwd pads the dT rows of each pair by up to 16 floats and the G2 rows
        // by up to 32 floats (bank spreading), on top of the plain sizes
        int g1f = 1, dtf = 1, g2f = 1;
        for (const TableDev& T : h->tabs) {
            const int Ns = T.q2 * (T.r2 / P.split);
            const int pb = bwd_batch_pairs(T.q1, Ns, T.r1);
            g1f = std::max(g1f, pb * T.q1 * T.r1);
            dtf = std::max(dtf, pb * (T.q1 * Ns + 16));
            g2f = std::max(g2f, (T.r1 + 32) * Ns);
        }
        P.g1s_floats = g1f;
        P.dts_floats = dtf;
        P.g2s_floats = g2f;
    }
    P.cache_rows = h->d_cache_rows;
    P.cache_n = h->cache_n;
    P.cache_vals = h->d_cache_vals;
    P.cache_hidx = h->d_cache_hidx;
    P.cache_claim = h->d_cache_claim;
    P.cache_stamp = h->d_cache_stamp;
    P.slice_stamp = h->d_slice_stamp;
    P.cache_train = (h->cache_train && h->cache_n > 0) ? 1 : 0;
    P.cache_acc = h->d_cache_acc;
    P.cache_state = h->d_cache_state;
    P.cache_grad = h->d_cache_grad;
    P.cache_gmax = h->d_cache_gmax;
    P.cache_touch = h->d_cache_touch;
    P.cache_list = h->d_cache_list;
    h->last_stream = s;
    h->has_fwd = false;
    if (num_bags == 0) {
        h->launches[0] = 0;
        h->nstage[0] = 0;
        h->has_fwd = true;
        return TT_OK;
    }
    Seq q(h, 0, s);
    if (nnz == 0) {
        if (cudaMemsetAsync(out, 0, sizeof(float) * (size_t)num_bags * P.D, s) != cudaSuccess) return TT_ERR_CUDA;
    } else {
        if (small) {
            q.run("decode", launch_decode_small);
        } else {
            q.run("decode_hist", launch_decode_hist);
            if (scan_segments(P, 0) > 2) q.run("scan_sums13", launch_scan_sums13);
            q.run("scan13", launch_scan13);
            q.run("scatter13", launch_scatter13);
            if (scan_segments(P, 1) > 1) q.run("scan_sums2", launch_scan_sums2);
            q.run("scan2_tiles", launch_scan2_tiles);
            q.run("scatter2", launch_scatter2);
        }
        q.run("fwd_T", launch_fwd_T);
        q.run("pool", launch_pool);
    }
    st = q.finish();
    if (st == TT_OK) {
        h->has_fwd = true;
    } else if (small) {
        // a pass cut short may not reach k_pool, which advances the epoch: clear the decode
        // stamps so that the next pass's k_fwd_T blocks cannot take them for its own
        cudaMemsetAsync(P.dec_done, 0, sizeof(int) * kDecDoneSlots, s);
    }
    return st;
}

tt_status tt_emb_backward(tt_emb* h, const float* grad_out, float lr, tt_stream stream) {
    if (!h) return TT_ERR_ARG;
    if (!h->has_fwd) return TT_ERR_STATE;
    Params& P = h->P;
    if (P.nbags > 0 && !grad_out) return TT_ERR_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    h->has_fwd = false;
    h->last_stream = s;
    P.grad_out = grad_out;
    P.lr = lr;
    P.slice_stamp = h->d_slice_stamp;
    Seq q(h, 1, s);
    if (P.opt == TT_OPT_GRAD) {  // untouched slices have a zero gradient
        for (const TableDev& T : h->tabs) {
            const size_t n[3] = {(size_t)T.p1 * T.q1 * T.r1, (size_t)T.p2 * T.r1 * T.q2 * T.r2,
                                 (size_t)T.p3 * T.r2 * T.q3};
            for (int k = 0; k < 3; ++k)
                if (cudaMemsetAsync(T.aux[k], 0, sizeof(float) * n[k], s) != cudaSuccess) return TT_ERR_CUDA;
        }
    }
    if (P.cache_train && P.opt == TT_OPT_GRAD &&
        cudaMemsetAsync(h->d_cache_grad, 0, sizeof(float) * (size_t)h->cache_n * P.D, s) != cudaSuccess)
        return TT_ERR_CUDA;
    if (P.nnz > 0) {
        q.run("tile_bwd", launch_tile_bwd);
        q.run("reduce13", launch_reduce13);
        if (P.cache_train) {
            q.run("cache_gmax", launch_cache_gmax);
            q.run("cache_acc", launch_cache_acc);
            q.run("cache_apply", launch_cache_apply);
        }
    }
    tt_status st = q.finish();
    return st;
}

tt_status tt_emb_set_optimizer(tt_emb* h, int32_t optim, float eps, float* const* aux) {
    if (!h) return TT_ERR_ARG;
    if (optim != TT_OPT_SGD && optim != TT_OPT_ADAGRAD && optim != TT_OPT_GRAD) return TT_ERR_ARG;
    if (optim == TT_OPT_ADAGRAD && !(eps >= 0.f && eps <= 3.0e38f)) return TT_ERR_ARG;
    if (optim != TT_OPT_SGD) {
        if (!aux) return TT_ERR_ARG;
        for (int i = 0; i < 3 * h->ntab; ++i)
            if (!aux[i] || ((uintptr_t)aux[i] & 15u) != 0) return TT_ERR_ARG;
    }
    std::vector<TableDev> tabs = h->tabs;
    for (int t = 0; t < h->ntab; ++t)
        for (int k = 0; k < 3; ++k) tabs[t].aux[k] = optim == TT_OPT_SGD ? nullptr : aux[3 * t + k];
    if (cudaMemcpy(h->d_tables, tabs.data(), sizeof(TableDev) * tabs.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return TT_ERR_CUDA;
    }
    h->tabs = tabs;
    h->P.opt = optim;
    h->P.eps = eps;
    return TT_OK;
}

tt_status tt_emb_full_weight(tt_emb* h, int32_t table, int64_t row0, int64_t nrows, float* out_dev,
                             tt_stream stream) {
    if (!h || table < 0 || table >= h->ntab || row0 < 0 || nrows < 0 || (nrows > 0 && !out_dev)) return TT_ERR_ARG;
    const TableDev& T = h->tabs[table];
    if (row0 > T.E || nrows > T.E - row0) return TT_ERR_ARG;
    if (nrows == 0) return TT_OK;
    if (nrows > (int64_t)8 * 0x7fffffff) return TT_ERR_ARG;  // grid limit of the warp-per-row launch
    const cudaError_t e = launch_full_weight(h->d_tables, table, row0, nrows, out_dev, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

static void cache_train_free(tt_emb* h) {
    cudaFree(h->d_cache_acc);
    cudaFree(h->d_cache_state);
    cudaFree(h->d_cache_grad);
    cudaFree(h->d_cache_gmax);
    cudaFree(h->d_cache_touch);
    cudaFree(h->d_cache_list);
    h->d_cache_list = nullptr;
    h->d_cache_acc = nullptr;
    h->d_cache_state = nullptr;
    h->d_cache_grad = nullptr;
    h->d_cache_gmax = nullptr;
    h->d_cache_touch = nullptr;
}

// Gradient state of the trainable cache rows, zeroed: fixed-point sums, Adagrad
// accumulators, last gradients, the two gmax words and the touch flags.
static tt_status cache_train_alloc(tt_emb* h, cudaStream_t s) {
    const size_t nd = (size_t)h->cache_n * h->tabs[0].D;
    if (cudaMalloc(&h->d_cache_acc, sizeof(unsigned long long) * nd) != cudaSuccess ||
        cudaMalloc(&h->d_cache_state, sizeof(float) * nd) != cudaSuccess ||
        cudaMalloc(&h->d_cache_grad, sizeof(float) * nd) != cudaSuccess ||
        cudaMalloc(&h->d_cache_gmax, sizeof(unsigned) * 4) != cudaSuccess ||
        cudaMalloc(&h->d_cache_touch, sizeof(int) * (size_t)h->cache_n) != cudaSuccess ||
        cudaMalloc(&h->d_cache_list, sizeof(int) * (size_t)h->cache_n) != cudaSuccess) {
        cudaGetLastError();
        cache_train_free(h);
        return TT_ERR_NOMEM;
    }
    if (cudaMemsetAsync(h->d_cache_acc, 0, sizeof(unsigned long long) * nd, s) != cudaSuccess ||
        cudaMemsetAsync(h->d_cache_state, 0, sizeof(float) * nd, s) != cudaSuccess ||
        cudaMemsetAsync(h->d_cache_grad, 0, sizeof(float) * nd, s) != cudaSuccess ||
        cudaMemsetAsync(h->d_cache_gmax, 0, sizeof(unsigned) * 4, s) != cudaSuccess ||
        cudaMemsetAsync(h->d_cache_touch, 0, sizeof(int) * (size_t)h->cache_n, s) != cudaSuccess)
        return TT_ERR_CUDA;
    return TT_OK;
}

// Allocate the cache arrays for n slots of table 0 and fill them from host row ids
// (-1 = empty slot); `sets` > 0 selects the set-associative layout.
static tt_status cache_install(tt_emb* h, const std::vector<int64_t>& rows, int sets, cudaStream_t s) {
    const int64_t n = (int64_t)rows.size();
    const TableDev& T = h->tabs[0];
    const int nslice = T.p1 + T.p2 + T.p3;
    if (cudaMalloc(&h->d_cache_rows, sizeof(int64_t) * n) != cudaSuccess ||
        cudaMalloc(&h->d_cache_vals, sizeof(float) * (size_t)n * T.D) != cudaSuccess ||
        cudaMalloc(&h->d_cache_stamp, sizeof(int) * n) != cudaSuccess ||
        cudaMalloc(&h->d_cache_claim, sizeof(int) * n) != cudaSuccess ||
        cudaMalloc(&h->d_slice_stamp, sizeof(int) * nslice) != cudaSuccess) {
        cudaGetLastError();
        tt_emb_cache_disable(h);
        return TT_ERR_NOMEM;
    }
    h->cache_n = n;
    if (h->cache_train) {
        const tt_status st = cache_train_alloc(h, s);
        if (st != TT_OK) {
            tt_emb_cache_disable(h);
            return st;
        }
    }
    if (cudaMemcpyAsync(h->d_cache_rows, rows.data(), sizeof(int64_t) * n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemsetAsync(h->d_slice_stamp, 0, sizeof(int) * nslice, s) != cudaSuccess ||
        cudaMemsetAsync(h->d_cache_claim, 0, sizeof(int) * n, s) != cudaSuccess)  // epochs start at 1
        return TT_ERR_CUDA;
    h->P.cache_sets = sets;
    if (sets == 0) {
        // explicit rows: open-addressing index (load <= 1/2, linear probing from mix64(row))
        int64_t M = 32;
        while (M < 2 * n) M <<= 1;
        std::vector<longlong2> hx((size_t)M, longlong2{-1, 0});
        int maxp = 1;
        for (int64_t i = 0; i < n; ++i) {
            uint64_t e = mix64((uint64_t)rows[i]) & (uint64_t)(M - 1);
            int p = 1;
            while (hx[e].x >= 0) {
                e = (e + 1) & (uint64_t)(M - 1);
                ++p;
            }
            hx[e] = longlong2{(long long)rows[i], (long long)i};
            maxp = std::max(maxp, p);
        }
        if (cudaMalloc(&h->d_cache_hidx, sizeof(longlong2) * M) != cudaSuccess) {
            cudaGetLastError();
            tt_emb_cache_disable(h);
            return TT_ERR_NOMEM;
        }
        if (cudaMemcpyAsync(h->d_cache_hidx, hx.data(), sizeof(longlong2) * M, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return TT_ERR_CUDA;
        h->P.cache_hmask = (int)(M - 1);
        h->P.cache_hprobe = maxp;
    }
    Params P = h->P;
    P.cache_rows = h->d_cache_rows;
    P.cache_n = n;
    P.cache_vals = h->d_cache_vals;
    P.cache_stamp = h->d_cache_stamp;
    if (launch_cache_fill(P, s) != cudaSuccess) return TT_ERR_CUDA;
    // the host vector must outlive the copy
    if (cudaStreamSynchronize(s) != cudaSuccess) return TT_ERR_CUDA;
    return TT_OK;
}

tt_status tt_emb_lfu_enable(tt_emb* h, int64_t cache_size, int64_t hashtbl_size) {
    if (!h || cache_size < 1 || hashtbl_size < 32 || (hashtbl_size & (hashtbl_size - 1)) != 0 ||
        hashtbl_size > ((int64_t)1 << 30) || cache_size > ((int64_t)1 << 30))
        return TT_ERR_ARG;
    if (h->ntab != 1) return TT_ERR_STATE;
    tt_emb_lfu_disable(h);
    if (cudaMalloc(&h->d_freq_keys, sizeof(unsigned long long) * hashtbl_size) != cudaSuccess ||
        cudaMalloc(&h->d_freq_counts, sizeof(unsigned) * hashtbl_size) != cudaSuccess) {
        cudaGetLastError();
        tt_emb_lfu_disable(h);
        return TT_ERR_NOMEM;
    }
    if (cudaMemset(h->d_freq_keys, 0xFF, sizeof(unsigned long long) * hashtbl_size) != cudaSuccess ||
        cudaMemset(h->d_freq_counts, 0, sizeof(unsigned) * hashtbl_size) != cudaSuccess)
        return TT_ERR_CUDA;
    h->freq_size = hashtbl_size;
    h->lfu_slots = (cache_size + kLfuWays - 1) / kLfuWays * kLfuWays;
    h->P.freq_keys = h->d_freq_keys;
    h->P.freq_counts = h->d_freq_counts;
    h->P.freq_mask = (int)(hashtbl_size - 1);
    return TT_OK;
}

tt_status tt_emb_lfu_disable(tt_emb* h) {
    if (!h) return TT_ERR_ARG;
    if (h->d_freq_keys) cudaDeviceSynchronize();
    cudaFree(h->d_freq_keys);
    cudaFree(h->d_freq_counts);
    h->d_freq_keys = nullptr;
    h->d_freq_counts = nullptr;
    h->freq_size = 0;
    h->lfu_slots = 0;
    h->P.freq_keys = nullptr;
    h->P.freq_counts = nullptr;
    h->P.freq_mask = 0;
    return TT_OK;
}

// The frequency table's (row, count) entries, sorted by row.
static tt_status lfu_entries(tt_emb* h, std::vector<std::pair<int64_t, unsigned>>& out) {
    std::vector<unsigned long long> keys(h->freq_size);
    std::vector<unsigned> counts(h->freq_size);
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(keys.data(), h->d_freq_keys, sizeof(unsigned long long) * h->freq_size, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(counts.data(), h->d_freq_counts, sizeof(unsigned) * h->freq_size, cudaMemcpyDeviceToHost) != cudaSuccess)
        return TT_ERR_CUDA;
    out.clear();
    for (int64_t i = 0; i < h->freq_size; ++i)
        if (keys[i] != ~0ull) out.emplace_back((int64_t)keys[i], counts[i]);
    std::sort(out.begin(), out.end());
    return TT_OK;
}

tt_status tt_emb_lfu_read(tt_emb* h, int64_t* rows_host, uint32_t* counts_host, int64_t cap, int64_t* n_out) {
    if (!h || !n_out || cap < 0 || (cap > 0 && (!rows_host || !counts_host))) return TT_ERR_ARG;
    if (!h->d_freq_keys) return TT_ERR_STATE;
    std::vector<std::pair<int64_t, unsigned>> e;
    tt_status st = lfu_entries(h, e);
    if (st != TT_OK) return st;
    *n_out = (int64_t)e.size();
    for (int64_t i = 0; i < (int64_t)e.size() && i < cap; ++i) {
        rows_host[i] = e[i].first;
        counts_host[i] = e[i].second;
    }
    return TT_OK;
}

tt_status tt_emb_lfu_populate(tt_emb* h, tt_stream stream) {
    if (!h) return TT_ERR_ARG;
    if (!h->d_freq_keys) return TT_ERR_STATE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::vector<std::pair<int64_t, unsigned>> e;
    tt_status st = lfu_entries(h, e);
    if (st != TT_OK) return st;
    tt_emb_cache_disable(h);
    const int sets = (int)(h->lfu_slots / kLfuWays);
    // per set: the kLfuWays most frequent counted rows (ties: the smaller row id)
    std::vector<std::vector<std::pair<int64_t, int64_t>>> by_set(sets);  // (-count, row)
    for (const auto& x : e) by_set[lfu_set_of(x.first, sets)].emplace_back(-(int64_t)x.second, x.first);
    std::vector<int64_t> rows((size_t)sets * kLfuWays, -1);
    for (int k = 0; k < sets; ++k) {
        auto& v = by_set[k];
        const size_t take = std::min(v.size(), (size_t)kLfuWays);
        std::partial_sort(v.begin(), v.begin() + take, v.end());
        for (size_t w = 0; w < take; ++w) rows[(size_t)k * kLfuWays + w] = v[w].second;
    }
    return cache_install(h, rows, sets, s);
}

tt_status tt_emb_lfu_cached_rows(tt_emb* h, int64_t* rows_host, int64_t cap, int64_t* n_out) {
    if (!h || !n_out || cap < 0 || (cap > 0 && !rows_host)) return TT_ERR_ARG;
    *n_out = h->cache_n;
    if (h->cache_n == 0) return TT_OK;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(rows_host, h->d_cache_rows, sizeof(int64_t) * (size_t)std::min(cap, h->cache_n),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return TT_ERR_CUDA;
    return TT_OK;
}

tt_status tt_emb_cache_populate(tt_emb* h, const int64_t* rows_dev, int64_t n, tt_stream stream) {
    if (!h || n < 0 || (n > 0 && !rows_dev) || n > ((int64_t)1 << 29)) return TT_ERR_ARG;
    if (h->ntab != 1) return TT_ERR_STATE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    tt_emb_cache_disable(h);
    if (n == 0) return TT_OK;
    // rows are sorted on the host once so that lookups can binary-search them
    std::vector<int64_t> rows(n);
    if (cudaMemcpyAsync(rows.data(), rows_dev, sizeof(int64_t) * n, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return TT_ERR_CUDA;
    std::sort(rows.begin(), rows.end());
    const TableDev& T = h->tabs[0];
    for (int64_t i = 0; i < n; ++i)
        if (rows[i] < 0 || rows[i] >= T.E || (i > 0 && rows[i] == rows[i - 1])) return TT_ERR_ARG;
    return cache_install(h, rows, 0, s);
}

tt_status tt_emb_cache_disable(tt_emb* h) {
    if (!h) return TT_ERR_ARG;
    if (h->cache_n > 0 || h->d_cache_rows) cudaDeviceSynchronize();
    if (h->P.cache_train) {  // the last forward's hit slots refer to this cache
        h->P.cache_train = 0;
        h->has_fwd = false;
    }
    cache_train_free(h);
    cudaFree(h->d_cache_rows);
    cudaFree(h->d_cache_vals);
    cudaFree(h->d_cache_stamp);
    cudaFree(h->d_slice_stamp);
    cudaFree(h->d_cache_hidx);
    cudaFree(h->d_cache_claim);
    h->d_cache_hidx = nullptr;
    h->d_cache_claim = nullptr;
    h->P.cache_hmask = 0;
    h->P.cache_hprobe = 0;
    h->d_cache_rows = nullptr;
    h->d_cache_vals = nullptr;
    h->d_cache_stamp = nullptr;
    h->d_slice_stamp = nullptr;
    h->cache_n = 0;
    h->P.cache_n = 0;
    h->P.cache_sets = 0;
    h->P.slice_stamp = nullptr;
    return TT_OK;
}

tt_status tt_emb_cache_set_trainable(tt_emb* h, int32_t trainable, tt_stream stream) {
    if (!h || (trainable != 0 && trainable != 1)) return TT_ERR_ARG;
    if (h->ntab != 1) return TT_ERR_STATE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (h->cache_n > 0) cudaDeviceSynchronize();
    if (h->P.cache_train) {  // the last forward's hit slots refer to this cache state
        h->P.cache_train = 0;
        h->has_fwd = false;
    }
    cache_train_free(h);
    h->cache_train = trainable != 0;
    if (h->cache_n == 0) return TT_OK;
    if (h->cache_train) {
        const tt_status st = cache_train_alloc(h, s);
        if (st != TT_OK) {
            tt_emb_cache_disable(h);
            return st;
        }
    }
    // the cached values start again from the cores
    Params P = h->P;
    P.cache_rows = h->d_cache_rows;
    P.cache_n = h->cache_n;
    P.cache_vals = h->d_cache_vals;
    P.cache_stamp = h->d_cache_stamp;
    if (launch_cache_fill(P, s) != cudaSuccess) return TT_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

tt_status tt_emb_cache_read(tt_emb* h, float* vals_dev, float* grads_dev, tt_stream stream) {
    if (!h) return TT_ERR_ARG;
    if (grads_dev && !h->cache_train) return TT_ERR_STATE;
    if (h->cache_n == 0) return TT_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t bytes = sizeof(float) * (size_t)h->cache_n * h->tabs[0].D;
    if (vals_dev && cudaMemcpyAsync(vals_dev, h->d_cache_vals, bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return TT_ERR_CUDA;
    if (grads_dev && cudaMemcpyAsync(grads_dev, h->d_cache_grad, bytes, cudaMemcpyDeviceToDevice, s) != cudaSuccess)
        return TT_ERR_CUDA;
    return TT_OK;
}

tt_status tt_emb_cache_write(tt_emb* h, const float* vals_dev, tt_stream stream) {
    if (!h || !vals_dev) return TT_ERR_ARG;
    if (!h->cache_train) return TT_ERR_STATE;
    if (h->cache_n == 0) return TT_OK;
    const size_t bytes = sizeof(float) * (size_t)h->cache_n * h->tabs[0].D;
    return cudaMemcpyAsync(h->d_cache_vals, vals_dev, bytes, cudaMemcpyDeviceToDevice,
                           reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}

tt_status tt_emb_get_decoded(tt_emb* h, int32_t* table_dev, int32_t* i1_dev, int32_t* i2_dev, int32_t* i3_dev,
                             int32_t* bag_dev, tt_stream stream) {
    if (!h) return TT_ERR_ARG;
    if (!h->has_fwd) return TT_ERR_STATE;
    const Params& P = h->P;
    if (P.nnz == 0) return TT_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t bytes = sizeof(int) * (size_t)P.nnz;
    cudaError_t e = cudaSuccess;
    if (i1_dev && e == cudaSuccess) e = cudaMemcpyAsync(i1_dev, P.lk_i1, bytes, cudaMemcpyDeviceToDevice, s);
    if (i2_dev && e == cudaSuccess) e = cudaMemcpyAsync(i2_dev, P.lk_i2, bytes, cudaMemcpyDeviceToDevice, s);
    if (i3_dev && e == cudaSuccess) e = cudaMemcpyAsync(i3_dev, P.lk_i3, bytes, cudaMemcpyDeviceToDevice, s);
    if (bag_dev && e == cudaSuccess) e = cudaMemcpyAsync(bag_dev, P.lk_bag, bytes, cudaMemcpyDeviceToDevice, s);
    if (table_dev && e == cudaSuccess) {
        // table = bag / bags_per_table; derived on the host side of the copy for 1 table
        if (h->ntab == 1) {
            e = cudaMemsetAsync(table_dev, 0, bytes, s);
        } else {
            std::vector<int32_t> bag(P.nnz);
            e = cudaMemcpyAsync(bag.data(), P.lk_bag, bytes, cudaMemcpyDeviceToHost, s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
            for (int64_t n = 0; n < P.nnz && e == cudaSuccess; ++n) bag[n] = (int32_t)(bag[n] / P.bags_per_table);
            if (e == cudaSuccess) e = cudaMemcpyAsync(table_dev, bag.data(), bytes, cudaMemcpyHostToDevice, s);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        }
    }
    return cuda_status(e);
}

tt_status tt_emb_get_last_error(tt_emb* h) {
    if (!h) return TT_ERR_ARG;
    if (cudaStreamSynchronize(h->last_stream) != cudaSuccess) return TT_ERR_CUDA;
    int err = 0;
    if (cudaMemcpy(&err, h->P.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TT_ERR_CUDA;
    if (err && cudaMemset(h->P.err, 0, sizeof(int)) != cudaSuccess) return TT_ERR_CUDA;
    if (err & kErrIndex) return TT_ERR_INDEX;
    if (err & kErrOffsets) return TT_ERR_ARG;
    if (err & kErrTimeout) return TT_ERR_TIMEOUT;
    if (err & kErrBounds) return TT_ERR_BOUNDS;
    return TT_OK;
}

tt_status tt_emb_apply_gradients(tt_emb* h, int32_t optim, float lr, float eps, float* const* grads_dev,
                                 float* const* state_dev, tt_stream stream) {
    if (!h || !grads_dev) return TT_ERR_ARG;
    if (optim != TT_OPT_SGD && optim != TT_OPT_ADAGRAD) return TT_ERR_ARG;
    if (optim == TT_OPT_ADAGRAD && (!state_dev || !(eps >= 0.f && eps <= 3.0e38f))) return TT_ERR_ARG;
    for (int i = 0; i < 3 * h->ntab; ++i) {
        if (!grads_dev[i] || ((uintptr_t)grads_dev[i] & 15u) != 0) return TT_ERR_ARG;
        if (optim == TT_OPT_ADAGRAD && (!state_dev[i] || ((uintptr_t)state_dev[i] & 15u) != 0)) return TT_ERR_ARG;
    }
    if (h->cache_train && h->cache_n > 0) return TT_ERR_STATE;  // cached values have gradients of their own
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ApplyArgs a{};
    a.opt = optim;
    a.lr = lr;
    a.eps = eps;
    a.dstep = h->P.dstep;
    for (int t = 0; t < h->ntab; ++t) {
        const TableDev& T = h->tabs[t];
        const int64_t sz[3] = {(int64_t)T.q1 * T.r1, (int64_t)T.r1 * T.q2 * T.r2, (int64_t)T.r2 * T.q3};
        const int64_t np[3] = {T.p1, T.p2, T.p3};
        float* G[3] = {T.G1, T.G2, T.G3};
        const int64_t soff[3] = {0, T.p1, (int64_t)T.p1 + T.p2};
        for (int k = 0; k < 3; ++k) {
            const int sg = a.nseg;
            a.G[sg] = G[k];
            a.g[sg] = grads_dev[3 * t + k];
            a.s[sg] = optim == TT_OPT_ADAGRAD ? state_dev[3 * t + k] : nullptr;
            a.n[sg] = np[k] * sz[k];
            a.slice_elems[sg] = sz[k];
            a.stamp[sg] = (t == 0 && h->d_slice_stamp && !h->cache_train) ? h->d_slice_stamp + soff[k] : nullptr;
            a.start[sg + 1] = a.start[sg] + (a.n[sg] + 3) / 4;
            ++a.nseg;
            if (a.nseg == kApplySegs || (t == h->ntab - 1 && k == 2)) {
                if (launch_apply_grads(a, h->P.sms, s) != cudaSuccess) return TT_ERR_CUDA;
                a.nseg = 0;
                a.start[0] = 0;
            }
        }
    }
    h->last_stream = s;
    return TT_OK;
}

tt_status tt_emb_set_wait_limit(tt_emb* h, uint32_t polls) {
    if (!h) return TT_ERR_ARG;
    h->P.wait_polls = polls;
    return TT_OK;
}

tt_status tt_emb_set_stage_timing(tt_emb* h, int enable) {
    if (!h) return TT_ERR_ARG;
    h->timing = enable != 0;
    return TT_OK;
}

int tt_emb_stage_times(tt_emb* h, int which, float* ms, const char** names, int cap) {
    if (!h || which < 0 || which > 1 || cap < 0) return -1;
    const int n = h->nstage[which];
    if (n == 0) return h->launches[which];
    if (cudaEventSynchronize(h->ev[which][n]) != cudaSuccess) return -1;
    for (int i = 0; i < n && i < cap; ++i) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, h->ev[which][i], h->ev[which][i + 1]) != cudaSuccess) return -1;
        if (ms) ms[i] = t;
        if (names) names[i] = h->names[which][i];
    }
    return h->launches[which];
}

int tt_emb_last_launch_count(tt_emb* h, int which) {
    if (!h || which < 0 || which > 1) return -1;
    return h->launches[which];
}

}  // extern "C"
