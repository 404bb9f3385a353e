// tt_noalloc.cu -- a forward pass that allocates no device memory.
//
// Some callers cannot call cudaMalloc: code that runs under a memory manager
// which owns all device memory (a framework's caching allocator, a serving
// runtime with a fixed budget), and code that must not synchronize the device
// (cudaMalloc and cudaFree may do so) or that runs while a stream is being
// captured into a CUDA graph, where allocating is not allowed.  For them,
// tt_emb_forward_noalloc() computes the same pooled output as tt_emb_forward()
// without a handle and without any allocation: the caller passes the cores,
// the bags and the output, and the kernel's only scratch (one partial product
// T = G1[i1] G2[i2] per warp) lives in the file-scope array below.
//
// The array is TT_NOALLOC_SCRATCH_BYTES (8 MiB) per GPU, held by every GPU
// that loads the library until the process exits.  All calls share it and it keeps the
// previous call's contents; the kernel writes each slot before reading it, so
// nothing needs clearing.  Calls whose kernels overlap on the GPU (different
// streams without ordering) race on the array and give wrong results.
#include <mutex>

#include "../../include/tt_emb.h"
#include "tt_internal.cuh"

namespace {

constexpr int64_t kScratchFloats = TT_NOALLOC_SCRATCH_BYTES / sizeof(float);
constexpr int kWarps = 8;       // warps per block
constexpr int kWarpsPerSm = 16; // grid cap: resident warps per SM the grid aims for
constexpr int kMaxDevices = 256;

static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];

float* g_scratch_addr[kMaxDevices];  // device address of the array, per device
int g_sm_count[kMaxDevices];         // multiprocessors of the device
std::mutex g_setup_mutex;

struct NoAllocArgs {
    int64_t E;
    int p1, p2, p3, q1, q2, q3, r1, r2, D;
    const float* G1;
    const float* G2;
    const float* G3;
    const int64_t* idx;
    const int64_t* off;
    const float* w;
    int mean;
    int64_t nnz;
    int64_t nbags;
    float* out;
    int* err;
};

// One warp per bag (grid-stride over bags).  For every lookup the warp forms
// T = G1[i1] G2[i2] in its scratch slot, then row = T G3[i3], pooled in registers.
__global__ void __launch_bounds__(kWarps * 32) k_pool_noalloc(const __grid_constant__ NoAllocArgs a, float* scratch) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * kWarps;
    const int N = a.q2 * a.r2, TS = a.q1 * N;
    float* Tw = scratch + warp * TS;
    if (warp == 0 && lane == 0 && (a.off[0] != 0 || a.off[a.nbags] != a.nnz) && a.err) atomicOr(a.err, 2);
    for (int64_t bag = warp; bag < a.nbags; bag += nwarps) {
        int64_t lo = a.off[bag], hi = a.off[bag + 1];
        if (hi < lo && a.err && lane == 0) atomicOr(a.err, 2);
        lo = lo < 0 ? 0 : (lo > a.nnz ? a.nnz : lo);
        hi = hi < lo ? lo : (hi > a.nnz ? a.nnz : hi);
        float acc[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) acc[m] = 0.f;
        for (int64_t n = lo; n < hi; ++n) {
            int64_t row = a.idx[n];
            float s = a.w ? a.w[n] : 1.f;
            if (row < 0 || row >= a.E) {
                if (a.err && lane == 0) atomicOr(a.err, 1);
                continue;
            }
            if (a.mean) s = s / (float)(hi - lo);
            const int64_t p23 = (int64_t)a.p2 * a.p3;
            const int i1 = (int)(row / p23), i2 = (int)((row / a.p3) % a.p2), i3 = (int)(row % a.p3);
            const float* g1 = a.G1 + (int64_t)i1 * a.q1 * a.r1;
            const float* g2 = a.G2 + (int64_t)i2 * a.r1 * N;
            for (int e = lane; e < TS; e += 32) {
                const int j1 = e / N, jc = e - j1 * N;
                float t = 0.f;
                for (int c = 0; c < a.r1; ++c) t = fmaf(g1[j1 * a.r1 + c], g2[c * N + jc], t);
                Tw[e] = t;
            }
            __syncwarp();
            const float* g3 = a.G3 + (int64_t)i3 * a.r2 * a.q3;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int j = lane + 32 * m;
                if (j < a.D) {
                    const int j12 = j / a.q3, j3 = j - j12 * a.q3;
                    float v = 0.f;
                    for (int c = 0; c < a.r2; ++c) v = fmaf(Tw[j12 * a.r2 + c], g3[c * a.q3 + j3], v);
                    acc[m] = fmaf(s, v, acc[m]);
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int j = lane + 32 * m;
            if (j < a.D) a.out[bag * a.D + j] = acc[m];
        }
    }
}

// Device address of the scratch array on the current device and the device's
// multiprocessor count, looked up once per device.
tt_status scratch_address(float** out, int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TT_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return TT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        int n = 0;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            return TT_ERR_CUDA;
        }
        g_sm_count[dev] = n;
        g_scratch_addr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_addr[dev];
    *sms = g_sm_count[dev];
    return TT_OK;
}

}  // namespace

extern "C" tt_status tt_emb_forward_noalloc(int64_t num_embeddings, const int64_t p[3], const int32_t q[3],
                                            const int32_t ranks[2], const float* const cores_dev[3],
                                            const int64_t* indices_dev, int64_t nnz, const int64_t* offsets_dev,
                                            int64_t num_bags, const float* per_sample_weights_dev, tt_pool mode,
                                            float* out_dev, int32_t* err_dev, tt_stream stream) {
    if (!p || !q || !ranks || !cores_dev || nnz < 0 || num_bags < 0) return TT_ERR_ARG;
    if (mode != TT_POOL_SUM && mode != TT_POOL_MEAN) return TT_ERR_ARG;
    if (!cores_dev[0] || !cores_dev[1] || !cores_dev[2]) return TT_ERR_ARG;
    if (num_bags > 0 && (!offsets_dev || !out_dev)) return TT_ERR_ARG;
    if (nnz > 0 && (!indices_dev || num_bags == 0)) return TT_ERR_ARG;
    if (num_embeddings <= 0) return TT_ERR_SHAPE;
    for (int k = 0; k < 3; ++k)
        if (p[k] <= 0 || p[k] > TT_MAX_P || q[k] <= 0 || q[k] > TT_MAX_Q) return TT_ERR_SHAPE;
    if (ranks[0] <= 0 || ranks[1] <= 0 || ranks[0] > TT_MAX_RANK || ranks[1] > TT_MAX_RANK) return TT_ERR_SHAPE;
    if (p[0] * p[1] * p[2] < num_embeddings) return TT_ERR_SHAPE;
    const int64_t D = (int64_t)q[0] * q[1] * q[2];
    if (D > TT_MAX_D) return TT_ERR_SHAPE;
    // one partial product per warp must fit the static scratch (at least one block of warps)
    const int64_t ts = (int64_t)q[0] * q[1] * ranks[1];
    if (ts * kWarps > kScratchFloats) return TT_ERR_SHAPE;
    float* scratch = nullptr;
    int sms = 0;
    tt_status st = scratch_address(&scratch, &sms);
    if (st != TT_OK) return st;
    if (num_bags == 0) return TT_OK;
    NoAllocArgs a{};
    a.E = num_embeddings;
    a.p1 = (int)p[0]; a.p2 = (int)p[1]; a.p3 = (int)p[2];
    a.q1 = q[0]; a.q2 = q[1]; a.q3 = q[2];
    a.r1 = ranks[0]; a.r2 = ranks[1];
    a.D = (int)D;
    a.G1 = cores_dev[0]; a.G2 = cores_dev[1]; a.G3 = cores_dev[2];
    a.idx = indices_dev;
    a.off = offsets_dev;
    a.w = per_sample_weights_dev;
    a.mean = mode == TT_POOL_MEAN;
    a.nnz = nnz;
    a.nbags = num_bags;
    a.out = out_dev;
    a.err = err_dev;
    // whole blocks of warps, every warp's slot inside the array
    int64_t warps = (num_bags + kWarps - 1) / kWarps * kWarps;
    if (warps > (int64_t)sms * kWarpsPerSm) warps = (int64_t)sms * kWarpsPerSm;
    if (warps * ts > kScratchFloats) warps = (kScratchFloats / ts) / kWarps * kWarps;
    const unsigned blocks = (unsigned)(warps / kWarps);
    k_pool_noalloc<<<blocks, kWarps * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a, scratch);
    return cudaGetLastError() == cudaSuccess ? TT_OK : TT_ERR_CUDA;
}
