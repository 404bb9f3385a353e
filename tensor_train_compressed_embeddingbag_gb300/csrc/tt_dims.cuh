// tt_dims.cuh -- compile-time or run-time TT dimensions for the kernel bodies.
//
// Each kernel body is a template over a dimension type: SDims<q1,q2,q3,r1,r2>
// makes every loop bound a constant (fully unrolled register tiles), DDims
// carries the dimensions of an arbitrary table at run time.  A table's
// `dclass` (set when the handle is created) selects the instantiation.
#pragma once

#include "tt_internal.cuh"

namespace ttemb {

template <int Q1, int Q2, int Q3, int R1, int R2>
struct SDims {
    static constexpr bool kStatic = true;
    __device__ __forceinline__ static constexpr int q1() { return Q1; }
    __device__ __forceinline__ static constexpr int q2() { return Q2; }
    __device__ __forceinline__ static constexpr int q3() { return Q3; }
    __device__ __forceinline__ static constexpr int r1() { return R1; }
    __device__ __forceinline__ static constexpr int r2() { return R2; }
};

struct DDims {
    static constexpr bool kStatic = false;
    int q1_, q2_, q3_, r1_, r2_;
    __device__ __forceinline__ int q1() const { return q1_; }
    __device__ __forceinline__ int q2() const { return q2_; }
    __device__ __forceinline__ int q3() const { return q3_; }
    __device__ __forceinline__ int r1() const { return r1_; }
    __device__ __forceinline__ int r2() const { return r2_; }
};

// Dimension classes with a compiled fast path (TableDev::dclass).
enum DimClass { kDynamic = 0, kQ444R32 = 1, kQ444R16 = 2, kQ444R64 = 3, kQ448R64 = 4 };

inline int dim_class(int q1, int q2, int q3, int r1, int r2) {
    if (q1 == 4 && q2 == 4 && q3 == 4 && r1 == r2) {
        if (r1 == 32) return kQ444R32;
        if (r1 == 16) return kQ444R16;
        if (r1 == 64) return kQ444R64;
    }
    if (q1 == 4 && q2 == 4 && q3 == 8 && r1 == 64 && r2 == 64) return kQ448R64;
    return kDynamic;
}

}  // namespace ttemb
