// Exhaustive check of div6_rn (the quantizer's division by 6) against IEEE
// division: for every non-negative float x, the E4M3 scale code of the
// quotient must be the same.  Built and run by tests/test_gpu_scale_math.py.
#include <cstdint>
#include <cuda_runtime.h>

#include "scale_math.cuh"

namespace {

__device__ __forceinline__ uint32_t e4m3_code(float s)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
    return r & 0xFFu;
}

__global__ void check(unsigned long long *counts)
{
    unsigned long long code_diff = 0, quot_diff_normal = 0;
    for (uint32_t b = blockIdx.x * blockDim.x + threadIdx.x; b < 0x80000000u; b += gridDim.x * blockDim.x) {
        const float x = __uint_as_float(b);
        const float ref = __fdiv_rn(x, 6.0f), got = nvfp4::div6_rn(x);
        if (e4m3_code(ref) != e4m3_code(got)) ++code_diff;
        const bool both_nan = isnan(ref) && isnan(got);
        const bool normal_quotient = __float_as_uint(ref) >= 0x00800000u;   // (sign bit clear here)
        if (!both_nan && normal_quotient && __float_as_uint(ref) != __float_as_uint(got)) ++quot_diff_normal;
    }
    atomicAdd(&counts[0], code_diff);
    atomicAdd(&counts[1], quot_diff_normal);
}

}  // namespace

// counts[0]: inputs whose scale code differs; counts[1]: inputs whose IEEE
// quotient is normal but whose div6_rn quotient differs.  Returns a cudaError_t value.
extern "C" int run_check_div6(unsigned long long *counts_host)
{
    unsigned long long *d = nullptr;
    cudaError_t e = cudaMalloc(&d, 2 * sizeof(unsigned long long));
    if (e == cudaSuccess) e = cudaMemset(d, 0, 2 * sizeof(unsigned long long));
    if (e == cudaSuccess) {
        check<<<2048, 256>>>(d);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(counts_host, d, 2 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(d);
    return (int)e;
}
