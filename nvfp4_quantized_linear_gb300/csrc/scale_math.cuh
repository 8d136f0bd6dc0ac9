// Scale arithmetic shared by the quantizer kernels.
#pragma once

#include <cuda_runtime.h>

namespace nvfp4 {

// x / 6 for the block-scale step s = (amax * gs) / 6.  Markstein's FMA
// correction (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q0 = x * RN(1/6),
// the residual r = x - 6 q0 is exact in one FMA, and q0 + r * RN(1/6) rounds
// to the correctly rounded quotient.  An exhaustive GPU test
// (tests/test_gpu_scale_math.py) checks, over every non-negative float, that
// e4m3(div6_rn(x)) == e4m3(x / 6) with IEEE division, and that the quotients
// agree wherever the IEEE quotient is normal; they can differ only where it is
// subnormal (x < 6 * 2^-126), whose scale code is 0 either way.
// Infinity is passed through (the residual would be NaN).
__device__ __forceinline__ float div6_rn(float x)
{
    const float c = 0.16666667f;                       // RN(1/6)
    const float q0 = __fmul_rn(x, c);
    const float r = __fmaf_rn(-q0, 6.0f, x);
    const float q1 = __fmaf_rn(r, c, q0);
    return isinf(x) ? x : q1;
}

}  // namespace nvfp4
