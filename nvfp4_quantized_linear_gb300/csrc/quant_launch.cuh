// Launchers of the MXFP4 quantizer and of the dynamic global-scale pass
// (quant.cu), declared apart from the headers the GEMM kernels share.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace nvfp4 {

// MXFP4 quantizer: p.nb = kp / 32 scale columns, p.nbp = roundup(nb, 4), no gs.
cudaError_t launch_quant_mx(const QuantParams &p, int num_sms, cudaStream_t s);

// Dynamic global scale: max |v| over the activation (of the transformed y when
// p.bs != 0) into *gs_out as bf16 bits, then gs = fl32(2688 / amax) in place
// (FLT_MAX on overflow, 1 for amax == 0) and, with w_gs, alpha = 1/(gs * w_gs).
cudaError_t launch_act_global_scale(const QuantParams &p, const float *w_gs, float *gs_out, float *alpha_out,
                                    int num_sms, cudaStream_t s, const char **why);

}  // namespace nvfp4
