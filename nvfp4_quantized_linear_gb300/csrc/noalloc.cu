// nvfp4_linear_noalloc: the NVFP4 linear layer with built-in scratch memory.
//
// nvfp4_linear needs a caller-provided workspace (the quantized activation and
// its block scales).  Some callers have no way to provide one: code that runs
// inside a host framework which owns every device allocation and hands a
// plugin only its inputs and outputs, or latency-critical code that must never
// call cudaMalloc (it can synchronise the whole device and may fail under
// memory pressure at a bad moment).  For them this entry point uses a fixed
// scratch array compiled into the library instead; it allocates nothing.
//
// The scratch is a file-scope __device__ array of kScratchBytes (16 MiB).
// Every GPU that loads the library holds it until the process exits.  In host
// code the array's name is only a host-side stand-in, never a device address:
// the device address is looked up with cudaGetSymbolAddress, with the device
// current, by the first call made on that device, checked, and kept.  That
// first call should therefore come before any stream capture.  The address
// belongs to the device's current CUDA context: if that context is torn down
// and re-created (cudaDeviceReset), the module holding the array is loaded
// again and may sit elsewhere, so the kept address is tagged with the
// context's id and the look-up is repeated when the id changes.  All calls on
// a device share the one array, so calls whose work overlaps on the GPU (for
// instance on two streams) race on it.
#include <cstdio>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "nvfp4.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;   // 16 MiB

// Shared by every call on a device; it keeps the previous call's contents.
// Nothing in it has to start at zero: each call rewrites every byte of the
// quantized activation and scales that its GEMM reads.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
    void *ptr = nullptr;                  // device address of g_noalloc_scratch
    unsigned long long ctx_id = 0;        // id of the context it was looked up in
};
ScratchSlot g_scratch[kMaxDevices];
std::mutex g_scratch_mutex;

nvfp4_status noalloc_fail(nvfp4_status st, const char *msg)
{
    return static_cast<nvfp4_status>(nvfp4::record_error(st, msg));
}

// Id of the calling thread's current CUDA context (the device's primary
// context once the runtime has set it up), through the driver entry points
// the runtime exposes; false if it cannot be read.
bool current_context_id(unsigned long long *id)
{
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    return get_current != nullptr && get_id != nullptr && get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
           get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of this device's scratch array: looked up on the first call
// made on the device, and again whenever the device's context has changed.
nvfp4_status scratch_address(void **ptr)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return noalloc_fail(NVFP4_ERR_CUDA, "nvfp4_linear_noalloc: cannot determine the current CUDA device");
    }
    // A thread that has made no runtime call needing the context yet may have
    // none current; the symbol look-up below then makes the device's primary
    // context current, and its id is read after it.
    unsigned long long ctx = 0;
    const bool have_ctx = current_context_id(&ctx);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ScratchSlot &slot = g_scratch[dev];
    if (!have_ctx || slot.ptr == nullptr || slot.ctx_id != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            char msg[200];
            snprintf(msg, sizeof msg, "nvfp4_linear_noalloc: cudaGetSymbolAddress of the scratch array failed: %s",
                     cudaGetErrorString(e));
            return noalloc_fail(NVFP4_ERR_CUDA, msg);
        }
        if (!current_context_id(&ctx))
            return noalloc_fail(NVFP4_ERR_CUDA, "nvfp4_linear_noalloc: cannot identify the current CUDA context");
        slot.ptr = p;
        slot.ctx_id = ctx;
    }
    *ptr = slot.ptr;
    return NVFP4_OK;
}

}  // namespace

extern "C" {

nvfp4_status nvfp4_linear_noalloc(const void *x_bf16, int64_t m, int64_t k, int64_t ldx, const float *gs_dev,
                                  const void *transform_bf16, int bs, const uint8_t *w_fp4, const uint8_t *w_sf,
                                  int64_t n_w, int64_t n_out, const float *alpha_dev, const void *bias_bf16,
                                  void *out_bf16, int64_t ldo, nvfp4_stream_t stream)
{
    if (m == 0)   // an empty call needs no scratch; let the regular checks answer it
        return nvfp4_linear(x_bf16, m, k, ldx, gs_dev, transform_bf16, bs, w_fp4, w_sf, n_w, n_out, alpha_dev,
                            bias_bf16, out_bf16, ldo, nullptr, 0, stream);
    const size_t need = nvfp4::linear_min_workspace_bytes(m, k);
    if (m < 0 || k < 1 || need > kScratchBytes) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "nvfp4_linear_noalloc: m=%lld, k=%lld needs %zu bytes of scratch; the built-in scratch holds %zu "
                 "bytes (use nvfp4_linear with a workspace instead)",
                 (long long)m, (long long)k, need, kScratchBytes);
        return noalloc_fail(m < 0 || k < 1 ? NVFP4_ERR_INVALID_ARG : NVFP4_ERR_WORKSPACE, msg);
    }
    void *scratch = nullptr;
    nvfp4_status st = scratch_address(&scratch);
    if (st != NVFP4_OK) return st;
    return nvfp4_linear(x_bf16, m, k, ldx, gs_dev, transform_bf16, bs, w_fp4, w_sf, n_w, n_out, alpha_dev,
                        bias_bf16, out_bf16, ldo, scratch, kScratchBytes, stream);
}

}  // extern "C"
