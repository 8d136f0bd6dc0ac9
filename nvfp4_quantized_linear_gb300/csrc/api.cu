// C ABI of the NVFP4 linear layer (declared and documented in include/nvfp4.h).
// Host-side argument validation, size queries and kernel launches; no memory
// is allocated and no stream is synchronised here.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "quant_launch.cuh"
#include "nvfp4.h"

namespace {

thread_local std::string g_last_error;

nvfp4_status fail(nvfp4_status st, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

nvfp4_status ok()
{
    g_last_error.clear();
    return NVFP4_OK;
}

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int num_sms = 0;
    char reason[160] = {0};
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_dev_mutex;

// Probes (once) whether `dev` can run the sm_103a kernels of this library.
const DeviceInfo *device_info(int dev)
{
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &d = g_devices[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            snprintf(d.reason, sizeof d.reason, "cannot query CUDA device %d", dev);
            return &d;   // not marked probed: a later call may succeed
        }
        d.num_sms = sms;
        d.supported = (major == 10 && minor == 3);
        if (!d.supported)
            snprintf(d.reason, sizeof d.reason,
                     "NVFP4 GB300 kernels are built for sm_103a only; device %d is sm_%d%d", dev, major, minor);
        d.probed = true;
    }
    return &d;
}

nvfp4_status current_device(int *num_sms)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(NVFP4_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    }
    const DeviceInfo *d = device_info(dev);
    if (d == nullptr || !d->probed) return fail(NVFP4_ERR_CUDA, "%s", d ? d->reason : "device index out of range");
    if (!d->supported) return fail(NVFP4_ERR_UNSUPPORTED_DEVICE, "%s", d->reason);
    *num_sms = d->num_sms;
    return NVFP4_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;   // [lo, hi)
    const char *name;
};

Range range(const void *p, size_t bytes, const char *name)
{
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return {lo, lo + bytes, name};
}

// Strided 2-D bf16 matrix: rows x cols elements, row stride ld elements.
Range range2d(const void *p, int64_t rows, int64_t cols, int64_t ld, const char *name)
{
    size_t bytes = rows > 0 ? (size_t)((rows - 1) * ld + cols) * 2 : 0;
    return range(p, bytes, name);
}

bool overlap(const Range &a, const Range &b) { return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo; }

nvfp4_status check_aliases(const Range *outs, int n_out, const Range *ins, int n_in)
{
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_in; ++j)
            if (overlap(outs[i], ins[j]))
                return fail(NVFP4_ERR_ALIAS, "output %s overlaps input %s", outs[i].name, ins[j].name);
        for (int j = i + 1; j < n_out; ++j)
            if (overlap(outs[i], outs[j]))
                return fail(NVFP4_ERR_ALIAS, "output %s overlaps output %s", outs[i].name, outs[j].name);
    }
    return NVFP4_OK;
}

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1024;

nvfp4_status check_quant_args(const void *x, int64_t m, int64_t k, int64_t ldx, const float *gs, const void *t,
                              int bs, const uint8_t *x_fp4, const uint8_t *x_sf, const char *xname)
{
    if (m < 0 || m > kMaxDim) return fail(NVFP4_ERR_INVALID_ARG, "rows of %s out of range: %lld", xname, (long long)m);
    if (k < 1 || k > kMaxDim) return fail(NVFP4_ERR_INVALID_ARG, "k out of range: %lld", (long long)k);
    if (ldx < k) return fail(NVFP4_ERR_INVALID_ARG, "row stride of %s (%lld) < k (%lld)", xname, (long long)ldx, (long long)k);
    if ((int64_t)((m + 127) / 128) * 128 * nvfp4::scale_cols_padded(k) > (int64_t(1) << 40) ||
        nvfp4::rows_padded(m) * ((nvfp4::padded_k(k) + 511) / 512) >= (int64_t(1) << 31))
        return fail(NVFP4_ERR_INVALID_ARG, "tensor too large (%lld x %lld)", (long long)m, (long long)k);
    if (m == 0) return NVFP4_OK;
    if (!x || !gs || !x_fp4 || !x_sf) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    if (bs != 0 || t != nullptr) {
        if (!t) return fail(NVFP4_ERR_INVALID_ARG, "bs = %d given without a transform matrix", bs);
        if (bs != 16 && bs != 32 && bs != 64 && bs != 128)
            return fail(NVFP4_ERR_INVALID_ARG, "transform block size must be 16, 32, 64 or 128 (got %d)", bs);
        if (k % bs != 0) return fail(NVFP4_ERR_INVALID_ARG, "transform block size %d does not divide k = %lld", bs, (long long)k);
        if (!aligned16(t)) return fail(NVFP4_ERR_ALIGNMENT, "transform matrix not 16-byte aligned");
    }
    if (!aligned16(x) || (ldx % 8) != 0)
        return fail(NVFP4_ERR_ALIGNMENT, "%s rows must start on 16-byte boundaries (pointer and ld %% 8 == 0)", xname);
    if (!aligned16(x_fp4) || !aligned16(x_sf)) return fail(NVFP4_ERR_ALIGNMENT, "packed / scale outputs must be 16-byte aligned");
    return NVFP4_OK;
}

nvfp4::QuantParams quant_params(const void *x, int64_t m, int64_t k, int64_t ldx, const float *gs, const void *t,
                                int bs, uint8_t *x_fp4, uint8_t *x_sf)
{
    nvfp4::QuantParams p;
    p.x = static_cast<const uint16_t *>(x);
    p.ldx = ldx;
    p.m = (int32_t)m;
    p.k = (int32_t)k;
    p.kp = (int32_t)nvfp4::padded_k(k);
    p.nb = (int32_t)nvfp4::scale_cols(k);
    p.nbp = (int32_t)nvfp4::scale_cols_padded(k);
    p.mp = (int32_t)nvfp4::rows_padded(m);
    p.gs = gs;
    p.out = x_fp4;
    p.sf = x_sf;
    p.t = static_cast<const uint16_t *>(t);
    p.bs = t ? bs : 0;
    p.err_flag = nullptr;
    p.y_out = nullptr;
    return p;
}

nvfp4_status launch_status(cudaError_t e, const char *what)
{
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(NVFP4_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
    }
    return ok();
}

nvfp4_status run_quant(nvfp4::QuantParams p, int num_sms, cudaStream_t s)
{
    if (p.bs) {
        cudaError_t e = nvfp4::device_error_word(&p.err_flag);
        if (e != cudaSuccess) return launch_status(e, "transform-quantize kernel (error word)");
        const char *why = nullptr;
        e = nvfp4::launch_quant_transform(p, num_sms, s, &why);
        if (why) return fail(NVFP4_ERR_CUDA, "%s", why);
        return launch_status(e, "transform-quantize kernel");
    }
    return launch_status(nvfp4::launch_quant(p, num_sms, s), "quantize kernel");
}

nvfp4_status check_gemm_args(const uint8_t *a, const uint8_t *a_sf, int64_t m, const uint8_t *w, const uint8_t *w_sf,
                             int64_t n_w, int64_t n_out, int64_t k, const float *alpha, const void *bias, void *out,
                             int64_t ldo)
{
    if (m < 0 || m > kMaxDim) return fail(NVFP4_ERR_INVALID_ARG, "m out of range: %lld", (long long)m);
    if (k < 1 || k > kMaxDim) return fail(NVFP4_ERR_INVALID_ARG, "k out of range: %lld", (long long)k);
    if (n_w < 1 || n_w > kMaxDim) return fail(NVFP4_ERR_INVALID_ARG, "n_w out of range: %lld", (long long)n_w);
    if (n_out < 1 || n_out > n_w)
        return fail(NVFP4_ERR_INVALID_ARG, "n_out must satisfy 1 <= n_out <= n_w (got %lld, n_w %lld)", (long long)n_out, (long long)n_w);
    if (ldo < n_out) return fail(NVFP4_ERR_INVALID_ARG, "ldo (%lld) < n_out (%lld)", (long long)ldo, (long long)n_out);
    if (m == 0) return NVFP4_OK;
    if (!w || !w_sf || !out) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(w) || !aligned16(w_sf)) return fail(NVFP4_ERR_ALIGNMENT, "weight buffers must be 16-byte aligned");
    if (!aligned16(out) || (ldo % 8) != 0)
        return fail(NVFP4_ERR_ALIGNMENT, "output rows must start on 16-byte boundaries (pointer and ldo %% 8 == 0)");
    if (bias && !aligned16(bias)) return fail(NVFP4_ERR_ALIGNMENT, "bias must be 16-byte aligned");
    if (a != nullptr || a_sf != nullptr) {   // standalone GEMM: check the activation too
        if (!a || !a_sf) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
        if (!aligned16(a) || !aligned16(a_sf)) return fail(NVFP4_ERR_ALIGNMENT, "activation buffers must be 16-byte aligned");
    }
    return NVFP4_OK;
}

// Scale columns (padded to 4) of an operand with logical K = k: NVFP4 has one
// per 16 elements of the padded K, MXFP4 one per 32.
int64_t scale_cols_of(int64_t k, bool mx)
{
    return mx ? (nvfp4::padded_k(k) / 32 + 3) / 4 * 4 : nvfp4::scale_cols_padded(k);
}

nvfp4::GemmParams gemm_params(const uint8_t *a_sf, int64_t m, const uint8_t *w_sf, int64_t n_w, int64_t n_out,
                              int64_t k, const float *alpha, const void *bias, void *out, int64_t ldo,
                              unsigned int *err, bool mx = false)
{
    nvfp4::GemmParams g;
    g.m = (int32_t)m;
    g.n_w = (int32_t)n_w;
    g.n_out = (int32_t)n_out;
    g.kp = (int32_t)nvfp4::padded_k(k);
    const int64_t nbp = scale_cols_of(k, mx);
    g.num_k64 = (int32_t)((g.kp + 63) / 64);
    g.sf_tiles = (int32_t)(nbp / 4);
    g.mx = mx ? 1 : 0;
    g.num_m_blk = (int32_t)((m + 127) / 128);
    g.num_n_blk = (int32_t)((n_out + 255) / 256);
    g.sfa = a_sf;
    g.sfb = w_sf;
    g.sfa_band_bytes = 128 * nbp;
    g.sfb_band_bytes = 128 * nbp;
    g.alpha = alpha;
    g.bias = static_cast<const uint16_t *>(bias);
    g.out = static_cast<uint16_t *>(out);
    g.ldo = ldo;
    g.err_flag = err;
    g.splits = 1;
    g.stages_per_split = (g.num_k64 + 3) / 4;
    g.group_offsets = nullptr;
    g.num_groups = 0;
    g.group_n = 0;
    g.wait_ns = nvfp4::kDefaultWaitNs;
    g.drill = 0;
    return g;
}

// Split-K plan for small m (a single 128-row band), where one CTA per 128 x 256
// output tile leaves SMs idle while the weight streams.  K is cut into
// `splits` ranges of whole 256-element stages; the ranges of a tile run as one
// thread-block cluster and sum their partials through distributed shared
// memory.  The count is the one with the fewest waves of clusters,
// ceil(tiles / clusters resident at once), and among those the most ranges:
// more SMs stream the weight, each a shorter range, while a second wave of
// clusters costs more than any range length saves.  (Measured per layer for
// every count at m = 1 .. 128 on the Llama and Qwen shapes: the largest
// one-wave count was the fastest or within 1 us of it; e.g. Llama down at
// m = 1, 16 tiles: 45.2 us unsplit, 16.9 us with 6 ranges, 26.7 us with 7,
// whose clusters no longer fit in one wave.)  Every range non-empty; at most
// kMaxSplits.  Returns the number of splits (1: none) and the stages per
// split.
int split_k_plan(const nvfp4::GemmParams &g, int num_sms, int *stages_per_split)
{
    const int num_ks = (g.num_k64 + 3) / 4;
    *stages_per_split = num_ks;
    if (g.m > 128 || num_sms <= 0) return 1;
    const int64_t tiles = g.num_n_blk;
    int best_s = 1;
    int64_t best_waves = (tiles + num_sms - 1) / num_sms;
    for (int s = 2; s <= nvfp4::kMaxSplits && s <= num_ks; ++s) {
        const int sps = (num_ks + s - 1) / s;
        if ((num_ks + sps - 1) / sps != s) continue;         // some range would be empty
        const int clusters = nvfp4::gemm_split_clusters(s, num_sms);
        if (clusters < 1) continue;
        const int64_t waves = (tiles + clusters - 1) / clusters;
        if (waves <= best_waves) {
            best_waves = waves;
            best_s = s;
        }
    }
    *stages_per_split = (num_ks + best_s - 1) / best_s;
    return best_s;
}

// Launches the GEMM; with allow_split and a small m it may split K (the
// linear entry points; nvfp4_gemm does not split).  after_quant: the
// kernel just before on `s` is the quantizer of `a` (and nothing else), so the
// GEMM may start as its programmatic dependent.
// GEMM kernel choice: the CTA-pair kernel (256 x 256 tiles, half of B per SM)
// for m > 128, the one-CTA kernel (which can split K) otherwise.  Both compute
// the same result; nvfp4_gemm_ex lets a test pick either.
enum GemmKernel { kGemmAuto = 0, kGemmOneCta = 1, kGemmPair = 2, kGemmOneCtaSplit = 3 };

// nvfp4_linear's fused path (the GEMM quantizes x itself) for m up to this.
constexpr int64_t kFusedLinearMaxRows = 16;

nvfp4_status run_gemm(const uint8_t *a, const uint8_t *a_sf, int64_t m, const uint8_t *w, const uint8_t *w_sf,
                      int64_t n_w, int64_t n_out, int64_t k, const float *alpha, const void *bias, void *out,
                      int64_t ldo, int num_sms, cudaStream_t s, bool allow_split = false,
                      bool after_quant = false, int kernel = kGemmAuto, uint64_t wait_ns = 0, int drill = 0,
                      bool mx = false, const nvfp4::QuantParams *fuse_quant = nullptr)
{
    unsigned int *err = nullptr;
    cudaError_t e = nvfp4::device_error_word(&err);
    if (e != cudaSuccess) return launch_status(e, "GEMM (error word)");
    nvfp4::GemmParams g = gemm_params(a_sf, m, w_sf, n_w, n_out, k, alpha, bias, out, ldo, err, mx);
    if (wait_ns != 0) g.wait_ns = wait_ns;
    g.drill = drill;
    if (allow_split && !(kernel == kGemmPair || (kernel == kGemmAuto && m > 128))) {
        int sps = 0;
        const int splits = split_k_plan(g, num_sms, &sps);
        if (splits > 1) {
            g.splits = splits;
            g.stages_per_split = sps;
        }
    }
    const char *why = nullptr;
    const bool pair = kernel == kGemmPair || (kernel == kGemmAuto && m > 128);
    if (fuse_quant != nullptr) {                     // the fused small-m linear: quantizer inside the GEMM
        g.quant = *fuse_quant;
        e = nvfp4::launch_linear_fused(g, w, num_sms, s, &why);
    } else {
        e = pair ? nvfp4::launch_gemm_pair(g, a, w, num_sms, s, &why, after_quant)
                 : nvfp4::launch_gemm(g, a, w, num_sms, s, &why, after_quant);
    }
    if (why) return fail(NVFP4_ERR_CUDA, "%s", why);
    return launch_status(e, fuse_quant ? "fused linear kernel" : "GEMM kernel");
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

// Smallest workspace of nvfp4_mxfp4_linear: the MXFP4 activation and its scales.
static size_t mx_min_workspace_bytes(int64_t m, int64_t k)
{
    if (m <= 0 || k <= 0) return 0;
    return align256(nvfp4_packed_bytes(m, k)) + align256(nvfp4_mxfp4_scale_bytes(m, k));
}

size_t nvfp4::linear_min_workspace_bytes(int64_t m, int64_t k)
{
    if (m <= 0 || k <= 0) return 0;
    return align256(nvfp4_packed_bytes(m, k)) + align256(nvfp4_scale_bytes(m, k));
}

int nvfp4::record_error(int st, const char *msg)
{
    g_last_error = msg;
    return st;
}

extern "C" {

int nvfp4_abi_version(void) { return NVFP4_ABI_VERSION; }

const char *nvfp4_last_error_string(void) { return g_last_error.c_str(); }

nvfp4_status nvfp4_is_supported(int device, char *reason, size_t reason_len)
{
    const DeviceInfo *d = device_info(device);
    nvfp4_status st = NVFP4_OK;
    const char *why = "";
    if (d == nullptr) {
        st = NVFP4_ERR_CUDA;
        why = "device index out of range";
    } else if (!d->probed) {
        st = NVFP4_ERR_CUDA;
        why = d->reason;
    } else if (!d->supported) {
        st = NVFP4_ERR_UNSUPPORTED_DEVICE;
        why = d->reason;
    }
    if (reason && reason_len) {
        strncpy(reason, why, reason_len - 1);
        reason[reason_len - 1] = 0;
    }
    return st == NVFP4_OK ? ok() : fail(st, "%s", why);
}

nvfp4_status nvfp4_device_error(int clear)
{
    unsigned int *ptr = nullptr;
    cudaError_t e = nvfp4::device_error_word(&ptr);
    unsigned int word = 0;
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&word, ptr, sizeof word, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && clear) e = cudaMemset(ptr, 0, sizeof word);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(NVFP4_ERR_CUDA, "reading the device error word failed: %s", cudaGetErrorString(e));
    }
    if (word & nvfp4::kErrTimeout)
        return fail(NVFP4_ERR_TIMEOUT, "a kernel abandoned a pipeline wait (error word 0x%x)", word);
    return ok();
}

size_t nvfp4_packed_bytes(int64_t rows, int64_t k)
{
    if (rows <= 0 || k <= 0) return 0;
    return (size_t)rows * (size_t)(nvfp4::padded_k(k) / 2);
}

size_t nvfp4_scale_bytes(int64_t rows, int64_t k)
{
    if (rows <= 0 || k <= 0) return 0;
    return (size_t)nvfp4::rows_padded(rows) * (size_t)nvfp4::scale_cols_padded(k);
}

size_t nvfp4_mxfp4_scale_bytes(int64_t rows, int64_t k)
{
    if (rows <= 0 || k <= 0) return 0;
    return (size_t)nvfp4::rows_padded(rows) * (size_t)((nvfp4::padded_k(k) / 32 + 3) / 4 * 4);
}

size_t nvfp4_linear_workspace_bytes(int64_t m, int64_t k, int64_t n_w)
{
    (void)n_w;
    if (m <= 0 || k <= 0) return 0;
    return nvfp4::linear_min_workspace_bytes(m, k);
}

nvfp4_status nvfp4_quant_act(const void *x_bf16, int64_t m, int64_t k, int64_t ldx, const float *gs_dev,
                             const void *transform_bf16, int bs, uint8_t *x_fp4, uint8_t *x_sf, nvfp4_stream_t stream)
{
    nvfp4_status st = check_quant_args(x_bf16, m, k, ldx, gs_dev, transform_bf16, bs, x_fp4, x_sf, "x");
    if (st != NVFP4_OK) return st;
    if (m == 0) return ok();
    Range outs[2] = {range(x_fp4, nvfp4_packed_bytes(m, k), "x_fp4"), range(x_sf, nvfp4_scale_bytes(m, k), "x_sf")};
    Range ins[3] = {range2d(x_bf16, m, k, ldx, "x"), range(gs_dev, 4, "gs"),
                    range(transform_bf16, transform_bf16 ? (size_t)bs * bs * 2 : 0, "transform")};
    if ((st = check_aliases(outs, 2, ins, 3)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    return run_quant(quant_params(x_bf16, m, k, ldx, gs_dev, transform_bf16, bs, x_fp4, x_sf), num_sms,
                     reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_quant_act_export_y(const void *x_bf16, int64_t m, int64_t k, int64_t ldx, const float *gs_dev,
                                      const void *transform_bf16, int bs, uint8_t *x_fp4, uint8_t *x_sf, void *y_bf16,
                                      nvfp4_stream_t stream)
{
    nvfp4_status st = check_quant_args(x_bf16, m, k, ldx, gs_dev, transform_bf16, bs, x_fp4, x_sf, "x");
    if (st != NVFP4_OK) return st;
    if (transform_bf16 == nullptr) return fail(NVFP4_ERR_INVALID_ARG, "y export needs a transform");
    if (m == 0) return ok();
    if (y_bf16 == nullptr) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    if (!aligned16(y_bf16)) return fail(NVFP4_ERR_ALIGNMENT, "y must be 16-byte aligned");
    Range outs[3] = {range(x_fp4, nvfp4_packed_bytes(m, k), "x_fp4"), range(x_sf, nvfp4_scale_bytes(m, k), "x_sf"),
                     range(y_bf16, (size_t)m * (size_t)k * 2, "y")};
    Range ins[3] = {range2d(x_bf16, m, k, ldx, "x"), range(gs_dev, 4, "gs"),
                    range(transform_bf16, (size_t)bs * bs * 2, "transform")};
    if ((st = check_aliases(outs, 3, ins, 3)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    nvfp4::QuantParams p = quant_params(x_bf16, m, k, ldx, gs_dev, transform_bf16, bs, x_fp4, x_sf);
    p.y_out = static_cast<uint16_t *>(y_bf16);
    return run_quant(p, num_sms, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_mxfp4_quant_act(const void *x_bf16, int64_t m, int64_t k, int64_t ldx, uint8_t *x_fp4, uint8_t *x_sf,
                                   nvfp4_stream_t stream)
{
    // MXFP4 has no global scale: x_sf stands in for check_quant_args' scale pointer
    nvfp4_status st = check_quant_args(x_bf16, m, k, ldx, reinterpret_cast<const float *>(x_sf), nullptr, 0, x_fp4,
                                       x_sf, "x");
    if (st != NVFP4_OK) return st;
    if (m == 0) return ok();
    Range outs[2] = {range(x_fp4, nvfp4_packed_bytes(m, k), "x_fp4"), range(x_sf, nvfp4_mxfp4_scale_bytes(m, k), "x_sf")};
    Range ins[1] = {range2d(x_bf16, m, k, ldx, "x")};
    if ((st = check_aliases(outs, 2, ins, 1)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    nvfp4::QuantParams p = quant_params(x_bf16, m, k, ldx, nullptr, nullptr, 0, x_fp4, x_sf);
    p.nb = (int32_t)(nvfp4::padded_k(k) / 32);
    p.nbp = (p.nb + 3) / 4 * 4;
    return launch_status(nvfp4::launch_quant_mx(p, num_sms, reinterpret_cast<cudaStream_t>(stream)),
                         "MXFP4 quantize kernel");
}

nvfp4_status nvfp4_act_global_scale(const void *x_bf16, int64_t m, int64_t k, int64_t ldx, const void *transform_bf16,
                                    int bs, const float *w_gs_dev, float *gs_out, float *alpha_out, nvfp4_stream_t stream)
{
    // the quantizer's checks, with gs_out standing in for the (absent) outputs' alignment
    if (!gs_out) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    if ((alpha_out != nullptr) != (w_gs_dev != nullptr))
        return fail(NVFP4_ERR_INVALID_ARG, "alpha_out and w_gs_dev go together");
    if ((reinterpret_cast<uintptr_t>(gs_out) & 3) || (reinterpret_cast<uintptr_t>(alpha_out) & 3) ||
        (reinterpret_cast<uintptr_t>(w_gs_dev) & 3))
        return fail(NVFP4_ERR_ALIGNMENT, "scalars must be 4-byte aligned");
    const uint8_t *dummy = reinterpret_cast<const uint8_t *>(16);
    nvfp4_status st = check_quant_args(m > 0 ? x_bf16 : nullptr, m, k, ldx, gs_out, transform_bf16, bs, dummy, dummy,
                                       "x");
    if (st != NVFP4_OK) return st;
    Range outs[2] = {range(gs_out, 4, "gs_out"), range(alpha_out, alpha_out ? 4 : 0, "alpha_out")};
    Range ins[3] = {range2d(m > 0 ? x_bf16 : nullptr, m, k, ldx, "x"), range(w_gs_dev, w_gs_dev ? 4 : 0, "w_gs"),
                    range(transform_bf16, transform_bf16 ? (size_t)bs * bs * 2 : 0, "transform")};
    if ((st = check_aliases(outs, 2, ins, 3)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    nvfp4::QuantParams p = quant_params(x_bf16, m, k, ldx, nullptr, transform_bf16, bs, nullptr, nullptr);
    cudaError_t e = nvfp4::device_error_word(&p.err_flag);
    if (e != cudaSuccess) return launch_status(e, "global-scale pass (error word)");
    const char *why = nullptr;
    e = nvfp4::launch_act_global_scale(p, w_gs_dev, gs_out, alpha_out, num_sms, reinterpret_cast<cudaStream_t>(stream),
                                       &why);
    if (why) return fail(NVFP4_ERR_CUDA, "%s", why);
    return launch_status(e, "global-scale pass");
}

nvfp4_status nvfp4_prepare_weight(const void *w_bf16, int64_t n, int64_t k, int64_t ldw, const float *w_gs_dev,
                                  uint8_t *w_fp4, uint8_t *w_sf, nvfp4_stream_t stream)
{
    nvfp4_status st = check_quant_args(w_bf16, n, k, ldw, w_gs_dev, nullptr, 0, w_fp4, w_sf, "w");
    if (st != NVFP4_OK) return st;
    if (n == 0) return ok();
    Range outs[2] = {range(w_fp4, nvfp4_packed_bytes(n, k), "w_fp4"), range(w_sf, nvfp4_scale_bytes(n, k), "w_sf")};
    Range ins[2] = {range2d(w_bf16, n, k, ldw, "w"), range(w_gs_dev, 4, "w_gs")};
    if ((st = check_aliases(outs, 2, ins, 2)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    return run_quant(quant_params(w_bf16, n, k, ldw, w_gs_dev, nullptr, 0, w_fp4, w_sf), num_sms,
                     reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_gemm_ex(const uint8_t *a_fp4, const uint8_t *a_sf, int64_t m, const uint8_t *w_fp4,
                           const uint8_t *w_sf, int64_t n_w, int64_t n_out, int64_t k, const float *alpha_dev,
                           const void *bias_bf16, void *out_bf16, int64_t ldo, int kernel, uint64_t wait_limit_ns,
                           int drill, nvfp4_stream_t stream)
{
    if (kernel < kGemmAuto || kernel > kGemmOneCtaSplit)
        return fail(NVFP4_ERR_INVALID_ARG,
                    "kernel must be 0 (automatic), 1 (one CTA), 2 (CTA pair) or 3 (one CTA, split K), got %d", kernel);
    if (kernel == kGemmPair && m > 0 && m <= 128)
        return fail(NVFP4_ERR_INVALID_ARG, "the CTA-pair kernel needs m > 128 (got %lld)", (long long)m);
    if (wait_limit_ns != 0 && (wait_limit_ns < 1000000ull || wait_limit_ns > 10000000000ull))
        return fail(NVFP4_ERR_INVALID_ARG, "wait_limit_ns must be 0 or within [1e6, 1e10] (got %llu)",
                    (unsigned long long)wait_limit_ns);
    if (drill != 0 && drill != 1) return fail(NVFP4_ERR_INVALID_ARG, "drill must be 0 or 1 (got %d)", drill);
    nvfp4_status st = check_gemm_args(m > 0 ? a_fp4 : nullptr, m > 0 ? a_sf : nullptr, m, w_fp4, w_sf, n_w, n_out, k,
                                      alpha_dev, bias_bf16, out_bf16, ldo);
    if (st != NVFP4_OK) return st;
    if (m == 0) return ok();
    if (!a_fp4 || !a_sf || !alpha_dev) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    Range outs[1] = {range2d(out_bf16, m, n_out, ldo, "out")};
    Range ins[6] = {range(a_fp4, nvfp4_packed_bytes(m, k), "a_fp4"), range(a_sf, nvfp4_scale_bytes(m, k), "a_sf"),
                    range(w_fp4, nvfp4_packed_bytes(n_w, k), "w_fp4"), range(w_sf, nvfp4_scale_bytes(n_w, k), "w_sf"),
                    range(alpha_dev, 4, "alpha"), range(bias_bf16, bias_bf16 ? (size_t)n_out * 2 : 0, "bias")};
    if ((st = check_aliases(outs, 1, ins, 6)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    // kernel 3: the one-CTA kernel with the linear's split-K plan (test hook)
    const bool split = kernel == kGemmOneCtaSplit;
    return run_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, alpha_dev, bias_bf16, out_bf16, ldo, num_sms,
                    reinterpret_cast<cudaStream_t>(stream), split, false, split ? (int)kGemmOneCta : kernel,
                    wait_limit_ns, drill);
}

nvfp4_status nvfp4_gemm(const uint8_t *a_fp4, const uint8_t *a_sf, int64_t m, const uint8_t *w_fp4,
                        const uint8_t *w_sf, int64_t n_w, int64_t n_out, int64_t k, const float *alpha_dev,
                        const void *bias_bf16, void *out_bf16, int64_t ldo, nvfp4_stream_t stream)
{
    return nvfp4_gemm_ex(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, alpha_dev, bias_bf16, out_bf16, ldo, kGemmAuto,
                         0, 0, stream);
}

nvfp4_status nvfp4_linear(const void *x_bf16, int64_t m, int64_t k, int64_t ldx, const float *gs_dev,
                          const void *transform_bf16, int bs, const uint8_t *w_fp4, const uint8_t *w_sf, int64_t n_w,
                          int64_t n_out, const float *alpha_dev, const void *bias_bf16, void *out_bf16, int64_t ldo,
                          void *workspace, size_t workspace_bytes, nvfp4_stream_t stream)
{
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t need = nvfp4::linear_min_workspace_bytes(m, k);   // quantized activation + scales
    uint8_t *a_fp4 = ws;
    uint8_t *a_sf = ws ? ws + align256(nvfp4_packed_bytes(m, k)) : nullptr;
    nvfp4_status st = check_quant_args(x_bf16, m, k, ldx, gs_dev, transform_bf16, bs, m > 0 ? a_fp4 : nullptr,
                                       m > 0 ? a_sf : nullptr, "x");
    if (st == NVFP4_ERR_INVALID_ARG && m > 0 && workspace == nullptr)
        return fail(NVFP4_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", need);
    if (st != NVFP4_OK) return st;
    st = check_gemm_args(nullptr, nullptr, m, w_fp4, w_sf, n_w, n_out, k, alpha_dev, bias_bf16, out_bf16, ldo);
    if (st != NVFP4_OK) return st;
    if (m == 0) return ok();
    if (!alpha_dev) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    if (workspace_bytes < need)
        return fail(NVFP4_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
    Range outs[2] = {range2d(out_bf16, m, n_out, ldo, "out"), range(workspace, workspace_bytes, "workspace")};
    Range ins[7] = {range2d(x_bf16, m, k, ldx, "x"), range(gs_dev, 4, "gs"),
                    range(transform_bf16, transform_bf16 ? (size_t)bs * bs * 2 : 0, "transform"),
                    range(w_fp4, nvfp4_packed_bytes(n_w, k), "w_fp4"), range(w_sf, nvfp4_scale_bytes(n_w, k), "w_sf"),
                    range(alpha_dev, 4, "alpha"), range(bias_bf16, bias_bf16 ? (size_t)n_out * 2 : 0, "bias")};
    if ((st = check_aliases(outs, 2, ins, 7)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const nvfp4::QuantParams qp = quant_params(x_bf16, m, k, ldx, gs_dev, transform_bf16, bs, a_fp4, a_sf);
    // Decode sizes: the GEMM quantizes its own activation (its eight epilogue
    // warps, each K stage as its slice lands, one 16-element block per lane).
    if (m <= kFusedLinearMaxRows && transform_bf16 == nullptr)
        return run_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, alpha_dev, bias_bf16, out_bf16, ldo, num_sms,
                        s, true, false, kGemmAuto, 0, 0, false, &qp);
    st = run_quant(qp, num_sms, s);
    if (st != NVFP4_OK) return st;
    return run_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, alpha_dev, bias_bf16, out_bf16, ldo, num_sms, s,
                    true, true);
}

size_t nvfp4_mxfp4_linear_workspace_bytes(int64_t m, int64_t k, int64_t n_w)
{
    (void)n_w;
    if (m <= 0 || k <= 0) return 0;
    return mx_min_workspace_bytes(m, k);
}

nvfp4_status nvfp4_mxfp4_gemm(const uint8_t *a_fp4, const uint8_t *a_sf, int64_t m, const uint8_t *w_fp4,
                              const uint8_t *w_sf, int64_t n_w, int64_t n_out, int64_t k, const void *bias_bf16,
                              void *out_bf16, int64_t ldo, nvfp4_stream_t stream)
{
    nvfp4_status st = check_gemm_args(m > 0 ? a_fp4 : nullptr, m > 0 ? a_sf : nullptr, m, w_fp4, w_sf, n_w, n_out, k,
                                      nullptr, bias_bf16, out_bf16, ldo);
    if (st != NVFP4_OK) return st;
    if (m == 0) return ok();
    if (!a_fp4 || !a_sf) return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    Range outs[1] = {range2d(out_bf16, m, n_out, ldo, "out")};
    Range ins[5] = {range(a_fp4, nvfp4_packed_bytes(m, k), "a_fp4"), range(a_sf, nvfp4_mxfp4_scale_bytes(m, k), "a_sf"),
                    range(w_fp4, nvfp4_packed_bytes(n_w, k), "w_fp4"),
                    range(w_sf, nvfp4_mxfp4_scale_bytes(n_w, k), "w_sf"),
                    range(bias_bf16, bias_bf16 ? (size_t)n_out * 2 : 0, "bias")};
    if ((st = check_aliases(outs, 1, ins, 5)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    return run_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, nullptr, bias_bf16, out_bf16, ldo, num_sms,
                    reinterpret_cast<cudaStream_t>(stream), false, false, kGemmAuto, 0, 0, true);
}

nvfp4_status nvfp4_mxfp4_linear(const void *x_bf16, int64_t m, int64_t k, int64_t ldx, const uint8_t *w_fp4,
                                const uint8_t *w_sf, int64_t n_w, int64_t n_out, const void *bias_bf16,
                                void *out_bf16, int64_t ldo, void *workspace, size_t workspace_bytes,
                                nvfp4_stream_t stream)
{
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t need = mx_min_workspace_bytes(m, k);           // MXFP4 activation + scales
    uint8_t *a_fp4 = ws;
    uint8_t *a_sf = ws ? ws + align256(nvfp4_packed_bytes(m, k)) : nullptr;
    // the quantizer's checks, with a_sf standing in for the (absent) global scale
    nvfp4_status st = check_quant_args(x_bf16, m, k, ldx, reinterpret_cast<const float *>(a_sf), nullptr, 0,
                                       m > 0 ? a_fp4 : nullptr, m > 0 ? a_sf : nullptr, "x");
    if (st == NVFP4_ERR_INVALID_ARG && m > 0 && workspace == nullptr)
        return fail(NVFP4_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", need);
    if (st != NVFP4_OK) return st;
    st = check_gemm_args(nullptr, nullptr, m, w_fp4, w_sf, n_w, n_out, k, nullptr, bias_bf16, out_bf16, ldo);
    if (st != NVFP4_OK) return st;
    if (m == 0) return ok();
    if (workspace_bytes < need)
        return fail(NVFP4_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
    Range outs[2] = {range2d(out_bf16, m, n_out, ldo, "out"), range(workspace, workspace_bytes, "workspace")};
    Range ins[4] = {range2d(x_bf16, m, k, ldx, "x"), range(w_fp4, nvfp4_packed_bytes(n_w, k), "w_fp4"),
                    range(w_sf, nvfp4_mxfp4_scale_bytes(n_w, k), "w_sf"),
                    range(bias_bf16, bias_bf16 ? (size_t)n_out * 2 : 0, "bias")};
    if ((st = check_aliases(outs, 2, ins, 4)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    nvfp4::QuantParams p = quant_params(x_bf16, m, k, ldx, nullptr, nullptr, 0, a_fp4, a_sf);
    p.nb = (int32_t)(nvfp4::padded_k(k) / 32);
    p.nbp = (p.nb + 3) / 4 * 4;
    // decode sizes: the GEMM quantizes its own activation, as nvfp4_linear's fused path
    if (m <= kFusedLinearMaxRows)
        return run_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, nullptr, bias_bf16, out_bf16, ldo, num_sms, s,
                        true, false, kGemmAuto, 0, 0, true, &p);
    st = launch_status(nvfp4::launch_quant_mx(p, num_sms, s), "MXFP4 quantize kernel");
    if (st != NVFP4_OK) return st;
    return run_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, nullptr, bias_bf16, out_bf16, ldo, num_sms, s,
                    true, true, kGemmAuto, 0, 0, true);
}

nvfp4_status nvfp4_grouped_gemm(const uint8_t *a_fp4, const uint8_t *a_sf, int64_t rows,
                                const int32_t *group_offsets_dev, int num_groups, const uint8_t *w_fp4,
                                const uint8_t *w_sf, int64_t n, int64_t k, const float *alpha_dev,
                                const void *bias_bf16, void *out_bf16, int64_t ldo, nvfp4_stream_t stream)
{
    if (num_groups < 1 || num_groups > (1 << 16))
        return fail(NVFP4_ERR_INVALID_ARG, "num_groups must be in [1, 65536] (got %d)", num_groups);
    if (n < 128 || n % 128 != 0 || n * (int64_t)num_groups > kMaxDim)
        return fail(NVFP4_ERR_INVALID_ARG, "n must be a positive multiple of 128 with num_groups * n < 2^31 (got %lld)",
                    (long long)n);
    nvfp4_status st = check_gemm_args(rows > 0 ? a_fp4 : nullptr, rows > 0 ? a_sf : nullptr, rows, w_fp4, w_sf,
                                      n * num_groups, n, k, alpha_dev, bias_bf16, out_bf16, ldo);
    if (st != NVFP4_OK) return st;
    if (rows == 0) return ok();
    if (!a_fp4 || !a_sf || !alpha_dev || !group_offsets_dev)
        return fail(NVFP4_ERR_INVALID_ARG, "null pointer argument");
    if ((reinterpret_cast<uintptr_t>(group_offsets_dev) & 3) || (reinterpret_cast<uintptr_t>(alpha_dev) & 3))
        return fail(NVFP4_ERR_ALIGNMENT, "group offsets and alphas must be 4-byte aligned");
    const int64_t wrows = n * num_groups;
    Range outs[1] = {range2d(out_bf16, rows, n, ldo, "out")};
    Range ins[7] = {range(a_fp4, nvfp4_packed_bytes(rows, k), "a_fp4"), range(a_sf, nvfp4_scale_bytes(rows, k), "a_sf"),
                    range(w_fp4, nvfp4_packed_bytes(wrows, k), "w_fp4"),
                    range(w_sf, nvfp4_scale_bytes(wrows, k), "w_sf"),
                    range(alpha_dev, (size_t)num_groups * 4, "alpha"),
                    range(bias_bf16, bias_bf16 ? (size_t)wrows * 2 : 0, "bias"),
                    range(group_offsets_dev, (size_t)(num_groups + 1) * 4, "group_offsets")};
    if ((st = check_aliases(outs, 1, ins, 7)) != NVFP4_OK) return st;
    int num_sms = 0;
    if ((st = current_device(&num_sms)) != NVFP4_OK) return st;
    unsigned int *err = nullptr;
    cudaError_t e = nvfp4::device_error_word(&err);
    if (e != cudaSuccess) return launch_status(e, "grouped GEMM (error word)");
    nvfp4::GemmParams g = gemm_params(a_sf, rows, w_sf, wrows, n, k, alpha_dev, bias_bf16, out_bf16, ldo, err);
    g.group_offsets = group_offsets_dev;
    g.num_groups = num_groups;
    g.group_n = (int32_t)n;
    const char *why = nullptr;
    e = nvfp4::launch_gemm(g, a_fp4, w_fp4, num_sms, reinterpret_cast<cudaStream_t>(stream), &why, false);
    if (why) return fail(NVFP4_ERR_CUDA, "%s", why);
    return launch_status(e, "grouped GEMM kernel");
}

}  // extern "C"
