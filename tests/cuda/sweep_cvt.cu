// Exhaustive probe of the hardware encoders the quantizers use -- cvt with
// .rn.satfinite to E2M1 (through cvt_e2m1x8) and to E4M3 (through cvt_e4m3x2),
// both from nvfp4_quantized_linear_gb300/csrc/ptx.cuh -- against the CPU
// oracle's encoders: every finite float for E2M1 (both signs), every finite
// non-negative float for E4M3 (block scales are never negative).  The GPU
// writes the codes; host threads compare them with the oracle's functions,
// loaded from the oracle's shared library.  Built and run by
// tests/test_gpu_encoders.py.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <dlfcn.h>
#include <thread>
#include <vector>

#include <cuda_runtime.h>

#include "ptx.cuh"

namespace {

constexpr uint64_t kFinite = 0x7F800000ull;          // patterns [0, 0x7F800000): +0 .. largest finite

// byte p of e2m1: code of +float(p) in the low nibble, of -float(p) in the high one
__global__ void encode(uint8_t *e2m1, uint8_t *e4m3)
{
    for (uint64_t p = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; p < kFinite;
         p += (uint64_t)gridDim.x * blockDim.x) {
        const float pos = __uint_as_float((uint32_t)p);
        const float neg = __uint_as_float((uint32_t)p | 0x80000000u);
        const float v[8] = {pos, neg, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        e2m1[p] = (uint8_t)(nvfp4::cvt_e2m1x8(v) & 0xFFu);
        e4m3[p] = (uint8_t)(nvfp4::cvt_e4m3x2(0.0f, pos) & 0xFFu);
    }
}

}  // namespace

// counts[0]: E2M1 mismatches over both signs; counts[1]: E4M3 mismatches.
// first_bad[0..1]: the smallest pattern of each kind that differs (or ~0u).
// Returns 0, a cudaError_t value, or -1 if the oracle cannot be loaded.
extern "C" int run_sweep(const char *oracle_so, unsigned long long *counts, unsigned int *first_bad)
{
    void *h = dlopen(oracle_so, RTLD_NOW | RTLD_LOCAL);
    if (h == nullptr) return -1;
    auto enc_e2m1 = reinterpret_cast<uint8_t (*)(float)>(dlsym(h, "oracle_enc_e2m1"));
    auto enc_e4m3 = reinterpret_cast<uint8_t (*)(float)>(dlsym(h, "oracle_enc_e4m3"));
    if (enc_e2m1 == nullptr || enc_e4m3 == nullptr) return -1;

    uint8_t *d = nullptr;
    cudaError_t e = cudaMalloc(&d, 2 * kFinite);
    std::vector<uint8_t> e2m1, e4m3;
    if (e == cudaSuccess) {
        int sms = 0;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
        encode<<<sms * 8, 256>>>(d, d + kFinite);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) {
        e2m1.resize(kFinite);
        e4m3.resize(kFinite);
        e = cudaMemcpy(e2m1.data(), d, kFinite, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(e4m3.data(), d + kFinite, kFinite, cudaMemcpyDeviceToHost);
    }
    cudaFree(d);
    if (e != cudaSuccess) return (int)e;

    const unsigned nt = std::max(1u, std::thread::hardware_concurrency());
    std::vector<unsigned long long> c2(nt, 0), c4(nt, 0);
    std::vector<unsigned int> f2(nt, ~0u), f4(nt, ~0u);
    std::vector<std::thread> th;
    for (unsigned t = 0; t < nt; ++t)
        th.emplace_back([&, t] {
            const uint64_t lo = kFinite * t / nt, hi = kFinite * (t + 1) / nt;
            for (uint64_t p = lo; p < hi; ++p) {
                float pos, neg;
                const uint32_t pb = (uint32_t)p, nb = (uint32_t)p | 0x80000000u;
                memcpy(&pos, &pb, 4);
                memcpy(&neg, &nb, 4);
                const uint8_t want2 = (uint8_t)(enc_e2m1(pos) | (enc_e2m1(neg) << 4));
                if (e2m1[p] != want2) {
                    ++c2[t];
                    if (f2[t] == ~0u) f2[t] = (uint32_t)p;
                }
                if (e4m3[p] != enc_e4m3(pos)) {
                    ++c4[t];
                    if (f4[t] == ~0u) f4[t] = (uint32_t)p;
                }
            }
        });
    for (auto &x : th) x.join();
    counts[0] = counts[1] = 0;
    first_bad[0] = first_bad[1] = ~0u;
    for (unsigned t = 0; t < nt; ++t) {
        counts[0] += c2[t];
        counts[1] += c4[t];
        first_bad[0] = std::min(first_bad[0], f2[t]);
        first_bad[1] = std::min(first_bad[1], f4[t]);
    }
    dlclose(h);
    return 0;
}
