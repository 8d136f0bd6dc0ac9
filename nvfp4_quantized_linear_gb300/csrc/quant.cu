// NVFP4 quantizer kernels: bf16 rows -> packed E2M1 + tiled E4M3 block scales.
//
// Page "TorchNvFp4LinearKernel" (vLLM PR #53319), section 关键源码片段:
// apply_weights calls scaled_fp4_quant(x, global_scale, swizzled layout,
// padded K); process_weights_after_loading needs the same packed/tiled form of
// the weight.  Page "QUTLASS fusedQuantizeNv" (vLLM PR #43229), 实现拆解 items
// 3 and 6: an optional block-diagonal transform (1/sqrt(n) folded into it,
// result in bf16) runs first, fused into the same kernel.
//
// Per 16-element block (all fp32, round-to-nearest-even, IEEE division):
//   s = (amax * gs) / 6;  sf = e4m3(s);  inv = sf ? gs / e4m3(sf) : 0;
//   q_i = e2m1(v_i * inv)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "scale_math.cuh"

namespace nvfp4 {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Scale code and element multiplier of a block with absolute maximum `amax`:
//   s = (amax * gs) / 6;  sf = e4m3(s);  inv = sf ? gs / e4m3(sf) : 0.
// The division by 6 is div6_rn (scale_math.cuh), which gives the same code sf
// as the IEEE quotient for every input.  gs / e4m3(code) comes from a table of
// the 128 non-negative codes (s >= 0, and satfinite never yields the NaN code)
// that each block fills once with the IEEE division (fill_inv_table).
__device__ __forceinline__ uint32_t block_scale_tab(float amax, float gs, const float *inv_tab, float &inv)
{
    const float s = div6_rn(__fmul_rn(amax, gs));
    const uint32_t sf = cvt_e4m3x2(0.0f, s) & 0x7Fu;
    inv = inv_tab[sf];
    return sf;
}

__device__ __forceinline__ void fill_inv_table(float *inv_tab, float gs)
{
    for (int c = threadIdx.x; c < 128; c += blockDim.x) {
        const float d = e4m3_to_f32((uint32_t)c);
        inv_tab[c] = (d == 0.0f) ? 0.0f : __fdiv_rn(gs, d);
    }
}

// q_i = e2m1(v_i * inv), the products two at a time (mul.rn.f32x2: each lane
// of the pair rounds like a scalar fp32 multiply).
__device__ __forceinline__ uint32_t quant8(const float (&v)[8], float inv)
{
    float q[8];
    uint64_t iv;
    asm("mov.b64 %0, {%1, %1};" : "=l"(iv) : "f"(inv));
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        uint64_t a, d;
        asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(v[i]), "f"(v[i + 1]));
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(iv));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(q[i]), "=f"(q[i + 1]) : "l"(d));
    }
    return cvt_e2m1x8(q);
}

// ---------------------------------------------------------------------------
// Plain quantizer.  A warp task is one 512-element segment of one row: lane l
// owns block l of the segment (elements [16l, 16l+16), two 16-byte loads), so
// the block maximum and the scale arithmetic are done once per block, in one
// lane.  Each lane stores its 8 packed bytes (the warp writes 256 contiguous
// bytes) and lanes 0, 4, 8, ... store the 4 scale bytes of 4 consecutive blocks
// as one word of a 512-byte scale tile.  Tasks run over the padded row count
// so the scale rows beyond m are zeroed (those rows store no packed data).  A
// warp loads the raw bytes of U consecutive tasks before processing any of
// them, to keep enough bytes in flight.
struct Raw16 {
    uint4 a, b;
};

__device__ __forceinline__ Raw16 load16(const uint16_t *row, int k0, int k, bool row_ok)
{
    Raw16 r;
    if (row_ok && k0 + 16 <= k) {
        r.a = ld_stream_v4(row + k0);
        r.b = ld_stream_v4(row + k0 + 8);
    } else {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = (row_ok && k0 + 2 * i < k) ? row[k0 + 2 * i] : 0u;
            const uint32_t hi = (row_ok && k0 + 2 * i + 1 < k) ? row[k0 + 2 * i + 1] : 0u;
            w[i] = lo | (hi << 16);
        }
        r.a = make_uint4(w[0], w[1], w[2], w[3]);
        r.b = make_uint4(w[4], w[5], w[6], w[7]);
    }
    return r;
}

__device__ __forceinline__ void unpack8(const uint4 &w, float (&v)[8])
{
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
    v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
    v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

template <int U>
__global__ void __launch_bounds__(256) quant_kernel(const QuantParams p)
{
    const int lane = threadIdx.x & 31;
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    // A programmatic dependent (the GEMM of the linear layer) may start its
    // prologue now; it waits for this grid before touching its data.
    if (threadIdx.x == 0) griddep_launch_dependents();
    __shared__ float inv_tab[128];
    const float gs = __ldg(p.gs);
    fill_inv_table(inv_tab, gs);
    __syncthreads();
    const int segs = (p.kp + 511) >> 9;
    const int tasks = p.mp * segs;                    // < 2^31: checked on the host
    const int64_t out_ld = p.kp >> 1;

    for (int base = warp * U; base < tasks; base += nwarps * U) {
        // (row, segment) of the first task; the next ones follow along the row
        int r0 = base / segs;
        int s0 = base - r0 * segs;
        Raw16 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            int r = r0, s = s0 + u;
            while (s >= segs) { s -= segs; ++r; }
            const bool row_ok = (base + u < tasks) && (r < p.m);
            raw[u] = load16(row_ok ? p.x + (int64_t)r * p.ldx : p.x, s * 512 + lane * 16, p.k, row_ok);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u >= tasks) break;                 // uniform across the warp
            int r = r0, s = s0 + u;
            while (s >= segs) { s -= segs; ++r; }
            const int k0 = s * 512 + lane * 16;
            float v0[8], v1[8];
            unpack8(raw[u].a, v0);
            unpack8(raw[u].b, v1);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(v0[i]), fabsf(v1[i])));
            float inv;
            const uint32_t sf = block_scale_tab(amax, gs, inv_tab, inv);
            if (r < p.m && k0 < p.kp) {
                uint2 pk;
                pk.x = quant8(v0, inv);
                pk.y = quant8(v1, inv);
                *reinterpret_cast<uint2 *>(p.out + (int64_t)r * out_ld + (k0 >> 1)) = pk;
            }
            const uint32_t s1 = __shfl_down_sync(kFull, sf, 1);
            const uint32_t s2 = __shfl_down_sync(kFull, sf, 2);
            const uint32_t s3 = __shfl_down_sync(kFull, sf, 3);
            const int c = s * 32 + lane;
            if ((lane & 3) == 0 && c < p.nb)
                *reinterpret_cast<uint32_t *>(p.sf + sf_offset(r, c, p.nbp)) = sf | (s1 << 8) | (s2 << 16) | (s3 << 24);
        }
    }
}

// ---------------------------------------------------------------------------
// Transform + quantizer.  A CTA tile is 32 rows x 256 columns.  The tile is
// staged in shared memory (row stride 129 words: conflict-free column reads),
// T is held in shared memory as fp32.  Thread (warp w, lane l) computes, for
// row l, the 16 outputs of units w and w+8 (a unit = 16 consecutive columns =
// one scale block): y_j = bf16(acc_j), acc_j an fp32 fused multiply-add chain
// over i = 0..bs-1 in index order, then quantizes the 16 values in-thread.
constexpr int kXRowWords = 129;

__global__ void __launch_bounds__(256) quant_transform_kernel(const QuantParams p)
{
    extern __shared__ float smem_f[];
    const int bs = p.bs;
    float *sT = smem_f;
    uint32_t *sX = reinterpret_cast<uint32_t *>(smem_f + bs * bs);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) griddep_launch_dependents();    // as in quant_kernel

    __shared__ float inv_tab[128];
    for (int i = tid; i < bs * bs; i += 256) sT[i] = __uint_as_float((uint32_t)p.t[i] << 16);
    const float gs = __ldg(p.gs);
    fill_inv_table(inv_tab, gs);                           // visible after the first tile's barrier
    const int segs = (p.kp + 255) >> 8;
    const int64_t tiles = (int64_t)(p.mp / 32) * segs;
    const int64_t out_ld = p.kp >> 1;

    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t r0 = (tile / segs) * 32;
        const int kseg = (int)(tile % segs) * 256;
        __syncthreads();                                   // previous tile fully consumed
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int idx = it * 256 + tid;
            const int rr = idx >> 5, ch = idx & 31;
            const int64_t r = r0 + rr;
            const int k = kseg + ch * 8;
            uint4 w = make_uint4(0, 0, 0, 0);
            if (r < p.m && k < p.k) w = ld_stream_v4(p.x + r * p.ldx + k);   // k % 16 == 0: whole chunk valid
            uint32_t *dst = sX + rr * kXRowWords + ch * 4;
            dst[0] = w.x; dst[1] = w.y; dst[2] = w.z; dst[3] = w.w;
        }
        __syncthreads();

        const int64_t r = r0 + lane;
#pragma unroll 1
        for (int uu = 0; uu < 2; ++uu) {
            const int u = warp + uu * 8;
            const int c0 = kseg + u * 16;
            if (c0 >= p.kp) continue;                      // uniform across the warp
            float acc[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
            if (c0 < p.k) {
                const int blk = (u * 16) / bs * bs;         // first column of the bs-block in this segment
                const int j0 = (u * 16) % bs;
                const uint32_t *xr = sX + lane * kXRowWords + (blk >> 1);
#pragma unroll 2
                for (int i = 0; i < bs; i += 2) {
                    const uint32_t xw = xr[i >> 1];
                    const float x0 = bf16_lo(xw), x1 = bf16_hi(xw);
                    const float4 *t0 = reinterpret_cast<const float4 *>(sT + i * bs + j0);
                    const float4 *t1 = reinterpret_cast<const float4 *>(sT + (i + 1) * bs + j0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 a = t0[q];
                        acc[4 * q + 0] = __fmaf_rn(x0, a.x, acc[4 * q + 0]);
                        acc[4 * q + 1] = __fmaf_rn(x0, a.y, acc[4 * q + 1]);
                        acc[4 * q + 2] = __fmaf_rn(x0, a.z, acc[4 * q + 2]);
                        acc[4 * q + 3] = __fmaf_rn(x0, a.w, acc[4 * q + 3]);
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 a = t1[q];
                        acc[4 * q + 0] = __fmaf_rn(x1, a.x, acc[4 * q + 0]);
                        acc[4 * q + 1] = __fmaf_rn(x1, a.y, acc[4 * q + 1]);
                        acc[4 * q + 2] = __fmaf_rn(x1, a.z, acc[4 * q + 2]);
                        acc[4 * q + 3] = __fmaf_rn(x1, a.w, acc[4 * q + 3]);
                    }
                }
            }
            float y0[8], y1[8];
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                y0[j] = __bfloat162float(__float2bfloat16_rn(acc[j]));
                y1[j] = __bfloat162float(__float2bfloat16_rn(acc[8 + j]));
                amax = fmaxf(amax, fmaxf(fabsf(y0[j]), fabsf(y1[j])));
            }
            float inv;
            const uint32_t sf = block_scale_tab(amax, gs, inv_tab, inv);
            if (r < p.m) {
                uint2 pk;
                pk.x = quant8(y0, inv);
                pk.y = quant8(y1, inv);
                *reinterpret_cast<uint2 *>(p.out + r * out_ld + (c0 >> 1)) = pk;
            }
            const int cb = c0 >> 4;
            p.sf[sf_offset(r, cb, p.nbp)] = (uint8_t)sf;
            if (cb == p.nb - 1)                             // zero the column padding of this row
                for (int c = p.nb; c < p.nbp; ++c) p.sf[sf_offset(r, c, p.nbp)] = 0;
        }
    }
}

}  // namespace

cudaError_t launch_quant(const QuantParams &p, int num_sms, cudaStream_t s)
{
    constexpr int U = 4;
    const int64_t segs = (p.kp + 511) / 512;
    const int64_t tasks = (int64_t)p.mp * segs;
    const int64_t warps_needed = (tasks + U - 1) / U;
    int64_t blocks = (warps_needed + 7) / 8;
    const int64_t cap = (int64_t)num_sms * 8;          // 8 x 256 threads fill an SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quant_kernel<U><<<(unsigned)blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_quant_transform(const QuantParams &p, int num_sms, cudaStream_t s)
{
    const size_t smem = (size_t)p.bs * p.bs * sizeof(float) + 32 * kXRowWords * sizeof(uint32_t);
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(quant_transform_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(128 * 128 * sizeof(float) + 32 * kXRowWords * sizeof(uint32_t)));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int64_t segs = (p.kp + 255) / 256;
    const int64_t tiles = (int64_t)(p.mp / 32) * segs;
    int64_t blocks = tiles;
    const int64_t cap = (int64_t)num_sms * 2;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quant_transform_kernel<<<(unsigned)blocks, 256, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace nvfp4
