// NVFP4 quantizer core shared by quant_kernel (quant.cu) and the fused
// small-m linear (gemm.cu): the per-block arithmetic and the grid-stride loop
// over 512-element row segments.  Page "TorchNvFp4LinearKernel" (vLLM PR
// #53319), section 关键源码片段: scaled_fp4_quant with the activation global
// scale, swizzled scales and K padded to the weight's padding.
//
// Per 16-element block (all fp32, round-to-nearest-even, IEEE division):
//   s = (amax * gs) / 6;  sf = e4m3(s);  inv = sf ? gs / e4m3(sf) : 0;
//   q_i = e2m1(v_i * inv)
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "scale_math.cuh"

namespace nvfp4 {
namespace quant_core {

constexpr unsigned kFull = 0xFFFFFFFFu;

// max(|a|, |b|, |c|): the three-input max.abs.f32 of sm_100 and later (one
// instruction where two two-input maxima with abs operands were needed).
__device__ __forceinline__ float max_abs3(float a, float b, float c)
{
    float d;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// MXFP4 scale code of a 32-element block with absolute maximum `amax`:
//     s = clamp(floor(log2 amax) - 2, -127, 127)  (-127 for a zero block),
//     code = s + 127 (UE8M0), and the elements are quantized as e2m1(v * 2^-s).
// floor(log2 amax) comes from the fp32 bits (exponent field, or the top set
// bit of a subnormal).
__device__ __forceinline__ uint32_t mx_scale_code(float amax)
{
    if (amax == 0.0f) return 0;
    const uint32_t u = __float_as_uint(amax);
    const int e = (int)(u >> 23);                       // amax >= 0: no sign bit
    const int fl = e != 0 ? e - 127 : -149 + (31 - __clz((int)u));
    const int s = min(max(fl - 2, -127), 127);
    return (uint32_t)(s + 127);
}

// 2^-s for a scale code (s = code - 127 <= 125 for finite input), built from bits.
__device__ __forceinline__ float mx_scale_mul(uint32_t code) { return __uint_as_float((254u - code) << 23); }

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

// Quantizes the tasks (512-element segments of the padded rows) that fall to
// warp `warp` of `nwarps`, U at a time: the body of quant_kernel.  inv_tab
// holds fill_inv_table(gs) and is visible to the calling thread.
template <int U>
__device__ __forceinline__ void quantize_rows(const QuantParams &p, const float *inv_tab, float gs, int warp,
                                              int nwarps, int lane)
{
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

}  // namespace quant_core
}  // namespace nvfp4
