// Quantizer kernels: bf16 rows -> packed E2M1 + tiled block scales.
//
// Page "TorchNvFp4LinearKernel" (vLLM PR #53319), section 关键源码片段:
// apply_weights calls scaled_fp4_quant(x, global_scale, swizzled layout,
// padded K); process_weights_after_loading needs the same packed/tiled form of
// the weight.  Page "QUTLASS fusedQuantizeNv" (vLLM PR #43229), 实现拆解 items
// 3 and 6: an optional block-diagonal transform (1/sqrt(n) folded into it,
// result in bf16) runs first, fused into the same kernel.
//
// Kernels in this file:
//   quant_kernel               NVFP4 (16-element blocks, E4M3 scales, global scale)
//   quant_mx_kernel            MXFP4 (32-element blocks, E8M0 scales; page "B12X"'s
//                              MXFP4 backend)
//   act_amax_kernel            per-tensor max |x| for the dynamic global scale
//   act_scale_finalize_kernel  gs = 448 * 6 / amax and alpha from that maximum
//   quant_transform_kernel     transform on the tensor cores (tcgen05 kind::f16)
//                              fused with the NVFP4 quantizer; its kAmaxOnly
//                              variant reduces max |y| for the dynamic scale
//
// Per 16-element block (all fp32, round-to-nearest-even, IEEE division):
//   s = (amax * gs) / 6;  sf = e4m3(s);  inv = sf ? gs / e4m3(sf) : 0;
//   q_i = e2m1(v_i * inv)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"
#include "quant_launch.cuh"
#include "quant_core.cuh"
#include "scale_math.cuh"

namespace nvfp4 {
namespace {

using namespace quant_core;

__device__ __forceinline__ uint64_t l2_policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}


template <int U>
__global__ void __launch_bounds__(256) quant_kernel(const QuantParams p)
{
    const int lane = threadIdx.x & 31;
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    // Launched as a programmatic dependent, this grid may start while the
    // kernel before it still runs: nothing is read or written before that
    // kernel has completed (gs or x may be its output, the outputs its input).
    // Only then may this grid's own dependent (the GEMM of the linear layer)
    // start: its weight side reads without waiting, and every kernel before
    // this one has completed by now.  The GEMM waits for this grid before it
    // reads the quantized activation.
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();
    __shared__ float inv_tab[128];
    const float gs = __ldg(p.gs);
    fill_inv_table(inv_tab, gs);
    __syncthreads();
    quantize_rows<U>(p, inv_tab, gs, warp, nwarps, lane);
}

// ---------------------------------------------------------------------------
// MXFP4 quantizer (OCP MX: 32-element blocks, E8M0 scale 2^s, no global
// scale).  The task split and loads of quant_kernel; a block is the 32
// elements of a lane pair, whose maxima meet through one shuffle:
//     s = clamp(floor(log2 amax) - 2, -127, 127)  (-127 for a zero block),
//     code = s + 127,  q_i = e2m1(fl32(v_i * 2^-s)).
// floor(log2 amax) comes from the fp32 bits (exponent field, or the top set
// bit of a subnormal); 2^-s is built from bits (s <= 125 for finite input).
// Lanes 0, 8, 16, 24 store the codes of four consecutive blocks as one word
// of a 512-byte scale tile (the tiled layout of the NVFP4 scales, one column
// per 32 elements); p.nb / p.nbp count these columns.  The scale code is
// quant_core::mx_scale_code.

template <int U>
__global__ void __launch_bounds__(256) quant_mx_kernel(const QuantParams p)
{
    const int lane = threadIdx.x & 31;
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    if (threadIdx.x == 0) griddep_launch_dependents();
    const int segs = (p.kp + 511) >> 9;
    const int tasks = p.mp * segs;                    // < 2^31: checked on the host
    const int64_t out_ld = p.kp >> 1;

    for (int base = warp * U; base < tasks; base += nwarps * U) {
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
            amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
            const uint32_t code = quant_core::mx_scale_code(amax);
            const float mul = quant_core::mx_scale_mul(code);          // 2^-s
            if (r < p.m && k0 < p.kp) {
                uint2 pk;
                pk.x = quant8(v0, mul);
                pk.y = quant8(v1, mul);
                *reinterpret_cast<uint2 *>(p.out + (int64_t)r * out_ld + (k0 >> 1)) = pk;
            }
            const uint32_t c1 = __shfl_down_sync(kFull, code, 2);
            const uint32_t c2 = __shfl_down_sync(kFull, code, 4);
            const uint32_t c3 = __shfl_down_sync(kFull, code, 6);
            const int c = s * 16 + (lane >> 1);
            if ((lane & 7) == 0 && c < p.nb)
                *reinterpret_cast<uint32_t *>(p.sf + sf_offset(r, c, p.nbp)) = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
        }
    }
}

// ---------------------------------------------------------------------------
// Per-tensor amax of the activation (no transform): the task split of
// quant_kernel (512-element row segments, U per warp loaded before use), an
// integer max over the bf16 magnitudes (the bits without the sign order like
// the values), one atomic max per warp.  Loads keep the default L2 policy so
// that a tensor smaller than L2 is still there for the quantizer.
template <int U>
__global__ void __launch_bounds__(256) act_amax_kernel(const QuantParams p, unsigned int *amax_out)
{
    const int lane = threadIdx.x & 31;
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int nwarps = (int)((gridDim.x * blockDim.x) >> 5);
    const int segs = (p.k + 511) >> 9;
    const int tasks = p.m * segs;                     // < 2^31: checked on the host
    uint32_t mx = 0;                                  // two 16-bit maxima
    for (int base = warp * U; base < tasks; base += nwarps * U) {
        Raw16 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int t = base + u;
            const int r = t / segs;
            const bool ok = t < tasks;
            raw[u] = load16(ok ? p.x + (int64_t)r * p.ldx : p.x, (t - r * segs) * 512 + lane * 16, p.k, ok);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t w[8] = {raw[u].a.x, raw[u].a.y, raw[u].a.z, raw[u].a.w,
                                   raw[u].b.x, raw[u].b.y, raw[u].b.z, raw[u].b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) mx = __vmaxu2(mx, w[i] & 0x7FFF7FFFu);
        }
    }
    const uint32_t v = __reduce_max_sync(~0u, max(mx & 0xFFFFu, mx >> 16));
    if (lane == 0 && v != 0) atomicMax(amax_out, v);
}

// gs = fl32(448 * 6 / amax) from the bf16 bits left in *word by the amax
// pass, written over it; FLT_MAX if the quotient overflows, 1 for amax == 0.
// With w_gs: alpha = fl32(1 / fl32(gs * w_gs)).
__global__ void act_scale_finalize_kernel(unsigned int *word, const float *w_gs, float *alpha)
{
    const float amax = __uint_as_float(*word << 16);
    float gs = 1.0f;
    if (amax > 0.0f) {
        gs = __fdiv_rn(2688.0f, amax);
        if (isinf(gs)) gs = 3.402823466e38f;
    }
    *reinterpret_cast<float *>(word) = gs;
    if (alpha != nullptr) *alpha = __fdiv_rn(1.0f, __fmul_rn(gs, *w_gs));
}

// ---------------------------------------------------------------------------
// Transform + quantizer on the tensor cores.  y = x * blockdiag(T) is a dense
// contraction per bs-block, so each 128-row x 128-column tile of x goes
// through tcgen05.mma (kind::f16: bf16 operands, fp32 accumulation in TMEM):
// for every bs-block g of the tile, bs/16 MMAs of M = 128, N = bs, K = 16 give
//     D[:, g*bs : (g+1)*bs] = X[:, g*bs : (g+1)*bs] * T,
// always 8 MMAs per tile.  The bf16 x bf16 products are exact in fp32; the
// sum is accumulated in fp32 by the tensor core and rounded to bf16 once, in
// the epilogue, which then quantizes y exactly as the plain quantizer does.
//
// One CTA per SM, persistent over the tiles (column tiles of a 128-row band
// consecutive):
//   warp 0      lane 0: TMA loads of the x tile (two boxes of 64 columns x
//               128 rows, 128-byte swizzle, zero fill past m and k) into a
//               4-stage ring;
//   warp 1      allocates the 256 TMEM columns (two 128-column accumulators);
//               an elected lane issues each tile's MMAs and commits;
//   warps 2..9  epilogue, two per TMEM lane quarter (64 columns each): read
//               the accumulator, hand it back, round to bf16, block scale,
//               E2M1 codes, stores (packed rows < m, scale rows < mp; and y
//               itself when the caller asks for it).
// T^T is the B operand: row n holds column n of T, in the same swizzled
// K-major form; K-chunk c (rows 64c .. 64c+63 of T) at byte c * bs * 128.
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel raises the
// device error word and exits.
constexpr int kXfRows = 128;                               // tile rows = MMA M
constexpr int kXfCols = 128;                               // tile columns
constexpr int kXfStages = 4;
constexpr uint32_t kXfBoxBytes = 128 * 128;                // 128 rows x 64 bf16
constexpr uint32_t kXfStageBytes = 2 * kXfBoxBytes;
constexpr uint32_t kXfOffT = kXfStages * kXfStageBytes;    // T^T: up to 2 K-chunks of 128 rows
constexpr uint32_t kXfOffBar = kXfOffT + 2 * kXfBoxBytes;
constexpr uint32_t kXfSmemBytes = kXfOffBar + 256 + 1024;  // barriers + alignment slack
constexpr int kXfEpiWarp0 = 2;
constexpr int kXfEpiCols = 64;                             // columns of a tile per epilogue warp
constexpr int kXfEpiWarps = 4 * (kXfCols / kXfEpiCols);    // kXfCols / kXfEpiCols per TMEM lane quarter
constexpr int kXfUnits = kXfEpiCols / 16;                  // scale blocks per thread and tile
constexpr int kXfThreads = 32 * (kXfEpiWarp0 + kXfEpiWarps);
constexpr uint32_t kXfTmemCols = 2 * kXfCols;
constexpr uint64_t kXfWaitNs = 2000000000ull;
static_assert(kXfSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ float round_bf16(float f) { return __bfloat162float(__float2bfloat16_rn(f)); }

// kAmaxOnly: the same pipeline computes y and only reduces max |y| over the
// tensor into *amax_out, as bf16 bits (no codes, scales or y written).
template <bool kAmaxOnly>
__global__ void __launch_bounds__(kXfThreads, 1)
    quant_transform_kernel(const __grid_constant__ CUtensorMap tmX, const QuantParams p, unsigned int *amax_out)
{
    extern __shared__ uint8_t xf_smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(xf_smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kXfOffBar);
    uint64_t *empty = full + kXfStages;
    uint64_t *tmem_full = empty + kXfStages;      // [2]
    uint64_t *tmem_empty = tmem_full + 2;         // [2]
    uint64_t *mma_done = tmem_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
    __shared__ float inv_tab[128];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int bs = p.bs;
    const int n_ct = (p.nbp * 16 + kXfCols - 1) / kXfCols;   // covers every scale column
    const int num_tiles = (p.mp / kXfRows) * n_ct;
    // x is read once; the amax pass leaves it in L2 for the quantizer that follows
    const uint64_t x_pol = kAmaxOnly ? l2_policy_evict_normal() : l2_policy_evict_first();
    // T (in 16-byte pieces, 8 consecutive n of one row i; T is 16-byte
    // aligned) and gs are loaded first, all loads in flight at once: issued
    // after the x tiles' copies they would queue behind ~20 MB of them and
    // hold back the first tile by about 2 us.
    constexpr int kPieces = (128 * 128 / 8 + kXfThreads - 1) / kXfThreads;
    const int pieces = bs * bs / 8;
    uint4 tv[kPieces];
#pragma unroll
    for (int u = 0; u < kPieces; ++u) {
        const int c = (int)threadIdx.x + u * kXfThreads;
        if (c < pieces) tv[u] = __ldg(reinterpret_cast<const uint4 *>(p.t) + c);
    }
    const float gs = kAmaxOnly ? 1.0f : __ldg(p.gs);   // the amax pass has no scale yet
    int pre_issued = 0;                           // (thread 0, the producer) stages issued before the role split
    if (threadIdx.x == 0) {
        griddep_launch_dependents();              // as in quant_kernel
        for (int s = 0; s < kXfStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tmem_full[b], 1);
            mbar_init(&tmem_empty[b], kXfEpiWarps);
        }
        mbar_init(mma_done, 1);
        fence_mbarrier_init();
        prefetch_tensormap(&tmX);
        // The first stages' x tiles are requested now, so that they load while
        // the block stages T and allocates its TMEM (their stages are free).
        for (int tile = blockIdx.x; tile < num_tiles && pre_issued < kXfStages; tile += gridDim.x, ++pre_issued) {
            const int rb = tile / n_ct, ct = tile - rb * n_ct;
            uint8_t *dst = smem + pre_issued * kXfStageBytes;
            mbar_arrive_expect_tx(&full[pre_issued], kXfStageBytes);
            tma_load_2d(dst, &tmX, &full[pre_issued], ct * kXfCols, rb * kXfRows, x_pol);
            tma_load_2d(dst + kXfBoxBytes, &tmX, &full[pre_issued], ct * kXfCols + 64, rb * kXfRows, x_pol);
        }
    }
    // T^T into shared memory: element T[i][n] -> row n, K index i, written
    // where the 128-byte swizzle puts it (16-byte chunk index XOR row % 8).
    uint8_t *sT = smem + kXfOffT;
    {
        const int lg = 31 - __clz(bs);                    // bs = 2^lg
#pragma unroll
        for (int u = 0; u < kPieces; ++u) {
            const int c = (int)threadIdx.x + u * kXfThreads;
            if (c < pieces) {
                const int i = c >> (lg - 3);
                const int n0 = (c & ((bs >> 3) - 1)) << 3;
                const uint32_t kb = (uint32_t)(i & 63) * 2;
                const uint32_t row0 = (uint32_t)(i >> 6) * bs * 128 + (kb & 15);
                const uint32_t w[4] = {tv[u].x, tv[u].y, tv[u].z, tv[u].w};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int n = n0 + q;
                    *reinterpret_cast<uint16_t *>(sT + row0 + n * 128 + (((kb >> 4) ^ (n & 7)) << 4)) =
                        (uint16_t)(w[q >> 1] >> ((q & 1) * 16));
                }
            }
        }
    }
    fence_proxy_async_shared();                   // the MMAs read T^T through the async proxy
    if (!kAmaxOnly) fill_inv_table(inv_tab, gs);
    if (warp == 1) {
        tmem_alloc(tmem_slot, kXfTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp >= kXfEpiWarp0) {
        // ---------------------------------------------------------- epilogue --
        const int q = warp & 3;
        const int h = (warp - kXfEpiWarp0) >> 2;
        const int64_t out_ld = p.kp >> 1;
        float tmax = 0.0f;                                // kAmaxOnly: this thread's max |y|
        int it = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
            const int b = it & 1;
            if (!__all_sync(~0u, mbar_wait(&tmem_full[b], (uint32_t)(it >> 1) & 1u, p.err_flag, kErrTimeout,
                                           kXfWaitNs)))
                break;
            tc_fence_after_sync();
            const uint32_t src = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * kXfCols + h * kXfEpiCols);
            uint32_t v[kXfEpiCols];
#pragma unroll
            for (int c = 0; c < kXfEpiCols / 32; ++c)
                tmem_ld_32cols(src + 32 * c, reinterpret_cast<uint32_t(&)[32]>(v[32 * c]));
#pragma unroll
            for (int c = 0; c < kXfEpiCols / 32; ++c) tmem_ld_wait_regs(reinterpret_cast<uint32_t(&)[32]>(v[32 * c]));
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tmem_empty[b]);

            const int rb = tile / n_ct, ct = tile - rb * n_ct;
            const int64_t r = (int64_t)rb * kXfRows + q * 32 + lane;
            const int c0 = ct * kXfCols + h * kXfEpiCols;
            uint32_t pk[2 * kXfUnits];
            uint32_t sfw = 0;
#pragma unroll
            for (int u = 0; u < kXfUnits; ++u) {
                const uint32_t *a = v + 16 * u;
                float y0[8], y1[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    y0[j] = round_bf16(__uint_as_float(a[j]));
                    y1[j] = round_bf16(__uint_as_float(a[8 + j]));
                }
                // The block maximum of the rounded values is the rounded
                // maximum of the fp32 sums (rounding to nearest is monotone
                // and symmetric): eight three-input maxima on the sums, then
                // one rounding, off the path of the element roundings.
                float m = quant_core::max_abs3(__uint_as_float(a[0]), __uint_as_float(a[1]), __uint_as_float(a[2]));
#pragma unroll
                for (int j = 3; j < 15; j += 2) m = quant_core::max_abs3(m, __uint_as_float(a[j]), __uint_as_float(a[j + 1]));
                m = quant_core::max_abs3(m, __uint_as_float(a[15]), __uint_as_float(a[15]));
                const float amax = round_bf16(m);
                if constexpr (kAmaxOnly) {
                    tmax = fmaxf(tmax, amax);
                    continue;
                }
                float inv;
                const uint32_t sf = block_scale_tab(amax, gs, inv_tab, inv);
                pk[2 * u] = quant8(y0, inv);
                pk[2 * u + 1] = quant8(y1, inv);
                sfw |= sf << (8 * u);
                if (p.y_out != nullptr && r < p.m && c0 + 16 * u < p.k) {   // k % 16 == 0
                    uint32_t w[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        w[j] = (__float_as_uint(y0[2 * j]) >> 16) | (__float_as_uint(y0[2 * j + 1]) & 0xFFFF0000u);
                        w[4 + j] = (__float_as_uint(y1[2 * j]) >> 16) | (__float_as_uint(y1[2 * j + 1]) & 0xFFFF0000u);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(p.y_out + r * p.k + c0 + 16 * u);
                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            if constexpr (kAmaxOnly) continue;
            if (r < p.m) {
                uint8_t *o = p.out + r * out_ld + (c0 >> 1);
#pragma unroll
                for (int pr = 0; pr < kXfUnits / 2; ++pr)           // 32 columns = 16 bytes (kp % 32 == 0)
                    if (c0 + 32 * pr < p.kp)
                        *reinterpret_cast<uint4 *>(o + 16 * pr) =
                            make_uint4(pk[4 * pr], pk[4 * pr + 1], pk[4 * pr + 2], pk[4 * pr + 3]);
            }
            const int cs = c0 >> 4;                       // columns >= k were zero-filled: codes 0
            if (cs < p.nbp) {                             // nbp % 4 == 0: the whole group is inside
                if (kXfUnits == 4)
                    *reinterpret_cast<uint32_t *>(p.sf + sf_offset(r, cs, p.nbp)) = sfw;
                else
                    *reinterpret_cast<uint16_t *>(p.sf + sf_offset(r, cs, p.nbp)) = (uint16_t)sfw;
            }
        }
        if constexpr (kAmaxOnly) {
            // max |y| is a bf16 value (a max of bf16 values): its top 16 bits
            // order like the magnitudes, so an integer max over bits is exact
            const uint32_t v = __reduce_max_sync(~0u, __float_as_uint(tmax) >> 16);
            if (lane == 0 && v != 0) atomicMax(amax_out, v);
        }
    } else if (warp == 0) {
        if (lane == 0) {
            // --------------------------------------------------------- producer --
            int it = pre_issued;
            for (int tile = blockIdx.x + pre_issued * (int)gridDim.x; tile < num_tiles; tile += gridDim.x, ++it) {
                const int stage = it % kXfStages;
                if (!mbar_wait(&empty[stage], ((uint32_t)(it / kXfStages) & 1u) ^ 1u, p.err_flag, kErrTimeout,
                               kXfWaitNs))
                    break;
                const int rb = tile / n_ct, ct = tile - rb * n_ct;
                uint8_t *dst = smem + stage * kXfStageBytes;
                mbar_arrive_expect_tx(&full[stage], kXfStageBytes);
                tma_load_2d(dst, &tmX, &full[stage], ct * kXfCols, rb * kXfRows, x_pol);
                tma_load_2d(dst + kXfBoxBytes, &tmX, &full[stage], ct * kXfCols + 64, rb * kXfRows, x_pol);
            }
            // Every copy issued has landed before the CTA may exit (the last
            // issue of each stage is its newest phase).
            for (int j = max(0, it - kXfStages); j < it; ++j)
                mbar_wait(&full[j % kXfStages], (uint32_t)(j / kXfStages) & 1u, p.err_flag, kErrTimeout, kXfWaitNs);
        }
    } else {
        // ---------------------------------------------------------------- MMA --
        const bool leader = elect_one();
        const uint32_t idesc = idesc_bf16(128, (uint32_t)bs);
        const uint32_t x_base = smem_u32(smem);
        const uint32_t t_base = smem_u32(sT);
        int it = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
            const int stage = it % kXfStages;
            const int b = it & 1;
            if (!__all_sync(~0u, mbar_wait(&tmem_empty[b], ((uint32_t)(it >> 1) & 1u) ^ 1u, p.err_flag, kErrTimeout,
                                           kXfWaitNs)))
                break;
            if (!__all_sync(~0u, mbar_wait(&full[stage], (uint32_t)(it / kXfStages) & 1u, p.err_flag, kErrTimeout,
                                           kXfWaitNs)))
                break;
            tc_fence_after_sync();
            if (leader) {
                const uint32_t d0 = tmem + (uint32_t)(b * kXfCols);
                const uint32_t xs = x_base + stage * kXfStageBytes;
                for (int g = 0; g < kXfCols / bs; ++g) {
                    for (int kk = 0; kk < bs / 16; ++kk) {
                        // K-step of 16: 32 bytes further into the swizzled 128-byte rows
                        const int c = g * bs + kk * 16;       // column of the x tile
                        const int i = kk * 16;                // row of T
                        const uint32_t a_addr = xs + (uint32_t)(c >> 6) * kXfBoxBytes + (uint32_t)(c & 63) * 2;
                        const uint32_t b_addr = t_base + (uint32_t)(i >> 6) * bs * 128 + (uint32_t)(i & 63) * 2;
                        tc_mma_bf16(d0 + (uint32_t)(g * bs), smem_desc_sw128(a_addr), smem_desc_sw128(b_addr), idesc,
                                    kk != 0);
                    }
                }
                tc_commit(&empty[stage]);
                tc_commit(&tmem_full[b]);
            }
            __syncwarp();
        }
        // No MMA may still be running when the TMEM is released.
        if (leader) tc_commit(mma_done);
        __syncwarp();
        mbar_wait(mma_done, 0, p.err_flag, kErrTimeout, kXfWaitNs);
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem, kXfTmemCols);
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
    // a programmatic dependent of whatever precedes it on the stream: its
    // blocks may be scheduled early, then wait (griddepcontrol.wait) for it
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quant_kernel<U>, p);
}

namespace {

// Sets the shared-memory attribute of both transform-kernel variants (once
// per device), encodes the activation's tensor map and launches one variant.
template <bool kAmaxOnly>
cudaError_t launch_transform_variant(const QuantParams &p, unsigned int *amax_out, int num_sms, cudaStream_t s,
                                     const char **why)
{
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(quant_transform_kernel<kAmaxOnly>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kXfSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    CUtensorMap tmX;
    if (!gemm_detail::make_bf16_rows_map(&tmX, p.x, (uint64_t)p.k, (uint64_t)p.m, (uint64_t)p.ldx)) {
        *why = "cuTensorMapEncodeTiled failed for the activation";
        return cudaErrorInvalidValue;
    }
    const int64_t n_ct = ((int64_t)p.nbp * 16 + kXfCols - 1) / kXfCols;
    const int64_t tiles = (int64_t)(p.mp / kXfRows) * n_ct;
    const int grid = (int)(tiles < num_sms ? tiles : num_sms);
    quant_transform_kernel<kAmaxOnly><<<(unsigned)grid, kXfThreads, kXfSmemBytes, s>>>(tmX, p, amax_out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_transform(const QuantParams &p, int num_sms, cudaStream_t s, const char **why)
{
    return launch_transform_variant<false>(p, nullptr, num_sms, s, why);
}

cudaError_t launch_quant_mx(const QuantParams &p, int num_sms, cudaStream_t s)
{
    constexpr int U = 4;
    const int64_t segs = (p.kp + 511) / 512;
    const int64_t tasks = (int64_t)p.mp * segs;
    int64_t blocks = ((tasks + U - 1) / U + 7) / 8;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quant_mx_kernel<U><<<(unsigned)blocks, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_act_global_scale(const QuantParams &p, const float *w_gs, float *gs_out, float *alpha_out,
                                    int num_sms, cudaStream_t s, const char **why)
{
    unsigned int *word = reinterpret_cast<unsigned int *>(gs_out);
    cudaError_t e = cudaMemsetAsync(word, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    if (p.m > 0) {
        if (p.bs) {
            e = launch_transform_variant<true>(p, word, num_sms, s, why);
        } else {
            constexpr int U = 4;
            const int64_t tasks = (int64_t)p.m * ((p.k + 511) / 512);
            int64_t blocks = ((tasks + U - 1) / U + 7) / 8;
            const int64_t cap = (int64_t)num_sms * 8;
            if (blocks > cap) blocks = cap;
            if (blocks < 1) blocks = 1;
            act_amax_kernel<U><<<(unsigned)blocks, 256, 0, s>>>(p, word);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
    }
    act_scale_finalize_kernel<<<1, 1, 0, s>>>(word, alpha_out != nullptr ? w_gs : nullptr, alpha_out);
    return cudaGetLastError();
}

}  // namespace nvfp4
