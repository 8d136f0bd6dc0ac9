// Block-scaled FP4 GEMM with fused epilogue on the sm_103a tensor cores.
//
// Page "TorchNvFp4LinearKernel" (vLLM PR #53319), section 关键源码片段:
// apply_weights computes torch._scaled_mm(x_fp4, weight.t(), scale_a, scale_b,
// out_dtype), then out * alpha, slice_nvfp4_output, + bias.  Here that is one
// kernel:
//     out[m, n] = bf16( alpha * sum_k A[m,k] B[n,k] + bias[n] ),  n < n_out,
// A, B packed E2M1 (K-major) with one UE4M3 scale per 16 K-elements.
//
// Design (one CTA per SM, persistent over output tiles of 128 x 256):
//   warp 0      TMA producer: A tile 128 x 256 FP4 (16 KB), B tile 256 x 256 FP4
//               (32 KB), both 128-byte swizzled, plus the matching 512-byte
//               scale tiles by bulk copy, into a 4-stage shared-memory ring;
//   warps 2,3   scale copiers (lane 0 of each): tcgen05.cp moves the stage's
//               scale tiles into that stage's TMEM columns, two K-steps per
//               copier, and each commits to sf_ready[stage];
//   warp 1      MMA issuer: 4 x tcgen05.mma (M=128, N=256, K=64,
//               kind::mxf4nvf4, scale_vec::4X) per stage accumulate into a
//               128 x 256 fp32 TMEM tile; tcgen05.commit releases the smem
//               stage / signals the epilogue;
//   warp 2      also allocates and frees the 512 TMEM columns;
//   warps 4..7  epilogue: tcgen05.ld of their 32-lane quarter, fma with alpha
//               and bias, bf16 round into registers, release of the TMEM tile,
//               then masked stores (rows < m, cols < n_out) that overlap the
//               next tile's MMAs.
// TMEM columns: [0,256) accumulator; stage s scales at 256 + 48 s (A: 16
// columns = 4 K-steps x 4; B: 32 columns = 4 K-steps x 2 row-halves x 4).
// Every mbarrier wait is bounded (about 2 s); on expiry the kernel raises the
// device error word, drains what it issued and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace nvfp4 {

__device__ unsigned int g_error_word;

cudaError_t device_error_word(unsigned int **ptr)
{
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_error_word);
}

namespace {

using namespace gemm_detail;

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBKBytes = 128;                 // 256 FP4 elements of K per stage
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBKBytes;  // 16 KB
constexpr uint32_t kBBytes = kBN * kBKBytes;  // 32 KB
constexpr uint32_t kSfaBytes = 4 * 512;       // 4 K-steps of one 128-row band
constexpr uint32_t kSfbBytes = 2 * 4 * 512;   // two 128-row bands
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffSfa = kOffB + kStages * kBBytes;
constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfaBytes;
constexpr uint32_t kOffBias = kOffSfb + kStages * kSfbBytes;   // per epilogue warp: one tile of bias
constexpr uint32_t kOffBar = kOffBias + 4 * kBN * 2;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;   // barriers + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSf = 256;
constexpr uint32_t kSfColsPerStage = 48;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4;                  // warps 4..7: epilogue, one per TMEM lane quarter
constexpr int kEpiWarps = 4;
constexpr int kCopiers = 2;                   // lane 0 of warps 2 and 3: two K-steps of each stage each

// Copier index of a thread (-1 if it does not copy scales).  The copiers sit
// in different warps: a warp issues a tcgen05 instruction for one lane only.
__device__ __forceinline__ int copier_of(int warp, int lane)
{
    return lane == 0 ? (warp == 2 ? 0 : warp == 3 ? 1 : -1) : -1;
}

static_assert(kSmemBytes <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *empty = full + kStages;
    uint64_t *sf_ready = empty + kStages;
    uint64_t *tmem_full = sf_ready + kStages;
    uint64_t *tmem_empty = tmem_full + 1;
    uint64_t *mma_done = tmem_empty + 1;
    uint64_t *cp_done = mma_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cp_done + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], kCopiers);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, kEpiWarps);
        mbar_init(mma_done, 1);
        mbar_init(cp_done, kCopiers);
        fence_mbarrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int num_tiles = p.num_m_blk * p.num_n_blk;
    const int num_ks = (p.num_k64 + 3) / 4;
    const int n_bands_w = (p.n_w + 127) / 128;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ producer --
        const uint64_t pol_a = l2_policy_evict_last();
        const uint64_t pol_b = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk);
            const int n_rows = min(kBN, p.n_out - t.nb * kBN);
            const int halves = n_rows > 128 ? 2 : 1;
            for (int ks = 0; ks < num_ks; ++ks) {
                if (!mbar_wait(&empty[stage], phase ^ 1, p.err_flag, kErrTimeout, kWaitNs)) { ok = false; break; }
                const int kcount = min(4, p.num_k64 - ks * 4);
                const uint32_t sf_bytes = (uint32_t)kcount * 512;
                mbar_arrive_expect_tx(&full[stage], kABytes + kBBytes + sf_bytes * (1 + halves));
                tma_load_2d(smem + kOffA + stage * kABytes, &tmA, &full[stage], ks * kBKBytes, t.mb * kBM, pol_a);
                tma_load_2d(smem + kOffB + stage * kBBytes, &tmB, &full[stage], ks * kBKBytes, t.nb * kBN, pol_b);
                bulk_load(smem + kOffSfa + stage * kSfaBytes, p.sfa + t.mb * p.sfa_band_bytes + (int64_t)ks * 2048,
                          sf_bytes, &full[stage], pol_a);
                for (int h = 0; h < halves; ++h)    // halves == 2 implies band t.nb*2+1 < n_bands_w
                    bulk_load(smem + kOffSfb + stage * kSfbBytes + h * 2048,
                              p.sfb + (t.nb * 2 + h) * p.sfb_band_bytes + (int64_t)ks * 2048, sf_bytes, &full[stage],
                              pol_b);
                issued_mask |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
        }
        (void)n_bands_w;
        // Every copy this thread issued has landed before the CTA may exit.
        for (int s = 0; s < kStages; ++s)
            if (issued_mask & (1u << s))
                mbar_wait(&full[s], (issued_phase >> s) & 1u, p.err_flag, kErrTimeout, kWaitNs);
    } else if (copier_of(warp, lane) >= 0) {
        // --------------------------------------------------- scale copiers --
        // Copier c moves K-steps 2c and 2c+1 of each stage (the A band's tile
        // and the B bands' tiles) from shared memory into that stage's TMEM
        // columns and commits to sf_ready[stage], which completes once both
        // have.  Two issuing threads keep the copies off the MMA's critical path.
        // A stage's TMEM columns are rewritten only after the producer
        // refilled the stage, i.e. after the MMAs that read them completed.
        const int cidx = copier_of(warp, lane);
        int stage = 0;
        uint32_t phase = 0;
        const uint32_t sfa_base = smem_u32(smem + kOffSfa);
        const uint32_t sfb_base = smem_u32(smem + kOffSfb);
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk);
            const int n_rows = min(kBN, p.n_out - t.nb * kBN);
            const int halves = n_rows > 128 ? 2 : 1;
            for (int ks = 0; ks < num_ks; ++ks) {
                if (!mbar_wait(&full[stage], phase, p.err_flag, kErrTimeout, kWaitNs)) { ok = false; break; }
                tc_fence_after_sync();
                const int kcount = min(4, p.num_k64 - ks * 4);
                const uint32_t sf_col = tmem + kTmemSf + stage * kSfColsPerStage;
                for (int kk = 2 * cidx; kk < 2 * cidx + 2 && kk < kcount; ++kk) {
                    tc_cp_32x128b_warpx4(sf_col + kk * 4, smem_desc_sf(sfa_base + stage * kSfaBytes + kk * 512));
                    for (int h = 0; h < halves; ++h)
                        tc_cp_32x128b_warpx4(sf_col + 16 + kk * 8 + h * 4,
                                             smem_desc_sf(sfb_base + stage * kSfbBytes + h * 2048 + kk * 512));
                }
                tc_commit(&sf_ready[stage]);
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
        }
        tc_commit(cp_done);
        mbar_wait(cp_done, 0, p.err_flag, kErrTimeout, kWaitNs);
    } else if (warp == 1 && lane == 0) {
        // ----------------------------------------------------------- MMA --
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        const uint32_t a_base = smem_u32(smem + kOffA);
        const uint32_t b_base = smem_u32(smem + kOffB);
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk);
            const int n_rows = min(kBN, p.n_out - t.nb * kBN);
            const uint32_t idesc = n_rows > 128 ? idesc_nvf4(128, 256) : idesc_nvf4(128, 128);
            if (!mbar_wait(tmem_empty, acc_phase ^ 1, p.err_flag, kErrTimeout, kWaitNs)) break;
            tc_fence_after_sync();
            for (int ks = 0; ks < num_ks; ++ks) {
                if (!mbar_wait(&sf_ready[stage], phase, p.err_flag, kErrTimeout, kWaitNs) ||
                    !mbar_wait(&full[stage], phase, p.err_flag, kErrTimeout, kWaitNs)) { ok = false; break; }
                tc_fence_after_sync();
                const int kcount = min(4, p.num_k64 - ks * 4);
                const uint32_t sf_col = tmem + kTmemSf + stage * kSfColsPerStage;
                const uint64_t adesc = smem_desc_sw128(a_base + stage * kABytes);
                const uint64_t bdesc = smem_desc_sw128(b_base + stage * kBBytes);
                for (int kk = 0; kk < kcount; ++kk) {
                    // K-step kk starts 32 bytes further into the swizzled 128-byte rows
                    tc_mma_nvf4(tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc,
                                sf_col + kk * 4, sf_col + 16 + kk * 8, (ks | kk) != 0);
                }
                tc_commit(&empty[stage]);
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            tc_commit(tmem_full);
            acc_phase ^= 1;
        }
        // No MMA may still be running when the TMEM is released.
        tc_commit(mma_done);
        mbar_wait(mma_done, 0, p.err_flag, kErrTimeout, kWaitNs);
    } else if (warp >= kEpiWarp0) {
        // ------------------------------------------------------ epilogue --
        // Drain the whole 128 x 256 accumulator into registers as packed bf16
        // (alpha and bias applied), release the TMEM to the MMA thread, and only
        // then write the tile out, so the stores overlap the next tile's MMAs.
        const int q = warp & 3;
        uint16_t *s_bias = reinterpret_cast<uint16_t *>(smem + kOffBias) + (warp - kEpiWarp0) * kBN;
        const float alpha = __ldg(p.alpha);
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk);
            const int n_rows = min(kBN, p.n_out - t.nb * kBN);
            const int col_base = t.nb * kBN;
            if (p.bias != nullptr) {                            // this warp's copy of the tile's bias
                __syncwarp();                                   // previous tile done reading it
                for (int j = lane; j < kBN; j += 32)
                    s_bias[j] = (j < n_rows) ? p.bias[col_base + j] : (uint16_t)0;
                __syncwarp();
            }
            if (!mbar_wait(tmem_full, acc_phase, p.err_flag, kErrTimeout, kWaitNs)) break;
            tc_fence_after_sync();
            uint32_t packed[kBN / 2];
#pragma unroll
            for (int ch = 0; ch < kBN / 32; ++ch) {
                if (ch * 32 < n_rows) {                         // uniform across the warp
                    uint32_t r[32];
                    tmem_ld_32cols(tmem + ((uint32_t)(q * 32) << 16) + ch * 32, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        float b0 = 0.0f, b1 = 0.0f;
                        if (p.bias != nullptr) {
                            const uint32_t bw = *reinterpret_cast<const uint32_t *>(s_bias + ch * 32 + j);
                            b0 = __uint_as_float(bw << 16);
                            b1 = __uint_as_float(bw & 0xFFFF0000u);
                        }
                        const uint32_t lo = bf16_bits_rn(__fmaf_rn(__uint_as_float(r[j]), alpha, b0));
                        const uint32_t hi = bf16_bits_rn(__fmaf_rn(__uint_as_float(r[j + 1]), alpha, b1));
                        packed[ch * 16 + j / 2] = lo | (hi << 16);
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(tmem_empty);
            acc_phase ^= 1;

            const int64_t row = (int64_t)t.mb * kBM + q * 32 + lane;
            if (row < p.m) {
                uint16_t *orow = p.out + row * p.ldo + col_base;
#pragma unroll
                for (int v = 0; v < kBN / 8; ++v) {
                    if (v * 8 + 8 <= n_rows) {
                        *reinterpret_cast<uint4 *>(orow + v * 8) =
                            make_uint4(packed[v * 4], packed[v * 4 + 1], packed[v * 4 + 2], packed[v * 4 + 3]);
                    } else if (v * 8 < n_rows) {
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if (v * 8 + e < n_rows)
                                orow[v * 8 + e] = (uint16_t)(packed[v * 4 + e / 2] >> ((e & 1) * 16));
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_gemm(const GemmParams &p, const uint8_t *a, const uint8_t *w, int num_sms, cudaStream_t s,
                        const char **why)
{
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e =
            cudaFuncSetAttribute(gemm_nvf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    CUtensorMap tmA, tmB;
    const uint64_t row_bytes = (uint64_t)p.kp / 2;
    if (!make_operand_map(&tmA, a, row_bytes, (uint64_t)p.m, kBM) ||
        !make_operand_map(&tmB, w, row_bytes, (uint64_t)p.n_w, kBN)) {
        *why = "cuTensorMapEncodeTiled failed for an FP4 operand";
        return cudaErrorInvalidValue;
    }
    const int tiles = p.num_m_blk * p.num_n_blk;
    const int grid = tiles < num_sms ? tiles : num_sms;
    gemm_nvf4_kernel<<<grid, kThreads, kSmemBytes, s>>>(tmA, tmB, p);
    return cudaGetLastError();
}

}  // namespace nvfp4
