// Block-scaled FP4 GEMM on CTA pairs (tcgen05 cta_group::2), for m > 128.
//
// Same operation as gemm.cu (page "TorchNvFp4LinearKernel", vLLM PR #53319,
// section 关键源码片段: _scaled_mm, * alpha, slice, + bias), with each output
// tile of 256 x 256 computed by a cluster of two CTAs on two SMs.  Per CTA
// r (r = 0, 1; rank 0 leads), sixteen warps in four warpgroups:
//   warps 0, 3  TMA producers of the operand ring (5 stages of 32 KB): warp 0
//               this CTA's A rows [128r, 128r + 128) of the tile, warp 3 its
//               half of B (rows [128r, 128r + 128) of the tile's 256);
//   warp 2      TMA producer of the scale ring (5 stages of 6 KB): this CTA's
//               A scale band and the scale tiles of both B bands (each CTA's
//               TMEM needs the scales of all 256 B rows);
//   warp 1      allocates the pair's TMEM; in the leader it issues, from one
//               elected lane of the converged warp, tcgen05.mma.cta_group::2
//               (M = 256, N = 256, K = 64): each CTA's tensor core reads its
//               own A rows and both B halves and accumulates its 128 x 256
//               fp32 tile in its own TMEM; the commits multicast to both CTAs'
//               barriers;
//   warps 4..7  one per TMEM lane quarter: read a stage's scales from the
//               scale ring (and release it), write them into the stage's TMEM
//               columns once the MMAs of the slot's previous use are done
//               (tcgen05.st), wait for the stage's operands in this CTA and
//               arrive on the leader's sf_ready[stage], which therefore
//               completes once both CTAs hold the stage's operands and scales;
//   warps 8..15 epilogue, two per TMEM lane quarter: load this CTA's whole
//               accumulator into registers (four loads in flight), hand it
//               back to the MMA warp, then apply alpha and bias, round to bf16
//               and TMA-store the rows.
// Per SM and stage this moves 38 KB into shared memory instead of 54 KB, so
// five stages fit where the one-CTA kernel holds four.  Every mbarrier wait is
// bounded; all threads meet at one final cluster barrier before the TMEM is
// released.
#include <cuda_bf16.h>

#include "common.cuh"
#include "gemm_common.cuh"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

using namespace gemm_detail;

constexpr int kTileM = 256;                     // per pair (128 rows per CTA)
constexpr int kWalkGroup = 32;                  // pair tiles per group of the tile walk (8192 rows)
constexpr int kTileN = 256;
constexpr int kRowsCta = 128;
constexpr int kBKBytes = 128;                   // 256 FP4 elements of K per stage
constexpr int kStages = 5;
constexpr int kEpiColsBias = 128;                     // bias columns per epilogue warp
constexpr uint32_t kABytes = kRowsCta * kBKBytes;     // 16 KB: this CTA's A rows
constexpr uint32_t kBBytes = kRowsCta * kBKBytes;     // 16 KB: this CTA's half of B
constexpr uint32_t kSfaBytes = 4 * 512;               // this CTA's A band, 4 K-steps
constexpr uint32_t kSfbBytes = 2 * 4 * 512;           // both B bands of the tile
constexpr uint32_t kOutChunkBytes = 32 * 64 * 2;      // output staging: 32 rows x 64 columns bf16 (4 KB)
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffSfa = kOffB + kStages * kBBytes;
constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfaBytes;
constexpr uint32_t kOffBias = kOffSfb + kStages * kSfbBytes;  // per epilogue warp: its 128 bias columns (bf16)
constexpr uint32_t kOffOut = (kOffBias + 8 * kEpiColsBias * 2 + 1023) / 1024 * 1024;   // one chunk per epilogue warp
constexpr uint32_t kOffBar = kOffOut + 8 * kOutChunkBytes;
constexpr uint32_t kSmemBytes = kOffBar + 512 + 1024;         // barriers + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSf = 256;
constexpr uint32_t kSfColsPerStage = 48;
constexpr int kThreads = 512;
constexpr int kSfWarp0 = 4;
constexpr int kEpiWarp0 = 8;
constexpr int kEpiWarps = 8;
constexpr int kEpiCols = kTileN / 2;
constexpr uint16_t kBothCtas = 0x3;
// registers per thread after setmaxnreg: the epilogue holds a whole 128-column
// accumulator slice (128 registers) at once
constexpr uint32_t kRegsCtl = 56, kRegsSf = 88, kRegsEpi = 184;

static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffOut % 1024 == 0, "128-byte-swizzled TMA store sources are 1024-byte aligned");
static_assert(kTmemSf + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
static_assert(128 * (kRegsCtl + kRegsSf + 2 * kRegsEpi) <= kThreads * 128, "register reallocation budget");

// kMx: MXFP4 operands (UE8M0 scales per 32 K-elements, scale_vec::2X), else NVFP4.
template <bool kMx>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmSfb, const __grid_constant__ CUtensorMap tmOut,
                          const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar);   // this CTA's operands of the stage landed
    uint64_t *empty = full + kStages;                                 // the pair's MMAs released the stage
    uint64_t *sf_ready = empty + kStages;                             // (leader) both CTAs' scales staged
    uint64_t *tmem_full = sf_ready + kStages;                         // accumulator complete
    uint64_t *tmem_empty = tmem_full + 1;                             // (leader) both CTAs drained it
    uint64_t *mma_done = tmem_empty + 1;
    uint64_t *sf_full = mma_done + 1;                                 // the stage's scale tiles landed
    uint64_t *sf_empty = sf_full + kStages;                           // the scale warps have read them
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sf_empty + kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool is_leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 2);             // the activation and the weight producer
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], 2 * 4);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, 2 * kEpiWarps);
        mbar_init(mma_done, 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sf_full[s], 1);          // the scale producer
            mbar_init(&sf_empty[s], 4);         // the four scale warps
        }
        fence_mbarrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        prefetch_tensormap(&tmSfb);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncwarp();
    cluster_sync_all();                 // barrier inits and the TMEM allocation visible in both CTAs
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int pair_id = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;
    const int num_tiles = p.num_m_blk * p.num_n_blk;       // num_m_blk counts 256-row tiles here
    const int num_ks = (p.num_k64 + 3) / 4;
    const int a_bands = (p.m + 127) / 128;

    if (warp >= kEpiWarp0) {
        setmaxnreg_inc<kRegsEpi>();
        // ------------------------------------------------------ epilogue --
        const int q = warp & 3;
        const int hcol = ((warp - kEpiWarp0) >> 2) * kEpiCols;
        const uint32_t acc = tmem + ((uint32_t)(q * 32) << 16) + hcol;
        const uint32_t out_stage = smem_u32(smem + kOffOut) + (warp - kEpiWarp0) * kOutChunkBytes;
        const uint32_t leader_tmem_empty = mapa_shared(tmem_empty, 0);
        const bool use_bias = p.bias != nullptr;
        const bool bias_vec = (reinterpret_cast<uintptr_t>(p.bias) & 7) == 0;   // 8-byte loads of 4 columns
        const float alpha = p.alpha != nullptr ? __ldg(p.alpha) : 1.0f;
        const uint64_t out_policy = l2_policy_evict_first();   // the output is written once
        uint32_t acc_phase = 0;
        int it = 0;
        for (int tile = pair_id; tile < num_tiles; tile += num_pairs, ++it) {
            const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk, kWalkGroup);
            const int n_cols = min(kEpiCols, p.n_out - t.nb * kTileN - hcol);   // may be <= 0
            const int col_base = t.nb * kTileN + hcol;
            // this warp's 128 bias columns into its own buffer (four per lane)
            // while the accumulator is still being computed
            uint16_t *s_bias = reinterpret_cast<uint16_t *>(smem + kOffBias) + (warp - kEpiWarp0) * kEpiColsBias;
            if (use_bias) {
                const int c0 = col_base + 4 * lane;
                uint2 bw = make_uint2(0u, 0u);
                if (bias_vec && c0 + 4 <= p.n_out) {
                    bw = __ldg(reinterpret_cast<const uint2 *>(p.bias + c0));
                } else {
                    uint16_t e[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) e[i] = (c0 + i < p.n_out) ? p.bias[c0 + i] : (uint16_t)0;
                    bw = make_uint2(e[0] | ((uint32_t)e[1] << 16), e[2] | ((uint32_t)e[3] << 16));
                }
                *reinterpret_cast<uint2 *>(s_bias + 4 * lane) = bw;
                __syncwarp();
            }
            if (!__all_sync(~0u, mbar_wait(tmem_full, acc_phase, p.err_flag, kErrTimeout, p.wait_ns))) break;
            tc_fence_after_sync();
            acc_phase ^= 1;

            // Load this warp's 128 accumulator columns with all four 32-column
            // loads in flight and hand the accumulator back to the MMA warp
            // as soon as they have landed: the next tile's MMAs wait only for
            // the loads, not for the arithmetic and stores below.
            uint32_t acc_regs[kEpiCols / 32][32];
            if (n_cols > 0) {                                   // uniform across the warp
#pragma unroll
                for (int ch = 0; ch < kEpiCols / 32; ++ch) tmem_ld_32cols(acc + ch * 32, acc_regs[ch]);
#pragma unroll
                for (int ch = 0; ch < kEpiCols / 32; ++ch) tmem_ld_wait_regs(acc_regs[ch]);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (is_leader) mbar_arrive(tmem_empty);          // the leader's own barrier: local arrive
                else mbar_arrive_remote(leader_tmem_empty);
            }

            // alpha, bias and bf16 rounding, 32 columns at a time, straight
            // into this warp's staging buffer; then TMA stores of two 32-row
            // x 64-column chunks (128-byte rows, the TMA's 128-byte swizzle:
            // 16-byte piece j of row r sits at piece j ^ (r % 8), which also
            // spreads the 32 lanes' writes over all banks).  Rows >= m and
            // columns >= n_out are clipped by the TMA.
            const int row0 = t.mb * kTileM + (int)rank * kRowsCta + q * 32;
#pragma unroll
            for (int c = 0; c < kEpiCols / 64; ++c) {
                if (c * 64 < n_cols) {                          // uniform across the warp
                    if (lane == 0) bulk_wait_group_read<0>();   // the previous store has read the buffer
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int ch = c * 2 + h;
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            float b0 = 0.0f, b1 = 0.0f;
                            if (use_bias) {
                                const uint32_t bw = *reinterpret_cast<const uint32_t *>(s_bias + ch * 32 + j);
                                b0 = __uint_as_float(bw << 16);
                                b1 = __uint_as_float(bw & 0xFFFF0000u);
                            }
                            pk[j / 2] = bf16x2_rn(__fmaf_rn(__uint_as_float(acc_regs[ch][j]), alpha, b0),
                                                  __fmaf_rn(__uint_as_float(acc_regs[ch][j + 1]), alpha, b1));
                        }
#pragma unroll
                        for (int j4 = 0; j4 < 4; ++j4) {
                            const int piece = h * 4 + j4;
                            st_shared_v4(out_stage + lane * 128 + ((piece ^ (lane & 7)) << 4), pk[j4 * 4],
                                         pk[j4 * 4 + 1], pk[j4 * 4 + 2], pk[j4 * 4 + 3]);
                        }
                    }
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmOut, out_stage, col_base + c * 64, row0, out_policy);
                        bulk_commit_group();
                    }
                }
            }
            __syncwarp();                                       // every lane has read the bias buffer
        }
        if (lane == 0) bulk_wait_group<0>();                    // all output written before the CTA exits
    } else if (warp >= kSfWarp0) {
        setmaxnreg_dec<kRegsSf>();
        // ----------------------------------------------- scale staging --
        // tcgen05.cp 32x128b.warpx4 layout: lane 32q + i of quarter q gets
        // bytes [16i, 16i + 16) of each 512-byte scale tile.  A stage's TMEM
        // scale columns are rewritten only after the MMAs of its previous use
        // have completed (their commit on `empty`).
        const int q = warp & 3;
        const uint32_t sf_tmem = tmem + ((uint32_t)(q * 32) << 16) + kTmemSf;
        const uint32_t sfa_smem = smem_u32(smem + kOffSfa) + lane * 16;
        const uint32_t sfb_smem = smem_u32(smem + kOffSfb) + lane * 16;
        const uint32_t leader_sf_ready = mapa_shared(sf_ready, 0);
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
            for (int ks = 0; ks < num_ks; ++ks) {
                ok = __all_sync(~0u, mbar_wait(&sf_full[stage], phase, p.err_flag, kErrTimeout, p.wait_ns));
                if (!ok) break;
                constexpr int kT = kSfTilesPerStage<kMx>;
                uint32_t a[4 * kT], b[8 * kT];
#pragma unroll
                for (int j = 0; j < kT; ++j) {
                    const uint4 v = ld_shared_v4(sfa_smem + stage * kSfaBytes + j * 512);
                    a[j * 4 + 0] = v.x; a[j * 4 + 1] = v.y; a[j * 4 + 2] = v.z; a[j * 4 + 3] = v.w;
                }
#pragma unroll
                for (int j = 0; j < kT; ++j)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 v = ld_shared_v4(sfb_smem + stage * kSfbBytes + h * (kT * 512) + j * 512);
                        uint32_t *d = b + j * 8 + h * 4;
                        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
                    }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_empty[stage]);   // the scale slot may be refilled
                // The stage's TMEM scale columns are free once the MMAs of the
                // slot's previous use are done (the commit on `empty`).
                ok = __all_sync(~0u, mbar_wait(&empty[stage], phase ^ 1, p.err_flag, kErrTimeout, p.wait_ns));
                if (!ok) break;
                // (tiles past the valid K-steps, B rows or A rows hold stale
                // bytes; what they meet in the MMA is never stored)
                if constexpr (kMx) {
                    tmem_st_8cols(sf_tmem + stage * kSfColsPerStage, a);
                    tmem_st_16cols(sf_tmem + stage * kSfColsPerStage + 4 * kT, b);
                } else {
                    tmem_st_16cols(sf_tmem + stage * kSfColsPerStage, a);
                    tmem_st_32cols(sf_tmem + stage * kSfColsPerStage + 4 * kT, b);
                }
                tmem_st_wait();
                tc_fence_before_sync();
                // and this CTA's operands of the stage have landed: then the
                // leader's MMA may read them (sf_ready counts both CTAs)
                ok = __all_sync(~0u, mbar_wait(&full[stage], phase, p.err_flag, kErrTimeout, p.wait_ns));
                if (!ok) break;
                __syncwarp();
                if (lane == 0) {
                    if (is_leader) mbar_arrive(&sf_ready[stage]);      // the leader's own barrier: local arrive
                    else mbar_arrive_remote(leader_sf_ready + stage * (uint32_t)sizeof(uint64_t));
                }
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
        }
    } else {
        setmaxnreg_dec<kRegsCtl>();
        if ((warp == 0 || warp == 3) && lane == 0 && !p.drill) {   // (a timeout drill issues no copies)
            // ---------------------------------------------- operand producers --
            // Two threads per CTA fill the operand ring, each with its half of
            // every stage and one arrival on `full` (count 2): warp 0 this
            // CTA's A rows (after the wait for the preceding grid, the
            // activation quantizer when launched as its dependent), warp 3
            // this CTA's half of B.
            const bool act_side = warp == 0;
            const uint64_t pol = l2_policy_evict_last();
            if (act_side) griddep_wait();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
                const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk, kWalkGroup);
                const int band_a = t.mb * 2 + (int)rank;
                for (int ks = 0; ks < num_ks; ++ks) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, p.err_flag, kErrTimeout, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    // (a box past the last row is zero-filled and still counts
                    // its full bytes)
                    mbar_arrive_expect_tx(&full[stage], act_side ? kABytes : kBBytes);
                    if (act_side)
                        tma_load_2d(smem + kOffA + stage * kABytes, &tmA, &full[stage], ks * kBKBytes,
                                    band_a * kRowsCta, pol);
                    else
                        tma_load_2d(smem + kOffB + stage * kBBytes, &tmB, &full[stage], ks * kBKBytes,
                                    t.nb * kTileN + (int)rank * kRowsCta, pol);
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) { stage = 0; phase ^= 1; }
                }
            }
            for (int s = 0; s < kStages; ++s)
                    if (issued_mask & (1u << s))
                    mbar_wait(&full[s], (issued_phase >> s) & 1u, p.err_flag, kErrTimeout, p.wait_ns);
        } else if (warp == 2 && lane == 0 && !p.drill) {
            // ------------------------------------------------- scale producer --
            // The scale tiles travel apart from the operands, in a ring of
            // their own that frees as soon as the scale warps have read it:
            // so they are requested stages ahead, and a stage's scales are in
            // TMEM before its operands land.  Per stage: this CTA's A band
            // (kT tiles, bulk copy) and both B bands of the tile (one 2-D copy,
            // 8-byte elements, box of kT tiles x 2 bands; the TMA fills zeros
            // past the last band or K-step).  The A scales may be the
            // preceding grid's output (the quantizer): wait for it first.
            constexpr int kT = kSfTilesPerStage<kMx>;
            const uint64_t pol = l2_policy_evict_last();
            griddep_wait();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
                const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk, kWalkGroup);
                const int band_a = t.mb * 2 + (int)rank;
                const bool a_here = band_a < a_bands;
                for (int ks = 0; ks < num_ks; ++ks) {
                    if (!mbar_wait(&sf_empty[stage], phase ^ 1, p.err_flag, kErrTimeout, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sfa_bytes = (uint32_t)min(kT, p.sf_tiles - ks * kT) * 512;
                    mbar_arrive_expect_tx(&sf_full[stage], (a_here ? sfa_bytes : 0) + 2 * kT * 512);
                    if (a_here)
                        bulk_load(smem + kOffSfa + stage * kSfaBytes,
                                  p.sfa + band_a * p.sfa_band_bytes + (int64_t)ks * kT * 512, sfa_bytes, &sf_full[stage],
                                  pol);
                    tma_load_2d(smem + kOffSfb + stage * kSfbBytes, &tmSfb, &sf_full[stage], ks * kT * 64, t.nb * 2, pol);
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) { stage = 0; phase ^= 1; }
                }
            }
            for (int s = 0; s < kStages; ++s)
                if (issued_mask & (1u << s))
                    mbar_wait(&sf_full[s], (issued_phase >> s) & 1u, p.err_flag, kErrTimeout, p.wait_ns);
        } else if (warp == 1 && is_leader) {
            // ---------------------------------------------------- MMA (leader) --
            // The whole warp runs the loop (warp-uniform values); one elected
            // lane issues the MMAs and commits for both CTAs.
            const bool issuer = elect_one();
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            const uint32_t a_base = smem_u32(smem + kOffA);
            const uint32_t b_base = smem_u32(smem + kOffB);
            const uint32_t idesc = idesc_nvf4(kTileM, kTileN);
            bool ok = true;
            for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
                if (!__all_sync(~0u, mbar_wait(tmem_empty, acc_phase ^ 1, p.err_flag, kErrTimeout, p.wait_ns)))
                    break;
                tc_fence_after_sync();
                for (int ks = 0; ks < num_ks; ++ks) {
                    // the stage's scales in both CTAs' TMEM, its operands in both
                    // CTAs' shared memory
                    if (!__all_sync(~0u, mbar_wait(&sf_ready[stage], phase, p.err_flag, kErrTimeout, p.wait_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const int kcount = min(4, p.num_k64 - ks * 4);
                    const uint32_t sf_col = tmem + kTmemSf + stage * kSfColsPerStage;
                    const uint64_t adesc = smem_desc_sw128(a_base + stage * kABytes);
                    const uint64_t bdesc = smem_desc_sw128(b_base + stage * kBBytes);
                    if (issuer) {
                        for (int kk = 0; kk < kcount; ++kk) {
                            const uint64_t ad = adesc + (uint64_t)(kk * 2), bd = bdesc + (uint64_t)(kk * 2);
                            if constexpr (kMx)      // two UE8M0 scales per row and K-step: half a scale word
                                tc_mma_pair_mxf4(tmem, ad, bd, idesc_mxf4(kTileM, kTileN, (kk & 1) * 2),
                                                 sf_col + (kk >> 1) * 4, sf_col + 8 + (kk >> 1) * 8, (ks | kk) != 0);
                            else
                                tc_mma_pair_nvf4(tmem, ad, bd, idesc, sf_col + kk * 4, sf_col + 16 + kk * 8,
                                                 (ks | kk) != 0);
                        }
                        tc_commit_pair_multicast(&empty[stage], kBothCtas);
                    }
                    if (++stage == kStages) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if (issuer) tc_commit_pair_multicast(tmem_full, kBothCtas);
                __syncwarp();
                acc_phase ^= 1;
            }
            if (issuer) tc_commit_pair(mma_done);
            __syncwarp();
            mbar_wait(mma_done, 0, p.err_flag, kErrTimeout, p.wait_ns);
        }
    }

    tc_fence_before_sync();
    __syncwarp();                       // reconverge the role lanes before the aligned cluster barrier
    cluster_sync_all();                 // no peer access to this CTA's smem or TMEM after this point
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmParams &p_in, const uint8_t *a, const uint8_t *w, int num_sms, cudaStream_t s,
                             const char **why, bool dependent)
{
    static int configured_device = -1;
    static int max_pairs = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(gemm_nvf4_pair_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_nvf4_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t probe = {};
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        probe.gridDim = dim3(2 * (num_sms / 2), 1, 1);
        probe.blockDim = dim3(kThreads, 1, 1);
        probe.dynamicSmemBytes = kSmemBytes;
        probe.attrs = &attr;
        probe.numAttrs = 1;
        int clusters = 0;
        e = cudaOccupancyMaxActiveClusters(&clusters, gemm_nvf4_pair_kernel<false>, &probe);
        if (e != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            clusters = num_sms / 2;
        }
        max_pairs = clusters;
        configured_device = dev;
    }
    if (p_in.splits != 1) {
        *why = "the CTA-pair GEMM does not split K";
        return cudaErrorInvalidValue;
    }
    GemmParams p = p_in;
    p.num_m_blk = (p.m + kTileM - 1) / kTileM;
    CUtensorMap tmA, tmB, tmSfb, tmOut;
    const uint64_t row_bytes = (uint64_t)p.kp / 2;
    if (!make_operand_map(&tmA, a, row_bytes, (uint64_t)p.m, kRowsCta) ||
        !make_operand_map(&tmB, w, row_bytes, (uint64_t)p.n_w, kRowsCta)) {
        *why = "cuTensorMapEncodeTiled failed for an FP4 operand";
        return cudaErrorInvalidValue;
    }
    const uint32_t sf_box = (uint32_t)(p.mx ? kSfTilesPerStage<true> : kSfTilesPerStage<false>) * 64;
    if (!make_scale_bands_map(&tmSfb, p.sfb, (uint64_t)p.sfb_band_bytes, (uint64_t)(p.n_w + 127) / 128, sf_box)) {
        *why = "cuTensorMapEncodeTiled failed for the weight scales";
        return cudaErrorInvalidValue;
    }
    if (!make_output_map_sw128(&tmOut, p.out, (uint64_t)p.n_out, (uint64_t)p.m, (uint64_t)p.ldo)) {
        *why = "cuTensorMapEncodeTiled failed for the output";
        return cudaErrorInvalidValue;
    }
    const int tiles = p.num_m_blk * p.num_n_blk;
    const int pairs = tiles < max_pairs ? tiles : max_pairs;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 2;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attrs;
    cfg.numAttrs = dependent ? 2 : 1;
    return p.mx ? cudaLaunchKernelEx(&cfg, gemm_nvf4_pair_kernel<true>, tmA, tmB, tmSfb, tmOut, p)
                : cudaLaunchKernelEx(&cfg, gemm_nvf4_pair_kernel<false>, tmA, tmB, tmSfb, tmOut, p);
}

}  // namespace nvfp4
