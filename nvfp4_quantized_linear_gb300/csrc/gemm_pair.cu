// Block-scaled FP4 GEMM on CTA pairs (tcgen05 cta_group::2), for m > 128.
//
// Same operation as gemm.cu (page "TorchNvFp4LinearKernel", vLLM PR #53319,
// section 关键源码片段: _scaled_mm, * alpha, slice, + bias), with each output
// tile of 256 x 256 computed by a cluster of two CTAs on two SMs:
//   - CTA r (r = 0, 1) loads A rows [128r, 128r+128) of the tile and B rows
//     [128r, 128r+128) of the tile (its half of N), plus the scale tiles of its
//     A band and of both B bands, into a 5-stage shared-memory ring;
//   - the leader CTA (r = 0) issues everything on the tensor cores for both:
//     tcgen05.cp.cta_group::2 moves each CTA's scale tiles into that CTA's
//     TMEM, tcgen05.mma.cta_group::2 (M=256, N=256, K=64) accumulates each
//     CTA's 128 rows x 256 columns in that CTA's TMEM, and the commits
//     multicast to both CTAs' barriers;
//   - the peer CTA's copy completions reach the leader through a relay thread
//     that arrives on a leader barrier at cluster scope;
//   - each CTA's four epilogue warps drain its own accumulator, arrive on the
//     leader's "accumulator free" barrier and store their rows.
// Per SM and K-step this moves 8 KB of operand tiles instead of 12 KB, and the
// scale copies and MMAs are issued once per pair.  Every mbarrier wait is
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
constexpr int kTileN = 256;
constexpr int kRowsCta = 128;
constexpr int kBKBytes = 128;                   // 256 FP4 elements of K per stage
constexpr int kStages = 5;
constexpr uint32_t kABytes = kRowsCta * kBKBytes;     // 16 KB: this CTA's A rows
constexpr uint32_t kBBytes = kRowsCta * kBKBytes;     // 16 KB: this CTA's half of B
constexpr uint32_t kSfaBytes = 4 * 512;               // this CTA's A band, 4 K-steps
constexpr uint32_t kSfbBytes = 2 * 4 * 512;           // both B bands of the tile
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + kStages * kABytes;
constexpr uint32_t kOffSfa = kOffB + kStages * kBBytes;
constexpr uint32_t kOffSfb = kOffSfa + kStages * kSfaBytes;
constexpr uint32_t kOffBias = kOffSfb + kStages * kSfbBytes;   // per epilogue warp: one tile of bias
constexpr uint32_t kOffBar = kOffBias + 4 * kTileN * 2;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSf = 256;
constexpr uint32_t kSfColsPerStage = 48;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kThreads = 256;
constexpr int kEpiWarp0 = 4;
constexpr int kEpiWarps = 4;
constexpr int kCopiers = 2;                     // lane 0 of warps 2 and 3 (leader): two K-steps each

// Copier index of a thread (-1 if it does not copy scales).  The copiers sit
// in different warps: a warp issues a tcgen05 instruction for one lane only.
__device__ __forceinline__ int copier_of(int warp, int lane)
{
    return lane == 0 ? (warp == 2 ? 0 : warp == 3 ? 1 : -1) : -1;
}
constexpr uint16_t kBothCtas = 0x3;

static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kTmemSf + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");

__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar);   // this CTA's copies landed
    uint64_t *empty = full + kStages;                                 // the pair's MMAs released the stage
    uint64_t *peer_full = empty + kStages;                            // (leader) the peer's copies landed
    uint64_t *sf_ready = peer_full + kStages;                         // (leader) scales are in both TMEMs
    uint64_t *tmem_full = sf_ready + kStages;                         // accumulator complete
    uint64_t *tmem_empty = tmem_full + 1;                             // (leader) both CTAs drained it
    uint64_t *mma_done = tmem_empty + 1;
    uint64_t *cp_done = mma_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(cp_done + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&peer_full[s], 1);
            mbar_init(&sf_ready[s], kCopiers);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, 2 * kEpiWarps);
        mbar_init(mma_done, 1);
        mbar_init(cp_done, kCopiers);
        fence_mbarrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 2) {
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

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------------ producer --
        const uint64_t pol = l2_policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_phase = 0;
        bool ok = true;
        for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
            const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk);
            const int band_a = t.mb * 2 + (int)rank;
            const bool a_here = band_a < a_bands;
            const int n_rows = min(kTileN, p.n_out - t.nb * kTileN);
            const int halves = n_rows > 128 ? 2 : 1;
            for (int ks = 0; ks < num_ks; ++ks) {
                if (!mbar_wait_cluster(&empty[stage], phase ^ 1, p.err_flag, kErrTimeout, kWaitNs)) { ok = false; break; }
                const int kcount = min(4, p.num_k64 - ks * 4);
                const uint32_t sf_bytes = (uint32_t)kcount * 512;
                mbar_arrive_expect_tx(&full[stage], kABytes + kBBytes + sf_bytes * ((a_here ? 1 : 0) + halves));
                tma_load_2d(smem + kOffA + stage * kABytes, &tmA, &full[stage], ks * kBKBytes, band_a * kRowsCta, pol);
                tma_load_2d(smem + kOffB + stage * kBBytes, &tmB, &full[stage], ks * kBKBytes,
                            t.nb * kTileN + (int)rank * kRowsCta, pol);
                if (a_here)
                    bulk_load(smem + kOffSfa + stage * kSfaBytes, p.sfa + band_a * p.sfa_band_bytes + (int64_t)ks * 2048,
                              sf_bytes, &full[stage], pol);
                for (int h = 0; h < halves; ++h)
                    bulk_load(smem + kOffSfb + stage * kSfbBytes + h * 2048,
                              p.sfb + (t.nb * 2 + h) * p.sfb_band_bytes + (int64_t)ks * 2048, sf_bytes, &full[stage],
                              pol);
                issued_mask |= 1u << stage;
                issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
        }
        for (int s = 0; s < kStages; ++s)
            if (issued_mask & (1u << s))
                mbar_wait(&full[s], (issued_phase >> s) & 1u, p.err_flag, kErrTimeout, kWaitNs);
    } else if (copier_of(warp, lane) >= 0 && (leader || warp == 3)) {
        // -------------------- scale copiers (leader) / relay thread (peer) --
        // In the leader, copier c moves K-steps 2c and 2c+1 of each stage's
        // scale tiles into both CTAs' TMEM (tcgen05.cp.cta_group::2) once both
        // CTAs' copies have landed, and commits to sf_ready[stage] (two arrivals).  In the
        // peer, one thread relays "this CTA's stage landed" to the leader.
        const int cidx = copier_of(warp, lane);
        int stage = 0;
        uint32_t phase = 0;
        const uint32_t sfa_base = smem_u32(smem + kOffSfa);
        const uint32_t sfb_base = smem_u32(smem + kOffSfb);
        const uint32_t leader_peer_full = mapa_shared(peer_full, 0);
        bool ok = true;
        for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
            const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk);
            const int n_rows = min(kTileN, p.n_out - t.nb * kTileN);
            const int halves = n_rows > 128 ? 2 : 1;
            for (int ks = 0; ks < num_ks; ++ks) {
                if (!mbar_wait(&full[stage], phase, p.err_flag, kErrTimeout, kWaitNs)) { ok = false; break; }
                if (!leader) {
                    mbar_arrive_cluster(leader_peer_full + stage * (uint32_t)sizeof(uint64_t));
                } else {
                    if (!mbar_wait_cluster(&peer_full[stage], phase, p.err_flag, kErrTimeout, kWaitNs)) { ok = false; break; }
                    tc_fence_after_sync();
                    const int kcount = min(4, p.num_k64 - ks * 4);
                    const uint32_t sf_col = tmem + kTmemSf + stage * kSfColsPerStage;
                    for (int kk = 2 * cidx; kk < 2 * cidx + 2 && kk < kcount; ++kk) {
                        tc_cp_pair_32x128b_warpx4(sf_col + kk * 4, smem_desc_sf(sfa_base + stage * kSfaBytes + kk * 512));
                        for (int h = 0; h < halves; ++h)
                            tc_cp_pair_32x128b_warpx4(sf_col + 16 + kk * 8 + h * 4,
                                                      smem_desc_sf(sfb_base + stage * kSfbBytes + h * 2048 + kk * 512));
                    }
                    tc_commit_pair(&sf_ready[stage]);
                }
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
        }
        if (leader) {
            tc_commit_pair(cp_done);
            mbar_wait(cp_done, 0, p.err_flag, kErrTimeout, kWaitNs);
        }
    } else if (warp == 1 && lane == 0 && leader) {
        // ---------------------------------------------------- MMA (leader) --
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        const uint32_t a_base = smem_u32(smem + kOffA);
        const uint32_t b_base = smem_u32(smem + kOffB);
        const uint32_t idesc = idesc_nvf4(kTileM, kTileN);
        bool ok = true;
        for (int tile = pair_id; tile < num_tiles && ok; tile += num_pairs) {
            if (!mbar_wait_cluster(tmem_empty, acc_phase ^ 1, p.err_flag, kErrTimeout, kWaitNs)) break;
            tc_fence_after_sync();
            for (int ks = 0; ks < num_ks; ++ks) {
                if (!mbar_wait(&sf_ready[stage], phase, p.err_flag, kErrTimeout, kWaitNs)) { ok = false; break; }
                tc_fence_after_sync();
                const int kcount = min(4, p.num_k64 - ks * 4);
                const uint32_t sf_col = tmem + kTmemSf + stage * kSfColsPerStage;
                const uint64_t adesc = smem_desc_sw128(a_base + stage * kABytes);
                const uint64_t bdesc = smem_desc_sw128(b_base + stage * kBBytes);
                for (int kk = 0; kk < kcount; ++kk)
                    tc_mma_pair_nvf4(tmem, adesc + (uint64_t)(kk * 2), bdesc + (uint64_t)(kk * 2), idesc,
                                     sf_col + kk * 4, sf_col + 16 + kk * 8, (ks | kk) != 0);
                tc_commit_pair_multicast(&empty[stage], kBothCtas);
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            tc_commit_pair_multicast(tmem_full, kBothCtas);
            acc_phase ^= 1;
        }
        tc_commit_pair(mma_done);
        mbar_wait(mma_done, 0, p.err_flag, kErrTimeout, kWaitNs);
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
        // ------------------------------------------------------ epilogue --
        const int q = warp & 3;
        uint16_t *s_bias = reinterpret_cast<uint16_t *>(smem + kOffBias) + (warp - kEpiWarp0) * kTileN;
        const uint32_t leader_tmem_empty = mapa_shared(tmem_empty, 0);
        const float alpha = __ldg(p.alpha);
        uint32_t acc_phase = 0;
        for (int tile = pair_id; tile < num_tiles; tile += num_pairs) {
            const Tile t = tile_coord(tile, p.num_m_blk, p.num_n_blk);
            const int n_rows = min(kTileN, p.n_out - t.nb * kTileN);
            const int col_base = t.nb * kTileN;
            if (p.bias != nullptr) {
                __syncwarp();
                for (int j = lane; j < kTileN; j += 32)
                    s_bias[j] = (j < n_rows) ? p.bias[col_base + j] : (uint16_t)0;
                __syncwarp();
            }
            if (!mbar_wait_cluster(tmem_full, acc_phase, p.err_flag, kErrTimeout, kWaitNs)) break;
            tc_fence_after_sync();
            uint32_t packed[kTileN / 2];
#pragma unroll
            for (int ch = 0; ch < kTileN / 32; ++ch) {
                if (ch * 32 < n_rows) {
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
            if (lane == 0) mbar_arrive_cluster(leader_tmem_empty);
            acc_phase ^= 1;

            const int64_t row = (int64_t)t.mb * kTileM + (int64_t)rank * kRowsCta + q * 32 + lane;
            if (row < p.m) {
                uint16_t *orow = p.out + row * p.ldo + col_base;
#pragma unroll
                for (int v = 0; v < kTileN / 8; ++v) {
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
    __syncwarp();                       // reconverge the role lanes before the aligned cluster barrier
    cluster_sync_all();                 // no peer access to this CTA's smem or TMEM after this point
    tc_fence_after_sync();
    if (warp == 2) tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmParams &p_in, const uint8_t *a, const uint8_t *w, int num_sms, cudaStream_t s,
                             const char **why)
{
    static int configured_device = -1;
    static int max_pairs = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(gemm_nvf4_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
        e = cudaOccupancyMaxActiveClusters(&clusters, gemm_nvf4_pair_kernel, &probe);
        if (e != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            clusters = num_sms / 2;
        }
        max_pairs = clusters;
        configured_device = dev;
    }
    GemmParams p = p_in;
    p.num_m_blk = (p.m + kTileM - 1) / kTileM;
    CUtensorMap tmA, tmB;
    const uint64_t row_bytes = (uint64_t)p.kp / 2;
    if (!make_operand_map(&tmA, a, row_bytes, (uint64_t)p.m, kRowsCta) ||
        !make_operand_map(&tmB, w, row_bytes, (uint64_t)p.n_w, kRowsCta)) {
        *why = "cuTensorMapEncodeTiled failed for an FP4 operand";
        return cudaErrorInvalidValue;
    }
    const int tiles = p.num_m_blk * p.num_n_blk;
    const int pairs = tiles < max_pairs ? tiles : max_pairs;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_nvf4_pair_kernel, tmA, tmB, p);
}

}  // namespace nvfp4
