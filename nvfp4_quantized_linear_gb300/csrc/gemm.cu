// Block-scaled FP4 GEMM with fused epilogue on the sm_103a tensor cores.
//
// Page "TorchNvFp4LinearKernel" (vLLM PR #53319), section 关键源码片段:
// apply_weights computes torch._scaled_mm(x_fp4, weight.t(), scale_a, scale_b,
// out_dtype), then out * alpha, slice_nvfp4_output, + bias.  Here that is one
// kernel:
//     out[m, n] = bf16( alpha * sum_k A[m,k] B[n,k] + bias[n] ),  n < n_out,
// A, B packed E2M1 (K-major) with one UE4M3 scale per 16 K-elements.
//
// Design (one CTA per SM, persistent over output tiles of 128 x 256; 16 warps):
//   warps 0, 3  TMA producers (lane 0 of each): warp 0 the A tile 128 x 256
//               FP4 (16 KB) and its scale tile, warp 3 the B tile 256 x 256 FP4
//               (32 KB) and its two scale tiles, 128-byte swizzled, into a
//               4-stage shared-memory ring.  Only warp 0 waits for the
//               preceding grid (programmatic dependent launch), so the weights
//               stream while the activation quantizer finishes;
//   warp 1      allocates / frees the 512 TMEM columns; lane 0 issues the
//               MMAs: 4 x tcgen05.mma (M=128, N=256, K=64, kind::mxf4nvf4,
//               scale_vec::4X) per stage into a 128 x 256 fp32 TMEM tile;
//               tcgen05.commit releases the smem stage / signals the epilogue;
//   warps 4..7  one per TMEM lane quarter: stage each landed stage's scale
//               tiles into TMEM with tcgen05.st, keeping the tensor pipe for
//               the MMAs alone;
//   warps 8..15 epilogue, two per TMEM lane quarter (128 columns each):
//               tcgen05.ld of finished accumulators, fma with alpha and bias, bf16 round into
//               registers, release of the TMEM tile, then masked stores
//               (rows < m, cols < n_out) that overlap the next tile's MMAs.
// Split-K (small m): the K ranges of a tile run as the CTAs of one thread-block
// cluster, one range each; the drain writes the raw fp32 sums into the CTA's
// own shared memory, and after a cluster barrier every CTA sums its share of
// the tile's columns over all ranks' partials (distributed shared memory, rank
// order) and applies alpha, bias and the bf16 rounding.
// Registers are moved between the warpgroups at start (setmaxnreg).
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
#include "quant_core.cuh"

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
constexpr uint32_t kOffBias = kOffSfb + kStages * kSfbBytes;   // two tiles of bias (bf16), double-buffered
constexpr uint32_t kOutChunkBytes = 32 * 16 * 2;              // output staging: 32 rows x 16 columns bf16
constexpr uint32_t kOffOut = kOffBias + 2 * kBN * 2;          // per epilogue warp: one staging chunk
constexpr uint32_t kOffBar = kOffOut + 8 * kOutChunkBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;      // + alignment slack
constexpr int kFusedMaxRows = 16;                          // the fused linear's largest m
constexpr int kXSliceRows = 16;                             // rows of the fused linear's activation copies
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemSf = 256;
constexpr uint32_t kSfColsPerStage = 48;
constexpr int kThreads = 512;                 // four warpgroups
constexpr int kSfWarp0 = 4;                   // warps 4..7: scale staging, lane quarter warp % 4
constexpr int kEpiWarp0 = 8;                  // warps 8..15: epilogue, lane quarter warp % 4,
constexpr int kEpiWarps = 8;                  // columns [128 h, 128 h + 128) for h = (warp - 8) / 4
constexpr int kEpiCols = kBN / 2;
// Registers per thread after the reallocation at kernel start (launched with
// 65536 / 512 = 128): 128 x (56 + 96 + 2 x 176) = 64512 <= 512 x 128 = 65536.
constexpr uint32_t kRegsCtl = 56, kRegsSf = 96, kRegsEpi = 176;
static_assert(128 * (kRegsCtl + kRegsSf + 2 * kRegsEpi) <= kThreads * 128, "register reallocation budget");

static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kOffOut % 128 == 0, "TMA store sources are 128-byte aligned");

// Work item of a persistent CTA: output tile, K-stage range [ks0, ks1) and,
// for a grouped GEMM, the group of the tile's row band (-1: no group, skip).
struct Work {
    Tile t;
    int split, ks0, ks1, g;
};

// Group of the 128-row band mb: the last g with offsets[g] <= 128 mb, or -1
// for a band outside [offsets[0], offsets[num_groups]).
__device__ __forceinline__ int group_of_band(const GemmParams &p, int mb)
{
    const int row = mb * 128;
    if (row < __ldg(p.group_offsets) || row >= __ldg(p.group_offsets + p.num_groups)) return -1;
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(p.group_offsets + mid) <= row) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ Work work_of(int item, const GemmParams &p, int num_ks)
{
    // split-K: consecutive items (the CTAs of one cluster) are the K ranges
    // of one tile
    Work w;
    w.split = item % p.splits;
    w.t = tile_coord(item / p.splits, p.num_m_blk, p.num_n_blk);
    w.ks0 = w.split * p.stages_per_split;
    w.ks1 = min(num_ks, w.ks0 + p.stages_per_split);
    w.g = p.group_offsets != nullptr ? group_of_band(p, w.t.mb) : 0;
    return w;
}

// Split-K partial sums in shared memory: row r of the tile at r * kPartLd
// floats (256 columns, padded by 4 so that the 32 rows a warp writes at once
// fall on different banks).
constexpr int kPartLd = kBN + 4;
// Up to this many rows below m in an epilogue warp's 32, the rows are written
// straight from registers instead of through the staging buffer and the TMA.
constexpr int kDirectStoreRows = 16;
static_assert((uint32_t)kBM * kPartLd * 4 <= kOffSfa, "the partials fit in the idle operand ring");

// Cluster split-K finish, by the 256 epilogue threads of CTA `rank` of the
// tile's p.splits CTAs.  The tile's valid 4-column groups (rows r < m,
// columns < n_out, row-major) are cut into p.splits equal ranges; for each
// group of its range this CTA forms out[r, c..c+3] = bf16(alpha * (((part_0 +
// part_1) + part_2) + ...) + bias[c]), the ranks' partials added in rank order
// (deterministic), its own from its shared memory and the others' through
// distributed shared memory, all loads of a group issued before the sum.
// Equal ranges rather than whole column chunks per rank: at m = 128 the
// distributed-shared-memory reads (m x 1 KB per rank) set the reduction's
// time, and chunks of 32 columns gave two ranks of six twice the reads.
__device__ __forceinline__ void cluster_reduce(const GemmParams &p, const Tile &t, uint32_t part_smem, uint32_t rank,
                                               int tid)
{
    const float alpha = p.alpha != nullptr ? __ldg(p.alpha) : 1.0f;
    const int rows = min(kBM, p.m - t.mb * kBM);
    const int cols = min(kBN, p.n_out - t.nb * kBN);
    const int quads = (cols + 3) >> 2;
    const int items = rows * quads;
    const int i0 = (int)((int64_t)items * rank / p.splits);
    const int i1 = (int)((int64_t)items * (rank + 1) / p.splits);
    for (int i = i0 + tid; i < i1; i += kEpiWarps * 32) {
        const int r = i / quads;
        const int col = (i - r * quads) * 4;                        // tile column
        const int gcol = t.nb * kBN + col;
        const uint32_t off = part_smem + (uint32_t)(r * kPartLd + col) * 4;
        float4 v[kMaxSplits];
#pragma unroll
        for (int sp = 0; sp < kMaxSplits; ++sp)
            if (sp < p.splits) {
                if (sp == (int)rank) {
                    const uint4 u = ld_shared_v4(off);
                    v[sp] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                        __uint_as_float(u.w));
                } else {
                    v[sp] = ld_dsmem_v4(mapa_shared_addr(off, (uint32_t)sp));
                }
            }
        float4 acc = v[0];
#pragma unroll
        for (int sp = 1; sp < kMaxSplits; ++sp)
            if (sp < p.splits) { acc.x += v[sp].x; acc.y += v[sp].y; acc.z += v[sp].z; acc.w += v[sp].w; }
        const float a[4] = {acc.x, acc.y, acc.z, acc.w};
        uint32_t h[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float b = (p.bias != nullptr && gcol + e < p.n_out) ? __uint_as_float((uint32_t)p.bias[gcol + e] << 16)
                                                                     : 0.0f;
            h[e] = bf16_bits_rn(__fmaf_rn(a[e], alpha, b));
        }
        uint16_t *o = p.out + (int64_t)(t.mb * kBM + r) * p.ldo + gcol;
        if (gcol + 4 <= p.n_out) {      // 8-byte aligned: rows start on 16 bytes, gcol % 4 == 0
            *reinterpret_cast<uint2 *>(o) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (gcol + e < p.n_out) o[e] = (uint16_t)h[e];
        }
    }
}

// The activation side of the fused small-m linear, run by the eight epilogue
// warps (idle during the mainloop) before each work item's epilogue: for every
// stage of the work item, the weight producer has fetched the stage's 256
// columns of the m <= kFusedMaxRows activation rows (bf16, one 2-D TMA of 16
// rows x 256 columns, zeros past m and k) into bytes [2 KB, 10 KB) of the
// stage's own A tile -- rows 16..127 of that tile, which the MMA reads but
// whose output rows are never stored.  Epilogue warp w quantizes block
// 32 w + lane of the m x 16 blocks exactly as quant_kernel does into the
// tile's first 16 rows (128-byte rows with the TMA's 128-byte swizzle, the
// layout of the MMA's descriptor) and its scale into the stage's four scale
// tiles, whose rows >= m were zeroed once at kernel start (their A bytes are
// finite FP4 codes whatever they hold).  Then the async-proxy fence and the
// warp's arrival on the stage's `full` barrier (eight of its nine).  One warp
// quantizing every block fell behind the weight stream from m = 8 on.  The
// slice's copy is requested by the weight producer together with the stage's
// weights, as soon as the stage frees (up to kStages ahead): a warp that
// fetched each slice itself after quantizing the previous one paid the copy's
// round trip once per stage.  inv = gs / e4m3(code) with the IEEE division,
// the value quant_kernel's table holds.  kMx (MXFP4, quant_mx_kernel's
// arithmetic): a lane holds half of a 32-element block, the two halves' maxima
// meet through one shuffle, and the even lane stores the block's UE8M0 code
// (scale column j / 2 of the stage, two scale tiles).  Returns false when a
// wait expired.
constexpr uint32_t kXSliceOff = 16 * 128;                    // rows 16.. of an A tile
constexpr uint32_t kXSliceBytes = kXSliceRows * 256 * 2;     // 16 rows x 256 bf16
static_assert(kXSliceOff + kXSliceBytes <= kABytes, "the activation slice fits in the A tile's spare rows");
static_assert(kFusedMaxRows * 16 <= kEpiWarps * 32, "one 16-element block per epilogue lane and stage");

template <bool kMx>
__device__ __forceinline__ bool fused_quant_stages(const GemmParams &p, uint8_t *smem, uint64_t *full,
                                                   uint64_t *x_full, const Work &wk, int &stage, uint32_t &phase,
                                                   float gs, int wq, int lane)
{
    const QuantParams &q = p.quant;
    for (int ks = wk.ks0; ks < wk.ks1; ++ks) {
        if (!__all_sync(~0u, mbar_wait(&x_full[stage], phase, p.err_flag, kErrTimeout, p.wait_ns))) return false;
        const uint32_t a_dst = smem_u32(smem + kOffA + stage * kABytes);
        const uint32_t x_src = a_dst + kXSliceOff;
        const uint32_t sf_dst = smem_u32(smem + kOffSfa + stage * kSfaBytes);
        const int b = wq * 32 + lane;
        // warps with any block of the m rows; their lanes past it (zero rows
        // of the slice) compute too, for the shuffle, but store nothing
        if (wq * 32 < q.m * 16) {
            const int r = b >> 4, j = b & 15;
            quant_core::Raw16 raw;
            raw.a = ld_shared_v4(x_src + (uint32_t)r * 512 + (uint32_t)j * 32);
            raw.b = ld_shared_v4(x_src + (uint32_t)r * 512 + (uint32_t)j * 32 + 16);
            float v0[8], v1[8];
            quant_core::unpack8(raw.a, v0);
            quant_core::unpack8(raw.b, v1);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(v0[i]), fabsf(v1[i])));
            uint32_t sf, sf_off;
            float inv;
            if constexpr (kMx) {
                amax = fmaxf(amax, __shfl_xor_sync(~0u, amax, 1));   // the block's other half
                sf = quant_core::mx_scale_code(amax);
                inv = quant_core::mx_scale_mul(sf);
                const int jb = j >> 1;                               // scale column of the stage
                sf_off = (uint32_t)(jb >> 2) * 512 + (uint32_t)(r & 31) * 16 + (uint32_t)((r >> 5) & 3) * 4 +
                         (uint32_t)(jb & 3);
            } else {
                sf = cvt_e4m3x2(0.0f, div6_rn(__fmul_rn(amax, gs))) & 0x7Fu;
                const float d = e4m3_to_f32(sf);
                inv = (d == 0.0f) ? 0.0f : __fdiv_rn(gs, d);
                // scale column j of the stage: tile j / 4, the tiled layout inside it
                sf_off = (uint32_t)(j >> 2) * 512 + (uint32_t)(r & 31) * 16 + (uint32_t)((r >> 5) & 3) * 4 +
                         (uint32_t)(j & 3);
            }
            const uint32_t lo = quant_core::quant8(v0, inv), hi = quant_core::quant8(v1, inv);
            // packed bytes [8j, 8j + 8) of row r: 16-byte piece j / 2 of the
            // row, at piece (j / 2) ^ (r % 8) after the swizzle
            const uint32_t a_off = (uint32_t)(r >> 3) * 1024 + (uint32_t)(r & 7) * 128 +
                                   ((uint32_t)((j >> 1) ^ (r & 7)) << 4) + (uint32_t)(j & 1) * 8;
            if (b < q.m * 16) {
                asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a_dst + a_off), "r"(lo), "r"(hi) : "memory");
                if (!kMx || (lane & 1) == 0)
                    asm volatile("st.shared.u8 [%0], %1;" ::"r"(sf_dst + sf_off), "r"(sf) : "memory");
            }
        }
        fence_proxy_async_shared();                          // the MMA reads the A tile through the async proxy
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1; }
    }
    return true;
}

// kMx: MXFP4 operands (one UE8M0 scale per 32 K-elements, two 512-byte scale
// tiles per band and stage, scale_vec::2X MMAs); otherwise NVFP4 (one UE4M3
// scale per 16 K-elements, four tiles per band and stage, scale_vec::4X).
// kFused: the fused small-m linear (m <= kFusedMaxRows, NVFP4 or with kMx
// MXFP4): no A tensor is read; the epilogue warps quantize each stage's slice
// of the activation p.quant.x (the body of quant_kernel, or quant_mx_kernel,
// for the stage's 256 columns of every row) straight into the stage's A tile
// and scale tiles in shared memory.
template <bool kMx, bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmX,
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
    uint64_t *bias_full = mma_done + 1;     // [2]
    uint64_t *bias_empty = bias_full + 2;   // [2]
    uint64_t *x_full = bias_empty + 2;      // [kStages] fused linear: the stage's activation slice landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(x_full + kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // the activation and the weight producer (fused: the weight
            // producer and the eight quantizing epilogue warps)
            mbar_init(&full[s], kFused ? 1 + kEpiWarps : 2);
            mbar_init(&empty[s], 1);
            mbar_init(&sf_ready[s], 4);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, kEpiWarps);
        mbar_init(mma_done, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bias_full[b], 1);
            mbar_init(&bias_empty[b], kEpiWarps);
        }
        if constexpr (kFused)
            for (int s = 0; s < kStages; ++s) mbar_init(&x_full[s], 1);
        fence_mbarrier_init();
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if constexpr (kFused) prefetch_tensormap(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if constexpr (kFused) {             // scale rows >= m stay zero in every stage
        for (uint32_t o = threadIdx.x * 16; o < kStages * kSfaBytes; o += kThreads * 16)
            st_shared_v4(smem_u32(smem + kOffSfa) + o, 0, 0, 0, 0);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int num_tiles = p.num_m_blk * p.num_n_blk * p.splits;     // work items
    const int num_ks = (p.num_k64 + 3) / 4;
    const int n_bands_w = (p.n_w + 127) / 128;

    // The next kernel on the stream, if launched as a programmatic dependent
    // (this library's quantizer or GEMM), may get resident now: it waits for
    // this grid before it reads anything.
    if (threadIdx.x == 0) griddep_launch_dependents();

    // Roles by warpgroup; each warpgroup first resizes its register file.
    if (warp >= kEpiWarp0) {
        setmaxnreg_inc<kRegsEpi>();
        // ------------------------------------------------------ epilogue --
        // Drain the finished 128 x 256 accumulator (this warp: TMEM lane
        // quarter warp % 4, one row per thread) into registers as packed bf16
        // with alpha and bias applied, hand the TMEM back to the MMA thread,
        // then store the rows (rows < m, columns < n_out) while the next
        // tile's MMAs run.  With split-K the drain writes raw fp32 sums.
        const int q = warp & 3;
        const int hcol = ((warp - kEpiWarp0) >> 2) * kEpiCols;    // this warp's first column of the tile
        const uint32_t acc = tmem + ((uint32_t)(q * 32) << 16) + hcol;
        const uint32_t out_stage = smem_u32(smem + kOffOut) + (warp - kEpiWarp0) * kOutChunkBytes;
        const bool use_bias = p.splits == 1 && p.bias != nullptr;
        const uint64_t out_policy = l2_policy_evict_first();   // the output is written once
        uint32_t acc_phase = 0;
        int it = 0;
        int q_stage = 0;                                        // fused linear: the quantized stages
        uint32_t q_phase = 0;
        float q_gs = 0.0f;
        if constexpr (kFused) {
            griddep_wait();                                     // x and gs may be the preceding kernel's output
            if constexpr (!kMx) q_gs = __ldg(p.quant.gs);       // (MXFP4 has no global scale)
        }
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
            const Work wk = work_of(tile, p, num_ks);
            if (wk.g < 0) continue;                             // every role skips the same tiles
            // (a timeout drill quantizes nothing: its stages never fill)
            if (kFused && !p.drill &&
                !fused_quant_stages<kMx>(p, smem, full, x_full, wk, q_stage, q_phase, q_gs, warp - kEpiWarp0, lane))
                break;
            const float alpha = p.alpha != nullptr ? __ldg(p.alpha + wk.g) : 1.0f;
            const Tile t = wk.t;
            const int n_cols = min(kEpiCols, p.n_out - t.nb * kBN - hcol);   // may be <= 0
            const int col_base = t.nb * kBN + hcol;
            const uint16_t *s_bias = reinterpret_cast<const uint16_t *>(smem + kOffBias) + (it & 1) * kBN + hcol;
            if (use_bias &&
                !__all_sync(~0u, mbar_wait(&bias_full[it & 1], (it >> 1) & 1, p.err_flag, kErrTimeout, p.wait_ns)))
                break;
            if (!__all_sync(~0u, mbar_wait(tmem_full, acc_phase, p.err_flag, kErrTimeout, p.wait_ns))) break;
            tc_fence_after_sync();
            acc_phase ^= 1;
            const int64_t row = (int64_t)t.mb * kBM + q * 32 + lane;
            const int row0 = t.mb * kBM + q * 32;
            // columns of this warp's slice that hold output, 0 when all of
            // its 32 rows are at or past m (small m: most warps)
            const int cols_here = p.m > row0 ? n_cols : 0;
            uint32_t r0[32], r1[32];

            if (p.splits > 1) {
                // split-K: raw fp32 sums of this K range for rows < m, into this
                // CTA's shared memory (the operand ring: every stage of the
                // CTA's one work item has been consumed)
                const uint32_t dst = smem_u32(smem) + (uint32_t)((row - t.mb * kBM) * kPartLd + hcol) * 4;
                if (cols_here > 0) tmem_ld_32cols(acc, r0);
#pragma unroll
                for (int ch = 0; ch < kEpiCols / 32; ++ch) {
                    uint32_t(&cur)[32] = (ch & 1) ? r1 : r0;
                    uint32_t(&nxt)[32] = (ch & 1) ? r0 : r1;
                    if (ch * 32 < cols_here) {                  // uniform across the warp
                        tmem_ld_wait_regs(cur);
                        if (ch + 1 < kEpiCols / 32 && (ch + 1) * 32 < cols_here)
                            tmem_ld_32cols(acc + (ch + 1) * 32, nxt);
                        if (row < p.m) {
#pragma unroll
                            for (int v = 0; v < 8; ++v)
                                st_shared_v4(dst + (uint32_t)(ch * 32 + 4 * v) * 4, cur[4 * v], cur[4 * v + 1],
                                             cur[4 * v + 2], cur[4 * v + 3]);
                        }
                    }
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(tmem_empty);
                continue;
            }

            uint32_t packed[kEpiCols / 2];
            if (cols_here > 0) tmem_ld_32cols(acc, r0);
#pragma unroll
            for (int ch = 0; ch < kEpiCols / 32; ++ch) {
                uint32_t(&cur)[32] = (ch & 1) ? r1 : r0;
                uint32_t(&nxt)[32] = (ch & 1) ? r0 : r1;
                if (ch * 32 < cols_here) {                      // uniform across the warp
                    tmem_ld_wait_regs(cur);
                    if (ch + 1 < kEpiCols / 32 && (ch + 1) * 32 < cols_here) tmem_ld_32cols(acc + (ch + 1) * 32, nxt);
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        float b0 = 0.0f, b1 = 0.0f;
                        if (use_bias) {
                            const uint32_t bw = *reinterpret_cast<const uint32_t *>(s_bias + ch * 32 + j);
                            b0 = __uint_as_float(bw << 16);
                            b1 = __uint_as_float(bw & 0xFFFF0000u);
                        }
                        packed[ch * 16 + j / 2] = bf16x2_rn(__fmaf_rn(__uint_as_float(cur[j]), alpha, b0),
                                                            __fmaf_rn(__uint_as_float(cur[j + 1]), alpha, b1));
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(tmem_empty);
                if (use_bias) mbar_arrive(&bias_empty[it & 1]);
            }

            // A few rows (small m): each of their lanes writes its row from
            // registers, 16 bytes at a time (rows start on 16 bytes, col_base
            // % 128 == 0); no round trips through the staging buffer.
            const int rows_here = min(32, p.m - row0);
            if (cols_here > 0 && rows_here <= kDirectStoreRows) {
                if (lane < rows_here) {
                    uint16_t *o = p.out + (int64_t)(row0 + lane) * p.ldo + col_base;
#pragma unroll
                    for (int g = 0; g < kEpiCols / 8; ++g) {
                        if (8 * g + 8 <= cols_here) {
                            *reinterpret_cast<uint4 *>(o + 8 * g) =
                                make_uint4(packed[4 * g], packed[4 * g + 1], packed[4 * g + 2], packed[4 * g + 3]);
                        } else if (8 * g < cols_here) {
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                if (8 * g + e < cols_here)
                                    o[8 * g + e] = (uint16_t)(packed[4 * g + e / 2] >> (16 * (e & 1)));
                        }
                    }
                }
                continue;
            }

            // Store through shared memory and the TMA: 16-column chunks of this
            // warp's 32 rows x 128 columns; the TMA clips rows >= m and
            // columns >= n_out.  (Thread-per-row global stores would touch 32
            // rows per instruction and congest the SM's memory pipeline that
            // the MMA thread's barrier and issue traffic also uses.)
#pragma unroll
            for (int c = 0; c < kEpiCols / 16; ++c) {
                if (c * 16 < cols_here) {                       // uniform across the warp
                    if (lane == 0) bulk_wait_group_read<0>();   // the previous chunk's store has read the buffer
                    __syncwarp();
                    st_shared_v4(out_stage + lane * 32, packed[c * 8], packed[c * 8 + 1], packed[c * 8 + 2],
                                 packed[c * 8 + 3]);
                    st_shared_v4(out_stage + lane * 32 + 16, packed[c * 8 + 4], packed[c * 8 + 5],
                                 packed[c * 8 + 6], packed[c * 8 + 7]);
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmOut, out_stage, col_base + c * 16, row0, out_policy);
                        bulk_commit_group();
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();                    // all output written before the CTA exits
        if (p.splits > 1) {
            // Cluster split-K: the first barrier phase completes once every
            // rank's partials are in its shared memory (this warp's arrival
            // releases its own); then this CTA sums its share of the columns.
            // The second phase, whose wait follows below, keeps the partials
            // until every peer has read them.
            cluster_arrive_release();
            cluster_wait_acquire();
            cluster_reduce(p, work_of(blockIdx.x, p, num_ks).t, smem_u32(smem), cluster_ctarank(),
                           (int)threadIdx.x - kEpiWarp0 * 32);
            cluster_arrive_release();
        }
    } else if (warp >= kSfWarp0) {
        setmaxnreg_dec<kRegsSf>();
        // ----------------------------------------------- scale staging --
        // When a stage lands, copy its scale tiles from shared memory into the
        // stage's TMEM columns with tcgen05.st (the tensor pipe's tcgen05.cp
        // would queue behind the MMAs) and arrive on sf_ready[stage].  The
        // tcgen05.cp 32x128b.warpx4 layout is reproduced: lane 32q + i of
        // the quarter q gets bytes [16i, 16i + 16) of each 512-byte tile.
        // A stage's columns are rewritten only after it landed again, i.e.
        // after the MMAs that read them completed and released the stage.
        const int q = warp & 3;
        const uint32_t sf_tmem = tmem + ((uint32_t)(q * 32) << 16) + kTmemSf;
        const uint32_t sfa_smem = smem_u32(smem + kOffSfa) + lane * 16;
        const uint32_t sfb_smem = smem_u32(smem + kOffSfb) + lane * 16;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const Work wk = work_of(tile, p, num_ks);
            if (wk.g < 0) continue;
            for (int ks = wk.ks0; ks < wk.ks1; ++ks) {
                ok = __all_sync(~0u, mbar_wait(&full[stage], phase, p.err_flag, kErrTimeout, p.wait_ns));
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
                        const uint4 v = ld_shared_v4(sfb_smem + stage * kSfbBytes + h * 2048 + j * 512);
                        uint32_t *d = b + j * 8 + h * 4;
                        d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
                    }
                // (tiles past the valid K-steps or B rows hold stale bytes; the
                // MMAs never read their columns)
                if constexpr (kMx) {
                    tmem_st_8cols(sf_tmem + stage * kSfColsPerStage, a);
                    tmem_st_16cols(sf_tmem + stage * kSfColsPerStage + 4 * kT, b);
                } else {
                    tmem_st_16cols(sf_tmem + stage * kSfColsPerStage, a);
                    tmem_st_32cols(sf_tmem + stage * kSfColsPerStage + 4 * kT, b);
                }
                tmem_st_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_ready[stage]);
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
        }
    } else {
        setmaxnreg_dec<kRegsCtl>();
        if (kFused && warp == 0) {
            // the fused linear reads no A tensor: the epilogue warps quantize it
        } else if ((warp == 0 || warp == 3) && lane == 0 && !p.drill) {   // (a timeout drill issues no copies)
            // ----------------------------------------------------- producers --
            // Two threads fill the ring, each with its half of every stage:
            // warp 0 the activation side (A tile + its scale tile), warp 3 the
            // weight side (B tile + the scale tiles of its two bands); each
            // arms the stage's `full` barrier (two arrivals) with its bytes.
            // One thread issuing all five copies of a stage took ~630 clocks,
            // longer than the stage's MMAs.  Only the activation side waits
            // for the preceding grid (the activation quantizer, when launched
            // as its programmatic dependent): the weights are not written by
            // it, so they stream while the quantizer finishes.
            const bool act_side = warp == 0;
            // weights are re-read by every 128-row band; with one band they stream once
            const uint64_t pol = act_side || p.num_m_blk > 1 ? l2_policy_evict_last() : l2_policy_evict_first();
            // The fused linear, a programmatic dependent of an arbitrary
            // kernel, waits on both sides: that kernel may write the weights.
            if (act_side || kFused) griddep_wait();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                const Work wk = work_of(tile, p, num_ks);
                if (wk.g < 0) continue;
                const Tile t = wk.t;
                const int b_row0 = wk.g * p.group_n + t.nb * kBN;          // weight rows of this tile
                const int b_band0 = b_row0 / 128;
                const int halves = min(kBN, p.n_out - t.nb * kBN) > 128 ? 2 : 1;
                for (int ks = wk.ks0; ks < wk.ks1; ++ks) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, p.err_flag, kErrTimeout, p.wait_ns)) { ok = false; break; }
                    constexpr int kT = kSfTilesPerStage<kMx>;
                    const uint32_t sf_bytes = (uint32_t)min(kT, p.sf_tiles - ks * kT) * 512;
                    if (act_side) {
                        mbar_arrive_expect_tx(&full[stage], kABytes + sf_bytes);
                        tma_load_2d(smem + kOffA + stage * kABytes, &tmA, &full[stage], ks * kBKBytes, t.mb * kBM, pol);
                        bulk_load(smem + kOffSfa + stage * kSfaBytes,
                                  p.sfa + t.mb * p.sfa_band_bytes + (int64_t)ks * kT * 512, sf_bytes, &full[stage], pol);
                    } else {
                        if constexpr (kFused) {
                            // the stage's activation slice for the fused linear's quantizing warps
                            // (every column tile's CTAs read the same slices: keep them in L2)
                            mbar_arrive_expect_tx(&x_full[stage], kXSliceBytes);
                            tma_load_2d(smem + kOffA + stage * kABytes + kXSliceOff, &tmX, &x_full[stage], ks * 256, 0,
                                        l2_policy_evict_last());
                        }
                        mbar_arrive_expect_tx(&full[stage], kBBytes + sf_bytes * halves);
                        tma_load_2d(smem + kOffB + stage * kBBytes, &tmB, &full[stage], ks * kBKBytes, b_row0, pol);
                        for (int h = 0; h < halves; ++h)    // halves == 2 implies band t.nb*2+1 exists
                            bulk_load(smem + kOffSfb + stage * kSfbBytes + h * 2048,
                                      p.sfb + (int64_t)(b_band0 + h) * p.sfb_band_bytes + (int64_t)ks * kT * 512, sf_bytes,
                                      &full[stage], pol);
                    }
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == kStages) { stage = 0; phase ^= 1; }
                }
            }
            (void)n_bands_w;
            // Every copy this thread issued has landed before the CTA may exit.
            for (int s = 0; s < kStages; ++s)
                if (issued_mask & (1u << s)) {
                    if (kFused && !act_side)
                        mbar_wait(&x_full[s], (issued_phase >> s) & 1u, p.err_flag, kErrTimeout, p.wait_ns);
                    mbar_wait(&full[s], (issued_phase >> s) & 1u, p.err_flag, kErrTimeout, p.wait_ns);
                }
        } else if (warp == 2 && p.splits == 1 && p.bias != nullptr) {
            // ---------------------------------------------------- bias loader --
            // The bias of each tile into one of two shared buffers, for the
            // four epilogue warps (bias_full / bias_empty per buffer).  As a
            // programmatic dependent this grid may start before the kernel
            // that writes the bias has finished: wait for it first.
            griddep_wait();
            uint16_t *s_bias_all = reinterpret_cast<uint16_t *>(smem + kOffBias);
            int it = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
                const Work wk = work_of(tile, p, num_ks);
                if (wk.g < 0) continue;
                const Tile t = wk.t;
                const int n_rows = min(kBN, p.n_out - t.nb * kBN);
                const int b = it & 1;
                if (!__all_sync(~0u, mbar_wait(&bias_empty[b], ((it >> 1) & 1) ^ 1, p.err_flag, kErrTimeout,
                                               p.wait_ns)))
                    break;
                for (int j = lane; j < kBN; j += 32)
                    s_bias_all[b * kBN + j] = (j < n_rows) ? p.bias[wk.g * p.group_n + t.nb * kBN + j] : (uint16_t)0;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bias_full[b]);
            }
        } else if (warp == 1) {
            // ----------------------------------------------------------- MMA --
            // The whole warp runs the loop, so every value in it stays
            // warp-uniform; one elected lane issues the tcgen05 instructions
            // (MMAs and the commits that track them).
            const bool leader = elect_one();
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            const uint32_t a_base = smem_u32(smem + kOffA);
            const uint32_t b_base = smem_u32(smem + kOffB);
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                const Work wk = work_of(tile, p, num_ks);
                if (wk.g < 0) continue;
                const int n_rows = min(kBN, p.n_out - wk.t.nb * kBN);
                const uint32_t n_mma = n_rows > 128 ? 256 : 128;
                const uint32_t idesc = idesc_nvf4(128, n_mma);
                if (!__all_sync(~0u, mbar_wait(tmem_empty, acc_phase ^ 1, p.err_flag, kErrTimeout, p.wait_ns))) break;
                tc_fence_after_sync();
                for (int ks = wk.ks0; ks < wk.ks1; ++ks) {
                    // sf_ready implies full: the scale warps arrive on it only
                    // after they saw the stage land (and read its scales).
                    if (!__all_sync(~0u, mbar_wait(&sf_ready[stage], phase, p.err_flag, kErrTimeout, p.wait_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const int kcount = min(4, p.num_k64 - ks * 4);
                    const uint32_t sf_col = tmem + kTmemSf + stage * kSfColsPerStage;
                    const uint64_t adesc = smem_desc_sw128(a_base + stage * kABytes);
                    const uint64_t bdesc = smem_desc_sw128(b_base + stage * kBBytes);
                    if (leader) {
                        for (int kk = 0; kk < kcount; ++kk) {
                            // K-step kk starts 32 bytes further into the swizzled 128-byte rows
                            const uint64_t ad = adesc + (uint64_t)(kk * 2), bd = bdesc + (uint64_t)(kk * 2);
                            const uint32_t acc_flag = (ks != wk.ks0 || kk != 0);
                            if constexpr (kMx)      // two UE8M0 scales per row and K-step: half a scale word
                                tc_mma_mxf4(tmem, ad, bd, idesc_mxf4(128, n_mma, (kk & 1) * 2),
                                            sf_col + (kk >> 1) * 4, sf_col + 8 + (kk >> 1) * 8, acc_flag);
                            else
                                tc_mma_nvf4(tmem, ad, bd, idesc, sf_col + kk * 4, sf_col + 16 + kk * 8, acc_flag);
                        }
                        tc_commit(&empty[stage]);
                    }
                    if (++stage == kStages) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                if (leader) tc_commit(tmem_full);
                __syncwarp();
                acc_phase ^= 1;
            }
            // No MMA may still be running when the TMEM is released.
            if (leader) tc_commit(mma_done);
            __syncwarp();
            mbar_wait(mma_done, 0, p.err_flag, kErrTimeout, p.wait_ns);
        }
    }

    if (p.splits > 1 && warp < kEpiWarp0) {
        // the other warps' arrivals on both phases of the epilogue's cluster
        // barrier (they hold nothing the reduction reads)
        cluster_arrive_release();
        cluster_wait_acquire();
        cluster_arrive_release();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (p.splits > 1) cluster_wait_acquire();          // every peer has read this CTA's partials
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

namespace {

// Launches the one-CTA kernel: the plain GEMM or, with `fused`, the fused
// small-m linear, optionally as a programmatic dependent of the kernel before
// it (only the activation side waits for that kernel; the weights stream at
// once).
cudaError_t launch_one_cta(const GemmParams &p, const uint8_t *a, const uint8_t *w, int num_sms, cudaStream_t s,
                           const char **why, bool dependent, bool fused)
{
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(gemm_nvf4_kernel<false, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_nvf4_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_nvf4_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(gemm_nvf4_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    CUtensorMap tmA, tmB, tmOut;
    const uint64_t row_bytes = (uint64_t)p.kp / 2;
    if (!make_operand_map(&tmA, a, row_bytes, (uint64_t)p.m, kBM) ||
        !make_operand_map(&tmB, w, row_bytes, (uint64_t)p.n_w, kBN)) {
        *why = "cuTensorMapEncodeTiled failed for an FP4 operand";
        return cudaErrorInvalidValue;
    }
    if (p.splits == 1) {
        if (!make_output_map(&tmOut, p.out, (uint64_t)p.n_out, (uint64_t)p.m, (uint64_t)p.ldo)) {
            *why = "cuTensorMapEncodeTiled failed for the output";
            return cudaErrorInvalidValue;
        }
    } else {
        tmOut = tmA;                                    // not used: the cluster reduction stores the output
    }
    // Persistent over the tiles (one CTA per SM at most); with split-K one CTA
    // per (tile, K range), the ranges of a tile forming one cluster.
    const int items = p.num_m_blk * p.num_n_blk * p.splits;
    if (p.splits > 1 && (p.splits > kMaxSplits || p.num_m_blk != 1 || p.group_offsets != nullptr)) {
        *why = "split-K takes one 128-row band, no groups, at most 8 ranges";
        return cudaErrorInvalidValue;
    }
    const int grid = p.splits > 1 ? items : (items < num_sms ? items : num_sms);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attrs[2];
    int n_attrs = 0;
    if (dependent) {
        attrs[n_attrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n_attrs].val.programmaticStreamSerializationAllowed = 1;
        ++n_attrs;
    }
    if (p.splits > 1) {
        attrs[n_attrs].id = cudaLaunchAttributeClusterDimension;
        attrs[n_attrs].val.clusterDim.x = (unsigned)p.splits;
        attrs[n_attrs].val.clusterDim.y = 1;
        attrs[n_attrs].val.clusterDim.z = 1;
        ++n_attrs;
    }
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = n_attrs ? attrs : nullptr;
    cfg.numAttrs = n_attrs;
    CUtensorMap tmX = tmA;                              // the plain GEMM reads no bf16 activation
    if (fused && !make_x_slice_map(&tmX, p.quant.x, (uint64_t)p.quant.k, (uint64_t)p.quant.m, (uint64_t)p.quant.ldx)) {
        *why = "cuTensorMapEncodeTiled failed for the activation";
        return cudaErrorInvalidValue;
    }
    if (fused)
        return p.mx ? cudaLaunchKernelEx(&cfg, gemm_nvf4_kernel<true, true>, tmA, tmB, tmOut, tmX, p)
                    : cudaLaunchKernelEx(&cfg, gemm_nvf4_kernel<false, true>, tmA, tmB, tmOut, tmX, p);
    return p.mx ? cudaLaunchKernelEx(&cfg, gemm_nvf4_kernel<true, false>, tmA, tmB, tmOut, tmX, p)
                : cudaLaunchKernelEx(&cfg, gemm_nvf4_kernel<false, false>, tmA, tmB, tmOut, tmX, p);
}

}  // namespace

int gemm_split_clusters(int splits, int num_sms)
{
    // clusters of `splits` one-CTA GEMM blocks resident at once on this device
    // (queried once per device and size; the SMs / splits if the query fails)
    static int cached_dev = -1;
    static int cached[kMaxSplits + 1];
    int dev = 0;
    cudaGetDevice(&dev);
    if (splits < 2 || splits > kMaxSplits) return num_sms;
    if (cached_dev != dev) {
        for (int i = 0; i <= kMaxSplits; ++i) cached[i] = 0;
        cached_dev = dev;
    }
    if (cached[splits] == 0) {
        int clusters = 0;
        cudaError_t e = cudaFuncSetAttribute(gemm_nvf4_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e == cudaSuccess) {
            cudaLaunchConfig_t probe = {};
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = (unsigned)splits;
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            probe.gridDim = dim3((unsigned)(splits * (num_sms / splits)), 1, 1);
            probe.blockDim = dim3(kThreads, 1, 1);
            probe.dynamicSmemBytes = kSmemBytes;
            probe.attrs = &attr;
            probe.numAttrs = 1;
            e = cudaOccupancyMaxActiveClusters(&clusters, gemm_nvf4_kernel<false, false>, &probe);
        }
        if (e != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            clusters = num_sms / splits;
        }
        cached[splits] = clusters;
    }
    return cached[splits];
}

cudaError_t launch_gemm(const GemmParams &p, const uint8_t *a, const uint8_t *w, int num_sms, cudaStream_t s,
                        const char **why, bool dependent)
{
    return launch_one_cta(p, a, w, num_sms, s, why, dependent, false);
}

cudaError_t launch_linear_fused(const GemmParams &p, const uint8_t *w, int num_sms, cudaStream_t s, const char **why)
{
    if (p.m > kFusedMaxRows || p.quant.bs != 0 || p.group_offsets != nullptr) {
        *why = "the fused linear takes activations of at most 16 rows, without a transform";
        return cudaErrorInvalidValue;
    }
    // A programmatic dependent of the kernel before it: the prologue (barrier
    // set-up, TMEM allocation, scale table) overlaps that kernel's tail, and
    // both producers wait for it before their first copy.
    return launch_one_cta(p, p.quant.out, w, num_sms, s, why, true, true);
}

}  // namespace nvfp4
