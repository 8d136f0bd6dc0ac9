// Internal declarations shared by the kernels and the C-ABI layer.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4 {

// Padded K of packed operands: a multiple of 32 FP4 elements (16 bytes), the
// row alignment the TMA needs for the packed rows.
__host__ __device__ constexpr int64_t padded_k(int64_t k) { return (k + 31) / 32 * 32; }
// Scale columns (one per 16 elements of the padded K) and their padding to 4.
__host__ __device__ constexpr int64_t scale_cols(int64_t k) { return padded_k(k) / 16; }
__host__ __device__ constexpr int64_t scale_cols_padded(int64_t k) { return (scale_cols(k) + 3) / 4 * 4; }
__host__ __device__ constexpr int64_t rows_padded(int64_t rows) { return (rows + 127) / 128 * 128; }

// Byte offset of block scale (r, c) in the tiled scale layout: 512-byte tiles
// of 128 rows x 4 columns, the tiles of a 128-row band consecutive along K;
// inside a tile, 16-byte line (r % 32) holds rows r%32 + {0,32,64,96}, four
// bytes each.  This is exactly the 32-row x 128-bit image that tcgen05.cp
// (32x128b, warpx4) moves into TMEM for the block-scaled MMA.
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t cols_padded)
{
    return ((r >> 7) * (cols_padded >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

struct QuantParams {
    const uint16_t *x;     // bf16 bits, [m, ldx]
    int64_t ldx;           // elements
    int32_t m, k;          // logical rows / K
    int32_t kp;            // padded K
    int32_t nb;            // kp / 16
    int32_t nbp;           // roundup(nb, 4)
    int32_t mp;            // roundup(m, 128)
    const float *gs;       // device fp32
    uint8_t *out;          // [m, kp/2]
    uint8_t *sf;           // tiled [mp, nbp]
    const uint16_t *t;     // transform (bf16 bits) or nullptr
    int32_t bs;
    unsigned int *err_flag;  // device error word (transform kernel's bounded waits)
    uint16_t *y_out;         // nullptr, or [m, k] bf16: the transform result (row stride k)
};

constexpr int kMaxSplits = 8;        // split-K ranges at most (the portable cluster size)

struct GemmParams {
    int32_t m, n_w, n_out, kp;
    int32_t num_k64;                 // kp / 64 rounded up: K-steps of the MMA
    int32_t sf_tiles;                // 512-byte scale tiles per 128-row band (scale columns / 4)
    int32_t mx;                      // 1: MXFP4 operands (UE8M0 scales per 32 elements, no alpha)
    int32_t num_m_blk, num_n_blk;
    const uint8_t *sfa, *sfb;        // tiled scales
    int64_t sfa_band_bytes;          // bytes per 128-row band of scales
    int64_t sfb_band_bytes;
    const float *alpha;              // device fp32; nullptr reads as 1 (MXFP4)
    const uint16_t *bias;            // bf16 bits or nullptr
    uint16_t *out;                   // bf16 bits
    int64_t ldo;
    unsigned int *err_flag;          // device error word
    // Split-K (small m, one-CTA kernel): K is cut into `splits` ranges of
    // `stages_per_split` 256-element stages; the ranges of a tile run as the
    // CTAs of one thread-block cluster, which sum their fp32 partials through
    // distributed shared memory before the epilogue's alpha, bias and bf16
    // rounding.  splits == 1: no split.
    int32_t splits;                  // 1 .. kMaxSplits
    int32_t stages_per_split;
    // Grouped GEMM (one-CTA kernel only): group_offsets [num_groups + 1] are
    // ascending row offsets, multiples of 128; the 128-row band of A at row r
    // belongs to the group g with offsets[g] <= r < offsets[g + 1] and is
    // multiplied by weight rows [g * group_n, (g + 1) * group_n) (stacked
    // weights), scaled by alpha[g], biased by bias[g * group_n + column].
    // Bands at or past offsets[num_groups] are skipped.  group_offsets ==
    // nullptr: a plain GEMM (group 0, group_n = 0).
    const int32_t *group_offsets;
    int32_t num_groups;
    int32_t group_n;
    uint64_t wait_ns;                // bound of every pipeline barrier wait (ns of %globaltimer)
    int32_t drill;                   // 1: timeout drill, the producers issue no copies (test hook)
    // Fused small-m linear (one-CTA kernel): the activation the kernel
    // quantizes itself, stage by stage, into shared memory.
    QuantParams quant;
};

constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // two seconds

// Launchers (return a cudaError_t; no host synchronisation).
cudaError_t launch_quant(const QuantParams &p, int num_sms, cudaStream_t s);
cudaError_t launch_quant_transform(const QuantParams &p, int num_sms, cudaStream_t s, const char **why);
// dependent = true launches the GEMM as a programmatic dependent of the
// preceding kernel, which must be the quantizer of its activation operand:
// the GEMM's weight-side loads then start before that kernel has finished.
cudaError_t launch_gemm(const GemmParams &p, const uint8_t *a, const uint8_t *w, int num_sms, cudaStream_t s,
                        const char **why, bool dependent = false);
// The fused small-m linear (m <= 16, NVFP4, no transform): p.quant describes
// the bf16 activation; the GEMM's epilogue warps quantize each stage of it
// into shared memory themselves, so no quantizer runs before it.  Launched as a
// programmatic dependent of the kernel before it, whose completion both of its
// producers wait for.
cudaError_t launch_linear_fused(const GemmParams &p, const uint8_t *w, int num_sms, cudaStream_t s,
                                const char **why);
// Clusters of `splits` one-CTA GEMM blocks that can be resident at once (the
// split-K plan's wave count).
int gemm_split_clusters(int splits, int num_sms);
// CTA-pair variant for m > 128 (tiles of 256 x 256 on two SMs).
cudaError_t launch_gemm_pair(const GemmParams &p, const uint8_t *a, const uint8_t *w, int num_sms, cudaStream_t s,
                             const char **why, bool dependent = false);

// Workspace of nvfp4_linear: the quantized activation and its scales (256-byte
// aligned inside).
size_t linear_min_workspace_bytes(int64_t m, int64_t k);

// Records `msg` as this thread's last error (read by nvfp4_last_error_string)
// and returns `st`; for entry points that live outside api.cu.
int record_error(int st, const char *msg);

// Device error word (bit 1: a pipeline wait timed out).
constexpr unsigned int kErrTimeout = 1u;
cudaError_t device_error_word(unsigned int **ptr);

}  // namespace nvfp4
