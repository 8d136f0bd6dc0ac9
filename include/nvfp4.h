/*
 * nvfp4.h -- C ABI of the GB300 (sm_103a) NVFP4 W4A4 linear layer.
 *
 * What the library computes (the pages are vLLM pull-request summaries; each
 * entry point names the one that defines its operation):
 *
 *   [torch-backend page]  "TorchNvFp4LinearKernel" (vLLM PR #53319), section
 *       关键源码片段 (key source snippets): process_weights_after_loading
 *       swizzles the weight block scales and pads the packed weight for the
 *       GEMM; apply_weights quantizes the activation with its global scale into
 *       packed FP4 plus swizzled block scales (K padded to the weight's padding),
 *       runs the block-scaled FP4 GEMM into the activation dtype, multiplies by
 *       alpha (product of the activation and weight global dequant scales),
 *       slices the padded output columns and adds the bias.
 *   [transform page]  "QUTLASS fusedQuantizeNv" (vLLM PR #43229), sections
 *       实现拆解 (implementation breakdown) items 3, 4 and 6 and the
 *       HadamardTransform snippet: an online block-diagonal transform of the
 *       input (block size 16/32/64/128, 1/sqrt(n) folded into the matrix, result
 *       in the activation dtype) fused with the NVFP4 quantization, writing into
 *       caller-preallocated outputs that never alias the inputs.
 *   [b12x page]  "B12X quantized linear backends" (vLLM PR #52016), NVFP4
 *       snippet: a non-contiguous 2-D view of the input goes straight into the
 *       quantizer (no contiguous copy); alpha is handed to the GEMM; packed
 *       weight storage is reused on reload so captured CUDA graphs stay valid.
 *       Its MXFP4 backend (dynamic activations) names the second format, whose
 *       activation quantizer is nvfp4_mxfp4_quant_act.
 *   Beyond the pages' calibrated scales, nvfp4_act_global_scale computes the
 *   activation global scale from the data on the device.
 *
 * Number formats.  FP4 = E2M1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their
 * negatives), two per byte, the even-index element in the low nibble.  Block
 * scale = FP8 E4M3 (max 448) per 16 consecutive K elements.  The per-tensor
 * global scale gs is an fp32 that MULTIPLIES into the block scale:
 *     s  = (amax(block) * gs) / 6      (fp32, each op rounded to nearest even)
 *     sf = e4m3_rne_satfinite(s)
 *     q  = e2m1_rne_satfinite(v * (gs / e4m3(sf)))   (0 when e4m3(sf) == 0)
 * so that v ~= e2m1(q) * e4m3(sf) / gs, and the linear's alpha = 1/(gs_x*gs_w).
 *
 * Layouts (all row-major, all caller-allocated device memory):
 *   Kp  = roundup(k, 32)                 padded K of every packed operand
 *   packed FP4   [rows, Kp/2] bytes      (row stride Kp/2; pad elements = 0)
 *   scales       [Rp, Cp] bytes, tiled:  Rp = roundup(rows,128), Cp = roundup(Kp/16,4)
 *       offset(r,c) = ((r/128)*(Cp/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4
 *       i.e. 512-byte tiles of 128 rows x 4 scale columns; padding bytes are 0.
 *
 * Conventions shared by every call:
 *   - Every pointer is device memory except where stated.  Buffers are owned
 *     by the caller; the library allocates nothing and never synchronises the
 *     stream: work is enqueued on `stream` (a cudaStream_t, 0 = legacy default).
 *   - All arguments are validated on the host before anything is launched; an
 *     invalid call returns a non-zero status, launches nothing and leaves the
 *     reason in nvfp4_last_error_string() (thread-local).
 *   - Outputs may not overlap any input (NVFP4_ERR_ALIAS).
 *   - Row strides are in elements; every base pointer and every row must start
 *     on a 16-byte boundary (NVFP4_ERR_ALIGNMENT).
 *   - m == 0 (or n == 0 for the weight) is a valid empty call: NVFP4_OK, no launch
 *     (nvfp4_act_global_scale still writes its defined result for m == 0).
 *   - Global scales and alpha are read on the device, so no call waits for the
 *     host or synchronises with it.
 *   - A kernel that waits longer than about two seconds on one of its own
 *     pipeline barriers abandons the launch and raises a device error flag
 *     that nvfp4_device_error() reports (NVFP4_ERR_TIMEOUT); it never hangs.
 */
#ifndef NVFP4_GB300_H
#define NVFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_ABI_VERSION 1

/* Opaque CUDA stream handle; pass a cudaStream_t. */
typedef struct CUstream_st *nvfp4_stream_t;

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,        /* null pointer, bad size, bad block size  */
    NVFP4_ERR_UNSUPPORTED_DEVICE = 2, /* current device is not compute 10.3       */
    NVFP4_ERR_ALIGNMENT = 3,          /* pointer or row stride not 16-B aligned   */
    NVFP4_ERR_ALIAS = 4,              /* an output overlaps an input              */
    NVFP4_ERR_CUDA = 5,               /* a CUDA runtime/driver call failed        */
    NVFP4_ERR_TIMEOUT = 6,            /* a kernel gave up on a barrier wait       */
    NVFP4_ERR_WORKSPACE = 7           /* workspace missing or too small           */
} nvfp4_status;

/* ABI version of the loaded library (NVFP4_ABI_VERSION at build time). */
int nvfp4_abi_version(void);

/* Capability check, modelled on the torch-backend page's is_supported (which
 * returns (False, reason) instead of raising): NVFP4_OK if `device` can run
 * this library (compute capability 10.3, the only target it is built for),
 * else NVFP4_ERR_UNSUPPORTED_DEVICE / NVFP4_ERR_CUDA with a reason copied into
 * `reason` (host buffer of reason_len bytes, may be NULL). */
nvfp4_status nvfp4_is_supported(int device, char *reason, size_t reason_len);

/* Text of the last error raised by a call on this host thread ("" if none).
 * The string stays valid until the next library call on the same thread. */
const char *nvfp4_last_error_string(void);

/* Reads (and, if clear != 0, resets) the device error flag of the current
 * device: NVFP4_OK or NVFP4_ERR_TIMEOUT.  This call synchronises the device. */
nvfp4_status nvfp4_device_error(int clear);

/* ---- size queries (pure host arithmetic; no device access) -------------- */

/* Bytes of a packed FP4 operand: rows * roundup(k,32)/2. */
size_t nvfp4_packed_bytes(int64_t rows, int64_t k);

/* Bytes of a tiled scale tensor: roundup(rows,128) * roundup(roundup(k,32)/16, 4). */
size_t nvfp4_scale_bytes(int64_t rows, int64_t k);

/* Workspace nvfp4_linear wants for an m x k activation against n_w weight
 * rows: the quantized activation and its scales, each 256-B aligned inside
 * (n_w is accepted for future use and does not change the size). */
size_t nvfp4_linear_workspace_bytes(int64_t m, int64_t k, int64_t n_w);

/* ---- operations ---------------------------------------------------------- */

/* Weight preparation, the torch-backend page's process_weights_after_loading
 * (swizzle_blockscale + pad_nvfp4_weight_for_cutlass), here starting from the
 * bf16 weight: quantize W [n, k] (row stride ldw) with global scale *w_gs_dev
 * (device fp32; the weight's counterpart of the activation global scale), pad
 * K to Kp = roundup(k,32) with zeros, pack to FP4 and write the tiled scales.
 *   w_bf16  in   [n, ldw] bf16
 *   w_fp4   out  nvfp4_packed_bytes(n, k) bytes
 *   w_sf    out  nvfp4_scale_bytes(n, k) bytes
 * Outputs are written in place, so a reload into the same buffers keeps the
 * weight addresses stable for captured graphs (b12x page, packed-storage reuse). */
nvfp4_status nvfp4_prepare_weight(const void *w_bf16, int64_t n, int64_t k, int64_t ldw,
                                  const float *w_gs_dev, uint8_t *w_fp4, uint8_t *w_sf,
                                  nvfp4_stream_t stream);

/* Activation quantization, the torch-backend page's scaled_fp4_quant call
 * (swizzled scales, K padded) with the transform page's optional fused
 * block-diagonal transform in front:
 *   x_bf16          in   [m, ldx] bf16, the first k columns are the data (a
 *                        strided view is fine: ldx >= k)
 *   gs_dev          in   device fp32, activation global scale
 *   transform_bf16  in   NULL (bs = 0) for none, else a bs x bs bf16 matrix T,
 *                        row-major, 1/sqrt(bs) already folded in; bs in
 *                        {16,32,64,128} and bs must divide k.  Then every bs-wide
 *                        block of a row is replaced by y = bf16(x_block * T)
 *                        before quantizing: the exact bf16 x bf16 products are
 *                        summed in fp32 on the tensor cores, in their own
 *                        order, and rounded to bf16 once.
 *   x_fp4           out  nvfp4_packed_bytes(m, k) bytes
 *   x_sf            out  nvfp4_scale_bytes(m, k) bytes                        */
nvfp4_status nvfp4_quant_act(const void *x_bf16, int64_t m, int64_t k, int64_t ldx,
                             const float *gs_dev, const void *transform_bf16, int bs,
                             uint8_t *x_fp4, uint8_t *x_sf, nvfp4_stream_t stream);

/* nvfp4_quant_act with a transform (transform_bf16 non-NULL), which also
 * writes the bf16 transform result y that the codes and scales were computed
 * from: y_bf16 (out, device, 16-byte aligned) is [m, k] bf16 with row stride
 * k, and must not overlap any other argument.  The codes are then a function
 * of y alone, so a checker can requantize y and compare bit for bit, and
 * compare y itself with x * blockdiag(T).  Same kernel and same x_fp4/x_sf
 * bytes as nvfp4_quant_act; the extra output costs 2 bytes per element. */
nvfp4_status nvfp4_quant_act_export_y(const void *x_bf16, int64_t m, int64_t k, int64_t ldx,
                                      const float *gs_dev, const void *transform_bf16, int bs,
                                      uint8_t *x_fp4, uint8_t *x_sf, void *y_bf16,
                                      nvfp4_stream_t stream);

/* MXFP4 activation quantization, the format of the B12X page's MXFP4 linear
 * backend (dynamic activations; OCP Microscaling v1.0): 32-element blocks of
 * E2M1 values sharing one E8M0 scale 2^s, no per-tensor scale:
 *   s    = clamp(floor(log2(amax)) - 2, -127, 127), -127 for an all-zero block;
 *   code = s + 127 (one byte per block);  q_i = e2m1_rne_satfinite(v_i * 2^-s).
 *   x_bf16  in   [m, ldx] bf16, the first k columns are the data
 *   x_fp4   out  nvfp4_packed_bytes(m, k) bytes: K padded to roundup(k,32) with
 *                zeros, two codes per byte, the even element in the low nibble
 *   x_sf    out  nvfp4_mxfp4_scale_bytes(m, k) bytes: the scale codes in the
 *                tiled layout of the NVFP4 scales (512-byte tiles of 128 rows x
 *                4 columns), one column per 32 elements, zero padding
 * Validation, aliasing and error behaviour as for nvfp4_quant_act. */
size_t nvfp4_mxfp4_scale_bytes(int64_t rows, int64_t k);   /* roundup(rows,128) * roundup(roundup(k,32)/32, 4) */
nvfp4_status nvfp4_mxfp4_quant_act(const void *x_bf16, int64_t m, int64_t k, int64_t ldx,
                                   uint8_t *x_fp4, uint8_t *x_sf, nvfp4_stream_t stream);

/* MXFP4 GEMM, the B12X page's MXFP4 linear backend (mm_mxfp4 on activations
 * from flashinfer_mxfp4_quantize; section 实现拆解), with the epilogue of
 * nvfp4_gemm minus alpha (the MX formats have no global scale):
 *   out[i, j] = bf16( sum_k deq(A)[i,k] * deq(W)[j,k] + bias[j] ),
 *   deq(q) = e2m1(q) * 2^(code - 127), one E8M0 code per 32 K-elements.
 *   a_fp4, a_sf     in   activation from nvfp4_mxfp4_quant_act
 *   w_fp4, w_sf     in   weight [n_w, k] quantized by the same conversion
 *                        (nvfp4_mxfp4_quant_act applied to the bf16 weight)
 *   k, n_out, bias_bf16, out_bf16, ldo   as for nvfp4_gemm
 * The operands' scales use the tiled layout with one column per 32
 * elements (nvfp4_mxfp4_scale_bytes). */
nvfp4_status nvfp4_mxfp4_gemm(const uint8_t *a_fp4, const uint8_t *a_sf, int64_t m,
                              const uint8_t *w_fp4, const uint8_t *w_sf, int64_t n_w, int64_t n_out,
                              int64_t k, const void *bias_bf16, void *out_bf16, int64_t ldo,
                              nvfp4_stream_t stream);

/* The whole MXFP4 linear (the B12X page's MXFP4 backend apply path):
 * nvfp4_mxfp4_quant_act of x into `workspace`, then nvfp4_mxfp4_gemm, on one
 * stream.  workspace: caller-owned device scratch of at least
 * align256(nvfp4_packed_bytes(m,k)) + align256(nvfp4_mxfp4_scale_bytes(m,k))
 * bytes (= nvfp4_mxfp4_linear_workspace_bytes); with m <= 128 the GEMM may
 * split K as nvfp4_linear does, and for m <= 16 the quantizer runs inside the
 * GEMM (its epilogue warps quantize each K stage of x; the workspace's
 * activation area is then not written), as in nvfp4_linear. */
size_t nvfp4_mxfp4_linear_workspace_bytes(int64_t m, int64_t k, int64_t n_w);
nvfp4_status nvfp4_mxfp4_linear(const void *x_bf16, int64_t m, int64_t k, int64_t ldx,
                                const uint8_t *w_fp4, const uint8_t *w_sf, int64_t n_w, int64_t n_out,
                                const void *bias_bf16, void *out_bf16, int64_t ldo,
                                void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* Dynamic activation global scale: the per-tensor AbsMax statistic of the
 * transform page's fusedQuantizeNv computed on the device, for activations
 * without a calibrated scale (the torch-backend page's input_global_scale_inv
 * then comes from the data):
 *   amax         = max |v| over the m x k activation, v = x, or with a
 *                  transform the bf16 y = x * blockdiag(T) exactly as
 *                  nvfp4_quant_act computes it (same kernel pipeline);
 *   gs_out[0]    = fl32(448 * 6 / amax); the largest finite float if that
 *                  overflows; 1 when amax == 0 (m == 0 included);
 *   alpha_out[0] = fl32(1 / fl32(gs_out[0] * w_gs_dev[0])) when alpha_out and
 *                  w_gs_dev are given (both or neither).
 *   x_bf16, k, ldx, transform_bf16, bs   as for nvfp4_quant_act
 *   gs_out      out  device fp32; also the pass's scratch word (it holds the
 *                    amax bits until the last kernel of the call)
 * gs_out and alpha_out feed nvfp4_quant_act / nvfp4_linear directly; nothing
 * leaves the device and nothing synchronises, so the sequence can be captured
 * in a CUDA graph.  Costs one read of x (2 bytes per element) before the
 * quantizer's; a tensor smaller than L2 is then re-read from L2. */
nvfp4_status nvfp4_act_global_scale(const void *x_bf16, int64_t m, int64_t k, int64_t ldx,
                                    const void *transform_bf16, int bs, const float *w_gs_dev,
                                    float *gs_out, float *alpha_out, nvfp4_stream_t stream);

/* Block-scaled FP4 GEMM with the fused epilogue (torch-backend page:
 * torch._scaled_mm, then * alpha, slice_nvfp4_output, + bias):
 *   out[i, j] = bf16( alpha * sum_k deq(A)[i,k] * deq(W)[j,k] + bias[j] ),
 *   deq(q) = e2m1(q) * e4m3(block scale), i < m, j < n_out.
 *   a_fp4, a_sf     in   quantized activation (as written by nvfp4_quant_act)
 *   w_fp4, w_sf     in   prepared weight with n_w rows (nvfp4_prepare_weight)
 *   k               in   logical K of both (their Kp = roundup(k,32) must match)
 *   n_out           in   1 <= n_out <= n_w: columns kept (the output slice)
 *   alpha_dev       in   device fp32
 *   bias_bf16       in   NULL or [n_out] bf16
 *   out_bf16        out  [m, ldo] bf16, ldo >= n_out; columns >= n_out untouched */
nvfp4_status nvfp4_gemm(const uint8_t *a_fp4, const uint8_t *a_sf, int64_t m,
                        const uint8_t *w_fp4, const uint8_t *w_sf, int64_t n_w, int64_t n_out,
                        int64_t k, const float *alpha_dev, const void *bias_bf16,
                        void *out_bf16, int64_t ldo, nvfp4_stream_t stream);

/* nvfp4_gemm with the two choices the library otherwise makes itself, for
 * testing its kernels and its failure path (the pages have no counterpart):
 *   kernel         0: as nvfp4_gemm (the CTA-pair kernel for m > 128, else the
 *                     one-CTA kernel);  1: the one-CTA kernel at any m;
 *                  2: the CTA-pair kernel (m > 128 only, else NVFP4_ERR_INVALID_ARG);
 *                  3: the one-CTA kernel with nvfp4_linear's split-K plan
 *                     (m <= 128 splits as nvfp4_linear would).
 *   wait_limit_ns  bound of every pipeline barrier wait of this launch, in
 *                  [1e6, 1e10] ns; 0 = the library's two seconds.
 *   drill          0: compute normally.  1: timeout drill -- the kernel's copy
 *                  producers issue nothing, so each of its barrier waits runs
 *                  out after wait_limit_ns; the kernel then sets the device
 *                  error flag (nvfp4_device_error() reports NVFP4_ERR_TIMEOUT)
 *                  and ends with nothing computed, stored or left in flight,
 *                  so the next call runs normally.  The call itself returns
 *                  NVFP4_OK (the wait runs out on the device, after the launch).
 * Every other argument, check and result is that of nvfp4_gemm. */
nvfp4_status nvfp4_gemm_ex(const uint8_t *a_fp4, const uint8_t *a_sf, int64_t m,
                           const uint8_t *w_fp4, const uint8_t *w_sf, int64_t n_w, int64_t n_out,
                           int64_t k, const float *alpha_dev, const void *bias_bf16,
                           void *out_bf16, int64_t ldo, int kernel, uint64_t wait_limit_ns, int drill,
                           nvfp4_stream_t stream);

/* Grouped NVFP4 GEMM for mixture-of-experts layers: one launch over the
 * token groups of all experts, each group multiplied by its own expert's
 * weight (the grouped NVFP4 MoE GEMM the transform page's related-work
 * section points to; the b12x page's packed-weight reuse keeps the stacked
 * weights in place).  The pages give no formula beyond nvfp4_gemm's, applied
 * per group:
 *   out[r, j] = bf16( alpha[g] * sum_k deq(A)[r,k] * deq(W)[g*n + j, k] + bias[g*n + j] )
 * for the rows r of group g and j < n.
 *   a_fp4, a_sf        in   activations of every group in one [rows, k] operand
 *                           (nvfp4_quant_act of the stacked rows, one global scale)
 *   group_offsets_dev  in   device int32 [num_groups + 1], ascending multiples
 *                           of 128: group g owns rows [offsets[g], offsets[g+1]),
 *                           the groups' real rows first and any padding rows
 *                           after them; 128-row bands at or past
 *                           offsets[num_groups] are not computed.  Being on the
 *                           device, the offsets can come from a routing kernel
 *                           of the same stream (no host synchronisation).
 *   w_fp4, w_sf        in   the experts' weights stacked as one [num_groups*n, k]
 *                           operand (nvfp4_prepare_weight per expert into the
 *                           slices w_fp4 + g*n*Kp/2 and w_sf + g*n*Cp, or once
 *                           over all of them); n a multiple of 128
 *   alpha_dev          in   device fp32 [num_groups]: 1/(gs_x * gs_w[g])
 *   bias_bf16          in   NULL or [num_groups * n] bf16
 *   out_bf16           out  [rows, ldo] bf16; every row of every computed band is
 *                           written (padding rows get unspecified values)
 * One 128 x 256 output tile per CTA step on the one-CTA kernel; no split-K. */
nvfp4_status nvfp4_grouped_gemm(const uint8_t *a_fp4, const uint8_t *a_sf, int64_t rows,
                                const int32_t *group_offsets_dev, int num_groups,
                                const uint8_t *w_fp4, const uint8_t *w_sf, int64_t n, int64_t k,
                                const float *alpha_dev, const void *bias_bf16,
                                void *out_bf16, int64_t ldo, nvfp4_stream_t stream);

/* The whole linear layer (torch-backend page apply_weights; b12x page
 * _apply_b12x_nvfp4_linear): nvfp4_quant_act of x into `workspace`, then
 * the GEMM of nvfp4_gemm, all on `stream`.  workspace (device) is scratch owned
 * by the caller, at least align256(nvfp4_packed_bytes(m,k)) +
 * align256(nvfp4_scale_bytes(m,k)) bytes (else NVFP4_ERR_WORKSPACE); its
 * contents after the call are unspecified.  With m <= 128, a GEMM whose
 * output has too few 128 x 256 tiles to fill the GPU splits K: the K ranges
 * of a tile run as the CTAs of one thread-block cluster, which add their fp32
 * partial sums through distributed shared memory in range order before alpha,
 * bias and the bf16 rounding (no extra launch, no partials in memory).  The
 * result is deterministic, but its fp32 rounding order differs from the
 * unsplit GEMM's (both are within the GEMM's accuracy).
 * For m <= 16 without a transform (decode batch sizes) the quantizer runs
 * inside the GEMM: its epilogue warps, idle until the accumulator is done,
 * quantize each K stage of x into the MMA's shared-memory tile themselves
 * (the workspace's activation area is then not written).  Codes, scales and output are those of nvfp4_quant_act
 * followed by nvfp4_gemm, bit for bit. */
nvfp4_status nvfp4_linear(const void *x_bf16, int64_t m, int64_t k, int64_t ldx,
                          const float *gs_dev, const void *transform_bf16, int bs,
                          const uint8_t *w_fp4, const uint8_t *w_sf, int64_t n_w, int64_t n_out,
                          const float *alpha_dev, const void *bias_bf16,
                          void *out_bf16, int64_t ldo,
                          void *workspace, size_t workspace_bytes, nvfp4_stream_t stream);

/* nvfp4_linear without a caller-provided workspace.  The pages have no
 * counterpart to this entry point: it exists for callers that cannot allocate
 * device memory -- a plugin whose host framework owns every device allocation
 * and gives it only its inputs and outputs, or latency-critical code that
 * must never call cudaMalloc (which can synchronise the device).  It computes
 * exactly what nvfp4_linear computes (same arguments minus the workspace),
 * using a scratch array built into the library instead of a workspace:
 *   - The scratch is 16 MiB of device memory that every GPU loading the
 *     library holds until the process exits.  Calls whose quantized activation
 *     and scales (nvfp4_linear's minimum workspace) exceed it are rejected with
 *     NVFP4_ERR_WORKSPACE before anything runs, e.g. up to m = 2048 at
 *     k = 14336 or m = 8192 at k = 3584 fit.
 *   - The first call on a device looks up the scratch's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  The address is kept with the id of the
 *     device's CUDA context; after the context is torn down and re-created
 *     (cudaDeviceReset) the next call looks it up again, so make that call
 *     outside a capture too.
 *   - It allocates nothing (no cudaMalloc / cudaFree, no allocating library
 *     call).  Every call on a device shares the one scratch array and leaves
 *     its contents behind; calls whose work overlaps on the GPU (e.g. on two
 *     streams) race on it. */
nvfp4_status nvfp4_linear_noalloc(const void *x_bf16, int64_t m, int64_t k, int64_t ldx,
                                  const float *gs_dev, const void *transform_bf16, int bs,
                                  const uint8_t *w_fp4, const uint8_t *w_sf, int64_t n_w, int64_t n_out,
                                  const float *alpha_dev, const void *bias_bf16,
                                  void *out_bf16, int64_t ldo, nvfp4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GB300_H */
