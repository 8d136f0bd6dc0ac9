/*
 * NVFP4 W4A4 linear: plain scalar CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg use
 * it.  It shares no code, header, table or constant generator with the CUDA
 * library; both sides are written independently from the same definitions.
 *
 * Sources of each definition (page titles as printed on the pages):
 *   [P1] "TorchNvFp4LinearKernel" PR page (vllm #53319), section "关键源码片段":
 *        apply_weights quantizes the activation with a global scale into packed
 *        float4_e2m1fn_x2 bytes plus swizzled block scales, pads K to the padded
 *        weight, runs the block-scaled FP4 GEMM, multiplies by alpha (the product
 *        of the two global dequant scales), slices the padded columns and adds
 *        the bias.
 *   [P2] "QUTLASS fusedQuantizeNv" PR page (vllm #43229), sections "实现拆解"
 *        items 3 and 6 and the HadamardTransform snippet: an online
 *        block-diagonal transform x * blockdiag(T) with 1/sqrt(n) folded into T,
 *        result cast back to the activation dtype (bf16), then NVFP4 quant with
 *        a per-block absmax scale.
 *   Format facts not printed on the pages (they name the formats only):
 *        FP4 E2M1 and FP8 E4M3 as defined by the OCP Microscaling (MX) v1.0 and
 *        OCP 8-bit floating point (OFP8) specifications; NVFP4 = blocks of 16
 *        E2M1 values sharing one E4M3 scale, under an FP32 per-tensor scale.
 *
 * Readings taken where the pages are silent (each is restated where it is used):
 *   R-scale  s = fl32(fl32(amax * gs) / 6), sf = e4m3_rne_satfinite(s).
 *   R-elem   q = e2m1_rne_satfinite(fl32(v * fl32(gs / dec(sf)))), 0 if dec(sf)==0.
 *   R-sign   e2m1 keeps the sign of values that round to zero (code 0x8).
 *   R-nibble the even element of a pair sits in the low nibble of its byte.
 *   R-pad    K is zero-extended to Kp = roundup(K, 32); padded elements are 0.
 *   R-swz    scale tiles of 128 rows x 4 columns, 512 bytes each,
 *            offset(r,c) = ((r/128)*(Cp/4) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4,
 *            rows padded to 128 and columns to 4 with zero bytes.
 *   R-xform  y[j] = bf16_rne(sum_i x[i]*T[i][j]) of the exact sum (no
 *            intermediate rounding; an exact zero sum gives +0).
 *   R-dyn    dynamic activation scale: gs = fl32(448*6 / amax|v|) over the whole
 *            tensor (of y with a transform), FLT_MAX on overflow, 1 if amax = 0.
 *   R-mx     MXFP4: blocks of 32, E8M0 scale 2^s with s = clamp(floor(log2 amax) - 2,
 *            -127, 127) (-127 for a zero block), q = e2m1(fl32(v * 2^-s)), no global scale.
 *   R-gemm   out[m,n] = alpha * sum_k deq(A)[m,k]*deq(B)[n,k] + bias[n] in FP64,
 *            where deq(q) = e2m1(q) * e4m3(sf) (the global scales live in alpha).
 *
 * Every floating-point step is IEEE binary32 or binary64 with round-to-nearest-
 * even; the file must be compiled without fast-math and with -ffp-contract=off
 * so that no multiply-add is fused behind our back.
 */
#include <assert.h>
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bits -- */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the upper half of an IEEE binary32. */
float oracle_bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* Round a finite binary32 to bf16, nearest-even: keep 8 significant bits and
 * decide on the 16 dropped bits (more than half: up; exactly half: up only if
 * the kept part is odd).  A carry out of the significand bumps the exponent,
 * which is the correct result (up to +inf on overflow). */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u = bits_from_f32(f);
    assert(((u >> 23) & 0xFF) != 0xFF && "oracle: bf16 rounding of a non-finite value");
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1;
    return (uint16_t)kept;
}

/* ------------------------------------------------------------------ E2M1 -- */
/* FP4 E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * exponent 0 is subnormal: value = m * 2^-1; otherwise 2^(e-1) * (1 + m/2). */
double oracle_dec_e2m1(uint8_t code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double mag = (e == 0) ? m * 0.5 : ldexp(1.0 + m * 0.5, e - 1);
    return s ? -mag : mag;
}

/* Nearest E2M1 value, ties to the code with even mantissa bit, magnitudes at or
 * above the largest finite value (6) clamp to it (satfinite).  The sign of the
 * input is kept, so a negative value that rounds to zero gives 0x8 (R-sign). */
uint8_t oracle_enc_e2m1(float f)
{
    assert(isfinite(f) && "oracle: e2m1 of a non-finite value");
    uint8_t sign = signbit(f) ? 0x8 : 0x0;
    double a = fabs((double)f);
    uint8_t best = 7;                               /* satfinite default */
    for (uint8_t c = 0; c < 7; ++c) {               /* walk up the magnitude grid */
        double lo = oracle_dec_e2m1(c), hi = oracle_dec_e2m1((uint8_t)(c + 1));
        double mid = 0.5 * (lo + hi);               /* exact in binary64 */
        if (a < mid) { best = c; break; }
        if (a == mid) { best = (c & 1) ? (uint8_t)(c + 1) : c; break; }
    }
    return (uint8_t)(sign | best);
}

/* ------------------------------------------------------------------ E4M3 -- */
/* FP8 E4M3 (the "fn" variant): bit 7 sign, bits 6..3 exponent (bias 7), bits
 * 2..0 mantissa; exponent 0 is subnormal (m/8 * 2^-6); 0x7F/0xFF are NaN, so
 * the largest finite magnitude is 1.75 * 2^8 = 448 (code 0x7E). */
double oracle_dec_e4m3(uint8_t code)
{
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* Round a finite binary32 to E4M3, nearest-even, saturating to +-448.
 * Exact integer manipulation: write |f| = M * 2^E with an integer significand
 * M, choose the E4M3 quantum 2^Q for that magnitude (2^(ea-3) for normal
 * targets, 2^-9 below the smallest normal 2^-6), and round M*2^E to a multiple
 * of 2^Q on the integer bits. */
uint8_t oracle_enc_e4m3(float f)
{
    assert(isfinite(f) && "oracle: e4m3 of a non-finite value");
    uint32_t u = bits_from_f32(f);
    uint8_t sign = (u >> 31) ? 0x80 : 0x00;
    uint32_t ebits = (u >> 23) & 0xFF, frac = u & 0x7FFFFFu;
    if (ebits == 0 && frac == 0) return sign;            /* +-0 */

    uint64_t M; int E;                                    /* |f| = M * 2^E */
    if (ebits == 0) { M = frac; E = -149; }               /* fp32 subnormal */
    else { M = frac | 0x800000u; E = (int)ebits - 127 - 23; }

    /* unbiased exponent of |f|: position of the top bit of M */
    int top = 63; while (!((M >> top) & 1u)) --top;
    int ea = E + top;

    int Q = (ea >= -6) ? ea - 3 : -9;                     /* E4M3 quantum exponent */
    int shift = Q - E;                                    /* >= 20 always */
    uint64_t n;
    if (shift >= 64) n = 0;                               /* far below half a quantum */
    else {
        n = M >> shift;
        uint64_t rem = M & ((1ull << shift) - 1);
        uint64_t half = 1ull << (shift - 1);
        if (rem > half || (rem == half && (n & 1))) n += 1;
    }
    /* now |result| = n * 2^Q.  With Q == -9 and n < 8 the result is subnormal
     * (exponent field 0, m = n); every other case is normal, n in [8, 16]
     * (a subnormal rounded up to 2^-6 arrives here as n == 8). */
    if (Q == -9 && n < 8) return (uint8_t)(sign | n);
    if (n == 16) { n = 8; Q += 1; }                       /* carry out of the mantissa */
    int efield = Q + 3 + 7;                               /* |result| = (n/8) * 2^(Q+3) */
    int m = (int)n - 8;
    if (efield > 15 || (efield == 15 && m == 7))          /* beyond 448: satfinite */
        return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (efield << 3) | m);
}

/* -------------------------------------------------------- block quantize -- */
/* Quantize `rows` rows of K bf16 values (row stride ld elements) with global
 * scale gs (it multiplies into the block scale, [P1] `input_global_scale_inv`).
 * K is zero-extended to Kp = roundup(K,32) (R-pad).  Outputs:
 *   packed  [rows, Kp/2] bytes, low nibble = even element (R-nibble);
 *   sf_lin  [rows, Kp/16] E4M3 codes, plain row-major (unswizzled).          */
void oracle_quantize_rows(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                          float gs, uint8_t *packed, uint8_t *sf_lin)
{
    const int64_t Kp = (K + 31) / 32 * 32, nb = Kp / 16;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * ld;
        for (int64_t b = 0; b < nb; ++b) {
            float v[16];
            float amax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                int64_t k = b * 16 + i;
                v[i] = (k < K) ? oracle_bf16_to_f32(xr[k]) : 0.0f;
                float a = fabsf(v[i]);
                if (a > amax) amax = a;
            }
            /* R-scale: two binary32 operations, each rounded */
            float t = amax * gs;
            float s = t / 6.0f;
            uint8_t sf = oracle_enc_e4m3(s);
            float d = (float)oracle_dec_e4m3(sf);         /* exact in binary32 */
            /* R-elem: reciprocal-free element multiplier */
            float inv = (d == 0.0f) ? 0.0f : gs / d;
            assert(isfinite(inv));
            sf_lin[r * nb + b] = sf;
            for (int i = 0; i < 16; i += 2) {
                float p0 = v[i] * inv, p1 = v[i + 1] * inv;
                uint8_t q0 = oracle_enc_e2m1(p0), q1 = oracle_enc_e2m1(p1);
                packed[r * (Kp / 2) + (b * 16 + i) / 2] = (uint8_t)(q0 | (q1 << 4));
            }
        }
    }
}

/* ------------------------------------------------------------------ MXFP4 -- */
/* MXFP4 (the B12X page's MXFP4 linear backend, dynamic activations; format of
 * the OCP Microscaling (MX) v1.0 specification): blocks of 32 E2M1 elements
 * sharing one E8M0 scale X = 2^s, code s + 127 (no sign; 0xFF is NaN), and
 * no per-tensor scale.  R-mx:
 *   s   = clamp(floor(log2(amax)) - 2, -127, 127), 2 being the exponent of the
 *         largest E2M1 value (6 = 1.5 * 2^2); an all-zero block gets s = -127;
 *   q_i = e2m1_rne_satfinite(fl32(v_i * 2^-s))   (|v_i| up to 7.99 * 2^s
 *         saturates to 6 * 2^s, as the specification's conversion does).     */
static int floor_log2_pos(float a)          /* a > 0, finite */
{
    const uint32_t u = bits_from_f32(a);
    const int e = (int)((u >> 23) & 0xFF);
    if (e != 0) return e - 127;
    uint32_t f = u & 0x7FFFFFu;
    int top = 22;
    while (!((f >> top) & 1u)) --top;
    return -149 + top;                      /* binary32 subnormal */
}

uint8_t oracle_mx_scale_code(float amax)
{
    assert(isfinite(amax) && amax >= 0.0f);
    if (amax == 0.0f) return 0;
    int s = floor_log2_pos(amax) - 2;
    if (s < -127) s = -127;
    if (s > 127) s = 127;
    return (uint8_t)(s + 127);
}

double oracle_dec_e8m0(uint8_t code)
{
    assert(code != 0xFF && "oracle: E8M0 NaN code");
    return ldexp(1.0, (int)code - 127);
}

/* Quantize `rows` rows of K bf16 values to MXFP4; K is zero-extended to
 * Kp = roundup(K, 32) (R-pad).  packed [rows, Kp/2] as for NVFP4 (R-nibble);
 * sf_lin [rows, Kp/32] E8M0 codes, row-major (unswizzled). */
void oracle_quantize_rows_mx(const uint16_t *x, int64_t rows, int64_t K, int64_t ld, uint8_t *packed,
                             uint8_t *sf_lin)
{
    const int64_t Kp = (K + 31) / 32 * 32, nb = Kp / 32;
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * ld;
        for (int64_t b = 0; b < nb; ++b) {
            float v[32];
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                const int64_t k = b * 32 + i;
                v[i] = (k < K) ? oracle_bf16_to_f32(xr[k]) : 0.0f;
                const float a = fabsf(v[i]);
                if (a > amax) amax = a;
            }
            const uint8_t code = oracle_mx_scale_code(amax);
            const float mul = (float)ldexp(1.0, 127 - (int)code);     /* 2^-s: exact in binary32 */
            sf_lin[r * nb + b] = code;
            for (int i = 0; i < 32; i += 2) {
                const float p0 = v[i] * mul, p1 = v[i + 1] * mul;
                packed[r * (Kp / 2) + (b * 32 + i) / 2] =
                    (uint8_t)(oracle_enc_e2m1(p0) | (oracle_enc_e2m1(p1) << 4));
            }
        }
    }
}

/* --------------------------------------------------------------- swizzle -- */
/* Byte offset of scale (r, c) in the tiled layout of an R x C scale matrix
 * padded to Rp = roundup(R,128), Cp = roundup(C,4) (R-swz). */
int64_t oracle_swizzle_offset(int64_t r, int64_t c, int64_t Cp)
{
    int64_t tile = (r / 128) * (Cp / 4) + c / 4;
    return tile * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

/* Scatter a linear [R, C] scale matrix into the tiled layout; the padded
 * region (rows >= R or columns >= C) is zero. */
void oracle_swizzle(const uint8_t *sf_lin, int64_t R, int64_t C, uint8_t *sf_swz)
{
    const int64_t Rp = (R + 127) / 128 * 128, Cp = (C + 3) / 4 * 4;
    memset(sf_swz, 0, (size_t)(Rp * Cp));
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            sf_swz[oracle_swizzle_offset(r, c, Cp)] = sf_lin[r * C + c];
}

/* Inverse: gather the linear [R, C] matrix back out of the tiled layout. */
void oracle_unswizzle(const uint8_t *sf_swz, int64_t R, int64_t C, uint8_t *sf_lin)
{
    const int64_t Cp = (C + 3) / 4 * 4;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t c = 0; c < C; ++c)
            sf_lin[r * C + c] = sf_swz[oracle_swizzle_offset(r, c, Cp)];
}

/* ------------------------------------------------------------- transform -- */
/* y = x * blockdiag(T, T, ...) for `rows` rows of K values (bs divides K),
 * T a bs x bs bf16 matrix, row-major T[i*bs + j], 1/sqrt(bs) already folded in
 * ([P2] HadamardTransform snippet).  R-xform: y[j] is the exact value of
 * sum_i x[i]*T[i][j], rounded once to bf16, nearest-even ([P2] `.to(value.dtype)`
 * of the product).  Output y is [rows, K] bf16 with row stride K.
 *
 * The exact sum: a bf16 value is an integer significand of at most 8 bits
 * times 2^e (e >= -133), so each product is a signed integer of at most 16
 * bits times 2^(ex+et) with ex+et >= -266.  The products are added as
 * integers into a fixed-point accumulator whose bit 0 weighs 2^-XF_LSB, held
 * in 32-bit digits of int64 limbs (each limb absorbs the carries of up to 2^15
 * additions of 48-bit values before the final normalisation). */
#define XF_LSB 300
#define XF_LIMBS 20                     /* bits of weight 2^-300 .. 2^339 */

static void bf16_split(uint16_t h, int64_t *sig, int *e2)
{
    const int e = (h >> 7) & 0xFF;
    int64_t m = h & 0x7F;
    assert(e != 0xFF);                  /* finite inputs only */
    if (e != 0) { m |= 0x80; *e2 = e - 134; } else { *e2 = -133; }   /* value = m * 2^e2 */
    *sig = (h & 0x8000) ? -m : m;
}

static void acc_normalise(int64_t *limb)
{
    for (int i = 0; i + 1 < XF_LIMBS; ++i) {
        const int64_t low = limb[i] & 0xFFFFFFFFLL;
        limb[i + 1] += (limb[i] - low) / 4294967296LL;   /* exact: a multiple of 2^32 */
        limb[i] = low;
    }
}

/* bit b (0-based, weight 2^(b - XF_LSB)) of a normalised non-negative accumulator */
static int acc_bit(const int64_t *limb, int b)
{
    if (b < 0) return 0;
    return (int)((limb[b / 32] >> (b % 32)) & 1);
}

/* Round the exact accumulator to bf16, nearest-even. */
static uint16_t acc_to_bf16(int64_t *limb)
{
    acc_normalise(limb);
    uint16_t sign = 0;
    if (limb[XF_LIMBS - 1] < 0) {       /* negative: take the magnitude */
        for (int i = 0; i < XF_LIMBS; ++i) limb[i] = -limb[i];
        acc_normalise(limb);
        sign = 0x8000;
    }
    int top = -1;                       /* highest set bit */
    int hi = XF_LIMBS - 1;
    while (hi >= 0 && limb[hi] == 0) --hi;
    if (hi >= 0)
        for (int b = 31; b >= 0; --b)
            if ((limb[hi] >> b) & 1) { top = hi * 32 + b; break; }
    if (top < 0) return 0;              /* an exact zero sum is +0 */
    int exp2 = top - XF_LSB;            /* value in [2^exp2, 2^(exp2+1)) */
    assert(exp2 <= 127);                /* no overflow of the bf16 range in this use */
    /* keep 8 significant bits, or fewer in the subnormal range (lsb >= 2^-133) */
    int lsb = top - 7;
    if (lsb - XF_LSB < -133) lsb = XF_LSB - 133;
    uint32_t keep = 0;
    for (int b = top; b >= lsb; --b) keep = (keep << 1) | (uint32_t)acc_bit(limb, b);
    const int half = acc_bit(limb, lsb - 1);
    int sticky = 0;                     /* any set bit in [0, lsb - 2] */
    const int sb = lsb - 2;
    if (sb >= 0) {
        const int q = sb / 32, r = sb % 32;
        const int64_t mask = (r == 31) ? (int64_t)0xFFFFFFFF : (((int64_t)1 << (r + 1)) - 1);
        sticky = (limb[q] & mask) != 0;
        for (int i = q - 1; i >= 0 && !sticky; --i) sticky = limb[i] != 0;
    }
    if (half && (sticky || (keep & 1))) ++keep;
    /* value = keep * 2^(lsb - XF_LSB); re-encode (keep may have carried to 2^8 or 2^(n+1)) */
    int e = lsb - XF_LSB;
    while (keep >= 0x100) { keep >>= 1; ++e; }      /* only a rounding carry: the dropped bit is 0 */
    uint16_t out;
    if (keep >= 0x80) {                 /* normal: keep = 1.m * 2^7 */
        const int biased = e + 7 + 127;
        assert(biased >= 1 && biased <= 254);
        out = (uint16_t)((biased << 7) | (keep & 0x7F));
    } else {                            /* subnormal: e == -133 */
        assert(e == -133);
        out = (uint16_t)keep;
    }
    return sign | out;
}

void oracle_transform_rows(const uint16_t *x, int64_t rows, int64_t K, int64_t ld,
                           const uint16_t *T, int bs, uint16_t *y)
{
    assert(bs > 0 && bs <= 32768 && K % bs == 0);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t g = 0; g < K / bs; ++g)
            for (int j = 0; j < bs; ++j) {
                int64_t limb[XF_LIMBS] = {0};
                for (int i = 0; i < bs; ++i) {
                    int64_t sx, st;
                    int ex, et;
                    bf16_split(x[r * ld + g * bs + i], &sx, &ex);
                    bf16_split(T[(int64_t)i * bs + j], &st, &et);
                    const int64_t p = sx * st;                 /* |p| < 2^16 */
                    if (p == 0) continue;
                    const int pos = ex + et + XF_LSB;          /* >= 34 */
                    assert(pos >= 0 && pos / 32 + 1 < XF_LIMBS);
                    const int64_t v = p * ((int64_t)1 << (pos % 32));   /* |v| < 2^47 */
                    limb[pos / 32] += v;
                }
                y[r * K + g * bs + j] = acc_to_bf16(limb);
            }
}

/* ------------------------------------------------- dynamic global scale -- */
/* Per-tensor activation scale computed from the data instead of calibrated
 * ([P2] the AbsMax statistic of fusedQuantizeNv; [P1] input_global_scale_inv
 * multiplies into the block scale, R-scale).  R-dyn:
 *   amax = max |v| over the rows x K bf16 values v (the transformed y when a
 *          transform applies: the caller passes y);
 *   gs   = fl32(448 * 6 / amax), the largest finite binary32 if that
 *          overflows, and 1 when amax == 0 (every block scale is 0 then). */
float oracle_act_global_scale(const uint16_t *x, int64_t rows, int64_t K, int64_t ld)
{
    float amax = 0.0f;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k) {
            const float a = fabsf(oracle_bf16_to_f32(x[r * ld + k]));
            assert(isfinite(a));
            if (a > amax) amax = a;
        }
    if (amax == 0.0f) return 1.0f;
    const float gs = 2688.0f / amax;        /* 448 * 6, exact in binary32 */
    return isinf(gs) ? FLT_MAX : gs;
}

/* alpha = fl32(1 / fl32(gs_x * gs_w)): the GEMM output scale of [P1]. */
float oracle_alpha(float gs_x, float gs_w)
{
    const float prod = gs_x * gs_w;
    return 1.0f / prod;
}

/* ------------------------------------------------------------------ GEMM -- */
/* Reference output of the NVFP4 linear for selected rows and columns (R-gemm):
 *   out[i][j] = alpha * sum_{k<Kp} e2m1(A[m,k]) e4m3(sfA[m,k/16])
 *                                  e2m1(B[n,k]) e4m3(sfB[n,k/16])  + bias[n]
 * with m = row_idx[i], n = col_idx[j]; A is [*, Kp/2] packed, sfA [*, Kp/16]
 * linear (unswizzled); same for B; bias may be NULL.  FP64 throughout; alpha
 * is the given binary32 value ([P1] `out * layer.alpha`). */
void oracle_gemm(const uint8_t *A, const uint8_t *sfA, const uint8_t *B, const uint8_t *sfB,
                 int64_t Kp, const int64_t *row_idx, int64_t n_rows,
                 const int64_t *col_idx, int64_t n_cols, float alpha,
                 const uint16_t *bias, double *out)
{
    const int64_t nb = Kp / 16, kb = Kp / 2;
    /* dequantized copies of the selected A rows and of one B row at a time */
    double *a_deq = (double *)malloc(sizeof(double) * (size_t)(Kp * (n_rows > 0 ? n_rows : 1)));
    double *b_deq = (double *)malloc(sizeof(double) * (size_t)Kp);
    assert(a_deq && b_deq);
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t m = row_idx[i];
        for (int64_t k = 0; k < Kp; ++k) {
            uint8_t byte = A[m * kb + k / 2];
            uint8_t q = (k & 1) ? (byte >> 4) : (byte & 0xF);
            a_deq[i * Kp + k] = oracle_dec_e2m1(q) * oracle_dec_e4m3(sfA[m * nb + k / 16]);
        }
    }
    for (int64_t j = 0; j < n_cols; ++j) {
        const int64_t n = col_idx[j];
        for (int64_t k = 0; k < Kp; ++k) {
            uint8_t byte = B[n * kb + k / 2];
            uint8_t q = (k & 1) ? (byte >> 4) : (byte & 0xF);
            b_deq[k] = oracle_dec_e2m1(q) * oracle_dec_e4m3(sfB[n * nb + k / 16]);
        }
        for (int64_t i = 0; i < n_rows; ++i) {
            double acc = 0.0;                          /* k ascending */
            for (int64_t k = 0; k < Kp; ++k) acc += a_deq[i * Kp + k] * b_deq[k];
            double o = (double)alpha * acc;
            if (bias) o += (double)oracle_bf16_to_f32(bias[n]);
            out[i * n_cols + j] = o;
        }
    }
    free(a_deq);
    free(b_deq);
}

/* ------------------------------------------------------------ MXFP4 GEMM -- */
/* Reference of an MXFP4 linear (R-mx operands): out[i][j] = sum_k
 * e2m1(A[m,k]) 2^(sfA[m,k/32]-127) e2m1(B[n,k]) 2^(sfB[n,k/32]-127) + bias[n],
 * FP64, k ascending; m = row_idx[i], n = col_idx[j]; sfA [*, Kp/32] and
 * sfB [*, Kp/32] linear E8M0 codes; no global scale (MX has none), bias may
 * be NULL.  Every product is a dyadic rational of at most 4 significant bits
 * times a power of two, so the FP64 sum is exact whenever the exponent span
 * of the terms stays within 49 bits. */
void oracle_gemm_mx(const uint8_t *A, const uint8_t *sfA, const uint8_t *B, const uint8_t *sfB, int64_t Kp,
                    const int64_t *row_idx, int64_t n_rows, const int64_t *col_idx, int64_t n_cols,
                    const uint16_t *bias, double *out)
{
    const int64_t nb = Kp / 32, kb = Kp / 2;
    double *a_deq = (double *)malloc(sizeof(double) * (size_t)(Kp * (n_rows > 0 ? n_rows : 1)));
    double *b_deq = (double *)malloc(sizeof(double) * (size_t)Kp);
    assert(a_deq && b_deq);
    for (int64_t i = 0; i < n_rows; ++i) {
        const int64_t m = row_idx[i];
        for (int64_t k = 0; k < Kp; ++k) {
            const uint8_t byte = A[m * kb + k / 2];
            const uint8_t q = (k & 1) ? (byte >> 4) : (byte & 0xF);
            a_deq[i * Kp + k] = oracle_dec_e2m1(q) * oracle_dec_e8m0(sfA[m * nb + k / 32]);
        }
    }
    for (int64_t j = 0; j < n_cols; ++j) {
        const int64_t n = col_idx[j];
        for (int64_t k = 0; k < Kp; ++k) {
            const uint8_t byte = B[n * kb + k / 2];
            const uint8_t q = (k & 1) ? (byte >> 4) : (byte & 0xF);
            b_deq[k] = oracle_dec_e2m1(q) * oracle_dec_e8m0(sfB[n * nb + k / 32]);
        }
        for (int64_t i = 0; i < n_rows; ++i) {
            double acc = 0.0;
            for (int64_t k = 0; k < Kp; ++k) acc += a_deq[i * Kp + k] * b_deq[k];
            if (bias) acc += (double)oracle_bf16_to_f32(bias[n]);
            out[i * n_cols + j] = acc;
        }
    }
    free(a_deq);
    free(b_deq);
}

