"""Pins of the CPU oracle against things other than itself (host only).

Each test ties one oracle function to an independent source: the published
format tables (tests/golden/*.txt, cited there), a library routine run on a
case the definition reduces to (torch's float8_e4m3fn and bfloat16 casts,
float64 matmul), brute force over every candidate, exact rational arithmetic,
or a closed form.  The cases are chosen so that a plausible slip -- a dropped
term, a wrong sign, an off-by-one index, a transposed operand, a tie broken the
wrong way -- fails at least one of them.
"""
import fractions
import math
import os

from fractions import Fraction

import numpy as np
import pytest
import torch

from nvfp4_quantized_linear_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _f32(x):
    return float(np.float32(x))


# ------------------------------------------------------------------ E2M1 ----

def test_e2m1_decode_matches_spec_table(oracle_mod):
    for code, val in _read_table("e2m1_grid.txt"):
        got = oracle_mod.dec_e2m1(int(code, 16))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_e2m1_roundtrip_every_code(oracle_mod):
    for c in range(16):
        assert oracle_mod.enc_e2m1(oracle_mod.dec_e2m1(c)) == c


def test_e2m1_ties_and_saturation(oracle_mod):
    for v, code in _read_table("e2m1_ties.txt"):
        assert oracle_mod.enc_e2m1(float(v)) == int(code, 16), v


def test_e2m1_is_nearest_by_brute_force(oracle_mod):
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.uniform(-7, 7, 4000), rng.normal(0, 0.3, 1000)]).astype(np.float32)
    mids = (grid[1:] + grid[:-1]) / 2
    # points one binary32 ulp either side of every midpoint
    near = np.concatenate([np.nextafter(mids.astype(np.float32), np.float32(np.inf)),
                           np.nextafter(mids.astype(np.float32), np.float32(-np.inf))])
    vals = np.concatenate([vals, near, -near])
    for v in vals:
        code = oracle_mod.enc_e2m1(float(v))
        a = min(abs(float(v)), 6.0)
        err = np.abs(grid - a)
        best = np.flatnonzero(err == err.min())
        assert (code & 7) in best, (v, code)
        if abs(v) > 0:
            assert (code >> 3) == (1 if v < 0 else 0)


def test_e2m1_keeps_sign_of_values_rounding_to_zero(oracle_mod):
    assert oracle_mod.enc_e2m1(-0.1) == 0x8
    assert oracle_mod.enc_e2m1(-0.0) == 0x8
    assert oracle_mod.enc_e2m1(0.1) == 0x0


# ------------------------------------------------------------------ E4M3 ----

def test_e4m3_points_match_spec(oracle_mod):
    for v, code in _read_table("e4m3_points.txt"):
        assert oracle_mod.enc_e4m3(float(v)) == int(code, 16), v
        assert oracle_mod.dec_e4m3(int(code, 16)) == float(v)


def test_e4m3_decode_matches_torch_for_all_codes(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle_mod.dec_e4m3(c)
        if np.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == ref[c], c


def test_e4m3_roundtrip_every_finite_code(oracle_mod):
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        if c == 0x80:   # -0 encodes back to the negative zero code
            assert oracle_mod.enc_e4m3(-0.0) == 0x80
            continue
        assert oracle_mod.enc_e4m3(oracle_mod.dec_e4m3(c)) == c, hex(c)


def test_e4m3_encode_matches_torch_cast(oracle_mod):
    """torch's fp32 -> float8_e4m3fn cast is RNE; it saturates to NaN (not 448)
    above 464, so the comparison stops at 464 and saturation is pinned apart."""
    rng = np.random.default_rng(2)
    finite = np.array([oracle_mod.dec_e4m3(c) for c in range(127)])
    mids = ((finite[1:] + finite[:-1]) / 2).astype(np.float32)
    vals = np.concatenate([
        np.exp2(rng.uniform(-14, 8.85, 20000)).astype(np.float32),
        mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
        np.float32([2.0 ** -10, 2.0 ** -10 * 1.001, 2.0 ** -11, 1e-30, 448, 463.9, 464.0]),
    ])
    vals = vals[vals <= 464.0]
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.enc_e4m3(float(v)) for v in vals], np.uint8)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_e4m3_saturates_to_448(oracle_mod):
    for v in [448.0, 464.0, 464.0001, 480.0, 1e4, 3e38]:
        assert oracle_mod.enc_e4m3(v) == 0x7E
        assert oracle_mod.enc_e4m3(-v) == 0xFE


def test_e4m3_is_nearest_by_brute_force(oracle_mod):
    finite = np.array([oracle_mod.dec_e4m3(c) for c in range(127)])
    rng = np.random.default_rng(3)
    vals = np.exp2(rng.uniform(-12, 8.8, 3000)).astype(np.float32)
    for v in vals:
        code = oracle_mod.enc_e4m3(float(v))
        err = np.abs(finite - min(float(v), 448.0))
        best = np.flatnonzero(err == err.min())
        assert code in best
        if best.size == 2:   # a tie goes to the even code
            assert code % 2 == 0


# ------------------------------------------------------------------ bf16 ----

def test_bf16_rounding_matches_torch(oracle_mod):
    rng = np.random.default_rng(4)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    bits = bits[((bits >> 23) & 0xFF) != 0xFF]                      # finite only
    bits = np.concatenate([bits, np.uint32([0x3F808000, 0x3F818000, 0x7F7FFFFF, 0x00008000])])
    f = bits.view(np.float32)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.f32_to_bf16(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------- block quant ----

def _bits(a):
    return syn.bf16_bits(torch.as_tensor(a, dtype=torch.float32).to(torch.bfloat16))


def test_quant_exact_roundtrip_of_representable_blocks(oracle_mod):
    """gs = 1 and blocks made of grid values times 2^e whose absmax is 6*2^e:
    the scale is exactly 2^e and every element comes back exactly."""
    rng = np.random.default_rng(5)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    rows = []
    for e in [-8, -3, -1, 0, 1, 4, 6]:
        blk = rng.choice(grid, size=(4, 64)) * rng.choice([-1, 1], size=(4, 64))
        blk[:, ::16] = 6.0                                       # absmax of each block
        rows.append(blk * 2.0 ** e)
    x = np.concatenate(rows)
    packed, sf = oracle_mod.quantize(_bits(x), 1.0)
    deq = oracle_mod.dequantize(packed, sf, 1.0)
    assert np.array_equal(deq, x)


def test_quant_zero_block_gives_zero_scale_and_codes(oracle_mod):
    x = np.zeros((3, 48), np.float32)
    x[1, 16:32] = np.linspace(-2, 2, 16)
    packed, sf = oracle_mod.quantize(_bits(x), 7.0)
    assert sf.shape == (3, 4) and packed.shape == (3, 32)
    assert (sf[0] == 0).all() and (packed[0] == 0).all()
    assert sf[1, 1] != 0 and (sf[1, [0, 2, 3]] == 0).all()


def test_quant_calibrated_global_scale_hits_448(oracle_mod):
    """gs = 448*6/amax(x) puts the block holding amax exactly on the largest
    E4M3 scale (0x7E) and its largest element on +-6."""
    x = syn.bf16_normal((32, 256), 1.0, seed=11)
    gs = syn.global_scale(x)
    xb = syn.bf16_bits(x)
    packed, sf = oracle_mod.quantize(xb, gs)
    xf = x.float().numpy()
    r, c = np.unravel_index(np.abs(xf).argmax(), xf.shape)
    assert sf[r, c // 16] == 0x7E
    assert sf.max() == 0x7E
    byte = packed[r, c // 2]
    code = (byte >> 4) if c % 2 else (byte & 0xF)
    assert code & 7 == 7


def test_quant_elements_are_nearest_grid_points(oracle_mod):
    """Every code is the E2M1 value nearest to v*gs/e4m3(sf) (brute force), and
    every scale is the E4M3 code nearest to amax*gs/6 (brute force)."""
    x = syn.bf16_student_t(8, 96, 3, seed=12)
    gs = _f32(syn.global_scale(x) * 0.37)
    packed, sf = oracle_mod.quantize(syn.bf16_bits(x), gs)
    xf = x.float().numpy().astype(np.float64)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    e4 = np.array([oracle_mod.dec_e4m3(c) for c in range(127)])
    for r in range(xf.shape[0]):
        for b in range(xf.shape[1] // 16):
            blk = xf[r, 16 * b:16 * b + 16]
            target = np.abs(blk).max() * gs / 6
            err = np.abs(e4 - target)
            assert sf[r, b] in np.flatnonzero(err <= err.min() * (1 + 1e-6) + 1e-12)
            d = oracle_mod.dec_e4m3(int(sf[r, b]))
            for i in range(16):
                k = 16 * b + i
                byte = packed[r, k // 2]
                code = (byte >> 4) if k % 2 else (byte & 0xF)
                v = abs(blk[i]) * gs / d
                e = np.abs(grid - min(v, 6.0))
                assert (code & 7) in np.flatnonzero(e <= e.min() * (1 + 1e-6) + 1e-9), (r, k, v)


def test_quant_low_nibble_holds_even_element(oracle_mod):
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 6.0     # element 0 -> code 7
    x[0, 3] = -1.0    # element 3 -> code 0xA in the high nibble of byte 1
    packed, sf = oracle_mod.quantize(_bits(x), 1.0)
    assert packed[0, 0] == 0x07 and packed[0, 1] == 0xA0


def test_quant_pads_k_to_32_with_zeros(oracle_mod):
    rng = np.random.default_rng(6)
    x = rng.normal(size=(5, 40)).astype(np.float32) + 3.0
    packed, sf = oracle_mod.quantize(_bits(x), 10.0)
    assert packed.shape == (5, 32) and sf.shape == (5, 4)
    assert (packed[:, 20:] == 0).all()            # elements 40..63
    assert (sf[:, 3] == 0).all() and (sf[:, 2] != 0).all()
    # the partial block (32..47) takes its absmax over the 8 real values only
    ref = np.abs(_bits(x).astype(np.uint32) << 16).view(np.float32)[:, 32:40].max(axis=1)
    for r in range(5):
        assert sf[r, 2] == oracle_mod.enc_e4m3(_f32(_f32(ref[r] * 10.0) / 6.0))


def test_quant_respects_row_stride(oracle_mod):
    x = syn.bf16_normal((6, 80), 1.0, seed=13)
    full = syn.bf16_bits(x)
    p1, s1 = oracle_mod.quantize(full, 3.0, k=64)
    p2, s2 = oracle_mod.quantize(np.ascontiguousarray(full[:, :64]), 3.0)
    assert np.array_equal(p1, p2) and np.array_equal(s1, s2)


def test_quant_dequant_error_is_nvfp4_sized(oracle_mod):
    x = syn.bf16_normal((64, 512), 1.0, seed=14)
    gs = syn.global_scale(x)
    packed, sf = oracle_mod.quantize(syn.bf16_bits(x), gs)
    deq = oracle_mod.dequantize(packed, sf, gs)
    xf = x.double().numpy()
    rel = np.linalg.norm(deq - xf) / np.linalg.norm(xf)
    assert 0.03 < rel < 0.15


# --------------------------------------------------------------- swizzle ----

def test_swizzle_hand_worked_offsets(oracle_mod):
    for r, c, cp, off in _read_table("swizzle_offsets.txt"):
        assert oracle_mod.swizzle_offset(int(r), int(c), int(cp)) == int(off), (r, c, cp)


@pytest.mark.parametrize("rows,cols", [(1, 1), (16, 16), (128, 4), (130, 9), (300, 258)])
def test_swizzle_is_a_bijection_and_inverts(oracle_mod, rows, cols):
    rp, cp = oracle_mod.swizzled_shape(rows, cols)
    offs = np.array([[oracle_mod.swizzle_offset(r, c, cp) for c in range(cp)] for r in range(rp)])
    assert np.array_equal(np.sort(offs.ravel()), np.arange(rp * cp))
    rng = np.random.default_rng(rows * 1000 + cols)
    s = rng.integers(1, 255, size=(rows, cols)).astype(np.uint8)
    swz = oracle_mod.swizzle(s)
    assert np.array_equal(oracle_mod.unswizzle(swz, rows, cols), s)
    mask = np.ones(rp * cp, bool)
    mask[offs[:rows, :cols].ravel()] = False
    assert (swz[mask] == 0).all()


def test_swizzle_tile_structure(oracle_mod):
    """Four scale columns of a row are adjacent bytes; rows 32 apart are 4 bytes
    apart; consecutive rows are 16-byte lines; a 128x4 tile is 512 bytes."""
    cp = 16
    off = oracle_mod.swizzle_offset
    for r in range(0, 256, 7):
        for c in range(cp):
            if c % 4 != 3:
                assert off(r, c + 1, cp) == off(r, c, cp) + 1
            if r % 128 < 96:
                assert off(r + 32, c, cp) == off(r, c, cp) + 4
            if r % 32 != 31:
                assert off(r + 1, c, cp) == off(r, c, cp) + 16
            assert off(r, c, cp) // 512 == (r // 128) * (cp // 4) + c // 4


# ------------------------------------------------------------- transform ----

@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_hadamard_transform_is_orthogonal(bs):
    t = syn.random_hadamard_transform(bs, seed=bs).double().numpy()
    prod = t @ t.T
    err = np.abs(prod - np.eye(bs)).max()
    if bs in (16, 64):          # 1/4 and 1/8 are exact in bf16
        assert err == 0.0
    else:                       # bf16(1/sqrt(bs)) is off by at most 2^-9 relative
        assert err <= 2.0 ** -8
    h = syn.sylvester_hadamard(bs)
    assert np.array_equal(h @ h.T, bs * np.eye(bs, dtype=np.int64))


def test_transform_identity_is_exact(oracle_mod):
    x = syn.bf16_student_t(4, 64, 3, seed=15)
    eye = syn.bf16_bits(torch.eye(32).to(torch.bfloat16))
    y = oracle_mod.transform(syn.bf16_bits(x), eye, 32)
    assert np.array_equal(y, syn.bf16_bits(x))


def test_transform_signed_permutation_catches_transpose(oracle_mod):
    """T[i][j] = s_j if i == perm[j]: y[:, j] = s_j * x[:, perm[j]] inside each
    block.  A transposed T would pick x[:, inv_perm[j]] instead."""
    bs = 16
    rng = np.random.default_rng(16)
    perm = rng.permutation(bs)
    s = rng.choice([-1.0, 1.0], bs)
    t = np.zeros((bs, bs), np.float32)
    t[perm, np.arange(bs)] = s
    x = syn.bf16_normal((3, 48), 1.0, seed=16)
    y = oracle_mod.transform(syn.bf16_bits(x), syn.bf16_bits(torch.from_numpy(t).to(torch.bfloat16)), bs)
    xf = x.float().numpy()
    yf = (y.astype(np.uint32) << 16).view(np.float32)
    for g in range(3):
        blk = xf[:, g * bs:(g + 1) * bs]
        assert np.array_equal(yf[:, g * bs:(g + 1) * bs], blk[:, perm] * s)


def test_transform_pm1_inputs_give_exact_hadamard_sums(oracle_mod):
    bs = 16
    h = syn.sylvester_hadamard(bs)
    t = torch.from_numpy(h / 4.0).to(torch.bfloat16)
    rng = np.random.default_rng(17)
    x = rng.choice([-1, 1], size=(8, 64)).astype(np.int64)
    y = oracle_mod.transform(_bits(x), syn.bf16_bits(t), bs)
    yf = (y.astype(np.uint32) << 16).view(np.float32)
    exact = np.concatenate([x[:, g * bs:(g + 1) * bs] @ h for g in range(4)], axis=1) / 4.0
    assert np.array_equal(yf.astype(np.float64), exact)


def _bf16_rne_exact(q: Fraction) -> float:
    """Nearest-even bf16 value of an exact rational (8 significant bits; the
    subnormal quantum is 2^-133)."""
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    quantum = Fraction(2) ** (max(e, -126) - 7)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * float(fl * quantum)


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_transform_is_the_exactly_rounded_sum(oracle_mod, bs):
    """y = bf16_rne(exact sum_i x_i T_ij), checked with rational arithmetic on
    a small sample (brute force, no floating-point sums)."""
    x = syn.bf16_student_t(3, 128, 3, seed=18 + bs)
    t = syn.random_hadamard_transform(bs, seed=19 + bs)
    y = oracle_mod.transform(syn.bf16_bits(x), syn.bf16_bits(t), bs)
    yf = (y.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xq = [[Fraction(float(v)) for v in row] for row in x.float().numpy()]
    tq = [[Fraction(float(v)) for v in row] for row in t.float().numpy()]
    for r in range(3):
        for g in range(128 // bs):
            for j in range(bs):
                exact = sum(xq[r][g * bs + i] * tq[i][j] for i in range(bs))
                assert yf[r, g * bs + j] == _bf16_rne_exact(exact), (r, g, j)


def test_transform_rounds_the_exact_sum_not_a_running_fp32_sum(oracle_mod):
    """(1 + 2^-8 + 2^-30) / 4 lies just above the bf16 midpoint 1/4 + 2^-10, so
    it rounds up to 1/4 + 2^-9; an fp32 running sum would lose the 2^-32 term,
    land on the midpoint and round to even (1/4)."""
    bs = 16
    t = np.full((bs, bs), 0.25, np.float32)
    x = np.zeros((1, bs), np.float32)
    x[0, :4] = [1.0, 2.0 ** -9, 2.0 ** -9, 2.0 ** -30]
    y = oracle_mod.transform(_bits(x), syn.bf16_bits(torch.from_numpy(t).to(torch.bfloat16)), bs)
    assert oracle_mod.bf16_to_f32(int(y[0, 0])) == 0.25 + 2.0 ** -9
    # exact cancellation gives +0; subnormal results keep their exact value
    x[0, :4] = [1.0, -1.0, 2.0 ** -126, 0.0]
    t2 = np.eye(bs, dtype=np.float32)
    t2[:2, 0] = 1.0
    y = oracle_mod.transform(_bits(x), syn.bf16_bits(torch.from_numpy(t2).to(torch.bfloat16)), bs)
    assert y[0, 0] == 0x0000
    assert oracle_mod.bf16_to_f32(int(y[0, 2])) == 2.0 ** -126


# ------------------------------------------------------------------- MXFP4 ----

def test_e8m0_decode_closed_forms(oracle_mod):
    assert oracle_mod.dec_e8m0(127) == 1.0
    assert oracle_mod.dec_e8m0(0) == 2.0 ** -127
    assert oracle_mod.dec_e8m0(254) == 2.0 ** 127
    assert oracle_mod.dec_e8m0(130) == 8.0


def test_mx_scale_rule(oracle_mod):
    """s = floor(log2 amax) - 2: amax in [4, 8) -> 2^0 (code 127), [8, 16) -> 2^1,
    [0.5, 1) -> 2^-3; clamped to [-127, 127]; zero block -> code 0."""
    code = oracle_mod.mx_scale_code
    assert code(4.0) == code(6.0) == code(7.99) == 127
    assert code(8.0) == 128 and code(0.75) == 124
    assert code(0.0) == 0
    assert code(2.0 ** -140) == 0                                   # clamped at s = -127
    assert code(float(np.finfo(np.float32).max)) == 127 + 125       # floor(log2) = 127 -> s = 125
    for e in range(-120, 120, 7):                                    # every power of two: s = e - 2
        assert code(2.0 ** e) == e - 2 + 127


def test_mx_exact_roundtrip_of_representable_blocks(oracle_mod):
    """Blocks of 32 E2M1 grid values times 2^e with 6 * 2^e present: the scale is
    2^e and every element comes back exactly."""
    rng = np.random.default_rng(50)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float64)
    for e in (-10, -3, 0, 2, 9):
        vals = rng.choice(grid, size=(4, 64)) * rng.choice([-1.0, 1.0], size=(4, 64))
        vals[:, 0] = 6.0
        vals[:, 32] = -6.0
        x = vals * 2.0 ** e
        packed, sf = oracle_mod.quantize_mx(_bits(x))
        assert (sf == e + 127).all()
        back = np.array([[oracle_mod.dec_e2m1(int((packed[r, c // 2] >> (4 * (c % 2))) & 0xF)) for c in range(64)]
                         for r in range(4)])
        assert np.array_equal(back * 2.0 ** e, x)


def test_mx_saturates_between_6_and_8_times_the_scale(oracle_mod):
    x = np.zeros((1, 32), np.float32)
    x[0, :3] = [7.5, -7.0, 5.0]                 # amax 7.5 -> s = 0: 7.5 and -7 clamp to +-6, 5 ties to 4
    packed, sf = oracle_mod.quantize_mx(_bits(x))
    assert sf[0, 0] == 127
    assert packed[0, 0] == (0x7 | (0xF << 4)) and (packed[0, 1] & 0xF) == 0x6


def test_mx_zero_block_and_padding(oracle_mod):
    x = syn.bf16_normal((3, 40), 1.0, seed=51).float().numpy()
    x[1, :32] = 0.0
    packed, sf = oracle_mod.quantize_mx(_bits(x), k=40)
    assert packed.shape == (3, 32) and sf.shape == (3, 2)        # Kp = 64: two blocks
    assert sf[1, 0] == 0 and (packed[1, :16] == 0).all()
    assert (packed[:, 20:] == 0).all()                           # columns 40..63 are zero padding


def test_mx_elements_are_nearest_grid_points(oracle_mod):
    """Brute force: each element's code decodes to a grid point nearest to
    v * 2^-s (ties to the even code), with the block's own s."""
    x = syn.bf16_student_t(4, 128, 3, seed=52)
    xf = x.float().numpy().astype(np.float64)
    packed, sf = oracle_mod.quantize_mx(syn.bf16_bits(x))
    mags = np.array([oracle_mod.dec_e2m1(c) for c in range(8)])
    for r in range(4):
        for c in range(128):
            code = (packed[r, c // 2] >> (4 * (c % 2))) & 0xF
            t = abs(xf[r, c]) * 2.0 ** (127 - int(sf[r, c // 32]))
            d = np.abs(mags - min(t, 6.0))
            assert d[code & 7] == d.min()


def _mx_deq_exact(packed, sf, r, k):
    """Exact rational value of element (r, k) of an MXFP4 operand."""
    code = int((packed[r, k // 2] >> (4 * (k % 2))) & 0xF)
    mag = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3), Fraction(4),
           Fraction(6)][code & 7]
    e = int(sf[r, k // 32]) - 127
    v = mag * (Fraction(2) ** e)
    return -v if code & 8 else v


def test_mx_gemm_matches_exact_rational_brute_force(oracle_mod):
    """Tiny MXFP4 GEMMs against exact rational sums of the decoded operands
    (scales spread over 2^-20 .. 2^20), plus a bf16 bias."""
    rng = np.random.default_rng(55)
    m, n, k = 5, 7, 96
    xa = rng.standard_normal((m, k)) * 2.0 ** rng.integers(-20, 20, (m, 1))
    xb = rng.standard_normal((n, k)) * 2.0 ** rng.integers(-20, 20, (n, 1))
    a, sa = oracle_mod.quantize_mx(_bits(xa))
    b, sb = oracle_mod.quantize_mx(_bits(xb))
    bias = _bits(rng.standard_normal(n))
    got = oracle_mod.gemm_mx(a, sa, b, sb, bias)
    for i in range(m):
        for j in range(n):
            exact = sum(_mx_deq_exact(a, sa, i, kk) * _mx_deq_exact(b, sb, j, kk) for kk in range(k))
            exact += Fraction(oracle_mod.bf16_to_f32(int(bias[j])))
            assert got[i, j] == float(exact), (i, j)


def test_mx_gemm_matches_float64_matmul_of_dequantized(oracle_mod):
    x = syn.bf16_normal((9, 160), 1.0, seed=56)
    w = syn.bf16_normal((11, 160), 0.02, seed=57)
    a, sa = oracle_mod.quantize_mx(syn.bf16_bits(x))
    b, sb = oracle_mod.quantize_mx(syn.bf16_bits(w))
    def deq(p, s):
        codes = np.stack([p & 0xF, p >> 4], axis=-1).reshape(p.shape[0], -1)
        mags = np.array([oracle_mod.dec_e2m1(c) for c in range(16)])[codes]
        return mags * np.repeat(2.0 ** (s.astype(np.float64) - 127), 32, axis=1)
    ref = deq(a, sa) @ deq(b, sb).T
    assert np.allclose(oracle_mod.gemm_mx(a, sa, b, sb), ref, rtol=1e-12, atol=0)


def test_mx_gemm_approximates_the_bf16_product(oracle_mod):
    """Quantization error of MXFP4 on both operands: relative Frobenius error of
    the product a few percent (E2M1's 3-bit grid, power-of-two scales)."""
    x = syn.bf16_normal((16, 512), 1.0, seed=58)
    w = syn.bf16_normal((24, 512), 0.02, seed=59)
    a, sa = oracle_mod.quantize_mx(syn.bf16_bits(x))
    b, sb = oracle_mod.quantize_mx(syn.bf16_bits(w))
    ref = x.double().numpy() @ w.double().numpy().T
    got = oracle_mod.gemm_mx(a, sa, b, sb)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert 0.02 < rel < 0.25, rel


# ------------------------------------------------- dynamic global scale ----

def test_dynamic_scale_closed_forms(oracle_mod):
    """gs = 448*6/amax: amax 448 -> 6, 2688 -> 1, 1 -> 2688, 0.75 -> 3584; the
    sign of the extreme element does not matter; an all-zero tensor gives 1;
    a scale that overflows binary32 is clamped to its largest finite value."""
    def gs_of(vals):
        return oracle_mod.act_global_scale(_bits(np.array(vals, np.float32).reshape(1, -1)))
    assert gs_of([1.0, -448.0, 3.0, 0.0]) == 6.0
    assert gs_of([2688.0, 5.0]) == 1.0
    assert gs_of([0.5, -1.0]) == 2688.0
    assert gs_of([0.75, 0.5]) == 3584.0
    assert gs_of([0.0, -0.0, 0.0]) == 1.0
    tiny = np.zeros((1, 8), np.uint16)
    tiny[0, 3] = 0x0001                                      # smallest bf16 subnormal, 2^-133
    assert oracle_mod.act_global_scale(tiny) == float(np.finfo(np.float32).max)


def test_dynamic_scale_matches_the_calibration_constant(oracle_mod):
    """The oracle's per-tensor pass equals the host calibration of the input
    generators (an independent numpy computation of fl32(2688 / amax))."""
    for seed, (m, k) in enumerate([(7, 256), (64, 4104), (3, 16)]):
        x = syn.bf16_student_t(m, k, 3, seed=40 + seed)
        assert oracle_mod.act_global_scale(syn.bf16_bits(x)) == syn.global_scale(x)


def test_dynamic_scale_under_transforms_that_keep_magnitudes(oracle_mod):
    """The identity and a signed permutation leave max |y| = max |x|, so the
    transformed scale equals the plain one; a Hadamard block changes it."""
    bs = 16
    x = syn.bf16_student_t(5, 64, 3, seed=44)
    xb = syn.bf16_bits(x)
    plain = oracle_mod.act_global_scale(xb)
    eye = syn.bf16_bits(torch.eye(bs).to(torch.bfloat16))
    assert oracle_mod.act_global_scale(xb, eye, bs) == plain
    rng = np.random.default_rng(45)
    t = np.zeros((bs, bs), np.float32)
    t[rng.permutation(bs), np.arange(bs)] = rng.choice([-1.0, 1.0], bs)
    assert oracle_mod.act_global_scale(xb, syn.bf16_bits(torch.from_numpy(t).to(torch.bfloat16)), bs) == plain
    h = syn.bf16_bits(syn.random_hadamard_transform(bs, seed=46))
    assert oracle_mod.act_global_scale(xb, h, bs) != plain


def test_dynamic_scale_puts_the_max_block_on_448(oracle_mod):
    x = syn.bf16_normal((16, 512), 1.0, seed=47)
    xb = syn.bf16_bits(x)
    gs = oracle_mod.act_global_scale(xb)
    _, sf = oracle_mod.quantize(xb, gs)
    assert sf.max() == 0x7E


def test_alpha_closed_forms(oracle_mod):
    assert oracle_mod.alpha(2.0, 4.0) == 0.125
    assert oracle_mod.alpha(6.0, 1.0) == float(np.float32(1.0) / np.float32(6.0))
    assert oracle_mod.alpha(3.0, 0.5) == float(np.float32(2.0) / np.float32(3.0))


# ------------------------------------------------------------------ GEMM ----

def _quantized_operands(oracle_mod, m, n, k, seed):
    x = syn.bf16_normal((m, k), 1.0, seed)
    w = syn.bf16_normal((n, k), 0.02, seed + 1)
    gx, gw = syn.global_scale(x), syn.global_scale(w)
    a, sa = oracle_mod.quantize(syn.bf16_bits(x), gx)
    b, sb = oracle_mod.quantize(syn.bf16_bits(w), gw)
    return a, sa, b, sb, gx, gw


def test_gemm_matches_exact_rational_brute_force(oracle_mod):
    m, n, k = 3, 5, 40
    a, sa, b, sb, gx, gw = _quantized_operands(oracle_mod, m, n, k, seed=20)
    alpha = syn.alpha_of(gx, gw)
    bias = syn.bf16_normal((n,), 0.1, seed=21)
    out = oracle_mod.gemm(a, sa, b, sb, alpha, syn.bf16_bits(bias))
    F = fractions.Fraction
    grid = [F(0), F(1, 2), F(1), F(3, 2), F(2), F(3), F(4), F(6)]

    def e2m1(q):
        return -grid[q & 7] if q & 8 else grid[q & 7]

    def e4m3(c):
        return F(oracle_mod.dec_e4m3(c))

    kp = a.shape[1] * 2
    for i in range(m):
        for j in range(n):
            acc = F(0)
            for kk in range(kp):
                qa = (a[i, kk // 2] >> 4) if kk % 2 else (a[i, kk // 2] & 0xF)
                qb = (b[j, kk // 2] >> 4) if kk % 2 else (b[j, kk // 2] & 0xF)
                acc += e2m1(qa) * e4m3(sa[i, kk // 16]) * e2m1(qb) * e4m3(sb[j, kk // 16])
            ref = F(alpha) * acc + F(float(bias[j].float()))
            assert abs(float(ref) - out[i, j]) <= 1e-12 * max(1.0, abs(float(ref)))


def test_gemm_matches_float64_matmul_of_dequantized(oracle_mod):
    m, n, k = 37, 70, 200
    a, sa, b, sb, gx, gw = _quantized_operands(oracle_mod, m, n, k, seed=22)
    alpha = syn.alpha_of(gx, gw)
    out = oracle_mod.gemm(a, sa, b, sb, alpha)
    da = oracle_mod.dequantize(a, sa, 1.0)
    db = oracle_mod.dequantize(b, sb, 1.0)
    ref = alpha * (torch.from_numpy(da) @ torch.from_numpy(db).T).numpy()
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    # row / column selection indexes the same entries
    rows, cols = np.array([36, 0, 5]), np.array([69, 1, 33, 2])
    sub = oracle_mod.gemm(a, sa, b, sb, alpha, rows=rows, cols=cols)
    assert np.array_equal(sub, out[np.ix_(rows, cols)])


def test_gemm_approximates_the_bf16_product(oracle_mod):
    """The dequantized product with alpha = 1/(gs_x gs_w) lands near x @ w.T."""
    m, n, k = 16, 64, 512
    x = syn.bf16_normal((m, k), 1.0, 23)
    w = syn.bf16_normal((n, k), 0.02, 24)
    gx, gw = syn.global_scale(x), syn.global_scale(w)
    a, sa = oracle_mod.quantize(syn.bf16_bits(x), gx)
    b, sb = oracle_mod.quantize(syn.bf16_bits(w), gw)
    out = oracle_mod.gemm(a, sa, b, sb, syn.alpha_of(gx, gw))
    ref = (x.double() @ w.double().T).numpy()
    rel = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    assert rel < 0.2


def test_gemm_exact_integer_case(oracle_mod):
    """Unit scales, gs = 1, alpha = 1: integer-valued products whose sums are
    exact; the oracle must return the integer matmul exactly."""
    rng = np.random.default_rng(25)
    grid = np.array([0, 1, 2, 3, 4, 6])
    xa = rng.choice(grid, (9, 64)) * rng.choice([-1, 1], (9, 64))
    xb = rng.choice(grid, (11, 64)) * rng.choice([-1, 1], (11, 64))
    xa[:, ::16] = 6
    xb[:, ::16] = 6
    a, sa = oracle_mod.quantize(_bits(xa), 1.0)
    b, sb = oracle_mod.quantize(_bits(xb), 1.0)
    assert (sa == 0x38).all() and (sb == 0x38).all()      # scale 1.0
    out = oracle_mod.gemm(a, sa, b, sb, 1.0)
    assert np.array_equal(out, (xa.astype(np.int64) @ xb.astype(np.int64).T).astype(np.float64))
