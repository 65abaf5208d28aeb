"""Pins of the CPU oracle against what the definitions and the mathematics fix.

Each test targets a plausible mistake (a wrong sign, a swapped nibble, a transposed
operand, an FMA where two roundings are required, a wrong tie rule) and must fail
if the oracle made it.  None of them re-derives an expected value with the oracle's
own formula: expected values are literals, closed forms, library routines (numpy
matmul, math.erf) or constructions whose answer is known by design.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import codebooks

CODE4 = codebooks.nf4_code4()
CODE8 = codebooks.dynamic_code8()
LIN8 = codebooks.linear_code8()


# --------------------------------------------------------------- codebooks ----

def test_code4_shape_endpoints_zero():
    # The NF4 codebook: 16 levels, an exact zero, endpoints -1 and +1.
    assert CODE4.dtype == np.float32 and CODE4.shape == (16,)
    assert np.all(np.diff(CODE4) > 0)
    assert CODE4[0] == -1.0 and CODE4[15] == 1.0 and CODE4[7] == 0.0
    assert (CODE4 < 0).sum() == 7 and (CODE4 > 0).sum() == 8


def _phi(x):
    return 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))


def _phi_inv_bisect(p):
    lo, hi = -10.0, 10.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if _phi(mid) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def test_code4_levels_are_normal_quantiles():
    # Each non-zero level times the normaliser is a standard-normal quantile at the
    # probabilities of the NormalFloat construction; checked through the forward CDF
    # (math.erf) and a bisection, not through the oracle's ndtri.
    delta = 0.5 * (1 / 30 + 1 / 32)
    z_top = _phi_inv_bisect(1 - delta)
    p_pos = np.linspace(1 - delta, 0.5, 9)[:-1][::-1]  # ascending, 8 values
    p_neg = np.linspace(1 - delta, 0.5, 8)[:-1]        # 7 values, largest first
    for j, p in zip(range(8, 16), p_pos):
        assert abs(_phi(float(CODE4[j]) * z_top) - p) < 2e-7, j
    for j, p in zip(range(0, 7), p_neg):
        assert abs(_phi(-float(CODE4[j]) * z_top) - p) < 2e-7, j


FP4 = codebooks.fp4_code4()


def test_fp4_levels_are_e2m1_scaled_to_unit():
    # E2M1: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (exponent bias 1, one mantissa
    # bit, subnormals at exponent 0), divided by the largest; ascending with -0
    # before +0.
    assert FP4.dtype == np.float32 and FP4.shape == (16,)
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for i, m in enumerate(e2m1):
        assert abs(float(FP4[8 + i]) * 6.0 - m) <= 4e-7 * max(m, 1.0), i
        assert abs(float(FP4[7 - i]) * 6.0 + m) <= 4e-7 * max(m, 1.0), i
    # levels that are dyadic are exact; the rest are the nearest fp32
    assert FP4[15] == 1.0 and FP4[0] == -1.0 and FP4[13] == 0.5 and FP4[11] == 0.25
    assert FP4[14] == np.float32(2.0 / 3.0) and FP4[9] == np.float32(1.0 / 12.0)
    # signed zero pair; every other neighbour strictly increasing; mirror symmetry
    assert FP4[7] == 0.0 and np.signbit(FP4[7]) and FP4[8] == 0.0 and not np.signbit(FP4[8])
    d = np.diff(FP4.astype(np.float64))
    assert np.all(d[np.arange(15) != 7] > 0) and d[7] == 0
    np.testing.assert_array_equal(FP4[::-1].view(np.uint32), (-FP4).view(np.uint32))


def test_fp4_round_trip_ties_and_zero_block():
    # Codebook-aligned blocks come back exactly (index 8, +0, is never produced:
    # an exact zero maps to index 7, -0, the first level equal to it).
    rng = np.random.default_rng(11)
    idx = rng.choice([j for j in range(16) if j != 8], size=(64, 64))
    idx[:, 0] = 15
    a = np.float32(0.75)
    w = (FP4[idx] * a).astype(np.float32)
    packed, absmax = oracle.quantize_nf4(w, FP4, 64)
    assert np.all(absmax == a)
    q = np.stack([packed >> 4, packed & 15], axis=1).reshape(-1)
    np.testing.assert_array_equal(q, idx.reshape(-1))
    st = oracle.QuantState(w.shape, 64, packed, absmax, FP4)
    np.testing.assert_array_equal(oracle.dequantize(st, "f32"), w)
    # Midpoint of 0 and 1/12 (exact: half an fp32) goes to the lower index (+0);
    # just above goes to 1/12; a small negative value to -0; 0 itself to -0.
    mid = np.float32(FP4[9] / np.float32(2))
    w = np.array([1.0, mid, np.nextafter(mid, np.float32(1)), np.float32(-1e-3), 0.0, 0.0],
                 np.float32)
    packed, _ = oracle.quantize_nf4(w, FP4, blocksize=6)
    assert packed.tolist() == [(15 << 4) | 8, (9 << 4) | 7, (7 << 4) | 7]
    packed, absmax = oracle.quantize_nf4(np.zeros(64, np.float32), FP4)
    assert absmax.tolist() == [0.0] and packed.tolist() == [0x77] * 32


E4M3 = codebooks.e4m3_code8()


def test_e4m3_levels():
    # 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, subnormals at exponent 0,
    # no NaN/inf codes; the largest magnitude (1.875 * 2**8 = 480) scaled to 1.
    assert E4M3.dtype == np.float32 and E4M3.shape == (256,)
    assert E4M3[255] == 1.0 and E4M3[0] == -1.0
    assert E4M3[254] == np.float32(448.0 / 480.0)          # e = 15, m = 6
    assert E4M3[247] == np.float32(0.5)                      # e = 14, m = 7: 240 / 480
    assert E4M3[136] == np.float32(2.0 ** -6 / 480.0)        # smallest normal
    assert E4M3[129] == np.float32(2.0 ** -9 / 480.0)        # smallest subnormal
    assert E4M3[127] == 0.0 and np.signbit(E4M3[127]) and E4M3[128] == 0.0 and not np.signbit(E4M3[128])
    d = np.diff(E4M3.astype(np.float64))
    assert np.all(d[np.arange(255) != 127] > 0) and d[127] == 0
    np.testing.assert_array_equal(E4M3[::-1].view(np.uint32), (-E4M3).view(np.uint32))
    # within each binade of the normals, 8 equally spaced levels: spacing 2**(e-10) / 480
    pos = E4M3[128:].astype(np.float64) * 480.0
    for e in range(1, 16):
        lv = pos[8 * e:8 * e + 8]
        assert np.allclose(np.diff(lv), 2.0 ** (e - 10), rtol=1e-6), e
        assert abs(lv[0] - 2.0 ** (e - 7)) <= 1e-6 * 2.0 ** (e - 7)


@pytest.mark.parametrize("table", ["dynamic", "e4m3"])
def test_8bit_round_trip_zero_block_and_ties(table):
    code = CODE8 if table == "dynamic" else E4M3
    zero = int(np.argmax(code == 0.0))  # first exact zero
    rng = np.random.default_rng(12)
    choices = [j for j in range(256) if code[j] != 0.0 or j == zero]
    idx = rng.choice(choices, size=(32, 64))
    idx[:, 0] = 255
    a = np.float32(1.25)
    w = (code[idx] * a).astype(np.float32)
    q, absmax = oracle.quantize_8bit(w, code, 64)
    assert np.all(absmax == a)
    np.testing.assert_array_equal(q, idx.reshape(-1))
    st = oracle.QuantState(w.shape, 64, q, absmax, code, bits=8)
    np.testing.assert_array_equal(oracle.dequantize(st, "f32"), w)
    q0, a0 = oracle.quantize_8bit(np.zeros(64, np.float32), code, 64)
    assert a0.tolist() == [0.0] and q0.tolist() == [zero] * 64
    # Around the fp64 midpoint of two adjacent positive levels: the fp32 values
    # just below and just above go to the lower and upper level, and a midpoint
    # that is itself an fp32 value goes to the lower level (the tie rule; the
    # 4-bit tests pin it with constructed ties).
    for j in (200, 230, 250):
        m64 = (np.float64(code[j]) + np.float64(code[j + 1])) / 2
        m32 = np.float32(m64)
        below = m32 if np.float64(m32) < m64 else np.nextafter(m32, np.float32(0))
        above = m32 if np.float64(m32) > m64 else np.nextafter(m32, np.float32(2))
        vals = [1.0, below, above] + ([m32] if np.float64(m32) == m64 else [])
        q, _ = oracle.quantize_8bit(np.array(vals, np.float32), code, len(vals))
        assert q.tolist() == [255, j, j + 1] + ([j] if len(vals) == 4 else []), (table, j)


def test_int8_storage_fidelity_beats_nf4_by_more_than_4x():
    # fork PR "Experts trainability", commit 1: int8 blockwise mean-abs
    # reconstruction error is more than 4x lower than nf4 on the same weights.
    rng = np.random.default_rng(13)
    w = (rng.standard_normal((256, 1024)) * 0.02).astype(np.float32)
    e4 = np.abs(oracle.dequantize(oracle.quantize(w, CODE4, 64), "f32") - w).mean()
    e8 = np.abs(oracle.dequantize(oracle.quantize(w, CODE8, 64), "f32") - w).mean()
    ef = np.abs(oracle.dequantize(oracle.quantize(w, E4M3, 64), "f32") - w).mean()
    assert e8 * 4 < e4, (e8, e4)
    assert ef < e4 and e8 < ef


def test_code8_dynamic_map_structure():
    assert CODE8.shape == (256,) and np.all(np.diff(CODE8) > 0)
    assert 0.0 in CODE8 and CODE8.max() == 1.0
    pos = CODE8[(CODE8 > 0) & (CODE8 < 1)]
    neg = CODE8[CODE8 < 0]
    assert pos.size == 127 and neg.size == 127
    np.testing.assert_array_equal(np.sort(-neg), pos)  # mirror image
    # 2**e fraction values in each decade (1e-7, 1e-6), ..., (0.1, 1)
    for e in range(7):
        lo, hi = 10.0 ** (e - 7), 10.0 ** (e - 6)
        assert ((pos > lo) & (pos < hi)).sum() == 2 ** e
    # the top decade: midpoints of 64 equal bins of [0.1, 1]
    assert abs(float(pos.max()) - (1.0 - 0.9 / 128)) < 1e-7


def test_linear_code8():
    assert LIN8[0] == -1.0 and LIN8[128] == 0.0 and np.all(np.diff(LIN8) > 0)


# ----------------------------------------------------------------- bf16 ----

@pytest.mark.parametrize("bits,expect", [
    (0x3F808000, 0x3F80),  # tie, even stays
    (0x3F818000, 0x3F82),  # tie, odd rounds up
    (0x3F808001, 0x3F81),  # above tie
    (0x3F807FFF, 0x3F80),  # below tie
    (0xBF818000, 0xBF82),  # negative tie
    (0x7F7FFFFF, 0x7F80),  # rounds to +inf
    (0x00000000, 0x0000),
    (0x80000000, 0x8000),
])
def test_bf16_round_to_nearest_even(oracle_lib, bits, expect):
    f = np.array([bits], dtype=np.uint32).view(np.float32)[0]
    assert oracle_lib.oracle_bf16_from_f32(float(f)) == expect


# -------------------------------------------------------- quantisation ----

def test_packing_hand_built_bytes():
    # indices 15, 0, 7, 12 at absmax 1: even element in the high nibble.
    w = np.array([1.0, -1.0, 0.0, CODE4[12]], dtype=np.float32)
    packed, absmax = oracle.quantize_nf4(w, CODE4, blocksize=4)
    assert packed.tolist() == [0xF0, 0x7C]
    assert absmax.tolist() == [1.0]
    # odd length: the missing low nibble is zero
    packed, _ = oracle.quantize_nf4(w[:3], CODE4, blocksize=4)
    assert packed.tolist() == [0xF0, 0x70]


def test_dequantize_hand_built_bytes():
    st = oracle.QuantState((4,), 4, np.array([0xF0, 0x7C], np.uint8), np.array([2.0], np.float32), CODE4)
    out = oracle.dequantize(st, "f32")
    assert out.tolist() == [2.0, -2.0, 0.0, float(np.float32(CODE4[12]) * np.float32(2.0))]


def _aligned_blocks(rng, nblocks, bs=64):
    """Blocks whose values are exactly fp32(code4[j] * a), with one value at +-a."""
    idx = rng.integers(0, 16, size=(nblocks, bs))
    pos = rng.integers(0, bs, size=nblocks)
    idx[np.arange(nblocks), pos] = rng.choice([0, 15], size=nblocks)
    a = (rng.uniform(0.5, 1.0, size=nblocks) * 2.0 ** rng.integers(-20, 5, size=nblocks)).astype(np.float32)
    w = (CODE4[idx] * a[:, None]).astype(np.float32)
    return w, idx, a


def test_round_trip_codebook_aligned_blocks():
    rng = np.random.default_rng(1)
    w, idx, a = _aligned_blocks(rng, 200)
    packed, absmax = oracle.quantize_nf4(w, CODE4, 64)
    np.testing.assert_array_equal(absmax, a)
    hi, lo = packed >> 4, packed & 15
    q = np.stack([hi, lo], axis=1).reshape(-1)
    np.testing.assert_array_equal(q, idx.reshape(-1))
    st = oracle.QuantState(w.shape, 64, packed, absmax, CODE4)
    np.testing.assert_array_equal(oracle.dequantize(st, "f32"), w)


def test_absmax_scaling_invariant():
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((64, 64)) * 0.02).astype(np.float32)
    p0, a0 = oracle.quantize_nf4(w, CODE4)
    for k in (-3, 1, 7):
        pk, ak = oracle.quantize_nf4(w * np.float32(2.0 ** k), CODE4)
        np.testing.assert_array_equal(pk, p0)
        np.testing.assert_array_equal(ak, a0 * np.float32(2.0 ** k))
    # every dequantised block reaches its absmax exactly
    st = oracle.QuantState(w.shape, 64, p0, a0, CODE4)
    wf = oracle.dequantize(st, "f32").reshape(-1, 64)
    np.testing.assert_array_equal(np.abs(wf).max(axis=1), a0)


def test_sign_flip_mirrors_where_codebook_is_symmetric():
    # Levels k/7 for k = -7..7 are symmetric about 0; the 16th level (-8/7) lies
    # outside [-1, 1] and is never nearest.  Negating a block must then negate
    # every dequantised value exactly.
    sym = np.array([-8 / 7] + [k / 7 for k in range(-7, 8)], np.float32)
    rng = np.random.default_rng(3)
    w = rng.uniform(-0.8, 0.8, size=(8, 64)).astype(np.float32)
    w[:, 0] = 0.9
    p, a = oracle.quantize_nf4(w, sym)
    pn, an = oracle.quantize_nf4(-w, sym)
    np.testing.assert_array_equal(a, an)
    d = oracle.dequantize(oracle.QuantState(w.shape, 64, p, a, sym), "f32")
    dn = oracle.dequantize(oracle.QuantState(w.shape, 64, pn, an, sym), "f32")
    np.testing.assert_array_equal(d, -dn)
    assert not np.any((p >> 4) == 0) and not np.any((p & 15) == 0)


def test_tie_goes_to_lower_index_and_nearest_otherwise():
    code = np.array([-1, -.875, -.75, -.625, -.5, -.375, -.25, 0, .125, .25, .375, .5, .625, .75, .875, 1],
                    np.float32)
    mid = np.float32(0.0625)  # exact midpoint of levels 7 (0) and 8 (0.125)
    above = np.nextafter(mid, np.float32(1))
    below = np.nextafter(mid, np.float32(0))
    w = np.array([1.0, mid, above, below], np.float32)
    packed, _ = oracle.quantize_nf4(w, code, blocksize=4)
    assert packed.tolist() == [(15 << 4) | 7, (8 << 4) | 7]


def test_zero_block():
    w = np.zeros(64, np.float32)
    packed, absmax = oracle.quantize_nf4(w, CODE4)
    assert absmax.tolist() == [0.0]
    assert packed.tolist() == [0x77] * 32
    st = oracle.QuantState(w.shape, 64, packed, absmax, CODE4)
    assert np.all(oracle.dequantize(st, "f32") == 0)


def test_short_last_block():
    rng = np.random.default_rng(4)
    w = (rng.standard_normal(64 * 3 + 17) * 0.02).astype(np.float32)
    packed, absmax = oracle.quantize_nf4(w, CODE4)
    assert absmax.size == 4 and packed.size == (w.size + 1) // 2
    assert absmax[3] == np.abs(w[192:]).max()
    # the last block is quantised on its own: same result as quantising it alone
    p_tail, a_tail = oracle.quantize_nf4(w[192:], CODE4)
    assert a_tail[0] == absmax[3]
    np.testing.assert_array_equal(p_tail, packed[96:])


def test_quantisation_error_bound():
    # nearest-level rounding: |w - wf| <= a * (largest half-gap of the codebook) + fp32 slack
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((32, 256)) * 0.02).astype(np.float32)
    st = oracle.quantize(w, CODE4)
    wf = oracle.dequantize(st, "f32").reshape(-1, 64)
    a = st.absmax[:, None]
    half_gap = float(np.max(np.diff(CODE4.astype(np.float64))) / 2)
    err = np.abs(wf - w.reshape(-1, 64))
    assert np.all(err <= a * (half_gap + 1e-6))


# ------------------------------------------------- double quantisation ----

def test_mean_offset_exact_for_exact_sums():
    absmax = np.array([0.5, 1.0, 1.5, 2.0] * 300, np.float32)  # 1200 values: two chunks
    _, _, off = oracle.double_quant(absmax, LIN8)
    assert off.tolist() == [1.25]


def test_double_quant_round_trip_linear_map():
    # residuals k/128 * na with sum 0 and max |r| = na: offset, na and every code exact.
    ks = [-128, 64, 64, 5, -5, 17, -17, 127, -127, 0, 33, -33]
    na = np.float32(0.125)
    r = np.array(ks, np.float64) / 128.0 * float(na)
    absmax = (1.0 + r).astype(np.float32)
    aq, nested, off = oracle.double_quant(absmax, LIN8)
    assert off.tolist() == [1.0] and nested.tolist() == [0.125]
    assert aq.tolist() == [k + 128 for k in ks]
    dec = oracle.decode_absmax(aq, nested, off, LIN8)
    np.testing.assert_array_equal(dec, absmax)


def test_double_quant_nested_blocks_and_error_bound():
    rng = np.random.default_rng(6)
    absmax = rng.uniform(0.01, 0.08, size=256 * 5 + 37).astype(np.float32)
    aq, nested, off = oracle.double_quant(absmax, CODE8)
    assert nested.size == 6
    r = absmax.astype(np.float64) - float(off[0])
    for c in range(6):
        blk = slice(256 * c, min(256 * (c + 1), absmax.size))
        assert nested[c] == np.float32(np.abs((absmax[blk] - off[0]).astype(np.float32)).max())
    dec = oracle.decode_absmax(aq, nested, off, CODE8).astype(np.float64)
    # nearest level of an 8-bit map: error at most half the local gap times na (+ rounding)
    gaps = np.diff(CODE8.astype(np.float64)).max()
    na = nested.astype(np.float64).repeat(256)[:absmax.size]
    assert np.all(np.abs(dec - absmax) <= na * (gaps / 2 + 1e-6) + 1e-7)
    del r


def test_decode_absmax_two_roundings_no_fma():
    # a*b+c with a = b = 1 + 2^-12, c = -1: two roundings give 2^-11, an FMA gives 2^-11 + 2^-24.
    a = np.float32(1.0 + 2.0 ** -12)
    code8 = np.linspace(-1.0, 1.0, 256).astype(np.float32)
    code8[128] = 0.0
    code8 = np.sort(code8)
    code8[255] = a
    dec = oracle.decode_absmax(np.array([255], np.uint8), np.array([a], np.float32),
                               np.array([-1.0], np.float32), code8)
    assert dec.tolist() == [2.0 ** -11]


def test_zero_nested_block_maps_to_exact_zero_code():
    absmax = np.full(256, 0.03125, np.float32)
    aq, nested, off = oracle.double_quant(absmax, CODE8)
    assert off.tolist() == [0.03125] and nested.tolist() == [0.0]
    assert np.all(CODE8[aq] == 0.0)
    np.testing.assert_array_equal(oracle.decode_absmax(aq, nested, off, CODE8), absmax)


# ------------------------------------------------------------- products ----

def _bf16(a):
    return oracle.f32_to_bf16_bits(np.asarray(a, np.float32))


def _small_weight(rng, N, K, dq=False):
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    st = oracle.quantize(w, CODE4, 64, dq, CODE8)
    return oracle.dequantize(st, "bf16")


@pytest.mark.parametrize("M,N,K", [(1, 1, 64), (3, 5, 128), (8, 8, 192), (7, 2, 64)])
def test_fwd_dgrad_brute_force_vs_numpy(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    wb = _small_weight(rng, N, K)
    x = _bf16(rng.standard_normal((M, K)))
    gy = _bf16(rng.standard_normal((M, N)))
    W = oracle.bf16_bits_to_f32(wb).astype(np.float64)
    X = oracle.bf16_bits_to_f32(x).astype(np.float64)
    GY = oracle.bf16_bits_to_f32(gy).astype(np.float64)
    np.testing.assert_allclose(oracle.linear_fwd(x, wb), X @ W.T, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(oracle.linear_dgrad(gy, wb), GY @ W, rtol=1e-12, atol=1e-14)


def test_identity_probe_is_exact():
    rng = np.random.default_rng(7)
    N, K = 24, 128
    wb = _small_weight(rng, N, K, dq=True)
    eye_k = _bf16(np.eye(K))
    eye_n = _bf16(np.eye(N))
    np.testing.assert_array_equal(oracle.linear_fwd(eye_k, wb), oracle.bf16_bits_to_f32(wb).T)
    np.testing.assert_array_equal(oracle.linear_dgrad(eye_n, wb), oracle.bf16_bits_to_f32(wb))


def test_constant_input_closed_form():
    rng = np.random.default_rng(8)
    wb = _small_weight(rng, 16, 256)
    ones = _bf16(np.ones((3, 256)))
    y = oracle.linear_fwd(ones, wb)
    rowsum = oracle.bf16_bits_to_f32(wb).astype(np.float64).sum(axis=1)
    np.testing.assert_allclose(y, np.broadcast_to(rowsum, y.shape), rtol=1e-12, atol=1e-15)


def test_dgrad_is_fwd_with_transposed_operand_exact():
    # Integer-valued bf16 data: every partial sum is exact, so any order gives the
    # same value and a transposed or shifted index shows as a mismatch.
    rng = np.random.default_rng(9)
    M, N, K = 5, 12, 64
    wb = _bf16(rng.integers(-8, 9, size=(N, K)))
    gy = _bf16(rng.integers(-8, 9, size=(M, N)))
    gx = oracle.linear_dgrad(gy, wb)
    np.testing.assert_array_equal(gx, oracle.linear_fwd(gy, np.ascontiguousarray(wb.T)))
    exact = oracle.bf16_bits_to_f32(gy).astype(np.int64) @ oracle.bf16_bits_to_f32(wb).astype(np.int64)
    np.testing.assert_array_equal(gx, exact.astype(np.float64))


def test_row_subset_matches_full():
    rng = np.random.default_rng(10)
    wb = _small_weight(rng, 8, 128)
    x = _bf16(rng.standard_normal((6, 128)))
    full = oracle.linear_fwd(x, wb)
    rows = np.array([5, 0, 3])
    np.testing.assert_array_equal(oracle.linear_fwd(x, wb, rows=rows), full[rows])
    gy = _bf16(rng.standard_normal((6, 8)))
    fullg = oracle.linear_dgrad(gy, wb)
    np.testing.assert_array_equal(oracle.linear_dgrad(gy, wb, rows=rows), fullg[rows])


def test_fp32_accumulation_is_well_inside_tolerance():
    # The GPU accumulates in fp32 and rounds to bf16; that arithmetic, emulated with
    # numpy, must sit far inside the 5e-3 relative Frobenius bound against fp64.
    rng = np.random.default_rng(11)
    M, N, K = 16, 64, 2048
    wb = _small_weight(rng, N, K)
    x = _bf16(rng.standard_normal((M, K)))
    ref = oracle.linear_fwd(x, wb)
    y32 = (oracle.bf16_bits_to_f32(x) @ oracle.bf16_bits_to_f32(wb).T).astype(np.float32)
    y16 = oracle.bf16_bits_to_f32(_bf16(y32)).astype(np.float64)
    rel = np.linalg.norm(y16 - ref) / np.linalg.norm(ref)
    assert rel < 5e-3 / 2
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.all(np.abs(y16 - ref) <= 1e-2 * (np.abs(ref) + rms))


def test_grouped_matches_per_expert_numpy():
    rng = np.random.default_rng(12)
    E, N, K = 4, 8, 64
    wbs = np.stack([_small_weight(rng, N, K) for _ in range(E)])
    offsets = np.array([0, 3, 3, 7, 10])
    x = _bf16(rng.standard_normal((10, K)))
    y = oracle.grouped_fwd(x, offsets, wbs)
    X = oracle.bf16_bits_to_f32(x).astype(np.float64)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        W = oracle.bf16_bits_to_f32(wbs[e]).astype(np.float64)
        np.testing.assert_allclose(y[a:b], X[a:b] @ W.T, rtol=1e-12, atol=1e-14)
    gy = _bf16(rng.standard_normal((10, N)))
    gx = oracle.grouped_dgrad(gy, offsets, wbs)
    GY = oracle.bf16_bits_to_f32(gy).astype(np.float64)
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        W = oracle.bf16_bits_to_f32(wbs[e]).astype(np.float64)
        np.testing.assert_allclose(gx[a:b], GY[a:b] @ W, rtol=1e-12, atol=1e-14)


def test_mean_offset_sums_in_fp64():
    # 2^24 followed by 1023 ones: an fp32 running sum loses every 1 (mean 16384.0);
    # the fp64 sum keeps them, and (2^24 + 1023) / 1024 rounds to 16385.0 in fp32.
    absmax = np.array([2.0 ** 24] + [1.0] * 1023, np.float32)
    _, _, off = oracle.double_quant(absmax, LIN8)
    assert off.tolist() == [16385.0]


# ------------------------------------------------------------- fp16 dtype ----

@pytest.mark.parametrize("value,bits", [
    (1.0, 0x3C00), (65504.0, 0x7BFF), (65520.0, 0x7C00), (65519.996, 0x7BFF),
    (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000), (1.5 * 2.0 ** -25, 0x0001), (3 * 2.0 ** -25, 0x0002),
    (1 + 2.0 ** -11, 0x3C00), (1 + 3 * 2.0 ** -11, 0x3C02), (-2.5, 0xC100), (0.1, 0x2E66),
    (6.1e-5, 0x03FF), (1e-8, 0x0000)])
def test_f16_round_to_nearest_even_literals(value, bits):
    # ties to even at the subnormal and normal boundaries, overflow at the half-ulp
    # above 65504, subnormals down to 2^-24
    assert int(oracle.f16_bits(np.array([value], np.float32))[0]) == bits


def test_f16_rounding_matches_numpy_and_decodes_every_pattern():
    rng = np.random.default_rng(14)
    r = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 12, 200000))).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = r.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(oracle.f16_bits(r), ref)
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = (pats & 0x7C00) != 0x7C00
    dec = np.array([oracle.lib().oracle_f32_from_f16(int(h)) for h in pats[finite]], np.float32)
    np.testing.assert_array_equal(dec, pats[finite].view(np.float16).astype(np.float32))
    np.testing.assert_array_equal(oracle.f16_bits(dec), pats[finite])


def test_f16_products_brute_force_vs_numpy():
    rng = np.random.default_rng(15)
    x = rng.standard_normal((5, 40)).astype(np.float16)
    w = (rng.standard_normal((7, 40)) * 0.05).astype(np.float16)
    gy = rng.standard_normal((5, 7)).astype(np.float16)
    xb, wb, gb = x.view(np.uint16), w.view(np.uint16), gy.view(np.uint16)
    np.testing.assert_allclose(oracle.linear_fwd(xb, wb, dtype="f16"),
                               x.astype(np.float64) @ w.astype(np.float64).T, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.linear_dgrad(gb, wb, dtype="f16"),
                               gy.astype(np.float64) @ w.astype(np.float64), rtol=1e-13, atol=1e-13)


# ------------------------------------------------------- expert epilogues ----

def test_interleave_gate_up_layout():
    E, H, K = 2, 128, 3
    gate = np.arange(E * H * K, dtype=np.float32).reshape(E * H, K)
    up = -gate - 1
    w = oracle.interleave_gate_up(gate, up, E)
    assert w.shape == (E * 2 * H, K)
    for e in range(E):
        for c in range(H):  # output column c of expert e
            r = e * 2 * H + 128 * (c // 64) + c % 64
            np.testing.assert_array_equal(w[r], gate[e * H + c])
            np.testing.assert_array_equal(w[r + 64], up[e * H + c])


def test_swiglu_bias_and_row_scale_literals():
    # One expert, N = 128 (64 gate + 64 up rows), K = 64, one-hot weights: the
    # accumulator of row t, column n is x[t, n % 64], so g and u are chosen by x.
    N, K = 128, 64
    w = np.zeros((1, N, K), np.float32)
    for n in range(N):
        w[0, n, n % 64] = 1.0
    wb = _bf16(w)
    x = np.zeros((2, K), np.float32)
    x[0, :4] = [0.0, 1.0, -1.0, 20.0]
    x[1, :4] = [2.0, 2.0, 2.0, 2.0]
    xb = _bf16(x)
    off = np.array([0, 2])
    bias = np.zeros(N, np.float32)
    bias[64:68] = 1.0              # up = x + 1
    h = oracle.grouped_fwd_epilogue(xb, off, wb, bias=bias, row_scale=np.array([1.0, 0.5], np.float32),
                                    swiglu=True)
    assert h.shape == (2, 64)
    # row 0: g = (0, 1, -1, 20), u = g + 1; silu(1) = 0.7310585786300049
    np.testing.assert_allclose(h[0, :4], [0.0, 0.7310585786300049 * 2.0, -0.2689414213699951 * 0.0,
                                          20.0 / (1 + math.exp(-20.0)) * 21.0], rtol=1e-12)
    # row 1: g = 2, u = 3, scaled by 0.5; silu(2) = 1.7615941559557649
    np.testing.assert_allclose(h[1, :4], [1.7615941559557649 * 3 * 0.5] * 4, rtol=1e-12)
    assert np.all(h[:, 4:] == 0.0)


# -------------------------------------------------- expert SwiGLU backward --
# h = silu(g) u r: gradients with respect to the gate and up pre-activations and
# the routing weight r, pinned by literal derivative values, by central
# differences of the (separately pinned) forward, and through the whole
# input-gradient composition with one-hot weights.

# silu(g) and silu'(g) = d/dg [g / (1 + exp(-g))] to 17 digits (computed
# symbolically, independent of the oracle's formula).
SILU = {0.0: 0.0, 1.0: 0.73105857863000488, -2.0: -0.23840584404423511, 4.0: 3.9280551601516338,
        0.5: 0.31122966560092728}
DSILU = {0.0: 0.5, 1.0: 0.92767051187148673, -2.0: -0.090784248784895479, 4.0: 1.0526646148910729,
         0.5: 0.73996118730265181}


def test_swiglu_backward_literals():
    gs = [0.0, 1.0, -2.0, 4.0, 0.5]
    a = np.zeros((2, 128))
    a[0, :5] = gs                 # gate columns
    a[0, 64:69] = [3.0, 2.0, -1.0, 0.25, 5.0]   # up columns of the same outputs
    a[1, :5] = gs
    a[1, 64:69] = 1.0
    dh = np.zeros((2, 64))
    dh[0, :5] = [1.0, 1.0, 2.0, -1.0, 0.5]
    dh[1, :5] = 1.0
    r = np.array([0.5, 2.0], np.float32)
    dgu, dr = oracle.swiglu_backward(a, dh, r)
    up0 = [3.0, 2.0, -1.0, 0.25, 5.0]
    for j, g in enumerate(gs):
        assert dgu[0, j] == pytest.approx(0.5 * dh[0, j] * up0[j] * DSILU[g], rel=1e-14, abs=1e-300)
        assert dgu[0, 64 + j] == pytest.approx(0.5 * dh[0, j] * SILU[g], rel=1e-14, abs=1e-300)
        assert dgu[1, j] == pytest.approx(2.0 * DSILU[g], rel=1e-14)
        assert dgu[1, 64 + j] == pytest.approx(2.0 * SILU[g], rel=1e-14, abs=1e-300)
    assert np.all(dgu[:, 5:64] == 0.0) and np.all(dgu[:, 69:] == 0.0)
    assert dr[0] == pytest.approx(sum(SILU[g] * u * d for g, u, d in zip(gs, up0, dh[0, :5])), rel=1e-14)
    assert dr[1] == pytest.approx(sum(SILU[g] for g in gs), rel=1e-14)
    # no routing weight: the same as r = 1, and no routing-weight gradient
    dgu1, dr1 = oracle.swiglu_backward(a, dh)
    assert dr1 is None
    np.testing.assert_array_equal(dgu1, oracle.swiglu_backward(a, dh, np.ones(2, np.float32))[0])


def test_swiglu_backward_matches_central_differences_of_the_forward():
    rng = np.random.default_rng(3)
    T, N = 3, 256
    a = rng.standard_normal((T, N)) * 2.0
    dh = rng.standard_normal((T, N // 2))
    r = rng.random(T).astype(np.float32)
    dgu, dr = oracle.swiglu_backward(a, dh, r)
    loss = lambda aa, rr: float(np.sum(oracle.swiglu_forward(aa, rr) * dh))
    eps = 1e-6
    for t in range(T):
        for c in list(range(0, N, 7)) + [63, 64, 127, 128, 255]:
            ap, am = a.copy(), a.copy()
            ap[t, c] += eps
            am[t, c] -= eps
            num = (loss(ap, r) - loss(am, r)) / (2 * eps)
            assert dgu[t, c] == pytest.approx(num, rel=1e-6, abs=1e-7), (t, c)
    # routing weight: the loss is linear in r (fp32 scales, so perturb in fp64 by hand)
    h1 = oracle.swiglu_forward(a)
    np.testing.assert_allclose(dr, np.sum(h1 * dh, axis=1), rtol=1e-12)


def test_grouped_swiglu_dgrad_one_hot_literals():
    # E = 1, N = 128 (64 gate + 64 up rows), K = 128, W = I: a[t, c] = x[t, c], and
    # grad_x[t, k] = bf16(dgu[t, k]).  Row 0: g = 1, u = 2, dh = 1, r = 0.5, so
    # dg = 0.5 * 2 * silu'(1) = 0.92767... -> bf16 0.92578125 and
    # du = 0.5 * silu(1) = 0.36552... -> bf16 0.365234375.
    N = K = 128
    w = np.eye(N, K, dtype=np.float32)[None]
    wb = _bf16(w)
    x = np.zeros((2, K), np.float32)
    x[0, 0], x[0, 64] = 1.0, 2.0
    x[1, 3], x[1, 67] = -2.0, 4.0
    dh = np.zeros((2, 64), np.float32)
    dh[0, 0] = 1.0
    dh[1, 3] = -0.5
    r = np.array([0.5, 1.0], np.float32)
    gx, dr = oracle.grouped_swiglu_dgrad(_bf16(x), np.array([0, 2]), wb, _bf16(dh), row_scale=r)
    assert gx.shape == (2, K) and dr.shape == (2,)
    assert gx[0, 0] == 0.92578125 and gx[0, 64] == 0.365234375
    # row 1: g = -2, u = 4, dh = -0.5: dg = -0.5 * 4 * silu'(-2) = 0.18156... -> 0.181640625,
    # du = -0.5 * silu(-2) = 0.11920... -> 0.119140625
    assert gx[1, 3] == 0.181640625 and gx[1, 67] == 0.119140625
    others = np.ones_like(gx, bool)
    others[0, [0, 64]] = others[1, [3, 67]] = False
    assert np.all(gx[others] == 0.0)
    assert dr[0] == pytest.approx(SILU[1.0] * 2.0, rel=1e-14)
    assert dr[1] == pytest.approx(SILU[-2.0] * 4.0 * -0.5, rel=1e-14)
    # a bias is added to the pre-activations before the derivative
    bias = np.zeros(N, np.float32)
    bias[0] = 1.0   # g of row 0 becomes 2
    gxb, _ = oracle.grouped_swiglu_dgrad(_bf16(x), np.array([0, 2]), wb, _bf16(dh), bias=bias,
                                         row_scale=r)
    s2 = 1.0 / (1.0 + math.exp(-2.0))
    assert gxb[0, 0] == oracle.bf16_bits_to_f32(oracle.f32_to_bf16_bits(
        np.float32(0.5 * 2.0 * s2 * (1 + 2.0 * (1 - s2)))))


def test_moe_combine_literals():
    """The top-k combine: token 0 takes rows 0 and 2, token 1 row 1 only (route 1
    absent); exact sums of bf16 values; the backward copies each token's gradient
    to its rows and leaves a row no route names at zero."""
    vals = np.array([[1.0, 2.0], [3.0, 4.0], [5.0, -6.5], [7.0, 8.0]], dtype=np.float32)
    rows = (vals.view(np.uint32) >> 16).astype(np.uint16)  # exact in bf16
    tr = np.array([[0, 2], [1, -1]], dtype=np.int32)
    out = oracle.moe_combine(rows, tr)
    np.testing.assert_array_equal(out, np.array([[6.0, -4.5], [3.0, 4.0]]))
    g = (np.array([[0.5, -1.0], [2.0, 0.25]], dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)
    gr = oracle.moe_combine_bwd(g, tr, 4)
    np.testing.assert_array_equal(gr[0], g[0])
    np.testing.assert_array_equal(gr[2], g[0])
    np.testing.assert_array_equal(gr[1], g[1])
    np.testing.assert_array_equal(gr[3], np.zeros(2, dtype=np.uint16))


def test_moe_combine_single_route_is_identity_and_sum_is_linear():
    rng = np.random.default_rng(3)
    R, H = 12, 16
    rows = oracle.f32_to_bf16_bits(rng.standard_normal((R, H)).astype(np.float32))
    perm = rng.permutation(R).astype(np.int32).reshape(R, 1)
    np.testing.assert_array_equal(oracle.moe_combine(rows, perm),
                                  oracle.bf16_bits_to_f32(rows[perm[:, 0]]).astype(np.float64))
    tr = rng.permutation(R).astype(np.int32).reshape(R // 3, 3)
    expect = sum(oracle.bf16_bits_to_f32(rows[tr[:, j]]).astype(np.float64) for j in range(3))
    np.testing.assert_allclose(oracle.moe_combine(rows, tr), expect, rtol=0, atol=1e-12)
