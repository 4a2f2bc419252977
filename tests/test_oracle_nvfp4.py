"""Pins of the oracle's NVFP4 layer matrices (e2m1 elements, an e4m3 scale per 16 elements of a
row, an fp32 scale per row) and of the seeded quantiser that produces them.

The element values are the format's definition written out (4-bit floating point E2M1: one sign
bit, two exponent bits with bias 1, one fraction bit, a subnormal for exponent 0); the whole
model is pinned by the float64 brute force in test_oracle_model.py, which dequantises the stored
bytes with its own code."""
import numpy as np
import pytest

import synth
from oracle import EXACT, PLAIN, OracleModel, brute
from oracle.oracle import lib

# every E2M1 code 0..15: +0, 0.5, 1, 1.5, 2, 3, 4, 6, then the same negated
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def test_e2m1_codes_decode_to_the_format_values():
    t = lib().orc_e2m1_table()
    got = [t[i] for i in range(16)]
    assert got == E2M1_VALUES
    assert [float(x) for x in brute.e2m1_decode(np.arange(16))] == E2M1_VALUES
    assert np.signbit(got[8])  # code 8 is negative zero


# e4m3 codes of the block scales used below (sign 0, exponent bias 7, three fraction bits)
E4M3_ONE, E4M3_ONE_AND_HALF = 0x38, 0x3C


def _pack(codes):
    """Element 2i in the low nibble of byte i."""
    c = np.asarray(codes, dtype=np.uint8)
    return np.ascontiguousarray(c[0::2] | (c[1::2] << 4))


def dot4(codes, bscale, x, mode):
    q = _pack(codes)
    b = np.ascontiguousarray(bscale, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    return lib().orc_dot_nvfp4(q.ctypes.data, b.ctypes.data, x.ctypes.data, len(x), mode)


@pytest.mark.parametrize("mode", [EXACT, PLAIN])
def test_nvfp4_dot_is_exact_when_every_partial_is_representable(mode):
    """Block scales that are powers of two and inputs that are small multiples of 1/4: every
    product and partial sum is exact in fp32, so both modes must return the rational dot of the
    format's values (a swapped nibble, a misplaced block, a mis-decoded scale or a dropped sign
    fails here)."""
    from fractions import Fraction
    rng = np.random.default_rng(77)
    K = 512
    codes = rng.integers(0, 16, K)
    k = rng.integers(-3, 4, K // 16)
    bscale = ((k + 7) << 3).astype(np.uint8)  # e4m3 code of 2^k
    x = (rng.integers(-3, 4, K) / 4.0).astype(np.float32)
    want = sum(Fraction(E2M1_VALUES[codes[j]]) * Fraction(2) ** int(k[j // 16]) * Fraction(float(x[j]))
               for j in range(K))
    assert Fraction(float(dot4(codes, bscale, x, mode))) == want


def test_nvfp4_dot_exact_assigns_vectors_to_lanes_and_folds_as_a_tree():
    """K = 512, all scales 1: vector 0 sums to 2^24 (code 4 times 2^22), vectors 1 and 33 to 1
    each. The contract puts vectors 1 and 33 in lane 1 (2, exact) and folds it into lane 0 last:
    2^24 + 2. The plain order adds each 1 to 2^24 and loses both (ties to even)."""
    K = 512
    codes = np.zeros(K, np.int64)
    x = np.zeros(K, np.float32)
    codes[0], x[0] = 6, 2.0 ** 22  # E2M1 code 6 is 4
    codes[8], x[8] = 2, 1.0        # code 2 is 1
    codes[264], x[264] = 2, 1.0
    bscale = np.full(K // 16, E4M3_ONE, np.uint8)
    assert dot4(codes, bscale, x, EXACT) == 2.0 ** 24 + 2
    assert dot4(codes, bscale, x, PLAIN) == 2.0 ** 24


def test_nvfp4_dot_exact_applies_the_block_scale_with_one_rounding():
    """Lane 0 holds a = 1 - 2^-24 from vector 0 (scale 1); vector 32 has t = 1 + 2^-23 and block
    scale 1.5. One fused step gives RN(1.5 t + a) = RN(2.5 + 2^-23): the midpoint between 2.5 and
    2.5 + 2^-22, so 2.5 (even). Rounding 1.5 t first (1.5 + 3 2^-24, a midpoint, rounds to
    1.5 + 2^-22) and then adding a gives 2.5 + 3 2^-24, which rounds to 2.5 + 2^-22; so does the
    plain order."""
    K = 512
    codes = np.zeros(K, np.int64)
    x = np.zeros(K, np.float32)
    a = np.float32(1.0) - np.float32(2.0 ** -24)
    t = np.float32(1.0) + np.float32(2.0 ** -23)
    codes[0], x[0] = 2, a
    codes[256], x[256] = 2, t
    bscale = np.full(K // 16, E4M3_ONE, np.uint8)
    bscale[16] = E4M3_ONE_AND_HALF
    assert dot4(codes, bscale, x, EXACT) == 2.5
    assert dot4(codes, bscale, x, PLAIN) == np.float32(2.5) + np.float32(2.0 ** -22)


@pytest.fixture(scope="module")
def quantised():
    return synth.normal_nvfp4_rows(1234, 5, 48, 320)


def test_quantiser_layout_and_ranges(quantised):
    codes, bscale, rscale = quantised
    assert codes.shape == (48, 160) and bscale.shape == (48, 20) and rscale.shape == (48,)
    assert codes.dtype == np.uint8 and bscale.dtype == np.uint8 and rscale.dtype == np.float32
    b = brute.e4m3_decode(bscale)
    assert np.all(np.isfinite(b)) and np.all(b >= 0) and np.all(b <= 448)
    w = synth.normal_f32(1234, 5, (48, 320), synth.WEIGHT_STD)
    # row scale: max |w| of the row over 6 * 448
    assert np.allclose(rscale.astype(np.float64) * 6 * 448, np.abs(w).max(axis=1), rtol=1e-6)


def test_quantiser_picks_a_nearest_code(quantised):
    """Each dequantised element is (row scale x block scale) times an E2M1 magnitude nearest to
    the draw's (saturating at 6), with the draw's sign."""
    codes, bscale, rscale = quantised
    w = synth.normal_f32(1234, 5, (48, 320), synth.WEIGHT_STD).astype(np.float64)
    deq = brute.nvfp4_dequant(codes, bscale, rscale)
    unit = rscale.astype(np.float64)[:, None] * np.repeat(brute.e4m3_decode(bscale), 16, axis=1)
    a = np.abs(w) / unit
    q = np.abs(deq) / unit
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    assert np.all(np.min(np.abs(q[..., None] - mags), axis=-1) <= 1e-9)  # q is an E2M1 magnitude
    nearest_err = np.min(np.abs(a[..., None] - mags), axis=-1)
    assert np.all(np.abs(a - q) <= nearest_err + 1e-6)
    assert np.all(np.sign(deq) * np.sign(w) >= 0)
    # every block's largest element lands at the top of the range (block scale = its max / 6)
    top = q.reshape(48, 20, 16).max(axis=2)
    assert np.all((top >= 4) & (top <= 6))


def test_ties_go_to_the_even_code():
    """Midpoints between E2M1 magnitudes round to the code with an even fraction bit."""
    mid = synth._E2M1_MID
    k = np.searchsorted(mid, mid, side="left")
    k = np.where(k % 2 == 1, k + 1, k)
    assert list(k) == [0, 2, 2, 4, 4, 6, 6]  # 0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4


def test_exact_and_plain_modes_agree_within_the_logit_tolerances():
    cfg = synth.shrink(synth.get_config("dense-2.3b-nvfp4"))
    W = synth.model_weights(cfg)
    a, b = OracleModel(cfg, W), OracleModel(cfg, W)
    for t in synth.prompt(cfg, 6):
        x = a.step(int(t), EXACT)["logits"].astype(np.float64)
        y = b.step(int(t), PLAIN)["logits"].astype(np.float64)
        assert np.max(np.abs(x - y)) <= 2e-2
        assert np.linalg.norm(x - y) / np.linalg.norm(y) <= 5e-3


def test_nvfp4_model_differs_from_its_fp16_source():
    """The quantisation is real: the nvfp4 model's logits are close to, but not equal to, those of
    the same seeded model kept in fp16 (a dropped scale or nibble swap would not be close)."""
    c4 = synth.shrink(synth.get_config("dense-2.3b-nvfp4"))
    c16 = dict(c4, weight_dtype="f16", embed_dtype=None, index=c4["index"])
    t = synth.prompt(c4, 4)
    l4 = brute.forward(c4, synth.model_weights(c4), t)[0]
    l16 = brute.forward(c16, synth.model_weights(c16), t)[0]
    d = np.abs(l4 - l16)
    assert d.max() > 1e-3  # not the same weights
    assert np.linalg.norm(l4 - l16) / np.linalg.norm(l16) < 0.3  # but the same model, quantised


def gemv(W, dt, rows, K, x, scale, bscale, mode):
    """The oracle's matrix-vector product (dt: 2 e4m3, 4 NVFP4), one output per row."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.ascontiguousarray(scale, dtype=np.float32)
    b = None if bscale is None else np.ascontiguousarray(bscale, dtype=np.uint8)
    y = np.zeros(rows, np.float32)
    rc = lib().orc_gemv(W.ctypes.data, dt, rows, K, x.ctypes.data, s.ctypes.data,
                        None if b is None else b.ctypes.data, y.ctypes.data, mode)
    assert rc == 0
    return y


@pytest.mark.parametrize("mode", [EXACT, PLAIN])
@pytest.mark.parametrize("fmt", ["e4m3", "nvfp4"])
def test_row_scale_multiplies_the_finished_dot(mode, fmt):
    """Row (+1, -1, 0, ...) against x = (1 + 2^-23, 1, 0, ...) with row scale s = 1 + 2^-23: the
    dot is 2^-23 exactly, and s times it, 2^-23 + 2^-46, is exact too. Scaling the elements first
    would round s (1 + 2^-23) to 1 + 2^-22 and return 2^-23."""
    K = 16
    x = np.zeros(K, np.float32)
    x[0], x[1] = np.float32(1.0) + np.float32(2.0 ** -23), 1.0
    s = np.array([np.float32(1.0) + np.float32(2.0 ** -23)], np.float32)
    if fmt == "e4m3":
        W = np.zeros(K, np.uint8)
        W[0], W[1] = 0x38, 0xB8  # e4m3 +1, -1
        y = gemv(W, 2, 1, K, x, s, None, mode)
    else:
        codes = np.zeros(K, np.int64)
        codes[0], codes[1] = 2, 10  # E2M1 +1, -1
        y = gemv(_pack(codes), 4, 1, K, x, s, np.array([E4M3_ONE], np.uint8), mode)
    assert float(y[0]) == 2.0 ** -23 + 2.0 ** -46


@pytest.mark.parametrize("mode", [EXACT, PLAIN])
def test_nvfp4_rows_are_exact_with_representable_operands(mode):
    """Several rows, power-of-two row and block scales, inputs in multiples of 1/4: each output is
    the exact rational row dot times its row scale (a row or block misplaced between rows fails)."""
    from fractions import Fraction
    rng = np.random.default_rng(5)
    rows, K = 6, 256
    codes = rng.integers(0, 16, (rows, K))
    kb = rng.integers(-2, 3, (rows, K // 16))
    kr = rng.integers(-4, 5, rows)
    x = (rng.integers(-3, 4, K) / 4.0).astype(np.float32)
    packed = np.stack([_pack(c) for c in codes])
    bscale = ((kb + 7) << 3).astype(np.uint8)
    scale = (2.0 ** kr).astype(np.float32)
    y = gemv(packed, 4, rows, K, x, scale, bscale, mode)
    for r in range(rows):
        want = sum(Fraction(E2M1_VALUES[codes[r, j]]) * Fraction(2) ** int(kb[r, j // 16]) * Fraction(float(x[j]))
                   for j in range(K)) * Fraction(2) ** int(kr[r])
        assert Fraction(float(y[r])) == want, r
