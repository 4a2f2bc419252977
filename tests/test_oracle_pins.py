"""Pins of the CPU oracle against what the mathematics, library routines and hand-worked
special cases fix (no GPU). Each test names the plausible mistake it catches."""
import ctypes
import math

import numpy as np
import pytest
import torch

from oracle import EXACT, PLAIN, lib

L = lib()
U = 2.0 ** -24  # unit roundoff of fp32


def f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def p(a):
    return a.ctypes.data


def dot(w, x, mode, vw=8):
    w, x = f32(w), f32(x)
    return L.orc_dot_exact(p(w), p(x), len(w), vw) if mode == EXACT else L.orc_dot_plain(p(w), p(x), len(w))


# ------------------------------------------------------------------ exp of the contract

def test_exp_c_special_values():
    assert L.orc_exp_c(0.0) == 1.0          # softmax of one element must be exactly 1
    assert L.orc_exp_c(-0.0) == 1.0
    assert L.orc_exp_c(-87.0) == 0.0 and L.orc_exp_c(-1000.0) == 0.0
    assert math.isinf(L.orc_exp_c(88.0)) and math.isinf(L.orc_exp_c(1e30))
    assert math.isnan(L.orc_exp_c(float("nan")))
    assert L.orc_exp_c(-86.9) > 0.0


def test_exp_c_within_two_ulp_of_exp():
    rng = np.random.default_rng(0)
    xs = np.concatenate([np.linspace(-86.9, 87.9, 40001), rng.uniform(-20, 5, 20000),
                         rng.uniform(-1e-3, 1e-3, 2000)]).astype(np.float32)
    worst = 0.0
    for x in xs:
        ref = math.exp(float(x))
        got = L.orc_exp_c(float(x))
        if ref < 2.0 ** -126:
            assert abs(got - ref) <= 2 * 2.0 ** -149
            continue
        ulp = float(np.spacing(np.float32(ref)))
        worst = max(worst, abs(got - ref) / ulp)
    assert worst <= 2.0, worst  # a wrong Taylor coefficient or ln2 split blows far past 2 ulp


# ------------------------------------------------------------------ dot products

@pytest.mark.parametrize("mode", [PLAIN, EXACT])
@pytest.mark.parametrize("K", [8, 16, 256, 688, 2560, 9728])
def test_dot_one_hot_is_exact(mode, K):
    rng = np.random.default_rng(K)
    x = rng.standard_normal(K).astype(np.float32)
    for k in (0, K // 3, K - 1):
        w = np.zeros(K, np.float32)
        w[k] = 1.0
        assert dot(w, x, mode) == x[k]  # a dropped or misplaced element fails here


@pytest.mark.parametrize("mode", [PLAIN, EXACT])
@pytest.mark.parametrize("K,vw", [(8, 8), (256, 8), (688, 8), (2560, 8), (9728, 8), (1408, 16), (2048, 16)])
def test_dot_within_forward_error_bound(mode, K, vw):
    rng = np.random.default_rng(K + vw)
    for _ in range(5):
        w = rng.standard_normal(K).astype(np.float32)
        x = rng.standard_normal(K).astype(np.float32)
        exact = math.fsum(float(a) * float(b) for a, b in zip(w, x))
        got = L.orc_dot_exact(p(w), p(x), K, vw) if mode == EXACT else L.orc_dot_plain(p(w), p(x), K)
        n = K + 5
        gamma = n * U / (1 - n * U)
        assert abs(got - exact) <= gamma * float(np.sum(np.abs(w.astype(np.float64) * x))) + 1e-30


def test_dot_exact_folds_partials_as_a_tree():
    # K = 256, VW = 8: one vector per partial. Partials a0 = 2^24, a8 = 1, a24 = 1, others 0.
    # Folds: (i, i+16) gives a0 = 2^24, a8 = 1 + 1 = 2; (i, i+8) gives a0 = 2^24 + 2 (representable).
    # A sequential sum adds each 1 to 2^24 separately and loses both (ties to even).
    K = 256
    w = np.zeros(K, np.float32)
    x = np.ones(K, np.float32)
    w[8 * 0] = 2.0 ** 24
    w[8 * 8] = 1.0
    w[8 * 24] = 1.0
    assert dot(w, x, EXACT) == 2.0 ** 24 + 2
    assert dot(w, x, PLAIN) == 2.0 ** 24


def test_dot_exact_assigns_vector_v_to_partial_v_mod_32():
    # K = 512, VW = 8: vector v covers elements 8v..8v+7. v0 = 2^24, v1 = 1, v33 = 1.
    # Contract: partial 1 chains v1 then v33 -> 2, which meets 2^24 at the last fold: 2^24 + 2.
    # A blocked assignment (partial l <- vectors 2l, 2l+1) would add v1 into 2^24 first and lose it.
    K = 512
    w = np.zeros(K, np.float32)
    x = np.ones(K, np.float32)
    w[0], w[8 * 1], w[8 * 33] = 2.0 ** 24, 1.0, 1.0
    assert dot(w, x, EXACT) == 2.0 ** 24 + 2


def test_dot_exact_chains_elements_of_a_vector_in_ascending_order():
    # One vector: elements 2^24, 1, 1 fused in ascending order -> each +1 is lost.
    w = np.zeros(8, np.float32)
    w[:3] = [2.0 ** 24, 1.0, 1.0]
    assert dot(w, np.ones(8, np.float32), EXACT) == 2.0 ** 24


def test_dot_exact_e4m3_vector_width_16():
    # Elements 0, 16, 24 hold 2^24, 1, 1 (K = 32).
    # VW = 16: vector 1 = elements 16..31 chains 1 + 1 = 2 in partial 1; final fold 2^24 + 2.
    # VW = 8: elements 16 and 24 start partials 2 and 3; fold (i, i+2) adds 1 to 2^24 (lost),
    #         fold (i, i+1) adds partial 1 (= 1 from partial 3) to 2^24 (lost): 2^24.
    K = 32
    w = np.zeros(K, np.float32)
    w[0], w[16], w[24] = 2.0 ** 24, 1.0, 1.0
    x = np.ones(K, np.float32)
    assert L.orc_dot_exact(p(w), p(x), K, 16) == 2.0 ** 24 + 2
    assert L.orc_dot_exact(p(w), p(x), K, 8) == 2.0 ** 24


# ------------------------------------------------------------------ RMSNorm

@pytest.mark.parametrize("mode", [PLAIN, EXACT])
def test_rmsnorm_matches_float64_definition(mode):
    rng = np.random.default_rng(1)
    d = 2560
    x = f32(rng.standard_normal(d) * 3)
    g = np.full(d, 0x3C00, np.uint16)  # fp16 1.0
    out = np.empty(d, np.float32)
    L.orc_rmsnorm(p(x), p(g), 0, d, 1e-5, mode, p(out))
    ref = x / np.sqrt(np.mean(x.astype(np.float64) ** 2) + 1e-5)
    assert np.max(np.abs(out - ref) / np.abs(ref)) < 4e-6  # a dropped eps or mean->sum fails
    # gain 2.0 (fp16 0x4000) doubles the result exactly
    g2 = np.full(d, 0x4000, np.uint16)
    out2 = np.empty(d, np.float32)
    L.orc_rmsnorm(p(x), p(g2), 0, d, 1e-5, mode, p(out2))
    assert np.array_equal(out2, 2 * out)


def test_rmsnorm_eps_inside_root():
    # x = c everywhere: mean(x^2) = c^2, so xn = c / sqrt(c^2 + eps); eps outside the root would give
    # c / (|c| + eps) and a missing eps would give exactly 1.
    d = 256
    c = np.float32(1e-3)
    x = np.full(d, c, np.float32)
    g = np.full(d, 0x3C00, np.uint16)
    out = np.empty(d, np.float32)
    L.orc_rmsnorm(p(x), p(g), 0, d, 1e-5, EXACT, p(out))
    assert out[0] == pytest.approx(1e-3 / math.sqrt(1e-6 + 1e-5), rel=1e-6)


# ------------------------------------------------------------------ RoPE

def rope(y, pos, theta=10000.0, mode=EXACT):
    y = f32(y).copy()
    L.orc_rope(p(y), len(y), pos, theta, mode)
    return y


@pytest.mark.parametrize("mode", [PLAIN, EXACT])
def test_rope_position_zero_is_identity(mode):
    y = np.random.default_rng(2).standard_normal(128).astype(np.float32)
    assert np.array_equal(rope(y, 0, mode=mode), y)


def test_rope_table_definition():
    cs, sn = np.empty(64, np.float32), np.empty(64, np.float32)
    L.orc_rope_row(10000.0, 128, 7, p(cs), p(sn))
    i = np.arange(64)
    ang = 7 * 10000.0 ** (-(2.0 * i) / 128)
    assert np.array_equal(cs, np.cos(ang).astype(np.float32))
    assert np.array_equal(sn, np.sin(ang).astype(np.float32))
    assert cs[0] == np.float32(math.cos(7.0))  # pair 0 turns by exactly p radians


def test_rope_preserves_pair_norms_and_is_relative():
    rng = np.random.default_rng(3)
    hd = 128
    q = rng.standard_normal(hd).astype(np.float32)
    k = rng.standard_normal(hd).astype(np.float32)
    for pos in (1, 17, 1000, 4095):
        r = rope(q, pos)
        a, b = q[:64].astype(np.float64), q[64:].astype(np.float64)
        ra, rb = r[:64].astype(np.float64), r[64:].astype(np.float64)
        assert np.allclose(ra ** 2 + rb ** 2, a ** 2 + b ** 2, rtol=1e-5)
    # q_m . k_n depends only on m - n (pairs are rotated, not swapped or sign-flipped)
    base = float(np.dot(rope(q, 10).astype(np.float64), rope(k, 3)))
    for t in (5, 100, 2000):
        assert float(np.dot(rope(q, 10 + t).astype(np.float64), rope(k, 3 + t))) == pytest.approx(base, rel=2e-4,
                                                                                                     abs=2e-4)


# ------------------------------------------------------------------ attention

def attend(q, K, V, n, mode, kvdt=0, hd=None):
    hd = hd or len(q)
    out = np.empty(hd, np.float32)
    L.orc_attention_head(p(f32(q)), p(K), p(V), kvdt, n, hd, float(np.float32(1 / math.sqrt(hd))), mode, p(out))
    return out


def to16(x, kvdt):
    x = f32(x)
    if kvdt == 0:
        return x.astype(np.float16).view(np.uint16)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def from16(b, kvdt):
    if kvdt == 0:
        return b.view(np.float16).astype(np.float64)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("mode", [PLAIN, EXACT])
@pytest.mark.parametrize("kvdt", [0, 1])
def test_attention_one_position_returns_v_exactly(mode, kvdt):
    rng = np.random.default_rng(4)
    hd = 128
    q = rng.standard_normal(hd)
    K = to16(rng.standard_normal((1, hd)), kvdt)
    V = to16(rng.standard_normal((1, hd)), kvdt)
    out = attend(q, K, V, 1, mode, kvdt)
    assert np.array_equal(out.astype(np.float64), from16(V[0], kvdt))


@pytest.mark.parametrize("mode", [PLAIN, EXACT])
@pytest.mark.parametrize("n", [2, 31, 32, 33, 64, 65, 300, 4096])
def test_attention_weights_sum_to_one(mode, n):
    rng = np.random.default_rng(n)
    hd = 128
    q = rng.standard_normal(hd) * 2
    K = to16(rng.standard_normal((n, hd)), 0)
    V = to16(np.ones((n, hd)), 0)
    out = attend(q, K, V, n, mode)
    assert np.max(np.abs(out - 1.0)) <= (n + 64) * U * 2  # softmax rows sum to 1 within rounding


@pytest.mark.parametrize("mode", [PLAIN, EXACT])
@pytest.mark.parametrize("n", [1, 5, 32, 33, 97, 513, 1024])
def test_attention_matches_float64_softmax(mode, n):
    rng = np.random.default_rng(100 + n)
    hd = 64
    q = rng.standard_normal(hd).astype(np.float32)
    K = to16(rng.standard_normal((n, hd)), 0)
    V = to16(rng.standard_normal((n, hd)), 0)
    out = attend(q, K, V, n, mode)
    s = from16(K, 0) @ q.astype(np.float64) * (1 / math.sqrt(hd))
    a = np.exp(s - s.max())
    a /= a.sum()
    ref = a @ from16(V, 0)
    assert np.max(np.abs(out - ref)) < 2e-6  # a wrong scale, mask or merge weight fails


def test_attention_masks_positions_beyond_n():
    # Rows past n hold NaN; reading them would poison the result.
    rng = np.random.default_rng(5)
    hd, n = 64, 40
    q = rng.standard_normal(hd)
    K = to16(np.concatenate([rng.standard_normal((n, hd)), np.full((24, hd), np.nan)]), 0)
    V = to16(np.concatenate([rng.standard_normal((n, hd)), np.full((24, hd), np.nan)]), 0)
    for mode in (PLAIN, EXACT):
        assert np.all(np.isfinite(attend(q, K, V, n, mode)))


# ------------------------------------------------------------------ storage types

def test_e4m3_table_matches_library_and_spec():
    tab = np.ctypeslib.as_array(L.orc_e4m3_table(), shape=(256,)).copy()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    both_nan = np.isnan(tab) & np.isnan(ref)
    assert np.array_equal(tab[~both_nan], ref[~both_nan])
    assert np.array_equal(np.isnan(tab), np.isnan(ref))
    # values written in the OCP FP8 specification
    assert tab[0x00] == 0.0 and tab[0x01] == 2.0 ** -9 and tab[0x07] == 7 * 2.0 ** -9
    assert tab[0x08] == 2.0 ** -6 and tab[0x38] == 1.0 and tab[0x7E] == 448.0 and tab[0xFE] == -448.0
    assert np.isnan(tab[0x7F]) and np.isnan(tab[0xFF])


def _edge_floats():
    rng = np.random.default_rng(6)
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e10, 6.1035156e-05, 5.96e-08, 2.98e-08,
            2.9802322e-08, 1e-9, 3.0517578e-05 + 1e-12, 1.0009765625, 1.00048828125, 1.000732421875,
            3.4e38, 1.1754944e-38, 1e-40, float("inf"), -float("inf")]
    vals += list(rng.standard_normal(20000) * 10 ** rng.uniform(-9, 5, 20000))
    return np.array(vals, dtype=np.float32)


def test_round_f16_is_ieee_round_to_nearest_even():
    x = _edge_floats()
    got = np.array([L.orc_round_f16(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, x.astype(np.float16).view(np.uint16))


def test_round_bf16_is_round_to_nearest_even():
    x = _edge_floats()
    got = np.array([L.orc_round_bf16(float(v)) for v in x], dtype=np.uint16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ routing

def route(r, k, mode=EXACT):
    r = f32(r)
    sel = np.zeros(k, np.int32)
    gate = np.zeros(k, np.float32)
    P = np.zeros(len(r), np.float32)
    L.orc_route(p(r), len(r), k, mode, p(sel), p(gate), p(P))
    return sel, gate, P


def test_route_ties_go_to_the_lower_index():
    sel, gate, _ = route([0.0, 1.0, 1.0, 0.5], 2)
    assert list(sel) == [1, 2]
    assert gate[0] == gate[1] == 0.5


@pytest.mark.parametrize("mode", [PLAIN, EXACT])
def test_route_top1_gate_is_one_and_gates_sum_to_one(mode):
    rng = np.random.default_rng(7)
    for _ in range(50):
        r = rng.standard_normal(32)
        sel, gate, P = route(r, 1, mode)
        assert gate[0] == 1.0 and sel[0] == int(np.argmax(r))
        sel, gate, P = route(r, 4, mode)
        assert abs(float(np.sum(gate, dtype=np.float64)) - 1.0) < 4 * U
        assert set(sel) == set(np.argsort(-r, kind="stable")[:4])
        ref = np.exp(r - r.max())
        assert np.allclose(P, ref / ref.sum(), rtol=1e-6, atol=1e-9)


# ------------------------------------------------------------------ sampling

@pytest.mark.parametrize("mode", [PLAIN, EXACT])
def test_sample_cold_temperature_is_argmax(mode):
    rng = np.random.default_rng(8)
    for V in (5, 300, 4096):
        l = f32(rng.standard_normal(V))
        for u in (0.0, 0.5, 0.999):
            assert L.orc_sample(p(l), V, 1e-3, u, mode) == L.orc_argmax(p(l), V) == int(np.argmax(l))


@pytest.mark.parametrize("mode", [PLAIN, EXACT])
def test_sample_matches_softmax_distribution(mode):
    # chi-square of 20000 inverse-CDF draws on a 16-token vocabulary against exp(l/T)/Z
    import synth
    from scipy.stats import chi2
    rng = np.random.default_rng(9)
    V, T = 16, 0.7
    l = f32(rng.standard_normal(V))
    us = synth.uniforms(12345, 0, 20000)
    counts = np.zeros(V)
    for u in us:
        counts[L.orc_sample(p(l), V, T, float(u), mode)] += 1
    pr = np.exp((l - l.max()) / T)
    pr /= pr.sum()
    stat = float(np.sum((counts - 20000 * pr) ** 2 / (20000 * pr)))
    assert chi2.sf(stat, V - 1) > 1e-4


def test_sample_inverse_cdf_matches_float64_away_from_boundaries():
    rng = np.random.default_rng(10)
    V, T = 32000, 0.7
    l = f32(rng.standard_normal(V))
    e = np.exp((l.astype(np.float64) - l.max()) / T)
    cdf = np.cumsum(e) / e.sum()
    for u in np.linspace(0.001, 0.999, 200):
        ref = int(np.searchsorted(cdf, u, side="right"))
        if min(abs(cdf[max(ref - 1, 0)] - u), abs(cdf[ref] - u)) < 1e-5:
            continue
        for mode in (PLAIN, EXACT):
            assert L.orc_sample(p(l), V, T, float(u), mode) == ref
