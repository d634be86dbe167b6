"""Pins of the fp64 oracle against facts that do not come from the oracle itself:
closed forms, invariants, brute force on tiny inputs and library routines.
Each test names the plausible mistake it would catch."""
import math

import numpy as np
import pytest

import oracle as O
import synth


# ---------------------------------------------------------------- storage dtypes
def test_upcast_known_bits():
    f16 = np.array([0x3C00, 0xC000, 0x0001, 0x7BFF, 0x3555], dtype=np.uint16)
    want = [1.0, -2.0, 2.0 ** -24, 65504.0, 0.333251953125]
    assert list(O.upcast(f16, "f16")) == want
    bf = np.array([0x3F80, 0x4049, 0xBF00, 0x0001], dtype=np.uint16)
    want = [1.0, 3.140625, -0.5, 2.0 ** -133]
    assert list(O.upcast(bf, "bf16")) == want


def test_round_ties_to_even():
    # fp16 spacing at 1 is 2^-10; bf16 spacing at 1 is 2^-7 (a wrong mantissa width fails)
    assert O.round_to_storage(np.array([1 + 2 ** -11]), "f16")[0] == 1.0
    assert O.round_to_storage(np.array([1 + 3 * 2 ** -11]), "f16")[0] == 1 + 2 ** -9
    assert O.round_to_storage(np.array([1 + 2 ** -8]), "bf16")[0] == 1.0
    assert O.round_to_storage(np.array([1 + 3 * 2 ** -8]), "bf16")[0] == 1 + 2 ** -6
    assert O.round_to_storage(np.array([-(1 + 3 * 2 ** -8)]), "bf16")[0] == -(1 + 2 ** -6)
    # not a truncation: just above the tie rounds up
    assert O.round_to_storage(np.array([1 + 2 ** -8 + 2 ** -20]), "bf16")[0] == 1 + 2 ** -7


def test_round_matches_library_conversions():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(20000) * rng.choice([1e-3, 1.0, 300.0], 20000)).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_storage(x.astype(np.float64), "bf16"), xb)
    xh = torch.from_numpy(x).to(torch.float16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_storage(x.astype(np.float64), "f16"), xh)


def test_synth_bits_roundtrip_through_oracle():
    # the generator's rounding and the oracle's upcast agree on the same bytes
    cfg = synth.CONFIGS["tiny"]
    w = synth.gen_tensor(cfg, "wq", 0)
    v = O.upcast(w, cfg.dtype)
    np.testing.assert_array_equal(O.round_to_storage(v, cfg.dtype), v)
    assert abs(v.std() - 0.02) < 0.002
    g = O.upcast(synth.gen_tensor(cfg, "attn_norm", 1), cfg.dtype)
    assert abs(g.mean() - 1.0) < 0.03 and abs(g.std() - 0.1) < 0.03


# ---------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_form_constant_vector():
    # h = c * 1 -> g * c / sqrt(c^2 + eps): catches sum-instead-of-mean and a missing sqrt
    c, eps = 0.37, 1e-5
    h = np.full((1, 64), c)
    g = np.linspace(0.5, 1.5, 64)
    np.testing.assert_allclose(O.rms_norm(h, g, eps)[0], g * c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(0)
    h = rng.standard_normal((3, 200))
    y = O.rms_norm(h, np.ones(200), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.rms_norm(7.5 * h, np.ones(200), 0.0), y, rtol=1e-13)


# ---------------------------------------------------------------- RoPE
def test_rope_two_dims_is_rotation_by_pos():
    # hd = 2: frequency theta^0 = 1, so the pair (x0, x1) turns by angle pos
    for pos in (0, 1, 5, 1000):
        a = O.apply_rope(np.array([1.0, 0.0]), pos, 10000.0)
        b = O.apply_rope(np.array([0.0, 1.0]), pos, 10000.0)
        np.testing.assert_allclose(a, [math.cos(pos), math.sin(pos)], atol=1e-15)
        np.testing.assert_allclose(b, [-math.sin(pos), math.cos(pos)], atol=1e-15)


def test_rope_pairing_and_frequencies():
    # hd = 4: dims (0, 2) turn at rate 1, dims (1, 3) at theta^(-1/2) -- catches an
    # interleaved (2i, 2i+1) pairing and a wrong exponent
    theta, pos = 10000.0, 7
    e1 = np.array([0.0, 1.0, 0.0, 0.0])
    r = O.apply_rope(e1, pos, theta)
    w = pos * theta ** -0.5
    np.testing.assert_allclose(r, [0.0, math.cos(w), 0.0, math.sin(w)], atol=1e-15)
    e0 = np.array([1.0, 0.0, 0.0, 0.0])
    np.testing.assert_allclose(O.apply_rope(e0, pos, theta), [math.cos(pos), 0, math.sin(pos), 0], atol=1e-15)


def test_rope_invariants():
    rng = np.random.default_rng(1)
    hd = 128
    q, k = rng.standard_normal(hd), rng.standard_normal(hd)
    np.testing.assert_array_equal(O.apply_rope(q, 0, 1e4), q)
    rq = O.apply_rope(q, 913, 1e4)
    for i in range(hd // 2):           # each pair keeps its norm
        assert math.isclose(rq[i] ** 2 + rq[i + 64] ** 2, q[i] ** 2 + q[i + 64] ** 2, rel_tol=1e-12)
    # <R_m q, R_n k> depends only on m - n
    a = O.apply_rope(q, 300, 1e4) @ O.apply_rope(k, 100, 1e4)
    b = O.apply_rope(q, 1200, 1e4) @ O.apply_rope(k, 1000, 1e4)
    c = O.apply_rope(q, 200, 1e4) @ k
    assert math.isclose(a, b, rel_tol=1e-10) and math.isclose(a, c, rel_tol=1e-10)


def test_rope_matches_complex_rotation():
    # independent formulation: z_i = x_i + 1j x_{i+hd/2} times exp(1j pos f_i)
    rng = np.random.default_rng(2)
    hd, pos, theta = 64, 4097, 10000.0
    x = rng.standard_normal(hd)
    f = theta ** (-np.arange(hd // 2) * 2.0 / hd)
    z = (x[: hd // 2] + 1j * x[hd // 2:]) * np.exp(1j * pos * f)
    np.testing.assert_allclose(O.apply_rope(x, pos, theta), np.concatenate([z.real, z.imag]), atol=1e-12)


# ---------------------------------------------------------------- softmax / attention
def test_softmax_rows_sum_to_one_and_library():
    scipy = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(3)
    s = rng.standard_normal((5, 37)) * 20
    p = O.softmax(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-12)
    np.testing.assert_allclose(p, scipy.softmax(s, axis=-1), rtol=1e-13)


def _attention_brute(q, k, v):
    Hq, hd = q.shape
    Hkv, T, _ = k.shape
    G = Hq // Hkv
    out = [[0.0] * hd for _ in range(Hq)]
    for i in range(Hq):
        j = i // G
        s = [sum(q[i][d] * k[j][t][d] for d in range(hd)) / math.sqrt(hd) for t in range(T)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = math.fsum(e)
        for d in range(hd):
            out[i][d] = math.fsum(e[t] * v[j][t][d] for t in range(T)) / z
    return np.array(out)


@pytest.mark.parametrize("Hq,Hkv,hd,T", [(4, 2, 8, 1), (4, 2, 8, 16), (6, 3, 4, 9), (4, 4, 8, 5), (8, 2, 8, 11)])
def test_attention_brute_force(Hq, Hkv, hd, T):
    rng = np.random.default_rng(Hq * 100 + T)
    q = rng.standard_normal((Hq, hd))
    k = rng.standard_normal((Hkv, T, hd))
    v = rng.standard_normal((Hkv, T, hd))
    np.testing.assert_allclose(O.attention(q, k, v), _attention_brute(q, k, v), rtol=1e-12, atol=1e-13)


def test_attention_single_position_is_v():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((4, 8))
    k = rng.standard_normal((2, 1, 8))
    v = rng.standard_normal((2, 1, 8))
    o = O.attention(q, k, v)
    np.testing.assert_array_equal(o, np.repeat(v[:, 0], 2, axis=0))


def test_gqa_grouping_is_contiguous():
    # kv head j carries a constant value vector j; query head i must read floor(i / G)
    Hq, Hkv, hd, T = 8, 2, 4, 6
    rng = np.random.default_rng(6)
    q = rng.standard_normal((Hq, hd))
    k = rng.standard_normal((Hkv, T, hd))
    v = np.zeros((Hkv, T, hd))
    v[1] += 1.0
    o = O.attention(q, k, v)
    np.testing.assert_allclose(o[:, 0], [0, 0, 0, 0, 1, 1, 1, 1], atol=1e-15)


@pytest.mark.parametrize("splits", [[0, 5, 9, 17], [0, 0, 3, 3, 17], [0, 17], [0, 1, 2, 16, 17, 17]])
def test_split_kv_merge_equals_unsplit(splits):
    rng = np.random.default_rng(7)
    hd, T = 16, 17
    q = rng.standard_normal(hd)
    k = rng.standard_normal((T, hd)) * 3
    v = rng.standard_normal((T, hd))
    bounds = list(zip(splits[:-1], splits[1:]))
    got = O.merge_partials(O.split_partials(q, k, v, bounds))
    want = O.attention(q[None], k[None], v[None])[0]
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- SwiGLU / GEMV / argmax
def test_silu_closed_forms():
    assert O.silu(np.array(0.0)) == 0.0
    assert math.isclose(O.silu(np.array(1.0)), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    x = np.linspace(-6, 6, 101)
    np.testing.assert_allclose(O.silu(x) - O.silu(-x), x, atol=1e-14)   # silu(x)-silu(-x)=x


def test_gemv_against_fsum():
    cfg = synth.CONFIGS["tiny"]
    W = O.upcast(synth.gen_tensor(cfg, "w_down", 0), cfg.dtype)
    x = np.random.default_rng(8).standard_normal(W.shape[1])
    y = W @ x
    for r in (0, 17, 255):
        assert math.isclose(y[r], math.fsum(W[r] * x), rel_tol=1e-12, abs_tol=1e-15)


def test_argmax_ties_lowest_index():
    z = np.array([[0.5, 2.0, -1.0, 2.0, 2.0], [3.0, 3.0, 3.0, 3.0, 3.0]])
    assert list(O.argmax_lowest(z)) == [1, 0]


def test_top2_margin():
    assert O.top2_margin(np.array([1.0, 4.0, 2.5, 4.0])) == 0.0
    assert O.top2_margin(np.array([1.0, 4.0, 2.5])) == 1.5
