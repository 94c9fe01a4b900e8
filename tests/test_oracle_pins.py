"""Pins of the scalar oracle against facts that do not come from the oracle:
closed forms, exact integer results, IEEE binary16 as numpy implements it,
values printed by the pages (tests/golden), invariants and brute force on
tiny shapes.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

import synth

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_fixtures.json")))


def np_dequant(w: np.ndarray, p: int, n: int) -> np.ndarray:
    """Independent numpy dequantisation for brute-force comparisons."""
    bpr = n // 32
    blk = w.reshape(p, bpr, 34)
    sc = blk[:, :, 0:2].copy().view("<f2").astype(np.float64).reshape(p, bpr, 1)
    q = blk[:, :, 2:].view(np.int8).astype(np.float64)
    return (sc * q).reshape(p, n)


# --------------------------------------------------------------------------- f16
def test_f16_widening_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([orc.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_widening_pages_scale(orc):
    g = GOLDEN["q8_test_scale"]
    bits = g["bytes"][0] | (g["bytes"][1] << 8)
    assert bits == g["bits"]
    assert orc.f16_to_f32(bits) == g["value"]
    # hand-decoded patterns
    assert orc.f16_to_f32(0x3C00) == 1.0
    assert orc.f16_to_f32(0x0001) == 2.0 ** -24
    assert orc.f16_to_f32(0x03FF) == 1023 * 2.0 ** -24
    assert orc.f16_to_f32(0x7BFF) == 65504.0
    assert math.copysign(1.0, orc.f16_to_f32(0x8000)) == -1.0
    assert orc.f16_to_f32(0xFC00) == -math.inf


def test_f16_rounding_representable_and_midpoints(orc):
    # every finite half value rounds to itself
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16)
    fin = np.isfinite(vals)
    f32 = vals[fin].astype(np.float32)
    got = orc.f32_to_f16_array(f32)
    assert np.array_equal(got, bits[fin])
    # midpoints between neighbouring positive halves tie to the even pattern
    pos = np.arange(0x0000, 0x7BFF, dtype=np.uint16)
    lo = pos.view(np.float16).astype(np.float64)
    hi = (pos + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    exact = mid.astype(np.float64) == (lo + hi) / 2   # midpoint representable in f32
    got = orc.f32_to_f16_array(mid[exact])
    even = np.where(pos[exact] % 2 == 0, pos[exact], pos[exact] + 1)
    assert np.array_equal(got, even.astype(np.uint16))


def test_f16_rounding_matches_numpy_random_and_extremes(orc):
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-5).astype(np.float32),      # subnormal halves
        (rng.standard_normal(5000) * 3e4).astype(np.float32),       # near overflow
        np.array([65504.0, 65519.99, 65520.0, 1e9, -65520.0, 2.0 ** -25, 2.0 ** -26,
                  3 * 2.0 ** -26, 0.0, -0.0], dtype=np.float32),
    ])
    got = orc.f32_to_f16_array(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
    assert orc.f32_to_f16(65520.0) == 0x7C00           # rounds up to infinity
    assert orc.f32_to_f16(65519.99) == 0x7BFF
    assert np.isnan(np.uint16(orc.f32_to_f16(float("nan"))).view(np.float16))


# --------------------------------------------------------------------------- matvec
def test_matvec_sum_of_x(orc):
    """All quants 1 and scale 1: out[r] = sum(x)."""
    n, p = 1024, 7
    w = synth.q8_const_matrix(p, n, 0x3C00, 1)
    x = synth.normal_f32(0, "x", n)
    out, ab = orc.q8_matvec(w, x, n, p)
    ref = math.fsum(float(v) for v in x)
    assert np.all(np.abs(out.astype(np.float64) - ref) <= 1e-7 * np.abs(x).sum())
    assert np.allclose(ab, np.abs(x.astype(np.float64)).sum(), rtol=1e-12)


@pytest.mark.parametrize("n,p", [(32, 1), (96, 5), (18944, 3)])
def test_matvec_exact_integer_sums(orc, n, p):
    """x = 1 and scale 1: out[r] = sum of the row's quants, an exact integer."""
    w = synth.q8_from_parts(3, "w", p, n, 0x3C00)
    q = w.reshape(p, n // 32, 34)[:, :, 2:].view(np.int8).astype(np.int64).reshape(p, n)
    out, _ = orc.q8_matvec(w, np.ones(n, np.float32), n, p)
    assert np.array_equal(out.astype(np.int64), q.sum(axis=1))


def test_matvec_minus_128_quant(orc):
    n, p = 64, 2
    w = synth.q8_const_matrix(p, n, 0x3C00, -128)
    out, _ = orc.q8_matvec(w, np.ones(n, np.float32), n, p)
    assert np.array_equal(out, np.full(p, -128.0 * n, np.float32))


def test_matvec_one_hot_every_column(orc):
    """x = e_j: out[r] = scale[r, j // 32] * q[r, j] for every (r, j)."""
    n, p = 64, 3
    w = synth.q8_matrix(11, "w", p, n)
    blk = w.reshape(p, n // 32, 34)
    sc = blk[:, :, 0:2].copy().view("<f2").astype(np.float64).reshape(p, n // 32)
    q = blk[:, :, 2:].view(np.int8).astype(np.float64).reshape(p, n)
    for j in range(n):
        x = np.zeros(n, np.float32)
        x[j] = 1.0
        out, _ = orc.q8_matvec(w, x, n, p)
        assert np.array_equal(out, (sc[:, j // 32] * q[:, j]).astype(np.float32)), j


@pytest.mark.parametrize("n,p", [(32, 1), (64, 3), (96, 50), (896, 33), (1024, 17)])
def test_matvec_brute_force(orc, n, p):
    w = synth.q8_matrix(1, f"w{n}", p, n)
    x = synth.normal_f32(1, f"x{n}", n)
    W = np_dequant(w, p, n)
    ref = W @ x.astype(np.float64)
    out, ab = orc.q8_matvec(w, x, n, p)
    assert np.allclose(ab, np.abs(W * x.astype(np.float64)).sum(axis=1), rtol=1e-12)
    assert np.all(np.abs(out.astype(np.float64) - ref) <= 1e-7 * ab + 1e-30)


def test_matvec_rows_matches_full(orc):
    n, p = 256, 40
    w = synth.q8_matrix(2, "w", p, n)
    x = synth.normal_f32(2, "x", n)
    full, ab = orc.q8_matvec(w, x, n, p)
    rows = np.array([0, 7, 39, 13], np.int64)
    part, pab = orc.q8_matvec_rows(w, x, n, rows)
    assert np.array_equal(part, full[rows]) and np.array_equal(pab, ab[rows])


def test_matvec_pages_fabricated_case(orc):
    """The pages' matvec test: fabricated 0x2C00-scale weights, LCG x; the
    oracle sits far inside the pages' 5e-4 bar of the exact float dot."""
    g = GOLDEN["matvec_test_shape"]
    p, n = g["p"], g["n"]
    w = synth.pages_fabricated_q8(p, n, g["w_seed"])
    lcg = synth.PagesLCG(g["x_seed"])
    x = np.array([lcg.next_f32() for _ in range(n)], np.float32)
    out, _ = orc.q8_matvec(w, x, n, p)
    W = np_dequant(w, p, n)
    scales = w.reshape(p, n // 32, 34)[:, :, 0:2]
    assert np.all(scales[:, :, 0] == 0x00) and np.all(scales[:, :, 1] == 0x2C)
    ref = W @ x.astype(np.float64)
    assert np.max(np.abs(out - ref)) < g["abs_bar"]
    # rounded once: within half an f32 ulp of the exact double result
    half_ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) / 2
    assert np.all(np.abs(out - ref) <= half_ulp * (1 + 1e-9))


def test_matmul_rows_are_matvecs(orc):
    n, p, m = 128, 9, 3
    w = synth.q8_matrix(4, "w", p, n)
    X = synth.normal_f32(4, "X", (m, n))
    Y, ab = orc.q8_matmul(w, X, n, p)
    W = np_dequant(w, p, n)
    ref = X.astype(np.float64) @ W.T
    assert np.all(np.abs(Y - ref) <= 1e-7 * ab)
    for i in range(m):
        yi, _ = orc.q8_matvec(w, X[i], n, p)
        assert np.array_equal(Y[i], yi)


# --------------------------------------------------------------------------- kv append
@pytest.mark.parametrize("dtype", [synth.KV_F32, synth.KV_F16])
def test_kv_append_row(orc, dtype):
    g = GOLDEN["append_test_shape"]
    w, pos, cap = g["width"], g["pos"], g["cap"]
    lcg = synth.PagesLCG(g["seed"])
    k = np.array([lcg.next_f32() for _ in range(w)], np.float32) * np.float32(300.0)
    v = np.array([lcg.next_f32() for _ in range(w)], np.float32)
    dt = np.float16 if dtype == synth.KV_F16 else np.float32
    kc = np.full((cap, w), 7, dt)
    vc = np.full((cap, w), 7, dt)
    orc.kv_append(k, v, kc, vc, dtype, pos)
    assert np.array_equal(kc[pos], k.astype(dt)) and np.array_equal(vc[pos], v.astype(dt))
    others = [r for r in range(cap) if r != pos]
    assert np.all(kc[others] == 7) and np.all(vc[others] == 7)


# --------------------------------------------------------------------------- attention
def np_attention(q, kc, vc, H, Hk, d, L, scale):
    G = H // Hk
    K = kc[:L].astype(np.float64).reshape(L, Hk, d)
    V = vc[:L].astype(np.float64).reshape(L, Hk, d)
    out = np.empty((H, d))
    for h in range(H):
        s = scale * (K[:, h // G, :] @ q[h * d:(h + 1) * d].astype(np.float64))
        e = np.exp(s - s.max())
        out[h] = (e / e.sum()) @ V[:, h // G, :]
    return out.ravel()


@pytest.mark.parametrize("dtype", [synth.KV_F32, synth.KV_F16])
def test_attention_single_position_returns_v(orc, dtype):
    H, Hk, d, cap = 6, 2, 64, 4
    dt = np.float16 if dtype == synth.KV_F16 else np.float32
    q = synth.normal_f32(0, "q", H * d) * 10
    kc = synth.normal_f32(0, "k", (cap, Hk * d)).astype(dt)
    vc = synth.normal_f32(0, "v", (cap, Hk * d)).astype(dt)
    out, _ = orc.gqa_decode_attn(q, kc, vc, dtype, H, Hk, d, 1, 0.125)
    for h in range(H):
        g = h // (H // Hk)
        assert np.array_equal(out[h * d:(h + 1) * d], vc[0, g * d:(g + 1) * d].astype(np.float32))


def test_attention_identical_keys_and_zero_query_give_mean_v(orc):
    H, Hk, d, L = 4, 2, 32, 37
    v = synth.normal_f32(1, "v", (L, Hk * d))
    krow = synth.normal_f32(1, "k", Hk * d)
    k = np.tile(krow, (L, 1))
    q = synth.normal_f32(1, "q", H * d)
    mean = v.astype(np.float64).mean(axis=0)
    for qq, kk in ((q, k), (np.zeros_like(q), synth.normal_f32(2, "k2", (L, Hk * d)))):
        out, _ = orc.gqa_decode_attn(qq, kk, v, synth.KV_F32, H, Hk, d, L, 1 / math.sqrt(d))
        for h in range(H):
            g = h // (H // Hk)
            assert np.allclose(out[h * d:(h + 1) * d], mean[g * d:(g + 1) * d], rtol=0, atol=1e-6)


@pytest.mark.parametrize("H,Hk,d,L", [(4, 2, 16, 9), (14, 2, 64, 33), (16, 8, 128, 5), (3, 3, 16, 2)])
def test_attention_brute_force(orc, H, Hk, d, L):
    cap = L + 3
    q = synth.normal_f32(7, "q", H * d)
    kc = synth.normal_f16(7, "k", (cap, Hk * d))
    vc = synth.normal_f16(7, "v", (cap, Hk * d))
    out, ab = orc.gqa_decode_attn(q, kc, vc, synth.KV_F16, H, Hk, d, L, 1 / math.sqrt(d))
    ref = np_attention(q, kc, vc, H, Hk, d, L, 1 / math.sqrt(d))
    assert np.all(np.abs(out - ref) <= 1e-7 * ab)


def test_attention_pages_shape_gqa_mapping(orc):
    """The pages' attention test shape; query head h reads KV head h // 2
    (contiguous groups), which differs from h % 2 for heads 1 and 2."""
    g = GOLDEN["attention_test_shape"]
    H, Hk, d, L = g["n_heads"], g["n_kv_heads"], g["head_dim"], g["seq"]
    lcg = synth.PagesLCG(g["seed"])
    q = np.array([lcg.next_f32() for _ in range(H * d)], np.float32)
    k = np.array([lcg.next_f32() for _ in range(L * Hk * d)], np.float32).reshape(L, Hk * d)
    v = np.array([lcg.next_f32() for _ in range(L * Hk * d)], np.float32).reshape(L, Hk * d)
    out, _ = orc.gqa_decode_attn(q, k, v, synth.KV_F32, H, Hk, d, L, 1 / math.sqrt(d))
    ref = np_attention(q, k, v, H, Hk, d, L, 1 / math.sqrt(d))
    assert np.max(np.abs(out - ref)) < g["abs_bar"] * 1e-3
    # the modulo mapping would give a different answer
    Kr = k.reshape(L, Hk, d)
    wrong = Kr[:, 1, :] @ q[d:2 * d]
    right = Kr[:, 0, :] @ q[d:2 * d]
    assert not np.allclose(wrong, right)


# --------------------------------------------------------------------------- glue
def test_rmsnorm(orc):
    x = synth.normal_f32(3, "x", 1024).astype(np.float64) * 5
    w = synth.gains(3, "w", 1024)
    out = orc.rmsnorm(x, w, 1e-6)
    ref = x / np.sqrt(np.mean(x * x) + 1e-6) * w
    assert np.allclose(out, ref, rtol=1e-13, atol=0)
    # unit gain: the output has mean square 1 (up to eps)
    out1 = orc.rmsnorm(x, np.ones(1024, np.float32), 0.0)
    assert abs(np.mean(out1 * out1) - 1.0) < 1e-12


def test_rope_rotation(orc):
    g = GOLDEN["rope_test_shape"]
    d, pos, theta = g["head_dim"], g["pos"], g["theta"]
    x = synth.normal_f32(g["seed"], "x", d).astype(np.float64)
    y = orc.rope_head(x, pos, theta)
    half = d // 2
    # each (i, i + d/2) pair keeps its length and turns by pos * theta^(-i/half)
    for i in range(half):
        a, b = x[i], x[i + half]
        c, s = y[i], y[i + half]
        assert abs((a * a + b * b) - (c * c + s * s)) < 1e-12 * (a * a + b * b + 1)
        ang = pos * theta ** (-i / half)
        assert abs(math.atan2(a * s - b * c, a * c + b * s) - math.remainder(ang, 2 * math.pi)) < 1e-9
    assert np.array_equal(orc.rope_head(x, 0, theta), x)    # position 0 is the identity
    # pair 0 rotates by exactly pos radians
    assert abs(y[0] - (x[0] * math.cos(pos) - x[half] * math.sin(pos))) < 1e-12


def test_silu(orc):
    assert orc.silu_mul(0.0, 5.0) == 0.0
    assert orc.silu_mul(50.0, 1.0) == pytest.approx(50.0, rel=1e-20)
    assert orc.silu_mul(-800.0, 1.0) == 0.0
    assert orc.silu_mul(1.0, 2.0) == pytest.approx(2.0 / (1 + math.exp(-1.0)), rel=1e-15)


def test_argmax_pages_planted_tie(orc):
    g = GOLDEN["argmax_tie"]
    lcg = synth.PagesLCG(g["lcg_seed"])
    x = np.array([lcg.next_f32() for _ in range(g["n"])], np.float32)
    for i in g["tie_indices"]:
        x[i] = g["tie_value"]
    assert orc.argmax(x) == g["expected"]
    x2 = x.copy()
    x2[5] = np.nan
    assert orc.argmax(x2) == g["expected"]


# --------------------------------------------------------------------------- decode step
def np_step(w, caches, token, pos):
    """Independent numpy composition of the step (f64), for the oracle's glue."""
    s = w.shape
    d, H, Hk = s.head_dim, s.n_heads, s.n_kv_heads
    x = np_dequant(w.embed, s.vocab, s.hidden)[token].copy()

    def rms(v, g):
        return v / np.sqrt(np.mean(v * v) + s.rms_eps) * g.astype(np.float64)

    def rope(v):
        v = v.reshape(-1, d).copy()
        half = d // 2
        i = np.arange(half)
        ang = pos * (1.0 / s.rope_theta ** (i / half))
        c, sn = np.cos(ang), np.sin(ang)
        a, b = v[:, :half].copy(), v[:, half:].copy()
        v[:, :half] = a * c - b * sn
        v[:, half:] = a * sn + b * c
        return v.ravel()

    dt = np.float16 if s.kv_dtype == synth.KV_F16 else np.float32
    for li, L in enumerate(w.layers):
        xn = rms(x, L["attn_norm"])
        q = np_dequant(L["wq"], s.q_width, s.hidden) @ xn
        k = np_dequant(L["wk"], s.kv_width, s.hidden) @ xn
        v = np_dequant(L["wv"], s.kv_width, s.hidden) @ xn
        if s.qkv_bias:
            q, k, v = q + L["bq"], k + L["bk"], v + L["bv"]
        if s.qk_norm:
            q = np.concatenate([rms(h, L["q_norm"]) for h in q.reshape(H, d)])
            k = np.concatenate([rms(h, L["k_norm"]) for h in k.reshape(Hk, d)])
        q, k = rope(q), rope(k)
        kc, vc = caches[li]
        kc[pos] = k.astype(np.float32).astype(dt)
        vc[pos] = v.astype(np.float32).astype(dt)
        att = np_attention(q, kc, vc, H, Hk, d, pos + 1, 1 / math.sqrt(d))
        x = x + np_dequant(L["wo"], s.hidden, s.q_width) @ att
        xn = rms(x, L["ffn_norm"])
        g = np_dequant(L["wg"], s.ffn, s.hidden) @ xn
        u = np_dequant(L["wu"], s.ffn, s.hidden) @ xn
        hh = g / (1 + np.exp(-g)) * u
        x = x + np_dequant(L["wd"], s.hidden, s.ffn) @ hh
    xn = rms(x, w.out_norm)
    return (np_dequant(w.lm_head, s.vocab, s.hidden) @ xn).astype(np.float32)


@pytest.mark.parametrize("pos", [0, 5])
def test_decode_step_composition(orc, pos):
    shape = synth.tiny_shape(2)
    w = synth.step_weights(shape, seed=3)
    cap = 8
    caches = [synth.kv_prefix(shape, 3, li, cap, pos) for li in range(shape.n_layers)]
    host = orc.HostStep(w, cap, [(k.copy(), v.copy()) for k, v in caches])
    logits, nxt = host.step(token=17, pos=pos)
    np_caches = [(k.copy(), v.copy()) for k, v in caches]
    ref = np_step(w, np_caches, 17, pos)
    scale = np.max(np.abs(ref))
    assert np.max(np.abs(logits - ref)) <= 1e-9 * scale
    assert nxt == int(np.argmax(logits))
    for (kc, vc), (rk, rv) in zip(host.caches, np_caches):
        assert np.array_equal(kc, rk) and np.array_equal(vc, rv)


def test_decode_step_pos0_attention_is_v(orc):
    """At position 0 attention sees one row, so the first layer's attention
    output equals the freshly appended V row: changing every K row leaves the
    logits unchanged, changing V changes them (control)."""
    shape = synth.tiny_shape(1)
    w = synth.step_weights(shape, seed=4)
    a = orc.HostStep(w, 4)
    la, _ = a.step(3, 0)
    w2 = synth.step_weights(shape, seed=4)
    w2.layers[0]["wk"] = synth.q8_matrix(99, "other", shape.kv_width, shape.hidden)
    b = orc.HostStep(w2, 4)
    lb, _ = b.step(3, 0)
    assert np.array_equal(la, lb)
    w3 = synth.step_weights(shape, seed=4)
    w3.layers[0]["wv"] = synth.q8_matrix(99, "other", shape.kv_width, shape.hidden)
    c = orc.HostStep(w3, 4)
    lc, _ = c.step(3, 0)
    assert not np.array_equal(la, lc)


# --------------------------------------------------------------------------- packed Q8_0 KV
def q8kv_parts(blk):
    """(scale as float64, quants as int) of one 34-byte block."""
    return float(blk[0:2].copy().view("<f2")[0]), blk[2:].view(np.int8).astype(np.int64)


def test_q8kv_quantize_zero_block(orc):
    assert np.array_equal(orc.q8_0_quantize_block(np.zeros(32, np.float32)), np.zeros(34, np.uint8))


def test_q8kv_quantize_exact_multiples_of_a_power_of_two(orc):
    """x = k * 2^-3 with integer k, max |k| = 127: d = 2^-3 exactly, so the
    block is the scale 0x3000 and the quants k."""
    k = synth.stream(0, "q8kv.k").integers(-127, 128, 32)
    k[5] = -127
    b = orc.q8_0_quantize_block((k * 0.125).astype(np.float32))
    assert b[0] == 0x00 and b[1] == 0x30
    assert np.array_equal(b[2:].view(np.int8), k.astype(np.int8))


def test_q8kv_quantize_halves_round_away_from_zero(orc):
    """amax = 127 makes d = 1: x * id is x itself, so halves show the rounding."""
    x = np.zeros(32, np.float32)
    x[:9] = [127, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, 0.49999997]
    b = orc.q8_0_quantize_block(x)
    assert b[0] == 0x00 and b[1] == 0x3C
    assert list(b[2:11].view(np.int8)) == [127, 3, -3, 1, -1, 2, -2, 127, 0]


@pytest.mark.parametrize("sigma", [1e-3, 1.0, 300.0])
def test_q8kv_quantize_round_trip_and_symmetry(orc, sigma):
    """Random blocks: the largest |x| maps to +-127; every element comes back
    within half a step of d = amax/127 plus the scale's f16 rounding; -x
    gives the same scale and negated quants."""
    X = (synth.normal_f32(3, f"q8kv.rt{sigma}", (64, 32)) * np.float32(sigma)).astype(np.float32)
    for x in X:
        b = orc.q8_0_quantize_block(x)
        s, q = q8kv_parts(b)
        d = np.max(np.abs(x.astype(np.float64))) / 127
        assert abs(s - d) <= 2.0 ** -11 * d + 2.0 ** -25  # (binary16 subnormals below 2^-14)
        assert np.max(np.abs(q)) == 127
        assert np.all(np.abs(x - s * q) <= 0.5 * d * (1 + 1e-6) + np.abs(s - d) * np.abs(q))
        bn = orc.q8_0_quantize_block(-x)
        assert np.array_equal(bn[:2], b[:2]) and np.array_equal(bn[2:].view(np.int8), -q)


def test_q8kv_pages_memory_ratio(orc):
    """The pages' 3.76x memory win of the packed cache over f32: 128 bytes of
    f32 per 32 elements against one 34-byte block."""
    g = GOLDEN["packed_kv_memory_ratio"]
    kvw = 512
    ratio = orc.kv_row_bytes(synth.KV_F32, kvw) / orc.kv_row_bytes(synth.KV_Q8_0, kvw)
    assert round(ratio, g["digits"]) == g["ratio"]


def test_q8kv_append_row(orc):
    g = GOLDEN["append_test_shape"]
    w, pos, cap = 2 * g["width"], g["pos"], g["cap"]
    lcg = synth.PagesLCG(g["seed"])
    k = np.array([lcg.next_f32() for _ in range(w)], np.float32) * np.float32(300.0)
    v = np.array([lcg.next_f32() for _ in range(w)], np.float32)
    rb = w // 32 * 34
    kc = np.full((cap, rb), 7, np.uint8)
    vc = np.full((cap, rb), 7, np.uint8)
    orc.kv_append(k, v, kc, vc, synth.KV_Q8_0, pos)
    for c, x in ((kc, k), (vc, v)):
        want = np.concatenate([orc.q8_0_quantize_block(x[32 * i:32 * i + 32]) for i in range(w // 32)])
        assert np.array_equal(c[pos], want)
        assert np.all(np.delete(c, pos, axis=0) == 7)


@pytest.mark.parametrize("H,Hk,d,L", [(4, 2, 32, 9), (14, 2, 64, 33), (28, 4, 128, 17)])
def test_q8kv_attention_equals_dequantized_cache(orc, H, Hk, d, L):
    """Attention over a packed cache equals, bit for bit, attention over an
    f32 cache holding its dequantised values (exact in f32), and matches
    numpy brute force."""
    cap = L + 2
    q = synth.normal_f32(5, "q8kv.q", H * d)
    kc = synth.q8_kv_cache(5, "q8kv.kc", cap, Hk * d)
    vc = synth.q8_kv_cache(5, "q8kv.vc", cap, Hk * d)
    kf = np_dequant(kc, cap, Hk * d).astype(np.float32)
    vf = np_dequant(vc, cap, Hk * d).astype(np.float32)
    out, ab = orc.gqa_decode_attn(q, kc, vc, synth.KV_Q8_0, H, Hk, d, L, 1 / math.sqrt(d))
    out2, ab2 = orc.gqa_decode_attn(q, kf, vf, synth.KV_F32, H, Hk, d, L, 1 / math.sqrt(d))
    assert np.array_equal(out, out2) and np.array_equal(ab, ab2)
    ref = np_attention(q, kf, vf, H, Hk, d, L, 1 / math.sqrt(d))
    assert np.all(np.abs(out - ref) <= 1e-7 * ab)


def test_q8kv_attention_single_position_returns_dequantized_v(orc):
    H, Hk, d = 6, 2, 64
    q = synth.normal_f32(6, "q8kv.q1", H * d) * 10
    kc = synth.q8_kv_cache(6, "q8kv.k1", 3, Hk * d)
    vc = synth.q8_kv_cache(6, "q8kv.v1", 3, Hk * d)
    out, _ = orc.gqa_decode_attn(q, kc, vc, synth.KV_Q8_0, H, Hk, d, 1, 0.125)
    v0 = np_dequant(vc, 3, Hk * d)[0].astype(np.float32)
    for h in range(H):
        g = h // (H // Hk)
        assert np.array_equal(out[h * d:(h + 1) * d], v0[g * d:(g + 1) * d])


# --------------------------------------------------------------------------- windowed attention
@pytest.mark.parametrize("dtype", [synth.KV_F32, synth.KV_F16, synth.KV_Q8_0])
def test_window_full_span_is_causal_attention(orc, dtype):
    H, Hk, d, L, cap = 6, 2, 64, 37, 50
    q = synth.normal_f32(11, "w.q", H * d)
    if dtype == synth.KV_Q8_0:
        kc, vc = synth.q8_kv_cache(11, "w.k", cap, Hk * d), synth.q8_kv_cache(11, "w.v", cap, Hk * d)
    else:
        dt = np.float16 if dtype == synth.KV_F16 else np.float32
        kc = synth.normal_f32(11, "w.k", (cap, Hk * d)).astype(dt)
        vc = synth.normal_f32(11, "w.v", (cap, Hk * d)).astype(dt)
    a, aa = orc.gqa_decode_attn(q, kc, vc, dtype, H, Hk, d, L, 0.125)
    b, bb = orc.gqa_decode_attn_runs(q, kc, vc, dtype, H, Hk, d, [(0, L)], 0.125)
    assert np.array_equal(a, b) and np.array_equal(aa, bb)


@pytest.mark.parametrize("cell", [0, 17, 49])
def test_window_one_cell_returns_that_v_row(orc, cell):
    """The pages' one-cell window gate: the named cell's V row, bitwise."""
    H, Hk, d, cap = 6, 3, 32, 50
    q = synth.normal_f32(12, "w1.q", H * d) * 20
    kc = synth.normal_f16(12, "w1.k", (cap, Hk * d))
    vc = synth.normal_f16(12, "w1.v", (cap, Hk * d))
    out, _ = orc.gqa_decode_attn_runs(q, kc, vc, synth.KV_F16, H, Hk, d, [(cell, 1), (0, 0)], 0.3)
    for h in range(H):
        g = h // (H // Hk)
        assert np.array_equal(out[h * d:(h + 1) * d], vc[cell, g * d:(g + 1) * d].astype(np.float32))


def test_window_runs_brute_force_and_shift_control(orc):
    """A shared prefix run plus a gapped private run against numpy over the
    gathered rows; shifting the private run by one cell changes the output;
    swapping the runs' order changes only rounding."""
    H, Hk, d, cap = 8, 2, 64, 120
    q = synth.normal_f32(13, "wr.q", H * d)
    kc = synth.normal_f32(13, "wr.k", (cap, Hk * d))
    vc = synth.normal_f32(13, "wr.v", (cap, Hk * d))
    runs = [(0, 20), (60, 15)]
    out, ab = orc.gqa_decode_attn_runs(q, kc, vc, synth.KV_F32, H, Hk, d, runs, 0.125)
    rows = list(range(0, 20)) + list(range(60, 75))
    ref = np_attention(q, kc[rows], vc[rows], H, Hk, d, len(rows), 0.125)
    assert np.all(np.abs(out - ref) <= 1e-7 * ab)
    shifted, _ = orc.gqa_decode_attn_runs(q, kc, vc, synth.KV_F32, H, Hk, d, [(0, 20), (61, 15)], 0.125)
    assert not np.array_equal(out, shifted)
    swapped, _ = orc.gqa_decode_attn_runs(q, kc, vc, synth.KV_F32, H, Hk, d, runs[::-1], 0.125)
    assert np.all(np.abs(out - swapped) <= 1e-7 * ab)


def test_window_refuses_bad_runs(orc):
    q = np.zeros(64, np.float32)
    kc = np.zeros((10, 64), np.float32)
    for runs in ([(0, 0)], [(-1, 3)], [(8, 3)], [(0, 5), (9, 2)]):
        with pytest.raises(ValueError):
            orc.gqa_decode_attn_runs(q, kc, kc, synth.KV_F32, 1, 1, 64, runs, 1.0)
