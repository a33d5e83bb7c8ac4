"""Pins of the fp64 oracle to things other than itself.

Each test checks the oracle against what the mathematics fixes: published
generator values, closed forms, invariants, brute force on tiny inputs and
special cases of the whole decoder that reduce to library routines.  They are
chosen so that a dropped term, a wrong sign or index, or a transposed operand
anywhere in oracle.c fails at least one of them (tests/test_oracle_mutants.py
plants such mistakes and checks that they are caught).
"""
from dataclasses import replace
import math
from pathlib import Path

import numpy as np
import pytest
from scipy.special import expit

import oracle
import synth
from synth.configs import ModelCfg

GOLDEN = Path(__file__).parent / "golden"
ONE_BF16 = 0x3F80


def f64(bits):
    return synth.bf16_to_f64(np.asarray(bits, dtype=np.uint16))


def to_bf16_bits(x):
    """Exact values only (small integers, 0, +-1): asserts exactness."""
    x = np.asarray(x, dtype=np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(f64(bits), x.astype(np.float64)), "value not exactly representable in bf16"
    return bits


def rng(seed=0):
    return np.random.default_rng(seed)


# ----------------------------------------------------------- generator pins

def test_splitmix64_published_values():
    rows = [l.split() for l in (GOLDEN / "splitmix64_state0.txt").read_text().splitlines() if l and l[0] != "#"]
    got = synth.stream(0, 0, len(rows))
    for (idx, val), g in zip(rows, got):
        assert int(g) == int(val, 16), f"output {idx}"


def test_stream_composition():
    # key(seed, tid) is output tid of the stream at state seed; u is output i of the stream at key
    seed, tid = 12345, 77
    key = int(synth.stream(seed, tid, 1)[0])
    assert np.array_equal(synth.u64(seed, tid, 5, 10), synth.stream(key, 5, 10))


def test_normal_generator_moments_and_bound():
    sigma = 0.02
    z = f64(synth.normal_bf16((1 << 20,), 3, 9, sigma))
    assert abs(z.mean()) < 4 * sigma / math.sqrt(z.size)
    assert abs(z.std() / sigma - 1) < 0.01
    # Irwin-Hall of four uniforms is bounded by sqrt(3) * 2 = 3.4641 sigma (plus bf16 rounding)
    assert np.abs(z).max() <= 3.4642 * sigma * (1 + 2 ** -8)
    # roughly normal: fraction within one sigma (normal: 0.6827; Irwin-Hall n=4: 0.6665)
    assert 0.65 < np.mean(np.abs(z) < sigma) < 0.69


def test_gain_generator_ones_and_offsets():
    ones = synth.normal_bf16((1000,), 0, 3, 0.0, 1.0)
    assert np.all(ones == ONE_BF16)
    g = f64(synth.normal_bf16((1 << 16,), 0, 3, 0.1, 1.0))
    assert abs(g.mean() - 1) < 0.005 and abs(g.std() - 0.1) < 0.003


def test_tokens_uniform_and_in_range():
    t = synth.tokens(200000, 0, 0, 1000)
    assert t.min() >= 0 and t.max() < 1000
    counts = np.bincount(t, minlength=1000)
    chi2 = ((counts - 200) ** 2 / 200).sum()
    assert chi2 < 1000 + 6 * math.sqrt(2000)


# ------------------------------------------------------------------ RMSNorm

def test_rmsnorm_unit_rms_and_scale_invariance():
    x = rng(1).normal(size=257) * 3.7
    ones = np.full(257, ONE_BF16, dtype=np.uint16)
    y = oracle.rmsnorm(x, ones, 0.0)
    assert abs(np.sqrt(np.mean(y ** 2)) - 1) < 1e-14
    assert np.allclose(oracle.rmsnorm(5.5 * x, ones, 0.0), y, rtol=1e-14, atol=0)
    assert np.allclose(y * np.sqrt(np.mean(x ** 2)), x, rtol=1e-13)  # direction kept


def test_rmsnorm_gain_is_elementwise():
    x = rng(2).normal(size=64)
    g = synth.normal_bf16((64,), 0, 5, 0.1, 1.0)
    ones = np.full(64, ONE_BF16, dtype=np.uint16)
    assert np.allclose(oracle.rmsnorm(x, g, 1e-5), f64(g) * oracle.rmsnorm(x, ones, 1e-5), rtol=1e-14)


def test_rmsnorm_eps_inside_sqrt():
    # constant vector c: y = g c / sqrt(c^2 + eps)
    c, eps = 0.01, 1e-3
    x = np.full(16, c)
    y = oracle.rmsnorm(x, np.full(16, ONE_BF16, dtype=np.uint16), eps)
    assert np.allclose(y, c / math.sqrt(c * c + eps), rtol=1e-14)
    assert np.all(oracle.rmsnorm(np.zeros(8), np.full(8, ONE_BF16, dtype=np.uint16), 1e-5) == 0)


# ------------------------------------------------------------------- matvec

def test_matvec_matches_library_matmul_nonsquare():
    W = synth.normal_bf16((7, 13), 0, 11, 0.5)
    x = rng(3).normal(size=13)
    assert np.allclose(oracle.matvec(W, x), f64(W) @ x, rtol=1e-13, atol=1e-15)


def test_bf16_widening_exact():
    assert oracle.bf16_value(0x3F80) == 1.0
    assert oracle.bf16_value(0xC040) == -3.0
    assert oracle.bf16_value(0x3C23) == float(np.float32(np.uint32(0x3C230000).view(np.float32)))


# --------------------------------------------------------------------- RoPE

@pytest.mark.parametrize("d", [4, 64, 128])
def test_rope_preserves_rotate_half_pair_norms(d):
    v = rng(d).normal(size=d)
    r = oracle.rope(v, 37, 1e4)
    h = d // 2
    assert np.allclose(v[:h] ** 2 + v[h:] ** 2, r[:h] ** 2 + r[h:] ** 2, rtol=1e-13)


def test_rope_position_zero_is_identity():
    v = rng(4).normal(size=64)
    assert np.array_equal(oracle.rope(v, 0, 5e5), v)


def test_rope_composes_additively():
    v = rng(5).normal(size=64)
    # rotating by a then b equals rotating by a + b (angle linear in position)
    assert np.allclose(oracle.rope(oracle.rope(v, 11, 1e4), 29, 1e4), oracle.rope(v, 40, 1e4), atol=1e-12)


def test_rope_relative_position_property():
    q, k = rng(6).normal(size=128), rng(7).normal(size=128)
    a = oracle.rope(q, 100, 5e5) @ oracle.rope(k, 93, 5e5)
    b = oracle.rope(q, 1007, 5e5) @ oracle.rope(k, 1000, 5e5)
    assert abs(a - b) < 1e-10 * (1 + abs(a))


def test_rope_d2_closed_form_direction():
    for p in (1, 2, 5):
        r = oracle.rope(np.array([1.0, 0.0]), p, 1e4)
        assert np.allclose(r, [math.cos(p), math.sin(p)], atol=1e-15)


def test_rope_frequency_exponent():
    # d = 4: element 1 pairs with element 3 and turns at theta^(-2/4) rad per position
    theta, p = 1e4, 3
    r = oracle.rope(np.array([0.0, 1.0, 0.0, 0.0]), p, theta)
    ang = p * theta ** -0.5
    assert np.allclose(r, [0.0, math.cos(ang), 0.0, math.sin(ang)], atol=1e-15)


# --------------------------------------------------------------- attention

def _attention_brute(q, K, V):
    d = len(q)
    s = [sum(q[e] * K[j][e] for e in range(d)) / math.sqrt(d) for j in range(len(K))]
    den = sum(math.exp(v) for v in s)
    return [sum(math.exp(s[j]) / den * V[j][e] for j in range(len(K))) for e in range(d)]


def test_attention_brute_force_tiny():
    r = rng(8)
    q, K, V = r.normal(size=4), r.normal(size=(5, 4)), r.normal(size=(5, 4))
    assert np.allclose(oracle.attention_head(q, K, V), _attention_brute(q, K, V), rtol=1e-13)


def test_attention_weights_sum_to_one():
    r = rng(9)
    q, K = r.normal(size=16) * 3, r.normal(size=(33, 16)) * 3
    assert np.allclose(oracle.attention_head(q, K, np.ones((33, 16))), 1.0, rtol=1e-14)


def test_attention_single_position_returns_value():
    r = rng(10)
    v = r.normal(size=(1, 8))
    assert np.allclose(oracle.attention_head(r.normal(size=8), r.normal(size=(1, 8)), v), v[0], rtol=1e-15)


def test_attention_identical_keys_give_mean():
    r = rng(11)
    k = r.normal(size=8)
    V = r.normal(size=(6, 8))
    assert np.allclose(oracle.attention_head(r.normal(size=8), np.tile(k, (6, 1)), V), V.mean(0), rtol=1e-13)


def test_attention_two_key_logistic_closed_form():
    # scores a/sqrt(d) and 0: weight of key 0 is expit(a / sqrt(d))
    d, a = 16, 3.0
    q = np.zeros(d)
    q[0] = a
    K = np.zeros((2, d))
    K[0, 0] = 1.0
    V = np.zeros((2, d))
    V[0, 0], V[1, 1] = 1.0, 1.0
    out = oracle.attention_head(q, K, V)
    w = expit(a / math.sqrt(d))
    assert abs(out[0] - w) < 1e-15 and abs(out[1] - (1 - w)) < 1e-15


def test_attention_large_scores_stable_and_permutation_invariant():
    r = rng(12)
    q, K, V = r.normal(size=8) * 100, r.normal(size=(9, 8)) * 100, r.normal(size=(9, 8))
    out = oracle.attention_head(q, K, V)
    assert np.all(np.isfinite(out))
    perm = r.permutation(9)
    assert np.allclose(oracle.attention_head(q, K[perm], V[perm]), out, rtol=1e-12, atol=1e-14)


# -------------------------------------------------------------------- SiLU

def test_silu_identities():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0)) < 1e-15
    for z in (0.3, 1.7, 5.0):
        # z sigma(z) - (-z) sigma(-z) = z
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-14
        assert abs(oracle.silu(z) - z * expit(z)) < 1e-15


# ----------------------------------------------------------- whole decoder

TINY_T = ModelCfg("pin", n_layers=2, hidden=32, n_q_heads=4, n_kv_heads=2, head_dim=8, ffn_dim=48, vocab=40,
                  rope_theta=1e4, weight_std=0.2)


def _model(cfg, seed=0, gains=False):
    if gains:
        cfg = replace(cfg, random_gains=True)
    return oracle.Model(cfg, synth.host_weights(cfg, seed)), synth.host_weights(cfg, seed)


def test_decode_equals_full_causal_forward():
    m, _ = _model(TINY_T, gains=True)
    toks = synth.tokens(12, 0, 0, TINY_T.vocab)
    full = m.full_forward(toks)
    kc, vc = m.new_cache(16)
    for p, t in enumerate(toks):
        step = m.decode_step(kc, vc, int(t), p)
        assert np.allclose(step, full[p], rtol=1e-11, atol=1e-12), f"position {p}"


def test_round_bf16_matches_fp32_round_to_nearest_even():
    """For values exactly representable in fp32, the nearest bf16 is fp32's
    top 16 bits rounded to nearest, ties to even: written here as integer bit
    manipulation, independent of the oracle's arithmetic on doubles."""
    r = rng(3)
    x = (r.standard_normal(20000) * 2.0 ** r.integers(-30, 30, 20000)).astype(np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    want = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    got = np.array([oracle.round_bf16(float(v)) for v in x])
    assert np.array_equal(got, want)
    # ties: 1 + 2^-8 is half way between 1 and 1 + 2^-7 (odd significand) -> 1;
    # 1 + 3 * 2^-8 is half way between 1 + 2^-7 and 1 + 2^-6 (even) -> 1 + 2^-6
    assert oracle.round_bf16(1 + 2 ** -8) == 1.0 and oracle.round_bf16(-(1 + 2 ** -8)) == -1.0
    assert oracle.round_bf16(1 + 3 * 2 ** -8) == 1 + 2 ** -6
    for v in (0.0, 1.0, -2.5, 2.0 ** -100, 3.0 * 2 ** 60):
        assert oracle.round_bf16(v) == v
    assert all(oracle.round_bf16(g) == g for g in got[:200])  # idempotent


def _is_bf16(a):
    a32 = np.asarray(a, dtype=np.float64).astype(np.float32)
    return np.array_equal(a32.astype(np.float64), np.asarray(a)) and not np.any(a32.view(np.uint32) & 0xFFFF)


def test_bf16_cache_holds_bf16_values_and_decode_equals_full_forward():
    """With a bf16 KV cache every stored key and value is a bf16 value, and
    token-by-token decode still equals the full causal forward, which rounds
    its keys and values in a separate code path; the rounding moves the
    logits, but only by a rounding-sized amount."""
    w = synth.host_weights(TINY_T, 0)
    m = oracle.Model(TINY_T, w, kv_bf16=True)
    toks = synth.tokens(12, 0, 2, TINY_T.vocab)
    full = m.full_forward(toks)
    kc, vc = m.new_cache(16)
    for p, t in enumerate(toks):
        step = m.decode_step(kc, vc, int(t), p)
        assert np.allclose(step, full[p], rtol=1e-11, atol=1e-12), f"position {p}"
    assert _is_bf16(kc[:, :12]) and _is_bf16(vc[:, :12])
    plain = oracle.Model(TINY_T, w).full_forward(toks)
    assert not np.allclose(full, plain, rtol=0, atol=1e-9)
    assert np.linalg.norm(full - plain) / np.linalg.norm(plain) < 1e-2


def test_full_forward_is_causal():
    m, _ = _model(TINY_T)
    toks = synth.tokens(10, 0, 1, TINY_T.vocab)
    other = toks.copy()
    other[6:] = (other[6:] + 7) % TINY_T.vocab
    a, b = m.full_forward(toks), m.full_forward(other)
    assert np.allclose(a[:6], b[:6], rtol=1e-14, atol=0)
    assert not np.allclose(a[6:], b[6:])


def _zero_layer(cfg):
    w = {}
    for name, shape in synth.layer_shapes(cfg).items():
        w[name] = np.full(shape, ONE_BF16, dtype=np.uint16) if name.endswith("norm") else np.zeros(shape, np.uint16)
    return w


def test_zero_layers_reduce_to_norm_and_head():
    # with every projection zero the residual stream is the embedding, so
    # logits = W_lm rmsnorm(emb[t]) (W_lm is vocab x hidden, not square)
    cfg = TINY_T
    w = synth.host_weights(replace(cfg, random_gains=True), 0)
    w["layers"] = [_zero_layer(cfg) for _ in range(cfg.n_layers)]
    m = oracle.Model(cfg, w)
    kc, vc = m.new_cache(8)
    for p, t in enumerate([3, 17, 39]):
        e = f64(w["embed"][t])
        xn = f64(w["final_norm"]) * e / np.sqrt(np.mean(e ** 2) + cfg.rms_eps)
        assert np.allclose(m.decode_step(kc, vc, t, p), f64(w["lm_head"]) @ xn, rtol=1e-12, atol=1e-14)


def test_uniform_attention_special_case():
    # Wq = 0 makes every score 0, so each q head h returns the mean over
    # positions 0..p of v[h // group]; Wo = I, MLP off, one layer.
    cfg = replace(TINY_T, n_layers=1)
    H, d, nq, nkv = cfg.hidden, cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    assert H == nq * d
    w = synth.host_weights(cfg, 4)
    lw = _zero_layer(cfg)
    lw["wk"] = w["layers"][0]["wk"]
    lw["wv"] = w["layers"][0]["wv"]
    lw["wo"] = to_bf16_bits(np.eye(H))
    lw["attn_norm"] = synth.normal_bf16((H,), 0, 99, 0.1, 1.0)
    w["layers"] = [lw]
    m = oracle.Model(cfg, w)
    toks = [5, 9, 2, 33, 9]
    kc, vc = m.new_cache(8)
    group = nq // nkv
    vs = []
    for p, t in enumerate(toks):
        e = f64(w["embed"][t])
        xn = f64(lw["attn_norm"]) * e / np.sqrt(np.mean(e ** 2) + cfg.rms_eps)
        vs.append(f64(lw["wv"]) @ xn)
        vmean = np.mean(vs, axis=0)  # positions 0..p, current one included
        att = np.concatenate([vmean[(h // group) * d:(h // group + 1) * d] for h in range(nq)])
        x = e + att
        xf = f64(w["final_norm"]) * x / np.sqrt(np.mean(x ** 2) + cfg.rms_eps)
        assert np.allclose(m.decode_step(kc, vc, t, p), f64(w["lm_head"]) @ xf, rtol=1e-11, atol=1e-13), p


def test_attention_only_layer_brute_force():
    # one layer, MLP off: brute-force RoPE + causal softmax attention per head
    cfg = replace(TINY_T, n_layers=1)
    H, d, nq, nkv = cfg.hidden, cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    w = synth.host_weights(cfg, 5)
    lw = dict(w["layers"][0])
    for n in ("w_gate", "w_up", "w_down"):
        lw[n] = np.zeros_like(lw[n])
    w["layers"] = [lw]
    m = oracle.Model(cfg, w)
    toks = [1, 2, 3, 4]
    kc, vc = m.new_cache(4)
    Ks, Vs = [], []

    def rot(v, p):
        h = d // 2
        out = list(v)
        for i in range(h):
            ang = p * cfg.rope_theta ** (-2 * i / d)
            out[i] = v[i] * math.cos(ang) - v[i + h] * math.sin(ang)
            out[i + h] = v[i] * math.sin(ang) + v[i + h] * math.cos(ang)
        return out

    for p, t in enumerate(toks):
        e = f64(w["embed"][t])
        xn = f64(lw["attn_norm"]) * e / np.sqrt(np.mean(e ** 2) + cfg.rms_eps)
        q = f64(lw["wq"]) @ xn
        k = f64(lw["wk"]) @ xn
        v = f64(lw["wv"]) @ xn
        Ks.append([rot(k[j * d:(j + 1) * d], p) for j in range(nkv)])
        Vs.append([v[j * d:(j + 1) * d] for j in range(nkv)])
        att = []
        for h in range(nq):
            j = h // (nq // nkv)
            att += _attention_brute(rot(q[h * d:(h + 1) * d], p), [K[j] for K in Ks], [V[j] for V in Vs])
        x = e + f64(lw["wo"]) @ np.array(att)
        xf = f64(w["final_norm"]) * x / np.sqrt(np.mean(x ** 2) + cfg.rms_eps)
        assert np.allclose(m.decode_step(kc, vc, t, p), f64(w["lm_head"]) @ xf, rtol=1e-11, atol=1e-13), p


def test_mlp_only_layer_closed_form():
    # attention off (Wo = 0): x = e + Wd (silu(Wg xn) * (Wu xn)) with random gains
    cfg = replace(TINY_T, n_layers=1, random_gains=True)
    w = synth.host_weights(cfg, 6)
    lw = dict(w["layers"][0])
    lw["wo"] = np.zeros_like(lw["wo"])
    w["layers"] = [lw]
    m = oracle.Model(cfg, w)
    kc, vc = m.new_cache(4)
    for p, t in enumerate([7, 8]):
        e = f64(w["embed"][t])
        xn = f64(lw["mlp_norm"]) * e / np.sqrt(np.mean(e ** 2) + cfg.rms_eps)
        g, u = f64(lw["w_gate"]) @ xn, f64(lw["w_up"]) @ xn
        x = e + f64(lw["w_down"]) @ (g * expit(g) * u)
        xf = f64(w["final_norm"]) * x / np.sqrt(np.mean(x ** 2) + cfg.rms_eps)
        assert np.allclose(m.decode_step(kc, vc, t, p), f64(w["lm_head"]) @ xf, rtol=1e-11, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv():
    cfg = replace(TINY_T, n_layers=1)
    group = cfg.n_q_heads // cfg.n_kv_heads
    d = cfg.head_dim
    w = synth.host_weights(cfg, 7)
    mha_cfg = replace(cfg, n_kv_heads=cfg.n_q_heads)
    lw = dict(w["layers"][0])
    rep = lambda W: np.concatenate([W[(h // group) * d:(h // group + 1) * d] for h in range(cfg.n_q_heads)])
    lw["wk"], lw["wv"] = rep(lw["wk"]), rep(lw["wv"])
    w2 = dict(w)
    w2["layers"] = [lw]
    a, b = oracle.Model(cfg, w), oracle.Model(mha_cfg, w2)
    toks = synth.tokens(6, 0, 3, cfg.vocab)
    assert np.allclose(a.full_forward(toks), b.full_forward(toks), rtol=1e-12, atol=1e-14)


def test_zero_second_layer_equals_one_layer_model():
    cfg = TINY_T
    w = synth.host_weights(cfg, 8)
    w1 = dict(w)
    w1["layers"] = [w["layers"][0]]
    w2 = dict(w)
    w2["layers"] = [w["layers"][0], _zero_layer(cfg)]
    toks = synth.tokens(5, 0, 4, cfg.vocab)
    a = oracle.Model(replace(cfg, n_layers=1), w1).full_forward(toks)
    b = oracle.Model(cfg, w2).full_forward(toks)
    assert np.allclose(a, b, rtol=1e-14, atol=0)


def test_layerwise_driver_matches_decode_step():
    cfg = TINY_T
    w = synth.host_weights(cfg, 9)
    m = oracle.Model(cfg, w)
    lm = oracle.Model(cfg, {k: w[k] for k in ("embed", "lm_head", "final_norm")})
    kc, vc = m.new_cache(8)
    kc2, vc2 = m.new_cache(8)
    for p, t in enumerate([4, 5, 6]):
        ref = m.decode_step(kc, vc, t, p)
        x = lm.embed_token(t)
        for l in range(cfg.n_layers):
            lm.layer_step(w["layers"][l], kc2[l], vc2[l], p, x)
        assert np.array_equal(lm.head(x), ref)


def test_rejects_out_of_range_token_and_position():
    m, _ = _model(TINY_T)
    kc, vc = m.new_cache(4)
    with pytest.raises(ValueError):
        m.decode_step(kc, vc, TINY_T.vocab, 0)
    with pytest.raises(ValueError):
        m.decode_step(kc, vc, 0, 4)
