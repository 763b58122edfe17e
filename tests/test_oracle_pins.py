"""Pins of the CPU oracle to facts other than itself.

The pages print no worked numeric example of the forward pass, so the oracle is
pinned by the BF16 rounding definition (hand-derived bit patterns), closed forms,
invariants, special cases that reduce to a known value, and brute force in FP64
on tiny inputs. Each test names the plausible mistake it would catch.
"""
import os
from dataclasses import replace

import numpy as np
import pytest

import oracle as O
import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- BF16 rounding
def _golden_bf16():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rne.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b = line.split()[:2]
            rows.append((int(a, 16), b))
    return rows


def test_bf16_rne_golden_bit_patterns():
    rows = _golden_bf16()
    f = np.array([r[0] for r in rows], np.uint32).view(np.float32)
    got = O.bf16_from_f32(f)
    for (src, want), g in zip(rows, got):
        if want == "nan":
            assert (g & 0x7F80) == 0x7F80 and (g & 0x007F) != 0, hex(src)
        else:
            assert int(g) == int(want, 16), (hex(src), hex(int(g)), want)


def test_bf16_widening_is_exact():
    b = np.arange(0, 1 << 16, dtype=np.uint16)
    fin = (b & 0x7F80) != 0x7F80
    f = O.f32_from_bf16(b[fin])
    assert np.array_equal(O.bf16_from_f32(f), b[fin])      # round trip is the identity


# ----------------------------------------------------------------- GEMV
def test_gemv_small_integers_is_exact():
    """Integer weights/activations in [-4, 4]: every partial sum is an integer below
    2^24, so FP32 is exact and the result must equal the integer dot product.
    Catches a transposed W, a dropped column, a wrong row stride."""
    rng = np.random.default_rng(7)
    for rows, cols in [(5, 7), (33, 2048), (17, 8192)]:
        Wi = rng.integers(-4, 5, size=(rows, cols))
        xi = rng.integers(-4, 5, size=cols)
        W = O.bf16_from_f32(Wi.astype(np.float32)).reshape(rows, cols)
        y = O.gemv(W, xi.astype(np.float32))
        assert np.array_equal(y.astype(np.int64), Wi @ xi)


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_vector_closed_form():
    """x = c * 1 gives g / sqrt(1 + eps / c^2)."""
    n, eps = 2048, 1e-5
    g = O.bf16_from_f32(np.linspace(-2, 2, n).astype(np.float32))
    for c in (0.5, 3.0, -0.125):
        out = O.rmsnorm(np.full(n, c, np.float32), g, eps)
        want = O.f32_from_bf16(g).astype(np.float64) * np.sign(c) / np.sqrt(1 + eps / c ** 2)
        np.testing.assert_allclose(out, want, rtol=2e-6, atol=1e-7)


def test_rmsnorm_power_of_two_scale_invariance_bitwise():
    """With eps = 0, scaling x by 2^k leaves every output bit unchanged."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal(1024).astype(np.float32)
    g = O.bf16_from_f32(rng.standard_normal(1024).astype(np.float32))
    base = O.rmsnorm(x, g, 0.0)
    for k in (-3, 1, 5):
        assert np.array_equal(O.rmsnorm(x * np.float32(2.0 ** k), g, 0.0), base)


def test_rmsnorm_unit_gain_has_unit_rms():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(4096).astype(np.float32) * 3
    out = O.rmsnorm(x, S.ones_bf16(4096), 0.0).astype(np.float64)
    assert abs(np.sqrt(np.mean(out ** 2)) - 1.0) < 1e-5


# ----------------------------------------------------------------- RoPE
def test_rope_frequencies_geometric_without_scaling():
    cfg = S.CONFIGS["qwen3_0_6b"]
    w = O.rope_inv_freq(cfg)
    assert w[0] == 1.0
    ratio = w[1:] / w[:-1]
    np.testing.assert_allclose(ratio, cfg.rope_theta ** (-2.0 / cfg.head_dim), rtol=1e-12)


def test_rope_llama3_scaling_regions():
    """High-frequency pairs unchanged, low-frequency pairs divided by the factor,
    the band between strictly between the two and continuous at both edges."""
    cfg = S.CONFIGS["llama1b"]
    base = O.rope_inv_freq(replace(cfg, rope_scaling=False))
    sc = O.rope_inv_freq(cfg)
    lam = 2 * np.pi / base
    hi = lam < cfg.rs_orig_max / cfg.rs_high
    lo = lam > cfg.rs_orig_max / cfg.rs_low
    mid = ~hi & ~lo
    assert hi.any() and lo.any() and mid.any()
    assert np.array_equal(sc[hi], base[hi])
    np.testing.assert_allclose(sc[lo], base[lo] / cfg.rs_factor, rtol=1e-15)
    assert np.all(sc[mid] < base[mid]) and np.all(sc[mid] > base[mid] / cfg.rs_factor)
    # the smoothing weight goes to 0 at lambda = orig/low and to 1 at orig/high
    sw = (sc[mid] - base[mid] / cfg.rs_factor) / (base[mid] - base[mid] / cfg.rs_factor)
    want = (cfg.rs_orig_max / lam[mid] - cfg.rs_low) / (cfg.rs_high - cfg.rs_low)
    np.testing.assert_allclose(sw, want, rtol=1e-9)
    assert np.all(np.diff(sc) < 0)                       # still strictly decreasing


def test_rope_position_zero_is_identity_bitwise():
    cfg = S.CONFIGS["llama1b"]
    c, s = O.rope_cos_sin(cfg, 0)
    v = np.random.default_rng(3).standard_normal(cfg.head_dim).astype(np.float32)
    assert np.array_equal(O.rope_apply(v, c, s), v)


def test_rope_rotate_half_pairing():
    """A unit vector on element j lands on (cos, sin) at elements (j, j + d/2):
    an interleaved (j, j+1) pairing or a flipped sign fails this."""
    cfg = S.CONFIGS["tiny"]
    d = cfg.head_dim
    c, s = O.rope_cos_sin(cfg, 7)
    for j in (0, 5, d // 2 - 1):
        e = np.zeros(d, np.float32)
        e[j] = 1.0
        r = O.rope_apply(e, c, s)
        assert r[j] == c[j] and r[j + d // 2] == s[j]
        assert np.count_nonzero(r) <= 2


def test_rope_preserves_pair_norms_and_relative_positions():
    cfg = S.CONFIGS["llama1b"]
    d = cfg.head_dim
    rng = np.random.default_rng(4)
    q = rng.standard_normal(d).astype(np.float32)
    k = rng.standard_normal(d).astype(np.float32)

    def rot(v, p):
        c, s = O.rope_cos_sin(cfg, p)
        return O.rope_apply(v, c, s).astype(np.float64)

    r = rot(q, 1234)
    n0 = q[: d // 2].astype(np.float64) ** 2 + q[d // 2:].astype(np.float64) ** 2
    n1 = r[: d // 2] ** 2 + r[d // 2:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-5)
    a = rot(q, 100) @ rot(k, 40)
    b = rot(q, 1100) @ rot(k, 1040)
    assert abs(a - b) < 1e-4 * (1 + abs(a))


# ----------------------------------------------------------------- attention
def _fp64_attention(q, K, V, scale):
    s = (K.astype(np.float64) @ q.astype(np.float64)) * scale
    p = np.exp(s - s.max())
    p /= p.sum()
    return p @ V.astype(np.float64)


@pytest.mark.parametrize("n,d", [(1, 4), (3, 8), (5, 8), (5, 2)])
def test_attention_matches_fp64_brute_force(n, d):
    rng = np.random.default_rng(10 * n + d)
    q = O.f32_from_bf16(O.bf16_from_f32(rng.standard_normal(d).astype(np.float32)))
    K = O.bf16_from_f32(rng.standard_normal((n, d)).astype(np.float32)).reshape(n, d)
    V = O.bf16_from_f32(rng.standard_normal((n, d)).astype(np.float32)).reshape(n, d)
    got = O.attention(q, K, V, 0.5)
    want = _fp64_attention(q, O.f32_from_bf16(K).reshape(n, d), O.f32_from_bf16(V).reshape(n, d), 0.5)
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-6)


def test_attention_single_position_returns_value_bitwise():
    rng = np.random.default_rng(11)
    q = rng.standard_normal(64).astype(np.float32)
    K = O.bf16_from_f32(rng.standard_normal(64).astype(np.float32)).reshape(1, 64)
    V = O.bf16_from_f32(rng.standard_normal(64).astype(np.float32)).reshape(1, 64)
    assert np.array_equal(O.attention(q, K, V, 0.125), O.f32_from_bf16(V).reshape(64))


def test_attention_equal_keys_average_values():
    rng = np.random.default_rng(12)
    n, d = 9, 64
    q = rng.standard_normal(d).astype(np.float32)
    K = np.tile(O.bf16_from_f32(rng.standard_normal(d).astype(np.float32)), (n, 1))
    V = O.bf16_from_f32(rng.standard_normal((n, d)).astype(np.float32)).reshape(n, d)
    got = O.attention(q, K, V, 0.125)
    np.testing.assert_allclose(got, O.f32_from_bf16(V).reshape(n, d).astype(np.float64).mean(0),
                               rtol=1e-5, atol=1e-6)


def test_split_partials_and_combine_equal_unsplit():
    rng = np.random.default_rng(13)
    n, d = 200, 64
    q = O.f32_from_bf16(O.bf16_from_f32(rng.standard_normal(d).astype(np.float32)))
    K = O.bf16_from_f32(rng.standard_normal((n, d)).astype(np.float32)).reshape(n, d)
    V = O.bf16_from_f32(rng.standard_normal((n, d)).astype(np.float32)).reshape(n, d)
    full = O.attention(q, K, V, 0.125)
    for bounds in ([0, 200], [0, 64, 128, 192, 200], [0, 0, 50, 50, 200], [0, 199, 200]):
        np.testing.assert_allclose(O.attention_split(q, K, V, 0.125, bounds), full,
                                   rtol=2e-5, atol=2e-6)


# ----------------------------------------------------------------- whole decoder
def _tiny_inputs(cfg):
    return S.model_weights(cfg), *S.kv_prefill(cfg), S.prompt(cfg)


def test_decoder_causal_invariance_bitwise(tiny_cfg):
    """Appending steps leaves the logits of earlier steps bit-for-bit unchanged."""
    w, k, v, p = _tiny_inputs(tiny_cfg)
    a = O.decode(tiny_cfg, w, k.copy(), v.copy(), p, 0, 4)
    b = O.decode(tiny_cfg, w, k.copy(), v.copy(), p, 0, 9)
    assert np.array_equal(b.logits[: a.logits.shape[0]], a.logits)
    assert np.array_equal(b.tokens[:4], a.tokens)


def test_decoder_resume_from_own_cache_equals_continuous_bitwise(tiny_cfg):
    w, k, v, p = _tiny_inputs(tiny_cfg)
    full = O.decode(tiny_cfg, w, k.copy(), v.copy(), p, 0, 10)
    k2, v2 = k.copy(), v.copy()
    first = O.decode(tiny_cfg, w, k2, v2, p[:20], 0, 1)
    second = O.decode(tiny_cfg, w, k2, v2, p[19:], 19, 10)
    assert np.array_equal(np.concatenate([first.logits, second.logits[1:]]), full.logits)
    assert np.array_equal(second.tokens, full.tokens)


def test_decoder_thread_count_does_not_change_bits(tiny_cfg):
    w, k, v, p = _tiny_inputs(tiny_cfg)
    a = O.decode(tiny_cfg, w, k.copy(), v.copy(), p, 0, 6, n_threads=1)
    b = O.decode(tiny_cfg, w, k.copy(), v.copy(), p, 0, 6, n_threads=4)
    assert np.array_equal(a.logits, b.logits)


def test_decoder_greedy_is_first_argmax_and_forcing_own_tokens_is_neutral(tiny_cfg):
    w, k, v, p = _tiny_inputs(tiny_cfg)
    r = O.decode(tiny_cfg, w, k.copy(), v.copy(), p, 0, 8)
    n_prompt = p.size
    assert np.array_equal(r.tokens, r.logits[n_prompt - 1:].argmax(1))
    srt = np.sort(r.logits, 1)
    np.testing.assert_array_equal(r.gaps, srt[:, -1] - srt[:, -2])
    f = O.decode(tiny_cfg, w, k.copy(), v.copy(), p, 0, 8, force_tokens=r.tokens[:-1])
    assert np.array_equal(f.logits, r.logits)


def _zero_like(a):
    return np.zeros_like(a)


def _perm_matrix(n_out, n_in, perm, value=1.0):
    W = np.zeros((n_out, n_in), np.uint16)
    W[np.arange(n_out), perm] = O.bf16_from_f32(np.float32(value))[0]
    return W


def test_decoder_attention_special_case_closed_form(tiny_cfg):
    """Keys all zero -> uniform softmax over positions 0..P; cached values are a
    constant vector per KV head, the new value is zero; Wo is a permutation;
    the FFN is zero. Then every layer adds R(P/(P+1) c_{i//G}) permuted, and the
    logits follow in closed form. A wrong GQA head mapping, an exclusive causal
    range, a transposed Wo or a wrong tied head fails it."""
    cfg = tiny_cfg
    rng = np.random.default_rng(21)
    w = S.model_weights(cfg)
    H, d, nkv, G = cfg.hidden, cfg.head_dim, cfg.n_kv_heads, cfg.n_q_heads // cfg.n_kv_heads
    perm = rng.permutation(H)
    for lw in w.layers:
        lw["wk"] = _zero_like(lw["wk"])
        lw["wv"] = _zero_like(lw["wv"])
        lw["wo"] = _perm_matrix(H, cfg.q_dim, perm)
        lw["w_gate"] = _zero_like(lw["w_gate"])
        lw["w_up"] = _zero_like(lw["w_up"])
        lw["w_down"] = _zero_like(lw["w_down"])
    P = 5
    k = np.zeros((cfg.n_layers, nkv, cfg.max_pos, d), np.uint16)
    v = np.zeros_like(k)
    consts = O.bf16_from_f32(rng.standard_normal((nkv, d)).astype(np.float32)).reshape(nkv, d)
    v[:, :, :P, :] = consts[None, :, None, :]
    tok = np.array([17], np.int32)
    r = O.decode(cfg, w, k, v, tok, P, 1)
    # closed form in float64, rounding to bf16 where the definition does
    c = O.f32_from_bf16(consts).reshape(nkv, d).astype(np.float64)
    o = np.concatenate([c[i // G] * P / (P + 1) for i in range(cfg.n_q_heads)])
    o = O.f32_from_bf16(O.bf16_from_f32(o.astype(np.float32))).astype(np.float64)
    x = O.f32_from_bf16(w.embed[tok[0]]).astype(np.float64)
    for _ in range(cfg.n_layers):
        x = O.f32_from_bf16(O.bf16_from_f32((x + o[perm]).astype(np.float32))).astype(np.float64)
    hf = x / np.sqrt(np.mean(x ** 2) + cfg.rms_eps)
    hf = O.f32_from_bf16(O.bf16_from_f32(hf.astype(np.float32))).astype(np.float64)
    logits = O.f32_from_bf16(w.embed).reshape(cfg.vocab, H).astype(np.float64) @ hf
    np.testing.assert_allclose(r.logits[0], logits, atol=2e-4)
    assert r.tokens[0] == int(np.argmax(logits))
    # the new K/V position was written (as zeros here) and nothing else moved
    assert np.array_equal(v[:, :, :P], np.broadcast_to(consts[None, :, None, :], v[:, :, :P].shape))


def test_decoder_ffn_special_case_closed_form(tiny_cfg):
    """Attention output projection zero; gate = rows 0..H-1 identity, up = 2x
    identity, down = a permutation: each layer adds R(silu(h) * 2h) permuted.
    Swapped gate/up, a wrong SiLU or a transposed down projection fails it."""
    cfg = tiny_cfg
    rng = np.random.default_rng(22)
    w = S.model_weights(cfg)
    H, F = cfg.hidden, cfg.ffn
    perm = rng.permutation(H)
    eye_g = np.zeros((F, H), np.uint16)
    eye_g[np.arange(H), np.arange(H)] = 0x3F80          # 1.0
    eye_u = np.zeros((F, H), np.uint16)
    eye_u[np.arange(H), np.arange(H)] = 0x4000          # 2.0
    down = np.zeros((H, F), np.uint16)
    down[np.arange(H), perm] = 0x3F80
    for lw in w.layers:
        lw["wo"] = _zero_like(lw["wo"])
        lw["w_gate"], lw["w_up"], lw["w_down"] = eye_g, eye_u, down
    k, v = S.kv_prefill(cfg, n_pos=3)
    tok = np.array([5], np.int32)
    r = O.decode(cfg, w, k, v, tok, 3, 1)

    def rb(a):
        return O.f32_from_bf16(O.bf16_from_f32(np.asarray(a, np.float32))).astype(np.float64)

    x = rb(O.f32_from_bf16(w.embed[tok[0]]))
    for _ in range(cfg.n_layers):
        h = rb(x / np.sqrt(np.mean(x ** 2) + cfg.rms_eps))
        a = rb(h / (1 + np.exp(-h)) * 2 * h)
        x = rb(x + a[perm])
    hf = rb(x / np.sqrt(np.mean(x ** 2) + cfg.rms_eps))
    logits = O.f32_from_bf16(w.embed).reshape(cfg.vocab, H).astype(np.float64) @ hf
    np.testing.assert_allclose(r.logits[0], logits, atol=2e-3)
    assert r.tokens[0] == int(np.argmax(logits))


def test_decoder_writes_kv_at_position_only(tiny_cfg):
    w, k, v, p = _tiny_inputs(tiny_cfg)
    k0, v0 = k.copy(), v.copy()
    O.decode(tiny_cfg, w, k, v, p[:3], 0, 1)
    changed = np.any(k != k0, axis=(0, 1, 3))
    assert set(np.nonzero(changed)[0]) <= {0, 1, 2}
    assert changed[:3].all()


def test_decoder_rejects_capacity_overflow(tiny_cfg):
    w, k, v, p = _tiny_inputs(tiny_cfg)
    with pytest.raises(ValueError):
        O.decode(tiny_cfg, w, k, v, p, tiny_cfg.max_pos - 2, 8)


def test_alternative_sum_order_build_is_the_same_function():
    """The noise-floor build differs only in rounding: exact on small integers,
    close on a small model (its rounding flips stay far inside the tolerance)."""
    rng = np.random.default_rng(31)
    Wi = rng.integers(-4, 5, size=(9, 1000))
    xi = rng.integers(-4, 5, size=1000)
    W = O.bf16_from_f32(Wi.astype(np.float32)).reshape(9, 1000)
    import ctypes
    y = np.empty(9, np.float32)
    xf = xi.astype(np.float32)
    O.lib("alt").orc_gemv(W.ctypes.data, 9, 1000, xf.ctypes.data, y.ctypes.data)
    assert np.array_equal(y.astype(np.int64), Wi @ xi)
    cfg = S.CONFIGS["tiny"]
    w, (k, v), p = S.model_weights(cfg), S.kv_prefill(cfg), S.prompt(cfg)
    a = O.decode(cfg, w, k.copy(), v.copy(), p, 0, 4)
    b = O.decode(cfg, w, k.copy(), v.copy(), p, 0, 4, variant="alt")
    assert np.abs(a.logits - b.logits).max() < 1e-2      # well inside 3e-2 at two layers
    del ctypes


# ----------------------------------------------------------------- INT8 weights
def _bf16_exact(vals):
    """float values that are exact in BF16 (checked), as BF16 bit patterns"""
    b = O.bf16_from_f32(np.asarray(vals, np.float32))
    assert np.array_equal(O.f32_from_bf16(b).ravel(), np.asarray(vals, np.float32).ravel())
    return b.reshape(np.shape(vals))


def test_quantize_power_of_two_scale_gives_exact_codes():
    """Row absmax 127/128 makes the scale exactly 2^-7, so every code is the
    value times 128. A divisor of 128 instead of 127, a dropped sign or a
    per-matrix instead of per-row scale fails it."""
    W = _bf16_exact(np.array([[127, -127, 64, 1, 0], [0, 0, 127, -2, 3]], np.float32) / 128)
    Q, s = O.quantize_rows(W)
    assert np.array_equal(Q, [[127, -127, 64, 1, 0], [0, 0, 127, -2, 3]])
    assert np.array_equal(s, np.array([2.0 ** -7, 2.0 ** -7], np.float32))


def test_quantize_ties_round_to_even():
    """Codes 2.5 and -2.5 go to 2 and -2, 3.5 to 4: round half to even (half
    away from zero would give 3, -3, 4)."""
    W = _bf16_exact(np.array([[127, 2.5, -2.5, 3.5]], np.float32) / 128)
    Q, _ = O.quantize_rows(W)
    assert np.array_equal(Q, [[127, 2, -2, 4]])


def test_quantize_zero_row_and_gemv_of_it():
    W = np.zeros((2, 8), np.uint16)
    W[1, 3] = 0x3F80                                   # 1.0
    Q, s = O.quantize_rows(W)
    assert s[0] == 0 and not Q[0].any()
    assert Q[1, 3] == 127 and s[1] == np.float32(1.0) / np.float32(127.0)
    y = O.gemv_q8(Q, s, np.arange(8, dtype=np.float32))
    assert y[0] == 0.0


def test_quantize_error_within_half_a_step_and_absmax_maps_to_127():
    """On a random matrix: |w - q s| <= s/2 plus the FP32 rounding of w / s
    (half an ulp of a quotient below 128: 128 * 2^-24 steps), and every row's
    largest magnitude gets code +-127. A wrong scale or rounding rule misses
    by a whole step."""
    rng = np.random.default_rng(31)
    W = O.bf16_from_f32(rng.normal(0, 0.02, (64, 257)).astype(np.float32)).reshape(64, 257)
    Q, s = O.quantize_rows(W)
    w = O.f32_from_bf16(W).reshape(64, 257).astype(np.float64)
    err = np.abs(w - Q.astype(np.float64) * s[:, None].astype(np.float64))
    assert (err <= s[:, None].astype(np.float64) * (0.5 + 128 * 2.0 ** -24)).all()
    assert (np.abs(Q).max(axis=1) == 127).all()
    assert (np.abs(Q[np.arange(64), np.abs(w).argmax(axis=1)]) == 127).all()


def test_gemv_q8_matches_fp64_of_codes_times_scale():
    """y = scale * (codes . x): against FP64 on a non-square matrix (a
    transposed operand or a scale from the wrong row fails)."""
    rng = np.random.default_rng(32)
    W = O.bf16_from_f32(rng.normal(0, 0.02, (37, 300)).astype(np.float32)).reshape(37, 300)
    Q, s = O.quantize_rows(W)
    x = O.f32_from_bf16(O.bf16_from_f32(rng.normal(0, 1, 300).astype(np.float32)))
    y = O.gemv_q8(Q, s, x)
    ref = s.astype(np.float64) * (Q.astype(np.float64) @ x.astype(np.float64))
    bound = 300 * 2.0 ** -23 * s.astype(np.float64) * (np.abs(Q).astype(np.float64) @ np.abs(x))
    assert (np.abs(y - ref) <= bound + 1e-12).all()


def test_decoder_int8_equals_bf16_when_weights_lie_on_the_int8_grid(tiny_cfg):
    """Every weight row (and the tied embedding) is q * 2^-12 with integer
    |q| <= 127 and one entry at +-127: quantizing gives back q with scale
    exactly 2^-12, and scaling by a power of two commutes with rounding, so
    the INT8 decode must equal the BF16 decode bit for bit. A mis-wired code
    matrix or scale anywhere in the decoder fails it."""
    cfg = tiny_cfg
    rng = np.random.default_rng(33)
    w = S.model_weights(cfg)

    def grid(shape):
        q = rng.integers(-127, 128, size=shape).astype(np.float32)
        q[:, 0] = np.where(rng.random(shape[0]) < 0.5, 127, -127)   # absmax 127 in every row
        return _bf16_exact(q * np.float32(2.0 ** -12))

    for lw in w.layers:
        for slot in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
            lw[slot] = grid(lw[slot].shape)
    w.embed = grid(w.embed.shape)
    qw = O.quantize_model(w)
    assert all((sc == np.float32(2.0 ** -12)).all() for ql in qw.layers for _, sc in ql.values())
    k, v = S.kv_prefill(cfg, n_pos=0)
    p = S.prompt(cfg)[:6]
    a = O.decode(cfg, w, k.copy(), v.copy(), p, 0, 5)
    b = O.decode(cfg, w, k.copy(), v.copy(), p, 0, 5, qweights=qw)
    assert np.array_equal(a.tokens, b.tokens)
    assert np.array_equal(a.logits.view(np.uint32), b.logits.view(np.uint32))


# ------------------------------------------------------------------ INT8 KV cache
def test_kv8_row_quantizer_scale_ties_and_zero_row():
    """A row with absmax 127/128 has scale exactly 2^-7: codes are value * 128,
    ties to even (2.5 -> 2, -2.5 -> -2, 3.5 -> 4); an all-zero row gets scale 0."""
    c, s = O.kv8_quantize_row(np.array([127, -127, 2.5, -2.5, 3.5, 0, 64], np.float32) / 128)
    assert s == np.float32(2.0 ** -7)
    assert np.array_equal(c, [127, -127, 2, -2, 4, 0, 64])
    c, s = O.kv8_quantize_row(np.zeros(8, np.float32))
    assert s == 0 and not c.any()


def test_kv8_key_mean_closed_form():
    K = _bf16_exact(np.array([[1, 2, -8], [3, 6, 0], [5, 10, 2]], np.float32))
    assert np.array_equal(O.kv8_key_mean(K), np.array([3, 6, -2], np.float32))
    assert not O.kv8_key_mean(K[:0]).any()                 # no prefill: no shift


def test_kv8_attention_matches_fp64_of_codes_times_scales():
    """Scores from ks_t Kq_t, weights from vs_t Vq_t, softmax in FP64 on the
    same dequantized rows (a swapped K/V scale, a transposed code matrix or a
    missing 1/sqrt(d) fails)."""
    rng = np.random.default_rng(41)
    n, d = 300, 64
    Kq = rng.integers(-127, 128, (n, d)).astype(np.int8)
    Vq = rng.integers(-127, 128, (n, d)).astype(np.int8)
    Ks = rng.uniform(0.005, 0.05, n).astype(np.float32)
    Vs = rng.uniform(0.005, 0.05, n).astype(np.float32)
    q = rng.normal(0, 1, d).astype(np.float32)
    out = O.attention_kv8(q, Kq, Ks, Vq, Vs, 1 / np.sqrt(d))
    K = Ks[:, None].astype(np.float64) * Kq
    V = Vs[:, None].astype(np.float64) * Vq
    sc = K @ q.astype(np.float64) / np.sqrt(d)
    p = np.exp(sc - sc.max())
    ref = (p / p.sum()) @ V
    assert np.allclose(out, ref, rtol=1e-4, atol=1e-5 * np.abs(ref).max())


def test_kv8_smoothing_removes_the_channel_offset_from_the_codes(tiny_cfg):
    """Keys = a per-channel offset mu + deviations on the grid s * code with
    zero mean per channel. The prefill conversion finds mu,
    quantizes only the deviations (exactly), and since a softmax ignores the
    q . mu added to every score, INT8 attention equals FP64 attention over the
    original keys. Quantizing the keys without the shift loses the deviations
    under a scale set by the offset, and fails by orders of magnitude."""
    cfg = tiny_cfg.with_workload(max_pos=64)
    rng = np.random.default_rng(42)
    n, d = 32, cfg.head_dim
    # offsets: integers in [-16, 16]; deviations: k / 4 with |k| <= 127 and
    # |k| = 127 in column 0 of every row (so every scale is exactly 1/4); keys
    # below 64 in magnitude on a 1/4 grid are exact in BF16
    mu = rng.integers(-16, 17, d).astype(np.float32)
    kdev = rng.integers(-127, 128, (n // 2, d)).astype(np.float32)
    kdev[:, 0] = 127
    dev = np.concatenate([kdev, -kdev]) * np.float32(0.25)               # zero mean per channel
    keys = _bf16_exact(mu[None, :] + dev)
    shape = (cfg.n_layers, cfg.n_kv_heads, cfg.max_pos, d)
    k = np.zeros(shape, np.uint16)
    v = np.zeros(shape, np.uint16)
    k[0, 0, :n] = keys
    vq = rng.integers(-127, 128, (n, d)).astype(np.float32)
    vq[:, 1] = 127                                        # every V scale exactly 2^-7 too
    v[0, 0, :n] = _bf16_exact(vq * np.float32(2.0 ** -7))
    kv = O.kv8_from_bf16(cfg, k, v, n)
    assert np.array_equal(kv.mu[0, 0], mu)
    deq = kv.ks[0, 0, :n, None].astype(np.float64) * kv.kq[0, 0, :n]
    assert np.array_equal(deq, dev.astype(np.float64))                   # deviations exact
    q = rng.normal(0, 0.05, d).astype(np.float32)      # scores of order 1: FP32 error ~1e-7
    out = O.attention_kv8(q, kv.kq[0, 0, :n], kv.ks[0, 0, :n], kv.vq[0, 0, :n], kv.vs[0, 0, :n],
                          1 / np.sqrt(d))
    K = O.f32_from_bf16(keys).reshape(n, d).astype(np.float64)
    V = O.f32_from_bf16(v[0, 0, :n]).reshape(n, d).astype(np.float64)
    sc = K @ q.astype(np.float64) / np.sqrt(d)
    p = np.exp(sc - sc.max())
    ref = (p / p.sum()) @ V
    err = np.abs(out - ref).max()
    assert err < 1e-5
    # without the shift: codes of the raw keys
    raw = [O.kv8_quantize_row(O.f32_from_bf16(r)) for r in keys]
    Kq0 = np.stack([c for c, _ in raw]); Ks0 = np.array([s for _, s in raw], np.float32)
    out0 = O.attention_kv8(q, Kq0, Ks0, kv.vq[0, 0, :n], kv.vs[0, 0, :n], 1 / np.sqrt(d))
    assert np.abs(out0 - ref).max() > 100 * max(err, 1e-7)


def test_kv8_decode_writes_each_new_row_with_the_prefill_shift(tiny_cfg):
    """Decoding with the INT8 cache: every row written during the run is the
    INT8 form of (the BF16 row the run cached) - mu, with mu from the prefill;
    the prefill rows are converted the same way; and the logits stay close to
    the BF16-cache decode (INT8 with about 8 bits per entry)."""
    cfg = tiny_cfg.with_workload(max_pos=96)
    w = S.model_weights(cfg)
    n0 = 40
    k, v = S.kv_prefill(cfg, n_pos=n0)
    p = S.prompt(cfg)[:3]
    kb, vb = k.copy(), v.copy()
    ref = O.decode(cfg, w, kb, vb, p, n0, 6)
    k8, v8 = k.copy(), v.copy()
    r8 = O.decode(cfg, w, k8, v8, p, n0, 6, kv_int8=True)
    kv = r8.kv8
    end = n0 + p.size - 1 + 6
    for l in range(cfg.n_layers):
        for h in range(cfg.n_kv_heads):
            mu = kv.mu[l, h]
            assert np.array_equal(mu, O.kv8_key_mean(k[l, h, :n0]))
            for t in (0, n0 - 1, n0, end - 1):
                c, s = O.kv8_quantize_row(O.f32_from_bf16(k8[l, h, t]) - mu)
                assert np.array_equal(kv.kq[l, h, t], c) and kv.ks[l, h, t] == s
                c, s = O.kv8_quantize_row(O.f32_from_bf16(v8[l, h, t]))
                assert np.array_equal(kv.vq[l, h, t], c) and kv.vs[l, h, t] == s
    assert not kv.kq[:, :, end:].any() and not kv.ks[:, :, end:].any()
    assert np.abs(r8.logits - ref.logits).max() < 0.1 * np.abs(ref.logits).max()
    assert np.abs(r8.logits - ref.logits).max() > 0                       # it is a different cache


# ------------------------------------------------------------------ multi-token verify
@pytest.fixture(scope="module")
def lively_model():
    """The tiny shape with its weights scaled by 8, so greedy decoding does not
    repeat one token (needed to see which draft each model token is compared
    with), and a 20-position prefill."""
    cfg = S.CONFIGS["tiny"]
    w = S.model_weights(cfg)

    def scale(a):
        f = O.f32_from_bf16(a).reshape(a.shape) * np.float32(8)
        return O.bf16_from_f32(f.astype(np.float32)).reshape(a.shape)

    for lw in w.layers:
        for slot in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
            lw[slot] = scale(lw[slot])
    w.embed = scale(w.embed)
    k, v = S.kv_prefill(cfg, n_pos=20)
    greedy = O.decode(cfg, w, k.copy(), v.copy(), np.array([5], np.int32), 20, 24).tokens
    assert len(set(greedy.tolist())) > 16
    return cfg, w, k, v, greedy


def test_verify_accepts_right_drafts_and_stops_at_the_first_wrong_one(lively_model):
    """Drafts equal to greedy's: all k accepted, k + 1 tokens out. A wrong
    draft at index j: j accepted, and the token after them is greedy's. An
    off-by-one comparing a_i with d_i instead of d_{i+1} accepts nothing here."""
    cfg, w, k, v, g = lively_model
    r = O.verify(cfg, w, k.copy(), v.copy(), 5, 20, g[:6])
    assert r.n_accepted == 6 and np.array_equal(r.tokens, g[:7])
    for j in (0, 3):
        d = g[:6].copy()
        d[j] = (d[j] + 1) % cfg.vocab
        r = O.verify(cfg, w, k.copy(), v.copy(), 5, 20, d)
        assert r.n_accepted == j and np.array_equal(r.tokens, g[:j + 1])
        assert np.array_equal(r.argmax[:j + 1], g[:j + 1])


def test_verify_loop_emits_exactly_the_greedy_tokens(lively_model):
    """Speculative greedy decoding is lossless: verify steps over drafts that
    are right for a random number of tokens and then wrong, each step starting
    where the last one's accepted prefix ended (its stale rows overwritten),
    emit greedy decoding's tokens."""
    cfg, w, k, v, g = lively_model
    rng = np.random.default_rng(43)
    kk, vv = k.copy(), v.copy()
    out, pos, last = [], 20, 5
    while len(out) < 20:
        i = len(out)
        good = int(rng.integers(0, 5))
        drafts = list(g[i:i + good]) + [int(rng.integers(0, cfg.vocab)) for _ in range(3)]
        r = O.verify(cfg, w, kk, vv, last, pos, drafts)
        assert r.n_accepted >= min(good, len(g) - i)
        out += r.tokens.tolist()
        pos += r.n_accepted + 1
        last = int(r.tokens[-1])
    assert out[:20] == g[:20].tolist()


# ----------------------------------------------------------------- decoder wiring
# The closed forms below read logits[j] = hf[j] for j < H: the tied embedding's
# rows 0..H-1 are the unit vectors e_j, so the LM head hands back the final
# normed vector itself, and every gain, rotation and softmax weight upstream is
# visible in it. The input token's own row is a seeded N(0, 1) vector.
def _rb(a):
    """FP32 -> BF16 round to nearest even, back as float64 (the R() of the definition)."""
    return O.f32_from_bf16(O.bf16_from_f32(np.asarray(a, np.float32))).astype(np.float64)


def _pow2_gain(n, shift):
    """Gains 2^((i + shift) mod 5 - 2) in {1/4 .. 4}: exact in BF16, and two
    vectors differ in every element unless their shifts agree mod 5."""
    e = (np.arange(n) + shift) % 5 - 2
    return O.bf16_from_f32((2.0 ** e).astype(np.float32))


def _unit_rows_embedding(cfg, tok, rng):
    H = cfg.hidden
    E = np.zeros((cfg.vocab, H), np.uint16)
    E[np.arange(H), np.arange(H)] = 0x3F80                          # e_j, value 1.0
    E[tok] = O.bf16_from_f32(rng.standard_normal(H).astype(np.float32))
    return E


def _rms(x, eps):
    return 1.0 / np.sqrt(np.mean(np.asarray(x, np.float64) ** 2) + eps)


def test_decoder_norm_gains_route_to_their_own_step_attention_path(tiny_cfg):
    """Each layer's attn_norm gain scales h, which reaches the residual through
    v = Wv h (uniform attention: all keys zero), Wo a permutation; the FFN is
    zero; the final gain scales hf. With distinct power-of-two gains per layer
    and per norm, a dropped gain, attn_norm and ffn_norm swapped, one layer's
    gain used for another, or the final gain dropped fails it."""
    cfg = replace(tiny_cfg, n_layers=2)
    rng = np.random.default_rng(31)
    H, d, nkv, G = cfg.hidden, cfg.head_dim, cfg.n_kv_heads, cfg.n_q_heads // cfg.n_kv_heads
    tok = H + 7
    w = S.model_weights(cfg)
    w.embed = _unit_rows_embedding(cfg, tok, rng)
    w.final_norm = _pow2_gain(H, 3)
    sel = rng.permutation(H)[: nkv * d]                            # v_g[j] = h[sel[g d + j]]
    perm = rng.permutation(H)                                      # (Wo o)_j = o[perm[j]]
    for l, lw in enumerate(w.layers):
        lw["attn_norm"] = _pow2_gain(H, l)
        lw["ffn_norm"] = _pow2_gain(H, l + 1)
        lw["wq"] = np.zeros_like(lw["wq"])
        lw["wk"] = np.zeros_like(lw["wk"])
        wv = np.zeros_like(lw["wv"])
        wv[np.arange(nkv * d), sel] = 0x3F80
        lw["wv"] = wv
        wo = np.zeros_like(lw["wo"])
        wo[np.arange(H), perm] = 0x3F80
        lw["wo"] = wo
        for m in ("w_gate", "w_up", "w_down"):
            lw[m] = np.zeros_like(lw[m])
    P = 4
    k = np.zeros((cfg.n_layers, nkv, cfg.max_pos, d), np.uint16)
    v = np.zeros_like(k)
    r = O.decode(cfg, w, k, v, np.array([tok], np.int32), P, 1)
    # closed form: uniform softmax over P + 1 positions, cached values zero
    p = np.float32(1.0) / np.float32(P + 1)
    x = O.f32_from_bf16(w.embed[tok]).astype(np.float64)
    for l in range(cfg.n_layers):
        g = O.f32_from_bf16(_pow2_gain(H, l)).astype(np.float64)
        h = _rb(x * _rms(x, cfg.rms_eps) * g)
        vg = h[sel].reshape(nkv, d)
        o = np.concatenate([_rb(np.float32(p) * vg[i // G].astype(np.float32)) for i in range(cfg.n_q_heads)])
        x = _rb(x + o[perm])
    gF = O.f32_from_bf16(_pow2_gain(H, 3)).astype(np.float64)
    hf = _rb(x * _rms(x, cfg.rms_eps) * gF)
    np.testing.assert_allclose(r.logits[0][:H], hf, rtol=2.0 ** -6, atol=1e-6)


def test_decoder_norm_gains_route_to_their_own_step_ffn_path(tiny_cfg):
    """Attention output zero; gate rows 0..H-1 the identity, up 2x the
    identity, down a permutation: each layer adds R(silu(h2) * 2 h2) permuted,
    h2 = R(rmsnorm(x) * g_ffn[l]). Distinct power-of-two gains catch a dropped
    ffn_norm, ffn_norm and attn_norm swapped, or a wrong layer's gain."""
    cfg = replace(tiny_cfg, n_layers=2)
    rng = np.random.default_rng(32)
    H, F = cfg.hidden, cfg.ffn
    tok = H + 3
    w = S.model_weights(cfg)
    w.embed = _unit_rows_embedding(cfg, tok, rng)
    w.final_norm = _pow2_gain(H, 4)
    perm = rng.permutation(H)
    eye_g = np.zeros((F, H), np.uint16)
    eye_g[np.arange(H), np.arange(H)] = 0x3F80
    eye_u = np.zeros((F, H), np.uint16)
    eye_u[np.arange(H), np.arange(H)] = 0x4000                    # 2.0
    down = np.zeros((H, F), np.uint16)
    down[np.arange(H), perm] = 0x3F80
    for l, lw in enumerate(w.layers):
        lw["attn_norm"] = _pow2_gain(H, l + 2)
        lw["ffn_norm"] = _pow2_gain(H, l)
        lw["wo"] = np.zeros_like(lw["wo"])
        lw["w_gate"], lw["w_up"], lw["w_down"] = eye_g, eye_u, down
    k, v = S.kv_prefill(cfg, n_pos=3)
    r = O.decode(cfg, w, k, v, np.array([tok], np.int32), 3, 1)
    x = O.f32_from_bf16(w.embed[tok]).astype(np.float64)
    for l in range(cfg.n_layers):
        g = O.f32_from_bf16(_pow2_gain(H, l)).astype(np.float64)
        h = _rb(x * _rms(x, cfg.rms_eps) * g)
        a = _rb(h / (1 + np.exp(-h)) * 2 * h)
        x = _rb(x + a[perm])
    gF = O.f32_from_bf16(_pow2_gain(H, 4)).astype(np.float64)
    hf = _rb(x * _rms(x, cfg.rms_eps) * gF)
    np.testing.assert_allclose(r.logits[0][:H], hf, rtol=2.0 ** -6, atol=1e-6)


def test_decoder_qk_norm_before_rope_and_both_rotated_at_the_position(tiny_cfg):
    """q/k RMSNorm with distinct per-dimension gains, then RoPE at P, for q and
    k alike. One hidden unit feeds dimension a of every q head and of KV head
    0's k, and dimension a + d/2 of KV head 1's k; the cached keys (already
    rotated) have components on a and a + d/2; cached values are unit vectors,
    so the output of each q head is its softmax weights. Closed form per score:
      q' = Q (cos t_a e_a + sin t_a e_{a+d/2}),   Q  = h_m / rms * g_q[a]
      k0' = K0 (cos t_a e_a + sin t_a e_{a+d/2}), K0 = h_m / rms * g_k[a]
      k1' = K1 (-sin t_a e_a + cos t_a e_{a+d/2}), K1 = h_m / rms * g_k[a + d/2]
    (t_a = P w_a), so the new key's score is Q K0 / sqrt(d) for KV head 0 and
    exactly 0 for KV head 1. Fails if the norm runs after RoPE (then g_q[a+d/2]
    enters), if q_norm and k_norm are swapped, if k is rotated at another
    position than q or not at all, or if q is rotated at another position."""
    cfg = replace(tiny_cfg, n_layers=1, qk_norm=True, rms_eps=1e-6)
    rng = np.random.default_rng(33)
    H, d, nkv, G, nq = cfg.hidden, cfg.head_dim, cfg.n_kv_heads, cfg.n_q_heads // cfg.n_kv_heads, cfg.n_q_heads
    half = d // 2
    tok, a, P = H + 11, 5, 6
    w = S.model_weights(cfg)
    w.embed = _unit_rows_embedding(cfg, tok, rng)
    x0 = O.f32_from_bf16(w.embed[tok]).astype(np.float64)
    h = _rb(x0 * _rms(x0, cfg.rms_eps))                            # attn_norm gain 1
    m = int(np.argmax(np.abs(h)))
    lw = w.layers[0]
    gq = np.full(d, 0x3F80, np.uint16)
    gk = np.full(d, 0x3F80, np.uint16)
    gq[a], gq[a + half] = O.bf16_from_f32(np.float32(0.5))[0], O.bf16_from_f32(np.float32(2.0))[0]
    gk[a], gk[a + half] = O.bf16_from_f32(np.float32(0.25))[0], O.bf16_from_f32(np.float32(1.0))[0]
    gk[0] = O.bf16_from_f32(np.float32(4.0))[0]                     # keeps g_k != g_q elementwise
    lw["q_norm"], lw["k_norm"] = gq, gk
    wq = np.zeros_like(lw["wq"])
    wq[np.arange(nq) * d + a, m] = 0x3F80
    wk = np.zeros_like(lw["wk"])
    wk[0 * d + a, m] = 0x3F80
    wk[1 * d + a + half, m] = 0x3F80
    lw["wq"], lw["wk"], lw["wv"] = wq, wk, np.zeros_like(lw["wv"])
    lw["wo"] = np.eye(H, nq * d, dtype=np.uint16) * np.uint16(0x3F80)
    for mm in ("w_gate", "w_up", "w_down"):
        lw[mm] = np.zeros_like(lw[mm])
    k = np.zeros((1, nkv, cfg.max_pos, d), np.uint16)
    v = np.zeros_like(k)
    alpha = O.bf16_from_f32((0.5 * np.cos(np.arange(P) * 1.3)).astype(np.float32))
    beta = O.bf16_from_f32((0.5 * np.sin(np.arange(P) * 0.7 + 0.3)).astype(np.float32))
    for g in range(nkv):
        k[0, g, :P, a] = alpha
        k[0, g, :P, a + half] = beta
        v[0, g, np.arange(P), np.arange(P)] = 0x3F80                 # V_t = e_t
    r = O.decode(cfg, w, k, v, np.array([tok], np.int32), P, 1)

    # closed form
    rms1 = 1.0 / np.sqrt(h[m] ** 2 / d + cfg.rms_eps)               # RMSNorm of h_m e_a over d
    f = lambda b: float(O.f32_from_bf16(b)[0])
    Q = h[m] * rms1 * f(gq[a])
    K0 = h[m] * rms1 * f(gk[a])
    K1 = h[m] * rms1 * f(gk[a + half])
    om = cfg.rope_theta ** (-2.0 * a / d)
    c, s = float(np.float32(np.cos(P * om))), float(np.float32(np.sin(P * om)))
    q_a, q_b = _rb(Q * c), _rb(Q * s)
    k_new = {0: (_rb(K0 * c), _rb(K0 * s)), 1: (_rb(-K1 * s), _rb(K1 * c))}
    al, be = O.f32_from_bf16(alpha).astype(np.float64), O.f32_from_bf16(beta).astype(np.float64)
    scale = 1.0 / np.sqrt(d)
    o = np.zeros(nq * d)
    for i in range(nq):
        g = i // G
        sc = np.append((q_a * al + q_b * be) * scale, (q_a * k_new[g][0] + q_b * k_new[g][1]) * scale)
        pr = np.exp(sc - sc.max())
        pr /= pr.sum()
        o[i * d: i * d + P] = pr[:P]                                 # V_P = 0
    assert abs(q_a * k_new[1][0] + q_b * k_new[1][1]) < 1e-2 * abs(Q * K1)
    x1 = _rb(x0 + _rb(o))
    hf = _rb(x1 * _rms(x1, cfg.rms_eps))
    np.testing.assert_allclose(r.logits[0][:H], hf, rtol=2.0 ** -6, atol=1e-6)
    # the new rows of the cache are the rotated, normed k (and v = 0)
    for g in range(nkv):
        np.testing.assert_allclose(O.f32_from_bf16(k[0, g, P, [a, a + half]]), np.ravel(k_new[g]), rtol=1e-6)
