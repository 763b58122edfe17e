"""The shared seeded input generator: definition, determinism, distribution."""
import numpy as np

import synthetic as S


def test_splitmix64_reference_outputs():
    """First outputs of SplitMix64 from state 1234567, the test vector that ships
    with the reference C implementation of the generator (Vigna, splitmix64.c)."""
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(v) for v in S.splitmix64_stream(1234567, 5)] == want


def test_counter_based_elements_are_position_independent():
    whole = S.normal_f32(0, 5, 1000, 1.0)
    part = S.normal_f32(0, 5, 300, 1.0, i0=401)
    assert np.array_equal(whole[401:701], part)
    assert not np.array_equal(S.normal_f32(0, 6, 1000), whole)   # other tensor id
    assert not np.array_equal(S.normal_f32(1, 5, 1000), whole)   # other seed


def test_normal_statistics():
    x = S.normal_f32(3, 9, 1 << 20, 0.02).astype(np.float64)
    assert abs(x.mean()) < 1e-4
    assert abs(x.std() - 0.02) < 1e-4
    assert abs(np.mean(np.abs(x) < 0.02) - 0.6827) < 3e-3       # one-sigma mass


def test_bf16_generation_rounds_the_float_values():
    f = S.normal_f32(0, 11, 4096, 0.02)
    b = S.normal_bf16(0, 11, (4096,), 0.02)
    back = S.bf16_to_f32(b)
    assert np.all(np.abs(back - f) <= np.abs(f) * 2.0 ** -8)


def test_tokens_in_range_and_spread():
    t = S.tokens(2, 0, 20000, 1024)
    assert t.min() >= 0 and t.max() < 1024
    assert len(np.unique(t)) > 1000


def test_kv_prefill_layout_and_tail_zero():
    cfg = S.CONFIGS["tiny"].with_workload(start_pos=10, max_pos=16)
    k, v = S.kv_prefill(cfg, n_pos=10)
    assert k.shape == (2, 2, 16, 64)
    assert not k[:, :, 10:].any() and not v[:, :, 10:].any()
    # element (h, p, j) of layer l is element (h * n_pos + p) * d + j of tensor 2l
    flat = S.normal_bf16(S.SEED_KV, 2 * 1, (2 * 10 * 64,), 1.0).reshape(2, 10, 64)
    assert np.array_equal(k[1, :, :10], flat)


def test_config_byte_counts():
    c = S.CONFIGS["llama1b"]
    assert c.weight_bytes() == 2 * (16 * (3072 * 2048 + 2048 * 2048 + 3 * 8192 * 2048 + 2 * 2048)
                                    + 128256 * 2048 + 2048)
    assert abs(c.algorithmic_bytes_per_token() - 2.5063e9) < 1e6


def test_config_byte_counts_equal_the_arrays_they_count():
    """weight_bytes counts what the arrays hold: every BF16 weight once, or the
    INT8 codes and FP32 row scales of the oracle's quantized model plus the
    BF16 norm weights."""
    import oracle
    for cfg in (S.CONFIGS["tiny"], S.CONFIGS["tiny"].with_workload(qk_norm=True)):
        w = S.model_weights(cfg)
        arrays = [w.embed, w.final_norm] + [a for lw in w.layers for a in lw.values() if a is not None]
        assert cfg.weight_bytes() == sum(a.nbytes for a in arrays)
        qw = oracle.quantize_model(w)
        norms = [lw[n] for lw in w.layers for n in ("attn_norm", "ffn_norm", "q_norm", "k_norm")
                 if lw[n] is not None]
        q_bytes = (sum(c.nbytes + s.nbytes for ql in qw.layers for c, s in ql.values())
                   + qw.lm[0].nbytes + qw.lm[1].nbytes + w.final_norm.nbytes
                   + sum(a.nbytes for a in norms))
        assert cfg.weight_bytes(int8=True) == q_bytes


def test_gains_default_to_one_and_are_seeded_distinct_vectors_when_asked():
    """The workload configs keep every norm gain at 1.0; gain_sigma > 0 gives
    each norm (per layer and slot, and the final one) its own seeded vector."""
    base = S.CONFIGS["tiny"].with_workload(qk_norm=True)
    w = S.model_weights(base)
    for lw in w.layers:
        for slot in ("attn_norm", "ffn_norm", "q_norm", "k_norm"):
            assert (lw[slot] == S.BF16_ONE).all()
    assert (w.final_norm == S.BF16_ONE).all()
    g = S.model_weights(base.with_workload(gain_sigma=0.25))
    vecs = [g.final_norm] + [lw[s] for lw in g.layers
                             for s in ("attn_norm", "ffn_norm", "q_norm", "k_norm")]
    f = [S.bf16_to_f32(v).astype(np.float64) for v in vecs]
    allf = np.concatenate(f)
    assert abs(allf.mean() - 1.0) < 0.02 and abs(allf.std() - 0.25) < 0.02
    for i in range(len(f)):
        for j in range(i + 1, len(f)):
            n = min(len(f[i]), len(f[j]))
            assert not np.array_equal(f[i][:n], f[j][:n])
    # the matrices are the same with or without seeded gains
    assert np.array_equal(g.layers[1]["wq"], w.layers[1]["wq"]) and np.array_equal(g.embed, w.embed)
