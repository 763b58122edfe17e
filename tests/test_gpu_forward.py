"""The multi-token pass (tiles_forward) and the verify step (tiles_verify)
against the CPU oracle, through the C ABI.

A pass of n tokens computes what n decode steps with those inputs compute, so
the oracle reference is its prompt path over the same inputs: every position's
logits within 3e-2 + 1e-2 |oracle|, the greedy choices identical except at
near-ties, the KV cache it writes close to the oracle's. The verify step is
held to oracle.verify (greedy acceptance) and, in a loop, to greedy decoding.
Norm gains are seeded non-unit.
"""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import synthetic as S
from gpu_helpers import GAINS, check_forward, inputs, with_gains

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tile_scheduled_persistent_gb300 as t
    t.build()
    return t


def _plan(tsp, cfg, w, **opts):
    return tsp.Plan(tsp.ModelDesc.from_config(cfg), tsp.upload_weights(w), tsp.make_opts(**opts))


def _forward(tsp, plan, cfg, k, v, tokens, start_pos, want_logits=True):
    import torch
    kc, vc = tsp.to_device_bf16(k), tsp.to_device_bf16(v)
    n = len(tokens)
    toks = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).cuda()
    am = torch.full((n,), -1, dtype=torch.int32, device="cuda")
    lg = torch.full((n, cfg.vocab), float("nan"), dtype=torch.float32, device="cuda") if want_logits else None
    plan.forward(kc, vc, toks, start_pos, am, lg)
    plan.check()
    torch.cuda.synchronize()
    return (am.cpu().numpy(), None if lg is None else lg.cpu().numpy(),
            kc.view(torch.int16).cpu().numpy().view(np.uint16), vc.view(torch.int16).cpu().numpy().view(np.uint16))


def _cache_close(got, want, end):
    np.testing.assert_allclose(S.bf16_to_f32(got[:, :, :end]).astype(np.float64),
                               S.bf16_to_f32(want[:, :, :end]).astype(np.float64), atol=3e-2, rtol=3e-2)


def test_prefill_tiny_prompt_matches_oracle(tsp):
    cfg = with_gains(S.CONFIGS["tiny"])
    w, k, v, prompt = inputs(cfg, n_pos=0)
    plan = _plan(tsp, cfg, w)
    am, lg, kc, vc = _forward(tsp, plan, cfg, k, v, prompt, 0)
    plan.close()
    _, rk, rv = check_forward(am, lg, cfg, w, k, v, prompt, 0, "tiny prefill")
    _cache_close(kc, rk, prompt.size)
    _cache_close(vc, rv, prompt.size)
    assert not kc[:, :, prompt.size:].any()                        # nothing written past the pass


SHAPES = {
    # head_dim 128, GQA group 8, q/k norm
    "d128_g8_qknorm": replace(S.CONFIGS["tiny"], name="f1", head_dim=128, n_q_heads=8, n_kv_heads=1,
                              qk_norm=True, rope_theta=1e6, rms_eps=1e-6, gain_sigma=GAINS),
    # no GQA sharing, llama3 RoPE, ragged widths
    "g1_llama3": replace(S.CONFIGS["tiny"], name="f2", n_q_heads=2, n_kv_heads=2, hidden=264, ffn=776,
                         vocab=1000, rope_scaling=True, rope_theta=5e5, gain_sigma=GAINS),
    # a prefilled cache crossing several 64-position blocks
    "g2_cache": replace(S.CONFIGS["tiny"], name="f3", start_pos=150, n_prompt=24, max_pos=200,
                        gain_sigma=GAINS),
    # long context with NaN past the written rows: nothing past a token's own position is read
    "d128_g2_long": replace(S.CONFIGS["tiny"], name="f4", head_dim=128, n_q_heads=4, n_kv_heads=2,
                            qk_norm=True, rope_theta=1e6, rms_eps=1e-6, start_pos=1000, n_prompt=17,
                            max_pos=1100, gain_sigma=GAINS),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_forward_shapes_match_oracle(tsp, name):
    cfg = SHAPES[name]
    w, k, v, _ = inputs(cfg)
    toks = S.tokens(S.SEED_TOKENS, 7, cfg.n_prompt, cfg.vocab)
    if name == "d128_g2_long":
        k[:, :, cfg.start_pos:, :] = 0x7FC0
        v[:, :, cfg.start_pos:, :] = 0x7FC0
    plan = _plan(tsp, cfg, w)
    am, lg, kc, vc = _forward(tsp, plan, cfg, k, v, toks, cfg.start_pos)
    plan.close()
    _, rk, rv = check_forward(am, lg, cfg, w, k, v, toks, cfg.start_pos, name)
    end = cfg.start_pos + toks.size
    _cache_close(kc, rk, end)
    if name == "d128_g2_long":
        assert (kc[:, :, end:] == 0x7FC0).all() and (vc[:, :, end:] == 0x7FC0).all()


def test_forward_of_more_than_one_pass_and_decode_continuation(tsp):
    """300 inputs run as two passes (256 + 44); then the decode kernel
    continues from the cache the passes wrote: its tokens and logits match
    the oracle's continuous run, and the pass's logits the oracle's prompt
    path."""
    import torch
    cfg = with_gains(S.CONFIGS["tiny"]).with_workload(max_pos=320)
    w, k, v, _ = inputs(cfg, n_pos=0)
    toks = S.tokens(S.SEED_TOKENS, 9, 300, cfg.vocab)
    plan = _plan(tsp, cfg, w)
    am, lg, kc, vc = _forward(tsp, plan, cfg, k, v, toks, 0)
    ref, rk, rv = check_forward(am, lg, cfg, w, k, v, toks, 0, "two passes")
    # decode 12 tokens after the prompt from the GPU-written cache
    kd, vd = tsp.to_device_bf16(kc), tsp.to_device_bf16(vc)
    out = torch.zeros(12, dtype=torch.int32, device="cuda")
    lgd = torch.zeros((12, cfg.vocab), dtype=torch.float32, device="cuda")
    plan.decode(kd, vd, torch.tensor([int(toks[-1])], dtype=torch.int32, device="cuda"), 299, 12, out, lgd)
    plan.check()
    plan.close()
    cont = oracle.decode(cfg, w, rk.copy(), rv.copy(), np.array([toks[-1]], np.int32), 299, 12)
    # the decode continues from the GPU's own cache; its first step is step 299 of the pass
    np.testing.assert_allclose(lgd.cpu().numpy()[0], lg[299], atol=3e-2, rtol=1e-2)
    err = np.abs(lgd.cpu().numpy() - cont.logits)
    assert (err <= 3e-2 + 1e-2 * np.abs(cont.logits)).all(), float(err.max())


def _verify(tsp, plan, cfg, k, v, inputs_, start_pos):
    import torch
    kc, vc = tsp.to_device_bf16(k), tsp.to_device_bf16(v)
    inp = torch.from_numpy(np.ascontiguousarray(inputs_, np.int32)).cuda()
    out = torch.full((len(inputs_),), -1, dtype=torch.int32, device="cuda")
    n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    lg = torch.zeros((len(inputs_), cfg.vocab), dtype=torch.float32, device="cuda")
    plan.verify(kc, vc, inp, start_pos, out, n, lg)
    plan.check()
    torch.cuda.synchronize()
    na = int(n.item())
    return na, out.cpu().numpy()[:na + 1], lg.cpu().numpy(), kc, vc


@pytest.fixture(scope="module")
def lively(tsp):
    """The tiny shape with weights x 3 (greedy decoding then does not repeat
    one token, so each draft is checked against a distinct model token),
    non-unit gains and a 20-position prefill; with the oracle's greedy run and
    tau, the reordered oracle's largest logit deviation per step."""
    cfg = with_gains(S.CONFIGS["tiny"])
    w = S.model_weights(cfg)

    def scale(a):
        return oracle.bf16_from_f32(oracle.f32_from_bf16(a).reshape(a.shape) * np.float32(3)).reshape(a.shape)

    for lw in w.layers:
        for slot in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
            lw[slot] = scale(lw[slot])
    w.embed = scale(w.embed)
    k, v = S.kv_prefill(cfg, n_pos=20)
    greedy = oracle.decode(cfg, w, k.copy(), v.copy(), np.array([5], np.int32), 20, 24)
    assert len(set(greedy.tokens.tolist())) > 16
    return cfg, w, k, v, greedy


def _near_tie(logits_row, tau):
    from gpu_helpers import near_tie_scale
    srt = np.sort(logits_row)
    return srt[-1] - srt[-2] < near_tie_scale(logits_row, tau, False)


@pytest.mark.parametrize("case", ["all_right", "wrong_at_0", "wrong_at_5", "k16"])
def test_verify_matches_oracle_verify(tsp, lively, case):
    """Logits of every input within 3e-2 + 1e-2 |oracle| + 1.5 tau; the accepted
    count and the emitted tokens the oracle's (a difference only where the
    oracle's choice was a near-tie)."""
    cfg, w, k, v, greedy = lively
    g = greedy.tokens
    kd = 16 if case == "k16" else 8
    drafts = g[:kd].copy()
    if case.startswith("wrong_at_"):
        j = int(case.split("_")[-1])
        drafts[j] = (drafts[j] + 1) % cfg.vocab
    inputs_ = np.concatenate([[5], drafts]).astype(np.int32)
    plan = _plan(tsp, cfg, w)
    na, toks, lg, *_ = _verify(tsp, plan, cfg, k, v, inputs_, 20)
    plan.close()
    ref = oracle.verify(cfg, w, k.copy(), v.copy(), 5, 20, drafts)
    alt = oracle.decode(cfg, w, k.copy(), v.copy(), inputs_, 20, 1, variant="alt")
    tau = np.abs(alt.logits - ref.logits).max(axis=1)
    err = np.abs(lg - ref.logits)
    assert (err <= 3e-2 + 1e-2 * np.abs(ref.logits) + 1.5 * tau[:, None]).all(), float(err.max())
    gpu_choice = lg.argmax(axis=1)
    first = next((i for i in range(kd + 1) if gpu_choice[i] != ref.argmax[i]), None)
    if first is not None and first <= ref.n_accepted:
        assert _near_tie(ref.logits[first], tau[first]), f"choice {first} differs away from a near-tie"
        return
    assert na == ref.n_accepted and np.array_equal(toks, ref.tokens), (na, toks, ref.n_accepted, ref.tokens)


def test_verify_loop_emits_the_greedy_tokens(tsp, lively):
    """Verify steps over drafts right for a random number of tokens and then
    wrong, each starting where the previous one's accepted prefix ended: the
    emitted stream is greedy decoding's (up to the first near-tie of the
    oracle's greedy run, where another valid FP32 order may choose the other
    token)."""
    import torch
    cfg, w, k, v, greedy = lively
    g = greedy.tokens
    rng = np.random.default_rng(61)
    plan = _plan(tsp, cfg, w)
    kc, vc = tsp.to_device_bf16(k), tsp.to_device_bf16(v)
    out_all, pos, last = [], 20, 5
    while len(out_all) < 20:
        i = len(out_all)
        good = int(rng.integers(0, 6))
        drafts = list(g[i:i + good]) + [int(rng.integers(0, cfg.vocab)) for _ in range(3)]
        inp = torch.tensor([last] + drafts, dtype=torch.int32, device="cuda")
        out = torch.full((len(drafts) + 1,), -1, dtype=torch.int32, device="cuda")
        n = torch.zeros(1, dtype=torch.int32, device="cuda")
        plan.verify(kc, vc, inp, pos, out, n)
        plan.check()
        na = int(n.item())
        emitted = out.cpu().numpy()[:na + 1].tolist()
        out_all += emitted
        pos += na + 1
        last = emitted[-1]
    plan.close()
    d = next((i for i in range(20) if out_all[i] != g[i]), 20)
    assert d >= 1
    if d < 20:
        alt = oracle.decode(cfg, w, k.copy(), v.copy(), np.array([5], np.int32), 20, 24, variant="alt",
                            force_tokens=g[:-1])
        tau = np.abs(alt.logits - greedy.logits).max(axis=1)
        assert _near_tie(greedy.logits[d], tau[d]), f"stream differs at {d} away from a near-tie"
    print({"verify loop agrees with greedy for": d})


@pytest.mark.parametrize("name,n", [("llama1b", 64), ("qwen3_0_6b", 40), ("llama1b", 512), ("llama1b", 17),
                                    ("qwen3_4b", 17)],
                         ids=["llama1b_64", "qwen3_0_6b_40", "llama1b_512", "llama1b_17", "qwen3_4b_17"])
def test_forward_full_width_one_layer_slice(tsp, name, n):
    """Full width (hidden, heads, FFN, vocab) at one layer: a pass of n tokens
    after the workload's cached positions (a 512-token prompt from position 0
    for the third case), every logit within the strict tolerance. 17 tokens
    of the Llama-1B and Qwen3-4B shapes (head_dim 64 and 128, q/k norm in
    the second) take the SwiGLU in the gate/up projection's epilogue (one
    split, a short pass); the others the separate kernel."""
    base = replace(S.CONFIGS[name], n_layers=1, gain_sigma=GAINS)
    cfg = base if n < 512 else base.with_workload(start_pos=0, max_pos=520)
    w, k, v, _ = inputs(cfg)
    toks = S.tokens(S.SEED_TOKENS, 11, n, cfg.vocab)
    plan = _plan(tsp, cfg, w)
    am, lg, *_ = _forward(tsp, plan, cfg, k, v, toks, cfg.start_pos)
    plan.close()
    check_forward(am, lg, cfg, w, k, v, toks, cfg.start_pos, f"{name} one layer, {n} tokens")


def test_forward_rejects_int8_plans_and_overflow(tsp):
    import torch
    cfg = S.CONFIGS["tiny"]
    w, k, v, prompt = inputs(cfg, n_pos=0)
    kc, vc = tsp.to_device_bf16(k), tsp.to_device_bf16(v)
    am = torch.zeros(8, dtype=torch.int32, device="cuda")
    toks = torch.zeros(8, dtype=torch.int32, device="cuda")
    q8 = _plan(tsp, cfg, w, weight_format=tsp.WEIGHTS_INT8)
    with pytest.raises(tsp.TilesError) as e:
        q8.forward(kc, vc, toks, 0, am)
    assert e.value.status == -2
    q8.close()
    plan = _plan(tsp, cfg, w)
    with pytest.raises(tsp.TilesError) as e:
        plan.forward(kc, vc, toks, cfg.max_pos - 4, am)
    assert e.value.status == -5
    plan.close()


@pytest.mark.parametrize("n,start", [(1, 0), (1, 37), (256, 0), (5, 123)], ids=["one_token", "one_token_cached",
                                                                                "exactly_one_pass", "up_to_max_pos"])
def test_forward_edge_lengths_match_oracle(tsp, n, start):
    """A pass of one token (a decode step), of exactly 256 tokens (one full
    pass), and one that ends on the last cache position (start + n =
    max_pos): every logit and greedy choice against the oracle's prompt path,
    the cache written up to the end and nothing past it."""
    max_pos = 260 if n == 256 else 128
    cfg = replace(S.CONFIGS["tiny"], name="edge", max_pos=max_pos, start_pos=start, gain_sigma=GAINS)
    w, k, v, _ = inputs(cfg)
    toks = S.tokens(S.SEED_TOKENS, 11, n, cfg.vocab)
    plan = _plan(tsp, cfg, w)
    am, lg, kc, vc = _forward(tsp, plan, cfg, k, v, toks, start)
    plan.close()
    _, kk, vv = check_forward(am, lg, cfg, w, k, v, toks, start, f"edge n={n} start={start}")
    _cache_close(kc, kk, start + n)
    _cache_close(vc, vv, start + n)
    assert not kc[:, :, start + n:].any() and not vc[:, :, start + n:].any()
