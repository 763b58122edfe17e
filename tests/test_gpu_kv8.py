"""GPU parity of the INT8 KV cache with smoothed keys ("History and roadmap",
M8: INT8 KV cache with smoothed keys; "Tried and not kept": queries stay
unquantized) against the oracle's INT8-cache decode, through the C ABI.

The cache built from a BF16 prefill is compared bit for bit (codes, scales
and key shifts); decodes are held to the same bar as the BF16 cache (every
logit within 3e-2 + 1e-2 |oracle| of the oracle run on the GPU's token
history, tokens exact except at near-ties), with seeded non-unit gains.
"""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import synthetic as S
from gpu_helpers import GAINS, check_parity, gpu_run_kv8, inputs

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
    return tsp.Plan(tsp.ModelDesc.from_config(cfg), tsp.upload_weights(w),
                    tsp.make_opts(kv_format=tsp.KV_INT8, **opts))


def _oracle_parts(cfg, kv8):
    """The oracle's INT8 cache in the GPU layout's index order, positions < max_pos."""
    Z, P, d = cfg.n_layers * cfg.n_kv_heads, cfg.max_pos, cfg.head_dim
    return {"kq": kv8.kq.reshape(Z, P, d), "vq": kv8.vq.reshape(Z, P, d).transpose(0, 2, 1),
            "ks": kv8.ks.reshape(Z, P), "vs": kv8.vs.reshape(Z, P), "mu": kv8.mu.reshape(Z, d)}


CONVERT = {
    # max_pos not a multiple of 16: the position stride is padded
    "d64": replace(S.CONFIGS["tiny"], name="k1", start_pos=100, max_pos=130, gain_sigma=GAINS),
    "d128": replace(S.CONFIGS["tiny"], name="k2", head_dim=128, n_q_heads=8, n_kv_heads=1,
                    qk_norm=True, start_pos=490, max_pos=520, gain_sigma=GAINS),
    "empty": replace(S.CONFIGS["tiny"], name="k3", start_pos=0, max_pos=64, gain_sigma=GAINS),
}


@pytest.mark.parametrize("name", list(CONVERT))
def test_cache_from_bf16_prefill_is_the_oracles_bit_for_bit(tsp, name):
    """Key shifts (FP64 channel sums in position order), codes and scales of
    every prefilled row, against oracle.kv8_from_bf16 on the same BF16 caches."""
    cfg = CONVERT[name]
    _, k, v, _ = inputs(cfg)
    n = cfg.start_pos
    cache = tsp.KV8Cache(tsp.ModelDesc.from_config(cfg))
    cache.from_bf16(tsp.to_device_bf16(k), tsp.to_device_bf16(v), n)
    g = cache.host()
    o = _oracle_parts(cfg, oracle.kv8_from_bf16(cfg, k, v, n))
    assert g["kq"].shape[1] % 16 == 0 and g["kq"].shape[1] >= cfg.max_pos
    assert np.array_equal(g["mu"].view(np.uint32), o["mu"].view(np.uint32))
    assert np.array_equal(g["kq"][:, :n], o["kq"][:, :n])
    assert np.array_equal(g["vq"][:, :, :n], o["vq"][:, :, :n])
    assert np.array_equal(g["ks"][:, :n].view(np.uint32), o["ks"][:, :n].view(np.uint32))
    assert np.array_equal(g["vs"][:, :n].view(np.uint32), o["vs"][:, :n].view(np.uint32))
    if n == 0:
        assert not g["mu"].any()
    else:
        assert np.abs(g["kq"][:, :n]).max() == 127 and g["ks"][:, :n].min() > 0


def _check_new_rows(cfg, g, o, p0, p1):
    """Rows the decode wrote (positions p0..p1-1): quantized from the GPU's own
    BF16 key/value rows, which may differ from the oracle's by a rounding now
    and then, so compared dequantized, within one code step (plus the BF16
    rounding), with most codes equal."""
    for q, s, tr in (("kq", "ks", False), ("vq", "vs", True)):
        gc = g[q][:, :, p0:p1].transpose(0, 2, 1) if tr else g[q][:, p0:p1]
        oc = o[q][:, :, p0:p1].transpose(0, 2, 1) if tr else o[q][:, p0:p1]
        gs, os_ = g[s][:, p0:p1, None], o[s][:, p0:p1, None]
        gd, od = gc * gs.astype(np.float64), oc * os_.astype(np.float64)
        tol = 1.01 * np.maximum(gs, os_) + 1e-2 * np.abs(od)
        assert (np.abs(gd - od) <= tol).all(), (q, float(np.abs(gd - od).max()))
        assert np.mean(gc == oc) > 0.9, (q, float(np.mean(gc == oc)))


DECODE = {
    # no prefill: key shifts 0, every row written by the decode
    "d64_scratch": (replace(S.CONFIGS["tiny"], name="d1", start_pos=0, gain_sigma=GAINS), None),
    # prefilled, crossing a 128-position chunk boundary while decoding
    "d64_prefill": (replace(S.CONFIGS["tiny"], name="d2", start_pos=230, n_prompt=2, n_new=40, max_pos=300,
                            gain_sigma=GAINS), None),
    # head_dim 128 (64-position chunks), GQA group 8, q/k norm
    "d128_g8_qknorm": (replace(S.CONFIGS["tiny"], name="d3", head_dim=128, n_q_heads=8, n_kv_heads=1,
                               qk_norm=True, rope_theta=1e6, rms_eps=1e-6, start_pos=490, n_prompt=2,
                               n_new=24, max_pos=520, gain_sigma=GAINS), None),
    # no GQA sharing, llama3 RoPE, padded position stride, two splits of several chunks
    "d64_g1_splits": (replace(S.CONFIGS["tiny"], name="d4", n_q_heads=2, n_kv_heads=2, hidden=264, ffn=776,
                              vocab=1000, rope_scaling=True, rope_theta=5e5, start_pos=1010, n_prompt=2,
                              n_new=12, max_pos=1030, gain_sigma=GAINS), 2),
    # one split of nine chunks: every warp owns chunks, the new row in the last
    "d64_one_split": (replace(S.CONFIGS["tiny"], name="d5", start_pos=1100, n_prompt=2, n_new=8,
                              max_pos=1200, gain_sigma=GAINS), 1),
}


@pytest.mark.parametrize("name", list(DECODE))
def test_decode_with_int8_cache_matches_oracle(tsp, name):
    cfg, splits = DECODE[name]
    w, k, v, prompt = inputs(cfg)
    prompt = prompt[: cfg.n_prompt] if cfg.start_pos else prompt
    n_new = cfg.n_new
    plan = _plan(tsp, cfg, w, **({"kv_splits": splits} if splits else {}))
    info = plan.info()
    assert info["kv_format"] == tsp.KV_INT8 and info["attn_tensor_cores"] == 1
    assert info["kv_block"] == 8192 // cfg.head_dim
    toks, logits, g = gpu_run_kv8(plan, cfg, k, v, prompt, cfg.start_pos, n_new)
    plan.close()
    _, ref, *_ = check_parity(toks, logits, cfg, w, k, v, prompt, cfg.start_pos, n_new, name + " int8 kv",
                              kv_int8=True)
    o = _oracle_parts(cfg, ref.kv8)
    n0 = cfg.start_pos
    n1 = n0 + prompt.size - 1 + n_new
    assert np.array_equal(g["mu"].view(np.uint32), o["mu"].view(np.uint32))
    assert np.array_equal(g["kq"][:, :n0], o["kq"][:, :n0])       # the prefill is untouched
    _check_new_rows(cfg, g, o, n0, n1)


def test_int8_cache_bitwise_across_schedulers_and_runs(tsp):
    cfg, _ = DECODE["d64_prefill"]
    w, k, v, prompt = inputs(cfg)
    prompt = prompt[: cfg.n_prompt]
    outs = []
    for sched in (2, 1, 0, 2):
        plan = _plan(tsp, cfg, w, scheduler=sched)
        outs.append(gpu_run_kv8(plan, cfg, k, v, prompt, cfg.start_pos, cfg.n_new))
        plan.close()
    for o in outs[1:]:
        assert np.array_equal(o[0], outs[0][0])
        assert np.array_equal(o[1].view(np.uint32), outs[0][1].view(np.uint32))
        for part in ("kq", "vq", "ks", "vs", "mu"):
            assert np.array_equal(o[2][part], outs[0][2][part])


def test_int8_weights_with_int8_cache_match_oracle(tsp):
    """Both INT8 forms together: weight-only INT8 GEMVs and the INT8 cache."""
    cfg, _ = DECODE["d64_prefill"]
    w, k, v, prompt = inputs(cfg)
    prompt = prompt[: cfg.n_prompt]
    plan = _plan(tsp, cfg, w, weight_format=tsp.WEIGHTS_INT8)
    toks, logits, _ = gpu_run_kv8(plan, cfg, k, v, prompt, cfg.start_pos, cfg.n_new)
    plan.close()
    check_parity(toks, logits, cfg, w, k, v, prompt, cfg.start_pos, cfg.n_new, "int8 weights + int8 kv",
                 qweights=oracle.quantize_model(w), kv_int8=True)


@pytest.mark.parametrize("name", ["llama1b_long", "llama1b"])
def test_full_width_one_layer_slice_with_int8_cache(tsp, name):
    """Full width at one layer with the INT8 cache: the long-context shape at
    32,767 cached positions and the 1,023-position one, strict tolerance."""
    cfg = replace(S.CONFIGS[name], n_layers=1, gain_sigma=GAINS)
    n_new = 8
    w, k, v, prompt = inputs(cfg)
    plan = _plan(tsp, cfg, w)
    toks, logits, g = gpu_run_kv8(plan, cfg, k, v, prompt, cfg.start_pos, n_new)
    plan.close()
    _, ref, *_ = check_parity(toks, logits, cfg, w, k, v, prompt, cfg.start_pos, n_new,
                              name + " one layer int8 kv", kv_int8=True)
    o = _oracle_parts(cfg, ref.kv8)
    n0 = cfg.start_pos
    assert np.array_equal(g["kq"][:, :n0], o["kq"][:, :n0])
    _check_new_rows(cfg, g, o, n0, n0 + prompt.size - 1 + n_new)


def test_multi_token_pass_rejects_int8_cache(tsp):
    import torch
    cfg = replace(S.CONFIGS["tiny"], gain_sigma=GAINS)
    w, *_ = inputs(cfg, n_pos=0)
    plan = _plan(tsp, cfg, w)
    cache = tsp.KV8Cache(tsp.ModelDesc.from_config(cfg))
    toks = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(tsp.TilesError) as e:
        plan.forward(cache.k, cache.v, toks, 0, out)
    assert e.value.status == -2                                   # TILES_ERR_UNSUPPORTED
    plan.close()
