"""Weight-only INT8 GEMV tiles against the INT8 oracle, through the C ABI.

The plan quantizes every GEMV matrix per output row on the device
(tiles_quantize_rows_int8). Its codes and scales must equal the oracle's
quantizer bit for bit, because a code is an integer decided in FP32 on both
sides. The decoder is then held to the same bars as the BF16 path
(gpu_helpers.check_parity): strict tolerance where the depth allows it, the
measured envelope at full depth, tokens identical up to the first near-tie.
"""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import synthetic as S
from gpu_helpers import GAINS, check_parity, gpu_run, inputs, with_gains

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
                    tsp.make_opts(weight_format=tsp.WEIGHTS_INT8, **opts))


def _oracle_q8(cfg, w, qw, k, v, prompt, start_pos, n_new, force=None, variant="seq"):
    return oracle.decode(cfg, w, k.copy(), v.copy(), prompt, start_pos, n_new,
                         force_tokens=force, qweights=qw, variant=variant)


@pytest.mark.parametrize("shape", [(7, 256), (64, 2048), (3, 8192), (128256, 64)])
def test_device_quantization_equals_oracle_bit_for_bit(tsp, shape):
    import torch
    rng = np.random.default_rng(shape[0] * 7 + shape[1])
    W = oracle.bf16_from_f32(rng.normal(0, 0.02, shape).astype(np.float32)).reshape(shape)
    W[0] = 0                                              # an all-zero row
    if shape[1] >= 4:                                     # ties: codes 2.5 and -2.5 (scale 2^-7)
        W[-1, :4] = oracle.bf16_from_f32(np.array([127, 2.5, -2.5, 3.5], np.float32) / 128)
        W[-1, 4:] = 0
    Wd = torch.from_numpy(W.view(np.int16)).cuda().view(torch.bfloat16)
    codes, scales = tsp.quantize_rows_int8(Wd)
    torch.cuda.synchronize()
    Q, s = oracle.quantize_rows(W)
    assert np.array_equal(codes.cpu().numpy(), Q)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), s.view(np.uint32))


def test_tiny_int8_matches_int8_oracle_and_is_bitwise_across_schedulers(tsp):
    cfg = with_gains(S.CONFIGS["tiny"])
    w, k, v, prompt = inputs(cfg, n_pos=0)
    qw = oracle.quantize_model(w)
    outs = []
    for sched in (2, 1, 0):
        plan = _plan(tsp, cfg, w, scheduler=sched)
        outs.append(gpu_run(plan, cfg, k, v, prompt, 0, cfg.n_new))
        plan.close()
    check_parity(outs[0][0], outs[0][1], cfg, w, k, v, prompt, 0, cfg.n_new, "tiny int8", qweights=qw)
    for o in outs[1:]:
        assert np.array_equal(o[0], outs[0][0])
        assert np.array_equal(o[1].view(np.uint32), outs[0][1].view(np.uint32))


VARIANTS = {
    "d128_g8_qknorm": replace(S.CONFIGS["tiny"], name="v1", head_dim=128, n_q_heads=8,
                              n_kv_heads=1, qk_norm=True, rope_theta=1e6, rms_eps=1e-6,
                              gain_sigma=GAINS),
    "g2_cache": replace(S.CONFIGS["tiny"], name="v3", start_pos=150, n_prompt=3, n_new=20,
                        max_pos=200, gain_sigma=GAINS),
}


@pytest.mark.parametrize("name", list(VARIANTS))
def test_int8_variants_match_int8_oracle(tsp, name):
    cfg = VARIANTS[name]
    w, k, v, prompt = inputs(cfg)
    prompt = prompt[: cfg.n_prompt]
    plan = _plan(tsp, cfg, w)
    toks, logits, *_ = gpu_run(plan, cfg, k, v, prompt, cfg.start_pos, cfg.n_new)
    check_parity(toks, logits, cfg, w, k, v, prompt, cfg.start_pos, cfg.n_new, name + " int8",
                 qweights=oracle.quantize_model(w))
    plan.close()


# long contexts: the kernel instances with the tensor-core attention path
MMA = {
    "d64_g2": replace(S.CONFIGS["tiny"], name="m1", start_pos=955, n_prompt=2, n_new=24, max_pos=1000,
                      gain_sigma=GAINS),
    "d128_g8_qknorm": replace(VARIANTS["d128_g8_qknorm"], name="m3", start_pos=490, n_prompt=2,
                              n_new=24, max_pos=520),
}


@pytest.mark.parametrize("name", list(MMA))
def test_int8_with_tensor_core_attention_matches_int8_oracle(tsp, name):
    cfg = MMA[name]
    w, k, v, prompt = inputs(cfg)
    prompt = prompt[: cfg.n_prompt]
    plan = _plan(tsp, cfg, w, kv_splits=2)
    toks, logits, *_ = gpu_run(plan, cfg, k, v, prompt, cfg.start_pos, cfg.n_new)
    check_parity(toks, logits, cfg, w, k, v, prompt, cfg.start_pos, cfg.n_new,
                 name + " int8, tensor-core attention", qweights=oracle.quantize_model(w))
    plan.close()


def test_int8_rejects_rows_not_a_multiple_of_16(tsp):
    cfg = replace(S.CONFIGS["tiny"], hidden=264, ffn=776, vocab=1000)
    d = tsp.ModelDesc.from_config(cfg)
    with pytest.raises(tsp.TilesError) as e:
        tsp.Schedule(d, 16, tsp.make_opts(weight_format=tsp.WEIGHTS_INT8))
    assert e.value.status == -2


@pytest.mark.parametrize("name", ["llama1b", "qwen3_0_6b", "llama1b_long"])
def test_int8_full_width_one_layer_slice_strict_tolerance(tsp, name):
    cfg = replace(S.CONFIGS[name], n_layers=1, gain_sigma=GAINS)
    n_new = 8
    w, k, v, prompt = inputs(cfg)
    plan = _plan(tsp, cfg, w)
    toks, logits, *_ = gpu_run(plan, cfg, k, v, prompt, cfg.start_pos, n_new)
    check_parity(toks, logits, cfg, w, k, v, prompt, cfg.start_pos, n_new, name + " int8 one layer",
                 qweights=oracle.quantize_model(w))
    plan.close()


def test_int8_full_depth_free_running_matches_int8_oracle_up_to_first_near_tie(tsp):
    """Llama-1B shape at full depth, 32 free-running steps: the same bar as the
    BF16 path, against the INT8 oracle and its reordered-summation build."""
    cfg = S.CONFIGS["llama1b"]
    n_new = 32
    w, k, v, prompt = inputs(cfg)
    qw = oracle.quantize_model(w)
    plan = _plan(tsp, cfg, w)
    toks, logits, *_ = gpu_run(plan, cfg, k, v, prompt, cfg.start_pos, n_new)
    plan.close()
    facts, ref, *_ = check_parity(toks, logits, cfg, w, k, v, prompt, cfg.start_pos, n_new,
                                  "llama1b int8 full depth", qweights=qw, envelope=True)
    free = _oracle_q8(cfg, w, qw, k, v, prompt, cfg.start_pos, n_new)
    d = n_new if facts["first_difference"] is None else facts["first_difference"]
    assert np.array_equal(free.tokens[:d], toks[:d])
