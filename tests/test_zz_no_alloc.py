"""The allocation-free decode entry point (tiles_decode_noalloc).

Some callers may not allocate device memory when they decode (their device
memory is all owned by their own allocator, or their runtime forbids
allocation after start-up). For them the library offers a decode whose working
memory is a fixed array compiled into the library. These tests call it through
the C ABI and hold it to the regular entry point's results, twice in a row
(the array keeps the first call's contents when the second one starts).

This file is collected last on purpose: a run that stops at the first failure
has run every other test before it gets here.
"""
import numpy as np
import pytest

from dataclasses import replace

import synthetic as S
from gpu_helpers import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tile_scheduled_persistent_gb300 as t
    t.build()
    return t


def _run(tsp, plan, cfg, k, v, prompt, use_noalloc, n_new=None):
    import torch
    n_new = cfg.n_new if n_new is None else n_new
    kc = tsp.to_device_bf16(k)
    vc = tsp.to_device_bf16(v)
    steps = prompt.size - 1 + n_new
    toks = torch.full((n_new,), -1, dtype=torch.int32, device="cuda")
    logits = torch.full((steps, cfg.vocab), float("nan"), dtype=torch.float32, device="cuda")
    dprompt = torch.from_numpy(np.ascontiguousarray(prompt, np.int32)).cuda()
    if use_noalloc:
        plan.decode_noalloc(kc, vc, dprompt, cfg.start_pos, n_new, toks, logits)
    else:
        plan.decode(kc, vc, dprompt, cfg.start_pos, n_new, toks, logits)
    plan.check()
    return (toks.cpu().numpy(), logits.cpu().numpy(),
            kc.view(torch.int16).cpu().numpy(), vc.view(torch.int16).cpu().numpy())


CASES = {
    # prompt then decode, one launch
    "tiny": (S.CONFIGS["tiny"], None),
    # cached positions across several KV blocks
    "g2_cache": (replace(S.CONFIGS["tiny"], name="v3", start_pos=150, n_prompt=3, n_new=20,
                         max_pos=200), None),
    # 31 + 80 = 111 steps: two launches in one call, so the array is cleared
    # again between launches of the same call
    "tiny_two_launches": (S.CONFIGS["tiny"].with_workload(max_pos=128), 80),
}


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_equals_regular_decode_bitwise_twice(tsp, name):
    """Same kernel, same inputs: tokens, logits and the caches written must be
    bit-identical to tiles_decode's, on two calls in a row (the second finds
    the array as the first left it)."""
    cfg, n_new = CASES[name]
    cfg = replace(cfg, gain_sigma=0.25)
    w, k, v, prompt = inputs(cfg, n_pos=cfg.start_pos)
    prompt = prompt[: cfg.n_prompt]
    plan = tsp.Plan(tsp.ModelDesc.from_config(cfg), tsp.upload_weights(w))
    ref = _run(tsp, plan, cfg, k, v, prompt, use_noalloc=False, n_new=n_new)
    assert not np.isnan(ref[1]).any()
    for _ in range(2):
        got = _run(tsp, plan, cfg, k, v, prompt, use_noalloc=True, n_new=n_new)
        assert np.array_equal(got[0], ref[0])
        assert np.array_equal(got[1].view(np.uint32), ref[1].view(np.uint32))
        assert np.array_equal(got[2], ref[2]) and np.array_equal(got[3], ref[3])
    plan.close()


def test_noalloc_with_int8_cache_equals_regular_decode_bitwise(tsp):
    """The INT8 KV cache plan through the allocation-free entry point: tokens,
    logits and every part of the INT8 cache bit-identical to tiles_decode's."""
    import torch
    cfg = replace(S.CONFIGS["tiny"], name="kv8", start_pos=230, n_prompt=2, n_new=40, max_pos=300,
                  gain_sigma=0.25)
    w, k, v, prompt = inputs(cfg)
    prompt = np.ascontiguousarray(prompt[: cfg.n_prompt], np.int32)
    desc = tsp.ModelDesc.from_config(cfg)
    plan = tsp.Plan(desc, tsp.upload_weights(w), tsp.make_opts(kv_format=tsp.KV_INT8))
    outs = []
    for use_noalloc in (False, True, True):
        cache = tsp.KV8Cache(desc).from_bf16(tsp.to_device_bf16(k), tsp.to_device_bf16(v), cfg.start_pos)
        steps = prompt.size - 1 + cfg.n_new
        toks = torch.full((cfg.n_new,), -1, dtype=torch.int32, device="cuda")
        logits = torch.full((steps, cfg.vocab), float("nan"), dtype=torch.float32, device="cuda")
        dprompt = torch.from_numpy(prompt).cuda()
        fn = plan.decode_noalloc if use_noalloc else plan.decode
        fn(cache.k, cache.v, dprompt, cfg.start_pos, cfg.n_new, toks, logits)
        plan.check()
        outs.append((toks.cpu().numpy(), logits.cpu().numpy(), cache.host()))
    assert not np.isnan(outs[0][1]).any()
    for got in outs[1:]:
        assert np.array_equal(got[0], outs[0][0])
        assert np.array_equal(got[1].view(np.uint32), outs[0][1].view(np.uint32))
        for part in ("kq", "vq", "ks", "vs", "mu"):
            assert np.array_equal(got[2][part], outs[0][2][part])
    plan.close()



def test_noalloc_rejects_a_plan_that_does_not_fit(tsp):
    """16 q heads of 128 dims in 64 KV splits need 1.06 MB of split partials
    (64-bit words), more than the fixed 1 MiB array."""
    import torch
    cfg = replace(S.CONFIGS["tiny"], name="wide", n_q_heads=16, head_dim=128)
    w, k, v, prompt = inputs(cfg, n_pos=0)
    plan = tsp.Plan(tsp.ModelDesc.from_config(cfg), tsp.upload_weights(w),
                    tsp.make_opts(kv_splits=64))
    kc, vc = tsp.to_device_bf16(k), tsp.to_device_bf16(v)
    out = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(tsp.TilesError) as e:
        plan.decode_noalloc(kc, vc, torch.tensor([3], dtype=torch.int32, device="cuda"), 0, 4, out)
    assert e.value.status == -5
    plan.close()
