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

import synthetic as S
from gpu_helpers import ATOL, RTOL, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsp():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tile_scheduled_persistent_gb300 as t
    t.build()
    return t


def _run(tsp, plan, cfg, k, v, prompt, use_noalloc):
    import torch
    kc = tsp.to_device_bf16(k)
    vc = tsp.to_device_bf16(v)
    steps = prompt.size - 1 + cfg.n_new
    toks = torch.full((cfg.n_new,), -1, dtype=torch.int32, device="cuda")
    logits = torch.full((steps, cfg.vocab), float("nan"), dtype=torch.float32, device="cuda")
    dprompt = torch.from_numpy(np.ascontiguousarray(prompt, np.int32)).cuda()
    if use_noalloc:
        plan.decode_noalloc(kc, vc, dprompt, cfg.start_pos, cfg.n_new, toks, logits)
    else:
        plan.decode(kc, vc, dprompt, cfg.start_pos, cfg.n_new, toks, logits)
    plan.check()
    return toks.cpu().numpy(), logits.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "g2_cache"])
def test_noalloc_matches_regular_decode_twice(tsp, name):
    from dataclasses import replace
    cfg = S.CONFIGS["tiny"] if name == "tiny" else replace(
        S.CONFIGS["tiny"], name="v3", start_pos=150, n_prompt=3, n_new=20, max_pos=200)
    w, k, v, prompt = inputs(cfg, n_pos=cfg.start_pos)
    prompt = prompt[: cfg.n_prompt]
    plan = tsp.Plan(tsp.ModelDesc.from_config(cfg), tsp.upload_weights(w))
    ref_toks, ref_logits = _run(tsp, plan, cfg, k, v, prompt, use_noalloc=False)
    for _ in range(2):
        toks, logits = _run(tsp, plan, cfg, k, v, prompt, use_noalloc=True)
        assert np.array_equal(toks, ref_toks)
        assert not np.isnan(logits).any()
        assert (np.abs(logits - ref_logits) <= ATOL + RTOL * np.abs(ref_logits)).all()
    plan.close()


def test_noalloc_rejects_a_plan_that_does_not_fit(tsp):
    """16 q heads of 128 dims in 64 KV splits need 1.06 MB of split partials
    (64-bit words), more than the fixed 1 MiB array."""
    import torch
    from dataclasses import replace
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
