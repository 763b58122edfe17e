"""Shared helpers of the GPU parity tests: seeded inputs, one decode through the
C ABI, and the comparison against the CPU oracle."""
from __future__ import annotations

import numpy as np

import oracle
import synthetic as S

# tolerance on logits (greedy tokens must match exactly):
# |gpu - oracle| <= ATOL + RTOL * |oracle|
ATOL = 3e-2
RTOL = 1e-2


def inputs(cfg, n_pos=None):
    w = S.model_weights(cfg)
    k, v = S.kv_prefill(cfg, n_pos=cfg.start_pos if n_pos is None else n_pos)
    return w, k, v, S.prompt(cfg)


def oracle_run(cfg, w, k, v, prompt, start_pos, n_new, force=None):
    kk, vv = k.copy(), v.copy()
    r = oracle.decode(cfg, w, kk, vv, prompt, start_pos, n_new, force_tokens=force)
    return r, kk, vv


def gpu_run(plan, cfg, k, v, prompt, start_pos, n_new, want_logits=True, split_at=None):
    """Decode on the GPU. With `split_at` = a step index past the prompt, the run
    is made of two calls: steps [0, a), then steps [a, end) resuming from the
    cache the first call wrote and fed the last token it produced. Returns
    tokens, logits, and the caches as numpy bf16 bit patterns."""
    import torch
    import tile_scheduled_persistent_gb300 as tsp
    kc = tsp.to_device_bf16(k)
    vc = tsp.to_device_bf16(v)
    prompt = np.asarray(prompt, np.int32)
    n_prompt = prompt.size
    steps = n_prompt - 1 + n_new
    toks = torch.full((max(n_new, 1),), -1, dtype=torch.int32, device="cuda")
    logits = (torch.full((max(steps, 1), cfg.vocab), float("nan"), dtype=torch.float32,
                         device="cuda") if want_logits else None)
    dprompt = torch.from_numpy(prompt).cuda()
    if split_at is None:
        plan.decode(kc, vc, dprompt, start_pos, n_new, toks, logits)
    else:
        a = int(split_at)
        assert n_prompt <= a < steps
        n1 = a - (n_prompt - 1)
        plan.decode(kc, vc, dprompt, start_pos, n1, toks[:n1],
                    logits[:a] if logits is not None else None)
        plan.check()
        plan.decode(kc, vc, toks[n1 - 1:n1].clone(), start_pos + a, n_new - n1, toks[n1:],
                    logits[a:] if logits is not None else None)
    plan.check()
    torch.cuda.synchronize()
    out_l = logits.cpu().numpy() if logits is not None else None
    return (toks.cpu().numpy()[:n_new], out_l,
            kc.view(torch.int16).cpu().numpy().view(np.uint16),
            vc.view(torch.int16).cpu().numpy().view(np.uint16))


def assert_parity(g_tokens, g_logits, ref, what=""):
    """Greedy tokens exact; logits within tolerance, with diagnostics on failure."""
    if g_logits is not None:
        err = np.abs(g_logits - ref.logits)
        bound = ATOL + RTOL * np.abs(ref.logits)
        bad = err > bound
        assert not np.isnan(g_logits).any(), f"{what}: NaN logits"
        assert not bad.any(), (f"{what}: {int(bad.sum())} logits out of tolerance, max err "
                               f"{float(err.max()):.3e}")
    if not np.array_equal(g_tokens, ref.tokens):
        i = int(np.nonzero(g_tokens != ref.tokens)[0][0])
        raise AssertionError(f"{what}: token mismatch at output {i}: gpu {g_tokens[i]} oracle "
                             f"{ref.tokens[i]}; oracle top-2 gaps {ref.gaps.tolist()}")
