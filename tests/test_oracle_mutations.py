"""The decoder-wiring pins fail on plausible slips in the oracle.

Each case plants one mistake in a copy of ``oracle/oracle.c`` (a gain routed to
the wrong step, a layer index reversed, q and k norms swapped, the q/k norm
moved after RoPE, q or k left unrotated), builds it with the same flags as the
oracle, and checks that the pins named beside it fail on that build. The real
oracle passes them (``test_oracle_pins.py``). The source lines a case replaces
must exist verbatim, so an edit of the oracle that moves them shows up here.
"""
import os
import subprocess

import pytest

import oracle as O
import test_oracle_pins as pins

ATTN = pins.test_decoder_norm_gains_route_to_their_own_step_attention_path
FFN = pins.test_decoder_norm_gains_route_to_their_own_step_ffn_path
QK = pins.test_decoder_qk_norm_before_rope_and_both_rotated_at_the_position

_Q_BLOCK = """            for (int i = 0; i < nq; ++i) {
                if (m->qk_norm) {
                    orc_rmsnorm(q + i * d, w->q_norm, d, m->rms_eps, tmp);
                    memcpy(q + i * d, tmp, sizeof(float) * d);
                }
                orc_rope_apply(q + i * d, d, cs, sn);
            }"""

MUTATIONS = {
    "attention prologue takes the ffn gain": (
        "orc_rmsnorm(x, w->attn_norm, H, m->rms_eps, h);",
        "orc_rmsnorm(x, w->ffn_norm, H, m->rms_eps, h);", [ATTN]),
    "ffn prologue takes the attention gain": (
        "orc_rmsnorm(x, w->ffn_norm, H, m->rms_eps, h);",
        "orc_rmsnorm(x, w->attn_norm, H, m->rms_eps, h);", [FFN]),
    "final norm takes the last layer's ffn gain": (
        "orc_rmsnorm(x, final_norm, H, m->rms_eps, h);",
        "orc_rmsnorm(x, layers[L - 1].ffn_norm, H, m->rms_eps, h);", [ATTN, FFN]),
    "layers visited in reverse": (
        "const orc_layer *w = &layers[l];",
        "const orc_layer *w = &layers[L - 1 - l];", [ATTN, FFN]),
    "q and k norms swapped": (
        "orc_rmsnorm(q + i * d, w->q_norm, d, m->rms_eps, tmp);",
        "orc_rmsnorm(q + i * d, w->k_norm, d, m->rms_eps, tmp);", [QK]),
    "q norm after RoPE": (
        _Q_BLOCK,
        _Q_BLOCK.replace("                orc_rope_apply(q + i * d, d, cs, sn);\n", "")
                .replace("                if (m->qk_norm) {",
                         "                orc_rope_apply(q + i * d, d, cs, sn);\n                if (m->qk_norm) {"),
        [QK]),
    "k not rotated": ("orc_rope_apply(k + i * d, d, cs, sn);", "", [QK]),
    "q not rotated": ("orc_rope_apply(q + i * d, d, cs, sn);", "", [QK]),
}


@pytest.fixture(scope="module")
def src():
    with open(O._SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_pins_catch_the_planted_mistake(name, src, tmp_path, monkeypatch, tiny_cfg):
    old, new, catchers = MUTATIONS[name]
    assert src.count(old) == 1, f"oracle source no longer holds the line this case mutates: {old!r}"
    path = tmp_path / "oracle_mutant.c"
    path.write_text(src.replace(old, new))
    so = str(tmp_path / "liboracle_mutant.so")
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           "-fno-fast-math", "-o", so, str(path), "-lm"])
    O.lib()                                             # the real build is loaded first
    monkeypatch.setitem(O._libs, "seq", O.load_library(so))
    for pin in catchers:
        with pytest.raises(AssertionError):
            pin(tiny_cfg)
    os.remove(so)
