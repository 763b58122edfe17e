"""CPU oracle for batch-1 greedy decoding (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path never does, and this
package imports nothing from it: the two share only the seeded input
generators in ``synthetic``.

The arithmetic lives in ``oracle.c`` (plain C, FP32 math, BF16 weights and
BF16 activations at the rounding points stated in that file's header); this
module builds it with gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_ALT_LIB_PATH = os.path.join(_HERE, "liboracle_alt.so")
_lock = threading.Lock()
_libs = {}


class OrcModel(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                 "max_pos", "qk_norm", "rope_scaling")] + \
               [(n, ctypes.c_double) for n in
                ("rope_theta", "rs_factor", "rs_low", "rs_high", "rs_orig_max")] + \
               [("rms_eps", ctypes.c_float)]


_SLOTS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ffn_norm", "w_gate",
          "w_up", "w_down")


class OrcLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _SLOTS]


_QSLOTS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


class OrcKV8(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("kq", "vq", "ks", "vs", "mu")]


class OrcQLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _QSLOTS] + \
               [(n, ctypes.c_void_p) for n in ("sq", "sk", "sv", "so", "s_gate", "s_up", "s_down")]


def _build_one(path, extra, force):
    if not force and os.path.exists(path) and os.path.getmtime(path) >= os.path.getmtime(_SRC):
        return path
    tmp = path + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           "-fno-fast-math", *extra, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, path)
    return path


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc -O2, OpenMP, no FP contraction) and
    the alternative-summation-order build liboracle_alt.so (noise-floor reference)."""
    _build_one(_ALT_LIB_PATH, ["-DORC_ALT_SUM_ORDER"], force)
    return _build_one(_LIB_PATH, [], force)


def load_library(path: str):
    """Loads an oracle build at `path` with the argument types of every entry point."""
    L = ctypes.CDLL(path)
    vp, i32, f32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64
    L.orc_bf16_from_f32.argtypes = [f32]
    L.orc_bf16_from_f32.restype = ctypes.c_uint16
    L.orc_f32_from_bf16.argtypes = [ctypes.c_uint16]
    L.orc_f32_from_bf16.restype = f32
    L.orc_bf16_round_array.argtypes = [vp, vp, i64]
    L.orc_rmsnorm.argtypes = [vp, vp, i32, f32, vp]
    L.orc_rope_inv_freq.argtypes = [ctypes.POINTER(OrcModel), vp]
    L.orc_rope_cos_sin.argtypes = [ctypes.POINTER(OrcModel), i32, vp, vp]
    L.orc_rope_apply.argtypes = [vp, i32, vp, vp]
    L.orc_gemv.argtypes = [vp, i32, i32, vp, vp]
    L.orc_attention.argtypes = [vp, vp, vp, i32, i32, f32, vp]
    L.orc_attention_split.argtypes = [vp, vp, vp, i32, i32, f32, i32, vp, vp]
    L.orc_quantize_rows.argtypes = [vp, i32, i32, vp, vp]
    L.orc_gemv_q8.argtypes = [vp, vp, i32, i32, vp, vp]
    L.orc_kv8_quantize_row.argtypes = [vp, i32, vp, vp]
    L.orc_kv8_key_mean.argtypes = [vp, i32, i32, vp]
    L.orc_kv8_from_bf16.argtypes = [ctypes.POINTER(OrcModel), vp, vp, i32, ctypes.POINTER(OrcKV8)]
    L.orc_attention_kv8.argtypes = [vp, vp, vp, vp, vp, i32, i32, f32, vp]
    L.orc_decode.argtypes = [ctypes.POINTER(OrcModel), ctypes.POINTER(OrcLayer), vp, vp,
                             vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, i32,
                             ctypes.POINTER(OrcQLayer), vp, vp, ctypes.POINTER(OrcKV8)]
    L.orc_decode.restype = i32
    return L


def lib(variant: str = "seq"):
    """The oracle library; variant "alt" is the build with the other GEMV summation order."""
    with _lock:
        if variant not in _libs:
            build()
            _libs[variant] = load_library(_ALT_LIB_PATH if variant == "alt" else _LIB_PATH)
    return _libs[variant]


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------- elementary ops
def bf16_from_f32(x) -> np.ndarray:
    x = _c(np.atleast_1d(x), np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_bf16_round_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def f32_from_bf16(b) -> np.ndarray:
    b = _c(np.atleast_1d(b), np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def rmsnorm(x, g_bf16, eps: float) -> np.ndarray:
    x = _c(x, np.float32)
    g = _c(g_bf16, np.uint16)
    out = np.empty_like(x)
    lib().orc_rmsnorm(x.ctypes.data, g.ctypes.data, x.size, eps, out.ctypes.data)
    return out


def model_struct(cfg) -> OrcModel:
    return OrcModel(n_layers=cfg.n_layers, hidden=cfg.hidden, n_q_heads=cfg.n_q_heads,
                    n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, ffn=cfg.ffn,
                    vocab=cfg.vocab, max_pos=cfg.max_pos, qk_norm=int(cfg.qk_norm),
                    rope_scaling=int(cfg.rope_scaling), rope_theta=cfg.rope_theta,
                    rs_factor=cfg.rs_factor, rs_low=cfg.rs_low, rs_high=cfg.rs_high,
                    rs_orig_max=float(cfg.rs_orig_max), rms_eps=cfg.rms_eps)


def rope_inv_freq(cfg) -> np.ndarray:
    m = model_struct(cfg)
    out = np.empty(cfg.head_dim // 2, np.float64)
    lib().orc_rope_inv_freq(ctypes.byref(m), out.ctypes.data)
    return out


def rope_cos_sin(cfg, pos: int):
    m = model_struct(cfg)
    c = np.empty(cfg.head_dim // 2, np.float32)
    s = np.empty(cfg.head_dim // 2, np.float32)
    lib().orc_rope_cos_sin(ctypes.byref(m), pos, c.ctypes.data, s.ctypes.data)
    return c, s


def rope_apply(v, cos, sin) -> np.ndarray:
    v = _c(v, np.float32).copy()
    cos = _c(cos, np.float32)
    sin = _c(sin, np.float32)
    lib().orc_rope_apply(v.ctypes.data, v.size, cos.ctypes.data, sin.ctypes.data)
    return v


def gemv(W_bf16, x) -> np.ndarray:
    W = _c(W_bf16, np.uint16)
    x = _c(x, np.float32)
    y = np.empty(W.shape[0], np.float32)
    lib().orc_gemv(W.ctypes.data, W.shape[0], W.shape[1], x.ctypes.data, y.ctypes.data)
    return y


def quantize_rows(W_bf16):
    """Weight-only INT8 of a [rows][cols] BF16 matrix: (codes int8 [rows][cols],
    scales float32 [rows]), scale = row absmax / 127, codes rounded to nearest
    even and clamped to +-127."""
    W = _c(W_bf16, np.uint16)
    Q = np.empty(W.shape, np.int8)
    sc = np.empty(W.shape[0], np.float32)
    lib().orc_quantize_rows(W.ctypes.data, W.shape[0], W.shape[1], Q.ctypes.data, sc.ctypes.data)
    return Q, sc


def gemv_q8(Q, scale, x) -> np.ndarray:
    Q = _c(Q, np.int8)
    sc = _c(scale, np.float32)
    x = _c(x, np.float32)
    y = np.empty(Q.shape[0], np.float32)
    lib().orc_gemv_q8(Q.ctypes.data, sc.ctypes.data, Q.shape[0], Q.shape[1], x.ctypes.data,
                      y.ctypes.data)
    return y


class QuantWeights:
    """INT8 copies of every GEMV matrix of a model (``quantize_model``)."""
    def __init__(self, layers, lm):
        self.layers = layers      # per layer: {slot: (codes, scales)}
        self.lm = lm              # (codes, scales) of the tied LM head


def quantize_model(weights) -> QuantWeights:
    layers = [{slot: quantize_rows(w[slot]) for slot in _QSLOTS} for w in weights.layers]
    return QuantWeights(layers, quantize_rows(weights.embed))


def attention(q, K_bf16, V_bf16, scale: float) -> np.ndarray:
    q = _c(q, np.float32)
    K = _c(K_bf16, np.uint16)
    V = _c(V_bf16, np.uint16)
    out = np.empty(q.size, np.float32)
    lib().orc_attention(q.ctypes.data, K.ctypes.data, V.ctypes.data, K.shape[0], q.size, scale,
                        out.ctypes.data)
    return out


def attention_split(q, K_bf16, V_bf16, scale: float, bounds) -> np.ndarray:
    q = _c(q, np.float32)
    K = _c(K_bf16, np.uint16)
    V = _c(V_bf16, np.uint16)
    b = _c(bounds, np.int32)
    out = np.empty(q.size, np.float32)
    lib().orc_attention_split(q.ctypes.data, K.ctypes.data, V.ctypes.data, K.shape[0], q.size,
                              scale, b.size - 1, b.ctypes.data, out.ctypes.data)
    return out


# ------------------------------------------------------------- INT8 KV cache
def kv8_quantize_row(x):
    """One cached row to INT8: (codes int8[d], FP32 scale), absmax / 127, ties to even."""
    x = _c(x, np.float32)
    c = np.empty(x.size, np.int8)
    s = np.zeros(1, np.float32)
    lib().orc_kv8_quantize_row(x.ctypes.data, x.size, c.ctypes.data, s.ctypes.data)
    return c, s[0]


def kv8_key_mean(K_bf16):
    """Per-channel mean of [n][d] BF16 keys (the key shift mu), FP32."""
    K = _c(K_bf16, np.uint16)
    mu = np.empty(K.shape[1], np.float32)
    lib().orc_kv8_key_mean(K.ctypes.data, K.shape[0], K.shape[1], mu.ctypes.data)
    return mu


def attention_kv8(q, Kq, Ks, Vq, Vs, scale: float) -> np.ndarray:
    q = _c(q, np.float32)
    Kq, Vq = _c(Kq, np.int8), _c(Vq, np.int8)
    Ks, Vs = _c(Ks, np.float32), _c(Vs, np.float32)
    out = np.empty(q.size, np.float32)
    lib().orc_attention_kv8(q.ctypes.data, Kq.ctypes.data, Ks.ctypes.data, Vq.ctypes.data,
                            Vs.ctypes.data, Kq.shape[0], q.size, scale, out.ctypes.data)
    return out


class KV8Cache:
    """The INT8 form of a [L][n_kv][max_pos][d] cache pair: codes kq, vq, FP32
    scales ks, vs ([L][n_kv][max_pos]) and key shifts mu ([L][n_kv][d])."""
    def __init__(self, cfg):
        shape = (cfg.n_layers, cfg.n_kv_heads, cfg.max_pos, cfg.head_dim)
        self.kq = np.zeros(shape, np.int8)
        self.vq = np.zeros(shape, np.int8)
        self.ks = np.zeros(shape[:3], np.float32)
        self.vs = np.zeros(shape[:3], np.float32)
        self.mu = np.zeros((cfg.n_layers, cfg.n_kv_heads, cfg.head_dim), np.float32)

    def struct(self):
        return OrcKV8(*(a.ctypes.data for a in (self.kq, self.vq, self.ks, self.vs, self.mu)))


def kv8_from_bf16(cfg, k_cache, v_cache, n_pos: int) -> KV8Cache:
    """INT8 cache of the prefilled positions 0..n_pos-1 (key shifts from them)."""
    kv = KV8Cache(cfg)
    st = kv.struct()
    m = model_struct(cfg)
    lib().orc_kv8_from_bf16(ctypes.byref(m), _c(k_cache, np.uint16).ctypes.data,
                            _c(v_cache, np.uint16).ctypes.data, n_pos, ctypes.byref(st))
    return kv


# ------------------------------------------------------------- whole decoder
class DecodeResult:
    def __init__(self, tokens, logits, gaps, kv8=None):
        self.tokens = tokens
        self.logits = logits
        self.gaps = gaps
        self.kv8 = kv8


def decode(cfg, weights, k_cache, v_cache, prompt, start_pos: int, n_new: int,
           force_tokens=None, want_logits: bool = True, n_threads: int = 0,
           variant: str = "seq", qweights: QuantWeights | None = None,
           kv_int8: bool = False) -> DecodeResult:
    """Run the oracle. ``weights`` is a ``synthetic.ModelWeights``; ``k_cache`` and
    ``v_cache`` are [L][n_kv][max_pos][d] uint16 arrays updated in place.
    ``variant="alt"`` runs the build with the other GEMV summation order.
    With ``qweights`` (``quantize_model(weights)``) every GEMV uses the INT8
    weights; the embedding lookup stays BF16. With ``kv_int8`` attention reads
    an INT8 KV cache with smoothed keys, built from the prefilled positions
    (``kv8_from_bf16``) and extended every step; it is returned as ``.kv8``."""
    prompt = _c(prompt, np.int32)
    n_prompt = prompt.size
    steps = n_prompt - 1 + n_new
    layers = (OrcLayer * cfg.n_layers)()
    keep = []
    for l, w in enumerate(weights.layers):
        for slot in _SLOTS:
            a = w.get(slot)
            if a is not None:
                a = _c(a, np.uint16)
                keep.append(a)
                setattr(layers[l], slot, a.ctypes.data)
            else:
                setattr(layers[l], slot, None)
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    assert v_cache.dtype == np.uint16 and v_cache.flags.c_contiguous
    embed = _c(weights.embed, np.uint16)
    fnorm = _c(weights.final_norm, np.uint16)
    out_tokens = np.zeros(max(n_new, 1), np.int32)
    logits = np.empty((steps, cfg.vocab), np.float32) if want_logits else None
    gaps = np.empty(max(steps, 1), np.float32)
    force = None if force_tokens is None else _c(force_tokens, np.int32)
    m = model_struct(cfg)
    qlayers, lm_q, lm_s = None, None, None
    if qweights is not None:
        qlayers = (OrcQLayer * cfg.n_layers)()
        for l, ql in enumerate(qweights.layers):
            for slot, sname in zip(_QSLOTS, ("sq", "sk", "sv", "so", "s_gate", "s_up", "s_down")):
                codes, sc = ql[slot]
                setattr(qlayers[l], slot, codes.ctypes.data)
                setattr(qlayers[l], sname, sc.ctypes.data)
        lm_q, lm_s = qweights.lm[0].ctypes.data, qweights.lm[1].ctypes.data
    kv8 = kv8_from_bf16(cfg, k_cache, v_cache, start_pos) if kv_int8 else None
    kv8_st = kv8.struct() if kv8 is not None else None
    rc = lib(variant).orc_decode(ctypes.byref(m), layers, embed.ctypes.data, fnorm.ctypes.data,
                          k_cache.ctypes.data, v_cache.ctypes.data, prompt.ctypes.data, n_prompt,
                          start_pos, n_new, _ptr(force), out_tokens.ctypes.data, _ptr(logits),
                          gaps.ctypes.data, n_threads, qlayers, lm_q, lm_s,
                          ctypes.byref(kv8_st) if kv8_st is not None else None)
    if rc != 0:
        raise ValueError(f"orc_decode rejected its arguments (rc={rc})")
    return DecodeResult(out_tokens[:n_new], logits, gaps[:steps], kv8)


# ------------------------------------------------------------- multi-token verify
class VerifyResult:
    def __init__(self, n_accepted, tokens, argmax, logits):
        self.n_accepted = n_accepted   # drafts accepted
        self.tokens = tokens           # emitted: the accepted drafts, then one model token
        self.argmax = argmax           # the model's token after each of the k + 1 inputs
        self.logits = logits           # [k + 1][vocab]


def verify(cfg, weights, k_cache, v_cache, last_token: int, start_pos: int, drafts,
           qweights: QuantWeights | None = None) -> VerifyResult:
    """One verify step over k draft tokens ("History and roadmap": 16-token
    verify steps on the split-KV decode kernels; the drafts' source is out of
    scope). The inputs last_token, d_1..d_k take positions start_pos ..
    start_pos + k (their K/V rows are written). a_i is the greedy token after
    input i. The step accepts the longest prefix with d_{i+1} = a_i, n drafts,
    and emits d_1..d_n, then a_n. Rows past start_pos + n are left as written
    and are stale; the caller's next step starts at start_pos + n + 1.
    Greedy decoding from the same state emits the same tokens."""
    drafts = [int(t) for t in drafts]
    inputs = np.array([int(last_token)] + drafts, np.int32)
    r = decode(cfg, weights, k_cache, v_cache, inputs, start_pos, 1, qweights=qweights)
    argmax = r.logits.argmax(axis=1).astype(np.int32)          # lowest index on ties
    n = 0
    while n < len(drafts) and drafts[n] == argmax[n]:
        n += 1
    tokens = np.array(drafts[:n] + [int(argmax[n])], np.int32)
    return VerifyResult(n, tokens, argmax, r.logits)

