"""Seeded synthetic inputs shared by the CPU oracle and the GPU path.

This package is input plumbing only. It builds and loads ``synth.c`` (the
counter-based SplitMix64 + Box-Muller generator defined in that file's header)
and describes the five decoder shapes and workloads used throughout:

  tiny          2 layers, hidden 256, 4/2 heads, head_dim 64, FFN 768, vocab 1024
  llama1b       Llama-3.2-1B shape: 16 layers, hidden 2048, 32/8 heads, head_dim 64,
                FFN 8192, vocab 128256, RoPE theta 5e5 with llama3 frequency scaling
  qwen3_0_6b    Qwen3-0.6B shape: 28 layers, hidden 1024, 16/8 heads, head_dim 128,
                FFN 3072, vocab 151936, q/k RMSNorm, RoPE theta 1e6
  qwen3_4b      Qwen3-4B shape: 36 layers, hidden 2560, 32/8 heads, head_dim 128,
                FFN 9728, vocab 151936, q/k RMSNorm, RoPE theta 1e6
  llama1b_long  llama1b with 32,767 cached positions

(shapes and workloads as stated on "Tiles: Scheduling LLM Decoding as a Graph of
Tiles", intro, and "History and roadmap", "Where it stands" table).

It holds none of the decoding arithmetic: no norm, GEMV, RoPE, attention or
activation rounding lives here. Weights are N(0, 0.02) bf16, norm gains 1.0
(the workloads' setting) or, with ``gain_sigma`` > 0, seeded 1 + N(0, gain_sigma)
bf16 gains, a different vector per norm (the parity tests' setting: a kernel that
dropped or swapped a gain would then disagree with the oracle). KV-cache prefill
N(0, 1) bf16, token ids uniform. Tensor ids (the `tid` of the generator) are
fixed:

  weights (seed 0): embed 0; final_norm gain 1; layer l slot m -> 16 + 16*l + m
      with m = 0 attn_norm, 1 wq, 2 wk, 3 wv, 4 q_norm, 5 k_norm, 6 wo,
      7 ffn_norm, 8 w_gate, 9 w_up, 10 w_down
  kv prefill (seed 1): layer l keys 2*l, values 2*l + 1; element index
      (head * n_pos + pos) * head_dim + j
  tokens (seed 2): prompt 0
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

SEED_WEIGHTS = 0
SEED_KV = 1
SEED_TOKENS = 2
WEIGHT_SIGMA = 0.02
KV_SIGMA = 1.0
BF16_ONE = 0x3F80

# layer matrix slots in the tensor-id scheme
LAYER_SLOTS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ffn_norm",
               "w_gate", "w_up", "w_down")


def build(force: bool = False) -> str:
    """Compile synth.c into libsynth.so next to it (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            u64, i64, i32, dbl, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int,
                                      ctypes.c_double, ctypes.c_void_p)
            lib.synth_splitmix64_stream.argtypes = [u64, vp, i64]
            lib.synth_raw.argtypes = [u64, u64, u64]
            lib.synth_raw.restype = u64
            lib.synth_normal_f32.argtypes = [u64, u64, i64, i64, dbl, vp]
            lib.synth_normal_bf16.argtypes = [u64, u64, i64, i64, dbl, vp]
            lib.synth_kv_prefill_bf16.argtypes = [u64, u64, i32, i32, i32, i32, dbl, vp]
            lib.synth_tokens.argtypes = [u64, u64, i64, i64, vp]
            lib.synth_fill_bf16.argtypes = [vp, i64, ctypes.c_uint16]
            lib.synth_gain_bf16.argtypes = [u64, u64, i64, dbl, vp]
            _lib = lib
    return _lib


# ---------------------------------------------------------------- primitives
def splitmix64_stream(state: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _load().synth_splitmix64_stream(state, out.ctypes.data, n)
    return out


def raw(seed: int, tid: int, c: int) -> int:
    return int(_load().synth_raw(seed, tid, c))


def normal_f32(seed: int, tid: int, n: int, sigma: float = 1.0, i0: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_normal_f32(seed, tid, i0, n, sigma, out.ctypes.data)
    return out


def normal_bf16(seed: int, tid: int, shape, sigma: float) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_normal_bf16(seed, tid, 0, out.size, sigma, out.ctypes.data)
    return out


def tokens(seed: int, tid: int, n: int, n_vocab: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_tokens(seed, tid, n, n_vocab, out.ctypes.data)
    return out


def ones_bf16(n: int) -> np.ndarray:
    return np.full(n, BF16_ONE, dtype=np.uint16)


def gain_bf16(seed: int, tid: int, n: int, sigma: float) -> np.ndarray:
    """Norm gains 1 + sigma * N(0, 1) as bf16 bit patterns (element c of tensor tid)."""
    out = np.empty(n, dtype=np.uint16)
    _load().synth_gain_bf16(seed, tid, n, sigma, out.ctypes.data)
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (a bit shift)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------- configs
@dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    rms_eps: float
    qk_norm: bool = False
    rope_scaling: bool = False          # llama3 frequency scaling
    rs_factor: float = 32.0
    rs_low: float = 1.0
    rs_high: float = 4.0
    rs_orig_max: int = 8192
    gain_sigma: float = 0.0             # 0: every norm gain 1.0; else 1 + N(0, gain_sigma)
    # workload
    n_prompt: int = 1
    start_pos: int = 1023
    n_new: int = 64
    max_pos: int = 1088

    @property
    def n_steps(self) -> int:
        return self.n_prompt - 1 + self.n_new

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def weight_bytes(self, int8: bool = False) -> int:
        """Bytes of every weight once (tied embedding counted once, as the LM head):
        BF16, or with the GEMV matrices and the LM head as INT8 codes plus one FP32
        scale per row (norm weights stay BF16)."""
        H, F = self.hidden, self.ffn
        qkv_rows = self.q_dim + 2 * self.kv_dim
        matrix = qkv_rows * H + H * self.q_dim + 3 * F * H        # weights per layer
        rows = qkv_rows + H + 2 * F + H                            # output rows per layer
        norms = 2 * H + (2 * self.head_dim if self.qk_norm else 0)
        if not int8:
            return 2 * (self.n_layers * (matrix + norms) + self.vocab * H + H)
        return (self.n_layers * (matrix + 4 * rows + 2 * norms)
                + self.vocab * H + 4 * self.vocab + 2 * H)

    def algorithmic_bytes_per_token(self, int8: bool = False, kv_int8: bool = False) -> float:
        """Weights once + one embedding row + K/V of positions 0..P read + new K/V write,
        averaged over the run's decode positions. With ``kv_int8`` a cached
        position is its key and value codes plus their two FP32 scales."""
        if kv_int8:
            kv_pos_bytes = self.n_layers * self.n_kv_heads * (2 * self.head_dim + 8)
        else:
            kv_pos_bytes = 2 * 2 * self.n_layers * self.kv_dim  # K and V, one position, all layers
        p0 = self.start_pos
        steps = self.n_steps
        avg_read_pos = p0 + (steps - 1) / 2.0 + 1.0              # positions 0..P inclusive
        return (self.weight_bytes(int8) + 2 * self.hidden
                + kv_pos_bytes * avg_read_pos + kv_pos_bytes)

    def with_workload(self, **kw) -> "ModelConfig":
        return replace(self, **kw)


CONFIGS = {
    "tiny": ModelConfig("tiny", 2, 256, 4, 2, 64, 768, 1024, 1e4, 1e-5,
                        n_prompt=32, start_pos=0, n_new=16, max_pos=128),
    "llama1b": ModelConfig("llama1b", 16, 2048, 32, 8, 64, 8192, 128256, 5e5, 1e-5,
                           rope_scaling=True, n_prompt=1, start_pos=1023, n_new=64,
                           max_pos=1088),
    "qwen3_0_6b": ModelConfig("qwen3_0_6b", 28, 1024, 16, 8, 128, 3072, 151936, 1e6, 1e-6,
                              qk_norm=True, n_prompt=1, start_pos=1023, n_new=64, max_pos=1088),
    "qwen3_4b": ModelConfig("qwen3_4b", 36, 2560, 32, 8, 128, 9728, 151936, 1e6, 1e-6,
                            qk_norm=True, n_prompt=1, start_pos=1023, n_new=64, max_pos=1088),
    "llama1b_long": ModelConfig("llama1b_long", 16, 2048, 32, 8, 64, 8192, 128256, 5e5, 1e-5,
                                rope_scaling=True, n_prompt=1, start_pos=32767, n_new=64,
                                max_pos=32832),
}


# ---------------------------------------------------------------- model inputs
@dataclass
class ModelWeights:
    """Host bf16 bit patterns (uint16), row-major [out][in]."""
    embed: np.ndarray
    final_norm: np.ndarray
    layers: list = field(default_factory=list)   # list of dict slot -> array (or None)


def _tid(layer: int, slot: str) -> int:
    return 16 + 16 * layer + LAYER_SLOTS.index(slot)


def layer_weights(cfg: ModelConfig, l: int, seed: int = SEED_WEIGHTS) -> dict:
    H, F, d = cfg.hidden, cfg.ffn, cfg.head_dim
    s = WEIGHT_SIGMA

    def gain(slot, n):
        if cfg.gain_sigma > 0:
            return gain_bf16(seed, _tid(l, slot), n, cfg.gain_sigma)
        return ones_bf16(n)

    w = {
        "attn_norm": gain("attn_norm", H),
        "wq": normal_bf16(seed, _tid(l, "wq"), (cfg.q_dim, H), s),
        "wk": normal_bf16(seed, _tid(l, "wk"), (cfg.kv_dim, H), s),
        "wv": normal_bf16(seed, _tid(l, "wv"), (cfg.kv_dim, H), s),
        "q_norm": gain("q_norm", d) if cfg.qk_norm else None,
        "k_norm": gain("k_norm", d) if cfg.qk_norm else None,
        "wo": normal_bf16(seed, _tid(l, "wo"), (H, cfg.q_dim), s),
        "ffn_norm": gain("ffn_norm", H),
        "w_gate": normal_bf16(seed, _tid(l, "w_gate"), (F, H), s),
        "w_up": normal_bf16(seed, _tid(l, "w_up"), (F, H), s),
        "w_down": normal_bf16(seed, _tid(l, "w_down"), (H, F), s),
    }
    return w


def model_weights(cfg: ModelConfig, seed: int = SEED_WEIGHTS) -> ModelWeights:
    embed = normal_bf16(seed, 0, (cfg.vocab, cfg.hidden), WEIGHT_SIGMA)
    fnorm = (gain_bf16(seed, 1, cfg.hidden, cfg.gain_sigma) if cfg.gain_sigma > 0
             else ones_bf16(cfg.hidden))
    mw = ModelWeights(embed=embed, final_norm=fnorm)
    mw.layers = [layer_weights(cfg, l, seed) for l in range(cfg.n_layers)]
    return mw


def kv_prefill(cfg: ModelConfig, n_pos: int | None = None, seed: int = SEED_KV):
    """K and V caches [L][n_kv][max_pos][d] bf16 with positions [0, n_pos) filled
    from N(0, 1); the rest zero."""
    n_pos = cfg.start_pos if n_pos is None else n_pos
    shape = (cfg.n_layers, cfg.n_kv_heads, cfg.max_pos, cfg.head_dim)
    k = np.zeros(shape, dtype=np.uint16)
    v = np.zeros(shape, dtype=np.uint16)
    if n_pos > 0:
        lib = _load()
        for l in range(cfg.n_layers):
            lib.synth_kv_prefill_bf16(seed, 2 * l, cfg.n_kv_heads, cfg.max_pos, n_pos,
                                      cfg.head_dim, KV_SIGMA, k[l].ctypes.data)
            lib.synth_kv_prefill_bf16(seed, 2 * l + 1, cfg.n_kv_heads, cfg.max_pos, n_pos,
                                      cfg.head_dim, KV_SIGMA, v[l].ctypes.data)
    return k, v


def prompt(cfg: ModelConfig, seed: int = SEED_TOKENS) -> np.ndarray:
    return tokens(seed, 0, cfg.n_prompt, cfg.vocab)
