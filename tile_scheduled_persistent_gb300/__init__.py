"""Python binding of the tile-scheduled persistent decoder (include/tiles.h).

Argument marshalling only: every step of the decode path runs in the CUDA
library ``libtiles.so``. Importing this package loads that library and raises
if it is missing; there is no fallback. Device buffers are PyTorch tensors
(PyTorch is used for device memory and streams only).
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB as _LIB_PATH, build  # noqa: F401

TILES_OK = 0
STATUS_NAMES = {0: "TILES_OK", -1: "TILES_ERR_INVALID_ARG", -2: "TILES_ERR_UNSUPPORTED",
                -3: "TILES_ERR_PLAN_INVALID", -4: "TILES_ERR_DEVICE_MISMATCH",
                -5: "TILES_ERR_CAPACITY", -6: "TILES_ERR_CUDA", -7: "TILES_ERR_TIMEOUT",
                -8: "TILES_ERR_DEVICE_BOUNDS"}
SCHED_WAVES, SCHED_COUNTERS, SCHED_FLAGS = 0, 1, 2
FLAG_INJECT_STALL = 1  # test hook: CTA 0's first wait is never met (the launch times out)
WEIGHTS_BF16, WEIGHTS_INT8 = 0, 1
KV_BF16, KV_INT8 = 0, 1
OPS = {1: "QKV", 2: "ATTN", 3: "COMBINE", 4: "OPROJ", 5: "GATEUP", 6: "DOWN", 7: "LMHEAD",
       8: "SYNC"}
NO_COUNTER = 0xFFFF


class TilesError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}"
                         f" ({_lib().tiles_status_string(status).decode()})")


class ModelDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                 "max_pos", "qk_norm", "rope_scaling", "tied_embeddings", "rs_orig_max")] + \
               [(n, ctypes.c_double) for n in ("rope_theta", "rs_factor", "rs_low", "rs_high")] + \
               [("rms_eps", ctypes.c_float)]

    @classmethod
    def from_config(cls, cfg) -> "ModelDesc":
        """From any object with the model-shape attributes (e.g. synthetic.ModelConfig)."""
        return cls(n_layers=cfg.n_layers, hidden=cfg.hidden, n_q_heads=cfg.n_q_heads,
                   n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim, ffn=cfg.ffn,
                   vocab=cfg.vocab, max_pos=cfg.max_pos, qk_norm=int(cfg.qk_norm),
                   rope_scaling=int(cfg.rope_scaling), tied_embeddings=1,
                   rs_orig_max=int(cfg.rs_orig_max), rope_theta=float(cfg.rope_theta),
                   rs_factor=float(cfg.rs_factor), rs_low=float(cfg.rs_low),
                   rs_high=float(cfg.rs_high), rms_eps=float(cfg.rms_eps))


LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "ffn_norm", "w_gate",
                "w_up", "w_down")


# Layer tensors a plan reads after tiles_plan_create returns, per weight format.
_NORMS = ("attn_norm", "q_norm", "k_norm", "ffn_norm")
_PLAN_READS_LATER = {WEIGHTS_BF16: _NORMS + ("wo", "w_down"), WEIGHTS_INT8: _NORMS}


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in LAYER_FIELDS]


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("layers", ctypes.POINTER(LayerWeights))]


class PlanOpts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("scheduler", "n_ctas", "slot_bytes", "ring_slots", "kv_splits", "timeout_ms",
                 "l2_prefetch_kb", "l2_prefetch_gbs", "weight_format")] + \
               [("flags", ctypes.c_uint32), ("kv_format", ctypes.c_int32)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_ctas", "threads_per_cta", "smem_bytes", "slot_bytes", "ring_slots",
                 "kv_splits", "scheduler", "n_tasks", "n_counters", "phases_per_step",
                 "max_tasks_per_cta", "kv_block", "attn_tensor_cores")] + \
               [("rows_per_chunk", ctypes.c_int32 * 5), ("weight_format", ctypes.c_int32),
                ("kv_format", ctypes.c_int32)] + \
               [(n, ctypes.c_int64) for n in
                ("weight_bytes_per_token", "max_cta_bytes", "min_cta_bytes")]

    def as_dict(self):
        d = {n: getattr(self, n) for n, _ in self._fields_}
        d["rows_per_chunk"] = dict(zip(("qkv", "o", "gateup", "down", "lm"), self.rows_per_chunk))
        return d


class KV8Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("k_bytes", "v_bytes", "k_scale_off", "k_mu_off", "v_scale_off")] + \
               [("pos_stride", ctypes.c_int32)]


class Task(ctypes.Structure):
    _fields_ = [("op", ctypes.c_uint8), ("phase_kind", ctypes.c_uint8), ("layer", ctypes.c_uint16),
                ("begin", ctypes.c_uint32), ("end", ctypes.c_uint32),
                ("wait_ctr", ctypes.c_uint16), ("signal_ctr", ctypes.c_uint16),
                ("wait_mul", ctypes.c_uint32), ("wait_add", ctypes.c_uint32)]


assert ctypes.sizeof(Task) == 24

# every function declared in include/tiles.h
EXPORTS = ("tiles_plan_create", "tiles_plan_destroy", "tiles_decode", "tiles_decode_host",
           "tiles_status", "tiles_status_string", "tiles_plan_get_info", "tiles_schedule_build",
           "tiles_schedule_validate", "tiles_schedule_tasks", "tiles_schedule_cta_bytes",
           "tiles_schedule_destroy", "tiles_copy_bw", "tiles_barrier_cost", "tiles_plan_set_trace",
           "tiles_decode_noalloc", "tiles_quantize_rows_int8", "tiles_schedule_get_info",
           "tiles_forward", "tiles_verify", "tiles_kv8_get_layout", "tiles_kv8_from_bf16")
MAX_FORWARD_TOKENS = 256

_lib_handle = None


def _lib():
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing: build it first "
                              "(python -m tile_scheduled_persistent_gb300.build)")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
        st = ctypes.c_int
        L.tiles_plan_create.argtypes = [ctypes.POINTER(ModelDesc), ctypes.POINTER(Weights),
                                        ctypes.POINTER(PlanOpts), ctypes.POINTER(vp)]
        L.tiles_plan_create.restype = st
        L.tiles_plan_destroy.argtypes = [vp]
        L.tiles_plan_destroy.restype = None
        L.tiles_decode.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.tiles_decode.restype = st
        L.tiles_decode_host.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.tiles_decode_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.tiles_decode_noalloc.restype = st
        L.tiles_decode_host.restype = st
        L.tiles_forward.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp]
        L.tiles_forward.restype = st
        L.tiles_verify.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, vp, vp]
        L.tiles_verify.restype = st
        L.tiles_status.argtypes = [vp, vp]
        L.tiles_status.restype = st
        L.tiles_status_string.argtypes = [st]
        L.tiles_status_string.restype = ctypes.c_char_p
        L.tiles_plan_set_trace.argtypes = [vp, vp, i32]
        L.tiles_plan_set_trace.restype = st
        L.tiles_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        L.tiles_plan_get_info.restype = st
        L.tiles_schedule_build.argtypes = [ctypes.POINTER(ModelDesc), ctypes.POINTER(PlanOpts), i32,
                                           ctypes.POINTER(vp)]
        L.tiles_schedule_build.restype = st
        L.tiles_schedule_validate.argtypes = [vp, ctypes.c_char_p, ctypes.c_size_t]
        L.tiles_schedule_validate.restype = st
        L.tiles_schedule_tasks.argtypes = [vp, ctypes.POINTER(ctypes.POINTER(Task)),
                                           ctypes.POINTER(i32), ctypes.POINTER(ctypes.POINTER(i32)),
                                           ctypes.POINTER(i32)]
        L.tiles_schedule_tasks.restype = st
        L.tiles_schedule_cta_bytes.argtypes = [vp, i32, ctypes.POINTER(i64)]
        L.tiles_schedule_cta_bytes.restype = st
        L.tiles_schedule_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        L.tiles_schedule_get_info.restype = st
        L.tiles_schedule_destroy.argtypes = [vp]
        L.tiles_schedule_destroy.restype = None
        L.tiles_copy_bw.argtypes = [vp, vp, ctypes.c_size_t, i32, vp]
        L.tiles_copy_bw.restype = st
        L.tiles_quantize_rows_int8.argtypes = [vp, i32, i32, vp, vp, vp]
        L.tiles_quantize_rows_int8.restype = st
        L.tiles_kv8_get_layout.argtypes = [ctypes.POINTER(ModelDesc), ctypes.POINTER(KV8Layout)]
        L.tiles_kv8_get_layout.restype = st
        L.tiles_kv8_from_bf16.argtypes = [ctypes.POINTER(ModelDesc), vp, vp, i32, vp, vp, vp]
        L.tiles_kv8_from_bf16.restype = st
        L.tiles_barrier_cost.argtypes = [i32, i32, ctypes.POINTER(ctypes.c_double)]
        L.tiles_barrier_cost.restype = st
        _lib_handle = L
        del u32
    return _lib_handle


def lib():
    return _lib()


def _check(status: int, what: str):
    if status != TILES_OK:
        raise TilesError(status, what)


def make_opts(scheduler=SCHED_FLAGS, n_ctas=0, slot_bytes=0, ring_slots=0, kv_splits=0,
              timeout_ms=0, l2_prefetch_kb=0, l2_prefetch_gbs=0, flags=0,
              weight_format=0, kv_format=0) -> PlanOpts:
    return PlanOpts(scheduler=scheduler, n_ctas=n_ctas, slot_bytes=slot_bytes,
                    ring_slots=ring_slots, kv_splits=kv_splits, timeout_ms=timeout_ms,
                    l2_prefetch_kb=l2_prefetch_kb, l2_prefetch_gbs=l2_prefetch_gbs, flags=flags,
                    weight_format=weight_format, kv_format=kv_format)


# ------------------------------------------------------------------ INT8 KV cache
def kv8_layout(desc: ModelDesc) -> dict:
    """Sizes and offsets of the two buffers of an INT8 KV cache (no GPU)."""
    lay = KV8Layout()
    _check(_lib().tiles_kv8_get_layout(ctypes.byref(desc), ctypes.byref(lay)), "tiles_kv8_get_layout")
    return {n: getattr(lay, n) for n, _ in lay._fields_}


class KV8Cache:
    """The two device buffers of an INT8 KV cache (uint8 CUDA tensors k, v),
    laid out as tiles_kv8_get_layout states. ``from_bf16`` fills the prefilled
    positions from BF16 caches; ``host()`` returns the parts as numpy arrays."""

    def __init__(self, desc: ModelDesc, device="cuda"):
        import torch
        self.desc = desc
        self.layout = kv8_layout(desc)
        self.k = torch.zeros(self.layout["k_bytes"], dtype=torch.uint8, device=device)
        self.v = torch.zeros(self.layout["v_bytes"], dtype=torch.uint8, device=device)

    def from_bf16(self, k_cache, v_cache, n_pos: int, stream=None) -> "KV8Cache":
        _check(_lib().tiles_kv8_from_bf16(ctypes.byref(self.desc), _ptr(k_cache), _ptr(v_cache), int(n_pos),
                                          _ptr(self.k), _ptr(self.v), _stream_ptr(stream)), "tiles_kv8_from_bf16")
        return self

    def host(self) -> dict:
        """kq [Z][MP][d] int8, vq [Z][d][MP] int8, ks / vs [Z][MP] float32, mu [Z][d] float32
        (Z = n_layers * n_kv_heads, MP = pos_stride)."""
        import numpy as np
        d, lay = self.desc, self.layout
        Z, mp, hd = d.n_layers * d.n_kv_heads, lay["pos_stride"], d.head_dim
        kb, vb = self.k.cpu().numpy(), self.v.cpu().numpy()

        def part(buf, off, n, dt, shape):
            return np.frombuffer(buf[off:off + n * np.dtype(dt).itemsize].tobytes(), dt).reshape(shape)
        return {"kq": part(kb, 0, Z * mp * hd, np.int8, (Z, mp, hd)),
                "ks": part(kb, lay["k_scale_off"], Z * mp, np.float32, (Z, mp)),
                "mu": part(kb, lay["k_mu_off"], Z * hd, np.float32, (Z, hd)),
                "vq": part(vb, 0, Z * hd * mp, np.int8, (Z, hd, mp)),
                "vs": part(vb, lay["v_scale_off"], Z * mp, np.float32, (Z, mp))}


# ------------------------------------------------------------------ schedule (host only)
class Schedule:
    """The planner's schedule for a model on n_ctas CTAs, without a GPU."""

    def __init__(self, desc: ModelDesc, n_ctas: int, opts: PlanOpts | None = None):
        h = ctypes.c_void_p()
        self._desc = desc
        _check(_lib().tiles_schedule_build(ctypes.byref(desc),
                                           ctypes.byref(opts) if opts is not None else None,
                                           n_ctas, ctypes.byref(h)), "tiles_schedule_build")
        self._h = h

    def validate(self):
        buf = ctypes.create_string_buffer(256)
        st = _lib().tiles_schedule_validate(self._h, buf, 256)
        return st, buf.value.decode()

    def tasks(self):
        """(tasks ctypes array view, offsets list). Mutating the view mutates the schedule."""
        tp = ctypes.POINTER(Task)()
        n = ctypes.c_int32()
        off = ctypes.POINTER(ctypes.c_int32)()
        nc = ctypes.c_int32()
        _check(_lib().tiles_schedule_tasks(self._h, ctypes.byref(tp), ctypes.byref(n),
                                           ctypes.byref(off), ctypes.byref(nc)), "tiles_schedule_tasks")
        arr = ctypes.cast(tp, ctypes.POINTER(Task * n.value)).contents
        return arr, [off[i] for i in range(nc.value + 1)]

    def info(self) -> dict:
        """The facts a plan made from this schedule would report (no GPU)."""
        inf = PlanInfo()
        _check(_lib().tiles_schedule_get_info(self._h, ctypes.byref(inf)), "tiles_schedule_get_info")
        return inf.as_dict()

    def cta_bytes(self, pos: int):
        n = self.tasks()[1]
        out = (ctypes.c_int64 * (len(n) - 1))()
        _check(_lib().tiles_schedule_cta_bytes(self._h, pos, out), "tiles_schedule_cta_bytes")
        return list(out)

    def close(self):
        if self._h:
            _lib().tiles_schedule_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------------ plans (GPU)
def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """A validated, uploaded schedule bound to device weights.

    ``weights``: dict with 'embed', 'final_norm' and 'layers' (a list of dicts
    keyed by LAYER_FIELDS) of CUDA tensors holding bf16 bit patterns, row-major
    [out][in]. The plan packs its own copies of wq/wk/wv and w_gate/w_up (with
    INT8 weights, of every GEMV matrix), so it keeps references only to the
    tensors the kernel still reads: the embedding, the norm gains and, for BF16,
    wo and w_down. The caller may drop the others once the plan exists."""

    def __init__(self, desc: ModelDesc, weights: dict, opts: PlanOpts | None = None):
        self.desc = desc
        read_later = _PLAN_READS_LATER[int(opts.weight_format) if opts is not None else WEIGHTS_BF16]
        self._keep = {"embed": weights["embed"], "final_norm": weights["final_norm"],
                      "layers": [{f: lw.get(f) for f in read_later} for lw in weights["layers"]]}
        n = desc.n_layers
        self._layers = (LayerWeights * n)()
        for l, lw in enumerate(weights["layers"]):
            for f in LAYER_FIELDS:
                t = lw.get(f)
                setattr(self._layers[l], f, None if t is None else t.data_ptr())
        self._w = Weights(embed=weights["embed"].data_ptr(),
                          final_norm=weights["final_norm"].data_ptr(),
                          layers=ctypes.cast(self._layers, ctypes.POINTER(LayerWeights)))
        h = ctypes.c_void_p()
        _check(_lib().tiles_plan_create(ctypes.byref(desc), ctypes.byref(self._w),
                                        ctypes.byref(opts) if opts is not None else None,
                                        ctypes.byref(h)), "tiles_plan_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def info(self) -> dict:
        inf = PlanInfo()
        _check(_lib().tiles_plan_get_info(self._h, ctypes.byref(inf)), "tiles_plan_get_info")
        return inf.as_dict()

    def set_trace(self, buf, steps: int) -> None:
        """Record a per-task timeline of the first `steps` steps of later decodes into
        `buf` (int64 CUDA tensor of n_ctas * steps * max_tasks_per_cta * 16 words)."""
        _check(_lib().tiles_plan_set_trace(self._h, _ptr(buf), steps), "tiles_plan_set_trace")

    def decode(self, k_cache, v_cache, prompt, start_pos: int, n_new: int, out_tokens,
               out_logits=None, stream=None) -> None:
        """Asynchronous greedy decode on `stream` (default: torch's current stream).
        prompt/out_tokens int32 CUDA tensors; out_logits float32 [steps][vocab] or None."""
        _check(_lib().tiles_decode(self._h, _ptr(k_cache), _ptr(v_cache), _ptr(prompt),
                                   int(prompt.numel()), start_pos, n_new, _stream_ptr(stream),
                                   _ptr(out_tokens), _ptr(out_logits)), "tiles_decode")

    def decode_noalloc(self, k_cache, v_cache, prompt, start_pos: int, n_new: int, out_tokens,
                       out_logits=None, stream=None) -> None:
        """Same as decode, but the kernel's working memory comes from the library's
        fixed 1 MiB device array instead of the plan's buffers (nothing is allocated;
        calls that overlap on the GPU must not share it)."""
        _check(_lib().tiles_decode_noalloc(self._h, _ptr(k_cache), _ptr(v_cache), _ptr(prompt),
                                           int(prompt.numel()), start_pos, n_new,
                                           _stream_ptr(stream), _ptr(out_tokens), _ptr(out_logits)),
               "tiles_decode_noalloc")

    def decode_host(self, k_cache, v_cache, prompt_np, start_pos: int, n_new: int,
                    out_tokens_np, out_logits_np=None, stream=None) -> None:
        """Same, with numpy host buffers; copies in and out and synchronises."""
        assert prompt_np.dtype.name == "int32" and out_tokens_np.dtype.name == "int32"
        _check(_lib().tiles_decode_host(
            self._h, _ptr(k_cache), _ptr(v_cache), prompt_np.ctypes.data_as(ctypes.c_void_p),
            int(prompt_np.size), start_pos, n_new, _stream_ptr(stream),
            out_tokens_np.ctypes.data_as(ctypes.c_void_p),
            None if out_logits_np is None else out_logits_np.ctypes.data_as(ctypes.c_void_p)),
            "tiles_decode_host")

    def forward(self, k_cache, v_cache, tokens, start_pos: int, out_argmax, out_logits=None,
                stream=None) -> None:
        """Runs the int32 CUDA tensor `tokens` through the model at positions start_pos..
        in passes of up to MAX_FORWARD_TOKENS (K/V written); out_argmax int32 [n] gets the
        greedy token after each input, out_logits float32 [n][vocab] (or None) the logits."""
        _check(_lib().tiles_forward(self._h, _ptr(k_cache), _ptr(v_cache), _ptr(tokens),
                                    int(tokens.numel()), start_pos, _stream_ptr(stream),
                                    _ptr(out_argmax), _ptr(out_logits)), "tiles_forward")

    def verify(self, k_cache, v_cache, inputs, start_pos: int, out_tokens, out_n_accepted,
               out_logits=None, stream=None) -> None:
        """One greedy verify step: inputs = [last token, d_1 .. d_k] (int32 CUDA tensor) at
        positions start_pos..; out_tokens int32 [k + 1] gets the accepted drafts and the
        model's next token, out_n_accepted int32 [1] the number of accepted drafts."""
        _check(_lib().tiles_verify(self._h, _ptr(k_cache), _ptr(v_cache), _ptr(inputs),
                                   int(inputs.numel()) - 1, start_pos, _stream_ptr(stream),
                                   _ptr(out_tokens), _ptr(out_n_accepted), _ptr(out_logits)),
               "tiles_verify")

    def status(self, stream=None) -> int:
        return _lib().tiles_status(self._h, _stream_ptr(stream))

    def check(self, stream=None):
        _check(self.status(stream), "tiles_status")

    def close(self):
        if getattr(self, "_h", None):
            _lib().tiles_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def quantize_rows_int8(w_bf16, stream=None):
    """Weight-only INT8 of a [rows][cols] BF16 CUDA tensor on the device (the
    kernel plans use): (codes int8 [rows][cols], scales float32 [rows])."""
    import torch
    assert w_bf16.is_cuda and w_bf16.dtype == torch.bfloat16 and w_bf16.dim() == 2
    w = w_bf16.contiguous()
    codes = torch.empty(w.shape, dtype=torch.int8, device=w.device)
    scales = torch.empty(w.shape[0], dtype=torch.float32, device=w.device)
    _check(_lib().tiles_quantize_rows_int8(_ptr(w), w.shape[0], w.shape[1], _ptr(codes), _ptr(scales),
                                           _stream_ptr(stream)), "tiles_quantize_rows_int8")
    return codes, scales


def copy_bw(dst, src, n_ctas: int = 0, stream=None) -> None:
    _check(_lib().tiles_copy_bw(_ptr(dst), _ptr(src), dst.numel() * dst.element_size(), n_ctas,
                                _stream_ptr(stream)), "tiles_copy_bw")


def barrier_cost(n_ctas: int = 0, rounds: int = 1000) -> float:
    ns = ctypes.c_double()
    _check(_lib().tiles_barrier_cost(n_ctas, rounds, ctypes.byref(ns)), "tiles_barrier_cost")
    return ns.value


# ------------------------------------------------------------------ helpers for bf16 arrays
def to_device_bf16(arr, device="cuda"):
    """numpy uint16 (bf16 bit patterns) -> CUDA tensor of dtype bfloat16 (bitwise copy)."""
    import numpy as np
    import torch
    a = np.ascontiguousarray(arr).view(np.int16)
    return torch.from_numpy(a).view(torch.bfloat16).to(device)


def upload_weights(model_weights, device="cuda") -> dict:
    """synthetic.ModelWeights-like object (numpy bf16 bit patterns) -> dict of CUDA tensors."""
    out = {"embed": to_device_bf16(model_weights.embed, device),
           "final_norm": to_device_bf16(model_weights.final_norm, device), "layers": []}
    for lw in model_weights.layers:
        out["layers"].append({k: (None if v is None else to_device_bf16(v, device))
                              for k, v in lw.items()})
    return out
