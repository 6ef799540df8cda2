"""Python binding of the qd C-ABI (``include/qd.h``): argument marshalling only.

Every step of the decode path runs in the CUDA kernels of ``libqd.so``; this
module converts Python/torch arguments into the C types the library takes.
PyTorch serves only to hold device memory and to name the caller's stream.
There is no fallback: importing fails loudly when ``libqd.so`` has not been
built (``python -c "import __graft_entry__ as g; g.build()"``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
# QD_LIBRARY names another build of the same library (the phase-timeline build of
# step_timeline.py); by default the in-tree libqd.so.
LIB_PATH = os.environ.get("QD_LIBRARY") or os.path.join(_PKG, "libqd.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                      "(transformer_autoregressive_decode_gb300.build.build())")

_lib = ctypes.CDLL(LIB_PATH)

QD_OK, QD_EINVAL, QD_ESTATE, QD_EKVFULL, QD_ENOMEM, QD_ECUDA, QD_EUNSUPPORTED, QD_EDEVICE = 0, -1, -2, -3, -4, -5, -6, -7
QD_F32, QD_BF16 = 0, 1
QD_MAX_BUCKETS = 8
QD_MAX_HEADS = 16
QD_FRAME_CODES = 16

# Every symbol the header declares (tests check the library exports each one).
EXPORTS = ("qd_create", "qd_destroy", "qd_reset", "qd_prefill", "qd_prefill_mrope", "qd_decode_step", "qd_decode_step_async",
           "qd_decode_greedy", "qd_grow_kv", "qd_get_hidden", "qd_set_debug_taps", "qd_set_graphs", "qd_set_sampling", "qd_copy_kv",
           "qd_get_emitted", "qd_get_pos", "qd_get_launch_count", "qd_time_kernel", "qd_last_error",
           "qd_status_string", "qd_head_argmax_noalloc", "qd_frame_create", "qd_frame_destroy",
           "qd_frame_generate", "qd_frame_set_graphs", "qd_gemm_bf16", "qd_quantize_q8", "qd_gemv_q8",
           "qd_quantize_q4k", "qd_gemv_q4k",
           "qd_conv1d_causal", "qd_conv_transpose1d_causal", "qd_conv1d_causal_tc",
           "qd_conv_transpose1d_causal_tc", "qd_batch_create", "qd_batch_destroy",
           "qd_batch_set_stream", "qd_batch_decode", "qd_batch_sync", "qd_batch_get_logits", "qd_batch_copy_kv",
           "qd_batch_get_pos", "qd_batch_get_launch_count", "qd_batch_set_graphs", "qd_batch_time_kernel", "qd_batch_prefill",
           "qd_batch_set_sampling")


class qd_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "embed_rows", "dtype",
        "qk_norm", "n_heads_out", "eos_mask_id", "n_buckets")] + [
        ("buckets", ctypes.c_int * QD_MAX_BUCKETS),
        ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double), ("rep_penalty", ctypes.c_double),
        ("mrope_section", ctypes.c_int * 3), ("weight_q8", ctypes.c_int)]


class qd_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "mlp_norm", "wg", "wu", "wd")]


class qd_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p * QD_MAX_HEADS), ("layers", ctypes.POINTER(qd_layer_weights))]


_vp, _i32, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
_P = ctypes.POINTER
_SIGS = {
    "qd_create": ([_P(qd_weights), _P(qd_config), _vp, _P(_vp)], _i32),
    "qd_destroy": ([_vp], _i32),
    "qd_reset": ([_vp], _i32),
    "qd_prefill": ([_vp, _vp, _vp, _i32, _i32, _P(ctypes.c_int32)], _i32),
    "qd_prefill_mrope": ([_vp, _vp, _vp, _i32, _i32, _vp, _P(ctypes.c_int32)], _i32),
    "qd_decode_step": ([_vp, _vp, ctypes.c_int32, _i32, _P(ctypes.c_int32)], _i32),
    "qd_decode_step_async": ([_vp, _vp, _vp, _i32, _vp], _i32),
    "qd_decode_greedy": ([_vp, _i32, ctypes.c_int32, _vp], _i32),
    "qd_grow_kv": ([_vp, _i32], _i32),
    "qd_get_hidden": ([_vp, _vp], _i32),
    "qd_set_debug_taps": ([_vp, _vp, _vp], _i32),
    "qd_set_graphs": ([_vp, _i32], _i32),
    "qd_set_sampling": ([_vp, _i32, ctypes.c_float, ctypes.c_float, ctypes.c_uint64], _i32),
    "qd_copy_kv": ([_vp, _vp, _P(_sz)], _i32),
    "qd_get_emitted": ([_vp, _vp], _i32),
    "qd_get_pos": ([_vp, _P(_i32), _P(_i32)], _i32),
    "qd_get_launch_count": ([_vp, _P(_i64), _P(_i32)], _i32),
    "qd_time_kernel": ([_vp, _i32, _i32, _P(ctypes.c_float)], _i32),
    "qd_last_error": ([_vp], ctypes.c_char_p),
    "qd_status_string": ([_i32], ctypes.c_char_p),
    "qd_head_argmax_noalloc": ([_vp, _vp, _i32, _i32, _i32, _vp, ctypes.c_double, _i32, _vp, _vp, _vp], _i32),
    "qd_frame_create": ([_vp, _vp, _P(_vp), _i32, _i32, _P(_vp)], _i32),
    "qd_frame_destroy": ([_vp], _i32),
    "qd_frame_generate": ([_vp, _i32, _vp, _vp, _vp, _vp], _i32),
    "qd_frame_set_graphs": ([_vp, _i32], _i32),
    "qd_gemm_bf16": ([_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _P(ctypes.c_float)], _i32),
    "qd_quantize_q8": ([_vp, _i32, _i32, _i32, _vp, _vp, _vp], _i32),
    "qd_conv1d_causal": ([_vp, _i32, _i32, _vp, _vp, _i32, _i32, _i32, _vp, _vp], _i32),
    "qd_conv_transpose1d_causal": ([_vp, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _vp], _i32),
    "qd_conv1d_causal_tc": ([_vp, _i32, _i32, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp], _i32),
    "qd_conv_transpose1d_causal_tc": ([_vp, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _i32, _vp], _i32),
    "qd_gemv_q8": ([_vp, _vp, _vp, _vp, _i32, _i32, _vp, _i32, _P(ctypes.c_float)], _i32),
    "qd_quantize_q4k": ([_vp, _i32, _i32, _i32, _vp, _vp], _i32),
    "qd_gemv_q4k": ([_vp, _vp, _vp, _i32, _i32, _vp, _i32, _P(ctypes.c_float)], _i32),
    "qd_batch_create": ([_vp, _i32, _i32, _P(_vp)], _i32),
    "qd_batch_destroy": ([_vp], _i32),
    "qd_batch_set_stream": ([_vp, _i32, _vp, _i32, ctypes.c_int32], _i32),
    "qd_batch_decode": ([_vp, _i32, _vp, _vp], _i32),
    "qd_batch_set_sampling": ([_vp, _i32, ctypes.c_float, ctypes.c_float, ctypes.c_uint64], _i32),
    "qd_batch_sync": ([_vp], _i32),
    "qd_batch_get_logits": ([_vp, _vp], _i32),
    "qd_batch_copy_kv": ([_vp, _i32, _vp, _P(_sz)], _i32),
    "qd_batch_get_pos": ([_vp, _i32, _P(_i32)], _i32),
    "qd_batch_get_launch_count": ([_vp, _P(_i64), _P(_i32)], _i32),
    "qd_batch_set_graphs": ([_vp, _i32], _i32),
    "qd_batch_time_kernel": ([_vp, _i32, _i32, _P(ctypes.c_float)], _i32),
    "qd_batch_prefill": ([_vp, _vp, _i32, _vp, _i32, _vp], _i32),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res


class QDError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_lib.qd_status_string(status).decode()}: {message}")
        self.status = status


def _ptr(t) -> Optional[int]:
    """Device address of a torch tensor (or None)."""
    if t is None:
        return None
    return t.data_ptr()


class Handle:
    """Owns a ``qd_handle``; destroyed with the object or by ``qd_destroy``."""

    def __init__(self, h: int, cfg: qd_config):
        self.h = h
        self.cfg = cfg

    def __del__(self):
        try:
            qd_destroy(self)
        except Exception:
            pass


def _check(h: Optional[Handle], st: int):
    if st != QD_OK:
        msg = _lib.qd_last_error(h.h if h is not None else None).decode(errors="replace") if h is not None else ""
        raise QDError(st, msg)


def make_config(hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab, embed_rows, bf16, qk_norm,
                n_heads_out=1, eos_mask_id=-1, buckets: Sequence[int] = (128,), rms_eps=1e-6, rope_theta=1e6,
                rep_penalty=1.0, mrope_section: Sequence[int] = (0, 0, 0), weight_q8: bool = False) -> qd_config:
    c = qd_config()
    c.hidden, c.n_layers, c.n_q_heads, c.n_kv_heads = hidden, n_layers, n_q_heads, n_kv_heads
    c.head_dim, c.ffn, c.vocab, c.embed_rows = head_dim, ffn, vocab, embed_rows
    c.dtype = QD_BF16 if bf16 else QD_F32
    c.qk_norm, c.n_heads_out, c.eos_mask_id = int(qk_norm), n_heads_out, eos_mask_id
    c.n_buckets = len(buckets)
    for i, b in enumerate(buckets):
        c.buckets[i] = b
    c.rms_eps, c.rope_theta, c.rep_penalty = rms_eps, rope_theta, rep_penalty
    for i, v in enumerate(mrope_section):
        c.mrope_section[i] = int(v)
    c.weight_q8 = int(bool(weight_q8))
    return c


LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "mlp_norm", "wg", "wu", "wd")


def qd_create(weights: Dict[str, "torch.Tensor"], cfg: qd_config, stream=None) -> Handle:
    """weights: device tensors keyed ``embed``, ``final_norm``, ``lm_head.{j}``,
    ``layers.{l}.{name}``.  ``stream``: a torch.cuda.Stream (default: current)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    w = qd_weights()
    w.embed = _ptr(weights.get("embed"))
    w.final_norm = _ptr(weights["final_norm"])
    for j in range(cfg.n_heads_out):
        w.lm_head[j] = _ptr(weights[f"lm_head.{j}"])
    layers = (qd_layer_weights * cfg.n_layers)()
    for l in range(cfg.n_layers):
        for k in LAYER_KEYS:
            setattr(layers[l], k, _ptr(weights.get(f"layers.{l}.{k}")))
    w.layers = layers
    out = ctypes.c_void_p()
    st = _lib.qd_create(ctypes.byref(w), ctypes.byref(cfg), ctypes.c_void_p(stream.cuda_stream), ctypes.byref(out))
    if st != QD_OK:
        raise QDError(st, "qd_create failed")
    return Handle(out.value, cfg)


def qd_destroy(h: Handle):
    if h is not None and h.h:
        _lib.qd_destroy(h.h)
        h.h = None


def qd_reset(h: Handle):
    _check(h, _lib.qd_reset(h.h))


def qd_prefill(h: Handle, tokens=None, embeds=None, head_idx: int = 0) -> int:
    """tokens: host int sequence; embeds: device fp32 tensor [n, hidden]."""
    fid = ctypes.c_int32(-1)
    if tokens is not None:
        arr = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        _check(h, _lib.qd_prefill(h.h, arr.ctypes.data, None, len(arr), head_idx, ctypes.byref(fid)))
    else:
        n = embeds.shape[0] if embeds is not None else 0
        _check(h, _lib.qd_prefill(h.h, None, _ptr(embeds), n, head_idx, ctypes.byref(fid)))
    return fid.value


def qd_prefill_mrope(h: Handle, positions, tokens=None, embeds=None, head_idx: int = 0) -> int:
    """qd_prefill with rotary positions: host int array [3, n] (t, h, w streams)."""
    fid = ctypes.c_int32(-1)
    n = len(tokens) if tokens is not None else (embeds.shape[0] if embeds is not None else 0)
    pos = np.ascontiguousarray(np.asarray(positions, dtype=np.int32))
    if pos.shape != (3, n):
        raise ValueError(f"positions must be [3, {n}], got {pos.shape}")
    if tokens is not None:
        arr = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        _check(h, _lib.qd_prefill_mrope(h.h, arr.ctypes.data, None, n, head_idx, pos.ctypes.data, ctypes.byref(fid)))
    else:
        _check(h, _lib.qd_prefill_mrope(h.h, None, _ptr(embeds), n, head_idx, pos.ctypes.data, ctypes.byref(fid)))
    return fid.value


def qd_decode_step(h: Handle, embed=None, token: int = -1, head_idx: int = 0) -> int:
    oid = ctypes.c_int32(-1)
    _check(h, _lib.qd_decode_step(h.h, _ptr(embed), int(token), head_idx, ctypes.byref(oid)))
    return oid.value


def qd_decode_step_async(h: Handle, embed=None, token_dev=None, head_idx: int = 0, out_id_dev=None):
    _check(h, _lib.qd_decode_step_async(h.h, _ptr(embed), _ptr(token_dev), head_idx, _ptr(out_id_dev)))


def qd_decode_greedy(h: Handle, n_steps: int, first_token: int, ids_dev):
    _check(h, _lib.qd_decode_greedy(h.h, int(n_steps), int(first_token), _ptr(ids_dev)))


def qd_grow_kv(h: Handle, new_smax: int):
    _check(h, _lib.qd_grow_kv(h.h, int(new_smax)))


def qd_get_hidden(h: Handle, out_dev):
    _check(h, _lib.qd_get_hidden(h.h, _ptr(out_dev)))


def qd_set_debug_taps(h: Handle, hidden_dev=None, logits_dev=None):
    _check(h, _lib.qd_set_debug_taps(h.h, _ptr(hidden_dev), _ptr(logits_dev)))


def qd_set_sampling(h: Handle, top_k: int, temperature: float = 1.0, top_p: float = 1.0, seed: int = 0):
    """Sample the heads' ids (top_k 0: greedy argmax); see qd_set_sampling in qd.h."""
    _check(h, _lib.qd_set_sampling(h.h, int(top_k), float(temperature), float(top_p), int(seed)))


def qd_set_graphs(h: Handle, enable: bool):
    _check(h, _lib.qd_set_graphs(h.h, int(bool(enable))))


def qd_copy_kv(h: Handle, dst_dev=None) -> int:
    n = ctypes.c_size_t(0 if dst_dev is None else dst_dev.numel() * dst_dev.element_size())
    _check(h, _lib.qd_copy_kv(h.h, _ptr(dst_dev), ctypes.byref(n)))
    return n.value


def qd_get_emitted(h: Handle, dst_dev):
    _check(h, _lib.qd_get_emitted(h.h, _ptr(dst_dev)))


def qd_get_pos(h: Handle):
    p, s = ctypes.c_int(0), ctypes.c_int(0)
    _check(h, _lib.qd_get_pos(h.h, ctypes.byref(p), ctypes.byref(s)))
    return p.value, s.value


def qd_get_launch_count(h: Handle):
    k, per = ctypes.c_longlong(0), ctypes.c_int(0)
    _check(h, _lib.qd_get_launch_count(h.h, ctypes.byref(k), ctypes.byref(per)))
    return k.value, per.value


def qd_time_kernel(h: Handle, which: int, reps: int) -> float:
    ms = ctypes.c_float(0.0)
    _check(h, _lib.qd_time_kernel(h.h, int(which), int(reps), ctypes.byref(ms)))
    return ms.value


def qd_last_error(h: Handle) -> str:
    return _lib.qd_last_error(h.h).decode(errors="replace")


def qd_status_string(status: int) -> str:
    return _lib.qd_status_string(int(status)).decode()


KERNEL_HEAD, KERNEL_QKV, KERNEL_GATE_UP, KERNEL_DOWN, KERNEL_ATTENTION, KERNEL_OPROJ, KERNEL_STEP = 0, 1, 2, 3, 4, 5, 6


def qd_head_argmax_noalloc(y_dev, w_dev, vocab: int, hidden: int, bf16: bool, emitted_dev, rep_penalty: float,
                           eos_mask_id: int, out_id_dev, logits_dev=None, stream=None):
    """Output head over device buffers the caller owns; allocates nothing."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    st = _lib.qd_head_argmax_noalloc(_ptr(y_dev), _ptr(w_dev), int(vocab), int(hidden), QD_BF16 if bf16 else QD_F32,
                                     _ptr(emitted_dev), float(rep_penalty), int(eos_mask_id), _ptr(out_id_dev),
                                     _ptr(logits_dev), ctypes.c_void_p(stream.cuda_stream))
    if st != QD_OK:
        raise QDError(st, "qd_head_argmax_noalloc failed")


class FrameHandle:
    """Owns a ``qd_frame_handle``; keeps the two model handles alive while it exists.
    Errors of its calls are described by ``qd_last_error(talker)``."""

    def __init__(self, f: int, talker: Handle, predictor: Handle):
        self.f = f
        self.talker = talker
        self.predictor = predictor

    def __del__(self):
        try:
            qd_frame_destroy(self)
        except Exception:
            pass


def qd_frame_create(talker: Handle, predictor: Handle, code_tables: Sequence["torch.Tensor"], bf16: bool) -> FrameHandle:
    """code_tables: the 15 device tables E_1..E_15, each [code_rows, hidden]."""
    if len(code_tables) != QD_FRAME_CODES - 1:
        raise ValueError(f"need {QD_FRAME_CODES - 1} code tables")
    rows = int(code_tables[0].shape[0])
    arr = (ctypes.c_void_p * len(code_tables))(*[_ptr(t) for t in code_tables])
    out = ctypes.c_void_p()
    _check(talker, _lib.qd_frame_create(talker.h, predictor.h, arr, rows, QD_BF16 if bf16 else QD_F32,
                                        ctypes.byref(out)))
    return FrameHandle(out.value, talker, predictor)


def qd_frame_destroy(f: FrameHandle):
    if f is not None and f.f:
        _lib.qd_frame_destroy(f.f)
        f.f = None


def qd_frame_set_graphs(f: FrameHandle, enable: bool):
    _check(f.talker, _lib.qd_frame_set_graphs(f.f, int(bool(enable))))


def qd_frame_generate(f: FrameHandle, n_frames: int, text_dev, codes_dev, force_dev=None, next_in_dev=None):
    """text_dev fp32 [n_frames, hidden]; codes_dev int32 [n_frames, 16] (written);
    force_dev int32 [n_frames, 16] or None; next_in_dev fp32 [hidden] or None."""
    _check(f.talker, _lib.qd_frame_generate(f.f, int(n_frames), _ptr(text_dev), _ptr(force_dev), _ptr(codes_dev),
                                            _ptr(next_in_dev)))


GEMM_STORE, GEMM_RESIDUAL, GEMM_SWIGLU = 0, 1, 2


def qd_gemm_bf16(w_dev, x_dev, out_dev, mode: int = GEMM_STORE, stream=None, time_reps: int = 0):
    """out = x @ W^T on the tensor cores (W bf16 [R, K], x fp32 [T, K]); see qd.h.
    With time_reps > 0, returns the kernel's mean duration in ms over that many launches."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    R, K = int(w_dev.shape[0]), int(w_dev.shape[1])
    T = int(x_dev.shape[0])
    ms = ctypes.c_float(0.0)
    st = _lib.qd_gemm_bf16(_ptr(w_dev), _ptr(x_dev), _ptr(out_dev), R, K, T, int(mode),
                           ctypes.c_void_p(stream.cuda_stream), int(time_reps),
                           ctypes.byref(ms) if time_reps > 0 else None)
    if st != QD_OK:
        raise QDError(st, "qd_gemm_bf16 failed")
    return ms.value if time_reps > 0 else None


class BatchHandle:
    """Owns a ``qd_batch_handle``; keeps its model handle alive.  Errors are described
    by ``qd_last_error(model)``."""

    def __init__(self, b: int, model: Handle, n_streams: int, smax: int):
        self.b = b
        self.model = model
        self.n_streams = n_streams
        self.smax = smax

    def __del__(self):
        try:
            qd_batch_destroy(self)
        except Exception:
            pass


def qd_batch_create(model: Handle, n_streams: int, smax: int) -> BatchHandle:
    out = ctypes.c_void_p()
    _check(model, _lib.qd_batch_create(model.h, int(n_streams), int(smax), ctypes.byref(out)))
    return BatchHandle(out.value, model, n_streams, smax)


def qd_batch_destroy(b: BatchHandle):
    if b is not None and b.b:
        _lib.qd_batch_destroy(b.b)
        b.b = None


def qd_batch_set_stream(b: BatchHandle, stream: int, kv_dev, length: int, token: int):
    """kv_dev: device bf16 tensor [n_layers, 2, n_kv_heads, length, head_dim] (or None when length is 0)."""
    _check(b.model, _lib.qd_batch_set_stream(b.b, int(stream), _ptr(kv_dev), int(length), int(token)))


def qd_batch_set_sampling(b: BatchHandle, top_k: int, temperature: float, top_p: float, seed: int):
    _check(b.model, _lib.qd_batch_set_sampling(b.b, int(top_k), float(temperature), float(top_p), int(seed)))


def qd_batch_decode(b: BatchHandle, n_steps: int, ids_dev, force_dev=None):
    _check(b.model, _lib.qd_batch_decode(b.b, int(n_steps), _ptr(force_dev), _ptr(ids_dev)))


def qd_batch_sync(b: BatchHandle):
    _check(b.model, _lib.qd_batch_sync(b.b))


def qd_batch_get_logits(b: BatchHandle, dst_dev):
    _check(b.model, _lib.qd_batch_get_logits(b.b, _ptr(dst_dev)))


def qd_batch_copy_kv(b: BatchHandle, stream: int, dst_dev=None) -> int:
    n = ctypes.c_size_t(0 if dst_dev is None else dst_dev.numel() * dst_dev.element_size())
    _check(b.model, _lib.qd_batch_copy_kv(b.b, int(stream), _ptr(dst_dev), ctypes.byref(n)))
    return n.value


def qd_batch_get_pos(b: BatchHandle, stream: int) -> int:
    p = ctypes.c_int(0)
    _check(b.model, _lib.qd_batch_get_pos(b.b, int(stream), ctypes.byref(p)))
    return p.value


def qd_batch_get_launch_count(b: BatchHandle):
    k, per = ctypes.c_longlong(0), ctypes.c_int(0)
    _check(b.model, _lib.qd_batch_get_launch_count(b.b, ctypes.byref(k), ctypes.byref(per)))
    return k.value, per.value


def qd_batch_set_graphs(b: BatchHandle, enable: bool):
    _check(b.model, _lib.qd_batch_set_graphs(b.b, int(bool(enable))))


BATCH_ATTENTION, BATCH_QKV, BATCH_OPROJ, BATCH_GATE_UP, BATCH_DOWN, BATCH_HEAD = 1, 2, 3, 4, 5, 6


def qd_batch_time_kernel(b: BatchHandle, which: int, reps: int) -> float:
    ms = ctypes.c_float(0.0)
    _check(b.model, _lib.qd_batch_time_kernel(b.b, int(which), int(reps), ctypes.byref(ms)))
    return ms.value


def qd_batch_prefill(b: BatchHandle, streams, embeds_dev, first_ids_dev):
    """streams: host ints; embeds_dev: device fp32 [ns, n, hidden]; first_ids_dev: device int32 [ns]."""
    arr = np.ascontiguousarray(np.asarray(streams, dtype=np.int32))
    ns, n = int(embeds_dev.shape[0]), int(embeds_dev.shape[1])
    if len(arr) != ns:
        raise ValueError("one stream index per prompt")
    _check(b.model, _lib.qd_batch_prefill(b.b, arr.ctypes.data, ns, _ptr(embeds_dev), n, _ptr(first_ids_dev)))


def qd_quantize_q8(w_dev, codes_dev, scales_dev, stream=None):
    """Weight-only 8-bit block quantisation of the device matrix w_dev [rows, K] (fp32 or
    bf16) into codes_dev (int8 [rows, K]) and scales_dev (half bits, int16/uint16
    [rows, K/32])."""
    import torch
    rows, K = w_dev.shape
    s = (stream or torch.cuda.current_stream()).cuda_stream
    st = _lib.qd_quantize_q8(_ptr(w_dev), QD_BF16 if w_dev.dtype == torch.bfloat16 else QD_F32, rows, K,
                             _ptr(codes_dev), _ptr(scales_dev), s)
    if st != QD_OK:
        raise QDError(st, "qd_quantize_q8 failed")


def qd_gemv_q8(codes_dev, scales_dev, x_dev, y_dev, stream=None, time_reps: int = 0):
    """y = dequant(codes, scales) x on the device; returns the mean kernel time (ms) of
    ``time_reps`` extra launches, or None."""
    import torch
    rows, K = codes_dev.shape
    s = (stream or torch.cuda.current_stream()).cuda_stream
    ms = ctypes.c_float(0.0)
    st = _lib.qd_gemv_q8(_ptr(codes_dev), _ptr(scales_dev), _ptr(x_dev), _ptr(y_dev), rows, K, s, int(time_reps),
                         ctypes.byref(ms) if time_reps else None)
    if st != QD_OK:
        raise QDError(st, "qd_gemv_q8 failed")
    return ms.value if time_reps else None


def qd_quantize_q4k(w_dev, blocks_dev, stream=None):
    """Q4_K super-blocks of the device matrix w_dev [rows, K] (fp32 or bf16, K a multiple
    of 256) into blocks_dev (uint8 [rows, K/256, 144])."""
    import torch
    rows, K = w_dev.shape
    s = (stream or torch.cuda.current_stream()).cuda_stream
    st = _lib.qd_quantize_q4k(_ptr(w_dev), QD_BF16 if w_dev.dtype == torch.bfloat16 else QD_F32, rows, K,
                              _ptr(blocks_dev), s)
    if st != QD_OK:
        raise QDError(st, "qd_quantize_q4k failed")


def qd_gemv_q4k(blocks_dev, x_dev, y_dev, stream=None, time_reps: int = 0):
    """y = dequant(blocks) x on the device (blocks uint8 [rows, K/256, 144]); returns the
    mean kernel time (ms) of ``time_reps`` extra launches, or None."""
    import torch
    rows, nsb = int(blocks_dev.shape[0]), int(blocks_dev.shape[1])
    s = (stream or torch.cuda.current_stream()).cuda_stream
    ms = ctypes.c_float(0.0)
    st = _lib.qd_gemv_q4k(_ptr(blocks_dev), _ptr(x_dev), _ptr(y_dev), rows, nsb * 256, s, int(time_reps),
                          ctypes.byref(ms) if time_reps else None)
    if st != QD_OK:
        raise QDError(st, "qd_gemv_q4k failed")
    return ms.value if time_reps else None


def qd_conv1d_causal(x_dev, w_dev, bias_dev=None, dilation: int = 1, stream=None):
    """Causal dilated convolution of the device signal x [Cin, T] with W [Cout, Cin, K];
    returns y [Cout, T] (fp32)."""
    import torch
    Cin, T = x_dev.shape
    Cout, _, K = w_dev.shape
    y = torch.empty((Cout, T), dtype=torch.float32, device=x_dev.device)
    s = (stream or torch.cuda.current_stream()).cuda_stream
    st = _lib.qd_conv1d_causal(_ptr(x_dev), Cin, T, _ptr(w_dev), _ptr(bias_dev), Cout, K, int(dilation), _ptr(y), s)
    if st != QD_OK:
        raise QDError(st, "qd_conv1d_causal failed")
    return y


def qd_conv_transpose1d_causal(x_dev, w_dev, bias_dev=None, stride: int = 2, stream=None):
    """Causal transposed convolution (kernel 2 * stride) of x [Cin, T] with W [Cin, Cout,
    2 * stride]; returns y [Cout, T * stride] (fp32)."""
    import torch
    Cin, T = x_dev.shape
    _, Cout, K = w_dev.shape
    if K != 2 * stride:
        raise ValueError("kernel must be 2 * stride")
    y = torch.empty((Cout, T * stride), dtype=torch.float32, device=x_dev.device)
    s = (stream or torch.cuda.current_stream()).cuda_stream
    st = _lib.qd_conv_transpose1d_causal(_ptr(x_dev), Cin, T, _ptr(w_dev), _ptr(bias_dev), Cout, int(stride),
                                         _ptr(y), s)
    if st != QD_OK:
        raise QDError(st, "qd_conv_transpose1d_causal failed")
    return y


def qd_conv1d_causal_tc(x_dev, w_dev, bias_dev=None, dilation: int = 1, stream=None, time_reps: int = 0):
    """qd_conv1d_causal on the tensor cores (weights rounded to bf16, x as bf16 hi + lo);
    returns y [Cout, T], and with time_reps > 0 also the mean ms of that many runs."""
    import torch
    Cin, T = x_dev.shape
    Cout, _, K = w_dev.shape
    y = torch.empty((Cout, T), dtype=torch.float32, device=x_dev.device)
    s = (stream or torch.cuda.current_stream()).cuda_stream
    ms = ctypes.c_float(0.0)
    st = _lib.qd_conv1d_causal_tc(_ptr(x_dev), Cin, T, _ptr(w_dev), _ptr(bias_dev), Cout, K, int(dilation), _ptr(y),
                                  s, int(time_reps), ctypes.byref(ms) if time_reps > 0 else None)
    if st != QD_OK:
        raise QDError(st, "qd_conv1d_causal_tc failed")
    return (y, ms.value) if time_reps > 0 else y


def qd_conv_transpose1d_causal_tc(x_dev, w_dev, bias_dev=None, stride: int = 2, stream=None, time_reps: int = 0):
    """qd_conv_transpose1d_causal on the tensor cores, per output phase (weights rounded to
    bf16, x as bf16 hi + lo); returns y [Cout, T * stride], and with time_reps > 0 also
    the mean ms of that many runs."""
    import torch
    Cin, T = x_dev.shape
    _, Cout, K = w_dev.shape
    if K != 2 * stride:
        raise ValueError("kernel must be 2 * stride")
    y = torch.empty((Cout, T * stride), dtype=torch.float32, device=x_dev.device)
    s = (stream or torch.cuda.current_stream()).cuda_stream
    ms = ctypes.c_float(0.0)
    st = _lib.qd_conv_transpose1d_causal_tc(_ptr(x_dev), Cin, T, _ptr(w_dev), _ptr(bias_dev), Cout, int(stride),
                                            _ptr(y), s, int(time_reps), ctypes.byref(ms) if time_reps > 0 else None)
    if st != QD_OK:
        raise QDError(st, "qd_conv_transpose1d_causal_tc failed")
    return (y, ms.value) if time_reps > 0 else y
