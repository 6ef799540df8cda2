"""CPU oracle for the decode step (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path never does: it shares no code
with it.  The arithmetic lives in ``oracle.c`` (plain C, fp32 with fp64 norm and
softmax accumulation); this file only compiles it and marshals arguments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

OK, EINVAL, ESTATE, EKVFULL, ENOMEM = 0, -1, -2, -3, -4
LAYER_SLOTS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "mlp_norm", "wg", "wu", "wd")


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what} failed with status {status}")
        self.status = status


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``liboracle.so`` (OpenMP, no FMA contraction).

    ``ORACLE_LIB`` in the environment names a prebuilt library to load instead;
    the mutation test uses it to run the pins against a deliberately broken copy."""
    override = os.environ.get("ORACLE_LIB")
    if override:
        return override
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "hidden", "n_layers", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab", "embed_rows",
        "w_bf16", "kv_bf16", "qk_norm", "n_heads_out", "eos_mask_id", "n_buckets")] + [
        ("buckets", ctypes.c_int * 8), ("acc64", ctypes.c_int), ("mrope_section", ctypes.c_int * 3),
        ("rms_eps", ctypes.c_double), ("rope_theta", ctypes.c_double), ("rep_penalty", ctypes.c_double)]


def _lib_handle():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            vp, i32, dp = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            P = ctypes.POINTER
            L.orc_create.argtypes = [P(Config), vp, P(i32)]
            L.orc_create.restype = vp
            L.orc_destroy.argtypes = [vp]
            L.orc_destroy.restype = None
            for f in (L.orc_reset, L.orc_pos, L.orc_smax):
                f.argtypes = [vp]
                f.restype = i32
            L.orc_forward.argtypes = [vp, vp, i32, i32, i32, i32, P(i32), vp, vp, P(dp)]
            L.orc_forward.restype = i32
            L.orc_prefill.argtypes = [vp, vp, vp, i32, i32, P(i32), vp, P(dp)]
            L.orc_prefill.restype = i32
            L.orc_prefill_positions.argtypes = [vp, vp, vp, i32, i32, vp, P(i32), vp, P(dp)]
            L.orc_prefill_positions.restype = i32
            L.orc_get_hidden.argtypes = [vp, vp]
            L.orc_get_hidden.restype = i32
            L.orc_get_kv.argtypes = [vp, i32, i32, vp]
            L.orc_get_kv.restype = i32
            L.orc_emitted_words.argtypes = [vp, vp]
            L.orc_emitted_words.restype = i32
            L.orc_recompute_logits.argtypes = [P(Config), vp, vp, vp, i32, i32, vp]
            L.orc_recompute_logits.restype = i32
            L.orc_rmsnorm.argtypes = [vp, vp, i32, dp, vp]
            L.orc_rmsnorm.restype = None
            L.orc_rope.argtypes = [vp, i32, i32, dp]
            L.orc_rope.restype = None
            L.orc_conv1d_causal.argtypes = [vp, i32, i32, vp, vp, i32, i32, i32, vp]
            L.orc_conv1d_causal.restype = i32
            L.orc_conv_transpose1d_causal.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp]
            L.orc_conv_transpose1d_causal.restype = i32
            L.orc_f32_to_f16.argtypes = [ctypes.c_float]
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_f32.restype = ctypes.c_float
            L.orc_quantize_q8.argtypes = [vp, i32, i32, vp, vp]
            L.orc_quantize_q8.restype = i32
            L.orc_gemv_q8.argtypes = [vp, vp, i32, i32, vp, vp]
            L.orc_gemv_q8.restype = i32
            L.orc_quantize_q4k.argtypes = [vp, i32, i32, vp]
            L.orc_quantize_q4k.restype = i32
            L.orc_gemv_q4k.argtypes = [vp, i32, i32, vp, vp]
            L.orc_gemv_q4k.restype = i32
            L.orc_rope_mrope.argtypes = [vp, i32, P(i32), P(i32), dp]
            L.orc_rope_mrope.restype = None
            L.orc_mrope_stream.argtypes = [i32, P(i32)]
            L.orc_mrope_stream.restype = i32
            L.orc_attend.argtypes = [vp, vp, vp, i32, i32, vp]
            L.orc_attend.restype = None
            L.orc_penalty_argmax.argtypes = [vp, i32, vp, ctypes.c_float, i32, P(dp)]
            L.orc_penalty_argmax.restype = i32
            L.orc_set_sampling.argtypes = [vp, i32, ctypes.c_double, ctypes.c_double, ctypes.c_uint64]
            L.orc_set_sampling.restype = i32
            L.orc_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            L.orc_splitmix64.restype = ctypes.c_uint64
            L.orc_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            L.orc_uniform.restype = ctypes.c_double
            L.orc_sample.argtypes = [vp, i32, i32, ctypes.c_double, ctypes.c_double, ctypes.c_double, P(dp)]
            L.orc_sample.restype = i32
            L.orc_silu_mul.argtypes = [ctypes.c_float, ctypes.c_float]
            L.orc_silu_mul.restype = ctypes.c_float
            L.orc_round_bf16.argtypes = [ctypes.c_float]
            L.orc_round_bf16.restype = ctypes.c_uint16
            L.orc_frame_sum.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
            L.orc_frame_sum.restype = i32
            L.orc_set_kv.argtypes = [vp, vp, i32]
            L.orc_set_kv.restype = i32
            L.orc_linear.argtypes = [vp, i32, i32, i32, vp, i32, vp]
            L.orc_linear.restype = i32
            L.orc_num_threads.argtypes = []
            L.orc_num_threads.restype = i32
            L.orc_set_threads.argtypes = [i32]
            L.orc_set_threads.restype = None
            _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def splitmix64(seed: int, counter: int) -> int:
    return int(_lib_handle().orc_splitmix64(seed, counter))


def uniform(seed: int, counter: int) -> float:
    return float(_lib_handle().orc_uniform(seed, counter))


def sample(logits: np.ndarray, top_k: int, temperature: float, top_p: float, u: float):
    """The oracle's sampler on final logits: (index, decision margin)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    mg = ctypes.c_double(0.0)
    i = _lib_handle().orc_sample(lg.ctypes.data, len(lg), int(top_k), float(temperature), float(top_p), float(u),
                           ctypes.byref(mg))
    return int(i), mg.value


def make_config(shape, acc64: bool = False, buckets: Optional[Sequence[int]] = None,
                weights_f32: bool = False) -> Config:
    """Oracle config from a ``workloads.Shape``; ``weights_f32`` takes every weight as
    float32 while the cache keeps the shape's type (a bf16 model whose matrices were
    replaced by their dequantised 8-bit rows, ``dequantize_q8``)."""
    c = Config()
    c.hidden, c.n_layers = shape.hidden, shape.n_layers
    c.n_q_heads, c.n_kv_heads, c.head_dim = shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    c.ffn, c.vocab, c.embed_rows = shape.ffn, shape.vocab, shape.embed_rows
    c.w_bf16 = 0 if weights_f32 else int(shape.bf16)
    c.kv_bf16 = int(shape.bf16)
    c.qk_norm, c.n_heads_out, c.eos_mask_id = int(shape.qk_norm), shape.n_heads_out, shape.eos_mask_id
    b = list(shape.buckets if buckets is None else buckets)
    c.n_buckets = len(b)
    for i, v in enumerate(b):
        c.buckets[i] = v
    c.acc64 = int(acc64)
    for i, v in enumerate(getattr(shape, "mrope_section", (0, 0, 0))):
        c.mrope_section[i] = int(v)
    c.rms_eps, c.rope_theta, c.rep_penalty = shape.rms_eps, shape.rope_theta, shape.rep_penalty
    return c


def weight_table(shape, weights: Dict[str, np.ndarray]):
    """Pointer table in the oracle's slot order; keeps the arrays alive."""
    keep = []

    def p(key):
        a = weights.get(key)
        if a is None:
            return None
        a = np.ascontiguousarray(a)
        keep.append(a)
        return a.ctypes.data

    ptrs = [p("embed"), p("final_norm")] + [p(f"lm_head.{j}") for j in range(shape.n_heads_out)]
    for l in range(shape.n_layers):
        ptrs += [p(f"layers.{l}.{s}") for s in LAYER_SLOTS]
    arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
    return arr, keep


class Oracle:
    """One decode stream on the CPU oracle."""

    def __init__(self, shape, weights: Dict[str, np.ndarray], acc64: bool = False,
                 buckets: Optional[Sequence[int]] = None, weights_f32: bool = False):
        self.L = _lib_handle()
        self.shape = shape
        self.cfg = make_config(shape, acc64, buckets, weights_f32)
        self._table, self._keep = weight_table(shape, weights)
        st = ctypes.c_int(0)
        self.h = self.L.orc_create(ctypes.byref(self.cfg), ctypes.cast(self._table, ctypes.c_void_p), ctypes.byref(st))
        if not self.h:
            raise OracleError(st.value, "create")

    def close(self):
        if self.h:
            self.L.orc_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st, what):
        if st != OK:
            raise OracleError(st, what)

    def reset(self):
        self._check(self.L.orc_reset(self.h), "reset")

    @property
    def pos(self) -> int:
        return self.L.orc_pos(self.h)

    @property
    def smax(self) -> int:
        return self.L.orc_smax(self.h)

    def prefill(self, embeds: Optional[np.ndarray] = None, tokens: Optional[np.ndarray] = None,
                head_idx: int = 0, want_logits: bool = True, positions: Optional[np.ndarray] = None):
        """Prefill from position 0; ``positions`` ([3, n] int32: the t, h, w rotary
        positions of each prompt position) replaces the default (i, i, i)."""
        n = len(embeds) if embeds is not None else len(tokens)
        e = None if embeds is None else np.ascontiguousarray(embeds, dtype=np.float32)
        t = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
        logits = np.empty(self.shape.vocab, np.float32) if want_logits else None
        fid, margin = ctypes.c_int(-1), ctypes.c_double(0.0)
        if positions is None:
            self._check(self.L.orc_prefill(self.h, _ptr(t), _ptr(e), n, head_idx, ctypes.byref(fid),
                                           _ptr(logits), ctypes.byref(margin)), "prefill")
        else:
            pos = np.ascontiguousarray(positions, dtype=np.int32)
            if pos.shape != (3, n):
                raise ValueError(f"positions must be [3, {n}], got {pos.shape}")
            self._check(self.L.orc_prefill_positions(self.h, _ptr(t), _ptr(e), n, head_idx, _ptr(pos),
                                                     ctypes.byref(fid), _ptr(logits), ctypes.byref(margin)),
                        "prefill_positions")
        return fid.value, logits, margin.value

    def step(self, token: int = -1, embed: Optional[np.ndarray] = None, head_idx: int = 0,
             want_head: bool = True, want_logits: bool = True, taps: bool = False,
             add_emitted: bool = True):
        """One decode position.  Returns (id, raw logits, top-2 margin, hidden taps)."""
        e = None if embed is None else np.ascontiguousarray(embed, dtype=np.float32)
        logits = np.empty(self.shape.vocab, np.float32) if (want_head and want_logits) else None
        tp = np.empty((self.shape.n_layers + 1, self.shape.hidden), np.float32) if taps else None
        oid, margin = ctypes.c_int(-1), ctypes.c_double(0.0)
        self._check(self.L.orc_forward(self.h, _ptr(e), int(token), int(add_emitted), int(want_head), head_idx,
                                       ctypes.byref(oid), _ptr(logits), _ptr(tp), ctypes.byref(margin)), "forward")
        return oid.value, logits, margin.value, tp

    def set_sampling(self, top_k: int, temperature: float = 1.0, top_p: float = 1.0, seed: int = 0):
        """Sample the heads' ids (top_k 0: greedy argmax); the draw counter is the
        number of ids produced since reset."""
        self._check(self.L.orc_set_sampling(self.h, int(top_k), float(temperature), float(top_p), int(seed)),
                    "set_sampling")

    def set_kv(self, kv: np.ndarray, length: int):
        """Start from a cache [n_layers, 2, n_kv_heads, length, head_dim] in the cache
        type (bf16 bits as uint16 on the bf16 path, else float32)."""
        k = np.ascontiguousarray(kv)
        self._check(self.L.orc_set_kv(self.h, k.ctypes.data if length else None, int(length)), "set_kv")

    def hidden(self) -> np.ndarray:
        out = np.empty(self.shape.hidden, np.float32)
        self._check(self.L.orc_get_hidden(self.h, out.ctypes.data), "get_hidden")
        return out

    def kv(self, layer: int, which: int) -> np.ndarray:
        s = self.shape
        out = np.empty((s.n_kv_heads, self.pos, s.head_dim), np.float32)
        self._check(self.L.orc_get_kv(self.h, layer, which, out.ctypes.data), "get_kv")
        return out

    def emitted(self) -> np.ndarray:
        out = np.zeros((self.shape.vocab + 31) // 32, np.uint32)
        self.L.orc_emitted_words(self.h, out.ctypes.data)
        return out


def recompute_logits(shape, weights, embeds=None, tokens=None, head_idx: int = 0, acc64: bool = False):
    L = _lib_handle()
    cfg = make_config(shape, acc64)
    table, keep = weight_table(shape, weights)
    n = len(embeds) if embeds is not None else len(tokens)
    e = None if embeds is None else np.ascontiguousarray(embeds, dtype=np.float32)
    t = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    out = np.empty(shape.vocab, np.float32)
    st = L.orc_recompute_logits(ctypes.byref(cfg), ctypes.cast(table, ctypes.c_void_p), _ptr(t), _ptr(e), n,
                                head_idx, out.ctypes.data)
    if st != OK:
        raise OracleError(st, "recompute")
    return out


# ---- two-level frame generation ----

FRAME_CODES = 16


def table_row(table: np.ndarray, i: int) -> np.ndarray:
    """Row i of an embedding table as float32 (bfloat16 bit patterns are widened)."""
    r = np.asarray(table[int(i)])
    if r.dtype == np.uint16:
        return (r.astype(np.uint32) << 16).view(np.float32)
    return r.astype(np.float32)


def frame_sum(tables: Sequence[np.ndarray], ids: Sequence[int], text: np.ndarray) -> np.ndarray:
    """((E_0[ids_0] + E_1[ids_1]) + ... ) + text in fp32, tables bf16 bits or float32."""
    bf16 = tables[0].dtype == np.uint16
    keep = [np.ascontiguousarray(t) for t in tables]
    if any((t.dtype == np.uint16) != bf16 for t in keep):
        raise ValueError("tables must share one dtype")
    hidden = keep[0].shape[1]
    ptrs = (ctypes.c_void_p * len(keep))(*[t.ctypes.data for t in keep])
    rows = np.array([t.shape[0] for t in keep], np.int32)
    idv = np.ascontiguousarray(ids, np.int32)
    tx = np.ascontiguousarray(text, np.float32)
    out = np.empty(hidden, np.float32)
    st = _lib_handle().orc_frame_sum(ctypes.cast(ptrs, ctypes.c_void_p), rows.ctypes.data, idv.ctypes.data,
                                     len(keep), hidden, int(bf16), tx.ctypes.data, out.ctypes.data)
    if st != OK:
        raise OracleError(st, "frame_sum")
    return out


class FrameLoop:
    """Two-level frame generation over two oracle streams.

    Per frame ("Qwen3-TTS ncnn port", section "Talker: non-standard structure and
    two-level generation"; "qwen3-tts-hip OPTIMIZATION_LOG", Code Predictor
    sub-stages), with p the Talker's last id and h_T its final-norm output:
      1. reset the predictor, prefill it with [h_T, E_0[p]], head 0 -> code_1;
      2. for j = 1..14: a step with input E_j[code_j] (code_j joins the predictor's
         emitted set), head j -> code_{j+1};
      3. next_in = E_0[p] + E_1[code_1] + ... + E_15[code_15] + text;
      4. unless it is the last frame: a Talker step with input next_in and token p.
    ``force`` [n, 16] replaces the fed-back ids (teacher forcing); the argmaxes are
    still reported."""

    def __init__(self, talker: Oracle, predictor: Oracle, e0: np.ndarray, code_tables: Sequence[np.ndarray]):
        if len(code_tables) != FRAME_CODES - 1:
            raise ValueError("need 15 code tables")
        self.talker, self.predictor = talker, predictor
        self.tables = [e0] + list(code_tables)

    def generate(self, n_frames: int, text: np.ndarray, primary: int, primary_margin: float = float("inf"),
                 force: Optional[np.ndarray] = None):
        """Returns (codes [n, 16] argmaxes, margins [n, 16], next_in [n, hidden],
        talker_hidden [n, hidden] = h_T of every frame)."""
        hidden = self.tables[0].shape[1]
        codes = np.zeros((n_frames, FRAME_CODES), np.int32)
        margins = np.zeros((n_frames, FRAME_CODES), np.float64)
        next_in = np.zeros((n_frames, hidden), np.float32)
        h_t = np.zeros((n_frames, hidden), np.float32)
        for f in range(n_frames):
            codes[f, 0], margins[f, 0] = primary, primary_margin
            p = int(force[f, 0]) if force is not None else primary
            h_t[f] = self.talker.hidden()
            self.predictor.reset()
            cid, _, cm = self.predictor.prefill(embeds=np.stack([h_t[f], table_row(self.tables[0], p)]),
                                                head_idx=0, want_logits=False)
            codes[f, 1], margins[f, 1] = cid, cm
            fed = [p]
            for j in range(1, FRAME_CODES - 1):
                c = int(force[f, j]) if force is not None else int(codes[f, j])
                fed.append(c)
                cid, _, cm, _ = self.predictor.step(token=c, embed=table_row(self.tables[j], c), head_idx=j,
                                                    want_logits=False)
                codes[f, j + 1], margins[f, j + 1] = cid, cm
            fed.append(int(force[f, FRAME_CODES - 1]) if force is not None else int(codes[f, FRAME_CODES - 1]))
            next_in[f] = frame_sum(self.tables, fed, text[f])
            if f < n_frames - 1:
                primary, _, primary_margin, _ = self.talker.step(token=p, embed=next_in[f], head_idx=0,
                                                                 want_logits=False)
        return codes, margins, next_in, h_t


def linear(W: np.ndarray, x: np.ndarray) -> np.ndarray:
    """out[t] = W x[t] for every row of x (W float32 or bfloat16 bits [R, K])."""
    Wc = np.ascontiguousarray(W)
    xc = np.ascontiguousarray(x, np.float32)
    R, K = Wc.shape
    T = xc.shape[0]
    out = np.empty((T, R), np.float32)
    st = _lib_handle().orc_linear(Wc.ctypes.data, int(Wc.dtype == np.uint16), R, K, xc.ctypes.data, T,
                                  out.ctypes.data)
    if st != OK:
        raise OracleError(st, "linear")
    return out


# ---- primitives (for the pins) ----

def rmsnorm(x, gamma, eps):
    x = np.ascontiguousarray(x, np.float32)
    g = np.ascontiguousarray(gamma, np.float32)
    out = np.empty_like(x)
    _lib_handle().orc_rmsnorm(x.ctypes.data, g.ctypes.data, len(x), eps, out.ctypes.data)
    return out


def rope(v, pos, theta):
    v = np.array(v, dtype=np.float32, copy=True)
    _lib_handle().orc_rope(v.ctypes.data, len(v), int(pos), float(theta))
    return v


def rope_mrope(v, pos3, section, theta):
    """Rotary embedding with one position per stream (t, h, w) and the interleaved
    section sizes ``section``."""
    v = np.array(v, dtype=np.float32, copy=True)
    p = (ctypes.c_int * 3)(*[int(x) for x in pos3])
    sec = (ctypes.c_int * 3)(*[int(x) for x in section])
    _lib_handle().orc_rope_mrope(v.ctypes.data, len(v), p, sec, float(theta))
    return v


def mrope_stream(m, section):
    """The position stream (0 t, 1 h, 2 w) frequency m takes."""
    sec = (ctypes.c_int * 3)(*[int(x) for x in section])
    return _lib_handle().orc_mrope_stream(int(m), sec)


def attend(q, K, V):
    q = np.ascontiguousarray(q, np.float32)
    K = np.ascontiguousarray(K, np.float32)
    V = np.ascontiguousarray(V, np.float32)
    out = np.empty(len(q), np.float32)
    _lib_handle().orc_attend(q.ctypes.data, K.ctypes.data, V.ctypes.data, K.shape[0], len(q), out.ctypes.data)
    return out


def penalty_argmax(logits, emitted_ids, penalty, eos_id=-1):
    lg = np.array(logits, dtype=np.float32, copy=True)
    mask = np.zeros((len(lg) + 31) // 32, np.uint32)
    for i in emitted_ids:
        mask[i >> 5] |= np.uint32(1 << (i & 31))
    margin = ctypes.c_double(0.0)
    idx = _lib_handle().orc_penalty_argmax(lg.ctypes.data, len(lg), mask.ctypes.data, float(penalty), int(eos_id),
                                           ctypes.byref(margin))
    return idx, lg, margin.value


def silu_mul(g, u):
    return _lib_handle().orc_silu_mul(float(g), float(u))


def round_bf16(f):
    return _lib_handle().orc_round_bf16(float(f))


def num_threads() -> int:
    return _lib_handle().orc_num_threads()


def set_threads(n: int):
    _lib_handle().orc_set_threads(int(n))


def f32_to_f16(f) -> int:
    """IEEE half bits of a float (round to nearest even)."""
    return int(_lib_handle().orc_f32_to_f16(float(np.float32(f))))


def f16_to_f32(h) -> float:
    return float(_lib_handle().orc_f16_to_f32(int(h)))


def quantize_q8(w: np.ndarray):
    """Codes int8 [rows, K] and half-bit scales uint16 [rows, K/32] of W [rows, K] (fp32)."""
    w = np.ascontiguousarray(w, np.float32)
    rows, K = w.shape
    codes = np.empty((rows, K), np.int8)
    scales = np.empty((rows, K // 32), np.uint16)
    st = _lib_handle().orc_quantize_q8(w.ctypes.data, rows, K, codes.ctypes.data, scales.ctypes.data)
    if st != OK:
        raise OracleError(st, "quantize_q8")
    return codes, scales


def dequantize_q8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """The matrix the 8-bit rows stand for: each code times its 32-weight block's half
    scale, float32 [rows, K] (exact: an 8-bit integer times an 11-bit significand)."""
    codes = np.asarray(codes, np.int8)
    d = np.asarray(scales, np.uint16).view(np.float16).astype(np.float32)
    return codes.astype(np.float32) * np.repeat(d, 32, axis=1)


def q8_model_weights(shape, weights: Dict[str, np.ndarray]) -> Dict[str, np.ndarray]:
    """Weights of a model whose layer matrices and output heads are held as 8-bit rows
    (the weight-only Q8_0 scheme of "audio.cpp Rockchip NPU build notes"): those are
    quantised from their float32 values and replaced by the dequantised matrices; the
    embedding table and the norm gammas are the same values as float32.  For an Oracle
    with ``weights_f32``."""
    mats = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")
    out = {}
    for k, v in weights.items():
        if v.dtype == np.uint16:                       # bfloat16 bits: the upper half of a float32
            f = (np.asarray(v).astype(np.uint32) << 16).view(np.float32)
        else:
            f = np.asarray(v, np.float32)
        if k.startswith("lm_head.") or k.rsplit(".", 1)[-1] in mats:
            f = dequantize_q8(*quantize_q8(f))
        out[k] = np.ascontiguousarray(f, np.float32)
    return out


def gemv_q8(codes: np.ndarray, scales: np.ndarray, x: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.int8)
    scales = np.ascontiguousarray(scales, np.uint16)
    x = np.ascontiguousarray(x, np.float32)
    rows, K = codes.shape
    y = np.empty(rows, np.float32)
    st = _lib_handle().orc_gemv_q8(codes.ctypes.data, scales.ctypes.data, rows, K, x.ctypes.data, y.ctypes.data)
    if st != OK:
        raise OracleError(st, "gemv_q8")
    return y


Q4K_BLOCK_BYTES = 144   # 256 weights: half d, half dm, 8 + 8 six-bit fields, 128 code bytes


def quantize_q4k(w: np.ndarray) -> np.ndarray:
    """Q4_K super-blocks of W [rows, K] (fp32, K a multiple of 256): uint8 [rows, K/256, 144]."""
    w = np.ascontiguousarray(w, np.float32)
    rows, K = w.shape
    out = np.zeros((rows, K // 256, Q4K_BLOCK_BYTES), np.uint8)
    st = _lib_handle().orc_quantize_q4k(w.ctypes.data, rows, K, out.ctypes.data)
    if st != OK:
        raise OracleError(st, "quantize_q4k")
    return out


def gemv_q4k(blocks: np.ndarray, x: np.ndarray) -> np.ndarray:
    blocks = np.ascontiguousarray(blocks, np.uint8)
    x = np.ascontiguousarray(x, np.float32)
    rows, nsb = blocks.shape[:2]
    y = np.empty(rows, np.float32)
    st = _lib_handle().orc_gemv_q4k(blocks.ctypes.data, rows, nsb * 256, x.ctypes.data, y.ctypes.data)
    if st != OK:
        raise OracleError(st, "gemv_q4k")
    return y


def conv1d_causal(x: np.ndarray, W: np.ndarray, bias: Optional[np.ndarray] = None, dilation: int = 1) -> np.ndarray:
    """x [Cin, T], W [Cout, Cin, K] -> y [Cout, T] (causal: zero history)."""
    x = np.ascontiguousarray(x, np.float32)
    W = np.ascontiguousarray(W, np.float32)
    Cin, T = x.shape
    Cout, _, K = W.shape
    b = None if bias is None else np.ascontiguousarray(bias, np.float32)
    y = np.empty((Cout, T), np.float32)
    st = _lib_handle().orc_conv1d_causal(x.ctypes.data, Cin, T, W.ctypes.data, _ptr(b), Cout, K, int(dilation),
                                         y.ctypes.data)
    if st != OK:
        raise OracleError(st, "conv1d_causal")
    return y


def conv_transpose1d_causal(x: np.ndarray, W: np.ndarray, bias: Optional[np.ndarray] = None,
                            stride: int = 2) -> np.ndarray:
    """x [Cin, T], W [Cin, Cout, 2*stride] -> y [Cout, T*stride]."""
    x = np.ascontiguousarray(x, np.float32)
    W = np.ascontiguousarray(W, np.float32)
    Cin, T = x.shape
    _, Cout, K = W.shape
    if K != 2 * stride:
        raise ValueError("kernel must be 2 * stride")
    b = None if bias is None else np.ascontiguousarray(bias, np.float32)
    y = np.empty((Cout, T * stride), np.float32)
    st = _lib_handle().orc_conv_transpose1d_causal(x.ctypes.data, Cin, T, W.ctypes.data, _ptr(b), Cout,
                                                   int(stride), y.ctypes.data)
    if st != OK:
        raise OracleError(st, "conv_transpose1d_causal")
    return y
