"""Seeded synthetic workloads: decoder shapes and the random tensors drawn for them.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It only defines shapes and draws numbers (see ``synth.c``); it holds
none of the decoder's arithmetic.

Shapes follow the five workloads the decode path is measured on:

* ``tiny``    -- one-layer fp32 decoder (hidden 256, 4 q / 2 kv heads, head_dim 64,
                 QK-RMSNorm, FFN 768, vocab 1024), prefill 35 + 8 greedy steps,
                 repetition penalty 1.05, one KV bucket of 128.
* ``asr``     -- the ASR decoder of "Audio8-ASR: dynamic KV-cache buckets"
                 (8 layers, hidden 512, 8 q / 8 kv heads, head_dim 64, so the
                 cache is [8, Smax, 64]; FFN 2048; vocab 151936; EOS 151645
                 masked off), prefill 110, greedy decode to KV length 400, buckets
                 128 -> 256 -> 512.
* ``talker``  -- the Qwen3-TTS Talker of the ncnn port (28 layers, hidden 1024,
                 16 q / 8 kv heads, head_dim 128, QK-RMSNorm, FFN 3072, codec
                 vocab 3072, repetition penalty 1.05), prefill 64 + 600 steps,
                 buckets 128 -> 256 -> 512 -> 1024.
* ``frame``   -- talker + the 5-layer Code Predictor (15 heads of vocab 2048).
* ``batched`` -- 64 independent talker streams with ragged KV lengths.

Random draws: every tensor has a name; its stream id is the 64-bit FNV-1a hash of
that name, so tensors can be drawn in any order and independently.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _get_lib():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, f64 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.synth_normal_f32.argtypes = [u64, u64, i64, f64, f64, vp]
            lib.synth_normal_bf16.argtypes = [u64, u64, i64, f64, f64, vp]
            lib.synth_uniform_int.argtypes = [u64, u64, i64, ctypes.c_int32, ctypes.c_int32, vp]
            lib.synth_raw_u64.argtypes = [u64, i64, vp]
            for f in (lib.synth_normal_f32, lib.synth_normal_bf16, lib.synth_uniform_int, lib.synth_raw_u64):
                f.restype = None
            _lib = lib
    return _lib


def tensor_id(name: str) -> int:
    """64-bit FNV-1a hash of a tensor name (its random stream id)."""
    h = 0xCBF29CE484222325
    for b in name.encode():
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def normal(name: str, shape, seed: int = 0, mean: float = 0.0, std: float = 1.0,
           bf16: bool = False) -> np.ndarray:
    """Draw N(mean, std^2) values for tensor ``name``.

    fp32 output is ``float32``; bf16 output is the raw bfloat16 bit pattern as
    ``uint16`` (round-to-nearest-even from the fp32 draw)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16 if bf16 else np.float32)
    lib = _get_lib()
    fn = lib.synth_normal_bf16 if bf16 else lib.synth_normal_f32
    fn(seed, tensor_id(name), n, float(mean), float(std), out.ctypes.data)
    return out.reshape(shape)


def uniform_int(name: str, n: int, lo: int, hi: int, seed: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _get_lib().synth_uniform_int(seed, tensor_id(name), n, lo, hi, out.ctypes.data)
    return out


def raw_u64(state: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint64)
    _get_lib().synth_raw_u64(state, n, out.ctypes.data)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32 (for host-side display)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------------------
# Decoder shapes
# --------------------------------------------------------------------------------------

@dataclass(frozen=True)
class Shape:
    name: str
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int                 # rows of each output head
    embed_rows: int            # rows of the input embedding table (0: inputs are embeddings)
    bf16: bool                 # weights (and the KV cache) in bf16, else fp32
    qk_norm: bool
    n_heads_out: int = 1       # output heads (15 for the Code Predictor)
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    rep_penalty: float = 1.0   # 1.0 = off
    eos_mask_id: int = -1      # id whose logit is forced to -inf (-1: none)
    buckets: tuple = (128,)
    mrope_section: tuple = (0, 0, 0)   # frequencies per rotary stream (t, h, w); 0s: plain RoPE
    # workload
    prefill: int = 0
    decode_steps: int = 0
    seed: int = 0

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def layer_matrix_params(self) -> int:
        h, q, kv, f = self.hidden, self.q_dim, self.kv_dim, self.ffn
        return q * h + 2 * kv * h + h * q + 3 * f * h

    def matrix_params(self) -> int:
        """Parameters of every matrix read per decode step (layers + one head)."""
        return self.n_layers * self.layer_matrix_params() + self.vocab * self.hidden

    def weight_bytes_per_step(self) -> int:
        """Bytes of weights streamed per decode step: all layer matrices, the norm
        gammas, and one output head (the embedding row gather is negligible)."""
        esize = 2 if self.bf16 else 4
        norms = self.n_layers * (2 * self.hidden + (2 * self.head_dim if self.qk_norm else 0)) + self.hidden
        return esize * (self.matrix_params() + norms)

    def kv_bytes_per_position(self) -> int:
        esize = 2 if self.bf16 else 4
        return esize * self.n_layers * 2 * self.kv_dim

    def step_bytes(self, L: int) -> int:
        """Algorithmic bytes of one decode step attending over L positions: weights
        read once, K/V read for L positions, the new K/V row written once."""
        return self.weight_bytes_per_step() + L * self.kv_bytes_per_position()


TINY = Shape("tiny", hidden=256, n_layers=1, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=768,
             vocab=1024, embed_rows=1024, bf16=False, qk_norm=True, rep_penalty=1.05,
             buckets=(128,), prefill=35, decode_steps=8)
ASR = Shape("asr", hidden=512, n_layers=8, n_q_heads=8, n_kv_heads=8, head_dim=64, ffn=2048,
            vocab=151936, embed_rows=151936, bf16=True, qk_norm=False, rep_penalty=1.0,
            eos_mask_id=151645, buckets=(128, 256, 512), prefill=110, decode_steps=290)
TALKER = Shape("talker", hidden=1024, n_layers=28, n_q_heads=16, n_kv_heads=8, head_dim=128,
               ffn=3072, vocab=3072, embed_rows=3072, bf16=True, qk_norm=True, rep_penalty=1.05,
               buckets=(128, 256, 512, 1024), prefill=64, decode_steps=600)
CODE_PREDICTOR = Shape("code_predictor", hidden=1024, n_layers=5, n_q_heads=16, n_kv_heads=8,
                       head_dim=128, ffn=3072, vocab=2048, embed_rows=0, bf16=True, qk_norm=True,
                       n_heads_out=15, rep_penalty=1.0, buckets=(32,), prefill=2, decode_steps=14)

CONFIGS: Dict[str, Shape] = {s.name: s for s in (TINY, ASR, TALKER, CODE_PREDICTOR)}

# Frame workload: talker frames, each followed by a 15-code predictor loop.
FRAME_COUNT = 150
FRAME_CODE_VOCAB = 2048
# Batched multi-stream workload.
BATCH_STREAMS = 64
BATCH_SMAX = 2048
BATCH_STEPS = 256
BATCH_L0 = (256, 1792)       # initial KV lengths, inclusive range, so L0 + 256 <= 2048
BATCH_PREFILL = (8, 512)     # streams x positions, timed separately


def scaled(shape: Shape, **kw) -> Shape:
    """A copy of ``shape`` with some fields replaced (for reduced test cases).  A new
    head_dim rescales the multimodal RoPE sections when they scale to whole numbers
    (else the copy uses plain RoPE)."""
    if "head_dim" in kw and "mrope_section" not in kw and any(shape.mrope_section):
        sec = [x * kw["head_dim"] for x in shape.mrope_section]
        ok = all(x % shape.head_dim == 0 for x in sec)
        kw["mrope_section"] = tuple(x // shape.head_dim for x in sec) if ok else (0, 0, 0)
    return replace(shape, **kw)


NORM_NAMES = ("attn_norm", "q_norm", "k_norm", "mlp_norm")
MATRIX_NAMES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def layer_tensor_shapes(s: Shape) -> Dict[str, tuple]:
    d = {
        "attn_norm": (s.hidden,),
        "wq": (s.q_dim, s.hidden),
        "wk": (s.kv_dim, s.hidden),
        "wv": (s.kv_dim, s.hidden),
        "wo": (s.hidden, s.q_dim),
        "mlp_norm": (s.hidden,),
        "wg": (s.ffn, s.hidden),
        "wu": (s.ffn, s.hidden),
        "wd": (s.hidden, s.ffn),
    }
    if s.qk_norm:
        d["q_norm"] = (s.head_dim,)
        d["k_norm"] = (s.head_dim,)
    return d


def model_weights(s: Shape, seed: Optional[int] = None, prefix: str = "") -> Dict[str, np.ndarray]:
    """All weights of decoder ``s``.  Matrices ~ N(0, 0.02), norm gammas ~ 1 + N(0, 0.1).

    Keys: ``embed`` (if embed_rows), ``final_norm``, ``lm_head.{j}``, ``layers.{l}.{name}``.
    Arrays are float32 for fp32 shapes and bfloat16 bit patterns (uint16) for bf16 shapes."""
    seed = s.seed if seed is None else seed
    pre = prefix or s.name
    out: Dict[str, np.ndarray] = {}

    def draw(key, shape, gamma):
        mean, std = (1.0, 0.1) if gamma else (0.0, 0.02)
        out[key] = normal(f"{pre}/{key}", shape, seed, mean, std, bf16=s.bf16)

    if s.embed_rows:
        draw("embed", (s.embed_rows, s.hidden), False)
    for l in range(s.n_layers):
        for name, shp in layer_tensor_shapes(s).items():
            draw(f"layers.{l}.{name}", shp, name in NORM_NAMES)
    draw("final_norm", (s.hidden,), True)
    for j in range(s.n_heads_out):
        draw(f"lm_head.{j}", (s.vocab, s.hidden), False)
    return out


def prefill_embeds(s: Shape, n: Optional[int] = None, seed: Optional[int] = None,
                   stream: str = "prefill") -> np.ndarray:
    """Prompt embeddings ~ N(0, 1), float32 [n, hidden]."""
    n = s.prefill if n is None else n
    seed = s.seed if seed is None else seed
    return normal(f"{s.name}/{stream}", (n, s.hidden), seed, 0.0, 1.0)


def grid_prompt_positions(n: int, text_before: int, grid_h: int, grid_w: int) -> np.ndarray:
    """Rotary positions [3, n] (t, h, w streams) of a prompt laid out as text, one
    grid_h x grid_w image, text: the text positions are equal in the three streams
    and count up; the image holds t at the next position while h and w run over its
    rows and columns from there; the text after it resumes at the largest position
    so far + 1.  (The shape of a multimodal prompt; no values of any dataset.)"""
    assert text_before + grid_h * grid_w <= n
    pos = np.empty((3, n), np.int32)
    pos[:, :text_before] = np.arange(text_before)
    k, b = text_before, text_before
    for r in range(grid_h):
        for c in range(grid_w):
            pos[:, k] = (b, b + r, b + c)
            k += 1
    nxt = b + max(grid_h, grid_w)
    pos[:, k:] = np.arange(nxt, nxt + n - k)
    return pos


def frame_tables(seed: int = 0, rows: int = FRAME_CODE_VOCAB, hidden: int = 1024,
                 bf16: bool = True) -> Dict[str, np.ndarray]:
    """Code-embedding tables of the frame workload: E1..E15 [rows, hidden] ~ N(0, 0.02)
    (bf16 bits by default).  E0 is the talker's own embedding table."""
    return {f"code_embed.{j}": normal(f"frame/code_embed.{j}", (rows, hidden), seed, 0.0, 0.02, bf16=bf16)
            for j in range(1, 16)}


def frame_text_embeds(n_frames: int = FRAME_COUNT, seed: int = 0, hidden: int = 1024) -> np.ndarray:
    """Per-frame text/pad embedding ~ N(0, 1), float32 [n_frames, hidden]."""
    return normal("frame/text_pad", (n_frames, hidden), seed, 0.0, 1.0)


def frame_bytes(talker_L: int, talker_step: bool = True) -> int:
    """Algorithmic bytes of one frame: the Talker step attending over talker_L
    positions (when the frame has one) and the Code Predictor's 15 weight passes
    (the two-position prefill needs its weights once; each pass reads one head and
    the K/V of the positions it attends, 2..16), plus the K/V row of position 0."""
    cp = CODE_PREDICTOR
    b = sum(cp.step_bytes(L) for L in range(2, 17)) + cp.kv_bytes_per_position()
    return b + (TALKER.step_bytes(talker_L) if talker_step else 0)


def batch_initial_lengths(seed: int = 0, n: int = BATCH_STREAMS, lo: int = BATCH_L0[0],
                          hi: int = BATCH_L0[1]) -> np.ndarray:
    """Cached length of each stream at the start of the batched workload, ~ U{lo..hi}."""
    return uniform_int("batched/L0", n, lo, hi, seed)


def batch_stream_kv(shape: "Shape", stream: int, length: int, seed: int = 0) -> np.ndarray:
    """Initial cache of one stream, [n_layers, 2, n_kv_heads, length, head_dim] ~ N(0, 1)
    as bf16 bits (the batched workload starts from filled caches, not from a prefill)."""
    return normal(f"batched/kv/{stream}", (shape.n_layers, 2, shape.n_kv_heads, length, shape.head_dim), seed,
                  0.0, 1.0, bf16=True)


def batch_first_tokens(n: int, vocab: int, seed: int = 0) -> np.ndarray:
    """Input token of each stream's first step, ~ U{0..vocab-1}."""
    return uniform_int("batched/first_token", n, 0, vocab - 1, seed)
