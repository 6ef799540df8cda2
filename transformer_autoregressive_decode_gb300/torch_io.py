"""Host <-> device marshalling helpers for callers of the binding.

``upload`` moves host arrays (float32, or bfloat16 bit patterns as uint16) to
torch device tensors; ``config_from_shape`` fills a ``qd_config`` from any object
with the decoder's shape attributes.  No decode arithmetic happens here.
"""
from __future__ import annotations

from typing import Dict

import numpy as np

from . import make_config, qd_config


def to_device(a: np.ndarray, device="cuda"):
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def upload(weights: Dict[str, np.ndarray], device="cuda") -> Dict[str, "torch.Tensor"]:
    return {k: to_device(v, device) for k, v in weights.items()}


def config_from_shape(s, buckets=None, weight_q8: bool = False) -> qd_config:
    return make_config(hidden=s.hidden, n_layers=s.n_layers, n_q_heads=s.n_q_heads, n_kv_heads=s.n_kv_heads,
                       head_dim=s.head_dim, ffn=s.ffn, vocab=s.vocab, embed_rows=s.embed_rows, bf16=s.bf16,
                       qk_norm=s.qk_norm, n_heads_out=s.n_heads_out, eos_mask_id=s.eos_mask_id,
                       buckets=tuple(s.buckets if buckets is None else buckets), rms_eps=s.rms_eps,
                       rope_theta=s.rope_theta, rep_penalty=s.rep_penalty,
                       mrope_section=tuple(getattr(s, "mrope_section", (0, 0, 0))), weight_q8=weight_q8)
