"""Drive the CUDA path (through the C-ABI binding) and the CPU oracle side by side.

Teacher forcing: both sides are fed the oracle's id stream, so every step is
comparable even after a low-margin step where the argmax may legitimately
differ.  Tolerances are the acceptance bar of the decode path: per-layer hidden
state and logits relative L2 <= 2e-3, and equal ids at every step whose oracle
top-2 margin exceeds 1e-2.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

REL_TOL = 2e-3
MARGIN = 1e-2


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@dataclass
class Trace:
    ids_gpu: List[int] = field(default_factory=list)
    ids_ref: List[int] = field(default_factory=list)
    margins: List[float] = field(default_factory=list)
    logits_rel: List[float] = field(default_factory=list)
    hidden_rel: List[float] = field(default_factory=list)   # worst layer per step
    mismatches: List[int] = field(default_factory=list)      # steps with id mismatch above the margin
    low_margin: List[int] = field(default_factory=list)

    def check(self, rel_tol: float = REL_TOL):
        assert max(self.logits_rel or [0.0]) <= rel_tol, f"logits rel L2 {max(self.logits_rel):.3e}"
        assert max(self.hidden_rel or [0.0]) <= rel_tol, f"hidden rel L2 {max(self.hidden_rel):.3e}"
        assert not self.mismatches, f"id mismatches above margin at steps {self.mismatches[:10]}"


class Pair:
    def __init__(self, shape, weights, buckets=None, taps: bool = True, graphs: bool = True, q8: bool = False):
        """``q8``: the GPU model holds its matrices as 8-bit rows (qd_config.weight_q8) and
        the oracle runs on the dequantised matrices (float32 weights, the shape's cache)."""
        import torch
        import oracle as O
        import transformer_autoregressive_decode_gb300 as qd
        from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload

        self.qd, self.torch, self.shape = qd, torch, shape
        self.dev_w = upload(weights)
        self.h = qd.qd_create(self.dev_w, config_from_shape(shape, buckets, weight_q8=q8))
        qd.qd_set_graphs(self.h, graphs)
        if q8:
            self.ref = O.Oracle(shape, O.q8_model_weights(shape, weights), buckets=buckets, weights_f32=True)
        else:
            self.ref = O.Oracle(shape, weights, buckets=buckets)
        self.taps = taps
        if taps:
            self.t_hidden = torch.empty((shape.n_layers + 1, shape.hidden), dtype=torch.float32, device="cuda")
            self.t_logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
            qd.qd_set_debug_taps(self.h, self.t_hidden, self.t_logits)
        self.y = torch.empty(shape.hidden, dtype=torch.float32, device="cuda")
        self.trace = Trace()

    def close(self):
        self.qd.qd_destroy(self.h)
        self.ref.close()

    def _record(self, got, rid, rlog, margin, rtaps=None):
        t = self.trace
        step = len(t.ids_ref)
        t.ids_gpu.append(got)
        t.ids_ref.append(rid)
        t.margins.append(margin)
        if self.taps:
            t.logits_rel.append(rel_l2(self.t_logits.cpu().numpy(), rlog))
            if rtaps is not None:
                g = self.t_hidden.cpu().numpy()
                t.hidden_rel.append(max(rel_l2(g[l], rtaps[l]) for l in range(len(rtaps))))
        else:
            self.qd.qd_get_hidden(self.h, self.y)
            t.hidden_rel.append(rel_l2(self.y.cpu().numpy(), self.ref.hidden()))
        if margin > MARGIN:
            if got != rid:
                t.mismatches.append(step)
        else:
            t.low_margin.append(step)

    def prefill(self, embeds=None, tokens=None, head_idx=0, positions=None):
        torch = self.torch
        e_dev = None if embeds is None else torch.from_numpy(np.ascontiguousarray(embeds)).cuda()
        if positions is None:
            got = self.qd.qd_prefill(self.h, tokens=tokens, embeds=e_dev, head_idx=head_idx)
        else:
            got = self.qd.qd_prefill_mrope(self.h, positions, tokens=tokens, embeds=e_dev, head_idx=head_idx)
        rid, rlog, margin = self.ref.prefill(embeds=embeds, tokens=tokens, head_idx=head_idx, positions=positions)
        self._record(got, rid, rlog, margin)
        return rid

    def step(self, token=-1, embed=None, head_idx=0):
        torch = self.torch
        e_dev = None if embed is None else torch.from_numpy(np.ascontiguousarray(embed, np.float32)).cuda()
        got = self.qd.qd_decode_step(self.h, embed=e_dev, token=token, head_idx=head_idx)
        rid, rlog, margin, rtaps = self.ref.step(token=token, embed=embed, head_idx=head_idx, taps=self.taps)
        self._record(got, rid, rlog, margin, rtaps)
        return rid

    def run_teacher_forced(self, embeds, n_steps):
        rid = self.prefill(embeds=embeds)
        for _ in range(n_steps):
            rid = self.step(token=rid)
        return self.trace

    def kv(self) -> np.ndarray:
        """GPU cache as float32 [n_layers, 2, kvh, Smax, hd]."""
        torch = self.torch
        s = self.shape
        n = self.qd.qd_copy_kv(self.h)
        buf = torch.empty(n, dtype=torch.uint8, device="cuda")
        self.qd.qd_copy_kv(self.h, buf)
        pos, smax = self.qd.qd_get_pos(self.h)
        if s.bf16:
            t = buf.view(torch.bfloat16).float()
        else:
            t = buf.view(torch.float32)
        return t.reshape(s.n_layers, 2, s.n_kv_heads, smax, s.head_dim).cpu().numpy(), pos
