"""Phase timeline of the persistent decode step.

Builds a variant of the library with ``-DQD_STEP_TRACE`` (``_build/libqd_trace.so``;
the in-tree ``libqd.so`` is untouched), runs a few decode steps of a workload on it in
a child process, and prints, for one layer, when every CTA passed each phase boundary
(thread 0's ``%globaltimer``, whose ticks on this GPU are 32 ns apart or coarser),
min / median / max over the CTAs, and the hops from the last writer of a vector to its
readers.

    python -m transformer_autoregressive_decode_gb300.step_timeline talker [layer]
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
TRACE_LIB = os.path.join(ROOT, "_build", "libqd_trace.so")
CTAS, SLOTS = 160, 24          # kStepTraceCtas, kStepTraceSlots

NAMES = {0: "QKV: start", 1: "QKV: input gathered", 2: "QKV: GEMV done", 3: "QKV: rows published",
         16: "attention: q/k/v polled", 17: "attention: done", 18: "attention: split published",
         19: "attention: merged published",
         4: "O-proj: start", 5: "O-proj: input gathered", 6: "O-proj: GEMV done", 7: "O-proj: rows published",
         8: "gate/up: start", 9: "gate/up: input gathered", 10: "gate/up: GEMV done", 11: "gate/up: act published",
         12: "down: start", 13: "down: input gathered", 14: "down: GEMV done", 15: "down: rows published",
         22: "next layer: input gathered"}
ORDER = [0, 1, 2, 3, 16, 17, 18, 19, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 22]
HOPS = [(3, 16, "QKV rows -> attention"), (18, 19, "split partials -> merge"), (19, 5, "merged -> O-proj"),
        (7, 9, "O-proj rows -> gate/up"), (11, 13, "act -> down"), (15, 22, "down rows -> next QKV")]


def build_traced() -> str:
    import importlib.util
    spec = importlib.util.spec_from_file_location("qd_build", os.path.join(PKG, "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    return b.build(force=True, extra_flags=["-DQD_STEP_TRACE"], lib=TRACE_LIB,
                   objdir=os.path.join(ROOT, "_build", "qd_trace"))


def run(workload: str, layer: int, reps: int = 5) -> None:
    """In a process whose QD_LIBRARY is the traced build."""
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    import transformer_autoregressive_decode_gb300 as qd
    import workloads as W
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload
    if os.path.abspath(qd.LIB_PATH) != os.path.abspath(TRACE_LIB):
        raise RuntimeError(f"not the traced build: {qd.LIB_PATH}")
    lib = ctypes.CDLL(qd.LIB_PATH)
    s = W.CONFIGS[workload]
    h = qd.qd_create(upload(W.model_weights(s)), config_from_shape(s))
    e = torch.from_numpy(W.prefill_embeds(s)).cuda()
    ids = torch.empty(64, dtype=torch.int32, device="cuda")
    first = qd.qd_prefill(h, embeds=e)
    qd.qd_decode_greedy(h, 20, first, ids)
    torch.cuda.synchronize()
    runs = []
    buf = (ctypes.c_ulonglong * (CTAS * SLOTS))()
    for _ in range(reps):
        if lib.qd_step_trace_reset(layer) != 0:
            raise RuntimeError("trace reset failed")
        qd.qd_decode_greedy(h, 1, -1, ids)
        torch.cuda.synchronize()
        if lib.qd_step_trace_read(buf, CTAS * SLOTS) != 0:
            raise RuntimeError("trace read failed")
        t = np.array(buf[:], dtype=np.float64).reshape(CTAS, SLOTS)[:152]
        t[t == 0] = np.nan
        runs.append((t - np.nanmin(t[:, 0])) / 1e3)
    pos, smax = qd.qd_get_pos(h)
    qd.qd_destroy(h)
    T = np.stack(runs)
    med = np.nanmedian(T, axis=0)            # per CTA, median over the steps
    print(f"== {workload}: layer {layer}, {reps} decode steps ending at position {pos}; "
          f"us after the first CTA started the layer, median over steps; min / median / max over CTAs")
    for k in ORDER:
        col = med[:, k]
        col = col[np.isfinite(col)]
        if len(col):
            print(f"  {NAMES[k]:30s} {col.min():7.2f} {np.median(col):7.2f} {col.max():7.2f}   ({len(col)} CTAs)")
    print("  hops: last writer -> readers' gather complete (median / last reader)")
    for a, b, lab in HOPS:
        last = np.nanmax(med[:, a])
        print(f"  {lab:30s} {np.nanmedian(med[:, b]) - last:6.2f} / {np.nanmax(med[:, b]) - last:6.2f}")
    gem = [np.nanmedian(med[:, 4 * p + 2] - med[:, 4 * p + 1]) for p in range(4)]
    print("  GEMV compute (median CTA): QKV %.2f  O-proj %.2f  gate/up %.2f  down %.2f;  attention %.2f" % (
        *gem, np.nanmedian(med[:, 17] - med[:, 16])))
    print("  layer: %.2f us" % np.nanmedian(med[:, 22]))


def main(argv) -> int:
    workload = argv[1] if len(argv) > 1 else "talker"
    layer = int(argv[2]) if len(argv) > 2 else 3
    if os.environ.get("QD_LIBRARY") == TRACE_LIB:
        run(workload, layer)
        return 0
    build_traced()
    env = dict(os.environ, QD_LIBRARY=TRACE_LIB)
    return subprocess.call([sys.executable, "-m", "transformer_autoregressive_decode_gb300.step_timeline",
                            workload, str(layer)], env=env, cwd=ROOT)


if __name__ == "__main__":
    sys.exit(main(sys.argv))
