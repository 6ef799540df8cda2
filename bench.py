#!/usr/bin/env python3
"""Decode throughput of the GB300 decode path.

Default (``--workload all``): one JSON line whose headline is the Talker decoder
(28 layers, hidden 1024, 16 q / 8 kv heads x 128, QK-norm, FFN 3072, vocab 3072,
repetition penalty 1.05, bf16 weights and KV cache) on seeded synthetic weights.  A
trajectory is reset, prefill 64 N(0,1) embeddings, then 600 greedy decode steps with
the bucket migrations 128 -> 256 -> 512 -> 1024.  A benchmark "step" is one decode
token; the timed region continues the trajectory in progress (graph replays of the
step) and restarts a trajectory (reset + prefill, timed with the tokens) when one
ends.  The same line carries, as keys ``asr``, ``frames`` and ``batch``, the ASR
decoder (8 layers, hidden 512, vocab 151936, EOS masked), the two-level frame loop
(Talker + 15-code predictor, 150 frames) and the batched 64-stream Talker decode, each
with its own value, roofline, CPU baseline and end-to-end figure.  ``--workload``
selects one of them alone.

``--impl reference`` times the CPU oracle instead (on the host cores, a bounded
sample of the headline's workload).  Under torchrun every rank runs the decoders as
replicas; the batched decode partitions its 64 streams over the ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s at 1 GB300; per-step HBM GB/s as fraction of peak"


# DRAM bytes (read + write) of one decode_step_kernel launch from one ncu capture
# (profiles/decode_step_kernel_asr.md, profiles/decode_step_kernel_talker.md), at
# attended length L, for the kernel sources
# with this digest; null in the JSON line once the sources differ.
_STEP_TRAFFIC = {"asr": {"digest": "51c8f2ba2df52b4f", "bytes": 224889088 + 3907840, "L": 116},
                 "talker": {"digest": "51c8f2ba2df52b4f", "bytes": 896905472 + 4811520, "L": 70}}
_STEP_SOURCES = ("decode_persistent.cu", "decode_common.cuh", "qd_device.cuh")
# DRAM bytes of one batch_attn_kernel launch (profiles/batch_attn_kernel_batch64.md) at
# the initial lengths + 3, for the kernel sources with this digest.
_BATT_TRAFFIC = {"digest": "15451e5cfb3ef81d", "bytes": 260572160 + 3373568, "rows": 62239 + 3 * 64}
_BATT_SOURCES = ("batch_kernels.cu", "decode_common.cuh", "qd_device.cuh", "mma_sync.cuh", "qd_internal.h")


def _step_digest(sources=_STEP_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, "transformer_autoregressive_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _workload(name):
    import workloads as W
    s = W.CONFIGS[name]
    desc = {
        "asr": "ASR decoder: 8 layers, hidden 512, 8q/8kv heads x 64, FFN 2048, vocab 151936, EOS 151645 masked; "
               "prefill 110, greedy to KV length 400, buckets 128->256->512, batch 1",
        "talker": "Talker decoder: 28 layers, hidden 1024, 16q/8kv heads x 128, QK-norm, FFN 3072, vocab 3072, "
                  "repetition penalty 1.05; prefill 64, 600 greedy steps, buckets 128->256->512->1024, batch 1",
        "tiny": "tiny fp32 decoder: 1 layer, hidden 256, 4q/2kv x 64, FFN 768, vocab 1024; prefill 35, 8 steps",
    }[name]
    return s, desc


class Clocks:
    """nvidia-smi sampler running during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-i", str(gpu_index), "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _init_dist():
    """One process per GPU: (world size, rank, local rank, device); NCCL process group
    when launched by torchrun with more than one rank."""
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        if not dist.is_initialized():
            dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return ws, rank, local, torch.cuda.current_device()


def _close_dist(ws):
    if ws > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


def stream_shard(n_streams: int, rank: int, ws: int):
    """The streams [lo, hi) of the batched workload that rank `rank` of `ws` decodes:
    contiguous, disjoint, covering all of them (streams are independent decoders, so
    the ranks exchange nothing)."""
    return n_streams * rank // ws, n_streams * (rank + 1) // ws


def max_over_ranks(ms: float, ws: int) -> float:
    """The slowest rank's time of the timed region: every rank takes part (a MAX
    all-reduce on the process group's device; CPU tensors under gloo); one rank: ms."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, ws: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return ws * units_per_rank / (ms / 1e3)


# ------------------------------------------------------------------------------ oracle arm


def run_oracle_sample(shape, max_tokens: int, budget_s: float = 20.0):
    """Time the CPU oracle on a bounded sample of the workload: prefill (untimed),
    then up to ``max_tokens`` greedy decode tokens or ``budget_s`` seconds."""
    import oracle as O
    import workloads as W
    w = W.model_weights(shape)
    e = W.prefill_embeds(shape)
    o = O.Oracle(shape, w)
    tok, _, _ = o.prefill(embeds=e, want_logits=False)
    n = 0
    t0 = time.perf_counter()
    limit = min(max_tokens, shape.decode_steps)
    while n < limit:
        tok, _, _, _ = o.step(token=tok, want_logits=False)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    o.close()
    return n / dt, n, dt, O.num_threads()


def reference_arm(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    wl = "talker" if args.workload == "all" else args.workload
    shape, desc = _workload(wl)
    run_oracle_sample(shape, max(1, min(args.warmup, 3)), budget_s=5.0)  # warm-up (untimed)
    tps, n, dt, cores = run_oracle_sample(shape, args.steps, budget_s=60.0)
    sample = (f"prefill {shape.prefill} untimed, then {n} greedy decode tokens of the {wl} workload "
              f"({dt:.1f} s)")
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": ws,
            "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(n, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if shape.bf16 else "f32", "data": "synthetic",
            "config": {"workload": desc},
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------ GPU arm


def gpu_line(args, workload, ctx):
    """The decode workload `workload` (asr, talker, tiny) on this rank: its JSON line
    (rank 0) or None."""
    import numpy as np
    import torch

    ws, rank, local, dev = ctx
    import workloads as W
    import __graft_entry__
    __graft_entry__.build_library()
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, upload

    shape, desc = _workload(workload)
    hbm_peak, _, peak_src = _peaks()
    w_np = W.model_weights(shape)
    e_np = W.prefill_embeds(shape)
    dev_w = upload(w_np)
    h = qd.qd_create(dev_w, config_from_shape(shape))
    del dev_w
    e_dev = torch.from_numpy(e_np).cuda()
    traj = shape.decode_steps
    ids = torch.empty(traj, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def tokens(n, events=None):
        """Produce n decode tokens, continuing the trajectory in progress: a trajectory
        is reset + prefill + greedy decode to its end.  With ``events``, each greedy
        segment is bracketed by a pair of CUDA events (used to time the decode steps
        without the prefill)."""
        done = 0
        pos_state = tokens.pos
        while done < n:
            if pos_state == 0 or pos_state >= traj:
                qd.qd_reset(h)
                tokens.prefills += 1
                first = qd.qd_prefill(h, embeds=e_dev)
                if events is not None:
                    events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True), 1))
                    events[-1][0].record(stream)
                qd.qd_decode_greedy(h, 1, first, ids)
                if events is not None:
                    events[-1][1].record(stream)
                pos_state = 1
                done += 1
                continue
            k = min(n - done, traj - pos_state)
            if events is not None:
                events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True), k))
                events[-1][0].record(stream)
            qd.qd_decode_greedy(h, k, -1, ids)
            if events is not None:
                events[-1][1].record(stream)
            pos_state += k
            done += k
        tokens.pos = pos_state

    tokens.pos = 0
    tokens.prefills = 0
    W_ = max(3, args.warmup)
    tokens(W_)
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    k0, per_step = qd.qd_get_launch_count(h)
    # clocks sampled from the timed region through the long decode-only pass below
    clocks = Clocks(dev if ws == 1 else local)
    barrier()
    pos0 = tokens.pos
    pf0 = tokens.prefills
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    torch.cuda.nvtx.range_push("timed")
    tokens(args.steps)
    torch.cuda.nvtx.range_pop()
    ev1.record(stream)
    barrier()
    timed_prefills = tokens.prefills - pf0
    ms = ev0.elapsed_time(ev1)
    k1, _ = qd.qd_get_launch_count(h)
    ms = max_over_ranks(ms, ws)
    value = whole_job_rate(args.steps, ws, ms)

    # decode steps alone (prefill excluded): events around every greedy segment of
    # one more pass over whole trajectories
    tokens.pos = 0
    evs = []
    tokens(2 * traj, evs)
    torch.cuda.synchronize()
    dec_ms = sum(a.elapsed_time(b) for a, b, _ in evs)
    dec_n = sum(k for _, _, k in evs)
    dec_step_us = 1e3 * dec_ms / dec_n
    clk = clocks.stop()

    # the same decode steps with on-device sampling at the wrapper's default generation
    # settings ("qwen3-tts-hip OPTIMIZATION_LOG", generation-defaults entry: top-k 50,
    # temperature 0.9, top-p 1.0): the head's candidate selection and draw on top of
    # the greedy step
    qd.qd_set_sampling(h, 50, 0.9, 1.0, 1)
    tokens.pos = 0
    evs = []
    tokens(traj, evs)
    torch.cuda.synchronize()
    samp_step_us = 1e3 * sum(a.elapsed_time(b) for a, b, _ in evs) / sum(k for _, _, k in evs)
    qd.qd_set_sampling(h, 0, 1.0, 1.0, 0)


    # whole-step HBM fraction of the decode step (algorithmic bytes: weights + KV at
    # the mean attended length of the trajectory)
    L_avg = shape.prefill + 0.5 * (traj + 1)
    step_bytes = shape.step_bytes(int(round(L_avg)))
    step_gbs = step_bytes / (dec_step_us / 1e6) / 1e9

    # dominant kernel: the persistent decode-step kernel (every phase of the step in one
    # launch); its algorithmic bytes per launch are the step's weights plus the KV rows
    # it reads, at the position the handle holds after the timed region.
    pos_now, smax_now = qd.qd_get_pos(h)
    reps = max(1, min(64, smax_now - pos_now - 4))
    kms = qd.qd_time_kernel(h, qd.KERNEL_STEP, reps)
    L_timed = pos_now + (reps + 1) // 2 + 3
    kbytes = shape.step_bytes(L_timed)
    achieved = kbytes / (kms / 1e3) / 1e9
    traffic, traffic_note = None, "no ncu capture for this workload and kernel build"
    tr = _STEP_TRAFFIC.get(workload)
    if tr and tr["digest"] == _step_digest():
        # scaled from the captured length to the timed one by the K/V rows read
        traffic = tr["bytes"] + (L_timed - tr["L"]) * shape.kv_bytes_per_position()
        traffic_note = (f"ncu dram__bytes_read+write of one launch at L={tr['L']} "
                        f"({tr['bytes']} B), plus {shape.kv_bytes_per_position()} B of K/V per position to L={L_timed}")
    kname = ("decode_step_kernel: RMSNorm+QKV, attention, O-proj, RMSNorm+gate/up+SwiGLU, down for every layer, "
             "then RMSNorm+LM head+penalty+EOS mask+argmax, one cooperative launch")
    # the output-head GEMV alone (per-phase kernel) as a pure streaming reference
    head_bytes = shape.vocab * shape.hidden * (2 if shape.bf16 else 4)
    head_ms = qd.qd_time_kernel(h, qd.KERNEL_HEAD, 20)

    # the same head as weight-only 8-bit blocks (qd_quantize_q8 / qd_gemv_q8): 1 + 1/16
    # bytes per weight; the GEMV alone, on the HBM roofline, beside the bf16 head GEMV
    q8 = None
    if shape.bf16 and shape.hidden in (512, 1024, 2048):
        from transformer_autoregressive_decode_gb300.torch_io import to_device
        w_head = to_device(w_np["lm_head.0"])
        codes = torch.empty((shape.vocab, shape.hidden), dtype=torch.int8, device="cuda")
        scales = torch.empty((shape.vocab, shape.hidden // 32), dtype=torch.int16, device="cuda")
        qd.qd_quantize_q8(w_head, codes, scales)
        del w_head
        xq = torch.from_numpy(W.normal("bench/q8_x", (shape.hidden,), 0, 0.0, 1.0)).cuda()
        yq = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        # L2 flushed (256 MB written) before every timed launch: the codes fit in L2
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        ts = []
        for _ in range(12):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            qd.qd_gemv_q8(codes, scales, xq, yq)
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        del flush
        q8_ms = float(np.median(ts[2:]))
        q8_bytes = shape.vocab * shape.hidden * (1 + 2 / 32)
        q8 = {"kernel": "gemv_q8_kernel (qd_gemv_q8)", "rows": shape.vocab, "K": shape.hidden,
              "bytes": q8_bytes, "avg_launch_ms": q8_ms, "achieved_gbs": q8_bytes / (q8_ms / 1e3) / 1e9,
              "frac": q8_bytes / (q8_ms / 1e3) / 1e9 / hbm_peak, "peak_source": peak_src,
              "bf16_head_gemv_ms": head_ms,
              "note": "the LM head quantised to 32-weight blocks with half scales; median of 10 launches "
                      "(after 2), each between CUDA events after a 256 MB write that flushes L2"}
        del codes, scales
        # the same head as Q4_K super-blocks (qd_quantize_q4k / qd_gemv_q4k): 144 bytes
        # per 256 weights, timed the same way
        w_head = to_device(w_np["lm_head.0"])
        q4b = torch.empty((shape.vocab, shape.hidden // 256, 144), dtype=torch.uint8, device="cuda")
        qd.qd_quantize_q4k(w_head, q4b)
        del w_head
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        ts = []
        for _ in range(12):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            qd.qd_gemv_q4k(q4b, xq, yq)
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        del flush, q4b
        q4_ms = float(np.median(ts[2:]))
        q4_bytes = shape.vocab * shape.hidden * 144 / 256
        q8["q4k"] = {"kernel": "gemv_q4k_kernel (qd_gemv_q4k)", "bytes": q4_bytes, "avg_launch_ms": q4_ms,
                     "achieved_gbs": q4_bytes / (q4_ms / 1e3) / 1e9,
                     "frac": q4_bytes / (q4_ms / 1e3) / 1e9 / hbm_peak, "peak_source": peak_src,
                     "note": "Q4_K super-blocks (256 weights: half d and dm, 6-bit sub-block scales and mins, "
                             "4-bit codes); median of 10 launches (after 2), L2 flushed before each"}
        # the whole decode step with every layer matrix and the head as 8-bit rows
        # (qd_config.weight_q8): the same trajectory's decode steps, and the step kernel
        # against the quantised bytes
        hq = qd.qd_create(upload(w_np), config_from_shape(shape, weight_q8=True))
        qd.qd_reset(hq)
        first = qd.qd_prefill(hq, embeds=e_dev)
        qd.qd_decode_greedy(hq, 4, first, ids)
        nq = traj - 4
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        qd.qd_decode_greedy(hq, nq, -1, ids)
        b.record(stream)
        torch.cuda.synchronize()
        q8_step_us = 1e3 * a.elapsed_time(b) / nq
        qd.qd_reset(hq)
        first = qd.qd_prefill(hq, embeds=e_dev)
        qd.qd_decode_greedy(hq, traj // 2, first, ids)
        pq, sq = qd.qd_get_pos(hq)
        if sq - pq - 4 < 16:
            # too close to the bucket's end to time a few steps: past the migration
            qd.qd_decode_greedy(hq, 8, -1, ids)
            pq, sq = qd.qd_get_pos(hq)
        rq = max(1, min(64, sq - pq - 4))
        q8_kms = qd.qd_time_kernel(hq, qd.KERNEL_STEP, rq)
        Lq = pq + (rq + 1) // 2 + 3
        mp = shape.matrix_params()
        q8_wb = mp * (1 + 2 / 32) + (shape.weight_bytes_per_step() - 2 * mp)
        q8_kb = q8_wb + Lq * shape.kv_bytes_per_position()
        qd.qd_destroy(hq)
        q8["step"] = {"config": "weight_q8: every layer matrix and the head as 8-bit rows; embedding, norms, "
                                "KV cache bf16",
                      "decode_step_us": q8_step_us, "bf16_decode_step_us": dec_step_us,
                      "kernel_ms": q8_kms, "kernel_bytes": q8_kb, "L": Lq,
                      "achieved_gbs": q8_kb / (q8_kms / 1e3) / 1e9,
                      "frac": q8_kb / (q8_kms / 1e3) / 1e9 / hbm_peak, "peak_source": peak_src}

    # the codec decoder's convolution stages (fp32, CUDA cores: "alu" bound against the
    # fp32 FMA rate of 152 SMs x 128 lanes x 2 flops at the sampled SM clock), each launch
    # after a 256 MB write that flushes L2
    codec = None
    if workload == "asr":
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

        def timed(fn, reps=6):
            fn()
            ts = []
            for _ in range(reps):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            return float(np.median(ts[1:]))
        cx = torch.from_numpy(W.normal("bench/codec_x", (512, 4096), 0, 0.0, 1.0)).cuda()
        cw = torch.from_numpy(W.normal("bench/codec_w", (512, 512, 7), 0, 0.0, 0.02)).cuda()
        tw = torch.from_numpy(W.normal("bench/codec_tw", (512, 256, 8), 0, 0.0, 0.02)).cuda()
        tx = cx[:, :1024].contiguous()
        conv_ms = timed(lambda: qd.qd_conv1d_causal(cx, cw, None, dilation=1))
        tconv_ms = timed(lambda: qd.qd_conv_transpose1d_causal(tx, tw, None, stride=4))
        sm_mhz = (clk or {}).get("sm_mhz") or 2070.0
        alu_peak = 152 * 128 * 2 * sm_mhz * 1e6 / 1e12
        conv_flop = 2 * 512 * 512 * 7 * 4096
        tconv_flop = 2 * 512 * 256 * 2 * 1024 * 4
        conv_tf = conv_flop / (conv_ms / 1e3) / 1e12
        tconv_tf = tconv_flop / (tconv_ms / 1e3) / 1e12
        # the tensor-core forms (bf16 weights, x as bf16 hi + lo: two products per
        # k-step, counted once): weight packing, signal transpose and the GEMMs, 20 runs
        # back to back between CUDA events (the inputs, 15 MB, stay in L2)
        torch.cuda.nvtx.range_push("codec_conv_tc")
        _, conv_tc_ms = qd.qd_conv1d_causal_tc(cx, cw, None, dilation=1, time_reps=20)
        torch.cuda.nvtx.range_pop()
        torch.cuda.nvtx.range_push("codec_tconv_tc")
        _, tconv_tc_ms = qd.qd_conv_transpose1d_causal_tc(tx, tw, None, stride=4, time_reps=20)
        torch.cuda.nvtx.range_pop()
        _, bf16_peak, peak_src = _peaks()
        conv_tc_tf = conv_flop / (conv_tc_ms / 1e3) / 1e12
        tconv_tc_tf = tconv_flop / (tconv_tc_ms / 1e3) / 1e12
        codec = {"conv1d_causal": {"shape": "512 -> 512 channels, K 7, 4096 frames", "ms": conv_ms,
                                   "tflops": conv_tf, "frac": conv_tf / alu_peak},
                 "conv_transpose1d_causal": {"shape": "512 -> 256 channels, stride 4, 1024 -> 4096 frames",
                                             "ms": tconv_ms, "tflops": tconv_tf, "frac": tconv_tf / alu_peak},
                 "bound": "alu", "peak_tflops": alu_peak,
                 "note": "fp32 CUDA-core kernels (parity first); peak = 152 SMs x 128 fp32 lanes x 2 flops x SM "
                         "clock; median of 5 after a warm launch, L2 flushed before each",
                 "tensor_cores": {
                     "conv1d_causal_tc": {"ms": conv_tc_ms, "tflops": conv_tc_tf, "frac": conv_tc_tf / bf16_peak,
                                          "speedup": conv_ms / conv_tc_ms},
                     "conv_transpose1d_causal_tc": {"ms": tconv_tc_ms, "tflops": tconv_tc_tf,
                                                    "frac": tconv_tc_tf / bf16_peak,
                                                    "speedup": tconv_ms / tconv_tc_ms},
                     "bound": "tensor", "peak_tflops": bf16_peak, "peak_source": peak_src,
                     "note": "qd_*_tc: shifted-tap tcgen05 GEMMs (one per transposed-convolution phase) with the "
                             "bias in the epilogue; the time includes packing the weights to bf16 and the signal "
                             "to time-major hi/lo parts; mean of 20 back-to-back runs (inputs L2-resident)"}}
        del flush, cx, cw, tw, tx

    # end to end through the public API with host buffers: the prompt embeddings
    # come from pinned host memory each trajectory, the token goes in and the id
    # comes out through host memory every step (synchronising call)
    e_host = torch.from_numpy(e_np).pin_memory()
    e_buf = torch.empty_like(e_dev)
    n_e2e = min(args.steps, 4 * traj)
    barrier()
    t0 = time.perf_counter()
    done = 0
    h2d = d2h = 0
    while done < n_e2e:
        qd.qd_reset(h)
        e_buf.copy_(e_host, non_blocking=True)
        h2d += e_host.numel() * 4
        tok = qd.qd_prefill(h, embeds=e_buf)
        d2h += 12
        for _ in range(min(traj, n_e2e - done)):
            tok = qd.qd_decode_step(h, token=tok)
            h2d += 16
            d2h += 12
            done += 1
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e = {"value": ws * n_e2e / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d / n_e2e,
           "d2h_bytes_per_step": d2h / n_e2e, "api": "qd_prefill + qd_decode_step (host token in, host id out)",
           "steps": n_e2e}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        tps, n, dt, cores = run_oracle_sample(shape, shape.decode_steps, budget_s=20.0)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"prefill {shape.prefill} untimed, then {n} greedy decode tokens ({dt:.1f} s)"}

    qd.qd_destroy(h)
    # the same Talker weights with the interleaved multimodal RoPE sections [24, 20, 20]:
    # a prompt with distinct rotary streams (text, a 6 x 8 image grid, text) beside the
    # plain prompt
    mrope = None
    if workload == "talker":
        ms_shape = W.scaled(shape, name="talker_mrope", mrope_section=(24, 20, 20))
        dev_w = upload(w_np)
        hm = qd.qd_create(dev_w, config_from_shape(ms_shape))
        del dev_w

        def prefill_ms(positions, reps=10):
            ts = []
            for _ in range(reps):
                qd.qd_reset(hm)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                if positions is None:
                    qd.qd_prefill(hm, embeds=e_dev)
                else:
                    qd.qd_prefill_mrope(hm, positions, embeds=e_dev)
                b.record(stream)
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            return float(np.median(ts[2:]))
        grid = W.grid_prompt_positions(shape.prefill, shape.prefill // 6, 6, 8)
        mrope = {"section": [24, 20, 20], "prefill_ms_plain_positions": prefill_ms(None),
                 "prefill_ms_grid_positions": prefill_ms(grid),
                 "note": f"a second handle on the same weights with mRoPE sections: qd_prefill vs "
                         f"qd_prefill_mrope of the {shape.prefill}-position prompt (median of 8 after 2), "
                         "text + 6 x 8 image grid + text positions"}
        qd.qd_destroy(hm)
    if rank != 0:
        return None
    if timed_prefills:
        timed = (f"{args.steps} decode tokens continuing the trajectory at position {pos0} of {traj} "
                 f"(graph replays of the step); {timed_prefills} trajectory restart(s) inside, each a reset and "
                 f"a {shape.prefill}-position prefill, timed with the tokens")
    else:
        timed = (f"{args.steps} decode tokens continuing the trajectory at position {pos0} of {traj} "
                 f"(graph replays of the step; no prefill inside the timed region)")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": W_, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if shape.bf16 else "f32",
        "data": "synthetic: seeded N(0,0.02) " + ("bf16" if shape.bf16 else "fp32") +
                " weights, 1+N(0,0.1) norm gammas, N(0,1) prompt embeddings",
        "config": {"workload": desc, "storage": ("bf16 weights and KV cache" if shape.bf16 else
                                                 "fp32 weights and KV cache") + ", fp32 activations and accumulation",
                   "timed": timed,
                   "l2": f"inputs larger than L2: {shape.weight_bytes_per_step() / 1e6:.1f} MB of weights per step",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": traffic, "traffic_note": traffic_note, "kernel": kname,
                     "bytes_per_launch": kbytes, "avg_launch_ms": kms, "peak_source": peak_src,
                     "timing": f"CUDA events on the library stream around {reps} decode steps (graph replays) at "
                               f"positions {pos_now}..{pos_now + reps + 2}",
                     "head_gemv_alone": {"bytes": head_bytes, "avg_launch_ms": head_ms,
                                         "achieved_gbs": head_bytes / (head_ms / 1e3) / 1e9}},
        "step_hbm": {"bytes_per_step": step_bytes, "decode_step_us": dec_step_us,
                     "decode_tokens_per_s": 1e6 / dec_step_us, "achieved_gbs": step_gbs,
                     "frac": step_gbs / hbm_peak, "peak_source": peak_src,
                     "note": f"decode steps only (prefill excluded), {dec_n} steps timed with CUDA events around "
                             f"each device greedy segment; weights + KV at mean L={L_avg:.0f}"},
        "sampling": {"top_k": 50, "temperature": 0.9, "top_p": 1.0, "decode_step_us": samp_step_us,
                     "greedy_decode_step_us": dec_step_us,
                     "note": "the same decode trajectories with qd_set_sampling on: per-CTA top-k selection in "
                             "the head, last-CTA merge and counter-based draw"},
        **({"mrope": mrope} if mrope else {}),
        **({"q8_head_gemv": q8} if q8 else {}),
        **({"codec_conv": codec} if codec else {}),
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(k1 - k0), "kernels_per_decode_step": per_step,
        "clocks": clk,
    }
    return line


def gpu_arm(args):
    ctx = _init_dist()
    line = gpu_line(args, args.workload, ctx)
    if line is not None:
        print(json.dumps(line), flush=True)
    _close_dist(ctx[0])


# ------------------------------------------------------------------------------ frame workload

FRAME_TRAJ = 150
FRAMES_DESC = ("two-level frame generation: 28-layer Talker (hidden 1024, 16q/8kv heads x 128, QK-norm, FFN 3072, "
               "vocab 3072, repetition penalty 1.05) emits the primary code, a 5-layer Code Predictor (same dims, 15 "
               "heads of vocab 2048) the 15 residual codes; 16 code embeddings + N(0,1) text embedding feed the "
               "Talker; prefill 64, 150 frames per trajectory, Talker buckets 128->256, batch 1")


def run_oracle_frames(max_frames: int, budget_s: float = 20.0):
    """Time the oracle's frame loop on a bounded sample: Talker prefill (untimed),
    then up to ``max_frames`` frames or ``budget_s`` seconds."""
    import oracle as O
    import workloads as W
    ts, cs = W.TALKER, W.CODE_PREDICTOR
    tw = W.model_weights(ts)
    tabs = W.frame_tables()
    talker, cp = O.Oracle(ts, tw), O.Oracle(cs, W.model_weights(cs))
    loop = O.FrameLoop(talker, cp, tw["embed"], [tabs[f"code_embed.{j}"] for j in range(1, 16)])
    text = W.frame_text_embeds(FRAME_TRAJ)
    p, _, m = talker.prefill(embeds=W.prefill_embeds(ts), want_logits=False)
    n = 0
    t0 = time.perf_counter()
    while n < min(max_frames, FRAME_TRAJ - 1):
        # one frame: the predictor loop and the sum, then the Talker step
        _, _, nxt, _ = loop.generate(1, text[n:n + 1], p, m)
        p, _, m, _ = talker.step(token=p, embed=nxt[0], want_logits=False)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    talker.close()
    cp.close()
    return n / dt, n, dt, O.num_threads()


def frames_reference_arm(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    run_oracle_frames(1, budget_s=5.0)                       # warm-up (untimed)
    fps, n, dt, cores = run_oracle_frames(args.steps, budget_s=60.0)
    sample = f"Talker prefill 64 untimed, then {n} frames ({dt:.1f} s)"
    line = {"impl": "reference", "metric": METRIC, "value": fps, "unit": "frames/s", "n_gpus": ws,
            "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(n, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": FRAMES_DESC},
            "cpu_baseline": {"value": fps, "unit": "frames/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": fps, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def frames_line(args, ctx):
    """The two-level frame workload on this rank: its JSON line (rank 0) or None."""
    import numpy as np
    import torch

    ws, rank, local, dev = ctx
    import workloads as W
    import __graft_entry__
    __graft_entry__.build_library()
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, to_device, upload

    ts, cs = W.TALKER, W.CODE_PREDICTOR
    hbm_peak, _, peak_src = _peaks()
    T = qd.qd_create(upload(W.model_weights(ts)), config_from_shape(ts))
    C = qd.qd_create(upload(W.model_weights(cs)), config_from_shape(cs))
    tabs = W.frame_tables()
    F = qd.qd_frame_create(T, C, [to_device(tabs[f"code_embed.{j}"]) for j in range(1, 16)], True)
    prompt_np = W.prefill_embeds(ts)
    text_np = W.frame_text_embeds(FRAME_TRAJ)
    prompt = torch.from_numpy(prompt_np).cuda()
    text = torch.from_numpy(text_np).cuda()
    codes = torch.empty((FRAME_TRAJ, 16), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def frames(n, events=None):
        """n frames as trajectories of up to 150 (reset + Talker prefill + frames)."""
        done = 0
        while done < n:
            k = min(FRAME_TRAJ, n - done)
            qd.qd_reset(T)
            qd.qd_prefill(T, embeds=prompt)
            if events is not None:
                events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True), k))
                events[-1][0].record(stream)
            qd.qd_frame_generate(F, k, text, codes)
            if events is not None:
                events[-1][1].record(stream)
            done += k

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    W_ = max(3, args.warmup)
    frames(W_)
    barrier()
    kt0, _ = qd.qd_get_launch_count(T)
    kc0, _ = qd.qd_get_launch_count(C)
    clocks = Clocks(dev if ws == 1 else local)
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    frames(args.steps)
    ev1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    kt1, _ = qd.qd_get_launch_count(T)
    kc1, _ = qd.qd_get_launch_count(C)
    ms = max_over_ranks(ms, ws)
    value = whole_job_rate(args.steps, ws, ms)

    # frame loop alone (Talker prefill excluded), two trajectories
    evs = []
    frames(2 * FRAME_TRAJ, evs)
    torch.cuda.synchronize()
    loop_ms = sum(a.elapsed_time(b) for a, b, _ in evs)
    loop_n = sum(k for _, _, k in evs)
    frame_us = 1e3 * loop_ms / loop_n
    traj_bytes = sum(W.frame_bytes(ts.prefill + f + 1, talker_step=f < FRAME_TRAJ - 1) for f in range(FRAME_TRAJ))
    frame_bytes = traj_bytes / FRAME_TRAJ
    frame_gbs = frame_bytes / (frame_us / 1e6) / 1e9

    # the step kernel on each model: predictor steps (positions 16..) and Talker steps
    # at the positions the handles hold after a trajectory
    pc, sc = qd.qd_get_pos(C)
    reps_c = max(1, min(12, sc - pc - 4))
    c_ms = qd.qd_time_kernel(C, qd.KERNEL_STEP, reps_c)
    c_bytes = cs.step_bytes(pc + (reps_c + 1) // 2 + 3)
    pt, st_ = qd.qd_get_pos(T)
    reps_t = max(1, min(32, st_ - pt - 4))
    t_ms = qd.qd_time_kernel(T, qd.KERNEL_STEP, reps_t)
    t_bytes = ts.step_bytes(pt + (reps_t + 1) // 2 + 3)
    c_gbs = c_bytes / (c_ms / 1e3) / 1e9

    # end to end through the public API: prompt and text embeddings from pinned host
    # memory every trajectory, the codes back to host memory
    prompt_h = torch.from_numpy(prompt_np).pin_memory()
    text_h = torch.from_numpy(text_np).pin_memory()
    codes_h = torch.empty((FRAME_TRAJ, 16), dtype=torch.int32).pin_memory()
    n_e2e = min(args.steps, 2 * FRAME_TRAJ)
    barrier()
    t0 = time.perf_counter()
    done = h2d = d2h = 0
    while done < n_e2e:
        k = min(FRAME_TRAJ, n_e2e - done)
        qd.qd_reset(T)
        prompt.copy_(prompt_h, non_blocking=True)
        text[:k].copy_(text_h[:k], non_blocking=True)
        h2d += prompt_h.numel() * 4 + k * ts.hidden * 4
        qd.qd_prefill(T, embeds=prompt)
        d2h += 12
        qd.qd_frame_generate(F, k, text, codes)
        codes_h[:k].copy_(codes[:k], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        d2h += k * 16 * 4
        done += k
    e2e_s = time.perf_counter() - t0
    e2e = {"value": ws * n_e2e / e2e_s, "unit": "frames/s", "h2d_bytes_per_step": h2d / n_e2e,
           "d2h_bytes_per_step": d2h / n_e2e, "steps": n_e2e,
           "api": "qd_prefill + qd_frame_generate (host embeddings in, host codes out per trajectory)"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        fps, n, dt, cores = run_oracle_frames(FRAME_TRAJ, budget_s=20.0)
        cpu = {"value": fps, "unit": "frames/s", "cores": cores, "kind": "oracle",
               "sample": f"Talker prefill 64 untimed, then {n} frames ({dt:.1f} s)"}

    qd.qd_frame_destroy(F)
    qd.qd_destroy(C)
    qd.qd_destroy(T)
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": ws, "steps": args.steps,
        "warmup": W_, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,0.02) bf16 weights and code tables, 1+N(0,0.1) norm gammas, N(0,1) prompt "
                "and text embeddings",
        "config": {"workload": FRAMES_DESC, "storage": "bf16 weights, tables and KV cache, fp32 activations",
                   "timed": f"{args.steps} frames as whole trajectories (reset + Talker prefill 64 + frames), "
                            "prefill time included; a step is one frame (16 codes)",
                   "l2": f"inputs larger than L2: {frame_bytes / 1e9:.2f} GB of weights per frame",
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "codes_per_s": 16 * value,
        "roofline": {"bound": "hbm", "achieved": c_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": c_gbs / hbm_peak,
                     "traffic": None, "traffic_note": "no ncu capture for this workload and kernel build",
                     "kernel": "decode_step_kernel on the Code Predictor (5 layers + one of 15 heads per launch)",
                     "bytes_per_launch": c_bytes, "avg_launch_ms": c_ms, "peak_source": peak_src,
                     "timing": f"CUDA events around {reps_c} predictor steps at positions {pc}..{pc + reps_c + 2}",
                     "talker_step": {"bytes": t_bytes, "avg_launch_ms": t_ms,
                                     "achieved_gbs": t_bytes / (t_ms / 1e3) / 1e9}},
        "frame_hbm": {"bytes_per_frame": frame_bytes, "frame_us": frame_us, "frames_per_s": 1e6 / frame_us,
                      "achieved_gbs": frame_gbs, "frac": frame_gbs / hbm_peak, "peak_source": peak_src,
                      "note": f"frame loop only (Talker prefill excluded), {loop_n} frames timed with CUDA events "
                              "around each qd_frame_generate call; algorithmic bytes per frame averaged over a "
                              "trajectory (149 Talker steps, 150 x 15 predictor weight passes)"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(kt1 - kt0 + kc1 - kc0), "clocks": clk,
    }
    return line


def frames_arm(args):
    ctx = _init_dist()
    line = frames_line(args, ctx)
    if line is not None:
        print(json.dumps(line), flush=True)
    _close_dist(ctx[0])


# ------------------------------------------------------------------------------ batched workload

BATCH_DESC = ("batched multi-stream decode: 64 independent streams of the 28-layer Talker (hidden 1024, 16q/8kv "
              "heads x 128, QK-norm, FFN 3072, vocab 3072, repetition penalty 1.05), each with its own bf16 cache "
              "(smax 2048) filled with N(0,1) K/V to a seeded length U{256..1792} and a seeded first token; 256 "
              "greedy steps per stream; projections, MLP and head as tcgen05 GEMMs over the 64 streams")


def run_oracle_batch_stream(max_steps: int, budget_s: float = 20.0):
    """The oracle decoding one stream of the batched workload (stream 0: its cache and
    first token), up to max_steps or budget_s seconds; stream-tokens/s."""
    import oracle as O
    import workloads as W
    s = W.TALKER
    L0 = int(W.batch_initial_lengths()[0])
    o = O.Oracle(s, W.model_weights(s), buckets=(W.BATCH_SMAX,))
    o.set_kv(W.batch_stream_kv(s, 0, L0), L0)
    tok = int(W.batch_first_tokens(W.BATCH_STREAMS, s.vocab)[0])
    n = 0
    t0 = time.perf_counter()
    while n < max_steps:
        tok, _, _, _ = o.step(token=tok, want_logits=False)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    o.close()
    return n / dt, n, dt, O.num_threads(), L0


def batch_reference_arm(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    run_oracle_batch_stream(1, budget_s=5.0)
    tps, n, dt, cores, L0 = run_oracle_batch_stream(args.steps, budget_s=60.0)
    sample = f"stream 0 of the batched workload (cache length {L0}), {n} greedy steps ({dt:.1f} s)"
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "stream-tokens/s", "n_gpus": ws,
            "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * dt / max(n, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": BATCH_DESC},
            "cpu_baseline": {"value": tps, "unit": "stream-tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": tps, "unit": "stream-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def batch_line(args, ctx):
    """The batched workload on this rank: its JSON line (rank 0) or None.  With more
    than one rank the 64 streams are partitioned: rank r decodes streams
    stream_shard(64, r, N) over a full weight replica, with no exchange."""
    import numpy as np
    import torch

    ws, rank, local, dev = ctx
    import workloads as W
    import __graft_entry__
    __graft_entry__.build_library()
    import transformer_autoregressive_decode_gb300 as qd
    from transformer_autoregressive_decode_gb300.torch_io import config_from_shape, to_device, upload

    s = W.TALKER
    if args.layers:
        # profiling case only: the same streams, lengths and per-layer kernels, fewer layers
        s = W.scaled(W.TALKER, n_layers=args.layers, name=f"talker{args.layers}")
    B_all, smax, traj = W.BATCH_STREAMS, W.BATCH_SMAX, W.BATCH_STEPS
    lo, hi = stream_shard(B_all, rank, ws)       # this rank's streams (all of them on one GPU)
    B = hi - lo
    hbm_peak, bf16_peak, peak_src = _peaks()
    h = qd.qd_create(upload(W.model_weights(s)), config_from_shape(s))
    bh = qd.qd_batch_create(h, B, smax)
    lens = [int(v) for v in W.batch_initial_lengths()][lo:hi]
    toks = [int(v) for v in W.batch_first_tokens(B_all, s.vocab)][lo:hi]
    kv_dev = [to_device(W.batch_stream_kv(s, lo + b, lens[b])) for b in range(B)]   # kept for restarts
    ids = torch.empty((traj, B), dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def restart():
        for b in range(B):
            qd.qd_batch_set_stream(bh, b, kv_dev[b], lens[b], toks[b])
        steps.pos = 0

    def steps(n):
        """n batched steps; a trajectory is 256 steps from the initial caches."""
        done = 0
        while done < n:
            if steps.pos >= traj:
                restart()
            k = min(n - done, traj - steps.pos)
            qd.qd_batch_decode(bh, k, ids[steps.pos:steps.pos + k])
            steps.pos += k
            done += k

    restart()
    W_ = max(3, args.warmup)
    steps(W_)
    qd.qd_batch_sync(bh)

    # per-kernel times at the start of a trajectory (positions = the initial lengths)
    restart()
    kms = {name: qd.qd_batch_time_kernel(bh, which, 10) for name, which in (
        ("attention", qd.BATCH_ATTENTION), ("qkv", qd.BATCH_QKV), ("oproj", qd.BATCH_OPROJ),
        ("gate_up", qd.BATCH_GATE_UP), ("down", qd.BATCH_DOWN), ("head", qd.BATCH_HEAD))}
    restart()
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    k0, per_step = qd.qd_batch_get_launch_count(bh)
    clocks = Clocks(dev if ws == 1 else local)
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    steps(args.steps)
    ev1.record(stream)
    barrier()
    clk = clocks.stop()
    qd.qd_batch_sync(bh)
    ms = ev0.elapsed_time(ev1)
    k1, _ = qd.qd_batch_get_launch_count(bh)
    ms = max_over_ranks(ms, ws)
    value = B_all * args.steps / (ms / 1e3)      # every stream of the workload over the slowest rank
    step_ms = ms / args.steps

    # algorithmic bytes: weights once per step + every stream's K/V over its attended
    # length (mean over a trajectory)
    kv_pos = s.kv_bytes_per_position()
    mean_L = sum(L + (traj + 1) / 2 for L in lens) / B
    step_bytes = s.weight_bytes_per_step() + B * mean_L * kv_pos
    step_gbs = step_bytes / (step_ms / 1e3) / 1e9
    # dominant kernel: attention of one layer, at the initial lengths (L = L0 + 1)
    att_bytes = sum(L + 1 for L in lens) * kv_pos / s.n_layers
    att_gbs = att_bytes / (kms["attention"] / 1e3) / 1e9
    att_traffic, att_note = None, "no ncu capture for this kernel build"
    if not args.layers and _BATT_TRAFFIC["digest"] == _step_digest(_BATT_SOURCES):
        rows = sum(L + 1 for L in lens)
        att_traffic = _BATT_TRAFFIC["bytes"] * rows / _BATT_TRAFFIC["rows"]
        att_note = (f"ncu dram__bytes_read+write of one launch with {_BATT_TRAFFIC['rows']} cached rows per group "
                    f"({_BATT_TRAFFIC['bytes']} B), scaled to {rows} rows")
    # the GEMMs: useful flops per step and their summed kernel time
    layer_params = s.layer_matrix_params()
    gemm_ms = s.n_layers * (kms["qkv"] + kms["oproj"] + kms["gate_up"] + kms["down"]) + kms["head"]
    gemm_flops = 2.0 * B * (s.n_layers * layer_params + s.vocab * s.hidden)
    gemm_tflops = gemm_flops / (gemm_ms / 1e3) / 1e12
    gemm_bytes = s.weight_bytes_per_step()

    # prefill of the workload: 8 prompt streams x 512 N(0,1) positions, timed alone
    ns_p, n_p = W.BATCH_PREFILL
    ns_p = min(ns_p, B)                         # this rank's share of the prompt streams fits its streams
    prompts = torch.from_numpy(np.stack([W.normal(f"batched/prompt/{i}", (n_p, s.hidden), 0)
                                         for i in range(ns_p)])).cuda()
    first = torch.empty(ns_p, dtype=torch.int32, device="cuda")
    pstreams = list(range(ns_p))
    for _ in range(2):
        qd.qd_batch_prefill(bh, pstreams, prompts, first)
    qd.qd_batch_sync(bh)
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    torch.cuda.nvtx.range_push("prefill")
    pe0.record(stream)
    for _ in range(reps):
        qd.qd_batch_prefill(bh, pstreams, prompts, first)
    pe1.record(stream)
    torch.cuda.nvtx.range_pop()
    qd.qd_batch_sync(bh)
    prefill_ms = pe0.elapsed_time(pe1) / reps
    T_p = ns_p * n_p
    pf_gemm_flops = 2.0 * T_p * s.n_layers * layer_params + 2.0 * ns_p * s.vocab * s.hidden
    pf_attn_flops = 4.0 * s.n_layers * ns_p * s.n_q_heads * s.head_dim * (n_p * (n_p + 1) / 2)
    pf_tflops = (pf_gemm_flops + pf_attn_flops) / (prefill_ms / 1e3) / 1e12
    prefill = {"streams": ns_p, "positions": n_p, "ms": prefill_ms, "tokens_per_s": T_p / (prefill_ms / 1e3),
               "useful_tflop": (pf_gemm_flops + pf_attn_flops) / 1e12, "useful_tflops": pf_tflops,
               "tensor_frac_useful": pf_tflops / bf16_peak, "bf16_peak_tflops": bf16_peak,
               "note": "qd_batch_prefill between CUDA events, mean of 5 after 2 warm-up calls; useful flops = "
                       "2 x tokens x weights (GEMMs) + causal attention; the hi/lo activation split issues two "
                       "MMAs per useful one"}

    # end to end: every step the 64 input tokens come from pinned host memory and the
    # 64 ids go back to it (the ids of a step are the next step's tokens)
    restart()
    n_e2e = min(args.steps, 64)
    tok_h = torch.tensor(toks, dtype=torch.int32).pin_memory()
    ids_h = torch.empty(B, dtype=torch.int32).pin_memory()
    force = torch.empty((1, B), dtype=torch.int32, device="cuda")
    one = torch.empty((1, B), dtype=torch.int32, device="cuda")
    barrier()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        force[0].copy_(tok_h, non_blocking=True)
        qd.qd_batch_decode(bh, 1, one, force)
        ids_h.copy_(one[0], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        tok_h.copy_(ids_h)
    e2e_s = time.perf_counter() - t0
    e2e = {"value": B_all * n_e2e / e2e_s, "unit": "stream-tokens/s", "h2d_bytes_per_step": 4 * B,
           "d2h_bytes_per_step": 4 * B, "steps": n_e2e,
           "api": "qd_batch_decode one step per call, tokens in from and ids out to pinned host memory"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        tps, n, dt, cores, L0 = run_oracle_batch_stream(traj, budget_s=20.0)
        cpu = {"value": tps, "unit": "stream-tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"stream 0 (cache length {L0}), {n} greedy steps ({dt:.1f} s)"}

    qd.qd_batch_destroy(bh)
    qd.qd_destroy(h)
    del kv_dev
    if rank != 0:
        return None
    line = {
        "metric": METRIC, "value": value, "unit": "stream-tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": W_, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "strong" if ws > 1 else "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,0.02) bf16 weights, 1+N(0,0.1) gammas, N(0,1) bf16 initial caches",
        "config": {"workload": BATCH_DESC if not args.layers else
                   f"PROFILING CASE, not the workload: {args.layers}-layer variant of: " + BATCH_DESC,
                   "storage": "bf16 weights and caches; activations fp32, entering the "
                                                      "GEMMs as bf16 hi + lo parts; fp32 accumulation",
                   "timed": f"{args.steps} batched steps (each 64 stream-tokens) from the initial caches",
                   "l2": f"inputs larger than L2: {step_bytes / 1e9:.2f} GB per step",
                   "parallelism": (f"streams partitioned: rank r of {ws} decodes streams "
                                   f"[64 r / {ws}, 64 (r + 1) / {ws}) over a full weight replica, no exchange")
                                  if ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": att_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": att_gbs / hbm_peak, "traffic": att_traffic, "traffic_note": att_note,
                     "kernel": "batch_attn_kernel: one layer's attention of all 64 streams over their caches "
                               "(QK-norm, RoPE, KV append, 8-way split, cluster merge)",
                     "bytes_per_launch": att_bytes, "avg_launch_ms": kms["attention"], "peak_source": peak_src,
                     "timing": "CUDA events around 10 graph-captured launches at the initial lengths"},
        "step_hbm": {"bytes_per_step": step_bytes, "step_ms": step_ms, "achieved_gbs": step_gbs,
                     "frac": step_gbs / hbm_peak, "peak_source": peak_src,
                     "note": f"weights {s.weight_bytes_per_step() / 1e9:.3f} GB + K/V of every stream at the "
                             f"trajectory's mean attended length {mean_L:.0f}"},
        "gemm": {"kernel_ms": {k: v for k, v in kms.items() if k != "attention"},
                 "per_step_ms": gemm_ms, "useful_tflops": gemm_tflops,
                 "tensor_frac_useful": gemm_tflops / bf16_peak, "bf16_peak_tflops": bf16_peak,
                 "weight_gbs": gemm_bytes / (gemm_ms / 1e3) / 1e9,
                 "note": "useful flops 2 x 64 x weights per step; the hi/lo activation split issues two MMAs per "
                         "useful one; at 64 streams the GEMMs stream their weights (HBM-bound)"},
        "prefill": prefill,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(k1 - k0), "kernels_per_step": per_step,
        "clocks": clk,
    }
    return line


def batch_arm(args):
    ctx = _init_dist()
    line = batch_line(args, ctx)
    if line is not None:
        print(json.dumps(line), flush=True)
    _close_dist(ctx[0])


def all_arm(args):
    """The default line: the Talker decode step (the DRAM-bound batch-1 decoder the metric
    is about) as the headline, with the ASR decoder, the two-level frame loop and the
    batched multi-stream decode as keys of the same line, each with its own value,
    roofline, CPU baseline and end-to-end number.  The --steps / --warmup arguments apply
    to the headline and the ASR decoder (decode tokens); the frame loop runs one
    150-frame trajectory and the batched decode 64 steps of its 256."""
    import copy
    ctx = _init_dist()
    line = gpu_line(args, "talker", ctx)
    sub = {}
    sub["asr"] = gpu_line(args, "asr", ctx)
    fa = copy.copy(args)
    fa.steps, fa.warmup = FRAME_TRAJ, 8
    sub["frames"] = frames_line(fa, ctx)
    ba = copy.copy(args)
    ba.steps, ba.warmup, ba.layers = 64, 8, 0
    sub["batch"] = batch_line(ba, ctx)
    if line is not None:
        for k, v in sub.items():
            line[k] = v
        line["config"]["also"] = ("keys asr, frames and batch: the ASR decoder, the two-level frame loop and the "
                                  "batched 64-stream decode, each measured in this run with its own value, "
                                  "roofline, cpu_baseline and e2e")
        print(json.dumps(line), flush=True)
    _close_dist(ctx[0])


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all", choices=["all", "asr", "talker", "tiny", "frames", "batch"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="batch workload only: run a variant with this many layers (a profiling case)")
    args = ap.parse_args()
    if args.workload == "frames":
        if args.steps == ap.get_default("steps"):
            args.steps = 4 * FRAME_TRAJ
        if args.warmup == ap.get_default("warmup"):
            args.warmup = FRAME_TRAJ
    if args.workload == "batch":
        if args.steps == ap.get_default("steps"):
            args.steps = 256
        if args.warmup == ap.get_default("warmup"):
            args.warmup = 8
    ref = {"frames": frames_reference_arm, "batch": batch_reference_arm}.get(args.workload, reference_arm)
    ours = {"frames": frames_arm, "batch": batch_arm, "all": all_arm}.get(args.workload, gpu_arm)
    (ref if args.impl == "reference" else ours)(args)


if __name__ == "__main__":
    main()
