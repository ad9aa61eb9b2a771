#!/usr/bin/env python
"""Benchmark of the GDN layer hot path on GB300.

Headline step: one fused GDN decode step (conv roll + conv + SiLU + L2 norm +
gates + gated delta rule) in the Qwen3-Next geometry (Hk=16, Hv=32, dk=dv=128,
8192 conv channels, width 4, bf16 conv cache, fp32 state) for B=256 rows
through a shuffled slot table over 512 slots. Metric: algorithmic HBM GB/s of
that step. Also reported: the decode batch sweep, the B=1024-over-2048-slot
case, and chunked-prefill tokens/s on one 4096-token sequence and on ~32k
packed varlen tokens.

Timing: W untimed warm-up steps, then exactly K timed steps. Each step is
bracketed by CUDA events on the stream the library launches on; L2 is flushed
between timed steps, outside the events: a 512 MiB buffer is overwritten, then a
256 MiB buffer is read, so that the dirty lines of the write are written back
before the step rather than during it.
Multi-GPU (torchrun): every rank runs its own workload on its own GPU (weak
scaling, no data-path collective); the step time is the max over ranks.

--impl reference times the fp64 CPU oracle (the only reference this build
has) on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("GDN decode HBM GB/s (% of peak) and chunked-prefill tokens/s per layer, 1 GB300")
HEADLINE_B = 256
NUM_SLOTS = 512
FALLBACK_HBM_GBS = 6800.0


def decode_bytes(B, geo, conv_f32=False, bias=True, out_bytes=2, state_bytes=4, gated=False):
    """Algorithmic bytes of one decode step: per row the state read + write (fp32, or bf16
    with state_bytes=2), x, the conv window read + write, the output and the gate inputs
    and slot; per call the conv weight and bias and the per-head gate parameters. With the
    output gate, per row the bf16 z and per call the fp32 norm weight."""
    s = 4 if conv_f32 else 2
    D = geo.D
    per_row = (2 * geo.Hv * geo.dv * geo.dk * state_bytes + 2 * D + 2 * D * (geo.W - 1) * s
               + out_bytes * geo.Hv * geo.dv + 2 * 2 * geo.Hv + 4)
    per_call = 2 * D * geo.W + (2 * D if bias else 0) + 8 * geo.Hv
    if gated:
        per_row += 2 * geo.Hv * geo.dv
        per_call += 4 * geo.dv
    return B * per_row + per_call


def prefill_flops_per_token(geo, C=64):
    """Dense-tile FLOPs per token of the chunked form (Gram and QK^T shared per k-head)."""
    dk, dv, r = geo.dk, geo.dv, geo.Hv // geo.Hk
    per_chunk_head = 2 * (C * C * dk / r * 2 + C * C * dv + C * C * dk + 2 * C * dk * dv
                          + C * C * dv + dv * C * dk)
    return per_chunk_head * geo.Hv / C


def prefill_bytes(T, N, geo, conv=True, conv_s=2):
    D = geo.D
    per_tok = 2 * D + 2 * 2 * geo.Hv + 2 * geo.Hv * geo.dv
    per_seq = 2 * geo.Hv * geo.dv * geo.dk * 4 + (2 * D * (geo.W - 1) * conv_s if conv else 0)
    return T * per_tok + N * per_seq


FALLBACK_BF16_TFLOPS = 1900.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def load_bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_digest():
    h = hashlib.sha256()
    for f in ("gdn_decode.cu", "gdn_common.cuh", "gdn_ptx.cuh"):
        with open(os.path.join(ROOT, "gated_deltanet_linear_gdn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(state="f32", batch=None, num_slots=None):
    """Per-launch DRAM bytes of the headline decode kernel (fp32 or bf16 state) from the
    committed ncu summary, if it was taken on the current kernel source and on this
    workload (rows, slot pool); else None."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    if j.get("source_digest") != kernel_source_digest():
        return None
    e = j.get("launches", {}).get(state)
    if e is None or e.get("batch") != batch or e.get("num_slots") != num_slots:
        return None
    return e


def prefill_launches(T, N, Hv, C, conv):
    """Kernels one tensor-core prefill call launches: prep (+ the conv and its final-window
    kernel), then an intra and a pass kernel per piece of the chunks. The piece rule is the
    library's (a call with at most 64 (sequence, value head) pairs and at least 16 chunks runs
    in pieces that grow by half, the first max(4, chunks / 8) long), restated here to count."""
    M = (T + N * (C - 1)) // C
    pieces = 1
    if N * Hv <= 64 and M >= 16:
        n, g, pieces = max(4, M // 8), 0, 0
        while g < M and pieces < 15:
            left = M - g
            g += left if (pieces == 14 or left < n + n // 2) else n
            pieces += 1
            n = n * 3 // 2
    return 1 + (2 if conv else 0) + 2 * pieces


def aggregate_ranks(mean_ms: float, bytes_per_rank: int, world: int, device=None):
    """Whole-job throughput over `world` ranks, each running its own copy of the workload:
    the step time is the max over ranks, the bytes are the sum. Returns (max_ms, GB/s).
    Uses torch.distributed (a timing-only reduction, not part of the data path)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        x = torch.tensor([mean_ms], dtype=torch.float64, device=device)
        dist.all_reduce(x, op=dist.ReduceOp.MAX)
        mean_ms = float(x.item())
    return mean_ms, bytes_per_rank * world / (mean_ms * 1e-3) / 1e9


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(ROOT, f".clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------- our arm

def run_ours(args, rank, world):
    import torch

    import gated_deltanet_linear_gdn_gb300 as gdn
    from gated_deltanet_linear_gdn_gb300 import inputs as gi

    gdn.lib()  # fails loudly if the CUDA library is missing
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    geo = gi.QWEN3_NEXT
    dims = gdn.Dims(geo.Hk, geo.Hv, geo.dk, geo.dv, geo.W)
    flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(64 << 20, dtype=torch.float32, device=dev)

    def flush():
        # a 512 MiB write evicts the workload from L2; the 256 MiB read after it replaces the
        # write's dirty lines with clean ones, so no write-back of the flush lands in the
        # timed step
        flush_buf.fill_(1)
        flush_rd.sum()

    def b16(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)

    def decode_setup(B, num_slots, seed, conv_f32=False, bias=True, silu=True, state_bf16=False):
        inp = gi.make_inputs(geo, [1] * B, num_slots, seed, state_pool=False, conv_f32=conv_f32,
                             bias=bias, silu=silu)
        t = dict(
            mixed=b16(inp.mixed).to(dev), a=b16(inp.a).to(dev), b=b16(inp.b).to(dev),
            A_log=torch.from_numpy(inp.A_log).to(dev), dt_bias=torch.from_numpy(inp.dt_bias).to(dev),
            conv_w=b16(inp.conv_w).to(dev), conv_b=None if inp.conv_b is None else b16(inp.conv_b).to(dev),
            conv=(torch.from_numpy(inp.conv_state) if conv_f32 else b16(inp.conv_state)).to(dev),
            ssm=gi.device_state_pool(num_slots, geo, 0.05, seed + 7, dev,
                                     dtype=torch.bfloat16 if state_bf16 else torch.float32),
            slot=torch.from_numpy(inp.slot).to(dev),
            out=torch.empty(B, geo.Hv, geo.dv, dtype=torch.bfloat16, device=dev),
            silu=silu, inp=inp)
        return t

    def decode_call(t, gate=None):
        gdn.gdn_decode_step(t["mixed"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["conv_w"],
                            t["conv_b"], t["conv"], t["ssm"], t["slot"], t["out"], dims,
                            silu=t["silu"], gate=gate, stream=stream)

    def central(ms):
        """Mean of the middle 80% of single-call times (of all but the extremes for fewer than 10). The events resolve about 1 us here, so a
        median of short calls sits on a tick; the trimmed mean averages the rounding out and
        still drops outliers."""
        x = np.sort(np.asarray(ms, dtype=np.float64))
        k = len(x) // 10 if len(x) >= 10 else min(1, (len(x) - 1) // 2)
        return float(np.mean(x[k:len(x) - k]))

    def timed(fn, steps, warmup, do_flush=True):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for e0, e1 in ev:
            if do_flush:
                flush()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return [e0.elapsed_time(e1) for e0, e1 in ev]

    result = {}
    clocks = ClockSampler(dev.index).start() if rank == 0 else None

    # ---- decode sweep (context) ----
    sweep = {}
    if not args.no_sweep:
        for B in (1, 2, 4, 8, 16, 64, 256):
            t = decode_setup(B, NUM_SLOTS, seed=B)
            ms = central(timed(lambda: decode_call(t), 50, 3))
            nb = decode_bytes(B, geo)
            sweep[str(B)] = {"us": round(ms * 1e3, 2), "GBps": round(nb / ms / 1e6, 1)}
            del t
        # CUDA-graph buckets (one replay = one graph launch of the fused step)
        for B in (1, 4, 16, 64, 256, 1024):
            t = decode_setup(B, NUM_SLOTS if B <= 256 else 2048, seed=B)
            g = gdn.DecodeGraph(t["mixed"], t["a"], t["b"], t["A_log"], t["dt_bias"], t["conv_w"],
                                t["conv_b"], t["conv"], t["ssm"], t["slot"], t["out"], dims)
            ms = central(timed(lambda: g.launch(stream), 50, 3))
            sweep[f"graph_c{B}"] = {"us": round(ms * 1e3, 2),
                                    "GBps": round(decode_bytes(B, geo) / ms / 1e6, 1)}
            g.close()
            del t
        for conv_f32 in (False, True):
            t = decode_setup(1024, 2048, seed=5, conv_f32=conv_f32)
            ms = central(timed(lambda: decode_call(t), 10, 2))
            nb = decode_bytes(1024, geo, conv_f32=conv_f32)
            key = "1024_of_2048_" + ("f32cache" if conv_f32 else "bf16cache")
            sweep[key] = {"us": round(ms * 1e3, 2), "GBps": round(nb / ms / 1e6, 1)}
            del t
        # bf16 recurrent state: half the state bytes per row
        for B, ns in ((HEADLINE_B, NUM_SLOTS), (1024, 2048)):
            t = decode_setup(B, ns, seed=6, state_bf16=True)
            ms = central(timed(lambda: decode_call(t), 20, 3))
            nb = decode_bytes(B, geo, state_bytes=2)
            sweep[f"bf16state_{B}_of_{ns}"] = {"us": round(ms * 1e3, 2),
                                               "GBps": round(nb / ms / 1e6, 1)}
            del t
        # the output gate (gated RMSNorm with z) fused into the step
        t = decode_setup(HEADLINE_B, NUM_SLOTS, seed=HEADLINE_B)
        gz = torch.randn(HEADLINE_B, geo.Hv, geo.dv, device=dev).to(torch.bfloat16)
        gw = torch.ones(geo.dv, device=dev)
        og = gdn.OutputGate(gz, gw)
        ms = central(timed(lambda: decode_call(t, og), 20, 3))
        nb = decode_bytes(HEADLINE_B, geo, gated=True)
        sweep[f"gated_{HEADLINE_B}_of_{NUM_SLOTS}"] = {"us": round(ms * 1e3, 2),
                                                      "GBps": round(nb / ms / 1e6, 1)}
        del t, gz, gw, og
        torch.cuda.empty_cache()

    # ---- chunked prefill ----
    prefill = {}
    cases = prefill_cases(args)
    if not args.no_prefill:
        for name, make in cases:
            inp = make()
            T, N = inp.total_tokens, inp.slot.size
            tt = dict(
                mixed=b16(inp.mixed).to(dev), a=b16(inp.a).to(dev), b=b16(inp.b).to(dev),
                A_log=torch.from_numpy(inp.A_log).to(dev),
                dt_bias=torch.from_numpy(inp.dt_bias).to(dev),
                conv_w=None if inp.conv_w is None else b16(inp.conv_w).to(dev),
                conv_b=None if inp.conv_b is None else b16(inp.conv_b).to(dev),
                conv=None if inp.conv_state is None else b16(inp.conv_state).to(dev),
                ssm=torch.from_numpy(inp.ssm_state).to(dev),
                cu=torch.from_numpy(inp.cu_seqlens).to(dev), slot=torch.from_numpy(inp.slot).to(dev),
                hi=None if inp.has_init is None else torch.from_numpy(inp.has_init).to(dev),
                out=torch.empty(T, geo.Hv, geo.dv, dtype=torch.bfloat16, device=dev))
            ws = torch.empty(gdn.gdn_chunked_prefill_workspace_size(T, N, dims, 64),
                             dtype=torch.uint8, device=dev)

            def pcall(tt=tt, ws=ws):
                gdn.gdn_chunked_prefill(tt["mixed"], tt["a"], tt["b"], tt["A_log"], tt["dt_bias"],
                                        tt["conv_w"], tt["conv_b"], tt["conv"], tt["ssm"], tt["cu"],
                                        tt["slot"], tt["hi"], tt["out"], ws, dims, chunk=64,
                                        stream=stream)
            ms = central(timed(pcall, 5, 2))
            launches = prefill_launches(T, N, geo.Hv, 64, inp.conv_w is not None)
            fl = prefill_flops_per_token(geo) * T
            tpk, tkind = load_bf16_peak()
            prefill[name] = {"tokens": T, "seqs": N, "ms": round(ms, 3),
                             "tokens_per_s": round(T / ms * 1e3, 1),
                             "TFLOPs": round(fl / ms / 1e9, 2),
                             "frac_of_bf16_tensor_peak": round(fl / ms / 1e9 / tpk, 4),
                             "peak_kind": tkind, "gpu_launches_per_call": launches,
                             "GBps": round(prefill_bytes(T, N, geo, conv=inp.conv_w is not None) / ms / 1e6, 1)}
            if name.startswith("single"):  # the same call with the output gate (+1 launch)
                og = gdn.OutputGate(torch.randn(T, geo.Hv, geo.dv, device=dev).to(torch.bfloat16),
                                    torch.ones(geo.dv, device=dev))

                def pcall_g(tt=tt, ws=ws, og=og):
                    gdn.gdn_chunked_prefill(tt["mixed"], tt["a"], tt["b"], tt["A_log"],
                                            tt["dt_bias"], tt["conv_w"], tt["conv_b"], tt["conv"],
                                            tt["ssm"], tt["cu"], tt["slot"], tt["hi"], tt["out"],
                                            ws, dims, chunk=64, gate=og, stream=stream)
                msg = central(timed(pcall_g, 5, 2))
                prefill[name + "_gated"] = {"tokens": T, "ms": round(msg, 3),
                                            "tokens_per_s": round(T / msg * 1e3, 1),
                                            "gate_us": round((msg - ms) * 1e3, 1)}
                del og
            del tt, ws
        torch.cuda.empty_cache()

    # ---- mixed step: 64 decode rows + one 4096-token prefill (with conv) ----
    mixed = {}
    if not args.no_prefill:
        nd, Tp = 64, 4096
        inp = gi.make_inputs(geo, [1] * nd + [Tp], NUM_SLOTS, seed=12, state_pool=False)
        mt = dict(mixed=b16(inp.mixed).to(dev), a=b16(inp.a).to(dev), b=b16(inp.b).to(dev),
                  A_log=torch.from_numpy(inp.A_log).to(dev),
                  dt_bias=torch.from_numpy(inp.dt_bias).to(dev),
                  conv_w=b16(inp.conv_w).to(dev), conv_b=b16(inp.conv_b).to(dev),
                  conv=b16(inp.conv_state).to(dev),
                  ssm=gi.device_state_pool(NUM_SLOTS, geo, 0.05, 13, dev),
                  slot=torch.from_numpy(inp.slot).to(dev),
                  cu=torch.tensor([0, Tp], dtype=torch.int32, device=dev),
                  out=torch.empty(nd + Tp, geo.Hv, geo.dv, dtype=torch.bfloat16, device=dev))
        ws = torch.empty(gdn.gdn_chunked_prefill_workspace_size(Tp, 1, dims, 64),
                         dtype=torch.uint8, device=dev)

        def mixed_call():
            gdn.gdn_mixed_step(mt["mixed"], mt["a"], mt["b"], mt["A_log"], mt["dt_bias"],
                               mt["conv_w"], mt["conv_b"], mt["conv"], mt["ssm"], mt["slot"], nd,
                               mt["cu"], None, mt["out"], ws, dims, chunk=64, stream=stream)

        def separate_calls():
            gdn.gdn_decode_step(mt["mixed"][:nd], mt["a"][:nd], mt["b"][:nd], mt["A_log"],
                                mt["dt_bias"], mt["conv_w"], mt["conv_b"], mt["conv"], mt["ssm"],
                                mt["slot"][:nd], mt["out"][:nd], dims, stream=stream)
            gdn.gdn_chunked_prefill(mt["mixed"][nd:], mt["a"][nd:], mt["b"][nd:], mt["A_log"],
                                    mt["dt_bias"], mt["conv_w"], mt["conv_b"], mt["conv"],
                                    mt["ssm"], mt["cu"], mt["slot"][nd:], None, mt["out"][nd:],
                                    ws, dims, chunk=64, stream=stream)
        ms_m = central(timed(mixed_call, 7, 3))
        ms_s = central(timed(separate_calls, 7, 3))
        mixed["decode64_prefill4096"] = {"mixed_us": round(ms_m * 1e3, 1),
                                         "separate_us": round(ms_s * 1e3, 1),
                                         "speedup": round(ms_s / ms_m, 3)}
        del mt, ws
        torch.cuda.empty_cache()

    # ---- e2e through the public API with pinned host buffers ----
    # A step's inputs (x, a, b, slot table) are staged in one pinned host buffer and copied
    # with one H2D copy into one device buffer whose sections the call reads as tensors;
    # the output comes back with one D2H copy.
    t = decode_setup(args.batch, args.num_slots, seed=args.batch, state_bf16=args.state_bf16)
    parts = [("mixed", t["mixed"]), ("a", t["a"]), ("b", t["b"]), ("slot", t["slot"])]
    offs, total = [], 0
    for _, x in parts:
        offs.append(total)
        total += (x.numel() * x.element_size() + 255) // 256 * 256
    h_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    for (name, x), o in zip(parts, offs):
        nb_ = x.numel() * x.element_size()
        h_buf[o:o + nb_].copy_(x.cpu().contiguous().view(-1).view(torch.uint8))
        t[name] = d_buf[o:o + nb_].view(x.dtype).view(x.shape)  # the call reads these views
    h_out = torch.empty_like(t["out"], device="cpu").pin_memory()

    def e2e_call():
        d_buf.copy_(h_buf, non_blocking=True)
        decode_call(t)
        h_out.copy_(t["out"], non_blocking=True)

    e2e_serial_ms = float(np.mean(timed(e2e_call, max(5, args.steps // 2), 3)))
    h2d = total  # the bytes the one H2D copy moves (the sections plus their alignment padding)
    d2h = h_out.numel() * h_out.element_size()

    # Pipelined like a serving loop: step n's inputs are copied in (own stream) while step
    # n-1 computes, and step n's output is copied out (own stream) while step n+1 computes;
    # inputs and outputs are double-buffered. Every step's H2D and D2H copies lie inside the
    # one timed region (start to the last D2H); the state pool (> L2) is not flushed.
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    d_in = [d_buf, torch.empty_like(d_buf)]
    views = []
    for db in d_in:
        v = dict(t)
        for (name, x), o in zip(parts, offs):
            nb_ = x.numel() * x.element_size()
            v[name] = db[o:o + nb_].view(x.dtype).view(x.shape)
        v["out"] = torch.empty_like(t["out"])
        views.append(v)
    h_outs = [h_out, torch.empty_like(h_out).pin_memory()]
    ev = lambda: torch.cuda.Event()
    in_ready, k_done, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def pipelined(steps):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        h2d_s.wait_event(start)
        d2h_s.wait_event(start)
        for n in range(steps):
            j = n & 1
            with torch.cuda.stream(h2d_s):
                if n >= 2:
                    h2d_s.wait_event(k_done[j])   # step n-2 no longer reads this input buffer
                d_in[j].copy_(h_buf, non_blocking=True)
                in_ready[j].record(h2d_s)
            stream.wait_event(in_ready[j])
            if n >= 2:
                stream.wait_event(out_free[j])    # step n-2's output has been copied out
            decode_call(views[j])
            k_done[j].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(k_done[j])
                h_outs[j].copy_(views[j]["out"], non_blocking=True)
                out_free[j].record(d2h_s)
        stream.wait_stream(d2h_s)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) / steps

    pipelined(3)
    e2e_ms = pipelined(max(10, args.steps))
    e2e_bytes = decode_bytes(args.batch, geo, state_bytes=2 if args.state_bf16 else 4)
    # whole-job figures: the slowest rank's time, every rank's bytes (all ranks call these)
    e2e_ms, e2e_gbs = aggregate_ranks(e2e_ms, e2e_bytes, world, dev)
    e2e_serial_ms, e2e_serial_gbs = aggregate_ranks(e2e_serial_ms, e2e_bytes, world, dev)

    # ---- headline: exactly K timed decode steps ----
    nbytes = decode_bytes(args.batch, geo, state_bytes=2 if args.state_bf16 else 4)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    step_ms = timed(lambda: decode_call(t), args.steps, args.warmup)
    torch.cuda.synchronize()
    mean_ms, value = aggregate_ranks(float(np.mean(step_ms)), nbytes, world, dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clk = clocks.stop() if clocks else None

    if rank != 0:
        return None
    peak, peak_kind = load_peaks()
    achieved = nbytes / (mean_ms * 1e-3) / 1e9
    traffic = ncu_traffic("bf16" if args.state_bf16 else "f32", args.batch, args.num_slots)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "GDN decode step, Qwen3-Next geometry Hk=16 Hv=32 dk=dv=128 "
                               f"D=8192 W=4, B={args.batch} rows over {args.num_slots} shuffled "
                               f"slots, bf16 conv cache, {'bf16' if args.state_bf16 else 'fp32'} "
                               "state, bf16 I/O",
                   "batch": args.batch, "num_slots": args.num_slots,
                   "bytes_per_step": nbytes,
                   "l2": "flushed between timed steps: a 512 MiB write, then a 256 MiB read, so "
                         "each step starts with none of its data and no dirty lines in L2"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "frac_of_8TBps_nominal": round(achieved / 8000.0, 4),
                     "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
                     "traffic_note": None if traffic is None else traffic.get("note")},
        "e2e": {"value": round(e2e_gbs, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5),
                "mode": "pipelined: step n+1's H2D and step n-1's D2H overlap step n's kernel",
                "serial": {"value": round(e2e_serial_gbs, 1),
                           "ms_per_step": round(e2e_serial_ms, 5),
                           "mode": "H2D, kernel, D2H in sequence per step, L2 flushed between"}},
        "gpu_launches": args.steps,
        "clocks": clk,
        "decode_sweep": sweep,
        "prefill": prefill,
        "mixed_step": mixed,
        "context": {"pages_gb10_c16_GBps": 175.14,
                    "note": "GB10 (SM121) whole GDN transition incl. W4A4 projections; context only"},
    }
    # prefill figures as flat keys beside the headline (the nested dict keeps the detail)
    for name, key in ((f"single_{args.prefill_tokens}_bypass", "prefill"),
                      ("varlen_8seq_conv", "prefill_varlen")):
        e = prefill.get(name)
        if e:
            line[f"{key}_tokens_per_s"] = e["tokens_per_s"]
            line[f"{key}_ms"] = e["ms"]
            line[f"{key}_tflops"] = e["TFLOPs"]
            line[f"{key}_frac_of_bf16_tensor_peak"] = e["frac_of_bf16_tensor_peak"]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
        line["cpu_baseline_1thread"] = cpu_baseline(seconds=args.cpu_seconds / 2, nthreads=1)
        if not args.no_prefill:
            pb = {}
            for name, make in prefill_cases(args):
                pb[name] = cpu_prefill_baseline(make(), name)
            line["cpu_baseline_prefill"] = pb
            for name, key in ((f"single_{args.prefill_tokens}_bypass", "prefill"),
                              ("varlen_8seq_conv", "prefill_varlen")):
                if name in pb:
                    line[f"{key}_oracle_tokens_per_s"] = pb[name]["value"]
    return line


def prefill_cases(args):
    """The chunked-prefill workloads: one sequence (conv bypassed), then ~32k varlen tokens."""
    from gated_deltanet_linear_gdn_gb300 import inputs as gi

    cases = []
    if not args.no_single:
        cases.append((f"single_{args.prefill_tokens}_bypass",
                      lambda: gi.prefill_single(args.prefill_tokens, seed=0)))
    if not args.no_varlen:
        name = "varlen_8seq_conv" if args.varlen_max == 8192 else f"varlen_8seq_conv_max{args.varlen_max}"
        cases.append((name, lambda: gi.prefill_varlen(8, args.varlen_max, seed=0)))
    return cases


# --------------------------------------------------------------------------- oracle arm

def oracle_decode_sample(rows, seed=HEADLINE_B):
    """Host inputs of a `rows`-row sample of the headline decode workload (compact pool)."""
    from gated_deltanet_linear_gdn_gb300 import inputs as gi

    geo = gi.QWEN3_NEXT
    inp = gi.make_inputs(geo, [1] * rows, rows + 1, seed, slots=np.arange(1, rows + 1))
    return inp


def _oracle_call(inp, conv, ssm, nthreads):
    import oracle

    g = inp.geo
    return oracle.layer(inp.mixed, inp.a, inp.b, False, inp.A_log, inp.dt_bias, inp.conv_w,
                        inp.conv_b, True, conv, False, 0, ssm, inp.cu_seqlens, inp.slot, None,
                        g.Hk, g.Hv, g.dk, g.dv, g.W, inp.scale, True, None, nthreads)


def cpu_baseline(seconds=10.0, rows=32, nthreads=None):
    import oracle

    oracle.lib()
    nthreads = nthreads or os.cpu_count() or 1
    inp = oracle_decode_sample(rows)
    conv = inp.conv_state.copy()
    ssm = inp.ssm_state.astype(np.float64)
    runs = 0
    t0 = time.perf_counter()
    while True:
        _oracle_call(inp, conv, ssm, nthreads)
        runs += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    nb = decode_bytes(rows, inp.geo) * runs
    return {"value": round(nb / el / 1e9, 4), "unit": "GB/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{rows} rows of the B=256 decode workload (Qwen3-Next geometry), "
                      f"{runs} oracle calls in {el:.1f} s, fp64, {nthreads} threads"}


def cpu_prefill_baseline(inp, name, head_stride=None, nthreads=None):
    """The oracle on one prefill workload, the same inputs as the GPU call. The token-by-token
    recurrence costs ~6 dv dk fp64 operations per token and value head, so long workloads are
    sampled by value head (every head_stride-th head; the conv runs in full) and the time is
    scaled to all heads -- which also scales the conv's share, so the figure slightly
    understates the oracle."""
    import oracle

    oracle.lib()
    nthreads = nthreads or os.cpu_count() or 1
    g = inp.geo
    T = inp.total_tokens
    if head_stride is None:
        head_stride = 1 if T <= 4096 else 4
    mask = (np.arange(g.Hv) % head_stride) == 0
    conv = None if inp.conv_state is None else inp.conv_state.copy()
    ssm = inp.ssm_state.astype(np.float64)
    t0 = time.perf_counter()
    oracle.layer(inp.mixed, inp.a, inp.b, inp.gate_direct, inp.A_log, inp.dt_bias, inp.conv_w,
                 inp.conv_b, inp.silu, conv, inp.conv_f32, inp.conv_layout, ssm, inp.cu_seqlens,
                 inp.slot, inp.has_init, g.Hk, g.Hv, g.dk, g.dv, g.W, inp.scale, inp.qk_l2norm,
                 mask, nthreads)
    el = time.perf_counter() - t0
    frac = float(mask.sum()) / g.Hv
    return {"value": round(T * frac / el, 1), "unit": "tokens/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{name}: {T} tokens, {int(mask.sum())} of {g.Hv} value heads "
                      f"(time scaled to all heads), fp64 token-by-token oracle, {el:.1f} s, "
                      f"{nthreads} threads"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle

    oracle.lib()
    nthreads = os.cpu_count() or 1
    rows = 16
    inp = oracle_decode_sample(rows)
    conv = inp.conv_state.copy()
    ssm = inp.ssm_state.astype(np.float64)
    for _ in range(args.warmup):
        _oracle_call(inp, conv, ssm, nthreads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_call(inp, conv, ssm, nthreads)
        times.append(time.perf_counter() - t0)
    nb = decode_bytes(rows, inp.geo)
    mean_s = float(np.mean(times))
    value = nb / mean_s / 1e9
    sample = (f"{rows} rows of the B=256 decode workload per step (Qwen3-Next geometry), fp64 "
              f"oracle, {nthreads} host threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "GDN decode step, Qwen3-Next geometry Hk=16 Hv=32 dk=dv=128 "
                               "D=8192 W=4, B=256 rows over 512 shuffled slots, bf16 conv cache, "
                               "fp32 state, bf16 I/O", "batch": HEADLINE_B,
                   "num_slots": NUM_SLOTS, "sampled_rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": nthreads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--batch", type=int, default=HEADLINE_B, help="headline decode rows")
    ap.add_argument("--num-slots", type=int, default=NUM_SLOTS, help="headline slot pool size")
    ap.add_argument("--state-bf16", action="store_true",
                    help="headline decode on a bf16 recurrent-state pool (default fp32)")
    ap.add_argument("--prefill-tokens", type=int, default=4096,
                    help="length of the single-sequence prefill case")
    ap.add_argument("--no-varlen", action="store_true", help="skip the ~32k-token varlen case")
    ap.add_argument("--no-single", action="store_true", help="skip the single-sequence prefill case")
    ap.add_argument("--varlen-max", type=int, default=8192,
                    help="upper bound of the varlen case's 8 sequence lengths (8192: ~32k tokens)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
