"""Decode-step benchmark for the paged FP8-KV GQA path.

One step = the step's new tokens appended to the FP8 cache (1 per sequence
where the workload appends) + decode attention over every cached token, on
one batch of synthetic Llama-3-shaped inputs already resident in HBM: by
default one append_decode_fp8 call (append fused into the decode launch),
with --separate kv_append_fp8 followed by paged_gqa_decode.  Prints ONE JSON line
(rank 0):

  value      effective HBM GB/s of the decode step: algorithmic KV bytes
             (sum_b L_b * Hkv * 2 * 128) / device time per step
  e2e        the same metric through the public Python API with the step's
             inputs copied from pinned host memory and the output copied back
  roofline   the decode call (partial + combine kernels) against the measured
             HBM copy bandwidth
  cpu_baseline  the CPU oracle on a bounded sample of the same workload

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 4] [--page 16]
    python bench.py --impl reference ...      # the oracle as the reference arm
    python bench.py --workload prefill        # chunked prefill: a 128K prompt as 8 x 16K
                                              # chunks (append + causal attention each),
                                              # TFLOP/s against the tensor roofline

With N > 1 (torchrun) every rank runs an independent replica: the path has no
exchange step, so there is no collective beyond the timing barrier.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged FP8-KV GQA decode: µs/step and effective HBM GB/s (% of GB300 peak)"
L2_BYTES = 129 * 1024 * 1024


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _tensor_peak():
    """Dense f16/bf16 tensor peak for a kernel timed inside a long step: the
    measured sustained cuBLAS bf16 rate (f16 has the same nominal rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        if "bf16_tflops_sustained" in p:
            return float(p["bf16_tflops_sustained"]), "measured (cuBLAS bf16, sustained; f16 same nominal rate)"
    return 1700.0, "fallback (sustained bf16; f16 same nominal rate)"


def _code_only(text: str) -> str:
    """C/CUDA source without comments and blank lines (a comment edit does
    not change the kernel the counters were taken on)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def _kernel_sha() -> str:
    h = hashlib.sha256()
    for f in ("decode.cu", "device.cuh", "internal.h"):
        with open(os.path.join(ROOT, "paged_fp8_kv_03_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _traffic(workload_name: str):
    """dram bytes per decode launch from the committed ncu summary, if it was
    taken on this exact kernel source and workload (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        t = json.load(fh)
    ent = t.get(workload_name)
    if not ent or ent.get("kernel_sha") != _kernel_sha():
        return None
    return ent.get("dram_bytes_per_launch")


class _HostStage:
    """Tensors packed into one pinned host buffer (each at a 256-byte aligned
    offset).  upload() copies the buffer with one H2D copy into a persistent
    device buffer and returns device views with the original names, dtypes
    and shapes (made once), as a serving loop keeps its input staging."""

    def __init__(self, parts):
        self.layout = []
        host = []
        off = 0
        for name, t in parts.items():
            t = t.detach().cpu().contiguous()
            n = t.numel() * t.element_size()
            self.layout.append((name, off, t.dtype, tuple(t.shape), n))
            host.append(t)
            off = (off + n + 255) // 256 * 256
        self.nbytes = off
        self.buf = torch.empty(off, dtype=torch.uint8).pin_memory()
        for (name, o, dt, shape, n), t in zip(self.layout, host):
            self.buf[o:o + n].copy_(t.view(-1).view(torch.uint8))

        self.dbuf = None
        self.views = None

    def upload(self, dev):
        if self.dbuf is None:
            self.dbuf = torch.empty(self.nbytes, dtype=torch.uint8, device=dev)
            self.views = {name: self.dbuf[o:o + n].view(dt).view(shape) for name, o, dt, shape, n in self.layout}
        self.dbuf.copy_(self.buf, non_blocking=True)
        return self.views


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed loop runs."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.path = tempfile.mktemp(prefix="pkv_clocks_", suffix=".csv")
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    sm.append(float(parts[2]))
                    smax.append(float(parts[3]))
                except ValueError:
                    continue
                n += 1
                for name, val in zip(names, parts[6:10]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value any rank holds (the slowest rank's time decides)."""
    if world <= 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- GPU arm
def _fill_layer(pkv, wl, layer, dev):
    P, H, D = wl.page_size, wl.hkv, wl.head_dim
    ks, vs = wl.scales(layer, device=dev)
    kc = torch.zeros((wl.num_pages, H, P, D), dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    chunk = 1 << 15
    for b, L in enumerate(wl.prefill_lens):
        for t0 in range(0, L, chunk):
            t1 = min(L, t0 + chunk)
            pkv.kv_append_fp8(wl.kv_rows(layer, 0, b, t0, t1, device=dev), wl.kv_rows(layer, 1, b, t0, t1, device=dev),
                              wl.slots(b, t0, t1).to(dev), ks, vs, kc, vc)
    return {"kc": kc, "vc": vc, "ks": ks, "vs": vs}


def _step_inputs(wl, layer, dev):
    """The per-step inputs: new K/V rows of the appended tokens [B, A, Hkv, D],
    their slots (for the two-call path), q."""
    A = wl.append
    if A:
        k_new = torch.stack([wl.kv_rows(layer, 0, b, L, L + A, device=dev) for b, L in enumerate(wl.prefill_lens)])
        v_new = torch.stack([wl.kv_rows(layer, 1, b, L, L + A, device=dev) for b, L in enumerate(wl.prefill_lens)])
        slots = torch.cat([wl.slots(b, L, L + A) for b, L in enumerate(wl.prefill_lens)]).to(dev)
    else:
        k_new = v_new = slots = None
    return {"k_new": k_new, "v_new": v_new, "slots": slots, "q": wl.q(layer, 0, device=dev)}


def run_gpu(args, rank, world):
    import paged_fp8_kv_03_gb300 as pkv
    from paged_fp8_kv_03_gb300 import build as pbuild

    if rank == 0 or not os.path.exists(pbuild.LIB):
        pbuild.build()
    if world > 1:
        torch.distributed.barrier()
    pkv.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl = workloads.config(args.config, page_size=args.page, dynamic_pages=args.dynamic_pages)
    kv_bytes = wl.kv_bytes()
    # distinct layer caches rotated step by step so a step never finds the
    # previous step's KV in L2 (each cache alone is already larger than L2)
    n_layers = max(1, args.rotate or max(2, int(math.ceil(3 * L2_BYTES / kv_bytes))))
    free, _ = torch.cuda.mem_get_info(dev)
    n_layers = max(1, min(n_layers, int(0.8 * free // (kv_bytes + (1 << 20)))))
    layers = [_fill_layer(pkv, wl, l, dev) for l in range(n_layers)]
    steps_in = [_step_inputs(wl, l, dev) for l in range(n_layers)]
    bt = wl.block_table().to(dev)
    lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=dev)
    psz = torch.tensor(wl.page_sizes, dtype=torch.int32, device=dev) if wl.page_sizes is not None else None
    max_len = wl.max_len
    out = torch.empty((wl.batch, wl.hq, wl.head_dim), dtype=torch.bfloat16, device=dev)
    ws = pkv.decode_workspace(wl.batch, wl.hq, wl.hkv, wl.page_size, dev, max_seq_len=max_len)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # Split weights: measured once per device on layer 0 of this workload
    # (setup, untimed; the library's calibration call), or the even split.
    split = "even"
    if not args.no_calibrate:
        c0, s0 = layers[0], steps_in[0]
        weights = pkv.pkv_decode_calibrate_split(s0["q"], c0["kc"], c0["vc"], c0["ks"], c0["vs"], bt, lens, out, ws,
                                                 rounds=args.calibrate_rounds, max_seq_len=max_len,
                                                 seq_page_sizes=psz)
        split = (f"calibrated per-CTA weights ({args.calibrate_rounds} rounds, {len(weights)} CTAs, "
                 f"weights {min(weights)}..{max(weights)})")
    else:
        pkv.pkv_decode_set_split_weights(None)

    per_step = wl.layers      # layer passes per decode step (80 for the mixed serving batch)

    def step(i, evs=None):
        for l in range(per_step):
            g = i * per_step + l
            c = layers[g % n_layers]
            s = steps_in[g % n_layers]
            if s["k_new"] is not None and args.separate:
                pkv.pkv_kv_append_fp8(s["k_new"].flatten(0, 1), s["v_new"].flatten(0, 1), s["slots"], c["ks"], c["vs"],
                                      c["kc"], c["vc"], err)
            if evs is not None:
                evs[l][0].record(stream)
            if s["k_new"] is not None and not args.separate:
                pkv.pkv_append_decode_fp8(s["k_new"], s["v_new"], s["q"], c["kc"], c["vc"], c["ks"], c["vs"], bt, lens,
                                          out, ws, device_error=err, max_seq_len=max_len, seq_page_sizes=psz)
            else:
                pkv.pkv_paged_gqa_decode(s["q"], c["kc"], c["vc"], c["ks"], c["vs"], bt, lens, out, ws,
                                         device_error=err, max_seq_len=max_len, seq_page_sizes=psz)
            if evs is not None:
                evs[l][1].record(stream)

    # nvidia-smi starts sampling before the warm-up, so no pause separates the
    # warm-up from the timed steps
    clocks = ClockSampler(dev.index)
    if rank == 0:
        clocks.start()
    graphs = None
    if args.graph:
        step(0)                 # first calls (library set-up) happen outside the capture
        torch.cuda.synchronize()
        # One graph per distinct layer-cache phase; each replays a whole step.
        n_phase = n_layers // math.gcd(n_layers, per_step)
        graphs = []
        for ph in range(n_phase):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(ph)
            graphs.append(g)
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream(dev)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(per_step)]
           for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    for i in range(args.warmup):
        if graphs is None:
            step(i)
        else:
            graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    h0 = time.perf_counter()
    t_start.record(stream)
    for i in range(args.steps):
        if graphs is None:
            step(i, evs[i])
        else:
            evs[i][0][0].record(stream)
            graphs[i % len(graphs)].replay()
            evs[i][-1][1].record(stream)
    t_end.record(stream)
    host_s = time.perf_counter() - h0        # host time to enqueue the timed steps
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if rank == 0 else None
    # Host cost of one call alone: enqueue a few layer passes behind a GPU
    # spin long enough that the launch queue never fills, so the time is the
    # binding's and the library's host work, not back-pressure from the GPU.
    # Always 16 calls (cycling over the layers), so every workload averages
    # over the same count.
    n_host = 16
    torch.cuda._sleep(int(2e8))
    hh0 = time.perf_counter()
    for l in range(n_host):
        c = layers[l % n_layers]
        s = steps_in[l % n_layers]
        if s["k_new"] is not None and not args.separate:
            pkv.pkv_append_decode_fp8(s["k_new"], s["v_new"], s["q"], c["kc"], c["vc"], c["ks"], c["vs"], bt, lens,
                                      out, ws, device_error=err, max_seq_len=max_len, seq_page_sizes=psz)
        else:
            pkv.pkv_paged_gqa_decode(s["q"], c["kc"], c["vc"], c["ks"], c["vs"], bt, lens, out, ws,
                                     device_error=err, max_seq_len=max_len, seq_page_sizes=psz)
    host_call_us = 1e6 * (time.perf_counter() - hh0) / n_host
    torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    if graphs is None:
        decode_ms = [a.elapsed_time(b) for ev in evs for a, b in ev]
    else:   # per-call times are not separable inside a graph: whole step / layer passes
        decode_ms = [ev[0][0].elapsed_time(ev[-1][1]) / per_step for ev in evs]
    total_ms = max_over_ranks(total_ms, world, dev)
    assert int(err.item()) == 0, f"device error word {int(err.item())}"

    # ---- kv_append_fp8 alone: one layer pass's new tokens (B x append rows of
    # every kv head) quantised into their pages, as the two-call path issues
    # it; the same rows rewrite the same bytes, so repeating it changes nothing.
    append_us = None
    if steps_in[0]["k_new"] is not None:
        c0, s0 = layers[0], steps_in[0]
        kf, vf = s0["k_new"].flatten(0, 1), s0["v_new"].flatten(0, 1)
        for _ in range(20):
            pkv.pkv_kv_append_fp8(kf, vf, s0["slots"], c0["ks"], c0["vs"], c0["kc"], c0["vc"], err)
        # The launches are enqueued behind a GPU spin longer than the host
        # needs to enqueue them, so they run back to back: the events time
        # the GPU, not the host's pace (a lone small launch would be timed
        # with the binding's host work inside it).
        n_app = 200
        torch.cuda.synchronize()
        torch.cuda._sleep(int(2e7))
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_app):
            pkv.pkv_kv_append_fp8(kf, vf, s0["slots"], c0["ks"], c0["vs"], c0["kc"], c0["vc"], err)
        a1.record(stream)
        torch.cuda.synchronize()
        append_us = {"us_per_call": round(1e3 * a0.elapsed_time(a1) / n_app, 3),
                     "calls": n_app, "tokens": int(kf.shape[0]), "kv_heads": wl.hkv,
                     "note": "kv_append_fp8 alone on one layer pass's new rows, launches back to back (in the "
                             "timed step the append is fused into the decode launch unless --separate)"}

    # ---- end to end through the public API with host buffers
    e2e_steps = min(args.steps, args.e2e_steps)
    # The step's block table and lengths cross once per step; each layer
    # pass's own inputs (q and the new K/V rows) are staged back to back
    # (256-byte aligned) in one pinned buffer and cross with one copy, as a
    # serving loop would stage them.
    seq_stage = _HostStage({"bt": bt, "lens": lens, **({"psz": psz} if psz is not None else {})})
    host = []
    for l in range(n_layers):
        s = steps_in[l]
        parts = {"q": s["q"]}
        if s["k_new"] is not None:
            parts.update(k_new=s["k_new"], v_new=s["v_new"], slots=s["slots"])
        host.append(_HostStage(parts))
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = seq_stage.nbytes + per_step * host[0].nbytes
    d2h = per_step * out.numel() * out.element_size()
    # As a serving loop would, the copies run on their own streams: layer
    # pass g+1's inputs cross while pass g computes, pass g-1's output while
    # pass g computes; events guard every reuse of a staging or output buffer.
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    outs = [out, torch.empty_like(out)]
    read_done = [None] * n_layers      # compute finished with staging buffer g % n_layers
    seq_done = [None]                  # compute finished with the step's block table and lengths
    out_free = [None, None]            # output buffer's copy to the host finished

    def upload(g):
        with torch.cuda.stream(s_in):
            if read_done[g % n_layers] is not None:
                s_in.wait_event(read_done[g % n_layers])
            d = host[g % n_layers].upload(dev)
            ready = torch.cuda.Event()
            ready.record(s_in)
        return d, ready

    def e2e_step_serial(i):
        # One layer pass per step: its copies and its compute depend on one
        # another, so there is nothing to overlap; all on the compute stream.
        sq = seq_stage.upload(dev)
        for l in range(per_step):
            g = i * per_step + l
            c = layers[g % n_layers]
            d = dict(host[g % n_layers].upload(dev), **sq)
            if "k_new" in d and args.separate:
                pkv.pkv_kv_append_fp8(d["k_new"].flatten(0, 1), d["v_new"].flatten(0, 1), d["slots"], c["ks"],
                                      c["vs"], c["kc"], c["vc"], err)
            if "k_new" in d and not args.separate:
                pkv.pkv_append_decode_fp8(d["k_new"], d["v_new"], d["q"], c["kc"], c["vc"], c["ks"], c["vs"],
                                          d["bt"], d["lens"], out, ws, device_error=err, max_seq_len=max_len,
                                          seq_page_sizes=d.get("psz"))
            else:
                pkv.pkv_paged_gqa_decode(d["q"], c["kc"], c["vc"], c["ks"], c["vs"], d["bt"], d["lens"], out, ws,
                                         device_error=err, max_seq_len=max_len, seq_page_sizes=d.get("psz"))
            out_host.copy_(out, non_blocking=True)

    def e2e_step(i):
        if per_step == 1:
            return e2e_step_serial(i)
        with torch.cuda.stream(s_in):
            if seq_done[0] is not None:
                s_in.wait_event(seq_done[0])
            sq = seq_stage.upload(dev)
            sq_ready = torch.cuda.Event()
            sq_ready.record(s_in)
        stream.wait_event(sq_ready)
        nxt = upload(i * per_step)
        for l in range(per_step):
            g = i * per_step + l
            c = layers[g % n_layers]
            d, ready = nxt
            stream.wait_event(ready)
            d = dict(d, **sq)
            ob = outs[g % 2]
            if out_free[g % 2] is not None:
                stream.wait_event(out_free[g % 2])
            if "k_new" in d and args.separate:
                pkv.pkv_kv_append_fp8(d["k_new"].flatten(0, 1), d["v_new"].flatten(0, 1), d["slots"], c["ks"],
                                      c["vs"], c["kc"], c["vc"], err)
            if "k_new" in d and not args.separate:
                pkv.pkv_append_decode_fp8(d["k_new"], d["v_new"], d["q"], c["kc"], c["vc"], c["ks"], c["vs"],
                                          d["bt"], d["lens"], ob, ws, device_error=err, max_seq_len=max_len,
                                          seq_page_sizes=d.get("psz"))
            else:
                pkv.pkv_paged_gqa_decode(d["q"], c["kc"], c["vc"], c["ks"], c["vs"], d["bt"], d["lens"], ob, ws,
                                         device_error=err, max_seq_len=max_len, seq_page_sizes=d.get("psz"))
            done = torch.cuda.Event()
            done.record(stream)
            read_done[g % n_layers] = done
            if l + 1 < per_step:
                nxt = upload(g + 1)                    # crosses while pass g computes
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                out_host.copy_(ob, non_blocking=True)
                freed = torch.cuda.Event()
                freed.record(s_out)
            out_free[g % 2] = freed
        seq_done[0] = done

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)                                # no copy starts before the timed region
    for i in range(e2e_steps):
        e2e_step(i)
    if per_step > 1:
        stream.wait_event(out_free[(e2e_steps * per_step - 1) % 2])   # the last output is on the host
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    assert int(err.item()) == 0, f"device error word {int(err.item())} (end-to-end steps)"

    ms_per_step = total_ms / args.steps
    step_bytes = per_step * kv_bytes
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = _peaks()
    dec_ms = statistics.mean(decode_ms)
    achieved = kv_bytes / (dec_ms * 1e-3) / 1e9
    traffic = _traffic(wl.name)
    launches_per_step = per_step * ((1 if (wl.append and args.separate) else 0) + 2)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 6),
        "us_per_step": round(ms_per_step * 1e3, 3),
        "frac_of_peak": round(value / world / peak, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "kv_dtype": "e4m3",
        "data": "synthetic",
        "config": {**wl.describe(), "kv_bytes_per_step": step_bytes, "layer_passes_per_step": per_step,
                   "layer_caches_resident": n_layers,
                   "l2": "inputs larger than L2: each layer cache exceeds the 129 MB L2 and "
                         f"{n_layers} distinct caches rotate layer pass by layer pass",
                   "parallelism": f"replicas x{world}", "split": split},
        "path": ("kv_append_fp8 + paged_gqa_decode (two calls)" if (wl.append and args.separate) else
                 "append_decode_fp8 (append fused into the decode launch)" if wl.append else "paged_gqa_decode")
                + (", CUDA-graph replay" if args.graph else ""),
        "roofline": {"bound": "hbm", "kernel": "decode call: paged_gqa_decode_kernel + splitk_merge_kernel",
                     "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": kv_bytes,
                     "avg_launch_us": round(dec_ms * 1e3, 3),
                     "median_launch_us": round(statistics.median(decode_ms) * 1e3, 3)},
        "e2e": {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 6), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "host": {"us_per_call": round(host_call_us, 2),
                 "enqueue_us_per_call_in_timed_loop": round(
                     1e6 * host_s / (args.steps * (1 if graphs is not None else per_step)), 2),
                 "note": "us_per_call: binding + library host work of one call with the GPU busy elsewhere; "
                         "the timed loop's enqueue time also includes waiting on a full launch queue"},
        "clocks": clk,
    }
    if append_us is not None:
        line["kv_append_fp8"] = append_us
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds, gen_device=dev)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- chunked prefill
PREFILL_METRIC = ("chunked-prefill attention over the paged FP8 cache: causal TFLOP/s "
                  "(append + attention of every chunk of one 128K prompt layer)")


def _prefill_flops(first: int, n: int, hq: int, d: int = 128) -> float:
    """Algorithmic FLOPs of n causal queries at positions first .. first+n-1:
    QK^T and PV, 2 * 2 * d per (query head, visible key)."""
    keys = n * first + n * (n + 1) // 2
    return 4.0 * d * hq * keys


def _prefill_setup(wl, chunk, dev):
    """Everything one chunked-prefill step needs, resident on the device: the
    fp32 K/V rows and slots of every chunk, the bf16 queries, per-chunk
    lengths and row offsets, an empty layer cache."""
    B, L = wl.batch, wl.seq_lens[0]
    n_chunks = L // chunk
    ks, vs = wl.scales(0, device=dev)
    kc = torch.zeros((wl.num_pages, wl.hkv, wl.page_size, wl.head_dim), dtype=torch.uint8, device=dev)
    chunks = []
    for c in range(n_chunks):
        t0, t1 = c * chunk, (c + 1) * chunk
        k = torch.cat([wl.kv_rows(0, 0, b, t0, t1, device=dev) for b in range(B)])
        v = torch.cat([wl.kv_rows(0, 1, b, t0, t1, device=dev) for b in range(B)])
        sl = torch.cat([wl.slots(b, t0, t1) for b in range(B)]).to(dev)
        q = wl.q_rows(0, B * chunk, step=c, device=dev)
        chunks.append({"k": k, "v": v, "slots": sl, "q": q,
                       "lens": torch.full((B,), t1, dtype=torch.int32, device=dev),
                       "cu": torch.arange(0, (B + 1) * chunk, chunk, dtype=torch.int32, device=dev),
                       "flops": B * _prefill_flops(t0, chunk, wl.hq, wl.head_dim)})
    return {"kc": kc, "vc": torch.zeros_like(kc), "ks": ks, "vs": vs, "chunks": chunks,
            "bt": wl.block_table().to(dev)}


def run_prefill_gpu(args, rank, world):
    import paged_fp8_kv_03_gb300 as pkv
    from paged_fp8_kv_03_gb300 import build as pbuild

    if rank == 0 or not os.path.exists(pbuild.LIB):
        pbuild.build()
    if world > 1:
        torch.distributed.barrier()
    pkv.load()
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    wl, chunk = workloads.prefill_config(page_size=args.page, prompt=args.prompt, chunk=args.chunk)
    st = _prefill_setup(wl, chunk, dev)
    B = wl.batch
    out = torch.empty((B * chunk, wl.hq, wl.head_dim), dtype=torch.bfloat16, device=dev)
    max_kv = wl.seq_lens[0]
    ws = torch.empty(pkv.pkv_prefill_workspace_size(B, wl.hkv, max_kv), dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    n_chunks = len(st["chunks"])

    def step(evs=None):
        for c, ch in enumerate(st["chunks"]):
            pkv.pkv_kv_append_fp8(ch["k"], ch["v"], ch["slots"], st["ks"], st["vs"], st["kc"], st["vc"], err)
            if evs is not None:
                evs[c][0].record(stream)
            pkv.pkv_paged_prefill(ch["q"], ch["cu"], st["kc"], st["vc"], st["ks"], st["vs"], st["bt"], ch["lens"],
                                  out, chunk, max_kv, ws, device_error=err)
            if evs is not None:
                evs[c][1].record(stream)

    clocks = ClockSampler(dev.index)
    if rank == 0:
        clocks.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_chunks)]
           for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if rank == 0 else None
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    assert int(err.item()) == 0, f"device error word {int(err.item())}"
    launch_ms = [[a.elapsed_time(b) for a, b in ev] for ev in evs]
    per_chunk_ms = [statistics.mean(launch_ms[i][c] for i in range(args.steps)) for c in range(n_chunks)]
    step_flops = sum(ch["flops"] for ch in st["chunks"])

    # ---- end to end through the public API: each chunk's q and K/V rows come
    # from pinned host memory and its output goes back.  As a serving loop
    # would, the copies run on their own streams: chunk c+1's inputs cross
    # while chunk c computes, chunk c-1's output while chunk c computes.
    stage = [_HostStage({"k": ch["k"], "v": ch["v"], "q": ch["q"], "slots": ch["slots"], "lens": ch["lens"],
                         "cu": ch["cu"]}) for ch in st["chunks"]]
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(n_chunks)]
    outs = [out, torch.empty_like(out)]
    h2d = sum(sg.nbytes for sg in stage)
    d2h = n_chunks * out.numel() * out.element_size()
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)
    read_done = [None] * n_chunks      # compute finished with chunk c's staged inputs
    out_free = [None, None]            # output buffer's copy to the host finished

    def e2e_step():
        for c in range(n_chunks):
            with torch.cuda.stream(s_in):
                if read_done[c] is not None:
                    s_in.wait_event(read_done[c])
                d = stage[c].upload(dev)
                ready = torch.cuda.Event()
                ready.record(s_in)
            stream.wait_event(ready)
            ob = outs[c % 2]
            if out_free[c % 2] is not None:
                stream.wait_event(out_free[c % 2])
            pkv.pkv_kv_append_fp8(d["k"], d["v"], d["slots"], st["ks"], st["vs"], st["kc"], st["vc"], err)
            pkv.pkv_paged_prefill(d["q"], d["cu"], st["kc"], st["vc"], st["ks"], st["vs"], st["bt"], d["lens"],
                                  ob, chunk, max_kv, ws, device_error=err)
            done = torch.cuda.Event()
            done.record(stream)
            read_done[c] = done
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                out_host[c].copy_(ob, non_blocking=True)
                freed = torch.cuda.Event()
                freed.record(s_out)
            out_free[c % 2] = freed

    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    e2e_step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)                                # no copy starts before the timed region
    for _ in range(e2e_steps):
        e2e_step()
    stream.wait_event(out_free[(n_chunks - 1) % 2])    # the last output is on the host
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)
    assert int(err.item()) == 0, f"device error word {int(err.item())} (end-to-end steps)"

    ms_per_step = total_ms / args.steps
    peak, peak_kind = _tensor_peak()
    prefill_ms = sum(per_chunk_ms)
    achieved = step_flops / (prefill_ms * 1e-3) / 1e12
    line = {
        "metric": PREFILL_METRIC,
        "value": round(world * step_flops / (ms_per_step * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 (QK^T) and f16 (PV) tensor-core operands, f32 accumulate",
        "kv_dtype": "e4m3",
        "data": "synthetic",
        "config": {**wl.describe(), "chunk": chunk, "chunks": n_chunks,
                   "flops_per_step": step_flops,
                   "l2": f"inputs larger than L2 ({wl.kv_bytes() / 1e6:.0f} MB of FP8 KV and "
                         f"{wl.seq_lens[0] * wl.batch * wl.hq * 256 / 1e6:.0f} MB of queries per step)",
                   "parallelism": f"replicas x{world}"},
        "path": "per chunk: kv_append_fp8 of its K/V, then paged_prefill (widen the visible FP8 K/V once, K to "
                "bf16 and V to f16, then the tcgen05 attention)",
        "per_chunk_ms": [round(x, 3) for x in per_chunk_ms],
        "roofline": {"bound": "tensor", "kernel": "paged_prefill_kernel",
                     "achieved": round(achieved, 2), "peak": peak, "peak_kind": peak_kind, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "algorithmic_flops_per_launch": step_flops / n_chunks,
                     "avg_launch_us": round(1e3 * prefill_ms / n_chunks, 1)},
        "e2e": {"value": round(world * step_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 3 * n_chunks * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(wl, chunk, args.cpu_seconds, scale_device=dev)
    if rank == 0:
        print(json.dumps(line), flush=True)


class OraclePrefillRig:
    """The CPU oracle on the chunked-prefill workload: pools of the whole
    prompt prepared once (untimed); sample() times the oracle on single query
    rows of the last chunk (all query heads of one kv head each)."""

    def __init__(self, wl, chunk, gen_device="cpu"):
        import oracle
        self.oracle, self.wl, self.chunk = oracle, wl, chunk
        L = wl.seq_lens[0]
        ks, vs = wl.scales(0, device=gen_device)
        self.ks, self.vs = ks.cpu().numpy(), vs.cpu().numpy()
        shape = (wl.num_pages, wl.hkv, wl.page_size, wl.head_dim)
        self.kc = np.zeros(shape, np.uint8)
        self.vc = np.zeros(shape, np.uint8)
        sl = wl.slots(0, 0, L).numpy()
        step = 1 << 15
        for t0 in range(0, L, step):
            t1 = min(L, t0 + step)
            oracle.kv_append(wl.kv_rows(0, 0, 0, t0, t1, device=gen_device).cpu().numpy(), sl[t0:t1], self.ks, self.kc)
            oracle.kv_append(wl.kv_rows(0, 1, 0, t0, t1, device=gen_device).cpu().numpy(), sl[t0:t1], self.vs, self.vc)
        last = L // chunk - 1
        self.q = wl.q_rows(0, chunk, step=last).view(torch.uint16).numpy()     # the last chunk's queries
        self.first = L - chunk
        self.bt = wl.block_table().numpy()[:1]

    def sample(self, row, h, threads):
        """Oracle time for query row `row` of the last chunk, the G heads of kv
        head h.  Returns (seconds, algorithmic FLOPs)."""
        wl = self.wl
        G = wl.group
        pos = self.first + row
        sel = np.array([[0, h * G + g] for g in range(G)], np.int32)
        t0 = time.perf_counter()
        self.oracle.paged_decode(self.q[row:row + 1], self.kc, self.vc, self.ks, self.vs, self.bt,
                                 np.array([pos + 1], np.int32), sel=sel, threads=threads)
        return time.perf_counter() - t0, 4.0 * wl.head_dim * G * (pos + 1)


def prefill_cpu_baseline(wl, chunk, budget_s, scale_device="cpu") -> dict:
    threads = len(os.sched_getaffinity(0))
    rig = OraclePrefillRig(wl, chunk, scale_device)
    rng = np.random.default_rng(0)
    secs, flops, n = 0.0, 0.0, 0
    while secs < budget_s and n < 4096:
        dt, f = rig.sample(int(rng.integers(chunk)), n % wl.hkv, threads)
        secs += dt
        flops += f
        n += 1
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} (query row, kv head) pairs of the last {chunk}-token chunk (positions from "
                      f"{rig.first}), the "
                      f"{wl.group} query heads of the kv head each, fp64 C oracle, {secs:.1f} s timed"}


def run_prefill_reference(args, rank, world):
    if rank != 0:
        return
    wl, chunk = workloads.prefill_config(page_size=args.page, prompt=args.prompt, chunk=args.chunk)
    threads = len(os.sched_getaffinity(0))
    rig = OraclePrefillRig(wl, chunk)
    dt1, _ = rig.sample(chunk - 1, 0, threads)
    per_step = max(1, int(args.ref_seconds / (args.warmup + args.steps) / max(dt1, 1e-9)))
    rng = np.random.default_rng(1)
    per, fl = [], []
    for i in range(args.warmup + args.steps):
        s, f = 0.0, 0.0
        for k in range(per_step):
            dt, ff = rig.sample(int(rng.integers(chunk)), k % wl.hkv, threads)
            s += dt
            f += ff
        if i >= args.warmup:
            per.append(s)
            fl.append(f)
    value = sum(fl) / sum(per) / 1e12
    line = {"impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * statistics.mean(per), 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**wl.describe(), "chunk": chunk},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: {per_step} (query row, kv head) pairs of the last chunk, the "
                                       f"{wl.group} query heads of the kv head each, fp64 C oracle"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- CPU oracle
def sample_sequences(wl, max_tokens: int = 131072) -> list:
    """The sequences the CPU oracle samples: the first ones in index order
    while their lengths add up to at most max_tokens (at least one), so that
    preparing their pages stays bounded on the mixed 512..128K batch."""
    seqs, tot = [], 0
    for b, L in enumerate(wl.seq_lens):
        if seqs and tot + L > max_tokens:
            break
        seqs.append(b)
        tot += L
    return seqs


class OracleRig:
    """The CPU oracle on this workload.  Pools, scales and prefill pages are
    prepared once from generated inputs (untimed; generation on gen_device,
    whose values are bit-identical to the host's); step() times the oracle's
    append of the step's tokens and its decode of whole sequences."""

    def __init__(self, wl, gen_device="cpu"):
        import oracle
        self.oracle = oracle
        self.wl = wl
        self.gen = gen_device
        ks, vs = wl.scales(0, device=gen_device)
        self.ks, self.vs = ks.cpu().numpy(), vs.cpu().numpy()
        shape = (wl.num_pages, wl.hkv, wl.page_size, wl.head_dim)
        self.kc = np.zeros(shape, np.uint8)
        self.vc = np.zeros(shape, np.uint8)
        self.q = wl.q().view(torch.uint16).numpy()
        self.bt = wl.block_table().numpy()
        self.lens = np.array(wl.seq_lens, np.int32)
        self.psz = np.array(wl.page_sizes, np.int32) if wl.page_sizes is not None else None
        self.filled = set()

    def _rows(self, which, b, t0, t1):
        return self.wl.kv_rows(0, which, b, t0, t1, device=self.gen).cpu().numpy()

    def fill(self, b):
        if b in self.filled:
            return
        wl, L = self.wl, self.wl.prefill_lens[b]
        sl = wl.slots(b, 0, L).numpy()
        step = 1 << 15
        for t0 in range(0, L, step):
            t1 = min(L, t0 + step)
            self.oracle.kv_append(self._rows(0, b, t0, t1), sl[t0:t1], self.ks, self.kc)
            self.oracle.kv_append(self._rows(1, b, t0, t1), sl[t0:t1], self.vs, self.vc)
        self.filled.add(b)

    def step(self, seqs, threads, n_kv_heads=None):
        """Times the oracle on sequences `seqs`: append of their step tokens and
        decode of the query heads of their first n_kv_heads kv heads (all by
        default).  Returns (seconds, algorithmic KV bytes covered)."""
        wl = self.wl
        hk = wl.hkv if n_kv_heads is None else max(1, min(wl.hkv, n_kv_heads))
        for b in seqs:
            self.fill(b)
        new = [(self._rows(0, b, wl.prefill_lens[b], wl.seq_lens[b]), self._rows(1, b, wl.prefill_lens[b], wl.seq_lens[b]),
                wl.slots(b, wl.prefill_lens[b], wl.seq_lens[b]).numpy()) for b in seqs]
        sel = np.array([[b, i] for b in seqs for i in range(hk * wl.group)], np.int32)
        t0 = time.perf_counter()
        for kn, vn, sl in new:
            if len(sl):
                self.oracle.kv_append(kn, sl, self.ks, self.kc)
                self.oracle.kv_append(vn, sl, self.vs, self.vc)
        self.oracle.paged_decode(self.q, self.kc, self.vc, self.ks, self.vs, self.bt, self.lens, sel=sel,
                                 threads=threads, seq_page_sizes=self.psz)
        dt = time.perf_counter() - t0
        return dt, sum(wl.seq_lens[b] for b in seqs) * hk * 2 * wl.head_dim


def cpu_baseline(wl, budget_s: float, gen_device="cpu") -> dict:
    threads = len(os.sched_getaffinity(0))
    rig = OracleRig(wl, gen_device)
    seqs = sample_sequences(wl)
    done, secs, nbytes, i = 0, 0.0, 0, 0
    while secs < budget_s and i < 256 * len(seqs):      # the time budget decides; the count only bounds it
        b = seqs[i % len(seqs)]
        dt, nb = rig.step([b], threads)
        done += 1
        secs += dt
        nbytes += nb
        i += 1
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} sequence decode steps over sequences {seqs[0]}..{seqs[-1]} "
                      f"({sum(wl.seq_lens[b] for b in seqs)} tokens) of {wl.batch}, all {wl.hq} query heads "
                      f"each, one layer, fp64 C oracle append+decode, {secs:.1f} s timed"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    wl = workloads.config(args.config, page_size=args.page, dynamic_pages=args.dynamic_pages)
    threads = len(os.sched_getaffinity(0))
    rig = OracleRig(wl)
    seqs = sample_sequences(wl)
    # Size each step's sample (kv heads of one sequence) so that all warm-up
    # and timed steps together take about args.ref_seconds of oracle time.
    t_full, _ = rig.step([seqs[-1]], threads)
    budget = args.ref_seconds / (args.warmup + args.steps)
    n_kv = max(1, min(wl.hkv, int(wl.hkv * budget / max(t_full, 1e-9))))
    per, nbytes = [], []
    for i in range(args.warmup + args.steps):
        b = seqs[i % len(seqs)]
        dt, nb = rig.step([b], threads, n_kv)
        if i >= args.warmup:
            per.append(dt)
            nbytes.append(nb)
    ms = 1e3 * statistics.mean(per)
    value = sum(nbytes) / sum(per) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**wl.describe(), "kv_bytes_per_step": wl.kv_bytes()},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: the {n_kv * wl.group} query heads of {n_kv} of the {wl.hkv} "
                                       f"kv heads of one sequence (sequences {seqs[0]}..{seqs[-1]} in turn, one "
                                       "layer), fp64 C oracle append + decode; value = algorithmic KV bytes "
                                       "covered / oracle time"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--workload", choices=["decode", "prefill"], default="decode",
                    help="decode: the decode-step line (default); prefill: chunked prefill of a 128K prompt")
    ap.add_argument("--prompt", type=int, default=131072, help="prefill: prompt tokens")
    ap.add_argument("--chunk", type=int, default=16384, help="prefill: tokens per chunk")
    ap.add_argument("--steps", type=int, default=None, help="timed steps (decode 3000, prefill 10)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (decode 50, prefill 3)")
    ap.add_argument("--config", type=int, default=4,
                    help="decode workload (default 4: the mixed 64-sequence 512..128K batch, 80 layers)")
    ap.add_argument("--page", type=int, default=None)
    ap.add_argument("--dynamic-pages", action="store_true",
                    help="mixed batch: 16-token pages, 64-token pages for sequences above 8192 tokens")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--rotate", type=int, default=0, help="distinct layer caches (0 = auto)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="oracle time budget of the whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-calibrate", action="store_true",
                    help="decode: keep the even split (no per-CTA split weights)")
    ap.add_argument("--calibrate-rounds", type=int, default=6)
    ap.add_argument("--graph", action="store_true", help="replay each step from a captured CUDA graph")
    ap.add_argument("--separate", action="store_true",
                    help="time kv_append_fp8 and paged_gqa_decode as two calls instead of the fused step")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = (3000 if args.config in (0, 1, 2) else 300 if args.config == 3 else 50) \
            if args.workload == "decode" else 10
    if args.warmup is None:
        args.warmup = (50 if args.config in (0, 1, 2, 3) else 5) if args.workload == "decode" else 3
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group(backend)
    try:
        if args.workload == "prefill":
            (run_prefill_reference if args.impl == "reference" else run_prefill_gpu)(args, rank, world)
        elif args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gpu(args, rank, world)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
