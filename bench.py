"""Benchmark of the KDA hot path on GB300.

One step = one pass of every hot-path call over synthetic inputs already resident in HBM:
  * kda_chunk_prefill  on the 16k-token prefill (H=32, T=16384, d=128, bf16 q/k/v);
  * the segment path on the same inputs split into 8 segments of 2048 tokens:
    kda_chunk_prepare (per-chunk records, once) -> kda_segment_package_prepared ->
    kda_package_scan -> kda_segment_replay_prepared;
  * kda_chunk_prefill and the same segment path on the long varlen workload (4 sequences of
    131072, 65536, 32768 and 8192 tokens with entry states; 44 leveled segments);
  * kda_decode_step    on 256 rows x 32 heads over a 4096-slot fp32 pool (8.6 GB).
After the timed steps, decode is also timed over 1000 back-to-back steps (the decode
workload's own definition), and the slot-table extensions each on their own.
`value` is the headline metric: prefill tokens per second of kda_chunk_prefill on the 16k
workload, from CUDA events around that call in each timed step; the other calls are reported
under "components" (tokens/s, achieved GB/s against the measured HBM peak). Every input is
larger than L2 (129 MB), so no flush is needed between timed iterations.

`--impl reference` times the CPU oracle (double precision, all host cores) on a bounded
sample of the same workload: the reference arm of this repository.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (H=32, d=128, T=16k) and decode state GB/s vs roofline"
UNIT = "tokens/s"

# Algorithmic bytes per unit (the minimum HBM traffic of each call: every input read once,
# every output written once). Token-head units for the prefill, (row, head) for decode.
D = 128
PREFILL_BYTES_PER_TOKEN_HEAD = 3 * D * 2 + D * 4 + 4 + D * 2   # q,k,v bf16 + g + beta + o
STATE_BYTES = D * D * 4                                       # one fp32 state
DECODE_BYTES_PER_ROW_HEAD = 2 * STATE_BYTES + 3 * D * 2 + D * 4 + 4 + D * 2


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one prefill_16k launch, from the
# ncu capture summarised in profiles/, and the SHA-256 prefix of the chunk kernels' source it
# was taken on: once that source changes the figure no longer describes the kernel that runs,
# and the roofline object reports traffic as null until a new capture replaces both.
TRAFFIC_PREFILL_16K = 929.2e6  # mean of 6 launches in two captures: 710.3 MB read + 218.9 written
TRAFFIC_SOURCE_SHA = "bbf7cd0786738437"
CHUNK_SOURCE = os.path.join(ROOT, "linear_attention_state_kda_gb300", "csrc", "kda_chunk_tc.cu")


def _traffic_prefill():
    import hashlib
    with open(CHUNK_SOURCE, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return (TRAFFIC_PREFILL_16K if sha == TRAFFIC_SOURCE_SHA else None), sha


WORKLOAD = ("prefill_16k: H=32, T=16384, dk=dv=128, chunk 64, bf16 q/k/v, fp32 g/beta/state "
            "(the headline); the step also runs segments_8x2048, varlen_long (4 sequences, "
            "237,568 tokens, single pass and 44 leveled segments) and decode_256 (256 rows x "
            "H32 over a 4096-slot pool)")
CONFIG = {"workload": WORKLOAD,
          "value_is": "tokens/s of kda_chunk_prefill on prefill_16k per GPU x n_gpus",
          "l2": "inputs larger than L2; no flush"}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, source="fallback")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(vals):
    """Element-wise maximum of a list of floats over all ranks (identity on one rank). The
    job's time is its slowest rank's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64)
    if dist.get_backend() == "nccl":
        t = t.cuda()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu().tolist()]


def weak_scaling_value(units_per_rank, world, ms):
    """Whole-job throughput when every rank processes `units_per_rank` units (replicas):
    all ranks' units over the slowest rank's time."""
    return world * units_per_rank / (ms * 1e-3)


def run_gb300(args):
    import torch
    import torch.distributed as dist
    from linear_attention_state_kda_gb300 import inputs, kda

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kda.lib()
    peaks = _peaks()

    x = inputs.make_workload("prefill_16k", device=dev)
    T, H = x.T, x.H
    segs = inputs.workload_segments("segments_8x2048")
    offs, seq_seg = inputs.segment_offsets(x.lens, segs)
    offs, seq_seg = offs.to(dev), seq_seg.to(dev)
    dec = inputs.make_workload("decode_256", device=dev)
    B = dec.q.shape[0]

    o = torch.empty_like(x.v)
    fin = torch.empty(1, H, D, D, device=dev)
    P = offs.numel() - 1
    M = torch.empty(P, H, D, D, device=dev)
    Dp = torch.empty(P, H, D, D, device=dev)
    seg_init = torch.empty(P, H, D, D, device=dev)
    fin2 = torch.empty(1, H, D, D, device=dev)
    o2 = torch.empty_like(x.v)
    ws = torch.empty(kda.package_scan_workspace(1, P, H, D, D), dtype=torch.uint8, device=dev)
    # chunk-path workspaces (per-chunk records), allocated once outside the timed region
    ws_pf = torch.empty(kda.chunk_workspace(torch.bfloat16, 1, T, H, D, D), dtype=torch.uint8,
                        device=dev)
    ws_seg = torch.empty(kda.chunk_workspace(torch.bfloat16, P, T, H, D, D), dtype=torch.uint8,
                         device=dev)
    od = torch.empty_like(dec.v)
    # the long varlen workload: 4 packed sequences with entry states, single pass and the
    # leveled segment path (one workspace serves both, used one after the other)
    xv = inputs.make_workload("varlen_long", device=dev)
    Tv = xv.T
    segs_v = inputs.workload_segments("varlen_long")
    offs_v, sso_v = inputs.segment_offsets(xv.lens, segs_v)
    offs_v, sso_v = offs_v.to(dev), sso_v.to(dev)
    Nv, Pv = len(xv.lens), offs_v.numel() - 1
    max_segs_v = max(len(sg) for sg in segs_v)
    ov = torch.empty_like(xv.v)
    finv = torch.empty(Nv, H, D, D, device=dev)
    Mv = torch.empty(Pv, H, D, D, device=dev)
    Dv = torch.empty(Pv, H, D, D, device=dev)
    siv = torch.empty(Pv, H, D, D, device=dev)
    finv2 = torch.empty(Nv, H, D, D, device=dev)
    ov2 = torch.empty_like(xv.v)
    ws_v = torch.empty(max(kda.chunk_workspace(torch.bfloat16, Nv, Tv, H, D, D),
                           kda.chunk_workspace(torch.bfloat16, Pv, Tv, H, D, D)),
                       dtype=torch.uint8, device=dev)
    ws_vs = torch.empty(kda.package_scan_workspace(Nv, max_segs_v, H, D, D), dtype=torch.uint8,
                        device=dev)
    stream = torch.cuda.current_stream()

    def prefill():
        kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta, o=o, final_state=fin, workspace=ws_pf)

    def package():  # the records serve both walks of the segment path
        kda.chunk_prepare(x.q, x.k, x.v, x.g, x.beta, offs, workspace=ws_seg)
        kda.segment_package_prepared(ws_seg, offs, T, H, D, D, M=M, D=Dp)

    def scan():
        kda.package_scan(M, Dp, seq_seg, P, seg_init=seg_init, final_state=fin2, workspace=ws)

    def replay():
        kda.segment_replay_prepared(ws_seg, offs, seg_init, T, H, D, D, o=o2)

    def decode():
        kda.decode_step(dec.q, dec.k, dec.v, dec.g, dec.beta, dec.slot_ids, dec.pool, o=od)

    def varlen():
        kda.chunk_prefill(xv.q, xv.k, xv.v, xv.g, xv.beta, cu_seqlens=xv.cu_seqlens,
                          init_state=xv.init_state, o=ov, final_state=finv, workspace=ws_v)

    def varlen_package():
        kda.chunk_prepare(xv.q, xv.k, xv.v, xv.g, xv.beta, offs_v, workspace=ws_v)
        kda.segment_package_prepared(ws_v, offs_v, Tv, H, D, D, M=Mv, D=Dv)

    def varlen_scan():
        kda.package_scan(Mv, Dv, sso_v, max_segs_v, init_state=xv.init_state, seg_init=siv,
                         final_state=finv2, workspace=ws_vs)

    def varlen_replay():
        kda.segment_replay_prepared(ws_v, offs_v, siv, Tv, H, D, D, o=ov2)

    # the segment paths are package -> scan -> replay; each call is timed on its own too
    parts = [("prefill_16k", prefill), ("seg_package", package), ("seg_scan", scan),
             ("seg_replay", replay), ("varlen_long", varlen), ("vseg_package", varlen_package),
             ("vseg_scan", varlen_scan), ("vseg_replay", varlen_replay), ("decode_256", decode)]
    for _ in range(args.warmup):
        for _, fn in parts:
            fn()
    torch.cuda.synchronize()

    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)] for n, _ in parts}
    step_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    launches0 = kda.launch_count()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # hold the stream on the device while the host enqueues the timed steps, so that the
        # events time device execution only (not the host's launch latency)
        torch.cuda._sleep(int(4e7))
        step_ev[0].record(stream)
        for i in range(args.steps):
            for n, fn in parts:
                ev[n][i][0].record(stream)
                fn()
                ev[n][i][1].record(stream)
        step_ev[1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = kda.launch_count() - launches0
    total_ms = step_ev[0].elapsed_time(step_ev[1])
    comp_ms = {n: sum(a.elapsed_time(b) for a, b in ev[n]) / args.steps for n, _ in parts}
    red = max_over_ranks([total_ms] + [comp_ms[n] for n, _ in parts])
    total_ms = red[0]
    for i, (n, _) in enumerate(parts):
        comp_ms[n] = red[1 + i]
    comp_ms["segments_8x2048"] = (comp_ms["seg_package"] + comp_ms["seg_scan"] +
                                  comp_ms["seg_replay"])
    comp_ms["varlen_long_segments"] = (comp_ms["vseg_package"] + comp_ms["vseg_scan"] +
                                       comp_ms["vseg_replay"])

    # decode as the workload states it: 1000 back-to-back steps over the same batch (the
    # states keep evolving), one event pair around all of them
    n_dec = 1000
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches_dec0 = kda.launch_count()
    torch.cuda._sleep(int(4e7))
    d0.record(stream)
    for _ in range(n_dec):
        decode()
    d1.record(stream)
    torch.cuda.synchronize()
    launches_dec = kda.launch_count() - launches_dec0
    dec1000_ms = max_over_ranks([d0.elapsed_time(d1) / n_dec])[0]

    hbm = peaks["hbm_gbs"]
    pf_bytes = T * H * PREFILL_BYTES_PER_TOKEN_HEAD + H * STATE_BYTES
    seg_bytes = (T * H * (2 * D * 2 + D * 4 + 4)            # package pass: k, v, g, beta
                 + P * H * 2 * STATE_BYTES                   # packages written
                 + P * H * 2 * STATE_BYTES + P * H * STATE_BYTES + H * STATE_BYTES  # scan
                 + T * H * PREFILL_BYTES_PER_TOKEN_HEAD + P * H * STATE_BYTES)     # replay
    dec_bytes = B * H * DECODE_BYTES_PER_ROW_HEAD + B * 4
    # varlen_long: every token's inputs read and output written once, plus the entry states
    # read and the exit states written; its segment path adds the package pass (k, v, g, beta
    # read, packages written), the scan (packages and entry states read, segment entry states
    # and exit states written) and the replay's segment entry states
    v_pf_bytes = Tv * H * PREFILL_BYTES_PER_TOKEN_HEAD + 2 * Nv * H * STATE_BYTES
    v_seg_bytes = (Tv * H * (2 * D * 2 + D * 4 + 4) + Pv * H * 2 * STATE_BYTES
                   + Pv * H * 2 * STATE_BYTES + Nv * H * STATE_BYTES + Pv * H * STATE_BYTES
                   + Nv * H * STATE_BYTES
                   + Tv * H * PREFILL_BYTES_PER_TOKEN_HEAD + Pv * H * STATE_BYTES)
    comps = {
        "prefill_16k": dict(ms=comp_ms["prefill_16k"],
                            tokens_per_s=T / (comp_ms["prefill_16k"] * 1e-3),
                            algorithmic_bytes=pf_bytes,
                            gbs=pf_bytes / (comp_ms["prefill_16k"] * 1e-3) / 1e9),
        "segments_8x2048": dict(ms=comp_ms["segments_8x2048"],
                                tokens_per_s=T / (comp_ms["segments_8x2048"] * 1e-3),
                                algorithmic_bytes=seg_bytes,
                                gbs=seg_bytes / (comp_ms["segments_8x2048"] * 1e-3) / 1e9,
                                package_ms=comp_ms["seg_package"], scan_ms=comp_ms["seg_scan"],
                                replay_ms=comp_ms["seg_replay"]),
        "varlen_long": dict(ms=comp_ms["varlen_long"],
                            tokens_per_s=Tv / (comp_ms["varlen_long"] * 1e-3),
                            algorithmic_bytes=v_pf_bytes,
                            gbs=v_pf_bytes / (comp_ms["varlen_long"] * 1e-3) / 1e9),
        "varlen_long_segments": dict(
            ms=comp_ms["varlen_long_segments"],
            tokens_per_s=Tv / (comp_ms["varlen_long_segments"] * 1e-3),
            algorithmic_bytes=v_seg_bytes,
            gbs=v_seg_bytes / (comp_ms["varlen_long_segments"] * 1e-3) / 1e9,
            package_ms=comp_ms["vseg_package"], scan_ms=comp_ms["vseg_scan"],
            replay_ms=comp_ms["vseg_replay"], segments=Pv),
        "decode_256": dict(ms=comp_ms["decode_256"], algorithmic_bytes=dec_bytes,
                           gbs=dec_bytes / (comp_ms["decode_256"] * 1e-3) / 1e9),
        "decode_256_x1000": dict(ms=dec1000_ms, steps=n_dec, launches=int(launches_dec),
                                 algorithmic_bytes=dec_bytes,
                                 gbs=dec_bytes / (dec1000_ms * 1e-3) / 1e9),
    }
    for c in comps.values():
        c["hbm_frac"] = c["gbs"] / hbm
    # dominant kernel: the longest single launch of the step, the prefill call (one fused
    # cooperative launch on this workload): algorithmic bytes of the call over its duration
    traffic, chunk_sha = _traffic_prefill()
    roofline = {"bound": "hbm", "achieved": round(comps["prefill_16k"]["gbs"], 1), "peak": hbm,
                "unit": "GB/s", "frac": round(comps["prefill_16k"]["gbs"] / hbm, 4),
                "traffic": traffic, "kernel": "prefill_16k (chunk_fused_kernel)",
                "kernel_source_sha": chunk_sha, "peak_source": peaks["source"]}

    # The extensions, timed on their own after the step (each over its own CUDA events, the
    # same number of iterations): a 4-token verify window per row with forked read slots and
    # logit write strengths, a checkpoint image of the decode rows' 256 slots (and its
    # restore), zeroing 256 slots, and the short conv over the 16k prefill's q, k, v channels.
    win = inputs.make_workload("window_256x4", device=dev)
    Bw, Ww = win.write_slots.shape
    ow = torch.empty_like(win.v)
    image = torch.empty(B, H, D, D, device=dev)
    named = torch.zeros(win.pool.shape[0], dtype=torch.bool, device=dev)
    named[win.read_slots.long()] = True
    named[win.write_slots.long().reshape(-1)] = True
    free_slots = torch.nonzero(~named).reshape(-1)[:B].to(torch.int32).contiguous()

    def window():
        kda.decode_window(win.q, win.k, win.v, win.g, win.beta_logit, win.read_slots,
                          win.write_slots, win.pool, beta_is_logit=True, o=ow)

    def checkpoint():
        kda.slot_copy(dec.pool, dec.slot_ids, image, None)

    def restore():
        kda.slot_copy(image, None, dec.pool, dec.slot_ids)

    def zero():
        kda.slot_zero(win.pool, free_slots)

    cv = inputs.make_workload("conv_16k", device=dev)
    cv_out = torch.empty_like(cv.x)

    def conv():
        kda.short_conv(cv.x, cv.weight, cv.cu_seqlens, silu=True, read_slots=cv.read_slots,
                       write_slots=cv.write_slots, conv_state=cv.state, out=cv_out)

    ext_parts = [("window_256x4", window), ("slot_checkpoint_256", checkpoint),
                 ("slot_restore_256", restore), ("slot_zero_256", zero),
                 ("short_conv_16k", conv)]
    for _ in range(args.warmup):
        for _, fn in ext_parts:
            fn()
    torch.cuda.synchronize()
    ext_ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)] for n, _ in ext_parts}
    torch.cuda._sleep(int(4e7))
    for i in range(args.steps):
        for n, fn in ext_parts:
            ext_ev[n][i][0].record(stream)
            fn()
            ext_ev[n][i][1].record(stream)
    torch.cuda.synchronize()
    ext_ms = {n: sum(a.elapsed_time(b) for a, b in ext_ev[n]) / args.steps for n, _ in ext_parts}
    red = max_over_ranks([ext_ms[n] for n, _ in ext_parts])
    for i, (n, _) in enumerate(ext_parts):
        ext_ms[n] = red[i]
    slot_bytes = H * STATE_BYTES
    ext_bytes = {
        "window_256x4": (Bw * H * (STATE_BYTES + Ww * STATE_BYTES)
                         + Bw * Ww * H * (3 * D * 2 + D * 4 + 4 + D * 2) + Bw * (Ww + 1) * 4),
        "slot_checkpoint_256": 2 * B * slot_bytes + B * 4,
        "slot_restore_256": 2 * B * slot_bytes + B * 4,
        "slot_zero_256": B * slot_bytes + B * 4,
        # x read once, out written once (bf16), weights, the two history windows
        "short_conv_16k": (2 * cv.x.numel() * cv.x.element_size() + cv.weight.numel() * 4
                           + 2 * cv.state[0].numel() * cv.state.element_size()),
    }
    extensions = {}
    for n, _ in ext_parts:
        gbs = ext_bytes[n] / (ext_ms[n] * 1e-3) / 1e9
        extensions[n] = {"ms": round(ext_ms[n], 4), "algorithmic_bytes": ext_bytes[n],
                         "gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4)}
    extensions["window_256x4"]["tokens_per_s"] = round(Bw * Ww / (ext_ms["window_256x4"] * 1e-3),
                                                       1)
    extensions["short_conv_16k"]["tokens_per_s"] = round(
        cv.x.shape[0] / (ext_ms["short_conv_16k"] * 1e-3), 1)
    del win, cv, cv_out

    # end to end through the public API with host buffers: every step copies its inputs in from
    # pinned host memory, runs kda_chunk_prefill and copies o and the final state back out.
    # Steps are pipelined over three streams (copy-in, compute, copy-out) with two buffer sets,
    # so that step i's copies overlap the neighbouring steps' prefill; step i + 2 reuses step
    # i's buffers once step i's prefill has read its inputs and its outputs are back on the host.
    h_in = [t.cpu().pin_memory() for t in (x.q, x.k, x.v, x.g, x.beta)]
    d_in = [[torch.empty_like(t) for t in (x.q, x.k, x.v, x.g, x.beta)] for _ in range(2)]
    o_b = [torch.empty_like(o) for _ in range(2)]
    f_b = [torch.empty_like(fin) for _ in range(2)]
    h_o = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
    h_f = [torch.empty(fin.shape, dtype=fin.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_o[0].numel() * h_o[0].element_size() + h_f[0].numel() * h_f[0].element_size()
    # (splitting the copy-in over several streams measured no faster: ~190 GB/s either way)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_k = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_k[b])  # step i - 2's prefill has read these inputs
            for h, d_ in zip(h_in, d_in[b]):
                d_.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if used[b]:
            stream.wait_event(ev_out[b])  # step i - 2's outputs are back on the host
        kda.chunk_prefill(*d_in[b], o=o_b[b], final_state=f_b[b], workspace=ws_pf)
        ev_k[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_k[b])
            h_o[b].copy_(o_b[b], non_blocking=True)
            h_f[b].copy_(f_b[b], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    def e2e_run(n):
        s_in.wait_stream(stream)
        for i in range(n):
            e2e_step(i)
        stream.wait_stream(s_out)

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_ms = max_over_ranks([e2e_ms])[0]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_heads, min_seconds=10.0)

    value = weak_scaling_value(T, world, comps["prefill_16k"]["ms"])
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; q,v~N(0,1), k L2-normalised, g=-softplus(N(0,1)), "
                "beta=sigmoid(N(0,1)))",
        "config": dict(CONFIG, parallelism=f"replicas{world}"),
        "components": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv)
                           for kk, vv in v.items()} for k, v in comps.items()},
        "roofline": roofline,
        "extensions": extensions,
        "e2e": {"value": round(weak_scaling_value(T, world, e2e_ms), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "what": "kda_chunk_prefill with pinned host inputs copied in and o/final state "
                        "copied out every step; steps pipelined over copy-in, compute and "
                        "copy-out streams with two buffer sets"},
        "gpu_launches": int(launches),
        "gpu_launches_per_step": launches / args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def cpu_baseline(heads, min_seconds=0.0, max_passes=30):
    """The oracle on a bounded sample of the prefill workload: `heads` of the 32 heads of the
    16k-token prompt (heads are independent), repeated as whole passes until at least
    `min_seconds` have elapsed (at most `max_passes`), scaled to whole-workload tokens/s."""
    import torch
    import oracle
    from linear_attention_state_kda_gb300 import inputs
    x = inputs.make_workload("prefill_16k", device="cpu")
    hs = list(range(heads))
    f = lambda t: t[:, hs].float().numpy().astype(np.float64)
    q, k, v, g, b = f(x.q), f(x.k), f(x.v), f(x.g), f(x.beta)
    cores = os.cpu_count() or 1
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.forward(q, k, v, g, b, threads=cores)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            break
    tokens_per_s = passes * x.T * (heads / x.H) / dt
    return {"value": round(tokens_per_s, 2), "unit": UNIT, "cores": min(cores, heads * 4),
            "kind": "oracle",
            "sample": f"{heads} of {x.H} heads of the 16k-token prefill (double precision, "
                      f"token by token), {passes} pass(es) in {dt:.2f} s, scaled by "
                      f"{x.H}/{heads} heads"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    per = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(args.cpu_heads)
        if i >= args.warmup:
            per.append(r)
    value = statistics.median([r["value"] for r in per])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": dict(CONFIG, parallelism=f"replicas{world}"),
        "cpu_baseline": {"value": value, "unit": UNIT, "kind": "oracle",
                         "cores": per[-1]["cores"], "sample": per[-1]["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """A small case of one call (inputs still larger than L2, a few GB on the device at most)
    for ncu captures: `--profile-case prefill|package|replay|scan|decode|window|slots|conv`,
    `--launches N`; `prefill16k` is the benchmark's full prefill launch, for single-pass
    counters only."""
    import torch
    from linear_attention_state_kda_gb300 import inputs, kda
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    case = args.profile_case
    if case == "decode":
        d = inputs.make_decode(256, 32, D, D, 1024, seed=1004, device=dev)
        fns = [lambda: kda.decode_step(d.q, d.k, d.v, d.g, d.beta, d.slot_ids, d.pool)]
    elif case == "window":
        w = inputs.make_window(128, 4, 32, D, D, 640, seed=1005, device=dev)
        fns = [lambda: kda.decode_window(w.q, w.k, w.v, w.g, w.beta_logit, w.read_slots,
                                         w.write_slots, w.pool, beta_is_logit=True)]
    elif case == "conv":
        cv = inputs.make_workload("conv_16k", device=dev)
        fns = [lambda: kda.short_conv(cv.x, cv.weight, cv.cu_seqlens, silu=True,
                                      read_slots=cv.read_slots, write_slots=cv.write_slots,
                                      conv_state=cv.state)]
    elif case == "slots":
        d = inputs.make_decode(256, 32, D, D, 1024, seed=1004, device=dev)
        image = torch.empty(256, 32, D, D, device=dev)
        fns = [lambda: kda.slot_copy(d.pool, d.slot_ids, image, None)]
    elif case == "prefill16k":  # the benchmark's own prefill launch (about 2 GB on the device)
        x = inputs.make_workload("prefill_16k", device=dev)
        fns = [lambda: kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta)]
    else:
        x = inputs.make_prefill([4096], 32, D, D, "bf16", seed=1001, device=dev)
        offs = torch.tensor([0, 2048, 4096], dtype=torch.int32, device=dev)
        sso = torch.tensor([0, 2], dtype=torch.int32, device=dev)
        M, Dp = kda.segment_package(x.k, x.v, x.g, x.beta, offs)
        si, _ = kda.package_scan(M, Dp, sso, 2)
        # the scan at the bench's tree shape: 8 packages per head (8 segments of 512 tokens)
        offs8 = torch.arange(0, 4097, 512, dtype=torch.int32, device=dev)
        sso8 = torch.tensor([0, 8], dtype=torch.int32, device=dev)
        M8, D8 = kda.segment_package(x.k, x.v, x.g, x.beta, offs8)
        si8, _ = kda.package_scan(M8, D8, sso8, 8)
        # the replay as the bench's segment path runs it: a walk over records prepared once
        # (the one-call kda_segment_replay takes the fused launch at this size)
        ws_r = kda.chunk_prepare(x.q, x.k, x.v, x.g, x.beta, offs) if case == "replay" else None
        fns = {
            "prefill": [lambda: kda.chunk_prefill(x.q, x.k, x.v, x.g, x.beta)],
            "package": [lambda: kda.segment_package(x.k, x.v, x.g, x.beta, offs, M=M, D=Dp)],
            "scan": [lambda: kda.package_scan(M8, D8, sso8, 8, seg_init=si8)],
            "replay": [lambda: kda.segment_replay_prepared(ws_r, offs, si, 4096, 32, D, D)],
        }[case]
    torch.cuda.synchronize()
    for _ in range(args.launches):
        for f in fns:
            f()
    torch.cuda.synchronize()
    print(f"profile case {case}: {args.launches} launch(es) done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile-case", default=None,
                    choices=["prefill", "prefill16k", "package", "scan", "replay", "decode",
                             "window", "slots", "conv"])
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-heads", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gb300(args)


if __name__ == "__main__":
    main()
