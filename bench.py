"""Benchmark of the window-attention hot path on GB300.

One step = the path between two NaDiT layers on the 720p-area workload
(T=21, H=45, W=80 -> 75,600 tokens, 24 heads x 128, bf16):
    regular-layout window attention (gather/scatter through the ids table)
 -> layout transition regular -> shifted of the hidden state [N, 3072]
 -> shifted-layout window attention.
Plans are built once per geometry (as a planner cache would) and timed
separately.  Inputs are seeded synthetic tensors resident in HBM; each of Q,
K, V is 464 MB, larger than the 129 MB L2, so no flush is needed between
steps.

`value` = window-attention FLOPs of both layers / step time (TFLOP/s).
Prints one JSON line on rank 0.  `--impl reference` times the fp64 CPU oracle
instead, on a bounded sample of the same workload.
"""

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The headline metric.  `value` is the attention FLOPs of all layers of a step
# divided by the step time (attention layers plus the transitions between
# them); tokens/s per layer and the fraction of tensor peak ride beside it.
METRIC = "window-attention TFLOP/s & tokens/s per layer (bf16, 1\u00d7GB300); % tensor peak"
# Clock event reasons that invalidate a timed region (power capping does not).
THROTTLE_REASONS = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one regular-layout attention launch of the
# 24-head 720p workload with canonical rows: an ncu capture of the same grid
# with 8 heads measured 886.1 MB (732.0 MB read, 154.1 MB written), scaled x3
# (each head's rows are disjoint, so traffic grows with the head count).
# Valid only for the kernel source and the work-list source (plan.cu, whose
# item order decides which key/value tiles are re-read) it was measured on.
MEASURED_TRAFFIC = {"kernel_sha1": "b89dd017275ec489", "plan_sha1": "2664da1284cc650f", "workload": "720p",
                    "heads": 24, "bytes": 2.658e9}


def source_sha1(name):
    import hashlib
    path = os.path.join(ROOT, "shifted_window_attention_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:16]


def kernel_sha1():
    return source_sha1("attention_tc.cu")


def attn_flops(offsets, heads, d, n_text=0):
    """Algorithmic attention FLOPs of one layer: 4 n^2 d per segment and head,
    a segment being a window's n_w video tokens plus n_text text tokens."""
    n = np.diff(np.asarray(offsets, dtype=np.float64)) + n_text
    return float(4.0 * np.sum(n * n) * d * heads)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(value, dist=None, device="cpu"):
    """The largest `value` over all ranks (the slowest rank sets a step's
    time); the value itself when not distributed."""
    import torch
    if dist is None or not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step, ms_per_step, world_size):
    """Aggregate throughput: every rank processes the same per-step work
    (weak scaling), in the time of the slowest rank."""
    return world_size * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return self.summarize(out)

    @staticmethod
    def summarize(out):
        """Median SM clock of the loaded samples, the maximum clock and the
        clock event reasons seen active, from nvidia-smi's CSV lines."""
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        busy = [s for s in sm if s > 0.5 * (max(smax) if smax else 1)] or sm
        return {"sm_mhz": float(np.median(busy)) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_config(wl, wsize, windows, packed=False, n_text=0, rope=-1, ws=1):
    """The bench line's `config`: the workload, named by what it is (grid,
    window sizes, heads, layers and what each step runs)."""
    N, C, L = wl.num_tokens, wl.channels, wl.layers
    desc = (f"{wl.name}: T={wl.T},H={wl.H},W={wl.W} ({N} tokens), nt,nh,nw={wl.nt},{wl.nh},{wl.nw} "
            f"-> wt,wh,ww={wsize[0]},{wsize[1]},{wsize[2]}; {wl.heads} heads x {wl.head_dim}; "
            f"{L} alternating layers ("
            + ("attention on rows in plan-packed order, full tiles by TMA" if packed
               else "attention gathers/scatters through ids")
            + f") with {L - 1} transitions of [N,{C}]"
            + (f"; segments [window, {n_text} text tokens], text mean over windows" if n_text else "")
            + (f"; window-local 3D RoPE of Q/K (text_len {rope}) before each attention" if rope >= 0 else ""))
    return {"workload": desc, "tokens": N, "heads": wl.heads, "head_dim": wl.head_dim, "layers": L,
            "text_tokens": n_text, "windows": list(windows),
            "l2": "inputs larger than L2 (Q/K/V >= 155 MB each); no flush",
            "parallelism": "replicas" if ws > 1 else "single"}


def host_link_gbs(host, device, stream):
    """Pinned host <-> device copy bandwidth (GB/s, each direction alone, best
    of three) measured right after the end-to-end leg: the host link is
    shared with the other GPUs of the machine, and this says what it gave."""
    import torch
    out = {}
    for name, dst, src in (("h2d", device, host), ("d2h", host, device)):
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                dst.copy_(src, non_blocking=True)
                b.record(stream)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        out[name] = round(src.numel() * src.element_size() / (best * 1e-3) / 1e9, 1)
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    import shifted_window_attention_gb300 as wsa
    import wsa_inputs

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = wsa_inputs.WORKLOADS[args.workload]
    if args.heads:
        # same grid, fewer heads: the small case used for detailed profiles
        wl = wsa_inputs.Workload(f"{wl.name}-{args.heads}h", wl.T, wl.H, wl.W, wl.nt, wl.nh, wl.nw,
                                 args.heads, wl.head_dim, wl.dtype, wl.dist, wl.layers)
    g = (wl.T, wl.H, wl.W, wl.nt, wl.nh, wl.nw)
    N, C, L = wl.num_tokens, wl.channels, wl.layers

    t0 = time.perf_counter()
    plans = [wsa.Plan(*g, wsa.REGULAR), wsa.Plan(*g, wsa.SHIFTED)]
    torch.cuda.synchronize()
    plan_ms = (time.perf_counter() - t0) * 1e3

    # Layer schedule: the layout each layer requires, as the model lists it
    # (NaDiT alternates regular and shifted windows).  Before every layer after
    # the first, ensure_layout(current, required) brings the hidden state
    # [N, C] into that layer's packed order; the transitions are derived from
    # this list, one wherever consecutive layers differ (L - 1 of them here).
    # Inputs: seeded Q/K/V per layer; schedules longer than 4 layers cycle 4
    # seeded input sets (the values do not change the work).
    layer_layouts = [(wsa.REGULAR, wsa.SHIFTED)[l % 2] for l in range(L)]
    n_sets = min(L, 4)
    sets = [wsa_inputs.qkv(wl, layer=i, device=dev) for i in range(n_sets)]
    canonical = not args.packed
    if args.packed:
        # rows in the plan-packed order of each set's layout (untimed setup)
        for i in range(n_sets):
            ids = plans[layer_layouts[i]].tables()[2].long()
            sets[i] = tuple(t[ids].contiguous() for t in sets[i])
    outs = [torch.empty_like(sets[i % n_sets][0]) for i in range(min(L, 2))]
    n_text = args.text
    if n_text:
        # replicated text tokens of each layer's segments (seeded like Q/K/V)
        tshape = (n_text, wl.heads, wl.head_dim)
        tsets = [tuple(wsa_inputs.randn(tshape, 900000 + 3 * i + j, dev).to(torch.bfloat16) for j in range(3))
                 for i in range(n_sets)]
        touts = [torch.empty(tshape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        wspace = [torch.empty(wsa.attention_text_workspace_bytes(p, n_text, wl.heads), dtype=torch.uint8, device=dev)
                  for p in plans]
    hidden = [wsa_inputs.activation(wl, device=dev), None]
    hidden[1] = torch.empty_like(hidden[0])
    stream = torch.cuda.current_stream()

    flops = [attn_flops(p.tables()[0].cpu().numpy(), wl.heads, wl.head_dim, n_text) for p in plans]
    fl_step = sum(flops[layer_layouts[l]] for l in range(L))
    trans_bytes = 2.0 * N * C * 2 + 2 * 4.0 * N  # read + write rows, two int32 table reads

    use_rope = args.rope >= 0
    if use_rope:
        # rotated Q/K of the current layer (window-local positions of its layout)
        qk_rot = [(torch.empty_like(sets[0][0]), torch.empty_like(sets[0][1])) for _ in range(2)]
        if n_text:
            tqk_rot = [(torch.empty_like(tsets[0][0]), torch.empty_like(tsets[0][1])) for _ in range(2)]
    # Q and K rows read + written, the ids table; the text rows when present
    rope_bytes = 2 * (2.0 * N * C * 2) + 4.0 * N + 2 * (2.0 * n_text * C * 2)

    # per layer: [before RoPE, before attention, after attention, after transition]
    n_ev = 4 * L
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]

    def step(i=None):
        """One pass over the layer list; returns the transitions it ran."""
        e = ev[i] if i is not None else None
        h, spare, moves = hidden[0], hidden[1], 0
        for l in range(L):
            p = plans[layer_layouts[l]]
            q, k, v = sets[l % n_sets]
            if e: e[4 * l].record(stream)
            if use_rope:
                qr, kr = qk_rot[l % 2]
                wsa.rope(p, q, k, q_out=qr, k_out=kr, canonical=canonical, text_len=args.rope)
                q, k = qr, kr
            if n_text:
                qt, kt, vt = tsets[l % n_sets]
                if use_rope:
                    qt, kt = wsa.rope_text(qt, kt, q_out=tqk_rot[l % 2][0], k_out=tqk_rot[l % 2][1])
            if e: e[4 * l + 1].record(stream)
            if n_text:
                wsa.attention_text(p, q, k, v, qt, kt, vt, out=outs[l % 2],
                                   out_txt=touts[l % 2], workspace=wspace[l % 2])
            else:
                wsa.attention(p, q, k, v, out=outs[l % 2], canonical=canonical)
            if e: e[4 * l + 2].record(stream)
            if l + 1 < L:
                # the hidden state enters the next layer's layout
                x = wsa.ensure_layout(p, plans[layer_layouts[l + 1]], h, out=spare)
                if x is not h:
                    h, spare, moves = x, h, moves + 1
            if e: e[4 * l + 3].record(stream)
        return moves

    for _ in range(args.warmup):
        transitions = step()
    torch.cuda.synchronize()
    if any(p.device_status() for p in plans):
        raise RuntimeError("device error during warm-up")

    def timed_region():
        clocks = ClockSampler(local)
        clocks.start()
        time.sleep(0.3)
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(args.steps):
            step(i)
        end.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        return start.elapsed_time(end), clocks.stop()

    total_ms, clk = timed_region()
    # A timed region that saw hardware or thermal slowdown is measured once more
    # (every rank together); the second measurement is the one reported.
    slow = float(bool(THROTTLE_REASONS & set(clk["reasons"])))
    if max_over_ranks(slow, dist if ws > 1 else None, dev) > 0:
        first = clk["reasons"]
        total_ms, clk = timed_region()
        clk["remeasured_after"] = first
    attn = np.array([[e[4 * l + 1].elapsed_time(e[4 * l + 2]) for l in range(L)] for e in ev])  # [steps, L]
    trans = np.array([[e[4 * l + 2].elapsed_time(e[4 * l + 3]) for l in range(L - 1)] for e in ev])
    rope_t = np.array([[e[4 * l].elapsed_time(e[4 * l + 1]) for l in range(L)] for e in ev])
    total_ms = max_over_ranks(total_ms, dist if ws > 1 else None, dev)
    ms_step = total_ms / args.steps
    if any(p.device_status() for p in plans):
        raise RuntimeError("device error during the timed region")

    # End to end through the public API with pinned host buffers (two-layer
    # workloads).  Every step uploads its inputs (Q/K/V of both layers and the
    # hidden rows) from pinned host memory, runs the three calls, and
    # downloads the two attention outputs and the transitioned rows.  Steps
    # are pipelined as a serving loop would run them: uploads, compute and
    # downloads go on three streams over two device buffer sets, so step i+1's
    # upload overlaps step i's compute and step i-1's download.  The timed
    # region runs from the first upload to the last download.
    e2e = None
    if L == 2 and not args.no_e2e and not n_text and not use_rope:
        dev_sets = [list(sets[0]) + list(sets[1]) + [hidden[0]]]
        dev_sets.append([torch.empty_like(t) for t in dev_sets[0]])
        out_sets = [[outs[0], outs[1], hidden[1]], [torch.empty_like(t) for t in (outs[0], outs[1], hidden[1])]]
        host_in = [t.cpu().pin_memory() for t in dev_sets[0]]
        host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in out_sets[0]] for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out[0])
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        in_ready = [torch.cuda.Event() for _ in range(2)]
        comp_done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        e2e_steps = max(2, args.steps)
        # per-step timeline of the timed run: [upload start, upload end,
        # compute start, compute end, download start, download end], each
        # recorded on the stream that does the work
        tl = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(e2e_steps)]

        def e2e_run(n, timeline=None):
            for i in range(n):
                b = i % 2
                t = timeline[i] if timeline else None
                din, dout = dev_sets[b], out_sets[b]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(comp_done[b])  # buffer set b no longer read by step i-2
                    if t: t[0].record(s_in)
                    for d_, h_ in zip(din, host_in):
                        d_.copy_(h_, non_blocking=True)
                    if t: t[1].record(s_in)
                    in_ready[b].record(s_in)
                stream.wait_event(in_ready[b])
                if i >= 2:
                    stream.wait_event(out_done[b])  # step i-2's outputs have left set b
                q0, k0, v0, q1, k1, v1, x = din
                if t: t[2].record(stream)
                wsa.attention(plans[0], q0, k0, v0, out=dout[0], canonical=canonical)
                wsa.transition(plans[0], plans[1], x, out=dout[2])
                wsa.attention(plans[1], q1, k1, v1, out=dout[1], canonical=canonical)
                if t: t[3].record(stream)
                comp_done[b].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(comp_done[b])
                    if t: t[4].record(s_out)
                    for h_, d_ in zip(host_out[b], dout):
                        h_.copy_(d_, non_blocking=True)
                    if t: t[5].record(s_out)
                    out_done[b].record(s_out)

        e2e_run(2)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        es.record(s_in)
        e2e_run(e2e_steps, tl)
        s_out.wait_stream(s_in)
        s_out.wait_stream(stream)
        ee.record(s_out)
        torch.cuda.synchronize()
        if any(p.device_status() for p in plans):
            raise RuntimeError("device error during the end-to-end leg")
        e2e_ms = max_over_ranks(es.elapsed_time(ee) / e2e_steps, dist if ws > 1 else None, dev)
        up = [t[0].elapsed_time(t[1]) for t in tl]
        comp = [t[2].elapsed_time(t[3]) for t in tl]
        down = [t[4].elapsed_time(t[5]) for t in tl]
        # time during which an upload and a download of different steps ran at once
        both = 0.0
        for i in range(1, e2e_steps):
            a0, a1 = es.elapsed_time(tl[i][0]), es.elapsed_time(tl[i][1])
            b0, b1 = es.elapsed_time(tl[i - 1][4]), es.elapsed_time(tl[i - 1][5])
            both += max(0.0, min(a1, b1) - max(a0, b0))
        timeline = {"upload_ms": round(float(np.mean(up)), 3), "compute_ms": round(float(np.mean(comp)), 3),
                    "download_ms": round(float(np.mean(down)), 3),
                    "upload_gbs": round(h2d / (np.mean(up) * 1e-3) / 1e9, 1),
                    "download_gbs": round(d2h / (np.mean(down) * 1e-3) / 1e9, 1),
                    "upload_download_overlap_ms_per_step": round(both / max(1, e2e_steps - 1), 3)}
        e2e = {"value": round(whole_job_tflops(fl_step, e2e_ms, ws), 2), "unit": "TFLOP/s",
               "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "steps": e2e_steps,
               "pipeline": "uploads, compute and downloads on three streams, two device buffer sets",
               "timeline": timeline,
               "host_link_gbs": host_link_gbs(host_in[0], dev_sets[0][0], s_in)}

    peaks, peak_kind = load_peaks()
    traffic, traffic_note = None, "no ncu capture for this kernel source / workload"
    mt = MEASURED_TRAFFIC
    if (kernel_sha1() == mt["kernel_sha1"] and source_sha1("plan.cu") == mt["plan_sha1"]
            and wl.name == mt["workload"] and wl.heads == mt["heads"]
            and not n_text and not args.packed):
        traffic = mt["bytes"]
        traffic_note = ("DRAM bytes of the regular-layout launch (ncu capture of the 8-head case scaled x3); "
                        f"algorithmic {4.0 * N * wl.channels * 2:.3e} B")
    fp32 = wl.dtype == "fp32"
    if fp32:
        # The fp32 path runs on the CUDA cores (FFMA): 128 fp32 lanes per SM,
        # 2 FLOP per FMA, at the SM clock sampled during the timed region.
        sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
        mhz = clk.get("sm_mhz") or 2070.0
        alu_peak = sm_count * 128 * 2 * mhz * 1e6 / 1e12
    kinds = np.array(layer_layouts)
    a_reg = attn[:, kinds == wsa.REGULAR].mean()
    a_sft = attn[:, kinds == wsa.SHIFTED].mean() if (kinds == wsa.SHIFTED).any() else float("nan")
    attn_ms = attn.mean()
    fl_launch = fl_step / L
    achieved = fl_launch / (attn_ms * 1e-3) / 1e12
    t_mean = float(trans.mean()) if L > 1 else float("nan")
    per_layer = {
        "attention_ms": [round(float(a_reg), 4), round(float(a_sft), 4)],
        "attention_tflops": [round(flops[0] / (a_reg * 1e9), 1), round(flops[1] / (a_sft * 1e9), 1)],
        "tokens_per_s": [round(N / (a_reg * 1e-3)), round(N / (a_sft * 1e-3))],
        "transition_ms": round(t_mean, 4),
        "transition_gbs": round(trans_bytes / (t_mean * 1e6), 1),
        "transition_frac_hbm": round(trans_bytes / (t_mean * 1e6) / peaks["hbm_gbs"], 4),
        "plan_build_ms_host_incl": round(plan_ms, 3),
    }
    if use_rope:
        r_mean = float(rope_t.mean())
        per_layer["rope_ms"] = round(r_mean, 4)
        per_layer["rope_gbs"] = round(rope_bytes / (r_mean * 1e6), 1)
        per_layer["rope_frac_hbm"] = round(rope_bytes / (r_mean * 1e6) / peaks["hbm_gbs"], 4)
    if L > 2:
        per_layer["attention_ms_by_layer"] = [round(float(x), 4) for x in attn.mean(axis=0)]
        per_layer["transition_ms_by_boundary"] = [round(float(x), 4) for x in trans.mean(axis=0)]
    dist_note = {"normal": "N(0,1)", "normal_half_var": "N(0,1)/sqrt(2)",
                 "outlier": "Q,K N(0,1) with 1% of channels x8, V N(0,1)"}[wl.dist]
    result = {
        "metric": METRIC,
        "value": round(whole_job_tflops(fl_step, ms_step, ws), 2),
        "unit": "TFLOP/s",
        "tokens_per_s": round(N * L * ws / (ms_step * 1e-3)),
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if fp32 else "bf16",
        "data": f"synthetic (seeded torch.randn, {dist_note}, {'fp32' if fp32 else 'bf16'})",
        "config": workload_config(wl, (plans[0].wt, plans[0].wh, plans[0].ww),
                                  [plans[0].num_windows, plans[1].num_windows], args.packed, n_text, args.rope, ws),
        "per_layer": per_layer,
        "roofline": {
            "bound": "tensor",
            "kernel": "attention_tc_kernel",
            "achieved": round(achieved, 2),
            "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": round(achieved / peaks["bf16_tflops"], 4),
            "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
            "peak_source": f"{peak_kind} bf16 burst",
            "traffic": traffic,
            "traffic_note": traffic_note,
        } if not fp32 else {
            "bound": "alu",
            "kernel": "attention_fp32_kernel",
            "achieved": round(achieved, 4),
            "peak": round(alu_peak, 2),
            "unit": "TFLOP/s",
            "frac": round(achieved / alu_peak, 5),
            "peak_source": "derived: SMs x 128 fp32 lanes x 2 FLOP x sampled SM clock",
            "traffic": None,
            "traffic_note": "launch-bound parity workload; no ncu capture",
        },
        "e2e": e2e,
        # per layer: attention (+ text reduction), RoPE pass(es)
        "gpu_launches": (((2 if n_text else 1) + (0 if not use_rope else 2 if n_text else 1)) * L + transitions)
                        * args.steps,
        "clocks": clk,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:  # the CPU baseline is an N = 1 figure
        q0, k0, v0 = sets[0]
        result["cpu_baseline"] = cpu_baseline(wl, tuple(t.float().cpu().numpy() for t in (q0, k0, v0)),
                                              seconds=args.cpu_seconds)
    if ws > 1:
        dist.destroy_process_group()
    return result if rank == 0 else None


def run_plan_a(args):
    """Plan A device kernels at a layout boundary, ranks emulated on one GPU.

    Each of R emulated ranks packs its rows (wsa_gather_rows through
    send_index) and unpacks its receive buffer (through recv_index), for both
    boundaries regular -> shifted and shifted -> regular.  The collective
    between them is not timed: on one GPU it is emulated by slicing the send
    buffers into receive buffers once, before the timed region.  Algorithmic
    bytes per boundary: every row is read and written once by a pack and once
    by an unpack, plus one int32 index read per row for each."""
    import torch
    import shifted_window_attention_gb300.sp as sp
    import wsa_inputs

    wl = wsa_inputs.WORKLOADS[args.workload]
    R = args.plan_a
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    grid = (wl.T, wl.H, wl.W, wl.nt, wl.nh, wl.nw)
    N, C = wl.num_tokens, wl.channels
    x = wsa_inputs.activation(wl, device=dev)
    legs = []
    for src_l, dst_l in ((0, 1), (1, 0)):
        plans = [sp.PlanA(*grid, src_l, dst_l, R, r) for r in range(R)]
        xl = [x[torch.from_numpy(sp.local_rows(*grid, src_l, R, r).astype(np.int64)).to(dev)].contiguous()
              for r in range(R)]
        sends = [torch.empty((p.n_send, C), dtype=x.dtype, device=dev) for p in plans]
        for r in range(R):
            plans[r].pack(xl[r], out=sends[r])
        bounds = [np.concatenate([[0], np.cumsum(p.input_split_sizes)]) for p in plans]
        recvs = [torch.cat([sends[r][bounds[r][d]:bounds[r][d + 1]] for r in range(R)]).contiguous()
                 for d in range(R)]
        outs = [torch.empty((p.n_recv, C), dtype=x.dtype, device=dev) for p in plans]
        legs.append((plans, xl, sends, recvs, outs))
    stream = torch.cuda.current_stream()

    def step():
        for plans, xl, sends, recvs, outs in legs:
            for r in range(R):
                plans[r].pack(xl[r], out=sends[r])
            for d in range(R):
                plans[d].unpack(recvs[d], out=outs[d])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    def timed_region():
        clocks = ClockSampler(0)
        clocks.start()
        time.sleep(0.3)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / args.steps, clocks.stop()

    ms, clk = timed_region()
    if THROTTLE_REASONS & set(clk["reasons"]):
        first = clk["reasons"]
        ms, clk = timed_region()
        clk["remeasured_after"] = first
    step_bytes = 2 * (2 * (2.0 * N * C * x.element_size()) + 2 * 4.0 * N)
    gbs = step_bytes / (ms * 1e-3) / 1e9
    peaks, peak_kind = load_peaks()
    hbm = peaks["hbm_gbs"]
    return {
        "metric": "Plan A pack + unpack bandwidth (both boundaries, ranks emulated on one GPU)",
        "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded torch.randn rows, bf16)",
        "config": {"workload": f"{wl.name}: [N={N}, C={C}] hidden rows, {R} emulated ranks, regular <-> shifted; "
                               "collective emulated outside the timed region",
                   "ranks": R, "l2": "inputs larger than L2 (464 MB of rows); no flush"},
        "roofline": {"bound": "hbm", "kernel": "transition_rows_kernel (one-level gather)",
                     "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(gbs / hbm, 4), "peak_source": f"{peak_kind} copy bandwidth", "traffic": None},
        "gpu_launches": 4 * R * args.steps,
        "clocks": clk,
    }


def cpu_inputs(wl):
    """The workload's layer-0 Q/K/V as fp32 numpy arrays (drawn on the GPU when
    one is present, which is faster; the CPU draw otherwise)."""
    import torch
    import wsa_inputs
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    return tuple(t.float().cpu().numpy() for t in wsa_inputs.qkv(wl, layer=0, device=dev))


def cpu_baseline(wl, inputs, seconds=15.0, layout=0, seed=0):
    """Time the fp64 oracle as it stands on a bounded sample of the workload:
    whole (window, head) problems of one layout, in seeded order, through
    oracle.window_attention_rows, until `seconds` of CPU work are done.
    Returns TFLOP/s of algorithmic attention work."""
    import oracle

    q, k, v = inputs
    g = (wl.T, wl.H, wl.W, wl.nt, wl.nh, wl.nw)
    p = oracle.make_plan(*g, layout)
    rng = np.random.default_rng(seed)
    order = [(int(w), int(h)) for w in rng.permutation(p.num_windows) for h in rng.permutation(wl.heads)]
    flops, done, t_total = 0.0, 0, 0.0
    for (w, h) in order:
        n = int(p.offsets[w + 1] - p.offsets[w])
        t0 = time.perf_counter()
        oracle.window_attention_rows(q, k, v, p, w, h, np.arange(n))
        t_total += time.perf_counter() - t0
        flops += 4.0 * n * n * wl.head_dim
        done += 1
        if t_total >= seconds:
            break
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count()
    return {"value": round(flops / t_total / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} whole (window, head) problems of the {wl.name} "
                      f"{'regular' if layout == 0 else 'shifted'} layer, fp64 numpy, {t_total:.1f} s"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    import wsa_inputs
    wl = wsa_inputs.WORKLOADS[args.workload]
    g = (wl.T, wl.H, wl.W, wl.nt, wl.nh, wl.nw)
    inputs = cpu_inputs(wl)
    vals = []
    per = max(2.0, 90.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(wl, inputs, seconds=per, layout=i % 2, seed=i)
        if i >= args.warmup:
            vals.append(r)
    value = float(np.mean([r["value"] for r in vals]))
    cores = vals[0]["cores"]
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, oracle.window_size(wl.T, wl.H, wl.W, wl.nt, wl.nh, wl.nw),
                                  [oracle.make_plan(*g, lay).num_windows for lay in (0, 1)], ws=ws),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: {vals[0]['sample']}"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="720p")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--heads", type=int, default=0, help="override the head count (small profiling case)")
    ap.add_argument("--text", type=int, default=0, help="replicated text tokens appended to every window segment")
    ap.add_argument("--rope", type=int, default=-1,
                    help="apply window-local 3D RoPE to Q/K before every attention, with this text_len (>= 0)")
    ap.add_argument("--packed", action="store_true",
                    help="attention on Q/K/V rows in plan-packed order (what the transition produces) instead of "
                         "canonical rows gathered through ids")
    ap.add_argument("--plan-a", type=int, default=0,
                    help="time the Plan A pack/unpack kernels for this many emulated ranks instead")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.plan_a and args.impl == "ours":
        res = run_plan_a(args)
    else:
        res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
