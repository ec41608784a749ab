"""Throughput of streaming two-stream paged-KV attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload steady_state_10k] [--impl reference]

A step is one frame-step of the whole hot path for one stream set: append of the
frame's K/V for every block, one evict, one plan, and attention (+ merge) for every
block.  The default workload is the 10,000-frame steady state (24 blocks, 16 heads
of 64, 256 patch + 6 special tokens per frame, 8 scale frames, 64-frame window):
the stream is fast-forwarded (append + evict for every block) to frame
10000 - K - W, then W warm-up and K timed frame-steps run on device-resident
inputs.  Visible K/V per block (~322 MB) exceeds L2, so no flush is needed between
steps.

Printed: one JSON line with the metric, a roofline object for the attention
launch (algorithmic bytes per block / CUDA-event launch time, against the
measured HBM copy bandwidth), an end-to-end figure through host buffers, the fp64
oracle timed on the host cores (cpu_baseline) and the SM clocks sampled during the
timed region.  With --gpus N > 1 (torchrun), every rank runs its own stream
(weak scaling, no collective on the data path); the slowest rank's time counts.

--impl reference times the fp64 CPU oracle itself (the only reference that
exists for this path) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)

import workloads as wl  # noqa: E402

METRIC = "paged-attn frame-steps/s (all blocks, 1 GB300); % of attention roofline"
UNIT = "frame-steps/s"


# ---------------------------------------------------------------- rank helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, world_size=world, rank=rank)
    return world, rank


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Max of a scalar over ranks (timing only: no data-path collective)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(steps_per_rank: int, world: int, max_seconds: float) -> float:
    """Whole-job frame-steps/s: every rank's steps over the slowest rank's time."""
    return steps_per_rank * world / max_seconds


# ---------------------------------------------------------------- roofline helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def fp32_alu_peak_tflops() -> float:
    """fp32 FMA peak of the CUDA cores: SMs x 128 FMA lanes x 2 FLOP x maximum SM clock
    (the clock from MEASURED_PEAKS.json, else the GB300's 2070 MHz)."""
    mhz = 2070.0
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            mhz = float(json.load(fh).get("sm_max_mhz", mhz))
    return 152 * 128 * 2 * mhz * 1e6 / 1e12


def visible_tokens(w: wl.Workload, f: int) -> int:
    """Visible keys per stream after f frames: (min(f,sc) + min(max(f-sc,0),w)) * P + f * S."""
    sc, win, P, S = w.scale_frames, w.sliding_window, w.patches_per_frame, w.specials_per_frame
    return (min(f, sc) + min(max(f - sc, 0), win)) * P + f * S


def block_work(w: wl.Workload, f: int):
    """Algorithmic FLOPs and bytes of one block's attention at frame f (all streams):
    F = 4 T N H D B, bytes = (2N + 2T) H D e B (visible K+V once, q read, out written)."""
    n = visible_tokens(w, f)
    t, h, d, b, e = w.tokens_per_frame, w.num_heads, w.head_dim, w.num_streams, wl.element_bytes(w)
    return 4.0 * t * n * h * d * b, (2.0 * n + 2.0 * t) * h * d * e * b


# ---------------------------------------------------------------- ncu traffic record

KERNEL_SOURCES = ("streaming_paged_kv_two_gb300/csrc/spk_attn_tc.cu", "streaming_paged_kv_two_gb300/csrc/ptx_sm100.cuh",
                  "streaming_paged_kv_two_gb300/csrc/spk_internal.h", "streaming_paged_kv_two_gb300/csrc/spk_kernels.cu")


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: line comments and blank lines are left out, so
    editing a comment does not retire the recorded counters."""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
            for line in fh:
                code = re.sub(r"//.*$", "", line).strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per attention launch (attention + merge kernels) from the committed ncu
    record, or None when the record is missing, for another workload, or older than the
    kernel sources."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    if rec.get("source_hash") != kernel_source_hash() or rec.get("workload") != workload:
        return None
    return float(rec["dram_bytes_per_launch"])


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.device_index = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
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
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0])); mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- CPU oracle sample

def oracle_block_sample(w: wl.Workload, frame_count: int, heads: int, reps: int, budget_s: float):
    """Time the fp64 oracle (bookkeeping of one frame + gather + dense attention of one
    block restricted to `heads` heads) at the steady state; returns per-rep seconds
    and the extrapolated frame-steps/s."""
    import oracle
    from oracle_cases import make_streams

    st = make_streams(w.replace(num_streams=1))[0]
    for _ in range(frame_count - 1):
        st.append(); st.evict()
    hs = slice(0, heads)
    # input generation is not timed: draw every frame a rep can see, once, head-sliced
    P = w.patches_per_frame
    last = frame_count + reps
    patch_frames = set(range(min(last, w.scale_frames))) | set(range(max(0, frame_count - w.sliding_window - 1), last))
    patch, special = {}, {}
    for frame in sorted(patch_frames):
        kp, vp = wl.frame_patch_kv(w, 0, 0, frame)
        patch[frame] = (wl.to_f64(kp, w.dtype)[:, hs], wl.to_f64(vp, w.dtype)[:, hs])
    for frame in range(last):
        ks, vs = wl.frame_special_kv(w, 0, 0, frame)
        special[frame] = (wl.to_f64(ks, w.dtype)[:, hs], wl.to_f64(vs, w.dtype)[:, hs])
    q = wl.to_f64(wl.frame_q(w, 0, 0, frame_count - 1), w.dtype)[:, hs]

    def fetch(frame, rows):
        rows = np.asarray(rows)
        if rows[0] < P:
            k, v = patch[frame]
            return k[rows], v[rows]
        k, v = special[frame]
        return k[rows - P], v[rows - P]

    times = []
    t_start = time.perf_counter()
    for i in range(reps):
        t0 = time.perf_counter()
        st.append(); st.evict()
        oracle.plan([st], w.tokens_per_frame)
        k, v = oracle.gather_visible(st.visible_sources(), fetch)
        oracle.attend(q, k, v)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > budget_s:
            break
    per_block = statistics.mean(times) * (w.num_heads / heads)
    value = 1.0 / (per_block * w.num_blocks)
    return times, value


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


# ---------------------------------------------------------------- reference arm

def run_reference(args, w: wl.Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    frame = w.frames
    heads = min(args.ref_heads, w.num_heads)
    # warm-up reps are discarded, then K reps timed
    oracle_block_sample(w.replace(frames=frame + 4), frame, heads, max(args.warmup, 1), budget_s=60.0)
    times, value = oracle_block_sample(w.replace(frames=frame + args.steps + 4), frame, heads, args.steps,
                                       budget_s=240.0)
    ms = 1000.0 / value
    cores = blas_threads()
    sample = (f"per step: one frame of bookkeeping + gather + fp64 attention of block 0 over {heads} of "
              f"{w.num_heads} heads at frame {frame} ({visible_tokens(w, frame)} visible keys); "
              f"frame-steps/s extrapolated x{w.num_heads // heads} heads x{w.num_blocks} blocks; "
              f"{len(times)} steps timed; ms_per_step is 1000/value, i.e. extrapolated the same way, "
              f"not a timed full step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": len(times), "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, frame),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def workload_config(w: wl.Workload, frame: int) -> dict:
    return {"workload": w.name, "blocks": w.num_blocks, "streams": w.num_streams, "heads": w.num_heads,
            "head_dim": w.head_dim, "page_size": w.page_size, "patches_per_frame": w.patches_per_frame,
            "specials_per_frame": w.specials_per_frame, "scale_frames": w.scale_frames,
            "sliding_window": w.sliding_window, "frames_streamed": frame,
            "visible_tokens_per_stream": visible_tokens(w, frame)}


# ---------------------------------------------------------------- GPU arm

def run_gpu(args, w: wl.Workload):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist_init("nccl")
    import streaming_paged_kv_two_gb300 as spk
    from workload_device import spk_config_for, to_device

    K, W = args.steps, args.warmup
    total_frames = w.frames
    extra = W + 2 * K + 8                   # the launch-timing, append-timing and e2e passes stream past the steady-state frame
    wk = w.replace(frames=total_frames + extra)
    cfg, keep = spk_config_for(wk, args.splits)
    pool_bytes, ws_bytes = spk.required_bytes(cfg)
    dev = torch.device("cuda", local)
    pools = [torch.empty(pool_bytes, dtype=torch.uint8, device=dev) for _ in range(w.num_blocks)]
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    cache = spk.Cache(cfg, pools, keep)
    stream = torch.cuda.current_stream()
    B, L, T = w.num_streams, w.num_blocks, w.tokens_per_frame

    # device-resident inputs: NV frame variants per (stream, block), drawn by the workload generator
    NV = 2
    qs = [[[to_device(wl.frame_q(w, s, b, vi), w.dtype) for b in range(L)] for s in range(B)] for vi in range(NV)]
    kvs = [[[tuple(to_device(x, w.dtype) for x in wl.frame_kv(w, s, b, vi)) for b in range(L)] for s in range(B)]
           for vi in range(NV)]
    qcat = [[torch.cat([qs[vi][s][b] for s in range(B)]) for b in range(L)] for vi in range(NV)]
    outs = [torch.empty_like(qcat[0][b]) for b in range(L)]
    # --rope: append through the fused rotary scatter; q is turned into qrot, which attention reads
    sections, theta = wl.rope_sections(w), 10000.0
    qrot = [torch.empty_like(qcat[0][b]) for b in range(L)] if args.rope else None
    pos_all = (torch.from_numpy(np.stack([wl.frame_positions(w, x) for x in range(wk.frames)])).to(dev)
               if args.rope else None)
    ev_app = []

    def append_one(f, s, b, k, v, q=None, pos=None):
        if not args.rope:
            cache.append_frame(s, b, k, v, stream)
            return
        pos = pos_all[f] if pos is None else pos
        cache.append_frame_rope(s, b, k, v, q if q is not None else qs[f % NV][s][b], qrot[b][s * T:(s + 1) * T],
                                pos, sections, theta, stream)

    def append_all(f, b, timed=False):
        vi = f % NV
        for s in range(B):
            k, v = kvs[vi][s][b]
            if timed:
                a0 = torch.cuda.Event(enable_timing=True)
                a1 = torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                append_one(f, s, b, k, v)
                a1.record(stream)
                ev_app.append((a0, a1))
            else:
                append_one(f, s, b, k, v)

    # fast-forward: frames whose attention is not timed only need their K/V appended
    t_ff = time.perf_counter()
    pre = max(0, total_frames - K - W)
    for f in range(pre):
        for s in range(B):
            k, v = kvs[f % NV][s][0]
            append_one(f, s, 0, k, v)
            cache.evict_frames(s)
        for b in range(1, L):
            append_all(f, b)
    torch.cuda.synchronize()
    t_ff = time.perf_counter() - t_ff

    ev_pairs = []

    def frame_step(f, timed_launches=False, timed_appends=False, q_override=None, out_override=None):
        vi = f % NV
        for s in range(B):
            k, v = kvs[vi][s][0]
            append_one(f, s, 0, k, v)
        for s in range(B):
            cache.evict_frames(s)
        cache.plan(ws, stream)
        for b in range(L):
            if b:
                append_all(f, b, timed=timed_appends)
            q = (qrot[b] if args.rope else qcat[vi][b]) if q_override is None else q_override[b]
            o = outs[b] if out_override is None else out_override[b]
            if timed_launches:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                cache.run_attention(b, q, o, ws, stream)
                e1.record(stream)
                ev_pairs.append((e0, e1))
            else:
                cache.run_attention(b, q, o, ws, stream)

    f = pre
    for _ in range(W):
        frame_step(f)
        f += 1
    info = cache.get_plan_info()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    f_first = f
    torch.cuda.nvtx.range_push("timed")
    t0.record(stream)
    for _ in range(K):
        frame_step(f)
        f += 1
    t1.record(stream)
    torch.cuda.nvtx.range_pop()
    # the same K frame-steps again with events around every spk_run_attention call, for
    # the per-launch time of the roofline (events between kernels keep a launch from
    # overlapping the kernel before it, so the step time above is taken without them)
    for _ in range(K):
        frame_step(f, timed_launches=True)
        f += 1
    torch.cuda.synchronize()
    clk = clocks.stop()
    elapsed = t0.elapsed_time(t1) / 1000.0
    barrier()
    max_elapsed = reduce_max(elapsed, device=dev)
    status = spk.read_device_status(ws, stream)
    launch_ms = [a.elapsed_time(b) for a, b in ev_pairs]
    # appends timed on their own, outside the timed region (events around every append
    # launch would slow the step they measure)
    for _ in range(2):
        frame_step(f, timed_appends=True)
        f += 1
    torch.cuda.synchronize()
    append_ms = [a.elapsed_time(b) for a, b in ev_app]

    # ------------------------------------------------ e2e: host buffers, copies in the timed region
    # Every step copies its q/k/v from pinned host memory and its outputs back.  A step's
    # inputs sit in one pinned host buffer (per frame variant: q of each block, then k and
    # v of each (stream, block)) and go to the device in one copy; its outputs come back
    # in one copy.  The copies run on their own streams and the device sets are double
    # buffered, so step f+1's inputs move while step f computes; events order each copy
    # against the compute stream.  Step f+1's input copy starts once step f's plan is
    # uploaded: the plan upload is itself a host->device copy on the compute stream and
    # would otherwise queue behind the larger input copy.
    q_elems = [qcat[0][b].numel() for b in range(L)]
    kv_elems = T * w.num_heads * w.head_dim
    per_block = q_elems[0] + 2 * B * kv_elems
    hin = []
    for vi in range(NV):
        parts = []
        for b in range(L):
            parts.append(qcat[vi][b].reshape(-1))
            for s in range(B):
                parts += [kvs[vi][s][b][0].reshape(-1), kvs[vi][s][b][1].reshape(-1)]
        hin.append(torch.cat(parts).cpu().pin_memory())
    din = [torch.empty_like(hin[0], device=dev) for _ in range(2)]

    def in_views(st):
        buf, dq, dkv = din[st], [], [[None] * L for _ in range(B)]
        for b in range(L):
            o = b * per_block
            dq.append(buf[o:o + q_elems[b]].view(qcat[0][b].shape))
            o += q_elems[b]
            for s in range(B):
                dkv[s][b] = (buf[o:o + kv_elems].view(kvs[0][s][b][0].shape),
                             buf[o + kv_elems:o + 2 * kv_elems].view(kvs[0][s][b][1].shape))
                o += 2 * kv_elems
        return dq, dkv

    views = [in_views(0), in_views(1)]
    dout = [torch.empty((L,) + tuple(outs[0].shape), dtype=outs[0].dtype, device=dev) for _ in range(2)]
    hout = torch.empty(dout[0].shape, dtype=dout[0].dtype).pin_memory()
    hpos = pos_all.cpu().pin_memory() if args.rope else None          # [frame, T, 3]
    dpos = [torch.empty_like(pos_all[0]) for _ in range(2)] if args.rope else None
    h2d = hin[0].numel() * hin[0].element_size() + (hpos[0].numel() * hpos[0].element_size() if args.rope else 0)
    d2h = hout.numel() * hout.element_size()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]      # inputs of set st landed
    ev_planned = torch.cuda.Event()                     # the last step's plan is uploaded (and the step
    planned = [False]                                   # before it is done with its inputs)
    ev_out = [torch.cuda.Event() for _ in range(2)]     # dout[st] written
    ev_back = [None, None]                              # dout[st] copied to the host

    def e2e_step(f):
        vi, st = f % NV, f % 2
        dq, dkv = views[st]
        with torch.cuda.stream(up):
            if planned[0]:
                up.wait_event(ev_planned)
            din[st].copy_(hin[vi], non_blocking=True)
            if args.rope:
                dpos[st].copy_(hpos[f], non_blocking=True)
            ev_in[st].record(up)
        stream.wait_event(ev_in[st])
        if ev_back[st] is not None:
            stream.wait_event(ev_back[st])           # step f-2's copy of dout[st] is done
        for s in range(B):
            append_one(f, s, 0, dkv[s][0][0], dkv[s][0][1], q=dq[0][s * T:(s + 1) * T],
                       pos=dpos[st] if args.rope else None)
        for s in range(B):
            cache.evict_frames(s)
        cache.plan(ws, stream)
        ev_planned.record(stream)
        planned[0] = True
        for b in range(L):
            if b:
                for s in range(B):
                    append_one(f, s, b, dkv[s][b][0], dkv[s][b][1], q=dq[b][s * T:(s + 1) * T],
                               pos=dpos[st] if args.rope else None)
            cache.run_attention(b, qrot[b] if args.rope else dq[b], dout[st][b], ws, stream)
        ev_out[st].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_out[st])
            hout.copy_(dout[st], non_blocking=True)
            ev_back[st] = torch.cuda.Event()
            ev_back[st].record(down)

    for _ in range(2):
        e2e_step(f)
        f += 1
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    for _ in range(K):
        e2e_step(f)
        f += 1
    for st in range(2):
        stream.wait_event(ev_back[st])             # every output is back on the host
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_elapsed = reduce_max(e0.elapsed_time(e1) / 1000.0, device=dev)
    # untimed check: the last e2e step's outputs, as copied back to the host, equal the
    # same frame's attention from the device-resident q (same plan, same kernels, so bit
    # for bit); with --rope q is produced by the appends themselves, so there is no
    # device-resident q to rerun from
    e2e_match = None
    if not args.rope:
        vi_last = (f - 1) % NV
        chk = torch.empty_like(outs[0])
        bits = torch.int16 if chk.element_size() == 2 else torch.int32
        e2e_match = True
        for b in range(L):
            cache.run_attention(b, qcat[vi_last][b], chk, ws, stream)
            torch.cuda.synchronize()
            e2e_match = e2e_match and bool(torch.equal(chk.cpu().view(bits), hout[b].view(bits)))

    # ------------------------------------------------ report
    hbm, tflops, tflops_sus, peak_kind = load_peaks()
    frames_launched = list(range(f_first + K + 1, f_first + 2 * K + 1))  # the frames of the per-launch pass
    flops = statistics.mean(block_work(w, x)[0] for x in frames_launched)
    byts = statistics.mean(block_work(w, x)[1] for x in frames_launched)
    avg_launch = statistics.mean(launch_ms) / 1000.0
    compute_peak, compute_bound, compute_src = tflops, "tensor", "bf16_tflops"
    if w.dtype == "f32":  # the fp32 path runs on the CUDA cores' FMA units
        compute_peak, compute_bound, compute_src = fp32_alu_peak_tflops(), "alu", "fp32 FMA: 152 SMs x 128 lanes x 2 x max SM clock"
    t_roof_block = max(flops / (compute_peak * 1e12), byts / (hbm * 1e9))
    bound = "hbm" if byts / (hbm * 1e9) >= flops / (compute_peak * 1e12) else compute_bound
    if bound == "hbm":
        achieved, peak, unit = byts / avg_launch / 1e9, hbm, "GB/s"
    else:
        achieved, peak, unit = flops / avg_launch / 1e12, compute_peak, "TFLOP/s"
    value = aggregate_throughput(K, world, max_elapsed)
    step_ms = max_elapsed / K * 1000.0
    launches_per_step = B * L + L + (L if info["merge_needed"] else 0)
    eb = wl.element_bytes(w)
    # K and V in and out; with the rotary embedding q in and q out as well
    append_bytes = (6 if args.rope else 4) * T * w.num_heads * w.head_dim * eb
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {**workload_config(w, f_first + K), "timed_frames": [f_first + 1, f_first + K],
                   **({"rope": {"sections": list(sections), "theta": theta}} if args.rope else {}),
                   "l2": "no flush: visible K/V per block exceeds L2",
                   "parallelism": f"replicas x{world} (independent streams, no data-path collective)"},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": recorded_traffic(w.name),
                     "kernel": ("attention (fp32 CUDA-core paged attention + LSE merge), per block launch"
                                if w.dtype == "f32" else
                                "attention (tcgen05 paged attention + LSE merge), per block launch"),
                     "peak_source": (f"{peak_kind} (hbm_gbs)" if bound == "hbm" else
                                     "derived (" + compute_src + ")" if bound == "alu" else
                                     f"{peak_kind} (bf16_tflops)"),
                     "avg_launch_us": avg_launch * 1e6, "algorithmic_bytes_per_launch": byts,
                     "algorithmic_flops_per_launch": flops,
                     "tensor_tflops": flops / avg_launch / 1e12, "hbm_gbs": byts / avg_launch / 1e9,
                     **({"frac_of_sustained": achieved / tflops_sus} if bound == "tensor" else {})},
        "attention_roofline_frac": t_roof_block * L / (max_elapsed / K),
        "roofline_frame_steps_per_s": 1.0 / (t_roof_block * L),
        "e2e": {"value": aggregate_throughput(K, world, e2e_elapsed), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "frames": [f - K + 1, f], "outputs_match_device_path": e2e_match},
        "append": {"kernel": "append_rope_kernel" if args.rope else "append_kernel",
                   "avg_launch_us": statistics.mean(append_ms) * 1e3,
                   "bytes_per_launch": append_bytes,
                   "gbs": append_bytes / (statistics.mean(append_ms) * 1e-3) / 1e9,
                   "note": "blocks 1..L-1 of two frames after the timed region, events around each launch "
                           "(launch overhead included)"},
        "gpu_launches": launches_per_step * K,
        "plan": info,
        "clocks": clk,
        "device_status": status,
        "fast_forward_s": t_ff,
    }
    cache.close()
    return line if rank == 0 else None


def add_cpu_baseline(line: dict, w: wl.Workload) -> None:
    """The fp64 oracle timed on the host cores on a bounded sample of the same workload
    (run after every GPU timing of the process, so that its host threads cannot slow a
    launching thread)."""
    reps = 50
    frame = line["config"]["timed_frames"][1]
    times, cpu_value = oracle_block_sample(w.replace(frames=frame + reps + 4), frame, heads=2, reps=reps,
                                           budget_s=20.0)
    line["cpu_baseline"] = {
        "value": cpu_value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
        "sample": (f"{len(times)} reps of one frame of bookkeeping + gather + fp64 attention of block 0 over 2 "
                   f"of {w.num_heads} heads at frame {frame}; extrapolated to all heads and "
                   f"{w.num_blocks} blocks")}


# (workload, variant, steps): the other streaming workloads, then the fp32 accuracy
# path, the fused rotary append and the scale-phase prefill
SECONDARY = (("lingbot_like_200", "", 20), ("high_res_999", "", 20), ("batched4_d128", "", 20),
             ("lingbot_like_200", "f32", 5), ("steady_state_10k", "rope", 20),
             ("steady_state_10k", "prefill8", 20))


def run_secondary(args) -> list:
    """The other workloads and paths, timed briefly in the same run after the headline
    line (device-resident and, for the streaming steps, end to end), so that one default
    run records every workload's throughput and roofline fraction.  A workload that
    fails is reported with its error instead."""
    import torch
    out = []
    for name, variant, steps in SECONDARY:
        sub = argparse.Namespace(**vars(args))
        sub.workload, sub.steps, sub.warmup, sub.no_cpu_baseline = name, steps, 5 if steps >= 20 else 3, True
        sub.f32, sub.rope, sub.query_frames = variant == "f32", variant == "rope", 8 if variant == "prefill8" else 1
        w = wl.CONFIGS[name]
        if sub.f32:
            w = w.replace(dtype="f32", name=f"{w.name}_f32")
        torch.cuda.empty_cache()
        try:
            d = run_prefill(sub, w) if sub.query_frames > 1 else run_gpu(sub, w)
        except Exception as e:  # noqa: BLE001 - the headline line must still print
            out.append({"workload": name, "variant": variant, "error": f"{type(e).__name__}: {e}"})
            continue
        r = d["roofline"]
        entry = {
            "workload": name, "variant": variant, "metric": d["metric"], "value": d["value"], "unit": d["unit"],
            "ms_per_step": d["ms_per_step"], "steps": d["steps"], "warmup": d["warmup"], "dtype": d["dtype"],
            "roofline": {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac", "avg_launch_us",
                                           "frac_of_sustained") if k in r},
            "gpu_launches": d["gpu_launches"], "clocks": d["clocks"], "device_status": d["device_status"]}
        if "e2e" in d:
            entry["e2e"] = {"value": d["e2e"]["value"],
                            "outputs_match_device_path": d["e2e"]["outputs_match_device_path"]}
        out.append(entry)
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------- scale-phase prefill

def run_prefill(args, w: wl.Workload):
    """Scale phase ("Frame Processing Loop", num_frames > 1): a new stream's first F
    frames are appended (all blocks) and then attend all of their F*T query rows over
    the F frames at once, every block.  A step is one such prefill of one stream set,
    on a cache reset before it; the inputs are resident in HBM."""
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist_init("nccl")
    import streaming_paged_kv_two_gb300 as spk
    from workload_device import spk_config_for, to_device

    F, K, W = args.query_frames, args.steps, args.warmup
    wk = w.replace(frames=F)
    cfg, keep = spk_config_for(wk, args.splits, max_query_frames=F)
    pool_bytes, ws_bytes = spk.required_bytes(cfg)
    dev = torch.device("cuda", local)
    pools = [torch.empty(pool_bytes, dtype=torch.uint8, device=dev) for _ in range(w.num_blocks)]
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    cache = spk.Cache(cfg, pools, keep)
    stream = torch.cuda.current_stream()
    B, L, T = w.num_streams, w.num_blocks, w.tokens_per_frame
    kvs = [[[tuple(to_device(x, w.dtype) for x in wl.frame_kv(w, s, b, f)) for b in range(L)] for s in range(B)]
           for f in range(F)]
    qcat = [torch.cat([to_device(wl.frame_q(w, s, b, f), w.dtype) for s in range(B) for f in range(F)])
            for b in range(L)]
    outs = [torch.empty_like(qcat[b]) for b in range(L)]
    ev_pairs = []

    def prefill(timed_launches=False):
        cache.reset()
        for f in range(F):
            for s in range(B):
                k, v = kvs[f][s][0]
                cache.append_frame(s, 0, k, v, stream)
                cache.evict_frames(s)
            for b in range(1, L):
                for s in range(B):
                    k, v = kvs[f][s][b]
                    cache.append_frame(s, b, k, v, stream)
        cache.plan_queries(F, ws, stream)
        for b in range(L):
            if timed_launches:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                cache.run_attention(b, qcat[b], outs[b], ws, stream)
                e1.record(stream)
                ev_pairs.append((e0, e1))
            else:
                cache.run_attention(b, qcat[b], outs[b], ws, stream)

    for _ in range(W):
        prefill()
    info = cache.get_plan_info()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(K):
        prefill(timed_launches=True)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    elapsed = reduce_max(t0.elapsed_time(t1) / 1000.0, device=dev)
    status = spk.read_device_status(ws, stream)
    hbm, tflops, tflops_sus, peak_kind = load_peaks()
    n_vis = visible_tokens(w, F)
    Tq = F * T
    flops = 4.0 * Tq * n_vis * w.num_heads * w.head_dim * B
    byts = (2.0 * n_vis + 2.0 * Tq) * w.num_heads * w.head_dim * wl.element_bytes(w) * B
    avg_launch = statistics.mean(a.elapsed_time(b) for a, b in ev_pairs) / 1000.0
    achieved = flops / avg_launch / 1e12
    line = {
        "metric": f"scale-phase prefills/s ({F} frames, all blocks, 1 GB300)", "value": K * world / elapsed,
        "unit": "prefills/s", "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": elapsed / K * 1000.0,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**workload_config(w, F), "workload": f"scale_phase_prefill_{F}x{T}", "query_rows": Tq,
                   "l2": "no flush: each step rewrites the pools and reads them once"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                     "frac": achieved / tflops, "traffic": None,
                     "kernel": "attention (tcgen05 paged attention), per block launch",
                     "peak_source": f"{peak_kind} (bf16_tflops)", "avg_launch_us": avg_launch * 1e6,
                     "algorithmic_flops_per_launch": flops, "algorithmic_bytes_per_launch": byts,
                     "frac_of_sustained": achieved / tflops_sus},
        "gpu_launches": (F * B * L + L * (2 if info["merge_needed"] else 1)) * K,
        "plan": info, "clocks": clk, "device_status": status,
    }
    cache.close()
    return line if rank == 0 else None


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="steady_state_10k", choices=sorted(wl.CONFIGS))
    ap.add_argument("--impl", default="spk", choices=["spk", "reference"])
    ap.add_argument("--ref-heads", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the brief runs of the other workloads that the plain default run appends")
    ap.add_argument("--rope", action="store_true",
                    help="streaming step: append through the fused 3-D rotary scatter (q and k turned)")
    ap.add_argument("--splits", type=int, default=0,
                    help="tuning only: force this many KV splits per stream (0 = the planner's choice)")
    ap.add_argument("--blocks", type=int, default=0,
                    help="profiling only: override the block count (smaller device footprint)")
    ap.add_argument("--f32", action="store_true",
                    help="the workload stored in fp32 and attended by the fp32 accuracy path")
    ap.add_argument("--query-frames", type=int, default=1,
                    help="F > 1: time the scale-phase prefill (F frames appended, then F*T query rows "
                         "attend over them) instead of the streaming step")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "spk":
        args.warmup = 3
    w = wl.CONFIGS[args.workload]
    if args.f32:
        w = w.replace(dtype="f32", name=f"{w.name}_f32")
    if args.blocks:
        w = w.replace(num_blocks=args.blocks, name=f"{w.name}_blocks{args.blocks}")
    if args.impl == "reference":
        return run_reference(args, w)
    if args.query_frames > 1:
        line = run_prefill(args, w)
        if line is not None:
            print(json.dumps(line))
        return 0
    line = run_gpu(args, w)
    if line is not None:
        plain_default = (args.workload == "steady_state_10k" and not (args.rope or args.f32 or args.blocks or args.splits)
                         and line["n_gpus"] == 1)
        if plain_default and not args.no_secondary:
            line["secondary"] = run_secondary(args)
        if line["n_gpus"] == 1 and not args.no_cpu_baseline:
            add_cpu_baseline(line, w)
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
