"""Benchmark of the selective-scan hot path on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--no-decode]

A step is one ssm_scan_fwd_ex over the Mamba-2.8B-shaped layer workload (batch 4,
d_inner 5120, L 4096, N 16, bf16 u/Δ/z/y, fp32 A/B/C/D/bias, seed 2), the largest
single-launch workload, with inputs resident in HBM.  Two copies of the inputs
alternate between steps, so a step never reads data the previous step left in L2
(each copy, 675 MB, is larger than the 126 MB L2).  The same line reports:

* the million-length sequence (batch 1, d_inner 1536, L 2^20, N 16) as 16 launches
  of 65 536 steps with the fp32 state carried from launch to launch, the whole
  loop timed;
* the Mamba-130M-shaped layer (batch 8, d_inner 1536, L 2048, N 16);
* the one-token decode step (batch 256, d_inner 5120, N 16; four such groups
  advanced round-robin so that the 336 MB of state exceeds L2), launched step by
  step and as the 1000 steps captured in one CUDA graph and replayed;
* the backward, the conv1d front end and Mamba-2 SSD;
* end-to-end figures through the C ABI with host buffers, the oracle's CPU
  throughput, the roofline of the scan kernel and the SM clocks sampled during
  the timed region.

Under torchrun (N > 1) every rank runs its own copy of the workload (the scan
shards by batch and channel with no exchange: weak scaling); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "scan HBM GB/s (% of B300 peak) & channel-steps/s; decode tokens/s"
L2_BYTES = 126 * 1024 * 1024
WS_HEADER = 256   # bytes of a scan workspace before its carry records (the status word)


def scan_bytes(w) -> int:
    """Algorithmic HBM bytes of one scan: u, Δ, z read and y written once (io dtype),
    B and C read once, A/D/bias read, final state written."""
    e = 4 if w.io == "f32" else 2
    chsteps = w.batch * w.dim * w.seqlen
    return (4 * e * chsteps + 2 * 4 * w.batch * w.dstate * w.seqlen
            + 4 * (w.dim * w.dstate + 2 * w.dim) + 4 * w.batch * w.dim * w.dstate)


def decode_bytes(batch, dim, N, e=2) -> int:
    """Algorithmic HBM bytes of one decode step: state read + written, u/Δ/z read,
    y written, B/C read, A/D/bias read."""
    return (2 * 4 * batch * dim * N + 4 * e * batch * dim + 2 * 4 * batch * N
            + 4 * (dim * N + 2 * dim))


def fp32_ops_per_channel_step(N: int) -> int:
    """FP32 operations the method needs per channel step, counted per state n:
    Δ·A, B·u, scaling by 1/A, the state update (add + fma) and the C·h readout."""
    return 6 * N


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk.get("sm_max_mhz", 2032.0)), "measured"
    except Exception:
        return 6400.0, 2032.0, "fallback"


def csrc_hash(names=None) -> str:
    """Hash of the library sources `names` (file names under csrc/; all when None)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "selective_state_space_128_b300", "csrc")
    for name in sorted(names or os.listdir(d)):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None when
    the summary is missing or was taken on different sources of that kernel (the
    entry lists the files the kernel is compiled from)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        ent = rec[kernel]
        if ent.get("csrc_hash") != csrc_hash(ent.get("sources")):
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def start(self):
        try:
            cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                   "-lms", "50"]
            if self.uuid:
                cmd += ["-i", self.uuid]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0=None, t1=None):
        """Summary of the samples read between host times t0 and t1 (all if None)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if t0 is not None and not (t0 <= ts <= t1 + 0.06):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (torchrun: one process per GPU)
# ---------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    """The largest of every rank's value (the slowest rank's time bounds the job)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(per_rank_units: float, max_seconds: float, world: int) -> float:
    """Weak scaling: every rank processes its own full workload, so the job's
    throughput is all ranks' units over the slowest rank's time."""
    return per_rank_units * world / max_seconds


# ---------------------------------------------------------------------------
# scan: device-resident throughput and end to end
# ---------------------------------------------------------------------------

def pinned(a):
    import torch
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    return t.pin_memory()


def to_dev(t_host, io_bf16=False):
    import torch
    d = t_host.to("cuda", non_blocking=True)
    return d.view(torch.bfloat16) if io_bf16 else d


def bench_scan(w, steps, warmup, world, e2e=True, clocks=True):
    """Per-launch time of ssm_scan_fwd_ex on workload `w` (two input copies alternated),
    and, with `e2e`, of ssm_scan_fwd_host on page-locked host copies of the same inputs."""
    import torch
    import selective_state_space_128_b300 as ssm
    x = synth.make_scan_inputs(w)
    bf = w.io == "bf16"
    host = {k: pinned(v) for k, v in x.items()}
    sets = []
    for _ in range(2):
        g = {k: to_dev(host[k], bf and k in ("u", "delta", "z")) for k in host}
        g["y"] = torch.empty_like(g["u"])
        g["h"] = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device="cuda")
        nb = ssm.ssm_scan_workspace_bytes(w.batch, w.dim, w.seqlen, w.dstate,
                                          ssm.SSM_BF16 if bf else ssm.SSM_F32)
        g["ws"] = torch.empty(nb, dtype=torch.uint8, device="cuda") if nb else None
        sets.append(g)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step(g):
        ssm.ssm_scan_fwd_ex(g["u"], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"], g["D"],
                            g["z"], True, g["y"], g["h"], None, g["ws"], stream=stream)

    for i in range(warmup):
        step(sets[i % 2])
    torch.cuda.synchronize()
    sampler = None
    if clocks:
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
            uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        sampler = ClockSampler(uuid)
        sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    e0.record(stream)
    for i in range(steps):
        step(sets[i % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    ck = sampler.stop(t0, t1) if sampler else None
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(world, ms)
    # a workspace larger than the status header means the plan splits the sequence
    # (two kernels per call)
    split = sets[0]["ws"] is not None and sets[0]["ws"].numel() > WS_HEADER
    out = dict(ms=ms, clocks=ck, inputs=sets[0], launches_per_step=2 if split else 1)
    if not e2e:
        return out

    # end to end through the C ABI with host buffers: ssm_scan_fwd_host copies the
    # step's inputs from page-locked host memory, scans and copies y and the final
    # state back, pipelined over units inside the call, every step
    e2e_steps = max(3, min(steps, 10))
    hin = {k: (host[k].view(torch.bfloat16) if (bf and k in ("u", "delta", "z")) else host[k])
           for k in host}
    yh = torch.empty(sets[0]["y"].shape, dtype=sets[0]["y"].dtype).pin_memory()
    hh = torch.empty(sets[0]["h"].shape, dtype=torch.float32).pin_memory()
    h2d = sum(host[k].numel() * host[k].element_size() for k in host)
    d2h = yh.numel() * yh.element_size() + hh.numel() * hh.element_size()
    flags = ssm.SSM_SOFTPLUS
    ws_bytes = ssm.ssm_scan_fwd_host_workspace_bytes(w.batch, w.dim, w.seqlen, w.dstate,
                                                     ssm.SSM_BF16 if bf else ssm.SSM_F32, flags)
    hws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")

    def e2e_step():
        ssm.ssm_scan_fwd_host(hin["u"], hin["delta"], hin["delta_bias"], hin["A"], hin["B"],
                              hin["C"], hin["D"], hin["z"], flags, yh, hh, None, hws, ws_bytes,
                              stream=stream)

    e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, f0.elapsed_time(f1))
    out.update(e2e_ms=e2e_ms, e2e_steps=e2e_steps, h2d=h2d, d2h=d2h)
    return out


# ---------------------------------------------------------------------------
# the million-length sequence: 16 launches with the fp32 state carried
# ---------------------------------------------------------------------------

def bench_million(w, reps, world, cpu=True, launches=None):
    """The million-length workload as w.launches launches of L / launches steps, each
    starting from the previous launch's fp32 final state; the whole loop is timed.

    Inputs are drawn on the device (seeded torch generator, the workload's
    distributions: u, z ~ N(0, 1), Δ_raw ~ N(0, 0.5^2), B, C ~ N(0, 1); A, D and the
    bias from the workload's generator): 16 chunks of u/Δ/z (3 x 201 MB each) and y,
    13 GB in all, far larger than L2.  End to end: the same loop through
    ssm_scan_fwd_host from page-locked host copies of every chunk.  CPU: the oracle on
    a sample of channels of the same inputs, over the whole length."""
    import torch
    import selective_state_space_128_b300 as ssm
    Lc = w.seqlen // w.launches
    K = w.launches if launches is None else max(1, min(w.launches, launches))
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1000 + w.seed)
    bf = torch.bfloat16
    shape = (w.batch, w.dim, Lc)
    chunks = []
    for _ in range(K):
        c = dict(u=torch.randn(shape, generator=gen, device="cuda").to(bf),
                 delta=(w.sigma_delta * torch.randn(shape, generator=gen, device="cuda")).to(bf),
                 z=torch.randn(shape, generator=gen, device="cuda").to(bf),
                 B=torch.randn((w.batch, w.dstate, Lc), generator=gen, device="cuda"),
                 C=torch.randn((w.batch, w.dstate, Lc), generator=gen, device="cuda"))
        c["y"] = torch.empty_like(c["u"])
        chunks.append(c)
    A = torch.from_numpy(synth.gen_A(w.dim, w.dstate)).cuda()
    D = torch.from_numpy(synth.gen_D(w)).cuda()
    bias = torch.from_numpy(synth.gen_delta_bias(w.seed, w.dim)).cuda()
    hs = [torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device="cuda")
          for _ in range(2)]
    nb = ssm.ssm_scan_workspace_bytes(w.batch, w.dim, Lc, w.dstate, ssm.SSM_BF16)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def loop():
        for k, c in enumerate(chunks):
            ssm.ssm_scan_fwd_ex(c["u"], c["delta"], bias, A, c["B"], c["C"], D, c["z"], True,
                                c["y"], hs[k % 2], None if k == 0 else hs[(k - 1) % 2], ws, nb,
                                stream=stream)

    loop()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        loop()
    e1.record(stream)
    torch.cuda.synchronize()
    loop_ms = max_over_ranks(world, e0.elapsed_time(e1)) / reps
    plan_split = nb > WS_HEADER
    out = dict(loop_ms=loop_ms, reps=reps, launches=K, chunk_len=Lc,
               kernels_per_launch=2 if plan_split else 1, workspace_bytes=nb)

    # end to end: page-locked host copies of every chunk, the same loop through
    # ssm_scan_fwd_host (copies in and out inside each call)
    hc = []
    for c in chunks:
        hc.append({k: c[k].cpu().pin_memory() for k in ("u", "delta", "z", "B", "C")})
    yh = torch.empty(shape, dtype=bf).pin_memory()
    hh = [torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32).pin_memory()
          for _ in range(2)]
    hA, hD, hb = A.cpu().pin_memory(), D.cpu().pin_memory(), bias.cpu().pin_memory()
    flags = ssm.SSM_SOFTPLUS
    hws_bytes = ssm.ssm_scan_fwd_host_workspace_bytes(w.batch, w.dim, Lc, w.dstate, ssm.SSM_BF16,
                                                      flags)
    hws = torch.empty(hws_bytes, dtype=torch.uint8, device="cuda")

    def e2e_loop():
        for k, c in enumerate(hc):
            ssm.ssm_scan_fwd_host(c["u"], c["delta"], hb, hA, c["B"], c["C"], hD, c["z"], flags,
                                  yh, hh[k % 2], None if k == 0 else hh[(k - 1) % 2], hws,
                                  hws_bytes, stream=stream)

    e2e_loop()
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    e2e_loop()
    e1.record(stream)
    torch.cuda.synchronize()
    out["e2e_ms"] = max_over_ranks(world, e0.elapsed_time(e1))
    out["h2d"] = sum(t.numel() * t.element_size() for c in hc for t in c.values())
    out["d2h"] = K * (yh.numel() * yh.element_size() + hh[0].numel() * 4)
    del hc

    if cpu:
        # the oracle over the whole length for a sample of channels of batch row 0
        import oracle
        nch = 32
        rows = {k: torch.cat([c[k][0, :nch] for c in chunks], dim=1).view(torch.int16).cpu()
                .numpy().view(np.uint16) for k in ("u", "delta", "z")}
        Bh = torch.cat([c["B"] for c in chunks], dim=2).cpu().numpy()
        Ch = torch.cat([c["C"] for c in chunks], dim=2).cpu().numpy()
        t = time.perf_counter()
        oracle.scan_rows(rows["u"], rows["delta"], rows["z"], np.zeros(nch, np.int64),
                         np.arange(nch), A.cpu().numpy(), Bh, Ch, D.cpu().numpy(),
                         bias.cpu().numpy(), True, None, y_stride=1021)
        secs = time.perf_counter() - t
        cs = nch * w.seqlen
        cores = min(oracle.max_threads(), nch)
        per_cs_bytes = scan_bytes(w) / w.channel_steps
        out["cpu"] = {"value": per_cs_bytes * cs / secs / 1e9, "unit": "GB/s", "cores": cores,
                      "kind": "oracle", "channel_steps_per_s": cs / secs,
                      "sample": "batch 0, channels 0..%d over the whole 2^20 steps (%d "
                                "channel-steps), %.1f s wall on %d threads; GB/s counts the "
                                "workload's algorithmic bytes per channel-step" % (
                                    nch - 1, cs, secs, cores)}
    return out


# ---------------------------------------------------------------------------
# the same scan with u/delta/z/y in the (batch, L, dim) layout
# ---------------------------------------------------------------------------

def bench_scan_bld(w, g, steps, warmup, world):
    """Per-launch time of the scan on the transposed (batch, L, dim) copies of the
    workload's inputs (one copy: 204 MB, larger than L2)."""
    import torch
    import selective_state_space_128_b300 as ssm
    t = {k: g[k].transpose(1, 2).contiguous() for k in ("u", "delta", "z")}
    y = torch.empty_like(t["u"])
    h = torch.empty((w.batch, w.dim, w.dstate), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    flags = ssm.SSM_SOFTPLUS | ssm.SSM_LAYOUT_BLD

    def step():
        ssm.ssm_scan_fwd_ex(t["u"], t["delta"], g["delta_bias"], g["A"], g["B"], g["C"], g["D"],
                            t["z"], flags, y, h, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    return max_over_ranks(world, e0.elapsed_time(e1)) / steps


# ---------------------------------------------------------------------------
# front end: causal conv1d (d_conv 4) + SiLU over the same layer's input
# ---------------------------------------------------------------------------

def bench_conv(w, steps, warmup, world, width=4, copies=3):
    """Per-launch time of ssm_conv1d_fwd on (batch, d_inner, L) bf16 input with a
    (d_inner, 4) kernel; `copies` input/output pairs (100 MB each) are rotated so
    the working set (300 MB) is larger than L2.  Seeded inputs drawn on the device."""
    import torch
    import selective_state_space_128_b300 as ssm
    gen = torch.Generator(device="cuda")
    gen.manual_seed(w.seed + 2000)
    shape = (w.batch, w.dim, w.seqlen)
    xs = [torch.randn(shape, generator=gen, device="cuda").to(torch.bfloat16) for _ in range(copies)]
    outs = [torch.empty_like(xs[0]) for _ in range(copies)]
    wt = 0.5 * torch.randn((w.dim, width), generator=gen, device="cuda")
    bias = 0.2 * torch.randn(w.dim, generator=gen, device="cuda")
    stream = torch.cuda.current_stream()
    for i in range(warmup):
        ssm.ssm_conv1d_fwd(xs[i % copies], wt, bias, None, True, outs[i % copies], None, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        ssm.ssm_conv1d_fwd(xs[i % copies], wt, bias, None, True, outs[i % copies], None, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(world, e0.elapsed_time(e1)) / steps
    nbytes = 2 * xs[0].numel() * 2 + wt.numel() * 4 + bias.numel() * 4
    # the backward on the same shapes: x and dout read, dx written (the outs
    # buffers serve as the cotangents, dxs rotate like the inputs)
    dxs = [torch.empty_like(xs[0]) for _ in range(copies)]
    dw = torch.empty_like(wt)
    db = torch.empty_like(bias)

    def bwd(i):
        ssm.ssm_conv1d_bwd(xs[i % copies], wt, bias, None, 1, outs[(i + 1) % copies], dxs[i % copies],
                           dw, db, None, stream)

    for i in range(warmup):
        bwd(i)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        bwd(i)
    e1.record(stream)
    torch.cuda.synchronize()
    bms = max_over_ranks(world, e0.elapsed_time(e1)) / steps
    bbytes = 3 * xs[0].numel() * 2 + 2 * (wt.numel() + bias.numel()) * 4
    return dict(step_ms=ms, steps=steps, bytes=nbytes, bwd_ms=bms, bwd_bytes=bbytes)


# ---------------------------------------------------------------------------
# Mamba-2 SSD (scalar-A SSM, chunked on the tensor cores): a Mamba-2-130M-shaped
# layer, batch 8, L 2048, 24 heads of 64, one group, N 128, bf16
# ---------------------------------------------------------------------------

SSD_SHAPE = dict(batch=8, L=2048, H=24, P=64, G=1, N=128)


def ssd_flops(batch, L, H, P, G, N, Q=64):
    """Tensor-core FLOPs the chunked algorithm needs per launch: the causal half of
    C Bᵀ and of (mask ∘ C Bᵀ) X inside each chunk, C Hᵀ and the chunk state."""
    nch = (L + Q - 1) // Q
    tri = Q * (Q + 1) // 2
    per = 2 * (tri * N + tri * P + Q * N * P + Q * P * N)
    return per * nch * H * batch


def ssd_bytes(batch, L, H, P, G, N):
    """Algorithmic HBM bytes: x, z, dt read, y written (bf16), B and C read (bf16),
    A, D, dt bias, and the final state written (fp32)."""
    return (3 * batch * L * H * P * 2 + batch * L * H * 2 + 2 * batch * L * G * N * 2 + 3 * H * 4
            + batch * H * P * N * 4)


def bench_ssd(steps, warmup, world, seed=5):
    import torch
    import selective_state_space_128_b300 as ssm
    sh = SSD_SHAPE
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    bf = torch.bfloat16
    b, L, H, P, G, N = sh["batch"], sh["L"], sh["H"], sh["P"], sh["G"], sh["N"]
    x = torch.randn((b, L, H, P), generator=gen, device="cuda").to(bf)
    z = torch.randn((b, L, H, P), generator=gen, device="cuda").to(bf)
    dt = (0.5 * torch.randn((b, L, H), generator=gen, device="cuda")).to(bf)
    B = torch.randn((b, L, G, N), generator=gen, device="cuda").to(bf)
    C = torch.randn((b, L, G, N), generator=gen, device="cuda").to(bf)
    A = -(1.0 + 7.0 * torch.rand(H, generator=gen, device="cuda"))
    D = 0.5 + torch.rand(H, generator=gen, device="cuda")
    bias = torch.from_numpy(synth.gen_delta_bias(seed, H)).cuda()
    y = torch.empty_like(x)
    h = torch.empty((b, H, P, N), dtype=torch.float32, device="cuda")
    nbytes = ssm.ssm_ssd_workspace_bytes(b, L, H, P, G, N)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        ssm.ssm_ssd_fwd(x, dt, bias, A, B, C, D, z, ssm.SSM_SOFTPLUS, y, h, None, ws, nbytes,
                        stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(world, e0.elapsed_time(e1)) / steps
    # the backward on the same layer (ssm_ssd_bwd, the chunked form), a few steps
    dy = torch.randn((b, L, H, P), generator=gen, device="cuda").to(bf)
    f32 = dict(dtype=torch.float32, device="cuda")
    dx, dz, ddt = torch.empty_like(x), torch.empty_like(z), torch.empty_like(dt)
    dA, dD, dbias = torch.empty(H, **f32), torch.empty(H, **f32), torch.empty(H, **f32)
    dB, dC = torch.empty(B.shape, **f32), torch.empty(C.shape, **f32)
    bwb = ssm.ssm_ssd_bwd_workspace_bytes(b, L, H, P, G, N)
    bws = torch.empty(bwb, dtype=torch.uint8, device="cuda")

    def bstep():
        ssm.ssm_ssd_bwd(x, dt, bias, A, B, C, D, z, ssm.SSM_SOFTPLUS, None, dy, None, dx, ddt, dA,
                        dB, dC, dD, dz, dbias, None, bws, bwb, stream)

    bsteps = 3
    bstep()
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    for _ in range(bsteps):
        bstep()
    e1.record(stream)
    torch.cuda.synchronize()
    bms = max_over_ranks(world, e0.elapsed_time(e1)) / bsteps
    del bws
    return dict(step_ms=ms, steps=steps, workspace_bytes=nbytes, bwd_ms=bms, bwd_steps=bsteps,
                bwd_workspace_bytes=bwb)


# ---------------------------------------------------------------------------
# backward pass on the same layer
# ---------------------------------------------------------------------------

def bench_backward(w, g, steps, warmup, world):
    """Per-step time of ssm_scan_bwd on the scan workload's device inputs `g`, with a
    seeded dy (N(0, 1), the I/O dtype) drawn on the device; outputs and workspace are
    allocated once.  u, delta, z and dy are 4 x 50 MB, larger than L2."""
    import torch
    import selective_state_space_128_b300 as ssm
    gen = torch.Generator(device="cuda")
    gen.manual_seed(w.seed + 1000)
    dy = torch.randn(g["u"].shape, generator=gen, device="cuda").to(g["u"].dtype)
    N = w.dstate
    f32 = dict(dtype=torch.float32, device="cuda")
    out = dict(du=torch.empty_like(g["u"]), ddelta=torch.empty_like(g["u"]),
               dz=torch.empty_like(g["u"]), dA=torch.empty((w.dim, N), **f32),
               dB=torch.empty((w.batch, N, w.seqlen), **f32),
               dC=torch.empty((w.batch, N, w.seqlen), **f32), dD=torch.empty(w.dim, **f32),
               dbias=torch.empty(w.dim, **f32))
    nbytes = ssm.ssm_scan_bwd_workspace_bytes(w.batch, w.dim, w.seqlen, N)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    y = torch.empty_like(g["u"])
    h = torch.empty((w.batch, w.dim, N), **f32)

    def step(flags=ssm.SSM_SOFTPLUS):
        ssm.ssm_scan_bwd(g["u"], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"], g["D"],
                         g["z"], flags, None, dy, None, out["du"], out["ddelta"], out["dA"],
                         out["dB"], out["dC"], out["dD"], out["dz"], out["dbias"], None, ws,
                         nbytes, stream=stream)

    def fwd_train():
        ssm.ssm_scan_fwd_train(g["u"], g["delta"], g["delta_bias"], g["A"], g["B"], g["C"],
                               g["D"], g["z"], True, y, h, None, None, 0, ws, nbytes, stream)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(world, e0.elapsed_time(e1)) / steps

    ms = timed(step)
    fwd_train()  # the workspace now holds the saved chunk-start states
    saved_ms = timed(lambda: step(ssm.SSM_SOFTPLUS | ssm.SSM_SAVED_STATES))
    train_ms = timed(lambda: (fwd_train(), step(ssm.SSM_SOFTPLUS | ssm.SSM_SAVED_STATES)))
    return dict(step_ms=ms, saved_ms=saved_ms, train_ms=train_ms, steps=steps,
                workspace_bytes=nbytes)


def bench_backward_million(w, reps, world):
    """ssm_scan_bwd over the million-length sequence in one call (batch 1, d_inner
    1536, L 2^20, N 16, bf16): 48 channel blocks of one batch row, so the library's
    plan splits the sequence into segments chained by their carries (the forward's
    first pass, the adjoint's carry pass, the per-block kernel, the fixed-order sums:
    4 launches a call).  Inputs drawn on the device with the workload's
    distributions (u, z, dy ~ N(0, 1), Δ_raw ~ N(0, 0.5^2), B, C ~ N(0, 1); A, D and
    the bias from the workload's generator): 4 x 3.2 GB in, 3 x 3.2 GB out."""
    import torch
    import selective_state_space_128_b300 as ssm
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2000 + w.seed)
    bf = torch.bfloat16
    shape = (w.batch, w.dim, w.seqlen)
    N = w.dstate
    f32 = dict(dtype=torch.float32, device="cuda")
    u = torch.randn(shape, generator=gen, device="cuda").to(bf)
    delta = (w.sigma_delta * torch.randn(shape, generator=gen, device="cuda")).to(bf)
    z = torch.randn(shape, generator=gen, device="cuda").to(bf)
    dy = torch.randn(shape, generator=gen, device="cuda").to(bf)
    B = torch.randn((w.batch, N, w.seqlen), generator=gen, **f32)
    C = torch.randn((w.batch, N, w.seqlen), generator=gen, **f32)
    A = torch.from_numpy(synth.gen_A(w.dim, N)).cuda()
    D = torch.from_numpy(synth.gen_D(w)).cuda()
    bias = torch.from_numpy(synth.gen_delta_bias(w.seed, w.dim)).cuda()
    du, ddelta, dz = torch.empty_like(u), torch.empty_like(u), torch.empty_like(u)
    dA, dD, dbias = torch.empty((w.dim, N), **f32), torch.empty(w.dim, **f32), torch.empty(w.dim, **f32)
    dB, dC = torch.empty_like(B), torch.empty_like(C)
    nbytes = ssm.ssm_scan_bwd_workspace_bytes(w.batch, w.dim, w.seqlen, N)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        ssm.ssm_scan_bwd(u, delta, bias, A, B, C, D, z, ssm.SSM_SOFTPLUS, None, dy, None, du,
                         ddelta, dA, dB, dC, dD, dz, dbias, None, ws, nbytes, stream=stream)

    call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(world, e0.elapsed_time(e1)) / reps
    del u, delta, z, dy, du, ddelta, dz, ws
    return dict(ms=ms, reps=reps, workspace_bytes=nbytes)


# ---------------------------------------------------------------------------
# decode: batch 256, d_inner 5120, N 16, one token per step
# ---------------------------------------------------------------------------

def bench_decode(dw, steps, world, groups=4):
    """Per-step time of ssm_state_update_ex at batch 256 x d_inner 5120, N 16.

    `groups` independent decode groups (each a batch of 256 sequences with its own
    84 MB state) are advanced round-robin, one step per launch, so every launch reads
    a state that is not in the 126 MB L2 and the write-back of earlier states'
    updates happens inside the timed region (336 MB of state in total).  Inputs are
    drawn on the device (seeded torch generator, the workload's distributions); the
    states start from a GPU scan over a 256-step prefill.  The same steps are also
    captured once in a CUDA graph and replayed: the device time without a host call
    per step."""
    import torch
    import selective_state_space_128_b300 as ssm
    gen = torch.Generator(device="cuda")
    gen.manual_seed(dw.seed)
    B_, D_, N = dw.batch, dw.dim, dw.dstate
    A = torch.from_numpy(synth.gen_A(D_, N)).cuda()
    Dp = torch.from_numpy(synth.fill(dw.seed, synth.S_D, 0, D_, synth.UNIFORM, 0.5, 1.5)).cuda()
    bias = torch.from_numpy(synth.gen_delta_bias(dw.seed, D_)).cuda()
    Lp = dw.prefill_len
    bf = torch.bfloat16
    pu = torch.randn((B_, D_, Lp), generator=gen, device="cuda").to(bf)
    pd = (0.5 * torch.randn((B_, D_, Lp), generator=gen, device="cuda")).to(bf)
    pz = torch.randn((B_, D_, Lp), generator=gen, device="cuda").to(bf)
    pB = torch.randn((B_, N, Lp), generator=gen, device="cuda")
    pC = torch.randn((B_, N, Lp), generator=gen, device="cuda")
    _, state0 = ssm.scan(pu, pd, A, pB, pC, Dp, pz, bias)
    del pu, pd, pz, pB, pC
    states = [state0.clone() for _ in range(groups)]
    u = torch.randn((steps, B_, D_), generator=gen, device="cuda").to(bf)
    dl = (0.5 * torch.randn((steps, B_, D_), generator=gen, device="cuda")).to(bf)
    z = torch.randn((steps, B_, D_), generator=gen, device="cuda").to(bf)
    Bs = torch.randn((steps, B_, N), generator=gen, device="cuda")
    Cs = torch.randn((steps, B_, N), generator=gen, device="cuda")
    y = torch.empty((steps, B_, D_), dtype=bf, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i, st):
        ssm.ssm_state_update_ex(st, u[i], dl[i], bias, True, A, Bs[i], Cs[i], Dp, z[i], y[i],
                                stream=stream)

    for i in range(2 * groups):
        step(i, states[i % groups])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        step(i, states[i % groups])
    e1.record(stream)
    torch.cuda.synchronize()
    step_ms = max_over_ranks(world, e0.elapsed_time(e1)) / steps
    # one group only, back to back: its state stays largely in L2 (context only)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for i in range(steps):
        step(i, states[0])
    g1.record(stream)
    torch.cuda.synchronize()
    l2_ms = max_over_ranks(world, g0.elapsed_time(g1)) / steps
    # the same round-robin steps captured once as a CUDA graph and replayed `replays`
    # times: the device time of the steps without a host call per step
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cs = torch.cuda.current_stream()
        for i in range(steps):
            ssm.ssm_state_update_ex(states[i % groups], u[i], dl[i], bias, True, A, Bs[i], Cs[i],
                                    Dp, z[i], y[i], stream=cs)
    graph.replay()
    torch.cuda.synchronize()
    replays = 5
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    r0.record(stream)
    for _ in range(replays):
        graph.replay()
    r1.record(stream)
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(world, r0.elapsed_time(r1)) / (replays * steps)
    del graph
    return dict(step_ms=step_ms, l2_resident_ms=l2_ms, steps=steps, groups=groups,
                graph_step_ms=graph_ms, graph_replays=replays)


# ---------------------------------------------------------------------------
# the oracle as CPU baseline / reference arm
# ---------------------------------------------------------------------------

def oracle_sample(w, channels, nthreads=0):
    """Run the fp64 oracle on batch 0, channels [0, channels) of workload w; returns
    (seconds, sample workload)."""
    import oracle
    sw = synth.scaled(w, batch=1, dim=channels)
    u = synth.gen_rows(w, "u", 0, 0, channels)
    dl = synth.gen_rows(w, "delta", 0, 0, channels)
    z = synth.gen_rows(w, "z", 0, 0, channels)
    B = synth.gen_bc(synth.scaled(w, batch=1), "B")
    C = synth.gen_bc(synth.scaled(w, batch=1), "C")
    A = synth.gen_A(w.dim, w.dstate)
    D = synth.gen_D(w)
    bias = synth.gen_delta_bias(w.seed, w.dim)
    t = time.perf_counter()
    oracle.scan_rows(u, dl, z, np.zeros(channels, np.int64), np.arange(channels), A, B, C, D, bias,
                     True, None, 1, nthreads)
    return time.perf_counter() - t, sw


def cpu_baseline(w):
    """The fp64 oracle on the whole workload (every batch row and channel, full length),
    all host threads; input generation is outside the timed region."""
    import oracle
    x = synth.make_scan_inputs(w)
    t = time.perf_counter()
    oracle.scan(x["u"], x["delta"], x["A"], x["B"], x["C"], x["D"], x["z"], x["delta_bias"])
    secs = time.perf_counter() - t
    cores = oracle.max_threads()
    return {"value": scan_bytes(w) / secs / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle", "channel_steps_per_s": w.channel_steps / secs,
            "sample": "the whole workload (%d channel-steps), %.1f s wall on %d threads "
                      "(%.0f core-s)" % (w.channel_steps, secs, cores, secs * cores)}


def run_reference(args, w):
    """The reference arm: the fp64 oracle as it stands, on the host cores."""
    import oracle
    secs, _ = oracle_sample(w, 32)
    per_ch = secs / 32
    budget = 90.0 / max(1, args.steps + args.warmup)
    ch = int(max(8, min(w.dim, budget / per_ch)))
    for _ in range(args.warmup):
        oracle_sample(w, ch)
    tot = 0.0
    sw = None
    for _ in range(args.steps):
        s, sw = oracle_sample(w, ch)
        tot += s
    ms = tot / args.steps * 1e3
    value = scan_bytes(sw) / (tot / args.steps) / 1e9
    cpu = {"value": value, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
           "sample": "each step: batch 0, channels 0..%d of the workload" % (ch - 1)}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w), "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "channel_steps_per_s": sw.channel_steps / (tot / args.steps)}
    print(json.dumps(line))


def workload_config(w):
    return {"workload": w.name, "batch": w.batch, "d_inner": w.dim, "seqlen": w.seqlen,
            "dstate": w.dstate, "io_dtype": w.io, "state_dtype": "f32", "seed": w.seed,
            "l2": "inputs larger than L2 (%.0f MB per copy > 126 MB), two copies alternated"
                  % (scan_bytes(w) / 1e6)}


def scan_roofline(w, ms_per_launch, hbm_peak, sm_max, peak_kind, traffic_key, kernel):
    """Roofline of one scan launch on workload w: the method's FP32 operations against
    the FP32 lanes (the bound) and its algorithmic bytes against the HBM copy peak."""
    step_s = ms_per_launch / 1e3
    nbytes = scan_bytes(w)
    ops = fp32_ops_per_channel_step(w.dstate) * w.channel_steps
    alu_peak = 148 * 128 * sm_max * 1e6 / 1e12          # FP32 lanes x max SM clock, TOP/s
    alu_ach = ops / step_s / 1e12
    gbs = nbytes / step_s / 1e9
    return {"bound": "alu", "achieved": alu_ach, "peak": alu_peak, "unit": "TOP/s",
            "frac": alu_ach / alu_peak, "traffic": profiled_traffic(traffic_key),
            "kernel": kernel, "ops_per_launch": ops,
            "peak_basis": "148 SMs x 128 FP32 lanes x %.0f MHz (max SM clock)" % sm_max,
            "hbm_achieved_gbs": gbs, "hbm_peak_gbs": hbm_peak, "hbm_peak_kind": peak_kind,
            "hbm_frac": gbs / hbm_peak, "algorithmic_bytes_per_launch": nbytes}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--bwd-steps", type=int, default=20)
    ap.add_argument("--no-bwd", action="store_true")
    ap.add_argument("--no-conv", action="store_true")
    ap.add_argument("--no-ssd", action="store_true")
    ap.add_argument("--no-million", action="store_true")
    ap.add_argument("--no-bwd-million", action="store_true")
    ap.add_argument("--million-reps", type=int, default=3)
    ap.add_argument("--million-launches", type=int, default=None,
                    help="time only the first K of the 16 launches (for profiling a smaller case)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = synth.MAMBA_2P8B          # the headline: the largest single-launch workload
    w1 = synth.MAMBA_130M
    wm = synth.MILLION
    world, rank, local = dist_setup()
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return
    import torch
    torch.cuda.set_device(local)
    import selective_state_space_128_b300 as ssm
    ssm.load()
    hbm_peak, sm_max, peak_kind = load_peaks()

    r = bench_scan(w, args.steps, args.warmup, world)
    r.pop("inputs")
    r1 = bench_scan(w1, max(20, min(args.steps, 200)), args.warmup, world, e2e=False,
                    clocks=False)
    bwd = None if args.no_bwd else bench_backward(w1, r1["inputs"], args.bwd_steps, args.warmup,
                                                  world)
    bld_ms = bench_scan_bld(w1, r1["inputs"], 50, args.warmup, world)
    r1.pop("inputs")
    torch.cuda.empty_cache()
    mil = None if args.no_million else bench_million(wm, max(1, args.million_reps), world,
                                                    cpu=(rank == 0 and world == 1
                                                         and not args.no_cpu),
                                                    launches=args.million_launches)
    torch.cuda.empty_cache()
    bmil = None if (args.no_bwd or args.no_bwd_million) else bench_backward_million(wm, 2, world)
    torch.cuda.empty_cache()
    conv = None if args.no_conv else bench_conv(w1, 50, args.warmup, world)
    ssd = None if args.no_ssd else bench_ssd(20, args.warmup, world)
    dec = None if args.no_decode else bench_decode(synth.DECODE, args.decode_steps, world)
    cpu = cpu_baseline(w) if (rank == 0 and world == 1 and not args.no_cpu) else None
    if rank != 0:
        return

    step_s = r["ms"] / 1e3 / args.steps
    nbytes = scan_bytes(w)
    gbs_rank = nbytes / step_s / 1e9
    value = job_throughput(nbytes / 1e9, step_s, world)   # GB/s over all ranks
    chsteps = job_throughput(w.channel_steps, step_s, world)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w),
        "channel_steps_per_s": chsteps,
        "hbm": {"achieved_gbs": gbs_rank, "peak_gbs": hbm_peak, "frac": gbs_rank / hbm_peak,
                "peak_kind": peak_kind, "frac_of_8000_nominal": gbs_rank / 8000.0,
                "bytes_per_step": nbytes},
        "roofline": scan_roofline(w, r["ms"] / args.steps, hbm_peak, sm_max, peak_kind,
                                  "scan_kernel@" + w.name,
                                  "scan_pair_kernel<0, 32> (blocks of two warps: 16 channels a block, 32-step chunks)"),
        "e2e": {"value": nbytes * r["e2e_steps"] / (r["e2e_ms"] / 1e3) / 1e9 * world,
                "unit": "GB/s", "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "steps": r["e2e_steps"],
                "call": "ssm_scan_fwd_host: page-locked host buffers, copies pipelined over "
                        "batch-row units inside the call",
                "note": "bounded by the host link (about 55 GB/s each way, the two directions "
                        "not overlapping on this box), so it cannot show kernel improvements "
                        "at this size"},
        "gpu_launches": args.steps * r["launches_per_step"],
        "clocks": r["clocks"],
    }
    n1 = max(20, min(args.steps, 200))
    s1 = r1["ms"] / 1e3 / n1
    line["mamba130m_layer"] = {
        "workload": w1.name, "config": workload_config(w1), "steps": n1,
        "us_per_step": s1 * 1e6, "channel_steps_per_s": w1.channel_steps / s1 * world,
        "hbm_gbs": scan_bytes(w1) / s1 / 1e9, "hbm_frac": scan_bytes(w1) / s1 / 1e9 / hbm_peak,
        "roofline": scan_roofline(w1, s1 * 1e3, hbm_peak, sm_max, peak_kind,
                                  "scan_kernel@" + w1.name,
                                  "scan_kernel<bf16,16,0> (the block kernel: 32 channels a block)"),
        "gpu_launches": n1 * r1["launches_per_step"]}
    if mil is not None:
        ls = mil["loop_ms"] / 1e3
        part = mil["launches"] / wm.launches   # 1 unless a prefix of the loop was timed
        mb = (scan_bytes(wm) + (wm.launches - 1) * 4 * wm.batch * wm.dim * wm.dstate) * part
        mo = {"workload": wm.name, "config": dict(workload_config(wm), launches=mil["launches"],
                                                   chunk_len=mil["chunk_len"],
                                                   l2="13 GB of chunk inputs and outputs, far "
                                                      "larger than L2"),
              "reps": mil["reps"], "ms_per_loop": mil["loop_ms"],
              "channel_steps_per_s": wm.channel_steps * part / ls * world,
              "hbm_gbs": mb / ls / 1e9, "hbm_frac": mb / ls / 1e9 / hbm_peak,
              "bytes_per_loop": mb,
              "kernels_per_launch": mil["kernels_per_launch"],
              "workspace_bytes": mil["workspace_bytes"],
              "gpu_launches": mil["reps"] * mil["launches"] * mil["kernels_per_launch"],
              "timing": "the whole 16-launch loop with the fp32 state carried, CUDA events, "
                        "mean of %d loops after one untimed loop" % mil["reps"],
              "e2e": {"value": mb / (mil["e2e_ms"] / 1e3) / 1e9 * world, "unit": "GB/s",
                      "h2d_bytes_per_loop": mil["h2d"], "d2h_bytes_per_loop": mil["d2h"],
                      "call": "ssm_scan_fwd_host per launch, state carried in host memory"}}
        ops = fp32_ops_per_channel_step(wm.dstate) * wm.channel_steps * part
        alu_peak = 148 * 128 * sm_max * 1e6 / 1e12
        mo["roofline"] = {"bound": "alu", "achieved": ops / ls / 1e12, "peak": alu_peak,
                          "unit": "TOP/s", "frac": ops / ls / 1e12 / alu_peak,
                          "hbm_frac": mb / ls / 1e9 / hbm_peak,
                          "note": "the split plan recomputes part of each segment in its "
                                  "first pass; the ops counted are the method's 6N per "
                                  "channel step"}
        if "cpu" in mil:
            mo["cpu_baseline"] = mil["cpu"]
        line["million_length"] = mo
    if bmil is not None:
        bs = bmil["ms"] / 1e3
        esz = 2
        # the method's bytes: u, Δ, z, dy read and du, dΔ, dz written; B, C read and
        # dB, dC written; A, D, bias and dA, dD, dbias
        bb = (7 * wm.channel_steps * esz + 4 * wm.batch * wm.dstate * wm.seqlen * 4
              + 2 * (wm.dim * wm.dstate + 2 * wm.dim) * 4)
        line["backward_million_length"] = {
            "workload": wm.name + " backward, one call over the whole length",
            "config": workload_config(wm), "reps": bmil["reps"], "ms_per_call": bmil["ms"],
            "channel_steps_per_s": wm.channel_steps / bs * world,
            "hbm_gbs_algorithmic": bb / bs / 1e9, "hbm_frac": bb / bs / 1e9 / hbm_peak,
            "bytes_per_call": bb, "workspace_bytes": bmil["workspace_bytes"],
            "gpu_launches": 4 * bmil["reps"],
            "call": "ssm_scan_bwd: the plan splits the sequence into segments (forward "
                    "carries, adjoint carries, per-block kernel, fixed-order sums)"}
    if dec is not None:
        db = decode_bytes(synth.DECODE.batch, synth.DECODE.dim, synth.DECODE.dstate)
        st = dec["step_ms"] / 1e3
        line["decode"] = {"workload": synth.DECODE.name, "steps": dec["steps"],
                          "us_per_step": dec["step_ms"] * 1e3,
                          "tokens_per_s": synth.DECODE.batch / st * world,
                          "hbm_gbs": db / st / 1e9, "hbm_frac": db / st / 1e9 / hbm_peak,
                          "bytes_per_step": db,
                          "l2": "%d groups of 256 sequences advanced round-robin: %.0f MB of "
                                "state, larger than L2" % (
                                    dec["groups"], dec["groups"] * 4.0 * synth.DECODE.batch *
                                    synth.DECODE.dim * synth.DECODE.dstate / 1e6),
                          "us_per_step_one_group_back_to_back": dec["l2_resident_ms"] * 1e3,
                          "graph": {"us_per_step": dec["graph_step_ms"] * 1e3,
                                    "tokens_per_s": synth.DECODE.batch /
                                                    (dec["graph_step_ms"] / 1e3) * world,
                                    "hbm_gbs": db / (dec["graph_step_ms"] / 1e3) / 1e9,
                                    "hbm_frac": db / (dec["graph_step_ms"] / 1e3) / 1e9 / hbm_peak,
                                    "replays": dec["graph_replays"],
                                    "call": "the same %d round-robin steps captured once in a "
                                            "CUDA graph (torch.cuda.CUDAGraph around "
                                            "ssm_state_update_ex), replayed %d times" % (
                                                dec["steps"], dec["graph_replays"]),
                                    "gpu_launches": dec["steps"] * dec["graph_replays"]},
                          "one_group_note": "one 84 MB state advanced back to back; the "
                                            "state's loads and stores carry evict-first "
                                            "hints, so it streams from HBM as well",
                          "gpu_launches": dec["steps"]}
    if bwd is not None:
        bs = bwd["step_ms"] / 1e3
        line["backward"] = {"workload": w1.name, "steps": bwd["steps"],
                            "us_per_step": bwd["step_ms"] * 1e3,
                            "channel_steps_per_s": w1.channel_steps / bs * world,
                            "time_vs_forward": bs / s1,
                            "us_per_step_from_saved_states": bwd["saved_ms"] * 1e3,
                            "train_step_us": bwd["train_ms"] * 1e3,
                            "train_step": "ssm_scan_fwd_train + ssm_scan_bwd(SSM_SAVED_STATES)",
                            "workspace_bytes": bwd["workspace_bytes"],
                            "gpu_launches": 2 * bwd["steps"],
                            "l2": "u, delta, z, dy: 4 x %.0f MB, larger than L2"
                                  % (w1.channel_steps * 2 / 1e6)}
    line["scan_bld_layout"] = {"workload": w1.name, "us_per_step": bld_ms * 1e3,
                               "channel_steps_per_s": w1.channel_steps / (bld_ms / 1e3) * world,
                               "layout": "u, delta, z, y as (batch, L, d_inner)", "steps": 50,
                               "gpu_launches": 50}
    if conv is not None:
        cs = conv["step_ms"] / 1e3
        line["conv1d"] = {"workload": "conv1d_silu d_conv 4 on %d x %d x %d bf16" % (
                              w1.batch, w1.dim, w1.seqlen),
                          "steps": conv["steps"], "us_per_step": conv["step_ms"] * 1e3,
                          "hbm_gbs": conv["bytes"] / cs / 1e9,
                          "hbm_frac": conv["bytes"] / cs / 1e9 / hbm_peak,
                          "bytes_per_step": conv["bytes"], "gpu_launches": conv["steps"],
                          "l2": "3 input/output pairs rotated: 300 MB, larger than L2",
                          "backward": {"us_per_step": conv["bwd_ms"] * 1e3,
                                       "hbm_gbs": conv["bwd_bytes"] / (conv["bwd_ms"] / 1e3) / 1e9,
                                       "hbm_frac": conv["bwd_bytes"] / (conv["bwd_ms"] / 1e3)
                                                   / 1e9 / hbm_peak,
                                       "bytes_per_step": conv["bwd_bytes"],
                                       "gpu_launches": conv["steps"],
                                       "call": "ssm_conv1d_bwd (dx, dweight, dbias)"}}
    if ssd is not None:
        sh = SSD_SHAPE
        ss = ssd["step_ms"] / 1e3
        fl = ssd_flops(**sh)
        nb = ssd_bytes(**sh)
        line["ssd"] = {"workload": "mamba2_130m_layer_ssd: batch %d, L %d, %d heads x %d, %d group, "
                                   "N %d, bf16, chunk 64" % (sh["batch"], sh["L"], sh["H"], sh["P"],
                                                            sh["G"], sh["N"]),
                       "steps": ssd["steps"], "us_per_step": ssd["step_ms"] * 1e3,
                       "tokens_per_s": sh["batch"] * sh["L"] / ss * world,
                       "tensor_tflops": fl / ss / 1e12, "flops_per_step": fl,
                       "hbm_gbs_algorithmic": nb / ss / 1e9, "bytes_per_step": nb,
                       "workspace_bytes": ssd["workspace_bytes"], "gpu_launches": 4 * ssd["steps"],
                       "l2": "x, z, y: 3 x 50 MB plus the 100 MB of bf16 chunk-entering states written and read per step, larger than L2",
                       "backward": {"us_per_step": ssd["bwd_ms"] * 1e3, "steps": ssd["bwd_steps"],
                                    "workspace_bytes": ssd["bwd_workspace_bytes"],
                                    "time_vs_forward": ssd["bwd_ms"] / ssd["step_ms"]}}
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line))


if __name__ == "__main__":
    main()
