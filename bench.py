"""Benchmark of the causal Taylor linear-attention hot path on GB300.

One JSON line on stdout (rank 0).  A timed step is one la_prefill call on the
long-prefill workload (B=16, H=16, N=32768, bf16, non-zero s0/z0 from a
4096-token prefill); ``value`` is its prefill tokens/s (B*N tokens per step,
each token covering all 16 heads), summed over ranks.  The same run also
times the other two calls of the path, reported under ``legs``:
  - prefix: la_prefix_prefill on the JRT-RNN workload (N=32768, M=16384);
  - prefix_padded: the same workload as a left-padded batch (per-row padding
    counts uniform in [0, M], la_prefix_prefill_padded);
  - jrt_prompt: the JRT-Prompt alternative, la_prefill over the prompt read
    twice (2N = 65536 tokens), timed against the prefix call;
  - prefill_decay / decode_decay: the long-prefill and decode workloads with a
    fixed per-head decay 1 - 2^-(4+h) (la_prefill_decay, la_decode_step_decay);
  - prefill_dk8/24/32: la_prefill_ws at other feature dimensions (d' = 8 on
    the tensor-core kernel at the long-prefill shape; d' = 24, 32 at B=4,
    H=16, N=4096 with cuBLASLt batched GEMMs and 4 kernels of the library);
  - decode: la_decode_step on B=128, H=16, 512 consecutive steps captured in
    one CUDA graph, state from a 2048-token prefill (tokens/s and HBM GB/s).
Inputs are seeded synthetic tensors already resident in HBM and larger than
L2 (2.1 GB of q/k/v per prefill step; the 145 MB decode state is read and
written every step).  ``e2e`` times the same prefill through the C-ABI's
host-memory call (la_prefill_host) with pinned host buffers: host->device
copies of q, k, v, s0, z0 and device->host copies of y, s, z inside the timed
region, overlapped with the kernels over slices of (b, h) rows.

Multi-GPU (torchrun): every rank runs its own batch (weak scaling, no
collective on the data path); the timed region is bracketed by barriers and
the max time over ranks is used.

``--impl reference`` times the fp64 CPU oracle (on a bounded sample per
step) on the same metric, for comparison only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from recurrent_lm_gb300 import inputs  # noqa: E402

METRIC = "prefill tokens/s & % bf16 TC peak (B=16,N=32K); decode tokens/s & % HBM BW"
FLOPS_PER_HEAD_TOKEN = 70980        # readout 2*273*65 + update 2*273*65
FLOPS_PER_PREFIX_TOKEN = 35490      # update only
BYTES_PER_HEAD_TOKEN_BF16 = 320     # q 32 + k 32 + v 128 + y 128
BYTES_PER_PREFIX_TOKEN_BF16 = 160   # k_e 32 + v_e 128
STATE_BYTES = 273 * 64 * 4 + 273 * 4  # one head's s and z (fp32)
COMPACT_STATE_BYTES = 153 * 64 * 4 + 153 * 4  # the same in the 153-row compact layout
COMPACT_LAYERS = 3   # compact decode leg: 3 x 81.5 MB of state, about 1.9x L2


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------- plumbing
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        t = torch.tensor([x], dtype=torch.float64,
                         device=f"cuda:{self.local}" if torch.cuda.is_available() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def done(self):
        if self.pg:
            self.pg.destroy_process_group()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def source_sha(paths) -> str:
    """Hash of the kernel's source files (relative to the repository root)."""
    h = hashlib.sha256()
    for rel in paths:
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()[:16]


def kernel_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu capture, if the capture was
    taken on the current kernel source (profiles/traffic.json records a hash
    of the source files); None otherwise."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    try:
        sha = source_sha(rec["sources"])
    except OSError:
        return None
    return rec["bytes_per_launch"] if sha == rec["source_sha"] else None


TIMED_WINDOWS = []   # (start, end) wall-clock seconds of every timed region


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons; only samples taken
    inside a timed region (TIMED_WINDOWS) are summarised."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: int):
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(dev).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = []

    def start(self):
        import tempfile
        # samples go to a file: a pipe that nobody reads would fill and stall them
        self.log = tempfile.TemporaryFile(mode="w+")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.log, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
            self.proc.wait()
        self.log.seek(0)
        out = self.log.read()
        self.log.close()
        import datetime
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[1]), float(f[2]), f))
            except ValueError:
                continue
        # samples inside the timed regions; if the regions were too short to
        # catch one, those between the first region's start and the last's end
        inside = [r for r in rows if any(a <= r[0] <= b for a, b in TIMED_WINDOWS)]
        scope = "timed regions"
        if not inside and TIMED_WINDOWS:
            lo, hi = min(a for a, _ in TIMED_WINDOWS), max(b for _, b in TIMED_WINDOWS)
            inside = [r for r in rows if lo <= r[0] <= hi]
            scope = "span of the timed regions"
        mhz, watts, reasons = [], [], set()
        mx = max((r[2] for r in rows), default=0.0)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, sm, _, f in inside:
            mhz.append(sm)
            try:
                watts.append(float(f[3]))
            except ValueError:
                pass
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": mx or None, "reasons": [],
                    "samples": 0, "samples_total": len(rows)}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(mhz), "samples_total": len(rows), "scope": scope,
                "power_w_median": statistics.median(watts) if watts else None}


LAST_MEDIAN_MS = [None]   # median per-step time of the last time_loop (this rank)


def time_loop(fn, steps, warmup, dist):
    """Run fn() warmup times untimed, then `steps` times with an event on the
    current stream before each step and after the last; returns the mean ms per
    step (max over ranks) and leaves the median step in LAST_MEDIAN_MS."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    t0 = time.time()
    for i in range(steps):
        ev[i].record(st)
        fn()
    ev[steps].record(st)
    ev[steps].synchronize()
    torch.cuda.synchronize()
    TIMED_WINDOWS.append((t0, time.time()))
    dist.barrier()
    per = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(steps))
    LAST_MEDIAN_MS[0] = per[steps // 2] if steps % 2 else 0.5 * (per[steps // 2 - 1] + per[steps // 2])
    return dist.max(ev[0].elapsed_time(ev[steps]) / steps)


def shard_seed(seed: int, rank: int) -> int:
    """Each rank draws its own batch (weak scaling over independent heads)."""
    return seed + 7919 * rank


def gen_device(shape, gen, dtype=torch.bfloat16, dev="cuda"):
    return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(dtype)


# ------------------------------------------------------------------ legs
def leg_prefill(la, args, dist, dev, clocks):
    w = inputs.WORKLOADS[3]
    B, H, N = w.B, w.H, w.N
    g = torch.Generator(device=dev)
    g.manual_seed(shard_seed(w.seed, dist.rank))
    q = gen_device((B, H, N, 16), g, dev=dev)
    k = gen_device((B, H, N, 16), g, dev=dev)
    v = gen_device((B, H, N, 64), g, dev=dev)
    qs = gen_device((B, H, w.s0_tokens, 16), g, dev=dev)
    ks = gen_device((B, H, w.s0_tokens, 16), g, dev=dev)
    vs = gen_device((B, H, w.s0_tokens, 64), g, dev=dev)
    _, s0, z0 = la.prefill(qs, ks, vs)
    del qs, ks, vs
    y = torch.empty((B, H, N, 64), dtype=torch.bfloat16, device=dev)
    s = torch.empty_like(s0)
    z = torch.empty_like(z0)
    # la_prefill_ws: the workspace lets the last wave's heads run split
    split = not args.no_split
    need = la.load_library().la_prefill_workspace_size(B, H, N, 16, la.binding.LA_DTYPE_BF16)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev) if split else None

    def step():
        la.prefill(q, k, v, s0, z0, y=y, s_out=s, z_out=z, workspace=ws, split=split)

    ms = time_loop(step, args.steps, args.warmup, dist)
    ms_median = LAST_MEDIAN_MS[0]
    la.check_device_status()
    r, n1 = la.prefill_split_info(B, H, N) if split else (0, 0)
    out = {"ms": ms, "ms_median": ms_median, "B": B, "H": H, "N": N, "split_heads": r, "split_chunk": n1,
           "finite": bool(torch.isfinite(y[:, :, -1].float()).all().item())}
    if not args.no_e2e:
        out["e2e"] = e2e_prefill(la, args, dist, q, k, v, s0, z0)
    return out


def e2e_prefill(la, args, dist, q, k, v, s0, z0):
    """Same prefill through the C-ABI's host-memory call (la_prefill_host) from
    pinned host buffers: the H2D copies of the inputs and the D2H copies of y,
    s, z are inside the timed region, pipelined with the kernels over slices
    of (b, h) rows."""
    hq, hk, hv, hs0, hz0 = (t.cpu().pin_memory() for t in (q, k, v, s0, z0))
    B, H, N = q.shape[:3]
    hy = torch.empty((B, H, N, 64), dtype=torch.bfloat16).pin_memory()
    hs = torch.empty(s0.shape, dtype=s0.dtype).pin_memory()
    hz = torch.empty(z0.shape, dtype=z0.dtype).pin_memory()
    ws = torch.empty(la.prefill_host_workspace_size(B, H, N), dtype=torch.uint8, device=q.device)

    def step():
        la.prefill_host(hq, hk, hv, hs0, hz0, y=hy, s_out=hs, z_out=hz, workspace=ws)

    steps = max(1, min(args.steps, 5))
    ms = time_loop(step, steps, max(1, min(args.warmup, 2)), dist)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hs0, hz0))
    d2h = sum(t.numel() * t.element_size() for t in (hy, hs, hz))
    ok = bool(torch.isfinite(hy[:, :, -1].float()).all().item())
    return {"ms": ms, "steps": steps, "h2d": h2d, "d2h": d2h, "finite": ok}


def leg_prefix(la, args, dist, dev):
    w = inputs.WORKLOADS[4]
    B, H, N, M = w.B, w.H, w.N, w.M
    g = torch.Generator(device=dev)
    g.manual_seed(shard_seed(w.seed, dist.rank))
    q = gen_device((B, H, N, 16), g, dev=dev)
    k = gen_device((B, H, N, 16), g, dev=dev)
    v = gen_device((B, H, N, 64), g, dev=dev)
    ke = gen_device((B, H, M, 16), g, dev=dev)
    ve = gen_device((B, H, M, 64), g, dev=dev)
    ws = torch.empty(la.prefix_workspace_size(B, H, M), dtype=torch.uint8, device=dev)
    y = torch.empty((B, H, N, 64), dtype=torch.bfloat16, device=dev)
    s = torch.empty((B, H, 273, 64), dtype=torch.float32, device=dev)
    z = torch.empty((B, H, 273), dtype=torch.float32, device=dev)

    def step():
        la.prefix_prefill(q, k, v, ke, ve, y=y, s_out=s, z_out=z, workspace=ws)

    ms = time_loop(step, max(1, args.steps // 2), max(3, args.warmup // 2), dist)
    la.check_device_status()
    return {"ms": ms, "B": B, "H": H, "N": N, "M": M}


def leg_prefix_padded(la, args, dist, dev):
    """The JRT-RNN prefix workload as a left-padded batch: row b's first p_b
    positions are padding, p_b drawn uniformly in [0, M] (seeded)."""
    w = inputs.WORKLOADS[4]
    B, H, N, M = w.B, w.H, w.N, w.M
    g = torch.Generator(device=dev)
    g.manual_seed(shard_seed(w.seed + 17, dist.rank))
    q = gen_device((B, H, N, 16), g, dev=dev)
    k = gen_device((B, H, N, 16), g, dev=dev)
    v = gen_device((B, H, N, 64), g, dev=dev)
    ke = gen_device((B, H, M, 16), g, dev=dev)
    ve = gen_device((B, H, M, 64), g, dev=dev)
    pads = torch.randint(0, M + 1, (B,), generator=g, device=dev, dtype=torch.int32)
    ws = torch.empty(la.prefix_workspace_size(B, H, M), dtype=torch.uint8, device=dev)
    y = torch.empty((B, H, N, 64), dtype=torch.bfloat16, device=dev)
    s = torch.empty((B, H, 273, 64), dtype=torch.float32, device=dev)
    z = torch.empty((B, H, 273), dtype=torch.float32, device=dev)

    def step():
        la.prefix_prefill(q, k, v, ke, ve, y=y, s_out=s, z_out=z, workspace=ws, left_pad=pads)

    ms = time_loop(step, max(1, args.steps // 2), max(3, args.warmup // 2), dist)
    la.check_device_status()
    valid = int((N - pads.to(torch.int64)).sum().item())
    return {"ms": ms, "B": B, "H": H, "N": N, "M": M, "valid_tokens": valid}


def leg_jrt_prompt(la, args, dist, dev):
    """JRT-Prompt: the prompt read twice by plain causal prefill, i.e.
    la_prefill at 2N = 65536 tokens (B=16, H=16), the pages' comparison
    point for the JRT-RNN prefix call on the same prompt."""
    w = inputs.WORKLOADS[4]
    B, H, N2 = w.B, w.H, 2 * w.N
    g = torch.Generator(device=dev)
    g.manual_seed(shard_seed(w.seed + 29, dist.rank))
    q = gen_device((B, H, N2, 16), g, dev=dev)
    k = gen_device((B, H, N2, 16), g, dev=dev)
    v = gen_device((B, H, N2, 64), g, dev=dev)
    y = torch.empty((B, H, N2, 64), dtype=torch.bfloat16, device=dev)
    s = torch.empty((B, H, 273, 64), dtype=torch.float32, device=dev)
    z = torch.empty((B, H, 273), dtype=torch.float32, device=dev)

    def step():
        la.prefill(q, k, v, y=y, s_out=s, z_out=z)

    ms = time_loop(step, max(1, args.steps // 4), max(3, args.warmup // 2), dist)
    la.check_device_status()
    return {"ms": ms, "B": B, "H": H, "N": w.N, "N_read": N2}


def decay_rates(H: int, dev) -> torch.Tensor:
    """Per-head decay rates 1 - 2^-(4 + h) (from 0.9375 to nearly 1)."""
    return torch.tensor([1.0 - 2.0 ** -(4 + h) for h in range(H)], dtype=torch.float32, device=dev)


def leg_prefill_decay(la, args, dist, dev):
    """The long-prefill workload with a fixed per-head decay (la_prefill_decay_ws)."""
    w = inputs.WORKLOADS[3]
    B, H, N = w.B, w.H, w.N
    g = torch.Generator(device=dev)
    g.manual_seed(shard_seed(w.seed + 31, dist.rank))
    q = gen_device((B, H, N, 16), g, dev=dev)
    k = gen_device((B, H, N, 16), g, dev=dev)
    v = gen_device((B, H, N, 64), g, dev=dev)
    s0 = torch.randn((B, H, 273, 64), generator=g, device=dev)
    z0 = torch.rand((B, H, 273), generator=g, device=dev) + 64.0
    gam = decay_rates(H, dev)
    y = torch.empty((B, H, N, 64), dtype=torch.bfloat16, device=dev)
    s = torch.empty_like(s0)
    z = torch.empty_like(z0)
    split = not args.no_split  # la_prefill_decay_ws: split heads of the last wave
    need = la.load_library().la_prefill_workspace_size(B, H, N, 16, la.binding.LA_DTYPE_BF16)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev) if split else None

    def step():
        la.prefill(q, k, v, s0, z0, y=y, s_out=s, z_out=z, gamma=gam, workspace=ws, split=split)

    ms = time_loop(step, max(1, args.steps // 2), max(3, args.warmup // 2), dist)
    la.check_device_status()
    return {"ms": ms, "B": B, "H": H, "N": N}


def leg_general_dk(la, args, dist, dev):
    """la_prefill_ws at other feature dimensions, bf16, with an initial state:
    d' = 8 on the tensor-core kernel (the padded map) at the long-prefill shape
    B=16, H=16, N=32768; d' = 24, 32 at B=4, H=16, N=4096 with the chunk
    contractions on the tensor cores (cuBLASLt batched GEMMs and the library's
    kernels, in the workspace)."""
    out = {}
    for dk in (8, 24, 32):
        D = 1 + dk + dk * dk
        B, H, N = (16, 16, 32768) if dk == 8 else (4, 16, 4096)
        g = torch.Generator(device=dev)
        g.manual_seed(shard_seed(1500 + dk, dist.rank))
        q = gen_device((B, H, N, dk), g, dev=dev)
        k = gen_device((B, H, N, dk), g, dev=dev)
        v = gen_device((B, H, N, 64), g, dev=dev)
        s0 = torch.randn((B, H, D, 64), generator=g, device=dev)
        z0 = torch.rand((B, H, D), generator=g, device=dev) + 64.0
        y = torch.empty((B, H, N, 64), dtype=torch.bfloat16, device=dev)
        s = torch.empty_like(s0)
        z = torch.empty_like(z0)
        need = la.prefill_workspace_size(B, H, N, dk)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

        def step():
            la.prefill(q, k, v, s0, z0, y=y, s_out=s, z_out=z, workspace=ws)

        ms = time_loop(step, max(1, args.steps // 4), 3, dist)
        la.check_device_status()
        out[dk] = {"ms": ms, "B": B, "H": H, "N": N, "D": D, "workspace_bytes": need,
                   "path": "tensor-core kernel (padded d' = 16 map)" if dk == 8 else
                           "tensor cores: cuBLASLt batched GEMMs + feature, scan, P and y kernels"}
    return out


def leg_decode(la, args, dist, dev, decay: bool = False, compact: bool = False):
    """512 decode steps in one CUDA graph (with decay: la_decode_step_decay;
    compact: the 153-row state from la_prefill_compact and
    la_decode_step_compact).  The 273-row state (143 MB at B=128, H=16) is
    larger than L2; the compact one (81.5 MB) is not, so that leg keeps
    COMPACT_LAYERS independent states (as the layers of a model would) and
    runs each step over all of them in turn: every state leaves L2 before it
    is used again, and the time per layer-step is reported."""
    w = inputs.WORKLOADS[5]
    B, H, T = w.B, w.H, args.decode_steps
    layers = COMPACT_LAYERS if compact else 1
    g = torch.Generator(device=dev)
    g.manual_seed(shard_seed(w.seed, dist.rank))
    states = []
    for _ in range(layers):
        qs = gen_device((B, H, w.s0_tokens, 16), g, dev=dev)
        ks = gen_device((B, H, w.s0_tokens, 16), g, dev=dev)
        vs = gen_device((B, H, w.s0_tokens, 64), g, dev=dev)
        _, s, z = (la.prefill_compact if compact else la.prefill)(qs, ks, vs)
        states.append((s, z))
        del qs, ks, vs
    qd = gen_device((T, B, H, 16), g, dev=dev)
    kd = gen_device((T, B, H, 16), g, dev=dev)
    vd = gen_device((T, B, H, 64), g, dev=dev)
    yd = torch.empty((T, B, H, 64), dtype=torch.bfloat16, device=dev)
    gam = decay_rates(H, dev) if decay else None

    def one(i):
        for s, z in states:
            if compact:
                la.decode_step_compact(qd[i], kd[i], vd[i], s, z, y=yd[i], inplace=True)
            else:
                la.decode_step(qd[i], kd[i], vd[i], s, z, y=yd[i], inplace=True, gamma=gam)
    # warm up the library (per-device set-up) before capture
    one(0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(T):
                one(i)
    torch.cuda.synchronize()
    ms = time_loop(graph.replay, max(1, args.steps // 4), max(3, args.warmup // 2), dist)
    la.check_device_status()
    ok = bool(torch.isfinite(yd[-1].float()).all().item() and torch.isfinite(s[0, 0]).all().item())
    return {"ms_per_graph": ms, "steps_per_graph": T * layers, "layers": layers, "B": B, "H": H,
            "finite": ok}


def cpu_baseline_prefill(sample_rows: int):
    """The fp64 oracle, as it stands, on the first `sample_rows` batch rows of
    the long-prefill workload (all 16 heads, all 32768 tokens, with an s0)."""
    import oracle
    w = inputs.WORKLOADS[3]
    q, k, v, _, _ = inputs.qkv(sample_rows, w.H, w.N, w.seed, w.dtype)
    s0, z0 = inputs.random_state(sample_rows, w.H, seed=w.seed + 1, tokens=float(w.s0_tokens))
    t = time.perf_counter()
    oracle.prefill(q, k, v, s0, z0)
    dt = time.perf_counter() - t
    return {"value": sample_rows * w.N / dt, "unit": "tokens/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"{sample_rows} of 16 batch rows x 16 heads x 32768 tokens with s0 "
                      f"({sample_rows * w.H * w.N} head-tokens, fp64, {dt:.1f} s)"}


# ------------------------------------------------------------------ ncu cases
def ncu_case(la, case: str):
    """Small launches for ncu captures (a few GB on the device at most, inputs
    still larger than L2): prefill B=16, H=16 at N=4096 then N=8192 with an
    initial state, two launches each (DRAM traffic is linear in N, so the
    full-length launch is extrapolated from the two sizes); decode (273-row or
    compact state) at the bench batch B=128, H=16, ten steps in place back to
    back (inputs generated first, so that nothing runs between the steps; the
    compact case over the bench leg's independent states in turn);
    prefix N=M=4096, three calls; the decayed prefill (the bench leg's rates)
    at B=16, H=16, N=8192 with an initial state, two launches (split heads);
    general_dk: d' = 24 then 32 at the bench leg's B=4, H=16, N=4096 with an
    initial state, two calls each (7 launches per call)."""
    dev = "cuda:0"
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    if case == "prefill":
        B, H = 16, 16
        s0 = torch.randn(B, H, 273, 64, device=dev, generator=g)
        z0 = torch.rand(B, H, 273, device=dev, generator=g) + 100.0
        for N in (4096, 8192):
            q = gen_device((B, H, N, 16), g, dev=dev)
            k = gen_device((B, H, N, 16), g, dev=dev)
            v = gen_device((B, H, N, 64), g, dev=dev)
            for _ in range(2):
                la.prefill(q, k, v, s0, z0)
            torch.cuda.synchronize()
            del q, k, v
    elif case in ("decode", "decode_compact"):
        B, H, T = 128, 16, 10
        compact = case == "decode_compact"
        D = 153 if compact else 273
        layers = COMPACT_LAYERS if compact else 1   # as in the bench leg
        states = [(torch.randn(B, H, D, 64, device=dev, generator=g),
                   torch.rand(B, H, D, device=dev, generator=g) + 100.0) for _ in range(layers)]
        q = gen_device((T, B, H, 16), g, dev=dev)
        k = gen_device((T, B, H, 16), g, dev=dev)
        v = gen_device((T, B, H, 64), g, dev=dev)
        y = torch.empty((T, B, H, 64), dtype=torch.bfloat16, device=dev)
        step = la.decode_step_compact if compact else la.decode_step
        torch.cuda.synchronize()
        for i in range(T):
            for s, z in states:
                step(q[i], k[i], v[i], s, z, y=y[i], inplace=True)
    elif case == "prefill_decay":
        B, H, N = 16, 16, 8192
        s0 = torch.randn(B, H, 273, 64, device=dev, generator=g)
        z0 = torch.rand(B, H, 273, device=dev, generator=g) + 64.0
        q = gen_device((B, H, N, 16), g, dev=dev)
        k = gen_device((B, H, N, 16), g, dev=dev)
        v = gen_device((B, H, N, 64), g, dev=dev)
        gam = decay_rates(H, dev)
        for _ in range(2):
            la.prefill(q, k, v, s0, z0, gamma=gam)
    elif case == "general_dk":
        B, H, N = 4, 16, 4096
        for dk in (24, 32):
            D = 1 + dk + dk * dk
            q, k = gen_device((B, H, N, dk), g, dev=dev), gen_device((B, H, N, dk), g, dev=dev)
            v = gen_device((B, H, N, 64), g, dev=dev)
            s0 = torch.randn((B, H, D, 64), generator=g, device=dev)
            z0 = torch.rand((B, H, D), generator=g, device=dev) + 64.0
            ws = torch.empty(la.prefill_workspace_size(B, H, N, dk), dtype=torch.uint8, device=dev)
            for _ in range(2):
                la.prefill(q, k, v, s0, z0, workspace=ws)
            torch.cuda.synchronize()
    elif case == "prefix":
        B, H, N, M = 16, 16, 4096, 4096
        q, k = gen_device((B, H, N, 16), g, dev=dev), gen_device((B, H, N, 16), g, dev=dev)
        v = gen_device((B, H, N, 64), g, dev=dev)
        ke, ve = gen_device((B, H, M, 16), g, dev=dev), gen_device((B, H, M, 64), g, dev=dev)
        for _ in range(3):
            la.prefix_prefill(q, k, v, ke, ve)
    else:
        raise SystemExit(f"unknown ncu case {case}")
    torch.cuda.synchronize()
    la.check_device_status()
    log(f"ncu case {case}: ok")


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--legs",
                    default="prefill,prefix,prefix_padded,jrt_prompt,prefill_decay,general_dk,decode,"
                            "decode_decay,decode_compact")
    ap.add_argument("--decode-steps", type=int, default=512)
    ap.add_argument("--cpu-sample-rows", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-split", action="store_true",
                    help="time la_prefill without the workspace (no split heads in the last wave)")
    ap.add_argument("--ncu-case", choices=["prefill", "decode", "decode_compact", "prefix", "prefill_decay",
                                           "general_dk"],
                    help="run one small case for an ncu capture and exit (no timing)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    dist = Dist()
    if args.impl == "reference":
        return main_reference(args, dist)

    if args.ncu_case:
        import recurrent_lm_gb300 as la
        la.load_library()
        return ncu_case(la, args.ncu_case)
    dist.init("nccl")
    dev = f"cuda:{dist.local}"
    torch.cuda.set_device(dev)
    import recurrent_lm_gb300 as la
    la.load_library()
    legs = set(args.legs.split(","))
    pk = peaks()
    clocks = Clocks(dist.local)

    clocks.start()  # sampled across every timed leg
    pre = leg_prefill(la, args, dist, dev, clocks)
    res = {}
    if "prefix" in legs:
        res["prefix"] = leg_prefix(la, args, dist, dev)
    if "prefix_padded" in legs:
        res["prefix_padded"] = leg_prefix_padded(la, args, dist, dev)
    if "jrt_prompt" in legs:
        res["jrt_prompt"] = leg_jrt_prompt(la, args, dist, dev)
    if "prefill_decay" in legs:
        res["prefill_decay"] = leg_prefill_decay(la, args, dist, dev)
    if "general_dk" in legs:
        res["general_dk"] = leg_general_dk(la, args, dist, dev)
    if "decode" in legs:
        res["decode"] = leg_decode(la, args, dist, dev)
    if "decode_decay" in legs:
        res["decode_decay"] = leg_decode(la, args, dist, dev, decay=True)
    if "decode_compact" in legs:
        res["decode_compact"] = leg_decode(la, args, dist, dev, compact=True)
    pre["clocks"] = clocks.stop()

    W = dist.world
    tokens = pre["B"] * pre["N"]
    head_tokens = pre["B"] * pre["H"] * pre["N"]
    s_ = pre["ms"] / 1e3
    flops = head_tokens * FLOPS_PER_HEAD_TOKEN
    # s0, z0 read once and s, z written once per head (STATE_BYTES covers s and z)
    nbytes = head_tokens * BYTES_PER_HEAD_TOKEN_BF16 + 2 * pre["B"] * pre["H"] * STATE_BYTES
    achieved_tf = flops / s_ / 1e12
    hbm_gbs = nbytes / s_ / 1e9
    traffic = kernel_traffic("prefill")
    line = {
        "metric": METRIC,
        "value": W * tokens / s_,
        "unit": "tokens/s",
        "n_gpus": W,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": pre["ms"],
        "ms_per_step_median": pre["ms_median"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 tensors resident in HBM)",
        "config": {"workload": inputs.WORKLOADS[3].name, "B": pre["B"], "H": pre["H"],
                   "N": pre["N"], "d_feat": 16, "d_v": 64, "D": 273, "s0_tokens": 4096,
                   "global_batch": W * pre["B"], "seq_len": pre["N"],
                   "parallelism": f"independent (b,h) shards x{W}",
                   "split_heads": pre["split_heads"], "split_chunk": pre["split_chunk"],
                   "l2": "inputs larger than L2 (2.1 GB of q,k,v per step)"},
        "roofline": {"bound": "tensor", "achieved": achieved_tf, "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved_tf / pk["bf16_tflops"],
                     "traffic": traffic, "peak_source": pk["source"] + " bf16 burst",
                     "algorithmic_flops_per_launch": flops,
                     "hbm_achieved_gbs": hbm_gbs, "hbm_peak_gbs": pk["hbm_gbs"],
                     "hbm_frac": hbm_gbs / pk["hbm_gbs"], "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": args.steps,
        "clocks": pre["clocks"],
        "clocks_note": "nvidia-smi samples every 100 ms inside the timed regions of all legs",
        "legs": {},
    }
    if "e2e" in pre:
        e = pre["e2e"]
        line["e2e"] = {"value": W * tokens / (e["ms"] / 1e3), "unit": "tokens/s",
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "ms_per_step": e["ms"], "steps": e["steps"]}
    launches = args.steps
    if "prefix" in res:
        r = res["prefix"]
        ht = r["B"] * r["H"]
        fl = ht * (r["N"] * FLOPS_PER_HEAD_TOKEN + r["M"] * FLOPS_PER_PREFIX_TOKEN)
        by = ht * (r["N"] * BYTES_PER_HEAD_TOKEN_BF16 + r["M"] * BYTES_PER_PREFIX_TOKEN_BF16)
        t = r["ms"] / 1e3
        line["legs"]["prefix"] = {
            "workload": inputs.WORKLOADS[4].name, "ms_per_call": r["ms"],
            "tokens_per_s": W * r["B"] * r["N"] / t, "achieved_tflops": fl / t / 1e12,
            "tc_frac": fl / t / 1e12 / pk["bf16_tflops"], "hbm_gbs": by / t / 1e9,
            "hbm_frac": by / t / 1e9 / pk["hbm_gbs"]}
        launches += 2 * max(1, args.steps // 2)
    if "prefix_padded" in res:
        r = res["prefix_padded"]
        t = r["ms"] / 1e3
        line["legs"]["prefix_padded"] = {
            "workload": inputs.WORKLOADS[4].name + "-leftpad-uniform0toM", "ms_per_call": r["ms"],
            "tokens_per_s": W * r["B"] * r["N"] / t,
            "valid_tokens_per_s": W * r["valid_tokens"] / t}
        launches += 2 * max(1, args.steps // 2)
    if "jrt_prompt" in res:
        r = res["jrt_prompt"]
        t = r["ms"] / 1e3
        fl = r["B"] * r["H"] * r["N_read"] * FLOPS_PER_HEAD_TOKEN
        entry = {"workload": f"jrt-prompt-bf16-B{r['B']}-H{r['H']}-N{r['N']}-read-twice",
                 "ms_per_call": r["ms"], "prompt_tokens_per_s": W * r["B"] * r["N"] / t,
                 "achieved_tflops": fl / t / 1e12, "tc_frac": fl / t / 1e12 / pk["bf16_tflops"]}
        if "prefix" in line["legs"]:
            entry["time_vs_jrt_rnn_prefix"] = r["ms"] / line["legs"]["prefix"]["ms_per_call"]
        line["legs"]["jrt_prompt"] = entry
        launches += max(1, args.steps // 4)
    if "prefill_decay" in res:
        r = res["prefill_decay"]
        t = r["ms"] / 1e3
        fl = r["B"] * r["H"] * r["N"] * FLOPS_PER_HEAD_TOKEN
        line["legs"]["prefill_decay"] = {
            "workload": inputs.WORKLOADS[3].name + "-decay-1-2^-(4+h)", "ms_per_call": r["ms"],
            "tokens_per_s": W * r["B"] * r["N"] / t, "achieved_tflops": fl / t / 1e12,
            "tc_frac": fl / t / 1e12 / pk["bf16_tflops"]}
        launches += max(1, args.steps // 2)
    if "general_dk" in res:
        for dk, r in res["general_dk"].items():
            t = r["ms"] / 1e3
            fl = r["B"] * r["H"] * r["N"] * 4 * r["D"] * 65   # readout + update, 2*D*(d_v+1) each
            line["legs"][f"prefill_dk{dk}"] = {
                "workload": f"prefill-bf16-B{r['B']}-H{r['H']}-N{r['N']}-dk{dk}-D{r['D']}-s0",
                "ms_per_call": r["ms"], "tokens_per_s": W * r["B"] * r["N"] / t,
                "achieved_tflops": fl / t / 1e12, "tc_frac": fl / t / 1e12 / pk["bf16_tflops"],
                "path": r["path"], "workspace_bytes": r["workspace_bytes"]}
            # the library's own kernels per call (d' = 24, 32: features, scan, P, y;
            # the three GEMMs are cuBLASLt's)
            launches += max(1, args.steps // 4) * (1 if dk == 8 else 4)
    suffix = {"decode": "", "decode_decay": "-decay-1-2^-(4+h)", "decode_compact": "-compact-state-153"}
    for dname in ("decode", "decode_decay", "decode_compact"):
        if dname not in res:
            continue
        r = res[dname]
        per_step_ms = r["ms_per_graph"] / r["steps_per_graph"]
        bh = r["B"] * r["H"]
        sbytes = COMPACT_STATE_BYTES if dname == "decode_compact" else STATE_BYTES
        by = bh * (2 * sbytes + BYTES_PER_HEAD_TOKEN_BF16)
        gbs = by / (per_step_ms / 1e3) / 1e9
        line["legs"][dname] = {
            "workload": inputs.WORKLOADS[5].name + suffix[dname],
            "us_per_step": per_step_ms * 1e3,
            "tokens_per_s": W * r["B"] / (per_step_ms / 1e3),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "traffic": kernel_traffic(dname) if dname != "decode_decay" else None,
                         "algorithmic_bytes_per_launch": by},
            "cuda_graph_steps": r["steps_per_graph"], "finite": r["finite"]}
        if r["layers"] > 1:
            line["legs"][dname]["layers"] = r["layers"]
            line["legs"][dname]["l2"] = (f"{r['layers']} independent B={r['B']} H={r['H']} states, "
                                         f"{r['layers'] * bh * sbytes / 1e6:.0f} MB, visited in turn "
                                         "each step (larger than L2); us_per_step is per layer-step")
        launches += r["steps_per_graph"] * max(1, args.steps // 4)
    line["gpu_launches"] = launches
    line["gpu_launches_note"] = ("prefill leg: 1 kernel per step; prefix legs: 2 per call; "
                                 "decode legs: 1 per decode step (per layer-step in decode_compact)")
    line["finite_outputs"] = pre["finite"]
    if dist.rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(args.cpu_sample_rows)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.done()


def main_reference(args, dist):
    """The fp64 CPU oracle, timed on host cores (rank 0 only)."""
    if dist.rank != 0:
        return
    import oracle
    w = inputs.WORKLOADS[3]
    n_sample = 4096
    q, k, v, _, _ = inputs.qkv(1, w.H, n_sample, w.seed, w.dtype)
    s0, z0 = inputs.random_state(1, w.H, seed=w.seed + 1, tokens=float(w.s0_tokens))
    for _ in range(args.warmup):
        oracle.prefill(q, k, v, s0, z0)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.prefill(q, k, v, s0, z0)
    dt = (time.perf_counter() - t) / args.steps
    val = n_sample / dt
    sample = f"1 of 16 batch rows x 16 heads x {n_sample} of 32768 tokens with s0, per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N},
        "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
