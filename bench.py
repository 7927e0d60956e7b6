"""Benchmark of the decode-step MLA query path on GB300.

Headline workload: 64 tokens, 128 local heads, fp8_ds_mla KV cache of 4096
pages x 64 tokens, 1% kv_c outliers ("tensorcore_b64_h128_ds"), the largest
batch the metric covers.  The same run then times the one-token 16-head case,
the one-token 64-head latency case and the 8-token 128-head case with the same
steps and warm-up (``per_config``).  A step is one mla_query_decode call:
q_a RMSNorm, Q_B projection, W_UK absorption and the paged KV insert for one
batch of synthetic tokens.

Timing: steps are captured in CUDA graphs and replayed; W warm-up steps, then
exactly K timed steps between CUDA events on the launching stream, with a
barrier and a device synchronise on both sides.  A spin kernel holds the
stream while the start event and the graph launches are queued, so the timed
region holds the steps and not the host's launch latency.  The weights rotate
over enough independent sets that their total exceeds 3x the L2 cache, so
every step streams its weights from HBM.

Prints one JSON line (rank 0).  ``--impl reference`` times the FP64 CPU oracle
on the same workload instead (host cores, bounded).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per MLA-query decode step and HBM GB/s vs ~8 TB/s peak, B=1..64"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
_CSRC = "mla_query_projection_gb300/csrc/"
# The files that define each kernel family: an ncu summary stays valid while
# they are unchanged.
KERNEL_SOURCES = {
    "fused": [_CSRC + f for f in ("mla_common.cuh", "mla_device.cuh", "mla_internal.h",
                                  "mla_fused.cu", "mla_split.cpp")],
    "wide": [_CSRC + f for f in ("mla_common.cuh", "mla_device.cuh", "mla_internal.h",
                                 "mla_wide.cu", "mla_split.cpp")],
    "qkv_a": [_CSRC + f for f in ("mla_device.cuh", "mla_qkv_a.cu")],
    "small": [_CSRC + f for f in ("mla_common.cuh", "mla_device.cuh", "mla_internal.h",
                                  "mla_small.cu", "mla_split.cpp")],
}


def kernel_sources(kernel: str) -> list[str]:
    """Source files of the kernel(s) named ("a+b" for a chain of launches)."""
    out = []
    for k in kernel.split("+"):
        fam = ("qkv_a" if "qkv_a" in k else "wide" if "wide" in k
               else "small" if "small" in k else "fused")
        out += [f for f in KERNEL_SOURCES[fam] if f not in out]
    return out


def algorithmic_bytes(batch: int, heads: int, layout: int, hidden: bool = False) -> int:
    """Bytes one decode step must move: W_QB (H*192*1536*2) + W_UK (H*128*512*2)
    + gammas (2*(1536+512)) + activations read (B*(1536+512+64)*2 + 8 slot)
    + outputs written (B*H*(512+64)*2 + q_c B*1536*2) + cache rows (576, 656
    or 352 bytes by layout).  A step from the hidden row adds the qkv_a
    projection: W_QKV_A (2112*7168*2), the hidden rows (B*7168*2) and the
    fused row it writes (B*2112*2)."""
    row = {0: 576, 1: 656, 2: 352}[layout]
    n = (heads * 192 * 1536 * 2 + heads * 128 * 512 * 2 + 2 * (1536 + 512)
         + batch * ((1536 + 512 + 64) * 2 + 8) + batch * heads * (512 + 64) * 2
         + batch * 1536 * 2 + batch * row)
    if hidden:
        n += QKV_ROW * HIDDEN * 2 + batch * HIDDEN * 2 + batch * QKV_ROW * 2
    return n


def algorithmic_flops(batch: int, heads: int, hidden: bool = False) -> int:
    f = 2 * batch * heads * (192 * 1536 + 128 * 512)
    return f + (2 * batch * QKV_ROW * HIDDEN if hidden else 0)


def kernel_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for p in kernel_sources(kernel):
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_peaks() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


QKV_ROW, HIDDEN = 2112, 7168


def dominant_kernel(kernels: str) -> str:
    """The kernel whose ncu summary a step's traffic comes from: of the kernels
    a decode launches ("a+b", as mla_query_kernel_for names them), the wide
    kernel, else the first."""
    names = kernels.split("+")
    return next((k for k in names if k.endswith("wide_kernel")), names[0])


def launches_per_step(kernels: str, batch: int, hidden: bool = False) -> int:
    """Kernels one step launches: those a decode names, once per 64 tokens on
    the wide path and once per 16 tokens when the 16-token paired kernel
    serves more than 16; a step from the hidden row first runs the qkv_a
    projection once per 8 tokens."""
    n = len(kernels.split("+"))
    if "wide_kernel" in kernels:
        n *= -(-batch // 64)
    elif batch > 16:
        n *= -(-batch // 16)
    return n + (-(-batch // 8) if hidden else 0)


def profile_name(kernel: str, workload: str) -> str:
    base = kernel.split("<")[0]
    return os.path.join(ROOT, "profiles", f"{base}_{workload}.txt")


def read_traffic(kernel: str, workload: str) -> float | None:
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if it was taken on the current kernel sources."""
    p = profile_name(kernel, workload)
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_sources_sha256_16") != kernel_hash(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- workloads

WORKLOAD_DEFAULT = "tensorcore_b64_h128_ds"


def workload_cfg(name: str) -> dict:
    from mla_query_projection_gb300 import synthetic as S

    if name in S.WORKLOADS:
        return dict(S.WORKLOADS[name])
    # sweep point: sweep_b{B}_h{H}_{e4m3|ds|nvfp4}
    parts = name.split("_")
    if parts[0] == "sweep":
        b, h = int(parts[1][1:]), int(parts[2][1:])
        lay = {"e4m3": S.LAYOUT_E4M3, "ds": S.LAYOUT_DS_MLA,
               "nvfp4": S.LAYOUT_NVFP4_DS_MLA}[parts[3]]
        return S.sweep_workload(b, h, lay)
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------- ranks


def max_over_ranks(values, device=None) -> list[float]:
    """Each value's maximum over all ranks: the slowest replica sets the time
    of a step.  Without an initialised process group, the values themselves."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_us(per_step_us: float, world: int) -> float:
    """Whole-job time per decode step when `world` replicas each run one step
    in the same (max-over-ranks) time: N steps complete per per-step time."""
    return per_step_us / world


def runs_reference_arm(rank: int) -> bool:
    """The oracle arm runs on rank 0 only; other ranks exit without work."""
    return rank == 0


# ---------------------------------------------------------------- GPU arm


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
            return
        t0 = time.time()
        while time.time() - t0 < 5.0:  # wait for the first sample
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                c = [x.strip() for x in line.split(",")]
                if len(c) < 9:
                    continue
                try:
                    sm.append(float(c[1]))
                    smax.append(float(c[2]))
                    power.append(float(c[3]))
                except ValueError:
                    continue
                for n, v in zip(names, c[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons),
            "samples": len(sm),
            "power_w_max": max(power) if power else None,
        }


def hold_stream(stream, cycles: int = 2_000_000) -> None:
    """Keep `stream` busy for about a millisecond (a spin kernel), so that the
    start event and the graph launches queued behind it are already on the
    device when it ends: the timed region then holds the steps and not the
    host's launch latency.  Outside the timed region."""
    import torch

    with torch.cuda.stream(stream):
        torch.cuda._sleep(cycles)


class Workload:
    """Device inputs, rotating weight sets and handles of one workload, and
    its decode call.  Weight set 0 is the seeded generator's; the others are
    drawn on the device from a seeded torch generator with the same
    distributions, until the sets total at least 3x the L2 size."""

    def __init__(self, name: str, rank: int, dev, path: int = 0, nsets: int = 0):
        import torch

        from mla_query_projection_gb300 import binding as B
        from mla_query_projection_gb300 import synthetic as S
        from mla_query_projection_gb300.runner import bf16_tensor

        self.B = B
        self.name = name
        self.dev = dev
        self.cfg = cfg = workload_cfg(name)
        inp = self.inp = S.make_inputs(**cfg)
        self.Bn, self.H, self.layout = cfg["batch"], cfg["heads"], cfg["layout"]
        H, hidden = self.H, bool(cfg.get("hidden", False))
        self.hidden = hidden
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.wbytes = H * (192 * 1536 + 128 * 512) * 2 + (QKV_ROW * HIDDEN * 2 if hidden else 0)
        self.nsets = nsets = nsets or max(1, -(-3 * self.l2 // self.wbytes))
        gen = torch.Generator(device=dev)
        gen.manual_seed(1234 + rank)
        self.sets = []
        for k in range(nsets):
            if k == 0:
                w = dict(w_qb=bf16_tensor(inp["w_qb"], dev), w_uk=bf16_tensor(inp["w_uk"], dev),
                         gamma_q=bf16_tensor(inp["gamma_q"], dev),
                         gamma_kv=bf16_tensor(inp["gamma_kv"], dev))
            else:
                w = dict(
                    w_qb=(torch.randn(H * 192, 1536, device=dev, generator=gen) * 0.02).bfloat16(),
                    w_uk=(torch.randn(H, 128, 512, device=dev, generator=gen) * 0.05).bfloat16(),
                    gamma_q=(1 + 0.1 * torch.randn(1536, device=dev, generator=gen)).bfloat16(),
                    gamma_kv=(1 + 0.1 * torch.randn(512, device=dev, generator=gen)).bfloat16())
            w["handle"] = B.mla_query_create(H, w["w_qb"], w["w_uk"], w["gamma_q"],
                                             w["gamma_kv"], float(inp["eps"]))
            if hidden:
                w["w_qkv_a"] = (bf16_tensor(inp["w_qkv_a"], dev) if k == 0 else
                                (torch.randn(QKV_ROW, HIDDEN, device=dev, generator=gen)
                                 * 0.012).bfloat16())
                w["qkv_a"] = B.mla_qkv_a_create(QKV_ROW, HIDDEN, w["w_qkv_a"])
            if path:
                B.mla_query_set_path(w["handle"], path)
            self.sets.append(w)
        self.q_a = bf16_tensor(inp["q_a"], dev)
        self.kv_c = bf16_tensor(inp["kv_c"], dev)
        self.k_pe = bf16_tensor(inp["k_pe"], dev)
        self.slots = torch.from_numpy(inp["slots"]).to(dev)
        self.cache = torch.from_numpy(inp["cache"]).to(dev)
        self.k_scale = torch.tensor([inp["k_scale"]], dtype=torch.float32, device=dev)
        self.q_latent = torch.empty(self.Bn, H, 512, dtype=torch.bfloat16, device=dev)
        self.q_pe = torch.empty(self.Bn, H, 64, dtype=torch.bfloat16, device=dev)
        self.q_c = torch.empty(self.Bn, 1536, dtype=torch.bfloat16, device=dev)
        self.pages, self.psize = self.cache.shape[0], self.cache.shape[1]
        if hidden:
            # the step from the hidden row: the projection writes the fused
            # row the decode step reads
            self.x_hidden = bf16_tensor(inp["hidden"], dev)
            self.y_row = torch.empty(self.Bn, QKV_ROW, dtype=torch.bfloat16, device=dev)
        self.kernels = B.mla_query_kernel_for(self.sets[0]["handle"], self.Bn)
        self.path = B.mla_query_path_for(self.sets[0]["handle"], self.Bn)

    def decode(self, j, stream, qa=None, kvc=None, kpe=None, sl=None, ql=None, qp=None, qc=None,
               stride=0, x=None, y=None):
        """Step j (weight set j mod nsets) on `stream`.  The keyword buffers
        replace the workload's own (the end-to-end loop's staging buffers):
        q_a, kv_c and k_pe rows with one row stride, or for the step from the
        hidden row the hidden rows x (stride 7168) and the fused row y."""
        B = self.B
        qa = self.q_a if qa is None else qa
        kvc = self.kv_c if kvc is None else kvc
        kpe = self.k_pe if kpe is None else kpe
        sl = self.slots if sl is None else sl
        ql = self.q_latent if ql is None else ql
        qp = self.q_pe if qp is None else qp
        qc = self.q_c if qc is None else qc
        w = self.sets[j % self.nsets]
        if self.hidden:
            xs = 0 if x is None else HIDDEN
            x = self.x_hidden if x is None else x
            y = self.y_row if y is None else y
            rc = B.mla_qkv_a_run(w["qkv_a"], self.Bn, x, xs, y, QKV_ROW, stream)
            if rc != B.MLA_OK:
                raise RuntimeError(f"mla_qkv_a_run: {B.strerror(rc)}")
            qa, kvc, kpe, stride = y, y[:, 1536:], y[:, 2048:], QKV_ROW
        rc = B.mla_query_decode(w["handle"], self.Bn, qa, stride, kvc, stride, kpe, stride, sl,
                                self.cache, self.pages, self.psize, self.layout, self.k_scale, ql,
                                qp, qc, stream)
        if rc != B.MLA_OK:
            raise RuntimeError(f"mla_query_decode: {B.strerror(rc)}")

    def flags(self, stream) -> int:
        f = 0
        for w in self.sets:
            f |= self.B.mla_query_get_error(w["handle"], stream)
            if self.hidden:
                f |= self.B.mla_qkv_a_get_error(w["qkv_a"], stream)
        return f

    def close(self):
        for w in self.sets:
            self.B.mla_query_destroy(w["handle"])
            if self.hidden:
                self.B.mla_qkv_a_destroy(w["qkv_a"])
        self.sets = []


def time_device(wl: Workload, steps: int, warmup: int, graph_steps: int, stream, barrier,
                sampler=None) -> float:
    """ms for exactly `steps` decode steps replayed from CUDA graphs of up to
    `graph_steps` steps, after `warmup` untimed steps (whole graphs).  Each
    graph launch adds a start-up of its own (the first step has no
    predecessor to overlap, the last no successor): about 8 us on GB300,
    spread over the graph's steps.  (Launching the steps one by one instead
    measured slower: 9.15 against 8.56 us per step for 20 one-token steps.)"""
    import torch

    dev = wl.dev
    G = max(1, min(graph_steps, steps))

    def capture(n, first=0):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for j in range(2):  # eager warm-up of the capture stream
                wl.decode(j, stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for j in range(first, first + n):
                    wl.decode(j, torch.cuda.current_stream())
        return g

    g_full = capture(G)
    # one untimed step, on the last weight set, replayed just before the start
    # event: the first timed step then starts as a graph that follows another
    # on the device, not after an idle front end (about 1.2 us less per timed
    # region); it completes before the start event is recorded
    g_lead = capture(1, first=wl.nsets - 1)
    rem = steps % G
    g_rem = capture(rem) if rem else None
    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-warmup // G))):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
    torch.cuda.synchronize(dev)
    if sampler is not None:
        sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    hold_stream(stream)
    with torch.cuda.stream(stream):
        g_lead.replay()
        e0.record(stream)
        for _ in range(steps // G):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop() if sampler is not None else None
    flags = wl.flags(stream)
    if flags:
        raise RuntimeError(f"device error flags {flags} during the timed run of {wl.name}")
    del g_full, g_rem, g_lead
    return e0.elapsed_time(e1), clocks


def time_e2e(wl: Workload, steps: int, nbuf: int, stream, barrier) -> tuple[float, int, int]:
    """ms for `steps` end-to-end steps, as a serving loop would run them:
    every step copies its inputs from pinned host memory to the device, runs
    the decode through the C ABI and copies its outputs back to pinned host
    memory.  `nbuf` staging buffers each way and three streams (copy in,
    compute, copy out) ordered by events, so that step j+1's upload and step
    j-1's download overlap step j's decode.  The inputs are the fused
    q_a|kv_c|k_pe rows (stride 2112; the hidden rows for the step from the
    hidden row) followed by the slots, the outputs q_latent|q_pe|q_c back to
    back.  Steps are captured in CUDA graphs of up to 50 steps."""
    import torch

    dev = wl.dev
    Bn, H, hidden = wl.Bn, wl.H, wl.hidden
    row = HIDDEN if hidden else QKV_ROW
    in_rows = Bn * row * 2
    in_bytes = in_rows + Bn * 8
    if hidden:
        fused = wl.x_hidden.cpu().contiguous()
    else:
        fused = torch.cat([wl.q_a.cpu(), wl.kv_c.cpu(), wl.k_pe.cpu()], dim=1).contiguous()
    o_sizes = [Bn * H * 512 * 2, Bn * H * 64 * 2, Bn * 1536 * 2]
    bufs = []
    for _ in range(nbuf):
        h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        h_in[:in_rows].copy_(fused.view(torch.uint8).reshape(-1))
        h_in[in_rows:].copy_(wl.slots.cpu().view(torch.uint8).reshape(-1))
        d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        d_out = torch.empty(sum(o_sizes), dtype=torch.uint8, device=dev)
        bufs.append(dict(
            h_in=h_in, d_in=d_in, d_out=d_out,
            rows=d_in[:in_rows].view(torch.bfloat16).view(Bn, row),
            sl=d_in[in_rows:].view(torch.int64),
            ql=d_out[:o_sizes[0]].view(torch.bfloat16),
            qp=d_out[o_sizes[0]:o_sizes[0] + o_sizes[1]].view(torch.bfloat16),
            qc=d_out[o_sizes[0] + o_sizes[1]:].view(torch.bfloat16),
            h_out=torch.empty(sum(o_sizes), dtype=torch.uint8).pin_memory(),
            row=torch.empty(Bn, QKV_ROW, dtype=torch.bfloat16, device=dev) if hidden else None,
            ev_in=torch.cuda.Event(), ev_done=torch.cuda.Event(), ev_out=torch.cuda.Event(),
        ))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_step(j, first):
        bf = bufs[j % nbuf]
        if not first:
            s_in.wait_event(bf["ev_done"])  # the decode that read this buffer is done
        with torch.cuda.stream(s_in):
            bf["d_in"].copy_(bf["h_in"], non_blocking=True)
            bf["ev_in"].record(s_in)
        stream.wait_event(bf["ev_in"])
        if not first:
            stream.wait_event(bf["ev_out"])  # this buffer's last outputs are downloaded
        r = bf["rows"]
        if hidden:
            wl.decode(j, stream, x=r, y=bf["row"], sl=bf["sl"], ql=bf["ql"], qp=bf["qp"],
                      qc=bf["qc"])
        else:
            wl.decode(j, stream, qa=r, kvc=r[:, 1536:], kpe=r[:, 2048:], sl=bf["sl"],
                      ql=bf["ql"], qp=bf["qp"], qc=bf["qc"], stride=QKV_ROW)
        bf["ev_done"].record(stream)
        s_out.wait_event(bf["ev_done"])
        with torch.cuda.stream(s_out):
            bf["h_out"].copy_(bf["d_out"], non_blocking=True)
            bf["ev_out"].record(s_out)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for j in range(2 * nbuf):  # eager warm-up of every stream and buffer
                e2e_step(j, j < nbuf)
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g, stream=stream):
                s_in.wait_stream(stream)
                s_out.wait_stream(stream)
                for j in range(n):
                    e2e_step(j, j < nbuf)
                stream.wait_stream(s_in)
                stream.wait_stream(s_out)
        return g

    G = min(steps, 50)
    g_full = capture(G)
    g_rem = capture(steps % G) if steps % G else None
    with torch.cuda.stream(stream):
        g_full.replay()
    torch.cuda.synchronize(dev)
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    hold_stream(stream)
    with torch.cuda.stream(stream):
        f0.record(stream)
        for _ in range(steps // G):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        f1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    flags = wl.flags(stream)
    if flags:
        raise RuntimeError(f"device error flags {flags} during the end-to-end run of {wl.name}")
    return f0.elapsed_time(f1), in_bytes, sum(o_sizes)


def gpu_arm(args, rank: int, world: int, local_rank: int) -> dict | None:
    """The headline workload (device-only and end-to-end), then each of
    `args.also` device-only, all with the same steps and warm-up."""
    import torch

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    out = {}
    wl = Workload(args.workload, rank, dev, args.path)
    sampler = ClockSampler(local_rank)
    ms, clocks = time_device(wl, args.steps, args.warmup, args.graph_steps, stream, barrier,
                             sampler)
    K_e = max(1, min(args.steps, args.e2e_steps))
    ms_e2e, h2d, d2h = time_e2e(wl, K_e, args.e2e_bufs, stream, barrier)
    out.update(clocks=clocks, nsets=wl.nsets, l2=wl.l2, wbytes=wl.wbytes, K_e=K_e, h2d=h2d,
               d2h=d2h, kernels=wl.kernels, path=wl.path)
    per_step_ms, per_step_e2e_ms = max_over_ranks([ms / args.steps, ms_e2e / K_e], dev)
    out.update(per_step_ms=per_step_ms, per_step_e2e_ms=per_step_e2e_ms)
    wl.close()
    del wl
    torch.cuda.empty_cache()
    others = {}
    for name in args.also:
        if name == args.workload:
            continue
        w2 = Workload(name, rank, dev, args.path)
        ms2, _ = time_device(w2, args.steps, args.warmup, args.graph_steps, stream, barrier)
        (per2,) = max_over_ranks([ms2 / args.steps], dev)
        others[name] = dict(per_step_ms=per2, kernels=w2.kernels, cfg=w2.cfg, nsets=w2.nsets)
        w2.close()
        del w2
        torch.cuda.empty_cache()
    out["others"] = others
    sweep = {}
    for name in (args.points if args.sweep else ()):
        w2 = Workload(name, rank, dev, args.path)
        ms2, _ = time_device(w2, args.steps, args.warmup, args.graph_steps, stream, barrier)
        (per2,) = max_over_ranks([ms2 / args.steps], dev)
        sweep[name] = dict(per_step_ms=per2, kernels=w2.kernels)
        w2.close()
        del w2
        torch.cuda.empty_cache()
    out["sweep"] = sweep
    return out


def sweep_profile(args, local_rank: int) -> None:
    """Three decode steps per sweep point with one weight set, in the order
    of --points (the 28 sweep points by default), for a short ncu pass
    (tensor-pipe utilisation and DRAM bytes per point): the third launch of
    each point is a warm step."""
    import torch

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    for name in args.points:
        wl = Workload(name, 0, dev, args.path, nsets=1)
        with torch.cuda.stream(stream):
            for j in range(3):
                wl.decode(j, stream)
        torch.cuda.synchronize(dev)
        if wl.flags(stream):
            raise RuntimeError(f"device error flags during {name}")
        print(name, wl.kernels, flush=True)
        wl.close()


# ---------------------------------------------------------------- CPU oracle

# Timing child: a fresh interpreter (no CUDA context to inherit) that loads the
# workload's inputs and times whole oracle steps.  With W > 1 workers the
# heads are split over W processes (spawned), each running the oracle's step
# on its heads; the KV insert runs once, on worker 0 (the others get skipped
# slots and a one-page cache), so the work of one step is done once.
_ORACLE_CHILD = r"""
import json, multiprocessing as mp, os, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np
path, budget, steps, warm, workers = sys.argv[2], float(sys.argv[3]), int(sys.argv[4]), int(sys.argv[5]), int(sys.argv[6])

def load(path):
    d = np.load(path)
    inp = {k: d[k] for k in d.files}
    inp["layout"] = int(inp["layout"])
    for k in ("k_scale", "eps"):
        inp[k] = float(inp[k])
    return inp

_INP = None

def part(inp, w, W):
    H = inp["w_uk"].shape[0]
    h0, h1 = H * w // W, H * (w + 1) // W
    p = dict(inp)
    p["w_qb"] = inp["w_qb"][h0 * 192:h1 * 192]
    p["w_uk"] = inp["w_uk"][h0:h1]
    if w > 0:
        p["slots"] = np.full_like(inp["slots"], -1)
        p["cache"] = inp["cache"][:1]
        p.pop("hidden", None)
    return p if h1 > h0 else None

def init(path, w_queue, W):
    global _INP
    w = w_queue.get()
    _INP = part(load(path), w, W)

def run_one(_):
    from oracle import mla_oracle as O
    if _INP is None:
        return 0
    if "hidden" in _INP:  # the step from the hidden row starts with the projection
        O.qkv_a_projection(_INP["hidden"], _INP["w_qkv_a"])
    O.decode_step(_INP)
    return 1

def main():
    global _INP
    if workers == 1:
        _INP = load(path)
        step = lambda: run_one(0)
    else:
        ctx = mp.get_context("spawn")
        q = ctx.Queue()
        for w in range(workers):
            q.put(w)
        pool = ctx.Pool(workers, initializer=init, initargs=(path, q, workers))
        step = lambda: pool.map(run_one, range(workers), chunksize=1)
        # every worker has its part before the clock starts
        step()
    for _ in range(max(1, warm)):
        step()
    t0 = time.perf_counter(); n = 0
    while True:
        step(); n += 1
        el = time.perf_counter() - t0
        if (steps and n >= steps) or (not steps and el >= budget):
            break
    print(json.dumps({"seconds": el, "samples": n}))
    if workers > 1:
        pool.close(); pool.join()

if __name__ == "__main__":
    main()
"""


def host_info() -> dict:
    """Host core count and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform

    return {"nproc": os.cpu_count(), "cpu_model": model or platform.machine()}


def oracle_time(cfg: dict, budget_s: float, steps: int = 0, warm: int = 1, workers: int = 1,
                sample_heads: int = 0) -> dict:
    """Seconds per oracle step on the workload (all its heads, or the first
    `sample_heads`), single-threaded BLAS in every process: `steps` steps, or
    as many as fit in `budget_s`, after `warm` untimed ones."""
    import numpy as np

    from mla_query_projection_gb300 import synthetic as S

    c = dict(cfg)
    if sample_heads:
        c["heads"] = sample_heads
    inp = S.make_inputs(**c)
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    np.savez(path, **{k: np.asarray(v) for k, v in inp.items()})
    # the child runs from a file: spawned workers re-import it by path
    fd, script = tempfile.mkstemp(suffix="_oracle_timing.py")
    with os.fdopen(fd, "w") as f:
        f.write(_ORACLE_CHILD)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, script, ROOT, path, str(budget_s), str(steps),
                              str(warm), str(workers)], capture_output=True, text=True, env=env,
                             check=True, timeout=max(600.0, 20 * budget_s))
    finally:
        os.unlink(path)
        os.unlink(script)
    r = json.loads(out.stdout.strip().splitlines()[-1])
    return dict(sec_per_step=r["seconds"] / r["samples"], samples=r["samples"],
                seconds=r["seconds"])


def cpu_baseline(cfg: dict, budget_s: float) -> dict:
    """The oracle's full decode step (every head, the workload's cache) on
    the host: one thread, then one process per host core (heads split over
    them).  The value is the single-threaded time."""
    host = host_info()
    cores = max(1, host["nproc"] or 1)
    t1 = oracle_time(cfg, budget_s / 2)
    tn = oracle_time(cfg, budget_s / 2, workers=cores) if cores > 1 else t1
    return {
        "value": t1["sec_per_step"] * 1e6,
        "unit": "us",
        "cores": 1,
        "kind": "oracle",
        "sample": (f"FP64 numpy oracle, the whole step (B={cfg['batch']}, all {cfg['heads']} "
                   f"heads, {cfg['pages']}-page cache), single-threaded BLAS: "
                   f"{t1['samples']} steps in {t1['seconds']:.1f} s"),
        "all_cores": {"value": tn["sec_per_step"] * 1e6, "unit": "us", "cores": cores,
                      "sample": (f"heads split over {cores} spawned processes, the KV insert on "
                                 f"one: {tn['samples']} steps in {tn['seconds']:.1f} s")},
        "host": host,
    }


# ---------------------------------------------------------------- main

KV_NAMES = {0: "fp8_e4m3_per_tensor", 1: "fp8_ds_mla", 2: "nvfp4_ds_mla"}
L2_POLICY = ("inputs larger than L2: the weights rotate over independent sets totalling at "
             "least 3x the L2 size")
ALSO_DEFAULT = ("tiny_b1_h16_e4m3", "latency_b1_h64_e4m3", "small_b8_h128_e4m3")
# The sweep of the metric: B in {1, 2, 4, 8, 16, 32, 64} x H in {64, 128} x
# the per-tensor E4M3 and fp8_ds_mla layouts (4096 pages, 1% kv_c outliers).
SWEEP_POINTS = tuple(f"sweep_b{b}_h{h}_{lay}" for h in (64, 128) for lay in ("e4m3", "ds")
                     for b in (1, 2, 4, 8, 16, 32, 64))


def workload_config(name: str, world: int) -> dict:
    """The `config` object of a workload: the same keys and values on both
    arms."""
    cfg = workload_cfg(name)
    config = {"workload": name, "batch": cfg["batch"], "heads": cfg["heads"],
              "kv_layout": KV_NAMES[cfg["layout"]], "pages": cfg["pages"], "page_size": 64,
              "l2_policy": L2_POLICY, "parallelism": f"replicas{world}"}
    if cfg.get("hidden"):
        config["input"] = f"hidden rows [{cfg['batch']}, {HIDDEN}] through the qkv_a projection"
    return config


def config_entry(name: str, per_step_ms: float, kernels: str, world: int, peak: float) -> dict:
    """One workload's figures: µs per step, tokens/s, GB/s on its algorithmic
    bytes, fraction of the measured copy bandwidth and of 8 TB/s."""
    cfg = workload_cfg(name)
    Bn, H, layout = cfg["batch"], cfg["heads"], cfg["layout"]
    hidden = bool(cfg.get("hidden", False))
    us = per_step_ms * 1e3
    nbytes = algorithmic_bytes(Bn, H, layout, hidden)
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us_per_step": us / world, "tokens_per_s": Bn * world / (per_step_ms * 1e-3),
            "hbm_gbs": gbs, "frac": gbs / peak, "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
            "algorithmic_bytes": nbytes, "kernels": kernels,
            "launches_per_step": launches_per_step(kernels, Bn, hidden)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD_DEFAULT)
    ap.add_argument("--also", default=",".join(ALSO_DEFAULT),
                    help="comma-separated workloads timed after the headline one, device-only "
                         "(reported under per_config); empty for none")
    ap.add_argument("--graph-steps", type=int, default=100)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--e2e-bufs", type=int, default=2,
                    help="staging buffers each way in the end-to-end loop")
    ap.add_argument("--path", type=int, default=0, help="force MLA_PATH_* (0 = auto)")
    ap.add_argument("--sweep", action="store_true",
                    help="also time every sweep point (B x H x layout), reported under sweep")
    ap.add_argument("--sweep-profile", action="store_true",
                    help="only run three decode steps per sweep point (for an ncu pass)")
    ap.add_argument("--points", default="",
                    help="comma list of sweep points (sweep_b{B}_h{H}_{e4m3|ds|nvfp4}) for "
                         "--sweep and --sweep-profile instead of the default 28")
    ap.add_argument("--cpu-budget", type=float, default=16.0)
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    args.also = [w for w in args.also.split(",") if w and w != "none"]
    args.points = [w for w in args.points.split(",") if w] or list(SWEEP_POINTS)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = workload_cfg(args.workload)
    Bn, H, layout = cfg["batch"], cfg["heads"], cfg["layout"]
    hidden = bool(cfg.get("hidden", False))
    config = workload_config(args.workload, world)

    if args.impl == "reference":
        # The reference arm is the FP64 CPU oracle; rank 0 alone runs it.
        if not runs_reference_arm(rank):
            return
        # the whole step when K + W steps fit the budget, else the first hs heads
        budget = 150.0
        probe = oracle_time(cfg, 0.0, steps=1, warm=0)["sec_per_step"]
        per_step_budget = budget / max(1, args.steps + args.warmup)
        hs = H if probe <= per_step_budget else max(1, int(H * per_step_budget / probe))
        r = oracle_time(cfg, 0.0, steps=args.steps, warm=min(args.warmup, 50),
                        sample_heads=hs if hs < H else 0)
        us = r["sec_per_step"] * 1e6 * H / hs
        host = host_info()
        sample = (f"each step: the FP64 oracle on {hs} of {H} heads (B={Bn}, "
                  f"{cfg['pages']}-page cache), single-threaded BLAS"
                  + (f", scaled by {H}/{hs}" if hs < H else ""))
        line = {
            "impl": "reference", "metric": METRIC, "value": us, "unit": "us",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
            "cpu_baseline": {"value": us, "unit": "us", "cores": 1, "kind": "oracle",
                             "sample": sample, "host": host},
            "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return

    import torch

    if args.sweep_profile:
        sweep_profile(args, local_rank)
        return

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    r = gpu_arm(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    if rank != 0:
        return

    per_step_us = r["per_step_ms"] * 1e3
    value = whole_job_us(per_step_us, world)
    nbytes = algorithmic_bytes(Bn, H, layout, hidden)
    achieved = nbytes / (per_step_us * 1e-6) / 1e9
    peak, peak_src = read_peaks()
    kernel = dominant_kernel(r["kernels"])
    if hidden:
        kernel = "mla_qkv_a_kernel+" + kernel
    per_config = {args.workload: config_entry(args.workload, r["per_step_ms"], r["kernels"],
                                              world, peak)}
    for name, o in r["others"].items():
        per_config[name] = config_entry(name, o["per_step_ms"], o["kernels"], world, peak)
    line = {
        "metric": METRIC, "value": value, "unit": "us", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["per_step_ms"], "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config,
        "tokens_per_s": Bn * world / (r["per_step_ms"] * 1e-3),
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_src} (MEASURED_PEAKS hbm_gbs)",
                     "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": nbytes,
                     "traffic": read_traffic(kernel, args.workload),
                     "kernel": kernel, "gflop_per_launch": algorithmic_flops(Bn, H, hidden) / 1e9},
        "e2e": {"value": r["per_step_e2e_ms"] * 1e3 / world, "unit": "us",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                "steps": r["K_e"],
                "note": ("every step: one pinned H2D copy of its inputs, the C-ABI decode, one "
                         "pinned D2H copy of its outputs; two staging buffers each way and "
                         "three streams, so step j+1's upload and step j-1's download overlap "
                         "step j's decode; captured in CUDA graphs of up to 50 steps")},
        "gpu_launches": args.steps * launches_per_step(r["kernels"], Bn, hidden),
        "kernels": r["kernels"],
        "clocks": r["clocks"],
        "timing": {"graph_steps": args.graph_steps,
                   "weight_sets": f"{r['nsets']} sets, {r['nsets'] * r['wbytes'] / 1e6:.0f} MB "
                                  f"against an L2 of {r['l2'] / 1e6:.0f} MB",
                   "launch": "CUDA graphs of up to graph_steps steps, queued behind a spin "
                             "kernel and one untimed step (a one-step graph on another "
                             "weight set) that completes before the start event"},
        "per_config": per_config,
    }
    if r["sweep"]:
        line["sweep"] = {name: config_entry(name, o["per_step_ms"], o["kernels"], world, peak)
                         for name, o in r["sweep"].items()}
    if not args.no_cpu and world == 1:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_budget)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
