"""Benchmark of the decode-step MLA query path on GB300.

Default workload: one token (B=1), 64 local heads, per-tensor FP8 E4M3 KV cache
of 1024 pages x 64 tokens ("latency_b1_h64_e4m3").  A step is one
mla_query_decode call: q_a RMSNorm, Q_B projection, W_UK absorption and the
paged KV insert for one batch of synthetic tokens.

Timing: steps are captured in CUDA graphs and replayed; W warm-up steps, then
exactly K timed steps between CUDA events on the launching stream, with a
barrier and a device synchronise on both sides.  The weights rotate over
enough independent sets that their total exceeds 3x the L2 cache, so every
step streams its weights from HBM.

Prints one JSON line (rank 0).  ``--impl reference`` times the FP64 CPU oracle
on the same workload instead (bounded samples, host cores).
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
}


def kernel_sources(kernel: str) -> list[str]:
    """Source files of the kernel(s) named ("a+b" for a chain of launches)."""
    out = []
    for k in kernel.split("+"):
        fam = "qkv_a" if "qkv_a" in k else "wide" if "wide" in k else "fused"
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

WORKLOAD_DEFAULT = "latency_b1_h64_e4m3"


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


def gpu_arm(args, rank: int, world: int, local_rank: int) -> dict | None:
    import numpy as np
    import torch

    from mla_query_projection_gb300 import binding as B
    from mla_query_projection_gb300 import synthetic as S
    from mla_query_projection_gb300.runner import bf16_tensor

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = workload_cfg(args.workload)
    inp = S.make_inputs(**cfg)
    Bn, H, layout = cfg["batch"], cfg["heads"], cfg["layout"]
    hidden = bool(cfg.get("hidden", False))
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    wbytes = H * (192 * 1536 + 128 * 512) * 2 + (QKV_ROW * HIDDEN * 2 if hidden else 0)
    nsets = max(1, -(-3 * l2 // wbytes))

    # Weight sets: set 0 from the seeded generator, the others drawn on the
    # device from a seeded torch generator with the same distributions.
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    sets = []
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
        w["handle"] = B.mla_query_create(H, w["w_qb"], w["w_uk"], w["gamma_q"], w["gamma_kv"],
                                         float(inp["eps"]))
        if hidden:
            w["w_qkv_a"] = (bf16_tensor(inp["w_qkv_a"], dev) if k == 0 else
                            (torch.randn(QKV_ROW, HIDDEN, device=dev, generator=gen)
                             * 0.012).bfloat16())
            w["qkv_a"] = B.mla_qkv_a_create(QKV_ROW, HIDDEN, w["w_qkv_a"])
        if args.path:
            B.mla_query_set_path(w["handle"], args.path)
        sets.append(w)

    q_a = bf16_tensor(inp["q_a"], dev)
    kv_c = bf16_tensor(inp["kv_c"], dev)
    k_pe = bf16_tensor(inp["k_pe"], dev)
    slots = torch.from_numpy(inp["slots"]).to(dev)
    cache = torch.from_numpy(inp["cache"]).to(dev)
    k_scale = torch.tensor([inp["k_scale"]], dtype=torch.float32, device=dev)
    q_latent = torch.empty(Bn, H, 512, dtype=torch.bfloat16, device=dev)
    q_pe = torch.empty(Bn, H, 64, dtype=torch.bfloat16, device=dev)
    q_c = torch.empty(Bn, 1536, dtype=torch.bfloat16, device=dev)
    pages, psize = cache.shape[0], cache.shape[1]
    if hidden:
        # the step from the hidden row: the projection writes the fused row
        # the decode step reads
        x_hidden = bf16_tensor(inp["hidden"], dev)
        y_row = torch.empty(Bn, QKV_ROW, dtype=torch.bfloat16, device=dev)

    def decode(j, stream, qa=q_a, kvc=kv_c, kpe=k_pe, sl=slots, ql=q_latent, qp=q_pe, qc=q_c):
        st = 0
        if hidden:
            rc = B.mla_qkv_a_run(sets[j % nsets]["qkv_a"], Bn, x_hidden, 0, y_row, QKV_ROW, stream)
            if rc != B.MLA_OK:
                raise RuntimeError(f"mla_qkv_a_run: {B.strerror(rc)}")
            qa, kvc, kpe, st = y_row, y_row[:, 1536:], y_row[:, 2048:], QKV_ROW
        rc = B.mla_query_decode(sets[j % nsets]["handle"], Bn, qa, st, kvc, st, kpe, st, sl, cache,
                                pages, psize, layout, k_scale, ql, qp, qc, stream)
        if rc != B.MLA_OK:
            raise RuntimeError(f"mla_query_decode: {B.strerror(rc)}")

    stream = torch.cuda.Stream(dev)
    G = max(1, min(args.graph_steps, args.steps))
    # graphs: G steps each (the step index inside a graph picks the weight set)
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for j in range(2):  # eager warm-up of the capture stream
                decode(j, stream)
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for j in range(n):
                    decode(j, torch.cuda.current_stream())
        return g

    g_full = capture(G)
    rem = args.steps % G
    g_rem = capture(rem) if rem else None

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    # warm-up (untimed)
    with torch.cuda.stream(stream):
        for _ in range(max(1, -(-args.warmup // G))):
            g_full.replay()
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local_rank)
    sampler.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps // G):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1)
    path = B.mla_query_path_for(sets[0]["handle"], Bn)
    kernels = B.mla_query_kernel_for(sets[0]["handle"], Bn)
    flags = 0
    for w in sets:
        flags |= B.mla_query_get_error(w["handle"], stream)
        if hidden:
            flags |= B.mla_qkv_a_get_error(w["qkv_a"], stream)
    if flags:
        raise RuntimeError(f"device error flags {flags} during the timed run")

    # e2e: every step copies its inputs from pinned host memory to the device,
    # runs the decode through the C ABI and copies its outputs back to pinned
    # host memory, as a serving loop would: two staging buffers each way and
    # three streams (copy in, compute, copy out) ordered by events, so that
    # step j+1's upload and step j-1's download overlap step j's decode.  The
    # inputs are the fused q_a|kv_c|k_pe rows (stride 2112; the hidden rows for
    # the step from the hidden row) followed by the slots, the outputs
    # q_latent|q_pe|q_c back to back.  Steps are captured in CUDA graphs of up
    # to 50 steps, like the device-only run.
    K_e = max(1, min(args.steps, args.e2e_steps))
    row = HIDDEN if hidden else QKV_ROW  # the step's input row: hidden, or q_a|kv_c|k_pe
    in_rows = Bn * row * 2
    in_bytes = in_rows + Bn * 8
    if hidden:
        fused = x_hidden.cpu().contiguous()
    else:
        fused = torch.cat([q_a.cpu(), kv_c.cpu(), k_pe.cpu()], dim=1).contiguous()
    o_sizes = [Bn * H * 512 * 2, Bn * H * 64 * 2, Bn * 1536 * 2]
    NBUF = args.e2e_bufs
    bufs = []
    for _ in range(NBUF):
        h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        h_in[:in_rows].copy_(fused.view(torch.uint8).reshape(-1))
        h_in[in_rows:].copy_(slots.cpu().view(torch.uint8).reshape(-1))
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
        bf = bufs[j % NBUF]
        if not first:
            s_in.wait_event(bf["ev_done"])  # the decode that read this buffer is done
        with torch.cuda.stream(s_in):
            bf["d_in"].copy_(bf["h_in"], non_blocking=True)
            bf["ev_in"].record(s_in)
        stream.wait_event(bf["ev_in"])
        if not first:
            stream.wait_event(bf["ev_out"])  # this buffer's last outputs are downloaded
        r_in = bf["rows"]
        if hidden:
            rc = B.mla_qkv_a_run(sets[j % nsets]["qkv_a"], Bn, bf["rows"], HIDDEN, bf["row"],
                                 QKV_ROW, stream)
            if rc != B.MLA_OK:
                raise RuntimeError(f"mla_qkv_a_run: {B.strerror(rc)}")
            r_in = bf["row"]
        rc = B.mla_query_decode(sets[j % nsets]["handle"], Bn, r_in, QKV_ROW, r_in[:, 1536:],
                                QKV_ROW, r_in[:, 2048:], QKV_ROW, bf["sl"], cache, pages, psize,
                                layout, k_scale, bf["ql"], bf["qp"], bf["qc"], stream)
        if rc != B.MLA_OK:
            raise RuntimeError(f"mla_query_decode: {B.strerror(rc)}")
        bf["ev_done"].record(stream)
        s_out.wait_event(bf["ev_done"])
        with torch.cuda.stream(s_out):
            bf["h_out"].copy_(bf["d_out"], non_blocking=True)
            bf["ev_out"].record(s_out)

    def capture_e2e(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            for j in range(2 * NBUF):  # eager warm-up of every stream and buffer
                e2e_step(j, j < NBUF)
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g, stream=stream):
                s_in.wait_stream(stream)
                s_out.wait_stream(stream)
                for j in range(n):
                    e2e_step(j, j < NBUF)
                stream.wait_stream(s_in)
                stream.wait_stream(s_out)
        return g

    G_e = min(K_e, 50)
    ge_full = capture_e2e(G_e)
    ge_rem = capture_e2e(K_e % G_e) if K_e % G_e else None
    with torch.cuda.stream(stream):
        ge_full.replay()
    torch.cuda.synchronize(dev)
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        f0.record(stream)
        for _ in range(K_e // G_e):
            ge_full.replay()
        if ge_rem is not None:
            ge_rem.replay()
        f1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms_e2e = f0.elapsed_time(f1)
    h2d = in_bytes
    d2h = sum(o_sizes)

    for w in sets:
        B.mla_query_destroy(w["handle"])
        if hidden:
            B.mla_qkv_a_destroy(w["qkv_a"])

    per_step_ms, per_step_e2e_ms = max_over_ranks([ms / args.steps, ms_e2e / K_e], dev)

    return dict(per_step_ms=per_step_ms, per_step_e2e_ms=per_step_e2e_ms, h2d=h2d, d2h=d2h,
                clocks=clocks, nsets=nsets, l2=l2, K_e=K_e, cfg=cfg, path=path, wbytes=wbytes,
                kernels=kernels)


# ---------------------------------------------------------------- CPU oracle

_ORACLE_CHILD = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np
from oracle import mla_oracle as O
d = np.load(sys.argv[2])
inp = {k: d[k] for k in d.files}
for k in ("layout",):
    inp[k] = int(inp[k])
for k in ("k_scale", "eps"):
    inp[k] = float(inp[k])
budget, steps = float(sys.argv[3]), int(sys.argv[4])
def step():
    if "hidden" in inp:  # the step from the hidden row starts with the projection
        O.qkv_a_projection(inp["hidden"], inp["w_qkv_a"])
    O.decode_step(inp)
step()  # warm
t0 = time.perf_counter(); n = 0
while True:
    step(); n += 1
    el = time.perf_counter() - t0
    if (steps and n >= steps) or (not steps and el >= budget):
        break
print(json.dumps({"seconds": el, "samples": n}))
"""


def oracle_time(cfg: dict, sample_heads: int, budget_s: float, steps: int = 0) -> dict:
    """Time the oracle (single-threaded BLAS) on `sample_heads` heads of the
    workload's batch with an 8-page cache; returns seconds per sample."""
    import numpy as np

    from mla_query_projection_gb300 import synthetic as S

    c = dict(cfg)
    c.update(heads=sample_heads, pages=8)
    inp = S.make_inputs(**c)
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    np.savez(path, **{k: np.asarray(v) for k, v in inp.items()})
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, "-c", _ORACLE_CHILD, ROOT, path, str(budget_s),
                              str(steps)], capture_output=True, text=True, env=env, check=True)
    finally:
        os.unlink(path)
    r = json.loads(out.stdout.strip().splitlines()[-1])
    return dict(sec_per_sample=r["seconds"] / r["samples"], samples=r["samples"],
                seconds=r["seconds"])


def cpu_baseline(cfg: dict, budget_s: float) -> dict:
    """Oracle us per full decode step, from two head counts (linear in H)."""
    H = cfg["heads"]
    h1, h2 = 1, min(H, 8)
    t1 = oracle_time(cfg, h1, budget_s / 3)
    t2 = oracle_time(cfg, h2, 2 * budget_s / 3) if h2 > h1 else t1
    per_head = (t2["sec_per_sample"] - t1["sec_per_sample"]) / max(1, h2 - h1)
    full = t1["sec_per_sample"] + per_head * (H - h1)
    return {
        "value": full * 1e6,
        "unit": "us",
        "cores": 1,
        "kind": "oracle",
        "sample": (f"FP64 numpy oracle, single-threaded BLAS, B={cfg['batch']} tokens on "
                   f"{h1} and {h2} heads (8-page cache), {t1['samples']}+{t2['samples']} "
                   f"samples in {t1['seconds'] + t2['seconds']:.1f} s, extrapolated linearly "
                   f"to {H} heads"),
    }


# ---------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD_DEFAULT)
    ap.add_argument("--graph-steps", type=int, default=100)
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--e2e-bufs", type=int, default=2,
                    help="staging buffers each way in the end-to-end loop")
    ap.add_argument("--path", type=int, default=0, help="force MLA_PATH_* (0 = auto)")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = workload_cfg(args.workload)
    Bn, H, layout = cfg["batch"], cfg["heads"], cfg["layout"]
    hidden = bool(cfg.get("hidden", False))
    config = {"workload": args.workload, "batch": Bn, "heads": H,
              "kv_layout": {0: "fp8_e4m3_per_tensor", 1: "fp8_ds_mla", 2: "nvfp4_ds_mla"}[layout],
              "pages": cfg["pages"], "page_size": 64}
    if hidden:
        config["input"] = f"hidden rows [{Bn}, {HIDDEN}] through the qkv_a projection"

    if args.impl == "reference":
        # The reference arm is the FP64 CPU oracle; rank 0 alone runs it.
        if not runs_reference_arm(rank):
            return
        t_full = oracle_time(cfg, min(H, 8), 2.0)["sec_per_sample"] * H / min(H, 8)
        budget = 150.0
        per_step_budget = budget / max(1, args.steps + args.warmup)
        hs = max(1, min(H, int(H * per_step_budget / max(t_full, 1e-9))))
        oracle_time(cfg, hs, 0.0, steps=min(args.warmup, 50))
        r = oracle_time(cfg, hs, 0.0, steps=args.steps)
        us = r["sec_per_sample"] * 1e6 * H / hs
        line = {
            "impl": "reference", "metric": METRIC, "value": us, "unit": "us",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
            "cpu_baseline": {"value": us, "unit": "us", "cores": 1, "kind": "oracle",
                             "sample": f"each step: the FP64 oracle on {hs} of {H} heads "
                                       f"(B={Bn}, 8-page cache), scaled by {H}/{hs}"},
            "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)
        return

    import torch

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
    config.update({
        "l2_policy": f"inputs larger than L2: {r['nsets']} rotating weight sets "
                     f"({r['nsets'] * r['wbytes'] / 1e6:.0f} MB vs L2 {r['l2'] / 1e6:.0f} MB)",
        "graph_steps": args.graph_steps, "parallelism": f"replicas{world}",
    })
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
    }
    if not args.no_cpu and world == 1:
        line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_budget)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
