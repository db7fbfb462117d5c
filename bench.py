"""Benchmark of the decode step: KV-read GB/s (fraction of HBM peak) and µs per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 13b|7b|70b|int8|tiny|...]
    python bench.py --impl reference ...   # the float64 CPU oracle as the reference arm

One step is one ``ftd_decode_mha`` call: bias add, KV append, scores, softmax,
P.V and the split-K merge for every slot of the batch.  Inputs are synthetic
(seeded, the workload shapes of the decode step's pages) and resident in HBM
before timing starts.  Consecutive steps rotate between cache pools whose
combined size is several times the 129 MB L2, so each step streams its KV
cache from HBM.  The default workload is the largest one, the 13B-shaped
ragged continuous batch.  Rank 0 prints one JSON line.

Every workload is timed two ways: back to back (graph-replayed steps; each
step may start while the previous one drains), and isolated (each step follows,
on the same stream, a projection-shaped GEMM that streams 285 MB of bf16
weights, as a decode step follows the projection kernels in a model: it starts
cold, with nothing of it in L2 and no early start).

With ``--gpus N`` under torchrun every rank runs an independent replica (its
own batch; the decode step needs no collective), ``value`` is the aggregate of
all ranks over the slowest rank's time and ``scaling`` is "weak".
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synthetic import WORKLOADS, gen_seq_lens  # noqa: E402

METRIC = "decode-attention KV-read GB/s (frac of 8 TB/s HBM); µs per decode step"
EB = {"f32": 4, "f16": 2, "bf16": 2, "i8": 1}
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("decode_step_masked_gb300/csrc/ftd_common.cuh",
                  "decode_step_masked_gb300/csrc/ftd_decode_splitk.cuh",
                  "decode_step_masked_gb300/csrc/ftd_decode_gqa_tc.cuh",
                  "decode_step_masked_gb300/csrc/ftd_decode_wide_tc.cuh")  # the kernels of the traffic captures


# option cases the bench times next to the plain step (half output, window, paged cache)
OPTION_CASES = [("13b", dict(out_dtype="bf16")), ("13b", dict(window=1024)), ("13b", dict(page_size=256)),
                ("70b", dict(out_dtype="bf16")), ("70b", dict(window=1024)), ("70b", dict(page_size=256)),
                ("int8", dict(page_size=256)), ("7b", dict(q_len=4)), ("7b", dict(q_len=8)),
                ("70b", dict(q_len=2)), ("70b", dict(q_len=4)), ("70b", dict(ragged=1)),
                ("7b", dict(proj_dim=4096)), ("13b", dict(proj_dim=5120)), ("70b", dict(proj_dim=8192))]


def kernel_name(w, q_len=1) -> str:
    """The kernel one step of workload ``w`` runs (the library's own selection rule)."""
    rows = max(1, q_len) * w.Hq // w.Hkv
    tc = (w.D == 128
          and ((w.cache_dtype in ("f16", "bf16") and rows % 4 == 0) or (w.cache_dtype == "i8" and rows % 8 == 0)))
    if tc and w.cache_dtype != "i8" and rows % 32 == 0:
        return "decode_wide_tc_kernel"
    return "decode_gqa_tc_kernel" if tc else "decode_splitk_kernel"


# ---------------------------------------------------------------- workload
def step_bytes(w, lens, window=0, out_dtype="f32", q_len=1, proj_dim=0) -> dict:
    """Algorithmic bytes of one step: each visible cached K/V row once per kv head
    (with a window, only rows some new token still sees), plus the q_len appended
    rows per slot; with an output projection, also its weight W_o [proj_dim][Hq D]
    read once, the hi / lo operand planes written and read, and y written."""
    lens = np.asarray(lens, np.int64)
    T = max(1, int(q_len))
    act = (lens >= 0) & (lens + T <= w.Lmax)
    vis = lens[act] + T                       # history rows read + new rows written
    if window > 0:
        vis = np.minimum(vis, window + T - 1)
    ctx = int(vis.sum())
    nact = int(act.sum())
    eb = EB[w.cache_dtype]
    qeb = EB[w.qkv_dtype]
    kv_read = 2 * w.Hkv * w.D * eb * (ctx - T * nact)
    kv_write = 2 * w.Hkv * w.D * eb * T * nact
    scale_rw = 8 * w.Hkv * ctx if w.cache_dtype == "i8" else 0
    small = ((w.B * w.Hq * w.D + 2 * w.B * w.Hkv * w.D) * qeb * T + 4 * w.B
             + EB[out_dtype] * w.B * T * w.Hq * w.D)
    proj = 0
    if proj_dim:
        K, tok = w.Hq * w.D, w.B * T
        proj = proj_dim * K * qeb + 2 * 2 * tok * K * qeb + tok * proj_dim * EB[out_dtype]
    return dict(kv=kv_read + kv_write + scale_rw, total=kv_read + kv_write + scale_rw + small + proj, ctx=ctx,
                proj=proj)


def kernel_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), source="measured")
    return dict(hbm_gbs=FALLBACK_HBM_GBS, source="fallback")


def load_traffic(workload: str):
    """DRAM bytes per launch from a committed ncu capture, if taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- device
def page_table(w, page_size, seed):
    """A paged pool covering every slot to Lmax, pages handed out in a seeded random order."""
    pps = -(-w.Lmax // page_size)
    perm = np.random.default_rng([seed, 77]).permutation(w.B * pps).astype(np.int32)
    return perm.reshape(w.B, pps), w.B * pps


def make_pools(w, npools, seed, device, page_size=0):
    """Seeded synthetic caches drawn on the device (same distributions as the parity inputs);
    with page_size, each pool is [num_pages][Hkv][page_size][D] (see page_table)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    pools = []
    lead = (w.B, w.Hkv, w.Lmax)
    if page_size:
        lead = (page_table(w, page_size, seed)[1], w.Hkv, page_size)
    shape = lead + (w.D,)
    for _ in range(npools):
        if w.cache_dtype == "i8":
            lo, hi = w.scale_range
            sc = torch.rand((2,) + lead, device=device, generator=g) * (hi - lo) + lo
            kc = torch.clamp(torch.round(torch.randn(shape, device=device, generator=g) / sc[0, ..., None]),
                             -128, 127).to(torch.int8)
            vc = torch.clamp(torch.round(torch.randn(shape, device=device, generator=g) / sc[1, ..., None]),
                             -128, 127).to(torch.int8)
        else:
            dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.cache_dtype]
            kc = torch.randn(shape, device=device, generator=g).to(dt)
            vc = torch.randn(shape, device=device, generator=g).to(dt)
            sc = None
        pools.append((kc, vc, sc))
    return pools


def make_step_inputs(w, lens, seed, device, out_dtype="f32", q_len=1, proj_dim=0):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1000)
    dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.qkv_dtype]
    tok = (q_len,) if q_len > 1 else ()
    q = torch.randn((w.B,) + tok + (w.Hq, w.D), device=device, generator=g).to(dt)
    kn = torch.randn((w.B,) + tok + (w.Hkv, w.D), device=device, generator=g).to(dt)
    vn = torch.randn((w.B,) + tok + (w.Hkv, w.D), device=device, generator=g).to(dt)
    bias = None
    if w.bias_std is not None:
        bias = (torch.randn(((w.Hq + 2 * w.Hkv) * w.D,), device=device, generator=g) * w.bias_std).to(dt)
    sl = torch.from_numpy(np.asarray(lens, np.int32)).to(device)
    odt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[out_dtype]
    out = torch.empty((w.B,) + tok + (w.Hq, w.D), dtype=odt, device=device)
    d = dict(q=q, k_new=kn, v_new=vn, bias=bias, seq_lens=sl, out=out)
    if proj_dim:  # W_o ~ N(0, 1/K) in the qkv dtype, y in the out dtype
        K = w.Hq * w.D
        d["w_o"] = (torch.randn((proj_dim, K), device=device, generator=g) / K ** 0.5).to(dt)
        d["y"] = torch.empty((w.B,) + tok + (proj_dim,), dtype=odt, device=device)
    return d


def n_pools_for(w, kv_bytes):
    # enough pools that a pool is re-read only after > 2x L2 (129 MB) of other traffic
    if kv_bytes < 1e6:
        return 1
    return int(max(2, min(4, np.ceil(300e6 / kv_bytes) + 1)))


# each isolated step follows a GEMM [16 x 8192] . [8192 x 17408] of bf16: 285 MB of weights (> 2x L2)
FLUSH_GEMM = (16, 8192, 17408)


def decode_call(step, pools, inp, stream):
    """A function that issues step i on ``stream`` (cache pool i mod the pool count)."""
    import decode_step_masked_gb300 as ftd
    n = len(pools)

    def one(i):
        kc, vc, sc = pools[i % n]
        common = (inp["q"].data_ptr(), inp["k_new"].data_ptr(), inp["v_new"].data_ptr(),
                  0 if inp["bias"] is None else inp["bias"].data_ptr(), kc.data_ptr(), vc.data_ptr())
        tail = (inp["seq_lens"].data_ptr(), 0 if sc is None else sc.data_ptr(), inp["out"].data_ptr(),
                stream.cuda_stream)
        if inp.get("block_table") is not None:
            ftd.check(ftd.ftd_decode_mha_paged(step.ctx, *common, inp["block_table"].data_ptr(), *tail))
        elif inp.get("w_o") is not None:
            ftd.check(ftd.ftd_decode_mha_proj(step.ctx, *common, *tail[:3], inp["w_o"].data_ptr(),
                                              inp["y"].data_ptr(), tail[3]))
        else:
            ftd.check(ftd.ftd_decode_mha(step.ctx, *common, *tail))
    return one


def make_flush(device):
    """The isolated steps' predecessor: a GEMM X . W (cuBLAS, bf16) whose weights W exceed
    2x L2, the shape of a decode step's projection; returns a function that issues it."""
    import torch
    m, k, n = FLUSH_GEMM
    g = torch.Generator(device=device)
    g.manual_seed(7)
    x = torch.randn((m, k), device=device, generator=g).to(torch.bfloat16)
    wt = torch.randn((k, n), device=device, generator=g).to(torch.bfloat16)
    y = torch.empty((m, n), dtype=torch.bfloat16, device=device)
    return lambda: torch.matmul(x, wt, out=y)


def run_isolated(step, pools, inp, n, stream, flush):
    """n steps, each preceded on the same stream by the projection-shaped GEMM of
    make_flush(): it streams more than 2x L2 of weights, so the step starts with
    nothing of its own in L2, and it is not a decode launch, so the step cannot
    overlap a previous step.  Each step is timed alone with CUDA events recorded
    right before and after it.  Returns the per-step times in µs."""
    import torch
    import decode_step_masked_gb300 as ftd
    one = decode_call(step, pools, inp, stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(3):  # warm-up
            flush()
            one(i)
        for i, (e0, e1) in enumerate(evs):
            flush()
            e0.record(stream)
            one(i)
            e1.record(stream)
    torch.cuda.synchronize()
    ftd.check(step.get_error())
    return np.array([e0.elapsed_time(e1) * 1e3 for e0, e1 in evs])


def run_timed(step, w, pools, inp, steps, warmup, stream, chunk=100):
    """W untimed steps, then exactly K steps timed with CUDA events on the launching stream.

    The K steps are replayed from CUDA graphs of ``chunk`` captured steps (plus
    one graph for the remainder), the pattern the pages recommend for the
    fixed-shape decode loop, so host launch latency does not starve the GPU.
    """
    import torch
    import decode_step_masked_gb300 as ftd
    one = decode_call(step, pools, inp, stream)

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        before = ftd.ftd_kernel_launches()
        with torch.cuda.graph(g, stream=stream):
            for i in range(nsteps):
                one(i)
        return g, ftd.ftd_kernel_launches() - before

    with torch.cuda.stream(stream):
        for i in range(warmup):
            one(i)
    torch.cuda.synchronize()
    chunk = max(1, min(chunk, steps))
    g_full, launches_full = capture(chunk)
    rem = steps % chunk
    g_rem, launches_rem = capture(rem) if rem else (None, 0)
    nrep = steps // chunk
    g_full.replay()  # graph upload, untimed
    if g_rem is not None:
        g_rem.replay()
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(nrep + 1)]
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for r in range(nrep):
            g_full.replay()
            evs[r + 1].record(stream)
        end = torch.cuda.Event(enable_timing=True)
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    per = np.array([evs[r].elapsed_time(evs[r + 1]) for r in range(nrep)]) * 1e3 / chunk  # µs per step
    total_ms = evs[0].elapsed_time(end)
    ftd.check(step.get_error())
    launches = launches_full * nrep + launches_rem
    return dict(total_ms=total_ms, per_us=per, launches=launches, wall=(t_wall0, t_wall1))


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, window):
        if not self.proc or not self.file:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=[], samples=0, note="nvidia-smi unavailable")
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
                except ValueError:
                    continue
        os.unlink(self.file.name)
        inside = [r for r in rows if window[0] <= r[0] <= window[1]]
        src = "timed region"
        if len(inside) < 3:
            inside = [r for r in rows if r[0] <= window[1]]
            src = "warm-up and timed region (timed region shorter than the sampling interval)"
        if not inside:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=[], samples=0, note="no samples")
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3][i + 1].lower().startswith("active")})
        return dict(sm_mhz=float(np.median([r[1] for r in inside])), sm_max_mhz=max(r[2] for r in inside),
                    reasons=reasons, samples=len(inside), window=src)


def gpu_id_for(local_rank: int) -> str:
    import torch
    props = torch.cuda.get_device_properties(local_rank)
    bus = getattr(props, "pci_bus_id", None)
    dom = getattr(props, "pci_domain_id", None)
    dev = getattr(props, "pci_device_id", None)
    if bus is not None and dom is not None and dev is not None:
        return f"{dom:08X}:{bus:02X}:{dev:02X}.0"
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[local_rank]
    return str(local_rank)


# ---------------------------------------------------------------- CPU oracle
def oracle_timing(w, seconds: float, nthreads: int, seed: int = 0):
    """Time the float64 oracle on bounded samples of the workload: whole slots, in turn."""
    import oracle
    from synthetic import gen_cache_slot, gen_qkv, gen_scales_slot
    o = oracle.load()
    lens = gen_seq_lens(w, seed or None)
    q, kn, vn, bias = gen_qkv(w, seed or None)
    w1 = w.with_(B=1)
    done_bytes, elapsed, slots = 0, 0.0, 0
    b = 0
    cache = {}
    while elapsed < seconds or slots == 0:
        L = int(lens[b])
        if b not in cache:  # input generation is not timed; each slot is drawn once
            sub = dict(q=q[b:b + 1], k_new=kn[b:b + 1], v_new=vn[b:b + 1], bias=bias,
                       k_cache=gen_cache_slot(w, seed or None, "k", b, L, "zero")[None],
                       v_cache=gen_cache_slot(w, seed or None, "v", b, L, "zero")[None],
                       seq_lens=lens[b:b + 1], scales=None)
            if w.cache_dtype == "i8":
                sub["scales"] = np.stack([gen_scales_slot(w, seed or None, "k", b, L, "zero")[None],
                                          gen_scales_slot(w, seed or None, "v", b, L, "zero")[None]])
            cache[b] = sub
        sub = cache[b]
        t0 = time.perf_counter()
        o.decode_step(w1, sub, nthreads=nthreads)
        elapsed += time.perf_counter() - t0
        done_bytes += step_bytes(w1, lens[b:b + 1])["kv"]
        slots += 1
        b = (b + 1) % w.B
    return dict(gbs=done_bytes / elapsed / 1e9, slots=slots, seconds=elapsed, bytes=done_bytes)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine() or "unknown"


def brute_tiny_ms() -> float:
    """Milliseconds of one tiny-workload step of the pure-Python brute force (oracle/brute.py)."""
    from oracle import brute
    from synthetic import gen_all
    w = WORKLOADS["tiny"]
    inp = gen_all(w)
    t0 = time.perf_counter()
    brute.decode_step(w, inp)
    return (time.perf_counter() - t0) * 1e3


def oracle_one_head_seconds(w, nthreads=1) -> float:
    import oracle
    from synthetic import gen_all
    lens = gen_seq_lens(w)
    L = int(np.max(lens))
    ws = w.with_(B=1, Hq=1, Hkv=1, Lmax=max(16, (L + 16) // 16 * 16), bias_std=None)
    inp = gen_all(ws, seq_lens=np.array([L], np.int32), fill_beyond="zero")
    t0 = time.perf_counter()
    oracle.load().decode_step(ws, inp, nthreads=nthreads)
    return time.perf_counter() - t0


# ---------------------------------------------------------------- multi-rank
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_over_ranks(local_ms: float, local_units: float, world: int, device=None):
    """Max of the per-rank timed-region length and the sum of the units processed."""
    if world == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    u = torch.tensor([local_units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ---------------------------------------------------------------- arms
def reference_arm(args):
    """The float64 CPU oracle, timed on the host cores on bounded samples of the same workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.config]
    lens = gen_seq_lens(w)
    per_step = step_bytes(w, lens)
    nthreads = os.cpu_count() or 1
    t_head = max(oracle_one_head_seconds(w, nthreads=1), 1e-4)
    budget = 90.0 / max(1, args.steps + args.warmup)  # the whole run ends within a few minutes
    heads = int(max(1, min(w.B * w.Hq, budget / t_head)))
    import oracle
    from synthetic import gen_all
    L = int(np.max(lens))
    ws = w.with_(B=1, Hq=heads, Hkv=heads, Lmax=max(16, (L + 16) // 16 * 16), bias_std=None)
    inp = gen_all(ws, seq_lens=np.array([L], np.int32), fill_beyond="zero")
    o = oracle.load()
    for _ in range(args.warmup):
        o.decode_step(ws, inp, nthreads=1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        o.decode_step(ws, inp, nthreads=1)
    dt = time.perf_counter() - t0
    sample_bytes = step_bytes(ws, [L])["kv"]
    gbs = sample_bytes * args.steps / dt / 1e9
    line = dict(metric=METRIC, value=gbs, unit="GB/s", n_gpus=args.gpus, steps=args.steps, warmup=args.warmup,
                ms_per_step=dt / args.steps * 1e3, higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic", impl="reference",
                config=dict(workload=w.description, name=w.name, B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D,
                            Lmax=w.Lmax, cache_dtype=w.cache_dtype),
                cpu_baseline=dict(value=gbs, unit="GB/s", cores=1, kind="oracle",
                                  sample=f"{heads} head(s) x context {L + 1} per step (float64 C oracle, one "
                                         f"thread); full step would be {per_step['kv'] / 1e6:.1f} MB"),
                e2e=dict(value=gbs, unit="GB/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def measure_config(name, steps, warmup, seed, device, stream, out_dtype="f32", window=0, page_size=0, q_len=1,
                   flush=None, isolated=0, proj_dim=0, ragged=0):
    """Time one workload; the options select a half-precision output, a sliding
    window, a paged cache (one shuffled block table shared by the rotated pools),
    several new tokens per slot (the cached lengths drop by q_len - 1 so the
    step's last position stays where the plain workload's is) or ragged contexts
    (uniform in 128 .. Lmax, the continuous-batch length mix).  With flush and
    isolated > 0, also time that many isolated steps (run_isolated)."""
    import torch
    import decode_step_masked_gb300 as ftd
    w = WORKLOADS[name]
    if ragged:
        w = w.with_(lens=("ctx_uniform", 128, w.Lmax))
    lens = gen_seq_lens(w) - (q_len - 1)
    by = step_bytes(w, lens, window, out_dtype, q_len, proj_dim)
    # rotation is sized on the bytes a step reads (the visible rows), so each pool leaves L2 between reads
    pools = make_pools(w, n_pools_for(w, by["kv"]), seed, device, page_size)
    inp = make_step_inputs(w, lens, seed, device, out_dtype, q_len, proj_dim)
    num_pages = 0
    if page_size:
        table, num_pages = page_table(w, page_size, seed)
        inp["block_table"] = torch.from_numpy(table).to(device)
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype, out_dtype=out_dtype,
                          window=window, page_size=page_size, num_pages=num_pages, q_len=q_len, proj_dim=proj_dim)
    r = run_timed(step, w, pools, inp, steps, warmup, stream)
    if isolated and flush is not None:
        r["isolated_us"] = run_isolated(step, pools, inp, isolated, stream, flush)
    step.close()
    us = r["total_ms"] * 1e3 / steps
    return w, lens, by, pools, inp, r, us


def roofline(w, by, r, us, peaks, q_len=1):
    """The roofline record of one workload: algorithmic bytes of one launch over its
    measured time, back to back and isolated, against the measured copy peak, with
    the DRAM traffic of a committed ncu capture of the same kernel source."""
    per = r["per_us"]
    d = dict(bound="hbm", achieved=by["total"] / (us * 1e-6) / 1e9, peak=peaks["hbm_gbs"], unit="GB/s",
             frac=by["total"] / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], traffic=load_traffic(w.name),
             peak_source=f"{peaks['source']} (STREAM-style copy)", kernel=kernel_name(w, q_len),
             bytes_per_launch=by["total"], launch_us=us, p50_us=float(np.median(per)),
             p99_us=float(np.percentile(per, 99)), p_note="per-step means of 100-step graph replays")
    iso = r.get("isolated_us")
    if iso is not None and len(iso):
        med = float(np.median(iso))
        d.update(isolated_us=med, isolated_p99_us=float(np.percentile(iso, 99)), isolated_steps=len(iso),
                 isolated_frac=by["total"] / (med * 1e-6) / 1e9 / peaks["hbm_gbs"],
                 isolated_after="bf16 GEMM %dx%dx%d (%.0f MB of weights), events around the step alone"
                 % (FLUSH_GEMM + (FLUSH_GEMM[1] * FLUSH_GEMM[2] * 2 / 1e6,)))
    return d


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--config", default="13b", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ftd", choices=["ftd", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip per-config, e2e and CPU-baseline legs")
    ap.add_argument("--isolated", type=int, default=200, help="isolated steps timed per workload")
    ap.add_argument("--ncu-launches", type=int, default=0,
                    help="profiling mode: launch N untimed steps of --config on one cache pool, print nothing")
    ap.add_argument("--ncu-batch", type=int, default=0,
                    help="profiling mode: only the first B slots of the workload (a smaller capture)")
    ap.add_argument("--ncu-window", type=int, default=0, help="profiling mode: sliding window W")
    ap.add_argument("--ncu-proj", type=int, default=0,
                    help="profiling mode: the step with an output projection to this many features")
    args = ap.parse_args()
    if args.ncu_launches:
        return profile_launches(args.config, args.ncu_launches, args.ncu_batch, args.ncu_window, args.ncu_proj)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import decode_step_masked_gb300 as ftd
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    ftd.build_library()
    ftd.load_library()
    stream = torch.cuda.Stream(device=device)
    peaks = load_peaks()
    flush = make_flush(device)  # the isolated steps' predecessor

    # ---- headline: the named workload, K timed steps ----
    sampler = ClockSampler(gpu_id_for(local))
    with sampler:
        if world > 1:
            torch.distributed.barrier()
        w, lens, by, pools, inp, r, us = measure_config(args.config, args.steps, args.warmup, 1234 + rank,
                                                        device, stream)
        if world > 1:
            torch.distributed.barrier()
    clocks = sampler.summary(r["wall"])
    max_ms, units = reduce_over_ranks(r["total_ms"], float(by["kv"]) * args.steps, world, device)
    value = units / (max_ms * 1e-3) / 1e9
    per = r["per_us"]
    kern_us = r["total_ms"] * 1e3 / args.steps
    line = dict(
        metric=METRIC, value=value, unit="GB/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
        ms_per_step=max_ms / args.steps, us_per_step=max_ms / args.steps * 1e3,
        us_per_step_median=float(np.median(per)), us_per_step_p99=float(np.percentile(per, 99)),
        frac_of_hbm_peak=value / world / peaks["hbm_gbs"], higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="f32", data="synthetic",
        config=dict(workload=w.description, name=w.name, B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, Lmax=w.Lmax,
                    cache_dtype=w.cache_dtype, qkv_dtype=w.qkv_dtype, context_tokens=by["ctx"],
                    kv_bytes_per_step=by["kv"], l2="caches rotated over %d pools of %.0f MB each (> L2 129 MB)"
                    % (len(pools), by["kv"] / 1e6), parallelism=f"replicas x{world}"),
        gpu_launches=int(r["launches"]), clocks=clocks)
    if rank == 0 and args.isolated > 0:
        # the headline's isolated steps, after its timed region (outside the clock window)
        step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
        r["isolated_us"] = run_isolated(step, pools, inp, args.isolated, stream, flush)
        step.close()
    line["roofline"] = roofline(w, by, r, kern_us, peaks)
    del pools

    if rank == 0 and not args.no_extras:
        # ---- end to end through the host-buffer entry point ----
        line["e2e"] = e2e_leg(w, lens, by, device, stream, min(args.steps, 2000))
        # ---- every large workload of the suite, same protocol, each with its roofline ----
        per_cfg = {}
        for name in ("7b", "13b", "70b", "int8", "mqa", "70b_i8", "tiny"):
            if name == w.name:
                per_cfg[name] = dict(us=line["us_per_step"], gbs=value / world, frac=value / world / peaks["hbm_gbs"],
                                     kv_mb=by["kv"] / 1e6, roofline=line["roofline"])
                continue
            w2, _, by2, pools2, _, r2, us2 = measure_config(name, 1000, 50, 99, device, stream, flush=flush,
                                                            isolated=args.isolated)
            per_cfg[name] = dict(us=us2, us_median=float(np.median(r2["per_us"])), gbs=by2["kv"] / us2 / 1e3,
                                 frac=by2["kv"] / us2 / 1e3 / peaks["hbm_gbs"], kv_mb=by2["kv"] / 1e6,
                                 roofline=roofline(w2, by2, r2, us2, peaks))
            del pools2
            torch.cuda.empty_cache()
        line["per_config"] = per_cfg
        # ---- the step's options, each on the workloads of both kernels ----
        opts = {}
        for name, kw in OPTION_CASES:
            w2, _, by2, pools2, _, r2, us2 = measure_config(name, 1000, 50, 99, device, stream, **kw)
            key = name + (":" + ",".join(f"{k}={v}" for k, v in kw.items()) if kw else "")
            opts[key] = dict(us=us2, gbs=by2["kv"] / us2 / 1e3, frac=by2["kv"] / us2 / 1e3 / peaks["hbm_gbs"],
                             kv_mb=by2["kv"] / 1e6, kernel=kernel_name(w2, kw.get("q_len", 1)))
            if kw.get("proj_dim"):
                # decode step + projection; the projection's share against the plain step's time
                extra = us2 - per_cfg[name]["us"]
                opts[key].update(kernel=kernel_name(w2) + " + out_proj_kernel", total_mb=by2["total"] / 1e6,
                                 gbs=by2["total"] / us2 / 1e3, frac=by2["total"] / us2 / 1e3 / peaks["hbm_gbs"],
                                 proj_mb=by2["proj"] / 1e6, proj_extra_us=extra,
                                 proj_gbs=by2["proj"] / extra / 1e3 if extra > 0 else None)
            del pools2
            torch.cuda.empty_cache()
        line["options"] = opts
        # ---- the float64 oracle on the host cores ----
        cores = os.cpu_count() or 1
        cb = oracle_timing(w, 10.0, cores)
        c1 = oracle_timing(w, 3.0, 1)  # the same oracle on one core
        line["cpu_baseline"] = dict(value=cb["gbs"], unit="GB/s", cores=cores, kind="oracle",
                                    sample=f"{cb['slots']} whole slot(s) of the {w.name} workload "
                                           f"({cb['bytes'] / 1e6:.0f} MB of KV) in {cb['seconds']:.1f} s, "
                                           f"OpenMP over (slot, head)",
                                    cpu_model=cpu_model(),
                                    single_thread=dict(value=c1["gbs"], unit="GB/s", cores=1,
                                                       sample=f"{c1['slots']} whole slot(s) in "
                                                              f"{c1['seconds']:.1f} s"),
                                    brute_tiny_ms=brute_tiny_ms())
    elif rank == 0:
        line["e2e"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def profile_launches(name, n, batch=0, window=0, proj_dim=0):
    """N plain launches of one workload on one cache pool (for ncu captures of a single launch);
    batch > 0 keeps only the workload's first slots (their seeded lengths), for a smaller capture;
    proj_dim > 0 adds the output projection (ftd_decode_mha_proj: two kernels per step)."""
    import torch
    import decode_step_masked_gb300 as ftd
    w = WORKLOADS[name]
    lens = gen_seq_lens(w)
    if batch:
        w = w.with_(B=batch)
        lens = lens[:batch]
    device = torch.device("cuda", 0)
    ftd.build_library()
    kc, vc, sc = make_pools(w, 1, 5, device)[0]
    inp = make_step_inputs(w, lens, 5, device, proj_dim=proj_dim)
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype, window=window,
                          proj_dim=proj_dim)
    for _ in range(n):
        if proj_dim:
            step.proj(inp["q"], inp["k_new"], inp["v_new"], inp["seq_lens"], inp["out"], inp["w_o"], inp["y"],
                      bias=inp["bias"], k_cache=kc, v_cache=vc, scales=sc)
        else:
            step(inp["q"], inp["k_new"], inp["v_new"], inp["seq_lens"], inp["out"], bias=inp["bias"], k_cache=kc,
                 v_cache=vc, scales=sc)
    torch.cuda.synchronize()
    ftd.check(step.get_error())
    step.close()


def e2e_leg(w, lens, by, device, stream, steps):
    """Same metric through ftd_decode_mha_host: pinned host inputs in, fp32 output back, every step."""
    import torch
    import decode_step_masked_gb300 as ftd
    step = ftd.DecodeStep(w.B, w.Hq, w.Hkv, w.D, w.Lmax, w.qkv_dtype, w.cache_dtype)
    kp, vp, sp = step.cache_ptrs()
    src = make_pools(w, 1, 7, device)[0]
    for ptr, t in ((kp, src[0]), (vp, src[1])):
        _copy_into(ptr, t)
    if src[2] is not None:
        _copy_into(sp, src[2])
    del src
    torch.cuda.synchronize()
    inp = make_step_inputs(w, lens, 7, device)
    host = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in inp.items() if k != "out"}
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32).pin_memory()
    args = [host["q"].data_ptr(), host["k_new"].data_ptr(), host["v_new"].data_ptr(),
            0 if host["bias"] is None else host["bias"].data_ptr(), 0, 0, host["seq_lens"].data_ptr(), 0,
            out.data_ptr(), stream.cuda_stream]
    for _ in range(20):
        ftd.check(ftd.ftd_decode_mha_host(step.ctx, *args))
    t0 = time.perf_counter()
    for _ in range(steps):
        ftd.check(ftd.ftd_decode_mha_host(step.ctx, *args))
    dt = time.perf_counter() - t0
    ftd.check(step.get_error())
    step.close()
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    return dict(value=by["kv"] * steps / dt / 1e9, unit="GB/s", us_per_step=dt / steps * 1e6,
                h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(out.numel() * 4), steps=steps,
                api="ftd_decode_mha_host (pinned host buffers, stream synchronised every step)")


def _copy_into(ptr, t):
    """Copy a device tensor into library-owned device memory at ``ptr``."""
    import torch

    class _CAI:
        __cuda_array_interface__ = {"shape": (t.numel() * t.element_size(),), "typestr": "|u1",
                                    "data": (int(ptr), False), "version": 3, "strides": None}

    dst = torch.as_tensor(_CAI(), device=t.device)
    dst.copy_(t.contiguous().view(-1).view(torch.uint8))


if __name__ == "__main__":
    main()
