"""Benchmark of the batched draft-verify step on the batch64-bf16 workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload: B=64 requests, N=7 drafts, V=128256 vocabulary, bf16 logits,
per-request draft noise sigma ~ U[0.2, 1.5] and temperature from
{0, 0.7, 1.0} (synthetic, seeded).  One step = one spec_verify call over the
whole batch (row statistics, walk, residual/bonus sampling).

Metric: verified draft positions per second (B*N per step), plus the
achieved HBM bandwidth of the row-statistics kernel against the measured
copy bandwidth of the GPU (its device time from a separate pass of calls
with events around each kernel, after the timed loop).  Under torchrun each
rank verifies its own batch (weak scaling, no collective on the data path);
the timed region is bracketed by barriers and the slowest rank's time is
used.

On one GPU the line also carries, unless --no-extras:
  per_config  the other workloads of the method statement (tiny-f32,
              single-bf16 at T=1 and T=0, mixture-bf16, alpha09-f32 with one
              verify seed), each timed alone per call with an L2 flush before
              every call, and the oracle on each on one thread and on every
              host core;
  rows_f      short measurements of the tree verify (tree222-bf16), the KV
              commit (32 layers x 64 sequences x 4 KB), the FC-norm fusion
              (T = d = d_out = 4096) and the lazy verify against the eager
              one (batch64-bf16 and lowaccept64-bf16).
cpu_baseline is the oracle on the headline workload, on every host core
(one process per core, one request per task) and on one thread.

--impl reference times the CPU oracle (float64) on the same metric on every
host core: one step is one draft position of oracle work per worker process.

--path lazy measures spec_verify_lazy on the same batch64-bf16 workload
(rows read only up to each request's first rejection); its roofline counts
the rows the walks actually read, averaged over 16 seeds.

--path tree measures spec_verify_tree instead, on tree222-bf16: B=64
requests, each a full [2, 2, 2] draft tree (14 nodes, 8 leaves) whose
children are independent draws from the drafter, V=128256 bf16; one step is
one tree verify of the batch, the metric counts the B*14 verified draft
nodes per step.

--path fcnorm measures spec_verify_fc_norm (EAGLE 3.1 LayerNorm fusion):
T=4096 tokens, three 4096-wide hidden states, a 4096 x 12288 bf16 FC weight
and bias; the metric is TFLOP/s of the FC (2 T 3d d_out per call), against
the measured bf16 tensor peak.

--path kv measures spec_verify_kv_commit (scratch mode): 32 layers x 64
sequences, 4 KB entries (8 KV heads x 128 dims x K and V in bf16), an
8-position window, the KV lengths of one batch64-bf16 verify; the metric is
the bytes the commit reads plus writes per second.
"""

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

METRIC = "verified draft positions/sec"
UNIT = "positions/s"
WORKLOAD = "batch64-bf16"
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC = os.path.join(ROOT, "profiles", "rowstats_traffic.json")
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--copies", type=int, default=3, help="rotating input copies in HBM")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-config and tree / KV / FC-norm measurements")
    ap.add_argument("--path", default="chain", choices=["chain", "lazy", "tree", "kv", "fcnorm"],
                    help="chain: spec_verify on batch64-bf16 (the headline); tree: "
                         "spec_verify_tree on tree222-bf16; kv: spec_verify_kv_commit; lazy: "
                         "spec_verify_lazy on batch64-bf16; fcnorm: spec_verify_fc_norm")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def ranks_max(value, device=None):
    """Max of a float over all ranks (the slowest rank's time); identity
    when torch.distributed is not initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step, steps, world, max_ms):
    """Units processed by all ranks divided by the slowest rank's time."""
    return units_per_rank_step * steps * world / (max_ms / 1e3)


def csrc_hash(files=("sv_device.cuh", "sv_internal.cuh", "sv_rowstats.cu", "sv_span.cuh")):
    """Hash of the row-statistics kernel's sources: the committed traffic
    figure is used only while these are unchanged."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "speculative_decoding_verification_73_gb300", "csrc")
    for f in files:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def hbm_peak():
    try:
        with open(PEAKS) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def traffic_per_launch():
    """DRAM bytes per row-statistics launch from the committed ncu summary, or
    None if the kernel sources changed since it was taken."""
    try:
        with open(TRAFFIC) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("csrc_hash") != csrc_hash():
        return None
    return t.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        self.t0 = time.time()

    def mark(self):
        return time.time()

    def stop(self, t_begin, t_end):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        # samples are 50 ms apart; attribute them to the timed region by order
        n = len(rows)
        span = max(time.time() - self.t0, 1e-9)
        sel = []
        for i, r in enumerate(rows):
            t = self.t0 + span * (i + 0.5) / max(n, 1)
            if t_begin - 0.05 <= t <= t_end + 0.05:
                sel.append(r)
        if not sel and rows:
            sel = rows[-max(1, n // 4):]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in sel if num(r[1]) is not None]
        mx = [num(r[2]) for r in sel if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in sel for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sel)}


# --------------------------------------------------------------------------- timing helpers

L2_FLUSH_BYTES = 256 << 20  # written before each call of a small workload (L2 is 129 MB)
PROFILE_CALLS = 256         # calls of the separate kernel-timing pass after the timed loop


def time_calls(stream, step, steps, warmup, flush=None):
    """Device time of each of `steps` calls of step(i), in microseconds: CUDA
    events on the launching stream around every call, each call preceded by a
    write of `flush` (a buffer larger than L2) when one is given, so the call
    reads its inputs from HBM and the host has queued it before it starts."""
    import torch
    for i in range(warmup):
        step(i)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(evs):
        if flush is not None:
            flush.fill_(i & 0xFF)
        a.record(stream)
        step(warmup + i)
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e3 for a, b in evs]


def kernel_pass(sv, step, calls, first):
    """Per-kernel device time of `calls` further calls with events around
    each kernel (the library's profiling hook), taken after the timed loop so
    the timed calls carry no events.  Returns ({kernel: us per call}, calls)."""
    from speculative_decoding_verification_73_gb300 import binding
    binding.spec_verify_profile_read(sv.ctx)  # clear
    binding.spec_verify_profile(sv.ctx, 1)
    for i in range(calls):
        step(first + i)
    ms, n = binding.spec_verify_profile_read(sv.ctx)
    binding.spec_verify_profile(sv.ctx, 0)
    return {k: v / max(n, 1) * 1e3 for k, v in ms.items()}, n


def direct_chain(lib, sv, wl, dev, copies=1, lazy=False):
    """step(i) that calls spec_verify (or spec_verify_lazy) through the C ABI
    with pointers prepared once, rotating over `copies` device copies of the
    inputs; also returns the output tensors."""
    import ctypes
    import torch
    from speculative_decoding_verification_73_gb300 import binding
    B, N, V = wl.shape
    target = [wl.target.to(dev) for _ in range(copies)]
    draft = [wl.draft.to(dev) for _ in range(copies)]
    tokens, temperature = wl.tokens.to(dev), wl.temperature.to(dev)
    out_t = sv.out_tokens[: B * (N + 1)].view(B, N + 1)
    out_a, out_k = sv.out_accept[:B], sv.out_kv[:B]
    P = ctypes.c_void_p
    ptrs = [(P(target[c].data_ptr()), P(draft[c].data_ptr())) for c in range(copies)]
    p_tok, p_temp = P(tokens.data_ptr()), P(temperature.data_ptr())
    p_ot, p_oa, p_ok = P(out_t.data_ptr()), P(out_a.data_ptr()), P(out_k.data_ptr())
    entry = lib.spec_verify_lazy if lazy else lib.spec_verify

    def step(i):
        zt, yt = ptrs[i % copies]
        rc = entry(sv.ctx, B, N, V, zt, yt, p_tok, p_temp, ctypes.c_uint64(i), p_ot, p_oa, p_ok)
        if rc != 0:
            raise binding.SpecVerifyError(rc, "spec_verify")

    bufs = {"target": target, "draft": draft, "tokens": tokens, "temperature": temperature,
            "out": (out_t, out_a, out_k)}
    return step, bufs


# --------------------------------------------------------------------------- oracle on the host
#
# The oracle, as it stands, timed on this machine's host cores: on one thread
# in this process and on a pool of one spawned process per core, each task
# one request (or one draft position) of a workload saved once to a temporary
# folder and memory-mapped by the workers.

def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


_POOL_DATA = {}
POOL_TIMEOUT_S = 600  # a pool that stops answering fails the run instead of hanging it


def _pool_rows(path):
    """A saved workload (metadata and memory-mapped arrays), loaded once per process."""
    if path not in _POOL_DATA:
        import numpy as np
        with open(os.path.join(path, "meta.json")) as f:
            meta = json.load(f)
        arrs = {k: np.load(os.path.join(path, k + ".npy"), mmap_mode="r") for k in ("z", "y", "d", "t")}
        _POOL_DATA[path] = (meta, arrs)
    return _POOL_DATA[path]


def _pool_warm(_):
    from oracle import verify  # noqa: F401  (import once per worker, outside the timing)
    return os.getpid()


def _pool_request(task):
    """The oracle on one whole request of a saved workload."""
    from oracle import verify as ov
    path, b, seed = task
    meta, a = _pool_rows(path)
    ov.verify_request(a["z"][b], a["y"][b], a["d"][b], float(a["t"][b]), seed, b, meta["dtype"])
    return 1


def _pool_position(task):
    """The oracle's work for draft position j (1-based) of request b, as it
    stands: widen the rows, then the argmax (T = 0) or both softmaxes, the
    Philox uniform and the accept test; at the request's last position also
    the residual of that row pair and its grouped draw (one draw per request)."""
    from oracle import philox as oph
    from oracle import verify as ov
    path, b, j, seed = task
    meta, a = _pool_rows(path)
    t = float(a["t"][b])
    zr = ov.logits_to_f64(a["z"][b, j - 1], meta["dtype"])
    if t == 0.0:
        ov.argmax_lowest(zr)
        return 1
    d = int(a["d"][b, j - 1])
    q = ov.softmax(zr, t)
    p = ov.softmax(ov.logits_to_f64(a["y"][b, j - 1], meta["dtype"]), t)
    ov.accept(q[d], p[d], oph.uniform(seed, b, j, oph.ACCEPT_DRAW))
    if j == meta["N"]:
        ov.sample_grouped(ov.residual(q, p), oph.uniforms4(seed, b, j, oph.SAMPLE_DRAW))
    return 1


class OracleHost:
    """Saved workloads plus a process pool for timing the oracle."""

    def __init__(self):
        self.dir = tempfile.mkdtemp(prefix="sv_oracle_")
        self.cores = host_cores()
        self.pool = None

    def start(self):
        """Spawn one worker per core (spawned, not forked: safe whatever this
        process has initialised) and wait until every one has imported the
        oracle."""
        import concurrent.futures
        import multiprocessing
        self.pool = concurrent.futures.ProcessPoolExecutor(
            max_workers=self.cores, mp_context=multiprocessing.get_context("spawn"))
        list(self.pool.map(_pool_warm, range(4 * self.cores), timeout=POOL_TIMEOUT_S))

    def save(self, name, wl):
        import numpy as np
        path = os.path.join(self.dir, name)
        os.makedirs(path, exist_ok=True)
        z, y = wl.raw()
        for k, arr in (("z", z), ("y", y), ("d", wl.tokens.numpy()), ("t", wl.temperature.numpy())):
            np.save(os.path.join(path, k + ".npy"), np.ascontiguousarray(arr))
        B, N, V = wl.shape
        with open(os.path.join(path, "meta.json"), "w") as f:
            json.dump({"dtype": wl.dtype, "B": B, "N": N, "V": V, "seed": int(wl.seed)}, f)
        return path

    def time_requests(self, name, wl, budget_s=1.5):
        """Positions per second of the oracle on whole requests of `wl`: one
        thread, then every core.  Each figure runs for about budget_s."""
        path = self.save(name, wl)
        B, N, _ = wl.shape
        seed = int(wl.seed)
        _pool_request((path, 0, seed))  # load the arrays here, outside the timing
        done, t0 = 0, time.perf_counter()
        while done == 0 or time.perf_counter() - t0 < budget_s:
            _pool_request((path, done % B, seed))
            done += 1
        el1 = time.perf_counter() - t0
        rate1 = done / el1
        out = {"single_thread": {"value": rate1 * N, "unit": UNIT, "cores": 1,
                                 "sample": f"{done} requests in {el1:.2f} s"}}
        if self.pool is not None:
            list(self.pool.map(_pool_request, [(path, b % B, seed) for b in range(self.cores)],
                               timeout=POOL_TIMEOUT_S))
            m = max(self.cores, int(round(rate1 * self.cores * budget_s)))
            t0 = time.perf_counter()
            list(self.pool.map(_pool_request, [(path, b % B, seed) for b in range(m)], chunksize=1,
                               timeout=POOL_TIMEOUT_S))
            el = time.perf_counter() - t0
            out.update({"value": m * N / el, "unit": UNIT, "cores": self.cores,
                        "sample": f"{m} requests (request i = i mod {B}) over {self.cores} "
                                  f"processes in {el:.2f} s"})
        return out

    def close(self):
        if self.pool is not None:
            self.pool.shutdown(wait=True, cancel_futures=True)
            self.pool = None
        import shutil
        shutil.rmtree(self.dir, ignore_errors=True)


# --------------------------------------------------------------------------- ours: the chain

# The other configurations of the method statement, each timed alone after
# the headline: (name, builder, what bounds one call).
def per_config_builders():
    from speculative_decoding_verification_73_gb300 import workloads
    return (
        ("tiny-f32", workloads.tiny_f32, "latency"),
        ("single-bf16-T1", lambda: workloads.single_bf16(1.0), "latency"),
        ("single-bf16-T0", lambda: workloads.single_bf16(0.0), "latency"),
        ("mixture-bf16", workloads.mixture_bf16, "hbm"),
        ("alpha09-f32", lambda: workloads.Alpha09().workload(0), "hbm"),
    )


def measure_config(lib, wl, dev, stream, bound, peak, steps=200, warmup=10):
    """One configuration: median device time per spec_verify call with an L2
    flush before every call, positions per second, and for a bandwidth-bound
    one the algorithmic bytes per second as a fraction of the HBM peak."""
    import statistics as st
    import torch
    from speculative_decoding_verification_73_gb300 import binding
    B, N, V = wl.shape
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    sv = binding.SpecVerify(B, max(N, 1), V, dt, stream=stream, device=dev)
    step, _ = direct_chain(lib, sv, wl, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    us = time_calls(stream, step, steps, warmup, flush)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    kern, _ = kernel_pass(sv, step, 64, warmup + steps)
    sv.close()
    med = st.median(us)
    nbytes = wl.bytes_read()
    gbs = nbytes / (med * 1e-6) / 1e9
    return {
        "B": B, "N": N, "V": V, "logits": wl.dtype,
        "us_per_step": med, "us_per_step_mean": st.fmean(us), "steps": steps,
        "positions_per_s": B * N / (med * 1e-6),
        "bytes_read_per_step": nbytes, "gb_per_s": gbs,
        "bound": bound, "hbm_frac": gbs / peak if bound == "hbm" else None,
        "kernel_us": ({"verify": kern["k0"]} if binding.spec_verify_launches_per_call() == 1
                      else {"rowstats": kern["k0"], "sample": kern["k1"]}),
        "l2": f"flushed before every call ({L2_FLUSH_BYTES >> 20} MB write)",
    }


def run_ours(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_73_gb300 import binding, build, workloads

    world, rank, local = dist_env()
    extras = world == 1 and not args.no_extras
    host = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = OracleHost()
        host.start()  # before any CUDA work
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    dev = torch.device("cuda", local)
    lib = binding.load()

    lazy = args.path == "lazy"
    wl = workloads.batch64_bf16(verify_seed=rank)
    B, N, V = wl.shape
    copies = max(1, args.copies)
    stream = torch.cuda.current_stream(dev)
    sv = binding.SpecVerify(B, N, V, torch.bfloat16, stream=stream, device=dev)
    step, bufs = direct_chain(lib, sv, wl, dev, copies, lazy)
    out_t, out_a, out_k = bufs["out"]

    for i in range(args.warmup):
        step(i)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    if world > 1:
        dist.barrier()
    elapsed_ms = ev0.elapsed_time(ev1)
    time.sleep(0.2)
    clk = clocks.stop(t_begin, t_end)
    elapsed_ms = ranks_max(elapsed_ms, dev)
    value = whole_job_rate(B * N, args.steps, world, elapsed_ms)

    # per-kernel device times from a separate pass after the timed loop
    kern, prof_calls = kernel_pass(sv, step, PROFILE_CALLS, args.warmup + args.steps)
    launches = 1 if lazy else binding.spec_verify_launches_per_call()
    names = ("lazy",) if lazy else ("verify",) if launches == 1 else ("rowstats", "sample")
    kernel_us = {n: kern[f"k{i}"] for i, n in enumerate(names)}
    first_kernel = names[0]
    rowstats_us = kernel_us[first_kernel]
    if lazy:
        bytes_per_launch = lazy_bytes(wl, sv, step, out_a)
        reread = 0
    else:
        # the rows streamed once, plus (one kernel doing both) the row pair or
        # bonus row each sampled request's draw reads again
        reread = reread_bytes(wl, step, out_a) if launches == 1 else 0
        bytes_per_launch = wl.bytes_read() + reread
    achieved = bytes_per_launch / (rowstats_us * 1e-6) / 1e9
    peak, peak_kind = hbm_peak()

    e2e = e2e_chain(sv, wl, bufs, dev, stream, copies, lazy, args, world)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 logits, f32 accumulate",
        "data": "synthetic (seeded Zipf logits, Gaussian draft noise)",
        "config": {
            "workload": WORKLOAD + ("-lazy" if lazy else ""), "B": B, "N": N, "V": V, "logits": "bf16",
            "temperatures": "per request from {0, 0.7, 1.0}",
            "sampled_requests": int((wl.temperature > 0).sum()),
            "bytes_read_per_step": bytes_per_launch,
            "reread_bytes_per_step": reread,
            "l2": f"inputs larger than L2: {bytes_per_launch / 1e6:.0f} MB read per step, "
                  f"{copies} rotating copies",
            "parallelism": f"replicas x{world} (requests shard, no collective)",
        },
        "roofline": {
            "bound": "hbm", "kernel": first_kernel, "achieved": achieved, "peak": peak,
            "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s", "frac": achieved / peak,
            "traffic": None if lazy else traffic_per_launch(),
            "algorithmic_bytes_per_launch": bytes_per_launch,
            "avg_launch_us": rowstats_us,
            "timed_launches": f"{prof_calls} calls after the timed loop, events around each kernel",
        },
        "kernel_us_per_step": kernel_us,
        "e2e": e2e,
        "gpu_launches": args.steps * launches,
        "clocks": clk,
    }
    if extras and not lazy:
        rp = read_stream_peak(dev, stream, bytes_per_launch)
        line["roofline"]["read_peak"] = rp
        line["roofline"]["frac_of_read_peak"] = achieved / rp["gb_per_s"]
        line["roofline"]["frac_of_read_at_step_bytes"] = achieved / rp["at_step_bytes"]["gb_per_s"]
        per = {WORKLOAD: {"B": B, "N": N, "V": V, "logits": "bf16",
                          "us_per_step": elapsed_ms / args.steps * 1e3, "steps": args.steps,
                          "positions_per_s": value, "bytes_read_per_step": bytes_per_launch,
                          "gb_per_s": bytes_per_launch / (elapsed_ms / args.steps * 1e-3) / 1e9,
                          "bound": "hbm",
                          "hbm_frac": bytes_per_launch / (elapsed_ms / args.steps * 1e-3) / 1e9 / peak,
                          "kernel_us": kernel_us, "l2": line["config"]["l2"]}}
        cfg_wls = {}
        for name, make, bound in per_config_builders():
            cfg_wls[name] = make()
            per[name] = measure_config(lib, cfg_wls[name], dev, stream, bound, peak)
        line["per_config"] = per
        line["rows_f"] = {
            "tree": tree_summary(dev, stream, peak),
            "kv_commit": kv_summary(dev, stream, peak),
            "fc_norm": fcnorm_summary(dev, stream),
            "lazy": lazy_summary(lib, dev, stream),
        }
    sv.close()
    if host is not None:
        line["cpu_baseline"] = dict(kind="oracle", **host.time_requests(WORKLOAD, wl, budget_s=6.0))
        if extras and not lazy:
            for name, cwl in cfg_wls.items():
                line["per_config"][name]["oracle"] = host.time_requests(name, cwl)
            line["per_config"][WORKLOAD]["oracle"] = {
                k: line["cpu_baseline"][k] for k in ("value", "unit", "cores", "sample", "single_thread")}
        host.close()
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def e2e_chain(sv, wl, bufs, dev, stream, copies, lazy, args, world):
    """The same metric end to end through the public API with host buffers:
    every step copies its inputs from pinned host memory and reads its
    outputs back.  Double-buffered: step i's inputs are copied on a copy
    stream into buffer i % 2 while the verify stream still runs step i - 1;
    the verify of step i waits for its copy, and a copy into a buffer waits
    for the verify that last read it.  Every copy and read-back is timed."""
    import torch
    from speculative_decoding_verification_73_gb300 import binding
    B, N, V = wl.shape
    out_t, out_a, out_k = bufs["out"]
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 200))
    h_target = wl.target.pin_memory()
    h_draft = wl.draft.pin_memory()
    h_tokens = wl.tokens.pin_memory()
    h_temp = wl.temperature.pin_memory()
    h_out_t = torch.empty(B, N + 1, dtype=torch.int32).pin_memory()
    h_out_a = torch.empty(B, dtype=torch.int32).pin_memory()
    h_out_k = torch.empty(B, dtype=torch.int32).pin_memory()
    target, draft = bufs["target"], bufs["draft"]
    tokens, temperature = bufs["tokens"], bufs["temperature"]
    dbufs = [(target[c % copies], draft[c % copies], torch.empty_like(tokens), torch.empty_like(temperature))
             for c in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (h_target, h_draft, h_tokens, h_temp))
    d2h = sum(t.numel() * t.element_size() for t in (h_out_t, h_out_a, h_out_k))
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        zb, yb, tb, pb = dbufs[i % 2]
        copy_stream.wait_event(consumed[i % 2])  # the verify two steps back is done with it
        with torch.cuda.stream(copy_stream):
            zb.copy_(h_target, non_blocking=True)
            yb.copy_(h_draft, non_blocking=True)
            tb.copy_(h_tokens, non_blocking=True)
            pb.copy_(h_temp, non_blocking=True)
        copied[i % 2].record(copy_stream)
        stream.wait_event(copied[i % 2])
        (binding.spec_verify_lazy if lazy else binding.spec_verify)(
            sv.ctx, zb, yb, tb, pb, i, out_t, out_a, out_k)
        consumed[i % 2].record(stream)
        h_out_t.copy_(out_t, non_blocking=True)
        h_out_a.copy_(out_a, non_blocking=True)
        h_out_k.copy_(out_k, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    copy_stream.wait_event(ev0)  # no copy of the timed steps starts before the clock
    for i in range(e2e_steps):
        e2e_step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = ranks_max(ev0.elapsed_time(ev1), dev)
    return {"value": whole_job_rate(B * N, e2e_steps, world, e2e_ms), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps}


def reread_bytes(wl, step, out_a, seeds=16):
    """Logit bytes the draws read a second time, averaged over `seeds` calls:
    the target and draft row at the first rejection (two rows) or the bonus
    row (one) of every sampled request."""
    import torch
    B, N, V = wl.shape
    esize = wl.target.element_size()
    sampled = wl.temperature.numpy() > 0
    total = 0
    for s in range(seeds):
        step(s)
        torch.cuda.synchronize()
        acc = out_a.cpu().numpy()
        total += sum((2 if a < N else 1) for a, smp in zip(acc, sampled) if smp and a >= 0)
    return total * V * esize // seeds


def lazy_bytes(wl, sv, step, out_a):
    """Logit bytes the lazy walks read, averaged over 16 seeds: per request
    the target rows up to its stop and, when sampled, the draft rows it
    tested plus the re-read of the row (pair) the final token is drawn from."""
    import torch
    B, N, V = wl.shape
    esize = wl.target.element_size()
    temps = wl.temperature.numpy()
    total = 0
    for s in range(16):
        step(s)
        torch.cuda.synchronize()
        acc = out_a.cpu().numpy()
        rows = 0
        for b in range(B):
            a = int(acc[b])
            if a < 0:
                continue
            rows += a + 1                                   # target rows 0..a
            if temps[b] > 0:
                rows += min(a + 1, N)                       # draft rows tested
                rows += 2 if a < N else 1                   # residual pair / bonus row re-read
        total += rows * V * esize
    return total // 16


# --------------------------------------------------------------------------- tree

TREE_WORKLOAD = "tree222-bf16"


def tree222(verify_seed=0):
    from speculative_decoding_verification_73_gb300 import workloads
    return workloads.make_tree(64, 128256, "bf16", gen_seed=1006, widths=(2, 2, 2),
                               verify_seed=verify_seed, name=TREE_WORKLOAD)


def tree_setup(dev, stream, wl, copies, lazy=False):
    import torch
    from speculative_decoding_verification_73_gb300 import binding
    B, M, V = wl.shape
    target = [wl.target.to(dev) for _ in range(copies)]
    draft = [wl.draft.to(dev) for _ in range(copies)]
    parents, tokens = wl.parents.to(dev), wl.tokens.to(dev)
    temperature = wl.temperature.to(dev)
    sv = binding.SpecVerify(B, M, V, torch.bfloat16, stream=stream, device=dev)
    outs = (sv.out_tokens[: B * (M + 1)].view(B, M + 1), sv.out_path[: B * M].view(B, M),
            sv.out_accept[:B], sv.out_kv[:B])

    def step(i, c=None):
        c = i % copies if c is None else c
        binding.spec_verify_tree(sv.ctx, wl.mode, target[c], draft[c], parents, tokens, temperature,
                                 i, *outs, lazy=lazy)

    return sv, step, (target, draft, parents, tokens, temperature), outs


def tree_lazy_bytes(wl, outs, step, seeds=8):
    """Bytes the lazy tree walk reads per call, averaged over `seeds` calls:
    the target row of every node on each request's walked path (root, then
    the accepted nodes) and, for a sampled request, the draft row of each of
    those nodes that has children."""
    from speculative_decoding_verification_73_gb300 import binding
    B, M, V = wl.shape
    par = wl.parents.numpy()
    inner = [set(int(v) for v in par[b]) for b in range(B)]  # nodes that have children
    temp = wl.temperature.numpy()
    row = V * wl.target.element_size()
    total = 0
    for i in range(seeds):
        step(i, 0)
        path, acc = outs[1].cpu().numpy(), outs[2].cpu().numpy()
        for b in range(B):
            nodes = [0] + [int(n) for n in path[b, : max(int(acc[b]), 0)]]
            total += len(nodes) * row
            if temp[b] > 0 and wl.mode == binding.SV_TREE_SAMPLED:
                total += sum(1 for n in nodes if n in inner[b]) * row
    return total // seeds


def tree_lazy_summary(dev, stream, steps=200, warmup=10, copies=3):
    """spec_verify_tree_lazy on tree222-bf16: device time per call (three
    rotating input copies, so rows come from HBM), verified nodes per second
    and the bytes its walks read."""
    import torch
    from speculative_decoding_verification_73_gb300 import binding
    wl = tree222()
    B, M, V = wl.shape
    sv, step, _, outs = tree_setup(dev, stream, wl, copies, lazy=True)
    nbytes = tree_lazy_bytes(wl, outs, step)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    us = ev0.elapsed_time(ev1) / steps * 1e3
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    sv.close()
    return {"workload": TREE_WORKLOAD, "us_per_step": us, "steps": steps,
            "verified_nodes_per_s": B * M / (us * 1e-6), "bytes_read_per_step": nbytes,
            "launches": 1, "l2": f"{copies} rotating input copies of {wl.bytes_read() / 1e6:.0f} MB"}


def tree_summary(dev, stream, peak, steps=200, warmup=10):
    """spec_verify_tree on tree222-bf16: device time per call, verified nodes
    per second, and tree_rowstats' bandwidth against the HBM peak."""
    import torch
    from speculative_decoding_verification_73_gb300 import binding
    wl = tree222()
    B, M, V = wl.shape
    sv, step, _, _ = tree_setup(dev, stream, wl, 1)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    us = ev0.elapsed_time(ev1) / steps * 1e3
    kern, _ = kernel_pass(sv, step, 64, warmup + steps)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    sv.close()
    nbytes = wl.bytes_read()
    rs = kern["k0"]
    return {"workload": TREE_WORKLOAD, "B": B, "M": M, "V": V, "us_per_step": us, "steps": steps,
            "verified_nodes_per_s": B * M / (us * 1e-6), "bytes_read_per_step": nbytes,
            "kernel_us": {"tree_rowstats": rs, "tree_walk": kern["k1"]},
            "roofline": {"kernel": "tree_rowstats", "achieved_gbs": nbytes / (rs * 1e-6) / 1e9,
                         "frac": nbytes / (rs * 1e-6) / 1e9 / peak},
            "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB per call)",
            "lazy": tree_lazy_summary(dev, stream)}


def run_tree(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_73_gb300 import binding, build

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    wl = tree222(verify_seed=rank)
    B, M, V = wl.shape
    copies = max(1, args.copies)
    sv, step, dev_in, outs = tree_setup(dev, stream, wl, copies)
    target, draft, parents, tokens, temperature = dev_in
    out_t, out_p, out_a, out_k = outs

    for i in range(args.warmup):
        step(i)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    if world > 1:
        dist.barrier()
    elapsed_ms = ranks_max(ev0.elapsed_time(ev1), dev)
    time.sleep(0.2)
    clk = clocks.stop(t_begin, t_end)
    kernel_us, calls = kernel_pass(sv, step, PROFILE_CALLS, args.warmup + args.steps)
    value = whole_job_rate(B * M, args.steps, world, elapsed_ms)
    bytes_per_launch = wl.bytes_read()
    rs_us = kernel_us["k0"]
    achieved = bytes_per_launch / (rs_us * 1e-6) / 1e9
    peak, peak_kind = hbm_peak()

    # end to end with pinned host buffers, through the Python binding;
    # double-buffered like the chain's (copies of step i on a copy stream
    # while the tree verify of step i - 1 runs)
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 200))
    hs = [t.pin_memory() for t in (wl.target, wl.draft, wl.parents, wl.tokens, wl.temperature)]
    dbufs = [[target[c % copies], draft[c % copies], torch.empty_like(parents), torch.empty_like(tokens),
              torch.empty_like(temperature)] for c in range(2)]
    hout = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (out_t, out_p, out_a, out_k)]
    h2d = sum(t.numel() * t.element_size() for t in hs)
    d2h = sum(t.numel() * t.element_size() for t in hout)
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        ds = dbufs[i % 2]
        copy_stream.wait_event(consumed[i % 2])  # the verify two steps back is done with it
        with torch.cuda.stream(copy_stream):
            for h, d in zip(hs, ds):
                d.copy_(h, non_blocking=True)
        copied[i % 2].record(copy_stream)
        stream.wait_event(copied[i % 2])
        binding.spec_verify_tree(sv.ctx, wl.mode, ds[0], ds[1], ds[2], ds[3], ds[4], i,
                                 out_t, out_p, out_a, out_k)
        consumed[i % 2].record(stream)
        for h, d in zip(hout, (out_t, out_p, out_a, out_k)):
            h.copy_(d, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    copy_stream.wait_event(ev0)  # no copy of the timed steps starts before the clock
    for i in range(e2e_steps):
        e2e_step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_value = whole_job_rate(B * M, e2e_steps, world, ranks_max(ev0.elapsed_time(ev1), dev))
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 logits, f32 accumulate",
        "data": "synthetic (seeded Zipf logits, Gaussian draft noise, children drawn from the drafter)",
        "config": {
            "workload": TREE_WORKLOAD, "B": B, "tree": "[2, 2, 2] (14 draft nodes, 8 leaves)",
            "M": M, "V": V, "logits": "bf16", "drafting": "independent draws (SV_TREE_SAMPLED)",
            "temperatures": "per request from {0, 0.7, 1.0}",
            "bytes_read_per_step": bytes_per_launch,
            "l2": f"inputs larger than L2: {bytes_per_launch / 1e6:.0f} MB read per step, "
                  f"{copies} rotating copies",
            "parallelism": f"replicas x{world} (requests shard, no collective)",
        },
        "roofline": {
            "bound": "hbm", "kernel": "tree_rowstats", "achieved": achieved, "peak": peak,
            "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s", "frac": achieved / peak,
            "traffic": None, "algorithmic_bytes_per_launch": bytes_per_launch,
            "avg_launch_us": rs_us,
            "timed_launches": f"{calls} calls after the timed loop, events around each kernel",
        },
        "kernel_us_per_step": {("tree_rowstats" if k == "k0" else "tree_walk"): v
                               for k, v in kernel_us.items()},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps * 2,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = tree_cpu_baseline(wl, budget_s=12.0)
    sv.close()
    if world == 1:
        line["lazy"] = tree_lazy_summary(dev, stream)
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


def tree_cpu_baseline(wl, budget_s):
    from oracle import tree as ot
    B, M, _ = wl.shape
    z, y = wl.raw()
    par, tok, t = wl.parents.numpy(), wl.tokens.numpy(), wl.temperature.numpy()
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        b = done % B
        ot.verify_request(z[b], y[b], par[b], tok[b], t[b], wl.seed, b, wl.dtype, wl.mode)
        done += 1
    el = time.perf_counter() - t0
    return {"value": done * M / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} requests of {TREE_WORKLOAD} (request i = i mod {B}), {el:.1f} s, "
                      f"float64 numpy on 1 host thread"}


# --------------------------------------------------------------------------- kv commit

KV_WORKLOAD = "kvcommit-32L-64seq-4KB"
KV_LAUNCHES_PER_COMMIT = 2


def kv_setup(dev, stream, copies, rank=0):
    """32 layers x 64 sequences x 4 KB entries, an 8-position window, the KV
    lengths of one batch64-bf16 verify; step(i) commits window copy i % copies."""
    import torch
    from speculative_decoding_verification_73_gb300 import binding, workloads
    wl = workloads.batch64_bf16(verify_seed=rank)
    B, N, V = wl.shape
    sv = binding.SpecVerify(B, N, V, torch.bfloat16, stream=stream, device=dev)
    _, _, kv = sv(wl.target.to(dev), wl.draft.to(dev), wl.tokens.to(dev), wl.temperature.to(dev), 0)
    kv = kv.clone()
    L, E, W, S = 32, 4096, N + 1, 1024
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    scratch = [torch.randint(0, 256, (L, B, W, E), generator=gen, dtype=torch.uint8, device=dev)
               for _ in range(copies)]
    cache = torch.zeros(L, B, S, E, dtype=torch.uint8, device=dev)
    # lengths start below 200 and grow by at most W per commit: reset every 100 commits
    seq0 = torch.randint(0, 200, (B,), generator=gen, dtype=torch.int32, device=dev)
    seq = seq0.clone()
    kv_host = kv.cpu().numpy()
    moved = int(sum(2 * max(int(n), 0) for n in kv_host)) * E * L

    def step(i):
        if i % 100 == 0:
            seq.copy_(seq0)
        binding.spec_verify_kv_commit(sv.ctx, binding.SV_KV_SCRATCH, cache, seq, kv,
                                      scratch=scratch[i % copies])

    shape = {"layers": L, "B": B, "entry_bytes": E, "window": W, "cache_positions": S,
             "kv_len_sum": int(sum(max(int(n), 0) for n in kv_host)),
             "l2": f"{copies} rotating scratch windows of {L * B * W * E / 1e6:.0f} MB"}
    return sv, step, moved, shape


def read_stream_peak(dev, stream, step_bytes, big=4 << 30):
    """The achievable streaming-read bandwidth on this GPU, by the library's
    read-stream hook (one plain read kernel per call): on a 4 GiB buffer
    (median of 10 single reads), and on buffers of the step's own size
    (3 rotating copies larger than L2 together, 300 back-to-back reads, the
    way the row statistics are timed), which carries the same fixed launch,
    ramp and drain cost per launch."""
    import torch
    from speculative_decoding_verification_73_gb300 import binding
    out = torch.zeros(1, dtype=torch.int64, device=dev)

    def timed(bufs, reps):
        for i in range(3):
            binding.spec_verify_debug_read_stream(bufs[i % len(bufs)], out, stream)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(reps):
            binding.spec_verify_debug_read_stream(bufs[i % len(bufs)], out, stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    buf = torch.ones(big, dtype=torch.uint8, device=dev)
    ms_big = statistics.median(timed([buf], 1) for _ in range(10))
    del buf
    n = step_bytes // 16 * 16
    bufs = [torch.ones(n, dtype=torch.uint8, device=dev) for _ in range(3)]
    ms_step = timed(bufs, 300)
    del bufs
    return {"gb_per_s": big / (ms_big * 1e-3) / 1e9, "bytes": big,
            "at_step_bytes": {"gb_per_s": n / (ms_step * 1e-3) / 1e9, "us": ms_step * 1e3, "bytes": n},
            "kernel": "spec_verify_debug_read_stream (8 CTAs per SM, 16-byte non-allocating loads)",
            "note": "context for the roofline; 'peak' stays the measured copy bandwidth"}


LAZY_WORKLOADS = ("batch64-bf16", "lowaccept64-bf16")


def lazy_summary(lib, dev, stream, steps=300, warmup=20):
    """spec_verify against spec_verify_lazy per step on batch64-bf16 and on
    lowaccept64-bf16 (drafter far from the target), three rotating input
    copies; the lazy walk reads rows only up to each request's first
    rejection, so it pays when few drafts are accepted."""
    import torch
    from speculative_decoding_verification_73_gb300 import binding, workloads
    res = {}
    for name in LAZY_WORKLOADS:
        wl = workloads.batch64_bf16() if name == "batch64-bf16" else workloads.low_accept_bf16()
        B, N, V = wl.shape
        sv = binding.SpecVerify(B, N, V, torch.bfloat16, stream=stream, device=dev)
        entry = {}
        for lazy in (False, True):
            step, bufs = direct_chain(lib, sv, wl, dev, copies=3, lazy=lazy)
            for i in range(warmup):
                step(i)
            torch.cuda.synchronize(dev)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for i in range(steps):
                step(warmup + i)
            ev1.record(stream)
            torch.cuda.synchronize(dev)
            entry["lazy_us_per_step" if lazy else "eager_us_per_step"] = ev0.elapsed_time(ev1) / steps * 1e3
            entry["mean_accepted"] = float(bufs["out"][1].float().mean())
            del bufs
        code, _ = sv.get_error()
        assert code == 0, binding.strerror(code)
        sv.close()
        entry.update(B=B, N=N, V=V, steps=steps)
        res[name] = entry
    return res


def kv_summary(dev, stream, peak, steps=500, warmup=20):
    import torch
    from speculative_decoding_verification_73_gb300 import binding
    sv, step, moved, shape = kv_setup(dev, stream, copies=3)
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(warmup + i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    us = ev0.elapsed_time(ev1) / steps * 1e3
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    sv.close()
    gbs = moved / (us * 1e-6) / 1e9
    return dict(workload=KV_WORKLOAD, us_per_commit=us, steps=steps, bytes_moved_per_commit=moved,
                gb_per_s=gbs, hbm_frac=gbs / peak, **shape)


def run_kv(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_73_gb300 import binding, build

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    copies = max(1, args.copies)
    sv, step, moved, shape = kv_setup(dev, stream, copies, rank)
    for i in range(args.warmup):
        step(i)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    ev0.record(stream)
    for i in range(args.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    if world > 1:
        dist.barrier()
    elapsed_ms = ranks_max(ev0.elapsed_time(ev1), dev)
    k_ms = elapsed_ms / args.steps  # the commit's launches are the whole step
    time.sleep(0.2)
    clk = clocks.stop(t_begin, t_end)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    peak, peak_kind = hbm_peak()
    value = moved * args.steps * world / (elapsed_ms / 1e3) / 1e9
    achieved = moved / (k_ms / 1e3) / 1e9
    line = {
        "metric": "KV commit bytes moved/sec", "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
        "data": "synthetic (random KV bytes; KV lengths from one batch64-bf16 verify)",
        "config": dict(workload=KV_WORKLOAD, mode="scratch", bytes_moved_per_step=moved,
                       parallelism=f"replicas x{world}", **shape),
        "roofline": {"bound": "hbm", "kernel": "kv_commit", "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": moved, "avg_launch_us": k_ms * 1e3,
                     "timed_launches": f"all {args.steps} commits of the timed loop (one length "
                                       f"reset per 100 commits)"},
        "e2e": None,
        "gpu_launches": args.steps * KV_LAUNCHES_PER_COMMIT,
        "clocks": clk,
    }
    sv.close()
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


# --------------------------------------------------------------------------- fc norm

FC_WORKLOAD = "fcnorm-T4096-d4096-o4096-layernorm"


def bf16_peak():
    try:
        with open(PEAKS) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def fcnorm_setup(dev, stream, rank=0, norm="layernorm"):
    """FC-norm at T = d = d_out = 4096; norm "layernorm" (the workload the
    row is measured on) or "none" (EAGLE-3's plain concatenation: the GEMM
    reads the hidden states directly)."""
    import torch
    from speculative_decoding_verification_73_gb300 import binding, workloads
    T, d, d_out = 4096, 4096, 4096
    wl = workloads.make_fcnorm(T, d, d_out, gen_seed=2026 + rank, name=FC_WORKLOAD)
    h = [x.to(dev) for x in wl.h]
    w, g, b, bias = wl.weight.to(dev), wl.gamma.to(dev), wl.beta.to(dev), wl.bias.to(dev)
    out = torch.empty(T, d_out, dtype=torch.bfloat16, device=dev)
    xbuf = torch.empty(T, 3 * d, dtype=torch.bfloat16, device=dev)
    sv = binding.SpecVerify(1, 1, 16, torch.float32, stream=stream, device=dev)

    layer = norm == "layernorm"

    def step(i=0):
        binding.spec_verify_fc_norm(sv.ctx, binding.SV_NORM_LAYER if layer else binding.SV_NORM_NONE, *h, w,
                                    gamma=g if layer else None, beta=b if layer else None, bias=bias,
                                    out=out, xbuf=xbuf)

    return sv, step, 2.0 * T * 3 * d * d_out, {"T": T, "d": d, "d_out": d_out, "norm": norm}


def fcnorm_summary(dev, stream, steps=30, warmup=3):
    import torch
    from speculative_decoding_verification_73_gb300 import binding
    peak, kind = bf16_peak()
    res = {}
    for norm in ("layernorm", "none"):
        sv, step, flops, shape = fcnorm_setup(dev, stream, norm=norm)
        for _ in range(warmup):
            step()
        torch.cuda.synchronize(dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        us = ev0.elapsed_time(ev1) / steps * 1e3
        code, _ = sv.get_error()
        assert code == 0, binding.strerror(code)
        sv.close()
        tf = flops / (us * 1e-6) / 1e12
        if norm == "layernorm":
            res = dict(workload=FC_WORKLOAD, us_per_call=us, steps=steps, flops_per_call=flops, tflops=tf,
                       tensor_frac=tf / peak, peak_kind=f"{kind} cuBLAS bf16 burst", **shape)
        else:
            res["norm_none"] = dict(us_per_call=us, tflops=tf, tensor_frac=tf / peak,
                                    launches=1, note="the GEMM alone, reading the three hidden states")
    return res


def run_fcnorm(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_73_gb300 import binding, build

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    sv, step, flops, shape = fcnorm_setup(dev, stream, rank)
    for _ in range(max(args.warmup, 3)):
        step()
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    steps = min(args.steps, 500)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    elapsed_ms = ranks_max(ev0.elapsed_time(ev1), dev)
    time.sleep(0.2)
    clk = clocks.stop(t_begin, t_end)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    per_ms = elapsed_ms / steps
    value = flops * steps * world / (elapsed_ms / 1e3) / 1e12
    peak, kind = bf16_peak()
    achieved = flops / (per_ms / 1e3) / 1e12
    line = {
        "metric": "FC-norm TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": per_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate",
        "data": "synthetic (Gaussian hidden states of three magnitudes, random weights)",
        "config": dict(workload=FC_WORKLOAD, flops_per_call=flops, parallelism=f"replicas x{world}",
                       **shape),
        "roofline": {"bound": "tensor", "kernel": "fc_gemm (+ fcnorm_prep)", "achieved": achieved,
                     "peak": peak, "peak_kind": f"{kind} cuBLAS bf16 burst", "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "algorithmic_flops_per_launch": flops, "avg_launch_us": per_ms * 1e3,
                     "timed_launches": f"{steps} calls of two launches each"},
        "e2e": None, "gpu_launches": steps * 2, "clocks": clk,
    }
    sv.close()
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


# --------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The oracle, as it stands, on this machine's host cores: one step is
    one draft position of batch64-bf16 per worker process (positions taken
    request-major, rotating over all B x N), all workers at once."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_73_gb300 import workloads
    host = OracleHost()
    host.start()
    wl = workloads.batch64_bf16()
    B, N, V = wl.shape
    path = host.save(WORKLOAD, wl)
    seed, cores = int(wl.seed), host.cores

    def step(i):
        ks = [(i * cores + c) % (B * N) for c in range(cores)]
        list(host.pool.map(_pool_position, [(path, k // N, k % N + 1, seed) for k in ks],
                           timeout=POOL_TIMEOUT_S))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    host.close()
    value = args.steps * cores / el
    sample = (f"{cores} draft positions of {WORKLOAD} per step, one per process (positions taken "
              f"request-major, rotating over all {B * N}; greedy positions cost an argmax, sampled "
              f"ones two softmaxes, the accept test and, at a request's last position, the residual "
              f"draw), float64 numpy")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "N": N, "V": V, "logits": "bf16"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.path == "tree":
        run_tree(args)
    elif args.path == "kv":
        run_kv(args)
    elif args.path == "fcnorm":
        run_fcnorm(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
