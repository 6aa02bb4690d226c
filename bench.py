"""Benchmark of the batched draft-verify step on the batch64-bf16 workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload: B=64 requests, N=7 drafts, V=128256 vocabulary, bf16 logits,
per-request draft noise sigma ~ U[0.2, 1.5] and temperature from
{0, 0.7, 1.0} (synthetic, seeded).  One step = one spec_verify call over the
whole batch (row statistics, walk, residual/bonus sampling).

Metric: verified draft positions per second (B*N per step), plus the
achieved HBM bandwidth of the row-statistics kernel against the measured
copy bandwidth of the GPU.  Under torchrun each rank verifies its own batch
(weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the slowest rank's time is used.

--impl reference times the CPU oracle (float64, one host thread) on the same
metric, one draft position of oracle work per step.

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
# Kernel durations come from CUDA events the library records around each
# kernel of every PROFILE_EVERY-th call of the timed loop; events between the
# two kernels stop them from overlapping, so only a sample of calls carry them.
PROFILE_EVERY = 16
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


# --------------------------------------------------------------------------- ours

def run_ours(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_73_gb300 import binding, build, workloads

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    dev = torch.device("cuda", local)

    wl = workloads.batch64_bf16(verify_seed=rank)
    B, N, V = wl.shape
    copies = max(1, args.copies)
    target = [wl.target.to(dev) for _ in range(copies)]
    draft = [wl.draft.to(dev) for _ in range(copies)]
    tokens = wl.tokens.to(dev)
    temperature = wl.temperature.to(dev)
    stream = torch.cuda.current_stream(dev)
    sv = binding.SpecVerify(B, N, V, torch.bfloat16, stream=stream, device=dev)
    out_t = sv.out_tokens[: B * (N + 1)].view(B, N + 1)
    out_a, out_k = sv.out_accept[:B], sv.out_kv[:B]

    # the timed loop calls the C ABI directly with pointers prepared once
    lib = binding.load()
    import ctypes
    P = ctypes.c_void_p
    ptrs = [(P(target[c].data_ptr()), P(draft[c].data_ptr())) for c in range(copies)]
    p_tok, p_temp = P(tokens.data_ptr()), P(temperature.data_ptr())
    p_ot, p_oa, p_ok = P(out_t.data_ptr()), P(out_a.data_ptr()), P(out_k.data_ptr())

    lazy = args.path == "lazy"
    entry = lib.spec_verify_lazy if lazy else lib.spec_verify

    def step(i):
        zt, yt = ptrs[i % copies]
        rc = entry(sv.ctx, B, N, V, zt, yt, p_tok, p_temp, ctypes.c_uint64(i), p_ot, p_oa, p_ok)
        if rc != 0:
            raise binding.SpecVerifyError(rc, "spec_verify")

    for i in range(args.warmup):
        step(i)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    binding.spec_verify_profile_read(sv.ctx)  # clear
    binding.spec_verify_profile(sv.ctx, PROFILE_EVERY)

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
    kernel_ms, calls = binding.spec_verify_profile_read(sv.ctx)
    binding.spec_verify_profile(sv.ctx, False)
    time.sleep(0.2)
    clk = clocks.stop(t_begin, t_end)
    elapsed_ms = ranks_max(elapsed_ms, dev)
    value = whole_job_rate(B * N, args.steps, world, elapsed_ms)
    bytes_per_launch = lazy_bytes(wl, sv, step, out_a) if lazy else wl.bytes_read()
    rowstats_ms = kernel_ms["rowstats"] / max(calls, 1)
    achieved = bytes_per_launch / (rowstats_ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()

    # ---- end to end through the C ABI with host buffers (pinned), rank-local.
    # Double-buffered: step i's inputs are copied on a copy stream into
    # buffer i % 2 while the verify stream still runs step i - 1; the verify
    # of step i waits for its copy, and a copy into a buffer waits for the
    # verify that last read it.  Every copy and read-back is timed.
    e2e_steps = args.e2e_steps or max(3, min(args.steps, 200))
    h_target = wl.target.pin_memory()
    h_draft = wl.draft.pin_memory()
    h_tokens = wl.tokens.pin_memory()
    h_temp = wl.temperature.pin_memory()
    h_out_t = torch.empty(B, N + 1, dtype=torch.int32).pin_memory()
    h_out_a = torch.empty(B, dtype=torch.int32).pin_memory()
    h_out_k = torch.empty(B, dtype=torch.int32).pin_memory()
    bufs = [(target[c % copies], draft[c % copies], torch.empty_like(tokens), torch.empty_like(temperature))
            for c in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (h_target, h_draft, h_tokens, h_temp))
    d2h = sum(t.numel() * t.element_size() for t in (h_out_t, h_out_a, h_out_k))
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        zb, yb, tb, pb = bufs[i % 2]
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
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    copy_stream.wait_event(ev0)  # no copy of the timed steps starts before the clock
    for i in range(e2e_steps):
        e2e_step(i)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = ev0.elapsed_time(ev1)
    e2e_ms = ranks_max(e2e_ms, dev)
    e2e_value = whole_job_rate(B * N, e2e_steps, world, e2e_ms)
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
            "l2": f"inputs larger than L2: {bytes_per_launch / 1e6:.0f} MB read per step, "
                  f"{copies} rotating copies",
            "parallelism": f"replicas x{world} (requests shard, no collective)",
        },
        "roofline": {
            "bound": "hbm", "kernel": "lazy" if lazy else "rowstats", "achieved": achieved, "peak": peak,
            "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s", "frac": achieved / peak,
            "traffic": None if lazy else traffic_per_launch(),
            "algorithmic_bytes_per_launch": bytes_per_launch,
            "avg_launch_us": rowstats_ms * 1e3,
            "timed_launches": f"{calls} of {args.steps} calls (every {PROFILE_EVERY}th)",
        },
        "kernel_us_per_step": ({"lazy": kernel_ms["rowstats"] / max(calls, 1) * 1e3} if lazy else
                               {k: v / max(calls, 1) * 1e3 for k, v in kernel_ms.items()}),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps * (1 if lazy else binding.spec_verify_launches_per_call()),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=12.0)
    sv.close()
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))


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
    target = [wl.target.to(dev) for _ in range(copies)]
    draft = [wl.draft.to(dev) for _ in range(copies)]
    parents, tokens = wl.parents.to(dev), wl.tokens.to(dev)
    temperature = wl.temperature.to(dev)
    sv = binding.SpecVerify(B, M, V, torch.bfloat16, stream=stream, device=dev)
    out_t = sv.out_tokens[: B * (M + 1)].view(B, M + 1)
    out_p = sv.out_path[: B * M].view(B, M)
    out_a, out_k = sv.out_accept[:B], sv.out_kv[:B]

    def step(i, c=None):
        c = i % copies if c is None else c
        binding.spec_verify_tree(sv.ctx, wl.mode, target[c], draft[c], parents, tokens, temperature,
                                 i, out_t, out_p, out_a, out_k)

    for i in range(args.warmup):
        step(i)
    code, _ = sv.get_error()
    assert code == 0, binding.strerror(code)
    binding.spec_verify_profile_read(sv.ctx)
    binding.spec_verify_profile(sv.ctx, PROFILE_EVERY)
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
    kernel_ms, calls = binding.spec_verify_profile_read(sv.ctx)
    binding.spec_verify_profile(sv.ctx, False)
    time.sleep(0.2)
    clk = clocks.stop(t_begin, t_end)
    value = whole_job_rate(B * M, args.steps, world, elapsed_ms)
    bytes_per_launch = wl.bytes_read()
    rs_ms = kernel_ms["rowstats"] / max(calls, 1)
    achieved = bytes_per_launch / (rs_ms / 1e3) / 1e9
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
            "avg_launch_us": rs_ms * 1e3,
            "timed_launches": f"{calls} of {args.steps} calls (every {PROFILE_EVERY}th)",
        },
        "kernel_us_per_step": {("tree_rowstats" if k == "rowstats" else "tree_walk"): v / max(calls, 1) * 1e3
                               for k, v in kernel_ms.items()},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps * 2,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = tree_cpu_baseline(wl, budget_s=12.0)
    sv.close()
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


def run_kv(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_73_gb300 import binding, build, workloads

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    wl = workloads.batch64_bf16(verify_seed=rank)
    B, N, V = wl.shape
    sv = binding.SpecVerify(B, N, V, torch.bfloat16, stream=stream, device=dev)
    _, _, kv = sv(wl.target.to(dev), wl.draft.to(dev), wl.tokens.to(dev), wl.temperature.to(dev), 0)
    kv = kv.clone()
    L, E, W, S = 32, 4096, N + 1, 1024
    copies = max(1, args.copies)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + rank)
    scratch = [torch.randint(0, 256, (L, B, W, E), generator=gen, dtype=torch.uint8, device=dev)
               for _ in range(copies)]
    cache = [torch.zeros(L, B, S, E, dtype=torch.uint8, device=dev) for _ in range(copies)]
    # lengths start below 200 and grow by at most W per commit: reset every 100 commits
    seq0 = torch.randint(0, 200, (B,), generator=gen, dtype=torch.int32, device=dev)
    seq = seq0.clone()
    kv_host = kv.cpu().numpy()
    moved = int(sum(2 * max(int(n), 0) for n in kv_host)) * E * L

    def step(i):
        if i % 100 == 0:
            seq.copy_(seq0)
        binding.spec_verify_kv_commit(sv.ctx, binding.SV_KV_SCRATCH, cache[i % copies], seq, kv,
                                      scratch=scratch[i % copies])

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
    k_ms = elapsed_ms / args.steps  # the commit's two launches are the whole step
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
        "config": {"workload": KV_WORKLOAD, "layers": L, "B": B, "entry_bytes": E, "window": W,
                   "cache_positions": S, "mode": "scratch", "kv_len_sum": int(sum(max(int(n), 0) for n in kv_host)),
                   "bytes_moved_per_step": moved,
                   "l2": f"{copies} rotating scratch windows of {L * B * W * E / 1e6:.0f} MB",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "kernel": "kv_commit", "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": moved, "avg_launch_us": k_ms * 1e3,
                     "timed_launches": f"all {args.steps} commits of the timed loop (copy + length "
                                       f"update launches, one length reset per 100 commits)"},
        "e2e": None,
        "gpu_launches": args.steps * 2,
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


def run_fcnorm(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_73_gb300 import binding, build, workloads

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    T, d, d_out = 4096, 4096, 4096
    wl = workloads.make_fcnorm(T, d, d_out, gen_seed=2026 + rank, name=FC_WORKLOAD)
    h = [x.to(dev) for x in wl.h]
    w, g, b, bias = wl.weight.to(dev), wl.gamma.to(dev), wl.beta.to(dev), wl.bias.to(dev)
    out = torch.empty(T, d_out, dtype=torch.bfloat16, device=dev)
    xbuf = torch.empty(T, 3 * d, dtype=torch.bfloat16, device=dev)
    sv = binding.SpecVerify(1, 1, 16, torch.float32, stream=stream, device=dev)

    def step():
        binding.spec_verify_fc_norm(sv.ctx, binding.SV_NORM_LAYER, *h, w, gamma=g, beta=b, bias=bias,
                                    out=out, xbuf=xbuf)

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
    flops = 2.0 * T * 3 * d * d_out
    per_ms = elapsed_ms / steps
    value = flops * steps * world / (elapsed_ms / 1e3) / 1e12
    peak, kind = bf16_peak()
    achieved = flops / (per_ms / 1e3) / 1e12
    line = {
        "metric": "FC-norm TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": per_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate",
        "data": "synthetic (Gaussian hidden states of three magnitudes, random weights)",
        "config": {"workload": FC_WORKLOAD, "T": T, "d": d, "d_out": d_out, "norm": "layernorm",
                   "flops_per_call": flops, "parallelism": f"replicas x{world}"},
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


# --------------------------------------------------------------------------- oracle

def oracle_requests(wl, idx):
    """Run the CPU oracle on the listed requests of a workload."""
    from oracle import verify as ov
    z, y = wl.raw()
    d = wl.tokens.numpy()
    t = wl.temperature.numpy()
    for b in idx:
        ov.verify_request(z[b], y[b], d[b], t[b], wl.seed, b, wl.dtype)


def cpu_baseline(wl, budget_s):
    """The oracle, as it stands, on whole requests of the workload until the
    budget is spent; one host thread (numpy float64)."""
    B, N, _ = wl.shape
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        oracle_requests(wl, [done % B])
        done += 1
    el = time.perf_counter() - t0
    return {"value": done * N / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} requests of {WORKLOAD} (request i = step i mod {B}), "
                      f"{el:.1f} s, float64 numpy on 1 host thread"}


def oracle_position(wl, z, y, b, j, seed):
    """The oracle's work for draft position j (1-based) of request b, as it
    stands: widen the rows, then the argmax (T = 0) or both softmaxes, the
    Philox uniform and the accept test; at the last position also the
    residual of that row pair and its grouped draw (one draw per request)."""
    from oracle import philox as oph
    from oracle import verify as ov
    _, N, _ = wl.shape
    t = float(wl.temperature[b])
    zr = ov.logits_to_f64(z[b, j - 1], wl.dtype)
    if t == 0.0:
        ov.argmax_lowest(zr)
        return
    d = int(wl.tokens[b, j - 1])
    q = ov.softmax(zr, t)
    p = ov.softmax(ov.logits_to_f64(y[b, j - 1], wl.dtype), t)
    ov.accept(q[d], p[d], oph.uniform(seed, b, j, oph.ACCEPT_DRAW))
    if j == N:
        ov.sample_grouped(ov.residual(q, p), oph.uniforms4(seed, b, j, oph.SAMPLE_DRAW))


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_73_gb300 import workloads
    wl = workloads.batch64_bf16()
    B, N, V = wl.shape
    z, y = wl.raw()
    # one step = the oracle's work for one draft position (request-major
    # order over all B x N positions, rotating), so any --steps stays bounded
    def step(i):
        k = i % (B * N)
        oracle_position(wl, z, y, k // N, k % N + 1, wl.seed)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    el = time.perf_counter() - t0
    value = args.steps / el
    sample = (f"one draft position of {WORKLOAD} per step (positions taken request-major, "
              f"rotating over all {B * N}; greedy positions cost an argmax, sampled ones two "
              f"softmaxes, the accept test and, at a request's last position, the residual draw), "
              f"float64 numpy, 1 host thread")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "N": N, "V": V, "logits": "bf16"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
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
