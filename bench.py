"""Benchmark of the speculative-decoding verify step on GB300.

One step = one spec_verify call over a batch of the c3 workload (B=256
sequences, K=8 drafts, V=152064, bf16 logits, temperature 0.7): temperature
softmax of 17 rows per sequence, gather, acceptance, first-rejection scan and
the residual / bonus draw.  Prints one JSON line (see the keys below).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 (torchrun), every rank verifies its own batch of B sequences
(independent sequences: weak scaling, no collective on the data path); the
timing uses a barrier on both sides and the maximum over ranks.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "c3"
METRIC = "verified sequences/sec (spec_verify, HBM-roofline reported)"
UNIT = "seq/s"
L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "spec_verify_c3_traffic.txt")


# --------------------------------------------------------------------------
# helpers shared with the multi-rank CPU tests
# --------------------------------------------------------------------------
def dist_env():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(rank: int, step: int) -> int:
    """Philox seed of one rank's batch at one step (independent batches)."""
    return (rank << 32) | step


def max_over_ranks(value: float, world: int) -> float:
    """Maximum of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# The sources that make up the sampling kernel and its launch configuration.
SAMPLE_SOURCES = ("api.cu", "sample_kernel.cu", "sv_common.cuh", "sv_kernels.h")


def source_hash() -> str:
    """sha256 over the sampling kernel's sources (ties a stored ncu traffic
    figure to the kernel it was measured on)."""
    csrc = os.path.join(ROOT, "speculative_decoding_verification_36_gb300", "csrc")
    h = hashlib.sha256()
    for name in SAMPLE_SOURCES:
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()


def stored_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    kv = {}
    for line in open(TRAFFIC_FILE):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha256") != source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"specverify_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            if self.uuid and self.uuid not in parts[0]:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------
# workload
# --------------------------------------------------------------------------
def workload_config(p, two_sets: bool):
    return {
        "workload": f"{p.name}: chain verify B={p.B} K={p.K} V={p.V} logits bf16 tau={p.temperature}; "
                    "target N(0,4^2) - 1.1 ln(v+1), draft = target + N(0,2^2), drafts sampled from "
                    "the draft softmax",
        "B": p.B, "K": p.K, "V": p.V, "logits": "bf16", "temperature": p.temperature,
        "bytes_per_step": algorithmic_bytes(p),
        "l2": ("inputs larger than L2 (%.2f GB per step vs 129 MB)" % (algorithmic_bytes(p) / 1e9))
              + ("; two input sets alternate" if two_sets else ""),
    }


def algorithmic_bytes(p) -> int:
    """Logits read once (2K+1 rows of V bf16 per sequence) plus the drafted
    tokens read and the outputs written."""
    return p.B * (2 * p.K + 1) * p.V * 2 + p.B * p.K * 4 + p.B * (p.K + 2) * 4


def oracle_seq_per_s(x_cpu, p, budget_s: float, max_seq: int):
    """The fp64 oracle timed on this host's cores on a bounded sample of the
    same inputs (sequence by sequence until the time budget is used).  Also
    returns the oracle's result for the first pass over the sample (seed 0,
    sequence ids 0..B-1), for the parity check of the bench line."""
    import oracle
    oracle.build()
    done = 0
    first = {}
    t0 = time.perf_counter()
    while done < max_seq:
        b = done % p.B
        r = oracle.spec_verify(x_cpu["target"][b:b + 1], x_cpu["draft"][b:b + 1], x_cpu["tokens"][b:b + 1],
                               p.temperature, 0, seq_ids=[b])
        if b not in first:
            first[b] = r
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, done, dt, first


def host_threads() -> int:
    """Threads for the all-cores oracle timing: the CPUs this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_parallel_seq_per_s(x_cpu, p, budget_s: float, threads: int):
    """The same oracle, one sequence per call, on `threads` host threads at
    once (the C oracle holds no global state, and ctypes releases the GIL
    during the call), cycling over the batch until the time budget is used
    and at least once over the whole batch.  Also returns the oracle's result
    for every sequence of the batch (seed 0, its batch index as sequence
    number), for the parity check of the bench line."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()
    results = {}

    def one(b):
        r = oracle.spec_verify(x_cpu["target"][b:b + 1], x_cpu["draft"][b:b + 1], x_cpu["tokens"][b:b + 1],
                               p.temperature, 0, seq_ids=[b])
        results.setdefault(b, r)

    done = 0
    with ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        while True:
            list(ex.map(one, [(done + t) % p.B for t in range(threads)]))
            done += threads
            if time.perf_counter() - t0 > budget_s and done >= p.B:
                break
        dt = time.perf_counter() - t0
    return done / dt, done, dt, results


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def parity_sample(gpu_tokens, gpu_n, first):
    """GPU outputs against the oracle's on the sequences the CPU leg ran:
    exact matches, sequences that differ only at a draw within 1e-6 of its
    decision boundary, other mismatches, and the oracle's boundary draws."""
    import numpy as np
    same = boundary = other = draws = 0
    for b, r in first.items():
        am, sm = r["acc_margin"][0], r["sample_margin"][0]
        draws += int(np.sum(am[np.isfinite(am)] < 1e-6)) + int(np.isfinite(sm) and sm < 1e-6)
        if int(gpu_n[b]) == int(r["n"][0]) and np.array_equal(gpu_tokens[b], r["tokens"][0]):
            same += 1
        elif (int(gpu_n[b]) != int(r["n"][0]) and min(int(gpu_n[b]), int(r["n"][0])) >= 0
              and am[min(int(gpu_n[b]), int(r["n"][0]))] < 1e-6) or (
                int(gpu_n[b]) == int(r["n"][0]) and np.isfinite(sm) and sm < 1e-6):
            boundary += 1
        else:
            other += 1
    return {"sequences": len(first), "identical": same, "boundary_only": boundary,
            "mismatch": other, "oracle_boundary_draws": draws}


# --------------------------------------------------------------------------
# the two arms
# --------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import torch
    from speculative_decoding_verification_36_gb300 import workloads as wl
    p = wl.preset(WORKLOAD)
    threads = host_threads()
    x = wl.make_chain(wl.preset(WORKLOAD, B=threads), device="cpu", seed=0)
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()

    def one(b):
        oracle.spec_verify(x["target"][b:b + 1], x["draft"][b:b + 1], x["tokens"][b:b + 1],
                           p.temperature, 0, seq_ids=[b])

    with ThreadPoolExecutor(max_workers=threads) as ex:
        def step(i):  # one sequence on every host thread
            list(ex.map(one, range(threads)))

        for i in range(args.warmup):
            step(i)
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(i)
        dt = time.perf_counter() - t0
    value = args.steps * threads / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(p, False),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{threads} c3 sequences (17 rows x 152064 each) per step, one per "
                                   f"host thread, fp64 C oracle"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def gpu_local_cpus(dev):
    """CPUs on the host socket the GPU is attached to (from the PCI device's
    local_cpulist), or None when the system does not say."""
    import torch
    try:
        pr = torch.cuda.get_device_properties(dev)
        path = "/sys/bus/pci/devices/%04x:%02x:%02x.0/local_cpulist" % (
            pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        cpus = set()
        for part in open(path).read().strip().split(","):
            if "-" in part:
                lo, hi = part.split("-")
                cpus.update(range(int(lo), int(hi) + 1))
            elif part:
                cpus.add(int(part))
        usable = cpus & os.sched_getaffinity(0)
        return usable or None
    except Exception:
        return None


def run_e2e(sv, sets, p, rank, world, dev, stream, e2e_steps):
    """The same metric through the public API with the inputs copied from
    pinned host memory and the outputs read back, every step.  The process is
    first bound to the CPUs of the GPU's own socket, so that the pinned
    buffers are allocated (first touch) in the memory next to the GPU, as a
    serving process would place them."""
    import torch
    local = gpu_local_cpus(dev)
    saved = os.sched_getaffinity(0)
    if local:
        os.sched_setaffinity(0, local)
    try:
        return _run_e2e(sv, sets, p, rank, world, dev, stream, e2e_steps, local)
    finally:
        os.sched_setaffinity(0, saved)


def _run_e2e(sv, sets, p, rank, world, dev, stream, e2e_steps, local):
    import torch
    host = [{k: sets[i][k].cpu().pin_memory() for k in ("target", "draft", "tokens")}
            for i in range(len(sets))]
    host_out = (torch.empty((p.B, p.K + 1), dtype=torch.int32).pin_memory(),
                torch.empty((p.B,), dtype=torch.int32).pin_memory())
    dbuf = {k: torch.empty_like(sets[0][k]) for k in ("target", "draft", "tokens")}
    h2d = sum(host[0][k].numel() * host[0][k].element_size() for k in host[0])
    d2h = host_out[0].numel() * 4 + host_out[1].numel() * 4

    def e2e_step(i):
        src = host[i % len(host)]
        for k in dbuf:
            dbuf[k].copy_(src[k], non_blocking=True)
        t, n = sv.spec_verify(dbuf["target"], dbuf["draft"], dbuf["tokens"], p.temperature,
                              rank_seed(rank, i), stream=stream)
        host_out[0].copy_(t, non_blocking=True)
        host_out[1].copy_(n, non_blocking=True)

    e2e_step(0)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = world * p.B * e2e_steps / (e2e_ms / 1e3)
    return e2e_value, h2d, d2h, (len(local) if local else None)


# --------------------------------------------------------------------------
# the other workloads and entry points, reported beside the headline
# --------------------------------------------------------------------------
def time_calls(call, steps, warm, stream, dev, flush=None):
    """Average device milliseconds per call: CUDA events on `stream` around
    each call, after `warm` untimed calls; `flush()` runs (untimed) before
    every timed call when given."""
    import torch
    for i in range(warm):
        call(i)
    torch.cuda.synchronize(dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        if flush is not None:
            flush()
        ev[i][0].record(stream)
        call(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in ev) / steps


def chain_rows_used(n, K):
    """Rows an early-exit verify depends on: target and draft rows 0..n, or
    all 2K + 1 rows when every draft is accepted (n = K)."""
    return sum(2 * K + 1 if int(v) >= K else 2 * (int(v) + 1) for v in n)


def extra_entry(ms, seqs, nbytes, peak, steps, l2, **more):
    gbs = nbytes / (ms / 1e3) / 1e9
    d = {"value": seqs / (ms / 1e3), "unit": "seq/s", "us_per_call": ms * 1e3, "bytes_per_step": int(nbytes),
         "achieved_gbs": gbs, "frac": gbs / peak, "steps": steps, "l2": l2}
    d.update(more)
    return d


def oracle_rates(one, B, budget_s, threads):
    """The oracle on this host's cores for one extra workload: `one(b)` runs
    it on item b of the batch; single-threaded, then on `threads` host
    threads at once (ctypes releases the GIL), each for about budget_s.
    Returns items per second for both."""
    from concurrent.futures import ThreadPoolExecutor
    done, t0 = 0, time.perf_counter()
    while True:
        one(done % B)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    single = done / (time.perf_counter() - t0)
    done = 0
    with ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        while True:
            list(ex.map(one, [(done + t) % B for t in range(threads)]))
            done += threads
            if time.perf_counter() - t0 > budget_s:
                break
        multi = done / (time.perf_counter() - t0)
    return {"single_thread": single, "all_cores": multi, "cores": threads, "kind": "oracle",
            "budget_s_each": budget_s}


def run_extras(sv, wl, dev, stream, steps, peak, cpu_budget=0.0):
    """CUDA-event timings, bytes per call and the fraction of the measured HBM
    bandwidth for every workload and entry point besides the headline: c1,
    c2 and c4 (full read and early exit), the c3 early exit, the c3 verify
    with row entropies or with the draft-length suggestion, the c5 tree
    (greedy, its early exit, and stochastic), and n-gram drafting."""
    import torch
    out = {}
    flushbuf = torch.empty(128 * 2**20, dtype=torch.float32, device=dev)  # 512 MB, read to evict L2
    flushbuf.fill_(1.0)

    def flush():
        flushbuf.sum()

    def big(nbytes):
        return nbytes >= 2 * L2_BYTES

    def l2_note(nbytes, sets):
        if big(nbytes):
            return f"inputs larger than L2 ({nbytes / 1e6:.0f} MB per call), {sets} input sets alternate"
        return f"L2 flushed before every call ({nbytes / 1e6:.1f} MB per call)"

    def chain(name, early=False):
        p = wl.preset(name)
        sets = [wl.make_chain(p, device=dev, seed=10 + i) for i in range(2)]
        esz = 4 if p.dtype == torch.float32 else 2
        rows = 2 * p.K + 1 if p.temperature > 0 else p.K + 1
        full = p.B * rows * p.V * esz
        fn = sv.spec_verify_early_exit if early else sv.spec_verify

        def call(i):
            x = sets[i % 2]
            fn(x["target"], x["draft"], x["tokens"], p.temperature, i, stream=stream)

        ms = time_calls(call, steps, 3, stream, dev, None if big(full) else flush)
        if early:
            x = sets[0]
            _, n = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 0, stream=stream)
            K = p.K
            used = chain_rows_used(n.cpu().tolist(), K) if p.temperature > 0 else \
                sum(int(v) + 1 for v in n.cpu().tolist())
            nbytes = used * p.V * esz
            e = extra_entry(ms, p.B, nbytes, peak, steps, l2_note(full, 2),
                            bytes_note="rows the result depends on (input set 0, seed 0)")
        else:
            e = extra_entry(ms, p.B, full, peak, steps, l2_note(full, 2))
        e["config"] = f"B={p.B} K={p.K} V={p.V} {str(p.dtype).split('.')[-1]} tau={p.temperature}"
        if cpu_budget > 0 and not early:
            import oracle
            oracle.build()
            xc = {k: (v.cpu() if v is not None else None) for k, v in sets[0].items() if k in ("target", "draft", "tokens")}
            if p.temperature > 0:
                def one(b):
                    oracle.spec_verify(xc["target"][b:b + 1], xc["draft"][b:b + 1], xc["tokens"][b:b + 1],
                                       p.temperature, 0, seq_ids=[b])
            else:
                def one(b):
                    oracle.spec_verify_greedy(xc["target"][b:b + 1], xc["tokens"][b:b + 1])
            e["cpu_oracle"] = oracle_rates(one, p.B, cpu_budget, host_threads())
            e["cpu_oracle"]["unit"] = "seq/s"
            del xc
        del sets
        return e

    out["c1"] = chain("c1")
    out["c2"] = chain("c2")
    out["c2_early_exit"] = chain("c2", early=True)
    out["c3_early_exit"] = chain("c3", early=True)
    out["c4"] = chain("c4")
    out["c4_early_exit"] = chain("c4", early=True)

    # c3 with the entropy pass: row entropies, and the draft-length suggestion
    p = wl.preset("c3")
    sets = [wl.make_chain(p, device=dev, seed=20 + i) for i in range(2)]
    full = p.B * (2 * p.K + 1) * p.V * 2

    def plain(i):
        x = sets[i % 2]
        sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, i, stream=stream)

    def khint(i):
        x = sets[i % 2]
        sv.spec_verify_khint(x["target"], x["draft"], x["tokens"], p.temperature, i, 1.0, 2.0, 1, 16,
                             stream=stream)

    def stats(i):
        x = sets[i % 2]
        sv.spec_verify_stats(x["target"], x["draft"], x["tokens"], p.temperature, i, stream=stream,
                             entropy=True)

    ms_plain = time_calls(plain, steps, 3, stream, dev)
    ms_k = time_calls(khint, steps, 3, stream, dev)
    ms_s = time_calls(stats, steps, 3, stream, dev)
    out["c3_khint"] = extra_entry(ms_k, p.B, full, peak, steps, l2_note(full, 2),
                                  entry_point="spec_verify_khint_bf16",
                                  cost_vs_spec_verify_pct=100.0 * (ms_k / ms_plain - 1.0),
                                  spec_verify_us_same_run=ms_plain * 1e3)
    out["c3_stats_entropy"] = extra_entry(ms_s, p.B, full, peak, steps, l2_note(full, 2),
                                          entry_point="spec_verify_stats_bf16 (row stats, p/q, residual "
                                                      "mass and row entropies)",
                                          cost_vs_spec_verify_pct=100.0 * (ms_s / ms_plain - 1.0))
    del sets

    # c5: tree greedy (full read and early exit) and stochastic tree
    p = wl.preset("c5")
    trees = [wl.make_tree(p, device=dev, seed=30 + i) for i in range(2)]
    full = p.B * (p.N + 1) * p.V * 2
    for early in (False, True):
        def tcall(i, early=early):
            x = trees[i % 2]
            sv.spec_tree_verify_greedy(x["target"], x["tokens"], x["parents"], stream=stream, early_exit=early)

        ms = time_calls(tcall, steps, 3, stream, dev, None if big(full) else flush)
        if early:
            x = trees[0]
            _, ln, _ = sv.spec_tree_verify_greedy(x["target"], x["tokens"], x["parents"], stream=stream)
            nbytes = sum(int(v) for v in ln.cpu().tolist()) * p.V * 2
            out["c5_early_exit"] = extra_entry(ms, p.B, nbytes, peak, steps, l2_note(full, 2),
                                               bytes_note="rows on the accepted path (input set 0)")
        else:
            out["c5"] = extra_entry(ms, p.B, full, peak, steps, l2_note(full, 2),
                                    config=f"B={p.B} N={p.N} V={p.V} bf16, complete binary tree depth {p.depth}")
    if cpu_budget > 0:
        import oracle
        tc = {k: trees[0][k].cpu() for k in ("target", "tokens", "parents")}

        def tone(b):
            oracle.tree_verify_greedy(tc["target"][b:b + 1], tc["tokens"][b:b + 1], tc["parents"][b:b + 1])

        out["c5"]["cpu_oracle"] = dict(oracle_rates(tone, p.B, cpu_budget, host_threads()), unit="seq/s")
        del tc
    del trees
    trees = [wl.make_tree_sampling(p, 1.0, device=dev, seed=40 + i) for i in range(2)]
    full_s = 2 * p.B * (p.N + 1) * p.V * 2

    def scall(i):
        x = trees[i % 2]
        sv.spec_tree_verify_sampling(x["target"], x["draft"], x["tokens"], x["parents"], 1.0, i, stream=stream)

    ms = time_calls(scall, steps, 3, stream, dev, None if big(full_s) else flush)
    out["c5_stochastic_tree"] = extra_entry(ms, p.B, full_s, peak, steps, l2_note(full_s, 2),
                                            config=f"B={p.B} N={p.N} V={p.V} bf16 target and draft, tau 1")
    if cpu_budget > 0:
        import oracle
        tc = {k: trees[0][k].cpu() for k in ("target", "draft", "tokens", "parents")}

        def sone(b):
            # sequence b alone draws with sequence number 0: a timing, not a parity check
            oracle.tree_verify_sampling(tc["target"][b:b + 1], tc["draft"][b:b + 1], tc["tokens"][b:b + 1],
                                        tc["parents"][b:b + 1], 1.0, b)

        out["c5_stochastic_tree"]["cpu_oracle"] = dict(oracle_rates(sone, p.B, cpu_budget, host_threads()),
                                                       unit="seq/s")
        del tc
    del trees

    # n-gram drafting: 256 histories of up to 131072 tokens (16 seeded
    # histories repeated), n 1..4, K = 8
    h = wl.make_ngram_histories(16, 131072, seed=1)
    tok = h["tokens"].repeat(16, 1).contiguous().to(dev)
    ln = h["lengths"].repeat(16).contiguous().to(dev)
    nbytes = int(ln.sum().item()) * 4

    def ncall(i):
        sv.spec_ngram_draft(tok, ln, 1, 4, 8, stream=stream)

    ms = time_calls(ncall, steps, 3, stream, dev, flush)
    out["ngram"] = extra_entry(ms, 256, nbytes, peak, steps, l2_note(nbytes, 1),
                               config="B=256 histories up to 131072 tokens, n 1..4, K=8")
    out["ngram"]["unit"] = "histories/s"
    if cpu_budget > 0:
        import oracle
        htok, hlen = tok[:16].cpu(), ln[:16].cpu()

        def gone(b):
            oracle.ngram_draft(htok[b:b + 1], hlen[b:b + 1], 1, 4, 8)

        out["ngram"]["cpu_oracle"] = dict(oracle_rates(gone, 16, cpu_budget, host_threads()), unit="histories/s")

    # A bare read of each entry's bytes: torch's max over a float32 buffer of
    # the same size, timed like the entry (L2 flushed first when the bytes
    # fit in twice L2).  One read pass of that size, nothing else, is the
    # practical ceiling the entry's call can be held against.
    reads = {}

    def plain_read_ms(nbytes):
        if nbytes not in reads:
            x = torch.ones(max(1, nbytes // 4), dtype=torch.float32, device=dev)
            reads[nbytes] = time_calls(lambda i: x.max(), steps, 3, stream, dev, None if big(nbytes) else flush)
            del x
        return reads[nbytes]

    for e in out.values():
        nb = e.get("bytes_per_step")
        if nb:
            ms = plain_read_ms(nb)
            e["plain_read"] = {"us_per_call": ms * 1e3, "call_vs_read": e["us_per_call"] / (ms * 1e3),
                               "kind": "torch max over a float32 buffer of the same bytes"}
    p3 = wl.preset("c3")
    c3_bytes = algorithmic_bytes(p3)
    ms = plain_read_ms(c3_bytes)
    out["c3_plain_read"] = {"us_per_call": ms * 1e3, "bytes": c3_bytes,
                            "kind": "torch max over a float32 buffer of the headline's bytes per step",
                            "l2": l2_note(c3_bytes, 1)}
    del tok, ln, flushbuf
    torch.cuda.synchronize(dev)
    return out


def read_sweep(dev, steps=50):
    """One read pass (torch max over a float32 buffer) at growing sizes, L2
    flushed before each call, CUDA events: what a bare read reaches at each
    size on this GPU."""
    import torch
    stream = torch.cuda.current_stream(dev)
    flushbuf = torch.ones(128 * 2**20, dtype=torch.float32, device=dev)
    rows = []
    for mib in (64, 105, 134, 180, 256, 512, 1024, 2048):
        x = torch.ones(mib * 2**20 // 4, dtype=torch.float32, device=dev)
        ms = time_calls(lambda i: x.max(), steps, 3, stream, dev, lambda: flushbuf.sum())
        rows.append({"MiB": mib, "us_per_call": round(ms * 1e3, 2), "GBs": round(x.numel() * 4 / ms / 1e6, 1)})
        del x
    return rows


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import speculative_decoding_verification_36_gb300 as sv
    from speculative_decoding_verification_36_gb300 import build as _build
    from speculative_decoding_verification_36_gb300 import workloads as wl
    _build.build()

    p = wl.preset(WORKLOAD, B=args.batch) if args.batch else wl.preset(WORKLOAD)
    sets = [wl.make_chain(p, device=dev, seed=rank * 2 + i) for i in range(args.sets)]
    stream = torch.cuda.current_stream(dev)
    outs = [(torch.empty((p.B, p.K + 1), dtype=torch.int32, device=dev),
             torch.empty((p.B,), dtype=torch.int32, device=dev)) for _ in range(2)]

    def step(i):
        x = sets[i % len(sets)]
        o = outs[i % 2]
        sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, rank_seed(rank, i),
                       out_tokens=o[0], out_n_accepted=o[1], stream=stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize(dev)
    assert sv.spec_get_status() == 0

    # device-resident timed region
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    with ClockSampler(uuid) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            step(i)
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    total_ms = t_start.elapsed_time(t_end)
    per_launch = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(total_ms, world)
    avg_launch_ms = max_over_ranks(sum(per_launch) / len(per_launch), world)
    value = world * p.B * args.steps / (total_ms / 1e3)
    flags = sv.spec_get_status()

    # the early-exit verify on the same inputs (reads only the rows the result
    # depends on): reported beside the full-read number, same timing rules
    ee_ms = None
    if args.early_exit_steps > 0:
        def ee_step(i):
            x = sets[i % len(sets)]
            o = outs[i % 2]
            sv.spec_verify_early_exit(x["target"], x["draft"], x["tokens"], p.temperature,
                                      rank_seed(rank, i), out_tokens=o[0], out_n_accepted=o[1],
                                      stream=stream)
        for i in range(max(args.warmup, 3)):
            ee_step(i)
        barrier(world)
        torch.cuda.synchronize(dev)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for i in range(args.early_exit_steps):
            ee_step(i)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        ee_ms = max_over_ranks(a0.elapsed_time(a1), world) / args.early_exit_steps

    # the oracle on the host cores, before the end-to-end leg binds the
    # process to the GPU's socket (rank 0 at N = 1 only), and the parity of
    # the whole batch of input set 0 (seed 0) against it
    cpu_line = parity = None
    if world == 1 and not args.no_cpu_baseline:
        threads = host_threads()
        x_cpu = {k: sets[0][k].cpu() for k in ("target", "draft", "tokens")}
        v, done, dt, _ = oracle_seq_per_s(x_cpu, p, args.cpu_budget, 1 << 30)
        vp, donep, dtp, results = oracle_parallel_seq_per_s(x_cpu, p, args.cpu_budget, threads)
        cpu_line = {"value": vp, "unit": UNIT, "cores": threads, "kind": "oracle",
                    "sample": f"{donep} c3 sequences (cycling over the batch of {p.B}) in {dtp:.1f} s, "
                              f"fp64 C oracle, one sequence per call on {threads} host threads",
                    "single_thread": {"value": v, "sample": f"{done} sequences in {dt:.1f} s"},
                    "cpu_model": cpu_model(), "os_cpu_count": os.cpu_count(),
                    "affinity_cpus": threads}
        x = sets[0]
        tok0, n0 = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 0, stream=stream)
        torch.cuda.synchronize(dev)
        parity = parity_sample(tok0.cpu().numpy(), n0.cpu().numpy(), results)
        del x_cpu

    # end to end through the public API from pinned host buffers
    e2e_steps = min(args.steps, args.e2e_steps)
    e2e_value, h2d, d2h, e2e_cpus = None, 0, 0, None
    if e2e_steps > 0:
        e2e_value, h2d, d2h, e2e_cpus = run_e2e(sv, sets, p, rank, world, dev, stream, e2e_steps)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peak, peak_kind = peaks()
    abytes = algorithmic_bytes(p)
    achieved = abytes / (avg_launch_ms / 1e3) / 1e9
    traffic = stored_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(p, len(sets) > 1),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "sv::sample_kernel<BF16,8>",
                     "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "avg_launch_ms": avg_launch_ms, "bytes_per_launch": abytes},
        "e2e": ({"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                 "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                 "host_buffers": ("pinned, allocated from the %d CPUs of the GPU's socket" % e2e_cpus)
                 if e2e_cpus else "pinned"} if e2e_steps > 0 else None),
        "early_exit": ({"value": world * p.B / (ee_ms / 1e3), "unit": UNIT, "ms_per_step": ee_ms,
                        "steps": args.early_exit_steps,
                        "entry_point": "spec_verify_early_exit_bf16",
                        "note": "reads only target/draft rows 0..n (and row K when all drafts are "
                                "accepted); identical tokens on valid inputs; bad data checked on "
                                "the rows used"} if ee_ms else None),
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "status_flags": flags,
    }
    if cpu_line is not None:
        line["cpu_baseline"] = cpu_line
        line["parity_sample"] = parity
    if world == 1 and args.extras_steps > 0:
        line["extra"] = run_extras(sv, wl, dev, stream, args.extras_steps, peak,
                                   0.0 if args.no_cpu_baseline else args.extras_cpu_budget)
        line["extra_status_flags"] = sv.spec_get_status()
    if world == 1:
        # acceptance statistics of one batch (spec_acceptance_stats on the GPU)
        x = sets[0]
        _, n0 = sv.spec_verify(x["target"], x["draft"], x["tokens"], p.temperature, 0, stream=stream)
        st = sv.spec_acceptance_stats(n0, p.K, stream=stream)
        torch.cuda.synchronize(dev)
        line["acceptance"] = {"mean_tokens_per_step": float(st["mean_tokens"]),
                              # null where no sequence reached the position
                              "alpha_per_position": [round(float(a), 4) if math.isfinite(float(a)) else None
                                                     for a in st["alpha"].cpu()],
                              "accepted_histogram": [int(h) for h in st["hist"].cpu()]}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20,
                    help="steps of the end-to-end (host buffers) measurement; 0 skips it")
    ap.add_argument("--early-exit-steps", type=int, default=500,
                    help="timed steps of the early-exit verify reported beside the main number; 0 skips it")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences per rank (default: the workload's B); for profiling runs")
    ap.add_argument("--sets", type=int, default=2, choices=[1, 2],
                    help="input sets alternated between steps")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--extras-cpu-budget", type=float, default=1.5,
                    help="seconds of oracle timing per extra workload, single-threaded and all cores")
    ap.add_argument("--extras-steps", type=int, default=100,
                    help="timed calls per extra workload (c1, c2, c4, c5, early exits, ...); 0 skips them")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--read-sweep", action="store_true",
                    help="print one JSON line of bare-read times over growing sizes and exit")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.read_sweep:
        import torch
        dev = torch.device("cuda", 0)
        print(json.dumps({"read_sweep": read_sweep(dev), "kind": "torch max over a float32 buffer, "
                          "L2 flushed by a 512 MB read before each call, CUDA events"}))
        return 0
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
