#!/usr/bin/env python
"""Benchmark of the decode/prefill hot path on one GB300 (or N replicas).

Default workload ("streaming"): B=1, Hq=16, Hkv=8, D=128, max_len=8192 bf16
static cache; one step = 8192 consecutive decode steps from position 0, each
one attn_decode_step_append launch (write the step's K/V row, then attend
rows 0..pos).  The 8192 launches of a step are captured once into a CUDA graph
and replayed; inputs for all 8192 positions are resident in HBM before timing.
L2 is flushed (a 512 MB read, which leaves only clean lines) between timed
steps, outside the timed events.

value = algorithmic decode bytes (K and V rows 0..pos of every KV head, plus
q and out) / device time of the step, in GB/s; `steps_per_s` is decode steps
per second.  Extra legs: per-position decode time (warm and cold L2), the
ragged B=64 batch, the B=256 g=8 stress batch, the ragged batch as a fused
append step with and without the rotary embedding, the ragged batch over a
1024-row local window, the ragged and stress batches with two new tokens per
sequence, and the causal prefill workloads (TFLOP/s; also GQA prompt chunks
at d_head=128), each against its roofline.  The cross-checks time the
same 8192 positions as separate append/decode launches, as decode launches
alone, and as fused steps with the rotary embedding.

``--impl reference`` times the fp64 CPU oracle (the only reference this
method has) on the host cores, on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

STEPS_STREAM = 8192
# DRAM bytes per launch of the streaming step's decode kernel, from an ncu
# launch list of `bench.py --only streaming_sample` (dram__bytes_read.sum +
# dram__bytes_write.sum, cold cache, mean over the sampled positions).  Set
# to None when the kernel changes until it is measured again.  It is 4.9%
# above the algorithmic bytes: every cluster rank fetches its first tile
# before the position is known, and tiles are whole 128-row boxes.
TRAFFIC_BYTES_PER_LAUNCH = 17.619e6
HQ, HKV, D, L = 16, 8, 128, 8192
METRIC = "decode-attn HBM GB/s (% of peak) & steps/s; causal prefill TFLOP/s"
FLUSH_BYTES = 512 << 20
# the nominal HBM3e bandwidth of the part (a second denominator beside the
# measured copy rate, which both reads and writes)
NOMINAL_HBM_GBS = 8000.0


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-legs", action="store_true", help="skip the extra workload legs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", type=str, default=None,
                    help="run one workload a few times and exit (for ncu captures): "
                         "streaming_sample, position:N, single_step, ragged, stress, prefill, "
                         "prefill_prefix, prefill_d128_chunk, prefill_d128")
    ap.add_argument("--reps", type=int, default=3, help="launches per --only run")
    ap.add_argument("--batch", type=int, default=None,
                    help="--only with a decode workload: use this batch size instead "
                         "(a smaller capture of the same kernel)")
    ap.add_argument("--window", type=int, default=None,
                    help="--only with a decode workload: attend the last WINDOW rows "
                         "(attn_decode_step_window)")
    ap.add_argument("--heads", type=int, default=None,
                    help="--only with a decode workload: use this many query heads "
                         "(another group size on the same cache shape)")
    ap.add_argument("--cpu-worker", type=str, default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _decode_bytes_stream(steps=STEPS_STREAM):
    import oracle
    return sum(oracle.decode_bytes([p], HQ, HKV, D) for p in range(steps))


# ------------------------------------------------------------- CPU oracle ---

def cpu_worker(kind: str):
    """Time the oracle, single-threaded, on a bounded sample of a workload."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(0)
    if kind == "streaming":
        sample = list(range(0, STEPS_STREAM, 64))  # every 64th position of the loop
        k = rng.standard_normal((STEPS_STREAM, HKV, D)).astype(np.float32).astype(np.float64)
        v = rng.standard_normal((STEPS_STREAM, HKV, D)).astype(np.float32).astype(np.float64)
        q = rng.standard_normal((STEPS_STREAM, 1, HQ, D)).astype(np.float32).astype(np.float64)
        kc = k.transpose(1, 0, 2)[None]
        vc = v.transpose(1, 0, 2)[None]
        t0 = time.perf_counter()
        nbytes = 0
        for p in sample:
            oracle.decode(q[p], kc[:, :, : p + 1], vc[:, :, : p + 1], [p], 1.0 / math.sqrt(D))
            nbytes += oracle.decode_bytes([p], HQ, HKV, D)
        dt = time.perf_counter() - t0
        print(json.dumps({"value": nbytes / dt / 1e9, "unit": "GB/s", "seconds": dt,
                          "steps_per_s": len(sample) / dt,
                          "sample": f"oracle.decode at every 64th position of the 8192-step loop "
                                    f"({len(sample)} steps, positions 0..8128)"}))
    else:
        raise ValueError(kind)


# Per-config oracle timing: a bounded sample of every workload, on one thread
# and on all host cores.  A sample is a list of "units" (decode: one
# (sequence, query head) row; prefill: one (token, head) row), each with its
# algorithmic bytes or flops; the full config's time is extrapolated from the
# sample's rate.  Inputs are drawn with numpy (exact bf16 values are not
# needed to time the oracle).

CPU_CONFIGS = {
    # name: (kind, shape, sample description)
    "single_step": ("decode", dict(B=1, Hq=16, Hkv=8, pos=[100]), "the whole step, 20 times"),
    "streaming_pos100": ("decode", dict(B=1, Hq=16, Hkv=8, pos=[100]), "one step at position 100, 20 times"),
    "streaming_pos1000": ("decode", dict(B=1, Hq=16, Hkv=8, pos=[1000]), "one step at position 1000, 4 times"),
    "streaming_pos4000": ("decode", dict(B=1, Hq=16, Hkv=8, pos=[4000]), "one step at position 4000"),
    "streaming_pos8000": ("decode", dict(B=1, Hq=16, Hkv=8, pos=[8000]), "one step at position 8000"),
    "ragged": ("decode", dict(B=64, Hq=32, Hkv=8, pos="ragged", sample_b=8),
               "8 of the 64 sequences, all heads"),
    "stress": ("decode", dict(B=256, Hq=64, Hkv=8, pos=[8191] * 256, sample_b=1),
               "1 of the 256 sequences, all 64 heads"),
    "prefill_prefix": ("prefill", dict(S=512, start_pos=2048, H=32, sample_rows=256),
                       "256 (token, head) rows spread over the 512 x 32"),
    "prefill": ("prefill", dict(S=2048, start_pos=0, H=32, sample_rows=256),
                "256 (token, head) rows spread over the 2048 x 32"),
}
_CPU_REPEAT = {"single_step": 20, "streaming_pos100": 20, "streaming_pos1000": 4}


def _cpu_units(name):
    """(unit list, units of the full config, unit name) for a config: each
    unit is (key, work) with key = (b, h) or (i, h)."""
    import numpy as np
    import oracle
    kind, sh, _ = CPU_CONFIGS[name]
    if kind == "decode":
        B, Hq, Hkv = sh["B"], sh["Hq"], sh["Hkv"]
        if sh["pos"] == "ragged":
            pos = np.random.default_rng(1).integers(0, L, B).tolist()
        else:
            pos = list(sh["pos"])
        bs = list(range(min(B, sh.get("sample_b", B))))
        per_row = lambda b: oracle.decode_bytes([pos[b]], Hq, Hkv, D) / Hq
        units = [((b, h), per_row(b)) for b in bs for h in range(Hq)]
        return units, float(oracle.decode_bytes(pos, Hq, Hkv, D)), pos
    S, sp, H = sh["S"], sh["start_pos"], sh["H"]
    rows = np.random.default_rng(2).choice(S * H, sh["sample_rows"], replace=False)
    units = [((int(r) // H, int(r) % H), 4.0 * 64 * (sp + int(r) // H + 1)) for r in sorted(rows)]
    return units, float(oracle.prefill_flops(S, sp, H, 64)), None


def _cpu_inputs(name, keys, pos):
    """Inputs for the given unit keys only (float32 storage of bf16-like values)."""
    import numpy as np
    kind, sh, _ = CPU_CONFIGS[name]
    rng = np.random.default_rng(sorted(CPU_CONFIGS).index(name) * 1000 + len(keys))
    if kind == "decode":
        Hq, Hkv = sh["Hq"], sh["Hkv"]
        bs = sorted({b for b, _ in keys})
        data = {}
        for b in bs:
            n = pos[b] + 1
            data[b] = (rng.standard_normal((1, Hq, D)).astype(np.float32),
                       rng.standard_normal((1, Hkv, n, D)).astype(np.float32),
                       rng.standard_normal((1, Hkv, n, D)).astype(np.float32))
        return data
    S, sp, H = sh["S"], sh["start_pos"], sh["H"]
    return (rng.standard_normal((S, H, 64)).astype(np.float32),
            rng.standard_normal((sp + S, H, 64)).astype(np.float32),
            rng.standard_normal((sp + S, H, 64)).astype(np.float32))


def _cpu_run(name, keys, pos, data):
    """The oracle on the given units; returns nothing (timed by the caller)."""
    import oracle
    kind, sh, _ = CPU_CONFIGS[name]
    if kind == "decode":
        by_b = {}
        for b, h in keys:
            by_b.setdefault(b, []).append(h)
        for b, hs in by_b.items():
            q, kc, vc = data[b]
            oracle.decode_rows(q, kc, vc, [pos[b]], 1.0 / math.sqrt(D), [(0, h) for h in hs])
    else:
        q, k, v = data
        oracle.prefill_rows(q, k, v, sh["start_pos"], 1.0 / 8.0, list(keys))


_POOL_BARRIER = None


def _pool_init(barrier):
    global _POOL_BARRIER
    _POOL_BARRIER = barrier


def _pool_job(name, keys, pos, reps):
    """One worker's share: build inputs, meet the others, time the oracle."""
    data = _cpu_inputs(name, keys, pos)
    _POOL_BARRIER.wait(timeout=300)
    t0 = time.time()
    for _ in range(reps):
        _cpu_run(name, keys, pos, data)
    return t0, time.time()


def cpu_configs_worker():
    """Every config's sample on 1 thread, then on all cores (spawn pool)."""
    import multiprocessing as mp
    ncpu = os.cpu_count() or 1
    out = {"cores_available": ncpu, "configs": {}}
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(ncpu)
    with ctx.Pool(ncpu, initializer=_pool_init, initargs=(barrier,)) as pool:
        for name in CPU_CONFIGS:
            units, full, pos = _cpu_units(name)
            keys = [k for k, _ in units]
            work = sum(w for _, w in units)
            reps = _CPU_REPEAT.get(name, 1)
            data = _cpu_inputs(name, keys, pos)
            t0 = time.perf_counter()
            for _ in range(reps):
                _cpu_run(name, keys, pos, data)
            t1 = (time.perf_counter() - t0) / reps
            del data
            chunks = [keys[i::ncpu] for i in range(ncpu)]
            spans = pool.starmap(_pool_job, [(name, c, pos, reps) for c in chunks])
            tn = (max(e for _, e in spans) - min(s0 for s0, _ in spans)) / reps
            kind = CPU_CONFIGS[name][0]
            unit, scale = ("GB/s", 1e9) if kind == "decode" else ("GFLOP/s", 1e9)
            out["configs"][name] = {
                "sample": CPU_CONFIGS[name][2], "unit": unit,
                "threads_1": {"value": round(work / t1 / scale, 4),
                              "full_config_s": round(full / (work / t1), 4)},
                f"threads_{ncpu}": {"value": round(work / tn / scale, 4),
                                    "full_config_s": round(full / (work / tn), 4)},
            }
    print(json.dumps(out))


def run_cpu_configs():
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", "configs"],
                       capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return {"error": r.stderr[-400:]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_cpu_baseline(kind="streaming"):
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker", kind],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        return {"error": r.stderr[-400:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["value"], "unit": d["unit"], "cores": 1, "kind": "oracle",
            "sample": d["sample"], "seconds": round(d["seconds"], 2),
            "steps_per_s": d["steps_per_s"]}


# -------------------------------------------------------------- clocks -----

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------ our arm ------

def _dist(set_device=None, backend="nccl"):
    """Rank setup of a replica: the GPU is LOCAL_RANK (set_device is
    torch.cuda.set_device unless a test passes its own), and with
    WORLD_SIZE > 1 a process group (NCCL on the GPU; a test may use gloo)
    for the barrier and the max-reduction of the step time only."""
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    (set_device or torch.cuda.set_device)(local)
    if ws > 1:
        import torch.distributed as dist
        if backend == "nccl":
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return ws, rank, local


def replica_seed(rank: int) -> int:
    """Seed of a replica's synthetic inputs: every rank streams its own
    sequence (weak scaling), not a copy of rank 0's."""
    return 7919 * rank


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(ws, x: float) -> float:
    """Slowest rank's value (the step time every replica must wait for)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(ws: int, units_per_rank: float, local_ms: float) -> float:
    """Whole-job throughput of ws independent replicas (weak scaling): all
    ranks' units over the slowest rank's time, in units per second."""
    ms = _max_over_ranks(ws, local_ms)
    return ws * units_per_rank / (ms * 1e-3)


class Stream:
    """The streaming job: 8192 decode steps captured in one CUDA graph.

    mode "fused": attn_decode_step_append per position (append fused into
    the decode launch) -- the product's streaming path and the timed step.
    mode "pair": attn_kv_append then attn_decode_step per position.
    mode "decode_only": attn_decode_step alone over a pre-filled cache.
    mode "rope": attn_decode_step_rope_append per position (the rotary
    embedding of q and the new key fused in as well; cos/sin rows of the
    usual base-10000 table at each position)."""

    def __init__(self, torch, ga, synth, mode="fused", seed=0):
        self.torch = torch
        dev = torch.device("cuda")
        self.q, self.k, self.v, self.pos = synth.streaming_inputs(
            steps=STEPS_STREAM, Hq=HQ, Hkv=HKV, D=D, seed=seed, device=dev)
        self.kc = torch.zeros((1, HKV, L, D), dtype=torch.bfloat16, device=dev)
        self.vc = torch.zeros_like(self.kc)
        self.ws = ga.decode_workspace(1, HQ, HKV, L, D, device=dev)
        self.outs = torch.empty((STEPS_STREAM, 1, HQ, D), dtype=torch.bfloat16, device=dev)
        self.scale = 1.0 / math.sqrt(D)
        self.ga = ga
        self.mode = mode
        if mode == "rope":
            self.cos, self.sin = synth.rope_tables(torch.arange(STEPS_STREAM), D, device=dev)
        if mode == "decode_only":  # fill the cache once so every position has its rows
            self._launch("append")
            torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self._launch(mode)  # eager warm-up
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._launch(mode)
        torch.cuda.synchronize()
        self.launches = STEPS_STREAM * (2 if mode == "pair" else 1)

    def _launch(self, mode):
        ga = self.ga
        for s in range(STEPS_STREAM):
            if mode == "fused":
                ga.attn_decode_step_append(self.q[s], self.k[s], self.v[s], self.pos[s], self.kc,
                                           self.vc, self.scale, out=self.outs[s],
                                           workspace=self.ws)
                continue
            if mode == "rope":
                ga.attn_decode_step_rope_append(self.q[s], self.k[s], self.v[s],
                                                self.cos[s:s + 1], self.sin[s:s + 1], self.pos[s],
                                                self.kc, self.vc, self.scale, out=self.outs[s],
                                                workspace=self.ws)
                continue
            if mode in ("pair", "append"):
                ga.attn_kv_append(self.k[s], self.v[s], self.pos[s], self.kc, self.vc)
            if mode in ("pair", "decode_only"):
                ga.attn_decode_step(self.q[s], self.pos[s], self.kc, self.vc, self.scale,
                                    out=self.outs[s], workspace=self.ws)

    def replay(self):
        self.graph.replay()


class _L2Flush:
    """Evicts L2 between timed launches by reading a buffer four times its
    size.  Reading leaves clean lines behind, so the timed kernel pays no
    write-back for them; a write-based flush would leave up to an L2's worth
    of dirty lines that the next kernel must write back to DRAM while it
    reads (about 15 us of HBM time on this part).  Capturable in a graph."""

    def __init__(self, torch, nbytes):
        self.torch = torch
        self.src = torch.ones(nbytes // 4, dtype=torch.int32, device="cuda")
        self.dst = torch.zeros((), dtype=torch.int64, device="cuda")

    def __call__(self):
        self.torch.sum(self.src, dim=0, dtype=self.torch.int64, out=self.dst)


def _time_graph(torch, fn, flush, reps, warm):
    for _ in range(warm):
        flush()
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    return times


def _launch_us(torch, one, flush, R=20):
    """Device time of one launch of `one` with a cold L2, in us, two ways:
    (a) a graph of R (flush, launch) pairs minus a graph of R flushes, over
    R -- the launch's time in a stream of launches, free of the event clock's
    coarse steps and of host launch latency; (b) the mean of R single
    flushed launches, each between two events (includes the launch latency
    and the event clock's granularity).  (a) is the leg's figure."""
    one()
    torch.cuda.synchronize()

    def graph(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def pairs():
        for _ in range(R):
            flush()
            one()

    def flushes():
        for _ in range(R):
            flush()
    g_pairs, g_flush = graph(pairs), graph(flushes)
    t_pairs = statistics.median(_time_graph(torch, g_pairs.replay, flush, 5, 1))
    t_flush = statistics.median(_time_graph(torch, g_flush.replay, flush, 5, 1))
    cold = (t_pairs - t_flush) * 1e3 / R
    single = statistics.mean(_time_graph(torch, one, flush, R, 3)) * 1e3
    del g_pairs, g_flush
    return cold, single


def _time_positions(torch, ga, q_of, kc, vc, ws, positions, flush, hbm, scale):
    """B=1 decode time at fixed positions: warm (graph of R back-to-back
    launches, cache in L2) and cold (each launch preceded by an L2 flush;
    flush-only time subtracted).  q_of(p) gives the query rows for p."""
    import oracle
    R = 50
    Hq, Hkv, Dd = q_of(0).shape[1], kc.shape[1], kc.shape[3]
    res = {}
    for p in positions:
        pos = torch.full((1,), p, dtype=torch.int32, device="cuda")
        out = torch.empty((1, Hq, Dd), dtype=torch.bfloat16, device="cuda")
        q = q_of(p)

        def one():
            ga.attn_decode_step(q, pos, kc, vc, scale, out=out, workspace=ws)
        one()
        torch.cuda.synchronize()
        g_warm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_warm):
            for _ in range(R):
                one()
        g_cold = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_cold):
            for _ in range(R):
                flush()
                one()
        g_flush = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_flush):
            for _ in range(R):
                flush()
        warm = statistics.median(_time_graph(torch, g_warm.replay, flush, 7, 2)) / R
        cold = (statistics.median(_time_graph(torch, g_cold.replay, flush, 7, 2)) -
                statistics.median(_time_graph(torch, g_flush.replay, flush, 7, 2))) / R
        nb = oracle.decode_bytes([p], Hq, Hkv, Dd)
        res[str(p)] = {"us_warm_l2": round(warm * 1e3, 3), "us_cold_l2": round(cold * 1e3, 3),
                       "GBs_cold": round(nb / (cold * 1e-3) / 1e9, 1),
                       "frac_cold": round(nb / (cold * 1e-3) / 1e9 / hbm, 3),
                       "frac_cold_8tbs": round(nb / (cold * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 3),
                       "bytes": nb}
    return res


def _per_position(torch, ga, st, flush, hbm):
    """The streaming workload's cache at positions 100/1000/4000/8000."""
    return _time_positions(torch, ga, lambda p: st.q[p], st.kc, st.vc, st.ws,
                           (100, 1000, 4000, 8000), flush, hbm, st.scale)


def _max_len_leg(torch, ga, flush, hbm):
    """Per-step cost against max_len: B=1, Hq=16, Hkv=8 at positions
    100/4000/8000 with max_len 8192 and with max_len 2^20 (two 2 GiB
    caches).  The step reads rows 0..pos only, so the times should agree."""
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    q = torch.randn((1, HQ, D), generator=g, device="cuda").to(torch.bfloat16)
    res = {}
    for Lx in (L, 1 << 20):
        kc = torch.empty((1, HKV, Lx, D), dtype=torch.bfloat16, device="cuda")
        vc = torch.empty_like(kc)
        for t in (kc, vc):  # N(0,1) rows, drawn in 64 Mi-element chunks
            flat = t.view(-1)
            for i in range(0, flat.numel(), 1 << 26):
                n = min(1 << 26, flat.numel() - i)
                flat[i:i + n] = torch.randn(n, generator=g, device="cuda").to(torch.bfloat16)
        ws = ga.decode_workspace(1, HQ, HKV, Lx, D)
        res[f"max_len_{Lx}"] = _time_positions(torch, ga, lambda p: q, kc, vc, ws,
                                               (100, 4000, 8000), flush, hbm, 1.0 / math.sqrt(D))
        del kc, vc
        torch.cuda.empty_cache()
    a, b = res[f"max_len_{L}"], res[f"max_len_{1 << 20}"]
    res["ratio_warm"] = {p: round(b[p]["us_warm_l2"] / a[p]["us_warm_l2"], 3) for p in a}
    res["ratio_cold"] = {p: round(b[p]["us_cold_l2"] / a[p]["us_cold_l2"], 3) for p in a}
    return res


def _decode_leg(torch, ga, synth, name, flush, hbm, B=None, Hq=None):
    """A decode workload (optionally with another batch size or head count:
    the cache shape, positions and value recipe stay the workload's)."""
    import oracle
    if B or Hq:
        w = dict(synth.generators.WORKLOADS[name])
        w.pop("kind")
        w["B"] = B or w["B"]
        w["Hq"] = Hq or w["Hq"]
        case = synth.generators.decode_case(seed=0, device="cuda", name=name, **w)
    else:
        case = synth.generators.workload_case(name, seed=0, device="cuda")
    B, Hq, Dd = case.q.shape
    Hkv, Ll = case.k_cache.shape[1], case.k_cache.shape[2]
    ga.attn_kv_append(case.k_new, case.v_new, case.positions, case.k_cache, case.v_cache)
    ws = ga.decode_workspace(B, Hq, Hkv, Ll, Dd)
    out = torch.empty_like(case.q)

    def one():
        ga.attn_decode_step(case.q, case.positions, case.k_cache, case.v_cache, case.scale,
                            out=out, workspace=ws)
    us, us1 = _launch_us(torch, one, flush)
    ms = us * 1e-3
    pos = case.positions.cpu().tolist()
    nb = oracle.decode_bytes(pos, Hq, Hkv, Dd)
    fl = oracle.decode_flops(pos, Hq, Dd)
    tc = Hq // Hkv == 16  # g = 16 runs on the tcgen05 kernel, g <= 8 on warp-level MMAs
    r = {"us": round(us, 2), "us_single_launch": round(us1, 2),
         "GBs": round(nb / (ms * 1e-3) / 1e9, 1),
         "frac_hbm": round(nb / (ms * 1e-3) / 1e9 / hbm, 3),
         "frac_hbm_8tbs": round(nb / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 3),
         "TFLOPs_tensor": round(fl / (ms * 1e-3) / 1e12, 2),
         "kernel": "decode_tc_kernel (tcgen05)" if tc else "decode kernel (mma.sync per warp)",
         "bytes": nb, "shape": {"B": B, "Hq": Hq, "Hkv": Hkv, "D": Dd, "L": Ll}}
    del case, ws, out
    torch.cuda.empty_cache()
    return r


def _append_leg(torch, ga, synth, name, flush, hbm, rope):
    """The fused step (append + decode, with or without the rotary embedding)
    on a decode workload.  Every launch rewrites the same rows with the same
    values, so repeated launches do identical work."""
    import oracle
    case = synth.generators.workload_case(name, seed=0, device="cuda")
    B, Hq, Dd = case.q.shape
    Hkv, Ll = case.k_cache.shape[1], case.k_cache.shape[2]
    ws = ga.decode_workspace(B, Hq, Hkv, Ll, Dd)
    out = torch.empty_like(case.q)
    cos, sin = synth.rope_tables(case.positions, Dd, device="cuda")

    def one():
        if rope:
            ga.attn_decode_step_rope_append(case.q, case.k_new, case.v_new, cos, sin,
                                            case.positions, case.k_cache, case.v_cache,
                                            case.scale, out=out, workspace=ws)
        else:
            ga.attn_decode_step_append(case.q, case.k_new, case.v_new, case.positions,
                                       case.k_cache, case.v_cache, case.scale, out=out,
                                       workspace=ws)
    us, us1 = _launch_us(torch, one, flush)
    ms = us * 1e-3
    pos = case.positions.cpu().tolist()
    nb = oracle.decode_bytes(pos, Hq, Hkv, Dd) + 2 * 2 * B * Hkv * Dd * 2
    r = {"us": round(us, 2), "us_single_launch": round(us1, 2),
         "GBs": round(nb / (ms * 1e-3) / 1e9, 1),
         "frac_hbm": round(nb / (ms * 1e-3) / 1e9 / hbm, 3),
         "frac_hbm_8tbs": round(nb / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 3), "bytes": nb,
         "shape": {"B": B, "Hq": Hq, "Hkv": Hkv, "D": Dd, "L": Ll}}
    del case, ws, out
    torch.cuda.empty_cache()
    return r


def _window_leg(torch, ga, synth, name, flush, hbm, window):
    """Local-window decode on a decode workload: algorithmic bytes count the
    window rows only (min(window, pos + 1) per sequence)."""
    import oracle
    case = synth.generators.workload_case(name, seed=0, device="cuda")
    B, Hq, Dd = case.q.shape
    Hkv, Ll = case.k_cache.shape[1], case.k_cache.shape[2]
    ws = ga.decode_workspace(B, Hq, Hkv, Ll, Dd)
    out = torch.empty_like(case.q)

    def one():
        ga.attn_decode_step_window(case.q, case.positions, case.k_cache, case.v_cache,
                                   case.scale, window, out=out, workspace=ws)
    us, us1 = _launch_us(torch, one, flush)
    ms = us * 1e-3
    rows_pos = [min(int(p), window - 1) for p in case.positions.cpu().tolist()]
    nb = oracle.decode_bytes(rows_pos, Hq, Hkv, Dd)
    r = {"us": round(us, 2), "us_single_launch": round(us1, 2),
         "GBs": round(nb / (ms * 1e-3) / 1e9, 1),
         "frac_hbm": round(nb / (ms * 1e-3) / 1e9 / hbm, 3),
         "frac_hbm_8tbs": round(nb / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 3), "bytes": nb, "window": window,
         "shape": {"B": B, "Hq": Hq, "Hkv": Hkv, "D": Dd, "L": Ll}}
    del case, ws, out
    torch.cuda.empty_cache()
    return r


def _multi_leg(torch, ga, synth, name, flush, hbm, S):
    """Multi-token decode on a decode workload: S new tokens per sequence
    (q and out [B, S, Hq, D], the tokens' rows already in the cache).
    Algorithmic bytes: K and V rows 0 .. pos + S - 1, plus q and out."""
    import oracle
    case = synth.generators.workload_case(name, seed=0, device="cuda")
    B, Hq, Dd = case.q.shape
    Hkv, Ll = case.k_cache.shape[1], case.k_cache.shape[2]
    pos = torch.clamp(case.positions, max=Ll - S).contiguous()
    q = torch.randn(B, S, Hq, Dd, device="cuda").to(torch.bfloat16)
    ws = ga.decode_workspace(B, S * Hq, Hkv, Ll, Dd)
    out = torch.empty_like(q)

    def one():
        ga.attn_decode_multi(q, pos, case.k_cache, case.v_cache, case.scale, out=out,
                             workspace=ws)
    us, us1 = _launch_us(torch, one, flush)
    ms = us * 1e-3
    last = [int(p) + S - 1 for p in pos.cpu().tolist()]
    nb = oracle.decode_bytes(last, Hq, Hkv, Dd) + 2 * (S - 1) * B * Hq * Dd * 2
    r = {"us": round(us, 2), "us_single_launch": round(us1, 2),
         "GBs": round(nb / (ms * 1e-3) / 1e9, 1),
         "frac_hbm": round(nb / (ms * 1e-3) / 1e9 / hbm, 3),
         "frac_hbm_8tbs": round(nb / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 3), "bytes": nb, "S": S,
         "shape": {"B": B, "Hq": Hq, "Hkv": Hkv, "D": Dd, "L": Ll}}
    del case, ws, out, q
    torch.cuda.empty_cache()
    return r


def _prefill_leg(torch, ga, synth, name, flush, tflops_peak):
    import oracle
    case = synth.generators.workload_case(name, seed=0, device="cuda")
    S, Hq, d = case.q.shape
    out = torch.empty_like(case.q)
    try:
        ga.attn_prefill_causal(case.q, case.k, case.v, case.start_pos, case.scale, out=out)
    except ga.AttnError as e:
        return {"unavailable": str(e)}

    def one():
        ga.attn_prefill_causal(case.q, case.k, case.v, case.start_pos, case.scale, out=out)
    us, us1 = _launch_us(torch, one, flush)
    ms = us * 1e-3
    fl = oracle.prefill_flops(S, case.start_pos, Hq, d)
    return {"us": round(us, 2), "us_single_launch": round(us1, 2),
            "TFLOPs": round(fl / (ms * 1e-3) / 1e12, 1),
            "frac_tensor": round(fl / (ms * 1e-3) / 1e12 / tflops_peak, 3), "flops": fl,
            "shape": {"S": S, "start_pos": case.start_pos, "Hq": Hq, "Hkv": case.k.shape[1],
                      "d": d}}


def run_ours(args):
    import torch
    import gqa_decode_attention_place_gb300 as ga
    import synth

    ws, rank, local = _dist()
    hbm, tf_burst, tf_sus, peak_src = _peaks()
    ga.load_library()
    flush = _L2Flush(torch, FLUSH_BYTES)
    st = Stream(torch, ga, synth, seed=replica_seed(rank))
    nbytes = _decode_bytes_stream()

    # ---- timed region: K replays of the streaming step -------------------
    for _ in range(max(3, args.warmup)):
        flush()
        st.replay()
    torch.cuda.synchronize()
    _barrier(ws)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    t_wall = time.perf_counter()
    ev = []
    for _ in range(args.steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        st.replay()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    _barrier(ws)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = _max_over_ranks(ws, statistics.mean(step_ms))
    status = ga.attn_read_device_status(st.ws)

    # ---- end to end: host inputs -> device -> step -> host outputs --------
    h_in = [t.cpu().pin_memory() for t in (st.q, st.k, st.v, st.pos)]
    h_out = torch.empty(st.outs.shape, dtype=st.outs.dtype).pin_memory()
    d_in = [st.q, st.k, st.v, st.pos]
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for h, dv in zip(h_in, d_in):
            dv.copy_(h, non_blocking=True)
        st.replay()
        h_out.copy_(st.outs, non_blocking=True)
        b.record()
        b.synchronize()
        if i >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    e2e = _max_over_ranks(ws, statistics.mean(e2e_ms))
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out.numel() * h_out.element_size()

    # ---- roofline of the dominant kernel ---------------------------------
    # The timed step is one launch per position of the fused append+decode
    # kernel, so its average launch is the step time / 8192.  Its algorithmic
    # bytes add the appended rows (read from k_new/v_new, written to the
    # cache) to the attention's.
    app_bytes = STEPS_STREAM * 2 * 2 * HKV * D * 2
    dec_avg_us = ms * 1e3 / STEPS_STREAM
    achieved = (nbytes + app_bytes) / (ms * 1e-3) / 1e9
    # cross-checks: the same positions as separate append/decode launches, and
    # the decode launches alone
    pair = Stream(torch, ga, synth, mode="pair", seed=1)
    pair_ms = statistics.mean(_time_graph(torch, pair.replay, flush, max(3, args.steps), 3))
    del pair
    dec = Stream(torch, ga, synth, mode="decode_only", seed=1)
    dec_ms = statistics.mean(_time_graph(torch, dec.replay, flush, max(3, args.steps), 3))
    del dec
    rope = Stream(torch, ga, synth, mode="rope", seed=1)
    rope_ms = statistics.mean(_time_graph(torch, rope.replay, flush, max(3, args.steps), 3))
    del rope

    value = replica_throughput(ws, nbytes, statistics.mean(step_ms)) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v rows)",
        "config": {"workload": "streaming decode loop: B=1, Hq=16, Hkv=8 (g=2), D=128, "
                               "max_len=8192, 8192 append+decode steps from position 0",
                   "B": 1, "Hq": HQ, "Hkv": HKV, "D": D, "max_len": L,
                   "decode_steps_per_step": STEPS_STREAM,
                   "l2": "512 MB read-based L2 flush between timed steps; inside a step the 33.5 MB "
                         "cache stays L2-resident, as the workload does on a 129 MB L2",
                   "launch": "one CUDA graph of 8192 attn_decode_step_append launches "
                             "(append fused into decode, programmatic dependent launch)",
                   "parallelism": f"replicas x{ws} (independent streams, no collective)"},
        "steps_per_s": round(ws * STEPS_STREAM / (ms * 1e-3), 1),
        "us_per_decode_step": round(ms * 1e3 / STEPS_STREAM, 3),
        "wall_s": round(wall, 3),
        "gpu_launches": args.steps * st.launches,
        "device_status": status,
        "e2e": {"value": round(ws * nbytes / (e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "roofline": {"kernel": "decode_cluster_kernel<2, 0> (mma.sync per warp on swizzled TMA tiles, append fused; clusters of 12)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 3), "traffic": TRAFFIC_BYTES_PER_LAUNCH,
                     "traffic_unit": "bytes per launch (ncu, cold cache)",
                     "peak_source": f"{peak_src} hbm_gbs",
                     "avg_launch_us": round(dec_avg_us, 3),
                     "bytes_per_launch_avg": (nbytes + app_bytes) // STEPS_STREAM,
                     "note": "the timed step's launches (one per position 0..8191); the "
                             "33.5 MB cache is L2-resident within the loop"},
        "cross_checks": {"pair_append_then_decode_ms": round(pair_ms, 3),
                         "decode_only_ms": round(dec_ms, 3),
                         "decode_only_GBs": round(nbytes / (dec_ms * 1e-3) / 1e9, 1),
                         "rope_fused_ms": round(rope_ms, 3),
                         "rope_fused_GBs": round(nbytes / (rope_ms * 1e-3) / 1e9, 1)},
    }
    if clk:
        line["clocks"] = clk
    if rank == 0 and not args.no_legs:
        legs = {"per_position": _per_position(torch, ga, st, flush, hbm)}
        del st
        torch.cuda.empty_cache()
        legs["max_len"] = _max_len_leg(torch, ga, flush, hbm)
        for name in ("ragged", "stress"):
            legs[name] = _decode_leg(torch, ga, synth, name, flush, hbm)
        # 16 query heads per KV head: the tcgen05 decode kernel
        legs["stress_g16_b32"] = _decode_leg(torch, ga, synth, "stress", flush, hbm, B=32, Hq=128)
        legs["ragged_append"] = _append_leg(torch, ga, synth, "ragged", flush, hbm, rope=False)
        legs["ragged_rope_append"] = _append_leg(torch, ga, synth, "ragged", flush, hbm,
                                                 rope=True)
        legs["ragged_window1024"] = _window_leg(torch, ga, synth, "ragged", flush, hbm, 1024)
        legs["ragged_multi_s2"] = _multi_leg(torch, ga, synth, "ragged", flush, hbm, 2)
        # the stress shapes (g = 8) with 2 new tokens: 16 heads per KV head
        legs["stress_multi_s2"] = _multi_leg(torch, ga, synth, "stress", flush, hbm, 2)
        for name in ("prefill_prefix", "prefill", "prefill_d128_chunk", "prefill_d128"):
            legs[name] = _prefill_leg(torch, ga, synth, name, flush, tf_burst)
        line["legs"] = legs
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = run_cpu_baseline("streaming")
        line["cpu_baseline"]["per_config"] = run_cpu_configs()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The oracle, as it stands, timed on the host cores (rank 0 only)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    times, vals = [], []
    info = None
    for i in range(args.warmup + args.steps):
        info = run_cpu_baseline("streaming")
        if "error" in info:
            print(json.dumps({"impl": "reference", "unavailable": info["error"][-200:]}))
            return
        if i >= args.warmup:
            times.append(info["seconds"])
            vals.append(info["value"])
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(statistics.mean(times) * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1))",
        "config": {"workload": "streaming decode loop: B=1, Hq=16, Hkv=8 (g=2), D=128, "
                               "max_len=8192, 8192 append+decode steps from position 0",
                   "sample": info["sample"]},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": info["sample"]},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_only(args):
    """A few launches of one workload, nothing else (for profiler captures)."""
    import torch
    import gqa_decode_attention_place_gb300 as ga
    import synth
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    ga.load_library()
    name = args.only
    if name == "streaming_sample" or name.startswith("position:"):
        # streaming_sample: the streaming step at every 64th position (cache
        # filled by a plain copy, then attn_decode_step_append, as the timed
        # step does); position:N: that one position, repeated
        q, k, v, pos = synth.streaming_inputs(steps=STEPS_STREAM, Hq=HQ, Hkv=HKV, D=D, seed=0,
                                              device="cuda")
        kc = k[:, 0].transpose(0, 1).contiguous().unsqueeze(0)
        vc = v[:, 0].transpose(0, 1).contiguous().unsqueeze(0)
        ws = ga.decode_workspace(1, HQ, HKV, L, D)
        out = torch.empty((1, HQ, D), dtype=torch.bfloat16, device="cuda")
        sample = (range(0, STEPS_STREAM, 64) if name == "streaming_sample"
                  else [int(name.split(":")[1])])
        for _ in range(args.reps):
            for p in sample:
                ga.attn_decode_step_append(q[p], k[p], v[p], pos[p], kc, vc, 1.0 / math.sqrt(D),
                                           out=out, workspace=ws)
        torch.cuda.synchronize()
        print(json.dumps({"only": name, "launches_per_rep": len(sample)}))
        return
    w = dict(synth.generators.WORKLOADS[name])
    if (args.batch or args.heads) and w["kind"] == "decode":
        w["B"] = args.batch or w["B"]
        w["Hq"] = args.heads or w["Hq"]
        kind = w.pop("kind")
        case = synth.generators.decode_case(seed=0, device="cuda", name=name, **w)
        w["kind"] = kind
    else:
        case = synth.generators.workload_case(name, seed=0, device="cuda")
    if w["kind"] == "decode":
        B, Hq, Dd = case.q.shape
        ws = ga.decode_workspace(B, Hq, case.k_cache.shape[1], case.k_cache.shape[2], Dd)
        out = torch.empty_like(case.q)
        ga.attn_kv_append(case.k_new, case.v_new, case.positions, case.k_cache, case.v_cache)
        for _ in range(args.reps):
            if args.window:
                ga.attn_decode_step_window(case.q, case.positions, case.k_cache, case.v_cache,
                                           case.scale, args.window, out=out, workspace=ws)
            else:
                ga.attn_decode_step(case.q, case.positions, case.k_cache, case.v_cache,
                                    case.scale, out=out, workspace=ws)
    else:
        out = torch.empty_like(case.q)
        for _ in range(args.reps):
            ga.attn_prefill_causal(case.q, case.k, case.v, case.start_pos, case.scale, out=out)
    torch.cuda.synchronize()
    print(json.dumps({"only": name, "reps": args.reps}))


def main():
    args = _args()
    if args.only:
        run_only(args)
        return
    if args.cpu_worker == "configs":
        cpu_configs_worker()
        return
    if args.cpu_worker:
        cpu_worker(args.cpu_worker)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
