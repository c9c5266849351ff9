"""Benchmark of the ReplaySSM decode path on one GB300 (or N replicas).

Default workload: the Mamba-2 layer at serving shape (nheads 128, headdim 64,
dstate 128, ngroups 8; 4 MiB FP32 state per sequence), batch 256, L = 16,
replay decode steps with the flush fused into every 16th step.  One step is
one replay decode of the whole batch (append, decay weights, record
contractions, checkpoint contraction, output, and on flush steps the fold).

Prints one JSON line (rank 0):
  value        sequences*tokens/s per layer over the K timed steps, inputs
               resident in HBM, device time (CUDA events on the launch stream)
  e2e          the same metric with each step's inputs copied from pinned host
               memory and y copied back inside the timed region
  roofline     algorithmic bytes per decode launch / its average duration
               against the measured HBM copy bandwidth
  cpu_baseline the CPU oracle (float64 stepwise recurrence) on a bounded
               sample of the same workload
`--impl reference` times the CPU oracle as the reference arm instead.

N > 1 (torchrun): every rank runs its own replica on its own GPU (the path
has no exchange step); value = all ranks' tokens / the slowest rank's time.
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

from ssm_decode_state_gb300 import bytes_model as bm  # noqa: E402
from ssm_decode_state_gb300 import inputs as gen  # noqa: E402

METRIC = "replay SSM decode tokens/s/layer at B=256; achieved HBM GB/s vs GB300 peak"
UNIT = "seq*tok/s/layer"
POOL = 32                       # distinct per-step input sets kept on the device
KERNEL_SOURCES = ["ssm_decode_state_gb300/csrc/mamba2_persist.cuh",
                  "ssm_decode_state_gb300/csrc/mamba2_persist_launch.cuh",
                  "ssm_decode_state_gb300/csrc/persist_common.cuh",
                  "ssm_decode_state_gb300/csrc/common.cuh"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def traffic_per_launch():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "replay_decode_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_sources_sha") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# --------------------------------------------------------------------------
# CPU oracle baseline (reference arm and cpu_baseline)
# --------------------------------------------------------------------------

def oracle_rate(shape: gen.Mamba2Shape, seed: int, seqs: int, steps: int):
    """Time the oracle's stepwise recurrence on `seqs` sequences x `steps`
    tokens of the workload; returns (seq*tok/s, seconds, sample text)."""
    from oracle.mamba2 import Mamba2Stepwise
    prm = gen.mamba2_params(shape, seed)
    sub = gen.Mamba2Shape(seqs, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L,
                          shape.bf16_io)
    h0 = gen.mamba2_random_state(shape, seed, batch_slice=slice(0, seqs))
    m = Mamba2Stepwise(prm.A, prm.D, shape.ngroups, h0)
    toks = [gen.mamba2_step_inputs(sub, prm, seed, t) for t in range(steps)]
    t0 = time.perf_counter()
    for st in toks:
        m.step(st.dt, st.x, st.B, st.C)
    el = time.perf_counter() - t0
    return seqs * steps / el, el, f"{seqs} sequences x {steps} decode steps of the batch-{shape.batch} shape"


def _oracle_worker(job):
    """One process of the all-cores baseline: the oracle on its own sequences."""
    os.environ["OMP_NUM_THREADS"] = "1"
    (B, H, P, N, G, L), seed, first, seqs, steps = job
    from oracle.mamba2 import Mamba2Stepwise
    shape = gen.Mamba2Shape(B, H, P, N, G, L, True)
    prm = gen.mamba2_params(shape, seed)
    sub = gen.Mamba2Shape(seqs, H, P, N, G, L, True)
    h0 = gen.mamba2_random_state(shape, seed, batch_slice=slice(first, first + seqs))
    m = Mamba2Stepwise(prm.A, prm.D, G, h0)
    toks = [gen.mamba2_step_inputs(sub, prm, seed, t) for t in range(steps)]
    t0 = time.perf_counter()
    for st in toks:
        m.step(st.dt, st.x, st.B, st.C)
    return time.perf_counter() - t0


def oracle_rate_all_cores(shape: gen.Mamba2Shape, seed: int, seqs_per_core: int, steps: int, cores: int = 0):
    """The oracle on every host core: one spawned process per core, each on its own
    `seqs_per_core` sequences (the oracle parallelises over sequences); rate =
    all processes' seq*tok over the slowest process's time."""
    import multiprocessing as mp
    cores = cores or os.cpu_count() or 1
    dims = (shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
    jobs = [(dims, seed, (i * seqs_per_core) % shape.batch, seqs_per_core, steps) for i in range(cores)]
    with mp.get_context("spawn").Pool(cores) as pool:
        times = pool.map(_oracle_worker, jobs)
    el = max(times)
    return (cores * seqs_per_core * steps / el, el, cores,
            f"{cores} processes x {seqs_per_core} sequences x {steps} decode steps of the batch-{shape.batch} shape")


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def _timed(stream, fn, steps):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for t in range(steps):
        fn(t)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def max_over_ranks(values, dist=None, device="cpu"):
    """Each value's maximum over the ranks (the slowest replica's times), after a
    barrier; one process (dist None): the values themselves."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    dist.barrier()
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def memory_report(H: int, P: int, N: int, G: int, L: int, layers: int = 24,
                  budget_bytes: int = 100 * 2 ** 30) -> dict:
    """Cache memory per sequence and layer for the replay variants against the
    conventional state, and the sequences a budget holds for `layers` SSM layers."""
    kw = dict(nheads=H, headdim=P, dstate=N, ngroups=G, L=L)
    out = {"layers": layers, "budget_GiB": budget_bytes / 2 ** 30}
    for name, extra in (("fp32", {}), ("fp32_fp8_copy", {"read_copy": 1}),
                        ("fp16_nvfp4_copy", {"read_copy": 2, "ckpt_f16": True})):
        c = bm.mamba2_cache_bytes(**kw, **extra)
        out[name] = {"bytes_per_seq_layer": c["total"], "ring_bytes": c["ring"],
                     "sequences": bm.sequences_that_fit(budget_bytes, layers, **kw, **extra)["replay"]}
    out["conventional"] = {"bytes_per_seq_layer": bm.mamba2_cache_bytes(**kw)["conventional"],
                           "sequences": bm.sequences_that_fit(budget_bytes, layers, **kw)["conventional"]}
    return out


def period_weighted(split: dict, L: int, batch: int, world: int = 1) -> dict | None:
    """Step time over one whole flush period from the per-step medians,
    ((L - 1) non-flush + 1 flush) / L, and its throughput: a figure that does
    not depend on where the timed window falls in the period."""
    if not split.get("nonflush") or not split.get("flush"):
        return None
    us = ((L - 1) * statistics.median(split["nonflush"]) + statistics.median(split["flush"])) / L
    return {"us_per_step": round(us, 2), "value": round(world * batch / (us / 1e6), 1)}


def replica_value(world: int, units_per_rank: float, ms: float) -> float:
    """Whole-job throughput of `world` independent replicas: every rank's units
    over the slowest rank's time (ms)."""
    return world * units_per_rank / (ms / 1e3)


def run_native(args, rank, world, local_rank):
    import torch
    import __graft_entry__
    dist = None
    if world > 1:
        import torch.distributed as dist
    if rank == 0:
        __graft_entry__.build()
    if dist is not None:
        dist.barrier()
    from ssm_decode_state_gb300 import replayssm as rs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = gen.workloads()["mamba2_b256"]
    shape = w.shape
    if args.batch:
        shape = gen.Mamba2Shape(args.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups,
                                shape.L, shape.bf16_io)
    B, H, P, N, G, L = shape.batch, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L
    seed = w.seed + 17 * rank
    prm = gen.mamba2_params(shape, seed)
    dims = rs.mamba2_dims(B, H, P, N, G, L, read_copy=0, io_bf16=True)

    gcuda = torch.Generator(device=dev)
    gcuda.manual_seed(seed)
    ckpt = torch.randn(B, H, P, N, device=dev, generator=gcuda).mul_(0.1)   # N(0, 0.1^2)
    cache = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D), ckpt=ckpt, device=dev)

    # pool of per-step inputs (seeded, the workload's distributions)
    host = [gen.mamba2_step_inputs(shape, prm, seed, t) for t in range(POOL)]
    pool = [(torch.from_numpy(s.dt).to(dev), torch.from_numpy(s.x).to(torch.bfloat16).to(dev),
             torch.from_numpy(s.B).to(torch.bfloat16).to(dev), torch.from_numpy(s.C).to(torch.bfloat16).to(dev))
            for s in host]
    y = torch.empty(B, H, P, device=dev)
    stream = torch.cuda.current_stream(dev)
    u = bm.mamba2_units(H, P, N, G)

    K, W = args.steps, args.warmup
    for t in range(W):
        rs.decode(cache, *pool[t % POOL], y=y)
    torch.cuda.synchronize(dev)
    start_len = int(cache.ring_len[0].item())
    alg_bytes, ln, nflush = 0, start_len, 0
    for _ in range(K):
        alg_bytes += bm.mamba2_replay_decode(u, ln, L) * B
        if ln + 1 >= L:
            ln, nflush = 0, nflush + 1
        else:
            ln += 1

    sampler = ClockSampler(local_rank)
    sampler.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ms = _timed(stream, lambda t: rs.decode(cache, *pool[(W + t) % POOL], y=y), K)
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    assert int(cache.err.item()) == 0, "device error word set"

    # ---- per-step split: each launch between its own events, two flush periods
    split = {"nonflush": [], "flush": []}
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2 * L)]
    ln0 = int(cache.ring_len[0].item())
    kinds = []
    for i, (s0, s1) in enumerate(evs):
        kinds.append("flush" if (ln0 + i) % L == L - 1 else "nonflush")
        s0.record(stream)
        rs.decode(cache, *pool[i % POOL], y=y)
        s1.record(stream)
    torch.cuda.synchronize(dev)
    for kind, (s0, s1) in zip(kinds, evs):
        split[kind].append(s0.elapsed_time(s1) * 1e3)

    # ---- staggered flushes: sequence b's ring length is set to b mod L over the records
    # already in its ring (real records of the earlier steps), so 1/L of the sequences
    # fold on every step instead of all of them on every L-th
    import numpy as np
    cache.ring_head.zero_()
    cache.ring_len.copy_(torch.arange(B, device=dev, dtype=torch.int32) % L)
    torch.cuda.synchronize(dev)
    Ks = max(L, (min(K, 512) // L) * L)
    lens = np.arange(B) % L
    stag_bytes = 0
    for _ in range(Ks):
        stag_bytes += sum(bm.mamba2_replay_decode(u, int(l), L) for l in lens)
        lens = np.where(lens + 1 >= L, 0, lens + 1)
    stag_ms = _timed(stream, lambda t: rs.decode(cache, *pool[t % POOL], y=y), Ks)
    assert int(cache.err.item()) == 0
    staggered = {"us_per_step": round(stag_ms * 1e3 / Ks, 1), "value": round(replica_value(world, B * Ks, stag_ms), 1),
                 "alg_GBps": round(stag_bytes / (stag_ms / 1e3) / 1e9, 1), "steps": Ks,
                 "ring_len_at_start": "b mod L"}
    cache.ring_len.zero_()                      # the later measurements start aligned again
    torch.cuda.synchronize(dev)

    # ---- conventional in-place decode on the same shape (comparison path)
    conv_ms = 0.0
    if not args.no_conventional:
        state = ckpt.clone()
        for t in range(W):
            rs.conventional_decode(dims, state, cache.A, cache.D, *pool[t % POOL], y=y)
        torch.cuda.synchronize(dev)
        conv_ms = _timed(stream, lambda t: rs.conventional_decode(dims, state, cache.A, cache.D,
                                                                  *pool[(W + t) % POOL], y=y), K)
        del state

    # ---- end to end: every step's inputs from pinned host memory and its y back to
    # pinned host memory, inside the timed region.  The copies run on a second stream,
    # double-buffered and ordered by events, so step t+1's inputs and step t's y move
    # while the next decode computes (how a serving loop would pipeline them).
    hpin = [tuple(t.to("cpu").pin_memory() for t in p) for p in pool]
    ypin = [torch.empty(B, H, P).pin_memory() for _ in range(2)]
    dbufs = [tuple(torch.empty_like(t) for t in pool[0]) for _ in range(2)]
    ys = [torch.empty_like(y) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in hpin[0])
    d2h = ypin[0].numel() * ypin[0].element_size()
    Ke = max(16, min(K, args.e2e_steps))
    cstream = torch.cuda.Stream(dev)

    def e2e_run(nsteps, first):
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_used = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        cstream.wait_stream(stream)
        with torch.cuda.stream(cstream):
            for d_, h_ in zip(dbufs[0], hpin[first % POOL]):
                d_.copy_(h_, non_blocking=True)
        ev_in[0].record(cstream)
        for t in range(nsteps):
            s_, n_ = t % 2, (t + 1) % 2
            if t + 1 < nsteps:
                if t >= 1:
                    cstream.wait_event(ev_used[n_])      # decode t-1 is done with slot n_
                with torch.cuda.stream(cstream):
                    for d_, h_ in zip(dbufs[n_], hpin[(first + t + 1) % POOL]):
                        d_.copy_(h_, non_blocking=True)
                ev_in[n_].record(cstream)
            stream.wait_event(ev_in[s_])
            if t >= 2:
                stream.wait_event(ev_out[s_])            # y of step t-2 has reached the host
            rs.decode(cache, *dbufs[s_], y=ys[s_])
            ev_used[s_].record(stream)
            cstream.wait_event(ev_used[s_])
            with torch.cuda.stream(cstream):
                ypin[s_].copy_(ys[s_], non_blocking=True)
            ev_out[s_].record(cstream)
        stream.wait_stream(cstream)

    e2e_run(W, 0)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    e2e_run(Ke, W)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1)

    ms, e2e_ms, conv_ms = max_over_ranks([ms, e2e_ms, conv_ms], dist, dev)
    if rank != 0:
        return
    value = replica_value(world, B * K, ms)
    per_launch_s = ms / 1e3 / K
    achieved = alg_bytes / K / per_launch_s / 1e9
    peak, peak_src = peaks()
    memory = memory_report(H, P, N, G, L)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": round(ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded; distributions of the workload)",
        "config": {"workload": f"mamba2 replay decode B={B} H={H} P={P} N={N} G={G} L={L}",
                   "batch": B, "state_bytes_per_seq": H * P * N * 4, "io": "bf16 x/B/C, f32 dt/A/D/y",
                   "flush_steps_timed": nflush, "ring_len_at_start": start_len,
                   "l2": "no flush needed: 1 GiB of checkpoint per step > 129 MB L2",
                   "parallelism": f"{world} independent replicas" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic_per_launch(),
                     "kernel": "m2_decode_persistent",
                     "alg_bytes_per_launch": int(alg_bytes / K),
                     "peak_source": f"{peak_src} hbm_gbs (copy), of measured"},
        "e2e": {"value": round(replica_value(world, B * Ke, e2e_ms), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
                "copies": "second stream, double-buffered, overlapping the decodes"},
        "step_us": {k: round(statistics.median(v), 1) for k, v in split.items() if v},
        "period_weighted": period_weighted(split, L, B, world),
        "staggered": staggered,
        "gpu_launches": K,
        "clocks": clocks,
        "memory": memory,
    }
    if conv_ms:
        line["conventional"] = {"value": round(replica_value(world, B * K, conv_ms), 1),
                                "ms_per_step": round(conv_ms / K, 5),
                                "alg_bytes_per_launch": bm.mamba2_conventional(u) * B,
                                "replay_speedup": round(conv_ms / ms, 3)}
    if world == 1 and not args.no_rows:
        line["rows"] = measure_rows(rs, dev, args.row_steps, 8)
    if world == 1 and not args.no_cpu_baseline:
        rate, el, sample = oracle_rate(shape, seed, args.cpu_seqs, args.cpu_steps)
        line["cpu_baseline_1core"] = {"value": round(rate, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                                      "sample": sample, "seconds": round(el, 2)}
        rate, el, cores, sample = oracle_rate_all_cores(shape, seed, args.cpu_seqs, args.cpu_steps)
        line["cpu_baseline"] = {"value": round(rate, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": sample, "seconds": round(el, 2)}
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """Replay vs conventional decode across batch sizes (device time, CUDA
    graphs of `steps` launches; inputs resident).  Batches up to 8 keep the
    whole state in L2 and are labelled so."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from ssm_decode_state_gb300 import replayssm as rs
    dev = torch.device("cuda", 0)
    w = gen.workloads()["mamba2_b256"]
    out = []
    for B in [int(v) for v in args.sweep.split(",")]:
        shape = gen.Mamba2Shape(B, w.shape.nheads, w.shape.headdim, w.shape.dstate, w.shape.ngroups,
                                w.shape.L, True)
        prm = gen.mamba2_params(shape, w.seed)
        dims = rs.mamba2_dims(B, shape.nheads, shape.headdim, shape.dstate, shape.ngroups, shape.L)
        g = torch.Generator(device=dev)
        g.manual_seed(w.seed)
        ck = torch.randn(B, shape.nheads, shape.headdim, shape.dstate, device=dev, generator=g).mul_(0.1)
        cache = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D), ckpt=ck, device=dev)
        state = ck.clone()
        pool = []
        for t in range(4):
            st = gen.mamba2_step_inputs(shape, prm, w.seed, t)
            pool.append((torch.from_numpy(st.dt).to(dev), torch.from_numpy(st.x).to(torch.bfloat16).to(dev),
                         torch.from_numpy(st.B).to(torch.bfloat16).to(dev),
                         torch.from_numpy(st.C).to(torch.bfloat16).to(dev)))
        y = torch.empty(B, shape.nheads, shape.headdim, device=dev)
        steps = args.steps
        res = {"batch": B, "state_MiB": B * 4, "l2_resident": B * 4 <= 64}
        for name, fn in (("replay", lambda t: rs.decode(cache, *pool[t % 4], y=y)),
                         ("conventional", lambda t: rs.conventional_decode(dims, state, cache.A, cache.D,
                                                                           *pool[t % 4], y=y))):
            for t in range(args.warmup):
                fn(t)
            torch.cuda.synchronize()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(gr, stream=s):
                    for t in range(steps):
                        fn(t)
            torch.cuda.synchronize()
            gr.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            res[name + "_us_per_step"] = round(ms * 1e3 / steps, 2)
            res[name + "_tok_s"] = round(B * steps / (ms / 1e3), 1)
            del gr
        res["replay_speedup"] = round(res["conventional_us_per_step"] / res["replay_us_per_step"], 3)
        out.append(res)
        assert int(cache.err.item()) == 0
        del cache, state, ck
        torch.cuda.empty_cache()
    print(json.dumps({"sweep": out}), flush=True)


ROWS = ("fp8", "nvfp4", "f16ckpt", "f16ckpt_nvfp4", "verify", "gdn", "gdn_verify")


def measure_rows(rs, dev, steps, warmup, which=ROWS):
    """The other hot-path rows, each on its own workload shape: FP8-read decode
    (batch 256), speculative verify + rollback (batch 512, T = 4) against the
    snapshot-per-draft path, Gated DeltaNet decode (batch 256) against its
    in-place decode.  Device time per step and algorithmic GB/s."""
    import numpy as np
    import torch
    wl = gen.workloads()
    out = {}
    stream = torch.cuda.current_stream(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(wl["mamba2_fp8read_b256"].seed)

    def dev_step(st):
        return (torch.from_numpy(st.dt).to(dev), torch.from_numpy(st.x).to(torch.bfloat16).to(dev),
                torch.from_numpy(st.B).to(torch.bfloat16).to(dev), torch.from_numpy(st.C).to(torch.bfloat16).to(dev))

    for rc, ckf, name, wname in ((1, False, "fp8", "mamba2_fp8read_b256"), (2, False, "nvfp4", "mamba2_nvfp4read_b256"),
                                 (0, True, "f16ckpt", "mamba2_f16ckpt_b256"),
                                 (2, True, "f16ckpt_nvfp4", "mamba2_f16ckpt_b256")):
        if name not in which:
            continue
        # ---- FP8 or NVFP4 read copy, and / or an FP16 checkpoint (stochastic rounding), batch 256
        w = wl[wname]
        sh = w.shape
        prm = gen.mamba2_params(sh, w.seed)
        dims = rs.mamba2_dims(sh.batch, sh.nheads, sh.headdim, sh.dstate, sh.ngroups, sh.L, read_copy=rc,
                              ckpt_f16=ckf)
        ck = torch.randn(sh.batch, sh.nheads, sh.headdim, sh.dstate, device=dev, generator=g).mul_(0.1)
        if ckf:
            ck = ck.half()
        cache = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D), ckpt=ck, device=dev)
        if rc:
            rs.requant(cache)
        pool = [dev_step(gen.mamba2_step_inputs(sh, prm, w.seed, t)) for t in range(8)]
        y = torch.empty(sh.batch, sh.nheads, sh.headdim, device=dev)
        for t in range(warmup):
            rs.decode(cache, *pool[t % 8], y=y)
        torch.cuda.synchronize(dev)
        ln = int(cache.ring_len[0].item())
        u = bm.mamba2_units(sh.nheads, sh.headdim, sh.dstate, sh.ngroups)
        K = (steps // sh.L) * sh.L
        alg = 0
        for _ in range(K):
            alg += bm.mamba2_replay_decode(u, ln, sh.L, read_copy=rc, ckpt_f16=ckf) * sh.batch
            ln = 0 if ln + 1 >= sh.L else ln + 1
        ms = _timed(stream, lambda t: rs.decode(cache, *pool[t % 8], y=y), K)
        assert int(cache.err.item()) == 0
        # per-step split over two flush periods, each launch between its own events
        ln0 = int(cache.ring_len[0].item())
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2 * sh.L)]
        for i, (s0, s1) in enumerate(evs):
            s0.record(stream)
            rs.decode(cache, *pool[i % 8], y=y)
            s1.record(stream)
        torch.cuda.synchronize(dev)
        split = {"nonflush": [], "flush": []}
        for i, (s0, s1) in enumerate(evs):
            split["flush" if (ln0 + i) % sh.L == sh.L - 1 else "nonflush"].append(s0.elapsed_time(s1) * 1e3)
        out[f"{name}_read_decode_b256"] = {"us_per_step": round(ms * 1e3 / K, 1),
                                           "seq_tok_s": round(sh.batch * K / (ms / 1e3), 1),
                                           "alg_GBps": round(alg / (ms / 1e3) / 1e9, 1),
                                           "step_us": {k: round(statistics.median(v), 1) for k, v in split.items()}}
        del cache, ck

    if "verify" in which:
        # ---- verify T = 4 + rollback, batch 512, and the snapshot-per-draft path
        w = wl["mamba2_verify_b512_T4"]
        sh, T = w.shape, w.T
        u = bm.mamba2_units(sh.nheads, sh.headdim, sh.dstate, sh.ngroups)
        prm = gen.mamba2_params(sh, w.seed)
        dims = rs.mamba2_dims(sh.batch, sh.nheads, sh.headdim, sh.dstate, sh.ngroups, sh.L)
        ck = torch.randn(sh.batch, sh.nheads, sh.headdim, sh.dstate, device=dev, generator=g).mul_(0.1)
        cache = rs.mamba2_cache(dims, torch.from_numpy(prm.A), torch.from_numpy(prm.D), ckpt=ck, device=dev)
        drafts = [dev_step(gen.mamba2_draft_inputs(sh, prm, w.seed, t, T)) for t in range(4)]
        accs = [gen.accepted_counts(sh.batch, T, w.seed, t) for t in range(steps + warmup)]
        accd = [torch.from_numpy(a).to(dev) for a in accs]
        y = torch.empty(sh.batch, T, sh.nheads, sh.headdim, device=dev)

        def vstep(t):
            rs.verify(cache, *drafts[t % 4], y=y)
            rs.rollback(cache, T, accd[t])

        for t in range(warmup):
            vstep(t)
        torch.cuda.synchronize(dev)
        lens = cache.ring_len.cpu().numpy().astype(np.int64)
        alg = 0
        for t in range(warmup, warmup + steps):
            alg += sum(bm.mamba2_verify(u, int(l), T, sh.L) for l in lens)
            lens = np.where(lens + T > sh.L, 0, lens) + T - (T - accs[t])
        ms = _timed(stream, lambda t: vstep(warmup + t), steps)
        assert int(cache.err.item()) == 0
        row = {"us_per_step": round(ms * 1e3 / steps, 1), "seq_verify_s": round(sh.batch * steps / (ms / 1e3), 1),
               "alg_GBps": round(alg / (ms / 1e3) / 1e9, 1)}
        del cache
        pool_t = torch.empty((sh.batch, T + 1) + tuple(ck.shape[1:]), device=dev)
        pool_t[:, 0] = ck
        del ck
        slot = torch.zeros(sh.batch, dtype=torch.int32, device=dev)
        err = torch.zeros(1, dtype=torch.int32, device=dev)
        Ad = torch.from_numpy(prm.A).to(dev)
        Dd = torch.from_numpy(prm.D).to(dev)

        def cstep(t):
            rs.conventional_verify(dims, pool_t, slot, Ad, Dd, *drafts[t % 4], err, y=y)
            rs.conventional_select(slot, T, accd[t], err)

        for t in range(warmup):
            cstep(t)
        ms_c = _timed(stream, lambda t: cstep(warmup + t), steps)
        row["snapshot_us_per_step"] = round(ms_c * 1e3 / steps, 1)
        row["snapshot_alg_GBps"] = round(bm.mamba2_conventional_verify(u, T) * sh.batch / (ms_c / steps / 1e3) / 1e9, 1)
        row["replay_speedup"] = round(ms_c / ms, 3)
        out["verify_T4_b512"] = row
        del pool_t

    if "gdn" in which:
        # ---- Gated DeltaNet, batch 256
        w = wl["gdn_b256"]
        sh = w.shape
        dims = rs.gdn_dims(sh.batch, sh.nheads, sh.dk, sh.dv, sh.L)
        S0 = torch.randn(sh.batch, sh.nheads, sh.dv, sh.dk, device=dev, generator=g).mul_(0.1)
        cache = rs.gdn_cache(dims, ckpt=S0, device=dev)
        state = S0.clone()
        gp = []
        for t in range(8):
            st = gen.gdn_step_inputs(sh, w.seed, t)
            gp.append(tuple(torch.from_numpy(a).to(torch.bfloat16).to(dev) for a in (st.q, st.k, st.v))
                      + (torch.from_numpy(st.alpha).to(dev), torch.from_numpy(st.beta).to(dev)))
        o = torch.empty(sh.batch, sh.nheads, sh.dv, device=dev)
        for t in range(warmup):
            rs.gdn_decode(cache, *gp[t % 8], o=o)
        torch.cuda.synchronize(dev)
        gu = bm.gdn_units(sh.nheads, sh.dk, sh.dv)
        ln = int(cache.ring_len[0].item())
        K = (steps // sh.L) * sh.L
        alg = 0
        for _ in range(K):
            alg += bm.gdn_replay_decode(gu, ln, sh.L) * sh.batch
            ln = 0 if ln + 1 >= sh.L else ln + 1
        ms = _timed(stream, lambda t: rs.gdn_decode(cache, *gp[t % 8], o=o), K)
        assert int(cache.err.item()) == 0
        # per-step split over two flush periods, each call (fold and decode kernels) between its own events
        ln0 = int(cache.ring_len[0].item())
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2 * sh.L)]
        for i, (s0, s1) in enumerate(evs):
            s0.record(stream)
            rs.gdn_decode(cache, *gp[i % 8], o=o)
            s1.record(stream)
        torch.cuda.synchronize(dev)
        split = {"nonflush": [], "flush": []}
        for i, (s0, s1) in enumerate(evs):
            split["flush" if (ln0 + i) % sh.L == sh.L - 1 else "nonflush"].append(s0.elapsed_time(s1) * 1e3)
        ms_c = _timed(stream, lambda t: rs.gdn_conventional_decode(dims, state, *gp[t % 8], o=o), K)
        assert int(cache.err.item()) == 0
        out["gdn_decode_b256"] = {"us_per_step": round(ms * 1e3 / K, 1), "seq_tok_s": round(sh.batch * K / (ms / 1e3), 1),
                                  "alg_GBps": round(alg / (ms / 1e3) / 1e9, 1),
                                  "step_us": {k: round(statistics.median(v), 1) for k, v in split.items()},
                                  "conventional_us_per_step": round(ms_c * 1e3 / K, 1),
                                  "replay_speedup": round(ms_c / ms, 3)}
    if "gdn_verify" in which:
        # ---- Gated DeltaNet verify of 4 drafts + rollback, batch 256
        w = wl["gdn_verify_b256_T4"]
        sh, T = w.shape, w.T
        dims = rs.gdn_dims(sh.batch, sh.nheads, sh.dk, sh.dv, sh.L)
        S0 = torch.randn(sh.batch, sh.nheads, sh.dv, sh.dk, device=dev, generator=g).mul_(0.1)
        cache = rs.gdn_cache(dims, ckpt=S0, device=dev)
        drafts = []
        for t in range(4):
            st = gen.gdn_draft_inputs(sh, w.seed, t, T)
            drafts.append(tuple(torch.from_numpy(a).to(torch.bfloat16).to(dev) for a in (st.q, st.k, st.v))
                          + (torch.from_numpy(st.alpha).to(dev), torch.from_numpy(st.beta).to(dev)))
        accs = [gen.accepted_counts(sh.batch, T, w.seed, t) for t in range(steps + warmup)]
        accd = [torch.from_numpy(a).to(dev) for a in accs]
        o = torch.empty(sh.batch, T, sh.nheads, sh.dv, device=dev)

        def gvstep(t):
            rs.gdn_verify(cache, *drafts[t % 4], o=o)
            rs.gdn_rollback(cache, T, accd[t])

        for t in range(warmup):
            gvstep(t)
        torch.cuda.synchronize(dev)
        gu = bm.gdn_units(sh.nheads, sh.dk, sh.dv)
        lens = cache.ring_len.cpu().numpy().astype(np.int64)
        alg = 0
        for t in range(warmup, warmup + steps):
            alg += sum(bm.gdn_verify(gu, int(l), T, sh.L) for l in lens)
            lens = np.where(lens + T > sh.L, 0, lens) + T - (T - accs[t])
        ms = _timed(stream, lambda t: gvstep(warmup + t), steps)
        assert int(cache.err.item()) == 0
        # context: T in-place decodes of a state copy (what scoring the drafts costs a
        # conventional step without the per-draft snapshots its rollback would need)
        state = S0.clone()
        o1 = torch.empty(sh.batch, sh.nheads, sh.dv, device=dev)
        step_in = [tuple(a[:, i].contiguous() for a in drafts[0]) for i in range(T)]
        ms_c = _timed(stream, lambda t: [rs.gdn_conventional_decode(dims, state, *step_in[i], o=o1)
                                         for i in range(T)], steps)
        out["gdn_verify_T4_b256"] = {"us_per_step": round(ms * 1e3 / steps, 1),
                                     "seq_verify_s": round(sh.batch * steps / (ms / 1e3), 1),
                                     "alg_GBps": round(alg / (ms / 1e3) / 1e9, 1),
                                     "T_inplace_decodes_us": round(ms_c * 1e3 / steps, 1)}
        del cache, state
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = gen.workloads()["mamba2_b256"]
    shape = w.shape
    seqs = args.cpu_seqs
    steps = max(1, min(args.cpu_steps, max(args.steps, 1)))
    oracle_rate(shape, w.seed, 1, 2)                  # warm-up pass, untimed
    # every host core: one spawned oracle process per core on its own sequences
    rate, el, cores, sample = oracle_rate_all_cores(shape, w.seed, seqs, steps)
    line = {
        "metric": METRIC, "value": round(rate, 3), "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"mamba2 replay decode B={shape.batch} H={shape.nheads} P={shape.headdim} "
                               f"N={shape.dstate} G={shape.ngroups} L={shape.L}",
                   "batch": shape.batch},
        "impl": "reference",
        "cpu_baseline": {"value": round(rate, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(rate, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2048)
    ap.add_argument("--warmup", type=int, default=32)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=512)
    ap.add_argument("--cpu-seqs", type=int, default=8)
    ap.add_argument("--cpu-steps", type=int, default=200)
    ap.add_argument("--no-conventional", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-rows", action="store_true", help="skip the FP8 / verify / GDN rows")
    ap.add_argument("--row-steps", type=int, default=128)
    ap.add_argument("--row", choices=ROWS, default="",
                    help="run only this row (FP8-read decode, verify, GDN) and print it")
    ap.add_argument("--sweep", type=str, default="",
                    help="comma-separated batch sizes: replay vs conventional table instead of the bench line")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.row:
        import torch
        import __graft_entry__
        __graft_entry__.build()
        from ssm_decode_state_gb300 import replayssm as rs
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        print(json.dumps({"rows": measure_rows(rs, dev, args.row_steps, args.warmup, (args.row,))}), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_native(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
