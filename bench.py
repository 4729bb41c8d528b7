#!/usr/bin/env python3
"""Benchmark of the paged decode step on one GB300 (or N replicas).

One step = pa_decode over every sequence's cached context (one query per
sequence and head) followed by pa_append_kv of one new token per sequence at
position L (the slot the host block manager assigns).  The step is
idempotent (the same slot is rewritten every step), so every timed step does
the same work.  copy_blocks has no pair in this workload (the OPT-13B-shaped
batch shares no block) and is not launched.

Prints ONE JSON line (rank 0).  Key numbers:
  value      decode KV GB/s = algorithmic KV bytes read per step / step time
             (K/V inputs already resident in HBM)
  e2e        the same metric through the public Python API with host
             buffers: per step the step's inputs (q, new K/V rows, slot
             mapping, context lengths, block tables) are copied from pinned
             host memory and the attention output is copied back
  roofline   pa_decode call (decode kernel + partition reduce) timed with
             CUDA events on its stream, against the measured HBM copy peak
  cpu_baseline  the fp64 CPU oracle on the host cores (rank 0, N = 1 only)

--impl reference times the CPU oracle alone as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak) and seq-layer steps/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=["opt13b", "gqa"], default="opt13b")
    ap.add_argument("--partition", type=int, default=0, help="pa_decode partition_size (0 = default)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU baseline budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: every rank runs its own copy of the workload)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world: int):
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (x itself at world size 1)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# peaks, clocks


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        except OSError:
            pass
        finally:
            if self.path:
                try:
                    os.unlink(self.path)
                except OSError:
                    pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        mine = [r for r in rows if r[0] == str(self.device_index)] or rows
        sm = [float(r[1]) for r in mine if _isnum(r[1])]
        smax = [float(r[2]) for r in mine if _isnum(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in mine for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(mine)}


def _isnum(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


# ---------------------------------------------------------------------------
# workload


def build_workload(name: str, device):
    """Inputs of one step, resident on `device`, plus host copies where needed."""
    from paged_kv_cache_251_gb300 import workloads as wl
    from paged_kv_cache_251_gb300.blocks import BlockManager

    if name == "opt13b":
        inp = wl.decode_inputs(wl.SHAPES["opt13b"], device=device)
    else:
        inp = wl.decode_inputs(wl.SHAPES["gqa"], device=device, room_for_append=True, fill=0.95)
    s = inp.shape
    # slots of the appended token (position L of every sequence): the host
    # block manager replays each sequence's blocks in table order
    held = inp.blocks_held.tolist()
    order = [b for row, n in zip(inp.block_tables.tolist(), held) for b in row[:n]]
    used = set(order)
    rest = [b for b in range(inp.num_blocks) if b not in used]
    bm = BlockManager(inp.num_blocks, s.block_size, s.num_seqs, inp.block_tables.shape[1],
                      free_order=order + rest)
    slots = torch.empty(s.num_seqs, dtype=torch.int64)
    for i in range(s.num_seqs):
        bm.add_sequence(i)
        sl, _ = bm.extend(i, int(inp.context_lens[i]) + 1)
        slots[i] = sl[-1]
    tables, _ = bm.tables()
    assert torch.equal(tables, inp.block_tables), "block manager replay disagrees with the generated tables"
    return inp, slots


def step_bytes(inp):
    from paged_kv_cache_251_gb300 import accounting as acc
    s = inp.shape
    elt = torch.tensor([], dtype=s.dtype).element_size()
    dec = acc.decode_bytes(inp.context_lens.cpu(), s.num_heads, s.num_kv_heads, s.head_dim, s.block_size, elt,
                           out_elt_bytes=4, window=s.window)
    app = acc.append_bytes(s.num_seqs, s.num_kv_heads, s.head_dim, elt)
    return dec, app


def traffic_from_profile(kernel_hash: str):
    """dram bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "pa_decode_opt13b.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)\s+source_hash:\s*([0-9a-f]+)", text)
    if m and m.group(2) == kernel_hash:
        return int(m.group(1))
    return None


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_251_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.startswith("pa_decode") or fn in ("pa_device.cuh", "pa_api.cu"):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# CPU oracle timing


def time_oracle(inp, slots, budget_s: float, threads: int, full_first: bool = True):
    """Run the oracle step (decode of all (seq, head) rows + append) on host
    copies; repeat while within budget.  Returns (seconds per step, reps, rows)."""
    import oracle
    s = inp.shape
    q, k, v = inp.q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu()
    bt, cl = inp.block_tables.cpu(), inp.context_lens.cpu()
    kn, vn = inp.k_new.cpu(), inp.v_new.cpu()
    scale = 1.0 / math.sqrt(s.head_dim)
    times = []
    t_start = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        oracle.paged_attention(q, k, v, bt, cl, num_kv_heads=s.num_kv_heads, scale=scale, threads=threads)
        oracle.append_kv(k, v, kn, vn, slots)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start + times[-1] > budget_s or len(times) >= 20:
            break
    return statistics.median(times), len(times), s.num_seqs * s.num_heads


# ---------------------------------------------------------------------------
# arms


def run_native(args):
    world, rank, local = dist_env()
    dist_init(world)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the native arm")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from paged_kv_cache_251_gb300 import pa

    inp, slots_h = build_workload(args.workload, dev)
    s = inp.shape
    bt = inp.block_tables.to(dev)
    cl = inp.context_lens.to(dev)
    slots = slots_h.to(dev)
    out = torch.empty(inp.q.shape, dtype=torch.float32, device=dev)
    ws = pa.workspace_for(inp.q, s.block_size, bt.shape[1], s.window, args.partition)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    scale = 1.0 / math.sqrt(s.head_dim)
    dec_b, app_b = step_bytes(inp)
    kv_bytes = dec_b["kv"]
    max_parts_gt1 = pa.pa_decode_workspace_size(s.num_seqs, s.num_heads, s.head_dim, s.block_size, bt.shape[1],
                                                s.window, args.partition) > 0
    launches_per_step = (2 if max_parts_gt1 else 1) + 1

    def decode():
        pa.pa_decode(out, inp.q, inp.k_cache, inp.v_cache, bt, cl, num_kv_heads=s.num_kv_heads, scale=scale,
                     window=s.window, partition_size=args.partition, workspace=ws, err_word=err, stream=stream)

    def append():
        pa.pa_append_kv(inp.k_new, inp.v_new, slots, inp.k_cache, inp.v_cache, err_word=err, stream=stream)

    for _ in range(max(args.warmup, 0)):
        decode()
        append()
    torch.cuda.synchronize(dev)
    assert err.item() == 0, f"device error word {err.item()}"

    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ds = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    de = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        ev0.record(stream)
        for i in range(K):
            ds[i].record(stream)
            decode()
            de[i].record(stream)
            append()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.summary()
    ms_step = ev0.elapsed_time(ev1) / K
    ms_dec = statistics.mean(ds[i].elapsed_time(de[i]) for i in range(K))
    ms_step_max = max_over_ranks(ms_step, world, dev)
    assert err.item() == 0, f"device error word {err.item()}"

    # spot parity of the benchmarked output against the oracle
    parity = None
    if rank == 0:
        import oracle
        from paged_kv_cache_251_gb300 import workloads as wl
        idx = wl.permutation(4242, 1, s.num_seqs * s.num_heads)[:16]
        pairs = torch.stack([idx // s.num_heads, idx % s.num_heads], 1).to(torch.int32)
        # the cache now also holds the appended token; the decode attended L tokens
        ref = oracle.paged_attention(inp.q.cpu(), inp.k_cache.cpu(), inp.v_cache.cpu(), inp.block_tables,
                                     inp.context_lens, num_kv_heads=s.num_kv_heads, scale=scale, pairs=pairs,
                                     threads=os.cpu_count() or 1)
        got = out.cpu()[pairs[:, 0].long(), pairs[:, 1].long()].double().numpy()
        parity = float(abs(got - ref).max())

    # end to end through the public API with host buffers
    pin = lambda t: t.cpu().pin_memory()  # noqa: E731
    q_h, kn_h, vn_h = pin(inp.q), pin(inp.k_new), pin(inp.v_new)
    sl_h, cl_h, bt_h = pin(slots_h), pin(inp.context_lens), pin(inp.block_tables)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_d, kn_d, vn_d = torch.empty_like(inp.q), torch.empty_like(inp.k_new), torch.empty_like(inp.v_new)
    sl_d, cl_d, bt_d = torch.empty_like(slots), torch.empty_like(cl), torch.empty_like(bt)
    h2d = sum(t.numel() * t.element_size() for t in (q_h, kn_h, vn_h, sl_h, cl_h, bt_h))
    d2h = out_h.numel() * out_h.element_size()

    def e2e_step():
        for dst, src in ((q_d, q_h), (kn_d, kn_h), (vn_d, vn_h), (sl_d, sl_h), (cl_d, cl_h), (bt_d, bt_h)):
            dst.copy_(src, non_blocking=True)
        pa.pa_decode(out, q_d, inp.k_cache, inp.v_cache, bt_d, cl_d, num_kv_heads=s.num_kv_heads, scale=scale,
                     window=s.window, partition_size=args.partition, workspace=ws, err_word=err, stream=stream)
        pa.pa_append_kv(kn_d, vn_d, sl_d, inp.k_cache, inp.v_cache, err_word=err, stream=stream)
        out_h.copy_(out, non_blocking=True)

    for _ in range(max(args.warmup, 0)):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / K, world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        t_step, reps, rows = time_oracle(inp, slots_h, args.cpu_seconds, threads)
        cpu = {"value": kv_bytes / t_step / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"the full step ({rows} (seq, head) rows of fp64 decode + the append), "
                         f"median of {reps} runs on {threads} host threads",
               "seconds_per_step": t_step}

    peak, peak_kind = hbm_peak()
    achieved = dec_b["total"] / (ms_dec * 1e-3) / 1e9
    khash = kernel_source_hash()
    traffic = traffic_from_profile(khash)
    value = world * kv_bytes / (ms_step_max * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}[s.dtype],
        "data": "synthetic (seeded SplitMix64 / Box-Muller N(0,1) q, K, V; seeded shuffle of the block pool)",
        "config": {
            "workload": ("opt13b: 64 seqs x 40 MHA heads, head_dim 128, block 16, fp16, context ~ U[512, 2048], "
                         "exact-need pool shuffled; step = pa_decode + pa_append_kv (1 token/seq)"
                         if args.workload == "opt13b" else
                         "gqa: 256 seqs, 32 q / 8 kv heads, head_dim 128, block 16, bf16, lognormal context "
                         "(median 1024, sigma 1) clipped to [16, 8192], 95%-full shuffled pool; "
                         "step = pa_decode + pa_append_kv"),
            "num_seqs": s.num_seqs, "num_heads": s.num_heads, "num_kv_heads": s.num_kv_heads,
            "head_dim": s.head_dim, "block_size": s.block_size, "context_tokens": dec_b["attended_tokens"],
            "partition_size": args.partition or 512, "accumulate": "f32", "out_dtype": "f32",
            "l2": f"no flush: the K/V read per step ({kv_bytes / 1e9:.2f} GB) is larger than L2 (129 MB)",
            "parallelism": f"replicas x{world} (each rank its own batch)",
        },
        "seq_layer_steps_per_s": round(world * s.num_seqs / (ms_step_max * 1e-3), 1),
        "hbm_frac_of_step": round(value / peak, 4),
        "decode_ms": round(ms_dec, 5),
        "roofline": {"bound": "hbm", "kernel": "pa_decode (decode + partition reduce)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} (hbm_gbs, STREAM-style copy)",
                     "algorithmic_bytes_per_launch": dec_b["total"], "traffic": traffic,
                     "traffic_source": "profiles/pa_decode_opt13b.md" if traffic else None,
                     "source_hash": khash},
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * kv_bytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 5),
                "api": "paged_kv_cache_251_gb300.pa (ctypes binding of libpa)"},
        "gpu_launches": K * launches_per_step,
        "clocks": clk,
        "parity_sampled_max_abs": parity,
        "impl": "native",
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return  # the reference arm runs on rank 0 only
    from paged_kv_cache_251_gb300 import workloads as wl
    import oracle
    s = wl.SHAPES[args.workload]
    if args.workload == "opt13b":
        inp = wl.decode_inputs(s)
    else:
        inp = wl.decode_inputs(s, room_for_append=True, fill=0.95)
    threads = os.cpu_count() or 1
    scale = 1.0 / math.sqrt(s.head_dim)
    # size the per-step sample so the whole run stays within a few minutes
    total_steps = max(1, args.steps + args.warmup)
    probe_n = min(4, s.num_seqs)
    t0 = time.perf_counter()
    oracle.paged_attention(inp.q[:probe_n], inp.k_cache, inp.v_cache, inp.block_tables[:probe_n],
                           inp.context_lens[:probe_n], num_kv_heads=s.num_kv_heads, scale=scale, threads=threads)
    per_seq = (time.perf_counter() - t0) / probe_n
    budget = 150.0 / total_steps
    n = max(1, min(s.num_seqs, int(budget / max(per_seq, 1e-9))))
    q, bt, cl = inp.q[:n].contiguous(), inp.block_tables[:n].contiguous(), inp.context_lens[:n].contiguous()
    dec_b, _ = step_bytes(inp)
    from paged_kv_cache_251_gb300 import accounting as acc
    elt = inp.k_cache.element_size()
    kv = acc.decode_bytes(cl, s.num_heads, s.num_kv_heads, s.head_dim, s.block_size, elt)["kv"]
    for _ in range(args.warmup):
        oracle.paged_attention(q, inp.k_cache, inp.v_cache, bt, cl, num_kv_heads=s.num_kv_heads, scale=scale,
                               threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_attention(q, inp.k_cache, inp.v_cache, bt, cl, num_kv_heads=s.num_kv_heads, scale=scale,
                               threads=threads)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = kv / dt / 1e9
    sample = (f"{n} of {s.num_seqs} sequences ({n * s.num_heads} (seq, head) rows, {int(cl.sum())} context tokens) "
              f"per step, fp64 oracle on {threads} host threads")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded workload as the native arm)",
        "config": {"workload": args.workload, "num_seqs_sampled": n, "num_heads": s.num_heads,
                   "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
