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
  cache_ops  pa_append_kv (and pa_copy_blocks where the step copies blocks):
             time per call, algorithmic bytes and GB/s, from CUDA events
             around each call in a second loop of the same steps (outside
             the timed region, so the events add nothing to it)

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
L2_FLUSH_BYTES = 256 * 1024 * 1024


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=["opt13b", "gqa", "window", "prefix_bs8", "prefix_bs16",
                                           "prefix_bs32", "tiny", "tiny_scaled", "swap"], default="opt13b")
    ap.add_argument("--partition", type=int, default=0, help="pa_decode partition_size (0 = default)")
    ap.add_argument("--shared-prefix", action="store_true",
                    help="prefix workloads: decode with pa_decode_shared_prefix (shared blocks read once per group)")
    ap.add_argument("--table", choices=["shuffled", "identity", "contiguous"], default="shuffled",
                    help="block hand-out order (identity: each sequence's blocks adjacent in memory; contiguous: "
                         "the same values in non-paged [N][H_kv][L][d] caches decoded by pa_decode_contiguous, "
                         "no block table and no append; opt13b / gqa / tiny_scaled)")
    ap.add_argument("--kv-format", choices=["native", "int8", "e4m3"], default="native",
                    help="opt13b / gqa / tiny_scaled: 8-bit cache (codes + one fp32 scale per row), decoded by "
                         "pa_decode_quant and appended by pa_append_kv_quant")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU baseline budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-others", action="store_true",
                    help="default run: skip the timing of the other workloads (other_workloads in the JSON line)")
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
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while active
    (the bench keeps the GPU busy with the timed step for the whole window)."""

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
# workloads: each defines one step on the GPU, its bytes, its end-to-end form
# (host buffers) and the oracle's version of the same step


class Step:
    """One workload's step.  Tensors the step reads are resident on the GPU;
    `host` holds pinned host copies of the per-step inputs for the end-to-end
    measurement."""

    name = ""
    description = ""

    def __init__(self, device, partition):
        self.device = device
        self.partition = partition
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    # the parts of a step, enqueued on `stream`
    def pre(self, stream):
        pass

    def decode(self, stream):
        raise NotImplementedError

    def post(self, stream):
        pass

    append_first = False   # prefix sharing writes the new tokens before it decodes
    append_bytes = 0       # algorithmic bytes of the step's append
    copy_bytes = 0         # and of its block copies (0: the step copies nothing)

    def run(self, stream, events=None):
        """One step; `events` maps a part of it ("copy", "append", "decode") to
        the (start, end) CUDA events that bracket that part."""
        ev = events or {}

        def part(name, fn):
            e = ev.get(name)
            if e:
                e[0].record(stream)
            fn(stream)
            if e:
                e[1].record(stream)

        part("copy", self.pre)
        if self.append_first:
            part("append", self.post)
        part("decode", self.decode)
        if not self.append_first:
            part("append", self.post)


def _elt(dtype):
    return torch.tensor([], dtype=dtype).element_size()


def describe(name, kv_format=None, tokens=None, pairs=None, shared=False):
    """The workload's description (the same words in both arms' JSON lines)."""
    if name == "tiny":
        d = ("tiny: 4 seqs x 4 MHA heads, head_dim 64, block 16, fp32, context ~ U[1, 100], "
             "64-block pool shuffled; step = pa_decode + pa_append_kv (launch-bound by size)")
    elif name == "tiny_scaled":
        d = ("tiny_scaled: the tiny shape (4 MHA heads, head_dim 64, block 16, fp32) with 4096 "
             "seqs, context ~ U[1, 2048], exact-need pool shuffled; step = pa_decode + pa_append_kv")
    elif name == "opt13b":
        d = ("opt13b: 64 seqs x 40 MHA heads, head_dim 128, block 16, fp16, context ~ U[512, 2048], "
             "exact-need pool shuffled; step = pa_decode + pa_append_kv (1 token/seq)")
    elif name == "gqa":
        d = ("gqa: 256 seqs, 32 q / 8 kv heads, head_dim 128, block 16, bf16, lognormal context "
             "(median 1024, sigma 1) clipped to [16, 8192], 95%-full shuffled pool; "
             "step = pa_decode + pa_append_kv (1 token/seq)")
    elif name == "window":
        d = ("window: 4 seqs x 131072 logical tokens, 32 q / 8 kv heads, head_dim 128, bf16, block 16, "
             "window 32768 over rings of 2049 physical blocks (table rewrite, no K/V movement), "
             "512-token partitions + LSE reduce; step = pa_decode + pa_append_kv (1 token/seq)")
    else:
        bs = int(name[len("prefix_bs"):].split("_")[0])
        d = (f"prefix: 32 prompts x 2000 tokens shared by 8 samples each (256 samples), U{{1..256}} new "
             f"tokens per sample ({tokens} in all), 40 MHA heads, head_dim 128, fp16, "
             f"block {bs}, {pairs} copy-on-write pairs; step = pa_copy_blocks + pa_append_kv + pa_decode")
        if shared:
            d += "; decode by pa_decode_shared_prefix (each prompt's whole blocks read once per group)"
    if kv_format:
        d += (f"; 8-bit cache: {kv_format.upper()} codes + one fp32 scale per (token, kv head) row in "
              f"(block, kv head) pages, step = pa_decode_quant + pa_append_kv_quant")
    return d


def _decode_inputs(name, device, shuffle):
    """The seeded inputs of the opt13b / gqa / tiny / tiny_scaled workloads."""
    from paged_kv_cache_251_gb300 import workloads as wl
    if name == "tiny":
        return wl.decode_inputs(wl.SHAPES["tiny"], device=device, num_blocks=64, shuffle=shuffle)
    if name == "gqa":
        return wl.decode_inputs(wl.SHAPES["gqa"], device=device, room_for_append=True, fill=0.95, shuffle=shuffle)
    return wl.decode_inputs(wl.SHAPES[name], device=device, shuffle=shuffle)


class OracleStep:
    """A workload's step as the CPU oracle runs it: the CPU baseline of the
    native arm and the whole of the reference arm.  Its inputs come from the
    seeded generator (workloads.py) and its block tables, slots and
    copy-on-write pairs from the oracle's own models (oracle.locate,
    oracle.RingModel, oracle.CowModel); nothing here loads the CUDA library or
    its host block manager."""

    def __init__(self, name, table="shuffled", kv_format="native", shared=False):
        import oracle
        from paged_kv_cache_251_gb300 import workloads as wl
        self.oracle = oracle
        self.kv_format = None if kv_format == "native" else kv_format
        self.window = 0
        self.pairs = None
        if name in ("opt13b", "gqa", "tiny", "tiny_scaled"):
            inp = _decode_inputs(name, "cpu", table == "shuffled")
            s = self.shape = inp.shape
            self.tables, self.lens = inp.block_tables, inp.context_lens
            slots = []
            for i in range(s.num_seqs):
                phys, off = oracle.locate(self.tables[i].tolist(), s.block_size, int(self.lens[i]))
                slots.append(phys * s.block_size + off)
            self.slots = torch.tensor(slots, dtype=torch.int64)
            self.q, self.k_new, self.v_new = inp.q, inp.k_new, inp.v_new
            if self.kv_format:
                self.k, self.v = wl.quant_pools(inp, self.kv_format)
            else:
                self.k, self.v = inp.k_cache, inp.v_cache
            self.description = describe(name, kv_format=self.kv_format)
        elif self.kv_format:
            raise SystemExit("--kv-format applies to the opt13b, gqa, tiny and tiny_scaled workloads")
        elif name == "window":
            self._window()
        else:
            self._prefix(int(name[len("prefix_bs"):]), shared)
            self.description = describe(name, tokens=self.slots.numel(), pairs=self.pairs.shape[0], shared=shared)

    def _window(self, context=131072, window=None):
        from paged_kv_cache_251_gb300 import workloads as wl
        s = self.shape = wl.SHAPES["window"]
        bs, W = s.block_size, (s.window if window is None else window)
        R = -(-W // bs) + 1
        nb = s.num_seqs * R
        M = -(-context // bs) + 8
        order = wl.permutation(s.seed, 2, nb).tolist()
        self.tables = torch.full((s.num_seqs, M), -1, dtype=torch.int32)
        slots = []
        for i in range(s.num_seqs):
            ring = self.oracle.RingModel(bs, order[i * R:(i + 1) * R], M)
            for t in range(context):
                ring.write(t)
            self.tables[i] = torch.tensor(ring.table, dtype=torch.int32)  # before token L is placed
            slots.append(ring.write(context))
        self.lens = torch.full((s.num_seqs,), context, dtype=torch.int32)
        self.slots = torch.tensor(slots, dtype=torch.int64)
        self.window = W
        kv_shape = (nb, s.num_kv_heads, bs, s.head_dim)
        self.q = wl.normal_tensor(s.seed, 3, (s.num_seqs, s.num_heads, s.head_dim), dtype=s.dtype)
        self.k = wl.normal_tensor(s.seed, 4, kv_shape, dtype=s.dtype)
        self.v = wl.normal_tensor(s.seed, 5, kv_shape, dtype=s.dtype)
        self.k_new = wl.normal_tensor(s.seed, 6, (s.num_seqs, s.num_kv_heads, s.head_dim), dtype=s.dtype)
        self.v_new = wl.normal_tensor(s.seed, 7, (s.num_seqs, s.num_kv_heads, s.head_dim), dtype=s.dtype)
        self.description = describe("window")

    def _prefix(self, bs, shared, prompts=32, samples=8, prompt_len=2000, max_new=256):
        from paged_kv_cache_251_gb300 import workloads as wl
        base = wl.SHAPES["prefix"]
        s = self.shape = wl.Shape(base.name, prompts * samples, base.num_heads, base.num_kv_heads, base.head_dim,
                                  bs, base.dtype, seed=base.seed + bs)
        n_new = wl.prefix_draws(base.seed, prompts * samples, 1, max_new)
        per_prompt = -(-prompt_len // bs)
        M = -(-(prompt_len + max_new) // bs) + 1
        nb = prompts * per_prompt + prompts * samples * (-(-max_new // bs) + 1)
        cow = self.oracle.CowModel(bs, wl.permutation(s.seed, 2, nb).tolist())
        length = [0] * (prompts * samples)
        for p in range(prompts):
            first = p * samples
            cow.add_sequence(first)
            for t in range(prompt_len):
                cow.write(first, t)
            for j in range(samples):
                length[first + j] = prompt_len
                if j:
                    cow.fork(first, first + j)
        slots, pairs = [], []
        for sid in range(prompts * samples):
            for _ in range(int(n_new[sid])):
                slot, copy = cow.write(sid, length[sid])
                length[sid] += 1
                slots.append(slot)
                if copy:
                    pairs.append(copy)
        self.tables = torch.full((prompts * samples, M), -1, dtype=torch.int32)
        for sid, row in cow.tables.items():
            self.tables[sid, :len(row)] = torch.tensor(row, dtype=torch.int32)
        self.lens = torch.tensor(length, dtype=torch.int32)
        self.slots = torch.tensor(slots, dtype=torch.int64)
        self.pairs = torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2)
        T = len(slots)
        kv_shape = (nb, s.num_kv_heads, bs, s.head_dim)
        self.q = wl.normal_tensor(s.seed, 3, (s.num_seqs, s.num_heads, s.head_dim), dtype=s.dtype)
        self.k = wl.normal_tensor(s.seed, 4, kv_shape, dtype=s.dtype)
        self.v = wl.normal_tensor(s.seed, 5, kv_shape, dtype=s.dtype)
        self.k_new = wl.normal_tensor(s.seed, 6, (T, s.num_kv_heads, s.head_dim), dtype=s.dtype)
        self.v_new = wl.normal_tensor(s.seed, 7, (T, s.num_kv_heads, s.head_dim), dtype=s.dtype)

    def run(self, threads, rows=None):
        """One step (copies, append, decode of the first `rows` sequences);
        returns the K/V bytes the decode read."""
        orc, s = self.oracle, self.shape
        n = s.num_seqs if rows is None else rows
        prefix = self.pairs is not None        # prefix sharing writes its tokens before it decodes
        if prefix:
            orc.copy_blocks(self.k, self.v, self.pairs)
            orc.append_kv(self.k, self.v, self.k_new, self.v_new, self.slots)
        orc.paged_attention(self.q[:n], self.k, self.v, self.tables[:n], self.lens[:n], num_kv_heads=s.num_kv_heads,
                            scale=1.0 / math.sqrt(s.head_dim), window=self.window, threads=threads)
        if self.kv_format:
            orc.append_kv_quant(self.k, self.v, self.k_new, self.v_new, self.slots)
        elif not prefix:
            orc.append_kv(self.k, self.v, self.k_new, self.v_new, self.slots)
        toks = self.lens[:n].to(torch.int64)
        if self.window:
            toks = toks.clamp_max(self.window)
        per_tok = 2 * s.num_kv_heads * (s.head_dim + 4 if self.kv_format else s.head_dim * _elt(s.dtype))
        return int(toks.sum()) * per_tok


class DecodeAppendStep(Step):
    """pa_decode over every sequence's L tokens, then pa_append_kv of token L
    (the slot the host block manager assigns); idempotent step."""

    kv_format = None

    def __init__(self, name, device, partition, shuffle=True, kv_format="native", contiguous=False):
        super().__init__(device, partition)
        self.kv_format = None if kv_format == "native" else kv_format
        from paged_kv_cache_251_gb300 import pa
        from paged_kv_cache_251_gb300 import workloads as wl
        from paged_kv_cache_251_gb300.blocks import BlockManager
        self.pa = pa
        self.name = name
        inp = _decode_inputs(name, device, shuffle)
        self.description = describe(name)
        s = self.shape = inp.shape
        # the host block manager replays each sequence's blocks in table order and
        # assigns the slot of the appended token (position L)
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
        self.inp = inp
        self.q, self.k_cache, self.v_cache = inp.q, inp.k_cache, inp.v_cache
        self.k_new, self.v_new = inp.k_new, inp.v_new
        self.bt, self.cl, self.slots = inp.block_tables.to(device), inp.context_lens.to(device), slots.to(device)
        self.host = {"q": inp.q, "k_new": inp.k_new, "v_new": inp.v_new, "slots": slots,
                     "context_lens": inp.context_lens, "block_tables": inp.block_tables}
        self.out = torch.empty(inp.q.shape, dtype=torch.float32, device=device)
        self.window = 0
        self.ws = pa.workspace_for(inp.q, s.block_size, self.bt.shape[1], 0, partition)
        elt = _elt(s.dtype)
        from paged_kv_cache_251_gb300 import accounting as acc
        if self.kv_format:
            # 8-bit pools: random codes and row scales from the seeded generator
            # (the 16-bit pools are dropped); the new tokens are quantised on append
            self.k_cache = self.v_cache = inp.k_cache = inp.v_cache = None
            self.kq, self.vq = wl.quant_pools(inp, self.kv_format, device=device)
            self.description = describe(name, kv_format=self.kv_format)
            self.dec_bytes = acc.decode_bytes(inp.context_lens, s.num_heads, s.num_kv_heads, s.head_dim,
                                              s.block_size, 1, out_elt_bytes=4, q_elt_bytes=elt, row_scale_bytes=4)
        else:
            self.dec_bytes = acc.decode_bytes(inp.context_lens, s.num_heads, s.num_kv_heads, s.head_dim,
                                              s.block_size, elt, out_elt_bytes=4)
        self.kv_bytes = self.dec_bytes["kv"]
        self.roof_bytes = self.dec_bytes["total"]
        self.launches = (2 if self.ws is not None else 1) + 1
        T = inp.k_new.shape[0]
        self.append_bytes = (acc.append_quant_bytes(T, s.num_kv_heads, s.head_dim, elt) if self.kv_format else
                             acc.append_bytes(T, s.num_kv_heads, s.head_dim, elt))
        self.contiguous = contiguous
        if contiguous:
            self._to_contiguous()

    def _to_contiguous(self):
        """The pool's values gathered into contiguous caches [N][H_kv][L][d]
        (L = the table width in tokens): decode reads them with no block
        table; the step has no append (its slots belong to the paged pool)."""
        s = self.shape
        bs = s.block_size
        L = self.bt.shape[1] * bs
        held = self.inp.blocks_held.tolist()
        self.kc = torch.zeros((s.num_seqs, s.num_kv_heads, L, s.head_dim), dtype=s.dtype, device=self.device)
        self.vc = torch.zeros_like(self.kc)
        for i in range(s.num_seqs):
            blocks = self.bt[i, :held[i]].long()
            for src, dst in ((self.k_cache, self.kc), (self.v_cache, self.vc)):
                dst[i, :, :held[i] * bs] = src[blocks].permute(1, 0, 2, 3).reshape(s.num_kv_heads, -1, s.head_dim)
        from paged_kv_cache_251_gb300 import accounting as acc
        n = self.pa.pa_decode_workspace_size(s.num_seqs, s.num_heads, s.head_dim, 16, L // 16, 0, self.partition)
        self.ws_c = None if n == 0 else torch.empty((n + 15) // 16 * 4, dtype=torch.float32, device=self.device)
        self.append_bytes = 0
        self.launches = 2 if self.ws_c is not None else 1
        self.description += ("; contiguous caches [N][H_kv][L][d] holding the same values, decoded by "
                             "pa_decode_contiguous (no block table); no append")

    def decode(self, stream, q=None, bt=None, cl=None):
        s = self.shape
        if getattr(self, "contiguous", False):
            self.pa.pa_decode_contiguous(self.out, self.q if q is None else q, self.kc, self.vc,
                                         self.cl if cl is None else cl, num_kv_heads=s.num_kv_heads,
                                         partition_size=self.partition, workspace=self.ws_c, err_word=self.err,
                                         stream=stream)
            return
        if self.kv_format:
            self.pa.pa_decode_quant(self.out, self.q if q is None else q, self.kq, self.vq,
                                    self.bt if bt is None else bt, self.cl if cl is None else cl,
                                    num_kv_heads=s.num_kv_heads, window=self.window, partition_size=self.partition,
                                    workspace=self.ws, err_word=self.err, stream=stream)
            return
        self.pa.pa_decode(self.out, self.q if q is None else q, self.k_cache, self.v_cache,
                          self.bt if bt is None else bt, self.cl if cl is None else cl, num_kv_heads=s.num_kv_heads,
                          window=self.window, partition_size=self.partition, workspace=self.ws, err_word=self.err,
                          stream=stream)

    def post(self, stream, k_new=None, v_new=None, slots=None):
        if getattr(self, "contiguous", False):
            return
        kn = self.k_new if k_new is None else k_new
        vn = self.v_new if v_new is None else v_new
        sl = self.slots if slots is None else slots
        if self.kv_format:
            self.pa.pa_append_kv_quant(kn, vn, sl, self.kq, self.vq, err_word=self.err, stream=stream)
            return
        self.pa.pa_append_kv(kn, vn, sl, self.k_cache, self.v_cache, err_word=self.err, stream=stream)

    def cache_args(self):
        """(k, v, extra oracle kwargs) of the cache for the oracle."""
        if self.kv_format:
            return self.kq, self.vq, {}
        return self.k_cache, self.v_cache, {}

    def e2e(self, stream, dev):
        """The step through the public API from host buffers (dev: device
        staging tensors filled here).  The decode's inputs go first on the
        step's stream; the append's inputs travel on a side stream while the
        decode runs, and the output comes back on it while the append runs.
        The step ends with the side stream joined, so the next step reuses
        the staging buffers and the output only after both copies are done.
        A step small enough to stay in L2 is launch-bound, and the extra
        cross-stream waits would cost more than they hide: it runs in order."""
        if self.kv_bytes < 2 * L2_BYTES:
            for k in ("q", "k_new", "v_new", "slots", "context_lens", "block_tables"):
                dev[k].copy_(self.host_pinned[k], non_blocking=True)
            self.decode(stream, q=dev["q"], bt=dev["block_tables"], cl=dev["context_lens"])
            self.post(stream, k_new=dev["k_new"], v_new=dev["v_new"], slots=dev["slots"])
            self.out_host.copy_(self.out, non_blocking=True)
            return
        if not hasattr(self, "_side"):
            self._side = torch.cuda.Stream(device=stream.device)
            self._ev_in = torch.cuda.Event()
            self._ev_dec = torch.cuda.Event()
        side = self._side
        side.wait_stream(stream)
        for k in ("q", "context_lens", "block_tables"):
            dev[k].copy_(self.host_pinned[k], non_blocking=True)
        with torch.cuda.stream(side):
            for k in ("k_new", "v_new", "slots"):
                dev[k].copy_(self.host_pinned[k], non_blocking=True)
            self._ev_in.record(side)
        self.decode(stream, q=dev["q"], bt=dev["block_tables"], cl=dev["context_lens"])
        self._ev_dec.record(stream)
        stream.wait_event(self._ev_in)
        self.post(stream, k_new=dev["k_new"], v_new=dev["v_new"], slots=dev["slots"])
        with torch.cuda.stream(side):
            side.wait_event(self._ev_dec)
            self.out_host.copy_(self.out, non_blocking=True)
        stream.wait_stream(side)


class WindowStep(DecodeAppendStep):
    """Sliding window: pa_decode with window 32768 (512-token partitions +
    reduce) over 4 x 131072-token sequences held in rings of 2049 blocks, then
    pa_append_kv of token L (a ring table rewrite on the host)."""

    def __init__(self, device, partition):
        Step.__init__(self, device, partition or 512)
        from paged_kv_cache_251_gb300 import pa, scenarios
        from paged_kv_cache_251_gb300 import accounting as acc
        self.pa = pa
        self.name = "window"
        self.description = describe("window")
        st = scenarios.window_state(device=device)
        s = self.shape = st.shape
        self.window = s.window
        tables0, lens0 = st.block_tables, st.context_lens
        slots, _ = st.manager.append(list(range(s.num_seqs)))   # token L of every sequence
        # decode over L tokens with the tables as they were before token L
        self.inp = type("I", (), {"block_tables": tables0, "context_lens": lens0})
        self.q, self.k_cache, self.v_cache, self.k_new, self.v_new = st.q, st.k_cache, st.v_cache, st.k_new, st.v_new
        self.bt, self.cl, self.slots = tables0.to(device), lens0.to(device), slots.to(device)
        self.host = {"q": st.q, "k_new": st.k_new, "v_new": st.v_new, "slots": slots, "context_lens": lens0,
                     "block_tables": tables0}
        self.out = torch.empty(st.q.shape, dtype=torch.float32, device=device)
        self.ws = pa.workspace_for(st.q, s.block_size, self.bt.shape[1], self.window, self.partition)
        self.dec_bytes = acc.decode_bytes(lens0, s.num_heads, s.num_kv_heads, s.head_dim, s.block_size,
                                          _elt(s.dtype), out_elt_bytes=4, window=self.window)
        self.kv_bytes = self.dec_bytes["kv"]
        self.roof_bytes = self.dec_bytes["total"]
        self.launches = 3
        self.append_bytes = acc.append_bytes(st.k_new.shape[0], s.num_kv_heads, s.head_dim, _elt(s.dtype))


class PrefixStep(DecodeAppendStep):
    """Prefix sharing: pa_copy_blocks (copy-on-write of the partly filled last
    prompt block, block 32 only), pa_append_kv of every sample's 1-256 new
    tokens, pa_decode over all 256 samples; idempotent step."""

    append_first = True

    def __init__(self, device, partition, block_size=16, shared=False):
        Step.__init__(self, device, partition)
        self.shared = shared
        from paged_kv_cache_251_gb300 import pa, scenarios
        from paged_kv_cache_251_gb300 import accounting as acc
        self.pa = pa
        self.name = f"prefix_bs{block_size}"
        st = scenarios.prefix_state(block_size, device=device)
        s = self.shape = st.shape
        self.description = describe(self.name, tokens=st.slots.numel(), pairs=st.pairs.shape[0])
        self.window = 0
        self.inp = type("I", (), {"block_tables": st.block_tables, "context_lens": st.context_lens})
        self.q, self.k_cache, self.v_cache, self.k_new, self.v_new = st.q, st.k_cache, st.v_cache, st.k_new, st.v_new
        self.bt, self.cl, self.slots = st.block_tables.to(device), st.context_lens.to(device), st.slots.to(device)
        self.pairs = st.pairs.to(device)
        self.host = {"q": st.q, "k_new": st.k_new, "v_new": st.v_new, "slots": st.slots,
                     "context_lens": st.context_lens, "block_tables": st.block_tables, "pairs": st.pairs}
        self.out = torch.empty(st.q.shape, dtype=torch.float32, device=device)
        self.ws = pa.workspace_for(st.q, s.block_size, self.bt.shape[1], 0, partition)
        elt = _elt(s.dtype)
        self.dec_bytes = acc.decode_bytes(st.context_lens, s.num_heads, s.num_kv_heads, s.head_dim, s.block_size, elt,
                                          out_elt_bytes=4)
        # logical bytes (every sample reads its own context) and unique bytes
        # (a prompt's shared blocks once): the roofline uses the unique bytes
        shared_blocks = st.prompts * (st.prompt_len // block_size)
        per_tok = 2 * s.num_kv_heads * s.head_dim * elt
        self.kv_bytes = self.dec_bytes["kv"]
        self.unique_kv = self.kv_bytes - (st.samples - 1) * shared_blocks * block_size * per_tok
        self.roof_bytes = self.dec_bytes["total"] - (self.kv_bytes - self.unique_kv)
        self.launches = (1 if st.pairs.shape[0] else 0) + 1 + (2 if self.ws is not None else 1)
        self.T = st.slots.numel()
        self.append_bytes = acc.append_bytes(self.T, s.num_kv_heads, s.head_dim, elt)
        self.copy_bytes = acc.copy_bytes(int(st.pairs.shape[0]), s.num_kv_heads, block_size, s.head_dim, elt)
        if shared:
            self.name += "_shared"
            self.description = describe(self.name, tokens=st.slots.numel(), pairs=st.pairs.shape[0], shared=True)
            self.group = st.samples
            self.shared_lens = torch.full((st.prompts,), st.prompt_len // block_size * block_size,
                                          dtype=torch.int32, device=device)
            n = pa.pa_decode_shared_prefix_workspace_size(s.num_seqs, s.num_heads, s.head_dim, block_size,
                                                          self.bt.shape[1], partition, self.group, s.dtype)
            self.ws_shared = torch.empty(n, dtype=torch.uint8, device=device)
            self.launches = (1 if st.pairs.shape[0] else 0) + 1 + 4

    def decode(self, stream, q=None, bt=None, cl=None):
        if not self.shared:
            return DecodeAppendStep.decode(self, stream, q, bt, cl)
        s = self.shape
        self.pa.pa_decode_shared_prefix(self.out, self.q if q is None else q, self.k_cache, self.v_cache,
                                        self.bt if bt is None else bt, self.cl if cl is None else cl,
                                        self.shared_lens, self.group, num_kv_heads=s.num_kv_heads,
                                        partition_size=self.partition, workspace=self.ws_shared, err_word=self.err,
                                        stream=stream)

    def pre(self, stream, pairs=None):
        self.pa.pa_copy_blocks(self.pairs if pairs is None else pairs, self.k_cache, self.v_cache,
                               err_word=self.err, stream=stream)

    def e2e(self, stream, dev):
        for k in ("q", "k_new", "v_new", "slots", "context_lens", "block_tables", "pairs"):
            dev[k].copy_(self.host_pinned[k], non_blocking=True)
        self.pre(stream, pairs=dev["pairs"])
        self.post(stream, k_new=dev["k_new"], v_new=dev["v_new"], slots=dev["slots"])
        self.decode(stream, q=dev["q"], bt=dev["block_tables"], cl=dev["context_lens"])
        self.out_host.copy_(self.out, non_blocking=True)


WORKLOADS = ["opt13b", "gqa", "window", "prefix_bs8", "prefix_bs16", "prefix_bs32", "tiny", "tiny_scaled"]


def make_step(name, device, partition, table="shuffled", shared=False, kv_format="native"):
    if table == "contiguous" and (name not in ("opt13b", "gqa", "tiny_scaled") or kv_format != "native"):
        raise SystemExit("--table contiguous applies to the 16/32-bit opt13b, gqa and tiny_scaled workloads")
    if name in ("opt13b", "gqa", "tiny", "tiny_scaled"):
        return DecodeAppendStep(name, device, partition, shuffle=(table == "shuffled"), kv_format=kv_format,
                                contiguous=(table == "contiguous"))
    if kv_format != "native":
        raise SystemExit("--kv-format applies to the opt13b, gqa, tiny and tiny_scaled workloads")
    if name == "window":
        return WindowStep(device, partition)
    if name.startswith("prefix_bs"):
        return PrefixStep(device, partition, int(name[len("prefix_bs"):]), shared=shared)
    raise ValueError(name)


def traffic_from_profile(name: str, kernel_hash: str):
    """dram bytes per decode launch from the committed ncu summary of this
    workload, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"pa_decode_{name}.md")
    try:
        text = open(path).read()
    except OSError:
        return None, None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)\s+source_hash:\s*([0-9a-f]+)", text)
    if m and m.group(2) == kernel_hash:
        return int(m.group(1)), os.path.relpath(path, ROOT)
    return None, None


def default_partition(s, kv_format):
    """The partition the library takes for partition_size 0 (include/pa.h):
    1024 tokens where a tensor-core kernel runs, else 512."""
    G = s.num_heads // s.num_kv_heads
    if kv_format == "native":
        tc = G in (2, 4, 8) and s.head_dim == 128 and s.dtype in (torch.float16, torch.bfloat16)
    else:
        tc = (kv_format == "e4m3" and s.head_dim == 128 and G in (2, 4) and s.block_size in (16, 32)
              and s.num_kv_heads % 4 == 0 and s.dtype in (torch.float16, torch.bfloat16))
    return 1024 if tc else 512


def host_call_times(st, stream, calls=100):
    """Host time of one decode call, in microseconds: through the Python
    binding (st.decode) and, for pa_decode, through the C ABI alone (ctypes
    with the arguments marshalled once).  The loops only submit work: they
    do not wait for the GPU, which runs behind them."""
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(calls):
        st.decode(stream)
    t_py = (time.perf_counter() - t0) / calls
    torch.cuda.synchronize()
    out = {"python_binding": round(t_py * 1e6, 2)}
    if type(st) is DecodeAppendStep and not st.kv_format and not getattr(st, "contiguous", False):
        pa, s = st.pa, st.shape
        lib = pa._lib
        args = (pa._ptr(st.out), pa._ptr(st.q), pa._ptr(st.k_cache), pa._ptr(st.v_cache), pa._ptr(st.bt),
                pa._ptr(st.cl), s.num_seqs, s.num_heads, s.num_kv_heads, s.head_dim, s.block_size,
                1.0 / math.sqrt(s.head_dim), st.window, pa.DTYPE_CODE[s.dtype], pa.DTYPE_CODE[st.out.dtype],
                st.bt.shape[1], st.k_cache.shape[0], st.partition, pa._ptr(st.ws),
                0 if st.ws is None else st.ws.numel() * st.ws.element_size(), pa._ptr(st.err), pa._stream(stream))
        f = lib.pa_decode
        t0 = time.perf_counter()
        for _ in range(calls):
            f(*args)
        t_c = (time.perf_counter() - t0) / calls
        torch.cuda.synchronize()
        out["c_abi"] = round(t_c * 1e6, 2)
    return out


def kernel_source_hash(csrc: str | None = None) -> str:
    """A hash of the decode kernels' code (comments and layout dropped), which
    keys the ncu traffic figures in profiles/ to the code they were taken on."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "paged_kv_cache_251_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.startswith("pa_decode") or fn in ("pa_device.cuh", "pa_api.cu", "pa_quant.cuh"):
            with open(os.path.join(csrc, fn), encoding="utf-8") as f:
                text = f.read()
            text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
            text = re.sub(r"//[^\n]*", " ", text)
            h.update(fn.encode() + " ".join(text.split()).encode())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# arms


# The other workloads, timed after the headline one in a default run (one
# GPU), so that one record carries every workload: (label, workload,
# kv_format, shared-prefix decode)
OTHER_WORKLOADS = [
    ("tiny", "tiny", "native", False),
    ("tiny_scaled", "tiny_scaled", "native", False),
    ("gqa", "gqa", "native", False),
    ("window", "window", "native", False),
    ("prefix_bs16_shared", "prefix_bs16", "native", True),
    ("opt13b_int8", "opt13b", "int8", False),
    ("opt13b_e4m3", "opt13b", "e4m3", False),
    ("gqa_int8", "gqa", "int8", False),
    ("gqa_e4m3", "gqa", "e4m3", False),
]


def time_workload(st, dev, steps, warmup, soak_s=0.3):
    """Decode-call and step times of a workload's step (CUDA events on the
    launching stream; L2 flushed before each step when its K/V would fit)."""
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(warmup, 3)):
        st.run(stream)
    torch.cuda.synchronize(dev)
    flush = (torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
             if int(st.kv_bytes) < 2 * L2_BYTES else None)
    ds = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    de = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    es = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(dev.index) as clocks:
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < soak_s:
            for _ in range(20):
                st.run(stream)
            torch.cuda.synchronize(dev)
        for i in range(steps):
            if flush is not None:
                flush.add_(1)
            es[i].record(stream)
            st.run(stream, {"decode": (ds[i], de[i])})
            ee[i].record(stream)
        torch.cuda.synchronize(dev)
    assert st.err.item() == 0, f"device error word {st.err.item()}"
    ms_dec = statistics.mean(ds[i].elapsed_time(de[i]) for i in range(steps))
    ms_step = statistics.mean(es[i].elapsed_time(ee[i]) for i in range(steps))
    return ms_dec, ms_step, clocks.summary(), flush is not None


def measure_others(dev, steps, warmup):
    peak, peak_kind = hbm_peak()
    out = {}
    for label, name, kv_format, shared in OTHER_WORKLOADS:
        st = make_step(name, dev, 0, "shuffled", shared, kv_format)
        ms_dec, ms_step, clk, flushed = time_workload(st, dev, steps, warmup)
        s = st.shape
        achieved = st.roof_bytes / (ms_dec * 1e-3) / 1e9
        out[label] = {
            "workload": st.description,
            "decode_ms": round(ms_dec, 5), "ms_per_step": round(ms_step, 5),
            "kv_gb_s": round(st.kv_bytes / (ms_step * 1e-3) / 1e9, 2),
            "roofline_frac": round(achieved / peak, 4), "algorithmic_bytes_per_decode": int(st.roof_bytes),
            "seq_layer_steps_per_s": round(s.num_seqs / (ms_step * 1e-3), 1),
            "partition_size": default_partition(s, kv_format) if name != "window" else 512,
            "l2_flushed_per_step": flushed, "clocks": clk,
        }
        if hasattr(st, "unique_kv"):
            out[label]["bytes_note"] = "unique K/V bytes (each shared prompt block counted once)"
        del st
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    return out


def run_native(args):
    world, rank, local = dist_env()
    dist_init(world)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the native arm")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    st = make_step(args.workload, dev, args.partition, args.table, args.shared_prefix, args.kv_format)
    s = st.shape
    tag = (args.workload + ("" if args.kv_format == "native" else "_" + args.kv_format) +
           ("_shared" if args.shared_prefix else ""))
    stream = torch.cuda.current_stream(dev)

    for _ in range(max(args.warmup, 0)):
        st.run(stream)
    torch.cuda.synchronize(dev)
    assert st.err.item() == 0, f"device error word {st.err.item()}"

    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ds = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    de = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    parts = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
             for n in ("append", "copy")}

    def part_events(i):
        ev = {"append": parts["append"][i]}
        if st.copy_bytes:
            ev["copy"] = parts["copy"][i]
        return ev

    es = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    flush = (torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
             if int(st.kv_bytes) < 2 * L2_BYTES else None)
    with ClockSampler(local) as clocks:
        # untimed soak of the same step (>= 0.6 s) so the 200 ms clock samples
        # see the GPU under this load; the timed region follows immediately
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 0.6:
            for _ in range(50):
                st.run(stream)
            torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        if flush is None:
            ev0.record(stream)
            for i in range(K):
                st.run(stream, {"decode": (ds[i], de[i])})
            ev1.record(stream)
        else:
            # the step's K/V would stay in L2: overwrite a buffer larger than L2
            # before every step and time each step on its own
            for i in range(K):
                flush.add_(1)
                es[i].record(stream)
                st.run(stream, {"decode": (ds[i], de[i])})
                ee[i].record(stream)
        torch.cuda.synchronize(dev)
        # the cache ops of the same steps, timed one by one in a loop of their
        # own (their events would add latency to a launch-bound timed step)
        for i in range(K):
            if flush is not None:
                flush.add_(1)
            st.run(stream, part_events(i))
        torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.summary()
    if flush is None:
        ms_step = ev0.elapsed_time(ev1) / K
    else:
        ms_step = statistics.mean(es[i].elapsed_time(ee[i]) for i in range(K))
    ms_dec = statistics.mean(ds[i].elapsed_time(de[i]) for i in range(K))
    cache_ops = {}
    for name, nbytes, what in (("append", st.append_bytes, "pa_append_kv"), ("copy_blocks", st.copy_bytes,
                                                                            "pa_copy_blocks")):
        if not nbytes:
            continue
        evs = parts["append" if name == "append" else "copy"]
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        cache_ops[name] = {"call": what + ("_quant" if name == "append" and args.kv_format != "native" else ""),
                           "ms": round(ms, 5), "algorithmic_bytes": int(nbytes),
                           "gb_s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    ms_step_max = max_over_ranks(ms_step, world, dev)
    assert st.err.item() == 0, f"device error word {st.err.item()}"

    # spot parity of the benchmarked output against the oracle
    parity = None
    if rank == 0:
        import oracle
        from paged_kv_cache_251_gb300 import workloads as wl
        idx = wl.permutation(4242, 1, s.num_seqs * s.num_heads)[:16]
        pairs = torch.stack([idx // s.num_heads, idx % s.num_heads], 1).to(torch.int32)
        kc, vc, extra = st.cache_args()
        extra = {k: v.cpu() for k, v in extra.items()}
        ref = oracle.paged_attention(st.q.cpu(), kc.cpu(), vc.cpu(), st.inp.block_tables,
                                     st.inp.context_lens, num_kv_heads=s.num_kv_heads,
                                     scale=1.0 / math.sqrt(s.head_dim), window=st.window, pairs=pairs,
                                     threads=os.cpu_count() or 1, **extra)
        got = st.out.cpu()[pairs[:, 0].long(), pairs[:, 1].long()].double().numpy()
        parity = float(abs(got - ref).max())

    # end to end through the public API with host buffers; its output is
    # compared with the device-resident path's (the decode kernels compute an
    # item in a fixed order whichever CTA claims it, so the two agree bit for
    # bit; the bound below only has to catch a wrong buffer or a race)
    out_device_path = st.out.clone()
    st.host_pinned = {k: v.cpu().pin_memory() for k, v in st.host.items()}
    dev_in = {k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in st.host.items()}
    st.out_host = torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in st.host_pinned.values())
    d2h = st.out_host.numel() * st.out_host.element_size()
    for _ in range(max(args.warmup, 0)):
        st.e2e(stream, dev_in)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        st.e2e(stream, dev_in)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / K, world, dev)
    e2e_diff = float((st.out_host.double() - out_device_path.cpu().double()).abs().max())
    assert e2e_diff <= 1e-4, f"the end-to-end output differs from the device-resident path's by {e2e_diff}"
    host_us = host_call_times(st, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        ost = OracleStep(args.workload, args.table, args.kv_format, args.shared_prefix)
        times, reps, kv_done = [], 0, 0
        t_start = time.perf_counter()
        while True:
            t0 = time.perf_counter()
            kv_done = ost.run(threads)
            times.append(time.perf_counter() - t0)
            if time.perf_counter() - t_start + times[-1] > args.cpu_seconds or len(times) >= 100:
                break
        t_step = statistics.median(times)
        cpu = {"value": kv_done / t_step / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"the full step ({s.num_seqs * s.num_heads} (seq, head) rows of fp64 decode plus the "
                         f"cache ops), median of {len(times)} runs on {threads} host threads",
               "seconds_per_step": t_step}

    others = None
    if (rank == 0 and world == 1 and not args.no_others and args.workload == "opt13b" and args.table == "shuffled"
            and args.kv_format == "native" and args.partition == 0):
        others = measure_others(dev, K, args.warmup)

    peak, peak_kind = hbm_peak()
    achieved = st.roof_bytes / (ms_dec * 1e-3) / 1e9
    khash = kernel_source_hash()
    traffic, traffic_src = traffic_from_profile(tag, khash)
    value = world * st.kv_bytes / (ms_step_max * 1e-3) / 1e9
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
        "dtype": ({"int8": "i8", "e4m3": "e4m3"}[args.kv_format] if args.kv_format != "native" else
                  {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}[s.dtype]),
        "data": "synthetic (seeded SplitMix64 / Box-Muller N(0,1) q, K, V; seeded shuffle of the block pool)",
        "config": {
            "workload": st.description,
            "num_seqs": s.num_seqs, "num_heads": s.num_heads, "num_kv_heads": s.num_kv_heads,
            "head_dim": s.head_dim, "block_size": s.block_size, "window": st.window,
            "context_tokens": st.dec_bytes["attended_tokens"],
            "partition_size": st.partition or default_partition(s, args.kv_format), "accumulate": "f32",
            "out_dtype": "f32",
            "block_order": args.table, "kv_format": args.kv_format,
            "l2": (f"no flush: the K/V read per step ({st.kv_bytes / 1e9:.2f} GB) is larger than L2 (129 MB)"
                   if flush is None else
                   f"L2 flushed before every timed step (a 256 MB buffer is overwritten); the K/V read per step "
                   f"({st.kv_bytes / 1e6:.2f} MB) would otherwise stay in L2; steps timed one by one"),
            "parallelism": f"replicas x{world} (each rank its own batch)",
        },
        "seq_layer_steps_per_s": round(world * s.num_seqs / (ms_step_max * 1e-3), 1),
        "hbm_frac_of_step": round(value / peak, 4),
        "decode_ms": round(ms_dec, 5),
        "cache_ops": cache_ops,
        "roofline": {"bound": "hbm", "kernel": "pa_decode (decode + partition reduce)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} (hbm_gbs, STREAM-style copy)",
                     "algorithmic_bytes_per_launch": st.roof_bytes, "traffic": traffic,
                     "traffic_source": traffic_src, "source_hash": khash},
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * st.kv_bytes / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 5),
                "api": "paged_kv_cache_251_gb300.pa (ctypes binding of libpa)",
                "max_abs_diff_vs_device_path": e2e_diff},
        "host_us_per_decode_call": host_us,
        "gpu_launches": K * st.launches,
        "clocks": clk,
        "parity_sampled_max_abs": parity,
        "impl": "native",
    }
    if others is not None:
        line["other_workloads"] = others
    if hasattr(st, "unique_kv"):
        line["config"]["unique_kv_bytes"] = st.unique_kv
        line["roofline"]["bytes_note"] = "unique K/V bytes (each shared prompt block counted once)"
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_swap(args):
    """Block swap between HBM and pinned host memory (the OPT-13B pool's
    blocks, 2048 of them = 655 MB of K+V, out to host and back in)."""
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from paged_kv_cache_251_gb300 import pa
    from paged_kv_cache_251_gb300 import workloads as wl
    inp = wl.decode_inputs(wl.SHAPES["opt13b"], device=dev)
    nblk = 2048
    hk = torch.empty((nblk,) + tuple(inp.k_cache.shape[1:]), dtype=inp.k_cache.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    src = wl.permutation(77, 1, inp.num_blocks)[:nblk]
    out_pairs = torch.stack([src, torch.arange(nblk)], 1).contiguous().to(dev)
    in_pairs = torch.stack([torch.arange(nblk), src], 1).contiguous().to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    bytes_dir = 2 * nblk * hk[0].numel() * hk.element_size()
    for _ in range(max(args.warmup, 3)):
        pa.pa_swap_blocks(out_pairs, inp.k_cache, inp.v_cache, hk, hv, err_word=err)
        pa.pa_swap_blocks(in_pairs, hk, hv, inp.k_cache, inp.v_cache, err_word=err)
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * K)]
    for i in range(K):
        ev[3 * i].record(stream)
        pa.pa_swap_blocks(out_pairs, inp.k_cache, inp.v_cache, hk, hv, err_word=err)
        ev[3 * i + 1].record(stream)
        pa.pa_swap_blocks(in_pairs, hk, hv, inp.k_cache, inp.v_cache, err_word=err)
        ev[3 * i + 2].record(stream)
    torch.cuda.synchronize(dev)
    assert err.item() == 0
    t_out = statistics.mean(ev[3 * i].elapsed_time(ev[3 * i + 1]) for i in range(K))
    t_in = statistics.mean(ev[3 * i + 1].elapsed_time(ev[3 * i + 2]) for i in range(K))

    # the copy engines instead of the kernel: one cudaMemcpyAsync (a torch
    # copy) per contiguous run of blocks, K and V; the bench's pairs are a
    # random permutation (runs of one block), and the same block count as one
    # run of consecutive blocks
    def ce_copy(src_k, src_v, dst_k, dst_v, runs):
        for a, b, n in runs:
            dst_k[b:b + n].copy_(src_k[a:a + n], non_blocking=True)
            dst_v[b:b + n].copy_(src_v[a:a + n], non_blocking=True)

    def as_runs(pairs):
        runs, p = [], pairs.cpu().tolist()
        for a, b in p:
            if runs and runs[-1][0] + runs[-1][2] == a and runs[-1][1] + runs[-1][2] == b:
                runs[-1][2] += 1
            else:
                runs.append([a, b, 1])
        return runs

    ce = {}
    first = 0
    for label, pairs_out in (("permuted", out_pairs), ("one_run", torch.stack([torch.arange(first, first + nblk),
                                                                                torch.arange(nblk)], 1))):
        r_out = as_runs(pairs_out)
        r_in = [[b, a, n] for a, b, n in r_out]
        for _ in range(2):
            ce_copy(inp.k_cache, inp.v_cache, hk, hv, r_out)
            ce_copy(hk, hv, inp.k_cache, inp.v_cache, r_in)
        torch.cuda.synchronize(dev)
        cev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * K)]
        t_host = time.perf_counter()
        for i in range(K):
            cev[3 * i].record(stream)
            ce_copy(inp.k_cache, inp.v_cache, hk, hv, r_out)
            cev[3 * i + 1].record(stream)
            ce_copy(hk, hv, inp.k_cache, inp.v_cache, r_in)
            cev[3 * i + 2].record(stream)
        t_host = (time.perf_counter() - t_host) / (2 * K)
        torch.cuda.synchronize(dev)
        co = statistics.mean(cev[3 * i].elapsed_time(cev[3 * i + 1]) for i in range(K))
        ci = statistics.mean(cev[3 * i + 1].elapsed_time(cev[3 * i + 2]) for i in range(K))
        ce[label] = {"copies_per_direction": 2 * len(r_out), "out_gbs": round(bytes_dir / (co * 1e-3) / 1e9, 2),
                     "in_gbs": round(bytes_dir / (ci * 1e-3) / 1e9, 2), "ms_out": round(co, 4), "ms_in": round(ci, 4),
                     "host_ms_per_direction": round(t_host * 1e3, 3)}
    # the kernel on one run of consecutive blocks, for the same comparison
    kp_out = torch.stack([torch.arange(first, first + nblk), torch.arange(nblk)], 1).contiguous().to(dev)
    kp_in = kp_out.flip(1).contiguous()
    for _ in range(2):
        pa.pa_swap_blocks(kp_out, inp.k_cache, inp.v_cache, hk, hv, err_word=err)
        pa.pa_swap_blocks(kp_in, hk, hv, inp.k_cache, inp.v_cache, err_word=err)
    kev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * K)]
    for i in range(K):
        kev[3 * i].record(stream)
        pa.pa_swap_blocks(kp_out, inp.k_cache, inp.v_cache, hk, hv, err_word=err)
        kev[3 * i + 1].record(stream)
        pa.pa_swap_blocks(kp_in, hk, hv, inp.k_cache, inp.v_cache, err_word=err)
        kev[3 * i + 2].record(stream)
    torch.cuda.synchronize(dev)
    assert err.item() == 0
    ko = statistics.mean(kev[3 * i].elapsed_time(kev[3 * i + 1]) for i in range(K))
    ki = statistics.mean(kev[3 * i + 1].elapsed_time(kev[3 * i + 2]) for i in range(K))
    line = {"metric": "KV block swap GB/s (HBM <-> pinned host memory)", "value": round(
        2 * bytes_dir / ((t_out + t_in) * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": 1, "steps": K,
        "warmup": max(args.warmup, 3), "higher_is_better": True, "dtype": "f16", "data": "synthetic",
        "config": {"workload": f"swap: {nblk} OPT-13B-shaped blocks (K+V {bytes_dir / 1e6:.0f} MB) out to pinned "
                               "host memory and back, pa_swap_blocks", "blocks": nblk},
        "swap_out_gbs": round(bytes_dir / (t_out * 1e-3) / 1e9, 2),
        "swap_in_gbs": round(bytes_dir / (t_in * 1e-3) / 1e9, 2),
        "ms_out": round(t_out, 4), "ms_in": round(t_in, 4),
        "kernel_one_run": {"out_gbs": round(bytes_dir / (ko * 1e-3) / 1e9, 2),
                           "in_gbs": round(bytes_dir / (ki * 1e-3) / 1e9, 2)},
        "copy_engine": ce, "gpu_launches": 2 * K, "impl": "native"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return  # the reference arm runs on rank 0 only
    st = OracleStep(args.workload, args.table, args.kv_format, args.shared_prefix)
    s = st.shape
    threads = os.cpu_count() or 1
    # size the per-step sample so the whole run stays within a few minutes
    total_steps = max(1, args.steps + args.warmup)
    probe = min(2, s.num_seqs)
    t0 = time.perf_counter()
    st.run(threads, rows=probe)
    per_seq = (time.perf_counter() - t0) / probe
    budget = 150.0 / total_steps
    n = max(1, min(s.num_seqs, int(budget / max(per_seq, 1e-9))))
    for _ in range(args.warmup):
        st.run(threads, rows=n)
    times, kv = [], 0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        kv = st.run(threads, rows=n)
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times) if times else float("nan")
    value = kv / dt / 1e9
    sample = (f"{n} of {s.num_seqs} sequences ({n * s.num_heads} (seq, head) rows) of fp64 decode plus the step's "
              f"cache ops per step, on {threads} host threads")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded workload as the native arm)",
        "config": {"workload": st.description, "num_seqs": s.num_seqs, "num_heads": s.num_heads,
                   "num_kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "block_size": s.block_size,
                   "window": st.window, "block_order": args.table, "kv_format": args.kv_format},
        "sequences_sampled_per_step": n,
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
    elif args.workload == "swap":
        run_swap(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
