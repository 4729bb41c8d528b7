"""GPU parity at the numerical edges of softmax(q K^T / sqrt(d)) V, the
definition in "PagedAttention: From Operating System Virtual Memory to Large
Language Model Memory Systems", section 2 (Background), for every decode kernel
family, against the fp64 oracle and, where the mathematics fixes the answer,
against that answer directly.

The seeded N(0, 1) inputs of the other parity tests keep every score within a
few units, so the online rescale, the partition merge and the reduced-precision
weight paths never meet a large jump.  The inputs here do:

  same_keys      every cached key of a kv head identical: the output is the mean
                 of the attended V rows (weights exactly uniform);
  zero_q         q = 0 for a whole sequence and for one head of another: again
                 the mean of V;
  dominant       one key planted per sequence with a score about 80 above the
                 rest: at the first attended token (first tile of the first
                 partition), at the last token (last tile of the last
                 partition) and at the last token of a middle partition; the
                 output of the aligned head is that token's V row;
  peaked_x8/x16  q scaled by 8 or 16: scores spread over tens of units;
  ramp_up        scores rising by 60 across the context, so the running maximum
                 jumps in every tile and every partition;
  ramp_down      the mirror image: later tiles' weights underflow;
  wide_q         query rows with one element at 1000 and the rest log-uniform
                 in [1e-3, 1] (a range above 2^19, well beyond the 2^14 that
                 the three-term E4M3 query encoding keeps exactly);
  wide_q_masked  the same rows with the keys' entry under the large element set
                 to zero, so the scores come from the small elements alone;
  bad_partition  every block of one partition an invalid table entry next to
                 valid partitions, and a sequence whose blocks are all invalid
                 (skipped and flagged; the all-invalid sequence gives zeros).

Families (which kernel each reaches is set by the library's dispatch on dtype,
group size, head_dim, block size and kv-head count): the MHA kernel, the
tensor-core grouped-head kernel at G = 2, 4, 8, the general CUDA-core kernel
(fp32 with grouped heads, head_dim 64 with grouped heads), the 8-bit
TMA-fed kernel (INT8 and E4M3), the tensor-core E4M3 kernel and the general
8-bit kernel, plus the shared-prefix decode.  Each runs with short partitions
(many partitions, the log-sum-exp reduce) and with one long partition.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_251_gb300 import workloads as wl
from paritylib import compare, make_groups, shape

pytestmark = pytest.mark.gpu

F16, BF16, F32 = torch.float16, torch.bfloat16, torch.float32

# name, N, H, H_kv, d, bs, query/cache dtype, 8-bit format (None = 16/32-bit cache), short partition, window
FAMILIES = [
    ("mha_f16", 3, 4, 4, 128, 16, F16, None, 64, 0),
    ("mha_bf16_d64_bs8", 3, 4, 4, 64, 8, BF16, None, 32, 0),
    ("mha_f32_d64", 3, 4, 4, 64, 16, F32, None, 64, 0),
    ("tc_g2_bs32", 3, 4, 2, 128, 32, BF16, None, 128, 0),
    ("tc_g4", 3, 8, 2, 128, 16, F16, None, 64, 0),
    ("tc_g8_bs8", 3, 16, 2, 128, 8, BF16, None, 64, 0),
    ("tc_g4_window", 3, 8, 2, 128, 16, BF16, None, 64, 700),
    ("gen_f32_g4", 3, 8, 2, 128, 16, F32, None, 64, 0),
    ("gen_d64_g4", 3, 8, 2, 64, 16, BF16, None, 64, 0),
    ("q8f_i8_g1", 3, 4, 4, 128, 16, F16, "int8", 64, 0),
    ("q8f_i8_g4", 3, 8, 2, 128, 16, BF16, "int8", 64, 0),
    ("q8f_e4m3_g1", 3, 4, 4, 128, 16, F16, "e4m3", 64, 0),
    ("q8f_e4m3_g4", 3, 8, 2, 128, 16, BF16, "e4m3", 64, 0),
    ("q8t_g2_bs32", 3, 8, 4, 128, 32, F16, "e4m3", 128, 0),
    ("q8t_g4", 3, 16, 4, 128, 16, BF16, "e4m3", 64, 0),
    ("q8t_g4_window", 3, 16, 4, 128, 16, F16, "e4m3", 64, 700),
    ("q8_gen_d64_i8", 3, 8, 2, 64, 16, F16, "int8", 64, 0),
    ("q8_gen_f32q_e4m3", 3, 8, 2, 128, 16, F32, "e4m3", 64, 0),
]
LENS = [1000, 77, 2049]
TRANSFORMS = ["same_keys", "zero_q", "dominant", "peaked_x8", "peaked_x16", "ramp_up", "ramp_down", "wide_q",
              "wide_q_masked", "bad_partition"]
BIG_SCORE = 80.0      # planted score above the rest, natural-log units
RAMP = 60.0


def _span(L, window):
    return (max(0, L - window) if window > 0 else 0), L


def _rows_of(table_row, bs, toks):
    """(physical block, offset) of logical tokens through one block table row."""
    toks = torch.as_tensor(toks, dtype=torch.int64)
    return table_row.to(torch.int64)[toks // bs], toks % bs


def _quantize(x, fmt):
    """Row-wise symmetric codes of x (float32 [..., d]) for building 8-bit test
    inputs: (codes int8 / float8_e4m3fn, scales float32 [...])."""
    q_max = 127.0 if fmt == "int8" else 448.0
    amax = x.abs().amax(-1, keepdim=True)
    s = amax / q_max
    y = x / torch.where(s > 0, s, torch.ones_like(s))
    if fmt == "int8":
        codes = torch.round(y).clamp(-127, 127).to(torch.int8)
    else:
        codes = y.clamp(-448, 448).to(torch.float8_e4m3fn)
    return codes, s.squeeze(-1).to(torch.float32)


def _dequantize(codes, scales):
    return codes.to(torch.float32) * scales[..., None]


class Case:
    """Inputs of one family in fp32 working form (q, K, V, tables, lengths)."""

    def __init__(self, fam, seed):
        name, n, h, hkv, d, bs, dt, fmt, part, window = fam
        self.name, self.n, self.h, self.hkv, self.d, self.bs = name, n, h, hkv, d, bs
        self.dt, self.fmt, self.part, self.window = dt, fmt, part, window
        self.G = h // hkv
        self.scale = 1.0 / math.sqrt(d)
        sh = shape(name, n, h, hkv, d, bs, dt, window=window, seed=seed)
        inp = wl.decode_inputs(sh, lens=torch.as_tensor(LENS[:n], dtype=torch.int32), room_for_append=False,
                               with_append=False)
        self.tables, self.lens, self.num_blocks = inp.block_tables.clone(), inp.context_lens.clone(), inp.num_blocks
        self.q = inp.q.to(F32)
        if fmt is None:
            self.k, self.v = inp.k_cache.to(F32), inp.v_cache.to(F32)
        else:
            kp, vp = wl.quant_pools(inp, fmt)
            self.k = _dequantize(*oracle.unpack_pages(kp))
            self.v = _dequantize(*oracle.unpack_pages(vp))

    # --- the tensors both sides read ------------------------------------------
    def materialise(self):
        """q in its dtype and the caches (16/32-bit pools or 8-bit pages)."""
        q = self.q.to(self.dt)
        if self.fmt is None:
            return q, self.k.to(self.dt), self.v.to(self.dt)
        return q, wl.page_pool(*_quantize(self.k, self.fmt)), wl.page_pool(*_quantize(self.v, self.fmt))

    def attended(self, s):
        return _span(int(self.lens[s]), self.window)

    def kv_rows(self, cache, s, kvh):
        """The attended rows of cache for (sequence s, kv head kvh), in token order."""
        a, b = self.attended(s)
        blk, off = _rows_of(self.tables[s], self.bs, range(a, b))
        return cache[blk, kvh, off]

    def set_rows(self, cache, s, kvh, toks, rows):
        blk, off = _rows_of(self.tables[s], self.bs, toks)
        cache[blk, kvh, off] = rows

    def n_parts(self, s, part):
        a, b = self.attended(s)
        first_blk = a // self.bs
        last_blk = (b - 1) // self.bs
        return (last_blk - first_blk) // (part // self.bs) + 1


def _direction(case, s, h):
    """A key row whose score with head h of sequence s is exactly 1 (pre-rounding)."""
    qv = case.q[s, h].to(torch.float64)
    return (qv / (float(qv @ qv) * case.scale)).to(F32)


def _wide_col(case, s, h, per_group):
    """Where the large element of a wide query row sits: one column per kv
    head (shared by its query heads) when the keys are masked there, else one
    per query head."""
    key = h // case.G if per_group else h
    return (7 * key + 3 * s) % case.d


def apply(case, transform, part):
    """Modify case's fp32 inputs in place; return the (s, h, expected row)
    closed-form checks the transform gives (expected rows are read back from the
    materialised caches, so they are the stored values)."""
    checks = []
    G, hkv = case.G, case.hkv
    if transform == "same_keys":
        for kvh in range(hkv):
            case.k[:, kvh] = case.k[0, kvh, 0]
        checks = [("mean", s, h) for s in range(case.n) for h in range(case.h)]
    elif transform == "zero_q":
        case.q[0] = 0.0
        case.q[1, 0] = 0.0
        checks = [("mean", 0, h) for h in range(case.h)] + [("mean", 1, 0)]
    elif transform == "dominant":
        for s in range(case.n):
            a, b = case.attended(s)
            P = part
            if s == 0:
                t = a                                   # first tile of the first partition
            elif s == 1:
                t = b - 1                               # last tile of the last partition
            else:                                       # last token of a middle partition
                first = a // case.bs * case.bs
                mid = case.n_parts(s, P) // 2
                t = min(b - 1, first + (mid + 1) * P - 1)
            for kvh in range(hkv):
                h = kvh * G + (s % G)
                row = BIG_SCORE * _direction(case, s, h)
                case.set_rows(case.k, s, kvh, [t], row[None])
                checks.append(("token", s, h, t))
    elif transform in ("peaked_x8", "peaked_x16"):
        case.q *= 8.0 if transform == "peaked_x8" else 16.0
    elif transform in ("ramp_up", "ramp_down"):
        for s in range(case.n):
            a, b = case.attended(s)
            n = b - a
            if n < 2:
                continue
            ramp = torch.linspace(0.0, RAMP, n) if transform == "ramp_up" else torch.linspace(RAMP, 0.0, n)
            for kvh in range(hkv):
                h = kvh * G + (s % G)
                rows = case.kv_rows(case.k, s, kvh) + ramp[:, None] * _direction(case, s, h)[None]
                case.set_rows(case.k, s, kvh, range(a, b), rows)
    elif transform in ("wide_q", "wide_q_masked"):
        d = case.d
        masked = transform == "wide_q_masked"
        for s in range(case.n):
            for h in range(case.h):
                u = wl.uniform01(500 + s, h, 2 * d)
                mag = torch.exp(math.log(1e-3) * (1.0 - u[:d]))            # log-uniform in [1e-3, 1]
                sign = torch.where(u[d:] < 0.5, -1.0, 1.0).to(torch.float64)
                row = (mag * sign).to(F32)
                row[_wide_col(case, s, h, masked)] = 1000.0
                case.q[s, h] = row
        if masked:
            # the large element meets zeros: its kv head's keys have that entry cleared
            for s in range(case.n):
                for kvh in range(hkv):
                    a, b = case.attended(s)
                    rows = case.kv_rows(case.k, s, kvh)
                    rows[:, _wide_col(case, s, kvh * G, True)] = 0.0
                    case.set_rows(case.k, s, kvh, range(a, b), rows)
    elif transform == "bad_partition":
        P_blk = part // case.bs
        t0 = case.tables
        # sequence 0: every block of its second partition invalid, both kinds of bad id
        a, _ = case.attended(0)
        first = a // case.bs
        lo = first + P_blk
        hi = min(lo + P_blk, int((case.lens[0] + case.bs - 1) // case.bs))
        for j, lb in enumerate(range(lo, hi)):
            t0[0, lb] = -3 if j % 2 else case.num_blocks + 11
        # the last sequence: every block invalid
        last = case.n - 1
        nb_last = int((case.lens[last] + case.bs - 1) // case.bs)
        t0[last, :nb_last] = -1 - torch.arange(nb_last, dtype=torch.int32)
    else:
        raise ValueError(transform)
    return checks


def _run_gpu(case, q, kc, vc, part):
    from paged_kv_cache_251_gb300 import pa
    out = torch.full(q.shape, float("nan"), dtype=F32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (out, q.cuda(), kc.cuda(), vc.cuda(), case.tables.cuda(), case.lens.cuda())
    kw = dict(num_kv_heads=case.hkv, scale=case.scale, window=case.window, partition_size=part, err_word=err)
    if case.fmt is None:
        pa.pa_decode(*args, **kw)
    else:
        pa.pa_decode_quant(*args, **kw)
    torch.cuda.synchronize()
    return out.cpu(), int(err.item())


def _closed_form_rows(case, checks, kc, vc):
    """Expected rows of the closed-form checks, from the stored cache values."""
    vals = vc.to(F32) if case.fmt is None else _dequantize(*oracle.unpack_pages(vc))
    rows = []
    for c in checks:
        s, h = c[1], c[2]
        kvh = h // case.G
        if c[0] == "mean":
            vr = case.kv_rows(vals, s, kvh).to(torch.float64)
            rows.append(vr.mean(0) if vr.shape[0] else torch.zeros(case.d, dtype=torch.float64))
        else:
            blk, off = _rows_of(case.tables[s], case.bs, [c[3]])
            rows.append(vals[blk[0], kvh, off[0]].to(torch.float64))
    return torch.stack(rows).numpy() if rows else None


@pytest.mark.parametrize("long_part", [False, True], ids=["short_parts", "one_part"])
@pytest.mark.parametrize("transform", TRANSFORMS)
@pytest.mark.parametrize("fam", FAMILIES, ids=[f[0] for f in FAMILIES])
def test_softmax_edges(fam, transform, long_part):
    case = Case(fam, seed=4000 + FAMILIES.index(fam))
    part = 256 * case.bs if long_part else case.part
    checks = apply(case, transform, part)
    q, kc, vc = case.materialise()
    got, err = _run_gpu(case, q, kc, vc, part)
    bad = transform == "bad_partition"
    assert (err & 1) if bad else err == 0
    ref = oracle.paged_attention(q, kc, vc, case.tables, case.lens, num_kv_heads=case.hkv, scale=case.scale,
                                 window=case.window, invalid_policy=1 if bad else 0, threads=8)
    kv_dt = F32 if (case.dt == F32 and case.fmt is None) else F16
    compare(got, ref, kv_dt)
    if bad:
        assert torch.equal(got[case.n - 1], torch.zeros_like(got[case.n - 1]))
    if checks:
        want = _closed_form_rows(case, checks, kc, vc)
        sel = torch.stack([got[c[1], c[2]] for c in checks])
        compare(sel, want, kv_dt)


# --- shared-prefix decode -----------------------------------------------------

SP_TRANSFORMS = ["dominant_prefix", "dominant_suffix", "peaked_x16", "ramp_up", "ramp_down"]


@pytest.mark.parametrize("transform", SP_TRANSFORMS)
@pytest.mark.parametrize("dtype", [F16, BF16])
def test_shared_prefix_softmax_edges(transform, dtype):
    """pa_decode_shared_prefix merges a prefix pass and a suffix pass; a
    dominant key in either part, peaked scores and ramps that put the maximum
    at either end must merge to the oracle's result."""
    from paged_kv_cache_251_gb300 import pa
    prompts, samples, H, hkv, bs = 2, 4, 8, 4, 16
    plens = [1300, 700]
    N = prompts * samples
    extra = wl.randint(7, 1, N, 1, 300).tolist()
    tables, lens, k, v = make_groups(prompts, samples, plens, extra, bs, hkv, 128, dtype, seed=61)
    q = wl.normal_tensor(9, 3, (N, H, 128), dtype=dtype).to(F32)
    kf = k.to(F32)
    scale = 1.0 / math.sqrt(128)
    G = H // hkv
    shared = [pl // bs * bs for pl in plens]

    def direction(s, h):
        qv = q[s, h].to(torch.float64)
        return (qv / (float(qv @ qv) * scale)).to(F32)

    checks = []
    if transform == "peaked_x16":
        q *= 16.0
    elif transform.startswith("dominant"):
        # a prompt key can only dominate one sample's head per group: plant it
        # for the first sample's head 0; suffix keys are private to each sample
        for s in range(N):
            g = s // samples
            L = int(lens[s])
            if transform == "dominant_prefix":
                if s % samples:
                    continue
                t = shared[g] // 2
            else:
                t = L - 1
            for kvh in range(hkv):
                h = kvh * G
                blk, off = _rows_of(tables[s], bs, [t])
                kf[blk[0], kvh, off[0]] = BIG_SCORE * direction(s, h)
                checks.append((s, h, t))
    else:
        # ramps over each sample's whole context (the prompt rows follow the
        # group's first sample, whose head 0 they are aimed at)
        for s in range(N):
            g = s // samples
            L = int(lens[s])
            first_member = s % samples == 0
            toks = torch.arange(0 if first_member else shared[g], L)
            if toks.numel() < 2:
                continue
            ramp = torch.linspace(0.0, RAMP, L)[toks] if transform == "ramp_up" else \
                torch.linspace(RAMP, 0.0, L)[toks]
            for kvh in range(hkv):
                blk, off = _rows_of(tables[s], bs, toks)
                kf[blk, kvh, off] = kf[blk, kvh, off] + ramp[:, None] * direction(s, kvh * G)[None]
    qd, kd = q.to(dtype), kf.to(dtype)
    out = torch.full((N, H, 128), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode_shared_prefix(out, qd.cuda(), kd.cuda(), v.cuda(), tables.cuda(), lens.cuda(),
                               torch.tensor(shared, dtype=torch.int32).cuda(), samples, num_kv_heads=hkv,
                               partition_size=64, err_word=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle.paged_attention(qd, kd, v, tables, lens, num_kv_heads=hkv, scale=scale, threads=8)
    got = out.cpu()
    compare(got, ref, dtype)
    if checks:
        want = []
        for s, h, t in checks:
            blk, off = _rows_of(tables[s], bs, [t])
            want.append(v[blk[0], h // G, off[0]].to(torch.float64))
        compare(torch.stack([got[s, h] for s, h, _ in checks]), torch.stack(want).numpy(), dtype)
