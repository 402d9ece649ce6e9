"""Benchmark: microseconds per MLA decode call on the synthetic workloads.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one mla_decode_fwd call (query preparation, split kernel and
log-sum-exp combine) over one batch, inputs resident in HBM, with the L2
flushed before every timed call (a 256 MiB device write); each call is
bracketed by CUDA events on its stream.  The headline workload is the
largest one, bs=64, kv_len=8192, e4m3 KV (302 MB of cache per call).  Under
torchrun (N > 1) every rank decodes its own batch of the same shape
(independent sequences, no collective on the data path: weak scaling); the
timed loop is bracketed by a barrier and synchronize, the per-call time is the
max over ranks.  Rank 0 prints one JSON line.

Extra keys:
  roofline     the split stage alone (query preparation + split kernel, timed
               in a second pass through the split/combine entry points, events
               on the launch stream) against the measured HBM copy bandwidth;
               algorithmic bytes = KV bytes.
  per_config   (one GPU) every one of the five workloads timed the same way in
               the same run: us per call, split stage, combine, roofline
               fraction, and the oracle's CPU time on a bounded sample.
  cpu_baseline the fp64 C oracle on the host cores (a bounded sample of
               sequences, scaled by KV rows to the full call).
  e2e          the same metric through the public call with the step's inputs
               (q and the index arrays) copied in from pinned host memory and
               out/lse copied back inside the timed region.
  clocks       nvidia-smi samples taken during the timed region.

--impl reference times the oracle (the pages' definition evaluated in fp64 on the
CPU) on the same workload and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mla_attention_decode_gb300 import synth  # noqa: E402

DEFAULT_WORKLOAD = "bs64_kv8192_fp8"
L2_FLUSH_BYTES = 256 << 20
L2_TEXT = "flushed before every timed call (256 MiB write)"
CODES = {"bf16": 0, "fp8": 1, "mxfp4": 2}
DTYPE_LABEL = {"bf16": "bf16 x bf16 -> f32", "fp8": "e4m3 x e4m3 -> f32", "mxfp4": "e4m3 x e4m3 -> f32 (e2m1 KV)"}
_CSRC = "mla_attention_decode_gb300/csrc/"
# sources of the split kernel timed for each KV format (the profiled traffic is
# only reported while these are unchanged since the capture)
KERNEL_SOURCES = {
    "bf16": [_CSRC + f for f in ("mla_stage1.cuh", "mla_common.cuh", "mla_ptx.cuh", "mla_internal.h")],
    "fp8": [_CSRC + f for f in ("mla_tc.cuh", "mla_common.cuh", "mla_ptx.cuh", "mla_internal.h")],
    "mxfp4": [_CSRC + f for f in ("mla_tc.cuh", "mla_common.cuh", "mla_ptx.cuh", "mla_internal.h",
                                  "mla_split_mxfp4.cu")],
    "mxfp4_bs": [_CSRC + f for f in ("mla_tc.cuh", "mla_common.cuh", "mla_ptx.cuh", "mla_internal.h",
                                     "mla_split_mxfp4_bs.cu")],
}
KERNEL_NAMES = {"bf16": "mla_split_kernel (mma.sync, bf16)",
                "fp8": "mla_prep_q_kernel + mla_split_tc_kernel (tcgen05, e4m3), launches overlapped",
                "mxfp4": "mla_prep_q_kernel + mla_split_tc_kernel (tcgen05, e2m1 dequantised to e4m3), "
                         "launches overlapped",
                "mxfp4_bs": "mla_prep_q_kernel + mla_split_tc_kernel (tcgen05 block-scaled e2m1 x e4m3 scores, "
                            "V dequantised to e4m3), launches overlapped"}
# the block-scaled form of the MXFP4 workload, timed beside the five in per_config
MX_BS_SUFFIX = "_block_scaled"
CLOCK_SOAK_S = 1.0
CPU_BUDGET_HEADLINE_S = 15.0
CPU_BUDGET_PER_CONFIG_S = 4.0


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=synth.WORKLOAD_ORDER)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline workload (per_config is otherwise added on one GPU)")
    ap.add_argument("--q-len", type=int, default=1,
                    help="query tokens per sequence (mla_decode_plan_multi; each token attends to the rows up "
                         "to its own entry)")
    ap.add_argument("--mx-block-scaled", action="store_true",
                    help="MXFP4 workload: scores by block-scaled MMAs on the e2m1 tile (plan.mx_scores = 1)")
    ap.add_argument("--page-size", type=int, default=0,
                    help="decode the workload's rows from a paged cache with pages of this many rows "
                         "(pages scattered at random; mla_decode_fwd_paged); 0 = contiguous cache")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(values, pg, device):
    """Element-wise maximum of per-rank values over the process group (the job
    takes as long as its slowest rank); the values themselves without one."""
    if pg is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_sha(kv_dtype: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kv_dtype]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kv_dtype: str):
    """dram bytes per split-kernel launch from the committed ncu summary of this
    workload key (e.g. "bs64_kv8192_fp8_q2"), if it was taken on the current
    kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_sha") != kernel_source_sha(kv_dtype):
        return None
    return e.get("dram_bytes_per_launch")


def workload_key(name: str, args) -> str:
    return (name + (MX_BS_SUFFIX if getattr(args, "mx_block_scaled", False) else "") +
            (f"_paged{args.page_size}" if args.page_size else "") + (f"_q{args.q_len}" if args.q_len > 1 else ""))


def workload_kv_bytes(name: str) -> int:
    """KV bytes (with scales) one call reads: the algorithmic bytes of the workload."""
    b, L, dt = synth.WORKLOADS[name]
    rows = b * L
    return {"bf16": rows * 1152, "fp8": rows * 576 + 4, "mxfp4": rows * (288 + 18)}[dt]


def workload_config(name: str, args, world: int) -> dict:
    """The `config` object of the JSON line; both arms print the same one."""
    b, L, dt = synth.WORKLOADS[name]
    return {"workload": workload_key(name, args), "batch": b, "kv_len": L, "kv_dtype": dt,
            "page_size": args.page_size or 1, "q_len": args.q_len, "kv_bytes_per_call": workload_kv_bytes(name),
            "l2": L2_TEXT, "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if not self.out:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


class L2Flush:
    """Evicts the L2 between timed calls: a write of 256 MiB, twice the L2."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def __call__(self, i: int):
        self.w.fill_(i & 0xFF)


def to_device(inp: synth.MLAInputs, dev):
    scale = inp.kv_scale if inp.kv_dtype == "fp8" else inp.block_scales
    return dict(q=inp.q.to(dev), kv=inp.kv.to(dev), kv_scale=None if scale is None else scale.to(dev),
                kv_indptr=inp.kv_indptr.to(dev), qo_indptr=inp.qo_indptr.to(dev))


def time_calls(fn, steps, flush, stream):
    """Per-call device times (us) of `steps` calls, L2 flushed before each."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush(i)
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e3 for a, b in ev]


def oracle_decoder(inp: synth.MLAInputs, q_len: int = 1, paged=None):
    """The fp64 C oracle as it stands, on the host cores: returns (decode(n), cores),
    decode(n) evaluating the first n sequences of the workload in its form
    (q_len tokens per sequence, or read through the page table)."""
    import oracle
    orc = oracle.load()
    cores = os.cpu_count() or 1
    code = CODES[inp.kv_dtype]
    kvs = None if inp.kv_scale is None else inp.kv_scale.numpy()
    bs = None if inp.block_scales is None else inp.block_scales.numpy()

    def decode(n):
        qo = inp.qo_indptr[:n + 1].numpy()
        if paged is not None:
            pbs = None if paged.block_scales is None else paged.block_scales.numpy()
            return orc.decode_paged(code, inp.q, paged.kv, paged.page_indptr[:n + 1].numpy(),
                                    paged.kv_indices.numpy(), paged.last_page_len[:n].numpy(), paged.page_size,
                                    qo, kvs, pbs, num_threads=cores)
        if q_len > 1:
            return orc.decode_multi(code, inp.q, inp.kv, inp.kv_indptr[:n + 1].numpy(), q_len, qo, kvs, bs,
                                    num_threads=cores)
        return orc.decode(code, inp.q, inp.kv, inp.kv_indptr[:n + 1].numpy(), qo, kvs, bs, num_threads=cores)

    return decode, cores


def cpu_baseline(inp: synth.MLAInputs, q_len: int = 1, paged=None, budget_s: float = CPU_BUDGET_HEADLINE_S):
    """Times the oracle as it stands on the host cores; returns (us per full call, cores, sample text)."""
    decode, cores = oracle_decoder(inp, q_len, paged)
    lens = (inp.kv_indptr[1:] - inp.kv_indptr[:-1]).tolist()
    # probe one sequence to size the sample
    t0 = time.perf_counter()
    decode(1)
    per_seq = max(time.perf_counter() - t0, 1e-4)
    nseq = max(1, min(inp.batch, int(budget_s / per_seq)))
    t0 = time.perf_counter()
    decode(nseq)
    dt = time.perf_counter() - t0
    us_call = dt * 1e6 * (sum(lens) / max(1, sum(lens[:nseq])))
    form = (f", {q_len} tokens each" if q_len > 1 else "") + (", through the page table" if paged is not None else "")
    sample = (f"{nseq} of {inp.batch} sequences (all 16 heads{form}), fp64 C oracle with OpenMP, "
              f"scaled by KV rows to the full call")
    return us_call, cores, sample


def make_workload_inputs(name, args, rank):
    """The seeded inputs of a workload in the form the run decodes it."""
    b, L, dt = synth.WORKLOADS[name]
    inp = synth.make_inputs([L] * b, dt, seed=rank)
    if args.q_len > 1:
        # q_len tokens per sequence: query rows b * q_len + i
        g = torch.Generator("cpu").manual_seed(1000 + rank)
        inp.q = torch.randn(b * args.q_len, 16, 576, generator=g).to(torch.bfloat16)
        inp.qo_indptr = torch.arange(b + 1, dtype=torch.int32) * args.q_len
    # the same rows in a paged cache: pages at random positions (no spare pages)
    paged = synth.make_paged(inp, args.page_size, seed=rank, spare_pages=0) if args.page_size else None
    return inp, paged


def run_reference(args, inp, name, paged=None):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return
    decode, cores = oracle_decoder(inp, args.q_len, paged)
    lens = (inp.kv_indptr[1:] - inp.kv_indptr[:-1]).tolist()

    # bound the whole run to about 100 s of CPU work: a sample of sequences per
    # step, scaled by rows
    t0 = time.perf_counter()
    decode(1)
    per_seq = max(time.perf_counter() - t0, 1e-4)
    budget = max(0.05, 100.0 / max(1, args.steps + args.warmup))
    nseq = max(1, min(inp.batch, int(budget / per_seq)))
    scale = sum(lens) / max(1, sum(lens[:nseq]))
    for _ in range(args.warmup):
        decode(nseq)
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        decode(nseq)
        ts.append((time.perf_counter() - t0) * 1e6 * scale)
    us = statistics.mean(ts)
    line = {
        "impl": "reference", "metric": "us_per_mla_decode_call", "value": round(us, 2), "unit": "us/call",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(name, args, world),
        "cpu_baseline": {"value": round(us, 2), "unit": "us/call", "cores": cores, "kind": "oracle",
                         "sample": f"{nseq} of {inp.batch} sequences per step, scaled by KV rows"},
        "e2e": {"value": round(us, 2), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def check_device(w, where: str):
    """The workload's device error word is clear; otherwise fail with the
    detail words the kernels leave (CTA, thread, tag, detail; mla_decode.h)."""
    err = w.dec.poll_error()
    if err:
        detail = w.dec.workspace[8:24].view(torch.int32).tolist()
        raise RuntimeError(f"{w.name} ({where}): device error {err}, detail {detail}")


class Workload:
    """One workload resident on the device, with its plan, workspace and the
    calls the bench times."""

    def __init__(self, name, args, rank, dev, mx_bs=False):
        from mla_attention_decode_gb300 import binding
        self.binding = binding
        self.name = name + (MX_BS_SUFFIX if mx_bs else "")
        b, L, self.dt = synth.WORKLOADS[name]
        assert not mx_bs or self.dt == "mxfp4"
        self.kind = "mxfp4_bs" if mx_bs else self.dt  # which kernel sources and name the roofline cites
        self.inp, self.paged = make_workload_inputs(name, args, rank)
        dt = self.dt
        d = to_device(self.inp, dev)
        if self.paged is not None:
            pg_ = self.paged
            d["kv"] = pg_.kv.to(dev)
            if dt == "mxfp4":
                d["kv_scale"] = pg_.block_scales.to(dev)
            d["page_indptr"] = pg_.page_indptr.to(dev)
            d["kv_indices"] = pg_.kv_indices.to(dev)
            d["last_page_len"] = pg_.last_page_len.to(dev)
            self.dec = binding.PagedMLADecoder(pg_.page_indptr, pg_.last_page_len, pg_.page_size, pg_.num_pages, dt,
                                               device=dev, mx_block_scaled=mx_bs)
        else:
            self.dec = binding.MLADecoder(self.inp.kv_indptr, dt, device=dev, q_len=args.q_len,
                                          mx_block_scaled=mx_bs)
        self.d = d
        self.plan = self.dec.plan
        self.out = torch.empty(self.plan.batch, 16, 512, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(self.plan.batch, 16, dtype=torch.float32, device=dev)
        self.scale_stride = int(d["kv_scale"].stride(0)) if dt == "mxfp4" else 0
        # query preparation (e4m3 and MXFP4 KV), split kernel, combine when split
        self.launches_per_call = (1 if dt == "bf16" else 2) + (1 if self.plan.splits_max > 1 else 0)

    def call(self, stream, src=None, out=None, lse=None):
        """One mla_decode_fwd (or _paged) call; src/out/lse override the inputs
        and results (host buffers for the end-to-end forms)."""
        b, d = self.binding, self.d
        s = d if src is None else src
        o = self.out if out is None else out
        l_ = self.lse if lse is None else lse
        if self.paged is not None:
            b.mla_decode_fwd_paged(s["q"], d["kv"], d["kv_scale"], s["page_indptr"], s["kv_indices"],
                                   s["last_page_len"], s["qo_indptr"], o, l_, self.plan, self.dec.workspace,
                                   scale_stride=self.scale_stride, stream=stream)
        else:
            b.mla_decode_fwd(s["q"], d["kv"], d["kv_scale"], s["kv_indptr"], s["qo_indptr"], o, l_, self.plan,
                             self.dec.workspace, scale_stride=self.scale_stride, stream=stream)

    def time_stages(self, steps, flush, stream, us_call):
        """(split stage us, combine us): the two entry points timed separately,
        L2 flushed before each call (the paged entry point has no separate
        stages: the whole call stands in)."""
        if self.paged is not None:
            return us_call, 0.0
        b, d = self.binding, self.d
        ev_split, ev_comb = [], []
        for i in range(steps):
            flush(i)
            e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e0.record(stream)
            b.mla_decode_split(d["q"], d["kv"], d["kv_scale"], d["kv_indptr"], d["qo_indptr"], self.out, self.lse,
                               self.plan, self.dec.workspace, scale_stride=self.scale_stride, stream=stream)
            e1.record(stream)
            b.mla_decode_combine(self.out, self.lse, self.plan, self.dec.workspace, stream=stream)
            e2.record(stream)
            ev_split.append((e0, e1))
            ev_comb.append((e1, e2))
        torch.cuda.synchronize()
        return (statistics.mean(a.elapsed_time(c) * 1e3 for a, c in ev_split),
                statistics.mean(a.elapsed_time(c) * 1e3 for a, c in ev_comb))


def roofline_entry(w: Workload, args, t_split: float, t_comb: float, peak: float, peak_kind: str) -> dict:
    kv_bytes = w.inp.kv_bytes()
    achieved = kv_bytes / (t_split * 1e-6) / 1e9
    key = w.name + (f"_q{args.q_len}" if args.q_len > 1 else "")
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": profiled_traffic(key, w.kind) if w.paged is None else None,
            "kernel": KERNEL_NAMES[w.kind] if w.paged is None else "whole paged call",
            "kernel_us": round(t_split, 3), "combine_us": round(t_comb, 3),
            "peak_kind": f"{peak_kind} (HBM copy)"}


def measure_per_config(args, rank, dev, stream, flush, peak, peak_kind, headline: dict) -> dict:
    """Every workload timed as the headline is (same flush, same events), one
    after another; the headline's own entry is the headline's numbers."""
    res = {}
    mx_name = next(n for n in synth.WORKLOAD_ORDER if synth.WORKLOADS[n][2] == "mxfp4")
    for name, mx_bs in [(n, False) for n in synth.WORKLOAD_ORDER] + [(mx_name, True)]:
        if name == args.workload and mx_bs == args.mx_block_scaled:
            res[name + (MX_BS_SUFFIX if mx_bs else "")] = headline
            continue
        w = Workload(name, args, rank, dev, mx_bs=mx_bs)
        for _ in range(max(3, args.warmup)):
            w.call(stream)
        check_device(w, "warm-up")
        # a device error in the timed calls voids them: they are taken once more
        # and the error is reported in the entry (a second one fails the bench)
        retried = None
        for attempt in range(2):
            us = statistics.mean(time_calls(lambda: w.call(stream), args.steps, flush, stream))
            t_split, t_comb = w.time_stages(args.steps, flush, stream, us)
            try:
                check_device(w, "timed calls")
                break
            except RuntimeError as e:
                if attempt == 1:
                    raise
                retried = str(e)
        entry = {"value": round(us, 3), "unit": "us/call", "kv_bytes_per_call": w.inp.kv_bytes(),
                 "kv_gbs": round(w.inp.kv_bytes() / (us * 1e-6) / 1e9, 1),
                 "roofline": roofline_entry(w, args, t_split, t_comb, peak, peak_kind),
                 "gpu_launches": args.steps * w.launches_per_call,
                 "plan": {k: w.plan.as_dict()[k] for k in ("num_work", "grid", "chunk_tokens", "splits_max",
                                                          "schedule")}}
        if retried:
            entry["device_error_then_retimed"] = retried
        if mx_bs:
            entry["form"] = "MXFP4 scores by block-scaled MMAs on the e2m1 tile (plan.mx_scores = 1)"
        if not args.no_cpu_baseline and not mx_bs:
            us_cpu, cores, sample = cpu_baseline(w.inp, args.q_len, w.paged, budget_s=CPU_BUDGET_PER_CONFIG_S)
            entry["cpu_baseline"] = {"value": round(us_cpu, 1), "unit": "us/call", "cores": cores, "kind": "oracle",
                                     "sample": sample}
        res[w.name] = entry
        del w
        torch.cuda.empty_cache()
    return res


def main(argv=None):
    args = parse(argv)
    rank, world, local = dist_env()
    name = args.workload
    assert args.page_size == 0 or args.q_len == 1, "--page-size and --q-len are not combined"
    if args.impl == "reference":
        inp, paged = make_workload_inputs(name, args, rank)
        run_reference(args, inp, name, paged)
        return

    from mla_attention_decode_gb300 import binding, build
    build.build()
    assert torch.cuda.is_available(), "bench.py needs a CUDA GPU"
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    w = Workload(name, args, rank, dev, mx_bs=args.mx_block_scaled)
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)
    for _ in range(max(3, args.warmup)):
        w.call(stream)
    check_device(w, "warm-up")

    # ---- headline: whole call, device time, L2 flushed before each call.  The
    # clock samples cover the timed steps and a soak of the same flushed calls
    # around them (the timed region alone is shorter than the sampling period).
    def soak(seconds):
        t_end = time.perf_counter() + seconds
        while time.perf_counter() < t_end:
            for i in range(20):
                flush(i)
                w.call(stream)
            torch.cuda.synchronize()

    barrier()
    with ClockSampler(local) as clk:
        soak(CLOCK_SOAK_S / 2)
        barrier()
        t_wall = time.perf_counter()
        per_call = time_calls(lambda: w.call(stream), args.steps, flush, stream)
        barrier()
        t_wall = time.perf_counter() - t_wall
        soak(CLOCK_SOAK_S / 2)
    us = max_over_ranks([statistics.mean(per_call)], pg, dev)[0]

    # ---- the split stage alone (roofline) and the combine, events on the launch stream
    t_split, t_comb = w.time_stages(args.steps, flush, stream, us)
    peak, peak_kind = measured_peaks()

    # ---- end to end through the public call, with the step's inputs (q and the
    # index arrays) in pinned host memory and out/lse read back to it.  Two
    # forms, both timed; the headline e2e value is always the "staged" form:
    # one host-to-device copy of the inputs, the call, one device-to-host copy
    # of out/lse.  "host_buffers" passes the pinned host buffers to the call
    # itself, so the kernels read the inputs and write the results over the
    # host link (NVLink-C2C on Grace) -- except q of bf16 KV, which that kernel
    # fetches with bulk copies and is therefore copied in first.
    inp, paged = w.inp, w.paged
    host_src = {"q": inp.q, "qo_indptr": inp.qo_indptr}
    if paged is None:
        host_src["kv_indptr"] = inp.kv_indptr
    else:
        host_src.update(page_indptr=paged.page_indptr, kv_indices=paged.kv_indices,
                        last_page_len=paged.last_page_len)
    ins = binding.PackedBuffers([(k, tuple(v.shape), v.dtype) for k, v in host_src.items()], dev)
    for k, v in host_src.items():
        ins.host[k].copy_(v)
    outs = binding.PackedBuffers([("out", tuple(w.out.shape), w.out.dtype), ("lse", tuple(w.lse.shape),
                                                                             w.lse.dtype)], dev)

    def staged_call():
        ins.to_device(stream)
        w.call(stream, ins.dev, outs.dev["out"], outs.dev["lse"])
        outs.to_host(stream)

    host_in = dict(ins.host)
    q_dev = ins.dev["q"]

    def host_call():
        src = host_in
        if w.dt == "bf16":
            q_dev.copy_(ins.host["q"], non_blocking=True)
            src = dict(host_in, q=q_dev)
        w.call(stream, src, outs.host["out"], outs.host["lse"])

    e2e_forms = {}
    for form, fn in (("staged", staged_call), ("host", host_call)):
        for _ in range(3):
            fn()
        barrier()
        times = time_calls(fn, args.steps, flush, stream)
        torch.cuda.synchronize()
        assert torch.equal(outs.host["out"], w.out.cpu()), f"end-to-end ({form}) output differs from the device call"
        e2e_forms[form] = statistics.mean(times)
    h2d, d2h = ins.nbytes, outs.nbytes
    check_device(w, "timed calls and end-to-end forms")
    e2e_staged, e2e_host, t_split, t_comb = max_over_ranks(
        [e2e_forms["staged"], e2e_forms["host"], t_split, t_comb], pg, dev)
    roof = roofline_entry(w, args, t_split, t_comb, peak, peak_kind)
    headline = {"value": round(us, 3), "unit": "us/call", "kv_bytes_per_call": inp.kv_bytes(),
                "kv_gbs": round(inp.kv_bytes() / (us * 1e-6) / 1e9, 1), "roofline": roof,
                "gpu_launches": args.steps * w.launches_per_call,
                "plan": {k: w.plan.as_dict()[k] for k in ("num_work", "grid", "chunk_tokens", "splits_max",
                                                         "schedule")}}
    plan_dict = {k: w.plan.as_dict()[k] for k in ("num_work", "grid", "chunk_tokens", "splits_max", "schedule",
                                                  "tokens_fused")}
    del w
    torch.cuda.empty_cache()

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            us_cpu, cores, sample = cpu_baseline(inp, args.q_len, paged)
            cpu = {"value": round(us_cpu, 1), "unit": "us/call", "cores": cores, "kind": "oracle", "sample": sample}
            headline["cpu_baseline"] = cpu
        per_config = None
        if world == 1 and not args.no_per_config and args.q_len == 1 and args.page_size == 0:
            per_config = measure_per_config(args, rank, dev, stream, flush, peak, peak_kind, headline)
        line = {
            "metric": "us_per_mla_decode_call", "value": round(us, 3), "unit": "us/call", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 6),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE_LABEL[synth.WORKLOADS[name][2]],
            "data": "synthetic (seeded N(0,1) q and KV, quantised as stated)",
            "config": workload_config(name, args, world),
            "plan": plan_dict,
            "kv_gbs": headline["kv_gbs"],
            "roofline": roof,
            "e2e": {"value": round(e2e_staged, 3), "unit": "us/call", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "form": "staged",
                    "staged_us": round(e2e_staged, 3), "host_buffers_us": round(e2e_host, 3),
                    "forms": "staged (the value): one pinned-host-to-device copy of q and the index arrays and "
                             "one copy of out/lse back, around the call; host_buffers: the call gets the pinned "
                             "host buffers and its kernels read and write them over the host link (q of bf16 KV "
                             "copied in first)"},
            "gpu_launches": headline["gpu_launches"],
            "clocks": dict(clk.summary(), window="timed steps plus a 1 s soak of the same calls"),
            "wall_s_timed_loop": round(t_wall, 4),
            "cpu_baseline": cpu,
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
