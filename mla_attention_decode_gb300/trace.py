"""Per-CTA timeline of the split kernels (bf16, e4m3 and MXFP4 KV).

    python -m mla_attention_decode_gb300.trace [--workload bs64_kv8192_fp8] [--runs 5] [--json PATH]
    python -m mla_attention_decode_gb300.trace --shape 64 8192 bf16    (any uniform batch)

Builds and loads the trace library (libmla_decode_trace.so: the same kernels
with global-timer stamps compiled in, see mla_decode_set_trace), decodes one
of the benchmark workloads with the L2 flushed before each call (as the
benchmark does), and prints where each CTA's time goes: kernel entry, set-up,
first KV copy, query preparation complete, each tile's scores, each unit's
epilogue, and exit, in microseconds from the first CTA's entry (the median
over the runs of each quantity).  Needs a GPU; times are global-timer times.
"""
from __future__ import annotations

import argparse
import json
import statistics
import sys

import numpy as np
import torch

from . import binding, build, synth

SLOTS = 128
ENTRY, SETUP, FIRST_LOAD, QUERY_READY, UNITS, TILES, EXIT, SCAN_DONE = 0, 1, 2, 3, 4, 5, 6, 7
UNIT_DONE, TILE_S, TILE_DATA, UNIT_LAST_PV = 8, 16, 80, 112
PREP_ENTRY, PREP_WAITED, PREP_DONE = 120, 121, 122  # rows < batch: the query-preparation CTAs
N_TILE_S, N_TILE_DATA = 64, 32


def run(workload: str, runs: int, flush_bytes: int = 256 << 20, lib: str | None = None, shape=None):
    """shape: (batch, kv_len, kv_dtype) in place of a named workload."""
    binding.load_library(lib or build.build(trace=True))
    dev = torch.device("cuda:0")
    b, L, dt = shape if shape is not None else synth.WORKLOADS[workload]
    inp = synth.make_inputs([L] * b, dt, seed=0)
    dec = binding.MLADecoder(inp.kv_indptr, dt, device=dev)
    scale = {"bf16": None, "fp8": inp.kv_scale, "mxfp4": inp.block_scales}[dt]
    q, kv, ind, qo = inp.q.to(dev), inp.kv.to(dev), inp.kv_indptr.to(dev), inp.qo_indptr.to(dev)
    sc = None if scale is None else scale.to(dev)
    grid = dec.plan.grid
    buf = torch.zeros(grid * SLOTS, dtype=torch.int64, device=dev)
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device=dev)
    lib_ = binding.load_library()
    import ctypes
    fn = lib_.mla_decode_set_trace
    fn.argtypes = [ctypes.c_void_p]
    fn.restype = ctypes.c_int
    for _ in range(3):
        dec(q, kv, ind, qo, kv_scale=sc)
    stream = torch.cuda.current_stream()
    out = []
    for r in range(runs):
        buf.zero_()
        rc = fn(ctypes.c_void_p(buf.data_ptr()))
        assert rc == 0, f"mla_decode_set_trace: {rc}"
        flush.fill_(r & 0xFF)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        _split(dec, q, kv, sc, ind, qo, dt, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        fn(ctypes.c_void_p(0))
        out.append((buf.view(grid, SLOTS).cpu().numpy().astype(np.int64), e0.elapsed_time(e1) * 1e3))
    assert dec.poll_error() == 0
    return dec.plan, out


_bufs = {}


def _split(dec, q, kv, sc, ind, qo, dt, stream):
    key = id(dec)
    if key not in _bufs:
        n = dec.plan.batch
        _bufs[key] = (torch.empty(n, 16, 512, dtype=torch.bfloat16, device=q.device),
                      torch.empty(n, 16, dtype=torch.float32, device=q.device))
    o, l_ = _bufs[key]
    binding.mla_decode_split(q, kv, sc, ind, qo, o, l_, dec.plan, dec.workspace,
                             scale_stride=int(sc.stride(0)) if dt == "mxfp4" else 0, stream=stream)


def analyse(stamps: np.ndarray, event_us: float) -> dict:
    """One run's stamps [grid, SLOTS] (ns) -> a summary in us from the first entry."""
    t0 = stamps[:, ENTRY].min()
    us = lambda v: (v - t0) / 1e3  # noqa: E731
    n_tiles = stamps[:, TILES]
    n_units = stamps[:, UNITS]
    periods, first_s, last_s, hold = [], [], [], []
    boundary_gaps, epilogue = [], []
    for c in range(stamps.shape[0]):
        nt = int(min(n_tiles[c], 64))
        s = stamps[c, TILE_S:TILE_S + nt]
        if nt >= 1:
            first_s.append(us(s[0]))
            last_s.append(us(s[-1]))
        if nt >= 4:
            periods.append(float(np.median(np.diff(s[1:]))) / 1e3)
        nd = int(min(nt, N_TILE_DATA))
        dsta = stamps[c, TILE_DATA:TILE_DATA + nd]
        if nd >= 2:
            hold.append(float(np.median(s[:nd] - dsta)) / 1e3)
        # a unit boundary: the gap between the unit's epilogue and the next tile's scores
        nu = int(min(n_units[c], 8))
        for k in range(nu):
            # a unit written after the next unit's last P.V (the e4m3 epilogue defers the
            # first of two) is left out: its span is the wait, not the write
            deferred = k + 1 < nu and stamps[c, UNIT_DONE + k] > stamps[c, UNIT_LAST_PV + k + 1] > 0
            if stamps[c, UNIT_DONE + k] > 0 and stamps[c, UNIT_LAST_PV + k] > 0 and not deferred:
                epilogue.append(float(stamps[c, UNIT_DONE + k] - stamps[c, UNIT_LAST_PV + k]) / 1e3)
        for k in range(nu - 1):
            done = stamps[c, UNIT_DONE + k]
            later = s[s > done]
            if done > 0 and later.size:
                boundary_gaps.append(float(later.min() - done) / 1e3)

    def stats(v):
        v = np.asarray(v, dtype=np.float64)
        if v.size == 0:
            return None
        return {"min": round(float(v.min()), 2), "median": round(float(np.median(v)), 2),
                "max": round(float(v.max()), 2)}

    def prep(slot):
        # the query-preparation grid (rows < batch; none for bf16 caches), relative to the
        # first split CTA's entry: negative before it
        v = stamps[:, slot]
        return stats(us(v[v > 0]))

    exit_ = us(stamps[:, EXIT])
    slowest = int(np.argmax(exit_))
    sc = stamps[slowest]
    nt = int(min(sc[TILES], 64))
    return {
        "event_us_split_stage": round(event_us, 2),
        "prep_entry_us": prep(PREP_ENTRY),
        "prep_waited_us": prep(PREP_WAITED),
        "prep_done_us": prep(PREP_DONE),
        "entry_us": stats(us(stamps[:, ENTRY])),
        "scan_done_us": stats(us(stamps[:, SCAN_DONE])),
        "setup_done_us": stats(us(stamps[:, SETUP])),
        "first_load_issued_us": stats(us(stamps[:, FIRST_LOAD])),
        "query_ready_us": stats(us(stamps[:, QUERY_READY])),
        "first_scores_us": stats(first_s),
        "last_scores_us": stats(last_s),
        "exit_us": stats(exit_),
        "tile_period_us": stats(periods),
        "data_to_scores_us": stats(hold),
        "unit_boundary_gap_us": stats(boundary_gaps),
        "epilogue_us": stats(epilogue),
        "tiles_per_cta": stats(n_tiles),
        "units_per_cta": stats(n_units),
        "slowest_cta": {"cta": slowest, "tiles": int(sc[TILES]), "units": int(sc[UNITS]),
                        "entry": round(us(sc[ENTRY]), 2), "first_scores": round(us(sc[TILE_S]), 2) if nt else None,
                        "last_scores": round(us(sc[TILE_S + nt - 1]), 2) if nt else None,
                        "unit_done": [round(us(sc[UNIT_DONE + k]), 2) for k in range(int(min(sc[UNITS], 8)))],
                        "exit": round(us(sc[EXIT]), 2)},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="bs64_kv8192_fp8", choices=synth.WORKLOAD_ORDER)
    ap.add_argument("--runs", type=int, default=5)
    ap.add_argument("--json", default=None, help="write the per-run summaries here")
    ap.add_argument("--lib", default=None, help="a prebuilt trace library (default: build libmla_decode_trace.so)")
    ap.add_argument("--shape", nargs=3, default=None, metavar=("BATCH", "KV_LEN", "DTYPE"),
                    help="a uniform batch in place of --workload (DTYPE: bf16, fp8 or mxfp4)")
    args = ap.parse_args(argv)
    shape = None
    if args.shape is not None:
        shape = (int(args.shape[0]), int(args.shape[1]), args.shape[2])
        assert shape[2] in ("bf16", "fp8", "mxfp4"), "DTYPE: bf16, fp8 or mxfp4"
        args.workload = f"bs{shape[0]}_kv{shape[1]}_{shape[2]}"
    plan, runs = run(args.workload, args.runs, lib=args.lib, shape=shape)
    summaries = [analyse(s, ev) for s, ev in runs]
    # the median run by split-stage event time
    order = sorted(range(len(summaries)), key=lambda i: summaries[i]["event_us_split_stage"])
    med = summaries[order[len(order) // 2]]
    print(f"workload {args.workload}: grid {plan.grid}, units {plan.num_work}, schedule {plan.schedule}")
    print(f"split-stage event times (us): {[s['event_us_split_stage'] for s in summaries]}")
    print(json.dumps(med, indent=1))
    if args.json:
        with open(args.json, "w") as f:
            raw = runs[order[len(order) // 2]][0]
            t0 = int(raw[:, ENTRY].min())
            rel = np.where(raw > 10**12, raw - t0, raw)  # times relative to the first entry; counts kept
            json.dump({"workload": args.workload, "plan": plan.as_dict(), "runs": summaries,
                       "median_run": med, "median_run_stamps_ns": rel.tolist()}, f)
    return 0


if __name__ == "__main__":
    sys.exit(main())
