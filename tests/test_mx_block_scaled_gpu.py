"""MXFP4 scores from block-scaled tensor-core MMAs (plan.mx_scores = 1): the
e2m1 tile is read as the A operand of tcgen05 kind::mxf8f6f4 with the cache's
e8m0 block scales as its scale factors, the query as two e4m3 terms with unit
scale factors (kernelindex "amd-mixed-mla" submission 754939, "Stage 1: Split-K
partial attention with native MXFP4 dot_scaled for scores").  Compared with
the fp64 oracle under the bounds of test_parity_gpu.py: the query's two-term
rounding and the e4m3 weights are the same as on the copy path, and the
scores carry no e4m3 rounding of K at all.
"""
import numpy as np
import pytest
import torch

from mla_attention_decode_gb300 import binding, synth
from test_paged_gpu import paged_gpu, paged_oracle
from test_parity_gpu import (assert_parity, gate_terms, gpu_decode, oracle_decode, orc, built,  # noqa: F401
                             v_absmax)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.mark.parametrize("num_splits", [0, 1, 3, 7])
def test_ragged_small(orc, num_splits):
    inp = synth.make_inputs([1, 33, 70, 0, 129, 200, 64, 2], "mxfp4", seed=31)
    got, lse, dec = gpu_decode(inp, num_splits=num_splits, mx_block_scaled=True)
    ref, ref_lse = oracle_decode(orc, inp)
    assert_parity(got, ref, lse, ref_lse, f"block-scaled ragged splits={num_splits}", gate_terms(inp, ref, ref_lse))
    assert got[3].max() == 0 and got[3].min() == 0, "empty sequence output must be exactly 0"
    assert dec.poll_error() == 0


@pytest.mark.parametrize("lens,num_sms,num_splits", [
    ([256] * 6, 1, 0),
    ([384, 512, 640], 1, 0),
    ([1024, 0, 0, 0, 1024, 1024], 1, 1),
    ([8192, 8192], 3, 0),
    ([3000, 1, 2047, 0, 700, 129], 5, 0),
])
def test_many_units_per_cta(orc, lens, num_sms, num_splits):
    """Grids planned for a few SMs: many tiles and unit boundaries per CTA
    (the ring, the scale chunks and the rope slots wrap many times)."""
    inp = synth.make_inputs(lens, "mxfp4", seed=len(lens) + num_sms)
    got, lse, dec = gpu_decode(inp, num_splits=num_splits, num_sms=num_sms, mx_block_scaled=True)
    ref, ref_lse = oracle_decode(orc, inp)
    assert_parity(got, ref, lse, ref_lse, f"block-scaled {lens} on {num_sms} SMs", gate_terms(inp, ref, ref_lse))
    assert dec.poll_error() == 0


def test_benchmark_workload_full(orc):
    """bs32 / kv8192 MXFP4 at full size, every sequence, head and feature."""
    inp = synth.make_workload("bs32_kv8192_mxfp4")
    got, lse, dec = gpu_decode(inp, mx_block_scaled=True)
    ref, ref_lse = oracle_decode(orc, inp)
    assert_parity(got, ref, lse, ref_lse, "block-scaled bs32_kv8192_mxfp4", gate_terms(inp, ref, ref_lse))
    assert dec.poll_error() == 0


def test_repeated_calls_are_identical():
    inp = synth.make_workload("bs32_kv8192_mxfp4")
    dec = binding.MLADecoder(inp.kv_indptr, "mxfp4", device=DEV, mx_block_scaled=True)
    args = (inp.q.to(DEV), inp.kv.to(DEV), inp.kv_indptr.to(DEV), inp.qo_indptr.to(DEV))
    sc = inp.block_scales.to(DEV)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=DEV)
    first = None
    for i in range(10):
        flush.fill_(i & 0xFF)
        out, lse = dec(*args, kv_scale=sc)
        torch.cuda.synchronize()
        assert dec.poll_error() == 0, f"call {i}: device error"
        if first is None:
            first = (out.clone(), lse.clone())
        else:
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1]), f"call {i} differs"


@pytest.mark.parametrize("spread", [6, 12])
def test_wide_block_exponents(orc, spread):
    """Block scales up to 2 x spread below the row's largest: the scores stay
    exact; the V copy rounds far-below blocks to e4m3's subnormal grid, which
    the looser bound covers (as on the copy path)."""
    inp = synth.make_inputs([700, 1, 2500, 130], "mxfp4", seed=spread, block_spread=spread)
    got, lse, _ = gpu_decode(inp, mx_block_scaled=True)
    ref, ref_lse = oracle_decode(orc, inp)
    assert_parity(got, ref, lse, ref_lse, f"block-scaled spread {spread}", vmax=v_absmax(inp))


@pytest.mark.parametrize("page_size,num_splits", [(64, 0), (64, 3), (128, 5), (256, 0)])
def test_paged(orc, page_size, num_splits):
    """Pages of 64 rows or more (two 64-row boxes per tile for 64), shuffled,
    with NaN poison in every row no sequence owns; identical bits to the
    contiguous decode of the same rows with the same splits."""
    lens = [130, 0, 64, 5, 1000, 257, 128, 1]
    inp = synth.make_inputs(lens, "mxfp4", seed=11)
    pg = synth.make_paged(inp, page_size, seed=3)
    out, lse, dec = paged_gpu(inp, pg, num_splits=num_splits, mx_block_scaled=True)
    assert dec.poll_error() == 0
    ref, ref_lse = paged_oracle(orc, inp, pg)
    assert_parity(out.double().cpu().numpy(), ref, lse.double().cpu().numpy(), ref_lse,
                  f"block-scaled paged P={page_size}", gate_terms(inp, ref, ref_lse))
    cdec = binding.MLADecoder(inp.kv_indptr, "mxfp4", device=DEV, num_splits=num_splits, mx_block_scaled=True)
    out_c, lse_c = cdec(inp.q.to(DEV), inp.kv.to(DEV), inp.kv_indptr.to(DEV), inp.qo_indptr.to(DEV),
                        kv_scale=inp.block_scales.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(out, out_c) and torch.equal(lse, lse_c), f"paged P={page_size} differs from contiguous"


def test_small_pages_take_the_copy():
    """Pages of fewer than 64 rows ignore mx_scores = 1: the same bits as the copy path."""
    inp = synth.make_inputs([300, 77, 0, 513], "mxfp4", seed=5)
    pg = synth.make_paged(inp, 8, seed=2)
    out_b, lse_b, _ = paged_gpu(inp, pg, mx_block_scaled=True)
    out_c, lse_c, _ = paged_gpu(inp, pg)
    assert torch.equal(out_b, out_c) and torch.equal(lse_b, lse_c)


def test_scores_closer_than_the_copy(orc):
    """Rows with widely spread block scales: the block-scaled scores are exact,
    so the lse (a function of the scores alone) is at least as close to the
    oracle as the copy path's, which rounds far-below K blocks."""
    inp = synth.make_inputs([2000, 900], "mxfp4", seed=44, block_spread=12)
    ref, ref_lse = oracle_decode(orc, inp)
    _, lse_b, _ = gpu_decode(inp, mx_block_scaled=True)
    _, lse_c, _ = gpu_decode(inp)
    eb, ec = np.abs(lse_b - ref_lse).max(), np.abs(lse_c - ref_lse).max()
    assert eb <= ec + 1e-4, (eb, ec)
