"""Paged KV cache on the GPU, through the C ABI: parity with the fp64 oracle's
paged decode, and identity with the contiguous decode of the same rows.

The page layout is the one the pages' AITER call takes (kernelindex
"amd-mixed-mla" submission 703488: kv.view(num_pages, page_size, 1, 576), a
page-counted kv_indptr, kv_indices and kv_last_page_lens; submission 616673
calls it with pages of 2 and 8 rows).  Page sizes run from 1 to 256 rows.  Every case scatters
a contiguous cache into pages at random positions, with partial last pages, an
empty sequence, and NaN poison in every row that no sequence owns (spare pages
and the tail of each last page): a kernel that reads anything else gives a
non-finite result.  Tolerances are those of test_parity_gpu.py.
"""
import numpy as np
import pytest
import torch

from mla_attention_decode_gb300 import binding, synth
from test_parity_gpu import CODES, assert_parity, gate_terms, orc, built  # noqa: F401 (fixtures)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
LENS = [130, 0, 64, 5, 1000, 257, 128, 1]


def paged_gpu(inp, pg, num_splits=0, kv_indices=None, mx_block_scaled=False):
    dec = binding.PagedMLADecoder(pg.page_indptr, pg.last_page_len, pg.page_size, pg.num_pages, inp.kv_dtype,
                                  device=DEV, num_splits=num_splits, mx_block_scaled=mx_block_scaled)
    scale = inp.kv_scale if inp.kv_dtype == "fp8" else pg.block_scales
    idx = pg.kv_indices if kv_indices is None else kv_indices
    out, lse = dec(inp.q.to(DEV), pg.kv.to(DEV), pg.page_indptr.to(DEV), idx.to(DEV), pg.last_page_len.to(DEV),
                   inp.qo_indptr.to(DEV), kv_scale=None if scale is None else scale.to(DEV))
    torch.cuda.synchronize()
    return out, lse, dec


def paged_oracle(orc, inp, pg):
    return orc.decode_paged(CODES[inp.kv_dtype], inp.q, pg.kv, pg.page_indptr, pg.kv_indices, pg.last_page_len,
                            pg.page_size, inp.qo_indptr,
                            kv_scale=None if inp.kv_scale is None else inp.kv_scale.numpy(),
                            block_scales=None if pg.block_scales is None else pg.block_scales.numpy())


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "mxfp4"])
@pytest.mark.parametrize("page_size", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_paged_parity(orc, dtype, page_size):
    inp = synth.make_inputs(LENS, dtype, seed=page_size + 5)
    pg = synth.make_paged(inp, page_size, seed=page_size)
    out, lse, dec = paged_gpu(inp, pg)
    assert dec.poll_error() == 0
    ref, ref_lse = paged_oracle(orc, inp, pg)
    assert_parity(out.double().cpu().numpy(), ref, lse.double().cpu().numpy(), ref_lse,
                  f"paged {dtype} P={page_size}", gate_terms(inp, ref, ref_lse))


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "mxfp4"])
@pytest.mark.parametrize("page_size,num_splits", [(1, 0), (2, 3), (4, 0), (8, 0), (16, 5), (32, 2), (64, 0), (64, 3), (128, 5)])
def test_paged_equals_contiguous(dtype, page_size, num_splits):
    """The same rows in pages or in one block, with the same splits: identical bits."""
    inp = synth.make_inputs(LENS, dtype, seed=11)
    pg = synth.make_paged(inp, page_size, seed=3)
    out_p, lse_p, dec = paged_gpu(inp, pg, num_splits=num_splits)
    assert dec.poll_error() == 0
    cdec = binding.MLADecoder(inp.kv_indptr, dtype, device=DEV, num_splits=num_splits)
    scale = inp.kv_scale if dtype == "fp8" else inp.block_scales
    out_c, lse_c = cdec(inp.q.to(DEV), inp.kv.to(DEV), inp.kv_indptr.to(DEV), inp.qo_indptr.to(DEV),
                        kv_scale=None if scale is None else scale.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_c), f"paged {dtype} P={page_size}: output differs from the contiguous decode"
    assert torch.equal(lse_p, lse_c)


def test_paged_long_sequences_split(orc):
    """Sequences of thousands of rows over 64-row pages, cut into many splits."""
    lens = [3000, 64, 4097, 0, 900]
    inp = synth.make_inputs(lens, "fp8", seed=17)
    pg = synth.make_paged(inp, 64, seed=9)
    out, lse, dec = paged_gpu(inp, pg)
    assert dec.plan.splits_max > 1
    assert dec.poll_error() == 0
    ref, ref_lse = paged_oracle(orc, inp, pg)
    assert_parity(out.double().cpu().numpy(), ref, lse.double().cpu().numpy(), ref_lse, "paged long",
                  gate_terms(inp, ref, ref_lse))


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "mxfp4"])
@pytest.mark.parametrize("page_size", [1, 2, 8, 16])
def test_small_pages_long_sequences(orc, dtype, page_size):
    """Pages of 1 to 16 rows with a shuffled page table under sequences of
    thousands of rows, split over several CTAs (the pages' own paged call uses
    pages of 2 and 8 rows)."""
    lens = [3000, 1, 2047, 0, 700]
    inp = synth.make_inputs(lens, dtype, seed=page_size + 29)
    pg = synth.make_paged(inp, page_size, seed=page_size + 3)
    out, lse, dec = paged_gpu(inp, pg)
    assert dec.plan.splits_max > 1
    assert dec.poll_error() == 0
    ref, ref_lse = paged_oracle(orc, inp, pg)
    assert_parity(out.double().cpu().numpy(), ref, lse.double().cpu().numpy(), ref_lse,
                  f"small pages {dtype} P={page_size}", gate_terms(inp, ref, ref_lse))


def test_paged_bad_page_index_is_reported():
    """A page index outside [0, num_pages) is flagged (and page 0 read instead)."""
    inp = synth.make_inputs([200, 70], "fp8", seed=23)
    pg = synth.make_paged(inp, 64, seed=1, spare_pages=0)
    bad = pg.kv_indices.clone()
    bad[1] = pg.num_pages
    _, _, dec = paged_gpu(inp, pg, kv_indices=bad)
    assert dec.poll_error() == binding.MLA_ERR_DEVICE_INDEX
    _, _, dec = paged_gpu(inp, pg)
    assert dec.poll_error() == 0
