"""Pins for the fp64 oracle: each pin checks the oracle against something other
than itself -- a library routine (torch's fp8 conversion, float64
scaled_dot_product_attention), a value table printed by the pages, a closed form,
or an invariant of the definition.  Each function raises AssertionError on a
mismatch.  ``ALL_PINS`` is run against the real oracle (all must pass) and
against planted-mistake builds of it (each must trip at least one pin).

Definition pinned: kernelindex "amd-mixed-mla" submission 593653, section
"Slow fallback" (``_bmm_reference``) -- scores = q . kv^T * sm_scale, softmax,
output = probs . kv[:, :512]; lse = max + ln(sum).
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

from mla_attention_decode_gb300 import synth

KV_CODES = {"bf16": 0, "fp8": 1, "mxfp4": 2}
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden_e2m1() -> np.ndarray:
    table = np.zeros(16, dtype=np.float64)
    with open(os.path.join(GOLDEN, "e2m1_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            code, val = line.split()
            table[int(code)] = float(val)
    return table


def golden_constants() -> dict:
    out = {}
    with open(os.path.join(GOLDEN, "constants.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                out[k] = float(v)
    return out


# --------------------------------------------------------------------------
# Independent dequantisation (library routines and the printed table only).
# --------------------------------------------------------------------------
def lib_dequant(inp: synth.MLAInputs) -> np.ndarray:
    """KV rows as float64 [N, 576], without using the oracle."""
    if inp.kv_dtype == "bf16":
        return inp.kv.to(torch.float64).numpy()
    if inp.kv_dtype == "fp8":
        return (inp.kv.view(torch.float8_e4m3fn).to(torch.float64) * float(inp.kv_scale[0])).numpy()
    tab = golden_e2m1()
    packed = inp.kv.numpy()
    n = packed.shape[0]
    nib = np.empty((n, 576), dtype=np.uint8)
    nib[:, 0::2] = packed & 0xF
    nib[:, 1::2] = packed >> 4
    scales = np.ldexp(1.0, inp.block_scales.numpy()[:, :18].astype(np.int32) - 127)
    return tab[nib] * np.repeat(scales, 32, axis=1)


def sdpa_reference(inp: synth.MLAInputs) -> np.ndarray:
    """torch float64 scaled_dot_product_attention with 1 shared KV head."""
    kv = torch.from_numpy(lib_dequant(inp))
    q = inp.q.to(torch.float64)
    ind = inp.kv_indptr.tolist()
    qo = inp.qo_indptr.tolist()
    outs = []
    for b in range(inp.batch):
        k = kv[ind[b]:ind[b + 1]]
        qb = q[qo[b]].view(1, 16, 1, 576)
        kb = k.view(1, 1, -1, 576).expand(1, 16, -1, 576)
        vb = kb[..., :512]
        outs.append(F.scaled_dot_product_attention(qb, kb, vb, scale=1.0 / 24.0).view(16, 512))
    return torch.stack(outs).numpy()


def run(orc, inp: synth.MLAInputs, q=None, kv=None, kv_indptr=None, qo_indptr=None):
    return orc.decode(KV_CODES[inp.kv_dtype], inp.q if q is None else q, inp.kv if kv is None else kv,
                      inp.kv_indptr if kv_indptr is None else kv_indptr,
                      inp.qo_indptr if qo_indptr is None else qo_indptr,
                      kv_scale=None if inp.kv_scale is None else inp.kv_scale.numpy(),
                      block_scales=None if inp.block_scales is None else inp.block_scales.numpy())


def _close(a, b, tol=1e-11, what=""):
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol * max(1.0, float(np.max(np.abs(b))) if b.size else 1.0), f"{what}: max err {err}"


# --------------------------------------------------------------------------
# Decoder pins
# --------------------------------------------------------------------------
def pin_e4m3_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.decode_e4m3(codes)
    nan_ref, nan_got = np.isnan(ref), np.isnan(got)
    assert np.array_equal(nan_ref, nan_got), "e4m3 NaN codes differ"
    assert np.array_equal(ref[~nan_ref], got[~nan_got]), "e4m3 values differ from torch float8_e4m3fn"
    assert np.array_equal(np.signbit(ref[~nan_ref]), np.signbit(got[~nan_got])), "e4m3 sign of zero"


def pin_e2m1_table(orc):
    got = orc.decode_e2m1(np.arange(16, dtype=np.uint8))
    ref = golden_e2m1()
    assert np.array_equal(got, ref), f"e2m1 table mismatch: {got}"
    assert np.array_equal(np.signbit(got), np.signbit(ref)), "e2m1 sign of zero"


def pin_e8m0_closed_form(orc):
    got = orc.decode_e8m0(np.arange(256, dtype=np.uint8))
    for e in range(255):
        assert got[e] == math.ldexp(1.0, e - 127), f"e8m0 {e}"
    assert math.isnan(got[255]), "e8m0 255 must be NaN"


def pin_bf16_widen(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # finite only
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(orc.decode_bf16(bits), ref), "bf16 widening"


def pin_constants(orc):
    c = golden_constants()
    assert c["sm_scale"] == 1.0 / math.sqrt(c["qk_head_dim"]) == 1.0 / 24.0
    assert c["qk_head_dim"] == c["q_nope_dim"] + c["q_rope_dim"] and c["v_head_dim"] == c["q_nope_dim"]
    # sm_scale pinned through the oracle: q = e_0 (unit vector), one row with k_0 = 24
    # gives a score of exactly 1, and with a second all-zero row lse = ln(e + 1).
    q = torch.zeros(1, 16, 576, dtype=torch.bfloat16)
    q[0, :, 0] = 1.0
    kv = torch.zeros(2, 576, dtype=torch.bfloat16)
    kv[0, 0] = 24.0
    out, lse = orc.decode(0, q, kv, [0, 2])
    _close(lse, np.full((1, 16), math.log(math.e + 1.0)), 1e-14, "sm_scale pin lse")
    _close(out[0, :, 0], np.full(16, 24.0 * math.e / (math.e + 1.0)), 1e-13, "sm_scale pin out")


# --------------------------------------------------------------------------
# Library special case: float64 SDPA
# --------------------------------------------------------------------------
def _pin_sdpa(orc, dt):
    inp = synth.make_inputs([1, 33, 70], dt, seed=11)
    out, _ = run(orc, inp)
    _close(out, sdpa_reference(inp), 1e-11, f"sdpa {dt}")


def pin_sdpa_bf16(orc):
    _pin_sdpa(orc, "bf16")


def pin_sdpa_fp8(orc):
    _pin_sdpa(orc, "fp8")


def pin_sdpa_mxfp4(orc):
    _pin_sdpa(orc, "mxfp4")


# --------------------------------------------------------------------------
# Invariants and closed forms
# --------------------------------------------------------------------------
def _with_rows(inp: synth.MLAInputs, rows: torch.Tensor, block_scales=None) -> synth.MLAInputs:
    return synth.MLAInputs(inp.kv_dtype, inp.q, inp.kv_bf16, rows.contiguous(), inp.kv_scale,
                           block_scales if block_scales is not None else inp.block_scales,
                           inp.kv_indptr, inp.qo_indptr)


def pin_identical_rows(orc):
    """L copies of one row r: out = dequant(r)[:512] for every head; lse(L) - lse(1) = ln L."""
    for dt in ("bf16", "fp8", "mxfp4"):
        base = synth.make_inputs([1], dt, seed=3)
        L = 37
        rows = base.kv.repeat(L, 1)
        bs = None if base.block_scales is None else base.block_scales.repeat(L, 1)
        ind = torch.tensor([0, L], dtype=torch.int32)
        inp = synth.MLAInputs(dt, base.q, base.kv_bf16, rows, base.kv_scale, bs, ind, base.qo_indptr)
        out, lse = run(orc, inp)
        r = lib_dequant(base)[0, :512]
        _close(out[0], np.broadcast_to(r, (16, 512)), 1e-12, f"identical rows {dt}")
        _, lse1 = run(orc, base)
        _close(lse - lse1, np.full_like(lse, math.log(L)), 1e-12, f"identical rows lse {dt}")


def pin_single_row(orc):
    """kv_len = 1: softmax weight 1, out = dequant(row)[:512], lse = the row's score."""
    for dt in ("bf16", "fp8", "mxfp4"):
        inp = synth.make_inputs([1, 1], dt, seed=5)
        out, lse = run(orc, inp)
        k = lib_dequant(inp)
        q = inp.q.to(torch.float64).numpy()
        for b in range(2):
            _close(out[b], np.broadcast_to(k[b, :512], (16, 512)), 1e-12, f"len1 out {dt}")
            s = np.array([math.fsum(q[b, h] * k[b]) / 24.0 for h in range(16)])
            _close(lse[b], s, 1e-12, f"len1 lse {dt}")


def pin_zero_query(orc):
    """q = 0: uniform weights, out = mean of the V rows, lse = ln L."""
    inp = synth.make_inputs([5, 64], "fp8", seed=9)
    q0 = torch.zeros_like(inp.q)
    out, lse = run(orc, inp, q=q0)
    k = lib_dequant(inp)
    ind = inp.kv_indptr.tolist()
    for b in range(2):
        mean = k[ind[b]:ind[b + 1], :512].mean(axis=0)
        _close(out[b], np.broadcast_to(mean, (16, 512)), 1e-12, "zero q mean")
        _close(lse[b], np.full(16, math.log(ind[b + 1] - ind[b])), 1e-12, "zero q lse")


def pin_permutation_and_isolation(orc):
    inp = synth.make_inputs([20, 31, 9], "mxfp4", seed=13)
    out, lse = run(orc, inp)
    ind = inp.kv_indptr.tolist()
    perm = torch.arange(inp.total_kv)
    g = torch.Generator().manual_seed(1)
    perm[ind[1]:ind[2]] = ind[1] + torch.randperm(ind[2] - ind[1], generator=g)
    p_inp = _with_rows(inp, inp.kv[perm], inp.block_scales[perm])
    out_p, lse_p = run(orc, p_inp)
    _close(out_p, out, 1e-12, "row permutation")
    _close(lse_p, lse, 1e-12, "row permutation lse")
    # perturb every row outside sequence 1: sequence 1 must not move at all
    rows = inp.kv.clone()
    rows[:ind[1]] ^= 0x5A
    rows[ind[2]:] ^= 0x33
    out_x, lse_x = run(orc, _with_rows(inp, rows))
    assert np.array_equal(out_x[1], out[1]) and np.array_equal(lse_x[1], lse[1]), "isolation"
    assert not np.array_equal(out_x[0], out[0]), "perturbation had no effect on sequence 0"


def pin_large_logits(orc):
    """q = 40 * row j: scores near 960 dominate -> out ~ row j, finite (max subtraction)."""
    inp = synth.make_inputs([8], "bf16", seed=17)
    j = 3
    q = (inp.kv[j].to(torch.float32) * 40.0).to(torch.bfloat16).view(1, 1, 576).expand(1, 16, 576).contiguous()
    out, lse = run(orc, inp, q=q)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse)), "overflow with large logits"
    _close(out[0], np.broadcast_to(lib_dequant(inp)[j, :512], (16, 512)), 1e-12, "large logits argmax row")


def pin_split_combine(orc):
    """Splitting a sequence anywhere and LSE-combining equals the unsplit result."""
    for dt in ("bf16", "fp8", "mxfp4"):
        inp = synth.make_inputs([50], dt, seed=19)
        out, lse = run(orc, inp)
        kvs = None if inp.kv_scale is None else inp.kv_scale.numpy()
        bs = None if inp.block_scales is None else inp.block_scales.numpy()
        for cuts in ([0, 50], [0, 1, 50], [0, 17, 17, 33, 50], [0, 10, 20, 30, 40, 49, 50]):
            parts = [orc.partial(KV_CODES[dt], inp.q, inp.kv, 0, cuts[i], cuts[i + 1], kvs, bs)
                     for i in range(len(cuts) - 1)]
            o = np.stack([p[0] for p in parts])
            l = np.stack([p[1] for p in parts])
            oc, lc = orc.combine(o, l)
            _close(oc, out[0], 1e-12, f"split/combine {dt} {cuts}")
            _close(lc, lse[0], 1e-12, f"split/combine lse {dt} {cuts}")


def pin_empty_sequence(orc):
    inp = synth.make_inputs([0, 4, 0], "fp8", seed=23)
    out, lse = run(orc, inp)
    for b in (0, 2):
        assert np.all(out[b] == 0.0), "empty sequence output must be 0"
        assert np.all(np.isneginf(lse[b])), "empty sequence lse must be -inf"
    ref = sdpa_reference(synth.MLAInputs(inp.kv_dtype, inp.q[1:2], inp.kv_bf16, inp.kv, inp.kv_scale, None,
                                         torch.tensor([0, 4], dtype=torch.int32),
                                         torch.tensor([0, 1], dtype=torch.int32)))
    _close(out[1], ref[0], 1e-11, "sequence between empties")


def pin_qo_indptr(orc):
    """qo_indptr selects the query row of each sequence."""
    inp = synth.make_inputs([6, 7, 8], "bf16", seed=29)
    q3 = inp.q
    q_big = torch.cat([q3[2:3], q3[0:1], torch.zeros_like(q3[0:1]), q3[1:2]], 0)
    qo = torch.tensor([1, 3, 0, 4], dtype=torch.int32)  # q row of b = qo[b]
    out_a, lse_a = run(orc, inp)
    out_b, lse_b = run(orc, inp, q=q_big, qo_indptr=qo)
    _close(out_b, out_a, 1e-14, "qo_indptr row selection")
    _close(lse_b, lse_a, 1e-14, "qo_indptr row selection lse")


def pin_paged_cache(orc):
    """A paged cache (submission 703488's kv.view(num_pages, page_size, 1, 576) with
    page-counted kv_indptr, kv_indices and kv_last_page_lens) holds the same rows as
    the contiguous cache it was scattered from, so the paged decode must equal the
    contiguous decode exactly -- with the pages in a random order, partial last
    pages, an empty sequence, and poison (NaN) in every row no sequence owns."""
    for dt in ("bf16", "fp8", "mxfp4"):
        inp = synth.make_inputs([130, 0, 64, 5, 200], dt, seed=41)
        ref_out, ref_lse = run(orc, inp)
        for page_size in (1, 3, 64):
            pg = synth.make_paged(inp, page_size, seed=page_size)
            out, lse = orc.decode_paged(KV_CODES[dt], inp.q, pg.kv, pg.page_indptr, pg.kv_indices,
                                        pg.last_page_len, page_size, inp.qo_indptr,
                                        kv_scale=None if inp.kv_scale is None else inp.kv_scale.numpy(),
                                        block_scales=None if pg.block_scales is None else pg.block_scales.numpy())
            assert np.array_equal(out, ref_out), f"paged {dt} P={page_size}: output differs"
            assert np.array_equal(lse, ref_lse), f"paged {dt} P={page_size}: lse differs"


def pin_multi_token_causal(orc):
    """q_len query tokens per sequence, the causal reading: token i sees the
    first L - (q_len - 1 - i) rows.  Checked against torch float64
    scaled_dot_product_attention with an explicit causal mask (a library
    routine), and q_len = 1 against the single-token decode."""
    for dt in ("bf16", "fp8", "mxfp4"):
        q_len = 3
        base = synth.make_inputs([5, 40, 3], dt, seed=17)
        qg = torch.Generator("cpu").manual_seed(5)
        q = torch.randn(3 * q_len, 16, 576, generator=qg).to(torch.bfloat16)
        out, lse = orc.decode_multi(KV_CODES[dt], q, base.kv, base.kv_indptr, q_len,
                                    kv_scale=None if base.kv_scale is None else base.kv_scale.numpy(),
                                    block_scales=None if base.block_scales is None else base.block_scales.numpy())
        k_all = torch.from_numpy(lib_dequant(base))
        ind = base.kv_indptr.tolist()
        for b in range(3):
            k = k_all[ind[b]:ind[b + 1]]
            L = k.shape[0]
            qb = q[b * q_len:(b + 1) * q_len].to(torch.float64).transpose(0, 1)  # [16, q_len, 576]
            mask = torch.arange(L)[None, :] <= (L - q_len + torch.arange(q_len))[:, None]
            ref = F.scaled_dot_product_attention(qb, k[None], k[None, :, :512], attn_mask=mask[None],
                                                 scale=1.0 / 24.0).transpose(0, 1)
            _close(out[b * q_len:(b + 1) * q_len], ref.numpy(), 1e-11, f"multi-token {dt} b={b}")
        one, lse1 = orc.decode_multi(KV_CODES[dt], base.q, base.kv, base.kv_indptr, 1,
                                     kv_scale=None if base.kv_scale is None else base.kv_scale.numpy(),
                                     block_scales=None if base.block_scales is None else base.block_scales.numpy())
        ref1, rlse1 = run(orc, base)
        _close(one, ref1, 1e-14, f"multi-token q_len=1 {dt}")
        _close(lse1, rlse1, 1e-14, f"multi-token q_len=1 lse {dt}")


ALL_PINS = [
    pin_e4m3_all_codes, pin_e2m1_table, pin_e8m0_closed_form, pin_bf16_widen, pin_constants,
    pin_sdpa_bf16, pin_sdpa_fp8, pin_sdpa_mxfp4, pin_identical_rows, pin_single_row,
    pin_zero_query, pin_permutation_and_isolation, pin_large_logits, pin_split_combine,
    pin_empty_sequence, pin_qo_indptr, pin_paged_cache, pin_multi_token_causal,
]

# Planted mistakes compiled into oracle variants (see mla_oracle.c, ORACLE_MUTANT).
MUTANTS = {
    1: "rope columns dropped from the scores",
    2: "V read from columns 64..575",
    3: "sm_scale ignored",
    4: "fp8 per-tensor scale ignored",
    5: "MXFP4 nibble order swapped",
    6: "e8m0 bias 128",
    7: "softmax without max subtraction",
    8: "lse in log2",
    9: "every head reads query head 0",
    10: "e4m3 subnormals decoded as normals",
    11: "paged cache: the last page read in full",
    12: "paged cache: the page table ignored",
    13: "multi-token: a token's own row left out",
}
