"""Seeded synthetic inputs for MLA decode (shared by tests and the benchmark).

This module only *draws and encodes* inputs; it holds none of the decode
arithmetic (no dequantisation, no attention).  Both the CUDA path and the CPU
oracle consume the tensors it returns.

Recipe (the pages' benchmark generator is not published, so this stands in for
it; see the workload table on kernelindex "amd-mixed-mla" submission 593653,
section "Dispatch", and the shapes named on submission 754939's docstring):

* one ``torch.Generator('cpu')`` seeded with ``seed`` (default 0);
* q is drawn first, float32 N(0,1) of shape [B, 16, 576], rounded to bf16 (RNE);
* the latent KV cache is drawn next, float32 N(0,1) of shape [sum(L_b), 576],
  rounded to bf16 -- rows of sequence b are contiguous (page size 1);
* kv_indptr = exclusive prefix sum of the lengths, qo_indptr = arange(B+1);
* fp8: per-tensor scale = amax(|kv|)/448 in fp32 (amax clamped to >= 1e-12),
  stored value = e4m3fn(clamp(kv / scale, +-448)) (submission 754939,
  ``quantize_fp8``), computed from the fp32 widening of the bf16 cache;
* MXFP4: each 576-wide row is cut into 18 blocks of 32; the block's e8m0 byte is
  clamp(ceil(log2(amax/6)) + 127, 0, 254) (127 for an all-zero block), i.e. the
  block amax/6 rounded *up* to a power of two so that no element clips; elements
  are divided by 2^(byte-127) and rounded to e2m1 (nearest, ties to the even
  code); element 2i goes to the low nibble of byte i, element 2i+1 to the high
  nibble (the unpack order of submission 754939's stage-1 kernel).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

NUM_HEADS = 16
QK_DIM = 576
V_DIM = 512
MX_BLOCK = 32
FP8_MAX = 448.0

KV_DTYPES = ("bf16", "fp8", "mxfp4")

# The five benchmark workloads: (batch, kv_len per sequence, kv dtype).
WORKLOADS = {
    "bs4_kv1024_bf16": (4, 1024, "bf16"),
    "bs32_kv1024_fp8": (32, 1024, "fp8"),
    "bs4_kv8192_fp8": (4, 8192, "fp8"),
    "bs64_kv8192_fp8": (64, 8192, "fp8"),
    "bs32_kv8192_mxfp4": (32, 8192, "mxfp4"),
}
WORKLOAD_ORDER = list(WORKLOADS)


@dataclasses.dataclass
class MLAInputs:
    """One synthetic decode batch (CPU tensors)."""
    kv_dtype: str
    q: torch.Tensor                 # bf16 [B, 16, 576]
    kv_bf16: torch.Tensor           # bf16 [N, 576] (the unquantised draw)
    kv: torch.Tensor                # bf16 [N,576] | uint8 e4m3 [N,576] | uint8 packed e2m1 [N,288]
    kv_scale: torch.Tensor | None   # fp32 [1] for fp8, else None
    block_scales: torch.Tensor | None  # uint8 e8m0 [N, 18] for mxfp4, else None
    kv_indptr: torch.Tensor         # int32 [B+1]
    qo_indptr: torch.Tensor         # int32 [B+1]

    @property
    def batch(self) -> int:
        return int(self.kv_indptr.numel() - 1)

    @property
    def total_kv(self) -> int:
        return int(self.kv_indptr[-1])

    def kv_bytes(self) -> int:
        """Bytes of KV cache (plus its scales) that one decode call reads."""
        n = self.total_kv
        if self.kv_dtype == "bf16":
            return n * QK_DIM * 2
        if self.kv_dtype == "fp8":
            return n * QK_DIM + 4
        return n * (QK_DIM // 2) + n * (QK_DIM // MX_BLOCK)


def quantize_fp8(kv_bf16: torch.Tensor):
    """Per-tensor e4m3 quantisation -> (uint8 codes [N,576], fp32 scale [1])."""
    x = kv_bf16.float()
    amax = x.abs().amax().clamp(min=1e-12)
    scale = (amax / FP8_MAX).to(torch.float32)
    q8 = (x / scale).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return q8.view(torch.uint8).contiguous(), scale.reshape(1).contiguous()


def _encode_e2m1(v: np.ndarray) -> np.ndarray:
    """Round to the nearest e2m1 value (ties to the even code), saturating at 6."""
    mag = np.abs(v)
    code = ((mag > 0.25).astype(np.uint8) + (mag >= 0.75) + (mag > 1.25) + (mag >= 1.75)
            + (mag > 2.5) + (mag >= 3.5) + (mag > 5.0)).astype(np.uint8)
    return code | (np.signbit(v).astype(np.uint8) << 3)


def quantize_mxfp4(kv_bf16: torch.Tensor):
    """MXFP4 encoding -> (packed e2m1 uint8 [N,288], e8m0 uint8 [N,18])."""
    x = kv_bf16.float().numpy().astype(np.float64)
    n = x.shape[0]
    xb = x.reshape(n, QK_DIM // MX_BLOCK, MX_BLOCK)
    amax = np.abs(xb).max(axis=2)
    with np.errstate(divide="ignore"):
        e = np.where(amax > 0, np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / 6.0)), 0.0)
    e8 = np.clip(e + 127, 0, 254).astype(np.uint8)
    scaled = xb / np.ldexp(1.0, e8.astype(np.int32) - 127)[..., None]
    nib = _encode_e2m1(scaled).reshape(n, QK_DIM)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return torch.from_numpy(np.ascontiguousarray(packed)), torch.from_numpy(np.ascontiguousarray(e8))


def make_inputs(kv_lens, kv_dtype: str = "bf16", seed: int = 0, q_mult: float = 1.0,
                block_spread: int = 0) -> MLAInputs:
    """Draw one decode batch.  ``kv_lens``: list of per-sequence lengths.
    ``block_spread`` > 0 scales the 32-element blocks 3j+1 and 3j+2 of every KV
    row by 2^-block_spread and 2^-2 block_spread before quantisation (rows
    whose block scales differ widely)."""
    if kv_dtype not in KV_DTYPES:
        raise ValueError(f"kv_dtype must be one of {KV_DTYPES}")
    lens = [int(x) for x in kv_lens]
    if any(x < 0 for x in lens):
        raise ValueError("negative kv length")
    b = len(lens)
    n = int(sum(lens))
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = (torch.randn(b, NUM_HEADS, QK_DIM, generator=g, dtype=torch.float32) * q_mult).to(torch.bfloat16)
    kv_f = torch.randn(n, QK_DIM, generator=g, dtype=torch.float32)
    if block_spread:
        gain = torch.ones(QK_DIM // MX_BLOCK, dtype=torch.float32)
        gain[1::3] = 2.0 ** -block_spread
        gain[2::3] = 2.0 ** (-2 * block_spread)
        kv_f = kv_f * gain.repeat_interleave(MX_BLOCK)
    kv_bf16 = kv_f.to(torch.bfloat16)
    ind = torch.zeros(b + 1, dtype=torch.int32)
    if b:
        ind[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    qo = torch.arange(b + 1, dtype=torch.int32)
    kv_scale = block_scales = None
    if kv_dtype == "bf16":
        kv = kv_bf16
    elif kv_dtype == "fp8":
        kv, kv_scale = quantize_fp8(kv_bf16)
    else:
        kv, block_scales = quantize_mxfp4(kv_bf16)
    return MLAInputs(kv_dtype, q.contiguous(), kv_bf16, kv.contiguous(), kv_scale, block_scales, ind, qo)


def make_workload(name: str, seed: int = 0) -> MLAInputs:
    batch, kv_len, dt = WORKLOADS[name]
    return make_inputs([kv_len] * batch, dt, seed=seed)


@dataclasses.dataclass
class PagedKV:
    """A paged copy of a contiguous cache (CPU tensors).

    Sequence b owns the pages ``kv_indices[page_indptr[b]:page_indptr[b+1]]`` in
    that order; its rows are those pages' rows in order, all ``page_size`` rows
    of each page but the last, which holds ``last_page_len[b]`` of them (the
    layout the pages' AITER call takes: ``kv.view(num_pages, page_size, 1, 576)``
    with ``kv_indptr`` counted in pages, ``kv_indices`` and ``kv_last_page_lens``).
    """
    page_size: int
    num_pages: int
    kv: torch.Tensor                   # num_pages * page_size rows, same row format as MLAInputs.kv
    block_scales: torch.Tensor | None  # uint8 e8m0 [num_pages * page_size, 18] for mxfp4
    page_indptr: torch.Tensor          # int32 [B+1], counted in pages
    kv_indices: torch.Tensor           # int32 [page_indptr[-1]]
    last_page_len: torch.Tensor        # int32 [B]


# Bytes no decode may use: NaN in every format that has one (bf16 0x7fc0, e4m3
# 0x7f, e8m0 0xff); e2m1 has no NaN, so for MXFP4 the rows' scales carry it.
_POISON_BF16 = 0x7FC0
_POISON_BYTE = {"fp8": 0x7F, "mxfp4": 0x77}
_POISON_E8M0 = 0xFF


def make_paged(inp: MLAInputs, page_size: int, seed: int = 0, spare_pages: int = 3) -> PagedKV:
    """Scatters the rows of ``inp`` into a paged cache: each sequence's rows go,
    ``page_size`` at a time, to pages at seeded random positions of the cache.
    ``spare_pages`` pages that no sequence references, and the unused rows of
    every last page, are filled with poison (NaN codes), so that a decode that
    reads anything but the sequences' own rows gives a non-finite result."""
    if page_size < 1:
        raise ValueError("page_size must be >= 1")
    ind = inp.kv_indptr.tolist()
    b = len(ind) - 1
    npages = [-(-(ind[i + 1] - ind[i]) // page_size) for i in range(b)]
    used = int(sum(npages))
    num_pages = used + int(spare_pages)
    g = torch.Generator("cpu").manual_seed(int(seed) + 7919)
    perm = torch.randperm(num_pages, generator=g)[:used].to(torch.int32)  # physical page of logical page j
    rows = num_pages * page_size
    if inp.kv_dtype == "bf16":
        kv = torch.full((rows, QK_DIM), 0, dtype=torch.int16)
        kv.fill_(_POISON_BF16)
        kv = kv.view(torch.bfloat16)
    else:
        kv = torch.full((rows, inp.kv.shape[1]), _POISON_BYTE[inp.kv_dtype], dtype=torch.uint8)
    bs = None
    if inp.kv_dtype == "mxfp4":
        bs = torch.full((rows, inp.block_scales.shape[1]), _POISON_E8M0, dtype=torch.uint8)
    page_indptr = torch.zeros(b + 1, dtype=torch.int32)
    last = torch.zeros(b, dtype=torch.int32)
    j = 0
    for i in range(b):
        start, L = ind[i], ind[i + 1] - ind[i]
        for k in range(npages[i]):
            n = min(page_size, L - k * page_size)
            dst = int(perm[j + k]) * page_size
            kv[dst:dst + n] = inp.kv[start + k * page_size:start + k * page_size + n]
            if bs is not None:
                bs[dst:dst + n] = inp.block_scales[start + k * page_size:start + k * page_size + n]
        if npages[i]:
            last[i] = L - (npages[i] - 1) * page_size
        j += npages[i]
        page_indptr[i + 1] = j
    return PagedKV(int(page_size), num_pages, kv.contiguous(), bs, page_indptr, perm.clone(), last)
