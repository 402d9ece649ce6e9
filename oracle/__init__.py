"""fp64 CPU oracle for single-token MLA decode -- TEST INFRASTRUCTURE ONLY.

This package is the checker that the CUDA path is compared against.  Only the
test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it.  The product library never loads it, and it shares no code with the
CUDA path: the arithmetic lives in ``mla_oracle.c`` (plain C, fp64, compiled with
gcc -O2, no fast-math), and this module only builds it and marshals numpy arrays.

What it computes is the definition on kernelindex "amd-mixed-mla" submission
593653, section "Slow fallback" (``_bmm_reference``): scores = q . kv^T * sm_scale,
softmax over the sequence, output = probs . kv[:, :512], evaluated without any
rounding, plus lse = max + ln(sum) per head.  See ``mla_oracle.c`` for the
dequantisation rules and their sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")

KV_BF16, KV_FP8_E4M3, KV_MXFP4 = 0, 1, 2
NUM_HEADS, QK_DIM, V_DIM = 16, 576, 512
SM_SCALE = 1.0 / 24.0  # 1/sqrt(576), exact

_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def lib_path(mutant: int = 0) -> str:
    name = "libmla_oracle.so" if mutant == 0 else f"libmla_oracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or a planted-mistake variant) with gcc; returns the .so path."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-shared", "-fPIC", "-std=c11",
           f"-DORACLE_MUTANT={mutant}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    for name in ("oracle_decode_bf16_array", "oracle_decode_e4m3_array",
                 "oracle_decode_e2m1_array", "oracle_decode_e8m0_array"):
        f = getattr(lib, name)
        f.argtypes = [P, P, i64]
        f.restype = None
    lib.oracle_mla_decode.argtypes = [i32, P, P, P, i64, dbl, P, P, i32, dbl, P, P, i32]
    lib.oracle_mla_decode.restype = i32
    lib.oracle_mla_decode_paged.argtypes = [i32, P, P, P, i64, dbl, P, P, P, i32, i64, P, i32, dbl, P, P, i32]
    lib.oracle_mla_decode_paged.restype = i32
    lib.oracle_mla_decode_multi.argtypes = [i32, P, P, P, i64, dbl, P, P, i32, i32, dbl, P, P, i32]
    lib.oracle_mla_decode_multi.restype = i32
    lib.oracle_mla_partial.argtypes = [i32, P, P, P, i64, dbl, i64, i64, i64, dbl, P, P]
    lib.oracle_mla_partial.restype = i32
    lib.oracle_mla_combine.argtypes = [i32, P, P, P, P]
    lib.oracle_mla_combine.restype = i32
    lib.oracle_mutant_id.argtypes = []
    lib.oracle_mutant_id.restype = i32
    return lib


def load(mutant: int = 0) -> "Oracle":
    with _lock:
        if mutant not in _libs:
            _libs[mutant] = _bind(ctypes.CDLL(build(mutant)))
        return Oracle(_libs[mutant])


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    """bf16 tensors/arrays -> contiguous uint16 bit patterns."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a).view(np.uint16))


def _u8(a) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            return np.ascontiguousarray(a.detach().cpu().contiguous().view(torch.uint8).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(a).view(np.uint8))


class Oracle:
    """numpy front end of one compiled oracle library."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib
        self.mutant = lib.oracle_mutant_id()

    # -- decoders ---------------------------------------------------------
    def _dec(self, fn, codes: np.ndarray) -> np.ndarray:
        codes = np.ascontiguousarray(codes)
        out = np.empty(codes.shape, dtype=np.float64)
        fn(_ptr(codes), _ptr(out), codes.size)
        return out

    def decode_bf16(self, bits) -> np.ndarray:
        return self._dec(self.lib.oracle_decode_bf16_array, _u16(bits))

    def decode_e4m3(self, codes) -> np.ndarray:
        return self._dec(self.lib.oracle_decode_e4m3_array, _u8(codes))

    def decode_e2m1(self, nibbles) -> np.ndarray:
        return self._dec(self.lib.oracle_decode_e2m1_array, _u8(nibbles))

    def decode_e8m0(self, codes) -> np.ndarray:
        return self._dec(self.lib.oracle_decode_e8m0_array, _u8(codes))

    # -- attention --------------------------------------------------------
    @staticmethod
    def _kv_args(kv_dtype: int, kv, kv_scale, block_scales):
        if kv_dtype == KV_BF16:
            kv_a = _u16(kv)
        else:
            kv_a = _u8(kv)
        sc = 1.0 if kv_scale is None else float(np.asarray(kv_scale, dtype=np.float64).reshape(-1)[0])
        bs, stride = None, 0
        if kv_dtype == KV_MXFP4:
            bs = _u8(block_scales)
            stride = bs.shape[-1]
        return kv_a, sc, bs, stride

    def decode(self, kv_dtype: int, q, kv, kv_indptr, qo_indptr=None, kv_scale=None,
               block_scales=None, sm_scale: float = SM_SCALE, num_threads: int = 0):
        """Returns (out [B,16,512] float64, lse [B,16] float64)."""
        q_a = _u16(q)
        kv_a, sc, bs, stride = self._kv_args(kv_dtype, kv, kv_scale, block_scales)
        ind = np.ascontiguousarray(np.asarray(kv_indptr, dtype=np.int32))
        batch = ind.size - 1
        qo = (np.arange(batch + 1, dtype=np.int32) if qo_indptr is None
              else np.ascontiguousarray(np.asarray(qo_indptr, dtype=np.int32)))
        out = np.zeros((batch, NUM_HEADS, V_DIM), dtype=np.float64)
        lse = np.zeros((batch, NUM_HEADS), dtype=np.float64)
        rc = self.lib.oracle_mla_decode(kv_dtype, _ptr(q_a), _ptr(kv_a), _ptr(bs), stride, sc,
                                        _ptr(ind), _ptr(qo), batch, float(sm_scale), _ptr(out),
                                        _ptr(lse), int(num_threads))
        if rc != 0:
            raise ValueError("oracle_mla_decode rejected its arguments")
        return out, lse

    def decode_paged(self, kv_dtype: int, q, kv, page_indptr, kv_indices, last_page_len, page_size: int,
                     qo_indptr=None, kv_scale=None, block_scales=None, sm_scale: float = SM_SCALE,
                     num_threads: int = 0):
        """Paged cache: kv holds num_pages * page_size rows; sequence b reads the pages
        kv_indices[page_indptr[b]:page_indptr[b+1]], the last one for last_page_len[b]
        rows.  Returns (out [B,16,512] float64, lse [B,16] float64)."""
        q_a = _u16(q)
        kv_a, sc, bs, stride = self._kv_args(kv_dtype, kv, kv_scale, block_scales)
        pin = np.ascontiguousarray(np.asarray(page_indptr, dtype=np.int32))
        idx = np.ascontiguousarray(np.asarray(kv_indices, dtype=np.int32).reshape(-1))
        last = np.ascontiguousarray(np.asarray(last_page_len, dtype=np.int32).reshape(-1))
        batch = pin.size - 1
        num_pages = kv_a.shape[0] // int(page_size)
        qo = (np.arange(batch + 1, dtype=np.int32) if qo_indptr is None
              else np.ascontiguousarray(np.asarray(qo_indptr, dtype=np.int32)))
        out = np.zeros((batch, NUM_HEADS, V_DIM), dtype=np.float64)
        lse = np.zeros((batch, NUM_HEADS), dtype=np.float64)
        rc = self.lib.oracle_mla_decode_paged(kv_dtype, _ptr(q_a), _ptr(kv_a), _ptr(bs), stride, sc,
                                              _ptr(pin), _ptr(idx if idx.size else None),
                                              _ptr(last if last.size else None), int(page_size),
                                              int(num_pages), _ptr(qo), batch, float(sm_scale),
                                              _ptr(out), _ptr(lse), int(num_threads))
        if rc != 0:
            raise ValueError("oracle_mla_decode_paged rejected its arguments")
        return out, lse

    def decode_multi(self, kv_dtype: int, q, kv, kv_indptr, q_len: int, qo_indptr=None, kv_scale=None,
                     block_scales=None, sm_scale: float = SM_SCALE, num_threads: int = 0):
        """q_len query tokens per sequence: token i of sequence b (query row
        qo_indptr[b] + i) attends causally to the first L_b - (q_len - 1 - i) rows.
        Returns (out [B*q_len,16,512], lse [B*q_len,16]) in (b, i) order."""
        q_a = _u16(q)
        kv_a, sc, bs, stride = self._kv_args(kv_dtype, kv, kv_scale, block_scales)
        ind = np.ascontiguousarray(np.asarray(kv_indptr, dtype=np.int32))
        batch = ind.size - 1
        qo = (np.arange(batch + 1, dtype=np.int32) * int(q_len) if qo_indptr is None
              else np.ascontiguousarray(np.asarray(qo_indptr, dtype=np.int32)))
        out = np.zeros((batch * q_len, NUM_HEADS, V_DIM), dtype=np.float64)
        lse = np.zeros((batch * q_len, NUM_HEADS), dtype=np.float64)
        rc = self.lib.oracle_mla_decode_multi(kv_dtype, _ptr(q_a), _ptr(kv_a), _ptr(bs), stride, sc, _ptr(ind),
                                              _ptr(qo), batch, int(q_len), float(sm_scale), _ptr(out), _ptr(lse),
                                              int(num_threads))
        if rc != 0:
            raise ValueError("oracle_mla_decode_multi rejected its arguments")
        return out, lse

    def partial(self, kv_dtype: int, q, kv, qrow: int, start: int, end: int, kv_scale=None,
                block_scales=None, sm_scale: float = SM_SCALE):
        """Normalised partial over KV rows [start, end): (o [16,512], lse [16])."""
        q_a = _u16(q)
        kv_a, sc, bs, stride = self._kv_args(kv_dtype, kv, kv_scale, block_scales)
        o = np.zeros((NUM_HEADS, V_DIM), dtype=np.float64)
        lse = np.zeros((NUM_HEADS,), dtype=np.float64)
        rc = self.lib.oracle_mla_partial(kv_dtype, _ptr(q_a), _ptr(kv_a), _ptr(bs), stride, sc,
                                         int(qrow), int(start), int(end), float(sm_scale),
                                         _ptr(o), _ptr(lse))
        if rc != 0:
            raise ValueError("oracle_mla_partial rejected its arguments")
        return o, lse

    def combine(self, o: np.ndarray, lse: np.ndarray):
        """LSE combine of partials o [n,16,512], lse [n,16] -> (out [16,512], lse [16])."""
        o = np.ascontiguousarray(o, dtype=np.float64)
        lse = np.ascontiguousarray(lse, dtype=np.float64)
        out = np.zeros((NUM_HEADS, V_DIM), dtype=np.float64)
        lo = np.zeros((NUM_HEADS,), dtype=np.float64)
        rc = self.lib.oracle_mla_combine(int(o.shape[0]), _ptr(o), _ptr(lse), _ptr(out), _ptr(lo))
        if rc != 0:
            raise ValueError("oracle_mla_combine rejected its arguments")
        return out, lo
