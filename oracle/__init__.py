"""CPU oracle for MXFP8 grouped-matmul-finalize-routing (FP64, plain C).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may use it; the product path never does.  It
shares no code with the CUDA library.  The arithmetic lives in
``gmmfr_oracle.c``; this module only compiles it and marshals arguments.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgmmfr_oracle.so")
_lock = threading.Lock()
_lib = None

BAD_GROUP_LIST = 1
BAD_ROW_INDEX = 2


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FMA contraction, no -march)."""
    src = os.path.join(_HERE, "gmmfr_oracle.c")
    hdr = os.path.join(_HERE, "gmmfr_oracle.h")
    os.makedirs(_BUILD, exist_ok=True)
    newest = max(os.path.getmtime(src), os.path.getmtime(hdr))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Args(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("N", ctypes.c_int64),
        ("E", ctypes.c_int64), ("batch", ctypes.c_int64),
        ("x1_fmt", ctypes.c_int32), ("x2_fmt", ctypes.c_int32),
        ("transpose_x2", ctypes.c_int32), ("scale_per_expert", ctypes.c_int32),
        ("group_list_type", ctypes.c_int32), ("_pad", ctypes.c_int32),
        ("x1", ctypes.c_void_p), ("x2", ctypes.c_void_p), ("scale", ctypes.c_void_p),
        ("pertoken_scale", ctypes.c_void_p), ("group_list", ctypes.c_void_p),
        ("logit", ctypes.c_void_p), ("row_index", ctypes.c_void_p),
        ("shared_input", ctypes.c_void_p), ("shared_rows", ctypes.c_int64),
        ("shared_offset", ctypes.c_int64), ("shared_weight", ctypes.c_double),
        ("out_init", ctypes.c_void_p), ("bias", ctypes.c_void_p),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # GMMFR_ORACLE_LIB: another build of gmmfr_oracle.c (the mutation test plants
            # mistakes in copies of it and checks that the pins catch each)
            lib = ctypes.CDLL(os.environ.get("GMMFR_ORACLE_LIB") or build())
            P = ctypes.POINTER(_Args)
            lib.oracle_decode_fp8.restype = ctypes.c_double
            lib.oracle_decode_fp8.argtypes = [ctypes.c_int, ctypes.c_uint32]
            lib.oracle_decode_e8m0.restype = ctypes.c_double
            lib.oracle_decode_e8m0.argtypes = [ctypes.c_uint32]
            lib.oracle_decode_bf16.restype = ctypes.c_double
            lib.oracle_decode_bf16.argtypes = [ctypes.c_uint32]
            lib.oracle_expert_ranges.restype = ctypes.c_int
            lib.oracle_expert_ranges.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_gmmfr.restype = ctypes.c_int
            lib.oracle_gmmfr.argtypes = [P, ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_gmmfr_sampled.restype = ctypes.c_int
            lib.oracle_gmmfr_sampled.argtypes = [P, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_void_p, ctypes.c_void_p]
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _np(x, dtype) -> Optional[np.ndarray]:
    """Contiguous host numpy array of ``dtype`` from a torch tensor or array, or None.
    bfloat16 tensors are passed as their raw 16-bit patterns."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        t = x.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        x = t.numpy()
    a = np.ascontiguousarray(x)
    if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" and np.dtype(dtype).kind in "iu":
        return a.view(dtype)
    return np.ascontiguousarray(a.astype(dtype))


class Problem:
    """Host copies of one call's inputs, held alive for the C call."""

    def __init__(self, *, M, K, N, E, batch, x1, x2, scale, pertoken_scale, group_list,
                 row_index, out, x1_dtype=0, x2_dtype=0, transpose_x2=False,
                 scale_per_expert=False, group_list_type=1, logit=None, shared_input=None,
                 shared_offset=0, shared_weight=1.0, bias=None):
        self.keep = dict(
            x1=_np(x1, np.uint8), x2=_np(x2, np.uint8), scale=_np(scale, np.uint8),
            pts=_np(pertoken_scale, np.uint8), gl=_np(group_list, np.int64),
            logit=_np(logit, np.float32), rows=_np(row_index, np.int64),
            shared=_np(shared_input, np.uint16), out=_np(out, np.float32), bias=_np(bias, np.uint16))
        k = self.keep
        p1 = 2 if int(x1_dtype) == 2 else 1
        p2 = 2 if int(x2_dtype) == 2 else 1
        assert k["x1"].size == M * K // p1 and k["x2"].size == E * K * N // p2
        assert k["out"].size == batch * N and k["rows"].size == M and k["gl"].size == E
        shared_rows = 0 if k["shared"] is None else k["shared"].size // max(N, 1)

        def ptr(a):
            return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

        self.args = _Args(
            M=M, K=K, N=N, E=E, batch=batch, x1_fmt=int(x1_dtype), x2_fmt=int(x2_dtype),
            transpose_x2=int(bool(transpose_x2)), scale_per_expert=int(bool(scale_per_expert)),
            group_list_type=int(group_list_type), _pad=0,
            x1=ptr(k["x1"]), x2=ptr(k["x2"]), scale=ptr(k["scale"]), pertoken_scale=ptr(k["pts"]),
            group_list=ptr(k["gl"]), logit=ptr(k["logit"]), row_index=ptr(k["rows"]),
            shared_input=ptr(k["shared"]), shared_rows=shared_rows, shared_offset=int(shared_offset),
            shared_weight=float(shared_weight), out_init=ptr(k["out"]), bias=ptr(k["bias"]))
        self.batch, self.N, self.E = batch, N, E


def problem_from_spec(spec, inputs) -> Problem:
    """Problem from a workloads.Spec and its input dict."""
    return Problem(M=spec.M, K=spec.K, N=spec.N, E=spec.E, batch=spec.batch,
                   x1=inputs["x1"], x2=inputs["x2"], scale=inputs["scale"],
                   pertoken_scale=inputs["pertoken_scale"], group_list=inputs["group_list"],
                   row_index=inputs["row_index"], out=inputs["out"], x1_dtype=spec.x1_dtype,
                   x2_dtype=spec.x2_dtype, transpose_x2=spec.transpose_x2,
                   scale_per_expert=spec.scale_per_expert, group_list_type=spec.group_list_type,
                   logit=inputs["logit"], shared_input=inputs["shared_input"],
                   shared_offset=spec.shared_offset, shared_weight=spec.shared_weight,
                   bias=inputs.get("bias"))


def run(p: Problem) -> Tuple[np.ndarray, np.ndarray, int]:
    """Full oracle: (out64 [batch,N], absb [batch,N], error flags)."""
    lib = _load()
    out = np.zeros((p.batch, p.N), dtype=np.float64)
    absb = np.zeros((p.batch, p.N), dtype=np.float64)
    flags = lib.oracle_gmmfr(ctypes.byref(p.args), out.ctypes.data_as(ctypes.c_void_p),
                             absb.ctypes.data_as(ctypes.c_void_p))
    return out, absb, int(flags)


def run_sampled(p: Problem, rows, cols) -> Tuple[np.ndarray, np.ndarray, int]:
    """Oracle on selected output elements (rows[i], cols[i])."""
    lib = _load()
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    cols = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    vals = np.zeros(rows.size, dtype=np.float64)
    bnd = np.zeros(rows.size, dtype=np.float64)
    flags = lib.oracle_gmmfr_sampled(ctypes.byref(p.args), rows.size, rows.ctypes.data_as(ctypes.c_void_p),
                                     cols.ctypes.data_as(ctypes.c_void_p), vals.ctypes.data_as(ctypes.c_void_p),
                                     bnd.ctypes.data_as(ctypes.c_void_p))
    return vals, bnd, int(flags)


def expert_ranges(p: Problem) -> Tuple[np.ndarray, np.ndarray, int]:
    lib = _load()
    s = np.zeros(max(p.E, 1), dtype=np.int64)
    e = np.zeros(max(p.E, 1), dtype=np.int64)
    f = lib.oracle_expert_ranges(ctypes.byref(p.args), s.ctypes.data_as(ctypes.c_void_p),
                                 e.ctypes.data_as(ctypes.c_void_p))
    return s[:p.E], e[:p.E], int(f)


def decode_fp8(fmt: int, code: int) -> float:
    return _load().oracle_decode_fp8(fmt, code)


def decode_e8m0(code: int) -> float:
    return _load().oracle_decode_e8m0(code)


def decode_bf16(bits: int) -> float:
    return _load().oracle_decode_bf16(bits)


def num_threads() -> int:
    return _load().oracle_num_threads()


def tolerance(out64: np.ndarray, absb: np.ndarray) -> np.ndarray:
    """Per-element parity bound |gpu - oracle| <= 1e-4 * absb + 1e-6, where absb sums
    |logit| * sum_k |a_k b_k| over the element's tokens: for an element with one token this
    is the operator's stated accuracy bound 1e-4 * |logit| * sum_k |a_k b_k| + 1e-6, and
    over several tokens each one's share of it.  The 1e-6 absolute term also covers the
    FP32 rounding of the initial value and the shared term (about 2^-24 of |out|), which
    keeps below it for |out| up to about 8."""
    return 1e-4 * absb + 1e-6
