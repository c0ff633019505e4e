"""ctypes binding of the gmmfr C ABI (include/gmmfr.h).

Argument marshalling only: every step of the computation runs in the CUDA
library.  The functions named like the C entry points take raw device
addresses (int) or None; :func:`tensor_args` and :func:`run` turn torch
tensors into those.  The library is loaded on first use; if it has not been
built, loading raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libgmmfr.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE = range(6)
E4M3, E5M2 = 0, 1
INDEX_I64, INDEX_I32 = 0, 1
DETERMINISTIC = 1
DEV_BAD_GROUP_LIST, DEV_BAD_ROW_INDEX, DEV_TIMEOUT, DEV_BAD_EXPERT_ID = 1, 2, 4, 8
PROFILE_SLOTS = 5
PROFILE_SLOT_NAMES = ("prep", "route", "gemm", "combine", "call")

# exported entry points, as declared in include/gmmfr.h
ENTRY_POINTS = (
    "gmmfr_prepared_weights_size", "gmmfr_prepare_weights", "gmmfr_workspace_size",
    "gmmfr_grouped_matmul_finalize_routing", "gmmfr_check_device_errors", "gmmfr_last_error",
    "gmmfr_profile_begin", "gmmfr_profile_end", "gmmfr_grouped_matmul_finalize_routing_static_scratch",
    "gmmfr_static_scratch_check_device_errors",
    "gmmfr_moe_route_workspace_size", "gmmfr_moe_route",
    "gmmfr_ffn_prepared_weights_size", "gmmfr_ffn_prepare_weights", "gmmfr_ffn_workspace_size",
    "gmmfr_llada2_moe_grouped_gemm",
)


DT_U8, DT_E4M3, DT_E5M2, DT_E2M1X2, DT_E8M0, DT_I64, DT_I32, DT_F32, DT_BF16 = range(9)
MAX_DIMS = 4


class Tensor(ctypes.Structure):
    """Mirror of gmmfr_tensor: a non-owning view of dense device memory."""
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * MAX_DIMS), ("strides", ctypes.c_int64 * MAX_DIMS)]


def raw_view(data, dtype: int, shape, strides=None) -> Tensor:
    """A view of `data` (an address, or None) with the given dtype code, shape and strides
    (dense row-major when not given)."""
    shape = tuple(int(x) for x in shape)
    if strides is None:
        strides, acc = [], 1
        for d in reversed(shape):
            strides.insert(0, acc)
            acc *= d
    t = Tensor()
    t.data = data
    t.dtype = dtype
    t.ndim = len(shape)
    for i, (d, st) in enumerate(zip(shape, strides)):
        t.shape[i] = d
        t.strides[i] = int(st)
    return t


class Problem(ctypes.Structure):
    """Mirror of gmmfr_problem."""
    _fields_ = [
        ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("N", ctypes.c_int64),
        ("E", ctypes.c_int64), ("batch", ctypes.c_int64),
        ("x1_format", ctypes.c_int32), ("x2_format", ctypes.c_int32),
        ("transpose_x2", ctypes.c_int32), ("scale_per_expert", ctypes.c_int32),
        ("group_list_type", ctypes.c_int32), ("row_index_type", ctypes.c_int32),
        ("shared_rows", ctypes.c_int64), ("shared_offset", ctypes.c_int64),
        ("shared_weight", ctypes.c_float), ("flags", ctypes.c_uint32),
        ("expected_tokens_per_expert", ctypes.c_int64),
    ]


class RouteProblem(ctypes.Structure):
    """Mirror of gmmfr_route_problem."""
    _fields_ = [
        ("batch", ctypes.c_int64), ("topk", ctypes.c_int64), ("K", ctypes.c_int64), ("E", ctypes.c_int64),
        ("ids_type", ctypes.c_int32), ("group_list_type", ctypes.c_int32),
    ]


class FfnProblem(ctypes.Structure):
    """Mirror of gmmfr_ffn_problem."""
    _fields_ = [("N", ctypes.c_int64), ("H", ctypes.c_int64), ("I", ctypes.c_int64), ("E", ctypes.c_int64)]


class GmmfrError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"gmmfr status {status}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it is missing: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"gmmfr CUDA library not built ({path}); run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            P = ctypes.POINTER(Problem)
            vp, sz = ctypes.c_void_p, ctypes.c_size_t
            lib.gmmfr_prepared_weights_size.argtypes = [P, ctypes.POINTER(sz)]
            T = ctypes.POINTER(Tensor)
            lib.gmmfr_prepare_weights.argtypes = [P, T, T, vp, sz, vp]
            lib.gmmfr_workspace_size.argtypes = [P, ctypes.c_int, ctypes.POINTER(sz)]
            lib.gmmfr_grouped_matmul_finalize_routing.argtypes = [P] + [T] * 10 + [vp, sz, vp, sz, vp]
            lib.gmmfr_grouped_matmul_finalize_routing_static_scratch.argtypes = [P] + [T] * 7 + [vp, sz, vp]
            lib.gmmfr_static_scratch_check_device_errors.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
            RP = ctypes.POINTER(RouteProblem)
            lib.gmmfr_moe_route_workspace_size.argtypes = [RP, ctypes.POINTER(sz)]
            lib.gmmfr_moe_route.argtypes = [RP] + [vp] * 11 + [sz, vp]
            FP = ctypes.POINTER(FfnProblem)
            lib.gmmfr_ffn_prepared_weights_size.argtypes = [FP, ctypes.POINTER(sz)]
            lib.gmmfr_ffn_prepare_weights.argtypes = [FP, vp, vp, vp, sz, vp]
            lib.gmmfr_ffn_workspace_size.argtypes = [FP, ctypes.POINTER(sz)]
            lib.gmmfr_llada2_moe_grouped_gemm.argtypes = [FP, vp, vp, vp, vp, vp, sz, vp]
            lib.gmmfr_check_device_errors.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
            lib.gmmfr_last_error.restype = ctypes.c_char_p
            lib.gmmfr_profile_begin.argtypes = [ctypes.c_int]
            lib.gmmfr_profile_end.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_int)]
            for name in ENTRY_POINTS:
                if name != "gmmfr_last_error":
                    getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def gmmfr_last_error() -> str:
    return load().gmmfr_last_error().decode()


def _check(status: int) -> None:
    if status != OK:
        raise GmmfrError(status, gmmfr_last_error())


def make_problem(*, M, K, N, E, batch, x1_format=E4M3, x2_format=E4M3, transpose_x2=False,
                 scale_per_expert=False, group_list_type=1, row_index_type=INDEX_I64, shared_rows=0,
                 shared_offset=0, shared_weight=1.0, deterministic=False,
                 expected_tokens_per_expert=0) -> Problem:
    return Problem(M=M, K=K, N=N, E=E, batch=batch, x1_format=x1_format, x2_format=x2_format,
                   transpose_x2=int(bool(transpose_x2)), scale_per_expert=int(bool(scale_per_expert)),
                   group_list_type=group_list_type, row_index_type=row_index_type,
                   shared_rows=shared_rows, shared_offset=shared_offset, shared_weight=shared_weight,
                   flags=DETERMINISTIC if deterministic else 0,
                   expected_tokens_per_expert=expected_tokens_per_expert)


def problem_from_spec(spec, deterministic: bool = False, row_index_type: int = INDEX_I64) -> Problem:
    """gmmfr_problem for a workloads.Spec."""
    return make_problem(M=spec.M, K=spec.K, N=spec.N, E=spec.E, batch=spec.batch, x1_format=spec.x1_dtype,
                        x2_format=spec.x2_dtype, transpose_x2=spec.transpose_x2,
                        scale_per_expert=spec.scale_per_expert, group_list_type=spec.group_list_type,
                        row_index_type=row_index_type, shared_rows=spec.n_shared,
                        shared_offset=spec.shared_offset, shared_weight=spec.shared_weight,
                        deterministic=deterministic)


def gmmfr_prepared_weights_size(problem: Problem) -> int:
    n = ctypes.c_size_t()
    _check(load().gmmfr_prepared_weights_size(ctypes.byref(problem), ctypes.byref(n)))
    return n.value


def _ref(view: Optional[Tensor]):
    return None if view is None else ctypes.byref(view)


def gmmfr_prepare_weights(problem: Problem, x2: Optional[Tensor], scale: Optional[Tensor], prepared: Optional[int],
                          prepared_bytes: int, stream: Optional[int] = None) -> None:
    _check(load().gmmfr_prepare_weights(ctypes.byref(problem), _ref(x2), _ref(scale), prepared, prepared_bytes,
                                        stream))


def gmmfr_workspace_size(problem: Problem, have_prepared: bool) -> int:
    n = ctypes.c_size_t()
    _check(load().gmmfr_workspace_size(ctypes.byref(problem), int(bool(have_prepared)), ctypes.byref(n)))
    return n.value


def gmmfr_grouped_matmul_finalize_routing(problem: Problem, x1, x2, scale, pertoken_scale, group_list, logit,
                                          row_index, shared_input, bias, out, prepared, prepared_bytes, workspace,
                                          workspace_bytes, stream=None) -> None:
    """Tensor arguments are Tensor views (or None); prepared and workspace are addresses."""
    _check(load().gmmfr_grouped_matmul_finalize_routing(
        ctypes.byref(problem), _ref(x1), _ref(x2), _ref(scale), _ref(pertoken_scale), _ref(group_list), _ref(logit),
        _ref(row_index), _ref(shared_input), _ref(bias), _ref(out), prepared, prepared_bytes, workspace,
        workspace_bytes, stream))


def gmmfr_grouped_matmul_finalize_routing_static_scratch(problem: Problem, x1, pertoken_scale, group_list, logit,
                                                         row_index, shared_input, out, prepared, prepared_bytes,
                                                         stream=None) -> None:
    """The operator with the library's own 16 MiB device scratch instead of a
    caller workspace (for callers that cannot allocate); needs prepared weights."""
    _check(load().gmmfr_grouped_matmul_finalize_routing_static_scratch(
        ctypes.byref(problem), _ref(x1), _ref(pertoken_scale), _ref(group_list), _ref(logit), _ref(row_index),
        _ref(shared_input), _ref(out), prepared, prepared_bytes, stream))


def gmmfr_static_scratch_check_device_errors(stream=None) -> int:
    """Synchronises `stream`; returns the device error bits of the last static-scratch call
    on the current device (0 when clean)."""
    bits = ctypes.c_uint32()
    st = load().gmmfr_static_scratch_check_device_errors(stream, ctypes.byref(bits))
    if st not in (OK, ERR_DEVICE):
        _check(st)
    return bits.value


def gmmfr_moe_route_workspace_size(problem: RouteProblem) -> int:
    n = ctypes.c_size_t()
    _check(load().gmmfr_moe_route_workspace_size(ctypes.byref(problem), ctypes.byref(n)))
    return n.value


def gmmfr_moe_route(problem: RouteProblem, topk_ids, topk_weights, x, x_scale, x1, pertoken_scale, group_list,
                    row_index, logit, perm, workspace, workspace_bytes, stream=None) -> None:
    _check(load().gmmfr_moe_route(ctypes.byref(problem), topk_ids, topk_weights, x, x_scale, x1, pertoken_scale,
                                  group_list, row_index, logit, perm, workspace, workspace_bytes, stream))


def gmmfr_ffn_prepared_weights_size(problem: FfnProblem) -> int:
    n = ctypes.c_size_t()
    _check(load().gmmfr_ffn_prepared_weights_size(ctypes.byref(problem), ctypes.byref(n)))
    return n.value


def gmmfr_ffn_prepare_weights(problem: FfnProblem, w13_flat, w2_flat, prepared, prepared_bytes, stream=None) -> None:
    _check(load().gmmfr_ffn_prepare_weights(ctypes.byref(problem), w13_flat, w2_flat, prepared, prepared_bytes, stream))


def gmmfr_ffn_workspace_size(problem: FfnProblem) -> int:
    n = ctypes.c_size_t()
    _check(load().gmmfr_ffn_workspace_size(ctypes.byref(problem), ctypes.byref(n)))
    return n.value


def gmmfr_llada2_moe_grouped_gemm(problem: FfnProblem, sorted_tokens, prepared, expert_cumsum, result, workspace,
                                  workspace_bytes, stream=None) -> None:
    _check(load().gmmfr_llada2_moe_grouped_gemm(ctypes.byref(problem), sorted_tokens, prepared, expert_cumsum,
                                                result, workspace, workspace_bytes, stream))


def gmmfr_check_device_errors(workspace: int, stream: Optional[int] = None) -> int:
    """Synchronises `stream`; returns the device error bits (0 when clean)."""
    bits = ctypes.c_uint32()
    st = load().gmmfr_check_device_errors(workspace, stream, ctypes.byref(bits))
    if st not in (OK, ERR_DEVICE):
        _check(st)
    return bits.value


def gmmfr_profile_begin(max_calls: int) -> None:
    _check(load().gmmfr_profile_begin(max_calls))


def gmmfr_profile_end(max_calls: int):
    """Per recorded call, the kernel times in ms by slot (-1 when not run)."""
    buf = (ctypes.c_float * (max_calls * PROFILE_SLOTS))()
    n = ctypes.c_int()
    _check(load().gmmfr_profile_end(buf, len(buf), ctypes.byref(n)))
    return [[buf[c * PROFILE_SLOTS + s] for s in range(PROFILE_SLOTS)] for c in range(n.value)]


# ---------------------------------------------------------------------------- torch marshalling
def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("gmmfr takes device tensors")
    if not t.is_contiguous():
        raise ValueError("gmmfr takes contiguous tensors")
    return t.data_ptr()


def _dtype_code(t) -> int:
    import torch
    codes = {torch.uint8: DT_U8, torch.int64: DT_I64, torch.int32: DT_I32, torch.float32: DT_F32,
             torch.bfloat16: DT_BF16, torch.float8_e4m3fn: DT_E4M3, torch.float8_e5m2: DT_E5M2}
    for name, code in (("float8_e8m0fnu", DT_E8M0), ("float4_e2m1fn_x2", DT_E2M1X2)):
        if hasattr(torch, name):
            codes[getattr(torch, name)] = code
    if t.dtype not in codes:
        raise ValueError(f"gmmfr has no element type for {t.dtype}")
    return codes[t.dtype]


def view(t) -> Optional[Tensor]:
    """The gmmfr_tensor view of a device tensor (None for None).  The library checks its
    element type, rank, shape and layout against the problem."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("gmmfr takes device tensors")
    return raw_view(t.data_ptr(), _dtype_code(t), tuple(t.shape), tuple(t.stride()))


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def prepare_weights(problem: Problem, x2, scale, stream=None):
    """Allocate (torch) and fill the prepared-weight buffer for x2/scale."""
    import torch
    n = gmmfr_prepared_weights_size(problem)
    buf = torch.empty(max(n, 16), dtype=torch.uint8, device=x2.device)
    gmmfr_prepare_weights(problem, view(x2), view(scale), _ptr(buf), n, _stream(stream))
    return buf


def workspace(problem: Problem, have_prepared: bool, device) -> "torch.Tensor":
    import torch
    n = gmmfr_workspace_size(problem, have_prepared)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def run(problem: Problem, inputs: dict, out, prepared=None, ws=None, stream=None) -> None:
    """One call of the operator on device tensors (``inputs`` as made by
    workloads.make_inputs); accumulates into ``out`` in place."""
    if ws is None:
        ws = workspace(problem, prepared is not None, out.device)
    gmmfr_grouped_matmul_finalize_routing(
        problem, view(inputs["x1"]), view(inputs["x2"]) if prepared is None else None,
        view(inputs["scale"]) if prepared is None else None, view(inputs["pertoken_scale"]),
        view(inputs["group_list"]), view(inputs.get("logit")), view(inputs["row_index"]),
        view(inputs.get("shared_input")), view(inputs.get("bias")), view(out), _ptr(prepared),
        0 if prepared is None else prepared.numel(), _ptr(ws), ws.numel(), _stream(stream))
    return ws


def run_static_scratch(problem: Problem, inputs: dict, out, prepared, stream=None) -> None:
    """One call of the allocation-free entry point on device tensors."""
    gmmfr_grouped_matmul_finalize_routing_static_scratch(
        problem, view(inputs["x1"]), view(inputs["pertoken_scale"]), view(inputs["group_list"]),
        view(inputs.get("logit")), view(inputs["row_index"]), view(inputs.get("shared_input")), view(out),
        _ptr(prepared), prepared.numel(), _stream(stream))


def route(topk_ids, topk_weights, x, x_scale, E: int, group_list_type: int = 1, stream=None, ws=None):
    """Run the routing step on device tensors; returns (dict of outputs, workspace)."""
    import torch
    batch, topk = topk_ids.shape
    K = x.shape[1]
    rp = RouteProblem(batch=batch, topk=topk, K=K, E=E,
                      ids_type=INDEX_I32 if topk_ids.dtype == torch.int32 else INDEX_I64,
                      group_list_type=group_list_type)
    M = batch * topk
    dev = x.device
    o = dict(x1=torch.empty((M, K), dtype=torch.uint8, device=dev),
             pertoken_scale=torch.empty((M,) + tuple(x_scale.shape[1:]), dtype=torch.uint8, device=dev),
             group_list=torch.empty(E, dtype=torch.int64, device=dev),
             row_index=torch.empty(M, dtype=torch.int64, device=dev),
             logit=torch.empty(M, dtype=torch.float32, device=dev),
             perm=torch.empty(M, dtype=torch.int32, device=dev))
    if ws is None:
        ws = torch.empty(max(gmmfr_moe_route_workspace_size(rp), 256), dtype=torch.uint8, device=dev)
    gmmfr_moe_route(rp, _ptr(topk_ids), _ptr(topk_weights), _ptr(x), _ptr(x_scale), _ptr(o["x1"]),
                    _ptr(o["pertoken_scale"]), _ptr(o["group_list"]), _ptr(o["row_index"]), _ptr(o["logit"]),
                    _ptr(o["perm"]), _ptr(ws), ws.numel(), _stream(stream))
    return o, ws


def ffn_prepare(H: int, I: int, E: int, w13_flat, w2_flat, stream=None):
    """Prepared-weight buffer (torch uint8) for the grouped FFN."""
    import torch
    fp = FfnProblem(N=0, H=H, I=I, E=E)
    n = gmmfr_ffn_prepared_weights_size(fp)
    buf = torch.empty(n, dtype=torch.uint8, device=w13_flat.device)
    gmmfr_ffn_prepare_weights(fp, _ptr(w13_flat), _ptr(w2_flat), _ptr(buf), n, _stream(stream))
    return buf


def ffn(sorted_tokens, prepared, expert_cumsum, H: int, I: int, E: int, result=None, ws=None, stream=None):
    """Run the grouped FFN on device tensors; returns (result, workspace)."""
    import torch
    N = sorted_tokens.shape[0]
    fp = FfnProblem(N=N, H=H, I=I, E=E)
    if result is None:
        result = torch.zeros((N, H), dtype=torch.bfloat16, device=sorted_tokens.device)
    if ws is None:
        ws = torch.empty(gmmfr_ffn_workspace_size(fp), dtype=torch.uint8, device=sorted_tokens.device)
    gmmfr_llada2_moe_grouped_gemm(fp, _ptr(sorted_tokens), _ptr(prepared), _ptr(expert_cumsum), _ptr(result),
                                  _ptr(ws), ws.numel(), _stream(stream))
    return result, ws
