"""ctypes binding of ``libw4a16_moe.so`` (the C ABI in include/w4a16_moe.h).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  Tensors are passed as raw pointers; streams as the raw
cudaStream_t handle of a ``torch.cuda.Stream``.  If the library has not been
built, loading fails loudly -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libw4a16_moe.so")

W4A16_OK = 0
PATH_AUTO, PATH_TENSOR_CORES, PATH_CUDA_CORES = 0, 1, 2
LAYOUT_CHECKPOINT, LAYOUT_INTERLEAVED = 0, 1
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE_TOO_SMALL",
                4: "CUDA", 5: "DEVICE_TIMEOUT"}

# Every entry point include/w4a16_moe.h declares.
EXPORTED = (
    "w4a16_moe_plan",
    "w4a16_moe_plan_destroy",
    "w4a16_moe_prepare_routes",
    "w4a16_moe_forward",
    "w4a16_moe_forward_host",
    "w4a16_moe_route_info",
    "w4a16_moe_set_overrides",
    "w4a16_moe_set_gemm_path",
    "w4a16_moe_check_device_error",
    "w4a16_moe_set_stage_events",
    "w4a16_moe_forward_static_workspace",
    "w4a16_moe_last_error",
    "w4a16_moe_route_topk",
    "w4a16_moe_forward_masked",
    "w4a16_moe_relayout_weights",
    "w4a16_moe_set_weight_layout",
    "w4a16_moe_set_fused_finalize",
    "w4a16_moe_route_and_prepare",
)


class W4A16Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_experts", "expert_offset", "hidden", "inter", "top_k", "max_tokens",
        "act", "scale_kind", "act_dtype", "global_experts")]


class RouteInfo(ctypes.Structure):
    _fields_ = [
        ("tile_rows", ctypes.c_int32), ("max_slots", ctypes.c_int32),
        ("max_tiles", ctypes.c_int32), ("gemm1_splits", ctypes.c_int32),
        ("gemm2_splits", ctypes.c_int32), ("gemm1_ctas", ctypes.c_int32),
        ("gemm2_ctas", ctypes.c_int32), ("pipeline_stages", ctypes.c_int32),
        ("gemm_path", ctypes.c_int32),
        ("off_counts", ctypes.c_size_t), ("off_offs", ctypes.c_size_t),
        ("off_perm", ctypes.c_size_t), ("off_inv", ctypes.c_size_t),
        ("off_tiles", ctypes.c_size_t), ("off_num_tiles", ctypes.c_size_t),
        ("off_inter", ctypes.c_size_t), ("off_expert_out", ctypes.c_size_t),
        ("fused_gemms", ctypes.c_int32), ("fused_finalize", ctypes.c_int32),
    ]


_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library (build it first with ``build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: the CUDA extension has not been built "
            "(run weight_only_int4_histogram_gb300.build.build()); there is no CPU fallback")
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32 = ctypes.c_int32
    st = ctypes.c_int
    L.w4a16_moe_plan.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(P), ctypes.POINTER(ctypes.c_size_t)]
    L.w4a16_moe_plan.restype = st
    L.w4a16_moe_plan_destroy.argtypes = [P]
    L.w4a16_moe_plan_destroy.restype = st
    L.w4a16_moe_prepare_routes.argtypes = [P, i32, P, P, P]
    L.w4a16_moe_prepare_routes.restype = st
    L.w4a16_moe_forward.argtypes = [P, i32, P, P, P, P, P, P, P, i32, P, P, P]
    L.w4a16_moe_forward.restype = st
    L.w4a16_moe_forward_host.argtypes = [P, i32, P, P, P, P, P, P, P, i32, P, P, P]
    L.w4a16_moe_forward_host.restype = st
    L.w4a16_moe_route_info.argtypes = [P, i32, ctypes.POINTER(RouteInfo)]
    L.w4a16_moe_route_info.restype = st
    L.w4a16_moe_set_overrides.argtypes = [P, i32, i32, i32, ctypes.POINTER(ctypes.c_size_t)]
    L.w4a16_moe_set_overrides.restype = st
    L.w4a16_moe_set_gemm_path.argtypes = [P, i32, ctypes.POINTER(ctypes.c_size_t)]
    L.w4a16_moe_set_gemm_path.restype = st
    L.w4a16_moe_check_device_error.argtypes = [P, P, P]
    L.w4a16_moe_check_device_error.restype = st
    L.w4a16_moe_set_stage_events.argtypes = [P, ctypes.POINTER(P), i32]
    L.w4a16_moe_set_stage_events.restype = st
    L.w4a16_moe_forward_static_workspace.argtypes = [P, i32, P, P, P, P, P, P, P, i32, P, P]
    L.w4a16_moe_forward_static_workspace.restype = st
    L.w4a16_moe_route_topk.argtypes = [P, i32, i32, i32, P, P, P]
    L.w4a16_moe_forward_masked.argtypes = [P, i32, P, P, P, P, P, P, P, P, P]
    L.w4a16_moe_forward_masked.restype = ctypes.c_int
    L.w4a16_moe_route_topk.restype = ctypes.c_int
    L.w4a16_moe_relayout_weights.argtypes = [P, i32, P, P, P]
    L.w4a16_moe_relayout_weights.restype = st
    L.w4a16_moe_route_and_prepare.argtypes = [P, i32, P, i32, P, P, P, P]
    L.w4a16_moe_route_and_prepare.restype = st
    L.w4a16_moe_set_weight_layout.argtypes = [P, i32]
    L.w4a16_moe_set_weight_layout.restype = st
    L.w4a16_moe_set_fused_finalize.argtypes = [P, i32]
    L.w4a16_moe_set_fused_finalize.restype = st
    L.w4a16_moe_last_error.argtypes = []
    L.w4a16_moe_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def check(status: int):
    if status != W4A16_OK:
        raise W4A16Error(status, load().w4a16_moe_last_error().decode())


def w4a16_moe_plan(desc: Desc):
    plan = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    check(load().w4a16_moe_plan(ctypes.byref(desc), ctypes.byref(plan), ctypes.byref(ws)))
    return plan, int(ws.value)


def w4a16_moe_plan_destroy(plan):
    check(load().w4a16_moe_plan_destroy(plan))


def w4a16_moe_prepare_routes(plan, num_tokens: int, topk_ids_ptr: int, workspace_ptr: int, stream: int):
    check(load().w4a16_moe_prepare_routes(plan, num_tokens, topk_ids_ptr, workspace_ptr, stream))


def w4a16_moe_forward(plan, num_tokens, x, w13, s13, w2, s2, topk_weights, topk_ids, renormalize,
                      out, workspace, stream):
    check(load().w4a16_moe_forward(plan, num_tokens, x, w13, s13, w2, s2, topk_weights, topk_ids,
                                   int(renormalize), out, workspace, stream))


def w4a16_moe_forward_host(plan, num_tokens, x_host, w13, s13, w2, s2, topk_weights_host,
                           topk_ids_host, renormalize, out_host, workspace, stream):
    check(load().w4a16_moe_forward_host(plan, num_tokens, x_host, w13, s13, w2, s2,
                                        topk_weights_host, topk_ids_host, int(renormalize),
                                        out_host, workspace, stream))


def w4a16_moe_route_info(plan, num_tokens: int) -> RouteInfo:
    info = RouteInfo()
    check(load().w4a16_moe_route_info(plan, num_tokens, ctypes.byref(info)))
    return info


def w4a16_moe_set_overrides(plan, tile_rows: int = 0, gemm1_splits: int = 0, gemm2_splits: int = 0) -> int:
    ws = ctypes.c_size_t()
    check(load().w4a16_moe_set_overrides(plan, tile_rows, gemm1_splits, gemm2_splits, ctypes.byref(ws)))
    return int(ws.value)


def w4a16_moe_set_gemm_path(plan, path: int) -> int:
    ws = ctypes.c_size_t()
    check(load().w4a16_moe_set_gemm_path(plan, path, ctypes.byref(ws)))
    return int(ws.value)


def w4a16_moe_check_device_error(plan, workspace_ptr: int, stream: int):
    check(load().w4a16_moe_check_device_error(plan, workspace_ptr, stream))


def w4a16_moe_forward_masked(plan, max_rows: int, counts_ptr: int, x_ptr: int, w13: int, s13: int, w2: int,
                             s2: int, y_ptr: int, workspace_ptr: int, stream: int):
    check(load().w4a16_moe_forward_masked(plan, max_rows, counts_ptr, x_ptr, w13, s13, w2, s2, y_ptr,
                                          workspace_ptr, stream))


def w4a16_moe_route_topk(logits_ptr: int, num_tokens: int, num_global: int, top_k: int, ids_ptr: int,
                         weights_ptr: int, stream: int):
    check(load().w4a16_moe_route_topk(logits_ptr, num_tokens, num_global, top_k, ids_ptr, weights_ptr, stream))


def w4a16_moe_relayout_weights(plan, which: int, in_ptr: int, out_ptr: int, stream: int):
    check(load().w4a16_moe_relayout_weights(plan, which, in_ptr, out_ptr, stream))


def w4a16_moe_route_and_prepare(plan, num_tokens: int, logits_ptr: int, num_global: int, ids_ptr: int,
                                weights_ptr: int, workspace_ptr: int, stream: int):
    check(load().w4a16_moe_route_and_prepare(plan, num_tokens, logits_ptr, num_global, ids_ptr, weights_ptr,
                                             workspace_ptr, stream))


def w4a16_moe_set_weight_layout(plan, layout: int):
    check(load().w4a16_moe_set_weight_layout(plan, layout))


def w4a16_moe_set_fused_finalize(plan, enable: bool):
    check(load().w4a16_moe_set_fused_finalize(plan, 1 if enable else 0))


def w4a16_moe_set_stage_events(plan, event_handles):
    """event_handles: list of 4 cudaEvent_t handles (ints), or [] to turn off."""
    n = len(event_handles)
    arr = (ctypes.c_void_p * max(n, 1))(*event_handles)
    check(load().w4a16_moe_set_stage_events(plan, arr if n else None, n))


STATIC_WORKSPACE_BYTES = 32 * 1024 * 1024


def w4a16_moe_forward_static_workspace(plan, num_tokens, x, w13, s13, w2, s2, topk_weights, topk_ids,
                                       renormalize, out, stream):
    """prepare_routes + forward on the library's fixed device workspace (no allocation)."""
    check(load().w4a16_moe_forward_static_workspace(plan, num_tokens, x, w13, s13, w2, s2, topk_weights,
                                                    topk_ids, int(renormalize), out, stream))
