"""GB300 (sm_103a) local W4A16 MoE forward.

The computation (optionally the router's softmax + top-k, route preparation,
expert-grouped gate/up GEMM over packed INT4 weights, SwiGLU / ReLU^2, down
GEMM, FP32 top-k combine) runs entirely in
the hand-written kernels of ``libw4a16_moe.so`` behind the C ABI declared in
``include/w4a16_moe.h``.  This package only marshals torch tensors (device
memory and streams) into that ABI.
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import (Desc, RouteInfo, W4A16Error, w4a16_moe_check_device_error,  # noqa: F401
                   w4a16_moe_forward, w4a16_moe_forward_host, w4a16_moe_plan,
                   w4a16_moe_plan_destroy, w4a16_moe_prepare_routes, w4a16_moe_route_info,
                   w4a16_moe_route_topk, w4a16_moe_set_gemm_path, w4a16_moe_set_overrides,
                   w4a16_moe_forward_masked, w4a16_moe_relayout_weights, w4a16_moe_set_weight_layout,
                   w4a16_moe_set_fused_finalize,
                   w4a16_moe_route_and_prepare)
from ._lib import PATH_AUTO, PATH_CUDA_CORES, PATH_TENSOR_CORES  # noqa: F401
from ._lib import LAYOUT_CHECKPOINT, LAYOUT_INTERLEAVED  # noqa: F401

ACT_SWIGLU, ACT_RELU2 = 0, 1
SCALE_GROUP32_K, SCALE_PER_CHANNEL = 0, 1
DT_BF16, DT_FP16 = 0, 1


def _ptr(t) -> int:
    if t is None:
        return 0
    if not t.is_contiguous():
        raise ValueError("tensors passed to the W4A16 MoE library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def route_topk(logits: torch.Tensor, top_k: int, stream=None):
    """Router softmax + top-k on the GPU (``w4a16_moe_route_topk``).

    logits: [T, G] FP32 CUDA tensor.  Returns (topk_ids int32 [T, k],
    topk_weights fp32 [T, k]): global expert indices by descending probability
    (ties to the lower index) and their softmax probabilities."""
    if logits.dtype != torch.float32 or not logits.is_cuda or logits.dim() != 2:
        raise ValueError("logits must be a 2-D float32 CUDA tensor")
    T, G = logits.shape
    ids = torch.empty(T, top_k, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, top_k, dtype=torch.float32, device=logits.device)
    w4a16_moe_route_topk(_ptr(logits), T, G, top_k, _ptr(ids), _ptr(w), _stream(stream))
    return ids, w


class W4A16MoE:
    """A plan plus its device workspace (owned by this object).

    ``weights`` arguments are any object with ``w13, s13, w2, s2`` tensors in
    the layouts documented in the C header.
    """

    def __init__(self, num_experts, hidden, inter, top_k, max_tokens, act=ACT_SWIGLU,
                 scale_kind=SCALE_GROUP32_K, act_dtype=DT_BF16, expert_offset=0, device="cuda",
                 global_experts=0):
        _lib.load()
        self.desc = Desc(num_experts, expert_offset, hidden, inter, top_k, max_tokens, act,
                         scale_kind, act_dtype, global_experts)
        self.plan, self.workspace_bytes = w4a16_moe_plan(self.desc)
        self.device = torch.device(device)
        self.workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=self.device)
        self.act_dtype = torch.bfloat16 if act_dtype == DT_BF16 else torch.float16

    @classmethod
    def from_config(cls, cfg, max_tokens=None, device="cuda"):
        return cls(cfg.num_experts, cfg.hidden, cfg.inter, cfg.top_k,
                   max_tokens or max(cfg.tokens), act=cfg.act, scale_kind=cfg.scale_kind,
                   act_dtype=cfg.act_dtype, expert_offset=cfg.expert_offset, device=device,
                   global_experts=cfg.global_experts)

    def close(self):
        if self.plan is not None:
            w4a16_moe_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_overrides(self, tile_rows=0, gemm1_splits=0, gemm2_splits=0):
        need = w4a16_moe_set_overrides(self.plan, tile_rows, gemm1_splits, gemm2_splits)
        if need > self.workspace.numel():
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        self.workspace_bytes = need

    def set_gemm_path(self, path=PATH_AUTO):
        """PATH_AUTO, PATH_TENSOR_CORES or PATH_CUDA_CORES for later calls."""
        need = w4a16_moe_set_gemm_path(self.plan, path)
        if need > self.workspace.numel():
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        self.workspace_bytes = need

    def set_fused_finalize(self, enable=True):
        """Combine the routes inside the fused CUDA-core launch (bit-identical
        to the separate combine; only forwards with fused_gemms use it)."""
        w4a16_moe_set_fused_finalize(self.plan, enable)

    def set_weight_layout(self, layout=LAYOUT_CHECKPOINT):
        """Layout of the packed weights later forwards receive."""
        w4a16_moe_set_weight_layout(self.plan, layout)

    def relayout_weights(self, weights, stream=None, in_place=False):
        """Plan-time relayout (``w4a16_moe_relayout_weights``) of both packed
        weight tensors into the interleaved layout, and switch this plan to it.
        Returns an object with the relaid-out ``w13``/``w2`` and the same
        scales (group scales: in place when ``in_place``)."""
        import copy
        out = copy.copy(weights)
        group = self.desc.scale_kind == SCALE_GROUP32_K
        E, H, I = self.desc.num_experts, self.desc.hidden, self.desc.inter
        N1 = 2 * I if self.desc.act == ACT_SWIGLU else I
        for which, name, rows, k in ((0, "w13", N1, H), (1, "w2", H, I)):
            src = getattr(weights, name)
            dst = src if (in_place and group) else torch.empty(E, rows, k // 2, dtype=torch.uint8,
                                                              device=src.device)
            w4a16_moe_relayout_weights(self.plan, which, _ptr(src), _ptr(dst), _stream(stream))
            setattr(out, name, dst)
        self.set_weight_layout(LAYOUT_INTERLEAVED)
        return out

    def route_info(self, num_tokens: int) -> RouteInfo:
        return w4a16_moe_route_info(self.plan, num_tokens)

    def route_and_prepare(self, logits, stream=None):
        """Router softmax + top-k and the route layout in one pass
        (``w4a16_moe_route_and_prepare``).  logits [T, G] FP32 CUDA tensor;
        returns (topk_ids int32 [T, k], topk_weights fp32 [T, k]) for the
        following ``forward``."""
        if logits.dtype != torch.float32 or not logits.is_cuda or logits.dim() != 2:
            raise ValueError("logits must be a 2-D float32 CUDA tensor")
        T, G = logits.shape
        k = self.desc.top_k
        ids = torch.empty(T, k, dtype=torch.int32, device=logits.device)
        w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
        w4a16_moe_route_and_prepare(self.plan, T, _ptr(logits), G, _ptr(ids), _ptr(w), _ptr(self.workspace),
                                    _stream(stream))
        return ids, w

    def prepare_routes(self, topk_ids, stream=None):
        w4a16_moe_prepare_routes(self.plan, topk_ids.shape[0], _ptr(topk_ids),
                                 _ptr(self.workspace), _stream(stream))

    def forward(self, x, weights, topk_weights, topk_ids, renormalize=False, out=None, stream=None):
        T = x.shape[0]
        if out is None:
            out = torch.empty(T, self.desc.hidden, dtype=self.act_dtype, device=x.device)
        w4a16_moe_forward(self.plan, T, _ptr(x), _ptr(weights.w13), _ptr(weights.s13),
                          _ptr(weights.w2), _ptr(weights.s2), _ptr(topk_weights), _ptr(topk_ids),
                          renormalize, _ptr(out), _ptr(self.workspace), _stream(stream))
        return out

    def forward_masked(self, x, weights, counts, out=None, stream=None):
        """Expert MLPs on the masked-count layout (``w4a16_moe_forward_masked``):
        x [E, max_rows, H], counts int32 [E] on the device; needs a plan built
        with top_k == 1 and max_tokens >= E * max_rows."""
        if x.dim() != 3 or x.shape[0] != self.desc.num_experts:
            raise ValueError("x must be [num_experts, max_rows, hidden]")
        if out is None:
            out = torch.empty_like(x)
        w4a16_moe_forward_masked(self.plan, x.shape[1], _ptr(counts), _ptr(x), _ptr(weights.w13),
                                 _ptr(weights.s13), _ptr(weights.w2), _ptr(weights.s2), _ptr(out),
                                 _ptr(self.workspace), _stream(stream))
        return out

    def __call__(self, x, weights, topk_weights, topk_ids, renormalize=False, out=None, stream=None):
        self.prepare_routes(topk_ids, stream)
        return self.forward(x, weights, topk_weights, topk_ids, renormalize, out, stream)

    def forward_host(self, x_host, weights, topk_weights_host, topk_ids_host, renormalize=False,
                     out_host=None, stream=None):
        """End-to-end call with host (ideally pinned) activations, ids, weights and output."""
        T = x_host.shape[0]
        if out_host is None:
            out_host = torch.empty(T, self.desc.hidden, dtype=self.act_dtype, pin_memory=True)
        w4a16_moe_forward_host(self.plan, T, _ptr(x_host), _ptr(weights.w13), _ptr(weights.s13),
                               _ptr(weights.w2), _ptr(weights.s2), _ptr(topk_weights_host),
                               _ptr(topk_ids_host), renormalize, _ptr(out_host),
                               _ptr(self.workspace), _stream(stream))
        return out_host

    def check_device_error(self, stream=None):
        w4a16_moe_check_device_error(self.plan, _ptr(self.workspace), _stream(stream))

    def read_route_layout(self, num_tokens: int):
        """Copy the route layout of the last prepare_routes back (tests)."""
        info = self.route_info(num_tokens)
        ws = self.workspace
        E = self.desc.num_experts

        def i32(off, n):
            return ws[off: off + 4 * n].view(torch.int32).cpu()

        offs = i32(info.off_offs, E + 1)
        nt = int(i32(info.off_num_tiles, 1)[0])
        return dict(tile_rows=info.tile_rows,
                    counts=i32(info.off_counts, E),
                    offs=offs,
                    perm=i32(info.off_perm, int(offs[E])),
                    inv=i32(info.off_inv, num_tokens * self.desc.top_k),
                    tiles=i32(info.off_tiles, 4 * nt).view(nt, 4),
                    num_tiles=nt)
