"""Seeded synthetic inputs for the local W4A16 MoE forward.

This module only *makes inputs*: activations, INT4 expert weights with their
BF16 scales, and top-k routes.  It holds none of the forward's arithmetic
(no unpacking, no dequantisation, no GEMM, activation or combine); both the
CPU oracle and the CUDA path receive exactly the tensors built here.

Recipes (restated from the pages' workload descriptions):

* "feat(pytorch): add CuTeDSL W4A16 MoE backend" (LMDeploy), section
  *Benchmark*: Kimi TP8 shard, 384 experts, hidden 7168, intermediate 256,
  top-k 8, INT4 group size 32, BF16 activations/scales, FP32 routing weights,
  INT32 ids, seed 20260908, renormalize=False.
* "perf: reduce split W4A16 routing and output overhead" (FlashInfer),
  sections *Validation* and *Final performance*: DeepSeek-like H7168/I2048,
  256 global experts of which 32 are local (simulated EP8), top-k 8, SwiGLU;
  widths 256 -> 384 -> 256 for the small functional case.
* "[None][feat] Add W4A16 per-channel weight-only support for Cutlass fused
  MoE" (TensorRT-LLM), sections *Checkpoint format* and *Validation*:
  symmetric per-output-channel INT4, scale = absmax / 7, packed two per byte
  along the output dim with the even index in the low nibble; up to 60
  experts at hidden 2048; a non-gated (Relu2) arm.

The quantiser below is the checkpoint-preparation rule of the TensorRT-LLM
page (*Checkpoint format*), applied per 32-group along K for the group mode.
Rounding of ``w / s`` is round-half-to-even (the pages do not name a mode).

All tensors are produced with ``torch`` generators so they can be made on the
CPU (small cases, oracle tests) or directly on a CUDA device (full sizes).  A
given (config, seed, device) always yields the same bytes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

ACT_SWIGLU = 0
ACT_RELU2 = 1
SCALE_GROUP32 = 0
SCALE_PER_CHANNEL = 1
DT_BF16 = 0
DT_FP16 = 1
GROUP = 32


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    num_experts: int          # E: experts held locally
    hidden: int               # H
    inter: int                # I
    top_k: int
    act: int = ACT_SWIGLU
    scale_kind: int = SCALE_GROUP32
    act_dtype: int = DT_BF16
    global_experts: int = 0   # ids are drawn over this many experts (0 -> E)
    expert_offset: int = 0    # global id of local expert 0
    tokens: tuple = (16,)
    seed: int = 20260908
    logits: str = "normal"    # "normal" N(0,1) or "uniform" U(0,1)
    hot_experts: tuple = ()   # experts given a logit bias
    hot_bias: float = 0.0
    forced_invalid: tuple = ()  # (token, slot) routes forced to -1
    weight_std: float = 0.02

    @property
    def n1(self) -> int:
        return 2 * self.inter if self.act == ACT_SWIGLU else self.inter

    @property
    def n_global(self) -> int:
        return self.global_experts or self.num_experts

    def torch_act_dtype(self):
        return torch.bfloat16 if self.act_dtype == DT_BF16 else torch.float16

    def with_(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


# The five workloads.  Names describe the shape, not where it was quoted.
TINY = MoEConfig("tiny_e8_h256_i384_k2", 8, 256, 384, 2, tokens=(16,), seed=0,
                 forced_invalid=((0, 1), (5, 0)))
KIMI = MoEConfig("kimi_tp8_e384_h7168_i256_k8", 384, 7168, 256, 8,
                 tokens=(1, 8, 32, 256, 1024, 2048), seed=20260908)
DEEPSEEK_LOCAL = MoEConfig("deepseek_local_e32of256_h7168_i2048_k8", 32, 7168, 2048, 8,
                           global_experts=256, expert_offset=0,
                           tokens=(1, 2, 4, 64, 512, 2048), seed=20260908,
                           logits="uniform")
PER_CHANNEL = MoEConfig("per_channel_e60_h2048_i1408_k4", 60, 2048, 1408, 4,
                        scale_kind=SCALE_PER_CHANNEL, tokens=(1, 8, 128, 1024),
                        seed=20260908)
PER_CHANNEL_FP16 = PER_CHANNEL.with_(name="per_channel_fp16_e60_h2048_i1408_k4",
                                     act_dtype=DT_FP16)
RELU2_SKEW = MoEConfig("relu2_skew_e64_h2688_i1856_k6", 64, 2688, 1856, 6,
                       act=ACT_RELU2, scale_kind=SCALE_PER_CHANNEL,
                       tokens=(32, 4096), seed=20260908,
                       hot_experts=(0, 1, 2, 3), hot_bias=3.0)

CONFIGS = {c.name: c for c in (TINY, KIMI, DEEPSEEK_LOCAL, PER_CHANNEL,
                               PER_CHANNEL_FP16, RELU2_SKEW)}


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    # Distinct, reproducible streams per tensor family.
    g.manual_seed((int(seed) * 1000003 + stream * 7919) % (2 ** 63))
    return g


# ----------------------------------------------------------------------------
# Quantiser and packers (checkpoint preparation, not the forward)
# ----------------------------------------------------------------------------

def quantize_symmetric(w: torch.Tensor, group: Optional[int]):
    """Symmetric INT4 quantisation, scale = absmax / 7 stored as BF16.

    ``group=None``: one scale per output row (per-channel).  ``group=32``: one
    scale per 32 consecutive K elements of a row.  The code is
    ``clamp(round_half_even(w / s), -8, 7)`` with ``s`` the BF16-rounded scale
    read back as FP32, and 0 where the scale is 0.
    Returns (q int8 [N, K], s bf16 [N] or [N, K/group]).
    """
    w = w.float()
    n, k = w.shape
    if group is None:
        amax = w.abs().amax(dim=1, keepdim=True)              # [N, 1]
    else:
        assert k % group == 0
        amax = w.view(n, k // group, group).abs().amax(dim=2)  # [N, K/g]
    s = (amax / 7.0).to(torch.bfloat16)
    s32 = s.float()
    if group is None:
        s_full = s32.expand(n, k)
    else:
        s_full = s32.repeat_interleave(group, dim=1)
    safe = torch.where(s_full == 0, torch.ones_like(s_full), s_full)
    q = torch.round(w / safe)
    q = torch.where(s_full == 0, torch.zeros_like(q), q)
    q = q.clamp(-8, 7).to(torch.int8)
    if group is None:
        s = s.view(n)
    return q, s


def pack_int4_along_k(q: torch.Tensor) -> torch.Tensor:
    """[N, K] int8 codes -> [N, K/2] bytes; byte b holds K index 2b in the low
    nibble and 2b+1 in the high nibble (two's complement nibbles)."""
    n, k = q.shape
    assert k % 2 == 0
    lo = q[:, 0::2].to(torch.int32) & 0xF
    hi = q[:, 1::2].to(torch.int32) & 0xF
    return (lo | (hi << 4)).to(torch.uint8)


def pack_int4_along_rows(q: torch.Tensor) -> torch.Tensor:
    """[N, K] int8 codes -> [N/2, K] bytes; byte [p, k] holds row 2p in the low
    nibble and row 2p+1 in the high nibble (the per-channel checkpoint rule:
    packed along dim 0, the output dim, even index low)."""
    n, k = q.shape
    assert n % 2 == 0
    lo = q[0::2, :].to(torch.int32) & 0xF
    hi = q[1::2, :].to(torch.int32) & 0xF
    return (lo | (hi << 4)).to(torch.uint8)


def _quant_pack(w: torch.Tensor, scale_kind: int):
    if scale_kind == SCALE_GROUP32:
        q, s = quantize_symmetric(w, GROUP)
        return pack_int4_along_k(q), s
    q, s = quantize_symmetric(w, None)
    return pack_int4_along_rows(q), s


# ----------------------------------------------------------------------------
# Inputs
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class ExpertWeights:
    w13: torch.Tensor   # uint8, group: [E, N1, H/2]; per-channel: [E, N1/2, H]
    s13: torch.Tensor   # bf16,  group: [E, N1, H/32]; per-channel: [E, N1]
    w2: torch.Tensor    # uint8, group: [E, H, I/2];  per-channel: [E, H/2, I]
    s2: torch.Tensor    # bf16,  group: [E, H, I/32]; per-channel: [E, H]

    def to(self, device) -> "ExpertWeights":
        return ExpertWeights(*(t.to(device) for t in (self.w13, self.s13, self.w2, self.s2)))

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.w13, self.s13, self.w2, self.s2))


def weight_shapes(cfg: MoEConfig):
    E, H, I, N1 = cfg.num_experts, cfg.hidden, cfg.inter, cfg.n1
    if cfg.scale_kind == SCALE_GROUP32:
        return dict(w13=(E, N1, H // 2), s13=(E, N1, H // GROUP),
                    w2=(E, H, I // 2), s2=(E, H, I // GROUP))
    return dict(w13=(E, N1 // 2, H), s13=(E, N1), w2=(E, H // 2, I), s2=(E, H))


def make_weights(cfg: MoEConfig, device="cpu", seed: Optional[int] = None) -> ExpertWeights:
    """Weights ~ N(0, weight_std) in FP32, quantised and packed one expert at a
    time (bounded host/device memory)."""
    seed = cfg.seed if seed is None else seed
    shp = weight_shapes(cfg)
    w13 = torch.empty(shp["w13"], dtype=torch.uint8, device=device)
    s13 = torch.empty(shp["s13"], dtype=torch.bfloat16, device=device)
    w2 = torch.empty(shp["w2"], dtype=torch.uint8, device=device)
    s2 = torch.empty(shp["s2"], dtype=torch.bfloat16, device=device)
    g1 = _gen(seed, 1, device)
    g2 = _gen(seed, 2, device)
    for e in range(cfg.num_experts):
        a = torch.randn(cfg.n1, cfg.hidden, generator=g1, device=device) * cfg.weight_std
        p, s = _quant_pack(a, cfg.scale_kind)
        w13[e].copy_(p)
        s13[e].copy_(s)
        b = torch.randn(cfg.hidden, cfg.inter, generator=g2, device=device) * cfg.weight_std
        p, s = _quant_pack(b, cfg.scale_kind)
        w2[e].copy_(p)
        s2[e].copy_(s)
    return ExpertWeights(w13, s13, w2, s2)


def make_activations(cfg: MoEConfig, tokens: int, device="cpu", seed: Optional[int] = None):
    """x ~ N(0, 1) in the activation dtype, [T, H]."""
    seed = cfg.seed if seed is None else seed
    g = _gen(seed, 3 + 17 * tokens, device)
    x = torch.randn(tokens, cfg.hidden, generator=g, device=device)
    return x.to(cfg.torch_act_dtype())


def make_logits(cfg: MoEConfig, tokens: int, device="cpu", seed: Optional[int] = None):
    """Router logits [T, n_global] FP32 of the workload (the draws make_routes uses)."""
    seed = cfg.seed if seed is None else seed
    g = _gen(seed, 4 + 31 * tokens, device)
    ng = cfg.n_global
    if cfg.logits == "uniform":
        logits = torch.rand(tokens, ng, generator=g, device=device)
    else:
        logits = torch.randn(tokens, ng, generator=g, device=device)
    if cfg.hot_experts:
        idx = torch.tensor(cfg.hot_experts, device=device)
        logits[:, idx] += cfg.hot_bias
    return logits.float().contiguous()


def make_routes(cfg: MoEConfig, tokens: int, device="cpu", seed: Optional[int] = None):
    """Router logits -> softmax -> top-k over the global experts.

    Returns (topk_ids int32 [T, k], topk_weights fp32 [T, k]).  Weights are the
    softmax probabilities (renormalize=False in every workload).  Global ids
    outside [expert_offset, expert_offset + E) stay as they are (the forward
    treats them as masked); ``forced_invalid`` routes become -1.
    """
    logits = make_logits(cfg, tokens, device, seed)
    probs = torch.softmax(logits.float(), dim=-1)
    w, ids = torch.topk(probs, cfg.top_k, dim=-1)
    ids = ids.to(torch.int32)
    for (t, j) in cfg.forced_invalid:
        if t < tokens:
            ids[t, j] = -1
    if cfg.global_experts and cfg.global_experts != cfg.num_experts:
        # single-GPU stand-in for expert parallelism: routes to experts that
        # live on other ranks are marked invalid.
        local = (ids >= cfg.expert_offset) & (ids < cfg.expert_offset + cfg.num_experts)
        ids = torch.where(local, ids, torch.full_like(ids, -1))
    return ids.contiguous(), w.float().contiguous()


def make_case(cfg: MoEConfig, tokens: int, device="cpu", weights: Optional[ExpertWeights] = None):
    if weights is None:
        weights = make_weights(cfg, device)
    x = make_activations(cfg, tokens, device)
    ids, tw = make_routes(cfg, tokens, device)
    return dict(x=x, ids=ids, topk_weights=tw, weights=weights)


# ----------------------------------------------------------------------------
# Accounting used by the roofline (bytes the method must move, FLOPs it does)
# ----------------------------------------------------------------------------

def algorithmic_bytes(cfg: MoEConfig, ids: torch.Tensor) -> int:
    """Packed INT4 + scale bytes of every *touched* local expert, plus x, out,
    ids and routing weights.  Intermediate, scratch and padding are excluded
    (they are implementation overhead)."""
    T = ids.shape[0]
    H, I, N1 = cfg.hidden, cfg.inter, cfg.n1
    loc = ids.long() - cfg.expert_offset
    valid = (ids >= 0) & (loc >= 0) & (loc < cfg.num_experts)
    touched = int(torch.unique(loc[valid]).numel())
    wbytes = (H * N1 + I * H) // 2
    if cfg.scale_kind == SCALE_GROUP32:
        sbytes = (H * N1 + I * H) // GROUP * 2
    else:
        sbytes = (N1 + H) * 2
    act = 2
    return touched * (wbytes + sbytes) + T * H * act * 2 + T * cfg.top_k * 8


def valid_routes(cfg: MoEConfig, ids: torch.Tensor) -> int:
    loc = ids.long() - cfg.expert_offset
    valid = (ids >= 0) & (loc >= 0) & (loc < cfg.num_experts)
    return int(valid.sum())


def algorithmic_flops(cfg: MoEConfig, ids: torch.Tensor) -> int:
    R = valid_routes(cfg, ids)
    return 2 * R * (cfg.hidden * cfg.n1 + cfg.inter * cfg.hidden)
