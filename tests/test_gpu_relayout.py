"""GPU checks of the plan-time weight relayout (``w4a16_moe_relayout_weights``)
and of forwards that read relaid-out weights.

The relayout is byte work: the GPU output must equal the oracle's
``relayout_interleaved`` bit for bit.  A forward on relaid-out weights computes
the same function: it must match the oracle within the parity tolerance on
both GEMM paths, and on the tensor-core path (where the dequantised operand
tile is the same in both layouts) reproduce the checkpoint-layout forward bit
for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import gen
from moe_testlib import case_on_gpu, compare, make_moe, oracle_rows, small_cfg

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

PATHS = {"tc": 1, "cc": 2}

SHAPES = [
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_GROUP32, dt=gen.DT_BF16),
    dict(act=gen.ACT_RELU2, scale=gen.SCALE_GROUP32, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_FP16),
    dict(act=gen.ACT_RELU2, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_BF16),
    dict(act=gen.ACT_SWIGLU, scale=gen.SCALE_GROUP32, dt=gen.DT_FP16),
]


@pytest.fixture(scope="module", autouse=True)
def _build():
    from weight_only_int4_histogram_gb300 import build
    build.build()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"a{s['act']}s{s['scale']}d{s['dt']}")
def test_relayout_bit_exact_against_oracle(shape):
    cfg = small_cfg(E=3, H=704, I=320, k=2, **shape)
    w = gen.make_weights(cfg, "cuda")
    moe = make_moe(cfg, 8)
    il = moe.relayout_weights(w)
    torch.cuda.synchronize()
    E, H, I, N1 = cfg.num_experts, cfg.hidden, cfg.inter, cfg.n1
    want13 = oracle.relayout_interleaved(w.w13.cpu(), cfg.scale_kind, E, N1, H)
    want2 = oracle.relayout_interleaved(w.w2.cpu(), cfg.scale_kind, E, H, I)
    np.testing.assert_array_equal(il.w13.cpu().numpy(), want13)
    np.testing.assert_array_equal(il.w2.cpu().numpy(), want2)
    # scales are untouched and shared
    assert il.s13.data_ptr() == w.s13.data_ptr() and il.s2.data_ptr() == w.s2.data_ptr()


def test_relayout_in_place_group_scales():
    cfg = small_cfg(E=4, H=512, I=256, k=2)
    w = gen.make_weights(cfg, "cuda")
    ref = oracle.relayout_interleaved(w.w13.cpu(), 0, cfg.num_experts, cfg.n1, cfg.hidden)
    moe = make_moe(cfg, 8)
    il = moe.relayout_weights(gen.ExpertWeights(w.w13.clone(), w.s13, w.w2.clone(), w.s2), in_place=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(il.w13.cpu().numpy(), ref)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"a{s['act']}s{s['scale']}d{s['dt']}")
@pytest.mark.parametrize("T", [7, 61])
def test_forward_on_relaid_out_weights(shape, T, path):
    cfg = small_cfg(E=5, H=704, I=320, k=3, **shape)
    w, x, ids, tw = case_on_gpu(cfg, T)
    base = make_moe(cfg, T)
    base.set_gemm_path(PATHS[path])
    want = base(x, w, tw, ids).clone()
    moe = make_moe(cfg, T)
    moe.set_gemm_path(PATHS[path])
    il = moe.relayout_weights(w)
    out = moe(x, il, tw, ids)
    torch.cuda.synchronize()
    moe.check_device_error()
    compare(out, oracle_rows(cfg, w, x, ids, tw), f"interleaved {cfg.name} T={T} {path}")
    if path == "tc":
        assert torch.equal(out.view(torch.int16), want.view(torch.int16))


@pytest.mark.parametrize("name,T", [("kimi_tp8_e384_h7168_i256_k8", 32), ("kimi_tp8_e384_h7168_i256_k8", 2048),
                                    ("relu2_skew_e64_h2688_i1856_k6", 4096)])
def test_full_size_relaid_out_sampled_rows(name, T):
    cfg = gen.CONFIGS[name]
    w = gen.make_weights(cfg, "cuda")
    moe = make_moe(cfg, T)
    il = moe.relayout_weights(w)
    _, x, ids, tw = case_on_gpu(cfg, T, weights_gpu=w)
    out = moe(x, il, tw, ids)
    torch.cuda.synchronize()
    moe.check_device_error()
    again = moe(x, il, tw, ids)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), out.view(torch.int16))
    rows = sorted(set([0, T - 1] + np.random.default_rng(T).integers(0, T, size=min(T, 30)).tolist()))
    compare(out[rows], oracle_rows(cfg, w, x, ids, tw, rows=rows), f"{name} T={T} interleaved")
