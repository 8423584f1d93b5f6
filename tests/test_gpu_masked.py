"""GPU parity of the masked-count layout entry point
(``w4a16_moe_forward_masked``: expert-major rows with per-expert counts, as a
low-latency expert-parallel dispatch hands them over) against the oracle's
masked forward, on both GEMM paths."""
import numpy as np
import pytest
import torch

import oracle
from workloads import gen
from moe_testlib import compare, make_moe, small_cfg

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

PATHS = {"tc": 1, "cc": 2}


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("shape", [dict(E=6, H=512, I=256), dict(E=5, H=704, I=320, scale=gen.SCALE_PER_CHANNEL),
                                   dict(E=4, H=640, I=192, act=gen.ACT_RELU2),
                                   dict(E=6, H=512, I=256, dt=gen.DT_FP16)])
def test_masked_layout_matches_oracle(shape, path):
    cfg = small_cfg(k=1, seed=41, **shape)
    E, M = cfg.num_experts, 24
    counts = torch.tensor([0, M, 7, 30, 1, 13][:E], dtype=torch.int32)  # one above max_rows: clamped
    w = gen.make_weights(cfg, "cuda")
    x = gen.make_activations(cfg, E * M, "cuda").view(E, M, cfg.hidden)
    moe = make_moe(cfg, E * M)
    moe.set_gemm_path(PATHS[path])
    # rows past the counts must come out +0 whatever the buffer held
    y = torch.full((E, M, cfg.hidden), float("nan"), dtype=x.dtype, device="cuda")
    moe.forward_masked(x, w, counts.cuda(), out=y)
    torch.cuda.synchronize()
    moe.check_device_error()
    acc, _ = oracle.masked_forward(cfg, x.view(E * M, cfg.hidden).cpu(), w.to("cpu"), counts, M)
    got = y.view(E * M, cfg.hidden)
    valid = np.zeros(E * M, bool)
    for e in range(E):
        valid[e * M:e * M + min(int(counts[e]), M)] = True
    compare(got[torch.from_numpy(valid).cuda()], acc[valid], f"masked layout {path}")
    assert (got[torch.from_numpy(~valid).cuda()] == 0).all()


def test_masked_layout_expert_offset_and_repeat():
    """A shard whose experts start at global id 16; two calls in a row on one
    workspace give bit-identical outputs."""
    cfg = small_cfg(E=8, H=512, I=256, k=1, seed=43, global_experts=32, expert_offset=16)
    E, M = cfg.num_experts, 16
    counts = torch.tensor([3, 16, 0, 9, 5, 1, 16, 2], dtype=torch.int32)
    w = gen.make_weights(cfg, "cuda")
    x = gen.make_activations(cfg, E * M, "cuda").view(E, M, cfg.hidden)
    moe = make_moe(cfg, E * M)
    y1 = moe.forward_masked(x, w, counts.cuda()).clone()
    y2 = moe.forward_masked(x, w, counts.cuda())
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    acc, _ = oracle.masked_forward(cfg, x.view(E * M, cfg.hidden).cpu(), w.to("cpu"), counts, M)
    valid = np.zeros(E * M, bool)
    for e in range(E):
        valid[e * M:e * M + int(counts[e])] = True
    compare(y1.view(E * M, -1)[torch.from_numpy(valid).cuda()], acc[valid], "masked layout, offset shard")
