"""Helpers shared by the GPU parity tests (not collected by pytest)."""
import numpy as np
import torch

import oracle
from workloads import gen

# Bar from the problem statement: max NRMSE <= 5e-3 and per-element
# |err| <= 2e-2 * max|ref|, against the oracle's FP32 combine before the cast.
NRMSE_TOL = 5e-3
ELEM_TOL = 2e-2


def compare(gpu_out: torch.Tensor, ref_acc: np.ndarray, what: str = ""):
    g = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    r = ref_acc.astype(np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    rn = np.linalg.norm(r)
    if rn == 0.0:
        assert np.all(g == 0.0), f"{what}: expected exact zeros"
        return 0.0, 0.0
    nrmse = np.linalg.norm(g - r) / rn
    maxerr = np.abs(g - r).max() / np.abs(r).max()
    assert nrmse <= NRMSE_TOL, f"{what}: NRMSE {nrmse:.3e} > {NRMSE_TOL}"
    assert maxerr <= ELEM_TOL, f"{what}: max|err|/max|ref| {maxerr:.3e} > {ELEM_TOL}"
    return nrmse, maxerr


def make_moe(cfg, max_tokens, **kw):
    from weight_only_int4_histogram_gb300 import W4A16MoE
    return W4A16MoE.from_config(cfg, max_tokens=max_tokens, **kw)


def case_on_gpu(cfg, T, weights_gpu=None, device="cuda"):
    """Inputs generated on the GPU (fast at full size)."""
    w = weights_gpu if weights_gpu is not None else gen.make_weights(cfg, device)
    x = gen.make_activations(cfg, T, device)
    ids, tw = gen.make_routes(cfg, T, device)
    return w, x, ids, tw


def oracle_rows(cfg, w, x, ids, tw, rows=None, renormalize=False, w_cpu=None):
    acc, _ = oracle.moe_forward(cfg, x.cpu(), w_cpu if w_cpu is not None else w.to("cpu"),
                                tw.cpu(), ids.cpu(), renormalize=renormalize, rows=rows)
    return acc


def small_cfg(E=6, H=512, I=256, k=2, act=gen.ACT_SWIGLU, scale=gen.SCALE_GROUP32,
              dt=gen.DT_BF16, seed=11, **kw):
    return gen.MoEConfig(f"small_e{E}_h{H}_i{I}_k{k}_a{act}_s{scale}_d{dt}", E, H, I, k,
                         act=act, scale_kind=scale, act_dtype=dt, seed=seed, **kw)
