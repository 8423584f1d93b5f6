"""The no-allocation entry point (fixed device workspace inside the library).

Some callers cannot allocate device memory themselves -- code running inside a
CUDA graph capture, applications whose memory is reserved up front by a pool,
or plug-in hosts that hand a library no allocator.  For them the library runs
route preparation and the forward on one fixed-size device array it owns.
This file checks, through the C ABI, that two calls in a row give the same
output as the regular workspace entry point (bit for bit, and within the
tolerance the parity tests use against the oracle), and that a batch too large
for the fixed array is refused before anything is launched.

Named so that pytest collects it last.
"""
import pytest
import torch

from workloads import gen
from moe_testlib import compare, make_moe, oracle_rows, small_cfg

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _ptr(t):
    return t.data_ptr()


def run_static(moe, x, w, tw, ids, out):
    from weight_only_int4_histogram_gb300 import _lib
    stream = torch.cuda.current_stream().cuda_stream
    _lib.w4a16_moe_forward_static_workspace(
        moe.plan, x.shape[0], _ptr(x), _ptr(w.w13), _ptr(w.s13), _ptr(w.w2), _ptr(w.s2), _ptr(tw),
        _ptr(ids), False, _ptr(out), stream)
    return out


@pytest.mark.parametrize("cfg,tokens", [
    (gen.TINY, (16, 11)),
    (small_cfg(E=16, H=1024, I=512, k=4, seed=21), (40, 7)),
    (small_cfg(E=6, H=704, I=320, k=3, scale=gen.SCALE_PER_CHANNEL, dt=gen.DT_FP16, seed=22), (25, 3)),
])
def test_static_workspace_matches_regular_entry_point(cfg, tokens):
    from weight_only_int4_histogram_gb300 import build
    build.build()
    w = gen.make_weights(cfg, "cuda")
    moe = make_moe(cfg, max(tokens))
    for call, T in enumerate(tokens):  # two calls in a row, different batches
        # fresh inputs per call so a stale result could not pass
        x = gen.make_activations(cfg, T, "cuda", seed=1000 + call)
        ids, tw = gen.make_routes(cfg, T, "cuda", seed=2000 + call)
        want = moe(x, w, tw, ids).clone()
        got = torch.full_like(want, float("nan"))
        run_static(moe, x, w, tw, ids, got)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"call {call}"
        compare(got, oracle_rows(cfg, w, x, ids, tw), f"static workspace call {call}")


def test_static_workspace_rejects_oversized_batch():
    from weight_only_int4_histogram_gb300 import _lib
    cfg = gen.KIMI
    moe = make_moe(cfg, 2048)
    info = moe.route_info(2048)
    assert info.max_slots * cfg.hidden * 4 > _lib.STATIC_WORKSPACE_BYTES
    with pytest.raises(_lib.W4A16Error) as ei:
        # pointers are never touched: the size check fails first
        _lib.w4a16_moe_forward_static_workspace(moe.plan, 2048, 16, 16, 16, 16, 16, 16, 16, False, 16, 0)
    assert ei.value.status == 3
    assert "static workspace" in str(ei.value)
