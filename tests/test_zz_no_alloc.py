"""moe_forward_noalloc against moe_forward (needs a B300).

moe_forward_noalloc serves callers that cannot allocate device memory (plugin
or custom-op hosts that supply only inputs and outputs, code under an
allocator that forbids direct cudaMalloc): it runs the same forward on the
library's fixed 32 MiB device scratch array instead of a caller workspace.
This file is collected last on purpose, and it also passes alone in a fresh
process: the first call sets the scratch address up on the device.
"""
import math

import pytest
import torch

from sparse_mixture_experts_66_b300 import moe
from sparse_mixture_experts_66_b300.workload import SMALL_FP32, WORKLOADS, custom, draw, draw_x_only

pytestmark = pytest.mark.gpu

CASES = [WORKLOADS[SMALL_FP32], custom(300, 256, 512, 8, 2, 1.0, router_bias="zipf", seed=21)]


def _dev(inp):
    return {k: (None if v is None else v.cuda()) for k, v in inp.items()}


def _reference(cfg, d, x):
    ws = moe.Workspace(cfg)
    y = torch.empty_like(x)
    moe.moe_forward(cfg, x, d["w_g"], d["router_bias"], d["w1"], d["b1"], d["w2"], d["b2"], y, ws.buf)
    ws.status()
    return y


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_moe_forward_on_two_calls_in_a_row(w):
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    cfg = moe.config_of(w)
    assert moe.moe_workspace_bytes(cfg) <= 32 << 20
    d = _dev(draw(w))
    batches = [d["x"], draw_x_only(w, seed=99).cuda()]  # two different batches, back to back
    outs = []
    for x in batches:
        y = torch.full_like(x, float("nan"))
        moe.moe_forward_noalloc(cfg, x, d["w_g"], d["router_bias"], d["w1"], d["b1"], d["w2"], d["b2"], y)
        outs.append(y)
    torch.cuda.synchronize()
    for x, y in zip(batches, outs):
        ref = _reference(cfg, d, x)
        assert torch.all(torch.isfinite(y))
        # the same launches on the same inputs, and no atomics decide any
        # output: anything but bit equality is a bug (e.g. stale scratch
        # carried over from the previous call)
        assert torch.equal(y, ref)


def test_noalloc_rejects_configs_beyond_its_scratch():
    cfg = moe.config_of(WORKLOADS["bf16_T4096_d1024_N8_k2_dff4096_cf1.25"])
    assert moe.moe_workspace_bytes(cfg) > 32 << 20
    x = torch.zeros(8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_forward_noalloc(cfg, x, x, None, x, x, x, x, x)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE
    assert "32" in str(ei.value) or "bytes" in str(ei.value)
    assert math.isfinite(float(moe.moe_workspace_bytes(cfg)))
