"""The bounded waits of the pipelined kernels give up cleanly (needs a B300).

Every wait inside the tensor-core kernels (on an mbarrier phase, or on a
completion counter raised by another CTA) has a time limit; when it passes, the
kernel records MOE_ERR_TIMEOUT in the workspace's status word and leaves, so a
lost signal surfaces as an error code instead of a stalled GPU. The library's
self-test entry point runs those same wait routines on a barrier that nothing
arms and a counter that nothing raises, with a 1 ms limit: no production
kernel is made to stall.
"""
import pytest
import torch

from sparse_mixture_experts_66_b300 import moe
from sparse_mixture_experts_66_b300.workload import custom, draw

pytestmark = pytest.mark.gpu


def test_bounded_waits_expire_with_timeout_status_and_the_workspace_recovers():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    w = custom(300, 256, 512, 8, 2, 1.0, router_bias="zipf", seed=5)
    cfg = moe.config_of(w)
    ws = moe.Workspace(cfg)
    ws.status()  # clean to start with
    result = torch.full((8,), -1, dtype=torch.int32, device="cuda")
    limit_ns = 1_000_000
    moe.moe_selftest_wait_timeout(ws.buf, limit_ns, result)
    with pytest.raises(moe.MoeError) as ei:
        ws.status()
    assert ei.value.status == moe.MOE_ERR_TIMEOUT
    assert "kernel 9" in str(ei.value)
    r = result.cpu().tolist()
    assert r[0] == 0 and r[1] == 0, r  # neither wait succeeded
    for waited_us in r[2:4]:  # each gave up after its limit, and not much later
        assert limit_ns // 1000 <= waited_us < 200_000, r
    assert r[4] == 0

    # the status word is sticky until the workspace is re-initialised; after
    # that, a forward on the same workspace is clean and matches a fresh one
    d = {k: (None if v is None else v.cuda()) for k, v in draw(w).items()}
    moe.moe_workspace_init(cfg, ws.buf)
    y, _ = moe.forward(cfg, d["x"], d["w_g"], d["w1"], d["b1"], d["w2"], d["b2"], d["router_bias"], ws=ws)
    ws.status()
    y_fresh, ws2 = moe.forward(cfg, d["x"], d["w_g"], d["w1"], d["b1"], d["w2"], d["b2"], d["router_bias"])
    ws2.status()
    assert torch.equal(y, y_fresh)


def test_selftest_rejects_limits_outside_its_range():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    result = torch.zeros(8, dtype=torch.int32, device="cuda")
    for bad in (0, 999, 2_000_000_000):
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_selftest_wait_timeout(ws, bad, result)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
