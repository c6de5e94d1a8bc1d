"""CUDA path against the CPU oracle, through the C ABI (needs a B300)."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from sparse_mixture_experts_66_b300 import moe
from sparse_mixture_experts_66_b300.workload import (DECODE, HEADLINE, PREFILL, SKEWED, SMALL_FP32, WORKLOADS,
                                                     as_f32_numpy, custom, draw)
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("no CUDA device: the GPU tests need a B300")
    moe.load()
    yield
    torch.cuda.synchronize()


# ---------------------------------------------------------------------------
# Stage-isolated checks
# ---------------------------------------------------------------------------
STAGE_CASES = [
    custom(1000, 256, 1408, 8, 2, 1.25, seed=1),
    custom(777, 512, 384, 6, 2, 1.0, router_bias="zipf", seed=2),
    custom(300, 128, 64, 64, 2, 1.0, router_bias="zipf", seed=3),
    custom(256, 64, 256, 4, 1, 1.25, dtype="f32", seed=0),
    custom(512, 64, 64, 256, 8, 1.0, seed=4),
    # every fp32 score of expert 0 rounds to 1.0: a full tie, resolved by token order
    custom(400, 128, 256, 8, 2, 1.0, router_bias="const:0:30", seed=9),
    # Above one CTA's registers (8192 requests) an expert's requests are split over a cluster of 2-8 CTAs,
    # one slice each. 12000 requests: 4 slices of 3000, with overflow
    custom(6000, 64, 64, 8, 2, 1.0, router_bias="zipf", seed=17),
    # 32000 requests, 8 slices of 4000; expert 0 receives nearly all tokens
    custom(16000, 64, 64, 4, 2, 1.0, router_bias="const:0:6", seed=22),
    # k = 1, 17000 requests: 8 slices of 2128 and a short last one (2104)
    custom(17000, 64, 64, 2, 1, 0.75, router_bias="const:1:3", seed=20),
    # 40000 and 48000 requests: 8 slices at 5000 and 6000
    custom(20000, 64, 64, 4, 2, 1.0, router_bias="const:0:6", seed=18),
    custom(24000, 64, 64, 4, 2, 1.0, router_bias="const:0:6", seed=19),
    # a full tie across slices: expert 0's 7000 requests all score 1.0 and the quota (C = 4375) ends inside
    # the third of four slices, so the ties and kept rows of the earlier slices decide the boundary
    custom(7000, 64, 64, 8, 2, 2.5, router_bias="const:0:30", seed=23),
    # eight slices of a fully tied expert: 32000 requests (L = 4000) and a quota C = 12000 that ends exactly at a
    # slice boundary (tokens 0..11999 are requests 0..23999); k = 1 with 30000 requests (L = 3752, a short last
    # slice) and a quota of 13500 that ends inside the fourth slice
    custom(16000, 64, 64, 4, 2, 1.5, router_bias="const:0:30", seed=29),
    custom(30000, 64, 64, 2, 1, 0.9, router_bias="const:0:30", seed=30),
    # the skewed batch's shape: 64 experts, 16384 requests in 2 slices, the head experts overflowing
    custom(8192, 64, 64, 64, 2, 1.0, router_bias="zipf", seed=26),
    # the single-CTA kernel streaming the list in passes: 66000 requests (more than 8 slices hold) and
    # 64 experts x 4 slices (more CTAs than one wave)
    custom(33000, 64, 64, 4, 2, 1.0, router_bias="const:0:6", seed=24),
    custom(10000, 64, 64, 64, 2, 1.0, router_bias="zipf", seed=25),
]


@pytest.mark.parametrize("w", STAGE_CASES, ids=lambda w: w.name)
def test_capacity_stage_is_bit_exact_on_gpu_routing(w):
    """The oracle's capacity step, run on the GPU's own picks and fp32 scores,
    must reproduce the GPU's counts, slots and drops exactly."""
    inp = draw(w)
    g = parity.run_gpu(w, inp)
    cr, ck, slot = O.load().capacity_assign(g["topk_idx"], g["score"].astype(np.float64), w.N,
                                            O.load().capacity(w.T, w.N, w.k, w.capacity_factor))
    assert np.array_equal(cr, g["counts_raw"])
    assert np.array_equal(ck, g["counts_kept"])
    assert np.array_equal(slot, parity.gpu_slots(g))
    parity.check_layout(g, w.k, parity.row_align(w))


@pytest.mark.parametrize("w", STAGE_CASES[:3], ids=lambda w: w.name)
def test_permute_is_an_exact_gather(w):
    inp = draw(w)
    g = parity.run_gpu(w, inp)
    xp = g["_ws"].views()["x_perm"].cpu()
    rows = int(g["offsets"][-1])
    rt = torch.from_numpy(g["row_token"][:rows]).long()
    x = inp["x"]
    used = rt >= 0
    assert torch.equal(xp[:rows][used], x[rt[used]])
    assert torch.all(xp[:rows][~used] == 0)


@pytest.mark.parametrize("w", STAGE_CASES[:3] + [custom(64, 1024, 4096, 8, 2, math.inf, seed=13)],
                         ids=lambda w: w.name)
def test_combine_is_the_fixed_order_fp32_sum(w):
    """y[t] = sum over kept picks in pick order of y_perm rows (x's dtype,
    widened exactly), in fp32, then rounded once to the storage dtype:
    reproduced bit for bit."""
    inp = draw(w)
    g = parity.run_gpu(w, inp)
    v = g["_ws"].views()
    yp = v["y_perm"].float().cpu().numpy()
    ys = v["y_split"].cpu().numpy()
    acc = np.zeros((w.T, w.d), dtype=np.float32)
    for j in range(w.k):
        r = g["row_of"][:, j]
        m = r >= 0
        term = yp[r[m]]
        for sl in range(ys.shape[0]):
            term = term + ys[sl][r[m]]
        acc[m] = acc[m] + term
    ref = torch.from_numpy(acc).to(g["_y"].dtype)
    assert torch.equal(g["_y"].cpu(), ref)


@pytest.mark.parametrize("w", STAGE_CASES[:3], ids=lambda w: w.name)
def test_expert_ffn_rows_against_oracle(w):
    """Each permuted row's y_perm equals row_gate * E_e(x_perm row) (oracle, fp64)."""
    inp = draw(w)
    g = parity.run_gpu(w, inp)
    v = g["_ws"].views()
    xp = v["x_perm"].float().cpu().numpy()
    yp = v["y_perm"].float().cpu().numpy()
    off = g["offsets"]
    w1, b1, w2, b2 = (as_f32_numpy(inp[n]) for n in ("w1", "b1", "w2", "b2"))
    rng = np.random.default_rng(0)
    orc = O.load()
    rows = int(off[-1])
    check = rng.choice(rows, size=min(rows, 96), replace=False)
    errs, scale = [], []
    for r in check:
        e = int(np.searchsorted(off, r, side="right") - 1)
        if g["row_token"][r] < 0:
            continue
        ref = g["row_gate"][r] * orc.expert_ffn(xp[r], w1[e], b1[e], w2[e], b2[e])
        errs.append(np.max(np.abs(yp[r] - ref)))
        scale.append(np.max(np.abs(ref)))
    assert max(errs) <= parity.TOL[w.dtype] * max(scale)


@pytest.mark.parametrize("w", [STAGE_CASES[0], WORKLOADS[HEADLINE], custom(1024, 520, 712, 16, 2, 1.0, seed=51)],
                         ids=lambda w: w.name)
def test_hidden_activations_within_bf16_rounding_of_exact_gelu(w):
    """h = GELU(x_perm W1^T + b1) from the first GEMM's epilogue equals the
    exact (erf) GELU of the oracle up to the bf16 rounding of h and the fp32
    accumulation error: |h - h_ref| <= 2^-8 |h_ref| + 1e-4."""
    inp = draw(w)
    g = parity.run_gpu(w, inp)
    v = g["_ws"].views()
    xp = v["x_perm"].float().cpu().numpy()
    hh = v["h"].float().cpu().numpy()
    off = g["offsets"]
    w1, b1, w2, b2 = (as_f32_numpy(inp[n]) for n in ("w1", "b1", "w2", "b2"))
    rng = np.random.default_rng(1)
    orc = O.load()
    rows = [r for r in rng.choice(int(off[-1]), size=64, replace=False) if g["row_token"][r] >= 0]
    worst = 0.0
    for r in rows:
        e = int(np.searchsorted(off, r, side="right") - 1)
        h_ref, _ = orc.expert_ffn_hidden(xp[r], w1[e], b1[e], w2[e], b2[e])
        excess = np.abs(hh[r] - h_ref) - (2.0 ** -8 * np.abs(h_ref) + 1e-4)
        worst = max(worst, float(excess.max()))
    assert worst <= 0.0, worst


ROUTER_CASES = [
    custom(2048, 1024, 64, 8, 2, math.inf, seed=5),  # d split over clusters of 4 CTAs
    custom(1100, 512, 64, 32, 2, math.inf, seed=6),  # 32 experts, split of 4, ragged last tile
    custom(1100, 512, 64, 64, 4, math.inf, router_bias="zipf", seed=7),  # 64 experts, k=4, no split
    custom(2500, 384, 64, 16, 2, math.inf, seed=8),  # split of 2 (6 k-blocks)
    # four column groups per token from 64 experts on: 40 experts leave group 2
    # part-padded and group 3 empty; 128 and 200 experts give 32 and 64 columns
    # per group (the top-k candidates of every group merged by group 0)
    custom(1100, 256, 64, 16, 4, math.inf, seed=53),  # k = 4 on the one-thread-per-token epilogue (8-step insertion)
    custom(1100, 512, 64, 40, 3, math.inf, router_bias="zipf", seed=9),
    custom(1300, 256, 64, 128, 6, math.inf, seed=10),
    custom(1500, 256, 64, 200, 8, math.inf, router_bias="zipf", seed=11),
]


@pytest.mark.parametrize("w", ROUTER_CASES, ids=lambda w: w.name)
def test_router_against_oracle(w):
    inp = draw(w)
    g = parity.run_gpu(w, inp)
    ref = parity.oracle_ref(w, inp, sel=np.array([0]))
    mg = parity.margins(ref["logits"], w.k)
    hi = mg > parity.MARGIN
    assert np.array_equal(g["topk_idx"][hi], ref["idx"][hi])
    assert np.allclose(g["gate"], ref["gate"], rtol=2e-5, atol=1e-6)
    assert np.allclose(g["gate"].sum(axis=1), 1.0, atol=1e-6)


@pytest.mark.parametrize("N,k", [(64, 4), (256, 8)])
def test_router_exact_ties_keep_the_lower_expert(N, k):
    """Experts with identical W_g rows and bias have bit-identical logits; placed
    in different column groups of the epilogue (every 16 or 64 experts) and
    biased above the rest, they must be picked in ascending expert order, the
    same order one pass over all columns gives."""
    w = custom(1100, 128, 64, N, k, math.inf, seed=12)  # T > 1024: the tensor-core router
    inp = draw(w)
    step = N // 4
    tied = [3 + step * j for j in range(4)]
    wg = inp["w_g"].clone()
    for e in tied[1:]:
        wg[e] = wg[tied[0]]
    bias = torch.zeros(N, dtype=torch.float32)
    bias[tied] = 20.0
    inp = dict(inp, w_g=wg, router_bias=bias)
    g = parity.run_gpu(w, inp)
    want = np.array(tied[: min(k, 4)])
    assert (g["topk_idx"][:, : len(want)] == want).all()
    if k > 4:  # the rest are ordinary picks, none of them tied experts
        assert not np.isin(g["topk_idx"][:, 4:], tied).any()
    assert np.allclose(g["gate"][:, : len(want)], g["gate"][:, :1], rtol=0, atol=0)


# ---------------------------------------------------------------------------
# End to end, every output element, small sizes spanning several tiles
# ---------------------------------------------------------------------------
E2E_CASES = [
    WORKLOADS[SMALL_FP32],
    custom(1000, 256, 1408, 8, 2, 1.25, seed=1),  # ragged d_ff tile, segments not multiples of 128
    custom(777, 512, 384, 6, 2, 1.0, router_bias="zipf", seed=2),  # skewed: drops
    custom(300, 128, 64, 64, 2, 1.0, router_bias="zipf", seed=3),  # d_ff below one tile, many experts
    custom(1, 256, 512, 8, 2, 1.25, seed=6),  # a single token
    custom(200, 128, 256, 1, 1, 1.0, seed=7),  # N = 1, k = 1: a dense FFN
    custom(200, 64, 64, 1, 1, 1.0, dtype="f32", seed=7),
    custom(130, 128, 256, 4, 4, math.inf, seed=8),  # k = N: the full soft mixture
    custom(512, 64, 64, 256, 8, 1.0, seed=4),  # the largest N and k
    custom(400, 128, 256, 8, 2, 1.0, router_bias="const:0:3", seed=9),  # most tokens want expert 0
    custom(640, 128, 128, 8, 2, 0.01, seed=10),  # tiny capacity: nearly everything dropped
    custom(333, 64, 128, 8, 2, 1.25, router_bias="const:3:-60", seed=11),  # an expert nobody picks
    custom(256, 64, 256, 4, 1, 1.25, dtype="f32", router_bias="zipf", seed=12),  # fp32 with drops
] + [
    # decode-shaped batches (bf16, T*k <= 64*N): swap-AB expert GEMMs, second GEMM split along d_ff;
    # 32-row token chunks while T*k <= 16*N, 64-row chunks above
    custom(64, 1024, 4096, 8, 2, math.inf, seed=13),
    custom(64, 512, 1024, 8, 2, math.inf, router_bias="const:0:3", seed=17),  # expert 0 spans two 32-row chunks
    custom(200, 512, 1024, 8, 2, math.inf, seed=18),  # 64-row chunks
    custom(48, 512, 2048, 8, 2, 1.0, router_bias="zipf", seed=14),  # drops
    custom(5, 768, 3072, 16, 4, math.inf, seed=15),  # fewer picks than experts
    custom(40, 520, 1000, 8, 2, 1.25, seed=16),  # ragged d and d_ff: partial k-blocks and weight tiles
    custom(700, 136, 200, 4, 2, 1.25, seed=50),  # CTA-pair path, d_ff = 8 mod 16: 16-byte h stores
    # the narrow CTA-pair form (C <= 256: 128-column tiles): every expert a masked 128-row tail, with ragged d
    # and d_ff (partial k-block, partial n-tiles); then full 256-row blocks mixed with tails
    custom(1024, 520, 712, 16, 2, 1.0, seed=51),
    custom(3000, 256, 640, 32, 2, 1.25, router_bias="zipf", seed=52),
]


@pytest.mark.parametrize("w", E2E_CASES, ids=lambda w: w.name)
def test_end_to_end(w):
    rep, g, ref, _ = parity.full_check(w)
    print(w.name, rep)


@pytest.mark.parametrize("flags", [moe.MOE_FLAG_RENORM_SURVIVORS, moe.MOE_FLAG_IDENTITY_FALLBACK, 3])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_flag_variants(flags, dtype):
    w = custom(500, 128, 256, 8, 2, 0.5, dtype=dtype, router_bias="zipf", seed=13)
    rep, g, ref, _ = parity.full_check(w, flags=flags)
    assert rep["dropped"] > 0
    print(w.name, flags, rep)


def test_deterministic_across_runs():
    w = custom(1500, 256, 512, 8, 2, 1.0, router_bias="zipf", seed=14)
    inp = draw(w)
    a = parity.run_gpu(w, inp)
    b = parity.run_gpu(w, inp, dev=a["_dev"], reps=3)
    assert torch.equal(a["_y"], b["_y"])
    assert np.array_equal(a["row_of"], b["row_of"])


@pytest.mark.parametrize("w", [
    custom(700, 256, 512, 8, 2, 1.0, router_bias="zipf", seed=15),
    # larger batches: 6000 rows (d = 1024) with drops and a zipf skew, 20000 rows over 16 experts
    custom(3000, 1024, 512, 8, 2, 1.0, router_bias="zipf", seed=27),
    custom(10000, 512, 256, 16, 2, 1.25, seed=28),
    # decode-shaped: the swap-AB expert FFN and the K-sliced combine
    custom(64, 1024, 4096, 8, 2, math.inf, seed=23),
], ids=lambda w: w.name)
def test_stage_calls_compose_to_forward(w):
    """moe_route + moe_dispatch + moe_expert_ffn + moe_combine on caller
    buffers give the same bits as moe_forward."""
    inp = draw(w)
    g = parity.run_gpu(w, inp)
    dev, cfg = g["_dev"], g["_cfg"]
    L = moe.moe_get_workspace_layout(cfg)
    ws = moe.Workspace(cfg)
    T, k, N, R = w.T, w.k, w.N, L.rows
    i32 = dict(dtype=torch.int32, device="cuda")
    f32 = dict(dtype=torch.float32, device="cuda")
    topk_idx, gate, score = torch.empty(T, k, **i32), torch.empty(T, k, **f32), torch.empty(T, k, **f32)
    moe.moe_route(cfg, dev["x"], dev["w_g"], dev["router_bias"], topk_idx, gate, score, ws.buf)
    counts_raw, counts_kept, offsets = torch.empty(N, **i32), torch.empty(N, **i32), torch.empty(N + 1, **i32)
    row_of, row_token, row_gate = torch.empty(T, k, **i32), torch.empty(R, **i32), torch.empty(R, **f32)
    x_perm = torch.empty(R, w.d, dtype=dev["x"].dtype, device="cuda")
    moe.moe_dispatch(cfg, dev["x"], topk_idx, gate, score, counts_raw, counts_kept, offsets, row_of, row_token,
                     row_gate, x_perm, ws.buf)
    h = torch.empty(R, w.d_ff, dtype=dev["x"].dtype, device="cuda")
    y_perm = torch.empty(R, w.d, dtype=dev["x"].dtype, device="cuda")
    moe.moe_expert_ffn(cfg, x_perm, offsets, dev["w1"], dev["b1"], dev["w2"], dev["b2"], row_gate, h, y_perm, ws.buf)
    y = torch.empty_like(dev["x"])
    moe.moe_combine(cfg, y_perm, row_of, gate, dev["x"], y, ws.buf)
    ws.status()
    assert torch.equal(y, g["_y"])
    assert np.array_equal(row_of.cpu().numpy(), g["row_of"])


def test_device_status_is_clean_after_runs():
    w = custom(64, 64, 64, 4, 2, 1.0, seed=16)
    g = parity.run_gpu(w, draw(w))
    g["_ws"].status()


# ---------------------------------------------------------------------------
# The published workloads at full size: routing and capacity on every token,
# outputs on a sample of tokens (cutoff tokens, dropped tokens, random tokens)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", [HEADLINE, SKEWED, DECODE, PREFILL])
def test_full_size_workloads(name):
    w = WORKLOADS[name]
    rep, g, ref, _ = parity.full_check(w, sample=48)
    print(name, rep)
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Router statistics (MOE_FLAG_ROUTER_STATS + moe_router_stats)
# ---------------------------------------------------------------------------
STATS_CASES = [
    custom(2048, 256, 64, 8, 2, 1.25, seed=21),  # bf16, tensor-core router
    custom(1500, 128, 64, 64, 2, 1.0, router_bias="zipf", seed=22),  # bf16, tensor-core router, N=64 + bias
    custom(1100, 128, 64, 200, 4, 1.0, seed=26),  # bf16, tensor-core router, four 64-column groups, padded tail
    # 64 experts with d split over clusters of 4 (8 k-blocks) and four column groups: the summed partials feed
    # the stored probability rows
    custom(1500, 512, 64, 64, 2, 1.0, router_bias="zipf", seed=31),
    custom(300, 128, 64, 16, 4, math.inf, seed=23),  # bf16, split-column router
    custom(1200, 64, 64, 4, 1, 1.25, dtype="f32", seed=24),  # fp32, N <= 8 register router
    custom(1100, 64, 64, 40, 3, 1.0, dtype="f32", seed=25),  # fp32, generic router
]


@pytest.mark.parametrize("w", STATS_CASES, ids=lambda w: w.name)
def test_router_stats_against_oracle(w):
    """Stored probability rows, f_e, P_e, the auxiliary loss and the z-loss
    against the oracle. f_e comes from the GPU's own picks (compared exactly);
    P_e, aux and z within 2e-5 relative (fp32 against fp64)."""
    inp = draw(w)
    g = parity.run_gpu(w, inp, flags=moe.MOE_FLAG_ROUTER_STATS)
    cfg, ws = g["_cfg"], g["_ws"]
    v = ws.views()
    f = torch.empty(w.N, dtype=torch.float32, device="cuda")
    P = torch.empty(w.N, dtype=torch.float32, device="cuda")
    losses = torch.empty(2, dtype=torch.float32, device="cuda")
    moe.moe_router_stats(cfg, ws.buf, v["counts_raw"], f, P, losses)
    ws.status()
    probs = v["probs"].cpu().numpy().astype(np.float64)
    ref = parity.oracle_ref(w, inp, sel=np.array([0]))
    # the stored rows are the softmax of the fp32 logits; the picks' rows equal their scores exactly
    assert np.max(np.abs(probs - ref["probs"])) <= 2e-5
    assert np.allclose(probs.sum(axis=1), 1.0, atol=1e-5)
    picked = np.take_along_axis(v["probs"].cpu().numpy(), g["topk_idx"].astype(np.int64), axis=1)
    assert np.array_equal(picked, g["score"])
    # the oracle's statistics on the GPU's own picks
    f_ref, P_ref, aux_ref, z_ref = O.load().router_stats(ref["logits"], ref["probs"], g["topk_idx"])
    assert np.array_equal(f.cpu().numpy(), (g["counts_raw"] / np.float32(w.T * w.k)).astype(np.float32))
    assert np.allclose(f.cpu().numpy(), f_ref, rtol=1e-6, atol=0)
    assert np.allclose(P.cpu().numpy(), P_ref, rtol=2e-5, atol=1e-7)
    aux, z = losses.cpu().numpy().astype(np.float64)
    assert abs(aux - aux_ref) <= 2e-5 * aux_ref
    assert abs(z - z_ref) <= 2e-5 * z_ref


def test_router_stats_leave_routing_unchanged():
    """The statistics flag changes no routing or output bit."""
    w = STATS_CASES[1]
    inp = draw(w)
    a = parity.run_gpu(w, inp)
    b = parity.run_gpu(w, inp, flags=moe.MOE_FLAG_ROUTER_STATS)
    for key in ("topk_idx", "gate", "score", "row_of", "offsets"):
        assert np.array_equal(a[key], b[key]), key
    assert torch.equal(a["_y"], b["_y"])


# ---------------------------------------------------------------------------
# Shared always-on expert (MOE_FLAG_SHARED_EXPERT)
# ---------------------------------------------------------------------------
SHARED_CASES = [
    custom(1000, 256, 1408, 8, 2, 1.25, seed=1),  # bf16, CTA-pair routed FFN
    custom(300, 256, 512, 8, 2, 1.25, router_bias="zipf", seed=30),  # T not a multiple of 128, drops
    custom(48, 512, 2048, 8, 2, 1.0, router_bias="zipf", seed=14),  # decode-shaped routed FFN
    WORKLOADS[SMALL_FP32],  # fp32 SIMT path
]


@pytest.mark.parametrize("w", SHARED_CASES, ids=lambda w: w.name)
def test_shared_expert_against_oracle(w):
    """moe_forward_shared equals the oracle's forward with the shared expert
    added to every token, under the same parity rules as the routed layer."""
    from sparse_mixture_experts_66_b300.workload import draw_shared
    inp = draw(w)
    sh = draw_shared(w)
    cfg = moe.config_of(w, moe.MOE_FLAG_SHARED_EXPERT)
    dev = parity.to_device(inp)
    shd = {k: v.cuda() for k, v in sh.items()}
    ws = moe.Workspace(cfg)
    y = torch.empty_like(dev["x"])
    moe.moe_forward_shared(cfg, dev["x"], dev["w_g"], dev["router_bias"], dev["w1"], dev["b1"], dev["w2"], dev["b2"],
                           shd["sw1"], shd["sb1"], shd["sw2"], shd["sb2"], y, ws.buf)
    ws.status()
    v = ws.views()
    g = {k: t.cpu().numpy() for k, t in v.items() if k not in ("x_perm", "h", "y_perm", "y_split", "y_shared")}
    g["y"] = y.float().cpu().numpy().astype(np.float64)
    ref = O.load().forward(*(as_f32_numpy(inp[n]) for n in ("x", "w_g", "w1", "b1", "w2", "b2")), k=w.k,
                           cf=w.capacity_factor, router_bias=as_f32_numpy(inp["router_bias"]),
                           shared=tuple(as_f32_numpy(sh[n]) for n in ("sw1", "sb1", "sw2", "sb2")))
    rep = parity.compare(w, g, ref)
    print(w.name, rep)


def test_shared_expert_stage_call_composes():
    """moe_shared_expert + moe_combine on the stage calls give moe_forward_shared's output bit for bit."""
    from sparse_mixture_experts_66_b300.workload import draw_shared
    w = SHARED_CASES[1]
    inp, sh = draw(w), draw_shared(w)
    cfg = moe.config_of(w, moe.MOE_FLAG_SHARED_EXPERT)
    d = parity.to_device(inp)
    s = {k: t.cuda() for k, t in sh.items()}
    ws = moe.Workspace(cfg)
    y1 = torch.empty_like(d["x"])
    moe.moe_forward_shared(cfg, d["x"], d["w_g"], d["router_bias"], d["w1"], d["b1"], d["w2"], d["b2"], s["sw1"],
                           s["sb1"], s["sw2"], s["sb2"], y1, ws.buf)
    ws2 = moe.Workspace(cfg)
    v = ws2.views()
    moe.moe_route(cfg, d["x"], d["w_g"], d["router_bias"], v["topk_idx"], v["gate"], v["score"], ws2.buf)
    moe.moe_dispatch(cfg, d["x"], v["topk_idx"], v["gate"], v["score"], v["counts_raw"], v["counts_kept"],
                     v["offsets"], v["row_of"], v["row_token"], v["row_gate"], v["x_perm"], ws2.buf)
    moe.moe_expert_ffn(cfg, v["x_perm"], v["offsets"], d["w1"], d["b1"], d["w2"], d["b2"], v["row_gate"], v["h"],
                       v["y_perm"], ws2.buf)
    moe.moe_shared_expert(cfg, d["x"], s["sw1"], s["sb1"], s["sw2"], s["sb2"], ws2.buf)
    y2 = torch.empty_like(d["x"])
    moe.moe_combine(cfg, v["y_perm"], v["row_of"], v["gate"], d["x"], y2, ws2.buf)
    ws.status()
    ws2.status()
    assert torch.equal(y1, y2)


# ---------------------------------------------------------------------------
# Expert-choice routing (MOE_FLAG_EXPERT_CHOICE)
# ---------------------------------------------------------------------------
EC_CASES = [
    custom(1000, 256, 512, 8, 2, 1.0, seed=41),  # bf16, CTA-pair FFN, k = N = 8 combine
    custom(800, 128, 256, 16, 2, 1.0, router_bias="zipf", seed=42),  # N = 16 > 8: the many-pick combine
    custom(40, 512, 1024, 8, 2, 1.0, seed=43),  # T <= 64: decode-shaped (swap-AB) FFN
    custom(256, 64, 256, 4, 1, 1.25, dtype="f32", seed=44),  # fp32 SIMT path
    # 64 experts on the tensor-core router (d split over clusters of 4, four column groups per token)
    custom(1100, 512, 256, 64, 2, 1.0, seed=45),
]


@pytest.mark.parametrize("w", EC_CASES, ids=lambda w: w.name)
def test_expert_choice_against_oracle(w):
    """Each expert takes its C most probable tokens (ties: lower token); a
    token's output sums p[t,e] E_e(x_t) over the experts that took it. Taken
    sets must equal the oracle's at every expert whose C-th and (C+1)-th fp64
    probabilities are not a near tie; outputs are compared on the tokens whose
    taken sets agree."""
    inp = draw(w)
    g = parity.run_gpu(w, inp, flags=moe.MOE_FLAG_EXPERT_CHOICE)
    C = O.load().capacity(w.T, w.N, w.k, w.capacity_factor)
    ref = parity.oracle_ref(w, inp, sel=np.array([0]))
    probs = ref["probs"]
    taken_ref, counts_ref, y_ref = O.load().expert_choice(
        as_f32_numpy(inp["x"]), probs, *(as_f32_numpy(inp[n]) for n in ("w1", "b1", "w2", "b2")), C)
    taken = (g["row_of"].reshape(w.T, w.N) >= 0).astype(np.int32)
    ties = set()
    for e in range(w.N):
        col = np.sort(probs[:, e])[::-1]
        if C < w.T and col[C - 1] - col[C] <= parity.NEAR_TIE * col[C - 1]:
            ties.add(e)
    ok_e = np.array([e not in ties for e in range(w.N)])
    assert np.array_equal(taken[:, ok_e], taken_ref[:, ok_e]), "taken sets differ"
    assert np.array_equal(g["counts_kept"], np.minimum(C, w.T) * np.ones(w.N, dtype=np.int32))
    tok_ok = np.all(taken == taken_ref, axis=1)
    assert tok_ok.sum() >= 0.99 * w.T
    # the GPU's weights are its fp32 probabilities: rows carry p[t, e]
    rows = g["row_of"].reshape(w.T, w.N)
    tt, ee = np.nonzero(rows >= 0)
    assert np.allclose(g["row_gate"][rows[tt, ee]], probs[tt, ee], rtol=2e-5, atol=1e-7)
    scale = np.max(np.abs(y_ref[tok_ok]))
    err = np.max(np.abs(g["y"][tok_ok] - y_ref[tok_ok]))
    assert err <= parity.TOL[w.dtype] * scale, (err, scale)


def test_expert_ffn_accepts_16_byte_aligned_outputs():
    """h and y_perm only 16-byte aligned (the ABI's minimum): the same rows as
    with the workspace's 256-byte aligned buffers, bit for bit."""
    w = STAGE_CASES[0]
    inp = draw(w)
    g = parity.run_gpu(w, inp)
    cfg, ws = g["_cfg"], g["_ws"]
    v = ws.views()
    R = ws.layout.rows
    hb = torch.empty(R * w.d_ff * 2 + 32, dtype=torch.uint8, device="cuda")
    yb = torch.empty(R * w.d * 2 + 32, dtype=torch.uint8, device="cuda")
    h16 = hb[16:16 + R * w.d_ff * 2].view(torch.bfloat16).view(R, w.d_ff)
    y16 = yb[16:16 + R * w.d * 2].view(torch.bfloat16).view(R, w.d)
    d = g["_dev"]
    moe.moe_expert_ffn(cfg, v["x_perm"], v["offsets"], d["w1"], d["b1"], d["w2"], d["b2"], v["row_gate"], h16, y16,
                       ws.buf)
    ws.status()
    rows = int(g["offsets"][-1])
    assert torch.equal(h16[:rows], v["h"][:rows])
    assert torch.equal(y16[:rows], v["y_perm"][:rows])


@pytest.mark.skipif(torch.cuda.is_available() and torch.cuda.device_count() < 2, reason="needs a second GPU")
def test_forward_on_a_second_device():
    """The one-time set-up of the tensor-core kernels (shared-memory opt-ins,
    SM and resident-pair counts) is kept per device: a forward on device 1
    after one on device 0 launches and gives the same bits."""
    w = custom(1100, 256, 512, 8, 2, 1.25, seed=29)
    inp = draw(w)
    outs = []
    for dev in (0, 1):
        with torch.cuda.device(dev):
            d = {k: (None if v is None else v.to(f"cuda:{dev}")) for k, v in inp.items()}
            cfg = moe.config_of(w)
            y, ws = moe.forward(cfg, d["x"], d["w_g"], d["w1"], d["b1"], d["w2"], d["b2"], d["router_bias"])
            ws.status()
            outs.append(y.cpu())
    assert torch.equal(outs[0], outs[1])
