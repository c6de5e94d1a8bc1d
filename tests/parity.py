"""Helpers shared by the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare them under the parity rules.

Parity rules (floating point decides the integer routing results, so both
sides are compared where the decision is robust):
  * Router: expert indices must equal the oracle's on every token whose k-th
    vs (k+1)-th logit margin (oracle logits) exceeds MARGIN; tokens under the
    margin are counted and reported.
  * Capacity: run alone on the GPU's own picks and scores (widened exactly to
    double), the oracle's capacity step must equal the GPU's counts, slots and
    drops bit for bit, always. End to end, slots and drops are compared at every
    expert that no routing disagreement touched and whose cutoff is not a
    near-tie (the C-th and (C+1)-th oracle scores within NEAR_TIE relative: fp32
    scores may order them differently); such experts are reported.
  * Output: max |y - y_ref| <= tol * max |y_ref| over the tokens whose picks and
    drops agree, tol = 1e-4 (fp32) or 2e-2 (bf16 with fp32 accumulation).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
from sparse_mixture_experts_66_b300 import moe
from sparse_mixture_experts_66_b300.workload import as_f32_numpy, draw

MARGIN = 1e-3
NEAR_TIE = 1e-5
TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_device(inp, device="cuda"):
    return {k: (None if v is None else v.to(device)) for k, v in inp.items()}


def run_gpu(w, inp, flags=0, dev=None, reps=1):
    """moe_forward on the GPU; returns numpy copies of y and the intermediates."""
    cfg = moe.config_of(w, flags)
    dev = dev or to_device(inp)
    ws = moe.Workspace(cfg)
    y = torch.empty_like(dev["x"])
    for _ in range(reps):
        moe.moe_forward(cfg, dev["x"], dev["w_g"], dev["router_bias"], dev["w1"], dev["b1"], dev["w2"], dev["b2"], y,
                        ws.buf)
    ws.status()
    v = ws.views()
    out = {k: t.cpu() for k, t in v.items() if k not in ("x_perm", "h", "y_perm", "y_split")}
    out = {k: (t.float() if t.dtype == torch.bfloat16 else t).numpy() for k, t in out.items()}
    out["y"] = y.float().cpu().numpy().astype(np.float64)
    out["_ws"], out["_cfg"], out["_dev"], out["_y"] = ws, cfg, dev, y
    return out


def oracle_ref(w, inp, flags=0, sel=None):
    orc = O.load()
    return orc.forward(as_f32_numpy(inp["x"]), as_f32_numpy(inp["w_g"]), as_f32_numpy(inp["w1"]),
                       as_f32_numpy(inp["b1"]), as_f32_numpy(inp["w2"]), as_f32_numpy(inp["b2"]), k=w.k,
                       cf=w.capacity_factor, router_bias=as_f32_numpy(inp["router_bias"]), flags=flags, sel=sel)


def margins(logits, k):
    s = -np.sort(-logits, axis=1)
    if k >= logits.shape[1]:
        return np.full(logits.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]


def near_tie_experts(ref, N):
    """Overflowing experts whose C-th and (C+1)-th oracle scores are within NEAR_TIE."""
    out = set()
    C = ref["C"]
    for e in range(N):
        sc = np.sort(ref["score"][ref["idx"] == e])[::-1]
        if len(sc) > C and C > 0 and (sc[C - 1] - sc[C]) <= NEAR_TIE * sc[C - 1]:
            out.add(e)
    return out


def gpu_slots(g):
    """Slot of each pick inside its expert's segment (-1 dropped)."""
    off = g["offsets"]
    slot = np.where(g["row_of"] >= 0, g["row_of"] - off[np.maximum(g["topk_idx"], 0)], -1)
    return slot


def row_align(w):
    """Segment alignment of the permuted buffers: the decode chunk size for
    decode-shaped bf16 batches (T*k <= 64*N: 64 rows, or 32 when
    T*k <= 16*N), else 128."""
    if w.dtype == "bf16" and w.T * w.k <= 64 * w.N:
        return 32 if w.T * w.k <= 16 * w.N else 64
    return 128


def check_layout(g, k, align=128):
    """Structural invariants of the GPU's dispatch outputs."""
    N = g["counts_raw"].shape[0]
    off, ck = g["offsets"], g["counts_kept"]
    assert off[0] == 0
    for e in range(N):
        assert off[e + 1] - off[e] == (ck[e] + align - 1) // align * align, e
    rt, rg, ro = g["row_token"], g["row_gate"], g["row_of"]
    T = ro.shape[0]
    kept = ro >= 0
    assert kept.sum() == ck.sum()
    tt, jj = np.nonzero(kept)
    rows = ro[tt, jj]
    assert len(np.unique(rows)) == len(rows)
    assert np.array_equal(rt[rows], tt)
    assert np.array_equal(rg[rows], g["gate"][tt, jj])
    used = np.zeros(off[N], dtype=bool)
    used[rows] = True
    assert np.all(rt[:off[N]][~used] == -1) and np.all(rg[:off[N]][~used] == 0.0)
    assert np.all(g["topk_idx"] >= 0) and np.all(g["topk_idx"] < N)
    assert T == g["topk_idx"].shape[0]


def compare(w, g, ref, sel=None, tol=None, max_excluded_frac=0.01):
    """Apply the parity rules; returns a report dict (raises on failure)."""
    T, N, k = w.T, w.N, w.k
    tol = TOL[w.dtype] if tol is None else tol
    check_layout(g, k, row_align(w))
    mg = margins(ref["logits"], k)
    low = mg <= MARGIN
    idx_eq = np.all(g["topk_idx"] == ref["idx"], axis=1)
    bad = ~idx_eq & ~low
    assert not bad.any(), f"router picks differ on {bad.sum()} high-margin tokens, e.g. {np.nonzero(bad)[0][:5]}"
    touched = set(np.unique(g["topk_idx"][~idx_eq]).tolist()) | set(np.unique(ref["idx"][~idx_eq]).tolist())
    ties = near_tie_experts(ref, N)
    affected = touched | ties
    ok_e = np.array([e not in affected for e in range(N)])
    for e in range(N):
        if ok_e[e]:
            assert g["counts_raw"][e] == ref["counts_raw"][e], e
            assert g["counts_kept"][e] == ref["counts_kept"][e], e
    # slots and drops on pairs at unaffected experts
    pair_ok = idx_eq[:, None] & ok_e[ref["idx"]]
    gs = gpu_slots(g)
    assert np.array_equal(gs[pair_ok], ref["slot"][pair_ok]), "capacity slots / drops differ"
    # gates and scores, fp32 against fp64
    assert np.allclose(g["gate"][idx_eq], ref["gate"][idx_eq], rtol=2e-5, atol=1e-6)
    assert np.allclose(g["score"][idx_eq], ref["score"][idx_eq], rtol=2e-5, atol=1e-6)
    tok_ok = np.all(pair_ok, axis=1)
    excluded = int((~tok_ok).sum())
    assert excluded <= max(2, max_excluded_frac * T), f"{excluded} tokens excluded"
    rows = np.arange(T) if sel is None else np.asarray(sel)
    yg = g["y"][rows]
    yr = ref["y"]
    m = tok_ok[rows]
    scale = np.max(np.abs(yr[m])) if m.any() else 0.0
    err = np.max(np.abs(yg[m] - yr[m])) if m.any() else 0.0
    assert np.all(np.isfinite(yg)), "non-finite output"
    assert err <= tol * max(scale, 1e-30) or scale == 0.0 and err == 0.0, \
        f"max|y-y_ref| = {err:.3e} > {tol} * {scale:.3e}"
    return dict(low_margin=int(low.sum()), idx_mismatch=int((~idx_eq).sum()), near_tie_experts=sorted(ties),
                excluded_tokens=excluded, max_err=float(err), max_ref=float(scale),
                rel_err=float(err / scale) if scale else 0.0, dropped=int((g["row_of"] < 0).sum()))


def sample_tokens(w, ref, g, n_random=48, seed=0):
    """Tokens for sampled full-size checks: the first and last token, tokens at
    every overflowing expert's cutoff, tokens with one or all picks dropped, and
    random tokens."""
    rng = np.random.default_rng(seed)
    T = w.T
    pick = {0, T - 1}
    C = ref["C"]
    for e in range(w.N):
        m = ref["idx"] == e
        if m.sum() > C:
            tt, jj = np.nonzero(m)
            order = np.lexsort((tt, -ref["score"][tt, jj]))
            for q in order[max(0, C - 2):C + 2]:
                pick.add(int(tt[q]))
    nk = (ref["slot"] >= 0).sum(axis=1)
    for cond in (nk == 0, (nk > 0) & (nk < w.k)):
        cand = np.nonzero(cond)[0]
        if len(cand):
            pick.update(rng.choice(cand, size=min(6, len(cand)), replace=False).tolist())
    pick.update(rng.choice(T, size=min(n_random, T), replace=False).tolist())
    return np.array(sorted(pick), dtype=np.int64)


def full_check(w, inp=None, flags=0, sample=None):
    """GPU forward vs the oracle: all tokens, or a sample of them."""
    inp = inp if inp is not None else draw(w)
    g = run_gpu(w, inp, flags)
    if sample is None:
        ref = oracle_ref(w, inp, flags)
        rep = compare(w, g, ref)
    else:
        ref0 = oracle_ref(w, inp, flags, sel=np.array([0], dtype=np.int64))
        sel = sample_tokens(w, ref0, g, n_random=sample)
        ref = oracle_ref(w, inp, flags, sel=sel)
        rep = compare(w, g, ref, sel=sel)
        rep["sampled_tokens"] = int(len(sel))
    return rep, g, ref, inp


def infinite(cf):
    return cf is None or math.isinf(cf)
