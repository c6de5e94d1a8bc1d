"""The C-ABI library loads and exports every declared symbol; host-side logic (CPU only)."""
import ctypes
import math
import os
import re

import pytest

import oracle as O
from sparse_mixture_experts_66_b300 import moe
from sparse_mixture_experts_66_b300.workload import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = moe.load()
    declared = header_functions()
    assert len(declared) >= 12
    for name in declared:
        assert hasattr(lib, name), name
    # the binding knows the same set, under the same names
    assert sorted(moe.SIGNATURES) == declared
    for name in declared:
        assert callable(getattr(moe, name))


def header_prototypes():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(moe_[a-z_]+)\s*\(([^)]*)\)\s*;", text):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_argument_counts_match_the_header():
    protos = header_prototypes()
    assert sorted(protos) == header_functions()
    for name, n in protos.items():
        assert len(moe.SIGNATURES[name][0]) == n, name


def test_version():
    assert "sm_103a" in moe.moe_version()


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_capacity_matches_oracle_formula(name):
    w = WORKLOADS[name]
    cfg = moe.config_of(w)
    assert moe.moe_capacity(cfg) == O.load().capacity(w.T, w.N, w.k, w.capacity_factor)


def test_capacity_edge_values():
    for T, N, k, cf, C in [(5, 4, 2, 0.8, 2), (10, 3, 1, 1.0, 4), (7, 2, 2, 100.0, 7), (100, 8, 2, math.inf, 100),
                           (100, 8, 2, 0.0, 100), (100, 8, 2, -1.0, 100), (1, 1, 1, 1.0, 1)]:
        cfg = moe.make_config(T, 8, 8, N, k, cf)
        assert moe.moe_capacity(cfg) == C


def test_workspace_layout_is_aligned_and_sized():
    for w in WORKLOADS.values():
        cfg = moe.config_of(w)
        L = moe.moe_get_workspace_layout(cfg)
        S = min(w.T * w.k, w.N * L.capacity)
        assert L.rows == (S + 127 * w.N) // 128 * 128
        offs = [getattr(L, f) for f, _ in moe.MoeWorkspaceLayout._fields_[:23]]
        assert all(o % 256 == 0 for o in offs)
        assert offs == sorted(offs)
        es = 2 if w.dtype == "bf16" else 4
        assert L.total >= L.y_perm + L.rows * w.d * es
        assert L.h - L.x_perm >= L.rows * w.d * es
        assert moe.moe_workspace_bytes(cfg) == L.total


@pytest.mark.parametrize("field,value", [("T", 0), ("N", 0), ("N", 257), ("k", 0), ("k", 9), ("d", 12),
                                         ("d_ff", 4), ("dtype", 7), ("flags", 32)])
def test_invalid_config_rejected_on_host(field, value):
    cfg = moe.make_config(64, 64, 64, 8, 2, 1.25)
    setattr(cfg, field, value)
    assert moe.moe_workspace_bytes(cfg) == 0
    assert moe.moe_capacity(cfg) == -1
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_get_workspace_layout(cfg)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG


def test_k_larger_than_N_rejected():
    cfg = moe.make_config(64, 64, 64, 2, 3, 1.25)
    assert moe.moe_workspace_bytes(cfg) == 0


def test_null_and_misaligned_pointers_rejected_before_any_launch():
    lib = moe.load()
    cfg = moe.make_config(64, 64, 64, 8, 2, 1.25)
    P = ctypes.c_void_p
    st = lib.moe_route(ctypes.byref(cfg), None, None, None, None, None, None, None, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    assert b"NULL" in lib.moe_last_error()
    # misaligned (never dereferenced: rejected on the host)
    bad = P(0x1003)
    st = lib.moe_forward(ctypes.byref(cfg), bad, bad, None, bad, bad, bad, bad, bad, bad, None)
    assert st == moe.MOE_ERR_INVALID_ARG
    assert b"aligned" in lib.moe_last_error()
    st = lib.moe_combine(ctypes.byref(cfg), None, None, None, None, None, None, None)
    assert st == moe.MOE_ERR_INVALID_ARG


def test_flag_variants_need_their_inputs():
    lib = moe.load()
    cfg = moe.make_config(64, 64, 64, 8, 2, 1.25, flags=moe.MOE_FLAG_RENORM_SURVIVORS)
    p = ctypes.c_void_p(0x1000)
    st = lib.moe_combine(ctypes.byref(cfg), p, p, None, None, p, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"gate" in lib.moe_last_error()
    cfg.flags = moe.MOE_FLAG_IDENTITY_FALLBACK
    st = lib.moe_combine(ctypes.byref(cfg), p, p, None, None, p, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"x" in lib.moe_last_error()


def test_router_stats_need_their_flag_and_buffers():
    """moe_router_stats reads what the router stored under MOE_FLAG_ROUTER_STATS;
    without the flag (or with a missing output) it is rejected on the host."""
    lib = moe.load()
    p = ctypes.c_void_p(0x1000)
    cfg = moe.make_config(64, 64, 64, 8, 2, 1.25)
    st = lib.moe_router_stats(ctypes.byref(cfg), p, p, p, p, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"MOE_FLAG_ROUTER_STATS" in lib.moe_last_error()
    cfg.flags = moe.MOE_FLAG_ROUTER_STATS
    st = lib.moe_router_stats(ctypes.byref(cfg), p, p, p, None, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"NULL" in lib.moe_last_error()
    # the statistics buffers exist in the workspace only under the flag
    L0 = moe.moe_get_workspace_layout(moe.make_config(64, 64, 64, 8, 2, 1.25))
    L1 = moe.moe_get_workspace_layout(cfg)
    assert L0.lse == L0.probs and L1.lse - L1.probs >= 64 * 8 * 4 and L1.total - L1.lse >= 64 * 4


def test_binding_refuses_cpu_tensors():
    import torch
    cfg = moe.make_config(8, 8, 8, 2, 1, 1.0, dtype=torch.float32)
    x = torch.zeros(8, 8)
    with pytest.raises(ValueError, match="CUDA"):
        moe.moe_forward(cfg, x, x, None, x, x, x, x, x, x, stream=None)


def test_shared_expert_entry_points_check_their_flag():
    lib = moe.load()
    p = ctypes.c_void_p(0x1000)
    cfg = moe.make_config(64, 64, 64, 8, 2, 1.25)
    st = lib.moe_shared_expert(ctypes.byref(cfg), p, p, p, p, p, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"MOE_FLAG_SHARED_EXPERT" in lib.moe_last_error()
    st = lib.moe_forward_shared(ctypes.byref(cfg), *([p] * 13), None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"MOE_FLAG_SHARED_EXPERT" in lib.moe_last_error()
    cfg.flags = moe.MOE_FLAG_SHARED_EXPERT
    # moe_forward has no shared weights to run it with
    st = lib.moe_forward(ctypes.byref(cfg), p, p, None, p, p, p, p, p, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"moe_forward_shared" in lib.moe_last_error()
    L = moe.moe_get_workspace_layout(cfg)
    assert L.y_shared - L.h_shared >= 128 * 64 * 2 and L.shared_sync - L.y_shared >= 128 * 64 * 2


def test_expert_choice_flag_rules():
    lib = moe.load()
    p = ctypes.c_void_p(0x1000)
    cfg = moe.make_config(64, 64, 64, 8, 2, 1.25, flags=moe.MOE_FLAG_EXPERT_CHOICE | moe.MOE_FLAG_RENORM_SURVIVORS)
    assert lib.moe_capacity(ctypes.byref(cfg)) == -1  # expert choice combines only with the statistics flag
    cfg.flags = moe.MOE_FLAG_EXPERT_CHOICE
    # the stage calls do not run expert choice
    st = lib.moe_route(ctypes.byref(cfg), p, p, None, p, p, p, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG and b"expert-choice" in lib.moe_last_error()
    # every token offers itself to every expert: the row maps are [T, N]
    L = moe.moe_get_workspace_layout(cfg)
    assert L.row_token - L.row_of >= 64 * 8 * 4
    C = moe.moe_capacity(cfg)
    assert C == 20 and L.rows >= 8 * 128  # C = ceil(1.25 * 64 * 2 / 8)


def test_selftest_checks_its_limit_before_touching_the_device():
    """The wait self-test validates its arguments on the host: a limit outside
    [1 us, 1 s] returns MOE_ERR_INVALID_ARG before anything is enqueued (so
    this runs without a GPU, on placeholder aligned pointers)."""
    lib = moe.load()
    for bad in (0, 999, 1_000_000_001):
        st = lib.moe_selftest_wait_timeout(ctypes.c_void_p(256), ctypes.c_int64(bad), ctypes.c_void_p(512), None)
        assert st == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_selftest_wait_timeout(None, ctypes.c_int64(10_000), ctypes.c_void_p(512), None) == \
        moe.MOE_ERR_INVALID_ARG
