"""Thin ctypes binding of the C ABI in ``include/moe.h``.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libmoe.so``. torch supplies device memory and streams. There is no CPU
fallback: if the library is missing, or a tensor is not on a CUDA device, the
call raises.

The functions keep the C names (``moe_route``, ``moe_dispatch``,
``moe_expert_ffn``, ``moe_combine``, ``moe_forward`` ...) and take torch
tensors where the C ABI takes device pointers.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_BOUNDS = 6
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_BOUNDS"}

MOE_DT_F32 = 0
MOE_DT_BF16 = 1
MOE_FLAG_RENORM_SURVIVORS = 1
MOE_FLAG_IDENTITY_FALLBACK = 2
MOE_FLAG_SHARED_EXPERT = 4
MOE_FLAG_ROUTER_STATS = 8
MOE_FLAG_EXPERT_CHOICE = 16

_DT_CODE = {torch.float32: MOE_DT_F32, torch.bfloat16: MOE_DT_BF16}
_DT_TORCH = {MOE_DT_F32: torch.float32, MOE_DT_BF16: torch.bfloat16}


class MoeError(RuntimeError):
    def __init__(self, status: int, text: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {text}")
        self.status = status


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("d_ff", ctypes.c_int64), ("N", ctypes.c_int32),
                ("k", ctypes.c_int32), ("capacity_factor", ctypes.c_double), ("dtype", ctypes.c_int),
                ("flags", ctypes.c_uint32)]

    @property
    def torch_dtype(self):
        return _DT_TORCH[self.dtype]


class MoeWorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "topk_idx", "gate", "score", "counts_raw", "counts_kept", "offsets", "sel_thr", "sel_eq",
        "row_of", "row_token", "row_gate", "x_perm", "h", "y_perm", "y_split", "ffn_sync", "probs", "lse", "shared_offsets", "h_shared", "y_shared",
        "shared_sync", "total")] + [
        ("rows", ctypes.c_int64), ("capacity", ctypes.c_int64)]


# Names and argument kinds of every symbol the header declares.
# kinds: C = config*, P = device pointer, S = stream, L = layout*, I = int64.
SIGNATURES = {
    "moe_version": ([], ctypes.c_char_p),
    "moe_last_error": ([], ctypes.c_char_p),
    "moe_capacity": (["C"], ctypes.c_int64),
    "moe_get_workspace_layout": (["C", "L"], ctypes.c_int),
    "moe_workspace_bytes": (["C"], ctypes.c_size_t),
    "moe_workspace_init": (["C", "P", "S"], ctypes.c_int),
    "moe_get_device_status": (["P", "S"], ctypes.c_int),
    "moe_route": (["C"] + ["P"] * 7 + ["S"], ctypes.c_int),
    "moe_dispatch": (["C"] + ["P"] * 12 + ["S"], ctypes.c_int),
    "moe_expert_ffn": (["C"] + ["P"] * 10 + ["S"], ctypes.c_int),
    "moe_combine": (["C"] + ["P"] * 6 + ["S"], ctypes.c_int),
    "moe_forward": (["C"] + ["P"] * 9 + ["S"], ctypes.c_int),
    "moe_forward_noalloc": (["C"] + ["P"] * 8 + ["S"], ctypes.c_int),
    "moe_router_stats": (["C"] + ["P"] * 5 + ["S"], ctypes.c_int),
    "moe_shared_expert": (["C"] + ["P"] * 6 + ["S"], ctypes.c_int),
    "moe_forward_shared": (["C"] + ["P"] * 13 + ["S"], ctypes.c_int),
    "moe_selftest_wait_timeout": (["P", "I", "P", "S"], ctypes.c_int),
}
_KIND = {"C": ctypes.POINTER(MoeConfig), "P": ctypes.c_void_p, "S": ctypes.c_void_p,
         "L": ctypes.POINTER(MoeWorkspaceLayout), "I": ctypes.c_int64}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libmoe.so not found at {path}: build it with "
                          "`python -m sparse_mixture_experts_66_b300.build`")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = [_KIND[a] for a in args]
        fn.restype = res
    _lib = lib
    return lib


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, moe_last_error())


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("tensor is not on a CUDA device: the library has no CPU path")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_config(T, d, d_ff, N, k, capacity_factor=math.inf, dtype=torch.bfloat16, flags=0) -> MoeConfig:
    if isinstance(dtype, str):
        dtype = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    return MoeConfig(int(T), int(d), int(d_ff), int(N), int(k), float(capacity_factor), _DT_CODE[dtype],
                     int(flags))


def config_of(workload, flags=0) -> MoeConfig:
    """Config of a :class:`workload.Workload`."""
    return make_config(workload.T, workload.d, workload.d_ff, workload.N, workload.k, workload.capacity_factor,
                       workload.dtype, flags)


# ---- sizing -----------------------------------------------------------------
def moe_version() -> str:
    return load().moe_version().decode()


def moe_last_error() -> str:
    return load().moe_last_error().decode()


def moe_capacity(cfg: MoeConfig) -> int:
    return int(load().moe_capacity(ctypes.byref(cfg)))


def moe_get_workspace_layout(cfg: MoeConfig) -> MoeWorkspaceLayout:
    out = MoeWorkspaceLayout()
    _check(load().moe_get_workspace_layout(ctypes.byref(cfg), ctypes.byref(out)))
    return out


def moe_workspace_bytes(cfg: MoeConfig) -> int:
    return int(load().moe_workspace_bytes(ctypes.byref(cfg)))


def moe_workspace_init(cfg, ws, stream=None):
    _check(load().moe_workspace_init(ctypes.byref(cfg), _ptr(ws), _stream(stream)))


def moe_get_device_status(ws, stream=None):
    _check(load().moe_get_device_status(_ptr(ws), _stream(stream)))


# ---- the five stage calls ---------------------------------------------------
def moe_route(cfg, x, w_g, router_bias, topk_idx, gate, score, ws, stream=None):
    _check(load().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(w_g), _ptr(router_bias), _ptr(topk_idx), _ptr(gate),
                            _ptr(score), _ptr(ws), _stream(stream)))


def moe_router_stats(cfg, ws, counts_raw, f, P, losses, stream=None):
    _check(load().moe_router_stats(ctypes.byref(cfg), _ptr(ws), _ptr(counts_raw), _ptr(f), _ptr(P), _ptr(losses),
                                   _stream(stream)))


def moe_dispatch(cfg, x, topk_idx, gate, score, counts_raw, counts_kept, offsets, row_of, row_token, row_gate,
                 x_perm, ws, stream=None):
    _check(load().moe_dispatch(ctypes.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(gate), _ptr(score),
                               _ptr(counts_raw), _ptr(counts_kept), _ptr(offsets), _ptr(row_of), _ptr(row_token),
                               _ptr(row_gate), _ptr(x_perm), _ptr(ws), _stream(stream)))


def moe_expert_ffn(cfg, x_perm, offsets, w1, b1, w2, b2, row_gate, h, y_perm, ws, stream=None):
    _check(load().moe_expert_ffn(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(w1), _ptr(b1), _ptr(w2),
                                 _ptr(b2), _ptr(row_gate), _ptr(h), _ptr(y_perm), _ptr(ws), _stream(stream)))


def moe_combine(cfg, y_perm, row_of, gate, x, y, ws, stream=None):
    _check(load().moe_combine(ctypes.byref(cfg), _ptr(y_perm), _ptr(row_of), _ptr(gate), _ptr(x), _ptr(y),
                              _ptr(ws), _stream(stream)))


def moe_forward(cfg, x, w_g, router_bias, w1, b1, w2, b2, y, ws, stream=None):
    _check(load().moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(w_g), _ptr(router_bias), _ptr(w1), _ptr(b1),
                              _ptr(w2), _ptr(b2), _ptr(y), _ptr(ws), _stream(stream)))


def moe_shared_expert(cfg, x, sw1, sb1, sw2, sb2, ws, stream=None):
    _check(load().moe_shared_expert(ctypes.byref(cfg), _ptr(x), _ptr(sw1), _ptr(sb1), _ptr(sw2), _ptr(sb2), _ptr(ws),
                                    _stream(stream)))


def moe_forward_shared(cfg, x, w_g, router_bias, w1, b1, w2, b2, sw1, sb1, sw2, sb2, y, ws, stream=None):
    _check(load().moe_forward_shared(ctypes.byref(cfg), _ptr(x), _ptr(w_g), _ptr(router_bias), _ptr(w1), _ptr(b1),
                                     _ptr(w2), _ptr(b2), _ptr(sw1), _ptr(sb1), _ptr(sw2), _ptr(sb2), _ptr(y),
                                     _ptr(ws), _stream(stream)))


def moe_forward_noalloc(cfg, x, w_g, router_bias, w1, b1, w2, b2, y, stream=None):
    """moe_forward without a workspace, for callers that cannot allocate device
    memory: the library's fixed 32 MiB device scratch array is used instead.
    Larger configs raise MOE_ERR_WORKSPACE; calls that overlap on the GPU race
    on the shared array."""
    _check(load().moe_forward_noalloc(ctypes.byref(cfg), _ptr(x), _ptr(w_g), _ptr(router_bias), _ptr(w1), _ptr(b1),
                                      _ptr(w2), _ptr(b2), _ptr(y), _stream(stream)))


def moe_selftest_wait_timeout(ws, limit_ns, result, stream=None):
    """Run the bounded-wait self-test: both waits must give up after limit_ns
    and leave MOE_ERR_TIMEOUT in ws's status word; result is a device int32[8]."""
    _check(load().moe_selftest_wait_timeout(_ptr(ws), ctypes.c_int64(int(limit_ns)), _ptr(result), _stream(stream)))


# ---- workspace helper -------------------------------------------------------
class Workspace:
    """A device workspace of one config, with typed views of its buffers."""

    def __init__(self, cfg: MoeConfig, device="cuda", stream=None):
        self.cfg = cfg
        self.layout = moe_get_workspace_layout(cfg)
        self.buf = torch.empty(self.layout.total, dtype=torch.uint8, device=device)
        moe_workspace_init(cfg, self.buf, stream)

    def view(self, name: str, dtype, shape):
        off = getattr(self.layout, name)
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return self.buf[off:off + nbytes].view(dtype).view(*shape)

    def views(self):
        c, L = self.cfg, self.layout
        T, k, N, R = c.T, c.k, c.N, L.rows
        if c.flags & MOE_FLAG_EXPERT_CHOICE:
            k = N  # every token offers itself to every expert
        dt = c.torch_dtype
        return dict(
            topk_idx=self.view("topk_idx", torch.int32, (T, k)), gate=self.view("gate", torch.float32, (T, k)),
            score=self.view("score", torch.float32, (T, k)), counts_raw=self.view("counts_raw", torch.int32, (N,)),
            counts_kept=self.view("counts_kept", torch.int32, (N,)),
            offsets=self.view("offsets", torch.int32, (N + 1,)), row_of=self.view("row_of", torch.int32, (T, k)),
            row_token=self.view("row_token", torch.int32, (R,)), row_gate=self.view("row_gate", torch.float32, (R,)),
            x_perm=self.view("x_perm", dt, (R, c.d)), h=self.view("h", dt, (R, c.d_ff)),
            y_perm=self.view("y_perm", dt, (R, c.d)),
            y_split=self.view("y_split", torch.float32, (self.splits - 1, R, c.d)),
            probs=self.view("probs", torch.float32,
                            (T, N) if c.flags & (MOE_FLAG_ROUTER_STATS | MOE_FLAG_EXPERT_CHOICE) else (0, N)),
            lse=self.view("lse", torch.float32,
                          (T,) if c.flags & (MOE_FLAG_ROUTER_STATS | MOE_FLAG_EXPERT_CHOICE) else (0,)),
            y_shared=self.view("y_shared", dt,
                               ((T + 127) // 128 * 128, c.d) if c.flags & MOE_FLAG_SHARED_EXPERT else (0, c.d)))

    @property
    def splits(self):
        """K slices of the decode-mode second GEMM (1 outside decode mode)."""
        L = self.layout
        return 1 + (L.ffn_sync - L.y_split) // (L.rows * self.cfg.d * 4)

    def status(self, stream=None):
        moe_get_device_status(self.buf, stream)


def forward(cfg, x, w_g, w1, b1, w2, b2, router_bias=None, ws: Workspace | None = None, y=None, stream=None):
    """One layer forward on device tensors; returns (y, workspace)."""
    if ws is None:
        ws = Workspace(cfg, device=x.device, stream=stream)
    if y is None:
        y = torch.empty_like(x)
    moe_forward(cfg, x, w_g, router_bias, w1, b1, w2, b2, y, ws.buf, stream)
    return y, ws
