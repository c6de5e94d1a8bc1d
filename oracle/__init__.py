"""ctypes wrapper around the CPU fp64 oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` import this package. The product path never does, and
it shares no code with the CUDA library.

All array arguments are numpy arrays; stored inputs are passed as exact
float32 copies (bf16 and fp32 values are exact in float32) and everything is
computed in double.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "libmoe_oracle.so")

FLAG_RENORM_SURVIVORS = 1
FLAG_IDENTITY_FALLBACK = 2
FLAG_SHARED_EXPERT = 4

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_F64 = ctypes.c_double


def compile_oracle(src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with plain -O2 (no fast-math, no FMA contraction)."""
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC",
           "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _needs_build(src: str, out: str) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src)


class Oracle:
    """One loaded oracle library (the real one, or a test's planted mutant)."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.moe_oracle_gelu.restype = _F64
        lib.moe_oracle_gelu.argtypes = [_F64]
        lib.moe_oracle_router_logits.argtypes = [_I64, _I64, _I32, _P, _P, _P, _P]
        lib.moe_oracle_softmax.argtypes = [_I64, _I32, _P, _P]
        lib.moe_oracle_topk.argtypes = [_I64, _I32, _I32, _P, _P]
        lib.moe_oracle_gates.argtypes = [_I64, _I32, _I32, _P, _P, _P, _P]
        lib.moe_oracle_capacity.restype = _I64
        lib.moe_oracle_capacity.argtypes = [_I64, _I32, _I32, _F64]
        lib.moe_oracle_capacity_assign.argtypes = [_I64, _I32, _I32, _I64, _P, _P, _P, _P, _P]
        lib.moe_oracle_expert_ffn.argtypes = [_I64, _I64, _P, _P, _P, _P, _P, _P, _P]
        lib.moe_oracle_forward.restype = ctypes.c_int
        lib.moe_oracle_forward.argtypes = [_I64, _I64, _I32, _I32, _I64, _F64, ctypes.c_uint32] + [_P] * 11 + [
            _I64] + [_P] * 10
        lib.moe_oracle_router_stats.argtypes = [_I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _P]
        lib.moe_oracle_expert_choice.argtypes = [_I64, _I64, _I32, _I64, _I64] + [_P] * 9
        self.lib = lib

    # -- helpers -------------------------------------------------------------
    @staticmethod
    def _f32(a):
        if a is None:
            return None
        return np.ascontiguousarray(a, dtype=np.float32)

    @staticmethod
    def _ptr(a):
        return None if a is None else a.ctypes.data_as(ctypes.c_void_p)

    # -- stages --------------------------------------------------------------
    def gelu(self, u: float) -> float:
        return self.lib.moe_oracle_gelu(float(u))

    def router_logits(self, x, w_g, router_bias=None):
        x, w_g, rb = self._f32(x), self._f32(w_g), self._f32(router_bias)
        T, d = x.shape
        N = w_g.shape[0]
        out = np.empty((T, N), dtype=np.float64)
        self.lib.moe_oracle_router_logits(T, d, N, self._ptr(x), self._ptr(w_g), self._ptr(rb), self._ptr(out))
        return out

    def softmax(self, logits):
        logits = np.ascontiguousarray(logits, dtype=np.float64)
        T, N = logits.shape
        out = np.empty_like(logits)
        self.lib.moe_oracle_softmax(T, N, self._ptr(logits), self._ptr(out))
        return out

    def topk(self, logits, k):
        logits = np.ascontiguousarray(logits, dtype=np.float64)
        T, N = logits.shape
        idx = np.empty((T, k), dtype=np.int32)
        self.lib.moe_oracle_topk(T, N, k, self._ptr(logits), self._ptr(idx))
        return idx

    def gates(self, probs, idx):
        probs = np.ascontiguousarray(probs, dtype=np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, N = probs.shape
        k = idx.shape[1]
        score = np.empty((T, k), dtype=np.float64)
        gate = np.empty((T, k), dtype=np.float64)
        self.lib.moe_oracle_gates(T, N, k, self._ptr(probs), self._ptr(idx), self._ptr(score), self._ptr(gate))
        return score, gate

    def capacity(self, T, N, k, cf):
        return int(self.lib.moe_oracle_capacity(T, N, k, float(cf)))

    def capacity_assign(self, idx, score, N, C):
        """Returns (counts_raw[N], counts_kept[N], slot[T,k])."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        score = np.ascontiguousarray(score, dtype=np.float64)
        T, k = idx.shape
        cr = np.empty(N, dtype=np.int32)
        ck = np.empty(N, dtype=np.int32)
        slot = np.empty((T, k), dtype=np.int32)
        self.lib.moe_oracle_capacity_assign(T, N, k, int(C), self._ptr(idx), self._ptr(score), self._ptr(cr),
                                            self._ptr(ck), self._ptr(slot))
        return cr, ck, slot

    def expert_ffn_hidden(self, xrow, w1e, b1e, w2e, b2e):
        """(h, out) of one expert on one row: h = GELU(W1 x + b1) (exact erf), out = W2 h + b2."""
        xrow, w1e, b1e, w2e, b2e = (self._f32(a) for a in (xrow, w1e, b1e, w2e, b2e))
        d_ff, d = w1e.shape
        h = np.empty(d_ff, dtype=np.float64)
        out = np.empty(d, dtype=np.float64)
        self.lib.moe_oracle_expert_ffn(d, d_ff, self._ptr(xrow), self._ptr(w1e), self._ptr(b1e), self._ptr(w2e),
                                       self._ptr(b2e), self._ptr(h), self._ptr(out))
        return h, out

    def expert_ffn(self, xrow, w1e, b1e, w2e, b2e):
        xrow, w1e, b1e, w2e, b2e = (self._f32(a) for a in (xrow, w1e, b1e, w2e, b2e))
        d_ff, d = w1e.shape
        h = np.empty(d_ff, dtype=np.float64)
        out = np.empty(d, dtype=np.float64)
        self.lib.moe_oracle_expert_ffn(d, d_ff, self._ptr(xrow), self._ptr(w1e), self._ptr(b1e), self._ptr(w2e),
                                       self._ptr(b2e), self._ptr(h), self._ptr(out))
        return out

    def forward(self, x, w_g, w1, b1, w2, b2, k, cf, router_bias=None, flags=0, sel=None, shared=None):
        """The full layer forward. Returns a dict with logits, probs, idx,
        score, gate, counts_raw, counts_kept, slot, C and y (rows of ``sel``,
        or of all tokens)."""
        x, w_g, w1, b1, w2, b2, rb = (self._f32(a) for a in (x, w_g, w1, b1, w2, b2, router_bias))
        T, d = x.shape
        N, d_ff, _ = w1.shape
        sw = [None] * 4
        if shared is not None:
            flags |= FLAG_SHARED_EXPERT
            sw = [self._f32(a) for a in shared]
        sel_arr = None if sel is None else np.ascontiguousarray(sel, dtype=np.int64)
        n_sel = T if sel_arr is None else sel_arr.shape[0]
        logits = np.empty((T, N), dtype=np.float64)
        probs = np.empty((T, N), dtype=np.float64)
        idx = np.empty((T, k), dtype=np.int32)
        score = np.empty((T, k), dtype=np.float64)
        gate = np.empty((T, k), dtype=np.float64)
        cr = np.empty(N, dtype=np.int32)
        ck = np.empty(N, dtype=np.int32)
        slot = np.empty((T, k), dtype=np.int32)
        y = np.empty((n_sel, d), dtype=np.float64)
        rc = self.lib.moe_oracle_forward(
            T, d, N, k, d_ff, float(cf), flags, self._ptr(x), self._ptr(w_g), self._ptr(rb), self._ptr(w1),
            self._ptr(b1), self._ptr(w2), self._ptr(b2), *[self._ptr(a) for a in sw], n_sel, self._ptr(sel_arr),
            self._ptr(logits), self._ptr(probs), self._ptr(idx), self._ptr(score), self._ptr(gate), self._ptr(cr),
            self._ptr(ck), self._ptr(slot), self._ptr(y))
        if rc != 0:
            raise ValueError("oracle rejected the sizes")
        return dict(logits=logits, probs=probs, idx=idx, score=score, gate=gate, counts_raw=cr, counts_kept=ck,
                    slot=slot, y=y, C=self.capacity(T, N, k, cf))

    def router_stats(self, logits, probs, idx):
        logits = np.ascontiguousarray(logits, dtype=np.float64)
        probs = np.ascontiguousarray(probs, dtype=np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, N = logits.shape
        k = idx.shape[1]
        f = np.empty(N, dtype=np.float64)
        P = np.empty(N, dtype=np.float64)
        aux = ctypes.c_double()
        z = ctypes.c_double()
        self.lib.moe_oracle_router_stats(T, N, k, self._ptr(logits), self._ptr(probs), self._ptr(idx), self._ptr(f),
                                         self._ptr(P), ctypes.byref(aux), ctypes.byref(z))
        return f, P, aux.value, z.value

    def expert_choice(self, x, probs, w1, b1, w2, b2, C):
        x, w1, b1, w2, b2 = (self._f32(a) for a in (x, w1, b1, w2, b2))
        probs = np.ascontiguousarray(probs, dtype=np.float64)
        T, d = x.shape
        N, d_ff, _ = w1.shape
        taken = np.empty((T, N), dtype=np.int32)
        counts = np.empty(N, dtype=np.int32)
        y = np.empty((T, d), dtype=np.float64)
        self.lib.moe_oracle_expert_choice(T, d, N, d_ff, int(C), self._ptr(x), self._ptr(probs), self._ptr(w1),
                                          self._ptr(b1), self._ptr(w2), self._ptr(b2), self._ptr(taken),
                                          self._ptr(counts), self._ptr(y))
        return taken, counts, y


_default = None


def load() -> Oracle:
    """The oracle built from ``moe_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        if _needs_build(_SRC, _LIB):
            compile_oracle()
        _default = Oracle(_LIB)
    return _default
