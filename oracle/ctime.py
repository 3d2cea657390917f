"""ctypes loader of the float32 timing baseline (oracle/h3time.c).

Test and measurement infrastructure only: bench.py times the block on the host's
cores (the CPU baseline beside the GPU line), and tests/test_oracle_time.py checks
it against the float64 oracle.  Nothing in the product library imports this
module.  The shared object is built with the host C compiler at -O3 with OpenMP
(without OpenMP, single-threaded, if the compiler lacks it) when it is missing or
older than its source; ``__graft_entry__.build()`` builds it too.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "h3time.c")
LIB = os.path.join(_HERE, "libh3time.so")
CFLAGS = ["-O3", "-std=gnu99", "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        cc = os.environ.get("CC", "gcc")
        r = subprocess.run([cc] + CFLAGS + ["-fopenmp", "-o", LIB, SRC, "-lm"],
                           capture_output=True, text=True)
        if r.returncode != 0:
            subprocess.run([cc] + CFLAGS + ["-o", LIB, SRC, "-lm"], check=True)
    return LIB


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("n_text", "n_audio", "n_video", "hidden", "heads", "head_dim", "mlp_width",
                 "topk", "qk_norm", "rope", "pooled", "swiglu")] + [
        ("eps", ctypes.c_float), ("theta", ctypes.c_float)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_qkvg_t", "b_qkvg", "w_o_t", "b_o", "w1_t", "b1", "w2_t", "b2", "mod",
                 "mod_prefix", "qnorm_w", "knorm_w")]


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        vp = ctypes.c_void_p
        _lib.h3time_scratch_floats.argtypes = [ctypes.POINTER(Shape)]
        _lib.h3time_scratch_floats.restype = ctypes.c_size_t
        _lib.h3time_block.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Weights), vp, vp,
                                      ctypes.c_int, vp]
        _lib.h3time_block.restype = ctypes.c_int
        _lib.h3time_threads.restype = ctypes.c_int
        _lib.h3time_attention.argtypes = [ctypes.POINTER(Shape)] + [vp] * 7
        _lib.h3time_attention.restype = ctypes.c_int
    return _lib


def threads() -> int:
    return int(lib().h3time_threads())


def make_shape(s) -> Shape:
    if getattr(s, "video_grid", None):
        raise ValueError("the float32 baseline tiles video rows as 64-row slices only")
    return Shape(s.n_text, s.n_audio, s.n_video, s.hidden, s.heads, s.head_dim, s.mlp_width,
                 s.topk, int(s.qk_norm), int(s.rope), int(s.pooled), int(s.mlp == "swiglu"),
                 s.rms_eps, s.rope_theta)


def input_major(wts: dict) -> dict:
    """float32 copies of a block's weights with the linear weights transposed to
    [in, out] (the layout h3time.c reads)."""
    f = lambda a: np.ascontiguousarray(np.asarray(a, np.float32))  # noqa: E731
    out = {n: f(np.asarray(wts[n]).T) for n in ("w_qkvg", "w_o", "w1", "w2")}
    for n in ("b_qkvg", "b_o", "b1", "b2", "mod", "qnorm_w", "knorm_w", "mod_prefix"):
        if wts.get(n) is not None:
            out[n] = f(wts[n])
    return out


class Block:
    """One block's float32 inputs held for repeated timed calls."""

    def __init__(self, shape, wts_input_major: dict):
        self.s = make_shape(shape)
        self.shape = shape
        self.w = wts_input_major
        g = self.w.get
        self.cw = Weights(*[(g(n).ctypes.data if g(n) is not None else None) for n in
                            ("w_qkvg", "b_qkvg", "w_o", "b_o", "w1", "b1", "w2", "b2", "mod",
                             "mod_prefix", "qnorm_w", "knorm_w")])
        self.scratch = np.zeros(lib().h3time_scratch_floats(ctypes.byref(self.s)), np.float32)

    def run(self, x: np.ndarray, sample: int = 1, want_idx: bool = False):
        """x: float32 [N, D], updated in place.  Returns the selections when asked."""
        assert x.dtype == np.float32 and x.flags.c_contiguous
        tv = -(-self.shape.n_video // 64)
        idx = np.zeros((self.shape.heads, tv, min(self.shape.topk, tv)), np.int32) \
            if want_idx else None
        rc = lib().h3time_block(ctypes.byref(self.s), ctypes.byref(self.cw), x.ctypes.data,
                                self.scratch.ctypes.data, int(sample),
                                idx.ctypes.data if idx is not None else None)
        if rc != 0:
            raise RuntimeError(f"h3time_block failed ({rc})")
        return idx


class Attention:
    """Router + routed/dense attention + pooled mix alone, float32, for repeated timed
    calls on the same inputs (q, k, v float32 [H, N, d]; g float32 [N, A] or None)."""

    def __init__(self, shape, q, k, v, g=None):
        self.s = make_shape(shape)
        self.shape = shape
        self.q, self.k, self.v = (np.ascontiguousarray(a, np.float32) for a in (q, k, v))
        self.g = None if g is None else np.ascontiguousarray(g, np.float32)
        self.out = np.zeros((shape.n_rows, shape.attn_width), np.float32)
        self.scratch = np.zeros(lib().h3time_scratch_floats(ctypes.byref(self.s)), np.float32)

    def run(self, want_idx: bool = False):
        tv = -(-self.shape.n_video // 64)
        idx = np.zeros((self.shape.heads, tv, min(self.shape.topk, tv)), np.int32) \
            if want_idx else None
        rc = lib().h3time_attention(ctypes.byref(self.s), self.q.ctypes.data, self.k.ctypes.data,
                                    self.v.ctypes.data,
                                    self.g.ctypes.data if self.g is not None else None,
                                    self.out.ctypes.data, self.scratch.ctypes.data,
                                    idx.ctypes.data if idx is not None else None)
        if rc != 0:
            raise RuntimeError(f"h3time_attention failed ({rc})")
        return self.out, idx
