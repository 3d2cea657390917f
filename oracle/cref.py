"""ctypes loader of the plain C reference block (oracle/h3ref.c), test infrastructure only.

The C file restates the block from the pages independently of the numpy oracle
(oracle/h3block.py); the tests run both on the same tiny inputs and require
them to agree.  Nothing in the product library imports this module.  The
shared object is built here with the host C compiler when it is missing or
older than its source (``__graft_entry__.build()`` builds it too).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "h3ref.c")
LIB = os.path.join(_HERE, "libh3ref.so")
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        cc = os.environ.get("CC", "gcc")
        subprocess.run([cc] + CFLAGS + ["-o", LIB, SRC, "-lm"], check=True)
    return LIB


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("n_text", "n_audio", "n_video", "hidden", "heads", "head_dim", "mlp_width",
                 "topk", "qk_norm", "rope", "pooled", "swiglu", "p_bf16")] + [
        ("grid", ctypes.c_int * 3), ("cube", ctypes.c_int * 3),
        ("eps", ctypes.c_double), ("theta", ctypes.c_double)]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_qkvg", "b_qkvg", "w_o", "b_o", "w1", "b1", "w2", "b2", "mod",
                 "mod_prefix", "qnorm_w", "knorm_w")]


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        ip, vp = ctypes.POINTER(ctypes.c_int), ctypes.c_void_p
        _lib.h3ref_tile_count.argtypes = [ctypes.POINTER(Shape)]
        _lib.h3ref_tiles.argtypes = [ctypes.POINTER(Shape), ip, ip]
        _lib.h3ref_attention_layer.argtypes = [ctypes.POINTER(Shape), vp, vp, vp, vp, vp, vp,
                                               vp, vp]
        _lib.h3ref_block_forward.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Weights),
                                             vp, vp, vp, vp]
        _lib.h3ref_bf16.argtypes = [ctypes.c_double]
        _lib.h3ref_bf16.restype = ctypes.c_double
    return _lib


def make_shape(s, p_bf16: bool = False) -> Shape:
    """The C struct of a ``synthetic.BlockShape``."""
    assert s.tile == 64
    c = Shape()
    for n in ("n_text", "n_audio", "n_video", "hidden", "heads", "head_dim", "mlp_width", "topk"):
        setattr(c, n, int(getattr(s, n)))
    c.qk_norm, c.rope, c.pooled = int(s.qk_norm), int(s.rope), int(s.pooled)
    c.swiglu, c.p_bf16 = int(s.mlp == "swiglu"), int(p_bf16)
    if s.video_grid is not None:
        c.grid[:] = list(s.video_grid)
        c.cube[:] = list(s.cube)
    c.eps, c.theta = float(s.rms_eps), float(s.rope_theta)
    return c


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def tiles(s) -> list:
    """Packed row indices of each video tile."""
    cs = make_shape(s)
    L = lib()
    tv = L.h3ref_tile_count(ctypes.byref(cs))
    rows = np.zeros(max(s.n_video, 1), np.int32)
    start = np.zeros(tv + 1, np.int32)
    L.h3ref_tiles(ctypes.byref(cs), rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
                  start.ctypes.data_as(ctypes.POINTER(ctypes.c_int)))
    return [rows[start[t]:start[t + 1]].astype(np.int64) for t in range(tv)]


def attention_layer(s, Q, K, V, G, p_bf16: bool = False) -> dict:
    """Router + attention + pooled branch + gate mix on Q, K, V [H, N, d], G [N, A]."""
    cs = make_shape(s, p_bf16)
    Q, K, V, G = _f64(Q), _f64(K), _f64(V), _f64(G)
    H, N, d = Q.shape
    tv = lib().h3ref_tile_count(ctypes.byref(cs))
    ks = min(s.topk, tv)
    o = np.zeros((N, H * d))
    idx = np.zeros((H, tv, ks), np.int32)
    scores = np.zeros((H, tv, tv))
    pooled = np.zeros((H, tv, d))
    rc = lib().h3ref_attention_layer(ctypes.byref(cs), _p(Q), _p(K), _p(V), _p(G), _p(o),
                                     _p(idx), _p(scores), _p(pooled))
    assert rc == 0
    return {"o_f64": o, "idx": idx, "scores": scores, "pooled": pooled}


def block_forward(x, wts: dict, s, p_bf16: bool = False) -> dict:
    """One block; ``wts`` holds float64 values (keys as in ``synthetic.block_weights``)."""
    cs = make_shape(s, p_bf16)
    x = _f64(x)
    keep = {k: _f64(v) for k, v in wts.items()}
    w = Weights()
    for n, _ in Weights._fields_:
        setattr(w, n, _p(keep.get(n)))
    N, D = x.shape
    x1 = np.zeros((N, D))
    x2 = np.zeros((N, D))
    o = np.zeros((N, s.attn_width))
    rc = lib().h3ref_block_forward(ctypes.byref(cs), ctypes.byref(w), _p(x), _p(x1), _p(x2),
                                   _p(o))
    assert rc == 0
    return {"x1": x1, "x2": x2, "o": o}


def bf16(x: float) -> float:
    return lib().h3ref_bf16(float(x))
