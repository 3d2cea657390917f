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
        i, d = ctypes.c_int, ctypes.c_double
        _lib.h3ref_euler.argtypes = [vp, vp, i, i, i, d, d, vp]
        _lib.h3ref_euler.restype = None
        _lib.h3ref_extrapolate.argtypes = [vp, vp, i, i, i, vp, vp, vp]
        _lib.h3ref_extrapolate.restype = None
        _lib.h3ref_patch_in.argtypes = [vp, i, i, vp, vp, i, vp]
        _lib.h3ref_patch_in.restype = None
        _lib.h3ref_output_head.argtypes = [vp, i, i, vp, vp, vp, i, d, vp]
        _lib.h3ref_output_head.restype = None
        _lib.h3ref_token_pool.argtypes = [vp, i, i, i, i, i, vp, vp]
        _lib.h3ref_token_pool.restype = None
        _lib.h3ref_token_restore.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
        _lib.h3ref_token_restore.restype = None
        _lib.h3ref_thin_layers.argtypes = [vp, i, i, i, vp]
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


def euler(z, v, dt, dt_prefix=None, n_prefix=0):
    z, v = _f64(z), _f64(v)
    N, D = z.shape
    out = np.zeros((N, D))
    lib().h3ref_euler(_p(z), _p(v), N, D, n_prefix, float(dt),
                      float(dt if dt_prefix is None else dt_prefix), _p(out))
    return out


def extrapolate(va, vb, sig_video, sig_prefix=None, n_prefix=0):
    va, vb = _f64(va), _f64(vb)
    N, D = va.shape
    sv = _f64(np.asarray(sig_video))
    sp = _f64(np.asarray(sig_video if sig_prefix is None else sig_prefix))
    out = np.zeros((N, D))
    lib().h3ref_extrapolate(_p(va), _p(vb), N, D, n_prefix, _p(sv), _p(sp), _p(out))
    return out


def patch_in(z, w_in, b_in):
    z, w_in, b_in = _f64(z), _f64(w_in), _f64(b_in)
    rows, c = z.shape
    D = w_in.shape[1]
    x = np.zeros((rows, D))
    lib().h3ref_patch_in(_p(z), rows, c, _p(w_in), _p(b_in), D, _p(x))
    return x


def output_head(x, mod2, w_out, b_out, eps=1e-6):
    x, mod2, w_out, b_out = _f64(x), _f64(mod2), _f64(w_out), _f64(b_out)
    rows, D = x.shape
    c = w_out.shape[0]
    v = np.zeros((rows, c))
    lib().h3ref_output_head(_p(x), rows, D, _p(mod2), _p(w_out), _p(b_out), c, float(eps), _p(v))
    return v


def token_pool(x, s):
    x = _f64(x)
    T, Hg, W = s.video_grid
    Wr = (W + 1) // 2
    D = x.shape[1]
    xr = np.zeros((s.n_prefix + T * Hg * Wr, D))
    base = np.zeros((T * Hg * Wr, D))
    lib().h3ref_token_pool(_p(x), s.n_prefix, T, Hg, W, D, _p(xr), _p(base))
    return xr, base


def token_restore(bypass, x_r, base, s):
    bypass, x_r, base = _f64(bypass), _f64(x_r), _f64(base)
    T, Hg, W = s.video_grid
    out = np.zeros(bypass.shape)
    lib().h3ref_token_restore(_p(bypass), _p(x_r), _p(base), s.n_prefix, T, Hg, W,
                              bypass.shape[1], _p(out))
    return out


def thin_layers(mods, keep):
    m = _f64(np.asarray(mods))
    L, _, D = m.shape
    kept = np.zeros(max(L, 1), np.int32)
    n = lib().h3ref_thin_layers(_p(m), L, D, keep, _p(kept))
    assert n >= 0
    return kept[:n].tolist()
