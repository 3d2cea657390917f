"""ctypes binding of libh3dit.so: argument marshalling only.

Every function here converts its arguments (torch tensors on the GPU, numpy
arrays on the host, shape objects) into the plain pointers and structs of
``include/h3dit.h`` and calls the C entry point of the same name.  No step of
the computation runs here; if the library is missing the import fails.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libh3dit.so")

H3DIT_QK_NORM = 0x1
H3DIT_ROPE = 0x2
H3DIT_POOLED = 0x4
H3DIT_SWIGLU = 0x8
H3DIT_TOKEN_REDUCTION = 0x10
H3DIT_KEEP_INTERMEDIATES = 0x20
H3DIT_WS_ABSENT = (1 << (8 * ctypes.sizeof(ctypes.c_size_t))) - 1

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported or inconsistent shape",
          3: "pointer not 16-byte aligned", 4: "workspace missing or too small",
          5: "CUDA call failed", 6: "a kernel wait timed out",
          7: "unsupported device or feature"}


class H3DitError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {STATUS.get(code, code)} (status {code})")
        self.code = code


class Shape(ctypes.Structure):
    _fields_ = [("n_text", ctypes.c_int), ("n_audio", ctypes.c_int), ("n_video", ctypes.c_int),
                ("hidden", ctypes.c_int), ("heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("attn_width", ctypes.c_int), ("mlp_width", ctypes.c_int), ("tile", ctypes.c_int),
                ("topk", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("flags", ctypes.c_uint),
                ("video_t", ctypes.c_int), ("video_h", ctypes.c_int), ("video_w", ctypes.c_int),
                ("cube_t", ctypes.c_int), ("cube_h", ctypes.c_int), ("cube_w", ctypes.c_int)]


class BlockWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_qkvg", "b_qkvg", "w_o", "b_o", "w1", "b1", "w2", "b2", "mod",
                 "qnorm_w", "knorm_w", "mod_prefix")]


class Schedule(ctypes.Structure):
    _fields_ = [("sigma_i", ctypes.c_float), ("sigma_a", ctypes.c_float),
                ("sigma_b", ctypes.c_float), ("dt", ctypes.c_float)]


class Ends(ctypes.Structure):
    _fields_ = [("c_video", ctypes.c_int), ("c_audio", ctypes.c_int)] + [
        (n, ctypes.c_void_p) for n in
        ("w_in_video", "b_in_video", "w_in_audio", "b_in_audio", "w_out_video", "b_out_video",
         "w_out_audio", "b_out_audio", "mod_out_video", "mod_out_audio", "text")]


class Reduction(ctypes.Structure):
    _fields_ = [("first", ctypes.c_int), ("last", ctypes.c_int)]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "q", "k", "v", "g", "o", "u", "h", "x1", "means", "scores", "idx",
                 "pooled", "total")]


H3DIT_PASS_FRESH, H3DIT_PASS_EXTRAPOLATE, H3DIT_PASS_CORE_REUSE = 0, 1, 2

_lib = None

# (name, restype, argtypes)
_SIGS = [
    ("h3dit_workspace_bytes", ctypes.c_size_t, [ctypes.POINTER(Shape)]),
    ("h3dit_check_shape", ctypes.c_int, [ctypes.POINTER(Shape)]),
    ("h3dit_block_forward", ctypes.c_int,
     [ctypes.POINTER(Shape), ctypes.POINTER(BlockWeights), ctypes.c_void_p, ctypes.c_void_p,
      ctypes.c_size_t, ctypes.c_void_p]),
    ("h3dit_routed_attention", ctypes.c_int,
     [ctypes.POINTER(Shape)] + [ctypes.c_void_p] * 8 + [ctypes.c_void_p, ctypes.c_size_t,
                                                        ctypes.c_void_p]),
    ("h3dit_routed_attention_static", ctypes.c_int,
     [ctypes.POINTER(Shape)] + [ctypes.c_void_p] * 8 + [ctypes.c_void_p]),
    ("h3dit_routed_attention_static_status", ctypes.c_int, [ctypes.c_void_p]),
    ("h3dit_get_workspace_layout", ctypes.c_int,
     [ctypes.POINTER(Shape), ctypes.POINTER(WorkspaceLayout)]),
    ("h3dit_denoise_step", ctypes.c_int,
     [ctypes.POINTER(Shape), ctypes.POINTER(BlockWeights), ctypes.POINTER(ctypes.c_int),
      ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(Schedule),
      ctypes.POINTER(Schedule), ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
      ctypes.c_void_p]),
    ("h3dit_sample_step", ctypes.c_int,
     [ctypes.POINTER(Shape), ctypes.POINTER(Ends), ctypes.POINTER(BlockWeights),
      ctypes.POINTER(ctypes.c_int), ctypes.c_int] + [ctypes.c_void_p] * 5
     + [ctypes.POINTER(Reduction), ctypes.c_int, ctypes.POINTER(Schedule),
        ctypes.POINTER(Schedule), ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t,
        ctypes.c_void_p]),
    ("h3dit_select_blocks", ctypes.c_int,
     [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    ("h3dit_tile_spans", ctypes.c_int,
     [ctypes.POINTER(Shape), ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int)]),
    ("h3dit_video_order", ctypes.c_int, [ctypes.POINTER(Shape), ctypes.c_void_p]),
    ("h3dit_linear", ctypes.c_int,
     [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
      ctypes.c_int, ctypes.c_int, ctypes.c_void_p]),
    ("h3dit_sync_status", ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    ("h3dit_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("h3dit_version", ctypes.c_char_p, []),
    ("h3dit_profile_begin", ctypes.c_int, [ctypes.c_int]),
    ("h3dit_profile_end", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]),
    ("h3dit_launch_count", ctypes.c_ulonglong, []),
    ("h3dit_gemm_cta_pairs", ctypes.c_int, [ctypes.c_int]),
    ("h3dit_selftest_timeout", ctypes.c_int,
     [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]),
]

STAGES = ["norm1", "qkvg", "router", "attention", "out_proj", "norm2", "fc1", "fc2", "sampler"]

EXPORTED = [s[0] for s in _SIGS]


def lib() -> ctypes.CDLL:
    """Loads libh3dit.so from the package directory (raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in _SIGS:
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(fn: str, code: int):
    if code != 0:
        raise H3DitError(fn, code)


def make_shape(s, flags=None) -> Shape:
    """ctypes shape from any object with the BlockShape attributes."""
    if flags is None:
        flags = ((H3DIT_QK_NORM if getattr(s, "qk_norm", False) else 0)
                 | (H3DIT_ROPE if getattr(s, "rope", False) else 0)
                 | (H3DIT_POOLED if getattr(s, "pooled", False) else 0)
                 | (H3DIT_SWIGLU if getattr(s, "mlp", "gelu") == "swiglu" else 0)
                 | (H3DIT_TOKEN_REDUCTION if getattr(s, "token_reduction", False) else 0))
    grid = getattr(s, "video_grid", None) or (0, 0, 0)
    cube = getattr(s, "cube", None) if getattr(s, "video_grid", None) else None
    cube = cube or (0, 0, 0)
    return Shape(s.n_text, s.n_audio, s.n_video, s.hidden, s.heads, s.head_dim, s.attn_width,
                 s.mlp_width, s.tile, s.topk, s.rms_eps, s.rope_theta, flags, *grid, *cube)


def attn_shape(s, flags=None) -> Shape:
    """Shape for h3dit_routed_attention alone (no hidden / MLP widths)."""
    sh = make_shape(s, flags)
    sh.hidden = 0
    sh.mlp_width = 0
    return sh


def _ptr(t):
    if t is None:
        return None
    if hasattr(t, "data_ptr"):
        if not t.is_contiguous():
            raise ValueError("tensor must be contiguous")
        if getattr(t, "is_cuda", True) is False:
            # the kernels read and write these buffers: a host tensor would reach them as
            # a host address, so it is refused here, before anything is launched
            raise ValueError("tensor must be in GPU memory")
        return t.data_ptr()
    return t


def _stream(stream):
    if stream is not None:
        return stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def workspace_bytes(shape: Shape) -> int:
    n = lib().h3dit_workspace_bytes(ctypes.byref(shape))
    if n == 0:
        raise H3DitError("h3dit_workspace_bytes", 2)
    return int(n)


def check_shape(shape: Shape) -> int:
    return int(lib().h3dit_check_shape(ctypes.byref(shape)))


def workspace_layout(shape: Shape) -> dict:
    """{region: byte offset} of the workspace regions (None where not reserved)."""
    out = WorkspaceLayout()
    _check("h3dit_get_workspace_layout",
           lib().h3dit_get_workspace_layout(ctypes.byref(shape), ctypes.byref(out)))
    return {n: (None if getattr(out, n) == H3DIT_WS_ABSENT else int(getattr(out, n)))
            for n, _ in WorkspaceLayout._fields_}


def block_weights(w: dict) -> BlockWeights:
    return BlockWeights(*[_ptr(w.get(n)) for n, _ in BlockWeights._fields_])


def block_forward(shape: Shape, weights: dict, x, workspace, stream=None):
    bw = block_weights(weights)
    _check("h3dit_block_forward", lib().h3dit_block_forward(
        ctypes.byref(shape), ctypes.byref(bw), _ptr(x), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def routed_attention(shape: Shape, q, k, v, gate, out, workspace, pooled=None, idx=None,
                     scores=None, stream=None):
    _check("h3dit_routed_attention", lib().h3dit_routed_attention(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out), _ptr(pooled),
        _ptr(idx), _ptr(scores), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def routed_attention_static(shape: Shape, q, k, v, gate, out, pooled=None, idx=None,
                            scores=None, stream=None):
    """h3dit_routed_attention on the library's fixed scratch array (no workspace)."""
    _check("h3dit_routed_attention_static", lib().h3dit_routed_attention_static(
        ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out), _ptr(pooled),
        _ptr(idx), _ptr(scores), _stream(stream)))


def routed_attention_static_status(stream=None) -> int:
    """Status word of the fixed scratch array (synchronises the stream, then clears it)."""
    return int(lib().h3dit_routed_attention_static_status(_stream(stream)))


def denoise_step(shape: Shape, blocks: list, block_ids, z, v_ring, fresh: bool, video,
                 n_fresh_so_far: int, workspace, prefix=None, stream=None):
    """One sampler step.  ``video`` and ``prefix`` are (sigma_i, sigma_a, sigma_b, dt)
    tuples; ``prefix`` (the text and audio rows' schedule) defaults to ``video``."""
    arr = (BlockWeights * max(1, len(blocks)))(*[block_weights(b) for b in blocks])
    ids = (ctypes.c_int * max(1, len(block_ids)))(*[int(i) for i in block_ids])
    sv = Schedule(*[float(x) for x in video])
    sp = Schedule(*[float(x) for x in prefix]) if prefix is not None else None
    _check("h3dit_denoise_step", lib().h3dit_denoise_step(
        ctypes.byref(shape), arr, ids, len(block_ids), _ptr(z), _ptr(v_ring), int(bool(fresh)),
        ctypes.byref(sv), ctypes.byref(sp) if sp is not None else None, int(n_fresh_so_far),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def tile_spans(shape: Shape):
    """(first_row, n_rows) int32 arrays of the shape's video routing tiles."""
    n = ctypes.c_int(0)
    lib().h3dit_tile_spans(ctypes.byref(shape), None, None, ctypes.byref(n))
    if n.value <= 0:
        _check("h3dit_tile_spans", lib().h3dit_check_shape(ctypes.byref(shape)))
    first = np.zeros(max(n.value, 1), np.int32)
    rows = np.zeros(max(n.value, 1), np.int32)
    _check("h3dit_tile_spans", lib().h3dit_tile_spans(ctypes.byref(shape), first.ctypes.data,
                                                      rows.ctypes.data, ctypes.byref(n)))
    return first[:n.value], rows[:n.value]


def video_order(shape: Shape) -> np.ndarray:
    """int32 [n_video]: raster index of each video row in the library's row order."""
    out = np.zeros(shape.n_video, np.int32)
    _check("h3dit_video_order", lib().h3dit_video_order(ctypes.byref(shape), out.ctypes.data))
    return out


def make_ends(ends: dict) -> Ends:
    """ctypes ends struct from a dict of device tensors (plus "c_video", "c_audio")."""
    return Ends(int(ends["c_video"]), int(ends.get("c_audio", 0)),
                *[_ptr(ends.get(n)) for n, _ in Ends._fields_[2:]])


def sample_step(shape: Shape, ends: dict, blocks: list, block_ids, z_video, z_audio,
                v_ring_video, v_ring_audio, core_residual, pass_kind: int, video, audio,
                n_fresh_so_far: int, workspace, stream=None, reduction=None):
    """One sampler step on the modality latents (both ends included).  ``video`` and
    ``audio`` are (sigma_i, sigma_a, sigma_b, dt) tuples; ``pass_kind`` one of
    H3DIT_PASS_FRESH / _EXTRAPOLATE / _CORE_REUSE; ``reduction`` = (first, last) block
    positions of token reduction, or None."""
    arr = (BlockWeights * max(1, len(blocks)))(*[block_weights(b) for b in blocks])
    ids = (ctypes.c_int * max(1, len(block_ids)))(*[int(i) for i in block_ids])
    e = make_ends(ends)
    sv = Schedule(*[float(x) for x in video])
    sa = Schedule(*[float(x) for x in (audio if audio is not None else video)])
    red = Reduction(*[int(x) for x in reduction]) if reduction is not None else None
    _check("h3dit_sample_step", lib().h3dit_sample_step(
        ctypes.byref(shape), ctypes.byref(e), arr, ids, len(block_ids), _ptr(z_video),
        _ptr(z_audio), _ptr(v_ring_video), _ptr(v_ring_audio), _ptr(core_residual),
        ctypes.byref(red) if red is not None else None,
        int(pass_kind), ctypes.byref(sv), ctypes.byref(sa), int(n_fresh_so_far),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def select_blocks(mods: np.ndarray, keep: int) -> list:
    m = np.ascontiguousarray(mods, dtype=np.float32)
    L, six, D = m.shape
    assert six == 6
    out = np.zeros(max(keep, 1) if keep < L else L, dtype=np.int32)
    _check("h3dit_select_blocks", lib().h3dit_select_blocks(
        m.ctypes.data, L, D, keep, out.ctypes.data))
    return out.tolist()


def linear(a, w, b, y, stream=None):
    M, K = a.shape
    N = w.shape[0]
    _check("h3dit_linear", lib().h3dit_linear(_ptr(a), _ptr(w), _ptr(b), _ptr(y), M, N, K,
                                              _stream(stream)))


def sync_status(workspace, stream=None) -> int:
    return int(lib().h3dit_sync_status(_ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream)))


def profile_begin(max_records: int = 65536):
    _check("h3dit_profile_begin", lib().h3dit_profile_begin(int(max_records)))


def profile_end() -> dict:
    """{stage: (milliseconds, kernel launches)} summed over the profiled calls."""
    ms = np.zeros(len(STAGES), np.float32)
    n = np.zeros(len(STAGES), np.int32)
    _check("h3dit_profile_end", lib().h3dit_profile_end(ms.ctypes.data, n.ctypes.data,
                                                        len(STAGES)))
    return {s: (float(ms[i]), int(n[i])) for i, s in enumerate(STAGES)}


def selftest_timeout(workspace, limit_ms: int = 200, stream=None):
    _check("h3dit_selftest_timeout", lib().h3dit_selftest_timeout(
        _ptr(workspace), workspace.numel() * workspace.element_size(), int(limit_ms),
        _stream(stream)))


def gemm_cta_pairs(enable: int = -1) -> int:
    """1: projection GEMMs on SM pairs (cluster kernel) where possible; 0: one SM per
    tile; -1: query.  Returns the previous setting."""
    return int(lib().h3dit_gemm_cta_pairs(int(enable)))


def launch_count() -> int:
    return int(lib().h3dit_launch_count())


def version() -> str:
    return lib().h3dit_version().decode()
