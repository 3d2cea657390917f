"""Host-only checks of the C-ABI library: it loads, exports every declared entry
point, rejects bad arguments before touching a GPU, and its host-side layer
thinning agrees with the oracle."""
import os
import re

import numpy as np
import pytest

import oracle
import synthetic as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "h3dit.h")


@pytest.fixture(scope="module")
def h3():
    import __graft_entry__
    __graft_entry__.build()
    import audio_diffusion_transformer_gb300 as pkg
    return pkg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(h3dit_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(h3):
    lib = h3.lib()
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(h3.EXPORTED)
    assert h3.version().startswith("h3dit")


def test_shape_checks_on_host(h3):
    good = S.BLOCK_4K.shape
    assert h3.check_shape(h3.make_shape(good)) == 0
    bad = [good.with_(tile=32), good.with_(head_dim=96),
           good.with_(hidden=3000), good.with_(mlp_width=1000), good.with_(n_video=0),
           good.with_(attn_width_override=2048),
           good.with_(video_grid=(7, 16, 32)),                  # 3,584 rows, grid holds 3,584?
           good.with_(video_grid=(7, 16, 32), cube=(4, 4, 2)),  # cube of 32 tokens
           good.with_(video_grid=(7, 16, 31))]                  # grid != n_video
    assert 7 * 16 * 32 == good.n_video
    for b in bad[-2:]:
        assert h3.check_shape(h3.make_shape(b)) == 2, b
    for b in bad[:-3]:
        assert h3.check_shape(h3.make_shape(b)) != 0, b
    assert h3.check_shape(h3.make_shape(bad[-3])) == 0  # a consistent grid is accepted
    # a prefix that is not a multiple of 64 rows (the receipt's 36 + 414) is accepted
    assert h3.check_shape(h3.make_shape(good.with_(n_text=36, n_audio=414))) == 0
    assert h3.check_shape(h3.make_shape(good.with_(topk=0))) == 1


def test_workspace_sizes(h3):
    for wl in S.WORKLOADS:
        s = wl.shape
        if wl is S.ATTN_TINY:
            n = h3.workspace_bytes(h3.attn_shape(s))
        else:
            n = h3.workspace_bytes(h3.make_shape(s))
        assert n > 0 and n % 256 == 0
    s3 = S.BLOCK_15K.shape
    n = h3.workspace_bytes(h3.make_shape(s3))
    # q, k, v, g, o, h, x at least: 7 * N * D * 2 bytes
    assert n >= 7 * s3.n_rows * s3.hidden * 2
    with pytest.raises(h3.H3DitError):
        h3.workspace_bytes(h3.make_shape(s3.with_(tile=16)))


def test_entry_points_reject_bad_arguments_without_gpu(h3):
    import ctypes
    lib = h3.lib()
    s = h3.make_shape(S.BLOCK_4K.shape)
    # null pointers are refused before any CUDA call
    assert lib.h3dit_block_forward(ctypes.byref(s), None, None, None, 0, None) == 1
    assert lib.h3dit_routed_attention(ctypes.byref(s), *([None] * 8), None, 0, None) == 1
    assert lib.h3dit_linear(None, None, None, None, 1, 256, 64, None) == 1
    assert lib.h3dit_linear(16, 16, None, 16, 1, 255, 64, None) == 2   # N not a multiple of 256
    assert lib.h3dit_linear(17, 16, None, 16, 1, 256, 64, None) == 3   # misaligned
    bad = h3.make_shape(S.BLOCK_4K.shape.with_(video_grid=(7, 16, 31)))  # grid != n_video
    assert lib.h3dit_block_forward(ctypes.byref(bad), None, None, None, 0, None) == 2
    # the fixed-scratch attention entry point: shape and size are checked, then pointers,
    # all before any CUDA call
    fn = lib.h3dit_routed_attention_static
    assert fn(None, *([None] * 9)) == 1
    small = h3.attn_shape(S.ATTN_TINY.shape)
    assert fn(ctypes.byref(small), *([None] * 9)) == 1
    big = h3.attn_shape(S.BLOCK_15K.shape)  # 26 MB of router scratch: beyond the 4 MiB
    dummy = ctypes.c_void_p(16)
    assert fn(ctypes.byref(big), dummy, dummy, dummy, None, dummy, None, None, None, None) == 4
    assert fn(ctypes.byref(bad), dummy, dummy, dummy, None, dummy, None, None, None, None) == 2
    # 4,096 rows x 24 heads x 128 needs 3.1 MB of router scratch and passes the size check;
    # a misaligned pointer is then refused, still before any CUDA call
    mid = h3.attn_shape(S.BLOCK_4K.shape)
    odd = ctypes.c_void_p(24)
    assert fn(ctypes.byref(mid), dummy, dummy, odd, None, dummy, None, None, None, None) == 3


@pytest.mark.parametrize("L,keep", [(50, 45), (50, 40), (6, 3), (5, 5), (3, 2)])
def test_select_blocks_matches_oracle(h3, L, keep):
    rng = np.random.default_rng(L * 100 + keep)
    mods = (rng.standard_normal((L, 6, 64)) * 0.1).astype(np.float32)
    got = h3.select_blocks(mods, keep)
    want = oracle.thin_layers([m.astype(np.float64) for m in mods], keep)
    assert got == want


def test_select_blocks_ties_drop_higher_index(h3):
    mods = np.zeros((6, 6, 4), np.float32)
    for b, g in enumerate([5.0, 1.0, 3.0, 1.0, 0.5, 9.0]):
        mods[b, 2, 0] = g
    assert h3.select_blocks(mods, 4) == [0, 1, 2, 5]
    assert h3.select_blocks(mods, 4) == oracle.thin_layers(list(mods.astype(np.float64)), 4)


def test_workspace_too_small_and_bad_weights_refused_on_host(h3):
    import ctypes
    lib = h3.lib()
    s = h3.make_shape(S.BLOCK_4K.shape)
    fake = {n: 4096 for n, _ in h3.BlockWeights._fields_}  # aligned, never dereferenced
    bw = h3.BlockWeights(*[fake[n] for n, _ in h3.BlockWeights._fields_])
    need = h3.workspace_bytes(s)
    assert lib.h3dit_block_forward(ctypes.byref(s), ctypes.byref(bw), 4096, 4096, need - 256,
                                   None) == 4  # H3DIT_ERR_WORKSPACE
    bw.w1 = 4097  # misaligned weight pointer
    assert lib.h3dit_block_forward(ctypes.byref(s), ctypes.byref(bw), 4096, 4096, need,
                                   None) == 3  # H3DIT_ERR_ALIGN
    bw.w1 = None
    assert lib.h3dit_block_forward(ctypes.byref(s), ctypes.byref(bw), 4096, 4096, need,
                                   None) == 1  # H3DIT_ERR_ARG
    assert lib.h3dit_selftest_timeout(None, 0, 100, None) == 1
    sv = h3.Schedule(0.5, 0.6, 0.7, -0.1)
    assert lib.h3dit_denoise_step(ctypes.byref(s), None, None, 0, 4096, 4096, 0, ctypes.byref(sv),
                                  None, 0, 4096, need, None) == 1  # nothing to extrapolate
    assert lib.h3dit_denoise_step(ctypes.byref(s), None, None, 0, 4096, 4096, 1, None, None, 0,
                                  4096, need, None) == 1  # no video schedule
    bad = h3.Schedule(0.5, 0.6, 0.6, -0.1)  # sigma_a == sigma_b: no extrapolation slope
    assert lib.h3dit_denoise_step(ctypes.byref(s), None, None, 0, 4096, 4096, 0, ctypes.byref(bad),
                                  None, 2, 4096, need, None) == 1


@pytest.mark.parametrize("grid", [None, (37, 15, 27), (5, 6, 7), (1, 3, 2), (8, 8, 8),
                                  (9, 1, 17)])
def test_tile_spans_and_video_order_match_oracle_tiles(h3, grid):
    """The library's contiguous tiles, mapped through its video order, are exactly the
    oracle's tiles of raster rows (same tile numbering, same order inside a tile)."""
    nv = 14985 if grid is None else int(np.prod(grid))
    shp = S.BlockShape(36, 414, nv, hidden=256, heads=2, head_dim=128, mlp_width=1024, topk=4,
                       video_grid=grid)
    cs = h3.make_shape(shp)
    first, nrows = h3.tile_spans(cs)
    order = h3.video_order(cs)
    P = shp.n_prefix
    assert np.array_equal(np.sort(order), np.arange(nv))
    want = oracle.shape_tiles(shp)
    assert len(first) == len(want) == shp.n_video_tiles
    assert first[0] == P and np.array_equal(first[1:], (first + nrows)[:-1])
    for i, rows in enumerate(want):
        lib_rows = P + order[first[i] - P:first[i] - P + nrows[i]]
        assert np.array_equal(lib_rows, rows), i


def test_sample_step_refuses_bad_arguments_on_host(h3):
    import ctypes
    lib = h3.lib()
    s = h3.make_shape(S.BLOCK_4K.shape)
    need = h3.workspace_bytes(s)
    fake = 4096  # aligned, never dereferenced: every case fails before a launch
    good = dict(c_video=96, c_audio=32, **{n: fake for n, _ in h3.Ends._fields_[2:]})
    sv = h3.Schedule(1.0, 0.0, 0.0, -0.125)

    def call(ends, pass_kind=0, z=fake, ws_bytes=need, nf=0, res=fake, sched=sv):
        e = h3.make_ends(ends)
        return lib.h3dit_sample_step(ctypes.byref(s), ctypes.byref(e), None, None, 0, z, fake,
                                     fake, fake, res, None, pass_kind,
                                     ctypes.byref(sched) if sched is not None else None,
                                     ctypes.byref(sv), nf, fake, ws_bytes, None)

    assert call(dict(good, c_video=100)) == 2             # latent width not a multiple of 32
    assert call(dict(good, c_audio=160)) == 2             # wider than 128
    assert call(dict(good, w_out_video=None)) == 1        # missing head
    assert call(dict(good, b_in_audio=fake + 4)) == 3     # misaligned
    assert call(good, pass_kind=7) == 1                   # unknown pass
    assert call(good, z=None) == 1
    assert call(good, ws_bytes=need - 256) == 4
    assert call(good, pass_kind=2, res=None) == 1         # core reuse needs the residual
    assert call(good, pass_kind=1, nf=0) == 1             # nothing to extrapolate from
    assert call(good, pass_kind=0) == 1                   # fresh pass without blocks array
    assert call(good, sched=None) == 1


def test_token_reduction_needs_its_buffers(h3):
    import ctypes
    lib = h3.lib()
    base = S.BlockShape(36, 92, 5 * 6 * 7, hidden=256, heads=2, head_dim=128, mlp_width=512,
                        topk=3, video_grid=(5, 6, 7))
    s_plain = h3.make_shape(base)
    s_red = h3.make_shape(base.with_(token_reduction=True))
    # the flag reserves a bypass of N x D bf16 and the pooled rows' baselines
    extra = h3.workspace_bytes(s_red) - h3.workspace_bytes(s_plain)
    assert extra >= (base.n_rows + 5 * 6 * 4) * 256 * 2
    # a grid is required; a 1-wide grid has nothing to pair
    assert h3.check_shape(h3.make_shape(base.with_(video_grid=None, token_reduction=True))) == 2
    one = S.BlockShape(36, 92, 5 * 6, hidden=256, heads=2, head_dim=128, mlp_width=512, topk=3,
                       video_grid=(5, 6, 1), token_reduction=True)
    assert h3.check_shape(h3.make_shape(one)) == 2
    # a reduction asked of a shape without the buffers is refused before any launch
    fake = 4096
    e = h3.make_ends(dict(c_video=96, c_audio=32, **{n: fake for n, _ in h3.Ends._fields_[2:]}))
    bw = h3.BlockWeights(*[fake] * len(h3.BlockWeights._fields_))
    ids = (ctypes.c_int * 1)(0)
    red = h3.Reduction(0, 1)
    sv = h3.Schedule(1.0, 0.0, 0.0, -0.125)
    st = lib.h3dit_sample_step(ctypes.byref(s_plain), ctypes.byref(e), ctypes.byref(bw), ids, 1,
                               fake, fake, fake, fake, None, ctypes.byref(red), 0,
                               ctypes.byref(sv), ctypes.byref(sv), 0, fake,
                               h3.workspace_bytes(s_plain), None)
    assert st == 2


def test_binding_struct_layouts_match_the_header(h3, tmp_path):
    """The ctypes structs of the binding have the sizes and field offsets of the C
    structs in include/h3dit.h, as the host C compiler lays them out."""
    import ctypes
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    from audio_diffusion_transformer_gb300 import _binding as B
    structs = {"h3dit_shape": B.Shape, "h3dit_block_weights": B.BlockWeights,
               "h3dit_schedule": B.Schedule, "h3dit_ends": B.Ends,
               "h3dit_reduction": B.Reduction, "h3dit_workspace_layout": B.WorkspaceLayout}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "h3dit.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'  printf("{cname} sizeof %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'  printf("{cname} {f} %zu\\n", offsetof({cname}, {f}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), "-o", str(exe),
                    str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {}
    for ln in out.splitlines():
        cname, field, val = ln.split()
        got[(cname, field)] = int(val)
    for cname, py in structs.items():
        assert got[(cname, "sizeof")] == ctypes.sizeof(py), cname
        for f, _ in py._fields_:
            assert got[(cname, f)] == getattr(py, f).offset, f"{cname}.{f}"


def test_binding_refuses_host_tensors_before_any_launch(h3):
    torch = pytest.importorskip("torch")
    shp = S.BlockShape(64, 0, 64, hidden=256, heads=2, head_dim=128, mlp_width=256, topk=1)
    cs = h3.make_shape(shp)
    w = {n: torch.zeros(16, dtype=torch.bfloat16) for n in ("w_qkvg", "b_qkvg")}
    x = torch.zeros(shp.n_rows, shp.hidden, dtype=torch.bfloat16)
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="GPU memory"):
        h3.block_forward(cs, w, x, ws, stream=0)
    with pytest.raises(ValueError, match="GPU memory"):
        h3.linear(x, x, None, x, stream=0)


def test_documented_size_limits_refused_on_host(h3):
    """The limits the header documents come back as H3DIT_ERR_SHAPE before any launch."""
    base = S.BlockShape(0, 0, 64, hidden=256, heads=4, head_dim=64, mlp_width=256, topk=1)
    assert h3.check_shape(h3.make_shape(base.with_(heads=1))) == 2  # attention width 64
    ok = lambda s: h3.check_shape(h3.make_shape(s))  # noqa: E731
    # at most 65,408 packed rows (a prefix query unit walks N / 128 key steps)
    assert ok(base.with_(n_video=1022 * 64)) == 0
    assert ok(base.with_(n_video=1022 * 64 + 1)) == 2
    # at most 1,024 video tiles: a 1 x 1 x W grid cut into clipped 4 x 4 x 4 cubes has
    # ceil(W / 4) tiles of at most 4 rows
    assert ok(base.with_(n_video=4096, video_grid=(1, 1, 4096))) == 0
    assert ok(base.with_(n_video=4097, video_grid=(1, 1, 4097))) == 2
    # a video query tile's steps, ceil(P / 128) + min(k, Tv), at most 512
    assert ok(base.with_(n_text=128 * 500, n_video=64 * 12, topk=12)) == 0
    assert ok(base.with_(n_text=128 * 500, n_video=64 * 13, topk=13)) == 2
    # head widths 64 and 128 only; hidden and MLP widths in multiples of 256 (SwiGLU 128)
    assert ok(base.with_(head_dim=32)) == 2
    assert ok(base.with_(hidden=384)) == 2
    assert ok(base.with_(mlp_width=384)) == 2
    assert ok(base.with_(mlp_width=384, mlp="swiglu")) == 0
    assert ok(base.with_(mlp_width=192, mlp="swiglu")) == 2
    # token reduction needs a video grid at least two tokens wide
    assert ok(base.with_(token_reduction=True)) == 2
    assert ok(base.with_(n_video=2 * 4 * 8, video_grid=(2, 4, 8), token_reduction=True)) == 0
    assert ok(base.with_(n_video=2 * 4 * 1, video_grid=(2, 4, 1), token_reduction=True)) == 2
    # the attention-only shape (hidden = mlp_width = 0) sizes its own, smaller workspace
    full = h3.workspace_bytes(h3.make_shape(base))
    attn = h3.workspace_bytes(h3.attn_shape(base))
    assert 0 < attn < full


def test_plain_c_program_links_and_calls_the_library(h3, tmp_path):
    """A C99 program includes the header, links libh3dit.so and calls its host-only
    entry points; its answers equal the Python binding's."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    src = tmp_path / "use.c"
    src.write_text(r'''
#include <stdio.h>
#include "h3dit.h"
int main(void) {
  h3dit_shape s = {.n_text = 512, .n_audio = 1024, .n_video = 13899, .hidden = 5120,
                   .heads = 40, .head_dim = 128, .attn_width = 5120, .mlp_width = 20480,
                   .tile = 64, .topk = 16, .rms_eps = 1e-6f, .rope_theta = 10000.f,
                   .flags = H3DIT_QK_NORM | H3DIT_ROPE | H3DIT_POOLED};
  int first[256], rows[256], n = 256;
  h3dit_status st = h3dit_tile_spans(&s, first, rows, &n);
  printf("%zu %d %d %d %d %d %s\n", h3dit_workspace_bytes(&s), (int)h3dit_check_shape(&s),
         (int)st, n, first[n - 1], rows[n - 1], h3dit_status_string(H3DIT_ERR_ALIGN));
  return 0;
}
''')
    from audio_diffusion_transformer_gb300._binding import LIB_PATH
    pkg = os.path.dirname(LIB_PATH)
    exe = tmp_path / "use"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), "-o", str(exe),
                    str(src), LIB_PATH, f"-Wl,-rpath,{pkg}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    shp = S.BLOCK_15K.shape
    cs = h3.make_shape(shp)
    first, nrows = h3.tile_spans(cs)
    assert int(out[0]) == h3.workspace_bytes(cs)
    assert out[1:4] == ["0", "0", str(shp.n_video_tiles)]
    assert int(out[4]) == first[-1] and int(out[5]) == nrows[-1] == 13899 - 217 * 64
    assert " ".join(out[6:]) == "pointer not 16-byte aligned"


def test_workspace_layout_regions(h3):
    """Attention alone reserves only the status word and the router's regions; a block
    reserves q..o, and with H3DIT_KEEP_INTERMEDIATES its MLP activations and x1 get
    regions of their own; regions never overlap."""
    shp = S.BLOCK_4K.shape
    att = h3.workspace_layout(h3.attn_shape(shp))
    assert att["total"] == h3.workspace_bytes(h3.attn_shape(shp))
    for n in ("q", "k", "v", "g", "o", "u", "h", "x1"):
        assert att[n] is None, n
    H, d, Tv, k = shp.heads, shp.head_dim, shp.n_video_tiles, min(shp.topk, shp.n_video_tiles)
    router = 3 * H * Tv * d * 4 + H * Tv * Tv * 4 + H * Tv * k * 4 + H * Tv * d * 4
    assert att["total"] <= 256 + router + 4 * 256
    assert att["total"] < 4 << 20  # fits the fixed scratch of the static entry point
    blk = h3.workspace_layout(h3.make_shape(shp))
    assert blk["u"] == blk["q"] and blk["x1"] is None  # u reuses the dead q..g region
    keep = h3.workspace_layout(h3.make_shape(shp, h3.make_shape(shp).flags
                                             | h3.H3DIT_KEEP_INTERMEDIATES))
    assert keep["total"] == h3.workspace_bytes(h3.make_shape(
        shp, h3.make_shape(shp).flags | h3.H3DIT_KEEP_INTERMEDIATES))
    N, D, A, F = shp.n_rows, shp.hidden, shp.attn_width, shp.mlp_width
    sizes = {"status": 4, "q": N * A * 2, "k": N * A * 2, "v": N * A * 2, "g": N * A * 2,
             "o": N * A * 2, "u": N * F * 2, "h": N * D * 2, "x1": N * D * 2,
             "means": 3 * H * Tv * d * 4, "scores": H * Tv * Tv * 4, "idx": H * Tv * k * 4,
             "pooled": H * Tv * d * 4}
    spans = sorted((keep[n], keep[n] + sz) for n, sz in sizes.items())
    for (a0, a1), (b0, _) in zip(spans, spans[1:]):
        assert a1 <= b0
    assert spans[-1][1] <= keep["total"]
    assert all(keep[n] % 256 == 0 for n in sizes)
