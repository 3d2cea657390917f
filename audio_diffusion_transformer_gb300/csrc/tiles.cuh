// tiles.cuh -- which packed rows form each video routing tile, and where a video
// row sits in the latent grid.  Host and device code share these closed forms.
//
// Two layouts:
//  * 1-D (no grid): video rows [P, P + V) cut into contiguous 64-row tiles in
//    packed order; the last tile may be partial.
//  * cubes (TensorFold #949 "Receipts": 280 video tiles at 864x480x124 from a
//    4x4x4 cube map): the video latent grid T x Hg x Wg is cut into cubes of
//    ct x ch x cw tokens (edge cubes clipped, not padded).  The library keeps
//    the video rows in cube order -- cubes in raster (cube_t, cube_h, cube_w)
//    order, the tokens of a cube in raster (t, h, w) order -- so every tile is a
//    contiguous run of at most 64 rows starting right after the previous one.
#pragma once

namespace h3 {

struct TileGeom {
  int P, V;        // prefix (text + audio) rows, video rows
  int gt, gh, gw;  // latent grid; gt == 0 selects the 1-D layout
  int ct, ch, cw;  // cube extents (product = 64)
  int nt, nh, nw;  // cubes along t, h, w
  int gw_full;     // token reduction: the full width whose horizontal pairs form this
                   // grid's columns (rotary w = 2j + 0.5, or 2j for a lone last token); 0 = none
};

__host__ __device__ __forceinline__ int tg_min(int a, int b) { return a < b ? a : b; }

__host__ __device__ __forceinline__ int tile_count_of(const TileGeom& g) {
  return g.gt == 0 ? (g.V + 63) / 64 : g.nt * g.nh * g.nw;
}

// First packed row and row count of video tile t (0 <= t < tile_count_of(g)).
__host__ __device__ __forceinline__ void tile_span(const TileGeom& g, int t, int* first,
                                                   int* count) {
  if (g.gt == 0) {
    *first = g.P + 64 * t;
    *count = tg_min(64, g.V - 64 * t);
    return;
  }
  const int a = t / (g.nh * g.nw), b = (t / g.nw) % g.nh, c = t % g.nw;
  const int et = tg_min(g.ct, g.gt - a * g.ct);
  const int eh = tg_min(g.ch, g.gh - b * g.ch);
  const int ew = tg_min(g.cw, g.gw - c * g.cw);
  // rows before this cube: whole t-slabs, then whole cube rows of this slab, then cubes
  *first = g.P + a * g.ct * g.gh * g.gw + et * (b * g.ch) * g.gw + et * eh * (c * g.cw);
  *count = et * eh * ew;
}

// Latent coordinates (t, h, w) of video row v (0 <= v < V) in cube order.
__host__ __device__ __forceinline__ void video_coord(const TileGeom& g, int v, int* tt, int* hh,
                                                     int* ww) {
  const int slab = g.ct * g.gh * g.gw;
  const int a = tg_min(v / slab, g.nt - 1);
  int rem = v - a * slab;
  const int et = tg_min(g.ct, g.gt - a * g.ct);
  const int crow = et * g.ch * g.gw;
  const int b = tg_min(rem / crow, g.nh - 1);
  rem -= b * crow;
  const int eh = tg_min(g.ch, g.gh - b * g.ch);
  const int cube = et * eh * g.cw;
  const int c = tg_min(rem / cube, g.nw - 1);
  rem -= c * cube;
  const int ew = tg_min(g.cw, g.gw - c * g.cw);
  *tt = a * g.ct + rem / (eh * ew);
  *hh = b * g.ch + (rem / ew) % eh;
  *ww = c * g.cw + rem % ew;
}

// Row (0 <= row < V, cube order) of the video token at latent (t, h, w).
__host__ __device__ __forceinline__ int video_row_of(const TileGeom& g, int tt, int hh, int ww) {
  const int a = tt / g.ct, b = hh / g.ch, c = ww / g.cw;
  int first, count;
  tile_span(g, (a * g.nh + b) * g.nw + c, &first, &count);
  const int eh = tg_min(g.ch, g.gh - b * g.ch);
  const int ew = tg_min(g.cw, g.gw - c * g.cw);
  return first - g.P + ((tt - a * g.ct) * eh + (hh - b * g.ch)) * ew + (ww - c * g.cw);
}

}  // namespace h3
