// Restructured KV cache: copy a run of frames from a monolithic
// [tokens][H][d] tensor into the per-archetype regions, all heads in one
// launch.  Used both to split the window after classification and, once per
// denoising step, to append the current block (with eviction implied by the
// ring: frame a lands in slot a mod window_frames, over the oldest frame).
//
//   Sink     block 0 only, rows [0, 3F)
//   Dummy    the newest block only, rows [0, 3F)
//   Global   ring slot s = a mod W, rows [s*F, (s+1)*F) in raster order
//            (also Spatial heads in the sliding mode)
//   Spatial  ring slot s, cell-major: cell (ci, cj) owns rows
//            W*tokens_before(ci, cj) + [0, W*|cell|), slot s of it the
//            |cell| rows at offset s*|cell|, row-major inside the cell
// [Pith review of HeadCast, "What carries the argument" (split along the
//  head dimension; single-block Sink/Dummy buffers, full-window Global,
//  Spatial full history partitioned by cell); Figure 2 phase 3.]
//
// Each thread moves 16-byte chunks; consecutive threads read consecutive
// chunks of the source, so reads are fully coalesced and every (token, head)
// row lands as one contiguous run in its region.
#include "hc_internal.h"

namespace hc {
namespace {

__global__ void __launch_bounds__(256) scatter_kernel(const ScatterParams p) {
  const Geom& g = p.g;
  const int cpr = g.d * p.esize / 16;
  const int64_t total = (int64_t)p.n_src_frames * g.F * g.H * cpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int c = (int)(idx % cpr);
    const int64_t rest = idx / cpr;
    const int h = (int)(rest % g.H);
    const int64_t tok = rest / g.H;
    const int f = (int)(tok / g.F);
    const int pos = (int)(tok - (int64_t)f * g.F);
    const int64_t a = p.src_frame0 + f;
    const HeadSlot hs = p.heads[h];
    int64_t row;
    if (hs.arch == HC_SINK) {
      if (a >= g.fpb) continue;
      row = a * g.F + pos;
    } else if (hs.arch == HC_DUMMY) {
      if (a < p.dummy_frame0) continue;
      row = (a - p.dummy_frame0) * g.F + pos;
    } else if (hs.arch == HC_GLOBAL || g.spatial_mode == HC_SPATIAL_SLIDING) {
      row = (a % g.Wf) * g.F + pos;
    } else {
      const int slot = (int)(a % g.Wf);
      const int hh = pos / g.Fw, ww = pos - hh * g.Fw;
      const int ci = cell_index(hh, g.cell_h, g.ncell_h);
      const int cj = cell_index(ww, g.cell_w, g.ncell_w);
      const int hz = cell_extent(ci, g.Fh, g.cell_h, g.ncell_h);
      const int wz = cell_extent(cj, g.Fw, g.cell_w, g.ncell_w);
      row = (int64_t)g.Wf * cell_tokens_before(g, ci, cj) + (int64_t)slot * hz * wz +
            (hh - ci * g.cell_h) * wz + (ww - cj * g.cell_w);
    }
    const int64_t src = (tok * g.H + h) * cpr + c;
    const int64_t dst = (hs.row0 + row) * cpr + c;
    static_cast<int4*>(p.k_dst)[dst] = static_cast<const int4*>(p.k_src)[src];
    static_cast<int4*>(p.v_dst)[dst] = static_cast<const int4*>(p.v_src)[src];
  }
}

}  // namespace

cudaError_t launch_scatter(const ScatterParams& p, cudaStream_t s) {
  const int64_t total = (int64_t)p.n_src_frames * p.g.F * p.g.H * (p.g.d * p.esize / 16);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 148 * 16) blocks = 148 * 16;
  scatter_kernel<<<(unsigned)blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hc
