// Internal declarations shared by the library's translation units.
//
// Geometry, work items and the cell arithmetic of the deployed Spatial path
// (non-overlapping cells of cell_h x cell_w tokens, the last cell along an
// axis taking the rounded remainder: n_cells = max(1, floor(N/c + 1/2))).
// [Pith review of HeadCast, Ledger "deployed spatial grid cell = 10x10 with
//  rounded remainder"; major comment 2; Figure 3 caption.]
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/headcast.h"

namespace hc {

#define HC_HD __host__ __device__ __forceinline__

// Layer geometry as the kernels see it.
struct Geom {
  int H, d, Fh, Fw, F, fpb, Wf, blk;   // blk = fpb * F (tokens per block)
  int cell_h, cell_w, ncell_h, ncell_w;
  int radius;
  int proxy_mode;                      // HC_PROXY_NEIGHBOURHOOD or HC_PROXY_CELL
  int spatial_mode;                    // HC_SPATIAL_CELLS or HC_SPATIAL_SLIDING
  float scale_log2;                    // softmax scale * log2(e)
};

HC_HD int n_cells(int n, int c) {            // max(1, floor(n/c + 1/2))
  int k = (2 * n + c) / (2 * c);
  return k < 1 ? 1 : k;
}
HC_HD int cell_index(int x, int c, int nc) {
  int i = x / c;
  return i < nc - 1 ? i : nc - 1;
}
HC_HD int cell_extent(int i, int n, int c, int nc) {
  return i < nc - 1 ? c : n - (nc - 1) * c;
}
// Tokens of one frame that precede cell (ci, cj) in cell-major order.  Every
// cell row above ci is cell_h tall; cells left of cj in row ci are cell_w
// wide and share row ci's height.
HC_HD int cell_tokens_before(const Geom& g, int ci, int cj) {
  int hz = cell_extent(ci, g.Fh, g.cell_h, g.ncell_h);
  return ci * g.cell_h * g.Fw + hz * cj * g.cell_w;
}

// Rows [h_lo, h_hi] and columns [w_lo, w_hi] of the classification proxy of
// a query at (h, w): the clipped (2r+1) x (2r+1) neighbourhood, or with
// HC_PROXY_CELL the query's deployed cell.  Both bounds are non-decreasing in
// h and in w, so the band of rows of a run of queries is [h_lo(first row),
// h_hi(last row)].
// [Pith review of HeadCast, major comment 2: proxy r = 2 vs deployed cells.]
HC_HD void proxy_window(const Geom& g, int h, int w, int& h_lo, int& h_hi, int& w_lo, int& w_hi) {
  if (g.proxy_mode == HC_PROXY_CELL) {
    const int ci = cell_index(h, g.cell_h, g.ncell_h), cj = cell_index(w, g.cell_w, g.ncell_w);
    h_lo = ci * g.cell_h;
    h_hi = h_lo + cell_extent(ci, g.Fh, g.cell_h, g.ncell_h) - 1;
    w_lo = cj * g.cell_w;
    w_hi = w_lo + cell_extent(cj, g.Fw, g.cell_w, g.ncell_w) - 1;
  } else {
    h_lo = h - g.radius < 0 ? 0 : h - g.radius;
    h_hi = h + g.radius > g.Fh - 1 ? g.Fh - 1 : h + g.radius;
    w_lo = w - g.radius < 0 ? 0 : w - g.radius;
    w_hi = w + g.radius > g.Fw - 1 ? g.Fw - 1 : w + g.radius;
  }
}

// Rows and columns of the sliding deployed Spatial window of a query at
// (h, w): cell_h x cell_w keys with the query at offset (cell_h/2, cell_w/2)
// from the top-left corner, clipped.  Bounds non-decreasing in h and w.
HC_HD void sliding_window(const Geom& g, int h, int w, int& h_lo, int& h_hi, int& w_lo, int& w_hi) {
  const int h0 = h - g.cell_h / 2, w0 = w - g.cell_w / 2;
  h_lo = h0 < 0 ? 0 : h0;
  h_hi = h0 + g.cell_h - 1 > g.Fh - 1 ? g.Fh - 1 : h0 + g.cell_h - 1;
  w_lo = w0 < 0 ? 0 : w0;
  w_hi = w0 + g.cell_w - 1 > g.Fw - 1 ? g.Fw - 1 : w0 + g.cell_w - 1;
}

// Window of a band item: the classification proxy or the sliding Spatial path.
enum : int32_t { WIN_PROXY = 0, WIN_SLIDING = 1 };
HC_HD void band_window(const Geom& g, int win, int h, int w, int& h_lo, int& h_hi, int& w_lo, int& w_hi) {
  if (win == WIN_SLIDING)
    sliding_window(g, h, w, h_lo, h_hi, w_lo, w_hi);
  else
    proxy_window(g, h, w, h_lo, h_hi, w_lo, w_hi);
}

// Work item kinds.
enum : int32_t {
  ITEM_RANGE = 0,   // queries q0.. (block-local tokens), keys: one run of rows
  ITEM_CELL = 1,    // queries: ordinals q0.. of one cell's 3-frame query set
  ITEM_PROXY = 2,   // queries q0.. inside one frame; keys: (2r+1) neighbourhood rows of every frame
  ITEM_BAND = 3,    // routed sliding Spatial (fp32 path): queries q0.. inside one frame; keys:
                    // the band of window rows in every filled ring slot of the head, masked
  ITEM_PATCH = 4,   // routed sliding Spatial (tensor-core path): a patch of query positions
                    // in every frame of the block; keys: its halo in every filled ring slot
};

// Query patches of the band attentions on the tensor cores (the
// classification proxy and the sliding deployed Spatial path).  A patch is
// ph x pw positions of the frame in each of the block's frames (every query
// at one position has the same key window).  Its keys in one key frame are
// the halo rows [h0 + dh, h0 + dh + kh) x columns [w0 + dw, w0 + dw + kw),
// covered by tpf boxes of bh rows x kw columns (bh * kw <= 128 keys, one key
// tile each), every query masked to its own window; boxes reaching outside
// the frame read zeros there (masked).  With `cells` the patches are the
// deployed cells (the classifier's cell proxy): halo = the cell, and a cell
// with more than 256 queries is cut into cpc chunks of 256.
struct PatchGeom {
  int32_t ph, pw;     // patch
  int32_t dh, dw;     // halo origin relative to the patch origin
  int32_t kh, kw;     // halo extent (cells: the largest cell)
  int32_t bh, tpf;    // box rows, boxes per key frame
  int32_t npw, n;     // patches per patch row, patches per frame
  int32_t cells, cpc; // patches are the deployed cells; query chunks per patch
};

// At most this many boxes per key frame: each softmax thread keeps its
// window mask for every box of a frame in shared memory.
constexpr int kMaxBoxesPerFrame = 4;

inline bool finish_patch_geom(PatchGeom& pg) {
  if (pg.kw > 128 || pg.kw < 1 || pg.kh < 1) return false;
  pg.bh = 128 / pg.kw;
  if (pg.bh > pg.kh) pg.bh = pg.kh;
  pg.tpf = (pg.kh + pg.bh - 1) / pg.bh;
  return pg.tpf <= kMaxBoxesPerFrame;
}

// Halo of a uniform patch for a window: the (2r+1) x (2r+1) neighbourhood
// (WIN_PROXY) or the centred cell_h x cell_w window (WIN_SLIDING).  False if
// no box fits (a halo row wider than 128 keys).
inline bool make_patch_geom(const Geom& g, int win, int ph, int pw, PatchGeom& pg) {
  pg.ph = ph;
  pg.pw = pw;
  pg.cells = 0;
  pg.cpc = 1;
  if (win == WIN_SLIDING) {
    pg.dh = -(g.cell_h / 2);
    pg.dw = -(g.cell_w / 2);
    pg.kh = ph + g.cell_h - 1;
    pg.kw = pw + g.cell_w - 1;
  } else {
    pg.dh = -g.radius;
    pg.dw = -g.radius;
    pg.kh = ph + 2 * g.radius;
    pg.kw = pw + 2 * g.radius;
  }
  pg.npw = (g.Fw + pw - 1) / pw;
  pg.n = ((g.Fh + ph - 1) / ph) * pg.npw;
  return finish_patch_geom(pg);
}

// The deployed cells as patches (the classifier's cell proxy).
inline bool make_cell_patch_geom(const Geom& g, PatchGeom& pg) {
  const int lh = cell_extent(g.ncell_h - 1, g.Fh, g.cell_h, g.ncell_h);
  const int lw = cell_extent(g.ncell_w - 1, g.Fw, g.cell_w, g.ncell_w);
  pg.cells = 1;
  pg.ph = pg.kh = g.ncell_h > 1 && lh < g.cell_h ? g.cell_h : lh;
  pg.pw = pg.kw = g.ncell_w > 1 && lw < g.cell_w ? g.cell_w : lw;
  pg.dh = pg.dw = 0;
  pg.npw = g.ncell_w;
  pg.n = g.ncell_h * g.ncell_w;
  pg.cpc = (g.fpb * pg.kh * pg.kw + 255) / 256;
  return finish_patch_geom(pg);
}

// The patch shape with the fewest key tiles over `frames` key frames (plus
// a boundary cost of 5 tiles per patch), over patches of at most 256 queries.
inline bool choose_patch_geom(const Geom& g, int win, int frames, PatchGeom& best) {
  long best_cost = -1;
  const int max_pos = 256 / g.fpb;
  for (int ph = 1; ph <= g.Fh && ph <= max_pos; ++ph)
    for (int pw = 1; pw <= g.Fw && ph * pw <= max_pos; ++pw) {
      PatchGeom pg;
      if (!make_patch_geom(g, win, ph, pw, pg)) continue;
      const long cost = (long)pg.n * ((long)pg.tpf * frames + 5);
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best = pg;
      }
    }
  return best_cost >= 0;
}

struct alignas(16) WorkItem {
  int32_t head;
  int32_t kind;
  int32_t q0;
  int32_t nq;
  int64_t k_row0;       // first key row in the key buffer's row space
  int32_t k_len;        // keys when k_per_frame == 0
  int32_t k_per_frame;  // > 0: k_len = k_per_frame * valid_frames
  int32_t cell;         // ITEM_CELL: ci * ncell_w + cj
  int32_t out_plane;
  int16_t chunk;        // split key run: this item covers key tiles
  int16_t n_chunks;     //   [chunk*T/n_chunks, (chunk+1)*T/n_chunks) of the run's T tiles
  int32_t part;         // >= 0: write an unnormalised partial output to slot `part`
};
static_assert(sizeof(WorkItem) == 48, "WorkItem layout");

// A query tile set whose key run is split across several work items: the
// partial outputs of slots part0 .. part0 + n_chunks - 1 are merged into the
// final output of queries q0 .. q0 + nq - 1 (block-local tokens) of `head`.
struct alignas(16) SplitItem {
  int32_t head, q0, nq, n_chunks;
  int32_t part0, pad0, pad1, pad2;
};
static_assert(sizeof(SplitItem) == 32, "SplitItem layout");

// Rows of one partial-output slot (the query rows of one work item).
constexpr int kPartRows = 256;

// Persistent launches: work items are laid out per CTA, CTA c running items
// sched[c] .. sched[c+1]-1 of the list.  Plans are made for this many CTAs
// (the SM count of a B300); the schedule array reserves room for kMaxCtas.
constexpr int kPlanCtas = 148;
constexpr int kMaxCtas = 1024;

// Item source for an attention launch.
enum : int32_t {
  ITEMS_LIST = 0,     // items[blockIdx.x]
  ITEMS_DENSE = 1,    // x: q tile, y: head, z: plane -> RANGE over plane_k0/plane_klen
  ITEMS_PROXY = 2,    // x: frame * tiles_per_frame + t, y: head -> PROXY
};

struct AttnParams {
  const void* q;            // [Nq][H][d]
  const void* k;            // key buffer base
  const void* v;            // value buffer base
  void* o;                  // output base (plane 0)
  int64_t k_stride;         // elements between consecutive key rows
  int64_t k_hstride;        // elements between heads inside a key row (0 for per-head buffers)
  int64_t o_plane_stride;   // elements between output planes
  int32_t nq_total;         // queries in the block (3F or caller's Nq)
  int32_t out_fp32;         // 1: fp32 output, 0: input dtype
  int32_t item_mode;
  int32_t n_items;          // work items of the launch
  const WorkItem* items;
  const int32_t* sched;     // ITEMS_LIST, tensor-core kernel: per-CTA item ranges (nullable)
  int32_t valid_frames;
  int32_t proxy_frames;     // frames of keys for ITEMS_PROXY
  int32_t tiles_per_frame;  // ITEMS_PROXY q tiles per frame
  int32_t n_planes;         // ITEMS_DENSE planes
  int64_t plane_k0[4];
  int32_t plane_klen[4];
  Geom g;
  int* status;
  float* part_o;            // split key runs: partial outputs [slot][kPartRows][d] (fp32, unnormalised)
  float* part_ml;           //   and their row max / row sum [slot][kPartRows][2] (log2 domain)
  // Classification full pass (cls != 0, ITEMS_DENSE with one plane): the
  // keys [0, nk) run as three segments, [0, seg_sink) the Sink block,
  // [seg_sink, seg_dummy) the middle and [seg_dummy, nk) the Dummy block.
  // The running state after the Sink segment and before the Dummy segment is
  // parked (unnormalised O, row max, row sum) and the accumulator restarts
  // for the Dummy segment; the epilogue merges them into the full output and
  // writes the per-token statistics.
  int32_t cls;
  int32_t seg_sink, seg_dummy;
  int32_t cls_n0, cls_n01;          // first key tile of the middle / the Dummy segment
  int32_t cls_v0, cls_v1, cls_v2;   // keys in the last tile of each segment
  void* park_o;               // bf16 [Nq][H][d]: the Sink state (unnormalised)
  float* park_o1;             // [Nq][H][d]: the state before the Dummy block (unnormalised);
                              // bf16 (in the same area) when park1_bf16 is set
  int32_t park1_bf16;         // no full-context output wanted: the cosines alone read it
  float* park_ml;             // [2][Nq][H][2]
  const void* proxy_o;        // bf16 [Nq][H][d] the proxy output (normalised)
  float* tok;                 // [4][H][Nq]: cos sink, cos dummy, cos proxy, squared error
  void* o_full;               // nullable: the full-context output in the input dtype
  int32_t band_win;           // WIN_PROXY / WIN_SLIDING window of band items
  int32_t band_frame0;        // tensor-core band items: frame index of the head's first key frame
                              // (cache launches add the head's row0 / F)
  PatchGeom pg;               // tensor-core band items: the patch geometry
  int32_t debug_stall;        // test hook: the K/V producer stops after the first tile
  uint64_t wait_limit_ns;     // bound of every device-side wait
};

// Test hook state (hc_debug_inject_stall).
bool debug_stall_enabled();

// Record a failure message for hc_last_error_message and return `s`.
hc_status record_error(hc_status s, const char* fmt, ...);

// Status codes a kernel may write to the device status word.
enum : int { DEV_OK = 0, DEV_TIMEOUT = 7, DEV_BOUNDS = 6 };

// Launchers (attn.cu).
cudaError_t launch_attention(const AttnParams& p, int dtype, dim3 grid, cudaStream_t s);
int attention_block_rows(int dtype, int d);   // queries per item tile

// tcgen05/TMA attention (attn_tc.cu), bf16 only.  K and V are read as
// [rows][heads][d] tensors; with heads == 1 the key rows of an item are
// absolute rows of that buffer (the restructured cache), otherwise token
// rows of a monolithic [tokens][H][d] window addressed with the item's head.
struct TcKV {
  const void* k;
  const void* v;
  int heads;
  int64_t rows;
};
// `ctas` persistent CTAs; with p.sched the CTA ranges come from it,
// otherwise CTA c runs items c, c + ctas, c + 2*ctas, ...
cudaError_t launch_attention_tc(const AttnParams& p, const TcKV& kv, int ctas, cudaStream_t s);
int tc_block_rows();                          // queries per tcgen05 item (256)
int tc_key_tile();                            // keys per tcgen05 key tile (128)
int proxy_block_rows();                       // queries per classification-proxy item
int device_sm_count();                        // SMs of the current device (cached)

// Merge of split key runs (attn_tc.cu): out[q][head] from the partial slots.
struct CombineParams {
  const SplitItem* items;
  int32_t n_items;
  int32_t out_fp32;
  const float* part_o;
  const float* part_ml;
  void* o;
  Geom g;
};
cudaError_t launch_combine(const CombineParams& c, cudaStream_t s);

// Classification post-processing (classify.cu).
struct ClassifyPost {
  const float* planes;      // 4 planes fp32 [Nq][H][d]: full, sink, dummy, proxy
  int64_t plane_stride;
  float* tok;               // [4][H][Nq]: cos_sink, cos_dummy, cos_spatial, sqerr
  void* o_full;             // nullable, dtype of the inputs
  int32_t o_full_fp32;
  int8_t* labels;
  float* stats;             // nullable [H][6]
  int32_t nq;
  Geom g;
  float theta_sink, theta_dummy, theta_spatial, theta_score, gamma;
  const int* status;        // device status word: set => the planes are incomplete
  int32_t tokens_ready;     // 1: tok already holds the per-token values (no planes)
};
cudaError_t launch_classify_post(const ClassifyPost& c, cudaStream_t s);

// Cache scatter (cache.cu).
struct HeadSlot {
  int32_t arch;
  int32_t pad;
  int64_t row0;
};
struct ScatterParams {
  const void* k_src;        // [n_src_frames*F][H][d]
  const void* v_src;
  void* k_dst;              // K area [rows][d]
  void* v_dst;              // V area [rows][d]
  int64_t src_frame0;       // absolute index of the first source frame
  int32_t n_src_frames;
  int32_t esize;            // bytes per element
  int64_t dummy_frame0;     // absolute first frame of the newest block (Dummy target)
  Geom g;
  HeadSlot heads[HC_MAX_HEADS];
};
cudaError_t launch_scatter(const ScatterParams& p, cudaStream_t s);

}  // namespace hc
