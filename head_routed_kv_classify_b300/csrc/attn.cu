// Softmax attention over per-item key sets.
//
// One CTA processes one work item: up to BM queries of one head against a
// key set that is either one contiguous run of rows (Sink, Dummy, Global,
// full attention, and a Spatial cell in the cell-major cache), or, for the
// classification proxy, the (2r+1)-row band of every window frame with a
// per-element |dh| <= r, |dw| <= r mask.  Online softmax (running max and
// sum, rescaled accumulator) over key tiles; rows are normalised at the end.
// [Pith review of HeadCast: "What carries the argument" (proxies), major
//  comment 2 (r = 2 neighbourhood, 10x10 deployed cells), Figure 3 caption.]
//
// This file holds the fp32 path (the tiny fp32 layer): a SIMT kernel with
// fp32 arithmetic, one warp per query row.  bf16 layers run on the
// tensor-core kernel in attn_tc.cu.
#include <math_constants.h>

#include "hc_internal.h"

namespace hc {
namespace {

constexpr int kBM = 64;   // queries per item tile

// ---------------------------------------------------------------------------
// Work-item decoding.

struct Item {
  int head, kind, q0, nq, out_plane;
  int64_t k_row0;
  int k_len;
  int h0, w0, hz, wz;           // ITEM_CELL: the cell
  int rlo, range_len, tpr;      // ITEM_PROXY: first band row, keys per frame band, tiles per band
  int n_tiles;
};

template <int BN>
__device__ __forceinline__ Item decode_item(const AttnParams& p) {
  const Geom& g = p.g;
  Item it;
  it.h0 = it.w0 = it.hz = it.wz = 0;
  it.rlo = it.range_len = it.tpr = 0;
  if (p.item_mode == ITEMS_LIST) {
    const WorkItem w = p.items[blockIdx.x];
    it.head = w.head;
    it.kind = w.kind;
    it.q0 = w.q0;
    it.nq = w.nq;
    it.out_plane = w.out_plane;
    it.k_row0 = w.k_row0;
    it.k_len = w.k_per_frame > 0 ? w.k_per_frame * p.valid_frames : w.k_len;
    if (w.kind == ITEM_CELL) {
      int ci = w.cell / g.ncell_w, cj = w.cell % g.ncell_w;
      it.h0 = ci * g.cell_h;
      it.hz = cell_extent(ci, g.Fh, g.cell_h, g.ncell_h);
      it.w0 = cj * g.cell_w;
      it.wz = cell_extent(cj, g.Fw, g.cell_w, g.ncell_w);
    } else if (w.kind == ITEM_BAND) {
      // Sliding Spatial: band of window rows over the head's filled ring slots.
      const int t0 = w.q0 % g.F;
      int hmin = t0 / g.Fw, hmax = (t0 + it.nq - 1) / g.Fw;
      int lo, hi, wl, wh, rhi;
      band_window(g, p.band_win, hmin, 0, it.rlo, hi, wl, wh);
      band_window(g, p.band_win, hmax, 0, lo, rhi, wl, wh);
      it.range_len = (rhi - it.rlo + 1) * g.Fw;
      it.tpr = (it.range_len + BN - 1) / BN;
      it.k_len = p.valid_frames * it.range_len;
    }
  } else if (p.item_mode == ITEMS_DENSE) {
    it.head = blockIdx.y;
    it.kind = ITEM_RANGE;
    it.q0 = blockIdx.x * kBM;
    it.nq = min(kBM, p.nq_total - it.q0);
    it.out_plane = blockIdx.z;
    it.k_row0 = p.plane_k0[blockIdx.z];
    it.k_len = p.plane_klen[blockIdx.z];
  } else {  // ITEMS_PROXY: a tile of queries inside one frame of the block
    int f = blockIdx.x / p.tiles_per_frame, t = blockIdx.x % p.tiles_per_frame;
    it.head = blockIdx.y;
    it.kind = ITEM_PROXY;
    it.q0 = f * g.F + t * kBM;
    it.nq = min(kBM, g.F - t * kBM);
    it.out_plane = 3;
    it.k_row0 = 0;
    int hmin = (t * kBM) / g.Fw;
    int hmax = (t * kBM + it.nq - 1) / g.Fw;
    int lo, hi, wl, wh, rhi;
    band_window(g, WIN_PROXY, hmin, 0, it.rlo, hi, wl, wh);
    band_window(g, WIN_PROXY, hmax, 0, lo, rhi, wl, wh);
    it.range_len = (rhi - it.rlo + 1) * g.Fw;
    it.tpr = (it.range_len + BN - 1) / BN;
    it.k_len = p.proxy_frames * it.range_len;
  }
  if (it.kind == ITEM_PROXY)
    it.n_tiles = p.proxy_frames * it.tpr;
  else if (it.kind == ITEM_BAND)
    it.n_tiles = p.valid_frames * it.tpr;
  else
    it.n_tiles = it.k_len > 0 ? (it.k_len + BN - 1) / BN : 0;
  return it;
}

// Block-local token of the r-th query of an item.
__device__ __forceinline__ int query_token(const Item& it, const Geom& g, int r) {
  if (it.kind != ITEM_CELL) return it.q0 + r;
  int ord = it.q0 + r;
  int csz = it.hz * it.wz;
  int fq = ord / csz, rem = ord - fq * csz;
  int hh = rem / it.wz, ww = rem - hh * it.wz;
  return fq * g.F + (it.h0 + hh) * g.Fw + it.w0 + ww;
}

// First key row of tile t, the number of valid keys in it, and (PROXY) the
// within-frame position of its first key.
template <int BN>
__device__ __forceinline__ void tile_rows(const Item& it, const Geom& g, int t, int64_t& row,
                                          int& valid, int& pos0) {
  if (it.kind == ITEM_PROXY || it.kind == ITEM_BAND) {
    int f = t / it.tpr, o = (t - f * it.tpr) * BN;
    pos0 = it.rlo * g.Fw + o;
    row = it.k_row0 + (int64_t)f * g.F + pos0;
    valid = min(BN, it.range_len - o);
  } else {
    row = it.k_row0 + (int64_t)t * BN;
    valid = min(BN, it.k_len - t * BN);
    pos0 = 0;
  }
}

// ---------------------------------------------------------------------------
// fp32 SIMT kernel: one warp per query row; 32 keys per step, one per lane;
// each lane owns head_dim/32 output channels.

template <int D>
__global__ void __launch_bounds__(128) attn_f32_kernel(const AttnParams p) {
  constexpr int NW = 4, BN = 32, PER = D / 32;
  __shared__ float sq[NW][D];
  const Geom& g = p.g;
  const Item it = decode_item<BN>(p);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t HD = (int64_t)g.H * D;
  const float* Q = static_cast<const float*>(p.q);
  const float* K = static_cast<const float*>(p.k);
  const float* V = static_cast<const float*>(p.v);
  const int64_t hoff = (int64_t)it.head * p.k_hstride;
  const float sl2 = g.scale_log2;

  for (int r = warp; r < it.nq; r += NW) {
    const int tok = query_token(it, g, r);
    for (int c = lane; c < D; c += 32) sq[warp][c] = Q[tok * HD + it.head * D + c];
    __syncwarp();
    int h_lo = 0, h_hi = 0, w_lo = 0, w_hi = 0;
    const bool band = it.kind == ITEM_PROXY || it.kind == ITEM_BAND;
    if (band) {
      const int tp = tok % g.F;
      const int hq = tp / g.Fw;
      band_window(g, it.kind == ITEM_BAND ? p.band_win : (int)WIN_PROXY, hq, tp - hq * g.Fw, h_lo, h_hi, w_lo,
                  w_hi);
    }
    float m = -CUDART_INF_F, l = 0.f, acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int t = 0; t < it.n_tiles; ++t) {
      int64_t row0;
      int valid, pos0;
      tile_rows<BN>(it, g, t, row0, valid, pos0);
      bool ok = lane < valid;
      if (ok && band) {
        int pos = pos0 + lane;
        int hk = pos / g.Fw, wk = pos - hk * g.Fw;
        ok = hk >= h_lo && hk <= h_hi && wk >= w_lo && wk <= w_hi;
      }
      float x = -CUDART_INF_F;
      if (ok) {
        const float* kr = K + (row0 + lane) * p.k_stride + hoff;
        float dot = 0.f;
        for (int c = 0; c < D; ++c) dot = fmaf(sq[warp][c], kr[c], dot);
        x = dot * sl2;
      }
      float mt = x;
      for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
      const float mn = fmaxf(m, mt);
      const float mu = mn == -CUDART_INF_F ? 0.f : mn;
      const float al = exp2f(m - mu);
      const float pj = exp2f(x - mu);
      float ps = pj;
      for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
      l = l * al + ps;
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] *= al;
      for (int j = 0; j < valid; ++j) {
        const float pb = __shfl_sync(0xffffffffu, pj, j);
        const float* vr = V + (row0 + j) * p.k_stride + hoff;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = fmaf(pb, vr[lane + 32 * i], acc[i]);
      }
      m = mn;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int64_t ob = (int64_t)it.out_plane * p.o_plane_stride + tok * HD + (int64_t)it.head * D;
#pragma unroll
    for (int i = 0; i < PER; ++i) static_cast<float*>(p.o)[ob + lane + 32 * i] = acc[i] * inv;
    __syncwarp();
  }
}

}  // namespace

int attention_block_rows(int dtype, int) { return dtype == HC_BF16 ? tc_block_rows() : kBM; }
int proxy_block_rows() { return kBM; }

cudaError_t launch_attention(const AttnParams& p, int dtype, dim3 grid, cudaStream_t s) {
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  // bf16 layers run on the tensor-core kernel (launch_attention_tc).
  if (dtype != HC_FP32 || p.out_fp32 == 0) return cudaErrorInvalidValue;
  if (p.g.d == 128) {
    attn_f32_kernel<128><<<grid, 128, 0, s>>>(p);
    return cudaGetLastError();
  }
  if (p.g.d == 64) {
    attn_f32_kernel<64><<<grid, 128, 0, s>>>(p);
    return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}

}  // namespace hc
