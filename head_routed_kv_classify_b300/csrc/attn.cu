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
// bf16 inputs run on warp-level tensor-core MMA (m16n8k16, fp32
// accumulate); fp32 inputs run on a SIMT kernel with fp32 arithmetic.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "hc_internal.h"

namespace hc {
namespace {

typedef __nv_bfloat16 bf16;

constexpr int kBM = 64;   // queries per item tile (both kernels)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------------------
// Work-item decoding shared by both kernels.

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
    it.rlo = max(0, hmin - g.radius);
    int rhi = min(g.Fh - 1, hmax + g.radius);
    it.range_len = (rhi - it.rlo + 1) * g.Fw;
    it.tpr = (it.range_len + BN - 1) / BN;
    it.k_len = p.proxy_frames * it.range_len;
  }
  if (it.kind == ITEM_PROXY)
    it.n_tiles = p.proxy_frames * it.tpr;
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
  if (it.kind == ITEM_PROXY) {
    int f = t / it.tpr, o = (t - f * it.tpr) * BN;
    pos0 = it.rlo * g.Fw + o;
    row = (int64_t)f * g.F + pos0;
    valid = min(BN, it.range_len - o);
  } else {
    row = it.k_row0 + (int64_t)t * BN;
    valid = min(BN, it.k_len - t * BN);
    pos0 = 0;
  }
}

// ---------------------------------------------------------------------------
// bf16 tensor-core kernel: 4 warps x 16 query rows, 64-key tiles, cp.async
// double buffering, XOR-swizzled shared tiles read with ldmatrix.

__device__ __forceinline__ int swz(int r, int ch, int D) { return r * D + ((ch ^ (r & 7)) << 3); }

template <int D>
__global__ void __launch_bounds__(128) attn_bf16_kernel(const AttnParams p) {
  constexpr int NW = 4, BM = kBM, BN = 64, CPR = D / 8;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  bf16* sQ = reinterpret_cast<bf16*>(smem_raw);
  bf16* sK = sQ + BM * D;
  bf16* sV = sK + 2 * BN * D;

  const Geom& g = p.g;
  const Item it = decode_item<BN>(p);
  if (it.nq <= 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t HD = (int64_t)g.H * D;
  const bf16* Q = static_cast<const bf16*>(p.q);
  const bf16* K = static_cast<const bf16*>(p.k);
  const bf16* V = static_cast<const bf16*>(p.v);

  for (int c = tid; c < BM * CPR; c += NW * 32) {
    int r = c / CPR, ch = c - r * CPR;
    bool ok = r < it.nq;
    int tok = ok ? query_token(it, g, r) : 0;
    cp_async16(smem_u32(sQ + swz(r, ch, D)), Q + tok * HD + it.head * D + ch * 8, ok);
  }
  cp_async_commit();

  auto load_kv = [&](int t, int stage) {
    int64_t row0;
    int valid, pos0;
    tile_rows<BN>(it, g, t, row0, valid, pos0);
    const int64_t hoff = (int64_t)it.head * p.k_hstride;
    for (int c = tid; c < BN * CPR; c += NW * 32) {
      int r = c / CPR, ch = c - r * CPR;
      bool ok = r < valid;
      int64_t off = (row0 + (ok ? r : 0)) * p.k_stride + hoff + ch * 8;
      cp_async16(smem_u32(sK + stage * BN * D + swz(r, ch, D)), K + off, ok);
      cp_async16(smem_u32(sV + stage * BN * D + swz(r, ch, D)), V + off, ok);
    }
  };

  if (it.n_tiles > 0) load_kv(0, 0);
  cp_async_commit();
  cp_async_wait<1>();
  __syncthreads();

  uint32_t qf[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    int r = warp * 16 + (lane & 15), ch = kk * 2 + (lane >> 4);
    ldsm_x4(smem_u32(sQ + swz(r, ch, D)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }

  // Query positions of this thread's two rows (for the proxy mask).
  const int qr0 = warp * 16 + (lane >> 2), qr1 = qr0 + 8;
  int hq0 = 0, wq0 = 0, hq1 = 0, wq1 = 0;
  if (it.kind == ITEM_PROXY) {
    int t0 = (query_token(it, g, qr0) % g.F), t1 = (query_token(it, g, qr1) % g.F);
    hq0 = t0 / g.Fw; wq0 = t0 - hq0 * g.Fw;
    hq1 = t1 / g.Fw; wq1 = t1 - hq1 * g.Fw;
  }

  float acc[D / 8][4];
#pragma unroll
  for (int j = 0; j < D / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  const float sl2 = g.scale_log2;

  for (int t = 0; t < it.n_tiles; ++t) {
    const int st = t & 1;
    if (t + 1 < it.n_tiles) load_kv(t + 1, st ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const bf16* cK = sK + st * BN * D;
    const bf16* cV = sV + st * BN * D;
    float s[BN / 8][4];
#pragma unroll
    for (int j = 0; j < BN / 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < BN / 16; ++np) {
        int r = np * 16 + ((lane >> 4) << 3) + (lane & 7);
        int ch = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(cK + swz(r, ch, D)), b0, b1, b2, b3);
        mma_bf16(s[2 * np], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b0, b1);
        mma_bf16(s[2 * np + 1], qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3], b2, b3);
      }
    }

    int64_t trow;
    int valid, pos0;
    tile_rows<BN>(it, g, t, trow, valid, pos0);
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < BN / 8; ++j) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        int col = j * 8 + 2 * (lane & 3) + e;
        bool ok0 = col < valid, ok1 = ok0;
        if (it.kind == ITEM_PROXY && ok0) {
          int pos = pos0 + col;
          int hk = pos / g.Fw, wk = pos - hk * g.Fw;
          ok0 = abs(hk - hq0) <= g.radius && abs(wk - wq0) <= g.radius;
          ok1 = abs(hk - hq1) <= g.radius && abs(wk - wq1) <= g.radius;
        }
        s[j][e] = ok0 ? s[j][e] * sl2 : -CUDART_INF_F;
        s[j][2 + e] = ok1 ? s[j][2 + e] * sl2 : -CUDART_INF_F;
        mx0 = fmaxf(mx0, s[j][e]);
        mx1 = fmaxf(mx1, s[j][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mu0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
    const float mu1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
    const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int j = 0; j < BN / 8; ++j) {
      s[j][0] = exp2f(s[j][0] - mu0);
      s[j][1] = exp2f(s[j][1] - mu0);
      s[j][2] = exp2f(s[j][2] - mu1);
      s[j][3] = exp2f(s[j][3] - mu1);
      rs0 += s[j][0] + s[j][1];
      rs1 += s[j][2] + s[j][3];
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      acc[j][0] *= al0;
      acc[j][1] *= al0;
      acc[j][2] *= al1;
      acc[j][3] *= al1;
    }
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
      uint32_t a0 = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      uint32_t a1 = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      uint32_t a2 = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      uint32_t a3 = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        int r = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        int ch = dp * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(cV + swz(r, ch, D)), b0, b1, b2, b3);
        mma_bf16(acc[2 * dp], a0, a1, a2, a3, b0, b1);
        mma_bf16(acc[2 * dp + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
  const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const bool w0 = qr0 < it.nq, w1 = qr1 < it.nq;
  const int64_t tok0 = w0 ? query_token(it, g, qr0) : 0;
  const int64_t tok1 = w1 ? query_token(it, g, qr1) : 0;
  const int64_t base = (int64_t)it.out_plane * p.o_plane_stride + (int64_t)it.head * D;
#pragma unroll
  for (int j = 0; j < D / 8; ++j) {
    int col = j * 8 + 2 * (lane & 3);
    if (p.out_fp32) {
      float* O = static_cast<float*>(p.o) + base + col;
      if (w0) *reinterpret_cast<float2*>(O + tok0 * HD) = make_float2(acc[j][0] * inv0, acc[j][1] * inv0);
      if (w1) *reinterpret_cast<float2*>(O + tok1 * HD) = make_float2(acc[j][2] * inv1, acc[j][3] * inv1);
    } else {
      bf16* O = static_cast<bf16*>(p.o) + base + col;
      if (w0)
        *reinterpret_cast<__nv_bfloat162*>(O + tok0 * HD) =
            __floats2bfloat162_rn(acc[j][0] * inv0, acc[j][1] * inv0);
      if (w1)
        *reinterpret_cast<__nv_bfloat162*>(O + tok1 * HD) =
            __floats2bfloat162_rn(acc[j][2] * inv1, acc[j][3] * inv1);
    }
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
    int hq = 0, wq = 0;
    if (it.kind == ITEM_PROXY) {
      int tp = tok % g.F;
      hq = tp / g.Fw;
      wq = tp - hq * g.Fw;
    }
    float m = -CUDART_INF_F, l = 0.f, acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    for (int t = 0; t < it.n_tiles; ++t) {
      int64_t row0;
      int valid, pos0;
      tile_rows<BN>(it, g, t, row0, valid, pos0);
      bool ok = lane < valid;
      if (ok && it.kind == ITEM_PROXY) {
        int pos = pos0 + lane;
        int hk = pos / g.Fw, wk = pos - hk * g.Fw;
        ok = abs(hk - hq) <= g.radius && abs(wk - wq) <= g.radius;
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

template <int D>
constexpr int bf16_smem_bytes() {
  return (kBM + 4 * 64) * D * 2;
}

template <int D>
cudaError_t launch_bf16(const AttnParams& p, dim3 grid, cudaStream_t s) {
  constexpr int smem = bf16_smem_bytes<D>();
  static bool configured = false;  // attribute is per function, per process
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_bf16_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  attn_bf16_kernel<D><<<grid, 128, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

int attention_block_rows(int dtype, int) { return dtype == HC_BF16 ? tc_block_rows() : kBM; }
int proxy_block_rows() { return kBM; }

cudaError_t launch_attention(const AttnParams& p, int dtype, dim3 grid, cudaStream_t s) {
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  if (dtype == HC_BF16) {
    if (p.g.d == 128) return launch_bf16<128>(p, grid, s);
    if (p.g.d == 64) return launch_bf16<64>(p, grid, s);
  } else {
    if (p.out_fp32 == 0) return cudaErrorInvalidValue;
    if (p.g.d == 128) {
      attn_f32_kernel<128><<<grid, 128, 0, s>>>(p);
      return cudaGetLastError();
    }
    if (p.g.d == 64) {
      attn_f32_kernel<64><<<grid, 128, 0, s>>>(p);
      return cudaGetLastError();
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace hc
