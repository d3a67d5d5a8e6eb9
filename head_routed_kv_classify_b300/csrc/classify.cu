// Classification statistics and the archetype decision.
//
// Per token and head: cosines between the full-context output and the Sink,
// Dummy and Spatial-proxy outputs, and the squared error of the proxy.  Per
// head: the three mean cosines, the 5th percentile of the proxy cosine
// (linear interpolation between the order statistics at rank 0.05*(Nq-1),
// selected exactly by radix select on the fp32 values), MSE over tokens and
// channels, score = P5 - gamma*MSE, and the first archetype to clear its
// gate in the order Sink, Dummy, Spatial (which also needs the score gate);
// Global otherwise.  Means, P5 interpolation and the comparisons are done in
// fp64.  [Pith review of HeadCast, "What carries the argument"; Ledger:
//  theta = 0.95, theta_sc = 0.755, gamma = 5.]
#include <cuda_bf16.h>

#include "hc_internal.h"

namespace hc {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Cosine with the convention cos(0, 0) = 1 and cos(x, 0) = 0.
__device__ __forceinline__ float cosine(float dot, float na2, float nb2) {
  if (na2 == 0.f && nb2 == 0.f) return 1.f;
  if (na2 == 0.f || nb2 == 0.f) return 0.f;
  return dot / (sqrtf(na2) * sqrtf(nb2));
}

// A set status word means an attention launch of this classification gave
// up on a bounded wait: its output planes are incomplete.
__device__ __forceinline__ bool planes_incomplete(const ClassifyPost& c) {
  return c.status && *reinterpret_cast<const volatile int*>(c.status) != DEV_OK;
}

// One warp per (token, head) row.
__global__ void cos_kernel(const ClassifyPost c) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int H = c.g.H, d = c.g.d;
  if (gw >= c.nq * H || planes_incomplete(c)) return;
  const int i = gw / H, h = gw - i * H;
  const int64_t row = ((int64_t)i * H + h) * d;
  const float* pf = c.planes + row;
  const float* ps = pf + c.plane_stride;
  const float* pd = ps + c.plane_stride;
  const float* pp = pd + c.plane_stride;
  float ff = 0, ss = 0, dd = 0, qq = 0, fs = 0, fd = 0, fq = 0, se = 0;
  for (int k = lane; k < d; k += 32) {
    float f = pf[k], s = ps[k], dm = pd[k], q = pp[k];
    ff = fmaf(f, f, ff);
    ss = fmaf(s, s, ss);
    dd = fmaf(dm, dm, dd);
    qq = fmaf(q, q, qq);
    fs = fmaf(f, s, fs);
    fd = fmaf(f, dm, fd);
    fq = fmaf(f, q, fq);
    float e = q - f;
    se = fmaf(e, e, se);
    if (c.o_full) {
      if (c.o_full_fp32)
        static_cast<float*>(c.o_full)[row + k] = f;
      else
        static_cast<__nv_bfloat16*>(c.o_full)[row + k] = __float2bfloat16_rn(f);
    }
  }
  ff = warp_sum(ff); ss = warp_sum(ss); dd = warp_sum(dd); qq = warp_sum(qq);
  fs = warp_sum(fs); fd = warp_sum(fd); fq = warp_sum(fq); se = warp_sum(se);
  if (lane == 0) {
    const int64_t n = c.nq;
    c.tok[(0 * (int64_t)H + h) * n + i] = cosine(fs, ff, ss);
    c.tok[(1 * (int64_t)H + h) * n + i] = cosine(fd, ff, dd);
    c.tok[(2 * (int64_t)H + h) * n + i] = cosine(fq, ff, qq);
    c.tok[(3 * (int64_t)H + h) * n + i] = se;
  }
}

// Order-preserving map of fp32 to uint32 and back.
__device__ __forceinline__ uint32_t f2key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

constexpr int kRedThreads = 1024;

// Exact k-th smallest (0-based) of x[0..n) by four 8-bit radix passes.
__device__ float block_select(const float* x, int n, int k, uint32_t* hist, int* sh) {
  uint32_t prefix = 0, mask = 0;
  int kk = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      uint32_t u = f2key(x[i]);
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // The bin holding rank kk: lane l sums bins [8l, 8l+8), an inclusive
      // scan over the lanes finds the first lane whose running count passes
      // kk, and that lane walks its eight bins.
      const int lane = threadIdx.x;
      uint32_t own[8];
      int sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        own[j] = hist[8 * lane + j];
        sum += (int)own[j];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, incl > kk);
      const int first = hit ? __ffs(hit) - 1 : 31;
      if (lane == first) {
        int cum = incl - sum, sel = 8 * lane + 7;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cum + (int)own[j] > kk) {
            sel = 8 * lane + j;
            break;
          }
          cum += (int)own[j];
        }
        sh[0] = sel;
        sh[1] = kk - cum;
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sh[0] << shift;
    mask |= 255u << shift;
    kk = sh[1];
    __syncthreads();
  }
  return key2f(prefix);
}

// Given v = the k-th smallest of x (0-based), the (k+1)-th: v itself when
// more than k+1 values are <= v, else the smallest value above v.  One pass.
__device__ float block_select_next(const float* x, int n, int k, float v, uint32_t* hist, int* sh) {
  const uint32_t kv = f2key(v);
  int le = 0;
  uint32_t gt = 0xffffffffu;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t u = f2key(x[i]);
    if (u <= kv) ++le;
    else gt = min(gt, u);
  }
  for (int o = 16; o > 0; o >>= 1) {
    le += __shfl_xor_sync(0xffffffffu, le, o);
    gt = min(gt, __shfl_xor_sync(0xffffffffu, gt, o));
  }
  if (threadIdx.x == 0) {
    sh[0] = 0;
    hist[0] = 0xffffffffu;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    atomicAdd(&sh[0], le);
    atomicMin(&hist[0], gt);
  }
  __syncthreads();
  const float r = sh[0] > k + 1 ? v : key2f(hist[0]);
  __syncthreads();
  return r;
}

__device__ double block_sum(double v, double* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[w] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0) {
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];
    red[32] = t;
  }
  __syncthreads();
  t = red[32];
  __syncthreads();
  return t;
}

__global__ void __launch_bounds__(kRedThreads) reduce_kernel(const ClassifyPost c) {
  __shared__ uint32_t hist[256];
  __shared__ int sh[2];
  __shared__ double red[33];
  __shared__ int incomplete;
  const int h = blockIdx.x, H = c.g.H, n = c.nq;
  // Read once and shared, so that the whole block takes the same branch.
  if (threadIdx.x == 0) incomplete = planes_incomplete(c) ? 1 : 0;
  __syncthreads();
  if (incomplete) {
    // No label can be decided: mark the head with an invalid label (-1),
    // which the cache calls reject.
    if (threadIdx.x == 0) c.labels[h] = -1;
    return;
  }
  const float* cs = c.tok + (0 * (int64_t)H + h) * n;
  const float* cd = c.tok + (1 * (int64_t)H + h) * n;
  const float* cp = c.tok + (2 * (int64_t)H + h) * n;
  const float* se = c.tok + (3 * (int64_t)H + h) * n;
  double a = 0, b = 0, e = 0, q = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    a += cs[i];
    b += cd[i];
    e += cp[i];
    q += se[i];
  }
  const double s_cs = block_sum(a, red), s_cd = block_sum(b, red);
  const double s_cp = block_sum(e, red), s_se = block_sum(q, red);
  const double pos = 0.05 * (double)(n - 1);
  const int lo = (int)floor(pos);
  const int hi = lo + 1 < n ? lo + 1 : n - 1;
  const float flo = block_select(cp, n, lo, hist, sh);
  const double vlo = flo;
  const double vhi = hi == lo ? vlo : (double)block_select_next(cp, n, lo, flo, hist, sh);
  if (threadIdx.x == 0) {
    const double c_s = s_cs / n, c_d = s_cd / n, c_sp = s_cp / n;
    const double p5 = vlo + (pos - lo) * (vhi - vlo);
    const double mse = s_se / ((double)n * c.g.d);
    const double score = p5 - (double)c.gamma * mse;
    int8_t label;
    if (c_s >= (double)c.theta_sink)
      label = HC_SINK;
    else if (c_d >= (double)c.theta_dummy)
      label = HC_DUMMY;
    else if (c_sp >= (double)c.theta_spatial && score >= (double)c.theta_score)
      label = HC_SPATIAL;
    else
      label = HC_GLOBAL;
    c.labels[h] = label;
    if (c.stats) {
      float* st = c.stats + h * 6;
      st[0] = (float)c_s;
      st[1] = (float)c_d;
      st[2] = (float)c_sp;
      st[3] = (float)p5;
      st[4] = (float)mse;
      st[5] = (float)score;
    }
  }
}

}  // namespace

cudaError_t launch_classify_post(const ClassifyPost& c, cudaStream_t s) {
  const int64_t rows = (int64_t)c.nq * c.g.H;
  const int threads = 256;
  const int64_t blocks = (rows * 32 + threads - 1) / threads;
  if (!c.tokens_ready) {
    cos_kernel<<<(unsigned)blocks, threads, 0, s>>>(c);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  reduce_kernel<<<c.g.H, kRedThreads, 0, s>>>(c);
  return cudaGetLastError();
}

}  // namespace hc
