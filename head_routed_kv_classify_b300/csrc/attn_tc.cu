// Softmax attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// with K/V tiles streamed by TMA.  Serves every bf16 attention of the
// library: the routed pathways (Sink / Dummy / Global key runs and Spatial
// cells of the restructured cache), the in-house full attention and the
// full / Sink / Dummy planes of classification.
// [Pith review of HeadCast: "The pith" and "Core claim" (each head attends
//  only over its pathway), "What carries the argument" (the classification
//  outputs), major comment 2 and Figure 3 caption (10x10 cells).]
//
// One CTA computes one work item: up to 256 queries of one head (two query
// tiles of 128) against one contiguous run of key rows, streamed in tiles of
// 128 keys.  Roles (320 threads):
//   warps 0-3, 4-7  softmax groups, one per query tile: thread r of group i
//              owns row r of tile i, i.e. TMEM lane r.  It reads its row of
//              S_i = Q_i K^T from TMEM (a max pass, then an exponent pass),
//              keeps the running max and sum, writes P_i (bf16, two per
//              32-bit column) back over the first half of S_i and, when the
//              max has grown by more than 2^8, rescales its row of O_i; at
//              the end it normalises O_i and stores it.
//   warp 8     TMA producer: K and V tiles into 2-stage rings.  V(j) and
//              K(j+1) travel together on one barrier, so the MMA issuer
//              makes one data wait and one release commit per key tile:
//              each barrier poll between two MMA batches leaves the tensor
//              pipe idle, since an MMA issue returns only once the pipe
//              accepts it.
//   warp 9     MMA issuer, in the order P_0 V, S_0, P_1 V, S_1 per key tile,
//              so the tensor core always has the other tile's products
//              queued while a softmax group works.  S uses Q and K from
//              shared memory; P V reads P from TMEM and V from shared memory.
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 after it.
// P_i(j) overwrites S_i(j) once it has been read; S_i(j+1) is written there
// only by an MMA issued after P_i(j) V(j), and MMAs issued by one thread
// execute in order.  The commit that signals S_i(j) also covers
// P_i(j-1) V(j-1), so a softmax group may rescale O_i as soon as it sees
// S_i(j).
// Band items -- the classification proxy (ITEMS_PROXY) and, with sliding
// deployed Spatial heads, their routed items (ITEM_BAND) -- run the same
// pipeline on the band of frame rows around a run of query tokens in every
// frame, with a per-row window mask (the (2r+1) x (2r+1) neighbourhood, the
// deployed cell, or the centred cell_h x cell_w window) applied to S.
// Hand-offs are mbarriers; every wait is bounded in wall-clock time and on
// expiry the CTA records HC_ERR_TIMEOUT in the status word, drains its own
// copies and MMAs (again bounded), frees TMEM and returns.
//
// Shared-memory operand layouts are the canonical 128-byte-swizzle ones:
// Q and K are K-major (rows of 64 bf16 = 128 B, 8-row atoms of 1 KB, one
// region per 64 columns); V is the MN-major B operand of P V (rows are keys,
// 128 B per 64 channels of d).
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

#include "hc_internal.h"

namespace hc {
namespace {

typedef __nv_bfloat16 bf16;

constexpr int BM = 128;            // queries per tile (one MMA M)
constexpr int QT = 2;              // query tiles per CTA
constexpr int BN = 128;            // keys per tile
constexpr int STAGES = 2;          // K and V ring depth
constexpr int NTHREADS = 320;
constexpr int W_PRODUCER = 8, W_MMA = 9;
constexpr uint32_t TMEM_COLS = 512;
constexpr float RESCALE_LOG2 = 8.f;  // rescale O when the row max grows by > 2^8
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;   // 1 s
constexpr unsigned long long STALL_WAIT_LIMIT_NS = 2000000ull; // 2 ms under the stall test hook
constexpr unsigned long long DRAIN_LIMIT_NS = 200000000ull;   // 0.2 s

template <int D>
struct Layout {
  static constexpr int NREG = D / 64;               // 64-column regions along d
  static constexpr int Q_REG = BM * 128;
  static constexpr int Q_BYTES = NREG * Q_REG;       // one query tile
  static constexpr int KV_REG = BN * 128;
  static constexpr int KV_BYTES = NREG * KV_REG;    // one K (or V) tile
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;
  static constexpr int BYTES = OFF_BAR + 256;
  static constexpr int ALLOC = BYTES + 1024;        // room to align the base to 1 KB
  static constexpr uint32_t COL_O = QT * BN;        // O_i at COL_O + i * D
  static_assert(COL_O + QT * D <= TMEM_COLS, "TMEM budget");
};

// Barrier slots (8 bytes each) after OFF_BAR.  Tile j's loads travel in
// load group j: V(j) and K(j+1) on one FULL barrier (K(0) alone on K0FULL);
// one EMPTY commit after the last MMA of key tile j releases both stages.
// S_0 has its own barrier (SFULL); S_1(j) is signalled by the EMPTY commit
// that follows it, which tracks the same MMAs.
enum { B_K0FULL = 0, B_FULL = 1, B_EMPTY = B_FULL + STAGES, B_SFULL = B_EMPTY + STAGES, B_PFULL = B_SFULL + 1,
       B_ODONE = B_PFULL + QT, B_FIN = B_ODONE + QT, B_COUNT = B_FIN + 1 };
// The barriers, the TMEM slot and the two flags fit the 256 bytes after OFF_BAR.
static_assert(8 * B_COUNT + 12 <= 256, "barrier area");

struct TcArgs {
  CUtensorMap tk;        // K as [rows][heads][D] (3-D map, box {64, 1, BN})
  CUtensorMap tv;        // V, same shape
  AttnParams p;
  int32_t kv_head_coord; // 1: the map's middle coordinate is the head; 0: always 0
};

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until phase `parity` of `bar` has completed, for at most `limit` ns
// or until another role has raised the CTA's abort flag.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                            unsigned long long limit) {
  const unsigned long long t0 = now_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (now_ns() - t0 > limit) return false;
  }
}

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  unsigned long long limit) {
  if (mbar_try(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, limit);
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 form): start address, leading and
// stride byte offsets (all >> 4), fixed version bits 46..48 = 0b001, and the
// 128-byte swizzle mode (2) in bits 61..63.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B,
// A K-major, B K-major or MN-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// As above with A (M x 16, K-major) read from TMEM at column a_tmem.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

#define HC_R32(i) "=r"(r[i])
#define HC_R32_8(b) HC_R32(b), HC_R32(b + 1), HC_R32(b + 2), HC_R32(b + 3), HC_R32(b + 4), HC_R32(b + 5), \
                    HC_R32(b + 6), HC_R32(b + 7)
// 32 consecutive TMEM columns of this thread's lane, waited for in the same
// asm statement so that no use of the registers can be scheduled before the
// load has completed.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : HC_R32_8(0), HC_R32_8(8), HC_R32_8(16), HC_R32_8(24)
      : "r"(taddr)
      : "memory");
}
// Two runs of 32 columns (64 registers) with one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t taddr0, uint32_t taddr1, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : HC_R32_8(0), HC_R32_8(8), HC_R32_8(16), HC_R32_8(24), HC_R32_8(32), HC_R32_8(40), HC_R32_8(48),
        HC_R32_8(56)
      : "r"(taddr0), "r"(taddr1)
      : "memory");
}
// 64 consecutive TMEM columns of this thread's lane together with their
// maximum, reduced by the load itself (tcgen05.ld.red), so that a tile
// without masked keys needs no max instructions.
__device__ __forceinline__ float tmem_ld64_max(uint32_t taddr, uint32_t* r) {
  float m;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x64.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,"
      "%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, %64, [%65];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : HC_R32_8(0), HC_R32_8(8), HC_R32_8(16), HC_R32_8(24), HC_R32_8(32), HC_R32_8(40), HC_R32_8(48),
        HC_R32_8(56), "=f"(m)
      : "r"(taddr)
      : "memory");
  return m;
}
#undef HC_R32
#define HC_W32(i) "r"(r[i])
#define HC_W32_8(b) HC_W32(b), HC_W32(b + 1), HC_W32(b + 2), HC_W32(b + 3), HC_W32(b + 4), HC_W32(b + 5), \
                    HC_W32(b + 6), HC_W32(b + 7)
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), HC_W32_8(0), HC_W32_8(8), HC_W32_8(16), HC_W32_8(24)
      : "memory");
}
#undef HC_W32
#undef HC_R32_8
#undef HC_W32_8
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// (d0, d1) = (a0, a1) * b + c as one packed two-lane fp32 FMA.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n mov.b64 rc, {%5, %5};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (s0, s1) += (a0, a1) as one packed two-lane fp32 add.
__device__ __forceinline__ void add2(float& s0, float& s1, float a0, float a1) {
  asm("{\n .reg .b64 rs, ra;\n mov.b64 rs, {%0, %1};\n mov.b64 ra, {%2, %3};\n add.rn.f32x2 rs, rs, ra;\n"
      " mov.b64 {%0, %1}, rs;\n}\n"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ---------------------------------------------------------------- work items

struct TcItem {
  int head, kind, q0, nq, out_plane;
  int64_t k_row0;
  int k_len;
  int h0, w0, hz, wz;   // ITEM_CELL: the cell
  int rlo, rlen, tpf;   // band items: first band row, keys per frame band, key tiles per frame
};

// Band of frame rows [h_lo(first row), h_hi(last row)] of a run of queries
// [t0, t0 + nq) inside one frame, over `frames` frames of keys.
__device__ __forceinline__ void tc_band(TcItem& it, const Geom& g, int win, int t0, int frames) {
  const int hmin = t0 / g.Fw, hmax = (t0 + it.nq - 1) / g.Fw;
  int lo, rhi, wl, wh;
  band_window(g, win, hmin, 0, it.rlo, rhi, wl, wh);
  band_window(g, win, hmax, 0, lo, rhi, wl, wh);
  it.rlen = (rhi - it.rlo + 1) * g.Fw;
  it.tpf = (it.rlen + BN - 1) / BN;
  it.k_len = frames * it.tpf * BN;
}

__device__ __forceinline__ TcItem tc_decode(const AttnParams& p) {
  const Geom& g = p.g;
  TcItem it;
  it.h0 = it.w0 = it.hz = it.wz = 0;
  it.rlo = it.rlen = it.tpf = 0;
  if (p.item_mode == ITEMS_PROXY) {
    // Up to 256 consecutive tokens of one frame of the block; keys: the
    // rows [h_min - r, h_max + r] of every window frame (one contiguous run
    // of tokens per frame), narrowed per query by the neighbourhood mask.
    const int f = blockIdx.x / p.tiles_per_frame, t0 = (blockIdx.x % p.tiles_per_frame) * (QT * BM);
    it.head = blockIdx.y;
    it.kind = ITEM_PROXY;
    it.q0 = f * g.F + t0;
    it.nq = min(QT * BM, g.F - t0);
    it.out_plane = 3;
    it.k_row0 = 0;
    tc_band(it, g, WIN_PROXY, t0, p.proxy_frames);
  } else if (p.item_mode == ITEMS_LIST) {
    const WorkItem w = p.items[blockIdx.x];
    it.head = w.head;
    it.kind = w.kind;
    it.q0 = w.q0;
    it.nq = w.nq;
    it.out_plane = w.out_plane;
    it.k_row0 = w.k_row0;
    it.k_len = w.k_per_frame > 0 ? w.k_per_frame * p.valid_frames : w.k_len;
    if (w.kind == ITEM_CELL) {
      const int ci = w.cell / g.ncell_w, cj = w.cell % g.ncell_w;
      it.h0 = ci * g.cell_h;
      it.hz = cell_extent(ci, g.Fh, g.cell_h, g.ncell_h);
      it.w0 = cj * g.cell_w;
      it.wz = cell_extent(cj, g.Fw, g.cell_w, g.ncell_w);
    } else if (w.kind == ITEM_BAND) {
      // Sliding Spatial: the head's ring slots in raster order from k_row0.
      tc_band(it, g, p.band_win, w.q0 % g.F, p.valid_frames);
    }
  } else {  // ITEMS_DENSE
    it.head = blockIdx.y;
    it.kind = ITEM_RANGE;
    it.q0 = blockIdx.x * (QT * BM);
    it.nq = min(QT * BM, p.nq_total - it.q0);
    it.out_plane = blockIdx.z;
    it.k_row0 = p.plane_k0[blockIdx.z];
    it.k_len = p.plane_klen[blockIdx.z];
  }
  return it;
}

// Block-local token of the r-th query of an item.
__device__ __forceinline__ int tc_query_token(const TcItem& it, const Geom& g, int r) {
  if (it.kind != ITEM_CELL) return it.q0 + r;
  const int ord = it.q0 + r;
  const int csz = it.hz * it.wz;
  const int fq = ord / csz, rem = ord - fq * csz;
  const int hh = rem / it.wz, ww = rem - hh * it.wz;
  return fq * g.F + (it.h0 + hh) * g.Fw + it.w0 + ww;
}

// ---------------------------------------------------------------- the kernel

template <int D, bool PROXY>
__global__ void __launch_bounds__(NTHREADS, 1) attn_tc_kernel(const __grid_constant__ TcArgs args) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + L::OFF_Q, sK = s_base + L::OFF_K, sV = s_base + L::OFF_V;
  const uint32_t bars = s_base + L::OFF_BAR;
  auto bar = [&](int slot) { return bars + 8u * slot; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_BAR + 8 * B_COUNT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * B_COUNT + 4);
  volatile int* skip_flag = reinterpret_cast<volatile int*>(smem + L::OFF_BAR + 8 * B_COUNT + 8);

  const AttnParams& p = args.p;
  const Geom& g = p.g;
  const unsigned long long wait_limit = p.wait_limit_ns;
  // Once any CTA has recorded an expired wait, the rest of the launch (and
  // later launches, until the status word is read and cleared) skip their
  // work so that a broken pipeline fails fast.
  if (threadIdx.x == 0) *skip_flag = p.status ? *reinterpret_cast<volatile int*>(p.status) : 0;
  __syncthreads();
  if (*skip_flag) return;
  const TcItem it = tc_decode(p);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = it.k_len > 0 ? (it.k_len + BN - 1) / BN : 0;
  const bool two = it.nq > BM;   // second query tile in use
  const int64_t HD = (int64_t)g.H * D;

  if (tid == 0) {
    mbar_init(bar(B_K0FULL), 1);
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(bar(B_FULL + st), 1);
      mbar_init(bar(B_EMPTY + st), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    for (int i = 0; i < QT; ++i) {
      mbar_init(bar(B_PFULL + i), 4);   // one arrival per softmax warp
      mbar_init(bar(B_ODONE + i), 1);
    }
    mbar_init(bar(B_FIN), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == W_MMA) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == W_PRODUCER && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&args.tk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&args.tv)) : "memory");
  }
  if (warp < 4 * QT) {
    // Query tiles: thread r of group i loads row i*128 + r of the item
    // (zeros past its queries) into the K-major 128-byte-swizzled layout.
    const int grp = warp >> 2, r = tid & 127, qrow = grp * BM + r;
    const bool ok = qrow < it.nq;
    const int tok = ok ? tc_query_token(it, g, qrow) : 0;
    const int4* src = reinterpret_cast<const int4*>(static_cast<const bf16*>(p.q) + tok * HD + (int64_t)it.head * D);
    const uint32_t q_tile = sQ + grp * L::Q_BYTES;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      int4 v = ok ? __ldg(src + c) : make_int4(0, 0, 0, 0);
      const uint32_t dst = q_tile + (c >> 3) * L::Q_REG + r * 128 + (((c & 7) ^ (r & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                   : "memory");
    }
    fence_proxy_async();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == W_PRODUCER) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && n_tiles > 0) {
      const int ycoord = args.kv_head_coord ? it.head : 0;
      // First key row of tile t.
      auto tile_row = [&](int t) -> int {
        if (PROXY) {
          const int f = t / it.tpf;
          return (int)it.k_row0 + f * g.F + it.rlo * g.Fw + (t - f * it.tpf) * BN;
        }
        return (int)(it.k_row0 + (int64_t)t * BN);
      };
      auto load_tile = [&](uint32_t dst, const CUtensorMap* map, int t, uint32_t b) {
#pragma unroll
        for (int rgn = 0; rgn < L::NREG; ++rgn) tma_load_3d(dst + rgn * L::KV_REG, map, rgn * 64, ycoord, tile_row(t), b);
      };
      mbar_expect_tx(bar(B_K0FULL), L::KV_BYTES);
      load_tile(sK, &args.tk, 0, bar(B_K0FULL));
      int issued = 0;   // load groups issued
      bool stalled = false;
      for (int t = 0; t < n_tiles; ++t) {
        if (p.debug_stall && t >= 1) {
          // Test hook: stop feeding without raising the abort flag, so that
          // the consumers' bounded waits expire.
          stalled = true;
          break;
        }
        // Group t reuses V stage t % 2 and K stage (t + 1) % 2, which key
        // tile t - 2's EMPTY commit releases (the MMA prologue's commit,
        // counted as tile -1, releases K(0)).
        const int st = t % STAGES;
        if (t >= 1 && !mbar_wait_bounded(bar(B_EMPTY + st), ((t - 1) / 2) & 1, abort_flag, wait_limit)) break;
        const bool knext = t + 1 < n_tiles;
        mbar_expect_tx(bar(B_FULL + st), knext ? 2 * L::KV_BYTES : L::KV_BYTES);
        load_tile(sV + st * L::KV_BYTES, &args.tv, t, bar(B_FULL + st));
        if (knext) load_tile(sK + ((t + 1) % STAGES) * L::KV_BYTES, &args.tk, t + 1, bar(B_FULL + st));
        issued = t + 1;
      }
      if (stalled || *abort_flag || issued < n_tiles) {
        if (!stalled) *abort_flag = 1;
        // Let the copies still in flight land before the CTA's memory goes.
        volatile int zero_flag = 0;   // drains ignore the abort flag
        (void)mbar_wait_bounded(bar(B_K0FULL), 0, &zero_flag, DRAIN_LIMIT_NS);
        for (int t = max(0, issued - STAGES); t < issued; ++t)
          (void)mbar_wait_bounded(bar(B_FULL + t % STAGES), (t / STAGES) & 1, &zero_flag, DRAIN_LIMIT_NS);
      }
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t ID_S = idesc_bf16(BM, BN, false);
      constexpr uint32_t ID_PV = idesc_bf16(BM, D, true);
      // Descriptors of query tile 0 and of the first K and V stage; the
      // start-address field is advanced by (byte offset >> 4), which cannot
      // carry out of its 14 bits (shared addresses stay below 256 KB).
      const uint64_t dq0 = sdesc(sQ, 16, 1024);
      const uint64_t dk0 = sdesc(sK, 16, 1024);
      const uint64_t dv0 = sdesc(sV, L::KV_REG, 1024);
      auto wait1 = [&](int slot, uint32_t parity) {
        return mbar_wait_bounded(bar(slot), parity, abort_flag, wait_limit);
      };
      // S_i(t) = Q_i K(t)^T into S_i's TMEM columns.
      auto mma_s = [&](int i, int t) {
        const uint64_t dk = dk0 + ((uint32_t)((t % STAGES) * L::KV_BYTES) >> 4);
        const uint64_t dq = dq0 + ((uint32_t)(i * L::Q_BYTES) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          // 16 columns of d = 32 B inside the 128-B row of region ks / 4.
          const uint32_t koff = (ks >> 2) * L::KV_REG + ((ks & 3) << 5);
          const uint32_t qoff = (ks >> 2) * L::Q_REG + ((ks & 3) << 5);
          mma_bf16_ss(tmem + i * BN, dq + (qoff >> 4), dk + (koff >> 4), ID_S, ks > 0 ? 1u : 0u);
        }
        if (i == 0) mma_commit(bar(B_SFULL));   // S_1: the EMPTY commit right after it
      };
      // O_i += P_i(j) V(j), P_i from the first half of S_i's columns.
      auto mma_pv = [&](int i, int j) {
        const uint64_t dv = dv0 + ((uint32_t)((j % STAGES) * L::KV_BYTES) >> 4);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          mma_bf16_ts(tmem + L::COL_O + i * D, tmem + i * BN + ks * 8, dv + ((ks * 16 * 128) >> 4), ID_PV,
                      (j > 0 || ks > 0) ? 1u : 0u);
      };
      bool ok = wait1(B_K0FULL, 0);
      if (ok) {
        tc_fence_after();
        mma_s(0, 0);
        if (two) mma_s(1, 0);
        mma_commit(bar(B_EMPTY + 1));   // tile -1: releases K(0)
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int st = j % STAGES;
        const bool more = j + 1 < n_tiles;
        // V(j) and K(j+1) arrive together.
        if (!(ok = wait1(B_FULL + st, (j / STAGES) & 1))) break;
        if (!(ok = wait1(B_PFULL + 0, j & 1))) break;
        tc_fence_after();
        mma_pv(0, j);
        if (more) mma_s(0, j + 1);
        if (two) {
          if (!(ok = wait1(B_PFULL + 1, j & 1))) break;
          tc_fence_after();
          mma_pv(1, j);
          if (more) mma_s(1, j + 1);
        }
        mma_commit(bar(B_EMPTY + st));   // releases V(j) and K(j+1)
      }
      if (ok) {
        mma_commit(bar(B_ODONE + 0));
        if (two) mma_commit(bar(B_ODONE + 1));
      } else {
        *abort_flag = 1;
        // Every MMA issued so far must finish before TMEM is released.
        volatile int zero_flag = 0;
        mma_commit(bar(B_FIN));
        (void)mbar_wait_bounded(bar(B_FIN), 0, &zero_flag, DRAIN_LIMIT_NS);
      }
    }
    __syncwarp();
  } else if (warp < 4 * QT) {
    // ---------------------------------------------------------------- softmax groups
    const int grp = warp >> 2, r = tid & 127, qrow = grp * BM + r;
    const bool active = grp == 0 || two;
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t t_s = t_lane + grp * BN;            // S_i (and P_i over its first half)
    const uint32_t t_o = t_lane + L::COL_O + grp * D;  // O_i
    const float sl2 = g.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    int h_lo = 0, h_hi = -1, w_lo = 0, w_hi = -1;   // PROXY: this row's key window in a frame
    if (PROXY) {
      const int pos = (it.q0 + qrow) % g.F;
      const int hq = pos / g.Fw;
      band_window(g, p.band_win, hq, pos - hq * g.Fw, h_lo, h_hi, w_lo, w_hi);
    }
    auto wait_warp = [&](int slot, uint32_t parity) -> bool {
      const bool w = mbar_wait_bounded(bar(slot), parity, abort_flag, wait_limit);
      return __all_sync(0xffffffffu, w);
    };
    for (int j = 0; active && j < n_tiles; ++j) {
      // S_1(j) is signalled by key tile j-1's EMPTY commit (the MMA
      // prologue's for j = 0): slot (j+1) % 2, its (j/2)-th completion.
      const int s_slot = grp == 0 ? (int)B_SFULL : B_EMPTY + (j + 1) % STAGES;
      if (!wait_warp(s_slot, grp == 0 ? (j & 1) : ((j / 2) & 1))) { ok = false; break; }
      tc_fence_after();
      const int valid = min(BN, it.k_len - j * BN);
      const bool full = PROXY || valid == BN;   // only a key run's last tile is partial
      // PROXY: bit e of mw[e / 32] marks key column e of this tile as inside
      // the row's proxy window (one run of keys per window row; the band's
      // rows are consecutive frame rows).
      uint32_t mw[BN / 32];
#pragma unroll
      for (int w = 0; w < BN / 32; ++w) mw[w] = 0u;
      if (PROXY) {
        const int o = (j % it.tpf) * BN;
        const int rhi = it.rlo + it.rlen / g.Fw - 1;
        for (int hk = max(it.rlo, h_lo); hk <= min(rhi, h_hi); ++hk) {
          const int a = max((hk - it.rlo) * g.Fw + w_lo - o, 0);
          const int b = min((hk - it.rlo) * g.Fw + w_hi - o, BN - 1);
#pragma unroll
          for (int w = 0; w < BN / 32; ++w) {
            const int lo = max(a, 32 * w), hi = min(b, 32 * w + 31);
            if (lo <= hi) mw[w] |= (uint32_t)(((1ull << (hi - lo + 1)) - 1ull) << (lo - 32 * w));
          }
        }
      }
      // Pass 1: row max over the tile.  Without masked keys the TMEM load
      // reduces it; otherwise 8 independent partial maxima (three-input max)
      // over the masked values.
      float pm[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
      if (!PROXY && full) {
#pragma unroll
        for (int h = 0; h < BN / 64; ++h) {
          uint32_t x[64];
          pm[h] = tmem_ld64_max(t_s + h * 64, x);
        }
      } else {
#pragma unroll
        for (int h = 0; h < BN / 64; ++h) {
          uint32_t x[64];
          tmem_ld32x2(t_s + h * 64, t_s + h * 64 + 32, x);
          if (PROXY) {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (!((mw[2 * h + e / 32] >> (e & 31)) & 1u)) x[e] = __float_as_uint(-INFINITY);
          } else if (!full) {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (h * 64 + e >= valid) x[e] = __float_as_uint(-INFINITY);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            pm[u] = max3f(pm[u], __uint_as_float(x[8 * u]), __uint_as_float(x[8 * u + 1]));
            pm[u] = max3f(pm[u], __uint_as_float(x[8 * u + 2]), __uint_as_float(x[8 * u + 3]));
            pm[u] = max3f(pm[u], __uint_as_float(x[8 * u + 4]), __uint_as_float(x[8 * u + 5]));
            pm[u] = max3f(pm[u], __uint_as_float(x[8 * u + 6]), __uint_as_float(x[8 * u + 7]));
          }
        }
      }
      pm[0] = max3f(pm[0], pm[1], pm[2]);
      pm[3] = max3f(pm[3], pm[4], pm[5]);
      pm[6] = fmaxf(pm[6], pm[7]);
      const float m_new = fmaxf(m_run, max3f(pm[0], pm[3], pm[6]) * sl2);
      if (j == 0) {
        m_run = m_new;
      } else if (__any_sync(0xffffffffu, m_new > m_run + RESCALE_LOG2)) {
        // O_i holds P_i(0..j-1) V, all of it complete (the commit that
        // signalled S_i(j) covers it): scale this warp's rows to the new max.
        // (A row still without any unmasked key keeps m = -inf and alpha 1.)
        const float alpha = m_new == -INFINITY ? 1.f : ex2(m_run - m_new);
        l_run *= alpha;
        m_run = m_new;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
  #pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(t_o + c * 32, o);
        }
        tmem_wait_st();
      }
      // Pass 2: probabilities 2^(s*scale*log2e - m), 64 keys at a time,
      // packed two per column into P_i.  Masked keys become -inf, whose
      // exponent is 0.
      // A row whose keys have all been masked so far keeps m = -inf; its
      // probabilities are all 0 (exponent of -inf), not NaN.
      const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
      float ps[8];   // 4 independent pairs of partial sums
#pragma unroll
      for (int u = 0; u < 8; ++u) ps[u] = 0.f;
#pragma unroll
      for (int h = 0; h < BN / 64; ++h) {
        // Keys [64h, 64h+64) of S_i; their probabilities go to P_i columns
        // [32h, 32h+32), which lie inside S_i columns already read.
        uint32_t x[64];
        tmem_ld32x2(t_s + h * 64, t_s + h * 64 + 32, x);
        if (PROXY) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (!((mw[2 * h + e / 32] >> (e & 31)) & 1u)) x[e] = __float_as_uint(-INFINITY);
        } else if (!full) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (h * 64 + e >= valid) x[e] = __float_as_uint(-INFINITY);
        }
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float a0, a1;
          fma2(a0, a1, __uint_as_float(x[2 * c]), __uint_as_float(x[2 * c + 1]), sl2, neg_m);
          const float e0 = ex2(a0), e1 = ex2(a1);
          add2(ps[2 * (c & 3)], ps[2 * (c & 3) + 1], e0, e1);
          pk[c] = pack_bf16(e0, e1);
        }
        tmem_st32(t_s + h * 32, pk);
      }
      l_run += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + grp));
    }
    // ---------------------------------------------------------------- epilogue
    if (active && ok && n_tiles > 0 && wait_warp(B_ODONE + grp, 0)) {
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const bool w = qrow < it.nq;
      const int64_t tok = w ? tc_query_token(it, g, qrow) : 0;
      const int64_t base = (int64_t)it.out_plane * p.o_plane_stride + tok * HD + (int64_t)it.head * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_o + c * 32, o);
        if (!w) continue;
        if (p.out_fp32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + base + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                 __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16*>(p.o) + base + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t* x = o + 8 * e;
            dst[e] = make_uint4(pack_bf16(__uint_as_float(x[0]) * inv, __uint_as_float(x[1]) * inv),
                                pack_bf16(__uint_as_float(x[2]) * inv, __uint_as_float(x[3]) * inv),
                                pack_bf16(__uint_as_float(x[4]) * inv, __uint_as_float(x[5]) * inv),
                                pack_bf16(__uint_as_float(x[6]) * inv, __uint_as_float(x[7]) * inv));
          }
        }
      }
    } else if (active && n_tiles == 0 && qrow < it.nq) {
      // No keys: the output is defined as zero.
      const int64_t tok = tc_query_token(it, g, qrow);
      const int64_t base = (int64_t)it.out_plane * p.o_plane_stride + tok * HD + (int64_t)it.head * D;
      for (int c = 0; c < D; ++c) {
        if (p.out_fp32) static_cast<float*>(p.o)[base + c] = 0.f;
        else static_cast<bf16*>(p.o)[base + c] = __float2bfloat16_rn(0.f);
      }
    } else if (active && n_tiles > 0) {
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag && p.status) atomicExch(p.status, DEV_TIMEOUT);
  if (warp == W_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// K or V as a 3-D bf16 tensor [rows][heads][d]; box {64, 1, BN}, 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* base, int d, int heads, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
  const cuuint32_t box[3] = {64, 1, BN};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, bool PROXY>
cudaError_t launch_d(const TcArgs& a, dim3 grid, cudaStream_t s) {
  constexpr int smem = Layout<D>::ALLOC;
  static_assert(smem <= 232448, "shared memory budget");
  // The dynamic shared-memory opt-in is a per-device attribute of the
  // function: set it once on every device the process launches on.
  constexpr int kMaxDevices = 128;
  static std::mutex mu;
  static bool configured[kMaxDevices] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(attn_tc_kernel<D, PROXY>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  attn_tc_kernel<D, PROXY><<<grid, NTHREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int tc_block_rows() { return QT * BM; }

cudaError_t launch_attention_tc(const AttnParams& p, const TcKV& kv, dim3 grid, cudaStream_t s) {
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  if (p.g.d != 64 && p.g.d != 128) return cudaErrorInvalidValue;
  if (kv.rows <= 0 || kv.rows > 0x7fffffffll) return cudaErrorInvalidValue;
  TcArgs a;
  memset(&a, 0, sizeof a);
  cudaError_t e = make_map(&a.tk, kv.k, p.g.d, kv.heads, kv.rows);
  if (e != cudaSuccess) return e;
  if ((e = make_map(&a.tv, kv.v, p.g.d, kv.heads, kv.rows)) != cudaSuccess) return e;
  a.p = p;
  a.p.debug_stall = debug_stall_enabled() ? 1 : 0;
  a.p.wait_limit_ns = a.p.debug_stall ? STALL_WAIT_LIMIT_NS : WAIT_LIMIT_NS;
  a.kv_head_coord = kv.heads > 1 ? 1 : 0;
  // Band items (classification proxy, routed sliding Spatial) run the masked
  // variant; the caller launches them separately from the other items.
  if (p.item_mode == ITEMS_PROXY || p.band_win == WIN_SLIDING)
    return p.g.d == 128 ? launch_d<128, true>(a, grid, s) : launch_d<64, true>(a, grid, s);
  return p.g.d == 128 ? launch_d<128, false>(a, grid, s) : launch_d<64, false>(a, grid, s);
}

}  // namespace hc
