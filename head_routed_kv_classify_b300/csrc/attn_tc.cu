// Softmax attention on the 5th-generation tensor cores (tcgen05 + TMEM),
// with K/V tiles streamed by TMA.  Serves every bf16 attention of the
// library: the routed pathways (Sink / Dummy / Global key runs and Spatial
// cells of the restructured cache, sliding Spatial patches), the in-house
// full attention, and classification (the proxy, and one pass that yields
// the full-context, Sink and Dummy outputs and the per-token statistics).
// [Pith review of HeadCast: "The pith" and "Core claim" (each head attends
//  only over its pathway), "What carries the argument" (the classification
//  outputs), major comment 2 and Figure 3 caption (10x10 cells).]
//
// A launch is persistent: each CTA runs a list of work items, each up to 256
// queries of one head (two query tiles of 128) against one run of key rows
// (or a patch's halo boxes), streamed in tiles of 128 keys.  Roles (320
// threads):
//   warps 0-3, 4-7  softmax groups, one per query tile: thread r of group i
//              owns row r of tile i, i.e. TMEM lane r.  It reads its row of
//              S_i = Q_i K^T from TMEM (a max pass, then an exponent pass),
//              keeps the running max and sum, writes P_i (bf16, two per
//              32-bit column) back over the first half of S_i and, when the
//              max has grown by more than 2^8, rescales its row of O_i; at
//              an item's end it gathers the next item's query rows and then
//              normalises O_i and stores it.
//   warp 8     TMA producer: K and V tiles into 2-stage rings.  V(j) and
//              K(j+1) travel together on one barrier, so the MMA issuer
//              makes one data wait and one release commit per key tile:
//              each barrier poll between two MMA batches leaves the tensor
//              pipe idle, since an MMA issue returns only once the pipe
//              accepts it.
//   warp 9     MMA issuer (the whole warp runs the loop with warp-uniform
//              descriptors; one elected lane issues), in the order
//              P_0 V, S_0, P_1 V, S_1 per key tile,
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
// deployed Spatial heads, their routed items (ITEM_PATCH) -- are patches of
// query positions in every frame of the block: every query at a position
// has the same key window, so a patch's keys in each key frame are its halo,
// read as 2-D TMA boxes of a [frames][Fh][Fw][heads][d] view of K and V and
// masked per query to its window (the (2r+1) x (2r+1) neighbourhood, the
// deployed cell, or the centred cell_h x cell_w window).
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
constexpr int ITEM_CACHE = 256;    // work items of a CTA kept in shared memory
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
  static constexpr int OFF_ITEMS = OFF_BAR + 256;   // the CTA's work items (list launches)
  static constexpr int OFF_MASK = OFF_ITEMS + ITEM_CACHE * (int)sizeof(WorkItem);   // band window masks
  static constexpr int BYTES = OFF_MASK + 4 * QT * 32 * kMaxBoxesPerFrame * 16;
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
       B_ODONE = B_PFULL + QT, B_QREADY = B_ODONE + QT, B_FIN = B_QREADY + QT, B_COUNT = B_FIN + 1 };
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
// 16 bytes global -> shared without a register round trip; with
// src_bytes = 0 nothing is read and the 16 bytes are zero-filled.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
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

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            int c4, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], "
      "[%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
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

// The MMA and commit wrappers are executed by the whole issuing warp, with
// warp-uniform operands; elect.sync picks the one lane that issues.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred e, p;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// As above with A (M x 16, K-major) read from TMEM at column a_tmem.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred e, p;\n elect.sync _|e, 0xffffffff;\n setp.ne.b32 p, %4, 0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
               " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
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
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : HC_R32_8(0), HC_R32_8(8)
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
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), HC_W32_8(0), HC_W32_8(8)
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
// The two bf16 halves of a 32-bit word as floats (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
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
  int rlo, rlen, tpf;   // band items: halo origin row and column, key tiles (boxes) per key frame
  int part;             // >= 0: partial output slot of a split key run
};

// A band item: patch `patch` of the launch's patch geometry, query chunk
// `chunk`, over `frames` key frames.
__device__ __forceinline__ void tc_patch(TcItem& it, const AttnParams& p, int patch, int chunk, int frames) {
  const Geom& g = p.g;
  const PatchGeom& pg = p.pg;
  if (pg.cells) {
    const int ci = patch / g.ncell_w, cj = patch - (patch / g.ncell_w) * g.ncell_w;
    it.h0 = ci * g.cell_h;
    it.hz = cell_extent(ci, g.Fh, g.cell_h, g.ncell_h);
    it.w0 = cj * g.cell_w;
    it.wz = cell_extent(cj, g.Fw, g.cell_w, g.ncell_w);
  } else {
    const int pi = patch / pg.npw, pj = patch - (patch / pg.npw) * pg.npw;
    it.h0 = pi * pg.ph;
    it.hz = min(pg.ph, g.Fh - it.h0);
    it.w0 = pj * pg.pw;
    it.wz = min(pg.pw, g.Fw - it.w0);
  }
  it.q0 = chunk * (QT * BM);
  it.nq = min(QT * BM, g.fpb * it.hz * it.wz - it.q0);
  it.rlo = it.h0 + pg.dh;
  it.rlen = it.w0 + pg.dw;
  it.tpf = pg.tpf;
  it.k_len = it.nq > 0 ? frames * pg.tpf * BN : 0;
}

// Work item w of the launch (`src`: where list launches read item w from).
__device__ __forceinline__ TcItem tc_decode(const AttnParams& p, int w, const WorkItem* src) {
  const Geom& g = p.g;
  TcItem it;
  it.h0 = it.w0 = it.hz = it.wz = 0;
  it.rlo = it.rlen = it.tpf = 0;
  it.part = -1;
  if (p.item_mode == ITEMS_PROXY) {
    // A patch of query positions in every frame of the block (a query chunk
    // of it with the cell proxy); keys: its halo in every window frame,
    // narrowed per query to its window by the mask.
    const int per_head = p.pg.n * p.pg.cpc;
    const int x = w % per_head;
    it.head = w / per_head;
    it.kind = ITEM_PROXY;
    it.out_plane = 3;
    it.k_row0 = 0;
    tc_patch(it, p, x / p.pg.cpc, x % p.pg.cpc, p.proxy_frames);
  } else if (p.item_mode == ITEMS_LIST) {
    const WorkItem wi = *src;
    it.head = wi.head;
    it.kind = wi.kind;
    it.q0 = wi.q0;
    it.nq = wi.nq;
    it.out_plane = wi.out_plane;
    it.k_row0 = wi.k_row0;
    it.k_len = wi.k_per_frame > 0 ? wi.k_per_frame * p.valid_frames : wi.k_len;
    if (wi.kind == ITEM_CELL) {
      const int ci = wi.cell / g.ncell_w, cj = wi.cell % g.ncell_w;
      it.h0 = ci * g.cell_h;
      it.hz = cell_extent(ci, g.Fh, g.cell_h, g.ncell_h);
      it.w0 = cj * g.cell_w;
      it.wz = cell_extent(cj, g.Fw, g.cell_w, g.ncell_w);
    } else if (wi.kind == ITEM_PATCH) {
      // Sliding Spatial: patch wi.cell; keys in the head's filled ring slots,
      // stored in raster order from row k_row0.
      tc_patch(it, p, wi.cell, 0, p.valid_frames);
    }
    if (wi.n_chunks > 1 && wi.kind != ITEM_PATCH) {
      // This item's share of the run's T key tiles (possibly none while the
      // window is still filling); the run's last, partial tile stays last.
      const int T = (it.k_len + BN - 1) / BN;
      const int t0 = (int)((int64_t)wi.chunk * T / wi.n_chunks);
      const int t1 = (int)((int64_t)(wi.chunk + 1) * T / wi.n_chunks);
      it.k_row0 += (int64_t)t0 * BN;
      it.k_len = t1 > t0 ? min(it.k_len - t0 * BN, (t1 - t0) * BN) : 0;
    }
    it.part = wi.part;
  } else {  // ITEMS_DENSE: w = ((plane * H) + head) * n_q_tiles + q_tile
    const int nx = (p.nq_total + QT * BM - 1) / (QT * BM);
    const int x = w % nx, rest = w / nx;
    const int z = rest / g.H;
    it.head = rest - z * g.H;
    it.kind = ITEM_RANGE;
    it.q0 = x * (QT * BM);
    it.nq = min(QT * BM, p.nq_total - it.q0);
    it.out_plane = z;
    it.k_row0 = p.plane_k0[z];
    it.k_len = p.plane_klen[z];
  }
  return it;
}

// Classification full pass: the key tiles run as Sink segment [0, cls_n0),
// middle [cls_n0, cls_n01) and Dummy segment [cls_n01, n), each ending in
// its own partial tile.  The boundaries are launch constants, so a tile
// needs a few compares against parameters and no live registers (this code
// runs on the critical path of every key tile).
__device__ __forceinline__ int tc_tiles(const AttnParams& p, const TcItem& it, bool cls) {
  if (it.k_len <= 0) return 0;
  if (cls) return p.cls_n01 + (it.k_len - p.seg_dummy + BN - 1) / BN;
  return (it.k_len + BN - 1) / BN;
}

// First key row of key tile j.
__device__ __forceinline__ int tile_row(const AttnParams& p, bool cls, int64_t k_row0, int j) {
  if (!cls) return (int)k_row0 + j * BN;
  const int seg0 = j < p.cls_n0 ? 0 : (j < p.cls_n01 ? p.seg_sink - p.cls_n0 * BN : p.seg_dummy - p.cls_n01 * BN);
  return (int)k_row0 + seg0 + j * BN;
}

// Keys in key tile j of n.
__device__ __forceinline__ int tile_valid(const AttnParams& p, bool cls, int k_len, int j, int n) {
  if (!cls) return min(BN, k_len - j * BN);
  int v = BN;
  v = j == p.cls_n0 - 1 ? p.cls_v0 : v;
  v = j == p.cls_n01 - 1 && p.cls_n01 > p.cls_n0 ? p.cls_v1 : v;
  v = j == n - 1 ? p.cls_v2 : v;
  return v;
}

// The items of this CTA: w0, w0 + step, ... below w1.
__device__ __forceinline__ void cta_items(const AttnParams& p, int& w0, int& w1, int& step) {
  if (p.sched) {
    w0 = p.sched[blockIdx.x];
    w1 = p.sched[blockIdx.x + 1];
    step = 1;
  } else {
    w0 = blockIdx.x;
    w1 = p.n_items;
    step = gridDim.x;
  }
}

// The CTA's list items: the first ITEM_CACHE from shared memory, the rest
// (of an unusually long list) from global memory.
struct ItemSrc {
  const WorkItem* smem;   // null: nothing staged
  const WorkItem* gmem;
  int w0;
  __device__ __forceinline__ const WorkItem* at(int w) const {
    return smem && w - w0 < ITEM_CACHE ? smem + (w - w0) : gmem + w;
  }
};

__device__ __forceinline__ TcItem tc_decode(const AttnParams& p, int w, const ItemSrc& src) {
  return tc_decode(p, w, p.item_mode == ITEMS_LIST ? src.at(w) : nullptr);
}

// First item at or after w with at least one key (w1 if none).
__device__ __forceinline__ int next_keyed(const AttnParams& p, int w, int w1, int step, const ItemSrc& src,
                                          TcItem& it) {
  for (; w < w1; w += step) {
    it = tc_decode(p, w, src);
    if (it.k_len > 0) return w;
  }
  return w1;
}

// Block-local token of the r-th query of an item (cells and patches: query
// ordinals in (frame, row, column) order inside the cell or patch).
__device__ __forceinline__ int tc_query_token(const TcItem& it, const Geom& g, int r) {
  if (it.kind == ITEM_RANGE) return it.q0 + r;
  const int ord = it.q0 + r;
  const int csz = it.hz * it.wz;
  const int fq = ord / csz, rem = ord - fq * csz;
  const int hh = rem / it.wz, ww = rem - hh * it.wz;
  return fq * g.F + (it.h0 + hh) * g.Fw + it.w0 + ww;
}

// ---------------------------------------------------------------- the kernel
//
// Persistent: each CTA runs its items back to back with one TMEM allocation
// and one set of barriers.  The key tiles of all its items form one global
// sequence g = 0, 1, ...: load group g carries V(g) and K(g+1), where K(g+1)
// may be the first key tile of the next item, so the producer runs ahead
// across item boundaries.  At a boundary each softmax group, once it has
// consumed S_i of the item's last tile, gathers its query tile of the next
// item into shared memory (arrival on QREADY_i) and then stores the item's
// output (after ODONE_i); the MMA issuer issues the next item's first S_i as
// soon as QREADY_i arrives, so the epilogue overlaps the next item's start.
// Every item runs both query tiles (rows past the item's queries are zero
// and never stored), so both softmax groups see every key tile.

// PROXY: band items (masked halo boxes); CLS: the classification pass
// (segmented keys, parked states, per-token statistics).
template <int D, bool PROXY, bool CLS>
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
  int w_begin, w_end, w_step;
  cta_items(p, w_begin, w_end, w_step);
  // Once any CTA has recorded an expired wait, the rest of the launch (and
  // later launches, until the status word is read and cleared) skip their
  // work so that a broken pipeline fails fast.
  if (threadIdx.x == 0) *skip_flag = p.status ? *reinterpret_cast<volatile int*>(p.status) : 0;
  __syncthreads();
  if (*skip_flag || w_begin >= w_end) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t HD = (int64_t)g.H * D;
  const bool staged = p.item_mode == ITEMS_LIST && w_step == 1;
  const ItemSrc isrc{staged ? reinterpret_cast<const WorkItem*>(smem + L::OFF_ITEMS) : nullptr, p.items, w_begin};
  if (PROXY) {
    // A band tile's box fills only its first bh*kw key rows; the rest of the
    // K and V stages must hold finite values (their probabilities are 0, and
    // 0 times a stale NaN would not be), so they start as zeros.
    int4* kv = reinterpret_cast<int4*>(smem + L::OFF_K);
    for (int i = tid; i < 2 * STAGES * L::KV_BYTES / 16; i += NTHREADS) kv[i] = make_int4(0, 0, 0, 0);
    fence_proxy_async();   // before the tensor core and TMA touch them
  }
  if (staged) {
    // Stage this CTA's items in shared memory: every role decodes each item
    // several times, and a decode must not wait on global memory at an item
    // boundary.  (List launches run a contiguous range: w_step == 1.)
    const int n = min(w_end - w_begin, ITEM_CACHE) * (int)(sizeof(WorkItem) / 16);
    const int4* src = reinterpret_cast<const int4*>(p.items + w_begin);
    int4* dst = reinterpret_cast<int4*>(smem + L::OFF_ITEMS);
    for (int i = tid; i < n; i += NTHREADS) dst[i] = src[i];
  }

  if (tid == 0) {
    mbar_init(bar(B_K0FULL), 1);
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(bar(B_FULL + st), 1);
      mbar_init(bar(B_EMPTY + st), 1);
    }
    mbar_init(bar(B_SFULL), 1);
    for (int i = 0; i < QT; ++i) {
      mbar_init(bar(B_PFULL + i), 4);    // one arrival per softmax warp
      mbar_init(bar(B_ODONE + i), 1);
      mbar_init(bar(B_QREADY + i), 4);   // one arrival per softmax warp
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == W_PRODUCER) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      auto load_tile = [&](uint32_t dst, const CUtensorMap* map, const TcItem& it, int t, uint32_t b) {
        const int y = args.kv_head_coord ? it.head : 0;
        if (PROXY) {
          // Box tt of key frame f of the item's halo: bh rows x kw columns
          // from (rlo + tt*bh, rlen), read as a [frames][Fh][Fw][heads][d]
          // tensor (zeros outside the frame).
          const int f = t / it.tpf, tt = t - f * it.tpf;
          const int fr = p.band_frame0 + (int)(it.k_row0 / g.F) + f;
#pragma unroll
          for (int rgn = 0; rgn < L::NREG; ++rgn)
            tma_load_5d(dst + rgn * L::KV_REG, map, rgn * 64, y, it.rlen, it.rlo + tt * p.pg.bh, fr, b);
          return;
        }
        const int z = tile_row(p, CLS, it.k_row0, t);
#pragma unroll
        for (int rgn = 0; rgn < L::NREG; ++rgn) tma_load_3d(dst + rgn * L::KV_REG, map, rgn * 64, y, z, b);
      };
      // Bytes one K (or V) tile brings: a whole tile, or for band items the
      // bh x kw rows of one halo box (out-of-frame rows included).
      const uint32_t tile_bytes = PROXY ? (uint32_t)(L::NREG * p.pg.bh * p.pg.kw * 128) : (uint32_t)L::KV_BYTES;
      TcItem it, nx;
      int w = next_keyed(p, w_begin, w_end, w_step, isrc, it);
      int issued = 0;   // load groups issued (global key tile count)
      bool k0 = false, stalled = false, fail = false;
      if (w < w_end) {
        mbar_expect_tx(bar(B_K0FULL), tile_bytes);
        load_tile(sK, &args.tk, it, 0, bar(B_K0FULL));
        k0 = true;
      }
      while (w < w_end && !fail && !stalled) {
        const int n = tc_tiles(p, it, CLS);
        const int wn = next_keyed(p, w + w_step, w_end, w_step, isrc, nx);
        for (int j = 0; j < n; ++j) {
          if (p.debug_stall && issued >= 1) {
            // Test hook: stop feeding without raising the abort flag, so that
            // the consumers' bounded waits expire.
            stalled = true;
            break;
          }
          // Group `issued` reuses V stage issued % 2 and K stage
          // (issued + 1) % 2, which key tile issued - 2's EMPTY commit
          // releases (the MMA prologue's commit, counted as tile -1,
          // releases K(0)).
          const int st = issued % STAGES;
          if (issued >= 1 && !mbar_wait_bounded(bar(B_EMPTY + st), ((issued - 1) / 2) & 1, abort_flag, wait_limit)) {
            fail = true;
            break;
          }
          const bool k_same = j + 1 < n, k_next = !k_same && wn < w_end;
          mbar_expect_tx(bar(B_FULL + st), (k_same || k_next) ? 2 * tile_bytes : tile_bytes);
          load_tile(sV + st * L::KV_BYTES, &args.tv, it, j, bar(B_FULL + st));
          const uint32_t kdst = sK + ((issued + 1) % STAGES) * L::KV_BYTES;
          if (k_same) load_tile(kdst, &args.tk, it, j + 1, bar(B_FULL + st));
          else if (k_next) load_tile(kdst, &args.tk, nx, 0, bar(B_FULL + st));
          ++issued;
        }
        w = wn;
        it = nx;
      }
      if (stalled || fail || *abort_flag) {
        if (!stalled) *abort_flag = 1;
        // Let the copies still in flight land before the CTA's memory goes.
        volatile int zero_flag = 0;   // drains ignore the abort flag
        if (k0) (void)mbar_wait_bounded(bar(B_K0FULL), 0, &zero_flag, DRAIN_LIMIT_NS);
        for (int t = max(0, issued - STAGES); t < issued; ++t)
          (void)mbar_wait_bounded(bar(B_FULL + t % STAGES), (t / STAGES) & 1, &zero_flag, DRAIN_LIMIT_NS);
      }
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ---------------------------------------------------------------- MMA issuer
    {
      constexpr uint32_t ID_S = idesc_bf16(BM, BN, false);
      constexpr uint32_t ID_PV = idesc_bf16(BM, D, true);
      // Descriptors of query tile 0 and of the first K and V stage; the
      // start-address field is advanced by (byte offset >> 4), which cannot
      // carry out of its 14 bits (shared addresses stay below 256 KB).
      const uint64_t dq0 = sdesc(sQ, 16, 1024);
      const uint64_t dk0 = sdesc(sK, 16, 1024);
      const uint64_t dv0 = sdesc(sV, L::KV_REG, 1024);
      // Every lane polls (the warp stays converged) and the warp agrees.
      auto wait1 = [&](int slot, uint32_t parity) {
        const bool r = mbar_wait_bounded(bar(slot), parity, abort_flag, wait_limit);
        return __all_sync(0xffffffffu, r);
      };
      // S_i = Q_i K(t)^T into S_i's TMEM columns (t: global key tile).
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
      // O_i (+)= P_i V(t), P_i from the first half of S_i's columns; the
      // item's first key tile (j == 0) starts O_i afresh.
      // (The classification pass also starts O_i afresh at the Dummy
      // segment's first tile.)
      const int j_restart = CLS ? p.cls_n01 : 0;
      auto mma_pv = [&](int i, int t, int j) {
        const uint64_t dv = dv0 + ((uint32_t)((t % STAGES) * L::KV_BYTES) >> 4);
        const bool fresh = j == 0 || j == j_restart;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          mma_bf16_ts(tmem + L::COL_O + i * D, tmem + i * BN + ks * 8, dv + ((ks * 16 * 128) >> 4), ID_PV,
                      (!fresh || ks > 0) ? 1u : 0u);
      };
      TcItem it, nx;
      int w = next_keyed(p, w_begin, w_end, w_step, isrc, it);
      int gt = 0;       // global key tile
      int qph = 0;      // QREADY phases consumed
      bool ok = true;
      if (w < w_end) {
        ok = wait1(B_K0FULL, 0) && wait1(B_QREADY + 0, 0);
        if (ok) {
          tc_fence_after();
          mma_s(0, 0);
          ok = wait1(B_QREADY + 1, 0);
        }
        if (ok) {
          tc_fence_after();
          mma_s(1, 0);
          mma_commit(bar(B_EMPTY + 1));   // tile -1: releases K(0), signals S_1(0)
        }
        qph = 1;
      }
      while (ok && w < w_end) {
        const int n = tc_tiles(p, it, CLS);
        const int wn = next_keyed(p, w + w_step, w_end, w_step, isrc, nx);
        for (int j = 0; j < n; ++j) {
          const int st = gt % STAGES;
          const bool last = j + 1 == n;
          // V(gt) and K(gt+1) arrive together.
          if (!(ok = wait1(B_FULL + st, (gt / STAGES) & 1))) break;
          if (!(ok = wait1(B_PFULL + 0, gt & 1))) break;
          tc_fence_after();
          mma_pv(0, gt, j);
          if (!last) mma_s(0, gt + 1);
          else mma_commit(bar(B_ODONE + 0));
          if (!(ok = wait1(B_PFULL + 1, gt & 1))) break;
          tc_fence_after();
          mma_pv(1, gt, j);
          if (!last) {
            mma_s(1, gt + 1);
          } else {
            mma_commit(bar(B_ODONE + 1));
            if (wn < w_end) {
              // The next item's first S: its query tiles, K(gt+1).
              if (!(ok = wait1(B_QREADY + 0, qph & 1))) break;
              tc_fence_after();
              mma_s(0, gt + 1);
              if (!(ok = wait1(B_QREADY + 1, qph & 1))) break;
              tc_fence_after();
              mma_s(1, gt + 1);
              ++qph;
            }
          }
          mma_commit(bar(B_EMPTY + st));   // releases V(gt) and K(gt+1), signals S_1(gt+1)
          ++gt;
        }
        w = wn;
        it = nx;
      }
      if (!ok) {
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
    const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t t_s = t_lane + grp * BN;            // S_i (and P_i over its first half)
    const uint32_t t_o = t_lane + L::COL_O + grp * D;  // O_i
    const float sl2 = g.scale_log2;
    const uint32_t q_tile = sQ + grp * L::Q_BYTES;
    const uint32_t mask_base = s_base + L::OFF_MASK + (uint32_t)(tid * kMaxBoxesPerFrame * 16);   // PROXY
    auto wait_warp = [&](int slot, uint32_t parity) -> bool {
      const bool w = mbar_wait_bounded(bar(slot), parity, abort_flag, wait_limit);
      return __all_sync(0xffffffffu, w);
    };
    // Row qrow of an item's query tile into the K-major 128-byte-swizzled
    // layout (zeros past its queries) by asynchronous copies; finish_q waits
    // for them and makes one arrival per warp on QREADY_i.
    // Row qrow of an item's query tile into the K-major 128-byte-swizzled
    // layout (zeros past its queries) by asynchronous copies (all 16-byte
    // pieces of the row in flight at once); finish_q waits for them and makes
    // one arrival per warp on QREADY_i.
    auto issue_q = [&](const TcItem& it) {
      const bool ok = qrow < it.nq;
      const int tok = ok ? tc_query_token(it, g, qrow) : 0;
      const int4* src = reinterpret_cast<const int4*>(static_cast<const bf16*>(p.q) + tok * HD + (int64_t)it.head * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        cp_async16(q_tile + (c >> 3) * L::Q_REG + r * 128 + (((c & 7) ^ (r & 7)) << 4), src + c, ok ? 16u : 0u);
      cp_async_commit();
    };
    auto finish_q = [&]() {
      cp_async_wait_all();
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QREADY + grp));
    };
    // Output rows of an item: the normalised output, or for a split key run
    // the unnormalised partial with its row max and sum.
    auto out_base = [&](const TcItem& it) -> int64_t {
      const int64_t tok = tc_query_token(it, g, qrow);
      return (int64_t)it.out_plane * p.o_plane_stride + tok * HD + (int64_t)it.head * D;
    };
    // Classification pass: park this row's running state (O as it stands in
    // TMEM, unnormalised, with the row max and sum) in slot 0 (after the
    // Sink segment; bf16) or 1 (before the Dummy segment; fp32 when the
    // full-context output is wanted, else bf16).
    auto park = [&](int w, int slot, float m, float l) {
      const TcItem it = tc_decode(p, w, isrc);
      const bool ok = qrow < it.nq;
      const int64_t tr = (int64_t)(it.q0 + qrow) * g.H + it.head;   // token row of a plane
      const int64_t row = (int64_t)slot * p.nq_total * g.H + tr;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_o + c * 32, o);
        if (!ok) continue;
        if (slot == 0 || p.park1_bf16) {   // bf16: feeds only the cosines
          uint4* dst = reinterpret_cast<uint4*>((slot == 0 ? static_cast<bf16*>(p.park_o)
                                                           : reinterpret_cast<bf16*>(p.park_o1)) +
                                                tr * D + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t* x = o + 8 * e;
            dst[e] = make_uint4(pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(p.park_o1 + tr * D + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                 __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
        }
      }
      if (ok) *reinterpret_cast<float2*>(p.park_ml + row * 2) = make_float2(m, l);
    };
    {
      TcItem f;
      if (next_keyed(p, w_begin, w_end, w_step, isrc, f) < w_end) {
        issue_q(f);
        finish_q();
      }
    }
    int gt = 0;     // global key tile
    int nitem = 0;  // keyed items done (ODONE phases)
    bool ok = true;
    for (int w = w_begin; ok && w < w_end; w += w_step) {
      // Only what the tile loop needs stays live across it; the item is
      // decoded again for the epilogue.
      int n, k_len, tpf = 1;
      {
        const TcItem it = tc_decode(p, w, isrc);
        n = tc_tiles(p, it, CLS);
        k_len = it.k_len;
        if (n == 0) {
          // No keys: the output is defined as zero (a split run's empty
          // share: row max -inf, sum 0).
          if (qrow < it.nq) {
            if (it.part >= 0) {
              float* po = p.part_o + ((int64_t)it.part * kPartRows + qrow) * D;
              for (int c = 0; c < D; ++c) po[c] = 0.f;
              p.part_ml[((int64_t)it.part * kPartRows + qrow) * 2 + 0] = -INFINITY;
              p.part_ml[((int64_t)it.part * kPartRows + qrow) * 2 + 1] = 0.f;
            } else {
              const int64_t base = out_base(it);
              for (int c = 0; c < D; ++c) {
                if (p.out_fp32) static_cast<float*>(p.o)[base + c] = 0.f;
                else static_cast<bf16*>(p.o)[base + c] = __float2bfloat16_rn(0.f);
              }
            }
          }
          continue;
        }
        if (PROXY) {
          // This row's window mask for each box of a key frame (the same in
          // every frame): bit e of word e / 32 marks key column e of the box
          // as inside the window.  Key column e of box tt is halo row
          // tt*bh + e / kw, halo column e % kw: one run of columns per window
          // row.
          tpf = it.tpf;
          int h_lo, h_hi, w_lo, w_hi;
          const int pos = tc_query_token(it, g, qrow) % g.F;
          const int hq = pos / g.Fw;
          band_window(g, p.band_win, hq, pos - hq * g.Fw, h_lo, h_hi, w_lo, w_hi);
          // As offsets into the halo (rows may start before the frame; the
          // window is clipped to the frame, so it lies inside the halo).
          h_lo -= it.rlo;
          h_hi -= it.rlo;
          w_lo -= it.rlen;
          w_hi -= it.rlen;
          const int bh = p.pg.bh, kw = p.pg.kw;
#pragma unroll 1
          for (int tt = 0; tt < tpf; ++tt) {
            uint32_t m4[BN / 32];
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) m4[q] = 0u;
            const int r0 = tt * bh;
            for (int hk = max(r0, h_lo); hk <= min(r0 + bh - 1, h_hi); ++hk) {
              const int a = (hk - r0) * kw + w_lo;
              const int b = (hk - r0) * kw + w_hi;
#pragma unroll
              for (int q = 0; q < BN / 32; ++q) {
                const int lo = max(a, 32 * q), hi = min(b, 32 * q + 31);
                if (lo <= hi) m4[q] |= (uint32_t)(((1ull << (hi - lo + 1)) - 1ull) << (lo - 32 * q));
              }
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(mask_base + tt * 16), "r"(m4[0]), "r"(m4[1]),
                         "r"(m4[2]), "r"(m4[3])
                         : "memory");
          }
        }
      }
      float m_run = -INFINITY, l_run = 0.f;
      int tt = 0;   // PROXY: box of the current key tile within its key frame
      for (int j = 0; j < n; ++j, ++gt) {
        // S_1(gt) is signalled by key tile gt-1's EMPTY commit (the MMA
        // prologue's for gt = 0): slot (gt+1) % 2, its (gt/2)-th completion.
        const int s_slot = grp == 0 ? (int)B_SFULL : B_EMPTY + (gt + 1) % STAGES;
        if (!wait_warp(s_slot, grp == 0 ? (gt & 1) : ((gt / 2) & 1))) { ok = false; break; }
        tc_fence_after();
        const int valid = tile_valid(p, CLS, k_len, j, n);
        if (CLS && (j == p.cls_n0 || j == p.cls_n01)) {
          // O_i holds the keys so far, complete (the commit that signalled
          // S_i(j) covers P_i(j-1) V).
          const int n0 = p.cls_n0, n01 = p.cls_n01;
          if (j == n0) park(w, 0, m_run, l_run);
          if (j == n01) {
            park(w, 1, m_run, l_run);
            m_run = -INFINITY;   // the Dummy segment starts afresh
            l_run = 0.f;
          }
        }
        const bool full = PROXY || valid == BN;   // only a key run's last tile is partial
        // PROXY: bit e of mw[e / 32] marks key column e of this tile as inside
        // the row's proxy window (one run of keys per window row; the band's
        // rows are consecutive frame rows).
        uint32_t mw[BN / 32];
#pragma unroll
        for (int q = 0; q < BN / 32; ++q) mw[q] = 0u;
        if (PROXY) {
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(mw[0]), "=r"(mw[1]), "=r"(mw[2]), "=r"(mw[3])
                       : "r"(mask_base + tt * 16)
                       : "memory");
          if (++tt == tpf) tt = 0;
        }
        // Pass 1: row max over the tile, reduced by the TMEM load itself.
        // Band tiles take it over the whole box, window or not: any value at
        // least the window's max stabilises the softmax equally (every score of
        // a band tile is finite -- rows outside the frame and past the box are
        // zero keys of the same head -- and the box's max exceeds the window's
        // by far less than the exponent range), so only the exponent pass
        // applies the mask.  A run's partial last tile takes 8 independent
        // partial maxima (three-input max) over its valid keys: the rows past
        // the run may hold another head's keys.
        // Keys [64, 128) are read first and only for their max; the scores of
        // keys [0, 64) stay in registers for pass 2 (band tiles, whose masking
        // needs the registers, read them again), whose probabilities then
        // overwrite only columns already read.
        float pm[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
        auto max_tree = [&](const uint32_t* x) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            pm[u] = max3f(pm[u], __uint_as_float(x[8 * u]), __uint_as_float(x[8 * u + 1]));
            pm[u] = max3f(pm[u], __uint_as_float(x[8 * u + 2]), __uint_as_float(x[8 * u + 3]));
            pm[u] = max3f(pm[u], __uint_as_float(x[8 * u + 4]), __uint_as_float(x[8 * u + 5]));
            pm[u] = max3f(pm[u], __uint_as_float(x[8 * u + 6]), __uint_as_float(x[8 * u + 7]));
          }
        };
        uint32_t x0[64];   // scores of keys [0, 64)
        if (full) {
          {
            uint32_t x[64];
            pm[1] = tmem_ld64_max(t_s + 64, x);
          }
          pm[0] = tmem_ld64_max(t_s, x0);
        } else {
          {
            uint32_t x[64];
            tmem_ld32x2(t_s + 64, t_s + 96, x);
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (64 + e >= valid) x[e] = __float_as_uint(-INFINITY);
            max_tree(x);
          }
          tmem_ld32x2(t_s, t_s + 32, x0);
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e >= valid) x0[e] = __float_as_uint(-INFINITY);
          max_tree(x0);
        }
        pm[0] = max3f(pm[0], pm[1], pm[2]);
        pm[3] = max3f(pm[3], pm[4], pm[5]);
        pm[6] = fmaxf(pm[6], pm[7]);
        const float m_new = fmaxf(m_run, max3f(pm[0], pm[3], pm[6]) * sl2);
        if (j == 0 || (CLS && j == p.cls_n01)) {
          m_run = m_new;
        } else if (__any_sync(0xffffffffu, m_new > m_run + RESCALE_LOG2)) {
          // O_i holds P_i(0..j-1) V, all of it complete (the commit that
          // signalled S_i(j) covers it): scale this warp's rows to the new max,
          // 16 columns at a time (the kept scores are live).
          // (A row still without any unmasked key keeps m = -inf and alpha 1.)
          const float alpha = m_new == -INFINITY ? 1.f : ex2(m_run - m_new);
          l_run *= alpha;
          m_run = m_new;
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            uint32_t o[16];
            tmem_ld16(t_o + c * 16, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(t_o + c * 16, o);
          }
          tmem_wait_st();
        }
        // Pass 2: probabilities 2^(s*scale*log2e - m), 64 keys at a time,
        // packed two per column into P_i (keys [64h, 64h+64) to columns
        // [32h, 32h+32)).  Masked keys become -inf, whose exponent is 0.
        // A row whose keys have all been masked so far keeps m = -inf; its
        // probabilities are all 0 (exponent of -inf), not NaN.
        const float neg_m = m_run == -INFINITY ? 0.f : -m_run;
        float ps[8];   // 4 independent pairs of partial sums
#pragma unroll
        for (int u = 0; u < 8; ++u) ps[u] = 0.f;
        auto exponents = [&](uint32_t* x, int h) {
          if (PROXY) {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (!((mw[2 * h + e / 32] >> (e & 31)) & 1u)) x[e] = __float_as_uint(-INFINITY);
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
        };
        if (PROXY) tmem_ld32x2(t_s, t_s + 32, x0);
        exponents(x0, 0);
        {
          uint32_t x[64];
          tmem_ld32x2(t_s + 64, t_s + 96, x);
          if (!full) {
#pragma unroll
            for (int e = 0; e < 64; ++e)
              if (64 + e >= valid) x[e] = __float_as_uint(-INFINITY);
          }
          exponents(x, 1);
        }
        l_run += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL + grp));
      }
      if (!ok) break;
      {
        // S_i of the item's last tile has been consumed: the query tile is
        // free for the next item, whose rows load in one round trip.
        TcItem nx;
        if (next_keyed(p, w + w_step, w_end, w_step, isrc, nx) < w_end) {
          issue_q(nx);
          finish_q();
        }
      }
      // ---------------------------------------------------------------- epilogue
      if (!wait_warp(B_ODONE + grp, nitem & 1)) { ok = false; break; }
      ++nitem;
      tc_fence_after();
      const TcItem it = tc_decode(p, w, isrc);
      // Final outputs are normalised; a split run's partial keeps O
      // unnormalised, with its row max and sum.
      const int mine_ok = qrow < it.nq ? 1 : 0;
      if (CLS) {
        // The Dummy segment's state is in TMEM; the Sink state and the state
        // before the Dummy segment are parked.  Full output = the two merged
        // (the softmax over all keys); then this token's cosines of the full
        // output with the Sink, Dummy and proxy outputs and the proxy's
        // squared error.
        const int token = it.q0 + qrow;
        const int64_t row = (int64_t)token * g.H + it.head;
        const int64_t row1 = ((int64_t)p.nq_total + token) * g.H + it.head;
        float2 ma = make_float2(0.f, 1.f), mb = make_float2(-INFINITY, 0.f);
        if (mine_ok) {
          ma = *reinterpret_cast<const float2*>(p.park_ml + row * 2);
          mb = *reinterpret_cast<const float2*>(p.park_ml + row1 * 2);
        }
        const float M = fmaxf(mb.x, m_run);
        const float fb = mb.x == -INFINITY ? 0.f : ex2(mb.x - M), fd = ex2(m_run - M);
        const float Lf = mb.y * fb + l_run * fd;
        const float inv_f = Lf > 0.f ? 1.f / Lf : 0.f, inv_a = ma.y > 0.f ? 1.f / ma.y : 0.f;
        const float inv_d = l_run > 0.f ? 1.f / l_run : 0.f;
        const float cb = fb * inv_f, cd = fd * inv_f;
        float ff = 0.f, ss = 0.f, dd = 0.f, pp = 0.f, fs = 0.f, fdm = 0.f, fq = 0.f, se = 0.f;
        const uint4* pa = reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.park_o) + row * D);
        const float4* pb = reinterpret_cast<const float4*>(p.park_o1 + row * D);
        const uint4* pb16 = reinterpret_cast<const uint4*>(reinterpret_cast<const bf16*>(p.park_o1) + row * D);
        const uint4* pq = reinterpret_cast<const uint4*>(static_cast<const bf16*>(p.proxy_o) + row * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
          if (!mine_ok) continue;
          uint32_t packed[16];
          uint4 a8[4], q8[4], b8[4];   // this chunk's 32 values of the bf16 planes
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            a8[e] = pa[c * 4 + e];
            q8[e] = pq[c * 4 + e];
            b8[e] = p.park1_bf16 ? pb16[c * 4 + e] : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const uint32_t aw0 = (&a8[e4 / 2].x)[2 * (e4 & 1)], aw1 = (&a8[e4 / 2].x)[2 * (e4 & 1) + 1];
            const uint32_t qw0 = (&q8[e4 / 2].x)[2 * (e4 & 1)], qw1 = (&q8[e4 / 2].x)[2 * (e4 & 1) + 1];
            const float av[4] = {bf16_lo(aw0), bf16_hi(aw0), bf16_lo(aw1), bf16_hi(aw1)};
            float bv[4];
            if (p.park1_bf16) {
              const uint32_t bw0 = (&b8[e4 / 2].x)[2 * (e4 & 1)], bw1 = (&b8[e4 / 2].x)[2 * (e4 & 1) + 1];
              bv[0] = bf16_lo(bw0);
              bv[1] = bf16_hi(bw0);
              bv[2] = bf16_lo(bw1);
              bv[3] = bf16_hi(bw1);
            } else {
              const float4 b4 = pb[c * 8 + e4];
              bv[0] = b4.x;
              bv[1] = b4.y;
              bv[2] = b4.z;
              bv[3] = b4.w;
            }
            const float qv[4] = {bf16_lo(qw0), bf16_hi(qw0), bf16_lo(qw1), bf16_hi(qw1)};
            float fv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float dv = __uint_as_float(o[4 * e4 + u]);
              const float f = bv[u] * cb + dv * cd;     // full
              const float sk = av[u] * inv_a;           // Sink
              const float dm = dv * inv_d;              // Dummy
              const float pr = qv[u];                   // proxy
              fv[u] = f;
              ff = fmaf(f, f, ff);
              ss = fmaf(sk, sk, ss);
              dd = fmaf(dm, dm, dd);
              pp = fmaf(pr, pr, pp);
              fs = fmaf(f, sk, fs);
              fdm = fmaf(f, dm, fdm);
              fq = fmaf(f, pr, fq);
              se = fmaf(pr - f, pr - f, se);
            }
            packed[2 * e4] = pack_bf16(fv[0], fv[1]);
            packed[2 * e4 + 1] = pack_bf16(fv[2], fv[3]);
            if (p.o_full && p.out_fp32)
              reinterpret_cast<float4*>(static_cast<float*>(p.o_full) + row * D + c * 32)[e4] =
                  make_float4(fv[0], fv[1], fv[2], fv[3]);
          }
          if (p.o_full && !p.out_fp32) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<bf16*>(p.o_full) + row * D + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
          }
        }
        if (mine_ok) {
          // Cosine with cos(0, 0) = 1 and cos(x, 0) = 0.
          auto cosine = [](float dot, float na2, float nb2) {
            if (na2 == 0.f && nb2 == 0.f) return 1.f;
            if (na2 == 0.f || nb2 == 0.f) return 0.f;
            return dot / (sqrtf(na2) * sqrtf(nb2));
          };
          const int64_t n = p.nq_total;
          p.tok[(0 * (int64_t)g.H + it.head) * n + token] = cosine(fs, ff, ss);
          p.tok[(1 * (int64_t)g.H + it.head) * n + token] = cosine(fdm, ff, dd);
          p.tok[(2 * (int64_t)g.H + it.head) * n + token] = cosine(fq, ff, pp);
          p.tok[(3 * (int64_t)g.H + it.head) * n + token] = se;
        }
      } else if (it.part >= 0) {
        float* po = p.part_o + ((int64_t)it.part * kPartRows + qrow) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
          if (!mine_ok) continue;
          float4* dst = reinterpret_cast<float4*>(po + c * 32);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                 __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
        }
      } else {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const int64_t base = mine_ok ? out_base(it) : 0;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
          if (!mine_ok) continue;
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
      }
      if (it.part >= 0 && mine_ok)
        *reinterpret_cast<float2*>(p.part_ml + ((int64_t)it.part * kPartRows + qrow) * 2) = make_float2(m_run, l_run);
      tc_fence_before();   // the next item's first P_i V overwrites O_i after the next PFULL
    }
    if (!ok) *abort_flag = 1;
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag && p.status) atomicExch(p.status, DEV_TIMEOUT);
  if (warp == W_MMA) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---------------------------------------------------------------- split-run merge
//
// One warp per query row of a split item: the partials of its chunks, each
// O_c = sum_j 2^(s_j - m_c) v_j with row sum l_c over the chunk's keys, merge
// into O = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c with M = max_c m_c,
// the softmax over the union of the chunks' keys.

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams c) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int s = gw / kPartRows, r = gw - s * kPartRows;
  if (s >= c.n_items) return;
  const SplitItem si = c.items[s];
  if (r >= si.nq) return;
  float M = -INFINITY;
  for (int k = 0; k < si.n_chunks; ++k) M = fmaxf(M, c.part_ml[((int64_t)(si.part0 + k) * kPartRows + r) * 2]);
  float acc[D / 32];
#pragma unroll
  for (int e = 0; e < D / 32; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int k = 0; k < si.n_chunks; ++k) {
    const int64_t row = (int64_t)(si.part0 + k) * kPartRows + r;
    const float m = c.part_ml[row * 2], l = c.part_ml[row * 2 + 1];
    if (m == -INFINITY) continue;   // an empty share
    const float f = exp2f(m - M);
    L = fmaf(l, f, L);
    const float* po = c.part_o + row * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) acc[e] = fmaf(po[lane + 32 * e], f, acc[e]);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  const int64_t base = ((int64_t)(si.q0 + r) * c.g.H + si.head) * D;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) {
    if (c.out_fp32) static_cast<float*>(c.o)[base + lane + 32 * e] = acc[e] * inv;
    else static_cast<bf16*>(c.o)[base + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
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

// K or V of band launches as a 5-D bf16 tensor [frames][Fh][Fw][heads][d];
// box {64, 1, kw, bh, 1} (one key box of a patch's halo), 128-byte swizzle.
cudaError_t make_band_map(CUtensorMap* m, const void* base, const Geom& g, int heads, int64_t frames, int kw,
                          int bh) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t e = 2;
  const cuuint64_t dims[5] = {(cuuint64_t)g.d, (cuuint64_t)heads, (cuuint64_t)g.Fw, (cuuint64_t)g.Fh, (cuuint64_t)frames};
  const cuuint64_t strides[4] = {(cuuint64_t)g.d * e, (cuuint64_t)heads * g.d * e, (cuuint64_t)g.Fw * heads * g.d * e,
                                 (cuuint64_t)g.F * heads * g.d * e};
  const cuuint32_t box[5] = {64, 1, (cuuint32_t)kw, (cuuint32_t)bh, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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

// Dynamic shared memory of a launch: the layout's bytes, but never less than
// half of an SM's shared memory, so that one CTA runs per SM (a second one
// would wait on its TMEM allocation while holding shared memory).
template <int D>
constexpr int smem_request() {
  return Layout<D>::ALLOC > 118 * 1024 ? Layout<D>::ALLOC : 118 * 1024;
}

template <int D, bool PROXY, bool CLS>
cudaError_t launch_d(const TcArgs& a, int ctas, cudaStream_t s) {
  constexpr int smem = smem_request<D>();
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
      e = cudaFuncSetAttribute(attn_tc_kernel<D, PROXY, CLS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  attn_tc_kernel<D, PROXY, CLS><<<ctas, NTHREADS, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int tc_block_rows() { return QT * BM; }
int tc_key_tile() { return BN; }

int device_sm_count() {
  constexpr int kMaxDevices = 128;
  static std::mutex mu;
  static int count[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kPlanCtas;
  std::lock_guard<std::mutex> lock(mu);
  if (count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = kPlanCtas;
    count[dev] = n;
  }
  return count[dev];
}

cudaError_t launch_attention_tc(const AttnParams& p, const TcKV& kv, int ctas, cudaStream_t s) {
  if (ctas <= 0 || p.n_items <= 0) return cudaSuccess;
  if (p.g.d != 64 && p.g.d != 128) return cudaErrorInvalidValue;
  if (kv.rows <= 0 || kv.rows > 0x7fffffffll) return cudaErrorInvalidValue;
  TcArgs a;
  memset(&a, 0, sizeof a);
  const bool band = p.item_mode == ITEMS_PROXY || p.band_win == WIN_SLIDING;
  cudaError_t e;
  if (band) {
    // Band launches read boxes of a patch's halo: K and V as frames of
    // Fh x Fw tokens (every key run of the cache is whole frames).
    if (kv.rows % p.g.F != 0 || p.pg.kw < 1 || p.pg.kw > 128 || p.pg.bh < 1 || p.pg.bh * p.pg.kw > BN)
      return cudaErrorInvalidValue;
    const int64_t frames = kv.rows / p.g.F;
    if ((e = make_band_map(&a.tk, kv.k, p.g, kv.heads, frames, p.pg.kw, p.pg.bh)) != cudaSuccess) return e;
    if ((e = make_band_map(&a.tv, kv.v, p.g, kv.heads, frames, p.pg.kw, p.pg.bh)) != cudaSuccess) return e;
  } else {
    if ((e = make_map(&a.tk, kv.k, p.g.d, kv.heads, kv.rows)) != cudaSuccess) return e;
    if ((e = make_map(&a.tv, kv.v, p.g.d, kv.heads, kv.rows)) != cudaSuccess) return e;
  }
  a.p = p;
  a.p.debug_stall = debug_stall_enabled() ? 1 : 0;
  a.p.wait_limit_ns = a.p.debug_stall ? STALL_WAIT_LIMIT_NS : WAIT_LIMIT_NS;
  a.kv_head_coord = kv.heads > 1 ? 1 : 0;
  // Band items (classification proxy, routed sliding Spatial) run the masked
  // variant; the caller launches them separately from the other items.
  if (band) return p.g.d == 128 ? launch_d<128, true, false>(a, ctas, s) : launch_d<64, true, false>(a, ctas, s);
  if (p.cls) return p.g.d == 128 ? launch_d<128, false, true>(a, ctas, s) : launch_d<64, false, true>(a, ctas, s);
  return p.g.d == 128 ? launch_d<128, false, false>(a, ctas, s) : launch_d<64, false, false>(a, ctas, s);
}

cudaError_t launch_combine(const CombineParams& c, cudaStream_t s) {
  if (c.n_items <= 0) return cudaSuccess;
  const int64_t threads = (int64_t)c.n_items * kPartRows * 32;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (c.g.d == 128) combine_kernel<128><<<blocks, 256, 0, s>>>(c);
  else if (c.g.d == 64) combine_kernel<64><<<blocks, 256, 0, s>>>(c);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace hc
