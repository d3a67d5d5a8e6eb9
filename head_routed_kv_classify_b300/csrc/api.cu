// Host side of the C ABI declared in include/headcast.h: argument checks,
// the restructured cache's layout and work list, and kernel launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include "hc_internal.h"

using hc::Geom;
using hc::HeadSlot;
using hc::SplitItem;
using hc::WorkItem;

// Device status word: kernels record bounded-wait expiry or a failed bounds
// check here instead of trapping; hc_get_last_error reads and clears it.
__device__ int g_hc_status_word;

struct hc_cache {
  hc_config cfg;
  Geom g;
  int8_t labels[HC_MAX_HEADS];
  HeadSlot heads[HC_MAX_HEADS];
  char* buf;
  size_t bytes, used, off_items, off_sched, off_split, off_k, off_v, off_part_o, off_part_ml;
  int n_items;
  int n_band;            // trailing band items (sliding Spatial heads), launched separately
  int n_cta_main, n_cta_band;
  int n_split;           // split key runs merged after the launch
  size_t split_bytes;    // partial-output workspace of the split runs
  int n_parts;           // pieces of the split runs
  int64_t plan_span, plan_total;   // the schedule's busiest CTA and total, key-tile steps
  hc::PatchGeom pg;      // patches of the sliding Spatial heads (tensor-core path)
  int64_t rows;
  int64_t rows_by_arch[4];
  int n_by_arch[4];
  int64_t newest;
  int valid_frames;
  bool sink_present;
};

namespace {

thread_local std::string g_msg;

hc_status fail(hc_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_msg = buf;
  return s;
}

hc_status cuda_fail(cudaError_t e, const char* what) {
  return fail(HC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define HC_CUDA(call, what)                        \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t esize_of(int dtype) { return dtype == HC_FP32 ? 4 : 2; }

Geom make_geom(const hc_config& c) {
  Geom g;
  g.H = c.n_heads;
  g.d = c.head_dim;
  g.Fh = c.frame_h;
  g.Fw = c.frame_w;
  g.F = c.frame_h * c.frame_w;
  g.fpb = c.frames_per_block;
  g.Wf = c.window_frames;
  g.blk = g.fpb * g.F;
  g.cell_h = c.cell_h;
  g.cell_w = c.cell_w;
  g.ncell_h = hc::n_cells(c.frame_h, c.cell_h);
  g.ncell_w = hc::n_cells(c.frame_w, c.cell_w);
  g.radius = c.proxy_radius;
  g.proxy_mode = c.proxy_mode;
  g.spatial_mode = c.spatial_mode;
  const double scale = c.softmax_scale > 0.f ? (double)c.softmax_scale : 1.0 / std::sqrt((double)c.head_dim);
  g.scale_log2 = (float)(scale * 1.4426950408889634);
  return g;
}

// Address of the status word on the current device.
hc_status status_ptr(int** out) {
  static std::mutex mu;
  static int* cached[128] = {nullptr};
  int dev = 0;
  HC_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= 128) return fail(HC_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    HC_CUDA(cudaGetSymbolAddress(&p, g_hc_status_word), "cudaGetSymbolAddress(status)");
    cached[dev] = static_cast<int*>(p);
  }
  *out = cached[dev];
  return HC_OK;
}

bool finite_all(std::initializer_list<float> xs) {
  for (float x : xs)
    if (!std::isfinite(x)) return false;
  return true;
}

// Per-head rows of the restructured cache.
int64_t head_rows(const Geom& g, int arch) {
  return (arch == HC_SINK || arch == HC_DUMMY) ? (int64_t)g.blk : (int64_t)g.Wf * g.F;
}

struct Plan {
  std::vector<WorkItem> items;       // main items in CTA order, then band items in CTA order
  std::vector<int32_t> sched_main;   // CTA c of the main launch: items [sched[c], sched[c+1])
  std::vector<int32_t> sched_band;   // the same for the band launch (offsets into the band items)
  std::vector<SplitItem> splits;
  int n_band = 0;
  int n_parts = 0;
  HeadSlot heads[HC_MAX_HEADS];
  int64_t rows = 0;
  int64_t rows_by_arch[4] = {0, 0, 0, 0};
  int n_by_arch[4] = {0, 0, 0, 0};
  size_t off_items = 0, off_sched = 0, off_split = 0, off_k = 0, off_v = 0, off_part_o = 0, off_part_ml = 0;
  size_t bytes = 0, split_bytes = 0;
  hc::PatchGeom pg;      // patches of the sliding Spatial heads (tensor-core path)
  int64_t span = 0;      // planned busiest CTA (main launch + band launch), key-tile steps
  int64_t total = 0;     // planned work over all CTAs, key-tile steps
  bool ok = true;        // false: no patch geometry fits the sliding window
};

hc_status check_labels(const hc_config* cfg, const int8_t* labels) {
  if (!labels) return fail(HC_ERR_INVALID_ARG, "labels_host is null");
  for (int h = 0; h < cfg->n_heads; ++h)
    if (labels[h] < HC_SINK || labels[h] > HC_GLOBAL)
      return fail(HC_ERR_INVALID_ARG, "label %d of head %d is not an archetype", labels[h], h);
  return HC_OK;
}

constexpr int kKeyTile = 128;   // keys per tile of the tensor-core kernel
constexpr int kMaxChunks = 8;   // most pieces a key run is split into
constexpr int kItemOverhead = 6;   // an item boundary, in key-tile steps (measured: about 8 us)

// Key tiles of an item with the window full (the steady state), plus the
// item boundary: the cost the schedule balances.
int64_t item_cost(const Geom& g, const WorkItem& w, const hc::PatchGeom* pg = nullptr) {
  int64_t keys;
  if (w.kind == hc::ITEM_PATCH && pg) return (int64_t)g.Wf * pg->tpf + kItemOverhead;
  if (w.kind == hc::ITEM_BAND) {
    int lo, rhi, wl, wh, rlo;
    const int t0 = w.q0 % g.F;
    hc::band_window(g, hc::WIN_SLIDING, t0 / g.Fw, 0, rlo, rhi, wl, wh);
    hc::band_window(g, hc::WIN_SLIDING, (t0 + w.nq - 1) / g.Fw, 0, lo, rhi, wl, wh);
    const int64_t tpf = ((int64_t)(rhi - rlo + 1) * g.Fw + kKeyTile - 1) / kKeyTile;
    return (int64_t)g.Wf * tpf + kItemOverhead;
  }
  keys = w.k_per_frame > 0 ? (int64_t)w.k_per_frame * g.Wf : w.k_len;
  const int64_t tiles = (keys + kKeyTile - 1) / kKeyTile;
  return (w.n_chunks > 1 ? (tiles + w.n_chunks - 1) / w.n_chunks : tiles) + kItemOverhead;
}

int64_t run_tiles(const Geom& g, const WorkItem& w) {
  const int64_t keys = w.k_per_frame > 0 ? (int64_t)w.k_per_frame * g.Wf : w.k_len;
  return (keys + kKeyTile - 1) / kKeyTile;
}

// Finishing time of the busiest CTA when items of these costs are dealt
// longest-first to `ctas` CTAs, each to the least loaded one.
int64_t lpt_makespan(std::vector<int64_t> costs, int ctas) {
  std::sort(costs.begin(), costs.end(), std::greater<int64_t>());
  std::priority_queue<int64_t, std::vector<int64_t>, std::greater<int64_t>> heap;
  for (int c = 0; c < ctas; ++c) heap.push(0);
  int64_t span = 0;
  for (int64_t x : costs) {
    const int64_t l = heap.top() + x;
    heap.pop();
    heap.push(l);
    span = std::max(span, l);
  }
  return span;
}

// Longest-processing-time-first assignment of items to `ctas` CTAs: items in
// decreasing cost, each to the CTA with the least work so far.  Returns the
// items regrouped per CTA (each CTA's in assignment order) and the ranges.
// The busiest CTA's cost is returned, the sum over CTAs added to *total.
int64_t lpt_schedule(const Geom& g, std::vector<WorkItem>& items, int max_ctas, std::vector<int32_t>& sched,
                     int64_t* total, const hc::PatchGeom* pg = nullptr) {
  const int n = (int)items.size();
  const int ctas = std::max(1, std::min(max_ctas, n));
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::vector<int64_t> cost(n);
  for (int i = 0; i < n; ++i) cost[i] = item_cost(g, items[i], pg);
  // Equal costs keep their list order, so items that read the same key run
  // (adjacent in the list) go to neighbouring CTAs and run at the same time,
  // and all but the first read the run from L2.
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  typedef std::pair<int64_t, int> Load;   // (work so far, cta)
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < ctas; ++c) heap.push(Load(0, c));
  std::vector<std::vector<int>> lists(ctas);
  int64_t span = 0;
  for (int i : order) {
    Load l = heap.top();
    heap.pop();
    lists[l.second].push_back(i);
    heap.push(Load(l.first + cost[i], l.second));
    span = std::max(span, l.first + cost[i]);
    *total += cost[i];
  }
  std::vector<WorkItem> out;
  out.reserve(n);
  sched.assign(ctas + 1, 0);
  for (int c = 0; c < ctas; ++c) {
    sched[c] = (int32_t)out.size();
    for (int i : lists[c]) out.push_back(items[i]);
  }
  sched[ctas] = (int32_t)out.size();
  items.swap(out);
  return span;
}

// Split-KV: some of the longest key runs (Sink, Dummy or Global items) are
// cut into pieces whose partial outputs are merged after the launch, where
// that shortens the launch's busiest CTA by more than 5 %.  It removes both a
// single item that outlasts the rest of the launch and the quantisation of a
// few long items over the CTAs (507 equal items on 148 CTAs leave 63 CTAs with
// a fourth item; splitting 63 of them in halves evens that out).  Searched:
// the m longest runs, each in c pieces.  Pieces replace their item in `main`;
// `splits` gets one entry per split run, `n_parts` counts the pieces.
void split_runs(const Geom& g, std::vector<WorkItem>& main, std::vector<SplitItem>& splits, int& n_parts) {
  if (main.empty()) return;
  const int n = (int)main.size();
  std::vector<int> runs;
  for (int i = 0; i < n; ++i)
    if (main[i].kind == hc::ITEM_RANGE) runs.push_back(i);
  std::stable_sort(runs.begin(), runs.end(),
                   [&](int a, int b) { return run_tiles(g, main[a]) > run_tiles(g, main[b]); });
  auto span_of = [&](const std::vector<int>& ch) {
    std::vector<int64_t> c;
    for (int i = 0; i < n; ++i) {
      const int64_t t = main[i].kind == hc::ITEM_RANGE ? run_tiles(g, main[i]) : item_cost(g, main[i]) - kItemOverhead;
      // A piece of a split run also writes its partial output and is read
      // back by the merge: one more step.
      for (int k = 0; k < ch[i]; ++k) c.push_back((t + ch[i] - 1) / ch[i] + kItemOverhead + (ch[i] > 1 ? 1 : 0));
    }
    return lpt_makespan(c, hc::kPlanCtas);
  };
  std::vector<int> best(n, 1);
  const int64_t base_span = span_of(best);
  int64_t best_span = base_span;
  const int nr = (int)runs.size();
  const int step = std::max(1, nr / 64);
  for (int c = 2; c <= kMaxChunks && nr > 0; ++c) {
    for (int m = std::min(step, nr);; m = std::min(m + step, nr)) {
      if ((run_tiles(g, main[runs[m - 1]]) + c - 1) / c < 8) break;   // pieces under 8 key tiles: no
      std::vector<int> ch(n, 1);
      for (int k = 0; k < m; ++k) ch[runs[k]] = c;
      const int64_t s = span_of(ch);
      if (s < best_span) {
        best_span = s;
        best = ch;
      }
      if (m == nr) break;
    }
  }
  if (best_span * 100 >= base_span * 95) best.assign(n, 1);
  std::vector<WorkItem> split;
  for (int i = 0; i < n; ++i) {
    const WorkItem& w = main[i];
    const int k = best[i];
    if (k <= 1) {
      split.push_back(w);
      continue;
    }
    SplitItem si;
    std::memset(&si, 0, sizeof si);
    si.head = w.head;
    si.q0 = w.q0;
    si.nq = w.nq;
    si.n_chunks = k;
    si.part0 = n_parts;
    splits.push_back(si);
    for (int c = 0; c < k; ++c) {
      WorkItem x = w;
      x.chunk = (int16_t)c;
      x.n_chunks = (int16_t)k;
      x.part = n_parts + c;
      split.push_back(x);
    }
    n_parts += k;
  }
  main.swap(split);
}

// Cache layout, the routed work list and its schedule.
void plan_cache(const hc_config& cfg, const int8_t* labels, Plan& P) {
  const Geom g = make_geom(cfg);
  const int BM = hc::attention_block_rows(cfg.dtype, cfg.head_dim);
  std::vector<WorkItem> main, band;
  std::memset(&P.pg, 0, sizeof P.pg);
  const bool patches = cfg.dtype == HC_BF16 && g.spatial_mode == HC_SPATIAL_SLIDING;
  if (patches) {
    bool any = false;
    for (int h = 0; h < g.H; ++h) any = any || labels[h] == HC_SPATIAL;
    if (any && !hc::choose_patch_geom(g, hc::WIN_SLIDING, g.Wf, P.pg)) P.ok = false;
  }
  for (int h = 0; h < g.H; ++h) {
    const int a = labels[h];
    P.heads[h].arch = a;
    P.heads[h].pad = 0;
    P.heads[h].row0 = P.rows;
    const int64_t r = head_rows(g, a);
    P.rows += r;
    P.rows_by_arch[a] += r;
    P.n_by_arch[a] += 1;
    auto push = [&](std::vector<WorkItem>& list, int kind, int q0, int nq, int64_t k_row0, int k_len,
                    int k_per_frame, int cell) {
      WorkItem w;
      std::memset(&w, 0, sizeof w);
      w.head = h;
      w.kind = kind;
      w.q0 = q0;
      w.nq = nq;
      w.k_row0 = k_row0;
      w.k_len = k_len;
      w.k_per_frame = k_per_frame;
      w.cell = cell;
      w.out_plane = 0;
      w.chunk = 0;
      w.n_chunks = 1;
      w.part = -1;
      list.push_back(w);
    };
    if (a == HC_SINK || a == HC_DUMMY) {
      for (int q0 = 0; q0 < g.blk; q0 += BM)
        push(main, hc::ITEM_RANGE, q0, std::min(BM, g.blk - q0), P.heads[h].row0, g.blk, 0, 0);
    } else if (a == HC_GLOBAL) {
      for (int q0 = 0; q0 < g.blk; q0 += BM)
        push(main, hc::ITEM_RANGE, q0, std::min(BM, g.blk - q0), P.heads[h].row0, 0, g.F, 0);
    } else if (g.spatial_mode == HC_SPATIAL_SLIDING && patches) {
      // Patches of query positions (in every frame of the block); the kernel
      // reads each patch's halo as boxes and masks each query's window.
      for (int k = 0; k < P.pg.n; ++k) push(band, hc::ITEM_PATCH, 0, 0, P.heads[h].row0, 0, g.F, k);
    } else if (g.spatial_mode == HC_SPATIAL_SLIDING) {
      // Runs of up to BM tokens inside one frame of the block; the kernel
      // derives the band of window rows and masks each query's window.
      for (int f = 0; f < g.fpb; ++f)
        for (int t0 = 0; t0 < g.F; t0 += BM)
          push(band, hc::ITEM_BAND, f * g.F + t0, std::min(BM, g.F - t0), P.heads[h].row0, 0, g.F, 0);
    } else {
      for (int ci = 0; ci < g.ncell_h; ++ci)
        for (int cj = 0; cj < g.ncell_w; ++cj) {
          const int hz = hc::cell_extent(ci, g.Fh, g.cell_h, g.ncell_h);
          const int wz = hc::cell_extent(cj, g.Fw, g.cell_w, g.ncell_w);
          const int csz = hz * wz, nq = g.fpb * csz;
          const int64_t k0 = P.heads[h].row0 + (int64_t)g.Wf * hc::cell_tokens_before(g, ci, cj);
          for (int q0 = 0; q0 < nq; q0 += BM)
            push(main, hc::ITEM_CELL, q0, std::min(BM, nq - q0), k0, 0, csz, ci * g.ncell_w + cj);
        }
    }
  }
  if (cfg.dtype == HC_BF16) split_runs(g, main, P.splits, P.n_parts);
  P.span = lpt_schedule(g, main, hc::kPlanCtas, P.sched_main, &P.total);
  if (!band.empty()) P.span += lpt_schedule(g, band, hc::kPlanCtas, P.sched_band, &P.total, &P.pg);
  P.n_band = (int)band.size();
  P.items = main;
  P.items.insert(P.items.end(), band.begin(), band.end());
  const size_t row_bytes = (size_t)g.d * esize_of(cfg.dtype);
  P.off_items = 256;
  P.off_sched = round_up(P.off_items + P.items.size() * sizeof(WorkItem), 256);
  P.off_split = round_up(P.off_sched + 2 * (hc::kMaxCtas + 1) * sizeof(int32_t), 256);
  P.off_k = round_up(P.off_split + P.splits.size() * sizeof(SplitItem), 256);
  P.off_v = round_up(P.off_k + (size_t)P.rows * row_bytes, 256);
  P.off_part_o = round_up(P.off_v + (size_t)P.rows * row_bytes, 256);
  P.off_part_ml = round_up(P.off_part_o + (size_t)P.n_parts * hc::kPartRows * g.d * sizeof(float), 256);
  P.bytes = round_up(P.off_part_ml + (size_t)P.n_parts * hc::kPartRows * 2 * sizeof(float), 256);
  P.split_bytes = P.bytes - P.off_part_o;
}

// Full attention's balanced schedule: every head's queries in 256-query
// items over the whole key window, dealt longest-first with long runs split
// (the routed launch's planner), and the workspace that holds the list, the
// schedule, the split table and the pieces' partial outputs.  Planning takes
// milliseconds, so plans are kept per shape.
struct FullPlan {
  std::vector<WorkItem> items;
  std::vector<int32_t> sched;
  std::vector<SplitItem> splits;
  int n_parts = 0;
  size_t off_items = 0, off_sched = 0, off_split = 0, off_part_o = 0, off_part_ml = 0, bytes = 0;
};

std::shared_ptr<const FullPlan> full_plan(const hc_config& cfg, int32_t n_q_tokens, int32_t n_key_frames) {
  static std::mutex mu;
  static std::map<std::vector<int64_t>, std::shared_ptr<const FullPlan>> plans;
  const std::vector<int64_t> key = {cfg.n_heads, cfg.head_dim, cfg.frame_h, cfg.frame_w, cfg.frames_per_block,
                                    cfg.window_frames, n_q_tokens, n_key_frames};
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = plans.find(key);
    if (it != plans.end()) return it->second;
  }
  const Geom g = make_geom(cfg);
  const int BM = hc::attention_block_rows(cfg.dtype, cfg.head_dim);
  const int64_t nk = (int64_t)n_key_frames * g.F;
  auto P = std::make_shared<FullPlan>();
  for (int h = 0; h < g.H; ++h)
    for (int q0 = 0; q0 < n_q_tokens; q0 += BM) {
      WorkItem w;
      std::memset(&w, 0, sizeof w);
      w.head = h;
      w.kind = hc::ITEM_RANGE;
      w.q0 = q0;
      w.nq = std::min(BM, n_q_tokens - q0);
      w.k_row0 = 0;
      w.k_len = (int32_t)nk;
      w.n_chunks = 1;
      w.part = -1;
      P->items.push_back(w);
    }
  split_runs(g, P->items, P->splits, P->n_parts);
  int64_t total = 0;
  lpt_schedule(g, P->items, hc::kPlanCtas, P->sched, &total);
  P->off_items = 0;
  P->off_sched = round_up(P->items.size() * sizeof(WorkItem), 256);
  P->off_split = round_up(P->off_sched + P->sched.size() * sizeof(int32_t), 256);
  P->off_part_o = round_up(P->off_split + P->splits.size() * sizeof(SplitItem), 256);
  P->off_part_ml = round_up(P->off_part_o + (size_t)P->n_parts * hc::kPartRows * g.d * sizeof(float), 256);
  P->bytes = round_up(P->off_part_ml + (size_t)P->n_parts * hc::kPartRows * 2 * sizeof(float), 256);
  std::lock_guard<std::mutex> lock(mu);
  plans[key] = P;
  return P;
}

}  // namespace

static std::atomic<int> g_debug_stall{0};
bool hc::debug_stall_enabled() { return g_debug_stall.load() != 0; }

hc_status hc::record_error(hc_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_msg = buf;
  return s;
}

// ===========================================================================

extern "C" {

int32_t hc_abi_version(void) { return HC_ABI_VERSION; }

const char* hc_status_string(hc_status s) {
  switch (s) {
    case HC_OK: return "ok";
    case HC_ERR_INVALID_ARG: return "invalid argument";
    case HC_ERR_SHAPE: return "unsupported or inconsistent shape";
    case HC_ERR_DTYPE: return "unsupported dtype";
    case HC_ERR_ALIGN: return "pointer not 16-byte aligned";
    case HC_ERR_STATE: return "call not valid in the current state";
    case HC_ERR_CUDA: return "CUDA error";
    case HC_ERR_TIMEOUT: return "device-side wait expired";
    case HC_ERR_UNSUPPORTED: return "unsupported";
    case HC_ERR_SIZE: return "buffer too small";
  }
  return "unknown status";
}

const char* hc_last_error_message(void) { return g_msg.c_str(); }

hc_status hc_config_default(hc_config* out) {
  if (!out) return fail(HC_ERR_INVALID_ARG, "out is null");
  std::memset(out, 0, sizeof *out);
  out->frames_per_block = 3;
  out->window_frames = 21;
  out->dtype = HC_BF16;
  out->softmax_scale = 0.f;
  out->theta_sink = 0.95f;
  out->theta_dummy = 0.95f;
  out->theta_spatial = 0.95f;
  out->theta_score = 0.755f;
  out->gamma = 5.f;
  out->proxy_radius = 2;
  out->cell_h = 10;
  out->cell_w = 10;
  return HC_OK;
}

hc_status hc_config_validate(const hc_config* c) {
  if (!c) return fail(HC_ERR_INVALID_ARG, "config is null");
  if (c->n_heads < 1 || c->n_heads > HC_MAX_HEADS)
    return fail(HC_ERR_SHAPE, "n_heads %d not in 1..%d", c->n_heads, HC_MAX_HEADS);
  if (c->head_dim != 64 && c->head_dim != 128)
    return fail(HC_ERR_SHAPE, "head_dim %d not 64 or 128", c->head_dim);
  if (c->frame_h < 1 || c->frame_w < 1 || c->frame_h > 4096 || c->frame_w > 4096)
    return fail(HC_ERR_SHAPE, "frame %dx%d out of range", c->frame_h, c->frame_w);
  if ((int64_t)c->frame_h * c->frame_w > (1 << 22))
    return fail(HC_ERR_SHAPE, "frame of %lld tokens too large", (long long)c->frame_h * c->frame_w);
  if (c->frames_per_block < 1 || c->frames_per_block > 64)
    return fail(HC_ERR_SHAPE, "frames_per_block %d out of range", c->frames_per_block);
  if (c->window_frames < c->frames_per_block || c->window_frames % c->frames_per_block != 0 ||
      c->window_frames > 4096)
    return fail(HC_ERR_SHAPE, "window_frames %d is not a positive multiple of frames_per_block %d",
                c->window_frames, c->frames_per_block);
  if ((int64_t)c->frames_per_block * c->frame_h * c->frame_w * c->n_heads * c->head_dim >= (1ll << 31) ||
      (int64_t)c->frames_per_block * c->frame_h * c->frame_w >= (1 << 24))
    return fail(HC_ERR_SHAPE, "block too large");
  if (c->dtype != HC_BF16 && c->dtype != HC_FP32) return fail(HC_ERR_DTYPE, "dtype %d", c->dtype);
  if (!finite_all({c->softmax_scale, c->theta_sink, c->theta_dummy, c->theta_spatial, c->theta_score, c->gamma}) ||
      c->softmax_scale < 0.f)
    return fail(HC_ERR_INVALID_ARG, "non-finite threshold or negative scale");
  if (c->proxy_radius < 0 || c->cell_h < 1 || c->cell_w < 1)
    return fail(HC_ERR_INVALID_ARG, "proxy_radius %d / cell %dx%d", c->proxy_radius, c->cell_h, c->cell_w);
  if (c->proxy_mode != HC_PROXY_NEIGHBOURHOOD && c->proxy_mode != HC_PROXY_CELL)
    return fail(HC_ERR_INVALID_ARG, "proxy_mode %d is not 0 or 1", c->proxy_mode);
  if (c->spatial_mode != HC_SPATIAL_CELLS && c->spatial_mode != HC_SPATIAL_SLIDING)
    return fail(HC_ERR_INVALID_ARG, "spatial_mode %d is not 0 or 1", c->spatial_mode);
  return HC_OK;
}

// ------------------------------------------------------------ classification

// Classification workspace.  bf16 layers (tensor-core path): the proxy
// output plane, the two parked states of the fused pass and their row
// max / sum, and the per-token statistics.  fp32 layers: four output planes
// (full, Sink, Dummy, proxy) and the per-token statistics.
struct ClassifyLayout {
  size_t plane, off_proxy, off_park, off_park1, off_park_ml, off_tok, total;
};

static ClassifyLayout classify_layout(const hc_config& c) {
  const int64_t nq = (int64_t)c.frames_per_block * c.frame_h * c.frame_w;
  ClassifyLayout L;
  L.plane = (size_t)nq * c.n_heads * c.head_dim * sizeof(float);
  const size_t tok = 4 * (size_t)c.n_heads * nq * sizeof(float);
  if (c.dtype == HC_BF16) {
    // bf16 planes for the proxy output and the parked Sink state; the state
    // before the Dummy block stays fp32 (the full-context output is made
    // from it).
    const size_t plane16 = L.plane / 2;
    L.off_proxy = 0;
    L.off_park = round_up(plane16, 256);
    L.off_park1 = round_up(L.off_park + plane16, 256);
    L.off_park_ml = round_up(L.off_park1 + L.plane, 256);
    L.off_tok = round_up(L.off_park_ml + 2 * (size_t)nq * c.n_heads * 2 * sizeof(float), 256);
  } else {
    L.off_proxy = 3 * L.plane;
    L.off_park = L.off_park1 = L.off_park_ml = 0;
    L.off_tok = round_up(4 * L.plane, 256);
  }
  L.total = round_up(L.off_tok + tok, 256);
  return L;
}

hc_status hc_classify_scratch_bytes(const hc_config* cfg, int32_t n_key_frames, size_t* bytes) {
  hc_status s = hc_config_validate(cfg);
  if (s != HC_OK) return s;
  if (!bytes) return fail(HC_ERR_INVALID_ARG, "bytes is null");
  (void)n_key_frames;
  *bytes = classify_layout(*cfg).total;
  return HC_OK;
}

hc_status hc_classify(const hc_config* cfg, const void* q, const void* k, const void* v,
                      int32_t n_key_frames, int8_t* labels_dev, int8_t* labels_host,
                      float* stats_dev, void* o_full, void* scratch, size_t scratch_bytes,
                      void* stream) {
  hc_status s = hc_config_validate(cfg);
  if (s != HC_OK) return s;
  if (!q || !k || !v || !labels_dev || !scratch)
    return fail(HC_ERR_INVALID_ARG, "q, k, v, labels_dev and scratch must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(scratch) ||
      (o_full && !aligned16(o_full)) || (stats_dev && !aligned16(stats_dev)))
    return fail(HC_ERR_ALIGN, "device pointers must be 16-byte aligned");
  if (n_key_frames < 2 * cfg->frames_per_block || n_key_frames % cfg->frames_per_block != 0 ||
      n_key_frames > 4096)
    return fail(HC_ERR_SHAPE, "n_key_frames %d must be a multiple of frames_per_block and hold >= 2 blocks",
                n_key_frames);
  const ClassifyLayout CL = classify_layout(*cfg);
  if (scratch_bytes < CL.total) return fail(HC_ERR_SIZE, "scratch %zu < %zu bytes", scratch_bytes, CL.total);
  char* sc = static_cast<char*>(scratch);
  int* status = nullptr;
  if ((s = status_ptr(&status)) != HC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Geom g = make_geom(*cfg);
  const int BM = hc::attention_block_rows(cfg->dtype, cfg->head_dim);
  const int64_t nk = (int64_t)n_key_frames * g.F;

  hc::AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.k_stride = (int64_t)g.H * g.d;
  p.k_hstride = g.d;
  p.nq_total = g.blk;
  p.out_fp32 = 1;
  p.g = g;
  p.status = status;
  if (cfg->dtype == HC_BF16) {
    const hc::TcKV kv{k, v, g.H, nk};
    // 1. The Spatial proxy output: patches of query positions with their
    //    halo in every window frame (with the cell proxy: the deployed cells).
    hc::AttnParams pp = p;
    pp.item_mode = hc::ITEMS_PROXY;
    pp.o = sc + CL.off_proxy;
    pp.o_plane_stride = 0;
    pp.out_fp32 = 0;
    pp.proxy_frames = n_key_frames;
    const bool pg_ok = g.proxy_mode == HC_PROXY_CELL ? hc::make_cell_patch_geom(g, pp.pg)
                                                      : hc::choose_patch_geom(g, hc::WIN_PROXY, n_key_frames, pp.pg);
    if (!pg_ok) return fail(HC_ERR_UNSUPPORTED, "the Spatial proxy window is too wide for the band kernel");
    pp.band_win = hc::WIN_PROXY;
    pp.n_items = g.H * pp.pg.n * pp.pg.cpc;
    HC_CUDA(hc::launch_attention_tc(pp, kv, std::min(pp.n_items, hc::device_sm_count()), st),
            "classification proxy attention");
    // 2. One pass over all keys per query tile: the full-context output,
    //    with the Sink block's and the current block's outputs taken from its
    //    running state, and each token's cosines and squared error.
    hc::AttnParams pc = p;
    pc.item_mode = hc::ITEMS_DENSE;
    pc.n_planes = 1;
    pc.plane_k0[0] = 0;
    pc.plane_klen[0] = (int32_t)nk;
    pc.cls = 1;
    pc.seg_sink = g.blk;
    pc.seg_dummy = (int32_t)(nk - g.blk);
    {
      const int kt = hc::tc_key_tile();
      const int n0 = (pc.seg_sink + kt - 1) / kt, n1 = (pc.seg_dummy - pc.seg_sink + kt - 1) / kt;
      const int n2 = ((int)nk - pc.seg_dummy + kt - 1) / kt;
      pc.cls_n0 = n0;
      pc.cls_n01 = n0 + n1;
      pc.cls_v0 = pc.seg_sink - (n0 - 1) * kt;
      pc.cls_v1 = n1 > 0 ? (pc.seg_dummy - pc.seg_sink) - (n1 - 1) * kt : 0;
      pc.cls_v2 = ((int)nk - pc.seg_dummy) - (n2 - 1) * kt;
    }
    pc.park_o = sc + CL.off_park;
    pc.park_o1 = reinterpret_cast<float*>(sc + CL.off_park1);
    // The state before the Dummy block builds the full-context output: fp32
    // when the caller wants that output, else bf16 (it then feeds only the
    // cosines and squared errors, as the parked Sink state does).
    pc.park1_bf16 = o_full ? 0 : 1;
    pc.park_ml = reinterpret_cast<float*>(sc + CL.off_park_ml);
    pc.proxy_o = sc + CL.off_proxy;
    pc.tok = reinterpret_cast<float*>(sc + CL.off_tok);
    pc.o_full = o_full;
    pc.out_fp32 = 0;
    pc.n_items = ((g.blk + BM - 1) / BM) * g.H;
    HC_CUDA(hc::launch_attention_tc(pc, kv, std::min(pc.n_items, hc::device_sm_count()), st),
            "classification attention");
  } else {
    // fp32 layers: the four outputs as planes, then the statistics kernel.
    p.o = scratch;
    p.o_plane_stride = (int64_t)(CL.plane / sizeof(float));
    p.item_mode = hc::ITEMS_DENSE;
    p.n_planes = 3;
    p.plane_k0[0] = 0;
    p.plane_klen[0] = (int32_t)nk;
    p.plane_k0[1] = 0;
    p.plane_klen[1] = g.blk;
    p.plane_k0[2] = nk - g.blk;
    p.plane_klen[2] = g.blk;
    HC_CUDA(hc::launch_attention(p, cfg->dtype, dim3((g.blk + BM - 1) / BM, g.H, 3), st),
            "classification attention");
    p.item_mode = hc::ITEMS_PROXY;
    p.proxy_frames = n_key_frames;
    const int PBM = hc::proxy_block_rows();
    p.tiles_per_frame = (g.F + PBM - 1) / PBM;
    HC_CUDA(hc::launch_attention(p, cfg->dtype, dim3(g.fpb * p.tiles_per_frame, g.H, 1), st),
            "classification proxy attention");
  }

  hc::ClassifyPost c;
  std::memset(&c, 0, sizeof c);
  c.planes = static_cast<const float*>(scratch);
  c.plane_stride = (int64_t)(CL.plane / sizeof(float));
  c.tok = reinterpret_cast<float*>(sc + CL.off_tok);
  c.tokens_ready = cfg->dtype == HC_BF16 ? 1 : 0;   // the fused pass wrote them
  c.o_full = o_full;
  c.o_full_fp32 = cfg->dtype == HC_FP32;
  c.labels = labels_dev;
  c.stats = stats_dev;
  c.nq = g.blk;
  c.g = g;
  c.theta_sink = cfg->theta_sink;
  c.theta_dummy = cfg->theta_dummy;
  c.theta_spatial = cfg->theta_spatial;
  c.theta_score = cfg->theta_score;
  c.gamma = cfg->gamma;
  c.status = status;
  HC_CUDA(hc::launch_classify_post(c, st), "classification statistics");
  if (labels_host) {
    HC_CUDA(cudaMemcpyAsync(labels_host, labels_dev, g.H, cudaMemcpyDeviceToHost, st), "label copy");
    HC_CUDA(cudaStreamSynchronize(st), "stream synchronize");
    // A bounded wait that expired in any of the kernels leaves its mark in
    // the status word (which stays set for hc_get_last_error): the labels
    // were then not computed from complete outputs.
    int word = 0;
    HC_CUDA(cudaMemcpy(&word, status, sizeof word, cudaMemcpyDeviceToHost), "status read");
    if (word == hc::DEV_TIMEOUT) return fail(HC_ERR_TIMEOUT, "a bounded device wait expired during classification");
    if (word != hc::DEV_OK) return fail(HC_ERR_CUDA, "device status word %d", word);
  }
  return HC_OK;
}

// ------------------------------------------------------------ cache

hc_status hc_cache_bytes(const hc_config* cfg, const int8_t* labels_host, size_t* bytes) {
  hc_status s = hc_config_validate(cfg);
  if (s != HC_OK) return s;
  if ((s = check_labels(cfg, labels_host)) != HC_OK) return s;
  if (!bytes) return fail(HC_ERR_INVALID_ARG, "bytes is null");
  Plan P;
  plan_cache(*cfg, labels_host, P);
  if (!P.ok)
    return fail(HC_ERR_UNSUPPORTED, "the sliding Spatial window (%dx%d) is too wide for the band kernel", cfg->cell_h,
                cfg->cell_w);
  *bytes = P.bytes;
  return HC_OK;
}

hc_status hc_cache_create(const hc_config* cfg, const int8_t* labels_host, void* buf, size_t bytes,
                          hc_cache** out) {
  hc_status s = hc_config_validate(cfg);
  if (s != HC_OK) return s;
  if ((s = check_labels(cfg, labels_host)) != HC_OK) return s;
  if (!buf || !out) return fail(HC_ERR_INVALID_ARG, "buf and out must be non-null");
  if ((reinterpret_cast<uintptr_t>(buf) & 255u) != 0) return fail(HC_ERR_ALIGN, "buf must be 256-byte aligned");
  Plan P;
  plan_cache(*cfg, labels_host, P);
  if (!P.ok)
    return fail(HC_ERR_UNSUPPORTED, "the sliding Spatial window (%dx%d) is too wide for the band kernel", cfg->cell_h,
                cfg->cell_w);
  if (bytes < P.bytes) return fail(HC_ERR_SIZE, "buffer %zu < %zu bytes", bytes, P.bytes);
  if (!P.items.empty())
    HC_CUDA(cudaMemcpy(static_cast<char*>(buf) + P.off_items, P.items.data(),
                       P.items.size() * sizeof(WorkItem), cudaMemcpyHostToDevice),
            "work-list upload");
  std::vector<int32_t> sched(2 * (hc::kMaxCtas + 1), 0);
  std::copy(P.sched_main.begin(), P.sched_main.end(), sched.begin());
  std::copy(P.sched_band.begin(), P.sched_band.end(), sched.begin() + hc::kMaxCtas + 1);
  HC_CUDA(cudaMemcpy(static_cast<char*>(buf) + P.off_sched, sched.data(), sched.size() * sizeof(int32_t),
                     cudaMemcpyHostToDevice),
          "schedule upload");
  if (!P.splits.empty())
    HC_CUDA(cudaMemcpy(static_cast<char*>(buf) + P.off_split, P.splits.data(), P.splits.size() * sizeof(SplitItem),
                       cudaMemcpyHostToDevice),
            "split-table upload");
  // Clear the K/V areas: a run's last key tile reads past its filled ring
  // slots while the window is still filling, and the masked probabilities
  // (0) times uninitialised V rows could be 0 * NaN.
  HC_CUDA(cudaMemset(static_cast<char*>(buf) + P.off_k, 0, P.off_part_o - P.off_k), "cache clear");
  HC_CUDA(cudaStreamSynchronize(0), "cache clear");
  hc_cache* c = new hc_cache;
  std::memset(c, 0, sizeof *c);
  c->cfg = *cfg;
  c->g = make_geom(*cfg);
  std::memcpy(c->labels, labels_host, cfg->n_heads);
  std::memcpy(c->heads, P.heads, sizeof(HeadSlot) * cfg->n_heads);
  c->buf = static_cast<char*>(buf);
  c->bytes = bytes;
  c->used = P.bytes;
  c->off_items = P.off_items;
  c->off_sched = P.off_sched;
  c->off_split = P.off_split;
  c->off_k = P.off_k;
  c->off_v = P.off_v;
  c->off_part_o = P.off_part_o;
  c->off_part_ml = P.off_part_ml;
  c->n_items = (int)P.items.size();
  c->n_band = P.n_band;
  c->n_cta_main = P.sched_main.empty() ? 0 : (int)P.sched_main.size() - 1;
  c->n_cta_band = P.sched_band.empty() ? 0 : (int)P.sched_band.size() - 1;
  c->n_split = (int)P.splits.size();
  c->split_bytes = P.split_bytes;
  c->n_parts = P.n_parts;
  c->plan_span = P.span;
  c->plan_total = P.total;
  c->pg = P.pg;
  c->rows = P.rows;
  for (int a = 0; a < 4; ++a) {
    c->rows_by_arch[a] = P.rows_by_arch[a];
    c->n_by_arch[a] = P.n_by_arch[a];
  }
  c->newest = -1;
  c->valid_frames = 0;
  c->sink_present = false;
  *out = c;
  return HC_OK;
}

hc_status hc_cache_destroy(hc_cache* cache) {
  delete cache;
  return HC_OK;
}

static size_t kv_row_bytes(const hc_config& cfg) { return (size_t)cfg.head_dim * esize_of(cfg.dtype); }

hc_status hc_cache_get_info(const hc_cache* c, hc_cache_info* out) {
  if (!c || !out) return fail(HC_ERR_INVALID_ARG, "null argument");
  std::memset(out, 0, sizeof *out);
  out->newest_block = c->newest;
  out->valid_frames = c->valid_frames;
  out->sink_present = c->sink_present ? 1 : 0;
  for (int a = 0; a < 4; ++a) {
    out->n_by_archetype[a] = c->n_by_arch[a];
    out->rows_by_archetype[a] = c->rows_by_arch[a];
  }
  out->bytes = c->used;
  out->kv_bytes = 2 * (size_t)c->rows * kv_row_bytes(c->cfg);
  out->split_bytes = c->split_bytes;
  out->n_work_items = c->n_items;
  out->n_split_runs = c->n_split;
  out->n_split_pieces = c->n_parts;
  out->planned_span = c->plan_span;
  out->planned_total = c->plan_total;
  out->monolithic_bytes = (size_t)2 * c->g.Wf * c->g.F * c->g.H * c->g.d * esize_of(c->cfg.dtype);
  return HC_OK;
}

hc_status hc_cache_plan_info(const hc_config* cfg, const int8_t* labels_host, hc_cache_info* out) {
  hc_status s = hc_config_validate(cfg);
  if (s != HC_OK) return s;
  if ((s = check_labels(cfg, labels_host)) != HC_OK) return s;
  if (!out) return fail(HC_ERR_INVALID_ARG, "out is null");
  Plan P;
  plan_cache(*cfg, labels_host, P);
  if (!P.ok)
    return fail(HC_ERR_UNSUPPORTED, "the sliding Spatial window (%dx%d) is too wide for the band kernel", cfg->cell_h,
                cfg->cell_w);
  const Geom g = make_geom(*cfg);
  std::memset(out, 0, sizeof *out);
  out->newest_block = -1;
  for (int a = 0; a < 4; ++a) {
    out->n_by_archetype[a] = P.n_by_arch[a];
    out->rows_by_archetype[a] = P.rows_by_arch[a];
  }
  out->bytes = P.bytes;
  out->kv_bytes = 2 * (size_t)P.rows * kv_row_bytes(*cfg);
  out->split_bytes = P.split_bytes;
  out->n_work_items = (int32_t)P.items.size();
  out->n_split_runs = (int32_t)P.splits.size();
  out->n_split_pieces = P.n_parts;
  out->planned_span = P.span;
  out->planned_total = P.total;
  out->monolithic_bytes = (size_t)2 * g.Wf * g.F * g.H * g.d * esize_of(cfg->dtype);
  return HC_OK;
}

hc_status hc_cache_plan_items(const hc_config* cfg, const int8_t* labels_host, hc_work_item* items_host,
                              int32_t capacity, int32_t* n_items) {
  hc_status s = hc_config_validate(cfg);
  if (s != HC_OK) return s;
  if ((s = check_labels(cfg, labels_host)) != HC_OK) return s;
  if (!n_items) return fail(HC_ERR_INVALID_ARG, "n_items is null");
  Plan P;
  plan_cache(*cfg, labels_host, P);
  if (!P.ok)
    return fail(HC_ERR_UNSUPPORTED, "the sliding Spatial window (%dx%d) is too wide for the band kernel", cfg->cell_h,
                cfg->cell_w);
  static_assert(HC_ITEM_RANGE == hc::ITEM_RANGE && HC_ITEM_CELL == hc::ITEM_CELL && HC_ITEM_BAND == hc::ITEM_BAND &&
                    HC_ITEM_PATCH == hc::ITEM_PATCH,
                "item kinds");
  const Geom g = make_geom(*cfg);
  const int n = (int)P.items.size();
  *n_items = n;
  if (!items_host) return HC_OK;
  if (capacity < n) return fail(HC_ERR_SIZE, "the plan has %d items, capacity %d", n, capacity);
  const int n_main = n - P.n_band;
  for (int launch = 0; launch < 2; ++launch) {
    const std::vector<int32_t>& sched = launch == 0 ? P.sched_main : P.sched_band;
    const int base = launch == 0 ? 0 : n_main;
    for (int c = 0; c + 1 < (int)sched.size(); ++c)
      for (int i = sched[c]; i < sched[c + 1]; ++i) {
        const WorkItem& w = P.items[base + i];
        hc_work_item& o = items_host[base + i];
        std::memset(&o, 0, sizeof o);
        o.head = w.head;
        o.kind = w.kind;
        o.q0 = w.q0;
        o.nq = w.nq;
        o.k_row0 = w.k_row0;
        o.k_len = w.k_per_frame > 0 ? (int64_t)w.k_per_frame * g.Wf : w.k_len;
        o.cell = w.cell;
        o.chunk = w.chunk;
        o.n_chunks = w.n_chunks;
        o.part = w.part;
        o.launch = launch;
        o.cta = c;
      }
  }
  return HC_OK;
}

static hc::ScatterParams scatter_params(const hc_cache* c, const void* k, const void* v) {
  hc::ScatterParams p;
  std::memset(&p, 0, sizeof p);
  p.k_src = k;
  p.v_src = v;
  p.k_dst = c->buf + c->off_k;
  p.v_dst = c->buf + c->off_v;
  p.esize = (int)esize_of(c->cfg.dtype);
  p.g = c->g;
  std::memcpy(p.heads, c->heads, sizeof(HeadSlot) * c->g.H);
  return p;
}

hc_status hc_cache_restructure(hc_cache* c, const void* k_win, const void* v_win,
                               int64_t first_block_id, int32_t n_blocks, void* stream) {
  if (!c || !k_win || !v_win) return fail(HC_ERR_INVALID_ARG, "null argument");
  if (!aligned16(k_win) || !aligned16(v_win)) return fail(HC_ERR_ALIGN, "k_win/v_win not 16-byte aligned");
  const Geom& g = c->g;
  if (first_block_id < 0 || n_blocks < 1 || (int64_t)n_blocks * g.fpb > g.Wf)
    return fail(HC_ERR_SHAPE, "window of %d blocks from block %lld does not fit %d frames", n_blocks,
                (long long)first_block_id, g.Wf);
  if (first_block_id != 0 && (int64_t)n_blocks * g.fpb != g.Wf)
    return fail(HC_ERR_STATE, "a window that does not start at block 0 must be full");
  hc::ScatterParams p = scatter_params(c, k_win, v_win);
  p.src_frame0 = first_block_id * g.fpb;
  p.n_src_frames = n_blocks * g.fpb;
  p.dummy_frame0 = (first_block_id + n_blocks - 1) * g.fpb;
  HC_CUDA(hc::launch_scatter(p, static_cast<cudaStream_t>(stream)), "cache restructure");
  c->newest = first_block_id + n_blocks - 1;
  c->valid_frames = first_block_id == 0 ? n_blocks * g.fpb : g.Wf;
  c->sink_present = c->sink_present || first_block_id == 0;
  return HC_OK;
}

hc_status hc_cache_append(hc_cache* c, int64_t block_id, const void* k_blk, const void* v_blk,
                          void* stream) {
  if (!c || !k_blk || !v_blk) return fail(HC_ERR_INVALID_ARG, "null argument");
  if (!aligned16(k_blk) || !aligned16(v_blk)) return fail(HC_ERR_ALIGN, "k_blk/v_blk not 16-byte aligned");
  if (c->newest < 0 ? block_id != 0 : (block_id != c->newest && block_id != c->newest + 1))
    return fail(HC_ERR_STATE, "block %lld after newest %lld: must repeat it or follow it",
                (long long)block_id, (long long)c->newest);
  const Geom& g = c->g;
  hc::ScatterParams p = scatter_params(c, k_blk, v_blk);
  p.src_frame0 = block_id * g.fpb;
  p.n_src_frames = g.fpb;
  p.dummy_frame0 = block_id * g.fpb;
  HC_CUDA(hc::launch_scatter(p, static_cast<cudaStream_t>(stream)), "cache append");
  c->newest = block_id;
  const int64_t seen = (block_id + 1) * g.fpb;
  c->valid_frames = std::max<int64_t>(c->valid_frames, std::min<int64_t>(seen, g.Wf));
  if (block_id == 0) c->sink_present = true;
  return HC_OK;
}

// ------------------------------------------------------------ attention

hc_status hc_routed_attention(const hc_cache* c, const void* q, void* o, void* stream) {
  if (!c || !q || !o) return fail(HC_ERR_INVALID_ARG, "null argument");
  if (!aligned16(q) || !aligned16(o)) return fail(HC_ERR_ALIGN, "q/o not 16-byte aligned");
  if (c->newest < 0) return fail(HC_ERR_STATE, "cache holds no block yet");
  if (c->n_by_arch[HC_SINK] > 0 && !c->sink_present)
    return fail(HC_ERR_STATE, "Sink heads present but block 0 was never written");
  int* status = nullptr;
  hc_status s = status_ptr(&status);
  if (s != HC_OK) return s;
  hc::AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.k = c->buf + c->off_k;
  p.v = c->buf + c->off_v;
  p.o = o;
  p.k_stride = c->g.d;
  p.k_hstride = 0;
  p.nq_total = c->g.blk;
  p.out_fp32 = c->cfg.dtype == HC_FP32;
  p.item_mode = hc::ITEMS_LIST;
  p.n_items = c->n_items;
  p.items = reinterpret_cast<const WorkItem*>(c->buf + c->off_items);
  p.valid_frames = c->valid_frames;
  p.g = c->g;
  p.status = status;
  if (c->cfg.dtype == HC_BF16) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const hc::TcKV kv{c->buf + c->off_k, c->buf + c->off_v, 1, c->rows};
    const int32_t* sched = reinterpret_cast<const int32_t*>(c->buf + c->off_sched);
    const int n_main = c->n_items - c->n_band;
    p.part_o = reinterpret_cast<float*>(c->buf + c->off_part_o);
    p.part_ml = reinterpret_cast<float*>(c->buf + c->off_part_ml);
    if (n_main > 0) {
      p.n_items = n_main;
      p.sched = sched;
      HC_CUDA(hc::launch_attention_tc(p, kv, c->n_cta_main, st), "routed attention");
    }
    if (c->n_band > 0) {
      // Sliding Spatial heads: the masked band variant over the list's tail.
      p.items += n_main;
      p.n_items = c->n_band;
      p.sched = sched + hc::kMaxCtas + 1;
      p.band_win = hc::WIN_SLIDING;
      p.pg = c->pg;
      HC_CUDA(hc::launch_attention_tc(p, kv, c->n_cta_band, st), "routed attention (sliding Spatial)");
    }
    if (c->n_split > 0) {
      // Merge the split key runs' partial outputs.
      hc::CombineParams m;
      std::memset(&m, 0, sizeof m);
      m.items = reinterpret_cast<const SplitItem*>(c->buf + c->off_split);
      m.n_items = c->n_split;
      m.out_fp32 = 0;
      m.part_o = p.part_o;
      m.part_ml = p.part_ml;
      m.o = o;
      m.g = c->g;
      HC_CUDA(hc::launch_combine(m, st), "routed attention (split-run merge)");
    }
  } else {
    p.band_win = hc::WIN_SLIDING;
    HC_CUDA(hc::launch_attention(p, c->cfg.dtype, dim3(c->n_items, 1, 1), static_cast<cudaStream_t>(stream)),
            "routed attention");
  }
  return HC_OK;
}

hc_status hc_full_attention(const hc_config* cfg, const void* q, const void* k, const void* v,
                            int32_t n_q_tokens, int32_t n_key_frames, void* o, void* stream) {
  hc_status s = hc_config_validate(cfg);
  if (s != HC_OK) return s;
  if (n_q_tokens == 0) return HC_OK;   // nothing to compute; q and o may be null
  if (!q || !k || !v || !o) return fail(HC_ERR_INVALID_ARG, "null argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(HC_ERR_ALIGN, "device pointers must be 16-byte aligned");
  if (n_q_tokens < 0 || n_key_frames < 1 || n_key_frames > 4096)
    return fail(HC_ERR_SHAPE, "n_q_tokens %d / n_key_frames %d", n_q_tokens, n_key_frames);
  const Geom g = make_geom(*cfg);
  const int64_t nk = (int64_t)n_key_frames * g.F;
  if (nk >= (1ll << 31)) return fail(HC_ERR_SHAPE, "too many keys");
  int* status = nullptr;
  if ((s = status_ptr(&status)) != HC_OK) return s;
  const int BM = hc::attention_block_rows(cfg->dtype, cfg->head_dim);
  hc::AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.k_stride = (int64_t)g.H * g.d;
  p.k_hstride = g.d;
  p.nq_total = n_q_tokens;
  p.out_fp32 = cfg->dtype == HC_FP32;
  p.item_mode = hc::ITEMS_DENSE;
  p.plane_k0[0] = 0;
  p.plane_klen[0] = (int32_t)nk;
  p.g = g;
  p.status = status;
  const dim3 grid((n_q_tokens + BM - 1) / BM, g.H, 1);
  p.n_planes = 1;
  if (cfg->dtype == HC_BF16) {
    const hc::TcKV kv{k, v, g.H, nk};
    p.n_items = (int)(grid.x * grid.y);
    HC_CUDA(hc::launch_attention_tc(p, kv, std::min(p.n_items, hc::device_sm_count()),
                                    static_cast<cudaStream_t>(stream)),
            "full attention");
  } else {
    HC_CUDA(hc::launch_attention(p, cfg->dtype, grid, static_cast<cudaStream_t>(stream)), "full attention");
  }
  return HC_OK;
}

hc_status hc_full_attention_ws_bytes(const hc_config* cfg, int32_t n_q_tokens, int32_t n_key_frames,
                                     size_t* bytes) {
  hc_status s = hc_config_validate(cfg);
  if (s != HC_OK) return s;
  if (!bytes) return fail(HC_ERR_INVALID_ARG, "bytes is null");
  if (n_q_tokens < 0 || n_key_frames < 1 || n_key_frames > 4096)
    return fail(HC_ERR_SHAPE, "n_q_tokens %d / n_key_frames %d", n_q_tokens, n_key_frames);
  *bytes = cfg->dtype == HC_BF16 && n_q_tokens > 0 ? full_plan(*cfg, n_q_tokens, n_key_frames)->bytes : 0;
  return HC_OK;
}

hc_status hc_full_attention_ws(const hc_config* cfg, const void* q, const void* k, const void* v,
                               int32_t n_q_tokens, int32_t n_key_frames, void* o, void* scratch,
                               size_t scratch_bytes, void* stream) {
  hc_status s = hc_config_validate(cfg);
  if (s != HC_OK) return s;
  if (cfg->dtype != HC_BF16 || n_q_tokens == 0)
    return hc_full_attention(cfg, q, k, v, n_q_tokens, n_key_frames, o, stream);
  if (!q || !k || !v || !o || !scratch) return fail(HC_ERR_INVALID_ARG, "null argument");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(scratch))
    return fail(HC_ERR_ALIGN, "device pointers must be 16-byte aligned");
  if (n_q_tokens < 0 || n_key_frames < 1 || n_key_frames > 4096)
    return fail(HC_ERR_SHAPE, "n_q_tokens %d / n_key_frames %d", n_q_tokens, n_key_frames);
  const Geom g = make_geom(*cfg);
  const int64_t nk = (int64_t)n_key_frames * g.F;
  if (nk >= (1ll << 31)) return fail(HC_ERR_SHAPE, "too many keys");
  const std::shared_ptr<const FullPlan> P = full_plan(*cfg, n_q_tokens, n_key_frames);
  if (scratch_bytes < P->bytes)
    return fail(HC_ERR_INVALID_ARG, "scratch_bytes %zu < %zu (hc_full_attention_ws_bytes)", scratch_bytes, P->bytes);
  int* status = nullptr;
  if ((s = status_ptr(&status)) != HC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(scratch);
  // The plan into the workspace (a few tens of KB; the host copies live in
  // the plan cache).
  HC_CUDA(cudaMemcpyAsync(ws + P->off_items, P->items.data(), P->items.size() * sizeof(WorkItem),
                          cudaMemcpyHostToDevice, st),
          "full attention work list upload");
  HC_CUDA(cudaMemcpyAsync(ws + P->off_sched, P->sched.data(), P->sched.size() * sizeof(int32_t),
                          cudaMemcpyHostToDevice, st),
          "full attention schedule upload");
  if (!P->splits.empty())
    HC_CUDA(cudaMemcpyAsync(ws + P->off_split, P->splits.data(), P->splits.size() * sizeof(SplitItem),
                            cudaMemcpyHostToDevice, st),
            "full attention split table upload");
  hc::AttnParams p;
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.k_stride = (int64_t)g.H * g.d;
  p.k_hstride = g.d;
  p.nq_total = n_q_tokens;
  p.out_fp32 = 0;
  p.item_mode = hc::ITEMS_LIST;
  p.items = reinterpret_cast<const WorkItem*>(ws + P->off_items);
  p.n_items = (int)P->items.size();
  p.sched = reinterpret_cast<const int32_t*>(ws + P->off_sched);
  p.part_o = reinterpret_cast<float*>(ws + P->off_part_o);
  p.part_ml = reinterpret_cast<float*>(ws + P->off_part_ml);
  p.valid_frames = n_key_frames;
  p.g = g;
  p.status = status;
  const hc::TcKV kv{k, v, g.H, nk};
  HC_CUDA(hc::launch_attention_tc(p, kv, (int)P->sched.size() - 1, st), "full attention");
  if (!P->splits.empty()) {
    hc::CombineParams m;
    std::memset(&m, 0, sizeof m);
    m.items = reinterpret_cast<const SplitItem*>(ws + P->off_split);
    m.n_items = (int)P->splits.size();
    m.out_fp32 = 0;
    m.part_o = p.part_o;
    m.part_ml = p.part_ml;
    m.o = o;
    m.g = g;
    HC_CUDA(hc::launch_combine(m, st), "full attention (split-run merge)");
  }
  return HC_OK;
}

hc_status hc_debug_inject_stall(int32_t enable) {
  g_debug_stall.store(enable != 0 ? 1 : 0);
  return HC_OK;
}

hc_status hc_get_last_error(void* stream) {
  HC_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream synchronize");
  int word = 0, zero = 0;
  HC_CUDA(cudaMemcpyFromSymbol(&word, g_hc_status_word, sizeof word), "status read");
  HC_CUDA(cudaMemcpyToSymbol(g_hc_status_word, &zero, sizeof zero), "status clear");
  if (word == hc::DEV_OK) return HC_OK;
  if (word == hc::DEV_TIMEOUT) return fail(HC_ERR_TIMEOUT, "a bounded device wait expired");
  return fail(HC_ERR_CUDA, "device status word %d", word);
}

}  // extern "C"
