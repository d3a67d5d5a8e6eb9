/*
 * headcast.h -- C ABI of the head-routed attention library (libheadcast.so).
 *
 * What it computes.  HeadCast ("HeadCast: Casting Attention Heads for
 * Efficient Autoregressive Video Generation"; method as restated in the Pith
 * review of that paper, sections "The pith", "Core claim", "What carries the
 * argument", "Referee Report" major comment 2, "Axiom & Free-Parameter
 * Ledger" and the Figure 2 / Figure 3 captions) types every attention head of
 * an autoregressive video diffusion transformer once, when the sliding window
 * of cached frames first fills, as Sink, Dummy, Spatial or Global, by the
 * cosine similarity between the head's full-context attention output and the
 * outputs over three restricted key sets.  The monolithic KV cache is then
 * split along the head dimension into per-archetype buffers and every head
 * attends only over its own pathway:
 *   Sink     the stream's first block (kept forever),
 *   Dummy    the newest block,
 *   Spatial  its own cell of a non-overlapping 10x10 partition of every
 *            cached frame,
 *   Global   the whole sliding window.
 *
 * Conventions shared by every call.
 *  - Tokens.  A frame is a frame_h x frame_w grid of F tokens; a block is
 *    frames_per_block frames; the window holds window_frames frames and
 *    includes the current block.  Inside a run of frames the token index is
 *    t = f*F + h*frame_w + w (frame-major raster order, oldest frame first).
 *  - Tensors.  Q, K, V and O are row-major [tokens][n_heads][head_dim]
 *    ("BSHD" with batch 1), contiguous, in the config's dtype (bf16 or fp32).
 *    Device pointers must be 16-byte aligned.
 *  - Pointers.  Every pointer is a DEVICE pointer unless its name ends in
 *    _host.  The caller owns every buffer; the library never allocates device
 *    memory.  Handles (hc_cache) are host objects owned by the library.
 *  - Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Calls are asynchronous on it unless marked SYNC.
 *  - Errors.  Arguments are validated on the host before anything is
 *    launched; a failed validation changes nothing and returns the status.
 *    A launch failure returns HC_ERR_CUDA.  Device-side failures never trap:
 *    they set a device status word that hc_get_last_error reports.
 *    hc_last_error_message() describes the most recent failure on the
 *    calling thread.
 *  - Thread safety.  Distinct handles may be used from distinct threads.  A
 *    handle must not be used on two streams at once.
 *  - Devices.  The library keeps a few per-device facts once it has seen a
 *    device (the addresses of its device-side status word and static
 *    workspace, kernel attributes, the SM count).  cudaDeviceReset, or any
 *    other way of replacing a device's primary context, while the library is
 *    in use is not supported: those cached addresses would then be stale.
 */
#ifndef HEADCAST_H
#define HEADCAST_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HC_ABI_VERSION 7
#define HC_MAX_HEADS 64

typedef enum { HC_SINK = 0, HC_DUMMY = 1, HC_SPATIAL = 2, HC_GLOBAL = 3 } hc_archetype;

typedef enum {
  HC_OK = 0,
  HC_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, negative size        */
  HC_ERR_SHAPE = 2,         /* unsupported or inconsistent shape            */
  HC_ERR_DTYPE = 3,         /* dtype not supported by this call             */
  HC_ERR_ALIGN = 4,         /* pointer not 16-byte aligned                  */
  HC_ERR_STATE = 5,         /* call not valid in the handle's current state */
  HC_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed         */
  HC_ERR_TIMEOUT = 7,       /* a bounded device-side wait expired           */
  HC_ERR_UNSUPPORTED = 8,   /* feature not built / no suitable device       */
  HC_ERR_SIZE = 9           /* caller buffer smaller than required          */
} hc_status;

typedef enum { HC_BF16 = 0, HC_FP32 = 1 } hc_dtype;

/* Layer geometry and the classifier's constants.  hc_config_default fills
 * the constants with the values the paper's free-parameter ledger gives
 * (theta 0.95 for all three cosine gates, spatial score threshold 0.755,
 * MSE weight gamma 5, proxy radius r = 2, deployed cell 10x10) and leaves
 * the shape fields for the caller. */
typedef struct {
  int32_t n_heads;          /* H, 1..HC_MAX_HEADS                             */
  int32_t head_dim;         /* d, 64 or 128                                   */
  int32_t frame_h;          /* token rows per frame                           */
  int32_t frame_w;          /* token columns per frame                        */
  int32_t frames_per_block; /* frames per AR block (3)                        */
  int32_t window_frames;    /* frames in the sliding window, a multiple of
                               frames_per_block, current block included       */
  int32_t dtype;            /* hc_dtype of Q, K, V and O                       */
  float softmax_scale;      /* 0 => 1/sqrt(head_dim)                          */
  float theta_sink;         /* Sink gate on the mean cosine (0.95)            */
  float theta_dummy;        /* Dummy gate (0.95)                              */
  float theta_spatial;      /* Spatial gate on the mean cosine (0.95)         */
  float theta_score;        /* Spatial gate on P5 - gamma*MSE (0.755)         */
  float gamma;              /* MSE penalty weight (5)                         */
  int32_t proxy_radius;     /* r of the (2r+1)x(2r+1) classification proxy   */
  int32_t cell_h;           /* deployed Spatial cell height (10)              */
  int32_t cell_w;           /* deployed Spatial cell width (10)               */
  int32_t proxy_mode;       /* Spatial proxy of the classifier:
                               HC_PROXY_NEIGHBOURHOOD (0, the paper's) = the
                               clipped (2r+1)x(2r+1) neighbourhood of the query;
                               HC_PROXY_CELL (1) = the query's deployed cell
                               (compares the proxy with the deployed path)    */
  int32_t spatial_mode;     /* deployed Spatial key set:
                               HC_SPATIAL_CELLS (0, default) = the query's own
                               non-overlapping cell_h x cell_w cell;
                               HC_SPATIAL_SLIDING (1) = the cell_h x cell_w
                               window centred on the query (rows
                               h - cell_h/2 .. h + cell_h - cell_h/2 - 1,
                               columns likewise, clipped), in every frame     */
} hc_config;

typedef enum { HC_SPATIAL_CELLS = 0, HC_SPATIAL_SLIDING = 1 } hc_spatial_mode;

typedef enum { HC_PROXY_NEIGHBOURHOOD = 0, HC_PROXY_CELL = 1 } hc_proxy_mode;

typedef struct hc_cache hc_cache;   /* opaque host handle, one per layer */

/* Summary of a cache handle (host-side bookkeeping, no device access). */
typedef struct {
  int64_t newest_block;     /* id of the newest block, -1 before any data     */
  int32_t valid_frames;     /* filled ring slots (<= window_frames)           */
  int32_t sink_present;     /* 1 once block 0 has been written                */
  int32_t n_by_archetype[4];/* heads per archetype                            */
  int64_t rows_by_archetype[4]; /* K rows reserved per archetype (V the same) */
  size_t bytes;             /* bytes of the backing store actually used       */
  size_t kv_bytes;          /* of which the per-archetype K and V regions     */
  size_t split_bytes;       /* of which the routed launch's workspace for key
                               runs split across CTAs (0 if none is split)    */
  size_t monolithic_bytes;  /* bytes a [window][H][d] K+V cache would take    */
  int32_t n_work_items;     /* work items of the routed launch(es)            */
  int32_t n_split_runs;     /* key runs split across CTAs and merged after    */
  int32_t n_split_pieces;   /* pieces of those runs                           */
  int32_t pad_;
  int64_t planned_span;     /* the schedule's busiest CTA, in key-tile steps
                               (an item boundary counts as 6) with the window
                               full; the band launch's added for sliding heads */
  int64_t planned_total;    /* the same summed over all CTAs                   */
} hc_cache_info;

/* Kinds of routed work items. */
typedef enum {
  HC_ITEM_RANGE = 0,   /* queries q0 .. q0+nq-1 of the block (block-local
                          tokens) against one contiguous key run: Sink,
                          Dummy and Global heads                            */
  HC_ITEM_CELL = 1,    /* query ordinals q0 .. q0+nq-1 of one deployed cell
                          (its 3-frame query set in frame, row, column order)
                          against the cell's key run: Spatial heads         */
  HC_ITEM_BAND = 3,    /* sliding Spatial, fp32 layers: queries q0 .. q0+nq-1
                          inside one frame, keys the band of window rows    */
  HC_ITEM_PATCH = 4    /* sliding Spatial, bf16 layers: patch `cell` of query
                          positions in every frame of the block (nq = 0: the
                          patch geometry fixes its queries)                 */
} hc_item_kind;

/* One work item of a routed launch as the planner deals it (host-side view
 * of the list hc_cache_create writes into the backing store). */
typedef struct {
  int32_t head;             /* head whose queries the item covers             */
  int32_t kind;             /* hc_item_kind                                   */
  int32_t q0, nq;           /* its queries (see hc_item_kind)                 */
  int64_t k_row0;           /* first K (and V) row of its key run, counted in
                               rows of the cache's per-archetype regions       */
  int64_t k_len;            /* rows of the whole run with the window full
                               (BAND, PATCH: the head's ring, of which the
                               item reads its queries' windows)                */
  int32_t cell;             /* CELL: ci * n_cells_w + cj, with
                               n_cells_w = max(1, floor(frame_w/cell_w + 1/2))
                               cells across a frame; PATCH: patch index        */
  int32_t chunk, n_chunks;  /* a key run split across CTAs: this item runs key
                               tiles [chunk*T/n_chunks, (chunk+1)*T/n_chunks)
                               of the run's T tiles of 128 keys; n_chunks = 1:
                               the whole run                                   */
  int32_t part;             /* partial-output slot of a split run's piece, -1
                               for an item that writes its output directly     */
  int32_t launch;           /* 0: the main launch; 1: the band launch of the
                               sliding Spatial heads                           */
  int32_t cta;              /* the CTA of that launch the schedule gives it    */
} hc_work_item;

/* ----------------------------------------------------------------------- */

int32_t hc_abi_version(void);
const char* hc_status_string(hc_status s);
/* Text of the most recent failure on the calling thread ("" if none). */
const char* hc_last_error_message(void);

/* Fill *out with the ledger constants; shape fields are zeroed, except
 * frames_per_block = 3, window_frames = 21, dtype = HC_BF16. */
hc_status hc_config_default(hc_config* out);
/* Check a config: H in 1..64, d in {64,128}, frame dims >= 1, window a
 * positive multiple of frames_per_block, finite thresholds, proxy_mode and
 * spatial_mode 0/1. */
hc_status hc_config_validate(const hc_config* cfg);

/* ---------------------------------------------------------------------------
 * Classification.  At the block where the window first fills (maximum-noise
 * step), each head's full-context output O_full is compared with its output
 * over (a) the window's first block (Sink proxy), (b) the window's last
 * block (Dummy proxy), (c) the (2r+1)x(2r+1) clipped neighbourhood of the
 * query's (h, w) in every window frame (Spatial proxy; with proxy_mode =
 * HC_PROXY_CELL, the query's deployed cell instead).  Per head:
 *   c_x   = mean over the block's queries of cos(O_full, O_x),
 *   P5    = 5th percentile of cos(O_full, O_spatial) (linear interpolation
 *           at rank 0.05*(Nq-1)),
 *   MSE   = mean over queries and channels of (O_spatial - O_full)^2,
 *   score = P5 - gamma*MSE,
 *   label = Sink if c_sink >= theta_sink, else Dummy if c_dummy >=
 *           theta_dummy, else Spatial if c_spatial >= theta_spatial and
 *           score >= theta_score, else Global.
 * [Pith review, "What carries the argument"; Ledger: theta, theta_sc,
 *  gamma, r; major comment 2 for the proxy shape.]
 *
 * q        [3F][H][d]  the current block's queries.
 * k, v     [n_key_frames*F][H][d]  the window, oldest frame first; its first
 *          block is block 0 of the stream, its last block the current one.
 * n_key_frames  a multiple of frames_per_block, >= 2 blocks.
 * labels_dev    int8 [H] out (device), required.
 * labels_host   int8 [H] out (host), nullable; if set the call is SYNC on
 *               `stream` (it copies the labels back and waits).
 * stats_dev     float [H][6] out (device), nullable: c_sink, c_dummy,
 *               c_spatial, P5, MSE, score.
 * o_full        [3F][H][d] out (device), nullable: the full-context output.
 * scratch       device workspace of at least hc_classify_scratch_bytes(),
 *               16-byte aligned, owned by the caller, contents undefined
 *               after the call.
 * If a bounded device-side wait expires in one of the call's kernels (or the
 * status word was already set when they ran), no label is decided:
 * labels_dev holds -1 for every head, and with labels_host the call returns
 * HC_ERR_TIMEOUT (the status word stays set for hc_get_last_error).
 * ------------------------------------------------------------------------- */
hc_status hc_classify_scratch_bytes(const hc_config* cfg, int32_t n_key_frames, size_t* bytes);
hc_status hc_classify(const hc_config* cfg, const void* q, const void* k, const void* v,
                      int32_t n_key_frames, int8_t* labels_dev, int8_t* labels_host,
                      float* stats_dev, void* o_full, void* scratch, size_t scratch_bytes,
                      void* stream);

/* ---------------------------------------------------------------------------
 * Classification with a library-held workspace.  The paper has no
 * counterpart to this call: it exists for callers that cannot allocate
 * device memory (for instance a plugin whose host framework owns all device
 * memory, or a real-time loop that allows no allocation after start-up).
 * It computes exactly what hc_classify computes, with the same arguments
 * except the workspace, which here is a fixed array of
 * HC_STATIC_SCRATCH_BYTES in the library's device image.  Every GPU that
 * loads the library holds that array until the process exits.  The call
 * itself allocates nothing (no cudaMalloc, no allocating library routine).
 *  - HC_ERR_SIZE if the layer's workspace (hc_classify_scratch_bytes) is
 *    larger than HC_STATIC_SCRATCH_BYTES; nothing is launched.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - All calls share the array and it keeps the last call's contents
 *    (nothing in it needs clearing between calls).  Calls whose kernels may
 *    overlap on the GPU (different streams or threads) race on it and must
 *    be serialised by the caller.
 * ------------------------------------------------------------------------- */
#define HC_STATIC_SCRATCH_BYTES (16u << 20)
hc_status hc_classify_static_scratch(const hc_config* cfg, const void* q, const void* k,
                                     const void* v, int32_t n_key_frames, int8_t* labels_dev,
                                     int8_t* labels_host, float* stats_dev, void* o_full,
                                     void* stream);

/* ---------------------------------------------------------------------------
 * Restructured cache.  The monolithic [window][H][d] K/V cache is replaced
 * by per-head regions in one caller-owned device buffer:
 *   Sink head     one block (3F rows): block 0 of the stream, fixed;
 *   Dummy head    one block: the newest block, overwritten in place;
 *   Spatial head  window_frames*F rows: a ring of frame slots (frame a lives
 *                 in slot a mod window_frames), stored cell-major: all slots
 *                 of one cell are contiguous, so a cell's keys across the
 *                 window form one run of rows (with HC_SPATIAL_SLIDING, in
 *                 raster order like a Global head);
 *   Global head   window_frames*F rows: the same ring in raster order.
 * K rows of all heads form one [rows][d] area, V rows a second one.
 * [Pith review, "What carries the argument" (split along the head
 *  dimension; Sink and Dummy keep a single block, Global the full window,
 *  Spatial the full history in time partitioned by cell); Figure 2 phase 3.]
 *
 * hc_cache_bytes     bytes the buffer needs for these labels (HOST only).
 * hc_cache_create    binds a handle to `buf` (device, >= hc_cache_bytes,
 *                    256-byte aligned), writes the work list into it and
 *                    clears its K/V areas (SYNC: waits for the clear).  The
 *                    caller keeps ownership of buf and must keep it alive
 *                    until hc_cache_destroy.
 * hc_cache_destroy   frees the handle only, never buf.
 * ------------------------------------------------------------------------- */
hc_status hc_cache_bytes(const hc_config* cfg, const int8_t* labels_host, size_t* bytes);
hc_status hc_cache_create(const hc_config* cfg, const int8_t* labels_host, void* buf,
                          size_t bytes, hc_cache** out);
hc_status hc_cache_destroy(hc_cache* cache);
hc_status hc_cache_get_info(const hc_cache* cache, hc_cache_info* out);
/* The same summary for a cache not yet created (HOST only, no device
 * access): what hc_cache_create would reserve for these labels.  The
 * steady-state memory comparison of the restructured cache with the
 * monolithic one [Pith review, Figure 9 caption / Appendix C]. */
hc_status hc_cache_plan_info(const hc_config* cfg, const int8_t* labels_host, hc_cache_info* out);
/* The routed work list hc_cache_create would write for these labels (HOST
 * only, no device access), in launch order: the main launch's items CTA by
 * CTA (each CTA's in the order it runs them), then the band launch's.  The
 * schedule deals items longest first, each to the least loaded of 148 CTAs,
 * after cutting the longest key runs where that shortens the busiest CTA.
 * items_host  [capacity] hc_work_item, or null to ask only for the count.
 * *n_items    set to the list's length in either case.
 * HC_ERR_SIZE if items_host is given and capacity < *n_items (nothing is
 * written to items_host then). */
hc_status hc_cache_plan_items(const hc_config* cfg, const int8_t* labels_host, hc_work_item* items_host,
                              int32_t capacity, int32_t* n_items);

/* Fill the per-archetype regions from a monolithic window.
 * k_win, v_win  [n_blocks*3F][H][d] holding blocks first_block_id ..
 *               first_block_id+n_blocks-1, oldest first.
 * Requires first_block_id == 0 (the window holds the Sink block) or a full
 * window (n_blocks*frames_per_block == window_frames); n_blocks*fpb <=
 * window_frames.  Resets the handle's state to this window.  Async. */
hc_status hc_cache_restructure(hc_cache* cache, const void* k_win, const void* v_win,
                               int64_t first_block_id, int32_t n_blocks, void* stream);

/* Write one block's K/V ([3F][H][d]) for the current denoising step.
 * block_id == newest      overwrite the newest block (a later denoising step);
 * block_id == newest + 1  advance: the block's frames replace the oldest ring
 *                         slots (eviction), Dummy buffers are overwritten;
 * block 0 is also written to the Sink heads.  Any other id: HC_ERR_STATE.
 * One fused launch for all heads.  Async.  [Figure 2 phase 3.] */
hc_status hc_cache_append(hc_cache* cache, int64_t block_id, const void* k_blk,
                          const void* v_blk, void* stream);

/* ---------------------------------------------------------------------------
 * Routed attention: every head over its own pathway, one launch.
 * q, o  [3F][H][d] the current block's queries / outputs.
 * softmax(q k^T * scale) v over: Sink -> block 0; Dummy -> newest block;
 * Spatial -> the query's cell in every filled ring slot (HC_SPATIAL_SLIDING:
 * the window centred on the query); Global -> every filled ring slot.  No
 * mask inside a block.  Async: one persistent launch over all heads and
 * pathways (plus one for sliding Spatial heads, and a light merge launch
 * when the plan splits long key runs across CTAs).  A handle's launches
 * share its split workspace, so one handle's calls must not overlap.
 * [Pith review, "The pith", "Core claim", Figure 3 caption.]
 * ------------------------------------------------------------------------- */
hc_status hc_routed_attention(const hc_cache* cache, const void* q, void* o, void* stream);

/* Full attention of every head over [n_key_frames*F] monolithic keys: the
 * comparison path (and the warm-up path before classification).
 * q, o [Nq][H][d] with Nq = n_q_tokens; k, v [n_key_frames*F][H][d].  Async.
 * n_q_tokens = 0 is a no-op (the pointers may then be null). */
hc_status hc_full_attention(const hc_config* cfg, const void* q, const void* k, const void* v,
                            int32_t n_q_tokens, int32_t n_key_frames, void* o, void* stream);

/* Full attention with a caller-owned workspace, for bf16 layers: the work is
 * planned like the routed launch -- 256-query items of every head over the
 * whole key window, dealt longest-first to the CTAs, with as many key runs
 * split across CTAs (and merged by a light second launch) as evens out the
 * CTAs -- instead of a plain strided assignment.  Plans are kept per shape
 * on the host and copied into the workspace at each call (a few tens of KB).
 * fp32 layers run as hc_full_attention (the workspace is then unused and may
 * be null).  Calls sharing a workspace must not overlap.  Async.
 * scratch  device workspace of at least hc_full_attention_ws_bytes() bytes,
 *          16-byte aligned, owned by the caller, contents undefined after the
 *          call; HC_ERR_INVALID_ARG if smaller. */
hc_status hc_full_attention_ws_bytes(const hc_config* cfg, int32_t n_q_tokens, int32_t n_key_frames,
                                     size_t* bytes);
hc_status hc_full_attention_ws(const hc_config* cfg, const void* q, const void* k, const void* v,
                               int32_t n_q_tokens, int32_t n_key_frames, void* o, void* scratch,
                               size_t scratch_bytes, void* stream);

/* Test hook for the failure path (no counterpart in the paper).  While
 * enabled (enable != 0), every tensor-core attention launch (routed, full
 * and classification attention) runs with its K/V producer stopping after
 * the first key tile and every device-side wait limited to 2 ms: the CTAs'
 * bounded waits expire, each CTA drains its own copies and MMAs, frees its
 * tensor memory and returns, and the launch leaves HC_ERR_TIMEOUT in the
 * device status word (read by hc_get_last_error).  Outputs of such launches
 * are undefined.  Process-wide; off by default; never faults or hangs. */
hc_status hc_debug_inject_stall(int32_t enable);

/* SYNC on `stream`: waits for it, returns and clears the device status word
 * (HC_OK, HC_ERR_TIMEOUT for an expired bounded wait, HC_ERR_CUDA for a
 * device-side bounds check).  A CUDA error in the wait is HC_ERR_CUDA. */
hc_status hc_get_last_error(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* HEADCAST_H */
