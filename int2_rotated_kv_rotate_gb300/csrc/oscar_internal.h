// Internal layout shared by the host side (oscar_host.cpp) and the kernels (*.cu).
// Plain structs only; the C ABI is include/oscar.h.
#pragma once

#include <cstddef>
#include <cstdint>

#include "oscar.h"

namespace oscar {

constexpr int kHeadDim = 128;
constexpr int kPage = 64;
constexpr int kRowBytes = kHeadDim / 4;  // 32 B of 2-bit codes per token
constexpr int kMaxWindow = 1024;

// One request of an append plan (same for every layer).
struct AppendReq {
  int slot;        // request slot
  int L0, H0;      // length and history end before the append
  int L1, H1;      // after
  int x_offset;    // first row of this request in k_new / v_new
};

// One work item of the append kernel.  kind 0: ring slots [begin, begin+count) of the
// request (evict old occupant to INT2, then write new occupant); kind 1: new positions
// [begin, begin+count) that go to sinks or directly to INT2.
struct AppendItem {
  int req;    // index into AppendReq array
  int kind;
  int begin;
  int count;
};

// One request of a decode plan.
struct DecodeReq {
  int slot;
  int L, H;          // length, history end (INT2 format); H = L for BF16 format
  int H_pre;         // history end (BF16 format: length) before this step's append: no
                     // kernel of the step writes the INT2 pages wholly below it (the BF16
                     // rows below it), so they may be copied before the wait on the
                     // preceding kernel
  int app_expect;    // fused append + decode: append tasks of this request per kv-head (K and
                     // V, times append_task_split, per append item); 0 = nothing to wait for
  int first_item;    // items of this request, kv-head-major: first_item + kvh*items_per_head ..
  int items_per_head;
};

// One split-K work item: pages [p0, p1) of the INT2 history (kind 0) or BF16 tokens
// [t0, t1) of the sink+ring list (kind 1; index < S is sink j, else ring position H + j - S)
// of request `req` (plan index), kv-head `kvh`.  Partial results go to partial slot
// `slot`; the last CTA to finish an item of (req, kvh) merges the head_count slots from
// head_first.  A plan stores its items in the order CTAs take them: the items that wait
// on no append task first, largest first.
struct DecodeItem {
  int req;
  int kvh;
  int kind;
  int begin;
  int end;
  int head_first;  // first partial slot of this (req, kvh)
  int head_count;  // number of partial slots of this (req, kvh)
  int dep;         // fused append + decode: what the item reads that this launch's append tasks
                   // write (kDepNone, kDepRing: BF16 rows of new tokens, kDepPages: INT2 pages
                   // that receive evicted or new tokens)
  int split;       // BF16 items: list index from which rows may be written by this step's
                   // append (rows before it may be copied before the wait); INT2 items: end
  int slot;        // partial slot: the item's index in the plan's (request, kv-head) order
};
constexpr int kDepNone = 0, kDepRing = 1, kDepPages = 2;

#ifdef __CUDACC__
#define OSCAR_HOST_DEVICE __host__ __device__
#else
#define OSCAR_HOST_DEVICE
#endif
// Warps of a split-kernel CTA: 16 for one-wave plans at GQA 4 ("wide"), else 8.
OSCAR_HOST_DEVICE constexpr int decode_warps(int gqa, bool wide) { return gqa == 4 && wide ? 16 : 8; }
// Fused append + decode: CTAs per append item and kv-head and K|V (a CTA of nw warps
// covers nw tokens of the item's 16).
OSCAR_HOST_DEVICE constexpr int append_task_split(int nw) { return 16 / nw; }

struct DeviceLayout {
  // pools (byte offsets in the device block)
  size_t codes, sz, sink, ring, bf16_pages;
  size_t codes_layer_stride, codes_page_stride, codes_head_stride;  // K at +0, V at +half
  size_t sz_layer_stride, sz_page_stride, sz_head_stride;
  size_t sink_slot_stride, sink_layer_stride, sink_head_stride;
  size_t ring_slot_stride, ring_layer_stride, ring_head_stride;
  size_t bf16_layer_stride, bf16_page_stride, bf16_head_stride;
  // params
  size_t R_K, R_V, R_Vt, clip_K, clip_V;  // fp32 [layer][H_kv][d][d] (R_Vt = R_V transposed), [layer][H_kv]
  // control
  size_t page_table;  // int32 [max_requests][max_pages_per_request]
  size_t status;      // uint32 flags
  size_t counters;    // uint32 [max_requests][H_kv] merge counters (items of a head done)
  // the append and the decode plan, each one block that one copy uploads: int32 counts[4]
  // at +0, the requests at +256, the items after them.  Append counts: items.  Decode
  // counts: items, requests, items that wait on no append task (stored first).
  size_t append_plan, append_counts, append_reqs, append_items;
  size_t decode_plan, decode_counts, decode_reqs, decode_items;
  size_t sched;         // uint32 [4]: dynamic work counter, CTA exit counter (self-resetting)
  size_t app_done;      // uint32 [layer][max_requests][H_kv][2]: append tasks of the running fused
                        // launch that have stored their sink and ring rows ([0]) and their INT2
                        // rows ([1]); the request's final merge takes the launch's count off again
  size_t max_append_items, max_decode_items;
  size_t total;
};

// Everything a kernel needs, passed by value.
struct KernelParams {
  uint8_t* base;
  int n_q_heads, n_kv_heads, gqa, group, n_sink, window, n_layers;
  int max_requests, max_pages, max_pages_per_request;
  uint32_t counter_polls;  // bounded waits on append-dependency counters give up after this many polls
  int v_cm;                // INT2 value pages channel-major (OSCAR_FORMAT_INT2_CM)
  int folded;              // decode: q arrives rotated, the output stays rotated (OSCAR_PLAN_FOLDED_ROTATIONS)
  DeviceLayout lay;
};
// Polls of a dependency-counter wait (each about 0.1-0.3 us: a sleep and an acquire load)
// unless oscar_set_wait_limit sets another count: roughly a second.
constexpr uint32_t kDefaultCounterPolls = 1u << 22;

// Decode workspace layout (per plan).
struct DecodeWorkspace {
  size_t partials;  // [n_items] slots of G x (fp32 m, l) then G x d fp32 o~ / l
  size_t total;
};

// Launchers (defined in the .cu files); return a cudaError_t as int.
// Work-item counts live in device memory (the plan blocks); `grid` is the number of CTAs the
// host launches, each CTA loops over items blockIdx.x, + gridDim.x, ... so a captured
// launch stays valid when a later plan has a different item count.
int launch_append(const KernelParams& kp, int layer, const void* k_new, const void* v_new, int n_items, int n_sm,
                  void* stream, int* launches);
int launch_bf16_append(const KernelParams& kp, int layer, const void* k_new, const void* v_new, int grid, void* stream,
                       int* launches);
// Decode; with `fused`, the same launch first runs the pending reservation's append tasks
// (k_new, v_new as for launch_append) and decode items wait for the ones they depend on.
// `wide`: the 16-warp CTA shape (GQA 4 only; the plan was made for it).
int launch_decode(const KernelParams& kp, int layer, const void* q, void* out, float* out_f32, uint8_t* ws,
                  const DecodeWorkspace& wl, bool wide, int n_sm, void* stream, int* launches,
                  const void* k_new = nullptr, const void* v_new = nullptr, bool fused = false);
// `deep`: the BF16 kernel with the deeper row pipeline (one-wave plans; the plan was made
// for it).
int launch_bf16_decode(const KernelParams& kp, int layer, const void* q, void* out, float* out_f32, uint8_t* ws,
                       const DecodeWorkspace& wl, bool deep, int n_sm, void* stream, int* launches);

// CTAs of the decode kernel of this shape that fit on the GPU at once (occupancy x SMs);
// the planner sizes work items so that one wave holds them all.
int decode_resident_ctas(int gqa, int group, bool wide, bool cm, int n_sm);
int bf16_decode_resident_ctas(int gqa, bool deep, int n_sm);

// Offline calibration of one layer on the GPU (calib.cu): workspace layout (byte offsets)
// and the launcher.  C_out (nullable): fp64 [2 H_kv][d][d], C_Q of every kv-head then C_S.
struct CalibWorkspace {
  size_t O, partials, C, U, lam, sweeps, keys;
  int splits;
  size_t total;
};
CalibWorkspace calib_workspace(int n_tokens, int n_q_heads, int n_kv_heads);
int launch_calibrate(const void* q, const void* k, const void* v, int n_tokens, int n_q_heads, int n_kv_heads,
                     long clip_rank, bool hadamard_only, float* R_K, float* R_V, float* clip_K, float* clip_V,
                     double* C_out, uint8_t* ws, void* stream, int* launches);

// Decode with the library's own fixed device scratch instead of a caller workspace
// (decode.cu).  Returns a cudaError_t as int; `too_big` is set when the plan's workspace
// exceeds static_scratch_bytes().
size_t static_scratch_bytes();
int launch_decode_static_scratch(const KernelParams& kp, int layer, const void* q, void* out, float* out_f32,
                                 const DecodeWorkspace& wl, bool wide, int n_sm, void* stream, int* launches,
                                 bool* too_big);

}  // namespace oscar
