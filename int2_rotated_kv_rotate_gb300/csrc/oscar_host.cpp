// Host side of the C ABI (include/oscar.h): configuration checks, the device-block layout,
// the page allocator with reference-counted prefix sharing, request state, append and
// split-K decode planning, uploads of plans and page-table rows, status readback.
//
// Paged KV with prefix caching, BF16 sinks / recent tokens and INT2 history follow the
// online-serving part of the OSCAR technical summary (gist.science), section 2.2-B.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "oscar_internal.h"

using namespace oscar;

constexpr int kUploadSlots = 6;  // pinned upload buffers (two uploads per step: reserve, plan)

namespace {

thread_local std::string g_error;
thread_local int g_launches = 0;

oscar_status fail(oscar_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
oscar_status fail(oscar_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_error = buf;
  return st;
}

#define CUDA_TRY(expr)                                                                        \
  do {                                                                                        \
    cudaError_t e_ = (expr);                                                                  \
    if (e_ != cudaSuccess) return fail(OSCAR_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
// offsets of the items inside a plan block (counts at 0, requests at 256)
size_t append_items_offset(size_t reqs) { return 256 + align256(reqs * sizeof(AppendReq)); }
size_t decode_items_offset(size_t reqs) { return 256 + align256(reqs * sizeof(DecodeReq)); }
int ceil_div(int a, int b) { return (a + b - 1) / b; }

constexpr int kAppendChunk = 16;     // tokens (or ring slots) per append work item
constexpr int kMaxAppendTokenItems = 65536;
constexpr int kBf16ItemTokens = 128;  // sink+ring tokens per decode work item (at least; one chunk of the CTA)

bool config_ok(const oscar_config* c, std::string* why) {
  auto bad = [&](const char* m) {
    *why = m;
    return false;
  };
  if (!c) return bad("config is NULL");
  if (c->format != OSCAR_FORMAT_INT2 && c->format != OSCAR_FORMAT_BF16 && c->format != OSCAR_FORMAT_INT2_CM)
    return bad("format must be INT2, INT2_CM or BF16");
  if (c->head_dim != kHeadDim) return bad("head_dim must be 128");
  if (c->page != kPage) return bad("page must be 64");
  if (c->n_kv_heads <= 0 || c->n_q_heads <= 0 || c->n_q_heads % c->n_kv_heads) return bad("bad head counts");
  int g = c->n_q_heads / c->n_kv_heads;
  if (g != 4 && g != 8) return bad("H_q / H_kv must be 4 or 8");
  if (c->n_layers <= 0 || c->max_requests <= 0 || c->max_pages <= 0 || c->max_pages_per_request <= 0)
    return bad("layers, requests and pages must be positive");
  if (c->max_pages_per_request > (1 << 20)) return bad("max_pages_per_request too large");
  if (c->format == OSCAR_FORMAT_INT2 || c->format == OSCAR_FORMAT_INT2_CM) {
    if (c->group != 32 && c->group != 128) return bad("group must be 32 or 128");
    if (c->format == OSCAR_FORMAT_INT2_CM && c->group == 32 && g != 4)
      return bad("the INT2_CM format supports group 32 at GQA 4 only");
    if (c->n_sink < 0 || c->n_sink > kPage) return bad("n_sink must be in [0, 64]");
    if (c->window < 0 || c->window > kMaxWindow || c->window % 16) return bad("window must be a multiple of 16 in [0, 1024]");
  }
  return true;
}

DeviceLayout compute_layout(const oscar_config& c) {
  DeviceLayout L;
  std::memset(&L, 0, sizeof L);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  const size_t d = kHeadDim, Hkv = c.n_kv_heads, layers = c.n_layers, pages = c.max_pages;
  const size_t reqs = c.max_requests;
  if (c.format == OSCAR_FORMAT_INT2 || c.format == OSCAR_FORMAT_INT2_CM) {
    const size_t ng = d / c.group;
    L.codes_head_stride = 2 * kPage * kRowBytes;
    L.codes_page_stride = Hkv * L.codes_head_stride;
    L.codes_layer_stride = pages * L.codes_page_stride;
    L.codes = take(layers * L.codes_layer_stride);
    L.sz_head_stride = 2 * kPage * ng * 4;
    L.sz_page_stride = Hkv * L.sz_head_stride;
    L.sz_layer_stride = pages * L.sz_page_stride;
    L.sz = take(layers * L.sz_layer_stride);
    L.sink_head_stride = 2 * size_t(c.n_sink) * d * 2;
    L.sink_layer_stride = Hkv * L.sink_head_stride;
    L.sink_slot_stride = layers * L.sink_layer_stride;
    L.sink = take(reqs * L.sink_slot_stride);
    L.ring_head_stride = 2 * size_t(c.window) * d * 2;
    L.ring_layer_stride = Hkv * L.ring_head_stride;
    L.ring_slot_stride = layers * L.ring_layer_stride;
    L.ring = take(reqs * L.ring_slot_stride);
    L.R_K = take(layers * Hkv * d * d * 4);
    L.R_V = take(layers * Hkv * d * d * 4);
    L.R_Vt = take(layers * Hkv * d * d * 4);
    L.clip_K = take(layers * Hkv * 4);
    L.clip_V = take(layers * Hkv * 4);
  } else {
    L.bf16_head_stride = 2 * kPage * d * 2;
    L.bf16_page_stride = Hkv * L.bf16_head_stride;
    L.bf16_layer_stride = pages * L.bf16_page_stride;
    L.bf16_pages = take(layers * L.bf16_layer_stride);
  }
  L.page_table = take(reqs * size_t(c.max_pages_per_request) * 4);
  L.status = take(256);
  L.counters = take(reqs * Hkv * 4);
  L.max_append_items = kMaxAppendTokenItems + reqs * (kMaxWindow / kAppendChunk + 1);  // + 1: a block-aligned split
  L.max_decode_items = reqs * Hkv * (2 + kMaxWindow / kBf16ItemTokens) + 16384;
  L.append_plan = take(append_items_offset(reqs) + L.max_append_items * sizeof(AppendItem));
  L.append_counts = L.append_plan;
  L.append_reqs = L.append_plan + 256;
  L.append_items = L.append_plan + append_items_offset(reqs);
  L.decode_plan = take(decode_items_offset(reqs) + L.max_decode_items * sizeof(DecodeItem));
  L.decode_counts = L.decode_plan;
  L.decode_reqs = L.decode_plan + 256;
  L.decode_items = L.decode_plan + decode_items_offset(reqs);
  L.sched = take(16);
  L.app_done = take(layers * reqs * Hkv * 8);
  L.total = off;
  return L;
}

struct Request {
  bool in_use = false;
  int L = 0, H = 0;
  std::vector<int> pages;
};

}  // namespace

struct oscar_cache {
  oscar_config cfg;
  DeviceLayout lay;
  uint8_t* base = nullptr;
  int n_sm = 148;
  std::vector<Request> reqs;
  std::vector<int> refcount;
  std::vector<int> free_pages;
  // host mirror of the page table, and a ring of pinned upload buffers: every upload copies
  // what it sends into the next buffer first, so the host never rewrites memory that an
  // enqueued copy still reads, and waits only when it runs kUploadSlots uploads ahead
  int32_t* h_page_table = nullptr;
  uint8_t* h_upload = nullptr;  // kUploadSlots x upload_bytes, pinned
  size_t upload_bytes = 0, staging_bytes = 0;
  cudaEvent_t upload_done[kUploadSlots] = {};
  bool upload_pending[kUploadSlots] = {};
  int upload_next = 0;
  uint32_t* h_status = nullptr;
  // pending append
  bool reserved = false;
  std::vector<AppendReq> app_reqs;
  std::vector<int> app_req_items;  // append items of each reservation request
  int app_items = 0, app_rows = 0;
  bool plan_covers_reservation = false;  // the plan lists every slot of the pending reservation
  bool dec_wide = false;                  // INT2: the plan is for 16-warp split-kernel CTAs; BF16: for the deep pipeline
  bool dec_folded = false;                // OSCAR_PLAN_FOLDED_ROTATIONS: q~ in, o~ out
  // decode plan
  bool planned = false;
  bool planned_with_reservation = false;  // the plan already counts the reserved tokens
  int dec_n_req = 0, dec_items = 0, dec_bf16_items = 0, dec_max_pages = 0;
  DecodeWorkspace ws{};
  int device = 0;              // the device current at creation (the device of `base`)
  uint32_t counter_polls = 0;  // oscar_set_wait_limit (0 = kDefaultCounterPolls)
  uint32_t inject = 0;         // oscar_inject_fault: host-side faults armed for the next plan
};

namespace {

// One upload buffer: page-table rows (max_requests rows), then the image of a plan block.
struct Upload {
  int32_t* rows;
  uint8_t* staging;
  int slot;
};

KernelParams kernel_params(const oscar_cache* c) {
  KernelParams kp;
  kp.base = c->base;
  kp.n_q_heads = c->cfg.n_q_heads;
  kp.n_kv_heads = c->cfg.n_kv_heads;
  kp.gqa = c->cfg.n_q_heads / c->cfg.n_kv_heads;
  kp.group = c->cfg.group;
  kp.n_sink = c->cfg.n_sink;
  kp.window = c->cfg.window;
  kp.n_layers = c->cfg.n_layers;
  kp.max_requests = c->cfg.max_requests;
  kp.max_pages = c->cfg.max_pages;
  kp.max_pages_per_request = c->cfg.max_pages_per_request;
  kp.counter_polls = c->counter_polls ? c->counter_polls : kDefaultCounterPolls;
  kp.v_cm = c->cfg.format == OSCAR_FORMAT_INT2_CM;
  kp.folded = c->dec_folded;
  kp.lay = c->lay;
  return kp;
}

// The next upload buffer of the ring, once the copies that last read it have run.
oscar_status begin_upload(oscar_cache* c, Upload* u) {
  const int i = c->upload_next;
  c->upload_next = (i + 1) % kUploadSlots;
  if (c->upload_pending[i]) {
    CUDA_TRY(cudaEventSynchronize(c->upload_done[i]));
    c->upload_pending[i] = false;
  }
  uint8_t* b = c->h_upload + size_t(i) * c->upload_bytes;
  u->rows = reinterpret_cast<int32_t*>(b);
  u->staging = b + align256(size_t(c->cfg.max_requests) * c->cfg.max_pages_per_request * 4);
  u->slot = i;
  return OSCAR_OK;
}

// Record that the copies enqueued on s so far read upload buffer u.
oscar_status end_upload(oscar_cache* c, const Upload& u, cudaStream_t s) {
  CUDA_TRY(cudaEventRecord(c->upload_done[u.slot], s));
  c->upload_pending[u.slot] = true;
  return OSCAR_OK;
}

// Every upload buffer is free again (teardown).
void drain_uploads(oscar_cache* c) {
  for (int i = 0; i < kUploadSlots; ++i)
    if (c->upload_pending[i]) {
      cudaEventSynchronize(c->upload_done[i]);
      c->upload_pending[i] = false;
    }
}

// Page-table rows of `slots` from the host mirror, through upload buffer u.
oscar_status upload_rows(oscar_cache* c, const Upload& u, const std::vector<int>& slots, cudaStream_t s) {
  const size_t n = size_t(c->cfg.max_pages_per_request);
  for (size_t k = 0; k < slots.size(); ++k) {
    int32_t* dst = u.rows + k * n;
    std::memcpy(dst, c->h_page_table + size_t(slots[k]) * n, n * 4);
    CUDA_TRY(cudaMemcpyAsync(c->base + c->lay.page_table + size_t(slots[k]) * n * 4, dst, n * 4,
                             cudaMemcpyHostToDevice, s));
  }
  return OSCAR_OK;
}

bool is_int2(const oscar_cache* c) {
  return c->cfg.format == OSCAR_FORMAT_INT2 || c->cfg.format == OSCAR_FORMAT_INT2_CM;
}
// Channel-major value pages, decoded on the tcgen05 tensor cores; never a fused launch.
bool is_cm(const oscar_cache* c) { return c->cfg.format == OSCAR_FORMAT_INT2_CM; }

// Pages a request needs to hold its stored tokens: the INT2 format pages positions < H
// (sinks and recent tokens live elsewhere), the BF16 format pages all L positions.
int pages_needed(const oscar_cache* c, int L, int H) {
  if (is_int2(c)) return H > c->cfg.n_sink ? ceil_div(H, kPage) : 0;
  return ceil_div(L, kPage);
}

oscar_status check_slot(const oscar_cache* c, int slot) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (slot < 0 || slot >= c->cfg.max_requests) return fail(OSCAR_ERR_INVALID_ARG, "slot %d out of range", slot);
  if (!c->reqs[slot].in_use) return fail(OSCAR_ERR_INVALID_ARG, "slot %d is not allocated", slot);
  return OSCAR_OK;
}

}  // namespace

extern "C" {

const char* oscar_last_error(void) { return g_error.c_str(); }
int oscar_last_launch_count(void) { return g_launches; }

size_t oscar_cache_device_bytes(const oscar_config* cfg) {
  std::string why;
  if (!config_ok(cfg, &why)) {
    g_error = why;
    return 0;
  }
  return compute_layout(*cfg).total;
}

oscar_status oscar_cache_create(const oscar_config* cfg, void* device_mem, size_t bytes, oscar_cache** out) {
  std::string why;
  if (!out) return fail(OSCAR_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!config_ok(cfg, &why)) return fail(OSCAR_ERR_INVALID_ARG, "%s", why.c_str());
  if (!device_mem) return fail(OSCAR_ERR_INVALID_ARG, "device_mem is NULL");
  if (reinterpret_cast<uintptr_t>(device_mem) % 256) return fail(OSCAR_ERR_INVALID_ARG, "device_mem must be 256-byte aligned");
  DeviceLayout lay = compute_layout(*cfg);
  if (bytes < lay.total) return fail(OSCAR_ERR_INVALID_ARG, "device block of %zu bytes < %zu needed", bytes, lay.total);
  oscar_cache* c = new (std::nothrow) oscar_cache();
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "host allocation failed");
  c->cfg = *cfg;
  c->lay = lay;
  c->base = static_cast<uint8_t*>(device_mem);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  c->device = dev;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->n_sm, cudaDevAttrMultiProcessorCount, dev);
  c->reqs.resize(cfg->max_requests);
  c->refcount.assign(cfg->max_pages, 0);
  c->free_pages.reserve(cfg->max_pages);
  for (int p = cfg->max_pages - 1; p >= 0; --p) c->free_pages.push_back(p);
  const size_t pt_bytes = size_t(cfg->max_requests) * cfg->max_pages_per_request * 4;
  // a plan block's image (the larger of the two)
  c->staging_bytes = std::max(append_items_offset(cfg->max_requests) + lay.max_append_items * sizeof(AppendItem),
                              decode_items_offset(cfg->max_requests) + lay.max_decode_items * sizeof(DecodeItem));
  c->upload_bytes = align256(pt_bytes) + align256(c->staging_bytes);
  if (e == cudaSuccess) e = cudaMallocHost(reinterpret_cast<void**>(&c->h_page_table), pt_bytes);
  if (e == cudaSuccess) e = cudaMallocHost(reinterpret_cast<void**>(&c->h_upload), kUploadSlots * c->upload_bytes);
  if (e == cudaSuccess) e = cudaMallocHost(reinterpret_cast<void**>(&c->h_status), 256);
  if (e == cudaSuccess) e = cudaMemset(c->base + lay.append_counts, 0, 16);
  if (e == cudaSuccess) e = cudaMemset(c->base + lay.decode_counts, 0, 16);
  for (int i = 0; i < kUploadSlots && e == cudaSuccess; ++i)
    e = cudaEventCreateWithFlags(&c->upload_done[i], cudaEventDisableTiming);
  if (e == cudaSuccess) {
    std::memset(c->h_page_table, 0xff, pt_bytes);  // -1 = unmapped
    e = cudaMemcpy(c->base + lay.page_table, c->h_page_table, pt_bytes, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaMemset(c->base + lay.status, 0, 256);
  if (e == cudaSuccess) e = cudaMemset(c->base + lay.counters, 0, size_t(cfg->max_requests) * cfg->n_kv_heads * 4);
  if (e == cudaSuccess) e = cudaMemset(c->base + lay.sched, 0, 16);
  // scale/zero words of rows no append has written yet (sink positions, the tail of a
  // page) are read with p = 0 by the decode: they must be finite, so the pool starts at 0
  if (e == cudaSuccess && is_int2(c)) e = cudaMemset(c->base + lay.sz, 0, size_t(cfg->n_layers) * lay.sz_layer_stride);
  if (e == cudaSuccess)
    e = cudaMemset(c->base + lay.app_done, 0, size_t(cfg->n_layers) * cfg->max_requests * cfg->n_kv_heads * 8);
  if (e == cudaSuccess && is_int2(c)) {
    // layer params start as zeros until oscar_set_layer_params
    e = cudaMemset(c->base + lay.R_K, 0, lay.clip_K - lay.R_K);
  }
  if (e != cudaSuccess) {
    fail(OSCAR_ERR_CUDA, "cache_create: %s", cudaGetErrorString(e));
    oscar_cache_destroy(c);
    return OSCAR_ERR_CUDA;
  }
  *out = c;
  return OSCAR_OK;
}

void oscar_cache_destroy(oscar_cache* c) {
  if (!c) return;
  drain_uploads(c);
  for (int i = 0; i < kUploadSlots; ++i)
    if (c->upload_done[i]) cudaEventDestroy(c->upload_done[i]);
  if (c->h_page_table) cudaFreeHost(c->h_page_table);
  if (c->h_upload) cudaFreeHost(c->h_upload);
  if (c->h_status) cudaFreeHost(c->h_status);
  delete c;
}

oscar_status oscar_cache_layout(const oscar_cache* c, oscar_layout* out) {
  if (!c || !out) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
  const DeviceLayout& L = c->lay;
  out->codes = L.codes;
  out->sz = L.sz;
  out->sink = L.sink;
  out->ring = L.ring;
  out->bf16_pages = L.bf16_pages;
  out->codes_page_bytes = L.codes_head_stride;
  out->sz_page_bytes = L.sz_head_stride;
  out->bf16_page_bytes = L.bf16_head_stride;
  out->sink_bytes_per_head = L.sink_head_stride;
  out->ring_bytes_per_head = L.ring_head_stride;
  out->page_table = L.page_table;
  out->total = L.total;
  return OSCAR_OK;
}

oscar_status oscar_set_layer_params(oscar_cache* c, int layer, const float* R_K, const float* R_V, const float* clip_K,
                                    const float* clip_V, void* stream) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (!is_int2(c)) return fail(OSCAR_ERR_STATE, "layer params apply to the INT2 format only");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(OSCAR_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (!R_K || !R_V || !clip_K || !clip_V) return fail(OSCAR_ERR_INVALID_ARG, "NULL parameter array");
  const int H = c->cfg.n_kv_heads, d = kHeadDim;
  for (int h = 0; h < H; ++h) {
    if (!(clip_K[h] > 0.f) || !(clip_V[h] > 0.f)) return fail(OSCAR_ERR_INVALID_ARG, "clip thresholds must be > 0");
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t mat = size_t(d) * d;
  std::vector<float> Vt(size_t(H) * mat);
  for (int h = 0; h < H; ++h)
    for (int i = 0; i < d; ++i)
      for (int j = 0; j < d; ++j) Vt[h * mat + size_t(j) * d + i] = R_V[h * mat + size_t(i) * d + j];
  const size_t lmat = size_t(layer) * H * mat * 4;
  CUDA_TRY(cudaMemcpyAsync(c->base + c->lay.R_K + lmat, R_K, H * mat * 4, cudaMemcpyHostToDevice, s));
  CUDA_TRY(cudaMemcpyAsync(c->base + c->lay.R_V + lmat, R_V, H * mat * 4, cudaMemcpyHostToDevice, s));
  CUDA_TRY(cudaMemcpyAsync(c->base + c->lay.R_Vt + lmat, Vt.data(), H * mat * 4, cudaMemcpyHostToDevice, s));
  CUDA_TRY(cudaMemcpyAsync(c->base + c->lay.clip_K + size_t(layer) * H * 4, clip_K, H * 4, cudaMemcpyHostToDevice, s));
  CUDA_TRY(cudaMemcpyAsync(c->base + c->lay.clip_V + size_t(layer) * H * 4, clip_V, H * 4, cudaMemcpyHostToDevice, s));
  CUDA_TRY(cudaStreamSynchronize(s));  // Vt is a temporary
  return OSCAR_OK;
}

oscar_status oscar_request_alloc(oscar_cache* c, int* slot) {
  if (!c || !slot) return fail(OSCAR_ERR_INVALID_ARG, "NULL argument");
  for (int i = 0; i < c->cfg.max_requests; ++i) {
    if (!c->reqs[i].in_use) {
      c->reqs[i] = Request();
      c->reqs[i].in_use = true;
      c->reqs[i].H = is_int2(c) ? c->cfg.n_sink : 0;
      *slot = i;
      return OSCAR_OK;
    }
  }
  return fail(OSCAR_ERR_OUT_OF_PAGES, "no free request slot");
}

oscar_status oscar_request_free(oscar_cache* c, int slot) {
  oscar_status st = check_slot(c, slot);
  if (st) return st;
  if (c->reserved)
    for (const AppendReq& r : c->app_reqs)
      if (r.slot == slot) return fail(OSCAR_ERR_STATE, "slot %d has a pending reservation", slot);
  Request& r = c->reqs[slot];
  for (int p : r.pages)
    if (--c->refcount[p] == 0) c->free_pages.push_back(p);
  // the device row keeps stale ids; it is rewritten before the slot is used again
  std::fill(c->h_page_table + size_t(slot) * c->cfg.max_pages_per_request,
            c->h_page_table + size_t(slot + 1) * c->cfg.max_pages_per_request, -1);
  r = Request();
  c->planned = false;
  return OSCAR_OK;
}

oscar_status oscar_cache_stats(const oscar_cache* c, int* free_pages, int* free_slots) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (free_pages) *free_pages = int(c->free_pages.size());
  if (free_slots) {
    int n = 0;
    for (const Request& r : c->reqs) n += !r.in_use;
    *free_slots = n;
  }
  return OSCAR_OK;
}

oscar_status oscar_request_info(const oscar_cache* c, int slot, int* length, int* history_end, int* n_pages) {
  oscar_status st = check_slot(c, slot);
  if (st) return st;
  const Request& r = c->reqs[slot];
  if (length) *length = r.L;
  if (history_end) *history_end = r.H;
  if (n_pages) *n_pages = int(r.pages.size());
  return OSCAR_OK;
}

oscar_status oscar_request_pages(const oscar_cache* c, int slot, int* pages, int n) {
  oscar_status st = check_slot(c, slot);
  if (st) return st;
  const Request& r = c->reqs[slot];
  if (!pages || n < 0 || n > int(r.pages.size())) return fail(OSCAR_ERR_INVALID_ARG, "bad page buffer");
  std::copy(r.pages.begin(), r.pages.begin() + n, pages);
  return OSCAR_OK;
}

oscar_status oscar_request_share_prefix(oscar_cache* c, int dst, int src, int n_tokens, void* stream) {
  oscar_status st = check_slot(c, dst);
  if (st) return st;
  st = check_slot(c, src);
  if (st) return st;
  if (dst == src) return fail(OSCAR_ERR_INVALID_ARG, "dst == src");
  if (c->reserved) return fail(OSCAR_ERR_STATE, "a reservation is pending");
  Request& d = c->reqs[dst];
  const Request& s = c->reqs[src];
  if (d.L != 0 || !d.pages.empty()) return fail(OSCAR_ERR_INVALID_ARG, "dst must be empty");
  if (n_tokens <= 0 || n_tokens % kPage) return fail(OSCAR_ERR_INVALID_ARG, "n_tokens must be a positive multiple of 64");
  const int limit = is_int2(c) ? s.H : s.L / kPage * kPage;
  if (n_tokens > limit)
    return fail(OSCAR_ERR_INVALID_ARG, "n_tokens %d exceeds the shareable prefix %d of src", n_tokens, limit);
  if (n_tokens / kPage > c->cfg.max_pages_per_request) return fail(OSCAR_ERR_INVALID_ARG, "prefix too long");
  Upload u;
  st = begin_upload(c, &u);
  if (st) return st;
  cudaStream_t strm = static_cast<cudaStream_t>(stream);
  const int n = n_tokens / kPage;
  d.pages.assign(s.pages.begin(), s.pages.begin() + n);
  for (int p : d.pages) ++c->refcount[p];
  int32_t* row = c->h_page_table + size_t(dst) * c->cfg.max_pages_per_request;
  std::fill(row, row + c->cfg.max_pages_per_request, -1);
  std::copy(d.pages.begin(), d.pages.end(), row);
  d.L = n_tokens;
  d.H = is_int2(c) ? n_tokens : n_tokens;
  st = upload_rows(c, u, {dst}, strm);
  if (st) return st;
  if (is_int2(c) && c->lay.sink_slot_stride > 0) {
    CUDA_TRY(cudaMemcpyAsync(c->base + c->lay.sink + size_t(dst) * c->lay.sink_slot_stride,
                             c->base + c->lay.sink + size_t(src) * c->lay.sink_slot_stride, c->lay.sink_slot_stride,
                             cudaMemcpyDeviceToDevice, strm));
  }
  st = end_upload(c, u, strm);
  if (st) return st;
  c->planned = false;
  return OSCAR_OK;
}

oscar_status oscar_reserve(oscar_cache* c, const int* slots, const int* n_new, int n_req, void* stream) {
  if (!c || !slots || !n_new || n_req <= 0 || n_req > c->cfg.max_requests)
    return fail(OSCAR_ERR_INVALID_ARG, "bad reserve arguments");
  if (c->reserved) return fail(OSCAR_ERR_STATE, "previous reservation not committed");
  std::vector<char> seen(c->cfg.max_requests, 0);
  long long rows = 0;
  int new_pages = 0;
  const int S = is_int2(c) ? c->cfg.n_sink : 0, W = c->cfg.window;
  std::vector<AppendReq> reqs(n_req);
  for (int i = 0; i < n_req; ++i) {
    oscar_status st = check_slot(c, slots[i]);
    if (st) return st;
    if (seen[slots[i]]) return fail(OSCAR_ERR_INVALID_ARG, "slot %d listed twice", slots[i]);
    seen[slots[i]] = 1;
    if (n_new[i] < 0) return fail(OSCAR_ERR_INVALID_ARG, "negative n_new");
    const Request& r = c->reqs[slots[i]];
    AppendReq& a = reqs[i];
    a.slot = slots[i];
    a.L0 = r.L;
    a.H0 = r.H;
    long long L1 = (long long)r.L + n_new[i];
    if (L1 > (long long)kPage * c->cfg.max_pages_per_request)
      return fail(OSCAR_ERR_INVALID_ARG, "request %d would exceed its page-table row", slots[i]);
    a.L1 = int(L1);
    a.H1 = is_int2(c) ? std::max(r.H, a.L1 - W) : a.L1;
    a.x_offset = int(rows);
    rows += n_new[i];
    new_pages += std::max(0, pages_needed(c, a.L1, a.H1) - int(r.pages.size()));
  }
  if (rows > (1 << 30)) return fail(OSCAR_ERR_INVALID_ARG, "too many rows");
  if (new_pages > int(c->free_pages.size()))
    return fail(OSCAR_ERR_OUT_OF_PAGES, "need %d pages, %zu free", new_pages, c->free_pages.size());
  // work items
  std::vector<AppendItem> items;
  for (int i = 0; i < n_req; ++i) {
    const AppendReq& a = reqs[i];
    if (is_int2(c) && W > 0) {
      std::vector<char> touched(W, 0);
      for (int p = a.H0; p < std::min(a.L0, a.H1); ++p) touched[p % W] = 1;   // evicted
      for (int p = std::max(a.L0, a.H1); p < a.L1; ++p) touched[p % W] = 1;  // new ring tokens
      for (int s0 = 0; s0 < W; s0 += kAppendChunk) {
        bool any = false;
        for (int s = s0; s < s0 + kAppendChunk; ++s) any |= touched[s] != 0;
        if (any) items.push_back({i, 0, s0, kAppendChunk});
      }
    }
    const int d0 = a.L0, d1 = is_int2(c) ? std::min(a.L1, a.H1) : a.L1;
    // channel-major value pages: an item's positions stay inside one 16-position block,
    // whose code words (one per channel) the append kernel writes whole
    for (int p = d0; p < d1;) {
      const int e = is_cm(c) ? std::min(d1, (p / kAppendChunk + 1) * kAppendChunk) : std::min(d1, p + kAppendChunk);
      items.push_back({i, 1, p, e - p});
      p = e;
    }
  }
  if (items.size() > c->lay.max_append_items)
    return fail(OSCAR_ERR_INVALID_ARG, "append of %lld tokens is too large for one reservation; split it", rows);
  Upload u;
  oscar_status st = begin_upload(c, &u);
  if (st) return st;
  // allocate pages and update the host mirror
  std::vector<int> changed;
  for (const AppendReq& a : reqs) {
    Request& r = c->reqs[a.slot];
    int need = pages_needed(c, a.L1, a.H1);
    if (need > int(r.pages.size())) {
      int32_t* row = c->h_page_table + size_t(a.slot) * c->cfg.max_pages_per_request;
      while (int(r.pages.size()) < need) {
        int p = c->free_pages.back();
        c->free_pages.pop_back();
        c->refcount[p] = 1;
        row[r.pages.size()] = p;
        r.pages.push_back(p);
      }
      changed.push_back(a.slot);
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = upload_rows(c, u, changed, s);
  if (st) return st;
  // the append plan block, one copy
  const size_t items_off = append_items_offset(c->cfg.max_requests);
  int32_t* counts = reinterpret_cast<int32_t*>(u.staging);
  counts[0] = int(items.size());
  counts[1] = counts[2] = counts[3] = 0;
  std::memcpy(u.staging + 256, reqs.data(), reqs.size() * sizeof(AppendReq));
  std::memcpy(u.staging + items_off, items.data(), items.size() * sizeof(AppendItem));
  CUDA_TRY(cudaMemcpyAsync(c->base + c->lay.append_plan, u.staging, items_off + items.size() * sizeof(AppendItem),
                           cudaMemcpyHostToDevice, s));
  st = end_upload(c, u, s);
  if (st) return st;
  c->app_reqs = reqs;
  c->app_req_items.assign(reqs.size(), 0);
  for (const AppendItem& it : items) ++c->app_req_items[it.req];
  c->app_items = int(items.size());
  c->app_rows = int(rows);
  c->reserved = true;
  c->planned = false;  // lengths change: plan again (a plan made now counts the new tokens)
  c->planned_with_reservation = false;
  return OSCAR_OK;
}

oscar_status oscar_commit_append(oscar_cache* c) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (!c->reserved) return fail(OSCAR_ERR_STATE, "no reservation to commit");
  for (const AppendReq& a : c->app_reqs) {
    c->reqs[a.slot].L = a.L1;
    c->reqs[a.slot].H = a.H1;
  }
  c->reserved = false;
  if (!c->planned_with_reservation) c->planned = false;
  c->planned_with_reservation = false;
  c->plan_covers_reservation = false;
  return OSCAR_OK;
}

oscar_status oscar_quantize_append(oscar_cache* c, int layer, const void* k_new, const void* v_new, void* stream) {
  g_launches = 0;
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (!is_int2(c)) return fail(OSCAR_ERR_STATE, "oscar_quantize_append needs the INT2 format");
  if (!c->reserved) return fail(OSCAR_ERR_STATE, "no reservation");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(OSCAR_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (c->app_rows > 0 && (!k_new || !v_new)) return fail(OSCAR_ERR_INVALID_ARG, "NULL token arrays");
  if (c->app_items == 0) return OSCAR_OK;
  int e = launch_append(kernel_params(c), layer, k_new, v_new, c->app_items, c->n_sm, stream, &g_launches);
  if (e) return fail(OSCAR_ERR_CUDA, "append launch: %s", cudaGetErrorString(cudaError_t(e)));
  return OSCAR_OK;
}

oscar_status oscar_bf16_append(oscar_cache* c, int layer, const void* k_new, const void* v_new, void* stream) {
  g_launches = 0;
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (is_int2(c)) return fail(OSCAR_ERR_STATE, "oscar_bf16_append needs the BF16 format");
  if (!c->reserved) return fail(OSCAR_ERR_STATE, "no reservation");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(OSCAR_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (c->app_rows > 0 && (!k_new || !v_new)) return fail(OSCAR_ERR_INVALID_ARG, "NULL token arrays");
  if (c->app_items == 0) return OSCAR_OK;
  int e = launch_bf16_append(kernel_params(c), layer, k_new, v_new, std::min(c->app_items, 4 * c->n_sm), stream,
                             &g_launches);
  if (e) return fail(OSCAR_ERR_CUDA, "bf16 append launch: %s", cudaGetErrorString(cudaError_t(e)));
  return OSCAR_OK;
}

oscar_status oscar_plan_decode(oscar_cache* c, const int* slots, int n_req, int max_split_pages, void* stream) {
  return oscar_plan_decode_ex(c, slots, n_req, max_split_pages, 0u, stream);
}

oscar_status oscar_plan_decode_ex(oscar_cache* c, const int* slots, int n_req, int max_split_pages, uint32_t flags,
                                  void* stream) {
  if (!c || !slots || n_req <= 0 || n_req > c->cfg.max_requests)
    return fail(OSCAR_ERR_INVALID_ARG, "bad plan arguments");
  if (flags & ~(OSCAR_PLAN_NARROW | OSCAR_PLAN_FOLDED_ROTATIONS))
    return fail(OSCAR_ERR_INVALID_ARG, "unknown plan flags %#x", flags);
  if ((flags & OSCAR_PLAN_FOLDED_ROTATIONS) && !is_int2(c))
    return fail(OSCAR_ERR_INVALID_ARG, "OSCAR_PLAN_FOLDED_ROTATIONS applies to the INT2 formats");
  if (max_split_pages < 0) return fail(OSCAR_ERR_INVALID_ARG, "max_split_pages < 0");
  std::vector<char> seen(c->cfg.max_requests, 0);
  const int Hkv = c->cfg.n_kv_heads, S = is_int2(c) ? c->cfg.n_sink : 0;
  // lengths the decode will see: a pending reservation's tokens count (append before decode)
  std::vector<int> Ls(n_req), Hs(n_req), Hpre(n_req), Lpre(n_req), app_items(n_req, 0), app_expect(n_req, 0);
  int n_reserved_planned = 0;
  long long total_pages = 0;
  for (int i = 0; i < n_req; ++i) {
    oscar_status st = check_slot(c, slots[i]);
    if (st) return st;
    if (seen[slots[i]]) return fail(OSCAR_ERR_INVALID_ARG, "slot %d listed twice", slots[i]);
    seen[slots[i]] = 1;
    const Request& r = c->reqs[slots[i]];
    Ls[i] = r.L;
    Hs[i] = r.H;
    Hpre[i] = r.H;
    Lpre[i] = r.L;
    if (c->reserved)
      for (size_t k = 0; k < c->app_reqs.size(); ++k) {
        const AppendReq& a = c->app_reqs[k];
        if (a.slot == slots[i]) {
          Ls[i] = a.L1;
          Hs[i] = a.H1;
          Hpre[i] = std::min(r.H, a.H0);
          Lpre[i] = std::min(r.L, a.L0);
          app_items[i] = c->app_req_items[k];
          ++n_reserved_planned;
        }
      }
    total_pages += (long long)Hkv * pages_needed(c, Ls[i], Hs[i]);
  }
  // Work items: per (request, kv-head) the BF16 sink+ring items and page ranges of
  // `chunk` pages.  Automatic chunk, from the bytes each resident CTA would stream:
  //  - small steps (latency-bound): the smallest chunk that lets one wave of resident CTAs
  //    hold every item (a second, partial wave would add a whole item's latency);
  //  - large steps: about kWaves items per resident CTA (at least kItemBytes each), taken
  //    dynamically by the CTAs, largest first, so the ragged tail stays short while the
  //    per-item costs (pipeline fill, partial store and merge) stay small.
  // Per request: INT2 pages np, BF16 sink+ring tokens n_bf, and the split points of the
  // items that do not (before) and may (after) read rows of this step's append: bf_new in
  // the BF16 list, pg_new in the pages.
  std::vector<int> np_of(n_req), nbf_of(n_req), bfnew_of(n_req), pgnew_of(n_req);
  int max_np = 1;
  const int ng = kHeadDim / (is_int2(c) ? c->cfg.group : kHeadDim);
  const long long page_bytes = is_int2(c) ? 2LL * kPage * (kRowBytes + 4 * ng) : 2LL * kPage * kHeadDim * 2;
  long long total_bytes = 0;
  for (int i = 0; i < n_req; ++i) {
    np_of[i] = pages_needed(c, Ls[i], Hs[i]);
    nbf_of[i] = is_int2(c) ? std::min(Ls[i], S) + std::max(0, Ls[i] - Hs[i]) : 0;
    bfnew_of[i] = nbf_of[i];
    pgnew_of[i] = np_of[i];
    // A fused launch's BF16 items of an appending request wait for its rows as a whole (the
    // new rows are a small part of the list); its INT2 items are not split: the append's
    // eviction rows are signalled before the launch's wait, and the one warp whose page
    // holds them waits for that signal before copying it.
    if (app_items[i] > 0) bfnew_of[i] = 0;
    max_np = std::max(max_np, np_of[i]);
    total_bytes += (long long)Hkv * (np_of[i] * page_bytes + nbf_of[i] * 2LL * kHeadDim * 2);
  }
  // CTA shape: at GQA 4 a step that one wave of 16-warp CTAs holds (one per SM) is planned
  // for them ("wide"); larger steps for 8-warp CTAs, two per SM.
  constexpr long long kItemBytes = 512 << 10;
  constexpr long long kWaves = 2;
  const int G = c->cfg.n_q_heads / Hkv;
  bool wide = false;
  if (is_int2(c) && G == 4 && !(flags & OSCAR_PLAN_NARROW)) {
    const int r_wide = decode_resident_ctas(G, c->cfg.group, true, is_cm(c), c->n_sm);
    wide = r_wide > 0 && total_bytes <= kItemBytes * r_wide;
  }
  if (!is_int2(c)) {  // BF16: the deeper row pipeline for steps that one wave holds
    const int r_deep = bf16_decode_resident_ctas(G, true, c->n_sm);
    wide = r_deep > 0 && total_bytes <= kItemBytes * r_deep;
  }
  const int nw = decode_warps(G, wide);
  for (int i = 0; i < n_req; ++i) app_expect[i] = 2 * append_task_split(nw) * app_items[i];  // per kv-head
  if ((c->inject & OSCAR_FAULT_LOST_APPEND_SIGNAL) && c->reserved)
    for (int i = 0; i < n_req; ++i)
      if (app_expect[i] > 0) {  // one signal more than the append tasks send: it never arrives
        ++app_expect[i];
        c->inject &= ~OSCAR_FAULT_LOST_APPEND_SIGNAL;
        break;
      }
  auto split_count = [](int a, int b, int step) { return (a > 0 ? ceil_div(a, step) : 0) + (b > a ? ceil_div(b - a, step) : 0); };
  long long n_bf_items = 0;
  // BF16 items of one CTA chunk: 16 tokens per warp
  const int bf_item = is_int2(c) ? 16 * nw : kBf16ItemTokens;
  for (int i = 0; i < n_req; ++i) n_bf_items += (long long)Hkv * split_count(bfnew_of[i], nbf_of[i], bf_item);
  auto count_items = [&](int ch) {
    long long n = n_bf_items;
    for (int i = 0; i < n_req; ++i) {
      const int pg = split_count(pgnew_of[i], np_of[i], ch);
      const int bf = split_count(bfnew_of[i], nbf_of[i], bf_item);
      n += (long long)Hkv * (pg + bf > 0 ? pg : 1);
    }
    return n;
  };
  int chunk = max_split_pages;
  if (chunk == 0) {
    int resident =
        is_int2(c) ? decode_resident_ctas(G, c->cfg.group, wide, is_cm(c), c->n_sm) : bf16_decode_resident_ctas(G, wide, c->n_sm);
    if (resident <= 0) resident = 2 * c->n_sm;
    if (total_bytes <= kItemBytes * resident) {
      // a fused append + decode launch runs the reservation's append tasks in the same wave
      const long long n_app_tasks =
          c->reserved && !is_cm(c) ? (long long)c->app_items * Hkv * 2 * append_task_split(nw) : 0;
      const long long slots = std::max<long long>(1, resident - n_bf_items - n_app_tasks);
      chunk = int(std::max<long long>(4, (total_pages + slots - 1) / slots));
      while (chunk < max_np && count_items(chunk) + n_app_tasks > resident) ++chunk;
    } else {
      const long long item_bytes = std::max(kItemBytes, total_bytes / (kWaves * resident));
      chunk = int(std::max<long long>(4, item_bytes / page_bytes));
    }
    // the plan must fit the item buffers
    while (chunk < max_np && count_items(chunk) > (long long)c->lay.max_decode_items)
      chunk = std::min(max_np, chunk + chunk / 4 + 1);
  }
  std::vector<DecodeReq> reqs(n_req);
  std::vector<DecodeItem> items;
  int n_bf16 = 0, max_pages = 0;
  for (int i = 0; i < n_req; ++i) {
    DecodeReq& q = reqs[i];
    q.slot = slots[i];
    q.L = Ls[i];
    q.H = is_int2(c) ? Hs[i] : Ls[i];
    q.H_pre = is_int2(c) ? Hpre[i] : Lpre[i];
    q.app_expect = is_int2(c) ? app_expect[i] : 0;
    const int np = np_of[i], n_bf = nbf_of[i], bf_new = bfnew_of[i], pg_new = pgnew_of[i];
    // BF16 list index of this step's first new row (index < min(L, S): sink, else ring
    // position H + index - min(L, S)); rows before it are final before the launch's wait
    int u_new = n_bf;
    if (is_int2(c) && Lpre[i] < Ls[i]) {
      const int n_s = std::min(q.L, S);
      u_new = std::min(n_bf, Lpre[i] < n_s ? Lpre[i] : n_s + std::max(0, Lpre[i] - q.H));
    }
    q.first_item = int(items.size());
    for (int h = 0; h < Hkv; ++h) {
      const int first = int(items.size());
      auto add = [&](int kind, int b, int e, int dep) {
        items.push_back({i, h, kind, b, e, first, 0, dep, kind == 1 ? std::min(e, std::max(b, u_new)) : e});
      };
      if (n_bf == 0 && np == 0) add(1, 0, 0, kDepNone);  // empty request: one empty item writes zeros
      // BF16 sink+ring list, split where this step's new tokens start (those items wait for
      // a fused launch's append tasks; the others do not)
      for (int part = 0; part < 2; ++part) {
        const int b0 = part == 0 ? 0 : bf_new, b1 = part == 0 ? bf_new : n_bf;
        for (int t = b0; t < b1; t += bf_item) {
          add(1, t, std::min(b1, t + bf_item), part == 0 ? kDepNone : kDepRing);
          ++n_bf16;
        }
      }
      // INT2 pages, split where pages that this step's append writes begin
      for (int part = 0; part < 2; ++part) {
        const int p0 = part == 0 ? 0 : pg_new, p1 = part == 0 ? pg_new : np;
        for (int p = p0; p < p1; p += chunk) {
          add(0, p, std::min(p1, p + chunk), part == 0 ? kDepNone : kDepPages);
          max_pages = std::max(max_pages, std::min(p1, p + chunk) - p);
        }
      }
      for (size_t k = first; k < items.size(); ++k) items[k].head_count = int(items.size()) - first;
    }
    q.items_per_head = (int(items.size()) - q.first_item) / Hkv;
  }
  if (items.size() > c->lay.max_decode_items)
    return fail(OSCAR_ERR_INVALID_ARG, "plan of %zu items exceeds %zu; raise max_split_pages", items.size(),
                c->lay.max_decode_items);
  // the order CTAs take items in (when they are more than one wave): the items that wait
  // on no append task first, then those that may wait; largest first within each (stable)
  std::vector<int> order(items.size());
  for (size_t k = 0; k < items.size(); ++k) order[k] = int(k);
  auto cost = [&](const DecodeItem& d) {
    return d.kind == 0 ? (long long)(d.end - d.begin) * page_bytes : (long long)(d.end - d.begin) * 2LL * kHeadDim * 2;
  };
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) {
    const bool wa = items[a].dep != kDepNone, wb = items[b].dep != kDepNone;
    if (wa != wb) return wb;
    return cost(items[a]) > cost(items[b]);
  });
  int n_front = 0;
  while (n_front < int(order.size()) && items[order[n_front]].dep == kDepNone) ++n_front;
  Upload u;
  oscar_status st = begin_upload(c, &u);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the decode plan block, one copy: the items in the order CTAs take them, each with its
  // partial slot (its index above)
  const size_t items_off = decode_items_offset(c->cfg.max_requests);
  int32_t* counts = reinterpret_cast<int32_t*>(u.staging);
  counts[0] = int(items.size());
  counts[1] = n_req;
  counts[2] = n_front;
  counts[3] = 0;
  std::memcpy(u.staging + 256, reqs.data(), reqs.size() * sizeof(DecodeReq));
  DecodeItem* staged = reinterpret_cast<DecodeItem*>(u.staging + items_off);
  for (size_t k = 0; k < order.size(); ++k) {
    staged[k] = items[order[k]];
    staged[k].slot = order[k];
  }
  CUDA_TRY(cudaMemcpyAsync(c->base + c->lay.decode_plan, u.staging, items_off + items.size() * sizeof(DecodeItem),
                           cudaMemcpyHostToDevice, s));
  st = end_upload(c, u, s);
  if (st) return st;
  DecodeWorkspace w;
  size_t off = 0;
  w.partials = off;
  off = align256(off + items.size() * size_t(G) * (8 + 4 * kHeadDim));  // partial slots
  w.total = off;
  c->ws = w;
  c->dec_n_req = n_req;
  c->dec_items = int(items.size());
  c->dec_bf16_items = n_bf16;
  c->dec_max_pages = max_pages;
  c->planned = true;
  c->planned_with_reservation = c->reserved;
  c->dec_wide = wide;
  c->dec_folded = (flags & OSCAR_PLAN_FOLDED_ROTATIONS) != 0;
  c->plan_covers_reservation = c->reserved && n_reserved_planned == int(c->app_reqs.size());
  return OSCAR_OK;
}

size_t oscar_decode_workspace_bytes(const oscar_cache* c) { return (c && c->planned) ? c->ws.total : 0; }

size_t oscar_decode_workspace_max_bytes(const oscar_cache* c) {
  if (!c) return 0;
  const size_t G = size_t(c->cfg.n_q_heads / c->cfg.n_kv_heads);
  return align256(c->lay.max_decode_items * G * (8 + 4 * kHeadDim));
}

oscar_status oscar_plan_info(const oscar_cache* c, int* n_items, int* n_bf16_items, int* max_item_pages) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (!c->planned) return fail(OSCAR_ERR_STATE, "no decode plan");
  if (n_items) *n_items = c->dec_items;
  if (n_bf16_items) *n_bf16_items = c->dec_bf16_items;
  if (max_item_pages) *max_item_pages = c->dec_max_pages;
  return OSCAR_OK;
}

static oscar_status check_decode(oscar_cache* c, int layer, const void* q, void* out, void* ws, size_t ws_bytes) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (!c->planned) return fail(OSCAR_ERR_STATE, "no decode plan (plan after every append commit)");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(OSCAR_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (!q || !out || !ws) return fail(OSCAR_ERR_INVALID_ARG, "NULL q, out or workspace");
  if (reinterpret_cast<uintptr_t>(ws) % 256) return fail(OSCAR_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < c->ws.total) return fail(OSCAR_ERR_INVALID_ARG, "workspace %zu < %zu bytes", ws_bytes, c->ws.total);
  return OSCAR_OK;
}

oscar_status oscar_decode_attention(oscar_cache* c, int layer, const void* q, void* out, void* workspace, size_t ws_bytes,
                                    float* out_f32, void* stream) {
  g_launches = 0;
  oscar_status st = check_decode(c, layer, q, out, workspace, ws_bytes);
  if (st) return st;
  if (!is_int2(c)) return fail(OSCAR_ERR_STATE, "oscar_decode_attention needs the INT2 format");
  int e = launch_decode(kernel_params(c), layer, q, out, out_f32, static_cast<uint8_t*>(workspace), c->ws, c->dec_wide,
                        c->n_sm, stream, &g_launches);
  if (e) return fail(OSCAR_ERR_CUDA, "decode launch: %s", cudaGetErrorString(cudaError_t(e)));
  return OSCAR_OK;
}

oscar_status oscar_append_decode_attention(oscar_cache* c, int layer, const void* k_new, const void* v_new,
                                           const void* q, void* out, void* workspace, size_t ws_bytes, float* out_f32,
                                           void* stream) {
  g_launches = 0;
  oscar_status st = check_decode(c, layer, q, out, workspace, ws_bytes);
  if (st) return st;
  if (!is_int2(c)) return fail(OSCAR_ERR_STATE, "oscar_append_decode_attention needs the INT2 format");
  if (!c->reserved) return fail(OSCAR_ERR_STATE, "no reservation");
  if (!c->plan_covers_reservation)
    return fail(OSCAR_ERR_STATE, "plan the decode after the reservation, over every reserved slot");
  if (c->app_rows > 0 && (!k_new || !v_new)) return fail(OSCAR_ERR_INVALID_ARG, "NULL token arrays");
  // The append tasks run in the same wave as the decode when they fit in it; more of them
  // (long chunks, many requests) would hold back the decode, so those go to the append
  // kernel, which is launched first.
  const int G = c->cfg.n_q_heads / c->cfg.n_kv_heads;
  const int resident = decode_resident_ctas(G, c->cfg.group, c->dec_wide, is_cm(c), c->n_sm);
  const long long n_tasks =
      (long long)c->app_items * c->cfg.n_kv_heads * 2 * append_task_split(decode_warps(G, c->dec_wide));
  const bool fused = !is_cm(c) && n_tasks <= (long long)resident;
  if (!fused && c->app_items > 0) {
    int e = launch_append(kernel_params(c), layer, k_new, v_new, c->app_items, c->n_sm, stream, &g_launches);
    if (e) return fail(OSCAR_ERR_CUDA, "append launch: %s", cudaGetErrorString(cudaError_t(e)));
  }
  int e = launch_decode(kernel_params(c), layer, q, out, out_f32, static_cast<uint8_t*>(workspace), c->ws, c->dec_wide,
                        c->n_sm, stream, &g_launches, k_new, v_new, fused);
  if (e) return fail(OSCAR_ERR_CUDA, "append + decode launch: %s", cudaGetErrorString(cudaError_t(e)));
  return OSCAR_OK;
}

oscar_status oscar_bf16_decode_attention(oscar_cache* c, int layer, const void* q, void* out, void* workspace,
                                         size_t ws_bytes, float* out_f32, void* stream) {
  g_launches = 0;
  oscar_status st = check_decode(c, layer, q, out, workspace, ws_bytes);
  if (st) return st;
  if (is_int2(c)) return fail(OSCAR_ERR_STATE, "oscar_bf16_decode_attention needs the BF16 format");
  int e = launch_bf16_decode(kernel_params(c), layer, q, out, out_f32, static_cast<uint8_t*>(workspace), c->ws,
                             c->dec_wide, c->n_sm, stream, &g_launches);
  if (e) return fail(OSCAR_ERR_CUDA, "bf16 decode launch: %s", cudaGetErrorString(cudaError_t(e)));
  return OSCAR_OK;
}

oscar_status oscar_decode_attention_noalloc(oscar_cache* c, int layer, const void* q, void* out, float* out_f32,
                                            void* stream) {
  g_launches = 0;
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (!is_int2(c)) return fail(OSCAR_ERR_STATE, "oscar_decode_attention_noalloc needs the INT2 format");
  if (!c->planned) return fail(OSCAR_ERR_STATE, "no decode plan (plan after every append commit)");
  if (layer < 0 || layer >= c->cfg.n_layers) return fail(OSCAR_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (!q || !out) return fail(OSCAR_ERR_INVALID_ARG, "NULL q or out");
  int dev = -1;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return fail(OSCAR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(de));
  if (dev != c->device)
    return fail(OSCAR_ERR_INVALID_ARG, "current device %d is not the cache's device %d (the library scratch is looked "
                "up on the current device)", dev, c->device);
  bool too_big = false;
  int e = launch_decode_static_scratch(kernel_params(c), layer, q, out, out_f32, c->ws, c->dec_wide,
                                       c->n_sm, stream, &g_launches, &too_big);
  if (too_big)
    return fail(OSCAR_ERR_INVALID_ARG,
                "decode plan needs %zu bytes of scratch, more than the library's fixed %zu; use "
                "oscar_decode_attention with a caller workspace or plan fewer requests / larger splits",
                c->ws.total, static_scratch_bytes());
  if (e) return fail(OSCAR_ERR_CUDA, "decode launch (library scratch): %s", cudaGetErrorString(cudaError_t(e)));
  return OSCAR_OK;
}

size_t oscar_calibration_workspace_bytes(int n_tokens, int n_q_heads, int n_kv_heads) {
  if (n_tokens <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads) return 0;
  return calib_workspace(n_tokens, n_q_heads, n_kv_heads).total;
}

oscar_status oscar_calibrate_layer(const void* q, const void* k, const void* v, int n_tokens, int n_q_heads,
                                   int n_kv_heads, long long clip_rank, int rotation, float* R_K, float* R_V,
                                   float* clip_K, float* clip_V, double* covariances, void* workspace,
                                   size_t ws_bytes, void* stream) {
  g_launches = 0;
  if (!q || !k || !v || !R_K || !R_V || !clip_K || !clip_V || !workspace)
    return fail(OSCAR_ERR_INVALID_ARG, "NULL input, output or workspace");
  if (n_tokens <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads)
    return fail(OSCAR_ERR_INVALID_ARG, "bad shape: %d tokens, %d query heads, %d kv-heads", n_tokens, n_q_heads,
                n_kv_heads);
  if (rotation != OSCAR_ROTATION_OSCAR && rotation != OSCAR_ROTATION_HADAMARD)
    return fail(OSCAR_ERR_INVALID_ARG, "unknown rotation %d", rotation);
  if (clip_rank < 1 || clip_rank > (long long)n_tokens * kHeadDim)
    return fail(OSCAR_ERR_INVALID_ARG, "clip_rank %lld outside [1, %lld]", clip_rank, (long long)n_tokens * kHeadDim);
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(OSCAR_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  const size_t need = calib_workspace(n_tokens, n_q_heads, n_kv_heads).total;
  if (ws_bytes < need) return fail(OSCAR_ERR_INVALID_ARG, "calibration workspace of %zu bytes < %zu needed", ws_bytes, need);
  const int e = launch_calibrate(q, k, v, n_tokens, n_q_heads, n_kv_heads, long(clip_rank),
                                 rotation == OSCAR_ROTATION_HADAMARD, R_K, R_V, clip_K, clip_V, covariances,
                                 static_cast<uint8_t*>(workspace), stream, &g_launches);
  if (e) return fail(OSCAR_ERR_CUDA, "calibration launch: %s", cudaGetErrorString(cudaError_t(e)));
  return OSCAR_OK;
}

oscar_status oscar_set_wait_limit(oscar_cache* c, uint32_t counter_polls) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  c->counter_polls = counter_polls;
  return OSCAR_OK;
}

oscar_status oscar_inject_fault(oscar_cache* c, uint32_t faults) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  if (faults & ~uint32_t(OSCAR_FAULT_LOST_APPEND_SIGNAL)) return fail(OSCAR_ERR_INVALID_ARG, "unknown faults %#x", faults);
  c->inject |= faults;
  return OSCAR_OK;
}

oscar_status oscar_get_status(oscar_cache* c, void* stream, uint32_t* flags) {
  if (!c) return fail(OSCAR_ERR_INVALID_ARG, "cache is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemcpyAsync(c->h_status, c->base + c->lay.status, 4, cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  uint32_t f = c->h_status[0];
  if (flags) *flags = f;
  if (f) {
    CUDA_TRY(cudaMemsetAsync(c->base + c->lay.status, 0, 4, s));
    if (f & OSCAR_FLAG_TIMEOUT) {
      // a wait gave up: the append-dependency counters may be off by the signals that never
      // came (or came late), so they restart from zero (no launch of this cache is in flight:
      // the stream is synchronised and a cache has one launch at a time)
      CUDA_TRY(cudaMemsetAsync(c->base + c->lay.app_done, 0,
                               size_t(c->cfg.n_layers) * c->cfg.max_requests * c->cfg.n_kv_heads * 8, s));
      CUDA_TRY(cudaMemsetAsync(c->base + c->lay.counters, 0, size_t(c->cfg.max_requests) * c->cfg.n_kv_heads * 4, s));
    }
    CUDA_TRY(cudaStreamSynchronize(s));
    if (f & OSCAR_FLAG_TIMEOUT) return fail(OSCAR_ERR_TIMEOUT, "device flags 0x%x: a bounded wait gave up", f);
    return fail(OSCAR_ERR_BAD_PAGE, "device flags 0x%x: an out-of-range page or slot was skipped", f);
  }
  return OSCAR_OK;
}

}  // extern "C"
