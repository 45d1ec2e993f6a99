/*
 * oscar.h -- C ABI of a GB300 (sm_103a) library for the hot path of OSCAR-style 2-bit
 * KV-cache serving: quantize-on-append into a mixed-precision paged cache, and fused
 * split-K decode attention over it, plus an uncompressed BF16 paged cache used as the
 * comparison.
 *
 * The method: "기술 요약: OSCAR - 2 비트 KV 캐시 양자화를 위한 오프라인 스펙트럴 공분산
 * 인지 회전" (gist.science technical summary of OSCAR), referred to below as [OSCAR].
 *   [OSCAR] §2.2-A.3  composite rotations R_K = U_Q H_Had P_br, R_V = U_S H_Had P_br;
 *   [OSCAR] §2.2-A.4  per-layer clip thresholds on rotated activations;
 *   [OSCAR] §2.2-B    paged KV cache: sink (initial) and recent tokens in BF16, the
 *                     history in INT2 after the fixed rotation and clipping; a fused
 *                     kernel that unpacks, dequantises, inverse-rotates and attends over
 *                     the INT2 history, compatible with paged attention and prefix caching.
 * The tilnote.io note on OSCAR restates the same layout (sink and recent tokens BF16,
 * long history INT2, paged KV).
 *
 * Conventions (every call):
 *   - Plain C types only.  `stream` is a cudaStream_t passed as void* (NULL = legacy
 *     default stream).  Device pointers are marked [dev], host pointers [host].
 *   - The caller owns all memory.  The cache lives in one caller-allocated device block;
 *     the library sub-allocates it and never calls cudaMalloc after creation.  Decode
 *     scratch is a caller-provided device workspace.
 *   - Launching calls are asynchronous on `stream`.  Host-side validation happens before
 *     any launch and returns a status; nothing is launched on error.
 *   - Device-side faults never trap: a kernel that meets a page id or slot out of range
 *     skips that access and sets a bit in a device status word (oscar_get_status).
 *   - No C++ exception crosses this ABI.  oscar_last_error() gives a thread-local text.
 *   - A cache is not thread-safe; at most one append or decode of a cache may be in
 *     flight on the GPU at a time (they share plan buffers and merge counters).
 *
 * Stored format (bit-exact contract, identical for every layer):
 *   head_dim d = 128.  Rotated value of a token x: r = bf16_rne(R^T x), where
 *   r_j = bf16(acc_j) with acc_j = +0 then acc_j = fmaf(R[i][j], x_i, acc_j) for
 *   i = 0..127 ascending (fp32, no contraction changes).  R is row-major R[i][j].
 *   Per request and layer: positions [0, min(L, S)) are BF16 sinks (r); positions
 *   [S, H) are INT2 history; positions [H, L) are BF16 recent tokens (r) in ring slot
 *   p % W.  H starts at S; after an append that brings L to L', H' = max(H, L' - W).
 *   INT2 of a token: x = fmaxf(fminf(r, c), -c) with the (layer, kv-head, K|V) clip c;
 *   per group of `group` consecutive channels s = bf16((max x - min x) / 3.0f),
 *   z = bf16(min x); code = 0 if s == 0 else fminf(fmaxf(rintf((x - z) / s), 0), 3);
 *   dequantised value fmaf(code, s, z).  A 32-byte token row holds channel
 *   c = 16 f + 2 w + h at bit 32 w + 16 h + 2 f (word w little-endian, half h, field f).
 *
 * Device pools (byte offsets are exposed through oscar_cache_layout for tests):
 *   codes : [layer][phys_page][kv_head][K|V][64 tokens][32 B]   (token-major rows)
 *           format OSCAR_FORMAT_INT2_CM: the K block as above; the V block (2048 B) is
 *           channel-major: 32-bit word 128 b + c holds channel c of the page's tokens
 *           16 b .. 16 b + 15, token 16 b + 8 h + f at bit 16 h + 2 f (b 0..3, h 0..1,
 *           f 0..7).  Codes, scale and zero are the same numbers as in OSCAR_FORMAT_INT2.
 *   sz    : [layer][phys_page][kv_head][K|V][64 tokens][d/group][scale, zero] bf16
 *   sink  : [request_slot][layer][kv_head][K|V][S][d] bf16
 *   ring  : [request_slot][layer][kv_head][K|V][W][d] bf16
 *   bf16 pages (format OSCAR_FORMAT_BF16): [layer][phys_page][kv_head][K|V][64][d] bf16
 *   A logical page p of a request holds positions [64 p, 64 p + 64); physical page ids
 *   come from the request's page table and are shared by all layers, K and V.  INT2
 *   slots of positions outside [S, H) are never read and hold unspecified bytes.
 */
#ifndef OSCAR_H_
#define OSCAR_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OSCAR_OK = 0,
  OSCAR_ERR_INVALID_ARG = 1,  /* a size, index or pointer is out of the documented range */
  OSCAR_ERR_UNSUPPORTED = 2,  /* a shape the library has no kernel for */
  OSCAR_ERR_OUT_OF_PAGES = 3, /* the page pool cannot hold the reservation; nothing changed */
  OSCAR_ERR_BAD_PAGE = 4,     /* device: a page-table entry or slot out of range was skipped */
  OSCAR_ERR_CUDA = 5,         /* a CUDA runtime call failed (text in oscar_last_error) */
  OSCAR_ERR_TIMEOUT = 6,      /* device: a bounded wait on a copy gave up */
  OSCAR_ERR_STATE = 7         /* call order violated (e.g. append without a reservation) */
} oscar_status;

/* Device status word bits (oscar_get_status). */
#define OSCAR_FLAG_BAD_PAGE 0x1u
#define OSCAR_FLAG_TIMEOUT 0x2u
#define OSCAR_FLAG_BAD_SLOT 0x4u

/* OSCAR_FORMAT_INT2: INT2 history, token-major pages, decoded with warp-level MMAs; the
 * step's append can run inside the decode launch.  OSCAR_FORMAT_INT2_CM: the same stored
 * numbers with channel-major value pages, decoded on the tcgen05 tensor cores with the
 * code operands in tensor memory (GQA 4 or 8 at group 128, GQA 4 at group 32); the append
 * always runs as its own launch.  OSCAR_FORMAT_BF16: the uncompressed comparison cache. */
typedef enum { OSCAR_FORMAT_INT2 = 0, OSCAR_FORMAT_BF16 = 1, OSCAR_FORMAT_INT2_CM = 2 } oscar_format;

typedef struct {
  int format;                /* oscar_format */
  int head_dim;              /* must be 128 */
  int n_q_heads;             /* H_q */
  int n_kv_heads;            /* H_kv; H_q / H_kv must be 4 or 8 */
  int group;                 /* INT2 quantisation group along head_dim: 32 or 128 */
  int page;                  /* tokens per page: must be 64 */
  int n_sink;                /* S, 0..64 (INT2 format; BF16 format ignores it) */
  int window;                /* W, 0..1024 and a multiple of 16 (INT2 format) */
  int n_layers;              /* >= 1 */
  int max_requests;          /* request slots */
  int max_pages;             /* physical pages in the pool (shared by all layers) */
  int max_pages_per_request; /* page-table row length: max context = 64 * this */
} oscar_config;

typedef struct oscar_cache oscar_cache;

/* Byte offsets of the pools inside the device block, and their strides (for tests and
 * debugging dumps).  All offsets are multiples of 256. */
typedef struct {
  size_t codes, sz, sink, ring, bf16_pages;          /* pool offsets (0 if absent) */
  size_t codes_page_bytes, sz_page_bytes;            /* per (layer, page, kv-head), K then V */
  size_t bf16_page_bytes;                            /* per (layer, page, kv-head), K then V */
  size_t sink_bytes_per_head, ring_bytes_per_head;   /* per (slot, layer, kv-head), K then V */
  size_t page_table;                                 /* int32 [max_requests][max_pages_per_request] */
  size_t total;
} oscar_layout;

/* Device bytes a cache of this configuration needs (0 if the configuration is invalid). */
size_t oscar_cache_device_bytes(const oscar_config* cfg);

/* Create a cache inside `device_mem` [dev] of `bytes` (>= oscar_cache_device_bytes).
 * Zeroes the control words with cudaMemset (synchronous).  *out receives the handle. */
oscar_status oscar_cache_create(const oscar_config* cfg, void* device_mem, size_t bytes, oscar_cache** out);
void oscar_cache_destroy(oscar_cache* cache);
oscar_status oscar_cache_layout(const oscar_cache* cache, oscar_layout* out);

/* Rotation and clip inputs of one layer ([OSCAR] §2.2-A.3, A.4), produced offline:
 * R_K, R_V [host] fp32 [H_kv][d][d] row-major (orthogonal), clip_K, clip_V [host] fp32
 * [H_kv] (> 0, +inf allowed).  Copied to the device on `stream` before return.
 * Only the INT2 format uses them. */
oscar_status oscar_set_layer_params(oscar_cache* cache, int layer, const float* R_K, const float* R_V,
                                    const float* clip_K, const float* clip_V, void* stream);

/* Request slots.  alloc gives an empty request (L = 0).  free drops its page references. */
oscar_status oscar_request_alloc(oscar_cache* cache, int* slot);
oscar_status oscar_request_free(oscar_cache* cache, int slot);
/* Free physical pages of the pool and free request slots (host view; a page shared by
 * several requests is free once the last of them is freed).  Either pointer may be NULL. */
oscar_status oscar_cache_stats(const oscar_cache* cache, int* free_pages, int* free_slots);
/* Host view of a request: length L, history end H (INT2 format), pages mapped. */
oscar_status oscar_request_info(const oscar_cache* cache, int slot, int* length, int* history_end, int* n_pages);
/* Host copy of a request's page-table row (n entries). */
oscar_status oscar_request_pages(const oscar_cache* cache, int slot, int* pages, int n);

/* Prefix caching ([OSCAR] §2.2-B): the empty request `dst` takes the first `n_tokens`
 * tokens of `src` by sharing src's physical pages (reference counted), and copies src's
 * sink tokens for every layer on `stream`.  n_tokens must be a positive multiple of 64
 * and, in the INT2 format, at most src's history end H (those pages are never rewritten,
 * so no copy-on-write is needed); in the BF16 format at most 64 * floor(L_src / 64).
 * Afterwards dst has L = H = n_tokens. */
oscar_status oscar_request_share_prefix(oscar_cache* cache, int dst, int src, int n_tokens, void* stream);

/* Append, step 1 (host): reserve pages for `n_new[i]` more tokens of request `slots[i]`
 * [host arrays of n_req distinct slots], upload the changed page-table rows and the append
 * plan on `stream`.  The plan serves every layer until oscar_commit_append.  On
 * OSCAR_ERR_OUT_OF_PAGES nothing is reserved. */
oscar_status oscar_reserve(oscar_cache* cache, const int* slots, const int* n_new, int n_req, void* stream);

/* Append, step 2 (device, per layer): quantize-on-append of the reserved tokens of one
 * layer.  k_new, v_new [dev] bf16 [sum n_new][H_kv][d], requests in reservation order.
 * Rotates by R^T, routes each position to its sink, ring slot or INT2 row, evicts ring
 * tokens that leave the recent window into INT2, clips, quantises and packs. */
oscar_status oscar_quantize_append(oscar_cache* cache, int layer, const void* k_new, const void* v_new, void* stream);

/* Append, step 3 (host): the reserved tokens count as held (L, H advance). */
oscar_status oscar_commit_append(oscar_cache* cache);

/* Decode, step 1 (host): plan split-K decode of requests `slots` [host, n_req distinct]
 * at their current lengths, upload on `stream`.  The plan serves every layer until the
 * next plan or append commit.  max_split_pages > 0 caps the INT2 pages per work item
 * (0 = automatic, balanced over the SMs). */
oscar_status oscar_plan_decode(oscar_cache* cache, const int* slots, int n_req, int max_split_pages, void* stream);

/* oscar_plan_decode with plan flags (OSCAR_PLAN_*, or-ed).  OSCAR_PLAN_NARROW plans for
 * the 8-warp CTA shape (two CTAs per SM at GQA 4), which the automatic choice takes only
 * for steps larger than one wave of 16-warp CTAs; results are the same either way. */
#define OSCAR_PLAN_NARROW 0x1u
/* OSCAR_PLAN_FOLDED_ROTATIONS (INT2 formats): the model folds the rotations into its
 * projections ([OSCAR] §2.2-A.3 and B: R_K into the query projection, R_V into the output
 * projection), so the decode calls of this plan take q already rotated, q~ = R_K^T q (bf16,
 * same layout as q), and write o~, the output in the rotated basis (o = R_V o~ is left to
 * the model).  The stored cache is the same; only the two matrix-vector products at the
 * ends of the decode are skipped. */
#define OSCAR_PLAN_FOLDED_ROTATIONS 0x2u
oscar_status oscar_plan_decode_ex(oscar_cache* cache, const int* slots, int n_req, int max_split_pages, uint32_t flags,
                                  void* stream);

/* Decode workspace bytes for the current plan (0 without a plan). */
size_t oscar_decode_workspace_bytes(const oscar_cache* cache);

/* Decode workspace bytes that cover every plan of this cache (0 for NULL).  A launch
 * captured into a CUDA graph keeps the workspace pointer it was given, and a replay after
 * a later plan writes that plan's partial results through it: a workspace of this size
 * keeps such replays in bounds whatever the later plans are. */
size_t oscar_decode_workspace_max_bytes(const oscar_cache* cache);

/* Number of split-K work items of the current plan, and of them BF16 (sink/ring) items. */
oscar_status oscar_plan_info(const oscar_cache* cache, int* n_items, int* n_bf16_items, int* max_item_pages);

/* Decode, step 2 (device, per layer): fused decode attention over the mixed-precision
 * cache ([OSCAR] §2.2-B): q~ = R_K^T q per query head; scores q~.k / sqrt(d) in the
 * rotated basis over BF16 sinks, the BF16 recent window and the INT2 history (2-bit codes
 * unpacked and dequantised in registers); online softmax merged across splits;
 * out = R_V o~ (inverse rotation, once per head).
 * q [dev] bf16 [n_req][H_q][d] in plan order; out [dev] bf16 same shape; out_f32 [dev]
 * nullable fp32 copy of the output before bf16 rounding; workspace [dev] of ws_bytes.
 * A request with L = 0 gets zeros. */
oscar_status oscar_decode_attention(oscar_cache* cache, int layer, const void* q, void* out, void* workspace,
                                    size_t ws_bytes, float* out_f32, void* stream);

/* Quantize-append and decode in one launch (device, per layer): oscar_quantize_append of
 * the pending reservation's tokens for `layer` (same k_new / v_new layout) followed by
 * oscar_decode_attention of q over the cache that includes them, as a single kernel: the
 * append tasks run first and each decode work item waits only for the append tasks of
 * its own (request, kv-head) before it reads a ring or sink row or an INT2 page that the
 * append writes ([OSCAR] §2.2-B: quantize on append, then fused decode over the
 * mixed-precision cache; one launch per layer is this library's scheduling, not the
 * paper's).  When the reservation has more append work than one wave of decode CTAs
 * holds (long chunks, many requests), the call launches the append kernel and then the
 * decode kernel instead (oscar_last_launch_count tells which).  Requires a reservation
 * and a plan made after it that lists every reserved slot (OSCAR_ERR_STATE otherwise);
 * oscar_commit_append afterwards as usual.  Results are those of the two separate calls.
 * Waits are bounded: a wait that runs out sets OSCAR_FLAG_TIMEOUT. */
oscar_status oscar_append_decode_attention(oscar_cache* cache, int layer, const void* k_new, const void* v_new,
                                           const void* q, void* out, void* workspace, size_t ws_bytes,
                                           float* out_f32, void* stream);

/* Uncompressed comparison path (format OSCAR_FORMAT_BF16, same page tables and calls
 * for requests, reserve, commit and plan): append writes plain bf16 K and V rows into
 * pages; decode is softmax(q K^T / sqrt(d)) V over all L tokens, with no rotation. */
oscar_status oscar_bf16_append(oscar_cache* cache, int layer, const void* k_new, const void* v_new, void* stream);
oscar_status oscar_bf16_decode_attention(oscar_cache* cache, int layer, const void* q, void* out, void* workspace,
                                         size_t ws_bytes, float* out_f32, void* stream);

/* oscar_decode_attention without a caller workspace.  The paper has no counterpart:
 * this exists for callers that cannot allocate device memory themselves, for example a
 * plugin whose host framework owns every device allocation and gives it none, or a
 * serving loop that must not allocate once it is running, and so cannot supply the
 * decode workspace.  The scratch is instead a fixed 8 MiB array inside the library
 * (static device memory, held on every GPU that loads the library until exit).
 *   - Same semantics, inputs and outputs as oscar_decode_attention (q, out, out_f32).
 *   - Returns OSCAR_ERR_INVALID_ARG, launching nothing, when the current plan needs more
 *     than 8 MiB (oscar_decode_workspace_bytes tells the need).
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The current device must be the cache's device (the one current at
 *     oscar_cache_create): the array's address is looked up on the current device, on
 *     every call; OSCAR_ERR_INVALID_ARG otherwise.  The first call on a device also loads
 *     the library's device code there if nothing has yet; make that first call before any
 *     stream capture.
 *   - Every call, on every cache and stream, shares the one array and leaves its
 *     contents behind; nothing in it needs to start at zero.  Calls that overlap on the
 *     GPU race on it: order them on one stream or serialise them. */
oscar_status oscar_decode_attention_noalloc(oscar_cache* cache, int layer, const void* q, void* out, float* out_f32,
                                            void* stream);

/* Offline calibration of one layer on the GPU ([OSCAR] §2.2-A.1 to A.4), in fp64:
 *   A.1  C_Q = (1/(G N)) sum over tokens and the G query heads of each kv-head of q^T q;
 *        C_S = (1/(G N)) sum_h O_h^T O_h, O_h = causal softmax(Q_h K^T / sqrt(d)) V
 *        (the score-aware value target V^T S^T S V / N);
 *   A.2  eigenbases by cyclic Jacobi: eigenvalues descending, each eigenvector's first
 *        largest-magnitude entry positive;
 *   A.3  R_K = U_Q H_Had P_br, R_V = U_S H_Had P_br (H_Had the Sylvester matrix / sqrt(d),
 *        P_br sending e_j to e_rev(j)), rounded to fp32;
 *   A.4  clip = the clip_rank-th smallest of |x R| over the N tokens x d channels of each
 *        kv-head's keys (values), with R as rounded; a nearest-rank percentile p is
 *        clip_rank = ceil(p / 100 * N * d).
 * rotation OSCAR_ROTATION_HADAMARD skips A.1 and A.2 (U = I: the Hadamard-only rotation).
 * q [dev] bf16 [N][H_q][d], k and v [dev] bf16 [N][H_kv][d] (d = 128); outputs [dev]:
 * R_K, R_V fp32 [H_kv][d][d] row-major (the inputs of oscar_set_layer_params), clip_K,
 * clip_V fp32 [H_kv]; covariances [dev] nullable fp64 [2 H_kv][d][d] (C_Q of every
 * kv-head, then C_S; untouched in the Hadamard-only mode).  workspace [dev], 256-byte
 * aligned, of oscar_calibration_workspace_bytes (0 for a bad shape).  Asynchronous on
 * `stream`. */
#define OSCAR_ROTATION_OSCAR 0
#define OSCAR_ROTATION_HADAMARD 1
size_t oscar_calibration_workspace_bytes(int n_tokens, int n_q_heads, int n_kv_heads);
oscar_status oscar_calibrate_layer(const void* q, const void* k, const void* v, int n_tokens, int n_q_heads,
                                   int n_kv_heads, long long clip_rank, int rotation, float* R_K, float* R_V,
                                   float* clip_K, float* clip_V, double* covariances, void* workspace,
                                   size_t ws_bytes, void* stream);

/* Bounded waits: a work item of oscar_append_decode_attention that waits for the append
 * tasks it depends on gives up after `counter_polls` polls of their counter (each poll
 * sleeps about 0.1 us; 0 restores the default of 2^22 polls, about a second), sets
 * OSCAR_FLAG_TIMEOUT and carries on.  Applies to launches made after the call. */
oscar_status oscar_set_wait_limit(oscar_cache* cache, uint32_t counter_polls);

/* Host-side fault injection, for tests of the failure paths (nothing faults on the GPU).
 * OSCAR_FAULT_LOST_APPEND_SIGNAL: the next decode plan made while a reservation is pending
 * expects one more append signal for its first appending request than the append tasks
 * send, so that request's waits in oscar_append_decode_attention run out (a signal that
 * never arrives); the kernel returns with OSCAR_FLAG_TIMEOUT set.  One-shot. */
#define OSCAR_FAULT_LOST_APPEND_SIGNAL 0x1u
oscar_status oscar_inject_fault(oscar_cache* cache, uint32_t faults);

/* Synchronises `stream`, returns the device status word in *flags (OSCAR_FLAG_*) and
 * clears it.  Returns OSCAR_ERR_BAD_PAGE / OSCAR_ERR_TIMEOUT if a flag was set.  After a
 * timeout it also resets the cache's append-dependency and merge counters, so the next
 * step starts from a consistent state. */
oscar_status oscar_get_status(oscar_cache* cache, void* stream, uint32_t* flags);

/* Text of the last error on this thread ("" if none). */
const char* oscar_last_error(void);

/* Number of kernels the last launching call on this thread put on its stream. */
int oscar_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* OSCAR_H_ */
