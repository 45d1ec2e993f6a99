// Device side of quantize-on-append, shared by the append kernel and the fused
// append + decode kernel.
//
// OSCAR technical summary (gist.science), §2.2-B: sink (initial) and recent tokens stay
// BF16; history is stored INT2 after the fixed rotation and clipping (§2.2-A.3, A.4).
// Tokens leaving the BF16 recent window are evicted into INT2 here.
//
// One item (x one kv-head x {K, V}) per CTA at a time.  An item is either
//   kind 0: ring slots [s0, s0+16) of one request: first the old occupants that leave the
//           window are quantised from their stored bf16 value into INT2, then (after a
//           barrier) the new tokens that land in those slots are rotated and stored.  The
//           slot partition makes the read-before-overwrite order local to the CTA;
//   kind 1: up to 16 new positions that go straight to a sink or an INT2 row.
// The rotation r_j = bf16(sum_i R[i][j] x_i) is one fp32 fma chain per output in the
// order i = 0..127, so codes match the format bit for bit.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace append_dev {

constexpr int kTok = 16;   // tokens (or ring slots) per item
constexpr int kTokPer = 4;  // tokens per thread

// Threads of a CTA working on (part of) one item: thread (g, j) owns rotated channel j of
// tokens kTokPer g .. kTokPer g + kTokPer - 1, so NTH threads cover kTokPer NTH / 128
// tokens (512 threads: a whole item; 256: half an item).
template <int NTH>
struct AppendShape {
  static constexpr int kTokens = kTokPer * NTH / kHeadDim;
  static_assert(NTH % kHeadDim == 0 && kTokens <= kTok, "whole channel groups, at most one item");
};

struct Smem {
  float xs[kHeadDim][kTok];  // fp32 inputs, transposed: xs[i][t]
  uint32_t words[kTok][8];   // packed code rows being assembled
  float red_mn[kTok][4];
  float red_mx[kTok][4];
  // INT2 destinations of the item's tokens: [0] evicted ring tokens, [1] new tokens
  // (nullptr = token not quantised here or page id out of range)
  uint8_t* code_row[2][kTok];
  uint8_t* sz_row[2][kTok];
};

// Byte address of the INT2 row / sz entry of position p, or nullptr (flagged) if the page
// table entry is out of range.
struct RowPtr {
  uint8_t* code;
  uint8_t* sz;
};

// Physical page of position p of the request in `slot` (-1, flagged, if out of range).
__device__ inline int int2_page(const KernelParams& kp, int slot, int p) {
  const int lp = p / kPage;
  if (lp >= kp.max_pages_per_request) {
    flag(kp, OSCAR_FLAG_BAD_PAGE);
    return -1;
  }
  const int phys = reinterpret_cast<const int*>(kp.base + kp.lay.page_table)[size_t(slot) * kp.max_pages_per_request + lp];
  if (phys < 0 || phys >= kp.max_pages) {
    flag(kp, OSCAR_FLAG_BAD_PAGE);
    return -1;
  }
  return phys;
}

// INT2 row and sz entry of position p in physical page phys (nullptr if phys < 0).
__device__ inline RowPtr int2_row_at(const KernelParams& kp, int phys, int layer, int kvh, int kv, int p) {
  RowPtr r{nullptr, nullptr};
  if (phys < 0) return r;
  const int ng = kHeadDim / kp.group;
  const int t = p % kPage;
  r.code = kp.base + kp.lay.codes + size_t(layer) * kp.lay.codes_layer_stride + size_t(phys) * kp.lay.codes_page_stride +
           size_t(kvh) * kp.lay.codes_head_stride + size_t(kv) * (kPage * kRowBytes) + size_t(t) * kRowBytes;
  r.sz = kp.base + kp.lay.sz + size_t(layer) * kp.lay.sz_layer_stride + size_t(phys) * kp.lay.sz_page_stride +
         size_t(kvh) * kp.lay.sz_head_stride + size_t(kv) * (kPage * ng * 4) + size_t(t) * ng * 4;
  return r;
}

__device__ inline RowPtr int2_row(const KernelParams& kp, int slot, int layer, int kvh, int kv, int p) {
  return int2_row_at(kp, int2_page(kp, slot, p), layer, kvh, kv, p);
}

__device__ __forceinline__ uint16_t* ring_ptr(const KernelParams& kp, int slot, int layer, int kvh, int kv, int p) {
  return reinterpret_cast<uint16_t*>(kp.base + kp.lay.ring + size_t(slot) * kp.lay.ring_slot_stride +
                                     size_t(layer) * kp.lay.ring_layer_stride + size_t(kvh) * kp.lay.ring_head_stride +
                                     size_t(kv) * (size_t(kp.window) * kHeadDim * 2)) +
         size_t(p % kp.window) * kHeadDim;
}

__device__ __forceinline__ uint16_t* sink_ptr(const KernelParams& kp, int slot, int layer, int kvh, int kv, int p) {
  return reinterpret_cast<uint16_t*>(kp.base + kp.lay.sink + size_t(slot) * kp.lay.sink_slot_stride +
                                     size_t(layer) * kp.lay.sink_layer_stride + size_t(kvh) * kp.lay.sink_head_stride +
                                     size_t(kv) * (size_t(kp.n_sink) * kHeadDim * 2)) +
         size_t(p) * kHeadDim;
}

// Quantise the item's tokens t with a destination row in sm.code_row[which][t], whose
// clipped value for channel j is x[t] (thread j), and store codes and scale/zero.
// Format: per group s = bf16((max-min)/3), z = bf16(min), code = s == 0 ? 0 :
// clamp(rint((x - z) / s), 0, 3); channel c = 16f + 2w + h at bit 16h + 2f of word w.
template <int GROUP, int NTH>
__device__ void quantize_tokens(Smem& sm, const float (&x)[kTokPer], int which) {
  const int tid = threadIdx.x, j = tid & 127, tg = tid >> 7, warp = tid >> 5, lane = tid & 31;
  if (tid < kTok * 8) (&sm.words[0][0])[tid] = 0u;
  float mn[kTokPer], mx[kTokPer];
#pragma unroll
  for (int u = 0; u < kTokPer; ++u) {
    mn[u] = x[u];
    mx[u] = x[u];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mn[u] = fminf(mn[u], __shfl_xor_sync(0xffffffffu, mn[u], off));
      mx[u] = fmaxf(mx[u], __shfl_xor_sync(0xffffffffu, mx[u], off));
    }
    if (GROUP == 128 && lane == 0) {
      sm.red_mn[kTokPer * tg + u][warp & 3] = mn[u];
      sm.red_mx[kTokPer * tg + u][warp & 3] = mx[u];
    }
  }
  __syncthreads();
  const int f = j >> 4, w = (j & 15) >> 1, h = j & 1;
  const int shift = 16 * h + 2 * f;
#pragma unroll
  for (int u = 0; u < kTokPer; ++u) {
    const int t = kTokPer * tg + u;
    uint8_t* szr = sm.sz_row[which][t];
    if (!szr) continue;
    float gmn = mn[u], gmx = mx[u];
    if (GROUP == 128) {
      gmn = fminf(fminf(sm.red_mn[t][0], sm.red_mn[t][1]), fminf(sm.red_mn[t][2], sm.red_mn[t][3]));
      gmx = fmaxf(fmaxf(sm.red_mx[t][0], sm.red_mx[t][1]), fmaxf(sm.red_mx[t][2], sm.red_mx[t][3]));
    }
    const uint16_t sb = bf16_rne(__fdiv_rn(__fsub_rn(gmx, gmn), 3.0f));
    const uint16_t zb = bf16_rne(gmn);
    const float sc = bf16_f32(sb), z = bf16_f32(zb);
    uint32_t code = 0;
    if (sc != 0.0f) {
      const float q = __fdiv_rn(__fsub_rn(x[u], z), sc);
      code = static_cast<uint32_t>(fminf(fmaxf(rintf(q), 0.0f), 3.0f));
    }
    atomicOr(&sm.words[t][w], code << shift);
    if ((j % GROUP) == 0) reinterpret_cast<uint32_t*>(szr)[j / GROUP] = uint32_t(sb) | (uint32_t(zb) << 16);
  }
  __syncthreads();
  if (tid < kTok * 8) {
    const int t = tid >> 3, wd = tid & 7;
    uint8_t* cr = sm.code_row[which][t];
    if (cr) reinterpret_cast<uint32_t*>(cr)[wd] = sm.words[t][wd];
  }
  __syncthreads();
}

// One work item.  Every memory access of a token is independent of the other tokens'
// (positions are plain arithmetic on the item), so all loads of the 16 tokens are issued
// together; thread j only ever touches channel j of a ring slot, so reading an evicted
// token's value before writing the slot's new token needs no barrier.
// Per-thread state of one item between its two halves.
struct ItemState {
  AppendReq a;
  float clip;
  int ev[kTokPer], nw[kTokPer];
  float xe[kTokPer];
  bool ok;
};

// First half of an item: everything that does not depend on the preceding kernel in the
// stream (the plan and page table were uploaded before it; the ring tokens it evicts were
// written by this layer's previous append, long complete), so it may run before the PDL
// wait: positions, INT2 row pointers, evicted ring values.
template <int GROUP, int NTH>
__device__ void prepare_item(Smem& sm, const KernelParams& kp, int layer, const AppendItem& it, int kvh, int kv,
                             ItemState& st) {
  st.a = reinterpret_cast<const AppendReq*>(kp.base + kp.lay.append_reqs)[it.req];
  const AppendReq& a = st.a;
  const int tid = threadIdx.x, j = tid & 127, tg = tid >> 7;
  st.ok = a.slot >= 0 && a.slot < kp.max_requests;
  if (!st.ok) return;
  st.clip = reinterpret_cast<const float*>(kp.base + (kv ? kp.lay.clip_V : kp.lay.clip_K))[layer * kp.n_kv_heads + kvh];
  const int W = kp.window, S = kp.n_sink;
  const int e0 = a.H0, e1 = min(a.L0, a.H1);  // evicted ring positions
  const int n0 = max(a.L0, a.H1), n1 = a.L1;  // new ring positions
  // positions of item token t (-1 = none): evicted occupant and new token of slot / position t
  auto position = [&](int t, int which) -> int {
    if (t >= it.count) return -1;
    if (it.kind == 1) return which == 0 ? -1 : it.begin + t;
    const int s = it.begin + t;
    if (which == 0) {
      if (e1 <= e0) return -1;
      const int p = e0 + ((s - e0 % W) % W + W) % W;
      return p < e1 ? p : -1;
    }
    if (n1 <= n0) return -1;
    const int p = n0 + ((s - n0 % W) % W + W) % W;
    return p < n1 ? p : -1;
  };
  // INT2 row pointers, one thread per (token, evicted|new)
  if (tid < 2 * kTok) {
    const int t = tid & (kTok - 1), which = tid >> 4;
    const int p = position(t, which);
    const bool q = which == 0 ? p >= 0 : (p >= S && p < a.H1);
    RowPtr rp{nullptr, nullptr};
    if (q) rp = int2_row(kp, a.slot, layer, kvh, kv, p);
    sm.code_row[which][t] = rp.code;
    sm.sz_row[which][t] = rp.sz;
  }
#pragma unroll
  for (int u = 0; u < kTokPer; ++u) {
    st.ev[u] = position(kTokPer * tg + u, 0);
    st.nw[u] = position(kTokPer * tg + u, 1);
    st.xe[u] = st.ev[u] >= 0 ? bf16_f32(ring_ptr(kp, a.slot, layer, kvh, kv, st.ev[u])[j]) : 0.f;
  }
}

// Eviction: the ring tokens that leave the window go to INT2 from their stored bf16 value,
// clipped (read by prepare_item before this step's new tokens overwrite their slots).
// Needs only what prepare_item read, so it may run before the PDL wait as well (it writes
// INT2 rows of this layer at positions >= H0, which no kernel still running reads or
// writes).  All threads, after a barrier that follows prepare_item.
template <int GROUP, int NTH>
__device__ void evict_item(Smem& sm, const AppendItem& it, const ItemState& st) {
  const AppendReq& a = st.a;
  if (!st.ok || it.kind != 0 || min(a.L0, a.H1) <= a.H0) return;
  float xe[kTokPer];
#pragma unroll
  for (int u = 0; u < kTokPer; ++u) xe[u] = fmaxf(fminf(st.xe[u], st.clip), -st.clip);
  quantize_tokens<GROUP, NTH>(sm, xe, 0);
}

// Second half: new input rows (written by the caller, so after the PDL wait), rotation of
// the new tokens and their sink / ring rows, then new tokens that go straight to INT2.
// Thread j only ever touches channel j of a ring slot, so reading an evicted token's value
// (prepare_item) before writing the slot's new token needs no barrier.
template <int GROUP, int NTH, typename OnRowsWritten>
__device__ void finish_item(Smem& sm, const float* Rs, const KernelParams& kp, int layer, const AppendItem& it,
                            int kvh, int kv, ItemState& st, const uint16_t* __restrict__ k_new,
                            const uint16_t* __restrict__ v_new, OnRowsWritten on_rows_written) {
  const AppendReq& a = st.a;
  const int tid = threadIdx.x, j = tid & 127, tg = tid >> 7;
  if (!st.ok) {
    if (tid == 0) flag(kp, OSCAR_FLAG_BAD_SLOT);
    on_rows_written();
    return;
  }
  const uint16_t* X = kv ? v_new : k_new;
  const float clip = st.clip;
  const int S = kp.n_sink;
  float xn[kTokPer];
#pragma unroll
  for (int u = 0; u < kTokPer; ++u)
    xn[u] = st.nw[u] >= 0 ? bf16_f32(X[(size_t(a.x_offset + st.nw[u] - a.L0) * kp.n_kv_heads + kvh) * kHeadDim + j])
                          : 0.f;
#pragma unroll
  for (int u = 0; u < kTokPer; ++u) sm.xs[j][kTokPer * tg + u] = xn[u];
  __syncthreads();
  // ---- rotate my new tokens: one fixed-order fp32 fma chain per output channel; the
  // shared-memory loads of 16 steps are issued ahead of their FMAs
  float acc[kTokPer];
#pragma unroll
  for (int u = 0; u < kTokPer; ++u) acc[u] = 0.0f;
  const float* Rc = Rs + j;  // column j of R, in shared memory
  for (int i0 = 0; i0 < kHeadDim; i0 += 16) {
    float r[16];
    float4 x4[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      r[k] = Rc[(i0 + k) * kHeadDim];
      x4[k] = *reinterpret_cast<const float4*>(&sm.xs[i0 + k][kTokPer * tg]);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      acc[0] = __fmaf_rn(r[k], x4[k].x, acc[0]);
      acc[1] = __fmaf_rn(r[k], x4[k].y, acc[1]);
      acc[2] = __fmaf_rn(r[k], x4[k].z, acc[2]);
      acc[3] = __fmaf_rn(r[k], x4[k].w, acc[3]);
    }
  }
  // ---- route: sink / ring (bf16 r) or INT2 (clip + quantise)
  float xq[kTokPer];
  bool any_q = false;
#pragma unroll
  for (int u = 0; u < kTokPer; ++u) {
    const int p = st.nw[u];
    const uint16_t rb = bf16_rne(acc[u]);
    xq[u] = fmaxf(fminf(bf16_f32(rb), clip), -clip);
    if (p < 0) continue;
    if (p < S) {
      sink_ptr(kp, a.slot, layer, kvh, kv, p)[j] = rb;
    } else if (p >= a.H1) {
      ring_ptr(kp, a.slot, layer, kvh, kv, p)[j] = rb;
    } else {
      any_q = true;
    }
  }
  // the bf16 rows of the step are in place (all threads call this)
  on_rows_written();
  if (__syncthreads_or(any_q)) quantize_tokens<GROUP, NTH>(sm, xq, 1);
}

}  // namespace append_dev
}  // namespace oscar
