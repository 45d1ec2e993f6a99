// Quantize-on-append into the mixed-precision paged cache, and the plain BF16 page append.
//
// OSCAR technical summary (gist.science), §2.2-B: sink (initial) and recent tokens stay
// BF16; history is stored INT2 after the fixed rotation and clipping (§2.2-A.3, A.4).
// Tokens leaving the BF16 recent window are evicted into INT2 here.
//
// One CTA = one work item x one kv-head x {K, V}; 128 threads, thread j owns rotated
// channel j.  An item is either
//   kind 0: ring slots [s0, s0+16) of one request: first the old occupants that leave the
//           window are quantised from their stored bf16 value into INT2, then (after a
//           barrier) the new tokens that land in those slots are rotated and stored.  The
//           slot partition makes the read-before-overwrite order local to the CTA;
//   kind 1: up to 16 new positions that go straight to a sink or an INT2 row.
// The rotation r_j = bf16(sum_i R[i][j] x_i) is one fp32 fma chain per output in the
// order i = 0..127, so codes match the format bit for bit.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr int kTok = 16;

struct Smem {
  float xs[kHeadDim][kTok];  // fp32 inputs, transposed: xs[i][t]
  uint32_t words[kTok][8];   // packed code rows being assembled
  float red_mn[kTok][4];
  float red_mx[kTok][4];
  int q_pos[kTok];  // positions to quantise into INT2 (this phase)
  int n_q;
};

// Byte address of the INT2 row / sz entry of position p, or nullptr (flagged) if the page
// table entry is out of range.
struct RowPtr {
  uint8_t* code;
  uint8_t* sz;
};

__device__ RowPtr int2_row(const KernelParams& kp, int slot, int layer, int kvh, int kv, int p) {
  const int lp = p / kPage;
  RowPtr r{nullptr, nullptr};
  if (lp >= kp.max_pages_per_request) {
    flag(kp, OSCAR_FLAG_BAD_PAGE);
    return r;
  }
  const int phys = reinterpret_cast<const int*>(kp.base + kp.lay.page_table)[size_t(slot) * kp.max_pages_per_request + lp];
  if (phys < 0 || phys >= kp.max_pages) {
    flag(kp, OSCAR_FLAG_BAD_PAGE);
    return r;
  }
  const int ng = kHeadDim / kp.group;
  const int t = p % kPage;
  r.code = kp.base + kp.lay.codes + size_t(layer) * kp.lay.codes_layer_stride + size_t(phys) * kp.lay.codes_page_stride +
           size_t(kvh) * kp.lay.codes_head_stride + size_t(kv) * (kPage * kRowBytes) + size_t(t) * kRowBytes;
  r.sz = kp.base + kp.lay.sz + size_t(layer) * kp.lay.sz_layer_stride + size_t(phys) * kp.lay.sz_page_stride +
         size_t(kvh) * kp.lay.sz_head_stride + size_t(kv) * (kPage * ng * 4) + size_t(t) * ng * 4;
  return r;
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

// Quantise sm.n_q tokens whose clipped value for channel j is x[t] (thread j), store
// codes and scale/zero.  Format: per group s = bf16((max-min)/3), z = bf16(min),
// code = s == 0 ? 0 : clamp(rint((x - z) / s), 0, 3); channel c = 16f + 2w + h at bit
// 16h + 2f of word w.
template <int GROUP>
__device__ void quantize_tokens(Smem& sm, const float (&x)[kTok], const KernelParams& kp, int slot, int layer, int kvh,
                                int kv) {
  const int j = threadIdx.x, warp = j >> 5, lane = j & 31;
  const int n = sm.n_q;
  if (j < kTok * 8) (&sm.words[0][0])[j] = 0u;
  float mn[kTok], mx[kTok];
#pragma unroll
  for (int t = 0; t < kTok; ++t) {
    mn[t] = x[t];
    mx[t] = x[t];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mn[t] = fminf(mn[t], __shfl_xor_sync(0xffffffffu, mn[t], off));
      mx[t] = fmaxf(mx[t], __shfl_xor_sync(0xffffffffu, mx[t], off));
    }
    if (GROUP == 128 && lane == 0) {
      sm.red_mn[t][warp] = mn[t];
      sm.red_mx[t][warp] = mx[t];
    }
  }
  __syncthreads();
  const int f = j >> 4, w = (j & 15) >> 1, h = j & 1;
  const int shift = 16 * h + 2 * f;
#pragma unroll
  for (int t = 0; t < kTok; ++t) {
    if (t >= n) break;
    float gmn = mn[t], gmx = mx[t];
    if (GROUP == 128) {
      gmn = fminf(fminf(sm.red_mn[t][0], sm.red_mn[t][1]), fminf(sm.red_mn[t][2], sm.red_mn[t][3]));
      gmx = fmaxf(fmaxf(sm.red_mx[t][0], sm.red_mx[t][1]), fmaxf(sm.red_mx[t][2], sm.red_mx[t][3]));
    }
    const uint16_t sb = bf16_rne(__fdiv_rn(__fsub_rn(gmx, gmn), 3.0f));
    const uint16_t zb = bf16_rne(gmn);
    const float s = bf16_f32(sb), z = bf16_f32(zb);
    uint32_t code = 0;
    if (s != 0.0f) {
      const float u = __fdiv_rn(__fsub_rn(x[t], z), s);
      code = static_cast<uint32_t>(fminf(fmaxf(rintf(u), 0.0f), 3.0f));
    }
    atomicOr(&sm.words[t][w], code << shift);
    if ((j % GROUP) == 0) {
      RowPtr rp = int2_row(kp, slot, layer, kvh, kv, sm.q_pos[t]);
      if (rp.sz) reinterpret_cast<uint32_t*>(rp.sz)[j / GROUP] = uint32_t(sb) | (uint32_t(zb) << 16);
    }
  }
  __syncthreads();
  if (j < kTok * 8) {
    const int t = j >> 3, wd = j & 7;
    if (t < n) {
      RowPtr rp = int2_row(kp, slot, layer, kvh, kv, sm.q_pos[t]);
      if (rp.code) reinterpret_cast<uint32_t*>(rp.code)[wd] = sm.words[t][wd];
    }
  }
  __syncthreads();
}

template <int GROUP>
__device__ void append_item(Smem& sm, const KernelParams& kp, int layer, const AppendItem& it,
                            const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new) {
  const AppendReq a = reinterpret_cast<const AppendReq*>(kp.base + kp.lay.append_reqs)[it.req];
  const int kvh = blockIdx.y, kv = blockIdx.z, j = threadIdx.x;
  if (a.slot < 0 || a.slot >= kp.max_requests) {
    if (j == 0) flag(kp, OSCAR_FLAG_BAD_SLOT);
    return;
  }
  const uint16_t* X = kv ? v_new : k_new;
  const size_t mat = size_t(kHeadDim) * kHeadDim;
  const float* R = reinterpret_cast<const float*>(kp.base + (kv ? kp.lay.R_V : kp.lay.R_K)) +
                   (size_t(layer) * kp.n_kv_heads + kvh) * mat;
  const float clip =
      reinterpret_cast<const float*>(kp.base + (kv ? kp.lay.clip_V : kp.lay.clip_K))[layer * kp.n_kv_heads + kvh];
  const int W = kp.window, S = kp.n_sink;

  // ---- phase 1 (ring items): old occupants of this item's slots leave the window -> INT2
  int rot_pos[kTok];  // new positions this CTA rotates; -1 = none
  int n_rot = 0;
  if (it.kind == 0) {
    const int e0 = a.H0, e1 = min(a.L0, a.H1);
    const int n0 = max(a.L0, a.H1), n1 = a.L1;
    int n_ev = 0;
    float x[kTok];
#pragma unroll
    for (int t = 0; t < kTok; ++t) x[t] = 0.f;
    for (int k = 0; k < it.count; ++k) {
      const int s = it.begin + k;
      if (e1 > e0) {
        const int p = e0 + ((s - e0 % W) % W + W) % W;
        if (p < e1) {
          if (j == 0) sm.q_pos[n_ev] = p;
          const float r = bf16_f32(ring_ptr(kp, a.slot, layer, kvh, kv, p)[j]);
#pragma unroll
          for (int t = 0; t < kTok; ++t)
            if (t == n_ev) x[t] = fmaxf(fminf(r, clip), -clip);
          ++n_ev;
        }
      }
      if (n1 > n0) {
        const int p = n0 + ((s - n0 % W) % W + W) % W;
        if (p < n1) rot_pos[n_rot++] = p;
      }
    }
    if (j == 0) sm.n_q = n_ev;
    __syncthreads();
    if (n_ev > 0) quantize_tokens<GROUP>(sm, x, kp, a.slot, layer, kvh, kv);
  } else {
    for (int k = 0; k < it.count; ++k) rot_pos[n_rot++] = it.begin + k;
  }
  for (int t = n_rot; t < kTok; ++t) rot_pos[t] = -1;
  if (n_rot == 0) return;

  // ---- phase 2: rotate the new tokens (fixed-order fp32 fma chain per output channel)
  for (int t = 0; t < kTok; ++t) {
    float v = 0.f;
    if (rot_pos[t] >= 0) {
      const size_t row = size_t(a.x_offset + rot_pos[t] - a.L0) * kp.n_kv_heads + kvh;
      v = bf16_f32(X[row * kHeadDim + j]);
    }
    sm.xs[j][t] = v;
  }
  __syncthreads();
  float acc[kTok];
#pragma unroll
  for (int t = 0; t < kTok; ++t) acc[t] = 0.0f;
  const float* Rc = R + j;
#pragma unroll 4
  for (int i = 0; i < kHeadDim; ++i) {
    const float rij = __ldg(Rc + size_t(i) * kHeadDim);
    const float4* xv = reinterpret_cast<const float4*>(&sm.xs[i][0]);
#pragma unroll
    for (int q = 0; q < kTok / 4; ++q) {
      const float4 x4 = xv[q];
      acc[4 * q + 0] = __fmaf_rn(rij, x4.x, acc[4 * q + 0]);
      acc[4 * q + 1] = __fmaf_rn(rij, x4.y, acc[4 * q + 1]);
      acc[4 * q + 2] = __fmaf_rn(rij, x4.z, acc[4 * q + 2]);
      acc[4 * q + 3] = __fmaf_rn(rij, x4.w, acc[4 * q + 3]);
    }
  }
  // ---- route: sink / ring (bf16 r) or INT2 (clip + quantise)
  float xq[kTok];
  int n_q = 0;
#pragma unroll
  for (int t = 0; t < kTok; ++t) xq[t] = 0.f;
#pragma unroll
  for (int t = 0; t < kTok; ++t) {
    const int p = rot_pos[t];
    if (p < 0) continue;
    const uint16_t rb = bf16_rne(acc[t]);
    if (p < S && p < a.H1) {
      sink_ptr(kp, a.slot, layer, kvh, kv, p)[j] = rb;
    } else if (p >= a.H1) {
      ring_ptr(kp, a.slot, layer, kvh, kv, p)[j] = rb;
    } else {
      const float r = bf16_f32(rb);
#pragma unroll
      for (int u = 0; u < kTok; ++u)
        if (u == n_q) xq[u] = fmaxf(fminf(r, clip), -clip);
      if (j == 0) sm.q_pos[n_q] = p;
      ++n_q;
    }
  }
  if (j == 0) sm.n_q = n_q;
  __syncthreads();
  if (n_q > 0) quantize_tokens<GROUP>(sm, xq, kp, a.slot, layer, kvh, kv);
}

template <int GROUP>
__global__ void __launch_bounds__(128) append_kernel(KernelParams kp, int layer, const uint16_t* __restrict__ k_new,
                                                     const uint16_t* __restrict__ v_new) {
  __shared__ Smem sm;
  pdl_wait();
  pdl_trigger();
  const int n_items = reinterpret_cast<const int*>(kp.base + kp.lay.plan_counts)[0];
  for (int ix = blockIdx.x; ix < n_items; ix += gridDim.x) {
    const AppendItem it = reinterpret_cast<const AppendItem*>(kp.base + kp.lay.append_items)[ix];
    append_item<GROUP>(sm, kp, layer, it, k_new, v_new);
    __syncthreads();  // shared memory is reused by the next item
  }
}

// Plain BF16 pages: copy K and V rows of new positions into [page][kvh][K|V][64][d].
__global__ void __launch_bounds__(128) bf16_append_kernel(KernelParams kp, int layer, const uint16_t* __restrict__ k_new,
                                                          const uint16_t* __restrict__ v_new) {
  pdl_wait();
  pdl_trigger();
  const int n_items = reinterpret_cast<const int*>(kp.base + kp.lay.plan_counts)[0];
  for (int ix = blockIdx.x; ix < n_items; ix += gridDim.x) {
  const AppendItem it = reinterpret_cast<const AppendItem*>(kp.base + kp.lay.append_items)[ix];
  const AppendReq a = reinterpret_cast<const AppendReq*>(kp.base + kp.lay.append_reqs)[it.req];
  const int kvh = blockIdx.y, kv = blockIdx.z;
  if (a.slot < 0 || a.slot >= kp.max_requests) {
    if (threadIdx.x == 0) flag(kp, OSCAR_FLAG_BAD_SLOT);
    continue;
  }
  const uint16_t* X = kv ? v_new : k_new;
  for (int e = threadIdx.x; e < it.count * 16; e += blockDim.x) {
    const int t = e >> 4, c16 = e & 15;
    const int p = it.begin + t;
    const int lp = p / kPage;
    if (lp >= kp.max_pages_per_request) {
      flag(kp, OSCAR_FLAG_BAD_PAGE);
      continue;
    }
    const int phys =
        reinterpret_cast<const int*>(kp.base + kp.lay.page_table)[size_t(a.slot) * kp.max_pages_per_request + lp];
    if (phys < 0 || phys >= kp.max_pages) {
      flag(kp, OSCAR_FLAG_BAD_PAGE);
      continue;
    }
    const size_t row = size_t(a.x_offset + p - a.L0) * kp.n_kv_heads + kvh;
    const uint4 v = reinterpret_cast<const uint4*>(X + row * kHeadDim)[c16];
    uint8_t* dst = kp.base + kp.lay.bf16_pages + size_t(layer) * kp.lay.bf16_layer_stride +
                   size_t(phys) * kp.lay.bf16_page_stride + size_t(kvh) * kp.lay.bf16_head_stride +
                   size_t(kv) * (kPage * kHeadDim * 2) + size_t(p % kPage) * (kHeadDim * 2);
    reinterpret_cast<uint4*>(dst)[c16] = v;
  }
  }
}

}  // namespace

int launch_append(const KernelParams& kp, int layer, const void* k_new, const void* v_new, int grid_x, void* stream,
                  int* launches) {
  dim3 grid(grid_x, kp.n_kv_heads, 2);
  const uint16_t* k = static_cast<const uint16_t*>(k_new);
  const uint16_t* v = static_cast<const uint16_t*>(v_new);
  int e = kp.group == 32 ? launch_ex(append_kernel<32>, grid, dim3(128), 0, stream, kp, layer, k, v)
                         : launch_ex(append_kernel<128>, grid, dim3(128), 0, stream, kp, layer, k, v);
  if (!e) *launches += 1;
  return e;
}

int launch_bf16_append(const KernelParams& kp, int layer, const void* k_new, const void* v_new, int grid_x,
                       void* stream, int* launches) {
  dim3 grid(grid_x, kp.n_kv_heads, 2);
  int e = launch_ex(bf16_append_kernel, grid, dim3(128), 0, stream, kp, layer, static_cast<const uint16_t*>(k_new),
                    static_cast<const uint16_t*>(v_new));
  if (!e) *launches += 1;
  return e;
}

}  // namespace oscar
