// Quantize-on-append into the mixed-precision paged cache, and the plain BF16 page append.
//
// Standalone append: one CTA takes passes of four work items x one kv-head x {K, V}
// (grid y, z), loading R once; see append_kernel.  The item logic of the fused append tasks
// (inside the decode launch) is in append_dev.cuh; both follow the same format.
#include <cuda_runtime.h>

#include <cstdint>

#include "append_dev.cuh"
#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

using namespace append_dev;
constexpr int kThreads = 512;

// R of this CTA's (layer, kv-head, K|V) arrives in shared memory by one bulk copy, issued
// before the wait on the preceding kernel (R is written long before, by
// oscar_set_layer_params).
constexpr int kRBytes = kHeadDim * kHeadDim * 4;
constexpr int kGroupItems = 4;                 // items (16 tokens or ring slots each) per CTA pass
constexpr int kGroupTok = kGroupItems * kTok;  // 64: warp w owns tokens 4w .. 4w + 3 of them
constexpr int kXsBytes = kHeadDim * kGroupTok * 4;  // new tokens' values, transposed: xs[i][token]
constexpr int kAppendSmem = kRBytes + kXsBytes + 16;

// INT2 codes of one token from the clipped values of the calling lane's four channels
// (lane l holds channels 4l .. 4l + 3; all 32 lanes of the warp call it together), and the
// (scale, zero) word of the lane's group.  Format: per group s = bf16((max - min) / 3),
// z = bf16(min), code = s == 0 ? 0 : clamp(rint((x - z) / s), 0, 3).
template <int GROUP>
__device__ __forceinline__ uint32_t quantize4(const float (&x)[4], uint32_t (&code)[4]) {
  float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  // group of 128 channels: the whole warp; of 32: lanes 8G .. 8G + 7
#pragma unroll
  for (int off = GROUP == 128 ? 16 : 4; off > 0; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  const uint16_t sb = bf16_rne(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
  const uint16_t zb = bf16_rne(mn);
  const float sc = bf16_f32(sb), z = bf16_f32(zb);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    code[c] = sc != 0.0f ? static_cast<uint32_t>(fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(x[c], z), sc)), 0.0f), 3.0f))
                         : 0u;
  return uint32_t(sb) | (uint32_t(zb) << 16);
}

// Store the (scale, zero) word of the lane's group at dst.sz.
template <int GROUP>
__device__ __forceinline__ void store_sz(uint32_t szw, const RowPtr& dst) {
  const int lane = threadIdx.x & 31;
  if (dst.sz && (lane & (GROUP / 4 - 1)) == 0) reinterpret_cast<uint32_t*>(dst.sz)[lane / (GROUP / 4)] = szw;
}

// Token-major 32-byte row: channel c = 16f + 2w + h at bit 32w + 16h + 2f, so lane l's
// channels land in words 2(l & 3) and 2(l & 3) + 1, field l >> 2.
template <int GROUP>
__device__ __forceinline__ void quantize_row(const float (&x)[4], const RowPtr& dst) {
  const int lane = threadIdx.x & 31;
  uint32_t code[4];
  const uint32_t szw = quantize4<GROUP>(x, code);
  const int f = lane >> 2;
  uint32_t wa = (code[0] << (2 * f)) | (code[1] << (16 + 2 * f));
  uint32_t wb = (code[2] << (2 * f)) | (code[3] << (16 + 2 * f));
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {  // the eight lanes sharing (l & 3) hold the eight fields
    wa |= __shfl_xor_sync(0xffffffffu, wa, off);
    wb |= __shfl_xor_sync(0xffffffffu, wb, off);
  }
  if (!dst.code) return;
  if (lane < 4) reinterpret_cast<uint2*>(dst.code)[lane] = make_uint2(wa, wb);
  store_sz<GROUP>(szw, dst);
}

// Channel-major value codes (format OSCAR_FORMAT_INT2_CM): a page's V block holds, per
// 16-position block b and channel c, the 32-bit word 128 b + c with position 16 b + 8 h + f
// at bit 16 h + 2 f.  A pass gathers the words of each item's blocks in shared memory
// (an item's positions fall in at most two blocks: a ring item's slots wrap once, a
// direct item never leaves its block) and writes them once the pass is quantised.
struct CmAgg {
  uint32_t bits[kGroupItems][2][kHeadDim];
  uint32_t mask[kGroupItems][2];  // positions of the block this pass writes (2 bits each)
  int base[kGroupItems][2];       // first position of the block
  int slot[kGroupItems];
};
constexpr int kAppendSmemCm = kAppendSmem + int(sizeof(CmAgg));  // the CmAgg after the barrier
static_assert(kAppendSmem % 16 == 0, "CmAgg alignment");

// Add the lane's four codes of position p (item i of the pass) to the block words.
__device__ __forceinline__ void cm_add(CmAgg& ag, int i, int p, int W, const uint32_t (&code)[4]) {
  const int lane = threadIdx.x & 31;
  const int sel = W > 0 ? (p / W) & 1 : 0;  // the two blocks of a wrapping ring item lie W apart
  const int sh = 16 * ((p >> 3) & 1) + 2 * (p & 7);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (code[c]) atomicOr(&ag.bits[i][sel][4 * lane + c], code[c] << sh);
  if (lane == 0) {
    atomicOr(&ag.mask[i][sel], 3u << sh);
    ag.base[i][sel] = p & ~15;
  }
}

// INT2 codes of position p (in physical page phys, looked up beforehand): the token-major
// row, or (channel-major V) the pass's block words.
template <int GROUP>
__device__ __forceinline__ void store_int2(bool cm, CmAgg& ag, int item, int W, const float (&x)[4],
                                           const KernelParams& kp, int phys, int layer, int kvh, int kv, int p) {
  const RowPtr dst = int2_row_at(kp, phys, layer, kvh, kv, p);
  if (!cm) {
    quantize_row<GROUP>(x, dst);
    return;
  }
  uint32_t code[4];
  const uint32_t szw = quantize4<GROUP>(x, code);
  if (!dst.code) return;  // page id out of range (flagged)
  store_sz<GROUP>(szw, dst);
  cm_add(ag, item, p, W, code);
}

// Write the pass's block words of the V pages (all threads, after a barrier): a block the
// pass fills whole is stored, one it fills in part is merged with atomics (other positions
// of it belong to earlier steps or to another item of this launch).
__device__ void cm_write(CmAgg& ag, const KernelParams& kp, int layer, int kvh) {
  for (int e = threadIdx.x; e < kGroupItems * 2 * kHeadDim; e += kThreads) {
    const int c = e % kHeadDim, sel = (e / kHeadDim) & 1, i = e / (2 * kHeadDim);
    const uint32_t mask = ag.mask[i][sel];
    if (mask == 0u) continue;
    const uint32_t bits = ag.bits[i][sel][c];
    ag.bits[i][sel][c] = 0u;
    const int slot = ag.slot[i], p0 = ag.base[i][sel];
    if (slot < 0) continue;
    const int lp = p0 / kPage;  // a page out of range gave no codes (store_int2 flags it)
    if (lp >= kp.max_pages_per_request) continue;
    const int phys = reinterpret_cast<const int*>(kp.base + kp.lay.page_table)[size_t(slot) * kp.max_pages_per_request + lp];
    if (phys < 0 || phys >= kp.max_pages) continue;
    uint32_t* w = reinterpret_cast<uint32_t*>(kp.base + kp.lay.codes + size_t(layer) * kp.lay.codes_layer_stride +
                                              size_t(phys) * kp.lay.codes_page_stride +
                                              size_t(kvh) * kp.lay.codes_head_stride + kPage * kRowBytes) +
                  kHeadDim * ((p0 % kPage) / 16) + c;
    if (mask == 0xffffffffu) {
      *w = bits;
    } else {
      atomicAnd(w, ~mask);
      atomicOr(w, bits);
    }
  }
}

// Column of warp w's four tokens in row i of xs: the token groups are swizzled by row, so
// that the transposing stores of a warp (lane l writes rows 4l .. 4l + 3) spread over the
// banks; a row's four tokens stay one aligned 16-byte load.
__device__ __forceinline__ int xs_col(int i, int w) { return 4 * (w ^ ((i >> 2) & 7)); }

// Four bf16 values (8 bytes) as floats.
__device__ __forceinline__ void load4(const uint16_t* p, float (&v)[4]) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  v[0] = bf16_lo(w.x);
  v[1] = bf16_hi(w.x);
  v[2] = bf16_lo(w.y);
  v[3] = bf16_hi(w.y);
}

// Quantize-on-append, standalone launch: grid (CTA passes, kv-heads, K|V), 512 threads.
// Each pass takes kGroupItems consecutive work items of the reservation (any requests) for
// this CTA's (kv-head, K|V), whose R is loaded once: warp w takes item w / 4, tokens (or
// ring slots) 4(w % 4) .. + 3 of it; lane l owns rotated channels 4l .. 4l + 3, so a thread
// computes 16 outputs, each one fixed-order fp32 fma chain over i = 0..127 (bit-exact with
// the format), from two 16-byte shared-memory loads per four steps of four chains.
// Per item (format, OSCAR technical summary §2.2-B): ring slots first quantise their old
// occupants that leave the window into INT2 (from the stored bf16 value; before the wait
// on the preceding kernel, as nothing still running reads those rows), then the new
// tokens are rotated and routed to their sink, ring slot or INT2 row.  A lane reads an
// evicted token's channels before it writes the same channels of the slot's new token.
// CM: channel-major value pages (the V CTAs gather code words in shared memory, CmAgg).
template <int GROUP, bool CM>
__global__ void __launch_bounds__(kThreads) append_kernel(KernelParams kp, int layer, const uint16_t* __restrict__ k_new,
                                                     const uint16_t* __restrict__ v_new) {
  extern __shared__ __align__(128) uint8_t dsm[];
  float* Rs = reinterpret_cast<float*>(dsm);
  float* xs = reinterpret_cast<float*>(dsm + kRBytes);
  uint64_t* bar = reinterpret_cast<uint64_t*>(dsm + kRBytes + kXsBytes);
  CmAgg& ag = *reinterpret_cast<CmAgg*>(dsm + kAppendSmem);
  const int kvh = blockIdx.y, kv = blockIdx.z, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool cm = CM && kv == 1;
  if (cm) {
    for (int e = threadIdx.x; e < int(sizeof(CmAgg) / 4); e += kThreads) reinterpret_cast<uint32_t*>(&ag)[e] = 0u;
    __syncthreads();
  }
  const float* R = reinterpret_cast<const float*>(kp.base + (kv ? kp.lay.R_V : kp.lay.R_K)) +
                   (size_t(layer) * kp.n_kv_heads + kvh) * kHeadDim * kHeadDim;
  const int n_items = reinterpret_cast<const int*>(kp.base + kp.lay.append_counts)[0];
  const int n_pass = (n_items + kGroupItems - 1) / kGroupItems;
  const bool work = int(blockIdx.x) < n_pass;
  if (threadIdx.x == 0 && work) {
    mbar_init(smem_u32(bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_expect_tx(smem_u32(bar), kRBytes);
    bulk_g2s(smem_u32(Rs), R, kRBytes, smem_u32(bar));
  }
  const int S = kp.n_sink, W = kp.window;
  const uint16_t* X = kv ? v_new : k_new;
  bool waited = false, have_r = false;
  for (int pass = blockIdx.x; pass < n_pass; pass += gridDim.x) {
    // ---- this warp's item and its four token (slot) positions
    const int ix = pass * kGroupItems + warp / 4, t0 = 4 * (warp % 4);
    AppendItem it{0, 1, 0, 0};
    AppendReq a{-1, 0, 0, 0, 0, 0};
    if (ix < n_items) {
      it = reinterpret_cast<const AppendItem*>(kp.base + kp.lay.append_items)[ix];
      a = reinterpret_cast<const AppendReq*>(kp.base + kp.lay.append_reqs)[it.req];
    }
    const bool ok = ix < n_items && a.slot >= 0 && a.slot < kp.max_requests;
    if (ix < n_items && !ok && lane == 0) flag(kp, OSCAR_FLAG_BAD_SLOT);
    if (cm && warp % 4 == 0 && lane == 0) ag.slot[warp / 4] = ok ? a.slot : -1;
    const float clip =
        ok ? reinterpret_cast<const float*>(kp.base + (kv ? kp.lay.clip_V : kp.lay.clip_K))[layer * kp.n_kv_heads + kvh]
           : 0.f;
    const int e0 = a.H0, e1 = min(a.L0, a.H1);  // evicted ring positions
    const int n0 = max(a.L0, a.H1), n1 = a.L1;  // new ring positions
    int ev[4], nw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t0 + u;
      ev[u] = nw[u] = -1;
      if (!ok || t >= it.count) continue;
      if (it.kind == 1) {
        nw[u] = it.begin + t;
      } else {
        const int sl = it.begin + t;
        if (e1 > e0) {
          const int p = e0 + ((sl - e0 % W) % W + W) % W;
          if (p < e1) ev[u] = p;
        }
        if (n1 > n0) {
          const int p = n0 + ((sl - n0 % W) % W + W) % W;
          if (p < n1) nw[u] = p;
        }
      }
    }
    // the tokens' INT2 pages and the evicted values, all loads issued before any is used
    // (a token's stores would otherwise wait for the next token's loads)
    int phys_ev[4], phys_nw[4];
    uint2 evw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      phys_ev[u] = ev[u] >= 0 ? int2_page(kp, a.slot, ev[u]) : -1;
      phys_nw[u] = nw[u] >= S && nw[u] < a.H1 ? int2_page(kp, a.slot, nw[u]) : -1;
      evw[u] = ev[u] >= 0 ? *reinterpret_cast<const uint2*>(ring_ptr(kp, a.slot, layer, kvh, kv, ev[u]) + 4 * lane)
                          : make_uint2(0u, 0u);
    }
    // ---- eviction: old ring occupants leave the window into INT2
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (ev[u] < 0) continue;  // warp-uniform
      const float xe[4] = {fmaxf(fminf(bf16_lo(evw[u].x), clip), -clip), fmaxf(fminf(bf16_hi(evw[u].x), clip), -clip),
                           fmaxf(fminf(bf16_lo(evw[u].y), clip), -clip), fmaxf(fminf(bf16_hi(evw[u].y), clip), -clip)};
      store_int2<GROUP>(cm, ag, warp / 4, W, xe, kp, phys_ev[u], layer, kvh, kv, ev[u]);
    }
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    // ---- new tokens' inputs (written by the caller) into xs, transposed
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float xv[4] = {0.f, 0.f, 0.f, 0.f};
      if (nw[u] >= 0) load4(X + (size_t(a.x_offset + nw[u] - a.L0) * kp.n_kv_heads + kvh) * kHeadDim + 4 * lane, xv);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = 4 * lane + c;
        xs[i * kGroupTok + xs_col(i, warp) + u] = xv[c];
      }
    }
    __syncthreads();
    if (!have_r) {
      const bool r_ok = mbar_wait(smem_u32(bar), 0);
      if (__syncthreads_or(!r_ok)) {  // the same decision in every thread
        if (threadIdx.x == 0) flag(kp, OSCAR_FLAG_TIMEOUT);
        mbar_wait(smem_u32(bar), 0);  // drain (bounded) before exit
        return;
      }
      have_r = true;
    }
    // ---- rotation: acc[u][c] = sum_i R[i][4l + c] x_u[i], i ascending
    float acc[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[u][c] = 0.0f;
    const float* rrow = Rs + 4 * lane;
#pragma unroll 8
    for (int i = 0; i < kHeadDim; ++i) {
      const float4 xv = *reinterpret_cast<const float4*>(xs + i * kGroupTok + xs_col(i, warp));
      const float4 rv = *reinterpret_cast<const float4*>(rrow + i * kHeadDim);
      const float xu[4] = {xv.x, xv.y, xv.z, xv.w}, rc[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[u][c] = __fmaf_rn(rc[c], xu[u], acc[u][c]);
    }
    // ---- route: sink / ring (bf16 r) or INT2 (clip + quantise)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int p = nw[u];
      if (p < 0) continue;  // warp-uniform
      uint16_t rb[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) rb[c] = bf16_rne(acc[u][c]);
      if (p < S || p >= a.H1) {
        uint16_t* row = p < S ? sink_ptr(kp, a.slot, layer, kvh, kv, p) : ring_ptr(kp, a.slot, layer, kvh, kv, p);
        *reinterpret_cast<uint2*>(row + 4 * lane) =
            make_uint2(uint32_t(rb[0]) | (uint32_t(rb[1]) << 16), uint32_t(rb[2]) | (uint32_t(rb[3]) << 16));
      } else {
        float xq[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) xq[c] = fmaxf(fminf(bf16_f32(rb[c]), clip), -clip);
        store_int2<GROUP>(cm, ag, warp / 4, W, xq, kp, phys_nw[u], layer, kvh, kv, p);
      }
    }
    __syncthreads();  // xs is refilled by the next pass
    if (cm) {
      cm_write(ag, kp, layer, kvh);
      __syncthreads();
      if (threadIdx.x < kGroupItems * 2) (&ag.mask[0][0])[threadIdx.x] = 0u;
      __syncthreads();
    }
  }
  if (work && !have_r) mbar_wait(smem_u32(bar), 0);  // (no pass ran) the copy lands before exit
  if (!waited) {
    pdl_wait();
    pdl_trigger();
  }
}

// Plain BF16 pages: copy K and V rows of new positions into [page][kvh][K|V][64][d].
__global__ void __launch_bounds__(128) bf16_append_kernel(KernelParams kp, int layer, const uint16_t* __restrict__ k_new,
                                                          const uint16_t* __restrict__ v_new) {
  pdl_wait();
  pdl_trigger();
  const int n_items = reinterpret_cast<const int*>(kp.base + kp.lay.append_counts)[0];
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

int launch_append(const KernelParams& kp, int layer, const void* k_new, const void* v_new, int n_items, int n_sm,
                  void* stream, int* launches) {
  // passes of kGroupItems items; at most one wave of resident CTAs, each looping over passes
  const int passes = (n_items + kGroupItems - 1) / kGroupItems;
  const int per_head = (2 * n_sm + 2 * kp.n_kv_heads - 1) / (2 * kp.n_kv_heads);  // two CTAs per SM
  dim3 grid(passes < per_head ? passes : per_head, kp.n_kv_heads, 2);
  const uint16_t* k = static_cast<const uint16_t*>(k_new);
  const uint16_t* v = static_cast<const uint16_t*>(v_new);
  static bool attr = false;
  if (!attr) {
    int e = int(cudaFuncSetAttribute(append_kernel<32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAppendSmem));
    if (!e)
      e = int(cudaFuncSetAttribute(append_kernel<128, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAppendSmem));
    if (!e)
      e = int(cudaFuncSetAttribute(append_kernel<32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAppendSmemCm));
    if (!e)
      e = int(cudaFuncSetAttribute(append_kernel<128, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAppendSmemCm));
    if (e) return e;
    attr = true;
  }
  const size_t smem = size_t(kp.v_cm ? kAppendSmemCm : kAppendSmem);
  int e;
  if (kp.v_cm)
    e = kp.group == 32 ? launch_ex(append_kernel<32, true>, grid, dim3(kThreads), smem, stream, kp, layer, k, v)
                       : launch_ex(append_kernel<128, true>, grid, dim3(kThreads), smem, stream, kp, layer, k, v);
  else
    e = kp.group == 32 ? launch_ex(append_kernel<32, false>, grid, dim3(kThreads), smem, stream, kp, layer, k, v)
                       : launch_ex(append_kernel<128, false>, grid, dim3(kThreads), smem, stream, kp, layer, k, v);
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
