// Uncompressed comparison: split-K decode attention over plain BF16 pages, no rotation.
// The pages' speed claims compare the INT2 kernel against BF16 decoding (OSCAR technical
// summary §4; the OScaR abstract compares against BF16 FlashDecoding-v2); this kernel is
// that comparison, on the same page tables and plans.
//
// Persistent-style grid: each CTA loops over work items (pages [p0, p1) of one (request,
// kv-head)); 64-token pages are staged by cp.async and attended with bf16 tensor-core
// MMAs (bf16_rows_mma); the last CTA of each (request, kv-head) merges the partials and
// stores bf16 (and optional fp32) output.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

// Row buffers of a CTA: chunks of 64 tokens, NBUF - 1 of them in flight while one is
// attended.  Plans of one wave (small steps, latency-bound) run the deeper pipeline
// (NBUF 3, two CTAs per SM); larger plans NBUF 2 (three CTAs per SM, more CTAs to overlap
// one another's prologues and merges).
template <int G, int NBUF>
constexpr int kBf16SlabSlots = Bf16Rows<4, NBUF>::kSmemBytes / PartialSlot<G>::kBytes;

template <int G, int NBUF>
__global__ void __launch_bounds__(128) bf16_split_kernel(KernelParams kp, int layer, const uint16_t* __restrict__ q,
                                                         uint8_t* __restrict__ partials, uint16_t* __restrict__ out,
                                                         float* __restrict__ out_f32) {
  extern __shared__ __align__(128) uint8_t smem[];
  float* qs = reinterpret_cast<float*>(smem + Bf16Rows<4, NBUF>::kSmemBytes);
  int* s_last_p = reinterpret_cast<int*>(smem + Bf16Rows<4, NBUF>::kSmemBytes + G * kQRow * 4);
  uint64_t* slab_bar = reinterpret_cast<uint64_t*>(smem + Bf16Rows<4, NBUF>::kSmemBytes + G * kQRow * 4 + 16);
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(slab_bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  uint32_t slab_phase = 0;
  // The plan and the page table were uploaded before the preceding kernels, and no kernel
  // of the step writes the rows below H_pre (the length before the step's append), so the
  // first item copies those of its first chunks before the wait on the preceding kernel.
  const int n_items = reinterpret_cast<const int*>(kp.base + kp.lay.decode_counts)[0];
  const WorkQueue wq{reinterpret_cast<unsigned*>(kp.base + kp.lay.sched), n_items, 0, n_items};
  int* s_next = s_last_p + 1;
  bool waited = false;
  for (int ix = wq.first(); ix >= 0; ix = wq.next(s_next)) {
    const DecodeItem it = reinterpret_cast<const DecodeItem*>(kp.base + kp.lay.decode_items)[ix];
    const DecodeReq dr = reinterpret_cast<const DecodeReq*>(kp.base + kp.lay.decode_reqs)[it.req];
    const size_t head0 = size_t(it.req) * kp.n_q_heads + size_t(it.kvh) * G;
    uint8_t* part = partials + size_t(it.slot) * PartialSlot<G>::kBytes;
    const bool slot_ok = dr.slot >= 0 && dr.slot < kp.max_requests;
    if (!slot_ok && threadIdx.x == 0) flag(kp, OSCAR_FLAG_BAD_SLOT);
    int t0 = 0, t1 = 0;
    if (slot_ok && it.kind == 0) {
      t0 = it.begin * kPage;
      t1 = min(it.end * kPage, dr.L);
    }
    const int* ptab =
        reinterpret_cast<const int*>(kp.base + kp.lay.page_table) + size_t(slot_ok ? dr.slot : 0) * kp.max_pages_per_request;
    const uint8_t* head_base = kp.base + kp.lay.bf16_pages + size_t(layer) * kp.lay.bf16_layer_stride +
                               size_t(it.kvh) * kp.lay.bf16_head_stride;
    // a bad page id reads page 0 of the pool instead and raises the flag
    auto page_of = [=](int u) -> const uint16_t* {
      int phys = ptab[u / kPage];
      if (phys < 0 || phys >= kp.max_pages) {
        flag(kp, OSCAR_FLAG_BAD_PAGE);
        phys = 0;
      }
      return reinterpret_cast<const uint16_t*>(head_base + size_t(phys) * kp.lay.bf16_page_stride);
    };
    auto rowK = [=](int u) { return page_of(u) + size_t(u % kPage) * kHeadDim; };
    auto rowV = [=](int u) { return page_of(u) + size_t(kPage + u % kPage) * kHeadDim; };
    int staged = 0;
    if (!waited) {
      if (threadIdx.x < 2 * G) prefetch_l2(q + head0 * kHeadDim + 64 * threadIdx.x);  // q's lines, loaded after the wait
      constexpr int kAheadTok = (NBUF > 1 ? NBUF - 1 : 1) * Bf16Rows<4, NBUF>::kChunk;
      const int upto = min(min(t1, dr.H_pre), t0 + kAheadTok);
      if (upto > t0) {
        bf16_prestage<4, NBUF>(rowK, rowV, t0, upto, smem);
        staged = upto - t0;
      }
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    for (int e = threadIdx.x; e < G * kHeadDim; e += 128) qs[(e / kHeadDim) * kQRow + e % kHeadDim] = bf16_f32(q[head0 * kHeadDim + e]);
    __syncthreads();
    bf16_rows_mma<G, 4, NBUF>(rowK, rowV, t0, t1, qs, part, smem, staged, [] {});

    MergeAcc<G, 128> acc;
    if (merge_partial<G, 128>(kp, it, partials, acc, s_last_p, smem, kBf16SlabSlots<G, NBUF>, smem_u32(slab_bar), slab_phase,
                              [] {})) {
      const int c = threadIdx.x;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float r = acc.L[h] > 0.f ? acc.O[h] / acc.L[h] : 0.f;
        out[(head0 + h) * kHeadDim + c] = bf16_rne(r);
        if (out_f32) out_f32[(head0 + h) * kHeadDim + c] = r;
      }
    }
    fence_proxy_async();  // generic use of the buffers is over before later bulk copies
  }
  if (!waited) {  // no item: the launch still orders itself after the preceding kernel
    pdl_wait();
    pdl_trigger();
  }
  wq.leave();
}

constexpr int kBf16KernelSmem(int G, int nbuf) {
  return (nbuf == 3 ? Bf16Rows<4, 3>::kSmemBytes : Bf16Rows<4, 2>::kSmemBytes) + G * kQRow * 4 + 32;  // + flags, barrier
}

template <int G, int NBUF>
int resident_ctas(int n_sm) {
  static int resident = 0;
  if (resident == 0) {
    int e = int(cudaFuncSetAttribute(bf16_split_kernel<G, NBUF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kBf16KernelSmem(G, NBUF)));
    int per_sm = 0;
    if (!e)
      e = int(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bf16_split_kernel<G, NBUF>, 128,
                                                            kBf16KernelSmem(G, NBUF)));
    if (e) return -e;
    resident = (per_sm > 0 ? per_sm : 1) * n_sm;
  }
  return resident;
}

template <int G, int NBUF>
int launch_t(const KernelParams& kp, int layer, const void* q, void* out, float* out_f32, uint8_t* ws,
             const DecodeWorkspace& wl, int n_sm, void* stream, int* launches) {
  uint8_t* partials = ws + wl.partials;
  const int resident = resident_ctas<G, NBUF>(n_sm);
  if (resident < 0) return -resident;
  const int grid = resident;  // persistent-style: CTAs loop over the plan's items
  int e = launch_ex(bf16_split_kernel<G, NBUF>, dim3(grid), dim3(128), size_t(kBf16KernelSmem(G, NBUF)), stream, kp,
                    layer, static_cast<const uint16_t*>(q), partials, static_cast<uint16_t*>(out), out_f32);
  if (!e) *launches += 1;
  return e;
}

}  // namespace

int bf16_decode_resident_ctas(int gqa, bool deep, int n_sm) {
  if (gqa == 4) return deep ? resident_ctas<4, 3>(n_sm) : resident_ctas<4, 2>(n_sm);
  if (gqa == 8) return deep ? resident_ctas<8, 3>(n_sm) : resident_ctas<8, 2>(n_sm);
  return n_sm;
}

int launch_bf16_decode(const KernelParams& kp, int layer, const void* q, void* out, float* out_f32, uint8_t* ws,
                       const DecodeWorkspace& wl, bool deep, int n_sm, void* stream, int* launches) {
  if (kp.gqa == 4)
    return deep ? launch_t<4, 3>(kp, layer, q, out, out_f32, ws, wl, n_sm, stream, launches)
                : launch_t<4, 2>(kp, layer, q, out, out_f32, ws, wl, n_sm, stream, launches);
  if (kp.gqa == 8)
    return deep ? launch_t<8, 3>(kp, layer, q, out, out_f32, ws, wl, n_sm, stream, launches)
                : launch_t<8, 2>(kp, layer, q, out, out_f32, ws, wl, n_sm, stream, launches);
  return int(cudaErrorInvalidValue);
}

}  // namespace oscar
