// Quantize-on-append into the mixed-precision paged cache, and the plain BF16 page append.
//
// One CTA = one work item x one kv-head x {K, V} (grid y, z); 512 threads: thread (g, j)
// owns rotated channel j of the item's tokens 4g..4g+3 (four token groups keep four warps
// per scheduler busy; one warp each left the kernel latency-bound).  The item logic is in
// append_dev.cuh.
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
constexpr int kAppendSmem = kRBytes + 16;

template <int GROUP>
__global__ void __launch_bounds__(kThreads) append_kernel(KernelParams kp, int layer, const uint16_t* __restrict__ k_new,
                                                     const uint16_t* __restrict__ v_new) {
  __shared__ Smem sm;
  extern __shared__ __align__(128) uint8_t dsm[];
  float* Rs = reinterpret_cast<float*>(dsm);
  uint64_t* bar = reinterpret_cast<uint64_t*>(dsm + kRBytes);
  const int kvh = blockIdx.y, kv = blockIdx.z;
  const float* R = reinterpret_cast<const float*>(kp.base + (kv ? kp.lay.R_V : kp.lay.R_K)) +
                   (size_t(layer) * kp.n_kv_heads + kvh) * kHeadDim * kHeadDim;
  const int n_items = reinterpret_cast<const int*>(kp.base + kp.lay.append_counts)[0];
  const bool work = int(blockIdx.x) < n_items;
  if (threadIdx.x == 0 && work) {
    mbar_init(smem_u32(bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_expect_tx(smem_u32(bar), kRBytes);
    bulk_g2s(smem_u32(Rs), R, kRBytes, smem_u32(bar));
  }
  ItemState st;
  AppendItem it{};
  if (work) {
    it = reinterpret_cast<const AppendItem*>(kp.base + kp.lay.append_items)[blockIdx.x];
    prepare_item<GROUP, kThreads>(sm, kp, layer, it, kvh, kv, st);
    __syncthreads();  // row pointers visible
    evict_item<GROUP, kThreads>(sm, it, st);
  }
  pdl_wait();
  pdl_trigger();
  if (!work) return;
  __syncthreads();  // barrier initialised
  if (!mbar_wait(smem_u32(bar), 0)) {
    if (threadIdx.x == 0) flag(kp, OSCAR_FLAG_TIMEOUT);
    mbar_wait(smem_u32(bar), 0);  // drain (bounded) before exit
    return;
  }
  for (int ix = blockIdx.x; ix < n_items; ix += gridDim.x) {
    if (ix != int(blockIdx.x)) {
      it = reinterpret_cast<const AppendItem*>(kp.base + kp.lay.append_items)[ix];
      prepare_item<GROUP, kThreads>(sm, kp, layer, it, kvh, kv, st);
      __syncthreads();
      evict_item<GROUP, kThreads>(sm, it, st);
    }
    finish_item<GROUP, kThreads>(sm, Rs, kp, layer, it, kvh, kv, st, k_new, v_new, [] {});
    __syncthreads();  // shared memory is reused by the next item
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

int launch_append(const KernelParams& kp, int layer, const void* k_new, const void* v_new, int grid_x, void* stream,
                  int* launches) {
  dim3 grid(grid_x, kp.n_kv_heads, 2);
  const uint16_t* k = static_cast<const uint16_t*>(k_new);
  const uint16_t* v = static_cast<const uint16_t*>(v_new);
  static bool attr = false;
  if (!attr) {
    int e = int(cudaFuncSetAttribute(append_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAppendSmem));
    if (!e) e = int(cudaFuncSetAttribute(append_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAppendSmem));
    if (e) return e;
    attr = true;
  }
  int e = kp.group == 32
              ? launch_ex(append_kernel<32>, grid, dim3(kThreads), size_t(kAppendSmem), stream, kp, layer, k, v)
              : launch_ex(append_kernel<128>, grid, dim3(kThreads), size_t(kAppendSmem), stream, kp, layer, k, v);
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
