// Device helpers shared by the kernels of this library (sm_103a).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "oscar_internal.h"

namespace oscar {

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kSpinLimit = 1u << 26;  // bounded mbarrier wait (~seconds of polling)

__device__ __forceinline__ uint16_t bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fffu;
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}
__device__ __forceinline__ float bf16_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Programmatic dependent launch: wait for the preceding grid's completion / allow the
// next grid to start its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void flag(const KernelParams& kp, uint32_t bit) {
  atomicOr(reinterpret_cast<uint32_t*>(kp.base + kp.lay.status), bit);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// ---------------------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false if the copy did not land within kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }


// Launch with programmatic stream serialization (PDL) allowed.
template <typename Kern, typename... Args>
int launch_ex(Kern kernel, dim3 grid, dim3 block, size_t smem, void* stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return int(cudaLaunchKernelEx(&cfg, kernel, args...));
}

// Softmax attention of G query heads (fp32 q in shared memory, qs[G][d], already in the
// keys' basis) over bf16 token rows u in [begin, end), CUDA cores, 128 threads, 32
// tokens per round: warp w scores heads {w, w + 4} with lane = token; every thread then
// rebuilds the same running statistics from the stored logits and accumulates channel
// t of the values.  Writes the partial m (log2 units), l, o~[d] (unnormalised) per head.
template <int G, typename RowK, typename RowV>
__device__ void rows_attention(RowK rowK, RowV rowV, int begin, int end, const float* qs, float* part, uint8_t* smem) {
  float* lgs = reinterpret_cast<float*>(smem);  // [G][32]
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const float scale = kLog2e * rsqrtf(float(kHeadDim));
  float m_run[G], l_run[G], o[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
    o[h] = 0.f;
  }
  for (int u0 = begin; u0 < end; u0 += 32) {
    const int u = u0 + lane;
    const bool valid = u < end;
#pragma unroll
    for (int hh = 0; hh < G / 4; ++hh) {
      const int h = warp + 4 * hh;
      float s = 0.f;
      if (valid) {
        const uint4* kr = reinterpret_cast<const uint4*>(rowK(u));
#pragma unroll 4
        for (int v = 0; v < kHeadDim / 8; ++v) {
          const uint4 x = kr[v];
          const float* qh = qs + h * kHeadDim + 8 * v;
          s = fmaf(qh[0], bf16_lo(x.x), s);
          s = fmaf(qh[1], bf16_hi(x.x), s);
          s = fmaf(qh[2], bf16_lo(x.y), s);
          s = fmaf(qh[3], bf16_hi(x.y), s);
          s = fmaf(qh[4], bf16_lo(x.z), s);
          s = fmaf(qh[5], bf16_hi(x.z), s);
          s = fmaf(qh[6], bf16_lo(x.w), s);
          s = fmaf(qh[7], bf16_hi(x.w), s);
        }
      }
      lgs[h * 32 + lane] = valid ? s * scale : -INFINITY;
    }
    __syncthreads();
    const int n = min(32, end - u0);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float cm = -INFINITY;
      for (int k = 0; k < n; ++k) cm = fmaxf(cm, lgs[h * 32 + k]);
      const float mnew = fmaxf(m_run[h], cm);
      const float muse = mnew == -INFINITY ? 0.f : mnew;
      const float alpha = ex2(m_run[h] - muse);
      l_run[h] *= alpha;
      o[h] *= alpha;
      m_run[h] = mnew;
    }
    for (int k = 0; k < n; ++k) {
      const float v = bf16_f32(rowV(u0 + k)[t]);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float lg = lgs[h * 32 + k];
        const float p = lg == -INFINITY ? 0.f : ex2(lg - m_run[h]);
        l_run[h] += p;
        o[h] = fmaf(p, v, o[h]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float* ph = part + size_t(h) * (kHeadDim + 2);
    if (t == 0) {
      ph[0] = m_run[h];
      ph[1] = l_run[h];
    }
    ph[2 + t] = o[h];
  }
}

}  // namespace oscar
