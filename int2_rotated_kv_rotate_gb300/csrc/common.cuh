// Device helpers shared by the kernels of this library (sm_103a).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "oscar_internal.h"

namespace oscar {

constexpr float kLog2e = 1.4426950408889634f;

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
// The same, suspending the thread until the phase completes or `ns` nanoseconds pass (a
// waiting warp takes no issue slots).
__device__ __forceinline__ bool mbar_try_wait_for(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}
// Bounded wait: false if the phase did not complete within kWaitPolls suspensions of at
// most 1 ms each (about a second or two).
constexpr uint32_t kWaitPolls = 2048;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitPolls; ++i)
    if (mbar_try_wait_for(bar, parity, 1000000u)) return true;
  return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }


// Ampere-style 16-byte asynchronous copy global -> shared; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Wait until at most n (0..3) of this thread's committed cp.async groups are pending.
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  if (n >= 3) cp_async_wait<3>();
  else if (n == 2) cp_async_wait<2>();
  else if (n == 1) cp_async_wait<1>();
  else cp_async_wait<0>();
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Pull the 128-byte line holding p into L2.  A prefetch only warms the cache, which stays
// coherent with every later write, so it may be issued for data that the preceding kernel
// is still writing, before the wait on it; the data is loaded after the wait.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// bf16 x bf16 -> fp32 tensor-core MMA, m16n8k16, A row-major, B column-major.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
// Two floats as bf16 (round to nearest even), first in the low half (one conversion).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// x rounded to the nearest bf16 (even on ties), as fp32 (finite x: the splits below).
__device__ __forceinline__ float bf16_round(float x) { return __uint_as_float(pack_bf16(0.f, x) & 0xffff0000u); }

// ---------------------------------------------------------------- partial slots
// The partial of one work item for the G heads of its kv group: float2 (m, l) per head
// (m in log2 units, l the softmax denominator), then the normalised output o~ / l per head
// and channel in fp32 (0 where l = 0).  fp16 here was measured to exceed the output
// tolerance on large values (its error is relative to the value).
template <int G>
struct PartialSlot {
  static constexpr int kMlBytes = G * 8;
  static constexpr int kBytes = G * (8 + 4 * kHeadDim);
  static_assert(kBytes % 16 == 0, "slots are bulk-copied");
};

// Store head h, channel c of a partial (unnormalised o); c == 0 also stores (m, l).
template <int G>
__device__ __forceinline__ void store_slot(uint8_t* slot, int h, int c, float m, float l, float o) {
  if (c == 0) reinterpret_cast<float2*>(slot)[h] = make_float2(m, l);
  reinterpret_cast<float*>(slot + PartialSlot<G>::kMlBytes)[h * kHeadDim + c] = l > 0.f ? o / l : 0.f;
}

// ---------------------------------------------------------------- BF16 rows on tensor cores
// A chunk is 16 tokens per warp; its K and V rows are staged in shared memory, each row
// padded to 272 bytes so that ldmatrix reads of 8 rows hit 8 distinct bank groups.
constexpr int kRowPad = 272;
template <int NW, int NBUF>
struct Bf16Rows {
  static constexpr int kChunk = 16 * NW;                   // tokens per chunk
  static constexpr int kBufBytes = 2 * kChunk * kRowPad;   // K and V rows of one chunk
  static constexpr int kPtrBytes = 2 * 2 * kChunk * 8;     // row pointers of two chunks
  static constexpr int kSmemBytes = NBUF * kBufBytes + kPtrBytes;
};

// Row stride (floats) of a CTA's q / q~ staging: the 4 heads of an MMA n-tile fall in
// different banks.
constexpr int kQRow = kHeadDim + 4;

// Softmax attention of G query heads over bf16 token rows u in [begin, end) (row pointers
// from rowK(u), rowV(u): 128 bf16 channels each), CTA of NW warps.  qg is fp32 [G][128]
// (shared, rows kQRow floats apart).  Chunks of 16 NW tokens are staged by cp.async
// (zero-filled past `end`) into NBUF buffers (2 = double buffered); warp w takes tokens
// 16w..16w+15 of each chunk.  Scores and values use mma.sync bf16 with q split into bf16 hi + lo columns
// (4 heads per n-tile) and p split the same way, so both products keep ~16 significant
// bits.  The first `staged` tokens may have been copied already (bf16_prestage; at most the
// chunks in flight before the first is attended, max(NBUF - 1, 1) of them); before_rest()
// runs (all threads) before the rest of them is copied.  Writes the
// partial slot (PartialSlot<G>) at part.  smem must hold
// Bf16Rows<NW, NBUF>::kSmemBytes and NW * G * (d + 2) floats (the two may alias).
// Issue the cp.async copies of the rows of tokens [begin, upto) in bf16_rows_mma<.., NBUF>'s
// layout (upto <= begin + max(NBUF - 1, 1) chunks: those that the first chunk's attention
// finds in flight), as one commit group: rows that may be copied early (before the wait on
// the preceding kernel).
template <int NW, int NBUF = 1, typename RowK, typename RowV>
__device__ void bf16_prestage(RowK rowK, RowV rowV, int begin, int upto, uint8_t* smem) {
  constexpr int kChunkTok = Bf16Rows<NW, NBUF>::kChunk;
  constexpr int kAhead = NBUF > 1 ? NBUF - 1 : 1;
  const int t = threadIdx.x, seg = t & 15;
  for (int c = 0; c < kAhead && begin + c * kChunkTok < upto; ++c) {
    const uint32_t buf = smem_u32(smem) + (c % NBUF) * Bf16Rows<NW, NBUF>::kBufBytes;
    for (int k = 0; k < 16; ++k) {
      const int row = (t >> 4) + 2 * NW * k;  // K rows then V rows
      const int u = begin + c * kChunkTok + (row & (kChunkTok - 1));
      if (u < upto) {
        const uint16_t* src = row < kChunkTok ? rowK(u) : rowV(u);
        cp_async16(buf + row * kRowPad + seg * 16, src + seg * 8, 16u);
      }
    }
  }
  cp_async_commit();
}

template <int G, int NW, int NBUF, typename RowK, typename RowV, typename BeforeRest>
__device__ void bf16_rows_mma(RowK rowK, RowV rowV, int begin, int end, const float* qg, uint8_t* part, uint8_t* smem,
                              int staged, BeforeRest before_rest) {
  constexpr int NT = G / 4;
  using B = Bf16Rows<NW, NBUF>;
  constexpr int kChunkTok = B::kChunk;
  constexpr int kBf16BufBytes = B::kBufBytes;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, gid = lane >> 2, tig = lane & 3;
  const float scale = kLog2e * rsqrtf(float(kHeadDim));
  // B fragments of q (k = channels 16kc + 2tig.., n = gid -> head 4j + gid/2, hi or lo)
  uint32_t bq[8][NT][2];
#pragma unroll
  for (int kc = 0; kc < 8; ++kc)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int head = 4 * j + (gid >> 1);
      const bool lo = gid & 1;
      const float* qh = qg + head * kQRow + 16 * kc + 2 * tig;
      float v[4] = {qh[0], qh[1], qh[8], qh[9]};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float hi = bf16_round(v[e]);
        v[e] = lo ? v[e] - hi : hi;
      }
      bq[kc][j][0] = pack_bf16(v[0], v[1]);
      bq[kc][j][1] = pack_bf16(v[2], v[3]);
    }
  float m_run[NT], l_part[NT], oacc[8][NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    m_run[j] = -INFINITY;
    l_part[j] = 0.f;
#pragma unroll
    for (int f = 0; f < 8; ++f)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[f][j][e] = 0.f;
  }
  const uint32_t sbase = smem_u32(smem);
  const int n_chunks = end > begin ? (end - begin + kChunkTok - 1) / kChunkTok : 0;
  // stage chunk c into buffer c & 1: thread t copies 16-byte segment (t & 15) of rows t/16 + 8k
  // row pointers of chunk c (thread t: row t, K rows then V rows; null past `end`), two
  // chunks' worth so that filling the next never races with issuing the current
  const uint16_t** rptr = reinterpret_cast<const uint16_t**>(smem + NBUF * kBf16BufBytes);
  static_assert(2 * kChunkTok == 32 * NW, "one row per thread");
  auto stage = [&](int c) {
    const uint16_t** rp = rptr + (c & 1) * 2 * kChunkTok;
    {
      const int tok = t & (kChunkTok - 1), u = begin + c * kChunkTok + tok;
      rp[t] = u < end ? (t < kChunkTok ? rowK(u) : rowV(u)) : nullptr;
    }
    __syncthreads();
    const uint32_t buf = sbase + (c % NBUF) * kBf16BufBytes;
    const int seg = t & 15;
    const uint16_t* any = rp[0];  // a valid row of the chunk (the chunk has one)
#pragma unroll 4
    for (int k = 0; k < 16; ++k) {
      const int row = (t >> 4) + 2 * NW * k;  // K rows then V rows
      if (c * kChunkTok + (row & (kChunkTok - 1)) < staged) continue;  // copied already
      const uint16_t* src = rp[row];
      cp_async16(buf + row * kRowPad + seg * 16, (src ? src : any) + seg * 8, src ? 16u : 0u);
    }
    cp_async_commit();
  };
  before_rest();
  // NBUF buffers: chunks c + 1 .. c + NBUF - 1 are in flight while chunk c is computed
  constexpr int kAhead = NBUF > 1 ? NBUF - 1 : 0;
  if (n_chunks > 0) stage(0);
  for (int c = 1; c < kAhead && c < n_chunks; ++c) stage(c);
  for (int c = 0; c < n_chunks; ++c) {
    if (NBUF > 1 && c + kAhead < n_chunks) stage(c + kAhead);  // into the buffer chunk c - 1 left
    cp_async_wait_upto(min(kAhead, n_chunks - 1 - c));       // chunk c has landed
    __syncthreads();
    const uint32_t kb = sbase + (c % NBUF) * kBf16BufBytes;
    const uint32_t vb = kb + kChunkTok * kRowPad;
    // ---- scores of my 16 tokens
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    {
      const int i = lane >> 3, r = lane & 7;
      const uint32_t a_row = kb + (16 * warp + (i & 1) * 8 + r) * kRowPad + (i >> 1) * 16;
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4(a_row + kc * 32, a0, a1, a2, a3);
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_bf16_16816(acc[j], a0, a1, a2, a3, bq[kc][j][0], bq[kc][j][1]);
      }
    }
    const int u0 = begin + c * kChunkTok + 16 * warp + gid, u1 = u0 + 8;
    float lg[NT][2], alpha[NT], muse[NT];
    bool rescale = false;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      lg[j][0] = u0 < end ? (acc[j][0] + acc[j][1]) * scale : -INFINITY;
      lg[j][1] = u1 < end ? (acc[j][2] + acc[j][3]) * scale : -INFINITY;
      float mx = fmaxf(lg[j][0], lg[j][1]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float mnew = fmaxf(m_run[j], mx);
      muse[j] = mnew == -INFINITY ? 0.f : mnew;
      alpha[j] = ex2(m_run[j] - muse[j]);
      rescale |= mnew > m_run[j];
      m_run[j] = mnew;
    }
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        l_part[j] *= alpha[j];
#pragma unroll
        for (int f = 0; f < 8; ++f)
#pragma unroll
          for (int e = 0; e < 4; ++e) oacc[f][j][e] *= alpha[j];
      }
    }
    // ---- P (bf16 hi, lo columns per head) as value-MMA B fragments
    uint32_t bp[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const float p0 = lg[j][0] == -INFINITY ? 0.f : ex2(lg[j][0] - muse[j]);
      const float p1 = lg[j][1] == -INFINITY ? 0.f : ex2(lg[j][1] - muse[j]);
      l_part[j] += p0 + p1;
      const float h0 = bf16_round(p0), h1 = bf16_round(p1);
      bp[j][0] = movmatrix_trans(pack_bf16(h0, p0 - h0));
      bp[j][1] = movmatrix_trans(pack_bf16(h1, p1 - h1));
    }
    // ---- values: A = V^T (16 channels x my 16 tokens) by ldmatrix.trans
    {
      const int i = lane >> 3, r = lane & 7;
      const uint32_t v_row = vb + (16 * warp + (i >> 1) * 8 + r) * kRowPad + (i & 1) * 16;
#pragma unroll
      for (int f = 0; f < 8; ++f) {
        uint32_t a0, a1, a2, a3;
        ldmatrix_x4_trans(v_row + f * 32, a0, a1, a2, a3);
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_bf16_16816(oacc[f][j], a0, a1, a2, a3, bp[j][0], bp[j][1]);
      }
    }
    __syncthreads();  // the buffer is refilled by the next stage()
    if (NBUF == 1 && c + 1 < n_chunks) stage(c + 1);
  }
  // ---- per-warp results -> shared memory, then merge the 4 warps into the partial
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    l_part[j] += __shfl_xor_sync(0xffffffffu, l_part[j], 4);
    l_part[j] += __shfl_xor_sync(0xffffffffu, l_part[j], 8);
    l_part[j] += __shfl_xor_sync(0xffffffffu, l_part[j], 16);
  }
  float* wres = reinterpret_cast<float*>(smem);  // [NW][G][2 + d], aliases the buffers
  float* mine = wres + size_t(warp) * G * (kHeadDim + 2);
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int head = 4 * j + tig;
    if (gid == 0) {
      mine[head * (kHeadDim + 2)] = m_run[j];
      mine[head * (kHeadDim + 2) + 1] = l_part[j];
    }
#pragma unroll
    for (int f = 0; f < 8; ++f) {
      mine[head * (kHeadDim + 2) + 2 + 16 * f + gid] = oacc[f][j][0] + oacc[f][j][1];
      mine[head * (kHeadDim + 2) + 2 + 16 * f + gid + 8] = oacc[f][j][2] + oacc[f][j][3];
    }
  }
  __syncthreads();
  for (int e = t; e < G * kHeadDim; e += 32 * NW) {
    const int h = e / kHeadDim, c = e % kHeadDim;
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) ms = fmaxf(ms, wres[(w * G + h) * (kHeadDim + 2)]);
    float l = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = wres[(w * G + h) * (kHeadDim + 2)];
      if (mw == -INFINITY) continue;
      const float a = ex2(mw - ms);
      l = fmaf(a, wres[(w * G + h) * (kHeadDim + 2) + 1], l);
      o = fmaf(a, wres[(w * G + h) * (kHeadDim + 2) + 2 + c], o);
    }
    store_slot<G>(part, h, c, ms, l, o);
  }
  __syncthreads();
}

// Counter increment that publishes the CTA's prior global writes and observes those of
// earlier incrementers: callers put a __syncthreads() before it (CTA-scope ordering of the
// other threads' writes, made cumulative by this gpu-scope release) and after it (so the
// acquire orders the whole CTA's later reads).
__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ---------------------------------------------------------------- merging partials
// Thread (c, hb) of an NTH-thread CTA owns channel c of heads hb, hb + NTH/128, ...
template <int G, int NTH>
struct MergeAcc {
  static constexpr int kStride = NTH / kHeadDim;
  static constexpr int HPT = G / kStride;
  static_assert(NTH % kHeadDim == 0 && G % kStride == 0, "thread count and group size");
  float M[HPT], L[HPT], O[HPT];  // running max (log2), sum of weights, weighted sum of o~ / l
};

// Online merge of n partial slots staged in shared memory into acc.
template <int G, int NTH>
__device__ void merge_slab(const uint8_t* slab, int n, MergeAcc<G, NTH>& acc) {
  using A = MergeAcc<G, NTH>;
  constexpr int S = PartialSlot<G>::kBytes;
  const int c = threadIdx.x & (kHeadDim - 1), hb = threadIdx.x / kHeadDim;
#pragma unroll
  for (int q = 0; q < A::HPT; ++q) {
    const int h = hb + A::kStride * q;
    float mx = acc.M[q];
    for (int i = 0; i < n; ++i) mx = fmaxf(mx, reinterpret_cast<const float2*>(slab + i * S)[h].x);
    if (mx == -INFINITY) continue;  // nothing but empty partials so far
    const float a = ex2(acc.M[q] - mx);  // acc.M = -inf gives 0
    float L = acc.L[q] * a, O = acc.O[q] * a;
#pragma unroll 4
    for (int i = 0; i < n; ++i) {
      const float2 ml = reinterpret_cast<const float2*>(slab + i * S)[h];
      if (ml.x == -INFINITY) continue;
      const float w = ex2(ml.x - mx) * ml.y;
      L += w;
      O = fmaf(w, reinterpret_cast<const float*>(slab + i * S + PartialSlot<G>::kMlBytes)[h * kHeadDim + c], O);
    }
    acc.M[q] = mx;
    acc.L[q] = L;
    acc.O[q] = O;
  }
}

// After the partial of item `it` is written, by every thread: the last CTA to finish an
// item of (request, kv-head) merges all of its partial slots into acc (true); the others
// return false.  on_last() runs (all threads) as soon as this CTA knows it merges.  The
// slots are bulk-copied into slab (shared, slab_slots of them per round) on the mbarrier
// slab_bar (phase tracked in slab_phase); waits are bounded.  s_flag: one int of shared
// memory.
template <int G, int NTH, typename OnLast>
__device__ bool merge_partial(const KernelParams& kp, const DecodeItem& it, const uint8_t* partials,
                              MergeAcc<G, NTH>& acc, int* s_flag, uint8_t* slab, int slab_slots, uint32_t slab_bar,
                              uint32_t& slab_phase, OnLast on_last) {
  constexpr int S = PartialSlot<G>::kBytes;
  fence_proxy_async();  // this thread's generic shared-memory accesses precede the bulk copies below
  __syncthreads();      // the partial is written (published by the release below)
  if (threadIdx.x == 0) {
    unsigned* hc = reinterpret_cast<unsigned*>(kp.base + kp.lay.counters) + size_t(it.req) * kp.n_kv_heads + it.kvh;
    const unsigned prev = atomic_add_acq_rel(hc, 1u);
    *s_flag = prev == unsigned(it.head_count - 1);
    if (*s_flag) *hc = 0u;  // every partial of (request, kv-head) has arrived
  }
  __syncthreads();
  if (!*s_flag) return false;
  on_last();
#pragma unroll
  for (int q = 0; q < MergeAcc<G, NTH>::HPT; ++q) {
    acc.M[q] = -INFINITY;
    acc.L[q] = 0.f;
    acc.O[q] = 0.f;
  }
  for (int base = 0; base < it.head_count; base += slab_slots) {
    const int n = min(slab_slots, it.head_count - base);
    if (threadIdx.x == 0) {
      fence_proxy_async();
      mbar_expect_tx(slab_bar, uint32_t(n * S));
      bulk_g2s(smem_u32(slab), partials + size_t(it.head_first + base) * S, uint32_t(n * S), slab_bar);
    }
    const bool ok = mbar_wait(slab_bar, slab_phase);
    if (!ok) {
      if (threadIdx.x == 0) flag(kp, OSCAR_FLAG_TIMEOUT);
      mbar_wait(slab_bar, slab_phase);  // drain (bounded) before the memory is reused
    }
    slab_phase ^= 1u;
    if (ok) merge_slab<G, NTH>(slab, n, acc);
    fence_proxy_async();
    __syncthreads();  // the slab is refilled by the next round
  }
  return true;
}

// Dynamic work distribution of a persistent-style decode grid: CTA b first takes position
// b (known before any wait, so its copies can be issued early), then the next free
// position gridDim.x + atomicAdd(work counter).  The last CTA to leave resets both counters
// for the next launch (launches of one cache never overlap).  A plan of at most one
// position per CTA uses neither counter.  Items are stored in the order they are taken
// (those that wait on no task first).  Call from all threads.
struct WorkQueue {
  unsigned* counters;  // [0] work, [1] exit
  int n_items;         // stored items
  int n_tasks;         // work ids 0 .. n_tasks - 1 that are not items (fused append tasks)
  int n_front;         // items that wait on no task (stored first)
  // One wave (every position has its own CTA): no counters, position b is CTA b's, tasks
  // first.  Several waves: the items that wait on nothing, the tasks, then the items that
  // wait on tasks, so that every task is handed out before any item that may wait on it.
  __device__ int n() const { return n_items + n_tasks; }
  __device__ bool one_wave() const { return n() <= int(gridDim.x); }
  // Work id of position p: a task t < n_tasks, or n_tasks + item index.
  __device__ int id_of(int p) const {
    if (p >= n()) return -1;
    if (one_wave() || p >= n_front + n_tasks) return p;
    if (p < n_front) return n_tasks + p;
    return p - n_front;
  }
  __device__ int first() const { return id_of(int(blockIdx.x)); }
  __device__ int next(int* s_slot) const {
    if (one_wave()) return -1;
    __syncthreads();
    if (threadIdx.x == 0) *s_slot = id_of(int(gridDim.x) + int(atomicAdd(&counters[0], 1u)));
    __syncthreads();
    return *s_slot;
  }
  __device__ void leave() const {
    if (one_wave()) return;
    if (threadIdx.x == 0) {
      __threadfence();  // this CTA's work-counter updates precede its exit
      if (atomicAdd(&counters[1], 1u) == gridDim.x - 1) {
        atomicExch(&counters[0], 0u);
        atomicExch(&counters[1], 0u);
      }
    }
  }
};

// Bounded wait (one thread) until *ctr >= expect, with acquire semantics: false after
// `polls` polls (kp.counter_polls; about a second by default).
__device__ __forceinline__ bool wait_counter(const unsigned* ctr, unsigned expect, uint32_t polls) {
  for (uint32_t i = 0; i < polls; ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= expect) return true;
    __nanosleep(128);
  }
  return false;
}

// Generic-proxy writes made visible to this thread (e.g. by an acquire) are ordered before
// its later async-proxy (bulk copy) reads of global memory.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

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

}  // namespace oscar
