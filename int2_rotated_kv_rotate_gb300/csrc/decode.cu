// Fused split-K decode attention over the mixed-precision paged cache (INT2 format).
//
// OSCAR technical summary (gist.science), §2.2-B (kernel integration): one kernel
// unpacks and dequantises the INT2 history, works in the rotated basis and applies the
// inverse rotation, over paged KV with prefix sharing, without extra memory traffic.
//
// One launch per layer: split_kernel, a persistent-style grid whose CTAs take work items
// (plan): either INT2 pages [p0, p1) of one (request, kv-head), or BF16 sink/ring tokens.
// Each item first rotates its query heads, q~ = R_K^T q (fp32, R_K columns loaded into
// registers before the wait on the preceding kernel), then writes a partial (m, l, o~) in
// the rotated basis; the last CTA of each (request, kv-head) merges the partials
// (log-sum-exp), applies o = R_V o~ and stores bf16 (and optional fp32) output.
//
// INT2 page pipeline (per warp, no block barriers): lane 0 issues cp.async.bulk copies of
// the page's code block (K 2 KB + V 2 KB) and scale/zero block into a private ring of
// kStages shared-memory stages, completion on an mbarrier; waits are bounded.
//
// Tensor-core formulation (mma.sync m16n8k16, fp16 in, fp32 accumulate), per 16 tokens:
//   scores  S[t, n] = sum_c code_K[t, c] * B[c, n],  B = q~ (hi and lo fp16 halves as two
//           columns per head, so q~ keeps ~22 bits).  Scale and zero factor out per
//           (token, group): q~.k^ = s * (q~ . code) + z * sum(q~).
//   values  O[c, n] += sum_t code_V[c, t] * P'[t, n],  P' = p * s_V (fp16), and
//           sum_t p * z_V is added per group at the end.
// A 2-bit field masked in place (w & 0x00030003 << 2k) is an fp16 subnormal equal to
// code * 4^k * 2^-24; the power of two is folded into B (keys) or into the output scale
// (values), so one AND turns two codes into an MMA operand.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "append_dev.cuh"
#include "common.cuh"
#include "oscar_internal.h"
#include "tmem.cuh"

namespace oscar {
namespace {

constexpr int kStages = 2;  // page stages per warp
constexpr int kSpareSMs = 8;  // SMs a one-per-SM grid leaves free (see resident_ctas_t)

// CTA shape of the split kernel.  NW = 16 (GQA 4, plans of one wave): one CTA per SM, 128
// registers a thread fill the register file.  NW = 8: two CTAs per SM, also 128 registers
// a thread (plans of several waves, and every plan at GQA 8: one CTA streams while the
// other is between items).  Each channel of the q rotation has kParts threads, each summing
// 128 / kParts rows of R_K.
template <int NW_>
struct Shape {
  static constexpr int NW = NW_;
  static constexpr int NTH = 32 * NW;
  static constexpr int kParts = NTH / kHeadDim;
  static constexpr int kRows = kHeadDim / kParts;        // rows of R_K per thread
  static constexpr int kQinRow = kHeadDim + 4 * kParts;  // padded staging row of q
  static_assert(append_task_split(NW) * append_dev::AppendShape<NTH>::kTokens == append_dev::kTok,
                "append tasks cover an item");
};

// ---------------------------------------------------------------- MMA helpers
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
// max(a, b, c) in one instruction (a NaN operand is ignored, as by fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// 2-bit field f (0..7) of each 16-bit half of w, as fp16 code * 4^(f&3) * 2^-24.
__device__ __forceinline__ uint32_t field(uint32_t w, uint32_t w_shr8, int f) {
  const uint32_t m = 0x00030003u << (2 * (f & 3));
  return (f < 4 ? w : w_shr8) & m;
}

// Token order inside a 16-token block used by both MMAs: row m of the score tile (and
// k-index m of the value MMA) is token tau(m); this makes every shared-memory read below
// bank-conflict free.
__device__ __forceinline__ int tau8(int m) { return (m >> 1) + 4 * (m & 1); }

// ---------------------------------------------------------------- q rotation
// Thread t of a split CTA holds column c = t / kParts of R_K, rows kRows (t % kParts) ..
// + kRows - 1, so the parts of a column sit in neighbouring lanes (R_K is written long
// before by oscar_set_layer_params, so this runs before the wait on the preceding kernel).
template <int NW>
__device__ __forceinline__ void load_rk_cols(const KernelParams& kp, int layer, int kvh,
                                             float (&rk)[Shape<NW>::kRows]) {
  using Sh = Shape<NW>;
  const int c = threadIdx.x / Sh::kParts, i0 = (threadIdx.x % Sh::kParts) * Sh::kRows;
  const float* R = reinterpret_cast<const float*>(kp.base + kp.lay.R_K) +
                   (size_t(layer) * kp.n_kv_heads + kvh) * kHeadDim * kHeadDim + size_t(i0) * kHeadDim + c;
#pragma unroll
  for (int u = 0; u < Sh::kRows; ++u) rk[u] = __ldg(R + u * kHeadDim);
}

// q~ = R_K^T q (fp32) for the G query heads at q_head0 into qts[G][kQRow] (shared), and per
// warp w the sum of q~ over its kHeadDim / NW channels into qpart[w][G] (shared).  qin:
// G * kQinRow floats of shared staging (channel i of a head at i + 4 (i / kRows), so that
// the parts a warp reads together fall in different banks).  All threads; two barriers.
template <int G, int NW>
__device__ void rotate_q(const uint16_t* __restrict__ q_head0, const float (&rk)[Shape<NW>::kRows], float* qin,
                         float* qts, float* qpart) {
  using Sh = Shape<NW>;
  constexpr int KP = Sh::kParts, KR = Sh::kRows;
  const int tid = threadIdx.x, c = tid / KP, part = tid % KP, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < G * kHeadDim; e += Sh::NTH) {
    const int h = e / kHeadDim, i = e % kHeadDim;
    qin[h * Sh::kQinRow + i + 4 * (i / KR)] = bf16_f32(q_head0[e]);
  }
  __syncthreads();
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll
  for (int u = 0; u < KR; u += 4)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float4 x = *reinterpret_cast<const float4*>(qin + h * Sh::kQinRow + (KR + 4) * part + u);
      acc[h] = fmaf(rk[u + 3], x.w, fmaf(rk[u + 2], x.z, fmaf(rk[u + 1], x.y, fmaf(rk[u], x.x, acc[h]))));
    }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    // the parts of the channel in ascending row order; every lane of the group gets the sum
    float v = acc[h];
    if (KP == 2) {
      const float o = __shfl_xor_sync(0xffffffffu, v, 1);
      v = part ? o + v : v + o;
    } else {
      const float p0 = __shfl_sync(0xffffffffu, v, lane & ~3), p1 = __shfl_sync(0xffffffffu, v, (lane & ~3) | 1);
      const float p2 = __shfl_sync(0xffffffffu, v, (lane & ~3) | 2), p3 = __shfl_sync(0xffffffffu, v, (lane & ~3) | 3);
      v = ((p0 + p1) + p2) + p3;
    }
    if (part == 0) qts[h * kQRow + c] = v;
    float sw = part == 0 ? v : 0.f;  // the warp's channels, each counted once
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sw += __shfl_xor_sync(0xffffffffu, sw, off);
    if (lane == 0) qpart[warp * G + h] = sw;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- split kernel
// Tensor-memory INT2 path (format OSCAR_FORMAT_INT2_CM): a warpgroup takes tiles of two
// pages (128 tokens).  B columns n = (group g, head h, hi|lo) = 2 G g + 2 h + hi|lo.
template <int G, int GROUP>
struct TcShape {
  static constexpr int NG = kHeadDim / GROUP;
  static constexpr int NCOL = NG * 2 * G;           // B columns in use
  static constexpr int N = NCOL < 16 ? 16 : NCOL;   // MMA N (M = 128 takes multiples of 16)
  static constexpr int NB = N / 8;                  // 8-column core blocks
  static constexpr int TS = GROUP == 32 ? 3 : 4;    // tile stages per warpgroup
  static constexpr int kCols = 128;                 // tensor-memory columns per warpgroup
  static constexpr int kColD = 64;                  // A: columns [0, 64) (128 x 128 fp16); D after it
  static constexpr int kColX = 96;                  // values of a tile's first page (written during the score MMA)
  static constexpr int kBqBytes = kHeadDim * N * 2;  // q~ columns, K-major
  static constexpr int kBpBytes = 128 * N * 2;       // P' of a tile, MN-major (per warpgroup)
  static constexpr int kRedFloats = G + NG * G;       // per warp: sums of p and of p z_V
};

template <int G, int GROUP, int NW_, bool CM = false>
struct Cfg {
  static constexpr int NW = NW_, NTH = Shape<NW>::NTH;
  static constexpr int kPerSM = NW == 8 ? 2 : 1;  // resident CTAs per SM (128 registers a thread)
  static constexpr int NG = kHeadDim / GROUP;           // groups per token
  static constexpr int NT = G / 4;                      // score n-tiles (4 heads x hi/lo each)
  static constexpr int kCodeBytes = 2 * kPage * kRowBytes;  // K then V codes
  static constexpr int kSzBytes = 2 * kPage * NG * 4;       // K then V (scale, zero)
  static constexpr int kStageBytes = kCodeBytes + kSzBytes;
  // tensor-memory path: tile stages, then each warpgroup's P' block, warp maxima and sums
  using T = TcShape<G, GROUP>;
  static constexpr int NWG = NW / 4;
  static constexpr int kTcBp = ((NWG * T::TS * 2 * kStageBytes + 127) / 128) * 128;
  static constexpr int kTcWmax = kTcBp + NWG * T::kBpBytes;  // fp32 [NW][G]
  static constexpr int kTcRed = kTcWmax + NW * G * 4;        // fp32 [NW][kRedFloats]
  static constexpr int kTcPok = kTcRed + NW * T::kRedFloats * 4;  // uint8 [NWG][TS]: pages copied per tile stage
  static constexpr int kTcEnd = kTcPok + 64;
  static constexpr int kPipeBytes = CM ? kTcEnd : NW * kStages * kStageBytes;
  // fused append tasks: R (fp32 [d][d]) then the append scratch, in the same memory
  static constexpr int kAppendR = kHeadDim * kHeadDim * 4;
  static constexpr int kAppendBytes = CM ? 0 : kAppendR + int(sizeof(append_dev::Smem));
  // the merge: R_V^T (64 KB) then a slab of at least 32 partial slots (64 / G at two CTAs per SM)
  static constexpr int kSlabOff = kHeadDim * kHeadDim * 4;
  static constexpr int kMergeBytes = kSlabOff + (kPerSM == 2 ? 64 / G : 32) * PartialSlot<G>::kBytes;
  static constexpr int kWorkBytes0 = kPipeBytes > kAppendBytes ? kPipeBytes : kAppendBytes;
  static constexpr int kWorkBytes = (((kWorkBytes0 > kMergeBytes ? kWorkBytes0 : kMergeBytes) + 127) / 128) * 128;
  static constexpr int kSlabSlots = (kWorkBytes - kSlabOff) / PartialSlot<G>::kBytes;
  static constexpr int kCtl = kWorkBytes;           // control area
  // control: page barriers (NW x kStages), merge flag, next item, R_V^T and slab barriers,
  // poison flag, per-warpgroup MMA barriers (tensor-memory path), tensor-memory base
  static constexpr int kCtlMma = kCtl + NW * kStages * 8 + 32;
  static constexpr int kCtlTmem = kCtlMma + 32;
  static constexpr int kCtlBytes = ((NW * kStages * 8 + 72 + 127) / 128) * 128;
  static constexpr int kQin = kCtl + kCtlBytes;     // fp32 [G][kQinRow] query staging
  static constexpr int kQts = kQin + G * Shape<NW>::kQinRow * 4;  // fp32 [G][kQRow] q~
  static constexpr int kQss = kQts + G * kQRow * 4;  // fp32 [NW][G] sums of q~ per warp's channels
  // packed B fragments of q~ for the INT2 pages: [4 NT chunks][32 lanes][4 words]; the
  // tensor-memory path keeps its K-major q~ columns there
  static constexpr int kQbWords = 16 * NT;  // per lane
  static constexpr int kQb = ((kQss + NW * G * 4 + 127) / 128) * 128;
  static constexpr int kQbBytes = CM && T::kBqBytes > 32 * kQbWords * 4 ? T::kBqBytes : 32 * kQbWords * 4;
  static constexpr int kSmemBytes = kQb + kQbBytes;
  static constexpr int kTmemCols = NWG * T::kCols;  // tensor-memory columns of a CTA (a power of two)
  static_assert(kSmemBytes + 1024 <= 228 * 1024 / kPerSM, "resident CTAs per SM");
  static_assert(kWorkBytes >= Bf16Rows<NW, 1>::kSmemBytes, "BF16 items reuse the page pipeline memory");
  static_assert(kWorkBytes >= (NW * G * (kHeadDim + 4) + 4 * ((G + 3) / 4)) * 4,
                "per-warp results reuse the page pipeline memory");
  static_assert(kSlabOff + (1 + NTH / kHeadDim) * G * kHeadDim * 4 <= kMergeBytes,
                "o~ and the partial sums of the output rotation are staged over the slab");
  static_assert(!CM || NWG * T::TS <= NW * kStages, "tile-stage barriers");
  static_assert(!CM || kTmemCols * kPerSM <= 512, "tensor memory of the resident CTAs");
};

// Start the bulk copy of R_V^T (64 KB) of (layer, kv-head) into smem[0, 64 KB).
__device__ void fetch_rvt(const KernelParams& kp, int layer, int kvh, uint8_t* smem, uint32_t mbar) {
  if (threadIdx.x == 0) {
    const float* RVt = reinterpret_cast<const float*>(kp.base + kp.lay.R_Vt) +
                       (size_t(layer) * kp.n_kv_heads + kvh) * kHeadDim * kHeadDim;
    fence_proxy_async();
    mbar_expect_tx(mbar, kHeadDim * kHeadDim * 4);
    bulk_g2s(smem_u32(smem), RVt, kHeadDim * kHeadDim * 4, mbar);
  }
}

// Final merge: o~ = O / L, then o = R_V o~ with R_V^T in smem (fetched by fetch_rvt; this
// waits for it), bf16 and optional fp32 store.
template <int G, int NW>
__device__ void finish_output(const KernelParams& kp, const DecodeItem& it, const MergeAcc<G, Shape<NW>::NTH>& acc,
                              uint16_t* out, float* out_f32, uint8_t* smem, uint32_t mbar, uint32_t& mphase) {
  using A = MergeAcc<G, Shape<NW>::NTH>;
  constexpr int HPT = A::HPT, KS = A::kStride, JR = kHeadDim / KS;
  const int t = threadIdx.x, c = t & (kHeadDim - 1), hb = t >> 7;
  const float* Rs = reinterpret_cast<const float*>(smem);   // R_V^T [128][128]
  float* os = reinterpret_cast<float*>(smem) + kHeadDim * kHeadDim;  // o~ [G][128]
  float* red = os + G * kHeadDim;                                      // [KS][G][128] partial sums
#pragma unroll
  for (int q = 0; q < HPT; ++q) os[(hb + KS * q) * kHeadDim + c] = acc.L[q] > 0.f ? acc.O[q] / acc.L[q] : 0.f;
  const bool ok = mbar_wait(mbar, mphase);
  if (!ok) {
    if (t == 0) flag(kp, OSCAR_FLAG_TIMEOUT);
    mbar_wait(mbar, mphase);  // drain (bounded) before the memory is reused
  }
  mphase ^= 1u;
  __syncthreads();
  // thread (c, hb): rows j of R_V^T in [JR hb, JR hb + JR) for every head, then the KS
  // partial sums of a (head, channel) are added in ascending row order
  float r[G];
#pragma unroll
  for (int h = 0; h < G; ++h) r[h] = 0.f;
#pragma unroll 2
  for (int j = JR * hb; j < JR * hb + JR; j += 4) {
    const float r0 = Rs[(j + 0) * kHeadDim + c], r1 = Rs[(j + 1) * kHeadDim + c];
    const float r2 = Rs[(j + 2) * kHeadDim + c], r3 = Rs[(j + 3) * kHeadDim + c];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float4 x = *reinterpret_cast<const float4*>(os + h * kHeadDim + j);
      r[h] = fmaf(r3, x.w, fmaf(r2, x.z, fmaf(r1, x.y, fmaf(r0, x.x, r[h]))));
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) red[(hb * G + h) * kHeadDim + c] = r[h];
  __syncthreads();
  const size_t head0 = size_t(it.req) * kp.n_q_heads + size_t(it.kvh) * G;
#pragma unroll
  for (int q = 0; q < HPT; ++q) {
    const int h = hb + KS * q;
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < KS; ++k) v += red[(k * G + h) * kHeadDim + c];
    out[(head0 + h) * kHeadDim + c] = bf16_rne(ok ? v : 0.f);
    if (out_f32) out_f32[(head0 + h) * kHeadDim + c] = ok ? v : 0.f;
  }
}

// Final merge with the rotations folded into the model's projections: o~ = O / L, bf16
// and optional fp32 store, no inverse rotation.
template <int G, int NW>
__device__ void finish_output_folded(const KernelParams& kp, const DecodeItem& it,
                                     const MergeAcc<G, Shape<NW>::NTH>& acc, uint16_t* out, float* out_f32) {
  using A = MergeAcc<G, Shape<NW>::NTH>;
  constexpr int HPT = A::HPT, KS = A::kStride;
  const int t = threadIdx.x, c = t & (kHeadDim - 1), hb = t >> 7;
  const size_t head0 = size_t(it.req) * kp.n_q_heads + size_t(it.kvh) * G;
#pragma unroll
  for (int q = 0; q < HPT; ++q) {
    const int h = hb + KS * q;
    const float v = acc.L[q] > 0.f ? acc.O[q] / acc.L[q] : 0.f;
    out[(head0 + h) * kHeadDim + c] = bf16_rne(v);
    if (out_f32) out_f32[(head0 + h) * kHeadDim + c] = v;
  }
}

// The rotated queries given (R_K folded into the model's query projection): q~ (bf16) into
// qts[G][kQRow] (fp32, shared), and per warp w the sum of q~ over the channels rotate_q gives
// warp w (kHeadDim / NW of them) into qpart[w][G].  All threads; one barrier.
template <int G, int NW>
__device__ void load_q_folded(const uint16_t* __restrict__ qt_head0, float* qts, float* qpart) {
  using Sh = Shape<NW>;
  constexpr int CPW = kHeadDim / NW;  // channels of warp w: [CPW w, CPW (w + 1))
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < G * kHeadDim; e += Sh::NTH) qts[(e / kHeadDim) * kQRow + e % kHeadDim] = bf16_f32(qt_head0[e]);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float v = lane < CPW ? bf16_f32(qt_head0[h * kHeadDim + CPW * warp + lane]) : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) qpart[warp * G + h] = v;
  }
  __syncthreads();
}

// BF16 rows of the sink + ring list of (request, kv-head): list index u < min(L, S) is
// sink u, otherwise position H + u - min(L, S) in ring slot p % W.
struct SinkRingRows {
  const uint16_t *sinkK, *sinkV, *ringK, *ringV;
  int n_s, W, hw;  // hw = H % W
  __device__ SinkRingRows(const KernelParams& kp, int layer, const DecodeItem& it, const DecodeReq& dr) {
    const int S = kp.n_sink;
    n_s = min(dr.L, S);
    W = kp.window;
    hw = W > 0 ? dr.H % W : 0;
    sinkK = reinterpret_cast<const uint16_t*>(kp.base + kp.lay.sink + size_t(dr.slot) * kp.lay.sink_slot_stride +
                                              size_t(layer) * kp.lay.sink_layer_stride +
                                              size_t(it.kvh) * kp.lay.sink_head_stride);
    sinkV = sinkK + size_t(S) * kHeadDim;
    ringK = reinterpret_cast<const uint16_t*>(kp.base + kp.lay.ring + size_t(dr.slot) * kp.lay.ring_slot_stride +
                                              size_t(layer) * kp.lay.ring_layer_stride +
                                              size_t(it.kvh) * kp.lay.ring_head_stride);
    ringV = ringK + size_t(W) * kHeadDim;
  }
  // ring slot of list index u >= n_s: (H + u - n_s) % W, with u - n_s < W
  __device__ int slot(int u) const {
    const int s = hw + u - n_s;
    return s >= W ? s - W : s;
  }
  __device__ const uint16_t* K(int u) const { return u < n_s ? sinkK + size_t(u) * kHeadDim : ringK + size_t(slot(u)) * kHeadDim; }
  __device__ const uint16_t* V(int u) const { return u < n_s ? sinkV + size_t(u) * kHeadDim : ringV + size_t(slot(u)) * kHeadDim; }
};

// Copy the rows of BF16 item `it` that are final before the wait on the preceding kernel
// (list indices below it.split) into the item's row buffer.
template <int NW>
__device__ void bf16_item_prestage(const KernelParams& kp, int layer, const DecodeItem& it, const DecodeReq& dr,
                                   uint8_t* smem) {
  const SinkRingRows rows(kp, layer, it, dr);
  bf16_prestage<NW>([&](int u) { return rows.K(u); }, [&](int u) { return rows.V(u); }, it.begin, it.split, smem);
}

// BF16 tokens [it.begin, it.end) of the sink + ring list; the rows below it.split were
// copied by bf16_item_prestage when `prestaged`; wait_rest() runs before the other rows
// are copied.
template <int G, int NW, typename WaitRest>
__device__ void bf16_tokens_item(const KernelParams& kp, int layer, const DecodeItem& it, const DecodeReq& dr,
                                 const float* qts, uint8_t* part, uint8_t* smem, bool prestaged, WaitRest wait_rest) {
  const SinkRingRows rows(kp, layer, it, dr);
  bf16_rows_mma<G, NW, 1>([&](int u) { return rows.K(u); }, [&](int u) { return rows.V(u); }, it.begin, it.end, qts,
                          part, smem, prestaged ? it.split - it.begin : 0, wait_rest);
}

// Issue (lane 0 of the calling warp) the bulk copies of the warp's k-th page of an INT2
// item into stage k % kStages; false (no copy) if the page id is out of range.
template <int G, int GROUP, int NW>
__device__ bool int2_issue_page(const KernelParams& kp, int layer, const DecodeItem& it, const DecodeReq& dr, int k,
                                uint8_t* smem) {
  using C = Cfg<G, GROUP, NW>;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int lp = it.begin + warp + C::NW * k;
  const int* ptab = reinterpret_cast<const int*>(kp.base + kp.lay.page_table) + size_t(dr.slot) * kp.max_pages_per_request;
  int phys = -1;
  if (lp < kp.max_pages_per_request) phys = ptab[lp];
  if (phys < 0 || phys >= kp.max_pages) return false;
  if (lane == 0) {
    const int st = k % kStages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kCtl) + warp * kStages;
    const uint32_t bar = smem_u32(&bars[st]);
    uint8_t* dst = smem + size_t(warp) * kStages * C::kStageBytes + size_t(st) * C::kStageBytes;
    const uint8_t* code = kp.base + kp.lay.codes + size_t(layer) * kp.lay.codes_layer_stride +
                          size_t(phys) * kp.lay.codes_page_stride + size_t(it.kvh) * kp.lay.codes_head_stride;
    const uint8_t* sz = kp.base + kp.lay.sz + size_t(layer) * kp.lay.sz_layer_stride +
                        size_t(phys) * kp.lay.sz_page_stride + size_t(it.kvh) * kp.lay.sz_head_stride;
    fence_proxy_async();
    mbar_expect_tx(bar, C::kStageBytes);
    bulk_g2s(smem_u32(dst), code, C::kCodeBytes, bar);
    bulk_g2s(smem_u32(dst + C::kCodeBytes), sz, C::kSzBytes, bar);
  }
  return true;
}

// INT2 history pages [it.begin, it.end) of one (request, kv-head).  Positions outside
// [S, H) inside those pages are masked.  Warp w takes pages begin + w, + NW, ...
template <int G, int GROUP, int NW>
__device__ void int2_pages_item(const KernelParams& kp, int layer, const DecodeItem& it, const DecodeReq& dr,
                                const float* qts, const float* qss, uint8_t* part, uint8_t* smem,
                                uint32_t& phase_bits, uint32_t pre_mask, const unsigned* pages_ctr, int* s_poison) {
  using C = Cfg<G, GROUP, NW>;
  constexpr int NG = C::NG, NT = C::NT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  uint8_t* pipe = smem + size_t(warp) * kStages * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kCtl) + warp * kStages;
  const int S = kp.n_sink, H = dr.H;

  // my pages: it.begin + warp + C::NW * k
  const int n_my = it.end - it.begin > warp ? (it.end - it.begin - warp + C::NW - 1) / C::NW : 0;
  // fused append: a page not wholly below H_pre may hold rows this launch's append tasks
  // write; the warp waits (once) for their signal before copying such a page
  bool pages_ready = pages_ctr == nullptr;
  auto issue = [&](int k) -> bool {
    if (!pages_ready && (it.begin + warp + C::NW * k + 1) * kPage > dr.H_pre) {
      if (lane == 0) {
        if (!wait_counter(pages_ctr, unsigned(dr.app_expect), kp.counter_polls)) flag(kp, OSCAR_FLAG_TIMEOUT);
        fence_proxy_async_global();
      }
      __syncwarp();
      pages_ready = true;
    }
    return int2_issue_page<G, GROUP, NW>(kp, layer, it, dr, k, smem);
  };
  // ok_mask bit st: stage st has a copy in flight; phase_bits (kept across items):
  // bit st = parity of the next completion of stage st.  The caller issued the first
  // stages it could (pre_mask); the rest are issued here.
  uint32_t ok_mask = pre_mask;
  for (int k = 0; k < min(kStages, n_my); ++k)
    if (!((pre_mask >> k) & 1u) && issue(k)) ok_mask |= 1u << k;

  // ---- B fragments of q~ (hi/lo fp16 columns), scaled by 4^-(kc & 3) for field kc: the
  // same for every warp, so the CTA packs them once.  Lane (gid, tig) word w = 2(NT kc + j) + r
  // holds head 4j + gid / 2, channels 16 kc + 4 tig + 2r, +1 (hi part for even gid, lo for odd).
  uint32_t* qb = reinterpret_cast<uint32_t*>(smem + C::kQb);
  for (int e = threadIdx.x; e < 32 * C::kQbWords; e += C::NTH) {
    const int ln = e & 31, w = e >> 5;  // consecutive threads: consecutive lanes of one word
    const int kc = w / (2 * NT), j = (w >> 1) % NT, r = w & 1;
    const int g_ = ln >> 2, t_ = ln & 3;
    const int head = 4 * j + (g_ >> 1);
    const float fs = 1.0f / float(1 << (2 * (kc & 3)));
    const float2 v2 = *reinterpret_cast<const float2*>(qts + head * kQRow + 16 * kc + 4 * t_ + 2 * r);
    const float v0 = v2.x * fs, v1 = v2.y * fs;
    const float h0 = __half2float(__float2half_rn(v0)), h1 = __half2float(__float2half_rn(v1));
    qb[((w >> 2) * 32 + ln) * 4 + (w & 3)] = (g_ & 1) ? pack_h2(v0 - h0, v1 - h1) : pack_h2(h0, h1);
  }
  __syncthreads();
  uint32_t bq[8][NT][2];
#pragma unroll
  for (int c4 = 0; c4 < 4 * NT; ++c4) {
    const uint4 u = reinterpret_cast<const uint4*>(qb)[c4 * 32 + lane];
    const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int w = 4 * c4 + i;
      bq[w / (2 * NT)][(w >> 1) % NT][w & 1] = ws[i];
    }
  }
  // per-thread heads: n-tile j gives head 4j + tig
  const float scale = kLog2e * rsqrtf(float(kHeadDim));
  float qs_scaled[NT][NG];  // sum(q~) over the group, times scale
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int g = 0; g < NG; ++g) {  // sum of q~ over group g: warps 8g / NG .. 8(g + 1) / NG - 1
      constexpr int WPG = C::NW / NG;
      float sq = 0.f;
#pragma unroll
      for (int w = 0; w < WPG; ++w) sq += qss[(WPG * g + w) * G + 4 * j + tig];
      qs_scaled[j][g] = sq * scale;
    }

  // m_run: the warp's running maximum per head; muse: the same, 0 while -inf
  float m_run[NT], muse[NT], l_part[NT], zv[NT][NG];
  float oacc[8][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    m_run[j] = -INFINITY;
    muse[j] = 0.f;
    l_part[j] = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) zv[j][g] = 0.f;
  }
#pragma unroll
  for (int f = 0; f < 8; ++f)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[f][e] = 0.f;

  const float two24 = 16777216.0f;
  const float scale24 = scale * two24;  // undoes the 2^-24 of the subnormal key codes
  const int tok_a = tau8(gid);  // rows gid and gid + 8 of the score tile: tokens tok_a, tok_a + 8
  bool broken = false;
  for (int k = 0; k < n_my; ++k) {
    const int st = k % kStages;
    const int lp = it.begin + warp + C::NW * k;
    const bool have = (ok_mask >> st) & 1u;
    if (have) {
      if (!mbar_wait(smem_u32(&bars[st]), (phase_bits >> st) & 1u)) {
        if (lane == 0) flag(kp, OSCAR_FLAG_TIMEOUT);
        broken = true;
        break;
      }
      phase_bits ^= 1u << st;
      ok_mask &= ~(1u << st);
    } else {
      // a page that was not copied (page id out of range) contributes nothing
      if (lane == 0) flag(kp, OSCAR_FLAG_BAD_PAGE);
      __syncwarp();
      if (k + kStages < n_my && issue(k + kStages)) ok_mask |= 1u << st;
      continue;
    }
    // positions [S, H) of the page: tokens t with t - vlo < vn (unsigned)
    const int vlo = max(S - lp * kPage, 0), vn = max(0, min(H - lp * kPage, kPage) - vlo);
    const uint8_t* stage = pipe + size_t(st) * C::kStageBytes;
    const uint8_t* kcodes = stage;
    const uint8_t* vcodes = stage + kPage * kRowBytes;
    const uint32_t* ksz = reinterpret_cast<const uint32_t*>(stage + C::kCodeBytes);
    const uint32_t* vsz = ksz + kPage * NG;

    // ---- scores for the 64 tokens of the page (4 blocks of 16)
    float lg[4][NT][2];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int t0 = 16 * b + tok_a, t1 = t0 + 8;
      const uint2 wa = *reinterpret_cast<const uint2*>(kcodes + t0 * kRowBytes + 8 * tig);
      const uint2 wb = *reinterpret_cast<const uint2*>(kcodes + t1 * kRowBytes + 8 * tig);
      const uint32_t wa0s = wa.x >> 8, wa1s = wa.y >> 8, wb0s = wb.x >> 8, wb1s = wb.y >> 8;
      // accumulators: one per group of 32 channels (fields 2g, 2g+1) at g = 32; two
      // (even / odd fields) at g = 128
      constexpr int NA = NG == 1 ? 2 : 4;
      float acc[NA][NT][4];
#pragma unroll
      for (int p = 0; p < NA; ++p)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[p][j][e] = 0.f;
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        const uint32_t a0 = field(wa.x, wa0s, kc), a1 = field(wb.x, wb0s, kc);
        const uint32_t a2 = field(wa.y, wa1s, kc), a3 = field(wb.y, wb1s, kc);
#pragma unroll
        for (int j = 0; j < NT; ++j)
          mma16816(acc[NG == 1 ? (kc & 1) : (kc >> 1)][j], a0, a1, a2, a3, bq[kc][j][0], bq[kc][j][1]);
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          float T0, T1;
          if (NG == 1) {
            T0 = (acc[0][j][0] + acc[0][j][1]) + (acc[1][j][0] + acc[1][j][1]);
            T1 = (acc[0][j][2] + acc[0][j][3]) + (acc[1][j][2] + acc[1][j][3]);
          } else {
            T0 = acc[g][j][0] + acc[g][j][1];
            T1 = acc[g][j][2] + acc[g][j][3];
          }
          const uint32_t sz0 = ksz[t0 * NG + g], sz1 = ksz[t1 * NG + g];
          s0 += fmaf(T0, bf16_lo(sz0) * scale24, bf16_hi(sz0) * qs_scaled[j][g]);
          s1 += fmaf(T1, bf16_lo(sz1) * scale24, bf16_hi(sz1) * qs_scaled[j][g]);
        }
        lg[b][j][0] = s0;
        lg[b][j][1] = s1;
      }
    }
    if (vlo != 0 || vn != kPage) {  // (warp-uniform) the page holds positions outside [S, H)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int t0 = 16 * b + tok_a, t1 = t0 + 8;
        const bool v0 = unsigned(t0 - vlo) < unsigned(vn), v1 = unsigned(t1 - vlo) < unsigned(vn);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (!v0) lg[b][j][0] = -INFINITY;
          if (!v1) lg[b][j][1] = -INFINITY;
        }
      }
    }
    // ---- online softmax over the page (per head: 8 scores per thread, 8 lanes per head):
    // the page's maxima are reduced over the head's lanes, and the sums rescaled, only
    // when some score exceeds the running maximum.  The maximum stays exact (not a lazy
    // reference), so the token that holds it gets p = 1 and an exact P' = s_V: with one
    // dominant token, the fp16 rounding of its P' would be the output's error.
    float mloc[NT];
    bool over = false;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      mloc[j] = fmax3(fmax3(lg[0][j][0], lg[0][j][1], lg[1][j][0]), fmax3(lg[1][j][1], lg[2][j][0], lg[2][j][1]),
                      fmaxf(lg[3][j][0], lg[3][j][1]));
      over |= mloc[j] > m_run[j];
    }
    if (__any_sync(0xffffffffu, over)) {
      float alpha[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        float mx = mloc[j];
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(m_run[j], mx);
        muse[j] = mnew == -INFINITY ? 0.f : mnew;
        alpha[j] = ex2(m_run[j] - muse[j]);  // 0 while the reference was -inf
        m_run[j] = mnew;
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        l_part[j] *= alpha[j];
#pragma unroll
        for (int g = 0; g < NG; ++g) zv[j][g] *= alpha[j];
      }
      // value accumulator columns: G = 4 -> head tig (and a column that stays 0); G = 8 -> heads tig, 4 + tig
#pragma unroll
      for (int f = 0; f < 8; ++f) {
        const float a0 = alpha[0], a1 = NT == 2 ? alpha[NT - 1] : alpha[0];
        oacc[f][0] *= a0;
        oacc[f][1] *= a1;
        oacc[f][2] *= a0;
        oacc[f][3] *= a1;
      }
    }
    // ---- values
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int t0 = 16 * b + tok_a, t1 = t0 + 8;
      float p[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        // masked tokens carry lg = -inf and muse is finite: ex2 gives exactly 0
        p[j][0] = ex2(lg[b][j][0] - muse[j]);
        p[j][1] = ex2(lg[b][j][1] - muse[j]);
        l_part[j] += p[j][0] + p[j][1];
      }
      // B fragments of P' = p * s_V per group (movmatrix turns score rows into value k-rows).
      // Masked rows have p = 0, and every scale/zero word of the pool is finite (the pool
      // starts zeroed and only finite words are written), so they need no select.
      uint32_t bp[NG][2];
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const uint32_t vz0 = vsz[t0 * NG + g], vz1 = vsz[t1 * NG + g];
        const float sv0 = bf16_lo(vz0), sv1 = bf16_lo(vz1);
        const float zv0 = bf16_hi(vz0), zv1 = bf16_hi(vz1);
        uint32_t x0, x1;
        if (NT == 1) {  // heads in the even columns; the odd (second-part) columns stay 0
          x0 = pack_h2(p[0][0] * sv0, 0.f);
          x1 = pack_h2(p[0][1] * sv1, 0.f);
        } else {
          x0 = pack_h2(p[0][0] * sv0, p[NT - 1][0] * sv0);
          x1 = pack_h2(p[0][1] * sv1, p[NT - 1][1] * sv1);
        }
        bp[g][0] = movtrans(x0);
        bp[g][1] = movtrans(x1);
#pragma unroll
        for (int j = 0; j < NT; ++j) zv[j][g] = fmaf(p[j][1], zv1, fmaf(p[j][0], zv0, zv[j][g]));
      }
      // A fragments: word gid of tokens tig, tig+4, tig+8, tig+12 (k = 2tig, 2tig+1, 2tig+8, 2tig+9)
      const uint32_t* vw = reinterpret_cast<const uint32_t*>(vcodes + (16 * b) * kRowBytes) + gid;
      const uint32_t wA = vw[(tig)*8], wB = vw[(tig + 4) * 8], wC = vw[(tig + 8) * 8], wD = vw[(tig + 12) * 8];
      const uint32_t X = prmt(wA, wB, 0x5410), Y = prmt(wA, wB, 0x7632);
      const uint32_t X2 = prmt(wC, wD, 0x5410), Y2 = prmt(wC, wD, 0x7632);
      const uint32_t Xs = X >> 8, Ys = Y >> 8, X2s = X2 >> 8, Y2s = Y2 >> 8;
#pragma unroll
      for (int f = 0; f < 8; ++f) {
        const int g = NG == 1 ? 0 : (f >> 1);
        mma16816(oacc[f], field(X, Xs, f), field(Y, Ys, f), field(X2, X2s, f), field(Y2, Y2s, f), bp[g][0], bp[g][1]);
      }
    }
    // ---- refill this stage with my page k + kStages
    __syncwarp();
    if (k + kStages < n_my && issue(k + kStages)) ok_mask |= 1u << st;
  }
  if (broken) {
    // drain copies still in flight (bounded) before the stages are reused or the CTA exits;
    // a stage whose copy does not land even then leaves its barrier phase unknown, so the
    // CTA takes no further work (s_poison) once this item is done
    bool drained = true;
    for (int st = 0; st < kStages; ++st)
      if ((ok_mask >> st) & 1u) {
        if (mbar_wait(smem_u32(&bars[st]), (phase_bits >> st) & 1u)) phase_bits ^= 1u << st;
        else drained = false;
      }
    if (!drained && lane == 0) *s_poison = 1;
  }

  // ---- per-warp results -> shared memory, then merge the 4 warps into the partial
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    l_part[j] += __shfl_xor_sync(0xffffffffu, l_part[j], 4);
    l_part[j] += __shfl_xor_sync(0xffffffffu, l_part[j], 8);
    l_part[j] += __shfl_xor_sync(0xffffffffu, l_part[j], 16);
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      zv[j][g] += __shfl_xor_sync(0xffffffffu, zv[j][g], 4);
      zv[j][g] += __shfl_xor_sync(0xffffffffu, zv[j][g], 8);
      zv[j][g] += __shfl_xor_sync(0xffffffffu, zv[j][g], 16);
    }
  }
  __syncthreads();  // every warp is done with its stages: reuse the pipeline memory
  // per-warp maxima, then every warp scales its (l, o) to the CTA's maximum and the
  // scaled parts are added over the warps in ascending order
  float* wm = reinterpret_cast<float*>(smem);  // [NW][G] maxima
  float* wl = wm + C::NW * G;                   // [NW][G] scaled l
  float* wmax = wl + C::NW * G;                 // [G] CTA maxima (4 floats reserved)
  float* wo = wmax + 4 * ((G + 3) / 4);         // [NW][G][d + 2] scaled o (rows padded against bank conflicts)
  constexpr int kRow = kHeadDim + 2;
  if (gid == 0) {
#pragma unroll
    for (int j = 0; j < NT; ++j) wm[warp * G + 4 * j + tig] = broken ? -INFINITY : m_run[j];
  }
  __syncthreads();
  float a[NT];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int head = 4 * j + tig;
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) ms = fmaxf(ms, wm[w * G + head]);
    a[j] = broken || ms == -INFINITY ? 0.f : ex2(m_run[j] - ms);
    if (gid == 0) {
      wl[warp * G + head] = l_part[j] * a[j];
      if (warp == 0) wmax[head] = ms;
    }
  }
#pragma unroll
  for (int f = 0; f < 8; ++f) {
    const float us = two24 / float(1 << (2 * (f & 3)));
    const int ch0 = 16 * f + 2 * gid, ch1 = ch0 + 1;
    const int g = NG == 1 ? 0 : (f >> 1);
    float* mine = wo + size_t(warp) * G * kRow;
    if (NT == 1) {
      mine[tig * kRow + ch0] = ((oacc[f][0] + oacc[f][1]) * us + zv[0][g]) * a[0];
      mine[tig * kRow + ch1] = ((oacc[f][2] + oacc[f][3]) * us + zv[0][g]) * a[0];
    } else {
      mine[tig * kRow + ch0] = (oacc[f][0] * us + zv[0][g]) * a[0];
      mine[(4 + tig) * kRow + ch0] = (oacc[f][1] * us + zv[NT - 1][g]) * a[NT - 1];
      mine[tig * kRow + ch1] = (oacc[f][2] * us + zv[0][g]) * a[0];
      mine[(4 + tig) * kRow + ch1] = (oacc[f][3] * us + zv[NT - 1][g]) * a[NT - 1];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * kHeadDim; e += C::NTH) {
    const int h = e / kHeadDim, c = e % kHeadDim;
    float l = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < C::NW; ++w) {
      l += wl[w * G + h];
      o += wo[(w * G + h) * kRow + c];
    }
    store_slot<G>(part, h, c, wmax[h], l, o);
  }
}

// ---------------------------------------------------------------- INT2 pages on tcgen05
// Named barrier of warpgroup u (128 threads; id 0 is __syncthreads), with immediate ids so
// that the kernel reserves only the barriers it uses; and the same with an OR of a
// predicate over the warpgroup.
#define OSCAR_BAR_WG(ID) asm volatile("bar.sync " #ID ", 128;" ::: "memory")
template <int NWG>
__device__ __forceinline__ void bar_wg(int u) {
  if (u == 0) OSCAR_BAR_WG(1);
  else if constexpr (NWG == 2) OSCAR_BAR_WG(2);
  else if (u == 1) OSCAR_BAR_WG(2);
  else if (u == 2) OSCAR_BAR_WG(3);
  else OSCAR_BAR_WG(4);
}
#undef OSCAR_BAR_WG
#define OSCAR_BAR_WG_OR(ID)                                                                                  \
  asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, " #ID                       \
               ", 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"                                                          \
               : "=r"(r)                                                                                     \
               : "r"(uint32_t(v))                                                                            \
               : "memory")
template <int NWG>
__device__ __forceinline__ bool bar_wg_or(int u, bool v) {
  uint32_t r;
  if (u == 0) OSCAR_BAR_WG_OR(1);
  else if constexpr (NWG == 2) OSCAR_BAR_WG_OR(2);
  else if (u == 1) OSCAR_BAR_WG_OR(2);
  else if (u == 2) OSCAR_BAR_WG_OR(3);
  else OSCAR_BAR_WG_OR(4);
  return r != 0;
}
#undef OSCAR_BAR_WG_OR
// One lane of the (converged) warp: true there, false elsewhere.
__device__ __forceinline__ bool elect_one() {
  uint32_t r;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n" : "=r"(r));
  return r != 0;
}
__device__ __forceinline__ float warp_max(float x) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
  return r;
}
// fp16 hi and lo parts of x (x ~ hi + lo to about 22 bits), as the two halves of a word
__device__ __forceinline__ uint32_t hi_lo(float x) {
  const float hi = __half2float(__float2half_rn(x));
  return pack_h2(hi, x - hi);
}

// INT2 history pages [it.begin, it.end) of one (request, kv-head) on the tcgen05 tensor
// cores (format OSCAR_FORMAT_INT2_CM).  Warpgroup u (warps 4u .. 4u + 3) takes tiles of two
// pages, tiles u, u + NWG, ...; per tile (128 tokens):
//   1. thread t = token t: its 32-byte key row, one AND per two codes (fp16 subnormals
//      code * 4^(f & 3) * 2^-24 of field f), into A (tensor memory, lane t);
//   2. one thread: S = A x B_q (8 MMAs of K = 16), B_q = q~ * 4^-(f & 3) as fp16 hi and lo
//      columns per (group, head), so q~ keeps about 22 bits.  Meanwhile thread c = channel
//      c moves its channel-major value words of the first page into X (lane c), one AND per
//      two codes (tokens 16 b + f and 16 b + 8 + f of word b share a column);
//   3. thread t: scores s = (S_hi + S_lo) s_K 2^24 + z_K sum(q~) per group, masked outside
//      [S, H); p = 2^(s - m) against the warpgroup's reference maximum m per head, which
//      is raised (and the sums rescaled) only when a score exceeds it by more than 8, so
//      p <= 2^8; P' = p s_V 4^-(f & 3) 2^kappa (fp16 hi and lo) into B_P, row k(t); the
//      second page's values into A;
//   4. one thread: D = [X | A] x B_P (8 MMAs, K = 16 tokens each); read back at the next
//      tile by thread c: o += D 2^(24 - kappa).
// The warpgroups of the SM overlap one another's MMA waits.
template <int G, int GROUP, int NW>
__device__ void int2_tc_item(const KernelParams& kp, int layer, const DecodeItem& it, const DecodeReq& dr,
                             const float* qts, const float* qss, uint8_t* part, uint8_t* smem, uint32_t& phase_bits,
                             uint32_t& mma_phase, uint32_t tmem_base, int* s_poison) {
  using C = Cfg<G, GROUP, NW, true>;
  using T = TcShape<G, GROUP>;
  constexpr int NG = T::NG, NWG = C::NWG, TS = T::TS, N = T::N, NB = T::NB;
  static_assert(T::kColD + N <= T::kColX && T::kColX + 32 <= T::kCols, "tensor-memory columns of a warpgroup");
  static_assert(N == 16 || N == 32, "D loads of 16 or 32 columns");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = warp >> 2, q = warp & 3, t = tid & 127;
  const bool leader = t == 0;
  const int S = kp.n_sink, H = dr.H;
  const uint32_t tm = tmem_base + uint32_t(u * T::kCols);  // this warpgroup's columns
  const uint32_t tl = tm + (uint32_t(32 * q) << 16);        // ... at this warp's lanes
  uint8_t* stages = smem + size_t(u) * TS * 2 * C::kStageBytes;
  uint64_t* sbars = reinterpret_cast<uint64_t*>(smem + C::kCtl) + u * TS;
  uint8_t* pok = smem + C::kTcPok + u * TS;  // per tile stage: bit p = page p was copied
  const uint32_t mbar = smem_u32(reinterpret_cast<uint64_t*>(smem + C::kCtlMma) + u);
  uint8_t* bp = smem + C::kTcBp + size_t(u) * T::kBpBytes;
  float* wmax = reinterpret_cast<float*>(smem + C::kTcWmax);
  float* wred = reinterpret_cast<float*>(smem + C::kTcRed);
  uint8_t* bq = smem + C::kQb;
  const int* ptab = reinterpret_cast<const int*>(kp.base + kp.lay.page_table) + size_t(dr.slot) * kp.max_pages_per_request;

  // ---- B_q (all threads): column n, channels 8 kb .. 8 kb + 7 per 16-byte core row
  for (int e = tid; e < N * 16; e += C::NTH) {
    const int n = e % N, kb = e / N;
    const int g = n / (2 * G), h = (n % (2 * G)) >> 1, hl = n & 1;
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float v[2];
#pragma unroll
      for (int z = 0; z < 2; ++z) {
        const int c = 8 * kb + 2 * i + z;
        v[z] = 0.f;
        if (n < T::NCOL && c / GROUP == g) {
          const float x = qts[h * kQRow + c] * (1.0f / float(1 << (2 * ((c >> 4) & 3))));
          const float hi = __half2float(__float2half_rn(x));
          v[z] = hl ? x - hi : hi;
        }
      }
      w[i] = pack_h2(v[0], v[1]);
    }
    *reinterpret_cast<uint4*>(bq + (kb * NB + n / 8) * 128 + (n % 8) * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  fence_proxy_async();  // generic writes of B_q before the tensor cores read them
  __syncthreads();

  const float scale = kLog2e * rsqrtf(float(kHeadDim));
  const float scale24 = scale * 16777216.0f;
  float qsc[NG][G];  // sum of q~ over group g, times scale
#pragma unroll
  for (int g = 0; g < NG; ++g)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      constexpr int WPG = NW / NG;
      float sq = 0.f;
#pragma unroll
      for (int w = 0; w < WPG; ++w) sq += qss[(WPG * g + w) * G + h];
      qsc[g][h] = sq * scale;
    }
  // P' scale 2^kappa keeps p s_V (p <= 2^8, s_V < clip_V) below 2^14 in fp16
  const float clipv = reinterpret_cast<const float*>(kp.base + kp.lay.clip_V)[layer * kp.n_kv_heads + it.kvh];
  const int kappa = clipv > 0.f && clipv < 1e30f ? min(60, max(-60, 5 - ilogbf(clipv))) : 0;
  const float pscale = ldexpf(1.0f, kappa - 2 * (t & 3));  // and 4^-(f & 3) of my token's field f = t & 7
  const float oscale = ldexpf(1.0f, 24 - kappa);
  const int kidx = (t & ~15) + 2 * (t & 7) + ((t >> 3) & 1);  // my token's row of B_P (K index)
  const int gc = GROUP == 32 ? q : 0;                         // group of my channel t

  const int n_tiles = (it.end - it.begin + 1) / 2;
  const int n_my = n_tiles > u ? (n_tiles - u + NWG - 1) / NWG : 0;
  auto tile_lp0 = [&](int k) { return it.begin + 2 * (u + NWG * k); };
  auto load_ids = [&](int k, int (&ph)[2]) {  // page ids of my k-th tile (-1: none or out of range)
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const int lp = tile_lp0(k) + p;
      ph[p] = lp < it.end && lp < kp.max_pages_per_request ? ptab[lp] : -1;
    }
  };
  auto issue = [&](int k, const int (&ph)[2]) {  // the leader: my k-th tile into stage k % TS
    const int st = k % TS, lp0 = tile_lp0(k);
    uint8_t* dst = stages + size_t(st) * 2 * C::kStageBytes;
    const uint32_t bar = smem_u32(&sbars[st]);
    uint32_t bytes = 0, ok = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      if (ph[p] >= 0 && ph[p] < kp.max_pages) {
        bytes += C::kStageBytes;
        ok |= 1u << p;
      } else if (lp0 + p < it.end) {
        flag(kp, OSCAR_FLAG_BAD_PAGE);
      }
    }
    pok[st] = uint8_t(ok);  // read by the warpgroup after the stage's barrier completes
    // (no proxy fence: the stage's earlier generic reads were all consumed before the
    // warpgroup barrier that precedes this)
    mbar_expect_tx(bar, bytes);  // the arrival; the phase completes once the bytes land
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      if (!((ok >> p) & 1u)) continue;
      const uint8_t* code = kp.base + kp.lay.codes + size_t(layer) * kp.lay.codes_layer_stride +
                            size_t(ph[p]) * kp.lay.codes_page_stride + size_t(it.kvh) * kp.lay.codes_head_stride;
      const uint8_t* sz = kp.base + kp.lay.sz + size_t(layer) * kp.lay.sz_layer_stride +
                          size_t(ph[p]) * kp.lay.sz_page_stride + size_t(it.kvh) * kp.lay.sz_head_stride;
      bulk_g2s(smem_u32(dst + p * C::kStageBytes), code, C::kCodeBytes, bar);
      bulk_g2s(smem_u32(dst + p * C::kStageBytes + C::kCodeBytes), sz, C::kSzBytes, bar);
    }
  };
  // warp 0 of the warpgroup issues the MMAs, warp 3 the page copies (one elected lane
  // each); the lanes of warp 3 all hold the page ids of the next tile to copy
  int nph[2] = {-1, -1};
  if (q == 3) {
    fence_proxy_async();  // the item's generic writes of this memory (B_q, the last results)
    for (int k = 0; k < min(TS, n_my); ++k) {
      int ph[2];
      load_ids(k, ph);
      if (elect_one()) issue(k, ph);
      __syncwarp();
    }
    if (TS < n_my) load_ids(TS, nph);
  }
  int n_issued = min(TS, n_my), next_wait = 0;  // tiles copied; first tile not yet waited for

  float m_ref[G], l_acc[G], zv[NG][G], o_acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_ref[h] = -INFINITY;
    l_acc[h] = 0.f;
    o_acc[h] = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) zv[g][h] = 0.f;
  }
  bool broken = false, mma_out = false;  // mma_out: a value MMA not yet read back
  bool mma_lost = false;                   // an MMA wait gave up (its barrier phase is unknown)
  // wait for this warpgroup's last commit (all threads of the warpgroup); false on timeout
  auto wait_mma = [&]() -> bool {
    const bool ok = mbar_wait(mbar, mma_phase & 1u);
    mma_phase ^= 1u;
    tmem::fence_after();
    return !bar_wg_or<NWG>(u, !ok);
  };
  // o += D 2^(24 - kappa) for my channel t, after the value MMA of the last tile
  auto read_values = [&]() -> bool {
    if (!wait_mma()) return false;
    uint32_t dv[2 * G];
    if constexpr (G == 4) tmem::ld_x8(tl + T::kColD + 2 * G * gc, dv);
    else tmem::ld_x16(tl + T::kColD + 2 * G * gc, dv);
    tmem::wait_ld();
#pragma unroll
    for (int h = 0; h < G; ++h)
      o_acc[h] = fmaf(__uint_as_float(dv[2 * h]) + __uint_as_float(dv[2 * h + 1]), oscale, o_acc[h]);
    return true;
  };
  // values of channel t in page pg of the stage into tensor-memory columns col .. col + 31
  auto put_values = [&](const uint8_t* stg, int pg, uint32_t col) {
    const uint32_t* vw = reinterpret_cast<const uint32_t*>(stg + pg * C::kStageBytes + kPage * kRowBytes) + t;
    uint32_t r[32];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const uint32_t W = vw[kHeadDim * b], Ws = W >> 8;
#pragma unroll
      for (int f = 0; f < 8; ++f) r[8 * b + f] = (f < 4 ? W : Ws) & (0x00030003u << (2 * (f & 3)));
    }
    tmem::st_x32(tl + col, r);
  };

  for (int k = 0; k < n_my; ++k) {
    const int st = k % TS, lp0 = tile_lp0(k);
    uint8_t* stg = stages + size_t(st) * 2 * C::kStageBytes;
    const bool landed = mbar_wait(smem_u32(&sbars[st]), (phase_bits >> st) & 1u);
    if (bar_wg_or<NWG>(u, !landed)) {
      if (leader) flag(kp, OSCAR_FLAG_TIMEOUT);
      broken = true;
      break;
    }
    phase_bits ^= 1u << st;
    ++next_wait;
    const uint32_t okp = pok[st];
    if (mma_out) {  // the last tile's values: frees A, X and D
      if (!read_values()) {
        if (leader) flag(kp, OSCAR_FLAG_TIMEOUT);
        broken = mma_lost = true;
        break;
      }
      mma_out = false;
    }
    // ---- 1. keys of token t into A
    const int tp = t >> 6, tr = t & 63;
    {
      const uint8_t* kr = stg + tp * C::kStageBytes + tr * kRowBytes;
      const uint4 a = *reinterpret_cast<const uint4*>(kr), b = *reinterpret_cast<const uint4*>(kr + 16);
      const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t r[32];
#pragma unroll
      for (int f = 0; f < 4; ++f)
#pragma unroll
        for (int w = 0; w < 8; ++w) r[8 * f + w] = wd[w] & (0x00030003u << (2 * f));
      tmem::st_x32(tl, r);
#pragma unroll
      for (int f = 0; f < 4; ++f)
#pragma unroll
        for (int w = 0; w < 8; ++w) r[8 * f + w] = (wd[w] >> 8) & (0x00030003u << (2 * f));
      tmem::st_x32(tl + 32, r);
    }
    tmem::wait_st();
    tmem::fence_before();
    bar_wg<NWG>(u);
    // ---- 2. scores; meanwhile the first page's values into X
    if (q == 0) {
      if (elect_one()) {
        tmem::fence_after();
        const uint32_t b0 = smem_u32(bq);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          tmem::mma_ts(tm + T::kColD, tm + 8 * s, tmem::sdesc(b0 + s * 2 * NB * 128, NB * 128, 128),
                       tmem::idesc_f16(128, N, false), s > 0);
        tmem::commit(mbar);
      }
      __syncwarp();
    }
    put_values(stg, 0, T::kColX);
    if (k > 0 && k + TS - 1 < n_my) {  // refill the last tile's stage while the MMA runs
      if (q == 3) {
        if (elect_one()) issue(k + TS - 1, nph);
        __syncwarp();
        if (k + TS < n_my) load_ids(k + TS, nph);
      }
      ++n_issued;
    }
    const int lp = lp0 + tp, pos = lp * kPage + tr;
    const bool valid = ((okp >> tp) & 1u) && pos >= S && pos < H;
    const uint32_t* ksz = reinterpret_cast<const uint32_t*>(stg + tp * C::kStageBytes + C::kCodeBytes) + tr * NG;
    const uint32_t* vsz = ksz + kPage * NG;
    uint32_t kszw[NG], vszw[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      kszw[g] = ksz[g];
      vszw[g] = vsz[g];
    }
    if (!wait_mma()) {
      if (leader) flag(kp, OSCAR_FLAG_TIMEOUT);
      broken = mma_lost = true;
      break;
    }
    uint32_t dsv[N];
    if constexpr (N == 16) tmem::ld_x16(tl + T::kColD, dsv);
    else tmem::ld_x32(tl + T::kColD, dsv);
    put_values(stg, 1, 0);  // the score MMA is done with A
    tmem::wait_ld();
    // ---- 3. softmax of token t against the reference maxima
    float sc[G];
    bool over = false;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float v = 0.f;
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const float T2 = __uint_as_float(dsv[2 * G * g + 2 * h]) + __uint_as_float(dsv[2 * G * g + 2 * h + 1]);
        v += fmaf(T2, bf16_lo(kszw[g]) * scale24, bf16_hi(kszw[g]) * qsc[g][h]);
      }
      sc[h] = valid ? v : -INFINITY;
      over |= sc[h] > m_ref[h] + 8.0f;
    }
    float sv[NG], zz[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {  // masked tokens: s_V = z_V = 0 (their words may be stale)
      sv[g] = valid ? bf16_lo(vszw[g]) * pscale : 0.f;
      zz[g] = valid ? bf16_hi(vszw[g]) : 0.f;
    }
    // row kidx of B_P (MN-major): 8 columns = 4 heads x hi|lo per 16-byte core row
    auto write_bp = [&](const float (&p)[G]) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = 8 * nb + 2 * i, g = n / (2 * G), h = (n % (2 * G)) >> 1;
          w[i] = n < T::NCOL ? hi_lo(p[h] * sv[g]) : 0u;
        }
        *reinterpret_cast<uint4*>(bp + ((kidx >> 3) * NB + nb) * 128 + (kidx & 7) * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    };
    float p[G];
#pragma unroll
    for (int h = 0; h < G; ++h) p[h] = over || !valid ? 0.f : ex2(sc[h] - m_ref[h]);
    write_bp(p);
    tmem::wait_st();
    fence_proxy_async();  // B_P rows before the tensor cores read them
    tmem::fence_before();
    if (bar_wg_or<NWG>(u, over)) {
      // a score above the reference by more than 8 (or the first scores): the tile's maxima
      // become the reference, the sums so far are rescaled, and p is taken again
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mx = warp_max(sc[h]);
        if (lane == 0) wmax[warp * G + h] = mx;
      }
      bar_wg<NWG>(u);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float* wm = wmax + 4 * u * G + h;
        const float mnew = fmaxf(m_ref[h], fmaxf(fmaxf(wm[0], wm[G]), fmaxf(wm[2 * G], wm[3 * G])));
        const float muse = mnew == -INFINITY ? 0.f : mnew;
        const float alpha = ex2(m_ref[h] - muse);  // 0 while the reference was -inf
        m_ref[h] = mnew;
        l_acc[h] *= alpha;
        o_acc[h] *= alpha;
#pragma unroll
        for (int g = 0; g < NG; ++g) zv[g][h] *= alpha;
        p[h] = ex2(sc[h] - muse);
      }
      write_bp(p);
      fence_proxy_async();
      tmem::fence_before();
      bar_wg<NWG>(u);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      l_acc[h] += p[h];
#pragma unroll
      for (int g = 0; g < NG; ++g) zv[g][h] = fmaf(p[h], zz[g], zv[g][h]);
    }
    // ---- 4. values; the stage is free again
    if (q == 0) {
      if (elect_one()) {
        tmem::fence_after();
        const uint32_t b0 = smem_u32(bp);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          tmem::mma_ts(tm + T::kColD, s < 4 ? tm + T::kColX + 8 * s : tm + 8 * (s - 4),
                       tmem::sdesc(b0 + s * 2 * NB * 128, NB * 128, 128), tmem::idesc_f16(128, N, true), s > 0);
        tmem::commit(mbar);
      }
      __syncwarp();
    }
    mma_out = true;
  }
  if (!broken && mma_out) {
    if (read_values()) mma_out = false;
    else {
      if (leader) flag(kp, OSCAR_FLAG_TIMEOUT);
      broken = mma_lost = true;
    }
  }
  if (broken) {
    // copies still in flight land (bounded) before the stages are reused or the CTA exits;
    // if one does not, or an MMA did not complete, the barrier phases are unknown and the
    // CTA takes no further work
    bool drained = !mma_lost && (!mma_out || wait_mma());
    for (int j = next_wait; j < n_issued; ++j) {
      const int st = j % TS;
      if (mbar_wait(smem_u32(&sbars[st]), (phase_bits >> st) & 1u)) phase_bits ^= 1u << st;
      else drained = false;
    }
    if (!drained) *s_poison = 1;
  }

  // ---- sums over the warpgroup's tokens, then the warpgroups into the partial
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l_acc[h] += __shfl_xor_sync(0xffffffffu, l_acc[h], off);
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) zv[g][h] += __shfl_xor_sync(0xffffffffu, zv[g][h], off);
  }
  if (lane == 0) {
    float* r = wred + warp * T::kRedFloats;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      r[h] = l_acc[h];
#pragma unroll
      for (int g = 0; g < NG; ++g) r[G + g * G + h] = zv[g][h];
    }
  }
  __syncthreads();  // every warpgroup is done with its stages and tensor memory
  constexpr int kRow = kHeadDim + 4;
  float* wm = reinterpret_cast<float*>(smem);  // [NWG][G] maxima
  float* wl = wm + NWG * G;                     // [NWG][G] l
  float* wo = wl + NWG * G;                     // [NWG][G][kRow] o
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float zsum = 0.f, lsum = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float* r = wred + (4 * u + w) * T::kRedFloats;
      lsum += r[h];
      zsum += r[G + gc * G + h];
    }
    wo[(u * G + h) * kRow + t] = broken ? 0.f : o_acc[h] + zsum;
    if (t == 0) {
      wm[u * G + h] = broken ? -INFINITY : m_ref[h];
      wl[u * G + h] = broken ? 0.f : lsum;
    }
  }
  __syncthreads();
  for (int e = tid; e < G * kHeadDim; e += C::NTH) {
    const int h = e / kHeadDim, c = e % kHeadDim;
    float ms = -INFINITY;
#pragma unroll
    for (int w = 0; w < NWG; ++w) ms = fmaxf(ms, wm[w * G + h]);
    float l = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < NWG; ++w) {
      const float a = ms == -INFINITY ? 0.f : ex2(wm[w * G + h] - ms);
      l = fmaf(wl[w * G + h], a, l);
      o = fmaf(wo[(w * G + h) * kRow + c], a, o);
    }
    store_slot<G>(part, h, c, ms, l, o);
  }
}

// One fused append task: part `half` (all 16 tokens or ring slots of the item at GQA 4, 8
// of them at GQA 8) of append item `item` of the pending reservation, for (kv-head kvh,
// K|V kv), as the append kernel does
// it, with release-increments of the (layer, request, kv-head) counters app_done[0] once
// its sink and ring rows are stored and app_done[1] once its INT2 rows are.  Before the
// wait on the preceding kernel (when this is the CTA's first work): R's bulk copy, the
// item's positions and evicted ring values, and the eviction into INT2 with its signal
// (ring items write no other INT2 rows).
template <int G, int GROUP, int NW>
__device__ void fused_append_task(const KernelParams& kp, int layer, int id, uint8_t* smem, uint32_t bar,
                                  uint32_t& phase, bool& waited, const uint16_t* k_new, const uint16_t* v_new) {
  using C = Cfg<G, GROUP, NW>;
  using namespace append_dev;
  constexpr int NTH = Shape<NW>::NTH, kSplit = append_task_split(NW);
  const int half = id % kSplit, rest = id / kSplit;
  const int kv = rest & 1, kvh = (rest >> 1) % kp.n_kv_heads, item = (rest >> 1) / kp.n_kv_heads;
  float* Rs = reinterpret_cast<float*>(smem);
  Smem& sm = *reinterpret_cast<Smem*>(smem + C::kAppendR);
  if (threadIdx.x == 0) {
    const float* R = reinterpret_cast<const float*>(kp.base + (kv ? kp.lay.R_V : kp.lay.R_K)) +
                     (size_t(layer) * kp.n_kv_heads + kvh) * kHeadDim * kHeadDim;
    fence_proxy_async();
    mbar_expect_tx(bar, C::kAppendR);
    bulk_g2s(smem_u32(Rs), R, C::kAppendR, bar);
  }
  AppendItem ait = reinterpret_cast<const AppendItem*>(kp.base + kp.lay.append_items)[item];
  constexpr int kHalf = AppendShape<NTH>::kTokens;
  ait.begin += kHalf * half;
  ait.count = max(0, min(kHalf, ait.count - kHalf * half));
  ItemState st;
  prepare_item<GROUP, NTH>(sm, kp, layer, ait, kvh, kv, st);
  unsigned* done = reinterpret_cast<unsigned*>(kp.base + kp.lay.app_done) +
                   ((size_t(layer) * kp.max_requests + (st.ok ? st.a.slot : 0)) * kp.n_kv_heads + kvh) * 2;
  auto signal = [&](int which) {
    __syncthreads();  // every store so far precedes the release below
    if (threadIdx.x == 0 && st.ok) atomic_add_acq_rel(done + which, 1u);
  };
  __syncthreads();  // row pointers visible
  evict_item<GROUP, NTH>(sm, ait, st);
  if (ait.kind == 0) signal(1);
  if (!waited) {
    pdl_wait();
    pdl_trigger();
    waited = true;
  }
  const bool ok = mbar_wait(bar, phase);
  if (!ok) {
    if (threadIdx.x == 0) flag(kp, OSCAR_FLAG_TIMEOUT);
    mbar_wait(bar, phase);  // drain (bounded) before the memory is reused
  }
  phase ^= 1u;
  __syncthreads();
  if (ok) finish_item<GROUP, NTH>(sm, Rs, kp, layer, ait, kvh, kv, st, k_new, v_new, [&] { signal(0); });
  else signal(0);
  if (ait.kind != 0) signal(1);
}

// CM: INT2 value pages channel-major, INT2 items on the tcgen05 tensor cores (never fused).
// FOLD: the plan's rotations are folded into the model (q~ in, o~ out).
template <int G, int GROUP, bool FUSED, int NW, bool CM, bool FOLD = false>
__global__ void __launch_bounds__(Shape<NW>::NTH, Cfg<G, GROUP, NW, CM>::kPerSM)
    split_kernel(KernelParams kp, int layer, const uint16_t* __restrict__ q, uint8_t* __restrict__ partials,
                 uint16_t* __restrict__ out, float* __restrict__ out_f32, const uint16_t* __restrict__ k_new,
                 const uint16_t* __restrict__ v_new) {
  static_assert(!(FUSED && CM), "the channel-major format appends in its own launch");
  constexpr bool fused = FUSED;
  extern __shared__ __align__(128) uint8_t smem[];
  using C = Cfg<G, GROUP, NW, CM>;
  constexpr int kWarps = C::NW, kThreads = C::NTH;
  int* s_last = reinterpret_cast<int*>(smem + C::kCtl + kWarps * kStages * 8);
  int* s_next = s_last + 1;
  uint64_t* merge_bar = reinterpret_cast<uint64_t*>(smem + C::kCtl + kWarps * kStages * 8 + 8);
  uint64_t* slab_bar = merge_bar + 1;
  int* s_poison = reinterpret_cast<int*>(slab_bar + 1);
  float* qin = reinterpret_cast<float*>(smem + C::kQin);
  float* qts = reinterpret_cast<float*>(smem + C::kQts);
  float* qss = reinterpret_cast<float*>(smem + C::kQss);
  if (threadIdx.x == 0) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kCtl);
    for (int i = 0; i < kWarps * kStages; ++i) mbar_init(smem_u32(&bars[i]), 1);
    mbar_init(smem_u32(merge_bar), 1);
    mbar_init(smem_u32(slab_bar), 1);
    *s_poison = 0;
    if constexpr (CM)
      for (int i = 0; i < C::NWG; ++i) mbar_init(smem_u32(reinterpret_cast<uint64_t*>(smem + C::kCtlMma) + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if constexpr (CM) {  // each warpgroup's tensor-memory columns, held until the CTA exits
    if (threadIdx.x < 32) tmem::alloc(smem_u32(smem + C::kCtlTmem), C::kTmemCols);
    tmem::fence_before();
  }
  __syncthreads();
  uint32_t tmem_base = 0, mma_phase = 0;
  if constexpr (CM) {
    tmem::fence_after();
    tmem_base = *reinterpret_cast<const uint32_t*>(smem + C::kCtlTmem);
  }
  // The plan, the page table and R_K were uploaded before the preceding kernels; of the
  // pages, only those wholly below H_pre are final before the wait (a preceding append may
  // still be writing the rest), so the first item copies those early.  Fused launches put
  // the reservation's append tasks (item x kv-head x K|V) ahead of the decode items.
  const int* counts = reinterpret_cast<const int*>(kp.base + kp.lay.decode_counts);
  const int n_items = counts[0];
  const int n_app =
      fused ? reinterpret_cast<const int*>(kp.base + kp.lay.append_counts)[0] * kp.n_kv_heads * 2 * append_task_split(NW)
            : 0;
  const WorkQueue wq{reinterpret_cast<unsigned*>(kp.base + kp.lay.sched), n_items, n_app, counts[2]};
  unsigned* app_done = reinterpret_cast<unsigned*>(kp.base + kp.lay.app_done);
  bool waited = false;
  uint32_t phase_bits = 0, merge_phase = 0, slab_phase = 0;
  // (a CTA whose page copies did not land takes no further work: *s_poison, written before
  // the item's last barriers)
  for (int id = wq.first(); id >= 0; id = *s_poison ? -1 : wq.next(s_next)) {
    if constexpr (FUSED) {
      if (id < n_app) {
        fused_append_task<G, GROUP, NW>(kp, layer, id, smem, smem_u32(merge_bar), merge_phase, waited, k_new, v_new);
        fence_proxy_async();  // generic use of the memory is over before later bulk copies
        continue;
      }
    }
    const int ix = id - n_app;
    const DecodeItem it = reinterpret_cast<const DecodeItem*>(kp.base + kp.lay.decode_items)[ix];
    const DecodeReq dr = reinterpret_cast<const DecodeReq*>(kp.base + kp.lay.decode_reqs)[it.req];
    const bool slot_ok = dr.slot >= 0 && dr.slot < kp.max_requests;
    // rows this launch's append tasks of (request, kv-head) write: an item marked dependent
    // waits for them first; INT2 pages at or above H_pre are waited for per warp
    const bool pending = fused && slot_ok && dr.app_expect > 0;
    const bool dep = pending && it.dep != kDepNone;
    const unsigned* ctrs = app_done + ((size_t(layer) * kp.max_requests + (slot_ok ? dr.slot : 0)) * kp.n_kv_heads + it.kvh) * 2;
    uint32_t pre_mask = 0;
    bool prestaged = false;
    if (it.kind == 1 && slot_ok && it.split > it.begin) {
      bf16_item_prestage<NW>(kp, layer, it, dr, smem);
      prestaged = true;
    }
    if (!CM && it.kind == 0 && slot_ok) {
      const int warp = threadIdx.x >> 5;
      const int n_my = it.end - it.begin > warp ? (it.end - it.begin - warp + kWarps - 1) / kWarps : 0;
      for (int k = 0; k < min(kStages, n_my); ++k) {
        const int lp = it.begin + warp + kWarps * k;
        if (((waited && !pending) || (lp + 1) * kPage <= dr.H_pre) && int2_issue_page<G, GROUP, NW>(kp, layer, it, dr, k, smem))
          pre_mask |= 1u << k;
      }
    }
    constexpr bool folded = FOLD;  // q arrives rotated and the output stays rotated
    if (!folded && threadIdx.x == 0 && it.slot == it.head_first)  // R_V^T for the merge of this (request, kv-head)
      bulk_prefetch_l2(reinterpret_cast<const float*>(kp.base + kp.lay.R_Vt) +
                           (size_t(layer) * kp.n_kv_heads + it.kvh) * kHeadDim * kHeadDim,
                       kHeadDim * kHeadDim * 4);
    float rk[Shape<NW>::kRows];
    if (!folded) load_rk_cols<NW>(kp, layer, it.kvh, rk);
    if (!waited) {
      pdl_wait();
      pdl_trigger();
      waited = true;
    }
    const size_t head0 = size_t(it.req) * kp.n_q_heads + size_t(it.kvh) * G;
    if (folded) load_q_folded<G, NW>(q + head0 * kHeadDim, qts, qss);
    else rotate_q<G, NW>(q + head0 * kHeadDim, rk, qin, qts, qss);
    // rows this launch's append tasks write: wait for their signal (all threads)
    auto wait_dep = [&] {
      if (!dep) return;
      const unsigned* ctr = ctrs + (it.dep == kDepPages ? 1 : 0);
      if (threadIdx.x == 0 && !wait_counter(ctr, unsigned(dr.app_expect), kp.counter_polls))
        flag(kp, OSCAR_FLAG_TIMEOUT);
      __syncthreads();
      fence_proxy_async_global();  // the append's rows, seen through the acquire, before bulk copies
    };
    if (it.kind == 0) wait_dep();
    uint8_t* part = partials + size_t(it.slot) * PartialSlot<G>::kBytes;
    if (!slot_ok) {
      if (threadIdx.x == 0) flag(kp, OSCAR_FLAG_BAD_SLOT);
      for (int e = threadIdx.x; e < G * kHeadDim; e += kThreads) store_slot<G>(part, e / kHeadDim, e % kHeadDim, -INFINITY, 0.f, 0.f);
    } else if (it.kind == 0) {
      if constexpr (CM)
        int2_tc_item<G, GROUP, NW>(kp, layer, it, dr, qts, qss, part, smem, phase_bits, mma_phase, tmem_base, s_poison);
      else
        int2_pages_item<G, GROUP, NW>(kp, layer, it, dr, qts, qss, part, smem, phase_bits, pre_mask,
                                      pending && it.dep == kDepNone ? ctrs + 1 : nullptr, s_poison);
    } else {
      bf16_tokens_item<G, NW>(kp, layer, it, dr, qts, part, smem, prestaged, wait_dep);
    }
    // ---- merge by the last CTA of (request, kv-head): R_V^T is fetched as soon as this CTA
    // knows it merges, the partial slots are bulk-copied after it
    MergeAcc<G, kThreads> acc;
    if (merge_partial<G, kThreads>(kp, it, partials, acc, s_last, smem + C::kSlabOff, C::kSlabSlots,
                                   smem_u32(slab_bar), slab_phase,
                                   [&] {
                                     if (!folded) fetch_rvt(kp, layer, it.kvh, smem, smem_u32(merge_bar));
                                   })) {
      // every item of (request, kv-head) is done, so are its waits: ready for the next launch
      // (subtracting the launch's count: a task's last increment may still be on its way)
      if (fused && slot_ok && dr.app_expect > 0 && threadIdx.x == 0) {
        unsigned* ctr = app_done + ((size_t(layer) * kp.max_requests + dr.slot) * kp.n_kv_heads + it.kvh) * 2;
        atomicSub(ctr, unsigned(dr.app_expect));
        atomicSub(ctr + 1, unsigned(dr.app_expect));
      }
      if (folded) finish_output_folded<G, NW>(kp, it, acc, out, out_f32);
      else finish_output<G, NW>(kp, it, acc, out, out_f32, smem, smem_u32(merge_bar), merge_phase);
    }
    // generic-proxy use of the stage memory is over before the next item's bulk copies
    fence_proxy_async();
  }
  wq.leave();
  if constexpr (CM) {  // every MMA of this CTA was waited for
    tmem::fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
      tmem::fence_after();
      tmem::dealloc(tmem_base, C::kTmemCols);
    }
  }
}

template <int G, int GROUP, bool FUSED, int NW, bool CM>
int resident_ctas_t(int n_sm) {
  using C = Cfg<G, GROUP, NW, CM>;
  static int resident = 0;  // CTAs of split_kernel that fit on the GPU at once
  if (resident == 0) {
    int e = int(cudaFuncSetAttribute(split_kernel<G, GROUP, FUSED, NW, CM>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes));
    if (!e)
      e = int(cudaFuncSetAttribute(split_kernel<G, GROUP, FUSED, NW, CM, true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes));
    int per_sm = 0;
    if (!e)
      e = int(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, split_kernel<G, GROUP, FUSED, NW, CM>, C::NTH,
                                                            C::kSmemBytes));
    if (CM && !e) {
      // The runtime's occupancy for a kernel that allocates tensor memory assumes one CTA
      // per SM; registers (128 a thread), shared memory and the 512 tensor-memory columns
      // of an SM decide here.  (A CTA that did not fit would start when another exits:
      // no CTA of this kernel waits for another.)
      int dev = 0, smem_sm = 0;
      e = int(cudaGetDevice(&dev));
      if (!e) e = int(cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev));
      const int by_regs = 65536 / (C::NTH * 128), by_smem = smem_sm / (C::kSmemBytes + 1024);
      per_sm = by_regs < by_smem ? by_regs : by_smem;
      if (per_sm * C::kTmemCols > 512) per_sm = 512 / C::kTmemCols;
    }
    if (e) return -e;
    resident = (per_sm > 0 ? per_sm : 1) * n_sm;
    // One CTA per SM (16-warp shape): leave a few SMs to the preceding launch's last CTAs
    // (its final merges), so that no CTA of this launch waits for an SM to drain.
    if (NW == 16 && resident > 4 * kSpareSMs) resident -= kSpareSMs;
  }
  return resident;
}

// The decode and the fused append + decode kernels of a shape get one plan: the smaller
// resident count of the two.
template <int G, int GROUP, int NW, bool CM>
int resident_ctas(int n_sm) {
  if constexpr (CM) return resident_ctas_t<G, GROUP, false, NW, true>(n_sm);
  const int a = resident_ctas_t<G, GROUP, false, NW, false>(n_sm), b = resident_ctas_t<G, GROUP, true, NW, false>(n_sm);
  if (a < 0) return a;
  if (b < 0) return b;
  return a < b ? a : b;
}

template <int G, int GROUP, int NW, bool CM>
int launch_decode_t(const KernelParams& kp, int layer, const void* q, void* out, float* out_f32, uint8_t* ws,
                    const DecodeWorkspace& wl, int n_sm, void* stream, int* launches, const void* k_new,
                    const void* v_new, bool fused) {
  using C = Cfg<G, GROUP, NW, CM>;
  uint8_t* partials = ws + wl.partials;
  const int resident = resident_ctas<G, GROUP, NW, CM>(n_sm);
  if (resident < 0) return -resident;
  // persistent-style grid: every resident CTA slot, each looping over work items, so a
  // captured launch serves later plans with other item counts
  const uint16_t* qb = static_cast<const uint16_t*>(q);
  uint16_t* ob = static_cast<uint16_t*>(out);
  const uint16_t* kb = static_cast<const uint16_t*>(k_new);
  const uint16_t* vb = static_cast<const uint16_t*>(v_new);
  auto go = [&](auto kernel) {
    return launch_ex(kernel, dim3(resident), dim3(C::NTH), size_t(C::kSmemBytes), stream, kp, layer, qb, partials, ob,
                     out_f32, kb, vb);
  };
  int e;
  if constexpr (CM)
    e = kp.folded ? go(split_kernel<G, GROUP, false, NW, true, true>) : go(split_kernel<G, GROUP, false, NW, true, false>);
  else if (fused)
    e = kp.folded ? go(split_kernel<G, GROUP, true, NW, false, true>) : go(split_kernel<G, GROUP, true, NW, false, false>);
  else
    e = kp.folded ? go(split_kernel<G, GROUP, false, NW, false, true>)
                  : go(split_kernel<G, GROUP, false, NW, false, false>);
  if (!e) *launches += 1;
  return e;
}

}  // namespace

int decode_resident_ctas(int gqa, int group, bool wide, bool cm, int n_sm) {
  const bool w = wide && gqa == 4;
  if (cm) {
    if (gqa == 4 && group == 128) return w ? resident_ctas<4, 128, 16, true>(n_sm) : resident_ctas<4, 128, 8, true>(n_sm);
    if (gqa == 4 && group == 32) return w ? resident_ctas<4, 32, 16, true>(n_sm) : resident_ctas<4, 32, 8, true>(n_sm);
    if (gqa == 8 && group == 128) return resident_ctas<8, 128, 8, true>(n_sm);
    return n_sm;
  }
  if (gqa == 4 && group == 128) return w ? resident_ctas<4, 128, 16, false>(n_sm) : resident_ctas<4, 128, 8, false>(n_sm);
  if (gqa == 4 && group == 32) return w ? resident_ctas<4, 32, 16, false>(n_sm) : resident_ctas<4, 32, 8, false>(n_sm);
  if (gqa == 8 && group == 128) return resident_ctas<8, 128, 8, false>(n_sm);
  if (gqa == 8 && group == 32) return resident_ctas<8, 32, 8, false>(n_sm);
  return n_sm;
}

int launch_decode(const KernelParams& kp, int layer, const void* q, void* out, float* out_f32, uint8_t* ws,
                  const DecodeWorkspace& wl, bool wide, int n_sm, void* stream, int* launches, const void* k_new,
                  const void* v_new, bool fused) {
  const bool w = wide && kp.gqa == 4;
#define OSCAR_DECODE_CASE(G_, GROUP_, NW_, CM_)                                                            \
  if (kp.gqa == G_ && kp.group == GROUP_ && (NW_ == 16) == w && bool(kp.v_cm) == CM_)                     \
    return launch_decode_t<G_, GROUP_, NW_, CM_>(kp, layer, q, out, out_f32, ws, wl, n_sm, stream, launches, \
                                                 k_new, v_new, fused);
  OSCAR_DECODE_CASE(4, 128, 16, false)
  OSCAR_DECODE_CASE(4, 128, 8, false)
  OSCAR_DECODE_CASE(4, 32, 16, false)
  OSCAR_DECODE_CASE(4, 32, 8, false)
  OSCAR_DECODE_CASE(8, 128, 8, false)
  OSCAR_DECODE_CASE(8, 32, 8, false)
  OSCAR_DECODE_CASE(4, 128, 16, true)
  OSCAR_DECODE_CASE(4, 128, 8, true)
  OSCAR_DECODE_CASE(4, 32, 16, true)
  OSCAR_DECODE_CASE(4, 32, 8, true)
  OSCAR_DECODE_CASE(8, 128, 8, true)
#undef OSCAR_DECODE_CASE
  return int(cudaErrorInvalidValue);
}


// ---------------------------------------------------------------- no-allocation variant
// Decode scratch (the split partials) owned by the
// library itself, for callers that cannot allocate device memory.  Every GPU that loads
// the library holds this array until the process exits; all calls share it.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

size_t static_scratch_bytes() { return kStaticScratchBytes; }

namespace {
// Device address of g_decode_scratch on the current device.  The host-side name of the
// array is only a stand-in, so the address is looked up with the device current, on every
// call (cheap after the first, which loads the module): a cached address would go stale
// when a host framework tears the context down and makes a new one.
int scratch_address(uint8_t** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess) return int(e);
  *out = static_cast<uint8_t*>(p);
  return 0;
}
}  // namespace

int launch_decode_static_scratch(const KernelParams& kp, int layer, const void* q, void* out, float* out_f32,
                                 const DecodeWorkspace& wl, bool wide, int n_sm, void* stream, int* launches,
                                 bool* too_big) {
  *too_big = wl.total > kStaticScratchBytes;
  if (*too_big) return int(cudaErrorInvalidValue);
  uint8_t* ws = nullptr;
  int e = scratch_address(&ws);
  if (e) return e;
  // Nothing in the scratch has to start at zero: every work item writes its partial
  // before the merge reads it.
  return launch_decode(kp, layer, q, out, out_f32, ws, wl, wide, n_sm, stream, launches);
}

}  // namespace oscar
