// Offline calibration of one layer on the GPU, in fp64 (sm_103a).
//
// OSCAR technical summary (gist.science), §2.2-A, steps A.1 to A.4:
//   A.1  query-aware key target C_Q = (1/N) sum q^T q and score-aware value target
//        C_S = (1/N) V^T S^T S V, S the attention probabilities (so C_S = O^T O / N with
//        O = S V);
//   A.2  eigenbases U_Q, U_S of C_Q and C_S;
//   A.3  R_K = U_Q H_Had P_br, R_V = U_S H_Had P_br;
//   A.4  per-layer clip thresholds on the rotated calibration activations.
// Readings where the page is silent (the same as the offline CPU calibration's): the G
// query heads of a kv-head are pooled (N counts token x head pairs), S is the causal
// softmax of q k^T / sqrt(d), eigenvalues descending with each eigenvector's
// largest-magnitude entry positive (the first such entry), H_Had the Sylvester matrix
// / sqrt(d), P_br sending e_j to e_rev(j), the clip the nearest-rank percentile of
// |R^T x| over all tokens and channels, with R as stored (fp32).
//
// Kernels (all fp64 arithmetic):
//   cov_kernel      C = X^T X / rows, split over row chunks; partial tiles summed in a
//                   fixed order by cov_reduce_kernel (deterministic)
//   attn_kernel     O = causal softmax(Q K^T / sqrt(d)) V per query head, online softmax
//   eigen_kernel    cyclic Jacobi on a 2-CTA cluster: CTA 0 holds the matrix, CTA 1 the
//                   accumulated rotations; the rotations of each round are sent to CTA 1
//                   through distributed shared memory (round-robin pairing, 64 disjoint
//                   pairs a round, 127 rounds a sweep)
//   compose_kernel  R = U H P: fast Walsh-Hadamard transform of each row of U, columns
//                   taken in bit-reversed order
//   rotate_abs_kernel, select_kernel
//                   |x R| for every token and channel, then the rank-th smallest by an
//                   8-pass radix select on the fp64 bit patterns (non-negative doubles
//                   order like their bits)
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "oscar_internal.h"

namespace cg = cooperative_groups;

namespace oscar {
namespace {

constexpr int D = kHeadDim;      // 128
constexpr int kCovRows = 2048;   // rows of one split of the covariance sum
constexpr int kCovStage = 32;    // rows staged in shared memory at a time
constexpr int kAttnRows = 32;    // query rows of one attention CTA
constexpr int kAttnKeys = 64;    // keys staged at a time
constexpr int kLd = D + 1;       // padded row of a staged fp64 matrix
constexpr int kMaxSweeps = 30;   // Jacobi sweeps (converges in about 8-12)

__device__ __forceinline__ double ld_in(const uint16_t* p) { return double(bf16_f32(*p)); }
__device__ __forceinline__ double ld_in(const double* p) { return *p; }

// Row r of the covariance input of matrix m (a kv-head): for the key target the rows are
// (token n, query head g) of q; for the value target the rows of O.
struct QRows {  // q bf16 [N][H_q][d], rows r = n G + g of kv-head m
  const uint16_t* q;
  int n_q_heads, G;
  __device__ const uint16_t* row(int m, int r) const {
    const int n = r / G, g = r % G;
    return q + (size_t(n) * n_q_heads + size_t(m) * G + g) * D;
  }
};
struct ORows {  // O fp64 [H_kv][G][N][d], rows r = g N + n of kv-head m
  const double* o;
  int rows;
  __device__ const double* row(int m, int r) const { return o + (size_t(m) * rows + r) * D; }
};

// Partial covariance of rows [split * kCovRows, +kCovRows) of matrix m, 64 x 64 tile
// (ti, tj): grid (4 tiles, splits, matrices), 256 threads, each a 4 x 4 block.
template <typename Rows>
__global__ void __launch_bounds__(256) cov_kernel(Rows X, int rows, double* partials) {
  __shared__ double si[kCovStage][64 + 1], sj[kCovStage][64 + 1];
  const int tile = blockIdx.x, split = blockIdx.y, m = blockIdx.z;
  const int ti = tile >> 1, tj = tile & 1, t = threadIdx.x, a = t >> 4, b = t & 15;
  const int r0 = split * kCovRows, r1 = min(rows, r0 + kCovRows);
  double acc[4][4] = {};
  for (int rs = r0; rs < r1; rs += kCovStage) {
    for (int e = t; e < kCovStage * 64; e += 256) {
      const int rr = e / 64, c = e % 64, r = rs + rr;
      si[rr][c] = r < r1 ? ld_in(X.row(m, r) + 64 * ti + c) : 0.0;
      sj[rr][c] = r < r1 ? ld_in(X.row(m, r) + 64 * tj + c) : 0.0;
    }
    __syncthreads();
    for (int rr = 0; rr < kCovStage; ++rr) {
      double x[4], y[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        x[u] = si[rr][4 * a + u];
        y[u] = sj[rr][4 * b + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fma(x[u], y[v], acc[u][v]);
    }
    __syncthreads();
  }
  double* out = partials + (size_t(m) * gridDim.y + split) * D * D;
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) out[(64 * ti + 4 * a + u) * D + 64 * tj + 4 * b + v] = acc[u][v];
}

// C[m] = (sum over splits, in order) / rows; grid (matrices), 256 threads.
__global__ void __launch_bounds__(256) cov_reduce_kernel(const double* partials, int splits, int rows, double* C) {
  const int m = blockIdx.x;
  for (int e = threadIdx.x; e < D * D; e += 256) {
    double s = 0.0;
    for (int k = 0; k < splits; ++k) s += partials[(size_t(m) * splits + k) * D * D + e];
    C[size_t(m) * D * D + e] = s / double(rows);
  }
}

// O[m][g][n] = sum_{j <= n} softmax_j(q_n . k_j / sqrt(d)) v_j for query head g of kv-head
// m, fp64 online softmax.  Grid (query blocks of kAttnRows, G, kv-heads), 256 threads:
// warp w owns query rows 4w .. 4w + 3 of the block; for the logits lane l takes keys l and
// l + 32 of a staged block of kAttnKeys; for the output lane l owns channels l + 32 u.
__global__ void __launch_bounds__(256) attn_kernel(const uint16_t* q, const uint16_t* k, const uint16_t* v, int N,
                                                   int n_q_heads, int n_kv_heads, double* O) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  double* sq = reinterpret_cast<double*>(smem_raw);  // [kAttnRows][D]
  double* sk = sq + kAttnRows * D;                    // [kAttnKeys][kLd]
  double* sv = sk + kAttnKeys * kLd;                  // [kAttnKeys][D]
  double* sp = sv + kAttnKeys * D;                    // [8 warps][4 rows][kAttnKeys]
  const int G = n_q_heads / n_kv_heads;
  const int n0 = blockIdx.x * kAttnRows, g = blockIdx.y, m = blockIdx.z;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const double inv_sqrt_d = 1.0 / sqrt(double(D));
  for (int e = t; e < kAttnRows * D; e += 256) {
    const int r = e / D, c = e % D, n = n0 + r;
    sq[e] = n < N ? double(bf16_f32(q[(size_t(n) * n_q_heads + size_t(m) * G + g) * D + c])) : 0.0;
  }
  double mx[4], l[4], o[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    mx[r] = -INFINITY;
    l[r] = 0.0;
#pragma unroll
    for (int u = 0; u < 4; ++u) o[r][u] = 0.0;
  }
  const int key_end = min(N, n0 + kAttnRows);  // keys any row of the block attends to
  for (int j0 = 0; j0 < key_end; j0 += kAttnKeys) {
    __syncthreads();  // the previous block's keys are used up (and sq is written)
    for (int e = t; e < kAttnKeys * D; e += 256) {
      const int r = e / D, c = e % D, j = j0 + r;
      const size_t src = (size_t(j) * n_kv_heads + m) * D + c;
      sk[r * kLd + c] = j < N ? double(bf16_f32(k[src])) : 0.0;
      sv[r * D + c] = j < N ? double(bf16_f32(v[src])) : 0.0;
    }
    __syncthreads();
    double s[4][2];
#pragma unroll
    for (int r = 0; r < 4; ++r) s[r][0] = s[r][1] = 0.0;
    const double* q0 = sq + (4 * warp) * D;
    for (int c = 0; c < D; ++c) {
      const double ka = sk[lane * kLd + c], kb = sk[(lane + 32) * kLd + c];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const double qv = q0[r * D + c];
        s[r][0] = fma(qv, ka, s[r][0]);
        s[r][1] = fma(qv, kb, s[r][1]);
      }
    }
    double* pw = sp + warp * 4 * kAttnKeys;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int n = n0 + 4 * warp + r;
      const int ja = j0 + lane, jb = ja + 32;
      const double la = (ja <= n && n < N) ? s[r][0] * inv_sqrt_d : -INFINITY;
      const double lb = (jb <= n && n < N) ? s[r][1] * inv_sqrt_d : -INFINITY;
      double bm = fmax(la, lb);
      for (int off = 16; off > 0; off >>= 1) bm = fmax(bm, __shfl_xor_sync(0xffffffffu, bm, off));
      const double mnew = fmax(mx[r], bm);
      if (mnew == -INFINITY) {  // no key of this block for this row yet
        pw[r * kAttnKeys + lane] = 0.0;
        pw[r * kAttnKeys + lane + 32] = 0.0;
        continue;
      }
      const double alpha = mx[r] == -INFINITY ? 0.0 : exp(mx[r] - mnew);
      const double pa = la == -INFINITY ? 0.0 : exp(la - mnew);
      const double pb = lb == -INFINITY ? 0.0 : exp(lb - mnew);
      double ps = pa + pb;
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l[r] = l[r] * alpha + ps;
#pragma unroll
      for (int u = 0; u < 4; ++u) o[r][u] *= alpha;
      mx[r] = mnew;
      pw[r * kAttnKeys + lane] = pa;
      pw[r * kAttnKeys + lane + 32] = pb;
    }
    __syncwarp();
    for (int j = 0; j < kAttnKeys; ++j) {
      double vv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) vv[u] = sv[j * D + lane + 32 * u];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const double p = pw[r * kAttnKeys + j];
#pragma unroll
        for (int u = 0; u < 4; ++u) o[r][u] = fma(p, vv[u], o[r][u]);
      }
    }
    __syncwarp();
  }
  const int rows = G * N;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int n = n0 + 4 * warp + r;
    if (n >= N) continue;
    double* dst = O + (size_t(m) * rows + size_t(g) * N + n) * D;
#pragma unroll
    for (int u = 0; u < 4; ++u) dst[lane + 32 * u] = o[r][u] / l[r];
  }
}

// Pair k (0..63) of round r (0..126) of the round-robin tournament on 128 indices: index
// 127 meets r; the others meet in pairs (r + k) mod 127, (r - k) mod 127.  Over the 127
// rounds every pair of indices meets exactly once.
__device__ __forceinline__ void tournament(int r, int k, int& p, int& q) {
  if (k == 0) {
    p = r;
    q = 127;
  } else {
    p = (r + k) % 127;
    q = (r - k + 127) % 127;
  }
  if (p > q) {
    const int x = p;
    p = q;
    q = x;
  }
}

struct EigenSmem {
  double M[D][kLd];   // CTA 0: the matrix; CTA 1: the accumulated rotations V
  double cs[2][64][2];  // CTA 1: the (c, s) of each pair of a round (written by CTA 0), double-buffered
  double lam[D];      // CTA 1: the eigenvalues (written by CTA 0)
  int rotated;        // CTA 0: rotations applied in the current sweep
  int done;           // both: the sweep loop is over (CTA 1's copy written by CTA 0)
};

// Cyclic Jacobi eigendecomposition of symmetric C[mat] (fp64, 128 x 128).  Cluster of two
// CTAs per matrix, 512 threads each.  A rotation of pair (p, q) is skipped when
// |A_pq| <= eps sqrt(|A_pp A_qq|) (eps = 2^-53); the sweeps end after one with no rotation
// (at most kMaxSweeps).  Output: U [mat] columns = eigenvectors, eigenvalues descending,
// each column's first largest-magnitude entry positive; lam [mat][128]; sweeps [mat].
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(512)
    eigen_kernel(const double* C, double* U, double* lam_out, int* sweeps_out) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  EigenSmem& sm = *reinterpret_cast<EigenSmem*>(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const int mat = blockIdx.x / 2, t = threadIdx.x;
  EigenSmem& peer = *cluster.map_shared_rank(&sm, 1);  // CTA 1's shared memory (CTA 0 writes it)
  const double* Cm = C + size_t(mat) * D * D;
  for (int e = t; e < D * D; e += 512) {
    const int i = e / D, j = e % D;
    sm.M[i][j] = rank == 0 ? Cm[e] : (i == j ? 1.0 : 0.0);
  }
  if (t == 0) {
    sm.done = 0;
    sm.rotated = 0;
  }
  cluster.sync();
  const double eps = 1.1102230246251565e-16;  // 2^-53
  int sweep = 0;
  for (; sweep < kMaxSweeps; ++sweep) {
    for (int r = 0; r < 127; ++r) {
      const int buf = r & 1;
      if (rank == 0 && t < 64) {
        int p, q;
        tournament(r, t, p, q);
        const double app = sm.M[p][p], aqq = sm.M[q][q], apq = sm.M[p][q];
        double c = 1.0, s = 0.0;
        if (apq != 0.0 && fabs(apq) > eps * sqrt(fabs(app * aqq))) {
          const double tau = (aqq - app) / (2.0 * apq);
          const double tt = tau >= 0.0 ? 1.0 / (tau + sqrt(1.0 + tau * tau)) : -1.0 / (-tau + sqrt(1.0 + tau * tau));
          c = 1.0 / sqrt(1.0 + tt * tt);
          s = tt * c;
          atomicAdd(&sm.rotated, 1);
        }
        sm.cs[buf][t][0] = c;
        sm.cs[buf][t][1] = s;
        peer.cs[buf][t][0] = c;
        peer.cs[buf][t][1] = s;
      }
      cluster.sync();  // this round's rotations are in both CTAs
      if (rank == 0) {
        // rows: A <- J^T A
        for (int e = t; e < 64 * D; e += 512) {
          const int k = e / D, j = e % D;
          int p, q;
          tournament(r, k, p, q);
          const double c = sm.cs[buf][k][0], s = sm.cs[buf][k][1];
          if (s == 0.0) continue;
          const double ap = sm.M[p][j], aq = sm.M[q][j];
          sm.M[p][j] = c * ap - s * aq;
          sm.M[q][j] = s * ap + c * aq;
        }
        __syncthreads();
        // columns: A <- A J
        for (int e = t; e < 64 * D; e += 512) {
          const int k = e / D, i = e % D;
          int p, q;
          tournament(r, k, p, q);
          const double c = sm.cs[buf][k][0], s = sm.cs[buf][k][1];
          if (s == 0.0) continue;
          const double ap = sm.M[i][p], aq = sm.M[i][q];
          sm.M[i][p] = c * ap - s * aq;
          sm.M[i][q] = s * ap + c * aq;
        }
        __syncthreads();
      } else {
        // V <- V J
        for (int e = t; e < 64 * D; e += 512) {
          const int k = e / D, i = e % D;
          int p, q;
          tournament(r, k, p, q);
          const double c = sm.cs[buf][k][0], s = sm.cs[buf][k][1];
          if (s == 0.0) continue;
          const double vp = sm.M[i][p], vq = sm.M[i][q];
          sm.M[i][p] = c * vp - s * vq;
          sm.M[i][q] = s * vp + c * vq;
        }
      }
    }
    // end of a sweep: CTA 0 decides, CTA 1 gets the decision before either reads it
    if (rank == 0 && t == 0) {
      const int d = sm.rotated == 0;
      sm.done = d;
      peer.done = d;
      sm.rotated = 0;
    }
    cluster.sync();
    if (sm.done) break;
  }
  if (rank == 0)
    for (int i = t; i < D; i += 512) peer.lam[i] = sm.M[i][i];
  cluster.sync();  // CTA 0 writes nothing more into CTA 1; it may exit
  if (rank == 0) return;
  // CTA 1: order by eigenvalue, descending (ties: lower index first), fix signs
  __shared__ int order[D];  // order[k] = index of the k-th largest eigenvalue
  if (t < D) {
    const double li = sm.lam[t];
    int rk = 0;
    for (int j = 0; j < D; ++j) rk += (sm.lam[j] > li) || (sm.lam[j] == li && j < t);
    order[rk] = t;
  }
  __syncthreads();
  if (t < D) {
    const int src = order[t];
    // first entry of largest magnitude of column src
    int arg = 0;
    double best = -1.0;
    for (int i = 0; i < D; ++i) {
      const double a = fabs(sm.M[i][src]);
      if (a > best) {
        best = a;
        arg = i;
      }
    }
    const double sign = sm.M[arg][src] < 0.0 ? -1.0 : 1.0;
    double* Um = U + size_t(mat) * D * D;
    for (int i = 0; i < D; ++i) Um[i * D + t] = sign * sm.M[i][src];
    lam_out[size_t(mat) * D + t] = sm.lam[src];
  }
  if (t == 0 && sweeps_out) sweeps_out[mat] = sweep + 1;
}

__device__ __forceinline__ int bitrev7(int j) { return int(__brev(unsigned(j)) >> 25); }

// R[mat] = U H P (fp32 out): row i of U H is the Walsh-Hadamard transform of row i of U
// over 1/sqrt(d); R[i][j] = (U H)[i][rev(j)].  U = nullptr: the identity (Hadamard-only).
// Grid (matrices), 128 threads (thread i: row i); dynamic shared memory D x kLd doubles.
__global__ void __launch_bounds__(128) compose_kernel(const double* U, float* R0, float* R1, int n_half) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  double* row = reinterpret_cast<double*>(smem_raw) + threadIdx.x * kLd;
  const int mat = blockIdx.x, i = threadIdx.x;
  for (int j = 0; j < D; ++j) row[j] = U ? U[size_t(mat) * D * D + i * D + j] : (i == j ? 1.0 : 0.0);
  for (int h = 1; h < D; h <<= 1)
    for (int j = 0; j < D; j += 2 * h)
      for (int u = j; u < j + h; ++u) {
        const double a = row[u], b = row[u + h];
        row[u] = a + b;
        row[u + h] = a - b;
      }
  const double inv = 1.0 / sqrt(double(D));
  float* R = (mat < n_half ? R0 : R1) + size_t(mat % n_half) * D * D;
  for (int j = 0; j < D; ++j) R[i * D + j] = float(row[bitrev7(j)] * inv);
}
constexpr size_t kComposeSmem = size_t(D) * kLd * 8;

// keys[mat][n * d + j] = bits of |sum_i x[n][i] R[i][j]| (fp64; x bf16, R fp32 as
// stored): mat < n_half are the keys (x = k, R = R_K of head mat), the rest the values.
// Grid (token blocks of kRotTok, matrices), 128 threads: thread j holds column j of R in
// registers and sums i = 0..127 in order for each token.
constexpr int kRotTok = 64;
__global__ void __launch_bounds__(128) rotate_abs_kernel(const uint16_t* k, const uint16_t* v, const float* RK,
                                                         const float* RV, int N, int n_kv_heads,
                                                         unsigned long long* keys) {
  __shared__ double xs[16][D];
  const int mat = blockIdx.y, h = mat % n_kv_heads, j = threadIdx.x;
  const uint16_t* X = mat < n_kv_heads ? k : v;
  const float* R = (mat < n_kv_heads ? RK : RV) + size_t(h) * D * D;
  float rc[D];
#pragma unroll
  for (int i = 0; i < D; ++i) rc[i] = R[i * D + j];
  for (int n0 = blockIdx.x * kRotTok; n0 < min(N, (blockIdx.x + 1) * kRotTok); n0 += 16) {
    __syncthreads();
    for (int e = j; e < 16 * D; e += 128) {
      const int r = e / D, c = e % D, n = n0 + r;
      xs[r][c] = n < N ? double(bf16_f32(X[(size_t(n) * n_kv_heads + h) * D + c])) : 0.0;
    }
    __syncthreads();
    for (int r = 0; r < 16 && n0 + r < N; ++r) {
      double acc = 0.0;
#pragma unroll
      for (int i = 0; i < D; ++i) acc = fma(xs[r][i], double(rc[i]), acc);
      keys[size_t(mat) * N * D + size_t(n0 + r) * D + j] = __double_as_longlong(fabs(acc));
    }
  }
}

// The rank-th smallest (1-based) of n non-negative fp64 values given as bit patterns,
// by eight 8-bit radix passes from the top byte; clip[mat] = that value rounded to fp32.
// Grid (matrices), 1024 threads.
__global__ void __launch_bounds__(1024) select_kernel(const unsigned long long* keys, long n, long rank, float* clip0,
                                                      float* clip1, int n_half) {
  __shared__ unsigned hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ long s_rank;
  const int mat = blockIdx.x, t = threadIdx.x;
  const unsigned long long* x = keys + size_t(mat) * n;
  if (t == 0) {
    s_prefix = 0ull;
    s_rank = rank;
  }
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    const unsigned long long hi_mask = pass == 0 ? 0ull : ~0ull << (shift + 8);
    if (t < 256) hist[t] = 0u;
    __syncthreads();
    const unsigned long long prefix = s_prefix;
    for (long e = t; e < n; e += 1024) {
      const unsigned long long b = x[e];
      if ((b & hi_mask) == prefix) atomicAdd(&hist[(b >> shift) & 0xffu], 1u);
    }
    __syncthreads();
    if (t == 0) {
      long r = s_rank;
      int d = 0;
      while (d < 255 && long(hist[d]) < r) r -= hist[d++];
      s_rank = r;
      s_prefix = prefix | (static_cast<unsigned long long>(d) << shift);
    }
    __syncthreads();
  }
  if (t == 0) {
    const float c = float(__longlong_as_double(static_cast<long long>(s_prefix)));
    (mat < n_half ? clip0 : clip1)[mat % n_half] = c;
  }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

CalibWorkspace calib_workspace(int n_tokens, int n_q_heads, int n_kv_heads) {
  CalibWorkspace w{};
  const int G = n_q_heads / n_kv_heads;
  const int splits_q = (n_tokens * G + kCovRows - 1) / kCovRows;
  const int splits = splits_q > 0 ? splits_q : 1;
  size_t off = 0;
  w.O = off;
  off += align256(size_t(n_q_heads) * n_tokens * D * 8);
  w.partials = off;
  off += align256(size_t(2) * n_kv_heads * splits * D * D * 8);
  w.C = off;
  off += align256(size_t(2) * n_kv_heads * D * D * 8);
  w.U = off;
  off += align256(size_t(2) * n_kv_heads * D * D * 8);
  w.lam = off;
  off += align256(size_t(2) * n_kv_heads * D * 8);
  w.sweeps = off;
  off += align256(size_t(2) * n_kv_heads * 4);
  w.keys = off;
  off += align256(size_t(2) * n_kv_heads * n_tokens * D * 8);
  w.splits = splits;
  w.total = off;
  return w;
}

int launch_calibrate(const void* q, const void* k, const void* v, int n_tokens, int n_q_heads, int n_kv_heads,
                     long clip_rank, bool hadamard_only, float* R_K, float* R_V, float* clip_K, float* clip_V,
                     double* C_out, uint8_t* ws, void* stream_, int* launches) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const CalibWorkspace w = calib_workspace(n_tokens, n_q_heads, n_kv_heads);
  const int H = n_kv_heads, G = n_q_heads / n_kv_heads;
  const uint16_t* qb = static_cast<const uint16_t*>(q);
  const uint16_t* kb = static_cast<const uint16_t*>(k);
  const uint16_t* vb = static_cast<const uint16_t*>(v);
  double* O = reinterpret_cast<double*>(ws + w.O);
  double* partials = reinterpret_cast<double*>(ws + w.partials);
  double* C = C_out ? C_out : reinterpret_cast<double*>(ws + w.C);
  double* U = reinterpret_cast<double*>(ws + w.U);
  cudaError_t e = cudaSuccess;
  auto count = [&](cudaError_t r) {
    if (r == cudaSuccess) r = cudaGetLastError();
    if (r == cudaSuccess) ++*launches;
    else if (e == cudaSuccess) e = r;
  };
  if (!hadamard_only) {
    const int rows_q = n_tokens * G;
    // A.1: C_Q over the (token, query head) rows; O per query head; C_S over the rows of O
    cov_kernel<QRows><<<dim3(4, w.splits, H), 256, 0, stream>>>(QRows{qb, n_q_heads, G}, rows_q, partials);
    count(cudaSuccess);
    cov_reduce_kernel<<<H, 256, 0, stream>>>(partials, w.splits, rows_q, C);
    count(cudaSuccess);
    const size_t attn_smem = size_t(kAttnRows * D + kAttnKeys * kLd + kAttnKeys * D + 8 * 4 * kAttnKeys) * 8;
    e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(attn_smem));
    if (e != cudaSuccess) return int(e);
    attn_kernel<<<dim3((n_tokens + kAttnRows - 1) / kAttnRows, G, H), 256, attn_smem, stream>>>(
        qb, kb, vb, n_tokens, n_q_heads, n_kv_heads, O);
    count(cudaSuccess);
    double* partials_s = partials + size_t(H) * w.splits * D * D;
    cov_kernel<ORows><<<dim3(4, w.splits, H), 256, 0, stream>>>(ORows{O, rows_q}, rows_q, partials_s);
    count(cudaSuccess);
    cov_reduce_kernel<<<H, 256, 0, stream>>>(partials_s, w.splits, rows_q, C + size_t(H) * D * D);
    count(cudaSuccess);
    // A.2: eigenbases of the 2 H matrices (C_Q of every head, then C_S)
    e = cudaFuncSetAttribute(eigen_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sizeof(EigenSmem)));
    if (e != cudaSuccess) return int(e);
    eigen_kernel<<<2 * (2 * H), 512, sizeof(EigenSmem), stream>>>(C, U, reinterpret_cast<double*>(ws + w.lam),
                                                                  reinterpret_cast<int*>(ws + w.sweeps));
    count(cudaSuccess);
  }
  // A.3: R = U H P (U = I for the Hadamard-only rotation)
  e = cudaFuncSetAttribute(compose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kComposeSmem));
  if (e != cudaSuccess) return int(e);
  compose_kernel<<<2 * H, 128, kComposeSmem, stream>>>(hadamard_only ? nullptr : U, R_K, R_V, H);
  count(cudaSuccess);
  // A.4: clip = nearest-rank percentile of |R^T x| over tokens x channels
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(ws + w.keys);
  rotate_abs_kernel<<<dim3((n_tokens + kRotTok - 1) / kRotTok, 2 * H), 128, 0, stream>>>(kb, vb, R_K, R_V,
                                                                                        n_tokens, H, keys);
  count(cudaSuccess);
  select_kernel<<<2 * H, 1024, 0, stream>>>(keys, long(n_tokens) * D, clip_rank, clip_K, clip_V, H);
  count(cudaSuccess);
  return int(e);
}

}  // namespace oscar
