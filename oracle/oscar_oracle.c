/*
 * oscar_oracle.c -- plain, slow CPU oracle for the OSCAR-style 2-bit rotated KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this file;
 * only the tests, the package's smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (web pages on the method):
 *   [OSCAR summary]  "기술 요약: OSCAR - 2 비트 KV 캐시 양자화를 위한 오프라인 스펙트럴 공분산 인지 회전"
 *                    (gist.science technical summary of OSCAR).
 *   [OSCAR note]     tilnote.io note on OSCAR (paged INT2 KV, BF16 sink/recent tokens).
 *
 * What the pages fix, and what this file follows:
 *   - history tokens are stored as INT2 after the fixed rotation and clipping
 *     ([OSCAR summary] §2.2-B, mixed-precision layout); sink and recent tokens stay BF16
 *     ([OSCAR summary] §2.2-B; [OSCAR note], "왜 실전 서빙에서 의미가 있나");
 *   - the rotation is R = U H P ([OSCAR summary] §2.2-A.3) and the clip threshold is
 *     estimated on rotated activations ([OSCAR summary] §2.2-A.4);
 *   - the fused kernel unpacks, dequantises, inverse-rotates and attends over the INT2
 *     history ([OSCAR summary] §2.2-B, kernel integration).
 * Everything finer (group size, asymmetric bf16 scale/zero, rounding, routing of ring
 * slots, code placement inside a 32-byte token row) is this library's documented format;
 * each reading is listed in the design notes.  The quantizer is an encoding, so it is
 * written step by step in fp32 exactly as the format states it (the bit-exact target);
 * attention is written in fp64 as its plain definition.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC.
 * -ffp-contract=off matters: the rotation is defined as an explicit chain of fmaf().
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------
 * bf16 <-> fp32.  Round to nearest, ties to even on the fp32 bit pattern; every NaN maps
 * to the canonical quiet NaN 0x7FFF.  (bf16 is the top half of an IEEE binary32.)
 * ---------------------------------------------------------------------------------- */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)0x7fffu;
  uint32_t keep_lsb = (u >> 16) & 1u;
  uint32_t rounded = u + 0x7fffu + keep_lsb;
  return (uint16_t)(rounded >> 16);
}

static float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t oo_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }
float oo_bf16_to_f32(uint16_t h) { return bf16_to_f32(h); }

/* ------------------------------------------------------------------------------------
 * Code placement in a 32-byte INT2 token row (format definition, d = 128).
 * Channel c = 16*f + 2*w + h  (f in 0..7, w in 0..7, h in 0..1) sits in 32-bit word w
 * (little-endian), 16-bit half h, 2-bit field f:  bit offset 32*w + 16*h + 2*f.
 * So channels 16f..16f+15 share field f, and a quantisation group of 32 channels owns
 * fields {2G, 2G+1}.
 * ---------------------------------------------------------------------------------- */
int oo_code_bitpos(int c) {
  int f = c >> 4;
  int w = (c & 15) >> 1;
  int h = c & 1;
  return 32 * w + 16 * h + 2 * f;
}

void oo_pack_row(const uint8_t* codes, int d, uint8_t* row) {
  memset(row, 0, (size_t)d / 4);
  for (int c = 0; c < d; ++c) {
    int pos = oo_code_bitpos(c);
    row[pos >> 3] |= (uint8_t)((codes[c] & 3u) << (pos & 7));
  }
}

void oo_unpack_row(const uint8_t* row, int d, uint8_t* codes) {
  for (int c = 0; c < d; ++c) {
    int pos = oo_code_bitpos(c);
    codes[c] = (uint8_t)((row[pos >> 3] >> (pos & 7)) & 3u);
  }
}

/* ------------------------------------------------------------------------------------
 * Rotation into the stored basis: r = R^T x (column vectors), R row-major R[i][j].
 * Format: acc_j starts at +0.0f and takes acc_j = fmaf(R[i][j], x_i, acc_j) for
 * i = 0..d-1 ascending; r_j = bf16_rne(acc_j).   ([OSCAR summary] §2.2-A.3, §2.2-B)
 * ---------------------------------------------------------------------------------- */
static void rotate_one(const float* R, const uint16_t* x, int d, uint16_t* r) {
  /* acc[j] takes its fmaf steps in the order i = 0..d-1; the outputs are independent, so
   * they advance together (j inner), which changes no output's sequence of operations */
  float acc[512];
  for (int j = 0; j < d; ++j) acc[j] = 0.0f;
  for (int i = 0; i < d; ++i) {
    const float xi = bf16_to_f32(x[i]);
    const float* Ri = R + (size_t)i * d;
    for (int j = 0; j < d; ++j) acc[j] = fmaf(Ri[j], xi, acc[j]);
  }
  for (int j = 0; j < d; ++j) r[j] = f32_to_bf16_rne(acc[j]);
}

void oo_rotate(const float* R, const uint16_t* x, long n_tok, int d, uint16_t* r) {
#pragma omp parallel for schedule(static)
  for (long t = 0; t < n_tok; ++t) rotate_one(R, x + (size_t)t * d, d, r + (size_t)t * d);
}

/* ------------------------------------------------------------------------------------
 * INT2 quantisation of one rotated token (bf16 values r[0..d-1]), format steps:
 *   1. clip:   x = fmaxf(fminf(r, c), -c)                 ([OSCAR summary] §2.2-A.4)
 *   2. per group of g consecutive channels: mn = min x, mx = max x
 *      s = bf16_rne((mx - mn) / 3.0f),  z = bf16_rne(mn)    (fp32 subtract and divide)
 *   3. code = 0 if s == 0, else fminf(fmaxf(rintf((x - z) / s), 0), 3)  (fp32, ties-even)
 *   4. pack with oo_code_bitpos; sz[2*grp] = s bits, sz[2*grp+1] = z bits.
 * ---------------------------------------------------------------------------------- */
void oo_quantize_token(const uint16_t* r, int d, int g, float clip, uint8_t* row, uint16_t* sz) {
  uint8_t codes[512];
  float x[512];
  for (int c = 0; c < d; ++c) x[c] = fmaxf(fminf(bf16_to_f32(r[c]), clip), -clip);
  for (int grp = 0; grp < d / g; ++grp) {
    const float* xg = x + grp * g;
    float mn = xg[0], mx = xg[0];
    for (int i = 1; i < g; ++i) {
      mn = fminf(mn, xg[i]);
      mx = fmaxf(mx, xg[i]);
    }
    float range = mx - mn;
    uint16_t s_bits = f32_to_bf16_rne(range / 3.0f);
    uint16_t z_bits = f32_to_bf16_rne(mn);
    float s = bf16_to_f32(s_bits), z = bf16_to_f32(z_bits);
    for (int i = 0; i < g; ++i) {
      float q = 0.0f;
      if (s != 0.0f) {
        float u = (xg[i] - z) / s;
        q = fminf(fmaxf(rintf(u), 0.0f), 3.0f);
      }
      codes[grp * g + i] = (uint8_t)q;
    }
    sz[2 * grp] = s_bits;
    sz[2 * grp + 1] = z_bits;
  }
  oo_pack_row(codes, d, row);
}

/* Dequantised value of every channel of one INT2 token: fmaf(code, s, z) in fp32. */
void oo_dequant_token(const uint8_t* row, const uint16_t* sz, int d, int g, float* out) {
  uint8_t codes[512];
  oo_unpack_row(row, d, codes);
  for (int c = 0; c < d; ++c) {
    int grp = c / g;
    out[c] = fmaf((float)codes[c], bf16_to_f32(sz[2 * grp]), bf16_to_f32(sz[2 * grp + 1]));
  }
}

/* ------------------------------------------------------------------------------------
 * Append state machine for ONE stream (one request x layer x kv-head x {K or V}).
 * State: L = tokens held; H = end of the INT2 history.  Positions [0, min(L,S)) are BF16
 * sinks, [S, H) INT2, [H, L) BF16 recent tokens in ring slot p % W.  H starts at S and
 * L - H <= W always holds, so exactly the last W tokens beyond the sinks stay BF16.
 * Appending n tokens: L' = L + n, H' = max(H, L' - W).
 *   (a) ring tokens whose positions fall below H' are evicted: quantised from their
 *       stored bf16 value (so a token's INT2 form does not depend on its route);
 *   (b) each new token is rotated; p < S -> sink, S <= p < H' -> INT2 directly,
 *       p >= H' -> ring slot p % W.
 * ([OSCAR summary] §2.2-B: sink/recent BF16, history INT2 after rotation and clipping.)
 * Arrays: sink[S*d], ring[W*d] (bf16 bits), rows[cap*(d/4)], sz[cap*(d/g)*2]; cap >= L'.
 * Returns 0, or -1 if cap is too small.
 * ---------------------------------------------------------------------------------- */
int oo_append(int d, int g, int S, int W, float clip, const float* R, int* L, int* H, uint16_t* sink,
              uint16_t* ring, uint8_t* rows, uint16_t* sz, long cap, const uint16_t* x, long n) {
  long L0 = *L, H0 = *H, L1 = L0 + n;
  long H1 = L1 - W > H0 ? L1 - W : H0;
  if (L1 > cap) return -1;
  int ng = d / g;
  long evict_end = L0 < H1 ? L0 : H1;
  for (long p = H0; p < evict_end; ++p)
    oo_quantize_token(ring + (size_t)(p % W) * d, d, g, clip, rows + (size_t)p * (d / 4), sz + (size_t)p * ng * 2);
  uint16_t* r = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1) * d);
  oo_rotate(R, x, n, d, r);
  for (long i = 0; i < n; ++i) {
    long p = L0 + i;
    const uint16_t* ri = r + (size_t)i * d;
    if (p < S)
      memcpy(sink + (size_t)p * d, ri, sizeof(uint16_t) * d);
    else if (p < H1)
      oo_quantize_token(ri, d, g, clip, rows + (size_t)p * (d / 4), sz + (size_t)p * ng * 2);
    else
      memcpy(ring + (size_t)(p % W) * d, ri, sizeof(uint16_t) * d);
  }
  free(r);
  *L = (int)L1;
  *H = (int)H1;
  return 0;
}

/* ------------------------------------------------------------------------------------
 * Decode attention for one (request, kv-head) over the mixed-precision stream, fp64.
 *   q~_h = R_K^T q_h;  keys/values in the stored (rotated) basis:
 *     sinks and ring tokens: their bf16 values; INT2 tokens: fmaf(code, s, z);
 *   logits = q~_h . k / sqrt(d); softmax (max-subtracted, two passes);
 *   o~_h = sum p v / sum p;  o_h = R_V o~_h   (inverse rotation of the output).
 * ([OSCAR summary] §2.2-B, kernel integration; §2.1: scores and outputs are what matter.)
 * q is bf16 [G][d]; out is fp64 [G][d]; L == 0 gives zeros.
 * ---------------------------------------------------------------------------------- */
static void stream_token_values(int d, int g, int S, int W, int H, long p, const uint16_t* sink,
                                const uint16_t* ring, const uint8_t* rows, const uint16_t* sz, double* out) {
  if (p < S) {
    for (int c = 0; c < d; ++c) out[c] = bf16_to_f32(sink[(size_t)p * d + c]);
  } else if (p < H) {
    float tmp[512];
    oo_dequant_token(rows + (size_t)p * (d / 4), sz + (size_t)p * (d / g) * 2, d, g, tmp);
    for (int c = 0; c < d; ++c) out[c] = tmp[c];
  } else {
    for (int c = 0; c < d; ++c) out[c] = bf16_to_f32(ring[(size_t)(p % W) * d + c]);
  }
}

/* Attention of G query heads over one (K, V) stream in the rotated basis: qt [G][d] (the
 * rotated queries), ot [G][d] (the rotated output, before the inverse value rotation).
 * Scores against the stored rotated keys, fp64 softmax, weighted stored rotated values. */
static void attend_rotated(int d, int G, int g, int S, int W, int L, int H, const uint16_t* sinkK,
                           const uint16_t* sinkV, const uint16_t* ringK, const uint16_t* ringV, const uint8_t* rowsK,
                           const uint16_t* szK, const uint8_t* rowsV, const uint16_t* szV, const double* qt,
                           double* ot) {
  double* logit = (double*)malloc(sizeof(double) * (size_t)G * L);
  double kv[512];
  double inv_sqrt_d = 1.0 / sqrt((double)d);
  for (long p = 0; p < L; ++p) {
    stream_token_values(d, g, S, W, H, p, sinkK, ringK, rowsK, szK, kv);
    for (int h = 0; h < G; ++h) {
      double s = 0.0;
      for (int c = 0; c < d; ++c) s += qt[(size_t)h * d + c] * kv[c];
      logit[(size_t)h * L + p] = s * inv_sqrt_d;
    }
  }
  for (int h = 0; h < G; ++h) {
    double m = -INFINITY;
    for (long p = 0; p < L; ++p) m = fmax(m, logit[(size_t)h * L + p]);
    double den = 0.0;
    for (long p = 0; p < L; ++p) {
      double e = exp(logit[(size_t)h * L + p] - m);
      logit[(size_t)h * L + p] = e;
      den += e;
    }
    for (long p = 0; p < L; ++p) logit[(size_t)h * L + p] /= den;
  }
  for (long p = 0; p < L; ++p) {
    stream_token_values(d, g, S, W, H, p, sinkV, ringV, rowsV, szV, kv);
    for (int h = 0; h < G; ++h) {
      double w = logit[(size_t)h * L + p];
      for (int c = 0; c < d; ++c) ot[(size_t)h * d + c] += w * kv[c];
    }
  }
  free(logit);
}

void oo_decode(int d, int G, int g, int S, int W, int L, int H, const uint16_t* sinkK, const uint16_t* sinkV,
               const uint16_t* ringK, const uint16_t* ringV, const uint8_t* rowsK, const uint16_t* szK,
               const uint8_t* rowsV, const uint16_t* szV, const uint16_t* q, const float* R_K, const float* R_V,
               double* out) {
  memset(out, 0, sizeof(double) * (size_t)G * d);
  if (L <= 0) return;
  double* qt = (double*)calloc((size_t)G * d, sizeof(double));
  double* ot = (double*)calloc((size_t)G * d, sizeof(double));
  for (int h = 0; h < G; ++h)
    for (int c = 0; c < d; ++c) {
      double s = 0.0;
      for (int i = 0; i < d; ++i) s += (double)R_K[(size_t)i * d + c] * (double)bf16_to_f32(q[(size_t)h * d + i]);
      qt[(size_t)h * d + c] = s;
    }
  attend_rotated(d, G, g, S, W, L, H, sinkK, sinkV, ringK, ringV, rowsK, szK, rowsV, szV, qt, ot);
  for (int h = 0; h < G; ++h)
    for (int c = 0; c < d; ++c) {
      double s = 0.0;
      for (int j = 0; j < d; ++j) s += (double)R_V[(size_t)c * d + j] * ot[(size_t)h * d + j];
      out[(size_t)h * d + c] = s;
    }
  free(qt);
  free(ot);
}

/* The same with the rotations folded into the model's projections: qt are the rotated
 * queries themselves (bf16, q~ = R_K^T q computed outside), and the output is left in the
 * rotated basis (o~; the inverse value rotation R_V is applied outside). */
void oo_decode_folded(int d, int G, int g, int S, int W, int L, int H, const uint16_t* sinkK, const uint16_t* sinkV,
                      const uint16_t* ringK, const uint16_t* ringV, const uint8_t* rowsK, const uint16_t* szK,
                      const uint8_t* rowsV, const uint16_t* szV, const uint16_t* qt_bf16, double* out) {
  memset(out, 0, sizeof(double) * (size_t)G * d);
  if (L <= 0) return;
  double* qt = (double*)calloc((size_t)G * d, sizeof(double));
  for (size_t e = 0; e < (size_t)G * d; ++e) qt[e] = (double)bf16_to_f32(qt_bf16[e]);
  attend_rotated(d, G, g, S, W, L, H, sinkK, sinkV, ringK, ringV, rowsK, szK, rowsV, szV, qt, out);
  free(qt);
}

/* Uncompressed comparison: plain softmax(q K^T / sqrt(d)) V over bf16 K, V [L][d]. */
void oo_bf16_decode(int d, int G, long L, const uint16_t* K, const uint16_t* V, const uint16_t* q, double* out) {
  memset(out, 0, sizeof(double) * (size_t)G * d);
  if (L <= 0) return;
  double* w = (double*)malloc(sizeof(double) * (size_t)L);
  double inv_sqrt_d = 1.0 / sqrt((double)d);
  for (int h = 0; h < G; ++h) {
    double m = -INFINITY;
    for (long p = 0; p < L; ++p) {
      double s = 0.0;
      for (int c = 0; c < d; ++c)
        s += (double)bf16_to_f32(q[(size_t)h * d + c]) * (double)bf16_to_f32(K[(size_t)p * d + c]);
      w[p] = s * inv_sqrt_d;
      m = fmax(m, w[p]);
    }
    double den = 0.0;
    for (long p = 0; p < L; ++p) {
      w[p] = exp(w[p] - m);
      den += w[p];
    }
    for (long p = 0; p < L; ++p) {
      double a = w[p] / den;
      for (int c = 0; c < d; ++c) out[(size_t)h * d + c] += a * (double)bf16_to_f32(V[(size_t)p * d + c]);
    }
  }
  free(w);
}

int oo_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oo_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
