/*
 * oracle.c — TEST INFRASTRUCTURE ONLY.  A plain, slow, single-threaded CPU
 * restatement of the batch-size-1 weight-only-quantised decode step described
 * on the gpt-fast pages (gpt-fast README, sections "Quantization: Int8
 * weight-only quantization", "Int4 weight-only quantization" and
 * "Benchmarks"; "Efficiently implementing the Mixtral 8x7B model with
 * gpt-fast", section "Key Features").  Only the tests, the package's smoke
 * check and the benchmark's CPU-baseline leg may load this library; the GPU
 * path never does, and this file shares no code with it.
 *
 * Precision.  The pages fix no precision.  Values the method rounds to bf16
 * are held here as doubles carrying bf16-exact values; every sum, product,
 * softmax and normalisation is done in fp64.  Where a float decides an
 * integer (a quantisation code or scale), the decision is taken in IEEE fp32
 * exactly as written below, because the GPU kernels take it in fp32 too.
 *
 * Readings of points the pages leave open are named in place as READING.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */
/* bf16 = the top 16 bits of an IEEE binary32; fp32 -> bf16 rounds to nearest,
 * ties to even.  NaN never occurs in this workload; it is kept quiet here. */
uint16_t orc_bf16_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

float orc_f32_from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round doubles to bf16 values in place (double -> fp32 -> bf16, RNE each). */
void orc_round_bf16(double* x, long n) {
  for (long i = 0; i < n; ++i) x[i] = orc_f32_from_bf16(orc_bf16_from_f32((float)x[i]));
}

void orc_bf16_to_double(const uint16_t* h, long n, double* out) {
  for (long i = 0; i < n; ++i) out[i] = orc_f32_from_bf16(h[i]);
}

/* ------------------------------------------------- int8 weight-only ---- */
/* Per output row n (gpt-fast README, "Int8 weight-only quantization";
 * READING: symmetric, one bf16 scale per output channel, code -128 unused):
 *   s_n = bf16( max_k |W[n,k]| / 127 )            fp32 divide, then RNE
 *   q   = clamp( rint( W[n,k] / s_n ), -127, 127 ) fp32 divide, ties to even
 * A row of zeros gets s = 0 and q = 0. */
void orc_quant_w8(const uint16_t* W, long N, long K, int8_t* q, uint16_t* s) {
  for (long n = 0; n < N; ++n) {
    const uint16_t* row = W + n * K;
    float mx = 0.0f;
    for (long k = 0; k < K; ++k) {
      float a = fabsf(orc_f32_from_bf16(row[k]));
      if (a > mx) mx = a;
    }
    float quotient = mx / 127.0f;
    uint16_t sb = orc_bf16_from_f32(quotient);
    float sv = orc_f32_from_bf16(sb);
    s[n] = sb;
    for (long k = 0; k < K; ++k) {
      long c = 0;
      if (sv != 0.0f) {
        float t = orc_f32_from_bf16(row[k]) / sv;
        c = (long)rintf(t);
        if (c > 127) c = 127;
        if (c < -127) c = -127;
      }
      q[n * K + k] = (int8_t)c;
    }
  }
}

/* ---------------------------------------------- int4 weight-only, G ---- */
/* Per row n and group g of G consecutive k (gpt-fast README, "Int4
 * weight-only quantization", --groupsize 32; READING: asymmetric min/max with
 * a float zero offset, dequantised value q*s + z, codes 0..15):
 *   z = bf16(min)   (exact: W is bf16)
 *   s = bf16( (max - min) / 15 )       fp32 subtract, fp32 divide, RNE
 *   q = clamp( rint( (W - min) / s ), 0, 15 )   fp32 subtract and divide
 * A group whose s is 0 (max == min) gets q = 0, so q*s + z == W exactly.
 * q holds one code per byte, [N][K]; s and z are [N][K/G]. */
void orc_quant_w4g(const uint16_t* W, long N, long K, int G, uint8_t* q, uint16_t* s,
                   uint16_t* z) {
  long ng = K / G;
  for (long n = 0; n < N; ++n) {
    for (long g = 0; g < ng; ++g) {
      const uint16_t* w = W + n * K + g * G;
      float mn = orc_f32_from_bf16(w[0]), mx = mn;
      for (int i = 1; i < G; ++i) {
        float v = orc_f32_from_bf16(w[i]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
      }
      float range = mx - mn;
      uint16_t sb = orc_bf16_from_f32(range / 15.0f);
      float sv = orc_f32_from_bf16(sb);
      s[n * ng + g] = sb;
      z[n * ng + g] = orc_bf16_from_f32(mn);
      for (int i = 0; i < G; ++i) {
        long c = 0;
        if (sv != 0.0f) {
          float t = (orc_f32_from_bf16(w[i]) - mn) / sv;
          c = (long)rintf(t);
          if (c > 15) c = 15;
          if (c < 0) c = 0;
        }
        q[n * K + g * G + i] = (uint8_t)c;
      }
    }
  }
}

/* ------------------------------------------------------ packed layout ---- */
/* The device layout of each weight type, restated from its definition: the
 * matrix is cut into slots of 32 rows (a tile) by 256 bytes of each row's
 * code bytes (a K-slot), stored one after another, tile-major (slot of tile
 * t, K-slot b at index t * nb + b, nb = ceil(row bytes / 256)).  A slot is
 * 128-byte lines: line h * 32 + r (h = 0, 1) holds bytes
 * [256 b + 128 h, 256 b + 128 h + 128) of the code bytes of row 32 t + r;
 * int4 slots add lines 64 + g (g < 512 / G), whose 32-bit word r is
 * s | z << 16 for row 32 t + r and group (512 / G) b + g.  Inside line L the
 * 16-byte unit u is stored at unit u XOR (L mod 8).  Bytes past a row, past
 * the last row or past the last group are zero.
 *   code bytes of a row: bf16 values (2 bytes each, little endian); int8
 *   q + 128 (offset binary); int4 byte i = q[2i] | q[2i+1] << 4. */
enum { ORC_BF16 = 0, ORC_INT8 = 1, ORC_INT4 = 2 };

static long row_bytes(int dt, long K) { return dt == ORC_BF16 ? 2 * K : dt == ORC_INT8 ? K : K / 2; }
static long slot_size(int dt, int G) { return 8192 + (dt == ORC_INT4 ? (512 / G) * 128 : 0); }
static long nslots_k(int dt, long K) { return (row_bytes(dt, K) + 255) / 256; }
/* byte b of line L of a slot, with the units of the line swizzled */
static long line_pos(long L, long b) { return L * 128 + (((b / 16) ^ (L % 8)) * 16) + b % 16; }

long orc_packed_bytes(int dt, long N, long K, int G) {
  return (N + 31) / 32 * nslots_k(dt, K) * slot_size(dt, G);
}

/* position in the packed buffer of code byte j of row n */
static long code_pos(int dt, long K, int G, long n, long j) {
  long t = n / 32, r = n % 32, b = j / 256, h = (j % 256) / 128;
  return (t * nslots_k(dt, K) + b) * slot_size(dt, G) + line_pos(h * 32 + r, j % 128);
}
/* position of the scale/zero word of (row n, group g) */
static long sz_pos(long K, int G, long n, long g) {
  long gps = 512 / G, t = n / 32, r = n % 32;
  return (t * nslots_k(ORC_INT4, K) + g / gps) * slot_size(ORC_INT4, G) + line_pos(64 + g % gps, 4 * r);
}

static void put32(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}
static uint32_t get32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

/* code byte j of row n, from the logical source */
static uint8_t code_byte(int dt, long K, const void* src, long n, long j) {
  if (dt == ORC_BF16) {
    uint16_t w = ((const uint16_t*)src)[n * K + j / 2];
    return (uint8_t)(j % 2 ? w >> 8 : w);
  }
  if (dt == ORC_INT8) return (uint8_t)(((const int8_t*)src)[n * K + j] + 128);
  const uint8_t* c = (const uint8_t*)src + n * K + 2 * j;
  return (uint8_t)((c[0] & 15u) | ((c[1] & 15u) << 4));
}

/* src: bf16 W [N][K] (uint16), int8 codes [N][K], or int4 codes [N][K] one per
 * byte; s, z: int4 [N][K/G] bf16 (ignored otherwise). */
void orc_pack(int dt, long N, long K, int G, const void* src, const uint16_t* s,
              const uint16_t* z, uint8_t* out) {
  memset(out, 0, (size_t)orc_packed_bytes(dt, N, K, G));
  long rb = row_bytes(dt, K);
  for (long n = 0; n < N; ++n)
    for (long j = 0; j < rb; ++j) out[code_pos(dt, K, G, n, j)] = code_byte(dt, K, src, n, j);
  if (dt == ORC_INT4) {
    long ng = K / G;
    for (long n = 0; n < N; ++n)
      for (long g = 0; g < ng; ++g)
        put32(out + sz_pos(K, G, n, g), (uint32_t)s[n * ng + g] | ((uint32_t)z[n * ng + g] << 16));
  }
}

/* Inverse of orc_pack (used only to show the layout is a bijection). */
void orc_unpack(int dt, long N, long K, int G, const uint8_t* in, void* dst, uint16_t* s,
                uint16_t* z) {
  long rb = row_bytes(dt, K);
  for (long n = 0; n < N; ++n)
    for (long j = 0; j < rb; ++j) {
      uint8_t v = in[code_pos(dt, K, G, n, j)];
      if (dt == ORC_BF16) {
        uint16_t* w = (uint16_t*)dst + n * K + j / 2;
        *w = (uint16_t)(j % 2 ? (*w & 0x00FF) | (v << 8) : (*w & 0xFF00) | v);
      } else if (dt == ORC_INT8) {
        ((int8_t*)dst)[n * K + j] = (int8_t)(v - 128);
      } else {
        uint8_t* c = (uint8_t*)dst + n * K + 2 * j;
        c[0] = (uint8_t)(v & 15u);
        c[1] = (uint8_t)(v >> 4);
      }
    }
  if (dt == ORC_INT4) {
    long ng = K / G;
    for (long n = 0; n < N; ++n)
      for (long g = 0; g < ng; ++g) {
        uint32_t v = get32(in + sz_pos(K, G, n, g));
        s[n * ng + g] = (uint16_t)v;
        z[n * ng + g] = (uint16_t)(v >> 16);
      }
  }
}

/* ---------------------------------------------------------- linear ---- */
/* Y[t][n] = sum_k X[t][k] * What[n][k] for t < T, in fp64, k ascending, with
 * What = W (bf16), q*s_n (int8) or q*s_{n,g} + z_{n,g} (int4, g = k/G): the
 * product y = x W^T of the pages' linear layers, against the dequantised
 * weight. */
void orc_linear(int dt, long N, long K, int G, const void* w, const uint16_t* s, const uint16_t* z,
                const double* X, long T, double* Y) {
  double* row = (double*)malloc(sizeof(double) * (size_t)K);
  long ng = K / G;
  for (long n = 0; n < N; ++n) {
    for (long k = 0; k < K; ++k) {
      if (dt == ORC_BF16) {
        row[k] = orc_f32_from_bf16(((const uint16_t*)w)[n * K + k]);
      } else if (dt == ORC_INT8) {
        row[k] = (double)((const int8_t*)w)[n * K + k] * (double)orc_f32_from_bf16(s[n]);
      } else {
        long g = k / G;
        row[k] = (double)((const uint8_t*)w)[n * K + k] * (double)orc_f32_from_bf16(s[n * ng + g]) +
                 (double)orc_f32_from_bf16(z[n * ng + g]);
      }
    }
    for (long t = 0; t < T; ++t) {
      const double* x = X + t * K;
      double acc = 0.0;
      for (long k = 0; k < K; ++k) acc += x[k] * row[k];
      Y[t * N + n] = acc;
    }
  }
  free(row);
}

/* ------------------------------------------------------- attention ---- */
/* Single-query attention of each of Hq heads over positions 0..T-1 of its
 * kv head h / (Hq/Hkv) (grouped-query sharing): o_h = sum_t p_t v_t with
 * p = softmax_t(q_h . k_t / sqrt(hd)), the max subtracted before exp.
 * q [Hq][hd]; Kc, Vc [Hkv][T][hd]; out [Hq][hd]; all fp64. */
void orc_attention(int Hq, int Hkv, int hd, long T, const double* q, const double* Kc,
                   const double* Vc, double* out) {
  double* p = (double*)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
  int group = Hq / Hkv;
  double scale = 1.0 / sqrt((double)hd);
  for (int h = 0; h < Hq; ++h) {
    int kvh = h / group;
    const double* qh = q + (long)h * hd;
    double m = -INFINITY;
    for (long t = 0; t < T; ++t) {
      const double* kt = Kc + ((long)kvh * T + t) * hd;
      double dot = 0.0;
      for (int d = 0; d < hd; ++d) dot += qh[d] * kt[d];
      p[t] = dot * scale;
      if (p[t] > m) m = p[t];
    }
    double L = 0.0;
    for (long t = 0; t < T; ++t) { p[t] = exp(p[t] - m); L += p[t]; }
    for (int d = 0; d < hd; ++d) {
      double acc = 0.0;
      for (long t = 0; t < T; ++t) acc += p[t] * Vc[((long)kvh * T + t) * hd + d];
      out[(long)h * hd + d] = acc / L;
    }
  }
  free(p);
}

/* ------------------------------------------------ elementwise steps ---- */
/* RMSNorm: out = x * (mean(x^2) + eps)^(-1/2) * g. */
void orc_rmsnorm(const double* x, const uint16_t* g, long d, double eps, double* out) {
  double ss = 0.0;
  for (long i = 0; i < d; ++i) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss / (double)d + eps);
  for (long i = 0; i < d; ++i) out[i] = x[i] * r * (double)orc_f32_from_bf16(g[i]);
}

/* Rotary position embedding at position pos, applied in place to nheads heads
 * of hd values.  READING: adjacent pairs (2i, 2i+1) rotate by the angle
 * pos * theta^(-2i/hd). */
void orc_rope(double* v, int nheads, int hd, long pos, double theta) {
  for (int h = 0; h < nheads; ++h) {
    double* x = v + (long)h * hd;
    for (int i = 0; i < hd / 2; ++i) {
      double f = pow(theta, -2.0 * (double)i / (double)hd);
      double a = (double)pos * f, c = cos(a), s = sin(a);
      double x0 = x[2 * i], x1 = x[2 * i + 1];
      x[2 * i] = x0 * c - x1 * s;
      x[2 * i + 1] = x0 * s + x1 * c;
    }
  }
}

/* SwiGLU gate: h = silu(gate) * up, silu(a) = a / (1 + e^(-a)). */
void orc_swiglu(const double* gate, const double* up, long n, double* h) {
  for (long i = 0; i < n; ++i) h[i] = gate[i] / (1.0 + exp(-gate[i])) * up[i];
}
