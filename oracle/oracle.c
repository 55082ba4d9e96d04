/*
 * ORACLE (test infrastructure only).  Plain, slow, obviously-correct CPU code
 * that the tests, the smoke check and the bench's CPU-baseline leg compare the
 * CUDA path against.  It shares no code with the CUDA library and nothing in
 * the product path may call it.
 *
 * Contents
 *   - W12, the lossless 12-bit weight format ("SpecPilot: AI Agent Framework
 *     Boosts Speculative Decoding 10.87x", section "(1) W12: Lossless 12-bit
 *     Weight Format"): each bf16 weight keeps its sign and 7-bit mantissa and
 *     replaces its 8-bit exponent by a 4-bit code into a per-tensor table of
 *     the 15 most frequent exponents; code 15 marks an escape whose exact bf16
 *     value sits in a sparse side list.  Restoration is bit-exact.
 *   - the packed byte layout (our definition; the page fixes only the fields),
 *     written here as a plain per-weight location function;
 *   - y = x W^T in fp64, summed in k order;
 *   - double -> bf16 round-to-nearest-even.
 *
 * Packed layout (N % 16 == 0, K % 64 == 0).  Rows are grouped in strips of
 * 16, columns in super-tiles of 64 split into four 16-wide sub-tiles.  A
 * super-tile of a strip occupies 384 consecutive 32-bit words, strips are
 * stored one after the other and within a strip the super-tiles follow in k
 * order:  word index = (s * (K/64) + t) * 384 + (p * 32 + lane) * 4 + j.
 * For weight (n, k):  s = n/16, r = n%16, t = k/64, j = (k%64)/16, c = k%16,
 *   g = r%8, lane = 4*g + (c%8)/2, half = c%2,
 *   pair = (c >= 8 ? 2 : 0) + (r >= 8 ? 1 : 0).
 * Its 12-bit field is f = sign<<11 | code<<7 | mantissa.
 *   pair 0,1,2: word p = pair holds f in bits 0..10 and its sign in bit 15
 *               (half 0) or in bits 16..26 and bit 31 (half 1);
 *   pair 3:     f is cut into three nibbles; nibble i goes to word p = i,
 *               bits 11..14 (half 0) or bits 27..30 (half 1).
 * An escaped weight stores f = 15<<7 (sign 0, mantissa 0).
 * Escapes are listed as (flat index n*K+k, bf16 bits) in increasing flat
 * index; row_ptr[n] counts the escapes with flat index < n*K.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 -- */

double or_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), with bf16 subnormals
 * and overflow to infinity. */
uint16_t or_double_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  frexp(a, &e);            /* a = m * 2^e, 0.5 <= m < 1 */
  int q = e - 8;           /* 8 significant bits */
  if (q < -133) q = -133;  /* subnormal quantum of bf16 */
  double r = nearbyint(ldexp(a, -q));
  double v = ldexp(r, q);
  if (v >= 0x1p128) return sign | 0x7F80;
  float f = (float)v; /* exact */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)(u >> 16);
}

void or_round_bf16(const double* x, int64_t n, uint16_t* out) {
#pragma omp parallel for schedule(static, 4096)
  for (int64_t i = 0; i < n; i++) out[i] = or_double_to_bf16(x[i]);
}

void or_bf16_to_f64(const uint16_t* b, int64_t n, double* out) {
#pragma omp parallel for schedule(static, 4096)
  for (int64_t i = 0; i < n; i++) out[i] = or_bf16_to_double(b[i]);
}

/* ----------------------------------------------------------------- W12 -- */

void or_w12_histogram(const uint16_t* w, int64_t n, uint64_t* hist) {
  for (int i = 0; i < 256; i++) hist[i] = 0;
  for (int64_t i = 0; i < n; i++) hist[(w[i] >> 7) & 0xFF]++;
}

/* The table: the (up to) 15 exponents with the largest counts, ties broken
 * by the smaller exponent, only exponents that occur; stored in ascending
 * exponent order.  Returns the number of entries. */
int or_w12_table(const uint64_t* hist, uint8_t* table) {
  int chosen[256] = {0};
  int n = 0;
  for (int round = 0; round < 15; round++) {
    int best = -1;
    for (int e = 0; e < 256; e++) {
      if (chosen[e] || hist[e] == 0) continue;
      if (best < 0 || hist[e] > hist[best]) best = e; /* ascending scan keeps the smaller e on ties */
    }
    if (best < 0) break;
    chosen[best] = 1;
    n++;
  }
  int k = 0;
  for (int e = 0; e < 256; e++)
    if (chosen[e]) table[k++] = (uint8_t)e;
  for (int i = k; i < 16; i++) table[i] = 0;
  return n;
}

/* Where weight (n,k) lives. */
typedef struct {
  int64_t tile_word; /* index of word (p=0, lane, j) of its super-tile */
  int pair;
  int half;
} w12_loc;

static w12_loc w12_locate(int64_t n, int64_t k, int64_t K) {
  int64_t s = n / 16, r = n % 16, t = k / 64;
  int j = (int)((k % 64) / 16), c = (int)(k % 16);
  int g = (int)(r % 8), lane = 4 * g + (c % 8) / 2;
  w12_loc L;
  L.half = c % 2;
  L.pair = (c >= 8 ? 2 : 0) + (r >= 8 ? 1 : 0);
  L.tile_word = (s * (K / 64) + t) * 384 + (int64_t)lane * 4 + j;
  return L;
}

#define W12_PLANE_STRIDE 128 /* words between plane p and p+1 of a super-tile */

static void w12_put(uint32_t* words, w12_loc L, uint32_t f) {
  int sh = 16 * L.half;
  if (L.pair < 3) {
    uint32_t v = (f & 0x7FFu) | ((f >> 11) << 15);
    uint32_t* w = &words[L.tile_word + (int64_t)L.pair * W12_PLANE_STRIDE];
    *w = (*w & ~(0x87FFu << sh)) | (v << sh);
  } else {
    for (int i = 0; i < 3; i++) {
      uint32_t nib = (f >> (4 * i)) & 0xFu;
      uint32_t* w = &words[L.tile_word + (int64_t)i * W12_PLANE_STRIDE];
      *w = (*w & ~(0xFu << (11 + sh))) | (nib << (11 + sh));
    }
  }
}

static uint32_t w12_get(const uint32_t* words, w12_loc L) {
  int sh = 16 * L.half;
  if (L.pair < 3) {
    uint32_t v = (words[L.tile_word + (int64_t)L.pair * W12_PLANE_STRIDE] >> sh) & 0xFFFFu;
    return (v & 0x7FFu) | (((v >> 15) & 1u) << 11);
  }
  uint32_t f = 0;
  for (int i = 0; i < 3; i++) f |= ((words[L.tile_word + (int64_t)i * W12_PLANE_STRIDE] >> (11 + sh)) & 0xFu) << (4 * i);
  return f;
}

int64_t or_w12_count_escapes(const uint16_t* w, int64_t n, const uint8_t* table, int n_table) {
  int in_table[256] = {0};
  for (int c = 0; c < n_table; c++) in_table[table[c]] = 1;
  int64_t cnt = 0;
  for (int64_t i = 0; i < n; i++) cnt += !in_table[(w[i] >> 7) & 0xFF];
  return cnt;
}

/* Pack W[N][K].  words: N*K*3/8 u32.  Escape arrays must hold esc_cap
 * entries; row_ptr holds N+1.  Returns the escape count, -1 on bad shape,
 * -2 if esc_cap is too small. */
int64_t or_w12_pack(const uint16_t* W, int64_t N, int64_t K, const uint8_t* table, int n_table, uint32_t* words,
                    uint32_t* esc_idx, uint16_t* esc_val, int64_t esc_cap, uint32_t* row_ptr) {
  if (N <= 0 || K <= 0 || N % 16 || K % 64 || n_table < 0 || n_table > 15) return -1;
  int code_of[256];
  for (int e = 0; e < 256; e++) code_of[e] = 15;
  for (int c = 0; c < n_table; c++) code_of[table[c]] = c;
  memset(words, 0, (size_t)(N * K / 8 * 3) * 4);
  int64_t ne = 0;
  for (int64_t n = 0; n < N; n++) {
    row_ptr[n] = (uint32_t)ne;
    for (int64_t k = 0; k < K; k++) {
      uint16_t b = W[n * K + k];
      int code = code_of[(b >> 7) & 0xFF];
      uint32_t f;
      if (code == 15) {
        if (ne >= esc_cap) return -2;
        esc_idx[ne] = (uint32_t)(n * K + k);
        esc_val[ne] = b;
        ne++;
        f = 15u << 7;
      } else {
        f = ((uint32_t)(b >> 15) << 11) | ((uint32_t)code << 7) | (b & 0x7Fu);
      }
      w12_put(words, w12_locate(n, k, K), f);
    }
  }
  row_ptr[N] = (uint32_t)ne;
  return ne;
}

/* Restore W[N][K] bit-exactly. */
int or_w12_unpack(const uint32_t* words, int64_t N, int64_t K, const uint8_t* table, int n_table,
                  const uint32_t* esc_idx, const uint16_t* esc_val, int64_t n_esc, uint16_t* W) {
  if (N <= 0 || K <= 0 || N % 16 || K % 64 || n_table < 0 || n_table > 15) return -1;
  uint8_t tab[16];
  for (int c = 0; c < 16; c++) tab[c] = c < n_table ? table[c] : 0;
  for (int64_t n = 0; n < N; n++)
    for (int64_t k = 0; k < K; k++) {
      uint32_t f = w12_get(words, w12_locate(n, k, K));
      W[n * K + k] = (uint16_t)(((f >> 11) << 15) | ((uint32_t)tab[(f >> 7) & 15] << 7) | (f & 0x7F));
    }
  for (int64_t e = 0; e < n_esc; e++) W[esc_idx[e]] = esc_val[e];
  return 0;
}

/* Read back the 12-bit field of weight (n,k) (for tests of the layout). */
uint32_t or_w12_field(const uint32_t* words, int64_t n, int64_t k, int64_t K) {
  return w12_get(words, w12_locate(n, k, K));
}

/* -------------------------------------------------------------- linear -- */

/* y[m][n] = sum_k x[m][k] * W[n][k], fp64, k ascending.  x is fp64 [M][K],
 * W bf16 [N][K], y fp64 [M][N]. */
void or_linear(const double* x, int64_t M, int64_t K, const uint16_t* W, int64_t N, double* y) {
  double* xt = (double*)malloc(sizeof(double) * (size_t)(M * K)); /* [K][M] so each k touches M values */
  for (int64_t m = 0; m < M; m++)
    for (int64_t k = 0; k < K; k++) xt[k * M + m] = x[m * K + k];
#pragma omp parallel
  {
    double* acc = (double*)malloc(sizeof(double) * (size_t)M);
#pragma omp for schedule(static, 16)
    for (int64_t n = 0; n < N; n++) {
      const uint16_t* wr = W + n * K;
      for (int64_t m = 0; m < M; m++) acc[m] = 0.0;
      for (int64_t k = 0; k < K; k++) {
        double wk = or_bf16_to_double(wr[k]);
        const double* xk = xt + k * M;
        for (int64_t m = 0; m < M; m++) acc[m] += xk[m] * wk;
      }
      for (int64_t m = 0; m < M; m++) y[m * N + n] = acc[m];
    }
    free(acc);
  }
  free(xt);
}
