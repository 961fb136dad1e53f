/*
 * kv4_oracle.c -- plain, slow CPU reference for 4-bit rotated KV-cache
 * decode attention (UltraQuant-style).  TEST INFRASTRUCTURE ONLY: only the
 * test-suite, the smoke check and the benchmark's CPU-baseline leg may load
 * this file.  It shares no code, header, table or constant with the CUDA
 * library; the two meet only through their inputs and outputs.
 *
 * Source of the method ("UltraQuant on AMD Instinct" blog, ioiotimes page):
 *   - section "What is UltraQuant": keys and values are stored on the FP4
 *     grid that MI355X supports, one shared power-of-two scale per 32
 *     channels, 17 bytes per 32-value group against 32 for the 8-bit cache;
 *     a Walsh-Hadamard rotation is applied first to spread outlier channels;
 *     the kernel consumes FP4 values directly, the power-of-two scale folded
 *     into the scaled MFMA (no lookup-table dequantisation).
 *   - section "Why UltraQuant beats 8-bit KV": FP4 codes plus UE8M0 scales;
 *     every new token re-reads the whole cache.
 *   - section "Throughput-latency trade-off": MTP verify rows (3 positions)
 *     share one paged cache.
 *
 * Readings of what the page leaves open (each is listed in the design notes):
 *   R1  H is the orthonormal Sylvester Walsh-Hadamard matrix of the full head
 *       dimension, natural order, no random signs, same for K, V, every head.
 *   R2  q is rotated by the same H (q.k is invariant); V is stored rotated,
 *       so the attention output is rotated back by H (H = H^T = H^-1).
 *   R3  rotation arithmetic: S = (+-1 matrix) . x computed EXACTLY, then
 *       y = fp32( fp64(S) * c_D ) with c_D = RN_fp64(1/sqrt(D)).
 *   R4  scale exponent (OCP MX rule): e = floor(log2(amax)) - 2, clamped to
 *       [-127, 127]; amax = 0 gives e = -127; UE8M0 byte = e + 127.
 *   R5  element code = round-to-nearest-even onto the E2M1 grid
 *       +-{0, .5, 1, 1.5, 2, 3, 4, 6}, saturating at 6; the sign bit is kept
 *       even when the value rounds to zero.
 *   R6  block layout per (page, kv-head) -- see the pack functions below.
 *   R7  FP8 comparator: E4M3 (OCP), RNE with saturation to +-448 of
 *       fp32(x * inv_scale[h]); no rotation.
 *
 * Everything here is fp64 unless a step is defined in fp32 above.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_INEXACT 2

/* ------------------------------------------------------------------ */
/* bf16 / fp32 bit helpers                                              */
/* ------------------------------------------------------------------ */
static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static int is_pow2_dim(int D) {
  return D == 64 || D == 128 || D == 256 || D == 512;
}

/* c_D = RN_fp64(1/sqrt(D)) written out as exact binary64 literals. */
static double inv_sqrt_dim(int D) {
  switch (D) {
    case 64:  return 0x1.0p-3;
    case 128: return 0x1.6a09e667f3bcdp-4;
    case 256: return 0x1.0p-4;
    case 512: return 0x1.6a09e667f3bcdp-5;
    default:  return 0.0;
  }
}

/* ------------------------------------------------------------------ */
/* Walsh-Hadamard matrix by the Sylvester recursion                     */
/*   H_1 = [1];  H_2n = [[H_n, H_n], [H_n, -H_n]]                        */
/* Entries are +-1 (unnormalised).                                      */
/* ------------------------------------------------------------------ */
int orc_hadamard_pm1(int D, int8_t* H) {
  if (D < 1 || (D & (D - 1)) != 0) return ORC_BAD_ARG;
  H[0] = 1;
  for (int n = 1; n < D; n *= 2) {
    /* H currently holds H_n in its top-left n x n corner (row stride D). */
    for (int i = 0; i < n; ++i)
      for (int j = 0; j < n; ++j) {
        int8_t h = H[i * D + j];
        H[i * D + (j + n)] = h;
        H[(i + n) * D + j] = h;
        H[(i + n) * D + (j + n)] = (int8_t)(-h);
      }
  }
  return ORC_OK;
}

/* Cached +-1 matrices for the supported head dimensions. */
static int8_t* g_H[10];
static const int8_t* hadamard_cached(int D) {
  int lg = 0;
  while ((1 << lg) < D) ++lg;
  if (!g_H[lg]) {
    int8_t* H = (int8_t*)malloc((size_t)D * D);
    orc_hadamard_pm1(D, H);
    g_H[lg] = H;
  }
  return g_H[lg];
}

/* ------------------------------------------------------------------ */
/* R3: exact rotation of one bf16 vector.                               */
/* Each nonzero bf16 value is an integer M (|M| < 256) times 2^E.  With */
/* Emin the smallest such E in the vector, every product +-x_j equals   */
/* an integer times 2^Emin, so S_i = sum_j H_ij x_j is an exact integer */
/* sum.  The vector is inside the exact domain when sum_j |M_j|         */
/* 2^(E_j - Emin) < 2^53: then S_i is exactly representable in binary64 */
/* and every summation order gives the same fp64 value.                 */
/* Returns ORC_INEXACT (and still fills y with the natural-order fp64   */
/* sum) for vectors outside that domain.                                */
/* ------------------------------------------------------------------ */
int orc_rotate_bf16(const uint16_t* x, int D, float* y) {
  if (!is_pow2_dim(D)) return ORC_BAD_ARG;
  const int8_t* H = hadamard_cached(D);
  const double c = inv_sqrt_dim(D);

  int64_t M[512];
  int E[512];
  int emin = 100000;
  for (int j = 0; j < D; ++j) {
    uint16_t b = x[j];
    int sign = (b >> 15) & 1;
    int ef = (b >> 7) & 0xFF;
    int mf = b & 0x7F;
    if (ef == 0xFF) return ORC_BAD_ARG; /* inf / nan are not encodable */
    int64_t m;
    int e;
    if (ef == 0) { m = mf; e = 1 - 127 - 7; }          /* subnormal */
    else { m = 0x80 | mf; e = ef - 127 - 7; }          /* normal */
    if (m == 0) { M[j] = 0; E[j] = 0; continue; }
    M[j] = sign ? -m : m;
    E[j] = e;
    if (e < emin) emin = e;
  }

  int exact = 1;
  int64_t T[512];
  uint64_t abs_sum = 0;
  for (int j = 0; j < D; ++j) {
    if (M[j] == 0) { T[j] = 0; continue; }
    int sh = E[j] - emin;
    if (sh > 45) { exact = 0; break; }
    T[j] = M[j] * ((int64_t)1 << sh);
    abs_sum += (uint64_t)(T[j] < 0 ? -T[j] : T[j]);
    if (abs_sum >= ((uint64_t)1 << 53)) { exact = 0; break; }
  }

  for (int i = 0; i < D; ++i) {
    double S;
    if (exact) {
      int64_t s = 0;
      for (int j = 0; j < D; ++j) s += (int64_t)H[i * D + j] * T[j];
      S = ldexp((double)s, emin == 100000 ? 0 : emin); /* exact: |s| < 2^53 */
    } else {
      S = 0.0;
      for (int j = 0; j < D; ++j) S += (double)H[i * D + j] * (double)bf16_to_float(x[j]);
    }
    y[i] = (float)(S * c);
  }
  return exact ? ORC_OK : ORC_INEXACT;
}

/* Plain fp64 rotation v -> H v (orthonormal H), used for q and the output. */
void orc_rotate_f64(const double* v, int D, double* out) {
  const int8_t* H = hadamard_cached(D);
  const double c = inv_sqrt_dim(D);
  for (int i = 0; i < D; ++i) {
    double s = 0.0;
    for (int j = 0; j < D; ++j) s += (double)H[i * D + j] * v[j];
    out[i] = s * c;
  }
}

/* ------------------------------------------------------------------ */
/* R4: UE8M0 group exponent from the fp32 group maximum.                */
/* ------------------------------------------------------------------ */
int orc_group_exponent(const float* y, int n) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(y[i]);
    if (a > amax) amax = a;
  }
  if (amax == 0.0f) return -127;
  int k;
  (void)frexpf(amax, &k); /* amax = f * 2^k, f in [0.5, 1): floor(log2 amax) = k - 1 */
  int e = (k - 1) - 2;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return e;
}

/* ------------------------------------------------------------------ */
/* R5: E2M1 code of z (already divided by 2^e), round-to-nearest-even   */
/* by comparison with the exact midpoints of the grid, saturating.      */
/* Code = sign<<3 | magnitude index; the index (0..7) is the standard   */
/* 3-bit E2M1 magnitude field (2 exponent bits, 1 mantissa bit).        */
/* ------------------------------------------------------------------ */
static const double kE2M1Grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

int orc_e2m1_encode(double z) {
  int sign = signbit(z) ? 1 : 0;
  double a = fabs(z);
  int idx = 0;
  for (int k = 0; k < 7; ++k) {
    double mid = 0.5 * (kE2M1Grid[k] + kE2M1Grid[k + 1]);
    if (a > mid) idx = k + 1;
    else if (a == mid) { idx = (k % 2 == 0) ? k : k + 1; break; }
    else break;
  }
  return (sign << 3) | idx;
}

double orc_e2m1_decode(int code) {
  double v = kE2M1Grid[code & 7];
  return (code & 8) ? -v : v;
}

/* Quantise an already rotated fp32 vector: per-32 exponent (R4), then
 * E2M1 codes of y / 2^e (R5).  codes: one code per channel (low 4 bits of
 * a byte); expo: D/32 signed, unbiased exponents. */
void orc_quantize_rotated(const float* y, int D, uint8_t* codes, int* expo) {
  for (int g = 0; g < D / 32; ++g) {
    int e = orc_group_exponent(y + 32 * g, 32);
    expo[g] = e;
    for (int i = 0; i < 32; ++i) {
      double z = ldexp((double)y[32 * g + i], -e); /* exact in binary64 */
      codes[32 * g + i] = (uint8_t)orc_e2m1_encode(z);
    }
  }
}

/* Quantise one bf16 head vector: rotation (R3), then orc_quantize_rotated. */
int orc_quantize_vector(const uint16_t* x, int D, uint8_t* codes, int* expo) {
  float y[512];
  int st = orc_rotate_bf16(x, D, y);
  if (st == ORC_BAD_ARG) return st;
  orc_quantize_rotated(y, D, codes, expo);
  return st;
}

/* ------------------------------------------------------------------ */
/* R6: block layout.  One block per (page, kv head); blocks are stored  */
/* page-major: block index = page * num_kv_heads + head.                */
/*   K block (also the latent cache):                                   */
/*     codes  in tiles of 8 tokens x 32 channels, 128 bytes each, tile  */
/*            (t/8, d/32) at byte ((t/8)*(D/32) + d/32)*128; inside a   */
/*            tile token t%8 takes 16 bytes and byte (d%32)/2 holds     */
/*            channel d, low nibble = even channel.  (This is the order */
/*            a block-scaled tensor-core MMA reads 8-row tiles in.)     */
/*     scales [P][D/32] UE8M0 byte per (token, 32-channel group)        */
/*   V block:                                                           */
/*     codes  [D][P/2]  channel-major; byte (d, j) holds token 2j in    */
/*                      the low nibble, token 2j+1 in the high nibble   */
/*     scales [P][D/32] as for K                                        */
/* Block bytes = P*D/2 + P*D/32 = 17 bytes per 32 values.               */
/* ------------------------------------------------------------------ */
size_t orc_block_bytes(int page_size, int D) {
  return (size_t)page_size * (size_t)D / 2 + (size_t)page_size * (size_t)D / 32;
}

static void put_nibble(uint8_t* byte, int high, int code) {
  if (high) *byte = (uint8_t)((*byte & 0x0F) | (code << 4));
  else *byte = (uint8_t)((*byte & 0xF0) | (code & 0x0F));
}

static int get_nibble(uint8_t byte, int high) {
  return high ? (byte >> 4) & 0xF : byte & 0xF;
}

/* Byte of (token t, channel d) in a K code plane (R6). */
static size_t k_code_byte(int D, int t, int d) {
  return ((size_t)(t / 8) * (D / 32) + d / 32) * 128 + (size_t)(t % 8) * 16 + (d % 32) / 2;
}

void orc_pack_k_token(uint8_t* block, int page_size, int D, int off,
                      const uint8_t* codes, const int* expo) {
  for (int d = 0; d < D; ++d) put_nibble(&block[k_code_byte(D, off, d)], d & 1, codes[d]);
  uint8_t* s = block + (size_t)page_size * D / 2 + (size_t)off * (D / 32);
  for (int g = 0; g < D / 32; ++g) s[g] = (uint8_t)(expo[g] + 127);
}

void orc_pack_v_token(uint8_t* block, int page_size, int D, int off,
                      const uint8_t* codes, const int* expo) {
  for (int d = 0; d < D; ++d) {
    uint8_t* b = block + (size_t)d * (page_size / 2) + off / 2;
    put_nibble(b, off & 1, codes[d]);
  }
  uint8_t* s = block + (size_t)page_size * D / 2 + (size_t)off * (D / 32);
  for (int g = 0; g < D / 32; ++g) s[g] = (uint8_t)(expo[g] + 127);
}

/* Dequantised (still rotated) value of one cached token, fp64, exact. */
void orc_unpack_k_token(const uint8_t* block, int page_size, int D, int off, double* out) {
  const uint8_t* s = block + (size_t)page_size * D / 2 + (size_t)off * (D / 32);
  for (int d = 0; d < D; ++d) {
    int code = get_nibble(block[k_code_byte(D, off, d)], d & 1);
    out[d] = ldexp(orc_e2m1_decode(code), (int)s[d / 32] - 127);
  }
}

void orc_unpack_v_token(const uint8_t* block, int page_size, int D, int off, double* out) {
  const uint8_t* s = block + (size_t)page_size * D / 2 + (size_t)off * (D / 32);
  for (int d = 0; d < D; ++d) {
    const uint8_t b = block[(size_t)d * (page_size / 2) + off / 2];
    int code = get_nibble(b, off & 1);
    out[d] = ldexp(orc_e2m1_decode(code), (int)s[d / 32] - 127);
  }
}

/* ------------------------------------------------------------------ */
/* Quantise-on-append: token i is written at slot_mapping[i] (negative  */
/* slots are skipped).  k, v: bf16 [num_tokens][Hkv][D]; v may be NULL  */
/* (latent cache: only the K cache is written).                         */
/* Returns ORC_INEXACT if any vector was outside the exact domain.      */
/* ------------------------------------------------------------------ */
int orc_append_quantize(const uint16_t* k, const uint16_t* v, int num_tokens,
                        int Hkv, int D, const int32_t* slot_mapping,
                        uint8_t* k_cache, uint8_t* v_cache, int num_pages,
                        int page_size) {
  if (!is_pow2_dim(D) || page_size <= 0 || (page_size & 1)) return ORC_BAD_ARG;
  const size_t bb = orc_block_bytes(page_size, D);
  for (int i = 0; i < num_tokens; ++i)
    if (slot_mapping[i] >= 0 && slot_mapping[i] / page_size >= num_pages) return ORC_BAD_ARG;
  int bad = 0, inexact = 0;
  (void)hadamard_cached(D);
  /* Heads write disjoint blocks, so they may run in parallel; the tokens of
   * one head run in order (two tokens share each V byte). */
#pragma omp parallel for schedule(static) reduction(|:bad, inexact)
  for (int h = 0; h < Hkv; ++h) {
    for (int i = 0; i < num_tokens; ++i) {
      int slot = slot_mapping[i];
      if (slot < 0) continue;
      int page = slot / page_size, off = slot % page_size;
      uint8_t codes[512];
      int expo[16];
      int st = orc_quantize_vector(k + ((size_t)i * Hkv + h) * D, D, codes, expo);
      if (st == ORC_BAD_ARG) { bad = 1; continue; }
      if (st == ORC_INEXACT) inexact = 1;
      orc_pack_k_token(k_cache + ((size_t)page * Hkv + h) * bb, page_size, D, off, codes, expo);
      if (v) {
        st = orc_quantize_vector(v + ((size_t)i * Hkv + h) * D, D, codes, expo);
        if (st == ORC_BAD_ARG) { bad = 1; continue; }
        if (st == ORC_INEXACT) inexact = 1;
        orc_pack_v_token(v_cache + ((size_t)page * Hkv + h) * bb, page_size, D, off, codes, expo);
      }
    }
  }
  return bad ? ORC_BAD_ARG : (inexact ? ORC_INEXACT : ORC_OK);
}

/* ------------------------------------------------------------------ */
/* Softmax attention of one query row over n keys, fp64.                */
/* out[d] = sum_t softmax(scale * q.k_t)_t * v_t[d]; also returns the   */
/* natural log of sum_t exp(scale*q.k_t) (the log-sum-exp).             */
/* ------------------------------------------------------------------ */
double orc_attend_row(const double* q, const double* K, const double* V, int n, int D,
                      double scale, double* out) {
  double* s = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
  double m = -INFINITY;
  for (int t = 0; t < n; ++t) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += q[d] * K[(size_t)t * D + d];
    s[t] = scale * acc;
    if (s[t] > m) m = s[t];
  }
  double l = 0.0;
  for (int t = 0; t < n; ++t) { s[t] = exp(s[t] - m); l += s[t]; }
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  for (int t = 0; t < n; ++t) {
    double p = s[t] / l;
    for (int d = 0; d < D; ++d) out[d] += p * V[(size_t)t * D + d];
  }
  free(s);
  return n > 0 ? m + log(l) : -INFINITY;
}

/* ------------------------------------------------------------------ */
/* Paged decode attention over the 4-bit cache.                         */
/*   q: bf16 [B][T][Hq][D] (not rotated); query head hq reads kv head   */
/*      hq / (Hq/Hkv).  context_lens[b] counts the T new tokens; query  */
/*      position j sees tokens t < context_lens[b] - T + 1 + j.         */
/*   latent != 0: one cache (k_cache) serves as both K and V.           */
/*   out: fp64 [B][T][Hq][D] in the original (unrotated) space.         */
/*   seqs / n_seqs: optional list of sequences to evaluate (NULL: all). */
/* ------------------------------------------------------------------ */
int orc_decode_attention(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                         const int32_t* block_tables, const int32_t* context_lens,
                         int B, int T, int Hq, int Hkv, int D, int page_size,
                         int max_pages, int num_pages, double scale, int latent,
                         const int32_t* seqs, int n_seqs, double* out) {
  if (!is_pow2_dim(D) || Hkv <= 0 || Hq % Hkv != 0 || T < 1) return ORC_BAD_ARG;
  const int G = Hq / Hkv;
  const size_t bb = orc_block_bytes(page_size, D);
  const int nsel = seqs ? n_seqs : B;
  int bad = 0;
  (void)hadamard_cached(D); /* build the matrix before the threads share it */
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(|:bad)
  for (int si = 0; si < nsel; ++si) {
    for (int h = 0; h < Hkv; ++h) {
      const int b = seqs ? seqs[si] : si;
      const int L = context_lens[b];
      if (L < T || L > max_pages * page_size) { bad = 1; continue; }
      double* Kd = (double*)malloc(sizeof(double) * (size_t)L * D);
      double* Vd = (double*)malloc(sizeof(double) * (size_t)L * D);
      for (int t = 0; t < L; ++t) {
        int page = block_tables[(size_t)b * max_pages + t / page_size];
        if (page < 0 || page >= num_pages) { bad = 1; page = 0; }
        const uint8_t* kb = k_cache + ((size_t)page * Hkv + h) * bb;
        orc_unpack_k_token(kb, page_size, D, t % page_size, Kd + (size_t)t * D);
        if (latent) memcpy(Vd + (size_t)t * D, Kd + (size_t)t * D, sizeof(double) * D);
        else orc_unpack_v_token(v_cache + ((size_t)page * Hkv + h) * bb, page_size, D,
                                t % page_size, Vd + (size_t)t * D);
      }
      for (int j = 0; j < T; ++j)
        for (int g = 0; g < G; ++g) {
          const int hq = h * G + g;
          double qv[512], qr[512], orot[512];
          for (int d = 0; d < D; ++d)
            qv[d] = (double)bf16_to_float(q[(((size_t)b * T + j) * Hq + hq) * D + d]);
          orc_rotate_f64(qv, D, qr);
          const int n = L - T + 1 + j;
          orc_attend_row(qr, Kd, Vd, n, D, scale, orot);
          orc_rotate_f64(orot, D, out + (((size_t)b * T + j) * Hq + hq) * D);
        }
      free(Kd);
      free(Vd);
    }
  }
  return bad ? ORC_BAD_ARG : ORC_OK;
}

/* ------------------------------------------------------------------ */
/* R7: FP8 E4M3 (OCP): 1 sign, 4 exponent (bias 7), 3 mantissa bits;   */
/* no infinities; S.1111.111 is NaN; largest finite 448; subnormals     */
/* m * 2^-9.                                                            */
/* ------------------------------------------------------------------ */
double orc_e4m3_decode(int byte) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 0xF, m = byte & 7;
  double v;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

int orc_e4m3_encode(float xf) {
  double x = (double)xf;
  int s = signbit(x) ? 1 : 0;
  double a = fabs(x);
  if (isnan(a)) return 0x7F | (s << 7);
  if (a >= 448.0) return (s << 7) | 0x7E; /* saturate (RNE never exceeds 448 below 464) */
  /* quantum of the binade holding a (subnormal binade shares 2^-9) */
  double quantum;
  if (a < 0x1.0p-6) quantum = 0x1.0p-9;
  else {
    int k;
    (void)frexp(a, &k); /* a in [2^(k-1), 2^k) */
    quantum = ldexp(1.0, (k - 1) - 3);
  }
  double n = a / quantum; /* exact */
  double fl = floor(n), fr = n - fl;
  double r;
  if (fr > 0.5) r = fl + 1.0;
  else if (fr < 0.5) r = fl;
  else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  double val = r * quantum;
  if (val > 448.0) val = 448.0;
  /* encode val exactly */
  int code;
  if (val == 0.0) code = 0;
  else if (val < 0x1.0p-6) code = (int)(val / 0x1.0p-9);
  else {
    int k;
    double f = frexp(val, &k); /* val = f 2^k, f in [0.5,1) => 1.m * 2^(k-1) */
    int e = (k - 1) + 7;
    int m = (int)((f * 2.0 - 1.0) * 8.0);
    code = (e << 3) | m;
  }
  return (s << 7) | code;
}

/* FP8 block layout per (page, kv head):
 *   K block: [P][D] token-major bytes;  V block: [D][P] channel-major bytes.
 * Code = E4M3(fp32(x * inv_scale[h])). */
int orc_fp8_append(const uint16_t* k, const uint16_t* v, int num_tokens, int Hkv, int D,
                   const int32_t* slot_mapping, const float* k_inv_scale,
                   const float* v_inv_scale, uint8_t* k_cache, uint8_t* v_cache,
                   int num_pages, int page_size) {
  const size_t bb = (size_t)page_size * D;
  for (int i = 0; i < num_tokens; ++i) {
    int slot = slot_mapping[i];
    if (slot < 0) continue;
    int page = slot / page_size, off = slot % page_size;
    if (page >= num_pages) return ORC_BAD_ARG;
    for (int h = 0; h < Hkv; ++h) {
      uint8_t* kb = k_cache + ((size_t)page * Hkv + h) * bb;
      uint8_t* vb = v_cache + ((size_t)page * Hkv + h) * bb;
      for (int d = 0; d < D; ++d) {
        float kx = bf16_to_float(k[((size_t)i * Hkv + h) * D + d]) * k_inv_scale[h];
        float vx = bf16_to_float(v[((size_t)i * Hkv + h) * D + d]) * v_inv_scale[h];
        kb[(size_t)off * D + d] = (uint8_t)orc_e4m3_encode(kx);
        vb[(size_t)d * page_size + off] = (uint8_t)orc_e4m3_encode(vx);
      }
    }
  }
  return ORC_OK;
}

int orc_fp8_decode_attention(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                             const float* k_scale, const float* v_scale,
                             const int32_t* block_tables, const int32_t* context_lens,
                             int B, int T, int Hq, int Hkv, int D, int page_size,
                             int max_pages, int num_pages, double scale,
                             const int32_t* seqs, int n_seqs, double* out) {
  if (Hkv <= 0 || Hq % Hkv != 0 || T < 1 || D <= 0 || D > 512) return ORC_BAD_ARG;
  const int G = Hq / Hkv;
  const size_t bb = (size_t)page_size * D;
  const int nsel = seqs ? n_seqs : B;
  int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(|:bad)
  for (int si = 0; si < nsel; ++si) {
    for (int h = 0; h < Hkv; ++h) {
      const int b = seqs ? seqs[si] : si;
      const int L = context_lens[b];
      if (L < T || L > max_pages * page_size) { bad = 1; continue; }
      double* Kd = (double*)malloc(sizeof(double) * (size_t)L * D);
      double* Vd = (double*)malloc(sizeof(double) * (size_t)L * D);
      for (int t = 0; t < L; ++t) {
        int page = block_tables[(size_t)b * max_pages + t / page_size];
        if (page < 0 || page >= num_pages) { bad = 1; page = 0; }
        const uint8_t* kb = k_cache + ((size_t)page * Hkv + h) * bb;
        const uint8_t* vb = v_cache + ((size_t)page * Hkv + h) * bb;
        const int off = t % page_size;
        for (int d = 0; d < D; ++d) {
          Kd[(size_t)t * D + d] = orc_e4m3_decode(kb[(size_t)off * D + d]) * (double)k_scale[h];
          Vd[(size_t)t * D + d] = orc_e4m3_decode(vb[(size_t)d * page_size + off]) * (double)v_scale[h];
        }
      }
      for (int j = 0; j < T; ++j)
        for (int g = 0; g < G; ++g) {
          const int hq = h * G + g;
          double qv[512];
          for (int d = 0; d < D; ++d)
            qv[d] = (double)bf16_to_float(q[(((size_t)b * T + j) * Hq + hq) * D + d]);
          const int n = L - T + 1 + j;
          orc_attend_row(qv, Kd, Vd, n, D, scale, out + (((size_t)b * T + j) * Hq + hq) * D);
        }
      free(Kd);
      free(Vd);
    }
  }
  return bad ? ORC_BAD_ARG : ORC_OK;
}

/* ------------------------------------------------------------------ */
/* Array helpers for the Python test wrapper.                           */
/* ------------------------------------------------------------------ */
void orc_e2m1_encode_array(const double* z, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e2m1_encode(z[i]);
}

void orc_e4m3_encode_array(const float* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)orc_e4m3_encode(x[i]);
}

void orc_e4m3_decode_array(const uint8_t* b, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(b[i]);
}

/* Quantise many vectors: x [n][D] bf16 -> codes [n][D] (one per byte),
 * expo [n][D/32]; returns the number of vectors outside the exact domain. */
int64_t orc_quantize_vectors(const uint16_t* x, int64_t n, int D, uint8_t* codes, int* expo) {
  int64_t inexact = 0;
  (void)hadamard_cached(D);
#pragma omp parallel for schedule(static) reduction(+:inexact)
  for (int64_t i = 0; i < n; ++i) {
    int st = orc_quantize_vector(x + i * D, D, codes + i * D, expo + i * (D / 32));
    if (st != ORC_OK) inexact += 1;
  }
  return inexact;
}

/* ------------------------------------------------------------------ */
/* Thread count of the OpenMP loops above.  Only the timing of the CPU  */
/* baseline uses it; no result depends on the thread count.             */
/* ------------------------------------------------------------------ */
void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
