/*
 * bitlinear_oracle.c -- plain, slow CPU oracle for the BitLinear W1.58A8 layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file:
 * only the tests, the smoke check and the CPU-baseline leg of the benchmark do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (BitNet b1.58 BitLinear, as used by the pages:
 *   "Add Support for BitNet Architecture Inference" (Candle PR), the
 *   answer that lists the changes made: every Linear in the MLP and the
 *   attention becomes a BitLinear, an RMSNorm sits before it, and
 *   `activation_quant` / `weight_quant` are implemented as in the BitNet
 *   paper; "Transformer Block", section "Feed-Forward Network": the gated
 *   FFN  hidden = ReLU^2(x W_gate) * (x W_up),  out = hidden W_down):
 *
 *   weight_quant (absmean):   sw = 1 / max(mean|W|, 1e-5)
 *                             Wq = clamp(round_half_even(W * sw), -1, 1)
 *   activation_quant (absmax, per token row):
 *                             sx = 127 / max(max_k |x|, 1e-5)
 *                             xq = clamp(round_half_even(x * sx), -128, 127)
 *   contraction:              acc[m,n] = sum_k xq[m,k] * Wq[n,k]   (exact integer)
 *   rescale:                  y[m,n] = acc[m,n] / (sx[m] * sw)
 *
 * Readings taken where the pages are silent (all stated, none invented):
 *  - Every quantisation decision (the products W*sw, x*sx and the scales
 *    themselves) is taken in IEEE fp32 with round-to-nearest-even, the
 *    precision of the data.  The rescale y is computed here in fp64.
 *  - mean|W| is the exact sum of |W| (every term is a float, the sum is
 *    carried exactly in a wide fixed-point integer), rounded once to fp64,
 *    divided by N*K in fp64 and rounded to fp32.  This makes the mean
 *    independent of summation order.
 *  - The optional RMSNorm prologue (Transformer Block "Architecture": an
 *    RMSNorm before each projection) is the LLaMA form
 *        inv = 1 / sqrt(sum_k h_k^2 / K + eps)      (fp64 from the exact sum)
 *        xn_k = (h_k * (float)inv) * gamma_k         (two fp32 products)
 *  - The optional gated prologue is h = (r*r)*u with r = max(g, 0), in fp32
 *    (ReLU squared, "BitNet uses relu_sqr, NOT silu" in the FFN section).
 *    When both prologues are requested the gate comes first, then the norm
 *    (the FFN sub-norm sits between the gating and the down projection).
 *
 * Packed weight layout (this library's own format, 2 bits per weight, the
 * 0.25 bytes per weight of the pages' memory tables):
 *   code = Wq + 1 in {0,1,2}; 3 is invalid; positions past K hold code 1 (0).
 *   The 16-byte chunk for row n and k-block kb = k/64 starts at byte
 *   (kb*N + n)*16.  Inside it, 32-bit little-endian word w = (k%64)/16 holds
 *   i = k%16 at bit 8*(i%4) + 2*(i/4).
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off (no fast-math).  The oracle asserts
 * that the FPU is in round-to-nearest mode before every entry point.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_SHAPE (-2)
#define ORACLE_ERR_CODE (-7)
#define ORACLE_ERR_ROUNDING (-8)

/* ------------------------------------------------------------------------ */
/* Exact sums of floats: a fixed-point integer with 32-bit digits.           */
/* value = sum_i digit[i] * 2^(32*i - FX_BIAS).  Every |float| and every     */
/* float squared is an integer times 2^(>= -298), below 2^256, so 24 digits  */
/* (768 bits) hold any sum of up to 2^40 such terms exactly.                 */
/* ------------------------------------------------------------------------ */
#define FX_BIAS 320
#define FX_DIGITS 24

typedef struct {
  uint64_t d[FX_DIGITS]; /* each digit kept below 2^32 after every add */
} fx_sum;

static void fx_clear(fx_sum* a) { memset(a, 0, sizeof(*a)); }

/* a += mant * 2^e2, mant < 2^48, e2 >= -FX_BIAS */
static void fx_add(fx_sum* a, uint64_t mant, int e2) {
  if (mant == 0) return;
  int pos = e2 + FX_BIAS;
  int i = pos / 32;
  int s = pos % 32;
  unsigned __int128 v = ((unsigned __int128)mant) << s;
  for (int j = i; j < FX_DIGITS && v != 0; ++j) {
    a->d[j] += (uint64_t)(v & 0xffffffffu);
    v >>= 32;
  }
  for (int j = i; j + 1 < FX_DIGITS; ++j) { /* propagate carries */
    uint64_t c = a->d[j] >> 32;
    a->d[j] &= 0xffffffffu;
    a->d[j + 1] += c;
  }
}

static int fx_bit(const fx_sum* a, int p) {
  return (int)((a->d[p / 32] >> (p % 32)) & 1u);
}

/* Round the exact value to the nearest double, ties to even. */
static double fx_to_double(const fx_sum* a) {
  int top = -1;
  for (int p = FX_DIGITS * 32 - 1; p >= 0; --p) {
    if (fx_bit(a, p)) { top = p; break; }
  }
  if (top < 0) return 0.0;
  if (top <= 52) { /* fits in 53 bits: exact */
    uint64_t m = 0;
    for (int p = top; p >= 0; --p) m = (m << 1) | (uint64_t)fx_bit(a, p);
    return ldexp((double)m, -FX_BIAS);
  }
  uint64_t m = 0;
  for (int p = top; p >= top - 52; --p) m = (m << 1) | (uint64_t)fx_bit(a, p);
  int round_bit = fx_bit(a, top - 53);
  int sticky = 0;
  for (int p = top - 54; p >= 0; --p) {
    if (fx_bit(a, p)) { sticky = 1; break; }
  }
  int lsb_exp = top - 52 - FX_BIAS;
  if (round_bit && (sticky || (m & 1u))) {
    m += 1;
    if (m == (1ull << 53)) { m >>= 1; lsb_exp += 1; }
  }
  return ldexp((double)m, lsb_exp);
}

/* |f| = mant * 2^e2 with mant < 2^24 */
static void float_abs_parts(float f, uint64_t* mant, int* e2) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t e = (u >> 23) & 0xffu;
  uint32_t frac = u & 0x7fffffu;
  if (e == 0) { *mant = frac; *e2 = -149; }
  else { *mant = (uint64_t)(frac | 0x800000u); *e2 = (int)e - 150; }
}

/* Exact sum of |v[i]|, rounded once to fp64. */
double oracle_exact_abs_sum(const float* v, int64_t n) {
  fx_sum a;
  fx_clear(&a);
  for (int64_t i = 0; i < n; ++i) {
    uint64_t m; int e2;
    float_abs_parts(v[i], &m, &e2);
    fx_add(&a, m, e2);
  }
  return fx_to_double(&a);
}

/* Exact sum of v[i]^2 (each square is exact in 48 bits), rounded once to fp64. */
double oracle_exact_sq_sum(const float* v, int64_t n) {
  fx_sum a;
  fx_clear(&a);
  for (int64_t i = 0; i < n; ++i) {
    uint64_t m; int e2;
    float_abs_parts(v[i], &m, &e2);
    fx_add(&a, m * m, 2 * e2);
  }
  return fx_to_double(&a);
}

static int rounding_ok(void) { return fegetround() == FE_TONEAREST; }

/* round half to even in the current (nearest) mode, then clamp */
static int32_t rne_clamp(float t, int32_t lo, int32_t hi) {
  float r = nearbyintf(t);
  if (r < (float)lo) return lo;
  if (r > (float)hi) return hi;
  return (int32_t)r;
}

/* ------------------------------------------------------------------------ */
/* weight_quant: absmean ternary quantiser.                                  */
/* ------------------------------------------------------------------------ */
int oracle_weight_quant(const float* W, int64_t N, int64_t K, int8_t* Wq,
                        float* sw_out, float* mean_out) {
  if (!rounding_ok()) return ORACLE_ERR_ROUNDING;
  if (N <= 0 || K <= 0) return ORACLE_ERR_SHAPE;
  double S = oracle_exact_abs_sum(W, N * K);
  float mean = (float)(S / (double)(N * K));
  float sw = 1.0f / fmaxf(mean, 1e-5f);
  for (int64_t i = 0; i < N * K; ++i) {
    float t = W[i] * sw;
    Wq[i] = (int8_t)rne_clamp(t, -1, 1);
  }
  *sw_out = sw;
  if (mean_out) *mean_out = mean;
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Pack / unpack of the 2-bit layout described in the header.                */
/* ------------------------------------------------------------------------ */
int64_t oracle_packed_bytes(int64_t N, int64_t K) {
  if (N <= 0 || K <= 0) return 0;
  return N * ((K + 63) / 64) * 16;
}

static int64_t code_byte(int64_t N, int64_t n, int64_t k, int* shift) {
  int64_t kb = k / 64;
  int64_t w = (k % 64) / 16;
  int64_t i = k % 16;
  *shift = (int)(2 * (i / 4));
  return (kb * N + n) * 16 + 4 * w + (i % 4);
}

int oracle_pack(const int8_t* Wq, int64_t N, int64_t K, uint8_t* packed) {
  if (N <= 0 || K <= 0) return ORACLE_ERR_SHAPE;
  memset(packed, 0x55, (size_t)oracle_packed_bytes(N, K)); /* every code = 1 */
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      int q = Wq[n * K + k];
      if (q < -1 || q > 1) return ORACLE_ERR_CODE;
      int sh;
      int64_t b = code_byte(N, n, k, &sh);
      packed[b] = (uint8_t)((packed[b] & ~(3u << sh)) | ((unsigned)(q + 1) << sh));
    }
  }
  return ORACLE_OK;
}

static int ternary_at(const uint8_t* packed, int64_t N, int64_t n, int64_t k, int* q) {
  int sh;
  int64_t b = code_byte(N, n, k, &sh);
  int code = (packed[b] >> sh) & 3;
  if (code == 3) return ORACLE_ERR_CODE;
  *q = code - 1;
  return ORACLE_OK;
}

int oracle_unpack(const uint8_t* packed, int64_t N, int64_t K, int8_t* Wq) {
  if (N <= 0 || K <= 0) return ORACLE_ERR_SHAPE;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t k = 0; k < K; ++k) {
      int q;
      if (ternary_at(packed, N, n, k, &q) != ORACLE_OK) return ORACLE_ERR_CODE;
      Wq[n * K + k] = (int8_t)q;
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* activation_quant with the optional gated and RMSNorm prologues.           */
/* mul == NULL: h = x.  mul != NULL: h = (r*r)*mul with r = max(x, 0).       */
/* gamma == NULL: no norm.  Otherwise h := (h * inv) * gamma.                */
/* h_out (optional) receives the fp32 row fed to the quantiser.              */
/* ------------------------------------------------------------------------ */
int oracle_act_quant(const float* x, const float* mul, int64_t M, int64_t K,
                     const float* gamma, double eps, int8_t* xq, float* sx,
                     float* h_out) {
  if (!rounding_ok()) return ORACLE_ERR_ROUNDING;
  if (M < 0 || K <= 0) return ORACLE_ERR_SHAPE;
  float* h = (float*)malloc((size_t)K * sizeof(float));
  if (!h) return ORACLE_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    const float* xr = x + m * K;
    for (int64_t k = 0; k < K; ++k) {
      if (mul) {
        float r = fmaxf(xr[k], 0.0f);
        float rr = r * r;
        h[k] = rr * mul[m * K + k];
      } else {
        h[k] = xr[k];
      }
    }
    if (gamma) {
      double S = oracle_exact_sq_sum(h, K);
      float inv = (float)(1.0 / sqrt(S / (double)K + eps));
      for (int64_t k = 0; k < K; ++k) {
        float t = h[k] * inv;
        h[k] = t * gamma[k];
      }
    }
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) amax = fmaxf(amax, fabsf(h[k]));
    float s = 127.0f / fmaxf(amax, 1e-5f);
    for (int64_t k = 0; k < K; ++k) {
      float t = h[k] * s;
      xq[m * K + k] = (int8_t)rne_clamp(t, -128, 127);
    }
    sx[m] = s;
    if (h_out) memcpy(h_out + m * K, h, (size_t)K * sizeof(float));
  }
  free(h);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Contraction on the packed weights and the rescale.                        */
/* acc (optional) gets the exact int32 sums, y (optional) the fp64 outputs.  */
/* ------------------------------------------------------------------------ */
int oracle_forward(const int8_t* xq, const float* sx, int64_t M,
                   const uint8_t* packed, float sw, int64_t N, int64_t K,
                   int32_t* acc, double* y) {
  if (M < 0 || N <= 0 || K <= 0) return ORACLE_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      int64_t a = 0;
      for (int64_t k = 0; k < K; ++k) {
        int q;
        if (ternary_at(packed, N, n, k, &q) != ORACLE_OK) return ORACLE_ERR_CODE;
        a += (int64_t)xq[m * K + k] * (int64_t)q;
      }
      if (acc) acc[m * N + n] = (int32_t)a;
      if (y) y[m * N + n] = (double)a / ((double)sx[m] * (double)sw);
    }
  }
  return ORACLE_OK;
}

/* Same contraction on unpacked ternary weights Wq [N,K] (used to check the
 * packed path against a layout-free one). */
int oracle_forward_unpacked(const int8_t* xq, const float* sx, int64_t M,
                            const int8_t* Wq, float sw, int64_t N, int64_t K,
                            int32_t* acc, double* y) {
  if (M < 0 || N <= 0 || K <= 0) return ORACLE_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      int64_t a = 0;
      for (int64_t k = 0; k < K; ++k) a += (int64_t)xq[m * K + k] * (int64_t)Wq[n * K + k];
      if (acc) acc[m * N + n] = (int32_t)a;
      if (y) y[m * N + n] = (double)a / ((double)sx[m] * (double)sw);
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Greedy choice after the LM head: out[m] = the first n whose y[m, n] is    */
/* the row's largest ("Hesper.Models.BitNet" page, "Performance (BitNet-3B   */
/* on A100)": the LM head is a BitLinear; greedy decoding takes the argmax   */
/* of its logits).  fp32 inputs are passed widened to fp64 (exact).          */
/* ------------------------------------------------------------------------ */
int oracle_argmax(const double* y, int64_t M, int64_t N, int32_t* out) {
  if (M < 0 || N <= 0) return ORACLE_ERR_SHAPE;
  for (int64_t m = 0; m < M; ++m) {
    int64_t best = 0;
    for (int64_t n = 1; n < N; ++n)
      if (y[m * N + n] > y[m * N + best]) best = n;
    out[m] = (int32_t)best;
  }
  return ORACLE_OK;
}
