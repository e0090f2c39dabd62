/*
 * skv_oracle.c -- plain, slow, single-threaded CPU oracle for speculative KV
 * coding (lossless coding of a target KV cache against a predictor's
 * approximation of it).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg load this library.  The CUDA library never
 * calls it, and the two share no source, header, table or constant.
 *
 * Parity pins (what fixes each function independently of its own code) are
 * listed in the test files; functions without an independent pin say so.
 *
 * Sources, cited by page title and section:
 *   [SKV]  "Speculative KV coding: losslessly compressing KV cache by up to
 *          ~4x" (Fergus Finn, summarised at aisparkup.com/posts/13411).
 *          Sections: "core idea" (residual of target against a deterministic
 *          predictor, coded losslessly; decoder re-runs the predictor and adds
 *          the decoded residual back), "which predictor" (residual statistics
 *          measured once on a little calibration data, then frozen).
 *   [DCKV] "DCKV compresses a hybrid language model's prompt KV cache with
 *          learned transform coding" (onedev.kr/papers/1428).  Sections:
 *          "how it works" (components whose scale/step ratio is below 0.05 are
 *          switched off in storage and reconstruction), "how it differs"
 *          (GPU rANS; static model = per-component Laplace integrated over the
 *          quantisation cells; a token-conditioned model shifts the Laplace
 *          by a predicted mean), "usage" (bit-identical decode across devices
 *          is not verified for a float model -> everything here is integer).
 *
 * Where the pages leave a step open, the plainest reading is taken; every
 * such reading is marked READING below.
 *
 * All arithmetic is integer (uint64_t / int64_t) except the one fp32 rounding
 * of a coefficient mean (COEF streams), done in IEEE single precision.
 * Build with -ffp-contract=off.  Every function is reentrant (no static
 * buffers), so callers may run chunks in parallel processes or threads.
 */
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#include <math.h>
#include <stdlib.h>

#define OR_FP8 1u
#define OR_BF16 2u
#define OR_COEF 3u

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_CAPACITY 3
#define OR_ERR_CORRUPT 4

/* Coding constants.  READING: the pages fix none of these numerically; they
 * are the plain choices of a 32-bit-state rANS coder with 16-bit
 * renormalisation and 12-bit probabilities over a 256-symbol alphabet. */
#define PROB_BITS 12u
#define PROB_SCALE 4096u          /* 2^PROB_BITS                          */
#define RANS_L 65536u             /* lower bound of the normalised state  */
#define NSYM 256u
#define ESC 255u                  /* escape symbol                        */
#define RMAX 127                  /* |r| <= RMAX is coded directly        */
#define LANES 32u                 /* lanes per chunk                      */
#define CHAIN_LEN 2056u           /* powers tau^0 .. tau^2055             */

typedef struct {
  uint32_t version;
  uint32_t dtype;     /* OR_FP8, OR_BF16, OR_COEF                          */
  uint32_t n_layers;  /* KV: layout [layer][kv][head][token][head_dim]      */
  uint32_t n_kv;
  uint32_t n_heads;
  uint32_t head_dim;
  uint64_t n_tokens;
  uint32_t n_coef;    /* COEF: layout [token][coef]                         */
  uint32_t lane_syms; /* K: positions per lane; a chunk is 32*K positions    */
  uint32_t n_calib;   /* calibration tokens per channel                      */
  uint32_t model;     /* residual model: 0 per-channel scale bins, 1 (FP8)  */
                      /* per-channel scale normalised by the prediction's   */
                      /* exponent (see O3b)                                  */
} or_params;

/* ------------------------------------------------------------------------ */
/* Geometry.  A "slice" is a contiguous run of positions that chunks never    */
/* straddle: one (layer, kv, head) block of n_tokens*head_dim positions for   */
/* a KV cache, the whole [token][coef] grid for a coefficient stream.         */
/* ------------------------------------------------------------------------ */

static uint32_t elem_bytes(const or_params *p) {
  return p->dtype == OR_FP8 ? 1u : 2u;
}
/* group size: consecutive positions a lane owns before the next lane starts */
uint32_t or_group(const or_params *p) { return p->dtype == OR_FP8 ? 16u : 8u; }
/* raw bytes carried by an escape: the residual width in bytes */
static uint32_t raw_bytes(const or_params *p) { return p->dtype == OR_FP8 ? 1u : 2u; }

uint64_t or_num_slices(const or_params *p) {
  if (p->dtype == OR_COEF) return 1;
  return (uint64_t)p->n_layers * p->n_kv * p->n_heads;
}
uint64_t or_slice_positions(const or_params *p) {
  if (p->dtype == OR_COEF) return p->n_tokens * (uint64_t)p->n_coef;
  return p->n_tokens * (uint64_t)p->head_dim;
}
uint64_t or_chunks_per_slice(const or_params *p) {
  uint64_t cs = (uint64_t)LANES * p->lane_syms;
  return (or_slice_positions(p) + cs - 1) / cs;
}
uint64_t or_num_chunks(const or_params *p) {
  return or_num_slices(p) * or_chunks_per_slice(p);
}
uint64_t or_num_lanes(const or_params *p) { return or_num_chunks(p) * LANES; }
uint64_t or_num_channels(const or_params *p) {
  if (p->dtype == OR_COEF) return p->n_coef;
  return or_num_slices(p) * p->head_dim;
}
/* sub-bins per octave of the scale grid: KV 4 (32 bins), COEF 8 (64 bins) */
uint32_t or_sub_bins(const or_params *p) { return p->dtype == OR_COEF ? 8u : 4u; }
uint32_t or_num_tables(const or_params *p) {
  return p->dtype == OR_COEF ? 64u * 16u : 32u;
}
/* worst-case 16-bit words of one lane stream: two state words plus at most
 * one renormalisation word per coding step, and an escaped position takes
 * 1 + raw_bytes steps */
uint64_t or_max_lane_words(const or_params *p) {
  return 2 + (uint64_t)p->lane_syms * (1 + raw_bytes(p));
}

int or_check_params(const or_params *p) {
  if (p->dtype != OR_FP8 && p->dtype != OR_BF16 && p->dtype != OR_COEF) return OR_ERR_ARG;
  if (p->model > 1u || (p->model == 1u && p->dtype != OR_FP8)) return OR_ERR_ARG;
  if (p->lane_syms == 0 || (p->lane_syms % or_group(p)) != 0) return OR_ERR_ARG;
  if (p->dtype != OR_COEF) {
    if (p->head_dim == 0 || (p->head_dim % or_group(p)) != 0) return OR_ERR_ARG;
  } else {
    if (p->n_coef == 0) return OR_ERR_ARG;
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* O1: monotone ordinal of a bit pattern.  [SKV] core idea codes the          */
/* difference between target and prediction; the difference is taken between */
/* ordinals so that neighbouring representable values differ by one.          */
/* READING: sign-magnitude patterns map to unsigned ordinals with            */
/*   non-negative b -> b | top,  negative b -> ~b (within the width),         */
/* a bijection on all patterns, monotone on all non-NaN values, -0 < +0.      */
/* ------------------------------------------------------------------------ */

uint32_t or_ordinal(uint32_t bits, uint32_t width) {
  uint32_t mask = (width == 32u) ? 0xFFFFFFFFu : ((1u << width) - 1u);
  uint32_t top = 1u << (width - 1u);
  bits &= mask;
  if (bits & top) return (~bits) & mask;
  return bits | top;
}

uint32_t or_ordinal_inv(uint32_t u, uint32_t width) {
  uint32_t mask = (width == 32u) ? 0xFFFFFFFFu : ((1u << width) - 1u);
  uint32_t top = 1u << (width - 1u);
  u &= mask;
  if (u & top) return u & ~top;
  return (~u) & mask;
}

/* ------------------------------------------------------------------------ */
/* O3: calibration.  [SKV] which predictor: residual statistics measured      */
/* once on a small calibration set and frozen.  READING: per channel, the     */
/* Laplace scale with location 0 has maximum-likelihood estimate mean|r| over */
/* the first n_calib tokens; it is quantised to a log grid of scale bins.     */
/* ------------------------------------------------------------------------ */

/* q = floor(beta * 2^16).  Bins: q < 2^13 -> 0, q >= 2^21 -> last bin,
 * otherwise octave p = floor(log2 q) in [13, 20] and the sub-bin is the
 * log2(sub) bits right below the leading one. */
uint32_t or_bin_from_q(uint64_t q, uint32_t sub) {
  uint32_t nbins = 8u * sub, sb = (sub == 8u) ? 3u : 2u, pw = 0;
  if (q < (1ull << 13)) return 0;
  if (q >= (1ull << 21)) return nbins - 1u;
  while ((q >> (pw + 1u)) != 0) pw++;            /* pw = floor(log2 q) */
  return sub * (pw - 13u) + (uint32_t)((q >> (pw - sb)) & (sub - 1u));
}

/* O3b: residual model 1 (FP8 only).  [SKV] names "more refined residual
 * models" as the next step; READING: ordinals are evenly spaced in bit
 * patterns, so a fixed value-space error spans 2^-e as many ordinals when the
 * prediction's exponent field e = (bits >> 3) & 15 is one higher.  The
 * channel's scale is therefore fitted on |r| 2^e (the scale at exponent 0),
 * S'_c = sum |r| 2^e over the calibration tokens, q_c = floor(S'_c 2^16 / N),
 * stored as its bin on the log grid extended upward without a cap (the base
 * bin; q below 2^13 -> 0).  A position whose prediction has exponent e uses
 * the table of the scale (base scale) / 2^e: the bin of the base bin's lower
 * edge shifted down e octaves. */
uint32_t or_bin_ext(uint64_t q) {
  uint32_t pw = 0;
  if (q < (1ull << 13)) return 0;
  while ((q >> (pw + 1u)) != 0) pw++;
  return 4u * (pw - 13u) + (uint32_t)((q >> (pw - 2u)) & 3u);
}
/* lower edge (Q16) of base bin b = 4 (p - 13) + j: leading one at p, j below */
static uint64_t bin_ext_lower_q(uint32_t b) {
  uint32_t pw = 13u + b / 4u, j = b % 4u;
  if (pw > 61u) return UINT64_MAX;   /* beyond 2^62: above every table at any e <= 15 */
  return (uint64_t)(4u + j) << (pw - 2u);
}
uint32_t or_model1_table(uint32_t base, uint32_t e) {
  return or_bin_from_q(bin_ext_lower_q(base) >> e, 4u);
}

static uint32_t load_bits(const void *base, uint64_t idx, uint32_t esz) {
  if (esz == 1) return ((const uint8_t *)base)[idx];
  return ((const uint16_t *)base)[idx];
}

/* KV: target/pred are the caches (raw bits).  sum_abs[c] receives the exact
 * sum of |r|, hist[c*256 + symbol] counts calibration symbols (either may be
 * NULL).  COEF: pred is beta_c = b_c/step_c (fp32, one per component); bins
 * 0xFF mark components switched off by the 0.05 rule ([DCKV] how it works). */
int or_calibrate(const or_params *p, const void *target, const void *pred,
                 uint8_t *bins, uint32_t *sum_abs, uint32_t *hist) {
  if (or_check_params(p) != OR_OK) return OR_ERR_ARG;
  if (p->dtype == OR_COEF) {
    const float *beta = (const float *)pred;
    for (uint32_t c = 0; c < p->n_coef; c++) {
      float b = beta[c];
      if (!(b >= 0.05f)) { bins[c] = 0xFF; continue; }     /* NaN -> off */
      if (b >= 32.0f) { bins[c] = 63; continue; }
      float scaled = b * 65536.0f;                          /* exact      */
      bins[c] = (uint8_t)or_bin_from_q((uint64_t)floorf(scaled), 8u);
    }
    return OR_OK;
  }
  uint32_t esz = elem_bytes(p), width = 8u * esz;
  uint64_t T = p->n_tokens, D = p->head_dim;
  uint64_t nc = p->n_calib < T ? p->n_calib : T;
  for (uint64_t s = 0; s < or_num_slices(p); s++) {
    for (uint64_t d = 0; d < D; d++) {
      uint64_t c = s * D + d, S = 0;
      for (uint64_t t = 0; t < nc; t++) {
        uint64_t idx = (s * T + t) * D + d;
        uint32_t pb = load_bits(pred, idx, esz);
        int64_t r = (int64_t)or_ordinal(load_bits(target, idx, esz), width) -
                    (int64_t)or_ordinal(pb, width);
        uint64_t a = (uint64_t)(r < 0 ? -r : r);
        S += p->model == 1u ? a << ((pb >> 3) & 15u) : a;
        if (hist) {
          uint32_t sym = (r >= -RMAX && r <= RMAX) ? (uint32_t)(r + RMAX) : ESC;
          hist[c * NSYM + sym]++;
        }
      }
      if (sum_abs) sum_abs[c] = S > 0xFFFFFFFFull ? 0xFFFFFFFFu : (uint32_t)S;
      uint64_t q = nc ? (S << 16) / nc : 0;     /* floor(S * 2^16 / N) */
      bins[c] = (uint8_t)(p->model == 1u ? or_bin_ext(q) : or_bin_from_q(q, 4u));
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* O4: integer probability tables.  [DCKV] how it differs: a per-component    */
/* Laplace integrated over the quantisation cells gives the probabilities.    */
/* The Laplace CDF is evaluated on a 1/16-step grid from integer powers of    */
/* tau = exp(-1/(16 beta)); every operation below is exact integer            */
/* arithmetic so that any machine reproduces the same table ([DCKV] usage:    */
/* bit-identical decode is not established for float models).                */
/* ------------------------------------------------------------------------ */

/* Representative scale of bin k = sub*e + j: the midpoint of its sub-bin,
 * beta = 2^(e-3) * (1 + (j + 1/2)/sub), returned in Q16. */
uint64_t or_beta_q(uint32_t bin, uint32_t sub) {
  uint32_t e = bin / sub, j = bin % sub;
  /* 2^(e-3) * (2 sub + 2 j + 1)/(2 sub) * 2^16 = 2^(e+13) / (2 sub) * (2sub+2j+1) */
  return ((1ull << (e + 13u)) / (2ull * sub)) * (2ull * sub + 2ull * j + 1ull);
}

/* tau_q = Q32 of exp(-x), x = 1/(16 beta), by the Taylor series up to n = 15:
 * a_0 = 2^32, a_n = round(a_{n-1} * x_q / (n 2^32)), tau = sum (-1)^n a_n. */
uint64_t or_tau_q(uint64_t beta_q) {
  uint64_t x_q = ((1ull << 44) + (beta_q >> 1)) / beta_q;   /* Q32 of 1/(16 beta) */
  uint64_t a = 1ull << 32;
  int64_t tau = (int64_t)a;
  for (uint64_t n = 1; n <= 15; n++) {
    a = (a * x_q + n * (1ull << 31)) / (n << 32);
    tau += (n & 1) ? -(int64_t)a : (int64_t)a;
  }
  return (uint64_t)tau;
}

/* P[n] = Q32 of tau^n, each power rounded from the previous one. */
void or_power_chain(uint64_t tau_q, uint64_t *P) {
  P[0] = 1ull << 32;
  for (uint32_t n = 1; n < CHAIN_LEN; n++) P[n] = (P[n - 1] * tau_q + (1ull << 31)) >> 32;
}

/* Laplace CDF at n/16 steps from the mean, Q32; READING: the halving
 * truncates. */
static uint64_t cdf16(const uint64_t *P, int64_t n) {
  if (n < 0) return P[-n] >> 1;
  return (1ull << 32) - (P[n] >> 1);
}

/* Q32 masses of the 256 symbols for scale bin `bin` (grid `sub`) and mean
 * fraction f/16 (f = 0 for KV).  Symbol i < 255 is the residual s = i - 127,
 * the cell [s - 1/2, s + 1/2) relative to a mean at f/16; the escape symbol
 * takes both tails beyond |s| = 127.  The masses add up to exactly 2^32. */
void or_masses(uint32_t bin, uint32_t sub, uint32_t f, uint64_t *m) {
  uint64_t P[CHAIN_LEN];
  or_power_chain(or_tau_q(or_beta_q(bin, sub)), P);
  for (int64_t i = 0; i < 255; i++) {
    int64_t s = i - RMAX;
    m[i] = cdf16(P, 16 * s + 8 - (int64_t)f) - cdf16(P, 16 * s - 8 - (int64_t)f);
  }
  m[255] = cdf16(P, -16 * RMAX - 8 - (int64_t)f) +
           ((1ull << 32) - cdf16(P, 16 * RMAX + 8 - (int64_t)f));
}

/* Frequencies summing to 4096 with a floor of 1: fr_i = 1 + floor(m_i*3840/2^32);
 * READING (minimum frequency 1, deficit shared by largest remainder): the
 * remaining 4096 - sum fr units go one each to the symbols with the largest
 * remainders (m_i*3840 mod 2^32), ties to the lower symbol index. */
void or_build_table(uint32_t bin, uint32_t sub, uint32_t f, uint16_t *freq, uint16_t *cum) {
  uint64_t m[NSYM], rem[NSYM];
  uint32_t fr[NSYM], total = 0;
  or_masses(bin, sub, f, m);
  for (uint32_t i = 0; i < NSYM; i++) {
    uint64_t scaled = m[i] * (uint64_t)(PROB_SCALE - NSYM);
    fr[i] = 1u + (uint32_t)(scaled >> 32);
    rem[i] = scaled & 0xFFFFFFFFull;
    total += fr[i];
  }
  uint32_t deficit = PROB_SCALE - total;
  for (uint32_t k = 0; k < deficit; k++) {       /* pick the k-th largest */
    uint32_t best = NSYM;
    for (uint32_t i = 0; i < NSYM; i++) {
      if (rem[i] == UINT64_MAX) continue;         /* already given one   */
      if (best == NSYM || rem[i] > rem[best]) best = i;
    }
    fr[best] += 1;
    rem[best] = UINT64_MAX;
  }
  uint32_t c = 0;
  for (uint32_t i = 0; i < NSYM; i++) {
    freq[i] = (uint16_t)fr[i];
    cum[i] = (uint16_t)c;
    c += fr[i];
  }
  cum[NSYM] = (uint16_t)c;   /* 4096 does not fit 12 bits but fits u16 */
}

/* All tables of a stream: KV table b is scale bin b (f = 0); COEF table
 * 16*b + f is scale bin b with mean fraction f/16. */
int or_build_tables(const or_params *p, uint16_t *freq_all, uint16_t *cum_all) {
  if (or_check_params(p) != OR_OK) return OR_ERR_ARG;
  uint32_t nt = or_num_tables(p), sub = or_sub_bins(p);
  for (uint32_t t = 0; t < nt; t++) {
    uint32_t bin = p->dtype == OR_COEF ? t / 16u : t;
    uint32_t f = p->dtype == OR_COEF ? t % 16u : 0u;
    or_build_table(bin, sub, f, freq_all + (uint64_t)t * NSYM, cum_all + (uint64_t)t * (NSYM + 1));
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* O2 + O5: position -> (table, symbol, raw residual).                        */
/* ------------------------------------------------------------------------ */

typedef struct {
  int present;     /* 0: position carries no symbol (switched-off component) */
  uint32_t table;
  uint32_t sym;    /* 0..254 = residual + 127, 255 = escape                  */
  uint32_t raw;    /* escape only: residual mod 2^(8*raw_bytes)              */
} or_sym;

/* READING (mean quantisation for COEF tables): mu_q = floor(16 mu + 1/2) in
 * fp32; integer part m = floor(mu_q / 16), fraction f = mu_q - 16 m.  Means
 * whose |16 mu + 1/2| is not below 2^26 (or NaN) count as 0. */
static void coef_mean(float mu, int32_t *m, uint32_t *f) {
  float t = mu * 16.0f;
  t = t + 0.5f;
  int32_t mq = 0;
  if (fabsf(t) < 67108864.0f) mq = (int32_t)floorf(t);
  int32_t mm = mq >= 0 ? mq / 16 : -((-mq + 15) / 16);
  *m = mm;
  *f = (uint32_t)(mq - 16 * mm);
}

/* residual -> symbol; |r| > 127 escapes with the residual mod 2^width */
static void residual_symbol(int64_t r, uint32_t width, or_sym *o) {
  if (r >= -RMAX && r <= RMAX) {
    o->sym = (uint32_t)(r + RMAX);
    o->raw = 0;
  } else {
    o->sym = ESC;
    o->raw = (uint32_t)((uint64_t)r & ((1ull << width) - 1ull));
  }
}

/* `tgt`, `prd` point at the data of global position `gpos` of slice `slice`
 * (i.e. already offset); `bins` covers all channels. */
static void position_symbol(const or_params *p, uint64_t slice, uint64_t pos_in_slice,
                            const void *tgt, const void *prd, uint64_t idx,
                            const uint8_t *bins, or_sym *o) {
  o->present = 1;
  if (p->dtype == OR_COEF) {
    uint32_t c = (uint32_t)(pos_in_slice % p->n_coef);
    if (bins[c] == 0xFF) { o->present = 0; return; }
    int32_t m; uint32_t f;
    coef_mean(((const float *)prd)[idx], &m, &f);
    int64_t q = ((const int16_t *)tgt)[idx];
    o->table = 16u * bins[c] + f;
    residual_symbol(q - (int64_t)m, 16u, o);
    return;
  }
  uint32_t esz = elem_bytes(p), width = 8u * esz;
  uint64_t c = slice * p->head_dim + pos_in_slice % p->head_dim;
  uint32_t pb = load_bits(prd, idx, esz);
  o->table = p->model == 1u ? or_model1_table(bins[c], (pb >> 3) & 15u) : bins[c];
  int64_t r = (int64_t)or_ordinal(load_bits(tgt, idx, esz), width) - (int64_t)or_ordinal(pb, width);
  residual_symbol(r, width, o);
}

/* ------------------------------------------------------------------------ */
/* O6/O7: rANS.  [DCKV] how it differs names rANS as the entropy coder       */
/* (the [SKV] page says "arithmetic coder"; rANS belongs to that family).     */
/* State x in [2^16, 2^32), 16-bit renormalisation words, probabilities       */
/* fr/2^prob_bits.  READING for the stream layout: a lane's words are         */
/*   [x_final >> 16, x_final & 0xFFFF, renormalisation words, last pushed     */
/*   first]                                                                   */
/* so that a decoder reads them front to back.                                */
/* ------------------------------------------------------------------------ */

typedef struct {
  uint64_t x;
  uint16_t *buf;   /* pushed words, in push order */
  uint64_t n, cap;
  int overflow;
} or_enc;

static void enc_step(or_enc *e, uint32_t prob_bits, uint32_t fr, uint32_t cum) {
  uint64_t x_max = (((uint64_t)RANS_L >> prob_bits) << 16) * fr;
  if (e->x >= x_max) {
    if (e->n < e->cap) e->buf[e->n] = (uint16_t)(e->x & 0xFFFF);
    else e->overflow = 1;
    e->n++;
    e->x >>= 16;
  }
  e->x = (e->x / fr) * ((uint64_t)1 << prob_bits) + (e->x % fr) + cum;
}

/* write [state, pushed words reversed] to out; returns words written */
static uint64_t enc_flush(const or_enc *e, uint16_t *out) {
  out[0] = (uint16_t)(e->x >> 16);
  out[1] = (uint16_t)(e->x & 0xFFFF);
  for (uint64_t k = 0; k < e->n; k++) out[2 + k] = e->buf[e->n - 1 - k];
  return e->n + 2;
}

typedef struct {
  uint64_t x;
  const uint16_t *w;
  uint64_t pos, n;
  int corrupt;
} or_dec;

static void dec_init(or_dec *d, const uint16_t *w, uint64_t n) {
  d->w = w; d->n = n; d->corrupt = 0;
  if (n < 2) { d->corrupt = 1; d->x = RANS_L; d->pos = n; return; }
  d->x = ((uint64_t)w[0] << 16) | w[1];
  d->pos = 2;
  if (d->x < RANS_L) d->corrupt = 1;
}

/* one decoding step given the symbol's (fr, cum) (already identified) */
static void dec_advance(or_dec *d, uint32_t prob_bits, uint32_t fr, uint32_t cum) {
  uint64_t mask = ((uint64_t)1 << prob_bits) - 1;
  uint64_t slot = d->x & mask;
  d->x = fr * (d->x >> prob_bits) + slot - cum;
  if (d->x < RANS_L) {
    uint64_t word = 0;
    if (d->pos < d->n) word = d->w[d->pos];
    else d->corrupt = 1;
    d->pos++;
    d->x = (d->x << 16) | word;
  }
}

/* the symbol whose cell holds the current slot: cum[i] <= slot < cum[i+1] */
static uint32_t dec_find(const or_dec *d, uint32_t prob_bits, const uint32_t *cum, uint32_t nsym) {
  uint64_t slot = d->x & (((uint64_t)1 << prob_bits) - 1);
  uint32_t i = 0;
  while (i + 1 < nsym && cum[i + 1] <= slot) i++;
  return i;
}

/* same search over a 16-bit cumulative table (the stream tables) */
static uint32_t dec_find16(const or_dec *d, const uint16_t *cum) {
  uint64_t slot = d->x & (PROB_SCALE - 1);
  uint32_t i = 0;
  while (i + 1 < NSYM && cum[i + 1] <= slot) i++;
  return i;
}

/* Generic coder over an arbitrary table, for hand-worked examples and brute
 * force: encodes syms[0..n) (decode order) into one lane stream. */
int or_rans_encode(uint32_t prob_bits, const uint32_t *freq, const uint32_t *cum,
                   const uint32_t *syms, uint64_t n, uint16_t *out, uint64_t cap,
                   uint64_t *n_out) {
  uint16_t *pushed = (uint16_t *)malloc((n + 1) * sizeof(uint16_t));
  if (!pushed) return OR_ERR_ARG;
  or_enc e = {RANS_L, pushed, 0, n + 1, 0};
  for (uint64_t k = n; k-- > 0;) enc_step(&e, prob_bits, freq[syms[k]], cum[syms[k]]);
  int st = OR_OK;
  if (e.overflow || e.n + 2 > cap) st = OR_ERR_CAPACITY;
  else *n_out = enc_flush(&e, out);
  free(pushed);
  return st;
}

int or_rans_decode(uint32_t prob_bits, const uint32_t *freq, const uint32_t *cum, uint32_t nsym,
                   const uint16_t *words, uint64_t n_words, uint64_t n, uint32_t *syms) {
  or_dec d;
  dec_init(&d, words, n_words);
  for (uint64_t k = 0; k < n; k++) {
    uint32_t i = dec_find(&d, prob_bits, cum, nsym);
    syms[k] = i;
    dec_advance(&d, prob_bits, freq[i], cum[i]);
  }
  if (d.corrupt || d.x != RANS_L || d.pos != d.n) return OR_ERR_CORRUPT;
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Chunks and lanes.  A chunk is 32*K consecutive positions of one slice (the */
/* last chunk of a slice may be short).  READING (interleaving): positions    */
/* come in groups of G (16 for FP8, 8 for 16-bit data, i.e. 16 bytes) and     */
/* lane l of a chunk owns the groups whose chunk-local index is l mod 32.     */
/* Each lane is an independent rANS stream; lanes are stored in global lane   */
/* order (chunk*32 + l) and lane_offsets[g] is the byte offset of lane g.     */
/* ------------------------------------------------------------------------ */

typedef struct {
  uint64_t slice, first;   /* slice index, first position within the slice */
  uint64_t n_pos;          /* positions in this chunk                       */
} or_chunk;

static or_chunk chunk_info(const or_params *p, uint64_t chunk) {
  or_chunk ch;
  uint64_t cps = or_chunks_per_slice(p), cs = (uint64_t)LANES * p->lane_syms;
  uint64_t sp = or_slice_positions(p);
  ch.slice = chunk / cps;
  ch.first = (chunk % cps) * cs;
  ch.n_pos = sp - ch.first < cs ? sp - ch.first : cs;
  return ch;
}

/* chunk-local positions of lane l, ascending; returns the count */
static uint64_t lane_positions(const or_params *p, uint64_t n_pos, uint32_t l, uint64_t *pos) {
  uint64_t G = or_group(p), n = 0;
  for (uint64_t g = l; g * G < n_pos; g += LANES)
    for (uint64_t e = 0; e < G && g * G + e < n_pos; e++) pos[n++] = g * G + e;
  return n;
}

/* Encode one chunk.  tgt/prd point at the chunk's first position (chunk data
 * is contiguous).  Writes the 32 lane streams back to back into out (words),
 * lane_words[l] = words of lane l.  Returns OR_OK or OR_ERR_CAPACITY. */
int or_encode_chunk(const or_params *p, uint64_t chunk, const uint16_t *freq_all,
                    const uint16_t *cum_all, const uint8_t *bins, const void *tgt,
                    const void *prd, uint16_t *out, uint64_t cap_words, uint32_t *lane_words) {
  if (or_check_params(p) != OR_OK || p->lane_syms > 65536) return OR_ERR_ARG;
  or_chunk ch = chunk_info(p, chunk);
  uint32_t rb = raw_bytes(p);
  uint64_t used = 0, max_pushed = (uint64_t)p->lane_syms * (1 + rb);
  uint64_t *pos_buf = (uint64_t *)malloc(p->lane_syms * sizeof(uint64_t));
  uint16_t *pushed = (uint16_t *)malloc(max_pushed * sizeof(uint16_t));
  int status = OR_OK;
  if (!pos_buf || !pushed) status = OR_ERR_ARG;
  for (uint32_t l = 0; l < LANES && status == OR_OK; l++) {
    uint64_t n = lane_positions(p, ch.n_pos, l, pos_buf);
    or_enc e = {RANS_L, pushed, 0, max_pushed, 0};
    for (uint64_t k = n; k-- > 0;) {                       /* reverse pass */
      or_sym s;
      position_symbol(p, ch.slice, ch.first + pos_buf[k], tgt, prd, pos_buf[k], bins, &s);
      if (!s.present) continue;
      if (s.sym == ESC) {
        /* raw residual bytes as uniform steps (fr 16 = 4096/256), coded
         * before the escape so that the decoder meets the escape first and
         * then reads the raw bytes high byte first */
        for (uint32_t b = 0; b < rb; b++) enc_step(&e, PROB_BITS, 16u, 16u * ((s.raw >> (8u * b)) & 0xFFu));
      }
      const uint16_t *fr = freq_all + (uint64_t)s.table * NSYM;
      const uint16_t *cm = cum_all + (uint64_t)s.table * (NSYM + 1);
      enc_step(&e, PROB_BITS, fr[s.sym], cm[s.sym]);
    }
    if (e.overflow || used + e.n + 2 > cap_words) { status = OR_ERR_CAPACITY; break; }
    lane_words[l] = (uint32_t)enc_flush(&e, out + used);
    used += lane_words[l];
  }
  free(pos_buf);
  free(pushed);
  return status;
}

static void store_bits(void *base, uint64_t idx, uint32_t esz, uint32_t v) {
  if (esz == 1) ((uint8_t *)base)[idx] = (uint8_t)v;
  else ((uint16_t *)base)[idx] = (uint16_t)v;
}

/* Decode one chunk: words = the chunk's 32 lane streams back to back,
 * lane_words[l] their lengths; prd at the chunk's first position; writes the
 * target at tgt_out (chunk-relative).  Switched-off COEF components decode
 * to 0 ([DCKV] how it works: switched off in reconstruction too). */
int or_decode_chunk(const or_params *p, uint64_t chunk, const uint16_t *freq_all,
                    const uint16_t *cum_all, const uint8_t *bins, const uint16_t *words,
                    const uint32_t *lane_words, const void *prd, void *tgt_out) {
  if (or_check_params(p) != OR_OK || p->lane_syms > 65536) return OR_ERR_ARG;
  or_chunk ch = chunk_info(p, chunk);
  uint32_t esz = elem_bytes(p), width = 8u * esz, rb = raw_bytes(p);
  uint64_t start = 0;
  int status = OR_OK;
  uint64_t *pos_buf = (uint64_t *)malloc(p->lane_syms * sizeof(uint64_t));
  if (!pos_buf) return OR_ERR_ARG;
  for (uint32_t l = 0; l < LANES; l++) {
    uint64_t n = lane_positions(p, ch.n_pos, l, pos_buf);
    or_dec d;
    dec_init(&d, words + start, lane_words[l]);
    for (uint64_t k = 0; k < n; k++) {
      uint64_t idx = pos_buf[k], pis = ch.first + idx;
      uint32_t table;
      int32_t m = 0;
      if (p->dtype == OR_COEF) {
        uint32_t c = (uint32_t)(pis % p->n_coef), f;
        if (bins[c] == 0xFF) { ((int16_t *)tgt_out)[idx] = 0; continue; }
        coef_mean(((const float *)prd)[idx], &m, &f);
        table = 16u * bins[c] + f;
      } else {
        uint32_t b = bins[ch.slice * p->head_dim + pis % p->head_dim];
        table = p->model == 1u ? or_model1_table(b, (load_bits(prd, idx, esz) >> 3) & 15u) : b;
      }
      const uint16_t *fr = freq_all + (uint64_t)table * NSYM;
      const uint16_t *cm = cum_all + (uint64_t)table * (NSYM + 1);
      uint32_t sym = dec_find16(&d, cm);
      dec_advance(&d, PROB_BITS, fr[sym], cm[sym]);
      uint64_t r;                         /* residual mod 2^width */
      if (sym == ESC) {
        uint32_t raw = 0;
        for (uint32_t b = rb; b-- > 0;) {     /* high byte first */
          uint32_t v = (uint32_t)((d.x & (PROB_SCALE - 1)) >> 4);
          dec_advance(&d, PROB_BITS, 16u, 16u * v);
          raw |= v << (8u * b);
        }
        r = raw;
      } else {
        r = (uint64_t)((int64_t)sym - RMAX);
      }
      if (p->dtype == OR_COEF) {
        ((int16_t *)tgt_out)[idx] = (int16_t)(uint16_t)(((uint64_t)(int64_t)m + r) & 0xFFFFu);
      } else {
        uint32_t up = or_ordinal(load_bits(prd, idx, esz), width);
        uint32_t ut = (uint32_t)((up + r) & ((1ull << width) - 1ull));
        store_bits(tgt_out, idx, esz, or_ordinal_inv(ut, width));
      }
    }
    if (d.corrupt || d.x != RANS_L || d.pos != d.n) status = OR_ERR_CORRUPT;
    start += lane_words[l];
  }
  free(pos_buf);
  return status;
}

/* ------------------------------------------------------------------------ */
/* Whole streams: chunks in order, lanes concatenated, byte offsets.          */
/* ------------------------------------------------------------------------ */

static uint64_t chunk_first_global(const or_params *p, uint64_t chunk) {
  or_chunk ch = chunk_info(p, chunk);
  return ch.slice * or_slice_positions(p) + ch.first;
}

int or_encode(const or_params *p, const uint16_t *freq_all, const uint16_t *cum_all,
              const uint8_t *bins, const void *target, const void *pred, uint8_t *bitstream,
              uint64_t cap_bytes, uint64_t *lane_offsets, uint64_t *total_bytes) {
  if (or_check_params(p) != OR_OK) return OR_ERR_ARG;
  uint32_t esz = elem_bytes(p), lw[LANES];
  uint32_t psz = p->dtype == OR_COEF ? 4u : esz;        /* mu is fp32 */
  uint64_t nch = or_num_chunks(p), off = 0;
  for (uint64_t c = 0; c < nch; c++) {
    uint64_t g0 = chunk_first_global(p, c);
    uint64_t cap_words = off / 2 <= cap_bytes / 2 ? cap_bytes / 2 - off / 2 : 0;
    int st = or_encode_chunk(p, c, freq_all, cum_all, bins,
                             (const uint8_t *)target + g0 * esz,
                             (const uint8_t *)pred + g0 * psz,
                             (uint16_t *)(bitstream + off), cap_words, lw);
    if (st != OR_OK) return st;
    for (uint32_t l = 0; l < LANES; l++) {
      lane_offsets[c * LANES + l] = off;
      off += 2ull * lw[l];
    }
  }
  lane_offsets[nch * LANES] = off;
  *total_bytes = off;
  return OR_OK;
}

int or_decode(const or_params *p, const uint16_t *freq_all, const uint16_t *cum_all,
              const uint8_t *bins, const uint8_t *bitstream, uint64_t n_bytes,
              const uint64_t *lane_offsets, const void *pred, void *target_out) {
  if (or_check_params(p) != OR_OK) return OR_ERR_ARG;
  uint32_t esz = elem_bytes(p), lw[LANES];
  uint32_t psz = p->dtype == OR_COEF ? 4u : esz;
  uint64_t nch = or_num_chunks(p);
  int status = OR_OK;
  if (lane_offsets[0] != 0 || lane_offsets[nch * LANES] != n_bytes) return OR_ERR_CORRUPT;
  for (uint64_t c = 0; c < nch; c++) {
    uint64_t g0 = chunk_first_global(p, c);
    for (uint32_t l = 0; l < LANES; l++) {
      uint64_t a = lane_offsets[c * LANES + l], b = lane_offsets[c * LANES + l + 1];
      if (b < a || (a & 1) || (b & 1) || b > n_bytes) return OR_ERR_CORRUPT;
      lw[l] = (uint32_t)((b - a) / 2);
    }
    int st = or_decode_chunk(p, c, freq_all, cum_all, bins,
                             (const uint16_t *)(bitstream + lane_offsets[c * LANES]), lw,
                             (const uint8_t *)pred + g0 * psz,
                             (uint8_t *)target_out + g0 * esz);
    if (st != OR_OK) status = st;
  }
  return status;
}

/* ------------------------------------------------------------------------ */
/* O8: Shannon reference for the coded length: sum over coding steps of       */
/* -log2(fr/4096), raw bytes counting exactly 8 bits.  Long double.          */
/* ------------------------------------------------------------------------ */

double or_shannon_bits(const or_params *p, const uint16_t *freq_all, const uint8_t *bins,
                       const void *target, const void *pred) {
  if (or_check_params(p) != OR_OK) return -1.0;
  uint32_t esz = elem_bytes(p), rb = raw_bytes(p);
  uint32_t psz = p->dtype == OR_COEF ? 4u : esz;
  long double bits = 0.0L;
  uint64_t sp = or_slice_positions(p);
  for (uint64_t s = 0; s < or_num_slices(p); s++) {
    const uint8_t *tg = (const uint8_t *)target + s * sp * esz;
    const uint8_t *pr = (const uint8_t *)pred + s * sp * psz;
    for (uint64_t i = 0; i < sp; i++) {
      or_sym o;
      position_symbol(p, s, i, tg, pr, i, bins, &o);
      if (!o.present) continue;
      uint32_t fr = freq_all[(uint64_t)o.table * NSYM + o.sym];
      bits += -log2l((long double)fr / (long double)PROB_SCALE);
      if (o.sym == ESC) bits += 8.0L * rb;
    }
  }
  return (double)bits;
}

/* symbols of every position, for tests: table id, symbol (-1 if absent) */
int or_symbols(const or_params *p, const uint8_t *bins, const void *target, const void *pred,
               uint32_t *table_out, int32_t *sym_out, uint32_t *raw_out) {
  if (or_check_params(p) != OR_OK) return OR_ERR_ARG;
  uint32_t esz = elem_bytes(p);
  uint32_t psz = p->dtype == OR_COEF ? 4u : esz;
  uint64_t sp = or_slice_positions(p), k = 0;
  for (uint64_t s = 0; s < or_num_slices(p); s++) {
    const uint8_t *tg = (const uint8_t *)target + s * sp * esz;
    const uint8_t *pr = (const uint8_t *)pred + s * sp * psz;
    for (uint64_t i = 0; i < sp; i++, k++) {
      or_sym o;
      position_symbol(p, s, i, tg, pr, i, bins, &o);
      table_out[k] = o.present ? o.table : 0;
      sym_out[k] = o.present ? (int32_t)o.sym : -1;
      raw_out[k] = o.raw;
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Checkerboard context ([DCKV] how it differs): the coefficient rows are     */
/* split by token parity; even rows are coded with the token-conditioned      */
/* means alone, odd rows with means that also depend on the decoded rows on   */
/* both sides through a rank-R linear map, so each parity decodes in one      */
/* token-parallel pass.  READING (the page's map is learned; none is given):  */
/* an integer map with factor matrices V [R][C], U [C][R] (int8 storage,      */
/* entries used clamped to [-8, 8]: 4-bit weights), and                       */
/*   x   = clamp(q_even[t] + q_even[t+1], -127, 127)  (missing row -> 0)      */
/*   g_r = clamp(floor((V x)_r / 2^s1), -127, 127)                            */
/*   k_c = floor((U g)_c / 2^s2)               (context shift, 1/16 steps)    */
/*   mu' = clamp(mu_q + k, +-(2^23 - 1)) / 16  (mu_q: the mean quantisation    */
/*         of the token-conditioned mean, as for every coefficient)           */
/* mu' is exact in fp32 and quantises back to mu_q + k, so the odd rows are   */
/* an ordinary coefficient stream whose means are mu'.                        */
/* ------------------------------------------------------------------------ */
static int64_t floor_shift(int64_t v, uint32_t s) {
  int64_t d = (int64_t)1 << s;
  return v >= 0 ? v / d : -((-v + d - 1) / d);
}
static int64_t clamp64(int64_t v, int64_t lo, int64_t hi) { return v < lo ? lo : (v > hi ? hi : v); }

int or_ctx_means(uint32_t C, uint32_t R, const int8_t *V, const int8_t *U, uint32_t s1, uint32_t s2,
                 const int16_t *q_even, uint64_t n_even, const float *mu_odd, uint64_t n_odd, float *out) {
  if (C == 0 || R == 0 || s1 > 30 || s2 > 30 || n_odd > n_even) return OR_ERR_ARG;
  int64_t *x = (int64_t *)malloc(C * sizeof(int64_t));
  int64_t *g = (int64_t *)malloc(R * sizeof(int64_t));
  if (!x || !g) { free(x); free(g); return OR_ERR_ARG; }
  for (uint64_t t = 0; t < n_odd; t++) {
    for (uint32_t c = 0; c < C; c++) {
      int64_t a = q_even[t * C + c], b = t + 1 < n_even ? q_even[(t + 1) * C + c] : 0;
      x[c] = clamp64(a + b, -127, 127);
    }
    for (uint32_t r = 0; r < R; r++) {
      int64_t h = 0;
      for (uint32_t c = 0; c < C; c++) h += clamp64(V[(uint64_t)r * C + c], -8, 8) * x[c];
      g[r] = clamp64(floor_shift(h, s1), -127, 127);
    }
    for (uint32_t c = 0; c < C; c++) {
      int64_t y = 0;
      for (uint32_t r = 0; r < R; r++) y += clamp64(U[(uint64_t)c * R + r], -8, 8) * g[r];
      int32_t m; uint32_t f;
      coef_mean(mu_odd[t * C + c], &m, &f);
      int64_t mq = 16 * (int64_t)m + f;
      int64_t mq2 = clamp64(mq + floor_shift(y, s2), -8388607, 8388607);
      out[t * C + c] = (float)mq2 / 16.0f;
    }
  }
  free(x); free(g);
  return OR_OK;
}
