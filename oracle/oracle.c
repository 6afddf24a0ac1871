/*
 * CPU oracle for the heterogeneous-batch LoRA delta -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * this file.  It shares no source, header, table or helper with the CUDA
 * library; it is deliberately slow and written to be checked by eye.
 *
 * What it computes ("S-LoRA: Serving Thousands of Concurrent LoRA Adapters",
 * abstract and method list of the nubint.ai review: every token of one batch
 * carries its own adapter, adapters of different ranks are batched together,
 * and the adapter weights sit in non-contiguous pages of one pool shared with
 * the KV cache; dongaigc.com summary, section 2 "heterogeneous batching"):
 *
 *     y_out[i, n] = round( y_in[i, n] + s * s_a * sum_k ( sum_c x[i, c] A_a[c, k] ) B_a[k, n] )
 *
 * where s_a is adapter a's own scale (LoRA's alpha / r; 1 when no per-adapter
 * scales are given), for every token i whose adapter a = a(i) is >= 0; tokens with a(i) = -1 are
 * copied unchanged.  Only -1 means "no adapter": a token naming any other id
 * outside [0, num_adapters), or an adapter of rank 0, is copied unchanged too
 * and makes the call return -1.  All arithmetic is fp64 on the exact values of the 16-bit
 * inputs, and round() is one IEEE round-to-nearest-even into the storage
 * type.  A and B are never dense here: every element is fetched through the
 * adapter's page table, exactly as the pages describe the non-contiguous
 * layout.
 *
 * Page-table layout of one adapter of rank r (the order its pages are listed):
 *   for each projection q in order:
 *     A rows k = 0..r-1, each split into ceil(h_in_q / H) page chunks,
 *     then B rows k = 0..r-1, each split into ceil(h_out_q / H) page chunks.
 * Row k of A holds column k of the H_in x r matrix A; row k of B holds row k
 * of the r x H_out matrix B.  Element c of a row sits in chunk c / H at
 * offset c % H of that chunk's page.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* ---- 16-bit float decoding (IEEE 754 binary16 and bfloat16) ------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);                    /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = (m == 0) ? INFINITY : NAN;
  else
    v = ldexp((double)(1024 + m), e - 25);        /* (1 + m/2^10) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int m = b & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)m, -133);                   /* subnormal: m * 2^-133 */
  else if (e == 255)
    v = (m == 0) ? INFINITY : NAN;
  else
    v = ldexp((double)(128 + m), e - 134);        /* (1 + m/2^7) * 2^(e-127) */
  return sign ? -v : v;
}

/* ---- round-to-nearest-even encoding ------------------------------------ */

/*
 * Generic encoder for a binary format with `mbits` fraction bits, exponent
 * bias `bias` and all-ones exponent field `emax_field`.  The magnitude is
 * expressed as an integer multiple of the quantum of its binade, and that
 * integer is rounded half-to-even with rint() (the C default rounding mode
 * is round-to-nearest-even).  Dividing by a power of two is exact in fp64,
 * so the only rounding is the one being defined.
 */
static uint16_t encode_rne(double v, int mbits, int bias, int emax_field) {
  uint16_t sign = (signbit(v) ? 1u : 0u) << 15;
  double a = fabs(v);
  if (isnan(v)) return (uint16_t)(sign | (emax_field << mbits) | (1u << (mbits - 1)));
  if (isinf(v)) return (uint16_t)(sign | (emax_field << mbits));
  int emin = 1 - bias;                            /* exponent of the smallest normal */
  int e;
  if (a == 0.0) return sign;
  frexp(a, &e);                                   /* a in [2^(e-1), 2^e) */
  int unb = e - 1;                                /* unbiased exponent of a */
  if (unb < emin) {
    /* subnormal range: quantum 2^(emin - mbits); n = 2^mbits encodes the
     * smallest normal, which is exactly the bit pattern n. */
    double n = rint(ldexp(a, mbits - emin));
    return (uint16_t)(sign | (uint16_t)n);
  }
  double n = rint(ldexp(a, mbits - unb));         /* in [2^mbits, 2^(mbits+1)] */
  long field = (long)(unb + bias);
  long bits = (field << mbits) + ((long)n - (1L << mbits));  /* n = 2^(mbits+1) carries */
  if ((bits >> mbits) >= emax_field) return (uint16_t)(sign | (emax_field << mbits));
  return (uint16_t)(sign | (uint16_t)bits);
}

uint16_t oracle_f64_to_f16(double v) { return encode_rne(v, 10, 15, 31); }
uint16_t oracle_f64_to_bf16(double v) { return encode_rne(v, 7, 127, 255); }

static double decode(uint16_t bits, int dtype) {
  return dtype == ORACLE_F16 ? oracle_f16_to_f64(bits) : oracle_bf16_to_f64(bits);
}
static uint16_t encode(double v, int dtype) {
  return dtype == ORACLE_F16 ? oracle_f64_to_f16(v) : oracle_f64_to_bf16(v);
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* Address of element c of a page-resident row whose first page-table entry
 * is page_table[entry].  `page_slot` maps a pool page to the row of `pool`
 * that holds its contents (NULL: the identity, i.e. `pool` is the whole
 * pool); the oracle's tests keep only the pages that hold adapter rows. */
static const uint16_t* row_elem(const uint16_t* pool, const int64_t* page_slot, int32_t H,
                                const int32_t* page_table, int64_t entry, int64_t c) {
  int64_t page = page_table[entry + c / H];
  int64_t slot = page_slot ? page_slot[page] : page;
  return pool + slot * (int64_t)H + (c % H);
}

/*
 * The delta for one projection `p`, over the tokens listed in `tokens`
 * (all T tokens when `tokens` is NULL, n_tokens ignored then).
 *   pool        16-bit page contents (see row_elem for page_slot)
 *   page_table  concatenated page tables; adapter a's entries start at pt_off[a]
 *   rank        rank of each adapter (0 = not resident)
 *   proj_in/out dims of every projection (the layout depends on all of them)
 *   x           T rows of proj_in[p] elements, row stride ldx
 *   y_in        T rows of proj_out[p] elements, row stride ldy
 *   y_out       receives round(y_in + s * delta) in the same layout
 *   y_exact     optional: the unrounded fp64 value y_in + s * delta
 *   v_out       optional: the fp64 shrink result, row stride v_ld
 * Returns 0, or -1 when a token names an id other than -1 outside
 * [0, num_adapters) or an adapter of rank 0 (its row is copied unchanged).
 */
int oracle_lora_apply(const uint16_t* pool, const int64_t* page_slot, int32_t H, int32_t dtype,
                      const int32_t* page_table, const int64_t* pt_off, const int32_t* rank,
                      int32_t num_adapters, int32_t num_proj, const int32_t* proj_in,
                      const int32_t* proj_out, int32_t p, const int32_t* token_adapter, int32_t T,
                      const int32_t* tokens, int32_t n_tokens, const uint16_t* x, int64_t ldx,
                      const uint16_t* y_in, int64_t ldy, double s, const double* adapter_scale, uint16_t* y_out,
                      double* y_exact, double* v_out, int64_t v_ld, int32_t num_threads) {
  int64_t rows_before = 0;               /* page chunks of one rank index in projections < p */
  for (int q = 0; q < p; q++) rows_before += ceil_div(proj_in[q], H) + ceil_div(proj_out[q], H);
  const int64_t ppi = ceil_div(proj_in[p], H), ppo = ceil_div(proj_out[p], H);
  const int64_t hin = proj_in[p], hout = proj_out[p];
  const int32_t n = tokens ? n_tokens : T;
  int bad = 0;
  (void)num_proj;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads > 0 ? num_threads : 1) reduction(| : bad)
#endif
  for (int32_t j = 0; j < n; j++) {
    const int32_t i = tokens ? tokens[j] : j;
    const int32_t a = token_adapter[i];
    const uint16_t* yi = y_in + (int64_t)i * ldy;
    uint16_t* yo = y_out + (int64_t)i * ldy;
    /* Only -1 means "base model only".  Any other id outside
     * [0, num_adapters), or an adapter of rank 0 (not resident), is an error:
     * the token is flagged and, like a base-only token, left unchanged. */
    const int is_bad = a != -1 && (a < 0 || a >= num_adapters || rank[a] <= 0 || rank[a] > 1024);
    if (a == -1 || is_bad) {
      for (int64_t c = 0; c < hout; c++) {
        yo[c] = yi[c];
        if (y_exact) y_exact[(int64_t)i * ldy + c] = decode(yi[c], dtype);
      }
      if (is_bad) bad = 1;
      continue;
    }
    const int64_t r = rank[a];
    const int64_t a_base = pt_off[a] + r * rows_before;     /* A rows of projection p */
    const int64_t b_base = a_base + r * ppi;                /* B rows follow the A rows */
    double v[1024];                                         /* r <= 1024 (checked above) */
    for (int64_t k = 0; k < r; k++) {                       /* shrink: v = x A */
      double acc = 0.0;
      for (int64_t c = 0; c < hin; c++) {
        double xc = decode(x[(int64_t)i * ldx + c], dtype);
        double akc = decode(*row_elem(pool, page_slot, H, page_table, a_base + k * ppi, c), dtype);
        acc += xc * akc;
      }
      v[k] = acc;
      if (v_out) v_out[(int64_t)i * v_ld + k] = acc;
    }
    for (int64_t c = 0; c < hout; c++) {                    /* expand: y += s v B */
      double acc = 0.0;
      for (int64_t k = 0; k < r; k++)
        acc += v[k] * decode(*row_elem(pool, page_slot, H, page_table, b_base + k * ppo, c), dtype);
      double y = decode(yi[c], dtype) + s * (adapter_scale ? adapter_scale[a] : 1.0) * acc;
      if (y_exact) y_exact[(int64_t)i * ldy + c] = y;
      yo[c] = encode(y, dtype);
    }
  }
  return bad ? -1 : 0;
}

/* Element-wise conversions over arrays (used by the tests' pins). */
void oracle_decode_array(const uint16_t* in, double* out, int64_t n, int32_t dtype) {
  for (int64_t i = 0; i < n; i++) out[i] = decode(in[i], dtype);
}
void oracle_encode_array(const double* in, uint16_t* out, int64_t n, int32_t dtype) {
  for (int64_t i = 0; i < n; i++) out[i] = encode(in[i], dtype);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
