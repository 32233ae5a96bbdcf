/*
 * mlora_oracle.c -- plain, slow fp64 CPU oracle for the gathered multi-LoRA delta.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline leg of the
 * bench may load this code. The CUDA library never includes, links or calls it, and it
 * includes nothing from the CUDA library: every definition below is local to this file.
 *
 * What it computes
 * ----------------
 * Punica (arXiv 2310.18547), section 3.4 "The SGMV Operator": the LoRA add-on x·A·B is
 * split into a shrink v = x·A (h1 -> r) and an expand y += v·B (r -> h2), with v starting
 * from zero. "Multi-LoRA Serving, in depth", section "Why a mixed batch needs special
 * kernels", gives the per-row specification with a slot per row (-1 = no adapter) and a
 * per-slot scale alpha/r applied to v·B. For every row i whose slot s is a valid adapter:
 *
 *     v[i][j]  = sum_{k < d_in} x[i][k] * A_s[k][j]                    j < rank[s]
 *     y'[i][n] = RNE( y[i][n] + scale[s] * sum_{j < rank[s]} v[i][j] * B_s[j][n] )
 *
 * SGMV (Punica section 3.4, segment boundaries s_0 = 0 <= ... <= s_n = M): the slot of row i
 * is the slot of the segment [off[t], off[t+1]) that contains i. BGMV (the "add_lora_bgmv"
 * semantics quoted in the zh-TW Punica digest, section 5.5): the slot of row i is
 * row_slot[i].
 *
 * Arithmetic: every bf16/fp16 input is decoded to fp64 exactly; sums run in fp64 in
 * increasing index order; y + delta is formed in fp64 and rounded ONCE to the I/O type by
 * round-to-nearest-even, written here from the IEEE-754 definition (no library conversion).
 *
 * Storage read by the oracle (the same pools the library reads):
 *   stacked pool  A^T [num_slots][num_layers][r_max][d_in]   (row j of A^T = column j of A;
 *                 Punica's LoraWeight.wa "[num_layers, r, in_features]", zh-TW digest 5.4)
 *                 B   [num_slots][num_layers][r_max][d_out]  (row-major B, LoraWeight.wb)
 *   paged pool    S-LoRA (arXiv 2311.03285) "Unified Paging": a page is one vector of
 *                 page_elems elements (one H-vector); A of rank R is R columns, B is R rows,
 *                 each a vector of d_in (A) or d_out (B) elements stored in pages. A vector
 *                 longer than a page (page_elems < d, e.g. the 13824-long rows of an MLP
 *                 projection in pages of hidden size 5120) spans ceil(d / page_elems) pages:
 *                 the page tables are [num_slots][num_layers][r_max][ceil(d / page_elems)],
 *                 and element k of a vector is element k % page_elems of the vector's
 *                 (k / page_elems)-th page. With page_elems >= d every vector is one page.
 *
 * Metadata the pages do not define (everything but slot -1) is reported with status bits
 * and the affected rows are left untouched:
 *   ORC_BAD_OFFSETS  SGMV offsets not 0 = off[0] <= ... <= off[n] = M; nothing is computed.
 *   ORC_BAD_SLOT     slot < -1 or slot >= num_slots.
 *   ORC_BAD_RANK     rank[s] outside [1, r_max].
 *   ORC_BAD_PAGE     a page id (of a vector j < rank[s]) outside [0, num_pages).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define ORC_DTYPE_BF16 0
#define ORC_DTYPE_FP16 1
#define ORC_POOL_STACKED 0
#define ORC_POOL_PAGED 1

#define ORC_BAD_OFFSETS 1
#define ORC_BAD_SLOT 2
#define ORC_BAD_RANK 4
#define ORC_BAD_PAGE 8

#define ORC_ERR_ARG (-1)

typedef struct {
  int32_t kind; /* ORC_POOL_STACKED or ORC_POOL_PAGED */
  int32_t dtype; /* ORC_DTYPE_BF16 or ORC_DTYPE_FP16 */
  int32_t num_slots, num_layers, r_max, d_in, d_out;
  const uint16_t *a_t; /* stacked A^T */
  const uint16_t *b; /* stacked B */
  const uint16_t *pages; /* paged: [num_pages][page_elems] */
  int32_t page_elems, num_pages;
  const int32_t *a_page_table; /* paged: [num_slots][num_layers][r_max][ceil(d_in / page_elems)] */
  const int32_t *b_page_table; /* paged: [num_slots][num_layers][r_max][ceil(d_out / page_elems)] */
  const int32_t *rank; /* [num_slots] */
  const float *scale; /* [num_slots] */
} orc_pool;

/* ---- IEEE-754 binary16 / bfloat16 <-> fp64, from the format definitions ---------------- */

typedef struct {
  int mant_bits; /* stored fraction bits */
  int exp_bits;
  int bias;
} orc_format;

static orc_format format_of(int dtype) {
  orc_format f;
  if (dtype == ORC_DTYPE_BF16) {
    f.mant_bits = 7;
    f.exp_bits = 8;
    f.bias = 127;
  } else {
    f.mant_bits = 10;
    f.exp_bits = 5;
    f.bias = 15;
  }
  return f;
}

/* Exact value of a bf16/fp16 bit pattern. */
double orc_decode(uint16_t bits, int dtype) {
  orc_format f = format_of(dtype);
  unsigned exp_all = (1u << f.exp_bits) - 1u;
  unsigned sign = (bits >> 15) & 1u;
  unsigned e = (bits >> f.mant_bits) & exp_all;
  unsigned m = bits & ((1u << f.mant_bits) - 1u);
  double mag;
  if (e == exp_all) {
    mag = (m == 0) ? INFINITY : NAN;
  } else if (e == 0) {
    /* subnormal: m * 2^(1 - bias - mant_bits) */
    mag = ldexp((double)m, 1 - f.bias - f.mant_bits);
  } else {
    mag = ldexp((double)((1u << f.mant_bits) | m), (int)e - f.bias - f.mant_bits);
  }
  return sign ? -mag : mag;
}

/* Round an fp64 value to the nearest bf16/fp16 value, ties to even, overflow to +-Inf,
 * gradual underflow to subnormals (and to signed zero). NaN maps to the canonical quiet NaN. */
uint16_t orc_round(double v, int dtype) {
  orc_format f = format_of(dtype);
  unsigned exp_all = (1u << f.exp_bits) - 1u;
  uint16_t sign = signbit(v) ? (uint16_t)0x8000u : (uint16_t)0;
  int emin = 1 - f.bias; /* exponent of the smallest normal */
  int emax = (int)exp_all - 1 - f.bias; /* exponent of the largest finite */
  if (isnan(v)) return (uint16_t)(0x7FFFu & ((exp_all << f.mant_bits) | (1u << (f.mant_bits - 1))));
  double a = fabs(v);
  if (isinf(a)) return (uint16_t)(sign | (exp_all << f.mant_bits));
  if (a == 0.0) return sign;

  int e2;
  (void)frexp(a, &e2); /* a = frac * 2^e2, frac in [0.5, 1) */
  int E = e2 - 1; /* a in [2^E, 2^(E+1)) */
  if (E < emin) E = emin; /* below the normal range the spacing stays 2^(emin - mant_bits) */
  double quantum = ldexp(1.0, E - f.mant_bits); /* distance between neighbours at this scale */
  double q = a / quantum; /* exact: division by a power of two */
  double fl = floor(q);
  double rem = q - fl; /* exact: q has few integer bits */
  if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
  double r = fl * quantum; /* the rounded magnitude */

  if (r >= ldexp(1.0, emax + 1)) return (uint16_t)(sign | (exp_all << f.mant_bits));
  if (r == 0.0) return sign;

  unsigned field_e, field_m;
  int er;
  (void)frexp(r, &er);
  int Er = er - 1;
  if (Er < emin) {
    field_e = 0;
    field_m = (unsigned)(r / ldexp(1.0, emin - f.mant_bits));
  } else {
    field_e = (unsigned)(Er + f.bias);
    field_m = (unsigned)((r / ldexp(1.0, Er) - 1.0) * ldexp(1.0, f.mant_bits));
  }
  return (uint16_t)(sign | (field_e << f.mant_bits) | field_m);
}

/* ---- element access -------------------------------------------------------------------- */

static size_t table_index(const orc_pool *p, int s, int layer, int j) {
  return ((size_t)s * (size_t)p->num_layers + (size_t)layer) * (size_t)p->r_max + (size_t)j;
}

/* Pages one vector of d elements spans (paged pools). */
static int pages_per_vector(const orc_pool *p, int d) { return (d + p->page_elems - 1) / p->page_elems; }

/* Page table entry of element k of vector j (paged pools): the vector's pages are consecutive
 * entries, element k sits in its (k / page_elems)-th page. */
static size_t page_entry(const orc_pool *p, int s, int layer, int j, int d, int k) {
  return table_index(p, s, layer, j) * (size_t)pages_per_vector(p, d) + (size_t)(k / p->page_elems);
}

/* A_s[k][j] of the given layer (A is d_in x rank). */
static double elem_a(const orc_pool *p, int s, int layer, int k, int j) {
  if (p->kind == ORC_POOL_STACKED) {
    size_t row = table_index(p, s, layer, j);
    return orc_decode(p->a_t[row * (size_t)p->d_in + (size_t)k], p->dtype);
  }
  int32_t page = p->a_page_table[page_entry(p, s, layer, j, p->d_in, k)];
  return orc_decode(p->pages[(size_t)page * (size_t)p->page_elems + (size_t)(k % p->page_elems)], p->dtype);
}

/* B_s[j][n] of the given layer (B is rank x d_out). */
static double elem_b(const orc_pool *p, int s, int layer, int j, int n) {
  if (p->kind == ORC_POOL_STACKED) {
    size_t row = table_index(p, s, layer, j);
    return orc_decode(p->b[row * (size_t)p->d_out + (size_t)n], p->dtype);
  }
  int32_t page = p->b_page_table[page_entry(p, s, layer, j, p->d_out, n)];
  return orc_decode(p->pages[(size_t)page * (size_t)p->page_elems + (size_t)(n % p->page_elems)], p->dtype);
}

/* Status bits for using slot s (s >= 0 assumed checked against num_slots by the caller).
 * need_a / need_b select which page tables must hold valid ids. */
static int32_t check_adapter(const orc_pool *p, int s, int layer, int need_a, int need_b) {
  int r = p->rank[s];
  if (r < 1 || r > p->r_max) return ORC_BAD_RANK;
  if (p->kind == ORC_POOL_PAGED) {
    for (int j = 0; j < r; ++j) {
      if (need_a) {
        for (int k = 0; k < p->d_in; k += p->page_elems) {
          int32_t pa = p->a_page_table[page_entry(p, s, layer, j, p->d_in, k)];
          if (pa < 0 || pa >= p->num_pages) return ORC_BAD_PAGE;
        }
      }
      if (need_b) {
        for (int n = 0; n < p->d_out; n += p->page_elems) {
          int32_t pb = p->b_page_table[page_entry(p, s, layer, j, p->d_out, n)];
          if (pb < 0 || pb >= p->num_pages) return ORC_BAD_PAGE;
        }
      }
    }
  }
  return 0;
}

static int check_pool(const orc_pool *p, int layer) {
  if (!p || !p->rank || !p->scale) return ORC_ERR_ARG;
  if (p->dtype != ORC_DTYPE_BF16 && p->dtype != ORC_DTYPE_FP16) return ORC_ERR_ARG;
  if (p->num_slots < 1 || p->num_layers < 1 || p->r_max < 1 || p->d_in < 1 || p->d_out < 1)
    return ORC_ERR_ARG;
  if (layer < 0 || layer >= p->num_layers) return ORC_ERR_ARG;
  if (p->kind == ORC_POOL_STACKED) {
    if (!p->a_t || !p->b) return ORC_ERR_ARG;
  } else if (p->kind == ORC_POOL_PAGED) {
    if (!p->pages || !p->a_page_table || !p->b_page_table) return ORC_ERR_ARG;
    if (p->page_elems < 1 || p->num_pages < 1) return ORC_ERR_ARG;
  } else {
    return ORC_ERR_ARG;
  }
  return 0;
}

/* Slot of row i under SGMV segments: the t with off[t] <= i < off[t+1] (plain scan). */
static int32_t sgmv_row_slot(const int32_t *off, const int32_t *seg_slot, int nseg, int i) {
  for (int t = 0; t < nseg; ++t)
    if (off[t] <= i && i < off[t + 1]) return seg_slot[t];
  return -1; /* unreachable when the offsets are valid */
}

static int sgmv_offsets_valid(const int32_t *off, int nseg, int M) {
  if (off[0] != 0 || off[nseg] != M) return 0;
  for (int t = 0; t < nseg; ++t)
    if (off[t + 1] < off[t]) return 0;
  return 1;
}

/* ---- the two phases, one row at a time ------------------------------------------------ */

/* Phase 1 (shrink) for row i: v[i][j] = sum_k x[i][k] A_s[k][j], j < rank[s]. */
static void shrink_row(const orc_pool *p, int layer, int s, const uint16_t *x_row, double *v_row) {
  int r = p->rank[s];
  for (int j = 0; j < r; ++j) {
    double acc = 0.0;
    for (int k = 0; k < p->d_in; ++k) acc += orc_decode(x_row[k], p->dtype) * elem_a(p, s, layer, k, j);
    v_row[j] = acc;
  }
}

/* Phase 2 (expand) for row i: y'[i][n] = RNE(y[i][n] + scale[s] * sum_j v[i][j] B_s[j][n]). */
static void expand_row(const orc_pool *p, int layer, int s, const double *v_row, uint16_t *y_row,
                       double *y_exact_row) {
  int r = p->rank[s];
  double sc = (double)p->scale[s];
  for (int n = 0; n < p->d_out; ++n) {
    double acc = 0.0;
    for (int j = 0; j < r; ++j) acc += v_row[j] * elem_b(p, s, layer, j, n);
    double out = orc_decode(y_row[n], p->dtype) + sc * acc;
    if (y_exact_row) y_exact_row[n] = out;
    y_row[n] = orc_round(out, p->dtype);
  }
}

/* Resolve, check and run one phase for one row. phase 1 = shrink, 2 = expand. */
static int32_t run_row(const orc_pool *p, int layer, int32_t s, int phase, int i, const uint16_t *x,
                       int64_t ldx, double *v, uint16_t *y, int64_t ldy, double *y_exact) {
  if (s == -1) return 0; /* no adapter: the row is not touched */
  if (s < -1 || s >= p->num_slots) return ORC_BAD_SLOT;
  int32_t bad = check_adapter(p, s, layer, phase == 1, phase == 2);
  if (bad) return bad;
  double *v_row = v + (size_t)i * (size_t)p->r_max;
  if (phase == 1) {
    shrink_row(p, layer, s, x + (size_t)i * (size_t)ldx, v_row);
  } else {
    expand_row(p, layer, s, v_row, y + (size_t)i * (size_t)ldy,
               y_exact ? y_exact + (size_t)i * (size_t)p->d_out : NULL);
  }
  return 0;
}

/* rows == NULL means every row 0..M-1, else the listed rows (for sampled checks). */
static int run_phase(const orc_pool *p, int layer, int phase, const int32_t *off, const int32_t *seg_slot,
                     int nseg, const int32_t *row_slot, int M, const int32_t *rows, int nrows,
                     const uint16_t *x, int64_t ldx, double *v, uint16_t *y, int64_t ldy, double *y_exact,
                     int32_t *status) {
  int rc = check_pool(p, layer);
  if (rc) return rc;
  if (M < 0 || (phase == 1 && (!x || !v || ldx < p->d_in)) || (phase == 2 && (!y || !v || ldy < p->d_out)))
    return ORC_ERR_ARG;
  int32_t st = 0;
  if (off) {
    if (nseg < 0 || !seg_slot) return ORC_ERR_ARG;
    if (!sgmv_offsets_valid(off, nseg, M)) {
      if (status) *status |= ORC_BAD_OFFSETS;
      return 0;
    }
  } else if (!row_slot && M > 0) {
    return ORC_ERR_ARG;
  }
  int count = rows ? nrows : M;
  for (int q = 0; q < count; ++q) {
    int i = rows ? rows[q] : q;
    if (i < 0 || i >= M) return ORC_ERR_ARG;
    int32_t s = off ? sgmv_row_slot(off, seg_slot, nseg, i) : row_slot[i];
    st |= run_row(p, layer, s, phase, i, x, ldx, v, y, ldy, y_exact);
  }
  if (status) *status |= st;
  return 0;
}

/* ---- exported entry points -------------------------------------------------------------- */

int orc_sgmv_shrink(const orc_pool *p, int layer, const uint16_t *x, int64_t ldx, const int32_t *off,
                    const int32_t *seg_slot, int nseg, int M, const int32_t *rows, int nrows, double *v,
                    int32_t *status) {
  if (!off) return ORC_ERR_ARG;
  return run_phase(p, layer, 1, off, seg_slot, nseg, NULL, M, rows, nrows, x, ldx, v, NULL, 0, NULL, status);
}

int orc_sgmv_expand(const orc_pool *p, int layer, const double *v, uint16_t *y, int64_t ldy,
                    const int32_t *off, const int32_t *seg_slot, int nseg, int M, const int32_t *rows,
                    int nrows, double *y_exact, int32_t *status) {
  if (!off) return ORC_ERR_ARG;
  return run_phase(p, layer, 2, off, seg_slot, nseg, NULL, M, rows, nrows, NULL, 0, (double *)v, y, ldy,
                   y_exact, status);
}

int orc_bgmv_shrink(const orc_pool *p, int layer, const uint16_t *x, int64_t ldx, const int32_t *row_slot,
                    int M, const int32_t *rows, int nrows, double *v, int32_t *status) {
  return run_phase(p, layer, 1, NULL, NULL, 0, row_slot, M, rows, nrows, x, ldx, v, NULL, 0, NULL, status);
}

int orc_bgmv_expand(const orc_pool *p, int layer, const double *v, uint16_t *y, int64_t ldy,
                    const int32_t *row_slot, int M, const int32_t *rows, int nrows, double *y_exact,
                    int32_t *status) {
  return run_phase(p, layer, 2, NULL, NULL, 0, row_slot, M, rows, nrows, NULL, 0, (double *)v, y, ldy, y_exact,
                   status);
}

/* Array forms of the conversions, for the Python side. */
void orc_round_array(const double *in, uint16_t *out, size_t n, int dtype) {
  for (size_t i = 0; i < n; ++i) out[i] = orc_round(in[i], dtype);
}

void orc_decode_array(const uint16_t *in, double *out, size_t n, int dtype) {
  for (size_t i = 0; i < n; ++i) out[i] = orc_decode(in[i], dtype);
}
