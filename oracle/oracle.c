/*
 * oracle.c -- the oracle: a plain, slow, obviously correct CPU statement of the
 * routed quantized mixture-of-experts step, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path calls, links or loads
 * this file; only the tests, the smoke check and the bench's CPU baseline do.
 * It shares no code, header, table or helper with the CUDA path.
 *
 * What it follows (pages of the qwen4_exp::gpu rustdoc and source):
 *  - `Gpu::router_b` (struct Gpu page): router over nb rows of x, softmax over
 *    experts, top-k.  Read here as: logits L = R x (R bf16), the k largest
 *    logits (ties to the lower expert id, ranked in float32, the precision the
 *    kernel decides in), weights = softmax over those k logits.
 *  - `union_of` (gpu.rs source page): the union of the rows' experts, unique
 *    ids in first-seen order over the row-major [nb][k] id table.
 *  - `slot_tab` / `wmap` fields (struct Gpu page): per union slot a record
 *    address; per row and slot the routing weight (0 when the row did not
 *    route to that expert).
 *  - `struct Q` and `Q::at_offset` (gpu.rs source page): an affine-quantized
 *    projection is byte offsets of codes / scales / biases relative to its
 *    record; 8 codes per uint32 word at 4 bits; groups of 64 codes (the
 *    "expert width must be a multiple of the 64-code quantization group"
 *    check in load.rs).  Weight = scale * code + bias, per 64-code group.
 *    Codes are a little-endian bitstream per row, LSB first (3-bit codes
 *    straddle words).
 *  - `Gpu::experts_b` (struct Gpu page): routed experts plus the shared
 *    expert summed per row; each expert is gate_up -> silu(gate)*up -> down.
 *    The shared expert's scalar gate is sigmoid(shared_gate . x) -- the pages
 *    name the gate but not its activation; sigmoid is the reading taken.
 *  - `expert_qmm_from` (struct Gpu page): low-bit (3/2-bit) records only for
 *    routed experts; "dense projections stay Q4", so the shared expert is 4-bit.
 *  - `encode_block` (struct Gpu page): fetched records carry the miss
 *    precision while resident ones keep theirs, so one union may mix 4-, 3-
 *    and 2-bit records; each routed expert is evaluated at its own width.
 *  - `cut_w` field (struct Gpu page), the deadline policy: a missing expert
 *    (here: one whose record is in host memory) whose weight is below w in
 *    every row is cut from the late part instead of waited for.  Read here
 *    as always cut (the deterministic worst case of the deadline), with the
 *    weights of the experts kept unchanged.
 *  - `encode_block` (struct Gpu page): the block output feeds the next block
 *    through a fused norm; stacked layers here use x_{l+1} = x_l + MoE(x^_l)
 *    with x^ the unit-weight RMSNorm (eps 1e-6) when the layer's flags ask.
 *
 * Every dot product accumulates in double; results are returned as double.
 * The bf16 "mirror" mode rounds the expert input, the dequantized weights,
 * the activation h and the output to bf16 (nearest-even) at the points where
 * the prefill tensor-core path stores bf16, so that path can be graded
 * against the same rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  uint64_t w, s, b; /* byte offsets inside the record */
  uint32_t out, inp;
} oq_t;

typedef struct {
  int32_t hidden, n_experts, top_k, inter, bits, flags;
  const uint16_t *router;        /* [E][H] bf16 bits */
  const uint16_t *shared_gate;   /* [H] bf16 bits; NULL = no shared expert */
  const uint8_t *shared_record;  /* 4-bit record of the shared expert */
  oq_t sh_gate_up, sh_down;
  const uint8_t *experts;        /* E records, `stride` bytes apart */
  uint64_t stride;
  oq_t gate_up, down;
  /* Mixed widths (NULL = every routed record has `bits`): the code width of
   * each routed record, and the projections' offsets inside a record of
   * width 4, 3 and 2 (index 4 - width). */
  const uint8_t *expert_bits;
  oq_t gate_up_w[3], down_w[3];
  /* Two tiers (NULL = every record in device memory): 1 marks a record held
   * in host memory; with cut_w > 0 such an expert whose weight is below
   * cut_w in every row of the call is cut (contributes nothing; the other
   * weights are left as they are). */
  const uint8_t *expert_tier;
  double cut_w;
} oracle_layer_t;

enum { ORACLE_RESIDUAL = 1, ORACLE_PRENORM = 2 };

/* Threads over output rows in the decode matvecs (router rows, projection
 * rows).  Off by default; each output is still computed by one thread in the
 * same order, so results do not depend on it.  Only used to time the oracle
 * on all host cores. */
static int g_par_rows = 0;
void oracle_set_parallel_rows(int on) { g_par_rows = on; }
static int par_rows(void) {
#ifdef _OPENMP
  return g_par_rows && !omp_in_parallel();
#else
  return 0;
#endif
}

/* ------------------------------------------------------------ scalars */

/* The value a bf16 bit pattern denotes (exact in double). */
double oracle_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even (via the exact
 * float-rounding of the bit pattern; doubles here are within float range). */
static double round_bf16(double v) {
  float f = (float)v; /* values reaching here are exact floats or close */
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return v;
  uint32_t lsb = (u >> 16) & 1u;
  u = (u + 0x7fffu + lsb) & 0xffff0000u;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double silu(double g) { return g / (1.0 + exp(-g)); }
static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

/* ------------------------------------------------------------ codes */

/* Code `i` of one row: bits [i*bits, i*bits+bits) of the row's bitstream,
 * taken one bit at a time, LSB first. */
uint32_t oracle_code_at(const uint32_t *row, int64_t i, int bits) {
  uint32_t v = 0;
  for (int j = 0; j < bits; j++) {
    int64_t p = i * bits + j;
    v |= ((row[p >> 5] >> (p & 31)) & 1u) << j;
  }
  return v;
}

/* Dequantize one projection into W[out][inp]: W = scale(group) * code + bias(group). */
void oracle_dequant(const uint8_t *rec, const oq_t *q, int bits, double *W) {
  const int64_t words_per_row = (int64_t)q->inp * bits / 32;
  const int64_t groups = q->inp / 64;
  const uint32_t *codes = (const uint32_t *)(rec + q->w);
  const uint16_t *sc = (const uint16_t *)(rec + q->s);
  const uint16_t *bi = (const uint16_t *)(rec + q->b);
  for (int64_t o = 0; o < q->out; o++) {
    const uint32_t *row = codes + o * words_per_row;
    for (int64_t i = 0; i < q->inp; i++) {
      int64_t g = i / 64;
      double s = oracle_bf16(sc[o * groups + g]);
      double b = oracle_bf16(bi[o * groups + g]);
      W[o * q->inp + i] = s * (double)oracle_code_at(row, i, bits) + b;
    }
  }
}

/* y[out] = W x for one projection (dequantized row by row), optionally
 * rounding each weight to bf16 first (mirror mode); yabs[out] (may be NULL)
 * receives sum_i |W[o][i] x[i]|. */
static void qmatvec(const uint8_t *rec, const oq_t *q, int bits, const double *x, double *y,
                    int mirror, double *yabs) {
  const int64_t words_per_row = (int64_t)q->inp * bits / 32;
  const int64_t groups = q->inp / 64;
  const uint32_t *codes = (const uint32_t *)(rec + q->w);
  const uint16_t *sc = (const uint16_t *)(rec + q->s);
  const uint16_t *bi = (const uint16_t *)(rec + q->b);
#pragma omp parallel for schedule(static) if (par_rows())
  for (int64_t o = 0; o < q->out; o++) {
    const uint32_t *row = codes + o * words_per_row;
    double acc = 0.0, aabs = 0.0;
    for (int64_t i = 0; i < q->inp; i++) {
      int64_t g = i / 64;
      double w = oracle_bf16(sc[o * groups + g]) * (double)oracle_code_at(row, i, bits) +
                 oracle_bf16(bi[o * groups + g]);
      if (mirror) w = round_bf16(w);
      acc += w * x[i];
      aabs += fabs(w * x[i]);
    }
    y[o] = acc;
    if (yabs) yabs[o] = aabs;
  }
}

/* One dequantized weight W[o][i] of a projection (bf16-rounded when mirror). */
static double qweight(const uint8_t *rec, const oq_t *q, int bits, int64_t o, int64_t i, int mirror) {
  const int64_t words_per_row = (int64_t)q->inp * bits / 32;
  const int64_t groups = q->inp / 64;
  const uint32_t *row = (const uint32_t *)(rec + q->w) + o * words_per_row;
  const uint16_t *sc = (const uint16_t *)(rec + q->s);
  const uint16_t *bi = (const uint16_t *)(rec + q->b);
  double w = oracle_bf16(sc[o * groups + i / 64]) * (double)oracle_code_at(row, i, bits) +
             oracle_bf16(bi[o * groups + i / 64]);
  return mirror ? round_bf16(w) : w;
}

/* bf16 neighbours of a bf16 value r (r != 0): the next value away from zero
 * and the next toward zero. */
static void bf16_neighbours(double r, double *away, double *toward) {
  float f = (float)r;
  uint32_t u, a, t;
  memcpy(&u, &f, 4);
  a = u + 0x10000u;
  t = u - 0x10000u;
  float fa, ft;
  memcpy(&fa, &a, 4);
  memcpy(&ft, &t, 4);
  *away = fa;
  *toward = ft;
}

/* One expert on one row: gu = W_gu x (2*inter outputs: gate then up),
 * h = silu(gate) * up, y = W_d h.  `y` has `hidden` entries.
 *
 * Tolerance helper of the bf16 mirror (test infrastructure, not a value of
 * the method): when `allow` is given, each h whose exact value lies within
 * the fp32 accuracy band of a bf16 rounding boundary may round to either
 * side in a kernel that accumulates in fp32; the largest output change one
 * such flip can cause, |weight * W_d[o][i] * (other side - rounded h)|, is
 * max-accumulated into allow[o].  The band is 2^-20 times the sums of
 * absolute products feeding gate and up (|silu'| <= 1.1), plus 2^-22 |h|
 * for the rounding of silu and the product. */
static void expert_row(const uint8_t *rec, const oq_t *gu, const oq_t *dn, int bits, int inter,
                       const double *x, double *y, int mirror, double weight, double *allow) {
  double *g = (double *)malloc(sizeof(double) * 2 * (size_t)inter);
  double *gabs = (double *)malloc(sizeof(double) * 2 * (size_t)inter);
  double *h = (double *)malloc(sizeof(double) * (size_t)inter);
  qmatvec(rec, gu, bits, x, g, mirror, gabs);
  for (int i = 0; i < inter; i++) {
    const double hs = silu(g[i]) * g[inter + i];
    h[i] = mirror ? round_bf16(hs) : hs;
    if (mirror && allow && h[i] != 0.0) {
      double away, toward;
      bf16_neighbours(h[i], &away, &toward);
      /* the boundary on hs's side of the rounded value, and the value across it */
      const int out_side = fabs(hs) > fabs(h[i]);
      const double other = out_side ? away : toward;
      const double boundary = 0.5 * (h[i] + other);
      const double band = ldexp(fabs(silu(g[i])) * gabs[inter + i] + 1.1 * fabs(g[inter + i]) * gabs[i], -20) +
                          ldexp(fabs(hs), -22);
      if (fabs(hs - boundary) <= band) {
        for (uint32_t o = 0; o < dn->out; o++) {
          const double d = fabs(weight * qweight(rec, dn, bits, o, i, 1) * (other - h[i]));
          if (d > allow[o]) allow[o] = d;
        }
      }
    }
  }
  qmatvec(rec, dn, bits, h, y, mirror, NULL);
  free(g);
  free(gabs);
  free(h);
}

/* Exported for the rounding pin: round_bf16 on one value. */
double oracle_round_bf16(double v) { return round_bf16(v); }

/* Exported for the allowance pin: one expert on one row in mirror mode, with
 * the one-flip allowance of its h rounding max-accumulated into allow[hidden]
 * (which the caller zeroes). */
void oracle_expert_mirror(const uint8_t *rec, const oq_t *gu, const oq_t *dn, int bits, int inter,
                          const double *x, double weight, double *y, double *allow) {
  expert_row(rec, gu, dn, bits, inter, x, y, 1, weight, allow);
}

/* Record, projections and width of routed expert e. */
static void routed_record(const oracle_layer_t *L, int e, const uint8_t **rec, const oq_t **gu, const oq_t **dn,
                          int *bits) {
  *rec = L->experts + (uint64_t)e * L->stride;
  if (L->expert_bits) {
    *bits = L->expert_bits[e];
    *gu = &L->gate_up_w[4 - *bits];
    *dn = &L->down_w[4 - *bits];
  } else {
    *bits = L->bits;
    *gu = &L->gate_up;
    *dn = &L->down;
  }
}

/* Exported for the brute-force pin: expert `e` of a layer on one row. */
void oracle_expert(const oracle_layer_t *L, int e, const double *x, double *y) {
  const uint8_t *rec;
  const oq_t *gu, *dn;
  int bits;
  routed_record(L, e, &rec, &gu, &dn, &bits);
  expert_row(rec, gu, dn, bits, L->inter, x, y, 0, 1.0, NULL);
}

/* Exported for the brute-force pin: the shared expert on one row (4-bit). */
void oracle_shared_expert(const oracle_layer_t *L, const double *x, double *y) {
  expert_row(L->shared_record, &L->sh_gate_up, &L->sh_down, 4, L->inter, x, y, 0, 1.0, NULL);
}

/* ------------------------------------------------------------ routing */

/* x^ = x / sqrt(mean(x^2) + 1e-6) (unit weight). */
static void rmsnorm(const double *x, int H, double *xn) {
  double ss = 0.0;
  for (int i = 0; i < H; i++) ss += x[i] * x[i];
  double r = 1.0 / sqrt(ss / H + 1e-6);
  for (int i = 0; i < H; i++) xn[i] = x[i] * r;
}

/* Router logits of one row: L[e] = sum_i R[e][i] x[i]. */
static void router_row(const oracle_layer_t *L, const double *x, double *logit) {
#pragma omp parallel for schedule(static) if (par_rows())
  for (int e = 0; e < L->n_experts; e++) {
    double acc = 0.0;
    const uint16_t *r = L->router + (int64_t)e * L->hidden;
    for (int i = 0; i < L->hidden; i++) acc += oracle_bf16(r[i]) * x[i];
    logit[e] = acc;
  }
}

/* Top-k of one row by repeated selection of the largest remaining logit,
 * compared as float32 (the kernel's precision), ties to the lower id; then
 * the softmax over the k chosen logits (in double). */
void oracle_topk_softmax(const double *logit, int E, int k, int32_t *idx, double *w) {
  char *taken = (char *)calloc((size_t)E, 1);
  for (int r = 0; r < k; r++) {
    int best = -1;
    float bv = 0.0f;
    for (int e = 0; e < E; e++) {
      if (taken[e]) continue;
      float v = (float)logit[e];
      if (best < 0 || v > bv) { /* strict: an equal later id never wins */
        best = e;
        bv = v;
      }
    }
    taken[best] = 1;
    idx[r] = best;
  }
  double m = logit[idx[0]];
  for (int r = 1; r < k; r++)
    if (logit[idx[r]] > m) m = logit[idx[r]];
  double z = 0.0;
  for (int r = 0; r < k; r++) z += exp(logit[idx[r]] - m);
  for (int r = 0; r < k; r++) w[r] = exp(logit[idx[r]] - m) / z;
  free(taken);
}

/* Union of ids in first-seen order (row-major over [nb][k]); returns its size. */
int oracle_union(const int32_t *idx, int n, int32_t *uni) {
  int u = 0;
  for (int i = 0; i < n; i++) {
    int seen = 0;
    for (int j = 0; j < u; j++)
      if (uni[j] == idx[i]) seen = 1;
    if (!seen) uni[u++] = idx[i];
  }
  return u;
}

/* Routing alone for nb rows (norm when the layer asks, router, top-k,
 * softmax): logits [nb][E], idx [nb][k], w [nb][k].  Returns the union size;
 * uni [64] (may be NULL) receives the union. */
int oracle_route(const oracle_layer_t *L, int nb, const double *x, double *logits, int32_t *idx,
                 double *w, int32_t *uni) {
  const int H = L->hidden, E = L->n_experts, k = L->top_k;
  double *xn = (double *)malloc(sizeof(double) * (size_t)H);
  int32_t un[64 * 4];
  for (int b = 0; b < nb; b++) {
    if (L->flags & ORACLE_PRENORM)
      rmsnorm(x + (int64_t)b * H, H, xn);
    else
      memcpy(xn, x + (int64_t)b * H, sizeof(double) * H);
    router_row(L, xn, logits + (int64_t)b * E);
    oracle_topk_softmax(logits + (int64_t)b * E, E, k, idx + b * k, w + b * k);
  }
  int U = oracle_union(idx, nb * k, un);
  if (uni) memcpy(uni, un, sizeof(int32_t) * (size_t)U);
  free(xn);
  return U;
}

/* ------------------------------------------------------------ one layer */

/* The deadline cut of one call: cut[e] = 1 for each routed expert whose
 * record is in host memory and whose weight is below cut_w in every one of
 * the nb rows (0 in a row that did not route to it).  cut [E], zeroed by the
 * caller.  Returns the number cut. */
int oracle_cut(const oracle_layer_t *L, int nb, const int32_t *idx, const double *w, uint8_t *cut) {
  const int k = L->top_k;
  int n = 0;
  if (!L->expert_tier || !(L->cut_w > 0.0)) return 0;
  for (int i = 0; i < nb * k; i++) {
    const int e = idx[i];
    if (!L->expert_tier[e] || cut[e]) continue;
    double wmax = 0.0;
    for (int j = 0; j < nb * k; j++)
      if (idx[j] == e && w[j] > wmax) wmax = w[j];
    if (wmax < L->cut_w) cut[e] = 1, n++;
  }
  return n;
}

/* One MoE layer over nb rows.
 *   x      [nb][H]   layer input
 *   out    [nb][H]   layer output (MoE, plus x when the layer is RESIDUAL)
 *   moe    [nb][H]   MoE part alone (before the residual), may be NULL
 *   logits [nb][E], idx [nb][k], w [nb][k], gamma [nb], uni [64], wmap [4][64]:
 *          routing results, each may be NULL.
 * Returns the union size. */
int oracle_moe_layer(const oracle_layer_t *L, int nb, const double *x, double *out, double *moe,
                     double *logits, int32_t *idx, double *w, double *gamma, int32_t *uni,
                     double *wmap) {
  const int H = L->hidden, E = L->n_experts, k = L->top_k;
  double *xn = (double *)malloc(sizeof(double) * (size_t)nb * H);
  double *lg = (double *)malloc(sizeof(double) * (size_t)nb * E);
  int32_t *id = (int32_t *)malloc(sizeof(int32_t) * (size_t)nb * k);
  double *wt = (double *)malloc(sizeof(double) * (size_t)nb * k);
  double *y = (double *)malloc(sizeof(double) * (size_t)H);
  int32_t un[64];

  for (int b = 0; b < nb; b++) {
    if (L->flags & ORACLE_PRENORM)
      rmsnorm(x + (int64_t)b * H, H, xn + (int64_t)b * H);
    else
      memcpy(xn + (int64_t)b * H, x + (int64_t)b * H, sizeof(double) * H);
    router_row(L, xn + (int64_t)b * H, lg + (int64_t)b * E);
    oracle_topk_softmax(lg + (int64_t)b * E, E, k, id + b * k, wt + b * k);
  }
  int U = oracle_union(id, nb * k, un);
  uint8_t *cut = (uint8_t *)calloc((size_t)E, 1);
  oracle_cut(L, nb, id, wt, cut);

  for (int b = 0; b < nb; b++) {
    const double *xb = xn + (int64_t)b * H;
    double *ob = out + (int64_t)b * H;
    for (int i = 0; i < H; i++) ob[i] = 0.0;
    for (int r = 0; r < k; r++) {
      if (cut[id[b * k + r]]) continue;
      oracle_expert(L, id[b * k + r], xb, y);
      for (int i = 0; i < H; i++) ob[i] += wt[b * k + r] * y[i];
    }
    double gm = 0.0;
    if (L->shared_gate) {
      double acc = 0.0;
      for (int i = 0; i < H; i++) acc += oracle_bf16(L->shared_gate[i]) * xb[i];
      gm = sigmoid(acc);
      oracle_shared_expert(L, xb, y);
      for (int i = 0; i < H; i++) ob[i] += gm * y[i];
    }
    if (gamma) gamma[b] = gm;
    if (moe) memcpy(moe + (int64_t)b * H, ob, sizeof(double) * H);
    if (L->flags & ORACLE_RESIDUAL)
      for (int i = 0; i < H; i++) ob[i] += x[(int64_t)b * H + i];
  }

  if (logits) memcpy(logits, lg, sizeof(double) * (size_t)nb * E);
  if (idx) memcpy(idx, id, sizeof(int32_t) * (size_t)nb * k);
  if (w) memcpy(w, wt, sizeof(double) * (size_t)nb * k);
  if (uni) memcpy(uni, un, sizeof(int32_t) * (size_t)U);
  if (wmap) {
    for (int i = 0; i < 4 * 64; i++) wmap[i] = 0.0;
    for (int b = 0; b < nb; b++)
      for (int r = 0; r < k; r++)
        for (int j = 0; j < U; j++)
          if (un[j] == id[b * k + r]) wmap[b * 64 + j] = wt[b * k + r];
  }
  free(xn);
  free(lg);
  free(id);
  free(wt);
  free(y);
  free(cut);
  return U;
}

/* Stacked layers: x_{l+1} = layer_l(x_l).  `inputs` (may be NULL) receives
 * each layer's input [n_layers][nb][H]; `idx` (may be NULL) receives
 * [n_layers][nb][k]. */
void oracle_moe_forward(const oracle_layer_t *layers, int n_layers, int nb, const double *x,
                        double *out, double *inputs, int32_t *idx) {
  const int H = layers[0].hidden;
  double *cur = (double *)malloc(sizeof(double) * (size_t)nb * H);
  double *nxt = (double *)malloc(sizeof(double) * (size_t)nb * H);
  memcpy(cur, x, sizeof(double) * (size_t)nb * H);
  for (int l = 0; l < n_layers; l++) {
    if (inputs) memcpy(inputs + (int64_t)l * nb * H, cur, sizeof(double) * (size_t)nb * H);
    oracle_moe_layer(&layers[l], nb, cur, nxt, NULL, NULL,
                     idx ? idx + (int64_t)l * nb * layers[l].top_k : NULL, NULL, NULL, NULL, NULL);
    double *t = cur;
    cur = nxt;
    nxt = t;
  }
  memcpy(out, cur, sizeof(double) * (size_t)nb * H);
  free(cur);
  free(nxt);
}

/* ------------------------------------------------------------ prefill rows */

/* Independent rows of a prefill chunk (one layer).  For each listed row:
 * route in double, then evaluate the experts either exactly (mirror = 0) or
 * with bf16 rounding of x^, W, h and the output (mirror = 1).  Rows are
 * independent, so they are spread over host threads.
 *   x [t][H] float32; rows [n]; out [n][H]; idx [n][k]; w [n][k];
 *   allow [n][H] or NULL: in mirror mode, the one-flip allowance of
 *   expert_row over the row's experts (max), a test tolerance term. */
void oracle_prefill_rows(const oracle_layer_t *L, const float *x, const int64_t *rows, int n,
                         int mirror, double *out, int32_t *idx, double *w, double *allow) {
  const int H = L->hidden, E = L->n_experts, k = L->top_k;
#pragma omp parallel for schedule(dynamic, 1)
  for (int n_i = 0; n_i < n; n_i++) {
    double *xb = (double *)malloc(sizeof(double) * H);
    double *xe = (double *)malloc(sizeof(double) * H);
    double *lg = (double *)malloc(sizeof(double) * E);
    double *y = (double *)malloc(sizeof(double) * H);
    int32_t *id = idx + (int64_t)n_i * k;
    double *wt = w + (int64_t)n_i * k;
    double *ob = out + (int64_t)n_i * H;
    double *al = allow ? allow + (int64_t)n_i * H : NULL;
    if (al)
      for (int i = 0; i < H; i++) al[i] = 0.0;
    const float *xr = x + rows[n_i] * H;
    for (int i = 0; i < H; i++) xb[i] = xr[i];
    if (L->flags & ORACLE_PRENORM) rmsnorm(xb, H, xb);
    router_row(L, xb, lg);
    oracle_topk_softmax(lg, E, k, id, wt);
    for (int i = 0; i < H; i++) xe[i] = mirror ? round_bf16(xb[i]) : xb[i];
    for (int i = 0; i < H; i++) ob[i] = 0.0;
    for (int r = 0; r < k; r++) {
      const uint8_t *rec;
      const oq_t *gu, *dn;
      int bits;
      routed_record(L, id[r], &rec, &gu, &dn, &bits);
      expert_row(rec, gu, dn, bits, L->inter, xe, y, mirror, wt[r], al);
      for (int i = 0; i < H; i++) ob[i] += wt[r] * y[i];
    }
    if (L->shared_gate) {
      double acc = 0.0;
      for (int i = 0; i < H; i++) acc += oracle_bf16(L->shared_gate[i]) * xb[i];
      double gm = sigmoid(acc);
      expert_row(L->shared_record, &L->sh_gate_up, &L->sh_down, 4, L->inter, xe, y, mirror, gm, al);
      for (int i = 0; i < H; i++) ob[i] += gm * y[i];
    }
    if (L->flags & ORACLE_RESIDUAL)
      for (int i = 0; i < H; i++) ob[i] += xr[i];
    if (mirror)
      for (int i = 0; i < H; i++) ob[i] = round_bf16(ob[i]);
    free(xb);
    free(xe);
    free(lg);
    free(y);
  }
}

/* ------------------------------------------------------------ prefill grouping */

/* Routing of n independent rows of a prefill chunk: per row, as in
 * oracle_route, the logits, the top-k ids and weights; gamma[r] =
 * sigmoid(shared_gate . x^_r) when the layer has a shared expert. */
void oracle_route_rows(const oracle_layer_t *L, const float *x, int n, double *logits, int32_t *idx,
                       double *w, double *gamma) {
  const int H = L->hidden, E = L->n_experts, k = L->top_k;
#pragma omp parallel for schedule(dynamic, 16)
  for (int r = 0; r < n; r++) {
    double *xb = (double *)malloc(sizeof(double) * H);
    for (int i = 0; i < H; i++) xb[i] = x[(int64_t)r * H + i];
    if (L->flags & ORACLE_PRENORM) rmsnorm(xb, H, xb);
    router_row(L, xb, logits + (int64_t)r * E);
    oracle_topk_softmax(logits + (int64_t)r * E, E, k, idx + (int64_t)r * k, w + (int64_t)r * k);
    if (L->shared_gate && gamma) {
      double acc = 0.0;
      for (int i = 0; i < H; i++) acc += oracle_bf16(L->shared_gate[i]) * xb[i];
      gamma[r] = sigmoid(acc);
    }
    free(xb);
  }
}

/* Rows grouped by expert (`ExpertJob` / `prepare_expert_jobs`, struct Gpu
 * page): group e lists, in ascending row order, the rows whose top-k holds e,
 * with the row's weight for e; with a shared expert, group E lists every row
 * with weight gamma[r].  Group g's entries are [offs[g], offs[g+1]).  Returns
 * the number of groups. */
int oracle_group(int E, int k, int n, const int32_t *idx, const double *w, const double *gamma,
                 int32_t *offs, int32_t *rows, double *wts) {
  int pos = 0;
  for (int e = 0; e < E; e++) {
    offs[e] = pos;
    for (int r = 0; r < n; r++)
      for (int j = 0; j < k; j++)
        if (idx[(int64_t)r * k + j] == e) {
          rows[pos] = r;
          wts[pos] = w[(int64_t)r * k + j];
          pos++;
        }
  }
  int G = E;
  if (gamma) {
    offs[E] = pos;
    for (int r = 0; r < n; r++) {
      rows[pos] = r;
      wts[pos] = gamma[r];
      pos++;
    }
    G = E + 1;
  }
  offs[G] = pos;
  return G;
}

/* Threads an OpenMP region here would use (1 without OpenMP). */
int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
