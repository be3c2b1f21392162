/*
 * Plain float64 CPU oracle for the MXFP8-activation x MXFP4-weight top-16 MoE
 * decode layer.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and the CPU
 * baseline leg of bench.py may load or call this library. The product path
 * (the CUDA library under mxfp4_weight_mxfp8_gb300/) never links, imports or
 * executes it, and it shares no code, header, table or helper with that path.
 *
 * Sources (web pages, cited by title and the class/function on them):
 *   [experts]  vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.experts
 *   [runtime]  vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.experts_runtime
 * The number formats (e2m1, e4m3 "FN", E8M0, block size 32) are the OCP
 * Microscaling Formats (MX) v1.0 definitions that the pages name.
 *
 * Everything is written the slow, obvious way: values are decoded by table or
 * by their textbook formula into float64, dot products are plain sequential
 * float64 loops, rounding picks the nearest representable value by search.
 * Parity status of every function is stated beside it; all are pinned by the
 * "not gpu" tests except where a line says "parity unpinned".
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_SLOTS 16 /* top-16 routing: 16 (token, slot) pairs per token */
#define ORC_UNIT_ROWS 8 /* a unit is (expert, <= 8 pair rows): [experts] ExpertsKernel.group */

/* ------------------------------------------------------------------------ */
/* Element formats (OCP MX v1.0).                                            */
/* ------------------------------------------------------------------------ */

/* e2m1 magnitudes by the low three code bits; bit 3 is the sign. */
static const double E2M1_MAGNITUDE[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(unsigned code) {
  double m = E2M1_MAGNITUDE[code & 7u];
  return (code & 8u) ? -m : m;
}

/* e4m3 (FN variant): bias 7, no infinities, 0x7F / 0xFF are NaN, subnormals
 * are m * 2^-9, largest finite magnitude 448. */
double orc_e4m3_value(unsigned code) {
  unsigned sign = (code >> 7) & 1u, exponent = (code >> 3) & 15u, mantissa = code & 7u;
  double v;
  if (exponent == 15u && mantissa == 7u) return NAN;
  if (exponent == 0u)
    v = ldexp((double)mantissa, -9);
  else
    v = ldexp(1.0 + (double)mantissa / 8.0, (int)exponent - 7);
  return sign ? -v : v;
}

/* E8M0 scale: 2^(b - 127); b = 0xFF is NaN. */
double orc_e8m0_value(unsigned b) {
  if ((b & 255u) == 255u) return NAN;
  return ldexp(1.0, (int)(b & 255u) - 127);
}

double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Nearest finite e4m3 value, ties to the even code, saturating at 448
 * ("satfinite"), sign kept (a negative value that rounds to zero gives 0x80).
 * Found by scanning all 127 non-negative finite codes: between two adjacent
 * codes exactly one has an even last mantissa bit, which is the code's last
 * bit. Parity: pinned (hand-worked values, exhaustive midpoint test). */
uint8_t orc_e4m3_encode(double v) {
  int negative = signbit(v) ? 1 : 0;
  double a = fabs(v);
  unsigned best = 0;
  if (a >= 448.0) {
    best = 0x7Eu;
  } else {
    double best_distance = a; /* distance to code 0 (value 0) */
    for (unsigned c = 1; c <= 0x7Eu; ++c) {
      double d = fabs(a - orc_e4m3_value(c));
      if (d < best_distance || (d == best_distance && (c & 1u) == 0u)) {
        best = c;
        best_distance = d;
      }
    }
  }
  return (uint8_t)(best | (negative ? 0x80u : 0u));
}

/* Round a float64 to bfloat16, to nearest with ties to even (8 significant
 * bits; quantum 2^-133 below the smallest normal 2^-126). The quotient by the
 * quantum is exact, so nearbyint (default rounding mode: nearest-even) is the
 * whole rounding step. Parity: pinned (hand-worked halfway cases). */
uint16_t orc_bf16_encode(double v) {
  int negative = signbit(v) ? 1 : 0;
  double a = fabs(v), r;
  uint32_t u;
  float f;
  if (isnan(v)) return 0x7FC0u;
  if (a == 0.0) {
    r = 0.0;
  } else {
    int e;
    frexp(a, &e); /* a in [2^(e-1), 2^e) */
    int quantum_exp = (e - 1 >= -126) ? (e - 8) : -133;
    r = ldexp(nearbyint(ldexp(a, -quantum_exp)), quantum_exp);
    if (r >= ldexp(1.0, 128)) r = INFINITY;
  }
  f = (float)r; /* exact: r is a bfloat16 value */
  memcpy(&u, &f, sizeof u);
  return (uint16_t)((u >> 16) | (negative ? 0x8000u : 0u));
}

/* ------------------------------------------------------------------------ */
/* MXFP8 block quantization ([experts] mx_block, plan_chunk,                 */
/* ExpertsKernel.store_hidden).                                              */
/* ------------------------------------------------------------------------ */

/* Shared exponent E of one 32-element block with largest magnitude amax.
 *  ceil rule  (floor_rule = 0): the smallest integer E with amax <= 448 * 2^E,
 *             so no element saturates;
 *  floor rule (floor_rule = 1): E = floor(log2(amax)) - 8, the OCP MX v1.0
 *             rule with emax(e4m3) = 8; elements may saturate at 448.
 * An all-zero block takes E = -127. E is clamped to the E8M0 range [-127, 127].
 * The ceil rule is found by stepping E until the defining inequality holds.
 * Parity: pinned (powers of two, the 1.75 boundary, floor-mode cases). */
int orc_mx_exponent(double amax, int floor_rule) {
  int e, E;
  if (!(amax > 0.0)) return -127;
  frexp(amax, &e); /* amax in [2^(e-1), 2^e) */
  if (floor_rule) {
    E = (e - 1) - 8;
  } else {
    E = e - 9;
    while (amax > ldexp(448.0, E)) ++E;
    while (amax <= ldexp(448.0, E - 1)) --E;
  }
  if (E < -127) E = -127;
  if (E > 127) E = 127;
  return E;
}

/* One block of 32 values: scale byte E + 127 and codes e4m3(v * 2^-E). */
void orc_mxfp8_block(const double* v, int floor_rule, uint8_t* codes, uint8_t* scale) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  int E = orc_mx_exponent(amax, floor_rule);
  *scale = (uint8_t)(E + 127);
  for (int i = 0; i < 32; ++i) codes[i] = orc_e4m3_encode(ldexp(v[i], -E));
}

/* Activation plan: every token row x[t, :] (BF16) in blocks of 32 with the
 * ceil rule ([experts] mx_block / ExpertsPlanKernel). codes [B, H],
 * scales [B, H/32]. */
void orc_quantize_x(const uint16_t* x, int B, int H, uint8_t* codes, uint8_t* scales) {
  double block[32];
  for (int t = 0; t < B; ++t)
    for (int b = 0; b < H / 32; ++b) {
      for (int i = 0; i < 32; ++i) block[i] = orc_bf16_value(x[(size_t)t * H + b * 32 + i]);
      orc_mxfp8_block(block, 0, codes + (size_t)t * H + b * 32, scales + (size_t)t * (H / 32) + b);
    }
}

/* ------------------------------------------------------------------------ */
/* Grouping ([experts] ExpertsKernel.group).                                 */
/* ------------------------------------------------------------------------ */

/* Canonical unit table: experts in ascending order; expert e's pairs
 * (token * 16 + slot) in token order fill ceil(n_e / 8) units of 8 rows,
 * the last padded with -1. Returns the unit count, or -1 if it would exceed
 * max_units. Parity: pinned (brute-force recount, invariants). */
int orc_group(const int32_t* ids, int B, int E, int32_t* unit_expert, int16_t* unit_rows,
              int max_units) {
  int units = 0, filled = ORC_UNIT_ROWS;
  for (int e = 0; e < E; ++e) {
    filled = ORC_UNIT_ROWS;
    for (int t = 0; t < B; ++t)
      for (int s = 0; s < ORC_SLOTS; ++s) {
        if (ids[t * ORC_SLOTS + s] != e) continue;
        if (filled == ORC_UNIT_ROWS) {
          if (units >= max_units) return -1;
          unit_expert[units] = e;
          for (int r = 0; r < ORC_UNIT_ROWS; ++r) unit_rows[units * ORC_UNIT_ROWS + r] = -1;
          ++units;
          filled = 0;
        }
        unit_rows[(units - 1) * ORC_UNIT_ROWS + filled] = (int16_t)(t * ORC_SLOTS + s);
        ++filled;
      }
  }
  return units;
}

/* ------------------------------------------------------------------------ */
/* One routed (token, slot) pair through its expert.                         */
/* ------------------------------------------------------------------------ */

typedef struct {
  const uint8_t* w13; /* [E, 2I, H/2] e2m1 pairs, element 2i in the low nibble of byte i */
  const uint8_t* s13; /* [E, 2I, H/32] E8M0 */
  const uint8_t* w2;  /* [E, H, I/2] */
  const uint8_t* s2;  /* [E, H, I/32] */
  int E, H, I;
} orc_weights;

/* Decode tables: the value of every e4m3 code and every E8M0 byte, filled
 * once from the functions above (decoding "by table"). */
static double E4M3_TABLE[256], E8M0_TABLE[256];
static int tables_ready = 0;

static void fill_tables(void) {
  if (tables_ready) return;
  for (unsigned c = 0; c < 256; ++c) {
    E4M3_TABLE[c] = orc_e4m3_value(c);
    E8M0_TABLE[c] = orc_e8m0_value(c);
  }
  tables_ready = 1;
}

/* Row `row` of an MXFP4 matrix with K columns, decoded to float64. */
static void decode_row(const uint8_t* w, const uint8_t* s, size_t row, int K, double* out) {
  const uint8_t* wr = w + row * (size_t)(K / 2);
  const uint8_t* sr = s + row * (size_t)(K / 32);
  for (int k = 0; k < K; ++k) {
    unsigned byte = wr[k / 2];
    unsigned code = (k & 1) ? (byte >> 4) : (byte & 15u);
    out[k] = orc_e2m1_value(code) * E8M0_TABLE[sr[k / 32]];
  }
}

/* FC1 of expert e on one dequantized activation row xv[H] (float64):
 * y[r] = sum_k W13[e, r, k] * xv[k], r in [0, 2I) (rows 0..I-1 gate,
 * I..2I-1 up). [experts] stage ("fc1": FP4 weights x MXFP8 activations,
 * block-scaled, FP32 accumulation on the GPU; exact sums here). */
static void fc1(const orc_weights* W, int e, const double* xv, double* y, double* wrow) {
  for (int r = 0; r < 2 * W->I; ++r) {
    decode_row(W->w13, W->s13, (size_t)e * 2 * W->I + r, W->H, wrow);
    double acc = 0.0;
    for (int k = 0; k < W->H; ++k) acc += wrow[k] * xv[k];
    y[r] = acc;
  }
}

/* Gated activation: h[j] = SiLU(gate[j]) * up[j], SiLU(z) = z / (1 + e^-z).
 * The pages call it "SiTU" with beta = 4, linear_beta = 25 ([experts]
 * ExpertsKernel.store_hidden; [runtime] PersistentExperts.__init__) but never
 * print its formula; this build reads it as SiLU(gate) * up (beta and
 * linear_beta unused). Parity: pinned by closed forms of SiLU; the true SiTU
 * is parity unpinned (no formula on the pages). */
double orc_gated(double gate, double up) { return gate / (1.0 + exp(-gate)) * up; }

/* FC2 of expert e on the dequantized hidden row hv[I]:
 * o[n] = sum_j W2[e, n, j] * hv[j], n in [0, H). [experts] stage ("fc2"). */
static void fc2(const orc_weights* W, int e, const double* hv, double* o, double* wrow) {
  for (int n = 0; n < W->H; ++n) {
    decode_row(W->w2, W->s2, (size_t)e * W->H + n, W->I, wrow);
    double acc = 0.0;
    for (int j = 0; j < W->I; ++j) acc += wrow[j] * hv[j];
    o[n] = acc;
  }
}

/* The hidden requant uses the floor rule exactly when 2I == 768 ([experts]
 * ExpertsKernel.store_hidden passes floor = (tp == 8); [runtime]
 * PersistentExperts.__init__ sets tp = 8 iff w13 has 768 rows). */
int orc_hidden_floor_rule(int I) { return 2 * I == 768; }

/* Full path for a list of pairs p = token * 16 + slot:
 *   xq, xs  : the activation plan (orc_quantize_x output);
 *   out     : [n, H] BF16 rows (RNE of the float64 FC2 result);
 *   hq, hs  : optional [n, I] / [n, I/32] hidden codes and scales;
 *   y       : optional [n, 2I] float64 FC1 results.
 * Pairs are independent; OpenMP runs them on `threads` host threads. */
void orc_pairs(const uint8_t* w13, const uint8_t* s13, const uint8_t* w2, const uint8_t* s2,
               int E, int H, int I, const uint8_t* xq, const uint8_t* xs, const int32_t* ids,
               const int32_t* pairs, int n, uint16_t* out, uint8_t* hq, uint8_t* hs, double* y,
               int threads) {
  orc_weights W = {w13, s13, w2, s2, E, H, I};
  int floor_rule = orc_hidden_floor_rule(I);
  fill_tables();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads > 0 ? threads : 1)
  for (int i = 0; i < n; ++i) {
    int pair = pairs[i], token = pair / ORC_SLOTS, e = ids[pair];
    double* xv = (double*)malloc(sizeof(double) * (size_t)H);
    double* yy = (double*)malloc(sizeof(double) * 2 * (size_t)I);
    double* hv = (double*)malloc(sizeof(double) * (size_t)I);
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
    uint8_t* codes = (uint8_t*)malloc((size_t)I);
    uint8_t* scales = (uint8_t*)malloc((size_t)(I / 32));
    /* one decoded weight row: FC1 rows hold H values, FC2 rows I */
    double* wrow = (double*)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    for (int k = 0; k < H; ++k)
      xv[k] = E4M3_TABLE[xq[(size_t)token * H + k]] * E8M0_TABLE[xs[(size_t)token * (H / 32) + k / 32]];
    fc1(&W, e, xv, yy, wrow);
    for (int j = 0; j < I; ++j) hv[j] = orc_gated(yy[j], yy[I + j]);
    for (int b = 0; b < I / 32; ++b) orc_mxfp8_block(hv + 32 * b, floor_rule, codes + 32 * b, scales + b);
    for (int j = 0; j < I; ++j) hv[j] = E4M3_TABLE[codes[j]] * E8M0_TABLE[scales[j / 32]];
    fc2(&W, e, hv, o, wrow);
    for (int c = 0; c < H; ++c) out[(size_t)i * H + c] = orc_bf16_encode(o[c]);
    if (hq) memcpy(hq + (size_t)i * I, codes, (size_t)I);
    if (hs) memcpy(hs + (size_t)i * (I / 32), scales, (size_t)(I / 32));
    if (y) memcpy(y + (size_t)i * 2 * I, yy, sizeof(double) * 2 * (size_t)I);
    free(xv), free(yy), free(hv), free(o), free(codes), free(scales), free(wrow);
  }
}

/* FC2 alone from given hidden codes/scales (used to separate hidden requant
 * flips from FC2 parity): out[i, :] = bf16(W2[experts[i]] . deq(hq[i], hs[i])). */
void orc_fc2_rows(const uint8_t* w2, const uint8_t* s2, int E, int H, int I, const int32_t* experts,
                  const uint8_t* hq, const uint8_t* hs, int n, uint16_t* out, int threads) {
  orc_weights W = {NULL, NULL, w2, s2, E, H, I};
  fill_tables();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads > 0 ? threads : 1)
  for (int i = 0; i < n; ++i) {
    double* hv = (double*)malloc(sizeof(double) * (size_t)I);
    double* o = (double*)malloc(sizeof(double) * (size_t)H);
    double* wrow = (double*)malloc(sizeof(double) * (size_t)I);
    for (int j = 0; j < I; ++j)
      hv[j] = E4M3_TABLE[hq[(size_t)i * I + j]] * E8M0_TABLE[hs[(size_t)i * (I / 32) + j / 32]];
    fc2(&W, experts[i], hv, o, wrow);
    for (int c = 0; c < H; ++c) out[(size_t)i * H + c] = orc_bf16_encode(o[c]);
    free(hv), free(o), free(wrow);
  }
}

/* ------------------------------------------------------------------------ */
/* Routing-weighted combine ([experts] ExpertsKernel.finalize, single GPU):  */
/* out[t, n] = BF16( sum over s of w[t, s] * row[t, s, n] ), where row is   */
/* the BF16 per-pair output and pairs that got no row (kept == 0) are left  */
/* out. The sum is taken in float64, in slot order, and rounded once.       */
/* Pinned by the "not gpu" tests (one-hot weights, zero weights, exact      */
/* power-of-two scaling, cancellation, skipped pairs).                      */
/* ------------------------------------------------------------------------ */
void orc_combine(const uint16_t* rows, const float* weights, const uint8_t* kept, int B, int H,
                 uint16_t* out) {
  for (int t = 0; t < B; ++t)
    for (int n = 0; n < H; ++n) {
      double acc = 0.0;
      for (int s = 0; s < ORC_SLOTS; ++s) {
        const size_t p = (size_t)t * ORC_SLOTS + (size_t)s;
        if (!kept[p]) continue;
        acc += (double)weights[p] * orc_bf16_value(rows[p * (size_t)H + (size_t)n]);
      }
      out[(size_t)t * (size_t)H + (size_t)n] = orc_bf16_encode(acc);
    }
}
