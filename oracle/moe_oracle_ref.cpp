// Plain C++ float64 reference of one small-batch MoE decode layer step.
//
// TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the tests, the smoke check and the
// bench's CPU legs load it (through oracle/cpp.py); the CUDA library never links
// it and the two share no code. Slow and obvious on purpose: plain loops, no
// BLAS, every sum accumulated in float64 in index order.
//
// What one step computes, per token row m (M = 1..16 rows):
//
//   1. router logits   l[e] = sum_h x[h] * Wr[e, h]
//        Ling-3.0-flash batch-1 decode blog, section "PDL: stacking the latency
//        floors of small kernels" (router chain: norm -> gate matvec -> top-k)
//        and section "bf16 router gate and lm_head" (a bf16 matvec).
//   2. selection and weights, by scoring rule:
//        SOFTMAX (0): the k largest l (ties to the lower expert id), weights
//          w_j = exp(l_j - l_max) / sum over the selected of exp(l_i - l_max),
//          which is softmax over all experts, then top-k, then renormalise (the
//          full-softmax denominator cancels). The pages never fix the rule; this
//          is the documented default reading.
//        SIGMOID_BIAS (1): s_e = 1 / (1 + exp(-l_e)); the k largest s_e + b_e
//          (b: a per-expert selection bias, ties to the lower id) are selected;
//          weights w_j = s_j / sum over the selected of s_i (the bias steers the
//          choice only). The Ling blog's router top-k "prefetches its bias"
//          (section "PDL: ...", figure on the router path); the rest of the rule
//          is the plainest reading of a bias-corrected sigmoid router.
//   3. each selected expert  g = Wg x, u = Wu x, a = silu(g) * u, y = Wd a,
//        silu(g) = g / (1 + exp(-g)); W13 = [Wg; Wu] is [2I, H], W2 = Wd is [H, I].
//        Same blog, section "Two fusions and a retune".
//   4. shared experts  the same MLP with the shared weights, weight 1
//        (Ling model table: 512 routed + 1 shared expert, top-8(+1)).
//   5. combine         out = r + routed_scale * sum_j w_j y_{e_j} + sum_s y_s
//        (section "PDL: ...": one sum times a scale, one final cast; the oracle
//        keeps float64 and does not round).
//
// Weight storage (bit patterns exactly as the GPU consumes them, widened exactly):
//   F64    double values;
//   BF16   uint16 bit patterns (the top half of a float32);
//   NVFP4  e2m1 codes two per byte along the reduction dim (even element in the
//          low nibble), one e4m3 scale byte per 16 consecutive elements, and a
//          float32 tensor scale per (expert, projection): w = e2m1 * e4m3 * ts.
//          (Muse Spark Open Ultrafast, section "The model": NVFP4 experts; the
//          format follows the OCP microscaling definitions of e2m1 and e4m3.)
//   FP8    one e4m3 code byte per element and one float32 scale per 128 x 128
//          block of the matrix, [rows / 128][cols / 128]: w = e4m3 * scale
//          (Ling-3.0-flash blog, section "Where the time goes now": fp8 weights,
//          block 128).
//
// Threads: the router loops over experts, and each expert's gate/up rows and
// down rows, split over OpenMP threads; every output element is one sequential
// sum, so the result does not depend on the thread count.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

// Planted mistakes for the pin tests (tests/test_oracle_pins.py builds one
// library per mutant with -DORACLE_MUTANT=n and checks that some pin fails);
// 0, the default, is the oracle itself.
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

namespace {

constexpr int kMutant = ORACLE_MUTANT;
enum Mutant {
  MUT_SWAP_GATE_UP = 1,
  MUT_SIGMOID_NOT_SILU = 2,
  MUT_SILU_SIGN = 3,
  MUT_NO_RENORM = 4,
  MUT_TIES_TO_HIGHER = 5,
  MUT_ROUTER_ROWS_REVERSED = 6,
  MUT_BOTTOM_K = 7,
  MUT_DROP_SHARED = 8,
  MUT_DROP_RESIDUAL = 9,
  MUT_BIAS_IN_WEIGHTS = 10,
  MUT_BF16_TRUNCATE = 11,
  MUT_NIBBLE_ORDER = 12,
  MUT_E4M3_BIAS = 13,
  MUT_NO_ROUTED_SCALE = 14,
  MUT_FP8_SCALE_TRANSPOSED = 15,
};

enum { FMT_F64 = 0, FMT_BF16 = 1, FMT_NVFP4 = 2, FMT_FP8 = 3 };
enum { SCORE_SOFTMAX = 0, SCORE_SIGMOID_BIAS = 1 };
enum { OK = 0, ERR_ARG = 1, ERR_MISSING_EXPERT = 2 };

double bf16_value(uint16_t bits) {
  const uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// e2m1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent field 0
// is subnormal (0.5 * mantissa). No infinities or NaNs.
double e2m1_value(unsigned code) {
  code &= 0xFu;
  const double sign = (code & 0x8u) ? -1.0 : 1.0;
  const unsigned ex = (code >> 1) & 0x3u, man = code & 0x1u;
  const double mag = ex == 0 ? 0.5 * man : std::ldexp(1.0 + man / 2.0, static_cast<int>(ex) - 1);
  return sign * mag;
}

// e4m3 (fn): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
// subnormal (2^-6 * mantissa / 8); exponent 15 with mantissa 7 is NaN; no infinity.
double e4m3_value(unsigned byte) {
  byte &= 0xFFu;
  const double sign = (byte & 0x80u) ? -1.0 : 1.0;
  const unsigned ex = (byte >> 3) & 0xFu, man = byte & 0x7u;
  if (ex == 0xFu && man == 0x7u) return std::nan("");
  const int bias = kMutant == MUT_E4M3_BIAS ? 8 : 7;
  const double mag = ex == 0 ? std::ldexp(man / 8.0, 1 - bias) : std::ldexp(1.0 + man / 8.0, static_cast<int>(ex) - bias);
  return sign * mag;
}

double sigmoid(double v) { return 1.0 / (1.0 + std::exp(-v)); }

double silu(double g) {
  if (kMutant == MUT_SIGMOID_NOT_SILU) return sigmoid(g);
  if (kMutant == MUT_SILU_SIGN) return g / (1.0 + std::exp(g));
  return g / (1.0 + std::exp(-g));
}

}  // namespace

extern "C" {

// One weight matrix set per expert; entries of unused experts may be NULL.
typedef struct {
  int32_t fmt;                      // FMT_F64, FMT_BF16, FMT_NVFP4 or FMT_FP8
  const void* const* w13;           // [n] -> [2I, H] values or e4m3 codes, or e2m1 codes [2I, H/2]
  const void* const* w2;            // [n] -> [H, I] values or e4m3 codes, or e2m1 codes [H, I/2]
  const uint8_t* const* w13_scale;  // NVFP4: [n] -> e4m3 [2I, H/16]; FP8: float [2I/128, H/128]
  const uint8_t* const* w2_scale;   // NVFP4: [n] -> e4m3 [H, I/16]; FP8: float [H/128, I/128]
  const float* w13_gscale;          // NVFP4: [n][2] tensor scale of the gate rows, of the up rows
  const float* w2_gscale;           // NVFP4: [n]
} moe_oracle_experts;

typedef struct {
  int32_t hidden, inter, num_experts, top_k, num_shared, rows;
  int32_t score;        // SCORE_SOFTMAX or SCORE_SIGMOID_BIAS
  int32_t router_fmt;   // FMT_F64 or FMT_BF16
  double routed_scale;
  int32_t threads;      // OpenMP threads (<= 0: the runtime's default)
} moe_oracle_shape;

int32_t moe_oracle_version(void) { return 1; }

int32_t moe_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

// Exact widening of bf16 bit patterns.
void moe_oracle_bf16_to_f64(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_value(in[i]);
}

// Round to the nearest bf16, ties to even. bf16 keeps 8 significant bits: for
// v = f * 2^e with 0.5 <= |f| < 1 the spacing near v is 2^(e-8), and below the
// smallest normal (2^-126) it stays 2^-133. nearbyint rounds halves to even in
// the default rounding mode. Values past the largest bf16 become infinities.
void moe_oracle_f64_to_bf16(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    const double v = in[i];
    uint32_t u;
    if (std::isnan(v)) {
      u = 0x7FC00000u;
    } else if (v == 0.0 || std::isinf(v)) {
      const float f = static_cast<float>(v);
      std::memcpy(&u, &f, sizeof u);
    } else {
      int e;
      std::frexp(v, &e);
      const double quantum = std::ldexp(1.0, (e > -125 ? e : -125) - 8);
      const double r = (kMutant == MUT_BF16_TRUNCATE ? std::trunc(v / quantum) : std::nearbyint(v / quantum)) * quantum;
      const float f = static_cast<float>(r);  // exact (8 significant bits) or overflows to inf
      std::memcpy(&u, &f, sizeof u);
    }
    out[i] = static_cast<uint16_t>(u >> 16);
  }
}

double moe_oracle_e2m1(int32_t code) { return e2m1_value(static_cast<unsigned>(code)); }
double moe_oracle_e4m3(int32_t byte) { return e4m3_value(static_cast<unsigned>(byte)); }

void moe_oracle_silu(const double* g, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = silu(g[i]);
}

// RMSNorm with gamma = 1 of bf16 rows, rounded once to bf16: the input of the
// next stacked layer, h / sqrt(mean(h^2) + eps) (router chain "norm" step).
void moe_oracle_rmsnorm_bf16(const uint16_t* h, uint16_t* out, int32_t rows, int32_t hidden, double eps) {
  std::vector<double> v(hidden);
  for (int32_t m = 0; m < rows; ++m) {
    double ss = 0.0;
    for (int32_t i = 0; i < hidden; ++i) {
      v[i] = bf16_value(h[static_cast<size_t>(m) * hidden + i]);
      ss += v[i] * v[i];
    }
    const double scale = 1.0 / std::sqrt(ss / hidden + eps);
    for (int32_t i = 0; i < hidden; ++i) v[i] *= scale;
    moe_oracle_f64_to_bf16(v.data(), out + static_cast<size_t>(m) * hidden, hidden);
  }
}

// Selection and weights of one row from its logits (step 2). idx in descending
// order of the selection key (equal keys: ascending expert id), w the weights.
int32_t moe_oracle_select(const double* logits, int32_t num_experts, int32_t top_k, int32_t score,
                          const double* bias, int64_t* idx, double* w) {
  if (top_k < 1 || top_k > num_experts) return ERR_ARG;
  if (score == SCORE_SIGMOID_BIAS && !bias) return ERR_ARG;
  std::vector<double> key(num_experts);
  for (int32_t e = 0; e < num_experts; ++e)
    key[e] = score == SCORE_SOFTMAX ? logits[e] : sigmoid(logits[e]) + bias[e];
  std::vector<char> taken(num_experts, 0);
  // k passes over all experts: the largest key not yet taken; the strict
  // comparison in ascending id order keeps the lower id on ties
  for (int32_t j = 0; j < top_k; ++j) {
    int32_t best = -1;
    for (int32_t e = 0; e < num_experts; ++e) {
      if (taken[e]) continue;
      const bool better = kMutant == MUT_BOTTOM_K       ? key[e] < key[best < 0 ? e : best]
                          : kMutant == MUT_TIES_TO_HIGHER ? key[e] >= key[best < 0 ? e : best]
                                                          : key[e] > key[best < 0 ? e : best];
      if (best < 0 || better) best = e;
    }
    taken[best] = 1;
    idx[j] = best;
  }
  if (score == SCORE_SOFTMAX) {
    double lmax = logits[idx[0]];
    for (int32_t j = 1; j < top_k; ++j) lmax = logits[idx[j]] > lmax ? logits[idx[j]] : lmax;
    double z = 0.0;
    for (int32_t j = 0; j < top_k; ++j) z += std::exp(logits[idx[j]] - lmax);
    if (kMutant == MUT_NO_RENORM) {  // the full softmax denominator
      z = 0.0;
      for (int32_t e = 0; e < num_experts; ++e) z += std::exp(logits[e] - lmax);
    }
    for (int32_t j = 0; j < top_k; ++j) w[j] = std::exp(logits[idx[j]] - lmax) / z;
  } else if (score == SCORE_SIGMOID_BIAS) {
    double z = 0.0;
    for (int32_t j = 0; j < top_k; ++j) z += kMutant == MUT_BIAS_IN_WEIGHTS ? key[idx[j]] : sigmoid(logits[idx[j]]);
    for (int32_t j = 0; j < top_k; ++j)
      w[j] = (kMutant == MUT_BIAS_IN_WEIGHTS ? key[idx[j]] : sigmoid(logits[idx[j]])) / z;
  } else {
    return ERR_ARG;
  }
  return OK;
}

// Router logits of every row (step 1): logits [rows, E].
int32_t moe_oracle_router(const double* x, const void* router_w, int32_t router_fmt, int32_t rows, int32_t hidden,
                          int32_t num_experts, int32_t threads, double* logits) {
  if (router_fmt != FMT_F64 && router_fmt != FMT_BF16) return ERR_ARG;
#ifdef _OPENMP
  if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for num_threads(threads) schedule(static)
#endif
  for (int32_t e = 0; e < num_experts; ++e) {
    for (int32_t m = 0; m < rows; ++m) {
      double acc = 0.0;
      for (int32_t h = 0; h < hidden; ++h) {
        const int32_t er = kMutant == MUT_ROUTER_ROWS_REVERSED ? num_experts - 1 - e : e;
        const size_t at = static_cast<size_t>(er) * hidden + h;
        const double wv = router_fmt == FMT_F64 ? static_cast<const double*>(router_w)[at]
                                                : bf16_value(static_cast<const uint16_t*>(router_w)[at]);
        acc += x[static_cast<size_t>(m) * hidden + h] * wv;
      }
      logits[static_cast<size_t>(m) * num_experts + e] = acc;
    }
  }
  return OK;
}

}  // extern "C"

namespace {

// Row r (of `cols` elements) of matrix `which` (0: w13, 1: w2) of expert e, widened.
bool expert_row(const moe_oracle_experts& ex, int e, int which, int r, int cols, int inter, double* dst) {
  const void* base = which == 0 ? ex.w13[e] : ex.w2[e];
  if (!base) return false;
  const size_t row0 = static_cast<size_t>(r) * cols;
  if (ex.fmt == FMT_F64) {
    const double* p = static_cast<const double*>(base) + row0;
    for (int c = 0; c < cols; ++c) dst[c] = p[c];
  } else if (ex.fmt == FMT_BF16) {
    const uint16_t* p = static_cast<const uint16_t*>(base) + row0;
    for (int c = 0; c < cols; ++c) dst[c] = bf16_value(p[c]);
  } else if (ex.fmt == FMT_FP8) {
    const uint8_t* q = static_cast<const uint8_t*>(base) + row0;
    const float* sc = reinterpret_cast<const float*>(which == 0 ? ex.w13_scale[e] : ex.w2_scale[e]);
    if (!sc) return false;
    const int rows = which == 0 ? 2 * inter : 0;  // only the transposed-index mutant needs it
    const int nb = cols / 128;
    for (int c = 0; c < cols; ++c) {
      const size_t bi = kMutant == MUT_FP8_SCALE_TRANSPOSED ? (size_t)(c / 128) * ((which == 0 ? rows : cols) / 128) + r / 128
                                                            : (size_t)(r / 128) * nb + c / 128;
      dst[c] = e4m3_value(q[c]) * static_cast<double>(sc[bi]);
    }
  } else {
    const uint8_t* q = static_cast<const uint8_t*>(base) + row0 / 2;
    const uint8_t* sc = (which == 0 ? ex.w13_scale[e] : ex.w2_scale[e]);
    if (!sc) return false;
    sc += row0 / 16;
    // gate rows (r < inter) and up rows carry their own tensor scale
    const double ts = which == 0 ? ex.w13_gscale[2 * e + (r < inter ? 0 : 1)] : ex.w2_gscale[e];
    for (int c = 0; c < cols; ++c) {
      const unsigned byte = q[c / 2];
      const bool hi = kMutant == MUT_NIBBLE_ORDER ? !(c & 1) : (c & 1);
      const unsigned code = hi ? (byte >> 4) : (byte & 0xFu);
      dst[c] = e2m1_value(code) * e4m3_value(sc[c / 16]) * ts;
    }
  }
  return true;
}

// y = W2 (silu(Wg x) * (Wu x)) for one expert and one row (step 3).
bool expert_mlp(const moe_oracle_experts& ex, int e, const double* x, int hidden, int inter, int threads,
                double* y) {
  std::vector<double> a(inter);
  bool ok = true;
#ifdef _OPENMP
#pragma omp parallel num_threads(threads)
#endif
  {
    std::vector<double> row(hidden > inter ? hidden : inter);
#ifdef _OPENMP
#pragma omp for schedule(static) reduction(&& : ok)
#endif
    for (int i = 0; i < inter; ++i) {
      double g = 0.0, u = 0.0;
      if (!expert_row(ex, e, 0, i, hidden, inter, row.data())) {
        ok = false;
        continue;
      }
      for (int h = 0; h < hidden; ++h) g += row[h] * x[h];
      if (!expert_row(ex, e, 0, inter + i, hidden, inter, row.data())) {
        ok = false;
        continue;
      }
      for (int h = 0; h < hidden; ++h) u += row[h] * x[h];
      a[i] = kMutant == MUT_SWAP_GATE_UP ? silu(u) * g : silu(g) * u;
    }
#ifdef _OPENMP
#pragma omp for schedule(static) reduction(&& : ok)
#endif
    for (int o = 0; o < hidden; ++o) {
      if (!expert_row(ex, e, 1, o, inter, inter, row.data())) {
        ok = false;
        continue;
      }
      double acc = 0.0;
      for (int i = 0; i < inter; ++i) acc += row[i] * a[i];
      y[o] = acc;
    }
  }
  return ok;
}

}  // namespace

extern "C" {

// The whole step (steps 1-5) for `rows` token rows.
//   x, residual   double [rows, H]
//   router_w      double or bf16 bits [E, H] (shape.router_fmt)
//   bias          double [E] (SIGMOID_BIAS only)
//   experts       per routed expert; only the selected ones are read
//   shared        per shared expert (shape.num_shared entries)
//   out           double [rows, H];  idx int64 [rows, k];  w double [rows, k]
//   logits        double [rows, E] or NULL
// Returns 0, ERR_ARG for a bad shape, or ERR_MISSING_EXPERT when a selected or
// shared expert's weights are NULL.
int32_t moe_oracle_layer(const moe_oracle_shape* s, const double* x, const double* residual, const void* router_w,
                         const double* bias, const moe_oracle_experts* experts, const moe_oracle_experts* shared,
                         double* out, int64_t* idx, double* w, double* logits) {
  if (!s || !x || !residual || !router_w || !experts || !out || !idx || !w) return ERR_ARG;
  const int H = s->hidden, I = s->inter, E = s->num_experts, K = s->top_k, S = s->num_shared, M = s->rows;
  if (H <= 0 || I <= 0 || E <= 0 || K <= 0 || K > E || S < 0 || M <= 0 || (S > 0 && !shared)) return ERR_ARG;
  int threads = s->threads;
#ifdef _OPENMP
  if (threads <= 0) threads = omp_get_max_threads();
#else
  threads = 1;
#endif
  std::vector<double> lg(static_cast<size_t>(M) * E);
  int32_t st = moe_oracle_router(x, router_w, s->router_fmt, M, H, E, threads, lg.data());
  if (st != OK) return st;
  if (logits) std::memcpy(logits, lg.data(), lg.size() * sizeof(double));
  std::vector<double> y(H);
  for (int m = 0; m < M; ++m) {
    const double* xm = x + static_cast<size_t>(m) * H;
    int64_t* im = idx + static_cast<size_t>(m) * K;
    double* wm = w + static_cast<size_t>(m) * K;
    st = moe_oracle_select(lg.data() + static_cast<size_t>(m) * E, E, K, s->score, bias, im, wm);
    if (st != OK) return st;
    std::vector<double> routed(H, 0.0);
    for (int j = 0; j < K; ++j) {
      if (!expert_mlp(*experts, static_cast<int>(im[j]), xm, H, I, threads, y.data())) return ERR_MISSING_EXPERT;
      for (int o = 0; o < H; ++o) routed[o] += wm[j] * y[o];
    }
    double* om = out + static_cast<size_t>(m) * H;
    const double rs = kMutant == MUT_NO_ROUTED_SCALE ? 1.0 : s->routed_scale;
    for (int o = 0; o < H; ++o)
      om[o] = (kMutant == MUT_DROP_RESIDUAL ? 0.0 : residual[static_cast<size_t>(m) * H + o]) + rs * routed[o];
    for (int t = 0; t < (kMutant == MUT_DROP_SHARED ? 0 : S); ++t) {
      if (!expert_mlp(*shared, t, xm, H, I, threads, y.data())) return ERR_MISSING_EXPERT;
      for (int o = 0; o < H; ++o) om[o] += y[o];
    }
  }
  return OK;
}

}  // extern "C"
