// Float64 CPU oracle for grouped-query attention with a learned per-head
// softmax sink.
//
// TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg may load this file's library. The product path
// (the CUDA kernels behind libsinkattn) never calls it, and the two share no
// code: no headers, helpers, tables or pre/post-processing.
//
// What it follows ("GPT-OSS on Day 0", Perplexity, section "Kernels for
// GPT-OSS / Sink attention"; "Attention: GQA with attention sinks"):
//   attn = softmax(q @ k^T * sm_scale + sink) * V
// read as: the sink s_h of query head h is one extra logit column whose value
// row is zero. Several query heads share one KV head (GQA); KV head of query
// head h is floor(h / G), G = Hq / Hkv. The KV cache is in HND order ("Hosting
// Qwen on Blackwell", section "Deployment on GB200 NVL72"): heads leading,
// tokens contiguous.
//
// The oracle never splits a row: for every (sequence, query row, query head)
// it materialises the whole visible logit row plus the sink column in
// float64, takes its maximum, and forms the softmax-weighted sum of V. The
// only rounding beyond the bf16 inputs is float64 arithmetic.
//
// The split/merge entry points state the two steps of the split-KV method
// (per-chunk partial state without the sink, then a fold that seeds the
// running max with the sink so it counts once) so that tests can pin the merge
// rule against the unsplit row, and so the GPU's per-split partials can be
// compared with values the oracle computes on its own.
//
// Conventions (readings of points the pages leave open):
//  * positions: query row i of a sequence with Lq queries and Lk keys sits at
//    position p = Lk - Lq + i (queries are the last Lq positions);
//  * causal: key j visible iff j <= p;
//  * window W > 0 (only with causal): key j visible iff j > p - W, i.e. the W
//    keys p-W+1 .. p including the query's own position;
//  * sink units: natural-log units of the scaled logits (added after the
//    scale, never multiplied by it);
//  * lse = M + ln Z includes the sink column;
//  * no keys and no sink (s = -inf): out = 0, lse = -inf.
//
// FP8 KV entry points (oracle_attend_rows_fp8, oracle_split_partials_fp8):
// K and V hold e4m3 codes (the OCP 8-bit floating-point format E4M3: sign,
// 4-bit exponent with bias 7, 3-bit mantissa, exponent 0 subnormal, the code
// S.1111.111 NaN, no infinities), and KV head g's values are code * k_scale[g]
// (keys) and code * v_scale[g] (values). Everything else is as above.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

// ORACLE_PLANT selects one deliberate mistake, for the test that checks the
// pins catch it. It is never defined in the library that tests load.
#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

namespace {

double bf16_bits_to_double(uint16_t bits) {
  // bf16 is the upper half of an IEEE binary32; widening is exact.
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

const double kNegInf = -std::numeric_limits<double>::infinity();

// e4m3 code -> value, from the format's definition.
double e4m3_to_double(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return std::numeric_limits<double>::quiet_NaN();
  const int bias = (ORACLE_PLANT == 10) ? 8 : 7;
  const double mag = (e == 0) ? std::ldexp(m / 8.0, 1 - bias) : std::ldexp(1.0 + m / 8.0, e - bias);
  return sign ? -mag : mag;
}

struct Problem {
  const uint16_t* q;      // [total_q, Hq, d]
  const void* k;          // ragged HND: sequence b at element Hkv*cu_k[b]*d, [Hkv, Lk_b, d]
  const void* v;          // same layout as k
  const double* sinks;    // [Hq] or nullptr (no sink column)
  const int32_t* cu_q;    // [B+1]
  const int32_t* cu_k;    // [B+1]
  int B, Hq, Hkv, d;
  double scale;
  int causal, window;
  // K/V element type: bf16 bits, or e4m3 codes with per-KV-head scales
  int fp8 = 0;
  const double* k_scale = nullptr;   // [Hkv]
  const double* v_scale = nullptr;   // [Hkv]
};

// Element e of the K (or V) array, as a value of KV head g.
double kv_elem(const Problem& P, const void* base, int64_t e, int g, bool is_v) {
  if (P.fp8) {
    const bool use_v = (ORACLE_PLANT == 9) ? !is_v : is_v;
    return e4m3_to_double(static_cast<const uint8_t*>(base)[e]) *
           (use_v ? P.v_scale[g] : P.k_scale[g]);
  }
  return bf16_bits_to_double(static_cast<const uint16_t*>(base)[e]);
}

bool key_visible(const Problem& P, int64_t j, int64_t pos) {
  if (P.causal && j > pos) return false;
  if (ORACLE_PLANT == 5) {
    if (P.window > 0 && j < pos - P.window) return false;
    return true;
  }
  if (P.window > 0 && j <= pos - P.window) return false;
  return true;
}

// Logit of query row `tok` (global token index), head h, against key j of
// sequence b. Exact float64 dot product of the bf16 values.
double logit(const Problem& P, int b, int64_t tok, int h, int64_t j) {
  const int G = P.Hq / P.Hkv;
  const int kvh = (ORACLE_PLANT == 3) ? h % P.Hkv : h / G;
  const int64_t Lk = P.cu_k[b + 1] - P.cu_k[b];
  const uint16_t* qrow = P.q + (tok * P.Hq + h) * static_cast<int64_t>(P.d);
  const int64_t krow = (static_cast<int64_t>(P.Hkv) * P.cu_k[b] + kvh * Lk + j) * P.d;
  double s = 0.0;
  for (int c = 0; c < P.d; ++c)
    s += bf16_bits_to_double(qrow[c]) * kv_elem(P, P.k, krow + c, kvh, false);
  if (ORACLE_PLANT == 7) return s;
  return P.scale * s;
}

// Value row of key j for query head h: element c is kv_elem(P, P.v, row + c, g, true).
int64_t value_row(const Problem& P, int b, int h, int64_t j, int* g) {
  const int G = P.Hq / P.Hkv;
  const int kvh = (ORACLE_PLANT == 3) ? h % P.Hkv : h / G;
  const int64_t Lk = P.cu_k[b + 1] - P.cu_k[b];
  *g = kvh;
  return (static_cast<int64_t>(P.Hkv) * P.cu_k[b] + kvh * Lk + j) * P.d;
}

int sequence_of(const Problem& P, int64_t tok) {
  // cu_q is non-decreasing; linear scan is fine for an oracle.
  for (int b = 0; b < P.B; ++b)
    if (tok >= P.cu_q[b] && tok < P.cu_q[b + 1]) return b;
  return -1;
}

// The plain definition for one (token, head) row: materialise the full row of
// visible logits plus the sink column, then softmax and weight V.
void attend_row(const Problem& P, int64_t tok, int h, double* out, double* lse) {
  const int b = sequence_of(P, tok);
  const int64_t Lq = P.cu_q[b + 1] - P.cu_q[b];
  const int64_t Lk = P.cu_k[b + 1] - P.cu_k[b];
  const int64_t pos = (ORACLE_PLANT == 4) ? (tok - P.cu_q[b]) : Lk - Lq + (tok - P.cu_q[b]);

  std::vector<double> l;
  std::vector<int64_t> idx;
  l.reserve(static_cast<size_t>(Lk));
  idx.reserve(static_cast<size_t>(Lk));
  for (int64_t j = 0; j < Lk; ++j) {
    if (!key_visible(P, j, pos)) continue;
    l.push_back(logit(P, b, tok, h, j));
    idx.push_back(j);
  }
  double sink = P.sinks ? P.sinks[h] : kNegInf;
  if (ORACLE_PLANT == 2) sink *= P.scale;

  double M = sink;
  for (double x : l) M = (x > M) ? x : M;
  for (int c = 0; c < P.d; ++c) out[c] = 0.0;
  if (M == kNegInf) {  // nothing in the row at all
    *lse = kNegInf;
    return;
  }
  double Z = std::exp(sink - M);  // the sink column (exp(-inf) = 0 when absent)
  if (ORACLE_PLANT == 1) Z = 0.0;
  std::vector<double> acc(static_cast<size_t>(P.d), 0.0);
  for (size_t t = 0; t < l.size(); ++t) {
    const double w = std::exp(l[t] - M);
    Z += w;
    int g = 0;
    const int64_t vr = value_row(P, b, h, idx[t], &g);
    for (int c = 0; c < P.d; ++c) acc[c] += w * kv_elem(P, P.v, vr + c, g, true);
  }
  // The sink's value row is zero: it contributes to Z only.
  for (int c = 0; c < P.d; ++c) out[c] = acc[c] / Z;
  *lse = M + std::log(Z);
  if (ORACLE_PLANT == 8) *lse = M + std::log(Z - std::exp(sink - M));
}

// Partial state of one chunk [lo, hi) of the keys, without the sink:
// m = max visible logit in the chunk, dsum = sum exp(l - m), acc = sum exp(l - m) v.
// Empty chunk: (-inf, 0, 0).
void chunk_partial(const Problem& P, int64_t tok, int h, int64_t lo, int64_t hi,
                   double* acc, double* m_out, double* d_out) {
  const int b = sequence_of(P, tok);
  const int64_t Lq = P.cu_q[b + 1] - P.cu_q[b];
  const int64_t Lk = P.cu_k[b + 1] - P.cu_k[b];
  const int64_t pos = Lk - Lq + (tok - P.cu_q[b]);
  std::vector<double> l;
  std::vector<int64_t> idx;
  for (int64_t j = lo; j < hi && j < Lk; ++j) {
    if (!key_visible(P, j, pos)) continue;
    l.push_back(logit(P, b, tok, h, j));
    idx.push_back(j);
  }
  for (int c = 0; c < P.d; ++c) acc[c] = 0.0;
  double m = kNegInf;
  for (double x : l) m = (x > m) ? x : m;
  double dsum = 0.0;
  for (size_t t = 0; t < l.size(); ++t) {
    const double w = std::exp(l[t] - m);
    dsum += w;
    int g = 0;
    const int64_t vr = value_row(P, b, h, idx[t], &g);
    for (int c = 0; c < P.d; ++c) acc[c] += w * kv_elem(P, P.v, vr + c, g, true);
  }
  *m_out = m;
  *d_out = dsum;
}

int check_problem(const Problem& P) {
  if (!P.q || !P.k || !P.v || !P.cu_q || !P.cu_k) return 1;
  if (P.B < 0 || P.Hq <= 0 || P.Hkv <= 0 || P.d <= 0) return 1;
  if (P.Hq % P.Hkv != 0) return 1;
  if (P.window > 0 && !P.causal) return 1;
  if (P.fp8 && (!P.k_scale || !P.v_scale)) return 1;
  for (int b = 0; b < P.B; ++b) {
    if (P.cu_q[b + 1] < P.cu_q[b] || P.cu_k[b + 1] < P.cu_k[b]) return 1;
    if (P.cu_q[b + 1] - P.cu_q[b] > P.cu_k[b + 1] - P.cu_k[b]) return 1;
  }
  return 0;
}

}  // namespace

extern "C" {

// Number of OpenMP threads the oracle runs on (1 when built without OpenMP).
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

// Full-row oracle over selected rows.
//   rows: n_rows flat row ids, row = token * Hq + head; nullptr = every row of
//         [total_q, Hq] in order.
//   out:  [n_rows, d] float64; lse: [n_rows] float64.
// Returns 0, or 1 on an invalid problem.
}  // extern "C"

namespace {

int attend_rows(const Problem& P, int64_t n_rows, const int64_t* rows, double* out,
                double* lse) {
  if (check_problem(P)) return 1;
  const int B = P.B, Hq = P.Hq, d = P.d;
  const int32_t* cu_q = P.cu_q;
  const int64_t total_rows = static_cast<int64_t>(cu_q[B]) * Hq;
  if (!rows) n_rows = total_rows;
  for (int64_t r = 0; r < (rows ? n_rows : 0); ++r)
    if (rows[r] < 0 || rows[r] >= total_rows) return 1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    const int64_t row = rows ? rows[r] : r;
    attend_row(P, row / Hq, static_cast<int>(row % Hq), out + r * d, lse + r);
  }
  return 0;
}

}  // namespace

extern "C" {

int oracle_attend_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const double* sinks, const int32_t* cu_q, const int32_t* cu_k,
                       int B, int Hq, int Hkv, int d, double sm_scale, int causal,
                       int window, int64_t n_rows, const int64_t* rows, double* out,
                       double* lse) {
  Problem P{q, k, v, sinks, cu_q, cu_k, B, Hq, Hkv, d, sm_scale, causal, window};
  return attend_rows(P, n_rows, rows, out, lse);
}

// The same with K and V as e4m3 codes (uint8, same layout) and per-KV-head
// scales k_scale, v_scale [Hkv].
int oracle_attend_rows_fp8(const uint16_t* q, const uint8_t* k, const uint8_t* v,
                           const double* k_scale, const double* v_scale, const double* sinks,
                           const int32_t* cu_q, const int32_t* cu_k, int B, int Hq, int Hkv,
                           int d, double sm_scale, int causal, int window, int64_t n_rows,
                           const int64_t* rows, double* out, double* lse) {
  Problem P{q, k, v, sinks, cu_q, cu_k, B, Hq, Hkv, d, sm_scale, causal, window};
  P.fp8 = 1;
  P.k_scale = k_scale;
  P.v_scale = v_scale;
  return attend_rows(P, n_rows, rows, out, lse);
}

// Value of every e4m3 code (256 entries; NaN codes give NaN).
int oracle_e4m3_table(double* out) {
  for (int c = 0; c < 256; ++c) out[c] = e4m3_to_double(static_cast<uint8_t>(c));
  return 0;
}

// Per-chunk partials of the split-KV method, without the sink. Sequence b's
// keys are cut into num_splits chunks of c = 64 * ceil(Lk_b / (64 * num_splits))
// keys (ceil(Lk_b / num_splits) rounded up to whole 64-key tiles); chunk s
// covers [s*c, min((s+1)*c, Lk_b)) and may be empty.
//   part_acc: [total_q, Hq, S, d]; part_m, part_d: [total_q, Hq, S].
}  // extern "C"

namespace {

int split_partials(const Problem& P, int num_splits, double* part_acc, double* part_m,
                   double* part_d) {
  if (check_problem(P) || num_splits < 1) return 1;
  const int Hq = P.Hq, d = P.d;
  const int32_t* cu_q = P.cu_q;
  const int32_t* cu_k = P.cu_k;
  const int B = P.B;
  const int64_t total_rows = static_cast<int64_t>(cu_q[B]) * Hq;
  const int S = num_splits;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t row = 0; row < total_rows; ++row) {
    const int64_t tok = row / Hq;
    const int h = static_cast<int>(row % Hq);
    const int b = sequence_of(P, tok);
    const int64_t Lk = cu_k[b + 1] - cu_k[b];
    const int64_t c = 64 * ((Lk + 64 * S - 1) / (64 * S));
    for (int s = 0; s < S; ++s) {
      const int64_t lo = s * c;
      const int64_t hi = (s + 1) * c < Lk ? (s + 1) * c : Lk;
      const int64_t slot = row * S + s;
      chunk_partial(P, tok, h, lo, hi, part_acc + slot * d, part_m + slot, part_d + slot);
    }
  }
  return 0;
}

}  // namespace

extern "C" {

int oracle_split_partials(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          const int32_t* cu_q, const int32_t* cu_k, int B, int Hq,
                          int Hkv, int d, double sm_scale, int causal, int window,
                          int num_splits, double* part_acc, double* part_m,
                          double* part_d) {
  Problem P{q, k, v, nullptr, cu_q, cu_k, B, Hq, Hkv, d, sm_scale, causal, window};
  return split_partials(P, num_splits, part_acc, part_m, part_d);
}

int oracle_split_partials_fp8(const uint16_t* q, const uint8_t* k, const uint8_t* v,
                              const double* k_scale, const double* v_scale,
                              const int32_t* cu_q, const int32_t* cu_k, int B, int Hq,
                              int Hkv, int d, double sm_scale, int causal, int window,
                              int num_splits, double* part_acc, double* part_m,
                              double* part_d) {
  Problem P{q, k, v, nullptr, cu_q, cu_k, B, Hq, Hkv, d, sm_scale, causal, window};
  P.fp8 = 1;
  P.k_scale = k_scale;
  P.v_scale = v_scale;
  return split_partials(P, num_splits, part_acc, part_m, part_d);
}

// Partial state of explicit chunk bounds [lo, hi) for one row; used by the
// split-invariance pins, which enumerate every contiguous partition.
int oracle_chunk_partial(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* cu_q, const int32_t* cu_k, int B, int Hq,
                         int Hkv, int d, double sm_scale, int causal, int window,
                         int64_t row, int64_t lo, int64_t hi, double* acc, double* m,
                         double* dsum) {
  Problem P{q, k, v, nullptr, cu_q, cu_k, B, Hq, Hkv, d, sm_scale, causal, window};
  if (check_problem(P)) return 1;
  if (row < 0 || row >= static_cast<int64_t>(cu_q[B]) * Hq || lo < 0 || hi < lo) return 1;
  chunk_partial(P, row / Hq, static_cast<int>(row % Hq), lo, hi, acc, m, dsum);
  return 0;
}

// Fold of S partials per row with the sink counted once: the running state
// starts at m = s_h, d = 1 (the sink's own term exp(s_h - s_h)), acc = 0 --
// or m = -inf, d = 0 when there is no sink -- and each partial (m_s, d_s,
// acc_s) is merged with the usual rescale to the larger maximum.
//   part_acc: [rows, Hq, S, d]; part_m, part_d: [rows, Hq, S];
//   sinks: [Hq] or nullptr; out: [rows, Hq, d]; lse: [rows, Hq].
int oracle_merge(const double* part_acc, const double* part_m, const double* part_d,
                 const double* sinks, int64_t rows, int Hq, int d, int num_splits,
                 double* out, double* lse) {
  if (!part_acc || !part_m || !part_d || !out || !lse || rows < 0 || Hq <= 0 || d <= 0 ||
      num_splits < 1)
    return 1;
  const int S = num_splits;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows * Hq; ++r) {
    const int h = static_cast<int>(r % Hq);
    const double sink = sinks ? sinks[h] : kNegInf;
    double m = sink;
    double dsum = (sink == kNegInf) ? 0.0 : 1.0;
    std::vector<double> acc(static_cast<size_t>(d), 0.0);
    for (int s = 0; s < S; ++s) {
      const int64_t slot = r * S + s;
      const double ms = part_m[slot];
      const double ds = part_d[slot];
      if (ms == kNegInf) continue;  // empty chunk: nothing to fold
      const double mn = ms > m ? ms : m;
      const double a_old = (m == kNegInf) ? 0.0 : std::exp(m - mn);
      const double a_new = std::exp(ms - mn);
      dsum = dsum * a_old + ds * a_new;
      if (ORACLE_PLANT == 6 && s > 0 && sink != kNegInf) dsum += std::exp(sink - mn);
      for (int c = 0; c < d; ++c) acc[c] = acc[c] * a_old + part_acc[slot * d + c] * a_new;
      m = mn;
    }
    if (dsum == 0.0) {
      for (int c = 0; c < d; ++c) out[r * d + c] = 0.0;
      lse[r] = kNegInf;
    } else {
      for (int c = 0; c < d; ++c) out[r * d + c] = acc[c] / dsum;
      lse[r] = m + std::log(dsum);
    }
  }
  return 0;
}

}  // extern "C"
