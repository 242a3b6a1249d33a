// fp64 CPU oracle for scaled-dot-product attention forward.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg load this library.  It shares no code, header,
// table or helper with the CUDA library, and neither side includes the other.
//
// What it computes (one query row at a time, two passes, no blocking):
//
//   kvh  = h / (Hq / Hkv)                         GQA: each KV head serves
//                                                 Hq/Hkv consecutive query heads
//                                                 (page "Xe2 ESIMD Flash Attention",
//                                                 section "GQA layout")
//   s_j  = scale * sum_d Q[b,i,h,d] K[b,j,kvh,d] + mask[b,i,j]
//   s_j  = -inf  when causal and j > i            (key j visible iff j <= i)
//   M    = max_j s_j
//   M == -inf  ->  O[b,i,h,:] = 0, LSE = -inf     (fully masked row; the page
//                                                 "Xe2 ESIMD Flash Attention",
//                                                 section "Correctness testing",
//                                                 names the all -inf row as the
//                                                 usual NaN source)
//   p_j  = exp(s_j - M),  l = sum_j p_j
//   O    = sum_j p_j V[b,j,kvh,:] / l,   LSE = M + ln l
//
// This is the plain definition softmax(scale * Q K^T + mask) V that the page
// "Xe SDPA Forward Mainloop" (section "Full simplified pseudocode", step 4
// "Online softmax") reaches block by block: the online update there is an exact
// rewrite of this two-pass form, so the kernels differ from it only by rounding.
// The mask is added after scaling and is not itself scaled; the natural
// exponential is used (exp2 with scale*log2(e) folded in, as in section
// "Arguments / params", is the same function).
//
// Layouts (contiguous, fp64):
//   q    [B, Sq, Hq, D]        k [B, Sk, Hkv, D]      v [B, Sk, Hkv, Dv]
//   mask [B, Sq, Sk] or null   o [B, Sq, Hq, Dv]      lse [B, Hq, Sq]
// When `rows` (nrows triples b, h, i) is given, only those rows are computed and
// o is [nrows, Dv], lse is [nrows].

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

namespace {

struct Problem {
  const double* q;
  const double* k;
  const double* v;
  const double* mask;
  int64_t B, Hq, Hkv, Sq, Sk, D, Dv;
  double scale;
  int causal;
};

// One query row (b, h, i): writes Dv outputs and the log-sum-exp.
void attend_row(const Problem& P, int64_t b, int64_t h, int64_t i, double* o_row, double* lse_out,
                std::vector<double>& s, std::vector<double>& acc) {
  const double neg_inf = -std::numeric_limits<double>::infinity();
  const int64_t group = P.Hq / P.Hkv;
  const int64_t kvh = h / group;
  const double* qrow = P.q + ((b * P.Sq + i) * P.Hq + h) * P.D;

  // pass 1: scores and their maximum
  double M = neg_inf;
  for (int64_t j = 0; j < P.Sk; ++j) {
    if (P.causal && j > i) {
      s[j] = neg_inf;
      continue;
    }
    const double* krow = P.k + ((b * P.Sk + j) * P.Hkv + kvh) * P.D;
    double dot = 0.0;
    for (int64_t d = 0; d < P.D; ++d) dot += qrow[d] * krow[d];
    double sj = P.scale * dot;
    if (P.mask) sj += P.mask[(b * P.Sq + i) * P.Sk + j];
    s[j] = sj;
    if (sj > M) M = sj;
  }

  if (M == neg_inf) {
    for (int64_t c = 0; c < P.Dv; ++c) o_row[c] = 0.0;
    *lse_out = neg_inf;
    return;
  }

  // pass 2: exponentials, their sum, and the weighted sum of V rows
  double l = 0.0;
  std::fill(acc.begin(), acc.end(), 0.0);
  for (int64_t j = 0; j < P.Sk; ++j) {
    if (s[j] == neg_inf) continue;  // exp(-inf) = 0 contributes nothing
    const double p = std::exp(s[j] - M);
    l += p;
    const double* vrow = P.v + ((b * P.Sk + j) * P.Hkv + kvh) * P.Dv;
    for (int64_t c = 0; c < P.Dv; ++c) acc[c] += p * vrow[c];
  }
  for (int64_t c = 0; c < P.Dv; ++c) o_row[c] = acc[c] / l;
  *lse_out = M + std::log(l);
}

int valid(const Problem& P) {
  if (!P.q || !P.k || !P.v) return 0;
  if (P.B < 0 || P.Sq < 0 || P.Sk < 0) return 0;
  if (P.Hq <= 0 || P.Hkv <= 0 || P.D <= 0 || P.Dv <= 0) return 0;
  if (P.Hq % P.Hkv != 0) return 0;
  return 1;
}

template <class F>
void parallel_rows(int64_t n, int nthreads, F&& body) {
  if (nthreads <= 0) nthreads = (int)std::max(1u, std::thread::hardware_concurrency());
  if (n < 2 * nthreads) nthreads = (int)std::max<int64_t>(1, std::min<int64_t>(nthreads, n));
  if (nthreads == 1) {
    body(0, n);
    return;
  }
  std::vector<std::thread> pool;
  const int64_t chunk = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    const int64_t lo = t * chunk, hi = std::min(n, lo + chunk);
    if (lo >= hi) break;
    pool.emplace_back([&, lo, hi] { body(lo, hi); });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Returns 0 on success, 1 on invalid arguments.
int oracle_sdpa_fwd(const double* q, const double* k, const double* v, const double* mask, double* o,
                    double* lse, int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t D,
                    int64_t Dv, double scale, int causal, const int64_t* rows, int64_t nrows, int nthreads) {
  Problem P{q, k, v, mask, B, Hq, Hkv, Sq, Sk, D, Dv, scale, causal};
  if (!valid(P) || !o || !lse) return 1;
  const int64_t n = rows ? nrows : B * Hq * Sq;
  if (rows) {
    for (int64_t r = 0; r < nrows; ++r) {
      const int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
      if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Sq) return 1;
    }
  }
  parallel_rows(n, nthreads, [&](int64_t lo, int64_t hi) {
    std::vector<double> s((size_t)std::max<int64_t>(Sk, 1)), acc((size_t)Dv);
    for (int64_t r = lo; r < hi; ++r) {
      int64_t b, h, i;
      double *orow, *lrow;
      if (rows) {
        b = rows[3 * r];
        h = rows[3 * r + 1];
        i = rows[3 * r + 2];
        orow = o + r * Dv;
        lrow = lse + r;
      } else {
        // r enumerates (b, h, i) with i fastest
        i = r % Sq;
        h = (r / Sq) % Hq;
        b = r / (Sq * Hq);
        orow = o + ((b * Sq + i) * Hq + h) * Dv;
        lrow = lse + (b * Hq + h) * Sq + i;
      }
      attend_row(P, b, h, i, orow, lrow, s, acc);
    }
  });
  return 0;
}

// Decode: one query token per (b, h) against the first kv_len[b] rows of a padded
// cache.  It is the same definition with Sq = 1, Sk = kv_len[b], no causal rule.
//   q [B, Hq, D]   k [B, max_kv, Hkv, D]   v [B, max_kv, Hkv, Dv]
//   o [B, Hq, Dv]  lse [B, Hq]
int oracle_sdpa_decode(const double* q, const double* k, const double* v, const int32_t* kv_len, double* o,
                       double* lse, int64_t B, int64_t Hq, int64_t Hkv, int64_t max_kv, int64_t D, int64_t Dv,
                       double scale, int nthreads) {
  if (!q || !k || !v || !kv_len || !o || !lse) return 1;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Dv <= 0 || Hq % Hkv != 0) return 1;
  for (int64_t b = 0; b < B; ++b)
    if (kv_len[b] < 0 || kv_len[b] > max_kv) return 1;
  parallel_rows(B * Hq, nthreads, [&](int64_t lo, int64_t hi) {
    std::vector<double> s((size_t)std::max<int64_t>(max_kv, 1)), acc((size_t)Dv);
    for (int64_t r = lo; r < hi; ++r) {
      const int64_t b = r / Hq, h = r % Hq;
      // view batch b as a single-batch problem with Sq = 1 and Sk = kv_len[b]
      Problem P{q + b * Hq * D, k + b * max_kv * Hkv * D, v + b * max_kv * Hkv * Dv, nullptr, 1, Hq, Hkv, 1,
                (int64_t)kv_len[b], D, Dv, scale, 0};
      attend_row(P, 0, h, 0, o + (b * Hq + h) * Dv, lse + b * Hq + h, s, acc);
    }
  });
  return 0;
}

}  // extern "C"
