// osattn_ref.cpp - fp64 CPU oracle for the attention forward pass and its
// gradients.
//
// TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
// benchmark's CPU-baseline leg load this library.  The product (libosattn)
// shares no code, header, table or helper with it, and it never calls into
// the product.
//
// Sources (the three web pages on online softmax; cited by title + section):
//   [Ch6]  "CUDA 算子工程：手写 FlashAttention v2 之路", chapter 6
//          "Softmax 与 Online Softmax" (yangyitao.com).  This page decides
//          what the method computes.
//   [XXQK] m.xxqk.cn/news/563265, the article on why softmax parallelises
//          and how FlashAttention uses online softmax (sections 1-7).
//
// What the oracle computes, for every query row i of every (b, h):
//   J   = { j : j < clamp(key_len[b], 0, Nkv)  and  (not causal or j <= i) }
//   s_j = scale * sum_k Q[i,k] K[j,k]                 ([XXQK] §1.1 steps 1-2,
//                                                       scale then mask)
//   J empty  ->  O[i,:] = 0, LSE = -inf               (fully masked row: the
//                                                       library's contract;
//                                                       [Ch6] §6.7.3 leaves
//                                                       it undefined)
//   else the three-pass safe softmax of [Ch6] §6.2:
//     pass 1  m = max_j s_j
//     pass 2  l = sum_j exp(s_j - m)
//     pass 3  p_j = exp(s_j - m) / l,  O[i,:] = sum_j p_j V[j,:]
//   LSE = m + log(l)                                   ([Ch6] §6.5)
// in double precision throughout, on the exact values the GPU reads (bf16 /
// fp32 inputs are widened to double without rounding).
//
// The scalar helpers below restate the other pieces of [Ch6] so that tests
// can pin them independently: the unguarded two-pass definition (§6.1), the
// one-element-at-a-time online recurrence (§6.3.1) with the -inf guard of
// §6.4, the (m, l) combine (§6.4.1), and the blocked attention loop of §6.6
// in both its forms (local max + beta, and the variant that exponentiates
// against the new running max directly).  Parity of everything here is
// pinned by tests/test_oracle.py (worked example, closed forms, library
// routines, brute force); no function here is "parity unpinned".

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

const double kNegInf = -std::numeric_limits<double>::infinity();

// Element formats the oracle can read.  bf16 is the top half of an IEEE
// binary32, so widening is a shift; fp16 is IEEE binary16, decoded from its
// fields below; every bf16/fp16/fp32 value is exact in double.
enum RefDtype { REF_BF16 = 0, REF_FP32 = 1, REF_FP64 = 2, REF_FP16 = 3 };

// IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
// bits.  Exponent 0 holds zero and the subnormals f * 2^-24; exponent 31
// holds infinity (f = 0) and NaN.
inline double decode_binary16(uint16_t h) {
  const int sign = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
  double mag;
  if (e == 0)
    mag = std::ldexp(static_cast<double>(f), -24);
  else if (e == 31)
    mag = f == 0 ? std::numeric_limits<double>::infinity()
                 : std::numeric_limits<double>::quiet_NaN();
  else
    mag = std::ldexp(static_cast<double>(1024 + f), e - 25);
  return sign ? -mag : mag;
}

inline double load_elem(const void* base, int dtype, int64_t idx) {
  if (dtype == REF_BF16) {
    uint16_t h;
    std::memcpy(&h, static_cast<const uint16_t*>(base) + idx, 2);
    uint32_t u = static_cast<uint32_t>(h) << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return static_cast<double>(f);
  }
  if (dtype == REF_FP16) {
    uint16_t h;
    std::memcpy(&h, static_cast<const uint16_t*>(base) + idx, 2);
    return decode_binary16(h);
  }
  if (dtype == REF_FP32) {
    float f;
    std::memcpy(&f, static_cast<const float*>(base) + idx, 4);
    return static_cast<double>(f);
  }
  double v;
  std::memcpy(&v, static_cast<const double*>(base) + idx, 8);
  return v;
}

struct AttnProblem {
  const void* Q;
  const void* K;
  const void* V;
  int dtype;
  int B, H, Nq, Nkv, d;
  double scale;
  int causal;
  const int32_t* key_len;  // host array [B] or null
};

// Number of keys the batch entry may see: key_len clamped to [0, Nkv].
int visible_keys(const AttnProblem& p, int b) {
  if (!p.key_len) return p.Nkv;
  int kl = p.key_len[b];
  if (kl < 0) kl = 0;
  if (kl > p.Nkv) kl = p.Nkv;
  return kl;
}

// Computes one output row by the definition above.  `s` is scratch of Nkv
// doubles.  flat_row = (b*H + h)*Nq + i.
void attention_row(const AttnProblem& p, int64_t flat_row, double* o_row,
                   double* lse, std::vector<double>& s) {
  const int64_t bh = flat_row / p.Nq;
  const int i = static_cast<int>(flat_row % p.Nq);
  const int b = static_cast<int>(bh / p.H);
  const int d = p.d;
  int jend = visible_keys(p, b);
  if (p.causal) jend = std::min(jend, i + 1);  // j <= i
  for (int c = 0; c < d; ++c) o_row[c] = 0.0;
  if (jend <= 0) {  // J is empty
    *lse = kNegInf;
    return;
  }
  const int64_t qoff = flat_row * d;
  const int64_t kvoff = bh * static_cast<int64_t>(p.Nkv) * d;
  // logits s_j = scale * <q_i, k_j>
  for (int j = 0; j < jend; ++j) {
    double acc = 0.0;
    const int64_t koff = kvoff + static_cast<int64_t>(j) * d;
    for (int k = 0; k < d; ++k)
      acc += load_elem(p.Q, p.dtype, qoff + k) * load_elem(p.K, p.dtype, koff + k);
    s[j] = p.scale * acc;
  }
  // pass 1: row max
  double m = kNegInf;
  for (int j = 0; j < jend; ++j) m = std::max(m, s[j]);
  // pass 2: denominator
  double l = 0.0;
  for (int j = 0; j < jend; ++j) l += std::exp(s[j] - m);
  // pass 3: probabilities and the weighted sum of V rows
  for (int j = 0; j < jend; ++j) {
    const double pj = std::exp(s[j] - m) / l;
    const int64_t voff = kvoff + static_cast<int64_t>(j) * d;
    for (int c = 0; c < d; ++c) o_row[c] += pj * load_elem(p.V, p.dtype, voff + c);
  }
  *lse = m + std::log(l);
}

int check_problem(const AttnProblem& p) {
  if (!p.Q || !p.K || !p.V) return 1;
  if (p.B < 1 || p.H < 1 || p.Nq < 1 || p.Nkv < 1 || p.d < 1) return 1;
  if (p.dtype < REF_BF16 || p.dtype > REF_FP16) return 1;
  return 0;
}

template <class F>
void parallel_rows(int64_t nrows, int nthreads, F&& body) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
  if (nthreads <= 0) nthreads = 1;
  if (nthreads > nrows) nthreads = static_cast<int>(std::max<int64_t>(nrows, 1));
  std::atomic<int64_t> next(0);
  const int64_t chunk = 16;
  auto worker = [&]() {
    for (;;) {
      int64_t r0 = next.fetch_add(chunk);
      if (r0 >= nrows) break;
      int64_t r1 = std::min(nrows, r0 + chunk);
      for (int64_t r = r0; r < r1; ++r) body(r);
    }
  };
  std::vector<std::thread> pool;
  for (int t = 1; t < nthreads; ++t) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

int osattn_ref_version(void) { return 1; }

// [Ch6] §6.1: the direct two-pass definition e^{x_i} / sum_j e^{x_j}, with no
// max subtraction (overflows for large inputs; used only on small ones).
int osattn_ref_softmax_naive(const double* x, int n, double* y) {
  if (!x || !y || n < 1) return 1;
  double sum = 0.0;
  for (int i = 0; i < n; ++i) sum += std::exp(x[i]);
  for (int i = 0; i < n; ++i) y[i] = std::exp(x[i]) / sum;
  return 0;
}

// [Ch6] §6.2: three-pass safe softmax.  Also returns m and l = sum e^{x-m}.
// A row of only -inf has no defined softmax; it yields y = 0, m = -inf, l = 0.
int osattn_ref_softmax_safe(const double* x, int n, double* y, double* m_out,
                            double* l_out) {
  if (!x || n < 1) return 1;
  double m = kNegInf;
  for (int i = 0; i < n; ++i) m = std::max(m, x[i]);
  double l = 0.0;
  if (m != kNegInf)
    for (int i = 0; i < n; ++i) l += std::exp(x[i] - m);
  if (y)
    for (int i = 0; i < n; ++i) y[i] = (m == kNegInf) ? 0.0 : std::exp(x[i] - m) / l;
  if (m_out) *m_out = m;
  if (l_out) *l_out = l;
  return 0;
}

// [Ch6] §6.3.1: the online recurrence from (m_0, l_0) = (-inf, 0),
//   m_{n+1} = max(m_n, x_{n+1}),  l_{n+1} = l_n e^{m_n - m_{n+1}} + e^{x_{n+1} - m_{n+1}},
// one element at a time, skipping the update while the running max is still
// -inf (the guard of §6.4).  l_trace (optional) receives l_1 .. l_n.
int osattn_ref_online_stats(const double* x, int n, double* m_out, double* l_out,
                            double* l_trace) {
  if (!x || n < 0 || !m_out || !l_out) return 1;
  double m = kNegInf, l = 0.0;
  for (int t = 0; t < n; ++t) {
    const double m_new = std::max(m, x[t]);
    if (m_new != kNegInf) {
      l = l * std::exp(m - m_new) + std::exp(x[t] - m_new);
      m = m_new;
    }
    if (l_trace) l_trace[t] = l;
  }
  *m_out = m;
  *l_out = l;
  return 0;
}

// [Ch6] §6.4.1: combine((m1,l1),(m2,l2)) = (M, l1 e^{m1-M} + l2 e^{m2-M}),
// M = max(m1, m2); two empty states (-inf, 0) give the empty state back.
void osattn_ref_combine(double m1, double l1, double m2, double l2, double* m_out,
                        double* l_out) {
  const double M = std::max(m1, m2);
  if (M == kNegInf) {
    *m_out = kNegInf;
    *l_out = 0.0;
    return;
  }
  *m_out = M;
  *l_out = l1 * std::exp(m1 - M) + l2 * std::exp(m2 - M);
}

// [Ch6] §6.5: LSE = m + log l (natural log); -inf for the empty state.
double osattn_ref_lse(double m, double l) {
  if (m == kNegInf || l == 0.0) return kNegInf;
  return m + std::log(l);
}

// Row softmax of a [rows, N] matrix by the three-pass safe softmax of
// [Ch6] §6.2, row by row: y = e^{x - m} / l with m = max x, l = sum e^{x - m},
// and lse = m + log l ([Ch6] §6.5).  A row of only -inf (all masked) has no
// defined softmax; it yields y = 0 and lse = -inf.  x is bf16 bits, fp32,
// fp64 or fp16 bits (dtype 0/1/2/3); y and lse are double; lse may be null.
int osattn_ref_softmax_rows(const void* x, int dtype, int64_t rows, int N, double* y,
                            double* lse, int nthreads) {
  if (!x || !y || rows < 1 || N < 1 || dtype < REF_BF16 || dtype > REF_FP16) return 1;
  parallel_rows(rows, nthreads, [&](int64_t r) {
    const int64_t base = r * N;
    double m = kNegInf;
    for (int i = 0; i < N; ++i) m = std::max(m, load_elem(x, dtype, base + i));
    double l = 0.0;
    if (m != kNegInf)
      for (int i = 0; i < N; ++i) l += std::exp(load_elem(x, dtype, base + i) - m);
    for (int i = 0; i < N; ++i)
      y[base + i] = (m == kNegInf) ? 0.0 : std::exp(load_elem(x, dtype, base + i) - m) / l;
    if (lse) lse[r] = (m == kNegInf) ? kNegInf : m + std::log(l);
  });
  return 0;
}

// Attention forward by the definition in the file header.
//   Q: [B,H,Nq,d], K/V: [B,H,Nkv,d], contiguous, element format `dtype`
//   (0 bf16 bits, 1 fp32, 2 fp64, 3 fp16 bits).  key_len: host int32 [B] or null.
//   rows == null: every row; O receives [B,H,Nq,d], LSE [B,H,Nq].
//   rows != null: only the nrows flat row indices (b*H+h)*Nq+i listed there;
//   O receives [nrows,d] and LSE [nrows], in list order.
//   nthreads <= 0 uses every hardware thread.
// Returns 0, or 1 for an invalid argument (nothing written).
int osattn_ref_attention_fwd(const void* Q, const void* K, const void* V, int dtype,
                             double* O, double* LSE, int B, int H, int Nq, int Nkv,
                             int d, double scale, int causal, const int32_t* key_len,
                             const int64_t* rows, int64_t nrows, int nthreads) {
  AttnProblem p{Q, K, V, dtype, B, H, Nq, Nkv, d, scale, causal, key_len};
  if (check_problem(p) || !O || !LSE) return 1;
  const int64_t total = static_cast<int64_t>(B) * H * Nq;
  if (rows) {
    if (nrows < 0) return 1;
    for (int64_t r = 0; r < nrows; ++r)
      if (rows[r] < 0 || rows[r] >= total) return 1;
  } else {
    nrows = total;
  }
  parallel_rows(nrows, nthreads, [&](int64_t r) {
    thread_local std::vector<double> s;
    if (static_cast<int>(s.size()) < Nkv) s.resize(Nkv);
    const int64_t flat = rows ? rows[r] : r;
    attention_row(p, flat, O + r * d, LSE + r, s);
  });
  return 0;
}

// [Ch6] §6.6 / [XXQK] §4.1: the blocked ("FlashAttention") loop over key
// blocks of `block` keys for every row, carrying (m, l, O).
//   form 0: the §6.6 listing's form - a block-local max m_b, P = e^{S - m_b},
//           l_b = rowsum P, then alpha = e^{m - m_new}, beta = e^{m_b - m_new},
//           O = O alpha + beta P V_b, l = l alpha + beta l_b.
//   form 1: the variant §6.6 notes as equivalent (and [XXQK] §4.1 prints):
//           P = e^{S - m_new} directly, O = O alpha + P V_b, l = l alpha + rowsum P.
// Masked keys (outside J) are skipped.  Blocks with no visible key leave the
// state untouched (the -inf guard).  At the end O /= l and LSE = m + log l;
// an empty J gives O = 0, LSE = -inf.  Same arguments/layout as
// osattn_ref_attention_fwd (all rows).
int osattn_ref_attention_blocked(const void* Q, const void* K, const void* V, int dtype,
                                 double* O, double* LSE, int B, int H, int Nq, int Nkv,
                                 int d, double scale, int causal, const int32_t* key_len,
                                 int block, int form, int nthreads) {
  AttnProblem p{Q, K, V, dtype, B, H, Nq, Nkv, d, scale, causal, key_len};
  if (check_problem(p) || !O || !LSE || block < 1 || (form != 0 && form != 1)) return 1;
  const int64_t total = static_cast<int64_t>(B) * H * Nq;
  parallel_rows(total, nthreads, [&](int64_t flat) {
    const int64_t bh = flat / Nq;
    const int i = static_cast<int>(flat % Nq);
    const int b = static_cast<int>(bh / H);
    int jend = visible_keys(p, b);
    if (causal) jend = std::min(jend, i + 1);
    double* o = O + flat * d;
    std::vector<double> sb(block), pv(d);
    double m = kNegInf, l = 0.0;
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    for (int j0 = 0; j0 < jend; j0 += block) {
      const int nb = std::min(block, jend - j0);
      for (int t = 0; t < nb; ++t) {
        double acc = 0.0;
        for (int k = 0; k < d; ++k)
          acc += load_elem(Q, dtype, flat * d + k) *
                 load_elem(K, dtype, (bh * Nkv + j0 + t) * d + k);
        sb[t] = scale * acc;
      }
      double m_b = kNegInf;
      for (int t = 0; t < nb; ++t) m_b = std::max(m_b, sb[t]);
      const double m_new = std::max(m, m_b);
      if (m_new == kNegInf) continue;
      const double alpha = std::exp(m - m_new);
      const double ref = (form == 0) ? m_b : m_new;
      double l_b = 0.0;
      for (int c = 0; c < d; ++c) pv[c] = 0.0;
      for (int t = 0; t < nb; ++t) {
        const double pt = std::exp(sb[t] - ref);
        l_b += pt;
        for (int c = 0; c < d; ++c) pv[c] += pt * load_elem(V, dtype, (bh * Nkv + j0 + t) * d + c);
      }
      const double beta = (form == 0) ? std::exp(m_b - m_new) : 1.0;
      for (int c = 0; c < d; ++c) o[c] = o[c] * alpha + beta * pv[c];
      l = l * alpha + beta * l_b;
      m = m_new;
    }
    if (l > 0.0) {
      for (int c = 0; c < d; ++c) o[c] /= l;
      LSE[flat] = m + std::log(l);
    } else {
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      LSE[flat] = kNegInf;
    }
  });
  return 0;
}

// Gradients of the forward pass above for an upstream gradient dO (one
// array shaped like O, element format `dtype`).  [Ch6] §6.5 keeps only LSE
// per row from the forward pass so that the backward pass can rebuild the
// probabilities, and [XXQK] §5.2 (last paragraph) recomputes S there; the
// derivatives are the chain rule applied to the definition in this file's
// header (nothing else is assumed):
//   P_ij  = exp(s_ij - LSE_i) for j in J_i, else 0
//   dV_j  = sum_i P_ij dO_i
//   dP_ij = <dO_i, V_j>
//   D_i   = sum_j P_ij dP_ij                 (equals <dO_i, O_i>)
//   dS_ij = P_ij (dP_ij - D_i)               (softmax Jacobian)
//   dQ_i  = scale * sum_j dS_ij K_j
//   dK_j  = scale * sum_i dS_ij Q_i
// Two passes, each parallel over rows so that whole heads of long sequences
// can be checked:
//   pass 1, one task per query row i: s_ij, LSE_i, P_ij, dP_ij, D_i and dQ_i;
//           LSE_i and D_i are kept;
//   pass 2, one task per key row j: for every query row i whose J_i holds j,
//           s_ij, P_ij = exp(s_ij - LSE_i), dP_ij and dS_ij again, summed
//           into dK_j and dV_j.
// A row with J empty contributes nothing.  dQ [B,H,Nq,d], dK and dV
// [B,H,Nkv,d], all double.  Returns 0, or 1 for an invalid argument
// (nothing written).
int osattn_ref_attention_bwd(const void* Q, const void* K, const void* V, const void* dO,
                             int dtype, double* dQ, double* dK, double* dV, int B, int H, int Nq,
                             int Nkv, int d, double scale, int causal, const int32_t* key_len,
                             int nthreads) {
  AttnProblem p{Q, K, V, dtype, B, H, Nq, Nkv, d, scale, causal, key_len};
  if (check_problem(p) || !dO || !dQ || !dK || !dV) return 1;
  // The inputs widened to double once (exact, as in load_elem).
  const int64_t nq = static_cast<int64_t>(B) * H * Nq * d;
  const int64_t nk = static_cast<int64_t>(B) * H * Nkv * d;
  std::vector<double> q(nq), g(nq), k(nk), v(nk);
  parallel_rows(static_cast<int64_t>(B) * H, nthreads, [&](int64_t bh) {
    for (int64_t e = bh * Nq * d; e < (bh + 1) * Nq * d; ++e) {
      q[e] = load_elem(Q, dtype, e);
      g[e] = load_elem(dO, dtype, e);
    }
    for (int64_t e = bh * Nkv * d; e < (bh + 1) * Nkv * d; ++e) {
      k[e] = load_elem(K, dtype, e);
      v[e] = load_elem(V, dtype, e);
    }
  });
  auto dot = [d](const double* a, const double* b) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += a[c] * b[c];
    return acc;
  };
  std::vector<double> row_lse(static_cast<int64_t>(B) * H * Nq), row_D(row_lse.size());

  // pass 1: query rows
  parallel_rows(static_cast<int64_t>(B) * H * Nq, nthreads, [&](int64_t r) {
    const int64_t bh = r / Nq;
    const int i = static_cast<int>(r % Nq);
    const int b = static_cast<int>(bh / H);
    const double* qi = q.data() + r * d;
    const double* gi = g.data() + r * d;
    const double* kb = k.data() + bh * Nkv * d;
    const double* vb = v.data() + bh * Nkv * d;
    double* dq = dQ + r * d;
    for (int c = 0; c < d; ++c) dq[c] = 0.0;
    int jend = visible_keys(p, b);
    if (causal) jend = std::min(jend, i + 1);
    row_lse[r] = kNegInf;
    row_D[r] = 0.0;
    if (jend <= 0) return;
    thread_local std::vector<double> s, pr, dp;
    s.resize(Nkv);
    pr.resize(Nkv);
    dp.resize(Nkv);
    for (int j = 0; j < jend; ++j) s[j] = scale * dot(qi, kb + static_cast<int64_t>(j) * d);
    double m = kNegInf;
    for (int j = 0; j < jend; ++j) m = std::max(m, s[j]);
    double den = 0.0;
    for (int j = 0; j < jend; ++j) den += std::exp(s[j] - m);
    const double lse = m + std::log(den);
    double D = 0.0;
    for (int j = 0; j < jend; ++j) {
      pr[j] = std::exp(s[j] - lse);
      dp[j] = dot(gi, vb + static_cast<int64_t>(j) * d);
      D += pr[j] * dp[j];
    }
    for (int j = 0; j < jend; ++j) {
      const double ds = pr[j] * (dp[j] - D);
      const double* kj = kb + static_cast<int64_t>(j) * d;
      for (int c = 0; c < d; ++c) dq[c] += scale * ds * kj[c];
    }
    row_lse[r] = lse;
    row_D[r] = D;
  });

  // pass 2: key rows
  parallel_rows(static_cast<int64_t>(B) * H * Nkv, nthreads, [&](int64_t r) {
    const int64_t bh = r / Nkv;
    const int j = static_cast<int>(r % Nkv);
    const int b = static_cast<int>(bh / H);
    const double* kj = k.data() + r * d;
    const double* vj = v.data() + r * d;
    double* dk = dK + r * d;
    double* dv = dV + r * d;
    for (int c = 0; c < d; ++c) {
      dk[c] = 0.0;
      dv[c] = 0.0;
    }
    if (j >= visible_keys(p, b)) return;  // no row sees key j
    const int i0 = causal ? j : 0;        // rows i with j <= i
    for (int i = i0; i < Nq; ++i) {
      const int64_t qr = bh * Nq + i;
      const double* qi = q.data() + qr * d;
      const double* gi = g.data() + qr * d;
      const double pij = std::exp(scale * dot(qi, kj) - row_lse[qr]);
      const double dsij = pij * (dot(gi, vj) - row_D[qr]);
      for (int c = 0; c < d; ++c) {
        dk[c] += scale * dsij * qi[c];
        dv[c] += pij * gi[c];
      }
    }
  });
  return 0;
}

}  // extern "C"
