// jvp_oracle.cpp -- float64 CPU oracle for attention forward + JVP (and its
// reverse mode).  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
// benchmark's CPU-baseline leg use it; the GPU library never links or calls it,
// and it shares no code, header or table with the GPU path.
//
// What it computes (the "JVP Flash Attention" project page, Description and
// Usage sections: a drop-in for scaled_dot_product_attention(q, k, v,
// attn_mask) whose `fwd_dual` returns the primal output together with its
// forward-mode tangent for use inside torch.func.jvp):
//
//   S  = scale * Q K^T + M          (M: additive bias, or -inf for excluded keys)
//   P  = softmax_row(S)             (over the keys a row keeps)
//   O  = P V
//   tO = d/de [ O(Q + e dQ, K + e dK, V + e dV) ] at e = 0
//
// The method reaches this exactly (up to rounding order), so the oracle is the
// plain definition evaluated with explicit dual numbers x + e*t (e^2 = 0).  It
// materialises every score of a row, never blocks, fuses or reorders beyond the
// definition, and accumulates in natural key order.  The log-sum-exp side
// output is lse = log sum_j exp(S_ij) (natural log); mu is the tangent of lse,
// which equals rowsum(P * dS).
//
// Readings where the pages are silent (each is listed in the design notes):
//   * boolean mask: nonzero = the key takes part (SDPA's attn_mask polarity);
//   * additive mask: added after scaling; it carries no tangent; an entry of
//     -inf excludes the key;
//   * causal: top-left aligned, key j kept iff j <= i;
//   * a row with no kept key: O = tO = 0, lse = -inf, mu = 0.
//
// Parity status: every function here is pinned by the CPU tests (finite
// differences, exact special cases, invariants and a library cross-check).

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------- dual numbers
struct Dual {
  double v;  // primal value
  double t;  // tangent (coefficient of e, e^2 = 0)
};
inline Dual operator+(Dual a, Dual b) { return {a.v + b.v, a.t + b.t}; }
inline Dual operator-(Dual a, Dual b) { return {a.v - b.v, a.t - b.t}; }
inline Dual operator*(Dual a, Dual b) { return {a.v * b.v, a.v * b.t + a.t * b.v}; }
inline Dual operator/(Dual a, Dual b) {
  return {a.v / b.v, (a.t * b.v - a.v * b.t) / (b.v * b.v)};
}
inline Dual dexp(Dual a) {
  const double e = std::exp(a.v);
  return {e, e * a.t};
}
inline Dual dlog(Dual a) { return {std::log(a.v), a.t / a.v}; }
inline Dual constant(double c) { return {c, 0.0}; }

// ---------------------------------------------------------------- problem view
enum MaskKind { MASK_NONE = 0, MASK_BOOL = 1, MASK_ADDITIVE = 2, MASK_CAUSAL = 3 };

struct Problem {
  int64_t B, H, Nq, Nk, D;
  const double *q, *k, *v, *dq, *dk, *dv;  // [B,H,N,D] contiguous; tangents may be null (= 0)
  int mask_kind;
  const void* mask;  // uint8 (bool) or double (additive); [B|1,H|1,Nq,Nk] via strides
  int64_t msb, msh, msq, msk;  // mask strides in elements (0 = broadcast)
  double scale;

  const double* row(const double* base, int64_t bh, int64_t n, int64_t N) const {
    return base + (bh * N + n) * D;
  }
  // Returns whether key j takes part in row i of head (b,h); *bias gets M_ij.
  bool keep(int64_t b, int64_t h, int64_t i, int64_t j, double* bias) const {
    *bias = 0.0;
    switch (mask_kind) {
      case MASK_NONE:
        return true;
      case MASK_CAUSAL:
        return j <= i;
      case MASK_BOOL: {
        const uint8_t* m = static_cast<const uint8_t*>(mask);
        return m[b * msb + h * msh + i * msq + j * msk] != 0;
      }
      case MASK_ADDITIVE: {
        const double* m = static_cast<const double*>(mask);
        const double x = m[b * msb + h * msh + i * msq + j * msk];
        if (std::isinf(x) && x < 0) return false;
        *bias = x;
        return true;
      }
    }
    return false;
  }
};

inline double tangent_at(const double* p, int64_t idx) { return p ? p[idx] : 0.0; }

// One query row of the forward dual computation.  Writes O (value) and tO
// (tangent) rows of length D, and lse / mu.
void forward_row(const Problem& pr, int64_t b, int64_t h, int64_t i, double* o_row,
                 double* to_row, double* lse, double* mu) {
  const int64_t bh = b * pr.H + h, D = pr.D;
  const double* qi = pr.row(pr.q, bh, i, pr.Nq);
  const int64_t qoff = (bh * pr.Nq + i) * D;

  // Step 1: dual logits z_j = scale * (q + e dq).(k_j + e dk_j) + M_ij for kept keys.
  std::vector<Dual> z;
  std::vector<int64_t> keys;
  for (int64_t j = 0; j < pr.Nk; ++j) {
    double bias;
    if (!pr.keep(b, h, i, j, &bias)) continue;
    const double* kj = pr.row(pr.k, bh, j, pr.Nk);
    const int64_t koff = (bh * pr.Nk + j) * D;
    Dual dot = constant(0.0);
    for (int64_t d = 0; d < D; ++d) {
      const Dual qd = {qi[d], tangent_at(pr.dq, qoff + d)};
      const Dual kd = {kj[d], tangent_at(pr.dk, koff + d)};
      dot = dot + qd * kd;
    }
    z.push_back(constant(pr.scale) * dot + constant(bias));
    keys.push_back(j);
  }

  if (keys.empty()) {  // no kept key: the convention stated in the header
    for (int64_t d = 0; d < D; ++d) o_row[d] = to_row[d] = 0.0;
    *lse = -std::numeric_limits<double>::infinity();
    *mu = 0.0;
    return;
  }

  // Step 2: softmax with a constant shift m (zero tangent; it cancels exactly).
  double m = z[0].v;
  for (const Dual& zj : z) m = std::max(m, zj.v);
  std::vector<Dual> e(z.size());
  Dual L = constant(0.0);
  for (size_t n = 0; n < z.size(); ++n) {
    e[n] = dexp(z[n] - constant(m));
    L = L + e[n];
  }

  // Step 3: O = sum_j P_j (v_j + e dv_j).
  for (int64_t d = 0; d < D; ++d) {
    Dual acc = constant(0.0);
    for (size_t n = 0; n < keys.size(); ++n) {
      const int64_t voff = (bh * pr.Nk + keys[n]) * D + d;
      const Dual P = e[n] / L;
      acc = acc + P * Dual{pr.v[voff], tangent_at(pr.dv, voff)};
    }
    o_row[d] = acc.v;
    to_row[d] = acc.t;
  }

  // Step 4: lse = m + log L; its tangent is mu = rowsum(P * dS).
  const Dual lse_dual = constant(m) + dlog(L);
  *lse = lse_dual.v;
  *mu = lse_dual.t;
}

// Reverse mode of the dual computation of one head (b,h): given cotangents gO
// and gtO of O and tO, accumulate the gradients of
//   Loss = <gO, O> + <gtO, tO>
// with respect to q, k, v, dq, dk, dv.  It walks back through exactly the
// steps of forward_row (logits, shifted exponentials, normaliser, weights,
// outputs), one adjoint per forward quantity.  The shift m is a constant: the
// outputs do not depend on it, so no gradient flows through it.
void backward_head(const Problem& pr, int64_t b, int64_t h, const double* go,
                   const double* gto, double* gq, double* gk, double* gv, double* gdq,
                   double* gdk, double* gdv) {
  const int64_t bh = b * pr.H + h, D = pr.D;
  for (int64_t i = 0; i < pr.Nq; ++i) {
    const int64_t qoff = (bh * pr.Nq + i) * D;
    const double* qi = pr.q + qoff;
    const double* go_i = go + qoff;
    const double* gto_i = gto + qoff;

    // Forward quantities of row i: values zv, tangents zt.
    std::vector<int64_t> keys;
    std::vector<double> zv, zt;
    for (int64_t j = 0; j < pr.Nk; ++j) {
      double bias;
      if (!pr.keep(b, h, i, j, &bias)) continue;
      const int64_t koff = (bh * pr.Nk + j) * D;
      double s_qk = 0.0, s_t = 0.0;
      for (int64_t d = 0; d < D; ++d) {
        s_qk += qi[d] * pr.k[koff + d];
        s_t += tangent_at(pr.dq, qoff + d) * pr.k[koff + d] +
               qi[d] * tangent_at(pr.dk, koff + d);
      }
      keys.push_back(j);
      zv.push_back(pr.scale * s_qk + bias);
      zt.push_back(pr.scale * s_t);
    }
    if (keys.empty()) continue;  // outputs are constant zero: no gradient
    const size_t n_keys = keys.size();
    double m = zv[0];
    for (double x : zv) m = std::max(m, x);
    std::vector<double> e(n_keys), et(n_keys);
    double L = 0.0, Lt = 0.0;
    for (size_t n = 0; n < n_keys; ++n) {
      e[n] = std::exp(zv[n] - m);  // e_j   = exp(z_j - m)
      et[n] = e[n] * zt[n];        // et_j  = tangent of e_j
      L += e[n];                   // L     = sum e_j
      Lt += et[n];                 // Lt    = sum et_j
    }
    // P_j = e_j / L ; Pt_j = et_j / L - e_j Lt / L^2 ;
    // O = sum P_j v_j ; tO = sum Pt_j v_j + P_j dv_j.
    std::vector<double> ge(n_keys, 0.0), get(n_keys, 0.0);
    double gL = 0.0, gLt = 0.0;
    for (size_t n = 0; n < n_keys; ++n) {
      const int64_t voff = (bh * pr.Nk + keys[n]) * D;
      const double P = e[n] / L;
      const double Pt = et[n] / L - e[n] * Lt / (L * L);
      double gP = 0.0, gPt = 0.0;
      for (int64_t d = 0; d < D; ++d) {
        const double vd = pr.v[voff + d];
        const double dvd = tangent_at(pr.dv, voff + d);
        gP += go_i[d] * vd + gto_i[d] * dvd;
        gPt += gto_i[d] * vd;
        gv[voff + d] += P * go_i[d] + Pt * gto_i[d];
        gdv[voff + d] += P * gto_i[d];
      }
      // through Pt_j = et_j / L - e_j Lt / L^2
      get[n] += gPt / L;
      ge[n] += -gPt * Lt / (L * L);
      gL += -gPt * et[n] / (L * L) + 2.0 * gPt * e[n] * Lt / (L * L * L);
      gLt += -gPt * e[n] / (L * L);
      // through P_j = e_j / L
      ge[n] += gP / L;
      gL += -gP * e[n] / (L * L);
    }
    for (size_t n = 0; n < n_keys; ++n) {
      ge[n] += gL;     // L  = sum e_j
      get[n] += gLt;   // Lt = sum et_j
      // et_j = e_j * zt_j
      ge[n] += get[n] * zt[n];
      const double gzt = get[n] * e[n];
      // e_j = exp(z_j - m)
      const double gz = ge[n] * e[n];
      // z_j = scale q.k_j + M ; zt_j = scale (dq.k_j + q.dk_j)
      const int64_t koff = (bh * pr.Nk + keys[n]) * D;
      for (int64_t d = 0; d < D; ++d) {
        const double kd = pr.k[koff + d];
        const double dkd = tangent_at(pr.dk, koff + d);
        const double dqd = tangent_at(pr.dq, qoff + d);
        gq[qoff + d] += pr.scale * (gz * kd + gzt * dkd);
        gdq[qoff + d] += pr.scale * gzt * kd;
        gk[koff + d] += pr.scale * (gz * qi[d] + gzt * dqd);
        gdk[koff + d] += pr.scale * gzt * qi[d];
      }
    }
  }
}

template <class Fn>
void parallel_for(int64_t n, int nthreads, Fn fn) {
  if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
  if (nthreads <= 0) nthreads = 1;
  if (nthreads > n) nthreads = static_cast<int>(n > 0 ? n : 1);
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (int64_t it = next.fetch_add(1); it < n; it = next.fetch_add(1)) fn(it);
  };
  std::vector<std::thread> pool;
  for (int t = 1; t < nthreads; ++t) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
}

Problem make_problem(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, const double* q,
                     const double* k, const double* v, const double* dq, const double* dk,
                     const double* dv, int mask_kind, const void* mask, int64_t msb,
                     int64_t msh, int64_t msq, int64_t msk, double scale) {
  Problem pr{B, H, Nq, Nk, D, q, k, v, dq, dk, dv, mask_kind, mask, msb, msh, msq, msk, scale};
  return pr;
}

}  // namespace

extern "C" {

// Number of worker threads a call with nthreads <= 0 uses.
int oracle_default_threads(void) {
  const int n = static_cast<int>(std::thread::hardware_concurrency());
  return n > 0 ? n : 1;
}

// Forward + JVP for a list of query rows.  row_ids[r] = (b*H + h)*Nq + i.
// Outputs are compact: o_rows/to_rows [nrows, D], lse_rows/mu_rows [nrows].
// Any of dq, dk, dv may be null (zero tangent).  Returns 0, or -1 on bad args.
int oracle_fwd_dual_rows(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D,
                         const double* q, const double* k, const double* v, const double* dq,
                         const double* dk, const double* dv, int mask_kind, const void* mask,
                         int64_t msb, int64_t msh, int64_t msq, int64_t msk, double scale,
                         const int64_t* row_ids, int64_t nrows, double* o_rows,
                         double* to_rows, double* lse_rows, double* mu_rows, int nthreads) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || D <= 0 || !q || !k || !v) return -1;
  if (mask_kind < MASK_NONE || mask_kind > MASK_CAUSAL) return -1;
  if ((mask_kind == MASK_BOOL || mask_kind == MASK_ADDITIVE) && !mask) return -1;
  const Problem pr =
      make_problem(B, H, Nq, Nk, D, q, k, v, dq, dk, dv, mask_kind, mask, msb, msh, msq, msk, scale);
  for (int64_t r = 0; r < nrows; ++r)
    if (row_ids[r] < 0 || row_ids[r] >= B * H * Nq) return -1;
  parallel_for(nrows, nthreads, [&](int64_t r) {
    const int64_t id = row_ids[r];
    const int64_t i = id % Nq, bh = id / Nq;
    forward_row(pr, bh / H, bh % H, i, o_rows + r * D, to_rows + r * D, lse_rows + r,
                mu_rows + r);
  });
  return 0;
}

// Forward + JVP over every row: o, t_o [B,H,Nq,D]; lse, mu [B,H,Nq].
int oracle_fwd_dual(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, const double* q,
                    const double* k, const double* v, const double* dq, const double* dk,
                    const double* dv, int mask_kind, const void* mask, int64_t msb,
                    int64_t msh, int64_t msq, int64_t msk, double scale, double* o,
                    double* t_o, double* lse, double* mu, int nthreads) {
  const int64_t rows = B * H * Nq;
  std::vector<int64_t> ids(static_cast<size_t>(rows));
  for (int64_t r = 0; r < rows; ++r) ids[static_cast<size_t>(r)] = r;
  return oracle_fwd_dual_rows(B, H, Nq, Nk, D, q, k, v, dq, dk, dv, mask_kind, mask, msb, msh,
                              msq, msk, scale, ids.data(), rows, o, t_o, lse, mu, nthreads);
}

// Gradients of <gO, O> + <gtO, tO> with respect to q, k, v, dq, dk, dv (all
// [B,H,N,D] contiguous; overwritten).  Tangent inputs must be non-null here.
int oracle_bwd_dual(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D, const double* q,
                    const double* k, const double* v, const double* dq, const double* dk,
                    const double* dv, int mask_kind, const void* mask, int64_t msb,
                    int64_t msh, int64_t msq, int64_t msk, double scale, const double* g_o,
                    const double* g_to, double* g_q, double* g_k, double* g_v, double* g_dq,
                    double* g_dk, double* g_dv, int nthreads) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || D <= 0) return -1;
  if (!q || !k || !v || !dq || !dk || !dv || !g_o || !g_to) return -1;
  if (!g_q || !g_k || !g_v || !g_dq || !g_dk || !g_dv) return -1;
  if (mask_kind < MASK_NONE || mask_kind > MASK_CAUSAL) return -1;
  if ((mask_kind == MASK_BOOL || mask_kind == MASK_ADDITIVE) && !mask) return -1;
  const Problem pr =
      make_problem(B, H, Nq, Nk, D, q, k, v, dq, dk, dv, mask_kind, mask, msb, msh, msq, msk, scale);
  const size_t nq = static_cast<size_t>(B * H * Nq * D), nk = static_cast<size_t>(B * H * Nk * D);
  std::memset(g_q, 0, nq * sizeof(double));
  std::memset(g_dq, 0, nq * sizeof(double));
  std::memset(g_k, 0, nk * sizeof(double));
  std::memset(g_v, 0, nk * sizeof(double));
  std::memset(g_dk, 0, nk * sizeof(double));
  std::memset(g_dv, 0, nk * sizeof(double));
  parallel_for(B * H, nthreads, [&](int64_t bh) {
    backward_head(pr, bh / H, bh % H, g_o, g_to, g_q, g_k, g_v, g_dq, g_dk, g_dv);
  });
  return 0;
}

}  // extern "C"
