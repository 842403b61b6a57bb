// Reference oracle for the Kalman Linear Attention scan: TEST INFRASTRUCTURE ONLY.
//
// Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
// leg may load this code. The product path (the CUDA library) never calls it.
//
// Source: "Technische Samenvatting: Kalman Linear Attention (KLA)"
// (gist.science/nl/paper/2602.10743), Methodologie §1 "Probabilistische
// Formulering" (OU dynamics prior with process noise p̄_t, observation operator
// k_t with value precision Λ^v_t, posterior-mean readout through q_t) and the
// diagonal structure stated under "Belangrijkste Bijdragen" item 1: every
// state element (i, j) of a head is its own scalar linear-Gaussian filter.
//
// What is computed, per head (b, h) and element (i, j), in the textbook
// variance (covariance) form of the scalar Kalman filter, starting from the
// prior P = 1/λ0, μ = η0/λ0 and for every token t = 0..T-1 in order:
//
//     P_pred = a_{t,i}² · P + p̄_{t,i}                       (OU predict)
//     μ_pred = a_{t,i} · μ
//     P      = 1 / (1/P_pred + k_{t,i}² · Λ^v_{t,j})          (observation of
//     μ      = P · (μ_pred/P_pred + k_{t,i} · Λ^v_{t,j} · v_{t,j})   v_{t,j} through k_{t,i})
//     y[t,j] += q_{t,i} · μ            (summed over i in increasing order)
//     y_var[t,j] += q_{t,i}² · P       (optional: the readout's variance under
//                                       the posterior, the layer's explicit
//                                       belief uncertainty, Belangrijkste
//                                       Bijdragen item 3)
//
// and at the end λ_T = 1/P, η_T = μ/P (information form). The readout uses the
// posterior that already includes token t.
//
// The same loop also returns condition scales used as the denominators of the
// relative-error tests: μ̂ follows the mean recursion with every term taken in
// absolute value (μ̂ = P·(|a|·μ̂/P_pred + |k·Λ^v·v|)), y_scale[t,j] = Σ_i |q|·μ̂
// and eta_scale = μ̂/P. They bound the magnitude of everything that is summed,
// so |error| / scale measures rounding error even where y or η cancel to ~0.
//
// It also counts, per element-step, violations of the invariants that exact
// filtering implies: λ_t > 0, λ_t ≥ k²Λ^v (the update adds that precision to
// a positive prior precision) and, when p̄ > 0, λ_t ≤ 1/p̄ + k²Λ^v (the
// predicted precision never exceeds 1/p̄).
//
// Inputs are float32 arrays (the exact values the GPU reads, bf16 inputs
// already widened); arithmetic is in R = double (the parity oracle) or
// R = float (a plain fp32 build of the same loop, timed as a CPU baseline).
// Layout: q, k, a, pbar [B,H,T,dk]; v, lam_v [B,H,T,dv]; y [B,H,T,dv];
// lam0, eta0, lamT, etaT [B,H,dk,dv]; all contiguous row-major.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <limits>
#include <thread>
#include <vector>
#include <algorithm>
#include <atomic>

// KLA_ORACLE_MUTANT (default 0) plants one deliberate mistake, for the test
// that checks the pins are sensitive to it; product and parity builds use 0.
#ifndef KLA_ORACLE_MUTANT
#define KLA_ORACLE_MUTANT 0
#endif

namespace {

template <typename R, typename In = float>
struct Args {
  const In *q, *k, *v, *lam_v, *a, *pbar, *lam0, *eta0;
  int B, H, T, dk, dv;
  R *y, *lamT, *etaT, *y_scale, *eta_scale;
  R* y_var = nullptr;  // Σ_i q_i² P (the readout's variance), or NULL
};

template <typename R, typename In>
long long run_head(const Args<R, In>& g, long long bh) {
  const int T = g.T, dk = g.dk, dv = g.dv;
  const size_t E = (size_t)dk * dv;
  std::vector<R> P(E), mu(E), muabs(E);
  for (size_t e = 0; e < E; ++e) {
    const R l0 = g.lam0 ? (R)g.lam0[bh * E + e] : (R)1;
    const R n0 = g.eta0 ? (R)g.eta0[bh * E + e] : (R)0;
    P[e] = (R)1 / l0;
    mu[e] = n0 / l0;
    muabs[e] = std::fabs(mu[e]);
  }
  long long violations = 0;
  std::vector<R> yacc(dv), ysc(dv), yvar(dv);
  for (int t = 0; t < T; ++t) {
    const size_t ri = ((size_t)bh * T + t) * dk;  // row of the per-i inputs
    const size_t rj = ((size_t)bh * T + t) * dv;  // row of the per-j inputs
    for (int j = 0; j < dv; ++j) { yacc[j] = 0; ysc[j] = 0; yvar[j] = 0; }
    for (int i = 0; i < dk; ++i) {
      const R ai = g.a[ri + i], pi = g.pbar[ri + i], ki = g.k[ri + i], qi = g.q[ri + i];
      for (int j = 0; j < dv; ++j) {
        const size_t e = (size_t)i * dv + j;
        const R Lj = g.lam_v[rj + j], vj = g.v[rj + j];
        R c = ki * ki * Lj;             // observation precision k²Λ^v
        R b = ki * Lj * vj;             // information added, kΛ^v v
        R Ppred = ai * ai * P[e] + pi;
        if (KLA_ORACLE_MUTANT == 1) Ppred = ai * ai * P[e];        // dropped p̄
        if (KLA_ORACLE_MUTANT == 2) Ppred = ai * P[e] + pi;        // a instead of a²
        if (KLA_ORACLE_MUTANT == 3) c = ki * Lj;                   // k instead of k²
        if (KLA_ORACLE_MUTANT == 5) b = ki * vj;                   // Λ^v missing
        const R mupred = ai * mu[e];
        const R Pn = (R)1 / ((R)1 / Ppred + c);
        R mun = Pn * (mupred / Ppred + b);
        if (KLA_ORACLE_MUTANT == 6) mun = Ppred * (mupred / Ppred + b);  // prior variance
        const R readout = (KLA_ORACLE_MUTANT == 4) ? mupred : mun;      // 4: prior mean read out
        muabs[e] = Pn * (std::fabs(ai) * muabs[e] / Ppred + std::fabs(b));
        if (KLA_ORACLE_MUTANT == 12) muabs[e] += Pn * std::fabs(b);  // 12: |b| counted twice in the scale
        P[e] = Pn;
        mu[e] = mun;
        yacc[j] += qi * readout;
        yvar[j] += qi * qi * (KLA_ORACLE_MUTANT == 10 ? Ppred : Pn);  // 10: prior variance read out
        ysc[j] += (KLA_ORACLE_MUTANT == 11 ? (R)2 : (R)1) * std::fabs(qi) * muabs[e];  // 11: |q| twice
        const R lam = (R)1 / Pn;
        if (!(lam > 0)) ++violations;
        // λ_t = λ_pred + c with λ_pred ∈ (0, 1/p̄]; allow one rounding step.
        const R tol = (R)8 * std::numeric_limits<R>::epsilon() * lam;
        if (lam < c - tol) ++violations;
        if (pi > 0 && lam > (R)1 / pi + c + tol) ++violations;
      }
    }
    for (int j = 0; j < dv; ++j) {
      if (g.y) g.y[rj + j] = yacc[j];
      if (g.y_scale) g.y_scale[rj + j] = ysc[j];
      if (g.y_var) g.y_var[rj + j] = yvar[j];
    }
  }
  for (size_t e = 0; e < E; ++e) {
    if (g.lamT) g.lamT[bh * E + e] = (R)1 / P[e];
    if (g.etaT) g.etaT[bh * E + e] = mu[e] / P[e];
    if (g.eta_scale) g.eta_scale[bh * E + e] = muabs[e] / P[e];
  }
  return violations;
}

// Run `head(bh)` for every head over nthreads std::threads; returns the sum
// of what the calls return.
template <typename F>
long long over_heads(long long nbh, int nthreads, F head) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nbh) nthreads = (int)nbh;
  std::atomic<long long> next(0), viol(0);
  auto worker = [&]() {
    long long local = 0;
    for (;;) {
      const long long bh = next.fetch_add(1);
      if (bh >= nbh) break;
      local += head(bh);
    }
    viol += local;
  };
  std::vector<std::thread> pool;
  for (int w = 1; w < nthreads; ++w) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return viol.load();
}

template <typename R, typename In>
long long run_all(const Args<R, In>& g, int nthreads) {
  return over_heads((long long)g.B * g.H, nthreads, [&](long long bh) { return run_head<R, In>(g, bh); });
}


// ---- backward (reverse-mode derivative of the loop above) ------------------
//
// The pages define the forward scan only; the gradient is its exact
// reverse-mode derivative (what autodiff of the loop would return), pinned in
// tests by central finite differences of the forward above. Given upstream
// gradients dy [B,H,T,dv] and (optionally) dλ_T, dη_T [B,H,dk,dv] of a scalar
// loss, it returns dq, dk, da, dp̄ [B,H,T,dk], dv, dΛ^v [B,H,T,dv] and dλ0, dη0
// [B,H,dk,dv].
//
// Per element (i, j), with the forward written as
//     P⁻ = a²P + p̄,  c = k²Λ^v,  b = kΛ^v v,  w = 1/(1 + cP⁻),
//     P' = wP⁻,      u = aμ + P⁻b,  μ' = wu,   y_j += q μ'
// (the same P' and μ' as above: 1/(1/P⁻ + c) = wP⁻ and P'(aμ/P⁻ + b) = wu),
// the adjoints (P̄, μ̄) of (P', μ') flow back one token at a time:
//     μ̄ += q·dy_j;  dq += dy_j·μ'
//     ū = μ̄w;  w̄ = μ̄u + P̄P⁻
//     P̄⁻ = P̄w + ūb − w̄cw²;  c̄ = −w̄P⁻w²;  b̄ = ūP⁻
//     da += ūμ + 2aP·P̄⁻;  dp̄ += P̄⁻
//     dk += 2kΛ^v·c̄ + Λ^v v·b̄;  dΛ^v += k²·c̄ + kv·b̄;  dv += kΛ^v·b̄
//     (P̄, μ̄) ← (a²P̄⁻, aū)                    — adjoints of (P, μ) before the token
// from (P̄, μ̄) = (−(dλ_T + dη_T μ_T)/P_T², dη_T/P_T) at the end, through
// λ_T = 1/P_T and η_T = μ_T/P_T; and at the start P = 1/λ0, μ = η0/λ0 give
//     dλ0 = −(P̄ + μ̄η0)/λ0²,  dη0 = μ̄/λ0.
// Each element is differentiated on its own (its forward states kept for all
// tokens), and its contributions are added to the per-row and per-column
// gradients in element order (i major, j minor), so the sums are
// deterministic.
//
// Condition scales (for the relative-error tests): the same recursion with
// every term in absolute value (shadow adjoints P̂̄, μ̂̄, and the forward's
// absolute mean μ̂), summed into *_scale arrays of the gradients' shapes.
template <typename In>
struct BwdArgs {
  const In *q, *k, *v, *lam_v, *a, *pbar, *lam0, *eta0;
  const In *dy, *dlamT, *detaT;
  int B, H, T, dk, dv;
  double *dq, *dk_, *dv_, *dlam_v, *da, *dpbar, *dlam0, *deta0;  // gradients (any may be NULL)
  double *sq, *sk, *sv, *slam_v, *sa, *spbar, *slam0, *seta0;    // condition scales (any may be NULL)
};

template <typename In>
long long bwd_head(const BwdArgs<In>& g, long long bh) {
  const int T = g.T, dk = g.dk, dv = g.dv;
  const size_t E = (size_t)dk * dv;
  std::vector<double> P(T + 1), mu(T + 1), muabs(T + 1);
  auto add = [](double* arr, size_t idx, double x) {
    if (arr) arr[idx] += x;
  };
  {  // this head's per-row and per-column gradient slices start at zero
    const size_t r0 = (size_t)bh * T * dk, c0 = (size_t)bh * T * dv;
    for (double* arr : {g.dq, g.dk_, g.da, g.dpbar, g.sq, g.sk, g.sa, g.spbar})
      if (arr) std::fill(arr + r0, arr + r0 + (size_t)T * dk, 0.0);
    for (double* arr : {g.dv_, g.dlam_v, g.sv, g.slam_v})
      if (arr) std::fill(arr + c0, arr + c0 + (size_t)T * dv, 0.0);
  }
  for (int i = 0; i < dk; ++i) {
    for (int j = 0; j < dv; ++j) {
      const size_t e = (size_t)i * dv + j, es = (size_t)bh * E + e;
      const double l0 = g.lam0 ? (double)g.lam0[es] : 1.0;
      const double n0 = g.eta0 ? (double)g.eta0[es] : 0.0;
      // forward for this element, keeping every state
      P[0] = 1.0 / l0;
      mu[0] = n0 / l0;
      muabs[0] = std::fabs(mu[0]);
      for (int t = 0; t < T; ++t) {
        const size_t ri = ((size_t)bh * T + t) * dk + i, rj = ((size_t)bh * T + t) * dv + j;
        const double at = g.a[ri], pt = g.pbar[ri], kt = g.k[ri];
        const double Lt = g.lam_v[rj], vt = g.v[rj];
        const double c = kt * kt * Lt, b = kt * Lt * vt;
        const double Pp = at * at * P[t] + pt;
        const double w = 1.0 / (1.0 + c * Pp);
        P[t + 1] = w * Pp;
        mu[t + 1] = w * (at * mu[t] + Pp * b);
        muabs[t + 1] = w * (std::fabs(at) * muabs[t] + Pp * std::fabs(b));
      }
      // terminal adjoints
      const double PT = P[T], dl = g.dlamT ? (double)g.dlamT[es] : 0.0, de = g.detaT ? (double)g.detaT[es] : 0.0;
      double Pb = -(dl + de * mu[T]) / (PT * PT);
      double mb = de / PT;
      double Pbh = (std::fabs(dl) + std::fabs(de) * muabs[T]) / (PT * PT);
      double mbh = std::fabs(de) / PT;
      for (int t = T - 1; t >= 0; --t) {
        const size_t ri = ((size_t)bh * T + t) * dk + i, rj = ((size_t)bh * T + t) * dv + j;
        const double at = g.a[ri], pt = g.pbar[ri], kt = g.k[ri], qt = g.q[ri];
        const double Lt = g.lam_v[rj], vt = g.v[rj], gy = g.dy ? (double)g.dy[rj] : 0.0;
        const double c = kt * kt * Lt, b = kt * Lt * vt;
        const double Pp = at * at * P[t] + pt;
        const double w = 1.0 / (1.0 + c * Pp);
        const double u = at * mu[t] + Pp * b, uabs = std::fabs(at) * muabs[t] + Pp * std::fabs(b);
        // readout y_j += q μ'
        mb += qt * gy;
        mbh += std::fabs(qt * gy);
        add(g.dq, ri, gy * mu[t + 1]);
        add(g.sq, ri, (KLA_ORACLE_MUTANT == 13 ? 2.0 : 1.0) * std::fabs(gy) * muabs[t + 1]);  // 13: scale doubled
        // through μ' = w u and P' = w P⁻
        const double ub = mb * w, ubh = mbh * w;
        const double wb = mb * u + Pb * Pp, wbh = mbh * uabs + Pbh * Pp;
        double Ppb = Pb * w + ub * b - wb * c * w * w;
        if (KLA_ORACLE_MUTANT == 7) Ppb = Pb * w + ub * b;  // dropped the path through w
        double Ppbh = Pbh * w + ubh * std::fabs(b) + wbh * c * w * w;
        if (KLA_ORACLE_MUTANT == 14) Ppbh += Pbh * w;  // 14: the carried term counted twice in the scale
        double cb = -wb * Pp * w * w;
        if (KLA_ORACLE_MUTANT == 8) cb = wb * Pp * w * w;   // sign of ∂w/∂c
        const double cbh = (KLA_ORACLE_MUTANT == 15 ? 2.0 : 1.0) * wbh * Pp * w * w;  // 15: scale doubled
        const double bb = ub * Pp, bbh = ubh * Pp;
        // per-row inputs
        add(g.da, ri, ub * mu[t] + 2.0 * at * P[t] * Ppb);
        add(g.sa, ri, ubh * muabs[t] + 2.0 * std::fabs(at) * P[t] * Ppbh);
        add(g.dpbar, ri, Ppb);
        add(g.spbar, ri, Ppbh);
        add(g.dk_, ri, 2.0 * kt * Lt * cb + Lt * vt * bb);
        add(g.sk, ri, 2.0 * std::fabs(kt) * Lt * cbh + Lt * std::fabs(vt) * bbh);
        // per-column inputs
        add(g.dlam_v, rj, kt * kt * cb + kt * vt * bb);
        add(g.slam_v, rj, kt * kt * cbh + std::fabs(kt * vt) * bbh);
        add(g.dv_, rj, kt * Lt * bb);
        add(g.sv, rj, std::fabs(kt) * Lt * bbh);
        // adjoints of the state before token t
        Pb = (KLA_ORACLE_MUTANT == 9 ? at : at * at) * Ppb;  // 9: a instead of a²
        mb = at * ub;
        Pbh = at * at * Ppbh;
        mbh = std::fabs(at) * ubh;
      }
      if (g.dlam0) g.dlam0[es] = -(Pb + mb * n0) / (l0 * l0);
      if (g.slam0) g.slam0[es] = (Pbh + mbh * std::fabs(n0)) / (l0 * l0);
      if (g.deta0) g.deta0[es] = mb / l0;
      if (g.seta0) g.seta0[es] = mbh / l0;
    }
  }
  return 0;
}

}  // namespace

#define KLA_BWD_PARAMS(In)                                                                       \
  const In *q, const In *k, const In *v, const In *lam_v, const In *a, const In *pbar,            \
      const In *lam0, const In *eta0, const In *dy, const In *dlamT, const In *detaT, int B, int H, \
      int T, int dk, int dv, double *dq, double *dk_, double *da, double *dpbar, double *dv_,       \
      double *dlam_v, double *dlam0, double *deta0, double *sq, double *sk, double *sa,            \
      double *spbar, double *sv, double *slam_v, double *slam0, double *seta0, int nthreads

template <typename In>
long long backward_all(KLA_BWD_PARAMS(In)) {
  if (!q || !k || !v || !lam_v || !a || !pbar || B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
    return -1;
  BwdArgs<In> g{q,  k,  v,  lam_v, a,     pbar,   lam0,  eta0, dy,    dlamT,  detaT, B,     H,
                T,  dk, dv, dq,    dk_,   dv_,    dlam_v, da,  dpbar, dlam0,  deta0, sq,    sk,
                sv, slam_v, sa,    spbar, slam0,  seta0};
  return over_heads((long long)B * H, nthreads, [&](long long bh) { return bwd_head<In>(g, bh); });
}

extern "C" {

// Returns the number of invariant violations seen (0 expected), or -1 on a
// bad argument. Any output pointer may be NULL. lam0/eta0 NULL mean λ0 = 1,
// η0 = 0. Heads are processed in parallel over nthreads std::threads; within a
// head the arithmetic order is fixed, so results do not depend on nthreads.
long long kla_oracle_forward_f64(const float* q, const float* k, const float* v,
                                 const float* lam_v, const float* a, const float* pbar,
                                 const float* lam0, const float* eta0,
                                 int B, int H, int T, int dk, int dv,
                                 double* y, double* lamT, double* etaT,
                                 double* y_scale, double* eta_scale, double* y_var, int nthreads) {
  if (!q || !k || !v || !lam_v || !a || !pbar || B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
    return -1;
  Args<double> g{q, k, v, lam_v, a, pbar, lam0, eta0, B, H, T, dk, dv, y, lamT, etaT, y_scale, eta_scale, y_var};
  return run_all<double>(g, nthreads);
}

long long kla_oracle_forward_f32(const float* q, const float* k, const float* v,
                                 const float* lam_v, const float* a, const float* pbar,
                                 const float* lam0, const float* eta0,
                                 int B, int H, int T, int dk, int dv,
                                 float* y, float* lamT, float* etaT, int nthreads) {
  if (!q || !k || !v || !lam_v || !a || !pbar || B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
    return -1;
  Args<float> g{q, k, v, lam_v, a, pbar, lam0, eta0, B, H, T, dk, dv, y, lamT, etaT, nullptr, nullptr};
  return run_all<float>(g, nthreads);
}

// Forward with fp64 inputs (finite-difference pins of the backward perturb
// inputs below float precision).
long long kla_oracle_forward_f64in(const double* q, const double* k, const double* v,
                                   const double* lam_v, const double* a, const double* pbar,
                                   const double* lam0, const double* eta0,
                                   int B, int H, int T, int dk, int dv,
                                   double* y, double* lamT, double* etaT, double* y_scale, double* eta_scale,
                                   int nthreads) {
  if (!q || !k || !v || !lam_v || !a || !pbar || B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
    return -1;
  Args<double, double> g{q, k, v, lam_v, a, pbar, lam0, eta0, B, H, T, dk, dv, y, lamT, etaT, y_scale, eta_scale};
  return run_all<double, double>(g, nthreads);
}

// Backward in fp64. Gradient outputs: dq, dk, da, dpbar [B,H,T,dk];
// dv, dlam_v [B,H,T,dv]; dlam0, deta0 [B,H,dk,dv]; scales: the same eight in
// that order (any output may be NULL). dy NULL means zero; dlamT/detaT NULL
// mean zero. Returns 0, or -1 on a bad argument.
long long kla_oracle_backward_f64(KLA_BWD_PARAMS(float)) {
  return backward_all<float>(q, k, v, lam_v, a, pbar, lam0, eta0, dy, dlamT, detaT, B, H, T, dk, dv, dq, dk_,
                             da, dpbar, dv_, dlam_v, dlam0, deta0, sq, sk, sa, spbar, sv, slam_v, slam0, seta0,
                             nthreads);
}

long long kla_oracle_backward_f64in(KLA_BWD_PARAMS(double)) {
  return backward_all<double>(q, k, v, lam_v, a, pbar, lam0, eta0, dy, dlamT, detaT, B, H, T, dk, dv, dq, dk_,
                              da, dpbar, dv_, dlam_v, dlam0, deta0, sq, sk, sa, spbar, sv, slam_v, slam0, seta0,
                              nthreads);
}

}  // extern "C"
