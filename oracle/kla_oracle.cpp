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
#include <atomic>

// KLA_ORACLE_MUTANT (default 0) plants one deliberate mistake, for the test
// that checks the pins are sensitive to it; product and parity builds use 0.
#ifndef KLA_ORACLE_MUTANT
#define KLA_ORACLE_MUTANT 0
#endif

namespace {

template <typename R>
struct Args {
  const float *q, *k, *v, *lam_v, *a, *pbar, *lam0, *eta0;
  int B, H, T, dk, dv;
  R *y, *lamT, *etaT, *y_scale, *eta_scale;
};

template <typename R>
long long run_head(const Args<R>& g, long long bh) {
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
  std::vector<R> yacc(dv), ysc(dv);
  for (int t = 0; t < T; ++t) {
    const size_t ri = ((size_t)bh * T + t) * dk;  // row of the per-i inputs
    const size_t rj = ((size_t)bh * T + t) * dv;  // row of the per-j inputs
    for (int j = 0; j < dv; ++j) { yacc[j] = 0; ysc[j] = 0; }
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
        P[e] = Pn;
        mu[e] = mun;
        yacc[j] += qi * readout;
        ysc[j] += std::fabs(qi) * muabs[e];
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
    }
  }
  for (size_t e = 0; e < E; ++e) {
    if (g.lamT) g.lamT[bh * E + e] = (R)1 / P[e];
    if (g.etaT) g.etaT[bh * E + e] = mu[e] / P[e];
    if (g.eta_scale) g.eta_scale[bh * E + e] = muabs[e] / P[e];
  }
  return violations;
}

template <typename R>
long long run_all(const Args<R>& g, int nthreads) {
  const long long nbh = (long long)g.B * g.H;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > nbh) nthreads = (int)nbh;
  std::atomic<long long> next(0), viol(0);
  auto worker = [&]() {
    long long local = 0;
    for (;;) {
      const long long bh = next.fetch_add(1);
      if (bh >= nbh) break;
      local += run_head<R>(g, bh);
    }
    viol += local;
  };
  std::vector<std::thread> pool;
  for (int w = 1; w < nthreads; ++w) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
  return viol.load();
}

}  // namespace

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
                                 double* y_scale, double* eta_scale, int nthreads) {
  if (!q || !k || !v || !lam_v || !a || !pbar || B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0)
    return -1;
  Args<double> g{q, k, v, lam_v, a, pbar, lam0, eta0, B, H, T, dk, dv, y, lamT, etaT, y_scale, eta_scale};
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

}  // extern "C"
