// Test infrastructure: the CPU oracle for the Mamba-2 SSD selective scan.
//
// This is NOT part of the product path.  Only the tests, the smoke check and
// the benchmark's CPU-baseline leg load it.  It shares no code, header or
// constant with the CUDA library.
//
// What it computes: the plain per-token recurrence of the selective state
// space model ("Optimizing Mamba-2 kernels for the B200", section "Why
// optimize Mamba-2?", Figure 1: the linear-time form of Mamba-2), in fp64,
// one (batch, head) pair at a time, one token after another:
//
//   delta_t = softplus(dt[b,t,h] + dt_bias[h])        (softplus(v) = v for v > 20)
//   alpha_t = exp(delta_t * A[h])
//   h_t     = alpha_t * h_{t-1} + delta_t * x_t (outer) B_t[g(h)]      (P x N)
//   y_t[p]  = sum_n h_t[p,n] * C_t[g(h)][n] + D[h] * x_t[p]
//   final   = h_{T-1},  h_{-1} = init (or 0)
//
// with g(h) = h / (H / G): contiguous blocks of H/G heads share B and C.
//
// The backward pass is the reverse sweep of the same recurrence for the
// loss L = <dy, y> + <dfinal, final>; the states h_t are recomputed from
// checkpoints (a storage choice that leaves the arithmetic unchanged).
//
// Layouts (row-major, all fp64):
//   x, y, dy, dx : (Bt, T, H, P)      dt, ddt : (Bt, T, H)
//   B, C, dB, dC : (Bt, T, G, N)      init, final, dfinal, dinit : (Bt, H, P, N)
//   dt_bias, A, D and their gradients : (H)
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

struct Dims {
  int64_t Bt, T, H, P, N, G;
};

inline double softplus(double v) { return v > 20.0 ? v : std::log1p(std::exp(v)); }
inline double softplus_grad(double v) { return v > 20.0 ? 1.0 : 1.0 / (1.0 + std::exp(-v)); }

template <class F>
void parallel_for(int64_t n, int nthreads, F f) {
  if (nthreads <= 0) nthreads = (int)std::thread::hardware_concurrency();
  if (nthreads <= 0) nthreads = 1;
  if (nthreads > n) nthreads = (int)n;
  std::atomic<int64_t> next(0);
  auto worker = [&]() {
    for (;;) {
      int64_t i = next.fetch_add(1);
      if (i >= n) break;
      f(i);
    }
  };
  if (nthreads <= 1) {
    worker();
    return;
  }
  std::vector<std::thread> pool;
  for (int i = 0; i < nthreads; ++i) pool.emplace_back(worker);
  for (auto& th : pool) th.join();
}

inline Dims read_dims(const int64_t* d) { return Dims{d[0], d[1], d[2], d[3], d[4], d[5]}; }

bool dims_ok(const Dims& d) {
  return d.Bt > 0 && d.T > 0 && d.H > 0 && d.P > 0 && d.N > 0 && d.G > 0 && d.H % d.G == 0;
}

// One token of the recurrence for head h of batch b: h <- alpha*h + delta*x (x) B.
inline void step_state(double* hs, const double* xt, const double* Bt, double alpha, double delta,
                       int64_t P, int64_t N) {
  for (int64_t p = 0; p < P; ++p) {
    const double dx = delta * xt[p];
    double* row = hs + p * N;
    for (int64_t n = 0; n < N; ++n) row[n] = alpha * row[n] + dx * Bt[n];
  }
}

}  // namespace

extern "C" {

int ssd_oracle_hardware_threads(void) { return (int)std::thread::hardware_concurrency(); }

// Forward recurrence.  dt_bias, D, init and final may be NULL (treated as 0 /
// not written).  Returns 0 on success, 1 on bad dimensions.
int ssd_oracle_fwd(const int64_t* dims, const double* x, const double* dt, const double* dt_bias,
                   const double* A, const double* Bm, const double* Cm, const double* D,
                   const double* init, double* y, double* final_state, int nthreads) {
  const Dims d = read_dims(dims);
  if (!dims_ok(d)) return 1;
  const int64_t hpg = d.H / d.G;
  parallel_for(d.Bt * d.H, nthreads, [&](int64_t task) {
    const int64_t b = task / d.H, h = task % d.H, g = h / hpg;
    std::vector<double> hs(d.P * d.N, 0.0);
    if (init) std::memcpy(hs.data(), init + (b * d.H + h) * d.P * d.N, sizeof(double) * d.P * d.N);
    const double bias = dt_bias ? dt_bias[h] : 0.0;
    const double Dh = D ? D[h] : 0.0;
    for (int64_t t = 0; t < d.T; ++t) {
      const double delta = softplus(dt[(b * d.T + t) * d.H + h] + bias);
      const double alpha = std::exp(delta * A[h]);
      const double* xt = x + ((b * d.T + t) * d.H + h) * d.P;
      const double* Bt = Bm + ((b * d.T + t) * d.G + g) * d.N;
      const double* Ct = Cm + ((b * d.T + t) * d.G + g) * d.N;
      step_state(hs.data(), xt, Bt, alpha, delta, d.P, d.N);
      double* yt = y + ((b * d.T + t) * d.H + h) * d.P;
      for (int64_t p = 0; p < d.P; ++p) {
        double acc = 0.0;
        for (int64_t n = 0; n < d.N; ++n) acc += hs[p * d.N + n] * Ct[n];
        yt[p] = acc + Dh * xt[p];
      }
    }
    if (final_state)
      std::memcpy(final_state + (b * d.H + h) * d.P * d.N, hs.data(), sizeof(double) * d.P * d.N);
  });
  return 0;
}

// Reverse sweep.  dfinal may be NULL (zero).  Outputs: dx, ddt (gradient
// w.r.t. the raw dt input), dA, dB, dC (summed over the heads of each group),
// dD, ddt_bias, dinit; dD, ddt_bias and dinit may be NULL.
int ssd_oracle_bwd(const int64_t* dims, const double* x, const double* dt, const double* dt_bias,
                   const double* A, const double* Bm, const double* Cm, const double* D,
                   const double* init, const double* dy, const double* dfinal, double* dx,
                   double* ddt, double* dA, double* dB, double* dC, double* dD, double* ddt_bias,
                   double* dinit, int nthreads) {
  const Dims d = read_dims(dims);
  if (!dims_ok(d)) return 1;
  const int64_t hpg = d.H / d.G;
  const int64_t PN = d.P * d.N;
  // Checkpoint spacing ~ sqrt(T): memory per task is O(sqrt(T) * P * N).
  int64_t K = (int64_t)std::ceil(std::sqrt((double)d.T));
  if (K < 16) K = 16;
  const int64_t nseg = (d.T + K - 1) / K;

  // Per-(b,h) partials, reduced in a fixed order afterwards (deterministic).
  std::vector<double> dB_h(d.Bt * d.T * d.H * d.N), dC_h(d.Bt * d.T * d.H * d.N);
  std::vector<double> dA_bh(d.Bt * d.H), dD_bh(d.Bt * d.H), dbias_bh(d.Bt * d.H);

  parallel_for(d.Bt * d.H, nthreads, [&](int64_t task) {
    const int64_t b = task / d.H, h = task % d.H, g = h / hpg;
    const double bias = dt_bias ? dt_bias[h] : 0.0;
    const double Ah = A[h];
    const double Dh = D ? D[h] : 0.0;
    auto tok = [&](int64_t t) { return (b * d.T + t) * d.H + h; };
    auto grp = [&](int64_t t) { return (b * d.T + t) * d.G + g; };

    // Forward pass keeping the state before each segment.
    std::vector<double> ckpt(nseg * PN), hs(PN, 0.0);
    if (init) std::memcpy(hs.data(), init + (b * d.H + h) * PN, sizeof(double) * PN);
    for (int64_t t = 0; t < d.T; ++t) {
      if (t % K == 0) std::memcpy(&ckpt[(t / K) * PN], hs.data(), sizeof(double) * PN);
      const double delta = softplus(dt[tok(t)] + bias);
      step_state(hs.data(), x + tok(t) * d.P, Bm + grp(t) * d.N, std::exp(delta * Ah), delta, d.P,
                 d.N);
    }

    std::vector<double> G(PN, 0.0), seg((K + 1) * PN), tmp(d.P > d.N ? d.P : d.N);
    if (dfinal) std::memcpy(G.data(), dfinal + (b * d.H + h) * PN, sizeof(double) * PN);
    double dA_acc = 0.0, dD_acc = 0.0, dbias_acc = 0.0;
    for (int64_t s = nseg - 1; s >= 0; --s) {
      const int64_t t0 = s * K, t1 = (t0 + K < d.T) ? t0 + K : d.T;
      // seg[0] = h_{t0-1}; seg[i+1] = h_{t0+i}
      std::memcpy(&seg[0], &ckpt[s * PN], sizeof(double) * PN);
      for (int64_t t = t0; t < t1; ++t) {
        double* hn = &seg[(t - t0 + 1) * PN];
        std::memcpy(hn, &seg[(t - t0) * PN], sizeof(double) * PN);
        const double delta = softplus(dt[tok(t)] + bias);
        step_state(hn, x + tok(t) * d.P, Bm + grp(t) * d.N, std::exp(delta * Ah), delta, d.P, d.N);
      }
      for (int64_t t = t1 - 1; t >= t0; --t) {
        const double* h_t = &seg[(t - t0 + 1) * PN];
        const double* h_prev = &seg[(t - t0) * PN];
        const double v = dt[tok(t)] + bias;
        const double delta = softplus(v);
        const double alpha = std::exp(delta * Ah);
        const double* xt = x + tok(t) * d.P;
        const double* dyt = dy + tok(t) * d.P;
        const double* Bt = Bm + grp(t) * d.N;
        const double* Ct = Cm + grp(t) * d.N;
        // G <- G + dy_t (x) C_t : now G = dL/dh_t
        for (int64_t p = 0; p < d.P; ++p)
          for (int64_t n = 0; n < d.N; ++n) G[p * d.N + n] += dyt[p] * Ct[n];
        // dC_t (this head's share) = sum_p dy_t[p] h_t[p,:]
        double* dCt = &dC_h[((b * d.T + t) * d.H + h) * d.N];
        for (int64_t n = 0; n < d.N; ++n) {
          double acc = 0.0;
          for (int64_t p = 0; p < d.P; ++p) acc += dyt[p] * h_t[p * d.N + n];
          dCt[n] = acc;
        }
        // dx_t = D dy_t + delta (G B_t)
        double* dxt = dx + tok(t) * d.P;
        double gxb = 0.0;  // <G, x_t (x) B_t>
        for (int64_t p = 0; p < d.P; ++p) {
          double acc = 0.0;
          for (int64_t n = 0; n < d.N; ++n) acc += G[p * d.N + n] * Bt[n];
          dxt[p] = Dh * dyt[p] + delta * acc;
          gxb += xt[p] * acc;
        }
        // dB_t (this head's share) = delta G^T x_t
        double* dBt = &dB_h[((b * d.T + t) * d.H + h) * d.N];
        for (int64_t n = 0; n < d.N; ++n) {
          double acc = 0.0;
          for (int64_t p = 0; p < d.P; ++p) acc += G[p * d.N + n] * xt[p];
          dBt[n] = delta * acc;
        }
        double gh = 0.0;  // <G, h_{t-1}>
        for (int64_t i = 0; i < PN; ++i) gh += G[i] * h_prev[i];
        const double ddelta = gxb + Ah * alpha * gh;
        const double dv = ddelta * softplus_grad(v);
        ddt[tok(t)] = dv;
        dbias_acc += dv;
        dA_acc += delta * alpha * gh;
        double dyx = 0.0;
        for (int64_t p = 0; p < d.P; ++p) dyx += dyt[p] * xt[p];
        dD_acc += dyx;
        // G <- alpha G : dL/dh_{t-1} before adding dy_{t-1}
        for (int64_t i = 0; i < PN; ++i) G[i] *= alpha;
      }
    }
    if (dinit) std::memcpy(dinit + (b * d.H + h) * PN, G.data(), sizeof(double) * PN);
    dA_bh[task] = dA_acc;
    dD_bh[task] = dD_acc;
    dbias_bh[task] = dbias_acc;
  });

  // Sum the head shares of each group, heads in increasing order.
  parallel_for(d.Bt * d.T, nthreads, [&](int64_t bt) {
    for (int64_t g = 0; g < d.G; ++g) {
      double* oB = dB + (bt * d.G + g) * d.N;
      double* oC = dC + (bt * d.G + g) * d.N;
      for (int64_t n = 0; n < d.N; ++n) {
        double sb = 0.0, sc = 0.0;
        for (int64_t h = g * hpg; h < (g + 1) * hpg; ++h) {
          sb += dB_h[(bt * d.H + h) * d.N + n];
          sc += dC_h[(bt * d.H + h) * d.N + n];
        }
        oB[n] = sb;
        oC[n] = sc;
      }
    }
  });
  for (int64_t h = 0; h < d.H; ++h) {
    double a = 0.0, dd = 0.0, bb = 0.0;
    for (int64_t b = 0; b < d.Bt; ++b) {
      a += dA_bh[b * d.H + h];
      dd += dD_bh[b * d.H + h];
      bb += dbias_bh[b * d.H + h];
    }
    dA[h] = a;
    if (dD) dD[h] = dd;
    if (ddt_bias) ddt_bias[h] = bb;
  }
  return 0;
}

}  // extern "C"
