// Host side of libsvdq: offline weight packing for the SVDQ W4A4 linear and
// the AWQ W4A16 GEMV, and the calibration statistic of the smoothing step.
//
// SVDQ packing follows the SVDQuant paragraph of dothoosh.com, "How Nunchaku
// Lite halves the VRAM of diffusion models": activation outliers are moved
// into the weights (smoothing by lambda), the hardest part of the smoothed
// weight is kept as a 16-bit low-rank branch, and the residual is quantized
// to NVFP4 (config block: group size 16, rank 32).  The truncated SVD is this
// file's own: randomized subspace iteration (Halko, Martinsson and Tropp,
// "Finding structure with randomness", SIAM Review 2011, algorithm 4.4) with
// classical Gram-Schmidt applied twice for orthonormalization, and a one-sided
// Jacobi SVD (Hestenes) of the small projected factor; small matrices take the
// one-sided Jacobi SVD directly.
//
// Compiled with -ffp-contract=off: the residual and every rounding decision
// are evaluated as written (one rounding per operation, no fused multiply-add)
// so that the packed codes are a deterministic function of the inputs.
#include <algorithm>
#include <atomic>
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include "../../include/svdq.h"

namespace {

// ---------------------------------------------------------------- threading
int num_threads() {
  unsigned h = std::thread::hardware_concurrency();
  if (h == 0) h = 1;
  return (int)std::min(h, 64u);
}

// f(begin, end) over contiguous chunks of [0, n); deterministic partition
template <class F>
void parallel_for(int64_t n, F f) {
  const int nt = (int)std::min<int64_t>(num_threads(), std::max<int64_t>(n, 1));
  if (nt <= 1 || n < 2) {
    f((int64_t)0, n);
    return;
  }
  std::vector<std::thread> th;
  th.reserve(nt);
  for (int t = 0; t < nt; ++t) {
    const int64_t b = n * t / nt, e = n * (t + 1) / nt;
    th.emplace_back([=] { f(b, e); });
  }
  for (auto& x : th) x.join();
}

// ---------------------------------------------------------------- formats
// nearest bfloat16 of a double (ties to even), as bits
uint16_t bf16_from_double(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const double a = std::fabs(x);
  uint32_t sign = std::signbit(x) ? 0x8000u : 0u;
  double r;
  if (a == 0.0) {
    return (uint16_t)sign;
  } else if (a < std::ldexp(1.0, -126)) {
    r = std::ldexp(std::nearbyint(std::ldexp(a, 133)), -133);
  } else {
    int e;
    const double m = std::frexp(a, &e);  // a = m 2^e, m in [0.5, 1)
    r = std::ldexp(std::nearbyint(std::ldexp(m, 8)), e - 8);
  }
  if (r > std::ldexp(255.0, 120)) return (uint16_t)(sign | 0x7F80u);  // overflow -> inf
  const float f = (float)r;                                          // exact
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}
double bf16_to_double(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// nearest binary16 of a double (ties to even): value and bits
double f16_round(double x, uint16_t* bits) {
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  const double a = std::fabs(x);
  if (std::isnan(x)) {
    *bits = 0x7E00;
    return x;
  }
  if (a >= 65520.0) {  // rounds past the largest finite value
    *bits = sign | 0x7C00;
    return std::copysign(INFINITY, x);
  }
  if (a < std::ldexp(1.0, -14)) {  // subnormal: step 2^-24
    const double t = std::nearbyint(std::ldexp(a, 24));
    *bits = (uint16_t)(sign | (uint16_t)t);  // t == 1024 is the smallest normal
    return std::copysign(std::ldexp(t, -24), x);
  }
  int e;
  const double m = std::frexp(a, &e);  // a = m 2^e
  int E = e - 1;
  int mant = (int)std::nearbyint((2.0 * m - 1.0) * 1024.0);
  if (mant == 1024) {
    mant = 0;
    E += 1;
  }
  *bits = (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)mant);
  return std::copysign(std::ldexp(1.0 + mant / 1024.0, E), x);
}

// e4m3 byte of a non-negative value: nearest, ties to even, saturating at 448
uint32_t rne_e4m3(double v) {
  if (!(v > 0.0)) return 0;
  if (v >= 448.0) return 0x7E;
  int e;
  const double m = std::frexp(v, &e);
  const int E = e - 1;           // v = (2m) 2^E, 2m in [1, 2)
  if (E < -6) return (uint32_t)std::nearbyint(std::ldexp(v, 9));  // subnormal step 2^-9
  int mant = (int)std::nearbyint((2.0 * m - 1.0) * 8.0);
  int ex = E + 7;
  if (mant == 8) {
    mant = 0;
    ex += 1;
  }
  const uint32_t code = ((uint32_t)ex << 3) | (uint32_t)mant;
  return std::min(code, 0x7Eu);
}
double e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xF, m = b & 7;
  return e == 0 ? std::ldexp((double)m, -9) : std::ldexp(1.0 + m / 8.0, (int)e - 7);
}

// e2m1 code of a value: nearest of {0,.5,1,1.5,2,3,4,6}, ties to the even
// code, saturating; sign bit = the value's sign bit
uint32_t rne_e2m1(double v) {
  const uint32_t sign = std::signbit(v) ? 8u : 0u;
  const double a = std::fabs(v);
  const uint32_t c = (uint32_t)(a > 0.25) + (uint32_t)(a >= 0.75) + (uint32_t)(a > 1.25) +
                     (uint32_t)(a >= 1.75) + (uint32_t)(a > 2.5) + (uint32_t)(a >= 3.5) +
                     (uint32_t)(a > 5.0);
  return sign | c;
}

// offset of scale (r, c) in the 512-byte tile layout with C scale columns
inline size_t sf_offset(size_t r, size_t c, size_t C) {
  return ((r / 128) * (C / 4) + c / 4) * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);
}

// ---------------------------------------------------------------- linear algebra
// Tall thin matrices are stored column-major: col j is v[j * n .. j * n + n).
struct Thin {
  int64_t n = 0;
  int l = 0;
  std::vector<double> v;
  Thin() = default;
  Thin(int64_t n_, int l_) : n(n_), l(l_), v((size_t)n_ * l_, 0.0) {}
  double* col(int j) { return v.data() + (size_t)j * n; }
  const double* col(int j) const { return v.data() + (size_t)j * n; }
};

double dot(const double* a, const double* b, int64_t n) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) s += a[i] * b[i];
  return s;
}

// counter-based standard normal (SplitMix64 mixing + Box-Muller)
uint64_t splitmix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}
double gauss(uint64_t idx) {
  const double u1 = ((splitmix64(2 * idx) >> 11) + 1.0) * 0x1.0p-53;  // (0, 1]
  const double u2 = (splitmix64(2 * idx + 1) >> 11) * 0x1.0p-53;
  return std::sqrt(-2.0 * std::log(u1)) * std::cos(6.283185307179586 * u2);
}

// Orthonormalize the columns in place (classical Gram-Schmidt, twice).
// Columns that vanish are replaced by a deterministic random direction.
// If R is given (l x l, row-major), it receives Q^T Y.
void orthonormalize(Thin& Y, std::vector<double>* R, uint64_t seed) {
  const int64_t n = Y.n;
  const int l = Y.l;
  if (R) R->assign((size_t)l * l, 0.0);
  std::vector<double> coef(l);
  for (int j = 0; j < l; ++j) {
    double* v = Y.col(j);
    const double norm0 = std::sqrt(dot(v, v, n));
    for (int pass = 0; pass < 2; ++pass) {
      // coefficients against all previous columns (classical GS: from the
      // same vector), computed in parallel over i
      parallel_for(j, [&](int64_t b, int64_t e) {
        for (int64_t i = b; i < e; ++i) coef[i] = dot(Y.col((int)i), v, n);
      });
      parallel_for(n, [&](int64_t b, int64_t e) {
        for (int i = 0; i < j; ++i) {
          const double c = coef[i];
          const double* q = Y.col(i);
          for (int64_t t = b; t < e; ++t) v[t] -= c * q[t];
        }
      });
      if (R)
        for (int i = 0; i < j; ++i) (*R)[(size_t)i * l + j] += coef[i];
    }
    double nv = std::sqrt(dot(v, v, n));
    if (!(nv > 1e-13 * std::max(norm0, 1e-300))) {
      // numerically dependent column: a random direction orthogonal to the rest
      for (int64_t t = 0; t < n; ++t) v[t] = gauss(seed + (uint64_t)j * (uint64_t)n + t);
      for (int pass = 0; pass < 2; ++pass)
        for (int i = 0; i < j; ++i) {
          const double c = dot(Y.col(i), v, n);
          const double* q = Y.col(i);
          for (int64_t t = 0; t < n; ++t) v[t] -= c * q[t];
        }
      if (R) (*R)[(size_t)j * l + j] = 0.0;
      nv = std::sqrt(dot(v, v, n));
      for (int64_t t = 0; t < n; ++t) v[t] /= nv;
      continue;
    }
    if (R) (*R)[(size_t)j * l + j] = nv;
    for (int64_t t = 0; t < n; ++t) v[t] /= nv;
  }
}

// One-sided Jacobi SVD of the n columns of C (each of length m; n <= m or
// not): on return C holds U*Sigma (orthogonal columns), V (n x n, row-major)
// the accumulated rotations, so that C_in = U Sigma V^T.
void jacobi_svd(Thin& C, std::vector<double>& V) {
  const int n = C.l;
  const int64_t m = C.n;
  V.assign((size_t)n * n, 0.0);
  for (int i = 0; i < n; ++i) V[(size_t)i * n + i] = 1.0;
  const double eps = 1e-15;
  for (int sweep = 0; sweep < 60; ++sweep) {
    bool rotated = false;
    for (int p = 0; p < n - 1; ++p) {
      for (int q = p + 1; q < n; ++q) {
        double* cp = C.col(p);
        double* cq = C.col(q);
        const double alpha = dot(cp, cp, m), beta = dot(cq, cq, m), gamma = dot(cp, cq, m);
        if (std::fabs(gamma) <= eps * std::sqrt(alpha * beta) || gamma == 0.0) continue;
        rotated = true;
        const double zeta = (beta - alpha) / (2.0 * gamma);
        const double t = (zeta >= 0 ? 1.0 : -1.0) / (std::fabs(zeta) + std::sqrt(1.0 + zeta * zeta));
        const double c = 1.0 / std::sqrt(1.0 + t * t), s = c * t;
        for (int64_t i = 0; i < m; ++i) {
          const double x = cp[i], y = cq[i];
          cp[i] = c * x - s * y;
          cq[i] = s * x + c * y;
        }
        for (int i = 0; i < n; ++i) {
          double& x = V[(size_t)i * n + p];
          double& y = V[(size_t)i * n + q];
          const double xv = x, yv = y;
          x = c * xv - s * yv;
          y = s * xv + c * yv;
        }
      }
    }
    if (!rotated) break;
  }
}

// Y(:, j) = A * T(:, j) for A (N x K row-major), T (K x l) -> Y (N x l)
void mul_A(const std::vector<double>& A, int64_t N, int64_t K, const Thin& T, Thin& Y) {
  Y = Thin(N, T.l);
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t r = b; r < e; ++r) {
      const double* a = A.data() + (size_t)r * K;
      for (int j = 0; j < T.l; ++j) Y.col(j)[r] = dot(a, T.col(j), K);
    }
  });
}
// Z(:, j) = A^T * Q(:, j) for A (N x K), Q (N x l) -> Z (K x l); rows of A
// accumulated in increasing order
void mul_At(const std::vector<double>& A, int64_t N, int64_t K, const Thin& Q, Thin& Z) {
  Z = Thin(K, Q.l);
  parallel_for(K, [&](int64_t b, int64_t e) {
    for (int64_t r = 0; r < N; ++r) {
      const double* a = A.data() + (size_t)r * K;
      for (int j = 0; j < Q.l; ++j) {
        const double c = Q.col(j)[r];
        double* z = Z.col(j);
        for (int64_t k = b; k < e; ++k) z[k] += c * a[k];
      }
    }
  });
}

// Rank-r factors of A (N x K row-major): U (N x r), sigma (r), Vk (K x r)
// with A ~= U diag(sigma) Vk^T.
void truncated_svd(const std::vector<double>& A, int64_t N, int64_t K, int r, Thin& U,
                   std::vector<double>& sigma, Thin& Vk) {
  const int64_t mn = std::min(N, K);
  const int l_want = r + 16;
  U = Thin(N, r);
  Vk = Thin(K, r);
  sigma.assign(r, 0.0);
  std::vector<double> Vrot;
  if (mn <= 256 || l_want >= mn) {
    // direct one-sided Jacobi on the shorter side
    if (K <= N) {
      Thin C(N, (int)K);  // columns of A
      parallel_for(K, [&](int64_t b, int64_t e) {
        for (int64_t k = b; k < e; ++k)
          for (int64_t n = 0; n < N; ++n) C.col((int)k)[n] = A[(size_t)n * K + k];
      });
      jacobi_svd(C, Vrot);  // A = Uc S Vrot^T
      std::vector<double> nrm(K);
      for (int j = 0; j < (int)K; ++j) nrm[j] = std::sqrt(dot(C.col(j), C.col(j), N));
      std::vector<int> ord(K);
      for (int j = 0; j < (int)K; ++j) ord[j] = j;
      std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return nrm[a] > nrm[b]; });
      for (int i = 0; i < r; ++i) {
        const int j = ord[i];
        sigma[i] = nrm[j];
        for (int64_t n = 0; n < N; ++n) U.col(i)[n] = nrm[j] > 0 ? C.col(j)[n] / nrm[j] : 0.0;
        for (int64_t k = 0; k < K; ++k) Vk.col(i)[k] = Vrot[(size_t)k * K + j];
      }
    } else {
      Thin C(K, (int)N);  // columns of A^T = rows of A
      for (int64_t n = 0; n < N; ++n)
        std::memcpy(C.col((int)n), A.data() + (size_t)n * K, sizeof(double) * K);
      jacobi_svd(C, Vrot);  // A^T = Uc S Vrot^T  ->  A = Vrot S Uc^T
      std::vector<double> nrm(N);
      for (int j = 0; j < (int)N; ++j) nrm[j] = std::sqrt(dot(C.col(j), C.col(j), K));
      std::vector<int> ord(N);
      for (int j = 0; j < (int)N; ++j) ord[j] = j;
      std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return nrm[a] > nrm[b]; });
      for (int i = 0; i < r; ++i) {
        const int j = ord[i];
        sigma[i] = nrm[j];
        for (int64_t k = 0; k < K; ++k) Vk.col(i)[k] = nrm[j] > 0 ? C.col(j)[k] / nrm[j] : 0.0;
        for (int64_t n = 0; n < N; ++n) U.col(i)[n] = Vrot[(size_t)n * N + j];
      }
    }
    return;
  }
  // randomized subspace iteration
  const int l = l_want;
  const int q_iters = 4;
  Thin Om(K, l);
  for (int j = 0; j < l; ++j)
    for (int64_t k = 0; k < K; ++k) Om.col(j)[k] = gauss(((uint64_t)j << 40) ^ (uint64_t)k);
  Thin Y, Z;
  mul_A(A, N, K, Om, Y);
  orthonormalize(Y, nullptr, 0x1000);
  for (int it = 0; it < q_iters; ++it) {
    mul_At(A, N, K, Y, Z);
    orthonormalize(Z, nullptr, 0x2000 + it);
    mul_A(A, N, K, Z, Y);
    orthonormalize(Y, nullptr, 0x3000 + it);
  }
  // B^T = A^T Q = Q2 R2;  R2 = Ur S J^T  ->  A ~= (Q J) S (Q2 Ur)^T
  Thin Bt;
  mul_At(A, N, K, Y, Bt);
  std::vector<double> R2;
  orthonormalize(Bt, &R2, 0x4000);  // Bt now holds Q2
  Thin Rc(l, l);
  for (int j = 0; j < l; ++j)
    for (int i = 0; i < l; ++i) Rc.col(j)[i] = R2[(size_t)i * l + j];
  jacobi_svd(Rc, Vrot);
  std::vector<double> nrm(l);
  for (int j = 0; j < l; ++j) nrm[j] = std::sqrt(dot(Rc.col(j), Rc.col(j), l));
  std::vector<int> ord(l);
  for (int j = 0; j < l; ++j) ord[j] = j;
  std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) { return nrm[a] > nrm[b]; });
  for (int i = 0; i < r; ++i) {
    const int j = ord[i];
    sigma[i] = nrm[j];
    // right factor: Q2 * (Rc(:, j) / nrm)   left factor: Q * J(:, j)
    double* vk = Vk.col(i);
    double* u = U.col(i);
    for (int t = 0; t < l; ++t) {
      const double cr = nrm[j] > 0 ? Rc.col(j)[t] / nrm[j] : 0.0;
      const double cj = Vrot[(size_t)t * l + j];
      const double* q2 = Bt.col(t);
      const double* q1 = Y.col(t);
      for (int64_t k = 0; k < K; ++k) vk[k] += cr * q2[k];
      for (int64_t n = 0; n < N; ++n) u[n] += cj * q1[n];
    }
  }
}

bool all_finite(const float* p, size_t n) {
  for (size_t i = 0; i < n; ++i)
    if (!std::isfinite(p[i])) return false;
  return true;
}

// Round-to-nearest for the scope of a packing call (the caller's mode is
// put back on every return path).
struct RoundingScope {
  int saved = std::fegetround();
  RoundingScope() { std::fesetround(FE_TONEAREST); }
  ~RoundingScope() { std::fesetround(saved); }
};

// Steps shared by the NVFP4 and INT4 packers: (1) smoothing, inv_lambda;
// (2) the rank-r factors of W_hat^T, L1s = bf16(inv (.) L1) written to L1s
// [rank][K] and bf16(L2) returned as doubles l2d [rank][N]; (3) the residual
// R[n][k] = (W[n][k] - sum_i L1s[i][k] L2[i][n]) / inv[k] (sum over i
// ascending) returned in A [N][K].  False if the smoothing is not finite.
bool factor_and_residual(const float* W, int N, int K, const float* x_absmax, int rank,
                         float* inv_lambda, uint16_t* L1s, std::vector<double>& A,
                         std::vector<double>& l2d) {
  const int64_t NN = N, KK = K;
  // (1) smoothing: lambda_j = sqrt(max|X_j| / max|W_j|), clamped
  std::vector<double> inv(K);
  for (int k = 0; k < K; ++k) {
    double wm = 0.0;
    for (int n = 0; n < N; ++n) wm = std::max(wm, (double)std::fabs(W[(size_t)n * K + k]));
    const double xm = (double)x_absmax[k];
    double lam = 1.0;
    if (xm > 0.0 && wm > 0.0) lam = std::sqrt(xm / wm);
    lam = std::min(std::max(lam, std::ldexp(1.0, -20)), std::ldexp(1.0, 20));
    inv_lambda[k] = (float)(1.0 / lam);
    inv[k] = (double)inv_lambda[k];
    if (!std::isfinite(inv[k])) return false;
  }
  // (2) W_hat = W diag(1/inv_lambda) (N x K); its transpose is the K x N
  // matrix the method factors
  A.assign((size_t)NN * KK, 0.0);
  parallel_for(NN, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n)
      for (int64_t k = 0; k < KK; ++k)
        A[(size_t)n * KK + k] = (double)W[(size_t)n * KK + k] / inv[k];
  });
  Thin U, Vk;
  std::vector<double> sig;
  truncated_svd(A, NN, KK, rank, U, sig, Vk);
  // W_hat^T ~= Vk S U^T  ->  L1 = Vk S (K x r), L2 = U^T (r x N)
  std::vector<uint16_t> l1s((size_t)rank * K), l2((size_t)rank * N);
  for (int i = 0; i < rank; ++i) {
    for (int k = 0; k < K; ++k)
      l1s[(size_t)i * K + k] = bf16_from_double(inv[k] * (Vk.col(i)[k] * sig[i]));
    for (int n = 0; n < N; ++n) l2[(size_t)i * N + n] = bf16_from_double(U.col(i)[n]);
  }
  std::memcpy(L1s, l1s.data(), l1s.size() * sizeof(uint16_t));
  std::vector<double> l1d((size_t)rank * K);
  l2d.assign((size_t)rank * N, 0.0);
  for (size_t i = 0; i < l1d.size(); ++i) l1d[i] = bf16_to_double(l1s[i]);
  for (size_t i = 0; i < l2d.size(); ++i) l2d[i] = bf16_to_double(l2[i]);
  // (3) residual, stored over A
  parallel_for(NN, [&](int64_t b, int64_t e) {
    std::vector<double> acc(KK);
    for (int64_t n = b; n < e; ++n) {
      std::fill(acc.begin(), acc.end(), 0.0);
      for (int i = 0; i < rank; ++i) {
        const double c = l2d[(size_t)i * N + n];
        const double* l1 = l1d.data() + (size_t)i * K;
        for (int64_t k = 0; k < KK; ++k) acc[k] += l1[k] * c;
      }
      double* rrow = A.data() + (size_t)n * KK;
      for (int64_t k = 0; k < KK; ++k)
        rrow[k] = ((double)W[(size_t)n * KK + k] - acc[k]) / inv[k];
    }
  });
  return true;
}

}  // namespace

extern "C" {

svdq_status svdq_calib_absmax(const uint16_t* X_bf16, int64_t M, int64_t K, float* x_absmax) {
  if (M < 0 || K <= 0) return SVDQ_ERR_SHAPE;
  if (!x_absmax || (M > 0 && !X_bf16)) return SVDQ_ERR_NULL;
  for (int64_t k = 0; k < K; ++k) x_absmax[k] = 0.0f;
  for (int64_t m = 0; m < M; ++m) {
    const uint16_t* row = X_bf16 + m * K;
    for (int64_t k = 0; k < K; ++k) {
      const float a = (float)std::fabs(bf16_to_double(row[k]));
      if (a > x_absmax[k]) x_absmax[k] = a;
    }
  }
  return SVDQ_OK;
}

svdq_status svdq_pack_weights(const float* W, int N, int K, const float* x_absmax, int rank,
                              float* inv_lambda, uint16_t* L1s, uint16_t* L2s,
                              uint8_t* w_codes, uint8_t* w_scales, float* w_tensor_scale) {
  if (N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return SVDQ_ERR_SHAPE;
  if (rank < 1 || rank > std::min(N, K)) return SVDQ_ERR_RANK;
  if (!W || !x_absmax || !inv_lambda || !L1s || !L2s || !w_codes || !w_scales || !w_tensor_scale)
    return SVDQ_ERR_NULL;
  if (!all_finite(W, (size_t)N * K) || !all_finite(x_absmax, (size_t)K)) return SVDQ_ERR_VALUE;
  for (int k = 0; k < K; ++k)
    if (x_absmax[k] < 0.0f) return SVDQ_ERR_VALUE;
  RoundingScope rounding;
  try {
    const int64_t NN = N, KK = K;
    std::vector<double> A, l2d;
    if (!factor_and_residual(W, N, K, x_absmax, rank, inv_lambda, L1s, A, l2d))
      return SVDQ_ERR_VALUE;
    double amax = 0.0;
    for (size_t i = 0; i < A.size(); ++i) amax = std::max(amax, std::fabs(A[i]));
    if (!std::isfinite(amax)) return SVDQ_ERR_VALUE;
    // (4) tensor scale: smallest power of two p with 6*448*p >= max|R|
    double sT = 1.0;
    if (amax > 0.0) {
      const double bound = 6.0 * 448.0;
      int e = (int)std::ceil(std::log2(amax / bound));
      while (bound * std::ldexp(1.0, e) < amax) ++e;
      while (bound * std::ldexp(1.0, e - 1) >= amax) --e;
      sT = std::ldexp(1.0, e);
    }
    if (sT < std::ldexp(1.0, -100) || sT > std::ldexp(1.0, 100)) return SVDQ_ERR_VALUE;
    *w_tensor_scale = (float)sT;
    // L2s[n][i] = bf16(L2)[i][n] / s_T: exact, s_T is a power of two
    for (int n = 0; n < N; ++n)
      for (int i = 0; i < rank; ++i)
        L2s[(size_t)n * rank + i] = bf16_from_double(l2d[(size_t)i * N + n] / sT);
    // (5) block scales and codes, 16 consecutive k of one output channel
    const size_t C = (size_t)K / 16;
    parallel_for(NN, [&](int64_t b, int64_t e) {
      for (int64_t n = b; n < e; ++n) {
        const double* rrow = A.data() + (size_t)n * KK;
        for (size_t cb = 0; cb < C; ++cb) {
          const double* blk = rrow + cb * 16;
          double bmax = 0.0;
          for (int i = 0; i < 16; ++i) bmax = std::max(bmax, std::fabs(blk[i]));
          const uint32_t sb = rne_e4m3(bmax / (6.0 * sT));
          w_scales[sf_offset((size_t)n, cb, C)] = (uint8_t)sb;
          const double scale = e4m3_value(sb) * sT;
          uint8_t* out = w_codes + (size_t)n * (KK / 2) + cb * 8;
          for (int i = 0; i < 8; ++i) {
            uint32_t lo = 0, hi = 0;
            if (scale > 0.0) {
              lo = rne_e2m1(blk[2 * i] / scale);
              hi = rne_e2m1(blk[2 * i + 1] / scale);
            }
            out[i] = (uint8_t)(lo | (hi << 4));
          }
        }
      }
    });
  } catch (const std::bad_alloc&) {
    return SVDQ_ERR_NOMEM;
  }
  return SVDQ_OK;
}

svdq_status svdq_pack_weights_int4(const float* W, int N, int K, const float* x_absmax, int rank,
                                   float* inv_lambda, uint16_t* L1s, uint16_t* L2,
                                   uint8_t* w_codes, uint16_t* w_scales) {
  if (N <= 0 || K <= 0 || N % 128 != 0 || K % 128 != 0) return SVDQ_ERR_SHAPE;
  if (rank < 1 || rank > std::min(N, K)) return SVDQ_ERR_RANK;
  if (!W || !x_absmax || !inv_lambda || !L1s || !L2 || !w_codes || !w_scales)
    return SVDQ_ERR_NULL;
  if (!all_finite(W, (size_t)N * K) || !all_finite(x_absmax, (size_t)K)) return SVDQ_ERR_VALUE;
  for (int k = 0; k < K; ++k)
    if (x_absmax[k] < 0.0f) return SVDQ_ERR_VALUE;
  RoundingScope rounding;
  try {
    const int64_t NN = N, KK = K;
    std::vector<double> A, l2d;
    if (!factor_and_residual(W, N, K, x_absmax, rank, inv_lambda, L1s, A, l2d))
      return SVDQ_ERR_VALUE;
    for (size_t i = 0; i < A.size(); ++i)
      if (!std::isfinite(A[i])) return SVDQ_ERR_VALUE;
    for (int n = 0; n < N; ++n)
      for (int i = 0; i < rank; ++i)
        L2[(size_t)n * rank + i] = bf16_from_double(l2d[(size_t)i * N + n]);
    // symmetric groups of 64 consecutive k of one output channel:
    // s = bf16(amax / 7), q = clamp(RNE(R / s), -8, 7), a zero scale gives 0
    const size_t G = (size_t)K / 64;
    parallel_for(NN, [&](int64_t b, int64_t e) {
      for (int64_t n = b; n < e; ++n) {
        const double* rrow = A.data() + (size_t)n * KK;
        for (size_t g = 0; g < G; ++g) {
          const double* grp = rrow + g * 64;
          double gmax = 0.0;
          for (int i = 0; i < 64; ++i) gmax = std::max(gmax, std::fabs(grp[i]));
          const uint16_t sbits = bf16_from_double(gmax / 7.0);
          w_scales[(size_t)n * G + g] = sbits;
          const double s = bf16_to_double(sbits);
          uint8_t* out = w_codes + (size_t)n * (KK / 2) + g * 32;
          for (int i = 0; i < 32; ++i) {
            int q[2] = {0, 0};
            for (int h = 0; h < 2; ++h)
              if (s > 0.0)
                q[h] = (int)std::min(7.0, std::max(-8.0, std::nearbyint(grp[2 * i + h] / s)));
            out[i] = (uint8_t)((q[0] & 0xF) | ((q[1] & 0xF) << 4));
          }
        }
      }
    });
  } catch (const std::bad_alloc&) {
    return SVDQ_ERR_NOMEM;
  }
  return SVDQ_OK;
}

svdq_status awq_pack_weights(const float* W, int N, int K, int group_size, uint8_t* qweight,
                             uint16_t* scales, uint16_t* zeros) {
  if (N <= 0 || K <= 0 || group_size != 64 || K % 64 != 0) return SVDQ_ERR_SHAPE;
  if (!W || !qweight || !scales || !zeros) return SVDQ_ERR_NULL;
  if (!all_finite(W, (size_t)N * K)) return SVDQ_ERR_VALUE;
  const int saved_round = std::fegetround();
  std::fesetround(FE_TONEAREST);
  const int G = K / 64;
  parallel_for(N, [&](int64_t b, int64_t e) {
    for (int64_t n = b; n < e; ++n) {
      for (int g = 0; g < G; ++g) {
        const float* w = W + (size_t)n * K + (size_t)g * 64;
        double mx = w[0], mn = w[0];
        for (int i = 1; i < 64; ++i) {
          mx = std::max(mx, (double)w[i]);
          mn = std::min(mn, (double)w[i]);
        }
        uint16_t sbits, zbits;
        double s = f16_round((mx - mn) / 15.0, &sbits);
        if (mx == mn || s == 0.0) s = f16_round(1.0, &sbits);
        const double zc = std::min(std::max(-mn / s, -65504.0), 65504.0);
        const double z = f16_round(zc, &zbits);
        scales[(size_t)n * G + g] = sbits;
        zeros[(size_t)n * G + g] = zbits;
        uint8_t* out = qweight + (size_t)n * (K / 2) + (size_t)g * 32;
        for (int i = 0; i < 32; ++i) {
          double q0 = std::nearbyint((double)w[2 * i] / s + z);
          double q1 = std::nearbyint((double)w[2 * i + 1] / s + z);
          q0 = std::min(std::max(q0, 0.0), 15.0);
          q1 = std::min(std::max(q1, 0.0), 15.0);
          out[i] = (uint8_t)((uint32_t)q0 | ((uint32_t)q1 << 4));
        }
      }
    }
  });
  std::fesetround(saved_round);
  return SVDQ_OK;
}

}  // extern "C"
