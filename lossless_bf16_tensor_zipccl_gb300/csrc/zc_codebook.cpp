// zc_codebook.cpp -- code tables of the exponent coder (host side).
//
// "ZipCCL: Efficient Lossless Data Compression of Communication Collectives
// for Accelerating LLM Training", abstract technique (1) and the shd-paper
// summary's key design: the exponent code comes from the Gaussian density, so
// frequent exponents get short codewords and no histogram is taken online.
//
// The tables the library codes with are the frozen integers of format v1
// (zc_format.h); rebuild_phase_table derives them again from the closed form,
// for the tests that check the frozen copy.
//
// For X ~ N(0, sigma^2) the biased BF16 exponent e has
//   P(e) = P(2^(e-127) <= |X| < 2^(e-126)),  1 <= e <= 254,
//   P(0) = P(|X| < 2^-126).
// The code is built for sigma = 2^(q/16).  On the normal range P only shifts
// with floor(q/16), so the tables depend on the phase r = q mod 16.  For each
// phase: the 15 consecutive exponents of largest mass form the window (lowest
// start on ties), the escape symbol takes the rest of the mass, and the code
// lengths are the optimal prefix code limited to 10 bits, found here by an
// exact dynamic program over Kraft sums in units of 2^-10.
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "zc_codebook.h"
#include "zc_format.h"

namespace zc {
namespace {

// P(a <= |X| < b) for X ~ N(0, sigma^2); erfc on the upper side keeps the
// relative accuracy of the tail.
double gaussian_abs_mass(double a, double b, double sigma) {
  const double s = sigma * sqrt(2.0);
  const double ua = a / s, ub = b / s;
  if (ua >= 0.5) return erfc(ua) - erfc(ub);
  return erf(ub) - erf(ua);
}

void exponent_masses(double sigma, double* p) {
  p[0] = gaussian_abs_mass(0.0, ldexp(1.0, -126), sigma);
  for (int e = 1; e <= 254; ++e) p[e] = gaussian_abs_mass(ldexp(1.0, e - 127), ldexp(1.0, e - 126), sigma);
  p[255] = 0.0;
}

// Minimum-cost length vector with every length in [1, lmax] and
// sum 2^-len <= 1.  dp over symbols in index order; state = Kraft units used.
void optimal_limited_lengths(const double* w, int n, int lmax, uint8_t* lens) {
  const int units = 1 << lmax;
  const double inf = 1e300;
  std::vector<double> dp((size_t)(n + 1) * (units + 1), inf);
  std::vector<uint8_t> pick((size_t)(n + 1) * (units + 1), 0);
  auto at = [&](int i, int k) -> size_t { return (size_t)i * (units + 1) + k; };
  dp[at(0, 0)] = 0.0;
  for (int i = 0; i < n; ++i) {
    for (int k = 0; k <= units; ++k) {
      const double cur = dp[at(i, k)];
      if (cur >= inf) continue;
      for (int len = 1; len <= lmax; ++len) {
        const int k2 = k + (1 << (lmax - len));
        if (k2 > units) continue;
        const double c = cur + w[i] * len;
        if (c < dp[at(i + 1, k2)]) {
          dp[at(i + 1, k2)] = c;
          pick[at(i + 1, k2)] = (uint8_t)len;
        }
      }
    }
  }
  int best_k = units;
  for (int k = 0; k <= units; ++k)
    if (dp[at(n, k)] < dp[at(n, best_k)]) best_k = k;
  for (int i = n, k = best_k; i > 0; --i) {
    const int len = pick[at(i, k)];
    lens[i - 1] = (uint8_t)len;
    k -= 1 << (lmax - len);
  }
}

PhaseTable g_tables[16];
std::once_flag g_once;

// The frozen tables of format v1 (zc_format.h), unpacked once.
void load_frozen() {
  for (int r = 0; r < 16; ++r) {
    g_tables[r].base_offset = kPhaseBaseOffset[r];
    g_tables[r].lens_packed = kPhaseLens[r];
    for (int s = 0; s < kNsym; ++s) g_tables[r].lens[s] = (uint8_t)((kPhaseLens[r] >> (4 * s)) & 15);
  }
}

}  // namespace

void rebuild_phase_table(int r, PhaseTable* out) {
  double p[256];
  exponent_masses(pow(2.0, r / 16.0), p);
  int best = 0;
  double best_mass = -1.0;
  for (int b = 0; b + kWindow <= 255; ++b) {
    double m = 0.0;
    for (int i = 0; i < kWindow; ++i) m += p[b + i];
    if (m > best_mass) {
      best_mass = m;
      best = b;
    }
  }
  double w[kNsym];
  double in_window = 0.0;
  for (int i = 0; i < kWindow; ++i) {
    w[i] = p[best + i];
    in_window += w[i];
  }
  w[kEsc] = 1.0 - in_window;
  out->base_offset = best - 127;
  optimal_limited_lengths(w, kNsym, kLmax, out->lens);
  uint64_t packed = 0;
  for (int s = 0; s < kNsym; ++s) packed |= (uint64_t)out->lens[s] << (4 * s);
  out->lens_packed = packed;
}

const PhaseTable* phase_tables() {
  std::call_once(g_once, load_frozen);
  return g_tables;
}

int base_for_q(int q) {
  const int k = q >= 0 ? q / 16 : -((15 - q) / 16);  // floor(q / 16)
  int b = k + 127 + phase_tables()[q - 16 * k].base_offset;
  return b < 0 ? 0 : (b > 240 ? 240 : b);
}

double expected_exponent_bits(double sigma, int q) {
  double p[256];
  exponent_masses(sigma, p);
  const int k = q >= 0 ? q / 16 : -((15 - q) / 16);
  const PhaseTable& t = phase_tables()[q - 16 * k];
  const int base = base_for_q(q);
  double bits = 0.0;
  for (int e = 0; e < 256; ++e) {
    const int x = e - base;
    bits += p[e] * (x >= 0 && x < kWindow ? (double)t.lens[x] : (double)(t.lens[kEsc] + 8));
  }
  return bits;
}

}  // namespace zc
