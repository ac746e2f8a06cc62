// zc_codebook.h -- per-phase code tables (built once on the host).
#pragma once
#include <stdint.h>

namespace zc {

struct PhaseTable {
  int base_offset;      // window start - 127 for q in [0, 16)
  uint8_t lens[16];     // code lengths of symbols 0..15 (15 = escape)
  uint64_t lens_packed; // lens[s] at bits 4s..4s+3
};

// The 16 phase tables of format v1 (the frozen integers, unpacked on first
// use; thread-safe).
const PhaseTable* phase_tables();

// Phase r rebuilt from the closed-form masses by the exact dynamic program
// (double precision, libm erf/erfc): for checking the frozen tables.
void rebuild_phase_table(int r, PhaseTable* out);

// Window start for scale q: floor(q/16) + 127 + the phase's offset, clamped
// to [0, 240] so that the window stays inside [0, 254].
int base_for_q(int q);

// Expected code bits of one exponent of X ~ N(0, sigma^2) under the code for
// scale q (window and lengths of phase q mod 16; an escape costs its
// codeword and 8 raw bits).
double expected_exponent_bits(double sigma, int q);

}  // namespace zc
