// zc_codebook.h -- per-phase code tables (built once on the host).
#pragma once
#include <stdint.h>

namespace zc {

struct PhaseTable {
  int base_offset;      // window start - 127 for q in [0, 16)
  uint8_t lens[16];     // code lengths of symbols 0..15 (15 = escape)
  uint64_t lens_packed; // lens[s] at bits 4s..4s+3
};

// The 16 phase tables, built on first use (thread-safe).
const PhaseTable* phase_tables();

}  // namespace zc
