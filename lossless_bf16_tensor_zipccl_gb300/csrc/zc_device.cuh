// zc_device.cuh -- device helpers of the GB300 exponent-coding kernels:
// memory-ordering primitives for the look-back, TMA bulk copies, bounded
// waits, canonical-code tables and the per-lane table-driven decoder.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "zc_format.h"

namespace zc {

constexpr unsigned kFull = 0xFFFFFFFFu;
// Bounded waits: a wait that exceeds this gives up and records kStTimeout.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void set_status(WsHeader* h, uint32_t code) {
  atomicCAS(&h->status, 0u, code);
}

// Streaming 16-byte load (read once, keep out of L1).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// (TMA) proxy; pair with a CTA barrier before the bulk copy is issued.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA bulk store shared -> global (no multicast); several may be issued
// before one commit.  bulk_commit_and_wait_read waits until shared memory has
// been read; the global writes complete on their own before the grid ends.
__device__ __forceinline__ void bulk_store_issue(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(ssrc)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ---- mbarrier-tracked TMA bulk load global -> shared (single use, phase 0)
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void bulk_load_async(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(sdst)),
               "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Wait for phase `parity` of the barrier, giving up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------- code tables
// Canonical codeword (MSB-first value) of symbol `sym` for packed lengths:
// codes are handed out in (length, symbol) order, so the code of s counts, at
// length L(s), every code value taken by a symbol that precedes it:
//   code(s) = sum_{t before s} 2^(L(s) - L(t)).
__device__ __forceinline__ uint32_t canonical_code(uint64_t lens, int sym) {
  const uint32_t L = (uint32_t)((lens >> (4 * sym)) & 15);
  uint32_t code = 0;
#pragma unroll
  for (int t = 0; t < kNsym; ++t) {
    const uint32_t lt = (uint32_t)((lens >> (4 * t)) & 15);
    if (lt < L || (lt == L && t < sym)) code += 1u << (L - lt);
  }
  return code;
}

__device__ __forceinline__ uint32_t bit_reverse(uint32_t v, int len) {
  return len ? (__brev(v) >> (32 - len)) : 0u;
}

// True when all 16 lengths are in [1, kLmax] and sum 2^-len == 1.
__host__ __device__ __forceinline__ bool lens_complete(uint64_t lens) {
  uint32_t kraft = 0;
  for (int s = 0; s < kNsym; ++s) {
    const uint32_t l = (uint32_t)((lens >> (4 * s)) & 15);
    if (l < 1 || l > (uint32_t)kLmax) return false;
    kraft += 1u << (kLmax - l);
  }
  return kraft == (1u << kLmax);
}

// Multi-symbol decode table: entry i describes the symbols that the 10-bit
// window i (next bits of the stream, LSB first) starts with, packed in 32 bits:
//   bits 0-19  up to 5 symbols, 4 bits each (first symbol lowest)
//   bits 20-23 bits consumed (<= 10)
//   bits 24-26 symbols decoded (1..5)
//   bit  27    the last symbol is the escape
// Decoding stops after an escape; its 8 raw bits are not in the window count.
constexpr uint32_t kLutEsc = 1u << 27;

__device__ __forceinline__ uint32_t lut_entry(uint32_t idx, uint64_t lens, const uint32_t (&rev)[kNsym]) {
  uint32_t pos = 0, ns = 0, nib = 0, esc = 0;
#pragma unroll 1
  while (ns < 5 && !esc) {
    int found = -1;
    uint32_t flen = 0;
#pragma unroll
    for (int s = 0; s < kNsym; ++s) {
      const uint32_t l = (uint32_t)((lens >> (4 * s)) & 15);
      if (l + pos <= (uint32_t)kLmax && ((idx >> pos) & ((1u << l) - 1u)) == rev[s]) {
        found = s;
        flen = l;
      }
    }
    if (found < 0) break;
    nib |= (uint32_t)found << (4 * ns);
    ++ns;
    pos += flen;
    esc = found == kEsc;
  }
  return nib | (pos << 20) | (ns << 24) | (esc << 27);
}

// Fill a 1024-entry table cooperatively (all threads of the block).
__device__ __forceinline__ void build_lut(uint64_t lens, uint32_t* lut) {
  uint32_t rev[kNsym];
#pragma unroll
  for (int s = 0; s < kNsym; ++s) rev[s] = bit_reverse(canonical_code(lens, s), (int)((lens >> (4 * s)) & 15));
  for (uint32_t i = threadIdx.x; i < kLutEntries; i += blockDim.x) lut[i] = lut_entry(i, lens, rev);
}

// ---------------------------------------------------------------- merge
// 4 exponent bytes + 4 sign/mantissa bytes -> 4 BF16 words (2 x u32).
__device__ __forceinline__ uint2 merge4(uint32_t e4, uint32_t sm4) {
  const uint32_t e01 = __byte_perm(e4, 0, 0x4140), e23 = __byte_perm(e4, 0, 0x4342);
  const uint32_t s01 = __byte_perm(sm4, 0, 0x4140), s23 = __byte_perm(sm4, 0, 0x4342);
  uint2 r;
  r.x = ((s01 & 0x00800080u) << 8) | (e01 << 7) | (s01 & 0x007F007Fu);
  r.y = ((s23 & 0x00800080u) << 8) | (e23 << 7) | (s23 & 0x007F007Fu);
  return r;
}

// ---------------------------------------------------------------- lane decoder
// Decodes one segment of a coded tile: symbols are taken 1-5 at a time from a
// 1024-entry table (in shared memory) indexed by the next 10 stream bits; the window is a funnel
// shift over two words with a third prefetched.  Pending symbols wait as
// nibbles in `acc`; escape exponents wait as bytes in escv (positions 0-7)
// and esch (8-11).
struct LaneDecoder {
  const uint32_t* seg;
  const uint32_t* lut;  // shared-memory copy of the chunk's table
  uint64_t acc, escv;
  uint32_t nw, wi, cur, nxt, nx2, boff, cnt, esch, base4;

  // seg points into shared memory (staged exponent region) or global memory
  __device__ __forceinline__ uint32_t word(uint32_t i) const { return i < nw ? seg[i] : 0u; }

  __device__ __forceinline__ void init(const uint32_t* s, uint32_t n_words, const uint32_t* table, uint32_t base) {
    seg = s;
    nw = n_words;
    lut = table;
    cur = word(0);
    nxt = word(1);
    nx2 = word(2);
    wi = 3;
    boff = 0;
    acc = 0;
    cnt = 0;
    escv = 0;
    esch = 0;
    base4 = base * 0x01010101u;
  }

  // Decode until at least `target` symbols are pending (target <= 8).
  __device__ __forceinline__ void fill(uint32_t target) {
    while (cnt < target) {
      const uint32_t win = __funnelshift_r(cur, nxt, boff);
      const uint32_t en = lut[win & (kLutEntries - 1)];
      uint32_t nb = (en >> 20) & 15u;
      acc |= (uint64_t)(en & 0xFFFFFu) << (4 * cnt);
      cnt += (en >> 24) & 7u;
      if (en & kLutEsc) {
        const uint32_t e = (win >> nb) & 0xFFu;
        const uint32_t p = cnt - 1;
        nb += 8;
        if (p < 8) {
          escv = (escv & ~(0xFFull << (8 * p))) | ((uint64_t)e << (8 * p));
        } else {
          const uint32_t q = 8 * (p - 8);
          esch = (esch & ~(0xFFu << q)) | (e << q);
        }
      }
      boff += nb;
      if (boff >= 32) {
        boff -= 32;
        cur = nxt;
        nxt = nx2;
        nx2 = word(wi);
        ++wi;
      }
    }
  }

  // Pop 8 pending symbols as exponent bytes (e0..e3, e4..e7).
  __device__ __forceinline__ void take8(uint32_t& lo, uint32_t& hi) {
    const uint32_t nib = (uint32_t)acc;
    const uint32_t ev = nib & 0x0F0F0F0Fu, od = (nib >> 4) & 0x0F0F0F0Fu;
    const uint32_t x0 = __byte_perm(ev, od, 0x5140), x1 = __byte_perm(ev, od, 0x7362);
    const uint32_t m0 = __vcmpeq4(x0, 0x0F0F0F0Fu), m1 = __vcmpeq4(x1, 0x0F0F0F0Fu);
    lo = ((x0 + base4) & ~m0) | ((uint32_t)escv & m0);
    hi = ((x1 + base4) & ~m1) | ((uint32_t)(escv >> 32) & m1);
    acc >>= 32;
    cnt = cnt > 8 ? cnt - 8 : 0;  // fewer than 8 only on a segment's last row
    escv = esch;
    esch = 0;
  }
};

}  // namespace zc
