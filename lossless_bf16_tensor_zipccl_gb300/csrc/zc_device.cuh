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

// Relaxed 64-bit loads and stores at GPU scope.  The look-back state words
// and the chunk-start slot each carry their flag and value in one word, and
// readers use only that word, so no fence is needed around them.
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Acquire load and release add at GPU scope: the per-chunk completion count
// of the compress-and-send call.  A writer's earlier stores (its own, and
// those ordered before by a fence) are visible to a reader whose acquire
// load sees the count.
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add_u64(uint64_t* p, uint64_t v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void set_status(WsHeader* h, uint32_t code) {
  atomicCAS(&h->status, 0u, code);
}

// Tagged status of a decompress or reduce call (tag: 56 bits, nonzero): the
// call's first error wins; a word with another tag is stale and is replaced.
// Only the call's own threads write the word, so after one stale word is
// replaced every further attempt finds this call's tag and stops.
__device__ __forceinline__ void set_status_tagged(WsHeader* h, uint64_t tag, uint32_t code) {
  unsigned long long* w = reinterpret_cast<unsigned long long*>(&h->status);
  const unsigned long long want = (tag << 8) | code;
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(w);
  for (int i = 0; i < 64; ++i) {
    if ((old >> 8) == tag && (old & 0xFFu) != 0) return;
    const unsigned long long prev = atomicCAS(w, old, want);
    if (prev == old) return;
    old = prev;
  }
}

__device__ __forceinline__ bool status_tagged_set(const WsHeader* h, uint64_t tag) {
  const unsigned long long v = *reinterpret_cast<const volatile unsigned long long*>(&h->status);
  return (v >> 8) == tag && (v & 0xFFu) != 0;
}

// Programmatic dependent launch.  A prep kernel lets the kernel after it in
// the stream be scheduled at once (pdl_trigger); that kernel, launched with
// programmatic stream serialisation, waits for the prep kernel to finish
// and its writes to be visible (pdl_wait) before it reads anything.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// Wait until at most one (all_but_last) or none (all) of this thread's bulk
// groups is still writing global memory, then order those writes (made by
// the async proxy) before this thread's later generic-proxy operations.
__device__ __forceinline__ void bulk_wait_written_all_but_last() {
  asm volatile("cp.async.bulk.wait_group 1;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_written_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ---- mbarrier-tracked TMA bulk loads global -> shared
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Arrive once on the barrier (release: this thread's earlier shared-memory
// writes are visible to a thread whose wait sees the phase complete).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive once on the barrier and announce `bytes` of TMA traffic for its phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// TMA bulk copy global -> shared (no multicast), completing `bytes` on the barrier.
__device__ __forceinline__ void bulk_copy_g2s(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(sdst)),
               "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// Wait for phase `parity` of the barrier, giving up after kWaitLimitNs.
// Each try_wait suspends the thread (up to the hint, 0.5 ms) until the phase
// completes, so a waiting warp does not take issue slots from working ones.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_addr(bar);
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(a), "r"(parity), "r"(500000u)
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
//   bits 0-19  up to 5 symbols, 4 bits each (last symbol lowest, so that a
//              queue shifted left by the entry's width takes them in order)
//   bits 20-23 bits consumed (<= 10)
//   bits 24-28 4 x symbols decoded (4..20): the entry's width in the queue
//   bit  29    the last symbol is the escape
// Decoding stops after an escape; its 8 raw bits are not in the window count.
constexpr uint32_t kLutEsc = 1u << 29;

// Fill entries [first, first + count) of a 1024-entry table; every thread
// of the block calls it, with complete lengths (lens_complete holds).  First
// the symbol that each 10-bit window starts with is found by matching the
// reversed codewords (the code is complete, so exactly one matches); then
// each entry chains up to five lookups in that first-symbol table.  A symbol
// found in the window shifted right by pos bits is real only if it ends
// within the 10 bits, since the shift brings in zeros from above.  Building
// a table is still split across several blocks.
__device__ __forceinline__ void build_lut(uint64_t lens, uint32_t* lut, uint32_t first, uint32_t count) {
  __shared__ uint32_t s_rev[kNsym];
  __shared__ uint8_t s_sym[kLutEntries];
  if (threadIdx.x < (uint32_t)kNsym) {
    const int s = (int)threadIdx.x;
    s_rev[s] = bit_reverse(canonical_code(lens, s), (int)((lens >> (4 * s)) & 15));
  }
  __syncthreads();
  uint32_t rev[kNsym], len[kNsym];
#pragma unroll
  for (int s = 0; s < kNsym; ++s) {
    rev[s] = s_rev[s];
    len[s] = (uint32_t)((lens >> (4 * s)) & 15);
  }
  for (uint32_t w = threadIdx.x; w < kLutEntries; w += blockDim.x) {
    uint32_t sym = 0;
#pragma unroll
    for (int s = 0; s < kNsym; ++s)
      if ((w & ((1u << len[s]) - 1u)) == rev[s]) sym = (uint32_t)s;
    s_sym[w] = (uint8_t)sym;
  }
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < count; i += blockDim.x) {
    const uint32_t idx = first + i;
    uint32_t pos = 0, ns = 0, nib = 0, esc = 0;
    while (ns < 5 && !esc) {
      const uint32_t s = s_sym[idx >> pos];
      const uint32_t l = (uint32_t)((lens >> (4 * s)) & 15);
      if (pos + l > (uint32_t)kLmax) break;
      nib = (nib << 4) | s;
      ++ns;
      pos += l;
      esc = s == (uint32_t)kEsc;
    }
    lut[idx] = nib | (pos << 20) | ((4 * ns) << 24) | (esc << 29);
  }
}

// ---------------------------------------------------------------- merge
// 4 exponent bytes + 4 sign/mantissa bytes (sign in bit 7) -> 4 BF16 words
// (2 x u32).  All four high bytes (sign, exponent bits 7..1) and all four low
// bytes (exponent bit 0, mantissa) are formed at once, then interleaved.
__device__ __forceinline__ uint2 merge4(uint32_t e4, uint32_t sm4) {
  const uint32_t hi = (sm4 & 0x80808080u) | ((e4 >> 1) & 0x7F7F7F7Fu);
  const uint32_t lo = ((e4 << 7) & 0x80808080u) | (sm4 & 0x7F7F7F7Fu);
  uint2 r;
  r.x = __byte_perm(lo, hi, 0x5140);
  r.y = __byte_perm(lo, hi, 0x7362);
  return r;
}

// ---------------------------------------------------------------- lane decoder
// Readable bytes a staged payload copy needs after its span.  A lane runs at
// most 8 symbols of at most kLmax + 8 bits past its segment's end (its queue
// holds 16, the last row takes 8), so its last table step starts before
// bit E + 144 (E: the span's last payload bit) and reads words up to two past
// the one holding that bit: less than E / 8 + 31 bytes.
constexpr uint32_t kStagePad = 48;

// Decodes one segment of a coded tile.  Symbols come 1-5 at a time from a
// 1024-entry table indexed by the next 10 stream bits; the window is a
// funnel shift over two words (boff < 32) and a third word is loaded one step
// ahead.  kStaged: the words are a copy in shared memory followed by at least
// kStagePad readable bytes, so loads need no bound; otherwise they are the
// region in place in global memory, never read past `end`.  Up to 16
// decoded symbols wait as nibbles in a 64-bit queue (qhi:qlo, newest lowest;
// a table entry enters it with one left shift by its own width), so a lane
// can decode ahead of the row its warp emits; escape exponents wait as bytes
// in esc0..esc3 with a mask, indexed by queue position from the oldest
// pending symbol.
template <bool kStaged>
struct LaneDecoder {
  const uint32_t* wp;    // next word to load
  const uint32_t* wend;  // one past the last readable word (in place)
  const uint32_t* lut;
  uint32_t qlo, qhi;     // pending symbols; the oldest at nibble cnt4 / 4 - 1
  uint32_t w0, w1, w2, boff, cnt4;  // cnt4: 4 x pending symbols
  uint32_t escm, esc0, esc1, esc2, esc3;
  uint32_t base4;

  __device__ __forceinline__ uint32_t next_word() {
    uint32_t w;
    if constexpr (kStaged) w = *wp;
    else w = wp < wend ? *wp : 0u;
    ++wp;
    return w;
  }

  // payload: first word of the tile's coded bitstream; start: this segment's
  // first bit in it; end: one past the last readable word.
  __device__ __forceinline__ void init(const uint32_t* payload, uint32_t start, const uint32_t* end,
                                       const uint32_t* table, uint32_t base) {
    wp = payload + (start >> 5);
    wend = end;
    lut = table;
    w0 = next_word();
    w1 = next_word();
    w2 = next_word();
    boff = start & 31;
    qlo = qhi = 0;
    cnt4 = 0;
    escm = esc0 = esc1 = esc2 = esc3 = 0;
    base4 = base * 0x01010101u;
  }

  __device__ __forceinline__ void place_escape(uint32_t p, uint32_t e) {
    const uint32_t sh = 8 * (p & 3), m = ~(0xFFu << sh), v = e << sh;
    switch (p >> 2) {
      case 0: esc0 = (esc0 & m) | v; break;
      case 1: esc1 = (esc1 & m) | v; break;
      case 2: esc2 = (esc2 & m) | v; break;
      default: esc3 = (esc3 & m) | v; break;
    }
    escm |= 1u << p;
  }

  // One table step.  Requires cnt4 <= 44 (room for 5 more symbols).
  __device__ __forceinline__ void step() {
    const uint32_t win = __funnelshift_r(w0, w1, boff);
    const uint32_t en = lut[win & (kLutEntries - 1)];
    const uint32_t sh = (en >> 24) & 31u;
    qhi = __funnelshift_l(qlo, qhi, sh);
    qlo = (qlo << sh) | (en & 0xFFFFFu);
    cnt4 += sh;
    uint32_t nb = (en >> 20) & 15u;
    if (__builtin_expect((en & kLutEsc) != 0, 0)) {
      place_escape((cnt4 >> 2) - 1, (win >> nb) & 0xFFu);
      nb += 8;
    }
    boff += nb;
    if (boff >= 32) {  // the window passed a word: slide by one
      boff -= 32;
      w0 = w1;
      w1 = w2;
      w2 = next_word();
    }
  }

  // Warp-wide: decode until every lane holds at least `need` symbols (need
  // <= 8); lanes that are there already keep decoding while they have room,
  // so the next row starts ahead.  All 32 lanes must call this together,
  // after init or take8, which leave at most 8 symbols pending: the first
  // step always has room.
  __device__ __forceinline__ void fill_warp(uint32_t need) {
    step();
    if (cnt4 <= 44) step();
    while (__any_sync(kFull, cnt4 < 4 * need)) {
      if (cnt4 <= 44) step();
    }
  }

  // Pop 8 pending symbols as exponent bytes (e0..e3, e4..e7); with fewer
  // pending (a segment's last row) the missing ones are garbage.  kRow8: at
  // least 8 are pending (every row of a full tile).  Escape bytes are kept
  // per queue position; bytes whose escm bit is clear are never read, so the
  // escape registers move only while an escape is pending.
  template <bool kRow8>
  __device__ __forceinline__ void take8(uint32_t& e_lo, uint32_t& e_hi) {
    // the oldest 8 symbols, oldest in the top nibble
    uint32_t e32;
    if constexpr (kRow8) e32 = __funnelshift_rc(qlo, qhi, cnt4 - 32);
    else e32 = cnt4 >= 32 ? __funnelshift_rc(qlo, qhi, cnt4 - 32) : __funnelshift_lc(0u, qlo, 32 - cnt4);
    const uint32_t ev = e32 & 0x0F0F0F0Fu, od = (e32 >> 4) & 0x0F0F0F0Fu;
    e_lo = __byte_perm(ev, od, 0x2637) + base4;
    e_hi = __byte_perm(ev, od, 0x0415) + base4;
    if (__builtin_expect(escm != 0, 0)) {
      const uint32_t m = escm;
      if (m & 0xFFu) {  // substitute the raw exponents of escapes
        const uint32_t m0 = (m & 1 ? 0xFFu : 0u) | (m & 2 ? 0xFF00u : 0u) | (m & 4 ? 0xFF0000u : 0u) |
                            (m & 8 ? 0xFF000000u : 0u);
        const uint32_t m1 = (m & 16 ? 0xFFu : 0u) | (m & 32 ? 0xFF00u : 0u) | (m & 64 ? 0xFF0000u : 0u) |
                            (m & 128 ? 0xFF000000u : 0u);
        e_lo = (e_lo & ~m0) | (esc0 & m0);
        e_hi = (e_hi & ~m1) | (esc1 & m1);
      }
      esc0 = esc2;
      esc1 = esc3;
      escm = m >> 8;
    }
    if constexpr (kRow8) cnt4 -= 32;
    else cnt4 = cnt4 > 32 ? cnt4 - 32 : 0;  // fewer than 8 only on a segment's last row
  }
};

}  // namespace zc
