// zc_encode.cu -- compressor kernels for sm_103a.
//
// "ZipCCL: Efficient Lossless Data Compression of Communication Collectives
// for Accelerating LLM Training":
//   - abstract, technique (1): exponent coding from the Gaussian law with no
//     online statistics -> zc_select_kernel takes the scale from a fixed
//     sample (one integer sum), never a histogram of the tensor;
//   - abstract, technique (2) and Fig. 5 / Fig. 6 captions: GPU compressor
//     with designed memory access, overlap of compression with memory
//     traffic, few launches, communication-aware layout -> one fused kernel
//     per tile computes lengths, packs bits in shared memory, finds its
//     output offset by decoupled look-back over the flat tile list of all
//     per-destination chunks, and writes the tile image with TMA bulk
//     stores;
//   - Fig. 7 caption (shared-memory data layout): the tile image is staged in
//     shared memory as header | sign/mantissa plane | exponent region.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "zc_device.cuh"
#include "zc_kernels.h"

namespace zc {

// ---------------------------------------------------------------- scale select
__device__ __forceinline__ int64_t floor_div_pos(int64_t a, int64_t b) {  // b > 0
  return a >= 0 ? a / b : -((-a + b - 1) / b);
}

// One block per chunk.  The code is built for sigma = 2^(q/16).  With a hint
// q is given; otherwise the mean biased exponent of a fixed sample (all
// elements when n <= 4096, else 64 blocks of 64 consecutive elements at
// floor(b n / 64)), skipping e = 0 and e = 255, gives
//   q = round-half-up(16 (mean - 127 + 1.4164)),
// 1.4164 being 1/2 + (gamma + ln 2)/(2 ln 2): the mean of floor(log2 |Z|)
// below log2(sigma) for a centred Gaussian.  The block also writes the
// chunk's code tables for the encoder.
__global__ void __launch_bounds__(256) zc_select_kernel(const __grid_constant__ SelectArgs a) {
  pdl_trigger();
  const SelectChunkArg ca = a.c[blockIdx.x];
  const uint32_t ci = a.chunk0 + blockIdx.x;
  __shared__ long long s_sum[8], s_cnt[8];
  __shared__ int s_q;
  if (ci == 0 && threadIdx.x == 0) {
    a.hdr->status = 0;
    a.hdr->status_hi = 0;
    a.hdr->epoch = 0;
  }
  if (ca.has_hint) {
    if (threadIdx.x == 0) s_q = ca.q_hint;
  } else {
    const uint16_t* x = a.in + ca.elem_start;
    long long S = 0, K = 0;
    // 16 samples per thread (256 threads), all loads issued before any is used
    uint32_t ev[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t s = threadIdx.x + 256u * i;
      uint64_t at;
      if (ca.n <= 4096) at = s;                                         // every element
      else at = ((uint64_t)(s >> 6) * ca.n) / 64 + (s & 63);            // block s/64, offset s%64
      ev[i] = at < ca.n ? x[at] : 0xFFFFu;                              // exponent 255: not counted
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t e = (ev[i] >> 7) & 0xFFu;
      if (e != 0 && e != 255) { S += e; ++K; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      S += __shfl_xor_sync(kFull, S, o);
      K += __shfl_xor_sync(kFull, K, o);
    }
    if ((threadIdx.x & 31) == 0) {
      s_sum[threadIdx.x >> 5] = S;
      s_cnt[threadIdx.x >> 5] = K;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      long long ts = 0, tk = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) { ts += s_sum[w]; tk += s_cnt[w]; }
      s_q = tk ? (int)floor_div_pos(40000ll * (ts - 127ll * tk) + 57906ll * tk, 2500ll * tk) : 0;
    }
  }
  __syncthreads();
  const int q = s_q;
  const int kq = (int)floor_div_pos(q, 16);
  const int r = q - 16 * kq;
  int base = kq + 127 + a.base_off[r];
  base = base < 0 ? 0 : (base > 240 ? 240 : base);
  const uint64_t lens = a.lens[r];
  if (threadIdx.x == 0) {
    EncChunk ec;
    ec.elem_start = ca.elem_start;
    ec.n = ca.n;
    ec.first_item = ca.first_item;
    ec.n_tiles = ca.n_tiles;
    ec.q = q;
    ec.base = (uint32_t)base;
    ec.lens = lens;
    ec.start_slot = 0;
    ec.done = 0;
    ec.end = 0;
    a.chunks[ci] = ec;
  }
  // Code tables of the chunk.  tab[e]: reversed codeword | length << 24 (an
  // escape entry carries the 8 raw exponent bits after the codeword).
  // pair[x0 | x1 << 4]: both reversed codewords, first lowest (bits 0-19) |
  // an escape flag (bit 20) | total length including 8 raw bits per escape
  // (bits 26-31); a pair with an escape is packed symbol by symbol.
  {
    // the 16 reversed codewords, once per block
    __shared__ uint32_t s_rev[kNsym];
    if (threadIdx.x < (uint32_t)kNsym) {
      const int sy = (int)threadIdx.x;
      s_rev[sy] = bit_reverse(canonical_code(lens, sy), (int)((lens >> (4 * sy)) & 15));
    }
    __syncthreads();
    uint32_t* tab = a.tables + (size_t)ci * kEncTableWords;
    const uint32_t e = threadIdx.x;
    const int xs = (int)e - base;
    const int sym = (xs >= 0 && xs < kWindow) ? xs : kEsc;
    const int L = (int)((lens >> (4 * sym)) & 15);
    const uint32_t rev = s_rev[sym];
    tab[e] = sym == kEsc ? ((rev | (e << L)) | ((uint32_t)(L + 8) << 24)) : (rev | ((uint32_t)L << 24));
    const uint32_t s0 = e & 15, s1 = e >> 4;
    const uint32_t l0 = (uint32_t)((lens >> (4 * s0)) & 15), l1 = (uint32_t)((lens >> (4 * s1)) & 15);
    const uint32_t c0 = s_rev[s0], c1 = s_rev[s1];
    const uint32_t raw = (s0 == (uint32_t)kEsc ? 8u : 0u) + (s1 == (uint32_t)kEsc ? 8u : 0u);
    tab[256 + e] = (c0 | (c1 << l0)) | (raw ? kPairEsc : 0u) | ((l0 + l1 + raw) << 26);
  }
  const uint32_t items = ca.n_tiles ? ca.n_tiles : 1u;
  for (uint32_t i = threadIdx.x; i < items; i += blockDim.x) {
    EncItem r;
    r.elem0 = ca.elem_start + (uint64_t)i * kTile;
    r.c = ci;
    r.k = i;
    r.nt = ca.n_tiles ? (uint32_t)min((uint64_t)kTile, ca.n - (uint64_t)i * kTile) : 0u;
    r.base = (uint32_t)base;
    r.pad[0] = r.pad[1] = 0;
    a.items[ca.first_item + i] = r;
    a.item_state[ca.first_item + i] = 0;
  }
}

// ---------------------------------------------------------------- encode
// Persistent CTAs, one per SM, all resident at once (cooperative launch);
// CTA b takes tiles b, b + G, b + 2G, ... (G CTAs), so every tile's
// predecessors are processed by running CTAs in the same order.
//
// Row warps 0..7 own the left half of every row (segments 0..31), row warps
// 8..15 the right half (segments 32..63), eight rows each; lane l of a row
// warp in half h works on segment 32 h + l.
//
// Single pass over the input: a row warp reads its rows once (the loads were
// issued one tile earlier), writes the sign/mantissa bytes into the tile
// image and packs each lane's codewords into its part slot, in the upper
// half of the image's exponent region (bit 0 of the part at bit 0 of word
// 0) -- phase A.  The layout warp (warp 16) then places the segments and
// publishes the tile's size -- phase B; each lane copies its part to its bit
// position in the lower half with funnel shifts -- phase D.  A row warp runs
// phase D of a tile after phase A of the next one: rather than wait at every
// tile boundary for the slowest row warp and the layout warp, it waits only
// when it gets a whole tile ahead of them.  Parts fit their
// slots at up to 4 bits per value, so a coded stream of fitting parts is at
// most 16 KB and never reaches the slots; a part longer than its slot (a lane
// with many escapes) sends the tile down a slower path that re-reads its
// input and packs in place; a raw tile re-reads its input to store the
// exponent bytes.
//
// The store warp (warp 17) runs the look-back for the tile's byte offset,
// writes the chunk header, tile table and chunk offsets, and stores the tile
// image with one TMA bulk copy -- phases C and E -- up to two tiles behind
// the row warps: the image is triple-buffered.  Named barriers hand tiles
// between the roles (i = tile number within the CTA, b = i mod 3):
//   kBarParts0 + b  row warps arrive after phase A; the layout warp waits;
//   kBarSeg0 + b    the layout warp arrives after phase B; row warps wait
//                   before phase D (after phase A of tile i + 1);
//   kBarB0 + b      the layout warp arrives after phase B; the store warp
//                   waits;
//   kBarImg0 + b    row warps arrive after phase D; the store warp waits;
//   kBarFree0 + b   the store warp arrives once image b has been read by its
//                   store; row warps wait before packing tile i + 3 into it.
// Each barrier has one id per buffer, since a role may reach it again
// before the other role has waited; barrier 0 is the block barrier.
//
// Shared memory: 3 tile images (header | sign/mantissa plane | exponent
// region with the part slots above kSlotOff) | 4 code tables (the layout
// warp stages tile i + 2's while tile i - 1's may still be in use) |
// per buffer: per-(row warp, lane) part bits, then offsets | per buffer:
// per-(row warp, lane) first word of each part.
constexpr int kRowWarpsPerHalf = 8;
constexpr int kRowWarps = 2 * kRowWarpsPerHalf;
constexpr int kLayoutWarp = kRowWarps;
constexpr int kStoreWarp = kRowWarps + 1;
constexpr int kSendWarp = kRowWarps + 2;  // compress-and-send only
constexpr int kRowThreads = 32 * kRowWarps;
constexpr int kEncThreads = 32 * (kRowWarps + 2);
constexpr int kEncThreadsSend = kEncThreads + 32;
constexpr uint32_t kBarThreads = kRowThreads + 32;      // row warps + one role warp
constexpr int kRowsPerWarp = kRows / kRowWarpsPerHalf;   // 8
constexpr uint32_t kPrivWords = 8;                        // 256 bits per lane part (4 bits per value)
constexpr uint32_t kPrivBytes = kRowWarps * 32 * kPrivWords * 4;
// Part slots, from the exponent region's start: above the segment table, a
// stream of fitting parts (kPrivBytes) and its padding to 16 bytes.
constexpr uint32_t kSlotOff = kSegTab + kPrivBytes + 16;
constexpr uint32_t kImgBytes = kTileHdr + kTile + kSlotOff + kPrivBytes;  // >= header + planes of a raw tile
constexpr uint32_t kImgBufs = 3;
constexpr uint32_t kTabBufs = 4;
constexpr uint32_t kEncSmem = kImgBufs * kImgBytes + kTabBufs * kEncTableWords * 4 + 2 * kImgBufs * kRowThreads * 4;
constexpr uint32_t kBarParts0 = 1, kBarSeg0 = 4, kBarB0 = 7, kBarImg0 = 10, kBarFree0 = 13;
static_assert(kBarFree0 + kImgBufs <= 16, "named barriers");
static_assert(kImgBytes >= kTileHdr + 2 * kTile, "raw tile image");

__device__ __forceinline__ void bar_arrive(uint32_t id, uint32_t n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void bar_wait(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Decoupled look-back over the flat tile list (warp-wide).  Each tile
// publishes its byte count (aggregate), then its inclusive prefix.  One pass
// reads the 64 nearest unfolded predecessors (2 per lane), folds them up to
// and including the nearest inclusive prefix, and stops there.  Returns the
// exclusive prefix; sets err on a timed-out wait or an upstream error.  The
// nearest inclusive prefix is usually a few tiles back, and every pass costs
// the store warp issue slots its scheduler's row warps would use: passes of
// 64 compress faster than passes of 256 (measured: -4 to -5%), and a 256-ns
// pause between passes that find a predecessor not ready is better than 64
// where many tiles are raw (measured: -1.5%).
constexpr int kLookbackDepth = 2;  // states per lane per pass

__device__ uint64_t lookback(const uint64_t* state, uint32_t item, uint32_t lane, bool& err) {
  uint64_t excl = 0;
  int64_t pred = (int64_t)item - 1;  // nearest predecessor not folded yet
  uint64_t t0 = 0;
  bool waiting = false;
  while (true) {
    uint64_t s[kLookbackDepth];
#pragma unroll
    for (int j = 0; j < kLookbackDepth; ++j) {
      const int64_t idx = pred - (int64_t)lane - 32 * j;  // position 32 j + lane back from pred
      s[j] = idx >= 0 ? ld_relaxed_u64(state + idx) : kFlagInc;
    }
    // nearest stop (inclusive prefix or error): group sj, lane sl
    uint32_t sj = kLookbackDepth, sl = 31;
#pragma unroll
    for (int j = kLookbackDepth - 1; j >= 0; --j) {
      const uint32_t b = __ballot_sync(kFull, (s[j] >> kFlagShift) >= 2);
      if (b) {
        sj = j;
        sl = __ffs(b) - 1;
      }
    }
    const uint32_t upto_sl = sl == 31 ? kFull : ((2u << sl) - 1u);
    bool not_ready = false, upstream_err = false;
#pragma unroll
    for (int j = 0; j < kLookbackDepth; ++j) {
      const uint32_t m = (uint32_t)j < sj ? kFull : ((uint32_t)j == sj ? upto_sl : 0u);
      not_ready |= (__ballot_sync(kFull, (s[j] >> kFlagShift) == 0) & m) != 0;
      upstream_err |= (__ballot_sync(kFull, (s[j] >> kFlagShift) == 3) & m) != 0;
    }
    if (not_ready) {
      // lane 0's clock decides for the whole warp, so all lanes leave together
      const uint64_t now = globaltimer_ns();
      if (!waiting) {
        waiting = true;
        t0 = now;
      }
      if (__shfl_sync(kFull, (now - t0 > kWaitLimitNs) ? 1u : 0u, 0)) {
        err = true;
        return 0;
      }
      __nanosleep(256);
      continue;
    }
    if (upstream_err) {
      err = true;
      return 0;
    }
    uint64_t v = 0;
#pragma unroll
    for (int j = 0; j < kLookbackDepth; ++j)
      if ((uint32_t)j < sj || ((uint32_t)j == sj && lane <= sl)) v += s[j] & kValMask;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    excl += v;
    if (sj < (uint32_t)kLookbackDepth) return excl;
    pred -= 32 * kLookbackDepth;
  }
}

// Bit sink for one lane's part of a segment in shared memory (32-bit,
// branch-free).  The part's first word may be shared with the previous part
// and its last word with the next one: both are OR-ed in at the end; the
// words in between belong to this part alone and are stored as they fill.
// code < 2^24, len <= 24, nacc < 32.
struct BitSink {
  uint32_t* sw;
  uint32_t acc, widx, nacc, first_idx, first_word, nfl;
  __device__ __forceinline__ void begin(uint32_t* words, uint32_t start_bit) {
    sw = words;
    acc = 0;
    widx = first_idx = start_bit >> 5;
    nacc = start_bit & 31;
    first_word = 0;
    nfl = 0;
  }
  __device__ __forceinline__ void put(uint32_t code, uint32_t len) {
    const uint32_t spill = __funnelshift_l(code, 0u, nacc);  // bits of code << nacc above bit 31
    acc |= code << nacc;
    nacc += len;
    const bool flush = nacc >= 32;
    if (flush && nfl) sw[widx] = acc;
    first_word = (flush && !nfl) ? acc : first_word;
    nfl |= flush ? 1u : 0u;
    widx += flush ? 1u : 0u;
    acc = flush ? spill : acc;
    nacc -= flush ? 32u : 0u;
  }
  __device__ __forceinline__ void finish() {
    if (nfl) atomicOr(sw + first_idx, first_word);
    if (nacc) atomicOr(sw + widx, acc);
  }
};

// Bit packer into a lane's part slot (word j at p[32 j]).  Counts every
// bit; words past kPrivWords are dropped and the caller sees the overflow in
// bits().  code < 2^len, len <= 32.
struct PrivSink {
  uint32_t* p;
  uint32_t acc, nacc, widx;
  __device__ __forceinline__ void begin(uint32_t* lane_words) {
    p = lane_words;
    acc = nacc = widx = 0;
  }
  __device__ __forceinline__ void put(uint32_t code, uint32_t len) {
    const uint32_t spill = __funnelshift_l(code, 0u, nacc);  // bits of code << nacc above bit 31
    acc |= code << nacc;
    nacc += len;
    if (nacc >= 32) {
      if (widx < kPrivWords) p[32 * widx] = acc;
      ++widx;
      nacc -= 32;
      acc = spill;
    }
  }
  __device__ __forceinline__ void finish() {
    if (nacc && widx < kPrivWords) p[32 * widx] = acc;
  }
  __device__ __forceinline__ uint32_t bits() const { return 32 * widx + nacc; }
};

// x << s for s < 32, 0 for s >= 32.
__device__ __forceinline__ uint32_t shl_clamped(uint32_t x, uint32_t s) { return __funnelshift_l(0u, x, s); }

// Sign/mantissa bytes (s << 7 | m) and exponent bytes of 4 BF16 values held
// in two words (value 2i in the low half of word i).
__device__ __forceinline__ void split4(uint32_t w0, uint32_t w1, uint32_t& sm, uint32_t& ex) {
  const uint32_t lo = __byte_perm(w0, w1, 0x6420);  // low byte of each value
  const uint32_t hi = __byte_perm(w0, w1, 0x7531);  // high byte of each value
  sm = (hi & 0x80808080u) | (lo & 0x7F7F7F7Fu);
  ex = ((hi << 1) & 0xFEFEFEFEu) | ((lo >> 7) & 0x01010101u);
}

// Pack the 8 exponents of one lane row (bytes of ex0, ex1) into the sink.
// Fast path: every x = e - base in 0..14, codes combined through the
// symbol-pair table into one put when the row fits 32 bits.
__device__ __forceinline__ void pack_row8(PrivSink& sink, uint32_t ex0, uint32_t ex1, uint32_t base4,
                                          const uint32_t* pair, const uint32_t* tab) {
  const uint32_t y0 = ex0 - base4, y1 = ex1 - base4;  // bytes x (borrows only when some x < 0)
  const bool in_window = ((y0 | y1) & 0xF0F0F0F0u) == 0;
  const uint32_t z0 = y0 | (y0 >> 4), z1 = y1 | (y1 >> 4);
  const uint32_t p0 = pair[z0 & 0xFFu], p1 = pair[(z0 >> 16) & 0xFFu];
  const uint32_t p2 = pair[z1 & 0xFFu], p3 = pair[(z1 >> 16) & 0xFFu];
  const bool fast = in_window && !((p0 | p1 | p2 | p3) & kPairEsc);
  const uint32_t l0 = p0 >> 26, l1 = p1 >> 26, l2 = p2 >> 26, l3 = p3 >> 26;
  const uint32_t s2 = l0 + l1, s3 = s2 + l2, tot = s3 + l3;
  if (fast && tot <= 32) {
    const uint32_t rc = (p0 & 0xFFFFFu) | shl_clamped(p1 & 0xFFFFFu, l0) | shl_clamped(p2 & 0xFFFFFu, s2) |
                        shl_clamped(p3 & 0xFFFFFu, s3);
    sink.put(rc, tot);
  } else if (fast) {
    sink.put(p0 & 0xFFFFFu, l0);
    sink.put(p1 & 0xFFFFFu, l1);
    sink.put(p2 & 0xFFFFFu, l2);
    sink.put(p3 & 0xFFFFFu, l3);
  } else {
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const uint32_t en = tab[((t < 4 ? ex0 : ex1) >> (8 * (t & 3))) & 0xFFu];
      sink.put(en & 0xFFFFFFu, en >> 24);
    }
  }
}

// The 8 (or fewer, cnt) values of one lane row as 4 words, from a 16-B
// aligned full group or element by element.
__device__ __forceinline__ void load_group(const uint16_t* x, uint32_t cnt, bool vec, uint32_t (&w)[4]) {
  if (vec && cnt == 8) {
    const uint4 v = ld_stream_v4(x);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  } else {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t lo = (2 * p < (int)cnt) ? x[2 * p] : 0u;
      const uint32_t hi = (2 * p + 1 < (int)cnt) ? x[2 * p + 1] : 0u;
      w[p] = lo | (hi << 16);
    }
  }
}

// Shared state of the encode CTA.  Plain pointers only: an array of
// pointers indexed by the buffer number would put the struct in local memory.
struct EncShared {
  uint8_t* img0;       // image b at img0 + b * kImgBytes
  uint32_t* tabs;      // kTabBufs x kEncTableWords
  uint32_t* part;      // per buffer: [row warp][lane] bits, then bit offsets in the segment
  uint32_t* first;     // per buffer: [row warp][lane] word 0 of each part
  uint32_t* segstart;  // per buffer: [kSegs]
  uint32_t* mode;      // per buffer: 0 coded, 1 coded with an overflowed part, 2 raw
  uint32_t* over;      // per buffer: a part overflowed its slot
  uint32_t* size;      // per buffer: tile bytes
  __device__ __forceinline__ uint8_t* img(uint32_t b) const { return img0 + b * kImgBytes; }
  // word 0 of this thread's part slot (words at a stride of 32)
  __device__ __forceinline__ uint32_t* slot(uint32_t b, uint32_t exp_off, uint32_t warp, uint32_t lane) const {
    return reinterpret_cast<uint32_t*>(img(b) + exp_off + kSlotOff) + warp * (32 * kPrivWords) + lane;
  }
};

__device__ __forceinline__ EncItem load_item(const EncodeArgs& a, uint32_t t) {
  EncItem r;
  if (t < a.n_items) {
    r = a.items[t];
  } else {
    r.elem0 = 0;
    r.c = r.k = r.nt = r.base = 0;
    r.pad[0] = r.pad[1] = 0;
  }
  return r;
}

__device__ __forceinline__ bool full_tile(const EncItem& r) { return r.nt == kTile && (r.elem0 & 7) == 0; }

// Row warps, phase A of one tile in image b with code tables tb.  v holds
// this tile's rows rb..rb+7 (full tiles); each row's registers are refilled
// with the next tile's row as soon as they are consumed, so the loads run a
// whole tile ahead.  Returns this lane's part length in bits.
__device__ __forceinline__ uint32_t phase_a(const EncodeArgs& a, const EncShared& S, uint32_t b, uint32_t tb,
                                            const EncItem& rec, uint4 (&v)[kRowsPerWarp], const EncItem& fut,
                                            bool fut_ok) {
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t half = warp / kRowWarpsPerHalf;
  const uint32_t rb = (warp % kRowWarpsPerHalf) * kRowsPerWarp;
  const uint32_t col = half * kHalf + lane * kLaneElems;
  uint8_t* img = S.img(b);
  const uint32_t* tab = S.tabs + tb * kEncTableWords;  // per exponent
  const uint32_t* pair = tab + 256;                   // per symbol pair
  const uint32_t nt = rec.nt;
  const uint16_t* x = a.in + rec.elem0;
  const bool vec = (rec.elem0 & 7) == 0;
  const bool full = nt == kTile && vec;
  const uint32_t base4 = rec.base * 0x01010101u;
  const uint32_t sm_pad = (uint32_t)pad16(nt);
  const uint32_t exp_off = kTileHdr + sm_pad;

  // Other than full tiles: zero the padding of the sign/mantissa plane and
  // the exponent area below the slots (the end words of each part are OR-ed
  // in; a raw tile's phase D zeroes its own padding).
  if (!full) {
    if (tid < 16 && nt + tid < sm_pad) img[kTileHdr + nt + tid] = 0;
    const uint32_t zend = min(sm_pad, kSlotOff);
    for (uint32_t o = tid * 16; o < zend; o += kRowThreads * 16)
      *reinterpret_cast<uint4*>(img + exp_off + o) = make_uint4(0, 0, 0, 0);
  }

  // sign/mantissa bytes to the image, codewords to the part slot
  PrivSink sink;
  uint32_t* my_slot = S.slot(b, exp_off, warp, lane);
  sink.begin(my_slot);
  const bool fut_full = fut_ok && full_tile(fut);
  const uint16_t* xf = a.in + fut.elem0 + rb * kRow + col;
  if (full) {
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      uint32_t sm0, sm1, ex0, ex1;
      split4(v[r].x, v[r].y, sm0, ex0);
      split4(v[r].z, v[r].w, sm1, ex1);
      if (fut_full) v[r] = ld_stream_v4(xf + r * kRow);
      *reinterpret_cast<uint2*>(img + kTileHdr + (rb + r) * kRow + col) = make_uint2(sm0, sm1);
      pack_row8(sink, ex0, ex1, base4, pair, tab);
    }
  } else {
    for (uint32_t row = rb; row < rb + kRowsPerWarp; ++row) {
      const uint32_t i0 = row * kRow + col;
      const uint32_t cnt = nt > i0 ? min(8u, nt - i0) : 0u;
      if (cnt == 0) break;
      uint32_t w[4];
      load_group(x + i0, cnt, vec, w);
      uint32_t sm0, sm1, ex0, ex1;
      split4(w[0], w[1], sm0, ex0);
      split4(w[2], w[3], sm1, ex1);
      if (cnt == 8) {
        *reinterpret_cast<uint2*>(img + kTileHdr + i0) = make_uint2(sm0, sm1);
        pack_row8(sink, ex0, ex1, base4, pair, tab);
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (t < (int)cnt) {
            img[kTileHdr + i0 + t] = (uint8_t)((t < 4 ? sm0 : sm1) >> (8 * (t & 3)));
            const uint32_t en = tab[((t < 4 ? ex0 : ex1) >> (8 * (t & 3))) & 0xFFu];
            sink.put(en & 0xFFFFFFu, en >> 24);
          }
        }
      }
    }
  }
  sink.finish();
  const uint32_t my_bits = sink.bits();
  S.part[b * kRowThreads + warp * 32 + lane] = my_bits;
  // word 0 of the part, for the part before it in the stream (phase D)
  S.first[b * kRowThreads + warp * 32 + lane] = my_slot[0];
  if (__any_sync(kFull, my_bits > 32 * kPrivWords) && lane == 0) S.over[b] = 1;
  if (!full && fut_full) {
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) v[r] = ld_stream_v4(xf + r * kRow);
  }
  return my_bits;
}

// Row warps, phase D of one tile in image b (code tables tb), after the
// layout warp's phase B: move each part from its slot to its bit position in
// the segment stream, or take the overflow or raw path.
__device__ __forceinline__ void phase_d(const EncodeArgs& a, const EncShared& S, uint32_t b, uint32_t tb,
                                        const EncItem& rec, uint32_t my_bits) {
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t half = warp / kRowWarpsPerHalf;
  const uint32_t rb = (warp % kRowWarpsPerHalf) * kRowsPerWarp;
  const uint32_t col = half * kHalf + lane * kLaneElems;
  uint8_t* img = S.img(b);
  const uint32_t* tab = S.tabs + tb * kEncTableWords;
  const uint32_t nt = rec.nt;
  const uint16_t* x = a.in + rec.elem0;
  const bool vec = (rec.elem0 & 7) == 0;
  const bool full = nt == kTile && vec;
  const uint32_t sm_pad = (uint32_t)pad16(nt);
  const uint32_t exp_off = kTileHdr + sm_pad;
  uint32_t* region = reinterpret_cast<uint32_t*>(img + exp_off + kSegTab);  // coded payload words
  const uint32_t* part = S.part + b * kRowThreads;
  const uint32_t* segstart = S.segstart + b * kSegs;
  const uint32_t mode = S.mode[b];
  if (mode == 0 && full) {
    // Full tile: every part holds >= 64 bits (64 codewords of >= 1 bit), so
    // a word of the stream holds bits of at most two parts.  Each word is
    // written once, by the part that holds its first bit; where the part
    // ends inside its last word, the rest of that word is the start of the
    // next part (its word 0).
    const uint32_t w8 = warp % kRowWarpsPerHalf;
    uint32_t nwarp = warp + 1, nlane = lane;  // the next part in stream order
    bool has_next = true;
    if (w8 + 1 == kRowWarpsPerHalf) {
      nwarp = half * kRowWarpsPerHalf;
      nlane = lane + 1;
      if (lane == 31) {
        nwarp = kRowWarpsPerHalf;
        nlane = 0;
        has_next = half == 0;
      }
    }
    const uint32_t next_w0 = has_next ? S.first[b * kRowThreads + nwarp * 32 + nlane] : 0u;
    const uint32_t St = segstart[half * 32 + lane] + part[warp * 32 + lane];
    const uint32_t sh = St & 31, nw = (my_bits + 31) >> 5, e = (St + my_bits) & 31;
    const uint32_t x0 = (St + 31) >> 5, x1 = (St + my_bits - 1) >> 5;
    const uint32_t* src = S.slot(b, exp_off, warp, lane);
    uint32_t pw[kPrivWords + 1];
#pragma unroll
    for (uint32_t j = 0; j < kPrivWords; ++j) pw[j] = j < nw ? src[32 * j] : 0u;
    pw[kPrivWords] = 0;
#pragma unroll
    for (uint32_t j = 0; j < kPrivWords; ++j) {
      const uint32_t xw = x0 + j;
      if (xw <= x1) {
        uint32_t w = sh ? __funnelshift_r(pw[j], pw[j + 1], 32 - sh) : pw[j];
        if (xw == x1 && e) w |= next_w0 << e;
        region[xw] = w;
      }
    }
    if (!has_next) {
      // the stream's last word: zero the padding words up to 16 bytes
      const uint32_t pend = ((kSegTab / 4 + x1 + 1 + 3) & ~3u) - kSegTab / 4;
      for (uint32_t xw = x1 + 1; xw < pend; ++xw) region[xw] = 0;
    }
  } else if (mode == 0) {
    // the part's end words are OR-ed into the zeroed area, the rest stored
    if (my_bits) {
      const uint32_t St = segstart[half * 32 + lane] + part[warp * 32 + lane];
      const uint32_t sh = St & 31, nw = (my_bits + 31) >> 5, nout = (sh + my_bits + 31) >> 5;
      const uint32_t* src = S.slot(b, exp_off, warp, lane);
      uint32_t* dst = region + (St >> 5);
      uint32_t pw[kPrivWords];
#pragma unroll
      for (uint32_t j = 0; j < kPrivWords; ++j) pw[j] = j < nw ? src[32 * j] : 0u;
      uint32_t prev = 0;
#pragma unroll
      for (uint32_t j = 0; j <= kPrivWords; ++j) {
        const uint32_t cur = j < kPrivWords ? pw[j] : 0u;
        const uint32_t w = __funnelshift_l(prev, cur, sh);
        if (j < nout) {
          if (j == 0 || j + 1 == nout) atomicOr(dst + j, w);
          else dst[j] = w;
        }
        prev = cur;
      }
    }
  } else if (mode == 1) {
    // A part overflowed its slot: re-read the rows and pack in place (the
    // layout warp has zeroed the payload area; boundary words are OR-ed).
    BitSink bs;
    bs.begin(region, segstart[half * 32 + lane] + part[warp * 32 + lane]);
#pragma unroll 1
    for (uint32_t row = rb; row < rb + kRowsPerWarp; ++row) {
      const uint32_t i0 = row * kRow + col;
      const uint32_t cnt = nt > i0 ? min(8u, nt - i0) : 0u;
      if (cnt == 0) break;
      uint32_t w[4];
      load_group(x + i0, cnt, vec, w);
      uint32_t sm0, sm1, ex0, ex1;
      split4(w[0], w[1], sm0, ex0);
      split4(w[2], w[3], sm1, ex1);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (t < (int)cnt) {
          const uint32_t en = tab[((t < 4 ? ex0 : ex1) >> (8 * (t & 3))) & 0xFFu];
          bs.put(en & 0xFFFFFFu, en >> 24);
        }
      }
    }
    bs.finish();
  } else {
    // Raw tile: re-read the rows and store the exponent bytes, then zero the
    // padding up to 16 bytes.
    if (tid < 16 && nt + tid < sm_pad) img[exp_off + nt + tid] = 0;
#pragma unroll 1
    for (uint32_t row = rb; row < rb + kRowsPerWarp; ++row) {
      const uint32_t i0 = row * kRow + col;
      const uint32_t cnt = nt > i0 ? min(8u, nt - i0) : 0u;
      if (cnt == 0) break;
      uint32_t w[4];
      load_group(x + i0, cnt, vec, w);
      uint32_t sm0, sm1, ex0, ex1;
      split4(w[0], w[1], sm0, ex0);
      split4(w[2], w[3], sm1, ex1);
      if (cnt == 8) {
        *reinterpret_cast<uint2*>(img + exp_off + i0) = make_uint2(ex0, ex1);
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t)
          if (t < (int)cnt) img[exp_off + i0 + t] = (uint8_t)((t < 4 ? ex0 : ex1) >> (8 * (t & 3)));
      }
    }
  }
  fence_proxy_async_smem();
  bar_arrive(kBarImg0 + b, kBarThreads);
}

// Layout warp, phase B of tile i (image b).  Also stages the code tables of
// tile i + 2 (`next2`) into table buffer (i + 2) mod kTabBufs: the row warps
// are past phase D of tile i - 2 once they have all finished phase A of
// tile i, and tile i - 1's tables may still be in use by its phase D.
__device__ __forceinline__ void layout_tile(const EncodeArgs& a, const EncShared& S, uint32_t b, uint32_t i,
                                            uint32_t item, uint32_t next2) {
  const uint32_t lane = threadIdx.x & 31;
  const EncItem rec = a.items[item];
  uint8_t* img = S.img(b);
  const uint32_t nt = rec.nt;
  const uint32_t sm_pad = (uint32_t)pad16(nt);
  const uint32_t exp_off = kTileHdr + sm_pad;
  const uint32_t hdr = (uint32_t)chunk_hdr_bytes(a.chunks[rec.c].n_tiles);
  // tile i + 2's code tables, staged in registers until the row warps are
  // past tile i's phase A
  uint4 nt4[kEncTableWords / 128];
  const bool has_next2 = next2 < a.n_items;
  if (has_next2) {
    const uint32_t cn = __ldg(&a.items[next2].c);
    const uint4* src = reinterpret_cast<const uint4*>(a.tables + (size_t)cn * kEncTableWords);
#pragma unroll
    for (uint32_t j = 0; j < kEncTableWords / 128; ++j) nt4[j] = __ldg(src + lane + 32 * j);
  }

  bar_wait(kBarParts0 + b, kBarThreads);
  // Bit offset of each row warp's part inside its segment, bit-granular
  // segment starts, raw/coded choice, publish the aggregate.  Lane l
  // handles segments l and 32 + l.
  uint32_t* part = S.part + b * kRowThreads;
  uint32_t seg[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pv[kRowWarpsPerHalf];
#pragma unroll
    for (int w = 0; w < kRowWarpsPerHalf; ++w) pv[w] = part[(h * kRowWarpsPerHalf + w) * 32 + lane];
    uint32_t off = 0;
#pragma unroll
    for (int w = 0; w < kRowWarpsPerHalf; ++w) {
      part[(h * kRowWarpsPerHalf + w) * 32 + lane] = off;
      off += pv[w];
    }
    seg[h] = off;
  }
  uint32_t start0 = seg[0], start1 = seg[1];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y0 = __shfl_up_sync(kFull, start0, o), y1 = __shfl_up_sync(kFull, start1, o);
    if (lane >= (uint32_t)o) {
      start0 += y0;
      start1 += y1;
    }
  }
  const uint32_t total0 = __shfl_sync(kFull, start0, 31), total1 = __shfl_sync(kFull, start1, 31);
  S.segstart[b * kSegs + lane] = start0 - seg[0];
  S.segstart[b * kSegs + 32 + lane] = total0 + start1 - seg[1];
  const uint32_t words = (total0 + total1 + 31) >> 5;
  const bool coded = kSegTab + 4ull * words < nt;
  const uint32_t exp_bytes = coded ? kSegTab + 4 * words : nt;
  const uint32_t over = S.over[b];
  if (coded) {
    reinterpret_cast<uint16_t*>(img + exp_off)[lane] = (uint16_t)seg[0];
    reinterpret_cast<uint16_t*>(img + exp_off)[32 + lane] = (uint16_t)seg[1];
    if (over) {
      // the overflow path packs in place over the whole payload area
      for (uint32_t o = kSegTab + lane * 16; o < sm_pad; o += 32 * 16)
        *reinterpret_cast<uint4*>(img + exp_off + o) = make_uint4(0, 0, 0, 0);
    }
  }
  const uint32_t size = nt ? (uint32_t)(kTileHdr + sm_pad + pad16(exp_bytes)) : 0u;
  const uint64_t agg = size + (rec.k == 0 ? hdr : 0u);
  __syncwarp();
  if (lane == 0) {
    S.mode[b] = coded ? (over ? 1u : 0u) : 2u;
    S.over[b] = 0;
    S.size[b] = size;
    *reinterpret_cast<uint4*>(img) = make_uint4(coded ? 0u : 1u, nt, exp_bytes, 0u);
  }
  if (has_next2) {
    uint4* dst = reinterpret_cast<uint4*>(S.tabs + ((i + 2) % kTabBufs) * kEncTableWords);
#pragma unroll
    for (uint32_t j = 0; j < kEncTableWords / 128; ++j) dst[lane + 32 * j] = nt4[j];
  }
  // Header and segment table are read by the TMA store.  The fence comes
  // before the aggregate's global store so that it does not wait for it.
  fence_proxy_async_smem();
  __syncwarp();
  bar_arrive(kBarSeg0 + b, kBarThreads);
  if (lane == 0) st_relaxed_u64(a.item_state + item, (item == 0 ? kFlagInc : kFlagAgg) | agg);
  bar_arrive(kBarB0 + b, 64);
}

// What the compress-and-send path publishes about a stored tile once its
// bytes are in global memory: its chunk, and the chunk's end offset when it
// is the chunk's last tile.
struct StoredTile {
  uint32_t c;
  uint32_t last;
  uint64_t end;
};

// Compress-and-send: the tile's stored bytes (and the headers and offsets its
// store warp wrote) become visible to the sender warps of every CTA.  Called
// by all lanes of the store warp after bulk_wait_written_*.
__device__ __forceinline__ void publish_stored(const EncodeArgs& a, const StoredTile& t) {
  __syncwarp();  // the other lanes' header and table stores come before the release
  if ((threadIdx.x & 31) == 0) {
    if (t.last) st_relaxed_u64(&a.chunks[t.c].end, t.end);
    red_release_add_u64(&a.chunks[t.c].done, 1);
  }
}

// Store warp, one tile: phases C and E.  `reuse`: the row warps will pack a
// later tile into this tile's image, so announce when its store has read it.
// `stored` receives what the compress-and-send path publishes later.
__device__ __forceinline__ void store_tile(const EncodeArgs& a, const EncShared& S, uint32_t buf, uint32_t item,
                                           const EncItem& rec, const EncChunk& ci, bool reuse, StoredTile& stored) {
  const uint32_t lane = threadIdx.x & 31;
  const uint32_t c = rec.c, k = rec.k, nt = rec.nt;
  const uint64_t hdr = chunk_hdr_bytes(ci.n_tiles);
  // Phase C: look-back for this tile's byte offset, chunk header / tile
  // table / chunk offsets.  The look-back and the wait for the chunk's start
  // need only earlier tiles, so they run before this tile's own size is
  // known, while its rows are still being packed and laid out.
  bool err = false;
  const uint64_t excl = item == 0 ? 0 : lookback(a.item_state, item, lane, err);
  uint64_t cs = 0;
  if (!err) {
    if (k == 0) {
      cs = excl;
      if (lane == 0) {
        st_relaxed_u64(&a.chunks[c].start_slot, kSlotValid | cs);
        a.offsets[c] = cs;
      }
    } else {
      // lane 0 waits for the chunk's first tile to publish the chunk start
      uint64_t v = 0;
      uint32_t to = 0;
      if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        v = ld_relaxed_u64(&a.chunks[c].start_slot);
        while (!(v & kSlotValid)) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            to = 1;
            break;
          }
          __nanosleep(64);
          v = ld_relaxed_u64(&a.chunks[c].start_slot);
        }
      }
      v = __shfl_sync(kFull, v, 0);
      err = __shfl_sync(kFull, to, 0) != 0;
      cs = v & ~kSlotValid;
    }
  }
  bar_wait(kBarB0 + buf, 64);
  const uint32_t size = S.size[buf];
  const uint64_t agg = size + (k == 0 ? hdr : 0);
  if (item != 0 && lane == 0) st_relaxed_u64(a.item_state + item, err ? kFlagErr : (kFlagInc | (excl + agg)));
  const uint64_t goff = excl + (k == 0 ? hdr : 0);
  const uint64_t lim = a.send && a.send_cap < a.cap ? a.send_cap : a.cap;  // both copies must fit
  if (!err && (goff + size > lim || cs + hdr > lim)) {
    err = true;
    if (lane == 0) set_status(a.hdr, kStCapacity);
  } else if (err && lane == 0) {
    set_status(a.hdr, kStTimeout);
  }
  // the chunk header and tile table go to the output and, with a send
  // buffer, to the same offsets there
  for (uint32_t copy = 0; !err && copy < (a.send ? 2u : 1u); ++copy) {
    uint8_t* cp = (copy ? a.send : a.out) + cs;
    if (k == 0) {
      if (lane < 8) {
        uint32_t v;
        switch (lane) {
          case 0: v = kMagic; break;
          case 1: v = kVersion | (kTileLog2 << 16) | (kSegLog2 << 24); break;
          case 2: v = (uint32_t)ci.n; break;
          case 3: v = (uint32_t)(ci.n >> 32); break;
          case 4: v = ci.n_tiles; break;
          case 5: v = ci.base | ((uint32_t)(uint16_t)(int16_t)ci.q << 16); break;
          case 6: v = (uint32_t)ci.lens; break;
          default: v = (uint32_t)(ci.lens >> 32); break;
        }
        reinterpret_cast<uint32_t*>(cp)[lane] = v;
      }
      // zero the tail of the tile table up to 16 bytes
      const uint32_t tail0 = 4 * ci.n_tiles, tail1 = (uint32_t)pad16(4ull * ci.n_tiles);
      if (tail0 + 4 * lane < tail1) reinterpret_cast<uint32_t*>(cp + kChunkHdr + tail0)[lane] = 0;
    }
    if (nt && lane == 0) reinterpret_cast<uint32_t*>(cp + kChunkHdr)[k] = (uint32_t)(goff - cs);
  }
  if (!err && item == a.n_items - 1 && lane == 0) a.offsets[a.n_chunks] = excl + agg;

  stored.c = c;
  stored.last = k + 1 >= ci.n_tiles ? 1u : 0u;  // an empty chunk's header-only item is its last
  stored.end = err ? 0 : goff + size;

  bar_wait(kBarImg0 + buf, kBarThreads);
  // Phase E: one TMA bulk store of the finished tile image, and with a send
  // buffer a second one of the same image there (the send costs HBM writes
  // only).  With a send buffer every tile commits one bulk group (empty when
  // nothing is stored), so that the group before last is always the
  // previous tile's.
  if (lane == 0) {
    if (!err && size) {
      bulk_store_issue(a.out + goff, S.img(buf), size);
      if (a.send) bulk_store_issue(a.send + goff, S.img(buf), size);
    }
    if (a.send || (!err && size)) bulk_commit_and_wait_read();
  }
  __syncwarp();
  if (reuse) bar_arrive(kBarFree0 + buf, kBarThreads);
}

// Sender warp of the compress-and-send path (CTA 0 only): the stand-in for
// the proxy that posts each chunk to its destination rank.  For chunks 0, 1,
// ... in order it waits until every tile of the chunk is stored in both
// buffers (the count published with release semantics by the store warps),
// then posts the chunk: here, it records %globaltimer in ready[c], so the
// caller sees how early each chunk could have left.  Waits are bounded; a
// wait that gives up records ZIPCCL_ERR_TIMEOUT and ends the posting, as does
// an error already recorded by the coding warps.
__device__ void send_chunks(const EncodeArgs& a) {
  const uint32_t lane = threadIdx.x & 31;
  for (uint32_t c = 0; c < a.n_chunks; ++c) {
    const uint32_t nt = a.chunks[c].n_tiles;
    const uint64_t want = nt ? nt : 1u;
    uint32_t ok = 1;
    if (lane == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_u64(&a.chunks[c].done) < want) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          ok = 0;
          break;
        }
        __nanosleep(128);
      }
      if (!ok) set_status(a.hdr, kStTimeout);
      else if (*reinterpret_cast<volatile uint32_t*>(&a.hdr->status) != 0) ok = 0;
      if (ok && a.ready) a.ready[c] = globaltimer_ns();
    }
    if (!__shfl_sync(kFull, ok, 0)) return;
  }
}

__global__ void __launch_bounds__(kEncThreadsSend, 1) zc_encode_kernel(EncodeArgs a) {
  pdl_wait();  // records and tables come from the select kernel
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t s_segstart[kImgBufs * kSegs], s_mode[kImgBufs], s_over[kImgBufs], s_size[kImgBufs];
  EncShared S;
  S.img0 = smem;
  S.tabs = reinterpret_cast<uint32_t*>(smem + kImgBufs * kImgBytes);
  S.part = S.tabs + kTabBufs * kEncTableWords;
  S.first = S.part + kImgBufs * kRowThreads;
  S.segstart = s_segstart;
  S.mode = s_mode;
  S.over = s_over;
  S.size = s_size;

  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t G = gridDim.x;
  const uint32_t t0 = blockIdx.x;
  const uint32_t count = (a.n_items - t0 + G - 1) / G;  // tiles of this CTA

  // Prologue: the code tables of the first two tiles.
  {
    const uint32_t c0 = a.items[t0].c;
    for (uint32_t i = tid; i < kEncTableWords; i += kEncThreads) S.tabs[i] = __ldg(a.tables + (size_t)c0 * kEncTableWords + i);
    if (t0 + G < a.n_items) {
      const uint32_t c1 = a.items[t0 + G].c;
      for (uint32_t i = tid; i < kEncTableWords; i += kEncThreads)
        S.tabs[kEncTableWords + i] = __ldg(a.tables + (size_t)c1 * kEncTableWords + i);
    }
    if (tid < kImgBufs) s_over[tid] = 0;
  }
  if (warp < kRowWarps) {
    const uint32_t half = warp / kRowWarpsPerHalf;
    const uint32_t rb = (warp % kRowWarpsPerHalf) * kRowsPerWarp;
    const uint32_t col = half * kHalf + lane * kLaneElems;
    uint4 v[kRowsPerWarp];
    EncItem rec = load_item(a, t0), nx = load_item(a, t0 + G), prv = rec;
    if (full_tile(rec)) {
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) v[r] = ld_stream_v4(a.in + rec.elem0 + (rb + r) * kRow + col);
    }
    __syncthreads();
    uint32_t b = 0, tb = 0, pb = 0, ptb = 0, prv_bits = 0;
    for (uint32_t i = 0; i < count; ++i) {
      const uint32_t t = t0 + i * G;
      const EncItem nx2 = load_item(a, t + 2 * G);  // records run two tiles ahead
      if (i >= kImgBufs) bar_wait(kBarFree0 + b, kBarThreads);
      const uint32_t bits = phase_a(a, S, b, tb, rec, v, nx, t + G < a.n_items);
      bar_arrive(kBarParts0 + b, kBarThreads);
      if (i > 0) {  // the previous tile, now that this one is packed
        bar_wait(kBarSeg0 + pb, kBarThreads);
        phase_d(a, S, pb, ptb, prv, prv_bits);
      }
      prv = rec;
      prv_bits = bits;
      pb = b;
      ptb = tb;
      rec = nx;
      nx = nx2;
      b = b + 1 == kImgBufs ? 0 : b + 1;
      tb = tb + 1 == kTabBufs ? 0 : tb + 1;
    }
    if (count > 0) {
      bar_wait(kBarSeg0 + pb, kBarThreads);
      phase_d(a, S, pb, ptb, prv, prv_bits);
    }
  } else if (warp == kLayoutWarp) {
    __syncthreads();
    uint32_t b = 0;
    for (uint32_t i = 0; i < count; ++i) {
      const uint32_t t = t0 + i * G;
      layout_tile(a, S, b, i, t, t + 2 * G);
      b = b + 1 == kImgBufs ? 0 : b + 1;
    }
  } else if (warp == kStoreWarp) {
    __syncthreads();
    // records are loaded one tile ahead
    EncItem rec = load_item(a, t0);
    EncChunk ch = a.chunks[rec.c];
    StoredTile prev = {0, 0, 0};
    for (uint32_t i = 0; i < count; ++i) {
      const uint32_t t = t0 + i * G;
      const EncItem rn = load_item(a, t + G);
      const EncChunk chn = a.chunks[rn.c];
      StoredTile cur;
      store_tile(a, S, i % kImgBufs, t, rec, ch, i + kImgBufs < count, cur);
      if (a.send && i > 0) {  // the previous tile's bulk group has written its bytes
        if (lane == 0) bulk_wait_written_all_but_last();
        publish_stored(a, prev);
      }
      prev = cur;
      rec = rn;
      ch = chn;
    }
    if (a.send && count > 0) {
      if (lane == 0) bulk_wait_written_all();
      publish_stored(a, prev);
    }
  } else if (warp == kSendWarp) {
    __syncthreads();
    if (a.send && blockIdx.x == 0) {
      if (lane == 0 && a.ready) a.ready[a.n_chunks] = globaltimer_ns();
      send_chunks(a);
    }
  }
}

// ---------------------------------------------------------------- bounded-wait self-test
// One warp waits, through the encoder's and the decoders' own code, on
// something no one completes: the look-back state of a predecessor tile
// (which = 0: tile 1 waits on tile 0, whose state stays 0), the phase of an
// mbarrier no one arrives on (which = 1), or the compress-and-send sender's
// wait for a chunk whose tiles are never stored (which = 2).  The wait gives up at its limit and
// the kernel records the timeout in the workspace status.
__global__ void zc_selftest_wait_kernel(WsHeader* hdr, uint64_t* state, int which) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t lane = threadIdx.x & 31;
  bool timed_out;
  if (which == 0) {
    bool err = false;
    (void)lookback(state, 1, lane, err);
    timed_out = err;
  } else if (which == 2) {
    // the compress-and-send sender's wait: one chunk of one tile whose
    // completion count stays 0 (the encoder never runs)
    EncodeArgs a = {};
    a.chunks = reinterpret_cast<EncChunk*>(state);
    a.offsets = state + sizeof(EncChunk) / 8;
    a.hdr = hdr;
    a.n_chunks = 1;
    a.send = reinterpret_cast<uint8_t*>(state);
    a.ready = nullptr;
    send_chunks(a);
    timed_out = false;  // send_chunks records the timeout itself
  } else {
    if (lane == 0) mbar_init(&bar, 1);
    __syncwarp();
    timed_out = __any_sync(kFull, !mbar_wait(&bar, 0));
  }
  if (lane == 0 && timed_out) set_status(hdr, kStTimeout);
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_selftest_wait(WsHeader* hdr, uint64_t* state, int which, cudaStream_t s) {
  zc_selftest_wait_kernel<<<1, 32, 0, s>>>(hdr, state, which);
  return cudaGetLastError();
}

cudaError_t launch_select(const SelectArgs& args, cudaStream_t s) {
  if (args.count == 0) return cudaSuccess;
  zc_select_kernel<<<args.count, 256, 0, s>>>(args);
  return cudaGetLastError();
}

// Co-resident encode CTAs per device (0: not set up).  Calls from several
// host threads may both do the set-up; each stores the same value.
static std::atomic<int> g_enc_ctas[64];

cudaError_t launch_encode(const EncodeArgs& args, uint32_t n_items, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int ctas = g_enc_ctas[dev].load(std::memory_order_acquire);
  if (!ctas) {
    e = cudaFuncSetAttribute(zc_encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kEncSmem);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, zc_encode_kernel, kEncThreadsSend, kEncSmem);
    if (e != cudaSuccess) return e;
    if (sms <= 0 || per_sm <= 0) return cudaErrorInvalidConfiguration;
    ctas = sms * per_sm;
    g_enc_ctas[dev].store(ctas, std::memory_order_release);
  }
  // Every CTA must be resident for the look-back order to make progress:
  // the cooperative launch guarantees it (or fails).
  const uint32_t grid = min(n_items, (uint32_t)ctas);
  cudaLaunchAttribute at[2];
  const int threads = args.send ? kEncThreadsSend : kEncThreads;  // the sender warp only with a send buffer
  const cudaLaunchConfig_t cfg = follow_config(dim3(grid), dim3(threads), kEncSmem, s, true, at);
  return cudaLaunchKernelEx(&cfg, zc_encode_kernel, args);
}

}  // namespace zc
