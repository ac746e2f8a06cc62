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
  const SelectChunkArg ca = a.c[blockIdx.x];
  const uint32_t ci = a.chunk0 + blockIdx.x;
  __shared__ long long s_sum[8], s_cnt[8];
  __shared__ int s_q;
  if (ci == 0 && threadIdx.x == 0) {
    a.hdr->status = 0;
    a.hdr->counter = 0;
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
    ec.pad[0] = ec.pad[1] = 0;
    a.chunks[ci] = ec;
  }
  // Code tables of the chunk.  tab[e]: reversed codeword | length << 24 (an
  // escape entry carries the 8 raw exponent bits after the codeword).
  // pair[x0 | x1 << 4]: both reversed codewords, first lowest (bits 0-19) |
  // an escape flag (bit 20) | total length including 8 raw bits per escape
  // (bits 26-31); a pair with an escape is packed symbol by symbol.
  {
    uint32_t* tab = a.tables + (size_t)ci * kEncTableWords;
    const uint32_t e = threadIdx.x;
    const int xs = (int)e - base;
    const int sym = (xs >= 0 && xs < kWindow) ? xs : kEsc;
    const int L = (int)((lens >> (4 * sym)) & 15);
    const uint32_t rev = bit_reverse(canonical_code(lens, sym), L);
    tab[e] = sym == kEsc ? ((rev | (e << L)) | ((uint32_t)(L + 8) << 24)) : (rev | ((uint32_t)L << 24));
    const uint32_t s0 = e & 15, s1 = e >> 4;
    const uint32_t l0 = (uint32_t)((lens >> (4 * s0)) & 15), l1 = (uint32_t)((lens >> (4 * s1)) & 15);
    const uint32_t c0 = bit_reverse(canonical_code(lens, (int)s0), (int)l0);
    const uint32_t c1 = bit_reverse(canonical_code(lens, (int)s1), (int)l1);
    const uint32_t raw = (s0 == (uint32_t)kEsc ? 8u : 0u) + (s1 == (uint32_t)kEsc ? 8u : 0u);
    tab[256 + e] = (c0 | (c1 << l0)) | (raw ? kPairEsc : 0u) | ((l0 + l1 + raw) << 26);
  }
  const uint32_t items = ca.n_tiles ? ca.n_tiles : 1u;
  for (uint32_t i = threadIdx.x; i < items; i += blockDim.x) {
    a.item_chunk[ca.first_item + i] = ci;
    a.item_state[ca.first_item + i] = 0;
  }
}

// ---------------------------------------------------------------- encode
// One CTA per tile.  Row warps 0..7 own the left half of every row
// (segments 0..31), row warps 8..15 the right half (segments 32..63), eight
// rows each; lane l of a row warp in half h works on segment 32 h + l.
// Warp 16 is the control warp: it lays out the segments, publishes the
// tile's size, runs the look-back and writes the chunk header while the row
// warps assemble the exponent region.
//
// Single pass over the input: a row warp reads its rows once, writes the
// sign/mantissa bytes into the tile image and packs each lane's codewords
// into a private word buffer in shared memory as it goes (bit 0 of the part
// at bit 0 of word 0).  Once every part's length is known, each lane copies
// its part to its bit position in the segment stream with funnel shifts:
// words that only this part touches are stored, the two end words are OR-ed.
// A part longer than its private buffer (a lane with many escapes) sends
// the tile down a slower path that re-reads its input and packs in place; a
// raw tile re-reads its input to store the exponent bytes.
//
// Shared memory: tile image (header | sign/mantissa plane | exponent region)
// | private part buffers | code tables | per-(row warp, lane) bit counts.
constexpr uint32_t kImgBytes = kTileHdr + kTile + kTile;
constexpr int kRowWarpsPerHalf = 8;
constexpr int kRowWarps = 2 * kRowWarpsPerHalf;
constexpr int kCtlWarp = kRowWarps;
constexpr int kEncThreads = 32 * (kRowWarps + 1);
constexpr int kRowsPerWarp = kRows / kRowWarpsPerHalf;   // 8
constexpr uint32_t kPrivWords = 16;                       // 512 bits per lane part (8 bits per value)
constexpr uint32_t kPrivBytes = kRowWarps * 32 * kPrivWords * 4;
constexpr uint32_t kEncSmem = kImgBytes + kPrivBytes + kEncTableWords * 4 + kRowWarps * 32 * 4;

// Decoupled look-back over the flat tile list (warp-wide).  Each tile
// publishes its byte count (aggregate), then its inclusive prefix.  Returns
// the exclusive prefix; sets err on a timed-out wait or an upstream error.
__device__ uint64_t lookback(uint64_t* state, uint32_t item, uint32_t lane, bool& err) {
  uint64_t excl = 0;
  int64_t pred = (int64_t)item - 1;
  uint64_t t0 = 0;
  bool waiting = false;
  while (true) {
    const int64_t idx = pred - (int64_t)lane;
    const uint64_t s = idx >= 0 ? ld_acquire_u64(state + idx) : kFlagInc;
    const uint32_t flag = (uint32_t)(s >> kFlagShift);
    const uint32_t not_ready = __ballot_sync(kFull, flag == 0);
    const uint32_t stop = __ballot_sync(kFull, flag >= 2);
    const uint32_t lim = stop ? (uint32_t)(__ffs(stop) - 1) : 31u;
    const uint32_t upto = lim == 31 ? kFull : ((2u << lim) - 1u);
    if (not_ready & upto) {
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
      __nanosleep(64);
      continue;
    }
    if (__ballot_sync(kFull, flag == 3) & upto) {
      err = true;
      return 0;
    }
    uint64_t v = lane <= lim ? (s & kValMask) : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    excl += v;
    if (stop) return excl;
    pred -= 32;
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

// Bit packer into a lane's private buffer (word j at p[32 j]).  Counts every
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

__global__ void __launch_bounds__(kEncThreads, 2) zc_encode_kernel(EncodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* img = smem;
  uint32_t* priv = reinterpret_cast<uint32_t*>(smem + kImgBytes);                    // [warp][word][lane]
  uint32_t* tab = reinterpret_cast<uint32_t*>(smem + kImgBytes + kPrivBytes);       // per exponent
  uint32_t* pair = tab + 256;                                                        // per symbol pair
  uint32_t* part = tab + kEncTableWords;  // [row warp][lane] bits, then bit offsets
  __shared__ uint32_t s_item, s_mode, s_err, s_size, s_over;
  __shared__ uint32_t s_segstart[kSegs];
  __shared__ unsigned long long s_goff;

  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    s_item = atomicAdd(&a.hdr->counter, 1u);  // tiles start in claim order
    s_err = 0;
    s_over = 0;
  }
  __syncthreads();
  const uint32_t item = s_item;
  const uint32_t c = a.item_chunk[item];
  const EncChunk ci = a.chunks[c];
  const uint32_t k = item - ci.first_item;
  const uint32_t nt = ci.n_tiles ? (uint32_t)min((uint64_t)kTile, ci.n - (uint64_t)k * kTile) : 0u;
  const uint64_t elem0 = ci.elem_start + (uint64_t)k * kTile;
  const uint16_t* x = a.in + elem0;
  const bool vec = (elem0 & 7) == 0;
  const uint32_t base = ci.base;
  const uint32_t base4 = base * 0x01010101u;
  const uint32_t sm_pad = (uint32_t)pad16(nt);
  const uint32_t exp_off = kTileHdr + sm_pad;
  uint32_t* region = reinterpret_cast<uint32_t*>(img + exp_off + kSegTab);  // coded payload words

  // Tables from the select kernel; zero the padding of the sign/mantissa
  // plane and the exponent area (the end words of each part are OR-ed in).
  for (uint32_t i = tid; i < kEncTableWords; i += kEncThreads) tab[i] = __ldg(a.tables + (size_t)c * kEncTableWords + i);
  if (tid < 16 && nt + tid < sm_pad) img[kTileHdr + nt + tid] = 0;
  for (uint32_t o = tid * 16; o < sm_pad; o += kEncThreads * 16)
    *reinterpret_cast<uint4*>(img + exp_off + o) = make_uint4(0, 0, 0, 0);
  __syncthreads();

  const uint32_t half = warp < kRowWarps ? warp / kRowWarpsPerHalf : 0u;
  const uint32_t rb = warp < kRowWarps ? (warp % kRowWarpsPerHalf) * kRowsPerWarp : kRows;
  const uint32_t col = half * kHalf + lane * kLaneElems;
  const bool full = nt == kTile && vec;

  // Phase A (row warps): read each row group once; sign/mantissa bytes to
  // the image, codewords to the private buffer.
  uint32_t my_bits = 0;
  if (warp < kRowWarps) {
    PrivSink sink;
    sink.begin(priv + warp * (32 * kPrivWords) + lane);
    if (full) {
      uint4 v[kRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) v[r] = ld_stream_v4(x + (rb + r) * kRow + col);
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        uint32_t sm0, sm1, ex0, ex1;
        split4(v[r].x, v[r].y, sm0, ex0);
        split4(v[r].z, v[r].w, sm1, ex1);
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
    my_bits = sink.bits();
    part[warp * 32 + lane] = my_bits;
    if (__any_sync(kFull, my_bits > 32 * kPrivWords) && lane == 0) s_over = 1;
  }
  __syncthreads();

  // Phase B (control warp): bit offset of each row warp's part inside its
  // segment, bit-granular segment starts, raw/coded choice, publish the
  // aggregate.  Lane l handles segments l and 32 + l.
  uint64_t agg = 0;
  if (warp == kCtlWarp) {
    uint32_t seg[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t off = 0;
#pragma unroll
      for (int w = 0; w < kRowWarpsPerHalf; ++w) {
        const uint32_t i = (h * kRowWarpsPerHalf + w) * 32 + lane;
        const uint32_t v = part[i];
        part[i] = off;
        off += v;
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
    s_segstart[lane] = start0 - seg[0];
    s_segstart[32 + lane] = total0 + start1 - seg[1];
    const uint32_t words = (total0 + total1 + 31) >> 5;
    const bool coded = kSegTab + 4ull * words < nt;
    const uint32_t exp_bytes = coded ? kSegTab + 4 * words : nt;
    if (coded) {
      reinterpret_cast<uint16_t*>(img + exp_off)[lane] = (uint16_t)seg[0];
      reinterpret_cast<uint16_t*>(img + exp_off)[32 + lane] = (uint16_t)seg[1];
    }
    const uint32_t size = nt ? (uint32_t)(kTileHdr + sm_pad + pad16(exp_bytes)) : 0u;
    agg = size + (k == 0 ? chunk_hdr_bytes(ci.n_tiles) : 0);
    if (lane == 0) {
      s_mode = coded ? 0u : 1u;
      s_size = size;
      *reinterpret_cast<uint4*>(img) = make_uint4(coded ? 0u : 1u, nt, exp_bytes, 0u);
      st_release_u64(a.item_state + item, (item == 0 ? kFlagInc : kFlagAgg) | agg);
    }
  }
  __syncthreads();

  if (warp == kCtlWarp) {
    // Phase C (control warp): look-back for this tile's byte offset, chunk
    // header / tile table / chunk offsets.
    bool err = false;
    uint64_t excl = item == 0 ? 0 : lookback(a.item_state, item, lane, err);
    if (item != 0 && lane == 0) st_release_u64(a.item_state + item, err ? kFlagErr : (kFlagInc | (excl + agg)));
    uint64_t cs = 0;
    if (!err) {
      if (k == 0) {
        cs = excl;
        if (lane == 0) {
          st_release_u64(&a.chunks[c].start_slot, kSlotValid | cs);
          a.offsets[c] = cs;
        }
      } else {
        // lane 0 waits for the chunk's first tile to publish the chunk start
        uint64_t v = 0;
        uint32_t to = 0;
        if (lane == 0) {
          const uint64_t t0 = globaltimer_ns();
          v = ld_acquire_u64(&a.chunks[c].start_slot);
          while (!(v & kSlotValid)) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
              to = 1;
              break;
            }
            __nanosleep(64);
            v = ld_acquire_u64(&a.chunks[c].start_slot);
          }
        }
        v = __shfl_sync(kFull, v, 0);
        err = __shfl_sync(kFull, to, 0) != 0;
        cs = v & ~kSlotValid;
      }
    }
    const uint64_t hdr = chunk_hdr_bytes(ci.n_tiles);
    const uint64_t goff = excl + (k == 0 ? hdr : 0);
    if (!err && (goff + s_size > a.cap || cs + hdr > a.cap)) {
      err = true;
      if (lane == 0) set_status(a.hdr, kStCapacity);
    } else if (err && lane == 0) {
      set_status(a.hdr, kStTimeout);
    }
    if (!err) {
      uint8_t* cp = a.out + cs;
      if (k == 0) {
        if (lane < 8) {
          uint32_t v;
          switch (lane) {
            case 0: v = kMagic; break;
            case 1: v = kVersion | (kTileLog2 << 16) | (kSegLog2 << 24); break;
            case 2: v = (uint32_t)ci.n; break;
            case 3: v = (uint32_t)(ci.n >> 32); break;
            case 4: v = ci.n_tiles; break;
            case 5: v = base | ((uint32_t)(uint16_t)(int16_t)ci.q << 16); break;
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
      if (item == a.n_items - 1 && lane == 0) a.offsets[a.n_chunks] = excl + agg;
    }
    if (lane == 0) {
      s_goff = goff;
      s_err = err ? 1u : 0u;
    }
  } else if (s_mode == 0 && !s_over) {
    // Phase D (row warps): move each part from its private buffer to its bit
    // position in the segment stream.
    if (my_bits) {
      const uint32_t S = s_segstart[half * 32 + lane] + part[warp * 32 + lane];
      const uint32_t sh = S & 31, nw = (my_bits + 31) >> 5, nout = (sh + my_bits + 31) >> 5;
      const uint32_t* src = priv + warp * (32 * kPrivWords) + lane;
      uint32_t* dst = region + (S >> 5);
      uint32_t prev = 0;
      for (uint32_t j = 0; j < nout; ++j) {
        const uint32_t cur = j < nw ? src[32 * j] : 0u;
        const uint32_t v = __funnelshift_l(prev, cur, sh);
        if (j == 0 || j + 1 == nout) atomicOr(dst + j, v);
        else dst[j] = v;
        prev = cur;
      }
    }
  } else if (s_mode == 0) {
    // Phase D, a part overflowed its buffer: re-read the rows and pack in place.
    BitSink sink;
    sink.begin(region, s_segstart[half * 32 + lane] + part[warp * 32 + lane]);
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
          sink.put(en & 0xFFFFFFu, en >> 24);
        }
      }
    }
    sink.finish();
  } else {
    // Phase D, raw tile: re-read the rows and store the exponent bytes.
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
  __syncthreads();

  // Phase E: one TMA bulk store of the finished tile image.  The CTA leaves
  // once shared memory has been read.
  if (tid == 0 && !s_err && s_size) {
    bulk_store_issue(a.out + s_goff, img, s_size);
    bulk_commit_and_wait_read();
  }
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_select(const SelectArgs& args, cudaStream_t s) {
  if (args.count == 0) return cudaSuccess;
  zc_select_kernel<<<args.count, 256, 0, s>>>(args);
  return cudaGetLastError();
}

static int g_enc_attr_done[64];

cudaError_t launch_encode(const EncodeArgs& args, uint32_t n_items, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !g_enc_attr_done[dev]) {
    e = cudaFuncSetAttribute(zc_encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kEncSmem);
    if (e != cudaSuccess) return e;
    g_enc_attr_done[dev] = 1;
  }
  zc_encode_kernel<<<n_items, kEncThreads, kEncSmem, s>>>(args);
  return cudaGetLastError();
}

}  // namespace zc
