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
    if (ca.n <= 4096) {
      for (uint64_t i = threadIdx.x; i < ca.n; i += blockDim.x) {
        const uint32_t e = (x[i] >> 7) & 0xFFu;
        if (e != 0 && e != 255) { S += e; ++K; }
      }
    } else {
      for (uint32_t s = threadIdx.x; s < 4096; s += blockDim.x) {
        const uint64_t b = s >> 6, off = s & 63;
        const uint32_t e = (x[(b * ca.n) / 64 + off] >> 7) & 0xFFu;
        if (e != 0 && e != 255) { S += e; ++K; }
      }
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
// One CTA per tile.  Row warps 0..6 own the left half of every row
// (segments 0..31), row warps 7..13 the right half (segments 32..63), each a
// run of 9 or 10 rows; lane l of a row warp in half h works on segment
// 32 h + l.  Warp 14 is the control warp: it lays out the segments,
// publishes the tile's size, runs the look-back and writes the chunk header
// while the row warps pack codewords.
// Shared memory: tile image (header | sign/mantissa plane | exponent region)
// | staged exponent bytes | code tables | per-(row warp, lane) bit counts.
constexpr uint32_t kImgBytes = kTileHdr + kTile + kTile;
constexpr int kRowWarpsPerHalf = 7;
constexpr int kRowWarps = 2 * kRowWarpsPerHalf;
constexpr int kCtlWarp = kRowWarps;
constexpr int kEncThreads = 32 * (kRowWarps + 1);
constexpr int kMaxRowsPerWarp = (kRows + kRowWarpsPerHalf - 1) / kRowWarpsPerHalf;
constexpr uint32_t kEncSmem = kImgBytes + kTile + kEncTableWords * 4 + kRowWarps * 32 * 4;

__device__ __forceinline__ uint32_t warp_row_begin(uint32_t w) {
  return (kRows * (w % kRowWarpsPerHalf)) / kRowWarpsPerHalf;
}
__device__ __forceinline__ uint32_t warp_row_end(uint32_t w) {
  return (kRows * (w % kRowWarpsPerHalf + 1)) / kRowWarpsPerHalf;
}

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

// Pair index x0 | x1 << 4 of the two BF16 values in word w, with
// x = e - base inside the window and 15 (escape) outside it.
__device__ __forceinline__ uint32_t pair_index(uint32_t w, uint32_t base) {
  const uint32_t x0 = min(((w >> 7) & 0xFFu) - base, 15u);  // wraps below base -> escape
  const uint32_t x1 = min(((w >> 23) & 0xFFu) - base, 15u);
  return x0 | (x1 << 4);
}

// The same from two exponent bytes at positions b and b + 1 of e4.
__device__ __forceinline__ uint32_t pair_index_bytes(uint32_t e4, uint32_t b, uint32_t base) {
  const uint32_t x0 = min(((e4 >> (8 * b)) & 0xFFu) - base, 15u);
  const uint32_t x1 = min(((e4 >> (8 * b + 8)) & 0xFFu) - base, 15u);
  return x0 | (x1 << 4);
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

// Sign/mantissa bytes and exponent bytes of the 8 values in 4 words.
__device__ __forceinline__ void split8(const uint32_t (&w)[4], uint32_t& sm0, uint32_t& sm1, uint32_t& ex0,
                                       uint32_t& ex1) {
  uint32_t e2[4], s2[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    e2[p] = (w[p] >> 7) & 0x00FF00FFu;
    s2[p] = ((w[p] >> 8) & 0x00800080u) | (w[p] & 0x007F007Fu);
  }
  ex0 = __byte_perm(e2[0], e2[1], 0x6420);
  ex1 = __byte_perm(e2[2], e2[3], 0x6420);
  sm0 = __byte_perm(s2[0], s2[1], 0x6420);
  sm1 = __byte_perm(s2[2], s2[3], 0x6420);
}

__global__ void __launch_bounds__(kEncThreads, 2) zc_encode_kernel(EncodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* img = smem;
  uint8_t* exps = smem + kImgBytes;  // exponent bytes in element order
  uint32_t* tab = reinterpret_cast<uint32_t*>(smem + kImgBytes + kTile);  // per exponent: code | len << 24
  uint32_t* pair = tab + 256;                                             // per symbol pair
  uint32_t* part = tab + kEncTableWords;  // [row warp][lane] bits, then bit offsets
  __shared__ uint32_t s_item, s_mode, s_err, s_size;
  __shared__ uint32_t s_segstart[kSegs];
  __shared__ unsigned long long s_goff;

  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    s_item = atomicAdd(&a.hdr->counter, 1u);  // tiles start in claim order
    s_err = 0;
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
  const uint32_t sm_pad = (uint32_t)pad16(nt);
  const uint32_t exp_off = kTileHdr + sm_pad;

  // Tables from the select kernel; zero the padding of the sign/mantissa
  // plane and staging, and the exponent area (boundary words are OR-ed in).
  for (uint32_t i = tid; i < kEncTableWords; i += kEncThreads) tab[i] = __ldg(a.tables + (size_t)c * kEncTableWords + i);
  if (tid < 16 && nt + tid < sm_pad) {
    img[kTileHdr + nt + tid] = 0;
    exps[nt + tid] = 0;
  }
  for (uint32_t o = tid * 16; o < sm_pad; o += kEncThreads * 16)
    *reinterpret_cast<uint4*>(img + exp_off + o) = make_uint4(0, 0, 0, 0);
  __syncthreads();

  const uint32_t rb = warp < kRowWarps ? warp_row_begin(warp) : kRows;
  const uint32_t re = warp < kRowWarps ? warp_row_end(warp) : kRows;
  const uint32_t col = (warp < kRowWarps ? (warp / kRowWarpsPerHalf) * kHalf : 0u) + lane * kLaneElems;

  // Phase A (row warps): 16-B loads; sign/mantissa bytes to the image,
  // exponent bytes to the staging area; sum the code lengths (pair table,
  // which counts the 8 raw bits of an escape).
  const bool full = nt == kTile && vec;
  if (warp < kRowWarps) {
    uint32_t bits = 0;
    if (full) {
      uint4 v[kMaxRowsPerWarp];
#pragma unroll
      for (int r = 0; r < kMaxRowsPerWarp; ++r)
        if (rb + r < re) v[r] = ld_stream_v4(x + (rb + r) * kRow + col);
#pragma unroll
      for (int r = 0; r < kMaxRowsPerWarp; ++r) {
        if (rb + r < re) {
          const uint32_t i0 = (rb + r) * kRow + col;
          const uint32_t w[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
          uint32_t sm0, sm1, ex0, ex1;
          split8(w, sm0, sm1, ex0, ex1);
          *reinterpret_cast<uint2*>(img + kTileHdr + i0) = make_uint2(sm0, sm1);
          *reinterpret_cast<uint2*>(exps + i0) = make_uint2(ex0, ex1);
          bits += (pair[pair_index(w[0], base)] >> 26) + (pair[pair_index(w[1], base)] >> 26) +
                  (pair[pair_index(w[2], base)] >> 26) + (pair[pair_index(w[3], base)] >> 26);
        }
      }
    } else {
      for (uint32_t row = rb; row < re; ++row) {
        const uint32_t i0 = row * kRow + col;
        const uint32_t cnt = nt > i0 ? min(8u, nt - i0) : 0u;
        uint32_t w[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint32_t lo = (2 * p < (int)cnt) ? x[i0 + 2 * p] : 0u;
          const uint32_t hi = (2 * p + 1 < (int)cnt) ? x[i0 + 2 * p + 1] : 0u;
          w[p] = lo | (hi << 16);
        }
        uint32_t sm0, sm1, ex0, ex1;
        split8(w, sm0, sm1, ex0, ex1);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (t < (int)cnt) {
            const uint32_t e = ((t < 4 ? ex0 : ex1) >> (8 * (t & 3))) & 0xFFu;
            img[kTileHdr + i0 + t] = (uint8_t)((t < 4 ? sm0 : sm1) >> (8 * (t & 3)));
            exps[i0 + t] = (uint8_t)e;
            bits += tab[e] >> 24;
          }
        }
      }
    }
    part[warp * 32 + lane] = bits;
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
  } else if (s_mode == 0) {
    // Phase D (row warps): pack codewords into the exponent region; raw tiles
    // are stored straight from the staging area.
    BitSink sink;
    sink.begin(reinterpret_cast<uint32_t*>(img + exp_off + kSegTab),
               s_segstart[(warp / kRowWarpsPerHalf) * 32 + lane] + part[warp * 32 + lane]);
#pragma unroll 1
    for (uint32_t row = rb; row < re; ++row) {
      const uint32_t i0 = row * kRow + col;
      const uint32_t cnt = full ? 8u : (nt > i0 ? min(8u, nt - i0) : 0u);
      if (cnt == 0) break;
      const uint2 e8 = *reinterpret_cast<const uint2*>(exps + i0);
      uint32_t p0 = 0, p1 = 0, p2 = 0, p3 = 0;
      if (cnt == 8) {
        p0 = pair[pair_index_bytes(e8.x, 0, base)];
        p1 = pair[pair_index_bytes(e8.x, 2, base)];
        p2 = pair[pair_index_bytes(e8.y, 0, base)];
        p3 = pair[pair_index_bytes(e8.y, 2, base)];
      }
      if (__builtin_expect(cnt == 8 && !((p0 | p1 | p2 | p3) & kPairEsc), 1)) {
        sink.put(p0 & 0xFFFFFu, p0 >> 26);
        sink.put(p1 & 0xFFFFFu, p1 >> 26);
        sink.put(p2 & 0xFFFFFu, p2 >> 26);
        sink.put(p3 & 0xFFFFFu, p3 >> 26);
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (t < (int)cnt) {
            const uint32_t en = tab[((t < 4 ? e8.x : e8.y) >> (8 * (t & 3))) & 0xFFu];
            sink.put(en & 0xFFFFFFu, en >> 24);
          }
        }
      }
    }
    sink.finish();
  }
  fence_proxy_async_smem();
  __syncthreads();

  // Phase E: TMA bulk store of the finished tile: one copy for a coded tile,
  // image head + staged exponents for a raw tile.  The CTA leaves once shared
  // memory has been read.
  if (tid == 0 && !s_err && s_size) {
    if (s_mode == 0) {
      bulk_store_issue(a.out + s_goff, img, s_size);
    } else {
      bulk_store_issue(a.out + s_goff, img, exp_off);
      bulk_store_issue(a.out + s_goff + exp_off, exps, sm_pad);
    }
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
