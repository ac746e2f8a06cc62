// zc_decode.cu -- decompressor and fused decompress + reduce kernels, sm_103a.
//
// "ZipCCL: Efficient Lossless Data Compression of Communication Collectives
// for Accelerating LLM Training":
//   - Fig. 6 caption: the GPU decompressor restores each value from its raw
//     sign/mantissa byte and its decoded exponent;  pith summary: lossless,
//     every byte restored;
//   - Fig. 3 / Fig. 5 captions: zipcclReduceScatter receives the peers'
//     compressed chunks, then decompresses and reduces them ->
//     zc_reduce_kernel decodes the same half tile of k peer chunks and sums in
//     fp32 in rank order, with no bf16 round trip through global memory.
//
// Decoding is table-driven: one 1024-entry table per chunk (built from the
// code lengths in the chunk header) returns up to five symbols per lookup.
// A tile's 64 segments are decoded by two warps, one lane per segment; the
// segments interleave 8 values at a time along each 512-value row, so a
// warp's stores of BF16 words stay coalesced while every lane runs its own
// bitstream.  The exponent bitstream and the sign/mantissa bytes arrive in
// shared memory by TMA bulk copies.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "zc_device.cuh"
#include "zc_kernels.h"

namespace zc {

__device__ __forceinline__ uint32_t ld_u32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint64_t ld_u64(const uint8_t* p) { return *reinterpret_cast<const uint64_t*>(p); }

// Header checks shared by both prep kernels; returns 0 or a status code.
struct HeaderInfo {
  uint64_t n;
  uint32_t n_tiles;
  uint32_t base;
  uint64_t lens;
};

__device__ uint32_t check_header(const uint8_t* ch, uint64_t bytes, HeaderInfo& h) {
  if (bytes < kChunkHdr) return kStCorrupt;
  if (ld_u32(ch) != kMagic) return kStCorrupt;
  const uint32_t w1 = ld_u32(ch + 4);
  if ((w1 & 0xFFFFu) != kVersion || ((w1 >> 16) & 0xFFu) != kTileLog2 || (w1 >> 24) != kSegLog2) return kStVersion;
  h.n = ld_u64(ch + 8);
  h.n_tiles = ld_u32(ch + 16);
  h.base = ch[20];
  h.lens = ld_u64(ch + 24);
  if (h.n >= (1ull << 40) || h.n_tiles != tiles_of(h.n)) return kStCorrupt;
  if (chunk_hdr_bytes(h.n_tiles) > bytes || h.base > 240 || !lens_complete(h.lens)) return kStCorrupt;
  return 0;
}

// Tile k of a chunk, validated against the chunk's extent, as seen by the
// warp decoding half `half` (segments 32 half .. 32 half + 31).
struct TileView {
  const uint8_t* tile;
  uint32_t mode, exp_off, exp_bytes;
  uint32_t start;           // this lane's segment: first bit in the payload (coded tiles)
  uint32_t hbit0, hbit1;    // bit range of this half's segments in the payload
  uint32_t bits;            // payload bits of the whole tile
};

__device__ bool open_tile(const uint8_t* ch, uint64_t bytes, uint32_t n_tiles, uint32_t k, uint32_t nt,
                          uint32_t half, uint32_t lane, TileView& tv) {
  tv.tile = ch;
  tv.mode = 1;
  tv.exp_off = tv.exp_bytes = tv.start = tv.hbit0 = tv.hbit1 = tv.bits = 0;
  const uint64_t toff = ld_u32(ch + kChunkHdr + 4ull * k);
  if ((toff & 15) || toff < chunk_hdr_bytes(n_tiles) || toff + kTileHdr > bytes) return false;
  const uint8_t* t = ch + toff;
  const uint4 h = *reinterpret_cast<const uint4*>(t);
  tv.tile = t;
  tv.mode = h.x;
  tv.exp_bytes = h.z;
  tv.exp_off = kTileHdr + (uint32_t)pad16(nt);
  if (h.y != nt || h.x > 1 || toff + tv.exp_off + pad16(h.z) > bytes) return false;
  if (tv.mode == 1) return h.z == nt;
  if (h.z < kSegTab || ((h.z - kSegTab) & 3)) return false;
  const uint16_t* segbits = reinterpret_cast<const uint16_t*>(t + tv.exp_off);
  const uint32_t b0 = segbits[lane], b1 = segbits[32 + lane];
  uint32_t i0 = b0, i1 = b1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y0 = __shfl_up_sync(kFull, i0, o), y1 = __shfl_up_sync(kFull, i1, o);
    if (lane >= (uint32_t)o) {
      i0 += y0;
      i1 += y1;
    }
  }
  const uint32_t t0 = __shfl_sync(kFull, i0, 31), t1 = __shfl_sync(kFull, i1, 31);
  tv.start = half == 0 ? i0 - b0 : t0 + i1 - b1;
  tv.hbit0 = half == 0 ? 0u : t0;
  tv.hbit1 = half == 0 ? t0 : t0 + t1;
  tv.bits = t0 + t1;
  return (t0 + t1 + 31) / 32 == (h.z - kSegTab) / 4;
}

__device__ __forceinline__ uint2 load_bytes8(const uint8_t* p, uint32_t cnt) {
  if (cnt == 8) return ld_stream_v2(p);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    if (t < (int)cnt) {
      const uint32_t b = p[t];
      if (t < 4) lo |= b << (8 * t);
      else hi |= b << (8 * (t - 4));
    }
  }
  return make_uint2(lo, hi);
}

// Where a decoder reads the coded payload: a copy of payload bytes
// [lo, lo + bytes) staged in shared memory, or the payload in place in global
// memory (bit_base 0).
struct ExpSource {
  const uint32_t* words;  // word holding payload bit 8 * lo
  uint32_t bit_base;      // 8 * lo
  const uint32_t* end;    // one past the last readable word
};

// Values of row r that this lane holds (col: its first value in a row).
__device__ __forceinline__ uint32_t lane_count(uint32_t nt, uint32_t col, uint32_t r) {
  const uint32_t i0 = r * kRow + col;
  return nt > i0 ? min(8u, nt - i0) : 0u;
}

// Decode one warp's 8-value lane group of row r into 4 words (8 BF16).
// kStaged: the payload words are a shared-memory copy (see LaneDecoder).
template <bool kStaged>
struct RowSource {
  TileView tv;
  LaneDecoder<kStaged> dec;
  uint32_t nt, col;  // col: first value of this lane in a row

  __device__ __forceinline__ void start(const TileView& view, uint32_t n, uint32_t c, const uint32_t* lut,
                                        uint32_t base, const ExpSource& xs) {
    tv = view;
    nt = n;
    col = c;
    if (tv.mode == 0) dec.init(xs.words, tv.start - xs.bit_base, xs.end, lut, base);
  }

  __device__ __forceinline__ uint32_t count(uint32_t r) const { return lane_count(nt, col, r); }

  __device__ __forceinline__ uint4 row(uint32_t r, uint2 sm) {
    const uint32_t cnt = count(r);
    uint32_t lo = 0, hi = 0;
    if (tv.mode == 0) {
      dec.fill_warp(cnt);
      dec.template take8<false>(lo, hi);
    } else {
      const uint2 e = load_bytes8(tv.tile + tv.exp_off + r * kRow + col, cnt);
      lo = e.x;
      hi = e.y;
    }
    const uint2 a = merge4(lo, sm.x), b = merge4(hi, sm.y);
    return make_uint4(a.x, a.y, b.x, b.y);
  }
};

// Bytes of the payload to stage for payload bits [bit0, bit1): from the
// 16-byte boundary below bit0 up to the words the decoders may read, within
// the exponent region; 0 when that does not fit `slot`.
__device__ __forceinline__ uint32_t stage_span(const TileView& tv, uint32_t bit0, uint32_t bit1, uint32_t slot,
                                               uint32_t& lo) {
  const uint32_t pay = (uint32_t)pad16(tv.exp_bytes) - kSegTab;  // payload bytes readable in the region
  lo = (bit0 >> 7) << 4;
  const uint32_t hi = min(pay, (uint32_t)pad16(((bit1 + 31) >> 5) * 4 + 12));
  const uint32_t bytes = hi > lo ? hi - lo : 0u;
  return bytes <= slot ? bytes : 0u;
}

// Copy one chunk's 4-KB decode table into shared memory (nthreads threads).
__device__ __forceinline__ void load_lut(uint32_t* dst, const uint32_t* src, uint32_t tid, uint32_t nthreads) {
  const uint4* g = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (uint32_t i = tid; i < kLutEntries / 4; i += nthreads) d[i] = __ldg(g + i);
}

__device__ __forceinline__ void store_row(uint16_t* y, uint32_t cnt, bool vec, uint4 v) {
  if (cnt == 8 && vec) {
    *reinterpret_cast<uint4*>(y) = v;
  } else {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if (t < (int)cnt) y[t] = (uint16_t)(w[t >> 1] >> (16 * (t & 1)));
  }
}

// ---------------------------------------------------------------- decompress
// Block c < n_chunks: validate chunk c's header, build its table.  Block
// n_chunks: prefix sums of element counts and tile counts over all chunks.
// Each chunk's (or peer's) decode table is built by kLutParts blocks.
constexpr uint32_t kLutParts = 8;
constexpr uint32_t kLutPart = kLutEntries / kLutParts;

// Blocks c * kLutParts + j (j < kLutParts): validate chunk c's header and
// build part j of its table (part 0 also writes the chunk record).  The last
// block: prefix sums of element counts and tile counts over all chunks.
__global__ void __launch_bounds__(256) zc_dprep_kernel(DprepArgs a) {
  pdl_trigger();
  const uint32_t tid = threadIdx.x;
  if (blockIdx.x == 0 && tid == 0) a.hdr->epoch = a.tag;  // the call's tag, before anything can fail
  if (blockIdx.x < a.n_chunks * kLutParts) {
    const uint32_t c = blockIdx.x / kLutParts, part = blockIdx.x % kLutParts;
    const uint64_t o0 = a.offsets[c], o1 = a.offsets[c + 1], total = a.offsets[a.n_chunks];
    HeaderInfo h;
    uint32_t st = (o1 < o0 || o1 > total || (o0 & 15)) ? kStCorrupt : check_header(a.stream + o0, o1 - o0, h);
    if (st) {
      if (tid == 0 && part == 0) {
        set_status_tagged(a.hdr, a.tag, st);
        a.chunks[c].ok = 0;
      }
      return;
    }
    build_lut(h.lens, a.luts + (size_t)c * kLutEntries, part * kLutPart, kLutPart);
    if (tid == 0 && part == 0) {
      DecChunk& d = a.chunks[c];
      d.stream_off = o0;
      d.bytes = o1 - o0;
      d.n = h.n;
      d.n_tiles = h.n_tiles;
      d.base = h.base;
      d.ok = 1;
    }
    return;
  }
  // scan block
  __shared__ unsigned long long s_n[8], s_t[8];
  __shared__ int s_bad;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  const uint32_t lane = tid & 31, warp = tid >> 5;
  uint64_t carry_n = 0, carry_t = 0;
  for (uint32_t c0 = 0; c0 < a.n_chunks; c0 += 256) {
    const uint32_t c = c0 + tid;
    uint64_t nc = 0, tc = 0;
    if (c < a.n_chunks) {
      const uint64_t o0 = a.offsets[c], o1 = a.offsets[c + 1];
      if (o1 >= o0 + kChunkHdr && o1 <= a.offsets[a.n_chunks] && !(o0 & 15) && ld_u32(a.stream + o0) == kMagic) {
        nc = ld_u64(a.stream + o0 + 8);
        if (nc > a.n) {
          nc = 0;
          s_bad = 1;
        }
        tc = tiles_of(nc);
      } else {
        s_bad = 1;
      }
    }
    uint64_t in = nc, it = tc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t yn = __shfl_up_sync(kFull, in, o), yt = __shfl_up_sync(kFull, it, o);
      if (lane >= (uint32_t)o) {
        in += yn;
        it += yt;
      }
    }
    if (lane == 31) {
      s_n[warp] = in;
      s_t[warp] = it;
    }
    __syncthreads();
    uint64_t wn = 0, wt = 0, bn = 0, bt = 0;
    for (uint32_t w = 0; w < 8; ++w) {
      if (w < warp) {
        wn += s_n[w];
        wt += s_t[w];
      }
      bn += s_n[w];
      bt += s_t[w];
    }
    if (c < a.n_chunks) {
      a.chunks[c].elem_start = carry_n + wn + in - nc;
      a.item_start[c] = (uint32_t)(carry_t + wt + it - tc);
    }
    carry_n += bn;
    carry_t += bt;
    __syncthreads();
  }
  if (tid == 0) {
    a.item_start[a.n_chunks] = (uint32_t)min(carry_t, (uint64_t)a.max_items);
    a.hdr->total_items = (uint32_t)min(carry_t, (uint64_t)a.max_items);
    if (s_bad || carry_n != a.n || carry_t > a.max_items) set_status_tagged(a.hdr, a.tag, kStCorrupt);
  }
}

// One CTA per tile: warp h decodes the tile's half h (segments 32h..32h+31).
// The coded payload comes into shared memory with one TMA bulk copy;
// sign/mantissa bytes are read straight from global memory (256 contiguous
// bytes per warp and row, four rows ahead).  Shared memory stays small
// enough for 14 CTAs per SM, so a whole 64M-value bucket decodes in one wave.
constexpr uint32_t kExpSlot = 11344;  // staged payload (~2.77 bits/value); larger ones are read in place
constexpr uint32_t kSmAhead = 4;      // rows of sign/mantissa bytes in flight per lane

// The rows of one warp's half tile.  sq: the first kSmAhead rows of this
// lane's sign/mantissa bytes (full tiles), already in flight.
template <bool kStaged>
__device__ __forceinline__ void decode_rows(RowSource<kStaged>& src, bool full, const uint8_t* smp, uint16_t* y,
                                            bool vec, uint2 (&sq)[kSmAhead]) {
  if (full) {
    // full coded tile: every lane has 8 values in every row
#pragma unroll kSmAhead
    for (uint32_t r = 0; r < kRows; ++r) {
      const uint2 sm = sq[r % kSmAhead];
      if (r + kSmAhead < kRows) sq[r % kSmAhead] = ld_stream_v2(smp + (r + kSmAhead) * kRow);
      uint32_t elo, ehi;
      src.dec.fill_warp(8);
      src.dec.template take8<true>(elo, ehi);
      const uint2 u = merge4(elo, sm.x), v = merge4(ehi, sm.y);
      *reinterpret_cast<uint4*>(y + r * kRow) = make_uint4(u.x, u.y, v.x, v.y);
    }
  } else {
    const uint32_t rows = (src.nt + kRow - 1) / kRow;
    for (uint32_t r = 0; r < rows; ++r) {
      const uint32_t cnt = src.count(r);
      const uint4 v = src.row(r, load_bytes8(smp + r * kRow, cnt));
      if (cnt) store_row(y + r * kRow, cnt, vec, v);
    }
  }
}

// The same rows with the tile's whole sign/mantissa plane already in shared
// memory (pl: this lane's bytes of row 0 there; plain loads, never the
// global-only streaming loads).
__device__ __forceinline__ uint2 plane_bytes8(const uint8_t* p, uint32_t cnt) {
  if (cnt == 8) return *reinterpret_cast<const uint2*>(p);
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    if (t < (int)cnt) {
      const uint32_t b = p[t];
      if (t < 4) lo |= b << (8 * t);
      else hi |= b << (8 * (t - 4));
    }
  }
  return make_uint2(lo, hi);
}

template <bool kStaged>
__device__ __forceinline__ void decode_rows_plane(RowSource<kStaged>& src, bool full, const uint8_t* pl, uint16_t* y,
                                                  bool vec) {
  if (full) {
#pragma unroll 4
    for (uint32_t r = 0; r < kRows; ++r) {
      const uint2 sm = *reinterpret_cast<const uint2*>(pl + r * kRow);
      uint32_t elo, ehi;
      src.dec.fill_warp(8);
      src.dec.template take8<true>(elo, ehi);
      const uint2 u = merge4(elo, sm.x), v = merge4(ehi, sm.y);
      *reinterpret_cast<uint4*>(y + r * kRow) = make_uint4(u.x, u.y, v.x, v.y);
    }
  } else {
    const uint32_t rows = (src.nt + kRow - 1) / kRow;
    for (uint32_t r = 0; r < rows; ++r) {
      const uint32_t cnt = src.count(r);
      const uint4 v = src.row(r, plane_bytes8(pl + r * kRow, cnt));
      if (cnt) store_row(y + r * kRow, cnt, vec, v);
    }
  }
}

// Chunks up to this count are found by each decode CTA itself while the prep
// kernel runs (one offset and one header per thread of the 64-thread CTA).
constexpr uint32_t kEarlyChunks = 64;

// kPlane: the tile's sign/mantissa plane also comes into shared memory by
// TMA (dynamic shared memory, 32 KB), for grids of a few tiles per SM, where
// each CTA's rows would otherwise wait on their own global loads.
template <bool kPlane>
__global__ void __launch_bounds__(64) zc_decode_kernel(DecodeArgs a) {
  __shared__ __align__(128) uint8_t s_exp[kExpSlot + kStagePad];
  extern __shared__ __align__(128) uint8_t s_plane[];  // kPlane only
  __shared__ __align__(16) uint32_t s_lut[kLutEntries];
  __shared__ __align__(8) uint64_t s_xbar;
  __shared__ uint32_t s_flag[3];
  __shared__ uint32_t s_map[2];  // early chunk search: chunk + 1 (0: none), first tile of the chunk
  __shared__ uint32_t s_wtot;    // early chunk search: warp 0's tile total
  const uint32_t tid = threadIdx.x, lane = tid & 31, half = tid >> 5;
  const uint32_t item = blockIdx.x;
  const uint32_t col = half * kHalf + lane * kLaneElems;
  if (tid == 0) s_map[0] = 0;
  __syncthreads();

  // This tile's chunk c and index k in it; its tile view, payload copy and
  // first sign/mantissa loads.
  uint32_t c = 0, k = 0, nt = 0, n_tiles = 0, sbytes = 0, pbytes = 0;
  const uint8_t* ch = nullptr;
  TileView tv = {};
  bool located = false;
  uint2 sq[kSmAhead];
  auto locate = [&](uint64_t chunk_bytes, uint64_t chunk_n) {
    nt = (uint32_t)min((uint64_t)kTile, chunk_n - (uint64_t)k * kTile);
    located = k < n_tiles && kChunkHdr + 4ull * (k + 1) <= chunk_bytes &&  // same in every thread
              open_tile(ch, chunk_bytes, n_tiles, k, nt, half, lane, tv);
    uint32_t slo = 0;
    sbytes = located && tv.mode == 0 ? stage_span(tv, 0, tv.bits, kExpSlot, slo) : 0u;  // the same in both warps
    pbytes = kPlane && located ? (uint32_t)pad16(nt) : 0u;  // within the chunk: open_tile checked the region after it
    if (tid == 0 && (sbytes || pbytes)) {
      mbar_init(&s_xbar, 1);
      mbar_arrive_expect_tx(&s_xbar, sbytes + pbytes);
      if (sbytes) bulk_copy_g2s(s_exp, tv.tile + tv.exp_off + kSegTab, sbytes, &s_xbar);
      if (pbytes) bulk_copy_g2s(s_plane, tv.tile + kTileHdr, pbytes, &s_xbar);
    }
    if (!kPlane && located && nt == kTile && tv.mode == 0) {
      const uint8_t* smp = tv.tile + kTileHdr + col;
#pragma unroll
      for (uint32_t r = 0; r < kSmAhead; ++r) sq[r] = ld_stream_v2(smp + r * kRow);
    }
  };

  // While the prep kernel runs (few chunks): the prefix of tile counts over
  // the chunks, as the prep kernel forms it, from the caller's offsets and
  // the headers' value counts.  Reads stay within the chunks' extents; after
  // the wait the prep kernel's validated records must agree.
  uint32_t early_first = 0;
  if (a.n_chunks <= kEarlyChunks) {
    uint32_t tiles = 0;
    uint64_t o0 = 0, o1 = 0, cn = 0;
    if (tid < a.n_chunks) {
      o0 = a.offsets[tid];
      o1 = a.offsets[tid + 1];
      if (o1 >= o0 + kChunkHdr && o1 <= a.offsets[a.n_chunks] && !(o0 & 15)) {
        cn = ld_u64(a.stream + o0 + 8);
        tiles = cn < (1ull << 40) ? (uint32_t)tiles_of(cn) : 0u;
      }
    }
    uint32_t incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, incl, o);
      if (lane >= (uint32_t)o) incl += y;
    }
    if (tid == 31) s_wtot = incl;
    __syncthreads();
    if (half) incl += s_wtot;
    const uint32_t excl = incl - tiles;
    if (tid < a.n_chunks && item >= excl && item < incl) {  // at most one thread
      s_map[0] = tid + 1;
      s_map[1] = excl;
    }
    __syncthreads();
    if (s_map[0]) {
      c = s_map[0] - 1;
      early_first = s_map[1];
      k = item - early_first;
      const uint64_t c0 = a.offsets[c], c1 = a.offsets[c + 1];
      ch = a.stream + c0;
      n_tiles = ld_u32(ch + 16);
      locate(c1 - c0, ld_u64(ch + 8));
    }
  }
  const bool early = s_map[0] != 0;

  pdl_wait();  // chunk records and tables come from the prep kernel
  // one read of the status word per block, so both warps take the same path
  if (tid == 0) s_flag[0] = status_tagged_set(a.hdr, a.tag) || item >= a.hdr->total_items;
  __syncthreads();
  if (s_flag[0]) {
    if (tid == 0 && (sbytes || pbytes)) mbar_wait(&s_xbar, 0);  // nothing left in flight
    return;
  }
  if (!early) {
    uint32_t lo = 0, hi = a.n_chunks;  // largest c with item_start[c] <= item
    while (hi - lo > 1) {
      const uint32_t mid = (lo + hi) >> 1;
      if (a.item_start[mid] <= item) lo = mid;
      else hi = mid;
    }
    c = lo;
  }
  const DecChunk d = a.chunks[c];
  bool ok;
  if (early) {
    ok = d.ok && d.n_tiles == n_tiles && a.item_start[c] == early_first && located;
  } else {
    k = item - a.item_start[c];
    ok = d.ok && k < d.n_tiles;
    if (ok) {
      ch = a.stream + d.stream_off;
      n_tiles = d.n_tiles;
      locate(d.bytes, d.n);
      ok = located;
    }
  }
  if (lane == 0) s_flag[1 + half] = ok ? 0u : 1u;
  load_lut(s_lut, a.luts + (size_t)(d.ok ? c : 0) * kLutEntries, tid, 64);
  __syncthreads();  // the table is in place; the payload barrier is initialised
  const bool bad = s_flag[1] | s_flag[2];
  const bool timeout = (sbytes || pbytes) && __any_sync(kFull, !mbar_wait(&s_xbar, 0));
  if (bad || timeout) {
    // the copy has arrived or was given up on; the status tells the caller
    if (lane == 0) set_status_tagged(a.hdr, a.tag, bad ? kStCorrupt : kStTimeout);
    return;
  }
  const uint64_t e0 = d.elem_start + (uint64_t)k * kTile;
  uint16_t* y = a.out + e0 + col;
  const bool vec = (e0 & 7) == 0;
  const uint8_t* smp = tv.tile + kTileHdr + col;  // this lane's sign/mantissa bytes of row 0
  const bool full = nt == kTile && vec && tv.mode == 0;
  const uint8_t* pl = s_plane + col;  // kPlane: this lane's bytes of row 0 in the staged plane
  if (sbytes) {
    RowSource<true> src;
    const ExpSource xs{reinterpret_cast<const uint32_t*>(s_exp), 0u, nullptr};
    src.start(tv, nt, col, s_lut, d.base, xs);
    if constexpr (kPlane) decode_rows_plane(src, full, pl, y, vec);
    else decode_rows(src, full, smp, y, vec, sq);
  } else {
    RowSource<false> src;
    const ExpSource xs{reinterpret_cast<const uint32_t*>(tv.tile + tv.exp_off + kSegTab), 0u,
                       reinterpret_cast<const uint32_t*>(tv.tile + tv.exp_off + pad16(tv.exp_bytes))};
    src.start(tv, nt, col, s_lut, d.base, xs);
    if constexpr (kPlane) decode_rows_plane(src, full, pl, y, vec);
    else decode_rows(src, full, smp, y, vec, sq);
  }
}

// ---------------------------------------------------------------- reduce
// Blocks p * kLutParts + j: validate peer p's header, build part j of its table.
__global__ void __launch_bounds__(256) zc_rprep_kernel(ReduceArgs a) {
  pdl_trigger();
  if (blockIdx.x == 0 && threadIdx.x == 0) a.hdr->epoch = a.tag;  // the call's tag, before anything can fail
  const uint32_t p = blockIdx.x / kLutParts, part = blockIdx.x % kLutParts;
  HeaderInfo h;
  uint32_t st = check_header(a.peers[p], a.bytes[p], h);
  if (!st && h.n != a.n) st = kStCorrupt;
  if (st) {
    if (threadIdx.x == 0 && part == 0) {
      set_status_tagged(a.hdr, a.tag, st);
      a.chunks[p].ok = 0;
    }
    return;
  }
  // Peers with the same code lengths share the first such peer's table.  The
  // owner's header is validated here too, so that a table is only ever
  // shared with a peer whose own block builds it.
  uint32_t owner = p;
  for (uint32_t j = 0; j < p; ++j) {
    HeaderInfo hj;
    if (check_header(a.peers[j], a.bytes[j], hj) == 0 && hj.n == a.n && hj.lens == h.lens) {
      owner = j;
      break;
    }
  }
  if (owner == p) build_lut(h.lens, a.luts + (size_t)p * kLutEntries, part * kLutPart, kLutPart);
  if (threadIdx.x == 0 && part == 0) {
    DecChunk& d = a.chunks[p];
    d.item_start = owner;
    d.stream_off = 0;
    d.bytes = a.bytes[p];
    d.n = h.n;
    d.n_tiles = h.n_tiles;
    d.base = h.base;
    d.elem_start = 0;
    d.ok = 1;
  }
}

__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return u >> 16;
}

// Two values as packed BF16 words (a low, b high), round to nearest even,
// subnormals kept; a NaN input gives a NaN whose payload the caller fixes.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2_rn(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// One block per half tile, one warp per peer.  Each warp stages the payload
// bits of its peer's half tile in shared memory with one TMA bulk copy and
// decodes its half rows with the sign/mantissa bytes read straight from
// global memory.  The fold runs along the warps in rank order: warp 0 writes
// its row into an fp32 row accumulator, warp p adds its row once warp p - 1
// has added its own, and the last warp rounds to BF16 and stores.  Each
// hand-off is an mbarrier phase; the accumulators form a ring of kRedBufs
// rows, so warp 0 starts row r + kRedBufs once the last warp has finished
// row r.  Peers with the
// same code lengths share one decode table; when the block's peers use at
// most two tables they sit in shared memory, else the tables are read
// through L1.  A block of 8 peers needs 55 KB of shared memory and 4 blocks
// fit per SM: a 64M-element reduce (512 half tiles) runs in one wave.
constexpr uint32_t kRedSlot = 5696;  // staged half payload per peer (~2.78 bits/value; a multiple of 16 for TMA)
constexpr uint32_t kRedBufs = 2;     // fp32 half-row accumulators in the ring
constexpr uint32_t kRedAcc = kRedBufs * kHalf * 4;

// Up to this many peers, the hand-off from warp p to warp p + 1 of buffer j
// is a hardware named barrier (ids 1 .. 2 (K - 1), two warps each: one
// arrives, one waits): cheaper than an mbarrier phase.  Every warp folds the
// same rows, so each barrier sees one arrival per wait; warp p arrives for
// row r + kRedBufs only after warp p + 1 has waited for row r, since warp 0
// reuses a buffer only after the last warp has finished with it.
constexpr uint32_t kNamedFoldPeers = 8;
static_assert(1 + 2 * (kNamedFoldPeers - 1) <= 15, "named barrier ids");
__device__ __forceinline__ uint32_t fold_barrier(uint32_t p, uint32_t j) { return 1 + kRedBufs * p + j; }

// An SM holds 64 hardware named barriers, and a barrier instruction with a
// register id makes ptxas reserve all 16 for the block, so at most 4 blocks
// are resident.  For up to this many peers a second instantiation names each
// hand-off barrier as an immediate (a warp-uniform switch): its blocks
// reserve only the 2 (K - 1) + 1 ids they use and are limited by registers
// and shared memory instead (K = 1..5: 13, 10, 8, 6, 5 blocks per SM).  It
// is launched only when that takes fewer waves of blocks than the register
// ids' 4 per SM (from the occupancy API at set-up); otherwise the register
// ids, which cost no switch per row, keep the grid.  From 6 peers on,
// registers allow at most 4 blocks anyway.
constexpr uint32_t kImmFoldPeers = 5;

template <uint32_t kMaxId, bool kArrive>
__device__ __forceinline__ void fold_bar_imm(uint32_t id) {
#define ZC_FOLD_BAR(n)                                                            \
  case n:                                                                         \
    if constexpr (kMaxId >= n) {                                                  \
      if constexpr (kArrive) asm volatile("bar.arrive " #n ", 64;" ::: "memory"); \
      else asm volatile("bar.sync " #n ", 64;" ::: "memory");                     \
    }                                                                             \
    break;
  switch (id) {
    ZC_FOLD_BAR(1) ZC_FOLD_BAR(2) ZC_FOLD_BAR(3) ZC_FOLD_BAR(4) ZC_FOLD_BAR(5)
    ZC_FOLD_BAR(6) ZC_FOLD_BAR(7) ZC_FOLD_BAR(8) ZC_FOLD_BAR(9) ZC_FOLD_BAR(10)
    default: break;
  }
#undef ZC_FOLD_BAR
}

// Hand-off barrier id of a K-peer block: wait (kArrive false) or arrive.
template <uint32_t K, bool kImm, bool kArrive>
__device__ __forceinline__ void fold_bar(uint32_t id) {
  if constexpr (kImm) {
    static_assert(K <= kImmFoldPeers, "immediate ids");
    fold_bar_imm<kRedBufs * (K - 1), kArrive>(id);
  } else if constexpr (kArrive) {
    asm volatile("bar.arrive %0, 64;" ::"r"(id) : "memory");
  } else {
    asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory");
  }
}

__host__ __device__ constexpr size_t reduce_smem_bytes(uint32_t k) {
  return 2 * kLutEntries * 4 + kRedAcc + (size_t)k * (kRedSlot + 16 + 8 * kRedBufs) + kStagePad;
}

// The rows of one half tile for warp p: decode, then take part in the fold.
// done: kRedBufs x K mbarriers (buffer j, warp q at done[kRedBufs q + j]),
// 32 arrivals each.  sq: the first kSmAhead rows of this lane's sign/mantissa bytes,
// already in flight.  Returns false if a hand-off wait gave up.
template <uint32_t K, bool kImm, bool kStaged>
__device__ __forceinline__ bool reduce_rows(RowSource<kStaged>& src, const uint8_t* smp, float* acc, uint64_t* done,
                                            uint16_t* y, uint2 (&sq)[kSmAhead]) {
  const uint32_t lane = threadIdx.x & 31, p = threadIdx.x >> 5;
  const uint32_t nt = src.nt, col = src.col;
  const uint32_t rows = (nt + kRow - 1) / kRow;
  const bool fast = nt == kTile && src.tv.mode == 0;  // same for every lane of the warp
  bool live = true;  // hand-off waits still bounded by their own limit
  // fold this lane's 8 values of row r (4 words of 2 BF16) into the row
  auto fold = [&](uint32_t r, uint4 v) {
    const uint32_t j = r % kRedBufs, use = r / kRedBufs;  // buffer, and its use count before row r
    // wait for the previous warp's row r, or (warp 0) for the last warp to
    // have finished the previous row in this buffer
    if (K <= kNamedFoldPeers) {
      // warp p - 1 -> p through a named barrier per (pair, buffer); the last
      // warp -> warp 0 (the buffer is free again) through its mbarrier
      if (K > 1 && p > 0) fold_bar<K, kImm, false>(fold_barrier(p - 1, j));
      else if (K > 1 && use > 0 && live) live = mbar_wait(done + kRedBufs * (K - 1) + j, (use - 1) & 1);
    } else if (live) {
      if (p > 0) live = mbar_wait(done + kRedBufs * (p - 1) + j, use & 1);
      else if (K > 1 && use > 0) live = mbar_wait(done + kRedBufs * (K - 1) + j, (use - 1) & 1);
    }
    float* a = acc + j * kHalf + lane * kLaneElems;
    float f[8];
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[2 * q] = __uint_as_float(w4[q] << 16);
      f[2 * q + 1] = __uint_as_float(w4[q] & 0xFFFF0000u);
    }
    if (p > 0) {
      const float4 a0 = *reinterpret_cast<const float4*>(a), a1 = *reinterpret_cast<const float4*>(a + 4);
      const float prev[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int q = 0; q < 8; ++q) f[q] = __fadd_rn(prev[q], f[q]);
    }
    if (p + 1 < K) {
      *reinterpret_cast<float4*>(a) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(a + 4) = make_float4(f[4], f[5], f[6], f[7]);
    } else {
      const uint32_t cnt = src.count(r);
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = f32x2_to_bf16x2_rn(f[2 * q], f[2 * q + 1]);
      // the sum of the 8 values is NaN when any of them is (or when infinities
      // cancel): only then are the words formed one by one, NaN as 0x7FC0
      const float any = ((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]));
      if (__builtin_expect(any != any, 0)) {
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = f32_to_bf16_rne(f[2 * q]) | (f32_to_bf16_rne(f[2 * q + 1]) << 16);
      }
      if (cnt) store_row(y + r * kRow + col, cnt, (reinterpret_cast<uintptr_t>(y) & 15) == 0, make_uint4(o[0], o[1], o[2], o[3]));
    }
    if (K > 1 && K <= kNamedFoldPeers && p + 1 < K) fold_bar<K, kImm, true>(fold_barrier(p, j));
    else mbar_arrive(done + kRedBufs * p + j);
  };
  if (fast) {
    // full coded tile: 8 values per lane in every row
#pragma unroll kSmAhead
    for (uint32_t r = 0; r < kRows; ++r) {
      uint32_t elo, ehi;
      src.dec.fill_warp(8);
      src.dec.template take8<true>(elo, ehi);
      const uint2 sm = sq[r % kSmAhead];
      if (r + kSmAhead < kRows) sq[r % kSmAhead] = ld_stream_v2(smp + (r + kSmAhead) * kRow);
      const uint2 u = merge4(elo, sm.x), w = merge4(ehi, sm.y);
      fold(r, make_uint4(u.x, u.y, w.x, w.y));
    }
  } else {
    for (uint32_t r = 0; r < rows; ++r) {
      const uint4 v = src.row(r, sq[0]);
#pragma unroll
      for (uint32_t q = 0; q + 1 < kSmAhead; ++q) sq[q] = sq[q + 1];
      const uint32_t rn = r + kSmAhead;
      sq[kSmAhead - 1] = rn < rows ? load_bytes8(smp + rn * kRow, src.count(rn)) : make_uint2(0, 0);
      fold(r, v);
    }
  }
  return live;
}

// Instantiated per peer count K (1..16), so the fold unrolls; kImm: the
// hand-off barriers are immediates (K <= kImmFoldPeers).
template <uint32_t K, bool kImm>
__global__ void __launch_bounds__(32 * K) zc_reduce_kernel(ReduceArgs a) {
  extern __shared__ __align__(128) uint8_t rsm[];
  const uint32_t lane = threadIdx.x & 31, p = threadIdx.x >> 5, tid = threadIdx.x;
  const uint32_t t = blockIdx.x >> 1, half = blockIdx.x & 1;
  // two decode tables | kRedBufs fp32 half rows | k x kRedSlot staged
  // payloads | kStagePad | k x (2 copy + kRedBufs hand-off) barrier words
  uint32_t* s_lut = reinterpret_cast<uint32_t*>(rsm);
  float* acc = reinterpret_cast<float*>(rsm + 2 * kLutEntries * 4);
  uint8_t* slots = rsm + 2 * kLutEntries * 4 + kRedAcc;
  uint64_t* bars = reinterpret_cast<uint64_t*>(slots + (size_t)K * kRedSlot + kStagePad);
  uint64_t* done = bars + 2 * K;
  __shared__ int s_bad;
  __shared__ uint32_t s_own[kMaxPeers];
  if (tid == 0) s_bad = 0;
  if (tid < kRedBufs * K) mbar_init(done + tid, 32);
  __syncthreads();
  // While the prep kernel runs: locate this half tile in the peer's chunk,
  // start the copy of its payload and the first sign/mantissa loads.  These
  // reads are bounded by the caller's byte count alone; the header is
  // validated by the prep kernel, and its tile count is checked against the
  // one used here after the wait.
  const uint32_t nt = (uint32_t)min((uint64_t)kTile, a.n - (uint64_t)t * kTile);
  const uint8_t* ch = a.peers[p];
  const uint64_t bytes = a.bytes[p];
  const uint32_t n_tiles = bytes >= kChunkHdr ? ld_u32(ch + 16) : 0u;
  const uint32_t col = half * kHalf + lane * kLaneElems;
  TileView tv = {};
  const bool located = t < n_tiles && kChunkHdr + 4ull * (t + 1) <= bytes &&  // same for the whole warp
                       open_tile(ch, bytes, n_tiles, t, nt, half, lane, tv);
  const uint8_t* payload = tv.tile + tv.exp_off + kSegTab;
  uint8_t* slot = slots + (size_t)p * kRedSlot;
  uint64_t* bar = bars + 2 * p;
  uint32_t slo = 0, sbytes = 0;
  if (located && tv.mode == 0) sbytes = stage_span(tv, tv.hbit0, tv.hbit1, kRedSlot, slo);
  if (lane == 0 && sbytes) {
    mbar_init(bar, 1);
    mbar_arrive_expect_tx(bar, sbytes);
    bulk_copy_g2s(slot, payload + slo, sbytes, bar);
  }
  __syncwarp();
  const uint8_t* smp = tv.tile + kTileHdr + col;  // this lane's sign/mantissa bytes of row 0
  const uint32_t rows = (nt + kRow - 1) / kRow;
  uint2 sq[kSmAhead];
#pragma unroll
  for (uint32_t r = 0; r < kSmAhead; ++r)
    sq[r] = located && r < rows ? load_bytes8(smp + r * kRow, lane_count(nt, col, r)) : make_uint2(0, 0);

  pdl_wait();  // peer records and tables come from the prep kernel
  const bool timeout = __any_sync(kFull, sbytes && !mbar_wait(bar, 0));
  const DecChunk d = a.chunks[p];
  const bool ok = located && d.ok && d.n_tiles == n_tiles;
  // one read of the status word per block, so every thread takes the same path
  if (tid == 0 && status_tagged_set(a.hdr, a.tag)) s_bad = 1;
  if (lane == 0) {
    s_own[p] = d.item_start;  // the peer owning this peer's table
    if (!ok || timeout) {
      s_bad = 1;
      set_status_tagged(a.hdr, a.tag, ok ? kStTimeout : kStCorrupt);
    }
  }
  // Decoders for the whole block: staged when every coded peer is staged (a
  // raw peer has none)
  const bool staged = __syncthreads_and(sbytes != 0 || tv.mode != 0) != 0;
  if (s_bad) return;  // uniform; a copy that did arrive has nothing left in flight
  // At most two tables (peer 0's and the first other one) go to shared memory.
  uint32_t o1 = 0;
  bool two = true;
#pragma unroll
  for (uint32_t q = 0; q < K; ++q) {
    const uint32_t o = s_own[q];
    if (o != 0 && o1 == 0) o1 = o;
    two = two && (o == 0 || o == o1);
  }
  if (p == 0) load_lut(s_lut, a.luts, lane, 32);  // peer 0 always owns its table
  if (p == (K > 1 ? 1u : 0u) && o1) load_lut(s_lut + kLutEntries, a.luts + (size_t)o1 * kLutEntries, lane, 32);
  __syncthreads();
  uint16_t* y = a.out + (uint64_t)t * kTile;
  const ExpSource sx{reinterpret_cast<const uint32_t*>(slot), 8 * slo, nullptr};
  bool live;
  if (staged && two) {
    RowSource<true> src;
    src.start(tv, nt, col, d.item_start == 0 ? s_lut : s_lut + kLutEntries, d.base, sx);
    live = reduce_rows<K, kImm>(src, smp, acc, done, y, sq);
  } else if (staged) {
    RowSource<true> src;
    src.start(tv, nt, col, a.luts + (size_t)d.item_start * kLutEntries, d.base, sx);
    live = reduce_rows<K, kImm>(src, smp, acc, done, y, sq);
  } else {
    RowSource<false> src;
    const ExpSource xs{reinterpret_cast<const uint32_t*>(payload), 0u,
                       reinterpret_cast<const uint32_t*>(tv.tile + tv.exp_off + pad16(tv.exp_bytes))};
    src.start(tv, nt, col, a.luts + (size_t)d.item_start * kLutEntries, d.base, xs);
    live = reduce_rows<K, kImm>(src, smp, acc, done, y, sq);
  }
  if (!live && lane == 0) set_status_tagged(a.hdr, a.tag, kStTimeout);
}

// ---------------------------------------------------------------- launchers
// Per device: the reduce kernels' shared-memory limits are set.  Calls from
// several host threads may both do the set-up; each stores the same value.
static std::atomic<int> g_red_attr_done[64];

// Per device: SM count for the choice of decode kernel (0: not read yet).
static std::atomic<int> g_dec_sms[64];
constexpr uint32_t kPlaneCtasPerSm = 4;  // the plane-staging decoder fits 4 CTAs per SM

cudaError_t launch_decode(const DprepArgs& prep, const DecodeArgs& args, uint32_t max_items, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms = g_dec_sms[dev].load(std::memory_order_acquire);
  if (!sms) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(zc_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTile);
    if (e != cudaSuccess) return e;
    g_dec_sms[dev].store(sms, std::memory_order_release);
  }
  zc_dprep_kernel<<<prep.n_chunks * kLutParts + 1, 256, 0, s>>>(prep);
  e = cudaGetLastError();
  if (e != cudaSuccess || max_items == 0) return e;
  cudaLaunchAttribute at[2];
  // A few tiles per SM: each CTA's latency is the time, so stage the plane
  // too; more: the small CTA keeps 14 tiles per SM in flight.
  if (max_items <= kPlaneCtasPerSm * (uint32_t)sms) {
    const cudaLaunchConfig_t cfg = follow_config(dim3(max_items), dim3(64), kTile, s, false, at);
    return cudaLaunchKernelEx(&cfg, zc_decode_kernel<true>, args);
  }
  const cudaLaunchConfig_t cfg = follow_config(dim3(max_items), dim3(64), 0, s, false, at);
  return cudaLaunchKernelEx(&cfg, zc_decode_kernel<false>, args);
}

// Per device and peer count: resident blocks per SM of the register-id
// [0] and immediate-id [1] instantiations (0: none).
static std::atomic<int> g_red_occ[64][kMaxPeers + 1][2];

template <uint32_t K>
static cudaError_t reduce_setup(int dev) {
  const int smem = (int)reduce_smem_bytes(K);
  cudaError_t e = cudaFuncSetAttribute(zc_reduce_kernel<K, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  int occ = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, zc_reduce_kernel<K, false>, 32 * K, smem);
  g_red_occ[dev][K][0].store(occ, std::memory_order_relaxed);
  occ = 0;
  if constexpr (K <= kImmFoldPeers) {
    if (e == cudaSuccess) e = cudaFuncSetAttribute(zc_reduce_kernel<K, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, zc_reduce_kernel<K, true>, 32 * K, smem);
  }
  g_red_occ[dev][K][1].store(occ, std::memory_order_relaxed);
  return e;
}

template <uint32_t K>
static cudaError_t reduce_launch(const ReduceArgs& args, uint32_t blocks, bool imm, cudaStream_t s) {
  cudaLaunchAttribute at[2];
  const cudaLaunchConfig_t cfg = follow_config(dim3(blocks), dim3(32 * K), reduce_smem_bytes(K), s, false, at);
  if constexpr (K <= kImmFoldPeers) {
    if (imm) return cudaLaunchKernelEx(&cfg, zc_reduce_kernel<K, true>, args);
  }
  return cudaLaunchKernelEx(&cfg, zc_reduce_kernel<K, false>, args);
}

// Per device: SM count for the reduce's choice of instantiation (0: not read yet).
static std::atomic<int> g_red_sms[64];

cudaError_t launch_reduce(const ReduceArgs& args, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_red_attr_done[dev].load(std::memory_order_acquire)) {
    const cudaError_t es[kMaxPeers] = {
        reduce_setup<1>(dev),  reduce_setup<2>(dev),  reduce_setup<3>(dev),  reduce_setup<4>(dev),
        reduce_setup<5>(dev),  reduce_setup<6>(dev),  reduce_setup<7>(dev),  reduce_setup<8>(dev),
        reduce_setup<9>(dev),  reduce_setup<10>(dev), reduce_setup<11>(dev), reduce_setup<12>(dev),
        reduce_setup<13>(dev), reduce_setup<14>(dev), reduce_setup<15>(dev), reduce_setup<16>(dev)};
    for (const cudaError_t x : es)
      if (x != cudaSuccess) return x;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_red_sms[dev].store(sms, std::memory_order_release);
    g_red_attr_done[dev].store(1, std::memory_order_release);
  }
  zc_rprep_kernel<<<args.k * kLutParts, 256, 0, s>>>(args);
  e = cudaGetLastError();
  if (e != cudaSuccess || args.n == 0) return e;
  const uint32_t blocks = 2 * (uint32_t)tiles_of(args.n);
  // the immediate-id instantiation only where it takes fewer waves
  const uint64_t sms = (uint64_t)g_red_sms[dev].load(std::memory_order_acquire);
  const uint64_t r0 = sms * (uint64_t)g_red_occ[dev][args.k][0].load(std::memory_order_relaxed);
  const uint64_t r1 = sms * (uint64_t)g_red_occ[dev][args.k][1].load(std::memory_order_relaxed);
  const bool imm = r0 && r1 && (blocks + r1 - 1) / r1 < (blocks + r0 - 1) / r0;
  switch (args.k) {
    case 1: return reduce_launch<1>(args, blocks, imm, s);
    case 2: return reduce_launch<2>(args, blocks, imm, s);
    case 3: return reduce_launch<3>(args, blocks, imm, s);
    case 4: return reduce_launch<4>(args, blocks, imm, s);
    case 5: return reduce_launch<5>(args, blocks, imm, s);
    case 6: return reduce_launch<6>(args, blocks, imm, s);
    case 7: return reduce_launch<7>(args, blocks, imm, s);
    case 8: return reduce_launch<8>(args, blocks, imm, s);
    case 9: return reduce_launch<9>(args, blocks, imm, s);
    case 10: return reduce_launch<10>(args, blocks, imm, s);
    case 11: return reduce_launch<11>(args, blocks, imm, s);
    case 12: return reduce_launch<12>(args, blocks, imm, s);
    case 13: return reduce_launch<13>(args, blocks, imm, s);
    case 14: return reduce_launch<14>(args, blocks, imm, s);
    case 15: return reduce_launch<15>(args, blocks, imm, s);
    default: return reduce_launch<16>(args, blocks, imm, s);
  }
}

}  // namespace zc
