// zc_format.h -- stream format v1 constants and workspace records of the
// GB300 ZipCCL path (product side; shared by host and device code).
//
// Stream format v1 (little-endian):
//   chunk  = ChunkHeader (32 B) | u32 tile_off[n_tiles] (from chunk start),
//            zero-padded to 16 B | tiles (each 16-B aligned, back to back)
//   ChunkHeader: u32 magic | u16 version | u8 tile_log2 (15) | u8 seg_log2 (9)
//            | u64 n_elems | u32 n_tiles | u8 base | u8 flags (0) | i16 q
//            | u8 lens[8]  (4-bit code lengths; symbol 2i in the low nibble)
//   tile   = TileHeader (16 B): u32 mode (0 coded, 1 raw) | u32 n_t
//            | u32 exp_bytes | u32 0
//            | sign/mantissa plane: n_t bytes (s << 7 | m), zero-padded to 16
//            | exponent region (exp_bytes, zero-padded to 16):
//                raw:   n_t exponent bytes in element order
//                coded: u16 seg_bits[64] | the 64 segment bitstreams back to
//                       back at bit granularity, zero-padded to a u32 word
//   Element i of a tile sits in row i / 512 and segment (i mod 512) / 8; a
//   segment holds its elements' exponent symbols in increasing i.  Symbol
//   x = e - base when 0 <= x <= 14, otherwise ESC (15) followed by the 8 raw
//   exponent bits.  Bits fill u32 words from the least significant bit; a
//   canonical codeword (assigned in (length, symbol) order) goes out most
//   significant bit first, i.e. it is stored bit-reversed.  Coded mode is used
//   only when 128 + 4 * ceil(sum(seg_bits) / 32) < n_t.
#pragma once
#include <stdint.h>

#ifndef __CUDACC__
#ifndef __host__
#define __host__
#endif
#ifndef __device__
#define __device__
#endif
#endif

namespace zc {

constexpr uint32_t kMagic = 0x4C43435Au;  // bytes 'Z' 'C' 'C' 'L'
constexpr uint32_t kVersion = 1;
constexpr uint32_t kTileLog2 = 15;
constexpr uint32_t kTile = 1u << kTileLog2;  // elements per tile
constexpr uint32_t kSegLog2 = 9;             // symbols per full segment: 512
constexpr uint32_t kRow = 512;               // elements per tile row
constexpr uint32_t kRows = kTile / kRow;     // 64
constexpr uint32_t kHalf = kRow / 2;         // one warp's 32 segments cover half a row
constexpr uint32_t kLaneElems = 8;           // consecutive elements of one segment per row
constexpr uint32_t kSegs = 64;
constexpr int kNsym = 16;
constexpr int kWindow = 15;
constexpr int kEsc = 15;
constexpr int kLmax = 10;
constexpr uint32_t kChunkHdr = 32;
constexpr uint32_t kTileHdr = 16;
constexpr uint32_t kSegTab = 2 * kSegs;  // u16 bit length per segment
constexpr uint32_t kMaxPeers = 16;
constexpr uint32_t kLutEntries = 1u << kLmax;

__host__ __device__ constexpr inline uint64_t pad16(uint64_t x) { return (x + 15u) & ~uint64_t(15); }
__host__ __device__ constexpr inline uint64_t tiles_of(uint64_t n) { return (n + kTile - 1) / kTile; }
__host__ __device__ constexpr inline uint64_t chunk_hdr_bytes(uint64_t n_tiles) {
  return kChunkHdr + pad16(4 * n_tiles);
}

// Code tables of format v1, frozen: for scale phase r = q mod 16, the window
// start relative to floor(q/16) + 127 and the 16 code lengths (symbol s at
// bits 4s..4s+3; symbols 0..14 are the window exponents, 15 the escape).
// They are the optimal 10-bit-limited prefix code over the closed-form
// Gaussian exponent masses at sigma = 2^(r/16) (window: the 15 consecutive
// exponents of largest mass).  The host builder in zc_codebook.cpp
// regenerates them for the tests; the library itself uses only these
// integers, so its streams do not depend on the host's erf.
constexpr int kPhaseBaseOffset[16] = {-13, -12, -12, -12, -12, -12, -12, -12,
                                      -12, -12, -12, -12, -12, -12, -12, -12};
constexpr uint64_t kPhaseLens[16] = {
    0xa5222355679aaaaaull, 0xaa4222445679aaaaull, 0xaa4222445679aaaaull, 0xaa4222445679aaaaull,
    0xaa3223345679aaaaull, 0xa932233456889aaaull, 0xa932233456889aaaull, 0xa832233456899aaaull,
    0xa8222345689aaaaaull, 0xa8222345689aaaaaull, 0xa7222345779aaaaaull, 0xa7222345779aaaaaull,
    0xa6222346679aaaaaull, 0xa6222346679aaaaaull, 0xa5222355679aaaaaull, 0xa5222355679aaaaaull};

// Look-back state word: 2-bit flag | 62-bit byte count.
constexpr uint64_t kFlagShift = 62;
constexpr uint64_t kFlagAgg = 1ull << kFlagShift;
constexpr uint64_t kFlagInc = 2ull << kFlagShift;
constexpr uint64_t kFlagErr = 3ull << kFlagShift;
constexpr uint64_t kValMask = (1ull << kFlagShift) - 1;
constexpr uint64_t kSlotValid = 1ull << 63;

// Device status codes (match zipccl_status).
constexpr uint32_t kStCorrupt = 3, kStVersion = 4, kStTimeout = 5, kStCapacity = 2;

// Workspace header, at the start of every workspace.  Compress (and the
// bounded-wait self-test) clear it first and keep a plain code in `status`.
// Decompress and reduce do not clear it: each call draws a 56-bit tag, its
// prep kernel stores the tag in `epoch`, and its kernels record an error as
// the 64-bit word (tag << 8 | code) over `status` and `status_hi`, so that a
// code left by an earlier call (or by whatever the memory held) reads as no
// error.  `epoch` = 0 marks the plain form.
struct alignas(256) WsHeader {
  uint32_t status;
  uint32_t status_hi;   // upper half of a tagged status (decompress, reduce)
  uint32_t total_items; // decode work items (decompress)
  uint32_t pad0;
  uint64_t epoch;       // the last decompress or reduce call's tag; 0: plain status
  uint64_t pad[29];
};
static_assert(sizeof(WsHeader) == 256, "ws header");
constexpr uint64_t kTagMask = (1ull << 56) - 1;

// Per-chunk record of the compress workspace.
struct alignas(64) EncChunk {
  uint64_t elem_start;  // first element of the chunk in the input
  uint64_t n;           // elements
  uint32_t first_item;  // first work item (tile) of the chunk
  uint32_t n_tiles;
  int32_t q;            // scale index: code built for sigma = 2^(q/16)
  uint32_t base;        // window start exponent
  uint64_t lens;        // 16 x 4-bit code lengths, symbol s at bits 4s..4s+3
  uint64_t start_slot;  // kSlotValid | chunk byte offset, published by tile 0
  uint64_t done;        // compress-and-send: tiles whose stores have completed
  uint64_t end;         // compress-and-send: chunk end offset, from its last tile
};
static_assert(sizeof(EncChunk) == 64, "enc chunk");

// Per-tile record of the compress workspace, written by the select kernel.
struct alignas(32) EncItem {
  uint64_t elem0;  // first input element of the tile
  uint32_t c;      // chunk
  uint32_t k;      // tile within the chunk
  uint32_t nt;     // values in the tile (0 for an empty chunk's header-only item)
  uint32_t base;   // window start exponent of the chunk
  uint32_t pad[2];
};
static_assert(sizeof(EncItem) == 32, "enc item");

// Per-chunk record of the decompress / reduce workspace.
struct alignas(64) DecChunk {
  uint64_t stream_off;  // chunk byte offset in the stream
  uint64_t bytes;       // chunk size in bytes
  uint64_t n;           // elements
  uint64_t elem_start;  // first output element
  uint32_t n_tiles;
  uint32_t base;
  uint32_t item_start;  // first decode work item
  uint32_t ok;
  uint64_t pad[2];
};
static_assert(sizeof(DecChunk) == 64, "dec chunk");

}  // namespace zc
