// zc_api.cu -- the C ABI declared in include/zipccl.h: argument checks,
// workspace layout and kernel launches.  Nothing here allocates device
// memory or synchronizes (except zipccl_get_device_status).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <memory>

#include "zipccl.h"
#include "zc_codebook.h"
#include "zc_device.cuh"
#include "zc_format.h"
#include "zc_kernels.h"

namespace zc {
namespace {

constexpr uint64_t kMaxChunkElems = (1ull << 31) - 1;

// Measurement hook (zipccl_profile_encode_events): the caller's events that
// compress records around its encode kernel, both null when off.
std::atomic<void*> g_prof_before{nullptr};
std::atomic<void*> g_prof_after{nullptr};

// Status tag of one decompress or reduce call (see WsHeader): 56 bits, never
// 0, spread by a splitmix64 step so that a workspace's leftover bytes match
// a tag only by a 2^-56 chance.
std::atomic<uint64_t> g_tag_counter{0};
uint64_t next_status_tag() {
  for (;;) {
    uint64_t z = g_tag_counter.fetch_add(1, std::memory_order_relaxed) + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z = (z ^ (z >> 31)) & kTagMask;
    if (z) return z;
  }
}

uint64_t pad256(uint64_t x) { return (x + 255) & ~uint64_t(255); }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct EncLayout {
  uint64_t n_items;
  uint64_t off_chunks, off_tables, off_items, off_state, total;
};

EncLayout enc_layout(const uint64_t* ce, uint32_t nc) {
  EncLayout L{};
  for (uint32_t c = 0; c < nc; ++c) {
    const uint64_t t = tiles_of(ce[c]);
    L.n_items += t ? t : 1;
  }
  L.off_chunks = sizeof(WsHeader);
  L.off_tables = L.off_chunks + pad256(sizeof(EncChunk) * (uint64_t)nc);
  L.off_items = L.off_tables + pad256(4ull * kEncTableWords * nc);
  L.off_state = L.off_items + pad256(sizeof(EncItem) * L.n_items);
  L.total = L.off_state + pad256(8 * L.n_items);
  return L;
}

struct DecLayout {
  uint64_t off_chunks, off_item_start, off_luts, total;
};

DecLayout dec_layout(uint32_t nc) {
  DecLayout L{};
  L.off_chunks = sizeof(WsHeader);
  L.off_item_start = L.off_chunks + pad256(sizeof(DecChunk) * (uint64_t)nc);
  L.off_luts = L.off_item_start + pad256(4 * ((uint64_t)nc + 1));
  L.total = L.off_luts + (uint64_t)nc * kLutEntries * sizeof(uint32_t);
  return L;
}

uint64_t red_ws(uint32_t k) {
  return sizeof(WsHeader) + pad256(sizeof(DecChunk) * (uint64_t)k) + (uint64_t)k * kLutEntries * sizeof(uint32_t);
}

zipccl_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ZIPCCL_OK : ZIPCCL_ERR_CUDA; }

// Worst-case bytes of one chunk: header, table, every tile raw.
bool chunk_bound(uint64_t n, uint64_t* out) {
  if (n > kMaxChunkElems) return false;
  const uint64_t T = tiles_of(n);
  uint64_t b = chunk_hdr_bytes(T);
  if (T) {
    b += (T - 1) * (kTileHdr + 2ull * kTile);
    b += kTileHdr + 2 * pad16(n - (T - 1) * kTile);
  }
  *out = b;
  return true;
}

}  // namespace
}  // namespace zc

using namespace zc;

extern "C" {

int zipccl_format_version(void) { return (int)kVersion; }

const char* zipccl_status_string(int s) {
  switch (s) {
    case ZIPCCL_OK: return "ok";
    case ZIPCCL_ERR_INVALID_ARG: return "invalid argument";
    case ZIPCCL_ERR_CAPACITY: return "buffer too small";
    case ZIPCCL_ERR_CORRUPT: return "corrupt stream";
    case ZIPCCL_ERR_VERSION: return "unsupported stream version";
    case ZIPCCL_ERR_TIMEOUT: return "device wait timed out";
    case ZIPCCL_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

zipccl_status zipccl_max_compressed_bytes(const uint64_t* chunk_elems, uint32_t n_chunks, uint64_t* out_bytes) {
  if (!out_bytes || !chunk_elems || n_chunks == 0) return ZIPCCL_ERR_INVALID_ARG;
  uint64_t total = 0;
  for (uint32_t c = 0; c < n_chunks; ++c) {
    uint64_t b;
    if (!chunk_bound(chunk_elems[c], &b) || total + b < total) return ZIPCCL_ERR_INVALID_ARG;
    total += b;
  }
  *out_bytes = total;
  return ZIPCCL_OK;
}

zipccl_status zipccl_compress_workspace_bytes(const uint64_t* chunk_elems, uint32_t n_chunks, uint64_t* out_bytes) {
  if (!out_bytes || !chunk_elems || n_chunks == 0) return ZIPCCL_ERR_INVALID_ARG;
  for (uint32_t c = 0; c < n_chunks; ++c)
    if (chunk_elems[c] > kMaxChunkElems) return ZIPCCL_ERR_INVALID_ARG;
  *out_bytes = enc_layout(chunk_elems, n_chunks).total;
  return ZIPCCL_OK;
}

zipccl_status zipccl_decompress_workspace_bytes(uint64_t n, uint32_t n_chunks, uint64_t* out_bytes) {
  (void)n;
  if (!out_bytes || n_chunks == 0) return ZIPCCL_ERR_INVALID_ARG;
  *out_bytes = dec_layout(n_chunks).total;
  return ZIPCCL_OK;
}

zipccl_status zipccl_reduce_workspace_bytes(uint32_t k, uint64_t* out_bytes) {
  if (!out_bytes || k == 0 || k > kMaxPeers) return ZIPCCL_ERR_INVALID_ARG;
  *out_bytes = red_ws(k);
  return ZIPCCL_OK;
}

}  // extern "C"

namespace {

// zipccl_compress and zipccl_compress_send: the same kernels; with a send
// buffer the encoder also runs its sender warps.
zipccl_status compress_impl(const uint16_t* d_in, uint64_t n, const uint64_t* chunk_elems, uint32_t n_chunks,
                            const float* sigma_hint, void* d_out, uint64_t out_capacity, uint64_t* d_chunk_offsets,
                            void* d_send, uint64_t send_capacity, uint64_t* d_chunk_ready, void* d_ws,
                            uint64_t ws_bytes, void* stream) {
  if (!chunk_elems || n_chunks == 0 || !d_out || !d_chunk_offsets || !d_ws) return ZIPCCL_ERR_INVALID_ARG;
  if (d_send && (!aligned(d_send, 16) || d_send == d_out)) return ZIPCCL_ERR_INVALID_ARG;
  if (d_chunk_ready && !aligned(d_chunk_ready, 8)) return ZIPCCL_ERR_INVALID_ARG;
  if ((n > 0 && !d_in) || !aligned(d_in, 16) || !aligned(d_out, 16) || !aligned(d_chunk_offsets, 8) ||
      !aligned(d_ws, 256))
    return ZIPCCL_ERR_INVALID_ARG;
  uint64_t sum = 0, bound = 0;
  for (uint32_t c = 0; c < n_chunks; ++c) {
    uint64_t b;
    if (!chunk_bound(chunk_elems[c], &b) || bound + b < bound) return ZIPCCL_ERR_INVALID_ARG;
    sum += chunk_elems[c];
    bound += b;
  }
  if (sum != n) return ZIPCCL_ERR_INVALID_ARG;
  const EncLayout L = enc_layout(chunk_elems, n_chunks);
  if (L.n_items >= (1ull << 31)) return ZIPCCL_ERR_INVALID_ARG;
  if (out_capacity < bound || ws_bytes < L.total || (d_send && send_capacity < bound)) return ZIPCCL_ERR_CAPACITY;

  const PhaseTable* tabs = phase_tables();
  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  std::unique_ptr<SelectArgs> sa(new SelectArgs);
  memset(sa.get(), 0, sizeof(SelectArgs));
  sa->in = d_in;
  sa->chunks = reinterpret_cast<EncChunk*>(ws + L.off_chunks);
  sa->tables = reinterpret_cast<uint32_t*>(ws + L.off_tables);
  sa->items = reinterpret_cast<EncItem*>(ws + L.off_items);
  sa->item_state = reinterpret_cast<uint64_t*>(ws + L.off_state);
  sa->hdr = reinterpret_cast<WsHeader*>(ws);
  for (int r = 0; r < 16; ++r) {
    sa->base_off[r] = tabs[r].base_offset;
    sa->lens[r] = tabs[r].lens_packed;
  }
  uint64_t elem = 0, item = 0;
  for (uint32_t c0 = 0; c0 < n_chunks; c0 += kSelectBatch) {
    const uint32_t cnt = (n_chunks - c0) < kSelectBatch ? (n_chunks - c0) : kSelectBatch;
    sa->chunk0 = c0;
    sa->count = cnt;
    for (uint32_t i = 0; i < cnt; ++i) {
      const uint64_t nc = chunk_elems[c0 + i];
      const uint64_t T = tiles_of(nc);
      SelectChunkArg& a = sa->c[i];
      a.elem_start = elem;
      a.n = nc;
      a.first_item = (uint32_t)item;
      a.n_tiles = (uint32_t)T;
      a.has_hint = 0;
      a.q_hint = 0;
      if (sigma_hint && sigma_hint[c0 + i] > 0.0f) {
        double v = floor(16.0 * log2((double)sigma_hint[c0 + i]) + 0.5);
        v = v < -32768.0 ? -32768.0 : (v > 32767.0 ? 32767.0 : v);
        a.q_hint = (int32_t)v;
        a.has_hint = 1;
      }
      elem += nc;
      item += T ? T : 1;
    }
    const cudaError_t e = launch_select(*sa, s);
    if (e != cudaSuccess) return ZIPCCL_ERR_CUDA;
  }
  EncodeArgs ea;
  ea.in = d_in;
  ea.out = static_cast<uint8_t*>(d_out);
  ea.cap = out_capacity;
  ea.send = static_cast<uint8_t*>(d_send);
  ea.send_cap = d_send ? send_capacity : 0;
  ea.ready = d_send ? d_chunk_ready : nullptr;
  ea.offsets = d_chunk_offsets;
  ea.chunks = sa->chunks;
  ea.tables = sa->tables;
  ea.items = sa->items;
  ea.item_state = sa->item_state;
  ea.hdr = sa->hdr;
  ea.n_chunks = n_chunks;
  ea.n_items = (uint32_t)L.n_items;
  // measurement hook: the caller's events around the encode kernel alone
  cudaEvent_t before = static_cast<cudaEvent_t>(g_prof_before.load(std::memory_order_acquire));
  cudaEvent_t after = static_cast<cudaEvent_t>(g_prof_after.load(std::memory_order_acquire));
  if (before && after && cudaEventRecord(before, s) != cudaSuccess) return ZIPCCL_ERR_CUDA;
  const zipccl_status st = cuda_status(launch_encode(ea, (uint32_t)L.n_items, s));
  if (st == ZIPCCL_OK && before && after && cudaEventRecord(after, s) != cudaSuccess) return ZIPCCL_ERR_CUDA;
  return st;
}

}  // namespace

extern "C" {

zipccl_status zipccl_compress(const uint16_t* d_in, uint64_t n, const uint64_t* chunk_elems, uint32_t n_chunks,
                              const float* sigma_hint, void* d_out, uint64_t out_capacity,
                              uint64_t* d_chunk_offsets, void* d_ws, uint64_t ws_bytes, void* stream) {
  return compress_impl(d_in, n, chunk_elems, n_chunks, sigma_hint, d_out, out_capacity, d_chunk_offsets, nullptr, 0,
                       nullptr, d_ws, ws_bytes, stream);
}

zipccl_status zipccl_compress_send(const uint16_t* d_in, uint64_t n, const uint64_t* chunk_elems, uint32_t n_chunks,
                                   const float* sigma_hint, void* d_out, uint64_t out_capacity,
                                   uint64_t* d_chunk_offsets, void* d_send, uint64_t send_capacity,
                                   uint64_t* d_chunk_ready, void* d_ws, uint64_t ws_bytes, void* stream) {
  if (!d_send) return ZIPCCL_ERR_INVALID_ARG;
  return compress_impl(d_in, n, chunk_elems, n_chunks, sigma_hint, d_out, out_capacity, d_chunk_offsets, d_send,
                       send_capacity, d_chunk_ready, d_ws, ws_bytes, stream);
}

zipccl_status zipccl_decompress(const void* d_stream, const uint64_t* d_chunk_offsets, uint32_t n_chunks,
                                uint16_t* d_out, uint64_t n, void* d_ws, uint64_t ws_bytes, void* stream) {
  if (!d_stream || !d_chunk_offsets || n_chunks == 0 || !d_ws || (n > 0 && !d_out)) return ZIPCCL_ERR_INVALID_ARG;
  if (!aligned(d_stream, 16) || !aligned(d_chunk_offsets, 8) || !aligned(d_out, 16) || !aligned(d_ws, 256))
    return ZIPCCL_ERR_INVALID_ARG;
  const uint64_t max_items = tiles_of(n) + n_chunks;
  if (max_items >= (1ull << 31)) return ZIPCCL_ERR_INVALID_ARG;
  const DecLayout L = dec_layout(n_chunks);
  if (ws_bytes < L.total) return ZIPCCL_ERR_CAPACITY;
  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint64_t tag = next_status_tag();  // no clear of the header: errors carry this call's tag
  DprepArgs pa;
  pa.stream = static_cast<const uint8_t*>(d_stream);
  pa.offsets = d_chunk_offsets;
  pa.chunks = reinterpret_cast<DecChunk*>(ws + L.off_chunks);
  pa.item_start = reinterpret_cast<uint32_t*>(ws + L.off_item_start);
  pa.luts = reinterpret_cast<uint32_t*>(ws + L.off_luts);
  pa.hdr = reinterpret_cast<WsHeader*>(ws);
  pa.n_chunks = n_chunks;
  pa.max_items = (uint32_t)max_items;
  pa.n = n;
  pa.tag = tag;
  DecodeArgs da;
  da.stream = pa.stream;
  da.offsets = d_chunk_offsets;
  da.chunks = pa.chunks;
  da.item_start = pa.item_start;
  da.luts = pa.luts;
  da.out = d_out;
  da.hdr = pa.hdr;
  da.n_chunks = n_chunks;
  da.tag = tag;
  return cuda_status(launch_decode(pa, da, (uint32_t)max_items, s));
}

zipccl_status zipccl_decompress_reduce(const void* const* d_peer_chunks, const uint64_t* peer_chunk_bytes, uint32_t k,
                                       uint64_t n, uint16_t* d_out, void* d_ws, uint64_t ws_bytes, void* stream) {
  if (!d_peer_chunks || !peer_chunk_bytes || k == 0 || k > kMaxPeers || !d_ws || (n > 0 && !d_out))
    return ZIPCCL_ERR_INVALID_ARG;
  if (!aligned(d_out, 16) || !aligned(d_ws, 256) || n > kMaxChunkElems) return ZIPCCL_ERR_INVALID_ARG;
  ReduceArgs ra;
  memset(&ra, 0, sizeof(ra));
  for (uint32_t p = 0; p < k; ++p) {
    if (!d_peer_chunks[p] || !aligned(d_peer_chunks[p], 16)) return ZIPCCL_ERR_INVALID_ARG;
    ra.peers[p] = static_cast<const uint8_t*>(d_peer_chunks[p]);
    ra.bytes[p] = peer_chunk_bytes[p];
  }
  if (ws_bytes < red_ws(k)) return ZIPCCL_ERR_CAPACITY;
  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ra.tag = next_status_tag();  // no clear of the header: errors carry this call's tag
  ra.hdr = reinterpret_cast<WsHeader*>(ws);
  ra.chunks = reinterpret_cast<DecChunk*>(ws + sizeof(WsHeader));
  ra.luts = reinterpret_cast<uint32_t*>(ws + sizeof(WsHeader) + pad256(sizeof(DecChunk) * (uint64_t)k));
  ra.out = d_out;
  ra.n = n;
  ra.k = k;
  return cuda_status(launch_reduce(ra, s));
}

zipccl_status zipccl_profile_encode_events(void* ev_before, void* ev_after) {
  if ((ev_before == nullptr) != (ev_after == nullptr)) return ZIPCCL_ERR_INVALID_ARG;
  g_prof_after.store(nullptr, std::memory_order_release);  // never one of a new pair with one of the old
  g_prof_before.store(ev_before, std::memory_order_release);
  g_prof_after.store(ev_after, std::memory_order_release);
  return ZIPCCL_OK;
}

zipccl_status zipccl_get_device_status(const void* d_ws, void* stream) {
  if (!d_ws) return ZIPCCL_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ZIPCCL_ERR_CUDA;
  WsHeader h;
  if (cudaMemcpy(&h, d_ws, 24, cudaMemcpyDeviceToHost) != cudaSuccess) return ZIPCCL_ERR_CUDA;
  if (h.epoch == 0) return static_cast<zipccl_status>(h.status);  // compress, self-test: plain code
  // decompress, reduce: the code counts only if it carries the last call's tag
  const uint64_t w = ((uint64_t)h.status_hi << 32) | h.status;
  return (w >> 8) == h.epoch ? static_cast<zipccl_status>(w & 0xFFu) : ZIPCCL_OK;
}

zipccl_status zipccl_predict_chunk_bytes(uint64_t n, float sigma, uint64_t* out_bytes, double* out_bits_per_value) {
  if (!out_bytes || !(sigma > 0.0f) || !(sigma < INFINITY) || n > kMaxChunkElems) return ZIPCCL_ERR_INVALID_ARG;
  // the scale a hint of sigma selects (as in zipccl_compress)
  double v = floor(16.0 * log2((double)sigma) + 0.5);
  v = v < -32768.0 ? -32768.0 : (v > 32767.0 ? 32767.0 : v);
  const double bits = expected_exponent_bits((double)sigma, (int)v);
  // format sizes: header and tile table, then per tile its header, the
  // sign/mantissa plane and the exponent region, coded only when smaller
  auto tile_bytes = [&](uint64_t nt) -> uint64_t {
    const uint64_t words = (uint64_t)ceil((double)nt * bits / 32.0);
    const uint64_t coded = kSegTab + 4 * words;
    return kTileHdr + pad16(nt) + pad16(coded < nt ? coded : nt);
  };
  const uint64_t T = tiles_of(n);
  uint64_t total = chunk_hdr_bytes(T);
  if (T) total += (T - 1) * tile_bytes(kTile) + tile_bytes(n - (T - 1) * kTile);
  *out_bytes = total;
  if (out_bits_per_value) *out_bits_per_value = n ? 8.0 * (double)total / (double)n : 0.0;
  return ZIPCCL_OK;
}

zipccl_status zipccl_choose_compressed(uint64_t n, float sigma, double link_gbs, double compress_gbs,
                                       double decompress_gbs, double margin, int* use_compressed,
                                       double* predicted_speedup) {
  if (!use_compressed || !(link_gbs > 0.0) || !(compress_gbs > 0.0) || !(decompress_gbs > 0.0) || !(margin >= 0.0))
    return ZIPCCL_ERR_INVALID_ARG;
  uint64_t bytes = 0;
  const zipccl_status st = zipccl_predict_chunk_bytes(n, sigma, &bytes, nullptr);
  if (st != ZIPCCL_OK) return st;
  const double raw = 2.0 * (double)n;
  const double t_raw = raw / link_gbs;
  const double t_zip = raw / compress_gbs + (double)bytes / link_gbs + raw / decompress_gbs;
  const double speedup = t_zip > 0.0 ? t_raw / t_zip : 0.0;
  *use_compressed = speedup > 1.0 + margin ? 1 : 0;
  if (predicted_speedup) *predicted_speedup = speedup;
  return ZIPCCL_OK;
}

zipccl_status zipccl_selftest_bounded_wait(int which, void* d_ws, uint64_t ws_bytes, void* stream) {
  // which 2 reads one chunk record and one offset after the status header
  const uint64_t need = sizeof(WsHeader) + (which == 2 ? sizeof(EncChunk) + 16 : 16);
  if (which < 0 || which > 2 || !d_ws || !aligned(d_ws, 256) || ws_bytes < need) return ZIPCCL_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(d_ws);
  if (cudaMemsetAsync(ws, 0, need, s) != cudaSuccess) return ZIPCCL_ERR_CUDA;
  return cuda_status(launch_selftest_wait(reinterpret_cast<WsHeader*>(ws), reinterpret_cast<uint64_t*>(ws + sizeof(WsHeader)),
                                          which, s));
}

zipccl_status zipccl_codebook_phase(int phase, int* base_offset, uint8_t* lens16) {
  if (phase < 0 || phase > 15 || !base_offset || !lens16) return ZIPCCL_ERR_INVALID_ARG;
  const PhaseTable& t = phase_tables()[phase];
  *base_offset = t.base_offset;
  for (int s = 0; s < kNsym; ++s) lens16[s] = t.lens[s];
  return ZIPCCL_OK;
}

zipccl_status zipccl_codebook_rebuild_phase(int phase, int* base_offset, uint8_t* lens16) {
  if (phase < 0 || phase > 15 || !base_offset || !lens16) return ZIPCCL_ERR_INVALID_ARG;
  PhaseTable t;
  rebuild_phase_table(phase, &t);
  *base_offset = t.base_offset;
  for (int s = 0; s < kNsym; ++s) lens16[s] = t.lens[s];
  return ZIPCCL_OK;
}

}  // extern "C"
