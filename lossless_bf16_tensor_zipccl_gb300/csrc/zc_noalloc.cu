// zc_noalloc.cu -- zipccl_decompress_reduce_noalloc: the decompress + reduce
// call for callers that may not allocate device memory.  Its workspace is a
// scratch area compiled into this library (one instance per device), so the
// caller passes no workspace and nothing is allocated on any call.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "zipccl.h"
#include "zc_format.h"

namespace {

constexpr uint64_t kScratchBytes = ZIPCCL_NOALLOC_SCRATCH_BYTES;
// status header | one record per peer (256-B padded) | one 4-KB decode table per peer
static_assert(kScratchBytes == sizeof(zc::WsHeader) +
                                   (sizeof(zc::DecChunk) * ZIPCCL_NOALLOC_MAX_PEERS + 255) / 256 * 256 +
                                   (uint64_t)ZIPCCL_NOALLOC_MAX_PEERS * zc::kLutEntries * sizeof(uint32_t),
              "scratch size must match the reduce workspace for the maximum peer count");

// The scratch itself: a __device__ variable has one instance on every device
// the library's module is loaded on.
__device__ __align__(256) uint8_t g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of the current device's scratch, looked up once per device.
zipccl_status current_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ZIPCCL_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return ZIPCCL_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ZIPCCL_OK;
}

}  // namespace

extern "C" zipccl_status zipccl_decompress_reduce_noalloc(const void* const* d_peer_chunks,
                                                          const uint64_t* peer_chunk_bytes, uint32_t k, uint64_t n,
                                                          uint16_t* d_out, void** d_scratch, void* stream) {
  if (!d_peer_chunks || !peer_chunk_bytes || k == 0 || k > ZIPCCL_NOALLOC_MAX_PEERS || (n > 0 && !d_out))
    return ZIPCCL_ERR_INVALID_ARG;
  uint64_t need = 0;
  zipccl_status st = zipccl_reduce_workspace_bytes(k, &need);
  if (st != ZIPCCL_OK) return st;
  if (need > kScratchBytes) return ZIPCCL_ERR_CAPACITY;
  void* ws = nullptr;
  st = current_scratch(&ws);
  if (st != ZIPCCL_OK) return st;
  if (d_scratch) *d_scratch = ws;
  return zipccl_decompress_reduce(d_peer_chunks, peer_chunk_bytes, k, n, d_out, ws, kScratchBytes, stream);
}
