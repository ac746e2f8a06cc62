// zc_kernels.h -- launch records and launchers of the sm_103a kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "zc_format.h"

namespace zc {

// Scale selection: chunk records travel as kernel parameters, kSelectBatch
// chunks per launch.
constexpr uint32_t kSelectBatch = 256;
constexpr uint32_t kEncTableWords = 512;  // per chunk: 256 per-exponent + 256 symbol-pair code entries
constexpr uint32_t kPairEsc = 1u << 20;   // symbol-pair entry holds an escape

struct SelectChunkArg {
  uint64_t elem_start;
  uint64_t n;
  uint32_t first_item;
  uint32_t n_tiles;
  int32_t q_hint;
  int32_t has_hint;
};

struct SelectArgs {
  const uint16_t* in;
  EncChunk* chunks;
  uint32_t* tables;  // per chunk: kEncTableWords code-table words
  EncItem* items;
  uint64_t* item_state;
  WsHeader* hdr;
  uint32_t chunk0;
  uint32_t count;
  int32_t base_off[16];
  uint64_t lens[16];
  SelectChunkArg c[kSelectBatch];
};

struct EncodeArgs {
  const uint16_t* in;
  uint8_t* out;
  uint64_t cap;
  uint8_t* send;       // compress-and-send: second copy of every tile (null: none)
  uint64_t send_cap;
  uint64_t* ready;     // compress-and-send: %globaltimer when chunk c was complete (nullable)
  uint64_t* offsets;
  EncChunk* chunks;
  const uint32_t* tables;
  const EncItem* items;
  uint64_t* item_state;
  WsHeader* hdr;
  uint32_t n_chunks;
  uint32_t n_items;
};

struct DprepArgs {
  const uint8_t* stream;
  const uint64_t* offsets;
  DecChunk* chunks;
  uint32_t* item_start;  // n_chunks + 1
  uint32_t* luts;        // n_chunks x 1024
  WsHeader* hdr;
  uint32_t n_chunks;
  uint32_t max_items;
  uint64_t n;
  uint64_t tag;  // the call's status tag (see WsHeader)
};

struct DecodeArgs {
  const uint8_t* stream;
  const uint64_t* offsets;  // the caller's chunk offsets (n_chunks + 1)
  const DecChunk* chunks;
  const uint32_t* item_start;
  const uint32_t* luts;
  uint16_t* out;
  WsHeader* hdr;
  uint32_t n_chunks;
  uint64_t tag;
};

struct ReduceArgs {
  const uint8_t* peers[kMaxPeers];
  uint64_t bytes[kMaxPeers];
  DecChunk* chunks;  // one per peer
  uint32_t* luts;    // k x 1024
  WsHeader* hdr;
  uint16_t* out;
  uint64_t n;
  uint32_t k;
  uint64_t tag;
};

// Launch configuration of a kernel that follows a prep kernel in the same
// stream: programmatic stream serialisation lets its CTAs be scheduled while
// the prep kernel finishes (the kernel waits for it before reading).
inline cudaLaunchConfig_t follow_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool cooperative,
                                        cudaLaunchAttribute (&at)[2]) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeCooperative;
  at[1].val.cooperative = cooperative ? 1 : 0;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cfg;
}

cudaError_t launch_select(const SelectArgs& args, cudaStream_t s);
cudaError_t launch_selftest_wait(WsHeader* hdr, uint64_t* state, int which, cudaStream_t s);
cudaError_t launch_encode(const EncodeArgs& args, uint32_t n_items, cudaStream_t s);
cudaError_t launch_decode(const DprepArgs& prep, const DecodeArgs& args, uint32_t max_items, cudaStream_t s);
cudaError_t launch_reduce(const ReduceArgs& args, cudaStream_t s);

}  // namespace zc
