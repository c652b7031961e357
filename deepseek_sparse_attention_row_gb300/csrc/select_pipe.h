// select_pipe.h -- host interface of the pipelined selection kernels
// (select_pipe.cu) for the C ABI in dsa_cb.cu. Internal to the library.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/dsa_cb.h"

namespace dsa {

// Row layouts, as in select_kernel.
constexpr int kPipeUnsharded = 0;      // [rows, ld], window [ks, ke)
constexpr int kPipeSharded = 1;        // [shards, rows, ld], windows from 0
constexpr int kPipeShardedStarts = 2;  // [shards, rows, ld], windows from each shard's start

// One selecting call, validated by the caller (dsa_cb.cu).
struct PipeCall {
  int elem_bytes;  // 4: fp32 logits and scores; 2: bf16
  int mode;        // kPipe*
  const void* logits;
  int64_t ld;            // row stride (elements)
  int64_t shard_stride;  // elements between shards (sharded modes)
  int32_t shards;        // 1 for the unsharded form
  int32_t width;         // unsharded width, or local width of each shard
  const int32_t* row_ks;  // nullable: unsharded starts or global starts
  const int32_t* row_ke;  // ends, or global ends
  int32_t row_repeat;
  int32_t block_size;  // unsharded block, or local block
  int32_t global_block_size;
  int32_t nb;       // blocks per output row
  int32_t nb_data;  // blocks that can hold data
  int32_t pin_newest;
  int32_t topk;
  int32_t* out;
  int64_t ld_out;
  void* scores;  // nullable, elem_bytes per entry
  int64_t ld_scores;
  int64_t rows;
  void* workspace;  // nullable
  size_t workspace_size;
};

// Whether the pipelined kernels take this call (device-memory logits, a
// block size they reduce, at most 16 shards, up to 4096 blocks and top-256).
bool pipe_takes(const PipeCall& c);

// Launches the pipelined selection. Call only when pipe_takes(c). Returns
// kPipeDeclined, with nothing enqueued, when no pipelined launch shape fits
// the call (shared memory); the caller then takes another kernel.
constexpr dsa_status kPipeDeclined = static_cast<dsa_status>(-100);
dsa_status pipe_select(const PipeCall& c, void* stream);

// Workspace layout shared by every selecting kernel: a 256-byte header whose
// first two words are the pipelined kernel's unit queue and finished-CTA
// count, then one arrival counter per row, then rows * nb block keys; each
// part 256-byte aligned. All of it is zero between calls.
inline size_t ws_align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
constexpr size_t kWsHeaderBytes = 256;
inline size_t ws_counts_offset() { return kWsHeaderBytes; }
inline size_t ws_keys_offset(int64_t rows) {
  return kWsHeaderBytes + ws_align256(static_cast<size_t>(rows) * 4);
}
inline size_t ws_total_bytes(int64_t rows, int64_t nb) {
  if (rows <= 0) return 0;  // a call without rows needs no workspace
  return ws_keys_offset(rows) + ws_align256(static_cast<size_t>(rows) * static_cast<size_t>(nb) * 4);
}

// Launch-shape overrides of the pipelined kernels (0: automatic), set through
// dsa_select_set_launch_override.
void pipe_set_override(int knob, int value);
int pipe_get_override(int knob);

}  // namespace dsa
