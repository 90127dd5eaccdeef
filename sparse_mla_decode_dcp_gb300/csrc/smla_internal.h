// Internal launcher interface shared by the C-ABI layer and the kernel
// translation units.  Not installed; the public surface is include/smla.h.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace smla {

struct IndexArgs {
  const int32_t* req_id;
  const int32_t* block_table;
  int64_t bt_row_stride;
  int32_t bt_width;
  int32_t num_reqs;
  const int32_t* topk;
  int32_t T, K, D, rank, block_size;
  int32_t* local_slots;
  int32_t* valid_count;  // may be null
};

struct DecodeArgs {
  const uint16_t* q;  // bf16 [T, H, 576]
  const uint8_t* kv;  // [num_slots, 656]
  int64_t num_slots;
  const int32_t* slots;  // [T, K]
  int32_t T, H, K;
  float sm_scale;
  uint16_t* out;  // bf16 [T, H, 512]
  float* lse;     // [T, H]
  void* workspace;
  size_t workspace_bytes;
};

constexpr int kMaxMerge = 16;

struct MergeArgs {
  const uint16_t* outs[kMaxMerge];
  const float* lses[kMaxMerge];
  int32_t D, T, H;
  uint16_t* out;
  float* lse;
};

cudaError_t launch_filter_convert(const IndexArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s);
size_t decode_workspace_bytes(int32_t T, int32_t H, int32_t K);

// Each kernel translation unit owns one device error word.
cudaError_t index_error_word(uint32_t* flags, bool clear);
cudaError_t decode_error_word(uint32_t* flags, bool clear);

}  // namespace smla
