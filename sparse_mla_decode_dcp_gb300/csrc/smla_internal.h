// Internal launcher interface shared by the C-ABI layer and the kernel
// translation units.  Not installed; the public surface is include/smla.h.
#pragma once

#include <cuda.h>
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
  int32_t interleave;  // I: runs of I consecutive positions per rank
  int32_t* local_slots;
  int32_t* valid_count;  // may be null
};

constexpr int kMaxMerge = 16;

// Division of a non-negative 32-bit int (< 2^31) by a divisor fixed for the
// whole launch, as a multiply-high, an add and a shift (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994):
// with s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1,
// n / d = (umulhi(n, m) + n) >> s.
struct FastDiv {
  uint32_t d, mul, shift;
};

inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  uint32_t s = 0;
  while ((uint64_t(1) << s) < d) ++s;
  f.shift = s;
  f.mul = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << s) - d)) / d + 1);
  return f;
}

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fastdiv(uint32_t n, const FastDiv& f) {
  return (__umulhi(n, f.mul) + n) >> f.shift;
}
#endif

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
  // filled by the launcher from the workspace (split-K partials)
  int32_t splits;
  uint16_t* ws_o;    // [T, splits, H, 512] fp16: each split's O / l (its own softmax average)
  float* ws_ml;      // [T, splits, 2 halves, 2, H]: log2-domain max, then sum
  int32_t* ws_tick;  // [T, 2] arrival counters, left at zero by every call
  int32_t combine_in_kernel;  // 1: the last split to arrive merges the row; 0: a second kernel
  int32_t single_split;       // set by the caller: no split-K whatever T (needs K <= 2048)
  // Fused DCP step only (D > 0): global top-k ids are converted per shard in
  // the kernel prologue and all shards' keys share one softmax.
  int32_t D, block_size, num_reqs, interleave;
  FastDiv div_I, div_D, div_bs;  // set by the fused and dense launchers
  // Dense decode only: row t belongs to request t / S, whose context length
  // is ctx_lens[t / S]; raw entries are positions (dense_rank < 0, all D
  // pools) or dense_rank's local positions; max_ctx bounds the positions.
  const int32_t* ctx_lens;
  int32_t S, dense_rank, max_ctx;
  // q [T*H, 576] bf16 for TMA, set by the launcher: boxes of 64 dims x 128
  // head rows (128-byte swizzle) and 32 dims x 128 head rows (64-byte swizzle)
  CUtensorMap q_lat, q_rope;
  const int32_t* req_id;
  const int32_t* topk;
  const uint8_t* pools[kMaxMerge];
  int64_t pool_slots[kMaxMerge];
  const int32_t* bts[kMaxMerge];
  int64_t bt_stride[kMaxMerge];
  int32_t bt_width[kMaxMerge];
};

struct TopkArgs {
  const float* scores;      // [T, row_stride]: select: by local position; merge: candidates
  const int32_t* cand_ids;  // merge only: [T, row_stride] global ids, -1 = none
  const int32_t* n_cand;    // select: [T] candidates per row; merge: see `chunk`
  int64_t row_stride;
  int32_t L, M, T, K, kp;   // kp: the sort's size, a power of two >= K (set by the launcher)
  int32_t D, rank, interleave;
  FastDiv div_I;            // set by the launcher
  int32_t* out_ids;         // [T, K]
  float* out_scores;        // [T, K] or null
  // Chunked selection (set by the launcher; 0 = one CTA per row).  Select:
  // CTA (i, c) takes positions [c chunk, (c + 1) chunk) of row i and writes
  // their K best, unsorted and -1 padded, to chunk_ids / chunk_scores
  // [T, gridDim.y, K].  Merge of those: row i's entries are its first
  // ceil(n_cand[i] / chunk) slabs of K (n_cand clipped to [0, L]).
  int32_t chunk;
  int32_t* chunk_ids;
  float* chunk_scores;
};

struct MergeArgs {
  const uint16_t* outs[kMaxMerge];
  const float* lses[kMaxMerge];
  int32_t D, T, H;
  uint16_t* out;
  float* lse;
};

cudaError_t launch_filter_convert(const IndexArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_fused(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_dense(const DecodeArgs& a, cudaStream_t s);
// Library-owned split-K scratch (no allocation by anyone at call time).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
// compacted entries one decode cluster handles (the key list in its shared
// memory): a decode without split-K needs K at most this
constexpr int32_t kDecodeMaxList = 2048;
cudaError_t launch_decode_noalloc(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s);
// workspace: null, or topk_workspace_bytes(T, L, K) bytes (16-byte aligned)
// that long rows' chunked selection uses
cudaError_t launch_topk_select(const TopkArgs& a, void* workspace, cudaStream_t s);
size_t topk_workspace_bytes(int32_t T, int32_t L, int32_t K);
cudaError_t launch_topk_merge(const TopkArgs& a, cudaStream_t s);
size_t decode_workspace_bytes(int32_t T, int32_t H, int32_t K);

// The fused step from and to host memory (smla_host.cu): the caller's host
// buffers and the device staging buffers their copies fill (the decode's q
// and topk point at the same staging memory).
struct HostBuffers {
  const void* q;        // host bf16 [T, H, 576]
  const int32_t* topk;  // host [T, K]
  void* out;            // host bf16 [T, H, 512]
  float* lse;           // host [T, H]
  uint16_t* q_dev;      // device staging [T, H, 576]
  int32_t* topk_dev;    // device staging [T, K]
};
cudaError_t launch_fused_host(const DecodeArgs& a, const HostBuffers& h, int groups,
                              cudaStream_t s);

// Each kernel translation unit owns one device error word.
cudaError_t index_error_word(uint32_t* flags, bool clear);
cudaError_t decode_error_word(uint32_t* flags, bool clear);

}  // namespace smla
