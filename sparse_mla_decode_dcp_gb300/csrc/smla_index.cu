// DCP filter + convert: global top-k token ids -> this rank's local slots.
//
// "FlashMLA sparse fp8 path + DCP + MTP", implementation breakdown step 2
// and the _forward_fp8_kv_mixed_batch snippet: ids owned by another rank
// become -1 in place; owned ids go through the rank's paged block table.
// With interleave size I, runs of I consecutive positions go to the ranks in
// turn: position t lives on rank (t div I) mod D at rank-local position
// (t div (I D)) I + t mod I (I = 1: rank t mod D, position t div D, the only
// size the pages validate -- implementation breakdown step 4).  The per-row
// count of surviving ids is emitted in the same pass (the "valid counts" of
// "[eldritch] attention: support DCP in SM120 FlashInfer sparse MLA",
// Summary).
//
// Layout: one CTA of 512 threads per query row; a thread converts four
// consecutive entries per 16-byte load and store (at K = 2048 the whole row
// in one step).  The CTA stages the request's block-table row in shared
// memory with coalesced loads issued together with its top-k loads, so an
// entry costs one memory round trip (not a top-k load followed by a
// dependent block-table load).  Divisions by I, D and the block size use
// multiply-shift constants fixed per launch; the row's valid count is a
// block reduction.
#include "../../include/smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

__device__ unsigned int g_index_error;

constexpr int kThreads = 512;
constexpr int kBtStage = 4096;  // block-table entries staged in shared memory

struct RowCtx {
  const int32_t* bt;    // this request's block-table row (global)
  const int32_t* bt_s;  // its first kBtStage entries (shared)
  int32_t bt_width, D, rank, I, block_size;
  FastDiv div_I, div_D, div_bs;
  bool bad_req;
};

__device__ __forceinline__ int32_t convert_one(int32_t t, const RowCtx& c, unsigned& err) {
  if (t < 0 || c.bad_req) return -1;
  const uint32_t g = fastdiv(uint32_t(t), c.div_I);  // run of I positions
  const uint32_t round = fastdiv(g, c.div_D);        // round of D runs
  const int32_t owner = int32_t(g - round * uint32_t(c.D));
  if (owner != c.rank) return -1;
  const int32_t lp = int32_t(round) * c.I + (t - int32_t(g) * c.I);  // rank-local position
  const int32_t col = int32_t(fastdiv(uint32_t(lp), c.div_bs));     // logical block
  if (col >= c.bt_width) {
    err |= SMLA_DEVERR_BLOCK_TABLE;
    return -1;
  }
  const int32_t blk = col < kBtStage ? c.bt_s[col] : __ldg(c.bt + col);
  if (blk < 0) {
    err |= SMLA_DEVERR_BLOCK_TABLE;
    return -1;
  }
  const int64_t slot = int64_t(blk) * c.block_size + (lp - col * c.block_size);
  if (slot > INT32_MAX) {
    err |= SMLA_DEVERR_BLOCK_TABLE;
    return -1;
  }
  return int32_t(slot);
}

template <bool kVec4>
__global__ void __launch_bounds__(kThreads)
    filter_convert_kernel(IndexArgs a, FastDiv div_I, FastDiv div_D, FastDiv div_bs) {
  __shared__ int32_t bt_s[kBtStage];
  __shared__ int warp_sum[kThreads / 32];
  const int64_t i = blockIdx.x;
  const int32_t r = a.req_id[i];
  RowCtx c;
  c.bad_req = (r < 0 || r >= a.num_reqs);
  c.bt = a.block_table + (c.bad_req ? 0 : int64_t(r) * a.bt_row_stride);
  c.bt_s = bt_s;
  c.bt_width = a.bt_width;
  c.D = a.D;
  c.rank = a.rank;
  c.I = a.interleave;
  c.block_size = a.block_size;
  c.div_I = div_I;
  c.div_D = div_D;
  c.div_bs = div_bs;
  unsigned err = (c.bad_req && threadIdx.x == 0) ? unsigned(SMLA_DEVERR_REQ_ID) : 0u;

  const int32_t* in = a.topk + i * a.K;
  int32_t* out = a.local_slots + i * a.K;
  // this thread's first group of entries, loaded before the block-table
  // staging so that both are in flight together
  const int first = kVec4 ? 4 * int(threadIdx.x) : int(threadIdx.x);
  int4 v0 = make_int4(-1, -1, -1, -1);
  int s0 = -1;
  if (first < a.K) {
    if (kVec4)
      v0 = *reinterpret_cast<const int4*>(in + first);
    else
      s0 = in[first];
  }
  if (!c.bad_req) {
    const int w = min(c.bt_width, kBtStage);
    for (int col = threadIdx.x; col < w; col += kThreads) bt_s[col] = __ldg(c.bt + col);
  }
  __syncthreads();

  int count = 0;
  if (kVec4) {
    for (int j = first; j < a.K; j += 4 * kThreads) {
      const int4 v = (j == first) ? v0 : *reinterpret_cast<const int4*>(in + j);
      int4 o;
      o.x = convert_one(v.x, c, err);
      o.y = convert_one(v.y, c, err);
      o.z = convert_one(v.z, c, err);
      o.w = convert_one(v.w, c, err);
      *reinterpret_cast<int4*>(out + j) = o;
      count += (o.x >= 0) + (o.y >= 0) + (o.z >= 0) + (o.w >= 0);
    }
  } else {
    for (int j = first; j < a.K; j += kThreads) {
      const int32_t o = convert_one(j == first ? s0 : in[j], c, err);
      out[j] = o;
      count += (o >= 0);
    }
  }
  if (err) atomicOr(&g_index_error, err);
  if (a.valid_count == nullptr) return;
  // the row's count: a block reduction
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) count += __shfl_xor_sync(0xffffffffu, count, off);
  if ((threadIdx.x & 31) == 0) warp_sum[threadIdx.x >> 5] = count;
  __syncthreads();
  if (threadIdx.x == 0) {
    int total = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) total += warp_sum[w];
    a.valid_count[i] = total;
  }
}

}  // namespace

cudaError_t launch_filter_convert(const IndexArgs& a, cudaStream_t s) {
  const bool vec = (a.K % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.topk) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.local_slots) % 16 == 0);
  const FastDiv div_I = make_fastdiv(uint32_t(a.interleave));
  const FastDiv div_D = make_fastdiv(uint32_t(a.D));
  const FastDiv div_bs = make_fastdiv(uint32_t(a.block_size));
  const dim3 grid(unsigned(a.T)), block(kThreads);
  if (vec)
    filter_convert_kernel<true><<<grid, block, 0, s>>>(a, div_I, div_D, div_bs);
  else
    filter_convert_kernel<false><<<grid, block, 0, s>>>(a, div_I, div_D, div_bs);
  return cudaGetLastError();
}

cudaError_t index_error_word(uint32_t* flags, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_index_error, sizeof(v));
  if (e != cudaSuccess) return e;
  *flags |= v;
  if (clear) {
    v = 0;
    e = cudaMemcpyToSymbol(g_index_error, &v, sizeof(v));
  }
  return e;
}

}  // namespace smla
