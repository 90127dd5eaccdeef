// DCP filter + convert: global top-k token ids -> this rank's local slots.
//
// "FlashMLA sparse fp8 path + DCP + MTP", implementation breakdown step 2
// and the _forward_fp8_kv_mixed_batch snippet: ids owned by another rank
// (interleave 1: position t lives on rank t mod D at local position t div D)
// become -1 in place; owned ids go through the rank's paged block table.
// The per-row count of surviving ids is emitted in the same pass (the
// "valid counts" of "[eldritch] attention: support DCP in SM120 FlashInfer
// sparse MLA", Summary).
//
// Layout: one CTA per query row.  Each thread converts four consecutive
// entries per step from one 16-byte load, so a warp moves 512 contiguous
// bytes of top-k ids per instruction; the block-table reads that follow hit
// L1/L2 (one row of the table serves the whole CTA).
#include "../../include/smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

__device__ unsigned int g_index_error;

constexpr int kThreads = 256;

struct RowCtx {
  const int32_t* bt;  // this request's block-table row
  int32_t bt_width, D, rank, block_size;
  bool bad_req;
};

__device__ __forceinline__ int32_t convert_one(int32_t t, const RowCtx& c,
                                               unsigned& err) {
  if (t < 0 || c.bad_req) return -1;
  const int32_t owner = t % c.D;
  if (owner != c.rank) return -1;
  const int32_t lp = t / c.D;            // rank-local position
  const int32_t col = lp / c.block_size;  // logical block
  if (col >= c.bt_width) {
    err |= SMLA_DEVERR_BLOCK_TABLE;
    return -1;
  }
  const int32_t blk = __ldg(c.bt + col);
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
    filter_convert_kernel(IndexArgs a) {
  const int64_t i = blockIdx.x;
  const int32_t r = a.req_id[i];
  RowCtx c;
  c.bad_req = (r < 0 || r >= a.num_reqs);
  c.bt = a.block_table + (c.bad_req ? 0 : int64_t(r) * a.bt_row_stride);
  c.bt_width = a.bt_width;
  c.D = a.D;
  c.rank = a.rank;
  c.block_size = a.block_size;
  unsigned err = (c.bad_req && threadIdx.x == 0) ? unsigned(SMLA_DEVERR_REQ_ID) : 0u;

  const int32_t* in = a.topk + i * a.K;
  int32_t* out = a.local_slots + i * a.K;
  int count = 0;
  if (kVec4) {
    for (int j = threadIdx.x * 4; j < a.K; j += kThreads * 4) {
      const int4 v = *reinterpret_cast<const int4*>(in + j);
      int4 o;
      o.x = convert_one(v.x, c, err);
      o.y = convert_one(v.y, c, err);
      o.z = convert_one(v.z, c, err);
      o.w = convert_one(v.w, c, err);
      *reinterpret_cast<int4*>(out + j) = o;
      count += (o.x >= 0) + (o.y >= 0) + (o.z >= 0) + (o.w >= 0);
    }
  } else {
    for (int j = threadIdx.x; j < a.K; j += kThreads) {
      const int32_t o = convert_one(in[j], c, err);
      out[j] = o;
      count += (o >= 0);
    }
  }
  if (err) atomicOr(&g_index_error, err);
  if (a.valid_count == nullptr) return;
  // block reduction of the row's count
  __shared__ int warp_sum[kThreads / 32];
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
  dim3 grid(a.T), block(kThreads);
  if (vec)
    filter_convert_kernel<true><<<grid, block, 0, s>>>(a);
  else
    filter_convert_kernel<false><<<grid, block, 0, s>>>(a);
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
