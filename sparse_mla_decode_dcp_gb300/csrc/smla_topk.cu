// Global top-k selection of indexer scores, the step that produces the
// sparse path's global top-k ids ("[eldritch] attention: support DCP in
// SM120 FlashInfer sparse MLA", Summary: global sparse top-k token ids;
// "FlashMLA sparse fp8 path + DCP + MTP", related PRs: the DCP sparse
// indexer's global top-k merge).
//
// The pages print no selection rule; the rule taken: a row keeps the K
// largest scores of its candidates, ranked by score descending and, among
// equal scores, by token id ascending, padded with -1 when it has fewer
// than K.  NaN ranks below every number and -0 equals +0 (the order of a
// stable ascending sort of the negated scores).  Under DCP each rank keeps
// the top-k of the positions it holds, as global ids, and the global top-k
// is the top-k of the union by the same rule.
//
// Method: every candidate gets a unique 64-bit key -- an order-preserving
// integer image of its score in the high half, the complement of its id in
// the low half -- so "the K best" is "the K largest keys".  One CTA per row
// finds the K-th largest key with a most-significant-digit radix select (8
// bits per pass over the row, stopping as soon as the boundary bucket holds
// exactly the keys still needed), gathers the keys at or above it into
// shared memory and sorts them with a bitonic network.
#include "../../include/smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kThreads = 1024;

// Order-preserving image of a float: larger score, larger key; every NaN
// maps to 0 (below -inf) and -0 to the key of +0.
__device__ __forceinline__ uint32_t score_key(float f) {
  if (f != f) return 0u;
  if (f == 0.f) f = 0.f;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

__device__ __forceinline__ uint64_t make_key(float score, int32_t id) {
  return (uint64_t(score_key(score)) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(id));
}

// Candidate j of row i: its key, or false when j is not a candidate.
template <bool kExplicit>
__device__ __forceinline__ bool candidate(const TopkArgs& a, int64_t i, int j, int n,
                                          uint64_t& key) {
  if (kExplicit) {
    const int32_t id = __ldg(a.cand_ids + i * a.row_stride + j);
    if (id < 0) return false;
    key = make_key(__ldg(a.scores + i * a.row_stride + j), id);
    return true;
  }
  if (j >= n) return false;
  // local position j of `rank` -> global position
  const uint32_t g = fastdiv(uint32_t(j), a.div_I);
  const int32_t id = int32_t(g) * a.interleave * a.D + a.rank * a.interleave +
                     (j - int32_t(g) * a.interleave);
  key = make_key(__ldg(a.scores + i * a.row_stride + j), id);
  return true;
}

template <bool kExplicit>
__global__ void __launch_bounds__(kThreads) topk_kernel(TopkArgs a) {
  extern __shared__ uint64_t buf[];  // kp keys
  __shared__ uint32_t hist[256];
  __shared__ uint64_t s_prefix, s_mask;
  __shared__ int s_need, s_done, s_count;
  const int64_t i = blockIdx.x;
  const int tid = threadIdx.x;
  const int n = kExplicit ? a.M : min(max(__ldg(a.n_cand + i), 0), a.L);
  const int span = kExplicit ? a.M : n;  // entries to scan

  // How many candidates: all of them are kept when they fit in K.
  if (tid == 0) {
    s_count = 0;
    s_prefix = 0;
    s_mask = 0;
    s_need = a.K;
    s_done = 0;
  }
  __syncthreads();
  int mine = 0;
  for (int j = tid; j < span; j += kThreads) {
    uint64_t k;
    mine += candidate<kExplicit>(a, i, j, n, k);
  }
  atomicAdd(&s_count, mine);
  __syncthreads();
  const bool select = s_count > a.K;
  __syncthreads();

  // Radix select of the K-th largest key, most significant 8 bits first.
  if (select) {
#pragma unroll 1
    for (int shift = 56; shift >= 0 && !s_done; shift -= 8) {
      for (int b = tid; b < 256; b += kThreads) hist[b] = 0;
      __syncthreads();
      const uint64_t prefix = s_prefix, mask = s_mask;
      for (int j = tid; j < span; j += kThreads) {
        uint64_t k;
        if (candidate<kExplicit>(a, i, j, n, k) && (k & mask) == prefix)
          atomicAdd(&hist[(k >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        // the bucket holding the need-th largest remaining key, from the top
        int need = s_need, sel = 0;
        for (int b = 255; b >= 0; --b) {
          const int c = int(hist[b]);
          if (c >= need) {
            sel = b;
            break;
          }
          need -= c;
        }
        s_prefix = prefix | (uint64_t(sel) << shift);
        s_mask = mask | (uint64_t(255) << shift);
        s_need = need;
        s_done = (int(hist[sel]) == need);  // the whole bucket is in
      }
      __syncthreads();
    }
  }

  // Gather the kept keys: every candidate when they fit, else those whose
  // key is at or above the boundary in the bits the select fixed (exactly K:
  // the keys are distinct).
  if (tid == 0) s_count = 0;
  __syncthreads();
  const uint64_t prefix = s_prefix, mask = s_mask;
  for (int j = tid; j < span; j += kThreads) {
    uint64_t k;
    if (candidate<kExplicit>(a, i, j, n, k) && (!select || (k & mask) >= prefix)) {
      const int p = atomicAdd(&s_count, 1);
      if (p < a.K) buf[p] = k;
    }
  }
  __syncthreads();
  const int kept = min(s_count, a.K);
  for (int p = kept + tid; p < a.kp; p += kThreads) buf[p] = 0;  // below every candidate
  __syncthreads();

  // Bitonic sort of the kp keys, descending.
#pragma unroll 1
  for (int size = 2; size <= a.kp; size <<= 1) {
#pragma unroll 1
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int p = tid; p < a.kp / 2; p += kThreads) {
        const int lo = 2 * p - (p & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t x = buf[lo], y = buf[hi];
        if ((x < y) == desc) {
          buf[lo] = y;
          buf[hi] = x;
        }
      }
      __syncthreads();
    }
  }

  for (int p = tid; p < a.K; p += kThreads) {
    const bool live = p < kept;
    const uint64_t k = buf[p];
    a.out_ids[i * a.K + p] = live ? int32_t(0xFFFFFFFFu - uint32_t(k)) : -1;
    if (a.out_scores) a.out_scores[i * a.K + p] = live ? key_score(uint32_t(k >> 32)) : 0.f;
  }
}

int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

template <bool kExplicit>
cudaError_t launch(TopkArgs a, cudaStream_t s) {
  a.kp = pow2_at_least(a.K);
  const size_t smem = size_t(a.kp) * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(topk_kernel<kExplicit>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  topk_kernel<kExplicit><<<dim3(unsigned(a.T)), dim3(kThreads), smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_topk_select(const TopkArgs& args, cudaStream_t s) {
  TopkArgs a = args;
  a.div_I = make_fastdiv(uint32_t(a.interleave));
  return launch<false>(a, s);
}

cudaError_t launch_topk_merge(const TopkArgs& args, cudaStream_t s) { return launch<true>(args, s); }

}  // namespace smla
