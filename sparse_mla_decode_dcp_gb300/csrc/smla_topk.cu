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
// the low half -- so "the K best" is "the K largest keys".  One CTA per row:
//   1. one pass over the row builds a histogram of the keys' top 12 bits
//      (sign, exponent and 3 mantissa bits of the score) in shared memory; a
//      block-wide suffix scan gives each bin its first place in the
//      descending order and finds the bin holding the K-th largest key;
//   2. a second pass puts every key of a higher bin at its bin's next place
//      (a counting sort by bin) and the boundary bin's keys in per-warp lists;
//   3. a most-significant-digit radix select over the boundary bin's keys (8
//      bits per step, in shared memory) picks those still needed;
//   4. the K selected keys are sorted: each warp's run in registers by a
//      bitonic network, then the runs by merges along the merge path (K up
//      to 4096; larger K: the bitonic network throughout).
// Only when the boundary bin overflows the per-warp lists (scores tied far
// beyond K) does step 3 read the row from global memory again, digit by
// digit.  Long rows get a cluster of two CTAs, each walking half of the
// row through steps 1 and 2, the second handing its queues to the first
// through distributed shared memory.  A call of few long rows may instead
// cut each row into chunks, one CTA each running steps 1-3 and writing its
// chunk's K best unsorted; a second launch of the same kernel (its merge
// front end) then selects and sorts each row's K best among its chunks'
// (the union holds them all).
#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/smla.h"
#include "smla_internal.h"
#include "smla_sm100.cuh"

namespace smla {
namespace {

constexpr int kThreads = 1024;
constexpr int kBinBits = 12;
constexpr int kBins = 1 << kBinBits;
constexpr int kBinShift = 64 - kBinBits;
constexpr int kSmemBytes = 226 * 1024;  // one CTA per SM: all of it but the static part
constexpr int kHistBytes = kBins * 4;
constexpr int kWarps = kThreads / 32;

// Distributed shared memory: a 16-byte load from, and 4- and 8-byte stores
// into, the shared memory of another CTA of the cluster (shared::cluster
// addresses from sm100::map_to_cta).
__device__ __forceinline__ uint4 ld_dsmem_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_dsmem_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" :: "r"(addr), "l"(v) : "memory");
}

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

__device__ __forceinline__ uint64_t make_key(uint32_t skey, int32_t id) {
  return (uint64_t(skey) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(id));
}

// Warp-aggregated append of `key` (for lanes with `take`) to list[*count].
// Returns nothing; entries at or past `cap` are dropped (the count still
// grows, so an overflow is visible).
__device__ __forceinline__ void append(bool take, uint64_t key, uint64_t* list, int* count, int cap) {
  const uint32_t m = __ballot_sync(0xffffffffu, take);
  if (m == 0) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(m) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(count, __popc(m));
  base = __shfl_sync(0xffffffffu, base, leader);
  if (take) {
    const int p = base + __popc(m & ((1u << lane) - 1u));
    if (p < cap) list[p] = key;
  }
}

// Global id of local position j of `rank` (select front end): runs of I
// positions go to the ranks in turn.
__device__ __forceinline__ int32_t global_id(const TopkArgs& a, int j) {
  const uint32_t g = fastdiv(uint32_t(j), a.div_I);  // run of I positions
  return int32_t(g) * a.interleave * a.D + a.rank * a.interleave + (j - int32_t(g) * a.interleave);
}

// Visit every candidate of row i, all lanes of a warp together: f(valid,
// score, x) is called by every lane, x the candidate's id (merge: entry
// j < M, skipped when its id is -1) or its local position j < n (select:
// global_id(x) is its id, computed only where needed; `base` is the first
// position a chunk-mode CTA visits).  A thread keeps
// kUnroll loads in flight: a gather's rate is set by the bytes in flight.
// The loads are issued unconditionally (at a clamped index, the result then
// masked): a branch around a load would make each wait for the one before.
// With kVec4 (select) the row's aligned middle is read 16 bytes at a time
// and its up to 3 leading and 3 trailing scores, outside any aligned quad,
// by warp 0 one per lane, so no load leaves the row whatever its alignment.
template <bool kExplicit, bool kVec4, typename F>
__device__ __forceinline__ void for_each_candidate(const TopkArgs& a, int64_t i, int base, int span,
                                                   F f) {
  const float* srow = a.scores + i * a.row_stride + base;
  if (kVec4) {
    // 16-byte loads, kUnroll per thread a step; the next step's are issued
    // before this step's scores are visited, so the loads overlap the work
    constexpr int kUnroll = 2;
    const int head = min(span, int((4u - ((reinterpret_cast<uintptr_t>(srow) >> 2) & 3u)) & 3u));
    const int nq = (span - head) >> 2;  // whole aligned quads
    const int tail = span - head - 4 * nq;
    const float4* quads = reinterpret_cast<const float4*>(srow + head);
    float4 next[kUnroll];
    if (nq > 0) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        next[u] = __ldg(quads + min(int(threadIdx.x) + u * kThreads, nq - 1));
    }
    for (int q0 = threadIdx.x; q0 - int(threadIdx.x) < nq; q0 += kThreads * kUnroll) {
      float4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) v[u] = next[u];
      const int qn = q0 + kThreads * kUnroll;  // the next step (block-uniform test)
      if (qn - int(threadIdx.x) < nq) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) next[u] = __ldg(quads + min(qn + u * kThreads, nq - 1));
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int q = q0 + u * kThreads;
        const int j = head + 4 * q;
        f(q < nq, v[u].x, base + j);
        f(q < nq, v[u].y, base + j + 1);
        f(q < nq, v[u].z, base + j + 2);
        f(q < nq, v[u].w, base + j + 3);
      }
    }
    if (threadIdx.x < 32 && head + tail > 0) {
      const int l = int(threadIdx.x);
      const bool ok = l < head + tail;
      const int j = l < head ? l : head + 4 * nq + (l - head);
      const float sc = ok ? __ldg(srow + j) : 0.f;
      f(ok, sc, base + (ok ? j : 0));
    }
    return;
  }
  const int32_t* irow = kExplicit ? a.cand_ids + i * a.row_stride : nullptr;
  constexpr int kUnroll = 8;  // 4-byte loads in flight per thread
  for (int j0 = threadIdx.x; j0 - int(threadIdx.x) < span; j0 += kThreads * kUnroll) {
    float sc[kUnroll];
    int32_t id[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int jc = min(j0 + u * kThreads, span - 1);
      sc[u] = __ldg(srow + jc);
      if (kExplicit) id[u] = __ldg(irow + jc);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = j0 + u * kThreads;
      if (kExplicit)
        f(j < span && id[u] >= 0, sc[u], id[u]);
      else
        f(j < span, sc[u], base + j);
    }
  }
}

// Warp 0 of the block: the bucket of `hist` (nb <= 256 buckets) holding the
// need-th largest key counting from the top, the keys still needed inside it
// and whether the whole bucket is needed.  Lane l owns buckets
// nb - 1 - 8l .. nb - 8 - 8l (high to low).
__device__ __forceinline__ void find_bucket(const uint32_t* hist, int nb, int need, int& pick,
                                            int& need_in, bool& whole) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8], own = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int b = nb - 1 - 8 * lane - q;
    c[q] = b >= 0 ? hist[b] : 0u;
    own += c[q];
  }
  uint32_t inc = own;  // inclusive prefix over lanes 0..l (higher buckets first)
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += y;
  }
  const uint32_t before = inc - own;
  int p = -1, nd = 0, wh = 0;
  if (before < uint32_t(need) && inc >= uint32_t(need)) {
    uint32_t acc = before;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (p < 0 && acc + c[q] >= uint32_t(need)) {
        p = nb - 1 - 8 * lane - q;
        nd = need - int(acc);
        wh = (int(c[q]) == nd);
      }
      acc += c[q];
    }
  }
  const uint32_t m = __ballot_sync(0xffffffffu, p >= 0);
  if (m == 0) {  // fewer keys than needed (cannot happen for distinct keys): stop here
    pick = 0;
    need_in = need;
    whole = true;
    return;
  }
  const int src = __ffs(m) - 1;
  pick = __shfl_sync(0xffffffffu, p, src);
  need_in = __shfl_sync(0xffffffffu, nd, src);
  whole = __shfl_sync(0xffffffffu, wh, src) != 0;
}

// Bitonic sort (descending) of the kp = E * 1024 keys at `sel` (E >= 2):
// strides of 32 E or more compare across warps in shared memory; the smaller
// ones run in registers (thread t holds keys E t .. E t + E - 1) and warp
// shuffles, without block barriers, the keys staying in registers from one
// size to the next until a stride crosses warps.
template <int E>
__device__ void bitonic_sort_regs(uint64_t* sel, int kp) {
  const int tid = threadIdx.x;
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = sel[E * tid + e];
  for (int size = 2; size <= kp; size <<= 1) {
    int stride = size >> 1;
    if (stride >= 32 * E) {
      // the keys go through shared memory only around strides that cross
      // warps; runs of sizes up to 32 E stay in registers
#pragma unroll
      for (int e = 0; e < E; ++e) sel[E * tid + e] = v[e];
      __syncthreads();
      for (; stride >= 32 * E; stride >>= 1) {
        for (int p = tid; p < kp / 2; p += kThreads) {
          const int lo = 2 * p - (p & (stride - 1));
          const int hi = lo + stride;
          const bool desc = (lo & size) == 0;
          const uint64_t x = sel[lo], y = sel[hi];
          if ((x < y) == desc) {
            sel[lo] = y;
            sel[hi] = x;
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int e = 0; e < E; ++e) v[e] = sel[E * tid + e];
    }
    for (; stride >= E; stride >>= 1) {
      // partner in lane ^ (stride / E), same slot; with stride >= E the
      // direction (bit `size`) and the side (bit `stride`) of key E t + e
      // are those of E t, so one flag serves the thread's E keys: the lower
      // index keeps the larger key when descending
      const int lm = stride / E;
      const bool keep_max = ((E * tid) & stride) == 0 ? ((E * tid) & size) == 0
                                                       : ((E * tid) & size) != 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint64_t w = __shfl_xor_sync(0xffffffffu, v[e], lm);
        v[e] = ((v[e] > w) == keep_max) ? v[e] : w;
      }
    }
    // strides below E: both keys in this thread (compile-time indices)
#pragma unroll
    for (int st = E / 2; st > 0; st >>= 1) {
      if (st <= stride) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & st) == 0) {
            const int g = E * tid + e;
            const bool desc = (g & size) == 0;
            const uint64_t x = v[e], y = v[e + st];
            if ((x < y) == desc) {
              v[e] = y;
              v[e + st] = x;
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) sel[E * tid + e] = v[e];
  __syncthreads();
}

// Descending sort of the kp = E * 1024 keys at `sel` by runs and merges:
// each warp first sorts its 32 E keys in registers (the bitonic network
// above, every run's last merge descending), then log2(kp / (32 E)) levels
// merge pairs of runs between `tmp` and `sel`: thread t writes outputs
// E t .. E t + E - 1 of its pair, finding how many of the first come from
// each run by a binary search along the merge path (equal keys -- only the
// zero padding -- are taken from the second run first, in the search as in
// the merge).  One block barrier per level instead of one per cross-warp
// stride of the bitonic network.
template <int E>
__device__ void merge_sort_desc(uint64_t* sel, uint64_t* tmp, int kp) {
  const int tid = threadIdx.x;
  constexpr int kRun = 32 * E;
  uint64_t v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = sel[E * tid + e];
  for (int size = 2; size <= kRun; size <<= 1) {
    const bool last = size == kRun;  // the run's final merge: all descending
    int stride = size >> 1;
    for (; stride >= E; stride >>= 1) {
      const int lm = stride / E;
      const bool desc = last || ((E * tid) & size) == 0;
      const bool keep_max = ((E * tid) & stride) == 0 ? desc : !desc;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const uint64_t w = __shfl_xor_sync(0xffffffffu, v[e], lm);
        v[e] = ((v[e] > w) == keep_max) ? v[e] : w;
      }
    }
#pragma unroll
    for (int st = E / 2; st > 0; st >>= 1) {
      if (st <= stride) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & st) == 0) {
            const bool desc = last || ((E * tid + e) & size) == 0;
            const uint64_t x = v[e], y = v[e + st];
            if ((x < y) == desc) {
              v[e] = y;
              v[e + st] = x;
            }
          }
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) tmp[E * tid + e] = v[e];
  __syncthreads();
  uint64_t* src = tmp;
  uint64_t* dst = sel;
  for (int R = kRun; R < kp; R <<= 1) {
    const int k = E * tid;
    const int base = k & ~(2 * R - 1);
    const int k0 = k - base;  // this thread's first output within the pair
    const uint64_t* A = src + base;
    const uint64_t* B = A + R;
    int lo = max(0, k0 - R), hi = min(k0, R);
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (A[mid] > B[k0 - mid - 1])
        lo = mid + 1;
      else
        hi = mid;
    }
    int ia = lo, ib = k0 - lo;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const bool take_a = ib >= R || (ia < R && A[ia] > B[ib]);
      dst[k + e] = take_a ? A[ia++] : B[ib++];
    }
    __syncthreads();
    uint64_t* t = src;
    src = dst;
    dst = t;
  }
  if (src != sel) {  // an even number of levels: the result is in tmp
    for (int p = tid; p < kp; p += kThreads) sel[p] = src[p];
    __syncthreads();
  }
}

// The plain shared-memory network, for kp < 2048 and kp = 16384 (whose 16
// keys per thread would not fit the registers).
__device__ void bitonic_sort_smem(uint64_t* sel, int kp) {
  const int tid = threadIdx.x;
  for (int size = 2; size <= kp; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int p = tid; p < kp / 2; p += kThreads) {
        const int lo = 2 * p - (p & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t x = sel[lo], y = sel[hi];
        if ((x < y) == desc) {
          sel[lo] = y;
          sel[hi] = x;
        }
      }
      __syncthreads();
    }
  }
}

// kPair (select only): a cluster of two CTAs per row, each walking half of
// it.  Each reads the other's histogram through distributed shared memory
// and so finds the same boundary bin; CTA 1 queues its half's candidates at
// or above it into CTA 0's shared memory (regions kWarps..2 kWarps - 1) and
// leaves, and CTA 0 goes on alone over both halves' queues.  Both CTAs pass
// both cluster barriers on every path: no return comes before the second.
template <bool kExplicit, bool kVec4, bool kPair = false>
__global__ void __launch_bounds__(kThreads, 1) topk_kernel(TopkArgs a, int cap) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem);                  // bin counts
  uint32_t* cur = hist + kBins;                                        // bin cursors
  uint64_t* sel = reinterpret_cast<uint64_t*>(smem + 2 * kHistBytes);  // kp keys
  uint64_t* bnd = sel + a.kp;  // boundary bin: one region of `reg` keys per warp
  constexpr int kRegions = kPair ? 2 * kWarps : kWarps;  // boundary regions in CTA 0
  const int reg = cap / kRegions;
  __shared__ uint32_t warp_sum[kWarps];
  __shared__ int wcount[kRegions];
  __shared__ int wend[kRegions];  // boundary keys in regions 0..r (inclusive prefix)
  __shared__ int s_nsel, s_need, s_bin, s_done, s_flag, s_nb;
  __shared__ uint32_t warp_above[kWarps], s_total;  // keys in the warps above; all keys
  __shared__ uint64_t s_prefix, s_mask;
  const int64_t i = kPair ? int64_t(blockIdx.x >> 1) : int64_t(blockIdx.x);  // the row
  const uint32_t crank = kPair ? sm100::cluster_ctarank() : 0u;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  // this CTA's candidates: positions [base, base + span) of the row (select)
  // or its first `span` entries (merge)
  int first = 0, span, row_n = 0;
  if (kExplicit) {
    span = a.M;
    if (a.chunk > 0) {  // the chunks' results: K entries per chunk the row has
      const int nr = min(max(__ldg(a.n_cand + i), 0), a.L);
      span = min(a.M, int((int64_t(nr) + a.chunk - 1) / a.chunk) * K);
    }
  } else {
    span = min(max(__ldg(a.n_cand + i), 0), a.L);
    row_n = span;
    if (kPair) {
      // CTA 0 takes the first ceil(n / 8) quads, CTA 1 the rest (maybe none)
      const int half = int(((int64_t(row_n) + 7) >> 3) << 2);
      first = crank ? half : 0;
      span = crank ? max(row_n - half, 0) : min(row_n, half);
    } else if (a.chunk > 0) {
      first = int(blockIdx.y) * a.chunk;
      span = min(span - first, a.chunk);
      if (span <= 0) return;  // past the row's end: the merge reads no slab of it
    }
  }

  // 1) histogram of the keys' top 12 bits
  for (int b = tid; b < kBins; b += kThreads) hist[b] = 0;
  __syncthreads();
  for_each_candidate<kExplicit, kVec4>(a, i, first, span, [&](bool ok, float sc, int32_t) {
    if (ok) atomicAdd(&hist[score_key(sc) >> (32 - kBinBits)], 1u);
  });
  __syncthreads();
  // suffix sums over bins: thread t owns bins 4t .. 4t + 3
  static_assert(kBins == 4 * kThreads, "four bins per thread");
  uint32_t own[4], own_sum = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) own[q] = hist[4 * tid + q];
  if (kPair) {
    sm100::cluster_sync();  // #1: both halves counted
    const uint4 o = ld_dsmem_v4(sm100::map_to_cta(sm100::smem_u32(hist + 4 * tid), crank ^ 1u));
    own[0] += o.x;
    own[1] += o.y;
    own[2] += o.z;
    own[3] += o.w;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) own_sum += own[q];
  uint32_t suf = own_sum;  // inclusive suffix within the warp (lanes >= this one)
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_down_sync(0xffffffffu, suf, off);
    if (lane + off < 32) suf += y;
  }
  if (lane == 0) warp_sum[warp] = suf;  // the warp's total
  __syncthreads();
  if (warp == 0) {  // lane l: the keys of warps above warp l
    const uint32_t x = warp_sum[lane];
    uint32_t above = x;  // inclusive suffix over lanes >= l
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_down_sync(0xffffffffu, above, off);
      if (lane + off < 32) above += y;
    }
    warp_above[lane] = above - x;
    if (lane == 0) s_total = above;
  }
  __syncthreads();
  const uint32_t higher = warp_above[warp], total = s_total;
  const bool select = total > uint32_t(K);
  {
    // keys strictly above each of this thread's bins: each bin's first place
    // in the descending order (its cursor); the boundary bin holds the K-th
    uint32_t above = higher + suf - own_sum;
#pragma unroll
    for (int q = 3; q >= 0; --q) {
      cur[4 * tid + q] = above;
      if (select && above < uint32_t(K) && above + own[q] >= uint32_t(K)) {
        s_bin = 4 * tid + q;
        s_need = K - int(above);
      }
      above += own[q];
    }
  }
  __syncthreads();
  const int bin = select ? s_bin : -1;
  const int need = select ? s_need : 0;
  const int nabove = select ? K - need : int(total);  // keys above the boundary bin
  // 2) keys of higher bins -> their bin's places in `sel`; the boundary bin ->
  //    this warp's region of `bnd`.  The pass over the row only queues the
  //    candidates at or above the boundary bin in the warp's region (score
  //    key and position packed; most candidates lie below: one ballot skips
  //    them), and each warp then places its queue: a warp whose lanes mostly
  //    skip then pays nothing for the few that take.  When a queue outgrows
  //    its region (ties or a narrow score range), the row is read again and
  //    every key placed as it comes.
  //    A candidate is at or above the boundary bin when its score is at
  //    least the bin's lower edge (one float compare; its key is built only
  //    when taken): the edge is the score whose key starts the bin, -inf for
  //    bins below -inf's key (only -inf lies there), and bin 0 (NaN's) or no
  //    boundary takes every candidate.
  const uint32_t lt = (1u << lane) - 1u;
  const bool take_all = bin <= 0;
  const float edge = key_score(max(uint32_t(max(bin, 0)) << (32 - kBinBits), score_key(-INFINITY)));
  int wc = 0;  // this warp's queued candidates (warp-uniform)
  const bool remote = kPair && crank != 0;  // CTA 1 queues into CTA 0
  const int rw = remote ? kWarps + warp : warp;  // this warp's region
  const uint32_t region_addr = sm100::smem_u32(bnd + rw * reg);
  const uint32_t region_cta0 = remote ? sm100::map_to_cta(region_addr, 0) : 0u;
  for_each_candidate<kExplicit, kVec4>(a, i, first, span, [&](bool ok, float sc, int32_t x) {
    const bool take = ok && (take_all || sc >= edge);
    const uint32_t m = __ballot_sync(0xffffffffu, take);
    if (m == 0) return;
    if (take) {
      const int q = wc + __popc(m & lt);
      const uint64_t e = (uint64_t(score_key(sc)) << 32) | uint32_t(x);
      if (q < reg) {
        if (remote)
          st_dsmem_u64(region_cta0 + 8u * uint32_t(q), e);
        else
          bnd[rw * reg + q] = e;
      }
    }
    wc += __popc(m);
  });
  if (lane == 0) {
    if (remote)
      st_dsmem_u32(sm100::map_to_cta(sm100::smem_u32(wcount + rw), 0), uint32_t(wc));
    else
      wcount[rw] = wc;
  }
  if (kPair) {
    __syncwarp();
    sm100::cluster_sync();  // #2: CTA 1's queues and counts are in CTA 0
    if (crank != 0) return;  // CTA 1 is done; CTA 0 no longer reads its memory
    first = 0;  // any later pass over the row covers all of it
    span = row_n;
  }
  __syncthreads();
  constexpr int kPer = kRegions / 32;  // regions a lane of warp 0 reads
  if (warp == 0) {
    bool fit = true;
#pragma unroll
    for (int r = 0; r < kPer; ++r) fit &= wcount[kPer * lane + r] <= reg;
    fit = __all_sync(0xffffffffu, fit);
    if (lane == 0) s_flag = fit;
  }
  __syncthreads();  // warp 0 has read the counts
  const bool queued = s_flag != 0;
  if (queued) {
    // place the queues of this warp's regions (kPair: also CTA 1's warp's);
    // their boundary keys move to the front of the region (an entry is read
    // before any write reaches its slot)
    for (int rr = warp; rr < kRegions; rr += kWarps) {
      const int nq = wcount[rr];
      int nbk = 0;  // the region's boundary keys
      uint64_t* region = bnd + rr * reg;
      for (int q0 = 0; q0 < nq; q0 += 32) {
        const int q = q0 + lane;
        const uint64_t e = q < nq ? region[q] : 0;
        const uint32_t sk = uint32_t(e >> 32);
        const int32_t x = int32_t(uint32_t(e));
        const int kb = int(sk >> (32 - kBinBits));
        const bool hi = q < nq && kb > bin;
        const bool bd = q < nq && kb == bin;
        const uint64_t key = make_key(sk, kExplicit ? x : (q < nq ? global_id(a, x) : 0));
        if (hi) sel[atomicAdd(&cur[kb], 1u)] = key;
        const uint32_t m = __ballot_sync(0xffffffffu, bd);
        if (bd) region[nbk + __popc(m & lt)] = key;
        nbk += __popc(m);
      }
      __syncwarp();
      if (lane == 0) wcount[rr] = nbk;
    }
  } else {
    // the queues are dropped: regions kWarps.. (kPair) stay empty
    for (int rr = kWarps + warp; rr < kRegions; rr += kWarps)
      if (lane == 0) wcount[rr] = 0;
    wc = 0;  // this warp's boundary keys
    for_each_candidate<kExplicit, kVec4>(a, i, first, span, [&](bool ok, float sc, int32_t x) {
      const uint32_t sk = score_key(sc);
      const int kb = int(sk >> (32 - kBinBits));
      const bool take = ok && kb >= bin;
      if (__ballot_sync(0xffffffffu, take) == 0) return;
      const uint64_t key = make_key(sk, kExplicit ? x : (take ? global_id(a, x) : 0));
      if (take && kb > bin) sel[atomicAdd(&cur[kb], 1u)] = key;
      const uint32_t m = __ballot_sync(0xffffffffu, take && kb == bin);
      if (take && kb == bin) {
        const int q = wc + __popc(m & lt);
        if (q < reg) bnd[warp * reg + q] = key;
      }
      wc += __popc(m);
    });
    if (lane == 0) wcount[warp] = wc;
  }
  __syncthreads();
  if (warp == 0) {
    bool of = false;
    int sum = 0;
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int c = wcount[kPer * lane + r];
      of |= c > reg;
      sum += c;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    of = __any_sync(0xffffffffu, of);
    if (lane == 0) {
      s_flag = of;
      s_nb = sum;
    }
  }
  __syncthreads();
  const bool overflow = s_flag != 0;
  const int nb = s_nb;
  const int kept = min(int(total), K);
  int32_t* out_ids = a.out_ids + i * K;
  float* out_scores = a.out_scores ? a.out_scores + i * K : nullptr;
  auto emit = [&](int pos, uint64_t k) {
    out_ids[pos] = int32_t(0xFFFFFFFFu - uint32_t(k));
    if (out_scores) out_scores[pos] = key_score(uint32_t(k >> 32));
  };

  // 3) the `need` largest keys of the boundary bin by a radix select over
  //    its keys, gathered into one list (a pass over global memory replaces
  //    the list when the bin overflowed the warps' regions: ties far beyond
  //    K), then a sort of `sel`
  if (tid == 0) s_nsel = nabove;
  if (select) {
    const bool in_smem = !overflow;
    if (in_smem) {
      // compact the regions in place, 1024 keys at a time: a key's place in
      // the list is never past its slot, and keys are read before written;
      // a key's region is found by a binary search of the regions' prefix
      // sums (warp 0 scans them: lane l holds regions kPer l .. kPer l + kPer - 1)
      if (warp == 0) {
        int own = 0;
#pragma unroll
        for (int r = 0; r < kPer; ++r) own += wcount[kPer * lane + r];
        int inc = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, inc, off);
          if (lane >= off) inc += y;
        }
        int acc = inc - own;
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
          acc += wcount[kPer * lane + r];
          wend[kPer * lane + r] = acc;
        }
      }
      __syncthreads();
      for (int c0 = 0; c0 < nb; c0 += kThreads) {
        const int u = c0 + tid;
        uint64_t x = 0;
        if (u < nb) {
          int lo = 0, hi = kRegions - 1;  // the first region whose prefix passes u
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (wend[mid] > u)
              hi = mid;
            else
              lo = mid + 1;
          }
          x = bnd[lo * reg + (u - (wend[lo] - wcount[lo]))];
        }
        __syncthreads();
        if (u < nb) bnd[u] = x;
        __syncthreads();
      }
    }
    if (tid == 0) {
      s_prefix = uint64_t(bin) << kBinShift;
      s_mask = ~uint64_t(0) << kBinShift;
      s_need = need;
      s_done = (nb == need);  // the whole bin is in
    }
    __syncthreads();
    // radix steps over the bits below the bin, 8 at a time (4 last); the
    // keys are distinct, so the last step leaves one key per bucket (the
    // bound on `shift` only matters for duplicate merge input)
#pragma unroll 1
    for (int shift = kBinShift - 8; !s_done && shift > -8; shift -= 8) {
      const int sh = max(shift, 0);
      const int bits = shift >= 0 ? 8 : 8 + shift;
      const uint32_t nbk = 1u << bits;
      for (int b = tid; b < 256; b += kThreads) hist[b] = 0;
      __syncthreads();
      const uint64_t prefix = s_prefix, mask = s_mask;
      auto count = [&](uint64_t key) {
        if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (nbk - 1)], 1u);
      };
      if (in_smem) {
        for (int u = tid; u < nb; u += kThreads) count(bnd[u]);
      } else {
        for_each_candidate<kExplicit, false>(a, i, first, span, [&](bool ok, float sc, int32_t x) {
          const uint32_t sk = score_key(sc);
          if (ok && int(sk >> (32 - kBinBits)) == bin)
            count(make_key(sk, kExplicit ? x : global_id(a, x)));
        });
      }
      __syncthreads();
      if (warp == 0) {
        int pick, nd;
        bool whole;
        find_bucket(hist, int(nbk), s_need, pick, nd, whole);
        if (lane == 0) {
          s_prefix = prefix | (uint64_t(pick) << sh);
          s_mask = mask | (uint64_t(nbk - 1) << sh);
          s_need = nd;
          s_done = whole;  // the whole bucket is in
        }
      }
      __syncthreads();
    }
    // append the boundary bin's keys at or above the selected prefix
    // (exactly `need` of them: the keys are distinct)
    const uint64_t prefix = s_prefix, mask = s_mask;
    if (in_smem) {
      for (int u0 = 0; u0 < nb; u0 += kThreads) {
        const int u = u0 + tid;
        const uint64_t key = u < nb ? bnd[u] : 0;
        append(u < nb && (key & mask) >= prefix, key, sel, &s_nsel, a.kp);
      }
    } else {
      for_each_candidate<kExplicit, false>(a, i, first, span, [&](bool ok, float sc, int32_t x) {
        const uint32_t sk = score_key(sc);
        const bool inbin = ok && int(sk >> (32 - kBinBits)) == bin;
        const uint64_t key = make_key(sk, kExplicit ? x : (inbin ? global_id(a, x) : 0));
        append(inbin && (key & mask) >= prefix, key, sel, &s_nsel, a.kp);
      });
    }
  }
  __syncthreads();
  if (!kExplicit && a.chunk > 0) {
    // chunk mode: the chunk's kept keys, unsorted, then -1 padding
    const int64_t slab = (i * gridDim.y + blockIdx.y) * K;
    for (int p = tid; p < K; p += kThreads) {
      const uint64_t k = p < kept ? sel[p] : 0;
      a.chunk_ids[slab + p] = p < kept ? int32_t(0xFFFFFFFFu - uint32_t(k)) : -1;
      a.chunk_scores[slab + p] = p < kept ? key_score(uint32_t(k >> 32)) : 0.f;
    }
    return;
  }
  for (int p = kept + tid; p < a.kp; p += kThreads) sel[p] = 0;  // below every candidate
  __syncthreads();
  // the histogram and cursors are free again: the merge sort's second buffer
  static_assert(2 * kHistBytes >= 4096 * 8, "the merge buffer holds 4096 keys");
  switch (a.kp) {
    case 2048: merge_sort_desc<2>(sel, reinterpret_cast<uint64_t*>(smem), a.kp); break;
    case 4096: merge_sort_desc<4>(sel, reinterpret_cast<uint64_t*>(smem), a.kp); break;
    case 8192: bitonic_sort_regs<8>(sel, a.kp); break;
    default: bitonic_sort_smem(sel, a.kp); break;
  }
  for (int p = tid; p < K; p += kThreads) {
    if (p < kept) {
      emit(p, sel[p]);
    } else {
      out_ids[p] = -1;
      if (out_scores) out_scores[p] = 0.f;
    }
  }
}

int pow2_at_least(int x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}

// The kernel's shared-memory opt-in, set once per device and kernel form.
constexpr int kMaxDevices = 64;
template <bool kExplicit, bool kVec4, bool kPair>
cudaError_t ensure_smem_attribute() {
  static std::atomic<bool> done[kMaxDevices];
  static std::mutex m;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  if (tracked && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(m);
  if (tracked && done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = cudaFuncSetAttribute(topk_kernel<kExplicit, kVec4, kPair>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess && tracked) done[dev].store(true, std::memory_order_release);
  return e;
}

template <bool kExplicit, bool kVec4>
cudaError_t launch(TopkArgs a, int cap, cudaStream_t s, int chunks = 1) {
  cudaError_t e = ensure_smem_attribute<kExplicit, kVec4, false>();
  if (e != cudaSuccess) return e;
  topk_kernel<kExplicit, kVec4>
      <<<dim3(unsigned(a.T), unsigned(chunks)), dim3(kThreads), kSmemBytes, s>>>(a, cap);
  return cudaGetLastError();
}

// The select with a cluster of two CTAs per row.
cudaError_t launch_pair(TopkArgs a, int cap, cudaStream_t s) {
  cudaError_t e = ensure_smem_attribute<false, true, true>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * unsigned(a.T));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel<false, true, true>, a, cap);
}

// Shared memory: the histogram and the bin cursors, the selection (kp keys),
// the boundary bin's regions (kPair: twice as many, half the size).
int boundary_cap(const TopkArgs& a) { return (kSmemBytes - 2 * kHistBytes) / 8 - a.kp; }

// Few long rows leave most SMs idle with one CTA (or one pair) per row.
// When there are at most kChunkRows rows and L is at least 2 kMaxChunks
// chunks of the smallest size (kChunkMin candidates, and kChunkPerK times
// the sort size), each row is cut into count = SMs / T chunks (2 to
// kMaxChunks): one CTA walks each chunk and keeps its K best, and a second
// launch selects and sorts the row's K best among those count K.  Each CTA
// costs about 10 us beyond its per-candidate work (the scan, the radix
// select; the merge adds a sort), so shorter rows, or more rows, are faster
// walked by a pair of CTAs each.
constexpr int kChunkMin = 16384;
constexpr int kChunkPerK = 8;
constexpr int kMaxChunks = 8;
constexpr int kChunkRows = 32;
// Rows of at least kPairMin candidates get two CTAs each (a cluster) when
// 2 T CTAs fit on the GPU at once.
constexpr int kPairMin = 16384;

bool chunkable(int32_t T, int32_t L, int32_t K) {
  const int64_t smallest = std::max<int64_t>(kChunkMin, int64_t(kChunkPerK) * pow2_at_least(K));
  return T >= 1 && T <= kChunkRows && int64_t(L) >= 2 * kMaxChunks * smallest;
}

// SMs of the current device, queried once per device.
cudaError_t sm_count(int* sms) {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  int v = tracked ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (v == 0) {
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (tracked) cached[dev].store(v, std::memory_order_relaxed);
  }
  *sms = v;
  return cudaSuccess;
}

}  // namespace

size_t topk_workspace_bytes(int32_t T, int32_t L, int32_t K) {
  if (!chunkable(T, L, K) || K <= 0) return 0;
  return size_t(T) * kMaxChunks * size_t(K) * (sizeof(int32_t) + sizeof(float));
}

cudaError_t launch_topk_select(const TopkArgs& args, void* workspace, cudaStream_t s) {
  TopkArgs a = args;
  a.div_I = make_fastdiv(uint32_t(a.interleave));
  a.kp = pow2_at_least(a.K);
  a.chunk = 0;
  int count = 1;
  if (workspace != nullptr && chunkable(a.T, a.L, a.K)) {
    int sms = 0;
    const cudaError_t e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    count = std::min(kMaxChunks, sms / a.T);
  }
  if (count < 2) {
    // 16-byte score loads over each row's aligned middle, whatever the stride
    if (a.L >= kPairMin) {
      int sms = 0;
      const cudaError_t e = sm_count(&sms);
      if (e != cudaSuccess) return e;
      if (2 * int64_t(a.T) <= sms) return launch_pair(a, boundary_cap(a), s);
    }
    return launch<false, true>(a, boundary_cap(a), s);
  }
  // whole quads a chunk: each chunk starts at the row's alignment
  const int64_t chunk = ((int64_t(a.L) + count - 1) / count + 3) & ~int64_t(3);
  const int64_t slabs = int64_t(a.T) * count * a.K;
  a.chunk = int32_t(chunk);
  a.chunk_scores = static_cast<float*>(workspace);
  a.chunk_ids = reinterpret_cast<int32_t*>(a.chunk_scores + slabs);
  cudaError_t e = launch<false, true>(a, boundary_cap(a), s, count);
  if (e != cudaSuccess) return e;
  TopkArgs m{};
  m.scores = a.chunk_scores;
  m.cand_ids = a.chunk_ids;
  m.n_cand = a.n_cand;
  m.row_stride = int64_t(count) * a.K;
  m.L = a.L;
  m.M = count * a.K;
  m.T = a.T;
  m.K = a.K;
  m.kp = a.kp;
  m.D = 1;
  m.interleave = 1;
  m.out_ids = a.out_ids;
  m.out_scores = a.out_scores;
  m.chunk = a.chunk;
  return launch<true, false>(m, boundary_cap(m), s);
}

cudaError_t launch_topk_merge(const TopkArgs& args, cudaStream_t s) {
  TopkArgs a = args;
  a.kp = pow2_at_least(a.K);
  a.chunk = 0;
  return launch<true, false>(a, boundary_cap(a), s);
}

}  // namespace smla
