// LSE-weighted merge of D partial (out, lse) results.
//
// "[eldritch] attention: support DCP in SM120 FlashInfer sparse MLA", Why:
// each DCP rank returns its partial attention with the softmax LSE and the
// common MLA layer merges them.  "FlashMLA sparse fp8 path + DCP + MTP",
// executive summary 1: (0, -inf) is the identity of that merge, so a rank
// with no candidate drops out without producing NaN.
//
// Per (token, head) row with M = max_d lse_d:
//   M = -inf -> out = 0, lse = -inf
//   else        lse = M + log(sum_d exp(lse_d - M)),
//               out = sum_d exp(lse_d - lse) * out_d    (fp32, bf16 RNE out)
//
// Memory-bound: one warp per row, each lane moves 2 x 16 bytes of every
// partial (bf16 x 8 per load), so every load is a full 512-byte warp
// transaction.  Every load of a row -- its D LSEs and all D partial rows --
// is issued before any of them is used, so a row costs one memory round
// trip; the kernel is instantiated per bound on D so the partials in flight
// fit in registers.
#include <cuda_bf16.h>

#include "../../include/smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    f[2 * k] = __uint_as_float(w[k] << 16);
    f[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float* f) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    __nv_bfloat162 p = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
    w[k] = *reinterpret_cast<uint32_t*>(&p);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

template <int kDMax>
__global__ void __launch_bounds__(kWarps * 32) merge_kernel(MergeArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t rows = int64_t(a.T) * a.H;
  if (row >= rows) return;

  // every load of the row first
  float l[kDMax];
  uint4 p0[kDMax], p1[kDMax];
#pragma unroll
  for (int d = 0; d < kDMax; ++d) {
    if (d < a.D) {
      l[d] = __ldg(a.lses[d] + row);
      const uint4* src = reinterpret_cast<const uint4*>(a.outs[d] + row * SMLA_V_DIM);
      p0[d] = ldg_stream(src + lane);
      p1[d] = ldg_stream(src + lane + 32);
    } else {
      l[d] = -INFINITY;
      p0[d] = p1[d] = make_uint4(0, 0, 0, 0);
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int d = 0; d < kDMax; ++d) M = fmaxf(M, l[d]);
  uint4* dst = reinterpret_cast<uint4*>(a.out + row * SMLA_V_DIM);
  if (M == -INFINITY) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    dst[lane] = z;
    dst[lane + 32] = z;
    if (lane == 0) a.lse[row] = -INFINITY;
    return;
  }
  float total = 0.f;
#pragma unroll
  for (int d = 0; d < kDMax; ++d) {
    l[d] = (d < a.D) ? expf(l[d] - M) : 0.f;  // weight before normalisation
    total += l[d];
  }
  const float inv = 1.f / total;
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
#pragma unroll
  for (int d = 0; d < kDMax; ++d) {
    const float w = l[d] * inv;
    float f[8];
    bf16x8_to_f32(p0[d], f);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = fmaf(w, f[k], acc[k]);
    bf16x8_to_f32(p1[d], f);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[8 + k] = fmaf(w, f[k], acc[8 + k]);
  }
  dst[lane] = f32x8_to_bf16(acc);
  dst[lane + 32] = f32x8_to_bf16(acc + 8);
  if (lane == 0) a.lse[row] = M + logf(total);
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t s) {
  const int64_t rows = int64_t(a.T) * a.H;
  const dim3 grid(unsigned((rows + kWarps - 1) / kWarps)), block(kWarps * 32);
  if (a.D <= 2)
    merge_kernel<2><<<grid, block, 0, s>>>(a);
  else if (a.D <= 4)
    merge_kernel<4><<<grid, block, 0, s>>>(a);
  else if (a.D <= 8)
    merge_kernel<8><<<grid, block, 0, s>>>(a);
  else
    merge_kernel<kMaxMerge><<<grid, block, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace smla
