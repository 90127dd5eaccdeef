// Sparse MLA decode, first CUDA-core version: semantics and layouts
// end to end, fp32 arithmetic, no tensor cores.
//
// "FlashMLA sparse fp8 path + DCP + MTP", implementation breakdown steps 1
// and 3: attention of each (token, head) over its valid local slots of the
// packed fp8_ds_mla cache, returning out and the natural-log softmax LSE;
// a row with no valid slot is written as (0, -inf).
//
// One CTA per (token, 16-head group).  The CTA scans its row's slots 256 at
// a time, compacts the valid ones, dequantises 16 keys at a time into
// shared memory and runs an online softmax per head.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "../../include/smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

__device__ unsigned int g_decode_error;

constexpr int kHB = 16;        // heads per CTA
constexpr int kKC = 16;        // keys per dequantised chunk
constexpr int kThreads = 256;  // = kHB * kKC
constexpr int kScan = 256;     // slots scanned per step
constexpr int kKPitch = SMLA_QK_DIM + 4;

constexpr size_t kSmemBytes =
    sizeof(float) * (kHB * SMLA_QK_DIM + kKC * kKPitch + kHB * kKC + 3 * kHB) +
    sizeof(int) * kScan;

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(uint32_t(b) << 16);
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(code, __NV_E4M3);
  return __half2float(__half(h));
}

__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeArgs a) {
  extern __shared__ float smem[];
  float* q_s = smem;                       // [kHB][576]
  float* k_s = q_s + kHB * SMLA_QK_DIM;    // [kKC][kKPitch]
  float* p_s = k_s + kKC * kKPitch;        // [kHB][kKC]
  float* m_s = p_s + kHB * kKC;            // running max per head
  float* l_s = m_s + kHB;                  // running sum per head
  float* alpha_s = l_s + kHB;              // rescale of the step
  int* list = reinterpret_cast<int*>(alpha_s + kHB);
  __shared__ int n_list;

  const int tid = threadIdx.x;
  const int64_t t = blockIdx.x;
  const int h0 = blockIdx.y * kHB;

  for (int idx = tid; idx < kHB * SMLA_QK_DIM; idx += kThreads) {
    const int h = idx / SMLA_QK_DIM, c = idx % SMLA_QK_DIM;
    q_s[idx] = (h0 + h < a.H)
                   ? bf16_bits_to_f32(a.q[(t * a.H + h0 + h) * SMLA_QK_DIM + c])
                   : 0.f;
  }
  if (tid < kHB) {
    m_s[tid] = -INFINITY;
    l_s[tid] = 0.f;
  }
  float acc[kHB][2];
#pragma unroll
  for (int h = 0; h < kHB; ++h) acc[h][0] = acc[h][1] = 0.f;

  const int32_t* srow = a.slots + t * a.K;
  for (int base = 0; base < a.K; base += kScan) {
    __syncthreads();
    if (tid == 0) n_list = 0;
    __syncthreads();
    const int j = base + tid;
    if (j < a.K) {
      const int32_t s = srow[j];
      if (s >= 0) {
        if (s >= a.num_slots) {
          atomicOr(&g_decode_error, SMLA_DEVERR_SLOT_RANGE);
        } else {
          list[atomicAdd(&n_list, 1)] = s;
        }
      }
    }
    __syncthreads();
    const int n = n_list;
    for (int c0 = 0; c0 < n; c0 += kKC) {
      const int nk = min(kKC, n - c0);
      for (int idx = tid; idx < kKC * SMLA_QK_DIM; idx += kThreads) {
        const int kk = idx / SMLA_QK_DIM, c = idx % SMLA_QK_DIM;
        float v = 0.f;
        if (kk < nk) {
          const uint8_t* row = a.kv + int64_t(list[c0 + kk]) * SMLA_ROW_BYTES;
          if (c < SMLA_V_DIM) {
            const float scale = reinterpret_cast<const float*>(row + 512)[c >> 7];
            v = e4m3_to_f32(row[c]) * scale;
          } else {
            v = bf16_bits_to_f32(reinterpret_cast<const uint16_t*>(row + 528)[c - 512]);
          }
        }
        k_s[kk * kKPitch + c] = v;
      }
      __syncthreads();
      {
        const int h = tid / kKC, kk = tid % kKC;
        float s = -INFINITY;
        if (kk < nk) {
          float dot = 0.f;
          for (int c = 0; c < SMLA_QK_DIM; ++c)
            dot = fmaf(q_s[h * SMLA_QK_DIM + c], k_s[kk * kKPitch + c], dot);
          s = dot * a.sm_scale;
        }
        p_s[h * kKC + kk] = s;
      }
      __syncthreads();
      if (tid < kHB) {
        const float m_old = m_s[tid];
        float mx = m_old;
        for (int kk = 0; kk < nk; ++kk) mx = fmaxf(mx, p_s[tid * kKC + kk]);
        const float alpha = expf(m_old - mx);  // 0 on the first chunk
        float sum = 0.f;
        for (int kk = 0; kk < kKC; ++kk) {
          const float p = (kk < nk) ? expf(p_s[tid * kKC + kk] - mx) : 0.f;
          p_s[tid * kKC + kk] = p;
          sum += p;
        }
        l_s[tid] = l_s[tid] * alpha + sum;
        m_s[tid] = mx;
        alpha_s[tid] = alpha;
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < kHB; ++h) {
        const float al = alpha_s[h];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int dv = tid + e * kThreads;
          float o = acc[h][e] * al;
          for (int kk = 0; kk < nk; ++kk)
            o = fmaf(p_s[h * kKC + kk], k_s[kk * kKPitch + dv], o);
          acc[h][e] = o;
        }
      }
      __syncthreads();
    }
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < kHB; ++h) {
    if (h0 + h >= a.H) break;
    const float l = l_s[h];
    const bool empty = !(l > 0.f) && !(l != l);  // no valid key (NaN stays NaN)
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(a.out) +
                       (t * a.H + h0 + h) * SMLA_V_DIM;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int dv = tid + e * kThreads;
      o[dv] = __float2bfloat16_rn(empty ? 0.f : acc[h][e] / l);
    }
    if (tid == 0) a.lse[t * a.H + h0 + h] = empty ? -INFINITY : m_s[h] + logf(l);
  }
}

}  // namespace

size_t decode_workspace_bytes(int32_t, int32_t, int32_t) { return 0; }

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(
        decode_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(a.T, (a.H + kHB - 1) / kHB);
  decode_simt_kernel<<<grid, kThreads, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

cudaError_t decode_error_word(uint32_t* flags, bool clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(v));
  if (e != cudaSuccess) return e;
  *flags |= v;
  if (clear) {
    v = 0;
    e = cudaMemcpyToSymbol(g_decode_error, &v, sizeof(v));
  }
  return e;
}

}  // namespace smla
