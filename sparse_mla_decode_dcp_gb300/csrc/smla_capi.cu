// C ABI of the library: host-side argument checks, then one launch per call
// (the host-buffer form of the fused step: its copies and a launch per row
// group).  Every check runs before anything touches the GPU, so a rejected
// call has no side effect and needs no device.
#include <cmath>
#include <cstdint>

#include "../../include/smla.h"
#include "smla_internal.h"

namespace {

inline bool misaligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) != 0;
}

inline smla_status from_cuda(cudaError_t e) {
  return e == cudaSuccess ? SMLA_OK : SMLA_ERR_CUDA;
}

}  // namespace

static_assert(SMLA_NOALLOC_SCRATCH_BYTES == smla::kNoAllocScratchBytes,
              "header and library agree on the scratch size");

extern "C" {

const char* smla_status_string(smla_status status) {
  switch (status) {
    case SMLA_OK: return "SMLA_OK";
    case SMLA_ERR_INVALID_ARG: return "SMLA_ERR_INVALID_ARG";
    case SMLA_ERR_UNSUPPORTED: return "SMLA_ERR_UNSUPPORTED";
    case SMLA_ERR_WORKSPACE: return "SMLA_ERR_WORKSPACE";
    case SMLA_ERR_CUDA: return "SMLA_ERR_CUDA";
    default: return "SMLA_UNKNOWN_STATUS";
  }
}

smla_status smla_get_device_error(uint32_t* flags, int clear) {
  if (flags == nullptr) return SMLA_ERR_INVALID_ARG;
  *flags = 0;
  cudaError_t e = smla::index_error_word(flags, clear != 0);
  if (e == cudaSuccess) e = smla::decode_error_word(flags, clear != 0);
  return from_cuda(e);
}

smla_status smla_dcp_filter_convert_index(
    const int32_t* req_id_per_token, const int32_t* block_table,
    int64_t bt_row_stride, int32_t bt_width, int32_t num_reqs,
    const int32_t* topk_global, int32_t T, int32_t K, int32_t D, int32_t rank,
    int32_t block_size, int32_t interleave, int32_t* local_slots, int32_t* valid_count,
    void* stream) {
  if (T < 0 || K < 1 || D < 1 || rank < 0 || rank >= D || block_size < 1 ||
      interleave < 1 || num_reqs < 1 || bt_width < 1 || bt_row_stride < bt_width)
    return SMLA_ERR_INVALID_ARG;
  if (T == 0) return SMLA_OK;
  if (!req_id_per_token || !block_table || !topk_global || !local_slots)
    return SMLA_ERR_INVALID_ARG;
  if (misaligned(req_id_per_token, 4) || misaligned(block_table, 4) ||
      misaligned(topk_global, 4) || misaligned(local_slots, 4) ||
      (valid_count && misaligned(valid_count, 4)))
    return SMLA_ERR_INVALID_ARG;
  smla::IndexArgs a;
  a.req_id = req_id_per_token;
  a.block_table = block_table;
  a.bt_row_stride = bt_row_stride;
  a.bt_width = bt_width;
  a.num_reqs = num_reqs;
  a.topk = topk_global;
  a.T = T;
  a.K = K;
  a.D = D;
  a.rank = rank;
  a.block_size = block_size;
  a.interleave = interleave;
  a.local_slots = local_slots;
  a.valid_count = valid_count;
  return from_cuda(smla::launch_filter_convert(a, static_cast<cudaStream_t>(stream)));
}

size_t smla_decode_workspace_size(int32_t T, int32_t H, int32_t K) {
  if (T < 0 || H < 1 || H > SMLA_MAX_HEADS || K < 1) return 0;
  return smla::decode_workspace_bytes(T, H, K);
}

smla_status smla_sparse_mla_decode(
    const uint16_t* q, const uint8_t* kv_cache, int64_t num_slots,
    const int32_t* local_slots, int32_t T, int32_t H, int32_t K,
    float sm_scale, uint16_t* out, float* lse, void* workspace,
    size_t workspace_bytes, void* stream) {
  if (T < 0 || K < 1 || H < 1 || num_slots < 0 || !std::isfinite(sm_scale) ||
      !(sm_scale > 0.f))
    return SMLA_ERR_INVALID_ARG;
  if (H > SMLA_MAX_HEADS) return SMLA_ERR_UNSUPPORTED;
  if (T == 0) return SMLA_OK;
  if (!q || !kv_cache || !local_slots || !out || !lse) return SMLA_ERR_INVALID_ARG;
  if (misaligned(q, 16) || misaligned(kv_cache, 16) || misaligned(out, 16) ||
      misaligned(local_slots, 4) || misaligned(lse, 4))
    return SMLA_ERR_INVALID_ARG;
  const size_t need = smla::decode_workspace_bytes(T, H, K);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                   misaligned(workspace, 256)))
    return SMLA_ERR_WORKSPACE;
  smla::DecodeArgs a{};
  a.q = q;
  a.kv = kv_cache;
  a.num_slots = num_slots;
  a.slots = local_slots;
  a.T = T;
  a.H = H;
  a.K = K;
  a.sm_scale = sm_scale;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return from_cuda(smla::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

smla_status smla_sparse_mla_decode_noalloc(
    const uint16_t* q, const uint8_t* kv_cache, int64_t num_slots,
    const int32_t* local_slots, int32_t T, int32_t H, int32_t K,
    float sm_scale, uint16_t* out, float* lse, void* stream) {
  if (T < 0 || K < 1 || H < 1 || num_slots < 0 || !std::isfinite(sm_scale) ||
      !(sm_scale > 0.f))
    return SMLA_ERR_INVALID_ARG;
  if (H > SMLA_MAX_HEADS) return SMLA_ERR_UNSUPPORTED;
  if (T == 0) return SMLA_OK;
  if (!q || !kv_cache || !local_slots || !out || !lse) return SMLA_ERR_INVALID_ARG;
  if (misaligned(q, 16) || misaligned(kv_cache, 16) || misaligned(out, 16) ||
      misaligned(local_slots, 4) || misaligned(lse, 4))
    return SMLA_ERR_INVALID_ARG;
  if (smla::decode_workspace_bytes(T, H, K) > SMLA_NOALLOC_SCRATCH_BYTES)
    return SMLA_ERR_WORKSPACE;
  smla::DecodeArgs a{};
  a.q = q;
  a.kv = kv_cache;
  a.num_slots = num_slots;
  a.slots = local_slots;
  a.T = T;
  a.H = H;
  a.K = K;
  a.sm_scale = sm_scale;
  a.out = out;
  a.lse = lse;
  return from_cuda(smla::launch_decode_noalloc(a, static_cast<cudaStream_t>(stream)));
}

// Checks of the fused step's arguments shared by its device and host forms;
// fills `a` with everything but the staging of q and the top-k ids.
static smla_status fused_args(
    const void* q, int32_t T, int32_t H, int32_t K, float sm_scale,
    const int32_t* req_id_per_token, const void* topk_global, int32_t num_reqs, int32_t D,
    int32_t block_size, int32_t interleave, const uint8_t* const* kv_caches,
    const int64_t* num_slots, const int32_t* const* block_tables,
    const int64_t* bt_row_strides, const int32_t* bt_widths, const void* out, const void* lse,
    smla::DecodeArgs& a) {
  if (T < 0 || K < 1 || H < 1 || D < 1 || block_size < 1 || interleave < 1 || num_reqs < 1 ||
      !std::isfinite(sm_scale) || !(sm_scale > 0.f))
    return SMLA_ERR_INVALID_ARG;
  if (H > SMLA_MAX_HEADS || D > SMLA_MAX_DCP) return SMLA_ERR_UNSUPPORTED;
  if (T == 0) return SMLA_OK;
  if (!q || !req_id_per_token || !topk_global || !out || !lse || !kv_caches ||
      !num_slots || !block_tables || !bt_row_strides || !bt_widths)
    return SMLA_ERR_INVALID_ARG;
  if (misaligned(q, 16) || misaligned(out, 16) || misaligned(lse, 4) ||
      misaligned(req_id_per_token, 4) || misaligned(topk_global, 4))
    return SMLA_ERR_INVALID_ARG;
  a = smla::DecodeArgs{};
  for (int d = 0; d < D; ++d) {
    if (!kv_caches[d] || misaligned(kv_caches[d], 16) || num_slots[d] < 0 ||
        !block_tables[d] || misaligned(block_tables[d], 4) || bt_widths[d] < 1 ||
        bt_row_strides[d] < bt_widths[d])
      return SMLA_ERR_INVALID_ARG;
    a.pools[d] = kv_caches[d];
    a.pool_slots[d] = num_slots[d];
    a.bts[d] = block_tables[d];
    a.bt_stride[d] = bt_row_strides[d];
    a.bt_width[d] = bt_widths[d];
  }
  a.T = T;
  a.H = H;
  a.K = K;
  a.sm_scale = sm_scale;
  a.D = D;
  a.block_size = block_size;
  a.interleave = interleave;
  a.num_reqs = num_reqs;
  a.req_id = req_id_per_token;
  return SMLA_OK;
}

smla_status smla_dcp_sparse_mla_decode_fused(
    const uint16_t* q, int32_t T, int32_t H, int32_t K, float sm_scale,
    const int32_t* req_id_per_token, const int32_t* topk_global, int32_t num_reqs,
    int32_t D, int32_t block_size, int32_t interleave, const uint8_t* const* kv_caches,
    const int64_t* num_slots, const int32_t* const* block_tables,
    const int64_t* bt_row_strides, const int32_t* bt_widths, uint16_t* out,
    float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  smla::DecodeArgs a;
  const smla_status st =
      fused_args(q, T, H, K, sm_scale, req_id_per_token, topk_global, num_reqs, D, block_size,
                 interleave, kv_caches, num_slots, block_tables, bt_row_strides, bt_widths, out,
                 lse, a);
  if (st != SMLA_OK || T == 0) return st;
  const size_t need = smla::decode_workspace_bytes(T, H, K);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                   misaligned(workspace, 256)))
    return SMLA_ERR_WORKSPACE;
  a.q = q;
  a.topk = topk_global;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  return from_cuda(smla::launch_decode_fused(a, static_cast<cudaStream_t>(stream)));
}

smla_status smla_dcp_sparse_mla_decode_fused_host(
    const uint16_t* q_host, const int32_t* topk_host, uint16_t* out_host, float* lse_host,
    uint16_t* q_dev, int32_t* topk_dev, uint16_t* out_dev, float* lse_dev,
    int32_t T, int32_t H, int32_t K, float sm_scale, const int32_t* req_id_per_token,
    int32_t num_reqs, int32_t D, int32_t block_size, int32_t interleave,
    const uint8_t* const* kv_caches, const int64_t* num_slots,
    const int32_t* const* block_tables, const int64_t* bt_row_strides,
    const int32_t* bt_widths, void* workspace, size_t workspace_bytes, int32_t chunks,
    void* stream) {
  smla::DecodeArgs a;
  smla_status st =
      fused_args(q_dev, T, H, K, sm_scale, req_id_per_token, topk_dev, num_reqs, D, block_size,
                 interleave, kv_caches, num_slots, block_tables, bt_row_strides, bt_widths,
                 out_dev, lse_dev, a);
  if (st != SMLA_OK) return st;
  if (chunks < 1 || chunks > SMLA_MAX_HOST_CHUNKS) return SMLA_ERR_INVALID_ARG;
  if (T == 0) return SMLA_OK;
  if (!q_host || !topk_host || !out_host || !lse_host) return SMLA_ERR_INVALID_ARG;
  const int groups = chunks < T ? chunks : T;
  if (groups > 1 && K > smla::kDecodeMaxList) return SMLA_ERR_UNSUPPORTED;
  if (groups == 1) {
    const size_t need = smla::decode_workspace_bytes(T, H, K);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                     misaligned(workspace, 256)))
      return SMLA_ERR_WORKSPACE;
    a.workspace = workspace;
    a.workspace_bytes = workspace_bytes;
  }
  a.q = q_dev;
  a.topk = topk_dev;
  a.out = out_dev;
  a.lse = lse_dev;
  smla::HostBuffers h{q_host, topk_host, out_host, lse_host, q_dev, topk_dev};
  return from_cuda(smla::launch_fused_host(a, h, groups, static_cast<cudaStream_t>(stream)));
}

// Raw entries per row of the dense decode: positions 0..max_ctx-1, or the
// largest count of them one rank holds.
static int32_t dense_entries(int32_t max_ctx, int32_t D, int32_t interleave, int32_t rank) {
  if (rank < 0) return max_ctx;
  const int64_t id = int64_t(interleave) * D;
  return int32_t(((int64_t(max_ctx) + id - 1) / id) * interleave);
}

size_t smla_dense_decode_workspace_size(int32_t T, int32_t H, int32_t max_ctx, int32_t D,
                                        int32_t interleave, int32_t rank) {
  if (T < 0 || H < 1 || H > SMLA_MAX_HEADS || max_ctx < 1 || D < 1 || interleave < 1 ||
      rank < -1 || rank >= D)
    return 0;
  return smla::decode_workspace_bytes(T, H, dense_entries(max_ctx, D, interleave, rank));
}

smla_status smla_dcp_dense_mla_decode(
    const uint16_t* q, int32_t B, int32_t S, int32_t H, float sm_scale,
    const int32_t* ctx_lens, int32_t max_ctx, int32_t D, int32_t rank,
    int32_t block_size, int32_t interleave, const uint8_t* const* kv_caches,
    const int64_t* num_slots, const int32_t* const* block_tables,
    const int64_t* bt_row_strides, const int32_t* bt_widths, uint16_t* out,
    float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || S < 1 || H < 1 || max_ctx < 1 || D < 1 || rank < -1 || rank >= D ||
      block_size < 1 || interleave < 1 || !std::isfinite(sm_scale) || !(sm_scale > 0.f))
    return SMLA_ERR_INVALID_ARG;
  if (H > SMLA_MAX_HEADS || D > SMLA_MAX_DCP) return SMLA_ERR_UNSUPPORTED;
  if (int64_t(B) * S > INT32_MAX) return SMLA_ERR_INVALID_ARG;
  const int32_t T = B * S;
  if (T == 0) return SMLA_OK;
  if (!q || !ctx_lens || !out || !lse || !kv_caches || !num_slots || !block_tables ||
      !bt_row_strides || !bt_widths)
    return SMLA_ERR_INVALID_ARG;
  if (misaligned(q, 16) || misaligned(out, 16) || misaligned(lse, 4) || misaligned(ctx_lens, 4))
    return SMLA_ERR_INVALID_ARG;
  smla::DecodeArgs a{};
  for (int d = 0; d < D; ++d) {
    const bool used = rank < 0 || d == rank;
    if (used && (!kv_caches[d] || misaligned(kv_caches[d], 16) || num_slots[d] < 0 ||
                 !block_tables[d] || misaligned(block_tables[d], 4) || bt_widths[d] < 1 ||
                 bt_row_strides[d] < bt_widths[d]))
      return SMLA_ERR_INVALID_ARG;
    a.pools[d] = used ? kv_caches[d] : nullptr;
    a.pool_slots[d] = used ? num_slots[d] : 0;
    a.bts[d] = used ? block_tables[d] : nullptr;
    a.bt_stride[d] = used ? bt_row_strides[d] : 0;
    a.bt_width[d] = used ? bt_widths[d] : 0;
  }
  const int32_t K = dense_entries(max_ctx, D, interleave, rank);
  const size_t need = smla::decode_workspace_bytes(T, H, K);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                   misaligned(workspace, 256)))
    return SMLA_ERR_WORKSPACE;
  a.q = q;
  a.T = T;
  a.H = H;
  a.K = K;
  a.sm_scale = sm_scale;
  a.out = out;
  a.lse = lse;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.D = D;
  a.block_size = block_size;
  a.interleave = interleave;
  a.num_reqs = B;
  a.ctx_lens = ctx_lens;
  a.S = S;
  a.dense_rank = rank;
  a.max_ctx = max_ctx;
  return from_cuda(smla::launch_decode_dense(a, static_cast<cudaStream_t>(stream)));
}

size_t smla_topk_select_workspace_size(int32_t T, int32_t L, int32_t K) {
  if (T < 0 || L < 0 || K < 1 || K > SMLA_MAX_TOPK) return 0;
  return smla::topk_workspace_bytes(T, L, K);
}

smla_status smla_topk_select(const float* scores, int64_t row_stride, int32_t L,
                             const int32_t* n_cand, int32_t T, int32_t K, int32_t D,
                             int32_t rank, int32_t interleave, int32_t* out_ids,
                             float* out_scores, void* workspace, size_t workspace_bytes,
                             void* stream) {
  if (T < 0 || L < 0 || row_stride < L || D < 1 || rank < 0 || rank >= D || interleave < 1)
    return SMLA_ERR_INVALID_ARG;
  if (K < 1 || K > SMLA_MAX_TOPK) return SMLA_ERR_UNSUPPORTED;
  if (T == 0) return SMLA_OK;
  if (!scores || !n_cand || !out_ids) return SMLA_ERR_INVALID_ARG;
  if (misaligned(scores, 4) || misaligned(n_cand, 4) || misaligned(out_ids, 4) ||
      (out_scores && misaligned(out_scores, 4)))
    return SMLA_ERR_INVALID_ARG;
  const size_t need = smla::topk_workspace_bytes(T, L, K);
  if (workspace != nullptr && (workspace_bytes < need || misaligned(workspace, 16)))
    return SMLA_ERR_WORKSPACE;
  smla::TopkArgs a{};
  a.scores = scores;
  a.n_cand = n_cand;
  a.row_stride = row_stride;
  a.L = L;
  a.T = T;
  a.K = K;
  a.D = D;
  a.rank = rank;
  a.interleave = interleave;
  a.out_ids = out_ids;
  a.out_scores = out_scores;
  return from_cuda(smla::launch_topk_select(a, need > 0 ? workspace : nullptr,
                                            static_cast<cudaStream_t>(stream)));
}

smla_status smla_dcp_topk_merge(const int32_t* cand_ids, const float* cand_scores,
                                int64_t row_stride, int32_t M, int32_t T, int32_t K,
                                int32_t* out_ids, float* out_scores, void* stream) {
  if (T < 0 || M < 0 || row_stride < M) return SMLA_ERR_INVALID_ARG;
  if (K < 1 || K > SMLA_MAX_TOPK) return SMLA_ERR_UNSUPPORTED;
  if (T == 0) return SMLA_OK;
  if (!cand_ids || !cand_scores || !out_ids) return SMLA_ERR_INVALID_ARG;
  if (misaligned(cand_ids, 4) || misaligned(cand_scores, 4) || misaligned(out_ids, 4) ||
      (out_scores && misaligned(out_scores, 4)))
    return SMLA_ERR_INVALID_ARG;
  smla::TopkArgs a{};
  a.scores = cand_scores;
  a.cand_ids = cand_ids;
  a.row_stride = row_stride;
  a.M = M;
  a.T = T;
  a.K = K;
  a.D = 1;
  a.interleave = 1;
  a.out_ids = out_ids;
  a.out_scores = out_scores;
  return from_cuda(smla::launch_topk_merge(a, static_cast<cudaStream_t>(stream)));
}

smla_status smla_dcp_lse_merge(const uint16_t* const* outs,
                               const float* const* lses, int32_t D, int32_t T,
                               int32_t H, uint16_t* out, float* lse,
                               void* stream) {
  if (D < 1 || T < 0 || H < 1) return SMLA_ERR_INVALID_ARG;
  if (D > SMLA_MAX_DCP) return SMLA_ERR_UNSUPPORTED;
  if (T == 0) return SMLA_OK;
  if (!outs || !lses || !out || !lse) return SMLA_ERR_INVALID_ARG;
  if (misaligned(out, 16) || misaligned(lse, 4)) return SMLA_ERR_INVALID_ARG;
  smla::MergeArgs a;
  for (int d = 0; d < D; ++d) {
    if (!outs[d] || !lses[d] || misaligned(outs[d], 16) || misaligned(lses[d], 4))
      return SMLA_ERR_INVALID_ARG;
    a.outs[d] = outs[d];
    a.lses[d] = lses[d];
  }
  for (int d = D; d < smla::kMaxMerge; ++d) {
    a.outs[d] = nullptr;
    a.lses[d] = nullptr;
  }
  a.D = D;
  a.T = T;
  a.H = H;
  a.out = out;
  a.lse = lse;
  return from_cuda(smla::launch_merge(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
