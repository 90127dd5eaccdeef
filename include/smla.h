/*
 * smla.h -- C ABI of the GB300 sparse MLA decode library under
 * decode-context-parallel (DCP).
 *
 * The hot path has three steps, one call each:
 *
 *   1. smla_dcp_filter_convert_index  global top-k ids -> this rank's slots
 *   2. smla_sparse_mla_decode         attention over the packed fp8 cache,
 *                                     returning out and the softmax LSE
 *   3. smla_dcp_lse_merge             LSE-weighted merge of D partials
 *
 * and three more entry points run it differently:
 *
 *   smla_dcp_sparse_mla_decode_fused  steps 1-3 for D pools held by one GPU,
 *                                     in a single launch
 *   smla_dcp_sparse_mla_decode_fused_host
 *                                     the same from and to pinned host
 *                                     memory, copies overlapping the decode
 *   smla_sparse_mla_decode_noalloc    step 2 with library-owned split-K
 *                                     scratch (no workspace argument)
 *
 * and the dense form of the decode (every cached position of a request's
 * causal context instead of a top-k list):
 *
 *   smla_dcp_dense_mla_decode         per rank or merged over D pools
 *
 * and the step before the path, the global top-k of indexer scores:
 *
 *   smla_topk_select                  per row (per rank: as global ids)
 *   smla_dcp_topk_merge               top-k of the ranks' candidates
 *
 * Sources (page title, then section):
 *   [P1] "[eldritch] attention: support DCP in SM120 FlashInfer sparse MLA"
 *   [P2] "[Bugfix][Attention] Stabilize sparse-MLA DCP for GLM PCP evals"
 *   [P3] "FlashMLA sparse fp8 path + DCP + MTP" (vLLM PR #46514 summary)
 *
 * Conventions shared by every call:
 *   - Pointers marked "device" point to memory of the current CUDA device;
 *     the caller allocates and owns all of it.  The library never allocates,
 *     frees or synchronises, and keeps no pointer after a call returns, with
 *     two exceptions: smla_sparse_mla_decode_noalloc's split-K scratch is a
 *     library-owned device array of SMLA_NOALLOC_SCRATCH_BYTES per GPU, whose
 *     device address the library looks up once per device and keeps, and
 *     smla_dcp_sparse_mla_decode_fused_host creates its streams and events
 *     once per device and keeps them.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*,
 *     NULL = legacy default stream) and takes every scalar by value, so no
 *     call issues a host->device copy of its own or a host sync [P2 "DCP
 *     decode rank scalar"]; smla_dcp_sparse_mla_decode_fused_host copies
 *     only the caller's host buffers it is given, asynchronously.
 *   - Arguments are checked on the host before any launch; a failing check
 *     returns a status and launches nothing.  A failed launch returns
 *     SMLA_ERR_CUDA.  No C++ exception crosses this boundary.
 *   - T = 0 is a no-op that returns SMLA_OK.
 *   - Inputs the host cannot check (an id that runs past its block table, a
 *     slot past the pool) are caught in the kernels: the offending entry is
 *     treated as -1 and a bit is set in the device error word, readable with
 *     smla_get_device_error.  No kernel traps.
 *   - Index tensors are int32, row-major and contiguous.
 */
#ifndef SMLA_H_
#define SMLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int smla_status;

enum {
  SMLA_OK = 0,
  SMLA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned buffer   */
  SMLA_ERR_UNSUPPORTED = 2, /* valid but outside the supported envelope    */
  SMLA_ERR_WORKSPACE = 3,   /* workspace missing, too small or misaligned  */
  SMLA_ERR_CUDA = 4         /* a CUDA runtime call or launch failed        */
};

/* Bits of the device error word. */
enum {
  SMLA_DEVERR_BLOCK_TABLE = 1u, /* id past the block table / unallocated block */
  SMLA_DEVERR_REQ_ID = 2u,      /* req_id_per_token outside [0, num_reqs)      */
  SMLA_DEVERR_SLOT_RANGE = 4u,  /* local slot >= num_slots                     */
  SMLA_DEVERR_TIMEOUT = 8u,     /* a bounded wait inside a kernel gave up      */
  SMLA_DEVERR_CONTEXT = 16u,    /* dense decode: a context shorter than its
                                   request's query tokens or past max_ctx     */
  SMLA_DEVERR_RANGE = 32u       /* a q or rope value, or a latent group scale,
                                   that the fp16 keys cannot carry (below)    */
};
/* The decode kernels compute QK^T and PV on fp16 operands: q and the rope
 * values are converted from bf16 and each latent value is dequantised as
 * e4m3 code x scale, rounded once to fp16.  SMLA_DEVERR_RANGE is set when a
 * q or rope value of a row has |x| >= 65536 (inf / NaN included), when a
 * group scale exceeds 65504 / 448 (its dequantised values would overflow
 * fp16), or when a nonzero scale is below 2^-22 (its keys would be fp16
 * subnormals and lose precision).  The result is still written; the bit says
 * it may be outside the stated tolerances. */
/* With SMLA_DEVERR_TIMEOUT, bits 8..31 of the word tell which of the decode
 * kernel's internal waits gave up (a diagnostic bitmask, one bit per site). */

/* Largest gathered head count the decode kernel takes [P3 implementation
 * breakdown step 4: heads pad to the 64/128 kernel envelope]. */
#define SMLA_MAX_HEADS 128
/* Largest number of partials smla_dcp_lse_merge combines in one call. */
#define SMLA_MAX_DCP 16
/* Packed fp8_ds_mla row: 512 e4m3 codes | 4 fp32 scales | 64 bf16 rope. */
#define SMLA_ROW_BYTES 656
#define SMLA_QK_DIM 576
#define SMLA_V_DIM 512

/* Human-readable name of a status code (static string, never NULL). */
const char* smla_status_string(smla_status status);

/* Reads the device error word of the current device into *flags (a host
 * pointer) as an OR of SMLA_DEVERR_* bits; clears it when `clear` != 0.
 * This call synchronises with the device (it is a diagnostic, not part of
 * the hot path). */
smla_status smla_get_device_error(uint32_t* flags, int clear);

/*
 * Step 1 -- DCP filter + convert [P3 implementation breakdown step 2 and
 * the _forward_fp8_kv_mixed_batch snippet; P1 Summary].
 *
 * For row i (request r = req_id_per_token[i]) and entry j, with t =
 * topk_global[i*K + j] and interleave size I (runs of I consecutive
 * positions go to the ranks in turn; the pages name the size,
 * cp_kv_cache_interleave_size, and validate only I = 1 [P3 implementation
 * breakdown step 4]):
 *   t < 0 or (t div I) mod D != rank  -> local_slots[i*K + j] = -1
 *   otherwise lp = (t div (I*D))*I + t mod I (rank-local position; I = 1:
 *             t div D), local_slots[i*K + j] = block_table[r*bt_row_stride +
 *             lp div block_size] * block_size + lp mod block_size
 * The -1s stay in place (compact_valid_to_front = False).  With D = 1 and
 * rank = 0 this is the plain paged request-index -> slot conversion.
 * valid_count[i] (optional, may be NULL) receives the number of
 * non-negative outputs of row i.
 *
 *   req_id_per_token  device int32 [T]
 *   block_table       device int32 [num_reqs, bt_row_stride]; columns
 *                     [0, bt_width) are meaningful, -1 = unallocated
 *   topk_global       device int32 [T, K], global token positions, -1 padded
 *   local_slots       device int32 [T, K] output (may not alias inputs)
 *   valid_count       device int32 [T] output or NULL
 * Errors: INVALID_ARG for null pointers (T > 0), T < 0, K < 1, D < 1,
 * rank outside [0, D), block_size < 1, interleave < 1, num_reqs < 1,
 * bt_width < 1 or bt_row_stride < bt_width.  On the device an out-of-range
 * request id or a position past the block table (or in a -1 block) yields -1
 * and sets a device error bit.
 */
smla_status smla_dcp_filter_convert_index(
    const int32_t* req_id_per_token, const int32_t* block_table,
    int64_t bt_row_stride, int32_t bt_width, int32_t num_reqs,
    const int32_t* topk_global, int32_t T, int32_t K, int32_t D, int32_t rank,
    int32_t block_size, int32_t interleave, int32_t* local_slots,
    int32_t* valid_count, void* stream);

/*
 * Bytes of caller-owned workspace smla_sparse_mla_decode needs for (T, H,
 * K); 0 means none.  The size follows from the shape alone, so a caller can
 * allocate it once at start-up for its largest batch [P1 Implementation
 * Notes: per-device scratch allocated at initialisation; P2 "FlashInfer
 * sparse-MLA DCP workspace": size derived from tokens x gathered heads].
 * Returns 0 for invalid shapes.
 */
size_t smla_decode_workspace_size(int32_t T, int32_t H, int32_t K);

/*
 * Step 2 -- sparse MLA decode with LSE return [P1 Why; P3 implementation
 * breakdown steps 1 and 3; the _forward_fp8_kv_mixed_batch snippet].
 *
 * For row i, head h, over the valid entries j of local_slots row i
 * (slot >= 0; every occurrence counts):
 *   k_j   = dequant(kv_cache row slot_j)              576 dims
 *           (latent dim c = e4m3(code c) * scale[c div 128], rope = bf16)
 *   s_j   = sm_scale * <q[i,h,:], k_j>
 *   lse   = log(sum_j exp(s_j))           natural log, sm_scale included
 *   out   = sum_j exp(s_j - lse) * latent_j           512 dims
 * A row with no valid entry is written as the merge identity out = 0,
 * lse = -inf [P3 executive summary 1, implementation breakdown step 3].
 *
 *   q           device bf16 [T, H, 576] (16-byte aligned); H is the
 *               gathered head count [P1 Implementation Notes]
 *   kv_cache    device uint8 [num_slots, 656] (16-byte aligned)
 *   local_slots device int32 [T, K], -1 = masked (scattered, any order)
 *   out         device bf16 [T, H, 512] output, contiguous, 16-byte aligned
 *   lse         device fp32 [T, H] output, row = token (spec decode rows
 *               b*S + s) [P3 implementation breakdown steps 1 and 5]
 *   workspace   device scratch of at least
 *               smla_decode_workspace_size(T, H, K) bytes, 256-byte aligned,
 *               zero-filled before its first use (every call, including one
 *               that sets SMLA_DEVERR_TIMEOUT, leaves its arrival counters
 *               zero again); may be NULL when that size is 0.  Calls that
 *               run concurrently need distinct workspaces.
 * When the size is not 0 the rows are split over several key ranges
 * (split-K) and each range's partial (its normalised output in fp16, its
 * maximum and sum in fp32) goes through the workspace.  The
 * partials are merged by their LSE in the decode kernel (the last range of
 * a row to finish merges it) when the decode grid is larger than one wave
 * on the GPU or there are fewer than four ranges per row; otherwise by a
 * second kernel launched on `stream` with programmatic stream
 * serialisation.  Without split-K the call is a single kernel launch.
 * Errors: INVALID_ARG for null pointers, T < 0, K < 1, H < 1, num_slots < 0,
 * sm_scale not finite and positive, misaligned q/kv_cache/out; UNSUPPORTED
 * for H > SMLA_MAX_HEADS; WORKSPACE
 * when the workspace is too small, NULL or misaligned.  A slot >= num_slots
 * is treated as -1 and sets SMLA_DEVERR_SLOT_RANGE.
 */
smla_status smla_sparse_mla_decode(
    const uint16_t* q, const uint8_t* kv_cache, int64_t num_slots,
    const int32_t* local_slots, int32_t T, int32_t H, int32_t K,
    float sm_scale, uint16_t* out, float* lse, void* workspace,
    size_t workspace_bytes, void* stream);

/*
 * Step 2 without caller scratch.  The pages have no counterpart to this call:
 * it exists for callers that cannot allocate device memory -- code that runs
 * inside CUDA stream capture, where cudaMalloc is not allowed, or hosts that
 * forbid device allocation after start-up -- and so cannot provide the
 * workspace smla_sparse_mla_decode wants.
 *
 * Same arguments, semantics and errors as smla_sparse_mla_decode minus the
 * workspace: the split-K scratch is a library-owned array of
 * SMLA_NOALLOC_SCRATCH_BYTES in device memory, which every GPU that loads the
 * library holds until the process exits.  A shape whose scratch need
 * (smla_decode_workspace_size) exceeds that size returns SMLA_ERR_WORKSPACE
 * and launches nothing.  The call allocates nothing (no cudaMalloc, no
 * cudaFree, no allocating library routine); it clears the scratch's arrival
 * counters with cudaMemsetAsync on `stream` before each launch.
 *
 * The first call on a device looks up the array's device address there (with
 * that device current); make that first call before any stream capture.
 * Every call on a device shares the one array and it keeps the last call's
 * contents, so calls that overlap on the GPU (e.g. on two streams at once)
 * race and must be serialised by the caller.
 */
#define SMLA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
smla_status smla_sparse_mla_decode_noalloc(
    const uint16_t* q, const uint8_t* kv_cache, int64_t num_slots,
    const int32_t* local_slots, int32_t T, int32_t H, int32_t K,
    float sm_scale, uint16_t* out, float* lse, void* stream);

/*
 * Steps 1-3 in one launch (fused DCP step for D shards held by one GPU; with
 * split-K, a second launch may merge the key ranges, as for
 * smla_sparse_mla_decode).
 *
 * Computes exactly what the three calls above compute for D shard pools --
 * filter + convert per shard, sparse MLA decode per shard, LSE merge -- in a
 * single kernel: the global-to-local conversion of "FlashMLA sparse fp8 path
 * + DCP + MTP" (implementation breakdown step 2) runs in the kernel's
 * prologue for every shard, the compacted keys of all shards share one online
 * softmax, and since the LSE merge of per-shard softmax partials equals the
 * softmax over the union of their keys ("[eldritch] attention: support DCP in
 * SM120 FlashInfer sparse MLA", Why: the merge reduces partial attention
 * results), the output is the merged (out, lse) directly.  A row whose ids
 * all map to nothing is written as (0, -inf).
 *
 *   q, T, H, K, sm_scale, out, lse   as in smla_sparse_mla_decode (out/lse
 *                                    receive the merged result)
 *   req_id_per_token, topk_global, num_reqs, D, block_size, interleave
 *                                    as in smla_dcp_filter_convert_index
 *   kv_caches      host array of D device pointers, pool d = uint8
 *                  [num_slots[d], 656], 16-byte aligned
 *   num_slots      host array of D pool sizes
 *   block_tables   host array of D device pointers, table d = int32
 *                  [num_reqs, bt_row_strides[d]], columns [0, bt_widths[d])
 *   workspace      >= smla_decode_workspace_size(T, H, K) bytes, same rules
 *                  as for smla_sparse_mla_decode
 * Errors: as the three calls above (INVALID_ARG for interleave < 1);
 * UNSUPPORTED for D > SMLA_MAX_DCP.
 * Device-side input errors (ids past a block table, bad request ids, slots
 * past a pool) drop the entry and set the device error word.
 */
smla_status smla_dcp_sparse_mla_decode_fused(
    const uint16_t* q, int32_t T, int32_t H, int32_t K, float sm_scale,
    const int32_t* req_id_per_token, const int32_t* topk_global, int32_t num_reqs,
    int32_t D, int32_t block_size, int32_t interleave, const uint8_t* const* kv_caches,
    const int64_t* num_slots, const int32_t* const* block_tables,
    const int64_t* bt_row_strides, const int32_t* bt_widths, uint16_t* out,
    float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The fused DCP step for callers whose q, top-k ids and results live in
 * host memory (the pages have no counterpart: it is the same step,
 * smla_dcp_sparse_mla_decode_fused, with its host<->device copies).
 *
 * The rows are cut into `chunks` contiguous groups (1 <= chunks <=
 * SMLA_MAX_HOST_CHUNKS, at most T).  Group g's q rows and top-k ids are
 * copied into the device staging buffers, its decode is launched as soon as
 * they have landed, and its out and lse rows are copied back as soon as its
 * decode ends, so the copies of some groups overlap the decode of others.
 * With chunks > 1 each group's decode runs without split-K (every group
 * keeps its own SM pairs, side by side with the others), which needs
 * K <= 2048; with chunks == 1 the copies, the decode (the usual split-K
 * policy and workspace) and the copies back run one after the other.
 *
 *   q_host, topk_host       pinned host bf16 [T, H, 576], int32 [T, K]
 *   out_host, lse_host      pinned host bf16 [T, H, 512], fp32 [T, H] outputs
 *   q_dev, topk_dev,        device staging buffers of the same shapes (16-byte
 *   out_dev, lse_dev        aligned; 4 for lse_dev), owned by the caller;
 *                           they hold the step's device copies afterwards
 *   other arguments         as for smla_dcp_sparse_mla_decode_fused
 *                           (req_id_per_token, pools, block tables and
 *                           workspace in device memory)
 * Everything is ordered after the work already queued on `stream`, and work
 * queued on `stream` after the call waits for the whole step, including the
 * copies back: the host buffers hold the results once `stream` has reached
 * that point.  The groups run on library-owned streams and events (created
 * on a device's first call, kept until the process exits); the call is
 * serialised per device, so concurrent calls from several host threads
 * queue one after the other.  Made inside CUDA stream capture on `stream`
 * (after one call outside it on the device), the library's streams join the
 * capture through those events and the graph replays the whole step.
 * Errors: as smla_dcp_sparse_mla_decode_fused, plus INVALID_ARG for a null
 * or misaligned host or staging buffer or chunks outside [1,
 * SMLA_MAX_HOST_CHUNKS]; UNSUPPORTED for chunks > 1 with K > 2048.
 */
#define SMLA_MAX_HOST_CHUNKS 8
smla_status smla_dcp_sparse_mla_decode_fused_host(
    const uint16_t* q_host, const int32_t* topk_host, uint16_t* out_host, float* lse_host,
    uint16_t* q_dev, int32_t* topk_dev, uint16_t* out_dev, float* lse_dev,
    int32_t T, int32_t H, int32_t K, float sm_scale, const int32_t* req_id_per_token,
    int32_t num_reqs, int32_t D, int32_t block_size, int32_t interleave,
    const uint8_t* const* kv_caches, const int64_t* num_slots,
    const int32_t* const* block_tables, const int64_t* bt_row_strides,
    const int32_t* bt_widths, void* workspace, size_t workspace_bytes, int32_t chunks,
    void* stream);

/*
 * Dense MLA decode with LSE return under DCP [P3 key snippets: the dense
 * FlashMLA decode path, whose LSE comes back as [batch, heads, seq_len] and
 * is flattened to [tokens, heads] for the DCP merge; implementation breakdown
 * step 5].
 *
 * Request b has S query tokens (S > 1: an MTP / speculative step); token s
 * sits at position p = ctx_lens[b] - S + s and attends every cached position
 * 0..p of its request (causal), with the attention of smla_sparse_mla_decode
 * over those positions' cache rows.  Position t lives on rank (t div I) mod
 * D at local position (t div (I*D))*I + t mod I, as in
 * smla_dcp_filter_convert_index.
 *   rank = -1       attend all D pools in one launch: out/lse are the merged
 *                   result (the LSE merge of the ranks' partials)
 *   rank in [0, D)  attend only rank's positions: out/lse are that rank's
 *                   partial, to be combined with smla_dcp_lse_merge
 * Rows come out in token order b*S + s: out [B*S, H, 512], lse [B*S, H] --
 * the pages' [batch, heads, seq_len] -> [tokens, heads] flattening.
 *
 *   q              device bf16 [B*S, H, 576]
 *   ctx_lens       device int32 [B], each in [S, max_ctx]
 *   max_ctx        host bound on every ctx_lens[b] (sizes the split-K)
 *   kv_caches, num_slots, block_tables, bt_row_strides, bt_widths
 *                  host arrays of D entries as in
 *                  smla_dcp_sparse_mla_decode_fused (block-table row b
 *                  belongs to request b); with rank >= 0 only entry [rank]
 *                  is read and the others may be NULL / 0
 *   workspace      >= smla_dense_decode_workspace_size(B*S, H, max_ctx, D,
 *                  interleave, rank) bytes, same rules as for
 *                  smla_sparse_mla_decode
 * Errors: INVALID_ARG for null pointers, B < 0, S < 1, H < 1, max_ctx < 1,
 * D < 1, rank outside [-1, D), block_size < 1, interleave < 1, a bad pool or
 * table entry that is read, misaligned q/out/lse; UNSUPPORTED for H >
 * SMLA_MAX_HEADS or D > SMLA_MAX_DCP; WORKSPACE as for smla_sparse_mla_decode.
 * On the device a request whose context is outside [S, max_ctx] comes out
 * as (0, -inf) in all its rows and sets SMLA_DEVERR_CONTEXT; a position past
 * a block table sets SMLA_DEVERR_BLOCK_TABLE.
 */
size_t smla_dense_decode_workspace_size(int32_t T, int32_t H, int32_t max_ctx, int32_t D,
                                        int32_t interleave, int32_t rank);
smla_status smla_dcp_dense_mla_decode(
    const uint16_t* q, int32_t B, int32_t S, int32_t H, float sm_scale,
    const int32_t* ctx_lens, int32_t max_ctx, int32_t D, int32_t rank,
    int32_t block_size, int32_t interleave, const uint8_t* const* kv_caches,
    const int64_t* num_slots, const int32_t* const* block_tables,
    const int64_t* bt_row_strides, const int32_t* bt_widths, uint16_t* out,
    float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Global top-k selection of indexer scores: the step that produces the
 * path's global top-k ids ["[eldritch] ..." Summary: global sparse top-k
 * token ids; P3 related PRs: the DCP sparse indexer's global top-k merge].
 * The pages print no rule; the rule taken: keep the K largest scores, ranked
 * by score descending and then token id ascending, -1 padded when a row has
 * fewer than K candidates; NaN ranks below every number, -0 equals +0.
 *
 * smla_topk_select: row i's candidates are the local positions
 * j < n_cand[i] (clipped to [0, L]) of rank `rank`, with scores
 * scores[i*row_stride + j]; the ids written are their global positions:
 * local position j of rank r is global position (j div I)*I*D + r*I +
 * j mod I, the inverse of smla_dcp_filter_convert_index's rule (D = 1,
 * rank = 0: the plain top-k of positions 0..n-1).
 *   scores      device fp32 [T, row_stride]
 *   n_cand      device int32 [T]
 *   out_ids     device int32 [T, K] output
 *   out_scores  device fp32 [T, K] output (the kept scores) or NULL
 *   workspace   NULL, or device scratch of at least
 *               smla_topk_select_workspace_size(T, L, K) bytes, 16-byte
 *               aligned (no initial contents); calls that run concurrently
 *               need distinct workspaces.  With it, a call of at most 32
 *               rows whose L is at least 16 x max(16384, 8 x K rounded up
 *               to a power of two) cuts each row into min(8, SMs / T)
 *               chunks, one CTA each keeping the chunk's K best, and a
 *               second launch selects the row's K best among those; without
 *               it (or when the size is 0) each row is walked whole, by two
 *               CTAs (a cluster) when L >= 16384 and 2 T CTAs fit on the
 *               GPU at once, else by one.  The result is the same either
 *               way.
 *
 * smla_dcp_topk_merge: row i's candidates are the entries j < M with
 * cand_ids[i*row_stride + j] >= 0 (global ids, unique per row) and their
 * cand_scores; writes the top K of the union by the same rule -- with each
 * rank's smla_topk_select output concatenated, exactly the unsharded top-k.
 *
 * Errors: INVALID_ARG for null pointers (T > 0), T < 0, L < 0, M < 0,
 * row_stride < L (or < M), D < 1, rank outside [0, D), interleave < 1,
 * misaligned buffers; UNSUPPORTED for K outside [1, SMLA_MAX_TOPK];
 * WORKSPACE for a non-NULL workspace smaller than the size below or not
 * 16-byte aligned.
 *
 * smla_topk_select_workspace_size: bytes of the optional workspace for
 * (T, L, K), from the shape alone; 0 when no row can be long enough to be
 * cut, or for invalid shapes.
 */
#define SMLA_MAX_TOPK 16384
size_t smla_topk_select_workspace_size(int32_t T, int32_t L, int32_t K);
smla_status smla_topk_select(const float* scores, int64_t row_stride, int32_t L,
                             const int32_t* n_cand, int32_t T, int32_t K, int32_t D,
                             int32_t rank, int32_t interleave, int32_t* out_ids,
                             float* out_scores, void* workspace, size_t workspace_bytes,
                             void* stream);
smla_status smla_dcp_topk_merge(const int32_t* cand_ids, const float* cand_scores,
                                int64_t row_stride, int32_t M, int32_t T, int32_t K,
                                int32_t* out_ids, float* out_scores, void* stream);

/*
 * Step 3 -- LSE-weighted merge of D partials [P1 Why, Scope / Limitations
 * (the ag_rs flow); P3 executive summary 1 and implementation breakdown
 * step 3].  With M = max_d lse_d[t,h]:
 *   M = -inf  -> out = 0, lse = -inf
 *   otherwise lse = M + log(sum_d exp(lse_d - M)),
 *             out = sum_d exp(lse_d - lse) * out_d
 * On one GPU this stands in for the cross-rank LSE all-gather plus output
 * reduce-scatter.
 *
 *   outs  host array of D device pointers, each bf16 [T, H, 512], 16-byte
 *         aligned
 *   lses  host array of D device pointers, each fp32 [T, H]
 *   out   device bf16 [T, H, 512] output (may alias none of the inputs)
 *   lse   device fp32 [T, H] output
 * Errors: INVALID_ARG for null pointers, D < 1, T < 0, H < 1, misaligned
 * buffers; UNSUPPORTED for D > SMLA_MAX_DCP.
 */
smla_status smla_dcp_lse_merge(const uint16_t* const* outs,
                               const float* const* lses, int32_t D, int32_t T,
                               int32_t H, uint16_t* out, float* lse,
                               void* stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* SMLA_H_ */
