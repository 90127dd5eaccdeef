// Sparse MLA decode over the packed fp8_ds_mla cache on tcgen05 tensor cores.
//
// What it computes ("FlashMLA sparse fp8 path + DCP + MTP", implementation
// breakdown steps 1 and 3; "[eldritch] attention: support DCP in SM120
// FlashInfer sparse MLA", Why): for query row t and head h, over the valid
// local slots j of row t,
//     s_j = sm_scale * <q[t,h,0:576], (latent_j || rope_j)>
//     lse = ln sum_j exp(s_j),   out = sum_j exp(s_j - lse) * latent_j
// with latent_j = e4m3(code) * scale[dim / 128].  A row with no valid slot is
// written as the merge identity (out = 0, lse = -inf).
//
// Design (GB300, one cluster of two CTAs per query row):
//   * Heads are the MMA M dimension (M = 128, heads padded with zero rows),
//     so the 576-wide latent keys are shared by all heads (MQA-style).
//   * The fp32 accumulator O[128 x 512] alone fills a whole SM's tensor
//     memory, so CTA c of the pair owns value dims [256c, 256c + 256).  The
//     QK^T contraction is split by key dimension the same way: CTA c
//     contracts latent dims [256c, 256c + 256) (its value half) and rope dims
//     [32c, 32c + 32), 288 key dims each, so every cache byte is fetched by
//     one CTA.  The two fp32 partial score tiles are exchanged through
//     distributed shared memory each tile, so no FLOP is recomputed.  Both
//     CTAs then run the identical online softmax.
//   * Q (this CTA's key-dim half) and P live in tensor memory as the A
//     operand; K/V tiles are the B operand in shared memory (128-byte
//     swizzle): one buffer serves as K (K-major) for QK^T and as V
//     (MN-major) for PV.
//   * Keys are dequantised to fp16 with a single rounding: the e4m3 code is
//     exact in fp16 and the fp32 scale is split into fp16 hi + lo parts, so
//     code*hi + code*lo is rounded once by a fused multiply-add.  fp16 keeps
//     3 more mantissa bits than bf16, which keeps score errors well inside
//     the LSE tolerance even for rows with a single valid slot.
//   * Valid slots are compacted in order in the prologue (-1 never costs a
//     load or an MMA).  Each gather thread loads its fixed share of every key
//     row straight into registers one tile ahead and converts it from there;
//     three operand tiles are in flight.
//   * The partial score tiles travel as asynchronous remote stores counted on
//     the receiving CTA's mbarrier (st.async + expect_tx).
//   * Softmax in the log2 domain with a lazily moved reference maximum: the
//     O accumulator in TMEM is rescaled only when the row maximum grows by
//     more than 2^8.
//
// Warp roles (384 threads): warps 0-3 softmax/epilogue (TMEM lanes 0-127,
// one head row per thread), warps 4-7 dequantise, warp 8 allocates TMEM and
// issues every MMA (one thread: QK^T of a tile, then PV of the tile two
// before it, once the softmax has stored that tile's P), warps 9-11 gather.
// Every wait is bounded; a wait that runs out sets SMLA_DEVERR_TIMEOUT and
// the CTA unwinds.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>
#include <mutex>

#include "../../include/smla.h"
#include "smla_internal.h"
#include "smla_sm100.cuh"

namespace smla {
namespace {

using namespace sm100;

__device__ unsigned int g_decode_error;

// What a row's raw entries are: local slots of one pool (per-shard decode),
// global top-k positions over D pools (fused DCP step), or the positions of
// the row's whole causal context (dense decode).
enum : int { kModeSlots = 0, kModeTopk = 1, kModeDense = 2 };

constexpr int kTileN = 64;        // keys per tile (MMA N of QK^T, K of PV)
constexpr int kThreads = 384;     // 12 warps
constexpr int kStages = 4;        // fp16 operand tiles in flight
constexpr int kRawStages = 1;     // raw cache-row tiles in shared memory (one more in registers)
constexpr int kMmaWarp = 8;
constexpr int kLoaderWarp0 = 9;   // warps 9..11 stage cache rows
constexpr int kLoaders = 96;
constexpr int kMaxList = kDecodeMaxList;  // compacted slots one cluster handles

// tensor-memory columns (512 allocated)
constexpr uint32_t kOCol = 0;     // O half: 256 fp32 columns
constexpr uint32_t kSCol = 256;   // S tile: 64 fp32 columns
constexpr uint32_t kPCol = 320;   // P tile: 64 fp16 = 32 columns
constexpr uint32_t kQCol = 352;   // Q part: 288 fp16 = 144 columns
constexpr uint32_t kTmemCols = 512;

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kKBlockBytes = kTileN * 128;          // 64 keys x 64 fp16, 128-byte swizzle
constexpr int kRopeBlock = 4 * kKBlockBytes;        // 64 keys x 32 fp16, 64-byte swizzle
constexpr int kOpTileBytes = kRopeBlock + kTileN * 64;  // 256 latent + 32 rope dims
constexpr int kRawStride = 336;                     // staged bytes of one cache row
constexpr int kRawTileBytes = kTileN * kRawStride;  // one tile of staged rows
// Per tile and direction the pair exchanges the fp32 partial scores of half
// the tile's keys (XA) and then the fp16 P of the other half plus each row's
// reference maximum and partial sum (XB).
constexpr int kXABytes = 128 * (kTileN / 2) * 4;
constexpr int kXBPBytes = 128 * (kTileN / 2) * 2;
constexpr int kXBBytes = kXBPBytes + 128 * 8;
constexpr int kXBytes = kXABytes + kXBBytes;         // one buffer set
constexpr int kOffOp = 0;
constexpr int kOffRaw = kOffOp + kStages * kOpTileBytes;
constexpr int kOffX = kOffRaw + kRawStages * kRawTileBytes;
constexpr int kOffList = kOffX + 2 * kXBytes;  // two buffer sets
constexpr int kBtStageMax = 2 * kXBytes / 4;    // staged block-table entries (fused prologue)
constexpr int kOffListShard = kOffList + kMaxList * 4;  // fused step: shard of each key
constexpr int kOffCtl = kOffListShard + kMaxList;
constexpr int kCtlBytes = 1024;
constexpr int kSmemBytes = kOffCtl + kCtlBytes + 1024;  // + control block + alignment slack

// Per shard: its staged block-table row's offset in the staging area, the
// row's meaningful columns and the pool's slot count (one 16-byte read).
struct __align__(16) ShardMeta {
  int32_t bt_off, bt_width;
  int64_t pool_slots;
};

struct Ctl {
  uint64_t q_tma, q_ready, full[kStages], freed[kStages], raw_full[kRawStages], raw_empty[kRawStages],
      s_full, s_free, pv_done, p_full, xa[2], xb[2], end;
  uint32_t tbase;
  int n_list;
  int abort;
  int is_last;
  int warp_cnt[8];  // the compacting warps' valid counts
  // fused step: per shard, its pool and this row's request row of its table
  const uint8_t* pool[kMaxMerge];
  const int32_t* bt_row[kMaxMerge];
  ShardMeta meta[kMaxMerge];
  int bt_staged;              // the rows fit the staging area
};
static_assert(sizeof(Ctl) <= kCtlBytes, "control block");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Programmatic dependent launch: a grid launched after this one with
// programmatic stream serialisation may be scheduled once every CTA here has
// signalled (or exited); it waits for this grid's completion and memory in
// griddepcontrol.wait.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait sites, recorded in bits 8.. of the device error word when a wait
// gives up (diagnostic).
enum WaitSite : uint32_t {
  kWsSFull = 0, kWsExchange, kWsPvDone, kWsPvLast, kWsFreed, kWsQReady, kWsFull, kWsSFree,
  kWsPFull, kWsDrain, kWsRaw, kWsRawEmpty, kWsExchangeP
};

// Every wait is bounded in time (kWaitNs of the global timer); a wait that
// gives up records TIMEOUT plus its site and raises the CTA's abort flag so
// the other roles stop waiting too.
constexpr uint64_t kWaitNs = 2000000000ull;

template <bool kCluster>
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort,
                                           uint32_t site) {
  auto probe = [&]() {
    return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (!probe()) {
    if (*abort) return false;
    if ((++it & 63u) == 0 && globaltimer_ns() - t0 > kWaitNs) {
      atomicOr(&g_decode_error, SMLA_DEVERR_TIMEOUT | (1u << (8 + site)));
      *abort = 1;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         uint32_t site) {
  return wait_phase<false>(bar, parity, abort, site);
}

__device__ __forceinline__ bool wait_bar_cluster(uint64_t* bar, uint32_t parity,
                                                 volatile int* abort, uint32_t site) {
  return wait_phase<true>(bar, parity, abort, site);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Nonzero when a bf16 of the pair in `w` would not fit fp16 (|x| >= 65536:
// bf16 has no value between 65280 and 65536, and fp16's largest is 65504;
// inf and NaN included): each 15-bit magnitude plus 0x3880 reaches bit 15
// exactly when it is >= 0x4780, with no carry between the halves.
__device__ __forceinline__ uint32_t bf16x2_over_fp16(uint32_t w) {
  return ((w & 0x7FFF7FFFu) + 0x38803880u) & 0x80008000u;
}

__device__ __forceinline__ uint32_t bf16x8_over_fp16(const uint4& v) {
  return bf16x2_over_fp16(v.x) | bf16x2_over_fp16(v.y) | bf16x2_over_fp16(v.z) |
         bf16x2_over_fp16(v.w);
}

// A latent group scale the fp16 keys cannot carry: its dequantised values
// (up to 448 x scale) overflow fp16, or a nonzero scale so small that
// 2^8 x scale is an fp16 subnormal (the keys lose precision); NaN included.
__device__ __forceinline__ bool scale_out_of_range(float s) {
  return !(s <= 65504.f / 448.f) || (s != 0.f && s < 0x1p-22f);
}

// 8 bf16 -> 8 fp16 (exact for values in fp16 range)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    o[k] = h2_bits(__floats2half2_rn(__uint_as_float(w[k] << 16),
                                     __uint_as_float(w[k] & 0xffff0000u)));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Two e4m3 codes (bytes `sel` picks) -> fp16x2 holding code * 2^-8, exactly,
// on the integer pipe: the sign moves to fp16's sign bit and the 7 exponent /
// mantissa bits drop in one position lower (4-bit exponent under fp16's
// 5-bit field, bias 7 vs 15), which makes normal and subnormal codes alike
// land on code * 2^-8.  (e4m3 NaN codes, which no quantiser emits, are not
// special-cased.)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled_down(uint32_t w, uint32_t sel) {
  const uint32_t y = __byte_perm(w, 0u, sel);  // code a in bits 15:8, code b in 31:24
  return (y & 0x80008000u) | ((y & 0x7F007F00u) >> 1);
}

// 8 e4m3 codes -> 8 fp16 values code * scale with one rounding: hi + lo is
// the fp32 scale * 2^8 split into two fp16 parts, and fma(c, hi, c * lo)
// rounds once.
__device__ __forceinline__ uint4 e4m3x8_scaled(uint2 codes, __half2 hi, __half2 lo) {
  const uint32_t w[2] = {codes.x, codes.y};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const uint32_t bits = e4m3x2_to_f16x2_scaled_down(w[k], p == 0 ? 0x1404u : 0x3424u);
      const __half2 c = *reinterpret_cast<const __half2*>(&bits);
      o[2 * k + p] = h2_bits(__hfma2(c, hi, __hmul2(c, lo)));
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 2^x; results below 2^-126 flush to zero (a softmax weight that small is
// zero in the fp16 P tile anyway)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The two CTAs of a pair split the work by key dimension, symmetrically:
// CTA c gathers and contracts latent dims [256c, 256c + 256) (the value dims
// of its O half) and rope dims [32c, 32c + 32), 288 key dims each, laid out
// in its operand tile as dims 0..255 (latent) and 256..287 (rope).  Every
// cache byte is fetched by one CTA (the 16 bytes of scales by both).  All of
// it is runtime data of the CTA's rank, so the two CTAs share one
// instruction stream (half the code, for the instruction cache).
constexpr int kQkDims = 288;
constexpr int kKSteps = kQkDims / 16;  // MMA K = 16

struct HalfRt {
  int c;  // CTA rank in the pair
};

__device__ __forceinline__ HalfRt half_of(uint32_t c) {
  HalfRt r;
  r.c = int(c);
  return r;
}

// The bytes of a cache row CTA c stages, at kRawStride per row, in 21
// pieces of 16 bytes:
//   pieces 0..15:  codes [256c, 256c + 256)      -> raw [0, 256)
//   piece  16:     the four fp32 scales [512, 528) -> raw [256, 272)
//   pieces 17..20: rope bf16 [528 + 64c, 592 + 64c) -> raw [272, 336)
constexpr int kPiecesPerRow = 21;
__device__ __forceinline__ int piece_src(int c, int j) {
  return j < 16 ? 256 * c + 16 * j : j == 16 ? 512 : 528 + 64 * c + 16 * (j - 17);
}
constexpr int kRawScales = 256;
constexpr int kRawRope = 272;

// Converter thread (key, part) of CTA c converts its key's code pieces
// [8 part, 8 part + 8) (tile dims 128 part .. 128 part + 127, all in scale
// group 2c + part) and rope pieces 2 part, 2 part + 1 (tile dims 256 + 16 part
// .. 256 + 16 part + 15).
constexpr int kCodePerPart = 8;
constexpr int kRopePerPart = 2;

// Cache row of entry `idx` of the compacted list.
template <int kMode>
__device__ __forceinline__ const uint8_t* row_ptr(const DecodeArgs& a, const Ctl* ctl,
                                                  const int* list, const uint8_t* shard,
                                                  int idx) {
  const uint8_t* pool = kMode != kModeSlots ? ctl->pool[shard[idx]] : a.kv;
  return pool + int64_t(list[idx]) * SMLA_ROW_BYTES;
}

__device__ __forceinline__ void split_scale(float s, __half2& hi, __half2& lo) {
  const float x = 256.f * s;  // the integer code decode leaves a factor 2^-8 out
  const __half h = __float2half_rn(x);
  hi = __half2half2(h);
  lo = __half2half2(__float2half_rn(x - __half2float(h)));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Operand tile address of 8 consecutive dims from tile dim `ldim` of `key`:
// dims 0..255 in four 128-byte-swizzled K-blocks, dims 256..287 (rope) in
// one 64-byte-swizzled block.
__device__ __forceinline__ uint32_t op_addr(uint32_t op, int key, int ldim) {
  return ldim < 256 ? op + (ldim >> 6) * kKBlockBytes + sw128_offset(key, (ldim & 63) >> 3)
                    : op + kRopeBlock + sw64_offset(key, (ldim - 256) >> 3);
}

// One converter thread's staged pieces of its key: 8 code pieces, 2 rope
// pieces and the scale of its code pieces' group.
struct ConvRegs {
  uint4 cur[kCodePerPart + kRopePerPart];
  float scale;
};

// Read this thread's staged pieces of its key (`row` = the key's staged row;
// zeros for a key past the row's valid count).  Lanes read rows kRawStride
// apart: 16-byte accesses of 8 consecutive keys hit 8 different bank groups.
__device__ __forceinline__ void read_row(uint32_t row, bool live, int c, int part, ConvRegs& r) {
  const uint32_t code0 = row + 16 * kCodePerPart * part;
  const uint32_t rope0 = row + kRawRope + 32 * part;
#pragma unroll
  for (int k = 0; k < kCodePerPart; ++k)
    r.cur[k] = live ? lds128(code0 + 16 * k) : make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int q = 0; q < kRopePerPart; ++q)
    r.cur[kCodePerPart + q] = live ? lds128(rope0 + 16 * q) : make_uint4(0, 0, 0, 0);
  // the one scale group of this thread's codes
  r.scale = live ? ld_shared_f32(row + kRawScales + 4 * (2 * c + part)) : 0.f;
}

// Convert the read pieces into the swizzled fp16 operand tile at `op` (the
// same code path for both CTA ranks and parts).
// Returns true when the key's scale or rope values do not fit the fp16 keys.
__device__ __forceinline__ bool convert_row(const ConvRegs& r, uint32_t op, int key, int part) {
  __half2 hi, lo;
  split_scale(r.scale, hi, lo);
#pragma unroll
  for (int k = 0; k < kCodePerPart; ++k) {
    const int ldim = 128 * part + 16 * k;
    sts128(op_addr(op, key, ldim), e4m3x8_scaled(make_uint2(r.cur[k].x, r.cur[k].y), hi, lo));
    sts128(op_addr(op, key, ldim + 8), e4m3x8_scaled(make_uint2(r.cur[k].z, r.cur[k].w), hi, lo));
  }
  uint32_t over = 0;
#pragma unroll
  for (int q = 0; q < kRopePerPart; ++q) {
    over |= bf16x8_over_fp16(r.cur[kCodePerPart + q]);
    sts128(op_addr(op, key, 256 + 16 * part + 8 * q), bf16x8_to_f16x8(r.cur[kCodePerPart + q]));
  }
  return over != 0 || scale_out_of_range(r.scale);
}

// The loader warps' loop.  Loader ld owns pieces ld + 96k (k < 14) of every
// tile (a tile has 64 rows x 21 pieces = 14 x 96), so consecutive lanes read
// consecutive 16 bytes of a row (whole sectors, few transactions).  A tile's
// pieces are loaded into registers while the raw stage holds the tile before
// it, and stored once the converter warps have read that tile out of the
// stage.  Load-issue stalls (the memory system's request slots) fall on these
// warps, not on the converters.
constexpr int kPiecesPerLoader = kTileN * kPiecesPerRow / kLoaders;
static_assert(kPiecesPerLoader * kLoaders == kTileN * kPiecesPerRow, "loaders share a tile evenly");
static_assert(kTileN * kRawStride <= (1 << 15) && SMLA_ROW_BYTES <= (1 << 10) && kTileN <= (1 << 7),
              "packed piece offsets fit their fields");

template <int kMode>
__device__ void loader_loop(const DecodeArgs& a, Ctl* ctl, uint8_t* sm, int n, int ntiles, int c,
                            int ld, volatile int* abort) {
  const int* list = reinterpret_cast<const int*>(sm + kOffList);
  const uint8_t* list_shard = sm + kOffListShard;
  const uint32_t raw0 = smem_u32(sm + kOffRaw);
  uint4 buf[kPiecesPerLoader];
  // Each piece's place is the same in every tile: its row r in the tile, its
  // source offset in the cache row and its destination offset in the raw
  // stage, packed once as r << 25 | src << 15 | dst (dst < 2^15, src < 2^10).
  uint32_t pk[kPiecesPerLoader];
#pragma unroll
  for (int k = 0; k < kPiecesPerLoader; ++k) {
    const int p = ld + kLoaders * k;                   // < 64 * 21
    const int r = int((uint32_t(p) * 3121u) >> 16);  // p / 21, exact for p < 64 * 21
    const int j = p - r * kPiecesPerRow;
    pk[k] = uint32_t(r) << 25 | uint32_t(piece_src(c, j)) << 15 |
            uint32_t(r * kRawStride + 16 * j);
  }
  auto load = [&](int tile) {
    const int base = tile * kTileN;
    const uint32_t rows = uint32_t(min(kTileN, n - base));
#pragma unroll
    for (int k = 0; k < kPiecesPerLoader; ++k) {
      const uint32_t r = pk[k] >> 25;
      if (r < rows) {
        const uint8_t* row = row_ptr<kMode>(a, ctl, list, list_shard, base + int(r));
        buf[k] = ldg_stream(row + ((pk[k] >> 15) & 1023u));
      }
    }
  };
  auto store = [&](int tile, uint32_t stage) {
    const uint32_t rows = uint32_t(min(kTileN, n - tile * kTileN));
#pragma unroll
    for (int k = 0; k < kPiecesPerLoader; ++k)
      if ((pk[k] >> 25) < rows) sts128(stage + (pk[k] & 0x7fffu), buf[k]);
  };
  if (ntiles > 0) load(0);
#pragma unroll 1
  for (int t = 0; t < ntiles; ++t) {
    const int st = t % kRawStages;
    if (t >= kRawStages &&
        !wait_bar(&ctl->raw_empty[st], ((t - kRawStages) / kRawStages) & 1, abort, kWsRawEmpty))
      break;
    store(t, raw0 + st * kRawTileBytes);
    mbar_arrive(&ctl->raw_full[st]);
    if (t + 1 < ntiles) load(t + 1);
  }
}

// The converter threads' tile loop: each staged tile is converted into the
// fp16 operand stage once the MMAs of the tile two back have released it,
// then handed back to the loaders (one arrival per warp).
__device__ void convert_loop(Ctl* ctl, uint8_t* sm, int n, int ntiles, int key, int c, int part,
                             int lane, volatile int* abort) {
  const uint32_t raw0 = smem_u32(sm + kOffRaw);
  const uint32_t op0 = smem_u32(sm + kOffOp);
  bool out_of_range = false;
#pragma unroll 1
  for (int i = 0; i < ntiles; ++i) {
    const int st = i % kRawStages;
    if (!wait_bar(&ctl->raw_full[st], (i / kRawStages) & 1, abort, kWsRaw)) break;
    ConvRegs r;
    read_row(raw0 + st * kRawTileBytes + key * kRawStride, key < n - i * kTileN, c, part, r);
    // the raw stage goes back to the loaders as soon as the warp has read it
    // (the warp barrier orders the lanes' reads before lane 0's release), so
    // they refill it while this tile is converted
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->raw_empty[st]);
    if (i >= kStages &&
        !wait_bar(&ctl->freed[i % kStages], ((i - kStages) / kStages) & 1, abort, kWsFreed))
      break;
    out_of_range |= convert_row(r, op0 + (i % kStages) * kOpTileBytes, key, part) &&
                    key < n - i * kTileN;
    fence_async_shared();
    mbar_arrive(&ctl->full[i % kStages]);
  }
  if (out_of_range) atomicOr(&g_decode_error, SMLA_DEVERR_RANGE);
}

// Split-K epilogue (softmax warps): write this split's unnormalised O half,
// its log2-domain reference maximum and its sum (-inf and 0 when it holds
// no partial).  With the in-kernel combine the split then counts itself in:
// the CTA whose split arrives last for its row and value half learns so in
// `ctl->is_last` and combines the row once all its warps are free (see
// combine_splits).  A split whose CTA gave up on a wait (`ok` false,
// SMLA_DEVERR_TIMEOUT set) still arrives, contributing nothing, so the
// counter always completes and the workspace stays valid for the next call.
__device__ void split_epilogue(const DecodeArgs& a, Ctl* ctl, int C, int64_t t, int split, int ntiles,
                               float m_ref, float l, uint32_t tb, int warp, int h, bool ok) {
  const int S = a.splits;
  const bool live = h < a.H;
  const int64_t row = (t * S + split) * a.H + (live ? h : 0);
  // the split's own normalised output O / l, in fp16: an average of the
  // fp16 value rows, so within their range, rounded once (2^-11 relative)
  uint4* wo = reinterpret_cast<uint4*>(a.ws_o + row * SMLA_V_DIM + C * 256);
  const bool has = ok && ntiles > 0;
  if (has) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
    for (int cc = 0; cc < 8; ++cc) {
      uint32_t r[32];
      tmem_ld32(tmem_addr(tb, 32 * warp, kOCol + 32 * cc), r);
      tmem_ld_wait();
      if (live) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            w[q] = h2_bits(__floats2half2_rn(__uint_as_float(r[8 * k + 2 * q]) * inv,
                                             __uint_as_float(r[8 * k + 2 * q + 1]) * inv));
          wo[cc * 4 + k] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }
  float* ml = a.ws_ml + ((t * S + split) * 2 + C) * 2 * a.H;
  if (live) {
    ml[h] = has ? m_ref : -INFINITY;
    ml[a.H + h] = has ? l : 0.f;
  }
  if (!a.combine_in_kernel) {  // split_combine_kernel merges after this grid
    if (h == 0) ctl->is_last = 0;
    return;
  }
  __threadfence();
  named_bar_sync(2, 128);
  if (h == 0) ctl->is_last = (atomicAdd(a.ws_tick + t * 2 + C, 1) == S - 1);
}

// Split-K combine of one row's value half, run by all 384 threads of the CTA
// whose split arrived last, after the roles have finished (TMEM released,
// the peer no longer writing into this CTA's shared memory).  With m_s and
// l_s the splits' log2-domain maxima and sums, M = max m_s over the splits
// that hold a partial, L = sum l_s 2^(m_s - M), out = sum 2^(m_s - M) O_s / L
// and LSE = (M + log2 L) ln 2: the same split merge as across shards, here
// over the key ranges of one shard.
//
// A split holds a partial for every head or for none (a split with a valid
// key has l >= 1 for each head: its largest key contributes 2^0), so the
// non-empty splits are listed once, from head 0's sums.  Each thread owns
// fixed float4 columns of the output (a warp covers 512 contiguous bytes of
// one head row) and accumulates them over the listed splits with independent
// loads, 11 columns per pass, two passes; the per-(split, head) weights sit
// in the operand stages, per head M and 1 / L beside the exchange buffers.
// Splits are taken kCombChunk at a time.  The sums run in split order, as
// the per-head M and L do.
constexpr int kCombItems = 11;                                      // float4 columns per pass
constexpr int kCombChunk = (kStages * kOpTileBytes) / (128 * 4);  // splits whose weights fit
static_assert(2 * kCombItems * kThreads >= 128 * (SMLA_V_DIM / 2) / 4, "two passes cover a value half");
static_assert(kCombChunk * 4 + 1024 + 16 <= 2 * kXBytes, "split list and head stats fit");

__device__ void combine_splits(const DecodeArgs& a, uint8_t* sm, int C, int64_t t) {
  const int S = a.splits;
  const int H = a.H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  float* s_m = reinterpret_cast<float*>(sm + kOffX);  // per head: M
  float* s_inv = s_m + 128;                           // per head: 1 / L (0 when empty)
  int* s_n = reinterpret_cast<int*>(s_m + 256);       // listed splits in this chunk
  int* s_list = s_n + 4;                              // the non-empty splits of the chunk
  float* s_w = reinterpret_cast<float*>(sm + kOffOp); // [listed split][head] weights
  const float* ml_row = a.ws_ml + (t * S * 2 + C) * 2 * H;  // split sp at + sp * 4H
  __threadfence();
  if (tid < H) {
    const float* ms = ml_row + tid;
    float M = -INFINITY;
    int sp = 0;
    for (; sp + 8 <= S; sp += 8) {
      float m8[8], l8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        m8[k] = __ldcg(ms + int64_t(sp + k) * 4 * H);
        l8[k] = __ldcg(ms + int64_t(sp + k) * 4 * H + H);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (l8[k] != 0.f && (m8[k] > M || m8[k] != m8[k])) M = m8[k];  // NaN propagates
    }
    for (; sp < S; ++sp) {
      const float m1 = __ldcg(ms + int64_t(sp) * 4 * H), l1 = __ldcg(ms + int64_t(sp) * 4 * H + H);
      if (l1 != 0.f && (m1 > M || m1 != m1)) M = m1;
    }
    float L = 0.f;
    if (M != -INFINITY) {
      sp = 0;
      for (; sp + 8 <= S; sp += 8) {
        float m8[8], l8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          m8[k] = __ldcg(ms + int64_t(sp + k) * 4 * H);
          l8[k] = __ldcg(ms + int64_t(sp + k) * 4 * H + H);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k)
          if (l8[k] != 0.f) L += l8[k] * ex2(m8[k] - M);
      }
      for (; sp < S; ++sp) {
        const float l1 = __ldcg(ms + int64_t(sp) * 4 * H + H);
        if (l1 != 0.f) L += l1 * ex2(__ldcg(ms + int64_t(sp) * 4 * H) - M);
      }
    }
    s_m[tid] = M;
    s_inv[tid] = (M == -INFINITY) ? 0.f : 1.f / L;
    if (C == 0) a.lse[t * H + tid] = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * kLn2;
  }
  const int n_items = H * (SMLA_V_DIM / 2) / 4;  // float4 columns of the value half
  const int n_chunks = (S + kCombChunk - 1) / kCombChunk;
  const uint16_t* o_row = a.ws_o + t * S * H * SMLA_V_DIM + C * 256;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int it0 = pass * kCombItems * kThreads + tid;
    if (pass * kCombItems * kThreads >= n_items) break;  // uniform
    int32_t off[kCombItems];  // float offset of the column in a split's O rows (head = off / 512)
#pragma unroll
    for (int k = 0; k < kCombItems; ++k) {
      const int it = it0 + k * kThreads;
      const int itc = it < n_items ? it : 0;
      off[k] = (itc >> 6) * SMLA_V_DIM + (itc & 63) * 4;
    }
    float4 acc[kCombItems];
#pragma unroll
    for (int k = 0; k < kCombItems; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int ch = 0; ch < n_chunks; ++ch) {
      const int sp0 = ch * kCombChunk;
      if (pass == 0 || n_chunks > 1) {
        __syncthreads();  // head stats written; the previous chunk's list and weights consumed
        if (warp == 0) {
          // non-empty splits of the chunk, in split order
          const int sp_end = min(S, sp0 + kCombChunk);
          int cnt = 0;
          for (int sb = sp0; sb < sp_end; sb += 32) {
            const int sp = sb + lane;
            const bool ne = sp < sp_end && __ldcg(ml_row + int64_t(sp) * 4 * H + H) != 0.f;
            const unsigned m = __ballot_sync(0xffffffffu, ne);
            if (ne) s_list[cnt + __popc(m & ((1u << lane) - 1u))] = sp;
            cnt += __popc(m);
          }
          if (lane == 0) *s_n = cnt;
        }
        __syncthreads();
        const int n = *s_n;
        for (int idx = tid; idx < n * H; idx += kThreads) {
          const int j = idx / H;
          const int hh = idx - j * H;
          const float* p = ml_row + int64_t(s_list[j]) * 4 * H + hh;
          const float m1 = __ldcg(p), l1 = __ldcg(p + H);
          s_w[idx] = (l1 != 0.f) ? l1 * ex2(m1 - s_m[hh]) * s_inv[hh] : 0.f;
        }
        __syncthreads();
      }
      const int n = *s_n;
#pragma unroll 1
      for (int j = 0; j < n; ++j) {
        const uint16_t* src = o_row + int64_t(s_list[j]) * H * SMLA_V_DIM;
        const float* wj = s_w + j * H;
#pragma unroll
        for (int k = 0; k < kCombItems; ++k) {
          const uint2 raw = __ldcg(reinterpret_cast<const uint2*>(src + off[k]));
          const float2 v0 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
          const float2 v1 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
          const float w = wj[off[k] >> 9];
          acc[k].x = fmaf(w, v0.x, acc[k].x);
          acc[k].y = fmaf(w, v0.y, acc[k].y);
          acc[k].z = fmaf(w, v1.x, acc[k].z);
          acc[k].w = fmaf(w, v1.y, acc[k].w);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kCombItems; ++k) {
      const int it = it0 + k * kThreads;
      if (it < n_items) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x, acc[k].y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z, acc[k].w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&lo);
        o.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(a.out + (t * H + (it >> 6)) * SMLA_V_DIM + C * 256 + (it & 63) * 4) = o;
      }
    }
  }
  if (tid == 0) a.ws_tick[t * 2 + C] = 0;
}

// Store 8 q loads (64 dims) as fp16 pairs into 32 (or 16) TMEM columns.
__device__ __forceinline__ void q_store_group(const uint4* raw, uint32_t addr, bool full) {
  uint32_t qr[32];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint4 v = bf16x8_to_f16x8(raw[k]);
    qr[4 * k + 0] = v.x;
    qr[4 * k + 1] = v.y;
    qr[4 * k + 2] = v.z;
    qr[4 * k + 3] = v.w;
  }
  if (full)
    tmem_st32(addr, qr);
  else
    tmem_st16(addr, qr);  // trailing 32 dims
}

// q staging in the prologue, in the operand stages (idle until the tile
// loop): four 16 KB boxes of 64 latent dims x 128 head rows (128-byte
// swizzle) and one 8 KB box of 32 rope dims x 128 head rows (64-byte
// swizzle).
constexpr int kQLatBox = 128 * 128;
constexpr int kQBytes = 4 * kQLatBox + 128 * 64;
static_assert(kQBytes <= kStages * kOpTileBytes, "q staging fits the operand stages");

// Issue the TMA loads of this CTA's 288 q dims of token t (latent dims
// [256c, 256c + 256), rope dims [32c, 32c + 32)) for 128 head rows.
__device__ __forceinline__ void issue_q_tma(const DecodeArgs& a, int64_t t, int c, uint32_t dst,
                                            uint64_t* bar) {
  mbar_arrive_expect_tx(bar, kQBytes);
  const int32_t y = int32_t(t * a.H);
#pragma unroll
  for (int k = 0; k < 4; ++k) tma_load_2d(dst + k * kQLatBox, &a.q_lat, 256 * c + 64 * k, y, bar);
  tma_load_2d(dst + 4 * kQLatBox, &a.q_rope, 512 + 32 * c, y, bar);
}

// Convert head row h of the staged q into tensor memory as fp16 pairs (the
// A operand of QK^T), 64 dims per group of 32 columns; reads follow the
// boxes' swizzles, so 8 consecutive rows hit 8 different bank groups.
// Returns true when a q value of the row does not fit fp16 (the operand
// precision of QK^T).
__device__ bool q_to_tmem(uint32_t tb, int warp, int h, bool live, uint32_t src) {
  const uint32_t base = tmem_addr(tb, 32 * warp, kQCol);
  uint32_t over = 0;
#pragma unroll 1
  for (int grp = 0; grp < 5; ++grp) {
    uint4 g[8];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      uint32_t addr;
      if (grp < 4)
        addr = src + grp * kQLatBox + sw128_offset(h, v);
      else
        addr = src + 4 * kQLatBox + sw64_offset(h, v & 3);
      g[v] = (live && (grp < 4 || v < 4)) ? lds128(addr) : make_uint4(0, 0, 0, 0);
      over |= bf16x8_over_fp16(g[v]);
    }
    q_store_group(g, base + 32 * grp, grp < 4);
  }
  tmem_st_wait();
  return over != 0;
}

// MMA issue, fully unrolled: one thread issues a tcgen05.mma every few tens
// of cycles at best, and computing each descriptor in the loop about doubles
// that, which for the N = 64 QK^T steps is slower than the tensor core runs
// them.  A descriptor's start address field is the byte address / 16, so
// stepping through a stage adds a constant to the stage's base descriptor
// (shared-memory addresses stay below 256 KB: no carry leaves the field).
__device__ __forceinline__ void issue_qk(uint32_t tb, uint32_t op) {
  constexpr uint32_t idesc = idesc_f16_f32(128, kTileN, false, false);
  const uint64_t lat = sdesc_sw128(op, 16, 1024);
  const uint64_t rope = sdesc_sw64(op + kRopeBlock, 16, 512);
#pragma unroll
  for (int k = 0; k < kKSteps; ++k) {
    // 16 dims = 32 bytes of a row; a 128-byte swizzled K-block holds 64 dims
    const uint64_t bd = k < 16 ? lat + uint64_t((k >> 2) * (kKBlockBytes >> 4) + (k & 3) * 2)
                               : rope + uint64_t((k - 16) * 2);
    mma_ts(tb + kSCol, tb + kQCol + 8 * k, bd, idesc, k > 0);
  }
}

// PV of one tile: P (TMEM) x V, V = the operand stage read MN-major, 16 keys
// = 2048 bytes per step.
__device__ __forceinline__ void issue_pv(uint32_t tb, uint32_t op, bool accumulate) {
  constexpr uint32_t idesc = idesc_f16_f32(128, 256, false, true);
  const uint64_t v = sdesc_sw128(op, kKBlockBytes, 1024);
#pragma unroll
  for (int k = 0; k < kTileN / 16; ++k)
    mma_ts(tb + kOCol, tb + kPCol + 8 * k, v + uint64_t(k * (2048 >> 4)), idesc, accumulate || k > 0);
}

template <int kMode>
__device__ void run_cta(const DecodeArgs& a, uint8_t* sm, Ctl* ctl, const HalfRt& hr, int64_t t,
                        int split, uint32_t peer) {
  const int C = hr.c;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  volatile int* abort = &ctl->abort;
  const int n = ctl->n_list;
  const int ntiles = (n + kTileN - 1) / kTileN;
  const uint32_t tb = ctl->tbase;

  if (warp < 4) {
    // ------------------------------------------------ softmax + epilogue
    const int h = tid;  // head row == TMEM lane
    const float scale_log2 = a.sm_scale * kLog2e;
    float m_ref = -INFINITY;  // log2-domain reference maximum
    float l = 0.f;
    // Key-column split of the softmax: CTA c finishes the scores of keys
    // [32c, 32c + 32) of each tile (its own partial plus the peer's, XA),
    // computes their P against a reference maximum, and sends that P, the
    // reference and the partial sum to the peer (XB); P of all 64 keys then
    // sits in both CTAs.  Both sides move the shared reference R to the same
    // max(own reference, peer reference), so O, l and P stay consistent.
    // Buffers alternate by tile parity: the peer writes tile i into buffer
    // set i % 2 only after it has received this CTA's tile-i partial scores,
    // which this CTA sent after it had read tile i - 2 out of that set.
    const int oc0 = 32 * C;  // this CTA's key columns (the peer's: 32 (1 - C) ..)
    uint8_t* xbase = sm + kOffX;
    const uint32_t peer_x = map_to_cta(smem_u32(xbase), peer);
    const uint32_t peer_xa0 = map_to_cta(smem_u32(&ctl->xa[0]), peer);
    const uint32_t peer_xa1 = map_to_cta(smem_u32(&ctl->xa[1]), peer);
    const uint32_t peer_xb0 = map_to_cta(smem_u32(&ctl->xb[0]), peer);
    const uint32_t peer_xb1 = map_to_cta(smem_u32(&ctl->xb[1]), peer);
    if (h == 0) {
      for (int b = 0; b < 2 && b < ntiles; ++b) {
        mbar_arrive_expect_tx(&ctl->xa[b], kXABytes);
        mbar_arrive_expect_tx(&ctl->xb[b], kXBBytes);
      }
    }
    // The loop is software-pipelined across tiles: while the P of tile i is
    // in flight between the CTAs, the scores of tile i + 1 are read and the
    // peer's half of them sent, so the two exchanges of consecutive tiles
    // overlap.
    float sown[32];  // this CTA's partial scores of its own columns, next tile
    // Read tile t's partial scores (QK^T of tile t done), release S for the
    // next QK^T, send the peer's columns, keep this CTA's.
    auto start_tile = [&](int t) -> bool {
      if (!__all_sync(0xffffffffu, wait_bar(&ctl->s_full, t & 1, abort, kWsSFull))) return false;
      tc_fence_after();
      float s[64];
      {
        uint32_t r[32];
        tmem_ld32(tmem_addr(tb, 32 * warp, kSCol), r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) s[j] = __uint_as_float(r[j]);
        tmem_ld32(tmem_addr(tb, 32 * warp, kSCol + 32), r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) s[32 + j] = __uint_as_float(r[j]);
      }
      tc_fence_before();
      mbar_arrive(&ctl->s_free);
      const int b = t & 1;
      const uint32_t xa_p = peer_x + b * kXBytes;
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        // columns 32 (1 - C) + 4 j4 ..: a select between two static indices
        const int lo = 4 * j4, hi = 32 + 4 * j4;
        st_async_v4(xa_p + (j4 * 128 + h) * 16, C ? s[lo] : s[hi], C ? s[lo + 1] : s[hi + 1],
                    C ? s[lo + 2] : s[hi + 2], C ? s[lo + 3] : s[hi + 3], b ? peer_xa1 : peer_xa0);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) sown[j] = C ? s[32 + j] : s[j];
      return true;
    };
    // A warp whose wait gave up leaves the loop (at give_up below); the
    // others' waits give up too, since every wait is an mbarrier wait that
    // sees the CTA's abort flag.  The four warps enter the loop on one
    // reduced decision and meet again only at the epilogue's barrier.
    bool ok = ntiles == 0 || start_tile(0);
    ok = !named_bar_or(5, 128, !ok);
    int i = 0;
    for (; i < ntiles && ok; ++i) {
      const int b = i & 1;
      const uint32_t xa_l = smem_u32(xbase) + b * kXBytes;  // this CTA's buffer set b
      const uint32_t xa_p = peer_x + b * kXBytes;           // the peer's
      // 1) full scores of this CTA's columns of tile i
      ok = __all_sync(0xffffffffu, wait_bar_cluster(&ctl->xa[b], (i >> 1) & 1, abort, kWsExchange));
      if (!ok) goto give_up;
      float f[32];
#pragma unroll
      for (int j4 = 0; j4 < 8; ++j4) {
        const float4 v = ld_shared_f4(xa_l + (j4 * 128 + h) * 16);
        f[4 * j4] = sown[4 * j4] + v.x;
        f[4 * j4 + 1] = sown[4 * j4 + 1] + v.y;
        f[4 * j4 + 2] = sown[4 * j4 + 2] + v.z;
        f[4 * j4 + 3] = sown[4 * j4 + 3] + v.w;
      }
      if (h == 0 && i + 2 < ntiles) mbar_arrive_expect_tx(&ctl->xa[b], kXABytes);
      const int valid = min(kTileN, n - i * kTileN) - oc0;  // valid columns of this CTA's 32
      if (valid < 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = (j < valid) ? f[j] : -INFINITY;
      }
      float mq[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mq[k] = f[k];
#pragma unroll
      for (int j = 8; j < 32; ++j) mq[j & 7] = fmaxf(mq[j & 7], f[j]);
      const float mx = scale_log2 * fmaxf(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])),
                                          fmaxf(fmaxf(mq[4], mq[5]), fmaxf(mq[6], mq[7])));
      // 2) P of this CTA's columns against its reference (R, or its own
      //    maximum when that exceeds R by more than 2^8)
      const float my_ref = (mx > m_ref + 8.f) ? mx : m_ref;
      uint32_t pk[16];
      float l_part = 0.f;
      // P against reference `ref` (fp16 pairs, one rounding) and its sum;
      // nothing valid yet: zeros
      auto own_p = [&](float ref) {
        l_part = 0.f;
        if (ref == -INFINITY) {
#pragma unroll
          for (int j = 0; j < 16; ++j) pk[j] = 0u;
          return;
        }
        float sums[4] = {0.f, 0.f, 0.f, 0.f};
        const float neg_m = -ref;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float p0 = ex2(fmaf(f[2 * j], scale_log2, neg_m));
          const float p1 = ex2(fmaf(f[2 * j + 1], scale_log2, neg_m));
          sums[j & 3] += p0 + p1;
          pk[j] = h2_bits(__floats2half2_rn(p0, p1));
        }
        l_part = (sums[0] + sums[1]) + (sums[2] + sums[3]);
      };
      own_p(my_ref);
      // 3) P, reference and partial sum go to the peer
      const uint32_t xb_p = xa_p + kXABytes;
      const uint32_t xbb = b ? peer_xb1 : peer_xb0;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st_async_v4(xb_p + (q * 128 + h) * 16, __uint_as_float(pk[4 * q]),
                    __uint_as_float(pk[4 * q + 1]), __uint_as_float(pk[4 * q + 2]),
                    __uint_as_float(pk[4 * q + 3]), xbb);
      st_async_v2(xb_p + kXBPBytes + h * 8, my_ref, l_part, xbb);
      // 4) while that is in flight: tile i + 1's scores (its QK^T could start
      //    once S(i) was read)
      if (i + 1 < ntiles && !start_tile(i + 1)) goto give_up;
      // 5) the peer's P of tile i
      ok = __all_sync(0xffffffffu, wait_bar_cluster(&ctl->xb[b], (i >> 1) & 1, abort, kWsExchangeP));
      if (!ok) goto give_up;
      const uint32_t xb_l = xa_l + kXABytes;
      uint32_t pp[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = lds128(xb_l + (q * 128 + h) * 16);
        pp[4 * q] = v.x;
        pp[4 * q + 1] = v.y;
        pp[4 * q + 2] = v.z;
        pp[4 * q + 3] = v.w;
      }
      const float2 peer_rl = ld_shared_f2(xb_l + kXBPBytes + h * 8);
      if (h == 0 && i + 2 < ntiles) mbar_arrive_expect_tx(&ctl->xb[b], kXBBytes);
      // 6) the shared reference moves to the larger of the two (identically
      //    on both CTAs); what was computed against a smaller one is redone
      const float r_new = fmaxf(my_ref, peer_rl.x);
      float alpha = 1.f;  // O and l
      bool rescale = false;
      if (r_new != m_ref) {
        alpha = ex2(m_ref - r_new);  // 0 while nothing was valid yet
        rescale = (i > 0);
      }
      // own P against a smaller reference: recomputed from the fp32 scores
      // (one rounding); the peer's: scaled in fp32 and rounded once more
      if (my_ref != r_new) own_p(r_new);
      float l_peer = peer_rl.y;
      if (peer_rl.x != r_new) {
        const float fp = (peer_rl.x == -INFINITY) ? 0.f : ex2(peer_rl.x - r_new);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&pp[j]));
          pp[j] = h2_bits(__floats2half2_rn(v.x * fp, v.y * fp));
        }
        l_peer *= fp;
      }
      const float l_own = l_part;
      m_ref = r_new;
      // the same sum on both CTAs: keys 0..31 first, then 32..63
      l = l * alpha + (C ? l_peer + l_own : l_own + l_peer);
      if (i > 0) {
        ok = __all_sync(0xffffffffu, wait_bar(&ctl->pv_done, (i - 1) & 1, abort, kWsPvDone));
        if (!ok) goto give_up;
        tc_fence_after();
      }
      // P(i) replaces P(i-1), which PV(i-1) has finished reading: keys
      // 0..31 in columns 0..15, keys 32..63 in columns 16..31
      tmem_st16(tmem_addr(tb, 32 * warp, kPCol + 16 * C), pk);
      tmem_st16(tmem_addr(tb, 32 * warp, kPCol + 16 * (1 - C)), pp);
      if (i > 0) {
        // tcgen05.ld/st are warp-collective: the warp rescales together when
        // any of its rows needs it, each lane by its own factor (1 if none)
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t r[32];
            const uint32_t addr = tmem_addr(tb, 32 * warp, kOCol + 32 * cc);
            tmem_ld32(addr, r);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) r[jj] = __float_as_uint(__uint_as_float(r[jj]) * alpha);
            tmem_st32(addr, r);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      // this thread's row of P(i) is in TMEM: once all 128 have arrived the
      // MMA thread issues PV(i); its completion releases the operand stage
      // and lets the next P overwrite this one
      mbar_arrive(&ctl->p_full);
    }
    if (false) {
    give_up:
      // this warp's wait gave up (the CTA's abort flag is up, so every
      // other wait of the CTA gives up too)
      ok = false;
    }
    // epilogue
    if (ok && ntiles > 0) {
      ok = __all_sync(0xffffffffu, wait_bar(&ctl->pv_done, (ntiles - 1) & 1, abort, kWsPvLast));
      tc_fence_after();
    }
    // one decision for all four softmax warps (the split epilogue below uses a
    // 128-thread named barrier)
    ok = !named_bar_or(4, 128, !ok);
    if (a.splits > 1) {
      split_epilogue(a, ctl, C, t, split, ntiles, m_ref, l, tb, warp, h, ok);
    } else if (ok) {
      // tcgen05.ld is warp-collective: every lane loads, only live heads store
      const bool live = h < a.H;
      uint4* dst = reinterpret_cast<uint4*>(a.out + (t * a.H + (live ? h : 0)) * SMLA_V_DIM +
                                            C * 256);
      if (ntiles == 0) {
        if (live) {
#pragma unroll 1
          for (int k = 0; k < 32; ++k) dst[k] = make_uint4(0, 0, 0, 0);
        }
      } else {
        const float inv = 1.f / l;
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem_addr(tb, 32 * warp, kOCol + 32 * cc), r);
          tmem_ld_wait();
          uint32_t o[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[2 * j]) * inv,
                                                     __uint_as_float(r[2 * j + 1]) * inv);
            o[j] = *reinterpret_cast<uint32_t*>(&v);
          }
          if (live) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[cc * 4 + k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
          }
        }
      }
      if (C == 0 && live)
        a.lse[t * a.H + h] = (ntiles == 0) ? -INFINITY : (m_ref + log2f(l)) * kLn2;
    }
  } else if (warp < 8) {
    // ------------------------------------------------ dequantise
    // Converter d owns key d % 64 of every tile and half d / 64 of its
    // pieces, so each warp stores 32 consecutive rows of one chunk column
    // (conflict-free under the 128-byte swizzle).
    const int d = tid - 128;
    convert_loop(ctl, sm, n, ntiles, d & (kTileN - 1), C, d >> 6, lane, abort);
  } else if (warp >= kLoaderWarp0) {
    // ------------------------------------------------ stage cache rows
    loader_loop<kMode>(a, ctl, sm, n, ntiles, C, tid - 32 * kLoaderWarp0, abort);
  } else if (lane == 0) {
    // ------------------------------------------------ MMA issue (one thread)
    // QK(i) needs its operand stage converted and S(i - 1) read by the
    // softmax, PV(i) the softmax's P(i); the thread sleeps on each barrier
    // until the hardware wakes it at the phase change.  Issuing PV here
    // rather than from a softmax thread keeps the MMA issue (~57 cycles an
    // instruction) and a per-tile barrier of the four softmax warps off the
    // softmax's chain.
    const uint32_t op0 = smem_u32(sm + kOffOp);
    bool ok = wait_bar(&ctl->q_ready, 0, abort, kWsQReady);
    // QK(j), then PV(j - 2): the softmax stores P(j - 2) after it has read
    // S(j - 1), which frees S for QK(j)
#pragma unroll 1
    for (int j = 0; j < ntiles + 2 && ok; ++j) {
      if (j < ntiles) {
        ok = wait_bar(&ctl->full[j % kStages], (j / kStages) & 1, abort, kWsFull) &&
             (j == 0 || wait_bar(&ctl->s_free, (j - 1) & 1, abort, kWsSFree));
        if (!ok) break;
        tc_fence_after();
        issue_qk(tb, op0 + (j % kStages) * kOpTileBytes);
        mma_commit(&ctl->s_full);
      }
      const int i = j - 2;
      if (i >= 0) {
        ok = wait_bar(&ctl->p_full, i & 1, abort, kWsPFull);
        if (!ok) break;
        tc_fence_after();
        issue_pv(tb, op0 + (i % kStages) * kOpTileBytes, i > 0);
        mma_commit(&ctl->pv_done);
        mma_commit(&ctl->freed[i % kStages]);
      }
    }
    // drain: every MMA issued above has completed before TMEM is released
    // (waited on even after an abort, with its own bound).  A CTA whose row
    // has no valid slot issued no MMA and has nothing to drain.
    if (ntiles > 0) {
      mma_commit(&ctl->end);
      int no_abort = 0;
      wait_bar(&ctl->end, 0, &no_abort, kWsDrain);
    }
  }
}

// Resolve raw entry v to (slot, shard).  Per-shard launch: the entry
// already is a local slot.  Fused DCP step and merged dense decode: the
// entry is a global position v; with interleave size I, runs of I positions
// go to the shards in turn, so v is owned by shard (v div I) mod D at local
// position (v div (I D)) I + v mod I (I = 1: shard v mod D, position
// v div D).  Dense decode of one rank: the entry is that rank's local
// position itself.  The local position then goes through that shard's
// block-table row for this request (staged in shared memory at `bt` when it
// fits, else read from global memory).  `limit` bounds the valid entries of
// a dense row (its last position + 1, or the rank's count of them).  Returns
// false for -1 / foreign / invalid entries, recording input errors in `err`.
template <int kMode>
__device__ __forceinline__ bool resolve_entry(const DecodeArgs& a, const Ctl* ctl, const int32_t* bt,
                                              bool staged, bool req_ok, int32_t limit, int32_t v,
                                              int32_t& slot, int& shard, unsigned& err) {
  if (kMode == kModeSlots) {
    if (v >= a.num_slots) {
      err |= SMLA_DEVERR_SLOT_RANGE;
      return false;
    }
    slot = v;
    shard = 0;
    return v >= 0;
  }
  // Pools: every entry takes the same straight-line path (no branch per
  // check), so the 16 entries of a thread overlap their shared-memory reads.
  const bool live = v >= 0 && req_ok && !(kMode == kModeDense && v >= limit);
  const int32_t vv = live ? v : 0;
  int d;
  int32_t lp;
  if (kMode == kModeDense && a.dense_rank >= 0) {
    d = a.dense_rank;
    lp = vv;
  } else {
    const uint32_t g = fastdiv(uint32_t(vv), a.div_I);  // run of I positions
    const uint32_t round = fastdiv(g, a.div_D);         // round of D runs
    d = int(g - round * uint32_t(a.D));
    lp = int32_t(round) * a.interleave + (vv - int32_t(g) * a.interleave);
  }
  const ShardMeta m = ctl->meta[d];
  const int32_t col = int32_t(fastdiv(uint32_t(lp), a.div_bs));
  const bool in_table = col < m.bt_width;
  const int32_t colc = in_table ? col : 0;  // every table has a column 0
  const int32_t blk = staged ? bt[m.bt_off + colc] : __ldg(ctl->bt_row[d] + colc);
  const int64_t s64 = int64_t(blk) * a.block_size + (lp - col * a.block_size);
  const bool in_pool = s64 < m.pool_slots;
  err |= (live && (!in_table || blk < 0)) ? unsigned(SMLA_DEVERR_BLOCK_TABLE) : 0u;
  err |= (live && in_table && blk >= 0 && !in_pool) ? unsigned(SMLA_DEVERR_SLOT_RANGE) : 0u;
  slot = int32_t(s64);
  shard = d;
  return live && in_table && blk >= 0 && in_pool;
}

// Dense decode: the request of row t and the bound on its raw entries (its
// own position + 1 in the merged form, that many positions' share of one
// rank in the per-rank form); false for every row of a request (and an error
// bit) when the request's context is shorter than its query tokens or runs
// past the raw range.
__device__ __forceinline__ bool dense_row(const DecodeArgs& a, int64_t t, int32_t& req,
                                          int32_t& limit, unsigned& err) {
  req = int32_t(t / a.S);
  const int32_t ctx = a.ctx_lens[req];
  if (ctx < a.S || ctx > a.max_ctx) {  // the request's query tokens are part of its context
    err |= SMLA_DEVERR_CONTEXT;
    limit = 0;
    return false;
  }
  const int32_t n = ctx - a.S + int32_t(t - int64_t(req) * a.S) + 1;  // positions 0..n-1
  if (a.dense_rank < 0) {
    limit = n;
  } else {
    // whole rounds of I*D positions give I each, then the partial round
    const int32_t ID = a.interleave * a.D;
    const int32_t full = n / ID, rem = n - full * ID;
    limit = full * a.interleave + min(max(rem - a.dense_rank * a.interleave, 0), a.interleave);
  }
  return true;
}

// A dense split with no position of its row (a short context under a long
// max_ctx) skips the set-up and publishes what the full path would: the
// row's (0, -inf) half without split-K, else an empty partial (-inf, 0)
// that counts in like any other split.  Both CTAs of the pair take this path
// together (the test depends only on the row and the split); it touches no
// tensor memory and no peer shared memory.
__device__ void publish_empty_split(const DecodeArgs& a, uint8_t* sm, Ctl* ctl, int64_t t, int split,
                                    int C) {
  const int tid = threadIdx.x;
  if (a.splits == 1) {
    for (int idx = tid; idx < a.H * 32; idx += kThreads) {  // 32 x 16 bytes per head half
      uint4* dst = reinterpret_cast<uint4*>(a.out + (t * a.H + (idx >> 5)) * SMLA_V_DIM + C * 256);
      dst[idx & 31] = make_uint4(0, 0, 0, 0);
    }
    if (C == 0)
      for (int h = tid; h < a.H; h += kThreads) a.lse[t * a.H + h] = -INFINITY;
    return;
  }
  float* ml = a.ws_ml + ((t * a.splits + split) * 2 + C) * 2 * a.H;
  for (int h = tid; h < a.H; h += kThreads) {
    ml[h] = -INFINITY;
    ml[a.H + h] = 0.f;
  }
  if (!a.combine_in_kernel) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) ctl->is_last = (atomicAdd(a.ws_tick + t * 2 + C, 1) == a.splits - 1);
  __syncthreads();
  if (ctl->is_last) combine_splits(a, sm, C, t);
}

template <int kMode>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    sparse_mla_decode_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr bool kPools = kMode != kModeSlots;  // entries resolve through D pools
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(sm + kOffCtl);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t c = cluster_ctarank();
  const uint32_t peer = c ^ 1u;
  const int64_t item = blockIdx.x >> 1;
  const int64_t t = item / a.splits;
  const int split = int(item - t * a.splits);
  const int per_split = (a.K + a.splits - 1) / a.splits;
  const int e_begin = split * per_split;
  const int e_end = min(a.K, e_begin + per_split);

  const HalfRt hr = half_of(c);
  // a separate split combine (if any) may be scheduled on SMs this grid
  // leaves idle
  griddep_launch_dependents();
  if (kMode == kModeDense) {
    int32_t r, limit = 0;
    unsigned e2 = 0;
    const bool row_ok = dense_row(a, t, r, limit, e2);
    if (!row_ok || min(e_end, limit) <= e_begin) {
      if (tid == 0 && e2) atomicOr(&g_decode_error, e2);
      publish_empty_split(a, sm, ctl, t, split, hr.c);
      return;
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tbase, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&ctl->q_tma, 1);
    mbar_init(&ctl->q_ready, 128);
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&ctl->full[st], 128);
      mbar_init(&ctl->freed[st], 1);
    }
    mbar_init(&ctl->s_full, 1);
    mbar_init(&ctl->s_free, 128);
    mbar_init(&ctl->pv_done, 1);
    mbar_init(&ctl->p_full, 128);  // one arrival per softmax thread
    for (int st = 0; st < kRawStages; ++st) {
      mbar_init(&ctl->raw_full[st], kLoaders);  // one arrival per loader
      mbar_init(&ctl->raw_empty[st], 4);        // one arrival per converter warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->xa[b], 1);  // one expect_tx arrival per phase
      mbar_init(&ctl->xb[b], 1);
    }
    mbar_init(&ctl->end, 1);
    ctl->abort = 0;
    fence_mbar_init_cluster();
    // q lands in the (still idle) operand stages while the CTA sets up
    issue_q_tma(a, t, hr.c, smem_u32(sm + kOffOp), &ctl->q_tma);
  }
  // The compacting warps' raw entries (kPer each of the row's split, see the
  // compaction below) are loaded before the set-up barrier, so that their
  // memory round trip overlaps the request id's.
  constexpr int kListThreads = kThreads - 128;  // every warp but the softmax warps
  constexpr int kPer = kMaxList / kListThreads;
  int32_t vs[kPer];
  if (kMode != kModeDense && warp >= 4) {
    const int j0 = e_begin + (tid - 128) * kPer;
    const int32_t* src = (kMode == kModeTopk ? a.topk : a.slots) + t * a.K;
    if (j0 + kPer <= e_end && (reinterpret_cast<uintptr_t>(src + j0) & 15u) == 0) {
#pragma unroll
      for (int q4 = 0; q4 < kPer / 4; ++q4) {
        const int4 w = __ldg(reinterpret_cast<const int4*>(src + j0) + q4);
        vs[4 * q4] = w.x;
        vs[4 * q4 + 1] = w.y;
        vs[4 * q4 + 2] = w.z;
        vs[4 * q4 + 3] = w.w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < kPer; ++k) vs[k] = (j0 + k < e_end) ? __ldg(src + j0 + k) : -1;
    }
  }
  if (kPools && tid < a.D) {
    // per-shard pointers of this row's request, read once
    const int32_t r = kMode == kModeDense ? int32_t(t / a.S) : a.req_id[t];
    const bool ok = r >= 0 && r < a.num_reqs;
    ctl->pool[tid] = a.pools[tid];
    ctl->bt_row[tid] = a.bts[tid] + (ok ? int64_t(r) * a.bt_stride[tid] : 0);
  }
  if (kPools && tid == 0) {
    // the request's block-table rows of all shards, staged in the exchange
    // buffers (idle until the tile loop) when they fit
    int off = 0;
    for (int d = 0; d < a.D; ++d) {
      ctl->meta[d].bt_off = off;
      ctl->meta[d].bt_width = a.bt_width[d];
      ctl->meta[d].pool_slots = a.pool_slots[d];
      off += a.bt_width[d];
    }
    ctl->bt_staged = off <= kBtStageMax;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp < 4) {
    // Q half -> TMEM, overlapping the compaction below
    // the whole q tile landed (issued by thread 0 before the set-up barrier)
    bool qok = wait_bar(&ctl->q_tma, 0, &ctl->abort, kWsQReady);
    if (q_to_tmem(ctl->tbase, warp, tid, qok && tid < a.H, smem_u32(sm + kOffOp)))
      atomicOr(&g_decode_error, SMLA_DEVERR_RANGE);
    tc_fence_before();
    mbar_arrive(&ctl->q_ready);
  } else {
    // Ordered compaction of the split's valid entries by the 256 threads of
    // warps 4-11 (idle until the tile loop): thread d owns the contiguous
    // entries [e_begin + 8d, e_begin + 8d + 8), resolves them with all loads
    // in flight at once, and a block scan gives each thread its output
    // offset.  Both CTAs of the pair build the same list, so their tiles hold
    // the same keys.
    const int d = tid - 128;
    int* list = reinterpret_cast<int*>(sm + kOffList);
    uint8_t* list_shard = sm + kOffListShard;
    unsigned err = 0;
    bool req_ok = true;
    int32_t limit = 0;
    if (kMode == kModeTopk) {
      const int32_t r = a.req_id[t];
      req_ok = r >= 0 && r < a.num_reqs;
      if (!req_ok && d == 0) err |= SMLA_DEVERR_REQ_ID;
    } else if (kMode == kModeDense) {
      int32_t r;
      unsigned e2 = 0;
      req_ok = dense_row(a, t, r, limit, e2);
      if (d == 0) err |= e2;
    }
    // 1) this thread's kPer raw entries (loaded before the set-up barrier,
    //    four 16-byte loads when the row allows; a dense row's entries are
    //    just their indices), and, with D pools, the request's block-table
    //    rows copied into shared memory by all the compacting threads
    const int j0 = e_begin + d * kPer;
    if (kMode == kModeDense) {
#pragma unroll
      for (int k = 0; k < kPer; ++k) vs[k] = j0 + k;
    }
    int32_t* bt = reinterpret_cast<int32_t*>(sm + kOffX);
    const bool staged = kPools && ctl->bt_staged;
    if (staged) {
      const uint32_t bt0 = smem_u32(bt);
#pragma unroll 1
      for (int sd = 0; sd < a.D; ++sd) {
#pragma unroll 1
        for (int col = d; col < ctl->meta[sd].bt_width; col += kListThreads)
          cp_async_4(bt0 + 4u * uint32_t(ctl->meta[sd].bt_off + col), ctl->bt_row[sd] + col);
      }
      cp_async_commit();
      cp_async_wait<0>();
      named_bar_sync(3, kListThreads);  // every thread's copies are visible
    }
    // 2) resolve the 16 entries from registers and shared memory
    int shards[kPer];
    unsigned keep = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int32_t v = vs[k];
      vs[k] = -1;
      shards[k] = 0;
      const bool ok = resolve_entry<kMode>(a, ctl, bt, staged, req_ok, limit,
                                           j0 + k < e_end ? v : -1, vs[k], shards[k], err);
      keep |= unsigned(ok) << k;
    }
    const int cnt = __popc(keep);
    int incl = cnt;  // inclusive warp scan
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) ctl->warp_cnt[warp - 4] = incl;
    named_bar_sync(3, kListThreads);
    int wbase = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kListThreads / 32; ++w) {
      const int x = ctl->warp_cnt[w];
      wbase += (w < warp - 4) ? x : 0;
      total += x;
    }
    int pos = wbase + incl - cnt;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      if (keep & (1u << k)) {
        list[pos] = vs[k];
        list_shard[pos] = uint8_t(shards[k]);
        ++pos;
      }
    }
    if (d == 0) ctl->n_list = total;
    if (err) atomicOr(&g_decode_error, err);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // peer barriers initialised before any remote arrive
  tc_fence_after();

  run_cta<kMode>(a, sm, ctl, hr, t, split, peer);

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer no longer writes into this CTA's shared memory
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(ctl->tbase, kTmemCols);
  }
  if (a.splits > 1 && ctl->is_last) combine_splits(a, sm, hr.c, t);
}

// Split-K combine of one row's value half for eight heads, one warp per
// head, launched after the decode grid with programmatic stream
// serialisation.  With m_s and l_s the splits' log2-domain maxima and sums,
// M = max m_s over the splits that hold a partial (l_s != 0), L = sum l_s
// 2^(m_s - M), out = sum_s 2^(m_s - M) O_s / L, LSE = (M + log2 L) ln 2: the
// merge of "partial attention results" by their LSE, here over the key ranges
// of one row.  A row whose splits all hold nothing comes out as the merge
// identity (0, -inf).  Lanes own float4 columns lane and lane + 32 of the
// head's value half (two 512-byte coalesced reads per split) and take the
// splits in ascending order, eight at a time, each load independent.
constexpr int kCombHeads = 8;

__device__ __forceinline__ float max_nan(float x, float y) {
  return (x != x || y != y) ? __int_as_float(0x7fc00000) : fmaxf(x, y);
}

__global__ void __launch_bounds__(kCombHeads * 32)
    split_combine_kernel(const uint16_t* __restrict__ ws_o, const float* __restrict__ ws_ml,
                         uint16_t* __restrict__ out, float* __restrict__ lse, int32_t H, int32_t S) {
  griddep_wait();  // the decode grid's partials are complete and visible
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = (H + kCombHeads - 1) / kCombHeads;
  const int64_t t = blockIdx.x / (2 * G);
  const int r = int(blockIdx.x - t * 2 * G);
  const int C = r / G;
  const int h = (r - C * G) * kCombHeads + warp;
  if (h >= H) return;
  const int64_t ml_stride = 4 * int64_t(H);  // floats from one split's stats to the next
  const float* ml = ws_ml + (t * S * 2 + C) * 2 * int64_t(H) + h;  // split sp: m at sp * 4H, l at + H
  float M = -INFINITY;
  for (int sp = lane; sp < S; sp += 32) {
    const float m1 = __ldcg(ml + sp * ml_stride), l1 = __ldcg(ml + sp * ml_stride + H);
    if (l1 != 0.f) M = max_nan(M, m1);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = max_nan(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
  if (M != -INFINITY) {
    for (int sp = lane; sp < S; sp += 32) {
      const float m1 = __ldcg(ml + sp * ml_stride), l1 = __ldcg(ml + sp * ml_stride + H);
      if (l1 != 0.f) L += l1 * ex2(m1 - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  }
  const float inv = (M == -INFINITY) ? 0.f : 1.f / L;
  const uint2* o_row =
      reinterpret_cast<const uint2*>(ws_o + (t * S * H + h) * SMLA_V_DIM + C * 256) + lane;
  const int64_t o_stride = int64_t(H) * SMLA_V_DIM / 4;  // 4-value groups from one split's row to the next
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
  for (int base = 0; base < S; base += 32) {
    const int sp = base + lane;
    float m1 = 0.f, l1 = 0.f;
    if (sp < S) {
      m1 = __ldcg(ml + sp * ml_stride);
      l1 = __ldcg(ml + sp * ml_stride + H);
    }
    const bool held = l1 != 0.f;  // this split wrote its partial
    const float w_lane = held ? l1 * ex2(m1 - M) * inv : 0.f;
    unsigned mask = __ballot_sync(0xffffffffu, held);
    while (mask) {
      int idx[8];
      float w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        idx[k] = mask ? __ffs(mask) - 1 : -1;
        w[k] = __shfl_sync(0xffffffffu, w_lane, idx[k] < 0 ? 0 : idx[k]);
        mask &= mask - 1u;
      }
      float4 v0[8], v1[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint2* src = o_row + (base + (idx[k] < 0 ? idx[0] : idx[k])) * o_stride;
        const uint2 r0 = __ldcg(src), r1 = __ldcg(src + 32);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&r0.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&r0.y));
        const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&r1.x));
        const float2 d = __half22float2(*reinterpret_cast<const __half2*>(&r1.y));
        v0[k] = make_float4(a.x, a.y, b.x, b.y);
        v1[k] = make_float4(c.x, c.y, d.x, d.y);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (idx[k] >= 0) {
          a0.x = fmaf(w[k], v0[k].x, a0.x);
          a0.y = fmaf(w[k], v0[k].y, a0.y);
          a0.z = fmaf(w[k], v0[k].z, a0.z);
          a0.w = fmaf(w[k], v0[k].w, a0.w);
          a1.x = fmaf(w[k], v1[k].x, a1.x);
          a1.y = fmaf(w[k], v1[k].y, a1.y);
          a1.z = fmaf(w[k], v1[k].z, a1.z);
          a1.w = fmaf(w[k], v1[k].w, a1.w);
        }
      }
    }
  }
  auto pack = [](float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    return make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  };
  uint2* dst = reinterpret_cast<uint2*>(out + (t * H + h) * SMLA_V_DIM + C * 256) + lane;
  dst[0] = pack(a0);
  dst[32] = pack(a1);
  if (C == 0 && lane == 0) lse[t * H + h] = (M == -INFINITY) ? -INFINITY : (M + log2f(L)) * kLn2;
}

// Which combine merges a row's splits.  The in-kernel one overlaps the CTAs
// still running, but one CTA reads every split's partial with a bounded
// number of loads in flight (two rounds of loads per split); the separate
// kernel spreads the reads over (row, half, 8 heads) CTAs for a fixed cost
// (its launch and the wait for this grid to drain).  So the separate kernel
// is taken when the decode grid fits in one wave on the GPU's SMs, whose
// other SMs then sit idle, and there are at least four splits per row.
bool combine_in_kernel(int64_t decode_ctas, int splits, int sms) {
  return decode_ctas > sms || splits < 4;
}

// Split-K policy, a function of the shape alone: enough clusters to cover the
// GB300's 76 SM pairs when there are few query rows, at least 256 top-k
// entries per split, and at most kMaxList entries per split.
constexpr int kClusterSlots = 76;

int decode_splits(int32_t T, int32_t K) {
  int s = (T > 0) ? kClusterSlots / T : 1;
  s = min(s, (K + 255) / 256);
  s = max(s, (K + kMaxList - 1) / kMaxList);
  return max(s, 1);
}

struct WsLayout {
  size_t o_off, ml_off, tick_off, total;
};

WsLayout ws_layout(int32_t T, int32_t H, int32_t K) {
  WsLayout w{0, 0, 0, 0};
  const int S = decode_splits(T, K);
  if (S == 1 || T <= 0) return w;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  w.o_off = 0;
  w.ml_off = up(size_t(T) * S * H * SMLA_V_DIM * sizeof(uint16_t));
  w.tick_off = w.ml_off + up(size_t(T) * S * 2 * 2 * H * sizeof(float));
  w.total = w.tick_off + up(size_t(T) * 2 * sizeof(int32_t));
  return w;
}

}  // namespace

size_t decode_workspace_bytes(int32_t T, int32_t H, int32_t K) {
  return ws_layout(T, H, K).total;
}

namespace {

// cuTensorMapEncodeTiled, looked up once through the runtime (no link-time
// dependency on the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t encode_tiled_fn(EncodeTiledFn* fn) {
  static std::mutex m;
  static EncodeTiledFn cached = nullptr;
  std::lock_guard<std::mutex> lock(m);
  if (cached == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || p == nullptr) return cudaErrorNotSupported;
    cached = reinterpret_cast<EncodeTiledFn>(p);
  }
  *fn = cached;
  return cudaSuccess;
}

// Tensor maps over q viewed as [T*H rows, 576] bf16: boxes of 64 dims x 128
// rows with 128-byte swizzle, and 32 dims x 128 rows with 64-byte swizzle.
// Rows past T*H read as zeros.
cudaError_t encode_q_maps(DecodeArgs& a) {
  EncodeTiledFn enc = nullptr;
  cudaError_t e = encode_tiled_fn(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {SMLA_QK_DIM, cuuint64_t(a.T) * cuuint64_t(a.H)};
  const cuuint64_t strides[1] = {SMLA_QK_DIM * sizeof(uint16_t)};
  const cuuint32_t box_lat[2] = {64, 128}, box_rope[2] = {32, 128}, ones[2] = {1, 1};
  void* q = const_cast<uint16_t*>(a.q);
  if (enc(&a.q_lat, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, dims, strides, box_lat, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      enc(&a.q_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q, dims, strides, box_rope, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return cudaSuccess;
}

// The kernels' shared-memory size attribute, set once per device and kernel,
// safe when several host threads make their first launch at once.
constexpr int kMaxDevices = 64;

template <int kMode>
cudaError_t ensure_smem_attribute(int dev) {
  static std::atomic<bool> done[kMaxDevices];
  static std::mutex m;
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  if (tracked && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(m);
  if (tracked && done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(sparse_mla_decode_kernel<kMode>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess && tracked) done[dev].store(true, std::memory_order_release);
  return e;
}

template <int kMode>
cudaError_t launch_impl(const DecodeArgs& args, cudaStream_t s) {
  DecodeArgs a = args;
  {
    const cudaError_t e = encode_q_maps(a);
    if (e != cudaSuccess) return e;
  }
  a.splits = a.single_split ? 1 : decode_splits(a.T, a.K);
  const WsLayout w = a.splits > 1 ? ws_layout(a.T, a.H, a.K) : WsLayout{0, 0, 0, 0};
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  a.ws_o = w.total ? reinterpret_cast<uint16_t*>(ws + w.o_off) : nullptr;
  a.ws_ml = w.total ? reinterpret_cast<float*>(ws + w.ml_off) : nullptr;
  a.ws_tick = w.total ? reinterpret_cast<int32_t*>(ws + w.tick_off) : nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = ensure_smem_attribute<kMode>(dev);
  if (e != cudaSuccess) return e;
  const int64_t ctas = 2 * int64_t(a.T) * a.splits;
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  a.combine_in_kernel = combine_in_kernel(ctas, a.splits, sms) ? 1 : 0;
  sparse_mla_decode_kernel<kMode><<<dim3(unsigned(ctas)), dim3(kThreads), kSmemBytes, s>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1 || a.T == 0 || a.combine_in_kernel) return e;
  // the separate split combine, scheduled while the decode grid drains
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(int64_t(a.T) * 2 * ((a.H + kCombHeads - 1) / kCombHeads)));
  cfg.blockDim = dim3(kCombHeads * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_combine_kernel, static_cast<const uint16_t*>(a.ws_o),
                            static_cast<const float*>(a.ws_ml), a.out, a.lse, a.H, a.splits);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
  return launch_impl<kModeSlots>(a, s);
}

cudaError_t launch_decode_fused(const DecodeArgs& args, cudaStream_t s) {
  DecodeArgs a = args;
  a.div_I = make_fastdiv(uint32_t(a.interleave));
  a.div_D = make_fastdiv(uint32_t(a.D));
  a.div_bs = make_fastdiv(uint32_t(a.block_size));
  return launch_impl<kModeTopk>(a, s);
}

cudaError_t launch_decode_dense(const DecodeArgs& args, cudaStream_t s) {
  DecodeArgs a = args;
  a.div_I = make_fastdiv(uint32_t(a.interleave));
  a.div_D = make_fastdiv(uint32_t(a.D));
  a.div_bs = make_fastdiv(uint32_t(a.block_size));
  return launch_impl<kModeDense>(a, s);
}

// ---------------------------------------------------------------------------
// Decode with library-owned scratch, for callers that cannot allocate device
// memory themselves.  The split-K scratch lives in this file-scope array; every
// GPU that loads the library holds it until the process exits.  Host code
// must not pass the array's name to a kernel (on the host it names a stand-in,
// not device memory): its device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call there.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

cudaError_t noalloc_scratch_ptr(void** ptr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  *ptr = g_noalloc_ptr[dev];
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_decode_noalloc(const DecodeArgs& args, cudaStream_t s) {
  const WsLayout w = ws_layout(args.T, args.H, args.K);
  if (w.total > kNoAllocScratchBytes) return cudaErrorInvalidValue;  // caller checks first
  DecodeArgs a = args;
  a.workspace = nullptr;
  a.workspace_bytes = 0;
  if (w.total > 0) {
    void* scratch = nullptr;
    cudaError_t e = noalloc_scratch_ptr(&scratch);
    if (e != cudaSuccess) return e;
    // the arrival counters must start at zero; a call that gave up part-way
    // could have left them otherwise
    e = cudaMemsetAsync(static_cast<uint8_t*>(scratch) + w.tick_off, 0, w.total - w.tick_off, s);
    if (e != cudaSuccess) return e;
    a.workspace = scratch;
    a.workspace_bytes = w.total;
  }
  return launch_impl<kModeSlots>(a, s);
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
