// The fused DCP step from and to host memory: row groups whose copies in,
// decode and copies out form a pipeline across library-owned streams.
//
// One decode launch of T rows takes about as long as its longest row (each
// row is one cluster's serial chain of key tiles), so cutting the rows into
// G groups and launching each group as soon as its q rows and top-k ids have
// landed lets the copies of later groups overlap the decode of earlier ones;
// each group's out and lse rows go back as soon as its decode ends.  The
// groups decode without split-K so that they run side by side on their own
// SM pairs instead of queueing behind one another.
//
// Per device the library keeps a stream per group, a copy-out stream and the
// events that order them, created on the device's first call.  A mutex serialises the calls: the events are shared, and two
// calls in flight on the same staging buffers would race anyway.
#include <mutex>

#include "../../include/smla.h"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int kHostMaxGroups = SMLA_MAX_HOST_CHUNKS;
constexpr int kHostMaxDevices = 64;

struct HostPipe {
  bool ready = false;
  cudaStream_t out = nullptr, group[kHostMaxGroups] = {};
  cudaEvent_t done = nullptr, landed[kHostMaxGroups] = {}, decoded[kHostMaxGroups] = {};
};

std::mutex g_host_mutex;
HostPipe g_host_pipe[kHostMaxDevices];

cudaError_t make_pipe(HostPipe& p) {
  if (p.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
  for (int g = 0; g < kHostMaxGroups && e == cudaSuccess; ++g)
    e = cudaStreamCreateWithFlags(&p.group[g], cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.done, cudaEventDisableTiming);
  for (int g = 0; g < kHostMaxGroups && e == cudaSuccess; ++g) {
    e = cudaEventCreateWithFlags(&p.landed[g], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.decoded[g], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) p.ready = true;  // a partial set is retried (and leaked) next time
  return e;
}

}  // namespace

cudaError_t launch_fused_host(const DecodeArgs& args, const HostBuffers& h, int groups,
                              cudaStream_t s) {
  const int64_t T = args.T, H = args.H, K = args.K;
  const size_t q_row = size_t(H) * SMLA_QK_DIM * sizeof(uint16_t);
  const size_t o_row = size_t(H) * SMLA_V_DIM * sizeof(uint16_t);
  const size_t l_row = size_t(H) * sizeof(float);
  const size_t k_row = size_t(K) * sizeof(int32_t);
  if (groups == 1) {
    // copies in, decode (the usual split-K policy) and copies out in order
    cudaError_t e = cudaMemcpyAsync(h.q_dev, h.q, T * q_row, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h.topk_dev, h.topk, T * k_row, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = launch_decode_fused(args, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h.out, args.out, T * o_row, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h.lse, args.lse, T * l_row, cudaMemcpyDeviceToHost, s);
    return e;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kHostMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_host_mutex);
  HostPipe& p = g_host_pipe[dev];
  e = make_pipe(p);
  if (e != cudaSuccess) return e;
  // The copies in run on the caller's stream (so after the work already
  // queued there); every group but the last branches off to a stream of its
  // own once its rows have landed and sends its rows back on the copy-out
  // stream.  The last group, whose rows land last, decodes and copies back
  // on the caller's stream itself, so no cross-stream hop sits on the step's
  // critical path; the caller's stream finally waits for the copy-out
  // stream (long done by then).
  int64_t r0 = 0;
  for (int g = 0; g < groups && e == cudaSuccess; ++g) {
    const int64_t rows = T / groups + (g < T % groups ? 1 : 0);
    const bool last = g == groups - 1;
    e = cudaMemcpyAsync(h.q_dev + r0 * H * SMLA_QK_DIM,
                        static_cast<const uint8_t*>(h.q) + r0 * q_row, rows * q_row,
                        cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h.topk_dev + r0 * K, h.topk + r0 * K, rows * k_row,
                          cudaMemcpyHostToDevice, s);
    cudaStream_t gs = s, os = s;
    if (!last) {
      gs = p.group[g];
      os = p.out;
      if (e == cudaSuccess) e = cudaEventRecord(p.landed[g], s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(gs, p.landed[g], 0);
    }
    if (e == cudaSuccess) {
      DecodeArgs a = args;
      a.T = int32_t(rows);
      a.q = args.q + r0 * H * SMLA_QK_DIM;
      a.topk = args.topk + r0 * K;
      a.req_id = args.req_id + r0;
      a.out = args.out + r0 * H * SMLA_V_DIM;
      a.lse = args.lse + r0 * H;
      a.single_split = 1;
      a.workspace = nullptr;
      a.workspace_bytes = 0;
      e = launch_decode_fused(a, gs);
    }
    if (!last) {
      if (e == cudaSuccess) e = cudaEventRecord(p.decoded[g], gs);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(os, p.decoded[g], 0);
    }
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(static_cast<uint8_t*>(h.out) + r0 * o_row,
                          args.out + r0 * H * SMLA_V_DIM, rows * o_row, cudaMemcpyDeviceToHost,
                          os);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(h.lse + r0 * H, args.lse + r0 * H, rows * l_row,
                          cudaMemcpyDeviceToHost, os);
    r0 += rows;
  }
  // the caller's later work waits for the other groups' copies back too
  if (e == cudaSuccess) e = cudaEventRecord(p.done, p.out);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p.done, 0);
  return e;
}

}  // namespace smla
