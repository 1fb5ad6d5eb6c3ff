// The end-to-end call on host buffers (sage_attn_host): the request is cut
// into chunks of whole kv-heads of one batch element -- independent problems
// with their own statistics and scales -- and the copies of one chunk overlap
// the kernels of the others: host -> device copies on one stream, the
// pre-pass and attention of even chunks on the caller's stream and of odd
// chunks on a second compute stream (each chunk in the workspace slot of its
// stream, so the next chunk's blocks fill the SMs the previous chunk's last
// blocks leave idle), device -> host copies on a fourth stream.  The internal
// streams and their events are created once per device on the first call (no
// device memory); the call is ordered after earlier work on the caller's
// stream, and later work on that stream after its last copy.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "layout.h"
#include "launch.h"

namespace sage {
namespace {

struct HostChunk {
  int b, g0, g1;  // batch element and its kv heads [g0, g1)
};

// chunks of about kHostChunkBlocks query blocks (a few waves of one CTA per
// SM each), at least kHostChunksMin and at most kHostChunksMax: the first
// chunk's copies in and the last chunk's copy out are what the pipeline
// cannot hide (video: 24 chunks measured 14.9 ms per step end to end against
// 16.2 with 6, the device alone taking 14.6)
constexpr int kHostChunkBlocks = 512, kHostChunksMin = 6, kHostChunksMax = 24;
constexpr size_t kHostStatusBytes = 1024;  // the call's status word at the start of dev_buf

std::vector<HostChunk> host_chunks(const sage_shape &s) {
  std::vector<HostChunk> out;
  const int64_t blocks = (int64_t)s.B * s.Hq * ((s.N + 127) / 128);
  const int target = (int)std::max<int64_t>(kHostChunksMin, std::min<int64_t>(kHostChunksMax, blocks / kHostChunkBlocks));
  const int per_b = std::max(1, std::min(s.Hkv, (target + s.B - 1) / s.B));
  for (int b = 0; b < s.B; ++b)
    for (int k = 0; k < per_b; ++k) {
      const int g0 = (int)((int64_t)k * s.Hkv / per_b), g1 = (int)((int64_t)(k + 1) * s.Hkv / per_b);
      if (g1 > g0) out.push_back(HostChunk{b, g0, g1});
    }
  return out;
}

sage_shape chunk_shape(const sage_shape &s, const HostChunk &c) {
  const int G = s.Hq / s.Hkv;
  return sage_shape{1, (c.g1 - c.g0) * G, c.g1 - c.g0, s.N, s.M, s.d};
}

size_t io_bytes(const sage_shape &s) {
  const size_t qn = (size_t)s.B * s.Hq * s.N * s.d * 2, kn = (size_t)s.B * s.Hkv * s.M * s.d * 2;
  return align_up(qn, 1024) * 2 + align_up(kn, 1024) * 2;  // q, k, v, o
}

// the largest chunk's workspace (every chunk's fits in a slot of this size)
sage_status slot_bytes(const sage_shape &s, int mode, int bq, int bk, size_t *bytes) {
  size_t best = 0;
  for (const HostChunk &c : host_chunks(s)) {
    const sage_shape cs = chunk_shape(s, c);
    sage_ws_layout L;
    const sage_status st = compute_layout(&cs, mode, bq, bk, &L);
    if (st != SAGE_OK) return st;
    best = std::max(best, L.total);
  }
  *bytes = align_up(best, 1024);
  return SAGE_OK;
}

struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr, cmp = nullptr;
  cudaEvent_t start = nullptr, done = nullptr, in_done[2] = {nullptr, nullptr}, cmp_done[2] = {nullptr, nullptr};
  bool ok = false;
};

// The copy streams and events of a device, created on its first call.
HostPipe *host_pipe() {
  constexpr int kMaxDevices = 64;
  static HostPipe pipes[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  HostPipe &p = pipes[dev];
  if (!p.ok) {
    const unsigned ef = cudaEventDisableTiming;
    bool good = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
                cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
                cudaStreamCreateWithFlags(&p.cmp, cudaStreamNonBlocking) == cudaSuccess &&
                cudaEventCreateWithFlags(&p.start, ef) == cudaSuccess &&
                cudaEventCreateWithFlags(&p.done, ef) == cudaSuccess;
    for (int i = 0; i < 2 && good; ++i)
      good = cudaEventCreateWithFlags(&p.in_done[i], ef) == cudaSuccess &&
             cudaEventCreateWithFlags(&p.cmp_done[i], ef) == cudaSuccess;
    if (!good) return nullptr;
    p.ok = true;
  }
  return &p;
}

// keep the first error of any chunk: the call's status word takes a chunk's
// when it holds none yet
__global__ void merge_status_kernel(const int *chunk, int *total) {
  if (threadIdx.x == 0 && chunk[0] != 0 && atomicCAS(&total[0], 0, chunk[0]) == 0) {
    total[1] = chunk[1];
    total[2] = chunk[2];
  }
}

}  // namespace

sage_status host_buffer_bytes(const sage_shape &s, int mode, int bq, int bk, size_t *bytes) {
  size_t slot = 0;
  const sage_status st = slot_bytes(s, mode, bq, bk, &slot);
  if (st != SAGE_OK) return st;
  *bytes = kHostStatusBytes + io_bytes(s) + 2 * slot;
  return SAGE_OK;
}

sage_status run_attn_host(const sage_shape &s, int causal, float sm_scale, int mode, int flags, int bq, int bk,
                          const void *q_host, const void *k_host, const void *v_host, void *o_host, void *dev_buf,
                          cudaStream_t stream) {
  size_t slot = 0;
  sage_status st = slot_bytes(s, mode, bq, bk, &slot);
  if (st != SAGE_OK) return st;
  HostPipe *hp = host_pipe();
  if (!hp) return SAGE_ERR_CUDA;
  const int G = s.Hq / s.Hkv;
  const size_t qrow = (size_t)s.N * s.d * 2, krow = (size_t)s.M * s.d * 2;  // bytes of one head
  const size_t qn = (size_t)s.B * s.Hq * qrow, kn = (size_t)s.B * s.Hkv * krow;
  char *base = (char *)dev_buf;
  int *status = (int *)base;
  char *dq = base + kHostStatusBytes;
  char *dk = dq + align_up(qn, 1024);
  char *dv = dk + align_up(kn, 1024);
  char *dO = dv + align_up(kn, 1024);
  char *slots = dO + align_up(qn, 1024);
  const char *qh = (const char *)q_host, *kh = (const char *)k_host, *vh = (const char *)v_host;
  char *oh = (char *)o_host;
#define SAGE_CK(x)                    \
  do {                                \
    if ((x) != cudaSuccess) return SAGE_ERR_CUDA; \
  } while (0)
  SAGE_CK(cudaMemsetAsync(status, 0, 16, stream));
  SAGE_CK(cudaEventRecord(hp->start, stream));
  SAGE_CK(cudaStreamWaitEvent(hp->in, hp->start, 0));
  SAGE_CK(cudaStreamWaitEvent(hp->out, hp->start, 0));
  SAGE_CK(cudaStreamWaitEvent(hp->cmp, hp->start, 0));
  cudaStream_t cmp[2] = {stream, hp->cmp};
  const std::vector<HostChunk> chunks = host_chunks(s);
  for (size_t i = 0; i < chunks.size(); ++i) {
    const HostChunk &c = chunks[i];
    const sage_shape cs = chunk_shape(s, c);
    const size_t qo = ((size_t)c.b * s.Hq + (size_t)c.g0 * G) * qrow, qb = (size_t)cs.Hq * qrow;
    const size_t ko = ((size_t)c.b * s.Hkv + c.g0) * krow, kb = (size_t)cs.Hkv * krow;
    const int r = (int)(i & 1);
    // host -> device: this chunk's q, k, v slices
    SAGE_CK(cudaMemcpyAsync(dq + qo, qh + qo, qb, cudaMemcpyHostToDevice, hp->in));
    SAGE_CK(cudaMemcpyAsync(dk + ko, kh + ko, kb, cudaMemcpyHostToDevice, hp->in));
    SAGE_CK(cudaMemcpyAsync(dv + ko, vh + ko, kb, cudaMemcpyHostToDevice, hp->in));
    SAGE_CK(cudaEventRecord(hp->in_done[r], hp->in));
    // the kernels on compute stream r, in workspace slot r (its previous
    // user, chunk i - 2, ran earlier on this same stream)
    cudaStream_t cst = cmp[r];
    SAGE_CK(cudaStreamWaitEvent(cst, hp->in_done[r], 0));
    char *ws = slots + r * slot;
    st = sage_quantize_qkv(&cs, mode, flags, bq, bk, dq + qo, dk + ko, dv + ko, ws, slot, (sage_stream_t)cst);
    if (st != SAGE_OK) return st;
    st = sage_attn_fwd(&cs, causal, sm_scale, mode, flags, bq, bk, ws, slot, dO + qo, (sage_stream_t)cst);
    if (st != SAGE_OK) return st;
    sage_ws_layout L;
    if ((st = compute_layout(&cs, mode, bq, bk, &L)) != SAGE_OK) return st;
    merge_status_kernel<<<1, 32, 0, cst>>>((const int *)(ws + L.status), status);
    SAGE_CK(cudaGetLastError());
    SAGE_CK(cudaEventRecord(hp->cmp_done[r], cst));
    // device -> host: this chunk's output rows
    SAGE_CK(cudaStreamWaitEvent(hp->out, hp->cmp_done[r], 0));
    SAGE_CK(cudaMemcpyAsync(oh + qo, dO + qo, qb, cudaMemcpyDeviceToHost, hp->out));
  }
  // the caller's stream after the last copy back (which follows both compute
  // streams' last chunks)
  SAGE_CK(cudaEventRecord(hp->done, hp->out));
  SAGE_CK(cudaStreamWaitEvent(stream, hp->done, 0));
#undef SAGE_CK
  return SAGE_OK;
}

}  // namespace sage
