// fa_host.cu -- one attention training step (forward + backward) whose inputs and results live
// in host memory, with the host <-> device copies overlapped with the kernels.
//
// Heads are independent in both passes, so the step is cut into chunks of heads: the copies
// of chunk c+1 in, the kernels of chunk c and the copies of chunk c-1 out run at once, on
// a copy-in stream, two compute streams (the caller's for even chunks, a second one for odd
// chunks, so that a chunk's kernels can fill the SMs the previous chunk's last CTAs leave
// idle) and a copy-out stream, ordered by events.  The copy engines work beside the SMs, so
// the step costs about its kernel time plus one chunk's copies instead of the sum of the
// three.  Each chunk is an ordinary fa_fwd / fa_bwd call on
// B*H' = (heads in the chunk) rows of the [B*H, N, d] tensors, with pointers offset to the
// chunk; every copy is one cudaMemcpyAsync of a contiguous range.  A chunk's forward waits only
// for its Q, K, V (dO follows them in), and its O and LSE leave as soon as the forward has
// written them, so the first chunk's start and the last chunk's finish each carry one tensor
// fewer of copies.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"

namespace {

constexpr int kMaxChunks = 64;
constexpr int kMaxDevices = 64;

// Per-device copy streams and events, created on first use and reused by every call (the
// enqueue phase of a call holds the lock; a later record of an event does not affect waits
// already enqueued on it).
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr, comp = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  // per chunk: Q, K, V in; dO in; forward done; backward done
  cudaEvent_t loaded[kMaxChunks] = {}, loaded_do[kMaxChunks] = {}, forwarded[kMaxChunks] = {},
              computed[kMaxChunks] = {};
};

std::mutex g_pipe_mu;
HostPipe g_pipes[kMaxDevices];

fa_status pipe_for_device(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  HostPipe& p = g_pipes[dev];
  if (p.in == nullptr) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.comp, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess || cudaEventCreateWithFlags(&p.done, ef) != cudaSuccess)
      return FA_ERR_CUDA;
    for (int c = 0; c < kMaxChunks; ++c)
      if (cudaEventCreateWithFlags(&p.loaded[c], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.loaded_do[c], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.forwarded[c], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.computed[c], ef) != cudaSuccess)
        return FA_ERR_CUDA;
  }
  *out = &p;
  return FA_OK;
}

// Heads per chunk: BH / requested chunks; by default BH / 16, but no fewer heads than give a
// launch 1.5 waves of 128-row tiles on a 152-SM part (smaller launches leave SMs idle: one
// head per chunk of the 4x16x8192x128 step ran at half the speed of four).  Rounded up so
// that every chunk starts LSE on a 16-byte boundary (heads * N a multiple of 4).
int heads_per_chunk(int BH, int N, int requested) {
  int per;
  if (requested > 0) {
    const int n = std::max(1, std::min({requested, BH, kMaxChunks}));
    per = (BH + n - 1) / n;
  } else {
    const int tiles = (N + 127) / 128;
    per = std::max((BH + 15) / 16, (228 + tiles - 1) / tiles);
  }
  if (N % 4 != 0) per = (per + 3) / 4 * 4;
  return std::min(per, BH);
}

}  // namespace

extern "C" {

// One backward workspace per compute stream, each sized for the largest chunk.
size_t fa_step_host_workspace_bytes(int B, int H, int N, int d, int num_chunks) {
  if (B < 1 || H < 1 || N < 1 || num_chunks > kMaxChunks) return 0;
  const size_t one = fa_bwd_workspace_bytes(1, heads_per_chunk(B * H, N, num_chunks), N, d);
  return one == 0 ? 0 : 2 * ((one + 255) & ~size_t(255));
}

fa_status fa_step_host(const void* q_h, const void* k_h, const void* v_h, const void* do_h, void* o_h,
                       float* lse_h, void* dq_h, void* dk_h, void* dv_h, void* q, void* k, void* v, void* dout,
                       void* o, float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                       int causal, int num_chunks, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  if (!q_h || !k_h || !v_h || !do_h || !o_h || !lse_h || !dq_h || !dk_h || !dv_h || !q || !k || !v || !dout ||
      !o || !lse || !dq || !dk || !dv || !workspace)
    return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || N < 1 || num_chunks > kMaxChunks) return num_chunks > kMaxChunks ? FA_ERR_UNSUPPORTED
                                                                                           : FA_ERR_INVALID_ARG;
  const size_t need = fa_step_host_workspace_bytes(B, H, N, d, num_chunks);
  if (need == 0) return FA_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  const int BH = B * H;
  const int per = heads_per_chunk(BH, N, num_chunks);
  const size_t ws_half = need / 2;
  const size_t row = size_t(N) * d * 2;  // bytes of one head of a bf16 tensor
  const size_t lrow = size_t(N) * 4;     // bytes of one head of LSE

  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe* p = nullptr;
  fa_status st = pipe_for_device(&p);
  if (st != FA_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto at = [](const void* base, size_t off) { return static_cast<const uint8_t*>(base) + off; };
  auto atw = [](void* base, size_t off) { return static_cast<uint8_t*>(base) + off; };
  // the library's streams start after the caller's earlier work on its stream
  if (cudaEventRecord(p->start, s) != cudaSuccess || cudaStreamWaitEvent(p->in, p->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->out, p->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(p->comp, p->start, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  for (int c = 0, h0 = 0; h0 < BH; ++c, h0 += per) {
    const int hc = std::min(per, BH - h0);
    const size_t off = size_t(h0) * row, bytes = size_t(hc) * row;
    const size_t loff = size_t(h0) * lrow, lbytes = size_t(hc) * lrow;
    // in: q, k, v of the chunk, then its dO (the forward needs only the first three)
    const void* src[4] = {q_h, k_h, v_h, do_h};
    void* dst[4] = {q, k, v, dout};
    for (int t = 0; t < 4; ++t) {
      if (cudaMemcpyAsync(atw(dst[t], off), at(src[t], off), bytes, cudaMemcpyHostToDevice, p->in) != cudaSuccess)
        return FA_ERR_CUDA;
      if (t == 2 && cudaEventRecord(p->loaded[c], p->in) != cudaSuccess) return FA_ERR_CUDA;
    }
    if (cudaEventRecord(p->loaded_do[c], p->in) != cudaSuccess) return FA_ERR_CUDA;
    // kernels: forward and backward of the chunk's heads, alternating compute streams
    const cudaStream_t cs = (c & 1) ? p->comp : s;
    void* ws = atw(workspace, (c & 1) * ws_half);
    if (cudaStreamWaitEvent(cs, p->loaded[c], 0) != cudaSuccess) return FA_ERR_CUDA;
    const fa_stream_t fs = reinterpret_cast<fa_stream_t>(cs);
    if ((st = fa_fwd(at(q, off), at(k, off), at(v, off), atw(o, off), reinterpret_cast<float*>(atw(lse, loff)), 1, hc,
                     N, d, scale, causal, fs)) != FA_OK)
      return st;
    // O and LSE leave as soon as the forward has written them
    if (cudaEventRecord(p->forwarded[c], cs) != cudaSuccess ||
        cudaStreamWaitEvent(p->out, p->forwarded[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(atw(o_h, off), at(o, off), bytes, cudaMemcpyDeviceToHost, p->out) != cudaSuccess ||
        cudaMemcpyAsync(atw(lse_h, loff), at(lse, loff), lbytes, cudaMemcpyDeviceToHost, p->out) != cudaSuccess)
      return FA_ERR_CUDA;
    if (cudaStreamWaitEvent(cs, p->loaded_do[c], 0) != cudaSuccess) return FA_ERR_CUDA;
    if ((st = fa_bwd(at(q, off), at(k, off), at(v, off), at(o, off), at(dout, off),
                     reinterpret_cast<const float*>(at(lse, loff)), atw(dq, off), atw(dk, off), atw(dv, off), 1, hc,
                     N, d, scale, causal, ws, ws_half, fs)) != FA_OK)
      return st;
    if (cudaEventRecord(p->computed[c], cs) != cudaSuccess ||
        cudaStreamWaitEvent(p->out, p->computed[c], 0) != cudaSuccess)
      return FA_ERR_CUDA;
    // out: dQ, dK, dV of the chunk
    const void* rsrc[3] = {dq, dk, dv};
    void* rdst[3] = {dq_h, dk_h, dv_h};
    for (int t = 0; t < 3; ++t)
      if (cudaMemcpyAsync(atw(rdst[t], off), at(rsrc[t], off), bytes, cudaMemcpyDeviceToHost, p->out) != cudaSuccess)
        return FA_ERR_CUDA;
  }
  // the caller's stream completes after the last copy out (which follows every chunk's kernels)
  if (cudaEventRecord(p->done, p->out) != cudaSuccess || cudaStreamWaitEvent(s, p->done, 0) != cudaSuccess)
    return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"
