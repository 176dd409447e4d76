// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument validation,
// TMA tensor-map encoding, launches, and the per-device error word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

// One error word per device, in static device memory.  Bit 0: a bounded wait timed out.
// Bit 1: shared memory was not 1024-byte aligned.
__device__ int g_fa_err_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};
int g_cc_ok[kMaxDevices] = {};  // 0 unknown, 1 sm_103, -1 other
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_withhold_k_tile{-1};  // one-shot test hook for the next fa_fwd launch
// one-shot profiling request of this host thread: events around the next backward main kernel
thread_local cudaEvent_t g_tl_main_events[2] = {nullptr, nullptr};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

fa_status cuda_fail(cudaError_t) { return FA_ERR_CUDA; }

// Resolves the device, checks it is compute capability 10.3 and returns its error word.
fa_status device_setup(int* dev_out, int** err_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_cc_ok[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return FA_ERR_CUDA;
    g_cc_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  if (g_cc_ok[dev] != 1) return FA_ERR_UNSUPPORTED;
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_err_word) != cudaSuccess) return FA_ERR_CUDA;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return FA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *dev_out = dev;
  *err_out = g_err_ptr[dev];
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_sizes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if ((long long)B * H > 65535 || N > (1 << 20)) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

fa_status check_scale(float scale) {
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// [BH, N, d] bf16, box (64 columns, rows, 1), 128-byte swizzle.
bool encode_bf16_rows(CUtensorMap* m, const void* p, int BH, int N, int d, int rows) {
  const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(N), cuuint64_t(BH)};
  const cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(N) * d * 2};
  const cuuint32_t box[3] = {64, cuuint32_t(rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [BH, rows, cols] bytes (E4M3), box (128 columns, 128 rows, 1), 128-byte swizzle.  `ld` is
// the row stride in bytes (a multiple of 16, >= cols).
bool encode_u8_rows(CUtensorMap* m, const void* p, int BH, int rows, int cols, int ld) {
  const cuuint64_t dims[3] = {cuuint64_t(cols), cuuint64_t(rows), cuuint64_t(BH)};
  const cuuint64_t strides[2] = {cuuint64_t(ld), cuuint64_t(ld) * rows};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(p), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [1, BH, Np] fp32 rows, box (box, 1, 1), no swizzle.
bool encode_f32_rows(CUtensorMap* m, const void* p, int BH, int Np, int box_len = 128) {
  const cuuint64_t dims[3] = {cuuint64_t(Np), cuuint64_t(BH), 1};
  const cuuint64_t strides[2] = {cuuint64_t(Np) * 4, cuuint64_t(Np) * 4 * BH};
  const cuuint32_t box[3] = {cuuint32_t(box_len), 1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(p), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t dvec_off, lse2_off, dq_off, total;
  int Np, n_q_tiles;
};

WsLayout ws_layout(int B, int H, int N, int d) {
  WsLayout w{};
  const size_t BH = size_t(B) * H;
  w.Np = (N + 3) & ~3;
  w.n_q_tiles = (N + 127) / 128;
  w.dvec_off = 0;
  w.lse2_off = round256(BH * w.Np * 4);
  w.dq_off = w.lse2_off + round256(BH * w.Np * 4);
  w.total = w.dq_off + BH * size_t(w.n_q_tiles) * 128 * d * 4;
  return w;
}


// Dropout parameters from the probability and seed: threshold t = round(p * 2^16) (ties to
// even, at most 2^16 - 1), scale 2^16 / (2^16 - t).
fa_status make_dropout(double p, unsigned long long seed, fa::DropoutParams* dp) {
  if (!(p >= 0.0 && p < 1.0)) return FA_ERR_INVALID_ARG;
  const double t = std::min(std::nearbyint(p * 65536.0), 65535.0);
  dp->threshold = uint32_t(t);
  dp->scale = float(65536.0 / (65536.0 - t));
  dp->seed_lo = uint32_t(seed & 0xFFFFFFFFull);
  dp->seed_hi = uint32_t(seed >> 32);
  return FA_OK;
}

// Forward of the square problem; `dp` null: no dropout.
fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                   float scale, int causal, const fa::DropoutParams* dp, fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;

  const int BH = B * H;
  fa::Maps maps;
  const int kv_rows = fa::fwd_kv_tile(d);
  if (!encode_bf16_rows(&maps.q, q, BH, N, d, 128) || !encode_bf16_rows(&maps.k, k, BH, N, d, kv_rows) ||
      !encode_bf16_rows(&maps.v, v, BH, N, d, kv_rows) || !encode_bf16_rows(&maps.o, o, BH, N, d, 128))
    return FA_ERR_CUDA;
  fa::FwdArgs a;
  a.lse = lse;
  a.N = N;
  a.Nk = N;
  a.num_splits = 1;
  a.tiles_per_split = (N + kv_rows - 1) / kv_rows;
  a.o_part = nullptr;
  a.lse_part = nullptr;
  a.BH = BH;
  a.n_q_tiles = (N + 127) / 128;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.err_word = err;
  a.withhold_k_tile = g_withhold_k_tile.exchange(-1);
  a.dropout = dp ? *dp : fa::DropoutParams{0u, 1.f, 0u, 0u};
  a.o_scale = 1.f;
  const cudaError_t e =
      fa::launch_fwd(maps, a, d, causal != 0, reinterpret_cast<cudaStream_t>(stream), dp != nullptr);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

// Backward; `dp` null: no dropout.  `accum` (three fp32 pointers dQ, dK, dV) selects the
// accumulate mode, where dq, dk, dv are not used.
fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                   int causal, const fa::DropoutParams* dp, void* workspace, size_t workspace_bytes,
                   fa_stream_t stream, float* const* accum = nullptr) {
  if (accum != nullptr) {
    if (!accum[0] || !accum[1] || !accum[2]) return FA_ERR_INVALID_ARG;
    if (!aligned16(accum[0]) || !aligned16(accum[1]) || !aligned16(accum[2])) return FA_ERR_MISALIGNED;
    dq = accum[0];  // stand-ins: the bf16 outputs are neither encoded for stores nor written
    dk = accum[1];
    dv = accum[2];
  }
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  const WsLayout w = ws_layout(B, H, N, d);
  if (workspace_bytes < w.total) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FA_ERR_MISALIGNED;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;

  const int BH = B * H;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  fa::BwdMaps maps;
  CUtensorMap m_lse2, m_dvec, m_dk, m_dv;
  if (!encode_bf16_rows(&maps.q, q, BH, N, d, 128) || !encode_bf16_rows(&maps.k, k, BH, N, d, 128) ||
      !encode_bf16_rows(&maps.v, v, BH, N, d, 128) || !encode_bf16_rows(&maps.dout, dout, BH, N, d, 128) ||
      !encode_bf16_rows(&m_dk, dk, BH, N, d, 128) || !encode_bf16_rows(&m_dv, dv, BH, N, d, 128) ||
      !encode_f32_rows(&m_lse2, ws + w.lse2_off, BH, w.Np) || !encode_f32_rows(&m_dvec, ws + w.dvec_off, BH, w.Np))
    return FA_ERR_CUDA;
  if (d == 256 && (!encode_bf16_rows(&maps.q64, q, BH, N, d, 64) ||
                   !encode_bf16_rows(&maps.dout64, dout, BH, N, d, 64) ||
                   !encode_f32_rows(&maps.lse2_64, ws + w.lse2_off, BH, w.Np, 64) ||
                   !encode_f32_rows(&maps.dvec_64, ws + w.dvec_off, BH, w.Np, 64)))
    return FA_ERR_CUDA;
  fa::BwdArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.o = static_cast<const uint16_t*>(o);
  a.dout = static_cast<const uint16_t*>(dout);
  a.lse = lse;
  a.dq = static_cast<uint16_t*>(dq);
  a.dk = static_cast<uint16_t*>(dk);
  a.dv = static_cast<uint16_t*>(dv);
  a.dvec = reinterpret_cast<float*>(ws + w.dvec_off);
  a.lse2 = reinterpret_cast<float*>(ws + w.lse2_off);
  a.dq_acc = reinterpret_cast<float*>(ws + w.dq_off);
  a.N = N;
  a.BH = BH;
  a.d = d;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.err_word = err;
  a.dropout = dp ? *dp : fa::DropoutParams{0u, 1.f, 0u, 0u};
  a.dq_accum = accum ? accum[0] : nullptr;
  a.dk_accum = accum ? accum[1] : nullptr;
  a.dv_accum = accum ? accum[2] : nullptr;
  a.causal_group = fa::kCausalGroup;  // the d = 256 launcher sets its own
  const cudaEvent_t events[2] = {g_tl_main_events[0], g_tl_main_events[1]};
  g_tl_main_events[0] = g_tl_main_events[1] = nullptr;
  const cudaError_t e = fa::launch_bwd_all(maps, m_lse2, m_dvec, m_dk, m_dv, a, causal != 0, w.Np,
                                           reinterpret_cast<cudaStream_t>(stream), dp != nullptr,
                                           events[0] != nullptr ? events : nullptr);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

}  // namespace

fa_status fa::check_problem_sizes(int B, int H, int N, int d) { return check_sizes(B, H, N, d); }

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

fa_status fa_profile_next_bwd_main(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return FA_ERR_INVALID_ARG;
  g_tl_main_events[0] = static_cast<cudaEvent_t>(start_event);
  g_tl_main_events[1] = static_cast<cudaEvent_t>(stop_event);
  return FA_OK;
}

int fa_test_withhold_kv_tile(int tile) { return g_withhold_k_tile.exchange(tile < 0 ? -1 : tile); }

uint64_t fa_set_wait_limit_ns(uint64_t ns) {
  if (ns < 1000000ull) ns = 1000000ull;
  return g_wait_limit_ns.exchange(ns);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                 int d, float scale, int causal, fa_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, nullptr, stream);
}

fa_status fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                         int d, float scale, int causal, double dropout_p, unsigned long long seed,
                         fa_stream_t stream) {
  fa::DropoutParams dp;
  const fa_status st = make_dropout(dropout_p, seed, &dp);
  if (st != FA_OK) return st;
  return fwd_impl(q, k, v, o, lse, B, H, N, d, scale, causal, &dp, stream);
}

namespace {

struct SplitPlan {
  int splits, tiles_per_split;
  size_t lse_off, total;
};

// Key-range split: `requested` <= 0 picks enough splits for about two CTAs per SM of a
// 152-SM part (independent of the device, so the workspace size is a pure function of the
// sizes); every split gets at least one key tile.
SplitPlan split_plan(int B, int H, int Nq, int Nk, int d, int requested) {
  SplitPlan p{};
  const int bc = fa::fwd_kv_tile(d);
  const int n_tiles = (Nk + bc - 1) / bc;
  const long long base = (long long)((Nq + 127) / 128) * B * H;
  int want = requested > 0 ? requested : int(std::min<long long>(256, (304 + base - 1) / base));
  want = std::max(1, std::min(want, n_tiles));
  p.tiles_per_split = (n_tiles + want - 1) / want;
  p.splits = (n_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  const size_t rows = size_t(B) * H * Nq;
  p.lse_off = round256(size_t(p.splits) * rows * d * 4);
  p.total = p.lse_off + size_t(p.splits) * rows * 4;
  return p;
}

}  // namespace

size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (check_sizes(B, H, Nq, d) != FA_OK || check_sizes(B, H, Nk, d) != FA_OK || num_splits > 1024) return 0;
  return split_plan(B, H, Nq, Nk, d, num_splits).total;
}

int fa_fwd_splitkv_num_splits(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (check_sizes(B, H, Nq, d) != FA_OK || check_sizes(B, H, Nk, d) != FA_OK || num_splits > 1024) return 0;
  return split_plan(B, H, Nq, Nk, d, num_splits).splits;
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                         int Nq, int Nk, int d, float scale, int num_splits, void* workspace,
                         size_t workspace_bytes, fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, Nq, d);
  if (st != FA_OK) return st;
  if ((st = check_sizes(B, H, Nk, d)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (num_splits > 1024) return FA_ERR_UNSUPPORTED;
  const SplitPlan plan = split_plan(B, H, Nq, Nk, d, num_splits);
  if (workspace_bytes < plan.total) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FA_ERR_MISALIGNED;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  const int BH = B * H;
  const int kv_rows = fa::fwd_kv_tile(d);
  fa::Maps maps;
  if (!encode_bf16_rows(&maps.q, q, BH, Nq, d, 128) || !encode_bf16_rows(&maps.k, k, BH, Nk, d, kv_rows) ||
      !encode_bf16_rows(&maps.v, v, BH, Nk, d, kv_rows) || !encode_bf16_rows(&maps.o, o, BH, Nq, d, 128))
    return FA_ERR_CUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  fa::FwdArgs a;
  a.lse = lse;
  a.N = Nq;
  a.Nk = Nk;
  a.num_splits = plan.splits;
  a.tiles_per_split = plan.tiles_per_split;
  a.o_part = reinterpret_cast<float*>(ws);
  a.lse_part = reinterpret_cast<float*>(ws + plan.lse_off);
  a.BH = BH;
  a.n_q_tiles = (Nq + 127) / 128;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.err_word = err;
  a.withhold_k_tile = -1;
  a.o_scale = 1.f;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_fwd(maps, a, d, false, s);
  if (e != cudaSuccess) return cuda_fail(e);
  e = fa::launch_splitkv_combine(a.o_part, a.lse_part, static_cast<uint16_t*>(o), lse,
                                 (long long)BH * Nq, plan.splits, d, s);
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

fa_status fa_fwd_partial(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int B,
                         int H, int Nq, int Nk, int d, float scale, int causal, fa_stream_t stream) {
  if (!q || !k || !v || !o_part || !lse_part) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, Nq, d);
  if (st != FA_OK) return st;
  if ((st = check_sizes(B, H, Nk, d)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (causal && Nq != Nk) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part) || !aligned16(lse_part))
    return FA_ERR_MISALIGNED;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  const int BH = B * H;
  const int kv_rows = fa::fwd_kv_tile(d);
  fa::Maps maps;
  if (!encode_bf16_rows(&maps.q, q, BH, Nq, d, 128) || !encode_bf16_rows(&maps.k, k, BH, Nk, d, kv_rows) ||
      !encode_bf16_rows(&maps.v, v, BH, Nk, d, kv_rows) || !encode_bf16_rows(&maps.o, q, BH, Nq, d, 128))
    return FA_ERR_CUDA;
  fa::FwdArgs a;
  a.lse = lse_part;
  a.N = Nq;
  a.Nk = Nk;
  a.num_splits = 1;
  a.tiles_per_split = (Nk + kv_rows - 1) / kv_rows;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.BH = BH;
  a.n_q_tiles = (Nq + 127) / 128;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.err_word = err;
  a.withhold_k_tile = -1;
  a.o_scale = 1.f;
  const cudaError_t e = fa::launch_fwd(maps, a, d, causal != 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

fa_status fa_merge_partials(const float* o_parts, const float* lse_parts, int num_parts, long long rows, int d,
                            void* o, float* lse, fa_stream_t stream) {
  if (!o_parts || !lse_parts || !o || !lse || num_parts < 1 || rows < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
  if (!aligned16(o_parts) || !aligned16(lse_parts) || !aligned16(o) || !aligned16(lse)) return FA_ERR_MISALIGNED;
  int dev = 0;
  int* err = nullptr;
  fa_status st = device_setup(&dev, &err);
  if (st != FA_OK) return st;
  const cudaError_t e = fa::launch_splitkv_combine(o_parts, lse_parts, static_cast<uint16_t*>(o), lse, rows,
                                                   num_parts, d, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d) != FA_OK) return 0;
  return ws_layout(B, H, N, d).total;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                 int causal, void* workspace, size_t workspace_bytes, fa_stream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, nullptr, workspace,
                  workspace_bytes, stream);
}

fa_status fa_bwd_accumulate(const void* q, const void* k, const void* v, const void* o, const void* dout,
                            const float* lse, float* dq_acc, float* dk_acc, float* dv_acc, int B, int H, int N,
                            int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                            fa_stream_t stream) {
  float* const accum[3] = {dq_acc, dk_acc, dv_acc};
  return bwd_impl(q, k, v, o, dout, lse, nullptr, nullptr, nullptr, B, H, N, d, scale, causal, nullptr,
                  workspace, workspace_bytes, stream, accum);
}

fa_status fa_e4m3_descale(const void* x, long long n, float* descale, fa_stream_t stream) {
  if (!x || !descale || n < 1) return FA_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(descale) & 3u) != 0) return FA_ERR_MISALIGNED;
  int dev = 0;
  int* err = nullptr;
  const fa_status st = device_setup(&dev, &err);
  if (st != FA_OK) return st;
  const cudaError_t e = fa::launch_e4m3_descale(static_cast<const uint16_t*>(x), n, descale,
                                                reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

fa_status fa_quantize_e4m3(const void* x, void* out8, int B, int H, int N, int d, int transpose, int ld,
                           const float* descale, fa_stream_t stream) {
  if (!x || !out8 || !descale) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if (transpose && (ld < N || ld % 16 != 0)) return FA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(out8) || (reinterpret_cast<uintptr_t>(descale) & 3u) != 0)
    return FA_ERR_MISALIGNED;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  const cudaError_t e = fa::launch_quantize_e4m3(static_cast<const uint16_t*>(x), static_cast<uint8_t*>(out8),
                                                 B * H, N, d, transpose != 0, ld, descale,
                                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

fa_status fa_convert_f32_to_bf16(const float* src, void* dst, long long n, fa_stream_t stream) {
  if (!src || !dst || n < 1) return FA_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return FA_ERR_MISALIGNED;
  int dev = 0;
  int* err = nullptr;
  const fa_status st = device_setup(&dev, &err);
  if (st != FA_OK) return st;
  const cudaError_t e = fa::launch_f32_to_bf16(src, static_cast<uint16_t*>(dst), n,
                                               reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

fa_status fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                         int causal, double dropout_p, unsigned long long seed, void* workspace,
                         size_t workspace_bytes, fa_stream_t stream) {
  fa::DropoutParams dp;
  const fa_status st = make_dropout(dropout_p, seed, &dp);
  if (st != FA_OK) return st;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, &dp, workspace,
                  workspace_bytes, stream);
}

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, int ldv, void* o, float* lse, int B,
                     int H, int N, int d, float scale, float q_descale, float k_descale, float v_descale,
                     int causal, fa_stream_t stream) {
  if (!q8 || !k8 || !vt8 || !o || !lse) return FA_ERR_INVALID_ARG;
  fa_status st = check_sizes(B, H, N, d);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if ((st = check_scale(scale)) != FA_OK || (st = check_scale(q_descale)) != FA_OK ||
      (st = check_scale(k_descale)) != FA_OK || (st = check_scale(v_descale)) != FA_OK)
    return st;
  if (ldv < N || ldv % 16 != 0) return FA_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  int dev = 0;
  int* err = nullptr;
  if ((st = device_setup(&dev, &err)) != FA_OK) return st;
  const int BH = B * H;
  fa::Maps maps;
  if (!encode_u8_rows(&maps.q, q8, BH, N, d, d) || !encode_u8_rows(&maps.k, k8, BH, N, d, d) ||
      !encode_u8_rows(&maps.v, vt8, BH, d, N, ldv) || !encode_bf16_rows(&maps.o, o, BH, N, d, 128))
    return FA_ERR_CUDA;
  fa::FwdArgs a;
  a.lse = lse;
  a.N = N;
  a.Nk = N;
  a.num_splits = 1;
  a.tiles_per_split = (N + 127) / 128;
  a.o_part = nullptr;
  a.lse_part = nullptr;
  a.BH = BH;
  a.n_q_tiles = (N + 127) / 128;
  a.scale_log2 = float(double(scale) * q_descale * k_descale * 1.4426950408889634);
  a.wait_limit_ns = g_wait_limit_ns.load();
  a.err_word = err;
  a.withhold_k_tile = -1;
  a.dropout = fa::DropoutParams{0u, 1.f, 0u, 0u};
  a.o_scale = v_descale;
  const cudaError_t e = fa::launch_fwd_fp8(maps, a, causal != 0, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : cuda_fail(e);
}

fa_status fa_status_check(fa_stream_t stream) {
  int dev = 0;
  int* err = nullptr;
  fa_status st = device_setup(&dev, &err);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_fa_err_word, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (word != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_err_word, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (word & 1) return FA_ERR_TIMEOUT;
  if (word != 0) return FA_ERR_CUDA;
  return FA_OK;
}

}  // extern "C"
