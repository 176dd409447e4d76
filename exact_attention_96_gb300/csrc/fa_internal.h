// fa_internal.h -- declarations shared by the host-side C ABI (fa_api.cu) and the kernel
// translation units.  Not part of the public interface (include/fa.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/fa.h"
#include "philox.cuh"

namespace fa {

// The size checks every entry point applies (B, H, N >= 1; d in {64, 128, 256}; B*H and N
// within the ABI's limits): FA_OK, FA_ERR_INVALID_ARG or FA_ERR_UNSUPPORTED (fa_api.cu).
fa_status check_problem_sizes(int B, int H, int N, int d);

#ifdef __CUDACC__
// Dispatch order of causal launches.  A causal CTA's work depends on its tile: with rank
// 0 the heaviest tile of a head, the CTA of rank r processes about (tiles - r) tiles.
// Dispatched head after head, the last head's heaviest CTA starts near the end and runs
// alone.  Instead the heads are taken in groups of kCausalGroup, and inside a group every
// head's rank-r CTA is dispatched before any rank-(r + 1) CTA: the heavy CTAs start first,
// and the few heads in flight still share their streamed tiles (and the dQ accumulator) in
// L2.  causal_order_of maps a linear index l in [0, tiles * heads) to a (rank, head), a
// bijection for any sizes; causal_dispatch_order applies it to the CTA's index in a
// (gridDim.x = tiles, gridDim.y = heads) grid.  Measured with groups of 2 to 32 heads at
// 4x16x8192x128 causal: 8 is best (larger groups spread the streamed tiles over more heads
// than L2 holds).
constexpr int kCausalGroup = 8;
struct RankHead {
  int rank, bh;
};
__device__ __forceinline__ RankHead causal_order_of(int l, int tiles, int heads, int group = kCausalGroup) {
  const int g0 = l / (group * tiles) * group;
  const int gs = min(group, heads - g0);
  const int r = l - g0 * tiles;
  return {r / gs, g0 + r % gs};
}
__device__ __forceinline__ RankHead causal_dispatch_order() {
  return causal_order_of(int(blockIdx.x) + int(gridDim.x) * int(blockIdx.y), int(gridDim.x), int(gridDim.y));
}

// Masking of a backward key row's 32 query columns as one bit mask, applied after the
// unmasked conversion loop of a tile that needs it (a diagonal tile of a causal head, or the
// sequence tail).  The loop then exists once, without per-element tests.  Testing inside the
// unrolled loop cost up to 12 % (2x8x16384x256 causal backward: 513 against 576 TFLOP/s).
// Bit c of visible_bits(qb, first, N) is set when query qb + c (c < 32) lies in [first, N).
__device__ __forceinline__ uint32_t visible_bits(int qb, int first, int N) {
  const int lo = min(max(first - qb, 0), 32), hi = min(max(N - qb, 0), 32);
  if (hi <= lo) return 0u;
  const uint32_t span = hi - lo == 32 ? 0xFFFFFFFFu : ((1u << (hi - lo)) - 1u);
  return span << lo;
}
// Zeroes the bf16 halves of w (word e holds columns 2e and 2e + 1) whose bit is clear.
__device__ __forceinline__ void apply_keep_mask(uint32_t (&w)[16], uint32_t bits) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint32_t kb = bits >> (2 * e);
    w[e] &= ((kb & 1u) ? 0x0000FFFFu : 0u) | ((kb & 2u) ? 0xFFFF0000u : 0u);
  }
}
#endif

// Everything a forward launch needs besides the four tensor maps.
struct FwdArgs {
  float* lse;           // [B*H, N] fp32
  int N;                // query rows per head
  int Nk;               // keys per head (== N for the square problem)
  int num_splits;       // key-range splits (grid.z); 1 for the square problem
  int tiles_per_split;  // key tiles per split
  float* o_part;        // split mode: fp32 [splits][B*H][N][d] partial outputs, else null
  float* lse_part;      // split mode: fp32 [splits][B*H][N] partial log-sum-exps
  int BH;               // B*H
  int n_q_tiles;        // ceil(N / 128)
  float scale_log2;     // scale * log2(e)
  uint64_t wait_limit_ns;
  int* err_word;        // per-device error word
  int withhold_k_tile;  // test hook: the producer never loads this K tile (-1: none)
  DropoutParams dropout;  // used by the dropout instantiation only
  float o_scale;          // final output multiplier (FP8: V's descale factor; else 1)
};

// Tensor maps of one [B*H, N, d] bf16 tensor: `rows128` boxes of 64 columns x 128 rows,
// `rows_kv` boxes of 64 columns x (key tile) rows.
struct Maps {
  CUtensorMap q, k, v, o;
};

// Forward: one launch.  Returns the cudaError_t of the launch.  With `dropout` the kernel
// applies the mask of a.dropout (square problem only: no split mode).
cudaError_t launch_fwd(const Maps& maps, const FwdArgs& a, int d, bool causal, cudaStream_t s,
                       bool dropout = false);
// FP8 forward for head dim 128, two query tiles per CTA (fa_fwd_fp8.cu): maps of E4M3 Q, K
// and of V transposed ([B*H, 128, ldv]), bf16 O.
cudaError_t launch_fwd_fp8(const Maps& maps, const FwdArgs& a, bool causal, cudaStream_t s);
// Key-tile height the forward kernel uses for head dim d (the K/V tensor-map box height).
int fwd_kv_tile(int d);

// Split-KV merge: o [rows, d] bf16 and lse [rows] from `splits` partial (o, lse) pairs,
// rows = B*H*Nq.
cudaError_t launch_splitkv_combine(const float* o_part, const float* lse_part, uint16_t* o, float* lse,
                                   long long rows, int splits, int d, cudaStream_t s);

struct BwdArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const uint16_t* o;
  const uint16_t* dout;
  const float* lse;
  uint16_t* dq;
  uint16_t* dk;
  uint16_t* dv;
  float* dvec;     // D [B*H, Np]
  float* lse2;     // LSE * log2(e) [B*H, Np]
  float* dq_acc;   // [B*H, N, d] fp32
  int N;
  int BH;
  int d;
  float scale;
  float scale_log2;
  uint64_t wait_limit_ns;
  int* err_word;
  DropoutParams dropout;  // threshold 0 with scale 1: no dropout
  // Accumulate mode (all three set, or all null): the gradients are added in fp32 into these
  // caller buffers ([B*H, N, d] row-major, dQ already multiplied by the scale) instead of
  // being written as bf16 dq, dk, dv.
  float* dq_accum;
  float* dk_accum;
  float* dv_accum;
  // Heads per causal dispatch group of the d = 256 kernel (set by its launcher).
  int causal_group;
};

struct BwdMaps {
  CUtensorMap q, k, v, dout;  // 64-column x 128-row boxes
  // head dim 256 only: Q and dO with 64-row boxes, LSE*log2e and D with 64-entry boxes
  CUtensorMap q64, dout64, lse2_64, dvec_64;
};

// Backward main kernel for d = 256 (fa_bwd_d256.cu); with `dropout` it applies the mask of
// a.dropout.
cudaError_t launch_bwd_main_d256(const CUtensorMap& q64, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& dout64, const CUtensorMap& lse2_64,
                                 const CUtensorMap& d64, const CUtensorMap& dk, const CUtensorMap& dv,
                                 const BwdArgs& a, bool causal, cudaStream_t s, bool dropout);

// Backward: prep, main and dQ-convert launches.  `lse2` and `dvec` describe the fp32
// [B*H, Np] rows of the workspace (box 128 x 1 x 1); `dk`, `dv` the bf16 outputs.
// Np = N rounded up to a multiple of 4.
// With `dropout` the main kernel applies the mask of a.dropout.  `main_events` (optional, two
// events) are recorded on `s` just before and just after the main kernel's launch.
cudaError_t launch_bwd_all(const BwdMaps& m, const CUtensorMap& lse2, const CUtensorMap& dvec,
                           const CUtensorMap& dk, const CUtensorMap& dv, const BwdArgs& a,
                           bool causal, int Np, cudaStream_t s, bool dropout = false,
                           const cudaEvent_t* main_events = nullptr);

// FP8 quantisation (fa_quant.cu): descale = max|x| / 448 of n bf16 values (1 for all zeros),
// left in device memory; E4M3 codes of x / descale, as [BH, N, d] or transposed [BH, d, ld].
cudaError_t launch_e4m3_descale(const uint16_t* x, long long n, float* descale, cudaStream_t s);
cudaError_t launch_quantize_e4m3(const uint16_t* x, uint8_t* out, int BH, int N, int d, bool transpose, int ld,
                                 const float* descale, cudaStream_t s);

// fp32 -> bf16 (round to nearest even), n elements, 16-byte aligned pointers.
cudaError_t launch_f32_to_bf16(const float* src, uint16_t* dst, long long n, cudaStream_t s);

}  // namespace fa
