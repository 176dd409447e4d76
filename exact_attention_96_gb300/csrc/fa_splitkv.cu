// fa_splitkv.cu -- merge of split-KV partial results ("Flash Attention 原理与实践" §5.1:
// the key/value sequence is split across SMs, each part computes its own softmax-weighted
// output, and the parts are merged with log-sum-exp).
//
// Part s of row r holds O_s (normalised within its key range) and LSE_s.  With
// LSE = log sum_s exp(LSE_s), the merged output is O = sum_s exp(LSE_s - LSE) O_s, the same
// re-basing the streaming softmax applies between tiles ("FlashAttention 与显存" §08).
// One warp per row; lane l owns d/32 adjacent columns.

#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2eC = 1.4426950408889634f;
constexpr float kLn2C = 0.69314718055994531f;

template <int D>
__global__ void __launch_bounds__(256)
fa_splitkv_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                          uint16_t* __restrict__ o, float* __restrict__ lse, long long rows, int splits) {
  constexpr int kPerLane = D / 32;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  // LSE of the whole row, in base 2 internally
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s) m = fmaxf(m, lse_part[(size_t)s * rows + row] * kLog2eC);
  float sum = 0.f;
  for (int s = 0; s < splits; ++s) sum += ex2_approx(lse_part[(size_t)s * rows + row] * kLog2eC - m);
  const float lse2 = m + lg2_approx(sum);
  float acc[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) acc[i] = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float w = ex2_approx(lse_part[(size_t)s * rows + row] * kLog2eC - lse2);
    const float* src = o_part + ((size_t)s * rows + row) * D + lane * kPerLane;
#pragma unroll
    for (int i = 0; i < kPerLane; i += 2) {
      const float2 x = *reinterpret_cast<const float2*>(src + i);
      acc[i] = fmaf(w, x.x, acc[i]);
      acc[i + 1] = fmaf(w, x.y, acc[i + 1]);
    }
  }
  uint32_t packed[kPerLane / 2];
#pragma unroll
  for (int i = 0; i < kPerLane; i += 2) packed[i / 2] = pack_bf16x2(acc[i], acc[i + 1]);
  uint16_t* dst = o + row * D + lane * kPerLane;
  if constexpr (kPerLane == 2) {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  } else if constexpr (kPerLane == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  }
  if (lane == 0) lse[row] = lse2 * kLn2C;
}

}  // namespace

cudaError_t launch_splitkv_combine(const float* o_part, const float* lse_part, uint16_t* o, float* lse,
                                   long long rows, int splits, int d, cudaStream_t s) {
  const unsigned grid = unsigned((rows + 7) / 8);
  switch (d) {
    case 64: fa_splitkv_combine_kernel<64><<<grid, 256, 0, s>>>(o_part, lse_part, o, lse, rows, splits); break;
    case 128: fa_splitkv_combine_kernel<128><<<grid, 256, 0, s>>>(o_part, lse_part, o, lse, rows, splits); break;
    case 256: fa_splitkv_combine_kernel<256><<<grid, 256, 0, s>>>(o_part, lse_part, o, lse, rows, splits); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace fa
