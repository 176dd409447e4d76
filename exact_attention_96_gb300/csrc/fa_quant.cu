// fa_quant.cu -- FP8 (E4M3) quantisation of bf16 attention inputs on the device, for the FP8
// forward ("Flash Attention 原理与实践" §3.2: the third version's FP8 mode takes 8-bit Q, K, V).
//
//   fa_e4m3_descale   descale = max|x| / 448 (fp32, 1 when x is all zeros): one reduction
//                     launch (per-block maxima, then an atomic maximum on the fp32 bit pattern,
//                     which orders non-negative floats like unsigned integers) and a one-thread
//                     finishing launch.
//   fa_quantize_e4m3  code = E4M3(x / descale): the quotient in fp32 (IEEE division), rounded
//                     to the nearest E4M3 value with ties to the even code and magnitudes above
//                     448 saturated (cvt.rn.satfinite), either in place of each element or
//                     transposed per head ([BH, N, d] -> [BH, d, ld], the V layout of
//                     fa_fwd_fp8), the transposed form through a 64 x 64 shared-memory tile.
// Both are HBM-bound elementwise passes (2 bytes read, 1 byte written per element).
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// max |x| over n bf16 values into *amax_bits (the fp32 bit pattern of a non-negative float)
__global__ void __launch_bounds__(256) fa_absmax_kernel(const uint16_t* __restrict__ x, long long n,
                                                        unsigned int* __restrict__ amax_bits) {
  float m = 0.f;
  const long long n8 = n / 8;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 w = reinterpret_cast<const uint4*>(x)[i];
    const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(fabsf(bf16_lo(v[e])), fabsf(bf16_hi(v[e]))));
  }
  if (blockIdx.x == 0)
    for (long long i = n8 * 8 + threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, fabsf(__uint_as_float(uint32_t(x[i]) << 16)));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float warp_max[8];
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) m = fmaxf(m, warp_max[w]);
    atomicMax(amax_bits, __float_as_uint(m));
  }
}

__global__ void fa_descale_finish_kernel(float* descale) {
  const float amax = *descale;  // the reduction left max|x| here
  *descale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
}

// element-wise: 16 values per thread (d is a multiple of 16, so no thread straddles rows)
__global__ void __launch_bounds__(256) fa_quant_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ out,
                                                       long long n16, const float* __restrict__ descale) {
  const float s = *descale;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += stride) {
    const uint4 a = reinterpret_cast<const uint4*>(x)[2 * i];
    const uint4 b = reinterpret_cast<const uint4*>(x)[2 * i + 1];
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = pack_e4m3x4(__fdiv_rn(bf16_lo(v[2 * k]), s), __fdiv_rn(bf16_hi(v[2 * k]), s),
                         __fdiv_rn(bf16_lo(v[2 * k + 1]), s), __fdiv_rn(bf16_hi(v[2 * k + 1]), s));
    reinterpret_cast<uint4*>(out)[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// transposed: block (jt, ct, bh) converts x[bh][64 jt .. +64][64 ct .. +64] into
// out[bh][64 ct .. +64][64 jt .. +64] (row stride ld); positions N <= j < ld are written as 0
constexpr int kT = 64;
__global__ void __launch_bounds__(256) fa_quant_t_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ out,
                                                         int N, int d, int ld, const float* __restrict__ descale) {
  __shared__ uint8_t tile[kT][kT + 4];  // [c][j]
  const float s = *descale;
  const int j0 = blockIdx.x * kT, c0 = blockIdx.y * kT, bh = blockIdx.z;
  const uint16_t* xh = x + (size_t)bh * N * d;
  // load: thread -> (row j, 8 columns); 64 rows x 8 groups = 512 items, 2 per thread
  for (int item = threadIdx.x; item < kT * (kT / 8); item += blockDim.x) {
    const int jj = item >> 3, cg = (item & 7) * 8;
    const int j = j0 + jj;
    float f[8];
    if (j < N) {
      const uint4 w = *reinterpret_cast<const uint4*>(xh + (size_t)j * d + c0 + cg);
      const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        f[2 * e] = __fdiv_rn(bf16_lo(v[e]), s);
        f[2 * e + 1] = __fdiv_rn(bf16_hi(v[e]), s);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = 0.f;
    }
    const uint32_t lo = pack_e4m3x4(f[0], f[1], f[2], f[3]);
    const uint32_t hi = pack_e4m3x4(f[4], f[5], f[6], f[7]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      tile[cg + e][jj] = uint8_t(lo >> (8 * e));
      tile[cg + 4 + e][jj] = uint8_t(hi >> (8 * e));
    }
  }
  __syncthreads();
  // store: thread -> (row c, 16 positions j); 64 rows x 4 groups = 256 items
  const int cc = threadIdx.x >> 2, jg = (threadIdx.x & 3) * 16;
  const int j = j0 + jg;
  if (j >= ld) return;
  uint32_t w[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    w[e] = uint32_t(tile[cc][jg + 4 * e]) | (uint32_t(tile[cc][jg + 4 * e + 1]) << 8) |
           (uint32_t(tile[cc][jg + 4 * e + 2]) << 16) | (uint32_t(tile[cc][jg + 4 * e + 3]) << 24);
  // ld is a multiple of 16, so a group of 16 positions lies wholly inside or outside [0, ld)
  *reinterpret_cast<uint4*>(out + ((size_t)bh * d + c0 + cc) * ld + j) = make_uint4(w[0], w[1], w[2], w[3]);
}

unsigned grid_for(long long items) {
  const long long blocks = (items + 255) / 256;
  return unsigned(blocks < 152 * 8 ? (blocks > 0 ? blocks : 1) : 152 * 8);
}

}  // namespace

cudaError_t launch_e4m3_descale(const uint16_t* x, long long n, float* descale, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(descale, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  fa_absmax_kernel<<<grid_for(n / 8), 256, 0, s>>>(x, n, reinterpret_cast<unsigned int*>(descale));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fa_descale_finish_kernel<<<1, 1, 0, s>>>(descale);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const uint16_t* x, uint8_t* out, int BH, int N, int d, bool transpose, int ld,
                                 const float* descale, cudaStream_t s) {
  if (!transpose) {
    const long long n16 = (long long)BH * N * d / 16;
    fa_quant_kernel<<<grid_for(n16), 256, 0, s>>>(x, out, n16, descale);
  } else {
    const dim3 grid((ld + kT - 1) / kT, d / kT, BH);
    fa_quant_t_kernel<<<grid, 256, 0, s>>>(x, out, N, d, ld, descale);
  }
  return cudaGetLastError();
}

}  // namespace fa
