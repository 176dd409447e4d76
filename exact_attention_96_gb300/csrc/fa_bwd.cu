// fa_bwd.cu -- backward pass of exact attention on sm_103a.
//
// Only O and the per-row log-sum-exp were kept by the forward pass; S and P are recomputed
// block by block from Q, K, V ("FlashAttention 与显存" §09).  The gradients are those of
// O = softmax(scale * Q K^T) V:
//   dV = P^T dO,  dP = dO V^T,  D_i = rowsum(dO_i * O_i),  dS = P * (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Three launches on one stream:
//   1. fa_bwd_prep_kernel   D = rowsum(dO * O), LSE2 = LSE * log2(e) (both fp32, stored
//                           negated, rows padded to a multiple of 4), and a zeroed fp32 dQ
//                           accumulator.
//   2. fa_bwd_main_kernel   one CTA per tile of 128 keys of one (batch, head); it keeps K_j,
//                           V_j and the dK_j, dV_j accumulators on chip and loops over the
//                           query tiles, adding each tile's dQ contribution into the fp32
//                           accumulator in global memory (no second pass over S).
//   3. fa_bwd_dq_kernel     dQ accumulator * scale -> bf16 dQ.
//
// fa_bwd_main_kernel roles (448 threads; thread t of a warpgroup owns TMEM lane t):
//   warps 0-7   key rows, two warpgroups splitting each query tile's 128 columns in halves
//               of 64: P^T = 2^(S^T*scale*log2e - LSE2) (masked) -> bf16 into TMEM for the
//               dV product (kept in registers too); dS^T = P^T (dP^T - D) -> bf16 into
//               shared memory for the dK and dQ products; finally dV (first warpgroup) and
//               dK (second) -> bf16 -> TMA stores.
//   warps 8-11  dQ drain: read each finished dQ tile from TMEM and add it (fp32 vector
//               atomics, coalesced by the accumulator's tile layout) into global memory.
//   warp 12     TMA producer: K_j, V_j once; then Q_i, dO_i, LSE2_i, D_i through a ring.
//   warp 13     TMEM allocator and MMA issuer; per query tile i, in this order:
//                 dV  += P^T dO_i         (TS, P^T from TMEM inside the S^T columns)
//                 S^T_{i+1} = K_j Q^T     (SS, once dV_i has completed) -> TMEM [0,128)
//                 dQ_i = dS K_j           (SS, dS^T read M-major) -> TMEM [128,..), signalled
//                 dK  += dS^T Q_i         (SS, dS^T K-major)
//                 dP^T_{i+1} = V_j dO^T   (SS, once the drain has read the dQ_i columns under
//                                          it; at d = 128 in two halves of 64 queries, one per
//                                          key-row warpgroup) -> TMEM [128,256)
//   so the tensor core runs dV_i and S_{i+1} while the key rows compute dS_i, and dQ_i, dK_i
//   while they compute P_{i+1}.
// Persistent form (d = 64, non-causal, no dropout, at most 8 key tiles): one CTA per SM
// walks the (key tile, head) items w = blockIdx.x + r * gridDim.x.  Item r + 1's K, V and
// Q, dO loads start once item r's products have completed, while the key rows still read
// dV, dK out of TMEM; its first dV product waits for that read.  dV and dK are staged in the
// dS tile (idle between items) and stored by a drain warp.

// dQ accumulator layout (fp32): [B*H][q tile][d/4][128 rows][4] -- for a fixed group of four
// columns, the 128 rows of a tile are contiguous, so the 32 lanes of a warp adding one
// float4 each touch one contiguous 512-byte span.
//
// Dropout (template flag, d <= 128; "FlashAttention 与显存" §09: the mask is not stored but
// regenerated from the generator state): with Z = keep * scale_keep the gradients are
//   dV = (P * Z)^T dO,  dS = P * (dP * Z - D)   (D = rowsum(dO * O) as before).
// A key-row thread needs the keep bits of its key for 64 queries.  The eight lanes holding
// keys 8g .. 8g+7 share the generator calls of those keys: lane u draws the call of query
// 8b + u (8 bits, one per key), the octet exchanges its 8 bytes by shuffles and each lane
// takes its own bit column -- one call per lane per 8 queries, made before S^T is waited for
// (d = 128).  At d = 64 the dQ drain warps draw the next query tile's bits instead, one call
// per (8 keys, query), into a [key group][query] byte matrix in shared memory (two buffers);
// a key row gathers its 64 bits from 64 bytes.  Both give the same bits: the same generator
// call, coordinates and bit order.
// P^T * keep goes to TMEM for the dV product (scale_keep applied to dV at the end).

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ----------------------------------------------------------------- prep ----

template <int D>
__global__ void __launch_bounds__(256)
fa_bwd_prep_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                   const float* __restrict__ lse, float* __restrict__ dvec,
                   float* __restrict__ lse2, float* __restrict__ dq_acc, int N, int Np,
                   int n_q_tiles, int BH) {
  constexpr int kTPR = D / 8;              // threads per row, 8 elements each
  constexpr int kRowsPerBlock = 256 / kTPR;
  const int sub = threadIdx.x % kTPR;
  const long long prow = (long long)blockIdx.x * kRowsPerBlock + threadIdx.x / kTPR;  // padded row id
  const long long rows_padded = (long long)BH * n_q_tiles * 128;
  if (prow >= rows_padded) return;
  const int bh = int(prow / (n_q_tiles * 128));
  const int i = int(prow % (n_q_tiles * 128));

  // zero this row's part of the dQ accumulator (columns 8*sub .. 8*sub+7)
  if constexpr (D == 256) {  // row-major [B*H][padded rows][256]
    float4* row = reinterpret_cast<float4*>(dq_acc + (size_t)prow * D);
    row[2 * sub] = make_float4(0.f, 0.f, 0.f, 0.f);
    row[2 * sub + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {  // tile order [B*H][q tile][D/4][128][4]
    // Zeros have no layout: the block clears its rows' share (kRowsPerBlock rows of D floats,
    // whole tiles' worth over the grid) as one contiguous range, 32 bytes per thread.  (Zeroed
    // in the tile order, a warp's stores spread over 16 lines 2 KB apart: 4x16x8192x128
    // backward call 2.885 -> 2.866 ms.)
    float4* flat = reinterpret_cast<float4*>(dq_acc + (size_t)blockIdx.x * kRowsPerBlock * D);
    flat[2 * threadIdx.x] = make_float4(0.f, 0.f, 0.f, 0.f);
    flat[2 * threadIdx.x + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float acc = 0.f;
  if (i < N) {
    const size_t off = ((size_t)bh * N + i) * D + sub * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(o + off);
    const uint4 b = *reinterpret_cast<const uint4*>(dout + off);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(__uint_as_float(av[e] << 16), __uint_as_float(bv[e] << 16), acc);
      acc = fmaf(__uint_as_float(av[e] & 0xFFFF0000u), __uint_as_float(bv[e] & 0xFFFF0000u), acc);
    }
  }
#pragma unroll
  for (int w = kTPR / 2; w >= 1; w >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, w);
  if (sub == 0 && i < Np) {
    // stored negated: the main kernels add them with two-wide instructions
    dvec[(size_t)bh * Np + i] = (i < N) ? -acc : 0.f;
    lse2[(size_t)bh * Np + i] = (i < N) ? -(lse[(size_t)bh * N + i] * kLog2e) : 0.f;
  }
}

// ------------------------------------------------------------ dq convert ----

// dst[0..8) += scale * (a, b)
__device__ __forceinline__ void add_scaled8(float* dst, float4 a, float4 b, float scale) {
  float4* d4 = reinterpret_cast<float4*>(dst);
  float4 x = d4[0], y = d4[1];
  x.x += a.x * scale; x.y += a.y * scale; x.z += a.z * scale; x.w += a.w * scale;
  y.x += b.x * scale; y.y += b.y * scale; y.z += b.z * scale; y.w += b.w * scale;
  d4[0] = x;
  d4[1] = y;
}

// fp32 -> bf16, eight elements per thread (the tail element by element).
__global__ void __launch_bounds__(256)
fa_f32_to_bf16_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst, long long n) {
  const long long i0 = ((long long)blockIdx.x * 256 + threadIdx.x) * 8;
  if (i0 + 8 <= n) {
    const float4 a = *reinterpret_cast<const float4*>(src + i0);
    const float4 b = *reinterpret_cast<const float4*>(src + i0 + 4);
    *reinterpret_cast<uint4*>(dst + i0) =
        make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
  } else {
    for (long long i = i0; i < n; ++i) dst[i] = uint16_t(pack_bf16x2(src[i], 0.f) & 0xFFFFu);
  }
}

// With `dq_out` set (accumulate mode) scale * accumulator is added into that fp32 row-major
// buffer instead of being written as bf16: each element has one owner thread, and calls on one
// stream are ordered, so a plain read-add-write is enough.
template <int D>
__global__ void __launch_bounds__(256)
fa_bwd_dq_kernel(const float* __restrict__ dq_acc, uint16_t* __restrict__ dq, float* __restrict__ dq_out,
                 int N, int n_q_tiles, int BH, float scale) {
  constexpr int kK = D / 8;
  const long long gid = (long long)blockIdx.x * 256 + threadIdx.x;
  if constexpr (D == 256) {  // row-major accumulator: thread -> (padded row, 8 columns k)
    const long long prow = gid / kK;
    const int k = int(gid % kK);
    if (prow >= (long long)BH * n_q_tiles * 128) return;
    const int bh = int(prow / (n_q_tiles * 128));
    const int i = int(prow % (n_q_tiles * 128));
    if (i >= N) return;
    const float4* src = reinterpret_cast<const float4*>(dq_acc + (size_t)prow * D) + 2 * k;
    const float4 a = src[0], b = src[1];
    if (dq_out != nullptr) {
      add_scaled8(dq_out + ((size_t)bh * N + i) * D + k * 8, a, b, scale);
      return;
    }
    uint4 w;
    w.x = pack_bf16x2(a.x * scale, a.y * scale);
    w.y = pack_bf16x2(a.z * scale, a.w * scale);
    w.z = pack_bf16x2(b.x * scale, b.y * scale);
    w.w = pack_bf16x2(b.z * scale, b.w * scale);
    *reinterpret_cast<uint4*>(dq + ((size_t)bh * N + i) * D + k * 8) = w;
    return;
  }
  // tile-order accumulator: thread -> (tile row t = fastest, group of 8 columns k)
  const long long per_tile = 128LL * kK;
  const long long total = (long long)BH * n_q_tiles * per_tile;
  if (gid >= total) return;
  const long long tile = gid / per_tile;
  const int rem = int(gid % per_tile);
  const int t = rem & 127, k = rem >> 7;
  const int bh = int(tile / n_q_tiles), qt = int(tile % n_q_tiles);
  const int i = qt * 128 + t;
  if (i >= N) return;
  const float4* src = reinterpret_cast<const float4*>(dq_acc + (size_t)tile * 128 * D);
  const float4 a = src[(2 * k) * 128 + t];
  const float4 b = src[(2 * k + 1) * 128 + t];
  if (dq_out != nullptr) {
    add_scaled8(dq_out + ((size_t)bh * N + i) * D + k * 8, a, b, scale);
    return;
  }
  uint4 w;
  w.x = pack_bf16x2(a.x * scale, a.y * scale);
  w.y = pack_bf16x2(a.z * scale, a.w * scale);
  w.z = pack_bf16x2(b.x * scale, b.y * scale);
  w.w = pack_bf16x2(b.z * scale, b.w * scale);
  *reinterpret_cast<uint4*>(dq + ((size_t)bh * N + i) * D + k * 8) = w;
}

// ------------------------------------------------------------------ main ----

constexpr int kTile = 128;  // keys per CTA and queries per inner step
constexpr int kMainThreads = 448;
constexpr int kRowThreads = 256;     // warps 0-7: key rows, split into two column halves
constexpr int kDrainWarp0 = 8;       // warps 8-11: dQ drain
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;

template <int D, int NS>
struct BwdLayout {
  static constexpr int kSlabs = D / 64;
  static constexpr int kTileBytes = kTile * D * 2;   // one [128 x D] bf16 tile
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kTileBytes;
  static constexpr int kQOff = kVOff + kTileBytes;            // NS stages
  static constexpr int kdOOff = kQOff + NS * kTileBytes;      // NS stages
  static constexpr int kdSOff = kdOOff + NS * kTileBytes;     // [128 keys x 128 queries] bf16
  static constexpr int kdSBytes = kTile * kTile * 2;
  static constexpr int kLseOff = kdSOff + kdSBytes;           // NS x 128 fp32
  static constexpr int kDOff = kLseOff + NS * 512;            // NS x 128 fp32
  // D = 64: the dropout kernel's keep bits, drawn by the drain warps a tile ahead: two
  // buffers of [16 key groups][128 queries] bytes (bit u of byte [g][q]: key 8g + u)
  static constexpr int kBitsOff = kDOff + NS * 512;
  static constexpr int kBitsBytes = D == 64 ? 2 * 16 * kTile : 0;
  static constexpr int kBarOff = kBitsOff + kBitsBytes;
  static constexpr int kBarKV = 0;
  static constexpr int kBarQFull = 1;
  static constexpr int kBarQEmpty = kBarQFull + NS;
  static constexpr int kBarSFull = kBarQEmpty + NS;
  static constexpr int kHalves = D == 64 ? 1 : 2;  // dP products (one per query half at D = 128)
  static constexpr int kBarDPFull = kBarSFull + 1;    // kHalves
  static constexpr int kBarPReady = kBarDPFull + kHalves;
  static constexpr int kBarDSReady = kBarPReady + 1;
  static constexpr int kBarDVDone = kBarDSReady + 1;
  static constexpr int kBarDQFull = kBarDVDone + 1;
  static constexpr int kBarDQDrained = kBarDQFull + 1;  // kHalves: one per 64-column half of dQ
  static constexpr int kBarDSFree = kBarDQDrained + kHalves;
  static constexpr int kBarAccDone = kBarDSFree + 1;
  static constexpr int kBarEpi = kBarAccDone + 1;   // 2: one per column half
  static constexpr int kBarDrain = kBarEpi + 2;
  static constexpr int kBarBitsFull = kBarDrain + 1;   // 2: one per bits buffer
  static constexpr int kBarBitsFree = kBarBitsFull + 2;  // 2
  static constexpr int kBarEpiRead = kBarBitsFree + 2;    // key rows have read dV, dK from TMEM
  static constexpr int kBarStageFree = kBarEpiRead + 1;   // the stores have read the staging tiles
  static constexpr int kNumBars = kBarStageFree + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  // TMEM columns
  static constexpr int kColS = 0;      // S^T, then P^T (bf16 pairs) packed inside it
  static constexpr int kColDP = 128;   // dP^T, then the dQ tile
  static constexpr int kColDV = 256;
  static constexpr int kColDK = 256 + D;
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kStageTx = 2 * kTileBytes + 2 * 512;
  static_assert(256 + 2 * D <= 512, "TMEM budget");
  static_assert(kBytes <= 232448, "shared memory budget");
};

template <int D, int NS, bool CAUSAL, bool DROPOUT, bool PERSIST>
__global__ void __launch_bounds__(kMainThreads, 1)
fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const __grid_constant__ CUtensorMap tmLse2, const __grid_constant__ CUtensorMap tmD,
                   const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                   const BwdArgs args) {
  using L = BwdLayout<D, NS>;
  // D = 64 with dropout: the keep bits come from the drain warps, which have the issue slots to
  // spare, instead of 8 generator calls per tile in each key-row thread (16x8x4096x64 backward
  // with dropout 391 -> 444 TFLOP/s).  D = 128 has no shared memory left for the 4 KB of
  // buffers and keeps the key rows' own draws.
  constexpr bool kBitsFromDrain = DROPOUT && D == 64;
  // PERSIST (D = 64, non-causal, no dropout): one CTA per SM walks a list of (key tile, head)
  // items, so that an item's K / V loads and first products overlap the previous item's dK /
  // dV epilogue, and the CTA's set-up and teardown are paid once.  Every per-tile barrier
  // phase then counts tiles across items (g = items done x tiles per item + tile); the
  // per-item ones (K / V, accumulators done, epilogue) count items.
  constexpr bool kPersist = PERSIST;
  static_assert(!PERSIST || (D == 64 && !CAUSAL && !DROPOUT), "persistent form: d = 64, non-causal, no dropout");
  // key-row column halves unrolled (see the key rows)
  constexpr bool kUnrollHalves = D == 64 && (!CAUSAL || DROPOUT);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_addr(smem_raw);
  if (base & 1023u) {  // the 128-byte swizzle needs 1024-byte aligned tiles
    if (threadIdx.x == 0) atomicOr(args.err_word, 2);
    return;
  }
  uint8_t* smem = smem_raw;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // causal: key tile 0 (seen by every query tile) is the heaviest; heads in small groups
  const RankHead rh = CAUSAL ? causal_dispatch_order() : RankHead{int(blockIdx.x), int(blockIdx.y)};
  int bh = rh.bh;
  int kv_tile = rh.rank;
  int k0 = kv_tile * kTile;
  const int N = args.N;
  const int n_q_tiles = (N + kTile - 1) / kTile;
  const int it_first = CAUSAL ? kv_tile : 0;  // query tiles before the diagonal see none of these keys
  const int n_it = n_q_tiles - it_first;
  // items of this CTA: w = blockIdx.x + r * gridDim.x (persistent), else the one of the grid
  const int n_items = kPersist ? n_q_tiles * args.BH : 1;
  auto set_item = [&](int r) -> bool {  // false when this CTA has no r-th item
    if constexpr (kPersist) {
      const int w = int(blockIdx.x) + r * int(gridDim.x);
      if (w >= n_items) return false;
      kv_tile = w % n_q_tiles;
      bh = w / n_q_tiles;
      k0 = kv_tile * kTile;
      return true;
    } else {
      return r == 0;
    }
  };

  auto bar = [&](int i) -> uint32_t { return base + L::kBarOff + 8u * uint32_t(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const WaitCtl wc{abort_flag, args.err_word, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kBarKV), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(L::kBarQFull + s), 1);
      mbar_init(bar(L::kBarQEmpty + s), kRowThreads + 1);  // key-row warps + MMA commit
    }
    mbar_init(bar(L::kBarSFull), 1);
    for (int h = 0; h < L::kHalves; ++h) mbar_init(bar(L::kBarDPFull + h), 1);
    mbar_init(bar(L::kBarPReady), kRowThreads);
    mbar_init(bar(L::kBarDSReady), kRowThreads);
    mbar_init(bar(L::kBarDVDone), 1);
    mbar_init(bar(L::kBarDQFull), 1);
    for (int h = 0; h < L::kHalves; ++h) mbar_init(bar(L::kBarDQDrained + h), 128);
    mbar_init(bar(L::kBarDSFree), 1);
    mbar_init(bar(L::kBarAccDone), 1);
    mbar_init(bar(L::kBarEpi + 0), 128);
    mbar_init(bar(L::kBarEpi + 1), 128);
    mbar_init(bar(L::kBarDrain), 1);
    if constexpr (kPersist) {  // (in the one-item kernel these two inits alone cost 0.8 %)
      mbar_init(bar(L::kBarEpiRead), kRowThreads);
      mbar_init(bar(L::kBarStageFree), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::kBarBitsFull + b), 128);         // drain warps
      mbar_init(bar(L::kBarBitsFree + b), kRowThreads);  // key rows
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sK = base + L::kKOff, sV = base + L::kVOff, sdS = base + L::kdSOff;
  auto sQ = [&](int s) -> uint32_t { return base + L::kQOff + uint32_t(s) * L::kTileBytes; };
  auto sdO = [&](int s) -> uint32_t { return base + L::kdOOff + uint32_t(s) * L::kTileBytes; };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer ----
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      int arms[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s) arms[s] = 0;
      bool ok = true;
      int kv_arms = 0;
      for (int r = 0; ok && set_item(r); ++r) {
      // K and V of the item, once every product of the previous one has completed
      if (r > 0 && !mbar_wait(bar(L::kBarAccDone), (r - 1) & 1, wc)) { ok = false; break; }
      mbar_arrive_expect_tx(bar(L::kBarKV), 2 * L::kTileBytes);
      for (int s = 0; s < L::kSlabs; ++s) {
        tma_load_3d(sK + s * (kTile * 128), &tmK, bar(L::kBarKV), s * 64, k0, bh);
        tma_load_3d(sV + s * (kTile * 128), &tmV, bar(L::kBarKV), s * 64, k0, bh);
      }
      ++kv_arms;
      const int g0 = r * n_it;
      for (int it = 0; it < n_it; ++it) {
        const int gt = g0 + it;
        const int st = gt % NS;
        if (gt >= NS && !mbar_wait(bar(L::kBarQEmpty + st), ((gt / NS) - 1) & 1, wc)) { ok = false; break; }
        const int q0 = (it_first + it) * kTile;
        const uint32_t fb = bar(L::kBarQFull + st);
        mbar_arrive_expect_tx(fb, L::kStageTx);
        for (int s = 0; s < L::kSlabs; ++s) {
          tma_load_3d(sQ(st) + s * (kTile * 128), &tmQ, fb, s * 64, q0, bh);
          tma_load_3d(sdO(st) + s * (kTile * 128), &tmdO, fb, s * 64, q0, bh);
        }
        tma_load_3d(base + L::kLseOff + st * 512, &tmLse2, fb, q0, bh, 0);
        tma_load_3d(base + L::kDOff + st * 512, &tmD, fb, q0, bh, 0);
        ++arms[st];
      }
      }
      if (!ok) {
        auto drain = [&](uint32_t b, uint32_t parity) {
          for (uint64_t t0 = global_timer_ns();
               !mbar_try_wait(b, parity) && global_timer_ns() - t0 < wc.limit_ns;) {
          }
        };
        if (kv_arms > 0) drain(bar(L::kBarKV), (kv_arms - 1) & 1);
        for (int s = 0; s < NS; ++s)
          if (arms[s] > 0) drain(bar(L::kBarQFull + s), (arms[s] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------- MMA issuer ----
    // Order per query tile i:  dV_i | S_{i+1} | dK_i, dQ_i | dP_{i+1}
    // so that the key-row warps turn S_{i+1} into P_{i+1} while dK_i and dQ_i run.
    if (lane == 0) {
      constexpr uint32_t kIdSq = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, D, 0, 1);   // dV, dK: B N-major
      constexpr uint32_t kIdDQ = idesc_bf16_f32(128, D, 1, 1);    // dQ: A (dS) M-major, B N-major
      auto issue_s = [&](int it) -> bool {
        const int st = it % NS;
        if (!mbar_wait(bar(L::kBarQFull + st), (it / NS) & 1, wc)) return false;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
          mma_ss(tmem + L::kColS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ(st) + off, 16, 1024),
                 kIdSq, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kBarSFull));
        return true;
      };
      // D = 128: dP^T in two halves of 64 queries (columns kColDP + 64h), each with its own
      // signal: key-row warpgroup h reads only its half, and half h starts as soon as the drain
      // has read the dQ columns it overwrites (4x16x8192x128 causal: 933 -> 944 TFLOP/s).
      // D = 64: one 128-query product read by both warpgroups (halves measured 8 % slower:
      // the narrower products cost more than the earlier start gains).
      constexpr uint32_t kIdDPh = idesc_bf16_f32(128, 64, 0, 0);
      auto issue_dp = [&](int it) {
        const int st = it % NS;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
          mma_ss(tmem + L::kColDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sdO(st) + off, 16, 1024),
                 kIdSq, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kBarDPFull));
      };
      auto issue_dp_half = [&](int it, int h) {
        const int st = it % NS;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
          mma_ss(tmem + L::kColDP + 64 * h, sdesc_sw128(sV + off, 16, 1024),
                 sdesc_sw128(sdO(st) + off + h * (64 * 128), 16, 1024), kIdDPh, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kBarDPFull + h));
      };
      if constexpr (kPersist) {
        bool ok = true;
        for (int r = 0; ok && set_item(r); ++r) {
        const int g0 = r * n_it;
        ok = mbar_wait(bar(L::kBarKV), r & 1, wc) && issue_s(g0);
        // dP of the item's first tile overwrites the previous item's last dQ tile
        if (ok && r > 0) ok = mbar_wait(bar(L::kBarDQDrained), (g0 - 1) & 1, wc);
        if (ok) {
          if constexpr (D == 64) {
            issue_dp(g0);
          } else {
            issue_dp_half(g0, 0);
            issue_dp_half(g0, 1);
          }
        }
        for (int it = 0; ok && it < n_it; ++it) {
          const int gt = g0 + it;
          const int st = gt % NS;
          const uint32_t ph = gt & 1;
          if (!mbar_wait(bar(L::kBarPReady), ph, wc)) { ok = false; break; }
          // the item's first dV overwrites the accumulators: the key rows must have read the
          // previous item's out of TMEM
          if (kPersist && it == 0 && r > 0 && !mbar_wait(bar(L::kBarEpiRead), (r - 1) & 1, wc)) { ok = false; break; }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            // P^T of queries 16kk..16kk+15 sits in 8 columns of its half's S^T range
            mma_ts(tmem + L::kColDV, tmem + L::kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                   sdesc_sw128(sdO(st) + kk * (16 * 128), kTile * 128, 1024), kIdAcc,
                   (it > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(L::kBarDVDone));
          // S_{i+1} overwrites P^T_i, whose only reader is the dV product (the key-row warps
          // keep their own copy of P in registers): issue it as soon as dV_i has completed, so
          // the tensor core runs dV_i and S_{i+1} while the key rows compute dS_i.
          if (it + 1 < n_it && !(mbar_wait(bar(L::kBarDVDone), ph, wc) && issue_s(gt + 1))) {
            ok = false;
            break;
          }
          if (!mbar_wait(bar(L::kBarDSReady), ph, wc)) { ok = false; break; }
          tc_fence_after_sync();
          // dQ_i first, with its own completion signal, so the drain warps read it while dK_i
          // runs and dP_{i+1} (which reuses its columns) can follow dK_i without a gap.
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            mma_ss(tmem + L::kColDP, sdesc_sw128(sdS + kk * (16 * 128), kTile * 128, 1024),
                   sdesc_sw128(sK + kk * (16 * 128), kTile * 128, 1024), kIdDQ, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(L::kBarDQFull));
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t a_off = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;  // dS^T K-major
            mma_ss(tmem + L::kColDK, sdesc_sw128(sdS + a_off, 16, 1024),
                   sdesc_sw128(sQ(st) + kk * (16 * 128), kTile * 128, 1024), kIdAcc,
                   (it > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(L::kBarDSFree));
          mma_commit(bar(L::kBarQEmpty + st));
          // dP_{i+1} overwrites the dQ_i tile: each product waits until the drain warps have
          // read the dQ columns under it.  (At D = 64 the accumulators leave 128 TMEM columns
          // free.  Giving the dQ tile 64 of them, with dP_{i+1} issued ahead of dQ_i and dK_i,
          // measured slower: 1x8x65536x64 causal 764 -> 752 TFLOP/s, 16x8x4096x64 non-causal
          // 792 -> 710.)
          if (it + 1 < n_it) {
            if (!mbar_wait(bar(L::kBarDQDrained + 0), ph, wc)) { ok = false; break; }
            if constexpr (D == 64) {
              issue_dp(gt + 1);
            } else {
              issue_dp_half(gt + 1, 0);
              if (!mbar_wait(bar(L::kBarDQDrained + 1), ph, wc)) { ok = false; break; }
              issue_dp_half(gt + 1, 1);
            }
          }
        }
        if (ok) mma_commit(bar(L::kBarAccDone));
        }
      } else {
        // one item (an item loop around this, even one that runs once, measured 3 % slower
        // at 16x8x4096x64: the issuing thread is on the critical path)
        bool ok = mbar_wait(bar(L::kBarKV), 0, wc) && issue_s(0);
        if (ok) {
          if constexpr (D == 64) {
            issue_dp(0);
          } else {
            issue_dp_half(0, 0);
            issue_dp_half(0, 1);
          }
        }
        for (int it = 0; ok && it < n_it; ++it) {
          const int st = it % NS;
          const uint32_t ph = it & 1;
          if (!mbar_wait(bar(L::kBarPReady), ph, wc)) { ok = false; break; }
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            // P^T of queries 16kk..16kk+15 sits in 8 columns of its half's S^T range
            mma_ts(tmem + L::kColDV, tmem + L::kColS + (kk >> 2) * 64 + (kk & 3) * 8,
                   sdesc_sw128(sdO(st) + kk * (16 * 128), kTile * 128, 1024), kIdAcc,
                   (it > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(L::kBarDVDone));
          // S_{i+1} overwrites P^T_i, whose only reader is the dV product (the key-row warps
          // keep their own copy of P in registers): issue it as soon as dV_i has completed, so
          // the tensor core runs dV_i and S_{i+1} while the key rows compute dS_i.
          if (it + 1 < n_it && !(mbar_wait(bar(L::kBarDVDone), ph, wc) && issue_s(it + 1))) {
            ok = false;
            break;
          }
          if (!mbar_wait(bar(L::kBarDSReady), ph, wc)) { ok = false; break; }
          tc_fence_after_sync();
          // dQ_i first, with its own completion signal, so the drain warps read it while dK_i
          // runs and dP_{i+1} (which reuses its columns) can follow dK_i without a gap.
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            mma_ss(tmem + L::kColDP, sdesc_sw128(sdS + kk * (16 * 128), kTile * 128, 1024),
                   sdesc_sw128(sK + kk * (16 * 128), kTile * 128, 1024), kIdDQ, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(L::kBarDQFull));
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t a_off = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;  // dS^T K-major
            mma_ss(tmem + L::kColDK, sdesc_sw128(sdS + a_off, 16, 1024),
                   sdesc_sw128(sQ(st) + kk * (16 * 128), kTile * 128, 1024), kIdAcc,
                   (it > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(L::kBarDSFree));
          mma_commit(bar(L::kBarQEmpty + st));
          // dP_{i+1} overwrites the dQ_i tile: each product waits until the drain warps have
          // read the dQ columns under it.  (At D = 64 the accumulators leave 128 TMEM columns
          // free.  Giving the dQ tile 64 of them, with dP_{i+1} issued ahead of dQ_i and dK_i,
          // measured slower: 1x8x65536x64 causal 764 -> 752 TFLOP/s, 16x8x4096x64 non-causal
          // 792 -> 710.)
          if (it + 1 < n_it) {
            if (!mbar_wait(bar(L::kBarDQDrained + 0), ph, wc)) { ok = false; break; }
            if constexpr (D == 64) {
              issue_dp(it + 1);
            } else {
              issue_dp_half(it + 1, 0);
              if (!mbar_wait(bar(L::kBarDQDrained + 1), ph, wc)) { ok = false; break; }
              issue_dp_half(it + 1, 1);
            }
          }
        }
        if (ok) mma_commit(bar(L::kBarAccDone));
      }
      mma_commit(bar(L::kBarDrain));
      for (uint64_t t0 = global_timer_ns();
           !mbar_try_wait(bar(L::kBarDrain), 0) && global_timer_ns() - t0 < wc.limit_ns;) {
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ key rows ----
    // Two warpgroups split the 128 query columns of each tile: half h owns queries
    // [64h, 64h + 64).  P^T for query q (bf16 pairs) is packed into TMEM column
    // 64*(q/64) + (q%64)/2, inside the S^T columns the same warpgroup has already read.
    const int t = threadIdx.x & 127;       // key row within the tile = TMEM lane
    const int half = threadIdx.x >> 7;     // 0 or 1
    const int c0 = half * 64;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const float sl2 = args.scale_log2;
    bool ok = true;
    for (int r = 0; ok && set_item(r); ++r) {
    const int key = k0 + t;
    const int g0 = r * n_it;
    for (int it = 0; it < n_it; ++it) {
      const int gt = g0 + it;
      const int st = gt % NS;
      const uint32_t ph = gt & 1;
      const int q0 = (it_first + it) * kTile;
      const bool edge = (CAUSAL && it == 0) || (q0 + kTile > N);  // any masking in this tile
      const float* lse2 = reinterpret_cast<const float*>(smem + L::kLseOff + st * 512) + c0;
      const float* dvv = reinterpret_cast<const float*>(smem + L::kDOff + st * 512) + c0;
      uint32_t km[2] = {0u, 0u};  // dropout keep bits: bit c % 32 of word c / 32 = query q0 + c0 + c
      if constexpr (kBitsFromDrain) {
        // bytes [t / 8][c0 .. c0 + 63] of this tile's matrix; bit t % 8 of each is this key's
        const int bb = it & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(L::kBarBitsFull + bb), (it >> 1) & 1, wc))) { ok = false; break; }
        const uint4* src = reinterpret_cast<const uint4*>(smem + L::kBitsOff + bb * (16 * kTile) + (t >> 3) * kTile + c0);
        const uint32_t u = uint32_t(t & 7);
        uint64_t bits = 0;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 w = src[v];
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)  // bit u of each of the word's four bytes -> a nibble
            bits |= uint64_t((((ws[e] >> u) & 0x01010101u) * 0x01020408u) >> 24) << (16 * v + 4 * e);
        }
        mbar_arrive(bar(L::kBarBitsFree + bb));
        km[0] = uint32_t(bits);
        km[1] = uint32_t(bits >> 32);
      } else if constexpr (DROPOUT) {
        const uint64_t bits = dropout_key_bits<8>(args.dropout, key, q0 + c0, bh, lane);
        km[0] = uint32_t(bits);
        km[1] = uint32_t(bits >> 32);
        // keep the generator work here, ahead of the S^T wait, instead of letting it sink into
        // the register-heavy conversion below
        asm volatile("" : "+r"(km[0]), "+r"(km[1]));
      }
      // phase 1: P^T
      if (!__all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull), ph, wc))) { ok = false; break; }
      tc_fence_after_sync();
      // The two 32-column halves of this warpgroup's 64 query columns run as a rolled loop
      // (phase 2 likewise) for D = 128 and for the causal D = 64 kernel: unrolled, the key-row
      // code (with the diagonal tile's masking) crowds the instruction cache that the drain,
      // producer and MMA warps share (measured: 4x16x8192x128 causal backward 815 -> 895
      // TFLOP/s; 1x8x65536x64 causal 655 -> 715).  The non-causal D = 64 kernel, and its
      // dropout form, are smaller and run faster unrolled (16x8x4096x64: 775 against 676).
      // P^T of each half (bf16 pairs) is kept for phase 2 in its own register array, selected
      // without run-time indexing.
      uint32_t pk0[16], pk1[16];
#pragma unroll(kUnrollHalves ? 2 : 1)
      for (int cc = 0; cc < 64; cc += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + L::kColS + c0 + cc, r);
        float lv[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 x = *reinterpret_cast<const float4*>(lse2 + cc + e);
          lv[e] = x.x; lv[e + 1] = x.y; lv[e + 2] = x.z; lv[e + 3] = x.w;
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          // lv holds -LSE * log2(e): two keys' exponents in one instruction
          const float2 x = ffma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                 make_float2(sl2, sl2), make_float2(lv[e], lv[e + 1]));
          w[e / 2] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
        }
        if (edge) apply_keep_mask(w, visible_bits(q0 + c0 + cc, CAUSAL ? key : 0, N));
        if (cc == 0) {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk0[e] = w[e];
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk1[e] = w[e];
        }
        if constexpr (DROPOUT) {  // the dV product sees P^T * keep
          const uint32_t kmw = cc == 0 ? km[0] : km[1];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint32_t kb = kmw >> (2 * e);
            w[e] &= ((kb & 1u) ? 0x0000FFFFu : 0u) | ((kb & 2u) ? 0xFFFF0000u : 0u);
          }
        }
        tmem_st16(tmem + lane_off + L::kColS + c0 + cc / 2, w);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kBarPReady));
      // phase 2: dS^T = P^T (dP^T - D)
      bool got = mbar_wait(bar(L::kBarDPFull + (L::kHalves > 1 ? half : 0)), ph, wc);
      if (gt > 0) got = got && mbar_wait(bar(L::kBarDSFree), ph ^ 1, wc);
      // persistent: the previous item's dV, dK stores must have read their staging in dS
      if (kPersist && it == 0 && r > 0) got = got && mbar_wait(bar(L::kBarStageFree), (r - 1) & 1, wc);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after_sync();
#pragma unroll(kUnrollHalves ? 2 : 1)
      for (int cc = 0; cc < 64; cc += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + L::kColDP + c0 + cc, r);
        uint32_t pr[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pr[e] = cc == 0 ? pk0[e] : pk1[e];
        [[maybe_unused]] const uint32_t kmw = cc == 0 ? km[0] : km[1];
        float dl[32];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 x = *reinterpret_cast<const float4*>(dvv + cc + e);
          dl[e] = x.x; dl[e + 1] = x.y; dl[e + 2] = x.z; dl[e + 3] = x.w;
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = __uint_as_float(pr[e / 2] << 16);
          const float p1 = __uint_as_float(pr[e / 2] & 0xFFFF0000u);
          float dp0 = __uint_as_float(r[e]), dp1 = __uint_as_float(r[e + 1]);
          if constexpr (DROPOUT) {
            const uint32_t kb = kmw >> e;
            dp0 = (kb & 1u) ? dp0 * args.dropout.scale : 0.f;
            dp1 = (kb & 2u) ? dp1 * args.dropout.scale : 0.f;
          }
          // dl holds -D: dS = P (dP - D) two at a time
          const float2 ds = fmul2(make_float2(p0, p1), fadd2(make_float2(dp0, dp1), make_float2(dl[e], dl[e + 1])));
          w[e / 2] = pack_bf16x2(ds.x, ds.y);
        }
        if (q0 + kTile > N) apply_keep_mask(w, visible_bits(q0 + c0 + cc, 0, N));
        // dS^T row t, queries c0+cc .. c0+cc+31 -> slab `half`, 16-byte chunks cc/8 ..
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int phys = ((cc >> 3) + i) ^ (t & 7);
          *reinterpret_cast<uint4*>(smem + L::kdSOff + half * (kTile * 128) + t * 128 + phys * 16) =
              make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kBarDSReady));
      mbar_arrive(bar(L::kBarQEmpty + st));
    }
    // epilogue: half 0 stores dV, half 1 stores dK (scaled), each staged in a free stage-0
    // tile and written by one TMA store per 64-column slab
    bool fin = ok && __all_sync(0xffffffffu, mbar_wait(bar(L::kBarAccDone), r & 1, wc));
    const uint32_t col = half == 0 ? L::kColDV : L::kColDK;
    const float mul = half == 0 ? (DROPOUT ? args.dropout.scale : 1.f) : args.scale;
    // the persistent kernel stages in the dS tile (free once the item's products are done):
    // the stage-0 Q, dO tiles may already hold the next item's loads
    uint8_t* stage = kPersist ? smem + L::kdSOff + half * L::kTileBytes : smem + (half == 0 ? L::kQOff : L::kdOOff);
    const bool accum = args.dk_accum != nullptr;
    if (fin && accum) {
      // accumulate mode: add the fp32 rows into the caller's buffers (vector atomics)
      tc_fence_after_sync();
      float4* dst = reinterpret_cast<float4*>((half == 0 ? args.dv_accum : args.dk_accum) +
                                              ((size_t)bh * N + key) * D);
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + col + c, r);
        if (key < N) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            atomicAdd(dst + c / 4 + e, make_float4(__uint_as_float(r[4 * e]) * mul, __uint_as_float(r[4 * e + 1]) * mul,
                                                   __uint_as_float(r[4 * e + 2]) * mul, __uint_as_float(r[4 * e + 3]) * mul));
        }
      }
    } else if (fin) {
      tc_fence_after_sync();
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + col + c, r);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
        const int slab = c >> 6;
        const int chunk0 = (c & 63) >> 3;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int phys = (chunk0 + i) ^ (t & 7);
          *reinterpret_cast<uint4*>(stage + slab * (kTile * 128) + t * 128 + phys * 16) =
              make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      fence_proxy_async_smem();
    }
    if constexpr (kPersist) {  // dV, dK are out of TMEM: the next item's products may overwrite them
      tc_fence_before_sync();
      mbar_arrive(bar(L::kBarEpiRead));
    }
    mbar_arrive(bar(L::kBarEpi + half));
    if (!kPersist && t == 0 && fin && !accum && mbar_wait(bar(L::kBarEpi + half), 0, wc) && *abort_flag == 0) {
      const CUtensorMap* map = half == 0 ? &tmdV : &tmdK;
      const uint32_t src = half == 0 ? sQ(0) : sdO(0);
      for (int s = 0; s < L::kSlabs; ++s) tma_store_3d(map, src + s * (kTile * 128), s * 64, k0, bh);
      bulk_commit_group();
      bulk_wait_group_read_all();  // source read: the CTA may exit
    }
    if (!fin) ok = false;
    }
  } else if (warp < kProducerWarp) {
    // --------------------------------------------------------- dQ drain ----
    const int t = threadIdx.x - kDrainWarp0 * 32;   // query row within the tile = TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    // D = 64 with dropout: draw the keep bits of query tile `i` for this CTA's 128 keys, query
    // row t of the tile: byte [g][t] = keep bits of keys k0 + 8g .. k0 + 8g + 7
    [[maybe_unused]] auto draw_bits = [&](int i) {
      uint8_t* dst = smem + L::kBitsOff + (i & 1) * (16 * kTile) + t;
      const uint32_t q = uint32_t((it_first + i) * kTile + t);
#pragma unroll 4
      for (int g = 0; g < 16; ++g)
        dst[g * kTile] = uint8_t(dropout_keep8(args.dropout, uint32_t((k0 >> 3) + g), q, uint32_t(bh)));
      mbar_arrive(bar(L::kBarBitsFull + (i & 1)));
    };
    if constexpr (kBitsFromDrain) draw_bits(0);
    bool dok = true;
    for (int r = 0; dok && set_item(r); ++r) {
    const int g0 = r * n_it;
    for (int it = 0; it < n_it; ++it) {
      const int qt = it_first + it;
      if constexpr (kBitsFromDrain) {
        // the next tile's bits, into the buffer the key rows released after tile it - 1
        if (it + 1 < n_it) {
          if (it >= 1 && !__all_sync(0xffffffffu, mbar_wait(bar(L::kBarBitsFree + ((it + 1) & 1)), ((it - 1) >> 1) & 1, wc)))
            break;
          draw_bits(it + 1);
        }
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(L::kBarDQFull), (g0 + it) & 1, wc))) { dok = false; break; }
      tc_fence_after_sync();
      float4* dst = reinterpret_cast<float4*>(args.dq_acc + ((size_t)bh * n_q_tiles + qt) * 128 * D);
      const bool live = qt * kTile + t < N;
#pragma unroll
      for (int h = 0; h < D / 64; ++h) {
        uint32_t a[32], b[32];
        tmem_ld32(tmem + lane_off + L::kColDP + 64 * h, a);
        tmem_ld32(tmem + lane_off + L::kColDP + 64 * h + 32, b);
        // these 64 columns are in registers: the dP half over them may be written
        tc_fence_before_sync();
        mbar_arrive(bar(L::kBarDQDrained + h));
        if (live) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            atomicAdd(dst + (16 * h + g) * 128 + t,
                      make_float4(__uint_as_float(a[4 * g]), __uint_as_float(a[4 * g + 1]),
                                  __uint_as_float(a[4 * g + 2]), __uint_as_float(a[4 * g + 3])));
            atomicAdd(dst + (16 * h + 8 + g) * 128 + t,
                      make_float4(__uint_as_float(b[4 * g]), __uint_as_float(b[4 * g + 1]),
                                  __uint_as_float(b[4 * g + 2]), __uint_as_float(b[4 * g + 3])));
          }
        }
      }
    }
    if constexpr (kPersist) {
      // the item's dV and dK stores from the staging tiles, once both key-row halves have
      // written them; the staging tiles are free again when the stores have read them
      if (warp == kDrainWarp0) {
        if (lane == 0) {
          const bool got = dok && mbar_wait(bar(L::kBarEpi + 0), r & 1, wc) && mbar_wait(bar(L::kBarEpi + 1), r & 1, wc);
          if (got && args.dk_accum == nullptr && *abort_flag == 0) {
            tma_store_3d(&tmdV, base + L::kdSOff, 0, k0, bh);
            tma_store_3d(&tmdK, base + L::kdSOff + L::kTileBytes, 0, k0, bh);
            bulk_commit_group();
            bulk_wait_group_read_all();
          }
          mbar_arrive(bar(L::kBarStageFree));
        }
        __syncwarp();
      }
    }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Sequences of at most this many key tiles take the persistent form of the d = 64
// non-causal backward: there a CTA's set-up, K / V loads and epilogue are a large part of
// its few query tiles (backward, TFLOP/s: 128x16x512 457 -> 517, 64x16x1024 608 -> 645).
// Longer ones keep one CTA per item: at 16 key tiles both forms ran alike, at 32 the
// persistent one was 2 % slower (16x8x4096: 797 -> 779), with static item lists and the
// K / V loads of an item waiting for the previous item's products.
constexpr int kPersistMaxTiles = 8;

template <int D, int NS, bool CAUSAL>
cudaError_t launch_main(const BwdMaps& m, const CUtensorMap& lse2, const CUtensorMap& dmap,
                        const CUtensorMap& dk, const CUtensorMap& dv, const BwdArgs& a, cudaStream_t s,
                        bool dropout) {
  using L = BwdLayout<D, NS>;
  constexpr bool kCanPersist = D == 64 && !CAUSAL;
  dim3 grid((a.N + kTile - 1) / kTile, a.BH);
  const bool persist = kCanPersist && !dropout && int(grid.x) <= kPersistMaxTiles;
  auto kern = dropout   ? fa_bwd_main_kernel<D, NS, CAUSAL, true, false>
              : persist ? fa_bwd_main_kernel<D, NS, CAUSAL, false, kCanPersist>
                        : fa_bwd_main_kernel<D, NS, CAUSAL, false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
  if (e != cudaSuccess) return e;
  if (persist) {  // one CTA per SM over every (key tile, head) item
    static int sms = 0;
    if (sms == 0) {
      int dev = 0;
      if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
      if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    }
    const int items = int(grid.x * grid.y);
    grid = dim3(unsigned(items < sms ? items : sms), 1);
  }
  kern<<<grid, kMainThreads, L::kBytes, s>>>(m.q, m.k, m.v, m.dout, lse2, dmap, dk, dv, a);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_prep_and_convert(const BwdArgs& a, int Np, int n_q_tiles, cudaStream_t s, bool prep) {
  if (prep) {
    constexpr int kRowsPerBlock = 256 / (D / 8);
    const long long rows = (long long)a.BH * n_q_tiles * 128;
    const unsigned grid = unsigned((rows + kRowsPerBlock - 1) / kRowsPerBlock);
    fa_bwd_prep_kernel<D><<<grid, 256, 0, s>>>(a.o, a.dout, a.lse, a.dvec, a.lse2,
                                               a.dq_acc, a.N, Np, n_q_tiles, a.BH);
  } else {
    const long long total = (long long)a.BH * n_q_tiles * 128 * (D / 8);
    const unsigned grid = unsigned((total + 255) / 256);
    fa_bwd_dq_kernel<D><<<grid, 256, 0, s>>>(a.dq_acc, a.dq, a.dq_accum, a.N, n_q_tiles, a.BH, a.scale);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_f32_to_bf16(const float* src, uint16_t* dst, long long n, cudaStream_t s) {
  const long long threads = (n + 7) / 8;
  fa_f32_to_bf16_kernel<<<unsigned((threads + 255) / 256), 256, 0, s>>>(src, dst, n);
  return cudaGetLastError();
}

// Workspace: [D: BH x Np][LSE2: BH x Np][dQ accumulator: BH x n_q_tiles x 128 x d], fp32
// (tile order for d <= 128, row-major for d = 256).
cudaError_t launch_bwd_all(const BwdMaps& m, const CUtensorMap& lse2, const CUtensorMap& dmap,
                           const CUtensorMap& dk, const CUtensorMap& dv, const BwdArgs& a, bool causal,
                           int Np, cudaStream_t s, bool dropout, const cudaEvent_t* main_events) {
  const int n_q_tiles = (a.N + kTile - 1) / kTile;
  if (a.d != 64 && a.d != 128 && a.d != 256) return cudaErrorInvalidValue;
  cudaError_t e;
  switch (a.d) {
    case 64: e = launch_prep_and_convert<64>(a, Np, n_q_tiles, s, true); break;
    case 128: e = launch_prep_and_convert<128>(a, Np, n_q_tiles, s, true); break;
    default: e = launch_prep_and_convert<256>(a, Np, n_q_tiles, s, true); break;
  }
  if (e != cudaSuccess) return e;
  if (main_events != nullptr && (e = cudaEventRecord(main_events[0], s)) != cudaSuccess) return e;
  switch (a.d) {
    case 64:
      e = causal ? launch_main<64, 3, true>(m, lse2, dmap, dk, dv, a, s, dropout)
                 : launch_main<64, 3, false>(m, lse2, dmap, dk, dv, a, s, dropout);
      break;
    case 128:
      e = causal ? launch_main<128, 2, true>(m, lse2, dmap, dk, dv, a, s, dropout)
                 : launch_main<128, 2, false>(m, lse2, dmap, dk, dv, a, s, dropout);
      break;
    default:
      e = launch_bwd_main_d256(m.q64, m.k, m.v, m.dout64, m.lse2_64, m.dvec_64, dk, dv, a, causal, s, dropout);
      break;
  }
  if (e != cudaSuccess) return e;
  if (main_events != nullptr && (e = cudaEventRecord(main_events[1], s)) != cudaSuccess) return e;
  switch (a.d) {
    case 64: return launch_prep_and_convert<64>(a, Np, n_q_tiles, s, false);
    case 128: return launch_prep_and_convert<128>(a, Np, n_q_tiles, s, false);
    default: return launch_prep_and_convert<256>(a, Np, n_q_tiles, s, false);
  }
}

}  // namespace fa
