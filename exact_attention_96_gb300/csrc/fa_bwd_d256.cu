// fa_bwd_d256.cu -- backward main kernel for head dimension 256.
//
// Same mathematics as fa_bwd_main_kernel ("FlashAttention 与显存" §09: S and P recomputed
// block by block; gradients from calculus), re-tiled because at d = 256 the dK and dV
// accumulators of a 128-key tile would fill all 512 TMEM columns on their own:
//   - a CTA owns 128 keys of one (batch, head) and one 128-wide slice z of the head
//     dimension for its dK, dV accumulators (grid.z = 2 slices); it recomputes S^T and dP^T
//     over the full d from query tiles of 64 rows;
//   - dQ is produced transposed, dQ^T_z = K_z^T dS^T (M = the 128 d-lanes of the slice,
//     N = 64 queries), and added into a row-major fp32 accumulator [B*H][rows][256], where
//     the 32 lanes of a warp add 32 consecutive floats of one query row.
// TMEM columns: S^T [0,64) (P^T packed inside), dP^T [64,128), dQ^T [128,192), dV [192,320),
// dK [320,448).  Shared memory: K, V [128 x 256] (64 KB each), Q, dO [64 x 256] (32 KB
// each, one stage with separate full/empty barriers so dO_{i+1} can land while dK_i runs),
// dS^T [128 x 64] (16 KB), LSE*log2e and D tiles.
// Roles: warps 0-7 key rows (two warpgroups split the 64 query columns), warps 8-11 dQ
// drain, warp 12 TMA producer, warp 13 TMEM + MMA issuer.
// Dropout (template flag): as in the d <= 128 kernel, with Z = keep * scale_keep,
// dV = (P * Z)^T dO and dS = P * (dP * Z - D); a key row draws the keep bits of its key for
// its 32 queries by the shared octet scheme, writes P^T * keep for the dV product where the
// plain kernel writes P^T, and the unmasked P^T in the next 16 columns of its S^T range (read
// back for dS).

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kKeys = 128;   // keys per CTA
constexpr int kQ = 64;       // queries per inner step
constexpr int kDH = 128;     // width of the dK / dV slice
constexpr int kThreads = 448;
constexpr int kRowThreads = 256;
constexpr int kDrainWarp0 = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;

struct L256 {
  static constexpr int kKVBytes = kKeys * 256 * 2;   // 64 KB, 4 slabs of [128 x 128 B]
  static constexpr int kQBytes = kQ * 256 * 2;        // 32 KB, 4 slabs of [64 x 128 B]
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKVBytes;
  static constexpr int kQOff = kVOff + kKVBytes;
  static constexpr int kdOOff = kQOff + kQBytes;
  static constexpr int kdSOff = kdOOff + kQBytes;     // [128 keys x 64 queries] bf16, one slab
  static constexpr int kLseOff = kdSOff + kKeys * kQ * 2;
  static constexpr int kDOff = kLseOff + kQ * 4;
  static constexpr int kBarOff = kDOff + kQ * 4;
  enum {
    kBarKV, kBarQFull, kBarQEmpty, kBarOFull, kBarOEmpty, kBarSFull, kBarDPFull, kBarPReady,
    kBarDSReady, kBarDQFull, kBarDQDrained, kBarAccDone, kBarEpi0,
    kBarEpi1, kBarDrain, kNumBars
  };
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kColS = 0, kColDP = 64, kColDQ = 128, kColDV = 192, kColDK = 320;
  static constexpr int kTmemCols = 512;
  static_assert(kBytes <= 232448, "shared memory budget");
};

template <bool CAUSAL, bool DROPOUT>
__global__ void __launch_bounds__(kThreads, 1)
fa_bwd_d256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const __grid_constant__ CUtensorMap tmLse2, const __grid_constant__ CUtensorMap tmD,
                   const __grid_constant__ CUtensorMap tmdK, const __grid_constant__ CUtensorMap tmdV,
                   const BwdArgs args) {
  using L = L256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_addr(smem_raw);
  if (base & 1023u) {
    if (threadIdx.x == 0) atomicOr(args.err_word, 2);
    return;
  }
  uint8_t* smem = smem_raw;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The two head-dimension slices of a key tile are dispatched next to each other, so that
  // they stream the same Q and dO tiles at about the same time and share them in L2.
  const int tiles = int(gridDim.x), heads = int(gridDim.y);
  const int lin = int(blockIdx.x) + tiles * (int(blockIdx.y) + heads * int(blockIdx.z));
  const int z = lin & 1;                  // d slice [128z, 128z + 128)
  const int pair = lin >> 1;              // (key tile, head) pair
  const RankHead rh = CAUSAL ? causal_order_of(pair, tiles, heads, args.causal_group) : RankHead{pair % tiles, pair / tiles};
  const int bh = rh.bh;
  const int k0 = rh.rank * kKeys;         // causal: key tile 0 is the heaviest
  const int N = args.N;
  const int n_qt = (N + kQ - 1) / kQ;     // 64-row query tiles
  const int it_first = CAUSAL ? (k0 / kQ) : 0;
  const int n_it = n_qt - it_first;
  const int rows_padded = ((N + 127) / 128) * 128;  // accumulator rows per head

  auto bar = [&](int i) -> uint32_t { return base + L::kBarOff + 8u * uint32_t(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const WaitCtl wc{abort_flag, args.err_word, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kBarKV), 1);
    mbar_init(bar(L::kBarQFull), 1);
    mbar_init(bar(L::kBarQEmpty), kRowThreads + 1);   // key rows done with LSE + MMA dK done
    mbar_init(bar(L::kBarOFull), 1);
    mbar_init(bar(L::kBarOEmpty), kRowThreads + 1);   // key rows done with D + MMA dV done
    mbar_init(bar(L::kBarSFull), 1);
    mbar_init(bar(L::kBarDPFull), 1);
    mbar_init(bar(L::kBarPReady), kRowThreads);
    mbar_init(bar(L::kBarDSReady), kRowThreads);
    mbar_init(bar(L::kBarDQFull), 1);
    mbar_init(bar(L::kBarDQDrained), 128);
    mbar_init(bar(L::kBarAccDone), 1);
    mbar_init(bar(L::kBarEpi0), 128);
    mbar_init(bar(L::kBarEpi1), 128);
    mbar_init(bar(L::kBarDrain), 1);
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
  const uint32_t sK = base + L::kKOff, sV = base + L::kVOff, sQ = base + L::kQOff,
                 sdO = base + L::kdOOff, sdS = base + L::kdSOff;

  if (warp == kProducerWarp) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(L::kBarKV), 2 * L::kKVBytes);
      for (int s = 0; s < 4; ++s) {
        tma_load_3d(sK + s * (kKeys * 128), &tmK, bar(L::kBarKV), s * 64, k0, bh);
        tma_load_3d(sV + s * (kKeys * 128), &tmV, bar(L::kBarKV), s * 64, k0, bh);
      }
      int q_arms = 0, o_arms = 0;
      bool ok = true;
      for (int it = 0; it < n_it; ++it) {
        const int q0 = (it_first + it) * kQ;
        if (it > 0 && !mbar_wait(bar(L::kBarQEmpty), (it - 1) & 1, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(L::kBarQFull), L::kQBytes + kQ * 4);
        for (int s = 0; s < 4; ++s) tma_load_3d(sQ + s * (kQ * 128), &tmQ, bar(L::kBarQFull), s * 64, q0, bh);
        tma_load_3d(base + L::kLseOff, &tmLse2, bar(L::kBarQFull), q0, bh, 0);
        ++q_arms;
        if (it > 0 && !mbar_wait(bar(L::kBarOEmpty), (it - 1) & 1, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(L::kBarOFull), L::kQBytes + kQ * 4);
        for (int s = 0; s < 4; ++s) tma_load_3d(sdO + s * (kQ * 128), &tmdO, bar(L::kBarOFull), s * 64, q0, bh);
        tma_load_3d(base + L::kDOff, &tmD, bar(L::kBarOFull), q0, bh, 0);
        ++o_arms;
      }
      if (!ok) {
        auto drain = [&](uint32_t b, uint32_t parity) {
          for (uint64_t t0 = global_timer_ns();
               !mbar_try_wait(b, parity) && global_timer_ns() - t0 < wc.limit_ns;) {
          }
        };
        drain(bar(L::kBarKV), 0);
        if (q_arms > 0) drain(bar(L::kBarQFull), (q_arms - 1) & 1);
        if (o_arms > 0) drain(bar(L::kBarOFull), (o_arms - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // Order per query tile i: dV_i | dK_i | dQ^T_i | S_{i+1}, dP_{i+1}
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(128, kQ, 0, 0);     // S^T, dP^T
      constexpr uint32_t kIdAcc = idesc_bf16_f32(128, kDH, 0, 1);  // dV, dK (B N-major)
      constexpr uint32_t kIdDQ = idesc_bf16_f32(128, kQ, 1, 1);    // dQ^T: A = K_z^T (M-major), B = dS^T (N-major)
      auto issue_s = [&]() {
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          mma_ss(tmem + L::kColS, sdesc_sw128(sK + (kk >> 2) * (kKeys * 128) + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(sQ + (kk >> 2) * (kQ * 128) + (kk & 3) * 32, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kBarSFull));
      };
      auto issue_dp = [&]() {
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          mma_ss(tmem + L::kColDP, sdesc_sw128(sV + (kk >> 2) * (kKeys * 128) + (kk & 3) * 32, 16, 1024),
                 sdesc_sw128(sdO + (kk >> 2) * (kQ * 128) + (kk & 3) * 32, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kBarDPFull));
      };
      bool ok = mbar_wait(bar(L::kBarKV), 0, wc) && mbar_wait(bar(L::kBarQFull), 0, wc);
      if (ok) issue_s();
      ok = ok && mbar_wait(bar(L::kBarOFull), 0, wc);
      if (ok) issue_dp();
      for (int it = 0; ok && it < n_it; ++it) {
        const uint32_t ph = it & 1;
        if (!mbar_wait(bar(L::kBarPReady), ph, wc)) { ok = false; break; }
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk) {
          mma_ts(tmem + L::kColDV, tmem + L::kColS + 32 * (kk >> 1) + 8 * (kk & 1),
                 sdesc_sw128(sdO + (2 * z) * (kQ * 128) + kk * (16 * 128), kQ * 128, 1024), kIdAcc,
                 (it > 0 || kk > 0) ? 1u : 0u);
        }
        // one commit serves both: dO_i's stage (with the key rows' arrivals) and, for the
        // S_{i+1} issue below, the end of dV_i (see there)
        mma_commit(bar(L::kBarOEmpty));
        if (!mbar_wait(bar(L::kBarDSReady), ph, wc)) { ok = false; break; }
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kQ / 16; ++kk) {
          mma_ss(tmem + L::kColDK, sdesc_sw128(sdS + kk * 32, 16, 1024),
                 sdesc_sw128(sQ + (2 * z) * (kQ * 128) + kk * (16 * 128), kQ * 128, 1024), kIdAcc,
                 (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(L::kBarQEmpty));
        // dQ^T_i overwrites dQ^T_{i-1}: the drain warps must have read it
        if (it > 0 && !mbar_wait(bar(L::kBarDQDrained), ph ^ 1, wc)) { ok = false; break; }
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          mma_ss(tmem + L::kColDQ,
                 sdesc_sw128(sK + (2 * z) * (kKeys * 128) + kk * (16 * 128), kKeys * 128, 1024),
                 sdesc_sw128(sdS + kk * (16 * 128), kQ * 128, 1024), kIdDQ, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kBarDQFull));  // also frees dS^T_i (dQ^T_i is its last reader)
        if (it + 1 < n_it) {
          // S_{i+1} overwrites P^T_i (read by dV_i and by the key rows before dS_i was published).
          // dV_i has completed once the dO stage's empty barrier has: the key rows arrived on it
          // after publishing dS_i, which dQ^T_i above already waited for, so this wait is on
          // dV_i alone; the barrier cannot run a phase ahead (its next completion needs the key
          // rows' arrival for tile i+1, after dP_{i+1} is issued below).
          if (!mbar_wait(bar(L::kBarOEmpty), ph, wc) || !mbar_wait(bar(L::kBarQFull), (it + 1) & 1, wc)) {
            ok = false;
            break;
          }
          issue_s();
          if (!mbar_wait(bar(L::kBarOFull), (it + 1) & 1, wc)) { ok = false; break; }
          issue_dp();
        }
      }
      if (ok) mma_commit(bar(L::kBarAccDone));
      mma_commit(bar(L::kBarDrain));
      for (uint64_t t0 = global_timer_ns();
           !mbar_try_wait(bar(L::kBarDrain), 0) && global_timer_ns() - t0 < wc.limit_ns;) {
      }
    }
    __syncwarp();
  } else if (warp < 8) {
    // key rows; half h owns queries [32h, 32h + 32) of each 64-query tile and packs their P^T
    // into TMEM columns [32h, 32h + 16), inside the S^T columns it has already read
    const int t = threadIdx.x & 127;
    const int half = threadIdx.x >> 7;
    const int c0 = half * 32;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const int key = k0 + t;
    const float sl2 = args.scale_log2;
    const float* lse2 = reinterpret_cast<const float*>(smem + L::kLseOff) + c0;
    const float* dvv = reinterpret_cast<const float*>(smem + L::kDOff) + c0;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const uint32_t ph = it & 1;
      const int q0 = (it_first + it) * kQ;
      const bool edge = (CAUSAL && q0 < k0 + kKeys) || (q0 + kQ > N);
      uint32_t km = 0u;  // dropout keep bits: bit c = query q0 + c0 + c
      if constexpr (DROPOUT) {
        km = uint32_t(dropout_key_bits<4>(args.dropout, key, q0 + c0, bh, lane));
        asm volatile("" : "+r"(km));  // generator work ahead of the S^T wait
      }
      if (!__all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull), ph, wc))) { ok = false; break; }
      tc_fence_after_sync();
      {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + L::kColS + c0, r);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          // lse2 holds -LSE * log2(e) (stored negated by the prep kernel): two keys per instruction
          const float2 x = ffma2(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                 make_float2(sl2, sl2), make_float2(lse2[e], lse2[e + 1]));
          w[e / 2] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
        }
        if (edge) apply_keep_mask(w, visible_bits(q0 + c0, CAUSAL ? key : 0, N));
        if constexpr (DROPOUT) {
          // unmasked P^T for dS in the second 16 columns; P^T * keep for the dV product
          tmem_st16(tmem + lane_off + L::kColS + c0 + 16, w);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint32_t kb = km >> (2 * e);
            w[e] &= ((kb & 1u) ? 0x0000FFFFu : 0u) | ((kb & 2u) ? 0xFFFF0000u : 0u);
          }
        }
        tmem_st16(tmem + lane_off + L::kColS + c0, w);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kBarPReady));
      mbar_arrive(bar(L::kBarQEmpty));   // done with this tile's LSE
      bool got = mbar_wait(bar(L::kBarDPFull), ph, wc);
      // dS^T_{i-1} is free once dQ^T_{i-1} (its last reader) has completed; that barrier's
      // next completion needs this tile's dS, so it cannot run a phase ahead
      if (it > 0) got = got && mbar_wait(bar(L::kBarDQFull), ph ^ 1, wc);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after_sync();
      {
        uint32_t r[32];
        uint32_t pr[16];
        tmem_ld32(tmem + lane_off + L::kColDP + c0, r);
        tmem_ld16(tmem + lane_off + L::kColS + c0 + (DROPOUT ? 16 : 0), pr);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = __uint_as_float(pr[e / 2] << 16);
          const float p1 = __uint_as_float(pr[e / 2] & 0xFFFF0000u);
          float dp0 = __uint_as_float(r[e]), dp1 = __uint_as_float(r[e + 1]);
          if constexpr (DROPOUT) {
            const uint32_t kb = km >> e;
            dp0 = (kb & 1u) ? dp0 * args.dropout.scale : 0.f;
            dp1 = (kb & 2u) ? dp1 * args.dropout.scale : 0.f;
          }
          // dvv holds -D: dS = P (dP - D) two at a time
          const float2 ds = fmul2(make_float2(p0, p1), fadd2(make_float2(dp0, dp1), make_float2(dvv[e], dvv[e + 1])));
          w[e / 2] = pack_bf16x2(ds.x, ds.y);
        }
        if (q0 + kQ > N) apply_keep_mask(w, visible_bits(q0 + c0, 0, N));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int phys = ((c0 >> 3) + i) ^ (t & 7);
          *reinterpret_cast<uint4*>(smem + L::kdSOff + t * 128 + phys * 16) =
              make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kBarDSReady));
      mbar_arrive(bar(L::kBarOEmpty));   // done with this tile's D
    }
    // epilogue: half 0 stores the dV slice, half 1 the dK slice (scaled)
    const bool fin = ok && __all_sync(0xffffffffu, mbar_wait(bar(L::kBarAccDone), 0, wc));
    const uint32_t col = half == 0 ? L::kColDV : L::kColDK;
    const float mul = half == 0 ? (DROPOUT ? args.dropout.scale : 1.f) : args.scale;
    uint8_t* stage = smem + (half == 0 ? L::kQOff : L::kdOOff);   // 2 slabs of [128 x 128 B]
    const bool accum = args.dk_accum != nullptr;
    if (fin && accum) {
      // accumulate mode: add the fp32 slice rows into the caller's buffers (vector atomics)
      tc_fence_after_sync();
      float4* dst = reinterpret_cast<float4*>((half == 0 ? args.dv_accum : args.dk_accum) +
                                              ((size_t)bh * N + key) * 256 + kDH * z);
#pragma unroll 1
      for (int c = 0; c < kDH; c += 32) {
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
      for (int c = 0; c < kDH; c += 32) {
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
          *reinterpret_cast<uint4*>(stage + slab * (kKeys * 128) + t * 128 + phys * 16) =
              make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
      fence_proxy_async_smem();
    }
    const uint32_t epi = bar(half == 0 ? L::kBarEpi0 : L::kBarEpi1);
    mbar_arrive(epi);
    if (t == 0 && fin && !accum && mbar_wait(epi, 0, wc) && *abort_flag == 0) {
      const CUtensorMap* map = half == 0 ? &tmdV : &tmdK;
      const uint32_t src = half == 0 ? sQ : sdO;
      for (int s = 0; s < 2; ++s) tma_store_3d(map, src + s * (kKeys * 128), kDH * z + 64 * s, k0, bh);
      bulk_commit_group();
      bulk_wait_group_read_all();  // source read: the CTA may exit
    }
  } else if (warp < kProducerWarp) {
    // dQ drain: thread t owns column 128z + t of the head dimension (TMEM lane t of dQ^T)
    const int t = threadIdx.x - kDrainWarp0 * 32;
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    float* acc = args.dq_acc + (size_t)bh * rows_padded * 256 + kDH * z + t;
    for (int it = 0; it < n_it; ++it) {
      const int q0 = (it_first + it) * kQ;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(L::kBarDQFull), it & 1, wc))) break;
      tc_fence_after_sync();
      uint32_t a[32], b[32];
      tmem_ld32(tmem + lane_off + L::kColDQ, a);
      tmem_ld32(tmem + lane_off + L::kColDQ + 32, b);
      tc_fence_before_sync();
      mbar_arrive(bar(L::kBarDQDrained));
      const int nq = min(kQ, N - q0);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        if (c < nq) atomicAdd(acc + (size_t)(q0 + c) * 256, __uint_as_float(a[c]));
        if (c + 32 < nq) atomicAdd(acc + (size_t)(q0 + c + 32) * 256, __uint_as_float(b[c]));
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

}  // namespace

cudaError_t launch_bwd_main_d256(const CUtensorMap& q64, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& dout64, const CUtensorMap& lse2_64,
                                 const CUtensorMap& d64, const CUtensorMap& dk, const CUtensorMap& dv,
                                 const BwdArgs& a, bool causal, cudaStream_t s, bool dropout) {
  auto kern = dropout ? (causal ? fa_bwd_d256_kernel<true, true> : fa_bwd_d256_kernel<false, true>)
                      : (causal ? fa_bwd_d256_kernel<true, false> : fa_bwd_d256_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L256::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((a.N + kKeys - 1) / kKeys, a.BH, 2);
  // Causal heads are dispatched in groups whose streamed tensors (Q, K, V, dO and the fp32 dQ
  // accumulator) fit about 128 MB of L2 together, at most kCausalGroup heads.  At
  // 2x8x16384x256 (50 MB per head: groups of 2) this took the backward from 577 to 597
  // TFLOP/s.  DRAM traffic with groups of 8 was 4.3x the algorithmic bytes.  The d <= 128
  // kernels and the forward measured best with 8 at every size.
  BwdArgs a2 = a;
  const double head_bytes = double(a.N) * 256 * 2 * 4 + double((a.N + 127) / 128 * 128) * 256 * 4;
  a2.causal_group = int(std::min<double>(kCausalGroup, std::max(1.0, std::floor(128e6 / head_bytes))));
  kern<<<grid, kThreads, L256::kBytes, s>>>(q64, k, v, dout64, lse2_64, d64, dk, dv, a2);
  return cudaGetLastError();
}

}  // namespace fa
