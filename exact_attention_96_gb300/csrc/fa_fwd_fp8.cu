// fa_fwd_fp8.cu -- FP8 forward pass for head dim 128: E4M3 Q, K, V, bf16 O, fp32 LSE
// ("Flash Attention 原理与实践" §3.2: the third version's FP8 mode).
//
// Same computation as fa_fwd.cu (streaming softmax over key tiles, "FlashAttention 与显存"
// §07/§08) with both products on 8-bit operands (tcgen05.mma kind::f8f6f4, 32 elements of K
// per instruction).  Q and K are E4M3 [B*H, N, 128]; V is given transposed, E4M3
// [B*H, 128, ldv] (keys innermost), so that P V also reads a K-major operand.  The descale
// factors of Q and K are folded into the softmax scale, V's into the final normalisation.
// P is rounded to E4M3 after scaling by 2^8 (exact: a power of two), which keeps
// probabilities down to 2^-14 as normal numbers; the running sum l carries the same
// factor, so O = acc / l needs no correction and LSE subtracts 8 in base 2.
//
// A CTA owns 256 query rows of one head as two 128-row tiles that share every K/V tile it
// loads; each tile has its own softmax warpgroup and its own MMA-issuing thread, and the two
// softmax warpgroups take turns (the third version's ping-pong of softmax and products
// between warpgroups, "FlashAttention 与显存" §11, re-derived for tcgen05 + TMEM): while one
// converts S to P, the tensor core runs the other tile's P V and next Q K^T.
//
// Roles (352 threads):
//   warps 0-3 / 4-7  softmax of tile 0 / tile 1: thread = query row = TMEM lane.  Reads S,
//                    masks, updates (m, l), writes P back into the first 32 columns of its S
//                    (S is fully in registers by then), rescales O when the maximum grew,
//                    finally normalises O, stores it with TMA and writes LSE.
//   warp 8           TMA producer: both query tiles once, then K_j and V^T_j through a ring.
//   warps 9 / 10     MMA issuers of tile 0 / tile 1 (warp 9 also allocates TMEM).  Each tile
//                    alternates S_j = Q K_j^T -> (softmax) -> O += P_j V_j -> S_{j+1};
//                    S_{j+1} overwrites P_j, so it is issued once P_j V_j has completed.
//                    Issuing a group of tcgen05.mma holds the issuing thread until the tensor
//                    core has nearly finished it, hence one issuer per tile.
//
// TMEM (512 columns): tile t owns [256t, 256t + 256): S in the first 128 columns (P packed
// four E4M3 values per column into the first 32), O in the last 128.
//
// Every wait is bounded (WaitCtl); on timeout the roles unwind as in fa_fwd.cu.

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kD = 128;          // head dim
constexpr int kBM = 128;         // rows per query tile
constexpr int kBC = 128;         // keys per key tile
constexpr int kThreadsP = 352;   // two softmax warpgroups + producer warp + two MMA warps
constexpr int kProducerWarpP = 8;
constexpr int kMmaWarpP = 9;     // issuer of tile 0 (and TMEM allocator); warp 10 issues tile 1
constexpr float kLn2 = 0.69314718055994531f;

struct Fp8Layout {
  static constexpr int kNS = 3;                     // K/V ring stages
  static constexpr int kQBytes = kBM * kD;          // one query tile: 128 rows x 128 bytes
  static constexpr int kKBytes = kBC * kD;          // one K tile
  static constexpr int kVBytes = kD * kBC;          // one V^T tile: 128 rows x 128 keys
  static constexpr int kOBytes = kBM * kD * 2;      // bf16 output tile (two 64-column slabs)
  static constexpr int kQOff = 0;                   // two query tiles
  static constexpr int kKOff = kQOff + 2 * kQBytes;
  static constexpr int kVOff = kKOff + kNS * kKBytes;
  static constexpr int kStageOff = kVOff + kNS * kVBytes;  // two output staging tiles
  static constexpr int kBarOff = kStageOff + 2 * kOBytes;
  static constexpr int kBarQFull = 0;               // 2: one per tile
  static constexpr int kBarKFull = 2;
  static constexpr int kBarKEmpty = kBarKFull + kNS;
  static constexpr int kBarVFull = kBarKEmpty + kNS;
  static constexpr int kBarVEmpty = kBarVFull + kNS;
  static constexpr int kBarSFull = kBarVEmpty + kNS;  // 2
  static constexpr int kBarPFull = kBarSFull + 2;     // 2
  static constexpr int kBarODone = kBarPFull + 2;     // 2
  static constexpr int kBarOFinal = kBarODone + 2;    // 2, single use: every product of the tile landed
  static constexpr int kBarEpi = kBarOFinal + 2;      // 2
  static constexpr int kBarDrain = kBarEpi + 2;       // 2: one per issuer
  static constexpr int kBarTurn = kBarDrain + 2;      // 2: softmax turn of tile 0 / tile 1
  static constexpr int kNumBars = kBarTurn + 2;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem slot, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kSmemAlloc = kBytes + 1024;  // slack for the 1024-byte alignment
  static constexpr int kTileCols = 256;             // TMEM columns per query tile
  static constexpr int kColO = 128;                 // O within a tile's columns
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

template <bool CAUSAL>
__global__ void __launch_bounds__(kThreadsP, 1)
fa_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const FwdArgs args) {
  using L = Fp8Layout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const RankHead rh = CAUSAL ? causal_dispatch_order() : RankHead{int(blockIdx.x), int(blockIdx.y)};
  const int bh = rh.bh;
  const int n_pairs = (args.n_q_tiles + 1) / 2;
  const int pair = CAUSAL ? (n_pairs - 1 - rh.rank) : rh.rank;  // heavy pairs first
  const int q0 = pair * 2 * kBM;  // first row of tile 0; tile 1 starts at q0 + kBM
  const int N = args.N;
  const int n_kv_all = (N + kBC - 1) / kBC;
  const bool has1 = q0 + kBM < N;
  // key tiles each query tile sees (causal: up to its diagonal tile)
  const int ntile0 = CAUSAL ? min(n_kv_all, (q0 + kBM + kBC - 1) / kBC) : n_kv_all;
  const int ntile1 = !has1 ? 0 : (CAUSAL ? min(n_kv_all, (q0 + 2 * kBM + kBC - 1) / kBC) : n_kv_all);
  const int nkv = max(ntile0, ntile1);

  auto bar = [&](int i) -> uint32_t { return base + L::kBarOff + 8u * uint32_t(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const WaitCtl wc{abort_flag, args.err_word, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kBarQFull + t), 1);
      mbar_init(bar(L::kBarSFull + t), 1);
      mbar_init(bar(L::kBarPFull + t), 128);
      mbar_init(bar(L::kBarODone + t), 1);
      mbar_init(bar(L::kBarOFinal + t), 1);
      mbar_init(bar(L::kBarEpi + t), 128);
    }
    // a K/V stage is free once every tile that reads it has committed its product (the only
    // tile read by one query tile alone is the causal last one, whose stage is never reused)
    for (int s = 0; s < L::kNS; ++s) {
      mbar_init(bar(L::kBarKFull + s), 1);
      mbar_init(bar(L::kBarKEmpty + s), has1 ? 2 : 1);
      mbar_init(bar(L::kBarVFull + s), 1);
      mbar_init(bar(L::kBarVEmpty + s), has1 ? 2 : 1);
    }
    mbar_init(bar(L::kBarDrain), 1);
    mbar_init(bar(L::kBarDrain + 1), 1);
    mbar_init(bar(L::kBarTurn), 128);
    mbar_init(bar(L::kBarTurn + 1), 128);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarpP) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  auto sQ = [&](int t) -> uint32_t { return base + L::kQOff + uint32_t(t) * L::kQBytes; };
  auto sK = [&](int s) -> uint32_t { return base + L::kKOff + uint32_t(s) * L::kKBytes; };
  auto sV = [&](int s) -> uint32_t { return base + L::kVOff + uint32_t(s) * L::kVBytes; };

  if (warp == kProducerWarpP) {
    // ------------------------------------------------------------ producer ----
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
      for (int t = 0; t < (has1 ? 2 : 1); ++t) {
        mbar_arrive_expect_tx(bar(L::kBarQFull + t), L::kQBytes);
        tma_load_3d(sQ(t), &tmQ, bar(L::kBarQFull + t), 0, q0 + t * kBM, bh);
      }
      int k_arms[L::kNS], v_arms[L::kNS];
#pragma unroll
      for (int s = 0; s < L::kNS; ++s) k_arms[s] = v_arms[s] = 0;
      bool ok = true;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % L::kNS;
        const uint32_t ph = (j / L::kNS) & 1;
        if (j >= L::kNS && !mbar_wait(bar(L::kBarKEmpty + st), ph ^ 1, wc)) { ok = false; break; }
        if (j != args.withhold_k_tile) {  // the test hook leaves this tile's barrier unarmed
          mbar_arrive_expect_tx(bar(L::kBarKFull + st), L::kKBytes);
          tma_load_3d(sK(st), &tmK, bar(L::kBarKFull + st), 0, j * kBC, bh);
          ++k_arms[st];
        }
        if (j >= L::kNS && !mbar_wait(bar(L::kBarVEmpty + st), ph ^ 1, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(L::kBarVFull + st), L::kVBytes);
        // V^T tile: 128 keys (x) by the 128 rows of the head dim (y)
        tma_load_3d(sV(st), &tmV, bar(L::kBarVFull + st), j * kBC, 0, bh);
        ++v_arms[st];
      }
      if (!ok) {
        // let every copy this thread started land before shared memory is released
        auto drain = [&](uint32_t b, uint32_t parity) {
          for (uint64_t t0 = global_timer_ns();
               !mbar_try_wait(b, parity) && global_timer_ns() - t0 < wc.limit_ns;) {
          }
        };
        drain(bar(L::kBarQFull), 0);
        if (has1) drain(bar(L::kBarQFull + 1), 0);
        for (int s = 0; s < L::kNS; ++s) {
          if (k_arms[s] > 0) drain(bar(L::kBarKFull + s), (k_arms[s] - 1) & 1);
          if (v_arms[s] > 0) drain(bar(L::kBarVFull + s), (v_arms[s] - 1) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarpP || warp == kMmaWarpP + 1) {
    // ------------------------------------------------------- MMA issuers ----
    // One issuing thread per query tile (a single issuer would serialise the two tiles'
    // chains); tcgen05.commit covers only the committing thread's operations, and the tiles'
    // TMEM columns are disjoint.
    const int t = warp - kMmaWarpP;
    const int ntile_t = t == 0 ? ntile0 : ntile1;
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_e4m3_f32(kBM, kBC);  // Q K^T: both K-major
      constexpr uint32_t kIdO = idesc_e4m3_f32(kBM, kD);   // P V: P from TMEM, V^T K-major
      const uint32_t s_tmem = tmem + uint32_t(t) * L::kTileCols;  // S, and P inside it
      const uint32_t o_tmem = s_tmem + L::kColO;
      bool ok = ntile_t > 0 && mbar_wait(bar(L::kBarQFull + t), 0, wc);
      for (int j = 0; ok && j < ntile_t; ++j) {
        const int st = j % L::kNS;
        const uint32_t ph = (j / L::kNS) & 1;
        // S_j = Q K_j^T, once K_j is in and P_{j-1} V_{j-1} (which reads P inside S) is done
        if (!mbar_wait(bar(L::kBarKFull + st), ph, wc) ||
            (j > 0 && !mbar_wait(bar(L::kBarODone + t), (j - 1) & 1, wc))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kD / 32; ++kk) {  // 32 bytes of each 128-byte row per step
          const uint64_t a = sdesc_sw128(sQ(t) + kk * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sK(st) + kk * 32, 16, 1024);
          mma_ss_f8(s_tmem, a, b, kIdS, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(L::kBarSFull + t));
        mma_commit(bar(L::kBarKEmpty + st));
        // O += P_j V_j, once the softmax has written P_j and V_j is in
        if (!mbar_wait(bar(L::kBarPFull + t), j & 1, wc) || !mbar_wait(bar(L::kBarVFull + st), ph, wc)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < kBC / 32; ++kk) {  // 32 keys per step: 8 TMEM columns of P
          const uint64_t b = sdesc_sw128(sV(st) + kk * 32, 16, 1024);
          mma_ts_f8(o_tmem, s_tmem + kk * 8, b, kIdO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(L::kBarODone + t));
        mma_commit(bar(L::kBarVEmpty + st));
      }
      if (ok && ntile_t > 0) mma_commit(bar(L::kBarOFinal + t));
      // Every MMA this thread issued must be finished before TMEM is released.
      mma_commit(bar(L::kBarDrain + t));
      for (uint64_t t0 = global_timer_ns();
           !mbar_try_wait(bar(L::kBarDrain + t), 0) && global_timer_ns() - t0 < wc.limit_ns;) {
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax ----
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = threadIdx.x & 127;       // = TMEM lane
    const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tcol = tmem + uint32_t(t) * L::kTileCols + lane_off;
    const int row_g = q0 + t * kBM + row;
    const int ntile_t = t == 0 ? ntile0 : ntile1;
    const float sl2 = args.scale_log2;
    // P is scaled by 2^8 before its 8-bit rounding (and l with it)
    constexpr float kPBias = 8.f;
    float m_run = -INFINITY;  // running max of scale*log2(e)*s
    float l_run = 0.f;        // running sum of 2^(scaled s - m_run [+ 8])
    bool ok = true;
    // The two warpgroups take turns: tile 1 runs softmax j after tile 0 has finished softmax
    // j, tile 0 runs softmax j + 1 after tile 1 has finished softmax j.  Meanwhile the tensor
    // core runs the waiting tile's P V and next Q K^T, so products and softmax overlap instead
    // of both warpgroups converting at once and then both waiting for the tensor core.  Tile
    // 1's extra causal tile (j = ntile0) has no turn to wait for.
    for (int j = 0; j < ntile_t; ++j) {
      const bool my_turn = t == 0 ? (j == 0 || j - 1 >= ntile1 || mbar_wait(bar(L::kBarTurn), (j - 1) & 1, wc))
                                  : (j >= ntile0 || mbar_wait(bar(L::kBarTurn + 1), j & 1, wc));
      // tcgen05.ld is warp-collective: every wait outcome is made warp-uniform
      if (!__all_sync(0xffffffffu, my_turn && mbar_wait(bar(L::kBarSFull + t), j & 1, wc))) { ok = false; break; }
      tc_fence_after_sync();
      float s[kBC];
      {
        uint32_t r[kBC];
        tmem_ld128(tcol, r);
#pragma unroll
        for (int i = 0; i < kBC; ++i) s[i] = __uint_as_float(r[i]);
      }
      // keys kv0 + c are visible for c < lim (sequence tail; causal: key <= query)
      const int kv0 = j * kBC;
      int lim = N - kv0;
      if (CAUSAL) lim = min(lim, row_g - kv0 + 1);
      if (lim < kBC) {
#pragma unroll
        for (int c = 0; c < kBC; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      // four independent chains for the maximum and two for the sum: shorter dependency
      // chains (4x16x8192x128 causal 1341 -> 1351 TFLOP/s; the bf16 forward measured within
      // +-0.8 % either way and keeps two)
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]), mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
      for (int c = 8; c < kBC; c += 8) {
        mx0 = fmax3(mx0, s[c], s[c + 1]);
        mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
        mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
        mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
      }
      const float m_new = fmaxf(m_run, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2);
      const float alpha = ex2_approx(m_run - m_new);  // 0 on the first tile
      const bool grew = (j > 0) && (m_new > m_run);
      m_run = m_new;
      const float neg_m = kPBias - m_new;
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      // P_j into the first columns of S_j (all of S_j is in registers; the tensor core
      // touches this tile's S again only after P_j V_j)
      uint32_t pk[kBC / 4];
#pragma unroll
      for (int c = 0; c < kBC; c += 4) {
        // two keys per instruction for the scaling and the sums
        const float2 x01 = ffma2(make_float2(s[c], s[c + 1]), make_float2(sl2, sl2), make_float2(neg_m, neg_m));
        const float2 x23 = ffma2(make_float2(s[c + 2], s[c + 3]), make_float2(sl2, sl2), make_float2(neg_m, neg_m));
        const float p0 = ex2_approx(x01.x), p1 = ex2_approx(x01.y);
        const float p2 = ex2_approx(x23.x), p3 = ex2_approx(x23.y);
        sum2[(c >> 2) & 1] = fadd2(sum2[(c >> 2) & 1], fadd2(make_float2(p0, p1), make_float2(p2, p3)));
        pk[c / 4] = pack_e4m3x4(p0, p1, p2, p3);
      }
      tmem_st32(tcol, pk);
      const float2 sa = fadd2(sum2[0], sum2[1]);
      l_run = l_run * alpha + (sa.x + sa.y);
      // Rescale the accumulator when this warp's rows saw a larger maximum.  O holds
      // P_0 V_0 .. P_{j-1} V_{j-1}, all complete: S_j was issued after the last of them had
      // landed, and its commit covers them.
      if (__any_sync(0xffffffffu, grew)) {
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          uint32_t r[32];
          tmem_ld32(tcol + L::kColO + c, r);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 y = fmul2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                   make_float2(alpha, alpha));
            r[i] = __float_as_uint(y.x);
            r[i + 1] = __float_as_uint(y.y);
          }
          tmem_st32(tcol + L::kColO + c, r);
        }
      }
      tmem_wait_st();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kBarPFull + t));
      mbar_arrive(bar(L::kBarTurn + (1 - t)));  // the other tile's turn
    }

    // ------------------------------------------------------------ epilogue ----
    if (ntile_t > 0) {
      const bool fin = ok && __all_sync(0xffffffffu, mbar_wait(bar(L::kBarOFinal + t), 0, wc));
      uint8_t* stage = smem + L::kStageOff + t * L::kOBytes;
      if (fin) {
        tc_fence_after_sync();
        const float inv_l = args.o_scale / l_run;
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          uint32_t r[32];
          tmem_ld32(tcol + L::kColO + c, r);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l, __uint_as_float(r[2 * i + 1]) * inv_l);
          const int slab = c >> 6;
          const int chunk0 = (c & 63) >> 3;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int phys = (chunk0 + i) ^ (row & 7);
            *reinterpret_cast<uint4*>(stage + slab * (kBM * 128) + row * 128 + phys * 16) =
                make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
        fence_proxy_async_smem();
        if (row_g < N) args.lse[size_t(bh) * N + row_g] = (m_run + lg2_approx(l_run) - kPBias) * kLn2;
      }
      // every thread of the warpgroup arrives; one stores the tile when all rows are staged
      mbar_arrive(bar(L::kBarEpi + t));
      if (row == 0 && fin && mbar_wait(bar(L::kBarEpi + t), 0, wc) && *abort_flag == 0) {
        const uint32_t src = smem_addr(stage);
        for (int s = 0; s < 2; ++s) tma_store_3d(&tmO, src + s * (kBM * 128), s * 64, q0 + t * kBM, bh);
        bulk_commit_group();
        bulk_wait_group_read_all();  // source read: the CTA may exit
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarpP) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

template <bool CAUSAL>
cudaError_t launch_fp8_cfg(const Maps& m, const FwdArgs& a, cudaStream_t s) {
  auto kern = fa_fwd_fp8_kernel<CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Fp8Layout::kSmemAlloc);
  if (e != cudaSuccess) return e;
  dim3 grid((a.n_q_tiles + 1) / 2, a.BH);
  kern<<<grid, kThreadsP, Fp8Layout::kSmemAlloc, s>>>(m.q, m.k, m.v, m.o, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp8(const Maps& m, const FwdArgs& a, bool causal, cudaStream_t s) {
  return causal ? launch_fp8_cfg<true>(m, a, s) : launch_fp8_cfg<false>(m, a, s);
}

}  // namespace fa
