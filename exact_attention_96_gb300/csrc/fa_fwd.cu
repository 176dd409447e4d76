// fa_fwd.cu -- forward pass of exact attention on sm_103a.
//
// One CTA owns one tile of 128 query rows of one (batch, head) and streams every key /
// value tile of that head past it ("FlashAttention 与显存" §07: the second-version order,
// one Q block per SM with K and V flying in; "FlashAttention算子优化" §2), keeping the
// running maximum m and running sum l of each row and rescaling the output accumulator
// when the maximum grows ("FlashAttention 与显存" §08).  S and P never leave the SM.
//
// Roles (warp specialisation, as the third version does with producer / consumer
// warps, "FlashAttention 与显存" §11 -- re-derived here for TMA + tcgen05 + TMEM):
//   warps 0-3  softmax: thread t owns query row t (= TMEM lane t).  Reads S from TMEM,
//              masks, updates (m, l), writes P (bf16) back to TMEM, rescales O in TMEM
//              when its warp's maximum grew, and finally normalises O, stages it in
//              shared memory for a TMA store and writes LSE.  The scaling, sums and
//              rescale run two elements per instruction (fma/add/mul .f32x2) and the row
//              maximum three at a time: this warp's instruction count is on the critical
//              path.
//   warp 4     TMA producer: Q once, then K_j and V_j through an NS-stage ring.
//   warp 5     TMEM allocator and MMA issuer (one thread):
//                S_j = Q K_j^T        (tcgen05.mma, A and B from shared memory)
//                O  += P_j V_j        (tcgen05.mma, A = P from TMEM, B = V from smem)
//              S is double-buffered so S_{j+1} is computed while row softmax of S_j runs.
//
// TMEM columns (fp32 32-bit cells, 128 lanes): S0 [0, BC), S1 [BC, 2BC),
// P0 / P1 bf16 pairs [2BC, 2BC + BC/2) and [2BC + BC/2, 3BC), O [3BC, 3BC + D).
//
// Shared memory, 1024-byte aligned (128-byte swizzle atoms): Q [D/64 slabs x 128 rows x
// 128 B], K ring, V ring (each [D/64 slabs x BC rows x 128 B] per stage), the dropout
// generator words (dropout only), barriers.
// The Q region is reused to stage the bf16 output tile for the TMA store.
//
// Every wait is bounded (see WaitCtl): on timeout the kernel records the error, skips the
// rest of the work, waits for its own copies and MMAs to land and frees TMEM.
//
// Dropout (template flag; "FlashAttention 与显存" §07: applied inside the fused kernel): a
// softmax thread runs the generator for its row over the coming key tile (one call per 8
// keys, philox.cuh) before it waits for S, and stages the words in its own shared-memory
// slots; the softmax reads them back per 8 keys.  P enters the P V product with dropped
// entries zeroed; the running sum l and the LSE are those of the undropped P, and the
// inverse keep probability is folded into the final 1 / l.

#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;            // query rows per CTA (= TMEM lanes)
constexpr int kSoftmaxThreads = 128;
constexpr int kThreads = 192;       // 4 softmax warps + producer warp + MMA warp

template <int D, int BC, int NS, bool DROP = false>
struct FwdLayout {
  static constexpr int kSlabs = D / 64;
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kKVBytes = BC * D * 2;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + NS * kKVBytes;
  // dropout: the generator words of the current key tile, [BC/8 groups][128 rows] x 16 bytes
  static constexpr int kDropOff = kVOff + NS * kKVBytes;
  static constexpr int kDropBytes = DROP ? (BC / 8) * kBM * 16 : 0;
  static constexpr int kBarOff = kDropOff + kDropBytes;
  // barrier slots
  static constexpr int kBarQFull = 0;
  static constexpr int kBarKFull = 1;
  static constexpr int kBarKEmpty = kBarKFull + NS;
  static constexpr int kBarVFull = kBarKEmpty + NS;
  static constexpr int kBarVEmpty = kBarVFull + NS;
  static constexpr int kBarSFull = kBarVEmpty + NS;  // 2
  static constexpr int kBarSFree = kBarSFull + 2;    // 2
  static constexpr int kBarPFull = kBarSFree + 2;    // 2
  // The rescale of O waits for P_{j-1} V_{j-1}: at D = 128 on a barrier of its own, committed
  // after every P V product; otherwise on that product's V-empty barrier, which spares the
  // MMA thread a commit per tile (measured: d = 64 and 256 +2-4 %, d = 128 -0.4 %).
  static constexpr bool kOwnOBar = D == 128;
  static constexpr int kBarODone = kBarPFull + 2;
  static constexpr int kBarDrain = kBarODone + 1;
  static constexpr int kBarEpi = kBarDrain + 1;
  static constexpr int kBarOFinal = kBarEpi + 1;  // single use: every P V product has landed
  static constexpr int kNumBars = kBarOFinal + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem slot, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kSmemAlloc = kBytes + 1024;  // slack for the 1024-byte alignment
  // TMEM columns
  static constexpr int kColS = 0;
  static constexpr int kColP = 2 * BC;
  static constexpr int kColO = 3 * BC;
  static constexpr int kTmemUsed = 3 * BC + D;
  static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
  static_assert(D % 64 == 0 && BC % 32 == 0 && BC <= 256, "tile shape");
};

template <int D, int BC, int NS, bool CAUSAL, bool SPLIT, bool DROPOUT>
__global__ void __launch_bounds__(kThreads, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const FwdArgs args) {
  using L = FwdLayout<D, BC, NS, DROPOUT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // causal: heavy query tiles (late rows see more keys) first, heads in small groups
  const RankHead rh = CAUSAL ? causal_dispatch_order() : RankHead{int(blockIdx.x), int(blockIdx.y)};
  const int bh = rh.bh;
  const int q_tile = CAUSAL ? (args.n_q_tiles - 1 - rh.rank) : rh.rank;
  const int q0 = q_tile * kBM;
  const int N = args.N;    // query rows
  const int Nk = args.Nk;  // keys
  const int n_kv_all = (Nk + BC - 1) / BC;
  // this CTA's key tiles: [t_begin, t_begin + nkv) (split mode: one range per blockIdx.z)
  const int t_begin = SPLIT ? int(blockIdx.z) * args.tiles_per_split : 0;
  const int nkv = CAUSAL ? min(n_kv_all, (q0 + kBM + BC - 1) / BC)
                         : (SPLIT ? min(n_kv_all - t_begin, args.tiles_per_split) : n_kv_all);

  auto bar = [&](int i) -> uint32_t { return base + L::kBarOff + 8u * uint32_t(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const WaitCtl wc{abort_flag, args.err_word, args.wait_limit_ns};

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kBarQFull), 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar(L::kBarKFull + s), 1);
      mbar_init(bar(L::kBarKEmpty + s), 1);
      mbar_init(bar(L::kBarVFull + s), 1);
      mbar_init(bar(L::kBarVEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::kBarSFull + b), 1);
      mbar_init(bar(L::kBarSFree + b), kSoftmaxThreads);
      mbar_init(bar(L::kBarPFull + b), kSoftmaxThreads);
    }
    mbar_init(bar(L::kBarODone), 1);
    mbar_init(bar(L::kBarDrain), 1);
    mbar_init(bar(L::kBarEpi), kSoftmaxThreads);
    mbar_init(bar(L::kBarOFinal), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_addr(tmem_slot), L::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sQ = base + L::kQOff;
  auto sK = [&](int s) -> uint32_t { return base + L::kKOff + uint32_t(s) * L::kKVBytes; };
  auto sV = [&](int s) -> uint32_t { return base + L::kVOff + uint32_t(s) * L::kKVBytes; };

  if (warp == 4) {
    // ------------------------------------------------------------ producer ----
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmO);
      mbar_arrive_expect_tx(bar(L::kBarQFull), L::kQBytes);
      for (int s = 0; s < L::kSlabs; ++s)
        tma_load_3d(sQ + s * (kBM * 128), &tmQ, bar(L::kBarQFull), s * 64, q0, bh);
      int k_arms[NS], v_arms[NS];
#pragma unroll
      for (int s = 0; s < NS; ++s) k_arms[s] = v_arms[s] = 0;
      bool ok = true;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % NS;
        const uint32_t ph = (j / NS) & 1;
        // With two stages the stage and the S buffer of a tile coincide, and S_{j-2} landing
        // means K_{j-2} has been read: wait on the S barrier and spare the MMA thread a commit
        // (the barrier cannot run a phase ahead: S_j needs the K_j loaded below).
        if (j >= NS && !mbar_wait(bar((NS == 2 ? L::kBarSFull : L::kBarKEmpty) + st), ph ^ 1, wc)) {
          ok = false;
          break;
        }
        if (j != args.withhold_k_tile) {  // the test hook leaves this tile's barrier unarmed
          mbar_arrive_expect_tx(bar(L::kBarKFull + st), L::kKVBytes);
          for (int s = 0; s < L::kSlabs; ++s)
            tma_load_3d(sK(st) + s * (BC * 128), &tmK, bar(L::kBarKFull + st), s * 64, (t_begin + j) * BC, bh);
          ++k_arms[st];
        }
        if (j >= NS && !mbar_wait(bar(L::kBarVEmpty + st), ph ^ 1, wc)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(L::kBarVFull + st), L::kKVBytes);
        for (int s = 0; s < L::kSlabs; ++s)
          tma_load_3d(sV(st) + s * (BC * 128), &tmV, bar(L::kBarVFull + st), s * 64, (t_begin + j) * BC, bh);
        ++v_arms[st];
      }
      if (!ok) {
        // Let every copy this thread started land before shared memory is released: the
        // latest armed phase of each full barrier is the last copy issued into that stage.
        auto drain = [&](uint32_t b, uint32_t parity) {
          for (uint64_t t0 = global_timer_ns();
               !mbar_try_wait(b, parity) && global_timer_ns() - t0 < wc.limit_ns;) {
          }
        };
        drain(bar(L::kBarQFull), 0);
        for (int s = 0; s < NS; ++s) {
          if (k_arms[s] > 0) drain(bar(L::kBarKFull + s), (k_arms[s] - 1) & 1);
          if (v_arms[s] > 0) drain(bar(L::kBarVFull + s), (v_arms[s] - 1) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------------------------------------------------- MMA issuer ----
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kBM, BC, 0, 0);  // Q K^T: both K-major
      constexpr uint32_t kIdO = idesc_bf16_f32(kBM, D, 0, 1);   // P V: V is N(=d)-major
      auto issue_s = [&](int jj) -> bool {
        const int st = jj % NS;
        if (!mbar_wait(bar(L::kBarKFull + st), (jj / NS) & 1, wc)) return false;
        if (jj >= 2 && !mbar_wait(bar(L::kBarSFree + (jj & 1)), ((jj - 2) >> 1) & 1, wc)) return false;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + L::kColS + (jj & 1) * BC;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = sdesc_sw128(sQ + (kk >> 2) * (kBM * 128) + (kk & 3) * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sK(st) + (kk >> 2) * (BC * 128) + (kk & 3) * 32, 16, 1024);
          mma_ss(d_tmem, a, b, kIdS, kk > 0 ? 1u : 0u);
        }
        if constexpr (NS != 2) mma_commit(bar(L::kBarKEmpty + st));
        mma_commit(bar(L::kBarSFull + (jj & 1)));
        return true;
      };
      bool ok = mbar_wait(bar(L::kBarQFull), 0, wc);
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nkv; ++j) {
        if (j + 1 < nkv && !issue_s(j + 1)) { ok = false; break; }
        const int st = j % NS;
        if (!mbar_wait(bar(L::kBarVFull + st), (j / NS) & 1, wc) ||
            !mbar_wait(bar(L::kBarPFull + (j & 1)), (j >> 1) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t a_tmem = tmem + L::kColP + (j & 1) * (BC / 2);
#pragma unroll
        for (int kk = 0; kk < BC / 16; ++kk) {
          const uint64_t b = sdesc_sw128(sV(st) + kk * (16 * 128), BC * 128, 1024);
          mma_ts(tmem + L::kColO, a_tmem + kk * 8, b, kIdO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        if constexpr (L::kOwnOBar) mma_commit(bar(L::kBarODone));
        mma_commit(bar(L::kBarVEmpty + st));
      }
      // The epilogue cannot use the per-tile V-empty barriers: the softmax warps may run up to
      // two P V products ahead of the tensor core, and a parity wait cannot tell phases two
      // apart.  One commit after the last product marks the final O.
      if (ok) mma_commit(bar(L::kBarOFinal));
      // Every MMA issued above must be finished before TMEM is released.
      mma_commit(bar(L::kBarDrain));
      for (uint64_t t0 = global_timer_ns();
           !mbar_try_wait(bar(L::kBarDrain), 0) && global_timer_ns() - t0 < wc.limit_ns;) {
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax ----
    const int row = threadIdx.x;                 // 0..127 = TMEM lane
    const uint32_t lane_off = uint32_t(warp * 32) << 16;
    const int row_g = q0 + row;
    const float sl2 = args.scale_log2;
    float m_run = -INFINITY;  // running max of scale*log2(e)*s
    float l_run = 0.f;        // running sum of 2^(scaled s - m_run)
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int b = j & 1;
      const int kv0 = (t_begin + j) * BC;
      if constexpr (DROPOUT) {
        // The generator words of this row for the tile go to shared memory (the row's own
        // slots: no other thread reads them).  Four calls per iteration, interleaved; the loop
        // stays rolled, since unrolled the generator code overflows the instruction cache next
        // to the unrolled softmax.
        uint4* words = reinterpret_cast<uint4*>(smem + L::kDropOff) + row;
#pragma unroll 1
        for (int g = 0; g < BC / 8; g += 4) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            words[(g + u) * kBM] =
                dropout_words(args.dropout, uint32_t((kv0 >> 3) + g + u), uint32_t(row_g), uint32_t(bh));
        }
      }
      // tcgen05.ld is warp-collective: every wait outcome is made warp-uniform
      if (!__all_sync(0xffffffffu, mbar_wait(bar(L::kBarSFull + b), (j >> 1) & 1, wc))) { ok = false; break; }
      tc_fence_after_sync();
      float s[BC];
      {  // the whole S row in one TMEM load (one wait)
        uint32_t r[BC];
        if constexpr (BC == 128) tmem_ld128(tmem + lane_off + L::kColS + b * BC, r);
        else tmem_ld64(tmem + lane_off + L::kColS + b * BC, r);
#pragma unroll
        for (int i = 0; i < BC; ++i) s[i] = __uint_as_float(r[i]);
      }
      tc_fence_before_sync();
      mbar_arrive(bar(L::kBarSFree + b));

      // keys kv0 + c are visible for c < lim (sequence tail; causal: key <= query)
      int lim = Nk - kv0;
      if (CAUSAL) lim = min(lim, row_g - kv0 + 1);
      if (lim < BC) {
#pragma unroll
        for (int c = 0; c < BC; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      // row maximum: two chains of three-input maxima
      float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
#pragma unroll
      for (int c = 4; c < BC; c += 4) {
        mx0 = fmax3(mx0, s[c], s[c + 1]);
        mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
      }
      const float m_new = fmaxf(m_run, fmaxf(mx0, mx1) * sl2);
      const float alpha = ex2_approx(m_run - m_new);  // 0 on the first tile
      const bool grew = (j > 0) && (m_new > m_run);
      m_run = m_new;
      const float neg_m = -m_new;
      float2 sum2 = make_float2(0.f, 0.f);  // (even keys, odd keys)
      uint32_t pk[BC / 2];
      [[maybe_unused]] uint4 dw;  // dropout: words of keys c .. c+7
      [[maybe_unused]] const uint32_t t_lo = args.dropout.threshold, t_hi = args.dropout.threshold << 16;
#pragma unroll
      for (int c = 0; c < BC; c += 2) {
        // two keys per instruction for the scaling and the sums (same rounding as scalar)
        const float2 x = ffma2(make_float2(s[c], s[c + 1]), make_float2(sl2, sl2), make_float2(neg_m, neg_m));
        const float p0 = ex2_approx(x.x);
        const float p1 = ex2_approx(x.y);
        sum2 = fadd2(sum2, make_float2(p0, p1));
        if constexpr (DROPOUT) {
          // key c (even) is the low half of its word, key c + 1 the high half; the undropped
          // values stay in the sums
          if (c % 8 == 0) dw = reinterpret_cast<const uint4*>(smem + L::kDropOff)[(c / 8) * kBM + row];
          const uint32_t w = (c % 8 == 0) ? dw.x : (c % 8 == 2) ? dw.y : (c % 8 == 4) ? dw.z : dw.w;
          pk[c / 2] = pack_bf16x2((w & 0xFFFFu) >= t_lo ? p0 : 0.f, w >= t_hi ? p1 : 0.f);
        } else {
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
      }
      l_run = l_run * alpha + (sum2.x + sum2.y);
      // P_j into its TMEM buffer (its previous reader, P_{j-2} V_{j-2}, finished before
      // S_j was signalled).
#pragma unroll
      for (int c = 0; c < BC / 2; c += 32) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = pk[c + i];
        tmem_st32(tmem + lane_off + L::kColP + b * (BC / 2) + c, w);
      }
      // Rescale the accumulator when this warp's rows saw a larger maximum.  O holds
      // P_0..P_{j-1} V; wait until P_{j-1} V_{j-1} has landed.
      if (__any_sync(0xffffffffu, grew)) {
        // P_{j-1} V_{j-1} has landed when its V stage's empty barrier (or the O barrier)
        // completes; neither can lag two phases behind (S_j, already read, was issued after
        // P_{j-2} V_{j-2}) nor run one ahead (the next product needs a P this warp has not
        // written yet).
        const bool landed = L::kOwnOBar
                                ? mbar_wait(bar(L::kBarODone), (j - 1) & 1, wc)
                                : mbar_wait(bar(L::kBarVEmpty + (j - 1) % NS), ((j - 1) / NS) & 1, wc);
        if (!landed) ok = false;
        if (__all_sync(0xffffffffu, ok)) {
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + L::kColO + c, r);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const float2 y = fmul2(make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                     make_float2(alpha, alpha));
              r[i] = __float_as_uint(y.x);
              r[i + 1] = __float_as_uint(y.y);
            }
            tmem_st32(tmem + lane_off + L::kColO + c, r);
          }
        } else {
          ok = false;
        }
      }
      tmem_wait_st();
      tc_fence_before_sync();
      if (!ok) break;
      mbar_arrive(bar(L::kBarPFull + b));
    }

    // ------------------------------------------------------------ epilogue ----
    const bool fin = ok && __all_sync(0xffffffffu, mbar_wait(bar(L::kBarOFinal), 0, wc));
    constexpr bool split_mode = SPLIT;
    if (fin && split_mode) {
      // partial output of this key range: O normalised by its own l (fp32) and its LSE
      tc_fence_after_sync();
      const float inv_l = 1.f / l_run;
      const size_t prow = (size_t(blockIdx.z) * args.BH + bh) * N + row_g;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + L::kColO + c, r);
        if (row_g < N) {
          float4* dst = reinterpret_cast<float4*>(args.o_part + prow * D + c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]) * inv_l, __uint_as_float(r[4 * i + 1]) * inv_l,
                                 __uint_as_float(r[4 * i + 2]) * inv_l, __uint_as_float(r[4 * i + 3]) * inv_l);
        }
      }
      if (row_g < N) args.lse_part[prow] = (m_run + lg2_approx(l_run)) * 0.69314718055994531f;
    } else if (fin) {
      tc_fence_after_sync();
      const float inv_l = (DROPOUT ? args.dropout.scale : 1.f) / l_run;
      uint8_t* stage = smem + L::kQOff;  // Q is no longer read by any MMA
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + L::kColO + c, r);
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
      if (row_g < N)
        args.lse[size_t(bh) * N + row_g] = (m_run + lg2_approx(l_run)) * 0.69314718055994531f;
    }
    // Every softmax thread arrives (finished or not); thread 0 stores the tile only when all
    // 128 rows were staged and no wait in the CTA gave up.
    mbar_arrive(bar(L::kBarEpi));
    if (threadIdx.x == 0 && fin && !split_mode && mbar_wait(bar(L::kBarEpi), 0, wc) && *abort_flag == 0) {
      for (int s = 0; s < L::kSlabs; ++s) tma_store_3d(&tmO, sQ + s * (kBM * 128), s * 64, q0, bh);
      bulk_commit_group();
      bulk_wait_group_read_all();  // source read: the CTA may exit
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int D, int BC, int NS, bool CAUSAL>
cudaError_t launch_cfg(const Maps& m, const FwdArgs& a, cudaStream_t s, bool dropout) {
  const int smem = dropout ? FwdLayout<D, BC, NS, true>::kSmemAlloc : FwdLayout<D, BC, NS, false>::kSmemAlloc;
  // split-KV partial outputs and dropout are separate instantiations, so the plain square
  // problem's kernel carries none of that code
  if (dropout && a.o_part != nullptr) return cudaErrorInvalidValue;
  auto kern = dropout ? fa_fwd_kernel<D, BC, NS, CAUSAL, false, true>
                      : (a.o_part != nullptr ? fa_fwd_kernel<D, BC, NS, CAUSAL, true, false>
                                             : fa_fwd_kernel<D, BC, NS, CAUSAL, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_q_tiles, a.BH, a.num_splits);
  kern<<<grid, kThreads, smem, s>>>(m.q, m.k, m.v, m.o, a);
  return cudaGetLastError();
}

}  // namespace

int fwd_kv_tile(int d) { return d == 128 ? 128 : 64; }

cudaError_t launch_fwd(const Maps& m, const FwdArgs& a, int d, bool causal, cudaStream_t s, bool dropout) {
  switch (d) {
    case 64:
      // 64-key tiles keep TMEM at 256 columns and shared memory near 81 KB: two CTAs per SM
      return causal ? launch_cfg<64, 64, 4, true>(m, a, s, dropout) : launch_cfg<64, 64, 4, false>(m, a, s, dropout);
    case 128:
      return causal ? launch_cfg<128, 128, 2, true>(m, a, s, dropout)
                    : launch_cfg<128, 128, 2, false>(m, a, s, dropout);
    case 256:
      return causal ? launch_cfg<256, 64, 2, true>(m, a, s, dropout)
                    : launch_cfg<256, 64, 2, false>(m, a, s, dropout);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa
