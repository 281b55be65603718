// fa_bwd.cuh — tensor-core (tcgen05) exact-attention backward for sm_103a.
//
// Method: the backward kernel of "flash_attention_2.cu"
// (leloykun/flash-hyperbolic-attention-minimal): the probabilities are
// recomputed from the saved log-sum-exp, P = exp(scale * Q K^T - L), and with
// D = rowsum(dO * O) (computed per row by the prep kernel)
//     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D),
//     dQ = scale * dS K,   dK = scale * dS^T Q.
// Loop order as on that page: one CTA per key tile, the query tiles inner,
// dK and dV kept on chip; dQ is accumulated across key tiles with global
// atomic adds.  The page's dV update reads the upstream gradient of the key's
// row instead of the query's; the product above is the derivative.
//
// GB300 design (one CTA = one (batch, head, 128-key tile), 16 warps).  Each
// 128-query tile is processed as two halves h of 64 queries with their own
// tensor memory, so that one half's softmax overlaps the other half's
// products:
//   warps 0-7   per half: read S_h^T and dP_h^T from tensor memory (lane =
//               key, warp w covers lanes 32*(w%4) and queries 32*(w/4) of the
//               half), form P^T (packed to 16 bits, back into tensor memory:
//               the A operand of dV) and dS = scale * P (dP - D) (16 bits,
//               shared memory).  At the end, write dV and dK.
//   warps 8-11  dQ drain: dQ_h^T out of tensor memory, then fp32 atomic adds
//               into the accumulator (an SM adds about 21 bytes per clock
//               whatever the number of warps, so the adds run beside the
//               softmax instead of after it).
//   warp 12     TMA producer: K_j and V_j once, then per query tile Q_i, dO_i
//               (2-stage ring) and the 128 rows' LSE*log2(e) and D (bulk copies).
//   warp 13     UMMA issuer (one lane), owner of tensor memory, per half h:
//                 dV  += P_h^T dO_h                         (A in TMEM, B MN-major)
//                 dK  += dS_h^T Q_h                         (A K-major, B MN-major)
//                 dQ_h^T = K_j^T dS_h^T                     (A, B MN-major)
//               then at once the next tile's
//                 S_h^T = K_j Q_h^T,  dP_h^T = V_j dO_h^T   (both operands K-major)
//               so half 0 of the next tile need not wait for half 1's products.
// The block is launched with 128 registers a thread; setmaxnreg gives the
// softmax warpgroups 152, the drain 104 and the producer/issuer group 104
// (the issuer's fully unrolled UMMA loops need them: rolled, each UMMA took
// about twice as long to issue).
// dS_h is stored once, one 128-byte-swizzled row of 64 queries per key, and
// read as two operands: rows = keys with queries contiguous is dS_h^T K-major
// (dK) and dS_h^T MN-major (dQ^T).  dQ^T has the head dimension on the TMEM
// lanes, so a warp's 32 atomic adds cover 32 consecutive floats of one dQ
// row.  (For D = 64 the dQ^T product still has M = 128: its A operand reads
// one 64-column panel past K_j, into V_j, and lanes 64-127 are not drained.)
// Tensor memory (512 columns): dV [0, D), dK [D, 2D), then per half h
// S_h^T [2D + 128h, +64) and dP_h^T [2D + 128h + 64, +64).  P_h^T (32
// columns) goes over columns 16..47 of S_h^T: each query quarter then writes
// only columns it has itself read, so neither waits for the other.  dQ_h^T
// goes over dP_h^T once the softmax has read it; the next tile's dP_h^T is
// issued once the drain warps have taken dQ_h^T into registers.
//
// Every wait is bounded (globaltimer); on expiry the CTA raises an abort
// flag, records its role in the status word, drains in-flight copies and
// UMMAs, frees tensor memory and exits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_internal.h"
#include "fa_wait.cuh"
#include "ptx.cuh"

namespace fa {

template <int D>
struct BwdCfg {
  static constexpr int NCH = D * 2 / 128;                  // 128-byte chunks per 16-bit row
  static constexpr int CH_ELEMS = 64;                       // elements per chunk
  static constexpr int CHUNK_BYTES = 128 * 128;             // 128 rows of one chunk
  static constexpr int TILE_BYTES = NCH * CHUNK_BYTES;      // one 128-row tile
  static constexpr int UK = 16;                             // K extent of one UMMA
  static constexpr int NQS = 2;                             // Q / dO ring depth
  static constexpr int HQ = 64;                             // queries per half tile
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_DV = 0;
  static constexpr uint32_t COL_DK = D;
  static constexpr uint32_t COL_S0 = 2 * D;                 // + 128 h: S_h^T
  static constexpr uint32_t COL_HALF = 128;                 // columns per half
  static constexpr uint32_t DP_OFF = 64;                    // dP_h^T after S_h^T
  static constexpr uint32_t P_OFF = 16;                     // P_h^T inside S_h^T
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + TILE_BYTES;
  static constexpr int OFF_DO = OFF_Q + NQS * TILE_BYTES;
  static constexpr int OFF_DS = OFF_DO + NQS * TILE_BYTES;  // + 16 KB h: dS_h
  static constexpr int DS_HALF_BYTES = 128 * 128;           // 128 keys x 64 queries
  static constexpr int OFF_ROW = OFF_DS + 2 * DS_HALF_BYTES; // per stage: lse2[128], dd[128]
  static constexpr int ROW_BYTES = 1024;
  static constexpr int OFF_BAR = OFF_ROW + NQS * ROW_BYTES;
  // kv, qfull[NQS], qempty[NQS], then per half: sfull, pfull, dqfull,
  // dqfree, hdone; fin
  static constexpr int NBAR = 1 + 2 * NQS + 2 * 5 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;       // tmem base, abort flag
  static constexpr int USED = OFF_MISC + 16;
  static constexpr int MAX_SMEM = 227 * 1024;
  static constexpr int SMEM_BYTES = USED + 1024 <= MAX_SMEM ? USED + 1024 : MAX_SMEM;
  // 16 warps: 0-7 softmax, 8-11 dQ drain, 12 producer, 13 UMMA issuer and
  // TMEM owner (14, 15 idle).  The block is launched with 128 registers a
  // thread; setmaxnreg moves them to the softmax warpgroups.
  static constexpr int THREADS = 512;
  static constexpr int WARP_PROD = 12;
  static constexpr int WARP_MMA = 13;
  static constexpr uint32_t REG_SOFTMAX = 152, REG_DRAIN = 104, REG_MISC = 104;
  static_assert(8 * 32 * REG_SOFTMAX + 4 * 32 * REG_DRAIN + 4 * 32 * REG_MISC <= THREADS * 128,
                "the register split must fit in what the block is launched with");
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(COL_S0 + 2 * COL_HALF <= TMEM_COLS, "tensor memory budget");
  static_assert(USED + 16 <= SMEM_BYTES, "shared memory budget");
};

template <int D, bool CAUSAL, bool HALF>
__global__ void __launch_bounds__(512, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr unsigned kFullMask = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  // The layout needs 1024-byte alignment; the launch reserves what is left
  // below 227 KB for it.  A base that leaves too little is reported, not used.
  if (static_cast<int>(smem - smem_raw) + C::USED > C::SMEM_BYTES) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusSmemLayout);
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO;
  const uint32_t sDS = sbase + C::OFF_DS, sRow = sbase + C::OFF_ROW;
  const uint32_t bKV = sbase + C::OFF_BAR;
  const uint32_t bQfull = bKV + 8;                 // + 8*stage
  const uint32_t bQempty = bQfull + 8 * C::NQS;    // + 8*stage
  const uint32_t bSfull = bQempty + 8 * C::NQS;    // + 8*half
  const uint32_t bPfull = bSfull + 16;             // + 8*half
  const uint32_t bDQfull = bPfull + 16;            // + 8*half
  const uint32_t bDQfree = bDQfull + 16;           // + 8*half
  const uint32_t bHdone = bDQfree + 16;            // + 8*half
  const uint32_t bFin = bHdone + 16;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int jt = static_cast<int>(blockIdx.x);  // key tile
  const int bh = static_cast<int>(blockIdx.z) * p.H + static_cast<int>(blockIdx.y);
  const int k0 = jt * BN;
  // Head dim of the tensors in memory: D, or less when a narrower head dim
  // runs zero-padded to D (the TMA loads zero-fill the missing columns; the
  // plain dQ, dK, dV writes below stop at dio).
  const int dio = p.d_io > 0 ? p.d_io : D;
  // This CTA's problem: rows [q_row0, q_row0 + Nq) of Q/dO and
  // [k_row0, k_row0 + Nk) of K/V/dK/dV in TMA plane hc.  dK/dV element
  // offset of row 0 and the row stride: [B,H,N,d] (plane b*H+h, rows dio
  // apart) or, for variable-length batches, token-major [total, H, d] (plane
  // h, rows H*dio apart).  The fp32 dQ accumulator is plane-major in both
  // cases, [B*H][Nq][D] or [H][total_q][D], so its row stride is the
  // compile-time D (the drain's 32 adds then share one address register).
  const bool varlen = p.cu_q != nullptr;
  int Nq = p.Nq, Nk = p.Nk, q_row0 = 0, k_row0 = 0, hc = bh, n_qtiles = p.n_qtiles;
  size_t row_base = static_cast<size_t>(bh) * p.Nq_pad;  // LSE/D rows of this problem
  size_t acc_base = static_cast<size_t>(bh) * p.Nq * D;   // dQ accumulator row 0
  long long kv_base = static_cast<long long>(bh) * p.Nk * dio, kv_rs = dio;
  if (varlen) {
    const int b = static_cast<int>(blockIdx.z), h = static_cast<int>(blockIdx.y);
    // Offsets are clamped to [0, total] (row indices never leave the
    // tensors) and lengths to the stated maxima (the padded LSE/D rows).
    q_row0 = min(max(p.cu_q[b], 0), p.total_q);
    k_row0 = min(max(p.cu_k[b], 0), p.total_k);
    Nq = min(max(0, min(p.cu_q[b + 1], p.total_q) - q_row0), p.Nq);
    Nk = min(max(0, min(p.cu_k[b + 1], p.total_k) - k_row0), p.Nk);
    hc = h;
    n_qtiles = (Nq + BM - 1) / BM;
    row_base = (static_cast<size_t>(h) * gridDim.z + b) * p.Nq_pad;
    acc_base = (static_cast<size_t>(h) * p.total_q + q_row0) * D;
    kv_base = (static_cast<long long>(k_row0) * p.H + h) * dio;
    kv_rs = static_cast<long long>(p.H) * dio;
    if (k0 >= Nk) return;  // the grid covers the longest sequence
  }
  // Query tiles that see this key tile (top-left causal: query >= key).
  const int i_first = CAUSAL ? jt : 0;
  const int n_it = max(0, n_qtiles - i_first);

  if (threadIdx.x == 0) {
    mbar_init(bKV, 1);
#pragma unroll
    for (int s = 0; s < C::NQS; ++s) {
      mbar_init(bQfull + 8 * s, 1);
      mbar_init(bQempty + 8 * s, 1);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mbar_init(bSfull + 8 * h, 1);
      mbar_init(bPfull + 8 * h, 256);
      mbar_init(bDQfull + 8 * h, 1);
      mbar_init(bDQfree + 8 * h, 128);
      mbar_init(bHdone + 8 * h, 1);
    }
    mbar_init(bFin, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == C::WARP_PROD && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == C::WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  WaitCtl w{abort_flag, p.status, p.wait_limit_ns, 0u};

  const int wg = warp >> 2;  // warpgroup: 0, 1 softmax; 2 dQ drain; 3 producer, issuer
  if (wg == 3) {
    setmaxnreg_dec<C::REG_MISC>();
    if (warp == C::WARP_PROD) {
      // ------------------------------------------------------------ producer
      w.role = kStatusProducer;
      if (lane == 0 && n_it > 0) {
        const uint64_t pol_kv = l2_policy_evict_first();   // read by this CTA only
        const uint64_t pol_q = l2_policy_evict_last();     // read by every key tile
        mbar_arrive_expect_tx(bKV, 2 * C::TILE_BYTES);
  #pragma unroll
        for (int c = 0; c < C::NCH; ++c) {
          tma_load_3d(sK + c * C::CHUNK_BYTES, &tm_k, bKV, c * C::CH_ELEMS, k_row0 + k0, hc, pol_kv);
          tma_load_3d(sV + c * C::CHUNK_BYTES, &tm_v, bKV, c * C::CH_ELEMS, k_row0 + k0, hc, pol_kv);
        }
        int issued = 0;
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
          const int s = it % C::NQS, r = it / C::NQS;
          if (r > 0 && !(ok = bounded_wait(bQempty + 8 * s, (r - 1) & 1, w))) break;
          const int q0 = (i_first + it) * BM;
          const uint32_t bar = bQfull + 8 * s;
          mbar_arrive_expect_tx(bar, 2 * C::TILE_BYTES + C::ROW_BYTES);
  #pragma unroll
          for (int c = 0; c < C::NCH; ++c) {
            tma_load_3d(sQ + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_q, bar, c * C::CH_ELEMS,
                        q_row0 + q0, hc, pol_q);
            tma_load_3d(sDO + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_do, bar,
                        c * C::CH_ELEMS, q_row0 + q0, hc, pol_q);
          }
          // (debug build: a row block outside the buffers is replaced by
          // block 0, so the barrier still gets its bytes)
          const size_t roff = FA_IN(p.status, row_base + q0, 128, p.row_elems) ? row_base + q0 : 0;
          bulk_load(sRow + s * C::ROW_BYTES, p.lse2 + roff, 512, bar);
          bulk_load(sRow + s * C::ROW_BYTES + 512, p.dd + roff, 512, bar);
          ++issued;
        }
        (void)ok;
        // Drain: no copy may still be writing shared memory when the CTA exits.
        bounded_wait(bKV, 0, w, false);
        for (int s = 0; s < C::NQS; ++s) {
          const int cnt = (issued > s) ? (issued - 1 - s) / C::NQS + 1 : 0;
          if (cnt > 0) bounded_wait(bQfull + 8 * s, (cnt - 1) & 1, w, false);
        }
      }
      __syncwarp();
    } else if (warp == C::WARP_MMA) {
      // ------------------------------------------------------------ UMMA issuer
      w.role = kStatusMma;
      if (lane == 0 && n_it > 0) {
        constexpr uint32_t kFmt = HALF ? 0u : 1u;                        // f16 / bf16
        constexpr uint32_t kIdescS = make_idesc(kFmt, 128, C::HQ, 0u, 0u); // S^T, dP^T
        constexpr uint32_t kIdescAcc = make_idesc(kFmt, 128, D, 0u, 1u);   // dV, dK
        constexpr uint32_t kIdescDQ = make_idesc(kFmt, 128, C::HQ, 1u, 1u); // dQ^T
        // S_h^T = K_j Q_h^T (over P_h^T of the previous tile) and
        // dP_h^T = V_j dO_h^T (over dQ_h^T of the previous tile) of tile t.
        auto issue_s = [&](int t, int h) {
          const int s = t % C::NQS;
          const uint32_t qb = sQ + s * C::TILE_BYTES;
          const uint32_t col = C::COL_S0 + h * C::COL_HALF;
  #pragma unroll
          for (int kk = 0; kk < D / C::UK; ++kk) {
            const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
            umma_ss<false>(tmem + col, sdesc_sw128(sK + off, 16, 1024),
                           sdesc_sw128(qb + h * C::HQ * 128 + off, 16, 1024), kIdescS,
                           kk > 0 ? 1u : 0u);
          }
        };
        auto issue_dp = [&](int t, int h) {
          const int s = t % C::NQS;
          const uint32_t db = sDO + s * C::TILE_BYTES;
          const uint32_t col = C::COL_S0 + h * C::COL_HALF;
  #pragma unroll
          for (int kk = 0; kk < D / C::UK; ++kk) {
            const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
            umma_ss<false>(tmem + col + C::DP_OFF, sdesc_sw128(sV + off, 16, 1024),
                           sdesc_sw128(db + h * C::HQ * 128 + off, 16, 1024), kIdescS,
                           kk > 0 ? 1u : 0u);
          }
          tc_commit(bSfull + 8 * h);
        };
        bool ok = bounded_wait(bKV, 0, w) && bounded_wait(bQfull, 0, w);
        if (ok) {
          tc_fence_after();
  #pragma unroll
          for (int h = 0; h < 2; ++h) {
            issue_s(0, h);
            issue_dp(0, h);
          }
        }
        // Per half h of tile t: the products once its P^T and dS are written,
        // then at once the next tile's S_h^T, dP_h^T into the same columns (so
        // the softmax of half 0 of tile t+1 need not wait for half 1's
        // products of tile t).
        for (int it = 0; ok && it < n_it; ++it) {
          const int s = it % C::NQS;
          const uint32_t qb = sQ + s * C::TILE_BYTES, db = sDO + s * C::TILE_BYTES;
          const bool next = it + 1 < n_it;
  #pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t col = C::COL_S0 + h * C::COL_HALF;
            if (!(ok = bounded_wait(bPfull + 8 * h, it & 1, w))) break;
            tc_fence_after();
            const uint32_t ds = sDS + h * C::DS_HALF_BYTES;
            // dV += P_h^T dO_h and dK += dS_h^T Q_h: 16 queries per UMMA (8
            // packed TMEM columns of P^T, 32 bytes of a dS row; 16 rows of
            // 128 bytes of the MN-major B).
  #pragma unroll
            for (int kk = 0; kk < C::HQ / C::UK; ++kk) {
              const uint32_t brow = (h * C::HQ + kk * C::UK) * 128;
              const uint32_t acc = (it > 0 || h > 0 || kk > 0) ? 1u : 0u;
              umma_ts<false>(tmem + C::COL_DV, tmem + col + C::P_OFF + kk * 8,
                             sdesc_sw128(db + brow, C::CHUNK_BYTES, 1024), kIdescAcc, acc);
              umma_ss<false>(tmem + C::COL_DK, sdesc_sw128(ds + kk * 32, 16, 1024),
                             sdesc_sw128(qb + brow, C::CHUNK_BYTES, 1024), kIdescAcc, acc);
            }
            // dQ_h^T = K_j^T dS_h^T over dP_h^T: 16 keys per UMMA.
  #pragma unroll
            for (int kk = 0; kk < BN / C::UK; ++kk)
              umma_ss<false>(tmem + col + C::DP_OFF,
                             sdesc_sw128(sK + kk * C::UK * 128, C::CHUNK_BYTES, 1024),
                             sdesc_sw128(ds + kk * C::UK * 128, C::CHUNK_BYTES, 1024), kIdescDQ,
                             kk > 0 ? 1u : 0u);
            tc_commit(bHdone + 8 * h);
            tc_commit(bDQfull + 8 * h);
            if (next) {
              // Tile t+1 in its stage; half h's products complete (they read
              // P_h^T and dS_h, which S_h^T and the softmax overwrite); dQ_h^T
              // moved out of tensor memory by the drain warps.
              if (h == 0 && !(ok = bounded_wait(bQfull + 8 * ((it + 1) % C::NQS),
                                                ((it + 1) / C::NQS) & 1, w)))
                break;
              if (!(ok = bounded_wait(bHdone + 8 * h, it & 1, w))) break;
              tc_fence_after();
              issue_s(it + 1, h);
              if (!(ok = bounded_wait(bDQfree + 8 * h, it & 1, w))) break;
              tc_fence_after();
              issue_dp(it + 1, h);
            }
          }
          tc_commit(bQempty + 8 * s);
        }
        (void)ok;
        tc_commit(bFin);
        bounded_wait(bFin, 0, w, false);
      }
      __syncwarp();
    }
  } else if (wg == 2) {
    setmaxnreg_dec<C::REG_DRAIN>();
    // ------------------------------------------------------------ dQ drain
    // dQ_h^T -> dq_acc with fp32 atomic adds: lane r = head-dim index, the
    // half's 64 queries; the warp's 32 lanes add to 32 consecutive floats of
    // one dQ row.  The values are taken out of tensor memory first, so the
    // next tile's dP_h^T may go in while the adds (limited to about 21 bytes
    // per clock per SM) run beside the softmax warps.  (D = 64: lanes 64-127
    // hold no dQ.)
    w.role = kStatusSoftmax;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const int qt = i_first + it;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const uint32_t col = C::COL_S0 + h * C::COL_HALF;
        ok = __all_sync(kFullMask, bounded_wait(bDQfull + 8 * h, it & 1, w));
        if (!ok) break;
        tc_fence_after();
        uint32_t v[64];
        if (r < dio) {   // whole warps (dio is a multiple of 32)
          uint32_t (&v0)[32] = *reinterpret_cast<uint32_t (*)[32]>(v);
          uint32_t (&v1)[32] = *reinterpret_cast<uint32_t (*)[32]>(v + 32);
          tmem_ld32(tmem + lane_off + col + C::DP_OFF, v0);
          tmem_ld32(tmem + lane_off + col + C::DP_OFF + 32, v1);
          tmem_ld_wait();
          reg_fence32(v0);
          reg_fence32(v1);
        }
        tc_fence_before();
        mbar_arrive(bDQfree + 8 * h);
        if (r < dio) {
          const int qbase = qt * BM + h * C::HQ;
          float *dst = p.dq_acc + acc_base + static_cast<size_t>(qbase) * D + r;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (qbase + i < Nq &&
                FA_IN(p.status, acc_base + static_cast<size_t>(qbase + i) * D + r, 1, p.dq_elems))
              red_add(dst + i * D, __uint_as_float(v[i]));
        }
      }
    }
    __syncwarp();
  } else {
    setmaxnreg_inc<C::REG_SOFTMAX>();
    // ------------------------------------------------------------ softmax warps
    w.role = kStatusSoftmax;
    const int g = warp >> 2;                  // query quarter within a half
    const int wq = warp & 3;
    const int r = wq * 32 + lane;             // TMEM lane: key (S^T) or head dim (dQ^T)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int cq = 32 * g;                    // first query column of this quarter
    const float sl2 = p.scale_log2;
    const uint64_t sl2_2 = pk2(sl2, sl2);
    const uint64_t sc_2 = pk2(p.scale, p.scale);
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it % C::NQS;
      const int qt = i_first + it;
      ok = __all_sync(kFullMask, bounded_wait(bQfull + 8 * s, (it / C::NQS) & 1, w));
      if (!ok) break;
      const float *lse2 = reinterpret_cast<const float *>(smem + C::OFF_ROW + s * C::ROW_BYTES);
      const float *dd = lse2 + 128;
      const bool diag = CAUSAL && qt == jt;   // key r sees query c only if r <= c
      // Query columns past Nq have LSE = +inf (prep kernel), so P = 0 there.
      // Key rows past Nk: their dK, dV rows are not stored, and their dS is
      // zeroed below, so they add nothing to dQ (for variable-length batches
      // those rows hold the next sequence's keys, not zeros).
      const bool krow_ok = k0 + r < Nk;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t col = C::COL_S0 + h * C::COL_HALF;
        ok = __all_sync(kFullMask, bounded_wait(bSfull + 8 * h, it & 1, w));
        if (!ok) break;
        tc_fence_after();
        const int c0 = h * C::HQ + cq;          // query index in the tile of column 0
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lane_off + col + cq, sr);
        tmem_ld32(tmem + lane_off + col + C::DP_OFF + cq, dr);
        tmem_ld_wait();
        reg_fence32(sr);
        reg_fence32(dr);
        uint32_t pp[16], dsp[16];
#pragma unroll
        for (int t = 0; t < 32; t += 4) {
          const float4 l4 = *reinterpret_cast<const float4 *>(lse2 + c0 + t);
          const float4 d4 = *reinterpret_cast<const float4 *>(dd + c0 + t);
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const float la = u == 0 ? l4.x : l4.z, lb = u == 0 ? l4.y : l4.w;
            const float da = u == 0 ? d4.x : d4.z, db = u == 0 ? d4.y : d4.w;
            const int c = t + u;
            const uint64_t x2 = ffma2(pk2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                                      sl2_2, pk2(-la, -lb));
            float x0, x1;
            upk2(x2, x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (diag) {
              if (c0 + c < r) p0 = 0.f;
              if (c0 + c + 1 < r) p1 = 0.f;
            }
            const uint64_t g2 = fadd2(pk2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])),
                                      pk2(-da, -db));
            float s0, s1;
            upk2(fmul2(fmul2(pk2(p0, p1), g2), sc_2), s0, s1);
            pp[c >> 1] = HALF ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            dsp[c >> 1] = HALF ? pack_f16x2(s0, s1) : pack_bf16x2(s0, s1);
          }
        }
        if (!krow_ok) {
#pragma unroll
          for (int u = 0; u < 16; ++u) dsp[u] = 0u;
        }
        // P^T columns 16 + 16g ..: inside the 32 columns this quarter read.
        tmem_st16(tmem + lane_off + col + C::P_OFF + 16 * g, pp);
        // dS_h row r: 16-byte unit u holds queries 8u..8u+7 of the half; this
        // quarter's 32 queries are units 4g..4g+3.
        uint8_t *ds_row = smem + C::OFF_DS + h * C::DS_HALF_BYTES + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4 *>(ds_row + (((4 * g + u) ^ (r & 7)) << 4)) =
              make_uint4(dsp[4 * u], dsp[4 * u + 1], dsp[4 * u + 2], dsp[4 * u + 3]);
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bPfull + 8 * h);
      }
    }

    // ---------------------------------------------------------- dV, dK out
    // Quarter 0 writes dV, quarter 1 writes dK (row r = key k0 + r).  The
    // last tile's half-1 products complete after every earlier UMMA.
    if (ok && n_it > 0) ok = __all_sync(kFullMask, bounded_wait(bHdone + 8, (n_it - 1) & 1, w));
    if (ok) {
      tc_fence_after();
      const int key = k0 + r;
      uint8_t *dst = static_cast<uint8_t *>(g == 0 ? p.dv : p.dk) +
                     (kv_base + static_cast<long long>(key) * kv_rs) * 2;
      const uint32_t colv = g == 0 ? C::COL_DV : C::COL_DK;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t v[32];
        if (n_it > 0) {
          tmem_ld32(tmem + lane_off + colv + c, v);
          tmem_ld_wait();
          reg_fence32(v);
        } else {
          // no query sees these keys (causal, Nk > Nq): zero gradients
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (key < Nk && c < dio &&
            FA_IN(p.status, kv_base + static_cast<long long>(key) * kv_rs + c, 32, p.kv_elems)) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 val;
            auto pk = [](uint32_t a, uint32_t b) {
              return HALF ? pack_f16x2(__uint_as_float(a), __uint_as_float(b))
                          : pack_bf16x2(__uint_as_float(a), __uint_as_float(b));
            };
            val.x = pk(v[8 * u + 0], v[8 * u + 1]);
            val.y = pk(v[8 * u + 2], v[8 * u + 3]);
            val.z = pk(v[8 * u + 4], v[8 * u + 5]);
            val.w = pk(v[8 * u + 6], v[8 * u + 7]);
            reinterpret_cast<uint4 *>(dst + c * 2)[u] = val;
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == C::WARP_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool HALF>
cudaError_t launch_bwd(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                       const CUtensorMap &dout, const BwdParams &p, int B, int causal,
                       cudaStream_t stream) {
  using C = BwdCfg<D>;
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
               const BwdParams) =
      causal ? fa_bwd_kernel<D, true, HALF> : fa_bwd_kernel<D, false, HALF>;
  static std::atomic<unsigned long long> attr_done[2];  // per causal flag
  cudaError_t e = smem_attr_once(kern, C::SMEM_BYTES, &attr_done[causal ? 1 : 0]);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.n_ktiles), static_cast<unsigned>(p.H),
                     static_cast<unsigned>(B));
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, dout, p);
}

}  // namespace fa
