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
// GB300 design (one CTA = one (batch, head, 128-key tile)):
//   warps 0-7   per query tile: read S^T and dP^T from tensor memory (lane =
//               key, warp w covers lanes 32*(w%4) and query half w/4), form
//               P^T (packed to 16 bits, back into tensor memory: the A operand
//               of dV) and dS = scale * P (dP - D) (16 bits, shared memory).
//               Then drain dQ from tensor memory with fp32 atomic adds.  At
//               the end, write dV and dK.
//   warp 8      TMA producer: K_j and V_j once, then per query tile Q_i, dO_i
//               (2-stage ring) and the 128 rows' LSE*log2(e) and D (bulk copies).
//   warp 9      UMMA issuer (one lane), owner of tensor memory:
//                 S^T  = K_j Q_i^T,  dP^T = V_j dO_i^T      (both operands K-major)
//                 dV  += P^T dO_i                            (A in TMEM, B MN-major)
//                 dK  += dS^T Q_i                            (A K-major, B MN-major)
//                 dQ_i = dS K_j, for D = 128 as dQ_i^T = K_j^T dS^T (A, B MN-major)
// dS is stored once, one 128-byte-swizzled row of queries per key, and read
// as both A operands: rows = keys, queries contiguous is dS^T K-major and
// dS MN-major.
// Tensor memory (512 columns): dV [0, D), dK [D, 2D), S^T [2D, 2D+128),
// dP^T [2D+128, 2D+256), and for D = 64 dQ after them.  P^T (64 columns)
// goes over columns 32..95 of S^T: each query half then writes only columns
// it has itself read (the half with queries 0..63 reads its upper 32 columns
// first), so neither half waits for the other.  For D = 128, dQ goes over
// dP^T once the softmax has read it; the next S^T is issued as soon as the
// previous products complete and the next dP^T once dQ has been drained.
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
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_DV = 0;
  static constexpr uint32_t COL_DK = D;
  static constexpr uint32_t COL_S = 2 * D;
  static constexpr uint32_t COL_DP = 2 * D + 128;
  // dQ over dP^T when a separate region does not fit (D = 128)
  static constexpr bool ALIAS = 2 * D + 256 + D > static_cast<int>(TMEM_COLS);
  static constexpr uint32_t COL_P = COL_S + 32;                  // P^T, 64 columns
  // D = 128: dQ^T = K^T dS^T (lane = head-dim index), so that a warp's
  // atomic adds cover 32 consecutive floats of one dQ row.  D = 64 keeps
  // dQ = dS K (lane = query; an M = 64 product would use half the lanes).
  static constexpr bool DQT = D == 128;
  static constexpr uint32_t COL_DQ = ALIAS ? COL_DP : COL_DP + 128;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + TILE_BYTES;
  static constexpr int OFF_Q = OFF_V + TILE_BYTES;
  static constexpr int OFF_DO = OFF_Q + NQS * TILE_BYTES;
  static constexpr int OFF_DS = OFF_DO + NQS * TILE_BYTES;  // 2 panels of 64 queries
  static constexpr int DS_BYTES = 2 * CHUNK_BYTES;
  static constexpr int OFF_ROW = OFF_DS + DS_BYTES;          // per stage: lse2[128], dd[128]
  static constexpr int ROW_BYTES = 1024;
  static constexpr int OFF_BAR = OFF_ROW + NQS * ROW_BYTES;
  // kv, qfull[NQS], qempty[NQS], sfull, pfull, dqfull, dqfree, bdone, fin
  static constexpr int NBAR = 1 + 2 * NQS + 6;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;       // tmem base, abort flag
  static constexpr int USED = OFF_MISC + 16;
  static constexpr int MAX_SMEM = 227 * 1024;
  static constexpr int SMEM_BYTES = USED + 1024 <= MAX_SMEM ? USED + 1024 : MAX_SMEM;
  static constexpr int THREADS = 320;
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(COL_DQ + D <= TMEM_COLS, "tensor memory budget");
  static_assert(USED + 16 <= SMEM_BYTES, "shared memory budget");
};

template <int D, bool CAUSAL, bool HALF>
__global__ void __launch_bounds__(320, 1)
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
  const uint32_t bSfull = bQempty + 8 * C::NQS;
  const uint32_t bPfull = bSfull + 8;
  const uint32_t bDQfull = bPfull + 8;
  const uint32_t bDQfree = bDQfull + 8;
  const uint32_t bBdone = bDQfree + 8;
  const uint32_t bFin = bBdone + 8;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int jt = static_cast<int>(blockIdx.x);  // key tile
  const int bh = static_cast<int>(blockIdx.z) * p.H + static_cast<int>(blockIdx.y);
  const int k0 = jt * BN;
  // Query tiles that see this key tile (top-left causal: query >= key).
  const int i_first = CAUSAL ? jt : 0;
  const int n_it = max(0, p.n_qtiles - i_first);

  if (threadIdx.x == 0) {
    mbar_init(bKV, 1);
#pragma unroll
    for (int s = 0; s < C::NQS; ++s) {
      mbar_init(bQfull + 8 * s, 1);
      mbar_init(bQempty + 8 * s, 1);
    }
    mbar_init(bSfull, 1);
    mbar_init(bPfull, 256);
    mbar_init(bDQfull, 1);
    mbar_init(bDQfree, 256);
    mbar_init(bBdone, 1);
    mbar_init(bFin, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  WaitCtl w{abort_flag, p.status, p.wait_limit_ns, 0u};

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    w.role = kStatusProducer;
    if (lane == 0 && n_it > 0) {
      const uint64_t pol_kv = l2_policy_evict_first();   // read by this CTA only
      const uint64_t pol_q = l2_policy_evict_last();     // read by every key tile
      mbar_arrive_expect_tx(bKV, 2 * C::TILE_BYTES);
#pragma unroll
      for (int c = 0; c < C::NCH; ++c) {
        tma_load_3d(sK + c * C::CHUNK_BYTES, &tm_k, bKV, c * C::CH_ELEMS, k0, bh, pol_kv);
        tma_load_3d(sV + c * C::CHUNK_BYTES, &tm_v, bKV, c * C::CH_ELEMS, k0, bh, pol_kv);
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
                      q0, bh, pol_q);
          tma_load_3d(sDO + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_do, bar,
                      c * C::CH_ELEMS, q0, bh, pol_q);
        }
        const size_t roff = static_cast<size_t>(bh) * p.Nq_pad + q0;
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
  } else if (warp == 9) {
    // ------------------------------------------------------------ UMMA issuer
    w.role = kStatusMma;
    if (lane == 0 && n_it > 0) {
      constexpr uint32_t kFmt = HALF ? 0u : 1u;                         // f16 / bf16
      constexpr uint32_t kIdescT = make_idesc(kFmt, 128, 128, 0u, 0u);  // S^T, dP^T
      constexpr uint32_t kIdescAcc = make_idesc(kFmt, 128, D, 0u, 1u);  // dV
      // dQ: M = 128 queries, N = D; dQ^T: M = 128 = D, N = 128 queries
      constexpr uint32_t kIdescDQ = make_idesc(kFmt, 128, C::DQT ? 128 : D, 1u, 1u);
      constexpr uint32_t kIdescDK = make_idesc(kFmt, 128, D, 0u, 1u);  // dK
      bool ok = bounded_wait(bKV, 0, w);
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it % C::NQS;
        if (!(ok = bounded_wait(bQfull + 8 * s, (it / C::NQS) & 1, w))) break;
        // S^T overwrites P^T of the previous tile, and the softmax rewrites dS
        // in shared memory after it: the previous products must be complete.
        if (it > 0 && !(ok = bounded_wait(bBdone, (it - 1) & 1, w))) break;
        tc_fence_after();
        const uint32_t qb = sQ + s * C::TILE_BYTES, db = sDO + s * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / C::UK; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          umma_ss<false>(tmem + C::COL_S, sdesc_sw128(sK + off, 16, 1024),
                         sdesc_sw128(qb + off, 16, 1024), kIdescT, kk > 0 ? 1u : 0u);
        }
        // D = 128: dP^T overwrites the previous dQ, which must be drained.
        if (C::ALIAS && it > 0) {
          if (!(ok = bounded_wait(bDQfree, (it - 1) & 1, w))) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kk = 0; kk < D / C::UK; ++kk) {
          const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          umma_ss<false>(tmem + C::COL_DP, sdesc_sw128(sV + off, 16, 1024),
                         sdesc_sw128(db + off, 16, 1024), kIdescT, kk > 0 ? 1u : 0u);
        }
        tc_commit(bSfull);
        if (!(ok = bounded_wait(bPfull, it & 1, w))) break;
        tc_fence_after();
        // dV += P^T dO: 16 queries per UMMA (8 packed TMEM columns of A; 16
        // rows of 128 bytes of the MN-major B).
#pragma unroll
        for (int kk = 0; kk < BM / C::UK; ++kk)
          umma_ts<false>(tmem + C::COL_DV, tmem + C::COL_P + kk * 8,
                         sdesc_sw128(db + kk * C::UK * 128, C::CHUNK_BYTES, 1024), kIdescAcc,
                         (it > 0 || kk > 0) ? 1u : 0u);
        // dK += dS^T Q: A = dS rows (keys) K-major, 16 queries = 32 bytes per
        // UMMA, two 64-query panels.
#pragma unroll
        for (int kk = 0; kk < BM / C::UK; ++kk)
          umma_ss<false>(tmem + C::COL_DK,
                         sdesc_sw128(sDS + (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32, 16, 1024),
                         sdesc_sw128(qb + kk * C::UK * 128, C::CHUNK_BYTES, 1024), kIdescDK,
                         (it > 0 || kk > 0) ? 1u : 0u);
        if (!C::ALIAS && it > 0) {
          if (!(ok = bounded_wait(bDQfree, (it - 1) & 1, w))) break;
          tc_fence_after();
        }
        // dQ_i = dS K_j, or for D = 128 its transpose K_j^T dS^T: 16 keys per
        // UMMA; dS (two 64-query panels) and K_j are both read MN-major.
#pragma unroll
        for (int kk = 0; kk < BN / C::UK; ++kk) {
          const uint64_t ds_desc = sdesc_sw128(sDS + kk * C::UK * 128, C::CHUNK_BYTES, 1024);
          const uint64_t k_desc = sdesc_sw128(sK + kk * C::UK * 128, C::CHUNK_BYTES, 1024);
          if constexpr (C::DQT)
            umma_ss<false>(tmem + C::COL_DQ, k_desc, ds_desc, kIdescDQ, kk > 0 ? 1u : 0u);
          else
            umma_ss<false>(tmem + C::COL_DQ, ds_desc, k_desc, kIdescDQ, kk > 0 ? 1u : 0u);
        }
        tc_commit(bQempty + 8 * s);
        tc_commit(bBdone);
        tc_commit(bDQfull);
      }
      (void)ok;
      tc_commit(bFin);
      bounded_wait(bFin, 0, w, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    w.role = kStatusSoftmax;
    const int g = warp >> 2;                  // query half of the tile
    const int wq = warp & 3;
    const int r = wq * 32 + lane;             // TMEM lane: key (S^T) or query (dQ)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int cb = 64 * g;                    // first query column of this half
    const float sl2 = p.scale_log2;
    const uint64_t sl2_2 = pk2(sl2, sl2);
    const uint64_t sc_2 = pk2(p.scale, p.scale);
    uint8_t *ds_row = smem + C::OFF_DS + g * C::CHUNK_BYTES + r * 128;
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it % C::NQS;
      const int qt = i_first + it;
      ok = __all_sync(kFullMask, bounded_wait(bQfull + 8 * s, (it / C::NQS) & 1, w));
      if (ok) ok = __all_sync(kFullMask, bounded_wait(bSfull, it & 1, w));
      if (!ok) break;
      tc_fence_after();
      const float *lse2 = reinterpret_cast<const float *>(smem + C::OFF_ROW + s * C::ROW_BYTES);
      const float *dd = lse2 + 128;
      const bool diag = CAUSAL && qt == jt;   // key r sees query c only if r <= c
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        // P^T of query half g lands in columns 32 + 32g .. of S^T: half 0
        // handles its upper 32 queries first, so no column is written before
        // this thread has read it.
        const int h = g == 0 ? 1 - hh : hh;
        const int c0 = cb + 32 * h;
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lane_off + C::COL_S + c0, sr);
        tmem_ld32(tmem + lane_off + C::COL_DP + c0, dr);
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
        tmem_st16(tmem + lane_off + C::COL_P + (c0 >> 1), pp);
        // dS row r of panel g: 16-byte unit u holds queries 8u..8u+7 of the
        // half; this chunk is units 4h..4h+3.
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4 *>(ds_row + (((4 * h + u) ^ (r & 7)) << 4)) =
              make_uint4(dsp[4 * u], dsp[4 * u + 1], dsp[4 * u + 2], dsp[4 * u + 3]);
      }
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bPfull);

      // dQ_i -> dq_acc with fp32 atomic adds.
      ok = __all_sync(kFullMask, bounded_wait(bDQfull, it & 1, w));
      if (!ok) break;
      tc_fence_after();
      if constexpr (C::DQT) {
        // dQ^T: lane r = head-dim index, columns = this half's 64 queries; the
        // warp's 32 lanes add to 32 consecutive floats of one dQ row.
        const int qbase = qt * BM + cb;
        float *dst = p.dq_acc + (static_cast<size_t>(bh) * p.Nq + qbase) * D + r;
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + C::COL_DQ + cb + c, v);
          tmem_ld_wait();
          reg_fence32(v);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (qbase + c + i < p.Nq) red_add(dst + static_cast<size_t>(c + i) * D, __uint_as_float(v[i]));
        }
      } else {
        // dQ: lane r = query row, columns = this half of d.
        const int qrow = qt * BM + r;
        float *dst = p.dq_acc + (static_cast<size_t>(bh) * p.Nq + qrow) * D + g * (D / 2);
#pragma unroll
        for (int c = 0; c < D / 2; c += 32) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + C::COL_DQ + g * (D / 2) + c, v);
          tmem_ld_wait();
          reg_fence32(v);
          if (qrow < p.Nq) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              red_add_v4(dst + c + 4 * u, __uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                         __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3]));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bDQfree);
    }

    // ---------------------------------------------------------- dV, dK out
    // Query half 0 writes dV, half 1 writes dK (row r = key k0 + r).
    if (ok && n_it > 0) ok = __all_sync(kFullMask, bounded_wait(bBdone, (n_it - 1) & 1, w));
    if (ok) {
      tc_fence_after();
      const int key = k0 + r;
      uint8_t *dst = static_cast<uint8_t *>(g == 0 ? p.dv : p.dk) +
                     (static_cast<size_t>(bh) * p.Nk + key) * D * 2;
      const uint32_t col = g == 0 ? C::COL_DV : C::COL_DK;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t v[32];
        if (n_it > 0) {
          tmem_ld32(tmem + lane_off + col + c, v);
          tmem_ld_wait();
          reg_fence32(v);
        } else {
          // no query sees these keys (causal, Nk > Nq): zero gradients
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        if (key < p.Nk) {
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
  if (warp == 9) {
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
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
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
