// fa_tc.cuh — tensor-core (tcgen05) exact-attention forward for sm_103a.
//
// Method: the forward kernel of "flash_attention_2.cu"
// (leloykun/flash-hyperbolic-attention-minimal) — scores S = scale * Q K^T,
// online softmax with a running row max m and row sum l, the partial output
// rescaled by exp(m_old - m_new), and at the end O = O / l, L = m + log(l).
// Loop order: the swapped one from "parallel execution of read/write
// operations (paper vs implementation)" (query tiles outer, keys inner, O kept
// on chip and written once).  Parallelism: over queries as well as
// batch and heads, as in "Meta's xFormers has Attention kernel written in
// CUTLASS".  exp2 with log2(e) folded into the scale, as in "Add Fused
// Multi-Head Attention example" (cuTile.jl).
//
// GB300 design (one CTA = one (batch, head) and one to four 128-row query
// tiles, "items", run through one pipeline; see tc_items and item_qt):
//   warps 0-3    softmax, correction and epilogue: one query row per thread
//                (= one TMEM lane).  Where Q lives in tensor memory, first copy
//                the thread's Q row there from global memory (the A operand of
//                S = Q K^T).  Per key tile: load the
//                row's 128 scores, mask the causal diagonal / ragged key tail,
//                update m and l, write P back over S in TMEM.  At the
//                end of an item normalise O, stage it swizzled in shared
//                memory for a TMA store, and write LSE.
//   warp 4       TMA producer: Q (when in shared memory), then K_j / V_j
//                through shared-memory rings (full/empty mbarriers), L2
//                evict-last for K/V.
//   warp 5       UMMA issuer (one lane) for S_j = Q K_j^T (A = Q from TMEM or
//                shared memory, B = K_j K-major in shared memory) into score
//                buffer j % NS (NS = 3 for bf16: two score tiles can be
//                computed ahead of the softmax).  Owns the TMEM allocation.
//   warp 6       UMMA issuer (one lane) for O += P_j V_j (A = P from TMEM),
//                fp32 accumulation.  A tcgen05.mma issue returns at about the
//                rate the tensor pipe executes it, so one issuing thread would
//                leave the pipe idle during every wait and commit between its
//                batches; with two, each batch's bookkeeping overlaps the other
//                product's MMAs.
// bf16 inputs (kind::f16): P is bf16; V_j is an MN-major B operand as loaded.
// fp32 inputs (kind::tf32): the tensor core truncates fp32 operands to tf32,
// which biases the scores; so Q (on its way to TMEM) and K_j (in place, by the
// softmax warps, before S_j is issued) are rounded to nearest first.  P is
// tf32.  kind::tf32 takes its B operand K-major only, so the softmax warps
// also transpose each V_j into a tf32 V_j^T buffer (d rows of 128 keys).  At
// D=128 the fp32 tiles are 64 KB: one K, one V and one V^T buffer.  With
// staged operands (the S16 instantiations) a pre-pass has already split K
// into bf16 halves and written V^T once per call: the scores are three bf16
// products of the split Q and K, K_j's halves are used as loaded and V_j^T is
// loaded by TMA into the V^T buffers (through the V ring's barriers), so the
// softmax warps only do the softmax.
// Tensor memory: S_b cols [128b, 128b+128) for b < NS, then O (D cols), then Q
// when it fits (bf16 D=64, fp32 D=64); bf16 D=128 and D=256 keep Q in shared
// memory.  D=256 has two score buffers and single-stage K/V rings (64 KB
// tiles).
//
// Rescaling: the running max used as the exponent offset only moves when a
// row's max grows by more than 2^8; otherwise the stale offset is kept.  The
// softmax is invariant to the offset, so the result is exact up to rounding;
// unshifted terms are at most 2^8, far inside the fp32/bf16 range.
//
// Every wait is bounded (globaltimer); on expiry the CTA sets an abort flag,
// records its role in the device status word, drains in-flight TMA loads and
// UMMAs, frees tensor memory and exits.
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "fa_internal.h"
#include "fa_wait.cuh"
#include "ptx.cuh"

namespace fa {

// S16 (fp32 inputs with staged operands only): the scores are three bf16
// products of split operands instead of three tf32 ones (see NQSPLIT).
template <int D, bool TF32, bool S16 = false>
struct TcCfg {
  static_assert(!S16 || TF32, "bf16 split scores are a variant of the fp32 path");
  static constexpr int ESZ = TF32 ? 4 : 2;                 // bytes per element
  static constexpr int NCH = D * ESZ / 128;                 // 128-byte swizzle chunks per row
  static constexpr int CH_ELEMS = 128 / ESZ;                // elements per chunk
  static constexpr int CHUNK_BYTES = 128 * 128;             // one chunk of 128 rows
  static constexpr int TILE_BYTES = NCH * CHUNK_BYTES;      // one 128-row tile
  static constexpr int UK = 32 / ESZ;                       // K extent of one UMMA
  // Score buffers in tensor memory: S_j lives in buffer j % NS; S_j may be
  // issued once P_{j-NS} V_{j-NS} is done, so NS - 1 score tiles can be
  // computed ahead of the softmax.  (fp32 at D = 128: one buffer, because
  // both halves of the split Q fill the rest of tensor memory; with bf16
  // halves, half as wide, one more.)
  static constexpr int NS = TF32 ? (D >= 128 ? 1 : 2) + (S16 ? 1 : 0) : (D >= 256 ? 2 : 3);
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_O = NS * 128;               // O after the score buffers
  // 32-bit columns of one Q row (S16: of one bf16 half of the split Q)
  static constexpr int Q_COLS = S16 ? D / 2 : D * ESZ / 4;
  // fp32 path: S = Q K^T runs as three products of the split operands,
  // Q_hi K_hi + Q_hi K_lo + Q_lo K_hi, x_hi = r(x), x_lo = r(x - x_hi) with r
  // the rounding to tf32 (about 2^-22 of x left out), or (S16) to bf16 (about
  // 2^-16 left out, at twice the tf32 rate and half the instructions).  Either
  // way the scores carry far more than one product's accuracy (tf32: 2^-11).
  static constexpr int NQSPLIT = TF32 ? 2 : 1;
  // S16: K_hi and K_lo arrive as bf16 tiles (KCH chunks of 128 rows).
  static constexpr int KCH = S16 ? D * 2 / 128 : D * ESZ / 128;
  static constexpr int K_CH_ELEMS = S16 ? 64 : 128 / ESZ;
  static constexpr int K_TILE_BYTES = KCH * 128 * 128;
  // Q is the A operand of S = Q K^T.  The fp32 path rounds (splits) it on
  // its way into tensor memory; the 16-bit path loads it into shared memory
  // by TMA, even at D = 64 where it would fit in tensor memory: there the S
  // products' tensor-memory reads competed with the softmax warps' loads and
  // stores, and the kernel ran 3% slower.
  static constexpr bool QTMEM = TF32 && COL_O + D + NQSPLIT * Q_COLS <= TMEM_COLS;
  static constexpr uint32_t COL_Q = COL_O + D;
  static constexpr uint32_t COL_QLO = COL_Q + Q_COLS;      // fp32 path: Q_lo
  static constexpr int NQ = QTMEM ? 0 : 1;                  // Q tiles in shared memory
  // K / V ring depths: as deep as shared memory allows (64 KB tiles at
  // D = 256 leave room for one stage each beside Q).
  static constexpr int KST = TILE_BYTES >= 65536 ? 1 : TF32 ? 2 : TILE_BYTES <= 16384 ? 4 : 3;
  static constexpr int VST = KST;
  // fp32 path: V_j is transposed by the softmax warps into a K-major copy
  // (V^T, d rows of 128 keys, tf32-rounded) because P V runs as kind::tf32
  // with V^T as a K-major B operand.  Two copies alternate.
  static constexpr int NVT = TF32 ? (TILE_BYTES >= 65536 ? 1 : 2) : 0;
  static constexpr int VT_CHUNK_BYTES = D * 128;            // 32 keys x D rows
  // fp32 path, K_lo of the split: with staged operands it is loaded into the
  // V ring's stage s beside K_hi in K stage s (the V ring is free: V^T goes
  // straight to the V^T buffers).  Converted in the kernel, it goes to one
  // buffer of its own at D = 64, and at D = 128 to the one V^T buffer, which
  // holds K_lo_j until S_j completes and V_j^T after that.
  static constexpr int NKLO = (TF32 && NVT >= 2) ? 1 : 0;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + KST * TILE_BYTES;
  static constexpr int OFF_KLO = OFF_V + VST * TILE_BYTES;
  static constexpr int OFF_VT = OFF_KLO + NKLO * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_VT + NVT * TILE_BYTES;
  // q, kfull[KST], kempty[KST], vfull[VST], vempty[VST], sfull[NS], pfull[NS],
  // odone[NS], fin[2], kready[KST]
  // ... then qempty, ofree, ostaged[kItemRing] (several query tiles per CTA)
  static constexpr int NBAR = 1 + 2 * KST + 2 * VST + 3 * NS + 2 + KST + 2 + kItemRing;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;       // tmem base, abort flag
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // + alignment slack
  static constexpr int THREADS = 224;
  static_assert(NCH >= 1 && D % 32 == 0, "head dim must fill whole 128-byte chunks");
  static_assert(COL_O + D <= TMEM_COLS, "tensor memory budget");
  static_assert(!TF32 || QTMEM, "the fp32 path rounds Q on its way into tensor memory");
  static_assert(!TF32 || VST == NVT, "staged V^T tiles use the V ring's barriers");
  static_assert(!TF32 || KST == VST, "staged K_lo tiles sit in the V stage of their K stage");
  static_assert(!TF32 || S16 || NKLO == 1 || NS == 1,
                "K_lo shares the V^T buffer only where S_j completes before V_j^T is written");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(VST + 1 <= kItemRing, "items with O staged in a V stage fit the item ring");
};

constexpr float kRescaleThreshold = 8.0f;   // log2 units: factor 256
constexpr float kLn2 = 0.693147180559945309f;
constexpr unsigned kFull = 0xffffffffu;

// HALF selects fp16 instead of bf16 for the 16-bit path (kind::f16 either
// way; P and O are packed in the input type).
template <int D, bool TF32, bool CAUSAL, bool HALF, bool S16 = false>
__global__ void __launch_bounds__(224, 1)
    fa_tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_o,
                     const __grid_constant__ CUtensorMap tm_klo, const TcParams p) {
  using C = TcCfg<D, TF32, S16>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q;   // used when Q is not in tensor memory
  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;
  const uint32_t sVT = sbase + C::OFF_VT;
  const uint32_t sKLO = sbase + C::OFF_KLO;  // fp32, converted in the kernel, D = 64
  const uint32_t bQ = sbase + C::OFF_BAR;             // Q in place (TMEM or smem)
  const uint32_t bKfull = bQ + 8;                      // + 8*stage
  const uint32_t bKempty = bKfull + 8 * C::KST;
  const uint32_t bVfull = bKempty + 8 * C::KST;
  const uint32_t bVempty = bVfull + 8 * C::VST;
  const uint32_t bSfull = bVempty + 8 * C::VST;        // + 8*score buffer
  const uint32_t bPfull = bSfull + 8 * C::NS;          // + 8*score buffer
  const uint32_t bOdone = bPfull + 8 * C::NS;          // + 8*score buffer
  const uint32_t bFin = bOdone + 8 * C::NS;            // S issuer's teardown
  const uint32_t bFin2 = bFin + 8;                     // P V issuer's teardown
  const uint32_t bKready = bFin2 + 8;                  // + 8*stage (fp32 path)
  const uint32_t bQempty = bKready + 8 * C::KST;       // Q of an item read by its last S
  const uint32_t bOfree = bQempty + 8;                 // O of an item read by the epilogue
  const uint32_t bOstaged = bOfree + 8;                // + 8*(item % kItemRing): O staged
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Causal: heaviest query tiles first (blockIdx.x = 0 gets the last tile).
  const int nsp = p.n_splits;
  const int qidx = nsp > 1 ? static_cast<int>(blockIdx.x) / nsp : static_cast<int>(blockIdx.x);
  const int split = static_cast<int>(blockIdx.x) - qidx * nsp;
  const int bh = static_cast<int>(blockIdx.z) * p.H + static_cast<int>(blockIdx.y);
  // This CTA's sequence: rows [q_row0, q_row0 + Nq) of Q/O and [k_row0,
  // k_row0 + Nk) of K/V in head plane hc of the tensor maps.
  int Nq = p.Nq, Nk = p.Nk, q_row0 = 0, k_row0 = 0, hc = bh;
  int n_qtiles = p.n_qtiles, n_ktiles = p.n_ktiles;
  if (p.cu_q != nullptr) {
    griddep_wait();  // the offsets are in global memory
    const int b = static_cast<int>(blockIdx.z);
    // Offsets clamped to [0, total]: row indices never leave the tensors,
    // and bad offsets cannot make a CTA walk more key tiles than exist.
    q_row0 = min(max(p.cu_q[b], 0), p.total_q);
    k_row0 = min(max(p.cu_k[b], 0), p.total_k);
    Nq = max(0, min(p.cu_q[b + 1], p.total_q) - q_row0);
    Nk = max(0, min(p.cu_k[b + 1], p.total_k) - k_row0);
    hc = static_cast<int>(blockIdx.y);
    n_qtiles = (Nq + BM - 1) / BM;
    n_ktiles = (Nk + BN - 1) / BN;
    if (qidx >= n_qtiles) return;  // the grid covers the longest sequence
  }
  // Persistent schedule (plain problems, 16-bit types): the grid has about
  // one CTA per SM, and CTA x runs the query tiles fwd_item() deals it, of
  // any heads, one after another through one pipeline, so an item's loads
  // and first products overlap the previous item's epilogue and the CTA's
  // set-up is paid once.  (The fp32 path always runs one item: a constant, so
  // its kernels carry none of the multi-item code and keep their registers.)
  const bool persist = !TF32 && p.ctas > 0;
  // Query tile of this CTA's item g, or -1; *plane = its (batch, head) plane.
  auto item_qt = [&](int g, int *plane) -> int {
    if (!persist) {
      *plane = bh;
      return g == 0 ? (CAUSAL ? (n_qtiles - 1 - qidx) : qidx) : -1;
    }
    return fwd_item(g, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), p.planes,
                    n_qtiles, p.group_heads, p.block_items, plane);
  };
  // Key tiles of query tile t: [kt0, kt0 + n_kt) (top-left causal: keys <=
  // its last row; in split mode chunk `split` of them).
  auto item_nall = [&](int t) { return CAUSAL ? min(t + 1, n_ktiles) : n_ktiles; };
  int bh0;  // plane of item 0
  const int qt = item_qt(0, &bh0);
  if (qt < 0) return;  // no item for this CTA (a persistent grid larger than the work)
  const int q0 = qt * BM;
  // Head dim of the tensors in memory: D, or less when the kernel runs a
  // narrower head dim zero-padded to D (the TMA maps zero-fill the missing
  // columns on load and clip them on store; plain loads and stores below
  // stop at dio).
  const int dio = p.d_io > 0 ? p.d_io : D;
  // fp32 path with staged operands: K arrives rounded to tf32 and V as a
  // K-major tf32 V^T, so neither is converted here.
  const bool staged = TF32 && (S16 || p.kv_staged != 0);
  if (Nk == 0) {
    // A sequence without keys: the softmax over an empty set gives O = 0 and
    // LSE = log 0 = -inf (variable-length batches only).
    if (threadIdx.x < BM) {
      const int row = q0 + static_cast<int>(threadIdx.x);
      if (row < Nq) {
        const long long gr = q_row0 + row;
        const long long off = hc * p.q_head_stride + gr * p.q_row_stride;
        uint8_t *orow = static_cast<uint8_t *>(p.o) + off * C::ESZ;
        if (FA_IN(p.status, off, dio, p.q_elems))
          for (int x = 0; x < dio * C::ESZ; x += 16)
            *reinterpret_cast<uint4 *>(orow + x) = make_uint4(0, 0, 0, 0);
        const long long li = hc * p.lse_head_stride + gr;
        if (FA_IN(p.status, li, 1, p.lse_elems)) p.lse[li] = -INFINITY;
      }
    }
    return;
  }
  // Key tiles this query tile needs (top-left causal: keys <= last row).
  const int n_all = CAUSAL ? min(qt + 1, n_ktiles) : n_ktiles;
  // This CTA's key tiles: [kt0, kt0 + n_kt), chunk `split` of n_all.
  const int kt0 = static_cast<int>(static_cast<long long>(split) * n_all / nsp);
  const int n_kt = static_cast<int>(static_cast<long long>(split + 1) * n_all / nsp) - kt0;
  if (n_kt == 0) return;  // empty chunk (split mode only); the combine step skips it

  if (threadIdx.x == 0) {
    // Q: written to TMEM by the 128 softmax threads, or one TMA transaction
    mbar_init(bQ, C::QTMEM ? 128 : 1);
#pragma unroll
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(bKfull + 8 * s, 1);
      mbar_init(bKempty + 8 * s, 1);
    }
#pragma unroll
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(bVfull + 8 * s, 1);
      // fp32 path: the softmax warps release a V stage once they transposed it
      mbar_init(bVempty + 8 * s, (TF32 && !p.kv_staged) ? 128 : 1);
    }
#pragma unroll
    for (int s = 0; s < C::KST; ++s) mbar_init(bKready + 8 * s, 128);
#pragma unroll
    for (int b = 0; b < C::NS; ++b) {
      mbar_init(bSfull + 8 * b, 1);
      mbar_init(bPfull + 8 * b, 128);
      mbar_init(bOdone + 8 * b, 1);
    }
    mbar_init(bFin, 1);
    mbar_init(bFin2, 1);
    mbar_init(bQempty, 1);
    mbar_init(bOfree, 128);
#pragma unroll
    for (int g = 0; g < kItemRing; ++g) mbar_init(bOstaged + 8 * g, 128);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 4 && lane == 0) {
    if constexpr (!C::QTMEM) tma_prefetch_desc(&tm_q);
    if (staged) tma_prefetch_desc(&tm_klo);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // Launched with programmatic stream serialization, the set-up above
  // overlaps the previous kernel's tail; its outputs may be this kernel's
  // inputs, so no global memory is touched before this point.
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  WaitCtl w{abort_flag, p.status, p.wait_limit_ns, 0u};

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    w.role = kStatusProducer;
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_last();
      int nk = 0, nv = 0, nq = 0;  // loads issued (K and V ring positions, Q tiles)
      bool ok = true;
      // Several query tiles per CTA: the epilogue of every item but the last
      // stages O in the V stage of the item's last tile (free once its P V
      // completed).  This thread stores it with TMA, and refills that stage
      // only after the store has read it.
      int last_v[kItemRing];     // V ring position of item g's last tile, at g % kItemRing
      int n_items = 0, pend = 0;  // items loaded; next item whose O is stored here
      auto store_o = [&](int gi) -> bool {
        if (!bounded_wait(bOstaged + 8 * (gi % kItemRing), (gi / kItemRing) & 1, w))
          return false;
        const uint32_t src = sV + (last_v[gi % kItemRing] % C::VST) * C::TILE_BYTES;
        int sp;
        const int sq = item_qt(gi, &sp);
#pragma unroll
        for (int c = 0; c < C::NCH; ++c)
          if (c * C::CH_ELEMS < dio)  // a chunk wholly past the row is not stored
            tma_store_3d(&tm_o, src + c * C::CHUNK_BYTES, c * C::CH_ELEMS, sq * BM, sp);
        tma_store_commit();
        tma_store_wait_read_all();
        return true;
      };
      for (int g = 0; ok; ++g) {
        int gp;  // the item's plane
        const int tq = item_qt(g, &gp);
        if (tq < 0) break;
        const int hcg = persist ? gp : hc;
        const int kt0_g = persist ? 0 : kt0;
        const int n_kt_g = persist ? item_nall(tq) : n_kt;
        if constexpr (!C::QTMEM) {
          // The Q buffer is free once the previous item's last S has read it.
          if (g > 0 && !(ok = bounded_wait(bQempty, (g - 1) & 1, w))) break;
          mbar_arrive_expect_tx(bQ, C::TILE_BYTES);
#pragma unroll
          for (int c = 0; c < C::NCH; ++c)
            tma_load_3d(sQ + c * C::CHUNK_BYTES, &tm_q, bQ, c * C::CH_ELEMS, q_row0 + tq * BM, hcg,
                        l2_policy_evict_first());
          ++nq;
        }
        // Load order = consumption order: S runs NS - 1 tiles ahead of P V, so
        // K_{j+NS-1} is loaded just before V_j (K0, K1, K2, V0, K3, V1, ... for
        // NS = 3).
        constexpr int kAhead = C::NS - 1;
        for (int j = -kAhead; ok && j < n_kt_g; ++j) {
          const int jk = j + kAhead;  // next K tile
          if (jk < n_kt_g) {
            const int s = nk % C::KST, r = nk / C::KST;
            if (r > 0) ok = bounded_wait(bKempty + 8 * s, (r - 1) & 1, w);
            if (!ok) break;
            // staged fp32: K_hi, and K_lo into the V stage of the same index
            // (S16: bf16 tiles, half the bytes)
            mbar_arrive_expect_tx(bKfull + 8 * s,
                                  staged ? 2 * C::K_TILE_BYTES : C::K_TILE_BYTES);
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_load_3d(sK + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_k, bKfull + 8 * s,
                          c * C::K_CH_ELEMS, k_row0 + (kt0_g + jk) * BN, hcg, pol_kv);
            if (staged) {
#pragma unroll
              for (int c = 0; c < C::KCH; ++c)
                tma_load_3d(sV + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_klo, bKfull + 8 * s,
                            c * C::K_CH_ELEMS, k_row0 + (kt0_g + jk) * BN, hcg, pol_kv);
            }
            ++nk;
          }
          if (j >= 0) {
            if (p.skip_v_load && g == 0 && j == 0) {  // test hook: starve the MMA issuer
              atomicOr(p.status, kStatusInjected);
              ok = false;
              break;
            }
            const int s = nv % C::VST, r = nv / C::VST;
            if (pend < g && last_v[pend % kItemRing] == nv - C::VST) {
              if (!(ok = store_o(pend))) break;  // this stage holds item pend's O
              ++pend;
            }
            if (r > 0) ok = bounded_wait(bVempty + 8 * s, (r - 1) & 1, w);
            if (!ok) break;
            mbar_arrive_expect_tx(bVfull + 8 * s, C::TILE_BYTES);
            if (staged) {
              // V^T prepared by the staging kernel: D rows x 32 keys per chunk,
              // straight into the K-major V^T buffer the P V product reads.
#pragma unroll
              for (int c = 0; c < BN / 32; ++c)
                tma_load_3d(sVT + s * C::TILE_BYTES + c * C::VT_CHUNK_BYTES, &tm_v,
                            bVfull + 8 * s, (kt0_g + j) * BN + 32 * c, 0, hcg, pol_kv);
            } else {
#pragma unroll
              for (int c = 0; c < C::NCH; ++c)
                tma_load_3d(sV + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_v, bVfull + 8 * s,
                            c * C::CH_ELEMS, k_row0 + (kt0_g + j) * BN, hcg, pol_kv);
            }
            ++nv;
          }
        }
        if (ok) last_v[g % kItemRing] = nv - 1;
        n_items = g + 1;
      }
      // O of the items before the last whose V stage was not refilled.
      for (; ok && pend < n_items - 1; ++pend) ok = store_o(pend);
      // Drain: no TMA write may still be in flight when the CTA exits.
      if (nq > 0) bounded_wait(bQ, (nq - 1) & 1, w, false);
      for (int s = 0; s < C::KST; ++s) {
        const int cnt = (nk > s) ? (nk - 1 - s) / C::KST + 1 : 0;
        if (cnt > 0) bounded_wait(bKfull + 8 * s, (cnt - 1) & 1, w, false);
      }
      for (int s = 0; s < C::VST; ++s) {
        const int cnt = (nv > s) ? (nv - 1 - s) / C::VST + 1 : 0;
        if (cnt > 0) bounded_wait(bVfull + 8 * s, (cnt - 1) & 1, w, false);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------ UMMA issuer: S = Q K^T
    // Issues S_j = Q K_j^T into score buffer j % NS.  That buffer last held
    // P_{j-NS} (written over S_{j-NS}), read by P_{j-NS} V_{j-NS} from the
    // other issuer warp, so S_j waits for that P V to complete.
    w.role = kStatusMma;
    if (lane == 0) {
      constexpr uint32_t kFmt = TF32 ? 2u : (HALF ? 0u : 1u);  // tf32 / f16 / bf16
      constexpr uint32_t kIdescQK = make_idesc(kFmt, BM, BN, 0u, 0u);  // K is K-major
      // A negative scale is applied as S = (-Q) K^T (the descriptor's negate-A
      // bit) with |scale|, so the softmax only ever sees a positive scale.
      const uint32_t idesc_qk = kIdescQK | (p.scale_neg ? (1u << 13) : 0u);
      // S16: the split products in bf16 (kind::f16, format 1)
      const uint32_t idesc_qk16 = make_idesc(1u, BM, BN, 0u, 0u) | (p.scale_neg ? (1u << 13) : 0u);
      bool ok = true;
      int b = 0, bph = 0;   // score buffer of the next S and the parity of its use
      int s = 0, sph = 0;   // K stage of the next S and its parity
      int ns = 0;           // S products issued (all items)
      for (int g = 0; ok; ++g) {
      int gp;
      const int tq = item_qt(g, &gp);
      if (tq < 0) break;
      const int n_kt_g = persist ? item_nall(tq) : n_kt;
      // Q of item g in place (TMEM or shared memory).
      if (!(ok = bounded_wait(bQ, g & 1, w))) break;
      tc_fence_after();
      for (int j = 0; ok && j < n_kt_g; ++j, ++ns) {
        if (ns >= C::NS && !(ok = bounded_wait(bOdone + 8 * b, bph ^ 1, w))) break;
        // fp32 path: K_j must first be rounded to tf32 by the softmax warps
        if (!(ok = bounded_wait(((TF32 && !staged) ? bKready : bKfull) + 8 * s, sph, w))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * 128;
        const uint32_t kb = sK + s * C::TILE_BYTES;
        // fp32: K_lo of this tile (see TcCfg::NKLO)
        const uint32_t klo = staged ? sV + s * C::TILE_BYTES : C::NKLO ? sKLO : sVT;
        if constexpr (S16) {
          // Q_hi K_hi + Q_hi K_lo + Q_lo K_hi in bf16: 32 bytes (16 values) of
          // K per UMMA, 8 TMEM columns of Q.
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
            const uint64_t khi = sdesc_sw128(kb + off, 16, 1024);
            umma_ts<false>(d_tmem, tmem + C::COL_Q + kk * 8, khi, idesc_qk16, kk > 0 ? 1u : 0u);
            umma_ts<false>(d_tmem, tmem + C::COL_Q + kk * 8, sdesc_sw128(klo + off, 16, 1024),
                           idesc_qk16, 1u);
            umma_ts<false>(d_tmem, tmem + C::COL_QLO + kk * 8, khi, idesc_qk16, 1u);
          }
        } else
#pragma unroll
        for (int kk = 0; kk < D / C::UK; ++kk) {
          // 32 bytes of K per UMMA (4 steps per 128-byte swizzle chunk); the
          // matching Q slice is 8 TMEM columns or the same 32 bytes of Q.
          const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          if constexpr (TF32) {
            // Q_hi K_hi + Q_hi K_lo + Q_lo K_hi
            const uint64_t khi = sdesc_sw128(kb + off, 16, 1024);
            umma_ts<TF32>(d_tmem, tmem + C::COL_Q + kk * 8, khi, idesc_qk, kk > 0 ? 1u : 0u);
            umma_ts<TF32>(d_tmem, tmem + C::COL_Q + kk * 8, sdesc_sw128(klo + off, 16, 1024),
                          idesc_qk, 1u);
            umma_ts<TF32>(d_tmem, tmem + C::COL_QLO + kk * 8, khi, idesc_qk, 1u);
          } else if constexpr (C::QTMEM) {
            umma_ts<TF32>(d_tmem, tmem + C::COL_Q + kk * 8, sdesc_sw128(kb + off, 16, 1024),
                          idesc_qk, kk > 0 ? 1u : 0u);
          } else {
            umma_ss<TF32>(d_tmem, sdesc_sw128(sQ + off, 16, 1024),
                          sdesc_sw128(kb + off, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
          }
        }
        tc_commit(bKempty + 8 * s);
        tc_commit(bSfull + 8 * b);
        if (++b == C::NS) { b = 0; bph ^= 1; }
        if (++s == C::KST) { s = 0; sph ^= 1; }
      }
      // Q of item g is free once its S products complete.
      if (ok) tc_commit(bQempty);
      }
      // Every UMMA issued above must be complete before TMEM is freed.
      tc_commit(bFin);
      bounded_wait(bFin, 0, w, false);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------ UMMA issuer: O += P V
    // A second issuing warp, so that neither product's waits and commits
    // leave the tensor pipe idle while the other has work ready.
    w.role = kStatusMma;
    if (lane == 0) {
      constexpr uint32_t kFmt = TF32 ? 2u : (HALF ? 0u : 1u);  // tf32 / f16 / bf16
      // bf16: V is an MN-major B operand.  fp32: V^T is a K-major B operand.
      constexpr uint32_t kIdescPV = make_idesc(kFmt, BM, D, 0u, TF32 ? 0u : 1u);
      bool ok = true;
      int b = 0, bph = 0;   // score buffer of the next P V and the parity of its use
      int s = 0, sph = 0;   // V stage of the next P V and its parity
      for (int g = 0; ok; ++g) {
      int gp;
      const int tq = item_qt(g, &gp);
      if (tq < 0) break;
      const int n_kt_g = persist ? item_nall(tq) : n_kt;
      // O of the previous item has been read out by the epilogue.
      if (g > 0) {
        if (!(ok = bounded_wait(bOfree, (g - 1) & 1, w))) break;
        tc_fence_after();
      }
      for (int j = 0; ok && j < n_kt_g; ++j) {
        // P_j ready (fp32 path: also V_j^T written), V_j (or V_j^T) loaded.
        if (!(ok = bounded_wait(bPfull + 8 * b, bph, w))) break;
        if (!TF32 || staged) {
          if (!(ok = bounded_wait(bVfull + 8 * s, sph, w))) break;
        }
        tc_fence_after();
        const uint32_t a_tmem = tmem + b * 128;
#pragma unroll
        for (int kk = 0; kk < BN / C::UK; ++kk) {
          // UK keys per UMMA; the P slice is 8 TMEM columns.
          uint64_t bdesc;
          if constexpr (TF32) {
            // V^T: D rows of 128 keys, K-major, 32 keys per 128-byte chunk
            const uint32_t vt = sVT + (j % C::NVT) * C::TILE_BYTES;
            bdesc = sdesc_sw128(vt + (kk >> 2) * C::VT_CHUNK_BYTES + (kk & 3) * 32, 16, 1024);
          } else {
            // V: UK key rows of 128 bytes per step, MN-major
            bdesc = sdesc_sw128(sV + s * C::TILE_BYTES + kk * C::UK * 128, C::CHUNK_BYTES, 1024);
          }
          umma_ts<TF32>(tmem + C::COL_O, a_tmem + kk * 8, bdesc, kIdescPV,
                        (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (!TF32 || staged) tc_commit(bVempty + 8 * s);
        tc_commit(bOdone + 8 * b);
        if (++b == C::NS) { b = 0; bph ^= 1; }
        if (++s == C::VST) { s = 0; sph ^= 1; }
      }
      }
      tc_commit(bFin2);
      bounded_wait(bFin2, 0, w, false);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax + epilogue
    w.role = kStatusSoftmax;
    const int r = threadIdx.x;  // TMEM lane == row within the tile
    int row = q0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t o_tm = tmem + lane_off + C::COL_O;
    const float sl2 = p.scale_log2;
    int row_lim = CAUSAL ? min(row + 1, Nk) : Nk;  // keys [0, row_lim)
    float m_used = -INFINITY;  // exponent offset, log2 units of the scaled score
    float l = 0.f;
    bool ok = true;

    // fp32 path: split this thread's row r of K tile t (stage t % KST) into
    // K_hi = tf32(k), written in place, and K_lo = tf32(k - K_hi), written at
    // the same place of the K_lo buffer; then release both to the UMMA
    // issuer.  Row r occupies NCH * 8 16-byte units of the 128-byte-swizzled
    // tile.  The K_lo buffer must be free: S_{t-1} has completed (D = 64), or
    // P_{t-1} V_{t-1} has, whose V^T it shares (D = 128).
    auto split_k_row = [&](int t) -> bool {
      const int s = t % C::KST;
      if (!__all_sync(kFull, bounded_wait(bKfull + 8 * s, (t / C::KST) & 1, w))) return false;
      uint8_t *kt = smem + C::OFF_K + s * C::TILE_BYTES;
      uint8_t *kl = smem + (C::NKLO ? C::OFF_KLO : C::OFF_VT);
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int off = ch * C::CHUNK_BYTES + r * 128 + ((u ^ (r & 7)) << 4);
          uint4 *ptr = reinterpret_cast<uint4 *>(kt + off);
          const uint4 val = *ptr;
          const uint32_t e[4] = {val.x, val.y, val.z, val.w};
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            hi[i] = to_tf32(__uint_as_float(e[i]));
            lo[i] = to_tf32(__uint_as_float(e[i]) - __uint_as_float(hi[i]));
          }
          *ptr = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4 *>(kl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bKready + 8 * s);
      return true;
    };
    // fp32 path: transpose key row r of V tile j into column r of V^T
    // (tf32-rounded), then release the fp32 stage to the producer.  For a fixed
    // d the 32 threads of a warp write 32 consecutive keys of one 128-byte row
    // of V^T: one word each, no bank conflicts.
    auto transpose_v_row = [&](int j) -> bool {
      const int s = j % C::VST;
      if (!__all_sync(kFull, bounded_wait(bVfull + 8 * s, (j / C::VST) & 1, w))) return false;
      const uint8_t *vt32 = smem + C::OFF_V + s * C::TILE_BYTES;
      uint8_t *vtT = smem + C::OFF_VT + (j % C::NVT) * C::TILE_BYTES;
      const int key_chunk = r >> 5, key_unit = (r & 31) >> 2, key_word = r & 3;
#pragma unroll
      for (int ch = 0; ch < C::NCH; ++ch) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 val = *reinterpret_cast<const uint4 *>(
              vt32 + ch * C::CHUNK_BYTES + r * 128 + ((u ^ (r & 7)) << 4));
          const uint32_t e[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int dd = ch * C::CH_ELEMS + 4 * u + i;  // head-dim index
            *reinterpret_cast<uint32_t *>(vtT + key_chunk * C::VT_CHUNK_BYTES + dd * 128 +
                                          ((key_unit ^ (dd & 7)) << 4) + key_word * 4) =
                to_tf32(__uint_as_float(e[i]));
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bVempty + 8 * s);
      return true;
    };

    // Q row -> tensor memory (A operand layout: lane = row, 32-bit column c
    // holds bf16 elements 2c, 2c+1, or one tf32 element).  Rows past Nq are 0.
    // (Otherwise the producer loads Q into shared memory with TMA.)
    auto stage_q = [&](int tq, int plane) {
      const int qrow = tq * BM + r;
      const long long qoff =
          plane * p.q_head_stride + (q_row0 + (qrow < Nq ? qrow : 0)) * p.q_row_stride;
      const bool in = qrow < Nq && FA_IN(p.status, qoff, dio, p.q_elems);
      const uint4 *src = reinterpret_cast<const uint4 *>(
          static_cast<const uint8_t *>(p.q) + qoff * C::ESZ);
      if constexpr (S16) {
        // Q_hi = bf16(q) and Q_lo = bf16(q - Q_hi), two per column: 64
        // fp32 values of the row per block of 32 columns.
#pragma unroll
        for (int blk = 0; blk < C::Q_COLS / 32; ++blk) {
          uint32_t wh[32], wl[32];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const bool ld = in && (blk * 16 + u) * 16 < dio * C::ESZ;
            const uint4 val = ld ? __ldg(src + blk * 16 + u) : make_uint4(0u, 0u, 0u, 0u);
            const float x[4] = {__uint_as_float(val.x), __uint_as_float(val.y),
                                __uint_as_float(val.z), __uint_as_float(val.w)};
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
              const uint32_t h = pack_bf16x2(x[e], x[e + 1]);
              wh[2 * u + e / 2] = h;
              wl[2 * u + e / 2] = pack_bf16x2(x[e] - __uint_as_float(h << 16),
                                              x[e + 1] - __uint_as_float(h & 0xffff0000u));
            }
          }
          tmem_st32(tmem + lane_off + C::COL_Q + blk * 32, wh);
          tmem_st32(tmem + lane_off + C::COL_QLO + blk * 32, wl);
        }
      } else
#pragma unroll
      for (int blk = 0; blk < C::Q_COLS / 32; ++blk) {
        uint32_t wq[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const bool ld = in && (blk * 8 + u) * 16 < dio * C::ESZ;
          uint4 val = ld ? __ldg(src + blk * 8 + u) : make_uint4(0u, 0u, 0u, 0u);
          wq[4 * u + 0] = val.x;
          wq[4 * u + 1] = val.y;
          wq[4 * u + 2] = val.z;
          wq[4 * u + 3] = val.w;
        }
        if constexpr (TF32) {
          // Q_hi = tf32(q) and Q_lo = tf32(q - Q_hi), the A operands of the
          // split S product
          uint32_t wl[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float x = __uint_as_float(wq[i]);
            wq[i] = to_tf32(x);
            wl[i] = to_tf32(x - __uint_as_float(wq[i]));
          }
          tmem_st32(tmem + lane_off + C::COL_QLO + blk * 32, wl);
        }
        tmem_st32(tmem + lane_off + C::COL_Q + blk * 32, wq);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bQ);
    };
    if constexpr (C::QTMEM) stage_q(qt, persist ? bh0 : hc);
    if (TF32 && !staged) ok = split_k_row(0);

    int buf = 0, bph = 0;            // score buffer of tile j and the parity of its use
    int pbuf = C::NS - 1, pbph = 1;  // the same for tile j - 1
    int tiles_done = 0;              // key tiles of all items so far (= V ring position)
    for (int g = 0;; ++g) {
    int gp;  // the item's plane
    const int tq = item_qt(g, &gp);
    if (tq < 0) break;
    const int n_kt_g = persist ? item_nall(tq) : n_kt;
    row = tq * BM + r;
    row_lim = CAUSAL ? min(row + 1, Nk) : Nk;
    m_used = -INFINITY;
    l = 0.f;
    for (int j = 0; ok && j < n_kt_g; ++j) {
      ok = __all_sync(kFull, bounded_wait(bSfull + 8 * buf, bph, w));
      if (!ok) break;
      tc_fence_after();
      if (TF32 && !staged && C::NKLO && j + 1 < n_kt_g) {
        // S_j has completed, so its K_lo buffer is free: the next K tile is
        // split before this tile's softmax so that S_{j+1} overlaps it
        if (!(ok = split_k_row(j + 1))) break;
      }
      const uint32_t s_tm = tmem + lane_off + buf * 128;
      uint32_t sr[4][32];
      tmem_ld32(s_tm + 0, sr[0]);
      tmem_ld32(s_tm + 32, sr[1]);
      tmem_ld32(s_tm + 64, sr[2]);
      tmem_ld32(s_tm + 96, sr[3]);
      tmem_ld_wait();
      reg_fence32(sr[0]);
      reg_fence32(sr[1]);
      reg_fence32(sr[2]);
      reg_fence32(sr[3]);
      auto S = [&](int c) -> float { return __uint_as_float(sr[c >> 5][c & 31]); };

      const int lim = row_lim - (kt0 + j) * BN;  // valid columns c < lim
      // Masked tiles (causal diagonal, ragged key tail; at most two per CTA)
      // set the excluded scores to -inf, so one code path serves every tile:
      // they drop out of the max, and exp2(-inf) = 0 (the scale is > 0 here).
      if (__any_sync(kFull, lim < BN)) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c >= lim) sr[c >> 5][c & 31] = 0xff800000u;  // -inf
      }
      // After the first tile of an item, P is computed with the current
      // offset straight away, and the row max is taken only when the row sum
      // exceeds 2^kRescaleThreshold.  Any P above that bound (the max grew by
      // more than the threshold, the one case where the offset must move)
      // makes the sum exceed it, so the offsets, and with them P and l, are
      // those of taking the max first on every tile.  When that max shows no
      // row of the warp has to move, the first pass stands; otherwise the
      // rows that must move rescale O and the warp recomputes P.  The first
      // tile of an item takes its max first.
      constexpr float kSumLimit = 256.f;  // 2^kRescaleThreshold
      bool with_max = (j == 0);
      float tsum = 0.f;
      for (;;) {
        if (with_max) {
          // Row max: eight independent chains of three-input max keep the
          // dependency depth at 8 for the 128 columns.
          float mx;
          {
            float part[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) part[i] = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; c += 2)
              part[(c >> 1) & 7] = max3f(part[(c >> 1) & 7], S(c), S(c + 1));
            mx = max3f(max3f(part[0], part[1], part[2]), max3f(part[3], part[4], part[5]),
                       fmaxf(part[6], part[7]));
          }
          const float m_new = fmaxf(m_used, mx * sl2);
          if (j == 0) {
            m_used = m_new;
          } else {
            // P_j may overwrite P_{j-NS} without waiting: S_j was only
            // issued after P_{j-NS} V_{j-NS} had completed.  Only a rescale
            // of O has to wait, for P_{j-1} V_{j-1} (the last UMMA into O
            // before P_j V_j); the done-barriers are per score buffer, and the
            // previous use of tile j-1's buffer (P_{j-1-NS} V_{j-1-NS})
            // completed before S_{j-1} was issued, so a skipped wait never
            // makes a later one ambiguous.
            const bool need = (m_new - m_used) > kRescaleThreshold;
            if (!__any_sync(kFull, need)) break;  // P and tsum of the first pass stand
            ok = __all_sync(kFull, bounded_wait(bOdone + 8 * pbuf, pbph, w));
            if (!ok) break;
            tc_fence_after();
            const float alpha = need ? ex2_approx(m_used - m_new) : 1.f;
            const uint64_t a2 = pk2(alpha, alpha);
#pragma unroll
            for (int c = 0; c < D; c += 32) {
              uint32_t o[32];
              tmem_ld32(o_tm + c, o);
              tmem_ld_wait();
              reg_fence32(o);
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                float lo, hi;
                upk2(fmul2(pk2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2), lo, hi);
                o[i] = __float_as_uint(lo);
                o[i + 1] = __float_as_uint(hi);
              }
              tmem_st32(o_tm + c, o);
            }
            tmem_st_wait();
            if (need) {
              l *= alpha;
              m_used = m_new;
            }
          }
        }
        // P = exp2(s * scale*log2e - m_used), written over S in TMEM; pairs of
        // columns go through packed f32x2 arithmetic.
        const uint64_t sl2_2 = pk2(sl2, sl2);
        const uint64_t nm_2 = pk2(-m_used, -m_used);
        uint64_t acc[2] = {0ull, 0ull};  // packed partial row sums (+0.0f bits)
        {
          constexpr int kBlk = TF32 ? 16 : 32;  // column pairs per TMEM store
#pragma unroll
          for (int blk = 0; blk < 64 / kBlk; ++blk) {
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < kBlk; ++i) {
              const int c0 = 2 * (blk * kBlk + i);
              const uint64_t x2 = ffma2(pk2(S(c0), S(c0 + 1)), sl2_2, nm_2);
              float x0, x1;
              upk2(x2, x0, x1);
              const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              acc[i & 1] = fadd2(acc[i & 1], pk2(p0, p1));
              if constexpr (TF32) {
                pk[2 * i] = to_tf32(p0);
                pk[2 * i + 1] = to_tf32(p1);
              } else {
                pk[i] = HALF ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
              }
            }
            tmem_st32(s_tm + blk * 32, pk);
          }
        }
        {
          float a0, a1, b0, b1;
          upk2(acc[0], a0, a1);
          upk2(acc[1], b0, b1);
          tsum = (a0 + a1) + (b0 + b1);
        }
        if (with_max || __all_sync(kFull, tsum <= kSumLimit)) break;
        with_max = true;
        tmem_st_wait();  // the second pass rewrites the same P columns
      }
      if (!ok) break;
      l += tsum;
      if (TF32 && !staged) {
        // V^T buffer j % NVT was last read by P_{j-NVT} V_{j-NVT}: with two
        // buffers that completed before S_j was issued (NS = 2); the one
        // buffer of D = 128 held K_lo_j, free since S_j completed, and
        // P_{j-1} V_{j-1} completed before S_j was issued (NS = 1).
        if (!(ok = transpose_v_row(j))) break;
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bPfull + 8 * buf);
      if (TF32 && !staged && !C::NKLO && j + 1 < n_kt_g) {
        // D = 128: K_lo_{j+1} goes into the V^T buffer once P_j V_j has read
        // it (and S_{j+1} could not start before that anyway: one score
        // buffer)
        ok = __all_sync(kFull, bounded_wait(bOdone + 8 * buf, bph, w));
        if (!ok) break;
        if (!(ok = split_k_row(j + 1))) break;
      }
      ++tiles_done;
      pbuf = buf;
      pbph = bph;
      if (++buf == C::NS) { buf = 0; bph ^= 1; }
    }

    // Q-in-TMEM: the next item's Q rows go in once this item's S products
    // have read the current ones, so its first S overlaps this epilogue.
    int np;  // plane of the next item
    const int tn = item_qt(g + 1, &np);
    if constexpr (C::QTMEM) {
      if (ok && tn >= 0) {
        ok = __all_sync(kFull, bounded_wait(bQempty, g & 1, w));
        if (ok) stage_q(tn, np);
      }
    }

    // ------------------------------------------------ epilogue
    const bool last_item = tn < 0;
    // The last P V; its commit also covers every earlier UMMA.
    if (ok)
      ok = __all_sync(kFull, bounded_wait(bOdone + 8 * pbuf, pbph, w));
    if (nsp > 1) {
      // Split mode: this chunk's O / l (fp32) and LSE go to the workspace with
      // plain vector stores; the combine kernel merges the chunks.
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        const size_t prow = (static_cast<size_t>(split) * gridDim.z * p.H + bh) * p.Nq + row;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(o_tm + c, o);
          tmem_ld_wait();
          reg_fence32(o);
          if (row < Nq && c < dio &&
              FA_IN(p.status, prow * dio + c, 32, static_cast<long long>(nsp) * p.lse_elems * dio)) {
            float4 *dst = reinterpret_cast<float4 *>(p.ws_o + prow * dio + c);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              dst[u] = make_float4(__uint_as_float(o[4 * u + 0]) * inv_l,
                                   __uint_as_float(o[4 * u + 1]) * inv_l,
                                   __uint_as_float(o[4 * u + 2]) * inv_l,
                                   __uint_as_float(o[4 * u + 3]) * inv_l);
          }
        }
        if (row < Nq && FA_IN(p.status, prow, 1, static_cast<long long>(nsp) * p.lse_elems))
          p.ws_lse[prow] = m_used * kLn2 + logf(l);
      }
    } else if (p.cu_q != nullptr) {
      // Variable-length batches: the rows after this sequence belong to the
      // next one, so O is written row by row from registers (no TMA store).
      if (ok) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        const long long gr = q_row0 + row;
        const long long off = hc * p.q_head_stride + gr * p.q_row_stride;
        uint8_t *orow = static_cast<uint8_t *>(p.o) + off * C::ESZ;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(o_tm + c, o);
          tmem_ld_wait();
          reg_fence32(o);
          if (row < Nq && c < dio && FA_IN(p.status, off + c, 32, p.q_elems)) {
            if constexpr (TF32) {
#pragma unroll
              for (int u = 0; u < 8; ++u)
                reinterpret_cast<float4 *>(orow + c * 4)[u] =
                    make_float4(__uint_as_float(o[4 * u + 0]) * inv_l,
                                __uint_as_float(o[4 * u + 1]) * inv_l,
                                __uint_as_float(o[4 * u + 2]) * inv_l,
                                __uint_as_float(o[4 * u + 3]) * inv_l);
            } else {
              auto pack16 = [](float lo, float hi) {
                return HALF ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
              };
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                uint4 val;
                val.x = pack16(__uint_as_float(o[8 * u + 0]) * inv_l, __uint_as_float(o[8 * u + 1]) * inv_l);
                val.y = pack16(__uint_as_float(o[8 * u + 2]) * inv_l, __uint_as_float(o[8 * u + 3]) * inv_l);
                val.z = pack16(__uint_as_float(o[8 * u + 4]) * inv_l, __uint_as_float(o[8 * u + 5]) * inv_l);
                val.w = pack16(__uint_as_float(o[8 * u + 6]) * inv_l, __uint_as_float(o[8 * u + 7]) * inv_l);
                reinterpret_cast<uint4 *>(orow + c * 2)[u] = val;
              }
            }
          }
        }
        const long long li = hc * p.lse_head_stride + gr;
        if (row < Nq && FA_IN(p.status, li, 1, p.lse_elems)) p.lse[li] = m_used * kLn2 + logf(l);
      }
    } else if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      // Staging for the TMA store.  The last item: K stage 0 (every S_j is
      // complete, so no UMMA reads K any more and the producer has no K load
      // outstanding).  An earlier item: the V stage of its last tile, whose
      // P V has completed; the producer stores it and refills the stage
      // after that.
      uint8_t *stage = last_item ? smem + C::OFF_K
                                 : smem + C::OFF_V + ((tiles_done - 1) % C::VST) * C::TILE_BYTES;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(o_tm + c, o);
        tmem_ld_wait();
        reg_fence32(o);
        if constexpr (TF32) {
          // 32 fp32 = 8 units of 16 bytes = one full chunk (chunk c/32).
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint4 val;
            val.x = __float_as_uint(__uint_as_float(o[4 * u + 0]) * inv_l);
            val.y = __float_as_uint(__uint_as_float(o[4 * u + 1]) * inv_l);
            val.z = __float_as_uint(__uint_as_float(o[4 * u + 2]) * inv_l);
            val.w = __float_as_uint(__uint_as_float(o[4 * u + 3]) * inv_l);
            const int ch = c / 32;
            *reinterpret_cast<uint4 *>(stage + ch * C::CHUNK_BYTES + r * 128 +
                                       ((u ^ (r & 7)) << 4)) = val;
          }
        } else {
          // 32 16-bit values = 4 units of 16 bytes; global unit index c/8 + u.
          auto pack16 = [](float lo, float hi) {
            return HALF ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
          };
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 val;
            val.x = pack16(__uint_as_float(o[8 * u + 0]) * inv_l,
                                __uint_as_float(o[8 * u + 1]) * inv_l);
            val.y = pack16(__uint_as_float(o[8 * u + 2]) * inv_l,
                                __uint_as_float(o[8 * u + 3]) * inv_l);
            val.z = pack16(__uint_as_float(o[8 * u + 4]) * inv_l,
                                __uint_as_float(o[8 * u + 5]) * inv_l);
            val.w = pack16(__uint_as_float(o[8 * u + 6]) * inv_l,
                                __uint_as_float(o[8 * u + 7]) * inv_l);
            const int gu = c / 8 + u;
            const int ch = gu >> 3, uu = gu & 7;
            *reinterpret_cast<uint4 *>(stage + ch * C::CHUNK_BYTES + r * 128 +
                                       ((uu ^ (r & 7)) << 4)) = val;
          }
        }
      }
      const long long li = static_cast<long long>(gp) * Nq + row;
      if (row < Nq && FA_IN(p.status, li, 1, p.lse_elems)) p.lse[li] = m_used * kLn2 + logf(l);
      if (!last_item) {
        fence_proxy_async_smem();
        mbar_arrive(bOstaged + 8 * (g % kItemRing));   // the producer stores this item's O
      }
    }
    // O of this item has been read from tensor memory: the next item's
    // P V may start.
    if (ok && !last_item) {
      tc_fence_before();
      mbar_arrive(bOfree);
    }
    fence_proxy_async_smem();
    // All four warps reach this barrier once per item whatever their own
    // waits gave; the OR over it hands them one decision to go on or stop.
    const bool stop = named_bar_or(1, 128, !ok || *abort_flag != 0);
    if (last_item && nsp == 1 && p.cu_q == nullptr && threadIdx.x == 0 && !stop) {
#pragma unroll
      for (int c = 0; c < C::NCH; ++c)
        if (c * C::CH_ELEMS < dio)  // a chunk wholly past the row is not stored
          tma_store_3d(&tm_o, sK + c * C::CHUNK_BYTES, c * C::CH_ELEMS, tq * BM, gp);
      tma_store_commit();
      tma_store_wait_read_all();
    }
    // The same `stop` in all four warps: they leave the item loop together.
    // (Only with several items: with one the check is moot, and as a loop
    // exit it cost the fp32 kernels their last free registers.)
    if (persist && stop) break;
    }  // items
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool TF32, bool HALF = false, bool S16 = false>
cudaError_t launch_tc(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                      const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p, int B,
                      int causal, cudaStream_t stream) {
  using C = TcCfg<D, TF32, S16>;
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
               const CUtensorMap, const TcParams) =
      causal ? fa_tc_fwd_kernel<D, TF32, true, HALF, S16>
             : fa_tc_fwd_kernel<D, TF32, false, HALF, S16>;
  static std::atomic<unsigned long long> attr_done[2];  // per causal flag
  cudaError_t e = smem_attr_once(kern, C::SMEM_BYTES, &attr_done[causal ? 1 : 0]);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  if (p.ctas > 0 && !TF32)
    cfg.gridDim = dim3(static_cast<unsigned>(p.ctas), 1, 1);  // persistent
  else
    cfg.gridDim = dim3(static_cast<unsigned>(p.n_qtiles * p.n_splits), static_cast<unsigned>(p.H),
                       static_cast<unsigned>(B));
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q, k, v, o, klo, p);
}

}  // namespace fa
