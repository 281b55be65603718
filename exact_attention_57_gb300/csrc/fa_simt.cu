// fa_simt.cu — plain fp32 (no tensor cores) exact-attention forward.
//
// The same method as the tensor-core kernels — the forward kernel of
// "flash_attention_2.cu" (leloykun/flash-hyperbolic-attention-minimal):
// scores scaled before the row max, online softmax over key tiles with a
// running max m and sum l, partial output rescaled by exp(m_old - m_new),
// O = O / l and L = m + log(l) at the end — computed with fp32 FMAs.
//
// Differences from that page's kernel, each deliberate:
//   * one CTA per (batch, head, query tile of R rows) instead of one per
//     (batch, head), so the grid does not depend on B*H;
//   * O accumulates in registers and is written once (the page
//     read-modify-writes O in global memory every key tile and therefore
//     needs O zeroed first);
//   * rows past Nq stay in the loop until the end (the page breaks out of the
//     loop before a __syncthreads, a divergent-barrier hazard);
//   * keys past Nk and, when causal, keys after the query are excluded
//     element by element, on every tile, not only within a row's own tile.
//
// Work split.  G neighbouring lanes of a warp share one query row (R =
// 128/(G*KS) rows per 128-thread CTA, KS the key groups below).  For the scores the G lanes split the keys of a
// shared-memory tile (lane g takes keys g, g+G, ...), each holding the whole
// query row in registers.  The tile's row max is combined across the G lanes
// by shuffles; each lane turns its own scores into probabilities, and the
// lanes then hand them round (one shuffle per key) so that each lane
// accumulates P·V for its own output columns (4-column chunks g, g+G, ...).
// The online-softmax state (m, and the partial O) is therefore the same in
// all G lanes and needs no merge at the end beyond summing l.
//   G trades work per FMA against parallelism.  G = 1 (one thread per row,
// every K/V read a broadcast, no shuffles) is the cheapest per FMA but puts
// 128 rows in a CTA; G = 4, 8, 16 spread a smaller problem over 4, 8, 16
// times as many CTAs at the cost of one shuffle per key and the row-max
// shuffles.  The launcher takes the smallest G whose grid still gives every
// SM two CTAs; a grid still short of that also splits each row's keys over
// KS = 2 or 4 warp groups of the CTA, whose states are merged at the end.  Staged rows are padded by 16 B so that the G different key
// rows one access touches fall in different banks.
//   K/V tiles go through a ring of NS shared-memory stages filled by
// cp.async, NS - 1 tiles ahead of the arithmetic.  The dot products (for
// G >= 8) and the P·V sums (for at most two column chunks per lane) are split
// over independent partial sums so that consecutive FMAs do not wait on one
// another.
#include <atomic>
#include <cmath>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kSimtThreads = 128;  // threads per CTA
constexpr int kSimtKeys = 32;      // keys per shared-memory tile
constexpr int kSimtPad = 4;        // floats of padding after each staged row

// Asynchronous global -> shared copies (cp.async); when `valid` is false the
// destination is zero-filled and `src` is not read.
__device__ __forceinline__ void cp_async4(float *dst, const float *src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async16(float *dst, const float *src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>  // wait until at most N committed groups are still in flight
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int DP, int KS>
constexpr int simt_stages() {  // K/V ring depth: 2 to 4 stages within ~108 KB
  constexpr int stage = 2 * KS * kSimtKeys * (DP + kSimtPad) * static_cast<int>(sizeof(float));
  return 110592 / stage > 4 ? 4 : (110592 / stage < 2 ? 2 : 110592 / stage);
}
template <int DP, int KS>
constexpr int simt_smem_bytes() {  // K and V, simt_stages() stages each
  return 2 * simt_stages<DP, KS>() * KS * kSimtKeys * (DP + kSimtPad) *
         static_cast<int>(sizeof(float));
}

// KS: key groups.  The CTA's threads form KS groups of 128/KS (whole warps);
// group k takes key sub-tile k of every stage of KS*32 keys for the same
// rows, and the groups' softmax states are merged at the end.
template <int DP, int G, int KS>  // DP: head dim padded up to 32, 64 or 128
__global__ void __launch_bounds__(kSimtThreads, 1) fa_simt_fwd_kernel(const SimtParams p) {
  constexpr int TPG = kSimtThreads / KS;   // threads per key group
  constexpr int R = TPG / G;               // query rows per CTA
  constexpr int LD = DP + kSimtPad;        // staged row stride (floats)
  constexpr int KPL = kSimtKeys / G;       // scores per lane per sub-tile
  constexpr int CPL = DP / (4 * G);        // 4-column output chunks per lane
  constexpr int SUB = kSimtKeys * LD;      // floats of one staged K (or V) sub-tile
  constexpr int TILE = KS * SUB;           // floats of one stage of K (or V)
  constexpr int NS = simt_stages<DP, KS>();
  constexpr int PVA = CPL <= 2 ? 2 : 1;   // P·V partial sums per output (even/odd keys)
  constexpr int SP = KPL >= 8 ? 1 : 2;    // partial sums per dot product
  static_assert(KPL >= 1 && CPL >= 1 && 32 % G == 0, "G must divide the warp and the tile");
  static_assert(TPG % 32 == 0, "a key group is whole warps");
  static_assert(NS >= 2, "the ring needs two stages");
  extern __shared__ float4 simt_smem[];
  float *const Ks = reinterpret_cast<float *>(simt_smem);  // [NS][KS*kSimtKeys][LD]
  float *const Vs = Ks + NS * TILE;                        // [NS][KS*kSimtKeys][LD]

  const int qt = p.causal ? (p.n_qtiles - 1 - static_cast<int>(blockIdx.x))
                          : static_cast<int>(blockIdx.x);
  const size_t bh = static_cast<size_t>(blockIdx.z) * p.H + blockIdx.y;
  const int d = p.d;
  const int ks = static_cast<int>(threadIdx.x) / TPG;  // key group (warp-uniform)
  const int tig = static_cast<int>(threadIdx.x) % TPG;
  const int g = tig % G;  // lane within the row's group
  const int row = qt * R + tig / G;
  const bool active = row < p.Nq;
  const float *qh = p.q + bh * p.Nq * d;
  const float *kh = p.k + bh * p.Nk * d;
  const float *vh = p.v + bh * p.Nk * d;
  // extents for the debug build's index checks
  const long long planes = static_cast<long long>(p.B) * p.H;
  const long long q_elems = planes * p.Nq * d, kv_elems = planes * p.Nk * d;
  // Launched with programmatic stream serialization: wait for the previous
  // kernel on the stream before the first global access (the debug build's
  // index checks write the status word), then let the next one start
  // launching.
  griddep_wait();
  griddep_launch_dependents();
  const bool q_ok =
      active && FA_IN(p.status, static_cast<long long>(bh * p.Nq + row) * d, d, q_elems);

  float qr[DP];
  if ((d & 3) == 0) {  // 16-byte-aligned rows: four columns a load
    const float4 *q4 = reinterpret_cast<const float4 *>(qh + static_cast<size_t>(row) * d);
#pragma unroll
    for (int x = 0; x < DP; x += 4) {
      const float4 v = (q_ok && x < d) ? q4[x / 4] : make_float4(0.f, 0.f, 0.f, 0.f);
      qr[x] = v.x;
      qr[x + 1] = v.y;
      qr[x + 2] = v.z;
      qr[x + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int x = 0; x < DP; ++x)
      qr[x] = (q_ok && x < d) ? qh[static_cast<size_t>(row) * d + x] : 0.f;
  }

  // keys [0, row_lim) take part for this row; the CTA visits keys up to the
  // largest row_lim among its rows.
  const int row_lim = p.causal ? min(row + 1, p.Nk) : p.Nk;
  const int cta_lim = p.causal ? min(qt * R + R, p.Nk) : p.Nk;
  const int n_tiles = (cta_lim + KS * kSimtKeys - 1) / (KS * kSimtKeys);

  // Stage key tile t (K and V rows k0 .. k0 + KS*32 - 1) into buffer `buf`;
  // columns past d and keys past Nk are zero-filled.
  auto stage = [&](int t, int buf) {
    const int k0 = t * KS * kSimtKeys;
    float *kd = Ks + buf * TILE;
    float *vd = Vs + buf * TILE;
    if ((d & 3) == 0) {  // rows are whole 16-byte chunks
      constexpr int CPR = DP / 4;
      for (int e = static_cast<int>(threadIdx.x); e < KS * kSimtKeys * CPR; e += kSimtThreads) {
        const int c = e / CPR, x = (e % CPR) * 4;
        const int key = k0 + c;
        const bool in = key < p.Nk && x < d &&
                        FA_IN(p.status, static_cast<long long>(bh * p.Nk + key) * d + x, 4,
                              kv_elems);
        const size_t off = in ? static_cast<size_t>(key) * d + x : 0;
        cp_async16(kd + c * LD + x, kh + off, in);
        cp_async16(vd + c * LD + x, vh + off, in);
      }
    } else {
      for (int e = static_cast<int>(threadIdx.x); e < KS * kSimtKeys * DP; e += kSimtThreads) {
        const int c = e / DP, x = e % DP;
        const int key = k0 + c;
        const bool in = key < p.Nk && x < d &&
                        FA_IN(p.status, static_cast<long long>(bh * p.Nk + key) * d + x, 1,
                              kv_elems);
        const size_t off = in ? static_cast<size_t>(key) * d + x : 0;
        cp_async4(kd + c * LD + x, kh + off, in);
        cp_async4(vd + c * LD + x, vh + off, in);
      }
    }
    cp_async_commit();
  };

  float acc[PVA][CPL][4];
#pragma unroll
  for (int a = 0; a < PVA; ++a)
#pragma unroll
    for (int i = 0; i < CPL; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[a][i][u] = 0.f;
  float m = -INFINITY, l = 0.f;  // l: this lane's share of the row sum

  // Tiles 0 .. NS-2 in flight before the loop; one copy group per tile
  // (empty past the last tile), so that "at most NS-2 groups pending" at
  // iteration t means tile t has landed.
#pragma unroll 1
  for (int t = 0; t < NS - 1; ++t) {
    if (t < n_tiles)
      stage(t, t);
    else
      cp_async_commit();
  }
  for (int t = 0; t < n_tiles; ++t) {
    cp_async_wait<NS - 2>();
    __syncthreads();  // tile t visible to all; stage (t-1) % NS no longer read
    {
      const int tn = t + NS - 1;
      if (tn < n_tiles)
        stage(tn, tn % NS);
      else
        cp_async_commit();
    }
    const int buf = t % NS;
    const float *kt = Ks + buf * TILE + ks * SUB;  // this group's sub-tile
    const float *vt = Vs + buf * TILE + ks * SUB;
    const int lim = row_lim - (t * KS + ks) * kSimtKeys;  // valid sub-tile columns c < lim
    // A warp whose rows all end before this tile skips it (causal only);
    // the condition is the same in all its lanes.
    if (__any_sync(0xffffffffu, lim > 0)) {
      // partial dot products: SP of them per key (4-column chunks taken in turn)
      float sp[SP][KPL];
#pragma unroll
      for (int h = 0; h < SP; ++h)
#pragma unroll
        for (int j = 0; j < KPL; ++j) sp[h][j] = 0.f;
#pragma unroll
      for (int x = 0; x < DP; x += 4 * SP) {
#pragma unroll
        for (int j = 0; j < KPL; ++j) {
#pragma unroll
          for (int h = 0; h < SP; ++h) {
            const int xh = x + 4 * h;
            const float4 kv = *reinterpret_cast<const float4 *>(kt + (g + G * j) * LD + xh);
            sp[h][j] = fmaf(qr[xh], kv.x, sp[h][j]);
            sp[h][j] = fmaf(qr[xh + 1], kv.y, sp[h][j]);
            sp[h][j] = fmaf(qr[xh + 2], kv.z, sp[h][j]);
            sp[h][j] = fmaf(qr[xh + 3], kv.w, sp[h][j]);
          }
        }
      }
      float s[KPL];
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        float dot = sp[0][j];
#pragma unroll
        for (int h = 1; h < SP; ++h) dot += sp[h][j];
        s[j] = (g + G * j < lim) ? dot * p.scale : -INFINITY;
        mt = fmaxf(mt, s[j]);
      }
#pragma unroll
      for (int o = G / 2; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o, G));
      // A group that has seen no valid key of the row yet keeps m = -inf;
      // m_use = 0 then makes alpha and every p exactly 0 instead of NaN.
      // Otherwise m_use = m_new: alpha = 0 on the first valid sub-tile, and
      // 1 on a later fully masked one.
      const float m_new = fmaxf(m, mt);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = expf(m - m_use);
      l *= alpha;
#pragma unroll
      for (int a = 0; a < PVA; ++a)
#pragma unroll
        for (int i = 0; i < CPL; ++i)
#pragma unroll
          for (int u = 0; u < 4; ++u) acc[a][i][u] *= alpha;
      float pr[KPL];
#pragma unroll
      for (int j = 0; j < KPL; ++j) {
        pr[j] = expf(s[j] - m_use);  // 0 for masked keys
        l += pr[j];
      }
      m = m_new;
      // P·V: the probability of key c comes from lane c % G of the group.
#pragma unroll
      for (int c = 0; c < kSimtKeys; ++c) {
        float pc;
        if constexpr (G == 1)
          pc = pr[c];
        else
          pc = __shfl_sync(0xffffffffu, pr[c / G], c % G, G);
        const float *vr = vt + c * LD;
        float(&ac)[CPL][4] = acc[c % PVA];
#pragma unroll
        for (int i = 0; i < CPL; ++i) {
          const float4 vv = *reinterpret_cast<const float4 *>(vr + 4 * (i * G + g));
          ac[i][0] = fmaf(pc, vv.x, ac[i][0]);
          ac[i][1] = fmaf(pc, vv.y, ac[i][1]);
          ac[i][2] = fmaf(pc, vv.z, ac[i][2]);
          ac[i][3] = fmaf(pc, vv.w, ac[i][3]);
        }
      }
    }
  }
  cp_async_wait<0>();  // only empty groups can still be open; close them all
#pragma unroll
  for (int a = 1; a < PVA; ++a)
#pragma unroll
    for (int i = 0; i < CPL; ++i)
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[0][i][u] += acc[a][i][u];

  if constexpr (KS > 1) {
    // Key groups 1 .. KS-1 leave (m, l, O) per thread in shared memory (the
    // ring is no longer read); group 0 merges them into its own:
    // m' = max m_k, l' = sum l_k exp(m_k - m'), O' likewise.  Group 0 holds
    // key 0 of every row, so m' is finite.
    constexpr int W = 2 + 4 * CPL;  // floats per thread
    float *red = Ks;
    __syncthreads();
    if (ks > 0) {
      float *dst = red + ((ks - 1) * TPG + tig) * W;
      dst[0] = m;
      dst[1] = l;
#pragma unroll
      for (int i = 0; i < CPL; ++i)
#pragma unroll
        for (int u = 0; u < 4; ++u) dst[2 + 4 * i + u] = acc[0][i][u];
    }
    __syncthreads();
    if (ks > 0) return;  // whole warps: the shuffles below see full warps
#pragma unroll
    for (int k = 1; k < KS; ++k) {
      const float *src = red + ((k - 1) * TPG + tig) * W;
      const float mk = src[0];
      const float mm = fmaxf(m, mk);
      const float a0 = expf(m - mm), a1 = expf(mk - mm);  // a1 = 0 when mk = -inf
      l = l * a0 + src[1] * a1;
#pragma unroll
      for (int i = 0; i < CPL; ++i)
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[0][i][u] = acc[0][i][u] * a0 + src[2 + 4 * i + u] * a1;
      m = mm;
    }
  }

#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o, G);
  if (active) {
    const float inv_l = 1.f / l;
    float *orow = p.o + (bh * p.Nq + row) * d;
    if (FA_IN(p.status, static_cast<long long>(bh * p.Nq + row) * d, d, q_elems)) {
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        const int x = 4 * (i * G + g);
        if ((d & 3) == 0) {
          if (x < d)
            *reinterpret_cast<float4 *>(orow + x) =
                make_float4(acc[0][i][0] * inv_l, acc[0][i][1] * inv_l,
                            acc[0][i][2] * inv_l, acc[0][i][3] * inv_l);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (x + u < d) orow[x + u] = acc[0][i][u] * inv_l;
        }
      }
    }
    if (g == 0 && FA_IN(p.status, bh * p.Nq + row, 1, planes * p.Nq))
      p.lse[bh * p.Nq + row] = m + logf(l);
  }
}

template <int DP, int G, int KS = 1>
cudaError_t launch_simt_dp(const SimtParams &p_in, int B, cudaStream_t s) {
  constexpr int R = kSimtThreads / (G * KS);
  constexpr int smem = simt_smem_bytes<DP, KS>();
  static std::atomic<unsigned long long> attr_done;
  cudaError_t e = smem_attr_once(fa_simt_fwd_kernel<DP, G, KS>, smem, &attr_done);
  if (e != cudaSuccess) return e;
  SimtParams p = p_in;
  p.n_qtiles = (p.Nq + R - 1) / R;  // this kernel's row tiles
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.n_qtiles), static_cast<unsigned>(p.H),
                     static_cast<unsigned>(B));
  cfg.blockDim = dim3(kSimtThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_simt_fwd_kernel<DP, G, KS>, p);
}

}  // namespace

cudaError_t launch_simt(const SimtParams &p, int B, cudaStream_t s) {
  // The fewest lanes per row (the least shuffling and the fewest shared-memory
  // reads per FMA) whose grid still puts two CTAs on every SM; small problems
  // take the widest split.  G = 1 holds 64 output columns per thread at most,
  // and head dim 32 has only 8 four-column chunks to share out.  A grid still
  // short of that at the widest split also splits each row's keys over KS
  // warp groups (the most, up to 4, that keeps it within two CTAs per SM).
  const long long planes = static_cast<long long>(B) * p.H;
  const long long want = 2LL * (p.num_sms > 0 ? p.num_sms : 1);
  auto ctas = [&](int g, int ks) {
    const int r = kSimtThreads / (g * ks);
    return planes * ((p.Nq + r - 1) / r);
  };
  auto fills = [&](int g) { return ctas(g, 1) >= want; };
  auto key_groups = [&](int g, int most) {
    int k = 1;
    while (k < most && ctas(g, 2 * k) <= want) k *= 2;
    return k;
  };
  if (p.d <= 32) {
    if (fills(1)) return launch_simt_dp<32, 1>(p, B, s);
    if (fills(4)) return launch_simt_dp<32, 4>(p, B, s);
    const int k = key_groups(8, 4);
    return k == 4 ? launch_simt_dp<32, 8, 4>(p, B, s)
         : k == 2 ? launch_simt_dp<32, 8, 2>(p, B, s)
                  : launch_simt_dp<32, 8, 1>(p, B, s);
  }
  if (p.d <= 64) {
    if (fills(1)) return launch_simt_dp<64, 1>(p, B, s);
    if (fills(4)) return launch_simt_dp<64, 4>(p, B, s);
    const int k = key_groups(16, 4);
    return k == 4 ? launch_simt_dp<64, 16, 4>(p, B, s)
         : k == 2 ? launch_simt_dp<64, 16, 2>(p, B, s)
                  : launch_simt_dp<64, 16, 1>(p, B, s);
  }
  if (fills(4)) return launch_simt_dp<128, 4>(p, B, s);
  return key_groups(16, 2) == 2 ? launch_simt_dp<128, 16, 2>(p, B, s)
                                : launch_simt_dp<128, 16, 1>(p, B, s);
}

}  // namespace fa
