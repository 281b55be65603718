// fa_simt.cu — plain fp32 (no tensor cores) exact-attention forward.
//
// The same method as the tensor-core kernels — the forward kernel of
// "flash_attention_2.cu" (leloykun/flash-hyperbolic-attention-minimal):
// scores scaled before the row max, online softmax over key tiles with a
// running max m and sum l, partial output rescaled by exp(m_old - m_new),
// O = O / l and L = m + log(l) at the end — computed with fp32 FMAs.
//
// Differences from that page's kernel, each deliberate:
//   * one CTA per (batch, head, 128-row query tile) instead of one per
//     (batch, head), so the grid does not depend on B*H;
//   * O accumulates in registers and is written once (the page
//     read-modify-writes O in global memory every key tile and therefore
//     needs O zeroed first);
//   * rows past Nq stay in the loop until the end (the page breaks out of the
//     loop before a __syncthreads, a divergent-barrier hazard);
//   * keys past Nk and, when causal, keys after the query are excluded
//     element by element, on every tile, not only within a row's own tile.
// One thread owns one query row (64 rows per CTA, so that small problems
// still spread over several SMs); K/V tiles of 32 keys are staged in shared
// memory and read as broadcasts.  The 32 dot products of a tile run side by
// side (head-dim index outer, key inner), so no FMA waits on the previous
// one.
#include <cmath>

#include "fa_internal.h"

namespace fa {

namespace {

constexpr int kSimtRows = 64;   // query rows per CTA (one per thread)

// Asynchronous 4-byte copy global -> shared (cp.async; zero fill when
// `valid` is false, in which case `src` is not read).
__device__ __forceinline__ void cp_async4(float *dst, const float *src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src),
               "r"(valid ? 4 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}
constexpr int kSimtKeys = 32;   // keys per shared-memory tile

template <int DP>  // head dim padded up to 32, 64 or 128
__global__ void __launch_bounds__(kSimtRows) fa_simt_fwd_kernel(const SimtParams p) {
  __shared__ float Ks[kSimtKeys * DP];
  __shared__ float Vs[kSimtKeys * DP];
  const int qt = p.causal ? (p.n_qtiles - 1 - static_cast<int>(blockIdx.x))
                          : static_cast<int>(blockIdx.x);
  const size_t bh = static_cast<size_t>(blockIdx.z) * p.H + blockIdx.y;
  const int d = p.d;
  const int row = qt * kSimtRows + static_cast<int>(threadIdx.x);
  const bool active = row < p.Nq;
  const float *qh = p.q + bh * p.Nq * d;
  const float *kh = p.k + bh * p.Nk * d;
  const float *vh = p.v + bh * p.Nk * d;
  // extents for the debug build's index checks
  const long long planes = static_cast<long long>(p.B) * p.H;
  const long long q_elems = planes * p.Nq * d, kv_elems = planes * p.Nk * d;
  const bool q_ok =
      active && FA_IN(p.status, static_cast<long long>(bh * p.Nq + row) * d, d, q_elems);

  float qr[DP], acc[DP];
#pragma unroll
  for (int x = 0; x < DP; ++x) {
    qr[x] = (q_ok && x < d) ? qh[static_cast<size_t>(row) * d + x] : 0.f;
    acc[x] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  // keys [0, row_lim) take part for this row; the CTA visits keys up to the
  // largest row_lim among its rows.
  const int row_lim = p.causal ? min(row + 1, p.Nk) : p.Nk;
  const int cta_lim = p.causal ? min(qt * kSimtRows + kSimtRows, p.Nk) : p.Nk;

  for (int k0 = 0; k0 < cta_lim; k0 += kSimtKeys) {
    __syncthreads();
    // every copy of the tile in flight at once (one memory round trip)
    for (int e = threadIdx.x; e < kSimtKeys * DP; e += kSimtRows) {
      const int c = e / DP, x = e % DP;
      const int key = k0 + c;
      const bool in = key < p.Nk && x < d &&
                      FA_IN(p.status, static_cast<long long>(bh * p.Nk + key) * d + x, 1, kv_elems);
      const size_t off = in ? static_cast<size_t>(key) * d + x : 0;
      cp_async4(Ks + e, kh + off, in);
      cp_async4(Vs + e, vh + off, in);
    }
    cp_async_wait_all();
    __syncthreads();
    const int lim = row_lim - k0;  // valid columns c < lim
    if (active && lim > 0) {
      float s[kSimtKeys];
#pragma unroll
      for (int c = 0; c < kSimtKeys; ++c) s[c] = 0.f;
#pragma unroll
      for (int x = 0; x < DP; ++x) {
#pragma unroll
        for (int c = 0; c < kSimtKeys; ++c) s[c] = fmaf(qr[x], Ks[c * DP + x], s[c]);
      }
      float mt = -INFINITY;
#pragma unroll
      for (int c = 0; c < kSimtKeys; ++c) {
        s[c] *= p.scale;
        if (c < lim) mt = fmaxf(mt, s[c]);
      }
      const float m_new = fmaxf(m, mt);
      const float alpha = expf(m - m_new);  // 0 on the first visited tile
      l *= alpha;
#pragma unroll
      for (int x = 0; x < DP; ++x) acc[x] *= alpha;
#pragma unroll
      for (int c = 0; c < kSimtKeys; ++c) {
        const float pc = (c < lim) ? expf(s[c] - m_new) : 0.f;
        l += pc;
#pragma unroll
        for (int x = 0; x < DP; ++x) acc[x] = fmaf(pc, Vs[c * DP + x], acc[x]);
      }
      m = m_new;
    }
  }
  if (active) {
    const float inv_l = 1.f / l;
    float *orow = p.o + (bh * p.Nq + row) * d;
    if (FA_IN(p.status, static_cast<long long>(bh * p.Nq + row) * d, d, q_elems)) {
#pragma unroll
      for (int x = 0; x < DP; ++x)
        if (x < d) orow[x] = acc[x] * inv_l;
    }
    if (FA_IN(p.status, bh * p.Nq + row, 1, planes * p.Nq)) p.lse[bh * p.Nq + row] = m + logf(l);
  }
}

template <int DP>
cudaError_t launch_simt_dp(const SimtParams &p_in, int B, cudaStream_t s) {
  SimtParams p = p_in;
  p.n_qtiles = (p.Nq + kSimtRows - 1) / kSimtRows;  // this kernel's row tiles
  dim3 grid(static_cast<unsigned>(p.n_qtiles), static_cast<unsigned>(p.H),
            static_cast<unsigned>(B));
  fa_simt_fwd_kernel<DP><<<grid, kSimtRows, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt(const SimtParams &p, int B, cudaStream_t s) {
  if (p.d <= 32) return launch_simt_dp<32>(p, B, s);
  if (p.d <= 64) return launch_simt_dp<64>(p, B, s);
  return launch_simt_dp<128>(p, B, s);
}

}  // namespace fa
