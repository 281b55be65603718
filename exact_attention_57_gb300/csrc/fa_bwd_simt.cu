// fa_bwd_simt.cu — fp32 backward of exact attention on the CUDA cores (no
// tensor cores), the gradients of fa_fwd for FA_DTYPE_F32 and
// FA_DTYPE_F32_SIMT inputs.
//
// Method: the backward kernel of "flash_attention_2.cu"
// (leloykun/flash-hyperbolic-attention-minimal), from the saved LSE:
//   P = exp(scale * Q K^T - LSE),  D = rowsum(dO * O),
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//   dQ = scale * dS K,  dK = scale * dS^T Q,
// with top-left causal masking (key j allowed for query i iff j <= i).
// Like that page's kernel, one block owns a block of keys and walks the
// query tiles, accumulating dK and dV on chip; unlike it, dV takes the
// query's row of dO (the page reads the key's row there), dQ is added into
// the fp32 output with atomics from every key block instead of a
// read-modify-write, and the work is spread over 256 threads, each with a
// 4 x 4 register block of every product (S and dP of a 64 x 64 tile, dK and
// dV of 4 keys, dQ of 4 queries).  All arithmetic is fp32 (expf for the
// exponential).
#include <cmath>

#include "fa.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr int kSbKeys = 64;     // keys per block
constexpr int kSbQueries = 64;  // queries per tile
constexpr int kSbThreads = 256;

// D = rowsum(dO * O) per query row (one warp a row) and dq zeroed.
__global__ void __launch_bounds__(256)
    fa_bwd_simt_prep_kernel(const float *__restrict__ o, const float *__restrict__ dout,
                            float *__restrict__ dd, float *__restrict__ dq, long long rows, int d,
                            unsigned *status) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;  // whole warp
  float acc = 0.f;
  for (int x = lane; x < d; x += 32) {
    if (FA_IN(status, row * d + x, 1, rows * d)) {
      acc = fmaf(o[row * d + x], dout[row * d + x], acc);
      dq[row * d + x] = 0.f;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0 && FA_IN(status, row, 1, rows)) dd[row] = acc;
}

struct SimtBwdParams {
  const float *q, *k, *v, *dout, *lse, *dd;
  float *dq, *dk, *dv;
  unsigned *status;
  int B, H, Nq, Nk, d;
  float scale;
  int causal;
};

// Shared memory: K, V, Q, dO tiles of 64 rows of DP + 4 floats (columns
// past d zero; rows 16-byte aligned for float4 reads, and the 4-float
// offset puts eight consecutive rows on distinct banks), then P and dS (64 x
// 68 each, the same alignment), then the tile's LSE and D.
constexpr int kSbPL = 68;  // row stride of P and dS
__host__ __device__ inline size_t simt_bwd_smem(int dp) {
  const size_t row = static_cast<size_t>(dp) + 4;
  return (4 * 64 * row + 2 * 64 * kSbPL + 2 * 64) * sizeof(float);
}

__device__ __forceinline__ float4 ld4(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}
__device__ __forceinline__ void axpy4(float a, float4 x, float *y) {
  y[0] = fmaf(a, x.x, y[0]);
  y[1] = fmaf(a, x.y, y[1]);
  y[2] = fmaf(a, x.z, y[2]);
  y[3] = fmaf(a, x.w, y[3]);
}

// Register blocking: each of the 256 threads computes a 4 x 4 block of S and
// dP (queries lo + 16a, keys hi + 16b; lo = t % 16, hi = t / 16), of dK and
// dV (keys 4lo .. 4lo+3 x columns hi*CB ..), and of dQ (queries lo + 16a x
// columns hi*CB ..), CB = DP / 16: one 16-byte shared-memory read per 8
// FMAs or fewer, the lanes of a warp reading consecutive rows (no bank
// conflicts) or the same address (a broadcast).
template <int DP>  // head dim padded up to 64 or 128
// (two blocks an SM at 64; at 128 the accumulators need more than 128
// registers a thread)
__global__ void __launch_bounds__(kSbThreads, DP <= 64 ? 2 : 1)
    fa_bwd_simt_kernel(const SimtBwdParams p) {
  constexpr int rs = DP + 4;
  constexpr int PL = kSbPL;
  constexpr int CB = DP / 16;  // columns per thread (dK, dV, dQ)
  static_assert(CB % 4 == 0, "whole float4 column chunks");
  extern __shared__ float4 sm4[];
  float *sm = reinterpret_cast<float *>(sm4);
  const int d = p.d;
  float *Ks = sm, *Vs = Ks + 64 * rs, *Qs = Vs + 64 * rs, *dOs = Qs + 64 * rs;
  float *Ps = dOs + 64 * rs, *dSs = Ps + 64 * PL, *lse_s = dSs + 64 * PL, *dd_s = lse_s + 64;

  const int t = threadIdx.x;
  const int lo = t & 15, hi = t >> 4;
  const int k0 = blockIdx.x * kSbKeys;
  const long long bh = static_cast<long long>(blockIdx.z) * p.H + blockIdx.y;
  const long long q_elems = static_cast<long long>(p.B) * p.H * p.Nq * d;
  const long long kv_elems = static_cast<long long>(p.B) * p.H * p.Nk * d;
  const long long rows_q = static_cast<long long>(p.B) * p.H * p.Nq;
  const float *qh = p.q + bh * p.Nq * d, *doh = p.dout + bh * p.Nq * d;
  const int d4 = (d + 3) & ~3;  // columns past d are zero

  // K and V of this block (rows past Nk and columns past d read as zeros)
  for (int e = t; e < 64 * DP; e += kSbThreads) {
    const int j = e / DP, x = e % DP;
    const int key = k0 + j;
    const long long gi = (bh * p.Nk + key) * d + x;
    const bool in = key < p.Nk && x < d && FA_IN(p.status, gi, 1, kv_elems);
    Ks[j * rs + x] = in ? p.k[gi] : 0.f;
    Vs[j * rs + x] = in ? p.v[gi] : 0.f;
  }
  // dK, dV of keys 4lo + a, columns hi*CB + c
  const int cb = hi * CB;
  float dk_acc[4][CB], dv_acc[4][CB];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < CB; ++c) dk_acc[a][c] = dv_acc[a][c] = 0.f;

  const int n_qt = (p.Nq + kSbQueries - 1) / kSbQueries;
  // causal: query tiles whose last row is before the block's first key see
  // none of its keys
  const int qt_first = p.causal ? k0 / kSbQueries : 0;
  for (int qt = qt_first; qt < n_qt; ++qt) {
    const int q0 = qt * kSbQueries;
    __syncthreads();  // the previous tile's shared data is no longer read
    for (int e = t; e < 64 * DP; e += kSbThreads) {
      const int i = e / DP, x = e % DP;
      const int qr = q0 + i;
      const long long gi = (bh * p.Nq + qr) * d + x;
      const bool in = qr < p.Nq && x < d && FA_IN(p.status, gi, 1, q_elems);
      Qs[i * rs + x] = in ? qh[static_cast<long long>(qr) * d + x] : 0.f;
      dOs[i * rs + x] = in ? doh[static_cast<long long>(qr) * d + x] : 0.f;
    }
    if (t < 64) {
      const int qr = q0 + t;
      const bool in = qr < p.Nq && FA_IN(p.status, bh * p.Nq + qr, 1, rows_q);
      lse_s[t] = in ? p.lse[bh * p.Nq + qr] : INFINITY;  // P = 0 for padded rows
      dd_s[t] = in ? p.dd[bh * p.Nq + qr] : 0.f;
    }
    __syncthreads();
    // S, dP -> P, dS: queries lo + 16a, keys hi + 16b
    {
      float s[4][4], dp[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) s[a][b] = dp[a][b] = 0.f;
      for (int x = 0; x < d4; x += 4) {
        float4 qv[4], ov[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          qv[a] = ld4(Qs + (lo + 16 * a) * rs + x);
          ov[a] = ld4(dOs + (lo + 16 * a) * rs + x);
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const float4 kv = ld4(Ks + (hi + 16 * b) * rs + x);
          const float4 vv = ld4(Vs + (hi + 16 * b) * rs + x);
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            s[a][b] = dot4(qv[a], kv, s[a][b]);
            dp[a][b] = dot4(ov[a], vv, dp[a][b]);
          }
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = lo + 16 * a, qr = q0 + i;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int j = hi + 16 * b, key = k0 + j;
          const bool keep = key < p.Nk && (!p.causal || key <= qr);
          const float pv = keep ? expf(s[a][b] * p.scale - lse_s[i]) : 0.f;
          Ps[i * PL + j] = pv;
          dSs[i * PL + j] = pv * (dp[a][b] - dd_s[i]);
        }
      }
    }
    __syncthreads();
    // dV += P^T dO, dK += dS^T Q (scale applied at the store): keys 4lo + a
    // (columns past d hold zeros, so their sums stay 0 and are not stored)
    for (int i = 0; i < 64; ++i) {
      const float4 p4 = ld4(Ps + i * PL + 4 * lo), s4 = ld4(dSs + i * PL + 4 * lo);
      const float pa[4] = {p4.x, p4.y, p4.z, p4.w}, sa[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
      for (int c = 0; c < CB; c += 4) {
        const float4 ov = ld4(dOs + i * rs + cb + c), qv = ld4(Qs + i * rs + cb + c);
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          axpy4(pa[a], ov, &dv_acc[a][c]);
          axpy4(sa[a], qv, &dk_acc[a][c]);
        }
      }
    }
    // dQ += scale dS K: queries lo + 16a, columns cb .. cb + CB (atomic:
    // every key block adds into the same rows)
    {
      float acc[4][CB];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < CB; ++c) acc[a][c] = 0.f;
      for (int j = 0; j < 64; j += 4) {
        float4 ds[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) ds[a] = ld4(dSs + (lo + 16 * a) * PL + j);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
          for (int c = 0; c < CB; c += 4) {
            const float4 kv = ld4(Ks + (j + jj) * rs + cb + c);
#pragma unroll
            for (int a = 0; a < 4; ++a) {
              const float w = jj == 0 ? ds[a].x : jj == 1 ? ds[a].y : jj == 2 ? ds[a].z : ds[a].w;
              axpy4(w, kv, &acc[a][c]);
            }
          }
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int qr = q0 + lo + 16 * a;
        if (qr >= p.Nq) continue;
        const long long gbase = (bh * p.Nq + qr) * d + cb;
        if ((d & 3) == 0) {  // rows 16-byte aligned: four adds per instruction
#pragma unroll
          for (int c = 0; c < CB; c += 4)
            if (cb + c < d && FA_IN(p.status, gbase + c, 4, q_elems))
              red_add_v4(p.dq + gbase + c, acc[a][c] * p.scale, acc[a][c + 1] * p.scale,
                         acc[a][c + 2] * p.scale, acc[a][c + 3] * p.scale);
        } else {
#pragma unroll
          for (int c = 0; c < CB; ++c)
            if (cb + c < d && FA_IN(p.status, gbase + c, 1, q_elems))
              atomicAdd(p.dq + gbase + c, acc[a][c] * p.scale);
        }
      }
    }
  }
  // dK, dV of keys 4lo + a
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int key = k0 + 4 * lo + a;
    if (key >= p.Nk) continue;
    const long long gbase = (bh * p.Nk + key) * d + cb;
#pragma unroll
    for (int c = 0; c < CB; ++c) {
      if (cb + c < d && FA_IN(p.status, gbase + c, 1, kv_elems)) {
        p.dk[gbase + c] = dk_acc[a][c] * p.scale;
        p.dv[gbase + c] = dv_acc[a][c];
      }
    }
  }
}

template <int DP>
cudaError_t launch_bwd_simt_dp(const SimtBwdParams &p, cudaStream_t s) {
  const size_t smem = simt_bwd_smem(DP);
  static std::atomic<unsigned long long> attr_done;
  cudaError_t e = smem_attr_once(fa_bwd_simt_kernel<DP>, static_cast<int>(smem), &attr_done);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((p.Nk + kSbKeys - 1) / kSbKeys),
                  static_cast<unsigned>(p.H), static_cast<unsigned>(p.B));
  fa_bwd_simt_kernel<DP><<<grid, kSbThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_simt(const float *q, const float *k, const float *v, const float *o,
                            const float *lse, const float *dout, float *dq, float *dk, float *dv,
                            float *dd, int B, int H, int Nq, int Nk, int d, float scale,
                            int causal, unsigned *status, cudaStream_t s) {
  const long long rows = static_cast<long long>(B) * H * Nq;
  fa_bwd_simt_prep_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(o, dout, dd, dq,
                                                                               rows, d, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  SimtBwdParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.dout = dout;
  p.lse = lse;
  p.dd = dd;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.status = status;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.d = d;
  p.scale = scale;
  p.causal = causal;
  if (d <= 64) return launch_bwd_simt_dp<64>(p, s);
  return launch_bwd_simt_dp<128>(p, s);
}

}  // namespace fa
