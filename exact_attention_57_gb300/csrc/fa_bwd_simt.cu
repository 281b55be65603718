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
// read-modify-write, and the work is spread over 256 threads:
//   * S and dP for a 64 x 64 (query, key) tile: 16 entries a thread;
//   * dK, dV: thread t owns key t/4 and a quarter of the head dim;
//   * dQ: thread t owns query t/4 and a quarter of the head dim.
// All arithmetic is fp32 (expf for the exponential).
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
// offset spreads eight consecutive rows over all banks), then P and dS
// (64 x 65 each), then the tile's LSE and D.
__host__ __device__ inline size_t simt_bwd_smem(int dp) {
  const size_t row = static_cast<size_t>(dp) + 4;
  return (4 * 64 * row + 2 * 64 * 65 + 2 * 64) * sizeof(float);
}

__device__ __forceinline__ float4 ld4(const float *p) {
  return *reinterpret_cast<const float4 *>(p);
}

template <int DP>  // head dim padded up to 32, 64 or 128
// (two blocks an SM up to head dim 64; at 128 the accumulators need more
// than 128 registers a thread)
__global__ void __launch_bounds__(kSbThreads, DP <= 64 ? 2 : 1)
    fa_bwd_simt_kernel(const SimtBwdParams p) {
  extern __shared__ float4 sm4[];
  float *sm = reinterpret_cast<float *>(sm4);
  const int d = p.d;
  constexpr int rs = DP + 4;
  float *Ks = sm, *Vs = Ks + 64 * rs, *Qs = Vs + 64 * rs, *dOs = Qs + 64 * rs;
  float *Ps = dOs + 64 * rs, *dSs = Ps + 64 * 65, *lse_s = dSs + 64 * 65, *dd_s = lse_s + 64;

  const int t = threadIdx.x;
  const int k0 = blockIdx.x * kSbKeys;
  const long long bh = static_cast<long long>(blockIdx.z) * p.H + blockIdx.y;
  const long long q_elems = static_cast<long long>(p.B) * p.H * p.Nq * d;
  const long long kv_elems = static_cast<long long>(p.B) * p.H * p.Nk * d;
  const long long rows_q = static_cast<long long>(p.B) * p.H * p.Nq;
  const float *qh = p.q + bh * p.Nq * d, *doh = p.dout + bh * p.Nq * d;

  // K and V of this block (rows past Nk and columns past d read as zeros)
  for (int e = t; e < 64 * DP; e += kSbThreads) {
    const int j = e / DP, x = e % DP;
    const int key = k0 + j;
    const long long gi = (bh * p.Nk + key) * d + x;
    const bool in = key < p.Nk && x < d && FA_IN(p.status, gi, 1, kv_elems);
    Ks[j * rs + x] = in ? p.k[gi] : 0.f;
    Vs[j * rs + x] = in ? p.v[gi] : 0.f;
  }
  // this thread's share of dK, dV: key kr, columns [c0, c0 + DP/4)
  constexpr int CW = DP / 4;
  const int kr = t >> 2, c0 = (t & 3) * CW;
  float dk_acc[CW], dv_acc[CW];
#pragma unroll
  for (int c = 0; c < CW; ++c) dk_acc[c] = dv_acc[c] = 0.f;

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
    // S, dP -> P, dS for 16 entries: query i = t & 63, keys jb .. jb + 15
    {
      const int i = t & 63, jb = (t >> 6) * 16;
      float s[16], dp[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) s[jj] = dp[jj] = 0.f;
      const int d4 = (d + 3) & ~3;  // columns past d are zero
      for (int x = 0; x < d4; x += 4) {
        const float4 qv = ld4(Qs + i * rs + x), dov = ld4(dOs + i * rs + x);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const float4 kv = ld4(Ks + (jb + jj) * rs + x), vv = ld4(Vs + (jb + jj) * rs + x);
          s[jj] = fmaf(qv.x, kv.x, s[jj]);
          dp[jj] = fmaf(dov.x, vv.x, dp[jj]);
          s[jj] = fmaf(qv.y, kv.y, s[jj]);
          dp[jj] = fmaf(dov.y, vv.y, dp[jj]);
          s[jj] = fmaf(qv.z, kv.z, s[jj]);
          dp[jj] = fmaf(dov.z, vv.z, dp[jj]);
          s[jj] = fmaf(qv.w, kv.w, s[jj]);
          dp[jj] = fmaf(dov.w, vv.w, dp[jj]);
        }
      }
      const int qr = q0 + i;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        const int key = k0 + jb + jj;
        const bool keep = key < p.Nk && (!p.causal || key <= qr);
        const float pv = keep ? expf(s[jj] * p.scale - lse_s[i]) : 0.f;
        Ps[i * 65 + jb + jj] = pv;
        dSs[i * 65 + jb + jj] = pv * (dp[jj] - dd_s[i]);
      }
    }
    __syncthreads();
    // dV += P^T dO, dK += scale dS^T Q for key kr, columns c0 ..
    // (columns past d hold zeros, so their sums stay 0 and are not stored)
    for (int i = 0; i < 64; ++i) {
      const float pv = Ps[i * 65 + kr], ds = dSs[i * 65 + kr];
#pragma unroll
      for (int c = 0; c < CW; c += 4) {
        const float4 ov = ld4(dOs + i * rs + c0 + c), qv = ld4(Qs + i * rs + c0 + c);
        dv_acc[c] = fmaf(pv, ov.x, dv_acc[c]);
        dv_acc[c + 1] = fmaf(pv, ov.y, dv_acc[c + 1]);
        dv_acc[c + 2] = fmaf(pv, ov.z, dv_acc[c + 2]);
        dv_acc[c + 3] = fmaf(pv, ov.w, dv_acc[c + 3]);
        dk_acc[c] = fmaf(ds, qv.x, dk_acc[c]);
        dk_acc[c + 1] = fmaf(ds, qv.y, dk_acc[c + 1]);
        dk_acc[c + 2] = fmaf(ds, qv.z, dk_acc[c + 2]);
        dk_acc[c + 3] = fmaf(ds, qv.w, dk_acc[c + 3]);
      }
    }
    // dQ += scale dS K for query t / 4, columns c0 .. (atomic: every key
    // block adds into the same rows)
    {
      const int i = t >> 2, qr = q0 + i;
      if (qr < p.Nq) {
        float acc[CW];
#pragma unroll
        for (int c = 0; c < CW; ++c) acc[c] = 0.f;
        for (int j = 0; j < 64; ++j) {
          const float ds = dSs[i * 65 + j];
#pragma unroll
          for (int c = 0; c < CW; c += 4) {
            const float4 kv = ld4(Ks + j * rs + c0 + c);
            acc[c] = fmaf(ds, kv.x, acc[c]);
            acc[c + 1] = fmaf(ds, kv.y, acc[c + 1]);
            acc[c + 2] = fmaf(ds, kv.z, acc[c + 2]);
            acc[c + 3] = fmaf(ds, kv.w, acc[c + 3]);
          }
        }
        const long long gbase = (bh * p.Nq + qr) * d + c0;
        if ((d & 3) == 0) {  // rows 16-byte aligned: four adds per instruction
#pragma unroll
          for (int c = 0; c < CW; c += 4)
            if (c0 + c < d && FA_IN(p.status, gbase + c, 4, q_elems))
              red_add_v4(p.dq + gbase + c, acc[c] * p.scale, acc[c + 1] * p.scale,
                       acc[c + 2] * p.scale, acc[c + 3] * p.scale);
        } else {
#pragma unroll
          for (int c = 0; c < CW; ++c)
            if (c0 + c < d && FA_IN(p.status, gbase + c, 1, q_elems))
              atomicAdd(p.dq + gbase + c, acc[c] * p.scale);
        }
      }
    }
  }
  // dK, dV of key kr
  const int key = k0 + kr;
  if (key < p.Nk) {
    const long long gbase = (bh * p.Nk + key) * d + c0;
#pragma unroll
    for (int c = 0; c < CW; ++c) {
      if (c0 + c < d && FA_IN(p.status, gbase + c, 1, kv_elems)) {
        p.dk[gbase + c] = dk_acc[c] * p.scale;
        p.dv[gbase + c] = dv_acc[c];
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
  if (d <= 32) return launch_bwd_simt_dp<32>(p, s);
  if (d <= 64) return launch_bwd_simt_dp<64>(p, s);
  return launch_bwd_simt_dp<128>(p, s);
}

}  // namespace fa
