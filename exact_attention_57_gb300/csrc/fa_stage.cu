// fa_stage.cu — staging pre-pass of the fp32 (TF32) forward: K split once
// per call into bf16 halves K_hi = bf16(K) and K_lo = bf16(K - K_hi), the B
// operands of the three-product score (bf16 products at the 16-bit rate; the
// kernel splits Q the same way), and V rounded to tf32 and transposed into
// the K-major V^T the tf32 P V product takes, instead of both being
// converted by every query-tile CTA.  Rounding: to nearest even for bf16, to
// nearest (ties away) for tf32.
#include <atomic>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

// Two values x -> packed bf16 pairs hi = bf16(x) and lo = bf16(x - hi): the
// split operands of the three bf16 products (about 2^-16 of x left out).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  hi = pack_bf16x2(x0, x1);
  lo = pack_bf16x2(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xffff0000u));
}

// One launch for both passes, side by side: blocks [0, split_blocks) split K
// (a grid-stride loop over its float4s), the others transpose V, one
// 64-key x 32-column tile of one head at a time: v[n0 + r][x0 + c] ->
// vt[x0 + c][n0 + r], rounded to tf32; keys n0 + r >= Nk give 0 up to
// nk_pad.  Both are bound by memory; sharing the GPU, each fills the other's
// gaps, and the call pays one launch.
__global__ void __launch_bounds__(256)
    fa_stage_kernel(const float4 *__restrict__ k, uint2 *__restrict__ kr,
                    uint2 *__restrict__ kl, long long n4, int split_blocks,
                    const float *__restrict__ v, float *__restrict__ vt, long long BH, int Nk,
                    int nk_pad, int d) {
  if (static_cast<int>(blockIdx.x) < split_blocks) {
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<long long>(split_blocks) * blockDim.x) {
      const float4 a = k[i];
      uint2 h, l;
      split_bf16x2(a.x, a.y, h.x, l.x);
      split_bf16x2(a.z, a.w, h.y, l.y);
      kr[i] = h;
      kl[i] = l;
    }
    return;  // the whole block: no barrier below is shared with it
  }
  __shared__ float tile[64][33];
  const long long ntn = nk_pad / 64, ntx = (d + 31) / 32;
  const long long ntiles = ntn * ntx * BH;
  const int t = threadIdx.x;
  for (long long ti = static_cast<long long>(blockIdx.x) - split_blocks; ti < ntiles;
       ti += static_cast<long long>(gridDim.x) - split_blocks) {
    const int n0 = static_cast<int>(ti % ntn) * 64;
    const int x0 = static_cast<int>((ti / ntn) % ntx) * 32;
    const long long bh = ti / (ntn * ntx);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      // row r of the tile, columns 4c .. 4c+3 (d is a multiple of 32)
      const int r = (t >> 3) + 32 * i, c = t & 7;
      const int n = n0 + r, x = x0 + 4 * c;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (n < Nk && x < d) a = *reinterpret_cast<const float4 *>(v + (bh * Nk + n) * d + x);
      tile[r][4 * c + 0] = a.x;
      tile[r][4 * c + 1] = a.y;
      tile[r][4 * c + 2] = a.z;
      tile[r][4 * c + 3] = a.w;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      // output row x0 + xr, keys n0 + 4u .. n0 + 4u + 3
      const int xr = t >> 3, u = (t & 7) + 8 * i;
      const int x = x0 + xr, n = n0 + 4 * u;
      if (x < d && n < nk_pad) {
        float4 b;
        b.x = __uint_as_float(to_tf32(tile[4 * u + 0][xr]));
        b.y = __uint_as_float(to_tf32(tile[4 * u + 1][xr]));
        b.z = __uint_as_float(to_tf32(tile[4 * u + 2][xr]));
        b.w = __uint_as_float(to_tf32(tile[4 * u + 3][xr]));
        *reinterpret_cast<float4 *>(vt + (bh * d + x) * nk_pad + n) = b;
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_stage_f32(const float *k, const float *v, __nv_bfloat16 *kr,
                             __nv_bfloat16 *kl, float *vt, int BH, int Nk, int nk_pad, int d,
                             cudaStream_t s) {
  const long long n4 = static_cast<long long>(BH) * Nk * d / 4;  // d is a multiple of 32
  // 8 blocks of 256 threads fill an SM: half of them split K, half
  // transpose V (the two move the same bytes).  The SM count is read once
  // per device.
  static std::atomic<int> sm_cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = (dev >= 0 && dev < 64) ? sm_cache[dev].load(std::memory_order_relaxed) : 0;
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) sm_cache[dev].store(sms, std::memory_order_relaxed);
  }
  const int half = 4 * (sms > 0 ? sms : 1);
  fa_stage_kernel<<<2 * half, 256, 0, s>>>(reinterpret_cast<const float4 *>(k),
                                          reinterpret_cast<uint2 *>(kr),
                                          reinterpret_cast<uint2 *>(kl), n4, half, v, vt, BH,
                                          Nk, nk_pad, d);
  return cudaGetLastError();
}

}  // namespace fa
