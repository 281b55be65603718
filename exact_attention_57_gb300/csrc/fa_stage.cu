// fa_stage.cu — staging pre-pass of the fp32 (TF32) forward: K split once
// per call into K_hi = tf32(K) and K_lo = tf32(K - K_hi), the B operands of
// the three-product score, and V rounded and transposed into the K-major V^T
// the tf32 P V product takes, instead of both being converted by every
// query-tile CTA.  Rounding is to nearest (ties away), the rounding the kernel
// itself applies to Q.
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {

namespace {

// x_hi = tf32(x) and x_lo = tf32(x - x_hi): the split operands of the three
// tf32 products that give the scores about fp32 accuracy.
__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo) {
  hi = __uint_as_float(to_tf32(x));
  lo = __uint_as_float(to_tf32(x - hi));
}

__global__ void fa_stage_split_kernel(const float4 *__restrict__ k, float4 *__restrict__ kr,
                                      float4 *__restrict__ kl, long long n4) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = k[i];
    float4 h, l;
    split_tf32(a.x, h.x, l.x);
    split_tf32(a.y, h.y, l.y);
    split_tf32(a.z, h.z, l.z);
    split_tf32(a.w, h.w, l.w);
    kr[i] = h;
    kl[i] = l;
  }
}

// One 32 x 32 tile per block and head: v[n0 + r][x0 + c] -> vt[x0 + c][n0 + r];
// heads stride by gridDim.z (which is capped at 65535).
__global__ void __launch_bounds__(256)
    fa_stage_transpose_kernel(const float *__restrict__ v, float *__restrict__ vt, long long BH,
                              int Nk, int nk_pad, int d) {
  __shared__ float tile[32][33];
  const int n0 = blockIdx.x * 32, x0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (long long bh = blockIdx.z; bh < BH; bh += gridDim.z) {
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      const int n = n0 + ty + i, x = x0 + tx;
      tile[ty + i][tx] = (n < Nk && x < d) ? v[(bh * Nk + n) * d + x] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      const int x = x0 + ty + i, n = n0 + tx;
      if (x < d && n < nk_pad)
        vt[(bh * d + x) * nk_pad + n] = __uint_as_float(to_tf32(tile[tx][ty + i]));
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_stage_f32(const float *k, const float *v, float *kr, float *kl, float *vt,
                             int BH, int Nk, int nk_pad, int d, cudaStream_t s) {
  const long long n4 = static_cast<long long>(BH) * Nk * d / 4;  // d is a multiple of 32
  fa_stage_split_kernel<<<1216, 256, 0, s>>>(reinterpret_cast<const float4 *>(k),
                                             reinterpret_cast<float4 *>(kr),
                                             reinterpret_cast<float4 *>(kl), n4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(nk_pad / 32), static_cast<unsigned>((d + 31) / 32),
                  static_cast<unsigned>(BH < 65535 ? BH : 65535));
  fa_stage_transpose_kernel<<<grid, 256, 0, s>>>(v, vt, BH, Nk, nk_pad, d);
  return cudaGetLastError();
}

}  // namespace fa
