// fa_bwd_aux.cu — the two memory-bound steps around the tensor-core backward.
//
// Before it: per query row, D = rowsum(dO * O) (the D of the backward kernel
// of "flash_attention_2.cu", leloykun/flash-hyperbolic-attention-minimal),
// the saved LSE in log2 units, and a zeroed fp32 dQ accumulator row.  Rows
// from Nq up to the padded tile end get LSE = +inf and D = 0, which makes
// their probabilities exactly 0 in the main kernel.
// After it: dQ rounded from the fp32 accumulator to the input type.
//
// The accumulator is plane-major with rows of DA = max(d, 64) floats (the
// gradient kernel's head dim): [B*H][Nq][DA], or [H][total_q][DA] for
// variable-length batches; only the first d floats of a row are used.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "fa_internal.h"

namespace fa {

namespace {

constexpr int kPrepRowsPerBlock = 8;  // one warp per row

template <int D>
constexpr int acc_dim() { return D < 64 ? 64 : D; }

__device__ __forceinline__ float2 load2(const void *base, size_t idx, bool half) {
  const uint32_t w = *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(base) + idx);
  if (half) {
    const __half2 h = *reinterpret_cast<const __half2 *>(&w);
    return __half22float2(h);
  }
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&w);
  return __bfloat1622float2(b);
}

template <int D>
__global__ void __launch_bounds__(32 * kPrepRowsPerBlock)
    fa_bwd_prep_kernel(const void *__restrict__ o, const void *__restrict__ dout,
                       const float *__restrict__ lse, float *__restrict__ lse2,
                       float *__restrict__ dd, float *__restrict__ dq_acc, int BH, int Nq,
                       int Nq_pad, int half) {
  const int lane = threadIdx.x & 31;
  const long long prow =
      static_cast<long long>(blockIdx.x) * kPrepRowsPerBlock + (threadIdx.x >> 5);
  if (prow >= static_cast<long long>(BH) * Nq_pad) return;  // whole warp
  const int bh = static_cast<int>(prow / Nq_pad);
  const int q = static_cast<int>(prow - static_cast<long long>(bh) * Nq_pad);
  if (q >= Nq) {
    if (lane == 0) {
      lse2[prow] = INFINITY;
      dd[prow] = 0.f;
    }
    return;
  }
  const size_t row = static_cast<size_t>(bh) * Nq + q;
  // lane covers elements [2*lane + 64*i, +2)
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < (D + 63) / 64; ++i) {
    if (64 * i + 2 * lane < D) {
      const size_t idx = row * D + 64 * i + 2 * lane;
      const float2 a = load2(o, idx, half != 0), b = load2(dout, idx, half != 0);
      acc = fmaf(a.x, b.x, acc);
      acc = fmaf(a.y, b.y, acc);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  float *zrow = dq_acc + row * acc_dim<D>();
  // D / 4 float4 per row, 32 per pass
#pragma unroll
  for (int i = 0; i < (D / 4 + 31) / 32; ++i)
    if (32 * i + lane < D / 4)
      reinterpret_cast<float4 *>(zrow)[32 * i + lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane == 0) {
    lse2[prow] = lse[row] * 1.4426950408889634f;
    dd[prow] = acc;
  }
}

// Variable-length batches: padded row prow = (h*B + b)*Nq_pad + pos of the
// LSE/D buffers; token t = cu_q[b] + pos of q/o/dout (token-major
// [total_q, H, D]) and of accumulator plane h; lse [H, total_q].
template <int D>
__global__ void __launch_bounds__(32 * kPrepRowsPerBlock)
    fa_bwd_prep_varlen_kernel(const void *__restrict__ o, const void *__restrict__ dout,
                              const float *__restrict__ lse, float *__restrict__ lse2,
                              float *__restrict__ dd, float *__restrict__ dq_acc,
                              const int *__restrict__ cu_q, int B, int H, int total_q,
                              int Nq_pad, int half) {
  const int lane = threadIdx.x & 31;
  const long long prow =
      static_cast<long long>(blockIdx.x) * kPrepRowsPerBlock + (threadIdx.x >> 5);
  if (prow >= static_cast<long long>(H) * B * Nq_pad) return;  // whole warp
  const long long hb = prow / Nq_pad;
  const int pos = static_cast<int>(prow - hb * Nq_pad);
  const int b = static_cast<int>(hb % B), h = static_cast<int>(hb / B);
  const int t0 = min(max(cu_q[b], 0), total_q);  // clamped, as in the kernel
  const int nq = min(max(0, min(cu_q[b + 1], total_q) - t0), Nq_pad);
  if (pos >= nq) {
    if (lane == 0) {
      lse2[prow] = INFINITY;
      dd[prow] = 0.f;
    }
    return;
  }
  const size_t row = static_cast<size_t>(t0 + pos) * H + h;  // token-major row
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < (D + 63) / 64; ++i) {
    if (64 * i + 2 * lane < D) {
      const size_t idx = row * D + 64 * i + 2 * lane;
      const float2 a = load2(o, idx, half != 0), c = load2(dout, idx, half != 0);
      acc = fmaf(a.x, c.x, acc);
      acc = fmaf(a.y, c.y, acc);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  float *zrow = dq_acc + (static_cast<size_t>(h) * total_q + t0 + pos) * acc_dim<D>();
#pragma unroll
  for (int i = 0; i < (D / 4 + 31) / 32; ++i)
    if (32 * i + lane < D / 4)
      reinterpret_cast<float4 *>(zrow)[32 * i + lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane == 0) {
    lse2[prow] = lse[static_cast<size_t>(h) * total_q + t0 + pos] * 1.4426950408889634f;
    dd[prow] = acc;
  }
}

// Output row o of dq (d elements; 8 per thread): [B,H,Nq,d] order, which is
// also the accumulator's row order, or for variable-length batches
// token-major, o = t*H + h, read from accumulator row h*total_q + t.
template <bool VARLEN>
__global__ void fa_bwd_convert_kernel(const float *__restrict__ src, void *__restrict__ dst,
                                      long long rows, int chunk_shift, int acc_d, int H,
                                      int total_q, int half) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= (rows << chunk_shift)) return;
  const long long o = i >> chunk_shift;
  const int c = static_cast<int>(i - (o << chunk_shift)) * 8;
  long long srow = o;
  if (VARLEN) {
    const long long t = o / H;
    srow = static_cast<long long>(o - t * H) * total_q + t;
  }
  const float4 *in = reinterpret_cast<const float4 *>(src + srow * acc_d + c);
  const float4 a = in[0], b = in[1];
  uint4 out;
  if (half) {
    const __half2 h0 = __floats2half2_rn(a.x, a.y), h1 = __floats2half2_rn(a.z, a.w);
    const __half2 h2 = __floats2half2_rn(b.x, b.y), h3 = __floats2half2_rn(b.z, b.w);
    out = make_uint4(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1),
                     *reinterpret_cast<const uint32_t *>(&h2), *reinterpret_cast<const uint32_t *>(&h3));
  } else {
    const __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x, a.y), h1 = __floats2bfloat162_rn(a.z, a.w);
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(b.x, b.y), h3 = __floats2bfloat162_rn(b.z, b.w);
    out = make_uint4(*reinterpret_cast<const uint32_t *>(&h0), *reinterpret_cast<const uint32_t *>(&h1),
                     *reinterpret_cast<const uint32_t *>(&h2), *reinterpret_cast<const uint32_t *>(&h3));
  }
  // d is a multiple of 8, so o*d + c is a multiple of 8 elements (16 bytes).
  reinterpret_cast<uint4 *>(static_cast<uint16_t *>(dst) + (o << (chunk_shift + 3)) + c)[0] = out;
}

}  // namespace

cudaError_t launch_bwd_prep(const void *o, const void *dout, const float *lse, float *lse2,
                            float *dd, float *dq_acc, int BH, int Nq, int Nq_pad, int d, int half,
                            cudaStream_t s) {
  const long long rows = static_cast<long long>(BH) * Nq_pad;
  const unsigned blocks = static_cast<unsigned>((rows + kPrepRowsPerBlock - 1) / kPrepRowsPerBlock);
  if (d == 32)
    fa_bwd_prep_kernel<32><<<blocks, 32 * kPrepRowsPerBlock, 0, s>>>(o, dout, lse, lse2, dd,
                                                                     dq_acc, BH, Nq, Nq_pad, half);
  else if (d == 64)
    fa_bwd_prep_kernel<64><<<blocks, 32 * kPrepRowsPerBlock, 0, s>>>(o, dout, lse, lse2, dd,
                                                                     dq_acc, BH, Nq, Nq_pad, half);
  else
    fa_bwd_prep_kernel<128><<<blocks, 32 * kPrepRowsPerBlock, 0, s>>>(o, dout, lse, lse2, dd,
                                                                      dq_acc, BH, Nq, Nq_pad, half);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep_varlen(const void *o, const void *dout, const float *lse, float *lse2,
                                   float *dd, float *dq_acc, const int *cu_q, int B, int H,
                                   int total_q, int Nq_pad, int d, int half, cudaStream_t s) {
  const long long rows = static_cast<long long>(H) * B * Nq_pad;
  const unsigned blocks = static_cast<unsigned>((rows + kPrepRowsPerBlock - 1) / kPrepRowsPerBlock);
  const dim3 block(32 * kPrepRowsPerBlock);
  if (d == 32)
    fa_bwd_prep_varlen_kernel<32><<<blocks, block, 0, s>>>(o, dout, lse, lse2, dd, dq_acc, cu_q, B,
                                                           H, total_q, Nq_pad, half);
  else if (d == 64)
    fa_bwd_prep_varlen_kernel<64><<<blocks, block, 0, s>>>(o, dout, lse, lse2, dd, dq_acc, cu_q, B,
                                                           H, total_q, Nq_pad, half);
  else
    fa_bwd_prep_varlen_kernel<128><<<blocks, block, 0, s>>>(o, dout, lse, lse2, dd, dq_acc, cu_q, B,
                                                            H, total_q, Nq_pad, half);
  return cudaGetLastError();
}

cudaError_t launch_bwd_convert(const float *dq_acc, void *dq, long long rows, int d, int H,
                               int total_q, int half, cudaStream_t s) {
  // d is 32, 64 or 128: d / 8 = 1 << chunk_shift chunks per row.
  const int chunk_shift = d == 32 ? 2 : d == 64 ? 3 : 4;
  const int acc_d = d < 64 ? 64 : d;
  const long long n = rows << chunk_shift;
  const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
  if (total_q > 0)
    fa_bwd_convert_kernel<true><<<blocks, 256, 0, s>>>(dq_acc, dq, rows, chunk_shift, acc_d, H,
                                                       total_q, half);
  else
    fa_bwd_convert_kernel<false><<<blocks, 256, 0, s>>>(dq_acc, dq, rows, chunk_shift, acc_d, H,
                                                        0, half);
  return cudaGetLastError();
}

}  // namespace fa
