// fa_splitkv.cu — merge of the key-range chunks written by the tensor-core
// kernel in split mode.
//
// Chunk s of a row holds O_s = sum_{j in s} e^{s_j - m_s} v_j / l_s and
// LSE_s = m_s + log l_s (natural log, scaled score).  The row's result is
// the online-softmax update of the forward kernel of "flash_attention_2.cu"
// (leloykun/flash-hyperbolic-attention-minimal) applied across chunks instead
// of across tiles:
//     LSE = log sum_s e^{LSE_s},   O = sum_s e^{LSE_s - LSE} O_s.
// Splitting the key range gives a grid that fills the GPU when B*H and the
// number of query tiles are small ("parallel execution of read/write
// operations (paper vs implementation)": per-head parallelism needs B*H
// around 80 or more).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>

#include "fa.h"
#include "fa_internal.h"

namespace fa {

namespace {

constexpr int kRowsPerBlock = 4;  // one warp per output row

// Number of key tiles query tile qt covers, and whether chunk s of them is
// empty (the same split rule as the tensor-core kernel).
__device__ __forceinline__ bool chunk_empty(int s, int nsp, int n_all) {
  const long long a = static_cast<long long>(s) * n_all / nsp;
  const long long b = static_cast<long long>(s + 1) * n_all / nsp;
  return a == b;
}

template <int D, int OUT>  // OUT: an fa_dtype of the output (bf16, f16 or f32)
__global__ void __launch_bounds__(32 * kRowsPerBlock)
    fa_splitkv_combine_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_lse,
                              void *__restrict__ o, float *__restrict__ lse, int BH, int Nq,
                              int n_ktiles, int nsp, int causal, unsigned *status) {
  const int lane = threadIdx.x & 31;
  const long long row_g = static_cast<long long>(blockIdx.x) * kRowsPerBlock + (threadIdx.x >> 5);
  if (row_g >= static_cast<long long>(BH) * Nq) return;  // whole warp
  const int row = static_cast<int>(row_g % Nq);
  const int qt = row / BM;
  const int n_all = causal ? min(qt + 1, n_ktiles) : n_ktiles;
  const size_t plane = static_cast<size_t>(BH) * Nq;  // rows per chunk

  // LSE = log sum_s e^{LSE_s} over the non-empty chunks (at most 64: two per lane).
  const long long ws_rows = static_cast<long long>(nsp) * plane;  // debug index checks
  float l0 = -INFINITY, l1 = -INFINITY;
  if (lane < nsp && !chunk_empty(lane, nsp, n_all) &&
      FA_IN(status, lane * plane + row_g, 1, ws_rows))
    l0 = ws_lse[lane * plane + row_g];
  if (lane + 32 < nsp && !chunk_empty(lane + 32, nsp, n_all) &&
      FA_IN(status, (lane + 32) * plane + row_g, 1, ws_rows))
    l1 = ws_lse[(lane + 32) * plane + row_g];
  float m = fmaxf(l0, l1);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float sum = expf(l0 - m) + expf(l1 - m);  // exp(-inf) = 0 for empty chunks
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float L = m + logf(sum);

  // O = sum_s e^{LSE_s - LSE} O_s; lane handles columns lane + 32 i.
  float acc[D / 32];
#pragma unroll
  for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
  for (int s = 0; s < nsp; ++s) {
    if (chunk_empty(s, nsp, n_all)) continue;  // uniform across the warp
    if (!FA_IN(status, (s * plane + row_g) * D, D, ws_rows * D)) continue;
    const float w = expf(ws_lse[s * plane + row_g] - L);
    const float *src = ws_o + (s * plane + row_g) * D;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(w, src[lane + 32 * i], acc[i]);
  }
  const size_t obase = static_cast<size_t>(row_g) * D;
  if (!FA_IN(status, obase, D, static_cast<long long>(plane) * D)) return;
#pragma unroll
  for (int i = 0; i < D / 32; ++i) {
    const size_t idx = obase + lane + 32 * i;
    if constexpr (OUT == FA_DTYPE_BF16)
      static_cast<__nv_bfloat16 *>(o)[idx] = __float2bfloat16_rn(acc[i]);
    else if constexpr (OUT == FA_DTYPE_F16)
      static_cast<__half *>(o)[idx] = __float2half_rn(acc[i]);
    else
      static_cast<float *>(o)[idx] = acc[i];
  }
  if (lane == 0) lse[row_g] = L;
}

template <int D, int OUT>
cudaError_t launch_combine(const float *ws_o, const float *ws_lse, void *o, float *lse, int BH,
                           int Nq, int n_ktiles, int nsp, int causal, unsigned *status,
                           cudaStream_t s) {
  const long long rows = static_cast<long long>(BH) * Nq;
  const unsigned blocks = static_cast<unsigned>((rows + kRowsPerBlock - 1) / kRowsPerBlock);
  fa_splitkv_combine_kernel<D, OUT><<<blocks, 32 * kRowsPerBlock, 0, s>>>(
      ws_o, ws_lse, o, lse, BH, Nq, n_ktiles, nsp, causal, status);
  return cudaGetLastError();
}

}  // namespace

template <int D>
cudaError_t launch_combine_d(const float *ws_o, const float *ws_lse, void *o, float *lse, int BH,
                             int Nq, int n_ktiles, int nsp, int causal, int dtype,
                             unsigned *status, cudaStream_t s) {
  if (dtype == FA_DTYPE_BF16)
    return launch_combine<D, FA_DTYPE_BF16>(ws_o, ws_lse, o, lse, BH, Nq, n_ktiles, nsp, causal, status, s);
  if (dtype == FA_DTYPE_F16)
    return launch_combine<D, FA_DTYPE_F16>(ws_o, ws_lse, o, lse, BH, Nq, n_ktiles, nsp, causal, status, s);
  return launch_combine<D, FA_DTYPE_F32>(ws_o, ws_lse, o, lse, BH, Nq, n_ktiles, nsp, causal, status, s);
}

cudaError_t launch_splitkv_combine(const float *ws_o, const float *ws_lse, void *o, float *lse,
                                   int BH, int Nq, int d, int n_ktiles, int nsp, int causal,
                                   int dtype, unsigned *status, cudaStream_t s) {
  if (d == 32)
    return launch_combine_d<32>(ws_o, ws_lse, o, lse, BH, Nq, n_ktiles, nsp, causal, dtype, status, s);
  if (d == 64)
    return launch_combine_d<64>(ws_o, ws_lse, o, lse, BH, Nq, n_ktiles, nsp, causal, dtype, status, s);
  if (d == 128)
    return launch_combine_d<128>(ws_o, ws_lse, o, lse, BH, Nq, n_ktiles, nsp, causal, dtype, status, s);
  return launch_combine_d<256>(ws_o, ws_lse, o, lse, BH, Nq, n_ktiles, nsp, causal, dtype, status, s);
}

}  // namespace fa
