// fa_bwd_bf16.cu — instantiations of the tensor-core backward for bf16 inputs
// (tcgen05 kind::f16), head dims 64 and 128.
#include "fa_bwd.cuh"

namespace fa {

cudaError_t launch_bwd_bf16_d64(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                         const CUtensorMap &dout, const BwdParams &p, int B, int causal,
                         cudaStream_t s) {
  return launch_bwd<64, false>(q, k, v, dout, p, B, causal, s);
}

cudaError_t launch_bwd_bf16_d128(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                          const CUtensorMap &dout, const BwdParams &p, int B, int causal,
                          cudaStream_t s) {
  return launch_bwd<128, false>(q, k, v, dout, p, B, causal, s);
}

}  // namespace fa
