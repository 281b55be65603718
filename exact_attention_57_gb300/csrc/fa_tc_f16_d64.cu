// fa_tc_f16_d64.cu — instantiation of the tensor-core forward for head dim 64,
// fp16 inputs (tcgen05 kind::f16).
#include "fa_tc.cuh"

namespace fa {

cudaError_t launch_tc_f16_d64(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                              const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                              int B, int causal, cudaStream_t s) {
  return launch_tc<64, false, true>(q, k, v, o, klo, p, B, causal, s);
}

}  // namespace fa
