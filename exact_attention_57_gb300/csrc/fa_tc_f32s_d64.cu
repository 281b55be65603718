// fa_tc_f32s_d64.cu — instantiation of the tensor-core forward for head dim 64,
// fp32 inputs with staged operands: scores as three bf16 products of the
// split Q and K (kind::f16), P V in tf32 (kind::tf32).
#include "fa_tc.cuh"

namespace fa {

cudaError_t launch_tc_f32s_d64(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                               const CUtensorMap &o, const CUtensorMap &klo, const TcParams &p,
                               int B, int causal, cudaStream_t s) {
  return launch_tc<64, true, false, true>(q, k, v, o, klo, p, B, causal, s);
}

}  // namespace fa
