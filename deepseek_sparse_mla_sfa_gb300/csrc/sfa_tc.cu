// sfa_tc.cu -- tcgen05 / TMA path of sparse MLA decode (sm_103a).
#include "sfa_internal.h"

namespace sfa {

bool tc_supports(int h, int block_size) { (void)h; (void)block_size; return false; }

size_t tc_workspace_bytes(int T, int h, int top_k, int n_splits) {
  (void)T; (void)h; (void)top_k; (void)n_splits;
  return 0;
}

int tc_launches(int T, int h, int top_k, int n_splits) {
  (void)T; (void)h; (void)top_k; (void)n_splits;
  return 1;
}

cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t stream) {
  (void)p; (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace sfa
