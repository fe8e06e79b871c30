// mla_decode.cu -- placeholder until the decode kernel lands.
#include "common.cuh"

size_t mla_workspace_bytes(int B, int Hq, int max_blocks, int num_sms, int pages_per_split) {
  (void)B; (void)Hq; (void)max_blocks; (void)num_sms; (void)pages_per_split;
  return 16;
}

cudaError_t launch_mla_decode(const MlaArgs& a, cudaStream_t s) {
  (void)a; (void)s;
  attn_set_error("mla_decode: not built yet");
  return cudaErrorNotSupported;
}
