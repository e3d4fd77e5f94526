// bf16 tree attention on the tcgen05 tensor cores (placeholder until the kernel lands).
#include "common.cuh"

namespace spec {
size_t attention_tc_workspace_size(const spec_attn_params*) { return 256; }
spec_status_t launch_attention_tc(const spec_attn_params*, void*, size_t, cudaStream_t) {
  return SPEC_ERR_UNSUPPORTED;
}
}  // namespace spec
