// spec_tree_attention / spec_attention_workspace_size: argument validation and dispatch to the
// fp32 CUDA-core kernel or the bf16 tcgen05 kernel.
#include "common.cuh"

namespace spec {
spec_status_t launch_attention_f32(const spec_attn_params* p, cudaStream_t s);
size_t attention_tc_workspace_size(const spec_attn_params* p);
spec_status_t launch_attention_tc(const spec_attn_params* p, void* ws, size_t ws_bytes,
                                  cudaStream_t s);

static spec_status_t check_attn(const spec_attn_params* p) {
  if (!p) return SPEC_ERR_INVALID_ARG;
  if (p->dtype != SPEC_F32 && p->dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (p->B < 1 || p->N < 0 || p->T_max < 1 || p->T_max > SPEC_MAX_TREE) return SPEC_ERR_INVALID_ARG;
  if (p->H_q < 1 || p->H_kv < 1 || p->H_q % p->H_kv || p->head_dim < 1 || p->block_size < 1 ||
      p->num_blocks < 1 || p->max_blocks_per_req < 1)
    return SPEC_ERR_INVALID_ARG;
  if (!p->block_table || !p->prefix_len || !p->node_offset || !p->req_status)
    return SPEC_ERR_INVALID_ARG;
  if (p->N > 0 && (!p->q || !p->k_cache || !p->v_cache || !p->o || !p->anc_mask))
    return SPEC_ERR_INVALID_ARG;
  if (p->N > 0 && (!aligned16(p->q) || !aligned16(p->k_cache) || !aligned16(p->v_cache) ||
                   !aligned16(p->o)))
    return SPEC_ERR_INVALID_ARG;
  const int es = p->dtype == SPEC_BF16 ? 2 : 4;
  if ((p->head_dim * es) % 16) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}
}  // namespace spec

extern "C" {

size_t spec_attention_workspace_size(const spec_attn_params* p) {
  if (spec::check_attn(p) != SPEC_OK) return 0;
  if (p->dtype == SPEC_F32) return 256;
  return spec::attention_tc_workspace_size(p);
}

spec_status_t spec_tree_attention(const spec_attn_params* p, void* workspace, size_t ws_bytes,
                                  spec_stream_t stream) {
  using namespace spec;
  const spec_status_t st = check_attn(p);
  if (st != SPEC_OK) return st;
  if (p->N == 0) return SPEC_OK;
  if (p->dtype == SPEC_F32) return launch_attention_f32(p, (cudaStream_t)stream);
  return launch_attention_tc(p, workspace, ws_bytes, (cudaStream_t)stream);
}

}  // extern "C"
