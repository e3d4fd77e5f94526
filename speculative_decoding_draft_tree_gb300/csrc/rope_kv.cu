// spec_tree_rope_kv_write: rotary position embedding of the tree's q and k at the position ids a
// tree build produced, and the tree's K/V written into the paged slots the attention step reads
// (for callers that build the tree themselves; spec_tree_build_rope_kv_write fuses both).
//
// One CTA per tree node.  Every 16-byte vector of the node's q rows, new k rows and new v rows is
// loaded first (the loads depend on the node index only), while the CTA finds the node's request
// (a parallel scan of node_offset), checks that all of the request's tree slots map into the
// block pool, and turns each pair's angle into (cos, sin) once for all heads.
#include "rope.cuh"

namespace spec {

constexpr int kRopeThreads = 256;
constexpr int kRopeIter = 8;   // items in flight per thread

spec_status_t make_rope_dev(const spec_rope_params* p, RopeDev* d) {
  if (!p) return SPEC_ERR_INVALID_ARG;
  if (p->dtype != SPEC_F32 && p->dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (p->B < 1 || p->N < 0 || p->H_q < 1 || p->H_kv < 1 || p->head_dim < 1 ||
      p->block_size < 1 || p->num_blocks < 1 || p->max_blocks_per_req < 1)
    return SPEC_ERR_INVALID_ARG;
  if (!(p->base > 0.0) || !std::isfinite(p->base)) return SPEC_ERR_INVALID_ARG;
  const int es = p->dtype == SPEC_BF16 ? 2 : 4;
  const int epv = 16 / es;
  const int rd = p->rotary_dim;
  if ((p->head_dim * es) % 16 || rd < 2 || rd > p->head_dim || rd % 2) return SPEC_ERR_INVALID_ARG;
  // rotated pairs must not straddle 16-byte vectors
  if (p->interleaved ? rd % epv : (rd / 2) % epv) return SPEC_ERR_UNSUPPORTED;
  if (rd / 2 > kRopeMaxPairs) return SPEC_ERR_UNSUPPORTED;
  if (!p->node_offset || !p->prefix_len || !p->req_status) return SPEC_ERR_INVALID_ARG;
  if (p->N > 0) {
    const void* bufs[] = {p->q_in, p->q_out, p->k_new, p->v_new, p->k_cache, p->v_cache};
    for (const void* b : bufs)
      if (!b || !aligned16(b)) return SPEC_ERR_INVALID_ARG;
    if (!p->block_table || !p->pos_id) return SPEC_ERR_INVALID_ARG;
  }
  d->q_in = static_cast<const char*>(p->q_in);
  d->q_out = static_cast<char*>(p->q_out);
  d->k_new = static_cast<const char*>(p->k_new);
  d->v_new = static_cast<const char*>(p->v_new);
  d->k_cache = static_cast<char*>(p->k_cache);
  d->v_cache = static_cast<char*>(p->v_cache);
  d->block_table = p->block_table;
  d->prefix_len = p->prefix_len;
  d->node_offset = p->node_offset;
  d->pos_id = p->pos_id;
  d->req_status = p->req_status;
  d->B = p->B;
  d->N = p->N;
  d->H_q = p->H_q;
  d->H_kv = p->H_kv;
  d->row_bytes = p->head_dim * es;
  d->d_vecs = d->row_bytes / 16;
  d->rot_vecs = rd / epv;
  d->items_qk = p->interleaved ? d->d_vecs : d->d_vecs - d->rot_vecs / 2;
  d->items_node = (d->H_q + d->H_kv) * d->items_qk + d->H_kv * d->d_vecs;
  d->rot_pairs = rd / 2;
  d->interleaved = p->interleaved ? 1 : 0;
  d->bs = p->block_size;
  d->num_blocks = p->num_blocks;
  d->max_blocks = p->max_blocks_per_req;
  d->bf16 = p->dtype == SPEC_BF16 ? 1 : 0;
  for (int j = 0; j < kRopeMaxPairs; ++j)
    d->theta[j] = j < d->rot_pairs ? std::pow(p->base, -2.0 * j / rd) : 0.0;
  return SPEC_OK;
}

template <typename T>
__global__ void __launch_bounds__(kRopeThreads)
tree_rope_kv_kernel(const __grid_constant__ RopeDev a) {
  __shared__ float2 s_cs[kRopeMaxPairs];
  __shared__ int s_req;
  __shared__ int s_o, s_T, s_P, s_pos, s_status;
  pdl_wait();
  pdl_trigger();
  const int n = blockIdx.x;
  const int t = threadIdx.x;
  const int total = a.items_node;

  // 1. issue the node's first loads (they depend on n only); the destination is not known yet
  uint4 x0[kRopeIter], x1[kRopeIter];
#pragma unroll
  for (int u = 0; u < kRopeIter; ++u) {
    const int f = u * kRopeThreads + t;
    if (f < total) rope_load(rope_item(a, n, f, 0), x0[u], x1[u]);
  }

  // 2. the owning request: the one r with node_offset[r] <= n < node_offset[r+1].  A request
  //    whose range is empty or inverted cannot match, so at most one r does.
  if (t == 0) s_req = -1;
  __syncthreads();
  for (int r = t; r < a.B; r += kRopeThreads) {
    const int o = a.node_offset[r], e = a.node_offset[r + 1];
    if (o <= n && n < e) s_req = r;
  }
  __syncthreads();
  const int r = s_req;
  if (r < 0) return;   // node past the last request
  if (t == 0) {
    s_o = a.node_offset[r];
    s_T = a.node_offset[r + 1] - s_o;
    s_P = a.prefix_len[r];
    s_pos = a.pos_id[n];
    s_status = a.req_status[r];
  }
  __syncthreads();
  const int o = s_o, T_r = s_T, P = s_P, pos = s_pos;
  if (s_status != 0 || pos < 0 || P < 0) return;   // request rejected by the tree build
  // every tree slot P .. P+T-1 of the request must map into the pool, else none is written
  {
    const int lb0 = P / a.bs, lb1 = (P + T_r - 1) / a.bs;
    bool bad = false;
    for (int lb = lb0 + t; lb <= lb1; lb += kRopeThreads) {
      if (lb >= a.max_blocks) {
        bad = true;
      } else {
        const int blk = a.block_table[size_t(r) * a.max_blocks + lb];
        bad |= blk < 0 || blk >= a.num_blocks;
      }
    }
    if (__syncthreads_or(bad)) {
      if (t == 0 && n == o) atomicOr(&a.req_status[r], SPEC_REQ_BAD_BLOCK);
      return;
    }
  }
  const int slot = P + (n - o);
  const int blk = a.block_table[size_t(r) * a.max_blocks + slot / a.bs];
  const size_t kv_off = (size_t(blk) * a.H_kv * a.bs + slot % a.bs) * a.row_bytes;

  // 3. (cos, sin) of every pair's angle at this position
  for (int j = t; j < a.rot_pairs; j += kRopeThreads) s_cs[j] = rope_cos_sin(a, pos, j);
  __syncthreads();

  // 4. rotate and store; items past the first kRopeIter * kRopeThreads are loaded here
  for (int base = 0; base < total; base += kRopeIter * kRopeThreads) {
#pragma unroll
    for (int u = 0; u < kRopeIter; ++u) {
      const int f = base + u * kRopeThreads + t;
      if (f >= total) continue;
      const RopeItem it = rope_item(a, n, f, kv_off);
      if (base > 0) rope_load(it, x0[u], x1[u]);
      rope_store<T>(it, x0[u], x1[u], s_cs);
    }
  }
}

}  // namespace spec

extern "C" spec_status_t spec_tree_rope_kv_write(const spec_rope_params* p, spec_stream_t stream) {
  using namespace spec;
  RopeDev d;
  const spec_status_t st = make_rope_dev(p, &d);
  if (st != SPEC_OK) return st;
  if (p->N == 0) return SPEC_OK;
  cudaError_t e;
  if (d.bf16)
    e = launch_pdl(tree_rope_kv_kernel<__nv_bfloat16>, dim3(p->N), dim3(kRopeThreads), 0,
                   (cudaStream_t)stream, d);
  else
    e = launch_pdl(tree_rope_kv_kernel<float>, dim3(p->N), dim3(kRopeThreads), 0,
                   (cudaStream_t)stream, d);
  return launch_result(e);
}
