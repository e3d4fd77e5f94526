// fp32 tree attention on the CUDA cores (the fp32 path of spec_tree_attention).
//
// Sources: "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的验证——树形掩码 (ancestor mask over the
// flattened tree, KV cache and position ids adapted to the tree); "万字综述 10+ 种 LLM 投机采样推理加速
// 方案" 5.2 (tree-based parallel decoding shares the prefix through the mask).
//
// fp32 inputs rule out the bf16 tensor-core path (a TF32 contraction would not meet an fp32
// tolerance), and the fp32 workloads are small (a chain of a few tokens over a short prefix), so
// this is a plain kernel: one warp per (node, query head); lanes split head_dim, every key's
// score is a warp reduction, softmax is online in fp32.
#include <math.h>

#include "common.cuh"

namespace spec {

struct AttnF32Dev {
  const float* q;
  const float* k;
  const float* v;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* node_offset;
  const uint32_t* anc;
  float* o;
  float* lse;
  int32_t* req_status;
  int32_t B, N, H_q, H_kv, d, bs, num_blocks, max_blocks, W, T_max;
  float scale;
};

__global__ void __launch_bounds__(128) attention_f32_kernel(AttnF32Dev a) {
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long pair = long(blockIdx.x) * 4 + warp;
  if (pair >= long(a.N) * a.H_q) return;
  const int n = int(pair / a.H_q), h = int(pair % a.H_q);
  // request owning node n
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.node_offset[mid] <= n) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  if (a.req_status[r] != 0) return;
  const int o = a.node_offset[r];
  const int T = a.node_offset[r + 1] - o;
  const int P = a.prefix_len[r];
  const int kvh = h / (a.H_q / a.H_kv);
  const int kv_len = P + T;
  const int nblk = (kv_len + a.bs - 1) / a.bs;
  if (nblk > a.max_blocks) {
    if (lane == 0) atomicOr(&a.req_status[r], SPEC_REQ_BAD_BLOCK);
    return;
  }
  const int32_t* table = a.block_table + size_t(r) * a.max_blocks;
  for (int b = lane; b < nblk; b += 32) {
    const int pb = table[b];
    if (pb < 0 || pb >= a.num_blocks) atomicOr(&a.req_status[r], SPEC_REQ_BAD_BLOCK);
  }
  __syncwarp();
  if (a.req_status[r] & SPEC_REQ_BAD_BLOCK) return;
  constexpr int kMaxPerLane = 4;  // head_dim <= 128
  float qv[kMaxPerLane], acc[kMaxPerLane];
  const float* qrow = a.q + (size_t(n) * a.H_q + h) * a.d;
#pragma unroll
  for (int e = 0; e < kMaxPerLane; ++e) {
    const int c = lane + 32 * e;
    qv[e] = c < a.d ? qrow[c] : 0.f;
    acc[e] = 0.f;
  }
  const uint32_t* anc = a.anc + size_t(n) * a.W;
  float m = -INFINITY, l = 0.f;
  for (int j = 0; j < kv_len; ++j) {
    if (j >= P) {
      const int t = j - P;
      if (!((anc[t >> 5] >> (t & 31)) & 1u)) continue;
    }
    const int pb = table[j / a.bs];
    const size_t off = ((size_t(pb) * a.H_kv + kvh) * a.bs + (j % a.bs)) * a.d;
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < kMaxPerLane; ++e) {
      const int c = lane + 32 * e;
      if (c < a.d) part = fmaf(qv[e], a.k[off + c], part);
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) part += __shfl_xor_sync(0xffffffffu, part, s);
    const float sc = part * a.scale;
    const float mn = fmaxf(m, sc);
    const float corr = expf(m - mn);
    const float pj = expf(sc - mn);
    l = l * corr + pj;
#pragma unroll
    for (int e = 0; e < kMaxPerLane; ++e) {
      const int c = lane + 32 * e;
      const float vv = c < a.d ? a.v[off + c] : 0.f;
      acc[e] = acc[e] * corr + pj * vv;
    }
    m = mn;
  }
  float* orow = a.o + (size_t(n) * a.H_q + h) * a.d;
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < kMaxPerLane; ++e) {
    const int c = lane + 32 * e;
    if (c < a.d) orow[c] = acc[e] * inv;
  }
  if (a.lse && lane == 0) a.lse[size_t(n) * a.H_q + h] = m + logf(l);
}

spec_status_t launch_attention_f32(const spec_attn_params* p, cudaStream_t s) {
  if (p->head_dim > 128 || p->head_dim % 4) return SPEC_ERR_UNSUPPORTED;
  AttnF32Dev d;
  d.q = static_cast<const float*>(p->q);
  d.k = static_cast<const float*>(p->k_cache);
  d.v = static_cast<const float*>(p->v_cache);
  d.block_table = p->block_table;
  d.prefix_len = p->prefix_len;
  d.node_offset = p->node_offset;
  d.anc = p->anc_mask;
  d.o = static_cast<float*>(p->o);
  d.lse = p->lse;
  d.req_status = p->req_status;
  d.B = p->B; d.N = p->N; d.H_q = p->H_q; d.H_kv = p->H_kv; d.d = p->head_dim;
  d.bs = p->block_size; d.num_blocks = p->num_blocks; d.max_blocks = p->max_blocks_per_req;
  d.W = (p->T_max + 31) / 32; d.T_max = p->T_max;
  d.scale = p->scale > 0.f ? p->scale : 1.f / sqrtf(float(p->head_dim));
  const long pairs = long(p->N) * p->H_q;
  if (pairs == 0) return SPEC_OK;
  const unsigned grid = unsigned((pairs + 3) / 4);
  return launch_result(launch_pdl(attention_f32_kernel, dim3(grid), dim3(128), 0, s, d));
}

}  // namespace spec
