// fp32 tree attention on the CUDA cores (the fp32 path of spec_tree_attention).
//
// Sources: "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的验证——树形掩码 (ancestor mask over the
// flattened tree, KV cache and position ids adapted to the tree); "万字综述 10+ 种 LLM 投机采样推理加速
// 方案" 5.2 (tree-based parallel decoding shares the prefix through the mask).
//
// fp32 inputs rule out the bf16 tensor-core path (a TF32 contraction would not meet an fp32
// tolerance), and the fp32 workloads are small (a chain of a few tokens over a short prefix), so
// this is a plain kernel, built for latency: one CTA of 128 threads per (node, query head).  Keys
// go in chunks of 128, one key per thread: each thread looks its key's block up, forms the full
// dot product with the query and copies its V row into shared memory (all its loads in flight
// at once), so a chunk costs a few memory round trips instead of one per key; the chunk's
// softmax is a block reduction (online across chunks, fp32), and thread c < head_dim then
// accumulates output column c over the chunk's visible keys from shared memory.
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

constexpr int kF32Threads = 128;   // keys per chunk and threads per CTA; head_dim <= 128

__device__ __forceinline__ float block_reduce_f32(float v, float* red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, x) : v + x;
  }
  __syncthreads();   // red is reused by consecutive reductions
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kF32Threads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  return r;
}

__global__ void __launch_bounds__(kF32Threads) attention_f32_kernel(AttnF32Dev a) {
  extern __shared__ float4 sv4[];   // [kF32Threads keys][head_dim / 4 + 1]: the chunk's V rows
  __shared__ __align__(16) float sq[128];
  __shared__ float sp[kF32Threads];
  __shared__ int spb[kF32Threads];
  __shared__ float red[kF32Threads / 32];
  __shared__ int s_bad;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  const int n = int(blockIdx.x / unsigned(a.H_q)), h = int(blockIdx.x % unsigned(a.H_q));
  // request owning node n
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.node_offset[mid] <= n) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  if (a.req_status[r] != 0) return;   // uniform across the CTA
  const int o = a.node_offset[r];
  const int T = a.node_offset[r + 1] - o;
  const int P = a.prefix_len[r];
  const int kvh = h / (a.H_q / a.H_kv);
  const int kv_len = P + T;
  const int nblk = (kv_len + a.bs - 1) / a.bs;
  if (nblk > a.max_blocks) {
    if (tid == 0) atomicOr(&a.req_status[r], SPEC_REQ_BAD_BLOCK);
    return;
  }
  const int32_t* table = a.block_table + size_t(r) * a.max_blocks;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  for (int b = tid; b < nblk; b += kF32Threads) {
    const int pb = table[b];
    if (pb < 0 || pb >= a.num_blocks) s_bad = 1;
  }
  const float* qrow = a.q + (size_t(n) * a.H_q + h) * a.d;
  if (tid < a.d) sq[tid] = qrow[tid];
  __syncthreads();
  if (s_bad) {
    if (tid == 0) atomicOr(&a.req_status[r], SPEC_REQ_BAD_BLOCK);
    return;
  }
  const uint32_t* anc = a.anc + size_t(n) * a.W;
  const int d4 = a.d >> 2;
  const int vstride = d4 + 1;   // float4s per staged V row (padded against bank conflicts)
  float m = -INFINITY, l = 0.f, acc = 0.f;
  for (int c0 = 0; c0 < kv_len; c0 += kF32Threads) {
    // scores: one key per thread
    const int j = c0 + tid;
    bool vis = j < kv_len;
    if (vis && j >= P) {
      const int t = j - P;
      vis = (anc[t >> 5] >> (t & 31)) & 1u;
    }
    float sc = -INFINITY;
    int pb = -1;
    if (vis) {
      pb = table[j / a.bs];
      const size_t row = ((size_t(pb) * a.H_kv + kvh) * a.bs + (j % a.bs)) * a.d;
      const float4* krow = reinterpret_cast<const float4*>(a.k + row);
      const float4* vrow = reinterpret_cast<const float4*>(a.v + row);
      const float4* q4 = reinterpret_cast<const float4*>(sq);
      float dot = 0.f;
#pragma unroll 8
      for (int e = 0; e < d4; ++e) {
        const float4 kv = krow[e], qq = q4[e];
        sv4[tid * vstride + e] = vrow[e];
        dot = fmaf(qq.x, kv.x, dot);
        dot = fmaf(qq.y, kv.y, dot);
        dot = fmaf(qq.z, kv.z, dot);
        dot = fmaf(qq.w, kv.w, dot);
      }
      sc = dot * a.scale;
    }
    const float cmax = block_reduce_f32(sc, red, true);
    const float mn = fmaxf(m, cmax);
    const float corr = m == -INFINITY ? 0.f : expf(m - mn);
    const float pj = vis ? expf(sc - mn) : 0.f;
    sp[tid] = pj;
    spb[tid] = pb;
    const float psum = block_reduce_f32(pj, red, false);   // its barriers publish sp, spb, sv4
    l = l * corr + psum;
    m = mn;
    // output column tid: the chunk's visible keys
    if (tid < a.d) {
      const float* sv = reinterpret_cast<const float*>(sv4);
      float part = 0.f;
      const int nk = min(kF32Threads, kv_len - c0);
#pragma unroll 4
      for (int k = 0; k < nk; ++k)
        if (spb[k] >= 0) part = fmaf(sp[k], sv[k * 4 * vstride + tid], part);
      acc = acc * corr + part;
    }
    __syncthreads();   // sp, spb and sv4 are rewritten by the next chunk
  }
  if (tid < a.d) a.o[(size_t(n) * a.H_q + h) * a.d + tid] = acc / l;
  if (a.lse && tid == 0) a.lse[size_t(n) * a.H_q + h] = m + logf(l);
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
  if (pairs > 0x7fffffffL) return SPEC_ERR_UNSUPPORTED;
  const size_t dyn = sizeof(float4) * kF32Threads * size_t(p->head_dim / 4 + 1);   // <= 66 KB
  static DeviceOnce raised;
  const spec_status_t st = raise_dyn_smem_once(
      attention_f32_kernel, sizeof(float4) * kF32Threads * size_t(128 / 4 + 1), raised);
  if (st != SPEC_OK) return st;
  return launch_result(launch_pdl(attention_f32_kernel, dim3(unsigned(pairs)),
                                  dim3(kF32Threads), dyn, s, d));
}

}  // namespace spec
