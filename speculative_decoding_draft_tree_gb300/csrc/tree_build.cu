// spec_tree_build: flattened draft tree -> depth, position ids, ancestor mask, internal flags.
//
// Source: "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的验证——树形掩码 -- the tree is flattened
// ([root, A, B, C, D, E]) and each token attends only to its ancestors; the page's mask table
// has a 1 at (row i, column j) iff j is i or an ancestor of i; mask, KV cache and position ids
// must follow the tree (position id = prefix length + depth here).
//
// One CTA per request.  The request's parent array is staged in shared memory; thread i walks
// node i's parent chain (at most T_max - 1 steps) building its mask row in registers, so no
// thread waits on another.  Validation happens first, block-wide; req_status[r] is (re)written
// here -- 0, or the SPEC_REQ_* bit of a bad request, whose outputs become -1 / 0.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "rope.cuh"

namespace spec {

static thread_local int g_last_cuda_error = 0;
void set_last_cuda_error(cudaError_t e) { g_last_cuda_error = int(e); }

static std::atomic<unsigned long long> g_kernel_launches{0};
void count_launch() { g_kernel_launches.fetch_add(1, std::memory_order_relaxed); }

int sm_count_current_device() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

constexpr int kTreeThreads = SPEC_MAX_TREE;  // one thread per possible node
constexpr int kMaxWords = SPEC_MAX_TREE / 32;

struct TreeArgs {
  const int32_t* parent;
  const int32_t* node_offset;
  const int32_t* prefix_len;
  int32_t N, T_max, W;
  int32_t* depth;
  int32_t* pos_id;
  uint32_t* anc_mask;
  uint8_t* is_internal;
  int32_t* req_status;
};

struct TreeSmem {
  int16_t par[SPEC_MAX_TREE];
  int16_t depth[SPEC_MAX_TREE];
  uint8_t has_child[SPEC_MAX_TREE];
};

// Request r (nodes o .. e-1): validate its size and parent array, stage the parents in shared
// memory and give every node its depth (thread i walks node i's chain, at most T_max - 1 steps,
// building its mask row in registers, so no thread waits on another).  With kWrite the outputs
// depth / pos_id / anc_mask / is_internal are stored (-1 / 0 for a bad request).  Returns the
// request's status bits (0 = valid), the same in every thread; s.depth is valid when it is 0.
template <bool kWrite>
__device__ int build_request_tree(const TreeArgs& a, int r, int o, int e, TreeSmem& s) {
  const int i = threadIdx.x;
  const int T = e - o;
  // size check: the range must be a valid window of [0, N) with 1 <= T <= T_max
  const bool size_ok = (o >= 0) && (e <= a.N) && (T >= 1) && (T <= a.T_max);
  int p = -2;
  if (size_ok && i < T) p = a.parent[o + i];
  const bool bad_par = size_ok && i < T && (i == 0 ? (p != -1) : (p < 0 || p >= i));
  const int any_bad = __syncthreads_or(bad_par);
  if (!size_ok || any_bad) {
    if (kWrite && size_ok && i < T) {
      a.depth[o + i] = -1;
      a.pos_id[o + i] = -1;
      a.is_internal[o + i] = 0;
      for (int w = 0; w < a.W; ++w) a.anc_mask[size_t(o + i) * a.W + w] = 0u;
    }
    return size_ok ? SPEC_REQ_BAD_PARENT : SPEC_REQ_BAD_SIZE;
  }
  if (i < T) {
    s.par[i] = int16_t(p);
    s.has_child[i] = 0;
  }
  __syncthreads();
  if (i < T && i > 0) s.has_child[p] = 1;  // benign race: every writer stores 1
  if (i < T) {
    uint32_t words[kMaxWords];
#pragma unroll
    for (int w = 0; w < kMaxWords; ++w) words[w] = 0u;
    int d = 0;
    int j = i;
    while (j != -1) {  // terminates: parent[j] < j, validated above
      if (kWrite) {
#pragma unroll
        for (int w = 0; w < kMaxWords; ++w)
          if ((j >> 5) == w) words[w] |= 1u << (j & 31);
      }
      j = s.par[j];
      ++d;
    }
    s.depth[i] = int16_t(d - 1);
    if (kWrite) {
      a.depth[o + i] = d - 1;
      a.pos_id[o + i] = a.prefix_len[r] + d - 1;
#pragma unroll
      for (int w = 0; w < kMaxWords; ++w)
        if (w < a.W) a.anc_mask[size_t(o + i) * a.W + w] = words[w];
    }
  }
  __syncthreads();
  if (kWrite && i < T) a.is_internal[o + i] = s.has_child[i];
  return 0;
}

__global__ void __launch_bounds__(kTreeThreads) tree_build_kernel(const TreeArgs a) {
  __shared__ TreeSmem s;
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int st = build_request_tree<true>(a, r, a.node_offset[r], a.node_offset[r + 1], s);
  if (threadIdx.x == 0) a.req_status[r] = st;
}

// ------------------------------------------------------------------------------------------
// Tree build fused with the step before attention (rotary embedding of the tree's q and k at
// pos = prefix + depth, and the tree K/V written into its cache slots).  Grid (request, slice):
// every CTA rebuilds its request's tree in shared memory (the parent array is a few hundred
// bytes) and handles nodes [slice * npc, slice * npc + npc) of it; slice 0 also stores the tree
// outputs and the request's status.  The node rows' loads, the parent loads and the block-table
// loads are all issued before the first wait, so the kernel costs about two memory round trips
// beyond its data movement -- and no launch of its own between the tree build and attention.
constexpr int kFusedIter = 8;    // items in flight per thread
constexpr int kFusedNodes = 4;   // nodes per CTA at most

template <typename Elem>
__global__ void __launch_bounds__(kTreeThreads)
tree_build_rope_kernel(const TreeArgs ta, const __grid_constant__ RopeDev a, int npc) {
  __shared__ TreeSmem s;
  __shared__ float2 s_cs[kFusedNodes][kRopeMaxPairs];
  __shared__ int s_blk[SPEC_MAX_TREE + 1];
  // Dependents are released only after the stores (below): released at the start, the small
  // attention kernel's CTAs were placed while this kernel still ran and the step lost ~20 us.
  pdl_wait();
  const int r = blockIdx.x;
  const int t = threadIdx.x;
  const int o = ta.node_offset[r], e = ta.node_offset[r + 1];
  const int P = ta.prefix_len[r];
  const int T = e - o;
  const bool size_ok = (o >= 0) && (e <= ta.N) && (T >= 1) && (T <= ta.T_max);
  const int n0 = o + int(blockIdx.y) * npc;
  const int nn = size_ok ? max(0, min(npc, e - n0)) : 0;   // nodes of this CTA
  const int total = nn * a.items_node;
  if (nn == 0 && blockIdx.y != 0) {   // a slice past the tree: nothing to store
    pdl_trigger();
    return;
  }

  // 1. the CTA's node rows (addresses depend on the node only)
  uint4 x0[kFusedIter], x1[kFusedIter];
#pragma unroll
  for (int u = 0; u < kFusedIter; ++u) {
    const int f = u * kTreeThreads + t;
    if (f < total) {
      const int k = f / a.items_node;
      rope_load(rope_item(a, n0 + k, f - k * a.items_node, 0), x0[u], x1[u]);
    }
  }
  // 2. the block-table entries of the request's tree slots P .. P+T-1 (at most T + 1 entries)
  const int lb0 = P >= 0 ? P / a.bs : 0;
  const int nlb = (size_ok && P >= 0) ? (P + T - 1) / a.bs - lb0 + 1 : 0;
  bool bad_blk = false;
  if (t < nlb) {
    const int lb = lb0 + t;
    if (lb >= a.max_blocks) {
      bad_blk = true;
    } else {
      const int blk = a.block_table[size_t(r) * a.max_blocks + lb];
      bad_blk = blk < 0 || blk >= a.num_blocks;
      s_blk[t] = blk;
    }
  }
  // 3. the tree (slice 0 stores its outputs)
  int st = blockIdx.y == 0 ? build_request_tree<true>(ta, r, o, e, s)
                           : build_request_tree<false>(ta, r, o, e, s);
  if (__syncthreads_or(bad_blk) && st == 0) st = SPEC_REQ_BAD_BLOCK;
  if (blockIdx.y == 0 && t == 0) ta.req_status[r] = st;
  if (st != 0 || nn == 0 || P < 0) {   // uniform across the CTA
    pdl_trigger();
    return;
  }

  // 4. (cos, sin) per pair of each of the CTA's nodes
  for (int idx = t; idx < nn * a.rot_pairs; idx += kTreeThreads) {
    const int k = idx / a.rot_pairs;
    const int j = idx - k * a.rot_pairs;
    s_cs[k][j] = rope_cos_sin(a, P + s.depth[n0 + k - o], j);
  }
  __syncthreads();

  // 5. rotate and store; items past the first kFusedIter * kTreeThreads are loaded here
  for (int base = 0; base < total; base += kFusedIter * kTreeThreads) {
#pragma unroll
    for (int u = 0; u < kFusedIter; ++u) {
      const int f = base + u * kTreeThreads + t;
      if (f >= total) continue;
      const int k = f / a.items_node;
      const int slot = P + (n0 + k - o);
      const int blk = s_blk[slot / a.bs - lb0];
      const size_t kv_off = (size_t(blk) * a.H_kv * a.bs + slot % a.bs) * a.row_bytes;
      const RopeItem it = rope_item(a, n0 + k, f - k * a.items_node, kv_off);
      if (base > 0) rope_load(it, x0[u], x1[u]);
      rope_store<Elem>(it, x0[u], x1[u], s_cs[k]);
    }
  }
  pdl_trigger();
}

}  // namespace spec

extern "C" {

const char* spec_status_string(spec_status_t s) {
  switch (s) {
    case SPEC_OK: return "SPEC_OK";
    case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
    case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
    case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
    case SPEC_ERR_TIMEOUT: return "SPEC_ERR_TIMEOUT";
    case SPEC_ERR_BAD_INPUT_DATA: return "SPEC_ERR_BAD_INPUT_DATA";
  }
  return "SPEC_ERR_UNKNOWN";
}

int spec_last_cuda_error(void) { return spec::g_last_cuda_error; }

uint64_t spec_kernel_launches(void) {
  return uint64_t(spec::g_kernel_launches.load(std::memory_order_relaxed));
}

spec_status_t spec_tree_build(const int32_t* parent, const int32_t* node_offset,
                              const int32_t* prefix_len, int32_t B, int32_t N, int32_t T_max,
                              int32_t* depth, int32_t* pos_id, uint32_t* anc_mask,
                              uint8_t* is_internal, int32_t* req_status, spec_stream_t stream) {
  if (B < 1 || N < 0 || T_max < 1 || T_max > SPEC_MAX_TREE) return SPEC_ERR_INVALID_ARG;
  if (!node_offset || !prefix_len || !req_status) return SPEC_ERR_INVALID_ARG;
  if (N > 0 && (!parent || !depth || !pos_id || !anc_mask || !is_internal))
    return SPEC_ERR_INVALID_ARG;
  spec::TreeArgs a{parent, node_offset, prefix_len, N, T_max, (T_max + 31) / 32,
                   depth, pos_id, anc_mask, is_internal, req_status};
  return spec::launch_result(spec::launch_pdl(spec::tree_build_kernel, dim3(B),
                                              dim3(spec::kTreeThreads), 0, (cudaStream_t)stream,
                                              a));
}

spec_status_t spec_tree_build_rope_kv_write(const int32_t* parent, const int32_t* node_offset,
                                            const int32_t* prefix_len, int32_t B, int32_t N,
                                            int32_t T_max, int32_t* depth, int32_t* pos_id,
                                            uint32_t* anc_mask, uint8_t* is_internal,
                                            int32_t* req_status, const spec_rope_params* rope,
                                            spec_stream_t stream) {
  using namespace spec;
  if (B < 1 || N < 0 || T_max < 1 || T_max > SPEC_MAX_TREE) return SPEC_ERR_INVALID_ARG;
  if (!node_offset || !prefix_len || !req_status || !rope) return SPEC_ERR_INVALID_ARG;
  if (N > 0 && (!parent || !depth || !pos_id || !anc_mask || !is_internal))
    return SPEC_ERR_INVALID_ARG;
  // the rope block's request arrays are this call's (NULL there means "the same")
  spec_rope_params p = *rope;
  if (p.B != B || p.N != N) return SPEC_ERR_INVALID_ARG;
  if ((p.node_offset && p.node_offset != node_offset) ||
      (p.prefix_len && p.prefix_len != prefix_len) || (p.pos_id && p.pos_id != pos_id) ||
      (p.req_status && p.req_status != req_status))
    return SPEC_ERR_INVALID_ARG;
  p.node_offset = node_offset;
  p.prefix_len = prefix_len;
  p.pos_id = pos_id;
  p.req_status = req_status;
  RopeDev d;
  const spec_status_t st = make_rope_dev(&p, &d);
  if (st != SPEC_OK) return st;
  TreeArgs a{parent, node_offset, prefix_len, N, T_max, (T_max + 31) / 32,
             depth, pos_id, anc_mask, is_internal, req_status};
  // nodes per CTA: enough CTAs to cover the SMs a few times over, at most kFusedNodes, and no
  // more than the items one pass of loads keeps in registers
  const int sms = std::max(1, sm_count_current_device());
  const long long want = 4LL * sms;
  int npc = int((static_cast<long long>(B) * T_max + want - 1) / want);
  npc = std::min({kFusedNodes, npc, kFusedIter * kTreeThreads / d.items_node});
  npc = std::max(1, npc);
  const dim3 grid(B, (T_max + npc - 1) / npc);
  cudaError_t e;
  if (d.bf16)
    e = launch_pdl(tree_build_rope_kernel<__nv_bfloat16>, grid, dim3(kTreeThreads), 0,
                   (cudaStream_t)stream, a, d, npc);
  else
    e = launch_pdl(tree_build_rope_kernel<float>, grid, dim3(kTreeThreads), 0,
                   (cudaStream_t)stream, a, d, npc);
  return launch_result(e);
}

}  // extern "C"
