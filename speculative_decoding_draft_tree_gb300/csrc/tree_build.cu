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
#include <mutex>

#include "common.cuh"

namespace spec {

static thread_local int g_last_cuda_error = 0;
void set_last_cuda_error(cudaError_t e) { g_last_cuda_error = int(e); }

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

__global__ void __launch_bounds__(kTreeThreads)
tree_build_kernel(const int32_t* __restrict__ parent, const int32_t* __restrict__ node_offset,
                  const int32_t* __restrict__ prefix_len, int32_t N, int32_t T_max, int32_t W,
                  int32_t* __restrict__ depth, int32_t* __restrict__ pos_id,
                  uint32_t* __restrict__ anc_mask, uint8_t* __restrict__ is_internal,
                  int32_t* __restrict__ req_status) {
  __shared__ int16_t s_par[SPEC_MAX_TREE];
  __shared__ uint8_t s_has_child[SPEC_MAX_TREE];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int i = threadIdx.x;
  const int o = node_offset[r];
  const int e = node_offset[r + 1];
  const int T = e - o;
  // size check: the range must be a valid window of [0, N) with 1 <= T <= T_max
  const bool size_ok = (o >= 0) && (e <= N) && (T >= 1) && (T <= T_max);
  int p = -2;
  if (size_ok && i < T) p = parent[o + i];
  const bool bad_par = size_ok && i < T && (i == 0 ? (p != -1) : (p < 0 || p >= i));
  const int any_bad = __syncthreads_or(bad_par);
  if (i == 0) req_status[r] = size_ok ? (any_bad ? SPEC_REQ_BAD_PARENT : 0) : SPEC_REQ_BAD_SIZE;
  if (!size_ok || any_bad) {
    if (size_ok && i < T) {
      depth[o + i] = -1;
      pos_id[o + i] = -1;
      is_internal[o + i] = 0;
      for (int w = 0; w < W; ++w) anc_mask[size_t(o + i) * W + w] = 0u;
    }
    return;
  }
  if (i < T) {
    s_par[i] = int16_t(p);
    s_has_child[i] = 0;
  }
  __syncthreads();
  if (i < T && i > 0) s_has_child[p] = 1;  // benign race: every writer stores 1
  if (i < T) {
    uint32_t words[kMaxWords];
#pragma unroll
    for (int w = 0; w < kMaxWords; ++w) words[w] = 0u;
    int d = 0;
    int j = i;
    while (j != -1) {  // terminates: parent[j] < j, validated above
#pragma unroll
      for (int w = 0; w < kMaxWords; ++w)
        if ((j >> 5) == w) words[w] |= 1u << (j & 31);
      j = s_par[j];
      ++d;
    }
    depth[o + i] = d - 1;
    pos_id[o + i] = prefix_len[r] + d - 1;
#pragma unroll
    for (int w = 0; w < kMaxWords; ++w)
      if (w < W) anc_mask[size_t(o + i) * W + w] = words[w];
  }
  __syncthreads();
  if (i < T) is_internal[o + i] = s_has_child[i];
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

spec_status_t spec_tree_build(const int32_t* parent, const int32_t* node_offset,
                              const int32_t* prefix_len, int32_t B, int32_t N, int32_t T_max,
                              int32_t* depth, int32_t* pos_id, uint32_t* anc_mask,
                              uint8_t* is_internal, int32_t* req_status, spec_stream_t stream) {
  if (B < 1 || N < 0 || T_max < 1 || T_max > SPEC_MAX_TREE) return SPEC_ERR_INVALID_ARG;
  if (!node_offset || !prefix_len || !req_status) return SPEC_ERR_INVALID_ARG;
  if (N > 0 && (!parent || !depth || !pos_id || !anc_mask || !is_internal))
    return SPEC_ERR_INVALID_ARG;
  const int W = (T_max + 31) / 32;
  return spec::launch_result(spec::launch_pdl(
      spec::tree_build_kernel, dim3(B), dim3(spec::kTreeThreads), 0, (cudaStream_t)stream,
      parent, node_offset, prefix_len, N, T_max, W, depth, pos_id, anc_mask, is_internal,
      req_status));
}

}  // extern "C"
