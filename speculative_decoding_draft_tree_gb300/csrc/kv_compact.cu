// spec_kv_compact: commit the accepted path's K/V into contiguous cache slots, roll back the rest.
//
// Sources: "推测解码 2026" (guijiagi.com), 工程实践中的考量 / KV Cache管理 -- the K/V of rejected
// candidates is rolled back, which block (paged) caches make cheap; "【模型后训练与深度推理】9
// 推理加速：推测解码与级联推理" section 4 -- accepted tokens extend the prefix and the cache is reused.
//
// One CTA per (request, layer).  Slot P + d receives slot P + path[d] for d = 0..n_acc.  Because
// path[d] >= d (the accepted path descends one level per step and nodes are numbered
// breadth-first), copying in increasing d never overwrites a slot that a later step still has
// to read: a later step d' > d reads P + path[d'] with path[d'] >= d' > d.  The steps that move
// a row (path[d] != d; identity steps such as a fully accepted chain copy nothing) are taken in
// increasing d in groups of up to kCompactSteps: each thread takes one 16-byte position w of
// the heads' rows (w < H_kv * head_dim * es / 16, in chunks of the block size), loads its K and
// V vector of every step of the group, and after a barrier stores them -- gather semantics
// with one memory round trip per group and chunk instead of one per step (within a group
// every load precedes every store, positions of different chunks are disjoint, and groups
// follow each other in increasing d).  Slot offsets come from shared memory.
#include "common.cuh"
#include "kv_compact.cuh"

namespace spec {

constexpr int kCompactThreads = 512;
constexpr int kCompactSteps = 8;   // moving steps staged per group (K and V: 2 vectors each)

__global__ void __launch_bounds__(kCompactThreads) kv_compact_kernel(CompactDev a) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int layer = blockIdx.y;
  const int tid = threadIdx.x;
  const int P = a.prefix_len[r];
  const int na = a.n_acc[r];
  const int32_t* prow = a.path + size_t(r) * a.max_path;
  const int32_t* trow = a.block_table + size_t(r) * a.max_blocks;
  __shared__ int s_bad;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  bool ok = a.req_status[r] == 0 && na >= 0 && na < a.max_path && P >= 0;
  if (ok) {
    for (int d = tid; d <= na; d += blockDim.x) {
      const int pd = prow[d];
      bool good = (d == 0) ? (pd == 0) : (pd >= d);
      const int src = P + pd, dst = P + d;
      const int lsb = src / a.bs, ldb = dst / a.bs;
      good = good && lsb < a.max_blocks && ldb < a.max_blocks;
      int flag = good ? 0 : SPEC_REQ_BAD_PARENT;
      if (good) {
        const int sb = trow[lsb], db = trow[ldb];
        if (sb < 0 || sb >= a.num_blocks || db < 0 || db >= a.num_blocks) flag = SPEC_REQ_BAD_BLOCK;
      }
      if (flag) atomicOr(&s_bad, flag);
    }
  }
  __syncthreads();
  if (ok && s_bad) {
    if (layer == 0 && tid == 0) atomicOr(&a.req_status[r], s_bad);
    ok = false;
  }
  if (!ok) {
    if (layer == 0) {
      for (int k = tid; k < a.max_path; k += blockDim.x) {
        a.slot_map[(size_t(r) * a.max_path + k) * 2] = -1;
        a.slot_map[(size_t(r) * a.max_path + k) * 2 + 1] = -1;
      }
      if (tid == 0) {
        a.new_kv_len[r] = P;
        a.blocks_in_use[r] = (P + a.bs - 1) / a.bs;
      }
    }
    return;
  }
  const int vec_per_row = a.row_bytes / 16;
  const int per_step = a.H_kv * vec_per_row;   // vectors of one cache for one step
  const size_t head_stride = size_t(a.bs) * a.row_bytes;
  const size_t block_stride = size_t(a.H_kv) * head_stride;
  char* kb = a.k + layer * a.layer_stride_bytes;
  char* vb = a.v + layer * a.layer_stride_bytes;
  // the moving steps, in increasing d, with their source and destination slot offsets
  __shared__ int s_move[SPEC_MAX_TREE];
  __shared__ size_t s_src[SPEC_MAX_TREE], s_dst[SPEC_MAX_TREE];
  __shared__ int s_nmove;
  if (tid == 0) {
    int n = 0;
    for (int d = 1; d <= na && d < SPEC_MAX_TREE; ++d)
      if (prow[d] != d) s_move[n++] = d;
    s_nmove = n;
  }
  __syncthreads();
  const int nmove = s_nmove;
  if (nmove > 0) {
    for (int q = tid; q < nmove; q += kCompactThreads) {
      const int d = s_move[q];
      const int src = P + prow[d], dst = P + d;
      s_src[q] = size_t(trow[src / a.bs]) * block_stride + size_t(src % a.bs) * a.row_bytes;
      s_dst[q] = size_t(trow[dst / a.bs]) * block_stride + size_t(dst % a.bs) * a.row_bytes;
    }
    __syncthreads();
    for (int w0 = 0; w0 < per_step; w0 += kCompactThreads) {
      const int w = w0 + tid;
      const bool mine = w < per_step;
      const int h = mine ? w / vec_per_row : 0;
      const size_t in_row = size_t(h) * head_stride + size_t(w - h * vec_per_row) * 16;
      for (int g0 = 0; g0 < nmove; g0 += kCompactSteps) {
        const int gsteps = min(kCompactSteps, nmove - g0);
        uint4 kv[kCompactSteps][2];
  #pragma unroll
        for (int q = 0; q < kCompactSteps; ++q) {
          if (mine && q < gsteps) {
            const size_t o = s_src[g0 + q] + in_row;
            kv[q][0] = *reinterpret_cast<const uint4*>(kb + o);
            kv[q][1] = *reinterpret_cast<const uint4*>(vb + o);
          }
        }
        __syncthreads();   // every source of the group is read before any destination is written
  #pragma unroll
        for (int q = 0; q < kCompactSteps; ++q) {
          if (mine && q < gsteps) {
            const size_t o = s_dst[g0 + q] + in_row;
            *reinterpret_cast<uint4*>(kb + o) = kv[q][0];
            *reinterpret_cast<uint4*>(vb + o) = kv[q][1];
          }
        }
        __syncthreads();
      }
    }
  }
  if (layer == 0) {
    for (int k = tid; k < a.max_path; k += blockDim.x) {
      const bool in = k <= na;
      a.slot_map[(size_t(r) * a.max_path + k) * 2] = in ? P + prow[k] : -1;
      a.slot_map[(size_t(r) * a.max_path + k) * 2 + 1] = in ? P + k : -1;
    }
    if (tid == 0) {
      a.new_kv_len[r] = P + na + 1;
      a.blocks_in_use[r] = (P + na + 1 + a.bs - 1) / a.bs;
    }
  }
}

}  // namespace spec

spec_status_t spec::make_compact_dev(const spec_compact_params* p, CompactDev* d) {
  if (!p) return SPEC_ERR_INVALID_ARG;
  if (p->dtype != SPEC_F32 && p->dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (p->B < 1 || p->H_kv < 1 || p->head_dim < 1 || p->block_size < 1 || p->num_blocks < 1 ||
      p->max_blocks_per_req < 1 || p->num_layers < 1 || p->max_path < 1 || p->layer_stride < 0)
    return SPEC_ERR_INVALID_ARG;
  const int es = p->dtype == SPEC_BF16 ? 2 : 4;
  const int row_bytes = p->head_dim * es;
  if (row_bytes % 16) return SPEC_ERR_INVALID_ARG;
  if (!p->k_cache || !p->v_cache || !aligned16(p->k_cache) || !aligned16(p->v_cache))
    return SPEC_ERR_INVALID_ARG;
  if ((p->layer_stride * es) % 16) return SPEC_ERR_INVALID_ARG;
  if (!p->block_table || !p->prefix_len || !p->path || !p->n_acc || !p->req_status ||
      !p->new_kv_len || !p->slot_map || !p->blocks_in_use)
    return SPEC_ERR_INVALID_ARG;
  if (p->num_layers > 65535) return SPEC_ERR_UNSUPPORTED;
  d->k = static_cast<char*>(p->k_cache);
  d->v = static_cast<char*>(p->v_cache);
  d->layer_stride_bytes = p->layer_stride * es;
  d->block_table = p->block_table;
  d->prefix_len = p->prefix_len;
  d->path = p->path;
  d->n_acc = p->n_acc;
  d->req_status = p->req_status;
  d->new_kv_len = p->new_kv_len;
  d->slot_map = p->slot_map;
  d->blocks_in_use = p->blocks_in_use;
  d->H_kv = p->H_kv;
  d->row_bytes = row_bytes;
  d->bs = p->block_size;
  d->num_blocks = p->num_blocks;
  d->max_blocks = p->max_blocks_per_req;
  d->max_path = p->max_path;
  d->num_layers = p->num_layers;
  return SPEC_OK;
}

extern "C" spec_status_t spec_kv_compact(const spec_compact_params* p, spec_stream_t stream) {
  using namespace spec;
  CompactDev d;
  const spec_status_t st = make_compact_dev(p, &d);
  if (st != SPEC_OK) return st;
  dim3 grid(p->B, p->num_layers);
  return launch_result(
      launch_pdl(kv_compact_kernel, grid, dim3(kCompactThreads), 0, (cudaStream_t)stream, d));
}
