// spec_verify in one launch for small trees: each request's rows held on chip by a cluster.
//
// Sources: as the two-launch form (verify.cu) -- "推测解码 2026" (guijiagi.com), 数学基础：拒绝采样
// (accept with min(1, p/q), resample from relu(p - q) normalised); "【模型后训练与深度推理】9 推理
// 加速：推测解码与级联推理" 7.1, 7.2 (residual, bonus token); "投机推理算法的常见优化手段" (cnblogs
// zrq96), 草稿树的验证——树形掩码 (every node's logits are its children's target distribution);
// "万字综述 10+ 种 LLM 投机采样推理加速方案" (m.haoling.cc) 4.3 (argmax at temp = 0).
//
// One cluster of n CTAs per request (n <= 8, chosen at launch so that the batch's clusters fit
// the GPU at once).  CTA c of a cluster owns the vocabulary units [c * per, (c + 1) * per)
// (8 tokens each) and copies its slice of every row the request can need -- the target row of
// each of its T nodes and the draft row of each node with children -- into shared memory with
// 16-byte asynchronous copies from all its threads (the non-tensor bulk copy engine moved only
// ~24 GB/s per SM here).  The target slices are requested as soon as the request's node range
// is known and the draft slices right after its tree is read, so the copies overlap the
// validation; every row is read from HBM once and every later step runs on chip:
//   1. row statistics: four warps per row slice; the slice max first, then double-float sums of
//      2^((x - m) log2(e) / tau) against it (at tau = 0: max and lowest argmax); the CTAs
//      exchange their slices' (m, sum) through distributed shared memory and every CTA
//      combines the n partials of a row in one warp, rank by rank, so all hold the same (m, Z);
//   2. the walk: every CTA runs the same walk on the same values in the same order, so all
//      take the same decisions -- plain ratio tests from (m, Z), later siblings' residual
//      tests on thread 0 in fp64, as in the two-launch form;
//   3. vocabulary passes (a sibling's residual mass, the final residual or bonus draw): each
//      CTA sums the weights of its slice (block scan of double-float unit sums), the CTAs
//      exchange their totals, and the CTA whose prefix range holds u * total finds the token
//      in its slice.
// Leaves' target rows are reduced with the others, so the bonus draw needs no max pass, and at
// tau = 0 every row's argmax comes with the statistics: no pass runs at all.
// Every CTA of a cluster passes the same cluster barriers: its exits and every decision of the
// walk come from the same data in every CTA.  The kernel has no spin-wait: the copies end with
// cp.async.wait_all, the exchanges with hardware cluster barriers.
#include <math.h>

#include "common.cuh"
#include "cluster.cuh"
#include "tc_ptx.cuh"
#include "verify_cluster.cuh"

namespace spec {

namespace vcl {
constexpr int kMaxCl = 8;                      // CTAs per request at most (portable clusters)
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxT = 32;                      // nodes per request (one lane per node)
constexpr int kMaxRows = 2 * kMaxT;
constexpr int kParts = 4;                      // warps per row slice in the statistics
constexpr int kMaxDynSmem = 200 * 1024;        // row slices per CTA
constexpr int kCompactGroup = 4;               // moving steps a thread loads before storing
}  // namespace vcl

struct ClSmem {
  int16_t par[vcl::kMaxT], first_child[vcl::kMaxT], next_sib[vcl::kMaxT];
  int8_t dslot[vcl::kMaxT];                     // draft slice slot of a node, or -1
  int8_t slot_node[vcl::kMaxT];                 // node of a draft slice slot
  uint8_t dec0[vcl::kMaxT];                     // outcome of the node's plain ratio test
  int32_t path[vcl::kMaxT];
  int32_t tok[vcl::kMaxT], drow[vcl::kMaxT];
  float xt[vcl::kMaxT], xd[vcl::kMaxT];         // the node's token in its parent's rows
  float uacc[vcl::kMaxT], usamp[vcl::kMaxT];
  float st_m[vcl::kMaxT], sd_m[vcl::kMaxT], st_iz[vcl::kMaxT], sd_iz[vcl::kMaxT];
  double st_Z[vcl::kMaxT], sd_Z[vcl::kMaxT];
  int32_t st_arg[vcl::kMaxT];
  // statistics of the parts of this CTA's row slices
  float pm[vcl::kMaxRows][vcl::kParts], ps_hi[vcl::kMaxRows][vcl::kParts],
      ps_lo[vcl::kMaxRows][vcl::kParts];
  int32_t parg[vcl::kMaxRows][vcl::kParts];
  // read by the other CTAs of the cluster
  float xm[vcl::kMaxRows], xs_hi[vcl::kMaxRows], xs_lo[vcl::kMaxRows];
  int32_t xarg[vcl::kMaxRows];
  float px_hi[2], px_lo[2];                     // per pass (parity): this CTA's slice total
  int32_t px_last[2];                           // and its last unit with mass
  // block scan scratch
  dfloat wtot[vcl::kWarps];
  int32_t wlast[vcl::kWarps], wfirst[vcl::kWarps];
  double C, Nk;                                 // sibling residual state (thread 0)
  float Cf;
  int32_t decision, bad, nint, found;
  // KV compaction in the same launch: the moving steps and their slot offsets
  int32_t cmove[vcl::kMaxT];
  long long csrc[vcl::kMaxT], cdst[vcl::kMaxT];
  int32_t cnmove, cbad;
};

// 16-byte asynchronous global -> shared copy (L2 only), its commit and the wait for all of this
// thread's copies
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// copy `rows` row slices of `bytes` bytes (a multiple of 16) with all threads of the CTA:
// slice j from src(j) to dst + j * stride
template <typename Src>
__device__ __forceinline__ void copy_slices(uint8_t* dst, int stride, int rows, int bytes,
                                            Src src) {
  const int chunks = bytes / 16;
  for (int j = 0; j < rows; ++j) {
    const uint8_t* from = reinterpret_cast<const uint8_t*>(src(j));
    uint8_t* to = dst + size_t(j) * stride;
    for (int c = threadIdx.x; c < chunks; c += vcl::kThreads)
      cp_async16(to + size_t(c) * 16, from + size_t(c) * 16);
  }
}
__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float sum8_(const float (&w)[8]) {
  return ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
}
__device__ __forceinline__ bool df_above_(dfloat x, float th_hi, float th_lo) {
  return ((x.hi - th_hi) + (x.lo - th_lo)) > 0.f;
}
// (best, arg) pairs: the larger value, the lower index on ties
__device__ __forceinline__ void warp_argmax(float& best, int& arg) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, off);
    const int oa = __shfl_xor_sync(0xffffffffu, arg, off);
    if (ob > best || (ob == best && oa < arg)) { best = ob; arg = oa; }
  }
}

// unit k (8 values) of a row slice in shared memory
template <typename T>
__device__ __forceinline__ void smem_unit(const T* row, int k, float (&x)[8]) {
  if constexpr (sizeof(T) == 2) {
    elem<__nv_bfloat16>::unpack(*reinterpret_cast<const uint4*>(row + size_t(k) * 8), x);
  } else {
    const float4 a = *reinterpret_cast<const float4*>(row + size_t(k) * 8);
    const float4 b = *reinterpret_cast<const float4*>(row + size_t(k) * 8 + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
}

// Element weights of a pass: p up to 1 / Z (bonus draw, residual mass 0) or the sibling
// residual max(0, p - C q) -- the same arithmetic as the two-launch form.
struct ClWeight {
  bool residual, probs;
  float mt, md, k2, invZt, invZd, C;
  template <typename TT, typename TD>
  __device__ __forceinline__ void unit(const TT* trow, const TD* drow, int k, float (&w)[8]) const {
    float xt[8];
    smem_unit(trow, k, xt);
    if (!residual) {
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = ex2((xt[e] - mt) * k2);
      return;
    }
    float xd[8];
    smem_unit(drow, k, xd);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float p = ex2((xt[e] - mt) * k2) * invZt;
      const float q = probs ? xd[e] : ex2((xd[e] - md) * k2) * invZd;
      w[e] = fmaxf(0.f, p - C * q);
    }
  }
};

// One warp, units [k0, k1) of a row slice: the max (and, greedy, the lowest argmax).  (This
// kernel runs each phase once per launch, from a cold instruction cache: compact loops beat
// unrolled ones here.)
template <typename T>
__device__ __forceinline__ void part_max(const T* row, int k0, int k1, int u0, bool greedy,
                                         int lane, float& best, int& arg) {
  best = -INFINITY;
  arg = 0x7fffffff;
  for (int k = k0 + lane; k < k1; k += 32) {
    float x[8];
    smem_unit(row, k, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (greedy) {
        if (x[e] > best) { best = x[e]; arg = (u0 + k) * 8 + e; }
      } else {
        best = fmaxf(best, x[e]);
      }
    }
  }
  if (greedy) {
    warp_argmax(best, arg);
  } else {
    best = warp_max(best);
  }
}

// One warp, units [k0, k1): the compensated sum of 2^((x - m) k2), as a double-float.
template <typename T>
__device__ __forceinline__ dfloat part_sum(const T* row, int k0, int k1, float m, float k2,
                                           int lane) {
  float s = 0.f, c = 0.f;   // Kahan: the sum is s - c
  if (m != -INFINITY) {
    for (int k = k0 + lane; k < k1; k += 32) {
      float x[8], w[8];
      smem_unit(row, k, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = ex2((x[e] - m) * k2);
      const float y = sum8_(w) - c;
      const float t = s + y;
      c = (t - s) - y;
      s = t;
    }
  }
  return warp_sum_df(df_make(s - c));
}

struct ClPass {
  double total;   // the pass's total mass over the whole vocabulary
  bool pos;       // total > 0
  int owner;      // search passes: the rank that found the token (-1: no mass)
  int tok;        // the token, in the owner CTA only
};

// A vocabulary pass over the CTA's slices of one node's rows (same result in every CTA of the
// cluster; one cluster barrier).  Search: the smallest token x with
// sum_{y <= x} w(y) > u * total, found by the CTA whose range of the prefix holds u * total.
// A final draw (search with mass) arrives on the kernel's last cluster barrier right after its
// remote reads (*arrived), so the owner's search overlaps the other CTAs' exit.
template <typename TT, typename TD>
__device__ ClPass cl_pass(const TT* trow, const TD* drow, int nu, int u0, int per, int ncl,
                          const ClWeight& fn, bool search, float u, ClSmem& sh, int& npass,
                          int rank, bool* arrived) {
  using namespace vcl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int run = (nu + kThreads - 1) / kThreads;
  const int a0 = min(tid * run, nu), a1 = min(a0 + run, nu);
  dfloat mine = df_make(0.f);
  int lastp = -1;
  for (int k = a0; k < a1; ++k) {
    float w[8];
    fn.unit(trow, drow, k, w);
    const float su = sum8_(w);
    mine = df_add_f(mine, su);
    if (su > 0.f) lastp = k;
  }
  const dfloat incl = warp_scan_df(mine, lane);
  dfloat excl = df_shfl_up(incl, 1);
  if (lane == 0) excl = df_make(0.f);
  lastp = warp_max_int(lastp);
  if (lane == 31) sh.wtot[warp] = incl;
  if (lane == 0) sh.wlast[warp] = lastp;
  __syncthreads();
  const dfloat wsc = warp_scan_df(lane < kWarps ? sh.wtot[lane] : df_make(0.f), lane);
  dfloat wex = df_shfl_up(wsc, 1);
  if (lane == 0) wex = df_make(0.f);
  const dfloat wbase = {__shfl_sync(0xffffffffu, wex.hi, warp), __shfl_sync(0xffffffffu, wex.lo, warp)};
  const dfloat ctot = {__shfl_sync(0xffffffffu, wsc.hi, 31), __shfl_sync(0xffffffffu, wsc.lo, 31)};
  const int clast = warp_max_int(lane < kWarps ? sh.wlast[lane] : -1);   // local unit
  const int slot = npass & 1;
  ++npass;
  if (tid == 0) {
    sh.px_hi[slot] = ctot.hi;
    sh.px_lo[slot] = ctot.lo;
    sh.px_last[slot] = clast >= 0 ? u0 + clast : -1;
  }
  // the slot written two passes ago is free: every CTA read it before this barrier
  cluster_sync();
  dfloat rv = df_make(0.f);
  int rl = -1;
  if (lane < ncl) {
    rv.hi = ld_cluster_f32(&sh.px_hi[slot], lane);
    rv.lo = ld_cluster_f32(&sh.px_lo[slot], lane);
    rl = ld_cluster_s32(&sh.px_last[slot], lane);
  }
  const dfloat rincl = warp_scan_df(rv, lane);   // inclusive over ranks, in rank order
  const dfloat total = {__shfl_sync(0xffffffffu, rincl.hi, ncl - 1),
                        __shfl_sync(0xffffffffu, rincl.lo, ncl - 1)};
  const int lastall = warp_max_int(rl);
  ClPass res{df_to_d(total), total.hi > 0.f, -1, -1};
  if (!search || !res.pos) return res;
  cluster_arrive();   // this CTA reads no other CTA's shared memory after this point
  *arrived = true;
  // theta = u * total as a double-float
  const float ph = u * total.hi;
  const float pl = fmaf(u, total.hi, -ph) + u * total.lo;
  const float th_hi = ph + pl, th_lo = pl - (th_hi - ph);
  const unsigned rm = __ballot_sync(0xffffffffu, lane < ncl && df_above_(rincl, th_hi, th_lo));
  const int cstar = rm ? __ffs(rm) - 1 : -1;
  // no rank crossed (theta at the total by rounding): the last unit with mass decides
  res.owner = cstar >= 0 ? cstar : lastall / per;
  if (res.owner != rank) return res;
  dfloat rex = df_shfl_up(rincl, 1);
  if (lane == 0) rex = df_make(0.f);
  const dfloat rbase = {__shfl_sync(0xffffffffu, rex.hi, rank), __shfl_sync(0xffffffffu, rex.lo, rank)};
  if (tid == 0) sh.found = -1;
  if (cstar == rank) {
    const dfloat prefix = df_add(rbase, df_add(wbase, excl));
    const bool c = a0 < a1 && df_above_(df_add(rbase, df_add(wbase, incl)), th_hi, th_lo);
    const unsigned cm = __ballot_sync(0xffffffffu, c);
    if (lane == 0) sh.wfirst[warp] = cm ? warp * 32 + __ffs(cm) - 1 : 0x7fffffff;
    __syncthreads();
    int first = 0x7fffffff;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) first = min(first, sh.wfirst[w]);
    if (tid == first) {
      dfloat cum = prefix;
      int cross = -1, lastpos_unit = -1;
      for (int k = a0; k < a1; ++k) {
        float w[8];
        fn.unit(trow, drow, k, w);
        const float su = sum8_(w);
        const dfloat nx = df_add_f(cum, su);
        if (su > 0.f) lastpos_unit = k;
        if (df_above_(nx, th_hi, th_lo)) { cross = k; break; }
        cum = nx;
      }
      const int cu = cross >= 0 ? cross : lastpos_unit;
      int tok = -1, lastpos = -1;
      if (cu >= 0) {
        float w[8];
        fn.unit(trow, drow, cu, w);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          cum = df_add_f(cum, w[e]);
          if (w[e] > 0.f) lastpos = (u0 + cu) * 8 + e;
          if (tok < 0 && cross >= 0 && df_above_(cum, th_hi, th_lo)) tok = (u0 + cu) * 8 + e;
        }
      }
      sh.found = tok >= 0 ? tok : lastpos;
    }
  }
  __syncthreads();
  if (sh.found < 0) {
    // the crossing fell outside every thread's range by rounding: the slice's last element
    // with mass
    if (tid == 0 && clast >= 0) {
      float w[8];
      fn.unit(trow, drow, clast, w);
      int lp = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (w[e] > 0.f) lp = (u0 + clast) * 8 + e;
      sh.found = lp;
    }
    __syncthreads();
  }
  res.tok = sh.found;
  __syncthreads();   // sh.found and sh.wfirst are reused by the next pass
  return res;
}

// The KV compaction of spec_kv_compact for request r, run by every CTA of its cluster after
// the walk (path = sh.path[0 .. npath - 1]): the same validation (BAD_PARENT / BAD_BLOCK, the
// request rolled back), then slot P + d receives slot P + path[d] for every layer, KV head, K
// and V.  The CTAs split the 16-byte positions of the rows (layer, head, offset); each thread
// loads its position of every moving step of a group of kCompactGroup before storing any, so, with
// path[d] >= d and groups taken in increasing d, every source is read before it is overwritten
// (as in spec_kv_compact).  Rank 0 writes the slot map and the lengths.
__device__ void cl_compact(const ClusterVerifyArgs& a, ClSmem& sh, int r, int rank, int ncl,
                           int P, int npath) {
  using namespace vcl;
  const CompactDev& c = a.cd;
  const int tid = threadIdx.x;
  const int na = npath - 1;
  int32_t* sm_row = c.slot_map + size_t(r) * c.max_path * 2;
  const int32_t* trow = c.block_table + size_t(r) * c.max_blocks;
  if (tid == 0) sh.cbad = 0;
  __syncthreads();
  const bool ok = na >= 0 && na < c.max_path && P >= 0;
  if (ok) {
    for (int d = tid; d <= na; d += kThreads) {
      const int pd = sh.path[d];
      bool good = (d == 0) ? (pd == 0) : (pd >= d);
      const int lsb = (P + pd) / c.bs, ldb = (P + d) / c.bs;
      good = good && lsb < c.max_blocks && ldb < c.max_blocks;
      int flag = good ? 0 : SPEC_REQ_BAD_PARENT;
      if (good) {
        const int sb = trow[lsb], db = trow[ldb];
        if (sb < 0 || sb >= c.num_blocks || db < 0 || db >= c.num_blocks) flag = SPEC_REQ_BAD_BLOCK;
      }
      if (flag) atomicOr(&sh.cbad, flag);
    }
  }
  __syncthreads();
  if (!ok || sh.cbad) {
    if (rank == 0) {
      if (tid == 0 && ok) atomicOr(&a.req_status[r], sh.cbad);
      for (int k = tid; k < c.max_path; k += kThreads) { sm_row[2 * k] = -1; sm_row[2 * k + 1] = -1; }
      if (tid == 0) {
        c.new_kv_len[r] = P;
        c.blocks_in_use[r] = (P + c.bs - 1) / c.bs;
      }
    }
    return;
  }
  const size_t head_stride = size_t(c.bs) * c.row_bytes;
  const size_t block_stride = size_t(c.H_kv) * head_stride;
  if (tid == 0) {
    int n = 0;
    for (int d = 1; d <= na; ++d)
      if (sh.path[d] != d) sh.cmove[n++] = d;
    sh.cnmove = n;
  }
  __syncthreads();
  const int nmove = sh.cnmove;
  for (int q = tid; q < nmove; q += kThreads) {
    const int d = sh.cmove[q];
    const int src = P + sh.path[d], dst = P + d;
    sh.csrc[q] = (long long)(size_t(trow[src / c.bs]) * block_stride + size_t(src % c.bs) * c.row_bytes);
    sh.cdst[q] = (long long)(size_t(trow[dst / c.bs]) * block_stride + size_t(dst % c.bs) * c.row_bytes);
  }
  __syncthreads();
  if (nmove > 0) {
    const int vpr = c.row_bytes / 16;
    const long long per_layer = (long long)c.H_kv * vpr;
    const long long total = per_layer * c.num_layers;
    const long long w0 = total * rank / ncl, w1 = total * (rank + 1) / ncl;
    for (long long w = w0 + tid; w < w1; w += kThreads) {
      const int layer = int(w / per_layer);
      const int rem = int(w - layer * per_layer);
      const int h = rem / vpr;
      const size_t in_row = size_t(h) * head_stride + size_t(rem - h * vpr) * 16;
      char* kb = c.k + layer * c.layer_stride_bytes;
      char* vb = c.v + layer * c.layer_stride_bytes;
      for (int g0 = 0; g0 < nmove; g0 += kCompactGroup) {
        const int gs = min(kCompactGroup, nmove - g0);
        uint4 kv[kCompactGroup][2];
#pragma unroll
        for (int q = 0; q < kCompactGroup; ++q) {
          if (q < gs) {
            const size_t o = size_t(sh.csrc[g0 + q]) + in_row;
            kv[q][0] = *reinterpret_cast<const uint4*>(kb + o);
            kv[q][1] = *reinterpret_cast<const uint4*>(vb + o);
          }
        }
#pragma unroll
        for (int q = 0; q < kCompactGroup; ++q) {
          if (q < gs) {
            const size_t o = size_t(sh.cdst[g0 + q]) + in_row;
            *reinterpret_cast<uint4*>(kb + o) = kv[q][0];
            *reinterpret_cast<uint4*>(vb + o) = kv[q][1];
          }
        }
      }
    }
  }
  if (rank == 0) {
    for (int k = tid; k < c.max_path; k += kThreads) {
      const bool in = k <= na;
      sm_row[2 * k] = in ? P + sh.path[k] : -1;
      sm_row[2 * k + 1] = in ? P + k : -1;
    }
    if (tid == 0) {
      c.new_kv_len[r] = P + na + 1;
      c.blocks_in_use[r] = (P + na + 1 + c.bs - 1) / c.bs;
    }
  }
}

template <typename TT, typename TD>
__global__ void __launch_bounds__(vcl::kThreads, 1) verify_cluster_kernel(ClusterVerifyArgs a) {
  using namespace vcl;
  __shared__ ClSmem sh;
  extern __shared__ __align__(128) uint8_t rows_s[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) sh.bad = 0;
  // the first kernel of the call: the logits or the tree flags may come from the previous
  // kernel on the stream
  pdl_wait();
  pdl_trigger();
  const int rank = cluster_rank(), ncl = cluster_size();
  const int r = blockIdx.x / ncl;
  int32_t* path_row = a.path + size_t(r) * a.max_path;
  int32_t* tok_row = a.out_tokens + size_t(r) * a.max_path;
  const bool greedy = a.tau == 0.f;
  const TT* target = reinterpret_cast<const TT*>(a.target);
  const TD* draft = reinterpret_cast<const TD*>(a.draft);
  const int st0 = a.req_status[r];
  const int P = a.compact ? a.cd.prefix_len[r] : 0;
  const int o = a.node_offset[r];
  const int T = a.node_offset[r + 1] - o;
  const bool range_ok = o >= 0 && T >= 1 && T <= a.T_max && o + T <= a.N;
  // every CTA of the cluster takes the same exits: they read the same data
  auto fail_exit = [&](int bits) {
    if (rank == 0) {
      if (tid == 0 && bits) atomicOr(&a.req_status[r], bits);
      for (int k = tid; k < a.max_path; k += kThreads) { path_row[k] = -1; tok_row[k] = -1; }
      if (tid == 0) {
        a.out_len[r] = 0;
        a.n_acc[r] = -1;
        if (a.rejections) a.rejections[r] = 0;
      }
      if (a.compact) {   // the whole tree rolled back, as spec_kv_compact does for it
        int32_t* sm_row = a.cd.slot_map + size_t(r) * a.cd.max_path * 2;
        for (int k = tid; k < a.cd.max_path; k += kThreads) { sm_row[2 * k] = -1; sm_row[2 * k + 1] = -1; }
        if (tid == 0) {
          a.cd.new_kv_len[r] = P;
          a.cd.blocks_in_use[r] = (P + a.cd.bs - 1) / a.cd.bs;
        }
      }
    }
  };
  __syncthreads();   // sh.bad is initialised
  if (st0 != 0 || !range_ok) {
    fail_exit(range_ok ? 0 : SPEC_REQ_BAD_SIZE);
    return;   // before any cluster barrier, in every CTA of the cluster
  }
  const int V = a.V, nunits = (V + 7) / 8, full = V / 8;
  const int per = a.per_units;
  const int u0 = min(rank * per, nunits), u1 = min(u0 + per, nunits), nu = u1 - u0;
  const int nfull = max(0, min(u1, full) - u0);
  const int tbytes = nfull * 8 * int(sizeof(TT));
  const int dbytes = nfull * 8 * int(sizeof(TD));
  uint8_t* const drows_s = rows_s + size_t(a.T_max) * a.t_slice;
  // the target slices of all T nodes need only the node range
  copy_slices(rows_s, a.t_slice, T, tbytes,
              [&](int j) { return target + size_t(o + j) * a.tld + size_t(u0) * 8; });
  cp_async_commit();
  // the tree, tokens, depths, draft rows and uniforms, one lane per node (T <= 32); validation
  // of tokens, parents, depths; children and siblings from lanes sharing a parent; the draft
  // slices (one per node with children, tau > 0); then the operands of the ratio tests -- each
  // node's token in its parent's rows -- are requested, to be stored once the copies landed
  float xt_r = 0.f, xd_r = 0.f;
  bool has_t = false, has_d = false;
  if (warp == 0) {
    const int i = lane;
    const bool in = i < T;
    const int n = o + i;
    int p = -1, t = -1, dr = -1, bad = 0;
    bool pok = false;
    if (in) {
      p = a.parent[n];
      pok = i == 0 ? p == -1 : (p >= 0 && p < i);
      if (!pok) bad |= SPEC_REQ_BAD_PARENT;
      if (i > 0) {
        t = a.tokens[n];
        if (t < 0 || t >= V) bad |= SPEC_REQ_BAD_TOKEN;
      }
      if (a.depth[n] + 1 > a.max_path) bad |= SPEC_REQ_BAD_DEPTH;
      dr = greedy ? -1 : a.draft_row[n];
      sh.par[i] = int16_t(pok ? p : -1);
      sh.tok[i] = t;
      sh.drow[i] = dr;
      sh.uacc[i] = a.uniforms[2 * size_t(n)];
      sh.usamp[i] = a.uniforms[2 * size_t(n) + 1];
    }
    const bool child = in && i > 0 && pok;
    // lanes with the same parent are siblings, in index order; a unique key otherwise
    const unsigned peers = __match_any_sync(0xffffffffu, child ? p : -2 - i);
    const unsigned has_child = __reduce_or_sync(0xffffffffu, child ? (1u << p) : 0u);
    sh.first_child[i] = -1;
    __syncwarp();
    if (child) {
      const unsigned later = peers & ~((2u << i) - 1u);
      sh.next_sib[i] = int16_t(later ? __ffs(later) - 1 : -1);
      if ((peers & ((1u << i) - 1u)) == 0) sh.first_child[p] = int16_t(i);
    } else {
      sh.next_sib[i] = -1;
    }
    const bool need = !greedy && in && ((has_child >> i) & 1u);
    const bool row_ok = need && dr >= 0 && dr < a.R;
    const unsigned m = __ballot_sync(0xffffffffu, row_ok);
    const int slot = __popc(m & ((1u << i) - 1u));
    if (in) sh.dslot[i] = int8_t(row_ok ? slot : -1);
    if (row_ok) sh.slot_node[slot] = int8_t(i);
    if (need && !row_ok) bad |= SPEC_REQ_BAD_DRAFT_ROW;
    bad = __reduce_or_sync(0xffffffffu, bad);
    if (i == 0) {
      sh.nint = __popc(m);
      sh.bad = bad;
    }
    // the parent's draft row, from its lane
    const int pdr = __shfl_sync(0xffffffffu, dr, child ? p : 0);
    if (!greedy && child && t >= 0 && t < V) {
      xt_r = elem<TT>::load1(target + size_t(o + p) * a.tld + t);
      has_t = true;
      if (pdr >= 0 && pdr < a.R) {
        xd_r = elem<TD>::load1(draft + size_t(pdr) * a.dld + t);
        has_d = true;
      }
    }
  }
  __syncthreads();
  const int nint = sh.nint;
  copy_slices(drows_s, a.d_slice, nint, dbytes, [&](int k) {
    return draft + size_t(sh.drow[sh.slot_node[k]]) * a.dld + size_t(u0) * 8;
  });
  cp_async_commit();
  if (full < u1 && full >= u0) {
    // the ragged last unit (V % 8 != 0) element by element, padded with weight-0 values
    for (int idx = tid; idx < (T + nint) * 8; idx += kThreads) {
      const int j = idx >> 3, e = idx & 7, v = full * 8 + e;
      if (j < T) {
        TT* dst = reinterpret_cast<TT*>(rows_s + size_t(j) * a.t_slice) + size_t(full - u0) * 8 + e;
        *dst = v < V ? target[size_t(o + j) * a.tld + v] : TT(-INFINITY);
      } else {
        const int k = j - T;
        TD* dst = reinterpret_cast<TD*>(drows_s + size_t(k) * a.d_slice) + size_t(full - u0) * 8 + e;
        *dst = v < V ? draft[size_t(sh.drow[sh.slot_node[k]]) * a.dld + v]
                     : TD(a.probs ? 0.f : -INFINITY);
      }
    }
  }
  if (has_t) sh.xt[lane] = xt_r;   // warp 0 only; the loads have had the copies' time to land
  if (has_d) sh.xd[lane] = xd_r;
  cp_async_wait_all();
  __syncthreads();
  if (sh.bad) {
    fail_exit(sh.bad);
    return;   // uniform across the cluster: sh.bad comes from the same data everywhere
  }
  // 1. statistics of this CTA's slices: kParts warps per row, the slice max first
  const int nrows = (greedy || a.probs) ? T : T + nint;
  const int ntasks = nrows * kParts;
  auto row_ptr = [&](int j) -> const uint8_t* {
    return j < T ? rows_s + size_t(j) * a.t_slice : drows_s + size_t(j - T) * a.d_slice;
  };
  {
    for (int t = warp; t < ntasks; t += kWarps) {
      const int j = t / kParts, q = t % kParts;
      const int k0 = nu * q / kParts, k1 = nu * (q + 1) / kParts;
      float best;
      int arg;
      if (j < T)
        part_max(reinterpret_cast<const TT*>(row_ptr(j)), k0, k1, u0, greedy, lane, best, arg);
      else
        part_max(reinterpret_cast<const TD*>(row_ptr(j)), k0, k1, u0, false, lane, best, arg);
      if (lane == 0) { sh.pm[j][q] = best; sh.parg[j][q] = arg; }
    }
    __syncthreads();
    if (!greedy) {
      for (int t = warp; t < ntasks; t += kWarps) {
        const int j = t / kParts, q = t % kParts;
        const int k0 = nu * q / kParts, k1 = nu * (q + 1) / kParts;
        float m = sh.pm[j][0];
#pragma unroll
        for (int qq = 1; qq < kParts; ++qq) m = fmaxf(m, sh.pm[j][qq]);
        const dfloat s = j < T
                             ? part_sum(reinterpret_cast<const TT*>(row_ptr(j)), k0, k1, m, a.k2, lane)
                             : part_sum(reinterpret_cast<const TD*>(row_ptr(j)), k0, k1, m, a.k2, lane);
        if (lane == 0) { sh.ps_hi[j][q] = s.hi; sh.ps_lo[j][q] = s.lo; }
      }
      __syncthreads();
    }
    for (int j = tid; j < nrows; j += kThreads) {
      float best = sh.pm[j][0];
      int arg = sh.parg[j][0];
      dfloat s = {sh.ps_hi[j][0], sh.ps_lo[j][0]};
#pragma unroll
      for (int q = 1; q < kParts; ++q) {
        if (greedy) {
          if (sh.pm[j][q] > best || (sh.pm[j][q] == best && sh.parg[j][q] < arg)) {
            best = sh.pm[j][q];
            arg = sh.parg[j][q];
          }
        } else {
          best = fmaxf(best, sh.pm[j][q]);
          s = df_add(s, dfloat{sh.ps_hi[j][q], sh.ps_lo[j][q]});
        }
      }
      sh.xm[j] = best;
      sh.xarg[j] = arg;
      sh.xs_hi[j] = greedy ? 0.f : s.hi;
      sh.xs_lo[j] = greedy ? 0.f : s.lo;
    }
  }
  cluster_sync();
  // combine the ncl partials of every row, one warp per row, lanes = ranks (the same order and
  // arithmetic in every CTA)
  for (int j = warp; j < nrows; j += kWarps) {
    float mc = -INFINITY;
    int ac = 0x7fffffff;
    dfloat sc = df_make(0.f);
    if (lane < ncl) {
      mc = ld_cluster_f32(&sh.xm[j], lane);
      if (greedy) {
        ac = ld_cluster_s32(&sh.xarg[j], lane);
      } else {
        sc.hi = ld_cluster_f32(&sh.xs_hi[j], lane);
        sc.lo = ld_cluster_f32(&sh.xs_lo[j], lane);
      }
    }
    if (greedy) {
      warp_argmax(mc, ac);
      if (lane == 0) { sh.st_m[j] = mc; sh.st_arg[j] = ac; }
      continue;
    }
    const float M = warp_max(mc);
    const float f = mc == -INFINITY ? 0.f : ex2((mc - M) * a.k2);
    const dfloat Zd = warp_sum_df(dfloat{sc.hi * f, sc.lo * f});
    if (lane == 0) {
      const double Z = df_to_d(Zd);
      if (j < T) {
        sh.st_m[j] = M;
        sh.st_Z[j] = Z;
        sh.st_iz[j] = __frcp_rn(float(Z));   // fp32: no fp64 division on the critical path
      } else {
        const int n = sh.slot_node[j - T];
        sh.sd_m[n] = M;
        sh.sd_Z[n] = Z;
        sh.sd_iz[n] = __frcp_rn(float(Z));
      }
    }
  }
  if (!greedy && a.probs) {
    for (int i = tid; i < T; i += kThreads) {
      sh.sd_m[i] = 0.f;
      sh.sd_Z[i] = 1.0;
      sh.sd_iz[i] = 1.f;
    }
  }
  __syncthreads();
  // 2. plain ratio tests u < p / q of every non-root node
  if (!greedy) {
    for (int i = tid; i < T; i += kThreads) {
      if (i > 0) {
        const int p = sh.par[i];
        const double u = double(sh.uacc[i]);
        bool acc;
        if (!a.probs) {
          const float e = expf(((sh.xt[i] - sh.st_m[p]) - (sh.xd[i] - sh.sd_m[p])) * a.inv_tau);
          acc = u * sh.st_Z[p] < double(e) * sh.sd_Z[p];
        } else {
          const float e = expf((sh.xt[i] - sh.st_m[p]) * a.inv_tau);
          acc = u * double(sh.xd[i]) * sh.st_Z[p] < double(e);
        }
        sh.dec0[i] = acc ? 1 : 0;
      }
    }
  }
  if (tid == 0) sh.path[0] = 0;
  __syncthreads();

  int node = 0, npath = 1, rejections = 0, final_tok = -1, owner = 0, npass = 0;
  bool arrived = false;   // on the last cluster barrier
  while (true) {
    const int fc = sh.first_child[node];
    if (greedy) {
      const int best = sh.st_arg[node];
      int acc = -1, rej = 0;
      for (int c = fc; c >= 0; c = sh.next_sib[c]) {
        if (sh.tok[c] == best) { acc = c; break; }
        ++rej;
      }
      rejections += rej;
      if (acc >= 0) {
        if (tid == 0) sh.path[npath] = acc;
        ++npath;
        node = acc;
        continue;
      }
      final_tok = best;
      break;
    }
    const TT* trow = reinterpret_cast<const TT*>(rows_s + size_t(node) * a.t_slice);
    const float u_samp = sh.usamp[node];
    if (fc < 0) {   // leaf: bonus token from p_leaf
      ClWeight fn{};
      fn.residual = false;
      fn.mt = sh.st_m[node];
      fn.k2 = a.k2;
      const ClPass pr = cl_pass(trow, static_cast<const TD*>(nullptr), nu, u0, per, ncl, fn, true,
                                u_samp, sh, npass, rank, &arrived);
      final_tok = pr.tok;
      owner = pr.owner;
      break;
    }
    const TD* drow = reinterpret_cast<const TD*>(drows_s + size_t(sh.dslot[node]) * a.d_slice);
    ClWeight res{};
    res.residual = true;
    res.probs = a.probs != 0;
    res.mt = sh.st_m[node];
    res.md = sh.sd_m[node];
    res.k2 = a.k2;
    res.invZt = sh.st_iz[node];
    res.invZd = sh.sd_iz[node];
    res.C = 1.f;
    if (tid == 0) { sh.C = 0.0; sh.Nk = 1.0; }
    int accepted = -1;
    bool from_p = false;
    for (int c = fc; c >= 0; c = sh.next_sib[c]) {
      bool acc;
      if (c == fc || !a.residual_rule) {
        acc = sh.dec0[c] != 0;
      } else {
        if (tid == 0) {
          // u < max(0, p - C q) / (N q) as u * N * q < max(0, p - C q), both sides times Zt
          // (and Zd for draft logits): no fp64 division
          const double et = double(expf((sh.xt[c] - sh.st_m[node]) * a.inv_tau));
          const double Zt = sh.st_Z[node], u = double(sh.uacc[c]);
          if (a.probs) {
            const double qZ = double(sh.xd[c]) * Zt;
            sh.decision = u * (sh.Nk * qZ) < fmax(0.0, et - sh.C * qZ);
          } else {
            const double qZ = double(expf((sh.xd[c] - sh.sd_m[node]) * a.inv_tau)) * Zt;
            sh.decision = u * (sh.Nk * qZ) < fmax(0.0, et * sh.sd_Z[node] - sh.C * qZ);
          }
        }
        __syncthreads();
        acc = sh.decision != 0;
        __syncthreads();
      }
      if (acc) { accepted = c; break; }
      ++rejections;
      if (a.residual_rule) {
        // C_{k+1} = C_k + N_k, N_{k+1} = sum_x max(0, p(x) - C_{k+1} q(x))
        if (tid == 0) { sh.C += sh.Nk; sh.Cf = float(sh.C); }
        __syncthreads();
        res.C = sh.Cf;
        if (sh.next_sib[c] < 0) break;   // the final draw yields N_{k+1} itself
        const ClPass pr = cl_pass(trow, drow, nu, u0, per, ncl, res, false, 0.f, sh, npass, rank, &arrived);
        if (tid == 0) sh.Nk = pr.total;
        if (!pr.pos) { from_p = true; break; }
      }
    }
    if (accepted >= 0) {
      if (tid == 0) sh.path[npath] = accepted;
      ++npath;
      node = accepted;
      continue;
    }
    if (!from_p) {
      const ClPass pr = cl_pass(trow, drow, nu, u0, per, ncl, res, true, u_samp, sh, npass, rank, &arrived);
      final_tok = pr.tok;
      owner = pr.owner;
      if (!pr.pos) from_p = true;
    }
    if (from_p) {
      ClWeight fn{};
      fn.residual = false;
      fn.mt = res.mt;
      fn.k2 = a.k2;
      const ClPass pr = cl_pass(trow, drow, nu, u0, per, ncl, fn, true, u_samp, sh, npass, rank, &arrived);
      final_tok = pr.tok;
      owner = pr.owner;
    }
    break;
  }
  if (owner < 0) { owner = 0; final_tok = -1; }   // a row without mass: no token
  __syncthreads();
  if (rank == 0) {
    for (int k = tid; k < a.max_path; k += kThreads) {
      if (k < npath) {
        path_row[k] = sh.path[k];
        if (k + 1 < npath) tok_row[k] = sh.tok[sh.path[k + 1]];
        else if (owner == 0) tok_row[k] = final_tok;
      } else {
        path_row[k] = -1;
        tok_row[k] = -1;
      }
    }
    if (tid == 0) {
      a.out_len[r] = npath;
      a.n_acc[r] = npath - 1;
      if (a.rejections) a.rejections[r] = rejections;
    }
  } else if (owner == rank && tid == 0) {
    tok_row[npath - 1] = final_tok;
  }
  if (a.compact) cl_compact(a, sh, r, rank, ncl, P, npath);
  // no CTA leaves while another may still read its shared memory
  if (!arrived) cluster_arrive();
  cluster_wait();
}

// ---------------------------------------------------------------------------- host side
namespace {

// dynamic shared memory of one CTA for n CTAs per request (0: does not fit)
long long cluster_smem(const ClusterVerifyArgs& a, int n, int tes, int des, long long* per_out) {
  const long long nunits = (a.V + 7LL) / 8;
  const long long per = (nunits + n - 1) / n;
  const long long ts = per * 8 * tes;
  const long long ds = a.tau > 0.f ? per * 8 * des : 0;
  const long long smem = a.T_max * ts + (a.T_max - 1) * ds;
  if (per_out) *per_out = per;
  return smem <= vcl::kMaxDynSmem ? smem : 0;
}

}  // namespace

bool verify_cluster_fits(const ClusterVerifyArgs& a, int tes, int des) {
  if (a.T_max < 1 || a.T_max > vcl::kMaxT || a.V < 1 || a.B < 1) return false;
  return cluster_smem(a, vcl::kMaxCl, tes, des, nullptr) > 0;
}

template <typename TT, typename TD>
static cudaError_t launch_cl(ClusterVerifyArgs a, int tes, int des, cudaStream_t s) {
  using namespace vcl;
  static DeviceOnce raised;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kernel = verify_cluster_kernel<TT, TD>;
  if (!raised.test(dev)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e != cudaSuccess) return e;
    raised.set(dev);
  }
  // CTAs per request: the fewest waves per unit of work, i.e. the least
  // ceil(B / resident clusters) / n; ties to the larger n
  int best_n = 0;
  double best_cost = 0.0;
  for (int n = kMaxCl; n >= 1; --n) {
    const long long smem = cluster_smem(a, n, tes, des, nullptr);
    if (smem == 0) continue;
    const int resident = active_clusters(kernel, dev, n, vcl::kThreads, smem);
    if (resident < 1) continue;
    const double cost = double((a.B + resident - 1) / resident) / n;
    if (best_n == 0 || cost < best_cost) {
      best_n = n;
      best_cost = cost;
    }
  }
  if (best_n == 0) return cudaErrorNotSupported;   // the caller takes the two-launch form
  long long per = 0;
  const long long smem = cluster_smem(a, best_n, tes, des, &per);
  a.per_units = int(per);
  a.t_slice = int(per * 8 * tes);
  a.d_slice = int(a.tau > 0.f ? per * 8 * des : 0);
  a.smem = int(smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(a.B) * unsigned(best_n));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(a.smem);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(best_n);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, kernel, a);
  if (le == cudaSuccess) count_launch();
  return le;
}

cudaError_t launch_verify_cluster(const ClusterVerifyArgs& a, int tes, int des, cudaStream_t s) {
  if (tes == 2 && des == 2) return launch_cl<__nv_bfloat16, __nv_bfloat16>(a, tes, des, s);
  if (tes == 2 && des == 4) return launch_cl<__nv_bfloat16, float>(a, tes, des, s);
  return launch_cl<float, float>(a, tes, des, s);
}

}  // namespace spec
