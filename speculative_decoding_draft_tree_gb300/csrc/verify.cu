// spec_verify: ratio-test verification of packed draft trees with residual resampling.
//
// Sources (page title, section):
//   "推测解码 2026" (guijiagi.com), 数学基础：拒绝采样 -- accept with min(1, p/q); on rejection resample
//     from relu(p - q) normalised and drop the remaining candidates;
//   "【模型后训练与深度推理】9 推理加速：推测解码与级联推理", 7.1 -- alpha = min(1, p/q), residual
//     norm(max(0, p - q)); 7.2 -- the emitted count includes the final corrected / bonus token;
//   "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的验证——树形掩码 -- node i's logits give
//     P(. | ancestors(i)); verification walks every level of the tree;
//   "万字综述 10+ 种 LLM 投机采样推理加速方案" (m.haoling.cc) 4.3 -- argmax sampling at temp = 0.
//
// Calls that fit it (residual or independent sibling rule, trees of at most 32 nodes, a
// request's row slices within one CTA's shared memory) run as ONE cluster launch
// (verify_cluster.cu: the rows of each request held on chip by a cluster of CTAs); the others,
// and every call whose verify_path field is SPEC_VERIFY_PATH_SPLIT, take the two-launch form,
// except that with those rules and a vocabulary of 65536 or more (or SPEC_VERIFY_PATH_WALK) the
// walk runs alone and forms the statistics of the nodes it visits itself: one pass over each
// visited internal node's target and draft rows (online max and compensated sum per thread,
// combined over the block and the cluster in a fixed order), then that node's children's plain
// ratio tests -- a few rows per request instead of every internal node's.
// Two launches on the caller's stream:
//   1. rows  (one CTA per internal node's target row and, for tau > 0 with draft logits, per
//      draft row; 256 threads, several CTAs per SM): ONE streaming read of the row with 16-byte
//      loads; per-thread online max / sum of 2^((x - m) log2(e) / tau) over chunks of eight
//      8-element units (Kahan-compensated), then a block reduction (max, then a double-float
//      sum) -> (m, Z);
//      tau = 0 keeps (max, lowest argmax) instead;
//   2. walk  (one cluster of 1..8 CTAs of 512 threads per request; CTA k of a cluster owns the
//      k-th contiguous slice of the vocabulary): validates the request's tokens, draft rows
//      and depths, then walks the tree.  A parallel prologue gathers
//      every node's test operands and decides every plain ratio test u < p / q at once (thread
//      per node, from (m, Z)); only later siblings under the residual rule are tested on the way,
//      on thread 0.  Every vocab-wide step (sibling residual mass, residual / bonus inverse CDF,
//      leaf max / argmax) is a pass over each CTA's slice: 16 warps own contiguous ranges of
//      it, per-warp double-float sums are scanned in token order, the CTAs exchange their slice
//      totals through distributed shared memory (one cluster barrier) and combine them in rank
//      order, and the CTA whose range of the prefix holds the crossing rescans its unit sums
//      (kept in shared memory) to find the unit, then the unit's 8 elements.  Every CTA of a
//      cluster runs the same walk on the same values in the same order, so all take the same
//      decisions and pass the same barriers.  A pass costs two exponentials per token, so one
//      SM per request is bound by its special-function units; slicing the vocabulary over a
//      cluster divides that time by the cluster size.
// Under the multi-draft sibling rule (siblings proposed by different draft models, each with its
// own q) the running residual has no closed form: it is materialised per request in a
// double-buffered fp32 scratch row, one vocab pass per rejected sibling (the last one is folded
// into the final draw), and that case runs its own instantiation of the walk kernel, with one
// CTA per request: its ratio tests read single elements of the scratch row, which a slice
// owned by another CTA would have written.
// Randomness is never generated here: u_acc / u_samp come from the caller's uniforms.
#include <math.h>

#include <atomic>
#include <mutex>

#include "cluster.cuh"
#include "common.cuh"
#include "kv_compact.cuh"
#include "verify_cluster.cuh"

namespace spec {

struct RowStat {
  float m;      // row max of the raw logits
  int32_t arg;  // lowest index of the max (tau = 0 rows)
  double Z;     // sum over the row of 2^((x - m) * log2(e) / tau)
  float inv_Z;  // float(1 / Z), for the vocab-wide weights
  int32_t pad;
};


struct VerifyDev {
  const void* target;
  const void* draft;
  int64_t tld, dld;
  int32_t B, N, R, V, T_max, max_path;
  float tau, k2, inv_tau;  // k2 = log2(e) / tau
  int32_t probs, residual_rule, multi;   // multi: the multi-draft sibling rule
  const int32_t* draft_row;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* node_offset;
  const int32_t* depth;
  const uint8_t* is_internal;
  const float* uniforms;
  int32_t* req_status;
  int32_t* out_tokens;
  int32_t* out_len;
  int32_t* path;
  int32_t* n_acc;
  int32_t* rejections;
  RowStat* tstat;
  RowStat* dstat;
  float* rbuf;          // multi-draft: per request, two residual rows of rld floats
  int64_t rld;
  int32_t after_rows;   // the walk follows a rows kernel of the same call
  int32_t walk_per;     // 8-element vocabulary units of each CTA of a request's walk cluster
  int32_t lazy;         // no rows kernel: the walk forms the statistics of the nodes it visits
                        // (the kLazy walk)
};

// ---- 8-element units: one 16-byte load for bf16, two for fp32 ------------------------------
template <typename T>
__device__ __forceinline__ void load8(const T* __restrict__ row, int unit, int V, int full,
                                      float fill, float (&x)[8]) {
  if (unit < full) {
    if constexpr (sizeof(T) == 2) {
      uint4 v = ld_stream16(row + size_t(unit) * 8);
      elem<T>::unpack(v, x);
    } else {
      uint4 a = ld_stream16(row + size_t(unit) * 8);
      uint4 b = ld_stream16(row + size_t(unit) * 8 + 4);
      x[0] = __uint_as_float(a.x); x[1] = __uint_as_float(a.y);
      x[2] = __uint_as_float(a.z); x[3] = __uint_as_float(a.w);
      x[4] = __uint_as_float(b.x); x[5] = __uint_as_float(b.y);
      x[6] = __uint_as_float(b.z); x[7] = __uint_as_float(b.w);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      int idx = unit * 8 + k;
      x[k] = idx < V ? elem<T>::load1(row + idx) : fill;
    }
  }
}

__device__ __forceinline__ float sum8(const float (&w)[8]) {
  return ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
}

// One 8-element unit of a row as raw 16-byte vectors, so that several units' loads can be
// issued before any of them is used.
template <typename T>
struct RawUnit {
  static constexpr int kVec = int(sizeof(T)) / 2;   // 1 for bf16, 2 for fp32
  uint4 v[kVec];
  __device__ __forceinline__ void load(const T* row, int unit) {
#pragma unroll
    for (int k = 0; k < kVec; ++k) v[k] = ld_stream16(row + size_t(unit) * 8 + k * (8 / kVec));
  }
  // the unit's 8 values; the ragged last unit (unit >= full) is read element by element
  __device__ __forceinline__ void get(const T* row, int unit, int V, int full, float fill,
                                      float (&x)[8]) const {
    if (unit < full) {
      if constexpr (kVec == 1) {
        elem<T>::unpack(v[0], x);
      } else {
        elem<float>::unpack(v[0], x);
        float y[4];
        elem<float>::unpack(v[1], y);
        x[4] = y[0]; x[5] = y[1]; x[6] = y[2]; x[7] = y[3];
      }
    } else {
      load8(row, unit, V, full, fill, x);
    }
  }
};

// ---- 1. rows: (m, Z) or (max, argmax) in one streaming read --------------------------------
// One row's statistics take one CTA of kRowThreads threads (several CTAs fit on an SM, which
// keeps more loads in flight per SM than one large CTA per row).
constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;

struct RowScratch {
  float f[kRowWarps];
  int i[kRowWarps];
  float hi[kRowWarps], lo[kRowWarps];
  RowStat out;
};

// barrier over the kRowThreads threads of one row (named barrier `bar`)
__device__ __forceinline__ void row_sync(int bar) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "n"(kRowThreads) : "memory");
}

// pairwise sum of n values (n a power of two), a fixed tree
template <int n>
__device__ __forceinline__ float tree_sum(const float* t) {
  if constexpr (n == 1) {
    return t[0];
  } else {
    return tree_sum<n / 2>(t) + tree_sum<n / 2>(t + n / 2);
  }
}

// (m, Z) -- or (max, lowest argmax) for tau = 0 -- of one row, computed by kRowThreads threads
// and returned to each of them.  Each thread keeps kUnroll 16-byte loads in flight, then folds
// them into an online max / Kahan-compensated sum of 2^((x - m) log2(e) / tau); the block
// combines maxima, then double-float sums.
template <typename T>
__device__ RowStat row_stats(const T* row, const VerifyDev& a, RowScratch& sc, int bar) {
  constexpr int kUnroll = 8;
  constexpr int kStep = kUnroll * kRowThreads;
  const int tid = threadIdx.x % kRowThreads, lane = tid & 31, warp = tid >> 5;
  const int V = a.V, full = V / 8, nunits = (V + 7) / 8;
  if (a.tau == 0.f) {
    float best = -INFINITY;
    int arg = 0x7fffffff;
    for (int u0 = tid; u0 < nunits; u0 += kStep) {
      RawUnit<T> raw[kUnroll];
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) {
        const int unit = u0 + j * kRowThreads;
        if (unit < full) raw[j].load(row, unit);
      }
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) {
        const int unit = u0 + j * kRowThreads;
        if (unit < nunits) {
          float x[8];
          raw[j].get(row, unit, V, full, -INFINITY, x);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (x[k] > best) { best = x[k]; arg = unit * 8 + k; }
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float ob = __shfl_xor_sync(0xffffffffu, best, off);
      int oa = __shfl_xor_sync(0xffffffffu, arg, off);
      if (ob > best || (ob == best && oa < arg)) { best = ob; arg = oa; }
    }
    if (lane == 0) { sc.f[warp] = best; sc.i[warp] = arg; }
    row_sync(bar);
    if (tid == 0) {
      float bb = sc.f[0];
      int ba = sc.i[0];
      for (int w = 1; w < kRowWarps; ++w)
        if (sc.f[w] > bb || (sc.f[w] == bb && sc.i[w] < ba)) { bb = sc.f[w]; ba = sc.i[w]; }
      sc.out = RowStat{bb, ba, 0.0, 0.f, 0};
    }
  } else {
    const float k2 = a.k2;
    float m = -INFINITY, s = 0.f, c = 0.f;  // Kahan: true sum ~ s - c
    for (int u0 = tid; u0 < nunits; u0 += kStep) {
      RawUnit<T> raw[kUnroll];
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) {
        const int unit = u0 + j * kRowThreads;
        if (unit < full) raw[j].load(row, unit);
      }
      float cm = -INFINITY;
#pragma unroll
      for (int j = 0; j < kUnroll; ++j) {
        const int unit = u0 + j * kRowThreads;
        if (unit < nunits) {
          float x[8];
          raw[j].get(row, unit, V, full, -INFINITY, x);
#pragma unroll
          for (int k = 0; k < 8; ++k) cm = fmaxf(cm, x[k]);
        }
      }
      if (cm > m) {
        const float f = (m == -INFINITY) ? 0.f : ex2((m - cm) * k2);
        s *= f;
        c *= f;
        m = cm;
      }
      if (m != -INFINITY) {
        float tj[kUnroll];
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) {
          const int unit = u0 + j * kRowThreads;
          tj[j] = 0.f;
          if (unit < nunits) {
            float x[8], w[8];
            raw[j].get(row, unit, V, full, -INFINITY, x);
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = ex2((x[k] - m) * k2);
            tj[j] = sum8(w);
          }
        }
        const float chunk = tree_sum<kUnroll>(tj);
        const float y = chunk - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
      }
    }
    float M = warp_max(m);
    if (lane == 0) sc.f[warp] = M;
    row_sync(bar);
    M = sc.f[0];
#pragma unroll
    for (int w = 1; w < kRowWarps; ++w) M = fmaxf(M, sc.f[w]);
    const float mine = (m == -INFINITY) ? 0.f : (s - c) * ex2((m - M) * k2);
    dfloat acc = warp_sum_df(df_make(mine));
    if (lane == 0) { sc.hi[warp] = acc.hi; sc.lo[warp] = acc.lo; }
    row_sync(bar);
    if (tid == 0) {
      dfloat tot = {sc.hi[0], sc.lo[0]};
      for (int w = 1; w < kRowWarps; ++w) tot = df_add(tot, dfloat{sc.hi[w], sc.lo[w]});
      const double Z = df_to_d(tot);
      sc.out = RowStat{M, -1, Z, __frcp_rn(float(Z)), 0};   // fp32 reciprocal: no fp64 division
    }
  }
  row_sync(bar);
  const RowStat out = sc.out;
  row_sync(bar);
  return out;
}

template <typename T>
__global__ void __launch_bounds__(kRowThreads) verify_rows_kernel(VerifyDev a) {
  __shared__ RowScratch sc;
  // the first kernel of the call: the previous kernel on the stream may have produced the logits
  // or the tree flags, so wait for it before reading anything (the walk's early prologue relies
  // on this kernel having waited before it triggers)
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const T* row;
  RowStat* out;
  if (b < a.N) {
    // statistics of every internal node's target row (also in requests the walk will reject:
    // reading a row of [0, N) is always safe, and skipping them would need the validation first)
    if (!a.is_internal[b]) return;
    row = reinterpret_cast<const T*>(a.target) + size_t(b) * a.tld;
    out = a.tstat + b;
  } else {
    const int rr = b - a.N;
    row = reinterpret_cast<const T*>(a.draft) + size_t(rr) * a.dld;
    out = a.dstat + rr;
  }
  const RowStat st = row_stats<T>(row, a, sc, 1);
  if (threadIdx.x == 0) *out = st;
}

// ---- 2. walk -------------------------------------------------------------------------------
// fp64 runs on thread 0 (or one warp) only: GB300's fp64 rate is a small fraction of fp32, and a
// double division executed by all 32 warps of the block costs microseconds.
constexpr int kWalkThreads = 512;   // 128 registers per thread: four units' loads in flight
constexpr int kWalkWarps = kWalkThreads / 32;
static_assert(kWalkWarps <= 32, "one warp scans the per-warp totals");
// per-unit sums of a vocab pass stay in dynamic shared memory for vocabularies up to this many
// 8-element units (V <= 262144); the search step then rescans them instead of the rows
constexpr int kWalkMaxSmemUnits = 32768;
// a request's walk runs on a cluster of up to kWalkMaxCl CTAs, each with a vocabulary slice of
// at least kWalkMinUnits units (one per thread: below that a pass is bound by its barriers)
constexpr int kWalkMaxCl = 8;
constexpr int kWalkMinUnits = kWalkThreads;
// vocabularies from this size verify without the rows kernel by default (the kLazy walk)
constexpr int kLazyMinVocab = 65536;

// scratch of the block-wide vocabulary passes
struct PassSmem {
  dfloat wtot[kWalkWarps];   // per-warp inclusive sums of the threads' unit runs
  int wlast[kWalkWarps];     // per-warp last unit with mass
  int wfirst[kWalkWarps];    // per-warp first thread whose inclusive prefix passes theta
  float fred[kWalkWarps];
  int ired[kWalkWarps];
  double total;              // the pass's total mass (read by thread 0)
  int found;
  // read by the other CTAs of the cluster, per exchange (parity): this CTA's slice total (or
  // slice max) and its last unit with mass (or slice argmax)
  float px_hi[2], px_lo[2];
  int px_last[2];
  // the statistics pass of two rows: per-warp maxima and sums of the second row, and per
  // exchange (parity) this CTA's (max, sum hi, sum lo) of both rows
  float fred2[kWalkWarps];
  dfloat wtot2[kWalkWarps];
  float sx[2][6];
};

// This CTA's share of a request's walk: its rank in the request's cluster, the cluster's size,
// the slice length and its own units [u0, u1); npass counts exchanges (the parity of the
// exchange slot) and `arrived` records an early arrival on the kernel's last cluster barrier.
struct Slice {
  int rank, ncl, per, u0, u1;
  int npass;
  bool arrived;
};

// Publishes this CTA's (hi, lo, last) and returns, in lane k < ncl of every warp, rank k's
// values (other lanes: fill_hi, 0, -1).  One cluster barrier; the slot written two exchanges
// ago is free, since every CTA read it before arriving on the barrier of the exchange between.
__device__ __forceinline__ void slice_exchange(PassSmem& sh, Slice& sl, float hi, float lo,
                                               int last, float fill_hi, dfloat& rv, int& rl) {
  const int slot = sl.npass & 1;
  ++sl.npass;
  if (threadIdx.x == 0) {
    sh.px_hi[slot] = hi;
    sh.px_lo[slot] = lo;
    sh.px_last[slot] = last;
  }
  cluster_sync();
  const int lane = threadIdx.x & 31;
  rv = dfloat{fill_hi, 0.f};
  rl = -1;
  if (lane < sl.ncl) {
    rv.hi = ld_cluster_f32(&sh.px_hi[slot], lane);
    rv.lo = ld_cluster_f32(&sh.px_lo[slot], lane);
    rl = ld_cluster_s32(&sh.px_last[slot], lane);
  }
}

struct WalkSmem {
  int16_t par[SPEC_MAX_TREE];
  int16_t first_child[SPEC_MAX_TREE];
  int16_t next_sib[SPEC_MAX_TREE];
  int32_t path[SPEC_MAX_TREE];
  // per local node, gathered once in parallel before the walk
  int32_t tok[SPEC_MAX_TREE];
  int32_t drow[SPEC_MAX_TREE];     // draft row of the node's children (internal nodes); under
                                   // the multi-draft rule the row the node itself came from
  float xt[SPEC_MAX_TREE];         // target logit of the node's token in its parent's row
  float xd[SPEC_MAX_TREE];         // draft logit / probability of the node's token (parent's q)
  float uacc[SPEC_MAX_TREE], usamp[SPEC_MAX_TREE];
  float st_m[SPEC_MAX_TREE], sd_m[SPEC_MAX_TREE];     // row max of the node's target / draft row
  float st_iz[SPEC_MAX_TREE], sd_iz[SPEC_MAX_TREE];   // float(1 / Z) of those rows (draft
                                                      // stats per child under multi-draft)
  double st_Z[SPEC_MAX_TREE], sd_Z[SPEC_MAX_TREE];
  int32_t st_arg[SPEC_MAX_TREE];
  uint8_t dec0[SPEC_MAX_TREE];     // outcome of the node's plain ratio test u < p / q
  PassSmem ps;
  double C, Nk;                    // sibling residual state (thread 0 only)
  float Cf, Nf;
  int decision;
  int bad;                         // SPEC_REQ_* bits found by the validation
};

__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Calls f(unit, x) for this thread's units of the slice (sl.u0 + tid + i * kWalkThreads, in
// increasing i) with the unit's 8 values; kSlots units' loads stay in flight, each slot refilled
// as soon as its unit is unpacked.
template <int kSlots, typename T, typename F>
__device__ __forceinline__ void slice_units(const T* row, int V, float fill, const Slice& sl,
                                            F&& f) {
  const int full = V / 8, vend = min(full, sl.u1);
  const int first = sl.u0 + int(threadIdx.x);
  RawUnit<T> rv[kSlots];
#pragma unroll
  for (int j = 0; j < kSlots; ++j)
    if (first + j * kWalkThreads < vend) rv[j].load(row, first + j * kWalkThreads);
  for (int base = first; base < sl.u1; base += kSlots * kWalkThreads) {
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
      const int unit = base + j * kWalkThreads;
      if (unit < sl.u1) {
        float x[8];
        rv[j].get(row, unit, V, full, fill, x);
        const int nx = unit + kSlots * kWalkThreads;
        if (nx < vend) rv[j].load(row, nx);
        f(unit, x);
      }
    }
  }
}

// The row max: each CTA over its slice, then over the cluster's slices.
template <typename TT>
__device__ float slice_row_max(const TT* row, int V, PassSmem& sh, Slice& sl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float m = -INFINITY;
  slice_units<16 / int(sizeof(TT))>(row, V, -INFINITY, sl, [&](int, const float (&x)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) m = fmaxf(m, x[k]);
  });
  m = warp_max(m);
  if (lane == 0) sh.fred[warp] = m;
  __syncthreads();
  const float M = warp_max(lane < kWalkWarps ? sh.fred[lane] : -INFINITY);  // every warp reduces
  __syncthreads();
  dfloat rv;
  int rl;
  slice_exchange(sh, sl, M, 0.f, 0, -INFINITY, rv, rl);
  return warp_max(rv.hi);
}

// The lowest index of the row max: each CTA over its slice, then over the cluster's slices.
template <typename TT>
__device__ int slice_row_argmax(const TT* row, int V, PassSmem& sh, Slice& sl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float best = -INFINITY;
  int arg = 0x7fffffff;
  // a thread's units come in increasing order: a strict > keeps the lowest index
  slice_units<16 / int(sizeof(TT))>(row, V, -INFINITY, sl, [&](int unit, const float (&x)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (x[k] > best) { best = x[k]; arg = unit * 8 + k; }
  });
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ob = __shfl_xor_sync(0xffffffffu, best, off);
    int oa = __shfl_xor_sync(0xffffffffu, arg, off);
    if (ob > best || (ob == best && oa < arg)) { best = ob; arg = oa; }
  }
  if (lane == 0) { sh.fred[warp] = best; sh.ired[warp] = arg; }
  __syncthreads();
  float bb = lane < kWalkWarps ? sh.fred[lane] : -INFINITY;
  int ba = lane < kWalkWarps ? sh.ired[lane] : 0x7fffffff;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    float ob = __shfl_xor_sync(0xffffffffu, bb, off);
    int oa = __shfl_xor_sync(0xffffffffu, ba, off);
    if (ob > bb || (ob == bb && oa < ba)) { bb = ob; ba = oa; }
  }
  __syncthreads();
  dfloat rv;
  int rl;
  slice_exchange(sh, sl, bb, 0.f, ba, -INFINITY, rv, rl);
  float cb = rv.hi;
  int ca = lane < sl.ncl ? rl : 0x7fffffff;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, cb, off);
    const int oa = __shfl_xor_sync(0xffffffffu, ca, off);
    if (ob > cb || (ob == cb && oa < ca)) { cb = ob; ca = oa; }
  }
  return ca;
}

// The statistics of a node's target row and (drow non-null) of its draft row: each CTA reads its
// slices of both rows once, each thread keeping an online maximum and a Kahan-compensated sum of
// 2^((x - m) k2) per row (rescaled when the maximum grows), as the rows kernel forms them; the
// block combines the threads' maxima, then their sums rescaled to the block maximum in
// double-float; the CTAs exchange (max, sum) per row through distributed shared memory (one
// cluster barrier) and every CTA combines them in rank order, so all hold the same (m, Z).
template <typename TT, typename TD>
__device__ __noinline__ void slice_row_stats(const TT* trow, const TD* drow, int V, float k2, PassSmem& sh,
                                Slice& sl, float& mt, double& Zt, float& md, double& Zd) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool two = drow != nullptr;
  float m0 = -INFINITY, s0 = 0.f, c0 = 0.f, m1 = -INFINITY, s1 = 0.f, c1 = 0.f;
  // both rows in one sweep, each unit's pair of vectors loaded together (kUnits in flight)
  constexpr int kUnits = (sizeof(TT) == 2 && sizeof(TD) == 2) ? 4 : 2;
  const int full = V / 8, vend = min(full, sl.u1);
  auto add = [&](const float (&x)[8], float& m, float& sum, float& comp) {
    float cm = x[0];
#pragma unroll
    for (int k = 1; k < 8; ++k) cm = fmaxf(cm, x[k]);
    if (cm > m) {
      const float f = (m == -INFINITY) ? 0.f : ex2((m - cm) * k2);
      sum *= f;
      comp *= f;
      m = cm;
    }
    if (m != -INFINITY) {
      float w[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = ex2((x[k] - m) * k2);
      const float y = sum8(w) - comp;
      const float t = sum + y;
      comp = (t - sum) - y;
      sum = t;
    }
  };
  const int first = sl.u0 + tid;
  RawUnit<TT> rt[kUnits];
  RawUnit<TD> rd[kUnits];
#pragma unroll
  for (int j = 0; j < kUnits; ++j) {
    const int unit = first + j * kWalkThreads;
    if (unit < vend) {
      rt[j].load(trow, unit);
      if (two) rd[j].load(drow, unit);
    }
  }
  for (int base = first; base < sl.u1; base += kUnits * kWalkThreads) {
#pragma unroll
    for (int j = 0; j < kUnits; ++j) {
      const int unit = base + j * kWalkThreads;
      if (unit < sl.u1) {
        float xt[8], xd[8];
        rt[j].get(trow, unit, V, full, -INFINITY, xt);
        if (two) rd[j].get(drow, unit, V, full, -INFINITY, xd);
        const int nx = unit + kUnits * kWalkThreads;
        if (nx < vend) {
          rt[j].load(trow, nx);
          if (two) rd[j].load(drow, nx);
        }
        add(xt, m0, s0, c0);
        if (two) add(xd, m1, s1, c1);
      }
    }
  }
  // the block: maxima, then the threads' sums rescaled to them
  {
    const float w0 = warp_max(m0), w1 = warp_max(m1);
    if (lane == 0) { sh.fred[warp] = w0; sh.fred2[warp] = w1; }
  }
  __syncthreads();
  const float B0 = warp_max(lane < kWalkWarps ? sh.fred[lane] : -INFINITY);
  const float B1 = warp_max(lane < kWalkWarps ? sh.fred2[lane] : -INFINITY);
  {
    const dfloat t0 = warp_sum_df(df_make(m0 == -INFINITY ? 0.f : (s0 - c0) * ex2((m0 - B0) * k2)));
    const dfloat t1 = warp_sum_df(df_make(m1 == -INFINITY ? 0.f : (s1 - c1) * ex2((m1 - B1) * k2)));
    if (lane == 0) { sh.wtot[warp] = t0; sh.wtot2[warp] = t1; }
  }
  __syncthreads();
  const dfloat S0 = warp_sum_df(lane < kWalkWarps ? sh.wtot[lane] : df_make(0.f));
  const dfloat S1 = warp_sum_df(lane < kWalkWarps ? sh.wtot2[lane] : df_make(0.f));
  // the cluster: every rank's (max, sum) of both rows, combined in rank order
  const int slot = sl.npass & 1;
  ++sl.npass;
  if (tid == 0) {
    sh.sx[slot][0] = B0; sh.sx[slot][1] = S0.hi; sh.sx[slot][2] = S0.lo;
    sh.sx[slot][3] = B1; sh.sx[slot][4] = S1.hi; sh.sx[slot][5] = S1.lo;
  }
  cluster_sync();
  float r0 = -INFINITY, r1 = -INFINITY;
  dfloat q0 = df_make(0.f), q1 = df_make(0.f);
  if (lane < sl.ncl) {
    r0 = ld_cluster_f32(&sh.sx[slot][0], lane);
    q0 = dfloat{ld_cluster_f32(&sh.sx[slot][1], lane), ld_cluster_f32(&sh.sx[slot][2], lane)};
    r1 = ld_cluster_f32(&sh.sx[slot][3], lane);
    q1 = dfloat{ld_cluster_f32(&sh.sx[slot][4], lane), ld_cluster_f32(&sh.sx[slot][5], lane)};
  }
  mt = warp_max(r0);
  md = warp_max(r1);
  // a rank's double-float sum times its rescale factor f = 2^((r - M) k2), exactly rounded parts
  auto scaled = [&](dfloat q, float r, float M) -> dfloat {
    if (r == -INFINITY) return df_make(0.f);
    const float f = ex2((r - M) * k2);
    const float hi = q.hi * f;
    return dfloat{hi, fmaf(q.hi, f, -hi) + q.lo * f};
  };
  const dfloat i0 = warp_scan_df(scaled(q0, r0, mt), lane);
  const dfloat i1 = warp_scan_df(scaled(q1, r1, md), lane);
  Zt = df_to_d(dfloat{__shfl_sync(0xffffffffu, i0.hi, sl.ncl - 1), __shfl_sync(0xffffffffu, i0.lo, sl.ncl - 1)});
  Zd = df_to_d(dfloat{__shfl_sync(0xffffffffu, i1.hi, sl.ncl - 1), __shfl_sync(0xffffffffu, i1.lo, sl.ncl - 1)});
}

// Element weights of the distribution being summed / sampled: p itself (bonus token, up to the
// constant 1 / Z) or the sibling residual max(0, p - C q).
struct WeightFn {
  bool residual, probs;
  float mt, md, k2, invZt, invZd, C;
  __device__ __forceinline__ void operator()(const float (&xt)[8], const float (&xd)[8],
                                             float (&w)[8]) const {
    if (!residual) {
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = ex2((xt[k] - mt) * k2);
      return;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float p = ex2((xt[k] - mt) * k2) * invZt;
      const float q = probs ? xd[k] : ex2((xd[k] - md) * k2) * invZd;
      w[k] = fmaxf(0.f, p - C * q);
    }
  }
  // the functor interface of vocab_pass
  __device__ __forceinline__ bool loads_t() const { return true; }
  __device__ __forceinline__ bool loads_d() const { return residual; }
  __device__ __forceinline__ bool stores() const { return false; }
  __device__ __forceinline__ void apply(int, const float (&xt)[8], const float (&xd)[8],
                                        float (&w)[8]) const {
    (*this)(xt, xd, w);
  }
  __device__ __forceinline__ void store(int, const float (&)[8]) const {}
  template <typename TT, typename TD>
  __device__ __forceinline__ void unit(const TT* trow, const TD* drow, int u, int V, int full,
                                       float (&w)[8]) const {
    float xt[8], xd[8];
    load8(trow, u, V, full, -INFINITY, xt);
    if (residual) load8(drow, u, V, full, probs ? 0.f : -INFINITY, xd);
    (*this)(xt, xd, w);
  }
};

// Weights of the multi-draft residual: w = max(0, S(x) - Nprev q_c(x)), where S is the running
// residual R_{j-1} from the scratch row `src` (or p itself, src == nullptr, before the first
// rejection) and q_c the rejected sibling's own draft distribution.  An update pass stores w to
// `dst` (R_j); the final draw passes dst == nullptr.
struct MultiFn {
  bool probs;
  float mt, md, k2, invZt, invZd, Nprev;
  const float* src;
  float* dst;
  int V;
  __device__ __forceinline__ bool loads_t() const { return src == nullptr; }
  __device__ __forceinline__ bool loads_d() const { return true; }
  __device__ __forceinline__ bool stores() const { return dst != nullptr; }
  __device__ __forceinline__ void apply(int u, const float (&xt)[8], const float (&xd)[8],
                                        float (&w)[8]) const {
    float sv[8];
    if (src) {
      const float4 a = *reinterpret_cast<const float4*>(src + size_t(u) * 8);
      const float4 b = *reinterpret_cast<const float4*>(src + size_t(u) * 8 + 4);
      sv[0] = a.x; sv[1] = a.y; sv[2] = a.z; sv[3] = a.w;
      sv[4] = b.x; sv[5] = b.y; sv[6] = b.z; sv[7] = b.w;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (u * 8 + k >= V) sv[k] = 0.f;   // the row's padding was never written
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) sv[k] = ex2((xt[k] - mt) * k2) * invZt;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float q = probs ? xd[k] : ex2((xd[k] - md) * k2) * invZd;
      w[k] = fmaxf(0.f, sv[k] - Nprev * q);
    }
  }
  __device__ __forceinline__ void store(int u, const float (&w)[8]) const {
    *reinterpret_cast<float4*>(dst + size_t(u) * 8) = make_float4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<float4*>(dst + size_t(u) * 8 + 4) = make_float4(w[4], w[5], w[6], w[7]);
  }
  template <typename TT, typename TD>
  __device__ __forceinline__ void unit(const TT* trow, const TD* drow, int u, int Vv, int full,
                                       float (&w)[8]) const {
    float xt[8], xd[8];
    if (!src) load8(trow, u, Vv, full, -INFINITY, xt);
    load8(drow, u, Vv, full, probs ? 0.f : -INFINITY, xd);
    apply(u, xt, xd, w);
  }
};

struct PassResult {
  int tok;     // sampled token (search passes, in the owner CTA only), -1 otherwise
  bool pos;    // the total mass is > 0
  int owner;   // search passes with mass: the rank whose slice holds the token
};

// double-float value minus theta (th_hi + th_lo) is > 0
__device__ __forceinline__ bool df_above(dfloat x, float th_hi, float th_lo) {
  return ((x.hi - th_hi) + (x.lo - th_lo)) > 0.f;
}

// Pass over the vocabulary, each CTA of the cluster over its slice: total mass of the weights
// (sh.total, thread 0; the same value in every CTA) and, when `search`, the smallest token x with
// sum_{y<=x} w(y) > u * total.  Phase 1 reads the slice (kUnits units' loads in flight per
// thread); a mass pass ends with a block reduction of the threads' sums and the exchange of the
// slice totals, a search pass stores every 8-element unit's weight sum in shared memory and
// continues.  Phase 2 gives
// thread t the contiguous units [t * run, (t + 1) * run) of the slice: a block scan of the
// threads' double-float run sums gives every thread its prefix within the slice, the CTAs
// exchange their slice totals and scan them in rank order, and in the CTA whose range holds
// theta the first thread whose inclusive prefix passes it walks its units, then the crossing
// unit's 8 elements.  No fp64: theta is a double-float product.  Without `usum` (very large
// vocabularies) phase 2 recomputes unit sums.  A search pass with mass is the walk's final
// draw: each CTA arrives on the kernel's last cluster barrier right after its remote reads.
template <typename TT, typename TD, typename Fn>
__device__ PassResult vocab_pass(const TT* trow, const TD* drow, int V, const Fn& fn,
                                 bool search, float u, float* usum, PassSmem& sh, Slice& sl) {
  constexpr int kUnits = (sizeof(TT) == 2 && sizeof(TD) == 2) ? 4 : 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int full = V / 8;
  const int s0 = sl.u0, s1 = sl.u1, nu = s1 - s0;
  const int vend = min(full, s1);   // units of the slice read as whole vectors end here
  // phase 1, thread t's units s0 + t + i * kWalkThreads: kUnits units' loads in flight, each
  // slot refilled as soon as its unit is unpacked.  A search pass keeps the unit sums; a mass
  // pass only the thread's total.
  dfloat mine1 = df_make(0.f);
  if (!search || usum || fn.stores()) {
    const int first = s0 + tid;
    RawUnit<TT> rt[kUnits];
    RawUnit<TD> rd[kUnits];
#pragma unroll
    for (int j = 0; j < kUnits; ++j) {
      const int unit = first + j * kWalkThreads;
      if (unit < vend) {
        if (fn.loads_t()) rt[j].load(trow, unit);
        if (fn.loads_d()) rd[j].load(drow, unit);
      }
    }
    for (int base = first; base < s1; base += kUnits * kWalkThreads) {
#pragma unroll
      for (int j = 0; j < kUnits; ++j) {
        const int unit = base + j * kWalkThreads;
        if (unit < s1) {
          float xt[8], xd[8], w[8];
          if (fn.loads_t()) rt[j].get(trow, unit, V, full, -INFINITY, xt);
          if (fn.loads_d()) rd[j].get(drow, unit, V, full, fn.probs ? 0.f : -INFINITY, xd);
          const int nx = unit + kUnits * kWalkThreads;
          if (nx < vend) {
            if (fn.loads_t()) rt[j].load(trow, nx);
            if (fn.loads_d()) rd[j].load(drow, nx);
          }
          fn.apply(unit, xt, xd, w);
          if (fn.stores()) fn.store(unit, w);
          const float su = sum8(w);
          if (!search) mine1 = df_add_f(mine1, su);
          else if (usum) usum[unit - s0] = su;
        }
      }
    }
  }
  if (!search) {
    // a mass pass: the slice total is a block reduction of the threads' totals
    const dfloat wt = warp_sum_df(mine1);
    if (lane == 0) sh.wtot[warp] = wt;
    __syncthreads();
    const dfloat ctot = warp_sum_df(lane < kWalkWarps ? sh.wtot[lane] : df_make(0.f));
    dfloat rv;
    int rl;
    slice_exchange(sh, sl, ctot.hi, ctot.lo, -1, 0.f, rv, rl);
    const dfloat rincl = warp_scan_df(rv, lane);
    const dfloat total = {__shfl_sync(0xffffffffu, rincl.hi, sl.ncl - 1),
                          __shfl_sync(0xffffffffu, rincl.lo, sl.ncl - 1)};
    if (tid == 0) sh.total = df_to_d(total);
    // no barrier: every read of sh.wtot came before the exchange's cluster barrier
    return PassResult{-1, total.hi > 0.f, -1};
  }
  __syncthreads();
  auto unit_sum = [&](int unit) -> float {
    if (usum) return usum[unit - s0];
    float w[8];
    fn.unit(trow, drow, unit, V, full, w);
    return sum8(w);
  };
  // phase 2: this thread's run of units, scanned across the block
  const int run = (nu + kWalkThreads - 1) / kWalkThreads;
  const int a0 = s0 + min(tid * run, nu), a1 = min(a0 + run, s1);
  dfloat mine = df_make(0.f);
  int lastp = -1;
  for (int unit = a0; unit < a1; ++unit) {
    const float su = unit_sum(unit);
    mine = df_add_f(mine, su);
    if (su > 0.f) lastp = unit;
  }
  const dfloat incl_w = warp_scan_df(mine, lane);
  dfloat excl_w = df_shfl_up(incl_w, 1);
  if (lane == 0) excl_w = df_make(0.f);
  lastp = warp_max_i(lastp);
  if (lane == 31) sh.wtot[warp] = incl_w;
  if (lane == 0) sh.wlast[warp] = lastp;
  __syncthreads();
  // every warp scans the warp totals: its own base and the slice total
  const dfloat wsc = warp_scan_df(lane < kWalkWarps ? sh.wtot[lane] : df_make(0.f), lane);
  dfloat wex = df_shfl_up(wsc, 1);
  if (lane == 0) wex = df_make(0.f);
  const dfloat wbase = {__shfl_sync(0xffffffffu, wex.hi, warp), __shfl_sync(0xffffffffu, wex.lo, warp)};
  const dfloat ctot = {__shfl_sync(0xffffffffu, wsc.hi, 31), __shfl_sync(0xffffffffu, wsc.lo, 31)};
  const int fb = warp_max_i(lane < kWalkWarps ? sh.wlast[lane] : -1);   // slice's last unit with mass
  // the cluster: slice totals in rank order
  dfloat rv;
  int rl;
  slice_exchange(sh, sl, ctot.hi, ctot.lo, fb, 0.f, rv, rl);
  const dfloat rincl = warp_scan_df(rv, lane);
  const dfloat total = {__shfl_sync(0xffffffffu, rincl.hi, sl.ncl - 1),
                        __shfl_sync(0xffffffffu, rincl.lo, sl.ncl - 1)};
  const int lastall = warp_max_i(rl);
  const bool pos = total.hi > 0.f;
  if (tid == 0) sh.total = df_to_d(total);
  if (!pos) {
    __syncthreads();   // sh is reused by the next pass
    return PassResult{-1, pos, -1};
  }
  cluster_arrive();   // no CTA reads another's shared memory after the final draw's exchange
  sl.arrived = true;
  // theta = u * total as a double-float (exact product of u and total.hi, plus u * total.lo)
  const float ph = u * total.hi;
  const float pl = fmaf(u, total.hi, -ph) + u * total.lo;
  const float th_hi = ph + pl, th_lo = pl - (th_hi - ph);
  const unsigned rm = __ballot_sync(0xffffffffu, lane < sl.ncl && df_above(rincl, th_hi, th_lo));
  const int cstar = rm ? __ffs(rm) - 1 : -1;
  // no rank crossed (theta at the total by rounding): the last unit with mass decides
  const int owner = cstar >= 0 ? cstar : (lastall >= 0 ? lastall / sl.per : -1);
  if (owner != sl.rank) return PassResult{-1, pos, owner};
  dfloat rex = df_shfl_up(rincl, 1);
  if (lane == 0) rex = df_make(0.f);
  const dfloat rbase = {__shfl_sync(0xffffffffu, rex.hi, sl.rank),
                        __shfl_sync(0xffffffffu, rex.lo, sl.rank)};
  if (tid == 0) sh.found = -1;
  if (cstar == sl.rank) {
    const dfloat prefix = df_add(rbase, df_add(wbase, excl_w));
    const bool c = a0 < a1 && df_above(df_add(rbase, df_add(wbase, incl_w)), th_hi, th_lo);
    const unsigned cm = __ballot_sync(0xffffffffu, c);
    if (lane == 0) sh.wfirst[warp] = cm ? warp * 32 + __ffs(cm) - 1 : 0x7fffffff;
    __syncthreads();
    int first = 0x7fffffff;
#pragma unroll
    for (int w = 0; w < kWalkWarps; ++w) first = min(first, sh.wfirst[w]);
    if (tid == first) {
      dfloat cum = prefix;
      int cross_unit = -1, last_pos_unit = -1;
      for (int unit = a0; unit < a1; ++unit) {
        const float su = unit_sum(unit);
        const dfloat nx = df_add_f(cum, su);
        if (su > 0.f) last_pos_unit = unit;
        if (df_above(nx, th_hi, th_lo)) { cross_unit = unit; break; }
        cum = nx;
      }
      // rounding can leave the crossing inside the run total only: take its last live unit
      const int cu = cross_unit >= 0 ? cross_unit : last_pos_unit;
      int tok = -1, lastpos = -1;
      if (cu >= 0) {
        float w[8];
        fn.unit(trow, drow, cu, V, full, w);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          cum = df_add_f(cum, w[k]);
          if (w[k] > 0.f) lastpos = cu * 8 + k;
          if (tok < 0 && cross_unit >= 0 && df_above(cum, th_hi, th_lo)) tok = cu * 8 + k;
        }
      }
      sh.found = tok >= 0 ? tok : lastpos;
    }
  }
  __syncthreads();
  int tok = sh.found;
  if (tok < 0) {
    // no thread crossed (theta at the slice's end by rounding): its last element with mass
    if (tid == 0 && fb >= 0) {
      float w[8];
      fn.unit(trow, drow, fb, V, full, w);
      int lp = -1;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (w[k] > 0.f) lp = fb * 8 + k;
      sh.found = lp;
    }
    __syncthreads();
    tok = sh.found;
  }
  __syncthreads();   // sh is reused by the next pass
  return PassResult{tok, pos, owner};
}

// Thread 0: the ratio test of a later sibling under the sibling residual rule,
// u < max(0, p - C q) / (N q) written as u * N * q < max(0, p - C q) (q >= 0), with both sides
// multiplied by Zt (and Zd for draft logits), p = et / Zt, q = ed / Zd: no fp64 division (a
// long dependent chain on GB300's fp64 unit, on the walk's critical path).
template <typename TT, typename TD>
__device__ bool residual_ratio_test(const VerifyDev& a, const WalkSmem& sh, int node, int c) {
  const double et = double(expf((sh.xt[c] - sh.st_m[node]) * a.inv_tau));
  const double Zt = sh.st_Z[node];
  const double u = double(sh.uacc[c]);
  if (a.probs) {
    const double qZ = double(sh.xd[c]) * Zt;   // q Zt
    return u * (sh.Nk * qZ) < fmax(0.0, et - sh.C * qZ);
  }
  const double ed = double(expf((sh.xd[c] - sh.sd_m[node]) * a.inv_tau));
  const double qZ = ed * Zt;                    // q Zt Zd
  return u * (sh.Nk * qZ) < fmax(0.0, et * sh.sd_Z[node] - sh.C * qZ);
}

// Thread 0: the ratio test of a later sibling c under the multi-draft rule,
// u < R_{j-1}(tok) / (N_{j-1} q_c(tok)) written as u * N_{j-1} * q_c(tok) < R_{j-1}(tok) (times Zd
// for draft logits), with R_{j-1} the scratch row the previous update pass stored.
__device__ bool multi_ratio_test(const VerifyDev& a, const WalkSmem& sh, int c, const float* src) {
  const double num = double(src[sh.tok[c]]);
  if (a.probs) return double(sh.uacc[c]) * (sh.Nk * double(sh.xd[c])) < num;
  const double ed = double(expf((sh.xd[c] - sh.sd_m[c]) * a.inv_tau));
  return double(sh.uacc[c]) * (sh.Nk * ed) < num * sh.sd_Z[c];
}

// kLazy: no rows kernel before it; the walk forms the statistics of the nodes it visits (a
// separate instance, so that the other keeps its register allocation)
template <typename TT, typename TD, bool kMulti, bool kLazy>
__global__ void __launch_bounds__(kWalkThreads, 1) verify_walk_kernel(VerifyDev a) {
  __shared__ WalkSmem sh;
  extern __shared__ float usum_dyn[];
  // After the rows kernel (which waited for everything before this call before it let this
  // kernel launch), everything up to the row statistics is already complete, so validation and
  // the gather of the tree run while the rows kernel may still be running; pdl_wait() comes
  // before the statistics and before any store.  Without a rows kernel, wait first.
  if (!a.after_rows) pdl_wait();
  pdl_trigger();
  const int rank = cluster_rank(), ncl = cluster_size();
  const int r = blockIdx.x / ncl;
  const int tid = threadIdx.x;
  int32_t* path_row = a.path + size_t(r) * a.max_path;
  int32_t* tok_row = a.out_tokens + size_t(r) * a.max_path;
  // validation: the node range, then every node's token, depth and (tau > 0) draft row
  const int st0 = a.req_status[r];
  const int o = a.node_offset[r];
  const int T = a.node_offset[r + 1] - o;
  const bool range_ok = o >= 0 && T >= 1 && T <= a.T_max && o + T <= a.N;
  if (tid == 0) sh.bad = range_ok ? 0 : SPEC_REQ_BAD_SIZE;
  __syncthreads();
  if (st0 == 0 && range_ok) {
    int bad = 0;
    for (int i = tid; i < T; i += kWalkThreads) {
      const int n = o + i;
      if (i > 0) {
        const int tok = a.tokens[n];
        if (tok < 0 || tok >= a.V) bad |= SPEC_REQ_BAD_TOKEN;
      }
      if (a.depth[n] + 1 > a.max_path) bad |= SPEC_REQ_BAD_DEPTH;
      // the draft rows read: the children's row of every internal node, or under the
      // multi-draft rule every drafted node's own row
      if (a.tau > 0.f && (kMulti ? i > 0 : a.is_internal[n] != 0)) {
        const int dr = a.draft_row[n];
        if (dr < 0 || dr >= a.R) bad |= SPEC_REQ_BAD_DRAFT_ROW;
      }
    }
    if (bad) atomicOr(&sh.bad, bad);
  }
  __syncthreads();
  const int st = st0 | sh.bad;
  if (st != 0) {
    // the same exit in every CTA of the cluster (the same data), before any cluster barrier
    pdl_wait();
    if (rank == 0) {
      if (tid == 0 && sh.bad) atomicOr(&a.req_status[r], sh.bad);
      for (int k = tid; k < a.max_path; k += kWalkThreads) { path_row[k] = -1; tok_row[k] = -1; }
      if (tid == 0) {
        a.out_len[r] = 0;
        a.n_acc[r] = -1;
        if (a.rejections) a.rejections[r] = 0;
      }
    }
    return;
  }
  Slice sl;
  {
    const int nunits = (a.V + 7) / 8;
    sl.rank = rank;
    sl.ncl = ncl;
    sl.per = a.walk_per;
    sl.u0 = min(rank * a.walk_per, nunits);
    sl.u1 = min(sl.u0 + a.walk_per, nunits);
    sl.npass = 0;
    sl.arrived = false;
  }
  float* usum = a.walk_per <= kWalkMaxSmemUnits ? usum_dyn : nullptr;
  const TT* target = reinterpret_cast<const TT*>(a.target);
  const TD* draft = reinterpret_cast<const TD*>(a.draft);
  const bool greedy = a.tau == 0.f;
  // gather, in parallel, everything the scalar part of the walk will read: tree links, tokens,
  // uniforms and, for every non-root node, its token's target and draft values in its parent's
  // rows (the operands of its ratio test); then, once the rows kernel is done, the row
  // statistics of internal nodes and every node's plain ratio test
  for (int i = tid; i < T; i += kWalkThreads) {
    const int p = a.parent[o + i];
    const int t = a.tokens[o + i];
    sh.par[i] = int16_t(p);
    sh.tok[i] = t;
    sh.first_child[i] = -1;
    sh.next_sib[i] = -1;
    sh.uacc[i] = a.uniforms[2 * size_t(o + i)];
    sh.usamp[i] = a.uniforms[2 * size_t(o + i) + 1];
    if (!greedy && (kMulti ? i > 0 : a.is_internal[o + i] != 0)) sh.drow[i] = a.draft_row[o + i];
    if (i > 0 && !greedy) {
      sh.xt[i] = elem<TT>::load1(target + size_t(o + p) * a.tld + t);
      const int dr = kMulti ? a.draft_row[o + i] : a.draft_row[o + p];
      sh.xd[i] = elem<TD>::load1(draft + size_t(dr) * a.dld + t);
    }
  }
  __syncthreads();
  for (int i = tid; i < T; i += kWalkThreads) {
    if (i > 0) {
      const int p = sh.par[i];
      int nxt = -1;
      for (int k = i + 1; k < T; ++k)
        if (sh.par[k] == p) { nxt = k; break; }
      sh.next_sib[i] = int16_t(nxt);
      // first child of p: the sibling with no smaller sibling
      bool first = true;
      for (int k = p + 1; k < i; ++k)
        if (sh.par[k] == p) { first = false; break; }
      if (first) sh.first_child[p] = int16_t(i);
    }
  }
  pdl_wait();   // the rows kernel's statistics are complete
  constexpr bool lazy = kLazy && !kMulti;   // else the statistics come from the rows kernel
  for (int i = tid; i < T && !lazy; i += kWalkThreads) {
    if (a.is_internal[o + i]) {
      const RowStat ts = a.tstat[o + i];
      sh.st_m[i] = ts.m;
      sh.st_Z[i] = ts.Z;
      sh.st_iz[i] = ts.inv_Z;
      sh.st_arg[i] = ts.arg;
    }
    // draft statistics: of the node's children's row, or (multi-draft) of its own row
    if (kMulti ? i > 0 : a.is_internal[o + i] != 0) {
      if (!greedy) {
        if (!a.probs) {
          const RowStat ds = a.dstat[sh.drow[i]];
          sh.sd_m[i] = ds.m;
          sh.sd_Z[i] = ds.Z;
          sh.sd_iz[i] = ds.inv_Z;
        } else {
          sh.sd_m[i] = 0.f;
          sh.sd_Z[i] = 1.0;
          sh.sd_iz[i] = 1.f;
        }
      }
    }
  }
  __syncthreads();
  // the plain ratio test u < p / q of node i from its parent's statistics, as
  // u * Zt < exp(((xt - mt) - (xd - md)) / tau) * Zd for draft logits and
  // u * q * Zt < exp((xt - mt) / tau) for draft probabilities
  auto plain_test = [&](int i) {
    const int p = sh.par[i];
    const int qi = kMulti ? i : p;   // whose draft statistics hold q for node i
    const double u = double(sh.uacc[i]);
    bool acc;
    if (!a.probs) {
      const float e = expf(((sh.xt[i] - sh.st_m[p]) - (sh.xd[i] - sh.sd_m[qi])) * a.inv_tau);
      acc = u * sh.st_Z[p] < double(e) * sh.sd_Z[qi];
    } else {
      const float e = expf((sh.xt[i] - sh.st_m[p]) * a.inv_tau);
      acc = u * double(sh.xd[i]) * sh.st_Z[p] < double(e);
    }
    sh.dec0[i] = acc ? 1 : 0;
  };
  if (!greedy && !lazy)
    for (int i = tid; i < T; i += kWalkThreads)
      if (i > 0) plain_test(i);
  if (tid == 0) sh.path[0] = 0;
  __syncthreads();

  // this CTA's slice of a row (its whole 8-element units) moves into L2 ahead of the passes'
  // loads: the passes keep only a few units per thread in flight, and a node's rejected
  // siblings read the same two slices pass after pass
  auto prefetch_slice = [&](const void* row, int es) {
    constexpr int kPiece = 16384;
    const int u1 = min(sl.u1, a.V / 8);
    if (u1 <= sl.u0) return;
    const char* p0 = static_cast<const char*>(row) + size_t(sl.u0) * 8 * es;
    const int bytes = (u1 - sl.u0) * 8 * es;
    for (int i = tid; i * kPiece < bytes; i += kWalkThreads)
      prefetch_l2_bulk(p0 + size_t(i) * kPiece, min(kPiece, bytes - i * kPiece));
  };
  int node = 0, npath = 1, rejections = 0, final_tok = -1, owner = 0;
  while (true) {
    const TT* trow = target + size_t(o + node) * a.tld;
    const int fc = sh.first_child[node];
    if (!greedy) {
      prefetch_slice(trow, int(sizeof(TT)));
      if (fc >= 0 && !kMulti) prefetch_slice(draft + size_t(sh.drow[node]) * a.dld, int(sizeof(TD)));
    }
    if constexpr (lazy) if (!greedy && fc >= 0) {
      // this node's statistics, then its children's plain ratio tests
      const TD* dr = a.probs ? nullptr : draft + size_t(sh.drow[node]) * a.dld;
      float mt = 0.f, md = 0.f;
      double Zt = 1.0, Zd = 1.0;
      slice_row_stats<TT, TD>(trow, dr, a.V, a.k2, sh.ps, sl, mt, Zt, md, Zd);
      if (tid == 0) {
        sh.st_m[node] = mt;
        sh.st_Z[node] = Zt;
        sh.st_iz[node] = __frcp_rn(float(Zt));
        sh.sd_m[node] = dr ? md : 0.f;
        sh.sd_Z[node] = dr ? Zd : 1.0;
        sh.sd_iz[node] = dr ? __frcp_rn(float(Zd)) : 1.f;
      }
      __syncthreads();
      for (int i = tid; i < T; i += kWalkThreads)
        if (i > 0 && sh.par[i] == node) plain_test(i);
      __syncthreads();
    }
    if (greedy) {
      const int best = (fc >= 0 && !lazy) ? sh.st_arg[node] : slice_row_argmax(trow, a.V, sh.ps, sl);
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
    const float u_samp = sh.usamp[node];
    if (fc < 0) {  // leaf: bonus token from p_leaf
      WeightFn fn{};
      fn.residual = false;
      fn.mt = slice_row_max(trow, a.V, sh.ps, sl);
      fn.k2 = a.k2;
      const PassResult pr = vocab_pass(trow, draft, a.V, fn, true, u_samp, usum, sh.ps, sl);
      final_tok = pr.tok;
      owner = pr.owner;
      break;
    }
    if (kMulti) {
      // siblings from different draft models: R_0 = p, N_0 = 1; a rejected child c gives
      // R_j = max(0, R_{j-1} - N_{j-1} q_c) (stored), N_j = sum R_j; the last sibling's residual
      // is drawn from directly
      float* const rows2 = a.rbuf + size_t(r) * 2 * a.rld;   // this request's two rows
      const float* src = nullptr;
      int flip = 0, accepted = -1, last = -1;
      bool from_p = false;
      if (tid == 0) { sh.Nk = 1.0; sh.Nf = 1.f; }
      __syncthreads();
      for (int c = fc; c >= 0; c = sh.next_sib[c]) {
        bool acc;
        if (c == fc) {
          acc = sh.dec0[c] != 0;
        } else {
          if (tid == 0) sh.decision = multi_ratio_test(a, sh, c, src);
          __syncthreads();
          acc = sh.decision != 0;
          __syncthreads();
        }
        if (acc) { accepted = c; break; }
        ++rejections;
        last = c;
        if (sh.next_sib[c] < 0) break;
        MultiFn upd{};
        upd.probs = a.probs != 0;
        upd.mt = sh.st_m[node]; upd.k2 = a.k2; upd.invZt = sh.st_iz[node];
        upd.md = sh.sd_m[c]; upd.invZd = sh.sd_iz[c];
        upd.Nprev = sh.Nf;
        upd.src = src;
        upd.dst = rows2 + flip * a.rld;
        upd.V = a.V;
        const TD* drow_c = draft + size_t(sh.drow[c]) * a.dld;
        const PassResult pr = vocab_pass(trow, drow_c, a.V, upd, false, 0.f, usum, sh.ps, sl);
        if (tid == 0) { sh.Nk = sh.ps.total; sh.Nf = float(sh.ps.total); }
        __syncthreads();
        if (!pr.pos) { from_p = true; break; }
        src = rows2 + flip * a.rld;
        flip ^= 1;
      }
      if (accepted >= 0) {
        if (tid == 0) sh.path[npath] = accepted;
        ++npath;
        node = accepted;
        continue;
      }
      if (!from_p) {
        MultiFn fin{};
        fin.probs = a.probs != 0;
        fin.mt = sh.st_m[node]; fin.k2 = a.k2; fin.invZt = sh.st_iz[node];
        fin.md = sh.sd_m[last]; fin.invZd = sh.sd_iz[last];
        fin.Nprev = sh.Nf;
        fin.src = src;
        fin.dst = nullptr;
        fin.V = a.V;
        const TD* drow_c = draft + size_t(sh.drow[last]) * a.dld;
        const PassResult pr = vocab_pass(trow, drow_c, a.V, fin, true, u_samp, usum, sh.ps, sl);
        final_tok = pr.tok;
        owner = pr.owner;
        if (!pr.pos) from_p = true;
      }
      if (from_p) {
        WeightFn fn{};
        fn.residual = false;
        fn.mt = sh.st_m[node];
        fn.k2 = a.k2;
        const PassResult pr = vocab_pass(trow, draft, a.V, fn, true, u_samp, usum, sh.ps, sl);
        final_tok = pr.tok;
        owner = pr.owner;
      }
      break;
    }
    const TD* drow = draft + size_t(sh.drow[node]) * a.dld;
    WeightFn res{};
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
        // C_1 = C_0 + N_0 = 0 + 1
        if (!acc && a.residual_rule) {
          if (tid == 0) sh.C = 1.0;
          res.C = 1.f;
        }
      } else {
        // thread 0 decides and, on a rejection, advances C_{k+1} = C_k + N_k; one barrier
        // publishes both (they are rewritten only after the next pass's barriers)
        if (tid == 0) {
          const bool d = residual_ratio_test<TT, TD>(a, sh, node, c);
          sh.decision = d;
          if (!d) {
            sh.C += sh.Nk;
            sh.Cf = float(sh.C);
          }
        }
        __syncthreads();
        acc = sh.decision != 0;
        if (!acc) res.C = sh.Cf;
      }
      if (acc) { accepted = c; break; }
      ++rejections;
      if (a.residual_rule) {
        // N_{k+1} = sum_x max(0, p(x) - C_{k+1} q(x))
        // after the last sibling the final draw below yields N_{k+1} itself
        if (sh.next_sib[c] < 0) break;
        const PassResult pr = vocab_pass(trow, drow, a.V, res, false, 0.f, usum, sh.ps, sl);
        if (tid == 0) sh.Nk = sh.ps.total;
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
      const PassResult pr = vocab_pass(trow, drow, a.V, res, true, u_samp, usum, sh.ps, sl);
      final_tok = pr.tok;
      owner = pr.owner;
      if (!pr.pos) from_p = true;
    }
    if (from_p) {
      WeightFn fn{};
      fn.residual = false;
      fn.mt = res.mt;
      fn.k2 = a.k2;
      const PassResult pr = vocab_pass(trow, draft, a.V, fn, true, u_samp, usum, sh.ps, sl);
      final_tok = pr.tok;
      owner = pr.owner;
    }
    break;
  }
  if (owner < 0) { owner = 0; final_tok = -1; }   // a row without mass: no token
  __syncthreads();
  // rank 0 writes the outputs, the owner of the final draw its token
  if (rank == 0) {
    for (int k = tid; k < a.max_path; k += kWalkThreads) {
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
  // no CTA leaves while another may still read its shared memory
  if (!sl.arrived) cluster_arrive();
  cluster_wait();
}

struct VerifyWs {
  size_t tstat, dstat, rbuf, total;
  int64_t rld;   // floats per residual row (multi-draft), a multiple of 64
};

// multi_B > 0: the multi-draft rule's two residual rows per request (multi_B requests, vocab V)
static VerifyWs verify_ws_layout(int N, int R, int multi_B = 0, int V = 0) {
  VerifyWs w;
  size_t off = 0;
  w.tstat = off; off = align_up(off + sizeof(RowStat) * size_t(N > 0 ? N : 1), 256);
  w.dstat = off; off = align_up(off + sizeof(RowStat) * size_t(R > 0 ? R : 1), 256);
  w.rld = int64_t(align_up(size_t(V > 0 ? V : 1), 64));
  w.rbuf = off;
  if (multi_B > 0) off = align_up(off + sizeof(float) * 2 * size_t(multi_B) * size_t(w.rld), 256);
  w.total = off;
  return w;
}


template <typename TT, typename TD, bool kMulti>
static spec_status_t launch_verify(const VerifyDev& d, cudaStream_t s) {
  const int nunits = (d.V + 7) / 8;
  VerifyDev dw = d;
  {
    // draft-row statistics are needed only for tau > 0 with draft logits; with d.lazy the walk
    // forms the statistics of the nodes it visits instead
    const int rows = d.lazy ? 0 : d.N + ((d.tau > 0.f && !d.probs) ? d.R : 0);
    dw.after_rows = rows > 0 ? 1 : 0;
    if (rows > 0) {
      const cudaError_t e = launch_pdl(verify_rows_kernel<TT>, dim3(rows), dim3(kRowThreads), 0, s, d);
      if (e != cudaSuccess) return launch_result(e);
    }
  }
  static DeviceOnce raised_walk, raised_walk_lazy;   // the unit-sum array's maximum, per device
  // (the multi-draft rule always follows its rows kernel: no kLazy instance of it)
  auto kernel = verify_walk_kernel<TT, TD, kMulti, false>;
  if constexpr (!kMulti)
    if (d.lazy) kernel = verify_walk_kernel<TT, TD, false, true>;
  {
    const spec_status_t st = raise_dyn_smem_once(kernel, sizeof(float) * kWalkMaxSmemUnits,
                                                 d.lazy ? raised_walk_lazy : raised_walk);
    if (st != SPEC_OK) return st;
  }
  // CTAs per request: the largest cluster (at most kWalkMaxCl) whose slices keep at least
  // kWalkMinUnits units and whose clusters for the whole batch are resident at once; one CTA
  // under the multi-draft rule
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return launch_result(e);
  int ncl = 1;
  if (!kMulti) {
    for (int n = kWalkMaxCl; n >= 2; n >>= 1) {
      const int per = (nunits + n - 1) / n;
      if (per < kWalkMinUnits) continue;
      const long long smem = per <= kWalkMaxSmemUnits ? 4LL * per : 0;
      if (active_clusters(kernel, dev, n, kWalkThreads, smem) >= d.B) {
        ncl = n;
        break;
      }
    }
  }
  dw.walk_per = (nunits + ncl - 1) / ncl;
  const size_t dyn = dw.walk_per <= kWalkMaxSmemUnits ? sizeof(float) * size_t(dw.walk_per) : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(d.B) * unsigned(ncl));
  cfg.blockDim = dim3(kWalkThreads);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(ncl);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kernel, dw);
  if (e == cudaSuccess) count_launch();
  return launch_result(e);
}

}  // namespace spec

extern "C" {

size_t spec_verify_workspace_size(const spec_verify_params* p) {
  if (!p) return 0;
  const bool multi = p->sibling_rule == SPEC_SIBLING_MULTI_DRAFT && p->tau > 0.f;
  return spec::verify_ws_layout(p->N, p->R, multi ? p->B : 0, p->V).total;
}

}  // extern "C"

// spec_verify, and with c != nullptr spec_verify_compact: the compaction runs inside the
// one-launch verification when the call takes that form, else as spec_kv_compact after it.
static spec_status_t verify_impl(const spec_verify_params* p, const spec_compact_params* c,
                                 void* workspace, size_t ws_bytes, spec_stream_t stream) {
  using namespace spec;
  if (!p) return SPEC_ERR_INVALID_ARG;
  if (p->B < 1 || p->N < 0 || p->R < 0 || p->V < 1 || p->T_max < 1 ||
      p->T_max > SPEC_MAX_TREE || p->max_path < 1)
    return SPEC_ERR_INVALID_ARG;
  if (!(p->tau >= 0.f) || !isfinite(p->tau)) return SPEC_ERR_INVALID_ARG;
  if (p->logits_dtype != SPEC_F32 && p->logits_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (p->draft_kind != SPEC_DRAFT_LOGITS && p->draft_kind != SPEC_DRAFT_PROBS)
    return SPEC_ERR_INVALID_ARG;
  if (p->sibling_rule != SPEC_SIBLING_RESIDUAL && p->sibling_rule != SPEC_SIBLING_INDEPENDENT &&
      p->sibling_rule != SPEC_SIBLING_MULTI_DRAFT)
    return SPEC_ERR_INVALID_ARG;
  if (p->verify_path != SPEC_VERIFY_PATH_AUTO && p->verify_path != SPEC_VERIFY_PATH_SPLIT &&
      p->verify_path != SPEC_VERIFY_PATH_WALK)
    return SPEC_ERR_INVALID_ARG;
  if (!p->node_offset || !p->req_status || !p->out_tokens || !p->out_len || !p->path ||
      !p->n_acc)
    return SPEC_ERR_INVALID_ARG;
  if (p->N > 0 && (!p->target || !p->tokens || !p->parent || !p->depth || !p->is_internal ||
                   !p->uniforms || !p->draft_row))
    return SPEC_ERR_INVALID_ARG;
  const size_t tes = p->logits_dtype == SPEC_BF16 ? 2 : 4;
  const size_t des = p->draft_kind == SPEC_DRAFT_PROBS ? 4 : tes;
  if (p->target_ld < p->V || (size_t(p->target_ld) * tes) % 16 != 0) return SPEC_ERR_INVALID_ARG;
  if (p->target && !aligned16(p->target)) return SPEC_ERR_INVALID_ARG;
  if (p->R > 0) {
    if (!p->draft || !aligned16(p->draft)) return SPEC_ERR_INVALID_ARG;
    if (p->draft_ld < p->V || (size_t(p->draft_ld) * des) % 16 != 0) return SPEC_ERR_INVALID_ARG;
  }
  const bool multi = p->sibling_rule == SPEC_SIBLING_MULTI_DRAFT && p->tau > 0.f;
  const VerifyWs lay = verify_ws_layout(p->N, p->R, multi ? p->B : 0, p->V);
  if (!workspace || ws_bytes < lay.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return SPEC_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  VerifyDev d;
  d.after_rows = 0;
  d.target = p->target;
  d.draft = p->draft;
  d.tld = p->target_ld;
  d.dld = p->draft_ld;
  d.B = p->B; d.N = p->N; d.R = p->R; d.V = p->V; d.T_max = p->T_max; d.max_path = p->max_path;
  d.tau = p->tau;
  d.k2 = p->tau > 0.f ? float(1.4426950408889634 / double(p->tau)) : 0.f;
  d.inv_tau = p->tau > 0.f ? 1.0f / p->tau : 0.f;
  d.probs = p->draft_kind == SPEC_DRAFT_PROBS;
  d.residual_rule = p->sibling_rule == SPEC_SIBLING_RESIDUAL;
  d.multi = multi ? 1 : 0;
  d.draft_row = p->draft_row; d.tokens = p->tokens; d.parent = p->parent;
  d.node_offset = p->node_offset; d.depth = p->depth; d.is_internal = p->is_internal;
  d.uniforms = p->uniforms; d.req_status = p->req_status; d.out_tokens = p->out_tokens;
  d.out_len = p->out_len; d.path = p->path; d.n_acc = p->n_acc; d.rejections = p->rejections;
  d.tstat = reinterpret_cast<RowStat*>(ws + lay.tstat);
  d.dstat = reinterpret_cast<RowStat*>(ws + lay.dstat);
  d.rbuf = multi ? reinterpret_cast<float*>(ws + lay.rbuf) : nullptr;
  d.rld = lay.rld;
  CompactDev cdev = {};
  if (c) {
    const spec_status_t cst = make_compact_dev(c, &cdev);
    if (cst != SPEC_OK) return cst;
    // the compaction reads the verification's own path, counts and status
    if (c->B != p->B || c->path != p->path || c->n_acc != p->n_acc ||
        c->req_status != p->req_status || c->max_path != p->max_path)
      return SPEC_ERR_INVALID_ARG;
  }
  cudaStream_t s = (cudaStream_t)stream;
  // the walk visits one path, usually a short one: with a large vocabulary the statistics of the
  // few nodes it visits (a pass over their rows each) cost less than a rows kernel reading every
  // internal node's rows first; below it the walk's own passes (and its prologue, which the rows
  // kernel hides) cost more (measured: SpecInfer, vocab 128256, step 0.429 -> 0.386 ms; Medusa,
  // vocab 32000, 0.140 -> 0.172 ms)
  d.lazy = (!multi && (p->verify_path == SPEC_VERIFY_PATH_WALK ||
                       (p->verify_path == SPEC_VERIFY_PATH_AUTO && p->V >= kLazyMinVocab))) ? 1 : 0;
  if (!multi && p->verify_path == SPEC_VERIFY_PATH_AUTO) {
    ClusterVerifyArgs ca;
    ca.compact = c ? 1 : 0;
    ca.cd = cdev;
    ca.target = p->target; ca.draft = p->draft; ca.tld = p->target_ld; ca.dld = p->draft_ld;
    ca.B = p->B; ca.N = p->N; ca.R = p->R; ca.V = p->V; ca.T_max = p->T_max;
    ca.max_path = p->max_path;
    ca.tau = d.tau; ca.k2 = d.k2; ca.inv_tau = d.inv_tau;
    ca.probs = d.probs; ca.residual_rule = d.residual_rule;
    ca.draft_row = p->draft_row; ca.tokens = p->tokens; ca.parent = p->parent;
    ca.node_offset = p->node_offset; ca.depth = p->depth; ca.is_internal = p->is_internal;
    ca.uniforms = p->uniforms; ca.req_status = p->req_status; ca.out_tokens = p->out_tokens;
    ca.out_len = p->out_len; ca.path = p->path; ca.n_acc = p->n_acc;
    ca.rejections = p->rejections;
    if (verify_cluster_fits(ca, int(tes), int(des))) {
      const cudaError_t e = launch_verify_cluster(ca, int(tes), int(des), s);
      if (e != cudaErrorNotSupported) return launch_result(e);
    }
  }
  spec_status_t st;
  if (multi) {
    if (p->logits_dtype == SPEC_BF16)
      st = d.probs ? launch_verify<__nv_bfloat16, float, true>(d, s)
                   : launch_verify<__nv_bfloat16, __nv_bfloat16, true>(d, s);
    else
      st = launch_verify<float, float, true>(d, s);
  } else {
    if (p->logits_dtype == SPEC_BF16)
      st = d.probs ? launch_verify<__nv_bfloat16, float, false>(d, s)
                   : launch_verify<__nv_bfloat16, __nv_bfloat16, false>(d, s);
    else
      st = launch_verify<float, float, false>(d, s);
  }
  if (st != SPEC_OK || !c) return st;
  return spec_kv_compact(c, stream);
}

extern "C" {

spec_status_t spec_verify(const spec_verify_params* p, void* workspace, size_t ws_bytes,
                          spec_stream_t stream) {
  return verify_impl(p, nullptr, workspace, ws_bytes, stream);
}

spec_status_t spec_verify_compact(const spec_verify_params* v, const spec_compact_params* c,
                                  void* workspace, size_t ws_bytes, spec_stream_t stream) {
  if (!c) return SPEC_ERR_INVALID_ARG;
  return verify_impl(v, c, workspace, ws_bytes, stream);
}

}  // extern "C"

// ------------------------------------------------------------------------------------------
// spec_verify_noalloc: spec_verify for callers that may not allocate device memory at all --
// for example an inference engine that reserves its whole memory budget at start-up and
// forbids any allocation on the request path, or a plugin that is handed only tensors and a
// stream by a host framework.  The verification workspace lives in one fixed array in device
// memory that is part of this library; every GPU that loads the library holds it until the
// process exits.  It covers up to kNoAllocMaxNodes tree nodes and kNoAllocMaxDraftRows draft
// rows; larger batches are refused with SPEC_ERR_UNSUPPORTED.
// The first call on each device looks the array's device address up (cudaGetSymbolAddress)
// with that device current; make that first call before any stream capture.  Later calls look
// it up again unless their stream is being captured (then the address found before is used), so
// a device reset between calls does not leave a stale address behind.  All calls share the
// array: calls whose kernels overlap on the GPU (different streams, or different host threads
// on the same device) race on it.  Every call writes the statistics it reads before reading
// them, so the contents left by an earlier call do not matter.  The multi-draft sibling rule
// (tau > 0) needs residual rows on top of the statistics and is refused.
// ------------------------------------------------------------------------------------------
namespace spec {
constexpr int kNoAllocMaxNodes = 32768;
constexpr int kNoAllocMaxDraftRows = 32768;
constexpr size_t kNoAllocScratchBytes =
    align_up(sizeof(RowStat) * kNoAllocMaxNodes, 256) +
    align_up(sizeof(RowStat) * kNoAllocMaxDraftRows, 256);
static __device__ __align__(256) unsigned char g_verify_scratch[kNoAllocScratchBytes];
}  // namespace spec

extern "C" spec_status_t spec_verify_noalloc(const spec_verify_params* p, spec_stream_t stream) {
  using namespace spec;
  static std::mutex mu;
  static void* scratch_of[64] = {nullptr};
  if (!p) return SPEC_ERR_INVALID_ARG;
  if (p->sibling_rule == SPEC_SIBLING_MULTI_DRAFT && p->tau > 0.f) return SPEC_ERR_UNSUPPORTED;
  if (p->N > kNoAllocMaxNodes || p->R > kNoAllocMaxDraftRows) return SPEC_ERR_UNSUPPORTED;
  const size_t need = spec_verify_workspace_size(p);
  if (need > kNoAllocScratchBytes) return SPEC_ERR_UNSUPPORTED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return SPEC_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return SPEC_ERR_UNSUPPORTED;
  // look the address up again unless the stream is being captured (a lookup may not be allowed
  // then); a stream whose capture state cannot be read keeps the address found before
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusActive;
  if (cudaStreamIsCapturing((cudaStream_t)stream, &cap) != cudaSuccess) {
    cudaGetLastError();
    cap = cudaStreamCaptureStatusActive;
  }
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!scratch_of[dev] || cap == cudaStreamCaptureStatusNone) {
      void* found = nullptr;
      e = cudaGetSymbolAddress(&found, g_verify_scratch);
      if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return SPEC_ERR_CUDA;
      }
      scratch_of[dev] = found;
    }
    ptr = scratch_of[dev];
  }
  return spec_verify(p, ptr, kNoAllocScratchBytes, stream);
}
