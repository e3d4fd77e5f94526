// Building the draft tree on the device: EAGLE-2's expansion of the most probable leaves, the
// top-K tokens of each expanded draft row, and ECHO's batch-wide budget, packed into the layout
// the verification step reads.
//
// Source: "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的生成 -- expansion-based trees take the
// top-K tokens per step; EAGLE-2 expands only the K most probable leaves of the newest level,
// ranked by the product of the probabilities along the path; 动态草稿长度 -- ECHO shares one
// global budget K_max of verified tokens among the requests of a batch.
//
// Scores are sums of log q along the path (fp32).  Every selection compares the fp32 scores
// exactly, with the ties broken by index, so it is a pure function of the pool.
//   spec_draft_init          pool entry 0 = the root of every request
//   spec_draft_expand_select one CTA per request, thread per candidate: the rank of each
//                            newest-level candidate among them; the K best, in index order
//   spec_draft_topk_append   one CTA per expanded row: one streaming read of the row (online
//                            max / compensated sum for log-sum-exp, a running top-K list per
//                            thread), K-round warp and block merges, children written to the pool
//   spec_echo_select_pack    one CTA: radix select (8 byte passes) of the (K_max - B)-th best
//                            non-root key over the batch; then one CTA per request packs its
//                            kept candidates (block scans for local indices and offsets)
#include "common.cuh"
#include "tc_ptx.cuh"

namespace spec {

constexpr int kDraftThreads = 256;
constexpr int kTopkMax = 16;
constexpr int kEchoThreads = 1024;

struct PoolDev {
  int32_t B, cap;
  int32_t* parent;
  int32_t* token;
  int32_t* depth;
  float* score;
  int32_t* row;
  int32_t* count;
};

static PoolDev pool_dev(const spec_draft_pool* p) {
  return PoolDev{p->B, p->cap, p->parent, p->token, p->depth, p->score, p->row, p->count};
}

static bool pool_ok(const spec_draft_pool* p) {
  return p && p->B >= 1 && p->cap >= 1 && p->cap <= SPEC_MAX_TREE && p->parent && p->token &&
         p->depth && p->score && p->row && p->count;
}

// ------------------------------------------------------------------------------------------
__global__ void draft_init_kernel(PoolDev p, const int32_t* __restrict__ roots) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= p.B) return;
  const size_t e = size_t(r) * p.cap;
  p.parent[e] = -1;
  p.token[e] = roots[r];
  p.depth[e] = 0;
  p.score[e] = 0.f;
  p.row[e] = -1;
  p.count[r] = 1;
}

// ------------------------------------------------------------------------------------------
// One CTA per request, thread i = candidate i.  Candidates of depth level-1 compete; candidate
// i's rank is the number of competitors with a larger score (or an equal one and a smaller
// index); the K best are listed in index order.  The pool count grows by K per expansion, which
// the clamp keeps within the capacity (a clamped request gets SPEC_REQ_BAD_SIZE).
__global__ void __launch_bounds__(kDraftThreads)
draft_expand_select_kernel(PoolDev p, int level, int K, int32_t* __restrict__ expand,
                           int32_t* __restrict__ req_status) {
  __shared__ float s_score[SPEC_MAX_TREE];
  __shared__ uint8_t s_front[SPEC_MAX_TREE];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, i = threadIdx.x;
  const size_t e0 = size_t(r) * p.cap;
  const int count = min(p.count[r], p.cap);
  const bool front = i < count && (level == 1 ? i == 0 : p.depth[e0 + i] == level - 1);
  s_front[i] = front ? 1 : 0;
  s_score[i] = i < count ? p.score[e0 + i] : 0.f;
  __syncthreads();
  int rank = 0;
  const int nfront = __syncthreads_count(front);
  if (front) {
    const float si = s_score[i];
    for (int k = 0; k < count; ++k)
      if (s_front[k] && (s_score[k] > si || (s_score[k] == si && k < i))) ++rank;
  }
  // how many expansions fit: every expansion appends K candidates
  const int fit = (p.cap - count) / K;
  const int want = min(K, nfront);
  const int nsel = min(want, fit);
  const bool chosen = front && rank < nsel;
  // position in index order = number of chosen candidates with a smaller index
  __shared__ uint8_t s_chosen[SPEC_MAX_TREE];
  s_chosen[i] = chosen ? 1 : 0;
  __syncthreads();
  if (chosen) {
    int pos = 0;
    for (int k = 0; k < i; ++k) pos += s_chosen[k];
    expand[size_t(r) * K + pos] = i;
  }
  if (i >= nsel && i < K) expand[size_t(r) * K + i] = -1;
  if (i == 0) {
    p.count[r] = count + nsel * K;
    if (nsel < want && req_status) atomicOr(&req_status[r], SPEC_REQ_BAD_SIZE);
  }
}

// ------------------------------------------------------------------------------------------
// Top-K of one row.  (value, id) pairs are ordered by value, ties to the lower id.
__device__ __forceinline__ bool better(float v, int id, float w, int jd) {
  return v > w || (v == w && id < jd);
}

// The row streams straight into registers: thread t reads units u * kTopkThreads + t of each
// kChunkBytes chunk (16-byte loads), the next chunk's loads in flight while it works on this one.
// Each thread folds its units into an online max / compensated sum (log-sum-exp; the exponent
// arguments and the sums two at a time with packed fp32 pairs), and each warp keeps its top-K list
// distributed over lanes 0..K-1: a unit is offered only when its maximum reaches the warp's K-th
// value, and offers are inserted one by one under a warp-uniform ballot, so the common path is
// one compare per unit.
constexpr int kChunkBytes = 16384;
constexpr int kTopkThreads = 256;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr long long kStallWaitLimit = 2000000000LL;   // clock cycles (~1 s)

// Testing only (spec_debug_draft_copy_stall): >= 0 makes every launch wait, bounded, for a device
// flag that nothing sets, so that it takes its timeout path as a lost read would; -1 (the
// default) disables it.
__device__ int g_draft_copy_stall = -1;
__device__ int g_draft_never_set = 0;

// fp32 value -> unsigned key in the same order (for an atomic maximum)
__device__ __forceinline__ unsigned ordered_key(float v) {
  const unsigned b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// insert (v, id) into the warp's distributed list (lane q < K holds the q-th best)
__device__ __forceinline__ void warp_list_insert(float& lv, int& lid, float v, int id, int K,
                                                 int lane) {
  const unsigned ahead = __ballot_sync(0xffffffffu, lane < K && better(lv, lid, v, id));
  const int pos = __popc(ahead);
  if (pos >= K) return;   // not better than the K-th (uniform across the warp)
  const float uv = __shfl_up_sync(0xffffffffu, lv, 1);
  const int uid = __shfl_up_sync(0xffffffffu, lid, 1);
  if (lane == pos) { lv = v; lid = id; }
  else if (lane > pos && lane < K) { lv = uv; lid = uid; }
}

template <typename T>
__global__ void __launch_bounds__(kTopkThreads)
draft_topk_append_kernel(PoolDev p, int level, int K, const int32_t* __restrict__ expand,
                         const T* __restrict__ rows, int64_t ld, int V, float k2, float inv_tau,
                         int row_base, int32_t* __restrict__ req_status) {
  constexpr int kElems = kChunkBytes / int(sizeof(T));   // elements per chunk
  constexpr int kUnitsPerChunk = kElems / 8;
  constexpr int kPerThread = kUnitsPerChunk / kTopkThreads;
  constexpr int kVecs = int(sizeof(T)) / 2;              // 16-byte loads per 8-element unit
  static_assert(kPerThread * kTopkThreads == kUnitsPerChunk, "whole units per thread");
  __shared__ float s_v[kTopkWarps][kTopkMax];
  __shared__ int s_id[kTopkWarps][kTopkMax];
  __shared__ float s_m[kTopkWarps];
  __shared__ double s_s[kTopkWarps];
  __shared__ float s_best_v[kTopkMax];
  __shared__ int s_best_id[kTopkMax];
  __shared__ float s_logz;
  __shared__ int s_abort;
  // The CTA's admission floor: the largest of the warps' K-th values and first-chunk seeds.  An
  // element of the row's top K is not below any warp's K-th value (that warp would hold K better
  // elements), so a unit below the floor needs no offer; the floor only grows, and a stale read
  // only admits more.
  __shared__ unsigned s_floor;
  pdl_wait();
  const int row_i = blockIdx.x;
  const int r = row_i / K, j = row_i - r * K;
  const int cand = expand[row_i];
  if (cand < 0) {
    pdl_trigger();
    return;
  }
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const char* src = reinterpret_cast<const char*>(rows + size_t(row_i) * ld);
  const int row_bytes = (V * int(sizeof(T)) + 15) & ~15;   // within the padded row (ld)
  const int nchunks = (row_bytes + kChunkBytes - 1) / kChunkBytes;
  if (tid == 0) {
    s_abort = 0;
    s_floor = ordered_key(-INFINITY);
    if (g_draft_copy_stall >= 0) {   // testing only: a wait that never completes, bounded
      volatile int* flag = &g_draft_never_set;
      const long long t0 = clock64();
      while (*flag == 0 && clock64() - t0 < kStallWaitLimit) {
      }
      if (*flag == 0) s_abort = 1;
    }
  }
  __syncthreads();
  // this thread's units of chunk c (vectors past the row's padded end are not read)
  uint4 nxt[kPerThread][kVecs];
  auto fetch = [&](int c) {
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
      const int off = c * kChunkBytes + (u * kTopkThreads + tid) * 16 * kVecs;
#pragma unroll
      for (int q = 0; q < kVecs; ++q)
        nxt[u][q] = off + 16 * q < row_bytes ? ld_stream16(src + off + 16 * q) : make_uint4(0, 0, 0, 0);
    }
  };

  float m = -INFINITY, s = 0.f, comp = 0.f;
  float lv = -INFINITY;      // this lane's entry of the warp's top-K list (lanes < K)
  int lid = 0x7fffffff;
  if (s_abort == 0) {
    float thr = -INFINITY;   // the warp's K-th value
    float seed = -INFINITY;  // admission floor from the first chunk
    float mk2 = -INFINITY;   // m * k2
    fetch(0);
    for (int c = 0; c < nchunks; ++c) {
      const int base_id = c * kElems;
      // this thread's units of the chunk, all in registers: one max, one rescale check, the
      // exponentials as independent work, one compensated step for the chunk
      constexpr int kN = kPerThread * 8;
      float x[kN];
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        if constexpr (sizeof(T) == 2) {
          elem<T>::unpack(nxt[u][0], x + 8 * u);
        } else {
          elem<T>::unpack(nxt[u][0], x + 8 * u);
          elem<T>::unpack(nxt[u][kVecs - 1], x + 8 * u + 4);
        }
      }
      if (c + 1 < nchunks) fetch(c + 1);   // the next chunk's loads fly while this one is folded
      if (base_id + kElems > V) {   // the row's last chunk: elements past V do not exist
#pragma unroll
        for (int u = 0; u < kPerThread; ++u)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (base_id + (u * kTopkThreads + tid) * 8 + k >= V) x[8 * u + k] = -INFINITY;
      }
      float um[kPerThread];
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const float* xu = x + 8 * u;
        um[u] = fmax3(fmax3(xu[0], xu[1], xu[2]), fmax3(xu[3], xu[4], xu[5]), fmaxf(xu[6], xu[7]));
      }
      float cm = um[0];
#pragma unroll
      for (int u = 1; u < kPerThread; ++u) cm = fmaxf(cm, um[u]);
      if (cm > m) {
        const float sc = ex2(mk2 - cm * k2);
        s *= sc;
        comp *= sc;
        m = cm;
        mk2 = m * k2;
      }
      // exponentials 2^(x k2 - m k2): arguments and sums two at a time
      const uint64_t k2v = f2_pack(k2, k2), negv = f2_pack(-mk2, -mk2);
      uint64_t acc[4] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f),
                         f2_pack(0.f, 0.f)};
#pragma unroll
      for (int k = 0; k < kN; k += 2) {
        float y0, y1;
        f2_unpack(f2_fma(f2_pack(x[k], x[k + 1]), k2v, negv), y0, y1);
        acc[(k >> 1) & 3] = f2_add(acc[(k >> 1) & 3], f2_pack(ex2(y0), ex2(y1)));
      }
      float a0, a1, a2, a3;
      f2_unpack(f2_add(acc[0], acc[1]), a0, a1);
      f2_unpack(f2_add(acc[2], acc[3]), a2, a3);
      const float y = ((a0 + a1) + (a2 + a3)) - comp;   // compensated sum, one step per chunk
      const float t = s + y;
      comp = (t - s) - y;
      s = t;
      // The first chunk seeds the admission threshold: the K-th largest of the lanes' maxima is
      // a lower bound of the row's K-th value (those K maxima are elements of the row), so no
      // element below it can be in the top K.  Ties still pass: the id decides at insertion.
      if (c == 0) {
        int rank = 0;
        for (int q = 0; q < 32; ++q) {
          const float o = __shfl_sync(0xffffffffu, cm, q);
          rank += (o > cm || (o == cm && q < lane)) ? 1 : 0;
        }
        const unsigned at = __ballot_sync(0xffffffffu, rank == K - 1);
        seed = at ? __shfl_sync(0xffffffffu, cm, __ffs(at) - 1) : -INFINITY;
        if (lane == 0) atomicMax(&s_floor, ordered_key(seed));
      }
      seed = fmaxf(seed, key_value(*reinterpret_cast<volatile unsigned*>(&s_floor)));
      // offers to the warp's list, one unit at a time; the offering lane names its elements
      // that reach the threshold and only those are inserted
#pragma unroll
      for (int u = 0; u < kPerThread; ++u) {
        const float adm = fmaxf(thr, seed);
        unsigned offer = __ballot_sync(0xffffffffu, um[u] >= adm && um[u] > -INFINITY);
        while (offer) {
          const int src_lane = __ffs(offer) - 1;
          offer &= offer - 1;
          const float adm_now = fmaxf(thr, seed);
          unsigned bits = 0;
#pragma unroll
          for (int k = 0; k < 8; ++k)
            bits |= (x[8 * u + k] >= adm_now && x[8 * u + k] > -INFINITY) ? (1u << k) : 0u;
          bits = __shfl_sync(0xffffffffu, bits, src_lane);
          while (bits) {   // uniform across the warp
            const int k = __ffs(bits) - 1;
            bits &= bits - 1;
            float xk = x[8 * u];
#pragma unroll
            for (int q = 1; q < 8; ++q) xk = (k == q) ? x[8 * u + q] : xk;
            const float v = __shfl_sync(0xffffffffu, xk, src_lane);
            const int id = base_id + (u * kTopkThreads + src_lane + warp * 32) * 8 + k;
            if (v >= fmaxf(thr, seed)) {   // the list may have moved since the mask was taken
              warp_list_insert(lv, lid, v, id, K, lane);
              const float nt = __shfl_sync(0xffffffffu, lv, K - 1);
              if (lane == 0 && nt > thr) atomicMax(&s_floor, ordered_key(nt));
              thr = nt;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  const bool ok = s_abort == 0;
  if (!ok && tid == 0 && req_status) atomicOr(&req_status[r], SPEC_REQ_TIMEOUT);
  pdl_trigger();
  // log-sum-exp over the warps: every thread's (m, s) rescaled to the block max
  {
    const float wm = warp_max(m);
    if (lane == 0) s_m[warp] = wm;
    if (lane < K) { s_v[warp][lane] = lv; s_id[warp][lane] = lid; }
  }
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kTopkWarps; ++w) M = fmaxf(M, s_m[w]);
  {
    dfloat ds = df_make(m == -INFINITY ? 0.f : (s - comp) * ex2((m - M) * k2));
    ds = warp_sum_df(ds);
    if (lane == 0) s_s[warp] = df_to_d(ds);
  }
  __syncthreads();
  // the block's top-K from the warps' lists (warp 0, lane w < kTopkWarps walks list w)
  if (warp == 0) {
    int h = 0;
    for (int q = 0; q < K; ++q) {
      float bv = -INFINITY;
      int bid = 0x7fffffff;
      if (lane < kTopkWarps && h < K) { bv = s_v[lane][h]; bid = s_id[lane][h]; }
      float wv = bv;
      int wid = bid;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, wv, o);
        const int oid = __shfl_xor_sync(0xffffffffu, wid, o);
        if (better(ov, oid, wv, wid)) { wv = ov; wid = oid; }
      }
      if (lane < kTopkWarps && h < K && bid == wid && bv == wv) ++h;
      if (lane == 0) { s_best_v[q] = wv; s_best_id[q] = wid; }
    }
    if (lane == 0) {
      double S = 0.0;
      for (int w = 0; w < kTopkWarps; ++w) S += s_s[w];
      s_logz = float(log(S));
    }
  }
  __syncthreads();
  // append the children: this expansion's block of K slots after the level's base
  if (tid < K) {
    int nsel = 0;
    for (int q = 0; q < K; ++q) nsel += expand[size_t(r) * K + q] >= 0 ? 1 : 0;
    const size_t e0 = size_t(r) * p.cap;
    const int base = p.count[r] - nsel * K;
    const int pos = base + j * K + tid;
    const float logq = (s_best_v[tid] - M) * inv_tau - s_logz;
    p.parent[e0 + pos] = cand;
    p.token[e0 + pos] = ok ? s_best_id[tid] : -1;
    p.depth[e0 + pos] = level;
    p.score[e0 + pos] = ok ? p.score[e0 + cand] + logq : -INFINITY;
    p.row[e0 + pos] = -1;
    if (tid == 0) p.row[e0 + cand] = row_base + r * K + j;
  }
}

// ------------------------------------------------------------------------------------------
// ECHO.  Key of candidate (r, i): score bits mapped so that ascending keys mean descending
// scores, then r * cap + i -- ascending key order is (score desc, request, index).
__device__ __forceinline__ uint64_t echo_key(float score, int r, int cap, int i) {
  const uint32_t b = __float_as_uint(score);
  const uint32_t asc = (b & 0x80000000u) ? ~b : (b | 0x80000000u);   // ascending in the value
  return (uint64_t(~asc) << 32) | uint32_t(r * cap + i);
}

// One CTA: the M-th smallest key among all non-root candidates (M = K_max - B), found by eight
// byte-wide passes from the top: each pass histograms the byte of the keys that share the
// prefix found so far and descends into the bin holding the M-th.  kept[r][i] = key <= it.
// The keys are read from the pool once into shared memory (non-candidates hold kNoKey); one warp
// finds the bin (eight bins per lane and a shuffle scan); kept counts per request are summed
// with shared atomics while marking.
constexpr uint64_t kNoKey = ~0ull;
constexpr int kEchoMaxKeys = 16384;   // keys held in shared memory (128 KB)
constexpr int kEchoMaxB = 4096;       // requests whose kept counts are summed in shared memory

__global__ void __launch_bounds__(kEchoThreads)
echo_select_kernel(PoolDev p, int K_max, uint8_t* __restrict__ kept,
                   int32_t* __restrict__ kept_count) {
  extern __shared__ uint64_t s_key[];   // [B * cap]
  __shared__ int hist[256];
  __shared__ int s_cnt[kEchoMaxB];
  __shared__ uint64_t s_prefix;
  __shared__ int s_rank;
  __shared__ int s_total;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.B * p.cap;
  if (tid == 0) s_total = 0;
  for (int r = tid; r < p.B; r += kEchoThreads) s_cnt[r] = 0;
  __syncthreads();
  int mine = 0;
  for (int e = tid; e < n; e += kEchoThreads) {
    const int r = e / p.cap, i = e - r * p.cap;
    const bool cand = i > 0 && i < min(p.count[r], p.cap);
    s_key[e] = cand ? echo_key(p.score[e], r, p.cap, i) : kNoKey;
    mine += cand ? 1 : 0;
  }
  atomicAdd(&s_total, mine);
  __syncthreads();
  const int total = s_total;
  const int M = min(max(K_max - p.B, 0), total);   // keep the M best non-roots
  uint64_t prefix = 0;
  if (M > 0 && M < total) {
    int rank = M;   // 1-based rank of the threshold key among the keys with this prefix
    for (int pass = 7; pass >= 0; --pass) {
      const int shift = pass * 8;
      for (int b = tid; b < 256; b += kEchoThreads) hist[b] = 0;
      __syncthreads();
      const uint64_t hi_mask = pass == 7 ? 0ull : (~0ull << (shift + 8));
      for (int e = tid; e < n; e += kEchoThreads) {
        const uint64_t key = s_key[e];
        if (key != kNoKey && (key & hi_mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
      }
      __syncthreads();
      if (warp == 0) {   // the bin where the running count reaches rank
        int c8[8], sum = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) { c8[k] = hist[lane * 8 + k]; sum += c8[k]; }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const int excl = incl - sum;
        const unsigned hit = __ballot_sync(0xffffffffu, excl < rank && incl >= rank);
        if (lane == __ffs(hit) - 1) {
          int acc = excl, b = lane * 8;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (acc + c8[k] >= rank) { b = lane * 8 + k; break; }
            acc += c8[k];
          }
          s_prefix = prefix | (uint64_t(b) << shift);
          s_rank = rank - acc;
        }
      }
      __syncthreads();
      prefix = s_prefix;
      rank = s_rank;
      __syncthreads();
    }
  }
  // marks: roots always; non-roots by key (M == total: all; M == 0: none)
  for (int e = tid; e < n; e += kEchoThreads) {
    const int r = e / p.cap, i = e - r * p.cap;
    const uint64_t key = s_key[e];
    uint8_t k = 0;
    if (i == 0) {
      k = 1;
    } else if (key != kNoKey && M > 0) {
      k = (M >= total || key <= prefix) ? 1 : 0;
    }
    kept[e] = k;
    if (k) atomicAdd(&s_cnt[r], 1);
  }
  __syncthreads();
  for (int r = tid; r < p.B; r += kEchoThreads) kept_count[r] = s_cnt[r];
}

// One CTA per request: offsets by summing the earlier requests' counts, local indices by a
// block scan of the kept flags, parents remapped through them.
__global__ void __launch_bounds__(kDraftThreads)
echo_pack_kernel(PoolDev p, const uint8_t* __restrict__ kept,
                 const int32_t* __restrict__ kept_count, int32_t* __restrict__ node_offset,
                 int32_t* __restrict__ parent, int32_t* __restrict__ tokens,
                 int32_t* __restrict__ depth, int32_t* __restrict__ draft_row,
                 int32_t* __restrict__ source) {
  __shared__ int s_new[SPEC_MAX_TREE];
  __shared__ uint8_t s_has_child[SPEC_MAX_TREE];
  __shared__ int s_warp[kDraftThreads / 32];
  __shared__ int s_off;
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, i = threadIdx.x, lane = i & 31, warp = i >> 5;
  // offset of this request = sum of the kept counts before it
  int part = 0;
  for (int q = i; q < r; q += kDraftThreads) part += kept_count[q];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if (lane == 0) s_warp[warp] = part;
  __syncthreads();
  if (i == 0) {
    int t = 0;
    for (int w = 0; w < kDraftThreads / 32; ++w) t += s_warp[w];
    s_off = t;
  }
  __syncthreads();
  const int off = s_off;
  const size_t e0 = size_t(r) * p.cap;
  const int cnt = min(p.count[r], p.cap);
  const int k = (i < cnt) ? kept[e0 + i] : 0;
  // inclusive scan of the flags over the block
  int v = k;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = v;
  s_has_child[i] = 0;
  __syncthreads();
  int wbase = 0;
  for (int w = 0; w < warp; ++w) wbase += s_warp[w];
  const int local = wbase + v - k;   // exclusive
  s_new[i] = k ? local : -1;
  __syncthreads();
  const int par = (i < cnt) ? p.parent[e0 + i] : -1;
  if (k && par >= 0) s_has_child[par] = 1;   // benign race: every writer stores 1
  __syncthreads();
  if (k) {
    const int n = off + local;
    parent[n] = par >= 0 ? s_new[par] : -1;
    tokens[n] = p.token[e0 + i];
    depth[n] = p.depth[e0 + i];
    draft_row[n] = s_has_child[i] ? p.row[e0 + i] : -1;
    if (source) source[n] = i;
  }
  if (i == 0) {
    node_offset[r] = off;
    if (r == p.B - 1) node_offset[p.B] = off + kept_count[r];
  }
}

}  // namespace spec

extern "C" {

spec_status_t spec_draft_init(const spec_draft_pool* pool, const int32_t* root_tokens,
                              spec_stream_t stream) {
  using namespace spec;
  if (!pool_ok(pool) || !root_tokens) return SPEC_ERR_INVALID_ARG;
  const PoolDev p = pool_dev(pool);
  return launch_result(launch_pdl(draft_init_kernel, dim3((p.B + 255) / 256), dim3(256), 0,
                                  (cudaStream_t)stream, p, root_tokens));
}

spec_status_t spec_draft_expand_select(const spec_draft_pool* pool, int32_t level, int32_t K,
                                       int32_t* expand, int32_t* req_status,
                                       spec_stream_t stream) {
  using namespace spec;
  if (!pool_ok(pool) || !expand || level < 1 || K < 1 || K > kTopkMax) return SPEC_ERR_INVALID_ARG;
  const PoolDev p = pool_dev(pool);
  return launch_result(launch_pdl(draft_expand_select_kernel, dim3(p.B), dim3(kDraftThreads), 0,
                                  (cudaStream_t)stream, p, int(level), int(K), expand,
                                  req_status));
}

spec_status_t spec_draft_topk_append(const spec_draft_pool* pool, int32_t level, int32_t K,
                                     const int32_t* expand, spec_dtype_t dtype, const void* rows,
                                     int64_t ld, int32_t V, float tau, int32_t row_base,
                                     int32_t* req_status, spec_stream_t stream) {
  using namespace spec;
  if (!pool_ok(pool) || !expand || !rows || level < 1 || K < 1 || K > kTopkMax || V < K ||
      !(tau > 0.f) || !isfinite(tau))
    return SPEC_ERR_INVALID_ARG;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  const size_t es = dtype == SPEC_BF16 ? 2 : 4;
  if (ld < V || (size_t(ld) * es) % 16 || !aligned16(rows)) return SPEC_ERR_INVALID_ARG;
  const PoolDev p = pool_dev(pool);
  const float k2 = float(1.4426950408889634 / double(tau));
  const float inv_tau = 1.0f / tau;
  const dim3 grid(unsigned(p.B) * unsigned(K));
  const size_t dyn = 0;
  cudaError_t e;
  if (dtype == SPEC_BF16)
    e = launch_pdl(draft_topk_append_kernel<__nv_bfloat16>, grid, dim3(kTopkThreads), dyn,
                   (cudaStream_t)stream, p, int(level), int(K), expand,
                   static_cast<const __nv_bfloat16*>(rows), ld, int(V), k2, inv_tau,
                   int(row_base), req_status);
  else
    e = launch_pdl(draft_topk_append_kernel<float>, grid, dim3(kTopkThreads), dyn,
                   (cudaStream_t)stream, p, int(level), int(K), expand,
                   static_cast<const float*>(rows), ld, int(V), k2, inv_tau, int(row_base),
                   req_status);
  return launch_result(e);
}

spec_status_t spec_debug_draft_copy_stall(int32_t chunk) {
  const int v = chunk < 0 ? -1 : chunk;
  const cudaError_t e = cudaMemcpyToSymbol(spec::g_draft_copy_stall, &v, sizeof(v));
  if (e != cudaSuccess) {
    spec::set_last_cuda_error(e);
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

size_t spec_echo_workspace_size(int32_t B, int32_t cap) {
  if (B < 1 || cap < 1) return 0;
  return spec::align_up(size_t(B) * size_t(cap), 256) + spec::align_up(sizeof(int32_t) * B, 256);
}

spec_status_t spec_echo_select_pack(const spec_draft_pool* pool, int32_t K_max,
                                    int32_t* node_offset, int32_t* parent, int32_t* tokens,
                                    int32_t* depth, int32_t* draft_row, int32_t* source,
                                    void* workspace, size_t ws_bytes, spec_stream_t stream) {
  using namespace spec;
  if (!pool_ok(pool) || K_max < 0 || !node_offset || !parent || !tokens || !depth ||
      !draft_row)
    return SPEC_ERR_INVALID_ARG;
  const size_t need = spec_echo_workspace_size(pool->B, pool->cap);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return SPEC_ERR_INVALID_ARG;
  const PoolDev p = pool_dev(pool);
  uint8_t* kept = static_cast<uint8_t*>(workspace);
  int32_t* kept_count = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) +
                                                   align_up(size_t(p.B) * size_t(p.cap), 256));
  if (p.B * p.cap > kEchoMaxKeys || p.B > kEchoMaxB) return SPEC_ERR_UNSUPPORTED;
  const size_t dyn = sizeof(uint64_t) * size_t(p.B) * size_t(p.cap);
  static DeviceOnce raised;
  const spec_status_t st = raise_dyn_smem_once(echo_select_kernel, sizeof(uint64_t) * kEchoMaxKeys,
                                               raised);
  if (st != SPEC_OK) return st;
  cudaError_t e = launch_pdl(echo_select_kernel, dim3(1), dim3(kEchoThreads), dyn,
                             (cudaStream_t)stream, p, int(K_max), kept, kept_count);
  if (e == cudaSuccess)
    e = launch_pdl(echo_pack_kernel, dim3(p.B), dim3(kDraftThreads), 0, (cudaStream_t)stream, p,
                   static_cast<const uint8_t*>(kept), static_cast<const int32_t*>(kept_count),
                   node_offset, parent, tokens, depth, draft_row, source);
  return launch_result(e);
}

}  // extern "C"
