// bf16 tree attention on the tcgen05 tensor cores (sm_103a).
//
// Sources: "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的验证——树形掩码 -- one forward over the
// flattened tree with the ancestor mask, tree position ids and the KV cache; "万字综述 10+ 种 LLM
// 投机采样推理加速方案" (m.haoling.cc) 5.2 -- tree-based decoding shares the prefix through the mask
// instead of one KV copy per branch; 12.4.3 -- PagedAttention and FlashDecoding are the framework
// features verification has to fit (paged KV blocks, KV split across CTAs + log-sum-exp merge).
//
// Work unit = (request r, KV head h, M-tile mt): the G query heads of h times up to 128/G tree
// tokens, stacked token-major into 128 MMA rows (row m = t_local * G + g), against the
// request's P_r + T_r logical KV slots in tiles of 128 keys (8 paged blocks of 16).  The units
// are laid end to end (request, head, M-tile order) as one stream of KV tiles, and a one-CTA
// prep kernel cuts the stream into equal contiguous ranges, one per persistent CTA (one CTA per
// SM).  A unit cut by a range boundary is computed in pieces whose fp32 partial outputs and
// log-sum-exps a merge kernel combines; every other unit writes its output directly.
//
// CTA (384 threads):
//   warp 0      Q and K producer, warp 2 V producer: 128-byte-swizzled TMA boxes (one per
//               paged block and 64-column half, issued by 8 lanes); blocks past the request or
//               with a bad block id are read from an out-of-range row (TMA fills zeros).  K has
//               3 stages, released right after QK^T; V has 2, released after PV;
//   warp 1      one thread issues tcgen05.mma: S = Q K^T (M=128, N=128, K=16 x 8) into one of two
//               TMEM score buffers, O += P V (V as an MN-major operand) into the TMEM
//               accumulator, and commits completions to mbarriers;
//   warps 4..11 softmax: the two warps of a TMEM lane quarter own the same 32 rows; each reads
//               all 128 scores of its rows (the row max is computed redundantly, so no exchange
//               is needed per tile) and exponentiates its own 64 keys with a lazily updated
//               reference max (O rescaled only when the max grows by more than 2^8), writing P
//               into the swizzled K-major P tile; the epilogue adds the two halves' row sums
//               (one bounded exchange per item) and writes O columns 64*half .. 64*half+63.
// Every wait is bounded (clock64 limit); an expired wait flags SPEC_REQ_TIMEOUT and lets every
// role drain and exit; TMEM is always freed.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace spec {

namespace attn {
constexpr int kD = 128;
constexpr int kBS = 16;
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 384;                 // 4 control warps + 8 softmax warps
constexpr int kAtom = 16384;                  // 128 rows x 128 B
constexpr int kTile = 2 * kAtom;              // 128 x 128 bf16
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kSmemQ = 0;
constexpr int kSmemK = kSmemQ + kTile;
constexpr int kSmemV = kSmemK + kKStages * kTile;
constexpr int kSmemP = kSmemV + kVStages * kTile;
constexpr int kSmemBar = kSmemP + kTile;
constexpr int kSmemRed = kSmemBar + 256;      // [2 buffers][2 halves][128 rows] fp32 exchange
constexpr int kSmemEnd = kSmemRed + 2048;
constexpr int kSmemBytes = 232448;            // the per-CTA maximum; the slack aligns the base
constexpr long long kWaitLimit = 4000000000LL;     // clock cycles (~2 s)
constexpr float kLazyRescale = 8.0f;          // log2 units
constexpr int kMaxCtas = 1024;                // prep handles up to this many persistent CTAs
constexpr int kMinTilesPerRange = 4;          // small problems use fewer, longer ranges
}  // namespace attn

struct Item {
  int r, h, mt, j0, j1, slot, pad0, pad1;
};
struct CombineUnit {
  int r, h, mt, slot0, npieces, pad0, pad1, pad2;
};

struct TcDev {
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* node_offset;
  const uint32_t* anc;
  __nv_bfloat16* o;
  float* lse;
  int32_t* req_status;
  int* header;        // [0] items, [1] merge records
  int* cta_off;       // [ctas + 1] item range of each CTA
  int* req_tiles;     // [B + 1] exclusive prefix of tile work per request
  Item* items;
  CombineUnit* combine;
  float* part_o;
  float* part_lse;
  int B, N, H_q, H_kv, G, log2G, T_max, W, num_blocks, max_blocks, kv_rows, ctas;
  int max_items, max_combine;
  float scale_log2;
};

// ------------------------------------------------------------------------------ workspace
struct TcWs {
  size_t header, cta_off, req_tiles, items, combine, part_o, part_lse, total;
  int max_items, max_combine, max_slots;
};

static TcWs tc_ws_layout(const spec_attn_params* p, int ctas) {
  TcWs w;
  const int G = p->H_q / p->H_kv;
  const int tpt = attn::kBM / G;
  const long units = long(p->B) * p->H_kv * ((p->T_max + tpt - 1) / tpt);
  w.max_items = int(units + ctas);      // each range boundary adds at most one piece
  w.max_combine = ctas;                 // a cut unit spans >= 2 ranges
  w.max_slots = 2 * ctas;               // at most two partial pieces per range
  size_t off = 0;
  w.header = off; off = align_up(off + 64, 256);
  w.cta_off = off; off = align_up(off + sizeof(int) * size_t(ctas + 1), 256);
  w.req_tiles = off; off = align_up(off + sizeof(int) * size_t(p->B + 1), 256);
  w.items = off; off = align_up(off + sizeof(Item) * size_t(w.max_items), 256);
  w.combine = off; off = align_up(off + sizeof(CombineUnit) * size_t(w.max_combine), 256);
  w.part_o = off; off = align_up(off + sizeof(float) * size_t(w.max_slots) * attn::kBM * attn::kD, 256);
  w.part_lse = off; off = align_up(off + sizeof(float) * size_t(w.max_slots) * attn::kBM, 256);
  w.total = off;
  return w;
}

// ------------------------------------------------------------------------------ prep
struct ReqGeom {
  int o, T, P, mts, nts, units;
};

__device__ __forceinline__ ReqGeom req_geom(const TcDev& a, int r) {
  ReqGeom g;
  g.o = a.node_offset[r];
  g.T = a.node_offset[r + 1] - g.o;
  g.P = a.prefix_len[r];
  const int tpt = attn::kBM >> a.log2G;
  const bool ok = a.req_status[r] == 0 && g.T >= 1 && g.P >= 0;
  g.mts = ok ? (g.T + tpt - 1) / tpt : 0;
  g.nts = ok ? (g.P + g.T + attn::kBN - 1) / attn::kBN : 0;
  g.units = a.H_kv * g.mts;
  return g;
}

// Block-wide exclusive scan of one int per thread (1024 threads); returns the block total.
__device__ int block_excl_scan(int v, int* s_warp, int& excl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += t;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int y = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += t;
    }
    s_warp[lane] = y;
  }
  __syncthreads();
  const int warp_base = warp ? s_warp[warp - 1] : 0;
  excl = warp_base + x - v;
  const int total = s_warp[31];
  __syncthreads();
  return total;
}

// Per-request geometry used by the range walk: shared memory for batches up to kPrepSmemReqs
// requests (the usual case), global memory beyond.
constexpr int kPrepSmemReqs = 2048;

struct PrepGeo {
  const int* tiles;   // [B + 1] exclusive prefix of tile work
  const int* nts;     // [B] KV tiles per unit
  const int* mts;     // [B] M-tiles per KV head
};

// Walks range [t0, t1) of the global tile stream; calls emit(r, h, mt, j0, j1, nts, mts) for
// every piece of a unit that falls in the range, in stream order.
template <typename F>
__device__ void walk_range(const TcDev& a, const PrepGeo& geo, long long t0, long long t1,
                           F&& emit) {
  if (t0 >= t1) return;
  int lo = 0, hi = a.B - 1;  // last request whose work starts at or before t0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (geo.tiles[mid] <= t0) lo = mid; else hi = mid - 1;
  }
  long long t = t0;
  for (int r = lo; r < a.B && t < t1; ++r) {
    const long long rbeg = geo.tiles[r], rend = geo.tiles[r + 1];
    if (rend <= t) continue;
    const int nts = geo.nts[r], mts = geo.mts[r];
    while (t < t1 && t < rend) {
      const long long off = t - rbeg;
      const int u = int(off / nts);
      const int j0 = int(off - (long long)u * nts);
      const int j1 = int(min((long long)nts, (long long)j0 + (t1 - t)));
      emit(r, u / mts, u % mts, j0, j1, nts, mts);
      t += j1 - j0;
    }
  }
}

__global__ void __launch_bounds__(1024) attn_prep_kernel(TcDev a) {
  __shared__ int s_warp[32];
  __shared__ int s_tiles[kPrepSmemReqs + 1];
  __shared__ int s_nts[kPrepSmemReqs];
  __shared__ int s_mts[kPrepSmemReqs];
  const int tid = threadIdx.x;
  const bool in_smem = a.B <= kPrepSmemReqs;
  // per-request geometry and tile work, exclusive prefix (in chunks of 1024 requests); the
  // global copies (req_tiles, and nts / mts recomputed on the fly) back batches that do not fit
  int carry = 0;
  for (int r0 = 0; r0 < a.B; r0 += 1024) {
    const int r = r0 + tid;
    int tiles = 0;
    if (r < a.B) {
      const ReqGeom g0 = req_geom(a, r);
      const int nblk = (g0.P + g0.T + attn::kBS - 1) / attn::kBS;
      ReqGeom g = g0;
      if (g0.units > 0 && nblk > a.max_blocks) {
        atomicOr(&a.req_status[r], SPEC_REQ_BAD_BLOCK);
        g.mts = g.nts = g.units = 0;
      }
      tiles = g.units * g.nts;
      if (in_smem) {
        s_nts[r] = g.nts;
        s_mts[r] = g.mts;
      }
    }
    int e;
    const int tot = block_excl_scan(tiles, s_warp, e);
    if (r < a.B) {
      a.req_tiles[r] = carry + e;
      if (in_smem) s_tiles[r] = carry + e;
    }
    carry += tot;
  }
  if (tid == 0) {
    a.req_tiles[a.B] = carry;
    if (in_smem) s_tiles[a.B] = carry;
  }
  __syncthreads();
  PrepGeo geo;
  if (in_smem) {
    geo.tiles = s_tiles;
    geo.nts = s_nts;
    geo.mts = s_mts;
  } else {
    // large batches: global prefix; nts / mts are recomputed from the inputs per request
    geo.tiles = a.req_tiles;
    geo.nts = nullptr;
    geo.mts = nullptr;
  }
  const long long total = carry;
  const int C = int(max(1LL, min((long long)a.ctas, total / attn::kMinTilesPerRange)));
  const bool mine = tid < C;
  const long long t0 = mine ? total * tid / C : 0, t1 = mine ? total * (tid + 1) / C : 0;
  auto walk = [&](auto&& emit) {
    if (in_smem) {
      walk_range(a, geo, t0, t1, emit);
    } else {
      // same walk with geometry from global memory
      if (t0 >= t1) return;
      int lo = 0, hi = a.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.req_tiles[mid] <= t0) lo = mid; else hi = mid - 1;
      }
      long long t = t0;
      for (int r = lo; r < a.B && t < t1; ++r) {
        const long long rbeg = a.req_tiles[r], rend = a.req_tiles[r + 1];
        if (rend <= t) continue;
        const ReqGeom g = req_geom(a, r);
        while (t < t1 && t < rend) {
          const long long off = t - rbeg;
          const int u = int(off / g.nts);
          const int j0 = int(off - (long long)u * g.nts);
          const int j1 = int(min((long long)g.nts, (long long)j0 + (t1 - t)));
          emit(r, u / g.mts, u % g.mts, j0, j1, g.nts, g.mts);
          t += j1 - j0;
        }
      }
    }
  };
  // pass 1: pieces, partial pieces and merge records per range
  int n = 0, np = 0, nc = 0;
  walk([&](int, int, int, int j0, int j1, int nts, int) {
    ++n;
    if (j0 > 0 || j1 < nts) ++np;
    if (j0 == 0 && j1 < nts) ++nc;   // the unit starts here and continues in the next range
  });
  int e_items, e_part, e_comb;
  const int n_items = block_excl_scan(n, s_warp, e_items);
  block_excl_scan(np, s_warp, e_part);
  const int n_comb = block_excl_scan(nc, s_warp, e_comb);
  if (mine) a.cta_off[tid] = min(e_items, a.max_items);
  for (int c = C + tid; c <= a.ctas; c += 1024) a.cta_off[c] = min(n_items, a.max_items);
  if (tid == 0) {
    a.header[0] = min(n_items, a.max_items);
    a.header[1] = min(n_comb, a.max_combine);
  }
  // pass 2: items with partial slots (consecutive across ranges for a cut unit: its pieces are
  // the last partial piece of one range and the first of the following ones) + merge records
  int idx = e_items, slot = e_part, ci = e_comb;
  const int* tiles_pref = in_smem ? s_tiles : a.req_tiles;
  walk([&](int r, int h, int mt, int j0, int j1, int nts, int mts) {
    Item it;
    it.r = r; it.h = h; it.mt = mt; it.j0 = j0; it.j1 = j1; it.pad0 = it.pad1 = 0;
    const bool partial = j0 > 0 || j1 < nts;
    it.slot = partial ? slot : -1;
    if (j0 == 0 && j1 < nts) {
      const long long ubeg = tiles_pref[r] + (long long)(h * mts + mt) * nts;
      const long long uend = ubeg + nts;
      int pieces = 1;
      for (int c = tid + 1; c < C; ++c) {
        const long long c0 = total * c / C;
        if (c0 >= uend) break;
        if (total * (c + 1) / C > c0) ++pieces;
      }
      CombineUnit cu;
      cu.r = r; cu.h = h; cu.mt = mt; cu.slot0 = slot; cu.npieces = pieces;
      cu.pad0 = cu.pad1 = cu.pad2 = 0;
      if (ci < a.max_combine) a.combine[ci] = cu;
      ++ci;
    }
    if (partial) ++slot;
    if (idx < a.max_items) a.items[idx] = it;
    ++idx;
  });
}

// ------------------------------------------------------------------------------ main kernel
__device__ __forceinline__ uint32_t anc_window(const uint32_t (&anc)[8], int W, int pos) {
  // 32 mask bits starting at tree index `pos` (zero outside [0, 32 W))
  if (pos <= -32 || pos >= 32 * W) return 0u;
  const int wi = pos >= 0 ? (pos >> 5) : -1;
  const int sh = pos - 32 * wi;
  uint32_t lo = 0u, hi = 0u;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (k == wi && k < W) lo = anc[k];
    if (k == wi + 1 && k < W) hi = anc[k];
  }
  return sh == 0 ? lo : ((lo >> sh) | (hi << (32 - sh)));
}

// all 32 lanes wait; the outcome is made warp-uniform so warp-collective TMEM accesses that
// follow are executed by the full warp or by none of it
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  const bool ok = tc::mbar_wait(bar, parity, abort, attn::kWaitLimit);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(a), "f"(b));
  return r;
}

// In place: masked, log2-scaled scores of 32 columns starting at key `key0`; returns their max.
// Columns inside the prefix need no mask (one multiply and one max per score).
__device__ __forceinline__ float mask_max32(uint32_t (&x)[32], bool valid, int key0, int P,
                                            const uint32_t (&anc)[8], int W, float sl2) {
  float mx = -INFINITY;
  if (key0 + 32 <= P) {
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float v = __uint_as_float(x[c]) * sl2;
      x[c] = __float_as_uint(v);
      mx = fmaxf(mx, v);
    }
    return valid ? mx : -INFINITY;
  }
  const uint32_t wd = anc_window(anc, W, key0 - P);
  const int npre = P - key0;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const bool vis = valid && ((c < npre) || ((wd >> c) & 1u));
    const float v = vis ? __uint_as_float(x[c]) * sl2 : -INFINITY;
    x[c] = __float_as_uint(v);
    mx = fmaxf(mx, v);
  }
  return mx;
}

__global__ void __launch_bounds__(attn::kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mK8,
               const __grid_constant__ CUtensorMap mV8, TcDev a) {
  using namespace attn;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = base + kSmemQ;
  uint8_t* sK = base + kSmemK;
  uint8_t* sV = base + kSmemV;
  uint8_t* sP = base + kSmemP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kSmemBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;     // [kKStages]
  uint64_t* k_empty = bars + 5;    // [kKStages]
  uint64_t* v_full = bars + 8;     // [kVStages]
  uint64_t* v_empty = bars + 10;   // [kVStages]
  uint64_t* s_full = bars + 12;    // [2]
  uint64_t* s_free = bars + 14;    // [2]
  uint64_t* p_full = bars + 16;
  uint64_t* pv_done = bars + 17;
  uint64_t* o_free = bars + 18;
  uint64_t* drain = bars + 19;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 20);
  int* s_abort = reinterpret_cast<int*>(bars + 21);
  uint64_t* ex_bar = bars + 22;    // [4]: row-sum exchange of the two softmax halves

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_empty, 1);
    for (int s = 0; s < kKStages; ++s) {
      tc::mbar_init(k_full + s, 1);
      tc::mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::mbar_init(v_full + s, 1);
      tc::mbar_init(v_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(s_full + s, 1);
      tc::mbar_init(s_free + s, 8);
    }
    tc::mbar_init(p_full, 8);
    tc::mbar_init(pv_done, 1);
    tc::mbar_init(o_free, 8);
    tc::mbar_init(drain, 1);
    for (int q = 0; q < 4; ++q) tc::mbar_init(ex_bar + q, 2);
    // the 1024-byte aligned layout must fit in the dynamic allocation
    *s_abort = (tc::smem_u32(base) + kSmemEnd > tc::smem_u32(smem_raw) + kSmemBytes) ? 1 : 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int it_beg = a.cta_off[blockIdx.x], it_end = a.cta_off[blockIdx.x + 1];
  volatile int* abort_flag = s_abort;
  const int G = a.G, log2G = a.log2G, tpt = kBM >> log2G;
  const bool layout_ok = *abort_flag == 0;

  if (layout_ok && (warp == 0 || warp == 2)) {
    // ===================================================================== TMA producers
    // warp 0 loads Q and K, warp 2 loads V.  Lanes 0..7 fetch the eight block-table entries
    // of a tile (a tile ahead).  When the tile's pages are consecutive physical blocks one
    // 4-D box per 64-column half brings all eight (16 KB); otherwise each lane issues the two
    // boxes of its own page (2 KB each) -- small boxes cap the copy rate well below HBM speed.
    const bool is_k = warp == 0;
    if (lane == 0) {
      tc::prefetch_tensormap(is_k ? &mK : &mV);
      tc::prefetch_tensormap(is_k ? &mK8 : &mV8);
      if (is_k) tc::prefetch_tensormap(&mQ);
    }
    const CUtensorMap* map = is_k ? &mK : &mV;
    const CUtensorMap* map8 = is_k ? &mK8 : &mV8;
    const int nstage = is_k ? kKStages : kVStages;
    uint8_t* ring = is_k ? sK : sV;
    uint64_t* full = is_k ? k_full : v_full;
    uint64_t* empty = is_k ? k_empty : v_empty;
    int kt = 0, li = 0;
    bool ok = true;
    auto wait_lane0 = [&](uint64_t* bar, uint32_t parity) -> bool {
      bool r = true;
      if (lane == 0) r = tc::mbar_wait(bar, parity, abort_flag, kWaitLimit);
      return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    for (int idx = it_beg; idx < it_end && ok; ++idx, ++li) {
      const Item it = a.items[idx];
      const int o = a.node_offset[it.r];
      const int T = a.node_offset[it.r + 1] - o;
      const int P = a.prefix_len[it.r];
      const int nblk = (P + T + kBS - 1) / kBS;
      const int32_t* table = a.block_table + size_t(it.r) * a.max_blocks;
      // physical block of this lane's page of tile j: -1 past the request, -2 if invalid
      auto tile_pb = [&](int j) -> int {
        int pb = -1;
        const int lb = j * 8 + lane;
        if (lane < 8 && lb < nblk) {
          pb = table[lb];
          if (pb < 0 || pb >= a.num_blocks) {
            atomicOr(&a.req_status[it.r], SPEC_REQ_BAD_BLOCK);
            pb = -2;
          }
        }
        return pb;
      };
      if (is_k) {
        if (li > 0 && !wait_lane0(q_empty, (li - 1) & 1)) { ok = false; break; }
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(q_full, kTile);
          tc::tma_load_3d(sQ, &mQ, 0, it.h * G, o + it.mt * tpt, q_full);
          tc::tma_load_3d(sQ + kAtom, &mQ, 64, it.h * G, o + it.mt * tpt, q_full);
        }
      }
      int pb_cur = tile_pb(it.j0);
      for (int j = it.j0; j < it.j1; ++j, ++kt) {
        const int pb_next = (j + 1 < it.j1) ? tile_pb(j + 1) : -1;
        const int st = kt % nstage, use = kt / nstage;
        if (use > 0 && !wait_lane0(empty + st, (use - 1) & 1)) { ok = false; break; }
        const int pb0 = __shfl_sync(0xffffffffu, pb_cur, 0);
        const bool contig = __all_sync(0xffffffffu, lane >= 8 || pb_cur == -1 || pb_cur == pb0 + lane) && pb0 >= 0;
        if (lane == 0) tc::mbar_arrive_expect_tx(full + st, kTile);
        __syncwarp();
        uint8_t* dst = ring + st * kTile;
        if (contig) {
          if (lane == 0) {
            tc::tma_load_4d(dst, map8, 0, 0, it.h, pb0, full + st);
            tc::tma_load_4d(dst + kAtom, map8, 64, 0, it.h, pb0, full + st);
          }
        } else if (lane < 8) {
          const int row = pb_cur >= 0 ? (pb_cur * a.H_kv + it.h) * kBS : a.kv_rows;  // zeros
          tc::tma_load_2d(dst + lane * 2048, map, 0, row, full + st);
          tc::tma_load_2d(dst + kAtom + lane * 2048, map, 64, row, full + st);
        }
        __syncwarp();
        pb_cur = pb_next;
      }
    }
    if (lane == 0) {
      if (!ok) *abort_flag = 1;
      // drain: wait for the copies issued last (bounded), so none is in flight at exit
      for (int k = max(0, kt - nstage); k < kt; ++k)
        tc::mbar_wait(full + k % nstage, (k / nstage) & 1, abort_flag, kWaitLimit / 8);
      if (is_k && li > 0) tc::mbar_wait(q_full, (li - 1) & 1, abort_flag, kWaitLimit / 8);
    }
  } else if (layout_ok && warp == 1) {
    // ===================================================================== MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_pv = tc::idesc_bf16_f32(128, 128, false, true);
      const uint32_t aQ = tc::smem_u32(sQ), aK = tc::smem_u32(sK), aV = tc::smem_u32(sV),
                     aP = tc::smem_u32(sP);
      const uint32_t tO = tmem + 256;
      int kv_it = 0, li = 0;
      bool ok = true;
      auto issue_pv = [&](int prev, bool first_pv) -> bool {
        const int pst = prev % kVStages, puse = prev / kVStages;
        if (!tc::mbar_wait(p_full, prev & 1, abort_flag, kWaitLimit)) return false;
        if (!tc::mbar_wait(v_full + pst, puse & 1, abort_flag, kWaitLimit)) return false;
        if (first_pv && li > 0 && !tc::mbar_wait(o_free, (li - 1) & 1, abort_flag, kWaitLimit))
          return false;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t da = tc::smem_desc(aP + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024);
          const uint64_t db = tc::smem_desc(aV + pst * kTile + kk * 2048, kAtom, 1024);
          tc::mma_bf16_ss(tO, da, db, id_pv, (first_pv && kk == 0) ? 0u : 1u);
        }
        tc::mma_commit(v_empty + pst);
        tc::mma_commit(pv_done);
        return true;
      };
      for (int idx = it_beg; idx < it_end && ok; ++idx, ++li) {
        const Item it = a.items[idx];
        if (!tc::mbar_wait(q_full, li & 1, abort_flag, kWaitLimit)) { ok = false; break; }
        bool first_pv = true;
        for (int j = it.j0; j < it.j1; ++j, ++kv_it) {
          const int st = kv_it & 1, use = kv_it >> 1;
          const int kst = kv_it % kKStages, kuse = kv_it / kKStages;
          if (!tc::mbar_wait(k_full + kst, kuse & 1, abort_flag, kWaitLimit)) { ok = false; break; }
          if (use > 0 && !tc::mbar_wait(s_free + st, (use - 1) & 1, abort_flag, kWaitLimit)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t tS = tmem + st * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t da = tc::smem_desc(aQ + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024);
            const uint64_t db = tc::smem_desc(aK + kst * kTile + (kk >> 2) * kAtom + (kk & 3) * 32, 16, 1024);
            tc::mma_bf16_ss(tS, da, db, id_qk, kk > 0 ? 1u : 0u);
          }
          tc::mma_commit(s_full + st);
          tc::mma_commit(k_empty + kst);
          if (j == it.j1 - 1) tc::mma_commit(q_empty);
          if (j > it.j0) {
            if (!issue_pv(kv_it - 1, first_pv)) { ok = false; break; }
            first_pv = false;
          }
        }
        if (!ok) break;
        if (!issue_pv(kv_it - 1, first_pv)) { ok = false; break; }
      }
      if (!ok) *abort_flag = 1;
      // drain every tcgen05 operation issued by this thread before TMEM is released
      tc::mma_commit(drain);
      tc::mbar_wait(drain, 0, abort_flag, kWaitLimit / 8);
    }
  } else if (layout_ok && warp >= 4) {
    // ===================================================================== softmax + epilogue
    const int q4 = warp & 3, hh = (warp - 4) >> 2;
    const int m = q4 * 32 + lane;
    const uint32_t lane_addr = uint32_t(q4 * 32) << 16;
    const int t_loc = m >> log2G, g = m & (G - 1);
    const float sl2 = a.scale_log2;
    float* red = reinterpret_cast<float*>(base + kSmemRed);   // [2][2][128]
    int ex_cnt = 0;
    bool ex_ok = true;
    // partner's value for this row: one mbarrier phase per exchange, double-buffered, bounded
    auto exchange = [&](float v) -> float {
      float* buf = red + (ex_cnt & 1) * 256;
      buf[hh * 128 + m] = v;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(ex_bar + q4);
      ex_ok = ex_ok && warp_wait(ex_bar + q4, ex_cnt & 1, abort_flag);
      ++ex_cnt;
      return buf[(1 - hh) * 128 + m];
    };
    int kv_it = 0, li = 0;
    bool ok = true;
    for (int idx = it_beg; idx < it_end && ok; ++idx, ++li) {
      const Item it = a.items[idx];
      const int o = a.node_offset[it.r];
      const int T = a.node_offset[it.r + 1] - o;
      const int P = a.prefix_len[it.r];
      const int kv_len = P + T;
      const int t = it.mt * tpt + t_loc;
      const bool valid = t < T;
      uint32_t anc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) anc[k] = (valid && k < a.W) ? a.anc[size_t(o + t) * a.W + k] : 0u;
      float m_ref = -INFINITY, l = 0.f;   // l: this half's share of the row sum
      // a warp whose 32 rows are all padding keeps only the barrier handshakes (and clears
      // its V rows on the last tile): no TMEM traffic, no math, no P writes -- its O rows
      // are never stored and P rows feed only their own O rows
      const bool live = __any_sync(0xffffffffu, valid);
      for (int j = it.j0; j < it.j1; ++j, ++kv_it) {
        const int st = kv_it & 1, use = kv_it >> 1;
        if (!warp_wait(s_full + st, use & 1, abort_flag)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t srow = tmem + lane_addr + st * 128;
        const int kbase = j * kBN;
        if (!live) {
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(s_free + st);
          if (j > it.j0 && !warp_wait(pv_done, (kv_it - 1) & 1, abort_flag)) { ok = false; break; }
        } else {
        // the partner half's 64 scores: only their max is needed
        float tmax;
        {
          uint32_t x0[32], x1[32];
          tc::tmem_ld32(srow + 64 * (1 - hh), x0);
          tc::tmem_ld32(srow + 64 * (1 - hh) + 32, x1);
          tc::tmem_ld_wait();
          tmax = fmaxf(mask_max32(x0, valid, kbase + 64 * (1 - hh), P, anc, a.W, sl2),
                       mask_max32(x1, valid, kbase + 64 * (1 - hh) + 32, P, anc, a.W, sl2));
        }
        // this half's 64 scores, kept for the exponentials; the S buffer is free afterwards
        uint32_t s0[32], s1[32];
        tc::tmem_ld32(srow + 64 * hh, s0);
        tc::tmem_ld32(srow + 64 * hh + 32, s1);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_free + st);
        tmax = fmaxf(tmax, mask_max32(s0, valid, kbase + 64 * hh, P, anc, a.W, sl2));
        tmax = fmaxf(tmax, mask_max32(s1, valid, kbase + 64 * hh + 32, P, anc, a.W, sl2));
        const bool grow = tmax > m_ref + kLazyRescale;
        const float new_ref = grow ? tmax : m_ref;
        const float factor = (grow && m_ref != -INFINITY) ? ex2(m_ref - new_ref) : 1.f;
        const bool has_ref = new_ref != -INFINITY;
        // exponentials (kept packed in registers) before waiting for the previous PV
        uint32_t pk[32];
        float rowsum = 0.f;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = has_ref ? ex2(__uint_as_float(s0[c]) - new_ref) : 0.f;
          const float p1 = has_ref ? ex2(__uint_as_float(s0[c + 1]) - new_ref) : 0.f;
          rowsum += p0 + p1;
          pk[c >> 1] = pack_bf16(p0, p1);
        }
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = has_ref ? ex2(__uint_as_float(s1[c]) - new_ref) : 0.f;
          const float p1 = has_ref ? ex2(__uint_as_float(s1[c + 1]) - new_ref) : 0.f;
          rowsum += p0 + p1;
          pk[16 + (c >> 1)] = pack_bf16(p0, p1);
        }
        // PV of the previous tile must be complete before P and O are touched
        if (j > it.j0 && !warp_wait(pv_done, (kv_it - 1) & 1, abort_flag)) { ok = false; break; }
        uint8_t* rowp = sP + hh * kAtom + (m >> 3) * 1024 + (m & 7) * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          *reinterpret_cast<uint4*>(rowp + ((ch ^ (m & 7)) << 4)) =
              make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
        // lazy rescale of this warp's half of the O accumulator (warp-collective TMEM access)
        const bool any_rescale = __any_sync(0xffffffffu, factor != 1.f) && j > it.j0;
        if (any_rescale) {
          tc::tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < 64; c0 += 32) {
            uint32_t r32[32];
            tc::tmem_ld32(tmem + lane_addr + 256 + 64 * hh + c0, r32);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) r32[c] = __float_as_uint(__uint_as_float(r32[c]) * factor);
            tc::tmem_st32(tmem + lane_addr + 256 + 64 * hh + c0, r32);
          }
          tc::tmem_st_wait();
        }
        l = l * factor + rowsum;
        m_ref = new_ref;
        }  // live
        // last tile: zero V rows past the request's KV length (stale cache rows times P = 0
        // must not turn into NaN); TMA must have landed first.  Half hh clears d-atom hh.
        if (kbase + kBN > kv_len) {
          if (!warp_wait(v_full + st, use & 1, abort_flag)) { ok = false; break; }
          const int key = m;
          if (key >= kv_len - kbase) {
            uint8_t* vrow = sV + st * kTile + hh * kAtom + (key >> 3) * 1024 + (key & 7) * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(p_full);
      }
      if (!ok) break;
      // epilogue: this warp writes output columns 64*hh .. 64*hh+63 of its rows
      if (!warp_wait(pv_done, (kv_it - 1) & 1, abort_flag)) { ok = false; break; }
      tc::tc_fence_after();
      if (!live) {
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(o_free);
        continue;
      }
      const float lt = l + exchange(l);
      if (!ex_ok) { ok = false; break; }
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float lse2 = lt > 0.f ? m_ref + __log2f(lt) : -INFINITY;
      if (it.slot < 0) {
        __nv_bfloat16* orow = a.o + (size_t(o + t) * a.H_q + it.h * G + g) * kD + 64 * hh;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t r32[32];
          tc::tmem_ld32(tmem + lane_addr + 256 + 64 * hh + c0, r32);
          tc::tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(r32[c]) * inv, __uint_as_float(r32[c + 1]) * inv);
              v.y = pack_bf16(__uint_as_float(r32[c + 2]) * inv, __uint_as_float(r32[c + 3]) * inv);
              v.z = pack_bf16(__uint_as_float(r32[c + 4]) * inv, __uint_as_float(r32[c + 5]) * inv);
              v.w = pack_bf16(__uint_as_float(r32[c + 6]) * inv, __uint_as_float(r32[c + 7]) * inv);
              *reinterpret_cast<uint4*>(orow + c0 + c) = v;
            }
          }
        }
        if (valid && hh == 0 && a.lse) a.lse[size_t(o + t) * a.H_q + it.h * G + g] = lse2 * 0.6931471805599453f;
      } else {
        float* prow = a.part_o + (size_t(it.slot) * kBM + m) * kD + 64 * hh;
#pragma unroll 1
        for (int c0 = 0; c0 < 64; c0 += 32) {
          uint32_t r32[32];
          tc::tmem_ld32(tmem + lane_addr + 256 + 64 * hh + c0, r32);
          tc::tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<float4*>(prow + c0 + c) =
                  make_float4(__uint_as_float(r32[c]) * inv, __uint_as_float(r32[c + 1]) * inv,
                              __uint_as_float(r32[c + 2]) * inv, __uint_as_float(r32[c + 3]) * inv);
          }
        }
        if (valid && hh == 0) a.part_lse[size_t(it.slot) * kBM + m] = lse2;
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(o_free);
    }
    if (!ok) *abort_flag = 1;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) {
    // every request of this CTA's range is unreliable after an expired wait
    for (int idx = it_beg; idx < it_end; ++idx) atomicOr(&a.req_status[a.items[idx].r], SPEC_REQ_TIMEOUT);
  }
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------ merge
// One warp per output row of a cut unit: lane L covers output columns 4L .. 4L+3.
__global__ void __launch_bounds__(128) attn_combine_kernel(TcDev a) {
  const int n_comb = a.header[1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tpt = attn::kBM >> a.log2G;
  for (int u = blockIdx.x; u < n_comb; u += gridDim.x) {
    const CombineUnit cu = a.combine[u];
    const int o = a.node_offset[cu.r];
    const int T = a.node_offset[cu.r + 1] - o;
    for (int m = warp; m < attn::kBM; m += 4) {
      const int t = cu.mt * tpt + (m >> a.log2G);
      const int g = m & (a.G - 1);
      if (t >= T) break;   // rows are token-major: this warp's remaining rows are past T
      float M = -INFINITY;
      for (int s = 0; s < cu.npieces; ++s)
        M = fmaxf(M, a.part_lse[size_t(cu.slot0 + s) * attn::kBM + m]);
      float wsum = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < cu.npieces; ++s) {
        const float ls = a.part_lse[size_t(cu.slot0 + s) * attn::kBM + m];
        if (ls == -INFINITY) continue;
        const float w = ex2(ls - M);
        wsum += w;
        const float4 v = *reinterpret_cast<const float4*>(
            a.part_o + (size_t(cu.slot0 + s) * attn::kBM + m) * attn::kD + 4 * lane);
        acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
      }
      const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
      __nv_bfloat16* orow = a.o + (size_t(o + t) * a.H_q + cu.h * a.G + g) * attn::kD + 4 * lane;
      uint2 v;
      v.x = pack_bf16(acc.x * inv, acc.y * inv);
      v.y = pack_bf16(acc.z * inv, acc.w * inv);
      *reinterpret_cast<uint2*>(orow) = v;
      if (lane == 0 && a.lse)
        a.lse[size_t(o + t) * a.H_q + cu.h * a.G + g] = (M + __log2f(wsum)) * 0.6931471805599453f;
    }
  }
}

// ------------------------------------------------------------------------------ host
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static int attention_ctas() {
  const int sms = sm_count_current_device();
  return sms < attn::kMaxCtas ? sms : attn::kMaxCtas;
}

size_t attention_tc_workspace_size(const spec_attn_params* p) {
  return tc_ws_layout(p, attention_ctas()).total;
}

spec_status_t launch_attention_tc(const spec_attn_params* p, void* ws, size_t ws_bytes,
                                  cudaStream_t s) {
  using namespace attn;
  const int G = p->H_q / p->H_kv;
  if (p->dtype != SPEC_BF16 || p->head_dim != kD || p->block_size != kBS) return SPEC_ERR_UNSUPPORTED;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return SPEC_ERR_UNSUPPORTED;
  const long long kv_rows = (long long)p->num_blocks * p->H_kv * kBS;
  if (kv_rows + kBS >= (1LL << 31) || (long long)p->N + kBM >= (1LL << 31))
    return SPEC_ERR_UNSUPPORTED;
  const int ctas = attention_ctas();
  if (ctas <= 0) return SPEC_ERR_CUDA;
  const TcWs lay = tc_ws_layout(p, ctas);
  if (!ws || ws_bytes < lay.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return SPEC_ERR_INVALID_ARG;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return SPEC_ERR_CUDA;
  CUtensorMap mQ, mK, mV, mK8, mV8;
  {
    cuuint64_t dims[3] = {cuuint64_t(kD), cuuint64_t(p->H_q), cuuint64_t(p->N)};
    cuuint64_t strides[2] = {cuuint64_t(kD) * 2, cuuint64_t(p->H_q) * kD * 2};
    cuuint32_t box[3] = {64, cuuint32_t(G), cuuint32_t(kBM / G)};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->q), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SPEC_ERR_INVALID_ARG;
  }
  for (int which = 0; which < 2; ++which) {
    cuuint64_t dims[2] = {cuuint64_t(kD), cuuint64_t(kv_rows)};
    cuuint64_t strides[1] = {cuuint64_t(kD) * 2};
    cuuint32_t box[2] = {64, cuuint32_t(kBS)};
    cuuint32_t es[2] = {1, 1};
    void* ptr = const_cast<void*>(which ? p->v_cache : p->k_cache);
    if (enc(which ? &mV : &mK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SPEC_ERR_INVALID_ARG;
  }
  // 4-D view [num_blocks][H_kv][16 slots][128] of each cache: one box = 8 consecutive blocks
  for (int which = 0; which < 2; ++which) {
    cuuint64_t dims[4] = {cuuint64_t(kD), cuuint64_t(kBS), cuuint64_t(p->H_kv), cuuint64_t(p->num_blocks)};
    cuuint64_t strides[3] = {cuuint64_t(kD) * 2, cuuint64_t(kBS) * kD * 2,
                             cuuint64_t(p->H_kv) * kBS * kD * 2};
    cuuint32_t box[4] = {64, cuuint32_t(kBS), 1, 8};
    cuuint32_t es[4] = {1, 1, 1, 1};
    void* ptr = const_cast<void*>(which ? p->v_cache : p->k_cache);
    if (enc(which ? &mV8 : &mK8, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, ptr, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SPEC_ERR_INVALID_ARG;
  }
  char* w = static_cast<char*>(ws);
  TcDev d;
  d.block_table = p->block_table;
  d.prefix_len = p->prefix_len;
  d.node_offset = p->node_offset;
  d.anc = p->anc_mask;
  d.o = static_cast<__nv_bfloat16*>(p->o);
  d.lse = p->lse;
  d.req_status = p->req_status;
  d.header = reinterpret_cast<int*>(w + lay.header);
  d.cta_off = reinterpret_cast<int*>(w + lay.cta_off);
  d.req_tiles = reinterpret_cast<int*>(w + lay.req_tiles);
  d.items = reinterpret_cast<Item*>(w + lay.items);
  d.combine = reinterpret_cast<CombineUnit*>(w + lay.combine);
  d.part_o = reinterpret_cast<float*>(w + lay.part_o);
  d.part_lse = reinterpret_cast<float*>(w + lay.part_lse);
  d.B = p->B; d.N = p->N; d.H_q = p->H_q; d.H_kv = p->H_kv; d.G = G;
  d.log2G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : 4;
  d.T_max = p->T_max; d.W = (p->T_max + 31) / 32;
  d.num_blocks = p->num_blocks; d.max_blocks = p->max_blocks_per_req;
  d.kv_rows = int(kv_rows);
  d.ctas = ctas;
  d.max_items = lay.max_items; d.max_combine = lay.max_combine;
  const float scale = p->scale > 0.f ? p->scale : 1.f / sqrtf(float(kD));
  d.scale_log2 = scale * 1.4426950408889634f;
  static std::once_flag attr_once;
  std::call_once(attr_once, [] {
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  attn_prep_kernel<<<1, 1024, 0, s>>>(d);
  attn_tc_kernel<<<ctas, kThreads, kSmemBytes, s>>>(mQ, mK, mV, mK8, mV8, d);
  attn_combine_kernel<<<lay.max_combine, 128, 0, s>>>(d);
  return launch_status();
}

}  // namespace spec
