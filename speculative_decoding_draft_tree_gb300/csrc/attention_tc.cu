// bf16 tree attention on the tcgen05 tensor cores (sm_103a).
//
// Sources: "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的验证——树形掩码 -- one forward over the
// flattened tree with the ancestor mask, tree position ids and the KV cache; "万字综述 10+ 种 LLM
// 投机采样推理加速方案" (m.haoling.cc) 5.2 -- tree-based decoding shares the prefix through the mask
// instead of one KV copy per branch; 12.4.3 -- PagedAttention and FlashDecoding are the framework
// features verification has to fit (paged KV blocks, KV split across CTAs + log-sum-exp merge).
//
// Rows: the G query heads of KV head h times up to 128/G tree tokens, stacked token-major into
// 128 MMA rows per M-tile (row m = t_local * G + g).  Work unit = (request r, KV head h, pair of
// M-tiles): each K/V tile of the request's P_r + T_r logical KV slots (tiles of 128 keys = 8
// paged blocks of 16) is read from HBM once for both M-tiles of the pair, so a unit with 2 M-tiles
// (up to 256 rows) costs one pass over its K/V, not two.  A unit with one M-tile splits its K/V
// tiles between the two slots by parity and merges their softmax states at the end.  The units are
// laid end to end (request, head, pair order) as one stream of K/V tiles cut into equal
// contiguous ranges, one per persistent CTA (one CTA per SM); each CTA finds its own range with
// two block-wide passes over the requests at start-up, so there is no separate partition launch.
// A unit cut by a range boundary is computed in pieces that write fp32 partial outputs and
// log-sum-exps; the CTA holding a cut unit's first piece leaves a merge record, and a small merge
// kernel combines the pieces by log-sum-exp.  Every other unit writes its output directly.
//
// CTA (384 threads), two slots s = 0, 1 (an M-tile each, or half of the K/V tiles of one):
//   warp 0      Q and K producer, warp 2 V producer: 128-byte-swizzled TMA boxes (one 4-D box per
//               64-column half when a tile's 8 paged blocks are consecutive, else one per block,
//               issued by 8 lanes); blocks past the request or with a bad block id are read from
//               an out-of-range row (TMA fills zeros).  K has 3 stages, V 2; Q one tile per slot;
//   warp 1      one thread issues every tcgen05.mma: S_s = Q_s K^T (M = N = 128, K = 16 x 8)
//               into TMEM and O_s += P_s V (P_s read from TMEM, V as an MN-major operand) into
//               the slot's TMEM accumulator, the slots interleaved so that one slot's products
//               run while the other slot's softmax works;
//   warps 4..7 (slot 0), 8..11 (slot 1): softmax, one query row per thread: the row maximum over
//               the tile's visible keys (masked by the ancestor bits), exponentials against a
//               lazily updated reference (O_s rescaled only when the maximum grows by more than
//               2^8), P_s (bf16) written over the upper half of S_s in TMEM (a thread holds 64
//               scores at a time: keys 0..63 are read twice); the epilogue normalises O_s and writes
//               the output rows (a split unit: each slot writes 64 columns of the merged rows).
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
constexpr int kThreads = 384;                 // 4 control warps + 2 slots x 4 softmax warps
constexpr int kAtom = 16384;                  // 128 rows x 128 B
constexpr int kTile = 2 * kAtom;              // 128 x 128 bf16
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kSmemQ = 0;                     // one Q tile per slot
constexpr int kSmemK = kSmemQ + 2 * kTile;
constexpr int kSmemV = kSmemK + kKStages * kTile;
constexpr int kSmemBar = kSmemV + kVStages * kTile;
constexpr int kSmemX = kSmemBar + 256;        // [2 slots][reference, sum][128 rows] fp32
constexpr int kSmemEnd = kSmemX + 2048;
constexpr int kSmemBytes = 232448;            // the per-CTA maximum; the slack aligns the base
constexpr long long kWaitLimit = 4000000000LL;     // clock cycles (~2 s)
constexpr float kLazyRescale = 8.0f;          // log2 units
constexpr int kMaxCtas = 1024;                // persistent CTAs at most
constexpr int kMinTilesPerRange = 4;          // small problems use fewer, longer ranges
constexpr int kPartRows = 2 * kBM;            // rows of one partial piece (up to two M-tiles)
constexpr int kCtlRegs = 96;                  // registers per thread: control warpgroup
constexpr int kSoftmaxRegs = 200;             // and each softmax warpgroup (setmaxnreg)
static_assert(kCtlRegs * 128 + kSoftmaxRegs * 256 <= kThreads * 168, "register split fits");
// TMEM columns: slot s's scores S_s (fp32) in 128 s .. 128 s + 127, overwritten by its
// probabilities P_s (bf16 pairs) in 128 s + 64 .. 128 s + 127; slot s's output O_s in 256 + 128 s ..
}  // namespace attn

// A unit cut by range boundaries: its pieces lie in ranges ca .. ca + np - 1; the first piece's
// partial slot is slot0 (2 ca, or 2 ca + 1 when the unit starts inside range ca), piece p > 0
// starts range ca + p and uses slot 2 (ca + p).  The unit covers M-tiles mt .. mt + nmt - 1.
struct MergeRec {
  int np, h, mt, nmt, o, T, ca, slot0;
};

struct TcDev {
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* node_offset;
  const uint32_t* anc;
  __nv_bfloat16* o;
  float* lse;
  int32_t* req_status;
  struct MergeRec* recs;   // [ctas]: the cut unit whose first piece CTA c holds (np = 0: none)
  float* part_o;      // [2 ctas][kPartRows][128] partial outputs of the pieces of cut units
  float* part_lse;    // [2 ctas][kPartRows] their log2-sum-exps
  int B, N, H_q, H_kv, G, log2G, T_max, W, num_blocks, max_blocks, kv_rows, ctas;
  float scale_log2;
};

// ------------------------------------------------------------------------------ workspace
struct TcWs {
  size_t recs, part_o, part_lse, total;
};

static TcWs tc_ws_layout(int ctas) {
  TcWs w;
  const size_t slots = 2 * size_t(ctas);   // at most two partial pieces per range
  size_t off = 0;
  w.recs = off; off = align_up(off + sizeof(MergeRec) * size_t(ctas), 256);
  w.part_o = off; off = align_up(off + sizeof(float) * slots * attn::kPartRows * attn::kD, 256);
  w.part_lse = off; off = align_up(off + sizeof(float) * slots * attn::kPartRows, 256);
  w.total = off;
  return w;
}

// ------------------------------------------------------------------------------ partition
struct ReqGeom {
  int o, T, P, mts, ups, nts, units;   // ups: units per KV head, one per pair of M-tiles
};

// Geometry of request r.  The status bits this kernel sets itself (BAD_BLOCK, TIMEOUT) are
// ignored, so every role of every CTA derives the same work from the same inputs; a request whose
// KV slots do not fit its block-table row gets no work.
__device__ __forceinline__ ReqGeom req_geom(const TcDev& a, int r) {
  ReqGeom g;
  g.o = a.node_offset[r];
  g.T = a.node_offset[r + 1] - g.o;
  g.P = a.prefix_len[r];
  const int tpt = attn::kBM >> a.log2G;
  const int st = a.req_status[r] & ~(SPEC_REQ_BAD_BLOCK | SPEC_REQ_TIMEOUT);
  const bool ok = st == 0 && g.T >= 1 && g.P >= 0 &&
                  (g.P + g.T + attn::kBS - 1) / attn::kBS <= a.max_blocks;
  g.mts = ok ? (g.T + tpt - 1) / tpt : 0;
  g.ups = (g.mts + 1) >> 1;
  g.nts = ok ? (g.P + g.T + attn::kBN - 1) / attn::kBN : 0;
  g.units = a.H_kv * g.ups;
  return g;
}

// This CTA's share of the tile stream.
struct Range {
  long long total;   // tiles in the stream
  long long t0, t1;  // this CTA's range [t0, t1)
  int C;             // ranges (CTAs blockIdx.x >= C have none)
  int r0, r1;        // requests holding tiles t0 and t1 - 1
  long long rbeg0, rbeg1;   // stream indices of their first tiles
};

__device__ __forceinline__ long long range_start(long long total, int C, int c) {
  return total * c / C;
}
// the range holding tile t (0 <= t < total): the largest c with range_start(c) <= t
__device__ __forceinline__ int range_of(long long t, long long total, int C) {
  const long long c = ((t + 1) * C + total - 1) / total - 1;
  return int(c < 0 ? 0 : (c >= C ? C - 1 : c));
}
// slot of the piece of the unit starting at tile ubeg that lies in range c
__device__ __forceinline__ int piece_slot(long long ubeg, long long total, int C, int c) {
  const long long rs = range_start(total, C, c);
  return (ubeg > rs) ? 2 * c + 1 : 2 * c;
}

// Every thread of the CTA (kThreads of them) computes the same Range: pass 1 sums the tile work
// of all requests, pass 2 scans it in chunks of kThreads requests until the chunk holding
// t1 - 1.  `s64` is scratch of at least kThreads / 32 + 2 entries, `s32` of two.  Contains
// __syncthreads.
template <int kThreads>
__device__ Range cta_range(const TcDev& a, long long* s64, int* s32) {
  using attn::kMinTilesPerRange;
  constexpr int kW = kThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  long long mine = 0;
  for (int r = tid; r < a.B; r += kThreads) {
    const ReqGeom g = req_geom(a, r);
    mine += (long long)g.units * g.nts;
    if (blockIdx.x == 0 && g.units == 0 && a.req_status[r] == 0 && g.T >= 1 && g.P >= 0)
      atomicOr(&a.req_status[r], SPEC_REQ_BAD_BLOCK);   // KV slots beyond the table row
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) s64[warp] = mine;
  __syncthreads();
  long long total = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) total += s64[w];
  Range R;
  R.total = total;
  R.C = int(max(1LL, min((long long)a.ctas, total / kMinTilesPerRange)));
  R.t0 = R.t1 = 0;
  R.r0 = R.r1 = 0;
  R.rbeg0 = R.rbeg1 = 0;
  const int c = blockIdx.x;
  if (total == 0 || c >= R.C) return R;   // uniform: no work for this CTA
  R.t0 = range_start(total, R.C, c);
  R.t1 = range_start(total, R.C, c + 1);
  long long base = 0;
  for (int r00 = 0; r00 < a.B; r00 += kThreads) {
    __syncthreads();   // s64 is rewritten below
    const int r = r00 + tid;
    long long tiles = 0;
    if (r < a.B) {
      const ReqGeom g = req_geom(a, r);
      tiles = (long long)g.units * g.nts;
    }
    long long incl = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    if (lane == 31) s64[warp] = incl;
    __syncthreads();
    long long before = 0, chunk = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      if (w < warp) before += s64[w];
      chunk += s64[w];
    }
    const long long hi = base + before + incl, lo = hi - tiles;
    const bool found = base + chunk > R.t1 - 1;   // uniform
    __syncthreads();
    if (tiles > 0 && lo <= R.t0 && R.t0 < hi) {
      s32[0] = r;
      s64[kW] = lo;
    }
    if (tiles > 0 && lo <= R.t1 - 1 && R.t1 - 1 < hi) {
      s32[1] = r;
      s64[kW + 1] = lo;
    }
    __syncthreads();
    base += chunk;
    if (found) break;
  }
  R.r0 = s32[0];
  R.rbeg0 = s64[kW];
  R.r1 = s32[1];
  R.rbeg1 = s64[kW + 1];
  // the scan always finds both requests; anything else would index out of bounds: no work
  if (R.r0 < 0 || R.r0 >= a.B || R.r1 < R.r0 || R.r1 >= a.B || R.rbeg0 > R.t0 || R.rbeg1 > R.t1 - 1)
    R.t0 = R.t1 = 0;
  return R;
}

// One piece of work: tiles [j0, j1) of unit (r, h, pair of M-tiles starting at mt).  pair: the
// unit has M-tiles mt and mt + 1 (one per slot, both reading every K/V tile); otherwise it has
// M-tile mt alone and the slots take alternate K/V tiles.
struct Item {
  int r, h, mt, j0, j1;
  bool pair;
  int slot;           // >= 0: a partial piece of a cut unit, written to part_o[slot]
  int o, T, P, nts;
  long long ubeg;     // stream index of the unit's first tile
};

// Walks this CTA's range in stream order; every role runs its own copy.
struct ItemIter {
  long long t, rbeg, rend;
  int r;
  ReqGeom g;
  __device__ __forceinline__ void start(const TcDev& a, const Range& R) {
    t = R.t0;
    r = R.r0;
    rbeg = rend = R.rbeg0;
    if (t < R.t1) {
      g = req_geom(a, r);
      rend = rbeg + (long long)g.units * g.nts;
    }
  }
  __device__ __forceinline__ bool next(const TcDev& a, const Range& R, Item& it) {
    if (t >= R.t1) return false;
    while (t >= rend) {
      if (r + 1 >= a.B) return false;
      ++r;
      g = req_geom(a, r);
      rbeg = rend;
      rend = rbeg + (long long)g.units * g.nts;
    }
    const long long off = t - rbeg;
    const int u = int(off / g.nts);
    it.r = r;
    it.h = u / g.ups;
    it.mt = 2 * (u - it.h * g.ups);
    it.pair = it.mt + 1 < g.mts;
    it.j0 = int(off - (long long)u * g.nts);
    it.j1 = int(min((long long)g.nts, (long long)it.j0 + (R.t1 - t)));
    it.o = g.o;
    it.T = g.T;
    it.P = g.P;
    it.nts = g.nts;
    it.ubeg = rbeg + (long long)u * g.nts;
    const bool partial = it.j0 > 0 || it.j1 < g.nts;
    it.slot = partial ? (t == R.t0 ? 2 * int(blockIdx.x) : 2 * int(blockIdx.x) + 1) : -1;
    t += it.j1 - it.j0;
    return true;
  }
};

// Thread 0 of CTA c: the merge record of range c -- the unit holding the range's last tile, if it
// starts in this range and continues past it.
__device__ __forceinline__ void write_merge_record(const TcDev& a, const Range& R) {
  MergeRec rec;
  rec.np = 0;
  rec.h = rec.mt = rec.nmt = rec.o = rec.T = rec.ca = rec.slot0 = 0;
  if (R.t0 < R.t1) {
    const ReqGeom g = req_geom(a, R.r1);
    const long long u = (R.t1 - 1 - R.rbeg1) / g.nts;
    const long long ubeg = R.rbeg1 + u * g.nts;
    if (ubeg >= R.t0 && ubeg + g.nts > R.t1) {
      rec.ca = int(blockIdx.x);
      rec.np = range_of(ubeg + g.nts - 1, R.total, R.C) - rec.ca + 1;
      rec.h = int(u) / g.ups;
      rec.mt = 2 * (int(u) - rec.h * g.ups);
      rec.nmt = rec.mt + 1 < g.mts ? 2 : 1;
      rec.o = g.o;
      rec.T = g.T;
      rec.slot0 = piece_slot(ubeg, R.total, R.C, rec.ca);
    }
  }
  a.recs[blockIdx.x] = rec;
}

// ------------------------------------------------------------------------------ main kernel
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


// 32 exponentials 2^(x sl + add) of one key chunk (masked keys hold -inf), the arguments formed
// two at a time by a packed FMA and summed two at a time into the packed partial sum `acc`, and
// stored as 16 columns of bf16 pairs at TMEM address `dst`
__device__ __forceinline__ void exp_chunk(const uint32_t (&x)[32], uint64_t sl2, uint64_t add2,
                                          uint64_t& acc, uint32_t dst) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float y0, y1;
    f2_unpack(f2_fma(f2_pack(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1])), sl2, add2),
              y0, y1);
    const float p0 = ex2(y0), p1 = ex2(y1);
    acc = f2_add(acc, f2_pack(p0, p1));
    pk[i] = pack_bf16(p0, p1);
  }
  tc::tmem_st16(dst, pk);
}


// Maximum of 32 values as a tree of three-input maxima (17 operations, depth 4).
__device__ __forceinline__ float max32_tree(const uint32_t (&x)[32]) {
  float m[11];
#pragma unroll
  for (int c = 0; c < 10; ++c)
    m[c] = fmax3(__uint_as_float(x[3 * c]), __uint_as_float(x[3 * c + 1]),
                 __uint_as_float(x[3 * c + 2]));
  m[10] = fmaxf(__uint_as_float(x[30]), __uint_as_float(x[31]));
  const float a = fmax3(m[0], m[1], m[2]), b = fmax3(m[3], m[4], m[5]);
  const float c = fmax3(m[6], m[7], m[8]), d = fmaxf(m[9], m[10]);
  return fmaxf(fmax3(a, b, c), d);
}

// 32 ancestor-mask bits of a query row starting at tree index `pos` (zero outside [0, 32 W)),
// read from the row's words in global memory (only tiles that reach the tree need them)
__device__ __forceinline__ uint32_t anc_window_g(const uint32_t* row, int W, int pos) {
  if (row == nullptr || pos <= -32 || pos >= 32 * W) return 0u;
  const int wi = pos >= 0 ? (pos >> 5) : -1;
  const int sh = pos - 32 * wi;
  const uint32_t lo = wi >= 0 ? __ldg(row + wi) : 0u;
  const uint32_t hi = (sh != 0 && wi + 1 < W) ? __ldg(row + wi + 1) : 0u;
  return sh == 0 ? lo : ((lo >> sh) | (hi << (32 - sh)));
}

// Masked raw (unscaled) scores of 32 columns starting at key `key0`, in place: invisible keys
// become -inf; returns the maximum of the visible ones.  Columns inside the prefix need no mask.
// Scaling by a positive constant commutes with the maximum, so the caller scales the maximum
// once and folds the scale into the exponentials' FMA.  The row's ancestor bits are read from
// global memory (`row` is null for a padding row).
__device__ __forceinline__ float mask_max32_row(uint32_t (&x)[32], bool valid, int key0, int P,
                                                const uint32_t* row, int W) {
  if (key0 + 32 <= P) return valid ? max32_tree(x) : -INFINITY;
  const uint32_t wd = anc_window_g(row, W, key0 - P);
  const int npre = P - key0;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const bool vis = valid && ((c < npre) || ((wd >> c) & 1u));
    x[c] = vis ? x[c] : __float_as_uint(-INFINITY);
  }
  return max32_tree(x);
}

// One lane waits (bounded), the warp gets the outcome.
__device__ __forceinline__ bool lane0_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  bool r = true;
  if ((threadIdx.x & 31) == 0) r = tc::mbar_wait(bar, parity, abort, attn::kWaitLimit);
  return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
}

// TMA producer warp (K and Q: is_k; V otherwise) walking the CTA's items.  Lanes 0..7 fetch
// the eight block-table entries of a tile (a tile ahead).  When the tile's pages are
// consecutive physical blocks one 4-D box per 64-column half brings all eight (16 KB);
// otherwise each lane issues the two boxes of its own page (2 KB each) -- small boxes cap the
// copy rate well below HBM speed.  Pages past the request or with a bad block id are read from
// an out-of-range row (TMA fills zeros).  The K warp also loads each item's Q: for each M-tile
// b of the item (two for a pair item, else one), q_bytes from two boxes of `qmap` at
// (0 | 64, head * G, first tree token + (mt + b) * q_tokens) into buffer b (sQ + b * q_bytes,
// halves q_half apart), completing on q_full[b] once q_empty[b] released its previous contents.
// Inlined into the kernel so that every tensor map address is the kernel parameter's own; a map
// address in local or shared memory (which TMA cannot read) aborts without issuing a copy.
// Returns false if a wait expired; every copy issued is waited for (bounded) before return.
__device__ __forceinline__ bool tma_producer(
    const TcDev& a, const Range& R, bool is_k, const CUtensorMap* map, const CUtensorMap* map8,
    int nstage, uint8_t* ring, uint64_t* full, uint64_t* empty, const CUtensorMap* qmap,
    uint8_t* sQ, int q_half, int q_bytes, int q_tokens, uint64_t* q_full, uint64_t* q_empty,
    volatile int* abort_flag) {
  using namespace attn;
  const int lane = threadIdx.x & 31;
  int kt = 0, qn[2] = {0, 0};   // tiles and Q loads issued
  bool ok = !(__isLocal(map) || __isShared(map) || __isLocal(map8) || __isShared(map8) ||
              __isLocal(qmap) || __isShared(qmap));
  ItemIter iter;
  iter.start(a, R);
  Item it;
  while (ok && iter.next(a, R, it)) {
    const int nblk = (it.P + it.T + kBS - 1) / kBS;
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
      for (int b = 0; b < (it.pair ? 2 : 1); ++b) {
        if (qn[b] > 0 && !lane0_wait(q_empty + b, (qn[b] - 1) & 1, abort_flag)) { ok = false; break; }
        if (lane == 0) {
          tc::mbar_arrive_expect_tx(q_full + b, q_bytes);
          const int row = it.o + (it.mt + b) * q_tokens;
          uint8_t* dst = sQ + b * q_bytes;
          tc::tma_load_3d(dst, qmap, 0, it.h * a.G, row, q_full + b);
          tc::tma_load_3d(dst + q_half, qmap, 64, it.h * a.G, row, q_full + b);
        }
        ++qn[b];
      }
      if (!ok) break;
    }
    int pb_cur = tile_pb(it.j0);
    for (int j = it.j0; j < it.j1; ++j, ++kt) {
      const int pb_next = (j + 1 < it.j1) ? tile_pb(j + 1) : -1;
      const int st = kt % nstage, use = kt / nstage;
      if (use > 0 && !lane0_wait(empty + st, (use - 1) & 1, abort_flag)) { ok = false; break; }
      const int pb0 = __shfl_sync(0xffffffffu, pb_cur, 0);
      // one wide box only when all eight pages exist and are consecutive: on a request's last
      // tile the pages past its end are zero-filled per page (out of bounds, no DRAM traffic)
      // instead of being read from whatever blocks follow
      const bool contig = __all_sync(0xffffffffu, lane >= 8 || pb_cur == pb0 + lane) && pb0 >= 0;
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
    for (int b = 0; is_k && b < 2; ++b)
      if (qn[b] > 0) tc::mbar_wait(q_full + b, (qn[b] - 1) & 1, abort_flag, kWaitLimit / 8);
  }
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

__global__ void __launch_bounds__(attn::kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mK8,
               const __grid_constant__ CUtensorMap mV8, TcDev a) {
  using namespace attn;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = base + kSmemQ;                    // slot s's Q tile at sQ + s * kTile
  uint8_t* sK = base + kSmemK;
  uint8_t* sV = base + kSmemV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kSmemBar);
  uint64_t* q_full = bars + 0;                    // [2] per Q buffer
  uint64_t* q_empty = bars + 2;                   // [2]
  uint64_t* k_full = bars + 4;                    // [kKStages]
  uint64_t* k_empty = k_full + kKStages;          // [kKStages]
  uint64_t* v_full = k_empty + kKStages;          // [kVStages]
  uint64_t* v_empty = v_full + kVStages;          // [kVStages]
  uint64_t* s_full = v_empty + kVStages;          // [2] per slot: S_s = Q K^T landed
  uint64_t* p_full = s_full + 2;                  // [2]: P_s written (the slot's 4 warps)
  uint64_t* pv_done = p_full + 2;                 // [2]: O_s += P_s V completed
  uint64_t* o_free = pv_done + 2;                 // [2]: an item's epilogue has read O_s (8 warps)
  uint64_t* drain = o_free + 2;                   // the MMA issuer's last operations
  uint64_t* ex_bar = drain + 1;                   // [4] per lane quarter: the slots' exchange
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ex_bar + 4);
  int* s_abort = reinterpret_cast<int*>(ex_bar + 5);
  static_assert((4 + 2 * kKStages + 2 * kVStages + 8 + 1 + 4 + 2) * 8 <= 256,
                "barriers fit their 256-byte region");
  static_assert(kSmemK % 1024 == 0 && kSmemV % 1024 == 0, "swizzled tiles on 1024-byte bounds");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  // this CTA's range of the tile stream (the exchange area is free until the first epilogue)
  const Range R = cta_range<kThreads>(a, reinterpret_cast<long long*>(base + kSmemX),
                                      reinterpret_cast<int*>(base + kSmemX + 256));
  if (tid == 0) write_merge_record(a, R);
  if (R.t0 >= R.t1) return;   // uniform across the CTA: no work, nothing allocated yet
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(q_full + b, 1);
      tc::mbar_init(q_empty + b, 1);
      tc::mbar_init(s_full + b, 1);
      tc::mbar_init(p_full + b, 4);
      tc::mbar_init(pv_done + b, 1);
      tc::mbar_init(o_free + b, 8);
    }
    for (int s = 0; s < kKStages; ++s) {
      tc::mbar_init(k_full + s, 1);
      tc::mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      tc::mbar_init(v_full + s, 1);
      tc::mbar_init(v_empty + s, 1);
    }
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
  volatile int* abort_flag = s_abort;
  const int G = a.G, log2G = a.log2G, tpt = kBM >> log2G;
  const bool layout_ok = *abort_flag == 0;
  // registers move from the control warpgroup (warps 0..3: TMA, MMA issue) to the two softmax
  // warpgroups, which hold 64 of a row's scores at a time: 128 x 96 + 256 x 200 = 63488 of the
  // 384 x 168 the block was launched with
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtlRegs));
  if (layout_ok && (warp == 0 || warp == 2)) {
    // ===================================================================== TMA producers
    // warp 0 loads Q (one tile per M-tile of the item) and K, warp 2 loads V; on an expired wait
    // the producer raises the abort flag itself
    const bool is_k = warp == 0;
    if (lane == 0) {
      tc::prefetch_tensormap(is_k ? &mK : &mV);
      tc::prefetch_tensormap(is_k ? &mK8 : &mV8);
      if (is_k) tc::prefetch_tensormap(&mQ);
    }
    const CUtensorMap* map = is_k ? &mK : &mV;
    const CUtensorMap* map8 = is_k ? &mK8 : &mV8;
    tma_producer(a, R, is_k, map, map8, is_k ? kKStages : kVStages, is_k ? sK : sV,
                 is_k ? k_full : v_full, is_k ? k_empty : v_empty, &mQ, sQ, kAtom, kTile, tpt,
                 q_full, q_empty, abort_flag);
  } else if (layout_ok && warp == 1) {
    // ===================================================================== MMA issuer
    // One thread issues both products of both slots, in the order
    //   QK_0(0) QK_1(0) | PV_0(k) QK_0(k+1) PV_1(k) QK_1(k+1) | ...
    // (slot s's k-th tile: tile k of a pair item; tile 2k + s otherwise); slot 1's products
    // release the K/V stages of a pair item.  P_s lives in the columns of S_s: QK_s(k+1)
    // overwrites what PV_s(k) reads, and both come from this thread, whose tcgen05.mma
    // operations execute in issue order.  (Serving whichever slot's P is ready first, by
    // polling both barriers, measured slower.)
    if (lane == 0) {
      const uint32_t id_qk = tc::idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_pv = tc::idesc_bf16_f32(128, 128, false, true);
      const uint32_t aQ = tc::smem_u32(sQ), aK = tc::smem_u32(sK), aV = tc::smem_u32(sV);
      // base descriptors of the first Q buffer, K stage and V stage; buffer b's is kTile bytes
      // (kTile / 16 in the address field) further
      const uint64_t dQ0 = tc::smem_desc(aQ, 16, 1024), dK0 = tc::smem_desc(aK, 16, 1024);
      const uint64_t dV0 = tc::smem_desc(aV, kAtom, 1024);
      constexpr uint64_t kTileDesc = kTile >> 4;
      int g0 = 0, li = 0;            // ring index of the item's first tile; items
      int qn0 = 0, qn1 = 0;          // Q tiles consumed per buffer
      int pvn0 = 0, pvn1 = 0;        // PV products issued per slot
      bool ok = true;
      ItemIter iter;
      iter.start(a, R);
      Item it;
      for (; ok && iter.next(a, R, it); ++li) {
        const int nt = it.j1 - it.j0;
        const bool pair = it.pair;
        const int n0 = pair ? nt : (nt + 1) >> 1, n1 = pair ? nt : nt >> 1;
        const int nq = pair ? 2 : 1;
        ok = tc::mbar_wait(q_full, qn0 & 1, abort_flag, kWaitLimit);
        ++qn0;
        if (ok && pair) {
          ok = tc::mbar_wait(q_full + 1, qn1 & 1, abort_flag, kWaitLimit);
          ++qn1;
        }
        if (!ok) break;
        int qk_left = n0 + n1;
        // release: this product is the stage's last reader (a split tile has one reader)
        auto issue_qk = [&](int s, int k, bool release) -> bool {
          const int g = g0 + (pair ? k : 2 * k + s);
          const int kst = g % kKStages, kuse = g / kKStages;
          if (!tc::mbar_wait(k_full + kst, kuse & 1, abort_flag, kWaitLimit)) return false;
          tc::tc_fence_after();
          const uint32_t tS = tmem + 128 * s;
          // the tiles' base descriptors plus each K step's offset (in 16-byte units, inside the
          // 14-bit address field), all formed before the first product: the eight products
          // then go out back to back and the tensor pipe does not wait on this thread
          const uint64_t dq = dQ0 + (pair ? s : 0) * kTileDesc, dk = dK0 + uint64_t(kst) * kTileDesc;
          uint64_t da[8], db[8];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t off = uint64_t(((kk >> 2) * kAtom + (kk & 3) * 32) >> 4);
            da[kk] = dq + off;
            db[kk] = dk + off;
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) tc::mma_bf16_ss(tS, da[kk], db[kk], id_qk, kk > 0 ? 1u : 0u);
          tc::mma_commit(s_full + s);
          if (!pair || release) tc::mma_commit(k_empty + kst);
          if (--qk_left == 0)
            for (int b = 0; b < nq; ++b) tc::mma_commit(q_empty + b);
          return true;
        };
        auto issue_pv = [&](int s, int k, bool release) -> bool {
          const int g = g0 + (pair ? k : 2 * k + s);
          const int vst = g % kVStages, vuse = g / kVStages;
          int& pvn = s == 0 ? pvn0 : pvn1;
          if (!tc::mbar_wait(p_full + s, pvn & 1, abort_flag, kWaitLimit)) return false;
          if (!tc::mbar_wait(v_full + vst, vuse & 1, abort_flag, kWaitLimit)) return false;
          // the first product of an item overwrites O_s: the previous epilogue must have read it
          if (k == 0 && li > 0 && !tc::mbar_wait(o_free + s, (li - 1) & 1, abort_flag, kWaitLimit))
            return false;
          tc::tc_fence_after();
          const uint32_t tO = tmem + 256 + 128 * s, tP = tmem + 128 * s + 64;
          const uint64_t dv = dV0 + uint64_t(vst) * kTileDesc;
          const uint32_t acc0 = k > 0 ? 1u : 0u;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // P_s: 16 keys = 8 columns per MMA; V's rows of those keys 2048 bytes further per step
            tc::mma_bf16_ts(tO, tP + 8 * kk, dv + uint64_t(kk * (2048 >> 4)), id_pv,
                            kk > 0 ? 1u : acc0);
          }
          tc::mma_commit(pv_done + s);
          if (!pair || release) tc::mma_commit(v_empty + vst);
          ++pvn;
          return true;
        };
        if (n0 > 0) ok = issue_qk(0, 0, false);
        if (ok && n1 > 0) ok = issue_qk(1, 0, true);
        const int kmax = n0 > n1 ? n0 : n1;
        for (int k = 0; ok && k < kmax; ++k) {
          if (k < n0) {
            ok = issue_pv(0, k, false);
            if (ok && k + 1 < n0) ok = issue_qk(0, k + 1, false);
          }
          if (ok && k < n1) {
            ok = issue_pv(1, k, true);
            if (ok && k + 1 < n1) ok = issue_qk(1, k + 1, true);
          }
        }
        g0 += nt;
      }
      if (!ok) *abort_flag = 1;
      // drain every tcgen05 operation issued by this thread before TMEM is released (bounded,
      // and not cut short by the abort flag: TMEM must not be freed under a product)
      tc::mma_commit(drain);
      volatile int never = 0;
      tc::mbar_wait(drain, 0, &never, kWaitLimit / 8);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
  if (layout_ok) {
    // ===================================================================== softmax + epilogue
    // warps 4..7 serve slot 0, warps 8..11 slot 1; warp w reads TMEM lanes 32 (w & 3) ..
    // 32 (w & 3) + 31: one query row per thread, all 128 keys of a tile
    const int s = (warp - 4) >> 2, q4 = warp & 3;
    const int m = q4 * 32 + lane;
    const uint32_t lane_addr = uint32_t(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_addr + 128 * s;
    const int t_loc = m >> log2G, g = m & (G - 1);
    const float sl2 = a.scale_log2;
    float* xch = reinterpret_cast<float*>(base + kSmemX);   // [2 slots][reference, sum][128]
    int scnt = 0, ex_cnt = 0, g0 = 0, li = 0;
    int pv_mine = 0, pv_other = 0;   // PV products of this slot / the other slot so far
    bool ok = true;
    ItemIter iter;
    iter.start(a, R);
    Item it;
    for (; ok && iter.next(a, R, it); ++li) {
      const int nt = it.j1 - it.j0;
      const bool pair = it.pair;
      const int n0 = pair ? nt : (nt + 1) >> 1, n1 = pair ? nt : nt >> 1;
      const int ns = s == 0 ? n0 : n1;
      const int o = it.o, T = it.T, P = it.P;
      const int kv_len = P + T;
      const int t = (it.mt + (pair ? s : 0)) * tpt + t_loc;
      const bool valid = t < T;
      const uint32_t* arow = valid ? a.anc + size_t(o + t) * a.W : nullptr;
      float m_ref = -INFINITY, l = 0.f;
      // a warp whose 32 rows are all padding keeps only the barrier handshakes and the V
      // clearing: its P rows feed only its own O rows, which are never read
      const bool live = __any_sync(0xffffffffu, valid);
      for (int k = 0; k < ns; ++k) {
        const int ti = pair ? k : 2 * k + s;
        const int kbase = (it.j0 + ti) * kBN;
        if (!warp_wait(s_full + s, scnt & 1, abort_flag)) { ok = false; break; }
        ++scnt;
        tc::tc_fence_after();
        if (live) {
          // The maximum of the row's visible scores, then 128 independent exponentials
          // 2^(x sl2 - ref), one FMA each, written as bf16 P into the upper half of S_s's columns
          // (keys 32 c .. 32 c + 31 go to columns 64 + 16 c .. 64 + 16 c + 15).  At most 64
          // scores are held at once: keys 0..63 are read for the maximum, then keys 64..127,
          // whose exponentials go first (their P columns cover only their own scores), then keys
          // 0..63 again.  The reference is lazy: it moves only when the tile's maximum passes it
          // by more than 2^8, and then the row sum and O_s are rescaled.
          uint32_t x0[32], x1[32];
          tc::tmem_ld32(tS, x0);
          tc::tmem_ld32(tS + 32, x1);
          tc::tmem_ld_wait();
          const float max01 = fmaxf(mask_max32_row(x0, valid, kbase, P, arow, a.W),
                                    mask_max32_row(x1, valid, kbase + 32, P, arow, a.W));
          asm volatile("" ::"f"(max01));   // keys 0..63 are dead before 64..127 arrive
          tc::tmem_ld32(tS + 64, x0);
          tc::tmem_ld32(tS + 96, x1);
          tc::tmem_ld_wait();
          const float tmax = fmaxf(max01, fmaxf(mask_max32_row(x0, valid, kbase + 64, P, arow, a.W),
                                                mask_max32_row(x1, valid, kbase + 96, P, arow, a.W))) *
                             sl2;
          const bool up = tmax > m_ref + kLazyRescale;
          const float ref = up ? tmax : m_ref;
          const float factor = (up && m_ref != -INFINITY) ? ex2(m_ref - ref) : 1.f;
          // a row with no visible key yet (ref = -inf) computes 2^(x - inf) = 0 for every key
          // (masked keys hold -inf: -inf - inf = -inf, never -inf * 0)
          const float sl = ref == -INFINITY ? 1.f : sl2;
          const float add = ref == -INFINITY ? -INFINITY : -ref;
          const uint64_t sl2v = f2_pack(sl, sl), addv = f2_pack(add, add);
          uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = f2_pack(0.f, 0.f);
          exp_chunk(x1, sl2v, addv, acc1, tS + 64 + 48);
          exp_chunk(x0, sl2v, addv, acc0, tS + 64 + 32);
          tc::tmem_ld32(tS, x0);
          tc::tmem_ld32(tS + 32, x1);
          tc::tmem_ld_wait();
          mask_max32_row(x0, valid, kbase, P, arow, a.W);   // the masks again (max unused)
          mask_max32_row(x1, valid, kbase + 32, P, arow, a.W);
          exp_chunk(x1, sl2v, addv, acc1, tS + 64 + 16);
          exp_chunk(x0, sl2v, addv, acc0, tS + 64);
          // O_s carries the factor, after the exponentials (the scores are dead by then, which
          // keeps the register peak down); its previous product must have landed -- it has,
          // since S_s of this tile was computed after it -- and an item's first tile finds
          // nothing to rescale
          if (k > 0 && __any_sync(0xffffffffu, factor != 1.f)) {
            if (!warp_wait(pv_done + s, (pv_mine - 1) & 1, abort_flag)) { ok = false; break; }
            tc::tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
              uint32_t r32[32];
              const uint32_t ta = tmem + lane_addr + 256 + 128 * s + c0;
              tc::tmem_ld32(ta, r32);
              tc::tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 32; ++c)
                r32[c] = __float_as_uint(__uint_as_float(r32[c]) * factor);
              tc::tmem_st32(ta, r32);
            }
          }
          tc::tmem_st_wait();
          float ra, rb, rc, rd;
          f2_unpack(acc0, ra, rb);
          f2_unpack(acc1, rc, rd);
          l = l * factor + ((ra + rb) + (rc + rd));
          m_ref = ref;
        }
        // the request's last tile: zero the V rows past its KV length (stale cache rows times
        // P = 0 must not turn into NaN) before the tile's first product reads them; TMA must
        // have landed first.  Thread m clears key m in both 64-column atoms.
        if (kbase + kBN > kv_len && (!pair || s == 0)) {
          const int gv = g0 + ti;
          const int vst = gv % kVStages, vuse = gv / kVStages;
          if (!warp_wait(v_full + vst, vuse & 1, abort_flag)) { ok = false; break; }
          if (m >= kv_len - kbase) {
            uint8_t* vrow = sV + vst * kTile + (m >> 3) * 1024 + (m & 7) * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(vrow + kAtom + c * 16) = make_uint4(0, 0, 0, 0);
            }
          }
          tc::fence_proxy_async_smem();
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(p_full + s);
        ++pv_mine;
      }
      if (!ok) break;
      pv_other += s == 0 ? n1 : n0;   // the other slot's products of this item
      // epilogue: wait for the products whose O columns this warp reads (both slots' for a
      // split unit)
      if (ns > 0 && !warp_wait(pv_done + s, (pv_mine - 1) & 1, abort_flag)) { ok = false; break; }
      if (!pair && (s == 0 ? n1 : n0) > 0 &&
          !warp_wait(pv_done + (1 - s), (pv_other - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc::tc_fence_after();
      float lt, M, w0 = 0.f, w1 = 0.f;
      int c_lo, c_hi;     // output columns this warp writes
      if (pair) {
        lt = l;
        M = m_ref;
        c_lo = 0;
        c_hi = 128;
      } else {
        // merge the two slots' halves of the K/V range: exchange (reference, sum) with the
        // other slot's warp of this lane quarter; each slot then writes 64 output columns
        xch[(s * 2 + 0) * 128 + m] = m_ref;
        xch[(s * 2 + 1) * 128 + m] = l;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(ex_bar + q4);
        if (!warp_wait(ex_bar + q4, ex_cnt & 1, abort_flag)) { ok = false; break; }
        ++ex_cnt;
        const float m_o = xch[((1 - s) * 2 + 0) * 128 + m], l_o = xch[((1 - s) * 2 + 1) * 128 + m];
        const float m0 = s == 0 ? m_ref : m_o, l0 = s == 0 ? l : l_o;
        const float m1 = s == 0 ? m_o : m_ref, l1 = s == 0 ? l_o : l;
        M = fmaxf(m0, m1);
        w0 = (n0 > 0 && m0 != -INFINITY) ? ex2(m0 - M) : 0.f;
        w1 = (n1 > 0 && m1 != -INFINITY) ? ex2(m1 - M) : 0.f;
        lt = l0 * w0 + l1 * w1;
        c_lo = 64 * s;
        c_hi = c_lo + 64;
      }
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float lse2 = lt > 0.f ? M + __log2f(lt) : -INFINITY;
      if (live) {
        const int row = (pair ? s * kBM : 0) + m;   // row of a partial piece
        __nv_bfloat16* orow = a.o + (size_t(o + t) * a.H_q + it.h * G + g) * kD;
        float* prow = it.slot >= 0 ? a.part_o + (size_t(it.slot) * kPartRows + row) * kD : nullptr;
#pragma unroll 1
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
          uint32_t r32[32];
          float v[32];
          if (pair) {
            tc::tmem_ld32(tmem + lane_addr + 256 + 128 * s + c0, r32);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = __uint_as_float(r32[c]) * inv;
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) v[c] = 0.f;
            for (int u = 0; u < 2; ++u) {
              if ((u == 0 ? n0 : n1) == 0) continue;   // warp-uniform: that slot had no tiles
              tc::tmem_ld32(tmem + lane_addr + 256 + 128 * u + c0, r32);
              tc::tmem_ld_wait();
              const float wu = (u == 0 ? w0 : w1) * inv;
#pragma unroll
              for (int c = 0; c < 32; ++c) v[c] = fmaf(__uint_as_float(r32[c]), wu, v[c]);
            }
          }
          if (valid) {
            if (it.slot < 0) {
#pragma unroll
              for (int c = 0; c < 32; c += 8) {
                uint4 w4;
                w4.x = pack_bf16(v[c], v[c + 1]);
                w4.y = pack_bf16(v[c + 2], v[c + 3]);
                w4.z = pack_bf16(v[c + 4], v[c + 5]);
                w4.w = pack_bf16(v[c + 6], v[c + 7]);
                *reinterpret_cast<uint4*>(orow + c0 + c) = w4;
              }
            } else {
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(prow + c0 + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
            }
          }
        }
        if (valid && (pair || s == 0)) {
          if (it.slot < 0) {
            if (a.lse) a.lse[size_t(o + t) * a.H_q + it.h * G + g] = lse2 * 0.6931471805599453f;
          } else {
            a.part_lse[size_t(it.slot) * kPartRows + row] = lse2;
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(o_free + 0);
        tc::mbar_arrive(o_free + 1);
      }
      g0 += nt;
    }
    if (!ok) *abort_flag = 1;
  }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) {
    // every request of this CTA's range is unreliable after an expired wait
    ItemIter iter;
    iter.start(a, R);
    Item it;
    while (iter.next(a, R, it)) atomicOr(&a.req_status[it.r], SPEC_REQ_TIMEOUT);
  }
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------ one M-tile
// For launches in which every unit has one M-tile (at most 128 query rows: G x T <= 128), a
// kernel with one M-tile per CTA and its scores double-buffered, so that S = Q K^T of the next
// tile runs while the softmax works on this one: S buffers in TMEM columns 0-127 and 128-255,
// the O accumulator in 256-383, P (bf16) double-buffered in 384-447 and 448-511.  Warps: 0 Q/K
// producer, 2 V producer, 1 issues QK, 3 issues PV; warps 4..11 softmax, two per TMEM lane
// quarter, each exponentiating 64 of a tile's 128 keys against the full row's maximum (lazy
// reference, O rescaled when it grows by more than 2^8); the epilogue adds the two halves' row
// sums through a bounded exchange and each warp writes 64 output columns.
namespace attn1 {
using attn::kD;
using attn::kBS;
using attn::kBM;
using attn::kBN;
using attn::kAtom;
using attn::kTile;
using attn::kWaitLimit;
using attn::kLazyRescale;
using attn::kPartRows;
constexpr int kThreads = 384;                 // 4 control warps + 8 softmax warps
constexpr int kKStages = 4;
constexpr int kVStages = 2;
constexpr int kSmemQ = 0;
constexpr int kSmemK = kSmemQ + kTile;
constexpr int kSmemV = kSmemK + kKStages * kTile;
constexpr int kSmemBar = kSmemV + kVStages * kTile;
constexpr int kSmemRed = kSmemBar + 256;      // [2 buffers][2 halves][128 rows] fp32 exchange
constexpr int kSmemEnd = kSmemRed + 2048;
constexpr int kSmemBytes = 232448;            // the per-CTA maximum; the slack aligns the base
constexpr uint32_t kTmemP = 384;
}  // namespace attn1

__global__ void __launch_bounds__(attn1::kThreads, 1)
attn_tc_single_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mK8,
               const __grid_constant__ CUtensorMap mV8, TcDev a) {
  using namespace attn1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = base + kSmemQ;
  uint8_t* sK = base + kSmemK;
  uint8_t* sV = base + kSmemV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kSmemBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;                    // [kKStages]
  uint64_t* k_empty = k_full + kKStages;          // [kKStages]
  uint64_t* v_full = k_empty + kKStages;          // [kVStages]
  uint64_t* v_empty = v_full + kVStages;          // [kVStages]
  uint64_t* s_full = v_empty + kVStages;          // [2]
  uint64_t* s_free = s_full + 2;                  // [2]
  uint64_t* p_full = s_free + 2;                  // [2]: P buffer b written (8 softmax warps)
  uint64_t* pv_done = p_full + 2;                 // [2]: the PV that read P buffer b completed
  uint64_t* o_free = pv_done + 2;
  uint64_t* drain = o_free + 1;                   // [2]: the QK issuer's, the PV issuer's
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
  int* s_abort = reinterpret_cast<int*>(drain + 3);
  uint64_t* ex_bar = drain + 4;                   // [4]: row-sum exchange of the softmax halves
  static_assert(2 + 2 * kKStages + 2 * kVStages + 2 + 2 + 2 + 2 + 1 + 2 + 2 + 4 <= 32,
                "barriers fit their 256-byte region");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  // this CTA's range of the tile stream (the row-sum exchange area is free until the first
  // epilogue)
  const Range R = cta_range<kThreads>(a, reinterpret_cast<long long*>(base + kSmemRed),
                                      reinterpret_cast<int*>(base + kSmemRed + 256));
  if (tid == 0) write_merge_record(a, R);
  if (R.t0 >= R.t1) return;   // uniform across the CTA: no work, nothing allocated yet
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
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(p_full + b, 8);
      tc::mbar_init(pv_done + b, 1);
    }
    tc::mbar_init(o_free, 8);
    tc::mbar_init(drain, 1);
    tc::mbar_init(drain + 1, 1);
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
  volatile int* abort_flag = s_abort;
  const int G = a.G, log2G = a.log2G, tpt = kBM >> log2G;
  const bool layout_ok = *abort_flag == 0;

  if (layout_ok && (warp == 0 || warp == 2)) {
    // ===================================================================== TMA producers
    // warp 0 loads Q and K, warp 2 loads V
    const bool is_k = warp == 0;
    if (lane == 0) {
      tc::prefetch_tensormap(is_k ? &mK : &mV);
      tc::prefetch_tensormap(is_k ? &mK8 : &mV8);
      if (is_k) tc::prefetch_tensormap(&mQ);
    }
    // on an expired wait the producer raises the abort flag itself
    // Q: the unit's 128 rows (G heads x 128 / G tree tokens)
    const CUtensorMap* map = is_k ? &mK : &mV;
    const CUtensorMap* map8 = is_k ? &mK8 : &mV8;
    tma_producer(a, R, is_k, map, map8, is_k ? kKStages : kVStages, is_k ? sK : sV,
                 is_k ? k_full : v_full, is_k ? k_empty : v_empty, &mQ, sQ, kAtom, kTile, tpt,
                 q_full, q_empty, abort_flag);
  } else if (layout_ok && (warp == 1 || warp == 3)) {
    // ===================================================================== MMA issuers
    // warp 1 issues S = Q K^T, warp 3 issues O += P V, each tile after tile; each thread commits
    // its own operations, so a QK is never queued behind the wait for the previous P
    if (lane == 0) {
      const bool is_qk = warp == 1;
      const uint32_t id_qk = tc::idesc_bf16_f32(128, 128, false, false);
      const uint32_t id_pv = tc::idesc_bf16_f32(128, 128, false, true);
      // base descriptors (buffer b's is kTile bytes, kTile / 16 in the address field, further)
      const uint64_t dQ0 = tc::smem_desc(tc::smem_u32(sQ), 16, 1024);
      const uint64_t dK0 = tc::smem_desc(tc::smem_u32(sK), 16, 1024);
      const uint64_t dV0 = tc::smem_desc(tc::smem_u32(sV), kAtom, 1024);
      constexpr uint64_t kTileDesc = kTile >> 4;
      const uint32_t tO = tmem + 256;
      int kv_it = 0, li = 0;
      bool ok = true;
      ItemIter iter;
      iter.start(a, R);
      Item it;
      for (; ok && iter.next(a, R, it); ++li) {
        if (is_qk && !tc::mbar_wait(q_full, li & 1, abort_flag, kWaitLimit)) { ok = false; break; }
        for (int j = it.j0; j < it.j1; ++j, ++kv_it) {
          const int st = kv_it & 1, use = kv_it >> 1;
          if (is_qk) {
            const int kst = kv_it % kKStages, kuse = kv_it / kKStages;
            if (!tc::mbar_wait(k_full + kst, kuse & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            if (use > 0 && !tc::mbar_wait(s_free + st, (use - 1) & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            tc::tc_fence_after();
            const uint32_t tS = tmem + st * 128;
            // all eight products' descriptors first (base + the K step's offset): the products
            // then go out back to back
            const uint64_t dk = dK0 + uint64_t(kst) * kTileDesc;
            uint64_t da[8], db[8];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t off = uint64_t(((kk >> 2) * kAtom + (kk & 3) * 32) >> 4);
              da[kk] = dQ0 + off;
              db[kk] = dk + off;
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16_ss(tS, da[kk], db[kk], id_qk, kk > 0 ? 1u : 0u);
            tc::mma_commit(s_full + st);
            tc::mma_commit(k_empty + kst);
            if (j == it.j1 - 1) tc::mma_commit(q_empty);
          } else {
            const int pst = kv_it % kVStages, puse = kv_it / kVStages;
            const bool first_pv = j == it.j0;
            if (!tc::mbar_wait(p_full + st, use & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            if (!tc::mbar_wait(v_full + pst, puse & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            if (first_pv && li > 0 && !tc::mbar_wait(o_free, (li - 1) & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            tc::tc_fence_after();
            const uint64_t dv = dV0 + uint64_t(pst) * kTileDesc;
            const uint32_t acc0 = first_pv ? 0u : 1u;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // P buffer st in TMEM columns 384 + 64 st: 16 keys = 8 columns per MMA
              const uint32_t ta = tmem + kTmemP + 64 * st + 8 * kk;
              tc::mma_bf16_ts(tO, ta, dv + uint64_t(kk * (2048 >> 4)), id_pv, kk > 0 ? 1u : acc0);
            }
            tc::mma_commit(v_empty + pst);
            tc::mma_commit(pv_done + st);
          }
        }
      }
      if (!ok) *abort_flag = 1;
      // drain every tcgen05 operation issued by this thread before TMEM is released
      // (bounded, and not cut short by the abort flag: TMEM must not be freed under a product)
      uint64_t* my_drain = drain + (is_qk ? 0 : 1);
      tc::mma_commit(my_drain);
      volatile int never = 0;
      tc::mbar_wait(my_drain, 0, &never, kWaitLimit / 8);
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
    ItemIter iter;
    iter.start(a, R);
    Item it;
    for (; ok && iter.next(a, R, it); ++li) {
      const int o = it.o, T = it.T, P = it.P;
      const int kv_len = P + T;
      const int t = it.mt * tpt + t_loc;
      const bool valid = t < T;
      const uint32_t* arow = valid ? a.anc + size_t(o + t) * a.W : nullptr;
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
        // P buffer st was last read by the PV of tile kv_it - 2: it must be complete before the
        // buffer is rewritten and before this tile's P is declared ready (all warps, live or
        // not, so that no warp gets two tiles ahead on p_full)
        auto wait_p_buffer = [&]() -> bool {
          return kv_it < 2 || warp_wait(pv_done + st, (use - 1) & 1, abort_flag);
        };
        if (!live) {
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(s_free + st);
          if (!wait_p_buffer()) { ok = false; break; }
        } else {
        // the partner half's 64 scores: only their max is needed
        float tmax;
        {
          uint32_t x0[32], x1[32];
          tc::tmem_ld32(srow + 64 * (1 - hh), x0);
          tc::tmem_ld32(srow + 64 * (1 - hh) + 32, x1);
          tc::tmem_ld_wait();
          tmax = fmaxf(mask_max32_row(x0, valid, kbase + 64 * (1 - hh), P, arow, a.W),
                       mask_max32_row(x1, valid, kbase + 64 * (1 - hh) + 32, P, arow, a.W));
        }
        // this half's 64 scores, kept for the exponentials; the S buffer is free afterwards
        uint32_t s0[32], s1[32];
        tc::tmem_ld32(srow + 64 * hh, s0);
        tc::tmem_ld32(srow + 64 * hh + 32, s1);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_free + st);
        tmax = fmaxf(tmax, mask_max32_row(s0, valid, kbase + 64 * hh, P, arow, a.W));
        tmax = fmaxf(tmax, mask_max32_row(s1, valid, kbase + 64 * hh + 32, P, arow, a.W));
        tmax *= sl2;   // raw maximum -> log2 units (sl2 > 0; -inf stays -inf)
        const bool grow = tmax > m_ref + kLazyRescale;
        const float new_ref = grow ? tmax : m_ref;
        const float factor = (grow && m_ref != -INFINITY) ? ex2(m_ref - new_ref) : 1.f;
        const bool has_ref = new_ref != -INFINITY;
        // exponentials (kept packed in registers) before waiting for the previous PV
        uint32_t pk[32];
        float rowsum = 0.f;
#pragma unroll
        for (int c = 0; c < 32; c += 2) {   // 2^(x sl2 - ref): one FMA per score
          const float p0 = has_ref ? ex2(fmaf(__uint_as_float(s0[c]), sl2, -new_ref)) : 0.f;
          const float p1 = has_ref ? ex2(fmaf(__uint_as_float(s0[c + 1]), sl2, -new_ref)) : 0.f;
          rowsum += p0 + p1;
          pk[c >> 1] = pack_bf16(p0, p1);
        }
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = has_ref ? ex2(fmaf(__uint_as_float(s1[c]), sl2, -new_ref)) : 0.f;
          const float p1 = has_ref ? ex2(fmaf(__uint_as_float(s1[c + 1]), sl2, -new_ref)) : 0.f;
          rowsum += p0 + p1;
          pk[16 + (c >> 1)] = pack_bf16(p0, p1);
        }
        // P of this tile into TMEM buffer st: this warp's rows, keys 64 hh .. 64 hh + 63
        if (!wait_p_buffer()) { ok = false; break; }
        tc::tc_fence_after();
        tc::tmem_st32(tmem + lane_addr + kTmemP + 64 * st + 32 * hh, pk);
        // lazy rescale of this warp's half of the O accumulator (warp-collective TMEM access):
        // the previous tile's PV must have landed in O first
        const bool any_rescale = __any_sync(0xffffffffu, factor != 1.f) && j > it.j0;
        if (any_rescale) {
          const int pv = kv_it - 1;
          if (!warp_wait(pv_done + (pv & 1), (pv >> 1) & 1, abort_flag)) { ok = false; break; }
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
        }
        tc::tmem_st_wait();
        l = l * factor + rowsum;
        m_ref = new_ref;
        }  // live
        // last tile: zero V rows past the request's KV length (stale cache rows times P = 0
        // must not turn into NaN); TMA must have landed first.  Half hh clears d-atom hh.
        if (kbase + kBN > kv_len) {
          const int vst = kv_it % kVStages, vuse = kv_it / kVStages;
          if (!warp_wait(v_full + vst, vuse & 1, abort_flag)) { ok = false; break; }
          const int key = m;
          if (key >= kv_len - kbase) {
            uint8_t* vrow = sV + vst * kTile + hh * kAtom + (key >> 3) * 1024 + (key & 7) * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
          }
          tc::fence_proxy_async_smem();
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(p_full + st);
      }
      if (!ok) break;
      // epilogue: this warp writes output columns 64*hh .. 64*hh+63 of its rows
      if (!warp_wait(pv_done + ((kv_it - 1) & 1), ((kv_it - 1) >> 1) & 1, abort_flag)) { ok = false; break; }
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
        float* prow = a.part_o + (size_t(it.slot) * kPartRows + m) * kD + 64 * hh;
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
        if (valid && hh == 0) a.part_lse[size_t(it.slot) * kPartRows + m] = lse2;
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
    ItemIter iter;
    iter.start(a, R);
    Item it;
    while (iter.next(a, R, it)) atomicOr(&a.req_status[it.r], SPEC_REQ_TIMEOUT);
  }
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------ small units
// For units of at most 16 query rows (T x G <= 16: plain decode and short chains) the scores are
// computed transposed, S^T = K Q^T (M = 128 keys on the TMEM lanes, N = 16 query rows), so the
// softmax spends its lanes on keys instead of on padding rows: 16 exponentials per lane and tile,
// spread over the four TMEM lane quarters (one softmax warp each), where the row-major kernel
// runs 64 per lane on the one sub-partition that owns the live rows.  O^T += V^T P^T (V as an
// M-major A operand, P^T a 4 KB K-major B tile in shared memory) accumulates in TMEM.  The lazy
// rescale reference of each row is shared by the four warps through a bounded exchange per tile;
// row sums stay per lane until the epilogue.  Q is a 16-row (4 KB) box.
namespace attn_s {
constexpr int kRows = 16;                        // N of both MMAs
constexpr int kThreads = 256;                    // 4 control warps + 4 softmax warps
constexpr int kQAtom = kRows * 128;              // 16 rows x 128 B
constexpr int kQBytes = 2 * kQAtom;              // Q: 16 rows x 128 d (bf16)
constexpr int kPTile = 2 * kQAtom;               // P^T: 16 rows x 128 keys (bf16)
constexpr int kKStages = 3;
constexpr int kVStages = 3;
constexpr int kSmemQ = 0;
constexpr int kSmemP = kSmemQ + kQBytes;                       // 2 P^T buffers
constexpr int kSmemK = kSmemP + 2 * kPTile;                    // 1024-aligned
constexpr int kSmemV = kSmemK + kKStages * attn::kTile;
constexpr int kSmemBar = kSmemV + kVStages * attn::kTile;
constexpr int kSmemX = kSmemBar + 512;                         // exchanges between softmax warps
constexpr int kSmemEnd = kSmemX + 1280;
constexpr int kSmemBytes = kSmemEnd + 1024;                    // slack for 1024-byte alignment
constexpr uint32_t kTmemCols = 64;                             // S^T 0-15, 16-31; O^T 32-47
constexpr uint32_t kTmemO = 32;
static_assert(kSmemK % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
static_assert(kSmemBytes <= 232448, "fits one CTA's shared memory");

struct Xchg {
  int flag[2][4];          // per tile (parity): some key of warp q passed its row's reference
  float mx[2][4][kRows];   // per update (parity): warp q's row maxima
  float sum[2][4][kRows];  // per item (parity): warp q's row sums
};
static_assert(sizeof(Xchg) <= 1280, "exchange area");
}  // namespace attn_s

__global__ void __launch_bounds__(attn_s::kThreads, 1)
attn_tc_small_kernel(const __grid_constant__ CUtensorMap mQs, const __grid_constant__ CUtensorMap mK,
                     const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mK8,
                     const __grid_constant__ CUtensorMap mV8, TcDev a) {
  using namespace attn_s;
  using attn::kAtom;
  using attn::kBM;
  using attn::kBN;
  using attn::kD;
  using attn::kLazyRescale;
  using attn::kTile;
  using attn::kWaitLimit;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = base + kSmemQ;
  uint8_t* sPT = base + kSmemP;
  uint8_t* sK = base + kSmemK;
  uint8_t* sV = base + kSmemV;
  Xchg* xs = reinterpret_cast<Xchg*>(base + kSmemX);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kSmemBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;                    // [kKStages]
  uint64_t* k_empty = k_full + kKStages;          // [kKStages]
  uint64_t* v_full = k_empty + kKStages;          // [kVStages]
  uint64_t* v_empty = v_full + kVStages;          // [kVStages]
  uint64_t* s_full = v_empty + kVStages;          // [2]
  uint64_t* s_free = s_full + 2;                  // [2]
  uint64_t* p_full = s_free + 2;                  // [2]
  uint64_t* pv_done = p_full + 2;                 // [2]
  uint64_t* o_free = pv_done + 2;
  uint64_t* drain = o_free + 1;                   // [2]: the QK issuer's, the PV issuer's
  uint64_t* xa_bar = drain + 2;                   // [2] flag exchange
  uint64_t* xb_bar = xa_bar + 2;                  // [2] maxima exchange
  uint64_t* xc_bar = xb_bar + 2;                  // [2] row-sum exchange
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xc_bar + 2);
  int* s_abort = reinterpret_cast<int*>(xc_bar + 3);
  static_assert(2 + 2 * kKStages + 2 * kVStages + 2 + 2 + 2 + 2 + 3 + 6 + 2 <= 64,
                "barriers fit their 512-byte region");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_wait();
  pdl_trigger();
  const Range R = cta_range<kThreads>(a, reinterpret_cast<long long*>(base + kSmemX),
                                      reinterpret_cast<int*>(base + kSmemX + 256));
  if (tid == 0) write_merge_record(a, R);
  if (R.t0 >= R.t1) return;   // uniform across the CTA: no work, nothing allocated yet
  __syncthreads();            // the exchange area was scratch for the range computation
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
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(s_full + b, 1);
      tc::mbar_init(s_free + b, 4);
      tc::mbar_init(p_full + b, 4);
      tc::mbar_init(pv_done + b, 1);
      tc::mbar_init(xa_bar + b, 4);
      tc::mbar_init(xb_bar + b, 4);
      tc::mbar_init(xc_bar + b, 4);
    }
    tc::mbar_init(o_free, 4);
    tc::mbar_init(drain, 1);
    tc::mbar_init(drain + 1, 1);
    *s_abort = (tc::smem_u32(base) + kSmemEnd > tc::smem_u32(smem_raw) + kSmemBytes) ? 1 : 0;
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  volatile int* abort_flag = s_abort;
  const int G = a.G, log2G = a.log2G;
  const bool layout_ok = *abort_flag == 0;

  if (layout_ok && (warp == 0 || warp == 2)) {
    // ===================================================================== TMA producers
    const bool is_k = warp == 0;
    if (lane == 0) {
      tc::prefetch_tensormap(is_k ? &mK : &mV);
      tc::prefetch_tensormap(is_k ? &mK8 : &mV8);
      if (is_k) tc::prefetch_tensormap(&mQs);
    }
    // Q: the unit's rows (G heads x 16 / G tree tokens; one M-tile per unit)
    const CUtensorMap* map = is_k ? &mK : &mV;
    const CUtensorMap* map8 = is_k ? &mK8 : &mV8;
    tma_producer(a, R, is_k, map, map8, is_k ? kKStages : kVStages, is_k ? sK : sV,
                 is_k ? k_full : v_full, is_k ? k_empty : v_empty, &mQs, sQ, kQAtom, kQBytes,
                 kRows / G, q_full, q_empty, abort_flag);
  } else if (layout_ok && (warp == 1 || warp == 3)) {
    // ===================================================================== MMA issuers
    // warp 1 issues S^T = K Q^T, warp 3 issues O^T += V^T P^T, each tile after tile; each thread
    // commits its own operations, so a QK is never queued behind the wait for the previous P
    if (lane == 0) {
      const bool is_qk = warp == 1;
      const uint32_t id_qk = tc::idesc_bf16_f32(128, kRows, false, false);
      const uint32_t id_pv = tc::idesc_bf16_f32(128, kRows, true, false);
      // base descriptors (stage / buffer b's is its size / 16 further in the address field)
      const uint64_t dQ0 = tc::smem_desc(tc::smem_u32(sQ), 16, 1024);
      const uint64_t dK0 = tc::smem_desc(tc::smem_u32(sK), 16, 1024);
      const uint64_t dV0 = tc::smem_desc(tc::smem_u32(sV), kAtom, 1024);
      const uint64_t dP0 = tc::smem_desc(tc::smem_u32(sPT), 16, 1024);
      const uint32_t tO = tmem + kTmemO;
      int kv_it = 0, li = 0;
      bool ok = true;
      ItemIter iter;
      iter.start(a, R);
      Item it;
      for (; ok && iter.next(a, R, it); ++li) {
        if (is_qk && !tc::mbar_wait(q_full, li & 1, abort_flag, kWaitLimit)) { ok = false; break; }
        for (int j = it.j0; j < it.j1; ++j, ++kv_it) {
          const int st = kv_it & 1, use = kv_it >> 1;
          if (is_qk) {
            const int kst = kv_it % kKStages, kuse = kv_it / kKStages;
            if (!tc::mbar_wait(k_full + kst, kuse & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            if (use > 0 && !tc::mbar_wait(s_free + st, (use - 1) & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            tc::tc_fence_after();
            const uint32_t tS = tmem + st * kRows;
            // A = K (128 keys x 16 d per step, K-major), B = Q (16 rows x 16 d, K-major); all
            // descriptors first, then the eight products back to back
            const uint64_t dk = dK0 + uint64_t(kst) * uint64_t(kTile >> 4);
            uint64_t da[8], db[8];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              da[kk] = dk + uint64_t(((kk >> 2) * kAtom + (kk & 3) * 32) >> 4);
              db[kk] = dQ0 + uint64_t(((kk >> 2) * kQAtom + (kk & 3) * 32) >> 4);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16_ss(tS, da[kk], db[kk], id_qk, kk > 0 ? 1u : 0u);
            tc::mma_commit(s_full + st);
            tc::mma_commit(k_empty + kst);
            if (j == it.j1 - 1) tc::mma_commit(q_empty);
          } else {
            const int pst = kv_it % kVStages, puse = kv_it / kVStages;
            const bool first_pv = j == it.j0;
            if (!tc::mbar_wait(p_full + st, use & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            if (!tc::mbar_wait(v_full + pst, puse & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            if (first_pv && li > 0 && !tc::mbar_wait(o_free, (li - 1) & 1, abort_flag, kWaitLimit)) { ok = false; break; }
            tc::tc_fence_after();
            // A = V^T (M = d, M-major), B = P^T (16 rows x 16 keys per step, K-major)
            const uint64_t dv = dV0 + uint64_t(pst) * uint64_t(kTile >> 4);
            const uint64_t dp = dP0 + uint64_t(st) * uint64_t(kPTile >> 4);
            const uint32_t acc0 = first_pv ? 0u : 1u;
            uint64_t da[8], db[8];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              da[kk] = dv + uint64_t(kk * (2048 >> 4));
              db[kk] = dp + uint64_t(((kk >> 2) * kQAtom + (kk & 3) * 32) >> 4);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) tc::mma_bf16_ss(tO, da[kk], db[kk], id_pv, kk > 0 ? 1u : acc0);
            tc::mma_commit(v_empty + pst);
            tc::mma_commit(pv_done + st);
          }
        }
      }
      if (!ok) *abort_flag = 1;
      // drain every tcgen05 operation issued by this thread before TMEM is released
      // (bounded, and not cut short by the abort flag: TMEM must not be freed under a product)
      uint64_t* my_drain = drain + (is_qk ? 0 : 1);
      tc::mma_commit(my_drain);
      volatile int never = 0;
      tc::mbar_wait(my_drain, 0, &never, kWaitLimit / 8);
    }
  } else if (layout_ok && warp >= 4) {
    // ===================================================================== softmax + epilogue
    const int q = warp & 3;                       // TMEM lane quarter: keys (S^T) / d (O^T)
    const uint32_t lane_addr = uint32_t(q * 32) << 16;
    const int kl = q * 32 + lane;                 // this lane's key within a tile; its d in O^T
    const float sl2 = a.scale_log2;
    int kv_it = 0, li = 0, xa = 0, xb = 0, xc = 0;
    bool ok = true;
    // bounded exchange among the four softmax warps: one phase of bar[n & 1] per use
    auto xwait = [&](uint64_t* bar, int n) -> bool {
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar + (n & 1));
      return warp_wait(bar + (n & 1), (n >> 1) & 1, abort_flag);
    };
    ItemIter iter;
    iter.start(a, R);
    Item it;
    for (; ok && iter.next(a, R, it); ++li) {
      const int o = it.o, T = it.T, P = it.P;
      const int kv_len = P + T;
      const int nrows = min(T << log2G, kRows);   // valid rows: n < nrows
      float ref[kRows], lsum[kRows];
#pragma unroll
      for (int n = 0; n < kRows; ++n) { ref[n] = -INFINITY; lsum[n] = 0.f; }
      for (int j = it.j0; j < it.j1; ++j, ++kv_it) {
        const int st = kv_it & 1, use = kv_it >> 1;
        if (!warp_wait(s_full + st, use & 1, abort_flag)) { ok = false; break; }
        tc::tc_fence_after();
        uint32_t sv[kRows];
        tc::tmem_ld16(tmem + lane_addr + st * kRows, sv);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_free + st);
        // visibility of this lane's key for each row: the prefix is visible to every valid row;
        // a tree slot a = key - P only to the rows whose token has a as ancestor-or-self
        const int key = j * kBN + kl;
        uint32_t vis = 0;
        if (key < P) {
          vis = (nrows >= 32) ? 0xFFFFFFFFu : ((1u << nrows) - 1u);
        } else if (key < kv_len) {
          const int slot = key - P;
#pragma unroll
          for (int n = 0; n < kRows; ++n) {
            if (n < nrows) {
              const uint32_t w0 = a.anc[size_t(o + (n >> log2G)) * a.W + (slot >> 5)];
              vis |= ((w0 >> (slot & 31)) & 1u) << n;
            }
          }
        }
        float x[kRows];
        bool above = false;
#pragma unroll
        for (int n = 0; n < kRows; ++n) {
          x[n] = ((vis >> n) & 1u) ? __uint_as_float(sv[n]) * sl2 : -INFINITY;
          above = above || (x[n] > ref[n] + kLazyRescale);
        }
        // some key of some warp passed its row's reference: all four warps move the references
        const int flag = __any_sync(0xffffffffu, above) ? 1 : 0;
        if (lane == 0) xs->flag[xa & 1][q] = flag;
        if (!xwait(xa_bar, xa)) { ok = false; break; }
        const bool update = (xs->flag[xa & 1][0] | xs->flag[xa & 1][1] | xs->flag[xa & 1][2] |
                             xs->flag[xa & 1][3]) != 0;
        ++xa;
        if (update) {
          float mx[kRows];
#pragma unroll
          for (int n = 0; n < kRows; ++n) mx[n] = warp_max(x[n]);
          if (lane == 0) {
#pragma unroll
            for (int n = 0; n < kRows; ++n) xs->mx[xb & 1][q][n] = mx[n];
          }
          if (!xwait(xb_bar, xb)) { ok = false; break; }
          float factor[kRows];
          bool any_factor = false;
#pragma unroll
          for (int n = 0; n < kRows; ++n) {
            float nr = ref[n];
#pragma unroll
            for (int w = 0; w < 4; ++w) nr = fmaxf(nr, xs->mx[xb & 1][w][n]);
            factor[n] = (ref[n] == -INFINITY || nr == ref[n]) ? 1.f : ex2(ref[n] - nr);
            any_factor = any_factor || factor[n] != 1.f;
            ref[n] = nr;
          }
          ++xb;
          // rescale the accumulated O^T rows (this warp's d quarter) once the previous PV landed
          if (any_factor && j > it.j0) {
            const int pv = kv_it - 1;
            if (!warp_wait(pv_done + (pv & 1), (pv >> 1) & 1, abort_flag)) { ok = false; break; }
            tc::tc_fence_after();
            uint32_t ov[kRows];
            tc::tmem_ld16(tmem + lane_addr + kTmemO, ov);
            tc::tmem_ld_wait();
#pragma unroll
            for (int n = 0; n < kRows; ++n) ov[n] = __float_as_uint(__uint_as_float(ov[n]) * factor[n]);
            tc::tmem_st16(tmem + lane_addr + kTmemO, ov);
            tc::tmem_st_wait();
          }
#pragma unroll
          for (int n = 0; n < kRows; ++n) lsum[n] *= factor[n];
        }
        // P^T of this key into buffer st, once the PV that last read it (tile kv_it - 2) is done
        if (kv_it >= 2 && !warp_wait(pv_done + st, (use - 1) & 1, abort_flag)) { ok = false; break; }
        uint8_t* pcol = sPT + st * kPTile + (kl >> 6) * kQAtom;
        const int chunk = (kl & 63) >> 3, within = (kl & 7) * 2;
#pragma unroll
        for (int n = 0; n < kRows; ++n) {
          const float p = (x[n] == -INFINITY) ? 0.f : ex2(x[n] - ref[n]);
          lsum[n] += p;
          const __nv_bfloat16 pb = __float2bfloat16_rn(p);
          *reinterpret_cast<__nv_bfloat16*>(pcol + (n >> 3) * 1024 + (n & 7) * 128 +
                                            ((chunk ^ (n & 7)) << 4) + within) = pb;
        }
        // last tile: zero the V rows of keys past the KV length (stale rows times P = 0 must not
        // turn into NaN); the V copy must have landed first
        if (j * kBN + kBN > kv_len) {
          const int vst = kv_it % kVStages, vuse = kv_it / kVStages;
          if (!warp_wait(v_full + vst, vuse & 1, abort_flag)) { ok = false; break; }
          if (key >= kv_len) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint8_t* vrow = sV + vst * kTile + hh * kAtom + (kl >> 3) * 1024 + (kl & 7) * 128;
#pragma unroll
              for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
            }
          }
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(p_full + st);
      }
      if (!ok) break;
      // epilogue: row sums over lanes and warps, then this warp's d quarter of every valid row
      if (!warp_wait(pv_done + ((kv_it - 1) & 1), ((kv_it - 1) >> 1) & 1, abort_flag)) { ok = false; break; }
      tc::tc_fence_after();
      float tot[kRows];
#pragma unroll
      for (int n = 0; n < kRows; ++n) {
        float v = lsum[n];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        tot[n] = v;
      }
      if (lane == 0) {
#pragma unroll
        for (int n = 0; n < kRows; ++n) xs->sum[xc & 1][q][n] = tot[n];
      }
      if (!xwait(xc_bar, xc)) { ok = false; break; }
#pragma unroll
      for (int n = 0; n < kRows; ++n)
        tot[n] = ((xs->sum[xc & 1][0][n] + xs->sum[xc & 1][1][n]) + xs->sum[xc & 1][2][n]) + xs->sum[xc & 1][3][n];
      ++xc;
      uint32_t ov[kRows];
      tc::tmem_ld16(tmem + lane_addr + kTmemO, ov);
      tc::tmem_ld_wait();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(o_free);
#pragma unroll
      for (int n = 0; n < kRows; ++n) {
        if (n < nrows) {
          const float lt = tot[n];
          const float inv = lt > 0.f ? 1.f / lt : 0.f;
          const float lse2 = lt > 0.f ? ref[n] + __log2f(lt) : -INFINITY;
          const int t = n >> log2G, g = n & (G - 1);
          const float val = __uint_as_float(ov[n]) * inv;
          if (it.slot < 0) {
            a.o[(size_t(o + t) * a.H_q + it.h * G + g) * kD + kl] = __float2bfloat16_rn(val);
            if (q == 0 && lane == 0 && a.lse)
              a.lse[size_t(o + t) * a.H_q + it.h * G + g] = lse2 * 0.6931471805599453f;
          } else {
            a.part_o[(size_t(it.slot) * attn::kPartRows + n) * kD + kl] = val;
            if (q == 0 && lane == 0) a.part_lse[size_t(it.slot) * attn::kPartRows + n] = lse2;
          }
        }
      }
    }
    if (!ok) *abort_flag = 1;
  }
  tc::tc_fence_before();
  __syncthreads();
  if (*abort_flag && tid == 0) {
    // every request of this CTA's range is unreliable after an expired wait
    ItemIter iter;
    iter.start(a, R);
    Item it;
    while (iter.next(a, R, it)) atomicOr(&a.req_status[it.r], SPEC_REQ_TIMEOUT);
  }
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------ merge
// CTA (c, y, z) merges rows 32 z .. 32 z + 31 of M-tile mt + y of the cut unit of record c by
// log-sum-exp of its pieces, in range order, into O and lse.  Warp w takes rows w, w + 8, w + 16
// and w + 24 of those and lane l columns 4l .. 4l + 3, so that every load of a partial row is
// one 512-byte line and all of a thread's loads are in flight together (the merge is bound by
// the latency of reading the pieces back).  A unit has at most kMergeFast pieces in the common
// case: their log-sum-exps and values are loaded in one batch; longer units take the general
// loop.
constexpr int kMergeFast = 2;
constexpr int kMergeBatch = 4;
constexpr int kMergeSplit = attn::kBM / (8 * kMergeBatch);   // CTAs per M-tile

__global__ void __launch_bounds__(256) attn_merge_kernel(TcDev a) {
  using namespace attn;
  pdl_wait();
  pdl_trigger();
  const MergeRec rec = a.recs[blockIdx.x];
  const int y = blockIdx.y;
  if (rec.np < 2 || y >= rec.nmt) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tpt = kBM >> a.log2G;
  const int np = rec.np;
  auto slot_of = [&](int p) { return p == 0 ? rec.slot0 : 2 * (rec.ca + p); };
  auto lse_of = [&](int p, int row) { return a.part_lse[size_t(slot_of(p)) * kPartRows + row]; };
  auto part_of = [&](int p, int row) {
    return reinterpret_cast<const float4*>(a.part_o + (size_t(slot_of(p)) * kPartRows + row) * kD)[lane];
  };
  // row m of the M-tile: its output row (token t, head g) and its row in the pieces
  auto out_row = [&](int m, int& t, int& g) {
    t = (rec.mt + y) * tpt + (m >> a.log2G);
    g = m & (a.G - 1);
  };
  auto store = [&](int t, int g, const float (&acc)[4], float wsum, float M) {
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const size_t orow = size_t(rec.o + t) * a.H_q + rec.h * a.G + g;
    uint2 o2;
    o2.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    o2.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(a.o + orow * kD + 4 * lane) = o2;
    if (lane == 0 && a.lse) a.lse[orow] = (M + __log2f(wsum)) * 0.6931471805599453f;
  };
  for (int i0 = int(blockIdx.z) * kMergeBatch; i0 < int(blockIdx.z + 1) * kMergeBatch; i0 += kMergeBatch) {
    if (np <= kMergeFast) {
      float ls[kMergeBatch][kMergeFast];
      float4 v[kMergeBatch][kMergeFast];
#pragma unroll
      for (int b = 0; b < kMergeBatch; ++b) {
        const int m = warp + 8 * (i0 + b);
        int t, g;
        out_row(m, t, g);
#pragma unroll
        for (int p = 0; p < kMergeFast; ++p) {
          ls[b][p] = -INFINITY;
          if (p < np && t < rec.T) {
            ls[b][p] = lse_of(p, y * kBM + m);
            v[b][p] = part_of(p, y * kBM + m);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < kMergeBatch; ++b) {
        const int m = warp + 8 * (i0 + b);
        int t, g;
        out_row(m, t, g);
        if (t >= rec.T) continue;
        float M = -INFINITY, wsum = 0.f;
#pragma unroll
        for (int p = 0; p < kMergeFast; ++p) M = fmaxf(M, ls[b][p]);
        float wt[kMergeFast];
#pragma unroll
        for (int p = 0; p < kMergeFast; ++p) {
          wt[p] = ls[b][p] != -INFINITY ? ex2(ls[b][p] - M) : 0.f;
          wsum += wt[p];
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int p = 0; p < kMergeFast; ++p) {
          if (wt[p] != 0.f) {
            acc[0] += wt[p] * v[b][p].x; acc[1] += wt[p] * v[b][p].y;
            acc[2] += wt[p] * v[b][p].z; acc[3] += wt[p] * v[b][p].w;
          }
        }
        store(t, g, acc, wsum, M);
      }
    } else {
      for (int b = 0; b < kMergeBatch; ++b) {
        const int m = warp + 8 * (i0 + b);
        int t, g;
        out_row(m, t, g);
        if (t >= rec.T) continue;
        const int row = y * kBM + m;
        float M = -INFINITY, wsum = 0.f;
        for (int p = 0; p < np; ++p) M = fmaxf(M, lse_of(p, row));
        for (int p = 0; p < np; ++p) {
          const float ls = lse_of(p, row);
          if (ls != -INFINITY) wsum += ex2(ls - M);
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int p = 0; p < np; ++p) {
          const float ls = lse_of(p, row);
          if (ls == -INFINITY) continue;
          const float wt = ex2(ls - M);
          const float4 v = part_of(p, row);
          acc[0] += wt * v.x; acc[1] += wt * v.y; acc[2] += wt * v.z; acc[3] += wt * v.w;
        }
        store(t, g, acc, wsum, M);
      }
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

size_t attention_tc_workspace_size(const spec_attn_params*) {
  return tc_ws_layout(attention_ctas()).total;
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
  const TcWs lay = tc_ws_layout(ctas);
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
  d.recs = reinterpret_cast<MergeRec*>(w + lay.recs);
  d.part_o = reinterpret_cast<float*>(w + lay.part_o);
  d.part_lse = reinterpret_cast<float*>(w + lay.part_lse);
  d.B = p->B; d.N = p->N; d.H_q = p->H_q; d.H_kv = p->H_kv; d.G = G;
  d.log2G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : 4;
  d.T_max = p->T_max; d.W = (p->T_max + 31) / 32;
  d.num_blocks = p->num_blocks; d.max_blocks = p->max_blocks_per_req;
  d.kv_rows = int(kv_rows);
  d.ctas = ctas;
  const float scale = p->scale > 0.f ? p->scale : 1.f / sqrtf(float(kD));
  d.scale_log2 = scale * 1.4426950408889634f;
  static DeviceOnce raised_main, raised_single, raised_small;
  spec_status_t st = raise_dyn_smem_once(attn_tc_kernel, kSmemBytes, raised_main);
  if (st == SPEC_OK)
    st = raise_dyn_smem_once(attn_tc_single_kernel, attn1::kSmemBytes, raised_single);
  if (st == SPEC_OK)
    st = raise_dyn_smem_once(attn_tc_small_kernel, attn_s::kSmemBytes, raised_small);
  if (st != SPEC_OK) return st;
  cudaError_t le;
  if ((long long)p->T_max * G <= attn_s::kRows) {
    // every unit has at most 16 query rows: the transposed kernel with a 16-row Q box
    CUtensorMap mQs;
    cuuint64_t dims[3] = {cuuint64_t(kD), cuuint64_t(p->H_q), cuuint64_t(p->N)};
    cuuint64_t strides[2] = {cuuint64_t(kD) * 2, cuuint64_t(p->H_q) * kD * 2};
    cuuint32_t box[3] = {64, cuuint32_t(G), cuuint32_t(attn_s::kRows / G)};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&mQs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->q), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SPEC_ERR_INVALID_ARG;
    le = launch_pdl(attn_tc_small_kernel, dim3(ctas), dim3(attn_s::kThreads),
                    size_t(attn_s::kSmemBytes), s, mQs, mK, mV, mK8, mV8, d);
  } else if ((long long)p->T_max * G <= kBM) {
    // every unit has one M-tile: scores double-buffered, one M-tile per CTA
    le = launch_pdl(attn_tc_single_kernel, dim3(ctas), dim3(attn1::kThreads),
                    size_t(attn1::kSmemBytes), s, mQ, mK, mV, mK8, mV8, d);
  } else {
    le = launch_pdl(attn_tc_kernel, dim3(ctas), dim3(kThreads), size_t(kSmemBytes), s,
                    mQ, mK, mV, mK8, mV8, d);
  }
  // a record covers two M-tiles only when some unit has more than 128 query rows
  const unsigned merge_y = (long long)p->T_max * G > kBM ? 2u : 1u;
  if (le == cudaSuccess)
    le = launch_pdl(attn_merge_kernel, dim3(ctas, merge_y, kMergeSplit), dim3(256), 0, s, d);
  return launch_result(le);
}

}  // namespace spec
