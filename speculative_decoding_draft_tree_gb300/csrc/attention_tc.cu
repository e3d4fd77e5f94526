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
// request's P_r + T_r logical KV slots in tiles of 128 keys (8 paged blocks of 16).  A device
// prep kernel lists the units, splits long KV ranges so the persistent grid has about four
// items per SM, and sorts the items longest first.
//
// CTA (one per SM, 256 threads):
//   warp 0      TMA producer: Q tile once per item, then K and V tiles of each KV block
//               (128-byte swizzle) into a 2-stage ring; blocks past the request or with a bad
//               block id are fetched from an out-of-range row, which TMA fills with zeros;
//   warp 1      one thread issues tcgen05.mma: S = Q K^T (M=128, N=128, K=16 x 8) into one of two
//               TMEM score buffers, then O += P V (V as an MN-major operand) into the TMEM
//               accumulator, and commits completions to mbarriers;
//   warps 4..7  softmax: each thread owns one row (TMEM lane); tcgen05.ld of the scores, the
//               ancestor mask on the tiles that reach the tree slots, exp2 with a lazily updated
//               reference max (O and the row sum are rescaled only when the max grows by more
//               than 2^8), P written to shared memory in the swizzled K-major layout; epilogue
//               reads O from TMEM and writes bf16 O (+ LSE) or an fp32 partial for the merge.
// Every wait is bounded (clock64 limit) and an expired wait flags SPEC_REQ_TIMEOUT and lets
// every role drain and exit; TMEM is always freed.
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
constexpr int kThreads = 384;               // 4 control warps + 8 softmax warps
constexpr int kAtom = 16384;                  // 128 rows x 128 B
constexpr int kTile = 2 * kAtom;              // 128 x 128 bf16
constexpr int kKStages = 3;                   // K tiles are released right after QK^T
constexpr int kVStages = 2;                   // V tiles are released after PV
constexpr int kSmemQ = 0;
constexpr int kSmemK = kSmemQ + kTile;
constexpr int kSmemV = kSmemK + kKStages * kTile;
constexpr int kSmemP = kSmemV + kVStages * kTile;
constexpr int kSmemBar = kSmemP + kTile;
constexpr int kSmemRed = kSmemBar + 256;      // [2 buffers][2 halves][128 rows] fp32 exchange
constexpr int kSmemEnd = kSmemRed + 2048;
constexpr int kSmemBytes = 232448;            // the per-CTA maximum; the slack aligns the base
constexpr long long kWaitLimit = 4000000000LL;     // clock cycles (~2 s)
constexpr int kSplitMinTiles = 4;
constexpr int kItemsPerSm = 4;
constexpr float kLazyRescale = 8.0f;          // log2 units
}  // namespace attn

struct Item {
  int r, h, mt, j0, j1, slot, pad0, pad1;
};
struct CombineUnit {
  int r, h, mt, slot0, nsplit, pad0, pad1, pad2;
};

struct TcDev {
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* node_offset;
  const uint32_t* anc;
  __nv_bfloat16* o;
  float* lse;
  int32_t* req_status;
  int* header;  // [0] items, [1] combine units
  Item* items;
  Item* items_tmp;
  CombineUnit* combine;
  float* part_o;
  float* part_lse;
  int B, N, H_q, H_kv, G, log2G, T_max, W, num_blocks, max_blocks, kv_rows;
  int max_items, max_combine, split_target;
  float scale_log2;
};

// ------------------------------------------------------------------------------ workspace
struct TcWs {
  size_t header, items, items_tmp, combine, part_o, part_lse, total;
  int max_items, max_combine, max_slots, split_target;
};

static TcWs tc_ws_layout(const spec_attn_params* p, int sms) {
  TcWs w;
  const int G = p->H_q / p->H_kv;
  const int tpt = attn::kBM / G;
  const long units = long(p->B) * p->H_kv * ((p->T_max + tpt - 1) / tpt);
  w.split_target = attn::kItemsPerSm * (sms > 0 ? sms : 1);
  w.max_items = int(units + w.split_target);
  w.max_combine = w.split_target;
  w.max_slots = 2 * w.split_target;
  size_t off = 0;
  w.header = off; off = align_up(off + 64, 256);
  w.items = off; off = align_up(off + sizeof(Item) * size_t(w.max_items), 256);
  w.items_tmp = off; off = align_up(off + sizeof(Item) * size_t(w.max_items), 256);
  w.combine = off; off = align_up(off + sizeof(CombineUnit) * size_t(w.max_combine), 256);
  w.part_o = off; off = align_up(off + sizeof(float) * size_t(w.max_slots) * attn::kBM * attn::kD, 256);
  w.part_lse = off; off = align_up(off + sizeof(float) * size_t(w.max_slots) * attn::kBM, 256);
  w.total = off;
  return w;
}

// ------------------------------------------------------------------------------ prep
__device__ __forceinline__ void req_geom(const TcDev& a, int r, int& o, int& T, int& P, int& mts,
                                         int& nts) {
  o = a.node_offset[r];
  T = a.node_offset[r + 1] - o;
  P = a.prefix_len[r];
  const int tpt = attn::kBM >> a.log2G;
  mts = (T + tpt - 1) / tpt;
  nts = (P + T + attn::kBN - 1) / attn::kBN;
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

__global__ void __launch_bounds__(1024) attn_prep_kernel(TcDev a) {
  __shared__ int s_warp[32];
  __shared__ int s_hist[1024];
  __shared__ long long s_total;
  const int tid = threadIdx.x;
  // phase 1: total tile work over valid requests
  long long mine = 0;
  for (int r = tid; r < a.B; r += 1024) {
    int o, T, P, mts, nts;
    req_geom(a, r, o, T, P, mts, nts);
    const int nblk = (P + T + attn::kBS - 1) / attn::kBS;
    if (a.req_status[r] == 0 && nblk > a.max_blocks) atomicOr(&a.req_status[r], SPEC_REQ_BAD_BLOCK);
    if (a.req_status[r] == 0 && T >= 1 && P >= 0) mine += (long long)a.H_kv * mts * nts;
  }
  if (tid == 0) s_total = 0;
  __syncthreads();
  atomicAdd(reinterpret_cast<unsigned long long*>(&s_total), (unsigned long long)mine);
  s_hist[tid] = 0;
  __syncthreads();
  const long long total = s_total;
  const int S = int(max((long long)attn::kSplitMinTiles,
                        (total + a.split_target - 1) / a.split_target));
  // phase 2+3: offsets and item generation, 1024 requests at a time
  int item_base = 0, comb_base = 0, slot_base = 0;
  for (int r0 = 0; r0 < a.B; r0 += 1024) {
    const int r = r0 + tid;
    int o = 0, T = 0, P = 0, mts = 0, nts = 0, splits = 0;
    bool ok = false;
    if (r < a.B) {
      req_geom(a, r, o, T, P, mts, nts);
      ok = a.req_status[r] == 0 && T >= 1 && P >= 0;
    }
    if (ok) splits = (nts + S - 1) / S;
    const int n_items = ok ? a.H_kv * mts * splits : 0;
    const int n_comb = (ok && splits > 1) ? a.H_kv * mts : 0;
    const int n_slot = (ok && splits > 1) ? n_items : 0;
    int e_items, e_comb, e_slot;
    const int t_items = block_excl_scan(n_items, s_warp, e_items);
    const int t_comb = block_excl_scan(n_comb, s_warp, e_comb);
    const int t_slot = block_excl_scan(n_slot, s_warp, e_slot);
    if (ok) {
      for (int h = 0; h < a.H_kv; ++h)
        for (int mt = 0; mt < mts; ++mt) {
          const int u = h * mts + mt;
          for (int s = 0; s < splits; ++s) {
            Item it;
            it.r = r; it.h = h; it.mt = mt;
            it.j0 = int((long long)s * nts / splits);
            it.j1 = int((long long)(s + 1) * nts / splits);
            it.slot = splits > 1 ? slot_base + e_slot + u * splits + s : -1;
            it.pad0 = it.pad1 = 0;
            const int idx = item_base + e_items + u * splits + s;
            if (idx < a.max_items) a.items_tmp[idx] = it;
          }
          if (splits > 1) {
            CombineUnit c;
            c.r = r; c.h = h; c.mt = mt;
            c.slot0 = slot_base + e_slot + u * splits;
            c.nsplit = splits;
            c.pad0 = c.pad1 = c.pad2 = 0;
            const int ci = comb_base + e_comb + u;
            if (ci < a.max_combine) a.combine[ci] = c;
          }
        }
    }
    item_base += t_items;
    comb_base += t_comb;
    slot_base += t_slot;
  }
  const int n_items = min(item_base, a.max_items);
  __syncthreads();  // every thread's items_tmp writes are visible before the sort reads them
  // phase 4: counting sort by tile count, longest first
  for (int i = tid; i < n_items; i += 1024) {
    const Item it = a.items_tmp[i];
    atomicAdd(&s_hist[min(it.j1 - it.j0, 1023)], 1);
  }
  __syncthreads();
  // descending exclusive offsets: bucket b starts after all buckets > b
  const int rev = s_hist[1023 - tid];
  int e_rev;
  block_excl_scan(rev, s_warp, e_rev);
  __syncthreads();
  s_hist[1023 - tid] = e_rev;
  __syncthreads();
  for (int i = tid; i < n_items; i += 1024) {
    const Item it = a.items_tmp[i];
    const int pos = atomicAdd(&s_hist[min(it.j1 - it.j0, 1023)], 1);
    a.items[pos] = it;
  }
  if (tid == 0) {
    a.header[0] = n_items;
    a.header[1] = min(comb_base, a.max_combine);
  }
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

__global__ void __launch_bounds__(attn::kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, TcDev a) {
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
  uint64_t* ex_bar = bars + 22;    // [4]: row-max / row-sum exchange of the two softmax halves

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
  const int n_items = a.header[0];
  volatile int* abort_flag = s_abort;
  const int G = a.G, log2G = a.log2G, tpt = kBM >> log2G;
  const bool layout_ok = *abort_flag == 0;

  if (layout_ok && warp == 0) {
    // ===================================================================== TMA producer
    // The whole warp runs the loop: lanes 0..7 fetch the eight block-table entries of a tile
    // (prefetched one tile ahead), lane 0 waits for free stages and issues the copies.  K runs
    // one tile ahead of V so that QK^T of the next tile never waits behind a V stage.
    if (lane == 0) {
      tc::prefetch_tensormap(&mQ);
      tc::prefetch_tensormap(&mK);
      tc::prefetch_tensormap(&mV);
    }
    int kt = 0, vt = 0, li = 0;
    bool ok = true;
    int prev_row = a.kv_rows;
    bool prev_valid = false;
    auto tile_rows = [&](const int32_t* table, int nblk, int j, int r, int h) -> int {
      int row = a.kv_rows;  // out of range: TMA fills zeros
      const int lb = j * 8 + lane;
      if (lane < 8 && lb < nblk) {
        const int pb = table[lb];
        if (pb >= 0 && pb < a.num_blocks) row = (pb * a.H_kv + h) * kBS;
        else atomicOr(&a.req_status[r], SPEC_REQ_BAD_BLOCK);
      }
      return row;
    };
    auto issue_kv = [&](const CUtensorMap* map, uint8_t* dst, uint64_t* full, int row_lane) {
      // lane b (0..7) copies block b of the tile: both 64-column halves (one swizzle atom each)
      if (lane == 0) tc::mbar_arrive_expect_tx(full, kTile);
      __syncwarp();
      if (lane < 8) {
        tc::tma_load_2d(dst + lane * 2048, map, 0, row_lane, full);
        tc::tma_load_2d(dst + kAtom + lane * 2048, map, 64, row_lane, full);
      }
      __syncwarp();
    };
    auto wait_lane0 = [&](uint64_t* bar, uint32_t parity) -> bool {
      bool r = true;
      if (lane == 0) r = tc::mbar_wait(bar, parity, abort_flag, kWaitLimit);
      return __shfl_sync(0xffffffffu, r ? 1 : 0, 0) != 0;
    };
    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++li) {
      const Item it = a.items[idx];
      const int o = a.node_offset[it.r];
      const int T = a.node_offset[it.r + 1] - o;
      const int P = a.prefix_len[it.r];
      const int nblk = (P + T + kBS - 1) / kBS;
      const int32_t* table = a.block_table + size_t(it.r) * a.max_blocks;
      if (li > 0 && !wait_lane0(q_empty, (li - 1) & 1)) { ok = false; break; }
      if (lane == 0) {
        tc::mbar_arrive_expect_tx(q_full, kTile);
        tc::tma_load_3d(sQ, &mQ, 0, it.h * G, o + it.mt * tpt, q_full);
        tc::tma_load_3d(sQ + kAtom, &mQ, 64, it.h * G, o + it.mt * tpt, q_full);
      }
      int row_cur = tile_rows(table, nblk, it.j0, it.r, it.h);
      for (int j = it.j0; j < it.j1; ++j) {
        const int row_next = (j + 1 < it.j1) ? tile_rows(table, nblk, j + 1, it.r, it.h) : a.kv_rows;
        const int kst = kt % kKStages, kuse = kt / kKStages;
        if (kuse > 0 && !wait_lane0(k_empty + kst, (kuse - 1) & 1)) { ok = false; break; }
        issue_kv(&mK, sK + kst * kTile, k_full + kst, row_cur);
        ++kt;
        if (prev_valid) {
          const int vst = vt % kVStages, vuse = vt / kVStages;
          if (vuse > 0 && !wait_lane0(v_empty + vst, (vuse - 1) & 1)) { ok = false; break; }
          issue_kv(&mV, sV + vst * kTile, v_full + vst, prev_row);
          ++vt;
        }
        prev_row = row_cur;
        prev_valid = true;
        row_cur = row_next;
      }
    }
    if (ok && prev_valid) {
      const int vst = vt % kVStages, vuse = vt / kVStages;
      if (vuse > 0 && !wait_lane0(v_empty + vst, (vuse - 1) & 1)) ok = false;
      else {
        issue_kv(&mV, sV + vst * kTile, v_full + vst, prev_row);
        ++vt;
      }
    }
    if (lane == 0) {
      if (!ok) *abort_flag = 1;
      // drain: wait for the copies issued last (bounded), so none is in flight at exit
      for (int k = max(0, kt - kKStages); k < kt; ++k)
        tc::mbar_wait(k_full + k % kKStages, (k / kKStages) & 1, abort_flag, kWaitLimit / 8);
      for (int v = max(0, vt - kVStages); v < vt; ++v)
        tc::mbar_wait(v_full + v % kVStages, (v / kVStages) & 1, abort_flag, kWaitLimit / 8);
      if (li > 0) tc::mbar_wait(q_full, (li - 1) & 1, abort_flag, kWaitLimit / 8);
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
      for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++li) {
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
    // Warps 4..11: lane quarter q = warp % 4 owns TMEM lanes / rows 32q..32q+31; the two warps of
    // a quarter split the 128 keys of a score tile (half hh = 0: keys 0..63, 1: keys 64..127) and
    // the 128 output columns, exchanging row maxima and row sums through shared memory.
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
    for (int idx = blockIdx.x; idx < n_items && ok; idx += gridDim.x, ++li) {
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
      for (int j = it.j0; j < it.j1; ++j, ++kv_it) {
        const int st = kv_it & 1, use = kv_it >> 1;
        if (!warp_wait(s_full + st, use & 1, abort_flag)) { ok = false; break; }
        tc::tc_fence_after();
        // this warp's 64 scores, one TMEM round trip; the S buffer is released right away
        uint32_t sr[64];
        {
          uint32_t* lo = sr;
          tc::tmem_ld32(tmem + lane_addr + st * 128 + 64 * hh, *reinterpret_cast<uint32_t(*)[32]>(lo));
          tc::tmem_ld32(tmem + lane_addr + st * 128 + 64 * hh + 32,
                        *reinterpret_cast<uint32_t(*)[32]>(lo + 32));
          tc::tmem_ld_wait();
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(s_free + st);
        // mask + scale (log2 units)
        const int key0 = j * kBN + 64 * hh;
        const bool all_prefix = key0 + 64 <= P;
        const int npre = P - key0;    // columns below npre are prefix keys
        const uint32_t w0 = all_prefix ? 0xffffffffu : anc_window(anc, a.W, key0 - P);
        const uint32_t w1 = all_prefix ? 0xffffffffu : anc_window(anc, a.W, key0 - P + 32);
        float pmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const uint32_t wd = c < 32 ? w0 : w1;
          const bool vis = valid && ((c < npre) || ((wd >> (c & 31)) & 1u));
          const float x = vis ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
          sr[c] = __float_as_uint(x);
          pmax = fmaxf(pmax, x);
        }
        const float tmax = fmaxf(pmax, exchange(pmax));
        if (!ex_ok) { ok = false; break; }
        const bool grow = tmax > m_ref + kLazyRescale;
        const float new_ref = grow ? tmax : m_ref;
        const float factor = (grow && m_ref != -INFINITY) ? ex2(m_ref - new_ref) : 1.f;
        // PV of the previous tile must be complete before P and O are touched
        if (j > it.j0 && !warp_wait(pv_done, (kv_it - 1) & 1, abort_flag)) { ok = false; break; }
        float rowsum = 0.f;
        const bool live = new_ref != -INFINITY;
        uint8_t* rowp = sP + hh * kAtom + (m >> 3) * 1024 + (m & 7) * 128;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {   // 8 keys = one 16-byte chunk of the swizzled row
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float x0 = __uint_as_float(sr[ch * 8 + e]);
            const float x1 = __uint_as_float(sr[ch * 8 + e + 1]);
            const float p0 = live ? ex2(x0 - new_ref) : 0.f;
            const float p1 = live ? ex2(x1 - new_ref) : 0.f;
            rowsum += p0 + p1;
            pk[e >> 1] = pack_bf16(p0, p1);
          }
          *reinterpret_cast<uint4*>(rowp + ((ch ^ (m & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
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
        // last tile: zero V rows past the request's KV length (stale cache rows times P = 0
        // must not turn into NaN); TMA must have landed first.  Half hh clears d-atom hh.
        if (j * kBN + kBN > kv_len) {
          if (!warp_wait(v_full + st, use & 1, abort_flag)) { ok = false; break; }
          const int key = m;
          if (key >= kv_len - j * kBN) {
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
    // every request this CTA was assigned is unreliable after an expired wait
    for (int idx = blockIdx.x; idx < n_items; idx += gridDim.x)
      atomicOr(&a.req_status[a.items[idx].r], SPEC_REQ_TIMEOUT);
  }
  tc::tc_fence_after();
  if (warp == 0) tc::tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------------------ combine
__global__ void __launch_bounds__(128) attn_combine_kernel(TcDev a) {
  const int n_comb = a.header[1];
  const int m = threadIdx.x;
  for (int u = blockIdx.x; u < n_comb; u += gridDim.x) {
    const CombineUnit cu = a.combine[u];
    const int o = a.node_offset[cu.r];
    const int T = a.node_offset[cu.r + 1] - o;
    const int tpt = attn::kBM >> a.log2G;
    const int t = cu.mt * tpt + (m >> a.log2G);
    const int g = m & (a.G - 1);
    if (t >= T) continue;
    float M = -INFINITY;
    for (int s = 0; s < cu.nsplit; ++s) M = fmaxf(M, a.part_lse[size_t(cu.slot0 + s) * attn::kBM + m]);
    float wsum = 0.f;
    float acc[attn::kD];
#pragma unroll
    for (int c = 0; c < attn::kD; ++c) acc[c] = 0.f;
    for (int s = 0; s < cu.nsplit; ++s) {
      const float ls = a.part_lse[size_t(cu.slot0 + s) * attn::kBM + m];
      if (ls == -INFINITY) continue;
      const float w = ex2(ls - M);
      wsum += w;
      const float* prow = a.part_o + (size_t(cu.slot0 + s) * attn::kBM + m) * attn::kD;
#pragma unroll
      for (int c = 0; c < attn::kD; c += 4) {
        const float4 v = *reinterpret_cast<const float4*>(prow + c);
        acc[c] += w * v.x; acc[c + 1] += w * v.y; acc[c + 2] += w * v.z; acc[c + 3] += w * v.w;
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __nv_bfloat16* orow = a.o + (size_t(o + t) * a.H_q + cu.h * a.G + g) * attn::kD;
#pragma unroll
    for (int c = 0; c < attn::kD; c += 8) {
      uint4 v;
      v.x = pack_bf16(acc[c] * inv, acc[c + 1] * inv);
      v.y = pack_bf16(acc[c + 2] * inv, acc[c + 3] * inv);
      v.z = pack_bf16(acc[c + 4] * inv, acc[c + 5] * inv);
      v.w = pack_bf16(acc[c + 6] * inv, acc[c + 7] * inv);
      *reinterpret_cast<uint4*>(orow + c) = v;
    }
    if (a.lse) a.lse[size_t(o + t) * a.H_q + cu.h * a.G + g] = (M + __log2f(wsum)) * 0.6931471805599453f;
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

size_t attention_tc_workspace_size(const spec_attn_params* p) {
  return tc_ws_layout(p, sm_count_current_device()).total;
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
  const int sms = sm_count_current_device();
  if (sms <= 0) return SPEC_ERR_CUDA;
  const TcWs lay = tc_ws_layout(p, sms);
  if (!ws || ws_bytes < lay.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return SPEC_ERR_INVALID_ARG;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return SPEC_ERR_CUDA;
  CUtensorMap mQ, mK, mV;
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
  d.items = reinterpret_cast<Item*>(w + lay.items);
  d.items_tmp = reinterpret_cast<Item*>(w + lay.items_tmp);
  d.combine = reinterpret_cast<CombineUnit*>(w + lay.combine);
  d.part_o = reinterpret_cast<float*>(w + lay.part_o);
  d.part_lse = reinterpret_cast<float*>(w + lay.part_lse);
  d.B = p->B; d.N = p->N; d.H_q = p->H_q; d.H_kv = p->H_kv; d.G = G;
  d.log2G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : 4;
  d.T_max = p->T_max; d.W = (p->T_max + 31) / 32;
  d.num_blocks = p->num_blocks; d.max_blocks = p->max_blocks_per_req;
  d.kv_rows = int(kv_rows);
  d.max_items = lay.max_items; d.max_combine = lay.max_combine; d.split_target = lay.split_target;
  const float scale = p->scale > 0.f ? p->scale : 1.f / sqrtf(float(kD));
  d.scale_log2 = scale * 1.4426950408889634f;
  static std::once_flag attr_once;
  std::call_once(attr_once, [] {
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  attn_prep_kernel<<<1, 1024, 0, s>>>(d);
  attn_tc_kernel<<<sms, kThreads, kSmemBytes, s>>>(mQ, mK, mV, d);
  attn_combine_kernel<<<lay.max_combine, 128, 0, s>>>(d);
  return launch_status();
}

}  // namespace spec
