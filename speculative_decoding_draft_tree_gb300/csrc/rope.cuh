// Rotary position embedding of tree tokens and the tree K/V slot write: the pieces shared by the
// standalone kernel (rope_kv.cu) and the kernel fused with the tree build (tree_build.cu).
//
// Source: "投机推理算法的常见优化手段" (cnblogs zrq96), 草稿树的验证——树形掩码 -- the forward over the
// draft tree takes the tree, its mask, its position ids and the KV cache, and all of them must
// follow the tree.  Position ids enter as rotary embeddings (RoFormer, Su et al. 2021, section
// 3.2): pair j of a head vector turns by pos * base^(-2j / rotary_dim).
//
// Work is cut into 16-byte items per node: a q or k row contributes one item per vector, except
// that a half-split pair of vectors (j, j + rotary_dim/2) is one item; a v row is a plain copy.
// Each angle is formed and reduced modulo 2 pi in fp64 (positions reach tens of thousands of
// radians, where an fp32 product would already be off by ~1e-3), then sincosf of the reduced
// fp32 angle; rotation runs in fp32 and rounds to the storage type once.
#pragma once

#include <cmath>

#include "common.cuh"

namespace spec {

constexpr int kRopeMaxPairs = 128;   // rotary_dim <= 256

struct RopeDev {
  const char* q_in;
  char* q_out;
  const char* k_new;
  const char* v_new;
  char* k_cache;
  char* v_cache;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* node_offset;
  const int32_t* pos_id;
  int32_t* req_status;
  int32_t B, N, H_q, H_kv;
  int32_t row_bytes;   // head_dim * element size
  int32_t d_vecs;      // 16-byte vectors per head row
  int32_t rot_vecs;    // vectors holding rotated components (rotary_dim / elements per vector)
  int32_t items_qk;    // work items per q / k row
  int32_t items_node;  // work items per node: (H_q + H_kv) * items_qk + H_kv * d_vecs
  int32_t rot_pairs;   // rotary_dim / 2
  int32_t interleaved;
  int32_t bs, num_blocks, max_blocks;
  int32_t bf16;
  double theta[kRopeMaxPairs];   // base^(-2j / rotary_dim), formed on the host in fp64
};

// Host: validate a spec_rope_params block and fill the kernel arguments.
spec_status_t make_rope_dev(const spec_rope_params* p, RopeDev* d);

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <typename T>
__device__ __forceinline__ uint4 pack_vec(const float* x) {
  uint4 v;
  if constexpr (sizeof(T) == 2) {
    v.x = pack_bf16x2(x[0], x[1]); v.y = pack_bf16x2(x[2], x[3]);
    v.z = pack_bf16x2(x[4], x[5]); v.w = pack_bf16x2(x[6], x[7]);
  } else {
    v.x = __float_as_uint(x[0]); v.y = __float_as_uint(x[1]);
    v.z = __float_as_uint(x[2]); v.w = __float_as_uint(x[3]);
  }
  return v;
}

// Streaming 16-byte load through the coherent path: q may be rotated in place (q_out == q_in),
// so the read-only (non-coherent) path is not used.
__device__ __forceinline__ uint4 ld_cs16(const void* p) {
  uint4 v;
  asm volatile("ld.global.cs.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// What work item f of node n touches: source and destination rows, the vectors inside the row,
// and how to treat them.  kv_off = byte offset of the node's cache slot (block and row) in
// layer 0 of the cache, head 0.
struct RopeItem {
  const char* src;
  char* dst;
  int v0, v1;    // vector indices: v1 >= 0 only for a half-split pair (v0, v1)
  int kind;      // 0 copy, 1 rotate pairs inside v0 (interleaved), 2 rotate across (v0, v1)
};

__device__ __forceinline__ RopeItem rope_item(const RopeDev& a, int n, int f, size_t kv_off) {
  RopeItem it;
  const int nq = a.H_q * a.items_qk;
  const int nk = a.H_kv * a.items_qk;
  if (f < nq + nk) {
    const bool is_q = f < nq;
    const int g = is_q ? f : f - nq;
    const int h = g / a.items_qk;
    const int j = g - h * a.items_qk;
    if (is_q) {
      const size_t off = (size_t(n) * a.H_q + h) * a.row_bytes;
      it.src = a.q_in + off;
      it.dst = a.q_out + off;
    } else {
      it.src = a.k_new + (size_t(n) * a.H_kv + h) * a.row_bytes;
      it.dst = a.k_cache + kv_off + size_t(h) * a.bs * a.row_bytes;
    }
    const int half = a.rot_vecs / 2;
    if (a.interleaved) {
      it.v0 = j;
      it.v1 = -1;
      it.kind = j < a.rot_vecs ? 1 : 0;
    } else if (j < half) {
      it.v0 = j;
      it.v1 = j + half;
      it.kind = 2;
    } else {
      it.v0 = j + half;
      it.v1 = -1;
      it.kind = 0;
    }
  } else {
    const int g = f - nq - nk;
    const int h = g / a.d_vecs;
    const int j = g - h * a.d_vecs;
    it.src = a.v_new + (size_t(n) * a.H_kv + h) * a.row_bytes;
    it.dst = a.v_cache + kv_off + size_t(h) * a.bs * a.row_bytes;
    it.v0 = j;
    it.v1 = -1;
    it.kind = 0;
  }
  return it;
}

__device__ __forceinline__ void rope_load(const RopeItem& it, uint4& x0, uint4& x1) {
  x0 = ld_cs16(it.src + it.v0 * 16);
  if (it.v1 >= 0) x1 = ld_cs16(it.src + it.v1 * 16);
}

// (cos, sin) of pair j's angle at position pos
__device__ __forceinline__ float2 rope_cos_sin(const RopeDev& a, int pos, int j) {
  const double ang = double(pos) * a.theta[j];
  const double turns = rint(ang * 0.15915494309189535);   // 1 / (2 pi)
  const float red = float(fma(-turns, 6.283185307179586, ang));
  float s, c;
  sincosf(red, &s, &c);
  return make_float2(c, s);
}

// Rotate (or copy) one loaded item and store it; cs = the node's (cos, sin) per pair.
template <typename T>
__device__ __forceinline__ void rope_store(const RopeItem& it, const uint4& x0, const uint4& x1,
                                           const float2* cs) {
  constexpr int EPV = 16 / sizeof(T);
  if (it.kind == 0) {
    *reinterpret_cast<uint4*>(it.dst + it.v0 * 16) = x0;
    return;
  }
  float a0[EPV], o0[EPV];
  elem<T>::unpack(x0, a0);
  if (it.kind == 1) {   // pairs (2j, 2j+1) inside one vector
#pragma unroll
    for (int e = 0; e < EPV; e += 2) {
      const float2 c = cs[(it.v0 * EPV + e) >> 1];
      o0[e] = fmaf(a0[e], c.x, -a0[e + 1] * c.y);
      o0[e + 1] = fmaf(a0[e], c.y, a0[e + 1] * c.x);
    }
    *reinterpret_cast<uint4*>(it.dst + it.v0 * 16) = pack_vec<T>(o0);
  } else {              // pairs (j, j + rotary_dim/2) across two vectors
    float b0[EPV], o1[EPV];
    elem<T>::unpack(x1, b0);
#pragma unroll
    for (int e = 0; e < EPV; ++e) {
      const float2 c = cs[it.v0 * EPV + e];
      o0[e] = fmaf(a0[e], c.x, -b0[e] * c.y);
      o1[e] = fmaf(a0[e], c.y, b0[e] * c.x);
    }
    *reinterpret_cast<uint4*>(it.dst + it.v0 * 16) = pack_vec<T>(o0);
    *reinterpret_cast<uint4*>(it.dst + it.v1 * 16) = pack_vec<T>(o1);
  }
}

}  // namespace spec
