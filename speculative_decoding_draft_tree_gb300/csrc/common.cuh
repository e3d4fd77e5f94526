// Shared device and host helpers of the verification library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "spec_verify.h"

#define SPEC_HOST_DEVICE __host__ __device__ __forceinline__

namespace spec {

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
void set_last_cuda_error(cudaError_t e);
int sm_count_current_device();
void count_launch();   // one kernel enqueued by this library (spec_kernel_launches)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline spec_status_t launch_status() {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    return SPEC_ERR_CUDA;
  }
  return SPEC_OK;
}

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// One bit per device (ids 0..63) recording that a per-device host-side step (a kernel attribute)
// was done.  Safe to share between host threads: the steps it guards are idempotent, so two
// threads that both find the bit clear both do the step and both set the bit.
struct DeviceOnce {
  std::atomic<uint64_t> done{0};
  bool test(int dev) const {
    return ((done.load(std::memory_order_acquire) >> dev) & 1u) != 0;
  }
  void set(int dev) { done.fetch_or(uint64_t(1) << dev, std::memory_order_release); }
};

// Raises `kernel`'s dynamic shared memory limit to `bytes` on the current device, once per
// device (`once` belongs to the kernel).
template <typename K>
spec_status_t raise_dyn_smem_once(K kernel, size_t bytes, DeviceOnce& once) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    if (e != cudaSuccess) set_last_cuda_error(e);
    return SPEC_ERR_CUDA;
  }
  if (!once.test(dev)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e != cudaSuccess) {
      set_last_cuda_error(e);
      return SPEC_ERR_CUDA;
    }
    once.set(dev);
  }
  return SPEC_OK;
}

// Launch with programmatic stream serialization allowed: the kernel may be scheduled while the
// previous kernel on the stream is still running (once every CTA of that kernel has executed
// pdl_trigger or exited), and waits in pdl_wait until that kernel has completed and its memory
// is visible.  This hides the launch latency between the dependent kernels of one call and
// across calls.  After any other stream operation it behaves like a plain launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e == cudaSuccess) count_launch();
  return e;
}

inline spec_status_t launch_result(cudaError_t e) {
  if (e != cudaSuccess) {
    set_last_cuda_error(e);
    cudaGetLastError();   // the error is reported here; do not leave it for the next call
    return SPEC_ERR_CUDA;
  }
  return launch_status();
}

// ------------------------------------------------------------------------------------------
// device side
// ------------------------------------------------------------------------------------------
// Every kernel of the library calls pdl_wait() before its first global memory access (the
// previous kernel on the stream may still be writing its inputs) and pdl_trigger(), which lets
// the next kernel be scheduled early -- right after the wait in most kernels; after its stores
// in a kernel whose run overlapped by the next kernel's waiting CTAs measured slower (the tree
// build fused with the rotary step).  Both are no-ops for a plain launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <typename T> struct elem;
template <> struct elem<float> {
  static constexpr int per16 = 4;
  __device__ __forceinline__ static void unpack(const uint4& v, float* out) {
    out[0] = __uint_as_float(v.x); out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z); out[3] = __uint_as_float(v.w);
  }
  __device__ __forceinline__ static float load1(const float* p) { return __ldg(p); }
};
template <> struct elem<__nv_bfloat16> {
  static constexpr int per16 = 8;
  __device__ __forceinline__ static void unpack(const uint4& v, float* out) {
    out[0] = bf16_lo(v.x); out[1] = bf16_hi(v.x); out[2] = bf16_lo(v.y); out[3] = bf16_hi(v.y);
    out[4] = bf16_lo(v.z); out[5] = bf16_hi(v.z); out[6] = bf16_lo(v.w); out[7] = bf16_hi(v.w);
  }
  __device__ __forceinline__ static float load1(const __nv_bfloat16* p) {
    uint16_t b = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(uint32_t(b) << 16);
  }
};

// streaming 16-byte load (read once: do not keep in L1)
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (one 64-bit register pair): fma.rn.f32x2 / add.f32x2 do two lanes' worth of
// FMA / add in one instruction.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// three-input maximum (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) at global address p into L2: one
// instruction, no registers held while the data moves.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, int bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Double-float (unevaluated sum hi + lo) accumulation: Knuth's TwoSum followed by a
// renormalisation (Dekker 1971 / Hida-Li-Bailey double-double addition, fp32 edition).
struct dfloat {
  float hi, lo;
};
__device__ __forceinline__ dfloat df_make(float a) { return {a, 0.f}; }
__device__ __forceinline__ dfloat df_add(dfloat a, dfloat b) {
  float s = a.hi + b.hi;
  float v = s - a.hi;
  float e = (a.hi - (s - v)) + (b.hi - v);
  e += a.lo + b.lo;
  float hi = s + e;
  float lo = e - (hi - s);
  return {hi, lo};
}
__device__ __forceinline__ dfloat df_add_f(dfloat a, float b) { return df_add(a, df_make(b)); }
__device__ __forceinline__ double df_to_d(dfloat a) { return double(a.hi) + double(a.lo); }
__device__ __forceinline__ dfloat df_shfl_xor(dfloat a, int o) {
  return {__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ dfloat df_shfl_up(dfloat a, int o) {
  return {__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ dfloat warp_sum_df(dfloat v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_add(v, df_shfl_xor(v, o));
  return v;
}
// inclusive prefix sum across the warp
__device__ __forceinline__ dfloat warp_scan_df(dfloat v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    dfloat t = df_shfl_up(v, o);
    if (lane >= o) v = df_add(v, t);
  }
  return v;
}

}  // namespace spec
