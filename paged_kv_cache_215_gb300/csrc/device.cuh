// device.cuh -- sm_103a device helpers: inline PTX for mbarriers, TMA tensor
// loads, ldmatrix / movmatrix, mma.sync, grid-dependency control, and the
// element conversions the kernels use.  Included only by the library's .cu files.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Bounded spin: after this many failed polls a wait gives up, records
// PKV_ETIMEOUT and returns false.  try_wait suspends the thread for a
// hardware-chosen interval per poll, so this is on the order of seconds.
constexpr uint32_t kMaxPolls = 1u << 22;

__device__ __forceinline__ void record_error(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with this parity to complete; false after kMaxPolls polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kMaxPolls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// ---------------------------------------------------------------- TMA
// 3-D tiled tensor load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- PDL
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- ldmatrix / movmatrix / mma
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// D += A(16x16) * B(16x8), fp32 accumulate; `kBf16` selects bf16 or f16 inputs.
template <bool kBf16>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (kBf16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7},"
        " {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kBf16) return pack_bf16(lo, hi);
  else return pack_f16(lo, hi);
}
template <bool kBf16>
__device__ __forceinline__ float2 unpack2(uint32_t x) {
  if constexpr (kBf16) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&x);
    return __bfloat1622float2(v);
  } else {
    __half2 v = *reinterpret_cast<__half2*>(&x);
    return __half22float2(v);
  }
}

// Two E4M3 codes (low byte first) -> f16x2, exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(x), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Four E4M3 codes in one register (byte 0 first) -> two f16x2: lo = bytes 0,1;
// hi = bytes 2,3.  Exact.  The 16-bit halves are taken with a register unpack.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t x, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
}

__device__ __forceinline__ uint32_t byte_perm(uint32_t a, uint32_t b, uint32_t sel) {
  return __byte_perm(a, b, sel);
}

// Load one element of q/out dtype as float.
__device__ __forceinline__ float load_as_float(const void* base, size_t idx, int dtype) {
  switch (dtype) {
    case PKV_F32: return static_cast<const float*>(base)[idx];
    case PKV_F16: return __half2float(static_cast<const __half*>(base)[idx]);
    case PKV_BF16: return __bfloat162float(static_cast<const __nv_bfloat16*>(base)[idx]);
    default: return 0.f;
  }
}

__device__ __forceinline__ void store_from_float(void* base, size_t idx, int dtype, float v) {
  switch (dtype) {
    case PKV_F32: static_cast<float*>(base)[idx] = v; break;
    case PKV_F16: static_cast<__half*>(base)[idx] = __float2half_rn(v); break;
    case PKV_BF16: static_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v); break;
    default: break;
  }
}

// Generic-proxy writes to global memory made visible to later TMA (async-proxy) reads.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Eight consecutive elements of an f32 / f16 / bf16 array as floats (16-byte aligned).
__device__ __forceinline__ void load8_as_float(const void* src, size_t idx, int dtype,
                                               float (&x)[8]) {
  if (dtype == PKV_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + idx);
    const float4 a = p[0], b = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 r = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + idx);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = dtype == PKV_BF16 ? unpack2<true>(w[i]) : unpack2<false>(w[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
}

// Per-tensor E4M3 store rule: y = x / scale (IEEE fp32 division), round to
// nearest even, finite overflow and +-Inf saturate to +-448, NaN -> 0x7F.
__device__ __forceinline__ uint8_t encode_e4m3(float x, float scale) {
  const float y = __fdiv_rn(x, scale);
  if (isnan(y)) return 0x7F;
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3));
}

// Store 8 consecutive elements of one token row into the pool: a 16-byte copy
// for a pool of the input's dtype, or E4M3 encoding into 8 bytes.
__device__ __forceinline__ void store8_to_pool(void* pool, size_t dst, int kv_dtype,
                                               const void* src, size_t sidx, int in_dtype,
                                               float scale) {
  if (kv_dtype == PKV_FP8_E4M3) {
    float x[8];
    load8_as_float(src, sidx, in_dtype, x);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      lo |= static_cast<uint32_t>(encode_e4m3(x[e], scale)) << (8 * e);
      hi |= static_cast<uint32_t>(encode_e4m3(x[4 + e], scale)) << (8 * e);
    }
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(pool) + dst) = make_uint2(lo, hi);
  } else if (kv_dtype == PKV_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(src) + sidx);
    float4* q = reinterpret_cast<float4*>(static_cast<float*>(pool) + dst);
    q[0] = p[0];
    q[1] = p[1];
  } else {
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(pool) + dst) =
        *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) + sidx);
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace pkv
