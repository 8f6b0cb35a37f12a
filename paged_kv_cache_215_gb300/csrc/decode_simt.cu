// decode_simt.cu -- paged decode attention on the CUDA cores, for the shapes
// and dtypes the tensor-core kernel does not take (fp32 K/V, head_dim other
// than 128, more than 8 query heads per KV head).
//
// Same computation as decode_mma.cu ("Unlocking long context", sections 4.1
// and 5.1; long-context article at mhpn.cn, section 3.2; "The engineering truth
// of long-context inference 2026", sections 2.2 and 3.1): CTA (p, hkv, s) takes
// block-aligned partition p of sequence s for KV head hkv.  Each of its four
// warps walks every fourth token; lanes split the head dimension, a warp
// reduction gives each query head's score, and every warp keeps an online
// softmax (running max m and sum l, rescaled by exp2(m_old - m_new)).  The four
// warps' states are combined through shared memory at the end.
#include "device.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kWarps = 4;
constexpr int kMaxG = 16;
constexpr int kMaxDL = 8;   // head_dim / 32 per lane, head_dim <= 256

template <int KVT>
__device__ __forceinline__ float load_kv(const void* pool, size_t idx) {
  if constexpr (KVT == PKV_F32) return static_cast<const float*>(pool)[idx];
  else if constexpr (KVT == PKV_F16) return __half2float(static_cast<const __half*>(pool)[idx]);
  else if constexpr (KVT == PKV_BF16)
    return __bfloat162float(static_cast<const __nv_bfloat16*>(pool)[idx]);
  else {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<const uint8_t*>(pool)[idx], __NV_E4M3);
    return __half2float(__half(h));
  }
}

template <int KVT>
__global__ void __launch_bounds__(32 * kWarps) decode_simt_kernel(const DecodeArgs a) {
  const int p = blockIdx.x, hkv = blockIdx.y, s = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.G, D = a.D, DL = a.D / 32;
  extern __shared__ float sm[];
  float* qs = sm;                                   // [G][D], pre-scaled into log2 units
  float* wm = qs + G * D;                           // [kWarps][G] running max per warp
  float* wl = wm + kWarps * G;                      // [kWarps][G] running sum per warp
  float* wo = wl + kWarps * G;                      // [kWarps][G][D] accumulators per warp

  int n = __ldg(a.seq_lens + s);
  const int cap = a.max_blocks * a.BS;
  if (n < 0 || n > cap) {
    if (threadIdx.x == 0) record_error(a.status, PKV_EBOUNDS);
    n = n < 0 ? 0 : cap;
  }
  const int nb = (n + a.BS - 1) / a.BS;
  const int jb = (int)((long long)p * nb / a.S), je = (int)((long long)(p + 1) * nb / a.S);
  const int tb = jb * a.BS, te = min(je * a.BS, n);

  for (int i = threadIdx.x; i < G * D; i += blockDim.x)
    qs[i] = load_as_float(a.q, ((size_t)s * a.Hq + (size_t)hkv * G) * D + i, a.q_dtype) *
            a.qk_scale_log2;
  __syncthreads();

  float m[kMaxG], l[kMaxG], acc[kMaxG][kMaxDL];
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxDL; ++k) acc[g][k] = 0.f;
  }

  for (int t = tb + warp; t < te; t += kWarps) {
    int blk = __ldg(a.tables + (size_t)s * a.max_blocks + t / a.BS);
    if (blk < 0 || blk >= a.num_blocks) {
      if (lane == 0) record_error(a.status, PKV_EBOUNDS);
      blk = 0;
    }
    const size_t kb = ((((size_t)blk * 2 + 0) * a.L + a.layer) * a.Hkv + hkv) * a.BS + t % a.BS;
    const size_t vb = ((((size_t)blk * 2 + 1) * a.L + a.layer) * a.Hkv + hkv) * a.BS + t % a.BS;
    float kr[kMaxDL], vr[kMaxDL];
    // E4M3 block-wise scales: this token's K / V tile scales (the per-tensor
    // scales are folded into qs and into the output instead)
    float kbs = 1.f, vbs = 1.f;
    if (KVT == PKV_FP8_E4M3 && a.block_scales) {
      kbs = a.block_scales[(((size_t)blk * 2 + 0) * a.L + a.layer) * a.Hkv + hkv];
      vbs = a.block_scales[(((size_t)blk * 2 + 1) * a.L + a.layer) * a.Hkv + hkv];
    }
#pragma unroll
    for (int k = 0; k < kMaxDL; ++k) {
      if (k < DL) {
        kr[k] = load_kv<KVT>(a.pool, kb * D + lane + 32 * k) * kbs;
        vr[k] = load_kv<KVT>(a.pool, vb * D + lane + 32 * k) * vbs;
      }
    }
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      if (g < G) {
        float part = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxDL; ++k)
          if (k < DL) part = fmaf(kr[k], qs[g * D + lane + 32 * k], part);
        const float sc = warp_sum(part);
        const float mn = fmaxf(m[g], sc);
        const float al = exp2f(m[g] - mn), pr = exp2f(sc - mn);
        m[g] = mn;
        l[g] = l[g] * al + pr;
#pragma unroll
        for (int k = 0; k < kMaxDL; ++k)
          if (k < DL) acc[g][k] = fmaf(pr, vr[k], acc[g][k] * al);
      }
    }
  }

  // combine the warps
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) {
    if (g < G) {
      if (lane == 0) {
        wm[warp * G + g] = m[g];
        wl[warp * G + g] = l[g];
      }
#pragma unroll
      for (int k = 0; k < kMaxDL; ++k)
        if (k < DL) wo[((size_t)warp * G + g) * D + lane + 32 * k] = acc[g][k];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
    const int g = i / D, d = i % D;
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * G + g]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(wm[w * G + g] - M);
        L += wl[w * G + g] * f;
        O += wo[((size_t)w * G + g) * D + d] * f;
      }
    }
    const int h = hkv * G + g;
    const float o = L > 0.f ? O * a.v_scale / L : 0.f;
    if (a.S == 1) {
      store_from_float(a.out, ((size_t)s * a.Hq + h) * D + d, a.out_dtype, o);
    } else {
      const size_t row = ((size_t)s * a.Hq + h) * a.S + p;
      a.part_o[row * D + d] = o;
      if (d == 0) a.part_lse[row] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
    }
  }
  grid_launch_dependents();
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream) {
  if (a.G > kMaxG || a.D > 32 * kMaxDL || a.D % 32 != 0) return cudaErrorInvalidValue;
  const size_t smem = sizeof(float) * ((size_t)a.G * a.D + 2 * kWarps * a.G +
                                       (size_t)kWarps * a.G * a.D);
  dim3 grid(a.S, a.Hkv, a.B);
  cudaError_t e = cudaSuccess;
  switch (a.kv_dtype) {
    case PKV_F32:
      e = cudaFuncSetAttribute(decode_simt_kernel<PKV_F32>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_simt_kernel<PKV_F32><<<grid, 32 * kWarps, smem, stream>>>(a);
      break;
    case PKV_F16:
      e = cudaFuncSetAttribute(decode_simt_kernel<PKV_F16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_simt_kernel<PKV_F16><<<grid, 32 * kWarps, smem, stream>>>(a);
      break;
    case PKV_BF16:
      e = cudaFuncSetAttribute(decode_simt_kernel<PKV_BF16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess) decode_simt_kernel<PKV_BF16><<<grid, 32 * kWarps, smem, stream>>>(a);
      break;
    case PKV_FP8_E4M3:
      e = cudaFuncSetAttribute(decode_simt_kernel<PKV_FP8_E4M3>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e == cudaSuccess)
        decode_simt_kernel<PKV_FP8_E4M3><<<grid, 32 * kWarps, smem, stream>>>(a);
      break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace pkv
