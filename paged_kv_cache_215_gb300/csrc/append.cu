// append.cu -- write new tokens' k and v into their pool slots, and the amax
// reduction behind the per-tensor FP8 scale.
//
// "The engineering truth of long-context inference 2026", section 2.2
// (append_token): block_id = pos // block_size, offset = pos % block_size,
// pool[table[block_id], 0/1, layer, :, offset, :] = k, v.  For an E4M3 pool
// ("Unlocking long context: engineering practice for million-token LLM
// inference", section 3.2, per-tensor FP8) every element is stored as
// e4m3(x / scale): IEEE fp32 division, round to nearest even, saturating
// finite overflow and +-Inf to +-448, NaN to 0x7F.
//
// One thread moves 8 consecutive elements of one (token, k|v, head) row:
// 16-byte loads of the input and a 16-byte (8-byte for E4M3) store into the
// slot, so a warp covers whole rows with coalesced accesses.
#include <algorithm>

#include "device.cuh"
#include "launch.h"

namespace pkv {
namespace {

template <int IN, int KV>
__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
  const int per_row = a.D / 8;
  const long long total = a.num_tokens * 2 * a.Hkv * per_row;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int d8 = (int)(i % per_row);
    long long r = i / per_row;
    const int h = (int)(r % a.Hkv);
    r /= a.Hkv;
    const int kv = (int)(r % 2);
    const long long tok = r / 2;
    const int s = a.seq_ids ? __ldg(a.seq_ids + tok) : (int)tok;
    if (s < 0 || s >= a.B) {
      record_error(a.status, PKV_EBOUNDS);
      continue;
    }
    const int pos = a.positions ? __ldg(a.positions + tok) : __ldg(a.seq_lens + s) - 1;
    if (pos < 0) continue;   // padding: no token for this sequence
    if (pos / a.BS >= a.max_blocks) {
      record_error(a.status, PKV_EBOUNDS);
      continue;
    }
    const int blk = __ldg(a.tables + (size_t)s * a.max_blocks + pos / a.BS);
    if (blk < 0 || blk >= a.num_blocks) {
      record_error(a.status, PKV_EBOUNDS);
      continue;
    }
    const size_t src = ((size_t)tok * a.Hkv + h) * a.D + (size_t)d8 * 8;
    const size_t dst =
        (((((size_t)blk * 2 + kv) * a.L + a.layer) * a.Hkv + h) * a.BS + pos % a.BS) * a.D +
        (size_t)d8 * 8;
    const void* in = kv ? a.v : a.k;
    store8_to_pool(a.pool, dst, KV, in, src, IN, kv ? a.v_scale : a.k_scale);
  }
}

template <int IN>
__global__ void __launch_bounds__(256) absmax_kernel(const void* x, int64_t n, float* amax) {
  float m = 0.f;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    float v;
    if constexpr (IN == PKV_F32) v = static_cast<const float*>(x)[i];
    else if constexpr (IN == PKV_F16) v = __half2float(static_cast<const __half*>(x)[i]);
    else v = __bfloat162float(static_cast<const __nv_bfloat16*>(x)[i]);
    m = fmaxf(m, fabsf(v));   // fmaxf ignores NaN
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<int*>(amax), __float_as_int(m));
}

template <int IN, int KV>
cudaError_t run_append(const AppendArgs& a, int grid, cudaStream_t stream) {
  append_kernel<IN, KV><<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
  const long long total = a.num_tokens * 2 * a.Hkv * (a.D / 8);
  if (total == 0) return cudaSuccess;
  const int grid = (int)std::min<long long>((total + 255) / 256, 1LL << 16);
  cudaError_t e;
  if (a.kv_dtype == PKV_FP8_E4M3) {
    switch (a.in_dtype) {
      case PKV_F32: e = run_append<PKV_F32, PKV_FP8_E4M3>(a, grid, stream); break;
      case PKV_F16: e = run_append<PKV_F16, PKV_FP8_E4M3>(a, grid, stream); break;
      case PKV_BF16: e = run_append<PKV_BF16, PKV_FP8_E4M3>(a, grid, stream); break;
      default: return cudaErrorInvalidValue;
    }
  } else if (a.kv_dtype == a.in_dtype) {
    switch (a.kv_dtype) {
      case PKV_F32: e = run_append<PKV_F32, PKV_F32>(a, grid, stream); break;
      case PKV_F16: e = run_append<PKV_F16, PKV_F16>(a, grid, stream); break;
      case PKV_BF16: e = run_append<PKV_BF16, PKV_BF16>(a, grid, stream); break;
      default: return cudaErrorInvalidValue;
    }
  } else {
    return cudaErrorInvalidValue;
  }
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t launch_absmax(const void* x, int dtype, int64_t n, float* amax, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), stream);
  if (e != cudaSuccess || n == 0) return e;
  const int grid = (int)std::min<long long>((n + 255) / 256, 1LL << 12);
  switch (dtype) {
    case PKV_F32: absmax_kernel<PKV_F32><<<grid, 256, 0, stream>>>(x, n, amax); break;
    case PKV_F16: absmax_kernel<PKV_F16><<<grid, 256, 0, stream>>>(x, n, amax); break;
    case PKV_BF16: absmax_kernel<PKV_BF16><<<grid, 256, 0, stream>>>(x, n, amax); break;
    default: return cudaErrorInvalidValue;
  }
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace pkv
