// append.cu -- write new tokens' k and v into their pool slots, the amax
// reduction behind the per-tensor FP8 scale, and the scale itself.
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
    float sc = kv ? a.v_scale : a.k_scale;
    if (KV == PKV_FP8_E4M3 && a.block_scales)
      sc = a.block_scales[(((size_t)blk * 2 + kv) * a.L + a.layer) * a.Hkv + h];
    store8_to_pool(a.pool, dst, KV, in, src, IN, sc);
  }
}

// Scale group of token `tok`: a.group_tokens consecutive positions of its
// sequence (a multiple of the block size), named by its first block.  Returns
// the tile of that first block for (kv, h), or -1 when the token is skipped or
// out of range.
__device__ __forceinline__ long long tile_of(const AppendArgs& a, long long tok, int kv, int h) {
  const int s = a.seq_ids ? __ldg(a.seq_ids + tok) : (int)tok;
  const int pos = __ldg(a.positions + tok);
  if (pos < 0 || s < 0 || s >= a.B || pos / a.BS >= a.max_blocks) return -1;
  const int blk = __ldg(a.tables + (size_t)s * a.max_blocks + pos / a.BS);
  const int lead = __ldg(a.tables + (size_t)s * a.max_blocks +
                         (pos / a.group_tokens) * (a.group_tokens / a.BS));
  if (blk < 0 || blk >= a.num_blocks || lead < 0 || lead >= a.num_blocks) return -1;
  return (((long long)lead * 2 + kv) * a.L + a.layer) * a.Hkv + h;
}

// Block-wise scales, pass 1: mark the tile of every group the tokens land in
// (its first block's) with -0.0.
__global__ void __launch_bounds__(256) scales_mark_kernel(const AppendArgs a, float* scales) {
  const long long total = a.num_tokens * 2 * a.Hkv;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int h = (int)(i % a.Hkv), kv = (int)((i / a.Hkv) % 2);
    const long long t = tile_of(a, i / (2 * a.Hkv), kv, h);
    if (t >= 0) scales[t] = -0.0f;
  }
}

// Pass 2: fold |x| of every element into its tile as -amax (sign bit set): as
// unsigned integers, 0x80000000 | bits(|x|) orders like |x|, and the -0.0 marker
// is the smallest such value.
template <int IN>
__global__ void __launch_bounds__(256) scales_amax_kernel(const AppendArgs a, float* scales) {
  const long long total = a.num_tokens * 2 * a.Hkv * a.D;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int d = (int)(i % a.D);
    long long r = i / a.D;
    const int h = (int)(r % a.Hkv);
    r /= a.Hkv;
    const int kv = (int)(r % 2);
    const long long tok = r / 2;
    const long long t = tile_of(a, tok, kv, h);
    if (t < 0) continue;
    const float x = fabsf(load_as_float(kv ? a.v : a.k, ((size_t)tok * a.Hkv + h) * a.D + d, IN));
    if (!isfinite(x)) continue;   // NaN and +-Inf do not set a scale
    atomicMax(reinterpret_cast<unsigned int*>(scales) + t, 0x80000000u | __float_as_uint(x));
  }
}

// Pass 3: every tile holding -amax becomes amax / 448 (IEEE fp32 division;
// amax 0 -> 1); pass 4 copies it to the group's other blocks.
__global__ void __launch_bounds__(256) scales_finish_kernel(float* scales, long long tiles) {
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < tiles;
       t += (long long)gridDim.x * blockDim.x) {
    const unsigned int u = __float_as_uint(scales[t]);
    if (u & 0x80000000u) {
      const float amax = __uint_as_float(u & 0x7fffffffu);
      scales[t] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    }
  }
}

// Pass 4 (groups of several blocks): every block of a token's group takes the
// scale of the group's first block.  Tokens of one group write the same value.
__global__ void __launch_bounds__(256) scales_spread_kernel(const AppendArgs a, float* scales) {
  const int per = a.group_tokens / a.BS;
  const long long total = a.num_tokens * 2 * a.Hkv * (per - 1);
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int m = 1 + (int)(i % (per - 1));             // member of the group after the first
    long long r = i / (per - 1);
    const int h = (int)(r % a.Hkv);
    r /= a.Hkv;
    const int kv = (int)(r % 2);
    const long long tok = r / 2;
    const long long lt = tile_of(a, tok, kv, h);
    if (lt < 0) continue;
    const int s = a.seq_ids ? __ldg(a.seq_ids + tok) : (int)tok;
    const int e = (__ldg(a.positions + tok) / a.group_tokens) * per + m;
    if (e >= a.max_blocks) continue;
    const int blk = __ldg(a.tables + (size_t)s * a.max_blocks + e);
    if (blk < 0 || blk >= a.num_blocks) continue;        // not allocated yet
    scales[(((long long)blk * 2 + kv) * a.L + a.layer) * a.Hkv + h] = scales[lt];
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
    if (isfinite(v)) m = fmaxf(m, fabsf(v));   // NaN and +-Inf do not set a scale
  }
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<int*>(amax), __float_as_int(m));
}

// Per-tensor scale of a tensor held in n pieces: amax = the largest of the
// pieces' amax values, scale = amax / 448 (IEEE fp32 division), 1 when amax is 0.
__global__ void fp8_scale_kernel(const float* amax, int n, float* scale) {
  float m = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, amax[i]);
  m = warp_max(m);
  if (threadIdx.x == 0) *scale = m > 0.f ? __fdiv_rn(m, 448.f) : 1.f;
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

cudaError_t launch_block_scales(const AppendArgs& a, float* scales, cudaStream_t stream) {
  const long long tiles = (long long)a.num_blocks * 2 * a.L * a.Hkv;
  if (a.num_tokens > 0) {
    const long long t1 = a.num_tokens * 2 * a.Hkv, t2 = t1 * a.D;
    scales_mark_kernel<<<(int)std::min<long long>((t1 + 255) / 256, 1LL << 16), 256, 0, stream>>>(
        a, scales);
    const int g2 = (int)std::min<long long>((t2 + 255) / 256, 1LL << 16);
    switch (a.in_dtype) {
      case PKV_F32: scales_amax_kernel<PKV_F32><<<g2, 256, 0, stream>>>(a, scales); break;
      case PKV_F16: scales_amax_kernel<PKV_F16><<<g2, 256, 0, stream>>>(a, scales); break;
      case PKV_BF16: scales_amax_kernel<PKV_BF16><<<g2, 256, 0, stream>>>(a, scales); break;
      default: return cudaErrorInvalidValue;
    }
  }
  scales_finish_kernel<<<(int)std::min<long long>((tiles + 255) / 256, 1LL << 16), 256, 0,
                         stream>>>(scales, tiles);
  const int per = a.group_tokens / a.BS;
  const bool spread = a.num_tokens > 0 && per > 1;
  if (spread) {
    const long long t4 = a.num_tokens * 2 * a.Hkv * (per - 1);
    scales_spread_kernel<<<(int)std::min<long long>((t4 + 255) / 256, 1LL << 16), 256, 0,
                           stream>>>(a, scales);
  }
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess)
    for (int i = 0; i < (a.num_tokens > 0 ? 3 : 1) + (spread ? 1 : 0); ++i) count_launch();
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

cudaError_t launch_fp8_scale(const float* amax, int n, float* scale, cudaStream_t stream) {
  fp8_scale_kernel<<<1, 32, 0, stream>>>(amax, n, scale);
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace pkv
