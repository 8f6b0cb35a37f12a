// merge.cu -- log-sum-exp merge of partial attention results.
//
// "Sequence-parallel engineering for long-context LLM inference: Ring Attention
// and distributed KV cache" (numerically stable incremental softmax) combines
// results over disjoint key ranges with the correction exp(m_prev - m_new);
// "The engineering truth of long-context inference 2026", section 3.1 carries
// the running max and sum.  Here each partial p of a row holds its normalised
// output O_p and the natural log-sum-exp lse_p of its scores, so with
// M = max_p lse_p and w_p = exp(lse_p - M) the row's result is
// sum_p w_p O_p / sum_p w_p.  A partial with lse_p = -inf (an empty key range)
// has weight 0; a row with no finite partial is 0.
//
// One CTA of 256 threads merges one row: its eight warps take every eighth
// partial, lanes split the head dimension, and the warps' sums meet in shared
// memory.
#include "device.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDL = 8;   // head_dim <= 256

// Partial i of the row: lse at lse[i * lse_stride], O at o[i * o_stride + d].
__device__ void merge_row(const float* __restrict__ lse, size_t lse_stride,
                          const float* __restrict__ o, size_t o_stride, int count, int D,
                          void* out, size_t out_off, int out_dtype) {
  __shared__ float red[kWarps][32 * kMaxDL];
  __shared__ float redw[kWarps];
  __shared__ float redm[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  float M = -INFINITY;
  for (int i = threadIdx.x; i < count; i += kThreads) M = fmaxf(M, lse[i * lse_stride]);
  M = warp_max(M);
  if (lane == 0) redm[warp] = M;
  __syncthreads();
  M = redm[0];
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, redm[w]);

  float acc[kMaxDL];
#pragma unroll
  for (int k = 0; k < kMaxDL; ++k) acc[k] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int i = warp; i < count; i += kWarps) {
      const float w = exp2f((lse[i * lse_stride] - M) * kLog2e);
      wsum += w;
      const float* op = o + i * o_stride;
#pragma unroll
      for (int k = 0; k < kMaxDL; ++k)
        if (lane + 32 * k < D) acc[k] = fmaf(w, op[lane + 32 * k], acc[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < kMaxDL; ++k)
    if (lane + 32 * k < D) red[warp][lane + 32 * k] = acc[k];
  if (lane == 0) redw[warp] = wsum;
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += kThreads) {
    float W = 0.f, v = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      W += redw[w];
      v += red[w][d];
    }
    store_from_float(out, out_off + d, out_dtype, W > 0.f ? v / W : 0.f);
  }
}

// Balanced-stream partials: unit u = (s, hg) has `count` partials in slots
// first .. first+count-1, each with HG*G heads; count 1 means the attention
// kernel already wrote the output.
__global__ void __launch_bounds__(kThreads) merge_units_kernel(const DecodeArgs a) {
  grid_dependency_wait();
  const int u = blockIdx.x, hl = blockIdx.y;
  const int2 info = a.unit_info[u];
  if (info.y == 1) return;
  const int HGG = a.HG * a.G;
  const int s = u / a.NHG, hg = u % a.NHG;
  const size_t out_off = ((size_t)s * a.Hq + (size_t)hg * HGG + hl) * a.D;
  const size_t row0 = (size_t)info.x * HGG + hl;
  merge_row(a.part_lse + row0, HGG, a.part_o + row0 * a.D, (size_t)HGG * a.D, info.y, a.D, a.out,
            out_off, a.out_dtype);
}

// [rows, S, D] partials (the layout of the public merge_partials).
__global__ void __launch_bounds__(kThreads)
    merge_rows_kernel(void* out, int out_dtype, const float* part_o, const float* part_lse, int S,
                      int D) {
  grid_dependency_wait();
  const size_t r = blockIdx.x;
  merge_row(part_lse + r * S, 1, part_o + r * S * D, D, S, D, out, r * D, out_dtype);
}

}  // namespace

static cudaError_t launch_pdl(const void* func, dim3 grid, void** args, bool pdl,
                              cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelExC(&cfg, func, args);
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t launch_merge_units(const DecodeArgs& a, bool pdl, cudaStream_t stream) {
  if (a.D > 32 * kMaxDL) return cudaErrorInvalidValue;
  const int units = a.B * a.NHG;
  if (units == 0) return cudaSuccess;
  DecodeArgs copy = a;
  void* args[] = {&copy};
  return launch_pdl(reinterpret_cast<const void*>(merge_units_kernel),
                    dim3(units, a.HG * a.G), args, pdl, stream);
}

cudaError_t launch_merge_rows(void* out, int out_dtype, const float* part_o, const float* part_lse,
                              int rows, int S, int D, bool pdl, cudaStream_t stream) {
  if (D > 32 * kMaxDL) return cudaErrorInvalidValue;
  if (rows == 0) return cudaSuccess;
  void* args[] = {&out, &out_dtype, &part_o, &part_lse, &S, &D};
  return launch_pdl(reinterpret_cast<const void*>(merge_rows_kernel), dim3(rows), args, pdl,
                    stream);
}

}  // namespace pkv
