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
// For few rows with many partials (one long sequence), one CTA of 512 threads
// merges one row: the partials' weights are computed once into shared memory,
// each of the sixteen warps takes every sixteenth partial with four rows in
// flight, lanes split the head dimension, and the warps' sums meet in shared
// memory.  For many rows with few partials each, one warp merges one row.
#include "device.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxD = 256;
constexpr int kChunk = 1024;   // partial weights staged in shared memory per pass
constexpr int kUnroll = 4;     // partial rows in flight per warp

// Partial i of the row: lse at lse[i * lse_stride], O at o[i * o_stride + d].
// Vector path: D % 4 == 0 and 16-byte aligned rows; lane g holds columns 4g..4g+3
// (and 4(g+32)..) of one partial row per load, so a warp reads a whole row.
__device__ void merge_row(const float* __restrict__ lse, size_t lse_stride,
                          const float* __restrict__ o, size_t o_stride, int count, int D,
                          void* out, size_t out_off, int out_dtype, float* out_lse = nullptr) {
  __shared__ float wts[kChunk];
  __shared__ float red[kWarps][kMaxD];
  __shared__ float redw[kWarps];
  __shared__ float redm[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  float M = -INFINITY;
  for (int i = threadIdx.x; i < count; i += kThreads) M = fmaxf(M, lse[i * lse_stride]);
  M = warp_max(M);
  if (lane == 0) redm[warp] = M;
  __syncthreads();
  M = redm[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, redm[w]);

  const bool vec = (D % 4) == 0 && (o_stride % 4) == 0 &&
                   (reinterpret_cast<uintptr_t>(o) & 15u) == 0;
  const int groups = vec ? D / 4 : 0;
  float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
  float accs[kMaxD / 32];
#pragma unroll
  for (int k = 0; k < kMaxD / 32; ++k) accs[k] = 0.f;
  float wsum = 0.f;

  if (M != -INFINITY) {
    for (int base = 0; base < count; base += kChunk) {
      const int n = min(kChunk, count - base);
      __syncthreads();
      for (int i = threadIdx.x; i < n; i += kThreads)
        wts[i] = exp2f((lse[(size_t)(base + i) * lse_stride] - M) * kLog2e);
      __syncthreads();
      for (int i0 = warp; i0 < n; i0 += kWarps * kUnroll) {
        if (vec) {
          float4 v[kUnroll][2];
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int i = i0 + u * kWarps;
            const float4* row = reinterpret_cast<const float4*>(o + (size_t)(base + i) * o_stride);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int g = lane + 32 * h;
              v[u][h] = (i < n && g < groups) ? row[g] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int i = i0 + u * kWarps;
            const float w = i < n ? wts[i] : 0.f;
            wsum += w;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              acc[h].x = fmaf(w, v[u][h].x, acc[h].x);
              acc[h].y = fmaf(w, v[u][h].y, acc[h].y);
              acc[h].z = fmaf(w, v[u][h].z, acc[h].z);
              acc[h].w = fmaf(w, v[u][h].w, acc[h].w);
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int i = i0 + u * kWarps;
            if (i >= n) break;
            const float w = wts[i];
            wsum += w;
            const float* row = o + (size_t)(base + i) * o_stride;
#pragma unroll
            for (int k = 0; k < kMaxD / 32; ++k)
              if (lane + 32 * k < D) accs[k] = fmaf(w, row[lane + 32 * k], accs[k]);
          }
        }
      }
    }
  }
  if (vec) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int g = lane + 32 * h;
      if (g < groups) {
        red[warp][4 * g + 0] = acc[h].x;
        red[warp][4 * g + 1] = acc[h].y;
        red[warp][4 * g + 2] = acc[h].z;
        red[warp][4 * g + 3] = acc[h].w;
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kMaxD / 32; ++k)
      if (lane + 32 * k < D) red[warp][lane + 32 * k] = accs[k];
  }
  if (lane == 0) redw[warp] = wsum;
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += kThreads) {
    float W = 0.f, v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      W += redw[w];
      v += red[w][d];
    }
    store_from_float(out, out_off + d, out_dtype, W > 0.f ? v / W : 0.f);
    // the row's natural log-sum-exp: M + ln(sum of exp(lse_p - M))
    if (out_lse && d == 0) *out_lse = W > 0.f ? M + __logf(W) : -INFINITY;
  }
}

// A unit's (first slot, count) record names slots inside the workspace.  The
// attention kernel writes every record before the merge runs; a record outside
// that range can only be left over from a call whose attention kernel gave up
// (a bounded wait ran out): its row is skipped instead of read out of range.
__device__ __forceinline__ bool info_ok(const DecodeArgs& a, int2 info) {
  return info.x >= 0 && info.y >= 0 && (long long)info.x + info.y <= (long long)a.slots;
}

// Balanced-stream partials: unit u = (s, hg) has `count` partials in slots
// first .. first+count-1, each with HG*R rows (R = q_len * G); count 1 means the
// attention kernel already wrote the output.
__global__ void __launch_bounds__(kThreads) merge_units_kernel(const DecodeArgs a) {
  // the next launch may be scheduled now (it waits for this grid before it
  // writes anything this grid reads); this grid's own inputs come first
  grid_launch_dependents();
  grid_dependency_wait();
  const int u = blockIdx.x, hl = blockIdx.y;
  const int2 info = a.unit_info[u];
  if (info.y == 1 && !a.out_lse) return;       // the attention kernel wrote this row
  if (!info_ok(a, info)) {
    if (hl == 0 && threadIdx.x == 0) record_error(a.status, PKV_EBOUNDS);
    return;
  }
  // row hl of a unit: KV head w of the group, column r = i * G + g (query token i, head g)
  const int HGR = a.HG * a.R;
  const int s = u / a.NHG, hg = u % a.NHG;
  const int w = hl / a.R, r = hl % a.R;
  const int i = r / a.G, g = r % a.G;
  const size_t q_row = ((size_t)s * a.q_len + i) * a.Hq + (size_t)(hg * a.HG + w) * a.G + g;
  const size_t row0 = (size_t)info.x * HGR + hl;
  merge_row(a.part_lse + row0, HGR, a.part_o + row0 * a.D, (size_t)HGR * a.D, info.y, a.D, a.out,
            q_row * a.D, a.out_dtype, a.out_lse ? a.out_lse + q_row : nullptr);
}

// Many rows, few partials each (multi-token decode, large batches): one warp per
// row, 8 rows per CTA; lane l holds columns 4l .. 4l+3 (+128 ...), every lane
// reads each partial's lse (a broadcast) and computes its weight.
constexpr int kRowsPerCta = 8;
// partial rows the shared-prefix merge's warps load at once (a row there merges
// the decode's partials and every split of the prefix pass: about 20 on the
// long shared documents)
constexpr int kInFlight = 16;
__global__ void __launch_bounds__(32 * kRowsPerCta) merge_units_warp_kernel(const DecodeArgs a) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int HGR = a.HG * a.R;
  const long long row = (long long)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (row >= (long long)a.B * a.NHG * HGR) return;
  const int lane = threadIdx.x & 31;
  const int u = (int)(row / HGR), hl = (int)(row % HGR);
  const int2 info = a.unit_info[u];
  if (info.y == 1 && !a.out_lse) return;        // the attention kernel wrote this row
  if (!info_ok(a, info)) {
    if (hl == 0 && lane == 0) record_error(a.status, PKV_EBOUNDS);
    return;
  }
  const int s = u / a.NHG, hg = u % a.NHG;
  const int w = hl / a.R, r = hl % a.R;
  const int i = r / a.G, g = r % a.G;
  const size_t q_row = ((size_t)s * a.q_len + i) * a.Hq + (size_t)(hg * a.HG + w) * a.G + g;
  const size_t row0 = (size_t)info.x * HGR + hl;
  float M = -INFINITY;
  for (int p = lane; p < info.y; p += 32) M = fmaxf(M, a.part_lse[row0 + (size_t)p * HGR]);
  M = warp_max(M);
  for (int d0 = 4 * lane; d0 < a.D; d0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float W = 0.f;
    if (M != -INFINITY) {
      for (int p = 0; p < info.y; ++p) {
        const size_t pr = row0 + (size_t)p * HGR;
        const float wt = exp2f((a.part_lse[pr] - M) * kLog2e);
        const float4 v = *reinterpret_cast<const float4*>(a.part_o + pr * a.D + d0);
        W += wt;
        acc.x = fmaf(wt, v.x, acc.x);
        acc.y = fmaf(wt, v.y, acc.y);
        acc.z = fmaf(wt, v.z, acc.z);
        acc.w = fmaf(wt, v.w, acc.w);
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    store_from_float(a.out, q_row * a.D + d0 + 0, a.out_dtype, acc.x * inv);
    store_from_float(a.out, q_row * a.D + d0 + 1, a.out_dtype, acc.y * inv);
    store_from_float(a.out, q_row * a.D + d0 + 2, a.out_dtype, acc.z * inv);
    store_from_float(a.out, q_row * a.D + d0 + 3, a.out_dtype, acc.w * inv);
    if (a.out_lse && d0 == 0) a.out_lse[q_row] = W > 0.f ? M + __logf(W) : -INFINITY;
  }
}

// [rows, S, D] partials (the layout of the public merge_partials).
__global__ void __launch_bounds__(kThreads)
    merge_rows_kernel(void* out, int out_dtype, const float* part_o, const float* part_lse, int S,
                      int D) {
  grid_launch_dependents();
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
  if (a.D > kMaxD) return cudaErrorInvalidValue;
  const int units = a.B * a.NHG;
  if (units == 0) return cudaSuccess;
  DecodeArgs copy = a;
  void* args[] = {&copy};
  const long long rows = (long long)units * a.HG * a.R;
  // many rows (each with few partials): a warp per row; few rows (long sequences,
  // many partials each): a CTA per row
  if (rows >= 512 && a.D % 4 == 0) {
    const long long ctas = (rows + kRowsPerCta - 1) / kRowsPerCta;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(32 * kRowsPerCta);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(merge_units_warp_kernel),
                                        args);
    if (e == cudaSuccess) count_launch();
    return e;
  }
  return launch_pdl(reinterpret_cast<const void*>(merge_units_kernel),
                    dim3(units, a.HG * a.R), args, pdl, stream);
}

cudaError_t launch_merge_rows(void* out, int out_dtype, const float* part_o, const float* part_lse,
                              int rows, int S, int D, bool pdl, cudaStream_t stream) {
  if (D > kMaxD) return cudaErrorInvalidValue;
  if (rows == 0) return cudaSuccess;
  void* args[] = {&out, &out_dtype, &part_o, &part_lse, &S, &D};
  return launch_pdl(reinterpret_cast<const void*>(merge_rows_kernel), dim3(rows), args, pdl,
                    stream);
}

}  // namespace pkv

// ---------------------------------------------------------------- shared-prefix decode
namespace pkv {
namespace {

// One CTA per row (a thread per column, D <= 256): the decode's `count`
// partials of the row (slots first .. first+count-1, stride HG*R rows) and the
// ext_count partials computed over the shared prefix, combined by log-sum-exp
// as in merge_row.  The weights of up to kExtChunk partials at a time go to
// shared memory; each thread then sums its column with eight partial rows in
// flight.
constexpr int kExtChunk = 512;
__global__ void __launch_bounds__(128) merge_units_ext_kernel(const DecodeArgs a) {
  __shared__ float wts[kExtChunk];
  __shared__ const float* rowp[kExtChunk];
  __shared__ float red[4];
  // chained behind the attention kernel: it and the prefix pass have finished
  // (and their partials are visible) once past this wait
  grid_launch_dependents();
  grid_dependency_wait();
  const int HGR = a.HG * a.R;
  const long long row = blockIdx.x;
  const int u = (int)(row / HGR), hl = (int)(row % HGR);
  int2 info = a.unit_info[u];
  if (!info_ok(a, info)) {
    if (hl == 0 && threadIdx.x == 0) record_error(a.status, PKV_EBOUNDS);
    info = make_int2(0, 0);                                   // the prefix partials alone
  }
  const int s = u / a.NHG, hg = u % a.NHG;
  const int w = hl / a.R, r = hl % a.R;
  const int i = r / a.G, g = r % a.G;
  const size_t q_row = ((size_t)s * a.q_len + i) * a.Hq + (size_t)(hg * a.HG + w) * a.G + g;
  const size_t rows = (size_t)a.B * a.q_len * a.Hq;           // rows of one ext partial set
  const size_t row0 = (size_t)info.x * HGR + hl;
  const int total = info.y + a.ext_count;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // partial p < count: the decode's; else the prefix split p - count
  auto lse_of = [&](int p) {
    return p < info.y ? a.part_lse[row0 + (size_t)p * HGR]
                      : a.ext_lse[(size_t)(p - info.y) * rows + q_row];
  };
  auto o_of = [&](int p) {
    return p < info.y ? a.part_o + (row0 + (size_t)p * HGR) * a.D
                      : a.ext_o + ((size_t)(p - info.y) * rows + q_row) * a.D;
  };
  float M = -INFINITY;
  for (int p = threadIdx.x; p < total; p += blockDim.x) M = fmaxf(M, lse_of(p));
  M = warp_max(M);
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  float acc[2] = {0.f, 0.f}, W = 0.f;
  for (int base = 0; base < total && M != -INFINITY; base += kExtChunk) {
    const int n = min(kExtChunk, total - base);
    __syncthreads();
    for (int p = threadIdx.x; p < n; p += blockDim.x) {
      const float wt = exp2f((lse_of(base + p) - M) * kLog2e);
      wts[p] = wt;
      rowp[p] = o_of(base + p);
      W += wt;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int d = threadIdx.x + 128 * h;
      if (d >= a.D) continue;
      int p = 0;
      for (; p + 8 <= n; p += 8) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = rowp[p + k][d];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[h] = fmaf(wts[p + k], v[k], acc[h]);
      }
      for (; p < n; ++p) acc[h] = fmaf(wts[p], rowp[p][d], acc[h]);
    }
  }
  W = warp_sum(W);
  __syncthreads();
  if (lane == 0) red[warp] = W;
  __syncthreads();
  W = (red[0] + red[1]) + (red[2] + red[3]);
  const float inv = W > 0.f ? 1.f / W : 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int d = threadIdx.x + 128 * h;
    if (d < a.D) store_from_float(a.out, q_row * a.D + d, a.out_dtype, acc[h] * inv);
  }
}

// Many rows (head_dim 128): one warp per row, 8 rows per CTA.  Lane l holds
// columns 4l .. 4l+3; the partials' weights are computed 32 at a time, one per
// lane, and broadcast by shuffle while kInFlight partial rows are in flight.
__global__ void __launch_bounds__(256) merge_units_ext_warp_kernel(const DecodeArgs a) {
  grid_launch_dependents();
  grid_dependency_wait();
  const int HGR = a.HG * a.R;
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= (long long)a.B * a.NHG * HGR) return;
  const int lane = threadIdx.x & 31;
  const int u = (int)(row / HGR), hl = (int)(row % HGR);
  int2 info = a.unit_info[u];
  if (!info_ok(a, info)) {
    if (hl == 0 && lane == 0) record_error(a.status, PKV_EBOUNDS);
    info = make_int2(0, 0);                                   // the prefix partials alone
  }
  const int s = u / a.NHG, hg = u % a.NHG;
  const int w = hl / a.R, r = hl % a.R;
  const int i = r / a.G, g = r % a.G;
  const size_t q_row = ((size_t)s * a.q_len + i) * a.Hq + (size_t)(hg * a.HG + w) * a.G + g;
  const size_t rows = (size_t)a.B * a.q_len * a.Hq;           // rows of one ext partial set
  const size_t row0 = (size_t)info.x * HGR + hl;
  const int total = info.y + a.ext_count;
  auto lse_of = [&](int p) {
    return p < info.y ? a.part_lse[row0 + (size_t)p * HGR]
                      : a.ext_lse[(size_t)(p - info.y) * rows + q_row];
  };
  auto o_of = [&](int p) {
    return p < info.y ? a.part_o + (row0 + (size_t)p * HGR) * a.D
                      : a.ext_o + ((size_t)(p - info.y) * rows + q_row) * a.D;
  };
  // the first kInFlight partial rows are requested before the lse maximum is
  // known, so that their loads overlap the lse round trip
  float4 v[kInFlight];
#pragma unroll
  for (int e = 0; e < kInFlight; ++e)
    v[e] = e < total ? reinterpret_cast<const float4*>(o_of(e))[lane]
                     : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = -INFINITY;
  for (int p = lane; p < total; p += 32) M = fmaxf(M, lse_of(p));
  M = warp_max(M);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  if (M != -INFINITY) {
    for (int base = 0; base < total; base += 32) {
      const int cnt = min(32, total - base);
      const float wl = lane < cnt ? exp2f((lse_of(base + lane) - M) * kLog2e) : 0.f;
      for (int k = 0; k < cnt; k += kInFlight) {
        float wt[kInFlight];
#pragma unroll
        for (int e = 0; e < kInFlight; ++e) {
          wt[e] = __shfl_sync(0xffffffffu, wl, (k + e) & 31);
          if (base > 0 || k > 0)                     // the first rows are in already
            v[e] = k + e < cnt ? reinterpret_cast<const float4*>(o_of(base + k + e))[lane]
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int e = 0; e < kInFlight; ++e) {
          if (k + e >= cnt) break;
          W += wt[e];
          acc.x = fmaf(wt[e], v[e].x, acc.x);
          acc.y = fmaf(wt[e], v[e].y, acc.y);
          acc.z = fmaf(wt[e], v[e].z, acc.z);
          acc.w = fmaf(wt[e], v[e].w, acc.w);
        }
      }
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  const size_t o = q_row * a.D + 4 * lane;
  store_from_float(a.out, o + 0, a.out_dtype, acc.x * inv);
  store_from_float(a.out, o + 1, a.out_dtype, acc.y * inv);
  store_from_float(a.out, o + 2, a.out_dtype, acc.z * inv);
  store_from_float(a.out, o + 3, a.out_dtype, acc.w * inv);
}

// The shared-prefix check, one thread per (sequence, prefix entry): each
// sequence's prefix length is whole blocks within its length and the shared
// list, and its table starts with the shared blocks; a mismatch is reported as
// PKV_EINVAL (the decode then reads that sequence from its first token).  Nothing
// launched after it reads what it writes, so the next launch may start at once.
__global__ void prefix_check_kernel(const int32_t* tables, int max_blocks, const int32_t* seq_lens,
                                    const int32_t* prefix_table, int prefix_blocks,
                                    const int32_t* prefix_lens, int prefix_len_max, int B, int BS,
                                    int32_t* status) {
  grid_launch_dependents();
  const int s = blockIdx.y;
  if (s >= B) return;
  const int n = seq_lens[s], pl = prefix_lens[s];
  const bool bad = pl < 0 || pl % BS != 0 || pl > prefix_len_max || pl > n ||
                   pl / BS > prefix_blocks || n > max_blocks * BS;
  if (bad && threadIdx.x == 0 && blockIdx.x == 0) record_error(status, PKV_EINVAL);
  const int pb = bad ? 0 : pl / BS;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < pb; j += gridDim.x * blockDim.x)
    if (tables[(size_t)s * max_blocks + j] != prefix_table[j])
      record_error(status, PKV_EINVAL);                     // not the shared prefix
}

}  // namespace

cudaError_t launch_merge_units_ext(const DecodeArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.B * a.NHG * a.HG * a.R;
  if (rows == 0) return cudaSuccess;
  if (rows > 0x7fffffffLL || a.D > 256) return cudaErrorInvalidValue;
  const bool warp = a.D == 128;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(warp ? (rows + 7) / 8 : rows));
  cfg.blockDim = dim3(warp ? 256 : 128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;              // chained behind a chained attention launch
  DecodeArgs copy = a;
  void* args[] = {&copy};
  const cudaError_t e = cudaLaunchKernelExC(
      &cfg, warp ? reinterpret_cast<const void*>(merge_units_ext_warp_kernel)
                 : reinterpret_cast<const void*>(merge_units_ext_kernel), args);
  if (e == cudaSuccess) count_launch();
  return e;
}

cudaError_t launch_prefix_check(const int32_t* tables, int max_blocks, const int32_t* seq_lens,
                                const int32_t* prefix_table, int prefix_blocks,
                                const int32_t* prefix_lens, int prefix_len_max, int B, int BS,
                                int32_t* status, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const int span = std::min(max_blocks, prefix_blocks);
  const int gx = std::max(1, (span + 255) / 256);
  prefix_check_kernel<<<dim3(gx > 64 ? 64 : gx, B), 256, 0, stream>>>(
      tables, max_blocks, seq_lens, prefix_table, prefix_blocks, prefix_lens, prefix_len_max, B, BS,
      status);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace pkv
