// decode_mma.cuh -- paged decode attention for sm_103a: persistent CTAs, TMA
// page loads into a shared-memory ring, GQA scores and P.V on the tensor cores
// (mma.sync m16n8k16), online softmax in registers, split partials merged by
// log-sum-exp.
//
// What it computes ("Unlocking long context: engineering practice for
// million-token LLM inference", sections 4.1 and 5.1; long-context article at
// mhpn.cn, sections 1.1 and 3.2): for one new query token per sequence, each
// query head h attends over every cached token of its sequence through KV head
// h / G: out = softmax(scale * q K^T) V.  Token j of sequence s lives in block
// table[s][j / bs], slot j % bs of the pool [NB, 2, L, Hkv, bs, D] ("The
// engineering truth of long-context inference 2026", section 2.2).  The key
// range is streamed block by block with the online softmax of that page's
// section 3.1 (running max m, running sum l, rescale by exp(m_old - m_new)), and
// partial results over disjoint key ranges are combined by the log-sum-exp
// correction of "Sequence-parallel engineering for long-context LLM
// inference" (numerically stable incremental softmax).
//
// Layout of the work.  A CTA owns HG consecutive KV heads of one sequence at a
// time; a unit u = (sequence s, head group hg) has nb = ceil(n_s / bs) blocks.
// In balanced mode the units' blocks form one stream of T blocks that is cut
// into gridDim.x equal contiguous runs, one per CTA, so every SM moves the
// same number of bytes; a unit spanning several runs leaves one partial per
// run (slot = cta + u) and the merge kernel combines them.  In fixed mode the
// grid is (S, units) and CTA (p, u) takes partition p of unit u.
//
// Roles inside a CTA: warps 0..HG-1 are consumers, one per KV head; warp HG is
// the producer.  Per block the producer issues TMA loads of the K and V tiles
// of all HG heads (they are contiguous in the pool: HG*bs rows of D elements)
// into one stage of the ring, with 128-byte swizzling so that ldmatrix reads
// are free of bank conflicts.  Consumers compute S^T = K q^T with K as the
// 16-token A operand and the G query heads as the 8-column B operand, run the
// online softmax on the accumulator fragment, transpose P with movmatrix and
// accumulate O^T += V^T P^T with V read by ldmatrix.trans.  E4M3 pages are
// converted to f16 in registers (exact) and the per-tensor scales are applied
// to the scores and to the output.
#pragma once
#include <algorithm>

#include "device.cuh"
#include "launch.h"

namespace pkv {
namespace mma {

constexpr int kD = 128;            // head_dim of this kernel
constexpr int kMaxHG = 8;          // consumer warps per CTA
constexpr int kLineBytes = 128;    // one swizzled shared-memory line per row and region

template <int KVT>
struct KvTraits;
template <>
struct KvTraits<PKV_BF16> {
  static constexpr bool kFp8 = false, kBf16Mma = true;
  static constexpr int kRegions = 2;   // K and V each split into two 64-column halves
};
template <>
struct KvTraits<PKV_F16> {
  static constexpr bool kFp8 = false, kBf16Mma = false;
  static constexpr int kRegions = 2;
};
template <>
struct KvTraits<PKV_FP8_E4M3> {
  static constexpr bool kFp8 = true, kBf16Mma = false;
  static constexpr int kRegions = 1;   // 128 one-byte columns fill one line
};

// First token of sequence s that a shared-prefix launch (kOff, a.len_off set)
// reads: the end of the sequence's shared prefix, whole blocks; a prefix the
// check before the launch reported bad reads the sequence from token 0.
__device__ __forceinline__ int first_token(const DecodeArgs& a, int s, int n) {
  const int o = __ldg(a.len_off + s);
  return (o < 0 || o > n || o % a.BS != 0) ? 0 : o;
}

// Iteration state over the blocks a CTA processes; identical in every warp.
struct Cursor {
  int s, hg, j, n, nb;     // unit (s, hg), local block j, tokens and blocks of s
  int j0;                  // local block where the current piece began
  long long gb;            // global block index of block j in balanced mode
  long long remaining;     // blocks left in this CTA's run
};

template <bool kOff>
__device__ __forceinline__ int clamp_len(const DecodeArgs& a, int s) {
  int n = __ldg(a.seq_lens + s);
  int cap = a.max_blocks * a.BS;
  if (n < 0 || n > cap) {
    record_error(a.status, PKV_EBOUNDS);
    n = n < 0 ? 0 : cap;
  }
  if constexpr (kOff) n -= first_token(a, s, n);
  return n;
}

__device__ __forceinline__ int blocks_of(int n, int BS) { return (n + BS - 1) / BS; }

// Move to the next block; crosses into the next non-empty unit when needed.
template <bool kOff>
__device__ __forceinline__ void cursor_next(Cursor& c, const DecodeArgs& a) {
  ++c.j;
  ++c.gb;
  --c.remaining;
  if (c.j == c.nb && c.remaining > 0) {
    c.j = 0;
    c.j0 = 0;
    if (++c.hg == a.NHG) {
      c.hg = 0;
      do {
        ++c.s;
        c.n = clamp_len<kOff>(a, c.s);
        c.nb = blocks_of(c.n, a.BS);
      } while (c.nb == 0);
    }
  }
}

// CTA of the balanced stream that owns global block b: the largest c with
// floor(c * T / P) <= b, where P = min(grid, T) CTAs take part.
__device__ __forceinline__ long long owner_of(long long b, long long T, long long P) {
  return ((b + 1) * P - 1) / T;
}

struct SmemHeader {
  uint64_t full[16];
  uint64_t empty[16];
  float bscale[16][2][kMaxHG];   // E4M3 block-wise scales of each stage's tiles (K, V)
  long long total, gb0, gb1;
  int s, hg, j;
  volatile int abort_flag;
};

// ---------------------------------------------------------------- consumer math
//
// A warp owns one KV head.  Its query rows are R = q_len * G (query token i,
// head g) pairs, row r = i * G + g, held as NT n-tiles of 8 columns of the MMA
// B operand.  Query token i sits at position n - q_len + i of its sequence and
// sees keys 0 .. that position (causal within the chunk; q_len = 1 is plain
// decode).

template <int KVT, int BS, int NT, bool kCausal>
struct Consumer {
  using T = KvTraits<KVT>;
  static constexpr int kTiles = BS / 16;
  static constexpr bool kSplitP = T::kBf16Mma;   // bf16 P is split into hi + lo parts
  // f16 P (f16 and E4M3 pools) is computed as 2^(s - m + kPOff): the largest
  // weight of a block is 2^kPOff instead of 1, so weights down to 2^-28 of the
  // running maximum stay normal f16 numbers (a long tail of small weights would
  // otherwise round in f16's subnormal range); the factor cancels in O / l.
  static constexpr float kPOff = kSplitP ? 0.f : 14.f;

  uint32_t qf[NT][8][2];   // B fragments of the query rows (8 k-steps of 16)
  float acc[8][NT][4];     // O^T fragments: 8 tiles of 16 d x 8 rows, per n-tile
  float m[NT][2], l[NT][2];// running max (log2 units) and per-thread partial sums
  int lim[NT][2];          // last key position each of the thread's columns may see
  // E4M3 with block-wise scales: acc is held in units of 2^ev_ref_, the largest
  // power-of-two exponent of the V block scales seen in the current piece, and
  // each block's P carries its scale's remaining factor (at most 2), so that
  // P x scale never leaves f16's range whatever the scales' magnitudes.
  int ev_ref_;

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[i][nt][k] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
    }
    ev_ref_ = -100000;
  }

  // Block-wise E4M3 scales: split vs_b = mant x 2^ev (mant in [1, 2)); a block
  // whose exponent exceeds the piece's reference raises it, and acc (in units of
  // the old reference) is rescaled by 2^(old - new) through *acc_f.  Returns the
  // factor P carries for this block: mant x 2^(ev - reference) <= 2.
  __device__ __forceinline__ float v_block_factor(float vs_b, float* acc_f) {
    int ev;
    const float mant = 2.f * frexpf(vs_b, &ev);
    --ev;
    if (ev > ev_ref_) {
      *acc_f = ldexpf(1.f, max(ev_ref_ - ev, -300));   // 0 for the piece's first block
      ev_ref_ = ev;
    }
    return ldexpf(mant, max(ev - ev_ref_, -300));
  }


  // q row of column r (query token r / G, head r % G of this KV head), -1 if padding.
  __device__ __forceinline__ static long long q_row(const DecodeArgs& a, int s, int hkv, int r) {
    if (r >= a.R) return -1;
    const int i = r / a.G, g = r - (r / a.G) * a.G;
    return ((long long)s * a.q_len + i) * a.Hq + (long long)hkv * a.G + g;
  }

  __device__ __forceinline__ void load_q(const DecodeArgs& a, int s, int n, int hkv, int lane) {
    if constexpr (NT == 1 && !kCausal) {
      load_q_decode(a, s, hkv, lane);
      return;
    }
    const int c = lane & 3;
    float qscale = 1.f;
    if constexpr (T::kFp8) {
      // E4M3 pools run f16 MMAs: q x 2^e with the warp's largest |q| over all its
      // rows setting e (f16_fit_exponent), and 2^-e folded into the softmax scale
      float amax = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const long long qr = q_row(a, s, hkv, nt * 8 + (lane >> 2));
        if (qr < 0) continue;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
#pragma unroll
          for (int i = 0; i < 4; ++i)
            amax = fmaxf(amax, fabsf(load_as_float(a.q, (size_t)qr * kD + 16 * kk + 4 * c + i,
                                                   a.q_dtype)));
      }
      const int e = f16_fit_exponent(warp_max(amax));
      qscale = pow2i(e);
      qk_scale_log2_ = a.qk_scale_log2 * pow2i(-e);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const long long qr = q_row(a, s, hkv, nt * 8 + (lane >> 2));
      const bool live = qr >= 0;
      const size_t row = (size_t)(live ? qr : 0) * kD;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        if constexpr (T::kFp8) {
          // k-slot permutation matching the E4M3 A fragment: thread c holds d = 16kk + 4c .. 4c+3
          const int d = 16 * kk + 4 * c;
          float x0 = live ? load_as_float(a.q, row + d + 0, a.q_dtype) : 0.f;
          float x1 = live ? load_as_float(a.q, row + d + 1, a.q_dtype) : 0.f;
          float x2 = live ? load_as_float(a.q, row + d + 2, a.q_dtype) : 0.f;
          float x3 = live ? load_as_float(a.q, row + d + 3, a.q_dtype) : 0.f;
          qf[nt][kk][0] = pack_f16(x0 * qscale, x1 * qscale);
          qf[nt][kk][1] = pack_f16(x2 * qscale, x3 * qscale);
        } else {
          const uint32_t* qp = reinterpret_cast<const uint32_t*>(
              static_cast<const uint16_t*>(a.q) + row + 16 * kk + 2 * c);
          qf[nt][kk][0] = live ? __ldg(qp) : 0u;
          qf[nt][kk][1] = live ? __ldg(qp + 4) : 0u;
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = nt * 8 + 2 * c + h;           // the thread's accumulator columns
        if constexpr (kCausal) lim[nt][h] = r < a.R ? n - a.q_len + r / a.G : n - 1;
      }
    }
  }

  // The single-token path (one query token, G <= 8 heads as the 8 columns).
  // ks_b / vs_b: the block's own E4M3 scales (block-wise scaling), else 1.
  __device__ __forceinline__ void block_decode(uint32_t kbase, uint32_t vbase, uint32_t region_bytes,
                                        int row0, int valid, int lane, float ks_b, float vs_b) {
    const int c = lane & 3;
    const uint32_t sw = lane & 7;   // every ldmatrix row index is congruent to lane mod 8
    float s[kTiles][4];

    // ---- S^T = K q^T
#pragma unroll
    for (int mt = 0; mt < kTiles; ++mt) {
      float e[4] = {0.f, 0.f, 0.f, 0.f}, o[4] = {0.f, 0.f, 0.f, 0.f};
      const int row = row0 + mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
      if constexpr (!T::kFp8) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t chunk = ((kk & 3) << 1) | (lane >> 4);
          const uint32_t addr = kbase + (kk >> 2) * region_bytes + row * kLineBytes +
                                ((chunk ^ sw) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(addr, a0, a1, a2, a3);
          if (kk & 1) mma_16816<T::kBf16Mma>(o, a0, a1, a2, a3, qf[0][kk][0], qf[0][kk][1]);
          else mma_16816<T::kBf16Mma>(e, a0, a1, a2, a3, qf[0][kk][0], qf[0][kk][1]);
        }
      } else {
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          const uint32_t chunk = (jp << 1) | (lane >> 4);
          const uint32_t addr = kbase + row * kLineBytes + ((chunk ^ sw) << 4);
          uint32_t r0, r1, r2, r3;
          ldsm_x4(addr, r0, r1, r2, r3);
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          e4m3x4_to_f16x2x2(r0, a0, a2);
          e4m3x4_to_f16x2x2(r1, a1, a3);
          e4m3x4_to_f16x2x2(r2, b0, b2);
          e4m3x4_to_f16x2x2(r3, b1, b3);
          mma_16816<false>(e, a0, a1, a2, a3, qf[0][2 * jp][0], qf[0][2 * jp][1]);
          mma_16816<false>(o, b0, b1, b2, b3, qf[0][2 * jp + 1][0], qf[0][2 * jp + 1][1]);
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) s[mt][k] = e[k] + o[k];
    }

    // ---- online softmax (log2 domain); thread holds tokens lane/4 (+8), heads 2c, 2c+1
    const float qs = T::kFp8 ? qk_scale_log2_ * ks_b : qk_scale_log2_;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < kTiles; ++mt) {
      const int t0 = mt * 16 + (lane >> 2);
      const bool v0 = t0 < valid, v1 = t0 + 8 < valid;
      s[mt][0] = v0 ? s[mt][0] * qs : -INFINITY;
      s[mt][1] = v0 ? s[mt][1] * qs : -INFINITY;
      s[mt][2] = v1 ? s[mt][2] * qs : -INFINITY;
      s[mt][3] = v1 ? s[mt][3] * qs : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[mt][0], s[mt][2]));
      mx1 = fmaxf(mx1, fmaxf(s[mt][1], s[mt][3]));
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(m[0][0], mx0), mn1 = fmaxf(m[0][1], mx1);
    const float al0 = exp2f(m[0][0] - mn0), al1 = exp2f(m[0][1] - mn1);
    m[0][0] = mn0;
    m[0][1] = mn1;
    const float ref0 = mn0 - kPOff, ref1 = mn1 - kPOff;
    float p[kTiles][4];
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int mt = 0; mt < kTiles; ++mt) {
      p[mt][0] = exp2f(s[mt][0] - ref0);
      p[mt][1] = exp2f(s[mt][1] - ref1);
      p[mt][2] = exp2f(s[mt][2] - ref0);
      p[mt][3] = exp2f(s[mt][3] - ref1);
      ps0 += p[mt][0] + p[mt][2];
      ps1 += p[mt][1] + p[mt][3];
    }
    l[0][0] = l[0][0] * al0 + ps0;
    l[0][1] = l[0][1] * al1 + ps1;
    // E4M3 block-wise scales: the block's V scale rides on P (the row sums l keep
    // unscaled p), split so that P stays in f16's range
    float pv = 1.f, acc_f = 1.f;
    if (T::kFp8 && bscaled_) pv = v_block_factor(vs_b, &acc_f);
    const float a0 = al0 * acc_f, a1 = al1 * acc_f;
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
      acc[dt][0][0] *= a0;
      acc[dt][0][1] *= a1;
      acc[dt][0][2] *= a0;
      acc[dt][0][3] *= a1;
    }

    // ---- P^T as B operand: movmatrix transposes the 8x8 (token, head) quadrants
    uint32_t bh[kTiles][2], bl[kTiles][2];
#pragma unroll
    for (int mt = 0; mt < kTiles; ++mt) {
      const uint32_t x0 = pack2<T::kBf16Mma>(p[mt][0] * pv, p[mt][1] * pv);
      const uint32_t x1 = pack2<T::kBf16Mma>(p[mt][2] * pv, p[mt][3] * pv);
      bh[mt][0] = movmatrix_t(x0);
      bh[mt][1] = movmatrix_t(x1);
      if constexpr (kSplitP) {
        const float2 r0 = unpack2<true>(x0), r1 = unpack2<true>(x1);
        bl[mt][0] = movmatrix_t(pack_bf16(p[mt][0] - r0.x, p[mt][1] - r0.y));
        bl[mt][1] = movmatrix_t(pack_bf16(p[mt][2] - r1.x, p[mt][3] - r1.y));
      }
    }

    // ---- O^T += V^T P^T
    // Rows of V past the sequence's end are unwritten slots: their lanes are
    // zeroed (only in a tail block) so that 0 * NaN never reaches the sum.
    const bool tail = valid < BS;
#pragma unroll
    for (int mt = 0; mt < kTiles; ++mt) {
      // tokens of this thread in the A fragment: 2c, 2c+1 (regs 0,1) and 8+2c, 9+2c (regs 2,3)
      uint32_t mk_lo = 0xffffffffu, mk_hi = 0xffffffffu;
      if (tail) {
        const int tl = mt * 16 + 2 * c;
        mk_lo = (tl < valid ? 0x0000ffffu : 0u) | (tl + 1 < valid ? 0xffff0000u : 0u);
        mk_hi = (tl + 8 < valid ? 0x0000ffffu : 0u) | (tl + 9 < valid ? 0xffff0000u : 0u);
      }
      if constexpr (!T::kFp8) {
        const int q4 = lane >> 3;
        const int row = row0 + mt * 16 + ((q4 >> 1) << 3) + (lane & 7);
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
          const uint32_t chunk = ((dt & 3) << 1) | (q4 & 1);
          const uint32_t addr = vbase + (dt >> 2) * region_bytes + row * kLineBytes +
                                ((chunk ^ sw) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(addr, a0, a1, a2, a3);
          if (tail) {
            a0 &= mk_lo;
            a1 &= mk_lo;
            a2 &= mk_hi;
            a3 &= mk_hi;
          }
          mma_16816<T::kBf16Mma>(acc[dt][0], a0, a1, a2, a3, bh[mt][0], bh[mt][1]);
          if constexpr (kSplitP)
            mma_16816<T::kBf16Mma>(acc[dt][0], a0, a1, a2, a3, bl[mt][0], bl[mt][1]);
        }
      } else {
        const int q4 = lane >> 3;
        const int row = row0 + mt * 16 + ((q4 & 1) << 3) + (lane & 7);
#pragma unroll
        for (int dp = 0; dp < 4; ++dp) {
          const uint32_t chunk = (dp << 1) | (q4 >> 1);
          const uint32_t addr = vbase + row * kLineBytes + ((chunk ^ sw) << 4);
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(addr, r0, r1, r2, r3);
          // r = {V[2c][2i], V[2c][2i+1], V[2c+1][2i], V[2c+1][2i+1]} -> (d even, d odd) pairs
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          e4m3x4_to_f16x2x2(byte_perm(r0, 0, 0x3120), a0, a1);
          e4m3x4_to_f16x2x2(byte_perm(r1, 0, 0x3120), a2, a3);
          e4m3x4_to_f16x2x2(byte_perm(r2, 0, 0x3120), b0, b1);
          e4m3x4_to_f16x2x2(byte_perm(r3, 0, 0x3120), b2, b3);
          if (tail) {
            a0 &= mk_lo;
            a1 &= mk_lo;
            a2 &= mk_hi;
            a3 &= mk_hi;
            b0 &= mk_lo;
            b1 &= mk_lo;
            b2 &= mk_hi;
            b3 &= mk_hi;
          }
          mma_16816<false>(acc[2 * dp][0], a0, a1, a2, a3, bh[mt][0], bh[mt][1]);
          mma_16816<false>(acc[2 * dp + 1][0], b0, b1, b2, b3, bh[mt][0], bh[mt][1]);
        }
      }
    }
  }

  __device__ __forceinline__ void load_q_decode(const DecodeArgs& a, int s, int hkv, int lane) {
    const int g = lane >> 2, c = lane & 3;
    const bool live = g < a.G;
    const size_t row = ((size_t)s * a.Hq + (size_t)hkv * a.G + (live ? g : 0)) * kD;
    if constexpr (T::kFp8) {
      // q x 2^e in f16 (f16_fit_exponent over the warp's q), 2^-e on the softmax
      // scale; k-slot permutation matching the E4M3 A fragment: thread c holds
      // d = 16kk + 4c .. 4c+3
      float x[8][4];
      float amax = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[kk][i] = live ? load_as_float(a.q, row + 16 * kk + 4 * c + i, a.q_dtype) : 0.f;
          amax = fmaxf(amax, fabsf(x[kk][i]));
        }
      const int e = f16_fit_exponent(warp_max(amax));
      const float qscale = pow2i(e);
      qk_scale_log2_ = a.qk_scale_log2 * pow2i(-e);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qf[0][kk][0] = pack_f16(x[kk][0] * qscale, x[kk][1] * qscale);
        qf[0][kk][1] = pack_f16(x[kk][2] * qscale, x[kk][3] * qscale);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t* qp = reinterpret_cast<const uint32_t*>(
            static_cast<const uint16_t*>(a.q) + row + 16 * kk + 2 * c);
        qf[0][kk][0] = live ? __ldg(qp) : 0u;
        qf[0][kk][1] = live ? __ldg(qp + 4) : 0u;
      }
    }
  }

  // The single-token form of finish: base + g * stride is head g's partial row.
  __device__ __forceinline__ void finish_decode(const DecodeArgs& a, int s, int hkv, int lane, bool whole,
                                         size_t part_row_base, int part_row_stride) {
    float L0 = l[0][0], L1 = l[0][1];
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      L0 += __shfl_xor_sync(0xffffffffu, L0, o);
      L1 += __shfl_xor_sync(0xffffffffu, L1, o);
    }
    const int c = lane & 3;
    float inv0 = a.v_scale / L0, inv1 = a.v_scale / L1;
    if (T::kFp8 && bscaled_) {
      inv0 = ldexpf(inv0, ev_ref_);
      inv1 = ldexpf(inv1, ev_ref_);
    }
    const int g0 = 2 * c, g1 = 2 * c + 1;
    if (whole) {
      const size_t ob = ((size_t)s * a.Hq + (size_t)hkv * a.G) * kD;
#pragma unroll
      for (int dt = 0; dt < 8; ++dt)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int g = (k & 1) ? g1 : g0;
          if (g < a.G)
            store_from_float(a.out, ob + (size_t)g * kD + d_of(dt, k, lane), a.out_dtype,
                             acc[dt][0][k] * ((k & 1) ? inv1 : inv0));
        }
    } else {
#pragma unroll
      for (int dt = 0; dt < 8; ++dt)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int g = (k & 1) ? g1 : g0;
          if (g < a.G)
            a.part_o[(part_row_base + (size_t)g * part_row_stride) * kD + d_of(dt, k, lane)] =
                acc[dt][0][k] * ((k & 1) ? inv1 : inv0);
        }
      if ((lane >> 2) == 0) {
        if (g0 < a.G) a.part_lse[part_row_base + (size_t)g0 * part_row_stride] = (m[0][0] + __log2f(L0) - kPOff) * kLn2;
        if (g1 < a.G) a.part_lse[part_row_base + (size_t)g1 * part_row_stride] = (m[0][1] + __log2f(L1) - kPOff) * kLn2;
      }
    }
    reset();
  }

  // One block of BS tokens for this warp's KV head.  `kbase` / `vbase` point at
  // the first region of K / V in the stage; `row0` is the warp's first row;
  // `jbase` the block's first token position; `valid` its tokens inside the
  // sequence; `full`: no key of the block is hidden from any query row.
  __device__ __forceinline__ void block(uint32_t kbase, uint32_t vbase, uint32_t region_bytes,
                                        int row0, int jbase, int valid, bool full, int lane,
                                        float ks_b, float vs_b) {
    if constexpr (NT == 1 && !kCausal) {
      block_decode(kbase, vbase, region_bytes, row0, valid, lane, ks_b, vs_b);
      return;
    }
    const int c = lane & 3;
    const uint32_t sw = lane & 7;   // every ldmatrix row index is congruent to lane mod 8
    float s[kTiles][NT][4];

    // ---- S^T = K q^T
#pragma unroll
    for (int mt = 0; mt < kTiles; ++mt) {
      float e[NT][4], o[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) e[nt][k] = o[nt][k] = 0.f;
      const int row = row0 + mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
      if constexpr (!T::kFp8) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t chunk = ((kk & 3) << 1) | (lane >> 4);
          const uint32_t addr = kbase + (kk >> 2) * region_bytes + row * kLineBytes +
                                ((chunk ^ sw) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (kk & 1) mma_16816<T::kBf16Mma>(o[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
            else mma_16816<T::kBf16Mma>(e[nt], a0, a1, a2, a3, qf[nt][kk][0], qf[nt][kk][1]);
          }
        }
      } else {
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          const uint32_t chunk = (jp << 1) | (lane >> 4);
          const uint32_t addr = kbase + row * kLineBytes + ((chunk ^ sw) << 4);
          uint32_t r0, r1, r2, r3;
          ldsm_x4(addr, r0, r1, r2, r3);
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          e4m3x4_to_f16x2x2(r0, a0, a2);
          e4m3x4_to_f16x2x2(r1, a1, a3);
          e4m3x4_to_f16x2x2(r2, b0, b2);
          e4m3x4_to_f16x2x2(r3, b1, b3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_16816<false>(e[nt], a0, a1, a2, a3, qf[nt][2 * jp][0], qf[nt][2 * jp][1]);
            mma_16816<false>(o[nt], b0, b1, b2, b3, qf[nt][2 * jp + 1][0], qf[nt][2 * jp + 1][1]);
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int k = 0; k < 4; ++k) s[mt][nt][k] = e[nt][k] + o[nt][k];
    }

    // ---- online softmax (log2 domain); thread holds tokens lane/4 (+8), columns 2c, 2c+1
    const float qs = T::kFp8 ? qk_scale_log2_ * ks_b : qk_scale_log2_;
    float mx[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mx[nt][0] = mx[nt][1] = -INFINITY;
#pragma unroll
    for (int mt = 0; mt < kTiles; ++mt) {
      if constexpr (kCausal) {
        const int t0 = jbase + mt * 16 + (lane >> 2);   // key positions of the thread's rows
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int t = t0 + ((k >> 1) << 3);
            const bool ok = full || t <= lim[nt][k & 1];
            s[mt][nt][k] = ok ? s[mt][nt][k] * qs : -INFINITY;
            mx[nt][k & 1] = fmaxf(mx[nt][k & 1], s[mt][nt][k]);
          }
      } else {
        // one query token: every column sees exactly the block's `valid` first keys
        const int t0 = mt * 16 + (lane >> 2);
        const bool v0 = t0 < valid, v1 = t0 + 8 < valid;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          s[mt][nt][0] = v0 ? s[mt][nt][0] * qs : -INFINITY;
          s[mt][nt][1] = v0 ? s[mt][nt][1] * qs : -INFINITY;
          s[mt][nt][2] = v1 ? s[mt][nt][2] * qs : -INFINITY;
          s[mt][nt][3] = v1 ? s[mt][nt][3] * qs : -INFINITY;
          mx[nt][0] = fmaxf(mx[nt][0], fmaxf(s[mt][nt][0], s[mt][nt][2]));
          mx[nt][1] = fmaxf(mx[nt][1], fmaxf(s[mt][nt][1], s[mt][nt][3]));
        }
      }
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mx[nt][0] = fmaxf(mx[nt][0], __shfl_xor_sync(0xffffffffu, mx[nt][0], o));
        mx[nt][1] = fmaxf(mx[nt][1], __shfl_xor_sync(0xffffffffu, mx[nt][1], o));
      }
    float p[kTiles][NT][4];
    // E4M3 block-wise scales: the block's V scale rides on P, split so that P
    // stays in f16's range (see v_block_factor)
    float pv = 1.f, acc_f = 1.f;
    if (T::kFp8 && bscaled_) pv = v_block_factor(vs_b, &acc_f);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float mn = fmaxf(m[nt][h], mx[nt][h]);
        // causal: a column that sees no key of this block keeps its state (its max
        // may still be -inf); one query token always sees the block's first key
        float ref = mn;
        if constexpr (kCausal) ref = mn == -INFINITY ? 0.f : mn;
        const float al = exp2f(m[nt][h] - ref);
        m[nt][h] = mn;
        const float pref = ref - kPOff;
        float ps = 0.f;
#pragma unroll
        for (int mt = 0; mt < kTiles; ++mt) {
          p[mt][nt][h] = exp2f(s[mt][nt][h] - pref);
          p[mt][nt][h + 2] = exp2f(s[mt][nt][h + 2] - pref);
          ps += p[mt][nt][h] + p[mt][nt][h + 2];
        }
        l[nt][h] = l[nt][h] * al + ps;
        const float alv = al * acc_f;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
          acc[dt][nt][h] *= alv;
          acc[dt][nt][h + 2] *= alv;
        }
      }
    }

    // ---- P^T as B operand: movmatrix transposes the 8x8 (token, column) quadrants
    uint32_t bh[kTiles][NT][2], bl[kTiles][NT][2];
#pragma unroll
    for (int mt = 0; mt < kTiles; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t x0 = pack2<T::kBf16Mma>(p[mt][nt][0] * pv, p[mt][nt][1] * pv);
        const uint32_t x1 = pack2<T::kBf16Mma>(p[mt][nt][2] * pv, p[mt][nt][3] * pv);
        bh[mt][nt][0] = movmatrix_t(x0);
        bh[mt][nt][1] = movmatrix_t(x1);
        if constexpr (kSplitP) {
          const float2 r0 = unpack2<true>(x0), r1 = unpack2<true>(x1);
          bl[mt][nt][0] = movmatrix_t(pack_bf16(p[mt][nt][0] - r0.x, p[mt][nt][1] - r0.y));
          bl[mt][nt][1] = movmatrix_t(pack_bf16(p[mt][nt][2] - r1.x, p[mt][nt][3] - r1.y));
        }
      }

    // ---- O^T += V^T P^T
    // Rows of V past the sequence's end are unwritten slots: their lanes are
    // zeroed (only in a tail block) so that 0 * NaN never reaches the sum.
    const bool tail = valid < BS;
#pragma unroll
    for (int mt = 0; mt < kTiles; ++mt) {
      // tokens of this thread in the A fragment: 2c, 2c+1 (regs 0,1) and 8+2c, 9+2c (regs 2,3)
      uint32_t mk_lo = 0xffffffffu, mk_hi = 0xffffffffu;
      if (tail) {
        const int tl = mt * 16 + 2 * c;
        mk_lo = (tl < valid ? 0x0000ffffu : 0u) | (tl + 1 < valid ? 0xffff0000u : 0u);
        mk_hi = (tl + 8 < valid ? 0x0000ffffu : 0u) | (tl + 9 < valid ? 0xffff0000u : 0u);
      }
      if constexpr (!T::kFp8) {
        const int q4 = lane >> 3;
        const int row = row0 + mt * 16 + ((q4 >> 1) << 3) + (lane & 7);
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
          const uint32_t chunk = ((dt & 3) << 1) | (q4 & 1);
          const uint32_t addr = vbase + (dt >> 2) * region_bytes + row * kLineBytes +
                                ((chunk ^ sw) << 4);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(addr, a0, a1, a2, a3);
          if (tail) {
            a0 &= mk_lo;
            a1 &= mk_lo;
            a2 &= mk_hi;
            a3 &= mk_hi;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_16816<T::kBf16Mma>(acc[dt][nt], a0, a1, a2, a3, bh[mt][nt][0], bh[mt][nt][1]);
            if constexpr (kSplitP)
              mma_16816<T::kBf16Mma>(acc[dt][nt], a0, a1, a2, a3, bl[mt][nt][0], bl[mt][nt][1]);
          }
        }
      } else {
        const int q4 = lane >> 3;
        const int row = row0 + mt * 16 + ((q4 & 1) << 3) + (lane & 7);
#pragma unroll
        for (int dp = 0; dp < 4; ++dp) {
          const uint32_t chunk = (dp << 1) | (q4 >> 1);
          const uint32_t addr = vbase + row * kLineBytes + ((chunk ^ sw) << 4);
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(addr, r0, r1, r2, r3);
          // r = {V[2c][2i], V[2c][2i+1], V[2c+1][2i], V[2c+1][2i+1]} -> (d even, d odd) pairs
          uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
          e4m3x4_to_f16x2x2(byte_perm(r0, 0, 0x3120), a0, a1);
          e4m3x4_to_f16x2x2(byte_perm(r1, 0, 0x3120), a2, a3);
          e4m3x4_to_f16x2x2(byte_perm(r2, 0, 0x3120), b0, b1);
          e4m3x4_to_f16x2x2(byte_perm(r3, 0, 0x3120), b2, b3);
          if (tail) {
            a0 &= mk_lo;
            a1 &= mk_lo;
            a2 &= mk_hi;
            a3 &= mk_hi;
            b0 &= mk_lo;
            b1 &= mk_lo;
            b2 &= mk_hi;
            b3 &= mk_hi;
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_16816<false>(acc[2 * dp][nt], a0, a1, a2, a3, bh[mt][nt][0], bh[mt][nt][1]);
            mma_16816<false>(acc[2 * dp + 1][nt], b0, b1, b2, b3, bh[mt][nt][0], bh[mt][nt][1]);
          }
        }
      }
    }
  }

  // d index held by accumulator register k of tile dt.
  __device__ __forceinline__ static int d_of(int dt, int k, int lane) {
    if constexpr (T::kFp8) return 16 * dt + 2 * (lane >> 2) + (k >> 1);
    else return 16 * dt + (lane >> 2) + ((k >> 1) << 3);
  }

  // Write the piece's result: directly to out (whole = true) or as a partial
  // (balanced: rows part_base + column; fixed: part_base + q_row * S).
  __device__ __forceinline__ void finish(const DecodeArgs& a, int s, int hkv, int lane, bool whole,
                                         size_t part_base, bool balanced) {
    if constexpr (NT == 1 && !kCausal) {
      if (balanced) finish_decode(a, s, hkv, lane, whole, part_base, 1);
      else finish_decode(a, s, hkv, lane, whole,
                         part_base + ((size_t)s * a.Hq + (size_t)hkv * a.G) * a.S, a.S);
      return;
    }
    const int c = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float L[2] = {l[nt][0], l[nt][1]};
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        L[0] += __shfl_xor_sync(0xffffffffu, L[0], o);
        L[1] += __shfl_xor_sync(0xffffffffu, L[1], o);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = nt * 8 + 2 * c + h;
        const long long qr = q_row(a, s, hkv, r);
        if (qr < 0) continue;
        // a column that saw no key (a query before the sequence start) is empty
        const bool empty = m[nt][h] == -INFINITY;
        float inv = empty ? 0.f : a.v_scale / L[h];
        if (T::kFp8 && bscaled_) inv = ldexpf(inv, ev_ref_);
        const size_t prow = balanced ? part_base + (size_t)r : part_base + (size_t)qr * a.S;
#pragma unroll
        for (int dt = 0; dt < 8; ++dt)
#pragma unroll
          for (int k = h; k < 4; k += 2) {
            const int d = d_of(dt, k, lane);
            const float v = acc[dt][nt][k] * inv;
            if (whole) store_from_float(a.out, (size_t)qr * kD + d, a.out_dtype, v);
            else a.part_o[prow * kD + d] = v;
          }
        if (!whole && (lane >> 2) == 0)
          a.part_lse[prow] = empty ? -INFINITY : (m[nt][h] + __log2f(L[h]) - kPOff) * kLn2;
      }
    }
    reset();
  }

  float qk_scale_log2_;
  bool bscaled_;           // E4M3 pool with block-wise scales attached
};

// First partial row of a piece: balanced mode rows are slot * HG*R + w*R + column;
// fixed mode rows are ((s * q_len + i) * Hq + h) * S + p = q_row * S + p.
__device__ __forceinline__ size_t part_base(const DecodeArgs& a, int w, long long slot, int p) {
  if (a.mode == 0) return (size_t)slot * (a.HG * a.R) + (size_t)w * a.R;
  return (size_t)p;
}

// kOff: a shared-prefix launch, each sequence read from token a.len_off[s] on.
template <int KVT, int BS, int NT, bool kCausal, bool kOff>
__global__ void __launch_bounds__(32 * (kMaxHG + 1), 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeArgs a) {
  using T = KvTraits<KVT>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle pattern
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  const int rows = a.HG * BS;                              // rows per region
  const uint32_t region_bytes = (uint32_t)rows * kLineBytes;
  const uint32_t stage_bytes = region_bytes * 2 * T::kRegions;
  SmemHeader* hdr = reinterpret_cast<SmemHeader*>(smem + (size_t)a.stages * stage_bytes);
  const uint32_t ring = smem_u32(smem);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int producer = nwarps - 1;

  // ---- prologue: barriers and this CTA's run of the block stream
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(&hdr->full[i], 1);
      mbar_init(&hdr->empty[i], producer);
    }
    hdr->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == producer && lane == 0) prefetch_tensormap(&tmap);

  if (a.mode == 0 && warp == 0) {
    long long total = 0;
    for (int base = 0; base < a.B; base += 32) {
      const int s = base + lane;
      int nb = s < a.B ? blocks_of(clamp_len<kOff>(a, s), BS) : 0;
      total += (long long)__reduce_add_sync(0xffffffffu, (unsigned)nb);
      // units of a sequence with no tokens get no piece: mark them once
      if (blockIdx.x == 0 && __any_sync(0xffffffffu, s < a.B && nb == 0)) {
        if (a.pdl) grid_dependency_wait();
        if (s < a.B && nb == 0)
          for (int hg = 0; hg < a.NHG; ++hg) a.unit_info[(size_t)s * a.NHG + hg] = make_int2(0, 0);
      }
    }
    total *= a.NHG;
    // Only min(grid, total) CTAs take part, so that every run holds at least one
    // block: the CTAs between a unit's first and last owner then all leave a partial.
    const long long P = total < (long long)gridDim.x ? total : (long long)gridDim.x;
    const long long gb0 = blockIdx.x < P ? (long long)blockIdx.x * total / P : 0;
    const long long gb1 = blockIdx.x < P ? ((long long)blockIdx.x + 1) * total / P : 0;
    int fs = 0, fhg = 0, fj = 0;
    if (gb0 < gb1) {
      long long run = 0;
      bool found = false;
      for (int base = 0; base < a.B && !found; base += 32) {
        const int s = base + lane;
        const int nbs = s < a.B ? blocks_of(clamp_len<kOff>(a, s), BS) : 0;
        const int nbu = nbs * a.NHG;
        int incl = nbu;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const long long lo = run + incl - nbu, hi = run + incl;
        const unsigned hit = __ballot_sync(0xffffffffu, s < a.B && lo <= gb0 && gb0 < hi);
        if (hit) {
          const int src = __ffs(hit) - 1;
          const long long off = gb0 - __shfl_sync(0xffffffffu, lo, src);
          const int nb_src = __shfl_sync(0xffffffffu, nbs, src);
          fs = base + src;
          fhg = (int)(off / nb_src);
          fj = (int)(off % nb_src);
          found = true;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) {
      hdr->total = total;
      hdr->gb0 = gb0;
      hdr->gb1 = gb1;
      hdr->s = fs;
      hdr->hg = fhg;
      hdr->j = fj;
    }
  }
  __syncthreads();
  // Balanced mode runs one resident wave.  When the next launch in the stream is
  // this call's own merge (a.early_trigger), it may be scheduled now: it takes
  // SMs as this grid's CTAs retire and waits (griddepcontrol.wait) for the whole
  // grid before it reads a partial.  The merge in turn lets the next step's
  // attention start early; that kernel waits for this chain before it loads the
  // last two blocks of a sequence (the blocks this step's new token went to) and
  // before it writes anything.
  if (a.mode == 0 && a.early_trigger) grid_launch_dependents();

  // ---- this CTA's cursor (identical in every warp)
  Cursor cur;
  int part_p = 0;
  if (a.mode == 0) {
    cur.s = hdr->s;
    cur.hg = hdr->hg;
    cur.j = hdr->j;
    cur.gb = hdr->gb0;
    cur.remaining = hdr->gb1 - hdr->gb0;
    cur.n = cur.remaining > 0 ? clamp_len<kOff>(a, cur.s) : 0;
    cur.nb = blocks_of(cur.n, BS);
  } else {
    const int u = blockIdx.y;
    cur.s = u / a.NHG;
    cur.hg = u % a.NHG;
    cur.n = clamp_len<kOff>(a, cur.s);
    cur.nb = blocks_of(cur.n, BS);
    part_p = blockIdx.x;
    const int jb = (int)((long long)part_p * cur.nb / a.S);
    const int je = (int)((long long)(part_p + 1) * cur.nb / a.S);
    cur.j = jb;
    cur.gb = jb;
    cur.remaining = je - jb;
  }
  cur.j0 = cur.j;

  if (warp == producer) {
    // ---------------------------------------------------------------- producer
    int stage = 0;
    uint32_t round = 0;
    long long issued = 0;
    int ids = 0, id_base = -1, id_unit_s = -1;
    bool waited = false;
    while (cur.remaining > 0) {
      // refill 32 table entries of the current sequence when needed
      if (cur.s != id_unit_s || cur.j < id_base || cur.j >= id_base + 32) {
        id_unit_s = cur.s;
        id_base = cur.j;
        const int jj = id_base + lane;
        // shared-prefix decode: the sequence's private blocks, after its prefix
        // (offset from the length clamp_len clamps, so jo + cur.nb <= max_blocks)
        int jo = 0;
        if constexpr (kOff)
          jo = first_token(a, cur.s, min(max(__ldg(a.seq_lens + cur.s), 0), a.max_blocks * BS)) /
               BS;
        ids = jj < cur.nb ? __ldg(a.tables + (size_t)cur.s * a.max_blocks + jo + jj) : 0;
      }
      int blk = __shfl_sync(0xffffffffu, ids, cur.j - id_base);
      const bool blk_ok = blk >= 0 && blk < a.num_blocks;
      if (!blk_ok) {
        if (lane == 0) record_error(a.status, PKV_EBOUNDS);
        blk = 0;
      }
      // with programmatic dependent launch the kernels ahead in the stream may still
      // run: the last two blocks of a sequence may hold tokens they store
      if (a.pdl && !waited && cur.j >= cur.nb - 2) {
        grid_dependency_wait();
        waited = true;
      }
      if (a.k_new && cur.j == cur.nb - 1 && blk_ok) {
        // decode step: store the sequence's new token (position n - 1) for this
        // head group, then order those generic-proxy writes before the TMA read
        if (a.pdl && !waited) {
          grid_dependency_wait();
          waited = true;
        }
        const int t = (cur.n - 1) % BS;
        const int per_head = kD / 8;
        const int total8 = 2 * a.HG * per_head;
        for (int i = lane; i < total8; i += 32) {
          const int kv = i / (a.HG * per_head);
          const int r = i - kv * a.HG * per_head;
          const int h = cur.hg * a.HG + r / per_head;
          const int d8 = r % per_head;
          const size_t src = ((size_t)cur.s * a.Hkv + h) * kD + (size_t)d8 * 8;
          const size_t dst =
              (((((size_t)blk * 2 + kv) * a.L + a.layer) * a.Hkv + h) * BS + t) * kD +
              (size_t)d8 * 8;
          float sc = kv ? a.v_enc_scale : a.k_enc_scale;
          if (T::kFp8 && a.block_scales)
            sc = a.block_scales[(((size_t)blk * 2 + kv) * a.L + a.layer) * a.Hkv + h];
          store8_to_pool(const_cast<void*>(a.pool), dst, KVT, kv ? a.v_new : a.k_new, src,
                         a.new_dtype, sc);
        }
        fence_proxy_async_global();
        __syncwarp();
      }
      if (lane == 0) {
        const bool ok = mbar_wait_bounded(&hdr->empty[stage], (round & 1) ^ 1);
        if (!ok || hdr->abort_flag) {
          if (!ok) record_error(a.status, PKV_ETIMEOUT);
          hdr->abort_flag = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, (int)hdr->abort_flag, 0)) break;
      if (T::kFp8 && a.block_scales) {
        // the stage's per-tile scales, visible to the consumers through the full barrier
        if (lane < 2 * a.HG) {
          const int kv = lane / a.HG, hl = lane % a.HG;
          hdr->bscale[stage][kv][hl] =
              a.block_scales[(((size_t)blk * 2 + kv) * a.L + a.layer) * a.Hkv + cur.hg * a.HG + hl];
        }
        __syncwarp();
      }
      if (lane == 0) {
        {
          mbar_arrive_expect_tx(&hdr->full[stage], stage_bytes);
          uint8_t* st = smem + (size_t)stage * stage_bytes;
          const int hrow = cur.hg * a.HG * BS;   // first row of the head group in a (blk, kv, layer) slab
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const int z = (blk * 2 + kv) * a.L + a.layer;
#pragma unroll
            for (int r = 0; r < T::kRegions; ++r)
              tma_load_3d(st + (size_t)(kv * T::kRegions + r) * region_bytes, &tmap,
                          &hdr->full[stage], r * 64, hrow, z);
          }
        }
      }
      ++issued;
      if (++stage == a.stages) {
        stage = 0;
        ++round;
      }
      cursor_next<kOff>(cur, a);
    }
    // drain: every stage still in flight must land before the CTA may exit
    if (lane == 0) {
      const long long inflight = issued < a.stages ? issued : a.stages;
      for (long long i = 0; i < inflight; ++i) {
        long long it = issued - 1 - i;
        const int st = (int)(it % a.stages);
        const uint32_t par = (uint32_t)((it / a.stages) & 1);
        if (!mbar_wait_bounded(&hdr->full[st], par)) {
          record_error(a.status, PKV_ETIMEOUT);
          break;
        }
      }
    }
    grid_launch_dependents();
    return;
  }

  if (warp >= a.HG) return;   // no spare warps are launched; guard anyway

  // ---------------------------------------------------------------- consumers
  Consumer<KVT, BS, NT, kCausal> cons;
  cons.qk_scale_log2_ = a.qk_scale_log2;
  cons.bscaled_ = T::kFp8 && a.block_scales != nullptr;
  cons.reset();
  const int w = warp;
  bool waited = false;
  int hkv = cur.hg * a.HG + w;
  if (cur.remaining > 0) cons.load_q(a, cur.s, cur.n, hkv, lane);

  // fixed mode, empty partition: an empty partial (or zero output when S == 1)
  if (a.mode == 1 && cur.remaining <= 0) {
    if (a.pdl) grid_dependency_wait();
    for (int r = 0; r < a.R; ++r) {
      const long long qr = Consumer<KVT, BS, NT, kCausal>::q_row(a, cur.s, hkv, r);
      if (a.S == 1) {
        for (int d = lane; d < kD; d += 32) store_from_float(a.out, (size_t)qr * kD + d, a.out_dtype, 0.f);
      } else {
        const size_t prow = (size_t)qr * a.S + part_p;
        for (int d = lane; d < kD; d += 32) a.part_o[prow * kD + d] = 0.f;
        if (lane == 0) a.part_lse[prow] = -INFINITY;
      }
    }
    grid_launch_dependents();
    return;
  }

  // a shared-prefix decode merges every row with its prefix partials, and a call
  // that returns each row's log-sum-exp has the merge write every row
  const bool whole_ok = a.ext_lse == nullptr && a.out_lse == nullptr;
  int stage = 0;
  uint32_t round = 0;
  while (cur.remaining > 0) {
    if (!mbar_wait_bounded(&hdr->full[stage], round & 1)) {
      if (lane == 0) {
        record_error(a.status, PKV_ETIMEOUT);
        hdr->abort_flag = 1;
      }
      break;
    }
    const uint32_t sbase = ring + (uint32_t)stage * stage_bytes;
    const int valid = min(BS, cur.n - cur.j * BS);
    const int jbase = cur.j * BS;
    const bool full = !kCausal || jbase + BS - 1 <= cur.n - a.q_len;
    float ks_b = 1.f, vs_b = 1.f;
    if (T::kFp8 && a.block_scales) {
      ks_b = hdr->bscale[stage][0][w];
      vs_b = hdr->bscale[stage][1][w];
    }
    cons.block(sbase, sbase + T::kRegions * region_bytes, region_bytes, w * BS, jbase, valid,
               full, lane, ks_b, vs_b);
    __syncwarp();
    if (lane == 0) mbar_arrive(&hdr->empty[stage]);
    if (++stage == a.stages) {
      stage = 0;
      ++round;
    }

    const bool unit_end = cur.j == cur.nb - 1;
    const bool run_end = cur.remaining == 1;
    if (unit_end || run_end) {
      if (a.pdl && !waited) {
        grid_dependency_wait();
        waited = true;
      }
      const bool first = cur.j0 == 0;
      const long long u = (long long)cur.s * a.NHG + cur.hg;
      bool whole;
      long long slot = 0;
      if (a.mode == 0) {
        whole = first && unit_end && whole_ok;
        slot = (long long)blockIdx.x + u;
        if (first && w == 0 && lane == 0) {
          const long long unit_first_gb = cur.gb - cur.j;
          const long long parts = hdr->total < (long long)gridDim.x ? hdr->total : (long long)gridDim.x;
          const long long c_last = owner_of(unit_first_gb + cur.nb - 1, hdr->total, parts);
          a.unit_info[u] = make_int2((int)slot, (int)(c_last - blockIdx.x + 1));
        }
      } else {
        whole = a.S == 1;
      }
      cons.finish(a, cur.s, hkv, lane, whole, part_base(a, w, slot, part_p), a.mode == 0);
    }
    cursor_next<kOff>(cur, a);
    if (cur.remaining > 0 && cur.j == 0) {
      hkv = cur.hg * a.HG + w;
      cons.load_q(a, cur.s, cur.n, hkv, lane);
    }
  }
  // a chained launch ends only after the launches ahead of it (a CTA that wrote
  // nothing has not waited yet)
  if (a.pdl && !waited) grid_dependency_wait();
  grid_launch_dependents();
}

template <int KVT, int BS, int NT, bool kCausal, bool kOff = false>
cudaError_t launch_t(const CUtensorMap* map, const DecodeArgs& a, int gx, int gy,
                     cudaStream_t stream) {
  // the ring needs mma_smem_bytes; a larger request (a.smem_bytes) caps how many
  // CTAs can share an SM
  const size_t smem = std::max(mma_smem_bytes(KVT, BS, a.HG, a.stages), (size_t)a.smem_bytes);
  auto kern = decode_mma_kernel<KVT, BS, NT, kCausal, kOff>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, gy);
  cfg.blockDim = dim3(32 * (a.HG + 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, *map, a);
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace mma
}  // namespace pkv
