// prefill_tc.cu -- causal attention of a chunk of new tokens over the paged
// pool on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// The computation is the multi-token decode of paged_decode_attention_mq
// ("Unlocking long context: engineering practice for million-token LLM
// inference", section 5.2 chunked prefill; naive attention of section 4.1;
// paging of "The engineering truth of long-context inference 2026", section
// 2.2; online softmax of its section 3.1): query token i of sequence s sits at
// position n - q_len + i and attends over keys 0 .. that position.  When the
// chunk holds many query rows per KV head the q-tile x page product is a real
// dense contraction, so it runs here as UMMA tiles:
//
//   CTA (query tile, KV head hkv, sequence s): M = 128 rows = 128/G query
//   tokens x G heads, staged once in shared memory (128-byte swizzled).
//   K/V tiles of 64 tokens arrive by TMA from the pool (one box per block and
//   64-column half), double-buffered.
//     S_j = Q K_j^T         tcgen05.mma M128 N64 K128 -> TMEM (two S buffers, so
//                           S_{j+1} runs while the softmax of S_j does)
//     softmax               4 warps, one thread per row: tcgen05.ld of its S row,
//                           scale, causal mask, running max / sum, P_j -> smem (bf16/f16)
//     O += P_j V_j          tcgen05.mma M128 N128 K64, V as the MN-major operand
//   O lives in TMEM for the whole key range.  The softmax keeps a reference max
//   per row and rescales the row of O (tcgen05.ld/st) only when the true max
//   exceeds it by more than 8 (log2 units); P is then at most 2^8, exact in
//   fp32 accumulation, and O and the row sum share the same reference.
// One elected thread of warp 4 issues the TMA loads and the MMAs; mbarriers
// (all waits bounded) pass the tiles between the roles.
#include "device.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kM = 128;          // query rows per CTA
constexpr int kN = 64;           // keys per tile
constexpr uint32_t kHalf = 16384;            // 128 rows x 128 B: one 64-column half of Q
constexpr uint32_t kKVHalf = kN * 128;       // 64 rows x 128 B
constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemK = kSmemQ + 2 * kHalf;            // 2 buffers x 2 halves
constexpr uint32_t kSmemV = kSmemK + 2 * 2 * kKVHalf;
constexpr uint32_t kSmemP = kSmemV + 2 * 2 * kKVHalf;     // 128 rows x 64 keys
constexpr uint32_t kSmemBytes = kSmemP + kM * 128;
constexpr uint32_t kTmemCols = 256;          // S0 [0,64) S1 [64,128) O [128,256)
// Slack for aligning the tiles to 1024 bytes (the 128-byte swizzle atom).  Two
// CTAs per SM must fit in its 228 KB (each also holds 1 KB for the system):
// 114,688 B of tiles + the barriers + this slack stays under 115,712 B.  A
// base that needs more is refused in the kernel (an error, no access).
constexpr uint32_t kAlignSlack = 896;

struct Bars {
  uint64_t kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full, o_done;
  uint32_t tmem;
  volatile int abort_flag;
};

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}

template <bool kBf16>
__global__ void __launch_bounds__(160, 2)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t shift = ((raw + 1023u) & ~1023u) - raw;
  if (shift > kAlignSlack) {                    // uniform over the CTA
    if (threadIdx.x == 0) record_error(a.status, PKV_ECUDA);
    return;
  }
  uint8_t* sm = smem_raw + shift;
  Bars* bars = reinterpret_cast<Bars*>(sm + kSmemBytes);
  const uint32_t base = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x, hkv = blockIdx.y, s = blockIdx.z;
  const int G = a.G, QT = kM / G;                 // query tokens per tile
  const int t0 = qt * QT;                          // first query token of the tile

  int n = __ldg(a.seq_lens + s);
  const int cap = a.max_blocks * a.BS;
  if (n < 0 || n > cap) {
    if (tid == 0) record_error(a.status, PKV_EBOUNDS);
    n = n < 0 ? 0 : cap;
  }
  const int last_tok = min(t0 + QT, a.q_len) - 1;          // last query token of the tile
  const int p_last = n - a.q_len + last_tok;                // its key limit (position)
  const int tiles = (t0 < a.q_len && p_last >= 0) ? (p_last + kN) / kN : 0;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 128);
    }
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->o_done, 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(&bars->tmem, kTmemCols);
    tmem_relinquish();
  }
  // Q tile: thread r stages row r = (token t0 + r / G, head hkv*G + r % G), swizzled
  if (warp < 4) {
    const int r = tid, i = r / G, g = r % G;
    const bool live = t0 + i < a.q_len;
    const size_t qrow = ((size_t)s * a.q_len + t0 + i) * a.Hq + (size_t)hkv * G + g;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                      (live ? qrow : 0) * kD);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = live ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(sm + kSmemQ + (c >> 3) * kHalf + sw128(r, c & 7)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA + MMA issuer
    // The whole warp walks the loop and waits (so it stays converged); lane 0
    // issues the TMA loads, the MMAs and the commits.
    if (tiles > 0) {
      const bool leader = lane == 0;
      const int bpt = kN / a.BS;                               // blocks per key tile
      const int nblk = (n + a.BS - 1) / a.BS;
      const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
      auto load_tile = [&](int j) {
        if (!leader) return;
        const int b = j & 1;
        mbar_arrive_expect_tx(&bars->kv_full[b], 4 * kKVHalf);
        for (int bl = 0; bl < bpt; ++bl) {
          // blocks past the sequence's last one are replaced by its last block:
          // their keys are masked and their V rows zeroed before use
          const int jb = min(j * bpt + bl, nblk - 1);
          int blk = __ldg(trow + jb);
          if (blk < 0 || blk >= a.num_blocks) {
            record_error(a.status, PKV_EBOUNDS);
            blk = 0;
          }
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const int z = (blk * 2 + kv) * a.L + a.layer;
            uint8_t* dst = sm + (kv ? kSmemV : kSmemK) + b * 2 * kKVHalf + bl * a.BS * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_3d(dst + h * kKVHalf, &tmap, &bars->kv_full[b], h * 64, hkv * a.BS, z);
          }
        }
      };
      const uint32_t id_s = kBf16 ? idesc_bf16_f32(kM, kN, false, false)
                                  : (idesc_bf16_f32(kM, kN, false, false) & ~((7u << 7) | (7u << 10)));
      const uint32_t id_o = kBf16 ? idesc_bf16_f32(kM, kD, false, true)
                                  : (idesc_bf16_f32(kM, kD, false, true) & ~((7u << 7) | (7u << 10)));
      auto issue_s = [&](int j) {
        if (!leader) return;
        const int b = j & 1;
        const uint32_t kb = base + kSmemK + b * 2 * kKVHalf;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = (k & 3) * 32;
          const uint64_t da = smem_desc_sw128(base + kSmemQ + (k >> 2) * kHalf + off, 16, 1024);
          const uint64_t db = smem_desc_sw128(kb + (k >> 2) * kKVHalf + off, 16, 1024);
          tc_mma_f16(tmem + b * kN, da, db, id_s, k > 0);
        }
        tc_commit(&bars->s_full[b]);
      };
      // every lane waits; the warp agrees on the outcome
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        const bool got = mbar_wait_bounded(bar, parity);
        return __all_sync(0xffffffffu, got) && !bars->abort_flag;
      };
      bool ok = true;
      load_tile(0);
      if (tiles > 1) load_tile(1);
      ok = wait(&bars->kv_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int j = 0; j < tiles && ok; ++j) {
        if (j + 1 < tiles) {
          ok = wait(&bars->kv_full[(j + 1) & 1], ((j + 1) >> 1) & 1);
          if (ok && j >= 1) ok = wait(&bars->s_free[(j + 1) & 1], ((j - 1) >> 1) & 1);
          if (!ok) break;
          tc_fence_after();
          issue_s(j + 1);
        }
        ok = wait(&bars->p_full, j & 1);
        if (!ok) break;
        tc_fence_after();
        const int b = j & 1;
        if (leader) {
          const uint32_t vb = base + kSmemV + b * 2 * kKVHalf;
#pragma unroll
          for (int k = 0; k < 4; ++k) {                       // 16 keys per MMA
            const uint64_t dp = smem_desc_sw128(base + kSmemP + k * 32, 16, 1024);
            const uint64_t dv = smem_desc_sw128(vb + k * 2048, kKVHalf, 1024);
            tc_mma_f16(tmem + 128, dp, dv, id_o, (j > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(&bars->o_done);
          tc_commit(&bars->kv_empty[b]);
        }
        __syncwarp();
        if (j + 2 < tiles) {
          ok = wait(&bars->kv_empty[b], (j >> 1) & 1);
          if (!ok) break;
          load_tile(j + 2);
        }
      }
      if (!ok && leader) {
        record_error(a.status, PKV_ETIMEOUT);
        bars->abort_flag = 1;
      }
      // every TMA load issued must land before the CTA may exit
      if (leader) {
        for (int j = 0; j < tiles && j < 2; ++j) {
          const int last = ((tiles - 1 - j) >> 1) << 1 | j;   // last tile that used buffer j
          mbar_wait_bounded(&bars->kv_full[j], (last >> 1) & 1);
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax, one row per thread
    const int r = tid, i = r / G, g = r % G;
    const bool live = t0 + i < a.q_len;
    const int pos = n - a.q_len + t0 + i;                       // this query's last visible key
    const float qs = a.qk_scale_log2;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float mref = -INFINITY, lsum = 0.f;
    bool ok = true;
    // waits and TMEM accesses stay warp-uniform (tcgen05.ld/st are .sync.aligned)
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      const bool got = mbar_wait_bounded(bar, parity);
      return __all_sync(0xffffffffu, got) && !bars->abort_flag;
    };
    for (int j = 0; j < tiles; ++j) {
      const int b = j & 1;
      if (!wait(&bars->s_full[b], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[kN];
      tmem_ld64_sync(tmem + lane_base + b * kN, sv);
      tc_fence_before();
      mbar_arrive(&bars->s_free[b]);
      // scale, causal mask, row max (8 partial maxima: short dependency chains)
      const int kpos0 = j * kN;
      float mp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mp[e] = -INFINITY;
      if (__all_sync(0xffffffffu, live && kpos0 + kN - 1 <= pos)) {
        // the warp's rows see every key of the tile: no mask
#pragma unroll
        for (int c = 0; c < kN; ++c) {
          sv[c] *= qs;
          mp[c & 7] = fmaxf(mp[c & 7], sv[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kN; ++c) {
          const bool vis = live && kpos0 + c <= pos;
          sv[c] = vis ? sv[c] * qs : -INFINITY;
          mp[c & 7] = fmaxf(mp[c & 7], sv[c]);
        }
      }
      const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                             fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      bool rescale = false;
      float alpha = 1.f;
      if (mx > mref + 8.f) {            // also the first visible key (mref = -inf)
        alpha = exp2f(mref - mx);       // 0 when mref = -inf
        mref = mx;
        rescale = j > 0;
      }
      const float ref = mref == -INFINITY ? 0.f : mref;
      float pp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) pp[e] = 0.f;
      uint32_t pk[kN / 2];
#pragma unroll
      for (int c = 0; c < kN; c += 2) {
        const float p0 = exp2f(sv[c] - ref), p1 = exp2f(sv[c + 1] - ref);
        pp[(c >> 1) & 7] += p0 + p1;
        pk[c / 2] = pack2<kBf16>(p0, p1);
      }
      const float ps = ((pp[0] + pp[1]) + (pp[2] + pp[3])) + ((pp[4] + pp[5]) + (pp[6] + pp[7]));
      lsum = lsum * alpha + ps;
      // P_{j-1} must be consumed (and O stable) before P_j and any rescale
      if (j > 0) {
        if (!wait(&bars->o_done, (j - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? alpha : 1.f;
#pragma unroll
        for (int c = 0; c < kD; c += 32) {
          float o[32];
          tmem_ld32(tmem + lane_base + 128 + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= f;
          tmem_st32(tmem + lane_base + 128 + c, o);
        }
        tmem_st_wait();
      }
      // keys past the sequence end in this tile: zero their V rows (0 * NaN guard)
      const int valid = n - kpos0;
      if (valid < kN) {
        uint8_t* vbuf = sm + kSmemV + b * 2 * kKVHalf;
        for (int e = r; e < (kN - valid) * 16; e += 128) {
          const int row = valid + e / 16, c16 = e % 16;
          *reinterpret_cast<uint4*>(vbuf + (c16 >> 3) * kKVHalf + sw128(row, c16 & 7)) =
              make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(sm + kSmemP + sw128(r, c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    // epilogue: O row / l -> out (every lane reads TMEM; live rows store)
    if (ok && tiles > 0 && wait(&bars->o_done, (tiles - 1) & 1)) {
      tc_fence_after();
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      const size_t orow = (((size_t)s * a.q_len + t0 + i) * a.Hq + (size_t)hkv * G + g) * kD;
#pragma unroll
      for (int c = 0; c < kD; c += 32) {
        float o[32];
        tmem_ld32(tmem + lane_base + 128 + c, o);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            store_from_float(a.out, orow + c + e, a.out_dtype, o[e] * inv);
        }
      }
    } else if (tiles == 0 && live) {
      const size_t orow = (((size_t)s * a.q_len + t0 + i) * a.Hq + (size_t)hkv * G + g) * kD;
      for (int e = 0; e < kD; ++e) store_from_float(a.out, orow + e, a.out_dtype, 0.f);
    } else if (!ok || tiles > 0) {
      record_error(a.status, PKV_ETIMEOUT);
      bars->abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t prefill_tc_smem_bytes() { return kSmemBytes + sizeof(Bars) + kAlignSlack; }

bool prefill_tc_supported(int kv_dtype, int q_dtype, int BS, int D, int G) {
  return (kv_dtype == PKV_BF16 || kv_dtype == PKV_F16) && q_dtype == kv_dtype && D == kD &&
         (BS == 16 || BS == 32 || BS == 64) && G >= 1 && G <= kM && kM % G == 0;
}

cudaError_t launch_prefill_tc(const CUtensorMap* map, const DecodeArgs& a, cudaStream_t stream) {
  const int QT = kM / a.G;
  const int qtiles = (a.q_len + QT - 1) / QT;
  if (qtiles == 0 || a.B == 0) return cudaSuccess;
  const size_t smem = prefill_tc_smem_bytes();
  cudaError_t e;
  dim3 grid(qtiles, a.Hkv, a.B);
  if (a.kv_dtype == PKV_BF16) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess) prefill_tc_kernel<true><<<grid, 160, smem, stream>>>(*map, a);
  } else {
    e = cudaFuncSetAttribute(prefill_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess) prefill_tc_kernel<false><<<grid, 160, smem, stream>>>(*map, a);
  }
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace pkv
