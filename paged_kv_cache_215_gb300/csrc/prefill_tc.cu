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
//   CTA (pair of query tiles, KV head hkv, sequence s).  A query tile is
//   M = 128 rows = 128/G query tokens x G heads, staged once in shared memory
//   (128-byte swizzled).  Both tiles of the pair consume every K/V tile, so
//   each 64-token K/V tile loaded from L2 feeds 256 query rows: the loads
//   from L2 into shared memory, not the tensor cores, bound a one-tile CTA.
//   K/V tiles arrive by TMA from the pool (one box per block and 64-column
//   half) into a 4-stage ring.  Per query tile t and key tile j:
//     S_tj = Q_t K_j^T      tcgen05.mma M128 N64 K128 -> TMEM (two S buffers per
//                           query tile, so S_t,j+1 runs while the softmax of S_tj does)
//     softmax               one warpgroup per query tile, one thread per row:
//                           tcgen05.ld of its S row, scale, causal mask, running
//                           max / sum, P_tj -> shared memory (bf16/f16)
//     O_t += P_tj V_j       tcgen05.mma M128 N128 K64, V as the MN-major operand
//   O_t lives in TMEM for the whole key range (512 columns: 256 per query tile).
//   The softmax keeps a reference max per row and rescales the row of O
//   (tcgen05.ld/st) only when the true max exceeds it by more than 8 (log2
//   units); P is then at most 2^8, exact in fp32 accumulation, and O and the
//   row sum share the same reference.
// One thread of warp 8 issues the S MMAs, one thread of warp 9 the P V MMAs:
// a single thread issues a UMMA about every 70 cycles, well short of what an
// N = 64 tile takes on the tensor core, and two issuers nearly double the
// rate.  Warp 10 issues the K/V loads (16 boxes per tile at block size 16,
// from 16 lanes), off the MMA issuers' path.  mbarriers (all waits bounded)
// pass the tiles between the roles; a stage is refilled once both issuers'
// MMAs reading it have completed.
#include "device.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kM = 128;                      // query rows per query tile (one UMMA M)
constexpr int kQT = 2;                       // query tiles per CTA
constexpr int kN = 64;                       // keys per K/V tile
constexpr int kStages = 4;                   // K/V tiles in flight
constexpr int kSoftmaxWarps = 4 * kQT;
constexpr int kWarpS = kSoftmaxWarps;        // S MMAs
constexpr int kWarpPV = kSoftmaxWarps + 1;   // P V MMAs
constexpr int kWarpTMA = kSoftmaxWarps + 2;  // K/V loads
constexpr int kThreads = 32 * (kSoftmaxWarps + 3);
constexpr uint32_t kHalf = 16384;            // 128 rows x 128 B: one 64-column half of Q
constexpr uint32_t kKVHalf = kN * 128;       // 64 rows x 128 B
constexpr uint32_t kStageBytes = 4 * kKVHalf;        // K halves 0, 1 then V halves 0, 1
constexpr uint32_t kSmemQ = 0;                        // [query tile][half]
constexpr uint32_t kSmemKV = kSmemQ + kQT * 2 * kHalf;
constexpr uint32_t kSmemP = kSmemKV + kStages * kStageBytes;   // [query tile] 128 rows x 64 keys
constexpr uint32_t kSmemBytes = kSmemP + kQT * kM * 128;
constexpr uint32_t kTmemCols = 512;          // query tile t: S0 [256t, +64) S1 [+64, +128) O [+128, +256)
constexpr uint32_t kAlignSlack = 1024;       // the tiles start on a 1024-byte boundary

struct Bars {
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[kQT][2], s_free[kQT][2], p_full[kQT], o_done[kQT];
  uint32_t tmem;
  volatile int abort_flag;
};

__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}

// Key tiles query tile `qt` needs: up to the one holding its last row's last key.
__device__ __forceinline__ int key_tiles(const DecodeArgs& a, int n, int qt) {
  const int QT = kM / a.G, t0 = qt * QT;
  if (t0 >= a.q_len) return 0;
  const int last_tok = min(t0 + QT, a.q_len) - 1;
  const int p_last = n - a.q_len + last_tok;
  return p_last >= 0 ? (p_last + kN) / kN : 0;
}

template <bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  Bars* bars = reinterpret_cast<Bars*>(sm + kSmemBytes);
  const uint32_t base = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hkv = blockIdx.y, s = blockIdx.z;
  const int G = a.G, QT = kM / G;                 // query tokens per query tile

  int n = __ldg(a.seq_lens + s);
  const int cap = a.max_blocks * a.BS;
  if (n < 0 || n > cap) {
    if (tid == 0) record_error(a.status, PKV_EBOUNDS);
    n = n < 0 ? 0 : cap;
  }
  int tiles[kQT];
#pragma unroll
  for (int t = 0; t < kQT; ++t) tiles[t] = key_tiles(a, n, blockIdx.x * kQT + t);
  int T = 0;                                      // key tiles the CTA loads
#pragma unroll
  for (int t = 0; t < kQT; ++t) T = max(T, tiles[t]);

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 2);          // one commit from each issuer
    }
    for (int t = 0; t < kQT; ++t) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bars->s_full[t][b], 1);
        mbar_init(&bars->s_free[t][b], 128);
      }
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->o_done[t], 1);
    }
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpS) {
    tmem_alloc(&bars->tmem, kTmemCols);
    tmem_relinquish();
  }
  // Q tiles: thread (t, r) stages row r = (token t0 + r / G, head hkv*G + r % G), swizzled
  if (warp < kSoftmaxWarps) {
    const int t = warp / 4, r = tid - 128 * t, i = r / G, g = r % G;
    const int tok = (blockIdx.x * kQT + t) * QT + i;
    const bool live = tok < a.q_len;
    const size_t qrow = ((size_t)s * a.q_len + tok) * a.Hq + (size_t)hkv * G + g;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                      (live ? qrow : 0) * kD);
    uint8_t* qdst = sm + kSmemQ + t * 2 * kHalf;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = live ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(qdst + (c >> 3) * kHalf + sw128(r, c & 7)) = v;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp >= kSoftmaxWarps) {
    // ------------------------------------------------------------ issuers
    // Each issuer warp walks its loop and waits as a whole (so it stays
    // converged); its lane 0 issues the MMAs and the commits.
    if (T > 0) {
      const bool leader = lane == 0;
      const int bpt = kN / a.BS;                               // blocks per key tile
      const int nblk = (n + a.BS - 1) / a.BS;
      const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
      int last_load[kStages];                                  // last key tile requested per stage
#pragma unroll
      for (int i = 0; i < kStages; ++i) last_load[i] = -1;
      // block ids of the sequence, 32 at a time: lane i holds entry id_base + i
      // (one table read per 32 blocks instead of a dependent read per TMA)
      int ids = 0, id_base = -1;
      auto load_tile = [&](int j) {
        const int st = j % kStages;
        last_load[st] = j;
        const int first = j * bpt;                              // < nblk for every tile loaded
        if (id_base < 0 || first + bpt > id_base + 32) {
          id_base = first;
          ids = id_base + lane < nblk ? __ldg(trow + id_base + lane) : 0;
        }
        // lane l < 4 * bpt loads one box: block l / 4 of the tile, K or V ((l / 2) & 1),
        // 64-column half l & 1 (boxes issued from several lanes at once)
        // blocks past the sequence's last one are replaced by its last block:
        // their keys are masked and their V rows zeroed before use
        const int jb = min(first + (lane >> 2), nblk - 1);
        int blk = __shfl_sync(0xffffffffu, ids, jb - id_base);
        if (leader) mbar_arrive_expect_tx(&bars->kv_full[st], kStageBytes);
        __syncwarp();
        if (lane < 4 * bpt) {
          if (blk < 0 || blk >= a.num_blocks) {
            record_error(a.status, PKV_EBOUNDS);
            blk = 0;
          }
          const int kv = (lane >> 1) & 1, h = lane & 1;
          const int z = (blk * 2 + kv) * a.L + a.layer;
          tma_load_3d(sm + kSmemKV + st * kStageBytes + (kv * 2 + h) * kKVHalf +
                          (lane >> 2) * a.BS * 128,
                      &tmap, &bars->kv_full[st], h * 64, hkv * a.BS, z);
        }
      };
      // keys past the sequence end in the tile (only its last): zero their V
      // rows, so that P = 0 never meets an unwritten (possibly NaN) slot
      auto zero_tail = [&](int j) {
        const int valid = n - j * kN;
        if (valid >= kN) return;
        uint8_t* vbuf = sm + kSmemKV + (j % kStages) * kStageBytes + 2 * kKVHalf;
        for (int e = lane; e < (kN - valid) * 16; e += 32) {
          const int row = valid + e / 16, c16 = e % 16;
          *reinterpret_cast<uint4*>(vbuf + (c16 >> 3) * kKVHalf + sw128(row, c16 & 7)) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      };
      const uint32_t id_s = kBf16 ? idesc_bf16_f32(kM, kN, false, false)
                                  : (idesc_bf16_f32(kM, kN, false, false) & ~((7u << 7) | (7u << 10)));
      const uint32_t id_o = kBf16 ? idesc_bf16_f32(kM, kD, false, true)
                                  : (idesc_bf16_f32(kM, kD, false, true) & ~((7u << 7) | (7u << 10)));
      // Descriptors of the shared-memory base; a tile's descriptor adds its byte
      // offset / 16 to the start-address field (shared addresses stay below 256 KB,
      // so the 14-bit field never carries).
      const uint64_t d_k = smem_desc_sw128(base, 16, 1024);      // K-major operands
      const uint64_t d_v = smem_desc_sw128(base, kKVHalf, 1024); // V: MN-major
      auto issue_s = [&](int j, int t) {
        if (!leader) return;
        const int b = j & 1;
        const uint64_t kb = d_k + ((kSmemKV + (j % kStages) * kStageBytes) >> 4);
        const uint64_t qb = d_k + ((kSmemQ + t * 2 * kHalf) >> 4);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = ((k >> 2) * kHalf + (k & 3) * 32) >> 4;
          const uint32_t offk = ((k >> 2) * kKVHalf + (k & 3) * 32) >> 4;
          tc_mma_f16(tmem + t * 256 + b * kN, qb + off, kb + offk, id_s, k > 0);
        }
        tc_commit(&bars->s_full[t][b]);
      };
      auto issue_pv = [&](int j, int t) {
        if (!leader) return;
        const uint64_t vb = d_v + ((kSmemKV + (j % kStages) * kStageBytes + 2 * kKVHalf) >> 4);
        const uint64_t pb = d_k + ((kSmemP + t * kM * 128) >> 4);
#pragma unroll
        for (int k = 0; k < 4; ++k)                            // 16 keys per MMA
          tc_mma_f16(tmem + t * 256 + 128, pb + k * 2, vb + k * 128, id_o,
                     (j > 0 || k > 0) ? 1u : 0u);
        tc_commit(&bars->o_done[t]);
      };
      // every lane waits; the warp agrees on the outcome
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        const bool got = mbar_wait_bounded(bar, parity);
        return __all_sync(0xffffffffu, got) && !bars->abort_flag;
      };
      bool ok = true;
      if (warp == kWarpTMA) {
        for (int j = 0; j < T && j < kStages; ++j) load_tile(j);
        // key tile k goes into the stage of tile k - kStages once both issuers'
        // MMAs reading that tile have completed
        for (int k = kStages; k < T && ok; ++k) {
          ok = wait(&bars->kv_empty[(k - kStages) % kStages], ((k - kStages) / kStages) & 1);
          if (!ok) break;
          load_tile(k);
        }
      } else if (warp == kWarpS) {
        for (int j = 0; j < T && ok; ++j) {
          ok = wait(&bars->kv_full[j % kStages], (j / kStages) & 1);
          // S_tj reuses the TMEM buffer of S_t,j-2: its softmax must have read it
          for (int t = 0; t < kQT && ok; ++t)
            if (j < tiles[t] && j >= 2) ok = wait(&bars->s_free[t][j & 1], ((j - 2) >> 1) & 1);
          if (!ok) break;
          zero_tail(j);
          tc_fence_after();
          for (int t = 0; t < kQT; ++t)
            if (j < tiles[t]) issue_s(j, t);
          if (leader) tc_commit(&bars->kv_empty[j % kStages]);  // S_j has read K_j
          __syncwarp();
        }
      } else if (warp == kWarpPV) {
        for (int j = 0; j < T && ok; ++j) {
          for (int t = 0; t < kQT && ok; ++t) {
            if (j >= tiles[t]) continue;
            ok = wait(&bars->p_full[t], j & 1);
            if (!ok) break;
            tc_fence_after();
            issue_pv(j, t);
          }
          if (!ok) break;
          if (leader) tc_commit(&bars->kv_empty[j % kStages]);  // P_j V_j has read V_j
          __syncwarp();
        }
      }
      if (!ok && leader) {
        record_error(a.status, PKV_ETIMEOUT);
        bars->abort_flag = 1;
      }
      // every TMA load issued must land before the CTA may exit.  A stage's key
      // tile k is requested only after tile k - kStages landed and was read, so
      // waiting for the phase of the last tile requested into it covers all.
      if (leader && warp == kWarpTMA) {
        for (int st = 0; st < kStages; ++st)
          if (last_load[st] >= 0)
            mbar_wait_bounded(&bars->kv_full[st], (last_load[st] / kStages) & 1);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax, one row per thread
    const int t = warp / 4, r = tid - 128 * t, i = r / G, g = r % G;
    const int tok = (blockIdx.x * kQT + t) * QT + i;
    const bool live = tok < a.q_len;
    const int pos = n - a.q_len + tok;                          // this query's last visible key
    const int my_tiles = tiles[t];
    const float qs = a.qk_scale_log2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tcol = tmem + lane_base + t * 256;
    uint8_t* pbuf = sm + kSmemP + t * kM * 128;
    float mref = -INFINITY, lsum = 0.f;
    bool ok = true;
    // waits and TMEM accesses stay warp-uniform (tcgen05.ld/st are .sync.aligned)
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      const bool got = mbar_wait_bounded(bar, parity);
      return __all_sync(0xffffffffu, got) && !bars->abort_flag;
    };
    for (int j = 0; j < my_tiles; ++j) {
      const int b = j & 1;
      if (!wait(&bars->s_full[t][b], (j >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[kN];
      tmem_ld64_sync(tcol + b * kN, sv);
      tc_fence_before();
      mbar_arrive(&bars->s_free[t][b]);
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
        if (!wait(&bars->o_done[t], (j - 1) & 1)) {
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
          tmem_ld32(tcol + 128 + c, o);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= f;
          tmem_st32(tcol + 128 + c, o);
        }
        tmem_st_wait();
      }
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(pbuf + sw128(r, c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full[t]);
    }
    // epilogue: O row / l -> out (every lane reads TMEM; live rows store)
    const size_t orow = (((size_t)s * a.q_len + tok) * a.Hq + (size_t)hkv * G + g) * kD;
    if (ok && my_tiles > 0 && wait(&bars->o_done[t], (my_tiles - 1) & 1)) {
      tc_fence_after();
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
      for (int c = 0; c < kD; c += 32) {
        float o[32];
        tmem_ld32(tcol + 128 + c, o);
        tmem_ld_wait();
        if (live) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            store_from_float(a.out, orow + c + e, a.out_dtype, o[e] * inv);
        }
      }
    } else if (my_tiles == 0) {
      if (live)
        for (int e = 0; e < kD; ++e) store_from_float(a.out, orow + e, a.out_dtype, 0.f);
    } else {
      record_error(a.status, PKV_ETIMEOUT);
      bars->abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpS) tmem_dealloc(tmem, kTmemCols);
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
  dim3 grid((qtiles + kQT - 1) / kQT, a.Hkv, a.B);
  if (a.kv_dtype == PKV_BF16) {
    e = cudaFuncSetAttribute(prefill_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess) prefill_tc_kernel<true><<<grid, kThreads, smem, stream>>>(*map, a);
  } else {
    e = cudaFuncSetAttribute(prefill_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e == cudaSuccess) prefill_tc_kernel<false><<<grid, kThreads, smem, stream>>>(*map, a);
  }
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace pkv
