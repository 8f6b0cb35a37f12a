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
//   each 64-token K/V tile loaded from L2 feeds 256 query rows.  K/V tiles
//   arrive by TMA from the pool (one box per block and K/V, both 64-column
//   halves: bs x 256 bytes) into a 5-stage ring.  Per query tile t and key tile j:
//     S_tj = Q_t K_j^T      tcgen05.mma M128 N64 K128 -> TMEM (two buffers per
//                           query tile, so S_t,j+1 runs while the softmax of S_tj does)
//     softmax               one warpgroup per query tile, one thread per row:
//                           tcgen05.ld of its S row, causal mask, running max / sum,
//                           P_tj written back over S_tj in TMEM (tcgen05.st)
//     O_t += P_tj V_j       tcgen05.mma M128 N128 K64 with P read from TMEM and V
//                           (the MN-major operand) from shared memory
//   bf16 P is stored as two bf16 terms, hi = bf16(p) and lo = bf16(p - hi), and
//   both are multiplied with V: a single bf16 P would carry up to 2^-8 of
//   relative error, which a sharply peaked softmax passes to the output whole.
//   O_t lives in TMEM for the whole key range (512 columns: 256 per query tile).
//   The softmax keeps a reference max per row and rescales the row of O
//   (tcgen05.ld/st) only when the true max exceeds it by more than 8 (log2
//   units); P is then at most 2^8, exact in fp32 accumulation, and O and the
//   row sum share the same reference.
// Issuers, one thread each: warp 8 + t issues query tile t's S MMAs, warp 10 + t
// its P V MMAs (a single thread issues a UMMA about every 70 cycles, short of
// what these tiles take on the tensor core; issuers in different warps multiply
// the rate), warp 12 the K/V loads (8 boxes per tile at block size 16, from 8
// lanes).  One warp's TMA requests stream at about 17 B/clk into an SM, two
// warps' at the HBM rate: in the shared-prefix pass, where the loads are on the
// critical path, warp 13 takes every other key tile (in chunked prefill it
// stays idle: its polling there would cost the softmax warps issue slots).  mbarriers (all waits bounded) pass the tiles between the roles; a
// stage is refilled once every issuer's MMAs reading it have completed.
#include "device.cuh"
#include "launch.h"

namespace pkv {
namespace {

constexpr int kD = 128;
constexpr int kM = 128;                      // query rows per query tile (one UMMA M)
constexpr int kQT = 2;                       // query tiles per CTA
constexpr int kN = 64;                       // keys per K/V tile
constexpr int kSoftmaxWarps = 4 * kQT;
constexpr int kWarpS = kSoftmaxWarps;        // S MMAs of query tile t: warp kWarpS + t
constexpr int kWarpPV = kWarpS + kQT;        // P V MMAs of query tile t: warp kWarpPV + t
constexpr int kWarpTMA = kWarpPV + kQT;      // K/V loads
constexpr int kWarpConv = kWarpTMA + 1;      // E4M3 pools: warps converting K/V tiles to f16;
                                             // 16-bit pools: the second producer
constexpr int kIssuers = 2 * kQT;            // MMA issuers committing each stage's release
constexpr uint32_t kHalf = 16384;            // 128 rows x 128 B: one 64-column half of Q
constexpr uint32_t kKVHalf = kN * 128;       // 64 rows x 128 B
constexpr uint32_t kStageBytes = 4 * kKVHalf;        // K tile (16 KB) then V tile (16 KB)
constexpr uint32_t kStage8Bytes = 2 * kKVHalf;       // an E4M3 tile: K then V, 128 B a key
constexpr uint32_t kSmemQ = 0;                        // [query tile][half]
constexpr uint32_t kSmemKV = kSmemQ + kQT * 2 * kHalf;
constexpr uint32_t kTmemCols = 512;          // query tile t: S/P0 [256t, +64) S/P1 [+64, +128) O [+128, +256)
constexpr uint32_t kAlignSlack = 1024;       // the tiles start on a 1024-byte boundary
constexpr int kMaxStages = 6;

// Per pool dtype.  bf16 / f16: TMA fills kStages tiles the MMAs read directly.
// E4M3: TMA lands the E4M3 tile (one 128-byte line per key: half the boxes) in
// the V half of its stage, and kConvWarps warps convert it in place into the
// stage's f16 K and V; the MMAs then run as for an f16 pool.  Every E4M3 value is
// an f16 value, so with per-tensor scales the conversion is exact (k_scale rides
// on the softmax scale, v_scale on the output); per-block scales are multiplied
// in before the f16 rounding (relative error 2^-11).
template <int KVT>
struct PfCfg {
  static constexpr bool kFp8 = KVT == PKV_FP8_E4M3;
  static constexpr bool kBf16 = KVT == PKV_BF16;      // else f16 operands (f16 and E4M3 pools)
  static constexpr int kStages = 5;                   // K/V tiles in flight
  static constexpr int kConvWarps = kFp8 ? 3 : 0;
  // producer warps (16-bit pools: a second one, after warp 12, that the
  // shared-prefix pass uses; E4M3 tiles are half the bytes and their converters
  // fill the warp budget)
  static constexpr int kProducers = kFp8 ? 1 : 2;
  static constexpr int kThreads = 32 * (kWarpConv + kConvWarps + kProducers - 1);
  static constexpr uint32_t kSmemBytes = kSmemKV + kStages * kStageBytes;
};

struct Bars {
  uint64_t kv_full[kMaxStages], kv_empty[kMaxStages];
  uint64_t s8_full[kMaxStages];               // E4M3: the stage's E4M3 tile has landed
  uint64_t s_full[kQT][2], p_full[kQT][2], p_free[kQT][2], o_done[kQT];
  uint64_t o_final[kQT];                      // query tile t's last P V has completed
  uint64_t v_zeroed;                          // the tail tile's V rows past the end are zero
  uint64_t q_ready;                           // the Q tiles are staged
  uint64_t eref_ready;                        // E4M3 per-block scales: the reference exponent is in
  int eref[4];                                // per converter warp: largest exponent of the V scales
  uint32_t tmem;
  volatile int abort_flag;
};
// the ring, the barriers and the alignment slack fit the 227 KB a CTA may opt into
static_assert(PfCfg<PKV_BF16>::kSmemBytes + sizeof(Bars) + kAlignSlack <= 227u * 1024u, "smem");
static_assert(PfCfg<PKV_FP8_E4M3>::kSmemBytes + sizeof(Bars) + kAlignSlack <= 227u * 1024u, "smem");
// 16 warps at most: four to a scheduler keeps 128 registers a thread
static_assert(PfCfg<PKV_FP8_E4M3>::kThreads <= 512, "threads");
static_assert(PfCfg<PKV_BF16>::kThreads <= 512, "threads");

// Two FP32 lanes in one 64-bit register, for the f32x2 instructions (each lane
// rounds exactly as the scalar instruction does).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

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

template <int KVT>
__global__ void __launch_bounds__(PfCfg<KVT>::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeArgs a) {
  using C = PfCfg<KVT>;
  constexpr bool kBf16 = C::kBf16, kFp8 = C::kFp8;
  constexpr int kStages = C::kStages;
  constexpr bool kSplitP = kBf16;            // f16 P (11 bits) needs no low term
  // f16 P is 2^(s - ref + kPOff) <= 2^15: weights down to 2^-21 of the row's
  // reference stay normal f16 numbers (a long tail of small weights would
  // otherwise round in f16's subnormal range); the factor cancels in O / l.
  // bf16 P has fp32's exponent range and needs none.
  constexpr float kPOff = kSplitP ? 0.f : 7.f;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sm = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  Bars* bars = reinterpret_cast<Bars*>(sm + C::kSmemBytes);
  const uint32_t base = smem_u32(sm);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // shared-prefix mode: query token i is sequence i, one key table (the prefix),
  // blockIdx.y cuts the key range into a.S splits
  const bool casc = a.key_limit != nullptr;
  // blockIdx.x = KV head; y = sequence (shared-prefix mode: key split); z = pair of
  // query tiles, counted from the chunk's end in chunked prefill: the pairs nearest
  // the end see the most keys and are launched first, so the last, partial wave of
  // CTAs holds the shortest ones
  const int hkv = blockIdx.x, s = casc ? 0 : blockIdx.y, split = casc ? blockIdx.y : 0;
  const int pair = casc ? (int)blockIdx.z : (int)(gridDim.z - 1 - blockIdx.z);
  const int G = a.G, QT = kM / G;                 // query tokens per query tile

  // shared-prefix mode: the prefix length comes with the launch (nothing launched
  // before it in the stream needs to have finished)
  int n = casc ? a.casc_len : __ldg(a.seq_lens + s);
  const int cap = a.max_blocks * a.BS;
  if (n < 0 || n > cap) {
    if (tid == 0) record_error(a.status, PKV_EBOUNDS);
    n = n < 0 ? 0 : cap;
  }
  // key tiles jt0 .. jt0 + T - 1 of the sequence; local tile j is global tile jt0 + j
  int tiles[kQT], jt0 = 0;                        // key tiles each slot computes
  int T = 0;                                      // key tiles the CTA loads
  if (casc) {
    const int nt = (n + kN - 1) / kN;
    jt0 = (int)((long long)split * nt / a.S);
    const int jt1 = (int)((long long)(split + 1) * nt / a.S);
#pragma unroll
    for (int t = 0; t < kQT; ++t)
      tiles[t] = (pair * kQT + t) * QT < a.q_len ? jt1 - jt0 : 0;
  } else {
#pragma unroll
    for (int t = 0; t < kQT; ++t) tiles[t] = key_tiles(a, n, pair * kQT + t);
  }
#pragma unroll
  for (int t = 0; t < kQT; ++t) T = max(T, tiles[t]);
  // The K/V ring: kStages stages after the Q tiles; a CTA whose second query
  // tile is empty (a single 128-row tile: the shared-prefix pass, or the last
  // CTA of an odd tile count) also puts one in that tile's Q space, so one more
  // K/V tile is in flight while the memory system answers.
  const int nst = (T > 0 && tiles[kQT - 1] == 0) ? kStages + 1 : kStages;
  auto stage_off = [&](int st) -> uint32_t {
    return st < kStages ? kSmemKV + (uint32_t)st * kStageBytes : kSmemQ + (kQT - 1) * 2 * kHalf;
  };
  // the sequence's last key tile, if it is ragged and this CTA reads it (local index)
  const int jg_tail = (n % kN != 0) ? (n - 1) / kN : -1;
  const int j_tail = (jg_tail >= jt0 && jg_tail < jt0 + T) ? jg_tail - jt0 : -1;

  if (tid == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&bars->kv_full[i], kFp8 ? C::kConvWarps : 1);   // the converters, or TMA
      mbar_init(&bars->kv_empty[i], kIssuers);   // one commit from each MMA issuer
    }
    if (kFp8)
      for (int i = 0; i < kMaxStages; ++i) mbar_init(&bars->s8_full[i], 1);
    for (int t = 0; t < kQT; ++t) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&bars->s_full[t][b], 1);
        mbar_init(&bars->p_full[t][b], 128);
        mbar_init(&bars->p_free[t][b], 1);
      }
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_final[t], 1);
    }
    mbar_init(&bars->v_zeroed, 1);
    mbar_init(&bars->q_ready, 32 * kSoftmaxWarps);
    mbar_init(&bars->eref_ready, kFp8 ? C::kConvWarps : 1);
    bars->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpTMA) {
    tmem_alloc(&bars->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  // shared-prefix mode runs one wave: once every CTA is resident, the suffix
  // decode launched behind it may be scheduled (it reads nothing this kernel
  // writes, and waits for it before it writes); it takes SMs as CTAs retire
  if (casc) grid_launch_dependents();
  // Q tiles, staged while the first K/V tiles are in flight (the S issuers wait
  // for q_ready): thread (t, r) stages row r = (token t0 + r / G, head hkv*G + r % G), swizzled.
  // E4M3 pools run f16 MMAs: a bf16 q row is scaled by 2^q_e (f16_fit_exponent of
  // its largest |q|) before the f16 rounding, exactly, and the same thread's
  // softmax takes 2^-q_e onto the scale.
  int q_e = 0;
  if (warp < kSoftmaxWarps) {
    const int t = warp / 4, r = tid - 128 * t, i = r / G, g = r % G;
    // an empty tile is not staged: its S MMAs never run, and its Q space may
    // hold the ring's extra stage
    const int tok = (pair * kQT + t) * QT + i;
    const bool live = tok < a.q_len;
    const bool staged = tiles[t] > 0;
    const size_t qrow = ((size_t)s * a.q_len + tok) * a.Hq + (size_t)hkv * G + g;
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) +
                                                      (live ? qrow : 0) * kD);
    uint8_t* qdst = sm + kSmemQ + t * 2 * kHalf;
    // a negative softmax scale is moved onto Q (an exact sign flip), so that the
    // softmax may take its row max over the unscaled scores
    const uint32_t flip = a.qk_scale_log2 < 0.f ? 0x80008000u : 0u;
    const bool to_f16 = kFp8 && a.q_dtype == PKV_BF16;
    float qscale = 1.f;
    if (to_f16 && live) {
      float amax = 0.f;
#pragma unroll 4
      for (int c = 0; c < 16; ++c) {
        uint4 v = __ldg(src + c);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack2<true>(w[e]);
          amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
      q_e = f16_fit_exponent(amax);
      qscale = pow2i(q_e);
    }
#pragma unroll
    for (int c = 0; c < 16 && staged; ++c) {
      uint4 v = live ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      if (to_f16) {
        // the MMAs of an E4M3 pool run on f16 operands: q bf16 x 2^q_e -> f16
        uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack2<true>(w[e]);
          w[e] = pack_f16(f.x * qscale, f.y * qscale);
        }
      }
      v.x ^= flip;
      v.y ^= flip;
      v.z ^= flip;
      v.w ^= flip;
      *reinterpret_cast<uint4*>(qdst + (c >> 3) * kHalf + sw128(r, c & 7)) = v;
    }
    fence_proxy_async_smem();
    mbar_arrive(&bars->q_ready);
  }

  if (warp >= kSoftmaxWarps) {
    // ------------------------------------------------------------ issuers
    // Each issuer warp walks its loop and waits as a whole (so it stays
    // converged); its lane 0 issues the MMAs and the commits.
    if (T > 0) {
      const bool leader = lane == 0;
      // every lane waits; the warp agrees on the outcome
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        const bool got = mbar_wait_bounded(bar, parity);
        return __all_sync(0xffffffffu, got) && !bars->abort_flag;
      };
      const uint32_t id_s = kBf16 ? idesc_bf16_f32(kM, kN, false, false)
                                  : (idesc_bf16_f32(kM, kN, false, false) & ~((7u << 7) | (7u << 10)));
      const uint32_t id_o = kBf16 ? idesc_bf16_f32(kM, kD, false, true)
                                  : (idesc_bf16_f32(kM, kD, false, true) & ~((7u << 7) | (7u << 10)));
      // Descriptors of the shared-memory base; a tile's descriptor adds its byte
      // offset / 16 to the start-address field (shared addresses stay below 256 KB,
      // so the 14-bit field never carries).
      // Q: K-major, 8-row groups 1 KB apart.  16-bit K/V tiles: 8-key groups of
      // [half 0 | half 1] atoms, so K (K-major) has its groups 2 KB apart and V
      // (MN-major) its halves 1 KB and its groups 2 KB apart.  E4M3 tiles are
      // converted into 64-row halves: K groups 1 KB apart, V halves 8 KB apart.
      const uint64_t d_k = smem_desc_sw128(base, 16, 1024);
      const uint64_t d_kt = smem_desc_sw128(base, 16, kFp8 ? 1024 : 2048);
      const uint64_t d_v = kFp8 ? smem_desc_sw128(base, kKVHalf, 1024)
                                : smem_desc_sw128(base, 1024, 2048);
      bool ok = true;
      if (warp == kWarpTMA || (!kFp8 && warp >= kWarpConv)) {
        // producer prod of P loads key tiles prod, prod + P, ...
        const int P = casc ? C::kProducers : 1;
        const int prod = warp == kWarpTMA ? 0 : warp - kWarpConv + 1;
        const int bpt = kN / a.BS;                             // blocks per key tile
        const int nblk = (n + a.BS - 1) / a.BS;
        const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
        int last_load[kMaxStages];             // E4M3: last key tile requested per stage
#pragma unroll
        for (int i = 0; i < kMaxStages; ++i) last_load[i] = -1;
        // block ids of the sequence, 32 at a time: lane i holds entry id_base + i
        // (one table read per 32 blocks instead of a dependent read per box)
        int ids = 0, id_base = -1;
        auto load_tile = [&](int j) {
          const int st = j % nst;
          const int first = (jt0 + j) * bpt;                    // < nblk for every tile loaded
          if (id_base < 0 || first + bpt > id_base + 32) {
            id_base = first;
            ids = id_base + lane < nblk ? __ldg(trow + id_base + lane) : 0;
          }
          // lane l < 2 * bpt loads one box: block l / 2 of the tile, K or V (l & 1),
          // both 64-column halves (bs x 256 bytes).  Blocks past the sequence's
          // last one are replaced by its last block: their keys are masked and
          // their V rows zeroed before use.
          const int jb = min(first + (lane >> 1), nblk - 1);
          int blk = __shfl_sync(0xffffffffu, ids, jb - id_base);
          if (leader) mbar_arrive_expect_tx(&bars->kv_full[st], kStageBytes);
          __syncwarp();
          if (lane < 2 * bpt) {
            if (blk < 0 || blk >= a.num_blocks) {
              record_error(a.status, PKV_EBOUNDS);
              blk = 0;
            }
            const int kv = lane & 1;
            const int z = (blk * 2 + kv) * a.L + a.layer;
            tma_load_5d(sm + stage_off(st) + kv * 2 * kKVHalf +
                            (lane >> 1) * a.BS * 256,
                        &tmap, &bars->kv_full[st], 0, 0, 0, hkv * a.BS / 8, z);
          }
        };
        if constexpr (kFp8) {
          // E4M3: one box per block and K/V (128 one-byte columns: the whole row)
          // into the V half of the stage: E4M3 K where f16 V half 0 goes, E4M3 V
          // where half 1 goes; the converters then fill the stage in place
          auto load8 = [&](int j) {
            const int st = j % nst;
            last_load[st] = j;
            const int first = (jt0 + j) * bpt;
            if (id_base < 0 || first + bpt > id_base + 32) {
              id_base = first;
              ids = id_base + lane < nblk ? __ldg(trow + id_base + lane) : 0;
            }
            const int jb = min(first + (lane >> 1), nblk - 1);
            int blk = __shfl_sync(0xffffffffu, ids, jb - id_base);
            if (leader) mbar_arrive_expect_tx(&bars->s8_full[st], kStage8Bytes);
            __syncwarp();
            if (lane < 2 * bpt) {
              if (blk < 0 || blk >= a.num_blocks) {
                record_error(a.status, PKV_EBOUNDS);
                blk = 0;
              }
              const int kv = lane & 1;
              const int z = (blk * 2 + kv) * a.L + a.layer;
              tma_load_3d(sm + stage_off(st) + (2 + kv) * kKVHalf +
                              (lane >> 1) * a.BS * 128,
                          &tmap, &bars->s8_full[st], 0, hkv * a.BS, z);
            }
          };
          for (int j = 0; j < T && j < nst; ++j) load8(j);
          for (int k = nst; k < T && ok; ++k) {
            ok = wait(&bars->kv_empty[(k - nst) % nst], ((k - nst) / nst) & 1);
            if (!ok) break;
            load8(k);
          }
          if (leader)
            for (int st = 0; st < nst; ++st)
              if (last_load[st] >= 0)
                mbar_wait_bounded(&bars->s8_full[st], (last_load[st] / nst) & 1);
        } else {
        // key tile k goes into the stage of tile k - nst once every issuer's
        // MMAs reading that tile have completed (the issuers release the tiles in
        // order, whichever producer loaded them)
        for (int k = prod; prod < P && k < T && ok; k += P) {
          if (k >= nst) {
            ok = wait(&bars->kv_empty[(k - nst) % nst], ((k - nst) / nst) & 1);
            if (!ok) break;
          }
          load_tile(k);
        }
        // keys past the sequence end in its last tile: zero their V rows once the
        // tile has landed, so that P = 0 never meets an unwritten (possibly NaN) slot
        if (ok && j_tail >= 0 && j_tail % P == prod) {
          ok = wait(&bars->kv_full[j_tail % nst], (j_tail / nst) & 1);
          if (ok) {
            const int valid = n - (jt0 + j_tail) * kN;
            uint8_t* vbuf = sm + stage_off(j_tail % nst) + 2 * kKVHalf;
            for (int e = lane; e < (kN - valid) * 16; e += 32) {
              const int row = valid + e / 16, c16 = e % 16;
              *reinterpret_cast<uint4*>(vbuf + ((row >> 3) * 2 + (c16 >> 3)) * 1024 +
                                        sw128(row & 7, c16 & 7)) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (leader) mbar_arrive(&bars->v_zeroed);
          }
        }
        // every TMA load issued must land before the CTA may exit.  A stage's key
        // tile k is requested only after tile k - nst landed and was read, so
        // waiting for the phase of the last tile requested into each stage covers
        // all.  That wait belongs to the producer that requested it: with an odd
        // ring depth the producers take turns on a stage, and the other one's
        // earlier tile there is two or more phases back (its parity no longer
        // tells that phase from the current, incomplete one).
        if (leader)
          for (int st = 0; st < nst; ++st) {
            const int k_last = st < T ? st + (T - 1 - st) / nst * nst : -1;
            if (k_last >= 0 && k_last % P == prod)
              mbar_wait_bounded(&bars->kv_full[st], (k_last / nst) & 1);
          }
        }
      } else if (warp >= kWarpConv) {
        if constexpr (kFp8) {
        // ---------------------------------------------------------- E4M3 -> f16
        // A tile's 64 keys are 16 groups of 4 rows; converter c takes groups
        // [16c/W, 16(c+1)/W) of K and of V, a group per step: 4 rows x 8 16-byte
        // chunks.  A quarter warp takes chunks 0-3 of one row and 4-7 of the next
        // (rows of opposite parity, so their swizzles differ in the low bit): its
        // 16-byte loads and both of its 16-byte stores (f16 halves 0 and 1) then
        // hit 8 distinct bank groups.  E4M3 K row r and V row r sit exactly where
        // f16 V row r goes (half 0, half 1), so a group's f16 V rows overwrite
        // only the bytes the same step has read.
        constexpr int W = C::kConvWarps;
        const int c = warp - kWarpConv, g0 = 16 * c / W, g1 = 16 * (c + 1) / W;
        const int nblk = (n + a.BS - 1) / a.BS;
        const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
        const int up = (lane >> 2) & 1, ch = 4 * up + (lane & 3);   // f16 half, source chunk
        const int rsub = 2 * (lane >> 4) + (up ^ ((lane >> 3) & 1));  // row within the group
        // 16 E4M3 values d = 16ch .. 16ch+15 -> f16 (V with per-block scales:
        // times the block's scale over 2^EV)
        auto convert = [&](const uint4 x, float sc, bool scaled, uint32_t (&o)[8]) {
          const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) e4m3x4_to_f16x2x2(xw[e], o[2 * e], o[2 * e + 1]);
          if (scaled) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float2 f = unpack2<false>(o[e]);
              o[e] = pack_f16(f.x * sc, f.y * sc);
            }
          }
        };
        // ... into f16 half `up` of K (kv 0) or V (kv 1): chunks 2(ch % 4) and +1
        auto store = [&](uint8_t* dst, int kv, int row, const uint32_t (&o)[8]) {
          uint8_t* half = dst + (kv * 2 + up) * kKVHalf;
          *reinterpret_cast<uint4*>(half + sw128(row, 2 * (ch & 3))) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(half + sw128(row, 2 * (ch & 3) + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
        };
        // Per-block scales.  K stays exact (E4M3 -> f16); its block scales
        // multiply the scores in fp32 in the softmax.  V's scales are applied here,
        // each divided by 2^EV, the largest power-of-two exponent among the V
        // scales of the CTA's blocks, so the f16 values stay below 2 x 448 whatever
        // the scales' magnitudes; 2^EV rides on the output.  The three converter
        // warps find EV over the CTA's blocks first.
        int ev_ref = 0;
        if (a.block_scales) {
          const int bpt = kN / a.BS;
          const int b1 = min((jt0 + T) * bpt, nblk);
          int ev = -100000;
          for (int b = jt0 * bpt + c * 32 + lane; b < b1; b += W * 32) {
            int blk = __ldg(trow + b);
            blk = (blk < 0 || blk >= a.num_blocks) ? 0 : blk;
            const float vs =
                __ldg(a.block_scales + ((size_t)(blk * 2 + 1) * a.L + a.layer) * a.Hkv + hkv);
            if (vs > 0.f && isfinite(vs)) ev = max(ev, ilogbf(vs));
          }
          ev = __reduce_max_sync(0xffffffffu, ev);
          if (leader) {
            bars->eref[c] = ev;
            mbar_arrive(&bars->eref_ready);
          }
          ok = wait(&bars->eref_ready, 0);
          ev = -100000;
          for (int w = 0; w < W; ++w) ev = max(ev, bars->eref[w]);
          ev_ref = ev == -100000 ? 0 : ev;
        }
        for (int j = 0; j < T && ok; ++j) {
          const int st = j % nst;
          ok = wait(&bars->s8_full[st], (j / nst) & 1);
          if (!ok) break;
          uint8_t* dst = sm + stage_off(st);
          const uint8_t* src = dst + 2 * kKVHalf;              // E4M3 K rows, then V rows
          const int valid = n - (jt0 + j) * kN;                // keys of the tile in the sequence
          // two groups a step (eight loads in flight a lane before the warp syncs)
#pragma unroll 1
          for (int gr = g0; gr < g1; gr += 2) {
            const bool two = gr + 1 < g1;
            const int row0 = 4 * gr + rsub, row1 = row0 + 4;
            const uint4 xk0 = *reinterpret_cast<const uint4*>(src + sw128(row0, ch));
            const uint4 xv0 = *reinterpret_cast<const uint4*>(src + kKVHalf + sw128(row0, ch));
            uint4 xk1 = make_uint4(0, 0, 0, 0), xv1 = xk1;
            if (two) {
              xk1 = *reinterpret_cast<const uint4*>(src + sw128(row1, ch));
              xv1 = *reinterpret_cast<const uint4*>(src + kKVHalf + sw128(row1, ch));
            }
            // per-block V scales: those of the row's block (per-tensor: applied elsewhere)
            const bool scaled = a.block_scales != nullptr;
            float sv[2] = {1.f, 1.f};
            if (scaled) {
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int jb = min((jt0 + j) * (kN / a.BS) + (row0 + 4 * h) / a.BS, nblk - 1);
                int blk = __ldg(trow + jb);
                blk = (blk < 0 || blk >= a.num_blocks) ? 0 : blk;
                sv[h] = ldexpf(
                    __ldg(a.block_scales + ((size_t)(blk * 2 + 1) * a.L + a.layer) * a.Hkv + hkv),
                    -ev_ref);
              }
            }
            __syncwarp();                                       // the step's E4M3 bytes are read
            uint32_t o[8];
            convert(xk0, 1.f, false, o);
            store(dst, 0, row0, o);
            convert(xv0, sv[0], scaled, o);
            if (row0 >= valid) {
              // keys past the sequence end: zero V, so that P = 0 never meets NaN
#pragma unroll
              for (int e = 0; e < 8; ++e) o[e] = 0u;
            }
            store(dst, 1, row0, o);
            if (two) {
              convert(xk1, 1.f, false, o);
              store(dst, 0, row1, o);
              convert(xv1, sv[1], scaled, o);
              if (row1 >= valid) {
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = 0u;
              }
              store(dst, 1, row1, o);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (leader) mbar_arrive(&bars->kv_full[st]);
        }
        }
      } else if (warp < kWarpPV) {
        const int t = warp - kWarpS;                           // this warp's query tile
        const uint64_t qb = d_k + ((kSmemQ + t * 2 * kHalf) >> 4);
        ok = wait(&bars->q_ready, 0);
        for (int j = 0; j < T && ok; ++j) {
          ok = wait(&bars->kv_full[j % nst], (j / nst) & 1);
          const bool mine = j < tiles[t];
          const int jl = j;
          // S_tj overwrites the TMEM buffer of the tile's P two tiles back: its P V
          // must have read it
          if (ok && mine && jl >= 2) ok = wait(&bars->p_free[t][jl & 1], ((jl - 2) >> 1) & 1);
          if (!ok) break;
          tc_fence_after();
          if (mine && leader) {
            const uint64_t kb = d_kt + (stage_off(j % nst) >> 4);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint32_t off = ((k >> 2) * kHalf + (k & 3) * 32) >> 4;
              const uint32_t offk = ((k >> 2) * (kFp8 ? kKVHalf : 1024u) + (k & 3) * 32) >> 4;
              tc_mma_f16(tmem + t * 256 + (jl & 1) * kN, qb + off, kb + offk, id_s, k > 0);
            }
            tc_commit(&bars->s_full[t][jl & 1]);
          }
          if (leader) tc_commit(&bars->kv_empty[j % nst]);  // S_tj has read K_j
          __syncwarp();
        }
      } else {
        const int t = warp - kWarpPV;                          // this warp's query tile
        for (int j = 0; j < T && ok; ++j) {
          // paces this warp's releases: its arrival for the stage's next tile can
          // only follow that tile's load, which follows this tile's release
          ok = wait(&bars->kv_full[j % nst], (j / nst) & 1);
          const int jl = j;
          if (ok && j < tiles[t]) {
            const int b = jl & 1;
            ok = wait(&bars->p_full[t][b], (jl >> 1) & 1);
            if (!kFp8 && ok && j == j_tail) ok = wait(&bars->v_zeroed, 0);
            if (!ok) break;
            tc_fence_after();
            if (leader) {
              const uint64_t vb = d_v + ((stage_off(j % nst) + 2 * kKVHalf) >> 4);
              const uint32_t pa = tmem + t * 256 + b * kN;       // P hi: 32 columns, lo: the next 32
#pragma unroll
              for (int k = 0; k < 4; ++k) {                     // 16 keys (8 columns of P) per MMA
                const uint32_t vk = k * (kFp8 ? 128u : 256u);   // 16 keys: 2 KB / 4 KB on
                tc_mma_f16_ts(tmem + t * 256 + 128, pa + k * 8, vb + vk, id_o,
                              (jl > 0 || k > 0) ? 1u : 0u);
                if (kSplitP) tc_mma_f16_ts(tmem + t * 256 + 128, pa + 32 + k * 8, vb + vk, id_o, 1u);
              }
              tc_commit(&bars->o_done[t]);
              tc_commit(&bars->p_free[t][b]);
              if (jl == tiles[t] - 1) tc_commit(&bars->o_final[t]);
            }
          }
          if (!ok) break;
          if (leader) tc_commit(&bars->kv_empty[j % nst]);  // P_tj V_j has read V_j
          __syncwarp();
        }
      }
      if (!ok && leader) {
        record_error(a.status, PKV_ETIMEOUT);
        bars->abort_flag = 1;
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax, one row per thread
    const int t = warp / 4, r = tid - 128 * t, i = r / G, g = r % G;
    const int tok = (pair * kQT + t) * QT + i;
    const bool live = tok < a.q_len;
    // this query's last visible key: causal within the chunk, or its prefix length
    const int pos = casc ? (live ? __ldg(a.key_limit + tok) : 0) - 1 : n - a.q_len + tok;
    const int my_tiles = tiles[t];
    // Q carries the sign; 2^-q_e undoes the row's f16 prescale (E4M3 pools)
    float qs = fabsf(a.qk_scale_log2) * pow2i(-q_e);
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tcol = tmem + lane_base + t * 256;
    float mref = -INFINITY, lsum = 0.f;
    bool ok = true;
    // waits and TMEM accesses stay warp-uniform (tcgen05.ld/st are .sync.aligned)
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      const bool got = mbar_wait_bounded(bar, parity);
      return __all_sync(0xffffffffu, got) && !bars->abort_flag;
    };
    // E4M3 per-block scales: each 16-key group's scores take their block's K
    // scale in fp32 (qsb), and the V tiles were divided by 2^EV
    const bool bscaled = kFp8 && a.block_scales != nullptr;
    int ev_ref = 0;
    if (bscaled && my_tiles > 0) {
      ok = wait(&bars->eref_ready, 0);
      int ev = -100000;
      for (int w = 0; w < C::kConvWarps; ++w) ev = max(ev, bars->eref[w]);
      if (ev != -100000) ev_ref = ev;
    }
    const int32_t* trow = a.tables + (size_t)s * a.max_blocks;
    const int nblk = (n + a.BS - 1) / a.BS;
    for (int jl = 0; jl < my_tiles && ok; ++jl) {
      const int b = jl & 1;
      const int j = jl;
      const int kpos0 = (jt0 + j) * kN;
      float qsb[4] = {qs, qs, qs, qs};
      if (bscaled) {
        // issued before the wait for S, so the loads overlap it
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
          int blk = __ldg(trow + min((kpos0 + 16 * g4) / a.BS, nblk - 1));
          blk = (blk < 0 || blk >= a.num_blocks) ? 0 : blk;
          qsb[g4] = qs * __ldg(a.block_scales + ((size_t)blk * 2 * a.L + a.layer) * a.Hkv + hkv);
        }
      }
      if (!wait(&bars->s_full[t][b], (jl >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[kN];
      tmem_ld64_sync(tcol + b * kN, sv);
      // causal mask and row max over the raw scores (8 partial maxima, two per
      // 16-key group: short dependency chains); the scales are positive, so each
      // group's scale commutes with its max
      float mp[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mp[e] = -INFINITY;
      if (__all_sync(0xffffffffu, live && kpos0 + kN - 1 <= pos)) {
        // the warp's rows see every key of the tile: no mask
#pragma unroll
        for (int c = 0; c < kN; c += 2) {
          const int e = 2 * (c >> 4) + ((c >> 1) & 1);
          mp[e] = fmax3(mp[e], sv[c], sv[c + 1]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kN; c += 2) {
          const int e = 2 * (c >> 4) + ((c >> 1) & 1);
          sv[c] = live && kpos0 + c <= pos ? sv[c] : -INFINITY;
          sv[c + 1] = live && kpos0 + c + 1 <= pos ? sv[c + 1] : -INFINITY;
          mp[e] = fmax3(mp[e], sv[c], sv[c + 1]);
        }
      }
      const float mx = fmaxf(fmaxf(qsb[0] * fmaxf(mp[0], mp[1]), qsb[1] * fmaxf(mp[2], mp[3])),
                             fmaxf(qsb[2] * fmaxf(mp[4], mp[5]), qsb[3] * fmaxf(mp[6], mp[7])));
      bool rescale = false;
      float alpha = 1.f;
      if (mx > mref + 8.f) {            // also the first visible key (mref = -inf)
        alpha = exp2f(mref - mx);       // 0 when mref = -inf
        mref = mx;
        rescale = jl > 0;
      }
      const float ref = mref == -INFINITY ? 0.f : mref;
      uint64_t pp[4];                   // partial row sums, two lanes each
#pragma unroll
      for (int e = 0; e < 4; ++e) pp[e] = 0ull;
      // a rescale needs O stable: P_{t,j-1} V_{j-1} done (its phase is the only
      // one pending here: P_tj is not yet written, and S_tj came after P_t,j-2 V)
      if (__any_sync(0xffffffffu, rescale)) {
        if (jl > 0) {
          if (!wait(&bars->o_done[t], (jl - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
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
      }
      // P over S_tj in TMEM, packed pairs: hi in columns 0..31 of the buffer, lo
      // in 32..63; computed and stored 16 keys at a time (fewer live registers).
      // Two keys per FP32 instruction (f32x2 FMA / add / sub).
      const uint64_t nref2 = f2_pack(kPOff - ref, kPOff - ref);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint64_t qs2 = f2_pack(qsb[q4], qsb[q4]);
        uint32_t phi[8], plo[8];
#pragma unroll
        for (int c2 = 0; c2 < 8; ++c2) {
          const int c = q4 * 16 + 2 * c2;
          // p = 2^(s * scale - ref): one FMA per two keys and the SFU per key
          float x0, x1;
          f2_unpack(ffma2(f2_pack(sv[c], sv[c + 1]), qs2, nref2), x0, x1);
          const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
          const uint64_t p2 = f2_pack(p0, p1);
          pp[c2 & 3] = fadd2(pp[c2 & 3], p2);
          if (kSplitP) {
            // hi = p with the low 16 bits cut (bf16 truncation), lo = p - hi exactly,
            // then rounded to bf16: |lo| < 2^-8 p, so P carries 2^-17 relative error
            const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
            phi[c2] = __byte_perm(b0, b1, 0x7632u);
            float l0, l1;
            f2_unpack(fsub2(p2, f2_pack(__uint_as_float(b0 & 0xffff0000u),
                                        __uint_as_float(b1 & 0xffff0000u))), l0, l1);
            plo[c2] = pack_bf16(l0, l1);
          } else {
            phi[c2] = pack2<kBf16>(p0, p1);
          }
        }
        tmem_st8(tcol + b * kN + q4 * 8, phi);
        if (kSplitP) tmem_st8(tcol + b * kN + 32 + q4 * 8, plo);
      }
      float ps = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float u0, u1;
        f2_unpack(pp[e], u0, u1);
        ps += u0 + u1;
      }
      lsum = lsum * alpha + ps;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p_full[t][b]);
    }
    // epilogue: O row / l -> out (every lane reads TMEM; live rows store).  The
    // softmax waits for P V only before a rescale, so the last P V may be up to
    // two phases of o_done away: a one-shot barrier marks the end instead.
    // (shared-prefix mode: fp32 partial O and its natural log-sum-exp per split)
    const int pidx = split;                          // this split's partial set
    const size_t hrow = ((size_t)(casc ? pidx : s) * a.q_len + tok) * a.Hq + (size_t)hkv * G + g;
    const size_t orow = hrow * kD;
    const int odt = casc ? PKV_F32 : a.out_dtype;
    if (ok && my_tiles > 0 && wait(&bars->o_final[t], 0)) {
      tc_fence_after();
      float inv = lsum > 0.f ? a.v_scale / lsum : 0.f;
      if (kFp8 && a.block_scales) inv = ldexpf(inv, ev_ref);
#pragma unroll
      for (int c = 0; c < kD; c += 32) {
        float o[32];
        tmem_ld32(tcol + 128 + c, o);
        tmem_ld_wait();
        if (live) {
          // 16-byte stores of the row's 32 values (rows start on 256-byte
          // boundaries of the 16-byte-aligned output)
          if (odt == PKV_F32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow + c);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv,
                                   o[4 * e + 3] * inv);
          } else {
            uint32_t w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = odt == PKV_BF16 ? pack_bf16(o[2 * e] * inv, o[2 * e + 1] * inv)
                                     : pack_f16(o[2 * e] * inv, o[2 * e + 1] * inv);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + orow + c);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
      }
      if (casc && live)
        a.out_lse[hrow] = lsum > 0.f
                              ? ((mref == -INFINITY ? 0.f : mref) + __log2f(lsum) - kPOff) * kLn2
                              : -INFINITY;
    } else if (my_tiles == 0) {
      if (live) {
        for (int e = 0; e < kD; ++e) store_from_float(a.out, orow + e, odt, 0.f);
        if (casc) a.out_lse[hrow] = -INFINITY;
      }
    } else {
      record_error(a.status, PKV_ETIMEOUT);
      bars->abort_flag = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpTMA) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

template <int KVT>
size_t smem_bytes_t() { return PfCfg<KVT>::kSmemBytes + sizeof(Bars) + kAlignSlack; }

template <int KVT>
cudaError_t launch_t(const CUtensorMap* map, const DecodeArgs& a, dim3 grid, cudaStream_t stream) {
  const size_t smem = smem_bytes_t<KVT>();
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<KVT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(PfCfg<KVT>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<KVT>, *map, a);
}

bool prefill_tc_supported(int kv_dtype, int q_dtype, int BS, int D, int G) {
  const bool dt_ok = (kv_dtype == PKV_BF16 || kv_dtype == PKV_F16) ? q_dtype == kv_dtype
                     : kv_dtype == PKV_FP8_E4M3 ? (q_dtype == PKV_BF16 || q_dtype == PKV_F16)
                                                : false;
  return dt_ok && D == kD && (BS == 16 || BS == 32 || BS == 64) && G >= 1 && G <= kM &&
         kM % G == 0;
}

cudaError_t launch_prefill_tc(const CUtensorMap* map, const DecodeArgs& a, cudaStream_t stream) {
  const int QT = kM / a.G;
  const int qtiles = (a.q_len + QT - 1) / QT;
  if (qtiles == 0 || a.B == 0) return cudaSuccess;
  if (a.key_limit && (a.S < 1 || a.S > 65535 || a.B != 1 || !a.out_lse)) return cudaErrorInvalidValue;
  const int pairs = (qtiles + kQT - 1) / kQT;
  if (pairs > 65535 || a.B > 65535) return cudaErrorInvalidValue;
  dim3 grid(a.Hkv, a.key_limit ? a.S : a.B, pairs);
  cudaError_t e;
  switch (a.kv_dtype) {
    case PKV_BF16: e = launch_t<PKV_BF16>(map, a, grid, stream); break;
    case PKV_F16: e = launch_t<PKV_F16>(map, a, grid, stream); break;
    case PKV_FP8_E4M3: e = launch_t<PKV_FP8_E4M3>(map, a, grid, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e == cudaSuccess) count_launch();
  return e;
}

}  // namespace pkv
