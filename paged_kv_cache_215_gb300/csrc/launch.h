// launch.h -- internal interface between the host library (pkv.cpp) and the
// kernels (*.cu).  Not installed; the public ABI is include/pkv.h.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Decode attention arguments, shared by the tensor-core kernel, the SIMT kernel
// and the merge kernels.
struct DecodeArgs {
  const void* q;             // [B, Hq, D] q_dtype
  void* out;                 // [B, Hq, D] out_dtype
  const void* pool;          // [NB, 2, L, Hkv, BS, D] kv_dtype
  const int32_t* tables;     // [B, max_blocks]
  const int32_t* seq_lens;   // [B]
  float* part_o;             // partial outputs (layout depends on mode)
  float* part_lse;           // partial natural log-sum-exp
  int2* unit_info;           // balanced mode: per unit (first slot, piece count)
  int slots;                 // balanced mode: partial slots in the workspace (grid + units)
  int32_t* status;           // device error word or nullptr
  int B, Hq, Hkv, G, D, BS, L, layer, max_blocks, num_blocks;
  int q_dtype, out_dtype, kv_dtype;
  int HG;                    // kv heads per CTA (tensor-core kernel)
  int NHG;                   // Hkv / HG
  int stages;                // shared-memory pipeline depth
  int smem_bytes;            // dynamic shared memory to request, if above what the ring needs
  int mode;                  // 0 balanced token stream, 1 fixed S partitions per sequence
  int S;                     // partitions per sequence in mode 1
  int q_len;                 // query tokens per sequence (1: decode; >1: causal chunk)
  int R;                     // query rows per KV head: q_len * G
  float qk_scale_log2;       // softmax scale * log2(e) (* k_scale for E4M3)
  float v_scale;             // v_scale for E4M3, else 1
  // Fused append (decode step): when k_new is set, the new token of sequence s
  // ([B, Hkv, D] in new_dtype) is stored at position seq_lens[s] - 1 before the
  // block holding it is read; E4M3 pools encode with k_enc_scale / v_enc_scale.
  const void* k_new;
  const void* v_new;
  int new_dtype;
  float k_enc_scale, v_enc_scale;
  // E4M3 per-tile scales [NB, 2, L, Hkv] (block-wise scaling) or nullptr.
  const float* block_scales;
  // 1: launched with programmatic dependent launch; every write to out, the
  // workspace or the pool waits for the preceding kernel (griddepcontrol.wait).
  int pdl;
  int early_trigger;  // balanced mode, this call's merge next: let it be scheduled at the start
  int casc_len;       // tcgen05 kernel, shared-prefix mode: the prefix length in tokens
  // Shared-prefix decode (cascade).  Decode kernel + merge: ext_count partials per
  // output row computed elsewhere (over the shared prefix), [ext_count][B*Hq][D] and
  // [ext_count][B*Hq]; every unit then leaves partials and the merge adds these.
  const float* ext_o;
  const float* ext_lse;
  int ext_count;
  // with ext partials: per sequence, the tokens before its private part (the
  // shared prefix, whole blocks); the decode reads sequence s from token
  // len_off[s] on (table entry len_off[s] / BS on).  nullptr: from token 0.
  const int32_t* len_off;
  // Prefill kernel over a shared prefix: query token i is sequence i, it sees keys
  // [0, key_limit[i]) (no causal mask); the key range is cut into S splits
  // (blockIdx.y), each writing fp32 normalised O to out and its lse to out_lse at
  // row (split * q_len + i) * Hq + head.
  const int32_t* key_limit;
  float* out_lse;
};

// Shared memory the tensor-core kernel needs for one CTA.
size_t mma_stage_bytes(int kv_dtype, int BS, int HG);
size_t mma_smem_bytes(int kv_dtype, int BS, int HG, int stages);
bool mma_supported(int kv_dtype, int BS, int D, int G, int q_len);

cudaError_t launch_decode_mma(const CUtensorMap* map, const DecodeArgs& a, int grid_x, int grid_y,
                              cudaStream_t stream);
cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t stream);
// Chunked prefill on tcgen05 (one CTA per 128-row query tile, KV head, sequence).
bool prefill_tc_supported(int kv_dtype, int q_dtype, int BS, int D, int G);
cudaError_t launch_prefill_tc(const CUtensorMap* map, const DecodeArgs& a, cudaStream_t stream);
// Merge of the balanced-mode partials, one CTA per (unit, head in the unit).
cudaError_t launch_merge_units(const DecodeArgs& a, bool pdl, cudaStream_t stream);
// Cascade merge: the decode's balanced-mode partials of each row plus a.ext_count
// external partials.
cudaError_t launch_merge_units_ext(const DecodeArgs& a, cudaStream_t stream);
// Shared-prefix check: each sequence's prefix length is whole blocks, within its
// length and the shared list, and its table starts with the shared blocks; a
// mismatch is recorded as PKV_EINVAL.  Lets the next launch be scheduled at once.
cudaError_t launch_prefix_check(const int32_t* tables, int max_blocks, const int32_t* seq_lens,
                                const int32_t* prefix_table, int prefix_blocks,
                                const int32_t* prefix_lens, int prefix_len_max, int B, int BS,
                                int32_t* status, cudaStream_t stream);
// Merge of [rows, S, D] partials (the public merge_partials layout).
cudaError_t launch_merge_rows(void* out, int out_dtype, const float* part_o, const float* part_lse,
                              int rows, int S, int D, bool pdl, cudaStream_t stream);

struct AppendArgs {
  void* pool;
  const void* k;
  const void* v;
  const int32_t* tables;
  const int32_t* seq_ids;    // nullptr: token i belongs to sequence i
  const int32_t* positions;  // nullptr: position seq_lens[s] - 1 (the decode step's token)
  const int32_t* seq_lens;
  int32_t* status;
  int64_t num_tokens;
  int B, Hkv, D, BS, L, layer, max_blocks, num_blocks;
  int in_dtype, kv_dtype;
  float k_scale, v_scale;
  const float* block_scales;  // E4M3 per-tile scales [NB, 2, L, Hkv], or nullptr (per-tensor)
  int group_tokens;           // block-wise scales: positions per scale group (a multiple of BS)
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);
// E4M3 block-wise scales amax / 448 of the scale groups the tokens land in, stored
// in every block of each group (three launches, four for groups of several blocks).
cudaError_t launch_block_scales(const AppendArgs& a, float* scales, cudaStream_t stream);
cudaError_t launch_absmax(const void* x, int dtype, int64_t n, float* amax, cudaStream_t stream);
// scale = max(amax[0..n)) / 448 (1 when that is 0), one thread block.
cudaError_t launch_fp8_scale(const float* amax, int n, float* scale, cudaStream_t stream);

// Launch counter shared by every launcher.
void count_launch();

// One warp waits (bounded) on a barrier nothing arrives on and records
// PKV_ETIMEOUT in `status`: the failure-detection self-test.
cudaError_t launch_wait_selftest(int32_t* status, cudaStream_t stream);

}  // namespace pkv
