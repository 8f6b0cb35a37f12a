// decode_mma.cu -- launch-shape helpers and the dtype dispatch of the
// tensor-core paged decode kernel (decode_mma.cuh); the template instances live
// in one file per KV dtype so that they compile in parallel.
#include "decode_mma.cuh"

namespace pkv {

cudaError_t launch_decode_mma_bf16(const CUtensorMap*, const DecodeArgs&, int, int, cudaStream_t);
cudaError_t launch_decode_mma_f16(const CUtensorMap*, const DecodeArgs&, int, int, cudaStream_t);
cudaError_t launch_decode_mma_fp8(const CUtensorMap*, const DecodeArgs&, int, int, cudaStream_t);

using mma::kD;
using mma::kLineBytes;
using mma::kMaxHG;
using mma::SmemHeader;

size_t mma_stage_bytes(int kv_dtype, int BS, int HG) {
  const int regions = kv_dtype == PKV_FP8_E4M3 ? 1 : 2;
  return (size_t)HG * BS * kLineBytes * 2 * regions;
}

size_t mma_smem_bytes(int kv_dtype, int BS, int HG, int stages) {
  return (size_t)stages * mma_stage_bytes(kv_dtype, BS, HG) + sizeof(SmemHeader) + 1024;
}

bool mma_supported(int kv_dtype, int BS, int D, int G, int q_len) {
  const int R = G * q_len;
  return (kv_dtype == PKV_BF16 || kv_dtype == PKV_F16 || kv_dtype == PKV_FP8_E4M3) &&
         (BS == 16 || BS == 32 || BS == 64) && D == kD && G >= 1 && R <= 16 &&
         (R <= 8 || BS <= 32);
}

cudaError_t launch_decode_mma(const CUtensorMap* map, const DecodeArgs& a, int gx, int gy,
                              cudaStream_t stream) {
  if (a.stages < 2 || a.stages > 16 || a.HG < 1 || a.HG > kMaxHG) return cudaErrorInvalidValue;
  if (a.R < 1 || a.R > 16 || (a.R > 8 && a.BS == 64)) return cudaErrorInvalidValue;
  switch (a.kv_dtype) {
    case PKV_BF16: return launch_decode_mma_bf16(map, a, gx, gy, stream);
    case PKV_F16: return launch_decode_mma_f16(map, a, gx, gy, stream);
    case PKV_FP8_E4M3: return launch_decode_mma_fp8(map, a, gx, gy, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
