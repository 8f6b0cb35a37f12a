// decode_mma_bf16.cu -- instances of the tensor-core paged decode kernel
// (decode_mma.cuh) for bf16 KV pools: block sizes 16 / 32 / 64, one query
// token (NT = 1, not causal) or a causal chunk of up to 8 (NT = 1) or 16
// (NT = 2, block sizes 16 / 32) query rows per KV head; and, for the
// shared-prefix decode, one query token with each sequence read from the end of
// its prefix (kOff; up to 8 or 16 rows per KV head).
#include "decode_mma.cuh"

namespace pkv {

cudaError_t launch_decode_mma_bf16(const CUtensorMap* map, const DecodeArgs& a, int gx, int gy,
                                   cudaStream_t stream) {
  using mma::launch_t;
  const int nt = a.R <= 8 ? 1 : 2;
  // two n-tiles exist only as the causal instance; with one query token its
  // limits let every row see every key, as the plain decode does
  const bool causal = a.q_len > 1 || nt == 2;
  if (a.len_off) {
    // shared-prefix decode (one query token): each sequence from the end of its prefix
    switch (a.BS * 100 + nt * 10 + (causal ? 1 : 0)) {
      case 1610: return launch_t<PKV_BF16, 16, 1, false, true>(map, a, gx, gy, stream);
      case 3210: return launch_t<PKV_BF16, 32, 1, false, true>(map, a, gx, gy, stream);
      case 6410: return launch_t<PKV_BF16, 64, 1, false, true>(map, a, gx, gy, stream);
      case 1621: return launch_t<PKV_BF16, 16, 2, true, true>(map, a, gx, gy, stream);
      case 3221: return launch_t<PKV_BF16, 32, 2, true, true>(map, a, gx, gy, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.BS * 100 + nt * 10 + (causal ? 1 : 0)) {
    case 1610: return launch_t<PKV_BF16, 16, 1, false>(map, a, gx, gy, stream);
    case 3210: return launch_t<PKV_BF16, 32, 1, false>(map, a, gx, gy, stream);
    case 6410: return launch_t<PKV_BF16, 64, 1, false>(map, a, gx, gy, stream);
    case 1611: return launch_t<PKV_BF16, 16, 1, true>(map, a, gx, gy, stream);
    case 3211: return launch_t<PKV_BF16, 32, 1, true>(map, a, gx, gy, stream);
    case 6411: return launch_t<PKV_BF16, 64, 1, true>(map, a, gx, gy, stream);
    case 1621: return launch_t<PKV_BF16, 16, 2, true>(map, a, gx, gy, stream);
    case 3221: return launch_t<PKV_BF16, 32, 2, true>(map, a, gx, gy, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
