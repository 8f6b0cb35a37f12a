// pkv.cpp -- host side of the C ABI declared in include/pkv.h: argument
// validation, the host block allocator, TMA descriptors, launch heuristics and
// workspace layout.  Every step of the computation runs in the CUDA kernels;
// nothing here touches K, V, q or out.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <vector>

#include "launch.h"
#include "pkv.h"

namespace pkv {

static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static int elem_bytes(int dtype) {
  switch (dtype) {
    case PKV_F32: return 4;
    case PKV_F16: return 2;
    case PKV_BF16: return 2;
    case PKV_FP8_E4M3: return 1;
    default: return 0;
  }
}

static bool act_dtype(int dtype) { return dtype == PKV_F32 || dtype == PKV_F16 || dtype == PKV_BF16; }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
  int sms = 0, smem_optin = 0, smem_per_sm = 0, l2_bytes = 0;
};

static bool device_info(DeviceInfo* out) {
  static std::mutex mu;
  static std::map<int, DeviceInfo> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(dev);
  if (it == cache.end()) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      return false;
    it = cache.emplace(dev, d).first;
  }
  *out = it->second;
  return true;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// ---------------------------------------------------------------- launch plans

struct MmaPlan {
  int HG = 0, NHG = 0, stages = 0, ctas_per_sm = 1, grid = 0;
  size_t smem = 0;
};

static bool hg_ok(const pkv_geometry& g, int hg) {
  return hg >= 1 && hg <= 8 && g.num_kv_heads % hg == 0 && hg * g.block_size <= 256;
}

// Tensor-core kernel: KV heads per CTA, pipeline depth and persistent grid.
// Defaults (measured on GB300 over the 8K x 32, 128K, 1M, 70B-shaped and FP8
// workloads): two CTAs per SM; each CTA streams a head group of at most 4 KV
// heads whose per-block K+V stage is at most 32 KB; the ring keeps about 128 KB
// per SM in flight for 16-bit pools and 192 KB for E4M3 pools, whose
// conversion work needs deeper buffering.  Deeper 16-bit rings measured slower.
static bool plan_mma(const pkv_geometry& g, const DeviceInfo& dev, const pkv_launch_opts* o,
                     MmaPlan* p) {
  const int ctas = (o && o->ctas_per_sm > 0) ? o->ctas_per_sm : 2;
  if (ctas > 8) return false;
  int hg = (o && o->kv_heads_per_cta > 0) ? o->kv_heads_per_cta : 0;
  if (hg) {
    if (!hg_ok(g, hg)) return false;
  } else {
    for (int c = 4; c >= 1; --c)
      if (hg_ok(g, c) && mma_stage_bytes(g.kv_dtype, g.block_size, c) <= 32 * 1024) {
        hg = c;
        break;
      }
    if (!hg) return false;
  }
  const size_t stage = mma_stage_bytes(g.kv_dtype, g.block_size, hg);
  const size_t per_cta = std::min<size_t>((size_t)dev.smem_optin,
                                          (size_t)dev.smem_per_sm / ctas - 1024);
  const size_t fixed = mma_smem_bytes(g.kv_dtype, g.block_size, hg, 0);
  const int fit = per_cta > fixed ? (int)((per_cta - fixed) / stage) : 0;
  int stages = (o && o->stages > 0) ? o->stages : 0;
  if (!stages) {
    const size_t inflight = (g.kv_dtype == PKV_FP8_E4M3 ? 192 : 128) * 1024;
    stages = (int)(inflight / ((size_t)ctas * stage));
    stages = std::max(2, std::min(stages, std::min(fit, 8)));
  }
  if (stages < 2 || stages > 16 || stages > fit) return false;
  p->HG = hg;
  p->NHG = g.num_kv_heads / hg;
  p->stages = stages;
  p->ctas_per_sm = ctas;
  p->grid = dev.sms * ctas;
  p->smem = mma_smem_bytes(g.kv_dtype, g.block_size, hg, stages);
  if (p->smem > (size_t)dev.smem_optin) return false;
  // Request the SM's share of shared memory even when the ring needs less, so
  // that at most `ctas` CTAs share an SM.  The balanced split gives every CTA
  // the same bytes; small CTAs (one KV head each at block size 64) otherwise fit
  // three or more to an SM, and a launch that starts while the previous grid
  // drains (programmatic dependent launch) then stacks them unevenly.
  const size_t share = (size_t)dev.smem_per_sm / ctas - 1024;
  if (p->smem < share && share <= (size_t)dev.smem_optin) p->smem = share;
  return true;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Balanced-mode workspace: partial O and lse per (slot, head of the group), and
// per-unit (first slot, count).
struct BalancedWs {
  size_t o_off, lse_off, info_off, bytes;
};
static BalancedWs balanced_ws(const pkv_geometry& g, int batch, int q_len, const MmaPlan& p) {
  const size_t units = (size_t)batch * p.NHG;
  const size_t slots = (size_t)p.grid + units;
  const size_t hgg = (size_t)p.HG * (g.num_q_heads / g.num_kv_heads) * q_len;
  BalancedWs w;
  w.o_off = 0;
  w.lse_off = align256(slots * hgg * g.head_dim * sizeof(float));
  w.info_off = w.lse_off + align256(slots * hgg * sizeof(float));
  w.bytes = w.info_off + align256(units * sizeof(int2));
  return w;
}

// Fixed-split workspace: [B, q_len, Hq, S, D] and [B, q_len, Hq, S].
static size_t fixed_ws(const pkv_geometry& g, int batch, int q_len, int S, size_t* lse_off) {
  const size_t rows = (size_t)batch * q_len * g.num_q_heads * S;
  const size_t o = align256(rows * g.head_dim * sizeof(float));
  if (lse_off) *lse_off = o;
  return S > 1 ? o + align256(rows * sizeof(float)) : 0;
}

static int simt_auto_splits(const pkv_geometry& g, int batch, int max_seq_len, int sms) {
  const long long units = std::max<long long>(1, (long long)batch * g.num_kv_heads);
  long long s = (8LL * sms + units - 1) / units;
  const long long nb = std::max<long long>(1, ((long long)max_seq_len + g.block_size - 1) / g.block_size);
  s = std::min<long long>(s, nb);
  s = std::min<long long>(s, 1024);
  return (int)std::max<long long>(s, 1);
}

static bool geometry_ok(const pkv_geometry* g) {
  if (!g) return false;
  if (g->num_layers < 1 || g->num_kv_heads < 1 || g->num_q_heads < 1 || g->head_dim < 8 ||
      g->head_dim > 256 || g->head_dim % 8 != 0 || g->block_size < 1 || g->block_size > 256 ||
      g->num_blocks < 1 || g->num_q_heads % g->num_kv_heads != 0 || elem_bytes(g->kv_dtype) == 0)
    return false;
  if (g->kv_dtype == PKV_FP8_E4M3 && g->head_dim % 16 != 0) return false;
  // the tensor map addresses (block, k|v, layer) slabs with a 32-bit coordinate
  if ((long long)g->num_blocks * 2 * g->num_layers >= (1LL << 31)) return false;
  return true;
}

}  // namespace pkv

using namespace pkv;

struct pkv_pool {
  pkv_geometry g;
  void* d_pool = nullptr;
  size_t bytes = 0;
  int32_t* d_status = nullptr;
  float* d_block_scales = nullptr; // E4M3 per-tile scales [NB, 2, L, Hkv] (caller-owned) or null
  std::vector<int32_t> ref;        // reference count per block, 0 = free
  std::vector<int32_t> free_ids;   // stack of free ids
  std::vector<int32_t> free_pos;   // position of an id in free_ids, -1 if taken
  std::map<int, CUtensorMap> tmaps;
  std::mutex mu;

  void take(int32_t id) {
    const int32_t pos = free_pos[id];
    const int32_t last = free_ids.back();
    free_ids[pos] = last;
    free_pos[last] = pos;
    free_ids.pop_back();
    free_pos[id] = -1;
  }
  void give(int32_t id) {
    free_pos[id] = (int32_t)free_ids.size();
    free_ids.push_back(id);
  }
  size_t block_bytes() const {
    return (size_t)2 * g.num_layers * g.num_kv_heads * g.block_size * g.head_dim *
           elem_bytes(g.kv_dtype);
  }
  // TMA descriptor over the pool viewed as [NB*2*L, Hkv*bs, D] with a box of
  // HG*bs rows by one 128-byte line, swizzled 128B.
  const CUtensorMap* tmap(int hg) {
    std::lock_guard<std::mutex> lk(mu);
    auto it = tmaps.find(hg);
    if (it != tmaps.end()) return &it->second;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return nullptr;
    const int eb = elem_bytes(g.kv_dtype);
    CUtensorMapDataType dt = g.kv_dtype == PKV_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                             : g.kv_dtype == PKV_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cuuint64_t dims[3] = {(cuuint64_t)g.head_dim, (cuuint64_t)g.num_kv_heads * g.block_size,
                          (cuuint64_t)g.num_blocks * 2 * g.num_layers};
    cuuint64_t strides[2] = {(cuuint64_t)g.head_dim * eb,
                             (cuuint64_t)g.num_kv_heads * g.block_size * g.head_dim * eb};
    cuuint32_t box[3] = {(cuuint32_t)(128 / eb), (cuuint32_t)(hg * g.block_size), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMap m;
    CUresult r = enc(&m, dt, 3, d_pool, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return nullptr;
    return &tmaps.emplace(hg, m).first->second;
  }
  // TMA descriptor for the tcgen05 kernel's K/V tiles (2-byte pools, D = 128): one
  // box holds a whole block of one KV head, both 64-column halves, laid out in
  // shared memory as 8-token groups, each group's half 0 then half 1 (1 KB
  // swizzle atoms: [group][half][8 rows][128 B]).  The dimensions, innermost
  // first: column within a half (64), token within a group (stride one row),
  // half (stride 128 B), group of 8 rows over heads and tokens (stride 8 rows),
  // block plane (blk * 2 + kv) * L + layer.  E4M3 pools use tmap(1).
  const CUtensorMap* tmap_tiles() {
    if (g.kv_dtype == PKV_FP8_E4M3) return tmap(1);
    if (g.head_dim != 128 || g.block_size % 8 != 0 || g.block_size > 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    auto it = tmaps.find(0);
    if (it != tmaps.end()) return &it->second;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return nullptr;
    const cuuint64_t row = (cuuint64_t)g.head_dim * 2;
    CUtensorMapDataType dt = g.kv_dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[5] = {64, 8, 2, (cuuint64_t)g.num_kv_heads * g.block_size / 8,
                          (cuuint64_t)g.num_blocks * 2 * g.num_layers};
    cuuint64_t strides[4] = {row, 128, 8 * row, (cuuint64_t)g.num_kv_heads * g.block_size * row};
    cuuint32_t box[5] = {64, 8, 2, (cuuint32_t)g.block_size / 8, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUtensorMap m;
    CUresult r = enc(&m, dt, 5, d_pool, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return nullptr;
    return &tmaps.emplace(0, m).first->second;
  }
};

extern "C" {

size_t kv_pool_bytes(const pkv_geometry* g) {
  if (!geometry_ok(g)) return 0;
  return (size_t)2 * g->num_layers * g->num_kv_heads * g->head_dim *
         ((size_t)g->num_blocks * g->block_size) * elem_bytes(g->kv_dtype);
}

int kv_pool_create(const pkv_geometry* g, void* d_pool, size_t pool_bytes, int32_t* d_status,
                   pkv_pool** out) {
  if (!out || !geometry_ok(g) || !d_pool || !aligned16(d_pool) || pool_bytes < kv_pool_bytes(g))
    return PKV_EINVAL;
  pkv_pool* p = new (std::nothrow) pkv_pool();
  if (!p) return PKV_ENOMEM;
  p->g = *g;
  p->d_pool = d_pool;
  p->bytes = pool_bytes;
  p->d_status = d_status;
  p->ref.assign(g->num_blocks, 0);
  p->free_pos.assign(g->num_blocks, -1);
  p->free_ids.reserve(g->num_blocks);
  for (int32_t i = g->num_blocks - 1; i >= 0; --i) p->give(i);
  if (d_status && cudaMemset(d_status, 0, PKV_STATUS_BYTES) != cudaSuccess) {
    delete p;
    return PKV_ECUDA;
  }
  *out = p;
  return PKV_OK;
}

int kv_pool_destroy(pkv_pool* p) {
  delete p;
  return PKV_OK;
}

int kv_pool_geometry(const pkv_pool* p, pkv_geometry* out) {
  if (!p || !out) return PKV_EINVAL;
  *out = p->g;
  return PKV_OK;
}

int kv_pool_alloc(pkv_pool* p, int n, int32_t* ids) {
  if (!p || n < 0 || (n > 0 && !ids)) return PKV_EINVAL;
  std::lock_guard<std::mutex> lk(p->mu);
  if ((size_t)n > p->free_ids.size()) return PKV_ENOMEM;
  for (int i = 0; i < n; ++i) {
    const int32_t id = p->free_ids.back();
    p->take(id);
    p->ref[id] = 1;
    ids[i] = id;
  }
  return PKV_OK;
}

int kv_pool_reserve(pkv_pool* p, int n, const int32_t* ids) {
  if (!p || n < 0 || (n > 0 && !ids)) return PKV_EINVAL;
  std::lock_guard<std::mutex> lk(p->mu);
  std::vector<char> seen;
  for (int i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= p->g.num_blocks || p->ref[id] != 0) return PKV_EINVAL;
  }
  seen.assign(p->g.num_blocks, 0);
  for (int i = 0; i < n; ++i) {
    if (seen[ids[i]]) return PKV_EINVAL;
    seen[ids[i]] = 1;
  }
  for (int i = 0; i < n; ++i) {
    p->take(ids[i]);
    p->ref[ids[i]] = 1;
  }
  return PKV_OK;
}

int kv_pool_free(pkv_pool* p, int n, const int32_t* ids) {
  if (!p || n < 0 || (n > 0 && !ids)) return PKV_EINVAL;
  std::lock_guard<std::mutex> lk(p->mu);
  std::map<int32_t, int> drops;
  for (int i = 0; i < n; ++i) {
    const int32_t id = ids[i];
    if (id < 0 || id >= p->g.num_blocks) return PKV_EINVAL;
    if (++drops[id] > p->ref[id]) return PKV_EINVAL;
  }
  for (int i = 0; i < n; ++i)
    if (--p->ref[ids[i]] == 0) p->give(ids[i]);
  return PKV_OK;
}

int kv_pool_share(pkv_pool* p, int n, const int32_t* ids) {
  if (!p || n < 0 || (n > 0 && !ids)) return PKV_EINVAL;
  std::lock_guard<std::mutex> lk(p->mu);
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= p->g.num_blocks || p->ref[ids[i]] == 0) return PKV_EINVAL;
  for (int i = 0; i < n; ++i) ++p->ref[ids[i]];
  return PKV_OK;
}

int kv_pool_refcount(const pkv_pool* p, int32_t id) {
  if (!p || id < 0 || id >= p->g.num_blocks) return PKV_EINVAL;
  return p->ref[id];
}

int kv_pool_num_free(const pkv_pool* p) {
  if (!p) return PKV_EINVAL;
  return (int)p->free_ids.size();
}

int kv_pool_cow(pkv_pool* p, int32_t id, int32_t* out_id, cudaStream_t stream) {
  if (!p || !out_id || id < 0 || id >= p->g.num_blocks) return PKV_EINVAL;
  std::lock_guard<std::mutex> lk(p->mu);
  if (p->ref[id] <= 0) return PKV_EINVAL;
  if (p->ref[id] == 1) {
    *out_id = id;
    return PKV_OK;
  }
  if (p->free_ids.empty()) return PKV_ENOMEM;
  const int32_t nid = p->free_ids.back();
  const size_t bb = p->block_bytes();
  char* base = static_cast<char*>(p->d_pool);
  if (cudaMemcpyAsync(base + (size_t)nid * bb, base + (size_t)id * bb, bb,
                      cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return PKV_ECUDA;
  p->take(nid);
  p->ref[nid] = 1;
  --p->ref[id];
  *out_id = nid;
  return PKV_OK;
}

int kv_pool_prepare_append(pkv_pool* p, int batch, const int32_t* h_seq_lens,
                           const int32_t* h_new_tokens, int32_t* h_block_tables,
                           int max_blocks_per_seq, int32_t* h_first_changed,
                           cudaStream_t stream) {
  if (!p || batch < 0 || max_blocks_per_seq < 1) return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  if (!h_seq_lens || !h_block_tables) return PKV_EINVAL;
  const int bs = p->g.block_size;
  std::lock_guard<std::mutex> lk(p->mu);
  // plan: per sequence the table entries to fill and whether its tail block
  // (the partly filled block the first new token lands in) must be copied;
  // shared tails are resolved in sequence order, as the copies will be
  struct Plan { int s, first_new, end, cow; };
  std::vector<Plan> plan;
  std::map<int32_t, int> refs;   // simulated counts of the tail blocks touched
  long long need = 0;
  for (int s = 0; s < batch; ++s) {
    const long long n = h_seq_lens[s];
    const long long k = h_new_tokens ? h_new_tokens[s] : 1;
    if (n < 0 || k < 0) return PKV_EINVAL;
    if (k == 0) continue;
    const long long have = (n + bs - 1) / bs, want = (n + k + bs - 1) / bs;
    if (want > max_blocks_per_seq) return PKV_EINVAL;
    int cow = 0;
    if (n % bs != 0) {
      const int32_t id = h_block_tables[(size_t)s * max_blocks_per_seq + n / bs];
      if (id < 0 || id >= p->g.num_blocks || p->ref[id] <= 0) return PKV_EINVAL;
      auto it = refs.emplace(id, p->ref[id]).first;
      if (it->second > 1) {
        cow = 1;
        --it->second;
      }
    }
    need += (want - have) + cow;
    if (want > have || cow) plan.push_back({s, (int)have, (int)want, cow});
  }
  if (need > (long long)p->free_ids.size()) return PKV_ENOMEM;   // nothing changed
  // the blocks to take, from the top of the free stack (taken only below)
  std::vector<int32_t> ids(p->free_ids.end() - need, p->free_ids.end());
  std::reverse(ids.begin(), ids.end());
  // copies first: a failed copy leaves the host state as it was
  size_t next = 0;
  const size_t bb = p->block_bytes();
  char* base = static_cast<char*>(p->d_pool);
  for (const Plan& pl : plan) {
    if (!pl.cow) continue;
    const int32_t src = h_block_tables[(size_t)pl.s * max_blocks_per_seq + h_seq_lens[pl.s] / bs];
    if (cudaMemcpyAsync(base + (size_t)ids[next] * bb, base + (size_t)src * bb, bb,
                        cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
      return PKV_ECUDA;
    ++next;
  }
  // commit: take the blocks, move the references, write the tables
  if (h_first_changed)
    for (int s = 0; s < batch; ++s) h_first_changed[s] = -1;
  next = 0;
  size_t fresh = 0;
  for (const int32_t id : ids) {
    p->take(id);
    p->ref[id] = 1;
  }
  // copies took ids[0 .. copies); fresh blocks follow
  size_t copies = 0;
  for (const Plan& pl : plan) copies += pl.cow;
  fresh = copies;
  for (const Plan& pl : plan) {
    int32_t* row = h_block_tables + (size_t)pl.s * max_blocks_per_seq;
    int first = pl.first_new;
    if (pl.cow) {
      const int j = h_seq_lens[pl.s] / bs;
      --p->ref[row[j]];
      row[j] = ids[next++];
      first = j;
    }
    for (int j = pl.first_new; j < pl.end; ++j) row[j] = ids[fresh++];
    if (h_first_changed) h_first_changed[pl.s] = first;
  }
  return PKV_OK;
}

static int append_common(pkv_pool* p, int layer, const void* k, const void* v, pkv_dtype in_dtype,
                         const int32_t* tables, int max_blocks, int batch, const int32_t* seq_ids,
                         const int32_t* positions, int64_t num_tokens, float k_scale,
                         float v_scale, cudaStream_t stream) {
  if (!p || layer < 0 || layer >= p->g.num_layers || batch < 0 || num_tokens < 0)
    return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !tables || !positions || max_blocks < 1 || batch < 1) return PKV_EINVAL;
  if (!aligned16(k) || !aligned16(v)) return PKV_EINVAL;
  const bool fp8 = p->g.kv_dtype == PKV_FP8_E4M3;
  if (fp8) {
    if (!act_dtype(in_dtype)) return PKV_EINVAL;
    if (!p->d_block_scales &&
        (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale)))
      return PKV_EINVAL;
  } else if ((int)in_dtype != p->g.kv_dtype) {
    return PKV_EINVAL;
  }
  AppendArgs a{};
  a.pool = p->d_pool;
  a.k = k;
  a.v = v;
  a.tables = tables;
  a.seq_ids = seq_ids;
  a.positions = positions;
  a.seq_lens = nullptr;
  a.status = p->d_status;
  a.num_tokens = num_tokens;
  a.B = batch;
  a.Hkv = p->g.num_kv_heads;
  a.D = p->g.head_dim;
  a.BS = p->g.block_size;
  a.L = p->g.num_layers;
  a.layer = layer;
  a.max_blocks = max_blocks;
  a.num_blocks = p->g.num_blocks;
  a.in_dtype = in_dtype;
  a.kv_dtype = p->g.kv_dtype;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.block_scales = fp8 ? p->d_block_scales : nullptr;
  return launch_append(a, stream) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int kv_append(pkv_pool* p, int layer, const void* d_k, const void* d_v, pkv_dtype in_dtype,
              const int32_t* d_block_tables, int max_blocks_per_seq, const int32_t* d_positions,
              int batch, float k_scale, float v_scale, cudaStream_t stream) {
  return append_common(p, layer, d_k, d_v, in_dtype, d_block_tables, max_blocks_per_seq, batch,
                       nullptr, d_positions, batch, k_scale, v_scale, stream);
}

int kv_append_tokens(pkv_pool* p, int layer, const void* d_k, const void* d_v, pkv_dtype in_dtype,
                     const int32_t* d_block_tables, int max_blocks_per_seq, int batch,
                     const int32_t* d_seq_ids, const int32_t* d_positions, int64_t num_tokens,
                     float k_scale, float v_scale, cudaStream_t stream) {
  if (num_tokens > 0 && !d_seq_ids) return PKV_EINVAL;
  return append_common(p, layer, d_k, d_v, in_dtype, d_block_tables, max_blocks_per_seq, batch,
                       d_seq_ids, d_positions, num_tokens, k_scale, v_scale, stream);
}

int kv_pool_set_block_scales(pkv_pool* p, float* d_scales) {
  if (!p) return PKV_EINVAL;
  if (d_scales && (p->g.kv_dtype != PKV_FP8_E4M3 || !aligned16(d_scales))) return PKV_EINVAL;
  p->d_block_scales = d_scales;
  return PKV_OK;
}

int kv_block_scales(pkv_pool* p, int layer, const void* d_k, const void* d_v, pkv_dtype in_dtype,
                    const int32_t* d_block_tables, int max_blocks_per_seq, int batch,
                    const int32_t* d_seq_ids, const int32_t* d_positions, int64_t num_tokens,
                    int group_tokens, cudaStream_t stream) {
  if (!p || !p->d_block_scales || layer < 0 || layer >= p->g.num_layers || num_tokens < 0 ||
      batch < 0 || !act_dtype(in_dtype))
    return PKV_EINVAL;
  if (group_tokens == 0) group_tokens = p->g.block_size;
  if (group_tokens < p->g.block_size || group_tokens % p->g.block_size != 0) return PKV_EINVAL;
  if (num_tokens > 0 &&
      (!d_k || !d_v || !d_block_tables || !d_positions || max_blocks_per_seq < 1 || batch < 1))
    return PKV_EINVAL;
  AppendArgs a{};
  a.k = d_k;
  a.v = d_v;
  a.tables = d_block_tables;
  a.seq_ids = d_seq_ids;
  a.positions = d_positions;
  a.num_tokens = num_tokens;
  a.B = batch;
  a.Hkv = p->g.num_kv_heads;
  a.D = p->g.head_dim;
  a.BS = p->g.block_size;
  a.L = p->g.num_layers;
  a.layer = layer;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = p->g.num_blocks;
  a.in_dtype = in_dtype;
  a.kv_dtype = p->g.kv_dtype;
  a.group_tokens = group_tokens;
  return launch_block_scales(a, p->d_block_scales, stream) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int kv_absmax(const void* d_x, pkv_dtype dtype, int64_t n, float* d_amax, cudaStream_t stream) {
  if (!d_amax || n < 0 || (n > 0 && !d_x) || !act_dtype(dtype)) return PKV_EINVAL;
  return launch_absmax(d_x, dtype, n, d_amax, stream) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int kv_fp8_scale(const float* d_amax, int n, float* d_scale, cudaStream_t stream) {
  if (!d_amax || !d_scale || n < 1) return PKV_EINVAL;
  return launch_fp8_scale(d_amax, n, d_scale, stream) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

size_t paged_decode_workspace_bytes_mq(const pkv_geometry* g, int batch, int q_len,
                                       int max_seq_len, int num_splits) {
  if (!geometry_ok(g) || batch < 0 || q_len < 1 || max_seq_len < 0 || num_splits < 0) return 0;
  DeviceInfo dev;
  if (!device_info(&dev)) return 0;
  if (num_splits > 0) return fixed_ws(*g, batch, q_len, num_splits, nullptr) + 256;
  size_t need = fixed_ws(*g, batch, q_len, simt_auto_splits(*g, batch, max_seq_len, dev.sms),
                         nullptr);
  for (int hg = 1; hg <= 8; ++hg) {
    if (!hg_ok(*g, hg)) continue;
    for (int c = 1; c <= 8; ++c) {   // every CTAs-per-SM count plan_mma accepts
      MmaPlan p;
      p.HG = hg;
      p.NHG = g->num_kv_heads / hg;
      p.grid = dev.sms * c;
      need = std::max(need, balanced_ws(*g, batch, q_len, p).bytes);
    }
  }
  return need + 256;
}

size_t paged_decode_workspace_bytes(const pkv_geometry* g, int batch, int max_seq_len,
                                    int num_splits) {
  return paged_decode_workspace_bytes_mq(g, batch, 1, max_seq_len, num_splits);
}

// Partials computed over a shared prefix, merged into every output row.
struct ExtPartials {
  const float* o;          // [count][B * Hq][D]
  const float* lse;        // [count][B * Hq]
  int count;
  const int32_t* len_off;  // per sequence: the tokens before its private part
};

// Shared body of paged_decode_attention_ex and paged_decode_step.  With k_new
// set, every sequence's new token is first stored at position seq_lens[s] - 1
// (fused into the tensor-core kernel, or a separate append launch otherwise).
// With ext set (shared-prefix decode) the tensor-core kernel in balanced mode
// is required and the merge adds the external partials.
static int decode_common(void* d_out, pkv_dtype out_dtype, const void* d_q, pkv_dtype q_dtype,
                         int q_len, const void* d_k_new, const void* d_v_new, int new_dtype,
                         const pkv_pool* pool, int layer, const int32_t* d_block_tables,
                         int max_blocks_per_seq, const int32_t* d_seq_lens, int batch,
                         int max_seq_len, float scale, float k_scale, float v_scale,
                         int num_splits, void* d_workspace, size_t ws_bytes,
                         const pkv_launch_opts* opts, cudaStream_t stream,
                         const ExtPartials* ext = nullptr, float* out_lse = nullptr) {
  pkv_pool* p = const_cast<pkv_pool*>(pool);
  if (!p || batch < 0 || max_seq_len < 0 || num_splits < 0 || layer < 0 ||
      layer >= p->g.num_layers || q_len < 1)
    return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  const pkv_geometry& g = p->g;
  if (q_len > 1 && d_k_new) return PKV_EINVAL;
  if (!d_out || !d_q || !d_block_tables || !d_seq_lens || max_blocks_per_seq < 1)
    return PKV_EINVAL;
  if (!act_dtype(out_dtype) || !act_dtype(q_dtype) || !aligned16(d_q) || !aligned16(d_out))
    return PKV_EINVAL;
  if ((long long)max_seq_len > (long long)max_blocks_per_seq * g.block_size) return PKV_EINVAL;
  if (!std::isfinite(scale)) return PKV_EINVAL;
  const bool fp8 = g.kv_dtype == PKV_FP8_E4M3;
  const float* bscales = fp8 ? p->d_block_scales : nullptr;
  if (fp8 && !bscales &&
      (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale)))
    return PKV_EINVAL;
  if (bscales) k_scale = v_scale = 1.f;   // the per-tile scales take their place
  const bool fused_append = d_k_new != nullptr;
  if (fused_append) {
    if (!d_v_new || !aligned16(d_k_new) || !aligned16(d_v_new)) return PKV_EINVAL;
    if (fp8 ? !act_dtype(new_dtype) : new_dtype != g.kv_dtype) return PKV_EINVAL;
  }
  const int phase = opts ? opts->phase : 0;
  const int kernel = opts ? opts->kernel : 0;
  const int pdl = opts ? opts->pdl : 0;
  if (phase < 0 || phase > 2 || kernel < 0 || kernel > 3 || pdl < 0 || pdl > 1)
    return PKV_EINVAL;
  DeviceInfo dev;
  if (!device_info(&dev)) return PKV_ECUDA;

  const int G = g.num_q_heads / g.num_kv_heads;
  // the tensor-core kernel runs f16 MMAs on E4M3 pools: bf16 and f16 q fit them
  // exactly after a power-of-two prescale, f32 q would be rounded, so it goes to
  // the CUDA-core kernel (fp32) instead
  const bool q_ok_mma = fp8 ? (q_dtype == PKV_BF16 || q_dtype == PKV_F16)
                            : (g.kv_dtype == PKV_BF16 ? q_dtype == PKV_BF16 : q_dtype == PKV_F16);
  const bool mma_ok = mma_supported(g.kv_dtype, g.block_size, g.head_dim, G, q_len) && q_ok_mma;
  const bool simt_ok = g.head_dim % 32 == 0 && g.head_dim <= 256 && G <= 16 && q_len == 1;
  // chunks with more query rows per KV head than the mma.sync kernel holds go to
  // the tcgen05 chunked-prefill kernel (also forced with kernel = 3)
  const bool tc_ok = !fused_append && prefill_tc_supported(g.kv_dtype, q_dtype, g.block_size,
                                                           g.head_dim, G);
  if (kernel == 3 || (kernel == 0 && q_len > 1 && !mma_ok && tc_ok)) {
    if (!tc_ok) return PKV_EUNSUPPORTED;
    if (num_splits != 0 || phase == 2) return phase == 2 ? PKV_OK : PKV_EUNSUPPORTED;
    if (batch > 65535 || g.num_kv_heads > 65535) return PKV_EUNSUPPORTED;
    const CUtensorMap* map = p->tmap_tiles();
    if (!map) return PKV_ECUDA;
    DecodeArgs t{};
    t.q = d_q;
    t.out = d_out;
    t.tables = d_block_tables;
    t.seq_lens = d_seq_lens;
    t.status = p->d_status;
    t.B = batch;
    t.Hq = g.num_q_heads;
    t.Hkv = g.num_kv_heads;
    t.G = G;
    t.D = g.head_dim;
    t.BS = g.block_size;
    t.L = g.num_layers;
    t.layer = layer;
    t.max_blocks = max_blocks_per_seq;
    t.num_blocks = g.num_blocks;
    t.q_dtype = q_dtype;
    t.out_dtype = out_dtype;
    t.kv_dtype = g.kv_dtype;
    t.q_len = q_len;
    t.R = G * q_len;
    // E4M3 pools: per-tensor scales as for the decode kernel (k_scale on the
    // softmax scale, v_scale on the output); per-block ones when each tile is
    // converted to f16
    t.qk_scale_log2 = (float)((double)scale * 1.4426950408889634 * (fp8 ? (double)k_scale : 1.0));
    t.v_scale = fp8 ? v_scale : 1.f;
    t.block_scales = bscales;
    return launch_prefill_tc(map, t, stream) == cudaSuccess ? PKV_OK : PKV_ECUDA;
  }
  bool use_mma;
  if (ext || out_lse) {
    if (!mma_ok || num_splits != 0 || q_len != 1 || kernel == 1) return PKV_EUNSUPPORTED;
    use_mma = true;
  } else if (kernel == 2) {
    if (!mma_ok) return PKV_EUNSUPPORTED;
    use_mma = true;
  } else if (kernel == 1) {
    if (!simt_ok) return PKV_EUNSUPPORTED;
    use_mma = false;
  } else {
    if (!mma_ok && !simt_ok) return PKV_EUNSUPPORTED;
    use_mma = mma_ok;
  }

  DecodeArgs a{};
  a.q = d_q;
  a.out = d_out;
  a.pool = p->d_pool;
  a.tables = d_block_tables;
  a.seq_lens = d_seq_lens;
  a.status = p->d_status;
  a.B = batch;
  a.Hq = g.num_q_heads;
  a.Hkv = g.num_kv_heads;
  a.G = G;
  a.D = g.head_dim;
  a.BS = g.block_size;
  a.L = g.num_layers;
  a.layer = layer;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = g.num_blocks;
  a.q_dtype = q_dtype;
  a.out_dtype = out_dtype;
  a.kv_dtype = g.kv_dtype;
  a.qk_scale_log2 = (float)((double)scale * 1.4426950408889634 * (fp8 ? (double)k_scale : 1.0));
  a.v_scale = fp8 ? v_scale : 1.f;
  a.k_enc_scale = k_scale;
  a.v_enc_scale = v_scale;
  a.block_scales = bscales;
  a.new_dtype = new_dtype;
  a.q_len = q_len;
  a.R = G * q_len;
  if (d_workspace && !aligned16(d_workspace)) return PKV_EINVAL;
  char* ws = static_cast<char*>(d_workspace);

  // without the fused path the new tokens go in through the append kernel first
  auto append_first = [&]() -> int {
    if (!fused_append || phase == 2) return PKV_OK;
    AppendArgs ap{};
    ap.pool = p->d_pool;
    ap.k = d_k_new;
    ap.v = d_v_new;
    ap.tables = d_block_tables;
    ap.seq_ids = nullptr;
    ap.positions = nullptr;
    ap.seq_lens = d_seq_lens;
    ap.status = p->d_status;
    ap.num_tokens = batch;
    ap.B = batch;
    ap.Hkv = g.num_kv_heads;
    ap.D = g.head_dim;
    ap.BS = g.block_size;
    ap.L = g.num_layers;
    ap.layer = layer;
    ap.max_blocks = max_blocks_per_seq;
    ap.num_blocks = g.num_blocks;
    ap.in_dtype = new_dtype;
    ap.kv_dtype = g.kv_dtype;
    ap.k_scale = k_scale;
    ap.v_scale = v_scale;
    ap.block_scales = bscales;
    return launch_append(ap, stream) == cudaSuccess ? PKV_OK : PKV_ECUDA;
  };

  if (use_mma) {
    MmaPlan plan;
    if (!plan_mma(g, dev, opts, &plan)) return PKV_EUNSUPPORTED;
    a.HG = plan.HG;
    a.NHG = plan.NHG;
    a.stages = plan.stages;
    a.smem_bytes = (int)plan.smem;
    a.pdl = pdl;
    if (fused_append) {
      a.k_new = d_k_new;
      a.v_new = d_v_new;
    }
    const CUtensorMap* map = p->tmap(plan.HG);
    if (!map) return PKV_ECUDA;
    if (num_splits == 0) {
      const BalancedWs w = balanced_ws(g, batch, q_len, plan);
      if (!ws || ws_bytes < w.bytes) return PKV_ENOMEM;
      a.mode = 0;
      a.S = 0;
      a.part_o = reinterpret_cast<float*>(ws + w.o_off);
      a.part_lse = reinterpret_cast<float*>(ws + w.lse_off);
      a.unit_info = reinterpret_cast<int2*>(ws + w.info_off);
      a.slots = plan.grid + batch * plan.NHG;
      a.out_lse = out_lse;
      // the merge may be scheduled at the attention grid's start (E4M3 pools: at its
      // end, measured 0.4% faster there)
      a.early_trigger = phase == 0 && !fp8 ? 1 : 0;
      if (ext) {
        a.ext_o = ext->o;
        a.ext_lse = ext->lse;
        a.ext_count = ext->count;
        a.len_off = ext->len_off;
      }
      if (phase != 2 && launch_decode_mma(map, a, plan.grid, 1, stream) != cudaSuccess)
        return PKV_ECUDA;
      if (phase != 1) {
        const cudaError_t e = ext ? launch_merge_units_ext(a, stream)
                                  : launch_merge_units(a, phase == 0, stream);
        if (e != cudaSuccess) return PKV_ECUDA;
      }
      return PKV_OK;
    }
    size_t lse_off = 0;
    const size_t need = fixed_ws(g, batch, q_len, num_splits, &lse_off);
    if (num_splits > 1 && (!ws || ws_bytes < need)) return PKV_ENOMEM;
    a.mode = 1;
    a.S = num_splits;
    a.part_o = num_splits > 1 ? reinterpret_cast<float*>(ws) : nullptr;
    a.part_lse = num_splits > 1 ? reinterpret_cast<float*>(ws + lse_off) : nullptr;
    const long long units = (long long)batch * plan.NHG;
    if (units > 65535) return PKV_EUNSUPPORTED;
    if (phase != 2 && launch_decode_mma(map, a, num_splits, (int)units, stream) != cudaSuccess)
      return PKV_ECUDA;
    if (num_splits > 1 && phase != 1 &&
        launch_merge_rows(d_out, out_dtype, a.part_o, a.part_lse, batch * q_len * g.num_q_heads,
                          num_splits, g.head_dim, phase == 0, stream) != cudaSuccess)
      return PKV_ECUDA;
    return PKV_OK;
  }

  // SIMT kernel: fixed partitions (automatic count when num_splits == 0)
  const int S = num_splits > 0 ? num_splits : simt_auto_splits(g, batch, max_seq_len, dev.sms);
  if (batch > 65535 || g.num_kv_heads > 65535) return PKV_EUNSUPPORTED;
  size_t lse_off = 0;
  const size_t need = fixed_ws(g, batch, 1, S, &lse_off);
  if (S > 1 && (!ws || ws_bytes < need)) return PKV_ENOMEM;
  a.mode = 1;
  a.S = S;
  a.part_o = S > 1 ? reinterpret_cast<float*>(ws) : nullptr;
  a.part_lse = S > 1 ? reinterpret_cast<float*>(ws + lse_off) : nullptr;
  const int rc = append_first();
  if (rc != PKV_OK) return rc;
  if (phase != 2 && launch_decode_simt(a, stream) != cudaSuccess) return PKV_ECUDA;
  if (S > 1 && phase != 1 &&
      launch_merge_rows(d_out, out_dtype, a.part_o, a.part_lse, batch * g.num_q_heads, S,
                        g.head_dim, phase == 0, stream) != cudaSuccess)
    return PKV_ECUDA;
  return PKV_OK;
}

// ---------------------------------------------------------------- shared-prefix decode
// Workspace sections: prefix partials O [S][B*Hq][D] and lse [S][B*Hq], then the
// decode's own workspace.
struct CascadeWs {
  size_t o_off, lse_off, dec_off, bytes;
  int S;          // key splits of the prefix pass
};
static CascadeWs cascade_ws(const pkv_geometry& g, int batch, int max_blocks, int prefix_len_max,
                            int sms, size_t decode_bytes) {
  CascadeWs w;
  const int G = g.num_q_heads / g.num_kv_heads;
  const int qtiles = (batch * G + 127) / 128;           // 128-row query tiles of the prefix pass
  const int ctas = ((qtiles + 1) / 2) * g.num_kv_heads;  // CTAs per key split
  const int ktiles = (prefix_len_max + 63) / 64;
  // as many key splits as keep every CTA in the first wave (one CTA per SM: the
  // kernel takes the SM's shared and tensor memory); a second, partial wave
  // would double the pass's time
  int S = ctas > 0 ? std::max(1, sms / ctas) : 1;
  S = std::max(1, std::min(S, std::min(std::max(ktiles, 1), 64)));
  w.S = S;
  const size_t rows = (size_t)batch * g.num_q_heads;
  (void)max_blocks;
  w.o_off = 0;
  w.lse_off = w.o_off + align256((size_t)w.S * rows * g.head_dim * 4);
  w.dec_off = w.lse_off + align256((size_t)w.S * rows * 4);
  w.bytes = w.dec_off + decode_bytes;
  return w;
}

size_t paged_decode_workspace_bytes_cascade(const pkv_geometry* g, int batch,
                                            int max_blocks_per_seq, int max_seq_len,
                                            int prefix_len_max) {
  if (!geometry_ok(g) || batch < 0 || max_blocks_per_seq < 1 || max_seq_len < 0 ||
      prefix_len_max < 0)
    return 0;
  DeviceInfo dev;
  if (!device_info(&dev)) return 0;
  const size_t dec = paged_decode_workspace_bytes(g, batch, max_seq_len, 0);
  return cascade_ws(*g, batch, max_blocks_per_seq, prefix_len_max, dev.sms, dec).bytes;
}

int paged_decode_attention_cascade(void* d_out, pkv_dtype out_dtype, const void* d_q,
                                   pkv_dtype q_dtype, const pkv_pool* pool, int layer,
                                   const int32_t* d_prefix_table, int prefix_blocks,
                                   int prefix_len_max, const int32_t* d_prefix_lens,
                                   const int32_t* d_block_tables, int max_blocks_per_seq,
                                   const int32_t* d_seq_lens, int batch, int max_seq_len,
                                   float scale, float k_scale, float v_scale, void* d_workspace,
                                   size_t ws_bytes, const pkv_launch_opts* opts,
                                   cudaStream_t stream) {
  pkv_pool* p = const_cast<pkv_pool*>(pool);
  if (!p || batch < 0 || layer < 0 || layer >= p->g.num_layers || max_seq_len < 0 ||
      prefix_len_max < 0 || max_blocks_per_seq < 1)
    return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  const pkv_geometry& g = p->g;
  const int G = g.num_q_heads / g.num_kv_heads;
  if (!d_out || !d_q || !d_block_tables || !d_seq_lens || !d_prefix_lens || !d_workspace ||
      !aligned16(d_workspace) || !aligned16(d_q) || !aligned16(d_out) || !act_dtype(out_dtype))
    return PKV_EINVAL;
  if (prefix_len_max % g.block_size != 0 ||
      (prefix_len_max > 0 && (!d_prefix_table || prefix_blocks * g.block_size < prefix_len_max)))
    return PKV_EINVAL;
  if ((long long)max_seq_len > (long long)max_blocks_per_seq * g.block_size) return PKV_EINVAL;
  if (!std::isfinite(scale)) return PKV_EINVAL;
  const bool fp8 = g.kv_dtype == PKV_FP8_E4M3;
  const float* bscales = fp8 ? p->d_block_scales : nullptr;
  if (fp8 && !bscales &&
      (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale)))
    return PKV_EINVAL;
  if (!fp8 || bscales) k_scale = v_scale = 1.f;   // unused, or the per-block scales instead
  if (!prefill_tc_supported(g.kv_dtype, q_dtype, g.block_size, g.head_dim, G) ||
      !mma_supported(g.kv_dtype, g.block_size, g.head_dim, G, 1) || batch > 65535)
    return PKV_EUNSUPPORTED;
  const int kernel = opts ? opts->kernel : 0;
  const int phase = opts ? opts->phase : 0;
  if (kernel != 0 && kernel != 2 && kernel != 3) return PKV_EINVAL;
  if (phase < 0 || phase > 2) return PKV_EINVAL;
  DeviceInfo dev;
  if (!device_info(&dev)) return PKV_ECUDA;
  const size_t dec = paged_decode_workspace_bytes(&g, batch, max_seq_len, 0);
  const CascadeWs w = cascade_ws(g, batch, max_blocks_per_seq, prefix_len_max, dev.sms, dec);
  // A prefix whose K/V fill at most a quarter of L2 is already read from HBM
  // about once by the plain decode: every sequence reaches its first blocks at
  // the start of the launch and the repeats hit in L2.  The repeats still cost
  // the decode L2 traffic (measured on the 70B-shaped batch, 64 sequences
  // sharing 17 MB: about 23 TB/s of repeats saved by the prefix pass), while the
  // prefix pass costs about 30 us plus its K/V streamed once per pair of
  // 128-row query tiles at about 5 TB/s.  So such a call runs the prefix pass
  // only when the saving is larger, else (or with kernel = 2) the plain decode
  // over the sequences' own tables, after the same prefix check; kernel = 3
  // always takes the prefix pass.
  const size_t prefix_bytes = (size_t)prefix_len_max * 2 * g.num_kv_heads * g.head_dim *
                              elem_bytes(g.kv_dtype);
  const int pairs = ((batch * G + 127) / 128 + 1) / 2;
  const double saved_us = (batch - 1) * (double)prefix_bytes / 23e12 * 1e6;
  const double cost_us = 30.0 + pairs * (double)prefix_bytes / 5e12 * 1e6;
  const bool plain = kernel == 2 || (kernel == 0 && prefix_bytes * 4 <= (size_t)dev.l2_bytes &&
                                     saved_us <= cost_us);
  if (ws_bytes < w.bytes) return PKV_ENOMEM;
  char* ws = static_cast<char*>(d_workspace);
  float* ext_o = reinterpret_cast<float*>(ws + w.o_off);
  float* ext_lse = reinterpret_cast<float*>(ws + w.lse_off);

  // 1. the check that each sequence's prefix is the shared one (it lets the
  //    prefix pass be scheduled at once: nothing after it reads what it writes)
  if (phase != 2 && launch_prefix_check(d_block_tables, max_blocks_per_seq, d_seq_lens,
                                        prefix_len_max > 0 ? d_prefix_table : d_block_tables,
                                        prefix_len_max > 0 ? prefix_blocks : 0, d_prefix_lens,
                                        prefix_len_max, batch, g.block_size, p->d_status,
                                        stream) != cudaSuccess)
    return PKV_ECUDA;
  if (plain)
    return phase == 1 ? PKV_OK
                      : decode_common(d_out, out_dtype, d_q, q_dtype, 1, nullptr, nullptr, 0, pool,
                                      layer, d_block_tables, max_blocks_per_seq, d_seq_lens, batch,
                                      max_seq_len, scale, k_scale, v_scale, 0, ws + w.dec_off,
                                      ws_bytes - w.dec_off, nullptr, stream);
  // 2. the shared prefix once for every sequence: tcgen05 tiles of 128 query rows
  //    (sequences x heads of a KV head), key range cut into w.S splits
  if (prefix_len_max > 0 && phase != 2) {
    const CUtensorMap* map = p->tmap_tiles();
    if (!map) return PKV_ECUDA;
    DecodeArgs t{};
    t.q = d_q;
    t.out = ext_o;
    t.out_lse = ext_lse;
    t.key_limit = d_prefix_lens;
    t.tables = d_prefix_table;
    t.seq_lens = d_prefix_lens;                   // unread: the length comes with the launch
    t.status = p->d_status;
    t.B = 1;
    t.Hq = g.num_q_heads;
    t.Hkv = g.num_kv_heads;
    t.G = G;
    t.D = g.head_dim;
    t.BS = g.block_size;
    t.L = g.num_layers;
    t.layer = layer;
    t.max_blocks = prefix_blocks;
    t.num_blocks = g.num_blocks;
    t.q_dtype = q_dtype;
    t.out_dtype = PKV_F32;
    t.kv_dtype = g.kv_dtype;
    t.q_len = batch;
    t.R = G * batch;
    t.S = w.S;
    // chained behind the prefix check: the pass reads only the caller's inputs (the
    // prefix length comes with the launch)
    t.casc_len = prefix_len_max;
    t.pdl = 1;
    // E4M3: per-tensor scales on the softmax scale and the partial O (as the
    // decode kernel's partials carry them), per-block ones in the tile conversion
    t.qk_scale_log2 = (float)((double)scale * 1.4426950408889634 * (double)k_scale);
    t.v_scale = v_scale;
    t.block_scales = bscales;
    if (launch_prefill_tc(map, t, stream) != cudaSuccess) return PKV_ECUDA;
  }
  // 3. the private suffixes, merged with the prefix partials: the decode reads each
  //    sequence's own table from the end of its prefix (prefix_lens[s] tokens, whole
  //    blocks); chained behind the prefix pass when this call launched it (the
  //    decode takes SMs as the pass's CTAs retire and waits for the pass before it
  //    writes)
  if (phase == 1) return PKV_OK;
  const ExtPartials ext{ext_o, ext_lse, prefix_len_max > 0 ? w.S : 0,
                        prefix_len_max > 0 ? d_prefix_lens : nullptr};
  pkv_launch_opts chained{};
  chained.pdl = 1;
  const bool chain = prefix_len_max > 0 && phase == 0;
  return decode_common(d_out, out_dtype, d_q, q_dtype, 1, nullptr, nullptr, 0, pool, layer,
                       d_block_tables, max_blocks_per_seq, d_seq_lens, batch, max_seq_len, scale,
                       k_scale, v_scale, 0, ws + w.dec_off, ws_bytes - w.dec_off,
                       chain ? &chained : nullptr, stream, &ext);
}

int paged_decode_attention_ex(void* d_out, pkv_dtype out_dtype, const void* d_q, pkv_dtype q_dtype,
                              const pkv_pool* pool, int layer, const int32_t* d_block_tables,
                              int max_blocks_per_seq, const int32_t* d_seq_lens, int batch,
                              int max_seq_len, float scale, float k_scale, float v_scale,
                              int num_splits, void* d_workspace, size_t ws_bytes,
                              const pkv_launch_opts* opts, cudaStream_t stream) {
  return decode_common(d_out, out_dtype, d_q, q_dtype, 1, nullptr, nullptr, 0, pool, layer,
                       d_block_tables, max_blocks_per_seq, d_seq_lens, batch, max_seq_len, scale,
                       k_scale, v_scale, num_splits, d_workspace, ws_bytes, opts, stream);
}

int paged_decode_attention_partial(float* d_out, float* d_lse, const void* d_q,
                                   pkv_dtype q_dtype, const pkv_pool* pool, int layer,
                                   const int32_t* d_block_tables, int max_blocks_per_seq,
                                   const int32_t* d_seq_lens, int batch, int max_seq_len,
                                   float scale, float k_scale, float v_scale, void* d_workspace,
                                   size_t ws_bytes, cudaStream_t stream) {
  if (batch > 0 && !d_lse) return PKV_EINVAL;
  return decode_common(d_out, PKV_F32, d_q, q_dtype, 1, nullptr, nullptr, 0, pool, layer,
                       d_block_tables, max_blocks_per_seq, d_seq_lens, batch, max_seq_len, scale,
                       k_scale, v_scale, 0, d_workspace, ws_bytes, nullptr, stream, nullptr, d_lse);
}

int paged_decode_attention_mq(void* d_out, pkv_dtype out_dtype, const void* d_q,
                              pkv_dtype q_dtype, int q_len, const pkv_pool* pool, int layer,
                              const int32_t* d_block_tables, int max_blocks_per_seq,
                              const int32_t* d_seq_lens, int batch, int max_seq_len, float scale,
                              float k_scale, float v_scale, int num_splits, void* d_workspace,
                              size_t ws_bytes, const pkv_launch_opts* opts, cudaStream_t stream) {
  return decode_common(d_out, out_dtype, d_q, q_dtype, q_len, nullptr, nullptr, 0, pool, layer,
                       d_block_tables, max_blocks_per_seq, d_seq_lens, batch, max_seq_len, scale,
                       k_scale, v_scale, num_splits, d_workspace, ws_bytes, opts, stream);
}

int paged_decode_step(void* d_out, pkv_dtype out_dtype, const void* d_q, pkv_dtype q_dtype,
                      const void* d_k_new, const void* d_v_new, pkv_dtype new_dtype,
                      const pkv_pool* pool, int layer, const int32_t* d_block_tables,
                      int max_blocks_per_seq, const int32_t* d_seq_lens, int batch,
                      int max_seq_len, float scale, float k_scale, float v_scale, int num_splits,
                      void* d_workspace, size_t ws_bytes, const pkv_launch_opts* opts,
                      cudaStream_t stream) {
  if (!d_k_new) return PKV_EINVAL;
  return decode_common(d_out, out_dtype, d_q, q_dtype, 1, d_k_new, d_v_new, new_dtype, pool, layer,
                       d_block_tables, max_blocks_per_seq, d_seq_lens, batch, max_seq_len, scale,
                       k_scale, v_scale, num_splits, d_workspace, ws_bytes, opts, stream);
}

int paged_decode_attention(void* d_out, pkv_dtype out_dtype, const void* d_q, pkv_dtype q_dtype,
                           const pkv_pool* pool, int layer, const int32_t* d_block_tables,
                           int max_blocks_per_seq, const int32_t* d_seq_lens, int batch,
                           int max_seq_len, float scale, float k_scale, float v_scale,
                           int num_splits, void* d_workspace, size_t ws_bytes,
                           cudaStream_t stream) {
  return paged_decode_attention_ex(d_out, out_dtype, d_q, q_dtype, pool, layer, d_block_tables,
                                   max_blocks_per_seq, d_seq_lens, batch, max_seq_len, scale,
                                   k_scale, v_scale, num_splits, d_workspace, ws_bytes, nullptr,
                                   stream);
}

int merge_partials(void* d_out, pkv_dtype out_dtype, const float* d_part_o,
                   const float* d_part_lse, int batch, int num_q_heads, int head_dim,
                   int num_splits, cudaStream_t stream) {
  if (batch < 0 || num_q_heads < 1 || head_dim < 1 || head_dim > 256 || num_splits < 1 ||
      !act_dtype(out_dtype))
    return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  if (!d_out || !d_part_o || !d_part_lse) return PKV_EINVAL;
  const long long rows = (long long)batch * num_q_heads;
  if (rows > 0x7fffffffLL) return PKV_EINVAL;
  return launch_merge_rows(d_out, out_dtype, d_part_o, d_part_lse, (int)rows, num_splits,
                           head_dim, false, stream) == cudaSuccess
             ? PKV_OK
             : PKV_ECUDA;
}

int pkv_check_status(const pkv_pool* p, cudaStream_t stream) {
  if (!p) return PKV_EINVAL;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PKV_ECUDA;
  if (!p->d_status) return PKV_OK;
  int32_t w[PKV_STATUS_BYTES / 4] = {0};
  if (cudaMemcpy(w, p->d_status, PKV_STATUS_BYTES, cudaMemcpyDeviceToHost) != cudaSuccess)
    return PKV_ECUDA;
  if (w[0] != 0 && cudaMemset(p->d_status, 0, PKV_STATUS_BYTES) != cudaSuccess) return PKV_ECUDA;
  return w[0];
}

int pkv_wait_selftest(const pkv_pool* p, cudaStream_t stream) {
  if (!p || !p->d_status) return PKV_EINVAL;
  return launch_wait_selftest(p->d_status, stream) == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

const char* pkv_strerror(int s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument";
    case PKV_ENOMEM: return "out of blocks or workspace";
    case PKV_ECUDA: return "CUDA runtime error";
    case PKV_EBOUNDS: return "block id or position out of range (device)";
    case PKV_ETIMEOUT: return "bounded wait ran out (device)";
    case PKV_EUNSUPPORTED: return "no kernel for this combination";
    default: return "unknown status";
  }
}

uint64_t pkv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
