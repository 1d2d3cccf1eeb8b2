// tc_host.cu -- host helpers of the tcgen05 kernels: TMA tensor maps over the paged caches
// and the launch-error message.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "tc_kernels.cuh"

namespace pgqa {

namespace {

std::mutex g_tc_mu;
thread_local char t_tc_err[256] = "";

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to libcuda).
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  std::lock_guard<std::mutex> lk(g_tc_mu);
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

}  // namespace

void set_tc_error(const char* msg) { snprintf(t_tc_err, sizeof t_tc_err, "%s", msg); }

const char* tc_last_error() { return t_tc_err; }

namespace {

// Encoded maps of recent caches. A serving loop passes the same cache tensors on every
// call, so the map (a host-side encode of ~1-2 us each, two per kernel) is looked up
// instead of re-encoded. The key is everything the encode reads from the descriptor.
struct TmapKey {
  const void* data;
  int dtype;
  int64_t shape[4];
  int64_t stride[3];
  int P;
  bool operator==(const TmapKey& o) const {
    if (data != o.data || dtype != o.dtype || P != o.P) return false;
    for (int i = 0; i < 4; ++i)
      if (shape[i] != o.shape[i]) return false;
    for (int i = 0; i < 3; ++i)
      if (stride[i] != o.stride[i]) return false;
    return true;
  }
};
constexpr int kTmapCache = 16;
struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  bool used;
};
TmapEntry g_tmap_cache[kTmapCache];
int g_tmap_next = 0;
std::mutex g_tmap_mu;

bool encode_cache_tmap(CUtensorMap* m, const pg_tensor* t, int P);

}  // namespace

// 4-D map over a cache [NB, P, Hkv, 256] (see encode_cache_tmap), from the cache of
// recent maps when the same tensor view was seen before.
bool make_cache_tmap(CUtensorMap* m, const pg_tensor* t, int P) {
  TmapKey k{};
  k.data = t->data;
  k.dtype = t->dtype;
  for (int i = 0; i < 4; ++i) k.shape[i] = t->shape[i];
  for (int i = 0; i < 3; ++i) k.stride[i] = t->stride[i];
  k.P = P;
  {
    std::lock_guard<std::mutex> lk(g_tmap_mu);
    for (int i = 0; i < kTmapCache; ++i)
      if (g_tmap_cache[i].used && g_tmap_cache[i].key == k) {
        *m = g_tmap_cache[i].map;
        return true;
      }
  }
  if (!encode_cache_tmap(m, t, P)) return false;
  std::lock_guard<std::mutex> lk(g_tmap_mu);
  TmapEntry& e = g_tmap_cache[g_tmap_next];
  g_tmap_next = (g_tmap_next + 1) % kTmapCache;
  e.key = k;
  e.map = *m;
  e.used = true;
  return true;
}

namespace {

// 4-D map over a cache [NB, P, Hkv, 256]: box = 128 bytes of d x 1 head x the page's rows
// x 1 page, 128-byte swizzle, so one box lands those rows in the layout the MMA descriptors
// expect (8-row atoms of 128 B).
bool encode_cache_tmap(CUtensorMap* m, const pg_tensor* t, int P) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_tc_error("cuTensorMapEncodeTiled unavailable");
    return false;
  }
  // e4m3: a box is one 128-byte d-half of a page; bf16: one 128-byte d-quarter of a page, or
  // of half a page for 128-token pages (the bf16 kernel's sub-tiles hold 64 keys)
  const bool bf16 = t->dtype == PG_BF16;
  const cuuint64_t esz = bf16 ? 2 : 1;
  cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)t->shape[2], (cuuint64_t)t->shape[1],
                        (cuuint64_t)t->shape[0]};
  cuuint64_t strides[3] = {(cuuint64_t)t->stride[2] * esz, (cuuint64_t)t->stride[1] * esz,
                           (cuuint64_t)t->stride[0] * esz};
  cuuint32_t box[4] = {bf16 ? 64u : 128u, 1, (cuuint32_t)(bf16 && P > 64 ? 64 : P), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, t->data, dims,
                  strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[96];
    snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    set_tc_error(buf);
    return false;
  }
  return true;
}

}  // namespace

}  // namespace pgqa
