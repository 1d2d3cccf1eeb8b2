// noalloc.cu -- paged_gqa_attn_noalloc: the same call as paged_gqa_attn for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run attention: code inside
// a custom allocator or memory-pool callback, runtimes that forbid allocation after
// start-up so that their memory footprint stays fixed, or code that runs while another
// component owns every free byte of the device. paged_gqa_attn allocates its workspace on
// first need and paged_gqa_attn_ex needs the caller to provide one; this entry point
// instead uses a fixed scratch array that is part of the library's device image.
//
// Limits and sharing:
//   * the scratch is kNoAllocScratchBytes (64 MiB); every GPU on which the library's
//     device code is loaded holds that much memory until the process exits;
//   * a call whose workspace need (paged_gqa_workspace_size) exceeds it returns
//     PG_ERR_WORKSPACE with a message stating both sizes, and launches nothing;
//   * every call on a device uses the same array, which keeps whatever the last call left
//     there. The merge counters in it carry a per-call tag (nothing needs clearing), so
//     results do not depend on earlier calls, but two calls whose work can overlap on the
//     GPU (different streams without ordering between them) race on the array: order
//     them on one stream, or use paged_gqa_attn_ex with separate workspaces;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call before any
//     stream capture.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/paged_gqa.h"

namespace pgqa {
// Sets the calling thread's last-error message (api.cu) and returns `code`.
int report_error(int code, const char* what, cudaError_t e);
}

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up once per device).
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int paged_gqa_attn_noalloc(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                                      const pg_tensor* block_table, const pg_tensor* seq_lens,
                                      const pg_tensor* query_start_loc, float k_descale, float v_descale,
                                      float softmax_scale, pg_tensor* out, pg_stream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    // let the regular entry point validate and report (no workspace: it fails cleanly)
    return paged_gqa_attn_ex(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, 1.0f, k_descale,
                             v_descale, softmax_scale, out, nullptr, 0, stream);
  }
  void* ws = nullptr;
  const cudaError_t e = scratch_address(dev, &ws);
  if (e != cudaSuccess) return pgqa::report_error(PG_ERR_CUDA, "cudaGetSymbolAddress(no-alloc scratch)", e);
  // paged_gqa_attn_ex validates the call, checks the size against the scratch and
  // reports "workspace too small: <scratch> < <needed> bytes" when it does not fit.
  return paged_gqa_attn_ex(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, 1.0f, k_descale,
                           v_descale, softmax_scale, out, ws, kNoAllocScratchBytes, stream);
}
