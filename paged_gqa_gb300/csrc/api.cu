// api.cu -- host side of the C ABI declared in include/paged_gqa.h.
//
// Validates the descriptors, sizes the workspace from host-known bounds, and issues
// the launches on the caller's stream: the plan kernel, then one persistent attention
// kernel per class of row blocks (verify: q_len*G <= 64 rows; prefill: 128-row blocks).
// Nothing here reads device memory, so a call never synchronises.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>

#include "../../include/paged_gqa.h"
#include "common.cuh"
#include "plan.cuh"
#include "tc_kernels.cuh"

namespace pgqa {
__device__ uint32_t g_error_word;
int report_error(int code, const char* what, cudaError_t e);
}

using namespace pgqa;

namespace {

thread_local std::string t_last_error;
thread_local int64_t t_last_plan[8] = {0, 0, 0, 0, 0, 0, 0, 0};
std::atomic<int> g_path{0};
std::atomic<uint32_t> g_stall_test_ns{0};
std::atomic<uint32_t> g_call_seq{0};

// Nonzero, new on every call (Problem::call_tag).
uint32_t next_call_tag() {
  uint32_t t;
  do t = g_call_seq.fetch_add(1) + 1; while (t == 0);
  return t;
}
std::atomic<cudaEvent_t> g_ev_start[kNumClasses], g_ev_stop[kNumClasses];

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether the rows of a written tensor are pairwise disjoint: dims 0 .. nd-1 index rows of
// kHeadDim contiguous elements. Sufficient test: taken in increasing stride order, every
// dim of extent > 1 must step past everything the smaller dims span (no zero, negative or
// interleaved strides), so no two (index tuples) write the same element.
bool rows_disjoint(const pg_tensor* t, int nd) {
  long long ext[4], str[4];
  int n = 0;
  for (int i = 0; i < nd; ++i) {
    if (t->shape[i] <= 1) continue;
    if (t->stride[i] <= 0) return false;
    ext[n] = t->shape[i];
    str[n] = t->stride[i];
    ++n;
  }
  for (int i = 1; i < n; ++i)  // insertion sort by stride
    for (int j = i; j > 0 && str[j] < str[j - 1]; --j) {
      std::swap(str[j], str[j - 1]);
      std::swap(ext[j], ext[j - 1]);
    }
  long long span = kHeadDim;  // elements covered by one index of the dims taken so far
  for (int i = 0; i < n; ++i) {
    if (str[i] < span) return false;
    span = (ext[i] - 1) * str[i] + span;
  }
  return true;
}

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::mutex mu;
  int sms = 0;
  uint32_t* err = nullptr;   // address of g_error_word on this device
  void* ws = nullptr;        // library-owned workspace
  size_t ws_bytes = 0;
};
DeviceState g_dev[kMaxDevices];

int device_state(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(PG_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  DeviceState& s = g_dev[dev];
  std::lock_guard<std::mutex> lk(s.mu);
  if (s.sms == 0) {
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_error_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    s.err = static_cast<uint32_t*>(addr);
    s.sms = sms;
  }
  *out = &s;
  return PG_OK;
}

// ---------------------------------------------------------------- workspace layout --

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct ClassSizes {
  int num_ctas, max_blocks, max_items, max_slots, slot_rows;
};

struct WsLayout {
  ClassSizes cls[kNumClasses];
  size_t off[kNumClasses][8];
  size_t q_amax_off;  // per-CTA maxima of |q| (calls that quantise Q)
  size_t epoch_off;   // the split counters' epoch word
  size_t total;
};

WsLayout make_layout(int num_seqs, int T, int Hq, int Hkv, int sms) {
  WsLayout L{};
  const long long G = Hq / Hkv;
  const long long rows_all = (long long)T * G;
  // verify blocks: one per (sequence, kv head); prefill blocks: 128-row blocks
  const long long vb = (long long)num_seqs * Hkv;
  // a prefill block needs some sequence with q_len*G > 64, so none exist if T*G <= 64
  const long long pb =
      rows_all > kVerifyRows ? (long long)Hkv * ((rows_all + kPrefillRows - 1) / kPrefillRows + num_seqs) : 0;
  const long long nb[2] = {vb, pb};
  const int rows[2] = {kVerifyRows, kPrefillRows};
  size_t at = 0;
  for (int c = 0; c < kNumClasses; ++c) {
    ClassSizes& s = L.cls[c];
    s.num_ctas = sms;
    s.max_blocks = (int)std::max<long long>(1, nb[c]);
    s.max_items = s.max_blocks + s.num_ctas;
    // Split pieces take slots by split_slot_base: below 2 per CTA.
    s.max_slots = nb[c] == 0 ? 0 : 2 * s.num_ctas;
    s.slot_rows = rows[c];
    size_t sz[8] = {
        256,                                                          // n_blocks, n_items, total_tiles
        sizeof(int) * (size_t)(s.num_ctas + 1),                       // cta_item_begin
        sizeof(RowBlock) * (size_t)s.max_blocks,                      // blocks
        sizeof(WorkItem) * (size_t)s.max_items,                       // items
        sizeof(unsigned long long) * (size_t)s.max_blocks,            // counters
        sizeof(uint16_t) * (size_t)s.max_slots * s.slot_rows * kHeadDim, // part_o (f16)
        sizeof(float) * (size_t)s.max_slots * s.slot_rows,            // part_lse
        0};
    for (int i = 0; i < 8; ++i) {
      L.off[c][i] = at;
      at += align256(sz[i]);
    }
  }
  L.q_amax_off = at;
  at += align256(sizeof(float) * (size_t)q_amax_parts(sms));
  L.epoch_off = at;
  at += 256;
  L.total = at;
  return L;
}

ClassPlan class_plan(const WsLayout& L, int c, char* base) {
  ClassPlan cp{};
  const size_t* o = L.off[c];
  cp.n_blocks = reinterpret_cast<int*>(base + o[0]);
  cp.n_items = reinterpret_cast<int*>(base + o[0] + 8);
  cp.total_tiles = reinterpret_cast<long long*>(base + o[0] + 16);
  cp.cta_item_begin = reinterpret_cast<int*>(base + o[1]);
  cp.blocks = reinterpret_cast<RowBlock*>(base + o[2]);
  cp.items = reinterpret_cast<WorkItem*>(base + o[3]);
  cp.counters = reinterpret_cast<unsigned long long*>(base + o[4]);
  cp.epoch = reinterpret_cast<unsigned long long*>(base + L.epoch_off);
  cp.part_o = reinterpret_cast<uint16_t*>(base + o[5]);
  cp.part_lse = reinterpret_cast<float*>(base + o[6]);
  cp.num_ctas = L.cls[c].num_ctas;
  cp.max_blocks = L.cls[c].max_blocks;
  cp.max_items = L.cls[c].max_items;
  cp.max_slots = L.cls[c].max_slots;
  cp.slot_rows = L.cls[c].slot_rows;
  return cp;
}

// ---------------------------------------------------------------- validation --

struct Validated {
  Problem p;
  Pointers ptr;
};

int check_tensor(const pg_tensor* t, const char* name, int ndim) {
  if (!t) return fail(PG_ERR_INVALID_ARG, "%s: null descriptor", name);
  if (t->ndim != ndim) return fail(PG_ERR_INVALID_ARG, "%s: expected %d dims, got %d", name, ndim, t->ndim);
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return fail(PG_ERR_INVALID_ARG, "%s: negative extent", name);
  return PG_OK;
}

int validate(const pg_tensor* q, const pg_tensor* k, const pg_tensor* v, const pg_tensor* bt,
             const pg_tensor* sl, const pg_tensor* qsl, float q_descale, float k_descale,
             float v_descale, float softmax_scale, const pg_tensor* out, bool q_cast, Validated* res) {
  int st;
  if ((st = check_tensor(q, "q", 3)) || (st = check_tensor(k, "k_cache", 4)) ||
      (st = check_tensor(v, "v_cache", 4)) || (st = check_tensor(bt, "block_table", 2)) ||
      (st = check_tensor(sl, "seq_lens", 1)) || (st = check_tensor(qsl, "query_start_loc", 1)) ||
      (st = check_tensor(out, "out", 3)))
    return st;
  if (q->shape[2] != kHeadDim || k->shape[3] != kHeadDim)
    return fail(PG_ERR_UNSUPPORTED, "head_dim must be 256 (q %lld, cache %lld)", (long long)q->shape[2],
                (long long)k->shape[3]);
  if (q->dtype != PG_BF16 && q->dtype != PG_E4M3) return fail(PG_ERR_UNSUPPORTED, "q dtype must be bf16 or e4m3");
  if (k->dtype != PG_BF16 && k->dtype != PG_E4M3) return fail(PG_ERR_UNSUPPORTED, "cache dtype must be bf16 or e4m3");
  if (v->dtype != k->dtype) return fail(PG_ERR_INVALID_ARG, "k_cache and v_cache dtypes differ");
  if (q->dtype == PG_E4M3 && k->dtype != PG_E4M3)
    return fail(PG_ERR_UNSUPPORTED, "e4m3 q needs an e4m3 cache");
  if (out->dtype != PG_BF16) return fail(PG_ERR_UNSUPPORTED, "out must be bf16");
  if (q_cast && (q->dtype != PG_BF16 || k->dtype != PG_E4M3))
    return fail(PG_ERR_UNSUPPORTED, "quantising q needs a bf16 q and e4m3 caches");
  if (bt->dtype != PG_I32 || sl->dtype != PG_I32 || qsl->dtype != PG_I32)
    return fail(PG_ERR_INVALID_ARG, "block_table, seq_lens and query_start_loc must be int32");
  for (int i = 0; i < 4; ++i)
    if (k->shape[i] != v->shape[i]) return fail(PG_ERR_INVALID_ARG, "k_cache and v_cache shapes differ");
  const long long T = q->shape[0], Hq = q->shape[1];
  const long long NB = k->shape[0], P = k->shape[1], Hkv = k->shape[2];
  const long long S = sl->shape[0], W = bt->shape[1];
  if (out->shape[0] != T || out->shape[1] != Hq || out->shape[2] != kHeadDim)
    return fail(PG_ERR_INVALID_ARG, "out shape must equal q shape");
  if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0)
    return fail(PG_ERR_INVALID_ARG, "num_q_heads (%lld) must be a positive multiple of num_kv_heads (%lld)", Hq, Hkv);
  if (P != 16 && P != 32 && P != 64 && P != 128)
    return fail(PG_ERR_UNSUPPORTED, "page size %lld not in {16, 32, 64, 128}", P);
  if (bt->shape[0] != S || qsl->shape[0] != S + 1)
    return fail(PG_ERR_INVALID_ARG, "block_table rows / query_start_loc length must match seq_lens");
  if (T > INT32_MAX / 2 || NB > INT32_MAX || S > INT32_MAX / 2 || W > INT32_MAX / 2 || Hq > 65535)
    return fail(PG_ERR_UNSUPPORTED, "sizes beyond the supported range");
  if (q->stride[2] != 1 || k->stride[3] != 1 || v->stride[3] != 1 || out->stride[2] != 1)
    return fail(PG_ERR_INVALID_ARG, "the head_dim axis must be contiguous");
  if (W > 1 && bt->stride[1] != 1) return fail(PG_ERR_INVALID_ARG, "block_table rows must be contiguous");
  if ((S > 0 && sl->stride[0] != 1) || qsl->stride[0] != 1)
    return fail(PG_ERR_INVALID_ARG, "seq_lens and query_start_loc must be contiguous");
  if (!rows_disjoint(out, 2))
    return fail(PG_ERR_INVALID_ARG, "out strides make (token, head) rows overlap");
  const int qesz = q->dtype == PG_E4M3 ? 1 : 2, kesz = k->dtype == PG_E4M3 ? 1 : 2;
  if (!aligned16(q->data) || !aligned16(k->data) || !aligned16(v->data) || !aligned16(out->data))
    return fail(PG_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned");
  for (int i = 0; i < 2; ++i)
    if ((q->stride[i] * qesz) % 16 || (out->stride[i] * 2) % 16)
      return fail(PG_ERR_INVALID_ARG, "q/out strides must be multiples of 16 bytes");
  for (int i = 0; i < 3; ++i)
    if ((k->stride[i] * kesz) % 16 || (v->stride[i] * kesz) % 16)
      return fail(PG_ERR_INVALID_ARG, "cache strides must be multiples of 16 bytes");
  if ((T > 0 && (!q->data || !out->data)) || (NB > 0 && (!k->data || !v->data)) || !qsl->data ||
      (S > 0 && (!sl->data || (W > 0 && !bt->data))))
    return fail(PG_ERR_INVALID_ARG, "null data pointer");
  if (!std::isfinite(softmax_scale) || !std::isfinite(k_descale) || !std::isfinite(v_descale) ||
      !std::isfinite(q_descale))
    return fail(PG_ERR_INVALID_ARG, "scales must be finite");

  Problem& p = res->p;
  p.num_seqs = (int)S;
  p.T = (int)T;
  p.Hq = (int)Hq;
  p.Hkv = (int)Hkv;
  p.G = (int)(Hq / Hkv);
  p.P = (int)P;
  p.W = (int)W;
  p.NB = (int)NB;
  p.q_is_fp8 = q->dtype == PG_E4M3;
  p.kv_is_fp8 = k->dtype == PG_E4M3;
  p.q_cast = q_cast ? 1 : 0;
  p.q_amax_parts = 0;
  p.q_st = q->stride[0];
  p.q_sh = q->stride[1];
  p.k_sb = k->stride[0];
  p.k_sp = k->stride[1];
  p.k_sh = k->stride[2];
  p.v_sb = v->stride[0];
  p.v_sp = v->stride[1];
  p.v_sh = v->stride[2];
  p.o_st = out->stride[0];
  p.o_sh = out->stride[1];
  p.bt_stride = W > 0 ? bt->stride[0] : 1;
  p.score_scale_log2 = (float)((double)softmax_scale * (double)q_descale * (double)k_descale * 1.4426950408889634);
  p.out_scale = v_descale;
  p.stall_test_ns = g_stall_test_ns.load();
  Pointers& ptr = res->ptr;
  ptr.q = q->data;
  ptr.k = k->data;
  ptr.v = v->data;
  ptr.block_table = static_cast<const int32_t*>(bt->data);
  ptr.seq_lens = static_cast<const int32_t*>(sl->data);
  ptr.qsl = static_cast<const int32_t*>(qsl->data);
  ptr.out = out->data;
  ptr.err = nullptr;
  ptr.q_amax = nullptr;
  return PG_OK;
}

int run(const Validated& val, const pg_tensor* k, const pg_tensor* v, void* ws, size_t ws_bytes,
        const WsLayout& L, DeviceState* ds, cudaStream_t stream) {
  Problem p = val.p;
  Pointers ptr = val.ptr;
  ptr.err = ds->err;
  ClassPlan cp[kNumClasses];
  for (int c = 0; c < kNumClasses; ++c) cp[c] = class_plan(L, c, static_cast<char*>(ws));
  (void)ws_bytes;
  int64_t plan_info[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int path = g_path.load();
  // tcgen05 kernels: the verify and prefill kernels for e4m3 caches, the bf16 kernel (both
  // classes) for a bf16 q with bf16 caches; the warp-MMA kernel under paged_gqa_set_path(1).
  const bool fast_ok = path != 1 && p.kv_is_fp8;
  const bool bf16_ok = path != 1 && !p.kv_is_fp8 && !p.q_is_fp8;
  // Only the tcgen05 kernels cast Q per tensor; nothing else may stand in for them.
  if (p.q_cast && !fast_ok) return fail(PG_ERR_UNSUPPORTED, "quantising q needs the tcgen05 path");
  int launched = 0;
  cudaError_t e;
  if (p.q_cast) {
    p.q_amax_parts = q_amax_parts(ds->sms);
    ptr.q_amax = reinterpret_cast<const float*>(static_cast<char*>(ws) + L.q_amax_off);
    e = launch_q_amax(p, ptr, reinterpret_cast<float*>(static_cast<char*>(ws) + L.q_amax_off), stream);
    if (e != cudaSuccess) return cuda_fail(e, "q amax launch");
    ++launched;
  }
  p.call_tag = next_call_tag();
  // The verify kernel (FP8 or bf16) plans its own class when its CTAs can hold one entry per verify block
  // (sequence x kv head), the class's units fit 31 bits and a block's tiles 16: it then runs
  // first, and the plan kernel (prefill only) and the prefill kernel follow it as
  // programmatic dependents, off the critical path.
  const long long max_tiles = ((long long)p.W * p.P + kTileKeys - 1) / kTileKeys;
  // A single sequence whose q_len x G rows exceed a verify block is all prefill (its q_len is
  // T): then the plan kernel goes first, as the verify kernel would only find nothing to do.
  const bool single_prefill = p.num_seqs == 1 && (long long)p.T * p.G > kVerifyRows;
  p.fused_verify = (fast_ok || bf16_ok) && path != 3 && !single_prefill && (long long)p.num_seqs * p.Hkv <= kFusedMaxBlocks &&
                   max_tiles < (1 << 16) &&
                   (long long)p.num_seqs * p.Hkv * (max_tiles + fixed_cost(0)) < (1LL << 31);
  if (!p.fused_verify) {
    e = launch_plan(p, ptr, cp[0], cp[1], true, false, stream);
    if (e != cudaSuccess) return cuda_fail(e, "plan launch");
    ++launched;
  }
  int used = 0;
  bool prev_ev = false;  // an event was recorded after the previous class's kernel
  for (int c = 0; c < kNumClasses; ++c) {
    bool done = false;
    cudaEvent_t ev0 = g_ev_start[c].load(), ev1 = g_ev_stop[c].load();
    bool after_plan = false;  // this class's kernel directly follows the plan kernel
    if (c == 1 && p.fused_verify) {
      e = launch_plan(p, ptr, cp[0], cp[1], false, !prev_ev, stream);
      if (e != cudaSuccess) return cuda_fail(e, "plan launch");
      ++launched;
      after_plan = true;
    }
    if (ev0 && (e = cudaEventRecord(ev0, stream)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    if (fast_ok || bf16_ok) {
      // the prefill-class kernel follows the verify-class one (or the plan kernel, when the
      // verify kernel planned itself) as a programmatic dependent, when that one is a
      // tcgen05 kernel too and no event sits between them
      const bool dependent = c == 1 && !ev0 && (after_plan || ((used & 2) && !prev_ev));
      int r = bf16_ok ? launch_bf16_tc(p, ptr, cp[c], k, v, stream, dependent, c == 0 && p.fused_verify)
              : (c == 0) ? launch_verify_tc(p, ptr, cp[c], k, v, ds->sms, stream, !p.fused_verify && pdl_enabled())
                         : launch_prefill_tc(p, ptr, cp[c], k, v, ds->sms, stream, dependent);
      if (r < 0) return fail(PG_ERR_CUDA, "tcgen05 %s launch failed: %s", c == 0 ? "verify" : "prefill",
                             tc_last_error());
      if (r == 1) {
        done = true;
        used |= 2 << c;
      }
    }
    if (!done && p.q_cast) return fail(PG_ERR_UNSUPPORTED, "quantising q needs the tcgen05 path");
    if (!done) {
      e = launch_portable(p, ptr, cp[c], c == 0 ? kVerifyRows : kPrefillRows, stream);
      if (e != cudaSuccess) return cuda_fail(e, "portable kernel launch");
      used |= 8 << c;
    }
    ++launched;
    if (ev1 && (e = cudaEventRecord(ev1, stream)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    prev_ev = ev1 != nullptr;
  }
  plan_info[0] = cp[0].num_ctas;
  plan_info[1] = cp[1].num_ctas;
  plan_info[2] = launched;
  plan_info[3] = used;
  plan_info[4] = cp[0].max_blocks;
  plan_info[5] = cp[1].max_blocks;
  plan_info[6] = (int64_t)L.total;
  plan_info[7] = p.fused_verify;
  memcpy(t_last_plan, plan_info, sizeof plan_info);
  return PG_OK;
}

int attn_common(const pg_tensor* q, const pg_tensor* k, const pg_tensor* v, const pg_tensor* bt,
                const pg_tensor* sl, const pg_tensor* qsl, float q_descale, float k_descale,
                float v_descale, float softmax_scale, pg_tensor* out, void* user_ws,
                size_t user_ws_bytes, bool use_user_ws, cudaStream_t stream, bool q_cast = false) {
  Validated val;
  int st = validate(q, k, v, bt, sl, qsl, q_descale, k_descale, v_descale, softmax_scale, out, q_cast, &val);
  if (st) return st;
  if (val.p.num_seqs == 0 || val.p.T == 0) {
    t_last_error.clear();
    return PG_OK;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds))) return st;
  const WsLayout L = make_layout(val.p.num_seqs, val.p.T, val.p.Hq, val.p.Hkv, ds->sms);
  void* ws = nullptr;
  if (use_user_ws) {
    if (!user_ws || (reinterpret_cast<uintptr_t>(user_ws) & 255u))
      return fail(PG_ERR_WORKSPACE, "workspace must be non-null and 256-byte aligned");
    if (user_ws_bytes < L.total)
      return fail(PG_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", user_ws_bytes, L.total);
    ws = user_ws;
    st = run(val, k, v, ws, user_ws_bytes, L, ds, stream);
  } else {
    std::lock_guard<std::mutex> lk(ds->mu);
    if (ds->ws_bytes < L.total) {
      if (ds->ws) {
        // Work already queued may still use the old buffer.
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize before workspace growth");
        cudaFree(ds->ws);
        ds->ws = nullptr;
        ds->ws_bytes = 0;
      }
      size_t want = L.total + L.total / 4;
      e = cudaMalloc(&ds->ws, want);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
      // not required (the split counters are tagged per call), but keeps the first call's
      // workspace contents deterministic
      e = cudaMemsetAsync(ds->ws, 0, want, stream);
      if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace)");
      ds->ws_bytes = want;
    }
    st = run(val, k, v, ds->ws, ds->ws_bytes, L, ds, stream);
  }
  if (st == PG_OK) t_last_error.clear();
  return st;
}

}  // namespace

// Sets the calling thread's last-error message for a failed CUDA call; used by the
// no-alloc entry point (noalloc.cu).
int pgqa::report_error(int code, const char* what, cudaError_t e) {
  return fail(code, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

extern "C" {

int paged_gqa_attn(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                   const pg_tensor* block_table, const pg_tensor* seq_lens,
                   const pg_tensor* query_start_loc, float k_descale, float v_descale,
                   float softmax_scale, pg_tensor* out, pg_stream_t stream) {
  return attn_common(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, 1.0f, k_descale,
                     v_descale, softmax_scale, out, nullptr, 0, false, reinterpret_cast<cudaStream_t>(stream));
}

int paged_gqa_attn_ex(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                      const pg_tensor* block_table, const pg_tensor* seq_lens,
                      const pg_tensor* query_start_loc, float q_descale, float k_descale,
                      float v_descale, float softmax_scale, pg_tensor* out, void* workspace,
                      size_t workspace_bytes, pg_stream_t stream) {
  return attn_common(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, q_descale, k_descale,
                     v_descale, softmax_scale, out, workspace, workspace_bytes, true,
                     reinterpret_cast<cudaStream_t>(stream));
}

int paged_gqa_attn_quant_q(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                           const pg_tensor* block_table, const pg_tensor* seq_lens,
                           const pg_tensor* query_start_loc, float k_descale, float v_descale,
                           float softmax_scale, pg_tensor* out, pg_stream_t stream) {
  return attn_common(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, 1.0f, k_descale,
                     v_descale, softmax_scale, out, nullptr, 0, false, reinterpret_cast<cudaStream_t>(stream),
                     true);
}

int paged_gqa_sparse_attn(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                          const pg_tensor* block_table, const pg_tensor* seq_lens,
                          const pg_tensor* query_start_loc, const pg_tensor* indices, float k_descale,
                          float v_descale, float softmax_scale, pg_tensor* out, pg_stream_t stream) {
  Validated val;
  int st = validate(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, 1.0f, k_descale, v_descale,
                    softmax_scale, out, false, &val);
  if (st) return st;
  if ((st = check_tensor(indices, "indices", 3))) return st;
  if (q->dtype != PG_BF16 || k_cache->dtype != PG_E4M3)
    return fail(PG_ERR_UNSUPPORTED, "sparse attention takes a bf16 q and e4m3 caches");
  for (int i = 0; i < 3; ++i)
    if (k_cache->stride[i] != v_cache->stride[i])
      return fail(PG_ERR_INVALID_ARG, "sparse attention needs k_cache and v_cache with the same strides");
  const Problem& p = val.p;
  if (indices->dtype != PG_I32) return fail(PG_ERR_INVALID_ARG, "indices must be int32");
  if (indices->shape[0] != p.T || indices->shape[1] != p.Hkv)
    return fail(PG_ERR_INVALID_ARG, "indices must be [T, num_kv_heads, K]");
  const long long K = indices->shape[2];
  if (K > INT32_MAX / 2) return fail(PG_ERR_UNSUPPORTED, "sizes beyond the supported range");
  if (K > 1 && indices->stride[2] != 1) return fail(PG_ERR_INVALID_ARG, "indices rows must be contiguous");
  if (K > 0 && p.T > 0 && (!indices->data || (reinterpret_cast<uintptr_t>(indices->data) & 3u)))
    return fail(PG_ERR_INVALID_ARG, "indices must be non-null and 4-byte aligned");
  if (p.num_seqs == 0 || p.T == 0) {
    t_last_error.clear();
    return PG_OK;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds)) != PG_OK) return st;
  SparseArgs a;
  a.q = static_cast<const uint16_t*>(q->data);
  a.q_st = p.q_st;
  a.q_sh = p.q_sh;
  a.k = static_cast<const uint8_t*>(k_cache->data);
  a.v = static_cast<const uint8_t*>(v_cache->data);
  a.kv_sb = p.k_sb;
  a.kv_sp = p.k_sp;
  a.kv_sh = p.k_sh;
  a.bt = val.ptr.block_table;
  a.bt_stride = p.bt_stride;
  a.seq_lens = val.ptr.seq_lens;
  a.qsl = val.ptr.qsl;
  a.idx = static_cast<const int32_t*>(indices->data);
  a.idx_st = indices->stride[0];
  a.idx_sh = indices->stride[1];
  a.K = (int)K;
  a.out = static_cast<uint16_t*>(out->data);
  a.o_st = p.o_st;
  a.o_sh = p.o_sh;
  a.num_seqs = p.num_seqs;
  a.T = p.T;
  a.Hq = p.Hq;
  a.Hkv = p.Hkv;
  a.G = p.G;
  a.HG = (p.G + 15) / 16;
  a.P = p.P;
  a.p_shift = __builtin_ctz((unsigned)p.P);
  a.W = p.W;
  a.NB = p.NB;
  a.score_scale_log2 = (float)((double)softmax_scale * (double)k_descale * 1.4426950408889634);
  a.out_scale = v_descale;
  a.err = ds->err;
  // The warp-level kernel by default: on the sparse workloads of "Tune sparse GQA prefill
  // profile" it is the faster of the two (3.4 vs 4.4 ms on the TP1 shape; the tcgen05 kernel's
  // row gather is bound by the latency of 16-byte copies from L2 with two K stages in
  // flight). paged_gqa_set_path(2) selects the tcgen05 kernel for lists of at least two
  // tiles' worth of keys.
  int used = 0;
  if (g_path.load() == 2) {
    const int r = launch_sparse_tc(a, ds->sms, p.stall_test_ns, reinterpret_cast<cudaStream_t>(stream));
    if (r < 0) return fail(PG_ERR_CUDA, "tcgen05 sparse launch failed: %s", tc_last_error());
    if (r == 1) used = 32;
  }
  if (!used) {
    e = launch_sparse(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse attention launch");
    used = 64;
  }
  int64_t plan_info[8] = {0, 0, 1, used, 0, 0, 0, 0};
  memcpy(t_last_plan, plan_info, sizeof plan_info);
  t_last_error.clear();
  return PG_OK;
}

size_t paged_gqa_workspace_size(int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                                int page_size, int max_blocks_per_seq, int device) {
  (void)max_blocks_per_seq;
  if (num_seqs < 0 || total_q < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || page_size <= 0)
    return 0;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || sms <= 0) return 0;
  return make_layout(num_seqs, total_q, num_q_heads, num_kv_heads, sms).total;
}

const char* paged_gqa_last_error(void) { return t_last_error.c_str(); }

int paged_gqa_check_device_errors(pg_stream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceState* ds = nullptr;
  int st = device_state(dev, &ds);
  if (st) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof word);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  const uint32_t zero = 0;
  e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  if (word & kErrTimeout) return fail(PG_ERR_TIMEOUT, "device: a bounded wait gave up (word 0x%x)", word);
  if (word & (kErrBounds | kErrPage))
    return fail(PG_ERR_DEVICE_BOUNDS, "device: %s%s(word 0x%x)", (word & kErrBounds) ? "sequence bounds " : "",
                (word & kErrPage) ? "page id out of range " : "", word);
  t_last_error.clear();
  return PG_OK;
}

int paged_gqa_set_path(int path) {
  if (path < 0 || path > 3) return fail(PG_ERR_INVALID_ARG, "path must be 0, 1, 2 or 3");
  return g_path.exchange(path);
}

int paged_gqa_set_stall_test(uint32_t wait_ns) { return (int)g_stall_test_ns.exchange(wait_ns); }

int paged_gqa_last_plan(int64_t* out8) {
  if (!out8) return fail(PG_ERR_INVALID_ARG, "null output");
  memcpy(out8, t_last_plan, sizeof t_last_plan);
  return PG_OK;
}

int paged_gqa_set_kernel_events(int cls, void* start, void* stop) {
  if (cls < 0 || cls >= kNumClasses) return fail(PG_ERR_INVALID_ARG, "class must be 0 or 1");
  g_ev_start[cls].store(static_cast<cudaEvent_t>(start));
  g_ev_stop[cls].store(static_cast<cudaEvent_t>(stop));
  return PG_OK;
}

int paged_gqa_cache_write(const pg_tensor* k_new, const pg_tensor* v_new, const pg_tensor* k_cache,
                          const pg_tensor* v_cache, const pg_tensor* block_table, const pg_tensor* seq_lens,
                          const pg_tensor* query_start_loc, float k_descale, float v_descale, pg_stream_t stream) {
  int st;
  if ((st = check_tensor(k_new, "k_new", 3)) || (st = check_tensor(v_new, "v_new", 3)) ||
      (st = check_tensor(k_cache, "k_cache", 4)) || (st = check_tensor(v_cache, "v_cache", 4)) ||
      (st = check_tensor(block_table, "block_table", 2)) || (st = check_tensor(seq_lens, "seq_lens", 1)) ||
      (st = check_tensor(query_start_loc, "query_start_loc", 1)))
    return st;
  if (k_new->dtype != PG_BF16 || v_new->dtype != PG_BF16)
    return fail(PG_ERR_UNSUPPORTED, "k_new and v_new must be bf16");
  if (k_cache->dtype != PG_E4M3 || v_cache->dtype != PG_E4M3)
    return fail(PG_ERR_UNSUPPORTED, "the caches must be e4m3");
  for (int i = 0; i < 3; ++i)
    if (k_new->shape[i] != v_new->shape[i]) return fail(PG_ERR_INVALID_ARG, "k_new and v_new shapes differ");
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i]) return fail(PG_ERR_INVALID_ARG, "k_cache and v_cache shapes differ");
  const long long T = k_new->shape[0], Hkv = k_new->shape[1];
  const long long NB = k_cache->shape[0], P = k_cache->shape[1], S = seq_lens->shape[0], W = block_table->shape[1];
  if (k_new->shape[2] != kHeadDim || k_cache->shape[3] != kHeadDim)
    return fail(PG_ERR_UNSUPPORTED, "head_dim must be 256");
  if (k_cache->shape[2] != Hkv) return fail(PG_ERR_INVALID_ARG, "k_new and the caches disagree on num_kv_heads");
  if (P != 16 && P != 32 && P != 64 && P != 128)
    return fail(PG_ERR_UNSUPPORTED, "page size %lld not in {16, 32, 64, 128}", P);
  if (block_table->shape[0] != S || query_start_loc->shape[0] != S + 1)
    return fail(PG_ERR_INVALID_ARG, "block_table rows / query_start_loc length must match seq_lens");
  if (S == 0 && T > 0) return fail(PG_ERR_INVALID_ARG, "tokens without sequences");
  if (T > INT32_MAX / 2 || NB > INT32_MAX || S > INT32_MAX / 2 || W > INT32_MAX / 2 || Hkv > 65535)
    return fail(PG_ERR_UNSUPPORTED, "sizes beyond the supported range");
  if (block_table->dtype != PG_I32 || seq_lens->dtype != PG_I32 || query_start_loc->dtype != PG_I32)
    return fail(PG_ERR_INVALID_ARG, "block_table, seq_lens and query_start_loc must be int32");
  if (k_new->stride[2] != 1 || v_new->stride[2] != 1 || k_cache->stride[3] != 1 || v_cache->stride[3] != 1)
    return fail(PG_ERR_INVALID_ARG, "the head_dim axis must be contiguous");
  if (W > 1 && block_table->stride[1] != 1) return fail(PG_ERR_INVALID_ARG, "block_table rows must be contiguous");
  if ((S > 0 && seq_lens->stride[0] != 1) || query_start_loc->stride[0] != 1)
    return fail(PG_ERR_INVALID_ARG, "seq_lens and query_start_loc must be contiguous");
  if (!aligned16(k_new->data) || !aligned16(v_new->data) || !aligned16(k_cache->data) || !aligned16(v_cache->data))
    return fail(PG_ERR_INVALID_ARG, "k_new, v_new and the caches must be 16-byte aligned");
  for (int i = 0; i < 2; ++i)
    if ((k_new->stride[i] * 2) % 16 || (v_new->stride[i] * 2) % 16)
      return fail(PG_ERR_INVALID_ARG, "k_new/v_new strides must be multiples of 16 bytes");
  for (int i = 0; i < 3; ++i)
    if (k_cache->stride[i] % 16 || v_cache->stride[i] % 16)
      return fail(PG_ERR_INVALID_ARG, "cache strides must be multiples of 16 bytes");
  if (!rows_disjoint(k_cache, 3) || !rows_disjoint(v_cache, 3))
    return fail(PG_ERR_INVALID_ARG, "cache strides make (page, slot, head) rows overlap");
  if ((T > 0 && (!k_new->data || !v_new->data)) || (NB > 0 && (!k_cache->data || !v_cache->data)) ||
      !query_start_loc->data || (S > 0 && (!seq_lens->data || (W > 0 && !block_table->data))))
    return fail(PG_ERR_INVALID_ARG, "null data pointer");
  if (!(std::isfinite(k_descale) && k_descale > 0.f && std::isfinite(v_descale) && v_descale > 0.f))
    return fail(PG_ERR_INVALID_ARG, "descales must be finite and positive");
  if (T == 0) {  // nothing to write: no device is touched
    t_last_error.clear();
    return PG_OK;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceState* ds = nullptr;
  if ((st = device_state(dev, &ds)) != PG_OK) return st;
  CacheWriteArgs a;
  a.kn = static_cast<const uint16_t*>(k_new->data);
  a.vn = static_cast<const uint16_t*>(v_new->data);
  a.kn_st = k_new->stride[0];
  a.kn_sh = k_new->stride[1];
  a.vn_st = v_new->stride[0];
  a.vn_sh = v_new->stride[1];
  a.kc = static_cast<uint8_t*>(k_cache->data);
  a.vc = static_cast<uint8_t*>(v_cache->data);
  a.kc_sb = k_cache->stride[0];
  a.kc_sp = k_cache->stride[1];
  a.kc_sh = k_cache->stride[2];
  a.vc_sb = v_cache->stride[0];
  a.vc_sp = v_cache->stride[1];
  a.vc_sh = v_cache->stride[2];
  a.bt = static_cast<const int32_t*>(block_table->data);
  a.bt_stride = W > 0 ? block_table->stride[0] : 1;
  a.seq_lens = static_cast<const int32_t*>(seq_lens->data);
  a.qsl = static_cast<const int32_t*>(query_start_loc->data);
  a.num_seqs = (int)S;
  a.T = (int)T;
  a.Hkv = (int)Hkv;
  a.P = (int)P;
  a.p_shift = __builtin_ctz((unsigned)P);
  a.W = (int)W;
  a.NB = (int)NB;
  a.k_scale = 1.f / k_descale;
  a.v_scale = 1.f / v_descale;
  a.err = ds->err;
  e = launch_cache_write(a, ds->sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cache write launch");
  return PG_OK;
}

int paged_gqa_version(void) { return 100; }

}  // extern "C"
