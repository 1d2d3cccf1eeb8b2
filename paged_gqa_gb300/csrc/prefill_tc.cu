// prefill_tc.cu -- tcgen05 (TMEM, TMA) kernel for prefill blocks: 128 query rows (tokens x
// heads of one kv head) against an FP8 e4m3 paged KV cache, bottom-right causal.
//
// What the pages ask of this path ("asm FP8 FMHA for prefix-hit prefill", summary and
// Results): FP8 Q/K/V with head_dim 256, new tokens attending to cached plus new K/V
// (cu_seqlens_k longer than cu_seqlens_q) under a bottom-right causal mask, GQA group 8 per
// kv head; the pages gather the cached K/V into contiguous buffers and cast to FP8 first,
// this kernel reads the pages in place through the block table ("gfx1250 GDN prefill
// kernels ...; DP points on unified attention": no KV gather before the prefill).
//
// Layout for sm_103a:
//   * one row block = 128 rows (row r = token r / G, head r % G of the kv head); S = Q K^T
//     is one tcgen05.mma kind::f8f6f4 M=128 x N=128 keys x K=256 per tile (8 MMAs of
//     K=32; bf16 Q is split once per block into e4m3 hi + lo and costs 16);
//   * P = 2^(s - m + 4) is split into e4m3 hi + lo (about bf16 precision; a single e4m3 P
//     misses the 5e-3 relative-L2 bar), written into one of two P buffers in TMEM and used
//     from there as the A operand of O += P V: M=128 x N=256 (all of d, V as an MN-major
//     operand whose two 128-byte d-halves sit 16 KB apart), fp32 accumulators in TMEM (S:
//     128 columns, P: 2 x 64, O: 256). S(g+1) only waits for the softmax to have loaded
//     S(g), and P(g) for P.V(g-2), so the tensor pipe runs S(g+1) and P.V(g) while the
//     softmax works on tile g; with P written over its own S, S(g+2) had to wait for
//     P.V(g), a chain of ~2.4 us per two tiles against ~2 us of tensor work;
//   * online softmax with one row per TMEM lane: two threads share a row (64 keys each)
//     and exchange their partial maxima; a row's reference only moves, and its O row is only
//     rescaled, when a score exceeds the reference by 2^4;
//   * K and V pages arrive by TMA (one box per page and d-half) from two producer warps;
//     two threads issue the MMAs (S and P.V), since one thread issues tcgen05.mma slower
//     than the tensor pipe retires them; persistent CTAs walk contiguous ranges of key
//     tiles cut by the plan kernel, and blocks cut across CTAs are merged by their last piece.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdio>

#include "common.cuh"
#include "device_util.cuh"
#include "tc_kernels.cuh"
#include "tc_util.cuh"

namespace pgqa {

bool make_cache_tmap(CUtensorMap* m, const pg_tensor* t, int P);
void set_tc_error(const char* msg);

namespace {

using namespace tc;

constexpr int kRows = kPrefillRows;    // 128: MMA M
constexpr int kSoftWarps = 8;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kThreads = 128 + kSoftThreads;   // + K producer, 2 MMA issuers, V producer
constexpr int kVProducerWarp = 2 + kSoftWarps;
constexpr int kPVIssuerWarp = 3 + kSoftWarps;
constexpr int kHalfKeys = kTileKeys / 2;       // keys per softmax thread
constexpr int kKStages = 2;
constexpr float kTau = 4.f;
constexpr float kSigma = 4.f;
constexpr float kMInit = -1.0e30f;

constexpr uint32_t kQHalf = kRows * 128;        // [128 rows][128 B]
constexpr uint32_t kQPart = 2 * kQHalf;         // 32 KB
constexpr uint32_t kKVHalf = kTileKeys * 128;   // [128 keys][128 B]
constexpr uint32_t kKVTile = 2 * kKVHalf;       // 32 KB
// TMEM columns: S (128), two P buffers (2 x 64: P_hi 32 and P_lo 32, four e4m3 keys per
// column; the A operand of O += P V straight from TMEM), O d-half 0 and 1 (2 x 128).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColP = 128;
constexpr uint32_t kPBufCols = 64;
constexpr uint32_t kColO = 256;
constexpr uint32_t kPCols = kTileKeys / 4;  // 32 columns per P part

constexpr uint32_t kIdescS = idesc_e4m3(128, 128, false, false);  // Q (K-major) x K (K-major)
constexpr uint32_t kIdescO = idesc_e4m3(128, 256, false, true);   // P (TMEM) x V (MN-major, N = d = 256)

template <bool kQFp8>
struct Layout {
  static constexpr int kQParts = kQFp8 ? 1 : 2;
  static constexpr int kVStages = kQFp8 ? 3 : 2;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kQParts * kQPart;
  static constexpr uint32_t kOffV = kOffK + kKStages * kKVTile;
  static constexpr uint32_t kOffMisc = kOffV + kVStages * kKVTile;
};

struct Misc {
  alignas(16) float red[2][2][kRows];   // [tile parity][key half][row] partial maxima
  alignas(16) float lsum[2][kRows];     // [key half][row] row-sum halves (epilogue)
  alignas(16) long long out_off[2][kRows];
  alignas(16) int lim[2][kRows];
  alignas(16) float merge_w[kMergeMaxSplits * kSlotRows];
  alignas(8) uint64_t k_full[kKStages], k_empty[kKStages], v_full[3], v_empty[3];
  uint64_t s_full, s_free, pv_done[2];
  uint64_t p_full[2], q_full, q_free, o_ready, o_free, drain[2];
  uint64_t never;  // no thread ever arrives (the failure-path test waits on it)
  float qscale[2];
  float amax[kSoftWarps];
  uint32_t tmem_base;
  int abort_flag;
  int vote[2][kSoftWarps];
  int merge_flag;
};

template <bool kQFp8>
constexpr size_t smem_bytes() {
  return Layout<kQFp8>::kOffMisc + sizeof(Misc) + 1024;
}

struct Item {
  int block, seq, kvh, row0, nrows, kv_end, nsplit, split, slot_base;
  int tile_begin, ntiles, kv_hi;
  int q0, qn, L;
};

__device__ __forceinline__ Item load_item(const ClassPlan& cp, const Pointers& ptr, int it) {
  const WorkItem w = cp.items[it];
  const RowBlock b = cp.blocks[w.block];
  Item r;
  r.block = w.block;
  r.seq = b.seq;
  r.kvh = b.kvh;
  r.row0 = b.row0;
  r.nrows = b.nrows;
  r.kv_end = b.kv_end;
  r.nsplit = b.nsplit;
  r.split = w.split;
  r.slot_base = b.slot_base;
  r.tile_begin = w.tile_begin;
  r.ntiles = w.tile_end - w.tile_begin;
  r.kv_hi = min(w.tile_end * kTileKeys, b.kv_end);
  r.q0 = ptr.qsl[b.seq];
  r.qn = ptr.qsl[b.seq + 1] - r.q0;
  r.L = ptr.seq_lens[b.seq];
  return r;
}

__device__ __forceinline__ float2 bf2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

}  // namespace

template <int kQM>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  Problem p, Pointers ptr, ClassPlan cp) {
  constexpr bool kQFp8 = kQM != kQSplit;       // one e4m3 Q part in shared memory
  constexpr int kQEsz = kQM == kQGiven ? 1 : 2;  // bytes of a Q element in HBM
  using LY = Layout<kQFp8>;
  constexpr int kVStages = LY::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + LY::kOffMisc);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &ms.abort_flag;
  auto bar = [&](const uint64_t& b) { return smem_u32(&b); };
  // The plan is read once the previous grid (the plan kernel) has completed. A CTA with no
  // work (an empty class, or fewer items than CTAs) leaves before any set-up.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int item_begin = cp.cta_item_begin[blockIdx.x];
  const int item_end = cp.cta_item_begin[blockIdx.x + 1];
  if (item_begin >= item_end) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(ms.k_full[s]), 1);
      mbar_init(bar(ms.k_empty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(ms.v_full[s]), 1);
      mbar_init(bar(ms.v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(ms.pv_done[b]), 1);
    }
    mbar_init(bar(ms.s_full), 1);
    mbar_init(bar(ms.s_free), kSoftThreads);
    mbar_init(bar(ms.p_full[0]), kSoftThreads);
    mbar_init(bar(ms.p_full[1]), kSoftThreads);
    mbar_init(bar(ms.q_full), kSoftThreads);
    mbar_init(bar(ms.q_free), 1);
    mbar_init(bar(ms.o_ready), 1);
    mbar_init(bar(ms.o_free), kSoftThreads);
    mbar_init(bar(ms.drain[0]), 1);
    mbar_init(bar(ms.drain[1]), 1);
    mbar_init(bar(ms.never), 1);
    ms.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ms.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  // The next kernel on the stream (the other class) may start its own checks now.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0 || warp == kVProducerWarp) {
    // ------------------------------------------------------------ TMA producers (K, V)
    const bool is_k = warp == 0;
    const CUtensorMap* tmap = is_k ? &tmap_k : &tmap_v;
    const int nst = is_k ? kKStages : kVStages;
    const uint32_t region = sbase + (is_k ? LY::kOffK : LY::kOffV);
    uint64_t* full = is_k ? ms.k_full : ms.v_full;
    uint64_t* empty = is_k ? ms.k_empty : ms.v_empty;
    if (lane == 0) tma_prefetch_desc(tmap);
    // Every row block of a sequence re-reads the same K/V pages: keep them in L2.
    const uint64_t policy = policy_evict_last();
    const int ppt = kTileKeys / p.P;
    uint32_t g = 0;
    uint32_t issued[kVStages > kKStages ? kVStages : kKStages] = {};
    bool stop = false;
    for (int it = item_begin; it < item_end && !stop; ++it) {
      const Item I = load_item(cp, ptr, it);
      const int32_t* bt_row = ptr.block_table + (size_t)I.seq * p.bt_stride;
      const int page0 = I.tile_begin * ppt;
      const int npages = (I.kv_hi + p.P - 1) / p.P - page0;
      auto fetch = [&](int w) -> int {
        const int pg = w * 32 + lane;
        int blk = -1;
        if (pg < npages) {
          blk = bt_row[page0 + pg];
          if (blk < 0 || blk >= p.NB) {
            atomicOr(ptr.err, kErrPage);
            blk = 0;
          }
        }
        return blk;
      };
      int cur = fetch(0), nxt = fetch(1);
      int cur_w = 0;
      for (int j = 0; j < I.ntiles; ++j, ++g) {
        const int first = j * ppt;
        if (first / 32 != cur_w) {
          cur = nxt;
          cur_w = first / 32;
          nxt = fetch(cur_w + 1);
        }
        const int tile_pages = min(ppt, npages - first);
        const uint32_t st = g % nst, ph = (g / nst) & 1;
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(bar(empty[st]), ph ^ 1, abort_flag, ptr.err);
          if (ok) mbar_expect_tx(bar(full[st]), (uint32_t)tile_pages * p.P * 128u * 2u);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          stop = true;
          break;
        }
        for (int pg = 0; pg < tile_pages; ++pg) {
          const int blk = __shfl_sync(0xffffffffu, cur, (first + pg) & 31);
          if (lane == 0) {
            const uint32_t row = (uint32_t)pg * p.P * 128u;
            for (int h = 0; h < 2; ++h)
              tma_load_4d(region + st * kKVTile + h * kKVHalf + row, tmap, h * 128, I.kvh, 0, blk, bar(full[st]),
                          policy);
          }
        }
        issued[st] = g / nst + 1;
      }
    }
    if (lane == 0) {
      for (int s = 0; s < nst; ++s)
        if (issued[s]) mbar_drain(bar(full[s]), (issued[s] - 1) & 1, abort_flag, ptr.err);
    }
    __syncwarp();
  } else if (warp == 1 || warp == kPVIssuerWarp) {
    // ------------------------------------------------------------ MMA issuers
    // One thread cannot issue tcgen05.mma faster than about one per 44 ns, below the tensor
    // pipe's rate, so S = Q K^T and O += P V come from two warps. S(g) waits for the softmax
    // to have loaded S(g-1); P.V(g) waits for P(g) and V(g).
    if (lane == 0) {
      const bool is_s = warp == 1;
      uint32_t g = 0;
      int ii = 0;
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it, ++ii) {
        const Item I = load_item(cp, ptr, it);
        for (int j = 0; j < I.ntiles && ok; ++j, ++g) {
          const uint32_t b = g & 1;
          if (is_s) {
            if (j == 0 && !(ok = mbar_wait(bar(ms.q_full), ii & 1, abort_flag, ptr.err))) break;
            const uint32_t st = g % kKStages;
            if (!(ok = mbar_wait(bar(ms.k_full[st]), (g / kKStages) & 1, abort_flag, ptr.err))) break;
            if (g >= 1 && !(ok = mbar_wait(bar(ms.s_free), (g - 1) & 1, abort_flag, ptr.err))) break;
            tc_fence_after();
            const uint64_t k0 = smem_desc(sbase + LY::kOffK + st * kKVTile, 16, 1024, kSw128);
#pragma unroll
            for (int part = 0; part < LY::kQParts; ++part) {
              const uint64_t q0 = smem_desc(sbase + LY::kOffQ + part * kQPart, 16, 1024, kSw128);
#pragma unroll
              for (int kb = 0; kb < 8; ++kb) {
                const uint32_t qoff = (kb >> 2) * kQHalf + (kb & 3) * 32, koff = (kb >> 2) * kKVHalf + (kb & 3) * 32;
                mma_e4m3(tmem + kColS, q0 + (qoff >> 4), k0 + (koff >> 4), kIdescS, (part | kb) ? 1u : 0u);
              }
            }
            mma_commit(bar(ms.s_full));
            mma_commit(bar(ms.k_empty[st]));
            if (j == I.ntiles - 1) mma_commit(bar(ms.q_free));
          } else {
            // the first P.V of an item overwrites O: the previous epilogue must be done
            if (j == 0 && ii >= 1 && !(ok = mbar_wait(bar(ms.o_free), (ii - 1) & 1, abort_flag, ptr.err))) break;
            // one barrier per P buffer: P(g + 2) waits for P.V(g), so the softmax is never two
            // publications ahead of this wait
            if (!(ok = mbar_wait(bar(ms.p_full[b]), (g >> 1) & 1, abort_flag, ptr.err))) break;
            const uint32_t st = g % kVStages;
            if (!(ok = mbar_wait(bar(ms.v_full[st]), (g / kVStages) & 1, abort_flag, ptr.err))) break;
            tc_fence_after();
            // V as one N = 256 MN-major operand: d-half 1 is the second 128-byte atom, 16 KB on
            const uint64_t v0 = smem_desc(sbase + LY::kOffV + st * kKVTile, kKVHalf, 1024, kSw128);
            const uint32_t p_cols = tmem + kColP + b * kPBufCols;  // P of this tile
#pragma unroll
            for (int part = 0; part < 2; ++part) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_e4m3_ts(tmem + kColO, p_cols + part * kPCols + kk * 8, v0 + ((kk * 4096) >> 4), kIdescO,
                            (j == 0 && part == 0 && kk == 0) ? 0u : 1u);
            }
            mma_commit(bar(ms.v_empty[st]));
            mma_commit(bar(ms.pv_done[b]));
            if (j == I.ntiles - 1) mma_commit(bar(ms.o_ready));
          }
        }
      }
      // Every MMA this thread issued has completed before the CTA may release TMEM.
      uint64_t& drain = is_s ? ms.drain[0] : ms.drain[1];
      mma_commit(bar(drain));
      mbar_drain(bar(drain), 0, abort_flag, ptr.err);
    }
    __syncwarp();
  } else if (warp >= 2 && warp < kVProducerWarp) {
    // ------------------------------------------------------------ softmax + epilogue
    const int sw = warp - 2;               // 0..7
    const int gi = sw * 32 + lane;         // 0..255
    const int q4 = warp & 3;               // TMEM lane quarter
    const int kh = sw >> 2;                // key half of the tile this thread owns (0/1)
    const int row = q4 * 32 + lane;        // TMEM lane = row of the block
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const int pair_bar = 1 + q4;           // named barrier of the two threads of each row
    // {descale, 1/descale} of a per-tensor cast of Q (kQCast), the same in every thread
    const float2 q_cast = kQM == kQCast ? q_cast_scales(ptr.q_amax, p.q_amax_parts, lane) : make_float2(1.f, 1.f);
    bool bad = false;
    float m_ref = kMInit, l = 0.f;
    // Failure-path test: a bounded wait on a barrier nothing arrives on runs out in every
    // softmax thread (by its own limit or by the abort flag another thread raised); they
    // then skip the items, so no Q is published, the MMA issuers give up on q_full / p_full
    // and every producer drains the copies it issued.
    const bool stalled = p.stall_test_ns && !mbar_wait(bar(ms.never), 0, abort_flag, ptr.err, p.stall_test_ns);
    if (!stalled) {

    auto q_prep = [&](const Item& I, int ii) {
      const int pi = ii & 1;
      if (ii >= 1 && !mbar_wait(bar(ms.q_free), (ii - 1) & 1, abort_flag, ptr.err)) bad = true;
      if (gi < kRows) {
        const int n = gi;
        if (n < I.nrows) {
          const RowMap m = map_row(I.row0 + n, p.G, I.kvh);
          ms.lim[pi][n] = I.L - I.qn + m.t;
          ms.out_off[pi][n] = (long long)(I.q0 + m.t) * p.o_st + (long long)m.h * p.o_sh;
        } else {
          ms.lim[pi][n] = -1;
          ms.out_off[pi][n] = 0;
        }
      }
      // 128 rows x 16 chunks of 16 elements: thread gi takes chunks gi + 256k, k < 8
      auto src_of = [&](int r, int ch) -> const uint8_t* {
        const RowMap m = map_row(I.row0 + r, p.G, I.kvh);
        return static_cast<const uint8_t*>(ptr.q) +
               ((size_t)(I.q0 + m.t) * p.q_st + (size_t)m.h * p.q_sh + ch * 16) * kQEsz;
      };
      auto dst_of = [&](int part, int r, int ch) -> uint8_t* {
        const int h = ch >> 3, c = ch & 7;
        return smem + LY::kOffQ + part * kQPart + h * kQHalf + r * 128 + ((c ^ (r & 7)) << 4);
      };
      if (kQM == kQCast) {
#pragma unroll
        for (int k0 = 0; k0 < 8; k0 += 4) {
          uint4 v[4][2];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = gi + (k0 + k) * kSoftThreads, r = c >> 4, ch = c & 15;
            if (r < I.nrows) {
              const uint4* s = reinterpret_cast<const uint4*>(src_of(r, ch));
              v[k][0] = s[0];
              v[k][1] = s[1];
            } else {
              v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = gi + (k0 + k) * kSoftThreads, r = c >> 4, ch = c & 15;
            *reinterpret_cast<uint4*>(dst_of(0, r, ch)) = bf16x16_to_e4m3(v[k][0], v[k][1], q_cast.y);
          }
        }
        if (gi == 0) ms.qscale[pi] = q_cast.x;
      } else if (kQM == kQGiven) {
#pragma unroll
        for (int k0 = 0; k0 < 8; k0 += 4) {
          uint4 v[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = gi + (k0 + k) * kSoftThreads, r = c >> 4, ch = c & 15;
            v[k] = r < I.nrows ? *reinterpret_cast<const uint4*>(src_of(r, ch)) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = gi + (k0 + k) * kSoftThreads, r = c >> 4, ch = c & 15;
            *reinterpret_cast<uint4*>(dst_of(0, r, ch)) = v[k];
          }
        }
        if (gi == 0) ms.qscale[pi] = 1.f;
      } else {
        float amax = 0.f;
        for (int k = 0; k < 8; ++k) {
          const int c = gi + k * kSoftThreads, r = c >> 4, ch = c & 15;
          if (r < I.nrows) {
            const uint4* s = reinterpret_cast<const uint4*>(src_of(r, ch));
            const uint4 a = s[0], b = s[1];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 f = bf2(w[i]);
              amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
        }
        amax = warp_max(amax);
        if (lane == 0) ms.amax[sw] = amax;
        named_barrier(9, kSoftThreads);
        amax = 0.f;
#pragma unroll
        for (int w = 0; w < kSoftWarps; ++w) amax = fmaxf(amax, ms.amax[w]);
        named_barrier(9, kSoftThreads);
        int sig = 0;
        if (amax > 0.f && isfinite(amax)) sig = 7 - (int)((__float_as_uint(amax) >> 23) & 0xff) + 127;
        sig = max(-100, min(100, sig));
        const float scale = ldexpf(1.f, sig);
        for (int k = 0; k < 8; ++k) {
          const int c = gi + k * kSoftThreads, r = c >> 4, ch = c & 15;
          uint4 hv = make_uint4(0, 0, 0, 0), lv = make_uint4(0, 0, 0, 0);
          if (r < I.nrows) {
            const uint4* s = reinterpret_cast<const uint4*>(src_of(r, ch));
            const uint4 a = s[0], b = s[1];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f0 = bf2(w[2 * i]), f1 = bf2(w[2 * i + 1]);
              split4(f0.x * scale, f0.y * scale, f1.x * scale, f1.y * scale, hw[i], lw[i]);
            }
            hv = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            lv = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
          *reinterpret_cast<uint4*>(dst_of(0, r, ch)) = hv;
          *reinterpret_cast<uint4*>(dst_of(1, r, ch)) = lv;
        }
        if (gi == 0) ms.qscale[pi] = ldexpf(1.f, -sig);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(ms.q_full));
    };

    int ii = 0;
    uint32_t g = 0;
    if (item_end > item_begin) q_prep(load_item(cp, ptr, item_begin), 0);
    for (int it = item_begin; it < item_end; ++it, ++ii) {
      const Item I = load_item(cp, ptr, it);
      const int pi = ii & 1;
      named_barrier(9, kSoftThreads);  // q_prep's shared writes are visible
      const float c = p.score_scale_log2 * ms.qscale[pi];
      const int lim = ms.lim[pi][row];
      const int min_lim = I.L - I.qn + map_row(I.row0, p.G, I.kvh).t;
      m_ref = kMInit;
      l = 0.f;
      const int kv_hi = I.kv_hi, tile_begin = I.tile_begin, ntiles = I.ntiles;
      const int hi_key = min(kv_hi - 1, lim);  // keys <= hi_key are visible to this row
      const bool c_pos = c >= 0.f;
      // A failed wait (timeout or abort) does not leave the loop: every later wait then
      // fails fast, so all softmax warps still pass the same barriers and finish.
      for (int j = 0; j < ntiles; ++j, ++g) {
        const int b = g & 1;
        const int key0 = (tile_begin + j) * kTileKeys;
        const int kbase = key0 + kh * kHalfKeys;
        float t[kHalfKeys];
        if (!mbar_wait(bar(ms.s_full), g & 1, abort_flag, ptr.err)) bad = true;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kHalfKeys; k += 16) {
          float v[16];
          tmem_ld16(tmem + lane_addr + kColS + kh * kHalfKeys + k, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) t[k + i] = v[i];
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(ms.s_free));  // S(g+1) may overwrite S now
        // masked tiles hold scaled scores; unmasked tiles keep raw scores and take the
        // scale in the exponent's FFMA
        const bool need_mask = (key0 + kTileKeys > kv_hi) || (key0 + kTileKeys - 1 > min_lim);
        float mx;
        if (need_mask) {
#pragma unroll
          for (int i = 0; i < kHalfKeys; ++i) t[i] = (kbase + i <= hi_key) ? t[i] * c : -INFINITY;
          mx = extreme_of<true>(t);
        } else {
          // max of s c = c max(s) for c >= 0, c min(s) for c < 0
          mx = (c_pos ? extreme_of<true>(t) : extreme_of<false>(t)) * c;
        }
        // the row's maximum over both key halves (partner: same lane, the other warp)
        ms.red[g & 1][kh][row] = mx;
        named_barrier(pair_bar, 64);
        const float mt = fmaxf(mx, ms.red[g & 1][kh ^ 1][row]);
        float alpha = 1.f;
        const bool rescale = mt > m_ref + kTau;
        if (rescale) {
          alpha = ex2(m_ref - mt);
          m_ref = mt;
          l *= alpha;
        }
        // P = 2^(s c - m + sigma) in f16, split into e4m3 hi + lo, 4 keys per word
        uint32_t ph[kHalfKeys / 4], pl[kHalfKeys / 4];
        const float off = m_ref - kSigma;
        const float sc = need_mask ? 1.f : c;
        __half2 acc[4] = {__float2half2_rn(0.f), __float2half2_rn(0.f), __float2half2_rn(0.f),
                          __float2half2_rn(0.f)};
#pragma unroll
        for (int i = 0; i < kHalfKeys; i += 4) {
          __half2 s01, s23;
          p_split4_f16(fmaf(t[i], sc, -off), fmaf(t[i + 1], sc, -off), fmaf(t[i + 2], sc, -off),
                       fmaf(t[i + 3], sc, -off), ph[i / 4], pl[i / 4], s01, s23);
          acc[(i / 4) & 3] = __hadd2(acc[(i / 4) & 3], __hadd2(s01, s23));
        }
        const float2 ls = __half22float2(__hadd2(__hadd2(acc[0], acc[1]), __hadd2(acc[2], acc[3])));
        l += ls.x + ls.y;
        // tcgen05.ld/st are warp-collective: a warp rescales if any of its rows must,
        // lanes whose row keeps its reference multiply by 1. O may only be touched once the
        // previous tile's P.V has completed; otherwise that wait comes after publishing P
        // (each tile waits exactly once, so the barrier's parity stays unambiguous).
        const bool warp_rescale = __any_sync(0xffffffffu, rescale && j > 0);
        if (warp_rescale) {
          if (g >= 1 && !mbar_wait(bar(ms.pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort_flag, ptr.err)) bad = true;
          tc_fence_after();
          if (!(rescale && j > 0)) alpha = 1.f;
          // this thread's half of its O row: d-half kh
#pragma unroll 1
          for (int k = 0; k < 128; k += 16) {
            float v[16];
            const uint32_t a = tmem + lane_addr + kColO + kh * 128 + k;
            tmem_ld16(a, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= alpha;
            tmem_st16(a, v);
          }
          tmem_wait_st();
        }
        // P.V(g-2) has read P buffer b (and every earlier P.V has completed, so V(g - 2) and
        // before have landed). Each tile waits on pv_done[b] once, in order, and P.V(g) needs
        // P(g): the barrier is never a phase ahead of or two phases behind the one waited for.
        if (g >= 2 && !mbar_wait(bar(ms.pv_done[b]), ((g >> 1) - 1) & 1, abort_flag, ptr.err)) bad = true;
        tc_fence_after();
        if (key0 + kTileKeys > kv_hi) {
          // keys past the piece's end: their V rows (stale or NaN slots) become zeros.
          // thread (kh, row) zeroes d-half kh of key `row`. This wait skips the phases of
          // tiles without a tail, so it must not lag two phases: V(g - kVStages) has landed
          // (P.V(g - 2) above has completed), and V(g + kVStages) cannot land before P.V(g).
          const uint32_t st = g % kVStages;
          if (!mbar_wait(bar(ms.v_full[st]), (g / kVStages) & 1, abort_flag, ptr.err)) bad = true;
          if (key0 + row >= kv_hi) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            uint4* dst = reinterpret_cast<uint4*>(smem + LY::kOffV + st * kKVTile + kh * kKVHalf + row * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = z;
          }
        }
        // P into P buffer b: row `row`, keys 64*kh .. 64*kh+63 -> columns 16*kh .. 16*kh+15 of
        // P_hi (buffer columns 0..31) and P_lo (32..63)
        tmem_st16u(tmem + lane_addr + kColP + b * kPBufCols + kh * 16, ph);
        tmem_st16u(tmem + lane_addr + kColP + b * kPBufCols + kPCols + kh * 16, pl);
        tmem_wait_st();
        fence_proxy_async_smem();  // zeroed V rows, if any
        tc_fence_before();
        mbar_arrive(bar(ms.p_full[b]));
      }
      if (it + 1 < item_end) q_prep(load_item(cp, ptr, it + 1), ii + 1);

      // ---------------------------------------------------------- epilogue
      if (!mbar_wait(bar(ms.o_ready), ii & 1, abort_flag, ptr.err)) bad = true;
      tc_fence_after();
      ms.lsum[kh][row] = l;
      named_barrier(pair_bar, 64);
      const float lr = l + ms.lsum[kh ^ 1][row];
      const bool split = I.nsplit > 1;
      const int slot = I.slot_base + I.split;
      const bool valid = row < I.nrows;
      // a split piece's partial stays in code units (v_descale is applied by the merge)
      const float inv = lr > 0.f ? (split ? 1.f : p.out_scale) / lr : 0.f;
#pragma unroll 1
      for (int k = 0; k < 128; k += 16) {
        float v[16];
        tmem_ld16(tmem + lane_addr + kColO + kh * 128 + k, v);
        tmem_wait_ld();
        if (valid) {
          const int d = kh * 128 + k;
          if (split) {
            uint4* dst = reinterpret_cast<uint4*>(slot_o(cp, slot) + (size_t)row * kHeadDim + d);
#pragma unroll
            for (int i = 0; i < 2; ++i)
              dst[i] = make_uint4(pack_f16x2(v[8 * i] * inv, v[8 * i + 1] * inv),
                                  pack_f16x2(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                  pack_f16x2(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                  pack_f16x2(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(ptr.out) + ms.out_off[pi][row] + d);
#pragma unroll
            for (int i = 0; i < 2; ++i)
              dst[i] = make_uint4(pack_bf16x2(v[8 * i] * inv, v[8 * i + 1] * inv),
                                  pack_bf16x2(v[8 * i + 2] * inv, v[8 * i + 3] * inv),
                                  pack_bf16x2(v[8 * i + 4] * inv, v[8 * i + 5] * inv),
                                  pack_bf16x2(v[8 * i + 6] * inv, v[8 * i + 7] * inv));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(ms.o_free));
      if (split) {
        if (kh == 0 && valid) slot_lse(cp, slot)[row] = lr > 0.f ? m_ref - kSigma + log2f(lr) : -INFINITY;
        __threadfence();
        RowBlock rb;
        rb.seq = I.seq;
        rb.kvh = I.kvh;
        rb.row0 = I.row0;
        rb.nrows = I.nrows;
        rb.nsplit = I.nsplit;
        rb.slot_base = I.slot_base;
        finish_split_block(p, ptr, cp, I.block, rb, gi, kSoftThreads, 10, &ms.merge_flag, ms.merge_w);
      }
    }
    }  // !stalled
    (void)bad;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int launch_prefill_tc(const Problem& p, const Pointers& ptr, const ClassPlan& cp, const pg_tensor* k,
                      const pg_tensor* v, int sms, cudaStream_t stream, bool dependent) {
  (void)sms;
  if (!p.kv_is_fp8) return 0;
  CUtensorMap tk, tv;
  if (!make_cache_tmap(&tk, k, p.P) || !make_cache_tmap(&tv, v, p.P)) return -1;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e;
  const int mode = p.q_cast ? kQCast : p.q_is_fp8 ? kQGiven : kQSplit;
  auto kern = mode == kQCast ? prefill_tc_kernel<kQCast> : mode == kQGiven ? prefill_tc_kernel<kQGiven> : prefill_tc_kernel<kQSplit>;
  const size_t bytes = mode != kQSplit ? smem_bytes<true>() : smem_bytes<false>();
  const int which = 1 << mode;
  if (dev >= 0 && dev < 64 && !(attr_done[dev] & which)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) {
      char buf[160];
      snprintf(buf, sizeof buf, "cudaFuncSetAttribute(prefill): %s", cudaGetErrorString(e));
      set_tc_error(buf);
      return -1;
    }
    attr_done[dev] |= which;
  }
  e = launch_pdl(dependent, kern, cp.num_ctas, kThreads, bytes, stream, tk, tv, p, ptr, cp);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    char buf[160];
    snprintf(buf, sizeof buf, "prefill kernel launch: %s", cudaGetErrorString(e));
    set_tc_error(buf);
    return -1;
  }
  return 1;
}

}  // namespace pgqa
