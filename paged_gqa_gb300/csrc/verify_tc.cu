// verify_tc.cu -- tcgen05 (TMEM, TMA) kernel for verify blocks: q_len*G <= 64 query rows of
// one (sequence, kv head) against an FP8 e4m3 paged KV cache.
//
// What the pages ask of this path ("Optimize Qwen3.5 MTP unified attention on gfx950",
// Motivation and Modifications): all q_len x G query rows of a kv head share one load of
// each KV page (BLOCK_M covers tokens x heads), split-KV segments keep every SM busy, and
// the FP8 descales are per-tensor scalars. The launch shape on that page (BLOCK_M 32,
// TILE 32, 8-64 segments on gfx950) is prior art; this kernel is laid out for sm_103a:
//
//   * swap-AB: the 128 keys of a tile are the MMA's M dimension and the (padded) 64 query
//     rows are N, so a 64-row verify block fills the 128-lane tensor core. S^T = K Q^T and
//     O^T += V^T P^T, both tcgen05.mma kind::f8f6f4 with fp32 accumulators in TMEM;
//   * FP8 K and V go from HBM to shared memory by TMA (one 2-D box per page and d-half,
//     addressed through the block table) and into the MMA untouched; the dequant scales are
//     folded into the score scale (k_descale) and the output scale (v_descale);
//   * bf16 Q is split once per block into e4m3 hi + lo parts (q*2^s = hi + lo, exact to
//     ~2^-16 of the block's max), so S = K.hi + K.lo costs two FP8 MMAs and no K conversion;
//   * P is split the same way (p = hi + lo in e4m3, ~9 significant bits, about bf16's
//     precision); a single e4m3 P would miss the 5e-3 relative-L2 bar;
//   * online softmax over keys: keys live on TMEM lanes, so the row max is a cross-lane
//     reduction (redux.sync + shared memory). It is only taken when some score exceeds the
//     running reference by 2^4 (the reference then moves to the exact max and O^T and the
//     row sums are rescaled); otherwise P = 2^(s - m + 4) <= 256 fits e4m3 directly;
//   * persistent CTAs (one per SM) walk a contiguous range of key tiles cut by the plan
//     kernel; a block cut across CTAs is finished by the last piece with a log-sum-exp merge.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer (+ TMEM owner),
// warps 2-5 = softmax and epilogue (thread i <-> TMEM lane i <-> key i of the tile).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "device_util.cuh"
#include "tc_kernels.cuh"
#include "tc_util.cuh"

namespace pgqa {

namespace {

using namespace tc;

constexpr int kVN = 64;            // MMA N: query rows, padded
constexpr int kVThreads = 192;
constexpr int kStages = 2;         // K/V shared-memory stages
constexpr float kTau = 4.f;        // rescale when a score exceeds the reference by 2^kTau
constexpr float kSigma = 4.f;      // P is stored scaled by 2^kSigma (max 2^(kTau+kSigma) = 256)
constexpr float kMInit = -1.0e30f; // reference of a row before its first key

constexpr uint32_t kQHalf = kVN * 128;          // [64 rows][128 B] e4m3, one d-half
constexpr uint32_t kQPart = 2 * kQHalf;
constexpr uint32_t kKVHalf = kTileKeys * 128;   // [128 keys][128 B]
constexpr uint32_t kKVTile = 2 * kKVHalf;
constexpr uint32_t kPPart = kTileKeys * kVN;    // [128 keys][64 B]
constexpr uint32_t kOffQhi = 0;
constexpr uint32_t kOffQlo = kOffQhi + kQPart;
constexpr uint32_t kOffK = kOffQlo + kQPart;
constexpr uint32_t kOffV = kOffK + kStages * kKVTile;
constexpr uint32_t kOffPhi = kOffV + kStages * kKVTile;
constexpr uint32_t kOffPlo = kOffPhi + kPPart;
constexpr uint32_t kOffMisc = kOffPlo + kPPart;

// TMEM columns: S^T double buffer, then O^T (d-half 0, d-half 1).
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;

constexpr uint32_t kIdescS = idesc_e4m3(128, kVN, false, false);  // K (K-major) x Q^T (K-major)
constexpr uint32_t kIdescO = idesc_e4m3(128, kVN, true, true);    // V^T (MN-major) x P^T (MN-major)

struct Misc {
  // arrays read with 16-byte vector loads first
  alignas(16) float m[2][kVN];
  alignas(16) float red[4][kVN];
  alignas(16) float alpha[kVN];
  alignas(16) float lrow[kVN];
  alignas(16) int lim[2][kVN];
  alignas(16) long long out_off[2][kVN];
  alignas(8) uint64_t k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, p_free, q_full, q_free, o_ready, o_free, drain;
  float qscale[2];
  uint32_t tmem_base;
  int abort_flag;
  int vote[2][4];
  int merge_flag;
};
static_assert(offsetof(Misc, m) % 16 == 0 && offsetof(Misc, k_full) % 8 == 0, "Misc alignment");
constexpr size_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;

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

// bf16 pair -> floats
__device__ __forceinline__ float2 bf2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// y -> (hi, lo) e4m3 bytes of 4 values packed in two words.
__device__ __forceinline__ void split4(float a, float b, float c, float d, uint32_t& hi, uint32_t& lo) {
  const uint32_t h01 = e4m3x2(a, b), h23 = e4m3x2(c, d);
  const float2 f01 = e4m3x2_to_f2(h01), f23 = e4m3x2_to_f2(h23);
  const uint32_t l01 = e4m3x2(a - f01.x, b - f01.y), l23 = e4m3x2(c - f23.x, d - f23.y);
  hi = h01 | (h23 << 16);
  lo = l01 | (l23 << 16);
}

}  // namespace

template <bool kQFp8>
__global__ void __launch_bounds__(kVThreads, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 Problem p, Pointers ptr, ClassPlan cp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item_begin = cp.cta_item_begin[blockIdx.x];
  const int item_end = cp.cta_item_begin[blockIdx.x + 1];
  volatile int* abort_flag = &ms.abort_flag;

  auto bar = [&](const uint64_t& b) { return smem_u32(&b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(ms.k_full[s]), 1);
      mbar_init(bar(ms.v_full[s]), 1);
      mbar_init(bar(ms.k_empty[s]), 1);
      mbar_init(bar(ms.v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(ms.s_full[b]), 1);
      mbar_init(bar(ms.s_free[b]), 128);
    }
    mbar_init(bar(ms.p_full), 128);
    mbar_init(bar(ms.p_free), 1);
    mbar_init(bar(ms.q_full), 128);
    mbar_init(bar(ms.q_free), 1);
    mbar_init(bar(ms.o_ready), 1);
    mbar_init(bar(ms.o_free), 128);
    mbar_init(bar(ms.drain), 1);
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmap_k);
      tma_prefetch_desc(&tmap_v);
    }
    const uint64_t policy = policy_evict_first();
    const int ppt = kTileKeys / p.P;  // pages per tile (1..8)
    uint32_t g = 0;
    uint32_t issued_k[kStages] = {}, issued_v[kStages] = {};
    bool stop = false;
    for (int it = item_begin; it < item_end && !stop; ++it) {
      const Item I = load_item(cp, ptr, it);
      const int32_t* bt_row = ptr.block_table + (size_t)I.seq * p.bt_stride;
      auto fetch = [&](int j) -> int {
        const int key0 = (I.tile_begin + j) * kTileKeys + lane * p.P;
        int blk = -1;
        if (lane < ppt && key0 < I.kv_hi) {
          blk = bt_row[key0 / p.P];
          if (blk < 0 || blk >= p.NB) {
            atomicOr(ptr.err, kErrPage);
            blk = 0;
          }
        }
        return blk;
      };
      int cur = fetch(0);
      for (int j = 0; j < I.ntiles; ++j, ++g) {
        const int nxt = (j + 1 < I.ntiles) ? fetch(j + 1) : -1;
        const uint32_t st = g % kStages, ph = (g / kStages) & 1;
        const int npages = __popc(__ballot_sync(0xffffffffu, cur >= 0));
        int ok = 1;
        if (lane == 0) {
          const uint32_t bytes = (uint32_t)npages * p.P * 128u * 2u;
          ok = mbar_wait(bar(ms.k_empty[st]), ph ^ 1, abort_flag, ptr.err);
          if (ok) mbar_expect_tx(bar(ms.k_full[st]), bytes);
          if (ok) ok = mbar_wait(bar(ms.v_empty[st]), ph ^ 1, abort_flag, ptr.err);
          if (ok) mbar_expect_tx(bar(ms.v_full[st]), bytes);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          stop = true;
          break;
        }
        for (int pg = 0; pg < npages; ++pg) {
          const int blk = __shfl_sync(0xffffffffu, cur, pg);
          if (lane == 0) {
            const uint32_t row = (uint32_t)pg * p.P * 128u;
            for (int h = 0; h < 2; ++h) {
              tma_load_4d(sbase + kOffK + st * kKVTile + h * kKVHalf + row, &tmap_k, h * 128, I.kvh, 0, blk,
                          bar(ms.k_full[st]), policy);
              tma_load_4d(sbase + kOffV + st * kKVTile + h * kKVHalf + row, &tmap_v, h * 128, I.kvh, 0, blk,
                          bar(ms.v_full[st]), policy);
            }
          }
        }
        issued_k[st] = issued_v[st] = g / kStages + 1;
        cur = nxt;
      }
    }
    // Every issued copy has landed before the CTA may exit.
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        if (issued_k[s]) mbar_wait(bar(ms.k_full[s]), (issued_k[s] - 1) & 1, abort_flag, ptr.err);
        if (issued_v[s]) mbar_wait(bar(ms.v_full[s]), (issued_v[s] - 1) & 1, abort_flag, ptr.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t g = 0;
      int ii = 0;
      struct Pending {
        uint32_t g;
        int first, last, item;
      } pend = {0, 0, 0, -1};
      bool ok = true;
      auto issue_pv = [&](const Pending& t) -> bool {
        if (t.first && t.item >= 1 && !mbar_wait(bar(ms.o_free), (t.item - 1) & 1, abort_flag, ptr.err)) return false;
        if (!mbar_wait(bar(ms.p_full), t.g & 1, abort_flag, ptr.err)) return false;
        const uint32_t st = t.g % kStages;
        if (!mbar_wait(bar(ms.v_full[st]), (t.g / kStages) & 1, abort_flag, ptr.err)) return false;
        tc_fence_after();
        for (int h = 0; h < 2; ++h) {
          for (int part = 0; part < 2; ++part) {
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = smem_desc(sbase + kOffV + st * kKVTile + h * kKVHalf + kk * 4096, 1024, 1024, kSw128);
              const uint64_t b = smem_desc(sbase + (part ? kOffPlo : kOffPhi) + kk * 2048, 512, 512, kSw64);
              mma_e4m3(tmem + kColO + h * kVN, a, b, kIdescO, (t.first && part == 0 && kk == 0) ? 0u : 1u);
            }
          }
        }
        mma_commit(bar(ms.v_empty[st]));
        mma_commit(bar(ms.p_free));
        if (t.last) mma_commit(bar(ms.o_ready));
        return true;
      };
      for (int it = item_begin; it < item_end && ok; ++it, ++ii) {
        const Item I = load_item(cp, ptr, it);
        for (int j = 0; j < I.ntiles && ok; ++j, ++g) {
          if (j == 0 && !(ok = mbar_wait(bar(ms.q_full), ii & 1, abort_flag, ptr.err))) break;
          const uint32_t st = g % kStages, b = g & 1;
          if (!(ok = mbar_wait(bar(ms.k_full[st]), (g / kStages) & 1, abort_flag, ptr.err))) break;
          if (g >= 2 && !(ok = mbar_wait(bar(ms.s_free[b]), ((g >> 1) - 1) & 1, abort_flag, ptr.err))) break;
          tc_fence_after();
          const int parts = kQFp8 ? 1 : 2;
          for (int part = 0; part < parts; ++part) {
            for (int kb = 0; kb < 8; ++kb) {
              const int h = kb >> 2, kk = kb & 3;
              const uint64_t a = smem_desc(sbase + kOffK + st * kKVTile + h * kKVHalf + kk * 32, 16, 1024, kSw128);
              const uint64_t bq = smem_desc(sbase + (part ? kOffQlo : kOffQhi) + h * kQHalf + kk * 32, 16, 1024, kSw128);
              mma_e4m3(tmem + kColS + b * kVN, a, bq, kIdescS, (part | kb) ? 1u : 0u);
            }
          }
          mma_commit(bar(ms.s_full[b]));
          mma_commit(bar(ms.k_empty[st]));
          if (j == I.ntiles - 1) mma_commit(bar(ms.q_free));
          if (pend.item >= 0 && !(ok = issue_pv(pend))) break;
          pend = {g, j == 0, j == I.ntiles - 1, ii};
        }
      }
      if (ok && pend.item >= 0) issue_pv(pend);
      // Wait for every MMA issued by this thread before the CTA may release TMEM.
      mma_commit(bar(ms.drain));
      mbar_wait(bar(ms.drain), 0, abort_flag, ptr.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int q4 = warp & 3;                 // TMEM lane quarter
    const int ti = q4 * 32 + lane;           // TMEM lane = key in tile = d in half
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const size_t qesz = kQFp8 ? 1 : 2;
    float l[kVN];
#pragma unroll
    for (int n = 0; n < kVN; ++n) l[n] = 0.f;
    bool bad = false;

    auto q_prep = [&](const Item& I, int ii) {
      const int pi = ii & 1;
      if (ii >= 1 && !mbar_wait(bar(ms.q_free), (ii - 1) & 1, abort_flag, ptr.err)) bad = true;
      if (ti < kVN) {
        const int n = ti;
        if (n < I.nrows) {
          const RowMap m = map_row(I.row0 + n, p.G, I.kvh);
          ms.lim[pi][n] = I.L - I.qn + m.t;
          ms.out_off[pi][n] = (long long)(I.q0 + m.t) * p.o_st + (long long)m.h * p.o_sh;
        } else {
          ms.lim[pi][n] = -1;
          ms.out_off[pi][n] = 0;
        }
        // padding rows: a finite reference, so their (discarded) scores never vote
        ms.m[pi][n] = n < I.nrows ? kMInit : 0.f;
      }
      // rows x 16 chunks of 16 elements
      auto src_of = [&](int r, int ch) -> const uint8_t* {
        const RowMap m = map_row(I.row0 + r, p.G, I.kvh);
        return static_cast<const uint8_t*>(ptr.q) +
               ((size_t)(I.q0 + m.t) * p.q_st + (size_t)m.h * p.q_sh + ch * 16) * qesz;
      };
      auto dst_of = [&](uint32_t part_off, int r, int ch) -> uint8_t* {
        const int h = ch >> 3, c = ch & 7;
        return smem + part_off + h * kQHalf + r * 128 + ((c ^ (r & 7)) << 4);
      };
      if (kQFp8) {
        for (int c = ti; c < kVN * 16; c += 128) {
          const int r = c >> 4, ch = c & 15;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (r < I.nrows) v = *reinterpret_cast<const uint4*>(src_of(r, ch));
          *reinterpret_cast<uint4*>(dst_of(kOffQhi, r, ch)) = v;
        }
        if (ti == 0) ms.qscale[pi] = 1.f;
      } else {
        float amax = 0.f;
        for (int c = ti; c < kVN * 16; c += 128) {
          const int r = c >> 4, ch = c & 15;
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
        if (lane == 0) ms.red[q4][0] = amax;
        named_barrier(1, 128);
        amax = fmaxf(fmaxf(ms.red[0][0], ms.red[1][0]), fmaxf(ms.red[2][0], ms.red[3][0]));
        named_barrier(1, 128);
        // 2^sig * amax in [128, 256): exponent arithmetic on the bits
        int sig = 0;
        if (amax > 0.f && isfinite(amax)) sig = 7 - (int)((__float_as_uint(amax) >> 23) & 0xff) + 127;
        sig = max(-100, min(100, sig));
        const float scale = ldexpf(1.f, sig);
        for (int c = ti; c < kVN * 16; c += 128) {
          const int r = c >> 4, ch = c & 15;
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
          *reinterpret_cast<uint4*>(dst_of(kOffQhi, r, ch)) = hv;
          *reinterpret_cast<uint4*>(dst_of(kOffQlo, r, ch)) = lv;
        }
        if (ti == 0) ms.qscale[pi] = ldexpf(1.f, -sig);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(ms.q_full));
    };

    int ii = 0;
    uint32_t g = 0;
    const int n_items = item_end - item_begin;
    if (n_items > 0) q_prep(load_item(cp, ptr, item_begin), 0);
    for (int it = item_begin; it < item_end; ++it, ++ii) {
      const Item I = load_item(cp, ptr, it);
      const int pi = ii & 1;
      named_barrier(1, 128);  // q_prep's shared writes (lim, m, qscale) are visible
      const float c = p.score_scale_log2 * ms.qscale[pi];
      int min_lim = 0x7fffffff;
      {
        const RowMap m0 = map_row(I.row0, p.G, I.kvh);
        min_lim = I.L - I.qn + m0.t;
      }
      bool aborted = false;
      for (int j = 0; j < I.ntiles; ++j, ++g) {
        const int b = g & 1;
        const int key0 = (I.tile_begin + j) * kTileKeys;
        const int key = key0 + ti;
        float t[kVN];
        if (!mbar_wait(bar(ms.s_full[b]), (g >> 1) & 1, abort_flag, ptr.err)) bad = true;
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < kVN; c0 += 16) {
          float v[16];
          tmem_ld16(tmem + lane_addr + kColS + b * kVN + c0, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) t[c0 + i] = v[i];
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(ms.s_free[b]));
        const bool need_mask = (key0 + kTileKeys > I.kv_hi) || (key0 + kTileKeys - 1 > min_lim);
        if (need_mask) {
          const bool kin = key < I.kv_hi;
#pragma unroll
          for (int n = 0; n < kVN; ++n) {
            const bool vis = kin && key <= ms.lim[pi][n];
            t[n] = vis ? t[n] * c : -INFINITY;
          }
        } else {
#pragma unroll
          for (int n = 0; n < kVN; ++n) t[n] = t[n] * c;
        }
        // vote: does any score exceed its row reference by more than 2^kTau?
        bool mine = false;
#pragma unroll
        for (int n = 0; n < kVN; n += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(&ms.m[pi][n]);
          mine |= (t[n] - m4.x > kTau) | (t[n + 1] - m4.y > kTau) | (t[n + 2] - m4.z > kTau) |
                  (t[n + 3] - m4.w > kTau);
        }
        const int wv = (__any_sync(0xffffffffu, mine) ? 1 : 0) | ((bad || *abort_flag) ? 2 : 0);
        if (lane == 0) ms.vote[g & 1][q4] = wv;
        named_barrier(1, 128);
        const int votes = ms.vote[g & 1][0] | ms.vote[g & 1][1] | ms.vote[g & 1][2] | ms.vote[g & 1][3];
        if (votes & 2) {
          aborted = true;
          break;
        }
        const bool rescale = votes & 1;
        if (rescale) {
#pragma unroll
          for (int n = 0; n < kVN; ++n) {
            const float r = warp_max(t[n]);
            if (lane == (n & 31)) ms.red[q4][n] = r;
          }
          named_barrier(1, 128);
          if (ti < kVN) {
            const int n = ti;
            const float mt = fmaxf(fmaxf(ms.red[0][n], ms.red[1][n]), fmaxf(ms.red[2][n], ms.red[3][n]));
            const float mo = ms.m[pi][n];
            const float mn = fmaxf(mo, mt);
            ms.alpha[n] = ex2(mo - mn);
            ms.m[pi][n] = mn;
          }
          named_barrier(1, 128);
#pragma unroll
          for (int n = 0; n < kVN; ++n) l[n] *= ms.alpha[n];
        }
        // P = 2^(t - m + sigma), split into e4m3 hi + lo, 4 rows per word
        uint32_t ph[kVN / 4], pl[kVN / 4];
#pragma unroll
        for (int n = 0; n < kVN; n += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(&ms.m[pi][n]);
          const float p0 = ex2(t[n] - m4.x + kSigma), p1 = ex2(t[n + 1] - m4.y + kSigma);
          const float p2 = ex2(t[n + 2] - m4.z + kSigma), p3 = ex2(t[n + 3] - m4.w + kSigma);
          l[n] += p0;
          l[n + 1] += p1;
          l[n + 2] += p2;
          l[n + 3] += p3;
          split4(p0, p1, p2, p3, ph[n / 4], pl[n / 4]);
        }
        // P buffer and O^T are free once the previous tile's P.V has completed
        if (g >= 1 && !mbar_wait(bar(ms.p_free), (g - 1) & 1, abort_flag, ptr.err)) bad = true;
        tc_fence_after();
        if (rescale && j > 0) {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
#pragma unroll 1
            for (int c0 = 0; c0 < kVN; c0 += 16) {
              float v[16];
              const uint32_t a = tmem + lane_addr + kColO + h * kVN + c0;
              tmem_ld16(a, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] *= ms.alpha[c0 + i];
              tmem_st16(a, v);
            }
          }
          tmem_wait_st();
        }
        if (key0 + kTileKeys > I.kv_hi) {
          // keys past the piece's end: their V rows (stale or NaN slots) become zeros
          const uint32_t st = g % kStages;
          if (!mbar_wait(bar(ms.v_full[st]), (g / kStages) & 1, abort_flag, ptr.err)) bad = true;
          if (key >= I.kv_hi) {
            uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint4* row = reinterpret_cast<uint4*>(smem + kOffV + st * kKVTile + h * kKVHalf + ti * 128);
#pragma unroll
              for (int i = 0; i < 8; ++i) row[i] = z;
            }
          }
        }
        // store P^T rows: key ti, 64 bytes per part, 64-byte swizzle
        {
          const int sw = (ti >> 1) & 3;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const uint32_t off = ti * 64 + ((cc ^ sw) << 4);
            *reinterpret_cast<uint4*>(smem + kOffPhi + off) = make_uint4(ph[4 * cc], ph[4 * cc + 1], ph[4 * cc + 2], ph[4 * cc + 3]);
            *reinterpret_cast<uint4*>(smem + kOffPlo + off) = make_uint4(pl[4 * cc], pl[4 * cc + 1], pl[4 * cc + 2], pl[4 * cc + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(ms.p_full));
      }
      if (aborted) break;
      // Q of the next item while this item's last P.V runs
      if (it + 1 < item_end) q_prep(load_item(cp, ptr, it + 1), ii + 1);

      // ---------------------------------------------------------- epilogue
      if (!mbar_wait(bar(ms.o_ready), ii & 1, abort_flag, ptr.err)) bad = true;
      tc_fence_after();
      // row sums: reduce l over the 128 key lanes (warp reduce-scatter, then across warps)
      {
        float v[kVN];
#pragma unroll
        for (int n = 0; n < kVN; ++n) v[n] = l[n];
#pragma unroll
        for (int w = 32, o = 16; o >= 1; w >>= 1, o >>= 1) {
          const bool up = lane & o;
#pragma unroll
          for (int i = 0; i < w; ++i) {
            const float send = up ? v[i] : v[i + w];
            const float keep = up ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        // lane now holds rows 2*lane and 2*lane+1
        ms.red[q4][2 * lane] = v[0];
        ms.red[q4][2 * lane + 1] = v[1];
      }
      named_barrier(1, 128);
      if (ti < kVN) {
        const int n = ti;
        ms.lrow[n] = ms.red[0][n] + ms.red[1][n] + ms.red[2][n] + ms.red[3][n];
      }
      named_barrier(1, 128);
      const bool split = I.nsplit > 1;
      const int slot = I.slot_base + I.split;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
#pragma unroll 1
        for (int c0 = 0; c0 < kVN; c0 += 16) {
          if (c0 >= I.nrows) break;
          float v[16];
          tmem_ld16(tmem + lane_addr + kColO + h * kVN + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = c0 + i;
            if (n < I.nrows) {
              const float lr = ms.lrow[n];
              const float val = lr > 0.f ? v[i] * (p.out_scale / lr) : 0.f;
              const int d = h * 128 + ti;
              if (split) {
                slot_o(cp, slot)[(size_t)n * kHeadDim + d] = val;
              } else {
                static_cast<__nv_bfloat16*>(ptr.out)[ms.out_off[pi][n] + d] = __float2bfloat16_rn(val);
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(ms.o_free));
      if (split) {
        if (ti < I.nrows) {
          const float lr = ms.lrow[ti];
          slot_lse(cp, slot)[ti] = lr > 0.f ? ms.m[pi][ti] - kSigma + log2f(lr) : -INFINITY;
        }
        __threadfence();
        RowBlock rb;
        rb.seq = I.seq;
        rb.kvh = I.kvh;
        rb.row0 = I.row0;
        rb.nrows = I.nrows;
        rb.nsplit = I.nsplit;
        rb.slot_base = I.slot_base;
        finish_split_block(p, ptr, cp, I.block, rb, ti, 128, 2, &ms.merge_flag);
      }
#pragma unroll
      for (int n = 0; n < kVN; ++n) l[n] = 0.f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side --

namespace {

std::mutex g_tc_mu;
thread_local char t_tc_err[256] = "";

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  std::lock_guard<std::mutex> lk(g_tc_mu);
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &f, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

}  // namespace

// 4-D map over an e4m3 cache [NB, P, Hkv, 256]: box = one d-half (128 B) x 1 head x P rows
// x 1 page, 128-byte swizzle.
bool make_cache_tmap(CUtensorMap* m, const pg_tensor* t, int P) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    snprintf(t_tc_err, sizeof t_tc_err, "cuTensorMapEncodeTiled unavailable");
    return false;
  }
  cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)t->shape[2], (cuuint64_t)t->shape[1], (cuuint64_t)t->shape[0]};
  cuuint64_t strides[3] = {(cuuint64_t)t->stride[2], (cuuint64_t)t->stride[1], (cuuint64_t)t->stride[0]};
  cuuint32_t box[4] = {128, 1, (cuuint32_t)P, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, t->data, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(t_tc_err, sizeof t_tc_err, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return false;
  }
  return true;
}

const char* tc_last_error() { return t_tc_err; }

int launch_verify_tc(const Problem& p, const Pointers& ptr, const ClassPlan& cp, const pg_tensor* k,
                     const pg_tensor* v, int sms, cudaStream_t stream) {
  (void)sms;
  if (!p.kv_is_fp8) return 0;
  CUtensorMap tk, tv;
  if (!make_cache_tmap(&tk, k, p.P) || !make_cache_tmap(&tv, v, p.P)) return -1;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e;
  auto kern = p.q_is_fp8 ? verify_tc_kernel<true> : verify_tc_kernel<false>;
  const int which = p.q_is_fp8 ? 2 : 1;
  if (dev >= 0 && dev < 64 && !(attr_done[dev] & which)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) {
      snprintf(t_tc_err, sizeof t_tc_err, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      return -1;
    }
    attr_done[dev] |= which;
  }
  kern<<<cp.num_ctas, kVThreads, kSmemBytes, stream>>>(tk, tv, p, ptr, cp);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(t_tc_err, sizeof t_tc_err, "verify kernel launch: %s", cudaGetErrorString(e));
    return -1;
  }
  return 1;
}

}  // namespace pgqa
