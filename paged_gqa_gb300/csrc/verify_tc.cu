// verify_tc.cu -- tcgen05 (TMEM, TMA) kernel for verify blocks: q_len*G <= 64 query rows of
// one (sequence, kv head) against an FP8 e4m3 paged KV cache.
//
// What the pages ask of this path ("Optimize Qwen3.5 MTP unified attention on gfx950",
// Motivation and Modifications): all q_len x G query rows of a kv head share one load of
// each KV page (BLOCK_M covers tokens x heads), split-KV segments keep every SM busy, and
// the FP8 descales are per-tensor scalars. The launch shape on that page (BLOCK_M 32,
// TILE 32, 8-64 segments on gfx950) is prior art; this kernel is laid out for sm_103a:
//
//   * swap-AB: the 128 keys of a tile are the MMA's M dimension and the query rows are N,
//     so a short query still fills the 128-lane tensor core;
//   * FP8 K and V go from HBM to shared memory by TMA (one box per page and d-half,
//     addressed through the block table) and into tcgen05.mma kind::f8f6f4 untouched; the
//     dequant scales are folded into the score scale (k_descale) and the output scale
//     (v_descale);
//   * bf16 Q is split once per block into e4m3 hi + lo parts (q*2^s = hi + lo, exact to
//     ~2^-16 of the block's max); both parts are stacked as one N = 128 operand, so
//     [S_hi | S_lo] = K [Q_hi; Q_lo]^T is 8 MMAs that read each K tile once;
//   * P is split the same way (p = hi + lo in e4m3, about bf16's precision; a single e4m3
//     P would miss the 5e-3 relative-L2 bar) and stacked the same way, so
//     [O_hi | O_lo] = V^T [P_hi; P_lo]^T is 8 MMAs that read each V tile once; O = O_hi + O_lo;
//   * online softmax over keys: keys live on TMEM lanes, so the row max is a cross-lane
//     reduction (redux.sync + shared memory). It is only taken when some score exceeds the
//     running reference by 2^4 (the reference then moves to the exact max and O^T and the
//     row sums are rescaled); otherwise P = 2^(s - m + 4) <= 256 fits e4m3 directly;
//   * S and P.V are issued by two threads: one thread issues tcgen05.mma at about one per
//     44 ns, slower than the tensor pipe retires these shapes, and S can then run ahead of
//     the softmax while P.V of the previous tile completes;
//   * persistent CTAs (one per SM) walk a contiguous range of key tiles cut by the plan
//     kernel; a block cut across CTAs is finished by the last piece with a log-sum-exp merge.
//
// Warp roles (768 threads): warp 0 = S issuer (+ TMEM owner), warp 1 = P.V issuer, warps
// 2, 3, 20 = K producers (TMA), warps 4-19 = softmax and epilogue, warps 21-23 = V
// producers (TMA). Softmax thread (q, c, lane) owns TMEM lane 32q+lane (= key of the tile,
// = d within a d-half for O^T) and rows [16c, 16c+16). Shared memory: Q hi/lo 32 KB, 2 K
// and 2 V stages of 32 KB, two P hi/lo buffers of 16 KB, barriers and row state (~205 KB,
// one CTA per SM). TMEM: 2 S buffers of 128 columns, O^T 256 columns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdio>

#include "common.cuh"
#include "device_util.cuh"
#include "self_plan.cuh"
#include "tc_kernels.cuh"
#include "tc_util.cuh"

namespace pgqa {

namespace {

using namespace tc;

constexpr int kVN = 64;            // query rows of a verify block (MMA N per Q or P part)
constexpr int kSoftWarps = 16;     // four per TMEM lane quarter: the softmax is latency-bound
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kRowGroups = kSoftWarps / 4;
constexpr int kCols = kVN / kRowGroups;  // rows per softmax thread (16)
// 24 warps in six warpgroups. Warpgroup 0: warp 0 = S issuer (+ TMEM owner), warp 1 = P.V
// issuer, warps 2-3 = K producers; warpgroups 1-4 (warps 4-19) = softmax; warpgroup 5:
// warp 20 = K producer, warps 21-23 = V producers. The kernel starts with 80 registers a
// thread (65536 / 768, rounded down to 8); the softmax warpgroups then take 96 and the
// others 48 (setmaxnreg): 4 x 128 x 96 + 2 x 128 x 48 = 768 x 80.
constexpr int kVThreads = 768;
constexpr int kLaunchRegs = 80;
constexpr int kSoftRegs = 96, kOtherRegs = 48;
static_assert(kLaunchRegs == (65536 / kVThreads) / 8 * 8, "launch registers");
static_assert(4 * 128 * kSoftRegs + 2 * 128 * kOtherRegs == kVThreads * kLaunchRegs, "register split");
static_assert(kCols == 16, "the epilogue's row-sum reduction assumes 16 rows per thread");
constexpr int kSoftWarp0 = 4;
constexpr int kQChunks = kVN * 16 / kSoftThreads;  // Q chunks of 16 elements per softmax thread
static_assert(kQChunks * kSoftThreads == kVN * 16, "Q chunks");
constexpr int kProdPerOp = 3;  // TMA producer warps per operand (one thread issues too slowly)
constexpr int kKStages = 2;        // K tiles in shared memory (freed by S = K Q^T)
constexpr int kVStages = 2;        // V tiles in shared memory (held until O += P V)
constexpr int kPBufs = 2;          // P buffers: P(g+1) is written while P.V(g) runs
constexpr float kTau = 4.f;        // rescale when a score exceeds the reference by 2^kTau
constexpr float kSigma = 4.f;      // P is stored scaled by 2^kSigma (max 2^(kTau+kSigma) = 256)
constexpr float kMInit = -1.0e30f; // reference of a row before its first key

// Q: per d-half h, [Q_hi 64 rows][Q_lo 64 rows] x 128 B (K-major, 128B swizzle).
constexpr uint32_t kQHalf = 2 * kVN * 128;      // 16 KB
constexpr uint32_t kQPartOff = kVN * 128;       // Q_lo rows start 8 KB into the half
constexpr uint32_t kKVHalf = kTileKeys * 128;   // [128 keys][128 B]
constexpr uint32_t kKVTile = 2 * kKVHalf;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + 2 * kQHalf;
constexpr uint32_t kOffV = kOffK + kKStages * kKVTile;
constexpr uint32_t kOffP = kOffV + kVStages * kKVTile;  // [128 keys][P_hi 64 B | P_lo 64 B]
constexpr uint32_t kPBuf = kTileKeys * 128;  // 16 KB
constexpr uint32_t kOffMisc = kOffP + kPBufs * kPBuf;

// TMEM columns: S buffers [S_hi | S_lo] (2 x 128), O^T d-half h [O_hi | O_lo] (2 x 128).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 256;

template <int kQM>
struct Shapes {
  static constexpr int kSN = kQM != kQSplit ? kVN : 2 * kVN;  // S MMA N: Q, or [Q_hi; Q_lo]
  static constexpr int kQEsz = kQM == kQGiven ? 1 : 2;        // bytes of a Q element in HBM
};
constexpr uint32_t kIdescO = idesc_e4m3(128, 2 * kVN, true, true);  // V^T (MN) x [P_hi; P_lo]^T (MN)

struct Misc {
  // arrays read with 16-byte vector loads first
  alignas(16) float m[2][kVN];
  alignas(16) float mo[2][kVN];   // kSigma - m: the per-row offset of the exponent
  alignas(16) float red[4][kVN];
  alignas(16) float alpha[kVN];
  alignas(16) int lim[2][kVN];
  alignas(16) long long out_off[2][kVN];
  alignas(16) float merge_w[kMergeMaxSplits * kSlotRows];
  alignas(16) float lse_stage[kVN];  // a split piece's log2-sum-exp per row, for its bulk store
  alignas(8) uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[kPBufs], pv_done[kPBufs], q_full, q_free, o_ready, o_free, drain[2], merge_full;
  uint64_t never;  // no thread ever arrives (the failure-path test waits on it)
  float qscale[2];
  float amax[kSoftWarps];
  uint32_t tmem_base;
  int abort_flag;
  int merge_flag;
  // Self-planned verify class (Problem::fused_verify): this CTA's items, packed by
  // self_plan::plan_warp, and their count.
  int4 fitem[kFusedMaxBlocks];
  int4 fseq[kFusedMaxBlocks];  // each item's sequence: {first token, q_len, L, 0}
  int fcount;
};
static_assert(offsetof(Misc, m) % 16 == 0 && offsetof(Misc, k_full) % 8 == 0, "Misc alignment");
constexpr size_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
static_assert(sizeof(self_plan::Scratch) <= kKStages * kKVTile, "the self-plan scratch fits the K stages");

struct Item {
  int block, seq, kvh, row0, nrows, kv_end, nsplit, split, slot_base;
  int tile_begin, ntiles, kv_hi;
  int q0, qn, L;
};

// Item it of a self-planned CTA.
__device__ __forceinline__ Item load_item_fused(const Problem& p, const Pointers& ptr, const Misc& ms, int it) {
  const self_plan::Piece f = self_plan::unpack(p, ms.fitem[it]);
  Item r;
  r.block = f.block;
  r.seq = f.seq;
  r.kvh = f.kvh;
  r.tile_begin = f.tile_begin;
  r.ntiles = f.ntiles;
  r.split = f.split;
  r.nsplit = f.nsplit;
  r.slot_base = f.slot_base;
  const int4 sq = ms.fseq[it];
  r.q0 = sq.x;
  r.qn = sq.y;
  r.L = sq.z;
  r.row0 = 0;
  r.nrows = r.qn * p.G;
  r.kv_end = r.L;  // the causal limit of the last row (token qn - 1) is L
  r.kv_hi = min((r.tile_begin + r.ntiles) * kTileKeys, r.kv_end);
  return r;
}

template <bool kFused>
__device__ __forceinline__ Item load_item(const Problem& p, const ClassPlan& cp, const Pointers& ptr,
                                          const Misc& ms, int it) {
  if (kFused) return load_item_fused(p, ptr, ms, it);
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

}  // namespace

template <int kQM, bool kFused>
__global__ void __launch_bounds__(kVThreads, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 Problem p, Pointers ptr, ClassPlan cp) {
  constexpr int kSN = Shapes<kQM>::kSN;
  constexpr int kQEsz = Shapes<kQM>::kQEsz;
  constexpr uint32_t kIdescS = idesc_e4m3(128, kSN, false, false);  // K (K-major) x Q (K-major)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &ms.abort_flag;

  auto bar = [&](const uint64_t& b) { return smem_u32(&b); };
  // The plan is read once the previous grid (the plan kernel) has completed; a self-planned
  // CTA works out its own items first. A CTA with no work (an empty class, or fewer items
  // than CTAs) leaves before any set-up.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int item_begin = 0, item_end = 0;
  self_plan::Scratch& fs = *reinterpret_cast<self_plan::Scratch*>(smem + kOffK);
  if (kFused) {
    // The sequences' reads go out first; the set-up below overlaps them.
    self_plan::load(p, ptr, fs);
  } else {
    item_begin = cp.cta_item_begin[blockIdx.x];
    item_end = cp.cta_item_begin[blockIdx.x + 1];
    if (item_begin >= item_end) return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(ms.k_full[s]), kProdPerOp);
      mbar_init(bar(ms.k_empty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(ms.v_full[s]), kProdPerOp);
      mbar_init(bar(ms.v_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(ms.s_full[b]), 1);
      mbar_init(bar(ms.s_free[b]), kSoftThreads);
    }
    for (int b = 0; b < kPBufs; ++b) {
      mbar_init(bar(ms.p_full[b]), kSoftThreads);
      mbar_init(bar(ms.pv_done[b]), 1);
    }
    mbar_init(bar(ms.q_full), kSoftThreads);
    mbar_init(bar(ms.q_free), 1);
    mbar_init(bar(ms.o_ready), 1);
    mbar_init(bar(ms.o_free), kSoftThreads);
    mbar_init(bar(ms.drain[0]), 1);
    mbar_init(bar(ms.drain[1]), 1);
    mbar_init(bar(ms.merge_full), 1);
    mbar_init(bar(ms.never), 1);
    ms.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&ms.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (kFused) {
    __syncthreads();  // the sequences are staged
    if (warp == 1) self_plan::plan_warp(p, fs, cp.num_ctas, lane, ms.fitem, ms.fseq, &ms.fcount);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  if (kFused) {
    item_end = ms.fcount;
    if (item_end == 0) {  // no range or no tile in it: give the columns back and leave
      if (warp == 0) tmem_dealloc(tmem, kTmemCols);
      return;
    }
  }
  // The next kernel on the stream (the other class) may start its own checks now.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Warpgroup roles. setmaxnreg is executed by all four warps of a warpgroup, first thing
  // in its role's branch (the launcher checks that the kernel starts with kLaunchRegs).
  const int wg = warp >> 2;
  if (wg >= 1 && wg <= kRowGroups) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftRegs));
    // ------------------------------------------------------------ softmax + epilogue
    const int sw = warp - kSoftWarp0;        // 0..15
    const int gi = sw * 32 + lane;           // 0..511
    const int q4 = warp & 3;                 // TMEM lane quarter
    const int c0 = (sw >> 2) * kCols;        // first row (column) this thread owns
    const int group_bar = 3 + (sw >> 2);     // named barrier of the row group's four warps
    // {descale, 1/descale} of a per-tensor cast of Q (kQCast), the same in every thread
    const float2 q_cast = kQM == kQCast ? q_cast_scales(ptr.q_amax, p.q_amax_parts, lane) : make_float2(1.f, 1.f);
    const int ti = q4 * 32 + lane;           // TMEM lane = key in tile = d in half
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    float l[kCols];
#pragma unroll
    for (int n = 0; n < kCols; ++n) l[n] = 0.f;
    bool bad = false;
    uint32_t merge_phase = 0;  // phases of merge_full used so far
    // Failure-path test: a bounded wait on a barrier nothing arrives on runs out in every
    // softmax thread (by its own limit or by the abort flag another thread raised); they
    // then skip the items, so no Q is published, the MMA issuers give up on q_full / p_full
    // and every producer drains the copies it issued.
    const bool stalled = p.stall_test_ns && !mbar_wait(bar(ms.never), 0, abort_flag, ptr.err, p.stall_test_ns);
    if (!stalled) {
    // This call's split-counter tag, read once: the epoch word does not move while this grid
    // runs (the plan kernel advances it after this grid, or before it and before the wait
    // above), and the load's latency then stays off every arrival.
    const unsigned long long ctag = gi == 0 ? split_tag(p, cp) : 0ull;

    auto q_prep = [&](const Item& I, int ii) {
      const int pi = ii & 1;
      if (ii >= 1 && !mbar_wait(bar(ms.q_free), (ii - 1) & 1, abort_flag, ptr.err)) bad = true;
      if (gi < kVN) {
        const int n = gi;
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
        ms.mo[pi][n] = kSigma - ms.m[pi][n];
      }
      // 64 rows x 16 chunks of 16 elements; thread gi takes chunks gi + kSoftThreads k
      auto src_of = [&](int r, int ch) -> const uint8_t* {
        const RowMap m = map_row(I.row0 + r, p.G, I.kvh);
        return static_cast<const uint8_t*>(ptr.q) +
               ((size_t)(I.q0 + m.t) * p.q_st + (size_t)m.h * p.q_sh + ch * 16) * kQEsz;
      };
      // part 0 = hi rows 0..63, part 1 = lo rows 64..127 of the stacked operand
      auto dst_of = [&](int part, int r, int ch) -> uint8_t* {
        const int h = ch >> 3, c = ch & 7, rr = part * kVN + r;
        return smem + kOffQ + h * kQHalf + rr * 128 + ((c ^ (rr & 7)) << 4);
      };
      if (kQM == kQGiven) {
        uint4 v[kQChunks];
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) {
          const int c = gi + k * kSoftThreads, r = c >> 4, ch = c & 15;
          v[k] = r < I.nrows ? *reinterpret_cast<const uint4*>(src_of(r, ch)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) {
          const int c = gi + k * kSoftThreads, r = c >> 4, ch = c & 15;
          *reinterpret_cast<uint4*>(dst_of(0, r, ch)) = v[k];
        }
        if (gi == 0) ms.qscale[pi] = 1.f;
      } else if (kQM == kQCast) {
        uint4 v[kQChunks][2];
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) {
          const int c = gi + k * kSoftThreads, r = c >> 4, ch = c & 15;
          if (r < I.nrows) {
            const uint4* s = reinterpret_cast<const uint4*>(src_of(r, ch));
            v[k][0] = s[0];
            v[k][1] = s[1];
          } else {
            v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) {
          const int c = gi + k * kSoftThreads, r = c >> 4, ch = c & 15;
          *reinterpret_cast<uint4*>(dst_of(0, r, ch)) = bf16x16_to_e4m3(v[k][0], v[k][1], q_cast.y);
        }
        if (gi == 0) ms.qscale[pi] = q_cast.x;
      } else {
        uint4 v[kQChunks][2];
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) {
          const int c = gi + k * kSoftThreads, r = c >> 4, ch = c & 15;
          if (r < I.nrows) {
            const uint4* s = reinterpret_cast<const uint4*>(src_of(r, ch));
            v[k][0] = s[0];
            v[k][1] = s[1];
          } else {
            v[k][0] = v[k][1] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) {
          const uint32_t w[8] = {v[k][0].x, v[k][0].y, v[k][0].z, v[k][0].w,
                                 v[k][1].x, v[k][1].y, v[k][1].z, v[k][1].w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 f = bf2(w[i]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
        amax = warp_max(amax);
        if (lane == 0) ms.amax[sw] = amax;
        named_barrier(1, kSoftThreads);
        amax = 0.f;
#pragma unroll
        for (int w = 0; w < kSoftWarps; ++w) amax = fmaxf(amax, ms.amax[w]);
        // 2^sig * amax in [128, 256): exponent arithmetic on the bits
        int sig = 0;
        if (amax > 0.f && isfinite(amax)) sig = 7 - (int)((__float_as_uint(amax) >> 23) & 0xff) + 127;
        sig = max(-100, min(100, sig));
        const float scale = ldexpf(1.f, sig);
#pragma unroll
        for (int k = 0; k < kQChunks; ++k) {
          const int c = gi + k * kSoftThreads, r = c >> 4, ch = c & 15;
          const uint32_t w[8] = {v[k][0].x, v[k][0].y, v[k][0].z, v[k][0].w,
                                 v[k][1].x, v[k][1].y, v[k][1].z, v[k][1].w};
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f0 = bf2(w[2 * i]), f1 = bf2(w[2 * i + 1]);
            split4(f0.x * scale, f0.y * scale, f1.x * scale, f1.y * scale, hw[i], lw[i]);
          }
          *reinterpret_cast<uint4*>(dst_of(0, r, ch)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(dst_of(1, r, ch)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        if (gi == 0) ms.qscale[pi] = ldexpf(1.f, -sig);
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(ms.q_full));
    };

    // scores of this thread's key for its 32 rows: S_hi + S_lo (one part for FP8 Q)
    auto load_s = [&](int b, float (&t)[kCols]) {
#pragma unroll
      for (int k = 0; k < kCols; k += 16) {
        float v[16];
        tmem_ld16(tmem + lane_addr + kColS + b * 128 + c0 + k, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) t[k + i] = v[i];
        if (kQM == kQSplit) {
          tmem_ld16(tmem + lane_addr + kColS + b * 128 + kVN + c0 + k, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) t[k + i] += v[i];
        }
      }
    };

    int ii = 0;
    uint32_t g = 0;
    if (item_end > item_begin) q_prep(load_item<kFused>(p, cp, ptr, ms, item_begin), 0);
    for (int it = item_begin; it < item_end; ++it, ++ii) {
      const Item I = load_item<kFused>(p, cp, ptr, ms, it);
      const int pi = ii & 1;
      named_barrier(1, kSoftThreads);  // q_prep's shared writes (lim, m, qscale) are visible
      const float c = p.score_scale_log2 * ms.qscale[pi];
      const int min_lim = I.L - I.qn + map_row(I.row0, p.G, I.kvh).t;
      // A failed wait (timeout or abort) does not leave the loops: every later wait then
      // fails fast, so all softmax warps still pass the same barriers and finish.
      for (int j = 0; j < I.ntiles; ++j, ++g) {
        const int b = g & 1;
        const int key0 = (I.tile_begin + j) * kTileKeys;
        const int key = key0 + ti;
        float t[kCols];
        if (!mbar_wait(bar(ms.s_full[b]), (g >> 1) & 1, abort_flag, ptr.err)) bad = true;
        tc_fence_after();
        load_s(b, t);
        tmem_wait_ld();
        // x = s c - m + sigma: the exponent of P, one FFMA per score
        const bool need_mask = (key0 + kTileKeys > I.kv_hi) || (key0 + kTileKeys - 1 > min_lim);
        float xmax = -INFINITY;
        if (need_mask) {
          const bool kin = key < I.kv_hi;
#pragma unroll
          for (int n = 0; n < kCols; n += 4) {
            const float4 o4 = *reinterpret_cast<const float4*>(&ms.mo[pi][c0 + n]);
            const int4 l4 = *reinterpret_cast<const int4*>(&ms.lim[pi][c0 + n]);
            t[n] = (kin && key <= l4.x) ? fmaf(t[n], c, o4.x) : -INFINITY;
            t[n + 1] = (kin && key <= l4.y) ? fmaf(t[n + 1], c, o4.y) : -INFINITY;
            t[n + 2] = (kin && key <= l4.z) ? fmaf(t[n + 2], c, o4.z) : -INFINITY;
            t[n + 3] = (kin && key <= l4.w) ? fmaf(t[n + 3], c, o4.w) : -INFINITY;
            xmax = fmaxf(xmax, fmaxf(fmaxf(t[n], t[n + 1]), fmaxf(t[n + 2], t[n + 3])));
          }
        } else {
#pragma unroll
          for (int n = 0; n < kCols; n += 4) {
            const float4 o4 = *reinterpret_cast<const float4*>(&ms.mo[pi][c0 + n]);
            t[n] = fmaf(t[n], c, o4.x);
            t[n + 1] = fmaf(t[n + 1], c, o4.y);
            t[n + 2] = fmaf(t[n + 2], c, o4.z);
            t[n + 3] = fmaf(t[n + 3], c, o4.w);
            xmax = fmaxf(xmax, fmaxf(fmaxf(t[n], t[n + 1]), fmaxf(t[n + 2], t[n + 3])));
          }
        }
        // vote of the row group (its four warps hold all 128 keys of its rows): does any
        // score exceed its row reference by more than 2^kTau? Row groups do not wait for
        // one another, so their phases interleave.
        const bool rescale = barrier_or(group_bar, 128, xmax > kTau + kSigma);
        if (rescale) {
          // Reload the raw scores (S buffer b is released only after this block; x may have
          // lost s entirely against a -1e30 reference), take the exact tile maximum of s c
          // per row, then the new reference.
          tc_fence_after();
          load_s(b, t);
          tmem_wait_ld();
          const bool kin = key < I.kv_hi;
#pragma unroll
          for (int n = 0; n < kCols; ++n) {
            const bool vis = !need_mask || (kin && key <= ms.lim[pi][c0 + n]);
            t[n] = vis ? t[n] * c : -INFINITY;  // s c, masked
            const float r = warp_max(t[n]);
            if (lane == n) ms.red[q4][c0 + n] = r;
          }
          named_barrier(group_bar, 128);
          if (q4 == 0 && lane < kCols) {
            const int n = c0 + lane;
            const float mt = fmaxf(fmaxf(ms.red[0][n], ms.red[1][n]), fmaxf(ms.red[2][n], ms.red[3][n]));
            const float m_old = ms.m[pi][n];
            const float mn = fmaxf(m_old, mt);
            ms.alpha[n] = ex2(m_old - mn);
            ms.m[pi][n] = mn;
            ms.mo[pi][n] = kSigma - mn;
          }
          named_barrier(group_bar, 128);
#pragma unroll
          for (int n = 0; n < kCols; ++n) {
            t[n] += ms.mo[pi][c0 + n];
            l[n] *= ms.alpha[c0 + n];
          }
        }
        // S buffer b is read for the last time above (the rescale path reloads it): only now
        // may the S issuer overwrite it with S(g+2)
        tc_fence_before();
        mbar_arrive(bar(ms.s_free[b]));
        // P = 2^x in f16, split into e4m3 hi + lo (4 rows per word); row sums in fp32
        uint32_t ph[kCols / 4], pl[kCols / 4];
#pragma unroll
        for (int n = 0; n < kCols; n += 4) {
          __half2 s01, s23;
          p_split4_f16(t[n], t[n + 1], t[n + 2], t[n + 3], ph[n / 4], pl[n / 4], s01, s23);
          const float2 f01 = __half22float2(s01), f23 = __half22float2(s23);
          l[n] += f01.x;
          l[n + 1] += f01.y;
          l[n + 2] += f23.x;
          l[n + 3] += f23.y;
        }
        // P buffer g & 1 is free once P.V(g-2) has completed; O^T may be rescaled once
        // P.V(g-1) has. Each barrier's next phase needs a P these threads have not written yet,
        // so a late parity wait cannot mistake it for the phase it waits for.
        if (g >= 2 && !mbar_wait(bar(ms.pv_done[g & 1]), ((g >> 1) - 1) & 1, abort_flag, ptr.err)) bad = true;
        if (rescale && j > 0 && !mbar_wait(bar(ms.pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort_flag, ptr.err))
          bad = true;
        tc_fence_after();
        if (rescale && j > 0) {
          // O^T (both d-halves, both P parts), column by column
#pragma unroll 1
          for (int h = 0; h < 4; ++h) {
#pragma unroll 1
            for (int k = 0; k < kCols; k += 16) {
              float v[16];
              const uint32_t a = tmem + lane_addr + kColO + (h >> 1) * 128 + (h & 1) * kVN + c0 + k;
              tmem_ld16(a, v);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] *= ms.alpha[c0 + k + i];
              tmem_st16(a, v);
            }
          }
          tmem_wait_st();
        }
        if (key0 + kTileKeys > I.kv_hi) {
          // keys past the piece's end: their V rows (stale or NaN slots) become zeros
          const uint32_t st = g % kVStages;
          if (!mbar_wait(bar(ms.v_full[st]), (g / kVStages) & 1, abort_flag, ptr.err)) bad = true;
          if (key >= I.kv_hi) {
            const uint4 z = make_uint4(0, 0, 0, 0);
            // the kRowGroups threads of key ti zero 64 bytes each: d-half rg / 2, 16-byte
            // chunks 4 (rg % 2) .. 4 (rg % 2) + 3 of the (swizzled) 128-byte row
            const int rg = c0 / kCols;
            uint8_t* row = smem + kOffV + st * kKVTile + (rg >> 1) * kKVHalf + ti * 128;
#pragma unroll
            for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4*>(row + ((((rg & 1) * 4 + i) ^ (ti & 7)) << 4)) = z;
          }
        }
        // P^T row of key ti: [P_hi rows 0..63 | P_lo rows 0..63], 128-byte swizzle; this
        // thread writes rows [c0, c0 + kCols) of both parts
        {
#pragma unroll
          for (int cc = 0; cc < kCols / 16; ++cc) {
            const int chunk_hi = (c0 >> 4) + cc, chunk_lo = 4 + chunk_hi;
            *reinterpret_cast<uint4*>(smem + kOffP + (g & 1) * kPBuf + ti * 128 + ((chunk_hi ^ (ti & 7)) << 4)) =
                make_uint4(ph[4 * cc], ph[4 * cc + 1], ph[4 * cc + 2], ph[4 * cc + 3]);
            *reinterpret_cast<uint4*>(smem + kOffP + (g & 1) * kPBuf + ti * 128 + ((chunk_lo ^ (ti & 7)) << 4)) =
                make_uint4(pl[4 * cc], pl[4 * cc + 1], pl[4 * cc + 2], pl[4 * cc + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(ms.p_full[g & 1]));
      }
      // Q of the next item while this item's last P.V runs
      if (it + 1 < item_end) q_prep(load_item<kFused>(p, cp, ptr, ms, it + 1), ii + 1);

      // ---------------------------------------------------------- epilogue
      if (!mbar_wait(bar(ms.o_ready), ii & 1, abort_flag, ptr.err)) bad = true;
      tc_fence_after();
      // row sums: reduce l over the 128 key lanes (warp reduce-scatter, then across quarters)
      {
        float v[kCols];
#pragma unroll
        for (int n = 0; n < kCols; ++n) v[n] = l[n];
#pragma unroll
        for (int w = kCols / 2, o = 16; o >= 2; w >>= 1, o >>= 1) {
          const bool up = lane & o;
#pragma unroll
          for (int i = 0; i < w; ++i) {
            const float send = up ? v[i] : v[i + w];
            const float keep = up ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
        // lanes 2r and 2r+1 now hold row c0 + r
        if ((lane & 1) == 0) ms.red[q4][c0 + (lane >> 1)] = v[0];
      }
      named_barrier(1, kSoftThreads);
      const bool split = I.nsplit > 1;
      // a split piece's partial stays in code units (v_descale is applied by the merge)
      const float num = split ? 1.f : p.out_scale;
      float inv[kCols];
#pragma unroll
      for (int n = 0; n < kCols; ++n) {
        const float lr = ms.red[0][c0 + n] + ms.red[1][c0 + n] + ms.red[2][c0 + n] + ms.red[3][c0 + n];
        inv[n] = lr > 0.f ? __fdividef(num, lr) : 0.f;
      }
      float my_l = 0.f;  // row c0 + lane (lane < kCols), for the partial's log-sum-exp
      if (q4 == 0 && lane < kCols)
        my_l = ms.red[0][c0 + lane] + ms.red[1][c0 + lane] + ms.red[2][c0 + lane] + ms.red[3][c0 + lane];
      named_barrier(1, kSoftThreads);  // red is reused by the next item's first rescale
      const int slot = I.slot_base + I.split;
      if (split) {
        // The f16 partial (64 rows x 256 = 32 KB) and its log2-sum-exp per row leave through
        // the P buffers (free: every P.V of the item has completed) by two bulk stores from
        // one thread, so no warp waits on scattered stores and only that thread has global
        // writes to complete before the block's split counter moves.
        static_assert(kPBufs * kPBuf >= kVN * kHeadDim * 2, "the f16 partial fits the P buffers");
        __half* stage = reinterpret_cast<__half*>(smem + kOffP);  // 64 rows x 256 halves
        if (c0 < I.nrows) {  // warp-uniform
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            float v[16], w[16];
            tmem_ld16(tmem + lane_addr + kColO + h * 128 + c0, v);
            tmem_ld16(tmem + lane_addr + kColO + h * 128 + kVN + c0, w);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) stage[(c0 + i) * kHeadDim + h * 128 + ti] = __float2half_rn((v[i] + w[i]) * inv[i]);
          }
        }
        if (q4 == 0 && lane < kCols) {
          const int row = c0 + lane;
          ms.lse_stage[row] = my_l > 0.f ? ms.m[pi][row] - kSigma + log2f(my_l) : -INFINITY;
        }
        fence_proxy_async_smem();
        named_barrier(1, kSoftThreads);
        if (gi == 0) {
          // the counter's current word travels while the partial is written
          const unsigned long long seen = split_peek(cp.counters + I.block);
          bulk_store(slot_o(cp, slot), smem_u32(stage), (uint32_t)I.nrows * kHeadDim * 2u);
          bulk_store(slot_lse(cp, slot), smem_u32(ms.lse_stage), kVN * 4u);  // all 64 entries of the slot
          bulk_commit();
          bulk_wait_all();  // the partial is in global memory before the split counter moves
          fence_proxy_async_global();
          // is this piece the block's last? (merged below)
          fence_acq_rel_gpu();
          ms.merge_flag = split_arrive_from(cp.counters + I.block, seen, I.nsplit, ctag);
          fence_acq_rel_gpu();
        }
        named_barrier(1, kSoftThreads);  // the stage is reused by the next item's P; merge_flag
      } else {
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int k = 0; k < kCols; k += 16) {
            if (c0 + k < I.nrows) {  // warp-uniform
              float v[16], w[16];
              tmem_ld16(tmem + lane_addr + kColO + h * 128 + c0 + k, v);
              tmem_ld16(tmem + lane_addr + kColO + h * 128 + kVN + c0 + k, w);
              tmem_wait_ld();
              const int d = h * 128 + ti;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int n = c0 + k + i;
                if (n < I.nrows)
                  static_cast<__nv_bfloat16*>(ptr.out)[ms.out_off[pi][n] + d] =
                      __float2bfloat16_rn((v[i] + w[i]) * inv[k + i]);
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar(ms.o_free));
      if (split) {
        if (it + 1 == item_end && I.nsplit <= kMergeMaxSplits) {
          // The CTA's last item: its Q, K, V and P buffers are idle (every tile consumed,
          // every MMA complete), so if this piece is the block's last, the merge bulk-loads
          // the pieces' partials into them instead of reading them element by element (this
          // merge is the tail of the kernel). The counter moved right after the partial left.
          if (ms.merge_flag) {
            // the counter's reader fenced after its atomic; the barrier orders the rest after it
            const int ns = I.nsplit;
            constexpr uint32_t kRegion = kOffMisc - kOffQ;  // Q, K stages, V stages, P buffers
            constexpr uint32_t kRowBytes = kHeadDim * 2;  // f16
            const int rpp = min(kVN, (int)(kRegion / (ns * kRowBytes)) / 8 * 8);  // rows per pass
            for (int r0 = 0; r0 < I.nrows; r0 += rpp) {
              const int nr = min(rpp, I.nrows - r0);
              if (gi == 0) {
                fence_proxy_async_global();  // the partials are read by the async proxy
                fence_proxy_async_smem();    // after the generic accesses to these buffers
                mbar_expect_tx(bar(ms.merge_full), (uint32_t)(ns * nr) * kRowBytes);
                for (int i = 0; i < ns; ++i)
                  bulk_load(sbase + kOffQ + (uint32_t)(i * rpp) * kRowBytes,
                            slot_o(cp, I.slot_base + i) + (size_t)r0 * kHeadDim, (uint32_t)nr * kRowBytes,
                            bar(ms.merge_full));
              }
              if (r0 == 0) {
                // per-row weights 2^(lse_i - M) / sum while the partials load
                for (int r = gi; r < I.nrows; r += kSoftThreads) {
                  float lse[kMergeMaxSplits];
                  float M = -INFINITY;
#pragma unroll
                  for (int i = 0; i < kMergeMaxSplits; ++i) {
                    lse[i] = i < ns ? __ldcg(slot_lse(cp, I.slot_base + i) + r) : -INFINITY;
                    M = fmaxf(M, lse[i]);
                  }
                  float sum = 0.f;
#pragma unroll
                  for (int i = 0; i < kMergeMaxSplits; ++i) {
                    lse[i] = lse[i] == -INFINITY ? 0.f : exp2f(lse[i] - M);
                    sum += lse[i];
                  }
                  const float inv_sum = sum > 0.f ? p.out_scale / sum : 0.f;
#pragma unroll
                  for (int i = 0; i < kMergeMaxSplits; ++i)
                    if (i < ns) ms.merge_w[i * kSlotRows + r] = lse[i] * inv_sum;
                }
                named_barrier(2, kSoftThreads);
              }
              // the bulk loads are this CTA's own: wait for them even after an abort, before the
              // buffers are read or reloaded (and before the CTA may exit)
              if (!mbar_drain(bar(ms.merge_full), merge_phase & 1, abort_flag, ptr.err)) bad = true;
              ++merge_phase;
              for (int idx = gi; idx < nr * (kHeadDim / 4); idx += kSoftThreads) {
                const int r = idx / (kHeadDim / 4), d = (idx % (kHeadDim / 4)) * 4;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int i = 0; i < ns; ++i) {
                  const float w = ms.merge_w[i * kSlotRows + r0 + r];
                  const uint2 h = *reinterpret_cast<const uint2*>(smem + kOffQ + (size_t)(i * rpp + r) * kRowBytes + d * 2);
                  const float2 o01 = unpack_f16x2(h.x), o23 = unpack_f16x2(h.y);
                  acc.x += w * o01.x;
                  acc.y += w * o01.y;
                  acc.z += w * o23.x;
                  acc.w += w * o23.y;
                }
                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(ptr.out) + ms.out_off[pi][r0 + r] + d) =
                    make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
              }
              named_barrier(2, kSoftThreads);  // the buffers are reused by the next pass
            }
          }
        } else if (ms.merge_flag) {
          // a piece that is not its CTA's last item (or one of more than kMergeMaxSplits) and
          // arrived last: merge from global memory
          RowBlock rb;
          rb.seq = I.seq;
          rb.kvh = I.kvh;
          rb.row0 = I.row0;
          rb.nrows = I.nrows;
          rb.nsplit = I.nsplit;
          rb.slot_base = I.slot_base;
          merge_split_block(p, ptr, cp, rb, gi, kSoftThreads, 2, ms.merge_w);
        }
      }
#pragma unroll
      for (int n = 0; n < kCols; ++n) l[n] = 0.f;
    }
    }  // !stalled
    (void)bad;
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
    const bool k_prod = warp == 2 || warp == 3 || warp == 20;
    const bool v_prod = warp >= 21;
    if (k_prod || v_prod) {
      // ------------------------------------------------------------ TMA producers (K, V)
      // K and V have their own warps, so K tiles run ahead as soon as S = K Q^T frees a
      // stage, whatever the P.V of older tiles is doing; kProdPerOp warps share each tile
      // (producer i takes the pages whose index in the tile is i mod kProdPerOp, both
      // d-halves back to back), since one thread issues page-sized boxes too slowly to keep
      // HBM busy.
      const bool is_k = k_prod;
      const int pi = is_k ? (warp == 20 ? 2 : warp - 2) : warp - 21;
      const CUtensorMap* tmap = is_k ? &tmap_k : &tmap_v;
      const int nst = is_k ? kKStages : kVStages;
      const uint32_t region = sbase + (is_k ? kOffK : kOffV);
      uint64_t* full = is_k ? ms.k_full : ms.v_full;
      uint64_t* empty = is_k ? ms.k_empty : ms.v_empty;
      if (lane == 0) tma_prefetch_desc(tmap);
      const uint64_t policy = policy_evict_first();
      const int ppt = kTileKeys / p.P;  // pages per tile (1, 2, 4 or 8); 32 is a multiple
      uint32_t g = 0;
      uint32_t issued[kVStages > kKStages ? kVStages : kKStages] = {};
      bool stop = false;
      for (int it = item_begin; it < item_end && !stop; ++it) {
        const Item I = load_item<kFused>(p, cp, ptr, ms, it);
        const int32_t* bt_row = ptr.block_table + (size_t)I.seq * p.bt_stride;
        const int page0 = I.tile_begin * ppt;                 // first page of the piece
        const int npages = (I.kv_hi + p.P - 1) / p.P - page0; // pages the piece reads
        // a window of 32 block-table entries, one per lane, and the next one in flight
        // The window's entries are loaded without waiting for the piece's page count (its
        // sequence length may still be on its way): the index is clamped to the row, and an
        // entry is checked, or dropped past the piece's pages, when it is used.
        auto fetch_raw = [&](int w) -> int { return bt_row[min(page0 + w * 32 + lane, p.W - 1)]; };
        auto check = [&](int w, int raw) -> int {
          if (w * 32 + lane >= npages) return -1;
          if (raw < 0 || raw >= p.NB) {
            atomicOr(ptr.err, kErrPage);
            return 0;
          }
          return raw;
        };
        auto fetch = [&](int w) -> int { return check(w, fetch_raw(w)); };
        const int raw0 = fetch_raw(0), raw1 = fetch_raw(1);
        int cur = check(0, raw0), nxt = check(1, raw1);
        if (is_k && pi == 0) {
          // The softmax warps read this item's Q a few tiles from now (this warp runs ahead
          // by its stages): bring the rows into L2 so that read does not wait on HBM. Issued
          // after the block-table reads, which the first copies wait on.
          for (int r = lane; r < I.nrows; r += 32) {
            const RowMap m = map_row(I.row0 + r, p.G, I.kvh);
            const uint8_t* row = static_cast<const uint8_t*>(ptr.q) +
                                 ((size_t)(I.q0 + m.t) * p.q_st + (size_t)m.h * p.q_sh) * kQEsz;
#pragma unroll
            for (int c = 0; c < 256 * kQEsz; c += 128) prefetch_l2(row + c);
          }
        }
        int cur_w = 0;
        for (int j = 0; j < I.ntiles; ++j, ++g) {
          const int first = j * ppt;  // page of this tile, relative to the piece
          if (first / 32 != cur_w) {
            cur = nxt;
            cur_w = first / 32;
            nxt = fetch(cur_w + 1);
          }
          const int tile_pages = min(ppt, npages - first);
          const int mine = tile_pages > pi ? (tile_pages - pi + kProdPerOp - 1) / kProdPerOp : 0;
          const uint32_t st = g % nst, ph = (g / nst) & 1;
          int ok = 1;
          if (lane == 0) {
            ok = mbar_wait(bar(empty[st]), ph ^ 1, abort_flag, ptr.err);
            if (ok) mbar_expect_tx(bar(full[st]), (uint32_t)mine * p.P * 128u * 2u);
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) {
            stop = true;
            break;
          }
          for (int pg = pi; pg < tile_pages; pg += kProdPerOp) {
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
      // Every issued copy has landed before the CTA may exit.
      if (lane == 0) {
        for (int s = 0; s < nst; ++s)
          if (issued[s]) mbar_drain(bar(full[s]), (issued[s] - 1) & 1, abort_flag, ptr.err);
      }
      __syncwarp();
    } else if (warp == 0 || warp == 1) {
      // ------------------------------------------------------------ MMA issuers
      // One thread cannot issue tcgen05.mma faster than about one per 44 ns, below the tensor
      // pipe's rate for these shapes, so S = K Q^T and O^T += V^T P^T come from two warps:
      // S runs ahead as soon as a K tile and an S buffer are free, P.V as soon as P is
      // published. The two streams share no operand or accumulator.
      if (lane == 0) {
        const bool is_s = warp == 0;
        uint32_t g = 0;
        int ii = 0;
        bool ok = true;
        for (int it = item_begin; it < item_end && ok; ++it, ++ii) {
          const Item I = load_item<kFused>(p, cp, ptr, ms, it);
          for (int j = 0; j < I.ntiles && ok; ++j, ++g) {
            if (is_s) {
              if (j == 0 && !(ok = mbar_wait(bar(ms.q_full), ii & 1, abort_flag, ptr.err))) break;
              const uint32_t st = g % kKStages, b = g & 1;
              if (!(ok = mbar_wait(bar(ms.k_full[st]), (g / kKStages) & 1, abort_flag, ptr.err))) break;
              if (g >= 2 && !(ok = mbar_wait(bar(ms.s_free[b]), ((g >> 1) - 1) & 1, abort_flag, ptr.err))) break;
              tc_fence_after();
              const uint64_t a0 = smem_desc(sbase + kOffK + st * kKVTile, 16, 1024, kSw128);
              const uint64_t b0 = smem_desc(sbase + kOffQ, 16, 1024, kSw128);
#pragma unroll
              for (int kb = 0; kb < 8; ++kb) {
                const uint32_t off = (kb >> 2) * kKVHalf + (kb & 3) * 32, qoff = (kb >> 2) * kQHalf + (kb & 3) * 32;
                mma_e4m3(tmem + kColS + b * 128, a0 + (off >> 4), b0 + (qoff >> 4), kIdescS, kb ? 1u : 0u);
              }
              mma_commit(bar(ms.s_full[b]));
              mma_commit(bar(ms.k_empty[st]));
              if (j == I.ntiles - 1) mma_commit(bar(ms.q_free));
            } else {
              // the first P.V of an item overwrites O^T: the previous epilogue must be done
              if (j == 0 && ii >= 1 && !(ok = mbar_wait(bar(ms.o_free), (ii - 1) & 1, abort_flag, ptr.err))) break;
              if (!(ok = mbar_wait(bar(ms.p_full[g & 1]), (g >> 1) & 1, abort_flag, ptr.err))) break;
              const uint32_t st = g % kVStages;
              if (!(ok = mbar_wait(bar(ms.v_full[st]), (g / kVStages) & 1, abort_flag, ptr.err))) break;
              tc_fence_after();
              const uint64_t a0 = smem_desc(sbase + kOffV + st * kKVTile, 1024, 1024, kSw128);
              const uint64_t b0 = smem_desc(sbase + kOffP + (g & 1) * kPBuf, 1024, 1024, kSw128);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint32_t off = h * kKVHalf + kk * 4096, poff = kk * 4096;
                  mma_e4m3(tmem + kColO + h * 128, a0 + (off >> 4), b0 + (poff >> 4), kIdescO,
                           (j == 0 && kk == 0) ? 0u : 1u);
                }
              }
              mma_commit(bar(ms.v_empty[st]));
              mma_commit(bar(ms.pv_done[g & 1]));
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
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int launch_verify_tc(const Problem& p, const Pointers& ptr, const ClassPlan& cp, const pg_tensor* k,
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
  auto kern = p.fused_verify
                  ? (mode == kQCast ? verify_tc_kernel<kQCast, true>
                                    : mode == kQGiven ? verify_tc_kernel<kQGiven, true> : verify_tc_kernel<kQSplit, true>)
                  : (mode == kQCast ? verify_tc_kernel<kQCast, false>
                                    : mode == kQGiven ? verify_tc_kernel<kQGiven, false> : verify_tc_kernel<kQSplit, false>);
  const int which = 1 << (mode + (p.fused_verify ? 3 : 0));
  if (dev >= 0 && dev < 64 && !(attr_done[dev] & which)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) {
      char buf[160];
      snprintf(buf, sizeof buf, "cudaFuncSetAttribute(verify): %s", cudaGetErrorString(e));
      set_tc_error(buf);
      return -1;
    }
    // setmaxnreg.inc waits until the registers it asks for are free; the split adds up only
    // if the kernel starts with exactly kLaunchRegs per thread, so never launch otherwise.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess || fa.numRegs != kLaunchRegs) {
      char buf[160];
      snprintf(buf, sizeof buf, "verify kernel built with %d registers per thread; its warpgroup split needs %d",
               e == cudaSuccess ? fa.numRegs : -1, kLaunchRegs);
      set_tc_error(buf);
      return -1;
    }
    attr_done[dev] |= which;
  }
  e = launch_pdl(dependent, kern, cp.num_ctas, kVThreads, kSmemBytes, stream, tk, tv, p, ptr, cp);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    char buf[160];
    snprintf(buf, sizeof buf, "verify kernel launch: %s", cudaGetErrorString(e));
    set_tc_error(buf);
    return -1;
  }
  return 1;
}

}  // namespace pgqa
