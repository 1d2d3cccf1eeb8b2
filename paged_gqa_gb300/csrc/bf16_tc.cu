// bf16_tc.cu -- tcgen05 (TMEM, TMA) kernel for a bf16 Q against a bf16 paged KV cache, for
// both classes of row blocks (verify blocks of q_len x G <= 64 rows run as padded 128-row
// tiles; prefill blocks are 128 rows), bottom-right causal.
//
// The pages time this path in bf16 for the tiny verify case ("Optimize Qwen3.5 MTP unified
// attention on gfx950", Benchmarking: bf16 Q/K/V, context 600, q_len 2) and name FP8 as the
// variant for long contexts; this kernel is the bf16 counterpart of the FP8 prefill kernel:
//
//   * one row block = up to 128 rows (token r / G, head r % G of one kv head) as the MMA's
//     M; S = Q K^T is tcgen05.mma kind::f16 (bf16 inputs, fp32 accumulate) with N = 64 keys
//     per sub-tile (half of a 128-key plan tile: a bf16 row is 512 B, so a 64-key K or V
//     sub-tile is the 32 KB the FP8 kernels stage per 128 keys), K = 16 per instruction,
//     16 instructions per sub-tile;
//   * P = 2^(s - m + 4) is rounded to bf16 (8 significant bits, the precision the FP8
//     kernels reach with an e4m3 hi + lo split), written into TMEM over the sub-tile's S,
//     and used from there as the A operand of O += P V: M = 128 x N = 256 (all of d, V as
//     one MN-major operand of four 128-byte d-quarters) x K = 16 keys, 4 instructions;
//   * K and V pages arrive by TMA, one box per page (or half page, for 128-token pages)
//     and d-quarter, addressed through the block table;
//   * the softmax (two threads per row, 32 keys each, lazy rescale), the epilogue, split-KV
//     pieces and their merge are those of the FP8 prefill kernel.
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

constexpr int kRows = 128;                     // MMA M (rows of a block, padded)
constexpr int kSub = 64;                       // keys per sub-tile: S's N, P.V's K
constexpr int kSoftWarps = 8;
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kThreads = 128 + kSoftThreads;   // + K producer, 2 MMA issuers, V producer
constexpr int kVProducerWarp = 2 + kSoftWarps;
constexpr int kPVIssuerWarp = 3 + kSoftWarps;
constexpr int kHalfKeys = kSub / 2;            // keys per softmax thread
constexpr int kKStages = 2, kVStages = 2;
constexpr float kTau = 4.f;
constexpr float kSigma = 4.f;
constexpr float kMInit = -1.0e30f;

constexpr uint32_t kQQuarter = kRows * 128;    // [128 rows][64 d] bf16, one 128-byte d-quarter
constexpr uint32_t kKVQuarter = kSub * 128;    // [64 keys][64 d] bf16
constexpr uint32_t kKVTile = 4 * kKVQuarter;   // 32 KB
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + 4 * kQQuarter;
constexpr uint32_t kOffV = kOffK + kKStages * kKVTile;
constexpr uint32_t kOffMisc = kOffV + kVStages * kKVTile;
// TMEM columns: S double buffer (2 x 64: fp32 scores of 64 keys), O (256). P of a sub-tile
// (bf16, two keys per column) replaces the first 32 columns of its S buffer.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;
constexpr uint32_t kPCols = kSub / 2;

constexpr uint32_t kIdescS = idesc_bf16(kRows, kSub, false, false);  // Q (K-major) x K (K-major)
constexpr uint32_t kIdescO = idesc_bf16(kRows, 256, false, true);    // P (TMEM) x V (MN-major, N = d = 256)

struct Misc {
  alignas(16) float red[2][2][kRows];   // [sub-tile parity][key half][row] partial maxima
  alignas(16) float lsum[2][kRows];     // [key half][row] row-sum halves (epilogue)
  alignas(16) long long out_off[2][kRows];
  alignas(16) int lim[2][kRows];
  alignas(16) float merge_w[kMergeMaxSplits * kSlotRows];
  alignas(8) uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], pv_done[2];
  uint64_t p_full, q_full, q_free, o_ready, o_free, drain[2];
  uint64_t never;  // no thread ever arrives (the failure-path test waits on it)
  uint32_t tmem_base;
  int abort_flag;
  int merge_flag;
  // Self-planned verify class (Problem::fused_verify, class-0 launch): this CTA's items,
  // packed by self_plan::plan_warp, and their count.
  int4 fitem[kFusedMaxBlocks];
  int4 fseq[kFusedMaxBlocks];  // each item's sequence: {first token, q_len, L, 0}
  int fcount;
};
static_assert(offsetof(Misc, red) % 16 == 0 && offsetof(Misc, k_full) % 8 == 0, "Misc alignment");
constexpr size_t kSmemBytes = kOffMisc + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 232448, "fits the dynamic shared memory of a CTA");
static_assert(sizeof(self_plan::Scratch) <= kKStages * kKVTile, "the self-plan scratch fits the K stages");

struct Item {
  int block, seq, kvh, row0, nrows, kv_end, nsplit, split, slot_base;
  int tile_begin, nsub, kv_hi;
  int q0, qn, L;
};

// A work item of the plan (128-key tiles) as 64-key sub-tiles that end at the piece's last
// key: sub-tiles past it would read block-table entries the call does not define.
template <bool kFused>
__device__ __forceinline__ Item load_item(const Problem& p, const ClassPlan& cp, const Pointers& ptr,
                                          const Misc& ms, int it) {
  if (kFused) {  // a verify block of a self-planned CTA
    const self_plan::Piece f = self_plan::unpack(p, ms.fitem[it]);
    Item r;
    r.block = f.block;
    r.seq = f.seq;
    r.kvh = f.kvh;
    r.nsplit = f.nsplit;
    r.split = f.split;
    r.slot_base = f.slot_base;
    r.tile_begin = f.tile_begin;
    const int4 sq = ms.fseq[it];
    r.q0 = sq.x;
    r.qn = sq.y;
    r.L = sq.z;
    r.row0 = 0;
    r.nrows = r.qn * p.G;
    r.kv_end = r.L;  // the causal limit of the last row (token qn - 1) is L
    r.kv_hi = min((f.tile_begin + f.ntiles) * kTileKeys, r.kv_end);
    r.nsub = (r.kv_hi - f.tile_begin * kTileKeys + kSub - 1) / kSub;
    return r;
  }
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
  r.kv_hi = min(w.tile_end * kTileKeys, b.kv_end);
  r.nsub = (r.kv_hi - w.tile_begin * kTileKeys + kSub - 1) / kSub;
  r.q0 = ptr.qsl[b.seq];
  r.qn = ptr.qsl[b.seq + 1] - r.q0;
  r.L = ptr.seq_lens[b.seq];
  return r;
}

}  // namespace

template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
bf16_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
               Problem p, Pointers ptr, ClassPlan cp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Misc& ms = *reinterpret_cast<Misc*>(smem + kOffMisc);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &ms.abort_flag;
  auto bar = [&](const uint64_t& b) { return smem_u32(&b); };
  // The plan is read once the previous grid has completed; a self-planned CTA works out its
  // own items first (self_plan.cuh). A CTA with no work leaves before any set-up.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int item_begin = 0, item_end = 0;
  self_plan::Scratch& fs = *reinterpret_cast<self_plan::Scratch*>(smem + kOffK);
  if (kFused) {
    self_plan::load(p, ptr, fs);  // the set-up below overlaps these reads
  } else {
    item_begin = cp.cta_item_begin[blockIdx.x];
    item_end = cp.cta_item_begin[blockIdx.x + 1];
    if (item_begin >= item_end) return;
  }

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
      mbar_init(bar(ms.s_full[b]), 1);
      mbar_init(bar(ms.pv_done[b]), 1);
    }
    mbar_init(bar(ms.p_full), kSoftThreads);
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
  if (kFused) {
    __syncthreads();  // the sequences are staged
    if (warp == 0) self_plan::plan_warp(p, fs, cp.num_ctas, lane, ms.fitem, ms.fseq, &ms.fcount);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms.tmem_base;
  if (kFused) {
    item_end = ms.fcount;
    if (item_end == 0) {  // no range or no tile in it: give the columns back and leave
      if (warp == 1) tmem_dealloc(tmem, kTmemCols);
      return;
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0 || warp == kVProducerWarp) {
    // ------------------------------------------------------------ TMA producers (K, V)
    const bool is_k = warp == 0;
    const CUtensorMap* tmap = is_k ? &tmap_k : &tmap_v;
    const uint32_t region = sbase + (is_k ? kOffK : kOffV);
    uint64_t* full = is_k ? ms.k_full : ms.v_full;
    uint64_t* empty = is_k ? ms.k_empty : ms.v_empty;
    const int nst = is_k ? kKStages : kVStages;
    if (lane == 0) tma_prefetch_desc(tmap);
    const uint64_t policy = policy_evict_last();  // every row block of a sequence re-reads the pages
    const int R = min(p.P, kSub);                 // rows per box: a page, or half of a 128-token page
    const int ppsub = kSub / R;                   // boxes per sub-tile and d-quarter (1 for P >= 64)
    uint32_t g = 0;
    uint32_t issued[kVStages > kKStages ? kVStages : kKStages] = {};
    bool stop = false;
    for (int it = item_begin; it < item_end && !stop; ++it) {
      const Item I = load_item<kFused>(p, cp, ptr, ms, it);
      const int32_t* bt_row = ptr.block_table + (size_t)I.seq * p.bt_stride;
      const int key_begin = I.tile_begin * kTileKeys;     // a multiple of P (P divides 128)
      const int page0 = key_begin / p.P;                  // first page of the piece
      const int npages = (I.kv_hi + p.P - 1) / p.P - page0;
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
      int cur_w = 0;
      for (int s = 0; s < I.nsub; ++s, ++g) {
        const int first = (s * kSub) / p.P;      // page of this sub-tile, relative to the piece
        const int slot0 = (s * kSub) % p.P;      // first slot (nonzero only for 128-token pages)
        if (first / 32 != cur_w) {
          cur = nxt;
          cur_w = first / 32;
          nxt = fetch(cur_w + 1);
        }
        const int nb = min(ppsub, npages - first);
        const uint32_t st = g % nst, ph = (g / nst) & 1;
        int ok = 1;
        if (lane == 0) {
          ok = mbar_wait(bar(empty[st]), ph ^ 1, abort_flag, ptr.err);
          if (ok) mbar_expect_tx(bar(full[st]), (uint32_t)nb * 4u * (uint32_t)R * 128u);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
          stop = true;
          break;
        }
        for (int i = 0; i < nb; ++i) {
          const int blk = __shfl_sync(0xffffffffu, cur, (first + i) & 31);
          if (lane == 0) {
            const uint32_t row = (uint32_t)i * R * 128u;
            for (int qd = 0; qd < 4; ++qd)
              tma_load_4d(region + st * kKVTile + qd * kKVQuarter + row, tmap, qd * 64, I.kvh, slot0, blk,
                          bar(full[st]), policy);
          }
        }
        issued[st] = g / nst + 1;
      }
    }
    // Every issued copy has landed before the CTA may exit (also after an abort).
    if (lane == 0) {
      for (int s = 0; s < nst; ++s)
        if (issued[s]) mbar_drain(bar(full[s]), (issued[s] - 1) & 1, abort_flag, ptr.err);
    }
    __syncwarp();
  } else if (warp == 1 || warp == kPVIssuerWarp) {
    // ------------------------------------------------------------ MMA issuers
    // S = Q K^T and O += P V come from two warps. P of sub-tile g lives in S buffer g & 1,
    // so S(g) waits for P.V(g-2); P.V(g) waits for P(g) and V(g).
    if (lane == 0) {
      const bool is_s = warp == 1;
      uint32_t g = 0;
      int ii = 0;
      bool ok = true;
      for (int it = item_begin; it < item_end && ok; ++it, ++ii) {
        const Item I = load_item<kFused>(p, cp, ptr, ms, it);
        for (int j = 0; j < I.nsub && ok; ++j, ++g) {
          const uint32_t b = g & 1;
          if (is_s) {
            if (j == 0 && !(ok = mbar_wait(bar(ms.q_full), ii & 1, abort_flag, ptr.err))) break;
            const uint32_t st = g % kKStages;
            if (!(ok = mbar_wait(bar(ms.k_full[st]), (g / kKStages) & 1, abort_flag, ptr.err))) break;
            if (g >= 2 && !(ok = mbar_wait(bar(ms.pv_done[b]), ((g >> 1) - 1) & 1, abort_flag, ptr.err))) break;
            tc_fence_after();
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
              const uint64_t q0 = smem_desc(sbase + kOffQ + qd * kQQuarter, 16, 1024, kSw128);
              const uint64_t k0 = smem_desc(sbase + kOffK + st * kKVTile + qd * kKVQuarter, 16, 1024, kSw128);
#pragma unroll
              for (int k = 0; k < 4; ++k)  // 16 bf16 (32 bytes) of d per instruction
                mma_f16(tmem + kColS + b * kSub, q0 + ((k * 32) >> 4), k0 + ((k * 32) >> 4), kIdescS,
                        (qd | k) ? 1u : 0u);
            }
            mma_commit(bar(ms.s_full[b]));
            mma_commit(bar(ms.k_empty[st]));
            if (j == I.nsub - 1) mma_commit(bar(ms.q_free));
          } else {
            // the first P.V of an item overwrites O: the previous epilogue must be done
            if (j == 0 && ii >= 1 && !(ok = mbar_wait(bar(ms.o_free), (ii - 1) & 1, abort_flag, ptr.err))) break;
            if (!(ok = mbar_wait(bar(ms.p_full), g & 1, abort_flag, ptr.err))) break;
            const uint32_t st = g % kVStages;
            if (!(ok = mbar_wait(bar(ms.v_full[st]), (g / kVStages) & 1, abort_flag, ptr.err))) break;
            tc_fence_after();
            // V as one N = 256 MN-major operand: its four 128-byte d-quarters sit kKVQuarter
            // apart, 8-key row groups 1 KB apart; 16 keys (2 KB) per instruction
            const uint64_t v0 = smem_desc(sbase + kOffV + st * kKVTile, kKVQuarter, 1024, kSw128);
            const uint32_t p_cols = tmem + kColS + b * kSub;  // P of this sub-tile, in its S buffer
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts(tmem + kColO, p_cols + kk * 8, v0 + ((kk * 2048) >> 4), kIdescO,
                         (j == 0 && kk == 0) ? 0u : 1u);
            mma_commit(bar(ms.v_empty[st]));
            mma_commit(bar(ms.pv_done[b]));
            if (j == I.nsub - 1) mma_commit(bar(ms.o_ready));
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
    const int kh = sw >> 2;                // key half of the sub-tile this thread owns (0/1)
    const int row = q4 * 32 + lane;        // TMEM lane = row of the block
    const uint32_t lane_addr = (uint32_t)(q4 * 32) << 16;
    const int pair_bar = 1 + q4;           // named barrier of the two threads of each row
    bool bad = false;
    float m_ref = kMInit, l = 0.f;
    bool stalled = false;
    if (p.stall_test_ns) {  // failure-path test: a bounded wait on a barrier nothing arrives on
      int ok = 1;
      if (lane == 0) ok = mbar_wait(bar(ms.never), 0, abort_flag, ptr.err, p.stall_test_ns);
      stalled = __shfl_sync(0xffffffffu, ok, 0) == 0;
    }
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
      // 128 rows x 32 chunks of 8 bf16 (16 B); thread gi takes chunks gi + 256 k, k < 16
#pragma unroll
      for (int k0 = 0; k0 < 16; k0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = gi + (k0 + k) * kSoftThreads, r = c >> 5, ch = c & 31;
          v[k] = make_uint4(0, 0, 0, 0);
          if (r < I.nrows) {
            const RowMap m = map_row(I.row0 + r, p.G, I.kvh);
            v[k] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(ptr.q) +
                                                   (size_t)(I.q0 + m.t) * p.q_st + (size_t)m.h * p.q_sh + ch * 8);
          }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = gi + (k0 + k) * kSoftThreads, r = c >> 5, ch = c & 31;
          const int qd = ch >> 3, cc = ch & 7;
          *reinterpret_cast<uint4*>(smem + kOffQ + qd * kQQuarter + r * 128 + ((cc ^ (r & 7)) << 4)) = v[k];
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(bar(ms.q_full));
    };

    int ii = 0;
    uint32_t g = 0;
    const float c = p.score_scale_log2;
    if (item_end > item_begin) q_prep(load_item<kFused>(p, cp, ptr, ms, item_begin), 0);
    for (int it = item_begin; it < item_end; ++it, ++ii) {
      const Item I = load_item<kFused>(p, cp, ptr, ms, it);
      const int pi = ii & 1;
      named_barrier(9, kSoftThreads);  // q_prep's shared writes are visible
      const int lim = ms.lim[pi][row];
      const int min_lim = I.L - I.qn + map_row(I.row0, p.G, I.kvh).t;
      m_ref = kMInit;
      l = 0.f;
      const int kv_hi = I.kv_hi, key_begin = I.tile_begin * kTileKeys;
      const int hi_key = min(kv_hi - 1, lim);  // keys <= hi_key are visible to this row
      // A failed wait (timeout or abort) does not leave the loop: every later wait then
      // fails fast, so all softmax warps still pass the same barriers and finish.
      for (int j = 0; j < I.nsub; ++j, ++g) {
        const int b = g & 1;
        const int key0 = key_begin + j * kSub;
        const int kbase = key0 + kh * kHalfKeys;
        float t[kHalfKeys];
        if (!mbar_wait(bar(ms.s_full[b]), (g >> 1) & 1, abort_flag, ptr.err)) bad = true;
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kHalfKeys; k += 16) {
          float v[16];
          tmem_ld16(tmem + lane_addr + kColS + b * kSub + kh * kHalfKeys + k, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) t[k + i] = v[i];
        }
        tmem_wait_ld();
        // scaled scores, masked past the row's causal limit and the piece's end
        const bool need_mask = (key0 + kSub > kv_hi) || (key0 + kSub - 1 > min_lim);
#pragma unroll
        for (int i = 0; i < kHalfKeys; ++i) t[i] = (!need_mask || kbase + i <= hi_key) ? t[i] * c : -INFINITY;
        const float mx = extreme_of<true>(t);
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
        // P = 2^(s c - m + sigma), rounded to bf16, two keys per 32-bit column; row sums of
        // the rounded values (what P.V multiplies)
        uint32_t pk[kHalfKeys / 2];
        const float off = m_ref - kSigma;
        float ls = 0.f;
#pragma unroll
        for (int i = 0; i < kHalfKeys; i += 2) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(ex2(t[i] - off), ex2(t[i + 1] - off));
          pk[i / 2] = *reinterpret_cast<const uint32_t*>(&h);
          const float2 f = __bfloat1622float2(h);
          ls += f.x + f.y;
        }
        l += ls;
        // tcgen05.ld/st are warp-collective: a warp rescales if any of its rows must; lanes
        // whose row keeps its reference multiply by 1. O may only be touched once the
        // previous sub-tile's P.V has completed; otherwise that wait comes after publishing P.
        const bool warp_rescale = __any_sync(0xffffffffu, rescale && j > 0);
        if (warp_rescale) {
          if (g >= 1 && !mbar_wait(bar(ms.pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort_flag, ptr.err)) bad = true;
          tc_fence_after();
          if (!(rescale && j > 0)) alpha = 1.f;
#pragma unroll 1
          for (int k = 0; k < 128; k += 16) {  // this thread's half of its O row: d-half kh
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
        if (key0 + kSub > kv_hi) {
          // keys past the piece's end: their V rows (stale or NaN slots) become zeros; thread
          // (kh, row < 64) zeroes d-quarters 2 kh and 2 kh + 1 of key `row`
          const uint32_t st = g % kVStages;
          if (!mbar_wait(bar(ms.v_full[st]), (g / kVStages) & 1, abort_flag, ptr.err)) bad = true;
          if (row < kSub && key0 + row >= kv_hi) {
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
              uint4* dst = reinterpret_cast<uint4*>(smem + kOffV + st * kKVTile + (2 * kh + qq) * kKVQuarter + row * 128);
#pragma unroll
              for (int i = 0; i < 8; ++i) dst[i] = z;
            }
          }
        }
        // P into TMEM over this sub-tile's S: row `row`, keys 32 kh .. 32 kh + 31 -> columns
        // 16 kh .. 16 kh + 15
        tmem_st16u(tmem + lane_addr + kColS + b * kSub + kh * (kPCols / 2), pk);
        tmem_wait_st();
        fence_proxy_async_smem();  // zeroed V rows, if any
        tc_fence_before();
        mbar_arrive(bar(ms.p_full));
        // P.V(g-1) has a barrier of its own (its S buffer's), whose next phase needs P(g+1):
        // the wait cannot mistake a later phase for this one, however late it runs.
        if (!warp_rescale && g >= 1 &&
            !mbar_wait(bar(ms.pv_done[(g - 1) & 1]), ((g - 1) >> 1) & 1, abort_flag, ptr.err))
          bad = true;
      }
      if (it + 1 < item_end) q_prep(load_item<kFused>(p, cp, ptr, ms, it + 1), ii + 1);

      // ---------------------------------------------------------- epilogue
      if (!mbar_wait(bar(ms.o_ready), ii & 1, abort_flag, ptr.err)) bad = true;
      tc_fence_after();
      ms.lsum[kh][row] = l;
      named_barrier(pair_bar, 64);
      const float lr = l + ms.lsum[kh ^ 1][row];
      const bool split = I.nsplit > 1;
      const int slot = I.slot_base + I.split;
      const bool valid = row < I.nrows;
      // a split piece's partial stays unnormalised by v_descale (applied by the merge)
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

int launch_bf16_tc(const Problem& p, const Pointers& ptr, const ClassPlan& cp, const pg_tensor* k,
                   const pg_tensor* v, cudaStream_t stream, bool dependent, bool self_planned) {
  if (p.kv_is_fp8 || p.q_is_fp8 || p.q_cast) return 0;
  CUtensorMap tk, tv;
  if (!make_cache_tmap(&tk, k, p.P) || !make_cache_tmap(&tv, v, p.P)) return -1;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t e;
  auto kern = self_planned ? bf16_tc_kernel<true> : bf16_tc_kernel<false>;
  const int which = self_planned ? 2 : 1;
  if (dev >= 0 && dev < 64 && !(attr_done[dev] & which)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) {
      char buf[160];
      snprintf(buf, sizeof buf, "cudaFuncSetAttribute(bf16): %s", cudaGetErrorString(e));
      set_tc_error(buf);
      return -1;
    }
    attr_done[dev] |= which;
  }
  e = launch_pdl(dependent, kern, cp.num_ctas, kThreads, kSmemBytes, stream, tk, tv, p, ptr, cp);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) {
    char buf[160];
    snprintf(buf, sizeof buf, "bf16 kernel launch: %s", cudaGetErrorString(e));
    set_tc_error(buf);
    return -1;
  }
  return 1;
}

}  // namespace pgqa
