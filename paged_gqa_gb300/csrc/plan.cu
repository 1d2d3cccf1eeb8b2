// plan.cu -- device-side launch plan (one CTA).
//
// Reads query_start_loc and seq_lens on the device (the host never syncs on them),
// classifies each sequence (verify if q_len*G <= 64 rows, else prefill), builds the
// row blocks, and cuts the concatenated key tiles of each class into one contiguous
// range per persistent CTA. The pages describe the same decision as a host-side gate
// on max_q_len / kv length and a launch-profile ladder keyed on program count
// ("Optimize Qwen3.5 MTP unified attention on gfx950": dispatch gate and segment
// count chosen from CU parallelism and per-segment KV work; "Tune sparse GQA prefill
// profile": the >512-program profile branch). Here the split is exact per call.
#include <cstddef>

#include "common.cuh"
#include "plan.cuh"
#include "tc_kernels.cuh"

namespace pgqa {

namespace {

constexpr int kPlanThreads = 1024;

// Block-wide exclusive scan of one value per thread (any multiple of 32 threads up to 1024).
// Returns the exclusive prefix; *total receives the sum.
__device__ long long block_exclusive_scan(long long v, long long* total) {
  __shared__ long long warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  long long before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

struct SeqInfo {
  int q0, qn, L, ok;
};

__device__ SeqInfo seq_info(const Problem& p, const Pointers& ptr, int s) {
  SeqInfo r;
  r.q0 = ptr.qsl[s];
  int q1 = ptr.qsl[s + 1];
  r.qn = q1 - r.q0;
  r.L = ptr.seq_lens[s];
  r.ok = (r.qn >= 0) && (r.q0 >= 0) && (q1 <= p.T) && (r.qn <= r.L) &&
         ((long long)r.L <= (long long)p.W * p.P);
  return r;
}

// Number of row blocks sequence s contributes to class c (per kv head).
__device__ int blocks_per_head(const SeqInfo& si, int G, int cls) {
  if (!si.ok || si.qn == 0) return 0;
  const long long rows = (long long)si.qn * G;
  const bool verify = rows <= kVerifyRows;
  if (cls == 0) return verify ? 1 : 0;
  return verify ? 0 : (int)((rows + kPrefillRows - 1) / kPrefillRows);
}

}  // namespace

// Shared-memory caches: sequence info, per-sequence block prefixes and per-block tile
// counts / offsets for the first kSeqCache sequences and kBlockCache blocks of a class
// (beyond that, global memory). Later phases read them instead of re-reading what this
// CTA wrote to global memory, which keeps the plan to a few dependent global accesses.
constexpr int kSeqCache = 2048;
constexpr int kBlockCache = 12288;
constexpr int kMaxCtas = 1024;
// fixed_cost(cls) (common.cuh), what starting a row block costs a CTA in key tiles: per-CTA
// timestamps on the MTP verify batch put an item beyond a CTA's first at ~9 us, ~6.5 of its
// 1.42 us tiles; 6 ended the slowest CTA ~1 us earlier than 5 (8 no better); prefill blocks
// have longer tiles.
constexpr size_t kPlanSmem = sizeof(int4) * kSeqCache + sizeof(int) * (kSeqCache + 1) +
                             sizeof(long long) * kBlockCache + sizeof(int) * kBlockCache +
                             sizeof(int) * (kMaxCtas + 1);

struct PlanSmem {
  int4* seq;          // q0, qn, L, ok
  int* seq_pre;       // first block of each cached sequence (class being planned)
  long long* off;     // tile_off
  int* tiles;         // tiles
  int* bfirst;        // first block of CTA range c
  long long* total;   // scan total
  int* overflow;
};

__device__ __forceinline__ SeqInfo seq_of(const Problem& p, const Pointers& ptr, const PlanSmem& sm, int s) {
  if (s < kSeqCache) {
    const int4 v = sm.seq[s];
    return SeqInfo{v.x, v.y, v.z, v.w};
  }
  return seq_info(p, ptr, s);
}

// Block i (0-based within sequence s_j, kv heads major) of class cls, written as vectors.
__device__ __forceinline__ int write_block(const Problem& p, const ClassPlan& cp, int cls, long long bi, int s_j,
                                          int i, int nb_j, int qn_j, int L_j) {
  const int rb_rows = cls == 0 ? kVerifyRows : kPrefillRows;
  const int per_head = nb_j / p.Hkv;
  const int kvh = i / per_head, rb = i - kvh * per_head;
  const int row0 = rb * rb_rows;
  const int nrows = min(rb_rows, qn_j * p.G - row0);
  const int t_last = (row0 + nrows - 1) / p.G;
  const int kv_end = L_j - qn_j + t_last + 1;
  const int tiles = (kv_end + kTileKeys - 1) / kTileKeys;
  // RowBlocks are 40 bytes: 8-byte aligned, so at most 8-byte vectors
  int* d = reinterpret_cast<int*>(cp.blocks + bi);
  static_assert(sizeof(RowBlock) == 40 && offsetof(RowBlock, tile_off) == 24 && alignof(RowBlock) == 8,
                "RowBlock layout");
  *reinterpret_cast<int2*>(d) = make_int2(s_j, kvh);
  *reinterpret_cast<int2*>(d + 2) = make_int2(row0, nrows);
  *reinterpret_cast<int2*>(d + 4) = make_int2(kv_end, tiles);
  *reinterpret_cast<long long*>(d + 6) = 0;
  *reinterpret_cast<int2*>(d + 8) = make_int2(1, 0);
  return tiles;
}

__device__ __forceinline__ void plan_class(const Problem& p, const Pointers& ptr, const ClassPlan& cp, int cls,
                                           const PlanSmem& sm) {
  auto tiles_of = [&](int b) -> int { return b < kBlockCache ? sm.tiles[b] : cp.blocks[b].tiles; };
  auto off_of = [&](int b) -> long long { return b < kBlockCache ? sm.off[b] : cp.blocks[b].tile_off; };
  const int ncached = min(p.num_seqs, kSeqCache);
  // ---- blocks: per-sequence counts and scan. Cached sequences record their first block
  // (filled below by all threads at once); the others fill their blocks here, a warp at a
  // time (one lane per block).
  long long base = 0;
  for (int s0 = 0; s0 < p.num_seqs; s0 += blockDim.x) {
    const int s = s0 + threadIdx.x;
    SeqInfo si = {0, 0, 0, 0};
    int nb = 0;
    if (s < p.num_seqs) {
      si = seq_of(p, ptr, sm, s);
      nb = blocks_per_head(si, p.G, cls) * p.Hkv;
    }
    const long long pre = block_exclusive_scan(nb, sm.total) + base;
    if (s < ncached) sm.seq_pre[s] = (int)min(pre, (long long)cp.max_blocks);
    if (s == ncached - 1) sm.seq_pre[ncached] = (int)min(pre + nb, (long long)cp.max_blocks);
    if (s0 + (int)blockDim.x > kSeqCache) {
      const int lane = threadIdx.x & 31;
      for (int j = 0; j < 32; ++j) {
        const int nb_j = __shfl_sync(0xffffffffu, nb, j);
        const long long pre_j = __shfl_sync(0xffffffffu, pre, j);
        const int qn_j = __shfl_sync(0xffffffffu, si.qn, j);
        const int L_j = __shfl_sync(0xffffffffu, si.L, j);
        const int s_j = s0 + (threadIdx.x & ~31) + j;
        if (nb_j == 0 || s_j < kSeqCache) continue;
        for (int i = lane; i < nb_j; i += 32) {
          const long long bi = pre_j + i;
          if (bi >= cp.max_blocks) {
            *sm.overflow = 1;
            break;
          }
          const int t = write_block(p, cp, cls, bi, s_j, i, nb_j, qn_j, L_j);
          if (bi < kBlockCache) sm.tiles[bi] = t;
        }
      }
    }
    base += *sm.total;
    __syncthreads();  // the scan total is reused
  }
  if (base > cp.max_blocks && threadIdx.x == 0) *sm.overflow = 1;
  const int nblocks = (int)min(base, (long long)cp.max_blocks);
  // blocks of cached sequences: every thread a block; its sequence by binary search
  const int ncb = ncached > 0 ? sm.seq_pre[ncached] : 0;
  for (int bi = threadIdx.x; bi < ncb; bi += blockDim.x) {
    int lo = 0, hi = ncached - 1;  // largest s with seq_pre[s] <= bi
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sm.seq_pre[mid] <= bi) lo = mid; else hi = mid - 1;
    }
    const SeqInfo si = seq_of(p, ptr, sm, lo);
    const int nb_s = blocks_per_head(si, p.G, cls) * p.Hkv;
    const int t = write_block(p, cp, cls, bi, lo, bi - sm.seq_pre[lo], nb_s, si.qn, si.L);
    if (bi < kBlockCache) sm.tiles[bi] = t;
  }
  __syncthreads();

  // ---- unit prefix over blocks. A block spans fixed_cost(cls) units for what starting it
  // costs a CTA (loading Q, the epilogue, a merge) and then one unit per key tile; the
  // units are cut into equal CTA ranges, so a CTA that starts blocks gets fewer tiles.
  const int E = fixed_cost(cls);
  long long tbase = 0;
  for (int b0 = 0; b0 < nblocks; b0 += blockDim.x) {
    const int b = b0 + threadIdx.x;
    const long long t = b < nblocks ? tiles_of(b) + E : 0;
    const long long pre = block_exclusive_scan(t, sm.total) + tbase;
    if (b < nblocks) {
      cp.blocks[b].tile_off = pre;
      if (b < kBlockCache) sm.off[b] = pre;
    }
    tbase += *sm.total;
    __syncthreads();
  }
  const long long U = tbase;
  // At most U ranges, none empty in units (a range may hold no tile: that CTA has no item).
  const int C = cut_ctas(U, cp.num_ctas);

  // ---- per-block split count and partial slots (split_slot_base: no scan); block containing
  // the start of each range
  for (int b = threadIdx.x; b < nblocks; b += blockDim.x) {
    const long long span = off_of(b), real = span + E;  // tiles occupy [real, real + tiles)
    const int tiles = tiles_of(b);
    const int c0 = cta_of(real, U, C);
    const int ns = cta_of(real + tiles - 1, U, C) - c0 + 1;  // pieces: ranges meeting the tiles
    const int slot = split_slot_base(c0, range_begin(c0, U, C) < span);
    *reinterpret_cast<int2*>(reinterpret_cast<int*>(cp.blocks + b) + 8) = make_int2(ns, slot);
    if (ns > 1 && slot + ns > cp.max_slots) *sm.overflow = 1;
    // CTA c's range starts inside block b's span for c in (c_first, c_last], and at its
    // first unit when the range boundary falls exactly there
    const int c_first = cta_of(span, U, C), c_last = cta_of(span + E + tiles - 1, U, C);
    if (range_begin(c_first, U, C) == span) sm.bfirst[c_first] = b;
    for (int c = c_first + 1; c <= c_last; ++c) sm.bfirst[c] = b;
  }
  __syncthreads();

  // ---- items: count per CTA, scan, fill. The items of range [u0, u1) are the blocks whose
  // tiles meet it: from the block whose span holds u0 to the block whose span holds
  // u1 - 1, less that last one if u1 - 1 falls in its fixed-cost units.
  long long ibase = 0;
  for (int c0i = 0; c0i < cp.num_ctas; c0i += blockDim.x) {
    const int c = c0i + threadIdx.x;
    int cnt = 0, bfirst = 0;
    long long u0 = 0, u1 = 0;
    if (c < C) {
      u0 = range_begin(c, U, C);
      u1 = range_begin(c + 1, U, C);
      bfirst = sm.bfirst[c];
      int blast = nblocks - 1;
      if (c + 1 < C) {
        const int bn = sm.bfirst[c + 1];
        blast = off_of(bn) == u1 ? bn - 1 : bn;
      }
      if (u1 - 1 < off_of(blast) + E) --blast;
      cnt = max(0, blast - bfirst + 1);
    }
    const long long pre = block_exclusive_scan(cnt, sm.total) + ibase;
    if (c < cp.num_ctas) {
      cp.cta_item_begin[c] = (int)min(pre, (long long)cp.max_items);
      for (int i = 0; i < cnt; ++i) {
        const long long ii = pre + i;
        if (ii >= cp.max_items) {
          *sm.overflow = 1;
          break;
        }
        const int b = bfirst + i;
        const long long real = off_of(b) + E;
        const long long lo = max(u0, real), hi = min(u1, real + tiles_of(b));
        static_assert(sizeof(WorkItem) == 16, "WorkItem layout");
        *reinterpret_cast<int4*>(cp.items + ii) =
            make_int4(b, (int)(lo - real), (int)(hi - real), cta_of(lo, U, C) - cta_of(real, U, C));
      }
    }
    ibase += *sm.total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    cp.cta_item_begin[cp.num_ctas] = (int)min(ibase, (long long)cp.max_items);
    *cp.n_blocks = nblocks;
    *cp.n_items = (int)min(ibase, (long long)cp.max_items);
    *cp.total_tiles = U;
  }
  __syncthreads();
}

// A class without blocks: no items for any CTA.
__device__ __forceinline__ void empty_class(const ClassPlan& cp) {
  for (int c = threadIdx.x; c <= cp.num_ctas; c += blockDim.x) cp.cta_item_begin[c] = 0;
  if (threadIdx.x == 0) {
    *cp.n_blocks = 0;
    *cp.n_items = 0;
    *cp.total_tiles = 0;
  }
}

// With plan_verify false the verify class is planned by its own kernel (Problem::fused_verify),
// which runs first: this kernel then plans prefill only, and advances the epoch word once
// that kernel has completed.
__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(Problem p, Pointers ptr, ClassPlan c0, ClassPlan c1, int plan_verify) {
  __shared__ long long s_total;
  __shared__ int s_overflow;
  extern __shared__ __align__(16) unsigned char plan_smem[];
  PlanSmem sm;
  sm.seq = reinterpret_cast<int4*>(plan_smem);
  sm.off = reinterpret_cast<long long*>(sm.seq + kSeqCache);
  sm.tiles = reinterpret_cast<int*>(sm.off + kBlockCache);
  sm.seq_pre = sm.tiles + kBlockCache;
  sm.bfirst = sm.seq_pre + kSeqCache + 1;
  sm.total = &s_total;
  sm.overflow = &s_overflow;
  // The attention kernels may be launched as programmatic dependents: let them start their
  // prologue now; they wait for this grid's completion before reading the plan.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    s_overflow = 0;
    if (p.num_seqs > 0 && (ptr.qsl[0] != 0 || ptr.qsl[p.num_seqs] != p.T)) atomicOr(ptr.err, kErrBounds);
  }
  // Sequence info, once. Rows of invalid sequences are zeroed and flagged; they get no blocks.
  // Which classes have any block at all: an empty class gets an empty plan at once.
  int has_v = 0, has_p = 0;
  for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
    SeqInfo si = seq_info(p, ptr, s);
    if (s < kSeqCache) sm.seq[s] = make_int4(si.q0, si.qn, si.L, si.ok);
    has_v |= blocks_per_head(si, p.G, 0) > 0;
    has_p |= blocks_per_head(si, p.G, 1) > 0;
    if (!si.ok) {
      atomicOr(ptr.err, kErrBounds);
      int q0 = max(0, si.q0), q1 = min(p.T, max(q0, si.q0 + max(si.qn, 0)));
      uint16_t* o = (uint16_t*)ptr.out;
      for (int t = q0; t < q1; ++t)
        for (int h = 0; h < p.Hq; ++h)
          for (int d = 0; d < kHeadDim; ++d) o[t * p.o_st + h * p.o_sh + d] = 0;
    }
  }
  has_v = __syncthreads_or(has_v) && plan_verify;
  has_p = __syncthreads_or(has_p);
  if (plan_verify) {
    if (has_v) plan_class(p, ptr, c0, 0, sm); else empty_class(c0);
  }
  if (has_p) plan_class(p, ptr, c1, 1, sm); else empty_class(c1);
  if (threadIdx.x == 0 && s_overflow) {
    // Host-side bounds make this unreachable; flag it rather than run a partial plan.
    atomicOr(ptr.err, kErrBounds);
    if (plan_verify) {
      *c0.n_items = 0;
      for (int c = 0; c <= c0.num_ctas; ++c) c0.cta_item_begin[c] = 0;
    }
    *c1.n_items = 0;
    for (int c = 0; c <= c1.num_ctas; ++c) c1.cta_item_begin[c] = 0;
  }
  // New split-counter tag for the next call: every kernel of this call that reads the epoch
  // word reads it after this grid completes, or (a self-planned verify kernel, which this grid
  // may follow as a programmatic dependent) has completed before this point.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) *c0.epoch += 1ull;
}

cudaError_t launch_plan(const Problem& p, const Pointers& ptr, const ClassPlan& v,
                        const ClassPlan& f, bool plan_verify, bool dependent, cudaStream_t stream) {
  if (v.num_ctas > kMaxCtas || f.num_ctas > kMaxCtas) return cudaErrorInvalidConfiguration;
  static int attr_done[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPlanSmem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = 1;
  }
  // A small problem (up to 256 sequences and row blocks per class, 256 CTAs) is planned by
  // 256 threads: the plan is a chain of block-wide scans, and each barrier over 8 warps is
  // cheaper than over 32. Larger problems take 1024 threads.
  const long long rows = (long long)p.T * p.G;
  const long long blocks = (long long)p.Hkv * ((rows + kPrefillRows - 1) / kPrefillRows + p.num_seqs);
  const int threads = (p.num_seqs <= 256 && blocks <= 256 && v.num_ctas <= 255 && f.num_ctas <= 255) ? 256 : kPlanThreads;
  cudaError_t e = launch_pdl(dependent, plan_kernel, 1, threads, kPlanSmem, stream, p, ptr, v, f, plan_verify ? 1 : 0);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pgqa
