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
#include "common.cuh"
#include "plan.cuh"

namespace pgqa {

namespace {

constexpr int kPlanThreads = 1024;

// Block-wide exclusive scan of one value per thread (1024 threads). Returns the
// exclusive prefix; *total receives the sum.
__device__ long long block_exclusive_scan(long long v, long long* total) {
  __shared__ long long warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = warp_sums[lane];
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

// CTA that owns unit u when U units are cut into C ranges [floor(c*U/C), floor((c+1)*U/C)).
__device__ __forceinline__ int cta_of(long long u, long long U, int C) {
  return (int)(((u + 1) * C + U - 1) / U) - 1;
}

__device__ __forceinline__ long long range_begin(int c, long long U, int C) {
  return (long long)c * U / C;
}

// Index of the block whose tile range contains unit u (tile_off is non-decreasing).
__device__ int find_block(const RowBlock* b, int n, long long u) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (b[mid].tile_off <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace

__global__ void __launch_bounds__(kPlanThreads, 1)
plan_kernel(Problem p, Pointers ptr, ClassPlan c0, ClassPlan c1) {
  __shared__ long long s_total;
  __shared__ int s_overflow;
  ClassPlan plans[2] = {c0, c1};
  // The attention kernels are launched as programmatic dependents: let them start their
  // prologue now; they wait for this grid's completion before reading the plan.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    s_overflow = 0;
    if (p.num_seqs > 0 && (ptr.qsl[0] != 0 || ptr.qsl[p.num_seqs] != p.T)) atomicOr(ptr.err, kErrBounds);
  }

  // Rows of invalid sequences are zeroed and flagged; they get no blocks.
  for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
    SeqInfo si = seq_info(p, ptr, s);
    if (!si.ok) {
      atomicOr(ptr.err, kErrBounds);
      int q0 = max(0, si.q0), q1 = min(p.T, max(q0, si.q0 + max(si.qn, 0)));
      uint16_t* o = (uint16_t*)ptr.out;
      for (int t = q0; t < q1; ++t)
        for (int h = 0; h < p.Hq; ++h)
          for (int d = 0; d < kHeadDim; ++d) o[t * p.o_st + h * p.o_sh + d] = 0;
    }
  }

  for (int cls = 0; cls < kNumClasses; ++cls) {
    ClassPlan& cp = plans[cls];
    // ---- blocks: per-sequence counts, scan, then fill
    long long base = 0;
    for (int s0 = 0; s0 < p.num_seqs; s0 += blockDim.x) {
      int s = s0 + threadIdx.x;
      SeqInfo si = {0, 0, 0, 0};
      int nb = 0;
      if (s < p.num_seqs) {
        si = seq_info(p, ptr, s);
        nb = blocks_per_head(si, p.G, cls) * p.Hkv;
      }
      long long pre = block_exclusive_scan(nb, &s_total) + base;
      // The warp fills the blocks of its 32 sequences together: one lane per block.
      const int rb_rows = cls == 0 ? kVerifyRows : kPrefillRows;
      const int lane = threadIdx.x & 31;
      for (int j = 0; j < 32; ++j) {
        const int nb_j = __shfl_sync(0xffffffffu, nb, j);
        if (nb_j == 0) continue;
        const long long pre_j = __shfl_sync(0xffffffffu, pre, j);
        const int qn_j = __shfl_sync(0xffffffffu, si.qn, j);
        const int L_j = __shfl_sync(0xffffffffu, si.L, j);
        const int s_j = s0 + (threadIdx.x & ~31) + j;
        const int per_head = nb_j / p.Hkv;
        const int rows_total = qn_j * p.G;
        for (int i = lane; i < nb_j; i += 32) {
          const long long bi = pre_j + i;
          if (bi >= cp.max_blocks) {
            s_overflow = 1;
            break;
          }
          const int kvh = i / per_head, rb = i % per_head;
          RowBlock b;
          b.seq = s_j;
          b.kvh = kvh;
          b.row0 = rb * rb_rows;
          b.nrows = min(rb_rows, rows_total - b.row0);
          const int t_last = (b.row0 + b.nrows - 1) / p.G;
          b.kv_end = L_j - qn_j + t_last + 1;
          b.tiles = (b.kv_end + kTileKeys - 1) / kTileKeys;
          b.tile_off = 0;
          b.nsplit = 1;
          b.slot_base = 0;
          cp.blocks[bi] = b;
        }
      }
      base += s_total;
    }
    __syncthreads();
    const int nblocks = (int)min(base, (long long)cp.max_blocks);

    // ---- tile prefix over blocks
    long long tbase = 0;
    for (int b0 = 0; b0 < nblocks; b0 += blockDim.x) {
      int b = b0 + threadIdx.x;
      long long t = b < nblocks ? cp.blocks[b].tiles : 0;
      long long pre = block_exclusive_scan(t, &s_total) + tbase;
      if (b < nblocks) cp.blocks[b].tile_off = pre;
      tbase += s_total;
    }
    __syncthreads();
    const long long U = tbase;
    // Cut into at most U ranges so that every range is non-empty: a block then has
    // exactly one piece per range it intersects, and its split count is exact.
    const int C = (int)min((long long)cp.num_ctas, U);

    // ---- per-block split count and partial slots
    int slot_base = 0;
    for (int b0 = 0; b0 < nblocks; b0 += blockDim.x) {
      int b = b0 + threadIdx.x;
      int ns = 0;
      if (b < nblocks) {
        RowBlock& rb = cp.blocks[b];
        int c_first = cta_of(rb.tile_off, U, C);
        int c_last = cta_of(rb.tile_off + rb.tiles - 1, U, C);
        rb.nsplit = c_last - c_first + 1;
        ns = rb.nsplit > 1 ? rb.nsplit : 0;
        cp.counters[b] = 0;
      }
      long long pre = block_exclusive_scan(ns, &s_total) + slot_base;
      if (b < nblocks) {
        cp.blocks[b].slot_base = (int)pre;
        if (ns > 0 && pre + ns > cp.max_slots) s_overflow = 1;
      }
      slot_base += (int)s_total;
    }
    __syncthreads();

    // ---- items: count per CTA, scan, fill
    long long ibase = 0;
    for (int c0i = 0; c0i < cp.num_ctas; c0i += blockDim.x) {
      int c = c0i + threadIdx.x;
      int cnt = 0, bfirst = 0;
      long long u0 = 0, u1 = 0;
      if (c < C && U > 0) {
        u0 = range_begin(c, U, C);
        u1 = range_begin(c + 1, U, C);
        if (u1 > u0) {
          bfirst = find_block(cp.blocks, nblocks, u0);
          int blast = find_block(cp.blocks, nblocks, u1 - 1);
          cnt = blast - bfirst + 1;
        }
      }
      long long pre = block_exclusive_scan(cnt, &s_total) + ibase;
      if (c < cp.num_ctas) {
        cp.cta_item_begin[c] = (int)min(pre, (long long)cp.max_items);
        for (int i = 0; i < cnt; ++i) {
          long long ii = pre + i;
          if (ii >= cp.max_items) { s_overflow = 1; break; }
          const int b = bfirst + i;
          const RowBlock& rb = cp.blocks[b];
          long long lo = max(u0, rb.tile_off), hi = min(u1, rb.tile_off + rb.tiles);
          WorkItem it;
          it.block = b;
          it.tile_begin = (int)(lo - rb.tile_off);
          it.tile_end = (int)(hi - rb.tile_off);
          it.split = cta_of(lo, U, C) - cta_of(rb.tile_off, U, C);
          cp.items[ii] = it;
        }
      }
      ibase += s_total;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      cp.cta_item_begin[cp.num_ctas] = (int)min(ibase, (long long)cp.max_items);
      *cp.n_blocks = nblocks;
      *cp.n_items = (int)min(ibase, (long long)cp.max_items);
      *cp.total_tiles = U;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0 && s_overflow) {
    // Host-side bounds make this unreachable; flag it rather than run a partial plan.
    atomicOr(ptr.err, kErrBounds);
    for (int cls = 0; cls < kNumClasses; ++cls) {
      *plans[cls].n_items = 0;
      for (int c = 0; c <= plans[cls].num_ctas; ++c) plans[cls].cta_item_begin[c] = 0;
    }
  }
}

cudaError_t launch_plan(const Problem& p, const Pointers& ptr, const ClassPlan& v,
                        const ClassPlan& f, cudaStream_t stream) {
  plan_kernel<<<1, kPlanThreads, 0, stream>>>(p, ptr, v, f);
  return cudaGetLastError();
}

}  // namespace pgqa
