// self_plan.cuh -- a verify-class kernel that plans its own class (Problem::fused_verify).
//
// Every CTA works out the plan kernel's cut of the verify blocks (one per verify sequence
// and kv head, in sequence order, each fixed_cost(0) units and then its ceil(L / 128) key
// tiles) from query_start_loc and seq_lens, and keeps its own items in shared memory;
// nothing is written to global memory. The host guarantees num_seqs * Hkv <=
// kFusedMaxBlocks, U < 2^31 and key tiles per block < 2^16. The split-KV decision is then
// per call and exact with no plan kernel on the call's critical path ("Optimize Qwen3.5 MTP
// unified attention on gfx950": segments chosen from CU parallelism and per-segment KV work).
//
// The cut in 32-bit arithmetic: with U = q C + r, range c starts at floor(c U / C) =
// c q + floor(c r / C) (c r < 2^20), and the range holding unit u comes from a float
// estimate of u C / U (off by at most one) and a correction.
#pragma once
#include "common.cuh"

namespace pgqa {
namespace self_plan {

constexpr int kE = fixed_cost(0);

struct Cut {
  int U, C, q, r;
};
__device__ __forceinline__ Cut make_cut(int U, int C) { return Cut{U, C, U / C, U % C}; }
__device__ __forceinline__ int cut_begin(const Cut& k, int c) {
  return c * k.q + (int)(((unsigned)c * (unsigned)k.r) / (unsigned)k.C);
}
__device__ __forceinline__ int cut_cta(const Cut& k, int u) {
  int c = (int)((float)u * (float)k.C / (float)k.U);
  c = min(max(c, 0), k.C - 1);
  while (c > 0 && cut_begin(k, c) > u) --c;
  while (c + 1 < k.C && cut_begin(k, c + 1) <= u) ++c;
  return c;
}

// Scratch of the prologue (20 KB), in shared memory no copy has touched yet.
struct Scratch {
  long long v[kFusedMaxBlocks];  // per sequence: (units << 16) | 1 for a verify sequence, else 0
  int tiles[kFusedMaxBlocks];    // per sequence: key tiles of each of its blocks
  int4 seq[kFusedMaxBlocks];     // per sequence: {first token, q_len, L, 0} as read
  int fv_seq[kFusedMaxBlocks];   // per verify sequence j: its index,
  int fv_off[kFusedMaxBlocks];   // the first unit of its blocks,
  int fv_tiles[kFusedMaxBlocks]; // its tiles per block
};

// Step 1, every thread of the CTA: the sequences' reads and units, staged in the scratch.
__device__ __forceinline__ void load(const Problem& p, const Pointers& ptr, Scratch& fs) {
  for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
    const int q0 = ptr.qsl[s], q1 = ptr.qsl[s + 1], L = ptr.seq_lens[s];
    const int qn = q1 - q0;
    long long v = 0;
    int tiles = 0;
    // the plan kernel's validity test; invalid sequences are flagged and zeroed there
    const bool ok = qn >= 0 && q0 >= 0 && q1 <= p.T && qn <= L && (long long)L <= (long long)p.W * p.P;
    if (ok && qn > 0 && (long long)qn * p.G <= kVerifyRows) {
      tiles = (L + kTileKeys - 1) / kTileKeys;
      v = ((long long)p.Hkv * (tiles + kE) << 16) | 1;
    }
    fs.v[s] = v;
    fs.tiles[s] = tiles;
    fs.seq[s] = make_int4(q0, qn, L, 0);
  }
}

// Step 2, one warp, after a CTA barrier: the scan over sequences (each lane a contiguous
// run of them), this CTA's range and items. Packed item (fitem, at most kFusedMaxBlocks):
// x = block, y = sequence, z = first tile | tiles << 16, w = piece index | pieces << 15 |
// (1 << 30 if the block's first CTA's range starts in an earlier block); fseq gets the
// item's sequence {first token, q_len, L, 0}, so that no item load reads global memory.
// *fcount gets the number of items.
__device__ __forceinline__ void plan_warp(const Problem& p, Scratch& fs, int num_ctas, int lane, int4* fitem,
                                          int4* fseq, int* fcount) {
  const int n = p.num_seqs;
  const int per = (n + 31) / 32;
  const int s0 = lane * per, s1 = min(n, s0 + per);
  long long sum = 0;
  for (int s = s0; s < s1; ++s) sum += fs.v[s];
  long long x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  const long long total = __shfl_sync(0xffffffffu, x, 31);
  const int U = (int)(total >> 16);
  const int C = cut_ctas(U, num_ctas);
  const int c = blockIdx.x;
  if (c >= C) {  // warp-uniform: no range (C = 0: no verify block at all)
    if (lane == 0) *fcount = 0;
    return;
  }
  const Cut k = make_cut(U, C);
  const int u0 = cut_begin(k, c), u1 = cut_begin(k, c + 1);
  // the blocks holding u0 and u1 - 1: found by the lane whose run of sequences holds them
  int ib = -1, il = -1;
  long long pre = x - sum;
  for (int s = s0; s < s1; ++s) {
    const long long v = fs.v[s];
    if (v) {
      const int j = (int)(pre & 0xffff), off = (int)(pre >> 16), units = (int)(v >> 16);
      const int tiles = fs.tiles[s], span = tiles + kE;
      fs.fv_seq[j] = s;
      fs.fv_off[j] = off;
      fs.fv_tiles[j] = tiles;
      if (u0 >= off && u0 < off + units) ib = j * p.Hkv + (u0 - off) / span;
      if (u1 - 1 >= off && u1 - 1 < off + units) {
        const int kvh = (u1 - 1 - off) / span;
        // u1 - 1 in that block's fixed-cost units: none of its tiles is in this range
        il = j * p.Hkv + kvh - (u1 - 1 < off + kvh * span + kE ? 1 : 0);
      }
    }
    pre += v;
  }
  ib = __reduce_max_sync(0xffffffffu, ib);
  il = __reduce_max_sync(0xffffffffu, il);
  __syncwarp();  // the per-verify-sequence arrays are complete
  const int cnt = max(0, il - ib + 1);
  for (int t = lane; t < cnt; t += 32) {
    const int b = ib + t;
    const int j = b / p.Hkv, kvh = b - j * p.Hkv;
    const int tiles = fs.fv_tiles[j];
    const int off = fs.fv_off[j] + kvh * (tiles + kE), real = off + kE;
    const int lo = max(u0, real), hi = min(u1, real + tiles);
    const int c0 = cut_cta(k, real);
    const int nsplit = cut_cta(k, real + tiles - 1) - c0 + 1;
    const int later = cut_begin(k, c0) < off ? 1 : 0;
    fitem[t] = make_int4(b, fs.fv_seq[j], (lo - real) | ((hi - lo) << 16), (c - c0) | (nsplit << 15) | (later << 30));
    fseq[t] = fs.seq[fs.fv_seq[j]];
  }
  if (lane == 0) *fcount = cnt;
}

// A packed item, unpacked; the caller adds its sequence's record (fseq).
struct Piece {
  int block, seq, kvh, tile_begin, ntiles, split, nsplit, slot_base;
};
__device__ __forceinline__ Piece unpack(const Problem& p, int4 f) {
  Piece r;
  r.block = f.x;
  r.seq = f.y;
  r.kvh = f.x % p.Hkv;
  r.tile_begin = f.z & 0xffff;
  r.ntiles = (int)((unsigned)f.z >> 16);
  r.split = f.w & 0x7fff;
  r.nsplit = (f.w >> 15) & 0x7fff;
  r.slot_base = split_slot_base((int)blockIdx.x - r.split, (f.w >> 30) & 1);
  return r;
}

}  // namespace self_plan
}  // namespace pgqa
