// common.cuh -- types shared by the plan kernel, the attention kernels and the host API.
//
// Work decomposition (all on the device; the host knows only upper bounds):
//   * a "row block" is up to 128 query rows of one (sequence, kv head). Row r of a
//     (sequence, kv head) is query token t = r / G and head g = r % G, i.e. the q_len x G
//     rows of one kv head are packed into the M (or N) dimension of one tile, so each KV
//     page is read once per kv head, not once per query token ("Optimize Qwen3.5 MTP
//     unified attention on gfx950", Modifications: BLOCK_M covers tokens x heads);
//   * verify blocks hold all q_len*G <= 64 rows of a short query; prefill blocks cut
//     longer queries into 128-row blocks;
//   * a block's keys are [0, kv_end) with kv_end the causal limit of its last row;
//     they form ceil(kv_end / 128) key tiles;
//   * the tiles of all blocks of one class are concatenated and cut into equal
//     contiguous ranges, one per persistent CTA (split-KV); a block cut into several
//     pieces is finished by a log-sum-exp merge of the pieces' partial results
//     ("Optimize Qwen3.5 MTP unified attention on gfx950": split-KV segments
//     reduced after the 3D kernel).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace pgqa {

constexpr int kHeadDim = 256;
constexpr int kTileKeys = 128;        // keys per tile (every kernel)
constexpr int kVerifyRows = 64;       // max rows of a verify block
constexpr int kPrefillRows = 128;     // rows of a prefill block
constexpr int kSlotRows = 128;        // rows per partial-result slot
constexpr int kNumClasses = 2;        // 0 = verify, 1 = prefill

// How a tcgen05 attention kernel stages Q (its template argument).
constexpr int kQSplit = 0;  // bf16 Q as e4m3 hi + lo parts under a per-tile power-of-two scale
constexpr int kQGiven = 1;  // e4m3 Q as given (its descale folded into the score scale)
constexpr int kQCast = 2;   // bf16 Q cast to e4m3 with the call's per-tensor scale amax / 448

// device error word bits
constexpr uint32_t kErrBounds = 1u;   // qn > L, L > W*P, qsl not monotone
constexpr uint32_t kErrPage = 2u;     // block-table entry outside [0, NB)
constexpr uint32_t kErrTimeout = 4u;  // a bounded wait gave up

// Split-KV cut of one class (the plan kernel; a self-planned verify kernel does the same):
// block b spans fixed_cost(class) units (what starting it costs a CTA: Q load, epilogue,
// merge) and then one unit per key tile; the class's U units are cut into C equal ranges
// [floor(c U / C), floor((c + 1) U / C)), one per persistent CTA.
__host__ __device__ constexpr int fixed_cost(int cls) { return cls == 0 ? 6 : 2; }
// CTAs a class's U units are cut across: one range per CTA, but no range shorter than
// kMinRangeUnits (a piece that small costs more in its partial store and merge than it
// saves: a small problem runs on fewer CTAs, in fewer pieces). Measured on GB300 over 1-6,
// 8, 10, 12, 16, 32 for verify batches of 1-32 sequences: 6 was best or within 1 us of it
// everywhere (8 x q4 with L 2-5.5k: 38 us per call, against 96 us when every CTA took a
// range), and the 64- and 256-sequence workloads did not change.
constexpr int kMinRangeUnits = 6;
__host__ __device__ __forceinline__ int cut_ctas(long long U, int num_ctas) {
  const long long c = U / kMinRangeUnits;
  return (int)(c < 1 ? (U > 0 ? 1 : 0) : (c < num_ctas ? c : num_ctas));
}
// CTA whose range holds unit u.
__host__ __device__ __forceinline__ int cta_of(long long u, long long U, int C) {
  return (int)(((u + 1) * C + U - 1) / U) - 1;
}
__host__ __device__ __forceinline__ long long range_begin(int c, long long U, int C) {
  return (long long)c * U / C;
}
constexpr unsigned long long kSplitTagMask = (1ull << 48) - 1;
// Most verify blocks (sequences x kv heads) of a call whose verify kernel plans its own
// class (its CTAs keep one entry per block they work on in shared memory).
constexpr int kFusedMaxBlocks = 512;

struct RowBlock {
  int seq, kvh;
  int row0, nrows;      // rows [row0, row0 + nrows) of the (seq, kvh) row space
  int kv_end;           // keys [0, kv_end) are visible to the block's last row
  int tiles;            // ceil(kv_end / kTileKeys)
  long long tile_off;   // plan only: first unit of the block's span (fixed cost, then tiles)
  int nsplit;           // number of pieces (CTAs) the block is cut into
  int slot_base;        // first partial slot (valid when nsplit > 1): piece i uses slot_base + i
};

// Partial slots of a split block, without a prefix over blocks: a block whose first tile
// falls in CTA c0's range takes slots [2 c0 + x, 2 c0 + x + nsplit), x = 1 if c0's range
// starts in an earlier block, else 0. Pieces 1.. are the first items of CTAs c0 + 1, ..,
// and the next split block starts at CTA c0 + nsplit - 1 or later with x = 1, i.e. at slot
// 2 (c0 + nsplit - 1) + 1 >= 2 c0 + x + nsplit: ranges never overlap, and 2 C slots suffice.
__host__ __device__ __forceinline__ int split_slot_base(int c0, bool range_starts_earlier) {
  return 2 * c0 + (range_starts_earlier ? 1 : 0);
}

struct WorkItem {
  int block;            // index into the class's RowBlock array
  int tile_begin, tile_end;
  int split;            // piece index within the block, 0..nsplit-1
};

// Per-call sizes known on the host, shared with every kernel.
struct Problem {
  int num_seqs, T, Hq, Hkv, G, P, W, NB;
  int q_is_fp8, kv_is_fp8;
  int q_cast;              // bf16 Q quantised per tensor inside the call (kQCast)
  int q_amax_parts;        // entries of Pointers::q_amax (q_cast only)
  // strides in elements
  long long q_st, q_sh;
  long long k_sb, k_sp, k_sh;
  long long v_sb, v_sp, v_sh;
  long long o_st, o_sh;
  long long bt_stride;
  float score_scale_log2;  // softmax_scale * q_descale * k_descale * log2(e)
  float out_scale;         // v_descale
  // Failure-path test (0 = off): the softmax warps of every tcgen05 attention CTA first wait
  // this many ns on a barrier that nothing arrives on; the wait runs out, the CTA takes its
  // abort path and the device error word reports a timeout.
  uint32_t stall_test_ns;
  // Nonzero, and new on every eager call (a CUDA graph replays its captured value; the
  // workspace's epoch word still moves): mixed with that word into the split counters' tag.
  uint32_t call_tag;
  // The verify class is planned by its own kernel's CTAs (each works out its range from
  // query_start_loc and seq_lens in its prologue); the plan kernel then plans prefill only.
  int fused_verify;
};

struct Pointers {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* qsl;
  void* out;               // bf16
  uint32_t* err;           // device error word
  const float* q_amax;     // per-CTA maxima of |q| from the amax kernel (q_cast only)
};

// Plan output in the workspace, one instance per class.
struct ClassPlan {
  int* n_blocks;           // [1]
  int* n_items;            // [1]
  long long* total_tiles;  // [1]
  int* cta_item_begin;     // [num_ctas + 1]
  RowBlock* blocks;        // [max_blocks]
  WorkItem* items;         // [max_items]
  // [max_blocks] split counters: (48-bit tag << 16) | pieces arrived. A word whose tag is
  // not this call's counts as zero, so nothing has to clear them between calls (the tag
  // changes on every call, CUDA-graph replays included) and a workspace needs no zeroing.
  unsigned long long* counters;
  unsigned long long* epoch;  // [1] workspace word the plan kernel advances once per call
  uint16_t* part_o;        // [max_slots][slot_rows][kHeadDim] f16: O / l in cache-code units
                           // (v_descale is applied by the merge; |O / l| <= 448 fits f16)
  float* part_lse;         // [max_slots][slot_rows] (log2 units)
  int num_ctas;
  int max_blocks, max_items, max_slots;
  int slot_rows;           // rows of a block of this class (64 verify, 128 prefill)
};

}  // namespace pgqa
