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

struct RowBlock {
  int seq, kvh;
  int row0, nrows;      // rows [row0, row0 + nrows) of the (seq, kvh) row space
  int kv_end;           // keys [0, kv_end) are visible to the block's last row
  int tiles;            // ceil(kv_end / kTileKeys)
  long long tile_off;   // plan only: first unit of the block's span (fixed cost, then tiles)
  int nsplit;           // number of pieces (CTAs) the block is cut into
  int slot_base;        // first partial slot (valid when nsplit > 1)
};

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
  int* counters;           // [max_blocks]
  uint16_t* part_o;        // [max_slots][slot_rows][kHeadDim] f16: O / l in cache-code units
                           // (v_descale is applied by the merge; |O / l| <= 448 fits f16)
  float* part_lse;         // [max_slots][slot_rows] (log2 units)
  int num_ctas;
  int max_blocks, max_items, max_slots;
  int slot_rows;           // rows of a block of this class (64 verify, 128 prefill)
};

}  // namespace pgqa
