/*
 * paged_gqa.h -- C ABI of the GB300 (sm_103a) paged grouped-query attention library.
 *
 * One call computes, for a varlen batch of sequences, attention of the new query
 * tokens over a paged (block-tabled) KV cache with head_dim 256:
 *
 *   for each sequence s (q0 = query_start_loc[s], qn = query_start_loc[s+1] - q0,
 *   L = seq_lens[s]), query token t < qn and query head h:
 *     kvh = h / (Hq / Hkv)                         contiguous GQA head groups
 *     keys j = 0 .. L - qn + t                     bottom-right causal mask
 *     K_j  = k_cache[block_table[s, j / P], j % P, kvh, :] * k_descale
 *     V_j  = v_cache[block_table[s, j / P], j % P, kvh, :] * v_descale
 *     out[q0 + t, h, :] = softmax_j(softmax_scale * q . K_j) . V_j      (bf16)
 *
 * Where each piece comes from:
 *   - paged K/V with separate K and V views, one kv-head grid dimension, per-tensor
 *     FP8 descale scalars, query heads grouped per kv head:
 *     "Optimize Qwen3.5 MTP unified attention on gfx950" (sglang #36330), review
 *     thread on kv-head-generic launch and the Modifications section;
 *   - new tokens attending to cached + new K/V (cu_seqlens_k longer than
 *     cu_seqlens_q) under a bottom-right causal mask:
 *     "asm FP8 FMHA for prefix-hit prefill" (ROCm/ATOM #2534), summary;
 *   - a block table whose row stride is a runtime value and 64-token pages:
 *     "gfx1250 GDN prefill kernels ...; DP points on unified attention"
 *     (ROCm/ATOM #2830), description and commit 6.
 *
 * Conventions shared by every entry point:
 *   - Every pointer inside a pg_tensor is a DEVICE pointer on the current CUDA
 *     device. Shapes and strides are in elements. The innermost dimension of q,
 *     the caches and out must be contiguous (stride 1).
 *   - The caller owns every tensor. Calls are asynchronous and ordered on
 *     `stream`; the library keeps no pointer to caller memory once the call's
 *     work on `stream` has completed.
 *   - seq_lens[s] is the TOTAL K/V length of sequence s, new tokens included
 *     (their K/V must already be in the cache). 0 <= qn <= L <= W * P.
 *   - Block-table entries past ceil(L / P) are never read and may hold anything.
 *   - Cache slots at positions >= L are never read into the result: their
 *     contents (NaN included) do not change the output.
 *   - Return value: PG_OK (0) or a negative pg_status. A host-side error launches
 *     nothing; the message is available from paged_gqa_last_error().
 *   - Violations only visible on the device (qn > L, L > W * P, a block-table
 *     entry outside [0, NB)) never trap: the kernels record a code in a device
 *     error word, write zeros to the affected rows, and go on.
 *     paged_gqa_check_device_errors() reports and clears it.
 */
#ifndef PAGED_GQA_H_
#define PAGED_GQA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* pg_stream_t;

typedef enum {
  PG_BF16 = 1,
  PG_F16 = 2,   /* accepted by no entry point today; reserved */
  PG_E4M3 = 3,  /* OCP FP8 e4m3fn (max 448, no inf, 0x7F/0xFF are NaN) */
  PG_I32 = 4,
  PG_F32 = 5
} pg_dtype;

/* A strided view. Unused trailing shape/stride entries are ignored. */
typedef struct {
  void* data;
  int32_t dtype;      /* pg_dtype */
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];  /* elements */
} pg_tensor;

typedef enum {
  PG_OK = 0,
  PG_ERR_INVALID_ARG = -1,   /* null pointer, shape/stride mismatch, Hq % Hkv != 0,
                                misaligned base or row stride, non-contiguous last dim */
  PG_ERR_UNSUPPORTED = -2,   /* head_dim != 256, out not bf16, FP8 q with bf16 K/V,
                                page size not in {16, 32, 64, 128} */
  PG_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed */
  PG_ERR_TIMEOUT = -4,       /* device: a bounded wait gave up (reported by
                                paged_gqa_check_device_errors) */
  PG_ERR_DEVICE_BOUNDS = -5, /* device: qn > L, L > W*P or a page id outside [0, NB) */
  PG_ERR_WORKSPACE = -6      /* caller workspace too small or misaligned */
} pg_status;

/*
 * paged_gqa_attn -- the call.
 *
 *   q               [T, Hq, 256]        bf16, or e4m3 (then K/V must be e4m3;
 *                                        fold q's descale into softmax_scale)
 *   k_cache         [NB, P, Hkv, 256]   bf16 or e4m3; any strides on dims 0..2 that
 *                                        are multiples of 16 bytes; base 16-byte aligned
 *   v_cache         same shape and dtype as k_cache (its own strides)
 *   block_table     [num_seqs, W]       int32, physical page ids; any row stride
 *   seq_lens        [num_seqs]          int32, total K/V length per sequence
 *   query_start_loc [num_seqs + 1]      int32, [0] == 0, non-decreasing, [num_seqs] == T
 *   k_descale, v_descale                per-tensor dequant scales (pass 1 for bf16)
 *   softmax_scale                       multiplies q . k (usually 1/16 for hd 256)
 *   out             [T, Hq, 256]        bf16, written for every (token, head); its
 *                                        (token, head) rows must not overlap (strides
 *                                        positive and each at least the span of the
 *                                        smaller ones, else PG_ERR_INVALID_ARG)
 *   stream                              CUDA stream the work is ordered on
 *
 * Uses a library-owned workspace per device that grows on first need
 * (cudaMalloc: do not call this inside CUDA-graph capture on a new shape; use
 * paged_gqa_attn_ex with your own workspace there).
 */
int paged_gqa_attn(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                   const pg_tensor* block_table, const pg_tensor* seq_lens,
                   const pg_tensor* query_start_loc, float k_descale, float v_descale,
                   float softmax_scale, pg_tensor* out, pg_stream_t stream);

/*
 * paged_gqa_attn_ex -- the same call with an explicit q descale (multiplied into
 * softmax_scale) and a caller-owned device workspace of at least
 * paged_gqa_workspace_size(...) bytes, 256-byte aligned. Allocates nothing.
 * The workspace must not be shared by calls that can overlap on the device. Its contents
 * need no initialisation and may be left from any earlier use: the split-KV merge
 * counters in it carry a 48-bit per-call tag (a counter word that holds this call's tag
 * by chance, about 2^-48 per split block, would mistime that block's merge).
 */
int paged_gqa_attn_ex(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                      const pg_tensor* block_table, const pg_tensor* seq_lens,
                      const pg_tensor* query_start_loc, float q_descale, float k_descale,
                      float v_descale, float softmax_scale, pg_tensor* out,
                      void* workspace, size_t workspace_bytes, pg_stream_t stream);

/*
 * paged_gqa_attn_noalloc -- the same call as paged_gqa_attn, for callers that cannot
 * allocate device memory when they run attention (code inside an allocator or memory-pool
 * callback, runtimes that fix their device footprint after start-up). The pages have no
 * counterpart of this entry point.
 *
 * Arguments, layouts and results are those of paged_gqa_attn. Instead of a workspace it
 * uses a 64 MiB scratch array that is part of the library's device image: every GPU that
 * loads the library holds those 64 MiB until the process exits. It allocates nothing.
 * A call whose workspace need (paged_gqa_workspace_size) exceeds 64 MiB returns
 * PG_ERR_WORKSPACE and launches nothing. All calls on a device share the array; nothing
 * in it needs clearing (the split counters carry a per-call tag), but calls that can
 * overlap on the GPU (unordered streams) race on it. The first call on each device looks up the array's address with
 * that device current: make it before any stream capture.
 */
int paged_gqa_attn_noalloc(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                           const pg_tensor* block_table, const pg_tensor* seq_lens,
                           const pg_tensor* query_start_loc, float k_descale, float v_descale,
                           float softmax_scale, pg_tensor* out, pg_stream_t stream);

/*
 * paged_gqa_attn_quant_q -- paged_gqa_attn on a bf16 q that the call first quantises to
 * FP8 e4m3 with one per-tensor scale, so that Q . K^T runs as a single FP8 product
 * ("asm FP8 FMHA for prefix-hit prefill": the FP8 prefill attention takes an e4m3 Q with a
 * per-tensor scale, and its summary counts the Q cast inside the attention time).
 *
 * What it computes: amax = max |q| over the whole tensor (NaNs skipped); q_descale =
 * amax / 448 and inv = 1 / q_descale, each rounded to nearest in fp32 (both 1 when amax
 * is 0 or infinite); every element becomes the e4m3 code of q * inv (fp32 product, round
 * to nearest even, saturating at +-448); then exactly paged_gqa_attn with that e4m3 q and
 * q_descale. The e4m3 q is never written to memory: the attention kernels cast each Q
 * tile as they stage it, after one extra launch that reads q to find amax.
 *
 * Arguments are those of paged_gqa_attn, except: q must be bf16 and the caches e4m3
 * (else PG_ERR_UNSUPPORTED), and the tcgen05 path must be selected (paged_gqa_set_path
 * 0, the default, or 2; else PG_ERR_UNSUPPORTED). Uses the library-owned workspace like
 * paged_gqa_attn. Error behaviour as paged_gqa_attn.
 */
int paged_gqa_attn_quant_q(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                           const pg_tensor* block_table, const pg_tensor* seq_lens,
                           const pg_tensor* query_start_loc, float k_descale, float v_descale,
                           float softmax_scale, pg_tensor* out, pg_stream_t stream);

/*
 * paged_gqa_sparse_attn -- sparse paged GQA attention ("Tune sparse GQA prefill profile on
 * gfx942 and gfx950": each query row attends a selected list of tokens, ~2k per row,
 * head_dim 256, FP8 K/V). Row (token t, q head h) attends the keys listed in
 * indices[t, h / G, :]: for each entry p with 0 <= p <= L - q_len + (t - q_start) (the
 * row's bottom-right causal limit) the key at position p of t's sequence (page
 * block_table[s][p / P], slot p mod P) takes part in the softmax; other entries (negative,
 * or past the limit) are not used; an entry listed twice counts twice. A row with no
 * used entry is written as zeros.
 *
 * Arguments as paged_gqa_attn, plus
 *   indices  [T, num_kv_heads, K] int32 positions, last dim contiguous, 4-byte aligned;
 *            K may be 0 (every row zero). Caller-owned, read only.
 * q must be bf16 and the caches e4m3 with the same strides (else PG_ERR_UNSUPPORTED /
 * PG_ERR_INVALID_ARG). Allocates nothing. A block-table entry out of range sets
 * PG_ERR_DEVICE_BOUNDS in the device error word and the key is skipped. Two kernels compute
 * it: a warp-level one (the default) and a tcgen05 one for lists of 64 or more entries (four
 * (token, kv head) units share a tile), selected by paged_gqa_set_path(2).
 */
int paged_gqa_sparse_attn(const pg_tensor* q, const pg_tensor* k_cache, const pg_tensor* v_cache,
                          const pg_tensor* block_table, const pg_tensor* seq_lens,
                          const pg_tensor* query_start_loc, const pg_tensor* indices, float k_descale,
                          float v_descale, float softmax_scale, pg_tensor* out, pg_stream_t stream);

/*
 * paged_gqa_cache_write -- the step before the call: write the new tokens' K and V into
 * the paged FP8 cache it reads ("Optimize Qwen3.5 MTP unified attention on gfx950" and
 * "asm FP8 FMHA for prefix-hit prefill" read such a cache; this fills it).
 *
 *   k_new, v_new    [T, Hkv, 256]       bf16, the new tokens in query_start_loc order;
 *                                        head_dim contiguous, base and strides multiples
 *                                        of 16 bytes
 *   k_cache, v_cache [NB, P, Hkv, 256]  e4m3, written in place (same layout rules as the
 *                                        call's caches; in addition their (page, slot,
 *                                        head) rows must not overlap, else
 *                                        PG_ERR_INVALID_ARG)
 *   block_table, seq_lens, query_start_loc  as in paged_gqa_attn: sequence s's q_len =
 *                                        qsl[s+1] - qsl[s] new tokens take positions
 *                                        seq_lens[s] - q_len .. seq_lens[s] - 1
 *   k_descale, v_descale                the per-tensor descales the call multiplies back
 *                                        (finite, > 0)
 *
 * Token t of sequence s lands in page block_table[s][pos / P], slot pos % P, as the e4m3
 * codes of value * inv, where inv = 1 / descale rounded to fp32 once per call and the
 * product is taken in fp32 (then clamped to +-448, rounded to nearest even). For a
 * descale that is not a power of two this product can round to a different code than
 * an fp32 division value / descale would, at an e4m3 tie.
 * Nothing else in the caches changes. Host-side argument errors return a status before any
 * launch; a position or page id out of range is flagged in the device error word
 * (PG_ERR_DEVICE_BOUNDS via paged_gqa_check_device_errors) and that row is skipped.
 * Allocates nothing.
 */
int paged_gqa_cache_write(const pg_tensor* k_new, const pg_tensor* v_new, const pg_tensor* k_cache,
                          const pg_tensor* v_cache, const pg_tensor* block_table, const pg_tensor* seq_lens,
                          const pg_tensor* query_start_loc, float k_descale, float v_descale,
                          pg_stream_t stream);

/*
 * Workspace bytes for a call with these host-known sizes on `device`
 * (num_seqs, total query tokens T, heads, page size, block-table width W).
 * Returns 0 on invalid sizes. The size depends only on num_seqs, T, the head counts and
 * the device's SM count; page_size and max_blocks_per_seq (which bound every sequence's
 * length, L <= W * P) are accepted so that the signature stays valid if a later kernel
 * sizes anything by the longest sequence, and are otherwise unused.
 */
size_t paged_gqa_workspace_size(int num_seqs, int total_q, int num_q_heads, int num_kv_heads,
                                int page_size, int max_blocks_per_seq, int device);

/* Message of the last non-zero status returned on this host thread ("" if none). */
const char* paged_gqa_last_error(void);

/*
 * Synchronise `stream`, then read and clear the current device's error word.
 * Returns PG_OK, PG_ERR_DEVICE_BOUNDS, PG_ERR_TIMEOUT or PG_ERR_CUDA.
 */
int paged_gqa_check_device_errors(pg_stream_t stream);

/*
 * Kernel path selection, for tests and sweeps (process-wide):
 *   0 = automatic: the dense calls use the tcgen05 kernels where they apply (e4m3 caches)
 *       and warp-level MMA otherwise; sparse calls use the warp-level kernel (measured the
 *       faster of the two on the sparse workloads)
 *   1 = warp-level MMA (mma.sync) kernel for every tile
 *   2 = as 0, but sparse calls with lists of 64 or more entries use the tcgen05 kernel
 *   3 = as 0, but the verify class is always planned by the plan kernel before its
 *       kernel runs (under 0 the tcgen05 verify kernel plans it itself when
 *       num_seqs x num_kv_heads <= 512; results are identical)
 * Returns the previous value, or PG_ERR_INVALID_ARG.
 */
int paged_gqa_set_path(int path);

/*
 * Failure-path test hook (process-wide; for tests of the error path only). With wait_ns
 * > 0, every CTA of the tcgen05 attention kernels first waits wait_ns nanoseconds on a
 * shared-memory barrier that nothing arrives on. That bounded wait runs out, the CTA
 * records PG_ERR_TIMEOUT in the device error word and takes its abort path (every other
 * wait gives up at once; each role still waits for its own TMA copies and MMAs, then TMEM
 * is freed), so the call's output is unspecified and paged_gqa_check_device_errors()
 * returns PG_ERR_TIMEOUT. Nothing faults, traps or hangs; the context stays usable.
 * wait_ns = 0 (the default) turns it off. Returns the previous value.
 * (The pages describe no such hook: it tests this library's bounded waits.)
 */
int paged_gqa_set_stall_test(uint32_t wait_ns);

/*
 * Host-side launch summary of the last successful call on this host thread, for
 * tests and the benchmark. out8 receives {verify CTAs, prefill CTAs, kernels
 * launched, path bits (2: tcgen05 verify, 4: tcgen05 prefill, 8: warp-MMA verify,
 * 16: warp-MMA prefill, 32: tcgen05 sparse, 64: warp-MMA sparse), verify block bound,
 * prefill block bound, workspace bytes, 1 if the verify kernel planned its own class}.
 * A sparse call sets only the launch count and the path bits.
 */
int paged_gqa_last_plan(int64_t* out8);

/*
 * Profiling hook (process-wide): while set, every call records `start` on its stream
 * immediately before the attention kernel of class `cls` (0 = verify blocks,
 * 1 = prefill blocks) and `stop` immediately after it. Both are cudaEvent_t handles
 * owned by the caller; pass NULLs to stop recording. Returns PG_OK or
 * PG_ERR_INVALID_ARG.
 */
int paged_gqa_set_kernel_events(int cls, void* start, void* stop);

/* Library ABI version (major * 100 + minor). */
int paged_gqa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* PAGED_GQA_H_ */
