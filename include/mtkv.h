/*
 * mtkv.h — C ABI of libmtkv: grouped-query decode attention over a paged KV
 * cache, and the kernels that feed it, for NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 *  - Plain pointers and sizes only. "device" pointers are CUDA device
 *    addresses (for example from a torch tensor's data_ptr()), "host"
 *    pointers are ordinary CPU memory.
 *  - Ownership: the caller owns every buffer. The library allocates no
 *    device memory; calls that need scratch take a caller-provided
 *    workspace whose size comes from the matching *_workspace_bytes call.
 *  - Execution: compute calls are asynchronous on `stream` (a cudaStream_t;
 *    NULL is the legacy default stream). Their kernels are launched with
 *    programmatic dependent launch: a kernel may start while the previous
 *    kernel of the stream finishes, and waits for it before touching memory
 *    that kernel may write. The decode kernels read their context lengths,
 *    windows (spans, kv_map) and block tables before that wait, so these
 *    arrays must not be written by a kernel of the stream that lets its
 *    dependents launch early (griddepcontrol.launch_dependents) before it
 *    completes; copies, and kernels that do not, are waited for as usual.
 *    Arguments that can be checked on
 *    the host are checked before anything is launched; a failed check
 *    returns a status and launches nothing. Checks that need device data
 *    (block ids, context lengths, cells) run inside the kernels: an
 *    out-of-range value is skipped (never dereferenced) and recorded in a
 *    caller-owned 32-bit device status word, read back with
 *    mt_check_device_status().
 *  - Errors: every call returns mt_status; mt_last_error() gives a
 *    human-readable reason for the last failure on the calling thread.
 *  - The storage format is an explicit argument of every call; there is no
 *    process-wide format setting.
 *  - No call aborts or traps; device-side waits are bounded and report
 *    MT_ERR_TIMEOUT through the status word instead of hanging.
 */
#ifndef MTKV_H
#define MTKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mt_stream; /* a cudaStream_t */

/* KV storage formats — "KV Cache Design — cells, format, sessions",
 * section 3 (KvFormat {f32, f16, q8_0}). An unknown value is an error. */
typedef enum { MT_KV_F32 = 0, MT_KV_F16 = 1, MT_KV_Q8_0 = 2 } mt_kv_format;

typedef enum {
  MT_OK = 0,
  MT_ERR_INVALID_ARG = 1,  /* null pointer, negative size, inconsistent shape  */
  MT_ERR_UNSUPPORTED = 2,  /* valid but outside the built kernels' shape set   */
  MT_ERR_ORDER = 3,        /* move list would overwrite a row not yet copied   */
  MT_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out               */
  MT_ERR_DEVICE_CHECK = 5, /* a kernel met an out-of-range id / length / cell  */
  MT_ERR_CUDA = 6          /* a CUDA runtime call failed                       */
} mt_status;

/* Device status word bits (see mt_check_device_status). */
#define MT_STATUS_BIT_DEVICE_CHECK 1u
#define MT_STATUS_BIT_TIMEOUT 2u

/* Hole marker in a block table — "Tiered KV cache — architecture",
 * sections "The paged-attention block model" (item 3, holes) and "Kernel
 * dispatch" (kInvalidBlockTableEntry): its positions get logit -infinity. */
#define MT_INVALID_BLOCK_ID (-1)

/* A run of `len` rows (cells) moving from cell `src` to cell `dst`. */
typedef struct {
  int64_t src;
  int64_t dst;
  int64_t len;
} mt_move;

/* Bytes of one cell (one token's K, or V, for all KV heads).
 * "KV Cache Design — cells, format, sessions", section 3: f32 4*Hkv*d,
 * f16 2*Hkv*d, q8_0 a whole number of 34-byte Q8_0 blocks ({f16 scale,
 * int8 q[32]}; head h owns blocks [h*d/32, (h+1)*d/32)) rounded up to whole
 * 4-byte words. Returns 0 for an unknown format, non-positive sizes, or
 * q8_0 with head_dim % 32 != 0. Host function. */
size_t mt_kv_row_bytes(mt_kv_format fmt, int n_kv_heads, int head_dim);

/* KV store: write freshly projected rows into their resolved cells.
 * "KV Cache Design — cells, format, sessions", section 1 (positions vs
 * cells: the store writes the cell the allocator resolved) and section 3
 * (one store quantiser: q8_0 scale amax/127 stored as f16, codes
 * round-ties-even of x divided by the float32 amax/127, clamped to
 * +-127; f16 round-to-nearest-even; f32 verbatim).
 *   k_pool, v_pool  device, n_cells rows of mt_kv_row_bytes(fmt, ...) bytes
 *                   each, 16-byte aligned.
 *   k_new, v_new    device float32 [n_rows][n_kv_heads*head_dim].
 *   cells           device int64 [n_rows]; a negative cell skips that row;
 *                   a cell >= n_cells is skipped and flagged in *status.
 *   status          device uint32 status word, or NULL (no reporting).
 * Rows with the same cell: the last one wins is NOT guaranteed (caller
 * error). */
mt_status mt_kv_store(mt_kv_format fmt, void *k_pool, void *v_pool, int64_t n_cells,
                      int n_kv_heads, int head_dim, const float *k_new, const float *v_new,
                      const int64_t *cells, int n_rows, uint32_t *status, mt_stream stream);

/* Arguments of paged decode attention (one query token per sequence). */
/* Runs per query of a set-valued (kv_map) window. The pages name the limit
 * KV_MAP_MAX_SPANS without a value; this library fixes 8. */
#define MT_KV_MAP_MAX_SPANS 8

typedef struct {
  mt_kv_format fmt;
  const float *q;              /* device float32 [n_seqs][n_heads][head_dim]        */
  const void *k_pool;          /* device, n_phys_blocks*block_size cells, 16B-aligned */
  const void *v_pool;          /* same shape as k_pool                                */
  const int32_t *block_table;  /* device int32 [n_seqs][max_blocks]; entry = physical
                                  block id in [0, n_phys_blocks) or MT_INVALID_BLOCK_ID */
  const int32_t *context_lens; /* device int32 [n_seqs], each in [0, max_blocks*block_size] */
  const int32_t *spans;        /* device int32 [n_seqs][2] windows [lo, hi), or NULL  */
  float *out;                  /* device float32 [n_seqs][n_heads][head_dim]          */
  float *lse;                  /* device float32 [n_seqs][n_heads] or NULL            */
  int n_seqs;
  int n_heads;                 /* query heads; a multiple of n_kv_heads               */
  int n_kv_heads;
  int head_dim;
  int block_size;
  int max_blocks;
  int64_t n_phys_blocks;
  float scale;                 /* softmax scale applied to q.k                        */
  int n_ctas;                  /* 0 = one persistent CTA per SM; >0 forces the split  */
  const int32_t *kv_map;       /* [n_seqs][MT_KV_MAP_MAX_SPANS][2] set-valued window:
                                  (start, len) runs of logical positions per query
                                  (len <= 0: unused run), or NULL. The third window
                                  mode: at most one of spans / kv_map.                */
} mt_paged_attn_args;

/* Workspace bytes mt_paged_attn_decode needs for `args` (0 on invalid args).
 * The first 4 bytes of the workspace are the call's device status word:
 * zero them once after allocating the workspace; mt_check_device_status()
 * reads and clears them. */
size_t mt_paged_attn_workspace_bytes(const mt_paged_attn_args *args);

/* Grouped-query decode attention read through a paged KV cache.
 * "Tiered KV cache — architecture", sections "The paged-attention block
 * model" (position p of sequence s lives in physical block
 * block_table[s][p / block_size], slot p % block_size, i.e. cell
 * block_table[s][p/bs]*bs + p%bs of each pool) and "Kernel dispatch"
 * (block table, context lengths; MT_INVALID_BLOCK_ID positions get logit
 * -infinity, so zero weight). "KV Cache Design — cells, format, sessions",
 * section 1: the optional window of each query — one [lo, hi) pair
 * (spans) or a set of (start, len) runs (kv_map) — read as logical
 * positions intersected with [0, context_len). spans and kv_map together
 * are MT_ERR_INVALID_ARG.
 * For each sequence s and query head h (KV head h / (n_heads/n_kv_heads)):
 *   out[s][h] = sum_p softmax_p(scale * q[s][h] . k_p) v_p over the valid
 *   positions p; lse[s][h] = log sum_p exp(scale * q . k_p) (natural log).
 * A sequence with no valid position gets out = 0 and lse = -infinity.
 * Shapes built: head_dim in {64, 128, 256}, block_size in {16, 32},
 * n_kv_heads <= 8, n_heads/n_kv_heads <= 8; others return
 * MT_ERR_UNSUPPORTED. Out-of-range block ids and context lengths are
 * skipped and flagged in the workspace status word. */
mt_status mt_paged_attn_decode(const mt_paged_attn_args *args, void *workspace,
                               size_t workspace_bytes, mt_stream stream);

/* Paged decode attention with the new token's K/V store fused in.
 * What is stored and where follows "KV Cache Design — cells, format,
 * sessions", section 1 (the store writes the cell the allocator resolved;
 * the paged model resolves position p of sequence s to cell
 * block_table[s][p/bs]*bs + p%bs) and section 3 (the one store quantiser).
 * Doing the store inside the decode launch is this library's own design:
 * the page's fused family (projection, RoPE and store in one op) has no
 * attention in it. Equivalent to mt_kv_store of row s of k_new/v_new
 * into the cell of position context_lens[s]-1 of every sequence with a
 * positive context length, followed by mt_paged_attn_decode(args): the
 * attention sees the new row when its position is inside the window.
 *   k_new, v_new  device float32 [n_seqs][n_kv_heads*head_dim], 16-byte
 *                 aligned; converted exactly as mt_kv_store converts.
 * The CTA whose share of the work loads the block of position ctx-1 writes
 * that row just before it copies the block, so no separate store launch is
 * needed. The appended block must belong to its sequence alone (copy on
 * write before a store into a shared block, as the pages' sharing rule
 * says); a sequence whose appended block is a hole or out of range stores
 * nothing and is flagged in the workspace status word. Other arguments,
 * workspace and errors as mt_paged_attn_decode. */
mt_status mt_paged_attn_decode_append(const mt_paged_attn_args *args, const float *k_new,
                                      const float *v_new, void *workspace,
                                      size_t workspace_bytes, mt_stream stream);

/* Arguments of multi-query (prefill) paged attention. Device pointers unless
 * stated; all arrays dense, row-major. */
typedef struct {
  mt_kv_format fmt;
  const float *q;               /* [n_tokens][n_heads][head_dim] float32, the
                                   queries of all sequences, sequence-major      */
  const void *k_pool;           /* as mt_paged_attn_args (the queries' own K/V
                                   rows already stored)                          */
  const void *v_pool;
  const int32_t *block_table;   /* [n_seqs][max_blocks]                          */
  const int32_t *context_lens;  /* [n_seqs], the queries' positions included     */
  const int32_t *q_start;       /* [n_seqs + 1]: sequence s owns query rows
                                   q_start[s] .. q_start[s+1]-1; its n queries sit
                                   at positions ctx - n .. ctx - 1               */
  const int32_t *spans;         /* [n_tokens][2] per-query [lo, hi), or NULL     */
  const int32_t *kv_map;        /* [n_tokens][MT_KV_MAP_MAX_SPANS][2] per-query
                                   (start, len) runs (len <= 0: unused), or NULL;
                                   at most one of spans / kv_map                 */
  float *out;                   /* [n_tokens][n_heads][head_dim] float32         */
  float *lse;                   /* [n_tokens][n_heads] natural log, or NULL      */
  int n_seqs;
  int n_tokens;                 /* rows of q / out                               */
  int n_heads;
  int n_kv_heads;
  int head_dim;
  int block_size;
  int max_blocks;
  int64_t n_phys_blocks;
  float scale;
} mt_paged_prefill_args;

/* Workspace bytes mt_paged_attn_prefill needs (its first 4 bytes are the
 * device status word; zero them once after allocating). For q8_0 and f32
 * pools of head_dim 64 or 128 it includes the staging of the call's blocks:
 * n_seqs x max_blocks x block_size rows of n_kv_heads x head_dim f16 (q8_0)
 * or f16 pairs (f32) for K and for V, plus a table of n_seqs x max_blocks
 * ids. */
size_t mt_paged_prefill_workspace_bytes(const mt_paged_prefill_args *args);

/* Multi-query (prefill, or chunked prefill) attention through the paged
 * cache. "Tiered KV cache — architecture", section "Kernel dispatch"
 * (per-sequence context and query lengths) and "The paged-attention block
 * model" (holes read as -infinity); "KV Cache Design — cells, format,
 * sessions", section 1 (causal positions, one [lo, hi) window or kv_map runs
 * per query, read as logical positions). For query row i of sequence s,
 * j = i - q_start[s], position p = ctx - n + j:
 *   out[i][h] = sum_t softmax_t(scale * q[i][h] . k_t) v_t over the positions
 *   t <= p, t < ctx, not in a hole, inside the query's window;
 *   lse[i][h] = log sum_t exp(scale * q . k_t). No valid t: out 0, lse -inf.
 * Shapes built: head_dim 64 or 128 (and 256 for f16 and q8_0 pools),
 * block_size 16 or 32, n_heads/n_kv_heads <= 8, n_kv_heads <= 8 (others
 * MT_ERR_UNSUPPORTED). Out-of-range block ids,
 * query counts above the context length and query rows outside
 * [0, n_tokens) are skipped and flagged in the workspace status word.
 * Arithmetic: f16 pools (head_dim 64, 128) run on the 5th-generation tensor
 * cores with q split into high and low f16 halves (scores to ~2^-22) and
 * f16 probabilities; q8_0 pools of those head sizes take the same kernel
 * after a pass that stages each block the call reads as f16 rows, every
 * value code * scale rounded once to the nearest f16 (relative error <=
 * 2^-11, inside the q8_0 tolerance; a staged value beyond the f16 range is
 * flagged in the status word); f32 pools of those head sizes after a pass
 * that stages each value x as an f16 pair (x rounded, and the remainder
 * rounded: x to ~2^-22 relative), scores and P.V each from three products
 * (float32 accuracy; a value beyond the f16 range is flagged); head_dim 256
 * runs a warp-level tensor-core kernel that keeps codes exact and applies
 * scales in float32. A q8_0 or f32 call whose staged rows (n_seqs x
 * max_blocks x block_size) would reach 2^31 returns MT_ERR_UNSUPPORTED. The
 * workspace (mt_paged_prefill_workspace_bytes) holds
 * the staged rows of q8_0 and f32 calls and must be 16-byte aligned. */
mt_status mt_paged_attn_prefill(const mt_paged_prefill_args *args, void *workspace,
                                size_t workspace_bytes, mt_stream stream);

/* A group of consecutive sequences whose block tables start with the same
 * n_prefix_blocks physical block ids: a prompt prefix shared through
 * refcounted blocks ("Tiered KV cache — architecture", section "The
 * paged-attention block model", point 2: forks share blocks by refcount,
 * copy on write). */
typedef struct {
  int32_t seq_begin;       /* first sequence of the group                   */
  int32_t seq_end;         /* one past the last                             */
  int32_t n_prefix_blocks; /* leading block-table entries all of them share */
} mt_prefix_group;

/* Workspace bytes mt_paged_attn_decode_cascade needs (0 on invalid
 * arguments). Like mt_paged_attn_workspace_bytes, its first 4 bytes are the
 * device status word. Queries the current device. */
size_t mt_paged_attn_cascade_workspace_bytes(const mt_paged_attn_args *args,
                                             const mt_prefix_group *groups, int n_groups);

/* Shared-prefix (cascade) paged decode: computes exactly what
 * mt_paged_attn_decode(args) computes (same outputs, same tolerances), for
 * batches whose sequences share prefix blocks. Each shared block is read once
 * per KV head for all sequences of its group (their queries form one
 * tensor-core tile), instead of once per sequence; each sequence's private
 * suffix goes through the ordinary decode; the two partial results merge by
 * log-sum-exp ("KV Cache Design — cells, format, sessions", section 1: a
 * sequence reads another's prefix in place, within its window; the
 * set-valued window of the kv_map input — shared prefix plus private run —
 * is the case that page names). All three window modes are accepted: none,
 * spans, or kv_map runs (each row of a prefix tile then masks its own runs).
 *   groups    host array of n_groups (<= 64) disjoint groups; sequences in no
 *             group are decoded as usual. Each group's sequences must hold
 *             identical first n_prefix_blocks table entries (holes included):
 *             the kernel checks this and flags a mismatch in the workspace
 *             status word (MT_ERR_DEVICE_CHECK), the affected outputs then
 *             being undefined.
 * Shapes the prefix kernel is not built for (f32 pools of head_dim 256) run
 * the ordinary decode. Errors as mt_paged_attn_decode, plus MT_ERR_INVALID_ARG for bad or
 * overlapping groups. */
mt_status mt_paged_attn_decode_cascade(const mt_paged_attn_args *args,
                                       const mt_prefix_group *groups, int n_groups,
                                       void *workspace, size_t workspace_bytes, mt_stream stream);

/* mt_paged_attn_decode_cascade with each sequence's new K/V row stored
 * into the cell of position context_lens[s]-1 in the same call, exactly as
 * mt_paged_attn_decode_append does it (see there). The appended block must
 * lie outside the group's shared prefix (copy on write first), so only the
 * suffix decode reads it. */
mt_status mt_paged_attn_decode_cascade_append(const mt_paged_attn_args *args,
                                              const mt_prefix_group *groups, int n_groups,
                                              const float *k_new, const float *v_new,
                                              void *workspace, size_t workspace_bytes,
                                              mt_stream stream);

/* Bytes of the scratch array built into the library for
 * mt_paged_attn_decode_static (8 MiB per device that loads the library). */
#define MT_STATIC_SCRATCH_BYTES ((size_t)8 << 20)

/* Paged decode attention that allocates nothing and takes no workspace.
 * This entry point has no counterpart in the paper; it is a convenience of
 * this library. It computes exactly what mt_paged_attn_decode computes, for
 * callers that cannot allocate device memory when they decode (a fixed
 * memory budget that must not grow, an embedder that gets no allocator from
 * its host, a thread that must not call into the CUDA allocator): the
 * split-K scratch lives in one array of MT_STATIC_SCRATCH_BYTES inside the
 * library, which every GPU that loads the library keeps until the process
 * exits. The caller still passes inputs and outputs in `args`.
 *   status  device uint32 status word, or NULL (no device-side reporting).
 * Refused with MT_ERR_UNSUPPORTED, launching nothing, when the call needs
 * more scratch than the array holds (compare
 * mt_paged_attn_workspace_bytes with MT_STATIC_SCRATCH_BYTES).
 * All calls on a device share the array and leave the last call's contents
 * in it; nothing in it needs to start at zero, but calls whose kernels
 * overlap on the GPU race on it, so order them on one stream. The first
 * call on each device looks up the array's device address and caches it:
 * make that first call before any stream capture begins. The cached
 * address belongs to the device's current context: after cudaDeviceReset
 * (or anything else that destroys that context) it is stale, and this
 * entry point must not be called again in the process. */
mt_status mt_paged_attn_decode_static(const mt_paged_attn_args *args, uint32_t *status,
                                      mt_stream stream);

/* order_moves — "KV Cache Design — cells, format, sessions", section 2:
 * upward moves (dst > src) first, top-down (source descending), then
 * downward moves bottom-up (source ascending), so a destination never lands
 * on a row that has not been copied yet. Sorts `moves` (host) in place,
 * dropping moves with len <= 0 or dst == src; *n_out receives the new
 * count. Host function. */
mt_status mt_order_moves(mt_move *moves, int n_moves, int *n_out);

/* Validate a move list (host): MT_OK if no move writes a row that a later
 * move still reads and every run lies in [0, n_cells); MT_ERR_ORDER
 * otherwise, with the index of the first offending move in *first_bad
 * (may be NULL). Host function. */
mt_status mt_check_moves(const mt_move *moves, int n_moves, int64_t n_cells, int *first_bad);

/* copy_cells: apply an ordered move list to every pool, rows verbatim.
 * "KV Cache Design — cells, format, sessions", section 2 (compaction moves
 * rows verbatim; overlapping runs copy ascending when sliding down and
 * descending when sliding up). The result equals applying each move in
 * list order as a memmove of len*row_bytes bytes in every pool.
 *   pools      host array of n_pools (<= 256) device pointers, 16-byte
 *              aligned, each n_cells rows of row_bytes bytes (% 4 == 0).
 *   moves      host array, already ordered (mt_order_moves). It is checked
 *              with mt_check_moves first; MT_ERR_ORDER launches nothing.
 * The schedule travels in kernel parameters (no workspace, no host-device
 * copy): consecutive moves share a launch (at most 1024, one CTA each) while
 * none writes rows another of them reads or writes; each move copies in
 * chunks of min(|dst-src|, len) rows in slide order with a barrier between
 * chunks (runs that fit in shared memory move in one staged round).
 *   status     device status word, or NULL. A staged move whose bounded wait
 *              for its load runs out leaves its rows unmoved and sets
 *              MT_STATUS_BIT_TIMEOUT here (mt_check_device_status then
 *              returns MT_ERR_TIMEOUT); with NULL such a failure cannot be
 *              reported, so callers that need the bit-exact guarantee pass
 *              a word and check it. */
mt_status mt_copy_cells(void *const *pools, int n_pools, size_t row_bytes, int64_t n_cells,
                        const mt_move *moves, int n_moves, uint32_t *status, mt_stream stream);

/* Cold-tier int4 quantise — "Tiered KV cache — architecture", section
 * "The three-tier model": per block one float32 scale and ceil(n_elts/2)
 * packed int4 nibbles. Reading: scale = amax/7 (float32), q =
 * clamp(rint(x/scale), -8, 7), nibble = q + 8, element 2j in the low nibble
 * of byte j; amax == 0 gives scale 0 and nibbles 8. A block's elements are
 * its block_size*n_kv_heads*head_dim values in pool order [slot][head][dim].
 *   fmt      MT_KV_F16 or MT_KV_F32 (the pool's format).
 *   pool     device pool of n_phys_blocks*block_size cells.
 *   blocks   device int32 [n_blocks] physical ids to quantise.
 *   scales   device float32 [n_blocks]; nibbles device uint8
 *            [n_blocks][n_elts/2], 16-byte aligned.
 *   status   device status word or NULL; out-of-range ids are skipped. */
mt_status mt_kv_quant_int4(mt_kv_format fmt, const void *pool, int block_size, int n_kv_heads,
                           int head_dim, int64_t n_phys_blocks, const int32_t *blocks,
                           int n_blocks, float *scales, uint8_t *nibbles, uint32_t *status,
                           mt_stream stream);

/* Cold-tier int4 dequantise into (fresh) physical blocks: element =
 * round_to_pool_type(float32(scale * (nibble - 8))). Same layout as
 * mt_kv_quant_int4; dst_blocks lists the blocks written. */
mt_status mt_kv_dequant_int4(mt_kv_format fmt, void *pool, int block_size, int n_kv_heads,
                             int head_dim, int64_t n_phys_blocks, const int32_t *dst_blocks,
                             int n_blocks, const float *scales, const uint8_t *nibbles,
                             uint32_t *status, mt_stream stream);

/* Grow-on-demand re-layout — "KV cache" (sipllm), section "Design": a
 * [layer][pos][row] store with the capacity as per-layer stride; growing
 * copies each layer's old_cap rows verbatim from stride old_cap (src) to
 * stride new_cap (dst). Rows [old_cap, new_cap) of dst are not written.
 * src, dst: device, 16-byte aligned, not overlapping; row_bytes % 4 == 0. */
mt_status mt_kv_relayout(const void *src, void *dst, int n_layers, int64_t old_cap,
                         int64_t new_cap, size_t row_bytes, mt_stream stream);

/* The same page's capacity rule: double `cap` until it holds `need`
 * positions, then cap at max_ctx. Returns -1 on invalid input. Host. */
int64_t mt_kv_grow_capacity(int64_t cap, int64_t need, int64_t max_ctx);

/* Diagnostic, no counterpart in the pages: launch one CTA that waits, with the
 * bounded wait every pipeline wait in this library uses, on a barrier nothing
 * will ever complete. After limit_ns (0 < limit_ns <= 2 s) the wait gives up
 * and sets MT_STATUS_BIT_TIMEOUT in *status (device word); the kernel returns
 * and the context stays usable. Used to test failure detection without
 * faulting or hanging the GPU. */
mt_status mt_selftest_bounded_wait(uint64_t limit_ns, uint32_t *status, mt_stream stream);

/* Synchronise `stream`, read the device status word, clear it, and map it
 * to MT_OK, MT_ERR_TIMEOUT or MT_ERR_DEVICE_CHECK. */
mt_status mt_check_device_status(uint32_t *status_word, mt_stream stream);

/* Reason for the calling thread's last non-OK status ("" if none). */
const char *mt_last_error(void);

/* Library version string. */
const char *mt_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MTKV_H */
