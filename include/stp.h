/*
 * stp.h -- C ABI of the prefix-tree packing + tree-attention library (libstp.so).
 *
 * The library packs tokenized sequences as one radix tree per training row
 * (a host packer) and runs causal tree attention over the packed rows on a
 * GB300 (sm_103a): tile classification, forward (O, LSE) and backward
 * (dQ, dK, dV).  Sources, by page and section:
 *
 *   [P1] "Prefix tree packing" (furtherai.github.io/blog/posts/prefix-tree-packing):
 *        tree-build section (the recursive walk, minimum shared-segment length,
 *        trainable tokens never shared, the join-token copy); global-tree
 *        section; bin-packing section (tree-aware best-fit-decreasing);
 *        attention section (ancestor-only visibility, DFS enter/exit interval
 *        check, empty blocks skipped); materialization section.
 *   [P2] "How to Configure Sequence Packing ..." (AReaL how-to), "Monitoring
 *        Packing Efficiency": the tree_token_ratio statistic.
 *   [P3] "ART-Optimized Megatron" (CoreWeave), "How do we implement shared
 *        prefix?": attention over the tree layout with a mask that lets tokens
 *        see the shared prefix and isolates sibling branches.
 *
 * Conventions
 *   - Every call returns an stp_status; no exception crosses the ABI.  On a
 *     non-zero status a thread-local message is available from stp_last_error().
 *   - Host buffers are caller-owned unless stated.  The opaque stp_plan is
 *     owned by the library (free it with stp_plan_free); it is immutable after
 *     stp_pack, so concurrent reads from several threads are safe.
 *   - Device buffers and workspaces are caller-owned; no call allocates
 *     device memory (stp_classify_noalloc uses a fixed array the library
 *     holds instead of caller scratch).  Device calls are asynchronous on the given
 *     stream (a cudaStream_t passed as void*; NULL = the legacy default
 *     stream).  Their status covers host-side validation and launch errors;
 *     device-side checks set an error word in the workspace that
 *     stp_device_status() reads.
 *   - Tensors are contiguous row-major: Q, O, dO, dQ [R, T, Hq, D];
 *     K, V, dK, dV [R, T, Hkv, D]; LSE float32 [R, Hq, T] (natural log);
 *     subtree_end int32 [R, T].
 */
#ifndef STP_H_
#define STP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t stp_status;
enum {
  STP_OK = 0,
  STP_EINVAL = 1,       /* bad argument: NULL pointer, size, alignment, shape     */
  STP_ETOOLONG = 2,     /* a sequence is longer than a row                        */
  STP_ENOMEM = 3,       /* host allocation failed                                 */
  STP_ECUDA = 4,        /* a CUDA launch or stream error                          */
  STP_EUNSUPPORTED = 5, /* dtype / head_dim / head ratio / row length not handled */
  STP_EDEVICE = 6       /* a device-side check tripped (see stp_device_status)    */
};

/* ------------------------------------------------------------------------ */
/* Host packer                                                              */
/* ------------------------------------------------------------------------ */

enum {
  STP_GLOBAL = 0u,        /* one global tree over every sequence ([P1] global-tree section) */
  STP_PER_FAMILY = 1u,    /* one tree per family, then the same placement (comparison arm)  */
  STP_IN_ORDER = 2u       /* fill rows in input order, moving on when a leaf does not fit
                             ([P1] "fill in the bins as you go"; comparison arm)             */
};

typedef struct stp_plan stp_plan;

typedef struct {
  int32_t n_rows;          /* R: rows (bins) in creation order                        */
  int32_t row_len;         /* T                                                       */
  int64_t input_tokens;    /* sum of sequence lengths                                 */
  int64_t packed_tokens;   /* real (non-pad) tokens over all rows                     */
  int64_t n_segments;      /* segments emitted by the walk, empty leaf segments too   */
  int64_t n_leaves;        /* = number of sequences                                   */
  int64_t useful_pairs;    /* visible (query, key) pairs over real tokens =
                              sum over real tokens of (position id + 1)               */
  double tree_token_ratio; /* input_tokens / packed_tokens ([P2] Monitoring)          */
} stp_plan_info_t;

/*
 * stp_pack -- build the global prefix tree and place its leaves into rows.
 *
 * [P1] tree-build section: the longest run every active sequence agrees on is
 * emitted once and the rest is split by next token.  A run shorter than
 * `min_shared` is not shared (it is repeated inside each sub-branch); runs stop
 * at trainable tokens; where a member's next token is trainable the shared run
 * gives up its last token and every branch below carries its own copy of it.
 * [P1] bin-packing section: leaves (one per sequence, cost = its length) are
 * placed best-fit-decreasing on their insertion delta (path segments the row
 * does not hold yet), families ordered by their largest leaf (stable), leaves
 * of a family in input order, the earliest row on ties.
 *
 *   tokens     int32 [offsets[n_seqs]]  token ids, sequences back to back (host)
 *   offsets    int64 [n_seqs + 1]       offsets[0] = 0, non-decreasing; every
 *                                       sequence must be non-empty (host)
 *   n_seqs     >= 0
 *   trainable  uint8 [offsets[n_seqs]] or NULL (= no trainable token)
 *   family     int32 [n_seqs] or NULL (= every sequence its own family)
 *   row_len    T > 0
 *   min_shared >= 1 (the pages' default is 64)
 *   flags      STP_GLOBAL, STP_PER_FAMILY or STP_IN_ORDER (may be OR-ed)
 *   out        receives the plan; *out is NULL on error
 * Errors: STP_EINVAL (bad pointer/offsets/arguments), STP_ETOOLONG (a sequence
 * longer than row_len), STP_ENOMEM.
 */
stp_status stp_pack(const int32_t* tokens, const int64_t* offsets, int32_t n_seqs,
                    const uint8_t* trainable, const int32_t* family, int32_t row_len,
                    int32_t min_shared, uint32_t flags, stp_plan** out);

/* Statistics of a plan (host). */
stp_status stp_plan_info(const stp_plan* plan, stp_plan_info_t* info);

/*
 * stp_plan_write -- materialize the plan into caller-owned host buffers
 * ([P1] materialization section: one pass slices the tokens into rows).
 * Rows hold the DFS pre-order of their segments, so a token's row index is its
 * DFS enter index and subtree_end[x] is the row index of the last token of the
 * subtree below x's segment (the exit index; [P1] attention section): key j is
 * visible to query i iff j <= i && subtree_end[j] >= i.  Pads fill each row
 * after its last real token with token 0, position 0, subtree_end = own index,
 * loss 0.
 *   token_ids, position_ids, subtree_end  int32 [R * T]
 *   loss_mask     uint8 [R * T]: 1 where the next token of the sequence is trainable
 *   gather_index  int64 [offsets[n_seqs]]: row-major flat index (r * T + x) of
 *                 every input token, sequences in input order
 * Any output pointer may be NULL (not written).
 */
stp_status stp_plan_write(const stp_plan* plan, int32_t* token_ids, int32_t* position_ids,
                          int32_t* subtree_end, uint8_t* loss_mask, int64_t* gather_index);

/*
 * stp_plan_times -- host wall time (milliseconds, steady clock) that stp_pack
 * spent building this plan: the trie walk and the placement of the leaves
 * into rows, measured apart ([P1] planning-cost table: "tree walk" and "bin
 * packing" columns).  Both pointers must be non-NULL (STP_EINVAL otherwise).
 */
stp_status stp_plan_times(const stp_plan* plan, double* walk_ms, double* place_ms);

/* Row index (bin) of every sequence, int32 [n_seqs] (host). */
stp_status stp_plan_rows_of(const stp_plan* plan, int32_t* row_of_seq);

void stp_plan_free(stp_plan* plan);

/*
 * stp_plan_rows -- "what if" planning ([P1] global-tree section: the pass that
 * packs a step is also run over sampled subsets of past data, to estimate how
 * many rows a candidate batch would need before committing to it).  Returns
 * the number of rows and of packed (real) tokens that stp_pack would produce
 * for the sequences subset[0..n_subset) of a pool, taken in that order, with
 * the same row_len, min_shared and flags; no plan is kept and nothing is
 * materialized.
 *   tokens, offsets, n_seqs, trainable, family   the pool, as for stp_pack
 *   subset     int32 [n_subset] indices into the pool (repeats allowed), or
 *              NULL for the whole pool in input order
 *   n_rows, packed_tokens   outputs
 * Errors: those of stp_pack; STP_EINVAL for an index outside [0, n_seqs).
 */
stp_status stp_plan_rows(const int32_t* tokens, const int64_t* offsets, int32_t n_seqs,
                         const uint8_t* trainable, const int32_t* family, const int32_t* subset,
                         int32_t n_subset, int32_t row_len, int32_t min_shared, uint32_t flags,
                         int32_t* n_rows, int64_t* packed_tokens);

/*
 * stp_plan_rows_many -- stp_plan_rows for many subsets at once, planned in
 * parallel on host threads (n_threads <= 0: one per hardware thread).
 * Subset i is subsets[subset_offsets[i] .. subset_offsets[i+1]);
 * subset_offsets int64 [n_subsets + 1], subset_offsets[0] = 0, non-decreasing.
 * n_rows int32 [n_subsets] and packed_tokens int64 [n_subsets] receive the
 * results.  On error the status and message are those of the first failing
 * subset (its index is in the message); the other outputs are unspecified.
 */
stp_status stp_plan_rows_many(const int32_t* tokens, const int64_t* offsets, int32_t n_seqs,
                              const uint8_t* trainable, const int32_t* family,
                              const int32_t* subsets, const int64_t* subset_offsets,
                              int32_t n_subsets, int32_t row_len, int32_t min_shared,
                              uint32_t flags, int32_t n_threads, int32_t* n_rows,
                              int64_t* packed_tokens);

/* ------------------------------------------------------------------------ */
/* Tree attention on the GPU                                                */
/* ------------------------------------------------------------------------ */

enum { STP_BF16 = 0, STP_FP32 = 1 };

typedef struct {
  int32_t n_rows;      /* R                                                        */
  int32_t row_len;     /* T, a multiple of 128, at most 131072                     */
  int32_t n_q_heads;   /* Hq                                                       */
  int32_t n_kv_heads;  /* Hkv; Hq % Hkv == 0; query head h reads kv head h/(Hq/Hkv) */
  int32_t head_dim;    /* D: 128 (bf16 or fp32) or 64 (fp32)                       */
  int32_t dtype;       /* STP_BF16 or STP_FP32, for Q, K, V, O, dO, dQ, dK, dV     */
  float scale;         /* softmax scale, usually 1/sqrt(D)                         */
  int32_t block_m;     /* must be 128 (or 0 = 128)                                 */
  int32_t block_n;     /* must be 128 (or 0 = 128)                                 */
  int32_t max_tile_pairs; /* bound on the non-empty (query tile, key tile) pairs
                             over all rows (stp_count_tile_pairs gives the exact
                             count); sizes the bf16 backward's dS workspace.
                             0 = every pair with key tile <= query tile,
                             R * NT * (NT + 1) / 2 with NT = T / 128            */
  int32_t ds_groups;   /* bf16 backward: kv-head groups whose dS tiles the
                          workspace holds at once.  The backward runs the kv
                          heads in n = min(Hkv, 8) groups of whole kv heads,
                          each on its own stream; with ds_groups in [1, n) a
                          group reuses the slot of the group ds_groups before
                          it and waits for that group's dQ pass, which bounds
                          the workspace by ds_groups groups instead of Hq
                          (less overlap between groups).  0 = n (all groups
                          at once, fastest)                                  */
} stp_attn_desc;

/*
 * Exact number of non-empty (query tile, key tile) pairs of 128-token tiles
 * over all rows of a host subtree_end array int32 [n_rows, row_len]:
 * key tile kt pairs with query tiles kt .. max_{j in kt} subtree_end[j] / 128
 * (the predicate j <= i && subtree_end[j] >= i).  Errors: STP_EINVAL (NULL,
 * row_len not a positive multiple of 128, subtree_end[j] outside [j, row_len)).
 */
stp_status stp_count_tile_pairs(const int32_t* subtree_end, int32_t n_rows, int32_t row_len,
                                int64_t* n_pairs);

/*
 * Byte sizes of the caller-owned device buffers for a descriptor:
 *   tile_meta  -- tile classes and work lists written by stp_classify
 *   fwd_ws     -- workspace of stp_attn_fwd (error word)
 *   bwd_ws     -- workspace of stp_attn_bwd (error word, per-query
 *                 Delta = dO . O and -LSE log2 e, and on the bf16 path one
 *                 32 KiB dS tile per (non-empty tile pair, query head of
 *                 the kv-head groups held at once), so
 *                 max_tile_pairs * S * ceil(Hkv / n) * (Hq / Hkv) * 32 KiB
 *                 with n = min(Hkv, 8) groups and S = ds_groups (or n))
 * Any pointer may be NULL.  Buffers must be 256-byte aligned.
 */
stp_status stp_workspace_size(const stp_attn_desc* desc, size_t* tile_meta_bytes,
                              size_t* fwd_ws_bytes, size_t* bwd_ws_bytes);

/*
 * stp_classify -- mark every (query tile, key tile) pair of each row EMPTY (0),
 * PARTIAL (1) or FULL (2) from subtree_end, and build the per-query-tile list
 * of non-empty key tiles and the per-key-tile list of non-empty query tiles
 * ([P1] attention section: most blocks of a packed row are empty and are
 * skipped; the rest are fully visible ancestor blocks or partial blocks).
 *   d_subtree_end  device int32 [R, T] as written by stp_plan_write
 *   d_tile_meta    device, tile_meta_bytes
 * Relies on subtree_end[j] >= j (true for any packed row).
 */
stp_status stp_classify(const stp_attn_desc* desc, const int32_t* d_subtree_end,
                        void* d_tile_meta, void* stream);

/*
 * stp_classify_noalloc -- stp_classify for callers that cannot allocate device
 * memory (for instance code being recorded into a CUDA graph, where cudaMalloc
 * is not allowed, or a plug-in host that only passes the buffers of its inputs
 * and outputs).  The paper has no counterpart; this is a library convenience.
 * Same arguments, outputs and checks as stp_classify, but the kernel's scratch
 * (per-key-tile min / max of subtree_end) lives in a fixed device array inside
 * the library, 1 MiB, held by every GPU that loads the library until the
 * process exits; no allocation is made by this call.
 *   - at most n_rows * (row_len / 128) <= 131072 tiles; larger sizes return
 *     STP_EINVAL with a message (use stp_classify);
 *   - the first call on a device looks up the array's device address with that
 *     device current (cudaGetSymbolAddress); make that first call before any
 *     stream capture;
 *   - all calls share the one array: calls that overlap on the GPU (different
 *     streams, or different host threads without ordering) race and may
 *     corrupt each other's result.  The array keeps the last call's contents;
 *     every entry is rewritten before it is read, so nothing needs clearing.
 */
stp_status stp_classify_noalloc(const stp_attn_desc* desc, const int32_t* d_subtree_end,
                                void* d_tile_meta, void* stream);

/* Copy the class matrix int8 [R, T/128, T/128] out of tile_meta (device to device). */
stp_status stp_read_tile_classes(const stp_attn_desc* desc, const void* d_tile_meta,
                                 int8_t* d_cls_out, void* stream);

/*
 * stp_attn_fwd -- tree attention forward ([P1] attention section; [P3]).
 * For query i of head h (kv head g = h / (Hq/Hkv)) over the visible keys
 * V(i) = { j : j <= i && subtree_end[j] >= i }:
 *   s_ij = scale * q_i . k_j,  LSE_i = ln sum_j exp(s_ij),
 *   O_i = sum_j exp(s_ij - LSE_i) v_j.
 * Empty tiles are skipped; the predicate is evaluated on partial tiles only.
 *   q, k, v   device, dtype of desc, layouts above, 16-byte aligned
 *   o         device [R, T, Hq, D], same dtype;  lse device float32 [R, Hq, T]
 *   d_ws      device, fwd_ws_bytes
 * d_tile_meta must come from stp_classify on the same subtree_end.
 */
stp_status stp_attn_fwd(const stp_attn_desc* desc, const void* q, const void* k, const void* v,
                        const int32_t* d_subtree_end, const void* d_tile_meta, void* o,
                        float* lse, void* d_ws, void* stream);

/*
 * stp_attn_bwd -- analytic backward of the forward above for L = sum dO . O:
 *   dP_ij = dO_i . v_j,  Delta_i = dO_i . O_i,  dS_ij = p_ij (dP_ij - Delta_i),
 *   dQ_i = scale sum_j dS_ij k_j,
 *   dK_j = scale sum_{i, h in group} dS_ij q_i,  dV_j = sum_{i, h in group} p_ij dO_i.
 *   o, lse     the forward's outputs;  d_o device [R, T, Hq, D]
 *   dq, dk, dv device outputs (overwritten), dtype of desc
 *   d_ws       device, bwd_ws_bytes
 */
stp_status stp_attn_bwd(const stp_attn_desc* desc, const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* d_o,
                        const int32_t* d_subtree_end, const void* d_tile_meta, void* dq,
                        void* dk, void* dv, void* d_ws, void* stream);

/*
 * stp_attn_step_host -- stp_attn_fwd followed by stp_attn_bwd on HOST buffers:
 * uploads Q, K, V, dO, runs both passes and writes O, LSE, dQ, dK, dV back to
 * host memory.  The paper computes the same two passes on device tensors; the
 * host-buffer pipeline is a library convenience.  The heads split into
 * n_chunks groups of whole kv heads (n_kv_heads % n_chunks == 0, at most 16);
 * group c holds kv heads [c Hkv/n, (c+1) Hkv/n) and their query heads.  Groups
 * are independent problems, so the copies of one group run while the kernels
 * of another do (library-owned streams, created on the first call on a
 * device and kept).  Results equal those of stp_attn_fwd / stp_attn_bwd on the
 * whole problem: O, LSE, dK, dV bit for bit, dQ up to the order of its float
 * reductions.
 *   q, k, v, d_o       host, layouts of stp_attn_fwd / stp_attn_bwd; page-locked
 *                      memory lets the copies run asynchronously
 *   d_subtree_end,
 *   d_tile_meta        device, as for stp_attn_fwd (stp_classify already
 *                      enqueued on `stream`)
 *   o, lse, dq, dk, dv host outputs, layouts of stp_attn_fwd / stp_attn_bwd
 *   d_scratch          device, 256-byte aligned, scratch_bytes >=
 *                      stp_step_scratch_size(desc, n_chunks); its first 4
 *                      bytes receive the step's device error word (read it
 *                      with stp_device_status(d_scratch, stream, &st))
 * Ordering: the step starts where `stream` stands at the call and `stream`
 * waits for all of it, so outputs are valid once `stream` is synchronized.
 * Host buffers must stay alive and untouched until then.  Calls made from
 * several host threads on one device are serialized by the library; steps
 * that share a scratch must be ordered on one stream.
 * Errors: STP_EINVAL (NULL pointer, bad n_chunks, short or unaligned
 * scratch), the checks of stp_attn_fwd / stp_attn_bwd, STP_ECUDA.
 */
stp_status stp_step_scratch_size(const stp_attn_desc* desc, int32_t n_chunks,
                                 size_t* scratch_bytes);
stp_status stp_attn_step_host(const stp_attn_desc* desc, int32_t n_chunks, const void* q,
                              const void* k, const void* v, const void* d_o,
                              const int32_t* d_subtree_end, const void* d_tile_meta, void* o,
                              float* lse, void* dq, void* dk, void* dv, void* d_scratch,
                              size_t scratch_bytes, void* stream);

/*
 * Tree-aware top-k indexer ([P1] attention section, the sparse top-k indexer
 * variants: the indexer scores candidates from a query's own ancestor chain
 * only -- the interval check of the mask -- so keys of a sibling branch are
 * never proposed).  For query i of a packed row:
 *   score(i, j) = sum_h w[i, h] * max(q[i, h] . k[j], 0)  over visible j
 * and the selection is the top_k visible keys of largest score (ties to the
 * smaller key index), listed in ascending key order, padded with index -1 and
 * score -inf when fewer keys are visible.  Scores are bf16 products summed in
 * float32 on the tensor cores; the selection is exact on those float32 scores.
 */
typedef struct {
  int32_t n_rows;         /* R                                                  */
  int32_t row_len;        /* T, a multiple of 128, at most 131072               */
  int32_t n_heads;        /* H indexer heads, H * head_dim <= 512               */
  int32_t head_dim;       /* D: 64 or 128                                       */
  int32_t top_k;          /* k in [1, 4096]                                     */
  int32_t max_tile_pairs; /* as in stp_attn_desc; sizes the score workspace     */
} stp_index_desc;

/* Device workspace of stp_index_topk: 256 bytes + 64 KiB per tile pair. */
stp_status stp_index_workspace_size(const stp_index_desc* desc, size_t* ws_bytes);

/*
 *   q           device bf16 [R, T, H, D]     k  device bf16 [R, T, D]
 *   w           device float32 [R, T, H]     (per-query head weights)
 *   d_subtree_end, d_tile_meta   as for stp_attn_fwd: stp_classify already run
 *               with an stp_attn_desc of the same n_rows, row_len and
 *               max_tile_pairs
 *   topk_idx    device int32 [R, T, top_k]  (row-local key indices)
 *   topk_score  device float32 [R, T, top_k]
 *   d_ws        device, stp_index_workspace_size bytes, 256-byte aligned; its
 *               first word is the device error word (stp_device_status)
 */
stp_status stp_index_topk(const stp_index_desc* desc, const void* q, const void* k, const float* w,
                          const int32_t* d_subtree_end, const void* d_tile_meta, int32_t* topk_idx,
                          float* topk_score, void* d_ws, void* stream);

/*
 * Next-token log-probabilities over packed rows ([P1] tree-build section: the
 * join copy keeps each trainable token's predecessor right before it in the
 * same row; materialization section: the loss mask marks those
 * predecessors).  For every position x = r * T + t with loss_mask[x] = 1:
 *   logprob[x] = h[x] . W[tok[x + 1]] - ln sum_v exp(h[x] . W[v])
 * and logprob[x] = 0 elsewhere.  The [positions, vocab] logits are never
 * stored: the products run on the tensor cores (bf16 in, float32 sums) and
 * the log-sum-exp is kept online in float32.
 */
typedef struct {
  int32_t n_rows;  /* R                                              */
  int32_t row_len; /* T, a positive multiple of 128; R * T <= 2^28   */
  int32_t hidden;  /* D, a multiple of 64 in [64, 16384]             */
  int32_t vocab;   /* V in [1, 2^24]                                 */
} stp_logprob_desc;

/* Device workspace of stp_logprob_gather: 512 bytes + 8 bytes per 128-position
 * tile + 12 * min(ceil(V / 256), 64) bytes per position (256-byte rounded). */
stp_status stp_logprob_workspace_size(const stp_logprob_desc* desc, size_t* ws_bytes);

/*
 *   hidden       device bf16 [R * T, D], 16-byte aligned (h, one row per position)
 *   w_vocab      device bf16 [V, D], 16-byte aligned (W, the vocabulary projection)
 *   d_token_ids  device int32 [R * T] (tok; read at x + 1 for each loss position x)
 *   d_loss_mask  device uint8 [R * T], nonzero = loss position
 *   logprob      device float32 [R * T], written in full
 *   d_ws         device, stp_logprob_workspace_size bytes, 256-byte aligned;
 *                its first word is the device error word (stp_device_status)
 * All buffers are the caller's; the call only enqueues work on `stream`.
 * Errors: STP_EINVAL / STP_EUNSUPPORTED for the descriptor, NULL or unaligned
 * pointers; STP_ECUDA.  A loss position that is the last of its row, or
 * whose target lies outside [0, V), sets the device error word
 * (stp_device_status then reports STP_EDEVICE) and its logprob is invalid.
 */
stp_status stp_logprob_gather(const stp_logprob_desc* desc, const void* hidden, const void* w_vocab,
                              const int32_t* d_token_ids, const uint8_t* d_loss_mask, float* logprob,
                              void* d_ws, void* stream);

/*
 * Tree-aware Gated DeltaNet layer core, forward ([P1] GDN section; [P3] the
 * Gated DeltaNet paragraphs).  The recurrent state is threaded along each
 * token's own path: forked at every branch point (a child segment starts
 * from its parent segment's final state), zero at every root; the short
 * convolution reads the previous tokens of the same path, so the parent's
 * last inputs are handed to each child.  Per token x of a packed row and
 * head h, with the path x_0 .. x_t = x:
 *   y        = SiLU(sum_{i=0..3} conv_w[:, i] * x_in[path token t-3+i])  (zero before the root)
 *   q, k, v  = channel blocks [0, Hd), [Hd, 2Hd), [2Hd, 3Hd) of y, split into
 *              heads of d; q, k scaled to unit norm (1 / sqrt(|.|^2 + 1e-6))
 *   S_x      = alpha S_prev + beta k (v - alpha S_prev^T k)^T,  alpha = exp(g[x, h])
 *   o[x, h]  = scale * S_x^T q                                  (S: [d, d], k-major)
 * equal, token for token, to the layer run on every sequence unpacked.
 * Computed chunk-wise (64 tokens per chunk) on the tensor cores: q, k, v and
 * the per-chunk operands are bf16, products are summed in float32, and the
 * state is kept in float32 between chunks.
 */
typedef struct {
  int32_t n_rows;    /* R                                                        */
  int32_t row_len;   /* T; R * T <= 2^26                                         */
  int32_t n_heads;   /* H in [1, 64] (q, k and v heads alike)                   */
  int32_t head_dim;  /* d; must be 128                                           */
  float scale;       /* output scale, e.g. 1 / sqrt(d)                           */
} stp_gdn_desc;

/* Upper bound of the plan size in bytes (from R and T only). */
stp_status stp_gdn_plan_bound(const stp_gdn_desc* desc, size_t* plan_bytes);

/*
 * Host planner: from subtree_end (host int32 [R, T], as written by
 * stp_plan_write) and the number of real tokens of each row (host int32 [R],
 * or NULL when no row holds pads; tokens at or past it are pads, which get
 * o = 0), writes the plan into `plan` (host, >= stp_gdn_plan_bound bytes):
 * the path predecessor of every token and its successors (the tokens whose
 * predecessor it is), the segments sorted by depth with their parents, and
 * the 64-token chunks.  Segments end at branch points; a root run of at least
 * 32 chunks is also cut once, after its first 16 chunks (the rest is its only
 * child), which changes no chunk and no result, only how the forward overlaps
 * the preparation of later chunks with the walk.  Its word 5 is the number of int32
 * words used; copy at least that much to the device for stp_gdn_fwd.
 * Errors: STP_EINVAL (NULL, short buffer, subtree_end outside [x, T) or not
 * nested, row_used outside [0, T]).
 */
stp_status stp_gdn_plan(const stp_gdn_desc* desc, const int32_t* subtree_end, const int32_t* row_used,
                        void* plan, size_t plan_bytes);

/* Device workspace of stp_gdn_fwd for a given host plan. */
stp_status stp_gdn_workspace_size(const stp_gdn_desc* desc, const void* plan, size_t* ws_bytes);

/*
 *   plan        host plan from stp_gdn_plan (launch sizes are read from it)
 *   d_plan      device copy of the same plan, 256-byte aligned
 *   x           device bf16 [R * T, 3 H d] (the projected q | k | v inputs), 16-byte aligned
 *   conv_w      device float32 [3 H d, 4] (tap 3 multiplies the token itself)
 *   g, beta     device float32 [R * T, H] (log decay <= 0, and the write strength)
 *   o           device float32 [R * T, H, d], written in full
 *   d_ws        device, stp_gdn_workspace_size bytes, 256-byte aligned; its
 *               first word is the device error word (stp_device_status)
 * The call enqueues 2 + (number of depths) kernels on `stream`.
 * Errors: STP_EINVAL / STP_EUNSUPPORTED for the descriptor, NULL or
 * unaligned pointers, a plan that is not one; STP_ECUDA.
 */
stp_status stp_gdn_fwd(const stp_gdn_desc* desc, const void* plan, const void* d_plan, const void* x,
                       const float* conv_w, const float* g, const float* beta, float* o, void* d_ws,
                       void* stream);

/*
 * Training: the same forward, keeping every chunk's starting state in the
 * workspace (stp_gdn_train_workspace_size bytes) for stp_gdn_bwd.
 */
stp_status stp_gdn_train_workspace_size(const stp_gdn_desc* desc, const void* plan, size_t* ws_bytes);
stp_status stp_gdn_fwd_train(const stp_gdn_desc* desc, const void* plan, const void* d_plan, const void* x,
                             const float* conv_w, const float* g, const float* beta, float* o, void* d_ws,
                             void* stream);

/*
 * Backward of the layer core for L = sum d_o . o ([P1] GDN section: a child
 * segment starts from its parent's final state, so the parent's final-state
 * gradient is the sum over its children).  Call after stp_gdn_fwd_train
 * with the same plan, inputs and workspace, on the same stream.
 *   d_o       device float32 [R * T, H, d], 16-byte aligned
 *   dx        device float32 [R * T, 3 H d], written in full (pads 0)
 *   dconv_w   device float32 [3 H d, 4], written in full
 *   dg, dbeta device float32 [R * T, H], written in full (pads 0)
 * The contractions run on the tensor core (bf16 operands, float32
 * accumulation, from the forward's bf16 chunk operands); every output is
 * summed in one fixed order (no float atomics), so repeated calls give the
 * same bits.  Device-side checks are OR-ed into the workspace's error word,
 * which stp_gdn_fwd_train clears: after the pair, stp_device_status on d_ws
 * reports a failure of either call.  Errors as for stp_gdn_fwd.
 */
stp_status stp_gdn_bwd(const stp_gdn_desc* desc, const void* plan, const void* d_plan, const void* x,
                       const float* conv_w, const float* g, const float* beta, const float* d_o, float* dx,
                       float* dconv_w, float* dg, float* dbeta, void* d_ws, void* stream);

/*
 * Read the device error word of a workspace (fwd_ws or bwd_ws): synchronizes
 * the stream, then *out = STP_OK or STP_EDEVICE (a device check tripped or a
 * bounded wait ran out; the kernel returned early and its outputs are invalid).
 * The word is cleared by the next call that uses the workspace.
 */
stp_status stp_device_status(const void* d_ws, void* stream, stp_status* out);

/* Thread-local text of the last error (empty string if none). */
const char* stp_last_error(void);

/* Library version string. */
const char* stp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* STP_H_ */
