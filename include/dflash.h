/*
 * dflash.h -- C ABI of the GB300 DFlash drafter round.
 *
 * The DFlash drafter (memra_engine::dflash module summary) is a small
 * Qwen3-class transformer that drafts a block of 16 tokens in ONE non-causal
 * forward, conditioned on the target model's hidden states at n tapped layers
 * (concatenated, then fc, then hidden_norm).  A drafting round has two halves:
 *
 *   dflash_ingest_ctx     appends newly committed context rows to the
 *                         per-layer draft KV cache (memra_engine::dflash::
 *                         DflashDraft, items ctx_features and ingest_ctx);
 *   dflash_forward_round  runs the 16 block rows through every layer over the
 *                         cached context K/V and returns the final normed
 *                         hidden states (DflashDraft, item forward_round).
 *
 * dflash_forward_full is the first-light path of the DflashDraft page (item
 * ctx_features, whose text carries the forward contract): context K/V are
 * recomputed on every call and no cache state is touched.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Device pointers are CUDA device addresses on the device that was
 *    current when dflash_create ran; host pointers are ordinary host memory
 *    that the call reads before it returns.
 *  - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *    void*, NULL = the legacy default stream).  Calls on one handle must be
 *    issued on one stream, or ordered by the caller.
 *  - Device f32 row buffers (taps, noise_emb, out) start on a 16-byte
 *    boundary (rows are moved as float4); a misaligned one is rejected with
 *    DFLASH_ERR_INVALID_ARG.  So do bf16 and e4m3 weight matrices
 *    (re-blocked at dflash_create with 16-byte moves).
 *  - The library never allocates device memory: the caller allocates the
 *    workspace (dflash_workspace_bytes) and owns every buffer.
 *  - Every call validates all of its arguments before it launches anything.
 *    On error it changes no state and returns a negative DFLASH_ERR_* code;
 *    dflash_last_error() gives a message (thread-local).  This mirrors the
 *    Result<_, Box<dyn Error>> of every DflashDraft method.
 *  - Layouts are row-major.  Weights are [out_features, in_features] (the
 *    nn.Linear convention of the checkpoint that DflashDraft::load reads);
 *    head h of a projection occupies rows [h*d, (h+1)*d); tap k occupies
 *    taps columns [k*H, (k+1)*H).
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dflash_handle dflash_t;

enum dflash_status {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = -1,  /* bad pointer, shape, id or count           */
  DFLASH_ERR_CAPACITY = -2,     /* pages, rows, batch or workspace too small  */
  DFLASH_ERR_CUDA = -3,         /* a CUDA runtime call failed                 */
  DFLASH_ERR_TIMEOUT = -4,      /* a bounded device-side wait gave up         */
  DFLASH_ERR_UNSUPPORTED = -5   /* a shape or format this build does not run  */
};

enum dflash_dtype { DFLASH_F32 = 0, DFLASH_BF16 = 1, DFLASH_FP8_E4M3 = 2 };
enum dflash_rope { DFLASH_ROPE_PLAIN = 0, DFLASH_ROPE_YARN = 1 };

/* e4m3 KV cache (the FP8 block attention named on the dflash_head page;
 * its storage format is not given there, this library's reading): every
 * cached K and V head row (one layer, one position, one kv head, d values)
 * is stored as OCP E4M3 codes with one f32 scale s = max|x| / 448 (an
 * all-zero row takes s = 1), each code the round-to-nearest-even,
 * saturating e4m3 value of x / s taken in f32.  The round's block K/V rows
 * pass through the same format, and so do its queries (one scale per token
 * and q head): the scores run on e4m3 tensor cores, the P V product in f16
 * with V decoded exactly from its codes.  The cache holds half the bytes of
 * a bf16 cache plus 4 bytes per row and kv head. */

/* Drafter shape and capacity (the pages' DflashCfg plus storage sizes). */
typedef struct dflash_config {
  int32_t n_layers;      /* L                                              */
  int32_t hidden;        /* H, a multiple of 128, at most 8192             */
  int32_t n_heads;       /* Hq query heads                                 */
  int32_t n_kv_heads;    /* Hkv, divides Hq, Hq/Hkv <= 8                   */
  int32_t head_dim;      /* d: 64 or 128                                   */
  int32_t intermediate;  /* I (SwiGLU), a multiple of 64                   */
  int32_t n_taps;        /* n tapped target layers                         */
  int32_t block;         /* b, must be 16                                  */
  double rms_eps;        /* RMSNorm epsilon                                */
  double rope_theta;     /* RoPE base                                      */
  int32_t rope_type;     /* DFLASH_ROPE_PLAIN or DFLASH_ROPE_YARN          */
  int32_t yarn_original_max_pos;
  double yarn_factor, yarn_beta_fast, yarn_beta_slow;
  int32_t weight_dtype;  /* DFLASH_F32, DFLASH_BF16 or DFLASH_FP8_E4M3     */
  int32_t kv_dtype;      /* DFLASH_F32 (f32 weights), DFLASH_BF16, or
                            DFLASH_FP8_E4M3 (bf16/e4m3 weights, head_dim
                            128): see "e4m3 KV cache" below               */
  int32_t page_size;     /* KV page rows, must be 64                       */
  int32_t max_seqs;      /* sequence slots: ids 0 .. max_seqs-1            */
  int32_t max_pages;     /* pages in the shared pool (all seqs, all calls) */
  int32_t max_seq_len;   /* committed rows + 16 a sequence may reach       */
  int32_t max_batch;     /* n_seq per dflash_forward_round, <= 64          */
  int32_t max_ingest_rows; /* sum of t per dflash_ingest_ctx, <= 512       */
  int32_t conv_groups;   /* DFlash2: channel groups of the grouped dynamic
                            causal conv around every sublayer (divides H,
                            H / conv_groups a multiple of 4, at most 256);
                            0 = DFlash (no conv)                            */
} dflash_config;

/* One decoder layer's tensors (DflashLayer).  Projections have the dtype
 * weight_dtype; *_scale are per-output-row f32 scales, required for
 * DFLASH_FP8_E4M3 and ignored otherwise (spark_model::layers::dflash_head,
 * DflashQuantization).  Norm gains are f32. */
typedef struct dflash_layer_weights {
  const void *q, *k, *v, *o, *gate, *up, *down;
  const float *q_scale, *k_scale, *v_scale, *o_scale, *gate_scale, *up_scale, *down_scale;
  const float *q_norm;    /* [d]  */
  const float *k_norm;    /* [d]  */
  const float *input_ln;  /* [H]  */
  const float *post_ln;   /* [H]  */
  /* DFlash2 (conv_groups = Gc > 0), sublayer s = 0 attention, 1 MLP
   * (memra_engine::dflash Dflash2Conv; DflashDraft d2_conv_prepare /
   * d2_conv_finish): conv_base[s] f32
   * [2][H][2] (half 0 wraps the sublayer input, half 1 its output; tap 0
   * weighs the previous block row, tap 1 this row); conv_dyn[s] the
   * dynamic-coefficient projection [4 Gc][H] in weight_dtype, output row
   * (half * Gc + group) * 2 + tap (+ conv_dyn_scale[s] [4 Gc] for e4m3).
   * Ignored when conv_groups is 0. */
  const float *conv_base[2];
  const void *conv_dyn[2];
  const float *conv_dyn_scale[2];
} dflash_layer_weights;

/* Backbone tensors (DflashDraft fields fc, hidden_norm, norm, layers): no fc
 * bias, no embedding or lm_head (the round reuses the target's). */
typedef struct dflash_weights {
  const void *fc;                     /* [H, n_taps*H]                   */
  const float *fc_scale;              /* [H] for fp8                     */
  const float *hidden_norm;           /* [H]                             */
  const float *norm;                  /* [H]                             */
  const dflash_layer_weights *layers; /* host array of n_layers          */
} dflash_weights;

/* Bytes of device workspace the handle needs for this config (256-byte
 * aligned start required).  It is the one allocation behind three items of
 * the pages: the per-layer draft KV cache (memra_engine::dflash, struct
 * DflashKv; paged with one block table shared by the layers as in
 * spark_model::layers::dflash_head, struct DflashProposerState), the
 * per-step scratch of the block forward (dflash_head, struct DflashScratch)
 * and the weights.  It holds the repacked weights, the paged KV pools, page
 * tables, activations and reduction scratch.  bf16 weights are stored as
 * 16 KB blocks for the tensor cores, e4m3 weights as 8 KB units of one byte
 * per weight (widened to f16 inside the projections; their per-row scales
 * are applied to the projections' sums), f32 weights as given.  A config
 * that dflash_create would reject fails here with the same code
 * (DFLASH_ERR_INVALID_ARG or DFLASH_ERR_UNSUPPORTED). */
int dflash_workspace_bytes(const dflash_config *cfg, size_t *bytes);

/* Validate cfg, carve the caller's workspace, copy and repack the weights
 * into it (the caller may free its weight buffers once the stream has
 * passed this call), resolve every kernel once and build the RoPE table.
 * Resolving the kernels once here, so that every later call only launches,
 * is the dflash_head page's struct DflashKernels (handles resolved once at
 * from_weights, each propose() only launches).  The workspace stays owned
 * by the caller and must outlive the handle; the handle itself is host
 * memory freed by dflash_destroy.  Returns a handle in *out; on error *out
 * is left untouched and nothing was launched. */
int dflash_create(const dflash_config *cfg, const dflash_weights *w, void *workspace,
                  size_t workspace_bytes, void *stream, dflash_t **out);

/* Append newly committed context rows to n_seq sequences (DflashDraft,
 * ctx_features then ingest_ctx): per row, feats = hidden_norm(fc(taps)); per
 * layer K = rope(k_norm(W_k feats)) * mscale and V = W_v feats are written at
 * rows len .. len+t-1 of that sequence, then len += t.
 *   seq_ids   host [n_seq]  distinct slot ids
 *   t_per_seq host [n_seq]  rows per sequence (0 allowed)
 *   pos_new   host [sum t]  absolute positions, sequence by sequence
 *   taps      device f32 [sum t, n_taps*H], rows in the same order */
int dflash_ingest_ctx(dflash_t *h, int32_t n_seq, const int32_t *seq_ids,
                      const int32_t *t_per_seq, const int32_t *pos_new,
                      const float *taps, void *stream);

/* One drafting forward of the 16-row block of each of n_seq sequences over
 * its cached context (DflashDraft, forward_round).  Block K/V land in the
 * cache rows len .. len+15 for the duration of the call only; len is not
 * changed.
 *   seq_ids   host [n_seq]
 *   pos_block host [n_seq, 16] absolute positions of the block rows
 *   noise_emb device f32 [n_seq, 16, H] (target embeddings of the block)
 *   out       device f32 [n_seq, 16, H] final normed hidden states */
int dflash_forward_round(dflash_t *h, int32_t n_seq, const int32_t *seq_ids,
                         const int32_t *pos_block, const float *noise_emb,
                         float *out, void *stream);

/* First-light forward: full non-causal attention over [ctx features ;
 * block] with the context K/V recomputed (no cache state touched).
 *   taps      device f32 [ctx, n_taps*H]
 *   noise_emb device f32 [16, H]
 *   pos       host [ctx + 16]: ctx rows' positions then the block rows'
 *   out       device f32 [16, H] */
int dflash_forward_full(dflash_t *h, int32_t ctx, const float *taps, const float *noise_emb,
                        const int32_t *pos, float *out, void *stream);

/* dflash_forward_full with its context K/V in a fixed device region compiled
 * into the library (16 MiB per device) instead of pages of the handle's KV
 * pool.  The pages have no counterpart of this entry point; it exists for
 * callers that cannot allocate: when every pool page belongs to a live
 * sequence, dflash_forward_full fails with DFLASH_ERR_CAPACITY, and more
 * pages would take a larger workspace -- a new device allocation plus a copy
 * of every live page.  This call uses no pool page and no buffer beyond its
 * arguments and the handle's workspace, and allocates nothing.
 *
 * Arguments, layouts and results are those of dflash_forward_full; no
 * sequence state changes.
 *
 * Limit: ctx + 16 rows must fit floor(16 MiB / (2 * L * Hkv * 64 * row))
 * pages of 64 rows, row = d * kv_bytes + (e4m3 KV ? 4 : 0) bytes (an e4m3
 * row carries its f32 scale) -- 16 pages, 1008 context rows, for the
 * 8-layer, 4-kv-head, head_dim-128 drafter with a bf16 KV cache; 31 pages,
 * 1968 rows, with an e4m3 one.  A larger ctx is rejected with
 * DFLASH_ERR_CAPACITY before anything is launched.  The current device must
 * be the handle's (the one current at dflash_create), else
 * DFLASH_ERR_INVALID_ARG.
 *
 * Set-up: the first call on a device (with that device current) looks the
 * region's address up once (cudaGetSymbolAddress; a failure returns
 * DFLASH_ERR_CUDA); make that first call before any stream capture.  The
 * region is zero when the library is loaded and calls write only finite
 * values into it (rows past the last key of a last page are read by the
 * attention and masked, so they must stay finite).  One region serves every
 * handle on that device in the process: calls that overlap in time (other
 * streams, threads or handles) race on it and must be serialised by the
 * caller. */
int dflash_forward_full_static(dflash_t *h, int32_t ctx, const float *taps, const float *noise_emb,
                               const int32_t *pos, float *out, void *stream);

/* Greedy draft tokens through the target model's lm_head (the pages'
 * DflashDraft page: the drafter reuses the target's lm_head on its block
 * rows; module index, dflash2_walk_greedy: argmax, lowest index on ties).
 *
 * The lm_head is packed once into a caller buffer of dflash_lm_head_bytes
 * (the library never allocates): vocab weight blocks for the tensor-core
 * projection, then a logits scratch of max_batch*16 rows.  Requires bf16 or
 * e4m3 drafter weights (the tensor-core path); vocab a multiple of 128.
 *
 *   dflash_lm_head_bytes  bytes of the packed buffer for `vocab` rows.
 *   dflash_pack_lm_head   lm_head: device bf16 [vocab, H] row-major, read
 *                         during the call; packed: device, 256-byte aligned.
 *   dflash_draft_tokens   hidden: device f32 [n_seq, 16, H] (16-byte aligned;
 *                         e.g. forward_round's out); tokens: device int32
 *                         [n_seq, 16].  Logits are f32-accurate sums of bf16
 *                         weights times the f32 rows (hi/lo split).  Calls
 *                         sharing one packed buffer must not overlap (its
 *                         logits scratch is reused). */
int dflash_lm_head_bytes(const dflash_t *h, int32_t vocab, size_t *bytes);
int dflash_pack_lm_head(dflash_t *h, const void *lm_head, int32_t vocab, void *packed, size_t bytes, void *stream);
int dflash_draft_tokens(dflash_t *h, int32_t n_seq, const float *hidden, const void *packed, int32_t vocab,
                        int32_t *tokens, void *stream);

/* Attention work plan (inspection; host only, no handle, no device).  The
 * block attention of a round runs over each sequence's [cached context ;
 * 16 block rows] (memra_engine::dflash::DflashDraft, forward_round) as work
 * items (sequence, kv head, split of split_pages 64-row pages), numbered in
 * that order; a round with these lengths plans them exactly so:
 *   cfg           as for dflash_create (same validation, same errors);
 *   n_sm          SMs of the device (0: the current device's count);
 *   lens          host int64 [n_seq]: committed rows of each sequence
 *                 (0 .. max_seq_len - 16), n_seq in 1..max_batch;
 *   kstart        host int64 [n_seq] or NULL (all 0): first attended row of
 *                 each sequence (the context window's start, 0 .. lens[i]);
 *   split_pages   out: pages per split (items cover the pages from the one
 *                 holding kstart through the block rows);
 *   n_items       out: work items of the round;
 *   item0         out (or NULL): host int32 [n_seq + 1], the first item of
 *                 each sequence and n_items last;
 *   launch_order  out (or NULL): host int32 [max_items], the item each
 *                 attention CTA runs, longest first (ties in item order).
 * The split size is the one whose list schedule (items launched in that
 * order, each to the SM that frees first) finishes first among a few
 * candidates.  DFLASH_ERR_CAPACITY when the items exceed the round's
 * scratch (forward_round refuses such a round the same way) or
 * launch_order is shorter than n_items; split_pages and n_items are set
 * either way. */
int dflash_attention_plan(const dflash_config *cfg, int32_t n_sm, int32_t n_seq, const int64_t *lens,
                          const int64_t *kstart, int32_t *split_pages, int32_t *n_items, int32_t *item0,
                          int32_t *launch_order, int32_t max_items);

/* Context window (spark_model::layers::dflash_head, dflash_ctx_cap: the
 * most recent target positions the drafter may accumulate and attend to).
 * cap = 0: unbounded (the default).  cap > 0: after every ingest a sequence
 * keeps only its most recent `cap` context positions -- pages wholly older
 * return to the pool, and the attention masks the older keys of the first
 * kept page -- and rounds attend to [len - cap, len) plus the block rows.
 * Setting the cap applies it to every sequence at once; positions already
 * dropped stay dropped when the cap is raised or cleared.  dflash_seq_len
 * still counts every committed position (RoPE positions keep growing);
 * dflash_kv_read rejects rows of dropped pages.  dflash_forward_full is not
 * windowed (the first-light forward attends to its whole context). */
int dflash_set_ctx_cap(dflash_t *h, int32_t cap);

/* Drop a sequence's cache (len = 0, pages back to the pool): a fresh
 * DflashKv (memra_engine::dflash, struct DflashKv) for slot seq_id, whose
 * pages return to the shared pool of the dflash_head page's
 * DflashProposerState.  Host-side bookkeeping only (no launch, no stream);
 * a null handle or an id out of [0, max_seqs) fails with
 * DFLASH_ERR_INVALID_ARG. */
int dflash_seq_reset(dflash_t *h, int32_t seq_id);

/* Committed rows of a sequence: the append-only len of its DflashKv
 * (memra_engine::dflash, struct DflashKv: block rows land transiently at
 * [len, len + 16) each round and are never committed, so len counts only
 * ingested context rows).  Written to *len on the host; a null argument or
 * an id out of [0, max_seqs) fails with DFLASH_ERR_INVALID_ARG. */
int dflash_seq_len(dflash_t *h, int32_t seq_id, int64_t *len);

/* Copy cached rows row0 .. row0+nrows-1 of one layer of a sequence out of
 * the paged pools as f32: k_out, v_out device [nrows, Hkv, d] (K normed and
 * roped, V raw; an e4m3 cache returns code times scale).  Inspection entry
 * point for tests. */
int dflash_kv_read(dflash_t *h, int32_t seq_id, int32_t layer, int32_t row0, int32_t nrows,
                   float *k_out, float *v_out, void *stream);

/* Synchronise the handle's last stream and report the device error word
 * (0 = none; else a DFLASH_ERR_* code a kernel recorded: DFLASH_ERR_TIMEOUT
 * when a bounded device-side wait gave up).  A reported error is cleared,
 * so the next call reports only what happens after it. */
int dflash_device_status(dflash_t *h, void *stream);

/* Failure-path self-test: launch one bounded wait on a device barrier that
 * nothing arrives on; after limit_ms (1..2000) of device time the kernel
 * records DFLASH_ERR_TIMEOUT in the error word and returns (no trap, the
 * context stays usable), which the next dflash_device_status reports. */
int dflash_selftest_wait_timeout(dflash_t *h, int32_t limit_ms, void *stream);

/* Kernel kinds reported by the measurement calls below. */
enum dflash_kernel_kind {
  DFLASH_KERNEL_GEMM = 0,       /* weight-streaming projections (fc, K/V, QKV, O, gate/up, down) */
  DFLASH_KERNEL_ATTENTION = 1,  /* split-KV block attention over the paged cache                 */
  DFLASH_KERNEL_COMBINE = 2,    /* merge of the split-KV partial softmaxes                        */
  DFLASH_KERNEL_INIT = 3,       /* per-call descriptor upload and residual / operand set-up       */
  DFLASH_KERNEL_NORM = 4,       /* final RMSNorm                                                  */
  DFLASH_KERNEL_FINISH = 5,     /* element-wise steps between projections (norm operands, q/k
                                   head-norm + RoPE and block K/V rows, SwiGLU)                   */
  DFLASH_KERNEL_KINDS = 6
};

/* Measurement (not needed to draft).  While enabled, every kernel launch
 * of the handle is bracketed by a CUDA event pair on its stream, tagged with
 * the launch's algorithmic bytes (weights, cached K/V, operands and outputs
 * it must move).  Enabling or disabling discards earlier records (it
 * synchronises the device if records exist). */
int dflash_profile_enable(dflash_t *h, int32_t enable);

/* Totals over the records of one kernel kind: launches, summed device time
 * in ms and summed algorithmic bytes (waits for the recorded events). */
int dflash_profile_read(dflash_t *h, int32_t kind, int64_t *launches, double *ms, double *bytes);

/* Launch trace (measurement).  While a buffer is set, every kernel launch of
 * the handle writes, per CTA, 16 u64 words into the next free region of
 * `device_buffer`: word 0 the SM id, word 1 the %globaltimer (ns) at entry,
 * word 15 the %globaltimer at exit (the latest of the CTA's warps' finishing
 * stamps, so a warp still draining counts); the tensor-core projection and attention
 * kernels also write words 2..14: SM clock cycles since entry at fixed
 * points of the kernel (set-up done, launch wait passed, last MMA issued,
 * epilogue steps, exit) or cycle counts spent waiting (projection points 9,
 * 11, 12: producer waiting for free stages, first MMA issuer waiting for
 * loaded stages and for a free accumulator).  Unused words stay as they
 * were.  Rounds still run as CUDA graphs while tracing, each captured afresh
 * with its own trace regions.  Launches that no longer fit are not traced.
 * NULL stops tracing (after a device synchronisation when traced rounds
 * ran).  The buffer is the caller's; the library never reads it. */
int dflash_trace_begin(dflash_t *h, void *device_buffer, size_t bytes);

/* Traced launches so far: kernel kind (dflash_kernel_kind), CTA count and the
 * word offset of each launch's region, up to max_launches entries;
 * *n_launches gets the total. */
int dflash_trace_launches(dflash_t *h, int32_t max_launches, int32_t *kinds, int32_t *grids, int64_t *offsets,
                          int32_t *n_launches);

/* Kernel launches issued by the handle since it was created. */
int dflash_launch_count(dflash_t *h, int64_t *launches);

/* Release the handle (the workspace stays the caller's). */
void dflash_destroy(dflash_t *h);

/* Message of the last failed call on this thread ("" if none). */
const char *dflash_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
