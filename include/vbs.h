/*
 * libvbs: one step of batched beam search over a vocabulary, the KV-cache
 * reorder that follows it, and the verify/accept step of blockwise parallel
 * decoding, as a C ABI for one NVIDIA GB300 (sm_103a).
 *
 * Sources of the operations (cited by page title and section):
 *   [BS] "Transformers中的Beam Search高效实现" (zhuanzhi.ai), section
 *        多个样本同时进行beam search: the batched step, BeamHypotheses, padding,
 *        the final choice.
 *   [LM] "9.2 贪心搜索与束搜索：确定性与近似搜索" (llm_internals): §9.2.2 the four
 *        sub-steps, the KV reorder paragraph and "何时结束"; §9.2.3 the length
 *        penalty; §9.2.4 prompt sharing.
 *   [BPD] "Blockwise Parallel Decoding for Deep Autoregressive Models"
 *        (papercache notes): §3 predict / verify / accept; §4 the combined
 *        scoring and proposal model.
 *   [LS] "推荐一款超高速、多特性的高性能序列推理引擎—— LightSeq": "层级式解码计算"
 *        names this path (vocabulary softmax, beam selection, cache refresh).
 *
 * Conventions for every call:
 *   - Return value: VBS_OK (0) or a negative VBS_E* status; vbs_strerror()
 *     names it.  Arguments are checked on the host before anything is
 *     launched; a call that returns an error has launched nothing, except
 *     VBS_ECUDA (the launch itself failed).
 *   - Pointers marked "device" are CUDA device pointers owned by the caller.
 *     The library reads and writes them only in work it enqueues on the
 *     stream given to the call (or to the context's init); they must stay
 *     valid until that work completes.  No call synchronises the stream unless
 *     its comment says so.  No call after an init allocates device memory.
 *   - Errors found on the device (bad input values, an exhausted block pool,
 *     a wait that gave up) are recorded in a status word of the context and
 *     reported by the *_status() calls; the kernels never trap.
 *   - Logits are row-major with a row stride `ld` (elements) >= V; dtype is
 *     VBS_F32 or VBS_BF16.  Logits must be finite or -inf, with at least one
 *     finite value per row that is read.
 *   - Devices: every call works on the device current on the calling thread,
 *     and the stream it is given must belong to that device.  The kernels'
 *     shared-memory attributes are set once per device, and the library's
 *     static device memory (bs_expand_static's scratch, bpd_verify's queue,
 *     the status word of the calls without a context) exists once per device.
 *     The bench runs one process per GPU.
 */
#ifndef VBS_H
#define VBS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* vbs_stream_t; /* the same type as cudaStream_t */

enum {
  VBS_OK = 0,
  VBS_EINVAL = -1,   /* an argument is out of range or inconsistent */
  VBS_ECUDA = -2,    /* a CUDA runtime call or kernel launch failed */
  VBS_ENOMEM = -3,   /* device memory (init) or the paged block pool (step) ran out */
  VBS_ESTATE = -4,   /* the call does not fit the context's state (e.g. more than max_len steps) */
  VBS_EALIGN = -5,   /* a pointer or stride is not aligned as the call needs */
  VBS_ETIMEOUT = -6, /* a bounded device-side wait gave up */
  VBS_EINPUT = -7,   /* the input data broke a precondition (NaN / +inf logits, ...) */
  VBS_ESCRATCH = -8, /* the problem is larger than bs_expand_static's static scratch allows */
  VBS_EBOUNDS = -9   /* a device bounds check failed (only the checked build, libvbs_checked.so, checks) */
};

enum { VBS_F32 = 0, VBS_BF16 = 1 };
/* length penalty ([LM] §9.2.3): GNMT ((5+|y|)/6)^alpha, or |y|^alpha */
enum { VBS_LP_GNMT = 0, VBS_LP_POWER = 1 };
/* early_stopping ([LM] §9.2.2 "何时结束"): False (heuristic), True (stop when W
   hypotheses are finished), "never" (stop only when no live beam can overtake) */
enum { VBS_ES_FALSE = 0, VBS_ES_TRUE = 1, VBS_ES_NEVER = 2 };

/* Name of a status code (static string, never NULL). */
const char* vbs_strerror(int status);
/* Library version, major * 10000 + minor * 100 + patch.  Never fails. */
int vbs_version(void);

/* =============================================================================
 * Batched beam search ([BS], [LM] §9.2.2-9.2.3)
 * ============================================================================= */
typedef struct vbs_bs vbs_bs;

/*
 * Create a beam-search context for `batch` sentences of W beams (R = batch*W
 * rows) over a vocabulary of V tokens; allocate every workspace it will use
 * (the streaming partials, the per-sentence finished sets, its own sequence
 * buffer) so that steps never allocate.
 *   eos            token that ends a hypothesis, or -1 for none
 *   alpha          length-penalty exponent ([LM] §9.2.3; 0 = no normalisation)
 *   early_stopping VBS_ES_*; lp_kind VBS_LP_*
 *   max_len        maximum number of steps (generated tokens); sequences have
 *                  max_len + 1 columns (BOS first)
 *   bos, pad       the BOS token of column 0 and the PAD token of finished rows
 *   dtype          VBS_F32 or VBS_BF16 logits
 *   stream         the stream all of this context's work is enqueued on
 * Limits: 1 <= W <= 16, V >= 2, 1 <= batch <= 32767, R*V < 2^31, 1 <= max_len.
 * Errors: VBS_EINVAL, VBS_ENOMEM, VBS_ECUDA.  *ctx is NULL on error.
 */
int bs_init(vbs_bs** ctx, int batch, int W, int V, int eos, double alpha, int early_stopping, int lp_kind,
            int max_len, int bos, int pad, int dtype, vbs_stream_t stream);

/*
 * Start a new decode ([BS]: beam_scores = 0 for beam 0 and -inf for the
 * others, input_ids = BOS): writes scores[R] (device, fp32) and seqs[R,
 * max_len+1] (device, int32, row-major; column 0 = BOS, the rest PAD), empties
 * the finished sets, clears the done flags and the step counter.
 * seqs may be NULL: the context then keeps the sequences in its own buffer
 * (bs_seqs() returns it), and every later call must also pass NULL.
 * Errors: VBS_EINVAL (NULL ctx or scores), VBS_ECUDA.
 */
int bs_reset(vbs_bs* ctx, float* scores, int32_t* seqs);

/*
 * One step for every sentence, in one kernel launch ([BS] loop body, [LM]
 * §9.2.2): row log-softmax of logits[R, V] (row stride ld elements, device),
 * add scores[r], rank each sentence's W*V candidates by (score desc, flat index
 * j = w*V + v asc), walk the best 2W: an EOS hit within the top W joins the
 * sentence's finished set with normalised score sum / lp(t) (t = this step's
 * number), an EOS hit at rank >= W is skipped, any other candidate becomes a
 * live beam until W are taken; then the sentence's stopping test runs once
 * with the best candidate score.  A sentence already finished before this step
 * emits score 0, token PAD and beam_idx -1 for its W rows.
 * Outputs (device): scores[R] (in/out, the new cumulative scores),
 *   beam_idx[R] (int32, the global parent row of each new row, -1 for a pad
 *   row), tokens[R] (int32), seqs (in/out: parents' rows gathered, token
 *   appended at column t; must be the buffer given to bs_reset), and, if
 *   all_done is not NULL, *all_done = 1 when every sentence is finished.
 * The logits are read once; a sentence already finished, and every row whose
 * score is -inf, is not read at all.
 * Errors: VBS_EINVAL (ld < V, NULL outputs), VBS_ESTATE (max_len steps already
 *   run, or a seqs pointer other than the one given to bs_reset), VBS_EALIGN
 *   never (unaligned logits take a slower element-wise path), VBS_ECUDA.
 */
int bs_step(vbs_bs* ctx, const void* logits, int64_t ld, float* scores, int32_t* seqs, int32_t* beam_idx,
            int32_t* tokens, int32_t* all_done);
/*
 * bs_step through the two-pass coarse selection of [LS] (an ablation, same
 * arguments and results): a first pass over each row computes its log-sum-exp
 * and R = the smallest of K group maxima (at most the row's K-th largest
 * logit; K = 2W), a second pass reads the row again and keeps the K best keys
 * among the logits >= R, then the per-sentence merge of bs_step runs.  It reads
 * the logits twice; bs_step reads them once.
 * Errors: those of bs_step.
 */
int bs_step_two_pass(vbs_bs* ctx, const void* logits, int64_t ld, float* scores, int32_t* seqs, int32_t* beam_idx,
                     int32_t* tokens, int32_t* all_done);
/*
 * Vocabulary shards (the row's logits split by column, e.g. across the ranks of
 * a vocabulary-parallel LM head): each shard reduces every row to a partial
 * (the shard's max, scaled sum of exponentials and its K = 2W best (logit,
 * token) keys, token ids global), the partials of all shards are exchanged
 * (the caller's job: one all-gather of bs_shard_partial_bytes() bytes per
 * shard), and one merge finishes the step exactly as bs_step would on the
 * whole rows (the row LSE is the log-sum-exp of the shards', the row's best 2W
 * come from the shards' lists).
 *   bs_shard_partial_bytes: the size of one shard's partial buffer.
 *   bs_step_shard: columns [v0, v0 + Vs) of the step's logits, logits_shard[R,
 *     ld] (device, row stride ld >= Vs), with the step's current scores (read
 *     only: rows of finished sentences and -inf scores are skipped); writes the
 *     partial to `partial` (device, 16-byte aligned).  Does not advance the step.
 *   bs_step_merge_shards: n_shards partials, contiguous ([n_shards][bytes],
 *     device), whose shards tile [0, V) (not checked); then as bs_step.
 *     n_shards <= min(256 / 2W, 128 / W) (VBS_EINVAL beyond).
 * Errors: VBS_EINVAL (NULL pointers; v0 < 0, Vs < 1, v0 + Vs > V or ld < Vs;
 *   n_shards out of range), VBS_EALIGN (partial not 16-byte aligned),
 *   VBS_ESTATE (no bs_reset yet, max_len steps already run, or another seqs
 *   buffer than bs_reset's), VBS_ECUDA.
 * The pages' vocabulary-parallel reading: the step reduces per row over V, so
 * per-shard (max, sum, top-2W) combine exactly; no pages' counterpart as calls.
 */
int bs_shard_partial_bytes(vbs_bs* ctx, int64_t* bytes);
int bs_step_shard(vbs_bs* ctx, const void* logits_shard, int64_t ld, int v0, int Vs, const float* scores,
                  void* partial);
int bs_step_merge_shards(vbs_bs* ctx, int n_shards, const void* partials, float* scores, int32_t* seqs,
                         int32_t* beam_idx, int32_t* tokens, int32_t* all_done);

/*
 * Final choice ([BS] after the loop): the live beams of every sentence not yet
 * finished are offered to its finished set with |y| = steps run; the winner is
 * the highest normalised score, ties going to the entry latest in the set's
 * insertion order.  out_seqs[batch, max_len+1] (device int32) gets BOS and the
 * winner's tokens, then EOS when shorter than max_len+1 columns, then PAD;
 * out_len[batch] the number of meaningful entries (EOS included);
 * out_score[batch] the winner's normalised score.  scores/seqs are the
 * buffers of the last bs_step (seqs NULL if the context keeps them).  The
 * context is not changed: finalize may be called more than once.
 * Errors: VBS_EINVAL (NULL pointers), VBS_ESTATE (no bs_reset yet, or another
 *   seqs buffer than bs_reset's), VBS_ECUDA.
 */
int bs_finalize(vbs_bs* ctx, const float* scores, const int32_t* seqs, int32_t* out_seqs, int32_t* out_len,
                float* out_score);
/*
 * bs_finalize returning the best n_return (1..W) hypotheses of every sentence
 * ([LM] §9.2.2: the first num_return_sequences by normalised score; [BS] pops
 * them from a stable ascending sort, so equal scores go latest-inserted
 * first).  Sentence b's j-th best is row b * n_return + j of out_seqs
 * [batch * n_return, max_len+1], out_len and out_score.  bs_finalize is the
 * n_return = 1 case.  Errors: those of bs_finalize; VBS_EINVAL for n_return
 * outside 1..W.
 */
int bs_finalize_n(vbs_bs* ctx, const float* scores, const int32_t* seqs, int n_return, int32_t* out_seqs,
                  int32_t* out_len, float* out_score);

/*
 * Copy the finished sets out (device buffers, for inspection):
 * count[batch] int32; ns[batch*W] double normalised scores; len[batch*W] int32
 * |y|; serial[batch*W] int32 insertion numbers (set order = ascending serial);
 * tokens[batch*W, max_len+1] int32 (the first len entries are BOS + tokens);
 * done[batch] int32.  Slots at or beyond count[b] are unused.  Any pointer may
 * be NULL to skip that array.  Errors: VBS_EINVAL (NULL ctx), VBS_ECUDA.
 */
int bs_finished(vbs_bs* ctx, int32_t* count, double* ns, int32_t* len, int32_t* serial, int32_t* tokens,
                int32_t* done);

/* The context's own sequence buffer [R, max_len+1] (device), used when bs_reset got NULL.
   Errors: VBS_EINVAL (NULL arguments). */
int bs_seqs(vbs_bs* ctx, int32_t** seqs);
/* Steps run since bs_reset.  Errors: VBS_EINVAL (NULL arguments). */
int bs_steps(vbs_bs* ctx, int* steps);
/* Synchronise the context's stream and return (then clear) its device status word:
   VBS_OK or the first VBS_E* a kernel recorded.  VBS_EINVAL for NULL, VBS_ECUDA when
   the synchronisation or the read fails. */
int bs_status(vbs_bs* ctx);
/* Free the context (synchronises its stream first). NULL is a no-op.  Returns VBS_OK. */
int bs_destroy(vbs_bs* ctx);

/*
 * One beam expansion with no context and no allocation.  The pages have no
 * counterpart: this exists for callers that cannot allocate device memory --
 * code running inside an allocator or a memory-pool callback, a host whose
 * memory budget is fixed up front, or an embedding runtime that forbids
 * cudaMalloc after start-up.
 *
 * Computes, for every sentence b of `batch` sentences of W beams, the W best
 * of log_softmax(logits[r, :]) + scores_in[r] over its W*V candidates, ranked
 * by (score desc, flat index j = w*V + v asc): exactly the beams bs_step would
 * keep when no token ends a hypothesis (eos = -1) and no sentence is finished.
 *   logits     [batch*W, V] device, row stride ld >= V elements, dtype VBS_*
 *   scores_in  [batch*W] device fp32 cumulative scores; a row at -inf is not read
 *   scores_out [batch*W] device fp32 new scores (may equal scores_in)
 *   beam_idx   [batch*W] device int32 global parent row; tokens [batch*W] int32
 * Scratch: a static device array of 4.5 MiB (the partial sums, partial top-K
 * lists and row maps), which every process that loads the library holds on
 * each device it uses until it exits.  Limit: batch*W <= 8192 rows, for any
 * 1 <= W <= 16 (the largest problem, 8192 rows at W = 16, needs 4,392,960
 * bytes of it), V >= 2, batch*W*V < 2^31; more rows return VBS_ESCRATCH
 * before anything is launched.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The call allocates nothing and frees nothing.  Every call shares
 * the one array and leaves its contents behind; each call rewrites what it
 * reads, but two calls that overlap on the GPU (different streams, or
 * different host threads) race on it and must be serialised by the caller.
 * Device-side errors go to the status word that vbs_stateless_status() reads.
 * Errors: VBS_EINVAL, VBS_ESCRATCH, VBS_ECUDA.
 */
int bs_expand_static(const void* logits, int64_t ld, int batch, int W, int V, int dtype, const float* scores_in,
                     float* scores_out, int32_t* beam_idx, int32_t* tokens, vbs_stream_t stream);

/* =============================================================================
 * KV-cache reorder ([LM] §9.2.2 KV paragraph; [LS] cache refresh)
 * ============================================================================= */

/* Geometry of a KV cache: layers L, KV heads H, head_dim D, positions t_max,
   elem_bytes per number.  Naive layout [L][2][rows][H][t_max][D] (K then V). */
typedef struct {
  int layers;
  int heads;
  int head_dim;
  int t_max;
  int elem_bytes;
} vbs_kv_desc;

/*
 * Naive reorder, out of place: for every row r with beam_idx[r] >= 0,
 * dst[l][kv][r][h][0:t_valid][:] = src[l][kv][beam_idx[r]][h][0:t_valid][:];
 * rows with beam_idx[r] = -1 are not written, positions >= t_valid neither.
 * src and dst (device) must not overlap.  beam_idx[rows] int32 (device).
 * Uses bulk (TMA) copies when head_dim * elem_bytes and both pointers are
 * 16-byte aligned, element copies otherwise.
 * Errors: VBS_EINVAL (t_valid > t_max, bad geometry, NULL), VBS_ECUDA.
 */
int kv_reorder(const vbs_kv_desc* desc, const void* src, void* dst, const int32_t* beam_idx, int rows,
               int t_valid, vbs_stream_t stream);

/*
 * Paged cache with copy-on-write ([LM] §9.2.2: rewrite block-table entries,
 * copy only when a shared block is written; §9.2.4 prompt sharing).
 * The pool (device, caller-owned) is [num_blocks][L][2][H][block][D], with
 * num_blocks = batch * blocks_per_sentence: sentence b owns blocks
 * [b*S, (b+1)*S) (blocks are never shared across sentences).  The library
 * owns the block table [R][max_blocks] int32 (row r's position p lives in pool
 * block table[r][p / block] at slot p % block), the reference counts and the
 * per-sentence free stacks.
 */
typedef struct vbs_pkv vbs_pkv;

/*
 * Create a paged cache for `batch` sentences of W rows over the caller's pool
 * (device, [batch * blocks_per_sentence][L][2][H][block][D] of desc's
 * elem_bytes): blocks_per_sentence blocks per sentence, `block` positions per
 * block, max_blocks table entries per row.  Allocates the table, counts, free
 * stacks, copy-task slots and the saved state once; later calls allocate
 * nothing.  All work goes to `stream`.
 * Errors: VBS_EINVAL (bad geometry, NULL pool, W outside 1..16, non-positive
 *   sizes, or a per-sentence table too large for one CTA's shared memory:
 *   W * max_blocks + 3 * blocks_per_sentence > 50000), VBS_ENOMEM, VBS_ECUDA.
 *   *pkv is NULL on error.
 */
int kv_paged_init(vbs_pkv** pkv, const vbs_kv_desc* desc, int batch, int W, int blocks_per_sentence, int block,
                  int max_blocks, void* pool, vbs_stream_t stream);
/*
 * The prompt: every sentence gets ceil(P / block) blocks that all W of its
 * rows point at (one copy per sentence).  The caller then writes the prompt's
 * K/V through the table of the sentence's first row and calls
 * kv_paged_prepare(P) before the first generated position is written.
 * Synchronises the stream (the tables are built on the host, once per decode).
 * Drops copies still pending.
 * Errors: VBS_EINVAL (P < 0, or the prompt needs more blocks than a sentence
 *   owns or a table row holds), VBS_ECUDA.
 */
int kv_paged_prefill(vbs_pkv* pkv, int P);
/*
 * Make the block that position t_write lands in exclusive to every live row:
 * a row whose table ends at that block boundary gets a fresh block; of the
 * rows sharing a partly filled block the lowest keeps it and every other row
 * gets a copy of its t_write % block filled slots (copy-on-write).
 * Errors: VBS_EINVAL (t_write < 0, or a block index beyond max_blocks),
 *   VBS_ESTATE (copies recorded by bs_step_paged still pending), VBS_ECUDA;
 *   an exhausted free stack is VBS_ENOMEM in kv_paged_status().
 */
int kv_paged_prepare(vbs_pkv* pkv, int t_write);
/*
 * Reorder by beam_idx[R] (device int32; -1 = pad row, left alone): table row r
 * becomes row beam_idx[r]'s, counts are raised for the new references before
 * the old ones are dropped, blocks reaching zero return to their sentence's
 * stack, then kv_paged_prepare(t_valid) runs.  Two launches, no host sync.
 * Errors: VBS_EINVAL (host checks as kv_paged_prepare, NULL beam_idx),
 * VBS_ESTATE (copies pending), VBS_ECUDA; VBS_ENOMEM / VBS_EINVAL on the device
 * are reported by kv_paged_status().
 */
int kv_paged_reorder(vbs_pkv* pkv, const int32_t* beam_idx, int t_valid);
/*
 * One beam step (bs_step, same arguments and outputs) followed by the remap
 * half of kv_paged_reorder(pkv, beam_idx, t_valid): the table, counts and free
 * stacks are updated and the copy-on-write tasks recorded, but nothing is
 * copied until kv_paged_copy(pkv).  bs_step_paged + kv_paged_copy has the
 * effect of bs_step + kv_paged_reorder ([LM] §9.2.2: the cache follows the
 * step's beam_idx).  When the beam-search context runs one cluster of CTAs per
 * sentence, the remap runs inside the beam-step kernel after each sentence's
 * merge, on the beam_idx it has just written (one launch instead of two);
 * otherwise it is a second launch.  pkv must describe the same batch and W and
 * use the same stream as ctx.  No pages' counterpart as one call: the pages
 * describe the two operations separately.
 * Until kv_paged_copy runs, the recorded copies are pending: another
 * bs_step_paged, kv_paged_reorder or kv_paged_prepare on pkv returns
 * VBS_ESTATE (kv_paged_restore and kv_paged_prefill drop pending copies).
 * Errors: those of bs_step and kv_paged_reorder; VBS_EINVAL for a pkv of
 * another batch, W or stream; VBS_ESTATE as above.  Device-side remap errors
 * go to kv_paged_status() (VBS_ESTATE there: more copy tasks than rows).
 */
int bs_step_paged(vbs_bs* ctx, const void* logits, int64_t ld, float* scores, int32_t* seqs, int32_t* beam_idx,
                  int32_t* tokens, int32_t* all_done, vbs_pkv* pkv, int t_valid);
/* The copy-on-write tasks recorded by bs_step_paged (one launch; none pending: no copy).
   Errors: VBS_EINVAL (NULL), VBS_ECUDA. */
int kv_paged_copy(vbs_pkv* pkv);
/* The device block table [R][max_blocks] and its row stride (library-owned, valid until
   kv_paged_destroy).  Errors: VBS_EINVAL (NULL arguments). */
int kv_paged_table(vbs_pkv* pkv, const int32_t** table, int* max_blocks);
/* Copy the reference counts [num_blocks] and per-row block counts [R] to device buffers
   (either may be NULL), on the stream.  Errors: VBS_EINVAL (NULL pkv), VBS_ECUDA. */
int kv_paged_counts(vbs_pkv* pkv, int32_t* refcnt, int32_t* nblk);
/* Copy the block table [R][max_blocks] to a device buffer (entries at or beyond a row's
   block count are stale), on the stream.  Errors: VBS_EINVAL (NULL), VBS_ECUDA. */
int kv_paged_copy_table(vbs_pkv* pkv, int32_t* out);
/*
 * Save / restore the allocator state (block table, block counts, reference
 * counts, free stacks) into / from the context's own copy, device to device on
 * the stream: a decode can restart from the state right after the prompt
 * without a host round trip.  Pool contents are not copied; positions the
 * restored tables do not cover are simply unused.  Restore drops copies still
 * pending.  Errors: VBS_EINVAL (NULL), VBS_ECUDA.
 */
int kv_paged_save(vbs_pkv* pkv);
int kv_paged_restore(vbs_pkv* pkv);
/* Synchronise the stream and return the number of filled slots copied by
   copy-on-write since init (one slot = one position of one (layer, k/v, head)
   run: head_dim * elem_bytes bytes read and the same written).
   Errors: VBS_EINVAL (NULL arguments), VBS_ECUDA. */
int kv_paged_cow_slots(vbs_pkv* pkv, int64_t* slots);
/* Synchronise the stream and return (then clear) the device status word: VBS_OK or
   the first VBS_E* a kernel recorded.  VBS_EINVAL for NULL, VBS_ECUDA when the
   synchronisation or the read fails. */
int kv_paged_status(vbs_pkv* pkv);
/* Free the cache's own memory (synchronises its stream first; the pool stays the
   caller's).  NULL is a no-op.  Returns VBS_OK. */
int kv_paged_destroy(vbs_pkv* pkv);

/* Synchronise `stream` and return (then clear) the status word of the calls
   that have no context (kv_reorder's and bpd_verify's bounded waits,
   bs_expand_static's input checks).  VBS_ECUDA when the synchronisation or the
   read fails. */
int vbs_stateless_status(vbs_stream_t stream);

/* =============================================================================
 * Blockwise parallel decoding ([BPD] §3-§4)
 * ============================================================================= */

/* The verify test of bpd_verify_approx ([BPD] §3 exact, §5.1 top-k, §5.2 distance). */
#define VBS_BPD_EXACT 0
#define VBS_BPD_TOPK 1
#define VBS_BPD_DISTANCE 2

/*
 * Predict: proposals[b, h] = argmax_v logits[b, h, v] for logits [B, k, V]
 * (device, dense rows); argmax ties go to the lower token id.  proposals[B, k]
 * int32 (device).  B = 0 launches nothing.
 * Errors: VBS_EINVAL (B < 0, k outside 1..32, V < 1, unknown dtype, NULL
 *   pointers with B > 0), VBS_ECUDA.
 */
int bpd_propose(const void* logits, int B, int k, int V, int dtype, int32_t* proposals, vbs_stream_t stream);

/*
 * Verify + accept on the combined model's logits [B, k, k, V] (device, dense):
 * logits[b, p, h, :] is head h+1 at proposal position p+1, i.e. given the
 * prefix extended by proposals[b, 0..p].  khat[b] = 1 + the number of leading
 * p = 0..k-2 with proposals[b, p+1] == argmax logits[b, p, 0, :]; if eos >= 0
 * and an accepted proposal e < khat equals eos, khat = e + 1.
 * next[b, h] = argmax logits[b, khat-1, h, :] (the next iteration's
 * proposals).  Only the rows this needs are read.  1 <= k <= 32.
 * For B <= 16384 the call runs as a persistent work queue whose counters and
 * ready list (4 MiB) are static device memory shared by every call (reset by
 * each call's last CTA): two bpd_verify calls that overlap on the GPU
 * (different streams or host threads) race and must be serialised by the
 * caller.  Calls on one stream are ordered: the kernel is launched as a
 * programmatic dependent, so its set-up may overlap the previous kernel, but it
 * touches memory only once that kernel has completed.  A wait that gives up is
 * reported by vbs_stateless_status().
 * Errors: VBS_EINVAL (B < 0, k outside 1..32, V < 1, eos >= V, unknown dtype,
 *   NULL pointers with B > 0), VBS_ECUDA.
 */
int bpd_verify(const void* logits, const int32_t* proposals, int B, int k, int V, int dtype, int eos,
               int32_t* khat, int32_t* next, vbs_stream_t stream);
/*
 * bpd_verify with the relaxed verify tests of [BPD] §5 (approximate inference:
 * the output may differ from greedy decoding).  The pages' formulas for the
 * criteria are missing from their text; these are the readings:
 *   criterion VBS_BPD_EXACT: proposal == argmax (bpd_verify; param ignored);
 *   VBS_BPD_TOPK (§5.1): the proposal's rank in head 0's row -- the number of
 *     tokens with a larger logit, or an equal logit and a lower id -- is below
 *     param (param >= 1; 1 is exact);
 *   VBS_BPD_DISTANCE (§5.2): |proposal - argmax| <= param, token ids read as
 *     intensities with d(u, v) = |u - v| (param >= 0; 0 is exact).
 * min_accept (§5.3, 1..k): khat = max(khat, min_accept) before the EOS cut;
 * min_accept = k decodes in fixed blocks of k.  The next proposals come from
 * position khat-1 as in bpd_verify.  Same layout, ownership and queue notes.
 * Errors: VBS_EINVAL for an unknown criterion or a parameter out of range.
 */
int bpd_verify_approx(const void* logits, const int32_t* proposals, int B, int k, int V, int dtype, int eos,
                      int criterion, int param, int min_accept, int32_t* khat, int32_t* next, vbs_stream_t stream);

/* =============================================================================
 * In-run memory peaks.  The pages have no counterpart: these measure, on the
 * running GPU, the bandwidth a roofline of the calls above is read against.
 * ============================================================================= */

/*
 * Copy `bytes` from src to dst (device, non-overlapping) with 16-byte vector
 * loads and stores, `grid` CTAs each taking one contiguous, equal share.  The
 * bandwidth is 2 * bytes / time (read + write).
 * Errors: VBS_EINVAL (NULL, bytes <= 0, grid outside 1..65535), VBS_EALIGN
 *   (a pointer not 16-byte aligned, bytes not a multiple of 16), VBS_ECUDA.
 */
int vbs_peak_copy(const void* src, void* dst, int64_t bytes, int grid, vbs_stream_t stream);
/*
 * Read `bytes` from src (device) and fold a maximum over them, `grid` CTAs each
 * taking one contiguous, equal share: mode 0 with 16-byte vector loads, mode 1
 * through a ring of bulk copies into shared memory (one producer lane, 16
 * consumer warps; the beam step's streaming pattern without its arithmetic).
 * sink[grid] (device uint32) receives one word per CTA, so no load is dead
 * code; its value carries no meaning.  A bounded wait that gives up is reported
 * by vbs_stateless_status().
 * Errors: VBS_EINVAL (NULL, bytes <= 0, grid outside 1..65535, unknown mode),
 *   VBS_EALIGN (src not 16-byte aligned, bytes not a multiple of 16), VBS_ECUDA.
 */
int vbs_peak_read(const void* src, int64_t bytes, int grid, int mode, uint32_t* sink, vbs_stream_t stream);

/*
 * The device bounds checks of the checked build.  The library can be built a second
 * time with VBS_CHECKED defined (libvbs_checked.so): then the indexed accesses whose index
 * comes from data (the streamed row ranges, partial slots, merge outputs and sequence
 * gathers, the KV parents and pool blocks, the verify queue's slots) are guarded; a
 * failed guard skips the access, sets VBS_EBOUNDS in the call's status word and records
 * the first failure.  Synchronises the device, then sets *checked (1 in the checked build,
 * 0 otherwise), and *site / *index of the first failed check since the last call (-1 / -1
 * when none; the record is then cleared).  The pages have no counterpart: this is a test
 * aid, the checks stand in for a memory checker.
 * Errors: VBS_EINVAL (NULL), VBS_ECUDA.
 */
int vbs_checked_record(int* checked, int* site, int64_t* index);

#ifdef __cplusplus
}
#endif

#endif /* VBS_H */
