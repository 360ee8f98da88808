/*
 * specng.h -- C ABI of the GB300 (sm_103a) library for the data-parallel hot
 * path of speculative decoding with n-gram drafts and Leviathan/Chen
 * verification.
 *
 * Sources (page title, section):
 *  [AX]  "AX Engine: An LLM Inference Engine Built Exclusively for Apple
 *        Silicon M4+", section "Core Technical Architecture & Methods":
 *        bigram/trigram tables built at runtime; up to 4 draft tokens per
 *        step; validation by the target forward; EMA acceptance gate
 *        (tau = 0.1, threshold = 0.5) that disables speculation; O(1)
 *        rollback by moving the sequence-length pointer.  Section "Supported
 *        Model Families" (table): Gemma's logit soft cap.
 *  [SW]  "SwiftLM: Apple Silicon native MLX Swift LLM inference server",
 *        paragraph on algorithmic equivalence (Leviathan et al.): accept a
 *        draft with probability P_target / P_draft and resample from the
 *        corrected distribution on rejection; M1 Ultra benchmark paragraph:
 *        --repeat-penalty 1.1, temperature 0.6; DFlash warning paragraph:
 *        greedy (argmax) verification is the temperature-0 case.
 *
 * Conventions shared by every call
 *  - Every array argument is caller-owned DEVICE memory unless stated
 *    otherwise; the library never frees it.  int32 arrays are row-major.
 *  - Every call is asynchronous and ordered on the given stream; none of
 *    them synchronises except specng_get_status() and specng_get_counters().
 *  - The stream must belong to the current device (make the device of the
 *    arrays current before the call); the verify calls check this and
 *    return EINVAL otherwise.
 *  - Return value: SPECNG_OK (0), or a negative code for an error found on
 *    the host before anything was enqueued (nothing ran in that case).
 *  - Errors found on the device (full table, out-of-range token, non-finite
 *    logits, history overflow, out-of-range k) never trap and never hang:
 *    the kernel skips the offending item and sets a bit in a per-device
 *    status word read with specng_get_status().
 *  - No kernel waits for another block: cross-block merges use a
 *    fence + atomic ticket, and the last block to arrive does the merge.
 *    Every hash probe loop is bounded by the table capacity.
 *  - The kernels of spec_verify, spec_append and spec_commit are launched
 *    with programmatic stream serialisation: each may start before the
 *    previous kernel on the stream has finished and waits (griddepcontrol)
 *    before it reads anything that kernel may have written, so stream
 *    order is kept for every caller.
 */
#ifndef SPECNG_H
#define SPECNG_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPECNG_API_VERSION 3

/* Host-detected return codes. */
#define SPECNG_OK      0
#define SPECNG_EINVAL (-1)  /* null pointer, size or parameter out of range   */
#define SPECNG_EALIGN (-2)  /* pointer alignment below what the call requires */
#define SPECNG_ECUDA  (-3)  /* a CUDA runtime call failed (message: strerror) */
#define SPECNG_ENOMEM (-4)  /* device allocation failed (table creation only) */
#define SPECNG_ESMALL (-5)  /* workspace smaller than spec_verify_workspace_bytes */

/* Logit element types accepted by spec_verify. */
#define SPECNG_F32  0
#define SPECNG_BF16 1

/* Device status bits (specng_get_status). */
#define SPECNG_DEV_TABLE_FULL     0x01u /* a hash probe met no free slot; insert skipped   */
#define SPECNG_DEV_TOKEN_OOR      0x02u /* a token outside [0, V) was met and skipped      */
#define SPECNG_DEV_NONFINITE      0x04u /* a logit row read at T > 0 had NaN or +Inf       */
#define SPECNG_DEV_HIST_OVERFLOW  0x08u /* spec_append would pass the history capacity     */
#define SPECNG_DEV_BAD_K          0x10u /* k[b] or accept_len[b] outside [0, K]; clamped   */
#define SPECNG_DEV_COUNT_SAT      0x20u /* an n-gram count passed 2^22 - 1 and saturated   */
#define SPECNG_DEV_HIST_SHRANK    0x40u /* lens[b] fell below what the table had indexed   */
#define SPECNG_DEV_TIMEOUT        0x80u /* a bounded wait for a bulk copy gave up; the call's
                                           outputs are incomplete and its workspace must be
                                           zeroed again (spec_verify_workspace_init)         */
#define SPECNG_DEV_KV_SHORT      0x200u /* specng_kv_reserve could not give a sequence all the
                                           blocks it needs: the pool ran empty or its table
                                           row is full (it keeps what it got)             */
#define SPECNG_DEV_CHECKED_OOB   0x100u /* checked build only (compiled with SPECNG_CHECKED):
                                           a computed index (vocabulary id, history position,
                                           draft slot, logit element) fell outside its array;
                                           it was clamped into range, nothing trapped        */

/* Limits checked on the host. */
#define SPECNG_MAX_K          16        /* drafts per sequence per call            */
#define SPECNG_MAX_REP_WINDOW 256       /* repetition-penalty window (tokens)      */
#define SPECNG_NGRAM_MAX_B    512       /* sequences per n-gram table              */
#define SPECNG_NGRAM_MAX_V    262144    /* vocabulary of an n-gram table (2^18)    */
#define SPECNG_NGRAM_MAX_POS  16777216  /* positions per sequence in a table (2^24) */
#define SPECNG_STATIC_SCRATCH_BYTES 16777216 /* scratch of spec_verify_noalloc (16 MiB) */

/* Diagnostic counters (specng_get_counters): how often a rarely taken exact
 * path ran.  Every decision that floating point takes is screened in fp32
 * with a margin and re-taken in fp64 inside the margin; these count the
 * re-takes, so a test can tell that a planted near-tie reached the fp64
 * code.  They are bumped only inside those cold paths. */
#define SPECNG_DIAG_ACCEPT_F64    0 /* accept test u q <= p re-taken in fp64              */
#define SPECNG_DIAG_SAMPLE_F64    1 /* top two Gumbel scores (point mass / bonus) in fp64 */
#define SPECNG_DIAG_RESIDUAL_F64  2 /* dense-residual decision taken in fp64              */
#define SPECNG_DIAG_GREEDY_F64    3 /* greedy argmax near-tie re-decided in fp64          */
#define SPECNG_DIAG_RESIDUAL_ZERO 4 /* all-zero residual: token sampled from p            */
#define SPECNG_DIAG_N             8

/* ------------------------------------------------------------------------
 * N-gram table  [AX]: "builds bigram/trigram tables at runtime, predicts up
 * to 4 draft tokens per step".
 *
 * One opaque object holds four open-addressed hash tables in device memory
 * (trigram pairs, bigram pairs, trigram contexts, bigram contexts) for B
 * sequences with token ids in [0, V).  A pair entry counts how often token
 * c followed a context and the latest position where it did; a context
 * entry holds its best continuation: the largest count, equal counts going
 * to the most recent occurrence.  Insertion is order-independent, so the
 * table is a pure function of the indexed histories (it can be rebuilt
 * from them after a restart).
 * --------------------------------------------------------------------- */
typedef struct specng_ngram specng_ngram;

/* Allocate and clear a table.  max_positions: upper bound on the number of
 * history positions that will ever be indexed, summed over all B sequences
 * (each table gets 2 * max_positions slots rounded up to a power of two, 16
 * bytes each).  B in [1, 512]; V in [1, 2^18].  The object owns its device
 * memory (allocated with cudaMalloc on the current device) until
 * specng_ngram_destroy.  Clearing is enqueued on stream s.
 * Errors: EINVAL, ENOMEM, ECUDA. */
int specng_ngram_create(specng_ngram** table, int B, int V, int64_t max_positions,
                        cudaStream_t s);

/* Free the table (synchronises the device first).  NULL is accepted. */
int specng_ngram_destroy(specng_ngram* table);

/* Draft only on repeated evidence ([AX] note under the decode table:
 * speculation "repeats n-gram evidence"): a context proposes its best
 * continuation only when that continuation was seen at least min_count
 * times (1, the default: any evidence).  A host-side setting of the table,
 * read by ngram_draft and spec_commit.  min_count in [1, 2^22 - 1]. */
int specng_ngram_set_min_count(specng_ngram* table, int min_count);

/* Remove every entry and mark every sequence as not indexed (stream s). */
int specng_ngram_reset(specng_ngram* table, cudaStream_t s);

/* Slots per hash table (a power of two). */
int specng_ngram_capacity(const specng_ngram* table, int64_t* slots);

/* Index the history positions added since the previous call.
 * history: int32 [B, hist_stride] (token i of sequence b at b*hist_stride+i);
 * lens: int32 [B], the number of valid tokens per sequence.  For every new
 * position i in [indexed_b, lens_b) (indexed_b = lens_b of the previous
 * call, 0 after create/reset) the bigram pair (h[i-1] -> h[i]) and, when
 * i >= 2, the trigram pair ((h[i-2], h[i-1]) -> h[i]) are counted, then the
 * contexts' best continuations are refreshed.  Three kernel launches (the
 * table keeps no state on the host, so a captured call replays right).
 * Device errors: TABLE_FULL, TOKEN_OOR, COUNT_SAT, HIST_SHRANK. */
int ngram_update(const int32_t* history, int64_t hist_stride, const int32_t* lens,
                 specng_ngram* table, cudaStream_t s);

/* Draft up to max_k tokens per sequence by chained lookups: the context is
 * the last two tokens of history ++ drafts so far; the trigram context is
 * tried first, then the bigram context; drafting stops at the first miss.
 * k_limit: optional int32 [B] per-sequence cap (NULL: max_k for all).
 * fallback: optional int32 [B, max_k] proposals of another drafter; when
 * given, the positions after the first miss (up to the cap) take
 * fallback[b, t] and are counted in out_k (NULL: drafting just stops).
 * out_drafts: int32 [B, max_k], padded with -1; out_k: int32 [B], the count.
 * The table is read only.  max_k in [0, 16].  One kernel launch. */
int ngram_draft(const specng_ngram* table, const int32_t* history, int64_t hist_stride,
                const int32_t* lens, int max_k, const int32_t* k_limit, const int32_t* fallback,
                int32_t* out_drafts, int32_t* out_k, cudaStream_t s);

/* ------------------------------------------------------------------------
 * Verification  [SW] Leviathan/Chen + [AX] EMA gate and rollback.
 * --------------------------------------------------------------------- */
typedef struct {
    float    temperature;   /* T; 0 selects greedy verification (argmax)          */
    float    softcap;       /* c: x -> c * tanh(x / c); <= 0 disables             */
    float    rep_penalty;   /* r > 0: x > 0 -> x / r, else x * r; 1 disables       */
    int32_t  rep_window;    /* W in [0, 256]: last W tokens of history ++ drafts   */
    float    ema_tau;       /* EMA rate (0.1 on the page)                          */
    float    ema_thresh;    /* gate threshold (0.5 on the page)                    */
    int32_t  gate_enabled;  /* 0: always verify k[b] drafts                        */
    uint32_t pad_;          /* must be 0                                           */
    uint64_t seed;          /* Philox key                                          */
    uint64_t step;          /* decode step (low 32 bits enter the Philox counter)  */
    int32_t  early_exit;    /* 1: rows past a sequence's known first rejection are
                               not read (single-kernel schedule only); the outputs
                               are the same, since those rows cannot change them   */
    int32_t  schedule;      /* SPECNG_SCHEDULE_*                                   */
    /* Gate variants ([AX] "Performance Evidence & Results", note under the
     * decode table: speculation "cools after partial acceptance"; the way a
     * disabled gate opens again is left open by the page).  Both 0: the
     * gate above alone, which stays shut once shut.                        */
    int32_t  probe_interval;/* P > 0: a gated-off sequence verifies its drafts on
                               the calls whose step is a multiple of P; that call
                               updates the EMA and may open the gate again       */
    int32_t  cool_steps;    /* C > 0: after a call with 0 < a < k_eff the sequence
                               verifies no drafts for its next C calls            */
    int32_t* gate_state;    /* device int32 [B], in/out: each sequence's remaining
                               cooling calls (zero-fill before the first call);
                               required when cool_steps > 0, else ignored         */
    const uint64_t* step_dev; /* device uint64 or NULL: when given, the kernels read
                               the decode step from it instead of `step` (a call
                               captured in a CUDA graph keeps its host arguments;
                               specng_step_advance moves this counter on).  Not
                               with the single-kernel schedule, whose state words
                               carry a per-call tag chosen on the host (EINVAL)   */
} specng_verify_params;

/* Kernel schedules of spec_verify (the outputs are the same under each). */
#define SPECNG_SCHEDULE_AUTO  0  /* the two-kernel schedule (SPLIT)                     */
#define SPECNG_SCHEDULE_FUSED 1  /* one persistent kernel (B <= 2048): every CTA streams
                                    whole rows, row index first, and decides each row
                                    it streamed as soon as it is streamed; the sequence
                                    whose accept length that settles is sampled at once;
                                    allows early exit                                  */
#define SPECNG_SCHEDULE_SPLIT 2  /* a streaming kernel over all active rows, then one
                                    CTA per sequence (accept tests, sample, epilogue),
                                    + a residual pass for dense drafts at T > 0        */
#define SPECNG_FUSED_MAX_B    2048

/* Bytes of device workspace spec_verify needs for (B, K, V). */
size_t spec_verify_workspace_bytes(int B, int K, int V);

/* Zero a workspace (stream-ordered).  A workspace must be zero-filled once
 * before its first spec_verify call; each call leaves it ready for the next
 * (see spec_verify's workspace argument). */
int spec_verify_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t s);

/* One verify call for B sequences with up to K drafts each.
 *
 * logits       [B, K+1, V] of logits_dtype (SPECNG_BF16 or SPECNG_F32);
 *              row j of sequence b is the target's next-token logits after
 *              history ++ d_1..d_j.  Rows j > k_eff(b) are never read.
 * drafts       int32 [B, K]: d_1..d_K (may be NULL when K = 0).
 * draft_probs  fp32 [B, K, V] draft distributions q_j, or NULL for
 *              point-mass drafts (q = one-hot(d), the n-gram case).
 * k            int32 [B]: drafts to verify per sequence, in [0, K].
 * history, hist_stride, lens: int32, as for ngram_update; read only for the
 *              repetition-penalty window (may be NULL when the penalty is off).
 * params       host pointer; see specng_verify_params.
 * kv_len       int32 [B], in/out: on entry the KV length after the verify
 *              forward (committed + k[b] + 1); on exit kv_len - k[b] + a.
 * ema          fp32 [B], in/out: acceptance EMA.  Gate (when enabled):
 *              k_eff = ema >= thresh ? k : 0, read before the update (a
 *              probe step, see probe_interval, counts as open; a cooling
 *              sequence, see cool_steps, has k_eff = 0); if k_eff > 0,
 *              ema <- (1 - tau) * ema + tau * a / k_eff.
 * out_tokens   int32 [B, K+1]: d_1..d_a, then the residual or bonus sample,
 *              then -1.
 * out_accept_len int32 [B]: a.
 * workspace    device scratch of at least spec_verify_workspace_bytes(B, K, V)
 *              bytes, 256-byte aligned, zero-filled before its first use
 *              (spec_verify_workspace_init or any zero fill).  Every call
 *              zeroes again the records it reads back (the rest is written
 *              before it is read), so later calls of any shape that fits may
 *              reuse it without another fill; one workspace per call in
 *              flight.
 *
 * Per row: x <- c tanh(x/c) (soft cap), repetition penalty over the window
 * (each distinct id once), temperature; online max and sum of exponentials.
 * Accept test for draft i: u_i * q(d_i) <= p(d_i), u_i from Philox4x32-10
 * keyed by (seed; draft index, step, sequence).  Sample at row a (residual
 * max(0, p_a - q_a) on a rejection, p_a when all k_eff drafts are accepted)
 * by Gumbel-max with Philox noise keyed by (seed; vocab id, row, step,
 * sequence).  T = 0: accept iff d_i is its row's argmax (lowest id on
 * ties); the emitted token is the argmax of row a.
 * Sampling noise: per block of 256 ids a block draw (the block minimum of
 * the block's Exp(1) variates and its slot), then one draw per id (that
 * minimum plus an Exp(1)), which leaves the variates i.i.d. Exp(1) and lets
 * whole blocks be ruled out by the bound z_max / T - ln(minimum).
 * Launches: two kernels (the streaming pass over the rows: block maxima and
 * the sums of exponentials; then one CTA per sequence: accept tests,
 * sample, epilogue); three with dense q at T > 0 (a residual pass over row a
 * of the rejected sequences).
 * Requirements: logits 16-byte aligned for the vectorised path (any
 * alignment works, slower); B in [1, 2^20]; K in [0, 16]; V in [1, 2^30].
 * Errors: EINVAL, ESMALL, ECUDA.  Device: NONFINITE, TOKEN_OOR, BAD_K. */
int spec_verify(const void* logits, int logits_dtype, int B, int K, int V,
                const int32_t* drafts, const float* draft_probs, const int32_t* k,
                const int32_t* history, int64_t hist_stride, const int32_t* lens,
                const specng_verify_params* params,
                int32_t* kv_len, float* ema,
                int32_t* out_tokens, int32_t* out_accept_len,
                void* workspace, size_t workspace_bytes, cudaStream_t s);

/* One step's commit in one kernel launch: exactly spec_append, then
 * ngram_update, then ngram_draft for the next step, with the same arguments
 * and results as those three calls made in that order (B must be the
 * table's B).  One warp per sequence: a sequence's history, lengths and
 * table keys belong to it alone, so no other sequence's work is waited for.
 * The fusion is an implementation choice, not a step of the pages; it
 * removes three of the four launches of the per-step bookkeeping, which are
 * bound by launch and memory latency rather than by bandwidth.
 * Errors: EINVAL, ECUDA.  Device: HIST_OVERFLOW, BAD_K, TABLE_FULL,
 * TOKEN_OOR, COUNT_SAT, HIST_SHRANK. */
int spec_commit(specng_ngram* table, int32_t* history, int64_t hist_stride, int32_t* lens,
                int64_t hist_cap, const int32_t* out_tokens, const int32_t* out_accept_len,
                int B, int K, int max_k, const int32_t* k_limit, const int32_t* fallback,
                int32_t* out_drafts, int32_t* out_k, cudaStream_t s);

/* spec_verify without a caller workspace.  The pages have no counterpart of
 * this call: it is an interface addition, for callers that cannot allocate
 * device memory where they verify -- a runtime whose allocator reserved the
 * device's memory up front and refuses requests while decoding, or a decode
 * loop that must not stall on cudaMalloc / cudaFree (both synchronise the
 * device) and has no buffer of its own to lend.
 *
 * Arguments, results, launches and errors as for spec_verify, minus the
 * workspace.  The scratch is a static device array of
 * SPECNG_STATIC_SCRATCH_BYTES inside the library, one per device; the call
 * allocates nothing (no cudaMalloc / cudaFree, no allocating library
 * routine).
 *   - Limit: spec_verify_workspace_bytes(B, K, V) must not exceed
 *     SPECNG_STATIC_SCRATCH_BYTES (e.g. B = 512, K = 4, V = 262144 fits);
 *     a larger shape returns SPECNG_ESMALL, with the sizes in
 *     specng_last_error().  spec_verify with a caller workspace has no
 *     such limit.
 *   - Every argument check, this one included, runs before anything is
 *     enqueued: a call that returns an error has enqueued nothing and has
 *     not touched the scratch.
 *   - Each call first zero-fills the part of the scratch it uses
 *     (cudaMemsetAsync on s), then enqueues the verify kernels on s.
 *   - The first call on a device looks the scratch address up
 *     (cudaGetSymbolAddress) and caches it; make that first call before any
 *     stream capture starts on that device.
 *   - All calls on one device share the scratch: calls whose executions
 *     overlap (unordered streams, or several host threads) race and give
 *     wrong results.  Order them, e.g. on one stream. */
int spec_verify_noalloc(const void* logits, int logits_dtype, int B, int K, int V,
                        const int32_t* drafts, const float* draft_probs, const int32_t* k,
                        const int32_t* history, int64_t hist_stride, const int32_t* lens,
                        const specng_verify_params* params,
                        int32_t* kv_len, float* ema,
                        int32_t* out_tokens, int32_t* out_accept_len, cudaStream_t s);

/* Fused LM head + verify.  The target model's last
 * projection and the verify of the drafts in one call: the logits of the
 * K + 1 positions are logits = hidden W^T (SwiftLM page, Leviathan
 * paragraph: the target scores the K drafts and the bonus position in one
 * forward), computed on the tensor cores, and the same kernel's epilogue
 * writes, per row and 256-id noise block, the block's largest logit and its
 * softmax record; the decision kernel of spec_verify then runs on those
 * records (no streaming pass over the logits), reading single logits back
 * only where a decision needs them.  Results, as for spec_verify with
 * logits_dtype SPECNG_BF16 and these logits.
 *
 * hidden       device, bf16 [B, K+1, d] row-major: the final hidden states
 *              of the K + 1 positions (d a multiple of 64, 16-byte aligned).
 * weight       device, bf16 [V, d] row-major: the LM head (16-byte aligned).
 * d            hidden size, a multiple of 64 in [64, 2^20].
 * logits       device, bf16 [B, K+1, V]: written by the call, each value the
 *              fp32 dot product rounded to bf16 (nearest, ties to even);
 *              V must be a multiple of 8 (16-byte rows).
 * workspace    device scratch of at least spec_verify_lmhead_workspace_bytes
 *              (B, K, V) bytes, 256-byte aligned, zero-filled before the
 *              first call; the call leaves it ready for the next
 *              spec_verify_lmhead call (every record is rewritten each
 *              call).  Its layout differs from spec_verify's: zero it again
 *              (spec_verify_workspace_init) before a spec_verify call uses
 *              the same buffer.
 * Other arguments as for spec_verify.  Not supported (SPECNG_EINVAL): the
 * repetition penalty (rep_penalty != 1 with rep_window > 0) and the
 * single-kernel schedule.  SPECNG_EINVAL also when the tensor maps of
 * hidden / weight cannot be encoded (the driver lacks
 * cuTensorMapEncodeTiled). */
size_t spec_verify_lmhead_workspace_bytes(int B, int K, int V);
int spec_verify_lmhead(const void* hidden, const void* weight, int d, void* logits,
                       int B, int K, int V, const int32_t* drafts, const float* draft_probs,
                       const int32_t* k, const int32_t* history, int64_t hist_stride,
                       const int32_t* lens, const specng_verify_params* params,
                       int32_t* kv_len, float* ema, int32_t* out_tokens, int32_t* out_accept_len,
                       void* workspace, size_t workspace_bytes, cudaStream_t s);

/* Measurement hook; the pages have no counterpart of it.  While
 * after_stream_kernel is not NULL, every spec_verify call records it on its
 * stream right after the streaming kernel, so a caller can time that kernel
 * alone (an event recorded before the call starts the span).  While it is
 * set, the decision kernel waits for the streaming kernel to finish instead
 * of starting during its tail.  One process-wide setting, not thread-safe;
 * NULL turns it off.  Always returns SPECNG_OK. */
int specng_set_verify_marker(cudaEvent_t after_stream_kernel);

/* Append the emitted tokens: history[b, lens_b + t] = out_tokens[b, t] for
 * t <= out_accept_len[b], then lens_b += out_accept_len[b] + 1.  A sequence
 * whose history would pass hist_cap tokens is left unchanged (HIST_OVERFLOW).
 * In place, one kernel launch. */
int spec_append(int32_t* history, int64_t hist_stride, int32_t* lens, int64_t hist_cap,
                const int32_t* out_tokens, const int32_t* out_accept_len, int B, int K,
                cudaStream_t s);

/* ------------------------------------------------------------------------
 * Decode-step bookkeeping  [AX] "Core Technical Architecture & Methods":
 * the KV cache grows inside preallocated buffers, and a speculation rollback
 * is O(1) -- only the sequence length moves (spec_verify's kv_len update);
 * the scheduler recovers memory blocks.  Graph compilation reuses the same
 * work across same-shape steps: a step (spec_verify, spec_commit, the KV
 * calls below, specng_step_advance) can be captured once in a CUDA graph and
 * replayed, with the decode step read from a device counter (step_dev).
 * --------------------------------------------------------------------- */

/* A pool of num_blocks KV blocks of block_size positions each, in the
 * caller's preallocated KV buffers; the library keeps the bookkeeping only.
 * All arrays are device int32 owned by the caller:
 *   free_stack [num_blocks]: the free block ids are free_stack[0 .. *free_top)
 *   free_top   [1]
 *   block_table[B, max_blocks]: row b lists sequence b's blocks in position
 *              order (position p of sequence b is in block row_b[p / block_size]),
 *              -1 past its count
 *   nblocks    [B]: blocks held by each sequence
 * Sizes: num_blocks in [1, 2^30], B in [1, 2^20], max_blocks >= 1 with
 * B * max_blocks <= 2^31 - 1, block_size >= 1. */
typedef struct {
    int32_t* free_stack;
    int32_t* free_top;
    int32_t* block_table;
    int32_t* nblocks;
    int32_t  num_blocks;
    int32_t  B;
    int32_t  max_blocks;
    int32_t  block_size;
} specng_kv_pool;

/* Every block free, every sequence without blocks (blocks are then handed out
 * in increasing id order by a single sequence).  One kernel launch. */
int specng_kv_init(const specng_kv_pool* pool, cudaStream_t s);

/* Sequence b takes blocks from the pool until it holds
 * ceil((kv_len[b] + extra) / block_size) of them (capped at max_blocks), e.g.
 * extra = K + 1 before a verify forward that writes K + 1 positions.  Which
 * free block a sequence gets depends on the order of the device's atomics.
 * kv_len: device int32 [B]; extra >= 0.  Device: KV_SHORT.  One launch. */
int specng_kv_reserve(const specng_kv_pool* pool, const int32_t* kv_len, int extra, cudaStream_t s);

/* Blocks past the ceil(kv_len[b] / block_size) that sequence b's positions
 * need go back to the pool (after a rollback, the blocks that held only
 * rejected positions).  kv_len: device int32 [B].  One launch. */
int specng_kv_trim(const specng_kv_pool* pool, const int32_t* kv_len, cudaStream_t s);

/* All blocks of the sequences with done[b] != 0 go back to the pool (a
 * finished request).  done: device int32 [B].  One launch. */
int specng_kv_release(const specng_kv_pool* pool, const int32_t* done, cudaStream_t s);

/* *step_dev += 1 on the stream (device uint64): the next call that reads
 * params.step_dev sees the next decode step.  One launch. */
int specng_step_advance(uint64_t* step_dev, cudaStream_t s);

/* ------------------------------------------------------------------------
 * Status and diagnostics
 * --------------------------------------------------------------------- */

/* Copy the current device's status bits to *bits (host pointer);
 * if clear != 0, reset them to 0.  Synchronises the device. */
int specng_get_status(uint32_t* bits, int clear);

/* Copy the current device's first n diagnostic counters (SPECNG_DIAG_*) to
 * counts (host array of n); if clear != 0, reset all of them to 0.  n in
 * [0, SPECNG_DIAG_N].  Synchronises the device.  The pages have no
 * counterpart of this call: it exists so that tests can show which exact
 * path a decision took. */
int specng_get_counters(uint32_t* counts, int n, int clear);

/* Static description of a return code. */
const char* specng_strerror(int code);

/* Description of the last host-detected error of the calling thread (names
 * the call and, for ECUDA, the CUDA error).  Valid until the next error. */
const char* specng_last_error(void);

/* Philox4x32-10 (Salmon et al., SC'11) on n counters: out[4i..4i+3] =
 * philox(ctr[4i..4i+3]; key = (seed mod 2^32, seed >> 32)).  The same
 * device routine keys the accept and Gumbel noise of spec_verify; exported
 * so that it can be compared bit for bit with an independent
 * implementation.  ctr, out: uint32 device arrays of 4n words. */
int specng_philox4x32_10(const uint32_t* ctr, uint64_t seed, uint32_t* out, int64_t n,
                         cudaStream_t s);

#ifdef __cplusplus
}
#endif
#endif /* SPECNG_H */
