/*
 * gdn.h -- C ABI of libgdn, the Gated DeltaNet linear-attention hot path for
 * one NVIDIA GB300 (sm_103a).
 *
 * The operation.  For each (sequence or decode row, value head h) the library
 * runs the gated delta rule of Gated DeltaNet (Yang, Kautz, Hatamizadeh,
 * "Gated Delta Networks: Improving Mamba2 with Delta Rule", ICLR 2025) on a
 * per-head fp32 state S in R^{d_k x d_v}:
 *
 *     alpha_t = exp(g_t)
 *     S_t     = alpha_t S_{t-1} - beta_t k_t (k_t^T (alpha_t S_{t-1})) + beta_t k_t v_t^T
 *     o_t     = scale * S_t^T q_t
 *
 * Value head h reads the q/k of key head h / (h_v / h_k) (grouped value
 * attention with contiguous groups).
 *
 * Routes, after the vLLM page "Enable batch-invariant mixed decode and
 * prefill for Qwen GDN" (sections "Why" and "How"): cached decode rows always
 * run on the packed recurrent decode kernel, also when fresh prefills share
 * the step, so a row's arithmetic never depends on what else is batched with
 * it; fresh prefill rows run through the chunked prefill on a fixed 64-token
 * chunk grid anchored at each sequence's first token of the call.  The
 * prefill can emit the carried state at chunk boundaries (the vLLM page
 * "GatedDeltaNet Automatic Prefix Caching", section "Purpose") so that prefix
 * caches can be filled and later resumed on the lcm(64, block) grid (the vLLM
 * page "Enable GDN batch-invariant prefix caching", section "Purpose").
 *
 * Conventions shared by every entry point.
 *   - All tensors are dense, row-major, in device memory unless the argument
 *     name ends in _host.  bf16 tensors are passed as gdn_bf16 (raw bits).
 *   - Token-major activations: q, k [T][h_k][d_k]; v, o [T][h_v][d_v];
 *     g, beta [T][h_v] fp32.  Decode rows are tokens.
 *   - State cache: float state[num_slots][h_v][d_v][d_k], i.e. each slot holds
 *     S^T per value head with d_k contiguous.  Slots are chosen per row or
 *     sequence by int32 index arrays in device memory.
 *   - Ownership: the caller owns every buffer.  The library allocates no
 *     device or host memory, keeps no state between calls, never
 *     synchronises the host, and enqueues all work on `stream` (a
 *     cudaStream_t; NULL = legacy default stream).
 *   - Errors: arguments are validated on the host before anything is
 *     launched; a bad argument returns GDN_ERR_INVALID_ARG or
 *     GDN_ERR_UNSUPPORTED and launches nothing.  A failed launch returns
 *     GDN_ERR_CUDA.  Problems only the device can see (a slot index out of
 *     range) skip the affected row or sequence, zero its outputs and OR a
 *     GDN_DEV_* bit into *dev_status when dev_status is not NULL; kernels
 *     never trap.
 *   - Only d_k == d_v in {64, 128} is supported; h_v % h_k == 0.
 *   - Slots: within one call, the set of slots a call writes (destination
 *     slots, snapshot slots, cache-block slots) must be disjoint from the
 *     slots that OTHER rows or sequences of the same call read, and no slot
 *     may be written twice; a row or sequence may write the slot it reads
 *     (in place).  Rows run concurrently, so an aliased slot would make the
 *     result depend on scheduling.  A state shift along slots (row r writes
 *     the slot row r+1 reads) must be split into calls that each satisfy
 *     this rule.  When the decode and prefill halves of a step are launched
 *     on two streams at once, their slot sets must be disjoint too.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gdn_bf16; /* bfloat16 bit pattern */

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null pointer, bad size, non-monotone cu_seqlens, ... */
    GDN_ERR_UNSUPPORTED = 2, /* head dims or shapes this build does not implement */
    GDN_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    GDN_ERR_WORKSPACE = 4,   /* workspace smaller than gdn_prefill_workspace_bytes() or misaligned */
    GDN_ERR_TIMEOUT = 5      /* from gdn_status_from_device(): a bounded wait expired in a kernel */
} gdn_status_t;

/* Bits ORed into *dev_status by kernels.  Kernels run asynchronously, so
 * these reach the host only when the caller reads the word back;
 * gdn_status_from_device() maps it to a gdn_status_t. */
#define GDN_DEV_BAD_SLOT 0x1 /* a slot index was >= num_slots; the row/sequence was skipped */
#define GDN_DEV_TIMEOUT 0x2  /* a bounded wait expired inside a kernel; its outputs are invalid */

typedef struct {
    int32_t h_k;  /* query/key heads */
    int32_t h_v;  /* value heads (multiple of h_k) */
    int32_t d_k;  /* key head dim */
    int32_t d_v;  /* value head dim */
    float scale;  /* multiplies o; the literal recurrence uses 1.0 */
} gdn_dims_t;

/*
 * Packed recurrent decode: one token per cached row.
 * vLLM page "Enable batch-invariant mixed decode and prefill for Qwen GDN",
 * section "How" (the shared packed recurrent decode helper for cached rows);
 * state recycling between slots after "GatedDeltaNet Automatic Prefix
 * Caching", section "Purpose" (copy the last computed block into the newly
 * scheduled slot).
 *
 *   num_rows   rows (tokens); 0 is a no-op.
 *   q, k       [num_rows][h_k][d_k] bf16;  v [num_rows][h_v][d_v] bf16
 *   g, beta    [num_rows][h_v] fp32 (alpha = exp(g))
 *   state      [num_slots][h_v][d_v][d_k] fp32, read at src_slot[r] and
 *              written at dst_slot[r] (in place when equal).
 *   src_slot   [num_rows] int32; a negative entry marks a padded row: it is
 *              skipped and its o rows are zeroed.
 *   dst_slot   [num_rows] int32, or NULL for dst == src.  Two rows of one
 *              call must not share a destination slot.
 *   o          [num_rows][h_v][d_v] bf16 output.
 *   dev_status optional device int32 (see GDN_DEV_*).
 * Each (row, head) reads and writes its 64 KiB (d=128) state exactly once;
 * results of a row depend only on that row's inputs and state, bit for bit.
 */
gdn_status_t gdn_decode_packed(const gdn_dims_t *dims, int32_t num_rows,
                               const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                               const float *g, const float *beta,
                               float *state, int64_t num_slots,
                               const int32_t *src_slot, const int32_t *dst_slot,
                               gdn_bf16 *o, int32_t *dev_status, void *stream);

/*
 * Input preparation ahead of the recurrence, from raw per-token projections.
 * The pages give no formula for this step (they consume prepared inputs);
 * the reading is the Gated DeltaNet layer's (Yang, Kautz, Hatamizadeh,
 * ICLR 2025):
 *     q = q_raw / sqrt(sum q_raw^2 + eps), k likewise   (per token and key head,
 *                                                         rounded to bf16)
 *     g = -exp(A_log[h]) * softplus(a + dt_bias[h]),  beta = sigmoid(b)
 *
 *   num_tokens       T >= 0 tokens.
 *   q_raw, k_raw     [T][h_k][d_k] bf16;  q, k outputs, same shape (may alias
 *                    the inputs).
 *   a, b             [T][h_v] fp32;  g, beta outputs [T][h_v] fp32.
 *   A_log, dt_bias   [h_v] fp32.
 *   eps              >= 0, added to the sum of squares.
 * The sum of squares and every later operation have one fixed order, shared
 * with gdn_decode_packed_raw: this call followed by gdn_decode_packed gives
 * the fused call's outputs and states bit for bit.
 */
gdn_status_t gdn_prep_inputs(const gdn_dims_t *dims, int64_t num_tokens,
                             const gdn_bf16 *q_raw, const gdn_bf16 *k_raw,
                             const float *a, const float *b,
                             const float *A_log, const float *dt_bias, float eps,
                             gdn_bf16 *q, gdn_bf16 *k, float *g, float *beta, void *stream);

/*
 * gdn_decode_packed with the input preparation of gdn_prep_inputs fused into
 * the kernel: q_raw, k_raw are normalised in registers and g, beta are formed
 * from a, b, A_log, dt_bias as they are loaded.  Other arguments as
 * gdn_decode_packed.
 */
gdn_status_t gdn_decode_packed_raw(const gdn_dims_t *dims, int32_t num_rows,
                                   const gdn_bf16 *q_raw, const gdn_bf16 *k_raw, const gdn_bf16 *v,
                                   const float *a, const float *b,
                                   const float *A_log, const float *dt_bias, float eps,
                                   float *state, int64_t num_slots,
                                   const int32_t *src_slot, const int32_t *dst_slot,
                                   gdn_bf16 *o, int32_t *dev_status, void *stream);

/*
 * Multi-token decode: tokens_per_row consecutive tokens per cached row, as a
 * speculative-decoding verifier feeds them.  The pages list speculative
 * decoding as unsupported ("Enable batch-invariant mixed decode and prefill
 * for Qwen GDN", section "Out of scope"; "GatedDeltaNet Automatic Prefix
 * Caching", section "Purpose", outstanding tasks); this entry point is the
 * plain reading: the recurrence of gdn_decode_packed applied token after
 * token, with the state after each token optionally kept in its own slot so
 * the caller can resume from the last accepted token.
 *
 *   num_rows, tokens_per_row  R rows of T >= 1 tokens; token t of row r is
 *              entry r*T + t of every token-major tensor.
 *   q, k       [R*T][h_k][d_k] bf16;  v, o [R*T][h_v][d_v] bf16
 *   g, beta    [R*T][h_v] fp32
 *   state      [num_slots][h_v][d_v][d_k] fp32 slot cache.
 *   src_slot   [R] int32: state entering token 0; negative = padded row
 *              (skipped, its o rows zeroed).
 *   dst_slots  [R*T] int32 or NULL.  Non-NULL: after token t the state is
 *              written to slot dst_slots[r*T + t] when that entry is >= 0
 *              (an entry >= num_slots sets GDN_DEV_BAD_SLOT and is skipped).
 *              NULL: the state after the last token is written back to
 *              src_slot[r].  Slots written by one call must be distinct,
 *              except that a row may write its own src slot.
 * The state is read once per (row, head) and kept on chip across the T
 * tokens; T tokens of one call equal T calls of gdn_decode_packed bit for
 * bit.
 */
gdn_status_t gdn_decode_multi(const gdn_dims_t *dims, int32_t num_rows, int32_t tokens_per_row,
                              const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                              const float *g, const float *beta,
                              float *state, int64_t num_slots,
                              const int32_t *src_slot, const int32_t *dst_slots,
                              gdn_bf16 *o, int32_t *dev_status, void *stream);

/*
 * Chunked varlen prefill on the 64-token chunk grid.
 * vLLM page "Enable batch-invariant mixed decode and prefill for Qwen GDN",
 * section "How" (fresh prefill rows go through chunk prefill), and
 * "GatedDeltaNet Automatic Prefix Caching", section "Purpose" (optional
 * per-chunk intermediate states as one flat stream).
 *
 *   num_seqs          sequences; sequence s holds tokens
 *                     [cu_seqlens[s], cu_seqlens[s+1]).  Empty sequences are
 *                     allowed (their final state is the initial state).
 *   cu_seqlens        device int32 [num_seqs+1], cu_seqlens[0] == 0.
 *   cu_seqlens_host   host mirror of cu_seqlens (same values), used for
 *                     validation and launch sizing; never dereferenced on
 *                     the device.
 *   q, k, v, g, beta  token-major as above, T = cu_seqlens_host[num_seqs].
 *   state, num_slots  slot cache as above.
 *   src_slot          device int32 [num_seqs]: initial state slot; a negative
 *                     entry (or src_slot == NULL) starts from S = 0.
 *   dst_slot          device int32 [num_seqs]: slot receiving the final state;
 *                     a negative entry (or dst_slot == NULL) skips the write.
 *   o                 [T][h_v][d_v] bf16.
 *   chunk_states      optional fp32 stream [n_emit][h_v][d_v][d_k].  When
 *   emit_every_chunks E > 0, after every E-th FULL 64-token chunk c of
 *                     sequence s (i.e. (c+1) % E == 0) the carried state is
 *                     written at entry emit_offset(s) + (c+1)/E - 1 where
 *                     emit_offset(s) = sum_{s' < s} floor(L_s' / (64 E)).
 *                     E = 17 puts states on the 1088-token block grid.
 *   chunk_states_capacity  entries available in chunk_states; must be at
 *                     least gdn_prefill_num_emits(...).  1 <= E <= 2^24.
 *                     Each sequence's first entry emit_offset(s) is computed
 *                     on the device from cu_seqlens (no caller-built cu_emit
 *                     array); gdn_prefill_emit_offsets() returns the same
 *                     values on the host.
 *   workspace, workspace_bytes  caller-owned device scratch of at least
 *                     gdn_prefill_workspace_bytes(dims, num_seqs, T) bytes,
 *                     256-byte aligned (NULL with 0 bytes when that is 0).
 *                     A smaller or misaligned workspace returns
 *                     GDN_ERR_WORKSPACE before any launch.
 * Resuming a sequence from the state emitted after token 64*E*j with its
 * tokens [64*E*j, L) reproduces the uninterrupted outputs and final state
 * bit for bit; so does running a sequence alone or inside any batch.
 */
gdn_status_t gdn_prefill_varlen(const gdn_dims_t *dims, int32_t num_seqs,
                                const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                const float *g, const float *beta,
                                float *state, int64_t num_slots,
                                const int32_t *src_slot, const int32_t *dst_slot,
                                gdn_bf16 *o,
                                float *chunk_states, int32_t emit_every_chunks,
                                int64_t chunk_states_capacity,
                                void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, void *stream);

/*
 * Device scratch that gdn_prefill_varlen, gdn_prefill_varlen_apc and the
 * prefill half of gdn_mixed_step need for num_seqs sequences of total_tokens
 * tokens (0 when the call needs none).  Host-only; returns (size_t)-1 for
 * bad dims or negative sizes.
 */
size_t gdn_prefill_workspace_bytes(const gdn_dims_t *dims, int32_t num_seqs, int64_t total_tokens);

/*
 * Chunked varlen prefill that writes its emitted states straight into the
 * prefix-cache blocks of the state cache, instead of a flat stream.
 * "GatedDeltaNet Automatic Prefix Caching", section "Purpose" (replay the
 * chunk history into persistent cache blocks so later requests hit the
 * prefix cache) and the review thread on its decode/prefill metadata
 * (block_idx_first_scheduled_token, block_idx_last_computed_token,
 * block_idx_last_scheduled_token); "Enable GDN batch-invariant prefix
 * caching", section "Purpose" (blocks on the 64-token chunk grid).
 *
 * Arguments as gdn_prefill_varlen, except:
 *   emit_every_chunks  E >= 1: chunks per cache block (block size 64 E).
 *   block_table        device int32 [num_seqs][block_table_stride]: the
 *                      sequence's cache slots by block index.
 *   block_first        device int32 [num_seqs]: block index that this call's
 *                      first token opens (the cached prefix length / 64 E,
 *                      i.e. block_idx_first_scheduled_token).
 * The state after token 64 E (k+1) of this call (full chunks only) goes to
 * slot block_table[s][block_first[s] + k].  A negative entry skips the
 * write; an index past the row or a slot >= num_slots sets
 * GDN_DEV_BAD_SLOT and skips it.  The values written are those that
 * gdn_prefill_varlen emits into its stream, bit for bit; o and the final
 * state (dst_slot) are the same too.
 */
gdn_status_t gdn_prefill_varlen_apc(const gdn_dims_t *dims, int32_t num_seqs,
                                    const int32_t *cu_seqlens, const int32_t *cu_seqlens_host,
                                    const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                    const float *g, const float *beta,
                                    float *state, int64_t num_slots,
                                    const int32_t *src_slot, const int32_t *dst_slot,
                                    gdn_bf16 *o, int32_t emit_every_chunks,
                                    const int32_t *block_table, int32_t block_table_stride,
                                    const int32_t *block_first,
                                    void *workspace, size_t workspace_bytes,
                                    int32_t *dev_status, void *stream);

/*
 * One mixed continuous-batching step: num_decodes cached decode rows at the
 * front of the token batch, then num_prefills fresh prefill sequences.
 * vLLM page "Enable batch-invariant mixed decode and prefill for Qwen GDN",
 * sections "How" and "Test plan" (the route regression: decode rows alone and
 * at the front of a mixed batch give bitwise equal outputs and states).
 *
 *   Token rows [0, num_decodes) are decode rows; prefill sequence s holds
 *   rows num_decodes + [cu_seqlens_p[s], cu_seqlens_p[s+1]).
 *   dec_src_slot/dec_dst_slot: as gdn_decode_packed (num_decodes entries).
 *   pre_src_slot/pre_dst_slot: as gdn_prefill_varlen (num_prefills entries).
 *   Remaining arguments as gdn_prefill_varlen; o covers all rows.  Both
 *   halves are validated before either is launched: a bad argument in the
 *   prefill half launches no decode work either.
 * The decode rows run on the same kernel and arithmetic as
 * gdn_decode_packed, so their outputs and states are bitwise identical to a
 * decode-only call, whatever prefills share the step.
 */
gdn_status_t gdn_mixed_step(const gdn_dims_t *dims, int32_t num_decodes, int32_t num_prefills,
                            const int32_t *cu_seqlens_p, const int32_t *cu_seqlens_p_host,
                            const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                            const float *g, const float *beta,
                            float *state, int64_t num_slots,
                            const int32_t *dec_src_slot, const int32_t *dec_dst_slot,
                            const int32_t *pre_src_slot, const int32_t *pre_dst_slot,
                            gdn_bf16 *o,
                            float *chunk_states, int32_t emit_every_chunks,
                            int64_t chunk_states_capacity,
                            void *workspace, size_t workspace_bytes,
                            int32_t *dev_status, void *stream);

/*
 * The same step with its two halves running at the same time: the prefill
 * on `stream`, the decode rows on `aux_stream` (cudaStream_t), so that the
 * decode blocks fill the SMs the prefill chains leave free.  Same page and
 * sections as gdn_mixed_step; the decode rows still run the decode kernel,
 * so their results are bitwise identical to gdn_mixed_step's.
 *
 *   fork_event, join_event: caller-created cudaEvent_t (no timing needed).
 *   The call records fork_event on `stream` and makes aux_stream wait for
 *   it, launches both halves, records join_event on aux_stream and makes
 *   `stream` wait for it: work issued on `stream` after the call sees both
 *   halves finished.  All of it can be captured in a CUDA graph.
 *   The decode half's slots must be disjoint from the prefill half's
 *   (the halves run concurrently).  aux_stream == NULL runs the step as
 *   gdn_mixed_step does, on `stream` alone; otherwise both events are
 *   required (GDN_ERR_INVALID_ARG).  Both halves are validated before
 *   anything is recorded or launched.
 */
gdn_status_t gdn_mixed_step_colaunch(const gdn_dims_t *dims, int32_t num_decodes, int32_t num_prefills,
                                     const int32_t *cu_seqlens_p, const int32_t *cu_seqlens_p_host,
                                     const gdn_bf16 *q, const gdn_bf16 *k, const gdn_bf16 *v,
                                     const float *g, const float *beta,
                                     float *state, int64_t num_slots,
                                     const int32_t *dec_src_slot, const int32_t *dec_dst_slot,
                                     const int32_t *pre_src_slot, const int32_t *pre_dst_slot,
                                     gdn_bf16 *o,
                                     float *chunk_states, int32_t emit_every_chunks,
                                     int64_t chunk_states_capacity,
                                     void *workspace, size_t workspace_bytes,
                                     int32_t *dev_status, void *stream,
                                     void *aux_stream, void *fork_event, void *join_event);

/* ---- host-only helpers (no device work) ------------------------------- */

/* Total emitted states of a prefill call: sum_s floor(L_s / (64 E)); 0 when
 * E <= 0; -1 on a bad argument. */
int64_t gdn_prefill_num_emits(const int32_t *cu_seqlens_host, int32_t num_seqs,
                              int32_t emit_every_chunks);

/* Per-sequence first entry in chunk_states: out[s] = emit_offset(s) for
 * s in [0, num_seqs], out[num_seqs] = total.  Returns GDN_OK or
 * GDN_ERR_INVALID_ARG. */
gdn_status_t gdn_prefill_emit_offsets(const int32_t *cu_seqlens_host, int32_t num_seqs,
                                      int32_t emit_every_chunks, int64_t *out);

/* Prefix-cache grid ("Enable GDN batch-invariant prefix caching", section
 * "Purpose"): the cache block size rounded up to a multiple of the 64-token
 * chunk (1056 -> 1088); returns -1 for block_size <= 0. */
int32_t gdn_align_block_size(int32_t block_size);

/* Usable prefix hit: floored onto the lcm(64, aligned block) grid unless the
 * hit covers the full prompt (1100 -> 1088, 200 -> 0 with 1056-token
 * blocks).  Returns -1 on a bad argument. */
int64_t gdn_floor_prefix_hit(int64_t hit_tokens, int64_t prompt_tokens, int32_t block_size);

/* Emission stride, in chunks, of the grid above (1088 / 64 = 17). */
int32_t gdn_grid_emit_every_chunks(int32_t block_size);

/* Status of a completed call from the device status word it wrote (read
 * back by the caller after the stream is done): GDN_ERR_TIMEOUT when
 * GDN_DEV_TIMEOUT is set, GDN_ERR_INVALID_ARG when only GDN_DEV_BAD_SLOT is
 * set, GDN_OK for 0. */
gdn_status_t gdn_status_from_device(int32_t dev_status_word);

const char *gdn_status_string(gdn_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
