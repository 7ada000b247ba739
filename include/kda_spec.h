/*
 * kda_spec.h -- C ABI of the GB300 (sm_103a) speculative-verify walk through a
 * Kimi-Delta-Attention (KDA) linear-attention layer.
 *
 * One verify round of K drafted tokens runs T = K+1 rows of a session through
 *   1. a depthwise causal short conv of width 4 with SiLU over the q, k, v raw
 *      rows, fed by a ring of the last 3 raw inputs,
 *   2. L2 normalisation of q and k, the forget gate g = -5 sigmoid(raw_g) per key
 *      channel and the write strength beta = sigmoid(raw_beta) per head,
 *   3. the gated delta rule on a resident f32 state S [d_k=128][d_v=128] per head:
 *        S' = diag(exp g) S;  u = S'^T k;  S = S' + beta k (v - u)^T;
 *        o = S^T q / sqrt(128)
 *      sequentially over the T rows inside one launch,
 * followed by greedy acceptance and accept-j rollback (snapshot + replay).
 * Passages (memra-engine docs.rs pages):
 *   glm_spec.rs 0.123.0, module doc "VERIFY-ROW BATCHING" (one launch per layer
 *     per round, T-loop inside the kernel, bit-identical to chained t=1 steps)
 *   glm_spec.rs, module doc "ROLLBACK" and the Glm5VerifyCkpt doc (one state
 *     snapshot per layer per round taken before row 0, stolen scan inputs,
 *     replay of rows 0..keep-1; 64 heads x 128 x 128 f32 = 4 MiB per layer)
 *   glm_spec.rs, glm5_verify_rollback / glm5_rollback_layer (keep = j+1 in 1..t;
 *     keep == t keeps the resident state)
 *   glm_spec.rs, glm5_spec_round step 4 (device argmax per verify row, lowest index
 *     wins; j = first mismatch; bonus = vam[j]) and guard_vocab_token (NaN rows)
 *   glm5_spec_ppn_gate.rs, mini fixture linear_attn_config (head_dim 128,
 *     short_conv_kernel_size 4, gate_lower_bound -5.0)
 *   glm_spec.rs, glm5_verify_rows (t <= 15: the decode-exact cap)
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller (the exceptions,
 *     pinned host memory: the source of kda_upload_rows_staged, the host rows of
 *     kda_verify_scan_deferred_host and the host buffers of kda_round_host); the
 *     library keeps none of them past the call except through the kda_stash it fills.
 *   - Every call is asynchronous on `stream` and never synchronises (the exception:
 *     kda_round_host, which waits for the round's results when asked to).
 *   - The library allocates no device memory.  spec_accept_sampled takes caller
 *     scratch; spec_accept ignores its scratch arguments.
 *   - Arguments are validated on the host before anything is launched; an
 *     invalid call returns KDA_EINVAL and enqueues nothing.  The reason is kept
 *     per thread for kda_last_error().
 *   - Conditions found on the device (a NaN row at the accept point, a device
 *     keep or row count out of range, a wait that ran out) are OR-ed as KDA_ST_*
 *     bits into the caller's device int `dev_status` (may be NULL); the caller
 *     reads it after synchronising.
 *   - Pointers to float / 16-byte vectors must be 16-byte aligned.
 */
#ifndef KDA_SPEC_H
#define KDA_SPEC_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_DK 128       /* key channels per head   (head_dim 128)            */
#define KDA_DV 128       /* value channels per head                          */
#define KDA_TMAX 15      /* rows per verify round: K <= 14 drafts            */
#define KDA_CONV_W 4     /* short_conv_kernel_size                           */
#define KDA_RING 3       /* ring slots: the last conv_w - 1 raw inputs       */
#define KDA_HOST_KEEP_MAX 2048 /* sessions per kda_rollback with host keep  */

/* return codes */
#define KDA_OK 0
#define KDA_EINVAL 1   /* bad argument; nothing was launched                 */
#define KDA_ENAN 2     /* reserved for host-side reports of KDA_ST_NAN       */
#define KDA_ECUDA 3    /* a CUDA launch or attribute call failed             */
#define KDA_ETIMEOUT 4 /* reserved for host-side reports of KDA_ST_TIMEOUT   */

/* bits OR-ed into *dev_status by kernels */
#define KDA_ST_NAN 0x1      /* accept: a consulted row holds a NaN (greedy: row j,
                               the bonus row; sampled: any row the walk reads) */
#define KDA_ST_BADKEEP 0x2  /* a device keep outside 1..T, or a device row count
                               outside 1..T (the *_var calls); that session is
                               left untouched                                    */
#define KDA_ST_TIMEOUT 0x4  /* a wait inside the scan kernel ran out (one second:
                               a bulk copy or a partner warp never arrived); the
                               CTA stopped early and its units are unfinished.
                               kda_verify_scan has no status word: a caller that
                               wants this report uses kda_verify_scan_var        */
/* 0x8 is reserved (no call raises it: the sampled filter is exact for any
   number of ties) */

/* element types of raw rows and logits */
#define KDA_F32 0
#define KDA_BF16 1

/* where kda_rollback finds keep[] */
#define KDA_MEM_HOST 0
#define KDA_MEM_DEVICE 1

/* Problem sizes.  L layers x B sessions x H heads, each an independent unit;
 * dk and dv must be 128; dtype is the element type of the raw rows. */
typedef struct kda_dims {
    int L, B, H;
    int dk, dv;
    int dtype; /* KDA_F32 or KDA_BF16 */
} kda_dims;

/* Resident per-layer state, updated in place by kda_verify_scan / kda_rollback.
 *   state     f32 [L][B][H][dk][dv]           S, d_v contiguous
 *   conv_ring f32 [L][B][H][3 stream][3 slot][dk]  raw q,k,v inputs of the last 3
 *             rows; slot 0 the oldest.  Streams in the order q, k, v.
 *   conv_w    f32 [L][H][3 stream][dk][4 tap]  tap 3 multiplies the current row,
 *             tap 0 the row three back. */
typedef struct kda_layer_state {
    float *state;
    float *conv_ring;
    const float *conv_w;
} kda_layer_state;

/* Raw (pre-conv, pre-activation) rows of one round, element type dims.dtype:
 *   q, k, v, g [L][B][T][H][128];  beta [L][B][T][H].
 * w (optional, NULL for none; zero-initialise the struct to leave it out): f32
 *   [L][B][T][H][128], 16-byte aligned, written by the verify of these rows with the
 *   update vector w_t = beta_t (v_t - S'^T k_t) of every row it runs.  A replay of
 *   these rows (kda_rollback, or the first part of the next deferred round) then
 *   reads w_t instead of forming S'^T k_t again: per row only S' = d S and
 *   S = S' + k w^T remain, the same operations on the same operands, so the state it
 *   leaves is bit-identical to a replay without w.  Like the raw rows, w is held by
 *   pointer in the stash and must stay unchanged until the replay has run; the next
 *   deferred round's rows need a different w buffer (two alternate).  The per-layer
 *   column-stash path (kda_verify_scan_cols) and kda_upload_rows_staged ignore it.
 *   Measured on GB300: a chain of deferred rounds runs 2-4 % faster with w (a
 *   replayed row costs about half a verify row); a verify followed by a separate
 *   kda_rollback runs slower with it (the verify ~3 %, the rollback 3-8 %: that
 *   replay is bound by the state's memory traffic, not by its rows), so leave w NULL
 *   for rounds committed by kda_rollback. */
typedef struct kda_rows {
    const void *q, *k, *v, *g, *beta;
    float *w;
} kda_rows;

/* Rollback material of one round (the KDA fields of the pages' verify
 * checkpoint).  The caller allocates state_snap (same shape as state) and
 * ring_snap (same shape as conv_ring); kda_verify_scan writes the pre-round state
 * and ring into them as it first reads them, and records `rows` and `T`.  The
 * stash holds the raw rows by pointer ("stolen", zero copies): they must stay
 * alive and unchanged until kda_rollback has run or the round is committed. */
typedef struct kda_stash {
    float *state_snap;
    float *ring_snap;
    kda_rows rows; /* filled by kda_verify_scan */
    int T;         /* filled by kda_verify_scan */
} kda_stash;

/*
 * kda_verify_scan -- one verify round over every (layer, session, head) unit.
 * glm_spec.rs, module doc VERIFY-ROW BATCHING (the T rows of a round run sequentially
 * inside one launch; the in-kernel T-loop over the register-resident state is the
 * chained t=1 program) and glm5_verify_rows (t <= 15); the snapshot is the pre-row-0
 * state of glm_spec.rs, ROLLBACK and the Glm5VerifyCkpt doc.
 * Rows 0..T-1 of `rows` pass through conv + SiLU, normalisation, gates and the
 * gated delta rule in one launch; state and conv_ring advance by T rows in place.
 *   out   f32 [L][B][T][H][dv] the attention outputs o_t, or NULL.
 *   stash NULL (no snapshot: a plain decode step), or a stash whose state_snap and
 *         ring_snap are non-NULL; they receive the pre-round state and ring.
 * T must lie in 1..KDA_TMAX.  With T = 1 this is exactly the chained per-row step:
 * running rows one call at a time gives bit-identical state, ring and outputs to
 * one call with all T rows.
 */
int kda_verify_scan(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows,
                    int T, float *out, kda_stash *stash, cudaStream_t stream);

/*
 * kda_rollback -- accept-j rollback of the round recorded in `stash`.
 * glm_spec.rs, glm5_verify_rollback and the KDA arm of glm5_rollback_layer (keep in
 * 1..t; keep == t keeps the resident state; else restore the snapshot and replay the
 * stolen rows 0..keep-1), module doc ROLLBACK.
 * keep[b] (= accepted drafts + 1, the anchor row is always kept) selects, per
 * session b, the state after row keep-1:
 *   keep == stash->T : nothing to do (the resident state is that state);
 *   keep <  stash->T : state <- replay of rows 0..keep-1 from state_snap, conv_ring
 *                      <- the ring after those rows, both bit-identical to a
 *                      kda_verify_scan of those rows from the snapshot.
 * keep_mem = KDA_MEM_HOST: keep is a host array [B], validated (1..T, B <=
 *   KDA_HOST_KEEP_MAX) before launch.
 * keep_mem = KDA_MEM_DEVICE: keep is a device array [B] (e.g. spec_accept's
 *   keep_out); a session whose keep is outside 1..T is left untouched and sets
 *   KDA_ST_BADKEEP in *dev_status.
 */
int kda_rollback(const kda_dims *dims, const kda_layer_state *st, const kda_stash *stash,
                 const int *keep, int keep_mem, int *dev_status, cudaStream_t stream);

/*
 * kda_verify_scan_pingpong -- a verify round with the state kept in two buffers whose
 * roles swap every round, so that the snapshot costs no copy (the pages' verify
 * snapshots the state with a device-to-device clone before row 0; glm_spec.rs,
 * ROLLBACK and the Glm5VerifyCkpt doc).
 * On entry stash->state_snap and stash->ring_snap hold the PRE-round state and conv
 * ring of every unit.  They are read and left untouched, and so are this round's
 * snapshot.  The post-round state and ring are written to st->state and
 * st->conv_ring, whose previous contents are ignored.  kda_rollback /
 * kda_rollback_var of the stash then restore from the pre-round buffers as usual.
 * Before the next round the caller swaps the buffers: st->state and st->conv_ring
 * (the committed state) become the next stash->state_snap and ring_snap, and the old
 * snapshot buffers become the next st->state and conv_ring.
 *   t_rows NULL: every session runs T rows; else per-session row counts with t_mem
 *   and dev_status as for kda_verify_scan_var (a session whose device count is out
 *   of range is not written at all and sets KDA_ST_BADKEEP).
 * State, ring and outputs are bit-identical to kda_verify_scan (or _var) run from the
 * same pre-round state.  Per head the state moves 2 x 64 KiB instead of 3 x 64 KiB.
 * The two buffers must not overlap.
 */
int kda_verify_scan_pingpong(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows, int T,
                             const int *t_rows, int t_mem, float *out, kda_stash *stash, int *dev_status,
                             cudaStream_t stream);

/*
 * kda_verify_scan_deferred -- a ping-pong verify round that first applies the
 * previous round's accept, in the same launch (the rollback of glm_spec.rs,
 * glm5_verify_rollback, deferred into the next round's verify).
 * On entry the stash and st describe the previous ping-pong round exactly as
 * kda_verify_scan_pingpong left them: stash->state_snap / ring_snap its pre-round
 * state and ring, stash->rows / stash->T its raw rows (still alive), st->state /
 * conv_ring its post-round state and ring.  prev_keep is a DEVICE int32 [B] array,
 * the previous round's keep (e.g. spec_accept's keep_out).
 * Per session b, the committed state is the previous post-round state when
 * prev_keep[b] == stash->T, else the replay of the previous rows 0..prev_keep[b]-1
 * from the previous pre-round state (bit-identical to kda_rollback); this round's T
 * rows (`rows`, outputs to `out`) then run from the committed state.
 * On return the library has exchanged st->state with stash->state_snap and
 * st->conv_ring with stash->ring_snap, and recorded `rows` and T in the stash, so that
 * the stash holds this round's snapshot (the committed state) and st its post-round
 * state: the pair is again as a ping-pong verify leaves it, ready for kda_rollback, a
 * further deferred round or (after swapping the pointers back) a ping-pong verify.
 * Results are bit-identical to kda_rollback of the previous round followed by
 * kda_verify_scan_pingpong of this one.  A session whose prev_keep lies outside
 * 1..stash->T is not processed at all (KDA_ST_BADKEEP is set in *dev_status, which
 * may be NULL).  Per head the state moves 3 x 64 KiB when the session rolls back and
 * 2 x 64 KiB when it kept every row, against 4 x 64 KiB for the two separate launches.
 * The last round of a sequence is committed with an ordinary kda_rollback.
 */
int kda_verify_scan_deferred(const kda_dims *dims, kda_layer_state *st, kda_stash *stash, const int *prev_keep,
                             const kda_rows *rows, int T, float *out, int *dev_status, cudaStream_t stream);

/*
 * kda_verify_scan_deferred_staged -- kda_verify_scan_deferred whose raw rows may still
 * be arriving when it starts (the round's inputs streamed in by range of (layer,
 * session) pairs, so that the host-to-device copy overlaps the scan of the pairs already
 * in place; glm_spec.rs, VERIFY-ROW BATCHING: one launch a round).
 * ready_flags: DEVICE array of unsigned flags; the raw rows of pair lb = l * B + b
 * (q, k, v, g and beta of layer l, session b) may be read once
 * ready_flags[lb / pairs_per_flag] has reached `epoch` (compared as
 * (int)(flag - epoch) >= 0, so a counter may wrap).  The caller copies each range of
 * pairs and then sets its flag in stream order after the copy (kda_upload_rows_staged,
 * or its own copies and kda_stream_write_u32 on the copy's stream).  The kernel waits
 * for a flag at most one second; a flag that does not arrive sets KDA_ST_TIMEOUT in
 * *dev_status and the launch ends early, its results undefined.  The previous round's
 * rows (stash->rows) must be in place.  Everything else, including the results, is as
 * for kda_verify_scan_deferred.  pairs_per_flag must be >= 1; ready_flags 4-byte aligned.
 */
int kda_verify_scan_deferred_staged(const kda_dims *dims, kda_layer_state *st, kda_stash *stash,
                                    const int *prev_keep, const kda_rows *rows, int T, float *out,
                                    const unsigned *ready_flags, int pairs_per_flag, unsigned epoch,
                                    int *dev_status, cudaStream_t stream);

/*
 * kda_verify_scan_deferred_host -- kda_verify_scan_deferred whose raw rows this round
 * are read in place from pinned host memory (host_rows: q, k, v, g, beta in the layout
 * of kda_rows, allocated so that the device can address them, e.g. cudaHostAlloc; the
 * call takes their device addresses from cudaHostGetDevicePointer) over the host link
 * while the launch runs, instead of being copied to the device first.  `rows` names
 * device tensors of the same shapes that receive a copy of them, written by the launch
 * (and rows->w, the update vectors, as for the other entry points); the stash records
 * `rows`, so the next round's replay reads the device copy and host_rows may change as
 * soon as the launch has completed.  Everything else, and the results, as for
 * kda_verify_scan_deferred.  A session whose prev_keep is invalid is not processed and
 * its rows are not copied.  KDA_EINVAL when host_rows is NULL or not addressable by the
 * device, and for whatever kda_verify_scan_deferred refuses.
 */
int kda_verify_scan_deferred_host(const kda_dims *dims, kda_layer_state *st, kda_stash *stash, const int *prev_keep,
                                  const kda_rows *host_rows, const kda_rows *rows, int T, float *out, int *dev_status,
                                  cudaStream_t stream);

/*
 * kda_stream_write_u32 -- *flag = value (a 4-byte aligned device address) in the order
 * of `stream`, written by the stream itself (a stream memory operation, no kernel), as
 * the ready flags of kda_verify_scan_deferred_staged want.  KDA_ECUDA when the driver
 * refuses it.
 */
int kda_stream_write_u32(unsigned *flag, unsigned value, cudaStream_t stream);

/*
 * kda_upload_rows_staged -- the host-to-device copy that feeds
 * kda_verify_scan_deferred_staged: for each range of pairs_per_flag (layer, session)
 * pairs (the last may be shorter), one cudaMemcpyAsync per raw-row tensor (q, k, v, g,
 * beta, layout as for kda_verify_scan) of that range from src (host memory, pinned for
 * the copies to be asynchronous) to dst (device), then ready_flags[range] = epoch, all in
 * the order of `stream` (a stream other than the launch's, so that the copies overlap
 * the scan).  Where q, k, v and g lie at one distance from each other in both dst and
 * src (four equal tensors in one allocation), a range of the four is one 2D copy.
 * dims gives L, B, H and the element type; T the rows a round.  Allocates nothing and
 * does not synchronise.  KDA_EINVAL for NULL pointers, T outside 1..15 or
 * pairs_per_flag < 1; KDA_ECUDA when a copy or the flag write is refused.
 */
int kda_upload_rows_staged(const kda_dims *dims, const kda_rows *dst, const kda_rows *src, int T,
                           unsigned *ready_flags, int pairs_per_flag, unsigned epoch, cudaStream_t stream);

/*
 * kda_round_host -- one speculative round end to end from host memory, in one call:
 * glm_spec.rs, glm5_spec_round (a round is verify, accept and rollback, and the next
 * round's drafts follow from this round's accept, so the host reads j every round).
 *   host_rows, host_logits [B][T][V] (logit_dtype), host_drafts int32 [B][T-1]: the
 *     round's inputs in host memory (pinned, for the copies to be asynchronous);
 *   dev_rows, dev_logits, dev_drafts: device buffers of the same shapes they go to.
 *     A deferred round replays the previous round's raw rows, so consecutive calls
 *     need different dev_rows (two sets alternate), and different dev_rows.w when
 *     the update vectors are kept;
 *   dev_jbk: device int32 [3][B]: j, bonus and keep of this round; the keep row is also
 *     the previous round's keep that this round's verify applies (same buffer every call);
 *   host_jb: host int32 [2][B] (pinned) receiving j and the bonus; where the device can
 *     address it (cudaHostGetDevicePointer succeeds) the accept writes them there
 *     directly and dev_jbk's j and bonus rows are not written, else they are copied back;
 *   ready_flags, pairs_per_flag, epoch: as for kda_verify_scan_deferred_staged (a new
 *     epoch each call);
 *   stream: the verify and the accept; copy_stream: the uploads (another stream);
 *   rows_in_place != 0: after the first call the raw rows are not copied: the verify
 *     reads them in place from host_rows and writes dev_rows as their device copy
 *     (kda_verify_scan_deferred_host; ready_flags and pairs_per_flag are then unused);
 *   wait != 0: return after the results are in host_jb: when the accept writes them
 *     there directly, the call fills host_jb with INT_MIN first and reads it until every
 *     entry has been written (at most one second, then cudaStreamSynchronize), which
 *     returns before the stream's own completion is signalled; else
 *     cudaStreamSynchronize(stream).  An earlier call made with wait == 0 must have
 *     completed first (its accept could otherwise still write host_jb);
 * First call of a chain (stash->T == 0): the committed state and ring are in
 * stash->state_snap / ring_snap, st's buffers are the spare pair; the rows, logits and
 * drafts go up on `stream`, then kda_verify_scan_pingpong, spec_accept and the copy of
 * j and the bonus.  Later calls: kda_verify_scan_deferred_staged on `stream` (the
 * previous round's accept folded in; it scans a range once its flag is set, so only
 * the first range's copy precedes the scan), then on copy_stream kda_upload_rows_staged
 * of the rows by range and the logits and drafts, spec_accept once those have landed,
 * then the results.  A copy refused after the launch leaves the launch waiting for its
 * flag until the one-second bound (KDA_ST_TIMEOUT in *dev_status).  On return st and stash describe this round as those entry points leave
 * them (the last round of a chain is committed with kda_rollback and the keep row of
 * dev_jbk).  The results are bit-identical to issuing those calls one by one.
 * Allocates no memory (one CUDA event is created and released per call).  KDA_EINVAL
 * for NULL buffers, T outside 1..15, V < 1, a bad logit_dtype or copy_stream ==
 * stream after the first call, and whatever the entry points it issues refuse.
 */
int kda_round_host(const kda_dims *dims, kda_layer_state *st, kda_stash *stash, int T, const kda_rows *host_rows,
                   const kda_rows *dev_rows, const void *host_logits, void *dev_logits, int logit_dtype, int V,
                   const int *host_drafts, int *dev_drafts, int *dev_jbk, int *host_jb, float *out,
                   unsigned *ready_flags, int pairs_per_flag, unsigned epoch, int *dev_status, cudaStream_t stream,
                   cudaStream_t copy_stream, int rows_in_place, int wait);

/*
 * Rounds whose length differs per session (variable T inside one batched grid).
 * glm_spec.rs, glm5_conf_keep and the p-min break of the draft chain, and dflash.rs,
 * DsparkVtPolicy / dspark_confidence_vt / dspark_slot_confidence_vt: each session
 * sends its own number of drafted rows through verify.  The raw-row, output and
 * logits layouts keep T (the cap) rows per session; session b uses rows
 * 0..t_rows[b]-1 of them and the rest are neither read nor written.
 *
 * kda_verify_scan_var -- kda_verify_scan where session b runs t_rows[b] rows
 *   (1 <= t_rows[b] <= T).  t_mem: KDA_MEM_HOST (validated before launch, B <=
 *   KDA_HOST_KEEP_MAX) or KDA_MEM_DEVICE (a session whose count is out of range is
 *   left untouched, its snapshot unwritten, and KDA_ST_BADKEEP is set in
 *   *dev_status, which may be NULL).  The stash records T; the row counts are
 *   passed again to kda_rollback_var.  Bit-identical, per session, to
 *   kda_verify_scan of that session's t_rows[b] rows.
 */
int kda_verify_scan_var(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows, int T,
                        const int *t_rows, int t_mem, float *out, kda_stash *stash, int *dev_status,
                        cudaStream_t stream);

/*
 * kda_rollback_var -- accept-j rollback of a round run by kda_verify_scan_var.
 *   t_rows and keep are both host arrays (mem = KDA_MEM_HOST, validated: 1 <= keep[b]
 *   <= t_rows[b] <= T) or both device arrays (mem = KDA_MEM_DEVICE; an invalid pair
 *   leaves the session untouched and sets KDA_ST_BADKEEP).  keep[b] == t_rows[b]:
 *   nothing to do for that session; otherwise rows 0..keep[b]-1 are replayed from the
 *   snapshot, as in kda_rollback.
 */
int kda_rollback_var(const kda_dims *dims, const kda_layer_state *st, const kda_stash *stash,
                     const int *t_rows, const int *keep, int mem, int *dev_status, cudaStream_t stream);

/*
 * Column-stash rollback, the alternative the pages weigh against snapshot + replay
 * (glm_spec.rs module doc, ROLLBACK: vLLM keeps num_spec + 1 KDA state columns and
 * commits the last accepted one; the pages keep the snapshot + replay, since the
 * columns cost 136 MiB per column per round).  Offered to measure that trade.
 *
 * kda_verify_scan_cols -- kda_verify_scan that also writes the state and conv ring
 *   after every row:
 *     state_cols f32 [L][B][H][T][dk][dv], ring_cols f32 [L][B][H][T][3][3][dk],
 *   caller-owned device memory, 16-byte aligned.  No snapshot is taken.  State, ring
 *   and outputs are bit-identical to kda_verify_scan; column t is bit-identical to the
 *   state (ring) a verify of rows 0..t leaves.
 * kda_rollback_cols -- commit keep[b] rows (1..T) of that round: for keep < T, state
 *   <- state_cols[keep-1] and conv_ring <- ring_cols[keep-1] (a copy, no replay);
 *   bit-identical to kda_rollback of a snapshot round.  keep as for kda_rollback.
 */
int kda_verify_scan_cols(const kda_dims *dims, const kda_layer_state *st, const kda_rows *rows, int T,
                         float *out, float *state_cols, float *ring_cols, cudaStream_t stream);
int kda_rollback_cols(const kda_dims *dims, const kda_layer_state *st, const float *state_cols,
                      const float *ring_cols, int T, const int *keep, int keep_mem, int *dev_status,
                      cudaStream_t stream);

/*
 * spec_accept_var -- spec_accept where session b's round has t_rows[b] rows
 *   (device int32 [B]).  logits stay [B][T][V] and drafts [B][T-1]; session b reads
 *   logits rows 0..t_rows[b]-1 and drafts 0..t_rows[b]-2: j = the first r <
 *   t_rows[b]-1 whose draft misses, else t_rows[b]-1; bonus = vam[j]; keep = j+1.
 *   A count outside 1..T gives j = -1, bonus = -1, keep = 0 and KDA_ST_BADKEEP.
 *   scratch, scratch_bytes: not used, as for spec_accept.
 */
int spec_accept_var(const void *logits, int logit_dtype, int B, int T, int V, const int *t_rows,
                    const int *drafts, int *j_out, int *bonus_out, int *keep_out, int *dev_status,
                    void *scratch, size_t scratch_bytes, cudaStream_t stream);

/* verify-window policies of spec_window */
#define KDA_WIN_CONF_KEEP 0       /* glm5_conf_keep: scores = draft-slot confidences q;
                                     param = p_min; pmin0 arms the break at slot 0;
                                     rows = 1 + kept drafts                          */
#define KDA_WIN_CONFIDENCE 1      /* dspark_confidence_vt: scores = pre-sigmoid slot
                                     scores; param = tau on the cumulative survival
                                     prod sigmoid(score); rows in [2, max(t_cap, 2)] */
#define KDA_WIN_SLOT_CONFIDENCE 2 /* dspark_slot_confidence_vt: per-slot
                                     sigmoid(score) >= tau; rows in [2, max(t_cap, 2)] */

/*
 * spec_window -- per-session verify rows from the drafter's slot scores, on the device.
 *   scores: device f32 [B][K] (slot k of session b: the score of draft k+1);
 *   t_out: device int32 [B], the rows of each session's round, capped at t_cap
 *   (1..15 for KDA_WIN_CONF_KEEP, 2..15 for the confidence policies).  Keeping
 *   stops at the first slot that fails (a kept draft after a dropped one could never
 *   be accepted).  The decisions are taken in f32: a strict "<" against the
 *   threshold, the survival multiplied in slot order, sigmoid(x) = 1 / (1 + exp(-x)).
 */
int spec_window(const float *scores, int B, int K, int policy, float param, int pmin0, int t_cap,
                int *t_out, cudaStream_t stream);

/*
 * Sampled acceptance.  glm_spec.rs module doc, SAMPLED ACCEPTANCE, and
 * glm5_sampled_accept / glm5_sampled_bonus: the rejection-sampling walk over the
 * verify rows.  Target p (verify rows) and draft q (the rows the drafts were drawn
 * from) go through one filter (filter_stats + softmax_gather_filtered):
 *   z = x / temperature, e = exp(z - max z) (both f32), S = sum e; a token is kept
 *   when it passes every enabled threshold on e: top_k (e >= the k-th largest e,
 *   ties kept), top_p (e >= e_(n), n the first count of the descending-sorted e
 *   whose running sum reaches top_p * S, ties kept), min_p (e >= min_p);
 *   p~ = e / Z over the kept tokens, Z their sum.  S, Z and every running sum are
 *   exact integer sums of the weights in units of 2^-46 (no sum depends on the order
 *   of its terms; a 64-bit sum of V weights of at most 1 holds V up to KDA_SAMPLED_VMAX,
 *   larger V is refused with KDA_EINVAL); top_p is exact for any top_k (0 included) and
 *   any number of ties.
 * Draft r is accepted iff u_r * q~_r(x_r) < p~_r(x_r), compared in double on the f32
 * values of p~ and q~ (the page's (u as f64) * (qj as f64) < pj as f64); the walk
 * stops at the first rejection j.  j < K: the token is drawn from max(0, p~_j - q~_j)
 * (from p~_j if that is zero everywhere); j = K: the bonus is drawn from p~_K.  A
 * draw takes the first token, in vocabulary order, whose running weight exceeds
 * u * (total weight).  Every result is reproducible bit for bit from the
 * inputs (and, for the session form, the counters).
 */
#define KDA_SAMPLED_VMAX 262143 /* 2^18 - 1: V * 2^46 stays below 2^64 */

typedef struct kda_sampling {
    float temperature; /* > 0                                                  */
    int top_k;         /* 0 off; >= 1 keeps the k largest (>= V: every token)  */
    float top_p;       /* (0, 1]; 1 off                                        */
    float min_p;       /* [0, 1); 0 off                                        */
} kda_sampling;

/*
 * spec_accept_sampled -- sampled acceptance for B sessions with caller uniforms.
 *   logits [B][T][V] and draft_logits [B][T-1][V] (logit_dtype), drafts int32
 *   [B][T-1], u_accept f32 [B][T-1] and u_sample f32 [B] in [0, 1), all device
 *   memory; sp a host struct.  Outputs device int32 [B]: j_out (accepted drafts),
 *   token_out (the residual draw, or the bonus at j = K), keep_out (j + 1, may be
 *   NULL).  A consulted row holding a NaN or no finite maximum gives token -1 and
 *   sets KDA_ST_NAN.  A draft id outside 0..V-1 is rejected.
 *   scratch: device memory of at least spec_accept_sampled_scratch_bytes(B, T)
 *   bytes, 16-byte aligned, for the per-row filter statistics (the target and draft
 *   rows are filtered in parallel, then each session walks); no initialisation needed.
 */
size_t spec_accept_sampled_scratch_bytes(int B, int T);
int spec_accept_sampled(const void *logits, const void *draft_logits, int logit_dtype, int B, int T, int V,
                        const int *drafts, const float *u_accept, const float *u_sample, const kda_sampling *sp,
                        int *j_out, int *token_out, int *keep_out, int *dev_status, void *scratch,
                        size_t scratch_bytes, cudaStream_t stream);

/*
 * spec_accept_sampled_session -- the same walk drawing its uniforms from each
 * session's own counter-based stream.  glm_spec.rs, SAMPLED ACCEPTANCE and the
 * Glm5SpecSession doc: the accept-test uniforms come from the session's uctr on the
 * Philox4x32-10 stream tagged 0xFFFF_FFFE (spec::host_u01), every device draw
 * advances its sctr, and the counters live on the session so randomness never
 * repeats across calls.
 *   seeds    uint64 [B], device: the key of session b's stream is (seed low, seed high)
 *   counters uint32 [B][2], device, read and written: (uctr, sctr) of session b
 * Uniform of counter n under tag t: output word 0 of Philox4x32-10 at counter
 * (n, 0, 0, t), its top 24 bits times 2^-24.  Accept test r of a round uses
 * (uctr + r, 0xFFFFFFFE); the residual or bonus draw uses (sctr, 0xFFFFFFFF).  After
 * the call uctr has advanced by the tests run (j + 1 when draft j was rejected, K
 * when every draft passed) and sctr by one.  Other arguments and results as
 * spec_accept_sampled; the same scratch size.  seeds and counters 8-byte aligned.
 */
int spec_accept_sampled_session(const void *logits, const void *draft_logits, int logit_dtype, int B, int T, int V,
                                const int *drafts, const unsigned long long *seeds, unsigned *counters,
                                const kda_sampling *sp, int *j_out, int *token_out, int *keep_out, int *dev_status,
                                void *scratch, size_t scratch_bytes, cudaStream_t stream);

/*
 * kda_philox4x32_10 -- the library's counter-based generator on the device:
 * out[i] = Philox4x32-10(ctr[i], key[i]) (Salmon, Moraes, Dror and Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3", SC'11; ten rounds), for i < n.
 *   ctr uint32 [n][4] and out uint32 [n][4], 16-byte aligned; key uint32 [n][2],
 *   8-byte aligned; device memory.
 */
int kda_philox4x32_10(const unsigned *ctr, const unsigned *key, unsigned *out, int n, cudaStream_t stream);

/* Bytes of the per-slice partial results of B sessions of T rows of V logits in the
 * two-launch accept (the bound of spec_accept_noalloc). */
size_t spec_accept_scratch_bytes(int B, int T, int V);

/*
 * spec_accept -- greedy acceptance for B sessions.
 * glm_spec.rs, glm5_spec_round step 4 (one device argmax per verify row, lowest index
 * wins, then the longest matching prefix; keep = j + 1) and guard_vocab_token (a NaN
 * row is refused).
 *   logits [B][T][V] (KDA_F32 or KDA_BF16, logit_dtype), drafts int32 [B][T-1]
 *   (drafts[b][r] is the token drafted for the position that row r predicts).
 * Per session: vam[r] = index of the maximum of row r, the lowest index winning
 * ties (bf16 compared after exact widening); a row holding a NaN has no argmax.
 * j = the first r < T-1 with drafts[r] != vam[r] (or a NaN row), else T-1;
 * bonus = vam[j]; keep = j + 1.
 * Outputs (device int32 [B], each may be NULL): j_out, bonus_out, keep_out.  If
 * row j holds a NaN, bonus is -1 and KDA_ST_NAN is set in *dev_status.
 * scratch, scratch_bytes: not used (NULL and 0 are fine).  The one launch of
 * thread-block clusters passes its partial results through shared memory; the
 * arguments remain for existing callers.  spec_accept_scratch_bytes(B, T, V) is the
 * size of the partial results of the two-launch form (spec_accept_noalloc).
 */
int spec_accept(const void *logits, int logit_dtype, int B, int T, int V, const int *drafts,
                int *j_out, int *bonus_out, int *keep_out, int *dev_status, void *scratch,
                size_t scratch_bytes, cudaStream_t stream);

/*
 * spec_accept_noalloc -- spec_accept without caller scratch.  The pages have no
 * counterpart: this entry point exists for callers of this library that cannot
 * allocate device memory when they accept a round, for example a serving loop
 * whose device memory is all handed out up front by a fixed arena, or a host
 * path that must not call cudaMalloc / cudaFree because those calls can
 * synchronise the device.
 * Arguments and results are those of spec_accept.  The partial results live in
 * one fixed device array of KDA_NOALLOC_SCRATCH_BYTES inside the library, which
 * every GPU that loads the library holds until the process exits.  Calls whose
 * spec_accept_scratch_bytes(B, T, V) exceeds it return KDA_EINVAL and launch
 * nothing.  The first call on a device looks up the array's device address with
 * that device current and keeps it with the context it belongs to; make that
 * first call before any stream capture.  A later call in another context (after
 * cudaDeviceReset, or in a context the caller made current) looks the address up
 * again, and the same advice holds for it.  The array keeps the last call's
 * contents; nothing in it needs to start at zero.
 * All calls share the one array, so calls that overlap on the GPU (for instance
 * on two streams at once) race; order them on one stream or with events.
 * The library calls no allocation routine for this entry point.
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)1 << 20)
int spec_accept_noalloc(const void *logits, int logit_dtype, int B, int T, int V, const int *drafts,
                        int *j_out, int *bonus_out, int *keep_out, int *dev_status, cudaStream_t stream);

/* Static description of a return code, and the calling thread's last error text. */
const char *kda_error_string(int code);
const char *kda_last_error(void);

/* Library version, for the binding's load check. */
int kda_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_SPEC_H */
