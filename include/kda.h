/*
 * kda.h: C ABI of libkda.so, the GB300 (sm_103a) implementation of the Kimi Delta Attention
 * (KDA) gated delta-rule state recurrence.
 *
 * The operation. Per sequence and head, with state S in R^{dk x dv} (row = key channel):
 *     S_t = (I - beta_t k_t k_t^T) Diag(a_t) S_{t-1} + beta_t k_t v_t^T,   a_t = exp(g_t)
 *     o_t = scale * S_t^T q_t
 * g_t in R^{dk} is a per-key-channel log-decay (g <= 0), beta_t a scalar write strength.
 * Every call accepts any g <= 0: the chunked calls compute a channel that decays by more than
 * 160 nats within one 64-token chunk without the chunk's shared exponent frame, so no decay
 * is too strong (results match the recurrence up to rounding).
 * This is the KDA linear-attention state that pegainfer PR #970 ("feat(k3): cross-process
 * CP whale gang - fleet-wide long-prompt prefill") prefills with FlashKDA per context-parallel
 * segment; each segment publishes its (M,D) package, and the packages are combined by an
 * exchange or, at lower traffic, a Blelloch prefix scan (whale-rendezvous and fabric
 * data-plane commit messages).
 * kern PR #44 keeps one KDA state block per packed sequence (varlen, cu_seqlens) and
 * ATOM PR #2709 ("feat(kimi-k3): PP8 prefill for P/D serving - KDA state under PP")
 * updates slot-addressed KDA state one decode token at a time.
 *
 * Layouts (all row-major, contiguous, device memory unless stated):
 *     q, k, g : [tokens, H, dk]     v, o : [tokens, H, dv]     beta : [tokens, H]
 *     states  : [n, H, dk, dv]      M : [n_segs, H, dk, dk]    D : [n_segs, H, dk, dv]
 * q, k, v and o have the dtype given by kda_dtype; g, beta and all states are fp32.
 * Sequences (or segments) are packed back to back along the token axis and delimited by
 * int32 offset arrays (cu_seqlens[0] = 0, non-decreasing, last = total tokens).
 *
 * Supported shapes: dk = dv in {64, 128}; chunk = 64.
 *
 * Ownership and ordering. The caller owns every buffer. Each call borrows the pointers for
 * the stream-ordered duration of the work it enqueues on `stream`; no call allocates device
 * memory, synchronises the device or keeps state between calls (the one exception being the
 * process-wide message returned by kda_last_error). Outputs must not alias inputs, except
 * that the decode pool is read and written in place.
 *
 * Errors. Argument checks run on the host before any launch and return
 * KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED / KDA_ERR_WORKSPACE without enqueuing work;
 * a failed launch returns KDA_ERR_CUDA. kda_last_error() then describes the failure.
 * Conditions only the device can see are OR-ed into the optional device word `status`
 * (see KDA_STATUS_*); the caller clears it and reads it back when convenient. Nothing
 * traps, and no call falls back to another implementation.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kda_stream_t; /* same type as cudaStream_t; NULL = legacy stream */

typedef enum {
  KDA_OK = 0,
  KDA_ERR_INVALID_ARG = 1, /* null pointer, negative size, misaligned pointer, bad offsets */
  KDA_ERR_UNSUPPORTED = 2, /* shape or dtype outside the supported set */
  KDA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the query returned */
  KDA_ERR_CUDA = 4         /* a CUDA runtime/launch error; see kda_last_error() */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype; /* dtype of q, k, v and o */

/* Bits OR-ed into the optional device status word. */
#define KDA_STATUS_BAD_SLOT 1u    /* decode: a slot id >= n_slots was skipped */
/* (bit 2u is not used) */
#define KDA_STATUS_BAD_OFFSETS 4u /* an offset array was decreasing or out of range, or a
                                     sequence had more segments than max_segs_per_seq; the
                                     offending range was treated as empty */
#define KDA_STATUS_TIMEOUT 8u     /* a tensor-core CTA waited more than 2 s for its own copies
                                     or MMAs and stopped early; its outputs are incomplete */

/* Message for the most recent non-OK status returned on this thread ("" if none). */
KDA_API const char* kda_last_error(void);

/* Library version string. */
KDA_API const char* kda_version(void);

/* Number of CUDA kernels this process has launched through the library so far (a
 * diagnostic counter for benchmarks; every successful entry point adds its launches). */
KDA_API uint64_t kda_launch_count(void);

/*
 * kda_chunk_workspace: bytes of device scratch that kda_chunk_prefill, kda_segment_package
 * and kda_segment_replay need for n_ranges sequences (or segments) over total_tokens tokens;
 * 0 when such a call needs none (fp32 inputs, dk = dv = 64, or H not a multiple of 4, all
 * served by the CUDA-core kernel). The tensor-core path precomputes every state-independent
 * factor of each (64-token chunk, head) into one record of 147,968 bytes; it keeps
 * R = (total_tokens / 64 + n_ranges) * H records, then a 4-byte ready flag per record
 * (rounded up to a multiple of 256 bytes): R * 147968 + roundup(4 R, 256) bytes.
 */
KDA_API size_t kda_chunk_workspace(kda_dtype dt, int n_ranges, int total_tokens, int H, int dk,
                                   int dv);

/*
 * kda_chunk_prefill: chunked (WY/UT form) prefill over packed sequences.
 *   n_seqs      number of sequences (>= 0); total_tokens = cu_seqlens[n_seqs].
 *   cu_seqlens  device int32 [n_seqs + 1]; may be NULL when n_seqs == 1 (one sequence of
 *               total_tokens tokens).
 *   init_state  [n_seqs, H, dk, dv] fp32 entry states, or NULL for zeros.
 *   o           [total_tokens, H, dv] output (dtype dt).
 *   final_state [n_seqs, H, dk, dv] fp32 exit states, or NULL.
 *   workspace   device scratch of at least kda_chunk_workspace(dt, n_seqs, total_tokens, H,
 *               dk, dv) bytes, 256-byte aligned, contents need not be initialised; may be
 *               NULL when that query returns 0 (KDA_ERR_WORKSPACE otherwise).
 *   status      optional device word (KDA_STATUS_BAD_OFFSETS, KDA_STATUS_TIMEOUT).
 * q, k, v, g, beta, o and the states must be 16-byte aligned (KDA_ERR_INVALID_ARG otherwise).
 * A shape whose workspace query is positive runs on the tensor-core kernels and on nothing
 * else: if the CUDA driver does not provide cuTensorMapEncodeTiled, the call returns
 * KDA_ERR_UNSUPPORTED. The same holds for every chunked call below.
 * Source: the chunked FlashKDA prefill of kern PR #44 (varlen build with cu_seqlens and
 * per-sequence state blocks) and pegainfer PR #970 (fabric data-plane commit message: the
 * segment replay runs the same per-chunk step as the prefill).
 */
KDA_API kda_status kda_chunk_prefill(kda_dtype dt, int n_seqs, int total_tokens,
                             const int32_t* cu_seqlens, int H, int dk, int dv, int chunk,
                             float scale, const void* q, const void* k, const void* v,
                             const float* g, const float* beta, const float* init_state,
                             void* o, float* final_state, void* workspace,
                             size_t ws_bytes, uint32_t* status, kda_stream_t stream);

/*
 * kda_segment_package: per-segment affine (M, D) packages. For each segment
 * [seg_offsets[p], seg_offsets[p+1]) and head, writes M [dk, dk] and D [dk, dv] such that
 * running the recurrence over the segment from any entry state S_in ends in
 * M S_in + D. No outputs o are produced and q is not read.
 *   seg_offsets device int32 [n_segs + 1].
 *   workspace   as for kda_chunk_prefill, sized by kda_chunk_workspace(dt, n_segs, ...).
 *   k, v, g, beta, M and D 16-byte aligned.
 * Source: pegainfer PR #970, fabric data-plane commit message (the (M,D) package each
 * context-parallel member publishes for its segment).
 */
KDA_API kda_status kda_segment_package(kda_dtype dt, int n_segs, int total_tokens,
                               const int32_t* seg_offsets, int H, int dk, int dv, int chunk,
                               const void* k, const void* v, const float* g,
                               const float* beta, float* M, float* D, void* workspace,
                               size_t ws_bytes, uint32_t* status, kda_stream_t stream);

/*
 * kda_package_scan: segmented exclusive prefix over packages with the composition
 * (M2, D2) o (M1, D1) = (M2 M1, M2 D1 + D2), applied to the entry state:
 *     seg_init[j]    = M_{<j} S_init + D_{<j}   (the state entering segment j)
 *     final_state[s] = M_{all} S_init + D_{all} (the state after the sequence)
 * Segments [seq_seg_offsets[s], seq_seg_offsets[s+1]) belong to sequence s, in token order.
 * Two schedules of the same prefix (equal up to rounding order): for dk = dv = 128 and
 * max_segs_per_seq <= 256, the sequential chain S_{j+1} = M_j S_j + D_j (one dependent product
 * per segment, the state's columns split over CTAs); otherwise a work-efficient (Blelloch)
 * up-sweep/down-sweep tree per (sequence, head).
 *   seq_seg_offsets   device int32 [n_seqs + 1] (last = n_segs).
 *   max_segs_per_seq  host upper bound on any sequence's segment count (1..65536); it picks
 *                     the schedule and sets the number of tree levels launched. A sequence
 *                     with more segments is malformed (KDA_STATUS_BAD_OFFSETS).
 *   init_state        [n_seqs, H, dk, dv] or NULL (zeros).
 *   seg_init          [n_segs, H, dk, dv] output.  final_state [n_seqs, H, dk, dv] or NULL.
 *   M, D, init_state, seg_init, final_state: 16-byte aligned.
 *   workspace         device scratch of at least kda_package_scan_workspace(...) bytes,
 *                     256-byte aligned; contents need not be initialised. It holds the
 *                     padded tree: n_seqs * (3/2) * P2 * H packages of (dk*dk + dk*dv) fp32,
 *                     P2 = max_segs_per_seq rounded up to a power of two (the sequential
 *                     chain leaves it untouched).
 *   status            optional device word (KDA_STATUS_BAD_OFFSETS; KDA_STATUS_TIMEOUT if a
 *                     tensor-core CTA's bounded wait expired).
 * Source: pegainfer PR #970, whale-rendezvous commit message (a Blelloch prefix scan over the
 * packages as the lower-traffic way to combine them).
 */
KDA_API size_t kda_package_scan_workspace(int n_seqs, int max_segs_per_seq, int H, int dk, int dv);
KDA_API kda_status kda_package_scan(int n_seqs, int n_segs, const int32_t* seq_seg_offsets,
                            int max_segs_per_seq, int H, int dk, int dv, const float* M,
                            const float* D, const float* init_state, float* seg_init,
                            float* final_state, void* workspace, size_t ws_bytes,
                            uint32_t* status, kda_stream_t stream);

/*
 * kda_package_scan_noalloc: kda_package_scan without a caller workspace, for callers that
 * cannot allocate device memory (for instance a serving loop that has reserved all of HBM for
 * its state pools, or a custom-op interface that provides no allocator). The pages have no
 * counterpart of this call; it is a deployment convenience.
 *   Arguments are those of kda_package_scan minus workspace/ws_bytes; the caller still passes
 *   every input and output buffer.
 *   Scratch: a 64 MiB, 256-byte aligned device array inside the library, reserved on every
 *   GPU that loads the library and held until the process exits. A scan whose
 *   kda_package_scan_workspace(...) exceeds 64 MiB returns KDA_ERR_WORKSPACE (use
 *   kda_package_scan then). The call allocates nothing (no cudaMalloc or cudaFree).
 *   The first call on a device looks up the array's device address with that device
 *   current; make it before any stream capture. The address is kept for the life of the
 *   process: do not call this entry point again after a cudaDeviceReset. All calls share
 *   the one array and it keeps the last call's contents (the scan writes all scratch it
 *   reads, so no clearing is needed); calls that overlap on the GPU race on it. Errors are
 *   reported under this entry point's name.
 */
KDA_API kda_status kda_package_scan_noalloc(int n_seqs, int n_segs,
                                            const int32_t* seq_seg_offsets,
                                            int max_segs_per_seq, int H, int dk, int dv,
                                            const float* M, const float* D,
                                            const float* init_state, float* seg_init,
                                            float* final_state, uint32_t* status,
                                            kda_stream_t stream);

/*
 * kda_segment_replay: replays every segment from its prefix state: the chunked prefill with
 * segments as the sequences and seg_init as their entry states. Writes o for every token and,
 * if seg_final is not NULL, each segment's exit state. workspace as for kda_chunk_prefill,
 * sized by kda_chunk_workspace(dt, n_segs, ...).
 * Source: pegainfer PR #970, each CP member prefills its own context segment.
 */
KDA_API kda_status kda_segment_replay(kda_dtype dt, int n_segs, int total_tokens,
                              const int32_t* seg_offsets, int H, int dk, int dv, int chunk,
                              float scale, const void* q, const void* k, const void* v,
                              const float* g, const float* beta, const float* seg_init,
                              void* o, float* seg_final, void* workspace, size_t ws_bytes,
                              uint32_t* status, kda_stream_t stream);

/*
 * kda_chunk_prepare: the state-independent half of the chunked calls, on its own. Writes into
 * `workspace` the per-(64-token chunk, head) records of n_ranges token ranges
 * [offsets[i], offsets[i+1]) (offsets may be NULL for one range of total_tokens tokens). The
 * records depend only on q, k, v, g, beta, the ranges and scale, so one preparation serves
 * both walks of the segment path over the same segments: kda_segment_package_prepared, and
 * (when q was given) kda_segment_replay_prepared. With q == NULL the records carry only what a
 * package walk reads.
 *   workspace  at least kda_chunk_workspace(dt, n_ranges, total_tokens, H, dk, dv) bytes,
 *              256-byte aligned; the tensor-core shapes only (that query > 0), others return
 *              KDA_ERR_UNSUPPORTED.
 *   beta       16-byte aligned. status: optional device word (KDA_STATUS_TIMEOUT).
 * The pages have no separate counterpart: their context-parallel members prepare a segment
 * once and both publish its package and replay it with the same per-chunk step (pegainfer
 * PR #970, fabric data-plane commit message).
 */
KDA_API kda_status kda_chunk_prepare(kda_dtype dt, int n_ranges, int total_tokens,
                                     const int32_t* offsets, int H, int dk, int dv, int chunk,
                                     float scale, const void* q, const void* k, const void* v,
                                     const float* g, const float* beta, void* workspace,
                                     size_t ws_bytes, uint32_t* status, kda_stream_t stream);

/*
 * kda_segment_package_prepared / kda_segment_replay_prepared: the state walks of
 * kda_segment_package / kda_segment_replay over records that kda_chunk_prepare wrote into
 * `workspace` for the same segments (same seg_offsets, total_tokens, H, dk, dv; the replay
 * also needs records prepared with q and the replay's scale). The workspace is only read.
 * Results equal those of the unprepared calls on the inputs that were prepared.
 */
KDA_API kda_status kda_segment_package_prepared(kda_dtype dt, int n_segs, int total_tokens,
                                                const int32_t* seg_offsets, int H, int dk,
                                                int dv, int chunk, float* M, float* D,
                                                const void* workspace, size_t ws_bytes,
                                                uint32_t* status, kda_stream_t stream);
KDA_API kda_status kda_segment_replay_prepared(kda_dtype dt, int n_segs, int total_tokens,
                                               const int32_t* seg_offsets, int H, int dk,
                                               int dv, int chunk, const float* seg_init,
                                               void* o, float* seg_final,
                                               const void* workspace, size_t ws_bytes,
                                               uint32_t* status, kda_stream_t stream);

/*
 * kda_debug_flag_wait: a diagnostic of the bounded waits. The state walk of
 * kda_segment_replay_prepared over the same records, except that before loading each record
 * the walk waits for that record's 4-byte ready flag to be non-zero, as the walk of a fused
 * prefill does, giving up after limit_ns nanoseconds (1e6 .. 4e9). The flags follow the
 * R = (total_tokens / 64 + n_segs) * H records: record r (chunk slot r / H, head r % H) has
 * its flag in the uint32 at byte R * 147968 + 4 r of the workspace. kda_chunk_prepare leaves
 * them as they were, so the caller sets them.
 * All flags non-zero: the results equal those of kda_segment_replay_prepared, bit for bit.
 * A zero flag: every walk that reaches it gives up, raises KDA_STATUS_TIMEOUT in *status,
 * lets its own copies and tensor-core work finish, frees its tensor memory and returns; its
 * outputs from that record on are not written. The device stays usable. The pages have no
 * counterpart: this exists so that the error path of the waits can be run without a fault.
 */
KDA_API kda_status kda_debug_flag_wait(kda_dtype dt, int n_segs, int total_tokens,
                                       const int32_t* seg_offsets, int H, int dk, int dv,
                                       int chunk, const float* seg_init, void* o,
                                       float* seg_final, const void* workspace,
                                       size_t ws_bytes, uint64_t limit_ns, uint32_t* status,
                                       kda_stream_t stream);

/*
 * kda_decode_step: one token per batch row over a slot-addressed fp32 state pool,
 * updated in place: for row b and head h, S = pool[slot_ids[b], h] becomes its successor
 * and o[b, h] = scale * S_new^T q.
 *   q, k, g [batch, H, dk]; v, o [batch, H, dv]; beta [batch, H].
 *   slot_ids   device int32 [batch]. A negative id marks a padding row: it is skipped and
 *              its o row is written as zeros. An id >= n_slots is skipped the same way and
 *              sets KDA_STATUS_BAD_SLOT in *status. Two rows naming the same slot race.
 *   state_pool [n_slots, H, dk, dv] fp32, read and written in place (16-byte aligned).
 *   batch * H at most 2^30.
 * Source: ATOM PR #2709 (slot-indexed KDA state for decode; read/write state indices) and
 * kern PR #44 (recurrent-state slots per sequence).
 */
KDA_API kda_status kda_decode_step(kda_dtype dt, int batch, int H, int dk, int dv, float scale,
                           const void* q, const void* k, const void* v, const float* g,
                           const float* beta, const int32_t* slot_ids, float* state_pool,
                           int64_t n_slots, void* o, uint32_t* status, kda_stream_t stream);

/* Bits of the `flags` argument of kda_decode_window. */
#define KDA_DECODE_BETA_LOGIT 1u /* beta holds logits; the write strength is 1/(1+exp(-beta)) */

/*
 * kda_decode_window: a verify window of `window` tokens per batch row with a state fork.
 * Row b reads its state from slot read_slots[b] (the read-side index: a forked sequence is
 * read from its source slot, nothing is copied onto the write slot first), runs the window's
 * tokens in order (token j of row b is row b*window + j of the token arrays) and, after token
 * j, stores the current state into slot write_slots[b*window + j]: one snapshot per window
 * column, so that a caller that accepts the first n tokens continues from the slot of column
 * n - 1 (and one that accepts all simply keeps the last). o[b*window + j] = scale * S_j^T q.
 *   q, k, g [batch*window, H, dk]; v, o [batch*window, H, dv]; beta [batch*window, H] (the
 *   write strength, or its logit when flags has KDA_DECODE_BETA_LOGIT).
 *   read_slots  device int32 [batch]. Negative: a padding row (skipped, its window's o rows
 *               written as zeros, nothing stored). >= n_slots: skipped the same way, and
 *               KDA_STATUS_BAD_SLOT is set in *status.
 *   write_slots device int32 [batch, window]. Negative: that column stores nothing.
 *               >= n_slots: that store is skipped and KDA_STATUS_BAD_SLOT is set. A write
 *               slot may equal the row's own read slot (the whole window reads the state
 *               before the first store). The slots named by different rows must be disjoint
 *               (a slot read by one row and written by another races).
 *   state_pool  [n_slots, H, dk, dv] fp32 (16-byte aligned).
 *   window      1 .. 16 (0 is a no-op). window = 1 with write_slots = read_slots is
 *               kda_decode_step with the option of logit write strengths. batch * window * H
 *               at most 2^30.
 * Source: ATOM PR #2709 ("feat(kimi-k3): PP8 prefill for P/D serving - KDA state under PP"),
 * the commits on reading a forked state through a read-side index and on resuming a verify
 * window from its last accepted column, and the sigmoid-gated delta-rule update they name.
 */
KDA_API kda_status kda_decode_window(kda_dtype dt, int batch, int window, int H, int dk, int dv,
                                     float scale, const void* q, const void* k, const void* v,
                                     const float* g, const float* beta, unsigned flags,
                                     const int32_t* read_slots, const int32_t* write_slots,
                                     float* state_pool, int64_t n_slots, void* o,
                                     uint32_t* status, kda_stream_t stream);

/*
 * kda_slot_zero: sets every listed slot of a state pool [n_slots, slot_elems] fp32 to zero.
 *   slot_ids device int32 [n], or NULL for slots 0 .. n-1. Negative ids are skipped; ids
 *            >= n_slots are skipped and set KDA_STATUS_BAD_SLOT.
 *   slot_elems elements per slot (H * dk * dv for a KDA pool), a multiple of 4; the pool
 *            16-byte aligned.
 * Source: kern PR #44 (Runtime::zero_slot: the state slot a new sequence is given starts at
 * zero).
 */
KDA_API kda_status kda_slot_zero(int n, const int32_t* slot_ids, float* state_pool,
                                 int64_t n_slots, int64_t slot_elems, uint32_t* status,
                                 kda_stream_t stream);

/*
 * kda_slot_copy: for i in [0, n) copies slot src[src_ids[i]] into slot dst[dst_ids[i]], where
 * src is [n_src, slot_elems] and dst [n_dst, slot_elems] fp32 (the same pool or two; NULL id
 * arrays mean 0 .. n-1). Taking a checkpoint image of some slots is a copy into a compact
 * buffer (dst_ids NULL); restoring it is the copy back (src_ids NULL). A pair with an id past
 * its pool's end is skipped and sets KDA_STATUS_BAD_SLOT; otherwise a pair with a negative id
 * is skipped. No slot may be both a source and a destination of one call.
 *   slot_elems a multiple of 4; both pools 16-byte aligned.
 * Source: ATOM PR #2709, PAGE-backed KDA state checkpoints (an image is a copy of a
 * sequence's state, made in stream order).
 */
KDA_API kda_status kda_slot_copy(int n, const float* src, const int32_t* src_ids, int64_t n_src,
                                 float* dst, const int32_t* dst_ids, int64_t n_dst,
                                 int64_t slot_elems, uint32_t* status, kda_stream_t stream);

/* Bits of the `flags` argument of kda_short_conv. */
#define KDA_CONV_SILU 1u /* out = y / (1 + exp(-y)) instead of y */

/*
 * kda_short_conv: short causal depthwise convolution over packed sequences, each with a
 * history window of the width - 1 inputs before it kept in a slot pool (the KDA short-conv
 * gather and window update). For sequence s and channel c, with h the window read from slot
 * read_slots[s] (oldest first; zeros for a negative id or read_slots == NULL) and
 * z = [h ; x rows of s]:
 *     y_t = sum_{i=0}^{width-1} weight[c, i] * z[t - (width - 1) + i]
 *     out_t = y_t, or y_t / (1 + exp(-y_t)) with KDA_CONV_SILU,
 * and the last width - 1 entries of z are stored into slot write_slots[s] (nothing for a
 * negative id or write_slots == NULL). An empty sequence passes its window through.
 *   cu_seqlens   device int32 [n_seqs + 1], or NULL for one sequence of total_tokens.
 *   x, out       [total_tokens, channels] (dtype dt), 16-byte aligned; out must not alias x.
 *   weight       [channels, width] fp32 (weight[c, width-1] weighs the current input).
 *   conv_state   [n_slots, width - 1, channels] (dtype dt), 16-byte aligned; may be NULL
 *                when both slot tables are NULL or width = 1.
 *   read_slots, write_slots  device int32 [n_seqs] or NULL. An id >= n_slots is treated as
 *                negative and sets KDA_STATUS_BAD_SLOT. read slot = write slot updates the
 *                window in place; slots named by different sequences must be disjoint.
 *   channels     a positive multiple of 8; width 1 .. 4 (else KDA_ERR_UNSUPPORTED).
 *   status       optional device word (KDA_STATUS_BAD_SLOT, KDA_STATUS_BAD_OFFSETS).
 * Source: kern PR #44, squash message (the short-conv gather and window update among the
 * per-sequence kernels generalised to varlen rows); ATOM PR #2709 (the speculative conv update
 * reads its window through a read-side index). Width and activation are not on the pages.
 */
KDA_API kda_status kda_short_conv(kda_dtype dt, int n_seqs, int total_tokens,
                                  const int32_t* cu_seqlens, int channels, int width,
                                  const void* x, const float* weight, unsigned flags,
                                  const int32_t* read_slots, const int32_t* write_slots,
                                  void* conv_state, int64_t n_slots, void* out,
                                  uint32_t* status, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
