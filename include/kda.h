/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention prefill library.
 *
 * The operation is the chunkwise KDA forward pass of "FlashKDA column split"
 * (mainlymatmul.com), section 1: for every sequence and head, with the state S
 * a 128 x 128 matrix (rows = value channels, columns = key channels), per
 * token t
 *     S <- S Diag(exp(g_t));  u_t = beta_t (v_t - S khat_t);
 *     S <- S + u_t khat_t^T;  o_t = s S qhat_t,   s = 1/sqrt(128),
 * evaluated 16 tokens at a time through the chunk quantities K^start, Q^start,
 * K^end, D_{0:15}, A^kk = (I + R)^{-1} and A^qk of that section.  q and k are
 * L2-normalised inside the operation, xhat = x / sqrt(sum x^2 + 1e-6)
 * (flashinfer kda_prefill, "Optimized Blackwell prefill subset",
 * use_qk_l2norm_in_kernel).  The log-decay g must lie in [-5, 0] ("K3's KDA
 * precision problem", introduction: the lower bound keeps exp(+-G) of a
 * 16-token chunk inside the FP32/BF16 range).
 *
 * Every pointer argument is a DEVICE pointer on the current CUDA device unless
 * stated otherwise.  The caller owns every buffer; the library keeps no
 * pointer after a call returns.  Calls are asynchronous on `stream` (a
 * cudaStream_t; NULL is the legacy default stream): the host never reads
 * device data and never synchronises.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
#define KDA_OK 0
#define KDA_ERR_NULL (-1)      /* a required pointer is NULL */
#define KDA_ERR_SHAPE (-2)     /* B, T or H out of range, or sizes overflow */
#define KDA_ERR_ALIGN (-3)     /* a pointer is not suitably aligned */
#define KDA_ERR_OVERLAP (-4)   /* an output overlaps an input or another output */
#define KDA_ERR_DEVICE (-5)    /* no CUDA device, or not compute capability 10.3 */
#define KDA_ERR_CUDA (-6)      /* a CUDA call (allocation, launch) failed */
#define KDA_ERR_ARG (-7)       /* an option value is out of range */
#define KDA_ERR_SCRATCH (-8)   /* shape too large for kda_prefill_noalloc's fixed scratch */
#define KDA_ERR_SEQLENS (-9)   /* kda_prefill_host: the host cu_seqlens break their contract */

/* Flags of kda_prefill_ex. */
#define KDA_FLAG_BETA_LOGIT 1u /* beta holds logits; the operation uses sigmoid(beta) */

/* Device-side status bits, reported by kda_device_status(). */
#define KDA_DEV_BAD_SEQLENS 1  /* cu_seqlens broke its contract; out/final_state untouched */
#define KDA_DEV_PIPE_TIMEOUT 2 /* an internal pipeline wait hit its bound; results incomplete */
#define KDA_DEV_BAD_CHECKPOINTS 4 /* a checkpoint had no valid row in checkpoint_cu_starts; skipped */

/*
 * KDA prefill, fixed or packed variable-length layout.
 *
 * Fixed layout (cu_seqlens == NULL): N = B sequences of T tokens each.
 *   q, k, v, out : BF16 [B, T, H, 128], contiguous (head dim innermost)
 *   g            : FP32 [B, T, H, 128], natural-log decay, alpha = exp(g), g in [-5, 0]
 *   beta         : BF16 [B, T, H], beta in [0, 1] (already passed through a sigmoid)
 * Packed layout (cu_seqlens != NULL): tensors are [1, T, H, ...] with T the
 *   total number of tokens, and B is read as the number of sequences N.
 *   cu_seqlens is a device int64 array of N + 1 offsets with cu[0] == 0,
 *   cu[n] <= cu[n+1] and cu[N] == T (flashinfer kda_prefill, "Optimized
 *   Blackwell prefill subset").  Equal neighbours are empty sequences, whose
 *   final state equals their initial state.  The offsets are validated on the
 *   device; a violation leaves out and final_state untouched and sets
 *   KDA_DEV_BAD_SEQLENS (see kda_device_status).
 * init_state  : BF16 [N, H, 128, 128] (value rows x key columns) or NULL for zeros.
 * final_state : BF16 [N, H, 128, 128] or NULL (not written).  final_state may be
 *   the same pointer as init_state (in-place update, as in flashinfer
 *   kda_prefill "State and graph semantics"); any other overlap is refused.
 *
 * Alignment: q, k, v, g, out, init_state and final_state 16 bytes; beta 2
 * bytes; cu_seqlens 8 bytes.  out must not overlap any input.
 * Limits: B >= 1, T >= 0, H >= 1, fewer than 2^31 tokens in total.  With no tokens (T = 0) only final_state is
 * written (a copy of init_state, or zeros) and q, k, v, g, beta and out may be NULL.
 *
 * Scratch: the call takes a workspace of about 13.5 KB per (chunk, head) from
 * a stream-ordered memory pool owned by the library (cudaMallocFromPoolAsync /
 * cudaFreeAsync on `stream`), so it allocates and frees in stream order.
 *
 * Returns KDA_OK or a negative KDA_ERR_* code; on an error nothing is launched.
 */
int kda_prefill(const void* q, const void* k, const void* v, const float* g, const void* beta,
                const void* init_state, void* out, void* final_state, int64_t B, int64_t T,
                int64_t H, const int64_t* cu_seqlens, void* stream);

/*
 * kda_prefill on HOST buffers: the same operation, arguments and layouts as
 * kda_prefill, except that q, k, v, g, beta, init_state, out, final_state and
 * cu_seqlens are HOST pointers (cu_seqlens: host int64 [B + 1] or NULL).  The
 * library copies the inputs to the device, runs the device path and copies
 * out and final_state back, overlapping the copies with the computation: the
 * batch is cut into at most 8 pieces, each a contiguous range of every tensor
 * (token ranges of whole chunks for a single fixed-length sequence, groups of
 * batch rows, or groups of whole packed sequences); while the caller's stream
 * computes one piece, a library stream copies the next one in and another
 * copies the previous piece's outputs back.  A single sequence cut into token
 * ranges carries its state from piece to piece as a BF16 state, as two
 * kda_prefill calls chained through final_state -> init_state would, so its
 * results can differ from one device call by that rounding (within the
 * operation's tolerance); batches cut between sequences give each sequence
 * the results of a device call on its group.
 *
 * Host memory: page-locked buffers (cudaHostAlloc, cudaHostRegister, or a
 * pinned framework tensor) let the copies run asynchronously and overlap;
 * pageable buffers are accepted, but the driver then stages each copy and the
 * overlap is lost (and a CUDA-graph capture of the call fails).
 * Asynchronous on `stream`: the call returns once everything is enqueued; the
 * inputs must stay unchanged and the outputs unread until `stream` has passed
 * the call.  Device memory: images of every tensor, taken from the library's
 * stream-ordered pool for the duration of the call, plus kda_prefill's
 * workspace per piece.  The copy streams are the library's, one pair per
 * device: calls from several host threads enqueue one after another, and
 * while a CUDA-graph capture that contains a kda_prefill_host call is open,
 * those streams belong to it: no other thread may call kda_prefill_host on
 * the device until the capture ends.
 *
 * Returns KDA_OK, kda_prefill's argument codes (shape, NULL, overlap of the
 * host ranges; no alignment rule), KDA_ERR_SEQLENS when the host cu_seqlens
 * break the contract of kda_prefill (nothing is enqueued then), or
 * KDA_ERR_CUDA when a copy or launch could not be enqueued (the copies already
 * enqueued are joined back into `stream` before the call returns).
 */
int kda_prefill_host(const void* q, const void* k, const void* v, const float* g, const void* beta,
                     const void* init_state, void* out, void* final_state, int64_t B, int64_t T,
                     int64_t H, const int64_t* cu_seqlens, void* stream);

/*
 * How many pieces kda_prefill_host cuts a call into: 0 (the default) chooses
 * automatically, 1 .. 8 sets the number (fewer when the batch has fewer
 * chunks, rows or sequences).  Process-wide, for comparing the choices;
 * KDA_ERR_ARG for other values.
 */
int kda_set_host_pieces(int n);

/*
 * Number of kernels (HOST out) that the last kda_prefill, kda_prefill_checkpointed
 * or kda_prefill_host call made on this host thread enqueued (memsets and copies
 * are not counted; after a call that returned an error the count may include
 * the launch that failed).
 */
int kda_last_call_launches(int64_t* n);

/* Human-readable text for a KDA_* status code (static storage). */
const char* kda_error_string(int status);

/*
 * Synchronise `stream`, then read and clear this device's KDA_DEV_* status
 * bits into *status (a HOST pointer).  The bits accumulate over every call on
 * the device since the last read.
 */
int kda_device_status(void* stream, int* status);

/*
 * Number of CTAs that share one (sequence, head) in the recurrence: each owns
 * 128 / nsplit value columns (value columns are independent recurrences,
 * "FlashKDA column split" section 3.1).  nsplit is one of 1, 2, 4, 8, 16, or 0
 * for the automatic choice (the largest split whose grid fits the SM count).
 * Process-wide setting; returns KDA_ERR_ARG for other values.
 */
int kda_set_split(int nsplit);

/*
 * Recurrence engine.  0 (default) and 1: the column-split kernel (warp-level
 * m16n8k16 MMAs, state in registers, `nsplit` CTAs per head).  Engine 0 gives
 * each warp 32 value columns at nsplit 1, 8 columns at nsplit 2, and at nsplit
 * 4, 8 and 16 splits each 8-column group's 128 keys over a pair of warps
 * (their partial sums over keys are added in a fixed order, so results agree
 * with the other variants to rounding, not bit for bit).  Engine 1 gives each
 * warp 8 columns and all 128 keys at every split.  2: the tcgen05
 * kernel (one CTA per (sequence, head); the value rows are the MMA's M = 128;
 * the FP32 state, its BF16 operand copy and every accumulator live in tensor
 * memory, the packets are read by the tensor cores from shared memory; the
 * split setting is ignored).
 * Process-wide; returns KDA_ERR_ARG for other values.
 */
int kda_set_engine(int engine);

/*
 * kda_prefill plus native state checkpoints ("flashinfer kda_prefill", Native
 * checkpoints): the recurrent state before each interval of
 * checkpoint_every_n_tokens tokens (a positive multiple of 16).  Every
 * non-empty sequence n contributes ceil(len_n / interval) rows: its initial
 * state (init_state, or zeros), then the states after one, two, ... intervals
 * that strictly precede its end; empty sequences contribute none.
 *
 *   state_checkpoints     BF16 [checkpoint_rows, H, 128 (value), 128 (key)], DEVICE,
 *                         written; 16-byte aligned; must not overlap any other
 *                         argument.
 *   checkpoint_cu_starts  int64 [N + 1], DEVICE, read: sequence n's rows are
 *                         checkpoint_cu_starts[n] ..; N = B (fixed layout) or the
 *                         number of sequences (packed).  Caller-provided and not
 *                         scanned at launch: a checkpoint whose row falls outside
 *                         [cu_starts[n], cu_starts[n + 1]) or [0, checkpoint_rows)
 *                         is not written and sets KDA_DEV_BAD_CHECKPOINTS.
 *
 * Everything else, including results and errors, is as kda_prefill (a call
 * that takes the segmented scan, kda_set_segments, writes the checkpoints
 * from its last pass: those at segment starts are the segments' BF16
 * incoming states); in addition KDA_ERR_ARG for an interval that is not a
 * positive multiple of 16 or negative checkpoint_rows, KDA_ERR_NULL for NULL
 * checkpoint pointers.
 * Under engine 2 (kda_set_engine) such calls run on the column-split kernels.
 */
int kda_prefill_checkpointed(const void* q, const void* k, const void* v, const float* g,
                             const void* beta, const void* init_state, void* out,
                             void* final_state, int64_t B, int64_t T, int64_t H,
                             const int64_t* cu_seqlens, int64_t checkpoint_every_n_tokens,
                             void* state_checkpoints, const int64_t* checkpoint_cu_starts,
                             int64_t checkpoint_rows, void* stream);

/*
 * kda_prefill with options: the same operation, arguments, layouts, results
 * and errors, plus
 *   flags  0, or KDA_FLAG_BETA_LOGIT: beta (BF16 [B, T, H]) holds logits x and
 *          the operation uses beta = sigmoid(x) = 1 / (1 + exp(-x)), formed in
 *          FP32 inside the chunk preparation ("flashinfer kda_prefill",
 *          "Optimized Blackwell prefill subset": beta_is_logit=True).  Other
 *          bits: KDA_ERR_ARG.
 *   checkpoint_every_n_tokens, state_checkpoints, checkpoint_cu_starts,
 *   checkpoint_rows: native checkpoints exactly as kda_prefill_checkpointed;
 *          state_checkpoints NULL for none (the other three are then ignored).
 */
int kda_prefill_ex(const void* q, const void* k, const void* v, const float* g, const void* beta,
                   const void* init_state, void* out, void* final_state, int64_t B, int64_t T,
                   int64_t H, const int64_t* cu_seqlens, uint32_t flags,
                   int64_t checkpoint_every_n_tokens, void* state_checkpoints,
                   const int64_t* checkpoint_cu_starts, int64_t checkpoint_rows, void* stream);

/*
 * Whether kda_prefill may run preparation and recurrence as one cooperative
 * launch (1, the default) or always as two kernels (0).  One launch is used
 * under engine 0 in two forms, each packet behind a ready flag in the
 * workspace: (a) fixed-length batches (cu_seqlens NULL) with few heads, whose
 * recurrence takes a split of 8 or 16 and leaves at least 16 SMs free: those
 * SMs prepare packets while the recurrence consumes them; (b) many heads, one
 * recurrence CTA per (sequence, head) and 3 N H <= 2 x the SM count, at
 * least 64 chunks per sequence (packed: on average), never with checkpoints:
 * one CTA per SM, the first N * H of them each run a head's recurrence and
 * prepare packets on two warp pairs, the others prepare on eight.  The
 * preparation walks the chunks in the order the recurrences consume them:
 * chunk index first across all heads (fixed layout), or, for a packed batch,
 * by each chunk's position relative to its sequence's length (a small kernel
 * ranks the chunks on the device after the offsets are checked), so that
 * every sequence's recurrence gets its packets at the pace its length needs.
 * The results are bit for bit those of the two-kernel path.
 * Process-wide; returns KDA_ERR_ARG for other values.
 */
int kda_set_fusion(int on);

/*
 * Whether kda_prefill would run a call of this shape as one launch on the
 * current device under the current settings (HOST out: 1 or 0).  Errors as
 * kda_prefill's shape checks, or KDA_ERR_DEVICE / KDA_ERR_CUDA without a
 * usable device.
 */
int kda_plan_fused(int64_t B, int64_t T, int64_t H, int packed, int* fused);

/*
 * For a packed call of n_seqs sequences (T tokens in all) and H heads: how
 * many of its longest sequences kda_prefill runs at split 2 in a second,
 * concurrent recurrence launch on a library-owned stream (HOST out; 0 when
 * the call uses a single recurrence launch or the many-head one-launch form).
 * That happens under engine 0 with the automatic split when the
 * one-CTA-per-head grid leaves SMs free and n_seqs <= 1024; the results are
 * bitwise those of split 1.
 */
int kda_plan_long_split(int64_t n_seqs, int64_t T, int64_t H, int64_t* k);

/*
 * Whether kda_prefill may use the segmented scan over chunks (1, the default)
 * or always runs each (sequence, head) as one serial chain of chunk steps (0).
 * The chunkwise state update is affine in the incoming state, so over a run
 * of chunks it is S -> S F + Z (the chunk equations of "FlashKDA column
 * split", section 1: S_{c+1} = S_c D_{0:15} + U_c K^end_c with
 * U_c = (V_c - S_c K^start_c) B_c (A^kk_c)^T affine in S_c).  When there
 * are too few (sequence, head) chains to fill the GPU (engine 0, automatic
 * split; fixed or packed layout; with or without checkpoints, which the last
 * pass writes), each sequence is cut into
 * segments: one launch forms every segment's F and Z, a short chain over the
 * segments forms each segment's incoming state, and one launch reruns every
 * segment from its incoming state and writes O.  The results agree with the
 * serial chain to rounding (the incoming states are rounded to BF16), not bit
 * for bit.  seg_chunks 0 lets a cost estimate decide whether and how to cut;
 * seg_chunks > 0 cuts every eligible call into segments of that many chunks
 * (for tests).  Process-wide; returns KDA_ERR_ARG for on not 0 or 1 or
 * seg_chunks negative or above 2^26.
 */
int kda_set_segments(int on, int64_t seg_chunks);

/*
 * Segments kda_prefill would use for a call of this shape on the current
 * device under the current settings (HOST out; 0: no segmented scan): per
 * sequence for the fixed layout; for the packed layout a bound on all
 * segments (the cut itself is made on the device from cu_seqlens).  Errors as
 * kda_plan_fused.
 */
int kda_plan_segments(int64_t B, int64_t T, int64_t H, int packed, int64_t* segs);

/* The split the automatic rule picks on the current device for N*H units (HOST out). */
int kda_auto_split(int64_t n_seqs, int64_t H, int* nsplit);

/*
 * Bytes of scratch kda_prefill takes for a given shape at most (HOST out);
 * `packed` is nonzero for the packed layout.  The ready flags of a fused
 * launch (kda_set_fusion) are counted whether or not a fixed-length call
 * fuses, and for a packed call, with its chunk order (4 bytes a chunk), when
 * the current device (a 152-SM one when there is none) would run it as the
 * many-head one-launch form; the segmented scan's three state buffers
 * (kda_set_segments) when that device would use it.
 */
int kda_workspace_bytes(int64_t B, int64_t T, int64_t H, int packed, int64_t* bytes);

/*
 * Test hook: run only the chunk preparation and write the per-(chunk, head)
 * packets into `packets` (device, capacity `packets_bytes`).  Packet
 * (chunk, head) starts at byte (chunk * H + head) * kda_packet_bytes(), with
 * chunks numbered sequence by sequence.  The packet layout is documented in
 * kda_common.cuh.  Arguments as for kda_prefill.
 */
int kda_prep_only(const void* q, const void* k, const float* g, const void* beta, int64_t B,
                  int64_t T, int64_t H, const int64_t* cu_seqlens, void* packets,
                  int64_t packets_bytes, void* stream);

/* Size in bytes of one (chunk, head) packet. */
int64_t kda_packet_bytes(void);

/*
 * Per-kernel timing for benchmarks.  kda_profile_begin(max_calls) creates
 * 5 * max_calls CUDA events on the current device; each of the next
 * max_calls kda_prefill calls then records, on its own stream, one event
 * before its preparation kernels, one after them, one after the transition
 * pass and one after the segment chain of a segmented scan (see
 * kda_set_segments; recorded right after the second otherwise), and one after
 * the recurrence.  When a call runs as one launch (see kda_set_fusion), the
 * first interval holds only the reset of the ready flags and the last the
 * fused kernel.  kda_profile_end synchronises those events, writes the summed
 * preparation time and recurrence time (the last three intervals) in
 * milliseconds and the number of calls timed (HOST pointers), and destroys
 * the events; kda_profile_end_detail does the same but writes the four
 * summed intervals to intervals_ms[0..3].  Process-wide; begin while active
 * returns KDA_ERR_ARG.
 */
int kda_profile_begin(int max_calls);
int kda_profile_end(double* prep_ms, double* recurrence_ms, int* calls);
int kda_profile_end_detail(double* intervals_ms, int* calls);

/*
 * Measurement hook: nanoseconds per step of the shortest dependent chain of
 * one chunk step on the current device (HOST out), for the critical-path
 * bound of a serial walk over the chunks ("FlashKDA column split" section 1:
 * chunk c + 1 needs chunk c's state).  One warp runs, 4,096 times, U^T = K'
 * S^T over 128 keys (two interleaved MMA accumulators and an add), the FP16
 * conversion and transpose of U^T, S^T <- D S^T + (K^end)^T U^T and the BF16
 * conversion and transpose of the new state, with operands in registers.
 * Synchronises the device; not for use on a hot path.  KDA_ERR_DEVICE
 * without a compute capability 10.3 device, KDA_ERR_CUDA on a CUDA error.
 */
int kda_chain_step_ns(double* ns);

/*
 * kda_prefill without any allocation.  The pages describe no such entry
 * point; it exists for callers that cannot let a library allocate device
 * memory: code running under an allocator that owns all of the GPU's memory
 * (a serving engine that carves HBM up front, a framework whose caching
 * allocator must account for every byte), callers that forbid driver
 * allocations on their hot path, or processes that have already handed out
 * nearly all HBM.
 *
 * Arguments, alignment and overlap rules and error codes are those of
 * kda_prefill; the caller still passes every input and output.  It runs the
 * plain plan -- the preparation kernel, then one recurrence launch at the
 * split kda_prefill would pick (kda_set_split and kda_set_engine apply) --
 * and never the one-launch form, the segmented scan or the longest-first
 * scheduling of packed sequences, so its results agree with kda_prefill's
 * within the operation's tolerance, not bit for bit.  The
 * scratch kda_prefill would take from its pool lives instead in one fixed
 * device array of kda_noalloc_scratch_bytes() bytes (48 MiB) inside this
 * library, which every GPU that loads the library holds until the process
 * exits.  A shape whose scratch does not fit -- about 13.5 KB per (chunk of
 * 16 tokens, head), plus (N + 1) * 8 + 512 bytes for packed input -- is
 * refused with KDA_ERR_SCRATCH before anything is launched.  No call
 * allocates or frees device or host memory.
 *
 * The first call on a device, with that device current, looks up the
 * array's device address (cudaGetSymbolAddress) once; make that first call
 * before any stream capture.  Every call on a device shares the one array
 * and leaves its contents behind; nothing in it has to start at zero.  Calls
 * whose kernels overlap on the GPU (on different streams, or from different
 * host threads) race on that array and corrupt each other's results: order
 * them on one stream, or with events.
 */
int kda_prefill_noalloc(const void* q, const void* k, const void* v, const float* g,
                        const void* beta, const void* init_state, void* out, void* final_state,
                        int64_t B, int64_t T, int64_t H, const int64_t* cu_seqlens, void* stream);

/* Size in bytes of kda_prefill_noalloc's fixed scratch array. */
int64_t kda_noalloc_scratch_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
