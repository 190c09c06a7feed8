// kda_launch.h -- host-side launch interface between the C ABI (kda_api.cu)
// and the kernel translation units.  Internal; not part of the public header.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

struct SeqGeometry {
    // Fixed layout: n_seqs sequences of tokens_per_seq tokens each.
    // Packed layout: cu_seqlens (device, n_seqs + 1) and metadata written by
    // the varlen metadata kernel (cu_chunks, valid flag).
    int64_t n_seqs;
    int64_t tokens;           // total tokens across all sequences
    int64_t tokens_per_seq;   // fixed layout only
    int64_t chunks_per_seq;   // fixed layout only
    int64_t chunk_ub;         // upper bound on the total number of chunks
    const int64_t* cu_seqlens;   // packed only (device)
    const int64_t* cu_chunks;    // packed only (device, n_seqs + 1)
    const int32_t* valid;        // packed only (device)
    // Packed only, may be null: the recurrence's sequence slots in
    // longest-first order (slot i runs sequence order[i]), from the metadata
    // kernel, so that the longest sequences start in the first wave.
    const int32_t* order;
    // Recurrence CTAs whose sequence slot is below first_slot return at once
    // (those sequences run in a second, concurrent launch).
    int64_t first_slot;
    // Fixed layout only, 0 for none: each sequence is cut into segments of
    // seg_chunks chunks (the last one shorter), and "sequence" n of the
    // recurrence is segment n % segs_per_seq of sequence n / segs_per_seq.
    int64_t seg_chunks;
    int64_t segs_per_seq;
    // Packed layout cut into segments (the segment table is cu_seqlens /
    // cu_chunks): the sequence of each segment and each sequence's first
    // chunk, for per-sequence checkpoint numbering.  Null otherwise.
    const int64_t* seg_seq;
    const int64_t* seq_chunks;
    int* status;                 // device status word (set by the launchers)
};

// Validates cu_seqlens, writes cu_chunks and, when `order` is not null
// (n_seqs <= kMaxOrdered), the longest-first order of the sequences.
constexpr int64_t kMaxOrdered = 1024;
cudaError_t launch_varlen_meta(const int64_t* cu_seqlens, int64_t n_seqs, int64_t total_tokens,
                               int32_t* valid, int64_t* cu_chunks, int32_t* order, int* status,
                               cudaStream_t stream);

// order[r] = the chunk of rank r when the chunks of a packed batch are ranked
// by their position relative to their sequence's length, and alone[n] = 1 for
// the sequences whose recurrences run without preparing pairs on their SMs in
// the many-head one-launch form of H heads on `grid` SMs (kda_meta.cu).
cudaError_t launch_chunk_order(const int64_t* cu_chunks, const int32_t* valid, int64_t n_seqs,
                               int64_t chunk_ub, int32_t* order, int32_t* alone, int64_t H,
                               int64_t grid, cudaStream_t stream);

// Consecutive groups of the sequences of a packed batch: group j is
// sequences first[j] .. first[j + 1] - 1 (first[0] = 0, first[n] = N).
constexpr int kMaxSeqGroups = 8;
struct SeqGroups {
    int64_t first[kMaxSeqGroups + 1];
    int n;
};
// Each group's offsets rebased to zero: out[first[j] + j + i] =
// cu_seqlens[first[j] + i] - cu_seqlens[first[j]] for i = 0 .. its sequence count
// (N + n entries in all).
cudaError_t launch_rebase_offsets(const int64_t* cu_seqlens, const SeqGroups& groups, int64_t* out,
                                  cudaStream_t stream);

// beta_logit: the beta tensor holds logits and the preparation applies
// beta = sigmoid(logit) ("flashinfer kda_prefill", beta_is_logit).
cudaError_t launch_prep(const void* q, const void* k, const float* g, const void* beta,
                        uint8_t* packets, const SeqGeometry& geo, int64_t H, float scale,
                        int* status, cudaStream_t stream, bool beta_logit = false);

// Native state checkpoints: the state before every `every`-chunk interval of
// each sequence (its initial state first), in rows cu_starts[n] ..
// cu_starts[n + 1] - 1 of states [rows, H, 128, 128] (BF16, DEVICE).
struct Checkpoints {
    __nv_bfloat16* states;       // null: no checkpoints
    const int64_t* cu_starts;    // [N + 1], DEVICE
    int64_t every;               // chunks per interval (>= 1)
    int64_t rows;                // rows of `states`
};

// Recurrence variants: `nsplit` CTAs share one (sequence, head); each owns
// 128 / nsplit value columns.  `ck` may be null (no checkpoints).
cudaError_t launch_recurrence(const void* v, void* out, const void* init_state,
                              void* final_state, const uint8_t* packets,
                              const SeqGeometry& geo, int64_t H, int nsplit, int* status,
                              cudaStream_t stream, const Checkpoints* ck = nullptr);

// First pass of the segmented scan (geo: a fixed layout with seg_chunks set):
// for every segment and head, the BF16 state the segment's chunks lead to
// from a zero state (zero_start_states) and from the identity with V taken as
// zero (transitions: the segment's state map S -> S F), each [segments][H] of
// 32 KB: F in fmap_frag_off order, the zero-start state in zmap_frag_off
// order (kda_segmap.cuh), the layouts the segment chain's MMA loads.
cudaError_t launch_transition(const void* v, const uint8_t* packets, const SeqGeometry& geo,
                              int64_t H, void* zero_start_states, void* transitions, int* status,
                              cudaStream_t stream);

// Second pass: per sequence and head, the segments' incoming states in order,
// S_0 = init (zero when null), S_{j+1} = S_j F_j + Z_j, written as BF16 to
// starts[segment * H + h] for the sequence's segments and the last one to
// final_state (when not null).  Fixed layout (seg_begin null): sequence n's
// segments are n segs .. n segs + segs - 1.  Packed layout: seg_begin[n] ..
// seg_begin[n + 1] - 1 from launch_segment_meta, `segs` bounds the total and
// `valid` is the metadata's verdict.
cudaError_t launch_segment_scan(const void* init_state, void* final_state, const void* transitions,
                                const void* zero_start_states, void* starts, int64_t n_seqs,
                                int64_t segs, const int64_t* seg_begin, const int32_t* valid,
                                int64_t H, int* status, cudaStream_t stream);

// Two-level chain (fixed layout, segs segments per sequence in groups of
// group_segs): first the composition inside each group — prefix maps
// (prefix_f, prefix_z: [segments][H][128][128] rows, entry s = the map of
// the group's segments up to s) and the group maps (group_f, group_z:
// [groups][H] in the fragment orders of transitions and zero_start_states);
// then launch_segment_scan over the group maps gives
// each group's incoming state; then launch_segment_apply forms every
// segment's incoming state from its group's and the prefix before it.
cudaError_t launch_segment_compose(const void* transitions, const void* zero_start_states,
                                   void* prefix_f, void* prefix_z, void* group_f, void* group_z,
                                   int64_t n_seqs, int64_t segs, int64_t group_segs,
                                   int64_t groups, int64_t H, int* status, cudaStream_t stream);
cudaError_t launch_segment_apply(const void* group_starts, const void* prefix_f, const void* prefix_z,
                                 void* starts, int64_t n_seqs, int64_t segs, int64_t group_segs,
                                 int64_t groups, int64_t H, int* status, cudaStream_t stream);

// Segments of a packed batch of n_seqs sequences (after launch_varlen_meta):
// ceil(chunks / seg_chunks_len) per sequence, at most s_ub in all; writes
// seg_begin [n_seqs + 1], per segment its first chunk and first token
// ([s_ub + 1] each, padded with the batch's end) and its sequence
// (seg_seq [s_ub], 0 for padding).
cudaError_t launch_segment_meta(const int64_t* cu_seqlens, const int64_t* cu_chunks, int32_t* valid,
                                int64_t n_seqs, int64_t seg_chunks_len, int64_t s_ub,
                                int64_t* seg_begin, int64_t* seg_chunks, int64_t* seg_tokens,
                                int64_t* seg_seq, int* status, cudaStream_t stream);

// The tcgen05 recurrence: one CTA per (sequence, head).
cudaError_t launch_recurrence_tc(const void* v, void* out, const void* init_state,
                                 void* final_state, const uint8_t* packets, const SeqGeometry& geo,
                                 int64_t H, int* status, cudaStream_t stream);

// Preparation and the key-split recurrence (nsplit 8 or 16) as one
// cooperative launch over all SMs, for fixed-length batches whose recurrence
// grid leaves SMs free.  `ready` holds chunk_ub * H flags that must be zero
// when the kernel starts; the packets go through `packets` as in the
// two-kernel path.
bool fused_supported(int64_t n_seqs, int64_t H, int nsplit, int sms);
cudaError_t launch_fused(const void* q, const void* k, const float* g, const void* beta,
                         const void* v, void* out, const void* init_state, void* final_state,
                         uint8_t* packets, uint32_t* ready, const SeqGeometry& geo, int64_t H,
                         int nsplit, float scale, int* status, cudaStream_t stream,
                         const Checkpoints* ck = nullptr, bool beta_logit = false);

// Preparation and the wide one-CTA-per-head recurrence as one cooperative
// launch of one 16-warp CTA per SM, for fixed-length batches of at most one
// (sequence, head) unit per SM (kda_fused.cu).  `ready` as for launch_fused,
// followed by one more zeroed word (the preparation's item counter).
bool fused_heads_supported(int64_t n_seqs, int64_t H, int sms);
cudaError_t launch_fused_heads(const void* q, const void* k, const float* g, const void* beta,
                               const void* v, void* out, const void* init_state, void* final_state,
                               uint8_t* packets, uint32_t* ready, const int32_t* chunk_order,
                               const int32_t* alone, const SeqGeometry& geo, int64_t H,
                               float scale, int* status, cudaStream_t stream, bool beta_logit);

// Tensor map of v viewed as a 2-D BF16 array [tokens][H * 128], boxes of
// 16 tokens x `cols` value columns.
cudaError_t encode_v_map(CUtensorMap* map, const void* v, int64_t tokens, int64_t H, int cols);
cudaError_t encode_v_map_sw128(CUtensorMap* map, const void* v, int64_t tokens, int64_t H);
cudaError_t encode_state_map(CUtensorMap* map, const void* base, int64_t rows, int box_rows);

// Recurrence engine: 0 automatic, 1 column-split warp MMA, 2 tcgen05.
int recurrence_engine();

// Per-device status word and the split kda_prefill picks for `units`
// (sequence x head) recurrences, for entry points outside kda_api.cu.
int device_context(int** status, int64_t units, int* nsplit);

}  // namespace kda
