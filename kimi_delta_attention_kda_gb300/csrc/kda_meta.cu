// kda_meta.cu -- packed variable-length metadata for KDA prefill (sm_103a).
//
// flashinfer kda_prefill ("Optimized Blackwell prefill subset" and "Packed
// scheduling") fixes the contract of cu_seqlens: int64, cu[0] == 0,
// non-decreasing, cu[N] == total tokens, equal neighbours meaning an empty
// sequence, and no host read of the device offsets.  This kernel checks that
// contract on the device and turns the offsets into a compact per-sequence
// chunk prefix cu_chunks[n] = sum_{m<n} ceil(len_m / 16), which the
// preparation kernel binary-searches and the recurrence indexes directly.
// On a violation it clears `valid` (every later kernel then returns without
// touching its outputs) and records kDevBadSeqlens in the status word.
// For up to kMaxOrdered sequences it can also write the longest-first order
// of the sequences (by chunk count, ties by index; "flashinfer kda_prefill",
// Packed scheduling, seq_order), which the recurrence uses to start the
// longest sequences in its first wave.
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kMetaThreads = 1024;

__global__ void __launch_bounds__(kMetaThreads)
varlen_meta_kernel(const int64_t* cu, int64_t N, int64_t total, int32_t* valid,
                   int64_t* cu_chunks, int32_t* order, int* status) {
    __shared__ int64_t warp_sums[kMetaThreads / 32];
    __shared__ int64_t counts[kMaxOrdered];
    __shared__ int64_t carry;
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        bad = (cu[0] != 0) || (cu[N] != total);
        cu_chunks[0] = 0;
    }
    __syncthreads();
    for (int64_t base = 0; base < N; base += kMetaThreads) {
        const int64_t n = base + tid;
        int64_t cnt = 0;
        if (n < N) {
            const int64_t len = cu[n + 1] - cu[n];
            if (len < 0) bad = 1;
            cnt = len > 0 ? (len + kChunk - 1) / kChunk : 0;
            if (order && n < kMaxOrdered) counts[n] = cnt;
        }
        // Inclusive scan: within the warp, then over warp totals.
        int64_t x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int64_t w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int64_t incl = x + (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
        if (n < N) cu_chunks[n + 1] = incl;
        __syncthreads();
        if (tid == kMetaThreads - 1) carry = incl;
        __syncthreads();
    }
    if (tid == 0) {
        *valid = bad ? 0 : 1;
        if (bad) atomicOr(status, kDevBadSeqlens);
    }
    if (order && N <= kMaxOrdered) {
        // Rank of sequence n: sequences with more chunks, or as many and a
        // smaller index, come first.
        __syncthreads();
        for (int64_t n = tid; n < N; n += kMetaThreads) {
            const int64_t cn = counts[n];
            int32_t rank = 0;
            for (int64_t m = 0; m < N; ++m) {
                const int64_t cm = counts[m];
                rank += (cm > cn || (cm == cn && m < n)) ? 1 : 0;
            }
            order[rank] = static_cast<int32_t>(n);
        }
    }
}

// The chunks of a packed batch in the order of their position relative to
// their sequence's length: chunk i of a sequence of n chunks has the key
// (2i + 1) / 2n, ties going to the lower sequence index.  order[r] is the
// global index of the chunk of rank r.  A preparation that produces the
// packets in this order brings every sequence along at the pace its length
// needs, so the longest sequence's recurrence gets its packets about as fast
// as it consumes them while the short ones are still being prepared.  The
// rank of a chunk is the number of chunks with a smaller key (or an equal key
// and a lower sequence index), counted per sequence in closed form: for
// sequence m with n_m chunks, chunk i' has a smaller key than chunk i of
// sequence n iff (2i' + 1) n < X with X = (2i + 1) n_m, i.e. for
// i' < ceil(X / n) / 2, and an equal key iff n divides X with an odd
// quotient.  The ranks of all chunks form a permutation of 0 .. total - 1.
//
// Block 0 also picks which sequences' recurrences run without preparing
// pairs beside them (alone[n] = 1): the k longest, with k minimising the
// larger of the preparation's time on the pairs that remain and the longest
// chain, a recurrence alone on its SM taking kAloneStepUs per chunk and one
// beside two pairs kSharedStepUs (the preparation rate and both step times
// measured on GB300 in the many-head one-launch form of a packed 8-sequence,
// 12-head batch).  Equal lengths give k = 0.
constexpr int kAloneMaxSeqs = 256;
// (FP32: an estimate, and FP64 arithmetic is slow on this GPU.)
constexpr float kPairItemsPerUs = 0.108f;
constexpr float kAloneStepUs = 1.02f;
constexpr float kSharedStepUs = 1.12f;

constexpr int64_t kOrderSmemSeqs = 1024;   // offsets staged in shared memory up to this many

__global__ void chunk_order_kernel(const int64_t* cu_chunks_g, const int32_t* valid, int64_t N,
                                   int64_t chunk_ub, int32_t* order, int32_t* alone, int64_t H,
                                   int64_t grid) {
    // The chunk offsets are read many times by every thread: stage them in
    // shared memory once per block (short chains of dependent global loads
    // were most of this kernel's time).
    __shared__ int64_t cu_s[kOrderSmemSeqs + 1];
    __shared__ int32_t valid_s;
    const bool staged = N <= kOrderSmemSeqs;
    if (staged)
        for (int64_t n = threadIdx.x; n <= N; n += blockDim.x) cu_s[n] = cu_chunks_g[n];
    if (threadIdx.x == 0) valid_s = *valid;
    __syncthreads();
    const int64_t* cu_chunks = staged ? cu_s : cu_chunks_g;
    if (blockIdx.x == 0 && alone) {
        __shared__ int64_t sorted[kAloneMaxSeqs];
        __shared__ int64_t best_k;
        const bool ok = valid_s && N <= kAloneMaxSeqs;
        int64_t rank[kAloneMaxSeqs / 256];
        for (int64_t n = threadIdx.x, j = 0; ok && n < N; n += blockDim.x, ++j) {
            const int64_t cn = cu_chunks[n + 1] - cu_chunks[n];
            int64_t r = 0;
            for (int64_t m = 0; m < N; ++m) {
                const int64_t cm = cu_chunks[m + 1] - cu_chunks[m];
                r += (cm > cn || (cm == cn && m < n)) ? 1 : 0;
            }
            rank[j] = r;
            sorted[r] = cn;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            best_k = 0;
            if (ok) {
                const float items = static_cast<float>(cu_chunks[N]) * static_cast<float>(H);
                const int64_t units = N * H;
                const float pairs0 = 2.f * static_cast<float>(units) + 8.f * static_cast<float>(grid - units);
                float best = 0.f;
                for (int64_t k = 0; k < N; ++k) {
                    const float pairs = pairs0 - 2.f * static_cast<float>(H * k);
                    if (pairs <= 0.f) break;
                    float t = items / (kPairItemsPerUs * pairs);
                    const float alone_t = static_cast<float>(sorted[0]) * kAloneStepUs;
                    const float shared_t = static_cast<float>(sorted[k]) * kSharedStepUs;
                    if (k > 0 && alone_t > t) t = alone_t;
                    if (shared_t > t) t = shared_t;
                    if (k == 0 || t < best) {
                        best = t;
                        best_k = k;
                    }
                }
            }
        }
        __syncthreads();
        for (int64_t n = threadIdx.x, j = 0; n < N; n += blockDim.x, ++j)
            alone[n] = ok && rank[j] < best_k ? 1 : 0;
    }
    const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= chunk_ub || !valid_s || c >= cu_chunks[N]) return;
    // The sequence of chunk c: the largest n with cu_chunks[n] <= c.
    int64_t lo = 0, hi = N;
    while (hi - lo > 1) {
        const int64_t mid = (lo + hi) >> 1;
        if (cu_chunks[mid] <= c)
            lo = mid;
        else
            hi = mid;
    }
    const int64_t n = lo;
    const int64_t nn = cu_chunks[n + 1] - cu_chunks[n];   // >= 1: chunk c is in it
    const int64_t i = c - cu_chunks[n];
    int64_t rank = i;
    for (int64_t m = 0; m < N; ++m) {
        if (m == n) continue;
        const int64_t nm = cu_chunks[m + 1] - cu_chunks[m];
        if (nm <= 0) continue;
        const int64_t X = (2 * i + 1) * nm;
        // q = floor(X / n), r = X mod n: in 32 bits when X fits (every batch
        // of fewer than about 46,000 chunks per sequence), exact either way.
        int64_t q, r;
        if (X < (int64_t(1) << 32)) {
            const uint32_t x32 = static_cast<uint32_t>(X), n32 = static_cast<uint32_t>(nn);
            const uint32_t q32 = x32 / n32;
            q = q32;
            r = x32 - q32 * n32;
        } else {
            q = X / nn;
            r = X - q * nn;
        }
        // Chunks of m with (2 i' + 1) n < (2 i + 1) nm: i' < ceil(X / n) / 2.
        int64_t less = (q + (r != 0 ? 1 : 0)) / 2;
        if (less > nm) less = nm;
        rank += less;
        if (m < n && r == 0 && (q & 1)) rank += 1;
    }
    order[rank] = static_cast<int32_t>(c);
}

// Group j of a packed batch (sequences first[j] .. first[j + 1] - 1) gets its
// offsets rebased to start at zero, at out[first[j] + j ..
// first[j + 1] + j]: a packed batch of its own over the group's tokens.
__global__ void rebase_offsets_kernel(const int64_t* cu, SeqGroups groups, int64_t* out) {
    const int j = blockIdx.x;
    const int64_t s0 = groups.first[j], s1 = groups.first[j + 1];
    const int64_t base = cu[s0];
    for (int64_t i = threadIdx.x; i <= s1 - s0; i += blockDim.x) out[s0 + j + i] = cu[s0 + i] - base;
}

}  // namespace

cudaError_t launch_rebase_offsets(const int64_t* cu_seqlens, const SeqGroups& groups, int64_t* out,
                                  cudaStream_t stream) {
    if (groups.n < 1 || groups.n > kMaxSeqGroups) return cudaErrorInvalidValue;
    rebase_offsets_kernel<<<groups.n, 256, 0, stream>>>(cu_seqlens, groups, out);
    return cudaGetLastError();
}

cudaError_t launch_chunk_order(const int64_t* cu_chunks, const int32_t* valid, int64_t n_seqs,
                               int64_t chunk_ub, int32_t* order, int32_t* alone, int64_t H,
                               int64_t grid, cudaStream_t stream) {
    if (chunk_ub <= 0) return cudaSuccess;
    if (chunk_ub >= (int64_t(1) << 31) || n_seqs < 1 || H < 1 || grid < 1)
        return cudaErrorInvalidValue;
    const int64_t blocks = (chunk_ub + 255) / 256;
    chunk_order_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        cu_chunks, valid, n_seqs, chunk_ub, order, alone, H, grid);
    return cudaGetLastError();
}

cudaError_t launch_varlen_meta(const int64_t* cu_seqlens, int64_t n_seqs, int64_t total_tokens,
                               int32_t* valid, int64_t* cu_chunks, int32_t* order, int* status,
                               cudaStream_t stream) {
    if (n_seqs > kMaxOrdered) order = nullptr;
    varlen_meta_kernel<<<1, kMetaThreads, 0, stream>>>(cu_seqlens, n_seqs, total_tokens, valid,
                                                      cu_chunks, order, status);
    return cudaGetLastError();
}

}  // namespace kda
