// kda_noalloc.cu -- kda_prefill_noalloc: KDA prefill for callers that cannot
// allocate device memory.
//
// kda_prefill takes its per-(chunk, head) workspace from a stream-ordered
// memory pool.  Some callers cannot let a library allocate: code running under
// an allocator that owns all device memory (a serving engine that carves the
// GPU up front, a framework with a caching allocator that must see every
// byte), callers that forbid driver allocations on their hot path, or
// processes that have already given nearly all HBM away.  This entry point
// serves them: its scratch is a fixed array in this file, created when the
// library's device code is loaded, so a call never allocates or frees
// anything.  The operation and its arguments are those of kda_prefill, but
// the launch plan is the plain one: the preparation kernel, then one
// recurrence launch at the split kda_prefill would pick (kda_set_split and
// kda_set_engine apply).  It never takes kda_prefill's other plans -- the
// one-launch form, the segmented scan, the longest-first order of packed
// sequences or their concurrent split-2 launch -- whose extra buffers would
// not fit the fixed scratch, so its results agree with kda_prefill's within
// the operation's tolerance rather than bit for bit, and its speed on shapes
// that kda_prefill segments (few heads, long sequences) is that of the serial
// chain.
#include <mutex>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

// 48 MiB: enough for B=1, H=6, T=8192 (3,072 chunk-heads, 42.5 MB) and any
// shape with at most 3,640 (chunk, head) packets minus the varlen metadata.
// Every GPU that loads this library holds the array until the process exits.
constexpr int64_t kNoAllocScratchBytes = int64_t(48) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint8_t* g_scratch_ptr[kMaxDevices] = {};   // device address of the array, per device

// Set-up, once per device, with that device current: the array's name is only
// a host-side stand-in, so ask the runtime for its device address.
int scratch_address(uint8_t** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return KDA_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return KDA_OK;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Span {
    uintptr_t lo, hi;
};
Span span(const void* p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Span{lo, lo + static_cast<uintptr_t>(bytes)};
}
bool intersects(Span a, Span b) {
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" int64_t kda_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" int kda_prefill_noalloc(const void* q, const void* k, const void* v, const float* g,
                                   const void* beta, const void* init_state, void* out,
                                   void* final_state, int64_t B, int64_t T, int64_t H,
                                   const int64_t* cu_seqlens, void* stream_ptr) {
    // Shape and scratch requirement (the same sizing rule as kda_prefill).
    constexpr int64_t kMaxElems = int64_t(1) << 56;
    const bool packed = cu_seqlens != nullptr;
    if (B < 1 || T < 0 || H < 1) return KDA_ERR_SHAPE;
    if (H > kMaxElems / (kHeadDim * kHeadDim)) return KDA_ERR_SHAPE;   // before dividing by H
    if (!packed && T > 0 && B > kMaxElems / T) return KDA_ERR_SHAPE;
    const int64_t tokens = packed ? T : B * T;
    if (tokens > kMaxElems / (H * kHeadDim) || B > kMaxElems / (H * kHeadDim * kHeadDim))
        return KDA_ERR_SHAPE;
    SeqGeometry geo = SeqGeometry{};
    geo.n_seqs = B;
    geo.tokens = tokens;
    int64_t meta_bytes = 0;
    if (packed) {
        geo.chunk_ub = (T + (kChunk - 1) * B) / kChunk;
        meta_bytes = 256 + ((8 * (B + 1) + 255) / 256) * 256;
    } else {
        geo.tokens_per_seq = T;
        geo.chunks_per_seq = (T + kChunk - 1) / kChunk;
        geo.chunk_ub = B * geo.chunks_per_seq;
    }
    if (geo.chunk_ub > kNoAllocScratchBytes / (H * static_cast<int64_t>(kPacketBytes)))
        return KDA_ERR_SCRATCH;
    const int64_t need = meta_bytes + geo.chunk_ub * H * static_cast<int64_t>(kPacketBytes);
    if (need > kNoAllocScratchBytes) return KDA_ERR_SCRATCH;

    // Pointers, alignment and overlap: the rules of kda_prefill.
    if (tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL;
    if (!is_aligned(q, 16) || !is_aligned(k, 16) || !is_aligned(v, 16) || !is_aligned(g, 16) ||
        !is_aligned(out, 16) || !is_aligned(beta, 2) ||
        (init_state && !is_aligned(init_state, 16)) ||
        (final_state && !is_aligned(final_state, 16)) ||
        (cu_seqlens && !is_aligned(cu_seqlens, 8)))
        return KDA_ERR_ALIGN;
    const int64_t x_bytes = tokens * H * kHeadDim * 2;
    const int64_t s_bytes = B * H * kHeadDim * kHeadDim * 2;
    const Span sq = span(q, x_bytes), sk = span(k, x_bytes), sv = span(v, x_bytes);
    const Span sg = span(g, tokens * H * kHeadDim * 4), sb = span(beta, tokens * H * 2);
    const Span so = span(out, x_bytes);
    const Span si = span(init_state, init_state ? s_bytes : 0);
    const Span sf = span(final_state, final_state ? s_bytes : 0);
    const Span sc = span(cu_seqlens, cu_seqlens ? 8 * (B + 1) : 0);
    for (Span in : {sq, sk, sv, sg, sb, si, sf, sc})
        if (intersects(so, in)) return KDA_ERR_OVERLAP;
    for (Span in : {sq, sk, sv, sg, sb, sc})
        if (intersects(sf, in)) return KDA_ERR_OVERLAP;
    if (final_state && init_state && final_state != init_state && intersects(sf, si))
        return KDA_ERR_OVERLAP;

    int* status = nullptr;
    int nsplit = 1;
    int rc = device_context(&status, B * H, &nsplit);
    if (rc != KDA_OK) return rc;
    uint8_t* scratch = nullptr;
    rc = scratch_address(&scratch);
    if (rc != KDA_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

    // Nothing in the scratch has to start at zero: the metadata kernel writes
    // the valid flag and the chunk prefix, and the preparation kernel writes
    // every packet the recurrence then reads, all within this call.
    uint8_t* packets = scratch + meta_bytes;
    if (packed) {
        int32_t* valid = reinterpret_cast<int32_t*>(scratch);
        int64_t* cu_chunks = reinterpret_cast<int64_t*>(scratch + 256);
        if (launch_varlen_meta(cu_seqlens, B, tokens, valid, cu_chunks, nullptr, status, stream) !=
            cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        geo.cu_seqlens = cu_seqlens;
        geo.cu_chunks = cu_chunks;
        geo.valid = valid;
    }
    const float scale = 0.08838834764831845f;   // 1 / sqrt(128)
    if (launch_prep(q, k, g, beta, packets, geo, H, scale, status, stream) != cudaSuccess ||
        launch_recurrence(v, out, init_state, final_state, packets, geo, H, nsplit, status,
                          stream) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}
