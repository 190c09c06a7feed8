// kda_api.cu -- the C ABI of the KDA prefill library (declared in include/kda.h).
//
// Host-side only: argument validation, workspace sizing, the choice of
// recurrence split, and the launches (varlen metadata -> chunk preparation ->
// recurrence) on the caller's stream.  No host <-> device synchronisation and
// no host reads of device data happen here (flashinfer kda_prefill, "Optimized
// Blackwell prefill subset": cu_seqlens is never inspected on the host).
#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

__device__ int g_device_status;   // KDA_DEV_* bits, one word per device

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool init = false;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    int* status = nullptr;            // device address of g_device_status
    cudaMemPool_t pool = nullptr;     // library-owned stream-ordered pool
    // Second stream and fork/join events for a concurrent second recurrence
    // launch (long packed sequences at split 2); created on first use.
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    // Copy streams and events of kda_prefill_host (host -> device, device ->
    // host); created on first use.
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t h_start = nullptr, h_in = nullptr, h_done = nullptr, h_out = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
// Kernels enqueued by the current (or last) entry-point call of this host thread.
thread_local int64_t t_launches = 0;
int g_split_override = 0;
int g_engine = 0;
int g_fusion = 1;
int g_segments = 1;
int64_t g_seg_chunks = 0;   // > 0: forced segment length (kda_set_segments)
int g_host_pieces = 0;      // > 0: kda_prefill_host cuts into at most this many pieces

// Optional per-kernel timing: when active, each kda_prefill call records three
// events on its stream (before the preparation kernels, between preparation
// and recurrence, after the recurrence).  Events are created up front by
// kda_profile_begin so that the calls themselves only record.
struct Profile {
    bool active = false;
    int max_calls = 0;
    int calls = 0;
    cudaEvent_t* ev = nullptr;   // 3 per call
};
Profile g_prof;

// Events per call: 0 before the preparation, 1 after it, 2 after the
// transition pass and 3 after the segment chain of a segmented scan (else
// recorded right after 1), 4 after the recurrence.
constexpr int kProfEvents = 5;

void prof_record(int which, cudaStream_t stream) {
    if (!g_prof.active || g_prof.calls >= g_prof.max_calls) return;
    cudaEventRecord(g_prof.ev[kProfEvents * g_prof.calls + which], stream);
}

int device_state(DeviceState** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return KDA_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_DEVICE;
        }
        if (d.cc_major != 10 || d.cc_minor != 3) return KDA_ERR_DEVICE;
        void* sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_device_status) != cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        d.status = static_cast<int*>(sym);
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        // Keep freed blocks in the pool: repeated calls then allocate without
        // going back to the driver.
        uint64_t threshold = UINT64_MAX;
        cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &threshold);
        d.init = true;
    }
    *out = &d;
    return KDA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
    uintptr_t lo, hi;
};
Range range(const void* p, int64_t bytes) {
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}
bool overlap(Range a, Range b) {
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}


int choose_split(int64_t units, int sms) {
    if (g_split_override) return g_split_override;
    // The widest split whose grid still fits on the SMs: with few heads the
    // recurrence is a per-warp latency chain, and more CTAs per head give each
    // warp fewer value columns and keys.
    const int options[] = {16, 8, 4, 2};
    for (int ns : options)
        if (units * ns <= sms) return ns;
    return 1;
}

constexpr int64_t kMaxElems = int64_t(1) << 56;
constexpr float kScale = 0.08838834764831845f;   // 1 / sqrt(128)

struct Plan {
    bool packed;
    int64_t N, tokens;
    SeqGeometry geo;
    int64_t meta_bytes;      // valid flag + cu_chunks + order (packed only), 256-aligned
    int64_t packet_bytes;    // chunk_ub * H * kPacketBytes
    int64_t ready_bytes;     // chunk_ub * H flags of the fused launch, 256-aligned
    int64_t order_bytes;     // packed: chunk order and alone flags of the many-head one-launch form
};

int make_plan(int64_t B, int64_t T, int64_t H, bool packed, Plan* p) {
    if (B < 1 || T < 0 || H < 1) return KDA_ERR_SHAPE;
    // H first: every bound below divides by a multiple of H, which must not
    // overflow (H * 128 * 128 wraps to 0 for H = 2^50).
    if (H > kMaxElems / (kHeadDim * kHeadDim)) return KDA_ERR_SHAPE;
    p->packed = packed;
    p->N = B;
    p->tokens = packed ? T : B * T;
    if (packed ? false : (T > 0 && B > kMaxElems / T)) return KDA_ERR_SHAPE;
    if (p->tokens > kMaxElems / (H * kHeadDim)) return KDA_ERR_SHAPE;
    if (p->tokens >= (int64_t(1) << 31)) return KDA_ERR_SHAPE;   // token index fits int32
    if (B > kMaxElems / (H * kHeadDim * kHeadDim)) return KDA_ERR_SHAPE;
    SeqGeometry& g = p->geo;
    g = SeqGeometry{};
    g.n_seqs = B;
    g.tokens = p->tokens;
    if (packed) {
        g.chunk_ub = (T + (kChunk - 1) * B) / kChunk;
        p->meta_bytes = 256 + ((8 * (B + 1) + 255) / 256) * 256 +
                        (B <= kMaxOrdered ? ((4 * B + 255) / 256) * 256 : 0);
    } else {
        g.tokens_per_seq = T;
        g.chunks_per_seq = (T + kChunk - 1) / kChunk;
        g.chunk_ub = B * g.chunks_per_seq;
        p->meta_bytes = 0;
    }
    if (g.chunk_ub > kMaxElems / (H * kPacketBytes)) return KDA_ERR_SHAPE;
    p->packet_bytes = g.chunk_ub * H * static_cast<int64_t>(kPacketBytes);
    // One flag per packet, then the many-head one-launch form's item counter.
    p->ready_bytes = g.chunk_ub > 0 ? ((g.chunk_ub * H * 4 + 4 + 255) / 256) * 256 : 0;
    p->order_bytes =
        packed && g.chunk_ub > 0 ? ((g.chunk_ub * 4 + 255) / 256) * 256 + ((B * 4 + 255) / 256) * 256
                                 : 0;
    return KDA_OK;
}

// Whether kda_prefill runs preparation and recurrence as one launch: the
// key-split recurrence on part of the SMs, with enough SMs left for the
// preparation to stay ahead of it.  A preparing warp takes about 25 times as
// long per packet as the recurrence takes per chunk, so the free SMs'
// 8 warps each must have at most ~chunks / 4 packets to make.
// Packed batches whose one-CTA-per-head recurrence fits one wave with SMs
// to spare: the k longest sequences (the first k of the metadata kernel's
// longest-first order) run at split 2 in a second, concurrent launch, the
// rest at split 1.  Returns k (0: no second launch).
int64_t long_split_count(const Plan& pl, int64_t H, int nsplit, int sms) {
    if (!pl.packed || g_engine != 0 || g_split_override || nsplit != 1 || pl.N > kMaxOrdered ||
        pl.tokens <= 0)
        return 0;
    const int64_t units = pl.N * H;
    if (units >= sms) return 0;
    const int64_t k = (sms - units) / H;
    return k < pl.N ? k : pl.N;
}

// Segmented scan over chunks (kda_segments.cu): with few (sequence, head)
// chains the serial recurrence leaves most SMs idle, so each sequence is cut
// into segments of seg_chunks chunks and run in three launches (every
// segment's zero-start state and state map; a short chain over each
// sequence's segments; every segment again from its true incoming state).
// The choice compares rough costs in microseconds, measured on GB300: a chunk
// step of the serial chain at the automatic split; a chunk of the transition
// pass and of the rerun; a step of the segment chain; the passes' fixed cost.
double serial_chunk_us(int nsplit) {
    return nsplit >= 16 ? 0.35 : nsplit == 8 ? 0.40 : nsplit == 4 ? 0.58 : nsplit == 2 ? 0.75 : 0.9;
}
constexpr double kTransChunkUs = 1.25;
constexpr double kQuadChunkUs = 1.0;
constexpr double kScanStepUs = 0.6;
constexpr double kSegFixedUs = 12.0;
// From this many segments per sequence (fixed layout) the chain over them
// runs in two levels: groups of about sqrt(segments), composed in parallel,
// then a chain over the groups, then every segment's incoming state.
constexpr int64_t kTwoLevelSegs = 48;
constexpr double kTwoLevelFixedUs = 10.0;

struct SegChoice {
    int64_t segs = 0;         // fixed: segments per sequence; packed: a bound on all segments (0: none)
    int64_t seg_chunks = 0;   // chunks per segment (the last one of a sequence shorter)
    int64_t total = 0;        // segments the three state buffers hold
    int64_t state_bytes = 0;  // bytes of each of the three [total][H][128][128] BF16 buffers
    int64_t meta_bytes = 0;   // packed: seg_begin, seg_chunks, seg_tokens (256-aligned each)
    int64_t group_segs = 0;   // two-level chain: segments per group (0: one level)
    int64_t groups = 0;       // two-level chain: groups per sequence
    int64_t group_bytes = 0;  // two-level chain: prefix and group buffers in all
};

// Segments per group of a two-level chain: about sqrt(segs), but large enough
// that the composition (32 CTAs per group and head, two per SM) fits one
// wave; 0 when one level is better (few segments, or no such size).
int64_t group_size(int64_t segs, int64_t units, int sms, bool forced) {
    if (segs < kTwoLevelSegs) return 0;
    int64_t m = static_cast<int64_t>(std::ceil(std::sqrt(static_cast<double>(segs))));
    if (!forced) {
        const int64_t max_groups = sms / (16 * units);
        if (max_groups < 4) return 0;
        const int64_t m_wave = (segs + max_groups - 1) / max_groups;
        if (m_wave > m) m = m_wave;
    }
    return m;
}

double chain_us(int64_t segs, int64_t m) {
    if (m == 0) return segs * kScanStepUs;
    return kTwoLevelFixedUs + (m - 1 + (segs + m - 1) / m) * kScanStepUs;
}

int64_t align256(int64_t b) { return ((b + 255) / 256) * 256; }

SegChoice plan_segments(const Plan& pl, int64_t H, int sms, bool checkpoints) {
    SegChoice sc;
    if (!g_segments || g_engine != 0 || g_split_override || pl.tokens <= 0) return sc;
    (void)checkpoints;   // the rerun writes them (per-sequence numbering)
    const int64_t units = pl.N * H;
    const double t_serial = serial_chunk_us(choose_split(units, sms));
    if (pl.packed) {
        // Sequence lengths stay on the device: plan on the bound of all
        // chunks; the longest sequence has at least the mean.
        const int64_t C = pl.geo.chunk_ub, N = pl.N;
        int64_t L = g_seg_chunks;
        if (L <= 0) {
            const int64_t budget = sms / H;   // segments per head in one wave
            if (budget < N + 4) return sc;
            L = (C + (budget - N) - 1) / (budget - N);
            const double mean = static_cast<double>(C) / static_cast<double>(N);
            const double seg_us = kSegFixedUs + L * (kTransChunkUs + kQuadChunkUs) +
                                  std::ceil(mean / L) * kScanStepUs;
            if (seg_us >= mean * t_serial) return sc;
        }
        sc.seg_chunks = L;
        sc.segs = C / L + N;
        sc.total = sc.segs;
        sc.meta_bytes = align256(8 * (N + 1)) + 2 * align256(8 * (sc.segs + 1)) + align256(8 * sc.segs);
    } else {
        const int64_t chunks = pl.geo.chunks_per_seq;
        int64_t L = g_seg_chunks;
        if (L <= 0) {
            const int64_t target = sms / units;   // segments per sequence: one wave
            if (target < 4) return sc;
            L = (chunks + target - 1) / target;
            const int64_t segs = (chunks + L - 1) / L;
            if (segs < 4) return sc;
            const double seg_us = kSegFixedUs + L * (kTransChunkUs + kQuadChunkUs) +
                                  chain_us(segs, group_size(segs, units, sms, false));
            if (seg_us >= chunks * t_serial) return sc;
        }
        sc.seg_chunks = L;
        sc.segs = (chunks + L - 1) / L;
        sc.total = pl.N * sc.segs;
        sc.group_segs = group_size(sc.segs, units, sms, g_seg_chunks > 0);
        if (sc.group_segs > 0) {
            sc.groups = (sc.segs + sc.group_segs - 1) / sc.group_segs;
            const int64_t st = H * kHeadDim * kHeadDim * 2;
            sc.group_bytes = (2 * sc.total + 3 * pl.N * sc.groups) * st;
        }
    }
    sc.state_bytes = sc.total * H * kHeadDim * kHeadDim * 2;
    return sc;
}

// Whether the outputs of a call stay clear of its inputs and of each other
// (final_state == init_state, the in-place update, is allowed): the byte
// ranges of the tensors of `pl` with H heads, device or host alike.
bool io_disjoint(const Plan& pl, int64_t H, const void* q, const void* k, const void* v,
                 const void* g, const void* beta, const void* init_state, const void* out,
                 const void* final_state, const void* cu_seqlens, const Checkpoints* ck,
                 const void* ck_cu_starts) {
    const int64_t x_bytes = pl.tokens * H * kHeadDim * 2;
    const int64_t s_bytes = pl.N * H * kHeadDim * kHeadDim * 2;
    const Range rq = range(q, x_bytes), rk = range(k, x_bytes), rv = range(v, x_bytes);
    const Range rg = range(g, pl.tokens * H * kHeadDim * 4), rb = range(beta, pl.tokens * H * 2);
    const Range ro = range(out, x_bytes);
    const Range ri = range(init_state, init_state ? s_bytes : 0);
    const Range rf = range(final_state, final_state ? s_bytes : 0);
    const Range rc = range(cu_seqlens, cu_seqlens ? 8 * (pl.N + 1) : 0);
    for (Range in : {rq, rk, rv, rg, rb, ri, rf, rc})
        if (overlap(ro, in)) return false;
    for (Range in : {rq, rk, rv, rg, rb, rc})
        if (overlap(rf, in)) return false;
    if (final_state && init_state && final_state != init_state && overlap(rf, ri)) return false;
    if (ck) {
        const Range rs = range(ck->states, ck->rows * H * kHeadDim * kHeadDim * 2);
        const Range rcs = range(ck_cu_starts, 8 * (pl.N + 1));
        for (Range in : {rq, rk, rv, rg, rb, ro, ri, rf, rc, rcs})
            if (overlap(rs, in)) return false;
    }
    return true;
}

// The side stream and events of device state d (under g_mu).
bool ensure_side(DeviceState* d) {
    if (d->side) return true;
    // Default (timing) events: with cudaEventDisableTiming ones the packed
    // H=12 call measured ~520 us instead of ~380 us per call on GB300 when
    // nothing else was recorded between its launches.
    if (cudaStreamCreateWithFlags(&d->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&d->fork, cudaEventDefault) != cudaSuccess ||
        cudaEventCreateWithFlags(&d->join, cudaEventDefault) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return true;
}

// The copy streams and events of kda_prefill_host (under g_mu).
bool ensure_host_streams(DeviceState* d) {
    if (d->h2d) return true;
    // Default (timing) events, as for the side stream's fork and join.
    if (cudaStreamCreateWithFlags(&d->h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&d->d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&d->h_start, cudaEventDefault) != cudaSuccess ||
        cudaEventCreateWithFlags(&d->h_in, cudaEventDefault) != cudaSuccess ||
        cudaEventCreateWithFlags(&d->h_done, cudaEventDefault) != cudaSuccess ||
        cudaEventCreateWithFlags(&d->h_out, cudaEventDefault) != cudaSuccess) {
        cudaGetLastError();
        d->h2d = nullptr;
        return false;
    }
    return true;
}

bool use_fusion(const Plan& pl, int64_t H, int nsplit, int sms) {
    if (!g_fusion || g_engine != 0 || pl.packed || pl.tokens <= 0) return false;
    if (!fused_supported(pl.N, H, nsplit, sms)) return false;
    const int64_t free_sms = sms - pl.N * H * nsplit;
    if (free_sms < 16) return false;
    return pl.geo.chunk_ub * H <= free_sms * pl.geo.chunks_per_seq / 4;
}

// Whether kda_prefill runs a fixed-length batch of one recurrence CTA per
// (sequence, head) as the many-head one-launch form (kda_fused.cu): every SM
// holds one CTA, the first N*H of them each run one head's recurrence while
// two warp pairs on each of them and eight on every other SM prepare the
// packets just ahead of it.  The preparation then has fewer pairs than alone
// (1,216 on 152 SMs), so the form gains while enough SMs are left to it.
// Measured on GB300, one launch against two kernels (eager, L2 flushed),
// T=8192: H=80 579 vs 703 us, H=96 664 vs 741, H=112 874 vs 782; T=2048,
// H=96 188 vs 203; B=2, T=4096, H=48 345 vs 383.  Hence the rule: at most two
// thirds of the SMs run a recurrence, and at least 64 chunks per sequence.
// Packed batches (their lengths are on the device only) qualify by the same
// rule on the mean length; their packets are made in the order of the chunks'
// positions relative to their sequence's length (launch_chunk_order).
bool use_fusion_heads(const Plan& pl, int64_t H, int nsplit, int sms, bool checkpoints) {
    if (!g_fusion || g_engine != 0 || g_split_override || pl.tokens <= 0 || checkpoints ||
        nsplit != 1)
        return false;
    if (!fused_heads_supported(pl.N, H, sms)) return false;
    if (3 * pl.N * H > 2 * static_cast<int64_t>(sms)) return false;
    if (pl.packed) return pl.N <= kMaxOrdered && pl.tokens >= 64 * kChunk * pl.N;
    return pl.geo.chunks_per_seq >= 64;
}

// Launch metadata (packed) and preparation into `ws` (meta) and `packets`.
// `ordered`: also have the metadata kernel order the sequences longest-first.
int run_prep(const Plan& pl, const void* q, const void* k, const float* g, const void* beta,
             int64_t H, const int64_t* cu_seqlens, uint8_t* meta, uint8_t* packets,
             DeviceState* d, cudaStream_t stream, SeqGeometry* geo_out, bool ordered = false,
             bool beta_logit = false) {
    SeqGeometry geo = pl.geo;
    if (pl.packed) {
        int32_t* valid = reinterpret_cast<int32_t*>(meta);
        int64_t* cu_chunks = reinterpret_cast<int64_t*>(meta + 256);
        int32_t* order = ordered && pl.N <= kMaxOrdered
                             ? reinterpret_cast<int32_t*>(meta + 256 + ((8 * (pl.N + 1) + 255) / 256) * 256)
                             : nullptr;
        if (launch_varlen_meta(cu_seqlens, pl.N, pl.tokens, valid, cu_chunks, order, d->status,
                               stream) != cudaSuccess)
            return KDA_ERR_CUDA;
        ++t_launches;
        geo.cu_seqlens = cu_seqlens;
        geo.cu_chunks = cu_chunks;
        geo.valid = valid;
        geo.order = order;
    }
    if (launch_prep(q, k, g, beta, packets, geo, H, kScale, d->status, stream, beta_logit) !=
        cudaSuccess)
        return KDA_ERR_CUDA;
    ++t_launches;
    *geo_out = geo;
    return KDA_OK;
}

}  // namespace

int recurrence_engine() { return g_engine; }

// Read-only view of the per-device state for other entry points in this
// library: the device status word and the recurrence split kda_prefill uses.
int device_context(int** status, int64_t units, int* nsplit) {
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != KDA_OK) return rc;
    *status = d->status;
    *nsplit = choose_split(units, d->sms);
    return KDA_OK;
}

}  // namespace kda

using namespace kda;

namespace kda {
namespace {

// kda_prefill and kda_prefill_checkpointed; `ck` null for no checkpoints.
int prefill_impl(const void* q, const void* k, const void* v, const float* g, const void* beta,
                 const void* init_state, void* out, void* final_state, int64_t B, int64_t T,
                 int64_t H, const int64_t* cu_seqlens, void* stream_ptr, const Checkpoints* ck,
                 const void* ck_cu_starts, uint32_t flags = 0) {
    const bool packed = cu_seqlens != nullptr;
    if (flags & ~static_cast<uint32_t>(KDA_FLAG_BETA_LOGIT)) return KDA_ERR_ARG;
    const bool beta_logit = (flags & KDA_FLAG_BETA_LOGIT) != 0;
    Plan pl;
    int rc = make_plan(B, T, H, packed, &pl);
    if (rc != KDA_OK) return rc;
    // Token tensors may be NULL only when there are no tokens to read or write.
    if (pl.tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) ||
        !aligned(out, 16) || !aligned(beta, 2) || (init_state && !aligned(init_state, 16)) ||
        (final_state && !aligned(final_state, 16)) || (cu_seqlens && !aligned(cu_seqlens, 8)))
        return KDA_ERR_ALIGN;

    if (!io_disjoint(pl, H, q, k, v, g, beta, init_state, out, final_state, cu_seqlens, ck,
                     ck_cu_starts))
        return KDA_ERR_OVERLAP;

    DeviceState* d = nullptr;
    rc = device_state(&d);
    if (rc != KDA_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

    const int nsplit = choose_split(pl.N * H, d->sms);
    const SegChoice sc = plan_segments(pl, H, d->sms, ck != nullptr);
    const bool fused_few = sc.segs == 0 && use_fusion(pl, H, nsplit, d->sms);
    const bool fused_many =
        !fused_few && sc.segs == 0 && use_fusion_heads(pl, H, nsplit, d->sms, ck != nullptr);
    const bool fused = fused_few || fused_many;
    const int64_t ws_bytes = pl.meta_bytes + pl.packet_bytes + (fused ? pl.ready_bytes : 0) +
                             (fused_many ? pl.order_bytes : 0) + 3 * sc.state_bytes +
                             sc.meta_bytes + sc.group_bytes;
    uint8_t* ws = nullptr;
    if (ws_bytes > 0) {
        if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&ws), static_cast<size_t>(ws_bytes),
                                    d->pool, stream) != cudaSuccess) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
    }
    SeqGeometry geo;
    prof_record(0, stream);
    bool done = false;
    if (fused) {
        // Reset the ready flags, then one cooperative launch.  If the device
        // refuses the cooperative launch (fewer SMs available to this
        // context), fall through to the two-kernel path.
        uint32_t* ready = reinterpret_cast<uint32_t*>(ws + pl.meta_bytes + pl.packet_bytes);
        int32_t* chunk_order = nullptr;
        int32_t* alone = nullptr;
        geo = pl.geo;
        if (pl.packed) {
            // Offsets checked and chunk offsets on the device, then the
            // preparation's chunk order.
            int32_t* valid = reinterpret_cast<int32_t*>(ws);
            int64_t* cu_chunks = reinterpret_cast<int64_t*>(ws + 256);
            chunk_order = reinterpret_cast<int32_t*>(ws + pl.meta_bytes + pl.packet_bytes +
                                                     pl.ready_bytes);
            alone = chunk_order + ((pl.geo.chunk_ub + 63) / 64) * 64;
            if (launch_varlen_meta(cu_seqlens, pl.N, pl.tokens, valid, cu_chunks, nullptr,
                                   d->status, stream) != cudaSuccess)
                rc = KDA_ERR_CUDA;
            ++t_launches;
            if (rc == KDA_OK && launch_chunk_order(cu_chunks, valid, pl.N, pl.geo.chunk_ub,
                                                   chunk_order, alone, H, d->sms,
                                                   stream) != cudaSuccess)
                rc = KDA_ERR_CUDA;
            ++t_launches;
            geo.cu_seqlens = cu_seqlens;
            geo.cu_chunks = cu_chunks;
            geo.valid = valid;
        }
        if (rc == KDA_OK &&
            cudaMemsetAsync(ready, 0, static_cast<size_t>(pl.ready_bytes), stream) != cudaSuccess)
            rc = KDA_ERR_CUDA;
        prof_record(1, stream);
        prof_record(2, stream);
        prof_record(3, stream);
        if (rc == KDA_OK) {
            const cudaError_t e =
                fused_many
                    ? launch_fused_heads(q, k, g, beta, v, out, init_state, final_state,
                                         ws + pl.meta_bytes, ready, chunk_order, alone, geo, H,
                                         kScale, d->status, stream, beta_logit)
                    : launch_fused(q, k, g, beta, v, out, init_state, final_state,
                                   ws + pl.meta_bytes, ready, pl.geo, H, nsplit, kScale, d->status,
                                   stream, ck, beta_logit);
            if (e == cudaSuccess) {
                done = true;
                ++t_launches;
            }
            else
                cudaGetLastError();
        }
    }
    if (rc == KDA_OK && !done && sc.segs > 0) {
        // Segmented scan: preparation, then the three recurrence passes.
        uint8_t* packets = ws + pl.meta_bytes;
        uint8_t* zstates = packets + pl.packet_bytes;
        uint8_t* maps = zstates + sc.state_bytes;
        uint8_t* starts = maps + sc.state_bytes;
        rc = run_prep(pl, q, k, g, beta, H, cu_seqlens, ws, packets, d, stream, &geo, false,
                      beta_logit);
        SeqGeometry sg = geo;
        int64_t* seg_begin = nullptr;
        if (pl.packed) {
            // Segment offsets from the device-side chunk offsets.
            seg_begin = reinterpret_cast<int64_t*>(starts + sc.state_bytes);
            int64_t* seg_chunk0 = seg_begin + align256(8 * (pl.N + 1)) / 8;
            int64_t* seg_tok0 = seg_chunk0 + align256(8 * (sc.segs + 1)) / 8;
            int64_t* seg_seq = seg_tok0 + align256(8 * (sc.segs + 1)) / 8;
            if (rc == KDA_OK &&
                launch_segment_meta(cu_seqlens, geo.cu_chunks, const_cast<int32_t*>(geo.valid), pl.N,
                                    sc.seg_chunks, sc.segs, seg_begin, seg_chunk0, seg_tok0, seg_seq,
                                    d->status, stream) != cudaSuccess)
                rc = KDA_ERR_CUDA;
            ++t_launches;
            sg.n_seqs = sc.segs;
            sg.cu_seqlens = seg_tok0;
            sg.cu_chunks = seg_chunk0;
            sg.order = nullptr;
            sg.seg_seq = seg_seq;
            sg.seq_chunks = geo.cu_chunks;
        } else {
            sg.n_seqs = pl.N * sc.segs;
            sg.seg_chunks = sc.seg_chunks;
            sg.segs_per_seq = sc.segs;
        }
        prof_record(1, stream);
        if (rc == KDA_OK &&
            launch_transition(v, packets, sg, H, zstates, maps, d->status, stream) != cudaSuccess)
            rc = KDA_ERR_CUDA;
        ++t_launches;
        prof_record(2, stream);
        if (rc == KDA_OK && sc.groups > 0) {
            // Two levels: compose inside groups, chain over the groups, apply.
            const int64_t st = H * kHeadDim * kHeadDim * 2;
            uint8_t* pf = starts + sc.state_bytes + sc.meta_bytes;
            uint8_t* pz = pf + sc.total * st;
            uint8_t* gf = pz + sc.total * st;
            uint8_t* gz = gf + pl.N * sc.groups * st;
            uint8_t* gs = gz + pl.N * sc.groups * st;
            if (launch_segment_compose(maps, zstates, pf, pz, gf, gz, pl.N, sc.segs, sc.group_segs,
                                       sc.groups, H, d->status, stream) != cudaSuccess ||
                launch_segment_scan(init_state, final_state, gf, gz, gs, pl.N, sc.groups, nullptr,
                                    nullptr, H, d->status, stream) != cudaSuccess ||
                launch_segment_apply(gs, pf, pz, starts, pl.N, sc.segs, sc.group_segs, sc.groups, H,
                                     d->status, stream) != cudaSuccess)
                rc = KDA_ERR_CUDA;
            t_launches += 3;
        } else if (rc == KDA_OK &&
                   launch_segment_scan(init_state, final_state, maps, zstates, starts, pl.N,
                                       sc.segs, seg_begin, pl.packed ? geo.valid : nullptr, H,
                                       d->status, stream) != cudaSuccess) {
            rc = KDA_ERR_CUDA;
        } else {
            ++t_launches;
        }
        prof_record(3, stream);
        if (rc == KDA_OK &&
            launch_recurrence(v, out, starts, nullptr, packets, sg, H, 1, d->status, stream, ck) !=
                cudaSuccess)
            rc = KDA_ERR_CUDA;
        ++t_launches;
        done = true;
    }
    if (rc == KDA_OK && !done) {
        // A recurrence grid of more than one wave starts the longest
        // sequences first; a grid of less than one wave gives the longest
        // sequences more CTAs (packed layout).
        const int64_t k_long = long_split_count(pl, H, nsplit, d->sms);
        const bool ordered = pl.packed && (pl.N * H * nsplit > d->sms || k_long > 0);
        rc = run_prep(pl, q, k, g, beta, H, cu_seqlens, ws, ws + pl.meta_bytes, d, stream, &geo,
                      ordered, beta_logit);
        prof_record(1, stream);
        prof_record(2, stream);
        prof_record(3, stream);
        if (rc == KDA_OK && k_long > 0) {
            // Fork: slots 0 .. k_long-1 (the longest) at split 2 on the side
            // stream, the rest at split 1 on the caller's stream; join.
            std::lock_guard<std::mutex> lock(g_mu);
            SeqGeometry g_long = geo, g_rest = geo;
            g_long.n_seqs = k_long;
            g_rest.first_slot = k_long;
            uint8_t* packets = ws + pl.meta_bytes;
            if (!ensure_side(d) || cudaEventRecord(d->fork, stream) != cudaSuccess ||
                cudaStreamWaitEvent(d->side, d->fork, 0) != cudaSuccess ||
                launch_recurrence(v, out, init_state, final_state, packets, g_long, H, 2, d->status,
                                  d->side, ck) != cudaSuccess ||
                launch_recurrence(v, out, init_state, final_state, packets, g_rest, H, 1, d->status,
                                  stream, ck) != cudaSuccess ||
                cudaEventRecord(d->join, d->side) != cudaSuccess ||
                cudaStreamWaitEvent(stream, d->join, 0) != cudaSuccess)
                rc = KDA_ERR_CUDA;
            t_launches += 2;
        } else if (rc == KDA_OK &&
                   launch_recurrence(v, out, init_state, final_state, ws + pl.meta_bytes, geo, H,
                                     nsplit, d->status, stream, ck) != cudaSuccess) {
            rc = KDA_ERR_CUDA;
        } else if (rc == KDA_OK) {
            ++t_launches;
        }
    }
    prof_record(4, stream);
    if (g_prof.active && g_prof.calls < g_prof.max_calls) g_prof.calls += 1;
    if (ws) cudaFreeAsync(ws, stream);
    if (rc != KDA_OK) cudaGetLastError();
    return rc;
}

// ---------------------------------------------------------------------------
// kda_prefill_host: the operation on HOST buffers, with the host <-> device
// copies overlapped with the computation.  The batch is cut into at most
// kMaxSeqGroups pieces, each a contiguous byte range of every tensor: token
// ranges (whole chunks) of a single fixed-length sequence, whose state passes
// from piece to piece through a BF16 state buffer on the device (as a
// final_state -> init_state hand-off of two calls); groups of batch rows of a
// fixed-length batch; or groups of whole sequences of a packed batch.  The
// library's host -> device stream copies piece p + 1 while the caller's stream
// computes piece p with the device path, and its device -> host stream
// returns piece p's outputs meanwhile.
// ---------------------------------------------------------------------------
constexpr int64_t kHostInBytesPerHT = 3 * kHeadDim * 2 + kHeadDim * 4 + 2;   // q, k, v, g, beta
// About this many input bytes per piece (the nearest count, 1 to 8): measured
// on GB300, fewer, larger pieces win where a piece's computation is
// latency-bound (few heads), and up to 8 pieces where it is not (B=1,
// T=8192: H=6 best at 2 pieces, H=96 at 6 to 8; B=1, T=65,536, H=1 at 2).
constexpr int64_t kHostPieceBytes = int64_t(40) << 20;
std::mutex g_host_mu;   // one kda_prefill_host enqueues on the copy streams at a time

struct HostPieces {
    int n = 1;
    int kind = 0;                        // 0 token ranges, 1 batch rows, 2 packed sequences
    int64_t first[kMaxSeqGroups + 1];    // bounds in tokens (kind 0), rows or sequences
};

HostPieces plan_host_pieces(const Plan& pl, int64_t T, int64_t H, const int64_t* cu) {
    HostPieces hp;
    const int64_t bytes = pl.tokens * H * kHostInBytesPerHT;
    int64_t want = (bytes + kHostPieceBytes / 2) / kHostPieceBytes;
    want = want < 1 ? 1 : (want > kMaxSeqGroups ? kMaxSeqGroups : want);
    if (g_host_pieces > 0) want = g_host_pieces;
    if (cu) {
        hp.kind = 2;
        const int64_t N = pl.N;
        if (want > N) want = N;
        hp.first[0] = 0;
        for (int64_t j = 1; j < want; ++j) {
            const int64_t target = T * j / want;
            int64_t s = std::lower_bound(cu, cu + N + 1, target) - cu;
            if (s < hp.first[j - 1] + 1) s = hp.first[j - 1] + 1;
            if (s > N - (want - j)) s = N - (want - j);
            hp.first[j] = s;
        }
        hp.first[want] = N;
        hp.n = static_cast<int>(want);
    } else if (pl.N == 1) {
        hp.kind = 0;
        const int64_t chunks = (T + kChunk - 1) / kChunk;
        if (want > chunks) want = chunks > 0 ? chunks : 1;
        // The last piece's call and outbound copy are not overlapped with
        // anything, so it gets about half the chunks of the others.
        const int64_t per = want > 1 ? (2 * chunks + 2 * want - 2) / (2 * want - 1) : chunks;
        hp.n = 0;
        hp.first[0] = 0;
        for (int64_t c = 0; c < chunks && hp.n < want; ++hp.n) {
            c = hp.n + 1 == want ? chunks : std::min(chunks, c + per);
            hp.first[hp.n + 1] = std::min<int64_t>(c * kChunk, T);
        }
        if (hp.n == 0) hp.n = 1;
        hp.first[hp.n] = T;
    } else {
        hp.kind = 1;
        if (want > pl.N) want = pl.N;
        for (int64_t j = 0; j <= want; ++j) hp.first[j] = pl.N * j / want;
        hp.n = static_cast<int>(want);
    }
    return hp;
}

// Byte offset into a host buffer that may be NULL (then nothing is copied).
void* at(void* p, int64_t bytes) { return p ? static_cast<char*>(p) + bytes : nullptr; }
const void* at(const void* p, int64_t bytes) {
    return p ? static_cast<const char*>(p) + bytes : nullptr;
}

int prefill_host_impl(const void* q, const void* k, const void* v, const float* g,
                      const void* beta, const void* init_state, void* out, void* final_state,
                      int64_t B, int64_t T, int64_t H, const int64_t* cu, void* stream_ptr) {
    const bool packed = cu != nullptr;
    Plan pl;
    int rc = make_plan(B, T, H, packed, &pl);
    if (rc != KDA_OK) return rc;
    if (pl.tokens > 0 && (!q || !k || !v || !g || !beta || !out)) return KDA_ERR_NULL;
    if (packed) {
        if (cu[0] != 0 || cu[pl.N] != T) return KDA_ERR_SEQLENS;
        for (int64_t n = 0; n < pl.N; ++n)
            if (cu[n + 1] < cu[n]) return KDA_ERR_SEQLENS;
    }
    const int64_t xb = pl.tokens * H * kHeadDim * 2, gb = pl.tokens * H * kHeadDim * 4;
    const int64_t bb = pl.tokens * H * 2, sb = pl.N * H * kHeadDim * kHeadDim * 2;
    if (!io_disjoint(pl, H, q, k, v, g, beta, init_state, out, final_state, cu, nullptr, nullptr))
        return KDA_ERR_OVERLAP;
    DeviceState* d = nullptr;
    rc = device_state(&d);
    if (rc != KDA_OK) return rc;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!ensure_host_streams(d)) return KDA_ERR_CUDA;
    }
    const HostPieces hp = plan_host_pieces(pl, T, H, cu);
    // Device images of the tensors (one allocation, 256-byte aligned parts).
    int64_t off = 0;
    auto part = [&off](int64_t bytes) {
        const int64_t at = off;
        off += align256(bytes);
        return at;
    };
    const int64_t oq = part(xb), ok_ = part(xb), ov = part(xb), og = part(gb), ob = part(bb);
    const int64_t oo = part(xb), os = part(sb);
    const int64_t ocu = part(packed ? 8 * (pl.N + 1) : 0);
    const int64_t orb = part(packed ? 8 * (pl.N + hp.n) : 0);
    cudaStream_t S = static_cast<cudaStream_t>(stream_ptr);
    std::lock_guard<std::mutex> hold(g_host_mu);
    uint8_t* buf = nullptr;
    if (cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf), static_cast<size_t>(off), d->pool,
                                S) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    auto* qd = buf + oq;
    auto* kd = buf + ok_;
    auto* vd = buf + ov;
    auto* gd = reinterpret_cast<float*>(buf + og);
    auto* bd = buf + ob;
    auto* od = buf + oo;
    auto* sd = buf + os;
    auto* cud = reinterpret_cast<int64_t*>(buf + ocu);
    auto* rbd = reinterpret_cast<int64_t*>(buf + orb);
    const int64_t xrow = H * kHeadDim * 2, grow = H * kHeadDim * 4, brow = H * 2;
    const int64_t srow = H * kHeadDim * kHeadDim * 2;

    // One piece: nothing to overlap, so every copy goes on the caller's
    // stream (no cross-stream hand-offs).
    const bool one = hp.n == 1;
    cudaStream_t in_st = one ? S : d->h2d, out_st = one ? S : d->d2h;
    cudaError_t e = cudaSuccess;
    if (!one) {
        e = cudaEventRecord(d->h_start, S);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(d->h2d, d->h_start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(d->d2h, d->h_start, 0);
    }
    auto copy = [&e](void* dst, const void* src, int64_t n, cudaMemcpyKind kind, cudaStream_t st) {
        if (e == cudaSuccess && n > 0) e = cudaMemcpyAsync(dst, src, static_cast<size_t>(n), kind, st);
    };
    const cudaMemcpyKind H2D = cudaMemcpyHostToDevice, D2H = cudaMemcpyDeviceToHost;
    if (packed) copy(cud, cu, 8 * (pl.N + 1), H2D, in_st);
    rc = KDA_OK;
    for (int p = 0; p < hp.n && e == cudaSuccess && rc == KDA_OK; ++p) {
        // Tokens [ta, tb) of the tensors and state rows [na, nb) of this piece.
        int64_t ta, tb, na = 0, nb = 1;
        if (hp.kind == 0) {
            ta = hp.first[p];
            tb = hp.first[p + 1];
        } else if (hp.kind == 1) {
            na = hp.first[p];
            nb = hp.first[p + 1];
            ta = na * T;
            tb = nb * T;
        } else {
            na = hp.first[p];
            nb = hp.first[p + 1];
            ta = cu[na];
            tb = cu[nb];
        }
        const int64_t nt = tb - ta;
        copy(qd + ta * xrow, at(q, ta * xrow), nt * xrow, H2D, in_st);
        copy(kd + ta * xrow, at(k, ta * xrow), nt * xrow, H2D, in_st);
        copy(gd + ta * H * kHeadDim, at(g, ta * grow), nt * grow, H2D, in_st);
        copy(bd + ta * brow, at(beta, ta * brow), nt * brow, H2D, in_st);
        copy(vd + ta * xrow, at(v, ta * xrow), nt * xrow, H2D, in_st);
        if (init_state && (hp.kind != 0 || p == 0))
            copy(sd + na * srow, at(init_state, na * srow), (nb - na) * srow, H2D, in_st);
        if (!one && e == cudaSuccess) e = cudaEventRecord(d->h_in, d->h2d);
        if (!one && e == cudaSuccess) e = cudaStreamWaitEvent(S, d->h_in, 0);
        if (e != cudaSuccess) break;
        if (packed && p == 0) {
            SeqGroups groups;
            groups.n = hp.n;
            for (int j = 0; j <= hp.n; ++j) groups.first[j] = hp.first[j];
            e = launch_rebase_offsets(cud, groups, rbd, S);
            if (e != cudaSuccess) break;
            ++t_launches;
        }
        const void* init_p;
        if (hp.kind == 0)
            init_p = (p == 0 && !init_state) ? nullptr : sd;
        else
            init_p = init_state ? sd + na * srow : nullptr;
        rc = prefill_impl(qd + ta * xrow, kd + ta * xrow, vd + ta * xrow, gd + ta * H * kHeadDim,
                          bd + ta * brow, init_p, od + ta * xrow, sd + na * srow,
                          hp.kind == 0 ? 1 : nb - na, hp.kind == 1 ? T : nt, H,
                          packed ? rbd + na + p : nullptr, S, nullptr, nullptr);
        if (rc != KDA_OK) break;
        if (!one) {
            e = cudaEventRecord(d->h_done, S);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(d->d2h, d->h_done, 0);
        }
        copy(at(out, ta * xrow), od + ta * xrow, nt * xrow, D2H, out_st);
        if (final_state && hp.kind != 0)
            copy(at(final_state, na * srow), sd + na * srow, (nb - na) * srow, D2H, out_st);
    }
    if (rc == KDA_OK && e == cudaSuccess && final_state && hp.kind == 0)
        copy(final_state, sd, srow, D2H, out_st);
    // Join both copy streams back into the caller's stream (also after an
    // error, so that the buffer is freed only after every copy issued so far),
    // then free the device images in stream order.
    bool joined = one || (cudaEventRecord(d->h_in, d->h2d) == cudaSuccess &&
                          cudaStreamWaitEvent(S, d->h_in, 0) == cudaSuccess &&
                          cudaEventRecord(d->h_out, d->d2h) == cudaSuccess &&
                          cudaStreamWaitEvent(S, d->h_out, 0) == cudaSuccess);
    if (!joined && e == cudaSuccess) e = cudaErrorUnknown;
    cudaFreeAsync(buf, S);
    if (rc == KDA_OK && e != cudaSuccess) rc = KDA_ERR_CUDA;
    if (rc != KDA_OK) cudaGetLastError();
    return rc;
}

}  // namespace
}  // namespace kda

extern "C" int kda_prefill(const void* q, const void* k, const void* v, const float* g,
                           const void* beta, const void* init_state, void* out,
                           void* final_state, int64_t B, int64_t T, int64_t H,
                           const int64_t* cu_seqlens, void* stream_ptr) {
    t_launches = 0;
    return prefill_impl(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens,
                        stream_ptr, nullptr, nullptr);
}

extern "C" int kda_prefill_host(const void* q, const void* k, const void* v, const float* g,
                                const void* beta, const void* init_state, void* out,
                                void* final_state, int64_t B, int64_t T, int64_t H,
                                const int64_t* cu_seqlens, void* stream_ptr) {
    t_launches = 0;
    return prefill_host_impl(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens,
                             stream_ptr);
}

extern "C" int kda_prefill_checkpointed(const void* q, const void* k, const void* v,
                                        const float* g, const void* beta, const void* init_state,
                                        void* out, void* final_state, int64_t B, int64_t T,
                                        int64_t H, const int64_t* cu_seqlens,
                                        int64_t checkpoint_every_n_tokens, void* state_checkpoints,
                                        const int64_t* checkpoint_cu_starts,
                                        int64_t checkpoint_rows, void* stream_ptr) {
    if (checkpoint_every_n_tokens <= 0 || checkpoint_every_n_tokens % kChunk != 0 ||
        checkpoint_rows < 0)
        return KDA_ERR_ARG;
    if (!checkpoint_cu_starts || !state_checkpoints) return KDA_ERR_NULL;
    if (!aligned(state_checkpoints, 16) || !aligned(checkpoint_cu_starts, 8)) return KDA_ERR_ALIGN;
    if (H < 1 || H > kMaxElems / (kHeadDim * kHeadDim)) return KDA_ERR_SHAPE;
    if (checkpoint_rows > kMaxElems / (H * kHeadDim * kHeadDim)) return KDA_ERR_SHAPE;
    Checkpoints ck;
    ck.states = static_cast<__nv_bfloat16*>(state_checkpoints);
    ck.cu_starts = checkpoint_cu_starts;
    ck.every = checkpoint_every_n_tokens / kChunk;
    ck.rows = checkpoint_rows;
    t_launches = 0;
    return prefill_impl(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens,
                        stream_ptr, &ck, checkpoint_cu_starts);
}

extern "C" int kda_prefill_ex(const void* q, const void* k, const void* v, const float* g,
                              const void* beta, const void* init_state, void* out,
                              void* final_state, int64_t B, int64_t T, int64_t H,
                              const int64_t* cu_seqlens, uint32_t flags,
                              int64_t checkpoint_every_n_tokens, void* state_checkpoints,
                              const int64_t* checkpoint_cu_starts, int64_t checkpoint_rows,
                              void* stream_ptr) {
    t_launches = 0;
    if (!state_checkpoints)
        return prefill_impl(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens,
                            stream_ptr, nullptr, nullptr, flags);
    if (checkpoint_every_n_tokens <= 0 || checkpoint_every_n_tokens % kChunk != 0 ||
        checkpoint_rows < 0)
        return KDA_ERR_ARG;
    if (!checkpoint_cu_starts) return KDA_ERR_NULL;
    if (!aligned(state_checkpoints, 16) || !aligned(checkpoint_cu_starts, 8)) return KDA_ERR_ALIGN;
    if (H < 1 || H > kMaxElems / (kHeadDim * kHeadDim)) return KDA_ERR_SHAPE;
    if (checkpoint_rows > kMaxElems / (H * kHeadDim * kHeadDim)) return KDA_ERR_SHAPE;
    Checkpoints ck;
    ck.states = static_cast<__nv_bfloat16*>(state_checkpoints);
    ck.cu_starts = checkpoint_cu_starts;
    ck.every = checkpoint_every_n_tokens / kChunk;
    ck.rows = checkpoint_rows;
    return prefill_impl(q, k, v, g, beta, init_state, out, final_state, B, T, H, cu_seqlens,
                        stream_ptr, &ck, checkpoint_cu_starts, flags);
}

extern "C" int kda_prep_only(const void* q, const void* k, const float* g, const void* beta,
                             int64_t B, int64_t T, int64_t H, const int64_t* cu_seqlens,
                             void* packets, int64_t packets_bytes, void* stream_ptr) {
    if (!q || !k || !g || !beta || !packets) return KDA_ERR_NULL;
    const bool packed = cu_seqlens != nullptr;
    Plan pl;
    int rc = make_plan(B, T, H, packed, &pl);
    if (rc != KDA_OK) return rc;
    if (packets_bytes < pl.packet_bytes) return KDA_ERR_SHAPE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(g, 16) || !aligned(beta, 2) ||
        !aligned(packets, 16) || (cu_seqlens && !aligned(cu_seqlens, 8)))
        return KDA_ERR_ALIGN;
    DeviceState* d = nullptr;
    rc = device_state(&d);
    if (rc != KDA_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    uint8_t* meta = nullptr;
    if (pl.meta_bytes > 0 &&
        cudaMallocFromPoolAsync(reinterpret_cast<void**>(&meta), static_cast<size_t>(pl.meta_bytes),
                                d->pool, stream) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    SeqGeometry geo;
    rc = run_prep(pl, q, k, g, beta, H, cu_seqlens, meta, static_cast<uint8_t*>(packets), d,
                  stream, &geo);
    if (meta) cudaFreeAsync(meta, stream);
    if (rc != KDA_OK) cudaGetLastError();
    return rc;
}

extern "C" int kda_set_host_pieces(int n) {
    if (n < 0 || n > kMaxSeqGroups) return KDA_ERR_ARG;
    g_host_pieces = n;
    return KDA_OK;
}

extern "C" int kda_last_call_launches(int64_t* n) {
    if (!n) return KDA_ERR_NULL;
    *n = t_launches;
    return KDA_OK;
}

extern "C" const char* kda_error_string(int status) {
    switch (status) {
        case KDA_OK: return "success";
        case KDA_ERR_NULL: return "a required pointer is NULL";
        case KDA_ERR_SHAPE: return "B, T or H out of range (or a size overflows)";
        case KDA_ERR_ALIGN: return "a pointer is not suitably aligned";
        case KDA_ERR_OVERLAP: return "an output overlaps an input or another output";
        case KDA_ERR_DEVICE: return "no CUDA device of compute capability 10.3 is current";
        case KDA_ERR_CUDA: return "a CUDA runtime call failed";
        case KDA_ERR_ARG: return "an option value is out of range";
        case KDA_ERR_SCRATCH:
            return "the shape needs more scratch than the fixed no-allocation buffer holds";
        case KDA_ERR_SEQLENS: return "host cu_seqlens break their contract";
        default: return "unknown KDA status";
    }
}

extern "C" int kda_device_status(void* stream_ptr, int* status) {
    if (!status) return KDA_ERR_NULL;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != KDA_OK) return rc;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    int zero = 0;
    if (cudaMemcpy(status, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

extern "C" int kda_set_split(int nsplit) {
    if (nsplit != 0 && nsplit != 1 && nsplit != 2 && nsplit != 4 && nsplit != 8 && nsplit != 16)
        return KDA_ERR_ARG;
    g_split_override = nsplit;
    return KDA_OK;
}

extern "C" int kda_plan_fused(int64_t B, int64_t T, int64_t H, int packed, int* fused) {
    if (!fused) return KDA_ERR_NULL;
    Plan pl;
    int rc = make_plan(B, T, H, packed != 0, &pl);
    if (rc != KDA_OK) return rc;
    DeviceState* d = nullptr;
    rc = device_state(&d);
    if (rc != KDA_OK) return rc;
    const int nsplit = choose_split(pl.N * H, d->sms);
    *fused = plan_segments(pl, H, d->sms, false).segs == 0 &&
                     (use_fusion(pl, H, nsplit, d->sms) ||
                      use_fusion_heads(pl, H, nsplit, d->sms, false))
                 ? 1
                 : 0;
    return KDA_OK;
}

extern "C" int kda_plan_long_split(int64_t n_seqs, int64_t T, int64_t H, int64_t* k) {
    if (!k) return KDA_ERR_NULL;
    Plan pl;
    int rc = make_plan(n_seqs, T, H, true, &pl);
    if (rc != KDA_OK) return rc;
    DeviceState* d = nullptr;
    rc = device_state(&d);
    if (rc != KDA_OK) return rc;
    const int nsplit = choose_split(pl.N * H, d->sms);
    // None when the call runs as the many-head one-launch form.
    const bool many = plan_segments(pl, H, d->sms, false).segs == 0 &&
                      use_fusion_heads(pl, H, nsplit, d->sms, false);
    *k = many ? 0 : long_split_count(pl, H, nsplit, d->sms);
    return KDA_OK;
}

extern "C" int kda_set_fusion(int on) {
    if (on != 0 && on != 1) return KDA_ERR_ARG;
    g_fusion = on;
    return KDA_OK;
}

extern "C" int kda_set_segments(int on, int64_t seg_chunks) {
    if ((on != 0 && on != 1) || seg_chunks < 0 || seg_chunks > (int64_t(1) << 26)) return KDA_ERR_ARG;
    g_segments = on;
    g_seg_chunks = seg_chunks;
    return KDA_OK;
}

extern "C" int kda_plan_segments(int64_t B, int64_t T, int64_t H, int packed, int64_t* segs) {
    if (!segs) return KDA_ERR_NULL;
    Plan pl;
    int rc = make_plan(B, T, H, packed != 0, &pl);
    if (rc != KDA_OK) return rc;
    DeviceState* d = nullptr;
    rc = device_state(&d);
    if (rc != KDA_OK) return rc;
    *segs = plan_segments(pl, H, d->sms, false).segs;
    return KDA_OK;
}

extern "C" int kda_set_engine(int engine) {
    if (engine < 0 || engine > 2) return KDA_ERR_ARG;
    g_engine = engine;
    return KDA_OK;
}

extern "C" int kda_auto_split(int64_t n_seqs, int64_t H, int* nsplit) {
    if (!nsplit) return KDA_ERR_NULL;
    if (n_seqs < 1 || H < 1) return KDA_ERR_SHAPE;
    DeviceState* d = nullptr;
    int rc = device_state(&d);
    if (rc != KDA_OK) return rc;
    *nsplit = choose_split(n_seqs * H, d->sms);
    return KDA_OK;
}

extern "C" int kda_workspace_bytes(int64_t B, int64_t T, int64_t H, int packed, int64_t* bytes) {
    if (!bytes) return KDA_ERR_NULL;
    Plan pl;
    int rc = make_plan(B, T, H, packed != 0, &pl);
    if (rc != KDA_OK) return rc;
    // The segmented scan's buffers as planned on the current device (on a
    // 152-SM device when there is none).
    int sms = 152;
    DeviceState* d = nullptr;
    if (device_state(&d) == KDA_OK) sms = d->sms;
    const SegChoice sc = plan_segments(pl, H, sms, false);
    // Fixed layout: the ready flags of a one-launch form are always counted;
    // packed: the flags and the chunk order when the many-head form is planned.
    const bool packed_fused =
        pl.packed && sc.segs == 0 && use_fusion_heads(pl, H, choose_split(pl.N * H, sms), sms, false);
    *bytes = pl.meta_bytes + pl.packet_bytes +
             (pl.packed ? (packed_fused ? pl.ready_bytes + pl.order_bytes : 0) : pl.ready_bytes) +
             3 * sc.state_bytes + sc.meta_bytes + sc.group_bytes;
    return KDA_OK;
}

extern "C" int64_t kda_packet_bytes(void) { return kPacketBytes; }

extern "C" int kda_profile_begin(int max_calls) {
    if (max_calls < 1 || max_calls > (1 << 20)) return KDA_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_prof.active) return KDA_ERR_ARG;
    g_prof.ev = new cudaEvent_t[kProfEvents * static_cast<size_t>(max_calls)];
    for (int i = 0; i < kProfEvents * max_calls; ++i) {
        if (cudaEventCreate(&g_prof.ev[i]) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(g_prof.ev[j]);
            delete[] g_prof.ev;
            g_prof.ev = nullptr;
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
    }
    g_prof.max_calls = max_calls;
    g_prof.calls = 0;
    g_prof.active = true;
    return KDA_OK;
}

extern "C" int kda_profile_end_detail(double* intervals_ms, int* calls) {
    if (!intervals_ms || !calls) return KDA_ERR_NULL;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_prof.active) return KDA_ERR_ARG;
    double t[kProfEvents - 1] = {};
    int rc = KDA_OK;
    for (int c = 0; c < g_prof.calls && rc == KDA_OK; ++c) {
        const cudaEvent_t* ev = g_prof.ev + kProfEvents * c;
        if (cudaEventSynchronize(ev[kProfEvents - 1]) != cudaSuccess) rc = KDA_ERR_CUDA;
        for (int i = 0; i + 1 < kProfEvents && rc == KDA_OK; ++i) {
            float ms = 0.f;
            if (cudaEventElapsedTime(&ms, ev[i], ev[i + 1]) != cudaSuccess)
                rc = KDA_ERR_CUDA;
            t[i] += ms;
        }
    }
    if (rc != KDA_OK) cudaGetLastError();
    for (int i = 0; i + 1 < kProfEvents; ++i) intervals_ms[i] = t[i];
    *calls = g_prof.calls;
    for (int i = 0; i < kProfEvents * g_prof.max_calls; ++i) cudaEventDestroy(g_prof.ev[i]);
    delete[] g_prof.ev;
    g_prof = Profile{};
    return rc;
}

extern "C" int kda_profile_end(double* prep_ms, double* recurrence_ms, int* calls) {
    if (!prep_ms || !recurrence_ms || !calls) return KDA_ERR_NULL;
    double t[kProfEvents - 1] = {};
    const int rc = kda_profile_end_detail(t, calls);
    *prep_ms = t[0];
    *recurrence_ms = t[1] + t[2] + t[3];
    return rc;
}
