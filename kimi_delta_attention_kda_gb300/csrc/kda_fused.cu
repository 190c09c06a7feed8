// kda_fused.cu -- chunk preparation and recurrence in one launch.
//
// With few (sequence, head) units the recurrence occupies only some of the
// SMs and is a latency-bound chain on each of them, while the preparation is
// a short parallel pass ahead of it.  This kernel runs both at once: CTAs
// 0 .. R-1 are the key-split recurrence (kda_rec_impl.cuh), CTAs R .. SMs-1
// prepare packets (kda_prep_impl.cuh) in chunk-major order.  A preparing warp
// publishes ready[chunk * H + head] = 1 (release, GPU scope) once that packet
// is complete in global memory; the recurrence's producer warp waits for the
// flag (acquire, bounded) before it copies the packet.  The launch is
// cooperative, so every CTA is resident at once and no wait depends on a CTA
// that has not started.  The arithmetic is that of the two separate kernels,
// so the results are bit for bit those of the unfused path.
#include <cuda.h>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_prep_impl.cuh"
#include "kda_rec_impl.cuh"

namespace kda {
namespace {

using namespace rec;

constexpr int kFusedThreads = prep::kPrepWarps * 32;

struct FusedArgs {
    prep::PrepArgs p;
    RecArgs r;
    int64_t rec_blocks;
    uint32_t* ready;
};

template <int NCG>
constexpr uint32_t fused_smem_bytes() {
    return KsLayout<NCG>::kSmemBytes > prep::kPrepSmemBytes + 32 ? KsLayout<NCG>::kSmemBytes
                                                                 : prep::kPrepSmemBytes + 32;
}

template <int NCG>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_kernel(FusedArgs f, const __grid_constant__ prep::PrepMaps maps,
                 const __grid_constant__ CUtensorMap vmap) {
    static_assert((2 * NCG + 1) * 32 <= kFusedThreads, "recurrence CTA must fit the block");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (blockIdx.x < f.rec_blocks) {
        ks_setup<NCG>(smem);
        __syncthreads();
        ks_run<NCG>(f.r, &vmap, smem, blockIdx.x, f.ready);
    } else {
        const int pair = warp >> 1, hw = warp & 1, bid = 1 + pair;
        uint64_t* bar = prep::pair_barrier(smem, pair, hw, lane, bid);
        const int64_t pb = static_cast<int64_t>(blockIdx.x) - f.rec_blocks;
        const int64_t pgrid = static_cast<int64_t>(gridDim.x) - f.rec_blocks;
        prep::PairCtl* ctl = reinterpret_cast<prep::PairCtl*>(
            smem + prep::kPrepPairs * prep::kPrepRegion + 8 * prep::kPrepPairs);
        if (threadIdx.x == 0) {
            ctl->ready = f.ready;
            ctl->counter = nullptr;
        }
        __syncthreads();
        prep::run_items(f.p, maps, smem + pair * prep::kPrepRegion, bar, bid, hw, lane,
                        pb * prep::kPrepPairs + pair, pgrid * prep::kPrepPairs, ctl);
    }
}

template <int NCG>
cudaError_t launch_fused_ncg(FusedArgs& f, const prep::PrepMaps& maps, const CUtensorMap& vmap,
                             int sms, cudaStream_t stream) {
    constexpr uint32_t smem = fused_smem_bytes<NCG>();
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(fused_kernel<NCG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    void* args[] = {&f, const_cast<prep::PrepMaps*>(&maps), const_cast<CUtensorMap*>(&vmap)};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fused_kernel<NCG>),
                                       dim3(static_cast<unsigned>(sms)), dim3(kFusedThreads), args,
                                       smem, stream);
}

// ---------------------------------------------------------------------------
// The one-launch form for many (sequence, head) units (fixed or packed
// layout, one recurrence CTA per unit, N*H <= SMs): every SM holds one 16-warp CTA,
// launched at 128 registers a thread.  CTAs 0 .. R-1 (R = N*H) each run a
// whole head's recurrence: warpgroup 0 (warps 0-3) is the quad form (32 value
// columns a warp, kda_rec_impl.cuh) and takes 256 registers a thread with
// setmaxnreg, which warpgroups 1 and 3 give up (down to 24: warp 4 is the
// producer, which waits for each packet's ready flag; warps 5-7 and 12-15
// leave); warpgroup 2 prepares packets (two warp pairs, 128 registers).  The
// other CTAs prepare packets on all 16 warps (eight pairs).  The shares,
// 128 x (256 + 24 + 128 + 24), stay within the launch's 512 x 128 registers.
// Every pair takes items in order from a counter, numbered chunk first (the
// preparation's interleaved order; packed batches by the chunks' positions
// relative to their sequence's length), so the packets of each chunk index
// appear for every head at about the same time and the recurrences stay close
// behind them, and the pairs that share an SM with a recurrence (slower) take
// fewer items than the others.  The preparation never waits on the recurrence, and
// the cooperative launch keeps every CTA resident, so every wait (bounded)
// ends.  The arithmetic is that of the preparation and quad kernels: the
// results are bit for bit those of the two-kernel path.
// ---------------------------------------------------------------------------
constexpr int kFhWarps = 16;
constexpr int kFhThreads = kFhWarps * 32;
constexpr int kFhRecWarps = 4;    // warpgroup 0
constexpr int kFhProdWarp = 4;    // first warp of warpgroup 1
constexpr int kFhRecPairs = 2;    // warpgroup 2 (warpgroup 3 gives its registers away)
constexpr int kFhPrepPairs = 8;   // all warps of a preparing CTA
constexpr int kFhStages = 8;
constexpr uint32_t kFhRecRegs = 256, kFhIdleRegs = 24;
static_assert(128 * (kFhRecRegs + 2 * kFhIdleRegs + 128) <= kFhThreads * 128,
              "register shares must fit the launch's registers");
constexpr uint32_t kFhRingBytes = kFhStages * kWideStageBytes;
constexpr uint32_t kFhRecPrepOff = kFhRingBytes + 1024;   // ring barriers in between
constexpr uint32_t kFhRecPairBarOff = kFhRecPrepOff + kFhRecPairs * prep::kPrepRegion;
constexpr uint32_t kFhPrepPairBarOff = kFhPrepPairs * prep::kPrepRegion;
// Each pair's mbarrier and its item slot (run_items' counter mode) follow the regions.
constexpr uint32_t kFhRecBytes = kFhRecPairBarOff + (8 + sizeof(prep::PairCtl)) * kFhRecPairs;
constexpr uint32_t kFhPrepBytes = kFhPrepPairBarOff + (8 + sizeof(prep::PairCtl)) * kFhPrepPairs;
constexpr uint32_t kFhSmemBytes = (kFhRecBytes > kFhPrepBytes ? kFhRecBytes : kFhPrepBytes) + 1024;
static_assert(kFhSmemBytes <= 227 * 1024, "one-launch CTA exceeds shared memory");
static_assert(2 * kFhStages * 8 <= 1024, "ring barriers overflow their slot");

struct FusedHeadsArgs {
    prep::PrepArgs p;
    RecArgs r;
    int64_t rec_blocks;
    uint32_t* ready;     // one flag per packet, then the item counter (all zero at launch)
    uint32_t* counter;
    const int32_t* alone;   // packed, may be null: alone[n] = 1, no preparing pairs beside n's heads
};

// The mbarrier of pair `pair` (at bars[pair]), initialised by the pair's
// first thread, then the pair's named barrier.
__device__ __forceinline__ uint64_t* fh_pair_barrier(uint64_t* bars, int pair, int hw, int lane,
                                                     int bid) {
    uint64_t* bar = bars + pair;
    if (hw == 0 && lane == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    pair_sync(bid);
    return bar;
}

__global__ void __launch_bounds__(kFhThreads, 1)
    fused_heads_kernel(FusedHeadsArgs f, const __grid_constant__ prep::PrepMaps maps,
                       const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t rec = f.rec_blocks;
    const int64_t pairs = rec * kFhRecPairs + (static_cast<int64_t>(gridDim.x) - rec) * kFhPrepPairs;
    if (blockIdx.x < rec) {
        const RecArgs& a = f.r;
        const int64_t n = blockIdx.x / a.H;
        const int64_t h = blockIdx.x - n * a.H;
        int64_t c_begin, nch, tok0, seqlen;
        // Packed offsets found invalid: the whole CTA leaves before any
        // register setting (every warp reads the same flag).
        if (!seq_span(a.geo, n, c_begin, nch, tok0, seqlen)) return;
        uint64_t* full = reinterpret_cast<uint64_t*>(smem + kFhRingBytes);
        uint64_t* empty = full + kFhStages;
        if (threadIdx.x == 0) {
            for (int s = 0; s < kFhStages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kFhRecWarps);
            }
            fence_barrier_init();
        }
        __syncthreads();
        if (warp < kFhRecWarps) {
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kFhRecRegs) : "memory");
            wide_consume<4, kFhStages, false>(a, smem, full, empty, warp, lane, n, h, c_begin, nch,
                                              tok0, seqlen);
        } else if (warp < 2 * kFhRecWarps) {
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kFhIdleRegs) : "memory");
            if (warp == kFhProdWarp)
                wide_produce<kFhStages>(a, &vmap, smem, full, empty, lane, h, c_begin, nch, tok0,
                                        f.ready);
        } else if (warp >= 3 * kFhRecWarps) {
            // Warpgroup 3 gives its registers to warpgroup 0 and leaves.
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kFhIdleRegs) : "memory");
        } else {
            // A long sequence's recurrence runs alone on its SM (its step is
            // the critical chain); both warps of every pair read the same flag.
            if (f.alone && f.alone[n]) return;
            const int pair = (warp - 2 * kFhRecWarps) >> 1, hw = warp & 1;
            const int bid = 1 + pair;
            uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kFhRecPairBarOff);
            uint64_t* bar = fh_pair_barrier(bars, pair, hw, lane, bid);
            prep::PairCtl* ctl = reinterpret_cast<prep::PairCtl*>(bars + kFhRecPairs) + pair;
            if (hw == 0 && lane == 0) {
                ctl->ready = f.ready;
                ctl->counter = f.counter;
            }
            pair_sync(bid);
            prep::run_items(f.p, maps, smem + kFhRecPrepOff + pair * prep::kPrepRegion, bar, bid, hw,
                            lane, 0, pairs, ctl);
        }
    } else {
        const int pair = warp >> 1, hw = warp & 1, bid = 1 + pair;
        uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kFhPrepPairBarOff);
        uint64_t* bar = fh_pair_barrier(bars, pair, hw, lane, bid);
        prep::PairCtl* ctl = reinterpret_cast<prep::PairCtl*>(bars + kFhPrepPairs) + pair;
        if (hw == 0 && lane == 0) {
            ctl->ready = f.ready;
            ctl->counter = f.counter;
        }
        pair_sync(bid);
        prep::run_items(f.p, maps, smem + pair * prep::kPrepRegion, bar, bid, hw, lane, 0, pairs, ctl);
    }
}

}  // namespace

bool fused_heads_supported(int64_t n_seqs, int64_t H, int sms) {
    const int64_t units = n_seqs * H;
    return units >= 1 && units <= sms;
}

cudaError_t launch_fused_heads(const void* q, const void* k, const float* g, const void* beta,
                               const void* v, void* out, const void* init_state, void* final_state,
                               uint8_t* packets, uint32_t* ready, const int32_t* chunk_order,
                               const int32_t* alone, const SeqGeometry& geo, int64_t H,
                               float scale, int* status, cudaStream_t stream, bool beta_logit) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (geo.seg_chunks || geo.tokens <= 0 || geo.tokens >= (int64_t(1) << 31) ||
        (geo.cu_chunks && (!chunk_order || !geo.valid || !geo.cu_seqlens)) ||
        !fused_heads_supported(geo.n_seqs, H, sms))
        return cudaErrorInvalidValue;
    FusedHeadsArgs f;
    if (!prep::make_prep_args(&f.p, beta, packets, geo, H, scale, status, beta_logit))
        return cudaErrorInvalidValue;
    // Items in the order the recurrences consume them: fixed layout chunk
    // index first; packed by the chunks' relative positions.
    if (geo.cu_chunks)
        f.p.chunk_order = chunk_order;
    else
        f.p.interleave = 1;
    f.r.v = static_cast<const __nv_bfloat16*>(v);
    f.r.out = static_cast<__nv_bfloat16*>(out);
    f.r.init_state = static_cast<const __nv_bfloat16*>(init_state);
    f.r.final_state = static_cast<__nv_bfloat16*>(final_state);
    f.r.packets = packets;
    f.r.geo = geo;
    f.r.H = H;
    f.r.nsplit = 1;
    f.r.status = status;
    f.r.ck = Checkpoints{nullptr, nullptr, 1, 0};
    f.r.final_ident = nullptr;
    f.rec_blocks = geo.n_seqs * H;
    f.ready = ready;
    f.counter = ready + geo.chunk_ub * H;
    f.alone = geo.cu_chunks ? alone : nullptr;
    prep::PrepMaps maps;
    e = prep::encode_maps(&maps, q, k, g, geo.tokens, H);
    if (e != cudaSuccess) return e;
    CUtensorMap vmap;
    e = encode_v_map_sw128(&vmap, v, geo.tokens, H);
    if (e != cudaSuccess) return e;
    static bool configured[64] = {};
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(fused_heads_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kFhSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    void* args[] = {&f, &maps, &vmap};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fused_heads_kernel),
                                       dim3(static_cast<unsigned>(sms)), dim3(kFhThreads), args,
                                       kFhSmemBytes, stream);
}

bool fused_supported(int64_t n_seqs, int64_t H, int nsplit, int sms) {
    if (nsplit != 8 && nsplit != 16) return false;
    const int64_t rec_blocks = n_seqs * H * nsplit;
    return rec_blocks >= 1 && rec_blocks < sms;
}

cudaError_t launch_fused(const void* q, const void* k, const float* g, const void* beta,
                         const void* v, void* out, const void* init_state, void* final_state,
                         uint8_t* packets, uint32_t* ready, const SeqGeometry& geo, int64_t H,
                         int nsplit, float scale, int* status, cudaStream_t stream,
                         const Checkpoints* ck, bool beta_logit) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (geo.cu_chunks || geo.tokens <= 0 || geo.tokens >= (int64_t(1) << 31) ||
        !fused_supported(geo.n_seqs, H, nsplit, sms))
        return cudaErrorInvalidValue;

    FusedArgs f;
    if (!prep::make_prep_args(&f.p, beta, packets, geo, H, scale, status, beta_logit))
        return cudaErrorInvalidValue;
    f.r.v = static_cast<const __nv_bfloat16*>(v);
    f.r.out = static_cast<__nv_bfloat16*>(out);
    f.r.init_state = static_cast<const __nv_bfloat16*>(init_state);
    f.r.final_state = static_cast<__nv_bfloat16*>(final_state);
    f.r.packets = packets;
    f.r.geo = geo;
    f.r.H = H;
    f.r.nsplit = nsplit;
    f.r.status = status;
    f.r.ck = ck ? *ck : Checkpoints{nullptr, nullptr, 1, 0};
    f.r.final_ident = nullptr;
    f.rec_blocks = geo.n_seqs * H * nsplit;
    f.ready = ready;

    prep::PrepMaps maps;
    e = prep::encode_maps(&maps, q, k, g, geo.tokens, H);
    if (e != cudaSuccess) return e;
    CUtensorMap vmap;
    e = encode_v_map(&vmap, v, geo.tokens, H, kHeadDim / nsplit);
    if (e != cudaSuccess) return e;
    return nsplit == 16 ? launch_fused_ncg<1>(f, maps, vmap, sms, stream)
                        : launch_fused_ncg<2>(f, maps, vmap, sms, stream);
}

}  // namespace kda
