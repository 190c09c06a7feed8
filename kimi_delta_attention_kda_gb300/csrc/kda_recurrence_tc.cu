// kda_recurrence_tc.cu -- the KDA recurrence on the tcgen05 tensor cores
// (sm_103a), one CTA per (sequence, head): eight state warps, an MMA-issuing
// warp and a producer warp (the roles of kda_tc_impl.cuh).  The whole chain
// (the FP32 state, its BF16 operand copy and every accumulator) lives in
// tensor memory; the ring of packet + V stages is in shared memory.
#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_tc_impl.cuh"

namespace kda {
namespace {

constexpr int kTcStages = 4;
constexpr uint32_t kTcOffUA = kTcStages * tcr::kStageBytes;   // U (FP16), 128 x 16, SW32
constexpr uint32_t kTcOffVT = kTcOffUA + 4096;                 // V^T (BF16), 128 x 16, SW32
constexpr uint32_t kTcOffBar = kTcOffVT + 4096;
constexpr int kTcNumBars = 2 * kTcStages + tcr::kExtraBars;
constexpr uint32_t kTcOffTmemPtr = kTcOffBar + kTcNumBars * 8;
constexpr uint32_t kTcSmemBytes = kTcOffTmemPtr + 16 + 1024;   // + alignment slack
constexpr int kMmaWarp = 8, kProdWarp = 9;
constexpr int kTcThreads = 320;

struct TcArgs {
    const __nv_bfloat16* v;
    __nv_bfloat16* out;
    const __nv_bfloat16* init_state;
    __nv_bfloat16* final_state;
    const uint8_t* packets;
    SeqGeometry geo;
    int64_t H;
    int* status;
};

__global__ void __launch_bounds__(kTcThreads, 2)
    recurrence_tc_kernel(TcArgs a, const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const tcr::Bars bars = tcr::make_bars<kTcStages>(reinterpret_cast<uint64_t*>(smem + kTcOffBar));
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + kTcOffTmemPtr);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n_slot = blockIdx.x / a.H;
    tcr::Chain ch;
    ch.h = blockIdx.x - n_slot * a.H;
    ch.n = a.geo.order ? a.geo.order[n_slot] : n_slot;   // longest-first (packed)
    if (a.geo.cu_chunks) {
        if (!*a.geo.valid) return;
        ch.c_begin = a.geo.cu_chunks[ch.n];
        ch.nch = a.geo.cu_chunks[ch.n + 1] - ch.c_begin;
        ch.tok0 = a.geo.cu_seqlens[ch.n];
        ch.seqlen = a.geo.cu_seqlens[ch.n + 1] - ch.tok0;
    } else {
        ch.c_begin = ch.n * a.geo.chunks_per_seq;
        ch.nch = a.geo.chunks_per_seq;
        ch.tok0 = ch.n * a.geo.tokens_per_seq;
        ch.seqlen = a.geo.tokens_per_seq;
    }
    ch.v = a.v;
    ch.out = a.out;
    ch.init_state = a.init_state;
    ch.final_state = a.final_state;
    ch.packets = a.packets;
    ch.ready = nullptr;
    ch.H = a.H;
    ch.status = a.status;

    if (threadIdx.x == 0) {
        tcr::init_bars<kTcStages>(bars);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_ptr, tcr::kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_ptr;

    if (warp == kProdWarp)
        tcr::produce<kTcStages>(ch, &vmap, smem, bars, lane);
    else if (warp == kMmaWarp)
        tcr::issue<kTcStages>(ch, smem, smem + kTcOffVT, smem + kTcOffUA, bars, tmem, lane);
    else
        tcr::state<kTcStages>(ch, smem, smem + kTcOffVT, smem + kTcOffUA, bars, tmem, warp, lane);

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, tcr::kTmemCols);
    }
}

}  // namespace

cudaError_t launch_recurrence_tc(const void* v, void* out, const void* init_state,
                                 void* final_state, const uint8_t* packets, const SeqGeometry& geo,
                                 int64_t H, int* status, cudaStream_t stream) {
    TcArgs a;
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.init_state = static_cast<const __nv_bfloat16*>(init_state);
    a.final_state = static_cast<__nv_bfloat16*>(final_state);
    a.packets = packets;
    a.geo = geo;
    a.H = H;
    a.status = status;
    const int64_t blocks = geo.n_seqs * H;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL || geo.tokens >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static bool configured[64] = {};
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(recurrence_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kTcSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    CUtensorMap vmap;
    alignas(64) static const char kZero[16] = {};
    const void* vbase = v ? v : static_cast<const void*>(kZero);
    cudaError_t e = encode_v_map(&vmap, vbase, geo.tokens, H, kHeadDim);
    if (e != cudaSuccess) return e;
    recurrence_tc_kernel<<<static_cast<unsigned>(blocks), kTcThreads, kTcSmemBytes, stream>>>(a, vmap);
    return cudaGetLastError();
}

}  // namespace kda
