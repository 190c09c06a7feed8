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
    return KsLayout<NCG>::kSmemBytes > prep::kPrepSmemBytes ? KsLayout<NCG>::kSmemBytes
                                                            : prep::kPrepSmemBytes;
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
        prep::run_items(f.p, maps, smem + pair * prep::kPrepRegion, bar, bid, hw, lane,
                        pb * prep::kPrepPairs + pair, pgrid * prep::kPrepPairs, f.ready);
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

}  // namespace

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
