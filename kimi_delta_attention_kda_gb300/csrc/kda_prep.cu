// kda_prep.cu -- chunk preparation for KDA prefill (sm_103a).
//
// A pair of warps prepares one (chunk, head): 16 tokens of q, k, g and beta
// in, one packet (kda_common.cuh) out.  Following "FlashKDA column split", section 1,
// for tokens i = 0..15 of the chunk and key channel c:
//   qhat, khat    per-token L2 normalisation (flashinfer kda_prefill,
//                 use_qk_l2norm_in_kernel): x / sqrt(sum x^2 + 1e-6)
//   G_i[c]        cumulative log-decay sum_{t<=i} g_t[c] in FP32
//                 ("K3's KDA precision problem", decay in tiles)
//   K^start_i     = exp(G_i) khat_i          (D_{0:i} inclusive of token i)
//   s Q^start_i   = s exp(G_i) qhat_i
//   K^end_i       = exp(G_15 - G_i) khat_i   (D_{i+1:15})
//   D_{0:15}      = exp(G_15)
//   A^qk_ij       = s <qhat_i exp(G_i), khat_j exp(-G_j)>,  j <= i
//   R_ij          = beta_i <khat_i exp(G_i), khat_j exp(-G_j)>, j < i
// The two score matrices use the split-exponent GEMM of "K3's KDA precision
// problem" (a 16 x 16 x 128 product of exp(G)-scaled and exp(-G)-scaled
// operands on the tensor cores); with g in [-5, 0] the factors stay within
// exp(+-80), inside the FP32/BF16 range.  Each operand is carried as a BF16
// high part plus a BF16 low part and the product is hi*hi + hi*lo + lo*hi, so
// a score keeps ~16 significant bits even when its 128 terms cancel (a nearly
// orthogonal q and k); plain BF16 operands lose that precision.  A^kk = (I + R)^{-1} is formed by
// forward substitution in FP32 and stored with column j scaled by beta_j.
//
// Tokens past the end of a sequence (a ragged last chunk) are zero: q = k = 0,
// g = 0, beta = 0.  They then contribute nothing to any output or state.
//
// The kernel is persistent (two CTAs of 4 warp pairs per SM): every pair walks
// a strided list of (chunk, head) items through one shared-memory region
// (kda_prep_impl.cuh has the split of the work between the two warps): 2-D
// TMA loads of the item's q, k and g tiles, the item's work (the region turns
// into scratch once the inputs are in registers, then into the packet image),
// and one bulk copy of the packet to global memory, which must have read the
// region before the next item's loads overwrite it.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_prep_impl.cuh"

namespace kda {
namespace {

using namespace prep;

__global__ void __launch_bounds__(kPrepWarps * 32, 2)
    prep_kernel(PrepArgs a, const __grid_constant__ PrepMaps maps) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int pair = warp >> 1, hw = warp & 1, bid = 1 + pair;
    uint64_t* bar = pair_barrier(smem, pair, hw, lane, bid);
    run_items(a, maps, smem + pair * kPrepRegion, bar, bid, hw, lane,
              static_cast<int64_t>(blockIdx.x) * kPrepPairs + pair,
              static_cast<int64_t>(gridDim.x) * kPrepPairs, nullptr);
}

PFN_cuTensorMapEncodeTiled_v12000 prep_tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// [tokens][H * 128] view of a token-major tensor, boxes of 16 tokens x 128 channels.
cudaError_t encode_rows_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt,
                            int64_t esize, int64_t tokens, int64_t H) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = prep_tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H * kHeadDim),
                                static_cast<cuuint64_t>(tokens)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(H * kHeadDim * esize)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadDim), static_cast<cuuint32_t>(kChunk)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

namespace prep {
cudaError_t encode_maps(PrepMaps* maps, const void* q, const void* k, const float* g,
                        int64_t tokens, int64_t H) {
    cudaError_t e = encode_rows_map(&maps->q, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, tokens, H);
    if (e == cudaSuccess)
        e = encode_rows_map(&maps->k, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, tokens, H);
    if (e == cudaSuccess)
        e = encode_rows_map(&maps->g, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, tokens, H);
    return e;
}
}  // namespace prep

using namespace prep;

cudaError_t launch_prep(const void* q, const void* k, const float* g, const void* beta,
                        uint8_t* packets, const SeqGeometry& geo, int64_t H, float scale,
                        int* status, cudaStream_t stream, bool beta_logit) {
    if (geo.chunk_ub * H <= 0 || geo.tokens <= 0) return cudaSuccess;
    if (geo.tokens >= (int64_t(1) << 31)) return cudaErrorInvalidValue;   // TMA coordinates are int32
    PrepArgs a;
    if (!make_prep_args(&a, beta, packets, geo, H, scale, status, beta_logit))
        return cudaErrorInvalidValue;
    PrepMaps maps;
    cudaError_t e = encode_maps(&maps, q, k, g, geo.tokens, H);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static bool configured[64] = {};
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kPrepSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // Two CTAs per SM (persistent); fewer when there are fewer items than pairs.
    int64_t blocks = (a.n_chunk_heads + kPrepPairs - 1) / kPrepPairs;
    if (blocks > 2 * sms) blocks = 2 * sms;
    prep_kernel<<<static_cast<unsigned>(blocks), kPrepWarps * 32, kPrepSmemBytes, stream>>>(a, maps);
    return cudaGetLastError();
}

}  // namespace kda
