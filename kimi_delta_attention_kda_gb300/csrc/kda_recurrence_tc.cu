// kda_recurrence_tc.cu -- the KDA recurrence on the tcgen05 tensor cores
// (sm_103a), one CTA per (sequence, head).
//
// Same chunk equations as kda_recurrence.cu ("FlashKDA column split",
// section 1, with the error term as one contraction over the keys), in the
// untransposed orientation where the 128 value rows of the state are the MMA's
// M dimension:
//   U   = V (A^kk B)^T + S K'^T          K' = -(A^kk B)(K^start)^T (packet)
//   O   = S (s Q^start) + U (A^qk)^T
//   S  <- S D_{0:15} + U K^end
// Roles (320 threads):
//   warps 0-7  epilogue: warp w serves TMEM lanes 32 (w % 4) .. + 31, i.e. value
//              rows r, and the key half h = w / 4 of those rows; each thread
//              keeps S[r][64 h .. 64 h + 63] in FP32 registers for the whole
//              sequence, writes its half of the BF16 operand copies of S, U and
//              V^T into shared memory, and stores its half of O and the final
//              state.  Warps 0-3 write the first 64-key slab of S, warps 4-7
//              the second, so the MMAs on either slab can start separately.
//   warp 8     MMA issuer (one thread) and tensor-memory owner.
//   warp 9     producer: per chunk one bulk copy of the packet and one 2-D
//              tensor-map TMA load of the 16 x 128 V tile.
// Tensor memory: U accumulator (16 columns), O accumulator (16), S update (128).
// All operands are K-major with the 128-byte (K = 128) or 32-byte (K = 16)
// swizzle, the layouts the packet tiles already have.  The V^T operand of the
// next chunk is built as soon as the current U is converted, off the state's
// dependent chain.  Every wait is bounded and warp-uniform.
#include "kda_common.cuh"
#include "kda_launch.h"
#include "kda_tcgen05.cuh"

namespace kda {
namespace {

constexpr int kTcStages = 6;
constexpr uint32_t kTcVTileBytes = kChunk * kHeadDim * 2;                                  // 4096
constexpr uint32_t kTcStageBytes = ((kPacketBytes + kTcVTileBytes + 1023) / 1024) * 1024;   // 18432
constexpr uint32_t kTcOffSA = kTcStages * kTcStageBytes;      // S (BF16), 128 x 128, SW128
constexpr uint32_t kTcOffUA = kTcOffSA + 32768;                // U (FP16), 128 x 16, SW32
constexpr uint32_t kTcOffVT = kTcOffUA + 4096;                 // V^T (BF16), 128 x 16, SW32
constexpr uint32_t kTcOffBar = kTcOffVT + 4096;
constexpr int kTcNumBars = 2 * kTcStages + 7;
constexpr uint32_t kTcOffTmemPtr = kTcOffBar + kTcNumBars * 8;
constexpr uint32_t kTcSmemBytes = kTcOffTmemPtr + 16 + 1024;   // + alignment slack
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColU = 0, kColO = 16, kColS = 32;
constexpr int kEpiWarps = 8;
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

__device__ __forceinline__ void st_shared_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

// Row r, tokens 8 hf .. 8 hf + 7 of V^T (from the stage's [16][128] V tile)
// into the SW32 K-major V^T operand.
__device__ __forceinline__ void build_vt(const uint8_t* stage, uint8_t* vT, int r, int hf) {
    const uint16_t* vt = reinterpret_cast<const uint16_t*>(stage + kPacketBytes);
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        p[j] = static_cast<uint32_t>(vt[(8 * hf + 2 * j) * kHeadDim + r]) |
               (static_cast<uint32_t>(vt[(8 * hf + 2 * j + 1) * kHeadDim + r]) << 16);
    st_shared_v4(vT + sw32_off(r, hf), p[0], p[1], p[2], p[3]);
}

__global__ void __launch_bounds__(kTcThreads, 1)
    recurrence_tc_kernel(TcArgs a, const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTcOffBar);
    uint64_t* full = bars;
    uint64_t* empty = bars + kTcStages;
    uint64_t* bar_vt = bars + 2 * kTcStages + 0;   // V^T(c) written          (8 warps)
    uint64_t* bar_u = bars + 2 * kTcStages + 1;    // U(c) accumulated        (commit)
    uint64_t* bar_ua = bars + 2 * kTcStages + 2;   // U(c) in BF16 in smem    (8 warps)
    uint64_t* bar_sa0 = bars + 2 * kTcStages + 3;  // S keys 0-63 in smem     (warps 0-3)
    uint64_t* bar_sa1 = bars + 2 * kTcStages + 4;  // S keys 64-127 in smem   (warps 4-7)
    uint64_t* bar_s = bars + 2 * kTcStages + 5;    // S update and O done     (commit)
    uint64_t* bar_done = bars + 2 * kTcStages + 6; // every MMA done          (commit)
    uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + kTcOffTmemPtr);
    uint8_t* sA = smem + kTcOffSA;
    uint8_t* uA = smem + kTcOffUA;
    uint8_t* vT = smem + kTcOffVT;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n_slot = blockIdx.x / a.H;
    const int64_t h = blockIdx.x - n_slot * a.H;
    const int64_t n = a.geo.order ? a.geo.order[n_slot] : n_slot;   // longest-first (packed)

    int64_t c_begin, nch, tok0, seqlen;
    if (a.geo.cu_chunks) {
        if (!*a.geo.valid) return;
        c_begin = a.geo.cu_chunks[n];
        nch = a.geo.cu_chunks[n + 1] - c_begin;
        tok0 = a.geo.cu_seqlens[n];
        seqlen = a.geo.cu_seqlens[n + 1] - tok0;
    } else {
        c_begin = n * a.geo.chunks_per_seq;
        nch = a.geo.chunks_per_seq;
        tok0 = n * a.geo.tokens_per_seq;
        seqlen = a.geo.tokens_per_seq;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kEpiWarps);
        }
        mbar_init(bar_vt, kEpiWarps);
        mbar_init(bar_u, 1);
        mbar_init(bar_ua, kEpiWarps);
        mbar_init(bar_sa0, kEpiWarps / 2);
        mbar_init(bar_sa1, kEpiWarps / 2);
        mbar_init(bar_s, 1);
        mbar_init(bar_done, 1);
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tc::tmem_alloc(tmem_ptr, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_ptr;

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ producer
        uint32_t fill_parity = 0, filled = 0;
        bool ok = true;
        for (int64_t c = 0; c < nch && ok; ++c) {
            const int s = static_cast<int>(c % kTcStages);
            if (c >= kTcStages)
                ok = mbar_wait_warp_sleep(&empty[s], ((c / kTcStages) - 1) & 1, a.status);
            if (!ok) break;
            uint8_t* stage = smem + s * kTcStageBytes;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], kPacketBytes + kTcVTileBytes);
                bulk_g2s(stage, a.packets + ((c_begin + c) * a.H + h) * static_cast<int64_t>(kPacketBytes),
                         kPacketBytes, &full[s]);
                tma_load_2d(stage + kPacketBytes, &vmap, static_cast<int32_t>(h * kHeadDim),
                            static_cast<int32_t>(tok0 + kChunk * c), &full[s]);
            }
            __syncwarp();
            fill_parity ^= (filled >> s & 1u) << s;
            filled |= 1u << s;
        }
        if (!ok)
            for (int s = 0; s < kTcStages; ++s)
                if (filled >> s & 1u) mbar_wait_bounded(&full[s], (fill_parity >> s) & 1u, a.status);
    } else if (warp == kMmaWarp) {
        // ---------------------------------------------------------- MMA issuer
        const uint32_t id16 = tc::idesc_bf16(128, 16);
        // U is FP16 in shared memory, and so are A^qk and K^end (see mma_f16).
        const uint32_t ih16 = tc::idesc_f16(128, 16), ih128 = tc::idesc_f16(128, 128);
        const uint64_t dVT = tc::smem_desc(vT, 256, tc::kSwizzle32B);
        const uint64_t dUA = tc::smem_desc(uA, 256, tc::kSwizzle32B);
        for (int64_t c = 0; c < nch; ++c) {
            const int s = static_cast<int>(c % kTcStages);
            const uint32_t ph = static_cast<uint32_t>(c & 1);
            const uint8_t* stage = smem + s * kTcStageBytes;
            if (!mbar_wait_warp(&full[s], (c / kTcStages) & 1, a.status)) break;
            if (!mbar_wait_warp(bar_vt, ph, a.status)) break;
            tc::fence_after_sync();
            // U = V (A^kk B)^T: does not depend on the state.
            if (lane == 0)
                tc::mma_bf16(tmem + kColU, dVT, tc::smem_desc(stage + kOffAKB, 256, tc::kSwizzle32B),
                             id16, 0);
            __syncwarp();
            // ... + S K'^T, keys 0-63 then 64-127 as each slab of S arrives.
            if (!mbar_wait_warp(bar_sa0, ph, a.status)) break;
            tc::fence_after_sync();
            if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16(tmem + kColU, tc::smem_desc(sA + 32 * kk, 1024, tc::kSwizzle128B),
                                 tc::smem_desc(stage + kOffKS + 32 * kk, 1024, tc::kSwizzle128B), id16, 1);
            }
            __syncwarp();
            if (!mbar_wait_warp(bar_sa1, ph, a.status)) break;
            tc::fence_after_sync();
            if (lane == 0) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16(tmem + kColU,
                                 tc::smem_desc(sA + 16384 + 32 * kk, 1024, tc::kSwizzle128B),
                                 tc::smem_desc(stage + kOffKS + 2048 + 32 * kk, 1024, tc::kSwizzle128B),
                                 id16, 1);
                tc::commit(bar_u);
                // O = S (s Q^start), off the state chain.
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    tc::mma_bf16(tmem + kColO,
                                 tc::smem_desc(sA + (kk >> 2) * 16384 + 32 * (kk & 3), 1024, tc::kSwizzle128B),
                                 tc::smem_desc(stage + kOffQS + (kk >> 2) * 2048 + 32 * (kk & 3), 1024,
                                               tc::kSwizzle128B),
                                 id16, kk > 0 ? 1u : 0u);
            }
            __syncwarp();
            if (!mbar_wait_warp(bar_ua, ph, a.status)) break;
            tc::fence_after_sync();
            if (lane == 0) {
                // O += U (A^qk)^T;  S update = U K^end
                tc::mma_bf16(tmem + kColO, dUA, tc::smem_desc(stage + kOffAQK, 256, tc::kSwizzle32B),
                             ih16, 1);
                tc::mma_bf16(tmem + kColS, dUA, tc::smem_desc(stage + kOffKE, 256, tc::kSwizzle32B),
                             ih128, 0);
                tc::commit(bar_s);
            }
            __syncwarp();
        }
        // Every MMA issued must be complete before tensor memory is released.
        if (lane == 0) tc::commit(bar_done);
        __syncwarp();
        mbar_wait_warp(bar_done, 0, a.status);
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3, hf = warp >> 2;
        const int r = 32 * quarter + lane;   // value row, TMEM lane
        const uint32_t trow = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
        const int64_t state_row = ((n * a.H + h) * kHeadDim + r) * kHeadDim + 64 * hf;
        uint64_t* bar_sa = hf ? bar_sa1 : bar_sa0;
        float S[64];   // keys 64 hf + i
        if (a.init_state) {
            const uint4* src = reinterpret_cast<const uint4*>(a.init_state + state_row);
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const uint4 w = src[x];
                S[8 * x + 0] = bf16_lo(w.x); S[8 * x + 1] = bf16_hi(w.x);
                S[8 * x + 2] = bf16_lo(w.y); S[8 * x + 3] = bf16_hi(w.y);
                S[8 * x + 4] = bf16_lo(w.z); S[8 * x + 5] = bf16_hi(w.z);
                S[8 * x + 6] = bf16_lo(w.w); S[8 * x + 7] = bf16_hi(w.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) S[i] = 0.f;
        }
        // BF16 operand copy of this half row: 8-key groups at SW128 positions.
#pragma unroll
        for (int x = 0; x < 8; ++x)
            st_shared_v4(sA + sw128_off(128, r, 8 * hf + x), pack_bf16(S[8 * x + 0], S[8 * x + 1]),
                         pack_bf16(S[8 * x + 2], S[8 * x + 3]), pack_bf16(S[8 * x + 4], S[8 * x + 5]),
                         pack_bf16(S[8 * x + 6], S[8 * x + 7]));
        fence_proxy_async_smem();
        __syncwarp();
        mbar_arrive_if(bar_sa, lane == 0);

        bool ok = true;
        if (nch > 0) {
            ok = mbar_wait_warp(&full[0], 0, a.status);
            if (ok) {
                build_vt(smem, vT, r, hf);
                fence_proxy_async_smem();
                __syncwarp();
                mbar_arrive_if(bar_vt, lane == 0);
            }
        }
        for (int64_t c = 0; c < nch && ok; ++c) {
            const int s = static_cast<int>(c % kTcStages);
            const uint32_t ph = static_cast<uint32_t>(c & 1);
            const uint8_t* stage = smem + s * kTcStageBytes;
            int64_t len = seqlen - kChunk * c;
            if (len > kChunk) len = kChunk;

            // U(c): accumulator -> BF16 operand (tokens 8 hf .. 8 hf + 7).
            if (!mbar_wait_warp(bar_u, ph, a.status)) { ok = false; break; }
            tc::fence_after_sync();
            {
                uint32_t u[8];
                tc::ld_x8(trow + kColU + 8 * hf, u);
                tc::wait_ld();
                st_shared_v4(uA + sw32_off(r, hf),
                             pack_f16_sat(__uint_as_float(u[0]), __uint_as_float(u[1])),
                             pack_f16_sat(__uint_as_float(u[2]), __uint_as_float(u[3])),
                             pack_f16_sat(__uint_as_float(u[4]), __uint_as_float(u[5])),
                             pack_f16_sat(__uint_as_float(u[6]), __uint_as_float(u[7])));
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            mbar_arrive_if(bar_ua, lane == 0);

            // V^T of the next chunk, while the MMA warp works on this one
            // (this chunk's V^T has been consumed: its MMA completed before U).
            if (c + 1 < nch) {
                const int s1 = static_cast<int>((c + 1) % kTcStages);
                if (!mbar_wait_warp(&full[s1], ((c + 1) / kTcStages) & 1, a.status)) { ok = false; break; }
                build_vt(smem + s1 * kTcStageBytes, vT, r, hf);
                fence_proxy_async_smem();
                __syncwarp();
                mbar_arrive_if(bar_vt, lane == 0);
            }

            // S(c+1) = S D + update (this half row), O(c).
            if (!mbar_wait_warp(bar_s, ph, a.status)) { ok = false; break; }
            tc::fence_after_sync();
            uint32_t o[8];
            tc::ld_x8(trow + kColO + 8 * hf, o);
            const float4* dq = reinterpret_cast<const float4*>(stage + kOffD);
#pragma unroll
            for (int qh = 0; qh < 2; ++qh) {
                const int q = 2 * hf + qh;   // keys 32 q .. 32 q + 31
                uint32_t upd[32];
                tc::ld_x32(trow + kColS + 32 * q, upd);
                tc::wait_ld();
                // The packet's D is permuted: float4 4*r7 + q holds the factors
                // of keys 32q + r7, 32q + r7 + 8, 32q + r7 + 16 and 32q + r7 + 24.
#pragma unroll
                for (int r7 = 0; r7 < 8; ++r7) {
                    const float4 d = dq[4 * r7 + q];
                    const int k0 = 32 * qh + r7;
                    S[k0] = fmaf(S[k0], d.x, __uint_as_float(upd[r7]));
                    S[k0 + 8] = fmaf(S[k0 + 8], d.y, __uint_as_float(upd[r7 + 8]));
                    S[k0 + 16] = fmaf(S[k0 + 16], d.z, __uint_as_float(upd[r7 + 16]));
                    S[k0 + 24] = fmaf(S[k0 + 24], d.w, __uint_as_float(upd[r7 + 24]));
                }
#pragma unroll
                for (int xx = 0; xx < 4; ++xx) {
                    const int x = 4 * qh + xx;   // local 8-key group
                    st_shared_v4(sA + sw128_off(128, r, 8 * hf + x), pack_bf16(S[8 * x + 0], S[8 * x + 1]),
                                 pack_bf16(S[8 * x + 2], S[8 * x + 3]),
                                 pack_bf16(S[8 * x + 4], S[8 * x + 5]),
                                 pack_bf16(S[8 * x + 6], S[8 * x + 7]));
                }
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            __syncwarp();
            mbar_arrive_if(bar_sa, lane == 0);

            // O rows of this chunk: tokens 8 hf + i, value r.
            __nv_bfloat16* orow = a.out + ((tok0 + kChunk * c + 8 * hf) * a.H + h) * kHeadDim + r;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (8 * hf + i < len) orow[i * a.H * kHeadDim] = __float2bfloat16_rn(__uint_as_float(o[i]));
            // This stage's V tile and D have been read.
            stage_release(&empty[s], lane);
        }
        if (ok && a.final_state) {
            uint4* dst = reinterpret_cast<uint4*>(a.final_state + state_row);
#pragma unroll
            for (int x = 0; x < 8; ++x)
                dst[x] = make_uint4(pack_bf16(S[8 * x + 0], S[8 * x + 1]), pack_bf16(S[8 * x + 2], S[8 * x + 3]),
                                    pack_bf16(S[8 * x + 4], S[8 * x + 5]), pack_bf16(S[8 * x + 6], S[8 * x + 7]));
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
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
