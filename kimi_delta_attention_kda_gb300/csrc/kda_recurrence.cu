// kda_recurrence.cu -- the serial-over-chunks KDA recurrence (sm_103a).
//
// For every chunk c of one (sequence, head), in the transposed layout of
// "FlashKDA column split", section 3.1 (one row per token, one column per
// value channel):
//   U^T   = (A^kk B)(V^T - (K^start)^T S^T) = (A^kk B) V^T + K' S^T
//   O^T   = s (Q^start)^T S^T + A^qk U^T
//   S^T  <- D_{0:15} S^T + (K^end)^T U^T
// with K' = -(A^kk B)(K^start)^T formed by the preparation kernel, so that the
// state enters the chunk's error term through a single contraction.
// Value columns are independent recurrences that share the per-chunk inputs
// (section 3.1), so the 128 value columns of a head are split over `nsplit`
// CTAs and, inside a CTA, over warps of 8 columns each.  Each warp keeps its
// 128 x 8 slice of S^T in registers in FP32 for the whole sequence (section
// 3.3); the BF16 copy used as an MMA operand is refreshed every chunk.  The
// accumulator -> operand layout change is an 8 x 8 transpose in registers
// (movmatrix).  No CTA ever waits on another CTA.
//
// A producer warp streams, per chunk, the packet (kda_common.cuh; one 1-D bulk
// copy) and the CTA's 16 x (value columns) tile of V (one 2-D tensor-map TMA
// load) into a ring of shared-memory stages, completing on mbarriers; every
// wait is bounded (kda_common.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_common.cuh"
#include "kda_segmap.cuh"
#include "kda_launch.h"
#include "kda_rec_impl.cuh"

namespace kda {
namespace {

using namespace rec;

template <int NW>
struct RecLayout {
    static constexpr int kCols = 8 * NW;                        // value columns per CTA
    static constexpr int kStages = NW <= 4 ? 8 : (NW <= 8 ? 6 : 4);
    static constexpr uint32_t kVRowBytes = kCols * 2;           // one token row of V
    static constexpr uint32_t kStageBytes =
        ((kPacketBytes + kChunk * kVRowBytes + 1023) / 1024) * 1024;
    static constexpr uint32_t kBarOff = kStages * kStageBytes;
    static constexpr uint32_t kSmemBytes = kBarOff + 2 * kStages * 8 + 1024;  // + align slack
    // With few warps per CTA every register is available, so each chunk's
    // operand fragments are loaded in one burst ahead of use.
    static constexpr bool kPrefetch = NW <= 4;
};

// Operand fragments of one chunk for one warp (m16n8k16 A-operand layout).
struct ChunkFrags {
    uint32_t ks[8][4];   // K' = -(A^kk B)(K^start)^T, k-steps over keys
    uint32_t qs[8][4];   // s (Q^start)^T
    uint32_t ke[8][4];   // (K^end)^T, one 16-key tile each
    uint32_t akb[4];     // A^kk B
    uint32_t aqk[4];     // A^qk
    float4 d[4];         // D for keys 16 m + g8 and 16 m + g8 + 8, m = 0..7
    uint32_t vb[2];      // V^T as a B operand (k = token, n = this warp's 8 values)
};

__device__ __forceinline__ void load_frags(const uint8_t* stage, uint32_t vrow_bytes, int warp,
                                           int lane, ChunkFrags& f) {
    const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t hiA = lane >> 4;
    const int g8 = lane >> 2;
    const uint32_t sKS = smem_u32(stage + kOffKS);
    const uint32_t sQS = smem_u32(stage + kOffQS);
    const uint32_t sKE = smem_u32(stage + kOffKE);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) ldsm_x4(f.ks[kk], sKS + sw128_off(16, rowA, 2 * kk + hiA));
    ldsm_x4(f.akb, smem_u32(stage + kOffAKB + sw32_off(rowA, hiA)));
    // V tile rows are tokens; lanes 0-7 address tokens 0-7, lanes 8-15 tokens 8-15.
    const uint8_t* sV = stage + kPacketBytes + (lane & 15) * vrow_bytes + 16 * warp;
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(f.vb[0]), "=r"(f.vb[1])
                 : "r"(smem_u32(sV)));
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) ldsm_x4(f.qs[kk], sQS + sw128_off(16, rowA, 2 * kk + hiA));
    const float4* dp = reinterpret_cast<const float4*>(stage + kOffD) + 4 * g8;
#pragma unroll
    for (int j = 0; j < 4; ++j) f.d[j] = dp[j];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) ldsm_x4(f.ke[mt], sKE + sw32_off(16 * mt + rowA, hiA));
    ldsm_x4(f.aqk, smem_u32(stage + kOffAQK + sw32_off(rowA, hiA)));
}

// The same loads in three groups, in the order a chunk step needs them: the
// error-term operands, K^end, then the output operands and D.
__device__ __forceinline__ void load_frags_u(const uint8_t* stage, uint32_t vrow_bytes, int warp,
                                             int lane, ChunkFrags& f) {
    const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t hiA = lane >> 4;
    const uint32_t sKS = smem_u32(stage + kOffKS);
    ldsm_x4(f.akb, smem_u32(stage + kOffAKB + sw32_off(rowA, hiA)));
    const uint8_t* sV = stage + kPacketBytes + (lane & 15) * vrow_bytes + 16 * warp;
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(f.vb[0]), "=r"(f.vb[1])
                 : "r"(smem_u32(sV)));
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) ldsm_x4(f.ks[kk], sKS + sw128_off(16, rowA, 2 * kk + hiA));
}
__device__ __forceinline__ void load_frags_ke(const uint8_t* stage, int lane, ChunkFrags& f) {
    const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t hiA = lane >> 4;
    const uint32_t sKE = smem_u32(stage + kOffKE);
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) ldsm_x4(f.ke[mt], sKE + sw32_off(16 * mt + rowA, hiA));
}
__device__ __forceinline__ void load_frags_o(const uint8_t* stage, int lane, ChunkFrags& f) {
    const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t hiA = lane >> 4;
    const int g8 = lane >> 2;
    const uint32_t sQS = smem_u32(stage + kOffQS);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) ldsm_x4(f.qs[kk], sQS + sw128_off(16, rowA, 2 * kk + hiA));
    ldsm_x4(f.aqk, smem_u32(stage + kOffAQK + sw32_off(rowA, hiA)));
    const float4* dp = reinterpret_cast<const float4*>(stage + kOffD) + 4 * g8;
#pragma unroll
    for (int j = 0; j < 4; ++j) f.d[j] = dp[j];
}

// One chunk for one warp: advances Sf (FP32 S^T slice) and returns O^T in o.
// Sb holds the BF16 B-operand fragments of the incoming state.
//   U^T = (A^kk B) V^T + K' S^T          (K' = -(A^kk B)(K^start)^T, from the packet)
//   O^T = s (Q^start)^T S^T + A^qk U^T
//   S^T <- D S^T + (K^end)^T U^T
// Token rows past the end of the sequence meet zero columns of A^kk B (beta
// is zero there), so they need no masking.
__device__ __forceinline__ void chunk_step(const ChunkFrags& f, float (&Sf)[8][4],
                                           const uint32_t (&Sb)[8][2], float (&o)[4]) {
    // (A^kk B) V^T does not depend on the state: it seeds the accumulator.
    float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
    mma_bf16(u0, f.akb, f.vb, u0);
    // U^T += K' S^T over the 128 keys, in two accumulators.
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) {
        mma_bf16(u0, f.ks[kk], Sb[kk], u0);
        mma_bf16(u1, f.ks[kk + 1], Sb[kk + 1], u1);
    }
    // D S^T, in place (the BF16 copy of the old state is already in Sb).
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const float d0 = dsel(f.d[mt >> 1], 2 * (mt & 1));
        const float d1 = dsel(f.d[mt >> 1], 2 * (mt & 1) + 1);
        mul2(Sf[mt][0], Sf[mt][1], d0);
        mul2(Sf[mt][2], Sf[mt][3], d1);
    }
    uint32_t Ub[2];   // U^T as the FP16 B operand of the update and the output term
    Ub[0] = movm_t(pack_f16_sat(u0[0] + u1[0], u0[1] + u1[1]));
    Ub[1] = movm_t(pack_f16_sat(u0[2] + u1[2], u0[3] + u1[3]));
    // S^T <- D S^T + (K^end)^T U^T.
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) mma_f16(Sf[mt], f.ke[mt], Ub, Sf[mt]);
    // P^T = s (Q^start)^T S^T, off the state chain.
    float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; kk += 2) {
        mma_bf16(p0, f.qs[kk], Sb[kk], p0);
        mma_bf16(p1, f.qs[kk + 1], Sb[kk + 1], p1);
    }
    // O^T = P^T + A^qk U^T.
    float pin[4] = {p0[0] + p1[0], p0[1] + p1[1], p0[2] + p1[2], p0[3] + p1[3]};
    mma_f16(o, f.aqk, Ub, pin);
}

// A warp's slice of a state (all 128 keys of 8 value columns), BF16, into a
// [128 value][128 key] state at dst.
__device__ __forceinline__ void narrow_store_state(__nv_bfloat16* dst, const float (&Sf)[8][4],
                                                   int vcol, int g8, int t4) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        const int key = 16 * mt + g8;
        const int val = vcol + 2 * t4;
        dst[(int64_t)val * kHeadDim + key] = __float2bfloat16_rn(Sf[mt][0]);
        dst[(int64_t)(val + 1) * kHeadDim + key] = __float2bfloat16_rn(Sf[mt][1]);
        dst[(int64_t)val * kHeadDim + key + 8] = __float2bfloat16_rn(Sf[mt][2]);
        dst[(int64_t)(val + 1) * kHeadDim + key + 8] = __float2bfloat16_rn(Sf[mt][3]);
    }
}

template <int NW>
__global__ void __launch_bounds__((NW + 1) * 32)
    recurrence_kernel(RecArgs a, const __grid_constant__ CUtensorMap vmap) {
    using L = RecLayout<NW>;
    constexpr int kStages = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the stages.
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* empty = full + kStages;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nh = blockIdx.x / a.nsplit;
    const int split = blockIdx.x - nh * a.nsplit;
    const int64_t n_slot = nh / a.H;
    const int64_t h = nh - n_slot * a.H;
    if (n_slot < a.geo.first_slot) return;   // runs in the other launch
    const int64_t n = a.geo.order ? a.geo.order[n_slot] : n_slot;   // longest-first (packed)
    const int v0 = split * L::kCols;

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
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------------------------------------ producer
        uint32_t fill_parity = 0;   // bit s: parity of the latest fill of stage s
        uint32_t filled = 0;        // bit s: stage s has been filled at least once
        bool ok = true;
        for (int64_t c = 0; c < nch && ok; ++c) {
            const int s = static_cast<int>(c % kStages);
            if (c >= kStages)
                ok = mbar_wait_warp_sleep(&empty[s], ((c / kStages) - 1) & 1, a.status);
            if (!ok) break;
            uint8_t* stage = smem + s * L::kStageBytes;
            if (lane == 0) {
                // The V box always lands whole: rows past the last token are
                // zero-filled, rows past this sequence are masked by the consumer.
                mbar_arrive_expect_tx(&full[s], kPacketBytes + kChunk * L::kVRowBytes);
                bulk_g2s(stage, a.packets + ((c_begin + c) * a.H + h) * static_cast<int64_t>(kPacketBytes),
                         kPacketBytes, &full[s]);
                tma_load_2d(stage + kPacketBytes, &vmap, static_cast<int32_t>(h * kHeadDim + v0),
                            static_cast<int32_t>(tok0 + kChunk * c), &full[s]);
            }
            __syncwarp();
            fill_parity ^= (filled >> s & 1u) << s;   // flip after the first fill
            filled |= 1u << s;
        }
        if (!ok) {
            // Let every copy already issued land before the CTA can exit.
            for (int s = 0; s < kStages; ++s)
                if (filled >> s & 1u) mbar_wait_bounded(&full[s], (fill_parity >> s) & 1u, a.status);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g8 = lane >> 2;     // fragment row group
    const int t4 = lane & 3;      // fragment column pair
    const int vcol = v0 + 8 * warp;   // first value column of this warp
    const int64_t state_base = (n * a.H + h) * kHeadDim * kHeadDim;

    // S^T slice: 8 key tiles of 16 rows x 8 value columns, FP32 accumulator layout.
    float Sf[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        if (a.init_state) {
            const __nv_bfloat16* src = a.init_state + state_base;
            const int key = 16 * mt + g8;
            const int val = vcol + 2 * t4;
            Sf[mt][0] = __bfloat162float(src[(int64_t)val * kHeadDim + key]);
            Sf[mt][1] = __bfloat162float(src[(int64_t)(val + 1) * kHeadDim + key]);
            Sf[mt][2] = __bfloat162float(src[(int64_t)val * kHeadDim + key + 8]);
            Sf[mt][3] = __bfloat162float(src[(int64_t)(val + 1) * kHeadDim + key + 8]);
        } else {
            Sf[mt][0] = Sf[mt][1] = Sf[mt][2] = Sf[mt][3] = 0.f;
        }
    }
    // BF16 B-operand fragments of S^T for k-step kk (keys 16kk..16kk+15).
    uint32_t Sb[8][2];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
        Sb[mt][0] = movm_t(pack_bf16(Sf[mt][0], Sf[mt][1]));
        Sb[mt][1] = movm_t(pack_bf16(Sf[mt][2], Sf[mt][3]));
    }

    bool ok = true;
    ChunkFrags f;
    int64_t ck_next = 0;   // next chunk whose incoming state is a checkpoint
    if (L::kPrefetch) {
        // Rolling prefetch: each group of chunk c+1's fragments is loaded as
        // soon as chunk c has issued its last use of that group, so the loads
        // are in flight behind the rest of chunk c.
        if (nch > 0) {
            ok = mbar_wait_warp(&full[0], 0, a.status);
            if (ok) load_frags(smem, L::kVRowBytes, warp, lane, f);
        }
        for (int64_t c = 0; c < nch && ok; ++c) {
            if (a.ck.states && c == ck_next) {
                ck_next += a.ck.every;
                __nv_bfloat16* dst = checkpoint_dst(a, n, h, c / a.ck.every);
                if (dst) narrow_store_state(dst, Sf, vcol, g8, t4);
            }
            const int s = static_cast<int>(c % kStages);
            const bool has_next = c + 1 < nch;
            const int s1 = static_cast<int>((c + 1) % kStages);
            const uint32_t par1 = static_cast<uint32_t>(((c + 1) / kStages) & 1);
            const uint8_t* stage1 = smem + s1 * L::kStageBytes;
            // Probe the next stage now; the answer is needed only after U.
            bool next_ready = has_next && mbar_try_wait(&full[s1], par1);
            int64_t len = seqlen - kChunk * c;
            if (len > kChunk) len = kChunk;

            float u0[4] = {0.f, 0.f, 0.f, 0.f}, u1[4] = {0.f, 0.f, 0.f, 0.f};
            mma_bf16(u0, f.akb, f.vb, u0);
#pragma unroll
            for (int kk = 0; kk < 8; kk += 2) {
                mma_bf16(u0, f.ks[kk], Sb[kk], u0);
                mma_bf16(u1, f.ks[kk + 1], Sb[kk + 1], u1);
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                const float d0 = dsel(f.d[mt >> 1], 2 * (mt & 1));
                const float d1 = dsel(f.d[mt >> 1], 2 * (mt & 1) + 1);
                mul2(Sf[mt][0], Sf[mt][1], d0);
                mul2(Sf[mt][2], Sf[mt][3], d1);
            }
            // Every read of this chunk's stage was issued during the previous
            // chunk (or before the loop): hand it back before the next
            // chunk's loads, so that the proxy fence finds nothing in flight.
            stage_release(&empty[s], lane);
            if (has_next) {
                if (!__all_sync(0xffffffffu, next_ready))
                    next_ready = mbar_wait_warp(&full[s1], par1, a.status);
                if (next_ready)
                    load_frags_u(stage1, L::kVRowBytes, warp, lane, f);
                else
                    ok = false;
            }
            uint32_t Ub[2];   // FP16 (see mma_f16)
            Ub[0] = movm_t(pack_f16_sat(u0[0] + u1[0], u0[1] + u1[1]));
            Ub[1] = movm_t(pack_f16_sat(u0[2] + u1[2], u0[3] + u1[3]));
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) mma_f16(Sf[mt], f.ke[mt], Ub, Sf[mt]);
            if (has_next && ok) load_frags_ke(stage1, lane, f);
            float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < 8; kk += 2) {
                mma_bf16(p0, f.qs[kk], Sb[kk], p0);
                mma_bf16(p1, f.qs[kk + 1], Sb[kk + 1], p1);
            }
            float o[4];
            {
                float pin[4] = {p0[0] + p1[0], p0[1] + p1[1], p0[2] + p1[2], p0[3] + p1[3]};
                mma_f16(o, f.aqk, Ub, pin);
            }
            if (has_next && ok) load_frags_o(stage1, lane, f);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                Sb[mt][0] = movm_t(pack_bf16(Sf[mt][0], Sf[mt][1]));
                Sb[mt][1] = movm_t(pack_bf16(Sf[mt][2], Sf[mt][3]));
            }
            __nv_bfloat16* orow = a.out + ((tok0 + kChunk * c + g8) * a.H + h) * kHeadDim + vcol + 2 * t4;
            st_global_u32_if(orow, pack_bf16(o[0], o[1]), g8 < len);
            st_global_u32_if(orow + 8 * a.H * kHeadDim, pack_bf16(o[2], o[3]), g8 + 8 < len);
        }
    } else {
        for (int64_t c = 0; c < nch; ++c) {
            if (a.ck.states && c == ck_next) {
                ck_next += a.ck.every;
                __nv_bfloat16* dst = checkpoint_dst(a, n, h, c / a.ck.every);
                if (dst) narrow_store_state(dst, Sf, vcol, g8, t4);
            }
            const int s = static_cast<int>(c % kStages);
            const uint8_t* stage = smem + s * L::kStageBytes;
            if (!mbar_wait_warp(&full[s], (c / kStages) & 1, a.status)) {
                ok = false;
                break;
            }
            load_frags(stage, L::kVRowBytes, warp, lane, f);
            int64_t len = seqlen - kChunk * c;
            if (len > kChunk) len = kChunk;

            float o[4];
            chunk_step(f, Sf, Sb, o);

            // BF16 operand copy of the new state: first, since the next chunk's
            // chain starts from it (warps issue in order).
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
                Sb[mt][0] = movm_t(pack_bf16(Sf[mt][0], Sf[mt][1]));
                Sb[mt][1] = movm_t(pack_bf16(Sf[mt][2], Sf[mt][3]));
            }
            // Every read of this stage is done: hand it back to the producer.
            stage_release(&empty[s], lane);

            // Store O (tokens g8 and g8 + 8, values vcol + 2 t4 .. + 1), predicated.
            __nv_bfloat16* orow = a.out + ((tok0 + kChunk * c + g8) * a.H + h) * kHeadDim + vcol + 2 * t4;
            st_global_u32_if(orow, pack_bf16(o[0], o[1]), g8 < len);
            st_global_u32_if(orow + 8 * a.H * kHeadDim, pack_bf16(o[2], o[3]), g8 + 8 < len);
        }
    }

    if (ok && a.final_state) narrow_store_state(a.final_state + state_base, Sf, vcol, g8, t4);
}

// ---------------------------------------------------------------------------
// Quad-width variant for one CTA per head (kda_rec_impl.cuh, wide_consume
// with four n-tiles per warp): 4 consumer warps of 32 value columns and a
// producer warp.
// ---------------------------------------------------------------------------
constexpr int kQuadWarps = 4;
constexpr int kQuadStages = 8;
constexpr uint32_t kQuadBarOff = kQuadStages * kWideStageBytes;
constexpr uint32_t kQuadSmemBytes = kQuadBarOff + 2 * kQuadStages * 8 + 1024;

template <int kMode>
__global__ void __launch_bounds__((kQuadWarps + 1) * 32, 1)
    recurrence_quad_kernel(RecArgs a, const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQuadBarOff);
    uint64_t* empty = full + kQuadStages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n_slot = blockIdx.x / a.H;
    const int64_t h = blockIdx.x - n_slot * a.H;
    if (n_slot < a.geo.first_slot) return;   // runs in the other launch
    const int64_t n = a.geo.order ? a.geo.order[n_slot] : n_slot;   // longest-first (packed)

    int64_t c_begin, nch, tok0, seqlen;
    if (!seq_span(a.geo, n, c_begin, nch, tok0, seqlen)) return;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQuadStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kQuadWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == kQuadWarps)
        wide_produce<kQuadStages>(a, &vmap, smem, full, empty, lane, h, c_begin, nch, tok0, nullptr);
    else
        wide_consume<4, kQuadStages, kMode == kWideCkpt>(a, smem, full, empty, warp, lane, n, h,
                                                         c_begin, nch, tok0, seqlen);
}

template <int kMode>
cudaError_t launch_quad_t(const RecArgs& a, int64_t blocks, cudaStream_t stream) {
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(recurrence_quad_kernel<kMode>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kQuadSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    CUtensorMap vmap;
    alignas(64) static const char kZero[16] = {};
    const void* vbase = a.v ? static_cast<const void*>(a.v) : static_cast<const void*>(kZero);
    cudaError_t e = encode_v_map_sw128(&vmap, vbase, a.geo.tokens, a.H);
    if (e != cudaSuccess) return e;
    recurrence_quad_kernel<kMode>
        <<<static_cast<unsigned>(blocks), (kQuadWarps + 1) * 32, kQuadSmemBytes, stream>>>(a, vmap);
    return cudaGetLastError();
}

cudaError_t launch_quad(const RecArgs& a, int64_t blocks, cudaStream_t stream) {
    return a.ck.states ? launch_quad_t<kWideCkpt>(a, blocks, stream)
                       : launch_quad_t<kWidePlain>(a, blocks, stream);
}

// ---------------------------------------------------------------------------
// Transition pass of the segmented scan.  For segment n of the batch and head
// h: the state the segment's chunks lead to from a zero state (Z, warps 0-3)
// and from the identity with V taken as zero (F, warps 4-7; S -> S F is the
// map of those chunks on the incoming state).  Both halves read the same
// packets; each warp holds 32 value columns of its state over all 128 keys as
// in the quad kernel and runs the U^T and S^T updates only (no P^T, no O).
// Under the state's registers eight warps leave no room for a producer warp,
// so warp 0 refills each stage once every warp has released it.  Z and F
// leave in the segment chain's fragment order.
// ---------------------------------------------------------------------------
constexpr int kTransWarps = 2 * kQuadWarps;

__global__ void __launch_bounds__(kTransWarps * 32, 1)
    transition_kernel(RecArgs a, const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kQuadBarOff);
    uint64_t* empty = full + kQuadStages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t n = blockIdx.x / a.H;
    const int64_t h = blockIdx.x - n * a.H;
    int64_t c_begin, nch, tok0, seqlen;
    if (!seq_span(a.geo, n, c_begin, nch, tok0, seqlen)) return;
    const bool ident = warp >= kQuadWarps;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kQuadStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kTransWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // Chunk c's packet and V tile into its stage (warp 0, lane 0).
    auto load = [&](int64_t c) {
        const int s = static_cast<int>(c % kQuadStages);
        uint8_t* stage = smem + s * kWideStageBytes;
        mbar_arrive_expect_tx(&full[s], kPacketBytes + kChunk * kWideVRowBytes);
        bulk_g2s(stage, a.packets + ((c_begin + c) * a.H + h) * static_cast<int64_t>(kPacketBytes),
                 kPacketBytes, &full[s]);
        wide_load_v(stage, &vmap, h, tok0 + kChunk * c, &full[s]);
    };
    int64_t issued = nch < kQuadStages ? nch : kQuadStages;
    if (warp == 0 && lane == 0)
        for (int64_t c = 0; c < issued; ++c) load(c);

    const int g8 = lane >> 2, t4 = lane & 3;
    const int vcol = 32 * (warp % kQuadWarps);
    const int64_t state_base = (n * a.H + h) * kHeadDim * kHeadDim;
    const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t hiA = lane >> 4;

    // Zero, or the identity (S[v][key] = 1 where v == key).
    float Sf[8][4][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int key = 16 * mt + g8;
            const int val = vcol + 8 * nt + 2 * t4;
            Sf[mt][nt][0] = ident && val == key ? 1.f : 0.f;
            Sf[mt][nt][1] = ident && val + 1 == key ? 1.f : 0.f;
            Sf[mt][nt][2] = ident && val == key + 8 ? 1.f : 0.f;
            Sf[mt][nt][3] = ident && val + 1 == key + 8 ? 1.f : 0.f;
        }

    bool ok = true;
    int64_t c = 0;
    for (; c < nch; ++c) {
        const int s = static_cast<int>(c % kQuadStages);
        if (!mbar_wait_warp(&full[s], (c / kQuadStages) & 1, a.status)) {
            ok = false;
            break;
        }
        const uint8_t* stage = smem + s * kWideStageBytes;
        const uint32_t sKS = smem_u32(stage + kOffKS);
        const uint32_t sKE = smem_u32(stage + kOffKE);

        // U^T = (A^kk B) V^T (zero-start half only) + K' S^T.
        float u[2][4][4];
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) u[x][nt][j] = 0.f;
        if (!ident) {
            uint32_t akb[4];
            ldsm_x4(akb, smem_u32(stage + kOffAKB + sw32_off(rowA, hiA)));
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
                uint32_t vb[4];
                const uint8_t* sV = stage + kWideVOff +
                                    sw128_off(kChunk, lane & 15, (vcol + 16 * hp) / 8 + (lane >> 4));
                asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                             : "=r"(vb[0]), "=r"(vb[1]), "=r"(vb[2]), "=r"(vb[3])
                             : "r"(smem_u32(sV)));
                mma_bf16(u[0][2 * hp], akb, vb, u[0][2 * hp]);
                mma_bf16(u[0][2 * hp + 1], akb, vb + 2, u[0][2 * hp + 1]);
            }
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t kf[4];
            ldsm_x4(kf, sKS + sw128_off(16, rowA, 2 * kk + hiA));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const uint32_t sb[2] = {movm_t(pack_bf16(Sf[kk][nt][0], Sf[kk][nt][1])),
                                        movm_t(pack_bf16(Sf[kk][nt][2], Sf[kk][nt][3]))};
                mma_bf16(u[kk & 1][nt], kf, sb, u[kk & 1][nt]);
            }
        }
        // D S^T in place.
        {
            const float4* dp = reinterpret_cast<const float4*>(stage + kOffD) + 4 * g8;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 d = dp[j];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    mul2(Sf[2 * j][nt][0], Sf[2 * j][nt][1], d.x);
                    mul2(Sf[2 * j][nt][2], Sf[2 * j][nt][3], d.y);
                    mul2(Sf[2 * j + 1][nt][0], Sf[2 * j + 1][nt][1], d.z);
                    mul2(Sf[2 * j + 1][nt][2], Sf[2 * j + 1][nt][3], d.w);
                }
            }
        }
        uint32_t Ub[4][2];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            add2(u[0][nt][0], u[0][nt][1], u[1][nt][0], u[1][nt][1]);
            add2(u[0][nt][2], u[0][nt][3], u[1][nt][2], u[1][nt][3]);
            Ub[nt][0] = movm_t(pack_f16_sat(u[0][nt][0], u[0][nt][1]));   // FP16 (mma_f16)
            Ub[nt][1] = movm_t(pack_f16_sat(u[0][nt][2], u[0][nt][3]));
        }
        // S^T <- D S^T + (K^end)^T U^T.
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t af[4];
            ldsm_x4(af, sKE + sw32_off(16 * mt + rowA, hiA));
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) mma_f16(Sf[mt][nt], af, Ub[nt], Sf[mt][nt]);
        }
        stage_release(&empty[s], lane);
        // Refill the stage of chunk c - 1 once every warp has released it.
        if (warp == 0 && c >= 1 && issued < nch) {
            const int64_t cp = c - 1;
            if (!mbar_wait_warp(&empty[cp % kQuadStages], (cp / kQuadStages) & 1, a.status)) {
                ok = false;
                ++c;
                break;
            }
            if (lane == 0) load(issued);
            __syncwarp();
            ++issued;
        }
    }
    if (!ok && warp == 0) {
        // Let the copies this warp issued and did not consume land before exiting.
        for (int64_t cc = c; cc < issued; ++cc)
            mbar_wait_bounded(&full[cc % kQuadStages], (cc / kQuadStages) & 1, a.status);
    }
    // F and Z leave in the segment chain's fragment order (fmap_frag_off,
    // zmap_frag_off): this warp's value tiles are 4 (warp % 4) + nt.
    __nv_bfloat16* dst = ident ? a.final_ident : a.final_state;
    if (ok && dst) {
        uint8_t* base = reinterpret_cast<uint8_t*>(dst + state_base);
        const uint32_t q = static_cast<uint32_t>(warp % kQuadWarps);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            if (ident) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const uint4 r = make_uint4(pack_bf16(Sf[mt][2 * p][0], Sf[mt][2 * p][1]),
                                               pack_bf16(Sf[mt][2 * p][2], Sf[mt][2 * p][3]),
                                               pack_bf16(Sf[mt][2 * p + 1][0], Sf[mt][2 * p + 1][1]),
                                               pack_bf16(Sf[mt][2 * p + 1][2], Sf[mt][2 * p + 1][3]));
                    *reinterpret_cast<uint4*>(base + fmap_frag_off(mt, 2 * q + p, lane)) = r;
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    const uint2 r = make_uint2(pack_bf16(Sf[mt][nt][0], Sf[mt][nt][1]),
                                               pack_bf16(Sf[mt][nt][2], Sf[mt][nt][3]));
                    *reinterpret_cast<uint2*>(base + zmap_frag_off(4 * q + nt, mt, lane)) = r;
                }
            }
        }
    }
}

template <int NCG>
__global__ void __launch_bounds__((2 * NCG + 1) * 32, 1)
    recurrence_ks_kernel(RecArgs a, const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    ks_setup<NCG>(smem);
    __syncthreads();
    ks_run<NCG>(a, &vmap, smem, blockIdx.x, nullptr);
}

template <int NCG>
cudaError_t launch_ks(const RecArgs& a, int64_t blocks, cudaStream_t stream) {
    using L = KsLayout<NCG>;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(recurrence_ks_kernel<NCG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(L::kSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    CUtensorMap vmap;
    alignas(64) static const char kZero[16] = {};
    const void* vbase = a.v ? static_cast<const void*>(a.v) : static_cast<const void*>(kZero);
    cudaError_t e = encode_v_map(&vmap, vbase, a.geo.tokens, a.H, L::kCols);
    if (e != cudaSuccess) return e;
    recurrence_ks_kernel<NCG><<<static_cast<unsigned>(blocks), (2 * NCG + 1) * 32, L::kSmemBytes, stream>>>(a, vmap);
    return cudaGetLastError();
}

template <int NW>
cudaError_t launch_nw(const RecArgs& a, int64_t blocks, cudaStream_t stream) {
    using L = RecLayout<NW>;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(recurrence_kernel<NW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(L::kSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    CUtensorMap vmap;
    alignas(64) static const char kZero[16] = {};
    // With no tokens nothing is loaded; still hand the kernel a well-formed map.
    const void* vbase = a.v ? static_cast<const void*>(a.v) : static_cast<const void*>(kZero);
    cudaError_t e = encode_v_map(&vmap, vbase, a.geo.tokens, a.H, L::kCols);
    if (e != cudaSuccess) return e;
    recurrence_kernel<NW><<<static_cast<unsigned>(blocks), (NW + 1) * 32, L::kSmemBytes, stream>>>(a, vmap);
    return cudaGetLastError();
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// Tensor map of v viewed as a 2-D BF16 array [tokens][H * 128] with boxes of
// 16 tokens x `cols` value columns.
cudaError_t encode_v_map(CUtensorMap* map, const void* v, int64_t tokens, int64_t H, int cols) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H * kHeadDim),
                                static_cast<cuuint64_t>(tokens > 0 ? tokens : 1)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(H * kHeadDim * 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(cols), static_cast<cuuint32_t>(kChunk)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(v), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The same view of v with boxes of 16 tokens x 64 value columns and the
// 128-byte swizzle (two boxes per 128 columns).
cudaError_t encode_v_map_sw128(CUtensorMap* map, const void* v, int64_t tokens, int64_t H) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(H * kHeadDim),
                                static_cast<cuuint64_t>(tokens > 0 ? tokens : 1)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(H * kHeadDim * 2)};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(kChunk)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(v), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map of BF16 states viewed as a 2-D array [rows][128], boxes of
// `box_rows` rows x 64 columns with the 128-byte swizzle.
cudaError_t encode_state_map(CUtensorMap* map, const void* base, int64_t rows, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim * 2)};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_recurrence(const void* v, void* out, const void* init_state,
                              void* final_state, const uint8_t* packets,
                              const SeqGeometry& geo, int64_t H, int nsplit, int* status,
                              cudaStream_t stream, const Checkpoints* ck) {
    RecArgs a;
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.out = static_cast<__nv_bfloat16*>(out);
    a.init_state = static_cast<const __nv_bfloat16*>(init_state);
    a.final_state = static_cast<__nv_bfloat16*>(final_state);
    a.packets = packets;
    a.geo = geo;
    a.H = H;
    a.nsplit = nsplit;
    a.status = status;
    a.ck = ck ? *ck : Checkpoints{nullptr, nullptr, 1, 0};
    a.final_ident = nullptr;
    // Engine 2 (opt-in): the tcgen05 kernel, one CTA per head (it writes no
    // checkpoints, so calls that ask for them take the column-split kernels).
    // Otherwise the column-split kernel with `nsplit` CTAs per head.
    if (recurrence_engine() == 2 && !a.ck.states)
        return launch_recurrence_tc(v, out, init_state, final_state, packets, geo, H, status, stream);
    const int64_t blocks = geo.n_seqs * H * nsplit;
    if (blocks <= 0) return cudaSuccess;
    if (geo.tokens >= (int64_t(1) << 31)) return cudaErrorInvalidValue;   // TMA coordinates are int32
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (recurrence_engine() == 1) {
        // Keys-major form only, 8 value columns per warp (for comparison).
        switch (nsplit) {
            case 1: return launch_nw<16>(a, blocks, stream);
            case 2: return launch_nw<8>(a, blocks, stream);
            case 4: return launch_nw<4>(a, blocks, stream);
            case 8: return launch_nw<2>(a, blocks, stream);
            case 16: return launch_nw<1>(a, blocks, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (nsplit) {
        case 1: return launch_quad(a, blocks, stream);     // 4 warps x 32 columns
        case 2: return launch_nw<8>(a, blocks, stream);    // 8 warps x 8 columns
        case 4: return launch_ks<4>(a, blocks, stream);    // key split: 4 pairs x 8 columns
        case 8: return launch_ks<2>(a, blocks, stream);
        case 16: return launch_ks<1>(a, blocks, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_transition(const void* v, const uint8_t* packets, const SeqGeometry& geo,
                              int64_t H, void* zero_start_states, void* transitions, int* status,
                              cudaStream_t stream) {
    RecArgs a;
    a.v = static_cast<const __nv_bfloat16*>(v);
    a.out = nullptr;
    a.init_state = nullptr;
    a.final_state = static_cast<__nv_bfloat16*>(zero_start_states);
    a.packets = packets;
    a.geo = geo;
    a.H = H;
    a.nsplit = 1;
    a.status = status;
    a.ck = Checkpoints{nullptr, nullptr, 1, 0};
    a.final_ident = static_cast<__nv_bfloat16*>(transitions);
    const int64_t blocks = geo.n_seqs * H;
    if (blocks <= 0) return cudaSuccess;
    if (geo.tokens >= (int64_t(1) << 31) || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(transition_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kQuadSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    CUtensorMap vmap;
    alignas(64) static const char kZero[16] = {};
    const void* vbase = a.v ? static_cast<const void*>(a.v) : static_cast<const void*>(kZero);
    cudaError_t e = encode_v_map_sw128(&vmap, vbase, a.geo.tokens, a.H);
    if (e != cudaSuccess) return e;
    transition_kernel<<<static_cast<unsigned>(blocks), kTransWarps * 32, kQuadSmemBytes, stream>>>(a,
                                                                                                  vmap);
    return cudaGetLastError();
}

}  // namespace kda
