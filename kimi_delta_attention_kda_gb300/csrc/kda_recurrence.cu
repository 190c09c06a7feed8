// kda_recurrence.cu -- the serial-over-chunks KDA recurrence (sm_103a).
//
// For every chunk c of one (sequence, head), in the transposed layout of
// "FlashKDA column split", section 3.1 (one row per token, one column per
// value channel):
//   W^T   = (K^start)^T S^T                        (16 tokens x values)
//   U^T   = (A^kk B)(V^T - W^T)
//   O^T   = s (Q^start)^T S^T + A^qk U^T
//   S^T  <- D_{0:15} S^T + (K^end)^T U^T
// Value columns are independent recurrences that share the per-chunk inputs
// (section 3.1), so the 128 value columns of a head are split over `nsplit`
// CTAs and, inside a CTA, over warps of 8 columns each.  Each warp keeps its
// 128 x 8 slice of S^T in registers in FP32 for the whole sequence (section
// 3.3); the BF16 copy used as an MMA operand is refreshed every chunk.  The
// accumulator -> operand layout change is an 8 x 8 transpose in registers
// (movmatrix).  No CTA ever waits on another CTA.
//
// A producer warp streams the per-chunk packets (kda_common.cuh) and the V
// rows into a ring of shared-memory stages with one-dimensional bulk copies
// (TMA), completing on mbarriers; every wait is bounded (kda_common.cuh).
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kStages = 4;

struct RecArgs {
    const __nv_bfloat16* v;
    __nv_bfloat16* out;
    const __nv_bfloat16* init_state;
    __nv_bfloat16* final_state;
    const uint8_t* packets;
    SeqGeometry geo;
    int64_t H;
    int nsplit;
    int* status;
};

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <int NW>
struct RecLayout {
    static constexpr int kCols = 8 * NW;                        // value columns per CTA
    static constexpr uint32_t kVRowBytes = kCols * 2;           // one token row of V
    static constexpr uint32_t kStageBytes =
        ((kPacketBytes + kChunk * kVRowBytes + 1023) / 1024) * 1024;
    static constexpr uint32_t kBarOff = kStages * kStageBytes;
    static constexpr uint32_t kSmemBytes = kBarOff + 2 * kStages * 8 + 1024;  // + align slack
};

template <int NW>
__global__ void __launch_bounds__((NW + 1) * 32) recurrence_kernel(RecArgs a) {
    using L = RecLayout<NW>;
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
    const int64_t n = nh / a.H;
    const int64_t h = nh - n * a.H;
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
        int64_t fills[kStages] = {0, 0, 0, 0};
        bool ok = true;
        for (int64_t c = 0; c < nch && ok; ++c) {
            const int s = static_cast<int>(c % kStages);
            if (c >= kStages) ok = mbar_wait_bounded(&empty[s], ((c / kStages) - 1) & 1, a.status);
            if (!ok) break;
            int64_t len = seqlen - kChunk * c;
            if (len > kChunk) len = kChunk;
            uint8_t* stage = smem + s * L::kStageBytes;
            if (lane == 0)
                mbar_arrive_expect_tx(&full[s], kPacketBytes + static_cast<uint32_t>(len) * L::kVRowBytes);
            __syncwarp();
            if (lane == 0)
                bulk_g2s(stage, a.packets + ((c_begin + c) * a.H + h) * static_cast<int64_t>(kPacketBytes),
                         kPacketBytes, &full[s]);
            if (lane < len)
                bulk_g2s(stage + kPacketBytes + lane * L::kVRowBytes,
                         a.v + ((tok0 + kChunk * c + lane) * a.H + h) * kHeadDim + v0,
                         L::kVRowBytes, &full[s]);
            fills[s] += 1;
        }
        if (!ok) {
            // Let every copy already issued land before the CTA can exit.
            for (int s = 0; s < kStages; ++s)
                if (fills[s] > 0) mbar_wait_bounded(&full[s], (fills[s] - 1) & 1, a.status);
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

    const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;   // A-operand ldmatrix row
    const uint32_t hiA = lane >> 4;                             // A-operand column half
    bool ok = true;
    for (int64_t c = 0; c < nch; ++c) {
        const int s = static_cast<int>(c % kStages);
        if (!mbar_wait_bounded(&full[s], (c / kStages) & 1, a.status)) {
            ok = false;
            break;
        }
        const uint8_t* stage = smem + s * L::kStageBytes;
        const uint32_t sKS = smem_u32(stage + kOffKS);
        const uint32_t sQS = smem_u32(stage + kOffQS);
        const uint32_t sKE = smem_u32(stage + kOffKE);
        const float* sD = reinterpret_cast<const float*>(stage + kOffD);
        const uint8_t* sV = stage + kPacketBytes;
        int64_t len = seqlen - kChunk * c;
        if (len > kChunk) len = kChunk;

        // W^T = (K^start)^T S^T, two accumulators to halve the dependent chain.
        float w0[4] = {0.f, 0.f, 0.f, 0.f}, w1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t af[4];
            ldsm_x4(af, sKS + sw128_off(16, rowA, 2 * kk + hiA));
            if (kk & 1)
                mma_bf16(w1, af, Sb[kk], w1);
            else
                mma_bf16(w0, af, Sb[kk], w0);
        }
        // Delta^T = V^T - W^T (tokens g8, g8 + 8; values 2 t4, 2 t4 + 1).
        float vv[4] = {0.f, 0.f, 0.f, 0.f};
        if (g8 < len) {
            const uint32_t x = *reinterpret_cast<const uint32_t*>(sV + g8 * L::kVRowBytes + (8 * warp + 2 * t4) * 2);
            vv[0] = bf16_lo(x);
            vv[1] = bf16_hi(x);
        }
        if (g8 + 8 < len) {
            const uint32_t x = *reinterpret_cast<const uint32_t*>(sV + (g8 + 8) * L::kVRowBytes + (8 * warp + 2 * t4) * 2);
            vv[2] = bf16_lo(x);
            vv[3] = bf16_hi(x);
        }
        uint32_t Db[2];
        Db[0] = movm_t(pack_bf16(vv[0] - (w0[0] + w1[0]), vv[1] - (w0[1] + w1[1])));
        Db[1] = movm_t(pack_bf16(vv[2] - (w0[2] + w1[2]), vv[3] - (w0[3] + w1[3])));

        // U^T = (A^kk B) Delta^T.
        float u[4] = {0.f, 0.f, 0.f, 0.f};
        {
            uint32_t af[4];
            ldsm_x4(af, smem_u32(stage + kOffAKB + sw32_off(rowA, hiA)));
            mma_bf16(u, af, Db, u);
        }
        // P^T = s (Q^start)^T S^T (off the state chain).
        float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t af[4];
            ldsm_x4(af, sQS + sw128_off(16, rowA, 2 * kk + hiA));
            if (kk & 1)
                mma_bf16(p1, af, Sb[kk], p1);
            else
                mma_bf16(p0, af, Sb[kk], p0);
        }
        uint32_t Ub[2];
        Ub[0] = movm_t(pack_bf16(u[0], u[1]));
        Ub[1] = movm_t(pack_bf16(u[2], u[3]));

        // S^T <- D S^T + (K^end)^T U^T.
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t af[4];
            ldsm_x4(af, sKE + sw32_off(16 * mt + rowA, hiA));
            const float d0 = sD[16 * mt + g8];
            const float d1 = sD[16 * mt + g8 + 8];
            float cin[4] = {Sf[mt][0] * d0, Sf[mt][1] * d0, Sf[mt][2] * d1, Sf[mt][3] * d1};
            mma_bf16(Sf[mt], af, Ub, cin);
        }
        // O^T = P^T + A^qk U^T.
        float o[4];
        {
            uint32_t af[4];
            ldsm_x4(af, smem_u32(stage + kOffAQK + sw32_off(rowA, hiA)));
            float pin[4] = {p0[0] + p1[0], p0[1] + p1[1], p0[2] + p1[2], p0[3] + p1[3]};
            mma_bf16(o, af, Ub, pin);
        }
        // Every read of this stage is done: hand it back to the producer.
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        // Store O (tokens g8 and g8 + 8, values vcol + 2 t4 .. + 1).
        const int64_t tok = tok0 + kChunk * c;
        if (g8 < len)
            *reinterpret_cast<uint32_t*>(a.out + ((tok + g8) * a.H + h) * kHeadDim + vcol + 2 * t4) =
                pack_bf16(o[0], o[1]);
        if (g8 + 8 < len)
            *reinterpret_cast<uint32_t*>(a.out + ((tok + g8 + 8) * a.H + h) * kHeadDim + vcol + 2 * t4) =
                pack_bf16(o[2], o[3]);

        // BF16 operand copy of the new state for the next chunk.
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            Sb[mt][0] = movm_t(pack_bf16(Sf[mt][0], Sf[mt][1]));
            Sb[mt][1] = movm_t(pack_bf16(Sf[mt][2], Sf[mt][3]));
        }
    }

    if (ok && a.final_state) {
        __nv_bfloat16* dst = a.final_state + state_base;
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
}

template <int NW>
cudaError_t launch_nw(const RecArgs& a, int64_t blocks, cudaStream_t stream) {
    using L = RecLayout<NW>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(recurrence_kernel<NW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(L::kSmemBytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    recurrence_kernel<NW><<<static_cast<unsigned>(blocks), (NW + 1) * 32, L::kSmemBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_recurrence(const void* v, void* out, const void* init_state,
                              void* final_state, const uint8_t* packets,
                              const SeqGeometry& geo, int64_t H, int nsplit, int* status,
                              cudaStream_t stream) {
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
    const int64_t blocks = geo.n_seqs * H * nsplit;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    switch (nsplit) {
        case 1: return launch_nw<16>(a, blocks, stream);
        case 2: return launch_nw<8>(a, blocks, stream);
        case 4: return launch_nw<4>(a, blocks, stream);
        case 8: return launch_nw<2>(a, blocks, stream);
        case 16: return launch_nw<1>(a, blocks, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kda
