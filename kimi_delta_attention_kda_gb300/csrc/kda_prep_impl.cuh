// kda_prep_impl.cuh -- device code of the chunk preparation, shared by the
// standalone preparation kernel (kda_prep.cu) and the fused kernel
// (kda_fused.cu).  See kda_prep.cu for what one item computes.
#pragma once

#include <cuda.h>

#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace prep {

// Division by a divisor fixed for a launch, as a multiply-high, an add and a
// shift: the round-up multiplier of Granlund and Montgomery ("Division by
// invariant integers using multiplication", 1994, section 4).  For d in
// [1, 2^31): s = ceil(log2 d), m = floor(2^32 (2^s - d) / d) + 1 (< 2^32),
// and floor(n / d) = (mulhi(n, m) + n) >> s for every n in [0, 2^31), where
// mulhi(n, m) + n < 2 n cannot overflow 32 bits.
struct FastDiv {
    uint32_t d, m, s;
};
inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t s = 0;
    while ((uint64_t(1) << s) < d) ++s;
    const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << s) - d)) / d + 1;
    return FastDiv{d, static_cast<uint32_t>(m), s};
}
__host__ __device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
#ifdef __CUDA_ARCH__
    return (__umulhi(n, f.m) + n) >> f.s;
#else
    return static_cast<uint32_t>(((static_cast<uint64_t>(n) * f.m >> 32) + n) >> f.s);
#endif
}

// A CTA has 8 warps: 4 pairs.  Each (chunk, head) is prepared by one pair:
// warp h (0 or 1) of the pair builds the operands of tokens 8 h .. 8 h + 7,
// and the pair splits the rest (step comments below).  The pair synchronises on its own
// named barrier at fixed points of the item, so both warps always pass the
// same barriers.
constexpr int kPrepWarps = 8;
constexpr int kPrepPairs = kPrepWarps / 2;
// Per-pair shared memory: one 28 KB region that holds, in turn, an item's
// TMA inputs, its scratch and its packet image:
//   inputs  : q [16][128] BF16 at 0, k at 4096, g [16][128] FP32 at 8192
//   scratch : [0,4K) K^start hi (packet KS) | [4K,8K) s Q^start hi (packet QS) |
//             [8K,12K) exp(-G) khat hi | [12K,16K) exp(-G) khat lo |
//             [16K,20K) K^start lo | [20K,24K) s Q^start lo | [24K,28K) K^end rows
//             (tiles 16 x 128 BF16, SW128; "lo" = BF16 rounding of what the
//             BF16 "hi" part left out)
//   packet  : once the score MMAs are done, [8K,12K) receives K^end^T, [12K,13.5K)
//             A^kk B, A^qk and D; R (FP32) and the low part of A^kk B go to
//             [20K,22.5K); finally -(A^kk B) K^start^T replaces K^start in [0,4K):
//             [0, 13824) is then the packet image.
constexpr uint32_t kInQ = 0, kInK = 4096, kInG = 8192, kInBytes = 16384;
constexpr uint32_t kPrepOffKinv = 8192;
constexpr uint32_t kPrepOffKinvLo = 12288;
constexpr uint32_t kPrepOffKsLo = 16384;
constexpr uint32_t kPrepOffQsLo = 20480;
constexpr uint32_t kPrepOffKen = 24576;
constexpr uint32_t kPrepOffAkbLo = 20480;     // 16 x 16 BF16 SW32, after the score MMAs
constexpr uint32_t kPrepOffR = 21504;          // 16 x 16 FP32, after the score MMAs
constexpr uint32_t kPrepRegion = 28672;
// Regions, then one mbarrier per pair; + slack to align the base to 128 bytes
// (TMA destinations).  Two CTAs fit on an SM.
constexpr uint32_t kPrepSmemBytes = kPrepPairs * kPrepRegion + kPrepPairs * 8 + 128;

struct PrepArgs {
    const __nv_bfloat16* beta;
    uint8_t* packets;
    SeqGeometry geo;
    int64_t H;
    int64_t n_chunk_heads;   // < 2^31, so item, chunk and head indices fit 32 bits
    float scale;
    int beta_logit;          // 1: the beta tensor holds logits, beta = sigmoid(logit)
    // Fixed layout only: 1 numbers the items chunk index first, sequence
    // second ((chunk-in-sequence * N + sequence) * H + head), so that a
    // launch whose recurrence consumes every sequence at once gets each
    // sequence's first chunks first; 0: sequence by sequence.
    int interleave;
    // Packed layout, may be null: the items are numbered by chunk rank
    // (rank * H + head), and chunk_order[rank] is the chunk (launch_chunk_order).
    const int32_t* chunk_order;
    FastDiv div_h;           // by H
    FastDiv div_cps;         // by geo.chunks_per_seq (fixed layout)
    FastDiv div_n;           // by geo.n_seqs (fixed layout, interleave)
};

// The preparation's arguments for `geo` and H heads; false when the item
// count leaves the 32-bit range of the item arithmetic.
inline bool make_prep_args(PrepArgs* a, const void* beta, uint8_t* packets, const SeqGeometry& geo,
                           int64_t H, float scale, int* status, bool beta_logit = false) {
    a->beta = static_cast<const __nv_bfloat16*>(beta);
    a->beta_logit = beta_logit ? 1 : 0;
    a->interleave = 0;
    a->chunk_order = nullptr;
    a->packets = packets;
    a->geo = geo;
    a->geo.status = status;
    a->H = H;
    a->n_chunk_heads = geo.chunk_ub * H;
    a->scale = scale;
    if (H <= 0 || H >= (int64_t(1) << 31) || a->n_chunk_heads >= (int64_t(1) << 31)) return false;
    const int64_t cps = geo.cu_chunks ? 1 : geo.chunks_per_seq;
    if (cps <= 0 || cps >= (int64_t(1) << 31)) return false;
    a->div_h = make_fastdiv(static_cast<uint32_t>(H));
    a->div_cps = make_fastdiv(static_cast<uint32_t>(cps));
    if (geo.n_seqs <= 0 || geo.n_seqs >= (int64_t(1) << 31)) return false;
    a->div_n = make_fastdiv(static_cast<uint32_t>(geo.n_seqs));
    return true;
}

struct PrepMaps {
    CUtensorMap q, k, g;   // [tokens][H * 128] views, boxes of 16 tokens x 128 channels
};

// Largest n in [0, N) with cu_chunks[n] <= c (cu_chunks non-decreasing,
// cu_chunks[0] = 0 <= c < cu_chunks[N]).
__device__ __forceinline__ int64_t find_sequence(const int64_t* cu_chunks, int64_t N, int64_t c) {
    int64_t lo = 0, hi = N;
    while (hi - lo > 1) {
        int64_t mid = (lo + hi) >> 1;
        if (cu_chunks[mid] <= c)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

constexpr float kLog2e = 1.4426950408889634f;

// (acc0, acc1) += (x0, x1) * (y0, y1) as one packed FP32x2 fused multiply-add
// (each lane rounded as fmaf).
__device__ __forceinline__ void fma2(float& acc0, float& acc1, float x0, float x1, float y0,
                                     float y1) {
    uint64_t a, x, y;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(acc0), "f"(acc1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(y) : "f"(y0), "f"(y1));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x), "l"(y));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc0), "=f"(acc1) : "l"(a));
}

// 2^x by the hardware's approximate base-2 exponential (relative error about
// 2^-22 over the range used here, |x| <= 16 * 5 * log2(e)).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of channels 4 lane .. 4 lane + 3 of token row t in a [16][128]
// BF16 SW128 tile.
__device__ __forceinline__ uint32_t row4_off(int t, int lane) {
    return sw128_off(16, t, (4 * lane) >> 3) + ((lane & 1) << 3);
}
// Store 4 BF16 (channels 4 lane .. 4 lane + 3) of token row t.
__device__ __forceinline__ void st_row4(uint8_t* tile, int t, int lane, float a, float b, float c,
                                        float d) {
    *reinterpret_cast<uint2*>(tile + row4_off(t, lane)) = make_uint2(pack_bf16(a, b), pack_bf16(c, d));
}
// Same in FP16 (the K^end rows: the state update's operand is FP16).
__device__ __forceinline__ void st_row4_f16(uint8_t* tile, int t, int lane, float a, float b,
                                            float c, float d) {
    *reinterpret_cast<uint2*>(tile + row4_off(t, lane)) = make_uint2(pack_f16(a, b), pack_f16(c, d));
}
// Same, storing the BF16 rounding in `hi` and the BF16 rounding of what it
// left out in `lo`, so that hi + lo carries about 16 significant bits.
__device__ __forceinline__ void st_row4_split(uint8_t* hi, uint8_t* lo, int t, int lane, float a,
                                              float b, float c, float d) {
    const uint32_t off = row4_off(t, lane);
    const uint32_t h0 = pack_bf16(a, b), h1 = pack_bf16(c, d);
    sub2(a, b, bf16_lo(h0), bf16_hi(h0));
    sub2(c, d, bf16_lo(h1), bf16_hi(h1));
    const uint32_t l0 = pack_bf16(a, b);
    const uint32_t l1 = pack_bf16(c, d);
    *reinterpret_cast<uint2*>(hi + off) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(lo + off) = make_uint2(l0, l1);
}


// Token range [t0, t0 + len) of item (chunk c, head h); false when the item
// does not exist (past the last chunk of a packed batch, or invalid offsets).
// Every quantity fits 32 bits: items < 2^31 (make_prep_args) and tokens
// < 2^31 (the C ABI's shape check), so the item loop keeps 32-bit
// bookkeeping (64-bit values there cost registers the item code needs).
__device__ __forceinline__ bool item_range(const PrepArgs& a, uint32_t item, int32_t* t0,
                                           int32_t* len, int32_t* c_out, int32_t* h_out) {
    const uint32_t c32 = fast_div(item, a.div_h);
    int32_t c = static_cast<int32_t>(c32);
    const int32_t h = static_cast<int32_t>(item - c32 * a.div_h.d);
    int64_t ln;
    if (a.geo.cu_chunks) {
        if (c >= a.geo.cu_chunks[a.geo.n_seqs]) return false;
        if (a.chunk_order) c = a.chunk_order[c];
        const int64_t n = find_sequence(a.geo.cu_chunks, a.geo.n_seqs, c);
        const int64_t t = a.geo.cu_seqlens[n] + kChunk * (c - a.geo.cu_chunks[n]);
        *t0 = static_cast<int32_t>(t);
        ln = a.geo.cu_seqlens[n + 1] - t;
    } else if (a.interleave) {
        // c32 = chunk-in-sequence * N + sequence; the packet goes to the
        // sequence-by-sequence chunk number.
        const uint32_t ci32 = fast_div(c32, a.div_n);
        const int64_t n = c32 - ci32 * a.div_n.d;
        const int64_t ci = ci32;
        *t0 = static_cast<int32_t>(n * a.geo.tokens_per_seq + kChunk * ci);
        ln = a.geo.tokens_per_seq - kChunk * ci;
        c = static_cast<int32_t>(n * a.geo.chunks_per_seq + ci);
    } else {
        const uint32_t n32 = fast_div(c32, a.div_cps);
        const int64_t n = n32;
        const int64_t ci = c32 - n32 * a.div_cps.d;
        *t0 = static_cast<int32_t>(n * a.geo.tokens_per_seq + kChunk * ci);
        ln = a.geo.tokens_per_seq - kChunk * ci;
    }
    *len = static_cast<int32_t>(ln > kChunk ? kChunk : ln);
    *c_out = c;
    *h_out = h;
    return true;
}

// One (chunk, head) by warp `hw` of a pair (named barrier `bid`): inputs from
// the TMA tiles in `region`, scratch in `region` once the inputs are in
// registers, packet image in `region` at the end.
__device__ __forceinline__ void prep_item(uint8_t* region, int bid, int hw, float beta_f,
                                          int32_t len, float scale, int lane) {
    const uint8_t* in = region;
    uint8_t* ws = region;
    uint8_t* sc = region;
    uint8_t* tKS = ws + kOffKS;
    uint8_t* tQS = ws + kOffQS;
    uint8_t* tKE = ws + kOffKE;
    uint8_t* tAKB = ws + kOffAKB;
    uint8_t* tAQK = ws + kOffAQK;
    float* tD = reinterpret_cast<float*>(ws + kOffD);
    uint8_t* tKinv = sc + kPrepOffKinv;
    uint8_t* tKinvLo = sc + kPrepOffKinvLo;
    uint8_t* tKsLo = sc + kPrepOffKsLo;
    uint8_t* tQsLo = sc + kPrepOffQsLo;
    uint8_t* tKen = sc + kPrepOffKen;
    float* tR = reinterpret_cast<float*>(sc + kPrepOffR);
    const int tb = 8 * hw;   // this warp's tokens in steps 1-3: tb .. tb + 7

    // ---- 0. A ragged last chunk: the tile rows past the end of the sequence
    // (the next sequence's tokens, or the tensor map's zero fill) are set to
    // zero, so that the steps below read all 16 rows unconditionally.
    if (len < kChunk) {
        for (int t = static_cast<int>(len) + hw; t < kChunk; t += 2) {
            *reinterpret_cast<float4*>(region + kInG + t * 512 + 16 * lane) =
                make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<uint2*>(region + kInQ + t * 256 + 8 * lane) = make_uint2(0u, 0u);
            *reinterpret_cast<uint2*>(region + kInK + t * 256 + 8 * lane) = make_uint2(0u, 0u);
        }
        pair_sync(bid);
    }

    // ---- 1. Lane l owns key channels 4 l .. 4 l + 3.  g's running sum (G, in
    // base-2 units so that each exponential below is one ex2) over all 16
    // tokens, keeping this warp's 8 tokens and G_15; q and k of this warp's 8
    // tokens.
    uint2 qv[8], kv[8];
    float G[8][4];
    float gl[4];             // G_15
    float red[16];           // partial sums of squares: q tokens tb..tb+7, k tokens tb..tb+7
    {
        float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
        if (hw == 1) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const float4 gg = *reinterpret_cast<const float4*>(in + kInG + t * 512 + 16 * lane);
                fma2(r0, r1, gg.x, gg.y, kLog2e, kLog2e);
                fma2(r2, r3, gg.z, gg.w, kLog2e, kLog2e);
            }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int t = tb + j;
            const float4 gg = *reinterpret_cast<const float4*>(in + kInG + t * 512 + 16 * lane);
            fma2(r0, r1, gg.x, gg.y, kLog2e, kLog2e);
            fma2(r2, r3, gg.z, gg.w, kLog2e, kLog2e);
            G[j][0] = r0;
            G[j][1] = r1;
            G[j][2] = r2;
            G[j][3] = r3;
            qv[j] = *reinterpret_cast<const uint2*>(in + kInQ + t * 256 + 8 * lane);
            kv[j] = *reinterpret_cast<const uint2*>(in + kInK + t * 256 + 8 * lane);
            const float q0 = bf16_lo(qv[j].x), q1 = bf16_hi(qv[j].x), q2 = bf16_lo(qv[j].y),
                        q3 = bf16_hi(qv[j].y);
            const float k0 = bf16_lo(kv[j].x), k1 = bf16_hi(kv[j].x), k2 = bf16_lo(kv[j].y),
                        k3 = bf16_hi(kv[j].y);
            red[j] = q0 * q0 + q1 * q1 + q2 * q2 + q3 * q3;
            red[8 + j] = k0 * k0 + k1 * k1 + k2 * k2 + k3 * k3;
        }
        if (hw == 0) {
#pragma unroll
            for (int t = 8; t < kChunk; ++t) {
                const float4 gg = *reinterpret_cast<const float4*>(in + kInG + t * 512 + 16 * lane);
                fma2(r0, r1, gg.x, gg.y, kLog2e, kLog2e);
                fma2(r2, r3, gg.z, gg.w, kLog2e, kLog2e);
            }
        }
        gl[0] = r0;
        gl[1] = r1;
        gl[2] = r2;
        gl[3] = r3;
    }

    // ---- 2. Sums of squares over the 128 channels: butterfly reduce-scatter
    // over lane bits 3..0, then the two lane halves.  Lane l ends with the
    // total of index l & 15 (q of token tb + l for l & 15 < 8, else k of
    // token tb + (l & 7)).
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? red[i] : red[i + o];
            const float keep = up ? red[i + o] : red[i];
            red[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    const float tot = red[0] + __shfl_xor_sync(0xffffffffu, red[0], 16);
    const float rnorm = rsqrtf(tot + 1e-6f);
    // Both warps have read the input tiles: from here on the region is scratch.
    pair_sync(bid);

    // ---- 3. Decayed operands of this warp's 8 tokens (the scale s rides on
    // the q norm factor).
    const float e_last0 = ex2_approx(gl[0]), e_last1 = ex2_approx(gl[1]);
    const float e_last2 = ex2_approx(gl[2]), e_last3 = ex2_approx(gl[3]);
    const float rnorm_q = (lane & 15) < 8 ? scale * rnorm : rnorm;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int t = tb + j;
        const float rq = __shfl_sync(0xffffffffu, rnorm_q, j);
        const float rk = __shfl_sync(0xffffffffu, rnorm, 8 + j);
        // The products below in packed pairs (bitwise the scalar products).
        float kh0 = bf16_lo(kv[j].x), kh1 = bf16_hi(kv[j].x);
        float kh2 = bf16_lo(kv[j].y), kh3 = bf16_hi(kv[j].y);
        float qh0 = bf16_lo(qv[j].x), qh1 = bf16_hi(qv[j].x);
        float qh2 = bf16_lo(qv[j].y), qh3 = bf16_hi(qv[j].y);
        mul2(kh0, kh1, rk);
        mul2(kh2, kh3, rk);
        mul2(qh0, qh1, rq);
        mul2(qh2, qh3, rq);
        const float e0 = ex2_approx(G[j][0]), e1 = ex2_approx(G[j][1]);
        const float e2 = ex2_approx(G[j][2]), e3 = ex2_approx(G[j][3]);
        const float i0 = ex2_approx(-G[j][0]), i1 = ex2_approx(-G[j][1]);
        const float i2 = ex2_approx(-G[j][2]), i3 = ex2_approx(-G[j][3]);
        float ks0 = e0, ks1 = e1, ks2 = e2, ks3 = e3;       // K^start
        float qs0 = e0, qs1 = e1, qs2 = e2, qs3 = e3;       // s Q^start
        float kv0 = i0, kv1 = i1, kv2 = i2, kv3 = i3;       // exp(-G) khat
        float ke0 = e_last0, ke1 = e_last1, ke2 = e_last2, ke3 = e_last3;   // K^end rows
        mul2v(ks0, ks1, kh0, kh1);
        mul2v(ks2, ks3, kh2, kh3);
        mul2v(qs0, qs1, qh0, qh1);
        mul2v(qs2, qs3, qh2, qh3);
        mul2v(kv0, kv1, kh0, kh1);
        mul2v(kv2, kv3, kh2, kh3);
        mul2v(ke0, ke1, kv0, kv1);   // exp(G_15) (exp(-G) khat)
        mul2v(ke2, ke3, kv2, kv3);
        st_row4_split(tKS, tKsLo, t, lane, ks0, ks1, ks2, ks3);
        st_row4_split(tQS, tQsLo, t, lane, qs0, qs1, qs2, qs3);
        st_row4_split(tKinv, tKinvLo, t, lane, kv0, kv1, kv2, kv3);
        st_row4_f16(tKen, t, lane, ke0, ke1, ke2, ke3);
    }
    // Every operand tile is complete.
    pair_sync(bid);

    // ---- 4. Scores, each as hi*hi + hi*lo + lo*hi of the split BF16 operands
    // (FP32 accumulate): warp 0 forms K^start (K exp(-G))^T (for R), warp 1
    // A^qk = (s Q^start)(K exp(-G))^T.  (A^qk from the BF16 s Q^start alone
    // lost 2.8e-2 of a one-token sequence's output: with q and k nearly
    // orthogonal, the rounding of q is large against their product.)
    const int gq = lane >> 2, tq = lane & 3;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
        const uint8_t* tA = hw == 0 ? tKS : tQS;
        const uint8_t* tAlo = hw == 0 ? tKsLo : tQsLo;
        const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
        const uint32_t rowB = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a4[4], b4[4], al4[4], bl4[4];
            const uint32_t offA = sw128_off(16, rowA, 2 * kk + (lane >> 4));
            const uint32_t offB = sw128_off(16, rowB, 2 * kk + ((lane >> 3) & 1));
            ldsm_x4(a4, smem_u32(tA + offA));
            ldsm_x4(b4, smem_u32(tKinv + offB));
            ldsm_x4(al4, smem_u32(tAlo + offA));
            ldsm_x4(bl4, smem_u32(tKinvLo + offB));
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                mma_bf16(acc[nt], a4, b4 + 2 * nt, acc[nt]);
                mma_bf16(acc[nt], a4, bl4 + 2 * nt, acc[nt]);
                mma_bf16(acc[nt], al4, b4 + 2 * nt, acc[nt]);
            }
        }
    }
    // Every read of the score operands is done; their tiles now take packet contents.
    pair_sync(bid);
    if (hw == 0) {
        tD[dperm_index(4 * lane + 0)] = e_last0;
        tD[dperm_index(4 * lane + 1)] = e_last1;
        tD[dperm_index(4 * lane + 2)] = e_last2;
        tD[dperm_index(4 * lane + 3)] = e_last3;
        const float beta_r0 = __shfl_sync(0xffffffffu, beta_f, gq);
        const float beta_r1 = __shfl_sync(0xffffffffu, beta_f, gq + 8);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int j0 = 8 * nt + 2 * tq;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = gq + 8 * hh;
                const float b = hh ? beta_r1 : beta_r0;
                const float r0 = (j0 < i) ? b * acc[nt][2 * hh] : 0.f;
                const float r1 = (j0 + 1 < i) ? b * acc[nt][2 * hh + 1] : 0.f;
                *reinterpret_cast<float2*>(tR + 16 * i + j0) = make_float2(r0, r1);
            }
        }
    } else {
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int j0 = 8 * nt + 2 * tq;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int i = gq + 8 * hh;
                const float q0 = (j0 <= i) ? acc[nt][2 * hh] : 0.f;
                const float q1 = (j0 + 1 <= i) ? acc[nt][2 * hh + 1] : 0.f;
                *reinterpret_cast<uint32_t*>(tAQK + sw32_off(i, nt) + 4 * tq) = pack_f16(q0, q1);
            }
        }
    }

    // ---- 5. K^end^T (key rows x token columns) by transposing 8 x 8 blocks:
    // warp 1, while warp 0 runs the forward substitution.
    if (hw == 1) {
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const int mi = lane >> 3;
            const int tok = 8 * (mi & 1) + (lane & 7);
            const int grp = 2 * p + (mi >> 1);
            uint32_t r[4];
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                         : "r"(smem_u32(tKen + sw128_off(16, tok, grp))));
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int key = 8 * (2 * p + (b >> 1)) + (lane >> 2);
                const int half = b & 1;
                *reinterpret_cast<uint32_t*>(tKE + sw32_off(key, half) + 4 * (lane & 3)) = r[b];
            }
        }
    }

    // ---- 6. A^kk = (I + R)^{-1} by forward substitution (warp 0, which wrote
    // R; lane m owns column m).
    if (hw == 0) {
        __syncwarp();
        if (lane < kChunk) {
            float x[kChunk];
#pragma unroll
            for (int i = 0; i < kChunk; ++i) x[i] = 0.f;
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                // Four partial sums, so that the dependent chain of row i is
                // ceil(i / 4) multiply-adds long instead of i.
                float a0 = (i == lane) ? 1.f : 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
                for (int jj = 0; jj < (i + 3) / 4; ++jj) {
                    const float4 rr = *reinterpret_cast<const float4*>(tR + 16 * i + 4 * jj);
                    a0 -= rr.x * x[4 * jj + 0];
                    a1 -= rr.y * x[4 * jj + 1];
                    a2 -= rr.z * x[4 * jj + 2];
                    a3 -= rr.w * x[4 * jj + 3];
                }
                x[i] = (a0 + a1) + (a2 + a3);
            }
            // Column `lane` of A^kk B (scaled by beta_lane), as BF16 high and low parts.
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                const float a = x[i] * beta_f;
                const __nv_bfloat16 hi = __float2bfloat16_rn(a);
                const __nv_bfloat16 lo = __float2bfloat16_rn(a - __bfloat162float(hi));
                const uint32_t off = sw32_off(i, lane >> 3) + 2 * (lane & 7);
                *reinterpret_cast<__nv_bfloat16*>(tAKB + off) = hi;
                *reinterpret_cast<__nv_bfloat16*>(sc + kPrepOffAkbLo + off) = lo;
            }
        }
    }
    // A^kk B and K^end^T are complete.
    pair_sync(bid);

    // ---- 7. K' = -(A^kk B) K^start^T (16 tokens x 128 keys; this warp's 64
    // keys), so that the recurrence gets U^T = (A^kk B) V^T + K' S^T from one
    // contraction over the keys: (V - S K^start)(A^kk B)^T = V (A^kk B)^T -
    // S (K^start (A^kk B)^T).  hi*hi + hi*lo + lo*hi of the split operands,
    // FP32 accumulation; it then replaces K^start in the packet (each warp
    // reads and writes only its own 64 key columns).
    {
        uint32_t ah[4], al[4];
        const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm_x4(ah, smem_u32(tAKB + sw32_off(rowA, lane >> 4)));
        ldsm_x4(al, smem_u32(sc + kPrepOffAkbLo + sw32_off(rowA, lane >> 4)));
        const int mi = lane >> 3;
        const int tok = 8 * (mi & 1) + (lane & 7);
        float kacc[8][4];
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
            // B fragments (k = token, n = key) of two 8-key tiles from the token-row tiles.
            uint32_t bh[4], bl[4];
            const uint32_t off = sw128_off(16, tok, 2 * (4 * hw + pp) + (mi >> 1));
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(bh[0]), "=r"(bh[1]), "=r"(bh[2]), "=r"(bh[3])
                         : "r"(smem_u32(tKS + off)));
            asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                         : "=r"(bl[0]), "=r"(bl[1]), "=r"(bl[2]), "=r"(bl[3])
                         : "r"(smem_u32(tKsLo + off)));
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float* d = kacc[2 * pp + half];
                d[0] = d[1] = d[2] = d[3] = 0.f;
                mma_bf16(d, ah, bh + 2 * half, d);
                mma_bf16(d, ah, bl + 2 * half, d);
                mma_bf16(d, al, bh + 2 * half, d);
            }
        }
        __syncwarp();   // every lane's K^start fragments are in registers
        const int gq2 = lane >> 2, tq2 = lane & 3;
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int nt = 8 * hw + n;
            *reinterpret_cast<uint32_t*>(tKS + sw128_off(16, gq2, nt) + 4 * tq2) =
                pack_bf16(-kacc[n][0], -kacc[n][1]);
            *reinterpret_cast<uint32_t*>(tKS + sw128_off(16, gq2 + 8, nt) + 4 * tq2) =
                pack_bf16(-kacc[n][2], -kacc[n][3]);
        }
    }
    // The packet image is complete; make it visible to the bulk copy.
    fence_proxy_async_smem();
    pair_sync(bid);
}

// Initialise pair `pair`'s mbarrier; both warps of the pair pass its named
// barrier `bid` afterwards.
__device__ __forceinline__ uint64_t* pair_barrier(uint8_t* smem, int pair, int hw, int lane,
                                                  int bid) {
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kPrepPairs * kPrepRegion) + pair;
    if (hw == 0 && lane == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
    }
    pair_sync(bid);
    return bar;
}

// What a pair needs beside its items when it runs in a one-launch kernel,
// kept in the pair's shared memory and read by its issuing thread where it is
// used (held in registers across an item, these values made the item code
// spill).
struct PairCtl {
    uint32_t* ready;     // ready[chunk * H + head] = 1 once that packet is in global memory
    uint32_t* counter;   // a zeroed global word the pairs take item numbers from, or null
    int64_t slot;        // counter mode: the next item's number, from the issuing thread
};

// A pair's share of the items: items first, first + stride, ... .  Both warps
// run this loop; warp 0's lane 0 issues the copies.  With `ctl` (one-launch
// kernels), ctl->ready[chunk * H + head] (the packet's index) becomes 1
// (release, GPU scope) once the item's packet is in global memory; the flag
// of an item is published when the pair has issued the next item's loads, or
// at the end.  With ctl->counter the pairs instead take items in order from
// it (atomicAdd by the pair's issuing thread once the item's loads are
// issued, handed to the other warp through ctl->slot), so that faster pairs
// take more items; `first` and `stride` are then unused.
__device__ __forceinline__ void run_items(const PrepArgs& a, const PrepMaps& maps, uint8_t* region,
                                          uint64_t* bar, int bid, int hw, int lane, int64_t first,
                                          int64_t stride, volatile PairCtl* ctl) {
    int32_t pending = -1;   // packet whose store is in flight, not yet published
    if (a.geo.cu_chunks && !*a.geo.valid) return;
    const bool issuer = hw == 0 && lane == 0;
    const uint32_t n_items = static_cast<uint32_t>(a.n_chunk_heads);
    const bool counted = ctl && ctl->counter;

    uint32_t phase = 0;
    uint32_t item = static_cast<uint32_t>(first);
    const uint32_t step = static_cast<uint32_t>(stride);
    if (counted) {
        if (issuer) ctl->slot = static_cast<int64_t>(atomicAdd(ctl->counter, 1u));
        pair_sync(bid);
        item = static_cast<uint32_t>(ctl->slot);
    }
    while (item < n_items) {
        int32_t t0, len, c, h;
        if (!item_range(a, item, &t0, &len, &c, &h)) break;   // items only grow past the end
        // (item + step cannot wrap: items < 2^31 and the pairs number far fewer.)
        uint32_t next = item + step;
        if (issuer) {
            // The previous packet store must have read the region before TMA
            // overwrites it; the region's generic-proxy writes were fenced
            // (fence.proxy.async) before that store.
            bulk_wait_read_all();
            mbar_arrive_expect_tx(bar, kInBytes);
            const int32_t x = h * kHeadDim, y = t0;
            tma_load_2d(region + kInQ, &maps.q, x, y, bar);
            tma_load_2d(region + kInK, &maps.k, x, y, bar);
            tma_load_2d(region + kInG, &maps.g, x, y, bar);
            // The next item's number, once this item's loads are on their way
            // (the atomic's round trip then overlaps them).
            if (counted) {
                next = atomicAdd(ctl->counter, 1u);
                ctl->slot = static_cast<int64_t>(next);   // read by the other warp after the barrier below
            }
            // This pair's next item: its tiles on their way to L2 while this
            // item is worked on, so that its loads above find them there.
            int32_t nt0, nlen, nc, nh;
            if (next < n_items && item_range(a, next, &nt0, &nlen, &nc, &nh)) {
                tma_prefetch_l2_2d(&maps.q, nh * kHeadDim, nt0);
                tma_prefetch_l2_2d(&maps.k, nh * kHeadDim, nt0);
                tma_prefetch_l2_2d(&maps.g, nh * kHeadDim, nt0);
            }
            if (ctl && pending >= 0) {
                // The previous packet is complete in global memory: publish it.
                bulk_wait_all();
                fence_proxy_async_global();
                st_release_gpu(ctl->ready + pending, 1u);
                pending = -1;
            }
        }
        float beta_f = lane < len ? __bfloat162float(a.beta[(static_cast<int64_t>(t0) + lane) * a.H + h]) : 0.f;
        // beta from a logit ("flashinfer kda_prefill", beta_is_logit):
        // sigmoid(x) = 1 / (1 + e^-x) in FP32; e^-x = inf for very negative x
        // gives 0, as it should.  Padding lanes stay 0.
        if (a.beta_logit && lane < len) beta_f = 1.f / (1.f + __expf(-beta_f));
        const bool got = mbar_wait_warp_sleep(bar, phase, a.geo.status);
        if (!pair_all(bid, got)) {
            // The loads may still land: wait for them (bounded) before leaving.
            if (!got) mbar_wait_bounded_sleep(bar, phase, a.geo.status);
            break;
        }
        if (counted) next = static_cast<uint32_t>(ctl->slot);   // the issuer's write precedes the barrier above
        phase ^= 1u;
        prep_item(region, bid, hw, beta_f, len, a.scale, lane);

        // Publish the packet with one bulk copy.
        if (issuer) {
            const int32_t pk = c * static_cast<int32_t>(a.H) + h;   // the packet's index
            bulk_s2g(a.packets + static_cast<int64_t>(pk) * kPacketBytes, region, kPacketBytes);
            bulk_commit();
            pending = pk;
        }
        item = next;
    }
    if (issuer) {
        bulk_wait_all();
        if (ctl && pending >= 0) {
            fence_proxy_async_global();
            st_release_gpu(ctl->ready + pending, 1u);
        }
    }
    __syncwarp();
}

// Tensor maps of q, k (BF16) and g (FP32) for the items' 2-D TMA loads.
cudaError_t encode_maps(PrepMaps* maps, const void* q, const void* k, const float* g,
                        int64_t tokens, int64_t H);

}  // namespace prep
}  // namespace kda
