// kda_tc_impl.cuh -- the recurrence of one (sequence, head) on the tcgen05
// tensor cores, as three warp roles that a kernel places in its CTA: a
// producer warp, an MMA-issuing warp and eight state warps.
//
// Chunk equations of "FlashKDA column split", section 1, with the error term
// as one contraction over the keys, in the orientation where the 128 value
// rows of the state are the MMA's M dimension:
//   U = V (A^kk B)^T + S K'^T       K' = -(A^kk B)(K^start)^T (packet)
//   O = S (s Q^start) + U (A^qk)^T
//   S <- S D_{0:15} + U K^end
// Tensor memory holds everything the chain carries (256 columns):
//   S      [0, 128)    the FP32 state; before the chunk's update it holds S D
//   P      [128, 144)  S (s Q^start), then O once U (A^qk)^T is added
//   U_S    [144, 160)  S K'^T
//   UV     [160, 176)  V (A^kk B)^T
//   S_A    [192, 256)  the state as the BF16 A operand of the next products
// Per chunk the issuer makes
//   UV       = V^T (A^kk B)^T                          1 MMA, N = 16
//   [P | U_S] = S_A [s Q^start ; K']^T                 8 MMAs, N = 32, 16 keys each
//   [S | P] += U [K^end ; A^qk]^T                      1 MMA, N = 144
// so the state update and O's U term are one instruction, and S D is formed
// by the state warps while the eight products run (the state update then only
// adds U K^end to it).  A state warp serves TMEM lanes 32 (w % 4) .. + 31
// (value rows) and the 32-key pieces w / 4 and 2 + w / 4 of those rows; it
// hands each piece back as BF16 as soon as it has it, so the products on keys
// 0-63 start while keys 64-127 are still being converted.  Every wait is
// bounded and warp-uniform.
#pragma once

#include "kda_common.cuh"
#include "kda_tcgen05.cuh"

namespace kda {
namespace tcr {

constexpr int kStateWarps = 8;
constexpr uint32_t kVTileBytes = kChunk * kHeadDim * 2;                                    // 4096
constexpr uint32_t kStageBytes = ((kPacketBytes + kVTileBytes + 1023) / 1024) * 1024;      // 18432
// Stage image (1024-aligned):
//   [0, 4096)      s Q^start keys 0-63 (16 rows), then K' keys 0-63 (16 rows): the
//                  N = 32 B operand of the 64-key slab, 8-row groups 1024 B apart
//   [4096, 8192)   the same for keys 64-127
//   [8192, 12288)  K^end^T (128 rows, FP16, SW32), then
//   [12288, 12800) A^qk (16 rows, FP16, SW32): one N = 144 B operand
//   [12800, 13312) A^kk B (BF16, SW32)
//   [13312, 13824) D_{0:15} (permuted, as in the packet)
//   [13824, 17920) the V tile [16 tokens][128 values]
constexpr uint32_t kStSlab = 4096;
constexpr uint32_t kStKE = 8192, kStAQK = 12288, kStAKB = 12800, kStD = 13312, kStV = 13824;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0, kColP = 128, kColU = 144, kColUV = 160, kColSA = 192;

// Barriers of one chain, after its ring's full/empty pairs.
struct Bars {
    uint64_t* full;    // [stages], producer: packet + V tile landed
    uint64_t* empty;   // [stages], state warps: stage released
    uint64_t* vt;      // V^T(c) written (8 warps)
    uint64_t* u;       // [P | U_S](c) and UV(c) accumulated (commit)
    uint64_t* ua;      // U(c) in FP16 in shared memory and S D stored (8 warps)
    uint64_t* sa;      // [4]: S_A piece p written (4 warps each)
    uint64_t* s;       // state update and O done (commit)
    uint64_t* done;    // every MMA done (commit)
};
constexpr int kExtraBars = 10;

template <int kStages>
__device__ __forceinline__ Bars make_bars(uint64_t* base) {
    Bars b;
    b.full = base;
    b.empty = base + kStages;
    b.vt = base + 2 * kStages + 0;
    b.u = base + 2 * kStages + 1;
    b.ua = base + 2 * kStages + 2;
    b.sa = base + 2 * kStages + 3;
    b.s = base + 2 * kStages + 7;
    b.done = base + 2 * kStages + 8;
    return b;
}

template <int kStages>
__device__ __forceinline__ void init_bars(const Bars& b) {
    for (int s = 0; s < kStages; ++s) {
        mbar_init(&b.full[s], 1);
        mbar_init(&b.empty[s], kStateWarps);
    }
    mbar_init(b.vt, kStateWarps);
    mbar_init(b.u, 1);
    mbar_init(b.ua, kStateWarps);
    for (int p = 0; p < 4; ++p) mbar_init(&b.sa[p], kStateWarps / 2);
    mbar_init(b.s, 1);
    mbar_init(b.done, 1);
}

// One chain's work: sequence n's chunks c_begin .. c_begin + nch - 1 of head h.
struct Chain {
    const __nv_bfloat16* v;
    __nv_bfloat16* out;
    const __nv_bfloat16* init_state;   // [.., H, 128, 128] at state index n, or null
    __nv_bfloat16* final_state;        // or null
    const uint8_t* packets;
    const uint32_t* ready;             // one flag per packet (one-launch form), or null
    int64_t H, h, n, c_begin, nch, tok0, seqlen;
    int* status;
};

__device__ __forceinline__ void st_shared_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    *reinterpret_cast<uint4*>(p) = make_uint4(a, b, c, d);
}

// ---------------------------------------------------------------- producer
template <int kStages>
__device__ __forceinline__ void produce(const Chain& ch, const CUtensorMap* vmap, uint8_t* ring,
                                        const Bars& b, int lane) {
    uint32_t fill_parity = 0, filled = 0;
    uint32_t ready_mask = 0;   // bit i: chunk ready_base + i seen ready
    int64_t ready_base = 0;
    bool ok = true;
    for (int64_t c = 0; c < ch.nch && ok; ++c) {
        const int s = static_cast<int>(c % kStages);
        if (c >= kStages) ok = mbar_wait_warp_sleep(&b.empty[s], ((c / kStages) - 1) & 1, ch.status);
        if (!ok) break;
        if (ch.ready && !((c - ready_base) < 32 && (ready_mask >> (c - ready_base)) & 1u)) {
            ready_base = c;
            ok = wait_ready_flags(ch.ready + (ch.c_begin + c) * ch.H + ch.h, ch.H, ch.nch - c,
                                  &ready_mask, ch.status);
            if (!ok) break;
            if (lane == 0) fence_proxy_async_global();
        }
        uint8_t* st = ring + s * kStageBytes;
        if (lane == 0) {
            const uint8_t* pk =
                ch.packets + ((ch.c_begin + c) * ch.H + ch.h) * static_cast<int64_t>(kPacketBytes);
            uint64_t* bar = &b.full[s];
            mbar_arrive_expect_tx(bar, kPacketBytes + kVTileBytes);
            bulk_g2s(st, pk + kOffQS, 2048, bar);
            bulk_g2s(st + 2048, pk + kOffKS, 2048, bar);
            bulk_g2s(st + kStSlab, pk + kOffQS + 2048, 2048, bar);
            bulk_g2s(st + kStSlab + 2048, pk + kOffKS + 2048, 2048, bar);
            bulk_g2s(st + kStKE, pk + kOffKE, kOffAKB - kOffKE, bar);
            bulk_g2s(st + kStAQK, pk + kOffAQK, 512, bar);
            bulk_g2s(st + kStAKB, pk + kOffAKB, 512, bar);
            bulk_g2s(st + kStD, pk + kOffD, 512, bar);
            tma_load_2d(st + kStV, vmap, static_cast<int32_t>(ch.h * kHeadDim),
                        static_cast<int32_t>(ch.tok0 + kChunk * c), bar);
        }
        __syncwarp();
        fill_parity ^= (filled >> s & 1u) << s;
        filled |= 1u << s;
    }
    if (!ok)
        for (int s = 0; s < kStages; ++s)
            if (filled >> s & 1u) mbar_wait_bounded(&b.full[s], (fill_parity >> s) & 1u, ch.status);
}

// -------------------------------------------------------------- MMA issuer
// vT, uA: the V^T and U operands in shared memory (128 x 16, SW32).
template <int kStages>
__device__ __forceinline__ void issue(const Chain& ch, const uint8_t* ring, const uint8_t* vT,
                                      const uint8_t* uA, const Bars& b, uint32_t tmem, int lane) {
    const uint32_t id16 = tc::idesc_bf16(128, 16), id32 = tc::idesc_bf16(128, 32);
    // U is FP16 in shared memory, and so are A^qk and K^end (see mma_f16).
    const uint32_t ih144 = tc::idesc_f16(128, 144);
    const uint64_t dVT = tc::smem_desc(vT, 256, tc::kSwizzle32B);
    const uint64_t dUA = tc::smem_desc(uA, 256, tc::kSwizzle32B);
    for (int64_t c = 0; c < ch.nch; ++c) {
        const int s = static_cast<int>(c % kStages);
        const uint32_t ph = static_cast<uint32_t>(c & 1);
        const uint8_t* st = ring + s * kStageBytes;
        if (!mbar_wait_warp(&b.full[s], (c / kStages) & 1, ch.status)) break;
        if (!mbar_wait_warp(b.vt, ph, ch.status)) break;
        tc::fence_after_sync();
        if (lane == 0)
            tc::mma_bf16(tmem + kColUV, dVT, tc::smem_desc(st + kStAKB, 256, tc::kSwizzle32B), id16, 0);
        __syncwarp();
        // [P | U_S] over keys 0-63 once pieces 0 and 1 are in, then 64-95, 96-127.
        bool ok = mbar_wait_warp(&b.sa[0], ph, ch.status) && mbar_wait_warp(&b.sa[1], ph, ch.status);
        if (!ok) break;
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if (kk >= 4 && (kk & 1) == 0) {
                if (!mbar_wait_warp(&b.sa[kk >> 1], ph, ch.status)) { ok = false; break; }
                tc::fence_after_sync();
            }
            if (lane == 0)
                tc::mma_ta(tmem + kColP, tmem + kColSA + 8 * kk,
                           tc::smem_desc(st + (kk >> 2) * kStSlab + 32 * (kk & 3), 1024, tc::kSwizzle128B),
                           id32, kk > 0 ? 1u : 0u);
            __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) tc::commit(b.u);
        __syncwarp();
        // S D + U K^end and P + U (A^qk)^T in one product.
        if (!mbar_wait_warp(b.ua, ph, ch.status)) break;
        tc::fence_after_sync();
        if (lane == 0) {
            tc::mma_bf16(tmem + kColS, dUA, tc::smem_desc(st + kStKE, 256, tc::kSwizzle32B), ih144, 1);
            tc::commit(b.s);
        }
        __syncwarp();
    }
    // Every MMA issued must be complete before tensor memory is released.
    if (lane == 0) tc::commit(b.done);
    __syncwarp();
    mbar_wait_warp(b.done, 0, ch.status);
}

// Row r, tokens 8 hf .. 8 hf + 7 of V^T (from the stage's V tile) into the
// SW32 K-major V^T operand.
__device__ __forceinline__ void build_vt(const uint8_t* st, uint8_t* vT, int r, int hf) {
    const uint16_t* vt = reinterpret_cast<const uint16_t*>(st + kStV);
    uint32_t p[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        p[j] = static_cast<uint32_t>(vt[(8 * hf + 2 * j) * kHeadDim + r]) |
               (static_cast<uint32_t>(vt[(8 * hf + 2 * j + 1) * kHeadDim + r]) << 16);
    st_shared_v4(vT + sw32_off(r, hf), p[0], p[1], p[2], p[3]);
}

// x[i] <- x[i] * D of key 32 p + i, with D from the stage's permuted vector
// (float4 4 r7 + p holds the factors of keys 32p + r7 + {0, 8, 16, 24}).
__device__ __forceinline__ void scale_by_d(uint32_t (&x)[32], const uint8_t* st, int p) {
    const float4* dq = reinterpret_cast<const float4*>(st + kStD);
#pragma unroll
    for (int r7 = 0; r7 < 8; ++r7) {
        const float4 d = dq[4 * r7 + p];
        x[r7] = __float_as_uint(__uint_as_float(x[r7]) * d.x);
        x[r7 + 8] = __float_as_uint(__uint_as_float(x[r7 + 8]) * d.y);
        x[r7 + 16] = __float_as_uint(__uint_as_float(x[r7 + 16]) * d.z);
        x[r7 + 24] = __float_as_uint(__uint_as_float(x[r7 + 24]) * d.w);
    }
}

// 32 FP32 values -> 16 packed BF16 pairs.
__device__ __forceinline__ void to_bf16(const uint32_t (&x)[32], uint32_t (&y)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = pack_bf16(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
}

// -------------------------------------------------------------- state warps
// w: 0 .. 7 (this chain's state warp index; warp w % 4 of its warpgroup must
// be the hardware warp that may access TMEM lanes 32 (w % 4) ..).
template <int kStages>
__device__ __forceinline__ void state(const Chain& ch, const uint8_t* ring, uint8_t* vT, uint8_t* uA,
                                      const Bars& b, uint32_t tmem, int w, int lane) {
    const int quarter = w & 3, hf = w >> 2;
    const int r = 32 * quarter + lane;   // value row, TMEM lane
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    const int64_t state_row = ((ch.n * ch.H + ch.h) * kHeadDim + r) * kHeadDim;
    bool ok = true;
    if (ch.nch > 0) ok = mbar_wait_warp(&b.full[0], 0, ch.status);
    // S_0: the BF16 operand copy is the initial state itself; the FP32 copy
    // is stored already multiplied by chunk 0's D.
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int p = 2 * j + hf;
        uint32_t wv[16];
        if (ch.init_state) {
            const uint4* src = reinterpret_cast<const uint4*>(ch.init_state + state_row + 32 * p);
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const uint4 q = src[x];
                wv[4 * x] = q.x; wv[4 * x + 1] = q.y; wv[4 * x + 2] = q.z; wv[4 * x + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) wv[i] = 0u;
        }
        if (ch.nch > 0 && ok) {
            tc::st_x16(trow + kColSA + 16 * p, wv);
            uint32_t f[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                f[2 * i] = __float_as_uint(bf16_lo(wv[i]));
                f[2 * i + 1] = __float_as_uint(bf16_hi(wv[i]));
            }
            scale_by_d(f, ring, p);
            tc::st_x32(trow + kColS + 32 * p, f);
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            mbar_arrive_if(&b.sa[p], lane == 0);
        } else if (ch.final_state) {
            // No chunks: the final state is the initial one.
            uint4* dst = reinterpret_cast<uint4*>(ch.final_state + state_row + 32 * p);
#pragma unroll
            for (int x = 0; x < 4; ++x) dst[x] = make_uint4(wv[4 * x], wv[4 * x + 1], wv[4 * x + 2], wv[4 * x + 3]);
        }
    }
    if (ch.nch > 0 && ok) {
        build_vt(ring, vT, r, hf);
        fence_proxy_async_smem();
        __syncwarp();
        mbar_arrive_if(b.vt, lane == 0);
    }
    for (int64_t c = 0; c < ch.nch && ok; ++c) {
        const int s = static_cast<int>(c % kStages);
        const uint32_t ph = static_cast<uint32_t>(c & 1);
        const uint8_t* st = ring + s * kStageBytes;
        int64_t len = ch.seqlen - kChunk * c;
        if (len > kChunk) len = kChunk;
        const bool more = c + 1 < ch.nch;
        const int s1 = static_cast<int>((c + 1) % kStages);
        const uint8_t* st1 = ring + s1 * kStageBytes;

        // U(c) = U_S + UV -> FP16 operand (tokens 8 hf .. 8 hf + 7).
        if (!mbar_wait_warp(b.u, ph, ch.status)) { ok = false; break; }
        tc::fence_after_sync();
        {
            uint32_t u[8], v[8];
            tc::ld_x8(trow + kColU + 8 * hf, u);
            tc::ld_x8(trow + kColUV + 8 * hf, v);
            tc::wait_ld();
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = __uint_as_float(u[i]) + __uint_as_float(v[i]);
            st_shared_v4(uA + sw32_off(r, hf), pack_f16_sat(f[0], f[1]), pack_f16_sat(f[2], f[3]),
                         pack_f16_sat(f[4], f[5]), pack_f16_sat(f[6], f[7]));
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        mbar_arrive_if(b.ua, lane == 0);

        // V^T of the next chunk, while the state update runs (this chunk's
        // V^T was read by an MMA that completed before U).
        if (more) {
            if (!mbar_wait_warp(&b.full[s1], ((c + 1) / kStages) & 1, ch.status)) { ok = false; break; }
            build_vt(st1, vT, r, hf);
            fence_proxy_async_smem();
            __syncwarp();
            mbar_arrive_if(b.vt, lane == 0);
        }

        // S(c+1) = S D + U K^end and O(c): hand each piece back as BF16, then
        // store it multiplied by the next chunk's D.
        if (!mbar_wait_warp(b.s, ph, ch.status)) { ok = false; break; }
        tc::fence_after_sync();
        uint32_t o[8];
        tc::ld_x8(trow + kColP + 8 * hf, o);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int p = 2 * j + hf;   // keys 32 p .. 32 p + 31
            uint32_t x[32];
            tc::ld_x32(trow + kColS + 32 * p, x);
            tc::wait_ld();
            uint32_t y[16];
            to_bf16(x, y);
            if (more) {
                tc::st_x16(trow + kColSA + 16 * p, y);
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                mbar_arrive_if(&b.sa[p], lane == 0);
                scale_by_d(x, st1, p);
                tc::st_x32(trow + kColS + 32 * p, x);
            } else if (ch.final_state) {
                uint4* dst = reinterpret_cast<uint4*>(ch.final_state + state_row + 32 * p);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = make_uint4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
            }
        }
        // O(c) rows: tokens 8 hf + i, value r.
        __nv_bfloat16* orow = ch.out + ((ch.tok0 + kChunk * c + 8 * hf) * ch.H + ch.h) * kHeadDim + r;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (8 * hf + i < len) orow[i * ch.H * kHeadDim] = __float2bfloat16_rn(__uint_as_float(o[i]));
        // S D stored before U(c+1) is handed over (its MMA adds to it).
        tc::wait_st();
        tc::fence_before_sync();
        // This stage's D and V tile have been read, and its MMAs are done.
        stage_release(&b.empty[s], lane);
    }
}

}  // namespace tcr
}  // namespace kda
