// kda_rec_impl.cuh -- device code of the recurrence shared by the
// standalone recurrence kernels (kda_recurrence.cu) and the fused kernel
// (kda_fused.cu): kernel arguments, small helpers, and the key-split variant.
#pragma once

#include <cuda.h>

#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace rec {

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
    Checkpoints ck;   // ck.states null: none
    // Transition launches only (segmented scan): where the identity-start
    // pass writes its final states.
    __nv_bfloat16* final_ident;
};

// Chunks and tokens of recurrence sequence n: a sequence of the batch, or
// with g.seg_chunks set, segment n % segs_per_seq of sequence
// n / segs_per_seq.  False when the packed metadata marked the batch invalid.
__device__ __forceinline__ bool seq_span(const SeqGeometry& g, int64_t n, int64_t& c_begin,
                                         int64_t& nch, int64_t& tok0, int64_t& seqlen) {
    if (g.cu_chunks) {
        if (!*g.valid) return false;
        c_begin = g.cu_chunks[n];
        nch = g.cu_chunks[n + 1] - c_begin;
        tok0 = g.cu_seqlens[n];
        seqlen = g.cu_seqlens[n + 1] - tok0;
    } else if (g.seg_chunks) {
        const int64_t sq = n / g.segs_per_seq;
        const int64_t c0 = (n - sq * g.segs_per_seq) * g.seg_chunks;
        c_begin = sq * g.chunks_per_seq + c0;
        nch = g.chunks_per_seq - c0;
        if (nch > g.seg_chunks) nch = g.seg_chunks;
        if (nch < 0) nch = 0;
        tok0 = sq * g.tokens_per_seq + kChunk * c0;
        seqlen = g.tokens_per_seq - kChunk * c0;
        if (seqlen > kChunk * g.seg_chunks) seqlen = kChunk * g.seg_chunks;
        if (seqlen < 0) seqlen = 0;
    } else {
        c_begin = n * g.chunks_per_seq;
        nch = g.chunks_per_seq;
        tok0 = n * g.tokens_per_seq;
        seqlen = g.tokens_per_seq;
    }
    return true;
}

// Where sequence n's checkpoint j of head h goes, or null (with the
// kDevBadCheckpoints status bit) when the caller's row offsets give it no
// row inside the buffer and inside the sequence's own range.
__device__ __forceinline__ __nv_bfloat16* checkpoint_dst(const RecArgs& a, int64_t n, int64_t h,
                                                         int64_t j) {
    const int64_t row = a.ck.cu_starts[n] + j;
    if (row < 0 || row >= a.ck.rows || row >= a.ck.cu_starts[n + 1]) {
        atomicOr(a.status, kDevBadCheckpoints);
        return nullptr;
    }
    return a.ck.states + (row * a.H + h) * kHeadDim * kHeadDim;
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void st_global_u32_if(void* p, uint32_t v, bool pred) {
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %2, 0;\n @p st.global.b32 [%0], %1;\n}\n"
                 ::"l"(p), "r"(v), "r"(static_cast<uint32_t>(pred))
                 : "memory");
}

__device__ __forceinline__ float dsel(const float4& a, int i) {
    return i == 0 ? a.x : (i == 1 ? a.y : (i == 2 ? a.z : a.w));
}

// ---------------------------------------------------------------------------
// Key-split variant for heads that get many CTAs (a latency-bound chain per
// warp).  Each 8-column group of S^T is held by a pair of warps, one per half
// of the 128 keys, so a warp issues half the operand loads and MMAs of the
// keys-major form.  Per chunk each warp forms its partial U^T (and partial
// P^T) over its 64 keys, the pair swaps partials through shared memory across
// its named barrier, and both add them in the same order (key half 0 + key
// half 1), so both warps continue from identical U^T.  The sums over
// keys are associated differently from the other variants, so results agree
// with them to rounding, not bit for bit.
// ---------------------------------------------------------------------------
template <int NCG>
struct KsLayout {
    static constexpr int kWarps = 2 * NCG;                        // consumer warps
    static constexpr int kCols = 8 * NCG;                         // value columns per CTA
    static constexpr int kStages = 8;
    static constexpr uint32_t kVRowBytes = kCols * 2;
    static constexpr uint32_t kStageBytes = ((kPacketBytes + kChunk * kVRowBytes + 1023) / 1024) * 1024;
    // Exchange buffers: [column group][chunk parity][key half][u, p][lane] float4.
    static constexpr uint32_t kXOff = kStages * kStageBytes;
    static constexpr uint32_t kXBytes = NCG * 2 * 2 * 2 * 32 * 16;
    static constexpr uint32_t kBarOff = kXOff + kXBytes;
    static constexpr uint32_t kSmemBytes = kBarOff + 2 * kStages * 8 + 1024;
};

struct HalfFrags {
    uint32_t ks[4][4];   // K' k-steps of this key half
    uint32_t qs[4][4];   // s (Q^start)^T k-steps of this key half
    uint32_t ke[4][4];   // (K^end)^T key tiles of this key half
    uint32_t akb[4];
    uint32_t aqk[4];
    float4 d[2];         // D for the key tiles of this key half
    uint32_t vb[2];
};

__device__ __forceinline__ void ks_load_uq(const uint8_t* stage, int kh, int lane, HalfFrags& f) {
    const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t hiA = lane >> 4;
    const uint32_t sKS = smem_u32(stage + kOffKS);
    const uint32_t sQS = smem_u32(stage + kOffQS);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ldsm_x4(f.ks[i], sKS + sw128_off(16, rowA, 2 * (4 * kh + i) + hiA));
        ldsm_x4(f.qs[i], sQS + sw128_off(16, rowA, 2 * (4 * kh + i) + hiA));
    }
}
__device__ __forceinline__ void ks_load_rest(const uint8_t* stage, uint32_t vrow_bytes, int cg, int kh,
                                             int lane, HalfFrags& f) {
    const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t hiA = lane >> 4;
    const int g8 = lane >> 2;
    const uint32_t sKE = smem_u32(stage + kOffKE);
#pragma unroll
    for (int i = 0; i < 4; ++i) ldsm_x4(f.ke[i], sKE + sw32_off(16 * (4 * kh + i) + rowA, hiA));
    ldsm_x4(f.akb, smem_u32(stage + kOffAKB + sw32_off(rowA, hiA)));
    ldsm_x4(f.aqk, smem_u32(stage + kOffAQK + sw32_off(rowA, hiA)));
    const uint8_t* sV = stage + kPacketBytes + (lane & 15) * vrow_bytes + 16 * cg;
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
                 : "=r"(f.vb[0]), "=r"(f.vb[1])
                 : "r"(smem_u32(sV)));
    const float4* dp = reinterpret_cast<const float4*>(stage + kOffD) + 4 * g8 + 2 * kh;
    f.d[0] = dp[0];
    f.d[1] = dp[1];
}

// This warp's slice of a state (its 64 keys of 8 value columns), BF16, into a
// [128 value][128 key] state at dst.
__device__ __forceinline__ void ks_store_state(__nv_bfloat16* dst, const float (&Sf)[4][4], int kh,
                                               int vcol, int g8, int t4) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int key = 16 * (4 * kh + i) + g8;
        const int val = vcol + 2 * t4;
        dst[(int64_t)val * kHeadDim + key] = __float2bfloat16_rn(Sf[i][0]);
        dst[(int64_t)(val + 1) * kHeadDim + key] = __float2bfloat16_rn(Sf[i][1]);
        dst[(int64_t)val * kHeadDim + key + 8] = __float2bfloat16_rn(Sf[i][2]);
        dst[(int64_t)(val + 1) * kHeadDim + key + 8] = __float2bfloat16_rn(Sf[i][3]);
    }
}

template <int NCG>
__device__ __forceinline__ void ks_setup(uint8_t* smem) {
    using L = KsLayout<NCG>;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* empty = full + L::kStages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < L::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], L::kWarps);
        }
        fence_barrier_init();
    }
}

// The CTA's work after ks_setup and a CTA-wide barrier: CTA `block` of the
// recurrence grid, warps 0 .. 2 NCG (the others do nothing here).  With
// `ready` set, the producer waits for ready[(chunk) * H + head] before it
// copies that chunk's packet (the packets are being written by the
// preparation running in the same launch).
template <int NCG>
__device__ __forceinline__ void ks_run(const RecArgs& a, const CUtensorMap* vmap, uint8_t* smem,
                                       int64_t block, const uint32_t* ready) {
    using L = KsLayout<NCG>;
    constexpr int kStages = L::kStages;
    constexpr int kWarps = L::kWarps;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* empty = full + kStages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nh = block / a.nsplit;
    const int split = static_cast<int>(block - nh * a.nsplit);
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

    if (warp > kWarps) return;
    if (warp == kWarps) {
        // ------------------------------------------------------------ producer
        uint32_t fill_parity = 0, filled = 0;
        uint32_t ready_mask = 0;   // bit i: chunk ready_base + i seen ready
        int64_t ready_base = 0;
        bool ok = true;
        for (int64_t c = 0; c < nch && ok; ++c) {
            const int s = static_cast<int>(c % kStages);
            if (c >= kStages)
                ok = mbar_wait_warp_sleep(&empty[s], ((c / kStages) - 1) & 1, a.status);
            if (!ok) break;
            uint8_t* stage = smem + s * L::kStageBytes;
            if (ready && !((c - ready_base) < 32 && (ready_mask >> (c - ready_base)) & 1u)) {
                // Poll the flags of chunks c .. c + 31 at once (lane i: chunk
                // c + i) until chunk c's is set; one proxy fence then orders
                // every copy of a chunk seen ready here after its packet.
                ready_base = c;
                ok = wait_ready_flags(ready + (c_begin + c) * a.H + h, a.H, nch - c, &ready_mask,
                                      a.status);
                if (!ok) break;
                if (lane == 0) fence_proxy_async_global();
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], kPacketBytes + kChunk * L::kVRowBytes);
                bulk_g2s(stage, a.packets + ((c_begin + c) * a.H + h) * static_cast<int64_t>(kPacketBytes),
                         kPacketBytes, &full[s]);
                tma_load_2d(stage + kPacketBytes, vmap, static_cast<int32_t>(h * kHeadDim + v0),
                            static_cast<int32_t>(tok0 + kChunk * c), &full[s]);
            }
            __syncwarp();
            fill_parity ^= (filled >> s & 1u) << s;
            filled |= 1u << s;
        }
        if (!ok)
            for (int s = 0; s < kStages; ++s)
                if (filled >> s & 1u) mbar_wait_bounded(&full[s], (fill_parity >> s) & 1u, a.status);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cg = warp >> 1;     // column group
    const int kh = warp & 1;      // key half
    const int g8 = lane >> 2, t4 = lane & 3;
    const int vcol = v0 + 8 * cg;
    const int64_t state_base = (n * a.H + h) * kHeadDim * kHeadDim;
    float4* xb = reinterpret_cast<float4*>(smem + L::kXOff) + cg * (2 * 2 * 2 * 32);

    // S^T rows (keys) of this half: tile i covers keys 16 (4 kh + i) + {g8, g8 + 8}.
    float Sf[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (a.init_state) {
            const __nv_bfloat16* src = a.init_state + state_base;
            const int key = 16 * (4 * kh + i) + g8;
            const int val = vcol + 2 * t4;
            Sf[i][0] = __bfloat162float(src[(int64_t)val * kHeadDim + key]);
            Sf[i][1] = __bfloat162float(src[(int64_t)(val + 1) * kHeadDim + key]);
            Sf[i][2] = __bfloat162float(src[(int64_t)val * kHeadDim + key + 8]);
            Sf[i][3] = __bfloat162float(src[(int64_t)(val + 1) * kHeadDim + key + 8]);
        } else {
            Sf[i][0] = Sf[i][1] = Sf[i][2] = Sf[i][3] = 0.f;
        }
    }
    uint32_t Sb[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        Sb[i][0] = movm_t(pack_bf16(Sf[i][0], Sf[i][1]));
        Sb[i][1] = movm_t(pack_bf16(Sf[i][2], Sf[i][3]));
    }

    bool ok = true;
    HalfFrags f;
    // The pair's named barrier (ids 1 .. NCG) also carries whether every wait
    // of both warps succeeded, so the two always leave the loop together.
    const int xbid = 1 + cg;
    if (nch > 0) {
        ok = mbar_wait_warp(&full[0], 0, a.status);
        if (ok) {
            ks_load_uq(smem, kh, lane, f);
            ks_load_rest(smem, L::kVRowBytes, cg, kh, lane, f);
        }
        ok = pair_all(xbid, ok);
    }
    int64_t ck_next = 0;   // next chunk whose incoming state is a checkpoint
    for (int64_t c = 0; c < nch && ok; ++c) {
        if (a.ck.states && c == ck_next) {
            ck_next += a.ck.every;
            __nv_bfloat16* dst = checkpoint_dst(a, n, h, c / a.ck.every);
            if (dst) ks_store_state(dst, Sf, kh, vcol, g8, t4);
        }
        const int s = static_cast<int>(c % kStages);
        const bool has_next = c + 1 < nch;
        const int s1 = static_cast<int>((c + 1) % kStages);
        const uint32_t par1 = static_cast<uint32_t>(((c + 1) / kStages) & 1);
        const uint8_t* stage1 = smem + s1 * L::kStageBytes;
        bool next_ready = has_next && mbar_try_wait(&full[s1], par1);
        int64_t len = seqlen - kChunk * c;
        if (len > kChunk) len = kChunk;

        // Partial U^T and P^T over this warp's 64 keys, from the incoming state.
        float ua[4] = {0.f, 0.f, 0.f, 0.f}, ub[4] = {0.f, 0.f, 0.f, 0.f};
        float pa[4] = {0.f, 0.f, 0.f, 0.f}, pb[4] = {0.f, 0.f, 0.f, 0.f};
        if (kh == 0) mma_bf16(ua, f.akb, f.vb, ua);
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
            mma_bf16(ua, f.ks[i], Sb[i], ua);
            mma_bf16(ub, f.ks[i + 1], Sb[i + 1], ub);
            mma_bf16(pa, f.qs[i], Sb[i], pa);
            mma_bf16(pb, f.qs[i + 1], Sb[i + 1], pb);
        }
        const int slot = static_cast<int>(c & 1);
        float4* mine = xb + ((slot * 2 + kh) * 2) * 32 + lane;
        const float4* theirs = xb + ((slot * 2 + (kh ^ 1)) * 2) * 32 + lane;
        // Own partials: all of U^T; of P^T the token rows the partner stores
        // (key half 0 stores tokens 0-7, i.e. fragment rows g8; half 1 rows g8 + 8).
        const float4 uh = make_float4(ua[0] + ub[0], ua[1] + ub[1], ua[2] + ub[2], ua[3] + ub[3]);
        const float2 ph_own = kh == 0 ? make_float2(pa[0] + pb[0], pa[1] + pb[1])
                                      : make_float2(pa[2] + pb[2], pa[3] + pb[3]);
        mine[0] = uh;
        *reinterpret_cast<float2*>(mine + 32) = kh == 0 ? make_float2(pa[2] + pb[2], pa[3] + pb[3])
                                                        : make_float2(pa[0] + pb[0], pa[1] + pb[1]);
        // D S^T for this half, in place (the BF16 copy is in Sb).
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float d0 = dsel(f.d[i >> 1], 2 * (i & 1));
            const float d1 = dsel(f.d[i >> 1], 2 * (i & 1) + 1);
            mul2(Sf[i][0], Sf[i][1], d0);
            mul2(Sf[i][2], Sf[i][3], d1);
        }
        // Every read of this chunk's stage was issued during the previous
        // chunk (or before the loop): hand it back before the next chunk's
        // loads, so that the proxy fence finds nothing in flight.
        stage_release(&empty[s], lane);
        // The K' and Q^start fragments are dead: load the next chunk's.
        if (has_next) {
            if (!__all_sync(0xffffffffu, next_ready))
                next_ready = mbar_wait_warp(&full[s1], par1, a.status);
            if (next_ready)
                ks_load_uq(stage1, kh, lane, f);
            else
                ok = false;
        }
        // The partner's partials (the pair barrier orders the stores above
        // before the loads below).
        ok = pair_all(xbid, ok);
        // Key half 0 + key half 1 (addition commutes, so both warps get the
        // same bits whichever half is their own).
        float u[4], pp[4];
        {
            const float4 tu = theirs[0];
            const float2 tp = *reinterpret_cast<const float2*>(theirs + 32);
            u[0] = uh.x + tu.x; u[1] = uh.y + tu.y; u[2] = uh.z + tu.z; u[3] = uh.w + tu.w;
            // P^T rows this warp stores; the other two entries are not used.
            const float2 pr = make_float2(ph_own.x + tp.x, ph_own.y + tp.y);
            pp[0] = kh == 0 ? pr.x : 0.f;
            pp[1] = kh == 0 ? pr.y : 0.f;
            pp[2] = kh == 0 ? 0.f : pr.x;
            pp[3] = kh == 0 ? 0.f : pr.y;
        }
        uint32_t Ub[2];
        Ub[0] = movm_t(pack_f16_sat(u[0], u[1]));   // FP16 (mma_f16)
        Ub[1] = movm_t(pack_f16_sat(u[2], u[3]));
        // S^T <- D S^T + (K^end)^T U^T for this half.
#pragma unroll
        for (int i = 0; i < 4; ++i) mma_f16(Sf[i], f.ke[i], Ub, Sf[i]);
        float o[4];
        mma_f16(o, f.aqk, Ub, pp);
        if (has_next && ok) ks_load_rest(stage1, L::kVRowBytes, cg, kh, lane, f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            Sb[i][0] = movm_t(pack_bf16(Sf[i][0], Sf[i][1]));
            Sb[i][1] = movm_t(pack_bf16(Sf[i][2], Sf[i][3]));
        }
        // Key half 0 stores tokens 0-7 of O, key half 1 tokens 8-15.
        const int tok = 8 * kh + g8;
        __nv_bfloat16* orow = a.out + ((tok0 + kChunk * c + tok) * a.H + h) * kHeadDim + vcol + 2 * t4;
        st_global_u32_if(orow, kh == 0 ? pack_bf16(o[0], o[1]) : pack_bf16(o[2], o[3]), tok < len);
    }

    if (ok && a.final_state) ks_store_state(a.final_state + state_base, Sf, kh, vcol, g8, t4);
}


// ---------------------------------------------------------------------------
// Wide variant for one CTA per (sequence, head): consumer warps of NT
// 8-column n-tiles (8 NT value columns) over all 128 keys, the n-tiles of a
// warp sharing every A fragment (K', Q^start, K^end), so the CTA reads each
// chunk's fragments from shared memory once per warp rather than once per 8
// columns.  The BF16 copy of the state is not kept: each k-step converts its
// slice of the incoming FP32 state just before the U and P MMAs that use it
// (the same conversions and order as the other full-key variants, so the
// results are bitwise theirs whatever NT is).  Used with NT = 4 (the quad
// kernel: 4 warps, up to 255 registers) and NT = 2 (the many-head one-launch
// form: 8 warps at 128 registers, kda_fused.cu).
// ---------------------------------------------------------------------------
constexpr uint32_t kWideVRowBytes = kHeadDim * 2;
// The V tile sits 1024-aligned after the packet as two [16][64] slabs with
// the 128-byte swizzle (rows 256 bytes apart would put the eight rows of
// each transposing load in the same banks).
constexpr uint32_t kWideVOff = ((kPacketBytes + 1023) / 1024) * 1024;
constexpr uint32_t kWideStageBytes = ((kWideVOff + kChunk * kWideVRowBytes + 1023) / 1024) * 1024;
// Modes: kWidePlain; kWideCkpt writes checkpoints (a separate instantiation
// keeps the check out of the loop of the plain call).
constexpr int kWidePlain = 0;
constexpr int kWideCkpt = 1;

// V rows tok .. tok + 15 of head h into the stage's two swizzled slabs.
__device__ __forceinline__ void wide_load_v(uint8_t* stage, const CUtensorMap* vmap, int64_t h,
                                            int64_t tok, uint64_t* bar) {
    tma_load_2d(stage + kWideVOff, vmap, static_cast<int32_t>(h * kHeadDim), static_cast<int32_t>(tok),
                bar);
    tma_load_2d(stage + kWideVOff + kChunk * 128, vmap, static_cast<int32_t>(h * kHeadDim + 64),
                static_cast<int32_t>(tok), bar);
}

// A warp's slice of a state (all 128 keys of 8 NT value columns), BF16, into
// a [128 value][128 key] state at dst.
template <int NT>
__device__ __forceinline__ void wide_store_state(__nv_bfloat16* dst, const float (&Sf)[8][NT][4],
                                                 int vcol, int g8, int t4) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int key = 16 * mt + g8;
            const int val = vcol + 8 * nt + 2 * t4;
            dst[(int64_t)val * kHeadDim + key] = __float2bfloat16_rn(Sf[mt][nt][0]);
            dst[(int64_t)(val + 1) * kHeadDim + key] = __float2bfloat16_rn(Sf[mt][nt][1]);
            dst[(int64_t)val * kHeadDim + key + 8] = __float2bfloat16_rn(Sf[mt][nt][2]);
            dst[(int64_t)(val + 1) * kHeadDim + key + 8] = __float2bfloat16_rn(Sf[mt][nt][3]);
        }
}

// Producer warp of a wide CTA: per chunk, one bulk copy of the packet and the
// two TMA loads of the 16 x 128 V tile into ring stage c % kStages.  With
// `ready` (one-launch form) it first waits for the packet's ready flag,
// polling the flags of 32 chunks at once.
template <int kStages>
__device__ __forceinline__ void wide_produce(const RecArgs& a, const CUtensorMap* vmap,
                                             uint8_t* smem, uint64_t* full, uint64_t* empty,
                                             int lane, int64_t h, int64_t c_begin, int64_t nch,
                                             int64_t tok0, const uint32_t* ready) {
    uint32_t fill_parity = 0, filled = 0;
    uint32_t ready_mask = 0;   // bit i: chunk ready_base + i seen ready
    int64_t ready_base = 0;
    bool ok = true;
    for (int64_t c = 0; c < nch && ok; ++c) {
        const int s = static_cast<int>(c % kStages);
        if (c >= kStages) ok = mbar_wait_warp_sleep(&empty[s], ((c / kStages) - 1) & 1, a.status);
        if (!ok) break;
        if (ready && !((c - ready_base) < 32 && (ready_mask >> (c - ready_base)) & 1u)) {
            ready_base = c;
            ok = wait_ready_flags(ready + (c_begin + c) * a.H + h, a.H, nch - c, &ready_mask,
                                  a.status);
            if (!ok) break;
            if (lane == 0) fence_proxy_async_global();
        }
        uint8_t* stage = smem + s * kWideStageBytes;
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[s], kPacketBytes + kChunk * kWideVRowBytes);
            bulk_g2s(stage, a.packets + ((c_begin + c) * a.H + h) * static_cast<int64_t>(kPacketBytes),
                     kPacketBytes, &full[s]);
            wide_load_v(stage, vmap, h, tok0 + kChunk * c, &full[s]);
        }
        __syncwarp();
        fill_parity ^= (filled >> s & 1u) << s;
        filled |= 1u << s;
    }
    if (!ok)
        for (int s = 0; s < kStages; ++s)
            if (filled >> s & 1u) mbar_wait_bounded(&full[s], (fill_parity >> s) & 1u, a.status);
}

// Consumer warp `warp` of a wide CTA: value columns 8 NT warp .. + 8 NT - 1
// of (sequence n, head h), every chunk of the sequence from the ring.
template <int NT, int kStages, bool kCkpt>
__device__ __forceinline__ void wide_consume(const RecArgs& a, const uint8_t* smem,
                                             uint64_t* full, uint64_t* empty, int warp, int lane,
                                             int64_t n, int64_t h, int64_t c_begin, int64_t nch,
                                             int64_t tok0, int64_t seqlen) {
    static_assert(NT % 2 == 0, "V fragments are loaded for two n-tiles at a time");
    const int g8 = lane >> 2, t4 = lane & 3;
    const int vcol = 8 * NT * warp;   // first of this warp's value columns
    const int64_t state_base = (n * a.H + h) * kHeadDim * kHeadDim;
    const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t hiA = lane >> 4;

    float Sf[8][NT][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if (a.init_state) {
                const __nv_bfloat16* src = a.init_state + state_base;
                const int key = 16 * mt + g8;
                const int val = vcol + 8 * nt + 2 * t4;
                Sf[mt][nt][0] = __bfloat162float(src[(int64_t)val * kHeadDim + key]);
                Sf[mt][nt][1] = __bfloat162float(src[(int64_t)(val + 1) * kHeadDim + key]);
                Sf[mt][nt][2] = __bfloat162float(src[(int64_t)val * kHeadDim + key + 8]);
                Sf[mt][nt][3] = __bfloat162float(src[(int64_t)(val + 1) * kHeadDim + key + 8]);
            } else {
                Sf[mt][nt][0] = Sf[mt][nt][1] = Sf[mt][nt][2] = Sf[mt][nt][3] = 0.f;
            }
        }

    bool ok = true;
    // Checkpoints are numbered per sequence: a segment's chunks start at
    // chunk c_off of sequence n_ck.
    int64_t n_ck = n, c_off = 0;
    if (kCkpt) {
        if (a.geo.seg_chunks) {
            n_ck = n / a.geo.segs_per_seq;
            c_off = (n - n_ck * a.geo.segs_per_seq) * a.geo.seg_chunks;
        } else if (a.geo.seg_seq) {
            n_ck = a.geo.seg_seq[n];
            c_off = c_begin - a.geo.seq_chunks[n_ck];
        }
    }
    // next chunk whose incoming state is a checkpoint
    int64_t ck_next = kCkpt ? ((c_off + a.ck.every - 1) / a.ck.every) * a.ck.every - c_off : 0;
    for (int64_t c = 0; c < nch; ++c) {
        if (kCkpt && c == ck_next) {
            ck_next += a.ck.every;
            __nv_bfloat16* dst = checkpoint_dst(a, n_ck, h, (c_off + c) / a.ck.every);
            if (dst) wide_store_state<NT>(dst, Sf, vcol, g8, t4);
        }
        const int s = static_cast<int>(c % kStages);
        if (!mbar_wait_warp(&full[s], (c / kStages) & 1, a.status)) {
            ok = false;
            break;
        }
        const uint8_t* stage = smem + s * kWideStageBytes;
        const uint32_t sKS = smem_u32(stage + kOffKS);
        const uint32_t sQS = smem_u32(stage + kOffQS);
        const uint32_t sKE = smem_u32(stage + kOffKE);
        int64_t len = seqlen - kChunk * c;
        if (len > kChunk) len = kChunk;

        // U^T = (A^kk B) V^T + K' S^T and P^T = s (Q^start)^T S^T from the
        // incoming state, NT n-tiles, two accumulators each.
        float u[2][NT][4], p[2][NT][4];
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) u[x][nt][j] = p[x][nt][j] = 0.f;
        {
            uint32_t akb[4];
            ldsm_x4(akb, smem_u32(stage + kOffAKB + sw32_off(rowA, hiA)));
#pragma unroll
            for (int hp = 0; hp < NT / 2; ++hp) {
                // lanes 0-15: tokens of columns vcol + 16 hp .. + 7; lanes 16-31: + 8.
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
            uint32_t kf[4], qf[4];
            ldsm_x4(kf, sKS + sw128_off(16, rowA, 2 * kk + hiA));
            ldsm_x4(qf, sQS + sw128_off(16, rowA, 2 * kk + hiA));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t sb[2] = {movm_t(pack_bf16(Sf[kk][nt][0], Sf[kk][nt][1])),
                                        movm_t(pack_bf16(Sf[kk][nt][2], Sf[kk][nt][3]))};
                mma_bf16(u[kk & 1][nt], kf, sb, u[kk & 1][nt]);
                mma_bf16(p[kk & 1][nt], qf, sb, p[kk & 1][nt]);
            }
        }
        // D S^T in place.
        {
            const float4* dp = reinterpret_cast<const float4*>(stage + kOffD) + 4 * g8;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 d = dp[j];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mul2(Sf[2 * j][nt][0], Sf[2 * j][nt][1], d.x);
                    mul2(Sf[2 * j][nt][2], Sf[2 * j][nt][3], d.y);
                    mul2(Sf[2 * j + 1][nt][0], Sf[2 * j + 1][nt][1], d.z);
                    mul2(Sf[2 * j + 1][nt][2], Sf[2 * j + 1][nt][3], d.w);
                }
            }
        }
        uint32_t Ub[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
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
            for (int nt = 0; nt < NT; ++nt) mma_f16(Sf[mt][nt], af, Ub[nt], Sf[mt][nt]);
        }
        // O^T = P^T + A^qk U^T.
        float o[NT][4];
        {
            uint32_t aq[4];
            ldsm_x4(aq, smem_u32(stage + kOffAQK + sw32_off(rowA, hiA)));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                add2(p[0][nt][0], p[0][nt][1], p[1][nt][0], p[1][nt][1]);
                add2(p[0][nt][2], p[0][nt][3], p[1][nt][2], p[1][nt][3]);
                mma_f16(o[nt], aq, Ub[nt], p[0][nt]);
            }
        }
        stage_release(&empty[s], lane);
        __nv_bfloat16* orow = a.out + ((tok0 + kChunk * c + g8) * a.H + h) * kHeadDim + vcol + 2 * t4;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            st_global_u32_if(orow + 8 * nt, pack_bf16(o[nt][0], o[nt][1]), g8 < len);
            st_global_u32_if(orow + 8 * a.H * kHeadDim + 8 * nt, pack_bf16(o[nt][2], o[nt][3]), g8 + 8 < len);
        }
    }

    if (ok && a.final_state) wide_store_state<NT>(a.final_state + state_base, Sf, vcol, g8, t4);
}

}  // namespace rec
}  // namespace kda
