// kda_segments.cu -- the middle pass of the segmented scan over chunks.
//
// The chunk equations of "FlashKDA column split", section 1, map the state of
// one chunk to the next by
//     S_{c+1} = S_c D_{0:15} + U_c K^end_c,   U_c = V_c (A^kk B)^T + S_c K'_c^T
// (U_c = (V_c - S_c K^start_c) B_c (A^kk_c)^T with K' = -(A^kk B) K^start^T),
// which is affine in S_c: S_{c+1} = S_c (D_{0:15} + K'^T K^end) + V_c (A^kk B)^T K^end.  Over a segment of consecutive chunks the map is
// therefore S -> S F + Z, with F the state the segment's chunks lead to from
// the identity with V taken as zero and Z the state they lead to from zero.
// The first pass (launch_transition) forms F and Z for every segment at
// once; this pass walks each sequence's segments in order,
//     S_0 = initial state,   S_{j+1} = S_j F_j + Z_j,
// and hands S_j to the last pass, which reruns segment j from S_j and writes
// its outputs.  With few heads this replaces one chain of all the chunks by
// chains of one segment's chunks plus this short chain of segment steps.
//
// One CTA per (sequence, head, 8 value rows of S): the rows of S update
// independently.  Four consumer warps each form 32 key columns of the new
// rows as (S_{j+1})^T = F_j^T S_j^T + Z_j^T on the warp MMA (BF16 operands,
// FP32 accumulation; the FP32 rows stay in registers), and swap their BF16
// slices through shared memory for the next step's operand.  A producer warp
// streams F_j and the CTA's rows of Z_j through a TMA ring.
#include <cuda.h>

#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kScanRows = 8;     // value rows of the state per CTA
constexpr int kScanWarps = 4;    // consumer warps, 32 keys each
constexpr int kScanStages = 3;
constexpr uint32_t kScanFBytes = kHeadDim * kHeadDim * 2;      // F: two SW128 slabs [128][64]
constexpr uint32_t kScanZBytes = kScanRows * kHeadDim * 2;     // Z rows: two SW128 slabs [8][64]
constexpr uint32_t kScanStageBytes = ((kScanFBytes + kScanZBytes + 1023) / 1024) * 1024;
constexpr uint32_t kScanXBytes = kScanRows * kHeadDim * 2;     // one BF16 copy of the CTA's rows
constexpr uint32_t kScanXOff = kScanStages * kScanStageBytes;
constexpr uint32_t kScanBarOff = kScanXOff + 2 * kScanXBytes;
constexpr uint32_t kScanSmemBytes = kScanBarOff + 2 * kScanStages * 8 + 1024;

// Byte offset of (row v, keys 8 ch .. 8 ch + 7) in a [8][128] BF16 copy of
// the CTA's rows; the 16-byte chunks of row v are XOR-swizzled by v so that
// the eight rows of one chunk fall in different banks.
__device__ __forceinline__ uint32_t x_off(uint32_t v, uint32_t ch) {
    return v * (kHeadDim * 2) + ((ch ^ v) << 4);
}

__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t* r, uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

struct ScanArgs {
    const __nv_bfloat16* init_state;   // [N][H][128][128] or null
    __nv_bfloat16* final_state;        // [N][H][128][128] or null
    __nv_bfloat16* starts;             // [segments][H][128][128]
    // Sequence n's segments: seg_begin[n] .. seg_begin[n + 1] - 1 (packed
    // layout), or n segs .. n segs + segs - 1 (seg_begin null: fixed layout).
    const int64_t* seg_begin;
    const int32_t* valid;              // packed layout: the metadata's verdict
    int64_t segs, H;
    int* status;
    // Composition in groups (first level of a two-level chain, fixed layout;
    // groups 0: off).  CTA sequence n is group n % groups of sequence
    // n / groups: segments gs = (n / groups) segs + (n % groups) group_segs
    // and on, up to group_segs of them.  The grid's first half composes the
    // F maps (src[0], no Z), the second half the Z maps (src[1], adding Z):
    // state_0 = src[gs], state_j = state_{j-1} F_{gs+j} (+ Z_{gs+j}); state_j
    // goes to prefix[p][gs + j] and the last one to gmap[p][n].
    int64_t groups, group_segs;
    const __nv_bfloat16* src[2];
    __nv_bfloat16* prefix[2];
    __nv_bfloat16* gmap[2];
};

// Warp w's slice (keys 32 w .. 32 w + 31 of the CTA's 8 rows) of a state in
// C-fragment form (m = key, n = value row), rounded to BF16, into the copy at x.
__device__ __forceinline__ void put_rows(uint8_t* x, const float (&c)[2][4], int w, int g8, int t4) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        const uint32_t lo = movm_trans(pack_bf16(c[mt][0], c[mt][1]));   // row g8, keys base + 2 t4
        const uint32_t hi = movm_trans(pack_bf16(c[mt][2], c[mt][3]));   // keys base + 8 + 2 t4
        const uint32_t base = 32 * w + 16 * mt;
        *reinterpret_cast<uint32_t*>(x + x_off(g8, base / 8) + 4 * t4) = lo;
        *reinterpret_cast<uint32_t*>(x + x_off(g8, base / 8 + 1) + 4 * t4) = hi;
    }
}

// The CTA's 8 rows from the copy at x into rows [8][128] at dst (thread tid
// of the 128 consumers copies 16 bytes).
__device__ __forceinline__ void copy_rows_out(const uint8_t* x, __nv_bfloat16* dst, int tid) {
    const int v = tid >> 4, ch = tid & 15;
    const uint4 val = *reinterpret_cast<const uint4*>(x + x_off(v, ch));
    *reinterpret_cast<uint4*>(dst + v * kHeadDim + 8 * ch) = val;
}

__global__ void __launch_bounds__((kScanWarps + 1) * 32, 1)
    segment_scan_kernel(ScanArgs a, const __grid_constant__ CUtensorMap fmap,
                        const __grid_constant__ CUtensorMap zmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kScanBarOff);
    uint64_t* empty = full + kScanStages;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int kGroups = kHeadDim / kScanRows;
    const bool compose = a.groups > 0;
    int part = 0;
    int64_t blk = blockIdx.x;
    if (compose) {
        const int64_t half = gridDim.x / 2;
        part = blk >= half ? 1 : 0;
        blk -= part * half;
    }
    const int64_t nh = blk / kGroups;
    const int v0 = kScanRows * static_cast<int>(blk - nh * kGroups);
    const int64_t n = nh / a.H;
    const int64_t h = nh - n * a.H;
    if (a.valid && !*a.valid) return;
    // Step j reads the maps of segment step0 + j and first carries no Z (or
    // its own when composing the Z maps); the state before step j goes to
    // segment first + j.
    int64_t first, nseg, step0;
    if (compose) {
        const int64_t sq = n / a.groups, gi = n - sq * a.groups;
        first = sq * a.segs + gi * a.group_segs;
        int64_t len = a.segs - gi * a.group_segs;
        if (len > a.group_segs) len = a.group_segs;
        nseg = len - 1;
        step0 = first + 1;
    } else {
        first = a.seg_begin ? a.seg_begin[n] : n * a.segs;
        nseg = a.seg_begin ? a.seg_begin[n + 1] - first : a.segs;
        step0 = first;
    }
    const bool add_z = !compose || part == 1;
    __nv_bfloat16* const starts = compose ? (part ? a.prefix[1] : a.prefix[0]) : a.starts;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kScanStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kScanWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kScanWarps) {
        // ------------------------------------------------------------ producer
        uint32_t fill_parity = 0, filled = 0;
        bool ok = true;
        for (int64_t j = 0; j < nseg && ok; ++j) {
            const int s = static_cast<int>(j % kScanStages);
            if (j >= kScanStages)
                ok = mbar_wait_warp_sleep(&empty[s], ((j / kScanStages) - 1) & 1, a.status);
            if (!ok) break;
            uint8_t* stage = smem + s * kScanStageBytes;
            if (lane == 0) {
                const int32_t row = static_cast<int32_t>(((step0 + j) * a.H + h) * kHeadDim);
                mbar_arrive_expect_tx(&full[s], kScanFBytes + kScanZBytes);
                tma_load_2d(stage, &fmap, 0, row, &full[s]);
                tma_load_2d(stage + kScanFBytes / 2, &fmap, 64, row, &full[s]);
                tma_load_2d(stage + kScanFBytes, &zmap, 0, row + v0, &full[s]);
                tma_load_2d(stage + kScanFBytes + kScanZBytes / 2, &zmap, 64, row + v0, &full[s]);
            }
            __syncwarp();
            fill_parity ^= (filled >> s & 1u) << s;
            filled |= 1u << s;
        }
        if (!ok)
            for (int s = 0; s < kScanStages; ++s)
                if (filled >> s & 1u) mbar_wait_bounded(&full[s], (fill_parity >> s) & 1u, a.status);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g8 = lane >> 2, t4 = lane & 3;
    const int tid = threadIdx.x;   // 0 .. 127
    uint8_t* xbuf = smem + kScanXOff;
    const int64_t rows0 = (n * a.H + h) * kHeadDim + v0;   // first row of this CTA in [N][H][128]
    // The initial state: the caller's (per sequence), or when composing the
    // group's first segment map.
    const __nv_bfloat16* init = compose ? (part ? a.src[1] : a.src[0]) + ((first * a.H + h) * kHeadDim + v0) * kHeadDim
                                        : (a.init_state ? a.init_state + rows0 * kHeadDim : nullptr);

    // S_0^T for keys 32 warp + 16 mt + {g8, g8 + 8}, rows v0 + 2 t4 + {0, 1}.
    float c[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        const int key = 32 * warp + 16 * mt + g8;
        if (init) {
            const __nv_bfloat16* src = init + 2 * t4 * kHeadDim;
            c[mt][0] = __bfloat162float(src[key]);
            c[mt][1] = __bfloat162float(src[kHeadDim + key]);
            c[mt][2] = __bfloat162float(src[key + 8]);
            c[mt][3] = __bfloat162float(src[kHeadDim + key + 8]);
        } else {
            c[mt][0] = c[mt][1] = c[mt][2] = c[mt][3] = 0.f;
        }
    }
    put_rows(xbuf, c, warp, g8, t4);
    bool ok = true;

    const uint32_t mi = lane >> 3, r8 = lane & 7;
    // Step j's operands from its stage into registers: F_j^T (m = new key,
    // k = old key) by transposing loads of F_j's rows (old key), and the C
    // fragments of Z_j^T.  The stage is released after the step that loads
    // it, once those loads have had the step's MMAs and barrier to complete.
    uint32_t af[2][8][4], zf[4];
    auto load_step = [&](int64_t j) -> bool {
        const int s = static_cast<int>(j % kScanStages);
        if (!mbar_wait_warp(&full[s], (j / kScanStages) & 1, a.status)) return false;
        const uint8_t* stage = smem + s * kScanStageBytes;
        ldsm_x4_trans(zf, smem_u32(stage + kScanFBytes + sw128_off(8, r8, 4 * warp + mi)));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const uint32_t row = 16 * kk + r8 + 8 * (mi >> 1);
                const uint32_t ch = 4 * warp + 2 * mt + (mi & 1);
                ldsm_x4_trans(af[mt][kk], smem_u32(stage + sw128_off(kHeadDim, row, ch)));
            }
        return true;
    };
    if (nseg > 0 && ok) {
        ok = load_step(0);
        if (ok) stage_release(&empty[0], lane);
    }
    ok = group_all<kScanWarps * 32>(1, ok);
    for (int64_t j = 0; j < nseg && ok; ++j) {
        const uint8_t* xc = xbuf + (j & 1) * kScanXBytes;
        // B operand: S_j^T (k = key of S_j, n = value row), all 8 k-steps.
        uint32_t b[8][2];
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
            uint32_t r[4];
            ldsm_x4(r, smem_u32(xc + x_off(r8, 4 * kp + mi)));
            b[2 * kp][0] = r[0];
            b[2 * kp][1] = r[1];
            b[2 * kp + 1][0] = r[2];
            b[2 * kp + 1][1] = r[3];
        }
        // Accumulators: Z_j^T (even k-steps; zero when composing the F maps)
        // and zero (odd k-steps).
        float acc[2][2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            acc[mt][0][0] = add_z ? bf_lo(zf[2 * mt]) : 0.f;
            acc[mt][0][1] = add_z ? bf_hi(zf[2 * mt]) : 0.f;
            acc[mt][0][2] = add_z ? bf_lo(zf[2 * mt + 1]) : 0.f;
            acc[mt][0][3] = add_z ? bf_hi(zf[2 * mt + 1]) : 0.f;
            acc[mt][1][0] = acc[mt][1][1] = acc[mt][1][2] = acc[mt][1][3] = 0.f;
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) mma_bf16(acc[mt][kk & 1], af[mt][kk], b[kk], acc[mt][kk & 1]);
        // While the MMAs run: S_j out as this segment's incoming state, and
        // the next step's operands in.
        copy_rows_out(xc, starts + (((first + j) * a.H + h) * kHeadDim + v0) * kHeadDim, tid);
        if (j + 1 < nseg && !load_step(j + 1)) ok = false;
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) c[mt][e] = acc[mt][0][e] + acc[mt][1][e];
        put_rows(xbuf + ((j + 1) & 1) * kScanXBytes, c, warp, g8, t4);
        ok = group_all<kScanWarps * 32>(1, ok);
        // Past the barrier the next step's loads have had time to complete.
        if (j + 1 < nseg && ok) stage_release(&empty[(j + 1) % kScanStages], lane);
    }
    __nv_bfloat16* const fin = compose ? (part ? a.gmap[1] : a.gmap[0]) : a.final_state;
    if (ok && fin) copy_rows_out(xbuf + (nseg & 1) * kScanXBytes, fin + rows0 * kHeadDim, tid);
}

// ---------------------------------------------------------------------------
// Last level of a two-level chain: for segment s, the i-th of its group g,
// the incoming state S_s = S_g P_F[s - 1] + P_Z[s - 1] (i >= 1; S_g itself for
// i = 0), where S_g is the group's incoming state and (P_F, P_Z) the map of
// the group's segments before s.  One CTA per (segment, head), all 128 value
// rows: four warps each form 32 key columns of S_s^T = P_F^T S_g^T + P_Z^T
// (warp MMA, BF16 operands, FP32 accumulation) from the three TMA-staged
// states, and the rows leave through shared memory in 16-byte stores.
// ---------------------------------------------------------------------------
constexpr int kApplyWarps = 4;
constexpr uint32_t kApplyTile = kHeadDim * kHeadDim * 2;   // one state, two SW128 slabs [128][64]
constexpr uint32_t kApplyOut = 3 * kApplyTile;            // output rows, XOR-swizzled [128][128]
constexpr uint32_t kApplyBar = 4 * kApplyTile;
constexpr uint32_t kApplySmemBytes = kApplyBar + 8 + 1024;

struct ApplyArgs {
    const __nv_bfloat16* group_starts;   // S_g: [N groups][H][128][128]
    __nv_bfloat16* starts;               // S_s: [N segs][H][128][128]
    int64_t segs, groups, group_segs, H;
    int* status;
};

__device__ __forceinline__ uint32_t out_off(uint32_t v, uint32_t ch) {
    return v * (kHeadDim * 2) + ((ch ^ (v & 7u)) << 4);
}

__global__ void __launch_bounds__(kApplyWarps * 32, 1)
    segment_apply_kernel(ApplyArgs a, const __grid_constant__ CUtensorMap pfmap,
                         const __grid_constant__ CUtensorMap pzmap,
                         const __grid_constant__ CUtensorMap sgmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kApplyBar);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tid = threadIdx.x;
    const int64_t sh = blockIdx.x;
    const int64_t seg = sh / a.H;
    const int64_t h = sh - seg * a.H;
    const int64_t sq = seg / a.segs;
    const int64_t sl = seg - sq * a.segs;
    const int64_t gi = sl / a.group_segs;
    const int64_t i = sl - gi * a.group_segs;
    const int64_t g = sq * a.groups + gi;
    __nv_bfloat16* dst = a.starts + (seg * a.H + h) * kHeadDim * kHeadDim;
    if (i == 0) {
        // The group's first segment starts from the group's incoming state.
        const uint4* src = reinterpret_cast<const uint4*>(a.group_starts + (g * a.H + h) * kHeadDim * kHeadDim);
        for (int q = tid; q < static_cast<int>(kApplyTile / 16); q += kApplyWarps * 32)
            reinterpret_cast<uint4*>(dst)[q] = src[q];
        return;
    }
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
        const int32_t prow = static_cast<int32_t>(((seg - 1) * a.H + h) * kHeadDim);
        const int32_t grow = static_cast<int32_t>((g * a.H + h) * kHeadDim);
        mbar_arrive_expect_tx(bar, 3 * kApplyTile);
        tma_load_2d(smem, &pfmap, 0, prow, bar);
        tma_load_2d(smem + kApplyTile / 2, &pfmap, 64, prow, bar);
        tma_load_2d(smem + kApplyTile, &pzmap, 0, prow, bar);
        tma_load_2d(smem + kApplyTile + kApplyTile / 2, &pzmap, 64, prow, bar);
        tma_load_2d(smem + 2 * kApplyTile, &sgmap, 0, grow, bar);
        tma_load_2d(smem + 2 * kApplyTile + kApplyTile / 2, &sgmap, 64, grow, bar);
    }
    __syncthreads();
    const bool ok = mbar_wait_warp(bar, 0, a.status);
    if (!__all_sync(0xffffffffu, ok)) return;   // bounded wait ran out (status is set)

    const uint8_t* tf = smem;                   // P_F rows (old key) x columns (new key)
    const uint8_t* tz = smem + kApplyTile;      // P_Z rows (value) x columns (new key)
    const uint8_t* ts = smem + 2 * kApplyTile;  // S_g rows (value) x columns (old key)
    uint8_t* out = smem + kApplyOut;
    const int g8 = lane >> 2, t4 = lane & 3;
    const uint32_t mi = lane >> 3, r8 = lane & 7;

    // Accumulators: P_Z^T tiles (m = new key 32 warp + 16 mt .., n = value 8 nt ..).
    float acc[2][16][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t z[4];
            const uint32_t v = 8 * (2 * np + (mi >> 1)) + r8;
            const uint32_t ch = 4 * warp + 2 * mt + (mi & 1);
            ldsm_x4_trans(z, smem_u32(tz + sw128_off(kHeadDim, v, ch)));
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                acc[mt][2 * np + e][0] = bf_lo(z[2 * e]);
                acc[mt][2 * np + e][1] = bf_hi(z[2 * e]);
                acc[mt][2 * np + e][2] = bf_lo(z[2 * e + 1]);
                acc[mt][2 * np + e][3] = bf_hi(z[2 * e + 1]);
            }
        }
    // + P_F^T S_g^T over the 128 old keys.
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t af[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
            const uint32_t row = 16 * kk + r8 + 8 * (mi >> 1);
            const uint32_t ch = 4 * warp + 2 * mt + (mi & 1);
            ldsm_x4_trans(af[mt], smem_u32(tf + sw128_off(kHeadDim, row, ch)));
        }
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t b[4];   // S_g^T (k = old key, n = value) for value tiles 2 np, 2 np + 1
            const uint32_t v = 8 * (2 * np + (mi >> 1)) + r8;
            ldsm_x4(b, smem_u32(ts + sw128_off(kHeadDim, v, 2 * kk + (mi & 1))));
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                mma_bf16(acc[mt][2 * np], af[mt], b, acc[mt][2 * np]);
                mma_bf16(acc[mt][2 * np + 1], af[mt], b + 2, acc[mt][2 * np + 1]);
            }
        }
    }
    // S_s rows (value) x key, BF16, through shared memory.
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const uint32_t lo = movm_trans(pack_bf16(acc[mt][nt][0], acc[mt][nt][1]));
            const uint32_t hi = movm_trans(pack_bf16(acc[mt][nt][2], acc[mt][nt][3]));
            const uint32_t v = 8 * nt + g8;
            const uint32_t base = 32 * warp + 16 * mt;
            *reinterpret_cast<uint32_t*>(out + out_off(v, base / 8) + 4 * t4) = lo;
            *reinterpret_cast<uint32_t*>(out + out_off(v, base / 8 + 1) + 4 * t4) = hi;
        }
    __syncthreads();
    for (int q = tid; q < static_cast<int>(kApplyTile / 16); q += kApplyWarps * 32) {
        const uint32_t v = q >> 4, ch = q & 15;
        reinterpret_cast<uint4*>(dst)[q] = *reinterpret_cast<const uint4*>(out + out_off(v, ch));
    }
}

// Segments of a packed batch (one block): sequence n, of c_n chunks, gets
// ceil(c_n / L) segments of L chunks (the last one shorter; none when empty),
// numbered sequence by sequence.  Writes seg_begin[0..N], and for segment s
// its first chunk seg_chunks[s] and first token seg_tokens[s]; entries from
// the last segment to bound s_ub repeat the batch's end, so segments past the
// real ones are empty.  Runs after the varlen metadata and exits when it found
// the offsets invalid (every later kernel then returns at once); a count
// above s_ub (impossible for valid offsets) invalidates the batch as well.
constexpr int kSegMetaThreads = 1024;

__global__ void __launch_bounds__(kSegMetaThreads)
    segment_meta_kernel(const int64_t* cu, const int64_t* cu_chunks, int32_t* valid, int64_t N,
                        int64_t L, int64_t s_ub, int64_t* seg_begin, int64_t* seg_chunks,
                        int64_t* seg_tokens, int64_t* seg_seq, int* status) {
    __shared__ int64_t warp_sums[kSegMetaThreads / 32];
    __shared__ int64_t carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!*valid) return;
    if (tid == 0) {
        carry = 0;
        seg_begin[0] = 0;
    }
    __syncthreads();
    for (int64_t base = 0; base < N; base += kSegMetaThreads) {
        const int64_t n = base + tid;
        const int64_t cnt = n < N ? (cu_chunks[n + 1] - cu_chunks[n] + L - 1) / L : 0;
        int64_t x = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int64_t w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int64_t incl = x + (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
        if (n < N) {
            seg_begin[n + 1] = incl;
            const int64_t s0 = incl - cnt;
            for (int64_t j = 0; j < cnt && s0 + j < s_ub; ++j) {
                seg_chunks[s0 + j] = cu_chunks[n] + j * L;
                seg_tokens[s0 + j] = cu[n] + kChunk * j * L;
                seg_seq[s0 + j] = n;
            }
        }
        __syncthreads();
        if (tid == kSegMetaThreads - 1) carry = incl;
        __syncthreads();
    }
    const int64_t total = carry;
    if (total > s_ub) {
        if (tid == 0) {
            *valid = 0;
            atomicOr(status, kDevBadSeqlens);
        }
        return;
    }
    for (int64_t sidx = total + tid; sidx <= s_ub; sidx += kSegMetaThreads) {
        seg_chunks[sidx] = cu_chunks[N];
        seg_tokens[sidx] = cu[N];
        if (sidx < s_ub) seg_seq[sidx] = 0;
    }
}

}  // namespace

cudaError_t launch_segment_scan(const void* init_state, void* final_state, const void* transitions,
                                const void* zero_start_states, void* starts, int64_t n_seqs,
                                int64_t segs, const int64_t* seg_begin, const int32_t* valid,
                                int64_t H, int* status, cudaStream_t stream) {
    const int64_t blocks = n_seqs * H * (kHeadDim / kScanRows);
    if (blocks <= 0) return cudaSuccess;
    const int64_t total_segs = seg_begin ? segs : n_seqs * segs;
    const int64_t rows = (total_segs > 0 ? total_segs : 1) * H * kHeadDim;
    if (rows >= (int64_t(1) << 31) || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    static bool configured[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(segment_scan_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kScanSmemBytes));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    CUtensorMap fmap, zmap;
    cudaError_t e = encode_state_map(&fmap, transitions, rows, kHeadDim);
    if (e == cudaSuccess) e = encode_state_map(&zmap, zero_start_states, rows, kScanRows);
    if (e != cudaSuccess) return e;
    ScanArgs a;
    a.init_state = static_cast<const __nv_bfloat16*>(init_state);
    a.final_state = static_cast<__nv_bfloat16*>(final_state);
    a.starts = static_cast<__nv_bfloat16*>(starts);
    a.segs = segs;
    a.seg_begin = seg_begin;
    a.valid = valid;
    a.groups = 0;
    a.group_segs = 0;
    a.src[0] = a.src[1] = nullptr;
    a.prefix[0] = a.prefix[1] = nullptr;
    a.gmap[0] = a.gmap[1] = nullptr;
    a.H = H;
    a.status = status;
    segment_scan_kernel<<<static_cast<unsigned>(blocks), (kScanWarps + 1) * 32, kScanSmemBytes,
                          stream>>>(a, fmap, zmap);
    return cudaGetLastError();
}

cudaError_t launch_segment_meta(const int64_t* cu_seqlens, const int64_t* cu_chunks, int32_t* valid,
                                int64_t n_seqs, int64_t seg_chunks_len, int64_t s_ub,
                                int64_t* seg_begin, int64_t* seg_chunks, int64_t* seg_tokens,
                                int64_t* seg_seq, int* status, cudaStream_t stream) {
    if (n_seqs <= 0 || seg_chunks_len <= 0) return cudaErrorInvalidValue;
    segment_meta_kernel<<<1, kSegMetaThreads, 0, stream>>>(cu_seqlens, cu_chunks, valid, n_seqs,
                                                          seg_chunks_len, s_ub, seg_begin,
                                                          seg_chunks, seg_tokens, seg_seq, status);
    return cudaGetLastError();
}

namespace {

bool configure_scan(int dev) {
    static bool configured[64] = {};
    if (dev < 0 || dev >= 64) return false;
    if (!configured[dev]) {
        if (cudaFuncSetAttribute(segment_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kScanSmemBytes)) != cudaSuccess ||
            cudaFuncSetAttribute(segment_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kApplySmemBytes)) != cudaSuccess)
            return false;
        configured[dev] = true;
    }
    return true;
}

}  // namespace

cudaError_t launch_segment_compose(const void* transitions, const void* zero_start_states,
                                   void* prefix_f, void* prefix_z, void* group_f, void* group_z,
                                   int64_t n_seqs, int64_t segs, int64_t group_segs,
                                   int64_t groups, int64_t H, int* status, cudaStream_t stream) {
    const int64_t blocks = 2 * n_seqs * groups * H * (kHeadDim / kScanRows);
    if (blocks <= 0) return cudaSuccess;
    const int64_t rows = n_seqs * segs * H * kHeadDim;
    if (rows >= (int64_t(1) << 31) || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !configure_scan(dev)) return cudaErrorInvalidDevice;
    CUtensorMap fmap, zmap;
    cudaError_t e = encode_state_map(&fmap, transitions, rows, kHeadDim);
    if (e == cudaSuccess) e = encode_state_map(&zmap, zero_start_states, rows, kScanRows);
    if (e != cudaSuccess) return e;
    ScanArgs a;
    a.init_state = nullptr;
    a.final_state = nullptr;
    a.starts = nullptr;
    a.seg_begin = nullptr;
    a.valid = nullptr;
    a.segs = segs;
    a.H = H;
    a.status = status;
    a.groups = groups;
    a.group_segs = group_segs;
    a.src[0] = static_cast<const __nv_bfloat16*>(transitions);
    a.src[1] = static_cast<const __nv_bfloat16*>(zero_start_states);
    a.prefix[0] = static_cast<__nv_bfloat16*>(prefix_f);
    a.prefix[1] = static_cast<__nv_bfloat16*>(prefix_z);
    a.gmap[0] = static_cast<__nv_bfloat16*>(group_f);
    a.gmap[1] = static_cast<__nv_bfloat16*>(group_z);
    segment_scan_kernel<<<static_cast<unsigned>(blocks), (kScanWarps + 1) * 32, kScanSmemBytes,
                          stream>>>(a, fmap, zmap);
    return cudaGetLastError();
}

cudaError_t launch_segment_apply(const void* group_starts, const void* prefix_f, const void* prefix_z,
                                 void* starts, int64_t n_seqs, int64_t segs, int64_t group_segs,
                                 int64_t groups, int64_t H, int* status, cudaStream_t stream) {
    const int64_t blocks = n_seqs * segs * H;
    if (blocks <= 0) return cudaSuccess;
    const int64_t rows = n_seqs * segs * H * kHeadDim;
    const int64_t grows = n_seqs * groups * H * kHeadDim;
    if (rows >= (int64_t(1) << 31) || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !configure_scan(dev)) return cudaErrorInvalidDevice;
    CUtensorMap pfmap, pzmap, sgmap;
    cudaError_t e = encode_state_map(&pfmap, prefix_f, rows, kHeadDim);
    if (e == cudaSuccess) e = encode_state_map(&pzmap, prefix_z, rows, kHeadDim);
    if (e == cudaSuccess) e = encode_state_map(&sgmap, group_starts, grows, kHeadDim);
    if (e != cudaSuccess) return e;
    ApplyArgs a;
    a.group_starts = static_cast<const __nv_bfloat16*>(group_starts);
    a.starts = static_cast<__nv_bfloat16*>(starts);
    a.segs = segs;
    a.groups = groups;
    a.group_segs = group_segs;
    a.H = H;
    a.status = status;
    segment_apply_kernel<<<static_cast<unsigned>(blocks), kApplyWarps * 32, kApplySmemBytes, stream>>>(
        a, pfmap, pzmap, sgmap);
    return cudaGetLastError();
}

}  // namespace kda
