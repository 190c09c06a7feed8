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
// independently.  Eight warps each form 16 key columns of the new rows as
// (S_{j+1})^T = F_j^T S_j^T + Z_j^T on the warp MMA (BF16 operands, FP32
// accumulation; the FP32 rows stay in registers), and swap their BF16 slices
// through shared memory for the next step's operand.  The transition pass
// stores F and Z in the MMA's fragment order (kda_segmap.cuh), so each warp
// loads its A tiles of F_j^T and its C tile of Z_j^T straight into registers,
// two steps ahead, with one coalesced load per tile: every CTA needs all of
// F_j each step, and staging it through shared memory (a TMA copy in, a
// transposing ldmatrix out) made that traffic the step's bound.
#include <cuda.h>

#include "kda_common.cuh"
#include "kda_segmap.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kScanRows = 8;     // value rows of the state per CTA
constexpr int kScanWarps = 8;    // warps, 16 keys (one m tile) each
constexpr int kScanThreads = kScanWarps * 32;
constexpr uint32_t kScanXBytes = kScanRows * kHeadDim * 2;     // one BF16 copy of the CTA's rows
constexpr int64_t kMapElems = int64_t(kHeadDim) * kHeadDim;    // one map or state

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

// Read-only loads of map fragments (the maps are written by an earlier launch).
__device__ __forceinline__ uint4 ld_map16(const uint8_t* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ld_map8(const uint8_t* p) {
    uint2 r;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

struct ScanArgs {
    const __nv_bfloat16* init_state;   // [N][H][128][128] or null
    __nv_bfloat16* final_state;        // [N][H][128][128] or null
    __nv_bfloat16* starts;             // [segments][H][128][128]
    // F maps (fmap_frag_off order) and Z states (zmap_frag_off order),
    // [total][H] of 32 KB each.
    const uint8_t* fmaps;
    const uint8_t* zmaps;
    int64_t total;
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
    // F maps (no Z), the second half the Z maps (adding Z):
    // state_0 = map gs, state_j = state_{j-1} F_{gs+j} (+ Z_{gs+j}); state_j
    // goes to prefix[p][gs + j] (rows) and the last one to gmap[p][n], in the
    // fragment order of its kind so that the chain over the groups reads it
    // like the segment maps.
    int64_t groups, group_segs;
    __nv_bfloat16* prefix[2];
    __nv_bfloat16* gmap[2];
};

// Warp w's slice (keys 16 w .. 16 w + 15 of the CTA's 8 rows) of a state in
// C-fragment form (m = key, n = value row), rounded to BF16, into the copy at x.
__device__ __forceinline__ void put_rows(uint8_t* x, const float (&c)[4], int w, int g8, int t4) {
    const uint32_t lo = movm_trans(pack_bf16(c[0], c[1]));   // row g8, keys 16 w + 2 t4
    const uint32_t hi = movm_trans(pack_bf16(c[2], c[3]));   // keys 16 w + 8 + 2 t4
    *reinterpret_cast<uint32_t*>(x + x_off(g8, 2 * w) + 4 * t4) = lo;
    *reinterpret_cast<uint32_t*>(x + x_off(g8, 2 * w + 1) + 4 * t4) = hi;
}

// The CTA's 8 rows from the copy at x into rows [8][128] at dst (thread tid
// < 128 copies 16 bytes).
__device__ __forceinline__ void copy_rows_out(const uint8_t* x, __nv_bfloat16* dst, int tid) {
    const int v = tid >> 4, ch = tid & 15;
    const uint4 val = *reinterpret_cast<const uint4*>(x + x_off(v, ch));
    *reinterpret_cast<uint4*>(dst + v * kHeadDim + 8 * ch) = val;
}

// Byte offset, within one map, of this lane's 8 bytes of C-fragment data for
// m tile mt and value tile nt: in an F map the half of A tile (mt, nt / 2)
// that holds value tile nt; in a Z map C tile (nt, mt).
__device__ __forceinline__ uint32_t cfrag_off(bool fmap, uint32_t mt, uint32_t nt, uint32_t lane) {
    return fmap ? fmap_frag_off(mt, nt >> 1, lane) + 8 * (nt & 1) : zmap_frag_off(nt, mt, lane);
}

__global__ void __launch_bounds__(kScanThreads, 2) segment_scan_kernel(ScanArgs a) {
    __shared__ __align__(128) uint8_t xbuf[2 * kScanXBytes];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tid = threadIdx.x;
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
    const int vt = static_cast<int>(blk - nh * kGroups);   // value tile: rows 8 vt .. 8 vt + 7
    const int v0 = kScanRows * vt;
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
    // Every map read below lies inside the [total][H] arrays.
    if (first < 0 || nseg < 0 || step0 + nseg > a.total) {
        if (tid == 0) atomicOr(a.status, kDevBadSeqlens);
        return;
    }
    const bool add_z = !compose || part == 1;
    __nv_bfloat16* const starts = compose ? (part ? a.prefix[1] : a.prefix[0]) : a.starts;
    const int g8 = lane >> 2, t4 = lane & 3;
    const int64_t rows0 = (n * a.H + h) * kHeadDim + v0;   // first row of this CTA in [N][H][128]

    // S_0^T for keys 16 warp + {g8, g8 + 8}, rows v0 + 2 t4 + {0, 1}: the
    // caller's initial state (rows), or when composing the group's first
    // segment map (fragment order).
    float c[4];
    if (compose) {
        const uint8_t* src = (part ? a.zmaps : a.fmaps) + (first * a.H + h) * kMapElems * 2;
        const uint2 p = ld_map8(src + cfrag_off(part == 0, warp, vt, lane));
        c[0] = bf_lo(p.x);
        c[1] = bf_hi(p.x);
        c[2] = bf_lo(p.y);
        c[3] = bf_hi(p.y);
    } else if (a.init_state) {
        const __nv_bfloat16* src = a.init_state + (rows0 + 2 * t4) * kHeadDim + 16 * warp + g8;
        c[0] = __bfloat162float(src[0]);
        c[1] = __bfloat162float(src[kHeadDim]);
        c[2] = __bfloat162float(src[8]);
        c[3] = __bfloat162float(src[kHeadDim + 8]);
    } else {
        c[0] = c[1] = c[2] = c[3] = 0.f;
    }
    put_rows(xbuf, c, warp, g8, t4);

    // Step j's operands straight into registers: this warp's eight A tiles of
    // F_j^T (m tile = warp) and its C tile of Z_j^T.  Two register sets: the
    // loads of step j + 2 go out as soon as step j's MMAs have taken theirs.
    uint32_t af[2][8][4], zf[2][2];
    const int64_t map_stride = a.H * kMapElems * 2;   // bytes from one segment's map to the next
    const uint8_t* fcur = a.fmaps + (step0 * a.H + h) * kMapElems * 2 + fmap_frag_off(warp, 0, lane);
    const uint8_t* zcur = a.zmaps + (step0 * a.H + h) * kMapElems * 2 + zmap_frag_off(vt, warp, lane);
    auto load_step = [&](int buf, int64_t j) {
        const uint8_t* fp = fcur + j * map_stride;
#pragma unroll
        for (int kt = 0; kt < 8; ++kt) {
            const uint4 r = ld_map16(fp + kt * 512);
            af[buf][kt][0] = r.x;
            af[buf][kt][1] = r.y;
            af[buf][kt][2] = r.z;
            af[buf][kt][3] = r.w;
        }
        if (add_z) {
            const uint2 r = ld_map8(zcur + j * map_stride);
            zf[buf][0] = r.x;
            zf[buf][1] = r.y;
        } else {
            zf[buf][0] = zf[buf][1] = 0u;
        }
    };
    if (nseg > 0) load_step(0, 0);
    if (nseg > 1) load_step(1, 1);
    __syncthreads();

    const uint32_t mi = lane >> 3, r8 = lane & 7;
    // One step with register set `buf`.
    auto step = [&](int buf, int64_t j) {
        const uint8_t* xc = xbuf + (j & 1) * kScanXBytes;
        // Accumulators: Z_j^T (even k tiles; zero when composing the F maps)
        // and zero (odd k tiles).
        float acc[2][4];
        acc[0][0] = bf_lo(zf[buf][0]);
        acc[0][1] = bf_hi(zf[buf][0]);
        acc[0][2] = bf_lo(zf[buf][1]);
        acc[0][3] = bf_hi(zf[buf][1]);
        acc[1][0] = acc[1][1] = acc[1][2] = acc[1][3] = 0.f;
        // B operand: S_j^T (k = key of S_j, n = value row), two k tiles per load.
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
            uint32_t r[4];
            ldsm_x4(r, smem_u32(xc + x_off(r8, 4 * kp + mi)));
            mma_bf16(acc[0], af[buf][2 * kp], r, acc[0]);
            mma_bf16(acc[1], af[buf][2 * kp + 1], r + 2, acc[1]);
        }
        if (j + 2 < nseg) load_step(buf, j + 2);
        // S_j out as this segment's incoming state.
        if (tid < 128) copy_rows_out(xc, starts + (((first + j) * a.H + h) * kHeadDim + v0) * kHeadDim, tid);
#pragma unroll
        for (int e = 0; e < 4; ++e) c[e] = acc[0][e] + acc[1][e];
        put_rows(xbuf + ((j + 1) & 1) * kScanXBytes, c, warp, g8, t4);
        __syncthreads();
    };
    for (int64_t j = 0; j < nseg; j += 2) {
        step(0, j);
        if (j + 1 < nseg) step(1, j + 1);
    }
    if (compose) {
        // The group's map, in the fragment order of its kind.
        uint8_t* dst = reinterpret_cast<uint8_t*>(part ? a.gmap[1] : a.gmap[0]) + (n * a.H + h) * kMapElems * 2;
        *reinterpret_cast<uint2*>(dst + cfrag_off(part == 0, warp, vt, lane)) =
            make_uint2(pack_bf16(c[0], c[1]), pack_bf16(c[2], c[3]));
    } else if (a.final_state && tid < 128) {
        copy_rows_out(xbuf + (nseg & 1) * kScanXBytes, a.final_state + rows0 * kHeadDim, tid);
    }
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
    if (total_segs * H * kHeadDim >= (int64_t(1) << 31) || blocks > 0x7fffffffLL)
        return cudaErrorInvalidValue;
    ScanArgs a;
    a.init_state = static_cast<const __nv_bfloat16*>(init_state);
    a.final_state = static_cast<__nv_bfloat16*>(final_state);
    a.starts = static_cast<__nv_bfloat16*>(starts);
    a.fmaps = static_cast<const uint8_t*>(transitions);
    a.zmaps = static_cast<const uint8_t*>(zero_start_states);
    a.total = total_segs;
    a.segs = segs;
    a.seg_begin = seg_begin;
    a.valid = valid;
    a.groups = 0;
    a.group_segs = 0;
    a.prefix[0] = a.prefix[1] = nullptr;
    a.gmap[0] = a.gmap[1] = nullptr;
    a.H = H;
    a.status = status;
    segment_scan_kernel<<<static_cast<unsigned>(blocks), kScanThreads, 0, stream>>>(a);
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
        if (cudaFuncSetAttribute(segment_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
    ScanArgs a;
    a.init_state = nullptr;
    a.final_state = nullptr;
    a.starts = nullptr;
    a.fmaps = static_cast<const uint8_t*>(transitions);
    a.zmaps = static_cast<const uint8_t*>(zero_start_states);
    a.total = n_seqs * segs;
    a.seg_begin = nullptr;
    a.valid = nullptr;
    a.segs = segs;
    a.H = H;
    a.status = status;
    a.groups = groups;
    a.group_segs = group_segs;
    a.prefix[0] = static_cast<__nv_bfloat16*>(prefix_f);
    a.prefix[1] = static_cast<__nv_bfloat16*>(prefix_z);
    a.gmap[0] = static_cast<__nv_bfloat16*>(group_f);
    a.gmap[1] = static_cast<__nv_bfloat16*>(group_z);
    segment_scan_kernel<<<static_cast<unsigned>(blocks), kScanThreads, 0, stream>>>(a);
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
