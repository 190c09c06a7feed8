// kda_prep.cu -- chunk preparation for KDA prefill (sm_103a).
//
// One warp prepares one (chunk, head): 16 tokens of q, k, g and beta in, one
// packet (kda_common.cuh) out.  Following "FlashKDA column split", section 1,
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
#include "kda_common.cuh"
#include "kda_launch.h"

namespace kda {
namespace {

constexpr int kPrepWarps = 2;
// Per-warp shared memory: the packet image, then scratch tiles (16 x 128 BF16,
// SW128): exp(-G) khat split into a BF16 high part and the BF16 rounding of
// the remainder, the low parts of K^start and s Q^start (their high parts are
// the packet tiles), K^end in token-row layout for the transpose, and R in FP32.
constexpr uint32_t kPrepOffKinv = kPacketBytes;
constexpr uint32_t kPrepOffKinvLo = kPacketBytes + 4096;
constexpr uint32_t kPrepOffKsLo = kPacketBytes + 8192;
constexpr uint32_t kPrepOffQsLo = kPacketBytes + 12288;
constexpr uint32_t kPrepOffKen = kPacketBytes + 16384;
constexpr uint32_t kPrepOffR = kPacketBytes + 20480;          // 16 x 16 FP32
constexpr uint32_t kPrepWarpSmem = kPacketBytes + 20480 + 1024;

struct PrepArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const float* g;
    const __nv_bfloat16* beta;
    uint8_t* packets;
    SeqGeometry geo;
    int64_t H;
    int64_t n_chunk_heads;
    float scale;
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

__device__ __forceinline__ uint2 ldg_nc_u2(const void* p) {
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ float4 ldg_nc_f4(const void* p) {
    float4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
                 : "l"(p));
    return r;
}

// Store 4 consecutive BF16 (channels 4*lane .. 4*lane+3) of token row t into a
// [16][128] SW128 tile.
__device__ __forceinline__ void st_row4(uint8_t* tile, int t, int lane, float a, float b, float c,
                                        float d) {
    uint32_t off = sw128_off(16, t, (4 * lane) >> 3) + ((lane & 1) << 3);
    uint2 v = make_uint2(pack_bf16(a, b), pack_bf16(c, d));
    *reinterpret_cast<uint2*>(tile + off) = v;
}
// Same, storing the BF16 rounding in `hi` and the BF16 rounding of what it
// left out in `lo`, so that hi + lo carries about 16 significant bits.
__device__ __forceinline__ void st_row4_split(uint8_t* hi, uint8_t* lo, int t, int lane, float a,
                                              float b, float c, float d) {
    uint32_t off = sw128_off(16, t, (4 * lane) >> 3) + ((lane & 1) << 3);
    const uint32_t h0 = pack_bf16(a, b), h1 = pack_bf16(c, d);
    const uint32_t l0 = pack_bf16(a - bf16_lo(h0), b - bf16_hi(h0));
    const uint32_t l1 = pack_bf16(c - bf16_lo(h1), d - bf16_hi(h1));
    *reinterpret_cast<uint2*>(hi + off) = make_uint2(h0, h1);
    *reinterpret_cast<uint2*>(lo + off) = make_uint2(l0, l1);
}

__global__ void __launch_bounds__(kPrepWarps * 32) prep_kernel(PrepArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * kPrepWarps + warp;
    if (wid >= a.n_chunk_heads) return;
    const int64_t c = wid / a.H;
    const int64_t h = wid - c * a.H;

    // Token range of this chunk.
    int64_t t0, len;
    if (a.geo.cu_chunks) {
        if (!*a.geo.valid) return;
        if (c >= a.geo.cu_chunks[a.geo.n_seqs]) return;
        const int64_t n = find_sequence(a.geo.cu_chunks, a.geo.n_seqs, c);
        t0 = a.geo.cu_seqlens[n] + kChunk * (c - a.geo.cu_chunks[n]);
        len = a.geo.cu_seqlens[n + 1] - t0;
    } else {
        const int64_t n = c / a.geo.chunks_per_seq;
        const int64_t ci = c - n * a.geo.chunks_per_seq;
        t0 = n * a.geo.tokens_per_seq + kChunk * ci;
        len = a.geo.tokens_per_seq - kChunk * ci;
    }
    if (len > kChunk) len = kChunk;

    uint8_t* ws = smem + warp * kPrepWarpSmem;
    uint8_t* tKS = ws + kOffKS;
    uint8_t* tQS = ws + kOffQS;
    uint8_t* tKE = ws + kOffKE;
    uint8_t* tAKB = ws + kOffAKB;
    uint8_t* tAQK = ws + kOffAQK;
    float* tD = reinterpret_cast<float*>(ws + kOffD);
    uint8_t* tKinv = ws + kPrepOffKinv;
    uint8_t* tKinvLo = ws + kPrepOffKinvLo;
    uint8_t* tKsLo = ws + kPrepOffKsLo;
    uint8_t* tQsLo = ws + kPrepOffQsLo;
    uint8_t* tKen = ws + kPrepOffKen;
    float* tR = reinterpret_cast<float*>(ws + kPrepOffR);

    // ---- 1. Load q, k (BF16, 4 channels per lane), g (running sum -> G), beta.
    uint2 qv[kChunk], kv[kChunk];
    float G[kChunk][4];
    float red[2 * kChunk];   // partial sums of squares: q tokens 0..15, k tokens 0..15
    float run0 = 0.f, run1 = 0.f, run2 = 0.f, run3 = 0.f;
#pragma unroll
    for (int t = 0; t < kChunk; ++t) {
        if (t < len) {
            const int64_t off = ((t0 + t) * a.H + h) * kHeadDim + 4 * lane;
            qv[t] = ldg_nc_u2(a.q + off);
            kv[t] = ldg_nc_u2(a.k + off);
            const float4 gg = ldg_nc_f4(a.g + off);
            run0 += gg.x;
            run1 += gg.y;
            run2 += gg.z;
            run3 += gg.w;
        } else {
            qv[t] = make_uint2(0u, 0u);
            kv[t] = make_uint2(0u, 0u);
        }
        G[t][0] = run0;
        G[t][1] = run1;
        G[t][2] = run2;
        G[t][3] = run3;
        const float q0 = bf16_lo(qv[t].x), q1 = bf16_hi(qv[t].x), q2 = bf16_lo(qv[t].y),
                    q3 = bf16_hi(qv[t].y);
        const float k0 = bf16_lo(kv[t].x), k1 = bf16_hi(kv[t].x), k2 = bf16_lo(kv[t].y),
                    k3 = bf16_hi(kv[t].y);
        red[t] = q0 * q0 + q1 * q1 + q2 * q2 + q3 * q3;
        red[kChunk + t] = k0 * k0 + k1 * k1 + k2 * k2 + k3 * k3;
    }
    float beta_f = 0.f;   // lane t < len holds beta of token t
    if (lane < len) beta_f = __bfloat162float(a.beta[(t0 + lane) * a.H + h]);

    // ---- 2. Sums of squares over the 128 channels: butterfly reduce-scatter.
    // After the step with offset o, element i stands for original index
    // i + o * (bit o of lane); at the end lane l holds the total of index l.
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = up ? red[i] : red[i + o];
            const float keep = up ? red[i + o] : red[i];
            red[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    const float rnorm = rsqrtf(red[0] + 1e-6f);   // lane < 16: 1/|q_lane|, else 1/|k_(lane-16)|

    // ---- 3. Decayed operands.
    const float e_last0 = __expf(G[kChunk - 1][0]), e_last1 = __expf(G[kChunk - 1][1]);
    const float e_last2 = __expf(G[kChunk - 1][2]), e_last3 = __expf(G[kChunk - 1][3]);
    *reinterpret_cast<float4*>(tD + 4 * lane) = make_float4(e_last0, e_last1, e_last2, e_last3);
    const float s = a.scale;
#pragma unroll
    for (int t = 0; t < kChunk; ++t) {
        const float rq = __shfl_sync(0xffffffffu, rnorm, t);
        const float rk = __shfl_sync(0xffffffffu, rnorm, kChunk + t);
        const float kh0 = bf16_lo(kv[t].x) * rk, kh1 = bf16_hi(kv[t].x) * rk;
        const float kh2 = bf16_lo(kv[t].y) * rk, kh3 = bf16_hi(kv[t].y) * rk;
        const float qh0 = bf16_lo(qv[t].x) * rq, qh1 = bf16_hi(qv[t].x) * rq;
        const float qh2 = bf16_lo(qv[t].y) * rq, qh3 = bf16_hi(qv[t].y) * rq;
        const float e0 = __expf(G[t][0]), e1 = __expf(G[t][1]);
        const float e2 = __expf(G[t][2]), e3 = __expf(G[t][3]);
        const float i0 = __expf(-G[t][0]), i1 = __expf(-G[t][1]);
        const float i2 = __expf(-G[t][2]), i3 = __expf(-G[t][3]);
        st_row4_split(tKS, tKsLo, t, lane, e0 * kh0, e1 * kh1, e2 * kh2, e3 * kh3);
        st_row4_split(tQS, tQsLo, t, lane, s * e0 * qh0, s * e1 * qh1, s * e2 * qh2, s * e3 * qh3);
        st_row4_split(tKinv, tKinvLo, t, lane, i0 * kh0, i1 * kh1, i2 * kh2, i3 * kh3);
        st_row4(tKen, t, lane, (e_last0 * i0) * kh0, (e_last1 * i1) * kh1,
                (e_last2 * i2) * kh2, (e_last3 * i3) * kh3);
    }
    __syncwarp();

    // ---- 4. Scores: A^qk = (s Q^start)(K exp(-G))^T and K^start (K exp(-G))^T,
    // each as hi*hi + hi*lo + lo*hi of the split BF16 operands (FP32 accumulate).
    const int gq = lane >> 2, tq = lane & 3;
    float acc_qk[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    float acc_kk[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
        const uint32_t rowA = (lane & 7) + ((lane >> 3) & 1) * 8;
        const uint32_t rowB = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t aq[4], ak[4], bk[4], aql[4], akl[4], bkl[4];
            const uint32_t offA = sw128_off(16, rowA, 2 * kk + (lane >> 4));
            const uint32_t offB = sw128_off(16, rowB, 2 * kk + ((lane >> 3) & 1));
            ldsm_x4(aq, smem_u32(tQS + offA));
            ldsm_x4(ak, smem_u32(tKS + offA));
            ldsm_x4(bk, smem_u32(tKinv + offB));
            ldsm_x4(aql, smem_u32(tQsLo + offA));
            ldsm_x4(akl, smem_u32(tKsLo + offA));
            ldsm_x4(bkl, smem_u32(tKinvLo + offB));
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                mma_bf16(acc_qk[nt], aq, bk + 2 * nt, acc_qk[nt]);
                mma_bf16(acc_qk[nt], aq, bkl + 2 * nt, acc_qk[nt]);
                mma_bf16(acc_qk[nt], aql, bk + 2 * nt, acc_qk[nt]);
                mma_bf16(acc_kk[nt], ak, bk + 2 * nt, acc_kk[nt]);
                mma_bf16(acc_kk[nt], ak, bkl + 2 * nt, acc_kk[nt]);
                mma_bf16(acc_kk[nt], akl, bk + 2 * nt, acc_kk[nt]);
            }
        }
    }
    const float beta_r0 = __shfl_sync(0xffffffffu, beta_f, gq);
    const float beta_r1 = __shfl_sync(0xffffffffu, beta_f, gq + 8);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int j0 = 8 * nt + 2 * tq;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int i = gq + 8 * hh;
            const float q0 = (j0 <= i) ? acc_qk[nt][2 * hh] : 0.f;
            const float q1 = (j0 + 1 <= i) ? acc_qk[nt][2 * hh + 1] : 0.f;
            *reinterpret_cast<uint32_t*>(tAQK + sw32_off(i, nt) + 4 * tq) = pack_bf16(q0, q1);
            const float b = hh ? beta_r1 : beta_r0;
            const float r0 = (j0 < i) ? b * acc_kk[nt][2 * hh] : 0.f;
            const float r1 = (j0 + 1 < i) ? b * acc_kk[nt][2 * hh + 1] : 0.f;
            *reinterpret_cast<float2*>(tR + 16 * i + j0) = make_float2(r0, r1);
        }
    }

    // ---- 5. K^end^T (key rows x token columns) by transposing 8 x 8 blocks.
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
    __syncwarp();

    // ---- 6. A^kk = (I + R)^{-1} by forward substitution; lane m owns column m.
    if (lane < kChunk) {
        float x[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) x[i] = 0.f;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            float acc = (i == lane) ? 1.f : 0.f;
#pragma unroll
            for (int jj = 0; jj < (i + 3) / 4; ++jj) {
                const float4 rr = *reinterpret_cast<const float4*>(tR + 16 * i + 4 * jj);
                acc -= rr.x * x[4 * jj + 0];
                acc -= rr.y * x[4 * jj + 1];
                acc -= rr.z * x[4 * jj + 2];
                acc -= rr.w * x[4 * jj + 3];
            }
            x[i] = acc;
        }
        // Column `lane` of A^kk B: scale by beta_lane.
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const __nv_bfloat16 v = __float2bfloat16_rn(x[i] * beta_f);
            *reinterpret_cast<__nv_bfloat16*>(tAKB + sw32_off(i, lane >> 3) + 2 * (lane & 7)) = v;
        }
    }

    // ---- 7. Publish the packet with one bulk copy.
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        uint8_t* dst = a.packets + (c * a.H + h) * static_cast<int64_t>(kPacketBytes);
        bulk_s2g(dst, ws, kPacketBytes);
        bulk_commit();
        bulk_wait_read_all();
    }
    __syncwarp();
}

}  // namespace

cudaError_t launch_prep(const void* q, const void* k, const float* g, const void* beta,
                        uint8_t* packets, const SeqGeometry& geo, int64_t H, float scale,
                        int* status, cudaStream_t stream) {
    (void)status;
    PrepArgs a;
    a.q = static_cast<const __nv_bfloat16*>(q);
    a.k = static_cast<const __nv_bfloat16*>(k);
    a.g = g;
    a.beta = static_cast<const __nv_bfloat16*>(beta);
    a.packets = packets;
    a.geo = geo;
    a.H = H;
    a.n_chunk_heads = geo.chunk_ub * H;
    a.scale = scale;
    if (a.n_chunk_heads <= 0) return cudaSuccess;
    const int64_t blocks = (a.n_chunk_heads + kPrepWarps - 1) / kPrepWarps;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const uint32_t smem = kPrepWarps * kPrepWarpSmem;
    static bool configured = false;   // attribute is per function; setting it twice is harmless
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    prep_kernel<<<static_cast<unsigned>(blocks), kPrepWarps * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kda
