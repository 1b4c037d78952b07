// intra.cu -- the intra-chunk stage of the chunked KDA forward (sm_103a).
//
// One CTA per (chunk of 64 tokens, head).  For the chunk's rows i, j and key
// dims d (kernel-fun "kda/_kernels/fwd_state.py", module docstring, for qg,
// kg, Aqk and the log2 gate; w and u solve the chunk's delta-rule system, the
// INV operand of "KDA源码剖析之FlashKDA（下）"):
//
//   g2[i,d]  = log2(e) * sum_{m<=i} g[m,d]          in-chunk cumsum, log2 space
//   G[d]     = g2[last valid row, d]                 -> gd (per-chunk decay)
//   qg       = q * exp2(g2)                          -> workspace
//   kg       = k * exp2(G - g2)                      -> workspace
//   Aqk[i,j] = sum_d q_id k_jd exp2(g2_id - g2_jd), j <= i, else 0
//              (stored WITHOUT scale; the scan kernel applies scale once to
//               qg@h + Aqk@v')                       -> workspace
//   A[i,j]   = beta_i sum_d k_id k_jd exp2(g2_id - g2_jd), j < i, else 0
//   T        = (I + A)^-1,   T' = T diag(beta)
//   w        = T' (k * exp2(g2)),   u = T' v         -> workspace
//
// GB300 mapping:
//  * q, k, v arrive by TMA (3-D maps over [rows, H, dim], 128-byte swizzle)
//    straight into the layouts the tensor core reads; g (fp32) by an
//    unswizzled TMA tile.  Rows past the end of the sequence are zeroed
//    on chip, so padding rows are inert (g = 0, beta = 0, q = k = v = 0).
//  * Gated products use one gate factorisation, (q exp2(g2)) . (k exp2(-g2)),
//    so Aqk and the k.k^T Gram matrix come out of ONE tcgen05 MMA with M = 128
//    (A operand = [qg ; k exp2(g2)] stacked, B = k exp2(-g2)), accumulated in
//    TMEM.  If a chunk's log2 decay span exceeds kSafeSpanLog2 (factors would
//    overflow), that chunk computes the gated sums exactly per element instead.
//  * T is found by a right-looking forward substitution in fp32, one column
//    per thread.  w and u are two more M = 128 MMAs with A = [T' ; unused
//    rows], reading k exp2(g2) and v as MN-major B operands in place.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kAmStride = 68;  // fp32 row stride of the A^T matrix in smem (bank spread)

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_at(const uint8_t* p) {
    return __uint_as_float(((uint32_t)(*(const uint16_t*)p)) << 16);
}

template <int KB, int VB>
struct IntraSmem {
    static constexpr int K = 64 * KB, V = 64 * VB;
    static constexpr uint32_t QK = 0;                   // per kb: [q / qg 8K | k / k*exp2(g2) 8K]
    static constexpr uint32_t TP = QK + 2 * KB * 8192;  // T' bf16 [64 i][64 j], SW128 K-major
    static constexpr uint32_t KINV = TP + 8192;         // k*exp2(-g2) per kb [64][64]; then A^T fp32
    static constexpr uint32_t KINV_BYTES = 18432;       // >= max(KB*8192, 64*68*4)
    static constexpr uint32_t VS = KINV + KINV_BYTES;   // v per vb [64][64], SW128
    static constexpr uint32_t G = VS + VB * 8192;       // g then g2, fp32 [64][K]
    static constexpr uint32_t GD = G + 64 * K * 4;      // G, fp32 [K]
    static constexpr uint32_t BETA = GD + K * 4;        // beta, fp32 [64]
    static constexpr uint32_t BYTES = BETA + 256;
    static constexpr uint32_t TX_BYTES = (2 * KB + VB) * 8192 + 64 * K * 4;
};

template <int KB, int VB>
__global__ void __launch_bounds__(256, 2)
    kda_intra_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                     const uint16_t* __restrict__ beta, uint8_t* __restrict__ ws, const WsLayout L,
                     const int H) {
    using S = IntraSmem<KB, VB>;
    constexpr int K = S::K, V = S::V;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_load, bar_mma;
    __shared__ uint32_t tmem_slot;

    const int64_t tile = blockIdx.x;  // chunk * H + head
    const int c = static_cast<int>(tile / H), h = static_cast<int>(tile % H);
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    const ChunkInfo ci = reinterpret_cast<const ChunkInfo*>(ws + L.chunk_info)[c];
    if (ci.valid <= 0 || *reinterpret_cast<volatile int32_t*>(status) != 0) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int valid = ci.valid, row0 = ci.row0;
    const uint32_t sbase = smem_u32(sm);
    float* G = reinterpret_cast<float*>(sm + S::G);
    float* GDs = reinterpret_cast<float*>(sm + S::GD);
    float* beta_s = reinterpret_cast<float*>(sm + S::BETA);
    float* AMT = reinterpret_cast<float*>(sm + S::KINV);  // A^T [m][i], valid after the Gram step

    if (tid == 0) {
        mbar_init(&bar_load, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar_load, S::TX_BYTES);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            tma_load_3d(sm + S::QK + kb * 16384, &tm_q, &bar_load, kb * 64, h, row0);
            tma_load_3d(sm + S::QK + kb * 16384 + 8192, &tm_k, &bar_load, kb * 64, h, row0);
        }
#pragma unroll
        for (int vb = 0; vb < VB; ++vb) tma_load_3d(sm + S::VS + vb * 8192, &tm_v, &bar_load, vb * 64, h, row0);
        tma_load_3d(sm + S::G, &tm_g, &bar_load, 0, h, row0);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, 256);
        tmem_relinquish();
    }
    if (tid >= 128 && tid < 192) {
        const int i = tid - 128;
        float b = 0.f;
        if (i < valid) b = __uint_as_float(((uint32_t)beta[(int64_t)(row0 + i) * H + h]) << 16);
        beta_s[i] = b;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    bool timed_out = false;
    if (!mbar_wait(&bar_load, 0, kWaitLimitNs)) timed_out = true;

    // ---- 1. in-chunk cumsum of g, log2 space; G; overflow guard --------------
    bool unsafe = false;
    if (tid < K) {
        float acc = 0.f, mx = 0.f;
#pragma unroll 8
        for (int i = 0; i < 64; ++i) {
            const float gi = (i < valid) ? G[i * K + tid] : 0.f;
            acc += gi;
            const float g2 = acc * kLog2e;
            G[i * K + tid] = g2;
            mx = fmaxf(mx, fabsf(g2));
        }
        const float Gd = acc * kLog2e;
        GDs[tid] = Gd;
        reinterpret_cast<float*>(ws + L.gd)[tile * K + tid] = Gd;
        unsafe = !(mx <= kSafeSpanLog2);
    }
    const bool exact_path = __syncthreads_or(unsafe) != 0;

    uint16_t* aqk_g = reinterpret_cast<uint16_t*>(ws + L.aqk) + tile * 64 * 64;

    // ---- 1b. (rare) exact gated sums for chunks with extreme decay -----------
    if (exact_path) {
        for (int e = tid; e < 64 * 64; e += 256) {
            const int i = e >> 6, j = e & 63;
            float sq = 0.f, sk = 0.f;
            if (j <= i && i < valid) {
                for (int d = 0; d < K; ++d) {
                    const uint8_t* base = sm + S::QK + (d >> 6) * 16384;
                    const float qi = bf16_at(base + sw128_offset(i, d & 63));
                    const float ki = bf16_at(base + 8192 + sw128_offset(i, d & 63));
                    const float kj = bf16_at(base + 8192 + sw128_offset(j, d & 63));
                    const float gate = ex2(G[i * K + d] - G[j * K + d]);
                    sq = fmaf(qi * kj, gate, sq);
                    sk = fmaf(ki * kj, gate, sk);
                }
            }
            aqk_g[i * 64 + j] = __bfloat16_as_ushort(__float2bfloat16_rn(sq));
            AMT[j * kAmStride + i] = (j < i) ? beta_s[i] * sk : 0.f;
        }
        __syncthreads();
    }

    // ---- 2. gate the operands in place; qg and kg to the workspace -----------
    {
        uint16_t* qg_g = reinterpret_cast<uint16_t*>(ws + L.qg) + tile * 64 * K;
        uint16_t* kg_g = reinterpret_cast<uint16_t*>(ws + L.kg) + tile * 64 * K;
        constexpr int CPR = 8 * KB;  // 16-byte chunks per row
        for (int e = tid; e < 64 * CPR; e += 256) {
            const int i = e / CPR, j8 = e % CPR, kb = j8 >> 3, cc = j8 & 7;
            const uint32_t off = i * 128 + ((cc ^ (i & 7)) << 4);
            uint4* qp = reinterpret_cast<uint4*>(sm + S::QK + kb * 16384 + off);
            uint4* kp = reinterpret_cast<uint4*>(sm + S::QK + kb * 16384 + 8192 + off);
            const int d0 = kb * 64 + cc * 8;
            const float4 ga = *reinterpret_cast<const float4*>(G + i * K + d0);
            const float4 gb = *reinterpret_cast<const float4*>(G + i * K + d0 + 4);
            const float4 Ga = *reinterpret_cast<const float4*>(GDs + d0);
            const float4 Gb = *reinterpret_cast<const float4*>(GDs + d0 + 4);
            const float g2[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
            const float Gv[8] = {Ga.x, Ga.y, Ga.z, Ga.w, Gb.x, Gb.y, Gb.z, Gb.w};
            uint4 qv = *qp, kv = *kp;
            if (i >= valid) qv = kv = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
            uint32_t o_qg[4], o_kga[4], o_kin[4], o_kg[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float q0 = bf_lo(qw[t]), q1 = bf_hi(qw[t]);
                const float k0 = bf_lo(kw[t]), k1 = bf_hi(kw[t]);
                const float a0 = g2[2 * t], a1 = g2[2 * t + 1];
                const float e0 = ex2(a0), e1 = ex2(a1);
                o_qg[t] = pack_bf16x2(q0 * e0, q1 * e1);
                o_kga[t] = pack_bf16x2(k0 * e0, k1 * e1);
                o_kin[t] = pack_bf16x2(k0 * ex2(-a0), k1 * ex2(-a1));
                o_kg[t] = pack_bf16x2(k0 * ex2(Gv[2 * t] - a0), k1 * ex2(Gv[2 * t + 1] - a1));
            }
            const uint4 vqg = make_uint4(o_qg[0], o_qg[1], o_qg[2], o_qg[3]);
            *qp = vqg;
            *kp = make_uint4(o_kga[0], o_kga[1], o_kga[2], o_kga[3]);
            if (!exact_path)
                *reinterpret_cast<uint4*>(sm + S::KINV + kb * 8192 + off) =
                    make_uint4(o_kin[0], o_kin[1], o_kin[2], o_kin[3]);
            *reinterpret_cast<uint4*>(qg_g + i * K + d0) = vqg;
            *reinterpret_cast<uint4*>(kg_g + i * K + d0) = make_uint4(o_kg[0], o_kg[1], o_kg[2], o_kg[3]);
        }
        for (int e = tid; e < (64 - valid) * 8 * VB; e += 256) {
            const int r = valid + e / (8 * VB), x = e % (8 * VB);
            *reinterpret_cast<uint4*>(sm + S::VS + (x >> 3) * 8192 + r * 128 + (x & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    uint32_t mma_phase = 0;
    // ---- 3. Gram MMA: [qg ; k exp2(g2)] @ (k exp2(-g2))^T -> TMEM ------------
    if (!exact_path) {
        if (warp == 1) {
            if (lane == 0) {
                tc_fence_after();
                constexpr uint32_t id = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const int kb = ks >> 2, kk = ks & 3;
                    const uint64_t ad = smem_desc(sbase + S::QK + kb * 16384 + kk * 32, 16, 1024);
                    const uint64_t bd = smem_desc(sbase + S::KINV + kb * 8192 + kk * 32, 16, 1024);
                    mma_bf16(tmem, ad, bd, id, ks > 0 ? 1u : 0u);
                }
                mma_commit(&bar_mma);
            }
            __syncwarp();
        }
        if (!mbar_wait(&bar_mma, mma_phase, kWaitLimitNs)) timed_out = true;
        mma_phase ^= 1;
        tc_fence_after();
        if (warp < 2) {
            // lanes 0..63: rows of q.k -> Aqk (lower triangle with diagonal)
            const int i = warp * 32 + lane;
            uint16_t* dst = aqk_g + i * 64;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
                float r[16];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, r);
                tmem_ld_wait();
                uint32_t wv[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const float lo = (c0 + 2 * t <= i) ? r[2 * t] : 0.f;
                    const float hi = (c0 + 2 * t + 1 <= i) ? r[2 * t + 1] : 0.f;
                    wv[t] = pack_bf16x2(lo, hi);
                }
                reinterpret_cast<uint4*>(dst + c0)[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                reinterpret_cast<uint4*>(dst + c0)[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
            }
        } else if (warp < 4) {
            // lanes 64..127: rows of k.k -> A^T (strictly lower A, beta on the row)
            const int i = (warp - 2) * 32 + lane;
            const float b = beta_s[i];
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
                float r[16];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, r);
                tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const int j = c0 + t;
                    AMT[j * kAmStride + i] = (j < i) ? b * r[t] : 0.f;
                }
            }
        }
        tc_fence_before();
        __syncthreads();
    }

    // ---- 4. T = (I + A)^-1, right-looking, one column per thread; T' = T diag(beta)
    if (tid < 64) {
        const int j = tid;
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < 63; ++m) {
            const float tm = acc[m];
            const float* arow = AMT + m * kAmStride;  // A[i][m] for all i (zero for i <= m)
#pragma unroll
            for (int i4 = ((m + 1) / 4) * 4; i4 < 64; i4 += 4) {
                const float4 a = *reinterpret_cast<const float4*>(arow + i4);
                acc[i4 + 0] = fmaf(-a.x, tm, acc[i4 + 0]);
                acc[i4 + 1] = fmaf(-a.y, tm, acc[i4 + 1]);
                acc[i4 + 2] = fmaf(-a.z, tm, acc[i4 + 2]);
                acc[i4 + 3] = fmaf(-a.w, tm, acc[i4 + 3]);
            }
        }
        const float bj = beta_s[j];
        uint8_t* TP = sm + S::TP;
#pragma unroll
        for (int i = 0; i < 64; ++i)
            *reinterpret_cast<uint16_t*>(TP + sw128_offset(i, j)) =
                __bfloat16_as_ushort(__float2bfloat16_rn(acc[i] * bj));
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 5. w = T' (k exp2(g2)), u = T' v  (M = 128: rows 64..127 unused) -----
    if (warp == 1) {
        if (lane == 0) {
            tc_fence_after();
            constexpr uint32_t idw = idesc_bf16_f32(128, K, 0, 1);
            constexpr uint32_t idu = idesc_bf16_f32(128, V, 0, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t ad = smem_desc(sbase + S::TP + ks * 32, 16, 1024);
                mma_bf16(tmem, ad, smem_desc(sbase + S::QK + 8192 + ks * 2048, 16384, 1024), idw,
                         ks > 0 ? 1u : 0u);
                mma_bf16(tmem + K, ad, smem_desc(sbase + S::VS + ks * 2048, 8192, 1024), idu,
                         ks > 0 ? 1u : 0u);
            }
            mma_commit(&bar_mma);
        }
        __syncwarp();
    }
    if (!mbar_wait(&bar_mma, mma_phase, kWaitLimitNs)) timed_out = true;
    tc_fence_after();

    // ---- 6. w (warps 0,1) and u (warps 4,5) rows to the workspace -------------
    if (warp < 2 || warp == 4 || warp == 5) {
        const int quad = warp & 3, i = quad * 32 + lane;
        const bool is_w = warp < 2;
        const int ncol = is_w ? K : V;
        const uint32_t col0 = is_w ? 0u : (uint32_t)K;
        uint16_t* dst = is_w ? reinterpret_cast<uint16_t*>(ws + L.w) + (tile * 64 + i) * K
                             : reinterpret_cast<uint16_t*>(ws + L.u) + (tile * 64 + i) * V;
        for (int c0 = 0; c0 < ncol; c0 += 16) {
            float r[16];
            tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + col0 + c0, r);
            tmem_ld_wait();
            uint32_t wv[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) wv[t] = pack_bf16x2(r[2 * t], r[2 * t + 1]);
            reinterpret_cast<uint4*>(dst + c0)[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            reinterpret_cast<uint4*>(dst + c0)[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
    if (timed_out) atomicOr(status, kStatusTimeout);
}

template <int KB, int VB>
cudaError_t launch_intra_t(const IntraArgs& a, cudaStream_t stream) {
    using S = IntraSmem<KB, VB>;
    const uint32_t smem = S::BYTES + 1024;
    auto kern = kda_intra_kernel<KB, VB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t ctas = a.max_chunks * a.H;
    if (ctas <= 0) return cudaSuccess;
    kern<<<(unsigned)ctas, 256, smem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_g, a.beta, a.ws, a.L, a.H);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_intra(const IntraArgs& a, cudaStream_t stream) {
    const int KB = a.K / 64, VB = a.V / 64;
    if (KB == 2 && VB == 2) return launch_intra_t<2, 2>(a, stream);
    if (KB == 2 && VB == 1) return launch_intra_t<2, 1>(a, stream);
    if (KB == 1 && VB == 2) return launch_intra_t<1, 2>(a, stream);
    if (KB == 1 && VB == 1) return launch_intra_t<1, 1>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace kda
