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
// GB300 mapping (256 threads; every phase uses all eight warps):
//  * q, k, v arrive by TMA (3-D maps over [rows, H, dim], 128-byte swizzle)
//    straight into the layouts the tensor core reads; g (fp32) by an
//    unswizzled TMA tile.  Rows past the end of the sequence are zeroed on
//    chip, so padding rows are inert (g = 0, beta = 0, q = k = v = 0).
//  * The cumsum runs as two passes of segment sums (P threads per key dim).
//  * Gated products use one gate factorisation, (q exp2(g2)) . (k exp2(-g2)),
//    so Aqk and the k.k^T Gram matrix come out of ONE tcgen05 MMA with M = 128
//    (A operand = [qg ; k exp2(g2)] stacked, B = k exp2(-g2)), accumulated in
//    TMEM.  If a chunk's |g2| exceeds kSafeSpanLog2 anywhere (factors would
//    overflow), that chunk computes the gated sums exactly per element instead.
//  * T is found block-wise in fp32: the four 16x16 diagonal blocks by
//    forward substitution, then the off-diagonal blocks level by level,
//    T_IJ = -T_II sum_{J<=K<I} A_IK T_KJ, as warp-level m16n8k8 MMAs with
//    both operands split into tf32 hi + lo parts (fp32-level accuracy).
//  * w and u are two more M = 128 MMAs with A = [T' ; unused rows], reading
//    k exp2(g2) and v as MN-major B operands in place.
//  * qg, Aqk and w leave through TMA stores from swizzled shared memory;
//    kg, u and gd through 16-byte stores.
//  * The kernel is persistent (two CTAs per SM loop over the tiles): the next
//    tile's g is fetched as soon as the inverse frees the g2 region, and its
//    q, k, v as soon as the w/u MMAs have read this tile's operands, so the
//    loads overlap this tile's tail.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kS = 68;  // fp32 row stride of the 64x64 matrices in smem (bank spread)

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

__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ void mma_tf32_16x8x8(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}
// d += a * b for one m16n8k8 fragment pair at fp32-level accuracy: both operands
// are split into tf32 hi + lo parts and the three significant cross products
// are accumulated (hi*hi into d, hi*lo + lo*hi into c).
__device__ __forceinline__ void mma3_tf32(float* d, float* c, const float* a, const float* b) {
    uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        ah[i] = tf32_rna(a[i]);
        al[i] = tf32_rna(a[i] - __uint_as_float(ah[i]));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        bh[i] = tf32_rna(b[i]);
        bl[i] = tf32_rna(b[i] - __uint_as_float(bh[i]));
    }
    mma_tf32_16x8x8(d, ah, bh);
    mma_tf32_16x8x8(c, ah, bl);
    mma_tf32_16x8x8(c, al, bh);
}

template <int KB, int VB>
struct IntraSmem {
    static constexpr int K = 64 * KB, V = 64 * VB;
    static constexpr uint32_t QK = 0;                   // per kb: [q / qg 8K | k / k*exp2(g2) 8K]; later w staging
    static constexpr uint32_t TP = QK + 2 * KB * 8192;  // Aqk staging, then T' bf16 [64 i][64 j] SW128
    static constexpr uint32_t KINV = TP + 8192;         // k*exp2(-g2) per kb [64][64]; then A^T fp32 [64][kS]
    static constexpr uint32_t KINV_BYTES = 18432;       // >= max(KB*8192, 64*kS*4)
    static constexpr uint32_t VS = KINV + KINV_BYTES;   // v per vb [64][64] SW128; later u staging
    static constexpr uint32_t G = VS + VB * 8192;       // g then g2, fp32 [64][K]; later T fp32 [64][kS] + X
    static constexpr uint32_t XS = G + 64 * kS * 4;     // per-warp X halves fp32 [6][16][8]
    static constexpr uint32_t G_BYTES = (64 * K * 4 > 64 * kS * 4 + 3 * 1024) ? 64 * K * 4 : 64 * kS * 4 + 3 * 1024;
    static constexpr uint32_t GD = G + G_BYTES;         // G, fp32 [K]
    static constexpr uint32_t EG = GD + K * 4;          // exp2(G), fp32 [K]
    static constexpr uint32_t PART = EG + K * 4;        // cumsum segment sums, fp32 [4][K]
    static constexpr uint32_t BETA = PART + 4 * K * 4;  // beta, fp32 [64]
    static constexpr uint32_t BYTES = BETA + 256;
    static constexpr uint32_t QKV_TX_BYTES = (2 * KB + VB) * 8192;
    static constexpr uint32_t G_TX_BYTES = 64 * K * 4;
    static_assert(XS + 3 * 256 * 4 <= GD, "T and X must fit in the g2 region");
};

// First tile index >= t whose chunk slot holds rows (unused varlen capacity
// slots have valid == 0), or `total` if none.
__device__ __forceinline__ int64_t next_tile(const ChunkInfo* chunks, int64_t t, int64_t total, int H,
                                             int64_t stride) {
    while (t < total && chunks[t / H].valid <= 0) t += stride;
    return t;
}

template <int KB, int VB>
__global__ void __launch_bounds__(256, 2)
    kda_intra_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                     const __grid_constant__ CUtensorMap st_qg, const __grid_constant__ CUtensorMap st_w,
                     const __grid_constant__ CUtensorMap st_aqk, const uint16_t* __restrict__ beta,
                     uint8_t* __restrict__ ws, const WsLayout L, const int H, const int64_t total) {
    using S = IntraSmem<KB, VB>;
    constexpr int K = S::K, V = S::V;
    constexpr int P = 256 / K;   // threads per key dim in the cumsum
    constexpr int R = 64 / P;    // rows per cumsum segment
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_qkv, bar_g, bar_mma;
    __shared__ uint32_t tmem_slot;

    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    const ChunkInfo* chunks = reinterpret_cast<const ChunkInfo*>(ws + L.chunk_info);
    if (*reinterpret_cast<volatile int32_t*>(status) != 0) return;
    const int64_t stride = gridDim.x;
    int64_t tile = next_tile(chunks, blockIdx.x, total, H, stride);  // chunk * H + head
    if (tile >= total) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);
    float* G = reinterpret_cast<float*>(sm + S::G);
    float* Tsm = reinterpret_cast<float*>(sm + S::G);  // reuses the g2 region after the gating
    float* Xsm = reinterpret_cast<float*>(sm + S::XS);
    float* GDs = reinterpret_cast<float*>(sm + S::GD);
    float* EGs = reinterpret_cast<float*>(sm + S::EG);
    float* PARTs = reinterpret_cast<float*>(sm + S::PART);
    float* beta_s = reinterpret_cast<float*>(sm + S::BETA);
    float* AMT = reinterpret_cast<float*>(sm + S::KINV);  // A^T [m][i], valid after the Gram step

    // TMA loads of a tile's inputs: q, k, v on bar_qkv; g on bar_g.
    auto load_qkv = [&](int64_t t) {
        const int hh = static_cast<int>(t % H), r0 = chunks[t / H].row0;
        mbar_arrive_expect_tx(&bar_qkv, S::QKV_TX_BYTES);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            tma_load_3d(sm + S::QK + kb * 16384, &tm_q, &bar_qkv, kb * 64, hh, r0);
            tma_load_3d(sm + S::QK + kb * 16384 + 8192, &tm_k, &bar_qkv, kb * 64, hh, r0);
        }
#pragma unroll
        for (int vb = 0; vb < VB; ++vb) tma_load_3d(sm + S::VS + vb * 8192, &tm_v, &bar_qkv, vb * 64, hh, r0);
    };
    auto load_g = [&](int64_t t) {
        const int hh = static_cast<int>(t % H), r0 = chunks[t / H].row0;
        mbar_arrive_expect_tx(&bar_g, S::G_TX_BYTES);
        tma_load_3d(sm + S::G, &tm_g, &bar_g, 0, hh, r0);
    };

    if (tid == 0) {
        mbar_init(&bar_qkv, 1);
        mbar_init(&bar_g, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        load_g(tile);
        load_qkv(tile);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    bool timed_out = false;
    uint32_t mma_phase = 0;

#pragma unroll 1
    for (uint32_t n = 0; tile < total; ++n) {
        const int c = static_cast<int>(tile / H), h = static_cast<int>(tile % H);
        const ChunkInfo ci = chunks[c];
        const int valid = ci.valid, row0 = ci.row0;
        const int trow = static_cast<int>(tile * 64);  // first row of this tile in the workspace maps
        const int64_t tile_next = next_tile(chunks, tile + stride, total, H, stride);

        if (tid >= 128 && tid < 192) {
            const int i = tid - 128;
            float b = 0.f;
            if (i < valid) b = __uint_as_float(((uint32_t)beta[(int64_t)(row0 + i) * H + h]) << 16);
            beta_s[i] = b;
        }
        if (warp == 0 && !mbar_wait(&bar_g, n & 1, kWaitLimitNs)) timed_out = true;
        __syncthreads();

        // ---- 1. in-chunk cumsum of g (log2 space), two passes of segment sums ---
        const int cd = tid % K, cp = tid / K;  // key dim, segment
        float gv[R];  // this thread's segment of column cd, loaded once
#pragma unroll
        for (int r = 0; r < R; ++r) gv[r] = G[(cp * R + r) * K + cd];
#pragma unroll
        for (int r = 0; r < R; ++r)
            if (cp * R + r >= valid) gv[r] = 0.f;
        {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int r = 0; r < R; r += 2) {
                s0 += gv[r];
                s1 += gv[r + 1];
            }
            PARTs[cp * K + cd] = s0 + s1;
        }
        __syncthreads();
        bool unsafe = false;
        {
            float acc = 0.f;
            for (int p = 0; p < cp; ++p) acc += PARTs[p * K + cd];
            float mx = fabsf(acc * kLog2e);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                acc += gv[r];
                gv[r] = acc * kLog2e;
                mx = fmaxf(mx, fabsf(gv[r]));
            }
#pragma unroll
            for (int r = 0; r < R; ++r) G[(cp * R + r) * K + cd] = gv[r];
            if (cp == P - 1) {
                const float Gd = acc * kLog2e;
                GDs[cd] = Gd;
                EGs[cd] = ex2(Gd);
                reinterpret_cast<float*>(ws + L.gd)[tile * K + cd] = Gd;
            }
            unsafe = !(mx <= kSafeSpanLog2);
        }
        // q, k, v of this tile (loaded behind the previous tile); the previous
        // tile's w store must have read its staging (the k*exp2(-g2) region).
        if (warp == 0 && !mbar_wait(&bar_qkv, n & 1, kWaitLimitNs)) timed_out = true;
        if (tid == 0) bulk_wait_read0();
        const bool exact_path = __syncthreads_or(unsafe) != 0;

        // ---- 1b. (rare) exact gated sums for chunks with extreme decay -----------
        if (exact_path) {
            uint16_t* aqk_st = reinterpret_cast<uint16_t*>(sm + S::TP);
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
                aqk_st[sw128_offset(i, j) >> 1] = __bfloat16_as_ushort(__float2bfloat16_rn(sq));
                AMT[j * kS + i] = (j < i) ? beta_s[i] * sk : 0.f;
            }
            __syncthreads();
        }
        // ---- 2. gate the operands in place; kg to the workspace ------------------
        {
            uint16_t* kg_g = reinterpret_cast<uint16_t*>(ws + L.kg) + tile * 64 * K;
            constexpr int CPR = 8 * KB;  // 16-byte chunks per row
#pragma unroll 2
            for (int e = tid; e < 64 * CPR; e += 256) {
                const int i = e / CPR, j8 = e % CPR, kb = j8 >> 3, cc = j8 & 7;
                const uint32_t off = i * 128 + ((cc ^ (i & 7)) << 4);
                uint4* qp = reinterpret_cast<uint4*>(sm + S::QK + kb * 16384 + off);
                uint4* kp = reinterpret_cast<uint4*>(sm + S::QK + kb * 16384 + 8192 + off);
                const int d0 = kb * 64 + cc * 8;
                const float4 ga = *reinterpret_cast<const float4*>(G + i * K + d0);
                const float4 gb = *reinterpret_cast<const float4*>(G + i * K + d0 + 4);
                const float g2[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                uint4 qv = *qp, kv = *kp;
                if (i >= valid) qv = kv = make_uint4(0u, 0u, 0u, 0u);
                const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w}, kw[4] = {kv.x, kv.y, kv.z, kv.w};
                uint32_t o_qg[4], o_kga[4], o_kin[4], o_kg[4];
                if (!exact_path) {
                    const float4 ea = *reinterpret_cast<const float4*>(EGs + d0);
                    const float4 eb = *reinterpret_cast<const float4*>(EGs + d0 + 4);
                    const float eG[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float q0 = bf_lo(qw[t]), q1 = bf_hi(qw[t]);
                        const float k0 = bf_lo(kw[t]), k1 = bf_hi(kw[t]);
                        const float e0 = ex2(g2[2 * t]), e1 = ex2(g2[2 * t + 1]);
                        const float n0 = ex2(-g2[2 * t]), n1 = ex2(-g2[2 * t + 1]);
                        o_qg[t] = pack_bf16x2(q0 * e0, q1 * e1);
                        o_kga[t] = pack_bf16x2(k0 * e0, k1 * e1);
                        o_kin[t] = pack_bf16x2(k0 * n0, k1 * n1);
                        o_kg[t] = pack_bf16x2((k0 * n0) * eG[2 * t], (k1 * n1) * eG[2 * t + 1]);
                    }
                    *reinterpret_cast<uint4*>(sm + S::KINV + kb * 8192 + off) =
                        make_uint4(o_kin[0], o_kin[1], o_kin[2], o_kin[3]);
                } else {
                    const float4 Ga = *reinterpret_cast<const float4*>(GDs + d0);
                    const float4 Gb = *reinterpret_cast<const float4*>(GDs + d0 + 4);
                    const float Gv[8] = {Ga.x, Ga.y, Ga.z, Ga.w, Gb.x, Gb.y, Gb.z, Gb.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float q0 = bf_lo(qw[t]), q1 = bf_hi(qw[t]);
                        const float k0 = bf_lo(kw[t]), k1 = bf_hi(kw[t]);
                        const float e0 = ex2(g2[2 * t]), e1 = ex2(g2[2 * t + 1]);
                        o_qg[t] = pack_bf16x2(q0 * e0, q1 * e1);
                        o_kga[t] = pack_bf16x2(k0 * e0, k1 * e1);
                        o_kg[t] = pack_bf16x2(k0 * ex2(Gv[2 * t] - g2[2 * t]),
                                              k1 * ex2(Gv[2 * t + 1] - g2[2 * t + 1]));
                    }
                }
                *qp = make_uint4(o_qg[0], o_qg[1], o_qg[2], o_qg[3]);
                *kp = make_uint4(o_kga[0], o_kga[1], o_kga[2], o_kga[3]);
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
        if (tid == 0) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) tma_store_2d(&st_qg, sm + S::QK + kb * 16384, kb * 64, trow);
            bulk_commit();
        }

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
                if (!mbar_wait(&bar_mma, mma_phase, kWaitLimitNs)) timed_out = true;
            }
            mma_phase ^= 1;
            __syncthreads();
            tc_fence_after();
            {
                // warp w: TMEM lane quadrant w & 3, column half w >> 2
                const int quad = warp & 3, c0 = (warp >> 2) * 32;
                float r[32];
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + c0, r);
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + c0 + 16, r + 16);
                tmem_ld_wait();
                if (quad < 2) {
                    // rows of q.k -> Aqk staging (lower triangle with diagonal), SW128 [64][64] bf16
                    const int i = quad * 32 + lane;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t wv[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int j = c0 + cc * 8 + 2 * t;
                            wv[t] = pack_bf16x2(j <= i ? r[cc * 8 + 2 * t] : 0.f, j + 1 <= i ? r[cc * 8 + 2 * t + 1] : 0.f);
                        }
                        const int chunk = (c0 >> 3) + cc;
                        *reinterpret_cast<uint4*>(sm + S::TP + i * 128 + ((chunk ^ (i & 7)) << 4)) =
                            make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                } else {
                    // rows of k.k -> A^T (strictly lower A, beta on the row)
                    const int i = (quad - 2) * 32 + lane;
                    const float b = beta_s[i];
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int j = c0 + t;
                        AMT[j * kS + i] = (j < i) ? b * r[t] : 0.f;
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
        }
        if (tid == 0) {
            tma_store_2d(&st_aqk, sm + S::TP, 0, trow);
            bulk_commit();
        }

        // ---- 4. T = (I + A)^-1 by 16x16 blocks, fp32 ------------------------------
        // level 0: diagonal blocks by forward substitution (column per thread)
        if (tid < 64) {
            const int I = tid >> 4, cc = tid & 15, b0 = 16 * I;
            float acc[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) acc[r] = (r == cc) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < 15; ++m) {
                const float tm = acc[m];
                const float* arow = AMT + (b0 + m) * kS + b0;  // A[b0 + r][b0 + m], zero for r <= m
#pragma unroll
                for (int r4 = ((m + 1) / 4) * 4; r4 < 16; r4 += 4) {
                    const float4 a = *reinterpret_cast<const float4*>(arow + r4);
                    acc[r4 + 0] = fmaf(-a.x, tm, acc[r4 + 0]);
                    acc[r4 + 1] = fmaf(-a.y, tm, acc[r4 + 1]);
                    acc[r4 + 2] = fmaf(-a.z, tm, acc[r4 + 2]);
                    acc[r4 + 3] = fmaf(-a.w, tm, acc[r4 + 3]);
                }
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tsm[(b0 + r) * kS + b0 + cc] = acc[r];
        }
        __syncthreads();
        // levels 1..3: T_IJ = -T_II * (sum_{J<=K<I} A_IK T_KJ), J = I - lev.  One warp per
        // (block, 8-column half): 16x8 outputs by warp-level m16n8k8 MMAs in 3xTF32
        // (hi/lo split of both operands: fp32-level accuracy), X staged per warp.
        {
            const int g = lane >> 2, t = lane & 3;
            float* xw = Xsm + warp * 128;  // this warp's X half, [16][8] fp32
#pragma unroll 1
            for (int lev = 1; lev < 4; ++lev) {
                if (warp < 2 * (4 - lev)) {
                    const int J = warp >> 1, nh = warp & 1, I = J + lev;
                    const int n0 = 16 * J + 8 * nh;
                    float acc[4] = {0.f, 0.f, 0.f, 0.f}, cor[4] = {0.f, 0.f, 0.f, 0.f};
                    for (int Kb = J; Kb < I; ++Kb) {
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks) {
                            const int kc = 16 * Kb + 8 * ks;
                            const float a[4] = {AMT[(kc + t) * kS + 16 * I + g], AMT[(kc + t) * kS + 16 * I + g + 8],
                                                AMT[(kc + t + 4) * kS + 16 * I + g],
                                                AMT[(kc + t + 4) * kS + 16 * I + g + 8]};
                            const float b[2] = {Tsm[(kc + t) * kS + n0 + g], Tsm[(kc + t + 4) * kS + n0 + g]};
                            mma3_tf32(acc, cor, a, b);
                        }
                    }
                    xw[g * 8 + 2 * t] = acc[0] + cor[0];
                    xw[g * 8 + 2 * t + 1] = acc[1] + cor[1];
                    xw[(g + 8) * 8 + 2 * t] = acc[2] + cor[2];
                    xw[(g + 8) * 8 + 2 * t + 1] = acc[3] + cor[3];
                    __syncwarp();
                    float d[4] = {0.f, 0.f, 0.f, 0.f}, dc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const int kc = 16 * I + 8 * ks;
                        const float a[4] = {Tsm[(16 * I + g) * kS + kc + t], Tsm[(16 * I + g + 8) * kS + kc + t],
                                            Tsm[(16 * I + g) * kS + kc + t + 4], Tsm[(16 * I + g + 8) * kS + kc + t + 4]};
                        const float b[2] = {xw[(8 * ks + t) * 8 + g], xw[(8 * ks + t + 4) * 8 + g]};
                        mma3_tf32(d, dc, a, b);
                    }
                    *reinterpret_cast<float2*>(Tsm + (16 * I + g) * kS + n0 + 2 * t) =
                        make_float2(-(d[0] + dc[0]), -(d[1] + dc[1]));
                    *reinterpret_cast<float2*>(Tsm + (16 * I + g + 8) * kS + n0 + 2 * t) =
                        make_float2(-(d[2] + dc[2]), -(d[3] + dc[3]));
                    __syncwarp();
                }
                __syncthreads();
            }
        }
        // T' = T diag(beta) -> bf16, K-major SW128 [64 i][64 j] (the Aqk store must have read TP)
        if (tid == 0) bulk_wait_read0();
        __syncthreads();
        {
            const int i = tid >> 2, j0 = (tid & 3) * 16;
            const float* trow = Tsm + i * kS + j0;
            uint32_t wv[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 t = *reinterpret_cast<const float4*>(trow + 4 * q);
                const float4 b = *reinterpret_cast<const float4*>(beta_s + j0 + 4 * q);
                const int j = j0 + 4 * q;
                wv[2 * q] = pack_bf16x2(j <= i ? t.x * b.x : 0.f, j + 1 <= i ? t.y * b.y : 0.f);
                wv[2 * q + 1] = pack_bf16x2(j + 2 <= i ? t.z * b.z : 0.f, j + 3 <= i ? t.w * b.w : 0.f);
            }
            const int ch = j0 >> 3;
            *reinterpret_cast<uint4*>(sm + S::TP + i * 128 + ((ch ^ (i & 7)) << 4)) =
                make_uint4(wv[0], wv[1], wv[2], wv[3]);
            *reinterpret_cast<uint4*>(sm + S::TP + i * 128 + (((ch + 1) ^ (i & 7)) << 4)) =
                make_uint4(wv[4], wv[5], wv[6], wv[7]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // the g2 region (T, X) is free now: fetch the next tile's g behind this one
        if (tid == 0 && tile_next < total) load_g(tile_next);

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
            if (!mbar_wait(&bar_mma, mma_phase, kWaitLimitNs)) timed_out = true;
        }
        if (tid == 0) bulk_wait_read0();  // the qg store has read QK
        mma_phase ^= 1;
        __syncthreads();
        tc_fence_after();
        // the MMAs have read QK and VS, and the qg store has read QK: fetch the
        // next tile's q, k, v behind this one
        if (tid == 0 && tile_next < total) load_qkv(tile_next);


        // ---- 6. w rows (warps 0,1) -> swizzled staging -> TMA store; u rows (warps 4,5) -> global
        if (warp < 2) {
            const int i = warp * 32 + lane;
            uint8_t* stg = sm + S::KINV;  // A^T and the unused MMA rows are dead now
#pragma unroll
            for (int blk = 0; blk < KB; ++blk) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float r[32];
                    const uint32_t col = blk * 64 + half * 32;
                    tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + col, r);
                    tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + col + 16, r + 16);
                    tmem_ld_wait();
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const int chunk = half * 4 + cc;
                        *reinterpret_cast<uint4*>(stg + blk * 8192 + i * 128 + ((chunk ^ (i & 7)) << 4)) =
                            make_uint4(pack_bf16x2(r[cc * 8 + 0], r[cc * 8 + 1]),
                                       pack_bf16x2(r[cc * 8 + 2], r[cc * 8 + 3]),
                                       pack_bf16x2(r[cc * 8 + 4], r[cc * 8 + 5]),
                                       pack_bf16x2(r[cc * 8 + 6], r[cc * 8 + 7]));
                    }
                }
            }
            fence_proxy_async_smem();
        } else if (warp == 4 || warp == 5) {
            const int quad = warp & 3, i = quad * 32 + lane;
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(ws + L.u) + (tile * 64 + i) * V);
#pragma unroll
            for (int c0 = 0; c0 < V; c0 += 32) {
                float r[32];
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + K + c0, r);
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + K + c0 + 16, r + 16);
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc)
                    dst[c0 / 8 + cc] = make_uint4(pack_bf16x2(r[cc * 8 + 0], r[cc * 8 + 1]),
                                                  pack_bf16x2(r[cc * 8 + 2], r[cc * 8 + 3]),
                                                  pack_bf16x2(r[cc * 8 + 4], r[cc * 8 + 5]),
                                                  pack_bf16x2(r[cc * 8 + 6], r[cc * 8 + 7]));
            }
        }
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) tma_store_2d(&st_w, sm + S::KINV + kb * 8192, kb * 64, trow);
            bulk_commit();
        }
        tile = tile_next;
    }

    if (tid == 0) bulk_wait_read0();  // smem must outlive the stores' reads; the writes complete with the grid
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
    const int64_t total = a.max_chunks * a.H;
    if (total <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 148;
    const int64_t ctas = total < 2 * (int64_t)sms ? total : 2 * (int64_t)sms;  // persistent: 2 per SM
    kern<<<(unsigned)ctas, 256, smem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_g, a.st_qg, a.st_w, a.st_aqk,
                                                a.beta, a.ws, a.L, a.H, total);
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
