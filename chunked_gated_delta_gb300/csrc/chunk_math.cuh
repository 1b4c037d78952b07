// chunk_math.cuh -- device arithmetic shared by the kernels: exponent and
// bf16 / fp16 helpers, the tf32 warp MMA, the fp32 64x64 matrix layout, and
// the intra-chunk stage's steps that the two-stage intra kernel (intra.cu) and
// the single-pass kernel (fused.cu) both run on a 256-thread CTA:
//
//   exact_sums_block   the gated sums of a chunk whose decay span is too large
//                      for the factored Gram MMA, per element
//   unit_lower_inverse T = (I + A)^-1 of the chunk's strictly lower A, in 16x16
//                      blocks: the diagonal blocks by forward substitution, the
//                      others level by level, T_IJ = -T_II sum_{J<=K<I} A_IK T_KJ
//   store_t_prime      T' = T diag(beta) rounded to bf16 as the w / u MMA operand
//
// (the chunked form of kernel-fun "kda/_kernels/fwd_state.py", module
// docstring; T is the INV operand of "KDA源码剖析之FlashKDA（下）").
// Everything here is internal to each translation unit that includes it.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace kda {
namespace {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint16_t bf16_bits(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }

// Inputs q, k, v, beta are bf16 or (F16) fp16.
template <bool F16>
__device__ __forceinline__ float in_lo(uint32_t w) {
    if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
    else return bf_lo(w);
}
template <bool F16>
__device__ __forceinline__ float in_hi(uint32_t w) {
    if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    else return bf_hi(w);
}
template <bool F16>
__device__ __forceinline__ float in_at(const uint8_t* p) {
    return in_lo<F16>((uint32_t)(*(const uint16_t*)p));
}

__device__ __forceinline__ uint32_t tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// d += a * b for one m16n8k8 fragment pair with tf32 operands (round to nearest)
// and fp32 accumulation.  A hi/lo operand split (3xTF32, fp32-level products)
// was measured to change no parity figure in the fourth digit: T' is rounded
// to bf16 right after, so single tf32 products suffice.
__device__ __forceinline__ void mma_tf32(float* d, const float* a, const float* b) {
    const uint32_t ah[4] = {tf32_rna(a[0]), tf32_rna(a[1]), tf32_rna(a[2]), tf32_rna(a[3])};
    const uint32_t bh[2] = {tf32_rna(b[0]), tf32_rna(b[1])};
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(ah[0]), "r"(ah[1]), "r"(ah[2]), "r"(ah[3]), "r"(bh[0]), "r"(bh[1]));
}

// fp32 64x64 matrix in shared memory, row-major with 64 floats per row and an
// XOR of the column's 8-float group by (row & 3): row-contiguous accesses,
// float4 row reads and the 4-row x 8-column fragment reads of the MMAs are
// all free of bank conflicts.  It holds A^T in its strict upper triangle and
// T in its strict lower triangle (T's diagonal 16x16 blocks whole, once A's
// have been consumed).
struct Mat64 {
    float* p;
    __device__ __forceinline__ float* at(int r, int c) const { return p + r * 64 + (c ^ ((r & 3) << 3)); }
};

constexpr int kChunkThreads = 256;  // threads of the CTAs that run the intra-chunk steps

// Exact gated sums of a chunk whose decay span is too large for the factored
// MMA (kept out of line so its registers do not weigh on the common path),
// accumulated over one 64-dim block of key dims: qs the block's raw q tile and
// the k tile 8 KB after it (SW128), g2h its g2 as fp32 [64][64].  For this
// thread's (i, j) pairs, ea += q_i . k_j gated (j <= i) and eb += k_i . k_j
// gated.
template <bool F16>
__device__ __noinline__ void exact_sums_block(const uint8_t* qs, const float* g2h, int valid, float* ea, float* eb) {
    const uint8_t* ks = qs + 8192;
    constexpr int kPairs = 64 * 64 / kChunkThreads;
    for (int n = 0; n < kPairs; ++n) {
        const int e = threadIdx.x + kChunkThreads * n, i = e >> 6, j = e & 63;
        if (j <= i && i < valid) {
            float a = ea[n], b = eb[n];
            for (int d = 0; d < 64; ++d) {
                const float qi = in_at<F16>(qs + ptx::sw128_offset(i, d));
                const float ki = in_at<F16>(ks + ptx::sw128_offset(i, d));
                const float kj = in_at<F16>(ks + ptx::sw128_offset(j, d));
                const float gate = ex2(g2h[i * 64 + d] - g2h[j * 64 + d]);
                a = fmaf(qi * kj, gate, a);
                b = fmaf(ki * kj, gate, b);
            }
            ea[n] = a;
            eb[n] = b;
        }
    }
}

// T = (I + A)^-1 in PM, from A^T in PM's strict upper triangle, by 16x16
// blocks in fp32; called by every thread of the CTA (block barriers inside;
// Xsm holds 8 warps x 128 floats).  Level 0: the diagonal blocks by forward
// substitution, one column per thread of the first 64; levels 1..3: T_IJ =
// -T_II (sum_{J<=K<I} A_IK T_KJ), J = I - lev, one warp per (block, 8-column
// half), 16x8 outputs by warp-level m16n8k8 tf32 MMAs.
__device__ __forceinline__ void unit_lower_inverse(const Mat64 PM, float* Xsm, int tid, int warp, int lane) {
    if (tid < 64) {
        const int I = tid >> 4, cc = tid & 15, b0 = 16 * I;
        float acc[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) acc[rr] = (rr == cc) ? 1.f : 0.f;
#pragma unroll
        for (int m = 0; m < 15; ++m) {
            const float tm = acc[m];
#pragma unroll
            for (int r4 = ((m + 1) / 4) * 4; r4 < 16; r4 += 4) {
                // A[b0 + r][b0 + m] for r = r4..r4+3: one float4 of A^T row b0 + m;
                // only r > m is A (the rest is T's storage)
                const float4 a = *reinterpret_cast<const float4*>(PM.at(b0 + m, b0 + r4));
                if (r4 + 0 > m) acc[r4 + 0] = fmaf(-a.x, tm, acc[r4 + 0]);
                if (r4 + 1 > m) acc[r4 + 1] = fmaf(-a.y, tm, acc[r4 + 1]);
                if (r4 + 2 > m) acc[r4 + 2] = fmaf(-a.z, tm, acc[r4 + 2]);
                acc[r4 + 3] = fmaf(-a.w, tm, acc[r4 + 3]);
            }
        }
        // acc is column cc of T_II whole (1 on the diagonal, 0 above it); it
        // replaces A's diagonal block once every column's substitution is done
        asm volatile("bar.sync 1, 64;" ::: "memory");
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) *PM.at(b0 + rr, b0 + cc) = acc[rr];
    }
    __syncthreads();
    const int gq = lane >> 2, t = lane & 3;
    float* xw = Xsm + warp * 128;  // this warp's X half, [16][8] fp32
#pragma unroll 1
    for (int lev = 1; lev < 4; ++lev) {
        for (int item = warp; item < 2 * (4 - lev); item += kChunkThreads / 32) {
            const int J = item >> 1, nh = item & 1, I = J + lev;
            const int n0 = 16 * J + 8 * nh;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int Kb = J; Kb < I; ++Kb) {
#pragma unroll
                for (int ks = 0; ks < 2; ++ks) {
                    const int kc = 16 * Kb + 8 * ks;
                    const float a[4] = {*PM.at(kc + t, 16 * I + gq), *PM.at(kc + t, 16 * I + gq + 8),
                                        *PM.at(kc + t + 4, 16 * I + gq), *PM.at(kc + t + 4, 16 * I + gq + 8)};
                    const float b[2] = {*PM.at(kc + t, n0 + gq), *PM.at(kc + t + 4, n0 + gq)};
                    mma_tf32(acc, a, b);
                }
            }
            xw[gq * 8 + 2 * t] = acc[0];
            xw[gq * 8 + 2 * t + 1] = acc[1];
            xw[(gq + 8) * 8 + 2 * t] = acc[2];
            xw[(gq + 8) * 8 + 2 * t + 1] = acc[3];
            __syncwarp();
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                const int kc = 16 * I + 8 * ks;
                const float a[4] = {*PM.at(16 * I + gq, kc + t), *PM.at(16 * I + gq + 8, kc + t),
                                    *PM.at(16 * I + gq, kc + t + 4), *PM.at(16 * I + gq + 8, kc + t + 4)};
                const float b[2] = {xw[(8 * ks + t) * 8 + gq], xw[(8 * ks + t + 4) * 8 + gq]};
                mma_tf32(d, a, b);
            }
            *reinterpret_cast<float2*>(PM.at(16 * I + gq, n0 + 2 * t)) = make_float2(-d[0], -d[1]);
            *reinterpret_cast<float2*>(PM.at(16 * I + gq + 8, n0 + 2 * t)) = make_float2(-d[2], -d[3]);
            __syncwarp();
        }
        __syncthreads();
    }
}

// T' = T diag(beta) -> bf16, K-major SW128 [64 i][64 j] at dst (which may
// overlay PM: it is written once every thread has read its part of T);
// called by every thread of the CTA.
__device__ __forceinline__ void store_t_prime(const Mat64 PM, const float* beta_s, uint8_t* dst, int tid) {
    const int i = tid >> 2, j0 = (tid & 3) * 16;
    uint4 x[2];
#pragma unroll
    for (int q8 = 0; q8 < 2; ++q8) {
        const int j = j0 + 8 * q8;
        const float4 ta = *reinterpret_cast<const float4*>(PM.at(i, j));
        const float4 tb = *reinterpret_cast<const float4*>(PM.at(i, j + 4));
        const float4 ba = *reinterpret_cast<const float4*>(beta_s + j);
        const float4 bb = *reinterpret_cast<const float4*>(beta_s + j + 4);
        const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
        const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = j + e <= i ? tv[e] * bv[e] : 0.f;
        x[q8] = make_uint4(ptx::pack_bf16x2(y[0], y[1]), ptx::pack_bf16x2(y[2], y[3]), ptx::pack_bf16x2(y[4], y[5]),
                           ptx::pack_bf16x2(y[6], y[7]));
    }
    __syncthreads();
#pragma unroll
    for (int q8 = 0; q8 < 2; ++q8) {
        const int j = j0 + 8 * q8;
        *reinterpret_cast<uint4*>(dst + i * 128 + (((j >> 3) ^ (i & 7)) << 4)) = x[q8];
    }
}

}  // namespace
}  // namespace kda
