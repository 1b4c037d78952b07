// fused.cu -- the single-pass forward (sm_103a): the intra-chunk stage and the
// state scan of one (sequence, head) in one CTA, chunk after chunk, with no
// intermediate leaving the chip.
//
// Per chunk c of the sequence (the same arithmetic as intra.cu followed by one
// step of scan.cu; kernel-fun "kda/_kernels/fwd_state.py", module docstring):
//
//   g2 = log2(e) cumsum(g), G = g2[last valid row]
//   qg = q exp2(g2),  kg = k exp2(G - g2),  Aqk[i,j] = q_i . k_j gated (j <= i)
//   A[i,j] = beta_i k_i . k_j gated (j < i),  T' = (I + A)^-1 diag(beta)
//   w = T' (k exp2(g2)),  u = T' v
//   v' = u - w h;  o = scale (qg h + Aqk v');  h <- exp2(G) h + kg^T v'
//
// Only q, k, v, g, beta and h0 are read and only o and ht written: the 1538
// bytes per token-head of the method's own inputs and outputs, against 3858
// for the two-stage path.  The price is that a sequence's chunks now run one
// after another on one SM: the intra work of a chunk (about 17 k cycles for
// one tile alone on an SM, against about 7 k cycles of SM time per tile when
// four tiles share an SM in the two-stage kernel) is no longer spread over the
// GPU, so this path is for problems too small to fill the GPU or to amortise
// three launches, and as the measured counterpart of the two-stage path.
//
// GB300 mapping: one CTA of 256 threads per (sequence, head) with all V
// columns, one CTA per SM (about 188 KB of shared memory at K = V = 128).
//  * Shared memory per 64-dim key block: [w | qg | k exp2(g2)], 8 KB each, so
//    that the scan's [w ; qg] and the Gram MMA's [qg ; k exp2(g2)] are both
//    contiguous 128-row operands; then kg, Aqk (the 8 KB before it is kg's last
//    block, the unused upper half of the [unused ; Aqk] operand), u (v until
//    the u MMA has read it), the 16 KB matrix region (segment sums, then
//    k exp2(-g2), then A^T + T in fp32, then T' in bf16), the bf16 copy of h
//    (MN-major), v', the [I ; 0] operand, and small buffers.
//  * TMEM: 128 columns for the intra MMAs (the Gram product, then w^T and
//    u^T), then the scan's accumulator (V columns) and DH (V columns).
//  * The state h: thread r of warp w (quadrant w & 3, V block w >> 2) owns row
//    r of V block (w >> 2) in 64 fp32 registers, as in the scan kernel.
//  * Phases are separated by block barriers; MMAs are issued by thread 0 and
//    completed through mbarriers whose waits are bounded (kWaitLimitNs): a
//    wait that runs out sets the status word and ends the CTA's walk.
//  * The next chunk's q, k, v and g are prefetched into L2 at the start of
//    each chunk.
#include <cuda_bf16.h>

#include "chunk_math.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = kChunkThreads;

template <int KB, int VB>
struct FusedSmem {
    static constexpr int K = 64 * KB, V = 64 * VB;
    static constexpr int NCG = K / 4;            // 4-column groups of g
    static constexpr int NSEG = kThreads / NCG;  // row segments
    static constexpr int RS = 64 / NSEG;         // rows per segment
    static constexpr uint32_t KBLK = 24576;      // per key block: [w 8K | qg 8K | k exp2(g2) 8K]
    __host__ __device__ static constexpr uint32_t W(int kb) { return kb * KBLK; }
    __host__ __device__ static constexpr uint32_t QG(int kb) { return kb * KBLK + 8192; }
    __host__ __device__ static constexpr uint32_t KX(int kb) { return kb * KBLK + 16384; }
    static constexpr uint32_t KG = KB * KBLK;            // kg per key block [64 tok][64 d]
    static constexpr uint32_t AQK = KG + KB * 8192;      // Aqk [64 i][64 j] (unscaled, zero above the diagonal)
    static constexpr uint32_t U = AQK + 8192;            // per V block [64 tok][64 v]: v, then u
    static constexpr uint32_t M = U + VB * 8192;         // 16 KB matrix region
    static constexpr uint32_t HS = M + 16384;            // per V block: h bf16 [K rows][64 v], MN-major
    static constexpr uint32_t HS_BLOCK = KB * 8192;
    static constexpr uint32_t VP = HS + VB * HS_BLOCK;   // per V block: v' bf16 [64 tok][64 v]
    static constexpr uint32_t IDN = VP + VB * 8192;      // [I_64 ; 0] bf16, K-major [128 rows][64 tok]
    static constexpr uint32_t XS = IDN + 16384;          // fp32 [8 warps][16][8]
    static constexpr uint32_t BETA = XS + 8 * 512;       // beta fp32 [64]
    static constexpr uint32_t GDS = BETA + 256;          // G fp32 [K]
    static constexpr uint32_t BYTES = GDS + K * 4;
    static constexpr uint32_t QKV_TX = (2 * KB + VB) * 8192;
    static constexpr uint32_t TMEM_COLS = VB == 2 ? 512 : 256;  // intra 128 + ACC V + DH V
    static_assert(NSEG * K * 4 == 4096, "segment sums are 4 KB");
    static_assert(KX(0) - QG(0) == 8192, "exact_sums_block reads k 8 KB after q");
};

struct FusedBars {
    uint64_t qkv, mma, wh, dh, acc;
    uint32_t tmem_slot;
};

// One CTA per (sequence, head).
template <int KB, int VB>
__global__ void __launch_bounds__(kThreads, 1)
    kda_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const float* __restrict__ g,
                     const uint16_t* __restrict__ beta, const float* __restrict__ h0, float* __restrict__ ht,
                     uint16_t* __restrict__ o, uint8_t* __restrict__ ws, const WsLayout L, const float scale,
                     const int H) {
    using S = FusedSmem<KB, VB>;
    constexpr int K = S::K, V = S::V, NCG = S::NCG, NSEG = S::NSEG, RS = S::RS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align_smem_1024(smem_raw);
    __shared__ FusedBars B;

    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    if (*reinterpret_cast<volatile int32_t*>(status) != 0) return;  // the planner rejected cu_seqlens
    const int s = blockIdx.x / H, h = blockIdx.x % H;
    const SeqInfo si = reinterpret_cast<const SeqInfo*>(ws + L.seq_info)[s];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);
    float* PARTs = reinterpret_cast<float*>(sm + S::M);
    float* Xsm = reinterpret_cast<float*>(sm + S::XS);
    float* beta_s = reinterpret_cast<float*>(sm + S::BETA);
    float* gds = reinterpret_cast<float*>(sm + S::GDS);
    const Mat64 PM{reinterpret_cast<float*>(sm + S::M)};

    if (tid == 0) {
        mbar_init(&B.qkv, 1);
        mbar_init(&B.mma, 1);
        mbar_init(&B.wh, 1);
        mbar_init(&B.dh, 1);
        mbar_init(&B.acc, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&B.tmem_slot, S::TMEM_COLS);
        tmem_relinquish();
    }
    // [I ; 0]: row r < 64 holds 1.0 at column r (16-byte chunk (r / 8) ^ (r & 7))
    for (int e = tid; e < 16384 / 16; e += kThreads) {
        const int row = e >> 3, ch = e & 7;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (row < 64 && ch == ((row >> 3) ^ (row & 7))) {
            uint32_t wv[4] = {0u, 0u, 0u, 0u};
            wv[(row & 7) >> 1] = (row & 1) ? 0x3F800000u : 0x00003F80u;
            x = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        *reinterpret_cast<uint4*>(sm + S::IDN + e * 16) = x;
    }

    // ---- the state: thread r of warp w owns row r of V block w >> 2 ---------
    const int quad = warp & 3, vb_own = warp >> 2;
    const int r = quad * 32 + lane;                 // state row (key dim) and, for r < 64, token row
    const bool has_row = r < K && vb_own < VB;      // warp-uniform
    float hreg[64];
    {
        const int64_t hrow = (((int64_t)s * H + h) * K + r) * V + vb_own * 64;
        if (has_row && h0 != nullptr) {
            const float4* src = reinterpret_cast<const float4*>(h0 + hrow);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float4 x = src[j];
                hreg[4 * j] = x.x;
                hreg[4 * j + 1] = x.y;
                hreg[4 * j + 2] = x.z;
                hreg[4 * j + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) hreg[j] = 0.f;
        }
    }
    auto write_h = [&]() {  // bf16 copy of h, MN-major SW128 [K rows][64 v] per V block
        if (has_row) {
            uint8_t* hs = sm + S::HS + vb_own * S::HS_BLOCK;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint4 x = make_uint4(pack_bf16x2(hreg[8 * cc], hreg[8 * cc + 1]),
                                           pack_bf16x2(hreg[8 * cc + 2], hreg[8 * cc + 3]),
                                           pack_bf16x2(hreg[8 * cc + 4], hreg[8 * cc + 5]),
                                           pack_bf16x2(hreg[8 * cc + 6], hreg[8 * cc + 7]));
                *reinterpret_cast<uint4*>(hs + r * 128 + ((cc ^ (r & 7)) << 4)) = x;
            }
        }
    };
    write_h();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B.tmem_slot;
    const uint32_t t_acc = tmem + 128;      // V columns: lanes 0-63 = v', 64-127 = -(qg h + Aqk v')
    const uint32_t t_dh = tmem + 128 + V;   // V columns: 128 lanes = K rows
    bool timed_out = false;
    uint32_t ph_qkv = 0, ph_mma = 0, ph_step = 0;
    auto wait0 = [&](uint64_t* bar, uint32_t parity) {  // warp 0 waits; the caller's barrier spreads it
        if (warp == 0 && !mbar_wait(bar, parity, kWaitLimitNs)) timed_out = true;
    };

    const int cg = tid % NCG, seg = tid / NCG;  // this thread's 4-column group and row segment of g
    const int d0 = 4 * cg, kb_d = d0 >> 6, col = d0 & 63;

    for (int c = 0; c < si.tiles; ++c) {
        const int row0 = si.bos + c * 64;
        const int valid = min(64, si.len - c * 64);
        // ---- 0. loads: q, k, v by TMA, g into registers, beta; L2 prefetch of the next chunk
        if (tid == 0) {
            mbar_arrive_expect_tx(&B.qkv, S::QKV_TX);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                tma_load_3d(sm + S::QG(kb), &tm_q, &B.qkv, kb * 64, h, row0);
                tma_load_3d(sm + S::KX(kb), &tm_k, &B.qkv, kb * 64, h, row0);
            }
#pragma unroll
            for (int vb = 0; vb < VB; ++vb) tma_load_3d(sm + S::U + vb * 8192, &tm_v, &B.qkv, vb * 64, h, row0);
        }
        if (warp == 1 && c + 1 < si.tiles) {
            const int prow = row0 + 64, pvalid = min(64, si.len - (c + 1) * 64);
            if (lane == 0) {
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_prefetch_3d(&tm_q, kb * 64, h, prow);
                    tma_prefetch_3d(&tm_k, kb * 64, h, prow);
                }
#pragma unroll
                for (int vb = 0; vb < VB; ++vb) tma_prefetch_3d(&tm_v, vb * 64, h, prow);
            }
            for (int i = lane; i < pvalid; i += 32) bulk_prefetch_l2(g + ((int64_t)(prow + i) * H + h) * K, K * 4);
        }
        float gv[RS][4];
        {
            const float* gp = g + ((int64_t)row0 * H + h) * K + d0;
            const int64_t rstride = (int64_t)H * K;
#pragma unroll
            for (int rr = 0; rr < RS; ++rr) {
                const int i = seg * RS + rr;
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if (i < valid) x = ldg_stream_f4(gp + i * rstride);
                gv[rr][0] = x.x;
                gv[rr][1] = x.y;
                gv[rr][2] = x.z;
                gv[rr][3] = x.w;
            }
        }
        if (tid >= 64 && tid < 128) {
            const int i = tid - 64;
            beta_s[i] = i < valid ? bf_lo((uint32_t)beta[(int64_t)(row0 + i) * H + h]) : 0.f;
        }
        // ---- 1. in-chunk cumsum of g: segment sums, then each row's prefix ----
        {
            float4 sacc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int rr = 0; rr < RS; ++rr) {
                sacc.x += gv[rr][0];
                sacc.y += gv[rr][1];
                sacc.z += gv[rr][2];
                sacc.w += gv[rr][3];
            }
            *reinterpret_cast<float4*>(PARTs + seg * K + d0) = sacc;
        }
        __syncthreads();
        float Gd[4], eG[4];
        bool unsafe;
        {
            float4 base = make_float4(0.f, 0.f, 0.f, 0.f), tot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int sgi = 0; sgi < NSEG; ++sgi) {
                const float4 p = *reinterpret_cast<const float4*>(PARTs + sgi * K + d0);
                if (sgi < seg) {
                    base.x += p.x;
                    base.y += p.y;
                    base.z += p.z;
                    base.w += p.w;
                }
                tot.x += p.x;
                tot.y += p.y;
                tot.z += p.z;
                tot.w += p.w;
            }
            float acc[4] = {base.x, base.y, base.z, base.w};
            float mx = 0.f;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) mx = fmaxf(mx, fabsf(acc[cc] * kLog2e));
#pragma unroll
            for (int rr = 0; rr < RS; ++rr)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    acc[cc] += gv[rr][cc];
                    gv[rr][cc] = acc[cc] * kLog2e;
                    mx = fmaxf(mx, fabsf(gv[rr][cc]));
                }
            Gd[0] = tot.x * kLog2e;
            Gd[1] = tot.y * kLog2e;
            Gd[2] = tot.z * kLog2e;
            Gd[3] = tot.w * kLog2e;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) eG[cc] = ex2(Gd[cc]);
            if (seg == 0) *reinterpret_cast<float4*>(gds + d0) = make_float4(Gd[0], Gd[1], Gd[2], Gd[3]);
            unsafe = !(mx <= kSafeSpanLog2);
        }
        wait0(&B.qkv, ph_qkv);
        ph_qkv ^= 1;
        const bool exact_path = __syncthreads_or(unsafe) != 0;
        if (exact_path && tid == 0) atomicAdd(status + kStatusExactTiles, 1);  // diagnostic count

        // ---- 1b. (rare) exact gated sums for a chunk with extreme decay -------
        if (exact_path) {
            constexpr int kPairs = 64 * 64 / kThreads;
            float* g2h = reinterpret_cast<float*>(sm + S::M);
            float ea[kPairs], eb[kPairs];
#pragma unroll
            for (int n = 0; n < kPairs; ++n) ea[n] = eb[n] = 0.f;
            for (int kb = 0; kb < KB; ++kb) {
                if (kb_d == kb) {
#pragma unroll
                    for (int rr = 0; rr < RS; ++rr)
                        *reinterpret_cast<float4*>(g2h + (seg * RS + rr) * 64 + col) =
                            make_float4(gv[rr][0], gv[rr][1], gv[rr][2], gv[rr][3]);
                }
                __syncthreads();
                exact_sums_block<false>(sm + S::QG(kb), g2h, valid, ea, eb);  // k exp2(g2) slot = qg slot + 8 KB
                __syncthreads();
            }
#pragma unroll
            for (int n = 0; n < kPairs; ++n) {
                const int e = tid + kThreads * n, i = e >> 6, j = e & 63;
                *reinterpret_cast<uint16_t*>(sm + S::AQK + sw128_offset(i, j)) = bf16_bits(ea[n]);
                if (j < i) *PM.at(j, i) = beta_s[i] * eb[n];
            }
        }

        // ---- 2. gating in place: qg, k exp2(g2); k exp2(-g2) -> M; kg -> KG ---
#pragma unroll
        for (int rr = 0; rr < RS; ++rr) {
            const int i = seg * RS + rr;
            const uint32_t off = i * 128 + ((((col >> 3) ^ (i & 7))) << 4) + (col & 7) * 2;
            uint8_t* qs = sm + S::QG(kb_d);
            uint8_t* ks = sm + S::KX(kb_d);
            uint2 qv = *reinterpret_cast<const uint2*>(qs + off);
            uint2 kv = *reinterpret_cast<const uint2*>(ks + off);
            if (i >= valid) qv = kv = make_uint2(0u, 0u);
            const float q4[4] = {bf_lo(qv.x), bf_hi(qv.x), bf_lo(qv.y), bf_hi(qv.y)};
            const float k4[4] = {bf_lo(kv.x), bf_hi(kv.x), bf_lo(kv.y), bf_hi(kv.y)};
            float qg4[4], kga4[4], kin4[4], kg4[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const float e = ex2(gv[rr][cc]);
                qg4[cc] = q4[cc] * e;
                kga4[cc] = k4[cc] * e;
                if (!exact_path) {
                    kin4[cc] = k4[cc] * ex2(-gv[rr][cc]);
                    kg4[cc] = kin4[cc] * eG[cc];
                } else {
                    kin4[cc] = 0.f;
                    kg4[cc] = k4[cc] * ex2(Gd[cc] - gv[rr][cc]);
                }
            }
            *reinterpret_cast<uint2*>(qs + off) = make_uint2(pack_bf16x2(qg4[0], qg4[1]), pack_bf16x2(qg4[2], qg4[3]));
            *reinterpret_cast<uint2*>(ks + off) = make_uint2(pack_bf16x2(kga4[0], kga4[1]), pack_bf16x2(kga4[2], kga4[3]));
            if (!exact_path)
                *reinterpret_cast<uint2*>(sm + S::M + kb_d * 8192 + off) =
                    make_uint2(pack_bf16x2(kin4[0], kin4[1]), pack_bf16x2(kin4[2], kin4[3]));
            *reinterpret_cast<uint2*>(sm + S::KG + kb_d * 8192 + off) =
                make_uint2(pack_bf16x2(kg4[0], kg4[1]), pack_bf16x2(kg4[2], kg4[3]));
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 3. Gram MMA: [qg ; k exp2(g2)] @ (k exp2(-g2))^T -> TMEM cols 0-63
        if (!exact_path) {
            if (tid == 0) {
                tc_fence_after();
                constexpr uint32_t id = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const int kb = ks >> 2, kk = ks & 3;
                    mma_bf16(tmem, smem_desc(sbase + S::QG(kb) + kk * 32, 16, 1024),
                             smem_desc(sbase + S::M + kb * 8192 + kk * 32, 16, 1024), id, ks > 0 ? 1u : 0u);
                }
                mma_commit(&B.mma);
            }
            wait0(&B.mma, ph_mma);
            ph_mma ^= 1;
            __syncthreads();
            tc_fence_after();
            {
                // warp w: TMEM lane quadrant w & 3, column half w >> 2
                const int c0 = (warp >> 2) * 32;
                float rv[32];
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + c0, rv);
                tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + c0 + 16, rv + 16);
                tmem_ld_wait();
                if (quad < 2) {  // Aqk rows (lower triangle with the diagonal) -> AQK, bf16 SW128
                    const int i = quad * 32 + lane;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t wv[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int j = c0 + cc * 8 + 2 * t;
                            wv[t] = pack_bf16x2(j <= i ? rv[cc * 8 + 2 * t] : 0.f,
                                                j + 1 <= i ? rv[cc * 8 + 2 * t + 1] : 0.f);
                        }
                        *reinterpret_cast<uint4*>(sm + S::AQK + sw128_offset(i, c0 + cc * 8)) =
                            make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
                } else {  // Gram rows -> A^T (strict upper triangle of M), beta on the row
                    const int i = (quad - 2) * 32 + lane;
                    const float b = beta_s[i];
#pragma unroll
                    for (int t = 0; t < 32; ++t) {
                        const int j = c0 + t;
                        if (j < i) *PM.at(j, i) = b * rv[t];
                    }
                }
            }
        }
        __syncthreads();

        // ---- 4. T = (I + A)^-1 by 16x16 blocks (fp32), then T' = T diag(beta) --
        unit_lower_inverse(PM, Xsm, tid, warp, lane);
        store_t_prime(PM, beta_s, sm + S::M, tid);
        // v rows past the end of the sequence -> 0 (inert in u)
        for (int e = tid; e < (64 - valid) * 8 * VB; e += kThreads) {
            const int rr = valid + e / (8 * VB), x = e % (8 * VB);
            *reinterpret_cast<uint4*>(sm + S::U + (x >> 3) * 8192 + rr * 128 + (x & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 5. w^T = (k exp2(g2))^T T'^T, u^T = v^T T'^T -> TMEM cols 0-63 / 64-127
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32(128, 64, 1, 0);  // A MN-major, B K-major
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t bd = smem_desc(sbase + S::M + ks * 32, 16, 1024);
                mma_bf16(tmem, smem_desc(sbase + S::KX(0) + ks * 2048, S::KBLK, 1024), bd, id, ks > 0 ? 1u : 0u);
                mma_bf16(tmem + 64, smem_desc(sbase + S::U + ks * 2048, 8192, 1024), bd, id, ks > 0 ? 1u : 0u);
            }
            mma_commit(&B.mma);
        }
        wait0(&B.mma, ph_mma);
        ph_mma ^= 1;
        __syncthreads();
        tc_fence_after();

        // ---- 6. w^T / u^T -> w into the w slots, u over v (stmatrix.trans) -----
        {
            const int i0 = (warp >> 2) * 32;     // token-row half
            const int mat = lane >> 3, mrow = lane & 7;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int L0 = quad * 32 + half * 16;  // dims L0 .. L0 + 15
#pragma unroll
                for (int wu = 0; wu < 2; ++wu) {
                    if (L0 >= (wu == 0 ? K : V)) continue;
                    uint32_t rv[16];
                    tmem_ld16x256_x4(tmem + ((uint32_t)L0 << 16) + wu * 64 + i0, rv);
                    tmem_ld_wait();
                    const uint32_t stg = sbase + (wu == 0 ? S::W(L0 >> 6) : S::U + (L0 >> 6) * 8192);
#pragma unroll
                    for (int g2i = 0; g2i < 2; ++g2i) {
                        const float* f = reinterpret_cast<const float*>(rv) + 8 * g2i;
                        const int tok = i0 + 16 * g2i + 8 * (mat >> 1) + mrow;
                        const int dim = (L0 & 63) + 8 * (mat & 1);
                        stmatrix_x4_trans(stg + sw128_offset(tok, dim), pack_bf16x2(f[0], f[1]),
                                          pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                    }
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- 7. the scan step: ACC = [I;0] u - [w;qg] h; v'; DH = kg^T v';
        //         ACC -= [.;Aqk] v'; h <- exp2(G) h + DH; o = -scale ACC[64..127]
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_h = idesc_bf16_f32(128, V, 0, 1);      // A K-major, B MN-major
            constexpr uint32_t id_hn = idesc_bf16_f32(128, V, 0, 1, 1);  // the same, A negated
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(t_acc, smem_desc(sbase + S::IDN + ks * 32, 16, 1024),
                         smem_desc(sbase + S::U + ks * 2048, 8192, 1024), id_h, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < K / 16; ++ks) {
                const int kb = ks >> 2, kk = ks & 3;
                mma_bf16(t_acc, smem_desc(sbase + S::W(kb) + kk * 32, 16, 1024),
                         smem_desc(sbase + S::HS + ks * 2048, S::HS_BLOCK, 1024), id_hn, 1u);
            }
            mma_commit(&B.wh);
        }
        wait0(&B.wh, ph_step);
        __syncthreads();
        tc_fence_after();
        if (quad < 2 && vb_own < VB) {  // v' rows (token rows = TMEM lanes 0-63) of V block vb_own
            uint8_t* vp = sm + S::VP + vb_own * 8192;
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
                float x[16];
                tmem_ld16(t_acc + (uint32_t)(vb_own * 64) + ((uint32_t)(quad * 32) << 16) + c0, x);
                tmem_ld_wait();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int cc = (c0 >> 3) + hh;
                    const float* y = x + 8 * hh;
                    *reinterpret_cast<uint4*>(vp + r * 128 + ((cc ^ (r & 7)) << 4)) =
                        make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                                   pack_bf16x2(y[6], y[7]));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_dh = idesc_bf16_f32(128, V, 1, 1);      // A = kg^T MN-major
            constexpr uint32_t id_hn = idesc_bf16_f32(128, V, 0, 1, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(t_dh, smem_desc(sbase + S::KG + ks * 2048, 8192, 1024),
                         smem_desc(sbase + S::VP + ks * 2048, 8192, 1024), id_dh, ks > 0 ? 1u : 0u);
            mma_commit(&B.dh);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                mma_bf16(t_acc, smem_desc(sbase + S::AQK - 8192 + ks * 32, 16, 1024),
                         smem_desc(sbase + S::VP + ks * 2048, 8192, 1024), id_hn, 1u);
            mma_commit(&B.acc);
        }
        wait0(&B.dh, ph_step);
        __syncthreads();
        tc_fence_after();
        if (has_row) {  // h <- exp2(G) h + DH
            const float decay = ex2(gds[r]);
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
                float dh[16];
                tmem_ld16(t_dh + (uint32_t)(vb_own * 64) + ((uint32_t)(quad * 32) << 16) + c0, dh);
                tmem_ld_wait();
#pragma unroll
                for (int t = 0; t < 16; ++t) hreg[c0 + t] = fmaf(decay, hreg[c0 + t], dh[t]);
            }
        }
        wait0(&B.acc, ph_step);
        ph_step ^= 1;
        tc_fence_before();
        __syncthreads();  // every read of the old h copy (by the WH MMA) is done; ACC is final
        tc_fence_after();
        write_h();
        if (quad >= 2 && vb_own < VB) {  // o rows (TMEM lanes 64-127) of V block vb_own
            // every lane of the warp takes part in the TMEM loads (they are
            // warp-collective); only the stores are masked to the valid rows
            const int i = (quad - 2) * 32 + lane;
            uint4* dst = reinterpret_cast<uint4*>(o + ((int64_t)(row0 + i) * H + h) * V + vb_own * 64);
            const float nscale = -scale;  // the accumulator holds -(qg h + Aqk v')
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
                float y[16];
                tmem_ld16(t_acc + (uint32_t)(vb_own * 64) + ((uint32_t)(quad * 32) << 16) + c0, y);
                tmem_ld_wait();
                if (i < valid) {
                    dst[c0 / 8] = make_uint4(pack_bf16x2(nscale * y[0], nscale * y[1]),
                                             pack_bf16x2(nscale * y[2], nscale * y[3]),
                                             pack_bf16x2(nscale * y[4], nscale * y[5]),
                                             pack_bf16x2(nscale * y[6], nscale * y[7]));
                    dst[c0 / 8 + 1] = make_uint4(pack_bf16x2(nscale * y[8], nscale * y[9]),
                                                 pack_bf16x2(nscale * y[10], nscale * y[11]),
                                                 pack_bf16x2(nscale * y[12], nscale * y[13]),
                                                 pack_bf16x2(nscale * y[14], nscale * y[15]));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        // the next chunk's loads overwrite qg, k, v / u; a wait that ran out ends the walk
        if (__syncthreads_or(timed_out)) break;
        tc_fence_after();
    }

    if (ht != nullptr && has_row && !timed_out) {
        float4* dst = reinterpret_cast<float4*>(ht + (((int64_t)s * H + h) * K + r) * V + vb_own * 64);
#pragma unroll
        for (int j = 0; j < 16; ++j) dst[j] = make_float4(hreg[4 * j], hreg[4 * j + 1], hreg[4 * j + 2], hreg[4 * j + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, S::TMEM_COLS);
    }
    if (timed_out) atomicOr(status, kStatusTimeout);
}

template <int KB, int VB>
cudaError_t launch_fused_t(const FusedArgs& a, cudaStream_t stream) {
    using S = FusedSmem<KB, VB>;
    const uint32_t smem = S::BYTES + 1024;
    auto kern = kda_fused_kernel<KB, VB>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t ctas = (int64_t)a.N * a.H;
    if (ctas <= 0) return cudaSuccess;
    kern<<<(unsigned)ctas, kThreads, smem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.g, a.beta, a.h0, a.ht, a.o, a.ws,
                                                     a.L, a.scale, a.H);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream) {
    const int KB = a.K / 64, VB = a.V / 64;
    if (KB == 2 && VB == 2) return launch_fused_t<2, 2>(a, stream);
    if (KB == 2 && VB == 1) return launch_fused_t<2, 1>(a, stream);
    if (KB == 1 && VB == 2) return launch_fused_t<1, 2>(a, stream);
    if (KB == 1 && VB == 1) return launch_fused_t<1, 1>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace kda
