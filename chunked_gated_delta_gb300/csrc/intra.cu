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
// GB300 mapping: 256 threads, 52 KB of shared memory, 128 TMEM columns and
// 64 registers per thread, so four tiles are in flight on every SM (the SM's
// 512 TMEM columns bound it there).
//  * q, k (3-D maps over [rows, H, dim], 128-byte swizzle, straight into the
//    layouts the tensor core reads) and, when it does not fit the q slots, v
//    arrive by TMA.  g never enters shared memory: each thread owns a block of
//    4 key dims x RS rows and reads it from global memory into registers with
//    16-byte loads (one warp reads whole 512-byte rows), forms its segment sums
//    (pass 1), then its g2 prefix from all segments' sums (pass 2), and gates
//    its q / k elements in place.  Rows past the end of the sequence are
//    zeroed on chip, so padding rows are inert.
//  * Gated products use one gate factorisation, (q exp2(g2)) . (k exp2(-g2)),
//    so Aqk and the k.k^T Gram matrix come out of ONE tcgen05 MMA with M = 128
//    (A operand = [qg ; k exp2(g2)] stacked, B = k exp2(-g2)), accumulated in
//    TMEM.  If a chunk's |g2| exceeds kSafeSpanLog2 anywhere (factors would
//    overflow), that chunk computes the gated sums exactly per element instead.
//  * T is found block-wise in fp32: the four 16x16 diagonal blocks by
//    forward substitution, then the off-diagonal blocks level by level,
//    T_IJ = -T_II sum_{J<=K<I} A_IK T_KJ, as warp-level m16n8k8 tf32 MMAs
//    with fp32 accumulation (16x16 products on the latency path, where a
//    tcgen05 round trip would cost more than the math).  A is strictly lower
//    triangular and T unit lower triangular, so both live in ONE 64x64 fp32
//    matrix: A^T in the strict upper triangle, T's strict lower triangle below
//    it.  Once the substitution has consumed A's diagonal blocks, T's diagonal
//    blocks are stored whole (unit diagonal, zeros above), so the later
//    products read T without masks.
//  * w and u are computed transposed, w^T = (k exp2(g2))^T T'^T and
//    u^T = v^T T'^T: the key / value dim is the MMA's M = 128, so every TMEM
//    lane holds real data, and 128 columns of TMEM suffice.
//  * qg, w and u leave through TMA stores from swizzled shared memory; Aqk,
//    kg and gd through direct stores.
//  * Shared memory, in order of use: the QK region holds q and k, gated in
//    place into qg and k exp2(g2); the qg slots receive v once the qg store and
//    the Gram MMA have read them (when V <= K), and finally the w staging; the
//    k exp2(g2) slots take the u staging once the w MMA has read them.  The
//    16 KB M region holds the segment sums, then k exp2(-g2), then A^T + T,
//    then T' (bf16, rewritten in place).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "chunk_math.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kThreads = kChunkThreads;

template <int KB, int VB>
struct IntraSmem {
    static constexpr int K = 64 * KB, V = 64 * VB;
    static constexpr int NCG = K / 4;             // 4-column groups
    static constexpr int NSEG = kThreads / NCG;   // row segments
    static constexpr int RS = 64 / NSEG;          // rows per segment
    // QK: per kb [q -> qg -> v block kb (V <= K) -> w staging 8K |
    //             k -> k exp2(g2) -> u staging 8K]
    static constexpr uint32_t QK = 0;
    // M (16 KB): segment sums fp32 [NSEG][K] -> k exp2(-g2) (KB x 8 KB) ->
    // A^T + T fp32 [64][64] -> T' bf16 SW128 [64][64] (g2 blocks on the exact path)
    static constexpr uint32_t M = QK + 2 * KB * 8192;
    static constexpr uint32_t XS = M + 16384;     // X halves fp32 [6][16][8]
    static constexpr uint32_t BETA = XS + 6 * 512;  // beta fp32 [64]
    // v takes the qg slots (block vb at QK + 16 KB * vb) unless V > K
    static constexpr bool V_OWN = VB > KB;
    static constexpr uint32_t VS = V_OWN ? ((BETA + 256 + 1023) / 1024) * 1024 : QK;
    static constexpr uint32_t VSTRIDE = V_OWN ? 8192 : 16384;
    __device__ static constexpr uint32_t ustg(int vb) { return V_OWN ? VS + vb * 8192 : QK + vb * 16384 + 8192; }
    // The transposed w / u MMAs with K or V = 64 read 8 KB past their operand
    // (rows that land in unused TMEM lanes): QK + 16 KB .. + 24 KB, inside
    // the allocation in every case.
    static constexpr uint32_t BYTES = V_OWN ? VS + VB * 8192 : BETA + 256;
    static constexpr uint32_t QK_TX = 2 * KB * 8192, V_TX = VB * 8192;
    static_assert(NSEG * K * 4 == 4096, "segment sums are 4 KB");
    static_assert(BYTES >= 24576, "operand over-reads stay inside the allocation");
};

// flags: kIntraBetaLogits = beta holds logits (sigmoid applied here).
// group: value heads per q/k head (value head h reads q/k head h / group).
// Four CTAs per SM (52 KB of shared memory, 64 registers, 128 TMEM columns).
template <int KB, int VB, bool F16>
__global__ void __launch_bounds__(kThreads, 4)
    kda_intra_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap st_qg,
                     const __grid_constant__ CUtensorMap st_w, const __grid_constant__ CUtensorMap st_u,
                     const float* __restrict__ g, const uint16_t* __restrict__ beta, uint8_t* __restrict__ ws,
                     const WsLayout L, const int H, const int flags, const int group, const int beta_stride,
                     const int beta_head0, const int pf_dist) {
    using S = IntraSmem<KB, VB>;
    constexpr int K = S::K, V = S::V, NCG = S::NCG, NSEG = S::NSEG, RS = S::RS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align_smem_1024(smem_raw);
    __shared__ uint64_t bar_qk, bar_v, bar_mma;
    __shared__ uint32_t tmem_slot;

    // launched after the planner: its chunk table and status word first
    grid_dep_launch();
    grid_dep_wait();
    const int64_t tile = blockIdx.x;  // chunk * H + head
    const int c = static_cast<int>(tile / H), h = static_cast<int>(tile % H);
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    const ChunkInfo ci = reinterpret_cast<const ChunkInfo*>(ws + L.chunk_info)[c];
    if (ci.valid <= 0 || *reinterpret_cast<volatile int32_t*>(status) != 0) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int valid = ci.valid, row0 = ci.row0;
    const int trow = static_cast<int>(tile * 64);  // first row of this tile in the workspace maps
    const uint32_t sbase = smem_u32(sm);
    float* PARTs = reinterpret_cast<float*>(sm + S::M);
    float* Xsm = reinterpret_cast<float*>(sm + S::XS);
    float* beta_s = reinterpret_cast<float*>(sm + S::BETA);
    const Mat64 PM{reinterpret_cast<float*>(sm + S::M)};

    // ---- 0. this thread's g block [RS rows][4 dims] -> registers ------------
    const int cg = tid % NCG, seg = tid / NCG;  // 4-column group, row segment
    const int d0 = 4 * cg, kb_d = d0 >> 6, col = d0 & 63;
    float gv[RS][4];
    {
        const float* gp = g + ((int64_t)row0 * H + h) * K + d0;
        const int64_t rstride = (int64_t)H * K;
#pragma unroll
        for (int r = 0; r < RS; ++r) {
            const int i = seg * RS + r;
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < valid) x = ldg_stream_f4(gp + i * rstride);
            gv[r][0] = x.x;
            gv[r][1] = x.y;
            gv[r][2] = x.z;
            gv[r][3] = x.w;
        }
    }
    // L2 prefetch of the inputs of the tile pf_dist ahead in launch order: the
    // tile a CTA starting about half a CTA lifetime from now takes, so its
    // loads find q, k, v and g in L2 instead of waiting on DRAM
    if (warp == 1 && pf_dist > 0 && tile + pf_dist < (int64_t)gridDim.x) {
        const int64_t pt = tile + pf_dist;
        const int pc = static_cast<int>(pt / H), ph = static_cast<int>(pt % H);
        const ChunkInfo pci = reinterpret_cast<const ChunkInfo*>(ws + L.chunk_info)[pc];
        if (pci.valid > 0) {
            if (lane == 0) {
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_prefetch_3d(&tm_q, kb * 64, ph / group, pci.row0);
                    tma_prefetch_3d(&tm_k, kb * 64, ph / group, pci.row0);
                }
#pragma unroll
                for (int vb = 0; vb < VB; ++vb) tma_prefetch_3d(&tm_v, vb * 64, ph, pci.row0);
            }
            for (int i = lane; i < pci.valid; i += 32)
                bulk_prefetch_l2(g + ((int64_t)(pci.row0 + i) * H + ph) * K, K * 4);
        }
    }
    if (tid == 0) {
        mbar_init(&bar_qk, 1);
        mbar_init(&bar_v, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar_qk, S::QK_TX);
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
            tma_load_3d(sm + S::QK + kb * 16384, &tm_q, &bar_qk, kb * 64, h / group, row0);
            tma_load_3d(sm + S::QK + kb * 16384 + 8192, &tm_k, &bar_qk, kb * 64, h / group, row0);
        }
        if constexpr (S::V_OWN) {
            mbar_arrive_expect_tx(&bar_v, S::V_TX);
#pragma unroll
            for (int vb = 0; vb < VB; ++vb)
                tma_load_3d(sm + S::VS + vb * 8192, &tm_v, &bar_v, vb * 64, h, row0);
        }
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, 128);
        tmem_relinquish();
    }
    if (tid >= 64 && tid < 128) {
        const int i = tid - 64;
        float b = 0.f;
        if (i < valid) {
            b = in_lo<F16>((uint32_t)beta[(int64_t)(row0 + i) * beta_stride + beta_head0 + h]);
            if (flags & kIntraBetaLogits) b = 1.f / (1.f + ex2(-b * kLog2e));  // sigmoid
        }
        beta_s[i] = b;
    }

    // ---- 1. pass 1: segment sums ---------------------------------------------
    {
        float4 sacc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < RS; ++r) {
            sacc.x += gv[r][0];
            sacc.y += gv[r][1];
            sacc.z += gv[r][2];
            sacc.w += gv[r][3];
        }
        *reinterpret_cast<float4*>(PARTs + seg * K + d0) = sacc;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    bool timed_out = false;

    // ---- 1'. pass 2: g2 prefix (log2 space), G, overflow guard ---------------
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
        for (int r = 0; r < RS; ++r)
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                acc[cc] += gv[r][cc];
                gv[r][cc] = acc[cc] * kLog2e;
                mx = fmaxf(mx, fabsf(gv[r][cc]));
            }
        Gd[0] = tot.x * kLog2e;
        Gd[1] = tot.y * kLog2e;
        Gd[2] = tot.z * kLog2e;
        Gd[3] = tot.w * kLog2e;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) eG[cc] = ex2(Gd[cc]);
        if (seg == 0)
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(ws + L.gd) + tile * K + d0) =
                make_float4(Gd[0], Gd[1], Gd[2], Gd[3]);
        unsafe = !(mx <= kSafeSpanLog2);
    }
    if (warp == 0 && !mbar_wait(&bar_qk, 0, kWaitLimitNs)) timed_out = true;
    const bool exact_path = __syncthreads_or(unsafe) != 0;
    if (exact_path && tid == 0) atomicAdd(status + kStatusExactTiles, 1);  // diagnostic count

    uint16_t* aqk_g = reinterpret_cast<uint16_t*>(ws + L.aqk) + tile * 64 * 64;

    // ---- 1b. (rare) exact gated sums for chunks with extreme decay -----------
    if (exact_path) {
        // one 64-dim block of g2 at a time in the M region (the segment sums
        // are dead), fp32 [64][64]
        constexpr int kPairs = 64 * 64 / kThreads;
        float* g2h = reinterpret_cast<float*>(sm + S::M);
        float ea[kPairs], eb[kPairs];
#pragma unroll
        for (int n = 0; n < kPairs; ++n) ea[n] = eb[n] = 0.f;
        for (int kb = 0; kb < KB; ++kb) {
            if (kb_d == kb) {
#pragma unroll
                for (int r = 0; r < RS; ++r)
                    *reinterpret_cast<float4*>(g2h + (seg * RS + r) * 64 + col) =
                        make_float4(gv[r][0], gv[r][1], gv[r][2], gv[r][3]);
            }
            __syncthreads();
            exact_sums_block<F16>(sm + S::QK + kb * 16384, g2h, valid, ea, eb);
            __syncthreads();  // every read of this g2 block is done
        }
#pragma unroll
        for (int n = 0; n < kPairs; ++n) {
            const int e = tid + kThreads * n, i = e >> 6, j = e & 63;
            aqk_g[e] = bf16_bits(ea[n]);  // zero above the diagonal
            if (j < i) *PM.at(j, i) = beta_s[i] * eb[n];
        }
    }

    // ---- 2. gate this thread's q / k block in place; kg to global ------------
    {
        uint8_t* qs = sm + S::QK + kb_d * 16384;
        uint16_t* kg_g = reinterpret_cast<uint16_t*>(ws + L.kg) + tile * 64 * K + d0;
#pragma unroll
        for (int r = 0; r < RS; ++r) {
            const int i = seg * RS + r;
            const uint32_t off = i * 128 + ((((col >> 3) ^ (i & 7))) << 4) + (col & 7) * 2;
            uint2 qv = *reinterpret_cast<const uint2*>(qs + off);
            uint2 kv = *reinterpret_cast<const uint2*>(qs + 8192 + off);
            if (i >= valid) qv = kv = make_uint2(0u, 0u);
            const float q4[4] = {in_lo<F16>(qv.x), in_hi<F16>(qv.x), in_lo<F16>(qv.y), in_hi<F16>(qv.y)};
            const float k4[4] = {in_lo<F16>(kv.x), in_hi<F16>(kv.x), in_lo<F16>(kv.y), in_hi<F16>(kv.y)};
            float qg4[4], kga4[4], kin4[4], kg4[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const float e = ex2(gv[r][cc]);
                qg4[cc] = q4[cc] * e;
                kga4[cc] = k4[cc] * e;
                if (!exact_path) {
                    kin4[cc] = k4[cc] * ex2(-gv[r][cc]);
                    kg4[cc] = kin4[cc] * eG[cc];
                } else {
                    kin4[cc] = 0.f;
                    kg4[cc] = k4[cc] * ex2(Gd[cc] - gv[r][cc]);
                }
            }
            *reinterpret_cast<uint2*>(qs + off) = make_uint2(pack_bf16x2(qg4[0], qg4[1]), pack_bf16x2(qg4[2], qg4[3]));
            *reinterpret_cast<uint2*>(qs + 8192 + off) =
                make_uint2(pack_bf16x2(kga4[0], kga4[1]), pack_bf16x2(kga4[2], kga4[3]));
            if (!exact_path)
                *reinterpret_cast<uint2*>(sm + S::M + kb_d * 8192 + off) =
                    make_uint2(pack_bf16x2(kin4[0], kin4[1]), pack_bf16x2(kin4[2], kin4[3]));
            *reinterpret_cast<uint2*>(kg_g + i * K) = make_uint2(pack_bf16x2(kg4[0], kg4[1]), pack_bf16x2(kg4[2], kg4[3]));
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

    uint32_t mma_phase = 0;
    // ---- 3. Gram MMA: [qg ; k exp2(g2)] @ (k exp2(-g2))^T -> TMEM ------------
    if (!exact_path) {
        if (warp == 0) {
            if (lane == 0) {
                tc_fence_after();
                constexpr uint32_t id = idesc_bf16_f32(128, 64, 0, 0);
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const int kb = ks >> 2, kk = ks & 3;
                    const uint64_t ad = smem_desc(sbase + S::QK + kb * 16384 + kk * 32, 16, 1024);
                    const uint64_t bd = smem_desc(sbase + S::M + kb * 8192 + kk * 32, 16, 1024);
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
                // rows of q.k -> Aqk (lower triangle with diagonal), direct stores
                const int i = quad * 32 + lane;
                uint4* dst = reinterpret_cast<uint4*>(aqk_g + i * 64 + c0);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t wv[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int j = c0 + cc * 8 + 2 * t;
                        wv[t] = pack_bf16x2(j <= i ? r[cc * 8 + 2 * t] : 0.f, j + 1 <= i ? r[cc * 8 + 2 * t + 1] : 0.f);
                    }
                    dst[cc] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            } else {
                // rows of k.k -> A^T, the strict upper triangle of M (A is
                // strictly lower, beta on the row); the Gram MMA has finished
                // reading k exp2(-g2) from M
                const int i = (quad - 2) * 32 + lane;
                const float b = beta_s[i];
#pragma unroll
                for (int t = 0; t < 32; ++t) {
                    const int j = c0 + t;
                    if (j < i) *PM.at(j, i) = b * r[t];
                }
            }
        }
    }
    if (tid == 0) {
        bulk_wait_read0();  // the qg store has read the qg slots
        if constexpr (!S::V_OWN) {
            // v into the qg slots (the Gram MMA has read them too); it is
            // needed only by the u MMA, after the inverse
            mbar_arrive_expect_tx(&bar_v, S::V_TX);
#pragma unroll
            for (int vb = 0; vb < VB; ++vb)
                tma_load_3d(sm + S::VS + vb * S::VSTRIDE, &tm_v, &bar_v, vb * 64, h, row0);
        }
    }
    __syncthreads();
    // ---- 4. T = (I + A)^-1 by 16x16 blocks, fp32, into M's strict lower
    // triangle; then T' = T diag(beta) in bf16 over M
    unit_lower_inverse(PM, Xsm, tid, warp, lane);
    store_t_prime(PM, beta_s, sm + S::M, tid);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 5. w^T = (k exp2(g2))^T T'^T, u^T = v^T T'^T  (M = 128 = key / value dims)
    if (warp == 0 && !mbar_wait(&bar_v, 0, kWaitLimitNs)) timed_out = true;
    __syncthreads();
    if constexpr (F16) {
        // fp16 v -> bf16 in place (the u MMA pairs it with the bf16 T'); rows
        // past the end -> 0
        for (int e = tid; e < 64 * 8 * VB; e += kThreads) {
            const int rr = e / (8 * VB), x = e % (8 * VB);
            uint4* p = reinterpret_cast<uint4*>(sm + S::VS + (x >> 3) * S::VSTRIDE + rr * 128 + (x & 7) * 16);
            uint4 y = make_uint4(0u, 0u, 0u, 0u);
            if (rr < valid) {
                const uint4 hv = *p;
                y = make_uint4(pack_bf16x2(in_lo<true>(hv.x), in_hi<true>(hv.x)),
                               pack_bf16x2(in_lo<true>(hv.y), in_hi<true>(hv.y)),
                               pack_bf16x2(in_lo<true>(hv.z), in_hi<true>(hv.z)),
                               pack_bf16x2(in_lo<true>(hv.w), in_hi<true>(hv.w)));
            }
            *p = y;
        }
    } else {
        for (int e = tid; e < (64 - valid) * 8 * VB; e += kThreads) {  // zero v rows past the end
            const int rr = valid + e / (8 * VB), x = e % (8 * VB);
            *reinterpret_cast<uint4*>(sm + S::VS + (x >> 3) * S::VSTRIDE + rr * 128 + (x & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        if (lane == 0) {
            tc_fence_after();
            constexpr uint32_t id = idesc_bf16_f32(128, 64, 1, 0);  // A MN-major, B K-major
            // For K or V = 64 the second 64 rows of the MMA's M read the
            // 8 KB one block stride further on (rows that land in unused TMEM
            // lanes).
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t bd = smem_desc(sbase + S::M + ks * 32, 16, 1024);
                mma_bf16(tmem, smem_desc(sbase + S::QK + 8192 + ks * 2048, KB == 2 ? 16384 : 8192, 1024), bd, id,
                         ks > 0 ? 1u : 0u);
                mma_bf16(tmem + 64, smem_desc(sbase + S::VS + ks * 2048, S::VSTRIDE, 1024), bd, id,
                         ks > 0 ? 1u : 0u);
            }
            mma_commit(&bar_mma);
        }
        __syncwarp();
        if (!mbar_wait(&bar_mma, mma_phase, kWaitLimitNs)) timed_out = true;
    }
    __syncthreads();
    tc_fence_after();

    // ---- 6. w^T / u^T -> swizzled [i][dim] staging -> TMA stores -------------
    // Each warp reads 16-lane (dim) x 32-column (token) blocks in the m16n8
    // fragment layout and writes them transposed, 8x8 bf16 matrices at a time.
    // w first: its stores read their staging while the warps stage u, so the
    // tile's end waits only for u's.
    {
        const int quad = warp & 3, i0 = (warp >> 2) * 32;  // TMEM lane quadrant, token-row half
        const int mat = lane >> 3, mrow = lane & 7;         // the stmatrix row this lane addresses
#pragma unroll
        for (int wu = 0; wu < 2; ++wu) {        // 0: w (columns i0..), 1: u (columns 64 + i0..)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int L0 = quad * 32 + half * 16;  // dims L0 .. L0 + 15
                if (L0 >= (wu == 0 ? K : V)) continue;
                uint32_t r[16];
                tmem_ld16x256_x4(tmem + ((uint32_t)L0 << 16) + wu * 64 + i0, r);
                tmem_ld_wait();
                const uint32_t stg = sbase + (wu == 0 ? S::QK + (L0 >> 6) * 16384 : S::ustg(L0 >> 6));
#pragma unroll
                for (int g2 = 0; g2 < 2; ++g2) {
                    // matrices: 0 = dims L0.., tokens i0 + 16 g2 ..; 1 = dims L0 + 8..;
                    // 2 and 3 the same for the next 8 tokens
                    const float* f = reinterpret_cast<const float*>(r) + 8 * g2;
                    const int tok = i0 + 16 * g2 + 8 * (mat >> 1) + mrow;
                    const int dim = (L0 & 63) + 8 * (mat & 1);
                    stmatrix_x4_trans(stg + sw128_offset(tok, dim), pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                }
            }
            fence_proxy_async_smem();
            if (wu == 1) tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                if (wu == 0) {
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb) tma_store_2d(&st_w, sm + S::QK + kb * 16384, kb * 64, trow);
                } else {
#pragma unroll
                    for (int vb = 0; vb < VB; ++vb) tma_store_2d(&st_u, sm + S::ustg(vb), vb * 64, trow);
                }
                bulk_commit();
            }
        }
    }
    if (tid == 0) bulk_wait_read0();  // smem must outlive the reads; the writes complete with the grid
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
    if (timed_out) atomicOr(status, kStatusTimeout);
}

template <int KB, int VB, bool F16>
cudaError_t launch_intra_t(const IntraArgs& a, cudaStream_t stream) {
    using S = IntraSmem<KB, VB>;
    const uint32_t smem = S::BYTES + 1024;
    auto kern = kda_intra_kernel<KB, VB, F16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // four CTAs per SM need the largest shared-memory carveout
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    const int64_t ctas = a.max_chunks * a.H;
    if (ctas <= 0) return cudaSuccess;
    // prefetch distance in tiles, measured at 4 tiles resident per SM: 1.25 x
    // SMs (about a third of a tile lifetime ahead) ran best at K = 128 (0.460
    // -> 0.434 ms at the headline; half an SM-count or less, and 4 x SMs, ran
    // slower than none); at K = 64 every distance tried ran slower, so off
    const int pf_dist = KB == 2 ? 5 * device_sm_count() / 4 : 0;
    if (a.after_planner)
        return launch_dependent(kern, dim3((unsigned)ctas), dim3(kThreads), smem, stream, a.tm_q, a.tm_k, a.tm_v,
                                a.st_qg, a.st_w, a.st_u, a.g, a.beta, a.ws, a.L, a.H, a.flags, a.group,
                                a.beta_stride, a.beta_head0, pf_dist);
    kern<<<(unsigned)ctas, kThreads, smem, stream>>>(a.tm_q, a.tm_k, a.tm_v, a.st_qg, a.st_w, a.st_u, a.g,
                                                     a.beta, a.ws, a.L, a.H, a.flags, a.group, a.beta_stride,
                                                     a.beta_head0, pf_dist);
    return cudaGetLastError();
}

template <bool F16>
cudaError_t launch_intra_d(const IntraArgs& a, cudaStream_t stream) {
    const int KB = a.K / 64, VB = a.V / 64;
    if (KB == 2 && VB == 2) return launch_intra_t<2, 2, F16>(a, stream);
    if (KB == 2 && VB == 1) return launch_intra_t<2, 1, F16>(a, stream);
    if (KB == 1 && VB == 2) return launch_intra_t<1, 2, F16>(a, stream);
    if (KB == 1 && VB == 1) return launch_intra_t<1, 1, F16>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_intra(const IntraArgs& a, cudaStream_t stream) {
    if (a.group < 1 || a.H % a.group != 0) return cudaErrorInvalidValue;
    return a.f16 ? launch_intra_d<true>(a, stream) : launch_intra_d<false>(a, stream);
}

}  // namespace kda
