// scan.cu -- fused inter-chunk state scan + output of the chunked KDA forward
// (sm_103a).
//
// One CTA per (sequence, head, V tile of 64*NVB columns), serial over the
// sequence's chunks.  Per chunk c, with h the K x (64*NVB) fp32 state tile
// (kernel-fun "kda/_kernels/fwd_state.py", module docstring):
//
//   WH = w @ h;   v' = u - WH  (rounded to bf16)
//   o  = scale * (qg @ h + Aqk @ v')        (Aqk is stored without scale)
//   h <- exp2(G) * h + kg^T @ v'
//
// GB300 mapping (warp-specialised, 256 threads for NVB = 1, 512 for NVB = 2):
//   warps 0..4*NVB-1   recurrence: warp w serves V block w/4; thread r owns
//                      state row r (h[r, 64 columns] in fp32 registers); the
//                      warps of TMEM quadrants 0-1 also form v' for token row r.
//   next warp          TMA producer: w, qg, kg, Aqk (shared by every V block),
//                      u (this V tile) and gd per chunk into a STAGES-deep ring.
//   next warp          tcgen05 issuer + TMEM owner.
//   2*NVB warps        epilogue (TMEM quadrants 2-3): o rows, scaled, bf16.
// Every MMA uses M = 128 (one TMEM lane per accumulator row):
//   ACC[buf] = [w ; qg] @ h           lanes 0-63 = WH, lanes 64-127 = qg@h
//   DH       = kg^T @ v'              (kg read MN-major; 128 lanes = K rows)
//   ACC[buf] += [unused ; Aqk] @ v'   lanes 64-127 become qg@h + Aqk@v'
// The critical path WH -> v' -> DH -> h -> next WH is issued first; the output
// MMA and the epilogue overlap it, ACC is double-buffered across chunks, and
// the input ring lets the loads of the next chunks overlap the current one.
// Every wait is bounded (kWaitLimitNs); a timeout sets the status word and the
// roles unwind without trapping.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

template <int KB, int NVB, int STAGES>
struct ScanCfg {
    static constexpr int K = 64 * KB;
    static constexpr int BV = 64 * NVB;                 // V columns per CTA
    static constexpr int REC_WARPS = 4 * NVB;
    static constexpr int TMA_WARP = REC_WARPS;
    static constexpr int MMA_WARP = REC_WARPS + 1;
    // NVB = 1: warps 0-3 recurrence, 4 TMA, 5 MMA, 6-7 epilogue.
    // NVB = 2: warps 0-7 recurrence, 8 TMA, 9 MMA, 10-11 and 14-15 epilogue
    //          (TMEM quadrants 2-3 for each V block), 12-13 idle.
    static constexpr int THREADS = NVB == 1 ? 256 : 512;
    static constexpr uint32_t TMEM_COLS = NVB == 1 ? 256 : 512;
    // the one-stage variant runs two CTAs per SM (registers capped at 128)
    static constexpr int MIN_CTAS = (NVB == 1 && STAGES == 1) ? 2 : 1;
    // one input stage
    static constexpr uint32_t AW = 0;                    // per kb: [w 8K | qg 8K]
    static constexpr uint32_t AQK = AW + 2 * KB * 8192;  // Aqk [64][64]; the 8K before it = rows 64..
    static constexpr uint32_t KG = AQK + 8192;           // kg per kb [64 tok][64 d]
    static constexpr uint32_t U = KG + KB * 8192;        // u per V block [64 tok][64 v]
    static constexpr uint32_t GD = U + NVB * 8192;       // gd fp32 [K]
    static constexpr uint32_t STAGE = GD + 1024;
    static constexpr uint32_t TX_BYTES = (3 * KB + 1 + NVB) * 8192 + K * 4;
    // persistent
    static constexpr uint32_t HS = STAGES * STAGE;       // h bf16 per V block [K rows][64 v], MN-major SW128
    static constexpr uint32_t HS_BLOCK = KB * 8192;
    static constexpr uint32_t VP = HS + NVB * HS_BLOCK;  // v' bf16 per V block [64 tok][64 v], MN-major SW128
    static constexpr uint32_t BYTES = VP + NVB * 8192;
};

template <int STAGES>
struct ScanBars {
    uint64_t full[STAGES], empty[STAGES];
    uint64_t h_ready, wh_full, vp_ready, dh_full;
    uint64_t acc_full[2], acc_empty[2];
    uint32_t tmem_slot;
    int abort_flag;
};

// Epilogue warp e (0 .. 2*NVB-1): TMEM quadrant 2 + (e & 1), V block e >> 1.
template <int NVB>
__device__ __forceinline__ int epilogue_index(int warp, int first) {
    const int e = warp - first;
    if (NVB == 1) return e;                 // warps first, first+1 = quadrants 2, 3
    return e < 2 ? e : (e >= 4 ? e - 2 : -1);  // warps first..+1 and first+4..+5; +2,+3 idle
}

template <int KB, int NVB, int STAGES>
__global__ void __launch_bounds__(ScanCfg<KB, NVB, STAGES>::THREADS, ScanCfg<KB, NVB, STAGES>::MIN_CTAS)
    kda_scan_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_qg,
                    const __grid_constant__ CUtensorMap tm_kg, const __grid_constant__ CUtensorMap tm_u,
                    const __grid_constant__ CUtensorMap tm_aqk, const void* __restrict__ h0,
                    void* __restrict__ ht, uint16_t* __restrict__ o, uint8_t* __restrict__ ws,
                    const WsLayout L, const float scale, const int H, const int V, const int flags) {
    using S = ScanCfg<KB, NVB, STAGES>;
    constexpr int K = S::K;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ ScanBars<STAGES> B;

    const int NT = V / S::BV;  // V tiles per head
    const int vt = blockIdx.x % NT;
    const int h = (blockIdx.x / NT) % H;
    const int s = blockIdx.x / (NT * H);
    const int v0 = vt * S::BV;
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    if (*reinterpret_cast<volatile int32_t*>(status) != 0) return;
    const SeqInfo si = reinterpret_cast<const SeqInfo*>(ws + L.seq_info)[s];
    const int tiles = si.tiles;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&B.full[i], 1);
            mbar_init(&B.empty[i], 1 + S::REC_WARPS);
        }
        mbar_init(&B.h_ready, S::REC_WARPS);
        mbar_init(&B.wh_full, 1);
        mbar_init(&B.vp_ready, 2 * NVB);
        mbar_init(&B.dh_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B.acc_full[i], 1);
            mbar_init(&B.acc_empty[i], 2 * NVB);
        }
        B.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == S::MMA_WARP) {
        tmem_alloc(&B.tmem_slot, S::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B.tmem_slot;
    const uint32_t t_acc = tmem;                 // 2 x BV columns
    const uint32_t t_dh = tmem + 2 * S::BV;      // BV columns
    volatile int* abort_flag = &B.abort_flag;
    bool timed_out = false;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
        timed_out = true;
        *abort_flag = 1;
        return false;
    };

    if (warp < S::REC_WARPS) {
        // ================= recurrence warps: v' and the state update =================
        const int quad = warp & 3, vb = warp >> 2;
        const int r = quad * 32 + lane;  // state row (key dim) and, for r < 64, token row
        const bool has_row = r < K;      // warp-uniform
        const int col = v0 + vb * 64;    // first V column of this warp's block
        float hreg[64];
        const int64_t hrow = (((int64_t)s * H + h) * K + r) * V + col;  // element offset of this row
        if (has_row && h0 != nullptr && (flags & kScanStateBF16)) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(h0) + hrow);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 x = src[j];
                const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    hreg[8 * j + 2 * t] = bf_lo(xw[t]);
                    hreg[8 * j + 2 * t + 1] = bf_hi(xw[t]);
                }
            }
        } else if (has_row && h0 != nullptr) {
            const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(h0) + hrow);
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
        uint8_t* hs = sm + S::HS + vb * S::HS_BLOCK;
        uint8_t* vp = sm + S::VP + vb * 8192;
        auto write_h = [&]() {
            if (has_row) {
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 x = make_uint4(pack_bf16x2(hreg[8 * cc], hreg[8 * cc + 1]),
                                               pack_bf16x2(hreg[8 * cc + 2], hreg[8 * cc + 3]),
                                               pack_bf16x2(hreg[8 * cc + 4], hreg[8 * cc + 5]),
                                               pack_bf16x2(hreg[8 * cc + 6], hreg[8 * cc + 7]));
                    *reinterpret_cast<uint4*>(hs + r * 128 + ((cc ^ (r & 7)) << 4)) = x;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.h_ready);
        };
        if (tiles > 0) write_h();
        for (int c = 0; c < tiles && !*abort_flag; ++c) {
            const int st = c % STAGES;
            const uint32_t sp = (c / STAGES) & 1;
            uint8_t* stage = sm + st * S::STAGE;
            if (!wait(&B.full[st], sp)) break;
            if (quad < 2) {
                // v'[r, :] = u[r, :] - WH[r, :]
                if (!wait(&B.wh_full, c & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    float wh[16];
                    tmem_ld16(t_acc + (uint32_t)((c & 1) * S::BV + vb * 64) + ((uint32_t)(quad * 32) << 16) + c0,
                              wh);
                    tmem_ld_wait();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int cc = (c0 >> 3) + hh;
                        const uint32_t off = r * 128 + ((cc ^ (r & 7)) << 4);
                        const uint4 uv = *reinterpret_cast<const uint4*>(stage + S::U + vb * 8192 + off);
                        const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
                        uint32_t pw[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t)
                            pw[t] = pack_bf16x2(bf_lo(uw[t]) - wh[8 * hh + 2 * t],
                                                bf_hi(uw[t]) - wh[8 * hh + 2 * t + 1]);
                        *reinterpret_cast<uint4*>(vp + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.vp_ready);
            }
            const float decay = has_row ? ex2(reinterpret_cast<const float*>(stage + S::GD)[r]) : 0.f;
            if (!wait(&B.dh_full, c & 1)) break;
            tc_fence_after();
            if (has_row) {
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    float dh[16];
                    tmem_ld16(t_dh + (uint32_t)(vb * 64) + ((uint32_t)(quad * 32) << 16) + c0, dh);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 16; ++t) hreg[c0 + t] = fmaf(decay, hreg[c0 + t], dh[t]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.empty[st]);
            write_h();
        }
        if (ht != nullptr && has_row && !timed_out && !*abort_flag) {
            if (flags & kScanStateBF16) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(ht) + hrow);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dst[j] = make_uint4(pack_bf16x2(hreg[8 * j], hreg[8 * j + 1]), pack_bf16x2(hreg[8 * j + 2], hreg[8 * j + 3]),
                                        pack_bf16x2(hreg[8 * j + 4], hreg[8 * j + 5]), pack_bf16x2(hreg[8 * j + 6], hreg[8 * j + 7]));
            } else {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(ht) + hrow);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    dst[j] = make_float4(hreg[4 * j], hreg[4 * j + 1], hreg[4 * j + 2], hreg[4 * j + 3]);
            }
        }
    } else if (warp == S::TMA_WARP) {
        // ================= TMA producer =================
        if (lane == 0 && tiles > 0) {
            prefetch_tmap(&tm_w);
            prefetch_tmap(&tm_qg);
            prefetch_tmap(&tm_kg);
            prefetch_tmap(&tm_u);
            prefetch_tmap(&tm_aqk);
            const float* gd = reinterpret_cast<const float*>(ws + L.gd);
            for (int c = 0; c < tiles && !*abort_flag; ++c) {
                const int st = c % STAGES;
                const uint32_t sp = (c / STAGES) & 1;
                if (!wait(&B.empty[st], sp ^ 1)) break;
                uint8_t* stage = sm + st * S::STAGE;
                const int64_t tile = (int64_t)(si.tile_base + c) * H + h;
                const int row = (int)(tile * 64);
                uint64_t* fb = &B.full[st];
                mbar_arrive_expect_tx(fb, S::TX_BYTES);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_load_2d(stage + S::AW + kb * 16384, &tm_w, fb, kb * 64, row);
                    tma_load_2d(stage + S::AW + kb * 16384 + 8192, &tm_qg, fb, kb * 64, row);
                    tma_load_2d(stage + S::KG + kb * 8192, &tm_kg, fb, kb * 64, row);
                }
                tma_load_2d(stage + S::AQK, &tm_aqk, fb, 0, row);
#pragma unroll
                for (int vb = 0; vb < NVB; ++vb) tma_load_2d(stage + S::U + vb * 8192, &tm_u, fb, v0 + vb * 64, row);
                bulk_load_1d(stage + S::GD, gd + tile * K, K * 4, fb);
            }
        }
    } else if (warp == S::MMA_WARP) {
        // ================= tcgen05 issuer =================
        if (lane == 0) {
            constexpr uint32_t id_h = idesc_bf16_f32(128, S::BV, 0, 1);   // A K-major, B (h, v') MN-major
            constexpr uint32_t id_dh = idesc_bf16_f32(128, S::BV, 1, 1);  // A = kg^T MN-major
            for (int c = 0; c < tiles && !*abort_flag; ++c) {
                const int st = c % STAGES;
                const uint32_t sp = (c / STAGES) & 1;
                const int buf = c & 1;
                const uint32_t bp = (c >> 1) & 1;
                const uint32_t stage = sbase + st * S::STAGE;
                if (!wait(&B.full[st], sp)) break;
                if (!wait(&B.h_ready, c & 1)) break;
                if (!wait(&B.acc_empty[buf], bp ^ 1)) break;
                tc_fence_after();
                const uint32_t d_acc = t_acc + buf * S::BV;
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const int kb = ks >> 2, kk = ks & 3;
                    mma_bf16(d_acc, smem_desc(stage + S::AW + kb * 16384 + kk * 32, 16, 1024),
                             smem_desc(sbase + S::HS + ks * 2048, S::HS_BLOCK, 1024), id_h, ks > 0 ? 1u : 0u);
                }
                mma_commit(&B.wh_full);
                if (!wait(&B.vp_ready, c & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(t_dh, smem_desc(stage + S::KG + ks * 2048, 8192, 1024),
                             smem_desc(sbase + S::VP + ks * 2048, 8192, 1024), id_dh, ks > 0 ? 1u : 0u);
                mma_commit(&B.dh_full);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(d_acc, smem_desc(stage + S::AQK - 8192 + ks * 32, 16, 1024),
                             smem_desc(sbase + S::VP + ks * 2048, 8192, 1024), id_h, 1u);
                mma_commit(&B.acc_full[buf]);
                mma_commit(&B.empty[st]);
            }
        }
    } else {
        // ================= epilogue: o = scale * (qg@h + Aqk@v') =================
        const int e = epilogue_index<NVB>(warp, S::MMA_WARP + 1);
        if (e >= 0) {
            const int quad = 2 + (e & 1);          // TMEM lanes 64..127
            const int vb = e >> 1;
            const int i = (quad - 2) * 32 + lane;  // token row within the chunk
            for (int c = 0; c < tiles && !*abort_flag; ++c) {
                const int buf = c & 1;
                const uint32_t bp = (c >> 1) & 1;
                if (!wait(&B.acc_full[buf], bp)) break;
                tc_fence_after();
                float acc[64];
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16)
                    tmem_ld16(t_acc + (uint32_t)(buf * S::BV + vb * 64) + ((uint32_t)(quad * 32) << 16) + c0,
                              acc + c0);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.acc_empty[buf]);
                const int valid = min(64, si.len - c * 64);
                if (i < valid) {
                    uint4* dst = reinterpret_cast<uint4*>(
                        o + ((int64_t)(si.bos + c * 64 + i) * H + h) * V + v0 + vb * 64);
                    if (flags & kScanOutF16) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_uint4(pack_f16x2(scale * acc[8 * j], scale * acc[8 * j + 1]),
                                                pack_f16x2(scale * acc[8 * j + 2], scale * acc[8 * j + 3]),
                                                pack_f16x2(scale * acc[8 * j + 4], scale * acc[8 * j + 5]),
                                                pack_f16x2(scale * acc[8 * j + 6], scale * acc[8 * j + 7]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            dst[j] = make_uint4(pack_bf16x2(scale * acc[8 * j], scale * acc[8 * j + 1]),
                                                pack_bf16x2(scale * acc[8 * j + 2], scale * acc[8 * j + 3]),
                                                pack_bf16x2(scale * acc[8 * j + 4], scale * acc[8 * j + 5]),
                                                pack_bf16x2(scale * acc[8 * j + 6], scale * acc[8 * j + 7]));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == S::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, S::TMEM_COLS);
    }
    if (timed_out) atomicOr(status, kStatusTimeout);
}

template <int KB, int NVB, int STAGES>
cudaError_t launch_scan_t(const ScanArgs& a, cudaStream_t stream) {
    using S = ScanCfg<KB, NVB, STAGES>;
    const uint32_t smem = S::BYTES + 1024;
    auto kern = kda_scan_kernel<KB, NVB, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t ctas = (int64_t)a.N * a.H * (a.V / S::BV);
    if (ctas <= 0) return cudaSuccess;
    kern<<<(unsigned)ctas, S::THREADS, smem, stream>>>(a.tm_w, a.tm_qg, a.tm_kg, a.tm_u, a.tm_aqk, a.h0,
                                                       a.ht, a.o, a.ws, a.L, a.scale, a.H, a.V, a.flags);
    return cudaGetLastError();
}

template <int KB>
cudaError_t launch_scan_k(const ScanArgs& a, cudaStream_t stream, int sms) {
    const int64_t ctas64 = (int64_t)a.N * a.H * (a.V / 64);
    // Few CTAs: each SM holds at most one, so give it a two-deep input ring.
    if (ctas64 <= sms) return launch_scan_t<KB, 1, 2>(a, stream);
    // Many CTAs with V = 128: one CTA per (sequence, head) covering all of V,
    // two-deep ring, w/qg/kg/Aqk loaded once per head.
    if (a.V % 128 == 0) return launch_scan_t<KB, 2, 2>(a, stream);
    // Many CTAs with V = 64: two CTAs per SM, one stage each.
    return launch_scan_t<KB, 1, 1>(a, stream);
}

}  // namespace

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 148;
    if (a.K == 128) return launch_scan_k<2>(a, stream, sms);
    if (a.K == 64) return launch_scan_k<1>(a, stream, sms);
    return cudaErrorInvalidValue;
}

}  // namespace kda
