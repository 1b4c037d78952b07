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
//   2*NVB warps        epilogue (TMEM quadrants 2-3): o rows, scaled, bf16,
//                      staged in shared memory and sent 32 rows per warp by
//                      TMA stores (a tail's partial rows from registers).
// Every MMA uses M = 128 (one TMEM lane per accumulator row):
//   ACC[buf]  = [I ; 0] @ u            lanes 0-63 = u (exact), 64-127 = 0
//   ACC[buf] += -[w ; qg] @ h          lanes 0-63 = u - WH = v', 64-127 = -qg@h
//   DH        = kg^T @ v'              (kg read MN-major; 128 lanes = K rows)
//   ACC[buf] += -[unused ; Aqk] @ v'   lanes 64-127 = -(qg@h + Aqk@v')
// (the A operand negated through the instruction descriptor; the epilogue
// scales by -scale).  The u term needs no state, so it is issued ahead, while
// the previous chunk's state update runs, and v' leaves TMEM ready to round.
// The critical path WH -> v' -> DH -> h -> next WH is issued first; the output
// MMA and the epilogue overlap it, ACC is double-buffered across chunks, and
// the input ring lets the loads of the next chunks overlap the current one.
// Every wait is bounded (kWaitLimitNs); a timeout sets the status word and the
// roles unwind without trapping.
#include <cuda_bf16.h>

#include "chunk_math.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;


// The descriptor of an operand `bytes` past the one that `d` describes, with
// the same strides: the offset (16-byte aligned) goes into the 14-bit start
// address field, which cannot carry since shared memory ends below 256 KB.
// The issue loop builds each operand's descriptor once and steps it with this.
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

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
    // One input stage, in two parts: part A holds what the u and WH MMAs read
    // (and gd), part B what DH and the output MMAs read.  In the 128-column
    // shape (SPLIT) each part has its own barriers, so part A of a later chunk
    // starts loading as soon as WH has read this one, about half a chunk
    // before DH and the output are done.  The 64-column shapes keep one
    // barrier phase per chunk: each phase of TMA loads costs an SM about as
    // much as seven 8 KB boxes of data (measured on GB300), more than the
    // earlier start of a 40 KB part A gains there.
    static constexpr bool SPLIT = NVB == 2;
    static constexpr uint32_t AW = 0;  // part A: per kb [w 8K | qg 8K]
    // split: [AW | u | kg | Aqk]; one phase: [AW | Aqk | kg | u] (the order
    // measured fastest for each)
    static constexpr uint32_t U = SPLIT ? AW + 2 * KB * 8192 : AW + (3 * KB + 1) * 8192;  // u per V block
    static constexpr uint32_t KG = SPLIT ? U + NVB * 8192 : AW + (2 * KB + 1) * 8192;     // part B: kg per kb
    static constexpr uint32_t AQK = SPLIT ? KG + KB * 8192 : AW + 2 * KB * 8192;          // Aqk [64][64]
    // the 8K before Aqk (kg, or qg in the one-phase order) are the unused A
    // rows 0..63 of the output MMA
    static constexpr uint32_t STAGE = AW + (3 * KB + 1 + NVB) * 8192;
    static constexpr uint32_t TXA_BYTES = (2 * KB + NVB) * 8192 + K * 4;
    static constexpr uint32_t TXB_BYTES = (KB + 1) * 8192;
    // persistent
    static constexpr uint32_t HS = STAGES * STAGE;       // h bf16 per V block [K rows][64 v], MN-major SW128
    static constexpr uint32_t HS_BLOCK = KB * 8192;
    static constexpr uint32_t VP = HS + NVB * HS_BLOCK;  // v' bf16 per V block [64 tok][64 v], MN-major SW128
    // [I_64 ; 0] bf16, K-major SW128 [128 rows][64 tok]: the A operand that puts u into the accumulator
    static constexpr uint32_t IDN = VP + NVB * 8192;
    static constexpr uint32_t GDS = IDN + 16384;         // gd fp32 [K] of each ring stage (stage st at GDS + st * 4K)
    // o leaves by TMA stores from a staging copy [64 tok][64 v] (SW128) per V
    // block, each epilogue warp storing its own 32 rows (a tail's partial rows
    // leave from registers); the two-CTAs-per-SM shape (one stage) has no
    // room for it and stores every row from registers
    static constexpr bool TMA_O = STAGES == 2;
    static constexpr uint32_t OST = (GDS + STAGES * K * 4 + 1023) / 1024 * 1024;
    static constexpr uint32_t BYTES = TMA_O ? OST + NVB * 8192 : GDS + STAGES * K * 4;
};

template <int STAGES>
struct ScanBars {
    uint64_t full_a[STAGES], empty_a[STAGES], full_b[STAGES], empty_b[STAGES];
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
                    const __grid_constant__ CUtensorMap tm_aqk, const __grid_constant__ CUtensorMap tm_o,
                    const void* __restrict__ h0,
                    void* __restrict__ ht, uint16_t* __restrict__ o, uint8_t* __restrict__ ws,
                    const WsLayout L, const float scale, const int N, const int H, const int V, const int flags,
                    const int mode, const int seg_base) {
    using S = ScanCfg<KB, NVB, STAGES>;
    constexpr int K = S::K;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align_smem_1024(smem_raw);
    __shared__ ScanBars<STAGES> B;

    // Column space: V columns of h (output mode) or, in map mode, K + V
    // columns [P | Q] of a segment's affine map h_out = P h_in + Q.
    const bool map_mode = mode == kScanModeMap;
    const int NCOL = map_mode ? K + V : V;
    const int NT = NCOL / S::BV;  // column tiles per head
    const int vt = blockIdx.x % NT;
    const int h = (blockIdx.x / NT) % H;
    const int s = blockIdx.x / (NT * H);
    const int seg = seg_base + (int)blockIdx.y;
    const int v0 = vt * S::BV;
    // launched after the kernel whose results this one reads (the intra
    // kernel, the map pass or the combine step)
    grid_dep_launch();
    grid_dep_wait();
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    if (*reinterpret_cast<volatile int32_t*>(status) != 0) return;
    const SeqInfo si = reinterpret_cast<const SeqInfo*>(ws + L.seq_info)[s];
    const int tiles = si.tiles;
    // this CTA's chunks [c_begin, c_end) of the sequence
    const int c_begin = seg * L.seg_len;
    const int c_end = min(tiles, c_begin + L.seg_len);
    const bool map_out = (flags & kScanMapOut) != 0;  // map of the whole sequence, to the caller
    if (seg > 0 && c_begin >= tiles) return;   // the sequence has fewer segments
    if (map_mode && !map_out && c_end >= tiles) return;  // the last segment's map is never used
    const int nit = c_end > c_begin ? c_end - c_begin : 0;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&B.full_a[i], 1);
            mbar_init(&B.empty_a[i], 1 + S::REC_WARPS);
            mbar_init(&B.full_b[i], 1);
            mbar_init(&B.empty_b[i], 1);
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
    // [I ; 0] operand; in map mode the u slots of P column blocks are never
    // loaded and hold zeros (those columns see u = 0)
    for (int e = tid; e < 16384 / 16; e += S::THREADS) {
        const int row = e >> 3, ch = e & 7;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        // row < 64: 1.0 at column row, i.e. in 16-byte chunk (row / 8) ^ (row & 7)
        if (row < 64 && ch == ((row >> 3) ^ (row & 7))) {
            uint32_t wv[4] = {0u, 0u, 0u, 0u};
            wv[(row & 7) >> 1] = (row & 1) ? 0x3F800000u : 0x00003F80u;
            x = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        *reinterpret_cast<uint4*>(sm + S::IDN + e * 16) = x;
    }
    if (map_mode) {
        for (int vb = 0; vb < NVB; ++vb) {
            if (v0 + vb * 64 >= K) continue;
            for (int e = tid; e < STAGES * 512; e += S::THREADS)
                *reinterpret_cast<uint4*>(sm + (e >> 9) * S::STAGE + S::U + vb * 8192 + (e & 511) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
        }
    }
    fence_proxy_async_smem();
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
        // map mode: P columns start as the identity and see u = 0; Q columns start at 0
        const bool p_block = map_mode && col < K;
        if (map_mode) {
#pragma unroll
            for (int j = 0; j < 64; ++j) hreg[j] = (p_block && r == col + j) ? 1.f : 0.f;
        } else if (seg > 0) {
            const float4* src = reinterpret_cast<const float4*>(
                reinterpret_cast<const float*>(ws + L.hin) + ((((int64_t)seg * N + s) * H + h) * K + r) * V + col);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float4 x = has_row ? src[j] : make_float4(0.f, 0.f, 0.f, 0.f);
                hreg[4 * j] = x.x;
                hreg[4 * j + 1] = x.y;
                hreg[4 * j + 2] = x.z;
                hreg[4 * j + 3] = x.w;
            }
        } else if (has_row && h0 != nullptr && (flags & kScanStateBF16)) {
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
        if (nit > 0) write_h();
        for (int it = 0; it < nit && !*abort_flag; ++it) {
            const int st = it % STAGES;
            const uint32_t sp = (it / STAGES) & 1;
            if (!wait(&B.full_a[st], sp)) break;
            // gd is the only part of the stage these warps read
            const float decay = has_row ? ex2(reinterpret_cast<const float*>(sm + S::GDS + st * K * 4)[r]) : 0.f;
            if (S::SPLIT) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.empty_a[st]);
            }
            if (quad < 2) {
                // v'[r, :] = u[r, :] - WH[r, :], formed in TMEM by the MMAs
                if (!wait(&B.wh_full, it & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    float x[16];
                    tmem_ld16(t_acc + (uint32_t)((it & 1) * S::BV + vb * 64) + ((uint32_t)(quad * 32) << 16) + c0,
                              x);
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
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.vp_ready);
            }
            if (!wait(&B.dh_full, it & 1)) break;
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
            if (!S::SPLIT) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.empty_a[st]);
            }
            write_h();
        }
        if (map_mode && has_row && !timed_out && !*abort_flag) {
            float* base = map_out ? static_cast<float*>(ht) : reinterpret_cast<float*>(ws + L.pq);
            float4* dst = reinterpret_cast<float4*>(base + ((((int64_t)seg * N + s) * H + h) * K + r) * (K + V) + col);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                dst[j] = make_float4(hreg[4 * j], hreg[4 * j + 1], hreg[4 * j + 2], hreg[4 * j + 3]);
        } else if (!map_mode && c_end < tiles && (flags & kScanExitToHin) && has_row && !timed_out &&
                   !*abort_flag) {
            // a chunk range of the staged forward: the exit state enters the next range
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(ws + L.hin) +
                                                    ((((int64_t)(seg + 1) * N + s) * H + h) * K + r) * V + col);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                dst[j] = make_float4(hreg[4 * j], hreg[4 * j + 1], hreg[4 * j + 2], hreg[4 * j + 3]);
        } else if (!map_mode && c_end == tiles && ht != nullptr && has_row && !timed_out && !*abort_flag) {
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
        if (lane == 0 && nit > 0) {
            prefetch_tmap(&tm_w);
            prefetch_tmap(&tm_qg);
            prefetch_tmap(&tm_kg);
            prefetch_tmap(&tm_u);
            prefetch_tmap(&tm_aqk);
            const float* gd = reinterpret_cast<const float*>(ws + L.gd);
            // map mode reads neither qg nor Aqk (no output) nor u for P columns
            uint32_t txa = S::TXA_BYTES, txb = S::TXB_BYTES;
            if (map_mode) {
                txa -= KB * 8192;  // no qg
                txb -= 8192;       // no Aqk
#pragma unroll
                for (int vb = 0; vb < NVB; ++vb)
                    if (v0 + vb * 64 < K) txa -= 8192;
            }
            for (int it = 0; it < nit && !*abort_flag; ++it) {
                const int c = c_begin + it;
                const int st = it % STAGES;
                const uint32_t sp = (it / STAGES) & 1;
                if (!wait(&B.empty_a[st], sp ^ 1)) break;
                uint8_t* stage = sm + st * S::STAGE;
                const int64_t tile = (int64_t)(si.tile_base + c) * H + h;
                const int row = (int)(tile * 64);
                uint64_t* fb = &B.full_a[st];
                mbar_arrive_expect_tx(fb, S::SPLIT ? txa : txa + txb);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb) {
                    tma_load_2d(stage + S::AW + kb * 16384, &tm_w, fb, kb * 64, row);
                    if (!map_mode) tma_load_2d(stage + S::AW + kb * 16384 + 8192, &tm_qg, fb, kb * 64, row);
                    if (!S::SPLIT) tma_load_2d(stage + S::KG + kb * 8192, &tm_kg, fb, kb * 64, row);
                }
                if (!S::SPLIT && !map_mode) tma_load_2d(stage + S::AQK, &tm_aqk, fb, 0, row);
#pragma unroll
                for (int vb = 0; vb < NVB; ++vb) {
                    const int cb = v0 + vb * 64;
                    if (!map_mode) tma_load_2d(stage + S::U + vb * 8192, &tm_u, fb, cb, row);
                    else if (cb >= K) tma_load_2d(stage + S::U + vb * 8192, &tm_u, fb, cb - K, row);
                }
                bulk_load_1d(sm + S::GDS + st * K * 4, gd + tile * K, K * 4, fb);
                if (S::SPLIT) {
                    if (!wait(&B.empty_b[st], sp ^ 1)) break;
                    fb = &B.full_b[st];
                    mbar_arrive_expect_tx(fb, txb);
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb) tma_load_2d(stage + S::KG + kb * 8192, &tm_kg, fb, kb * 64, row);
                    if (!map_mode) tma_load_2d(stage + S::AQK, &tm_aqk, fb, 0, row);
                }
            }
        }
    } else if (warp == S::MMA_WARP) {
        // ================= tcgen05 issuer =================
        if (lane == 0) {
            constexpr uint32_t id_h = idesc_bf16_f32(128, S::BV, 0, 1);   // A K-major, B (u, h, v') MN-major
            constexpr uint32_t id_hn = idesc_bf16_f32(128, S::BV, 0, 1, 1);  // the same with A negated
            constexpr uint32_t id_dh = idesc_bf16_f32(128, S::BV, 1, 1);  // A = kg^T MN-major
            // operand descriptors built once (the ring's at stage 0); the issue
            // loop steps them by constant offsets and the stage
            const uint64_t d_idn = smem_desc(sbase + S::IDN, 16, 1024);
            const uint64_t d_hs = smem_desc(sbase + S::HS, S::HS_BLOCK, 1024);
            const uint64_t d_vp = smem_desc(sbase + S::VP, 8192, 1024);
            const uint64_t d_u = smem_desc(sbase + S::U, 8192, 1024);
            const uint64_t d_aw = smem_desc(sbase + S::AW, 16, 1024);
            const uint64_t d_kg = smem_desc(sbase + S::KG, 8192, 1024);
            const uint64_t d_aqk = smem_desc(sbase + S::AQK - 8192, 16, 1024);
            for (int it = 0; it < nit && !*abort_flag; ++it) {
                const int st = it % STAGES;
                const uint32_t sp = (it / STAGES) & 1;
                const int buf = it & 1;
                const uint32_t bp = (it >> 1) & 1;
                const uint32_t so = (uint32_t)st * S::STAGE;  // this stage's offset in the ring
                if (!wait(&B.full_a[st], sp)) break;
                if (!wait(&B.acc_empty[buf], bp ^ 1)) break;
                tc_fence_after();
                const uint32_t d_acc = t_acc + buf * S::BV;
                // ACC = [I ; 0] @ u, ahead of the state
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(d_acc, desc_at(d_idn, ks * 32), desc_at(d_u, so + ks * 2048), id_h, ks > 0 ? 1u : 0u);
                if (!wait(&B.h_ready, it & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const int kb = ks >> 2, kk = ks & 3;
                    mma_bf16(d_acc, desc_at(d_aw, so + kb * 16384 + kk * 32), desc_at(d_hs, ks * 2048), id_hn, 1u);
                }
                mma_commit(&B.wh_full);
                if (S::SPLIT) mma_commit(&B.empty_a[st]);  // u and WH have read part A
                if (!wait(&B.vp_ready, it & 1)) break;
                if (S::SPLIT && !wait(&B.full_b[st], sp)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(t_dh, desc_at(d_kg, so + ks * 2048), desc_at(d_vp, ks * 2048), id_dh, ks > 0 ? 1u : 0u);
                mma_commit(&B.dh_full);
                if (!map_mode) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_bf16(d_acc, desc_at(d_aqk, so + ks * 32), desc_at(d_vp, ks * 2048), id_hn, 1u);
                }
                mma_commit(&B.acc_full[buf]);
                mma_commit(S::SPLIT ? &B.empty_b[st] : &B.empty_a[st]);
            }
        }
    } else {
        // ================= epilogue: o = scale * (qg@h + Aqk@v') =================
        const int e = epilogue_index<NVB>(warp, S::MMA_WARP + 1);
        if (e >= 0) {
            const int quad = 2 + (e & 1);          // TMEM lanes 64..127
            const int vb = e >> 1;
            const int i = (quad - 2) * 32 + lane;  // token row within the chunk
            for (int it = 0; it < nit && !*abort_flag; ++it) {
                const int c = c_begin + it;
                const int buf = it & 1;
                const uint32_t bp = (it >> 1) & 1;
                if (!wait(&B.acc_full[buf], bp)) break;
                tc_fence_after();
                if (map_mode) {  // no output: hand the accumulator back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&B.acc_empty[buf]);
                    continue;
                }
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
                const float nscale = -scale;  // the accumulator holds -(qg@h + Aqk@v')
                uint4 packed[8];  // this token row's 64 outputs, scaled and rounded
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float* y = acc + 8 * j;
                    packed[j] = (flags & kScanOutF16)
                                    ? make_uint4(pack_f16x2(nscale * y[0], nscale * y[1]),
                                                 pack_f16x2(nscale * y[2], nscale * y[3]),
                                                 pack_f16x2(nscale * y[4], nscale * y[5]),
                                                 pack_f16x2(nscale * y[6], nscale * y[7]))
                                    : make_uint4(pack_bf16x2(nscale * y[0], nscale * y[1]),
                                                 pack_bf16x2(nscale * y[2], nscale * y[3]),
                                                 pack_bf16x2(nscale * y[4], nscale * y[5]),
                                                 pack_bf16x2(nscale * y[6], nscale * y[7]));
                }
                const int row_lo = (quad - 2) * 32;  // this warp's 32 token rows
                if (S::TMA_O && valid >= row_lo + 32) {
                    // all 32 rows real: into this warp's staging copy, then one TMA
                    // store issued by lane 0 once its previous store has read the copy
                    uint8_t* stg = sm + S::OST + vb * 8192 + row_lo * 128;
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = packed[j];
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&tm_o, stg, v0 + vb * 64, h, si.bos + c * 64 + row_lo);
                        bulk_commit();
                    }
                } else if (i < valid) {
                    uint4* dst = reinterpret_cast<uint4*>(
                        o + ((int64_t)(si.bos + c * 64 + i) * H + h) * V + v0 + vb * 64);
#pragma unroll
                    for (int j = 0; j < 8; ++j) dst[j] = packed[j];
                }
            }
            if (S::TMA_O && lane == 0) bulk_wait_read0();  // the staging outlives the stores' reads
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

// Shared memory a scan CTA of the staged forward reserves: with it no
// intra-chunk CTA (about 55 KB including the per-CTA reservation) fits on the
// same SM, so the intra kernel of the next chunk range runs on the SMs the
// scan leaves idle and does not take issue slots from the scan's serial chain.
constexpr uint32_t kStageScanSmem = 180 * 1024;

// stage < 0: the plain or segmented scan (mode); stage >= 0: chunk range
// `stage` of the staged forward, one CTA per (sequence, head, V tile).
template <int KB, int NVB, int STAGES>
cudaError_t launch_scan_t(const ScanArgs& a, int mode, cudaStream_t stream, int stage = -1) {
    using S = ScanCfg<KB, NVB, STAGES>;
    uint32_t smem = S::BYTES + 1024;
    if (stage >= 0 && smem < kStageScanSmem) smem = kStageScanSmem;
    auto kern = kda_scan_kernel<KB, NVB, STAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int ncol = mode == kScanModeMap ? a.K + a.V : a.V;
    const int64_t ctas = (int64_t)a.N * a.H * (ncol / S::BV);
    const int segs = (stage >= 0 || (a.flags & kScanMapOut)) ? 1
                     : mode == kScanModeMap                 ? a.L.seg_count - 1
                                                            : a.L.seg_count;
    if (ctas <= 0 || segs <= 0) return cudaSuccess;
    WsLayout L = a.L;
    int flags = a.flags;
    if (stage >= 0) {  // the kernel's segment arithmetic over the chunk ranges
        L.seg_count = L.stage_count;
        L.seg_len = L.stage_len;
        flags |= kScanExitToHin;
    }
    const dim3 grid((unsigned)ctas, (unsigned)segs);
    if (stage < 0)  // the staged forward's ranges follow event waits: plain launches there
        return launch_dependent(kern, grid, dim3(S::THREADS), smem, stream, a.tm_w, a.tm_qg, a.tm_kg, a.tm_u,
                                a.tm_aqk, a.tm_o, a.h0, a.ht, a.o, a.ws, L, a.scale, a.N, a.H, a.V, flags, mode, 0);
    kern<<<grid, S::THREADS, smem, stream>>>(a.tm_w, a.tm_qg, a.tm_kg, a.tm_u, a.tm_aqk, a.tm_o, a.h0, a.ht, a.o, a.ws,
                                             L, a.scale, a.N, a.H, a.V, flags, mode, stage);
    return cudaGetLastError();
}

template <int KB>
cudaError_t launch_scan_k(const ScanArgs& a, int mode, cudaStream_t stream, int sms, int stage = -1) {
    const int ncol = mode == kScanModeMap ? a.K + a.V : a.V;
    const int segs = (stage >= 0 || (a.flags & kScanMapOut)) ? 1
                     : mode == kScanModeMap                 ? a.L.seg_count - 1
                                                            : a.L.seg_count;
    const ScanShape sh = scan_shape((int64_t)a.N * a.H * (ncol / 64) * segs, ncol, sms);
    // Few CTAs: each SM holds at most one, so give it a two-deep input ring.
    if (sh.nvb == 1 && sh.stages == 2) return launch_scan_t<KB, 1, 2>(a, mode, stream, stage);
    // Many CTAs with 128-column tiles: one CTA covers 128 columns, two-deep
    // ring, w/qg/kg/Aqk loaded once per 128 columns.
    if (sh.nvb == 2) return launch_scan_t<KB, 2, 2>(a, mode, stream, stage);
    // Many CTAs otherwise: two CTAs per SM, one stage each.
    return launch_scan_t<KB, 1, 1>(a, mode, stream, stage);
}

// Chains the segment maps of the map pass: for every (sequence, head, 16
// columns of V), h_in[0] = h0 and h_in[j+1] = P_j h_in[j] + Q_j in fp32, for
// the segments the sequence has.  Two threads per state row r (2K threads):
// each sums the products over one half of the key dims for the row's 16
// columns, and a lane exchange adds the halves, so a step's serial work is
// half a row.  P_j (K x K) streams into a double buffer by cp.async while the
// previous step computes; its rows keep their 16-byte chunks XOR-swizzled by
// (row & 7), and the second half walks its chunks four places rotated, so the
// two threads of a row read different banks.  h_in[j] (K x 16) is
// double-buffered and read as broadcast float4s; the second half takes the
// rows of each group of four in the order 1 0 3 2, so the two broadcast rows
// of a warp never share a bank.
constexpr int kCombineCols = 16;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// The same kernel chains the maps of consecutive token ranges for the
// context-parallel forward: explicit pointers, a fixed count of maps
// (nseg_fixed > 0, no sequence table, no status word) and h_in[0] = h0
// written out too.
template <int K>
__global__ void __launch_bounds__(2 * K) kda_seg_combine_kernel(const void* __restrict__ h0,
                                                                const float* __restrict__ pq,
                                                                float* __restrict__ hin,
                                                                const int32_t* __restrict__ status,
                                                                const SeqInfo* __restrict__ seqs, const int seg_len,
                                                                const int nseg_fixed, const int N, const int H,
                                                                const int V, const int flags) {
    constexpr int C = kCombineCols, K4 = K / 4, HK4 = K4 / 2, NTH = 2 * K;
    extern __shared__ float4 csm4[];
    float4* Ps = csm4;              // 2 x [K][K / 4], chunk-swizzled rows
    float4* Hs = csm4 + 2 * K * K4;  // 2 x [K][C / 4]
    const int NTV = V / C;
    const int vt = blockIdx.x % NTV, h = (blockIdx.x / NTV) % H, s = blockIdx.x / (NTV * H);
    grid_dep_launch();
    grid_dep_wait();  // the map pass (or the caller's earlier work) has written pq
    if (status != nullptr && *reinterpret_cast<const volatile int32_t*>(status) != 0) return;
    int nseg = nseg_fixed;
    if (nseg_fixed <= 0) {
        const SeqInfo si = seqs[s];
        nseg = (si.tiles + seg_len - 1) / seg_len;
    }
    const int tid = threadIdx.x;
    const int col0 = vt * C;
    const int r = tid >> 1, half = tid & 1;  // state row, half of the key dims
    if (nseg_fixed > 0 && half == 0) {  // h_in[0] = h0 (the first range's entry)
        float4* dst = reinterpret_cast<float4*>(hin + (((int64_t)s * H + h) * K + r) * V + col0);
        const float* src = h0 != nullptr ? static_cast<const float*>(h0) + (((int64_t)s * H + h) * K + r) * V + col0
                                         : nullptr;
#pragma unroll
        for (int c4 = 0; c4 < C / 4; ++c4)
            dst[c4] = src != nullptr ? *reinterpret_cast<const float4*>(src + 4 * c4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (nseg < 2) return;
    auto map_of = [&](int j) { return pq + (((int64_t)j * N + s) * H + h) * K * (K + V); };
    auto stage_p = [&](int j) {  // issue the copies of P_j into buffer j & 1
        const float* PQ = map_of(j);
        float4* dst = Ps + (j & 1) * K * K4;
        for (int e4 = tid; e4 < K * K4; e4 += NTH) {
            const int row = e4 / K4, c4 = e4 % K4;
            cp_async16(dst + row * K4 + (c4 ^ (row & 7)), PQ + (int64_t)row * (K + V) + 4 * c4);
        }
        cp_async_commit();
    };
    stage_p(0);
    if (half == 0) {
        float hr[C];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            float x = 0.f;
            if (h0 != nullptr) {
                const int64_t off = (((int64_t)s * H + h) * K + r) * V + col0 + c;
                x = (flags & kScanStateBF16)
                        ? __uint_as_float(((uint32_t) static_cast<const uint16_t*>(h0)[off]) << 16)
                        : static_cast<const float*>(h0)[off];
            }
            hr[c] = x;
        }
#pragma unroll
        for (int c4 = 0; c4 < C / 4; ++c4)
            Hs[r * (C / 4) + c4] = make_float4(hr[4 * c4], hr[4 * c4 + 1], hr[4 * c4 + 2], hr[4 * c4 + 3]);
    }
    for (int j = 0; j + 1 < nseg; ++j) {
        // this thread's half of Q_j's row (columns 8 half .. + 7), fetched ahead of the sums
        const float* qrow = map_of(j) + (int64_t)r * (K + V) + K + col0 + 8 * half;
        const float4 qa = *reinterpret_cast<const float4*>(qrow);
        const float4 qb = *reinterpret_cast<const float4*>(qrow + 4);
        if (j + 2 < nseg) {
            stage_p(j + 1);  // overlaps this step
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float4* P = Ps + (j & 1) * K * K4;
        const float4* Hc = Hs + (j & 1) * K * (C / 4);
        float4* Hn = Hs + ((j + 1) & 1) * K * (C / 4);
        float acc[C];
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] = 0.f;
#pragma unroll 2
        for (int i = 0; i < HK4; ++i) {
            const int k4 = half ? HK4 + ((i + 4) & (HK4 - 1)) : i;
            const float4 p4 = P[r * K4 + (k4 ^ (r & 7))];
            const float pk[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int kx = kk ^ half;  // the second half takes rows 1 0 3 2
                const float pv = half ? pk[kk ^ 1] : pk[kk];
#pragma unroll
                for (int c4 = 0; c4 < C / 4; ++c4) {
                    const float4 x = Hc[(4 * k4 + kx) * (C / 4) + c4];
                    acc[4 * c4] = fmaf(pv, x.x, acc[4 * c4]);
                    acc[4 * c4 + 1] = fmaf(pv, x.y, acc[4 * c4 + 1]);
                    acc[4 * c4 + 2] = fmaf(pv, x.z, acc[4 * c4 + 2]);
                    acc[4 * c4 + 3] = fmaf(pv, x.w, acc[4 * c4 + 3]);
                }
            }
        }
        // both halves of the row, then this thread's 8 columns plus Q
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], 1);
        float a8[8];  // this thread's columns, selected without indexing acc at run time
#pragma unroll
        for (int c = 0; c < 8; ++c) a8[c] = half ? acc[8 + c] : acc[c];
        const float4 x0 = make_float4(a8[0] + qa.x, a8[1] + qa.y, a8[2] + qa.z, a8[3] + qa.w);
        const float4 x1 = make_float4(a8[4] + qb.x, a8[5] + qb.y, a8[6] + qb.z, a8[7] + qb.w);
        Hn[r * (C / 4) + 2 * half] = x0;
        Hn[r * (C / 4) + 2 * half + 1] = x1;
        float4* dst = reinterpret_cast<float4*>(hin + ((((int64_t)(j + 1) * N + s) * H + h) * K + r) * V + col0 +
                                                8 * half);
        dst[0] = x0;
        dst[1] = x1;
        __syncthreads();
    }
}

template <int K>
cudaError_t launch_combine_raw(const void* h0, const float* pq, float* hin, const int32_t* status,
                               const SeqInfo* seqs, int seg_len, int nseg_fixed, int N, int H, int V, int flags,
                               cudaStream_t stream) {
    const uint32_t smem = (2 * K * (K / 4) + 2 * K * (kCombineCols / 4)) * sizeof(float4);
    auto kern = kda_seg_combine_kernel<K>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t ctas = (int64_t)N * H * (V / kCombineCols);
    if (ctas <= 0) return cudaSuccess;
    return launch_dependent(kern, dim3((unsigned)ctas), dim3(2 * K), smem, stream, h0, pq, hin, status, seqs, seg_len,
                            nseg_fixed, N, H, V, flags);
}

template <int K>
cudaError_t launch_combine_k(const ScanArgs& a, cudaStream_t stream) {
    return launch_combine_raw<K>(a.h0, reinterpret_cast<const float*>(a.ws + a.L.pq),
                                 reinterpret_cast<float*>(a.ws + a.L.hin),
                                 reinterpret_cast<const int32_t*>(a.ws + a.L.status),
                                 reinterpret_cast<const SeqInfo*>(a.ws + a.L.seq_info), a.L.seg_len, 0, a.N, a.H,
                                 a.V, a.flags, stream);
}

}  // namespace

cudaError_t launch_seg_combine(const void* h0, uint8_t* ws, const WsLayout& L, int N, int H, int K, int V,
                               int flags, cudaStream_t stream) {
    ScanArgs a{};
    a.h0 = h0;
    a.ws = ws;
    a.L = L;
    a.N = N;
    a.H = H;
    a.K = K;
    a.V = V;
    a.flags = flags;
    if (K == 128) return launch_combine_k<128>(a, stream);
    if (K == 64) return launch_combine_k<64>(a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream) {
    const int sms = device_sm_count();
    if (a.K != 128 && a.K != 64) return cudaErrorInvalidValue;
    auto run = [&](int mode) {
        return a.K == 128 ? launch_scan_k<2>(a, mode, stream, sms) : launch_scan_k<1>(a, mode, stream, sms);
    };
    if (a.L.seg_count > 1) {
        // segmented: maps of every segment but the last, chain them, then the
        // output pass over all segments in parallel
        cudaError_t e = run(kScanModeMap);
        if (e != cudaSuccess) return e;
        e = a.K == 128 ? launch_combine_k<128>(a, stream) : launch_combine_k<64>(a, stream);
        if (e != cudaSuccess) return e;
    }
    return run(kScanModeOutput);
}

cudaError_t launch_scan_map_out(const ScanArgs& a, cudaStream_t stream) {
    const int sms = device_sm_count();
    if (a.K != 128 && a.K != 64) return cudaErrorInvalidValue;
    ScanArgs m = a;
    m.flags |= kScanMapOut;
    m.L.seg_len = 0x7fffffff;  // one segment: every chunk of each sequence
    return a.K == 128 ? launch_scan_k<2>(m, kScanModeMap, stream, sms) : launch_scan_k<1>(m, kScanModeMap, stream, sms);
}

cudaError_t launch_chain_states(const float* pq, const float* h0, float* h_in, int ranges, int N, int H, int K, int V,
                                cudaStream_t stream) {
    if (ranges < 1) return cudaErrorInvalidValue;
    if (K == 128) return launch_combine_raw<128>(h0, pq, h_in, nullptr, nullptr, 1, ranges, N, H, V, 0, stream);
    if (K == 64) return launch_combine_raw<64>(h0, pq, h_in, nullptr, nullptr, 1, ranges, N, H, V, 0, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_scan_stage(const ScanArgs& a, int stage, cudaStream_t stream) {
    const int sms = device_sm_count();
    if (a.K != 128 && a.K != 64) return cudaErrorInvalidValue;
    if (a.L.stage_count < 2 || a.L.seg_count > 1 || stage < 0 || stage >= a.L.stage_count)
        return cudaErrorInvalidValue;
    return a.K == 128 ? launch_scan_k<2>(a, kScanModeOutput, stream, sms, stage)
                      : launch_scan_k<1>(a, kScanModeOutput, stream, sms, stage);
}

}  // namespace kda
