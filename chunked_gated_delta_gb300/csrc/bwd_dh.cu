// bwd_dh.cu -- reverse state scan of the chunked KDA forward (sm_103a): the
// gradient of the loss with respect to the recurrent state, chunk by chunk.
//
// One CTA per (sequence, head, V tile of 64*NVB columns), serial over the
// sequence's chunks, newest first.  With dh the gradient with respect to the
// state after the chunk (kernel-fun "kda/_kernels/bwd_dhu.py", module
// docstring; dh starts at dht):
//
//   dhck[c] = dh                          (bf16 checkpoint, before the update)
//   dv2     = kg @ dh + dv_in             (rounded to bf16; gradient w.r.t. v')
//   dh     <- exp2(G) * dh + scale * qg^T @ do - w^T @ dv2
//   dh0     = dh after the oldest chunk   (fp32)
//
// It reads qg, kg, w and gd from the workspace the intra-chunk kernel wrote
// for the same inputs, so a training step runs kda_fwd (or kda_fwd_intra)
// first and keeps its workspace.
//
// GB300 mapping (warp-specialised, the forward scan's layout):
//   warps 0..4*NVB-1   recurrence: thread r owns dh row r (fp32 registers) and,
//                      in TMEM quadrants 0-1, token row r of dv2.
//   next warp          TMA producer: kg, qg, w (workspace), do and dv_in (user
//                      tensors) and gd per chunk into a STAGES-deep ring; with
//                      fp16 gradients the warp also rewrites each landed do
//                      tile as bf16 for the qg^T @ do product.
//   next warp          tcgen05 issuer + TMEM owner.
//   next warp          TMA stores: each chunk's checkpoint from the bf16 dh
//                      copy and, for a full chunk, dv2 from its bf16 copy;
//                      then it releases both copies for the next chunk.
// MMAs, all M = 128:
//   DV  = [I ; *] @ dv_in     TMEM lanes 0-63 = dv_in exactly (lanes 64-127 unused)
//   DV += [kg ; qg] @ dh      lanes 0-63 = dv2 before rounding
//   QD  = qg^T @ do           qg read MN-major; 128 lanes = K rows; two buffers
//   WD  = w^T @ dv2           w read MN-major
// DV's dv_in term and QD need no state: they are issued as soon as a chunk's
// tiles land, during the previous chunk's update, so the chain
// DV -> dv2 -> WD -> dh -> next DV carries only the state-dependent products.
// Rows of a tail chunk past the sequence end have qg = kg = w = 0 in the
// workspace, so do there contributes nothing; dv2 rows there are masked.
//
// Segmented (few sequences x heads over long sequences, the forward's plan):
// the reverse update is affine in dh, dh_in = (Diag(2^G) - w^T kg) dh_out +
// (scale qg^T do - w^T dv_in), so a map pass runs every segment but the
// oldest from [I | 0] over K + V columns (do = dv_in = 0 on the P columns)
// and stores [P | Q]; the forward's combine kernel chains them newest first
// from dht; the output pass runs all segments in parallel from their entry
// gradients, each writing its own checkpoints and dv2 rows, the oldest dh0.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "chunk_math.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

__device__ __forceinline__ float h_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))); }
__device__ __forceinline__ float h_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

template <int KB, int NVB, int STAGES>
struct BwdCfg {
    static constexpr int K = 64 * KB;
    static constexpr int BV = 64 * NVB;
    static constexpr int REC_WARPS = 4 * NVB;
    static constexpr int TMA_WARP = REC_WARPS;
    static constexpr int MMA_WARP = REC_WARPS + 1;
    static constexpr int STORE_WARP = REC_WARPS + 2;
    static constexpr int THREADS = 32 * (REC_WARPS + 3);
    static constexpr uint32_t TMEM_COLS = NVB == 1 ? 256 : 512;
    static constexpr int MIN_CTAS = (NVB == 1 && STAGES == 1) ? 2 : 1;
    // one input stage
    static constexpr uint32_t AKQ = 0;                     // per kb: [kg 8K | qg 8K]
    static constexpr uint32_t W = AKQ + 2 * KB * 8192;     // w per kb [64 tok][64 d]
    static constexpr uint32_t DO = W + KB * 8192;          // do per V block [64 tok][64 v]
    static constexpr uint32_t DVIN = DO + NVB * 8192;      // dv_in per V block
    static constexpr uint32_t GD = DVIN + NVB * 8192;      // gd fp32 [K]
    static constexpr uint32_t STAGE = GD + 1024;
    static constexpr uint32_t TX_BYTES = (3 * KB + 2 * NVB) * 8192 + K * 4;
    // persistent
    static constexpr uint32_t HS = STAGES * STAGE;         // dh bf16 per V block [K rows][64 v], MN-major
    static constexpr uint32_t HS_BLOCK = KB * 8192;
    // I_64 (bf16, or fp16 with fp16 gradients), K-major SW128 [64 rows][64 tok]:
    // the A operand that puts dv_in into the accumulator; its rows 64-127 read
    // the next 8 KB (VP), which land in unused TMEM lanes
    static constexpr uint32_t IDN = HS + NVB * HS_BLOCK;
    static constexpr uint32_t VP = IDN + 8192;             // dv2 bf16 per V block [64 tok][64 v], MN-major
    static constexpr uint32_t BYTES = VP + NVB * 8192;
};

template <int STAGES>
struct BwdBars {
    uint64_t full[STAGES], empty[STAGES];
    uint64_t h_ready, dv_full, vp_ready, upd_full;
    uint64_t hs_free, vp_free;  // the store warp's copies have read the dh / dv2 operand copies
    uint64_t do_ready[STAGES];  // fp16 do converted to bf16 in the stage
    uint32_t tmem_slot;
    int abort_flag;
};

template <int KB, int NVB, int STAGES, bool F16>
__global__ void __launch_bounds__(BwdCfg<KB, NVB, STAGES>::THREADS, BwdCfg<KB, NVB, STAGES>::MIN_CTAS)
    kda_bwd_dh_kernel(const __grid_constant__ CUtensorMap tm_kg, const __grid_constant__ CUtensorMap tm_qg,
                      const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_dvin, const __grid_constant__ CUtensorMap tm_dv2,
                      const __grid_constant__ CUtensorMap tm_dhck, const void* __restrict__ dht,
                      uint16_t* __restrict__ dhck, uint16_t* __restrict__ dv2, void* __restrict__ dh0,
                      uint8_t* __restrict__ ws, const WsLayout L, const float scale, const int N, const int H,
                      const int V, const int mode, const int flags) {
    using S = BwdCfg<KB, NVB, STAGES>;
    constexpr int K = S::K;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align_smem_1024(smem_raw);
    __shared__ BwdBars<STAGES> B;

    // Column space: V columns of dh (output mode) or, in map mode, K + V
    // columns [P | Q] of a segment's affine map dh_in = P dh_out + Q.
    const bool map_mode = mode == kScanModeMap;
    const int NCOL = map_mode ? K + V : V;
    const int NT = NCOL / S::BV;
    const int vt = blockIdx.x % NT;
    const int h = (blockIdx.x / NT) % H;
    const int s = blockIdx.x / (NT * H);
    const int v0 = vt * S::BV;
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    if (*reinterpret_cast<volatile int32_t*>(status) != 0) return;
    const SeqInfo si = reinterpret_cast<const SeqInfo*>(ws + L.seq_info)[s];
    const int tiles = si.tiles;
    // segments of the sequence (all of it when the scan is not segmented);
    // the map pass covers segments 1.., the output pass segments 0..
    const int nseg = tiles == 0 ? 0 : (tiles - 1) / L.seg_len + 1;
    const int seg = map_mode ? (int)blockIdx.y + 1 : (int)blockIdx.y;
    if (seg > 0 && seg >= nseg) return;
    const int c_lo = seg * L.seg_len;                 // this CTA's chunks [c_lo, c_hi),
    const int c_hi = min(tiles, c_lo + L.seg_len);    // walked newest first
    const int nit = c_hi > c_lo ? c_hi - c_lo : 0;
    // the segment maps and entry states are stored newest segment first
    const int rev = nseg - 1 - seg;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);
    constexpr bool f16 = F16;  // do, dv_in, dv2 are fp16

    if (tid == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&B.full[i], 1);
            mbar_init(&B.empty[i], 1 + S::REC_WARPS);
        }
        mbar_init(&B.h_ready, S::REC_WARPS);
        mbar_init(&B.dv_full, 1);
        mbar_init(&B.vp_ready, 2 * NVB);
        mbar_init(&B.upd_full, 1);
        mbar_init(&B.hs_free, 1);
        mbar_init(&B.vp_free, 1);
        for (int i = 0; i < STAGES; ++i) mbar_init(&B.do_ready[i], 1);
        B.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == S::MMA_WARP) {
        tmem_alloc(&B.tmem_slot, S::TMEM_COLS);
        tmem_relinquish();
    }
    for (int e = tid; e < 8192 / 16; e += S::THREADS) {
        const int row = e >> 3, ch = e & 7;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        // 1.0 at column row, i.e. in 16-byte chunk (row / 8) ^ (row & 7)
        if (ch == ((row >> 3) ^ (row & 7))) {
            const uint32_t one = F16 ? 0x3C00u : 0x3F80u;
            uint32_t wv[4] = {0u, 0u, 0u, 0u};
            wv[(row & 7) >> 1] = (row & 1) ? one << 16 : one;
            x = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        *reinterpret_cast<uint4*>(sm + S::IDN + e * 16) = x;
    }
    fence_proxy_async_smem();
    if (map_mode) {
        // P columns see do = dv_in = 0: their tiles stay zero in every stage
        // (the TMA never writes them)
        for (int st = 0; st < STAGES; ++st)
#pragma unroll
            for (int b = 0; b < NVB; ++b)
                if (v0 + b * 64 < K)
                    for (int e = tid; e < 1024; e += S::THREADS) {
                        reinterpret_cast<uint4*>(sm + st * S::STAGE + S::DO + b * 8192)[e] = make_uint4(0u, 0u, 0u, 0u);
                        reinterpret_cast<uint4*>(sm + st * S::STAGE + S::DVIN + b * 8192)[e] = make_uint4(0u, 0u, 0u, 0u);
                    }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = B.tmem_slot;
    // TMEM columns: DV, WD, then QD for even and odd chunks
    const uint32_t t_dv = tmem, t_wd = tmem + S::BV, t_qd = tmem + 2 * S::BV;
    volatile int* abort_flag = &B.abort_flag;
    bool timed_out = false;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
        timed_out = true;
        *abort_flag = 1;
        return false;
    };

    if (warp < S::REC_WARPS) {
        // ================= recurrence warps =================
        const int quad = warp & 3, vb = warp >> 2;
        const int r = quad * 32 + lane;  // dh row (key dim) and, for r < 64, token row
        const bool has_row = r < K;      // warp-uniform
        const int col = v0 + vb * 64;
        float dh[64];
        // start: map mode [I | 0]; the newest segment dht (or 0); any other
        // segment the entry state the combine step chained for it
        const float* src_row = nullptr;
        const bool dht_row = !map_mode && has_row && (seg == nseg - 1 || nseg == 0) && dht != nullptr;
        if (!map_mode && has_row) {
            if (seg == nseg - 1 || nseg == 0) {
                if (dht != nullptr && !(flags & kBwdStateBF16))
                    src_row = static_cast<const float*>(dht) + (((int64_t)s * H + h) * K + r) * V + col;
            } else {
                src_row = reinterpret_cast<const float*>(ws + L.hin) + ((((int64_t)rev * N + s) * H + h) * K + r) * V + col;
            }
        }
        if (dht_row && (flags & kBwdStateBF16)) {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(dht) +
                                                              (((int64_t)s * H + h) * K + r) * V + col);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 x = src[j];
                const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    dh[8 * j + 2 * t] = bf_lo(xw[t]);
                    dh[8 * j + 2 * t + 1] = bf_hi(xw[t]);
                }
            }
        } else if (src_row != nullptr) {
            const float4* src = reinterpret_cast<const float4*>(src_row);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float4 x = src[j];
                dh[4 * j] = x.x;
                dh[4 * j + 1] = x.y;
                dh[4 * j + 2] = x.z;
                dh[4 * j + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) dh[j] = (map_mode && has_row && r == col + j) ? 1.f : 0.f;
        }
        uint8_t* hs = sm + S::HS + vb * S::HS_BLOCK;
        uint8_t* vp = sm + S::VP + vb * 8192;
        for (int it = 0; it < nit && !*abort_flag; ++it) {
            const int c = c_hi - 1 - it;
            const int st = it % STAGES;
            const uint32_t sp = (it / STAGES) & 1;
            uint8_t* stage = sm + st * S::STAGE;
            // MMA operand: dh before this chunk's update, bf16 (once the store
            // warp's copy of the previous chunk's checkpoint has read it)
            if (it > 0 && !wait(&B.hs_free, (it - 1) & 1)) break;
            if (has_row) {
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 x = make_uint4(pack_bf16x2(dh[8 * cc], dh[8 * cc + 1]), pack_bf16x2(dh[8 * cc + 2], dh[8 * cc + 3]),
                                               pack_bf16x2(dh[8 * cc + 4], dh[8 * cc + 5]), pack_bf16x2(dh[8 * cc + 6], dh[8 * cc + 7]));
                    *reinterpret_cast<uint4*>(hs + r * 128 + ((cc ^ (r & 7)) << 4)) = x;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.h_ready);
            // (the checkpoint leaves from this copy through the store warp)
            if (!wait(&B.full[st], sp)) break;
            if (quad < 2) {
                // dv2[r, :] = DV[r, :] + dv_in[r, :], rows past the sequence end = 0
                if (!wait(&B.dv_full, it & 1)) break;
                if (it > 0 && !wait(&B.vp_free, (it - 1) & 1)) break;
                tc_fence_after();
                const int valid = min(64, si.len - c * 64);
                const bool row_ok = r < valid;
                uint4* gdst = reinterpret_cast<uint4*>(dv2 + ((int64_t)(si.bos + c * 64 + r) * H + h) * V + col);
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    float dv[16];  // kg@dh + dv_in, summed by the MMAs
                    tmem_ld16(t_dv + (uint32_t)(vb * 64) + ((uint32_t)(quad * 32) << 16) + c0, dv);
                    tmem_ld_wait();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int cc = (c0 >> 3) + hh;
                        const uint32_t off = r * 128 + ((cc ^ (r & 7)) << 4);
                        const float* x = dv + 8 * hh;
                        uint32_t pw[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) pw[t] = row_ok ? pack_bf16x2(x[2 * t], x[2 * t + 1]) : 0u;
                        if constexpr (F16) {
                            // fp16 dv2 leaves from the fp32 values (the operand copy is bf16)
                            if (row_ok && !map_mode)
                                gdst[cc] = make_uint4(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]),
                                                      pack_f16x2(x[4], x[5]), pack_f16x2(x[6], x[7]));
                        }
                        *reinterpret_cast<uint4*>(vp + off) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&B.vp_ready);
                // dv2 rows of a tail chunk leave after the hand-off, read back from
                // the operand copy (full chunks leave through the store warp)
                if (row_ok && !map_mode && !f16 && valid < 64) {
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) gdst[cc] = *reinterpret_cast<const uint4*>(vp + r * 128 + ((cc ^ (r & 7)) << 4));
                }
            }
            const float decay = has_row ? ex2(reinterpret_cast<const float*>(stage + S::GD)[r]) : 0.f;
            if (!wait(&B.upd_full, it & 1)) break;
            tc_fence_after();
            if (has_row) {
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 8) {
                    float qd[8], wd[8];
                    tmem_ld8(t_qd + (uint32_t)((it & 1) * S::BV + vb * 64) + ((uint32_t)(quad * 32) << 16) + c0, qd);
                    tmem_ld8(t_wd + (uint32_t)(vb * 64) + ((uint32_t)(quad * 32) << 16) + c0, wd);
                    tmem_ld_wait();
#pragma unroll
                    for (int t = 0; t < 8; ++t) dh[c0 + t] = fmaf(decay, dh[c0 + t], fmaf(scale, qd[t], -wd[t]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.empty[st]);
        }
        if (map_mode && has_row && !timed_out && !*abort_flag) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(ws + L.pq) +
                                                    ((((int64_t)rev * N + s) * H + h) * K + r) * (K + V) + col);
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[j] = make_float4(dh[4 * j], dh[4 * j + 1], dh[4 * j + 2], dh[4 * j + 3]);
        } else if (!map_mode && seg == 0 && dh0 != nullptr && has_row && !timed_out && !*abort_flag) {
            const int64_t hrow = (((int64_t)s * H + h) * K + r) * V + col;  // element offset of this row
            if (flags & kBwdStateBF16) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(dh0) + hrow);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    dst[j] = make_uint4(pack_bf16x2(dh[8 * j], dh[8 * j + 1]), pack_bf16x2(dh[8 * j + 2], dh[8 * j + 3]),
                                        pack_bf16x2(dh[8 * j + 4], dh[8 * j + 5]), pack_bf16x2(dh[8 * j + 6], dh[8 * j + 7]));
            } else {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(dh0) + hrow);
#pragma unroll
                for (int j = 0; j < 16; ++j) dst[j] = make_float4(dh[4 * j], dh[4 * j + 1], dh[4 * j + 2], dh[4 * j + 3]);
            }
        }
    } else if (warp == S::TMA_WARP) {
        // ================= TMA producer =================
        // fp16 do: once a chunk's tiles have landed, the warp rewrites its do
        // tiles as bf16 in place (the qg^T @ do MMA takes bf16 operands)
        auto convert_do = [&](int j) {
            const int sj = j % STAGES;
            const bool ok = wait(&B.full[sj], (j / STAGES) & 1);
            __syncwarp();
            if (!ok) return;
            uint4* t = reinterpret_cast<uint4*>(sm + sj * S::STAGE + S::DO);
            for (int e = lane; e < NVB * 512; e += 32) {
                const int b = e >> 9;
                if (map_mode && v0 + b * 64 < K) continue;  // P columns: zero tiles
                const uint4 x = t[e];
                t[e] = make_uint4(pack_bf16x2(h_lo(x.x), h_hi(x.x)), pack_bf16x2(h_lo(x.y), h_hi(x.y)),
                                  pack_bf16x2(h_lo(x.z), h_hi(x.z)), pack_bf16x2(h_lo(x.w), h_hi(x.w)));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B.do_ready[sj]);
        };
        if (nit > 0 && (F16 || lane == 0)) {  // bf16: lane 0 alone; fp16: the warp also converts do
            if (lane == 0) {
                prefetch_tmap(&tm_kg);
                prefetch_tmap(&tm_qg);
                prefetch_tmap(&tm_w);
                prefetch_tmap(&tm_do);
                prefetch_tmap(&tm_dvin);
            }
            const float* gd = reinterpret_cast<const float*>(ws + L.gd);
            uint32_t tx = S::TX_BYTES;  // map mode: no do / dv_in for P columns
#pragma unroll
            for (int b = 0; b < NVB; ++b)
                if (map_mode && v0 + b * 64 < K) tx -= 2 * 8192;
            for (int it = 0; it < nit && !*abort_flag; ++it) {
                const int c = c_hi - 1 - it;
                const int st = it % STAGES;
                const uint32_t sp = (it / STAGES) & 1;
                bool issued = false;
                if (lane == 0 && wait(&B.empty[st], sp ^ 1)) {  // lane 0 issues the copies
                    issued = true;
                    uint8_t* stage = sm + st * S::STAGE;
                    const int64_t tile = (int64_t)(si.tile_base + c) * H + h;
                    const int row = (int)(tile * 64);
                    const int trow = si.bos + c * 64;
                    uint64_t* fb = &B.full[st];
                    mbar_arrive_expect_tx(fb, tx);
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb) {
                        tma_load_2d(stage + S::AKQ + kb * 16384, &tm_kg, fb, kb * 64, row);
                        tma_load_2d(stage + S::AKQ + kb * 16384 + 8192, &tm_qg, fb, kb * 64, row);
                        tma_load_2d(stage + S::W + kb * 8192, &tm_w, fb, kb * 64, row);
                    }
#pragma unroll
                    for (int vb = 0; vb < NVB; ++vb) {
                        const int cb = v0 + vb * 64, uc = map_mode ? cb - K : cb;  // column in the user tensors
                        if (uc < 0) continue;
                        tma_load_3d(stage + S::DO + vb * 8192, &tm_do, fb, uc, h, trow);
                        tma_load_3d(stage + S::DVIN + vb * 8192, &tm_dvin, fb, uc, h, trow);
                    }
                    bulk_load_1d(stage + S::GD, gd + tile * K, K * 4, fb);
                }
                if constexpr (F16) issued = __shfl_sync(0xffffffffu, issued, 0);
                if (!issued) break;
                if (f16 && it >= 1) convert_do(it - 1);
            }
            if (f16 && nit > 0 && !*abort_flag) convert_do(nit - 1);
        }
    } else if (warp == S::STORE_WARP) {
        // ================= stores through TMA =================
        // Per chunk: the checkpoint (dh before the update, the bf16 operand copy
        // in HS) and, for a full bf16 chunk, dv2 (the operand copy in VP) leave
        // by TMA stores; once their shared-memory reads are done, hs_free and
        // vp_free let the recurrence warps rewrite the copies.  Rows of a tail
        // chunk past the sequence end belong to the next sequence, so a tail's
        // dv2 rows are stored by the recurrence warps with a row mask.
        if (lane == 0 && nit > 0) {
            const bool ck = dhck != nullptr && !map_mode;
            if (ck) prefetch_tmap(&tm_dhck);
            if (!map_mode && !f16) prefetch_tmap(&tm_dv2);
            for (int it = 0; it < nit && !*abort_flag; ++it) {
                const int c = c_hi - 1 - it;
                if (!wait(&B.h_ready, it & 1)) break;
                if (ck) {
                    const int blk = (si.tile_base + c) * H + h;  // below 2^25: the host bounds chunks * H * 64
#pragma unroll
                    for (int vb = 0; vb < NVB; ++vb) tma_store_3d(&tm_dhck, sm + S::HS + vb * S::HS_BLOCK, v0 + vb * 64, 0, blk);
                }
                if (!wait(&B.vp_ready, it & 1)) break;
                if (!map_mode && !f16 && si.len - c * 64 >= 64) {
#pragma unroll
                    for (int vb = 0; vb < NVB; ++vb)
                        tma_store_3d(&tm_dv2, sm + S::VP + vb * 8192, v0 + vb * 64, h, si.bos + c * 64);
                }
                bulk_commit();
                bulk_wait_read0();
                mbar_arrive(&B.hs_free);
                mbar_arrive(&B.vp_free);
            }
            bulk_wait_read0();
        }
    } else if (warp == S::MMA_WARP) {
        // ================= tcgen05 issuer =================
        if (lane == 0) {
            constexpr uint32_t id_dv = idesc_bf16_f32(128, S::BV, 0, 1);  // A K-major, B (dh) MN-major
            constexpr uint32_t id_up = idesc_bf16_f32(128, S::BV, 1, 1);  // A (qg^T, w^T) MN-major
            // the dv_in term: fp16 operands with fp16 gradients
            constexpr uint32_t id_in = F16 ? idesc_f16_f32(128, S::BV, 0, 1) : idesc_bf16_f32(128, S::BV, 0, 1);
            for (int it = 0; it < nit && !*abort_flag; ++it) {
                const int st = it % STAGES;
                const uint32_t sp = (it / STAGES) & 1;
                const uint32_t stage = sbase + st * S::STAGE;
                if (!wait(&B.full[st], sp)) break;
                tc_fence_after();
                // DV = dv_in (the previous chunk's dv2 phase has read DV: its
                // vp_ready was waited on before this point)
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(t_dv, smem_desc(sbase + S::IDN + ks * 32, 16, 1024),
                             smem_desc(stage + S::DVIN + ks * 2048, 8192, 1024), id_in, ks > 0 ? 1u : 0u);
                // QD = qg^T @ do into this chunk's buffer (the update two chunks
                // back, which read it, finished before the last h_ready): the
                // qg blocks sit 16 KB apart (K = 64: the next 8 KB are unused rows)
                if (f16 && !wait(&B.do_ready[st], sp)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(t_qd + (uint32_t)((it & 1) * S::BV),
                             smem_desc(stage + S::AKQ + 8192 + ks * 2048, KB == 2 ? 16384 : 8192, 1024),
                             smem_desc(stage + S::DO + ks * 2048, 8192, 1024), id_up, ks > 0 ? 1u : 0u);
                if (!wait(&B.h_ready, it & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < K / 16; ++ks) {
                    const int kb = ks >> 2, kk = ks & 3;
                    mma_bf16(t_dv, smem_desc(stage + S::AKQ + kb * 16384 + kk * 32, 16, 1024),
                             smem_desc(sbase + S::HS + ks * 2048, S::HS_BLOCK, 1024), id_dv, 1u);
                }
                mma_commit(&B.dv_full);
                if (!wait(&B.vp_ready, it & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_bf16(t_wd, smem_desc(stage + S::W + ks * 2048, 8192, 1024),
                             smem_desc(sbase + S::VP + ks * 2048, 8192, 1024), id_up, ks > 0 ? 1u : 0u);
                mma_commit(&B.upd_full);
                mma_commit(&B.empty[st]);
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

template <int KB, int NVB, int STAGES, bool F16>
cudaError_t launch_bwd_f(const BwdArgs& a, int mode, cudaStream_t stream) {
    using S = BwdCfg<KB, NVB, STAGES>;
    const uint32_t smem = S::BYTES + 1024;
    auto kern = kda_bwd_dh_kernel<KB, NVB, STAGES, F16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int ncol = mode == kScanModeMap ? a.K + a.V : a.V;
    const int64_t ctas = (int64_t)a.N * a.H * (ncol / S::BV);
    const int segs = mode == kScanModeMap ? a.L.seg_count - 1 : a.L.seg_count;
    if (ctas <= 0 || segs <= 0) return cudaSuccess;
    const dim3 grid((unsigned)ctas, (unsigned)segs);
    kern<<<grid, S::THREADS, smem, stream>>>(a.tm_kg, a.tm_qg, a.tm_w, a.tm_do, a.tm_dvin, a.tm_dv2, a.tm_dhck,
                                             a.dht, a.dhck, a.dv2, a.dh0, a.ws, a.L, a.scale, a.N, a.H, a.V, mode,
                                             a.flags);
    return cudaGetLastError();
}

template <int KB, int NVB, int STAGES>
cudaError_t launch_bwd_t(const BwdArgs& a, int mode, cudaStream_t stream) {
    return (a.flags & kBwdF16) ? launch_bwd_f<KB, NVB, STAGES, true>(a, mode, stream)
                               : launch_bwd_f<KB, NVB, STAGES, false>(a, mode, stream);
}

template <int KB>
cudaError_t launch_bwd_k(const BwdArgs& a, int mode, cudaStream_t stream, int sms) {
    const int ncol = mode == kScanModeMap ? a.K + a.V : a.V;
    const int segs = mode == kScanModeMap ? a.L.seg_count - 1 : a.L.seg_count;
    const int64_t ctas64 = (int64_t)a.N * a.H * (ncol / 64) * segs;
    if (ctas64 <= sms) return launch_bwd_t<KB, 1, 2>(a, mode, stream);
    if (ncol % 128 == 0) return launch_bwd_t<KB, 2, 2>(a, mode, stream);
    return launch_bwd_t<KB, 1, 1>(a, mode, stream);
}

}  // namespace

cudaError_t launch_bwd_dh(const BwdArgs& a, cudaStream_t stream) {
    const int sms = device_sm_count();
    if (a.K != 128 && a.K != 64) return cudaErrorInvalidValue;
    auto run = [&](int mode) {
        return a.K == 128 ? launch_bwd_k<2>(a, mode, stream, sms) : launch_bwd_k<1>(a, mode, stream, sms);
    };
    if (a.L.seg_count > 1) {
        // segmented (the forward's plan): maps of every segment but the oldest,
        // chained newest first from dht, then all segments in parallel
        cudaError_t e = run(kScanModeMap);
        if (e != cudaSuccess) return e;
        e = launch_seg_combine(a.dht, a.ws, a.L, a.N, a.H, a.K, a.V, (a.flags & kBwdStateBF16) ? kScanStateBF16 : 0,
                               stream);
        if (e != cudaSuccess) return e;
    }
    return run(kScanModeOutput);
}

}  // namespace kda
