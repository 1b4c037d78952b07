// common.cuh -- constants, workspace layout and chunk planning shared by the
// host API and the two kernels.
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = 64;  // tokens per chunk (BT in the fwd_state.py kernel)

// Gate factorisation guard of the intra kernel.  The gated products
// q_i k_j exp2(g2_i - g2_j) are formed as (q_i exp2(g2_i)) . (k_j exp2(-g2_j));
// both factors stay finite in fp32/bf16 while the chunk's total log2 decay
// span -G is below this bound.  Chunks with a larger span take the exact
// per-element path instead.
constexpr float kSafeSpanLog2 = 96.0f;

// Pipeline waits give up after this long and record KDA_ERR_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Status word bits (workspace, int32).
constexpr int kStatusTimeout = 1;
constexpr int kStatusBadSeqlens = 2;
// Index of the int32 after the status word that counts the (chunk, head)
// tiles of the last forward whose gated sums took the exact per-element path
// (a diagnostic; the planner resets it with the status word).
constexpr int kStatusExactTiles = 1;

struct SeqInfo {
    int32_t bos, len, tile_base, tiles;
};
struct ChunkInfo {
    int32_t row0, valid;  // first packed token row, number of real rows (0 = unused slot)
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Upper bound on the number of 64-token chunks: sum_s ceil(L_s/64) <=
// floor((T + 63 N) / 64) for the packed case; B * ceil(T/64) for fixed length.
inline int64_t max_chunks(const kda_dims& d, bool varlen) {
    if (varlen) return ((int64_t)d.T + (int64_t)(kChunk - 1) * d.num_seqs) / kChunk;
    return (int64_t)d.B * (((int64_t)d.T + kChunk - 1) / kChunk);
}

struct WsLayout {
    size_t status, seq_info, chunk_info, gd, qg, kg, w, u, aqk, pq, hin, total;
    int64_t max_chunks;
    int32_t seg_count;    // segments per sequence of the segmented scan (1 = plain scan)
    int32_t seg_len;      // chunks per segment
    int32_t stage_count;  // chunk ranges of the staged forward (1 = not staged)
    int32_t stage_len;    // chunks per range
};

// Scan kernel shape for a launch of ctas64 64-column blocks over ncol
// columns per head (the same rule the launcher applies):
//   few blocks          -> 64-column CTAs, two-stage ring, one per SM
//   ncol % 128 == 0     -> 128-column CTAs, two-stage ring, one per SM
//   otherwise           -> 64-column CTAs, one stage, two per SM
// lat is the measured per-chunk latency of a CTA of that shape relative to
// the first (1.4 / 2.2 / 2.3 us per chunk at K = 128 on GB300).
struct ScanShape {
    int nvb, stages, per_sm;
    float lat;
};
inline ScanShape scan_shape(int64_t ctas64, int ncol, int sms) {
    if (ctas64 <= sms) return {1, 2, 1, 1.0f};
    if (ncol % 128 == 0) return {2, 2, 1, 1.6f};
    return {1, 1, 2, 1.7f};
}

// Segmented scan plan.  When the plain scan would leave most SMs idle (few
// sequences x heads over long sequences), each sequence's chunks are cut into
// seg_count segments of seg_len chunks: a map pass computes every segment's
// affine state map, a combine step chains them, and the output pass runs the
// segments in parallel.  The plan models each choice as chunks per CTA x
// relative per-chunk latency x waves (for an assumed kPlanSMs SMs), adds the
// fixed cost of the extra launches, and segments only for a gain of at least
// 10%; segments are never shorter than kSegMinChunks.  It depends on the dims
// only (so does the workspace size).
constexpr int kPlanSMs = 148;

// SMs of the current device (kPlanSMs if the query fails).
inline int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = kPlanSMs;
    return sms;
}
constexpr int kSegMinChunks = 16;
constexpr int kSegMaxCount = 64;

inline double scan_pass_cost(int64_t ctas64, int ncol) {
    if (ctas64 <= 0) return 0.0;
    const ScanShape sh = scan_shape(ctas64, ncol, kPlanSMs);
    const int64_t ctas = ctas64 / sh.nvb;
    const int64_t slots = (int64_t)kPlanSMs * sh.per_sm;
    return (double)sh.lat * (double)((ctas + slots - 1) / slots);
}

inline void seg_plan(const kda_dims& d, bool varlen, int32_t* count, int32_t* len) {
    const int64_t N = varlen ? d.num_seqs : d.B;
    const int64_t units = N * d.H * (d.V / 64);
    const int64_t maxt = (d.T + kChunk - 1) / kChunk;  // bound on any sequence's chunks
    int64_t best_S = 1, best_L = maxt > 0 ? maxt : 1;
    double best = (double)maxt * scan_pass_cost(units, d.V);
    const double plain = best;
    for (int64_t S = 2; S <= kSegMaxCount && units > 0 && S * kSegMinChunks <= maxt; ++S) {
        const int64_t L = (maxt + S - 1) / S;
        if ((maxt + L - 1) / L != S) continue;
        const double cost = (double)L * (scan_pass_cost((S - 1) * N * d.H * ((d.K + d.V) / 64), d.K + d.V) +
                                         scan_pass_cost(S * units, d.V)) +
                            8.0 + 2.0 * (double)(S - 1);
        if (cost < best) {
            best = cost;
            best_S = S;
            best_L = L;
        }
    }
    if (best_S > 1 && best > 0.9 * plain) best_S = 1;
    *count = (int32_t)best_S;
    *len = (int32_t)(best_S > 1 ? best_L : 0x7fffffff);
}

// Staged forward.  One sequence whose scan occupies at most half of the SMs
// (and that the segmented plan leaves unsegmented, e.g. 32 heads x 65536
// tokens at K = V = 128: 64 scan CTAs) is run as stage_count chunk ranges: the
// intra-chunk kernel of range j + 1 runs on the idle SMs while the scan walks
// range j, and the scan hands its fp32 state from range to range through the
// hin region.  Ranges are at least kStageMinChunks chunks long; at most
// kStageMax of them.  A function of the dims only (so is the workspace size).
constexpr int kStageMinChunks = 64;
constexpr int kStageMax = 8;

inline void stage_plan(const kda_dims& d, bool varlen, int32_t seg_count, int32_t* count, int32_t* len) {
    *count = 1;
    *len = 0x7fffffff;
    const int64_t N = varlen ? d.num_seqs : d.B;
    if (N != 1 || seg_count > 1) return;
    const int64_t ctas64 = (int64_t)d.H * (d.V / 64);  // the plain scan's 64-column blocks
    if (2 * ctas64 > kPlanSMs) return;
    const int64_t nt = ((int64_t)d.T + kChunk - 1) / kChunk;
    int64_t P = nt / kStageMinChunks;
    if (P > kStageMax) P = kStageMax;
    if (P < 2) return;
    const int64_t len_c = (nt + P - 1) / P;
    *count = (int32_t)((nt + len_c - 1) / len_c);
    *len = (int32_t)len_c;
}

inline WsLayout ws_layout(const kda_dims& d, bool varlen) {
    WsLayout L{};
    const int64_t N = varlen ? d.num_seqs : d.B;
    const int64_t NC = max_chunks(d, varlen);
    const size_t tiles = (size_t)NC * d.H;  // (chunk, head) tiles
    size_t off = 0;
    L.status = off;
    off = align_up(off + 256, 256);
    L.seq_info = off;
    off = align_up(off + sizeof(SeqInfo) * (size_t)(N > 0 ? N : 1), 256);
    L.chunk_info = off;
    off = align_up(off + sizeof(ChunkInfo) * (size_t)(NC > 0 ? NC : 1), 1024);
    L.gd = off;
    off = align_up(off + tiles * d.K * sizeof(float), 1024);
    L.qg = off;
    off = align_up(off + tiles * kChunk * d.K * 2, 1024);
    L.kg = off;
    off = align_up(off + tiles * kChunk * d.K * 2, 1024);
    L.w = off;
    off = align_up(off + tiles * kChunk * d.K * 2, 1024);
    L.u = off;
    off = align_up(off + tiles * kChunk * d.V * 2, 1024);
    L.aqk = off;
    off = align_up(off + tiles * kChunk * kChunk * 2, 1024);
    seg_plan(d, varlen, &L.seg_count, &L.seg_len);
    stage_plan(d, varlen, L.seg_count, &L.stage_count, &L.stage_len);
    const size_t seg_units = L.seg_count > 1 ? (size_t)L.seg_count * N * d.H : 0;
    const size_t stage_units = L.stage_count > 1 ? (size_t)L.stage_count * N * d.H : 0;
    L.pq = off;  // fp32 [S, N, H, K, K + V]: per segment [P | Q]
    off = align_up(off + seg_units * d.K * (d.K + d.V) * sizeof(float), 1024);
    L.hin = off;  // fp32 [S, N, H, K, V]: state entering each segment (or stage)
    off = align_up(off + (seg_units > stage_units ? seg_units : stage_units) * d.K * d.V * sizeof(float), 1024);
    L.total = off;
    L.max_chunks = NC;
    return L;
}

// Chunk planning shared by the host helper and the device planner:
// t_tiles = ceil(len / chunk); tile_base = exclusive prefix sum of t_tiles.
__host__ __device__ inline int32_t tiles_of(int32_t len, int32_t chunk) {
    return (len + chunk - 1) / chunk;
}

}  // namespace kda
