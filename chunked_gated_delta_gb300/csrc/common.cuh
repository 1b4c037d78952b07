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
    size_t status, seq_info, chunk_info, gd, qg, kg, w, u, aqk, total;
    int64_t max_chunks;
};

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
