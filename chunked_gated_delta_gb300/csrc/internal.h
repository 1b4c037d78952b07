// internal.h -- launchers shared between the C-ABI translation unit and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace kda {

struct IntraArgs {
    CUtensorMap tm_q, tm_k, tm_v, tm_g;      // user inputs, 3-D {dim, H, rows}
    CUtensorMap st_qg, st_w, st_u, st_aqk;   // workspace tiles (stores), 2-D {dim, tiles*64}
    const uint16_t* beta;                // bf16 bits [rows, H]
    uint8_t* ws;
    WsLayout L;
    int H, K, V;
    int64_t max_chunks;
};

struct ScanArgs {
    CUtensorMap tm_w, tm_qg, tm_kg, tm_u, tm_aqk;  // workspace tiles, 2-D {dim, tiles*64}
    const float* h0;  // [N, H, K, V] or null
    float* ht;        // [N, H, K, V] or null
    uint16_t* o;      // bf16 bits [rows, H, V]
    uint8_t* ws;
    WsLayout L;
    float scale;
    int N, H, K, V;
};

struct BwdArgs {
    CUtensorMap tm_kg, tm_qg, tm_w;  // workspace tiles, 2-D {dim, tiles*64}
    CUtensorMap tm_do, tm_dvin;      // user tensors, 3-D {V, H, rows}
    const float* dht;   // [N, H, K, V] or null
    uint16_t* dhck;     // bf16 [chunks, H, K, V] or null
    uint16_t* dv2;      // bf16 [rows, H, V]
    float* dh0;         // [N, H, K, V] or null
    uint8_t* ws;
    WsLayout L;
    float scale;
    int N, H, K, V;
};

cudaError_t launch_plan(const int32_t* cu_seqlens, int N, int B, int T, uint8_t* ws,
                        const WsLayout& L, cudaStream_t stream);
cudaError_t launch_intra(const IntraArgs& a, cudaStream_t stream);
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream);
cudaError_t launch_bwd_dh(const BwdArgs& a, cudaStream_t stream);

}  // namespace kda
