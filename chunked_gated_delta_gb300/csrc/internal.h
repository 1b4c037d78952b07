// internal.h -- launchers shared between the C-ABI translation unit and the
// kernel translation units.  Not part of the public ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace kda {

// Launches kern after the previous kernel in stream with programmatic stream
// serialization: its CTAs may become resident while that kernel's last CTAs
// run.  Every kernel launched this way calls grid_dep_wait() before it reads
// or writes global memory, so it is correct after any earlier work; the
// staged forward's launches, which follow event waits on the library's
// streams, stay plain launches all the same.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

struct IntraArgs {
    CUtensorMap tm_q, tm_k, tm_v;            // user inputs, 3-D {dim, H, rows}
    CUtensorMap st_qg, st_w, st_u;           // workspace tiles (stores), 2-D {dim, tiles*64}
    const float* g;                      // fp32 [rows, H, K]
    const uint16_t* beta;                // bf16 or fp16 bits [rows, H]
    uint8_t* ws;
    WsLayout L;
    int H, K, V;                         // H = value heads
    int64_t max_chunks;
    int beta_stride;                     // elements between beta rows (H, or more for a head group)
    int beta_head0;                      // beta column of value head 0
    int f16;                             // q, k, v, beta are fp16 (else bf16)
    int flags;                           // kIntraBetaLogits
    int group;                           // value heads per q/k head
    int after_planner;                   // launched right after the planner in the same stream (PDL)
};

constexpr int kIntraBetaLogits = 1;
constexpr int kScanOutF16 = 1;     // o is fp16 (else bf16)
constexpr int kScanStateBF16 = 2;  // h0 / ht are bf16 (else fp32)
constexpr int kScanModeOutput = 0;  // the scan with its output o (and ht)
constexpr int kScanModeMap = 1;     // per-segment affine maps [P | Q] (segmented scan)
constexpr int kScanExitToHin = 4;   // output mode: a segment that ends before its sequence
                                    // stores its exit state as the next one's entry (hin)
constexpr int kScanMapOut = 8;      // map mode over each whole sequence: [P | Q] to ScanArgs::ht
                                    // as fp32 [N, H, K, K + V] (the affine map of the tokens given)

struct ScanArgs {
    CUtensorMap tm_w, tm_qg, tm_kg, tm_u, tm_aqk;  // workspace tiles, 2-D {dim, tiles*64}
    CUtensorMap tm_o;                              // o (stores), 3-D {V, H, rows}
    const void* h0;   // fp32 (or bf16) [N, H, K, V] or null
    void* ht;         // fp32 (or bf16) [N, H, K, V] or null
    uint16_t* o;      // bf16 (or fp16) bits [rows, H, V]
    uint8_t* ws;
    WsLayout L;
    float scale;
    int N, H, K, V;
    int flags;        // kScanOutF16 | kScanStateBF16
};

struct BwdArgs {
    CUtensorMap tm_kg, tm_qg, tm_w;  // workspace tiles, 2-D {dim, tiles*64}
    CUtensorMap tm_do, tm_dvin;      // user tensors, 3-D {V, H, rows}
    CUtensorMap tm_dv2;              // dv2 (stores), 3-D {V, H, rows}
    CUtensorMap tm_dhck;             // checkpoints (stores), 3-D {V, K, chunks * H}
    const void* dht;    // fp32 (or bf16) [N, H, K, V] or null
    uint16_t* dhck;     // bf16 [chunks, H, K, V] or null
    uint16_t* dv2;      // bf16 (or fp16) [rows, H, V]
    void* dh0;          // fp32 (or bf16) [N, H, K, V] or null
    uint8_t* ws;
    WsLayout L;
    float scale;
    int N, H, K, V;
    int flags;          // kBwdF16 | kBwdStateBF16
};

constexpr int kBwdF16 = 1;         // do, dv_in, dv2 are fp16 (else bf16)
constexpr int kBwdStateBF16 = 2;   // dht, dh0 are bf16 (else fp32)

struct FusedArgs {
    CUtensorMap tm_q, tm_k, tm_v;  // user inputs, 3-D {dim, H, rows}
    const float* g;                // fp32 [rows, H, K]
    const uint16_t* beta;          // bf16 bits [rows, H]
    const float* h0;               // fp32 [N, H, K, V] or null
    float* ht;                     // fp32 [N, H, K, V] or null
    uint16_t* o;                   // bf16 bits [rows, H, V]
    uint8_t* ws;                   // status word and sequence table (the planner's)
    WsLayout L;
    float scale;
    int N, H, K, V;
};

cudaError_t launch_plan(const int32_t* cu_seqlens, int N, int B, int T, uint8_t* ws,
                        const WsLayout& L, cudaStream_t stream);
cudaError_t launch_intra(const IntraArgs& a, cudaStream_t stream);
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t stream);
// The scan over chunk range `stage` of the staged forward (a.L.stage_count >
// 1): from h0 (stage 0) or the entry state in hin, writing o for the range and
// the exit state to hin (or ht after the last range).  The CTAs reserve shared
// memory beyond their own need, so no intra-chunk CTA shares an SM with them.
cudaError_t launch_scan_stage(const ScanArgs& a, int stage, cudaStream_t stream);
cudaError_t launch_bwd_dh(const BwdArgs& a, cudaStream_t stream);
// The single-pass forward: one CTA per (sequence, head), intra-chunk stage and
// scan chunk by chunk on chip (bf16 I/O, fp32 state, activated beta).
cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream);
// Argument checks of the scan stage of kda_fwd (h0, o, ht, dims, workspace),
// with no driver call and no launch: lets an entry point that runs the two
// stages itself report every argument error before it enqueues anything.
kda_status check_scan_args(const void* h0, void* o, void* ht, const kda_dims* dims, void* workspace,
                           size_t workspace_bytes);
// h_in[j+1] = P_j h_in[j] + Q_j over the segment maps in L.pq (h_in[0] = h0)
cudaError_t launch_seg_combine(const void* h0, uint8_t* ws, const WsLayout& L, int N, int H, int K, int V,
                               int flags, cudaStream_t stream);
// The affine map [P | Q] of every (sequence, head) over all of its chunks, from
// the intermediates in a.ws, stored to a.ht as fp32 [N, H, K, K + V].
cudaError_t launch_scan_map_out(const ScanArgs& a, cudaStream_t stream);
// h_in[0] = h0 (fp32, or zeros if null) and h_in[r+1] = P_r h_in[r] + Q_r for
// r < ranges - 1 over pq fp32 [ranges, N, H, K, K + V]; h_in fp32 [ranges, N, H, K, V].
cudaError_t launch_chain_states(const float* pq, const float* h0, float* h_in, int ranges, int N, int H, int K,
                                int V, cudaStream_t stream);

}  // namespace kda
