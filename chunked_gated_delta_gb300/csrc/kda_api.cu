// kda_api.cu -- the C ABI (include/kda.h): argument validation, workspace
// layout, TMA descriptor creation, the chunk planner kernel, and the launches
// of the intra-chunk and scan kernels on the caller's stream.
#include <algorithm>
#include <cstring>

#include "../../include/kda.h"
#include <mutex>

#include "internal.h"
#include "tensormap.h"

namespace kda {
namespace {

// ---------------------------------------------------------------- planner
// One CTA.  Validates cu_seqlens (0 = c_0 <= ... <= c_N = T), writes the
// per-sequence table {bos, len, tile_base, tiles} and the per-chunk table
// {row0, valid}.  tile_base is the exclusive prefix sum of ceil(len / 64),
// the layout of "KDA源码剖析之FlashKDA（下）" (its workspace index
// head * total_tiles + tile_base + t is kept here as (tile_base + t) * H + head,
// i.e. chunk-major, so that one chunk's heads are adjacent).
constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads)
    kda_plan_kernel(const int32_t* __restrict__ cu, int N, int B, int T, uint8_t* __restrict__ ws,
                    WsLayout L) {
    int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
    SeqInfo* seqs = reinterpret_cast<SeqInfo*>(ws + L.seq_info);
    ChunkInfo* chunks = reinterpret_cast<ChunkInfo*>(ws + L.chunk_info);
    __shared__ int64_t part[kPlanThreads];
    __shared__ int bad;
    const int tid = threadIdx.x;
    if (tid == 0) bad = 0;
    __syncthreads();
    const bool varlen = cu != nullptr;
    const int nseq = varlen ? N : B;
    const int per = (nseq + kPlanThreads - 1) / kPlanThreads;
    const int s0 = tid * per, s1 = min(nseq, s0 + per);
    int64_t local = 0;
    int my_bad = 0;
    if (varlen && tid == 0 && (cu[0] != 0 || cu[N] != T)) my_bad = 1;
    for (int s = s0; s < s1; ++s) {
        const int len = varlen ? cu[s + 1] - cu[s] : T;
        if (len < 0) my_bad = 1;
        local += len > 0 ? tiles_of(len, kChunk) : 0;
    }
    part[tid] = local;
    if (my_bad) atomicOr(&bad, 1);
    __syncthreads();
    // inclusive Hillis-Steele scan of the per-thread tile counts
    for (int off = 1; off < kPlanThreads; off <<= 1) {
        const int64_t x = tid >= off ? part[tid - off] : 0;
        __syncthreads();
        part[tid] += x;
        __syncthreads();
    }
    const int64_t total = part[kPlanThreads - 1];
    if (total > L.max_chunks) bad = 1;  // benign race: every writer stores 1
    __syncthreads();
    const bool ok = bad == 0;
    int64_t base = part[tid] - local;
    for (int s = s0; s < s1; ++s) {
        const int len = varlen ? cu[s + 1] - cu[s] : T;
        const int bos = varlen ? cu[s] : s * T;
        const int t = (ok && len > 0) ? tiles_of(len, kChunk) : 0;
        seqs[s] = SeqInfo{bos, ok ? len : 0, (int32_t)base, t};
        base += t;
    }
    __syncthreads();
    __threadfence_block();
    for (int64_t c = tid; c < L.max_chunks; c += kPlanThreads) {
        ChunkInfo ci{0, 0};
        if (ok && c < total) {
            int lo = 0, hi = nseq - 1;  // largest s with tile_base <= c
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (seqs[mid].tile_base <= c) lo = mid;
                else hi = mid - 1;
            }
            const SeqInfo q = seqs[lo];
            const int t = (int)(c - q.tile_base);
            ci.row0 = q.bos + t * kChunk;
            ci.valid = min(kChunk, q.len - t * kChunk);
        }
        chunks[c] = ci;
    }
    if (tid == 0) {
        status[0] = ok ? 0 : kStatusBadSeqlens;
        status[kStatusExactTiles] = 0;
    }
}

// ---------------------------------------------------------------- validation
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_varlen(const kda_dims* d) { return d->num_seqs > 0; }

kda_status check_dims(const kda_dims* d, bool varlen) {
    if (!d) return KDA_ERR_INVALID_ARG;
    if (d->T < 0 || d->H < 1 || d->B < 1 || d->num_seqs < 0) return KDA_ERR_INVALID_ARG;
    if (varlen && d->B != 1) return KDA_ERR_INVALID_ARG;
    if (d->K != 64 && d->K != 128) return KDA_ERR_UNSUPPORTED;
    if (d->V != 64 && d->V != 128) return KDA_ERR_UNSUPPORTED;
    const int64_t rows = (int64_t)d->B * d->T;
    if (rows > INT32_MAX / 2) return KDA_ERR_UNSUPPORTED;
    const int64_t nc = max_chunks(*d, varlen);
    if (nc * d->H * kChunk > INT32_MAX) return KDA_ERR_UNSUPPORTED;  // TMA coordinates are int32
    return KDA_OK;
}

kda_status check_ws(const kda_dims* d, bool varlen, void* ws, size_t bytes, WsLayout* L) {
    *L = ws_layout(*d, varlen);
    if (!ws || !aligned(ws, 256)) return KDA_ERR_WORKSPACE;
    if (bytes < L->total) return KDA_ERR_WORKSPACE;
    return KDA_OK;
}

bool map3(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* base, int inner, int H,
          int64_t rows, uint32_t box_inner, CUtensorMapSwizzle sw) {
    const uint64_t dims[3] = {(uint64_t)inner, (uint64_t)H, (uint64_t)rows};
    const uint64_t strides[2] = {(uint64_t)inner * esize, (uint64_t)inner * esize * H};
    const uint32_t box[3] = {box_inner, 1, (uint32_t)kChunk};
    return make_tensormap(m, dt, 3, base, dims, strides, box, sw);
}

bool check_opts(const kda_fwd_opts* op, const kda_dims* d) {
    if (op->plan != KDA_PLAN_AUTO && op->plan != KDA_PLAN_TWO_STAGE && op->plan != KDA_PLAN_FUSED) return false;
    if (op->io_dtype != KDA_IO_BF16 && op->io_dtype != KDA_IO_F16) return false;
    if (op->state_dtype != KDA_STATE_F32 && op->state_dtype != KDA_STATE_BF16) return false;
    if (op->beta_logits != 0 && op->beta_logits != 1) return false;
    if (op->qk_heads < 0) return false;
    if (op->qk_heads > 0 && (op->qk_heads > d->H || d->H % op->qk_heads != 0)) return false;
    return true;
}

bool map2(CUtensorMap* m, const void* base, int inner, int64_t rows) {
    const uint64_t dims[2] = {(uint64_t)inner, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)inner * 2};
    const uint32_t box[2] = {64, (uint32_t)kChunk};
    return make_tensormap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

size_t kda_fwd_workspace_size(const kda_dims* dims) {
    if (!dims) return 0;
    const bool varlen = is_varlen(dims);
    if (check_dims(dims, varlen) != KDA_OK) return 0;
    return ws_layout(*dims, varlen).total;
}

kda_status kda_workspace_layout(const kda_dims* dims, kda_ws_layout* out) {
    if (!dims || !out) return KDA_ERR_INVALID_ARG;
    const bool varlen = is_varlen(dims);
    kda_status st = check_dims(dims, varlen);
    if (st != KDA_OK) return st;
    const WsLayout L = ws_layout(*dims, varlen);
    out->status = L.status;
    out->seq_info = L.seq_info;
    out->chunk_info = L.chunk_info;
    out->gd = L.gd;
    out->qg = L.qg;
    out->kg = L.kg;
    out->w = L.w;
    out->u = L.u;
    out->aqk = L.aqk;
    out->total = L.total;
    out->max_chunks = (int32_t)L.max_chunks;
    out->chunk = kChunk;
    out->seg_count = L.seg_count;
    out->seg_len = L.seg_len;
    out->pq = L.pq;
    out->hin = L.hin;
    out->stage_count = L.stage_count;
    out->stage_len = L.stage_len;
    return KDA_OK;
}

int32_t kda_chunk_table(const int32_t* cu_seqlens, int32_t num_seqs, int32_t chunk,
                        int32_t* tile_base, int32_t* t_tiles) {
    if (!cu_seqlens || num_seqs < 0 || chunk < 1 || (num_seqs > 0 && (!tile_base || !t_tiles)))
        return -1;
    int64_t base = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t len = cu_seqlens[s + 1] - cu_seqlens[s];
        if (len < 0) return -1;
        tile_base[s] = (int32_t)base;
        t_tiles[s] = tiles_of(len, chunk);
        base += t_tiles[s];
        if (base > INT32_MAX) return -1;
    }
    return (int32_t)base;
}

namespace {
// Validation and TMA descriptors of the intra-chunk stage, with beta read as
// rows of beta_stride elements starting at column beta_head0 (the host
// pipeline passes a head group's view of beta).  Launches nothing.  *run is
// false when there is nothing to compute past the planner (no rows or no
// chunks); a->ws and a->L are set either way.
kda_status intra_setup(const void* q, const void* k, const void* v, const float* g, const void* beta,
                       int beta_stride, int beta_head0, const int32_t* cu_seqlens, const kda_dims* dims,
                       const kda_fwd_opts* opts, void* workspace, size_t workspace_bytes, IntraArgs* a,
                       bool* run) {
    if (!dims) return KDA_ERR_INVALID_ARG;
    kda_fwd_opts op{};
    if (opts) op = *opts;
    if (!check_opts(&op, dims)) return KDA_ERR_INVALID_ARG;
    const bool varlen = is_varlen(dims);
    if (varlen != (cu_seqlens != nullptr)) return KDA_ERR_INVALID_ARG;
    kda_status st = check_dims(dims, varlen);
    if (st != KDA_OK) return st;
    WsLayout L;
    st = check_ws(dims, varlen, workspace, workspace_bytes, &L);
    if (st != KDA_OK) return st;
    const int64_t rows = (int64_t)dims->B * dims->T;
    if (varlen && !aligned(cu_seqlens, 4)) return KDA_ERR_ALIGNMENT;
    if (rows > 0) {
        if (!q || !k || !v || !g || !beta) return KDA_ERR_INVALID_ARG;
        if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) || !aligned(beta, 2))
            return KDA_ERR_ALIGNMENT;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    *a = IntraArgs{};
    a->ws = ws;
    a->L = L;
    *run = rows > 0 && L.max_chunks > 0;
    if (!*run) return KDA_OK;
    const CUtensorMapDataType io =
        op.io_dtype == KDA_IO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int hqk = op.qk_heads > 0 ? op.qk_heads : dims->H;
    bool ok = map3(&a->tm_q, io, 2, q, dims->K, hqk, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && map3(&a->tm_k, io, 2, k, dims->K, hqk, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && map3(&a->tm_v, io, 2, v, dims->V, dims->H, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    const int64_t trows = L.max_chunks * dims->H * kChunk;
    ok = ok && map2(&a->st_qg, ws + L.qg, dims->K, trows);
    ok = ok && map2(&a->st_w, ws + L.w, dims->K, trows);
    ok = ok && map2(&a->st_u, ws + L.u, dims->V, trows);
    if (!ok) return KDA_ERR_CUDA;
    a->g = g;
    a->beta = static_cast<const uint16_t*>(beta);
    a->H = dims->H;
    a->K = dims->K;
    a->V = dims->V;
    a->max_chunks = L.max_chunks;
    a->f16 = op.io_dtype == KDA_IO_F16;
    a->flags = op.beta_logits ? kIntraBetaLogits : 0;
    a->group = dims->H / hqk;
    a->beta_stride = beta_stride;
    a->beta_head0 = beta_head0;
    a->after_planner = 1;  // every caller launches the planner, then this kernel, on one stream
    return KDA_OK;
}

// The planner: validates cu_seqlens, builds the tables, resets the status word.
kda_status plan(const int32_t* cu_seqlens, const kda_dims* dims, const IntraArgs& a, cudaStream_t s) {
    const int N = is_varlen(dims) ? dims->num_seqs : dims->B;
    kda_plan_kernel<<<1, kPlanThreads, 0, s>>>(cu_seqlens, N, dims->B, dims->T, a.ws, a.L);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status intra_impl(const void* q, const void* k, const void* v, const float* g, const void* beta,
                      int beta_stride, int beta_head0, const int32_t* cu_seqlens, const kda_dims* dims,
                      const kda_fwd_opts* opts, void* workspace, size_t workspace_bytes, void* stream) {
    IntraArgs a;
    bool run = false;
    kda_status st = intra_setup(q, k, v, g, beta, beta_stride, beta_head0, cu_seqlens, dims, opts, workspace,
                                workspace_bytes, &a, &run);
    if (st != KDA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = plan(cu_seqlens, dims, a, s);
    if (st != KDA_OK || !run) return st;
    return launch_intra(a, s) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Argument checks of the scan stage (no driver call).
kda_status scan_check(const void* h0, void* o, void* ht, const kda_dims* dims, const kda_fwd_opts* opts,
                      void* workspace, size_t workspace_bytes) {
    if (!dims) return KDA_ERR_INVALID_ARG;
    kda_fwd_opts op{};
    if (opts) op = *opts;
    if (!check_opts(&op, dims)) return KDA_ERR_INVALID_ARG;
    const bool varlen = is_varlen(dims);
    kda_status st = check_dims(dims, varlen);
    if (st != KDA_OK) return st;
    WsLayout L;
    st = check_ws(dims, varlen, workspace, workspace_bytes, &L);
    if (st != KDA_OK) return st;
    const int64_t rows = (int64_t)dims->B * dims->T;
    if (rows > 0 && !o) return KDA_ERR_INVALID_ARG;
    if ((o && !aligned(o, 16)) || (h0 && !aligned(h0, 16)) || (ht && !aligned(ht, 16)))
        return KDA_ERR_ALIGNMENT;
    return KDA_OK;
}

// Validation and TMA descriptors of the scan stage.  Launches nothing.
// with_o = false: the map pass of kda_fwd_state_map (no o, no tensor map of it).
kda_status scan_setup(float scale, const void* h0, void* o, void* ht, const kda_dims* dims,
                      const kda_fwd_opts* opts, void* workspace, size_t workspace_bytes, ScanArgs* a,
                      bool with_o = true) {
    kda_status st = with_o ? scan_check(h0, o, ht, dims, opts, workspace, workspace_bytes) : KDA_OK;
    if (st != KDA_OK) return st;
    kda_fwd_opts op{};
    if (opts) op = *opts;
    const bool varlen = is_varlen(dims);
    const WsLayout L = ws_layout(*dims, varlen);
    const int64_t rows = (int64_t)dims->B * dims->T;
    *a = ScanArgs{};
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int64_t trows = L.max_chunks * dims->H * kChunk;
    if (trows > 0) {
        bool ok = map2(&a->tm_w, ws + L.w, dims->K, trows);
        ok = ok && map2(&a->tm_qg, ws + L.qg, dims->K, trows);
        ok = ok && map2(&a->tm_kg, ws + L.kg, dims->K, trows);
        ok = ok && map2(&a->tm_u, ws + L.u, dims->V, trows);
        ok = ok && map2(&a->tm_aqk, ws + L.aqk, kChunk, trows);
        if (rows > 0 && with_o) {  // o [rows, H, V]: a box is 32 token rows of one head's 64 columns
            const uint64_t odims[3] = {(uint64_t)dims->V, (uint64_t)dims->H, (uint64_t)rows};
            const uint64_t ostr[2] = {(uint64_t)dims->V * 2, (uint64_t)dims->V * 2 * dims->H};
            const uint32_t obox[3] = {64, 1, 32};
            ok = ok && make_tensormap(&a->tm_o,
                                      op.io_dtype == KDA_IO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                      3, o, odims, ostr, obox, CU_TENSOR_MAP_SWIZZLE_128B);
        }
        if (!ok) return KDA_ERR_CUDA;
    }
    a->h0 = h0;
    a->ht = ht;
    a->o = static_cast<uint16_t*>(o);
    a->ws = ws;
    a->L = L;
    a->scale = scale;
    a->N = varlen ? dims->num_seqs : dims->B;
    a->H = dims->H;
    a->K = dims->K;
    a->V = dims->V;
    a->flags = (op.io_dtype == KDA_IO_F16 ? kScanOutF16 : 0) | (op.state_dtype == KDA_STATE_BF16 ? kScanStateBF16 : 0);
    return KDA_OK;
}

// Streams and events of the staged forward, created once per device: the
// intra-chunk kernels of the chunk ranges run on `intra`, the scans on `scan`
// (the highest stream priority, so a range's scan CTAs are placed before the
// next range's intra CTAs when both are ready).
struct StageRes {
    bool ready = false;
    cudaStream_t intra = nullptr, scan = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, ev_intra[2] = {}, ev_scan[2] = {};
};
std::mutex g_stage_mutex;
StageRes g_stage[64];

StageRes* stage_res() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    StageRes& r = g_stage[dev];
    if (r.ready) return &r;
    int least = 0, greatest = 0;
    bool ok = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess;
    ok = ok && r.intra == nullptr && cudaStreamCreateWithFlags(&r.intra, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaStreamCreateWithPriority(&r.scan, cudaStreamNonBlocking, greatest) == cudaSuccess;
    cudaEvent_t* evs[] = {&r.start, &r.done, &r.ev_intra[0], &r.ev_intra[1], &r.ev_scan[0], &r.ev_scan[1]};
    for (cudaEvent_t* e : evs) ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    r.ready = ok;
    return ok ? &r : nullptr;
}

// The chunk ranges of the staged forward (one sequence, L.stage_count > 1).
// Range j's intra kernel waits for range j - 2's scan (so at most one range of
// intra work runs ahead and the scan finds its SMs free), range j's scan for
// range j's intra kernel and, by stream order, range j - 1's scan.  Forked
// from and joined back to the caller's stream s.
kda_status run_stages(const IntraArgs& ia, const ScanArgs& sa, cudaStream_t s) {
    std::unique_lock<std::mutex> lock(g_stage_mutex);
    StageRes* R = stage_res();
    if (!R) {  // no library streams: the same work in order on the caller's stream
        if (launch_intra(ia, s) != cudaSuccess || launch_scan(sa, s) != cudaSuccess) return KDA_ERR_CUDA;
        return KDA_OK;
    }
    if (cudaEventRecord(R->start, s) != cudaSuccess || cudaStreamWaitEvent(R->intra, R->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(R->scan, R->start, 0) != cudaSuccess)
        return KDA_ERR_CUDA;
    const WsLayout& L = ia.L;
    const int64_t H = ia.H;
    bool ok = true;
    for (int j = 0; j < L.stage_count && ok; ++j) {
        // range j's intra kernel sees the workspace from chunk c0 on: the same
        // kernel, its tile index counted from the range's first chunk
        const int64_t c0 = (int64_t)j * L.stage_len;
        const int64_t c1 = std::min<int64_t>(c0 + L.stage_len, L.max_chunks);
        IntraArgs aj = ia;
        aj.after_planner = 0;  // follows event waits on the library's intra stream
        aj.max_chunks = c1 - c0;
        aj.L.chunk_info += (size_t)c0 * sizeof(ChunkInfo);
        aj.L.gd += (size_t)(c0 * H) * ia.K * sizeof(float);
        aj.L.kg += (size_t)(c0 * H) * kChunk * ia.K * 2;
        aj.L.aqk += (size_t)(c0 * H) * kChunk * kChunk * 2;
        const int64_t rows = aj.max_chunks * H * kChunk;
        ok = map2(&aj.st_qg, ia.ws + L.qg + (size_t)(c0 * H) * kChunk * ia.K * 2, ia.K, rows) &&
             map2(&aj.st_w, ia.ws + L.w + (size_t)(c0 * H) * kChunk * ia.K * 2, ia.K, rows) &&
             map2(&aj.st_u, ia.ws + L.u + (size_t)(c0 * H) * kChunk * ia.V * 2, ia.V, rows);
        ok = ok && (j < 2 || cudaStreamWaitEvent(R->intra, R->ev_scan[j & 1], 0) == cudaSuccess) &&
             launch_intra(aj, R->intra) == cudaSuccess && cudaEventRecord(R->ev_intra[j & 1], R->intra) == cudaSuccess &&
             cudaStreamWaitEvent(R->scan, R->ev_intra[j & 1], 0) == cudaSuccess &&
             launch_scan_stage(sa, j, R->scan) == cudaSuccess &&
             cudaEventRecord(R->ev_scan[j & 1], R->scan) == cudaSuccess;
    }
    // join (also after a failed launch, so the caller's stream never runs ahead of enqueued work)
    const bool joined =
        cudaEventRecord(R->done, R->scan) == cudaSuccess && cudaStreamWaitEvent(s, R->done, 0) == cudaSuccess;
    return ok && joined ? KDA_OK : KDA_ERR_CUDA;
}
}  // namespace

}  // extern "C"

kda_status kda::check_scan_args(const void* h0, void* o, void* ht, const kda_dims* dims, void* workspace,
                                size_t workspace_bytes) {
    return scan_check(h0, o, ht, dims, nullptr, workspace, workspace_bytes);
}

extern "C" {

kda_status kda_fwd_intra_ex(const void* q, const void* k, const void* v, const float* g,
                            const void* beta, const int32_t* cu_seqlens, const kda_dims* dims,
                            const kda_fwd_opts* opts, void* workspace, size_t workspace_bytes,
                            void* stream) {
    return intra_impl(q, k, v, g, beta, dims ? dims->H : 0, 0, cu_seqlens, dims, opts, workspace,
                      workspace_bytes, stream);
}

kda_status kda_fwd_intra(const void* q, const void* k, const void* v, const float* g,
                         const void* beta, const int32_t* cu_seqlens, const kda_dims* dims,
                         void* workspace, size_t workspace_bytes, void* stream) {
    return kda_fwd_intra_ex(q, k, v, g, beta, cu_seqlens, dims, nullptr, workspace, workspace_bytes, stream);
}

kda_status kda_fwd_scan_ex(float scale, const void* h0, void* o, void* ht, const kda_dims* dims,
                           const kda_fwd_opts* opts, void* workspace, size_t workspace_bytes,
                           void* stream) {
    ScanArgs a;
    kda_status st = scan_setup(scale, h0, o, ht, dims, opts, workspace, workspace_bytes, &a);
    if (st != KDA_OK) return st;
    if (launch_scan(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_fwd_scan(float scale, const float* h0, void* o, float* ht, const kda_dims* dims,
                        void* workspace, size_t workspace_bytes, void* stream) {
    return kda_fwd_scan_ex(scale, h0, o, ht, dims, nullptr, workspace, workspace_bytes, stream);
}

kda_status kda_bwd_dh_ex(float scale, const void* do_, const void* dv_in, const void* dht, void* dhck, void* dv2,
                         void* dh0, const kda_dims* dims, const kda_fwd_opts* opts, void* workspace,
                         size_t workspace_bytes, void* stream) {
    if (!dims) return KDA_ERR_INVALID_ARG;
    kda_fwd_opts op{};
    if (opts) op = *opts;
    if (op.io_dtype != KDA_IO_BF16 && op.io_dtype != KDA_IO_F16) return KDA_ERR_INVALID_ARG;
    if (op.state_dtype != KDA_STATE_F32 && op.state_dtype != KDA_STATE_BF16) return KDA_ERR_INVALID_ARG;
    const CUtensorMapDataType io =
        op.io_dtype == KDA_IO_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const bool varlen = is_varlen(dims);
    kda_status st = check_dims(dims, varlen);
    if (st != KDA_OK) return st;
    WsLayout L;
    st = check_ws(dims, varlen, workspace, workspace_bytes, &L);
    if (st != KDA_OK) return st;
    const int64_t rows = (int64_t)dims->B * dims->T;
    if (rows > 0 && (!do_ || !dv_in || !dv2)) return KDA_ERR_INVALID_ARG;
    if ((do_ && !aligned(do_, 16)) || (dv_in && !aligned(dv_in, 16)) || (dv2 && !aligned(dv2, 16)) ||
        (dht && !aligned(dht, 16)) || (dhck && !aligned(dhck, 16)) || (dh0 && !aligned(dh0, 16)))
        return KDA_ERR_ALIGNMENT;
    BwdArgs a{};
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int64_t trows = L.max_chunks * dims->H * kChunk;
    if (trows > 0 && rows > 0) {
        bool ok = map2(&a.tm_kg, ws + L.kg, dims->K, trows);
        ok = ok && map2(&a.tm_qg, ws + L.qg, dims->K, trows);
        ok = ok && map2(&a.tm_w, ws + L.w, dims->K, trows);
        ok = ok && map3(&a.tm_do, io, 2, do_, dims->V, dims->H, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B);
        ok = ok && map3(&a.tm_dvin, io, 2, dv_in, dims->V, dims->H, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B);
        ok = ok && map3(&a.tm_dv2, io, 2, dv2, dims->V, dims->H, rows, 64, CU_TENSOR_MAP_SWIZZLE_128B);
        if (dhck) {  // [chunks * H] blocks of K rows x V columns; a box is one block's 64 columns
            const uint64_t cdims[3] = {(uint64_t)dims->V, (uint64_t)dims->K, (uint64_t)(L.max_chunks * dims->H)};
            const uint64_t cstr[2] = {(uint64_t)dims->V * 2, (uint64_t)dims->K * dims->V * 2};
            const uint32_t cbox[3] = {64, (uint32_t)dims->K, 1};
            ok = ok && make_tensormap(&a.tm_dhck, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, dhck, cdims, cstr, cbox,
                                      CU_TENSOR_MAP_SWIZZLE_128B);
        }
        if (!ok) return KDA_ERR_CUDA;
    }
    a.dht = dht;
    a.dhck = static_cast<uint16_t*>(dhck);
    a.dv2 = static_cast<uint16_t*>(dv2);
    a.dh0 = dh0;
    a.ws = ws;
    a.L = L;
    a.scale = scale;
    a.N = varlen ? dims->num_seqs : dims->B;
    a.H = dims->H;
    a.K = dims->K;
    a.V = dims->V;
    a.flags = (op.io_dtype == KDA_IO_F16 ? kBwdF16 : 0) | (op.state_dtype == KDA_STATE_BF16 ? kBwdStateBF16 : 0);
    if (launch_bwd_dh(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_bwd_dh(float scale, const void* do_, const void* dv_in, const float* dht, void* dhck, void* dv2,
                      float* dh0, const kda_dims* dims, void* workspace, size_t workspace_bytes, void* stream) {
    return kda_bwd_dh_ex(scale, do_, dv_in, dht, dhck, dv2, dh0, dims, nullptr, workspace, workspace_bytes, stream);
}

kda_status kda_fwd_ex(const void* q, const void* k, const void* v, const float* g, const void* beta,
                      float scale, const void* h0, const int32_t* cu_seqlens, void* o, void* ht,
                      const kda_dims* dims, const kda_fwd_opts* opts, void* workspace,
                      size_t workspace_bytes, void* stream) {
    // every argument of both stages is checked before any driver call or launch
    kda_status st = scan_check(h0, o, ht, dims, opts, workspace, workspace_bytes);
    if (st != KDA_OK) return st;
    kda_fwd_opts op{};
    if (opts) op = *opts;
    // the single-pass kernel runs on request only (it leaves no intermediates in
    // the workspace for kda_bwd_dh) and takes the default interface only
    const bool fused = op.plan == KDA_PLAN_FUSED;
    if (fused && (op.io_dtype != KDA_IO_BF16 || op.state_dtype != KDA_STATE_F32 || op.beta_logits != 0 ||
                  (op.qk_heads != 0 && op.qk_heads != dims->H)))
        return KDA_ERR_UNSUPPORTED;
    IntraArgs ia;
    bool run = false;
    st = intra_setup(q, k, v, g, beta, dims ? dims->H : 0, 0, cu_seqlens, dims, opts, workspace,
                                workspace_bytes, &ia, &run);
    if (st != KDA_OK) return st;
    if (fused) {
        FusedArgs fa{};
        fa.tm_q = ia.tm_q;
        fa.tm_k = ia.tm_k;
        fa.tm_v = ia.tm_v;
        fa.g = g;
        fa.beta = static_cast<const uint16_t*>(beta);
        fa.h0 = static_cast<const float*>(h0);
        fa.ht = static_cast<float*>(ht);
        fa.o = static_cast<uint16_t*>(o);
        fa.ws = ia.ws;
        fa.L = ia.L;
        fa.scale = scale;
        fa.N = is_varlen(dims) ? dims->num_seqs : dims->B;
        fa.H = dims->H;
        fa.K = dims->K;
        fa.V = dims->V;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        st = plan(cu_seqlens, dims, ia, s);
        if (st != KDA_OK) return st;
        return launch_fused(fa, s) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
    }
    ScanArgs sa;
    st = scan_setup(scale, h0, o, ht, dims, opts, workspace, workspace_bytes, &sa);
    if (st != KDA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = plan(cu_seqlens, dims, ia, s);
    if (st != KDA_OK) return st;
    if (run && ia.L.stage_count > 1) return run_stages(ia, sa, s);
    if (run && launch_intra(ia, s) != cudaSuccess) return KDA_ERR_CUDA;
    return launch_scan(sa, s) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_fwd_state_map(const void* q, const void* k, const void* v, const float* g, const void* beta,
                             const int32_t* cu_seqlens, float* pq, const kda_dims* dims, void* workspace,
                             size_t workspace_bytes, void* stream) {
    // every argument is checked before any driver call or launch
    if (!dims) return KDA_ERR_INVALID_ARG;
    kda_status st = check_dims(dims, is_varlen(dims));
    if (st != KDA_OK) return st;
    const int64_t N = is_varlen(dims) ? dims->num_seqs : dims->B;
    if (N * dims->H > 0 && !pq) return KDA_ERR_INVALID_ARG;
    if (pq && !aligned(pq, 16)) return KDA_ERR_ALIGNMENT;
    IntraArgs ia;
    bool run = false;
    st = intra_setup(q, k, v, g, beta, dims->H, 0, cu_seqlens, dims, nullptr, workspace, workspace_bytes, &ia, &run);
    if (st != KDA_OK) return st;
    ScanArgs sa;
    st = scan_setup(1.0f, nullptr, nullptr, pq, dims, nullptr, workspace, workspace_bytes, &sa, false);
    if (st != KDA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    st = plan(cu_seqlens, dims, ia, s);
    if (st != KDA_OK) return st;
    if (run && launch_intra(ia, s) != cudaSuccess) return KDA_ERR_CUDA;
    return launch_scan_map_out(sa, s) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_chain_states(const float* pq, const float* h0, float* h_in, int32_t ranges, int32_t num_seqs,
                            int32_t H, int32_t K, int32_t V, void* stream) {
    if (ranges < 1 || num_seqs < 0 || H < 1) return KDA_ERR_INVALID_ARG;
    if ((K != 64 && K != 128) || (V != 64 && V != 128)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return KDA_OK;
    if (!pq || !h_in) return KDA_ERR_INVALID_ARG;
    if (!aligned(pq, 16) || !aligned(h_in, 16) || (h0 && !aligned(h0, 16))) return KDA_ERR_ALIGNMENT;
    return launch_chain_states(pq, h0, h_in, ranges, num_seqs, H, K, V, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

kda_status kda_fwd(const void* q, const void* k, const void* v, const float* g, const void* beta,
                   float scale, const float* h0, const int32_t* cu_seqlens, void* o, float* ht,
                   const kda_dims* dims, void* workspace, size_t workspace_bytes, void* stream) {
    return kda_fwd_ex(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, dims, nullptr, workspace, workspace_bytes,
                      stream);
}

namespace {
// kda_fwd_host as a head-group pipeline: the value heads are cut into
// `pieces` groups; group p's inputs go host -> device on a copy stream while
// group p-1 computes on the caller's stream and group p-2's outputs go device
// -> host on a second copy stream (the link is full duplex), with two arena
// slots for the groups in flight.  Heads are independent, so each group is a
// problem of its own (its rows are strided 2-D copies of the host tensors);
// beta, one element per head, is copied whole and read with its full stride.
// Two groups: every group runs the full serial scan over all chunks with
// fewer heads, so more groups add compute (measured on the headline problem:
// 8.73 ms in one piece, 7.88 ms in two, 8.27 in four, 8.70 in eight, against
// 6.4 ms for the input copies alone).
constexpr int64_t kPipeMinRows = 4096;  // smaller problems: one piece

int host_pieces(const kda_dims* d) {
    if ((int64_t)d->B * d->T < kPipeMinRows || d->H % 2 != 0) return 1;
    return 2;
}

struct HostArena {
    int pieces, hp, slots;
    size_t q, k, v, g, beta, h0, o, ht, slot_bytes;  // offsets inside a slot
    size_t slot0, cu, ws, ws_bytes, total;
    kda_dims pd;  // one head group's dims
};
HostArena host_arena(const kda_dims* d) {
    const bool varlen = is_varlen(d);
    const size_t rows = (size_t)d->B * d->T;
    const size_t N = varlen ? (size_t)d->num_seqs : (size_t)d->B;
    HostArena A{};
    A.pieces = host_pieces(d);
    A.hp = d->H / A.pieces;
    A.slots = A.pieces > 1 ? 2 : 1;
    A.pd = *d;
    A.pd.H = A.hp;
    const size_t hp = A.hp;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 1024);
        return at;
    };
    A.q = take(rows * hp * d->K * 2);
    A.k = take(rows * hp * d->K * 2);
    A.v = take(rows * hp * d->V * 2);
    A.g = take(rows * hp * d->K * 4);
    A.beta = take(rows * d->H * 2);
    A.h0 = take(N * hp * d->K * d->V * 4);
    A.o = take(rows * hp * d->V * 2);
    A.ht = take(N * hp * d->K * d->V * 4);
    A.slot_bytes = off;
    off = 0;
    A.slot0 = take(A.slot_bytes * A.slots);
    A.cu = take((N + 1) * 4);
    A.ws_bytes = ws_layout(A.pd, varlen).total;
    A.ws = take(A.ws_bytes);
    A.total = off;
    return A;
}

// Streams and events of the pipeline, created once per device.
struct PipeRes {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, done = nullptr, ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
};
std::mutex g_pipe_mutex;
PipeRes g_pipe[64];

PipeRes* pipe_res() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    PipeRes& r = g_pipe[dev];
    if (r.ready) return &r;
    bool ok = cudaStreamCreateWithFlags(&r.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&r.out, cudaStreamNonBlocking) == cudaSuccess;
    cudaEvent_t* evs[] = {&r.start, &r.done, &r.ev_in[0], &r.ev_in[1], &r.ev_comp[0], &r.ev_comp[1],
                          &r.ev_out[0], &r.ev_out[1]};
    for (cudaEvent_t* e : evs) ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    r.ready = ok;
    return ok ? &r : nullptr;
}

// Fixed-length problems run kda_fwd_host as a pipeline over time slices: the
// tokens are cut into `slices` ranges of whole 64-token chunks; slice j's
// inputs (every sequence's rows of the range, one strided copy per tensor) go
// host -> device on a copy stream while slice j - 1 computes on the caller's
// stream and slice j - 2's outputs go device -> host on a second copy stream,
// with two arena slots.  Slice j is kda_fwd on the sub-problem [B, T_j] whose
// initial state is slice j - 1's final state (fp32, kept in the arena): the
// chunks and the per-chunk arithmetic are those of one call over all T tokens,
// so the results are the same bits.  Unlike head groups, every slice runs a
// fraction of the serial scan, and only the first slice's copies and the last
// slice's compute and output copies stay exposed.
constexpr int kSliceMax = 8;

bool use_slices(const kda_dims* d) {
    return !is_varlen(d) && (int64_t)d->B * d->T >= kPipeMinRows && d->T >= 2 * kChunk;
}

struct SliceArena {
    int slices, ts;  // slice count, tokens per slice (a multiple of 64; the last may be shorter)
    size_t q, k, v, g, beta, o, slot_bytes;  // offsets inside a slot
    size_t slot0, h0, state, ws, ws_bytes, total;
};
SliceArena slice_arena(const kda_dims* d) {
    SliceArena A{};
    const int64_t nt = ((int64_t)d->T + kChunk - 1) / kChunk;
    const int64_t per = (nt + kSliceMax - 1) / kSliceMax;  // chunks per slice
    A.ts = (int)(per * kChunk);
    A.slices = (int)((nt + per - 1) / per);
    const size_t rows = (size_t)d->B * A.ts, B = (size_t)d->B, H = (size_t)d->H, K = (size_t)d->K,
                 V = (size_t)d->V;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 1024);
        return at;
    };
    A.q = take(rows * H * K * 2);
    A.k = take(rows * H * K * 2);
    A.v = take(rows * H * V * 2);
    A.g = take(rows * H * K * 4);
    A.beta = take(rows * H * 2);
    A.o = take(rows * H * V * 2);
    A.slot_bytes = off;
    off = 0;
    A.slot0 = take(A.slot_bytes * 2);
    A.h0 = take(B * H * K * V * 4);
    A.state = take(2 * B * H * K * V * 4);  // two fp32 states, slice j writes state[j & 1]
    kda_dims sd = *d;
    sd.T = A.ts;  // the largest slice (workspace size grows with T)
    A.ws_bytes = ws_layout(sd, false).total;
    A.ws = take(A.ws_bytes);
    A.total = off;
    return A;
}

// rows x width bytes, source rows `src_pitch` apart, packed at dst (or the reverse)
cudaError_t copy_rows(void* dst, size_t dst_pitch, const void* src, size_t src_pitch, size_t width, size_t rows,
                      cudaMemcpyKind kind, cudaStream_t s) {
    if (rows == 0 || width == 0) return cudaSuccess;
    if (dst_pitch == width && src_pitch == width) return cudaMemcpyAsync(dst, src, width * rows, kind, s);
    return cudaMemcpy2DAsync(dst, dst_pitch, src, src_pitch, width, rows, kind, s);
}

// Tokens [t0, t0 + tj) of every one of B sequences: host [B, T, tok] <-> device
// [B, tj, tok] packed (tok = bytes per token).  One strided copy, or one copy
// per sequence when the host pitch is 512 MiB or more (2-D copies take
// pitches below that size here).
cudaError_t copy_slice(uint8_t* dev, const uint8_t* host_in, uint8_t* host_out, size_t tok, size_t T, size_t t0,
                       size_t tj, size_t B, cudaStream_t s) {
    const size_t hp = T * tok, dp = tj * tok, w = tj * tok;
    const bool up = host_in != nullptr;
    if (hp < ((size_t)1 << 29)) {
        return up ? copy_rows(dev, dp, host_in + t0 * tok, hp, w, B, cudaMemcpyHostToDevice, s)
                  : copy_rows(host_out + t0 * tok, hp, dev, dp, w, B, cudaMemcpyDeviceToHost, s);
    }
    for (size_t b = 0; b < B; ++b) {
        const cudaError_t e = up ? cudaMemcpyAsync(dev + b * dp, host_in + b * hp + t0 * tok, w,
                                                   cudaMemcpyHostToDevice, s)
                                 : cudaMemcpyAsync(host_out + b * hp + t0 * tok, dev + b * dp, w,
                                                   cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

kda_status fwd_host_slices(const void* q, const void* k, const void* v, const float* g, const void* beta,
                           float scale, const float* h0, void* o, float* ht, const kda_dims* dims, uint8_t* base,
                           cudaStream_t s) {
    const SliceArena A = slice_arena(dims);
    const size_t B = dims->B, T = dims->T, H = dims->H, K = dims->K, V = dims->V;
    const size_t state_bytes = B * H * K * V * 4;
    std::unique_lock<std::mutex> lock(g_pipe_mutex);
    PipeRes* R = pipe_res();
    // without the pipeline's streams every step runs in order on the caller's stream
    cudaStream_t s_in = R ? R->in : s, s_out = R ? R->out : s;
    auto wait = [&](cudaStream_t who, cudaEvent_t e) { return !R || cudaStreamWaitEvent(who, e, 0) == cudaSuccess; };
    auto record = [&](cudaEvent_t e, cudaStream_t who) { return !R || cudaEventRecord(e, who) == cudaSuccess; };
    if (R && (!record(R->start, s) || !wait(s_in, R->start) || !wait(s_out, R->start))) return KDA_ERR_CUDA;
    bool ok = !h0 || cudaMemcpyAsync(base + A.h0, h0, state_bytes, cudaMemcpyHostToDevice, s_in) == cudaSuccess;
    kda_status st = ok ? KDA_OK : KDA_ERR_CUDA;
    for (int j = 0; j < A.slices && st == KDA_OK; ++j) {
        const int slot = j & 1;
        uint8_t* sb = base + A.slot0 + slot * A.slot_bytes;
        const size_t t0 = (size_t)j * A.ts, tj = std::min<size_t>(A.ts, T - t0);
        // inputs of slice j (slice j - 2 has computed and its outputs have left the slot)
        ok = !(R && j >= 2) || wait(s_in, R->ev_out[slot]);
        auto up = [&](size_t off, const void* src, size_t tok) {
            return copy_slice(sb + off, static_cast<const uint8_t*>(src), nullptr, tok, T, t0, tj, B, s_in) ==
                   cudaSuccess;
        };
        ok = ok && up(A.q, q, H * K * 2) && up(A.k, k, H * K * 2) && up(A.v, v, H * V * 2) && up(A.g, g, H * K * 4) &&
             up(A.beta, beta, H * 2);
        ok = ok && record(R ? R->ev_in[slot] : nullptr, s_in) && wait(s, R ? R->ev_in[slot] : nullptr);
        if (!ok) {
            st = KDA_ERR_CUDA;
            break;
        }
        // slice j from slice j - 1's final state (or h0)
        kda_dims sd = *dims;
        sd.T = (int32_t)tj;
        const float* h_in = j == 0 ? (h0 ? reinterpret_cast<const float*>(base + A.h0) : nullptr)
                                   : reinterpret_cast<const float*>(base + A.state + ((j - 1) & 1) * state_bytes);
        float* h_out = reinterpret_cast<float*>(base + A.state + (j & 1) * state_bytes);
        st = kda_fwd(sb + A.q, sb + A.k, sb + A.v, reinterpret_cast<const float*>(sb + A.g), sb + A.beta, scale, h_in,
                     nullptr, sb + A.o, h_out, &sd, base + A.ws, A.ws_bytes, s);
        if (st != KDA_OK) break;
        // outputs of slice j (and the final state after the last one)
        ok = record(R ? R->ev_comp[slot] : nullptr, s) && wait(s_out, R ? R->ev_comp[slot] : nullptr) &&
             copy_slice(sb + A.o, nullptr, static_cast<uint8_t*>(o), H * V * 2, T, t0, tj, B, s_out) == cudaSuccess;
        if (ok && ht && j == A.slices - 1)
            ok = cudaMemcpyAsync(ht, h_out, state_bytes, cudaMemcpyDeviceToHost, s_out) == cudaSuccess;
        ok = ok && record(R ? R->ev_out[slot] : nullptr, s_out);
        if (!ok) st = KDA_ERR_CUDA;
    }
    // the caller's stream completes after the last output copy (joined also after a failure)
    if (R && (!record(R->done, s_out) || !wait(s, R->done)) && st == KDA_OK) st = KDA_ERR_CUDA;
    return st;
}
}  // namespace

size_t kda_fwd_host_arena_size(const kda_dims* dims) {
    if (!dims || check_dims(dims, is_varlen(dims)) != KDA_OK) return 0;
    if (use_slices(dims)) return slice_arena(dims).total;
    return host_arena(dims).total;
}

kda_status kda_fwd_host(const void* q, const void* k, const void* v, const float* g,
                        const void* beta, float scale, const float* h0, const int32_t* cu_seqlens,
                        void* o, float* ht, const kda_dims* dims, void* arena, size_t arena_bytes,
                        void* stream) {
    if (!dims) return KDA_ERR_INVALID_ARG;
    const bool varlen = is_varlen(dims);
    if (varlen != (cu_seqlens != nullptr)) return KDA_ERR_INVALID_ARG;
    kda_status st = check_dims(dims, varlen);
    if (st != KDA_OK) return st;
    if (!arena || !aligned(arena, 256) || arena_bytes < kda_fwd_host_arena_size(dims)) return KDA_ERR_WORKSPACE;
    const size_t rows = (size_t)dims->B * dims->T;
    const size_t N = varlen ? (size_t)dims->num_seqs : (size_t)dims->B;
    if (rows > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* base = static_cast<uint8_t*>(arena);
    if (use_slices(dims)) return fwd_host_slices(q, k, v, g, beta, scale, h0, o, ht, dims, base, s);
    const HostArena A = host_arena(dims);
    const size_t H = dims->H, K = dims->K, V = dims->V, hp = A.hp;

    std::unique_lock<std::mutex> lock(g_pipe_mutex);
    PipeRes* R = A.pieces > 1 ? pipe_res() : nullptr;
    // without the pipeline's streams every step runs in order on the caller's stream
    cudaStream_t s_in = R ? R->in : s, s_out = R ? R->out : s;
    auto wait = [&](cudaStream_t who, cudaEvent_t e) { return !R || cudaStreamWaitEvent(who, e, 0) == cudaSuccess; };
    auto record = [&](cudaEvent_t e, cudaStream_t who) { return !R || cudaEventRecord(e, who) == cudaSuccess; };
    if (R && (!record(R->start, s) || !wait(s_in, R->start) || !wait(s_out, R->start))) return KDA_ERR_CUDA;
    if (cu_seqlens && cudaMemcpyAsync(base + A.cu, cu_seqlens, (N + 1) * 4, cudaMemcpyHostToDevice, s_in) != cudaSuccess)
        return KDA_ERR_CUDA;
    for (int p = 0; p < A.pieces; ++p) {
        const int slot = p % A.slots;
        uint8_t* sb = base + A.slot0 + slot * A.slot_bytes;
        const size_t h0c = (size_t)p * hp;  // first head of the group
        // inputs of group p (the slot's previous group must have finished computing)
        if (R && p >= 2 && !wait(s_in, R->ev_comp[slot])) return KDA_ERR_CUDA;
        const cudaMemcpyKind up = cudaMemcpyHostToDevice;
        bool ok = copy_rows(sb + A.q, hp * K * 2, static_cast<const uint8_t*>(q) + h0c * K * 2, H * K * 2, hp * K * 2,
                            rows, up, s_in) == cudaSuccess;
        ok = ok && copy_rows(sb + A.k, hp * K * 2, static_cast<const uint8_t*>(k) + h0c * K * 2, H * K * 2, hp * K * 2,
                             rows, up, s_in) == cudaSuccess;
        ok = ok && copy_rows(sb + A.v, hp * V * 2, static_cast<const uint8_t*>(v) + h0c * V * 2, H * V * 2, hp * V * 2,
                             rows, up, s_in) == cudaSuccess;
        ok = ok && copy_rows(sb + A.g, hp * K * 4, reinterpret_cast<const uint8_t*>(g) + h0c * K * 4, H * K * 4,
                             hp * K * 4, rows, up, s_in) == cudaSuccess;
        ok = ok && copy_rows(sb + A.beta, H * 2, beta, H * 2, H * 2, rows, up, s_in) == cudaSuccess;
        if (h0)
            ok = ok && copy_rows(sb + A.h0, hp * K * V * 4, reinterpret_cast<const uint8_t*>(h0) + h0c * K * V * 4,
                                 H * K * V * 4, hp * K * V * 4, N, up, s_in) == cudaSuccess;
        if (!ok || !record(R ? R->ev_in[slot] : nullptr, s_in)) return KDA_ERR_CUDA;
        // compute group p on the caller's stream (the slot's outputs of group p - 2 must be out)
        if (R && (!wait(s, R->ev_in[slot]) || (p >= 2 && !wait(s, R->ev_out[slot])))) return KDA_ERR_CUDA;
        st = intra_impl(sb + A.q, sb + A.k, sb + A.v, reinterpret_cast<const float*>(sb + A.g), sb + A.beta, (int)H,
                        (int)h0c, cu_seqlens ? reinterpret_cast<const int32_t*>(base + A.cu) : nullptr, &A.pd, nullptr,
                        base + A.ws, A.ws_bytes, stream);
        if (st != KDA_OK) return st;
        st = kda_fwd_scan(scale, h0 ? reinterpret_cast<const float*>(sb + A.h0) : nullptr, sb + A.o,
                          ht ? reinterpret_cast<float*>(sb + A.ht) : nullptr, &A.pd, base + A.ws, A.ws_bytes, stream);
        if (st != KDA_OK) return st;
        if (!record(R ? R->ev_comp[slot] : nullptr, s) || !wait(s_out, R ? R->ev_comp[slot] : nullptr))
            return KDA_ERR_CUDA;
        // outputs of group p
        const cudaMemcpyKind down = cudaMemcpyDeviceToHost;
        ok = copy_rows(static_cast<uint8_t*>(o) + h0c * V * 2, H * V * 2, sb + A.o, hp * V * 2, hp * V * 2, rows, down,
                       s_out) == cudaSuccess;
        if (ht)
            ok = ok && copy_rows(reinterpret_cast<uint8_t*>(ht) + h0c * K * V * 4, H * K * V * 4, sb + A.ht,
                                 hp * K * V * 4, hp * K * V * 4, N, down, s_out) == cudaSuccess;
        if (!ok || !record(R ? R->ev_out[slot] : nullptr, s_out)) return KDA_ERR_CUDA;
    }
    // the caller's stream completes after the last output copy
    if (R && (!record(R->done, s_out) || !wait(s, R->done))) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status kda_fwd_status(const void* workspace, void* stream) {
    if (!workspace) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (word & kStatusBadSeqlens) return KDA_ERR_BAD_SEQLENS;
    if (word & kStatusTimeout) return KDA_ERR_TIMEOUT;
    return KDA_OK;
}

const char* kda_status_string(kda_status s) {
    switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported shape (K and V must be 64 or 128)";
    case KDA_ERR_ALIGNMENT: return "tensor base pointer not 16-byte aligned";
    case KDA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case KDA_ERR_CUDA: return "CUDA launch or driver error";
    case KDA_ERR_TIMEOUT: return "a kernel pipeline wait timed out";
    case KDA_ERR_BAD_SEQLENS: return "cu_seqlens must satisfy 0 = c0 <= c1 <= ... <= cN = T";
    }
    return "unknown status";
}

}  // extern "C"
