/*
 * kda.h -- C ABI of the GB300 (sm_103a) chunked forward of Kimi Delta
 * Attention (KDA): the gated delta rule with a decay per key dimension,
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T,
 *     o_t = scale * S_t^T q_t,
 *
 * computed in chunks of 64 tokens by two CUDA kernels: an intra-chunk kernel
 * (in-chunk cumsum of g in log2 space, the gated Aqk, the beta-weighted
 * lower-triangular system and its inverse, w, u, qg, kg) and a fused
 * inter-chunk state-scan + output kernel.  The chunked form is the one stated
 * in kernel-fun "kda/_kernels/fwd_state.py" (module docstring); its host
 * wrapper kda_cute_fwd_call takes (qg, kg, w, u, aqk, g2, h0, scale), and this
 * ABI starts one step earlier, from the raw (q, k, v, g, beta).  Packed
 * variable-length batches follow "KDA源码剖析之FlashKDA（下）" (sequence
 * boundaries bos/eos from cu_seqlens, per-sequence initial/final state).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers, row-major and contiguous, owned
 *    by the caller; the library allocates no memory and keeps no pointer
 *    after a call returns.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Kernel
 *    work is enqueued asynchronously on it; the return value reports argument
 *    validation and launch errors only.  Errors found by the kernels (bad
 *    cu_seqlens contents, a pipeline wait that timed out) are recorded in the
 *    workspace and returned by kda_fwd_status().
 *  - Supported shapes: K in {64, 128}, V in {64, 128}, H >= 1, T >= 0.
 *    Other K/V return KDA_ERR_UNSUPPORTED.
 *  - Every tensor base pointer must be 16-byte aligned (KDA_ERR_ALIGNMENT).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, inconsistent dims        */
    KDA_ERR_UNSUPPORTED = 2,  /* K or V outside the supported set                       */
    KDA_ERR_ALIGNMENT = 3,    /* a tensor base pointer is not 16-byte aligned           */
    KDA_ERR_WORKSPACE = 4,    /* workspace NULL, misaligned or smaller than required    */
    KDA_ERR_CUDA = 5,         /* a CUDA launch / driver call failed                     */
    KDA_ERR_TIMEOUT = 6,      /* a kernel pipeline wait ran out of time (kda_fwd_status) */
    KDA_ERR_BAD_SEQLENS = 7   /* cu_seqlens not 0 = c0 <= c1 <= ... <= cN = T          */
} kda_status;

/*
 * Problem dimensions.
 *   Fixed length: num_seqs = 0 and cu_seqlens == NULL; B >= 1 sequences of T
 *   tokens each (N = B).
 *   Packed variable length: num_seqs = N >= 1 and cu_seqlens != NULL; B must
 *   be 1 and T is the total number of tokens.
 *   A mismatch between num_seqs and cu_seqlens is KDA_ERR_INVALID_ARG.
 * K = key (state row) dim, V = value dim, H = heads.
 */
typedef struct kda_dims {
    int32_t B, T, H, K, V;
    int32_t num_seqs;
} kda_dims;

/*
 * Bytes of device workspace kda_fwd needs for these dims (an upper bound that
 * does not depend on the cu_seqlens contents).  Returns 0 for invalid dims.
 * The workspace holds the intra-chunk intermediates qg, kg, w (bf16,
 * [chunks, H, 64, K]), u (bf16 [chunks, H, 64, V]), Aqk (bf16 [chunks, H, 64,
 * 64]), the per-chunk log2 decay gd (fp32 [chunks, H, K]), the chunk and
 * sequence tables, and a status word: about 1160 bytes per token-head at
 * K = V = 128.
 */
size_t kda_fwd_workspace_size(const kda_dims* dims);

/*
 * Full forward: kda_fwd_intra followed by kda_fwd_scan.  Every argument of
 * both stages is checked before anything is launched.  One long sequence whose
 * scan would leave most SMs idle (kda_workspace_layout's stage_count > 1, e.g.
 * 32 heads x 65536 tokens at K = V = 128) runs as stage_count chunk ranges:
 * the intra-chunk kernel of range j + 1 beside the scan of range j, on two
 * streams the library creates once per device, forked from `stream` after the
 * planner and joined back to it before the call returns (work enqueued on
 * `stream` later runs after the whole forward; the fork and join are events,
 * so the call can be captured in a CUDA graph).  Its results are bit for bit
 * those of kda_fwd_intra followed by kda_fwd_scan (the state passes from
 * range to range in fp32).  Calls of the staged path from several host threads
 * are serialised while they enqueue.  The first staged call on a device
 * creates the two streams and their events: make it before any stream capture.
 *
 *   q, k      bf16 [B, T, H, K]   queries / keys (the kernels do not normalise)
 *   v         bf16 [B, T, H, V]
 *   g         fp32 [B, T, H, K]   natural-log decay per key dimension (g <= 0
 *                                 expected; any finite value is accepted)
 *   beta      bf16 [B, T, H]      write strength, already activated (in (0,1))
 *   scale     multiplies o only (usually K^-0.5)
 *   h0        fp32 [N, H, K, V]   initial state per sequence, or NULL = zeros
 *   cu_seqlens int32 [N + 1]      device, packed sequence offsets, or NULL
 *   o         bf16 [B, T, H, V]   output (every valid token row is written)
 *   ht        fp32 [N, H, K, V]   final state per sequence, or NULL = not stored
 *   workspace device, >= kda_fwd_workspace_size(dims) bytes, 256-byte aligned;
 *             its contents on entry do not matter, and it must not be shared by
 *             calls that may run concurrently.
 * Returns KDA_OK once both kernels are enqueued.
 */
kda_status kda_fwd(const void* q, const void* k, const void* v, const float* g, const void* beta,
                   float scale, const float* h0, const int32_t* cu_seqlens, void* o, float* ht,
                   const kda_dims* dims, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Intra-chunk stage alone: resets the status word, builds the chunk tables
 * from cu_seqlens (validating them), and writes qg, kg, w, u, Aqk and gd for
 * every (chunk, head) into the workspace.  Same argument meanings as kda_fwd.
 */
kda_status kda_fwd_intra(const void* q, const void* k, const void* v, const float* g,
                         const void* beta, const int32_t* cu_seqlens, const kda_dims* dims,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Inter-chunk stage alone: the serial state scan and the output, reading the
 * intermediates that kda_fwd_intra left in `workspace` for the same dims.
 * One CTA per (sequence, head, V tile of 64 or 128 columns), serial over the
 * sequence's chunks (or over a segment of them, for few sequences x heads).
 */
kda_status kda_fwd_scan(float scale, const float* h0, void* o, float* ht, const kda_dims* dims,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Interface variants of the forward.  A zero-initialised kda_fwd_opts (or a
 * NULL pointer) gives exactly kda_fwd / kda_fwd_intra / kda_fwd_scan.
 *   io_dtype     KDA_IO_BF16: q, k, v, beta and o are bf16.
 *                KDA_IO_F16: they are fp16 (kernel-fun "kda/_kernels/fwd_state.py",
 *                host wrapper: the io dtype is bf16 or fp16).  The
 *                intermediates in the workspace stay bf16 either way.
 *   state_dtype  KDA_STATE_F32: h0 and ht are fp32.  KDA_STATE_BF16: they are
 *                bf16 (FlashKDA's StateFP32 = false, "KDA源码剖析之FlashKDA（下）",
 *                initial / final state sections); the state is still carried
 *                in fp32 on chip.
 *   beta_logits  0: beta is given in (0, 1).  1: beta holds logits and the
 *                kernel applies the sigmoid in fp32 (FlashKDA's in-kernel
 *                sigmoid of beta).
 *   qk_heads     heads of q and k; 0 means dims->H.  Otherwise dims->H (the
 *                value heads: v, g, beta, o, h0, ht) must be a multiple of it,
 *                and value head h reads q / k head h / (dims->H / qk_heads)
 *                (grouped value heads, the "HV" heads of fwd_state.py).  q and
 *                k are then [B, T, qk_heads, K].
 *   plan         KDA_PLAN_AUTO and KDA_PLAN_TWO_STAGE: the intra-chunk kernel
 *                over every chunk, then the scan (segmented or staged as
 *                kda_workspace_layout reports), leaving the intermediates in
 *                the workspace for kda_bwd_dh.  KDA_PLAN_FUSED: the single-pass
 *                kernel, one CTA per (sequence, head) running the intra-chunk
 *                stage and the scan chunk by chunk on chip, so only q, k, v, g,
 *                beta, h0 are read and o, ht written; the workspace then holds
 *                only the status word and the tables (no intermediates: a
 *                kda_bwd_dh needs a two-stage forward).  It takes the default
 *                interface only (bf16 I/O, fp32 state, activated beta, equal
 *                heads); other options with it return KDA_ERR_UNSUPPORTED.  A
 *                sequence's chunks run one after another on one SM, so it is
 *                slower than the two stages wherever those fill the GPU.
 *                kda_fwd_intra_ex / kda_fwd_scan_ex ignore it.
 * The ABI types: h0 / ht pointers are `const void*` / `void*` here because
 * their element type follows state_dtype.  Invalid option values return
 * KDA_ERR_INVALID_ARG.
 */
#define KDA_IO_BF16 0
#define KDA_IO_F16 1
#define KDA_STATE_F32 0
#define KDA_STATE_BF16 1
#define KDA_PLAN_AUTO 0
#define KDA_PLAN_TWO_STAGE 1
#define KDA_PLAN_FUSED 2
typedef struct kda_fwd_opts {
    int32_t io_dtype;
    int32_t state_dtype;
    int32_t beta_logits;
    int32_t qk_heads;
    int32_t plan;
} kda_fwd_opts;

kda_status kda_fwd_ex(const void* q, const void* k, const void* v, const float* g, const void* beta,
                      float scale, const void* h0, const int32_t* cu_seqlens, void* o, void* ht,
                      const kda_dims* dims, const kda_fwd_opts* opts, void* workspace,
                      size_t workspace_bytes, void* stream);
kda_status kda_fwd_intra_ex(const void* q, const void* k, const void* v, const float* g,
                            const void* beta, const int32_t* cu_seqlens, const kda_dims* dims,
                            const kda_fwd_opts* opts, void* workspace, size_t workspace_bytes,
                            void* stream);
kda_status kda_fwd_scan_ex(float scale, const void* h0, void* o, void* ht, const kda_dims* dims,
                           const kda_fwd_opts* opts, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * kda_bwd_dh with interface variants.  Of `opts` (NULL = kda_bwd_dh) the
 * reverse scan reads io_dtype and state_dtype:
 *   io_dtype     KDA_IO_F16: do, dv_in and dv2 are fp16 (do is rounded to bf16
 *                on chip for the qg^T @ do product, whose other operand is the
 *                bf16 qg; dv_in is added and dv2 written from fp32).
 *   state_dtype  KDA_STATE_BF16: dht and dh0 are bf16 (dh is carried in fp32).
 * The checkpoints dhck stay bf16.  beta_logits and qk_heads shaped the forward
 * whose workspace this call reads; they are ignored here.
 */
kda_status kda_bwd_dh_ex(float scale, const void* do_, const void* dv_in, const void* dht, void* dhck,
                         void* dv2, void* dh0, const kda_dims* dims, const kda_fwd_opts* opts,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Reverse state scan (the backward of the inter-chunk stage): the gradient of
 * the loss with respect to the recurrent state at every chunk boundary, after
 * kernel-fun "kda/_kernels/bwd_dhu.py".  With dh the gradient w.r.t. the state
 * after a chunk (starting from dht), chunks newest first:
 *     dhck[c] = dh;   dv2 = kg @ dh + dv_in;
 *     dh = exp2(G) * dh + scale * qg^T @ do - w^T @ dv2;   dh0 = final dh.
 * `workspace` must hold the intra-chunk intermediates of the same inputs and
 * dims (kda_fwd or kda_fwd_intra run before, workspace kept).
 *   do        bf16 [B, T, H, V]   gradient of the loss w.r.t. o
 *   dv_in     bf16 [B, T, H, V]   the chunk-local part of the v' gradient
 *                                 (the Aqk^T do term), from an earlier stage
 *   dht       fp32 [N, H, K, V]   gradient w.r.t. the final state, or NULL = 0
 *   dhck      bf16 [chunks, H, K, V] checkpoints in chunk-table order (chunks =
 *             kda_workspace_layout().max_chunks), or NULL = not stored
 *   dv2       bf16 [B, T, H, V]   gradient w.r.t. v' (valid rows written)
 *   dh0       fp32 [N, H, K, V]   gradient w.r.t. h0, or NULL = not stored
 * Asynchronous on `stream`; kernel-side errors via kda_fwd_status(workspace).
 */
kda_status kda_bwd_dh(float scale, const void* do_, const void* dv_in, const float* dht, void* dhck,
                      void* dv2, float* dh0, const kda_dims* dims, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * End-to-end forward from HOST buffers.  Copies q, k, v, g, beta (and h0,
 * cu_seqlens when given) from host memory into `arena`, runs kda_fwd there,
 * and copies o (and ht) back to host memory -- one cudaMemcpyAsync per tensor,
 * everything enqueued on `stream`.  The caller synchronises `stream` before
 * reading o / ht.  Host buffers should be page-locked (cudaHostAlloc or
 * cudaHostRegister) for the copies to overlap; pageable memory works but the
 * copies then block the calling thread.
 *   All tensor pointers here are HOST pointers with the shapes and dtypes of
 *   kda_fwd; cu_seqlens (host int32 [N+1]) may be NULL for fixed length.
 *   arena: device memory of at least kda_fwd_host_arena_size(dims) bytes,
 *   256-byte aligned, owned by the caller; it holds the device copies of the
 *   inputs and outputs and the workspace.
 *   Problems of 4096 rows (B * T) or more run as a pipeline: fixed-length
 *   ones over up to 8 time slices of whole 64-token chunks (each slice a
 *   kda_fwd over every sequence's rows of the slice, started from the
 *   previous slice's fp32 final state kept in the arena: the same bits as one
 *   kda_fwd), packed ones with an even head count over two head groups.  One
 *   piece's host -> device copies overlap the previous piece's kernels and
 *   the one before's device -> host copies, on two streams the library
 *   creates once per device (the call returns after enqueuing; `stream`
 *   completes when every copy has).  Calls are serialised internally.
 */
size_t kda_fwd_host_arena_size(const kda_dims* dims);
kda_status kda_fwd_host(const void* q, const void* k, const void* v, const float* g,
                        const void* beta, float scale, const float* h0, const int32_t* cu_seqlens,
                        void* o, float* ht, const kda_dims* dims, void* arena, size_t arena_bytes,
                        void* stream);

/*
 * Scratch capacity of kda_fwd_noalloc: 64 MiB.  A problem fits when
 * kda_fwd_workspace_size(dims) is at most this size: at K = V = 128 that is
 * T <= 1792 tokens with H = 32, or T <= 53248 with H = 1 (a long single
 * sequence adds the segment maps of the segmented scan to the workspace, so
 * the token-head capacity is lower there than for many heads).
 */
#define KDA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

/*
 * kda_fwd without a caller workspace (the method's pages have no counterpart:
 * this is an interface convenience of this library).  Meant for callers that
 * cannot call cudaMalloc: a plugin running inside a host framework whose
 * caching allocator owns all of the GPU's memory and must not be bypassed,
 * and latency-critical paths where cudaMalloc / cudaFree would implicitly
 * synchronise the device.  The workspace lives instead in a file-scope
 * device array of KDA_NOALLOC_SCRATCH_BYTES that every GPU which loads the
 * library holds until the process exits.  This call allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *   Arguments are those of kda_fwd minus the workspace; the caller still
 *   passes every input and output buffer.
 *   Problems whose workspace (kda_fwd_workspace_size) exceeds the scratch
 *   capacity return KDA_ERR_WORKSPACE before anything is enqueued.
 *   The first call on each device looks up the array's device address with
 *   that device current (cudaGetSymbolAddress) and caches it; make that first
 *   call before any stream capture begins.
 *   All calls share the one array, which keeps the previous call's contents.
 *   The forward needs nothing in it to start at zero (the planner rewrites
 *   the status word and tables on every call).  Calls that may overlap on the
 *   GPU (different streams, or different host threads) race on the array and
 *   must be serialised by the caller.
 *   Errors that only the kernels can detect (bad cu_seqlens contents, a
 *   timed-out pipeline wait) are recorded in the array's status word, which
 *   this call does not expose: a caller that needs them uses kda_fwd with a
 *   workspace and kda_fwd_status.
 */
kda_status kda_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                           const void* beta, float scale, const float* h0,
                           const int32_t* cu_seqlens, void* o, float* ht, const kda_dims* dims,
                           void* stream);

/*
 * Context-parallel forward (sequences split along T across ranks), the pass
 * before the exchange.  The state after a run of tokens is an affine function
 * of the state before it: with the chunked update h <- exp2(G) * h + kg^T v',
 * v' = u - w h, of kernel-fun "kda/_kernels/fwd_state.py" (module docstring),
 * each chunk maps h to M_c h + kg^T u with M_c = Diag(exp2 G) - kg^T w, so a
 * range of chunks maps h_in to
 *     h_out = P h_in + Q,   P = the product of its M_c,  Q = h_out from h_in = 0.
 * For every sequence s and head h of the local problem (this rank's tokens of
 * each sequence; same dims, q, k, v, g, beta and cu_seqlens conventions as
 * kda_fwd), this call runs the intra-chunk stage and a scan over the K + V
 * columns [P | Q], started from [I | 0], and stores
 *   pq        fp32 [N, H, K, K + V]   P in columns 0..K-1, Q in K..K+V-1
 *             (device, 16-byte aligned; N = num_seqs or B).
 * An empty sequence gives P = I, Q = 0.  The intra-chunk intermediates stay
 * in `workspace` (>= kda_fwd_workspace_size(dims) bytes), so that after the
 * exchange kda_fwd_scan(scale, h_in, o, ht, dims, workspace, ...) on the same
 * workspace produces this rank's o and its exit state from the entry state
 * h_in (kda_chain_states).  P and Q are computed with the same bf16 operand
 * copies as the scan itself, so the composed result matches a single call to
 * the forward's tolerances (not bit for bit).  Asynchronous on `stream`;
 * kernel-side errors via kda_fwd_status(workspace).
 */
kda_status kda_fwd_state_map(const void* q, const void* k, const void* v, const float* g,
                             const void* beta, const int32_t* cu_seqlens, float* pq,
                             const kda_dims* dims, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * Context-parallel forward, after the exchange: the entry state of each of
 * `ranges` consecutive token ranges, from their maps gathered in rank order,
 *     h_in[0] = h0,   h_in[r + 1] = P_r h_in[r] + Q_r   (fp32),
 *   pq    fp32 [ranges, num_seqs, H, K, K + V]  (kda_fwd_state_map of range r at pq[r])
 *   h0    fp32 [num_seqs, H, K, V] or NULL = zeros
 *   h_in  fp32 [ranges, num_seqs, H, K, V] out (the last range's map is not needed)
 * All device pointers, 16-byte aligned.  K, V in {64, 128}.  Asynchronous on
 * `stream`; returns KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED / KDA_ERR_ALIGNMENT
 * before any launch.
 */
kda_status kda_chain_states(const float* pq, const float* h0, float* h_in, int32_t ranges,
                            int32_t num_seqs, int32_t H, int32_t K, int32_t V, void* stream);

/*
 * Synchronises `stream` and returns the error the kernels recorded in
 * `workspace` during the last kda_fwd / kda_fwd_intra / kda_fwd_scan on it
 * (KDA_OK, KDA_ERR_BAD_SEQLENS or KDA_ERR_TIMEOUT), or KDA_ERR_CUDA if the
 * stream itself reports an error.
 */
kda_status kda_fwd_status(const void* workspace, void* stream);

/*
 * Self-check of the kernels' failure path: one CTA waits, for at most
 * limit_ns nanoseconds (1 .. 2e9), on a pipeline barrier that nothing
 * releases, using the same bounded wait as the forward's kernels, and records
 * the expiry in the int32 status word at status_word (device memory, 4-byte
 * aligned, owned by the caller).  Synchronises `stream` and returns what
 * kda_fwd_status would: KDA_ERR_TIMEOUT when the wait expired as designed.
 * The context stays usable afterwards (no trap, no fault).
 */
kda_status kda_selftest_wait_timeout(void* status_word, unsigned long long limit_ns, void* stream);

/* Static description of a status code.  Never NULL. */
const char* kda_status_string(kda_status s);

/*
 * Host helper (no GPU needed): the chunk table of a packed batch, the same
 * routine the device planner runs.  For each sequence s, t_tiles[s] =
 * ceil((cu[s+1] - cu[s]) / chunk) and tile_base[s] = sum of t_tiles over the
 * earlier sequences ("KDA源码剖析之FlashKDA（下）", the tile_base / t_tiles table
 * of its sequence-information section).  Returns the total number of tiles, or
 * -1 if the arguments are invalid (NULL, num_seqs < 0, chunk < 1, or
 * decreasing offsets).
 */
int32_t kda_chunk_table(const int32_t* cu_seqlens, int32_t num_seqs, int32_t chunk,
                        int32_t* tile_base, int32_t* t_tiles);

/*
 * Byte offsets of the regions inside the workspace, for inspection of the
 * intra-chunk intermediates (tests).  `max_chunks` is the chunk capacity
 * the layout was sized for.  Returns KDA_ERR_INVALID_ARG for invalid dims.
 * The status region holds the status word (int32 at `status`) and, in the
 * int32 after it, a diagnostic count of the (chunk, head) tiles of the last
 * forward whose gated sums took the exact per-element path (chunks whose
 * log2 decay span exceeds 96, where the factored gate products would
 * overflow); the planner resets both.
 */
typedef struct kda_ws_layout {
    size_t status, seq_info, chunk_info, gd, qg, kg, w, u, aqk, total;
    int32_t max_chunks;
    int32_t chunk;
    /* Segmented scan (few sequences x heads over long sequences): each
     * sequence's chunks are cut into seg_count segments of seg_len chunks;
     * pq holds every segment's affine state map [P | Q] (fp32 [seg_count, N,
     * H, K, K + V]) and hin the state entering each segment (fp32 [seg_count,
     * N, H, K, V]).  seg_count = 1: the plain scan (pq, hin empty). */
    int32_t seg_count;
    int32_t seg_len;
    size_t pq, hin;
    /* Staged forward (one sequence whose scan leaves most SMs idle): kda_fwd
     * runs the sequence as stage_count chunk ranges of stage_len chunks, the
     * intra-chunk kernel of range j + 1 beside the scan of range j, and the
     * scan passes its fp32 state from range to range through hin (fp32
     * [stage_count, 1, H, K, V]).  stage_count = 1: not staged. */
    int32_t stage_count;
    int32_t stage_len;
} kda_ws_layout;
kda_status kda_workspace_layout(const kda_dims* dims, kda_ws_layout* out);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
