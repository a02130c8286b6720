/*
 * fa.h -- C ABI of the exact tiled attention forward for GB300 (sm_103a).
 *
 * The operation (sources are web pages, cited by page and section):
 *   "Flash Attention Memory Optimization Explained" (lzwjava.github.io),
 *   section "What is Flash Attention?": an exact scaled dot-product attention
 *   that never stores the T x T score matrix; the yelogs.com Flash
 *   Attention2/Triton tutorial, sections "核心 Kernel 實現" (tiled forward with
 *   online softmax that writes O and the per-row L), "Softmax 的在線計算"
 *   (running max m and normaliser l) and "2. 多查詢注意力（MQA）" (one KV head
 *   shared by all query heads).
 *
 *   For batch b, query head h, KV head hk = h / (Hq / Hkv), query row i:
 *     S[i][j] = scale * dot(Q[b][h][i][:], K[b][hk][j][:])
 *     keys j  = 0..T-1, or only j <= i when causal
 *     O[b][h][i][:] = sum_j softmax_j(S[i][:]) * V[b][hk][j][:]
 *     lse[b][h][i]  = m_i + ln(l_i)  (m_i = max_j S[i][j],
 *                                    l_i = sum_j exp(S[i][j] - m_i))
 *
 * Memory: every buffer is a DEVICE pointer owned by the caller; the library
 * never allocates, frees or keeps them.  Layouts are contiguous row-major:
 *   q   [B][Hq][T][d]    element type `dtype`
 *   k,v [B][Hkv][T][d]   element type `dtype`
 *   o   [B][Hq][T][d]    element type `dtype` (written; round-to-nearest-even)
 *   lse [B][Hq][T]       float32 (written; natural log)
 * o and lse must not overlap each other or the inputs.  All pointers must be
 * 16-byte aligned.
 *
 * Execution: fa_fwd validates its arguments on the host, then enqueues one
 * kernel on `stream` (a cudaStream_t; NULL = legacy default stream) and
 * returns without synchronising.  No host synchronisation and no device
 * allocation happen on this path.  The current CUDA device must be the one
 * that owns the buffers.
 *
 * Kernels by dtype (selection by the arithmetic type, not a fallback):
 *   FA_DTYPE_BF16, FA_DTYPE_F16: TMA-staged swizzled tiles, tcgen05 MMA into
 *                  tensor memory (bf16 or fp16 operands, fp32 accumulation),
 *                  warp-specialised softmax (d in {16, 32, 64, 128}); P is
 *                  rounded to the input type for the second product;
 *   FA_DTYPE_F32 : true-fp32 FFMA kernel on the CUDA cores (same d).
 * The pages name FP16 and BF16 as the tensor-core precisions ("Flash
 * Attention Memory Optimization Explained", section "Key Mechanisms"). 
 * Dropout and arbitrary attention masks are not supported.
 */
#ifndef FA_H_
#define FA_H_

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, size <= 0, Hq % Hkv != 0,
                             non-finite scale, causal not 0/1, overlap of an
                             output with another buffer, size overflow,
                             T >= 2^30 */
  FA_ERR_UNSUPPORTED = 2, /* d not in {16,32,64,128} or unknown dtype */
  FA_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
  FA_ERR_CUDA = 4,        /* a CUDA runtime/driver call failed (launch etc.) */
  FA_ERR_TIMEOUT = 5,     /* a kernel gave up waiting on a barrier (reported
                             by fa_debug_sync_check only) */
  FA_ERR_WORKSPACE = 6    /* the scratch workspace is missing or too small */
} fa_status;

typedef enum { FA_DTYPE_F32 = 0, FA_DTYPE_BF16 = 1, FA_DTYPE_F16 = 2 } fa_dtype;

/* Exact attention forward with log-sum-exp (see the header comment).
 *   q, k, v : device inputs; o, lse : device outputs
 *   B, Hq, Hkv, T, d : sizes (> 0; Hq a multiple of Hkv; d in {16,32,64,128})
 *   scale   : finite multiplier of every score (1/sqrt(d) is the usual one)
 *   causal  : 1 keeps key j for query i only when j <= i; 0 keeps all
 *   dtype   : element type of q, k, v and o
 *   stream  : cudaStream_t to enqueue on
 * Returns FA_OK once the kernel is enqueued; on any error nothing is
 * launched and the outputs are untouched. */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int Hq, int Hkv, int T, int d, float scale, int causal,
                 fa_dtype dtype, void* stream);

/* Band-masked (sliding-window) forward.  The yelogs.com Flash Attention2/
 * Triton tutorial, section "1. 稀疏注意力支持" (sparse-attention support),
 * restricts each query to the keys |i - j| <= window_size.  This call keeps
 * key j for query i iff  i - window_left <= j <= i + window_right  (and
 * j < T); -1 leaves that side unbounded.  The page's window is (w, w),
 * causal attention is (-1, 0), no mask is (-1, -1).  KV tiles outside every
 * row's band are skipped.  Other arguments, results and errors as fa_fwd
 * (non-causal); FA_ERR_INVALID_ARG also for a window value below -1. */
fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int Hq, int Hkv, int T, int d, float scale, int window_left,
                        int window_right, fa_dtype dtype, void* stream);

/* Local-global forward.  The yelogs.com Flash Attention2/Triton tutorial,
 * section "1. 稀疏注意力支持" (sparse-attention support), defines the
 * local-global mask: query i keeps key j iff |i - j| <= local_window OR j is
 * one of the global tokens (torch.isin over the key index) -- global tokens are
 * keys that every query attends to.  With causal = 1 the union is intersected
 * with j <= i.  The KV tiles a query tile visits are those of its band plus
 * the tiles holding a global key, or, with the larger workspace of
 * fa_fwd_local_global_packed_workspace_size, its band's tiles plus the global
 * keys gathered into packed 128-row tiles; all others are skipped.
 *   local_window  : >= 0
 *   global_tokens : DEVICE array of num_global int32 key indices, any order
 *                   (4-byte aligned; may be NULL when num_global = 0); repeats
 *                   and entries outside [0, T) select nothing more
 *   workspace     : DEVICE scratch of at least
 *                   fa_fwd_local_global_workspace_size(T) bytes, 16-byte
 *                   aligned, not overlapping any other buffer; contents on
 *                   entry ignored, on return undefined.  With at least
 *                   fa_fwd_local_global_packed_workspace_size(...) bytes the
 *                   global keys are packed (16-bit inputs, num_global > 0)
 * Other arguments and results as fa_fwd.  Enqueues a memset and three kernels
 * (key bitmask, list of tiles holding global keys, attention), and two more
 * when packing (the sorted token list, the gather of their K and V rows).  Errors: as
 * fa_fwd, plus FA_ERR_INVALID_ARG for local_window < 0, num_global < 0, a
 * NULL global_tokens with num_global > 0 or an overlapping workspace;
 * FA_ERR_MISALIGNED for a global_tokens pointer that is not 4-byte aligned;
 * FA_ERR_WORKSPACE for a NULL or too small workspace. */
fa_status fa_fwd_local_global(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int T, int d, float scale, int causal,
                              int local_window, const int* global_tokens, int num_global,
                              fa_dtype dtype, void* workspace,
                              unsigned long long workspace_bytes, void* stream);

/* Bytes of workspace fa_fwd_local_global needs for T keys (a bitmask of the
 * global keys and the list of 128-key tiles holding one: 20 bytes per tile,
 * plus 16); 0 for T <= 0. */
unsigned long long fa_fwd_local_global_workspace_size(int T);

/* Bytes of workspace with which fa_fwd_local_global packs the global keys
 * (bf16 and fp16 inputs): fa_fwd_local_global_workspace_size(T) plus the
 * sorted distinct tokens and their K and V rows gathered per (batch, KV head)
 * into 128-row tiles, R * 4 + 16 + 2 * B * Hkv * R * d * 2 bytes with R =
 * num_global rounded up to a multiple of 128 (at least 128).  A query tile
 * then visits its band's KV tiles plus ceil(#distinct tokens / 128) packed
 * tiles, instead of every 128-key tile that holds a global key; the results
 * are the same.  With a smaller workspace (at least the size above) the call
 * visits whole tiles.  For fp32 inputs, or num_global = 0, the same as
 * fa_fwd_local_global_workspace_size(T).  0 for invalid sizes or dtype. */
unsigned long long fa_fwd_local_global_packed_workspace_size(int B, int Hkv, int T, int d,
                                                             fa_dtype dtype, int num_global);

/* Split-KV forward (FlashDecoding-style; "Flash Attention Memory Optimization
 * Explained", section "Why It Matters", names FlashDecoding as the inference
 * extension).  Same operation, arguments and results as fa_fwd, for shapes
 * with too few (batch, head, 256-row block) work units to fill the GPU: the
 * keys of every row block are cut into num_splits contiguous ranges that run
 * on different SMs; each writes its normalised partial output O_s and
 * log-sum-exp L_s to `workspace`, and a second kernel merges them exactly,
 * L = m + ln sum_s exp(L_s - m) (m = max_s L_s), O = sum_s exp(L_s - L) O_s.
 *   num_splits : 1 .. 64 (1 = fa_fwd; fa_fwd_split_heuristic suggests one)
 *   workspace  : DEVICE scratch of at least fa_fwd_split_workspace_size(...)
 *                bytes, 16-byte aligned, not overlapping any other buffer;
 *                owned by the caller, contents on entry are ignored and on
 *                return are undefined; unused when num_splits = 1
 * fp32 inputs run the CUDA-core kernel, which needs no split (workspace
 * unused).  Errors: as fa_fwd, plus FA_ERR_INVALID_ARG for num_splits outside
 * 1..64 or an overlapping workspace, FA_ERR_WORKSPACE when num_splits > 1 and
 * the workspace is NULL or too small.  Calls that share a workspace and run
 * concurrently on the GPU race. */
fa_status fa_fwd_split(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int Hq, int Hkv, int T, int d, float scale, int causal,
                       fa_dtype dtype, int num_splits, void* workspace,
                       unsigned long long workspace_bytes, void* stream);

/* fa_fwd_split for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this is an interface choice of this library.)  Some
 * callers cannot call cudaMalloc: a plugin hosted by an application that
 * hands out all device memory through its own pool, where a raw cudaMalloc
 * would bypass the pool's accounting or fail once the pool has reserved the
 * device, or a latency-critical path that cannot afford cudaMalloc's implicit
 * device-wide synchronisation.  This entry point takes no workspace: its
 * scratch is a fixed 64 MiB array inside the library (every GPU that loads
 * libfa.so holds it until the process exits).  Arguments, results and errors
 * are those of fa_fwd_split without the workspace, plus FA_ERR_WORKSPACE when
 * fa_fwd_split_workspace_size(B, Hq, T, d, num_splits) exceeds 64 MiB (use a
 * smaller num_splits, or 1, which needs no scratch).
 * Set-up: the first call on each device looks up the scratch array's device
 * address (cudaGetSymbolAddress, no allocation).  The address is cached per device together with the id
 * of the CUDA context it belongs to; after cudaDeviceReset the next call
 * finds a new context and looks the address up again.  Every call on a device shares the one array and leaves
 * its partial results there; no call relies on earlier contents, but calls
 * that overlap on the GPU (for example on different streams) race. */
fa_status fa_fwd_split_static(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int Hq, int Hkv, int T, int d, float scale, int causal,
                              fa_dtype dtype, int num_splits, void* stream);

/* Bytes of workspace fa_fwd_split needs (num_splits * B * Hq * T * (d + 1) *
 * 4: fp32 partial outputs and log-sum-exps); 0 for invalid sizes. */
unsigned long long fa_fwd_split_workspace_size(int B, int Hq, int T, int d, int num_splits);

/* A split count for this shape on the current device: 1 when the row blocks
 * already occupy at least half of the SMs, else about one work unit per SM
 * with at least four 128-key tiles per split (at most 64 splits).  Returns 1
 * on invalid sizes. */
int fa_fwd_split_heuristic(int B, int Hq, int Hkv, int T, int d, int causal);

/* Backward pass: gradients of o = attention(q, k, v) with respect to q, k and
 * v for an upstream gradient d_o of o ("Flash Attention Memory Optimization
 * Explained", section "Key Mechanisms", item "Backward Checkpointing": the
 * forward's intermediates are recomputed, not stored).  The score matrix is
 * rebuilt tile by tile from q, k and the forward's lse, P = exp(S - lse), and
 *   dV  = sum over query heads of the group of P^T dO
 *   dP  = dO V^T,   D_i = sum_c dO[i][c] * O[i][c]  (= sum_j P_ij dP_ij)
 *   dS  = P * (dP - D)                              (softmax Jacobian)
 *   dQ  = scale * dS K,   dK = sum over the group of scale * dS^T Q
 * lse carries no gradient.
 *   q, k, v, o, lse : the forward's inputs and outputs (o and lse exactly as
 *                     a forward call with the same mask wrote them)
 *   d_o   : [B][Hq][T][d] upstream gradient, element type `dtype`
 *   dq    : [B][Hq][T][d], dk, dv : [B][Hkv][T][d]; written, element type
 *           `dtype` (round-to-nearest-even from fp32 accumulation)
 *   causal, window_left, window_right : the forward's mask (causal as
 *           fa_fwd; the band as fa_fwd_window, -1 = unbounded side; both
 *           combine by intersection)
 *   workspace : DEVICE scratch of at least fa_bwd_workspace_size(B, Hq, T)
 *           bytes, 16-byte aligned, not overlapping any other buffer; owned by
 *           the caller; contents on entry ignored, on return undefined
 * Kernels: bf16 and fp16 run on the tensor cores (two kernels, one over KV
 * tiles for dK and dV and one over query tiles for dQ, so that no gradient is
 * accumulated by atomics: results are deterministic); fp32 runs true-fp32
 * CUDA-core kernels.  Accumulation is fp32 throughout.
 * Errors: as fa_fwd, plus FA_ERR_INVALID_ARG when an output (dq, dk, dv)
 * overlaps another buffer or a window value is below -1, FA_ERR_WORKSPACE for
 * a NULL or too small workspace.  Enqueues three kernels on `stream` and
 * returns without synchronising. */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* d_o, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int T,
                 int d, float scale, int causal, int window_left, int window_right,
                 fa_dtype dtype, void* workspace, unsigned long long workspace_bytes,
                 void* stream);

/* Bytes of workspace fa_bwd needs: two fp32 values per query row (D_i and
 * lse_i * log2(e)), rows padded to a multiple of 128 per head; 0 for invalid
 * sizes. */
unsigned long long fa_bwd_workspace_size(int B, int Hq, int T);

/* Backward of the local-global forward (fa_fwd_local_global): the same
 * gradients as fa_bwd for the mask |i - j| <= local_window OR j in
 * global_tokens (intersected with j <= i when causal).  o and lse must come
 * from fa_fwd_local_global with the same mask.  Arguments as fa_bwd, with the
 * mask arguments of fa_fwd_local_global; the workspace is at least
 * fa_bwd_local_global_workspace_size(B, Hq, T) bytes (fa_bwd's rows plus the
 * key sets).  Errors: as fa_bwd and fa_fwd_local_global. */
fa_status fa_bwd_local_global(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* d_o, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int T, int d, float scale, int causal,
                              int local_window, const int* global_tokens, int num_global,
                              fa_dtype dtype, void* workspace,
                              unsigned long long workspace_bytes, void* stream);

/* Bytes of workspace fa_bwd_local_global needs: fa_bwd_workspace_size(B, Hq,
 * T) + fa_fwd_local_global_workspace_size(T); 0 for invalid sizes. */
unsigned long long fa_bwd_local_global_workspace_size(int B, int Hq, int T);

/* Forward from HOST buffers to HOST buffers.  Same operation, sizes and
 * layouts as fa_fwd, but q, k, v, o and lse are host pointers (pinned memory,
 * e.g. cudaHostAlloc, lets the copies run asynchronously and overlap; pageable
 * memory works, without overlap).  The batch is cut into `chunks` chunks of
 * whole batch entries; each chunk's inputs are copied to the device, its
 * attention computed and its outputs copied back, with the chunks alternating
 * between two streams of the library (created once per device) so that copies
 * overlap kernels.  The work is ordered after everything already on `stream`
 * and everything later on `stream` is ordered after it; the call returns
 * without synchronising (the host outputs are complete once `stream` has
 * reached this point).  Calls on one device run on the GPU in turn.  The
 * first call on a device creates the two streams and three events (kept
 * until the process exits); make it before any stream capture.
 *   chunks    : 1 .. B (larger values are clamped to B); each chunk should
 *               keep the GPU busy (B*Hq*ceil(T/256)/chunks work units of 256
 *               rows against the number of SMs)
 *   workspace : DEVICE scratch of at least fa_fwd_host_workspace_size(...)
 *               bytes (two chunks of q, k, v, o and lse), 16-byte aligned
 * Errors: as fa_fwd (for the host pointers), plus FA_ERR_INVALID_ARG for
 * chunks < 1 and FA_ERR_WORKSPACE for a NULL or too small workspace. */
fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int Hq, int Hkv, int T, int d, float scale, int causal,
                      fa_dtype dtype, int chunks, void* workspace,
                      unsigned long long workspace_bytes, void* stream);

/* Bytes of device workspace fa_fwd_host needs; 0 for invalid arguments. */
unsigned long long fa_fwd_host_workspace_size(int B, int Hq, int Hkv, int T, int d,
                                              fa_dtype dtype, int chunks);

/* Backward from HOST buffers to HOST buffers: fa_bwd's operation, sizes and
 * mask arguments with q, k, v, o, lse, d_o, dq, dk and dv on the host, in
 * `chunks` batch chunks pipelined over the library's two streams exactly as
 * fa_fwd_host does (same ordering, asynchrony and pinning notes).
 *   workspace : DEVICE scratch of at least fa_bwd_host_workspace_size(...)
 *               bytes (two chunk slots of every tensor and the rows' part)
 * Errors: as fa_bwd (for the host pointers), plus FA_ERR_INVALID_ARG for
 * chunks < 1. */
fa_status fa_bwd_host(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* d_o, void* dq, void* dk, void* dv, int B,
                      int Hq, int Hkv, int T, int d, float scale, int causal, int window_left,
                      int window_right, fa_dtype dtype, int chunks, void* workspace,
                      unsigned long long workspace_bytes, void* stream);

/* Bytes of device workspace fa_bwd_host needs; 0 for invalid arguments. */
unsigned long long fa_bwd_host_workspace_size(int B, int Hq, int Hkv, int T, int d,
                                              fa_dtype dtype, int chunks);

/* Static English text for a status code (never NULL). */
const char* fa_status_string(fa_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int fa_version(void);

/* Debug/test aid, not for the hot path: synchronises `stream`, then reads and
 * clears the device-side error word that kernels set when a barrier wait runs
 * out of time (each wait is bounded; on expiry the kernel abandons its work,
 * frees its tensor memory and exits instead of hanging).  Returns
 * FA_ERR_TIMEOUT if the word was set, FA_ERR_CUDA if the synchronisation
 * failed, else FA_OK. */
fa_status fa_debug_sync_check(void* stream);

/* Last CUDA error code seen by the library on this thread (0 if none);
 * detail for FA_ERR_CUDA. */
int fa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
