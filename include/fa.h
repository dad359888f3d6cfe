/* libfa — exact tiled attention forward (FlashAttention forward) for GB300 (sm_103a).
 *
 * O = softmax(scale * Q K^T) V, computed tile by tile with an online softmax
 * (running row max m and running sum l; the partial output is rescaled by
 * exp(m_old - m_new) when the max rises; O is divided by l once at the end),
 * so the N_q x N_k score and probability matrices never reach device memory.
 * Also returned: the FP32 log-sum-exp of each row's scaled scores, the small
 * per-row statistic the backward pass recomputes from. Around the forward:
 * its backward pass (fa_backward), decode over a paged K/V cache
 * (fa_decode_paged), FP16 tensors, FP8 E4M3 inputs (fa_forward_fp8),
 * host-memory requests, an allocation-free variant and the unfused baseline.
 *
 * Sources: "Why is standard attention memory-bound, and how does FlashAttention
 * fix it?" (interview.clozo.ai), Step 1 (definition), Step 3 (online softmax),
 * Step 4 (saved per-row statistics); "Flash Attention Mechanics: How Tiled
 * Attention Fits in SRAM" (interviewprepkit.dev), "The Tiling Algorithm";
 * "FlashAttention HBM bytes, one head, 8K" (inferenceinterviews.com),
 * "A strong answer" (FA2 query-block order, L2 reuse) and "What interviewers
 * probe next" (causal tile skipping; decode with GQA).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers of the CURRENT device, owned by
 *    the caller; the library keeps no reference after the call returns. A
 *    pointer to host memory (pinned or not) or to another GPU's memory is
 *    rejected with FA_ERR_INVALID_ARG before anything is enqueued.
 *  - Per-device state (the status word's address, the scratch array's
 *    address, the workspace pool) is looked up once per device and kept for
 *    the life of the process: do not use libfa across cudaDeviceReset.
 *  - q: BF16 [B][H_q][N_q][d];  k, v: BF16 [B][H_kv][N_k][d];  o: BF16
 *    [B][H_q][N_q][d]; lse: FP32 [B][H_q][N_q] or NULL. All contiguous,
 *    row-major, 16-byte aligned.
 *  - GQA: query head h reads KV head h / (H_q / H_kv); H_q % H_kv must be 0.
 *  - causal != 0: query row i sees key j iff j <= i + (N_k - N_q) (bottom-right
 *    aligned; the usual lower triangle when N_q == N_k). A row that sees no
 *    key gets O = 0 and LSE = -inf.
 *  - lse[i] = ln(sum_j exp(scale * q_i . k_j)) over the visible keys.
 *  - scale must be finite and > 0 (1/sqrt(d) is the usual value).
 *  - d must be 64 or 128, or 256 for the forward entry points fa_forward,
 *    fa_forward_fp16, fa_forward_noalloc and fa_forward_host[_packed]
 *    (FA_ERR_UNSUPPORTED otherwise; FP8 inputs: 64 or 128).
 *  - stream: a cudaStream_t (NULL = legacy default stream). Calls are
 *    asynchronous: they return once the work is enqueued. Argument errors are
 *    reported before anything is enqueued. Launch errors return FA_ERR_CUDA
 *    (details: fa_get_last_cuda_error). Errors during execution surface at the
 *    caller's next synchronisation; a kernel that gave up on a bounded wait
 *    records FA_ERR_TIMEOUT in the device status word (fa_device_status).
 */
#ifndef LIBFA_FA_H
#define LIBFA_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1, /* null/misaligned/overlapping pointer, bad size, H_q % H_kv, scale */
  FA_ERR_UNSUPPORTED = -2, /* valid request this build does not implement (head dim, entry point) */
  FA_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
  FA_ERR_NO_MEMORY = -4,   /* stream-ordered workspace allocation failed, or workspace too small */
  FA_ERR_TIMEOUT = -5,     /* a kernel gave up on a bounded wait (device status word) */
  FA_ERR_TOO_LARGE = -6,   /* fa_forward_noalloc: needs more than its static scratch holds */
  FA_ERR_BOUNDS = -7       /* FA_DEBUG builds: a device-side bounds check failed (status word) */
} fa_status;

/* Element type of q, k, v and o for the entry points that take one. */
typedef enum { FA_DTYPE_BF16 = 0, FA_DTYPE_FP16 = 1 } fa_dtype;

/* Exact attention forward, fused (the tiled online-softmax kernel).
 * Prefill: tcgen05/TMA kernel, two 128-row query tiles per CTA, K/V tiles of
 * 128 keys. Query blocks that do not fill a whole wave of the GPU have their
 * key range split over several CTAs. When every block is split (fewer blocks
 * than SMs), the CTAs of a block run as one thread-block cluster and merge
 * their partial (m, l, O) results through distributed shared memory at the
 * end of the kernel (no workspace, one launch); otherwise a second kernel
 * (programmatic dependent launch on the same stream) merges them. The main
 * kernel is itself a programmatic dependent launch: its set-up may overlap the
 * previous kernel on the stream, and it reads and writes global memory only
 * after that kernel has completed.
 * Decode / few queries (the H_q/H_kv * N_q query rows that share a KV head
 * number at most 16): one CTA per (batch, KV head, run of consecutive 128-key
 * chunks) reads each K and V chunk once for all those rows, the runs sized so
 * that the grid is about 1.7 CTAs per SM; run partials are merged the same way
 * (in a cluster when a KV head has at most 8 runs, else by a second kernel).
 * Every call can be captured into a CUDA graph once a first call has run on
 * the device outside the capture (it does one-time set-up).
 * Head dimension 256: one CTA per 128-row query tile (a 256-column output tile
 * fills half of the SM's tensor memory), two 128-key score buffers in turn,
 * K and V in 128-column halves; no key-range split, no workspace, one launch.
 * Split and decode partials live in a stream-ordered workspace taken from a
 * library-owned memory pool on the current device (cudaMallocFromPoolAsync /
 * cudaFreeAsync on `stream`); the pool keeps freed memory reserved for later
 * calls until the process exits. No pointer outlives the call. With
 * FA_TEST_WORKSPACE_FAIL=1 in the environment every workspace allocation fails
 * (FA_ERR_NO_MEMORY, nothing enqueued): a hook to test that error path.
 * Returns FA_OK or an fa_status code. */
int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
               int H_kv, int N_q, int N_k, int d, int causal, float scale, void* stream);

/* fa_forward on FP16 tensors: q, k, v and o hold IEEE binary16 values instead
 * of BF16, with the same layouts and every other convention, result and error
 * code of fa_forward (FP32 accumulation and LSE). The pages size their
 * tensors in FP16 ("Flash Attention Mechanics", its opening and "Why Standard
 * Attention Is Memory-Bound"; "Why is standard attention memory-bound...",
 * Step 1). P is rounded to FP16 before the P V product; a row's exponentials are kept
 * at most 2^15 against a reference max, so they never overflow FP16. */
int fa_forward_fp16(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int H_q, int H_kv, int N_q, int N_k, int d, int causal, float scale,
                    void* stream);

/* fa_forward on FP8 inputs ("Flash Attention Mechanics...", "FlashAttention 2
 * and FlashAttention 3": FP8 as the next precision step). q, k, v hold FP8
 * E4M3 codes (one byte per element: sign, 4 exponent bits with bias 7, 3
 * mantissa bits, subnormals, no infinities, 0x7F/0xFF NaN), in fa_forward's
 * layouts; each tensor stands for decode(code) * its factor (descale_q,
 * descale_k, descale_v: finite and > 0). The result is attention over those
 * values: o is BF16 [B][H_q][N_q][d], lse FP32 [B][H_q][N_q] as in fa_forward.
 * Arithmetic: S = Q K^T from the codes on the tensor cores (exact products,
 * FP32 accumulation), the factors of Q and K and `scale` folded into the
 * exponent; P rounded to E4M3 (nearest even, at most 2^8 against the row's
 * reference max) for the P V product; O multiplied by descale_v / l in FP32
 * and rounded to BF16. d must be 64 or 128 (FA_ERR_UNSUPPORTED otherwise). Every
 * request runs the prefill kernel (including one-query decode shapes). Pointers,
 * alignment, overlap, workspace and error codes as fa_forward. */
int fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H_q,
                   int H_kv, int N_q, int N_k, int d, int causal, float scale, float descale_q,
                   float descale_k, float descale_v, void* stream);

/* n forward requests of one shape whose tensors live in HOST memory (no
 * counterpart on the pages, which start from tensors in device memory: this is
 * the serving-side runtime around the same path). For request i, q[i], k[i],
 * v[i] are host pointers to its inputs and o[i], lse[i] to its outputs, in
 * fa_forward's layouts; `lse` (the array) or any lse[i] may be NULL (that LSE is
 * not copied back). dtype: FA_DTYPE_BF16 (fa_forward) or FA_DTYPE_FP16
 * (fa_forward_fp16). Host pointers need no alignment; page-locked memory
 * (cudaHostAlloc, cudaHostRegister) lets the copies run asynchronously.
 * Execution: each request's inputs are copied into one of three device slots
 * (stream-ordered memory from libfa's pool, on `stream`), the fused forward
 * runs on `stream`, and O, LSE are copied back. The copies run on two
 * library-owned streams of the current device, so later requests' copies in
 * and earlier requests' copies out overlap request i's kernels. Each tensor is its own
 * copy (fa_forward_host_packed moves a request with one copy each way).
 * Ordering: all of it runs after the work already on `stream`, and work
 * enqueued on `stream` later runs after all of it; the call returns once
 * everything is enqueued, so synchronise `stream` before reading outputs or
 * reusing inputs. Concurrent calls on one device enqueue one at a time.
 * Returns FA_OK; FA_ERR_INVALID_ARG (n < 0, NULL arrays or request pointers,
 * bad shape or scale, unknown dtype) or FA_ERR_UNSUPPORTED before anything is
 * enqueued; FA_ERR_NO_MEMORY if the slots cannot be allocated; FA_ERR_CUDA if a
 * copy or launch fails (requests before the failing one may have run; the
 * caller's stream still waits for everything that was enqueued). */
int fa_forward_host(int n, const void* const* q, const void* const* k, const void* const* v,
                    void* const* o, float* const* lse, int B, int H_q, int H_kv, int N_q, int N_k,
                    int d, int causal, float scale, int dtype, void* stream);

/* fa_forward_host with each request packed into two host buffers: qkv[i]
 * holds Q, K and V back to back (Q first, then K, then V, each in fa_forward's
 * layout, no padding) and out[i] receives O followed by LSE (FP32). Each
 * request then moves with one copy in and one copy out, which runs closer to
 * the host link's rate than several smaller copies. Everything else as
 * fa_forward_host. */
int fa_forward_host_packed(int n, const void* const* qkv, void* const* out, int B, int H_q, int H_kv,
                           int N_q, int N_k, int d, int causal, float scale, int dtype, void* stream);

/* Gradients of the exact attention forward: given q, k, v, the forward's o and
 * lse (FP32, required) and the upstream gradient dout (= dL/dO, o's layout),
 * writes dq (q's layout), dk and dv (k's layout), all of element type dtype
 * (FA_DTYPE_BF16 or FA_DTYPE_FP16) with FP32 accumulation. Same scale, causal
 * and GQA conventions as fa_forward: dk and dv of a KV head sum over the query
 * heads that read it. The scores are recomputed tile by tile from q, k and the
 * saved lse, not stored ("Why is standard attention memory-bound...", Step 4).
 * Work: a per-row preprocessing kernel (D = rowsum(dout * o)), then one
 * launch whose CTAs compute dK/dV over key blocks or dQ over query tiles, on
 * `stream`, with two B*H_q*roundup(N_q, 128) FP32 arrays of stream-ordered
 * workspace from libfa's pool. Deterministic (no atomics). Pointers: device, 16-byte aligned; the
 * outputs may not overlap any input or each other. When N_q or N_k is 0 the
 * gradients that exist are zero-filled. Returns FA_OK, FA_ERR_INVALID_ARG,
 * FA_ERR_UNSUPPORTED (d not 64/128; d = 256 is forward-only), FA_ERR_NO_MEMORY
 * or FA_ERR_CUDA. */
int fa_backward(const void* q, const void* k, const void* v, const void* o, const float* lse,
                const void* dout, void* dq, void* dk, void* dv, int B, int H_q, int H_kv, int N_q,
                int N_k, int d, int causal, float scale, int dtype, void* stream);

/* Decode attention over a paged K/V cache: for each sequence b, the N_q
 * query rows of q (layout as fa_forward) attend to that sequence's first
 * seqlens_k[b] keys, in order, exactly as fa_forward would over the same keys
 * stored contiguously (same scale, causal and GQA conventions; a sequence of
 * length 0, or a causal row that sees no key, gets O = 0 and LSE = -inf).
 * Decode is reading K and V once per KV head ("FlashAttention HBM bytes, one
 * head, 8K", "What interviewers probe next"); the pages describe no cache
 * layout, so this layout is the library's own:
 *  - k_cache, v_cache: element type dtype, [num_pages][H_kv][128][d]: a page
 *    holds 128 consecutive keys of one sequence for every KV head; device,
 *    16-byte aligned.
 *  - block_table: int32 [B][max_pages], device: key j of sequence b is row
 *    j % 128 of page block_table[b][j / 128]. Entries past a sequence's last
 *    page are not read; every entry that is read must lie in [0, num_pages)
 *    (an entry outside it reads as zeros, it does not fault).
 *  - seqlens_k: int32 [B], device; values are clamped to [0, max_pages * 128].
 *  - o: dtype [B][H_q][N_q][d]; lse: FP32 [B][H_q][N_q] or NULL.
 * Rows per KV head, (H_q / H_kv) * N_q, must be at most 16 (the decode
 * kernel's tile), else FA_ERR_UNSUPPORTED. Workspace for the partials of long
 * sequences comes from libfa's stream-ordered pool (none when they are merged
 * inside a thread-block cluster). Returns FA_OK, FA_ERR_INVALID_ARG,
 * FA_ERR_UNSUPPORTED, FA_ERR_NO_MEMORY or FA_ERR_CUDA. */
int fa_decode_paged(const void* q, const void* k_cache, const void* v_cache, const int* block_table,
                    const int* seqlens_k, void* o, float* lse, int B, int H_q, int H_kv, int N_q,
                    int num_pages, int max_pages, int d, int causal, float scale, int dtype, void* stream);

/* fa_forward without any device-memory allocation. (The pages have no
 * counterpart: this exists for callers, not for the method.)
 * For callers that cannot allocate device memory on this path: a serving loop
 * that must never block in cudaMalloc/cudaFree (they can synchronise the
 * device and take unbounded time), a process whose device memory is fully
 * reserved up front by another allocator, or a deployment that sizes all of
 * its memory before it starts. Same arguments, conventions, kernel and results
 * as fa_forward. The caller still provides q, k, v, o and lse.
 * Scratch: when a query block's key range is split over several CTAs, the
 * partial results go to a fixed 32 MiB array inside libfa's device image
 * (every GPU that loads libfa holds it until the process exits) instead of a
 * pool allocation. Requests whose partials would not fit return
 * FA_ERR_TOO_LARGE before anything is enqueued; requests that need no split
 * use no scratch at all.
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * Sharing: every call uses the same array, which keeps the last call's
 * contents (each call writes every partial it reads, so nothing needs
 * clearing). Calls whose execution overlaps on the GPU race on the array:
 * issue them on one stream, or order them with events. */
int fa_forward_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H_q, int H_kv, int N_q, int N_k, int d, int causal, float scale,
                       void* stream);

/* The unfused three-kernel path, kept as the measured traffic baseline
 * ("FlashAttention HBM bytes, one head, 8K", "A strong answer": S written,
 * read, P written, read). Kernel 1: S = scale * Q K^T stored as BF16 in
 * `workspace`; kernel 2: row softmax S -> P in place (BF16) and LSE; kernel
 * 3: O = P V. `workspace` is a caller-owned device buffer of at least
 * fa_naive_workspace_bytes(B, H_q, N_q, N_k) bytes (16-byte aligned); the
 * score rows are padded to a multiple of 8 elements. Same conventions and
 * return codes as fa_forward; FA_ERR_NO_MEMORY if workspace_bytes is short. */
int fa_naive_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H_q, int H_kv, int N_q, int N_k, int d, int causal, float scale,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace fa_naive_forward needs: B*H_q*N_q*roundup(N_k, 8)*2. 0 on bad sizes. */
size_t fa_naive_workspace_bytes(int B, int H_q, int N_q, int N_k);

/* How fa_forward would run a request on the current device, without running
 * it (no paper counterpart: a planning query for callers that size buffers or
 * count launches). Same shape checks as fa_forward (no pointers involved).
 * Outputs (each may be NULL): *ctas = CTAs of the main kernel; *launches =
 * kernels one call enqueues (0 for an empty request, 1, or 2 when a merge
 * kernel follows); *workspace_bytes = stream-ordered workspace the call
 * allocates, which is also the scratch fa_forward_noalloc needs (0 when the
 * split partials are merged inside thread-block clusters). The plan depends on
 * the device's SM count and cluster capacity, and on the environment switch
 * FA_CLUSTER_MERGE=0 (merge kernel instead of in-cluster merge). Returns FA_OK,
 * FA_ERR_INVALID_ARG or FA_ERR_UNSUPPORTED. */
int fa_forward_plan(int B, int H_q, int H_kv, int N_q, int N_k, int d, int causal, long long* ctas,
                    int* launches, size_t* workspace_bytes);

/* Failure-detection self-test (no counterpart on the pages; the kernels'
 * bounded waits are what it exercises). Enqueues on `stream` one CTA that runs
 * the same bounded mbarrier wait the kernels use, on a barrier nothing ever
 * arrives at, with a limit of timeout_ns (1 ns .. 10 s) instead of the kernels'
 * 2 s: the wait gives up, records FA_ERR_TIMEOUT in the device status word and
 * the kernel returns, leaving the context usable. Read the result with
 * fa_device_status. Returns FA_OK once enqueued, FA_ERR_INVALID_ARG for a limit
 * out of range, FA_ERR_CUDA on a launch failure. */
int fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

/* 1 if this library was compiled with FA_DEBUG (device-side bounds checks:
 * every tensor-memory column range, shared-memory offset and global row index
 * the kernels use is checked first; a failed check records FA_ERR_BOUNDS in the
 * device status word and the access is skipped, nothing faults), else 0. No
 * counterpart on the pages: it stands in for a memory checker. */
int fa_debug_build(void);

/* FA_DEBUG builds: enqueue on `stream` one CTA whose single bounds check fails
 * by construction (no memory is touched), so fa_device_status then reports
 * FA_ERR_BOUNDS: a test of the recording path. Release builds return
 * FA_ERR_UNSUPPORTED and enqueue nothing. */
int fa_selftest_bounds(void* stream);

/* Static description of an fa_status code. Never NULL. */
const char* fa_status_string(int status);

/* The cudaError_t of the last CUDA failure this thread saw inside libfa (0 if none). */
int fa_get_last_cuda_error(void);

/* Synchronises the current device, then returns FA_OK, FA_ERR_TIMEOUT (a
 * kernel's bounded wait ran out) or FA_ERR_BOUNDS (FA_DEBUG builds: a bounds
 * check failed) from the device status word; `reset` != 0 clears the word
 * afterwards. FA_ERR_CUDA if synchronisation fails. */
int fa_device_status(int reset);

/* Library version, (major << 16) | minor. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBFA_FA_H */
