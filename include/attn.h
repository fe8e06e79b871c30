/*
 * attn.h -- C ABI of libattn.so: attention forward with online softmax on
 * GB300 (sm_103a).
 *
 * Two forms of O = softmax(scale * Q K^T [+ causal mask]) V, both computed
 * without ever writing S or P to global memory:
 *
 *   attn_fwd    multi-head prefill, FlashAttention-2 loop order ("FP32
 *               CUDA-core FlashAttention-2 v2" blog, dandandamowang
 *               post_1787450400: section 1.1 Q-outer/KV-inner loop, 1.2
 *               on-chip m/l/O, 1.3 deferred 1/l, 1.4 and 3.4 causal block
 *               skipping with diagonal-block masking, 3.5 single write of O).
 *   mla_decode  MLA absorbed decode over a paged 576-wide latent cache ("MLA
 *               x FlashAttention-3 fusion" article, hnwysp news 119127:
 *               latent layout [c_kv 512 | k_rope 64], the absorption
 *               identity Q K^T = (Q W_UK) c^T + Q_R k_R^T, and the
 *               online-softmax "partial reduction" stage of its pipeline).
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers (cudaMalloc / torch CUDA
 *     memory) of the current device, except where a comment says HOST.
 *   - The caller owns every buffer.  The library allocates no device memory
 *     per call; the kernels allocate and free tensor memory (TMEM) inside
 *     each CTA.  Tensor-map descriptors are built on the host per call and
 *     passed by value as kernel parameters.
 *   - Calls are asynchronous: they validate, enqueue on `stream`
 *     (cudaStream_t; NULL = the legacy default stream) and return.  They
 *     never synchronise and never trap.  Errors that only the device can see
 *     (a bad block-table entry, a wait that ran out) are recorded in a
 *     device error word and returned later by attn_device_status().
 *   - Return value: ATTN_OK (0) or a negative ATTN_ERR_* code; on error
 *     nothing was launched and attn_last_error() describes the cause.
 *   - Thread safety: calls may be made from several host threads; the error
 *     message is thread-local.
 *   - Device addresses of the library's own device variables (the error
 *     word, the prefill work counters, the fixed decode scratch) are looked
 *     up once per device and cached for the life of the process.  Do not
 *     keep using the library after cudaDeviceReset() in the same process:
 *     the cached addresses belong to the destroyed context.
 */
#ifndef GB300_ATTN_H_
#define GB300_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define ATTN_OK 0
#define ATTN_ERR_INVALID_ARG (-1)      /* null pointer, size <= 0, non-finite scale */
#define ATTN_ERR_UNSUPPORTED (-2)      /* head dim / dtype / head count not built */
#define ATTN_ERR_MISALIGNED (-3)       /* a base pointer is not 16-byte aligned */
#define ATTN_ERR_WORKSPACE_TOO_SMALL (-4)
#define ATTN_ERR_CUDA (-5)             /* a CUDA runtime / driver call failed */
#define ATTN_ERR_BAD_BLOCK_TABLE (-6)  /* device: block id outside [0, num_blocks) */
#define ATTN_ERR_BAD_SEQLEN (-7)       /* device: seqlen < 0 or > max_blocks*64 */
#define ATTN_ERR_DEVICE_TIMEOUT (-8)   /* device: a pipeline wait ran out (~2 s) */

/* ---- data types -------------------------------------------------------- */
#define ATTN_DTYPE_F32 0   /* fp32 in, fp32 out, fp32 arithmetic (CUDA cores) */
#define ATTN_DTYPE_BF16 1  /* bf16 in, bf16 out, fp32 accumulate (tcgen05) */

/*
 * attn_fwd -- multi-head attention forward (prefill).
 *
 *   q, k, v : [B, H, N, D] contiguous, element type `dtype`.
 *   o       : [B, H, N, D] contiguous, element type `dtype` (written).
 *   lse     : [B, H, N] float32 (written): natural-log logsumexp of the
 *             scaled, masked scores of each row.  The pages never output it;
 *             it is kept so that split results can be merged.
 *   causal  : nonzero -> key j is visible to query i iff j <= i (blog 3.4).
 *   scale   : multiplies Q K^T before the softmax (blog 3.3); finite.
 *   dtype   : ATTN_DTYPE_F32 (D == 64) or ATTN_DTYPE_BF16 (D == 64 or 128).
 *   stream  : cudaStream_t or NULL.
 * Requirements: all pointers non-null and 16-byte aligned; B, H, N >= 1.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA.
 * The bf16 path is one persistent kernel (one CTA per SM) whose CTAs draw
 * Q-tile pairs from a work counter: the call enqueues a 4-byte
 * cudaMemsetAsync of that counter on `stream`, then the kernel.  Ordinary
 * calls take one of 64 counters per device in turn, so at most 64 bf16
 * attn_fwd launches may be in flight at once across streams of one device
 * (launches on one stream reuse counters in order and are always safe).
 * A call made while `stream` is being captured into a CUDA graph gets a
 * counter of its own that no other call uses (up to 1984 such calls per
 * device and process; beyond that the call fails with ATTN_ERR_CUDA), so a
 * replay of the graph may overlap any ordinary launch or any other graph.
 * Two instantiations of the same captured graph share its counters: do not
 * run them at the same time.
 */
ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int N, int D, int causal, float scale, int dtype,
             void* stream);

/*
 * attn_fwd_tf32x3_workspace_size -- bytes of device workspace that
 * attn_fwd_tf32x3 needs for (B, H, N, D): 2 x B*H*N*64 floats for the split
 * K (each part rounded up to 256 bytes) plus 2 x B*H*64*Np floats' worth for
 * the split, transposed V (V_hi in fp32, V and V - V_hi in bf16; Np = N
 * rounded up to a multiple of 64).  Returns 0 for invalid sizes or D != 64.
 * Pure host arithmetic: no CUDA call.
 */
ATTN_API size_t attn_fwd_tf32x3_workspace_size(int B, int H, int N, int D);

/*
 * attn_fwd_tf32x3 -- fp32 attention forward on the tensor cores, accurate to
 * fp32 level: the same operation as attn_fwd with ATTN_DTYPE_F32 (the fp32
 * FlashAttention-2 forward of the "FP32 CUDA-core FlashAttention-2 v2" blog,
 * sections 1.2-1.4 and 3.3-3.5, with the tensor cores of its section 5 list
 * of what is left to do).  Every fp32 operand x is split into
 * hi = tf32(x) and lo = x - hi.  Q K^T is lo*hi + hi*lo + hi*hi on tcgen05
 * kind::tf32 (lo rounded to tf32) with fp32 accumulation; in P V the two
 * cross terms, which carry about 2^-11 of each product, run on bf16 operands
 * (kind::f16, bf16(P_lo) bf16(V) + bf16(P) bf16(V_lo)) into the same fp32
 * accumulator as the tf32 hi*hi.  O and LSE stay within 1e-4 of the exact
 * result on the tested inputs (the fp32 bound).
 *
 *   q, k, v : [B, H, N, 64] float32, contiguous.
 *   o       : [B, H, N, 64] float32 (written).
 *   lse     : [B, H, N] float32 (written), as for attn_fwd.
 *   causal, scale : as for attn_fwd.
 *   workspace : device buffer of >= attn_fwd_tf32x3_workspace_size(B, H, N, D)
 *             bytes, owned by the caller; the call overwrites it (a split
 *             copy of K and a split, transposed copy of V) and it must not be
 *             used by another call that is in flight at the same time.
 *   stream  : cudaStream_t or NULL.
 * Two kernels are enqueued: the split pre-pass, then the attention kernel
 * as a programmatic dependent of it.  Nothing is allocated.
 * Requirements: pointers non-null and 16-byte aligned; B, H, N >= 1; D = 64;
 * B*H*N < 2^31.
 * Errors: INVALID_ARG (null, size <= 0, non-finite scale), UNSUPPORTED
 * (D != 64, too large), MISALIGNED, WORKSPACE_TOO_SMALL, CUDA.  A stuck
 * pipeline is reported later by attn_device_status as DEVICE_TIMEOUT.
 */
ATTN_API int attn_fwd_tf32x3(const float* q, const float* k, const float* v, float* o,
                    float* lse, int B, int H, int N, int D, int causal, float scale,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_fwd_host_workspace_size -- bytes of device workspace attn_fwd_host
 * needs: one or two chunk buffers of [q | k | v | o] (ceil(B*H / chunks) heads
 * of N x D elements each) plus the chunk's LSE, every part rounded up to 256
 * bytes; chunks = min(B*H, 4).  Returns 0 for a combination attn_fwd does not
 * build.  Pure host arithmetic: no CUDA call.
 */
ATTN_API size_t attn_fwd_host_workspace_size(int B, int H, int N, int D, int dtype);

/*
 * attn_fwd_host -- attn_fwd on HOST buffers: the same arguments and result,
 * but q, k, v are read from and o, lse written to host memory (page-locked
 * memory lets the copies run asynchronously and overlap; pageable memory
 * works, with copies that block the calling thread).
 *
 *   workspace : device buffer, 256-byte aligned, of at least
 *               attn_fwd_host_workspace_size(...) bytes, owned by the caller
 *               and not shared with another call in flight.
 *   stream    : cudaStream_t or NULL; when the stream reaches the end of the
 *               call's work, o and lse are in host memory.
 * The B*H heads are cut into up to 4 contiguous chunks.  Chunk c+1 is copied
 * in and chunk c-1 copied out on two copy streams the library keeps per
 * device (created on first use), while chunk c runs on `stream`; events order
 * every hand-over, and the call makes `stream` wait for the last copy out.
 * Returns after enqueue.  Errors: as attn_fwd, plus WORKSPACE_TOO_SMALL and
 * MISALIGNED for the workspace, and CUDA for a failed copy or event call.
 */
ATTN_API int attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                  int B, int H, int N, int D, int causal, float scale, int dtype,
                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_host_workspace_size -- bytes of device workspace mla_decode_host
 * needs for these sizes on a device with num_sms SMs: room for q, the pool,
 * the table, the lengths, o and lse, then mla_decode's own workspace.
 * Returns 0 for invalid sizes.  Pure host arithmetic: no CUDA call.
 */
ATTN_API size_t mla_decode_host_workspace_size(int B, int Hq, int max_blocks_per_seq,
                                      int num_blocks, int num_sms);

/*
 * mla_decode_host -- mla_decode on HOST buffers: q, kv_cache, block_table and
 * seqlens are copied in from host memory, mla_decode runs, and o, lse are
 * copied back, all in order on `stream` (any sequence may use any page, so
 * the pool is copied whole).  workspace: device buffer, 256-byte aligned, of
 * at least mla_decode_host_workspace_size(...) bytes.  Errors: as
 * mla_decode, plus MISALIGNED for the workspace and CUDA for a failed copy.
 */
ATTN_API int mla_decode_host(const void* q, const void* kv_cache, const int32_t* block_table,
                    const int32_t* seqlens, void* o, float* lse, int B, int Hq,
                    float scale, int max_blocks_per_seq, int num_blocks, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * mla_decode_workspace_size -- bytes of device workspace mla_decode needs.
 *
 *   B, Hq, max_blocks_per_seq : as for mla_decode.
 *   num_sms         : SM count of the device that will run the call
 *                     (cudaDevAttrMultiProcessorCount); must be >= 2.
 * Returns 0 if an argument is invalid.  Pure host arithmetic: no CUDA call.
 */
ATTN_API size_t mla_decode_workspace_size(int B, int Hq, int max_blocks_per_seq,
                                 int num_sms);

/*
 * mla_decode_split_workspace_size -- bytes of device workspace that
 * mla_decode_split needs: as mla_decode_workspace_size, for a fixed split
 * length of `pages_per_split` 64-token pages (0 = the automatic plan, the
 * same size as mla_decode_workspace_size).  A fixed split length can cut the
 * pages into more chunks than the automatic plan, each with its own partial
 * results, so the size depends on it.
 * Returns 0 if an argument is invalid.  Pure host arithmetic: no CUDA call.
 */
ATTN_API size_t mla_decode_split_workspace_size(int B, int Hq, int max_blocks_per_seq,
                                       int num_sms, int pages_per_split);

/*
 * mla_decode -- MLA absorbed decode, one query token per sequence.
 *
 *   q           : [B, Hq, 576] bf16 absorbed queries [q_nope W_UK | q_rope].
 *   kv_cache    : [num_blocks, 64, 576] bf16 latent pool; row t of a page is
 *                 [c_kv (512) | k_rope (64)].  K is the whole row, V is its
 *                 first 512 entries (the same bytes; nothing is decompressed).
 *   block_table : [B, max_blocks_per_seq] int32; page j of sequence b lives at
 *                 kv_cache[block_table[b * max_blocks_per_seq + j]].
 *   seqlens     : [B] int32, tokens t < seqlens[b] are visible (the single
 *                 query is the newest token, so no causal mask applies).
 *   o           : [B, Hq, 512] bf16 (written).
 *   lse         : [B, Hq] float32 (written); a sequence of length 0 gets
 *                 o = 0 and lse = -inf.
 *   scale       : finite multiplier of q . C_t.
 *   workspace   : device buffer of >= mla_decode_workspace_size(...) bytes,
 *                 used for the split plan and split partials; 16-byte
 *                 aligned; contents need not be initialised.  It must not be
 *                 shared by calls that may run concurrently.
 * Supported: Hq == 128.  Device-side checks: a block id outside
 * [0, num_blocks) or a length outside [0, max_blocks_per_seq*64] is never
 * dereferenced: the affected pages are skipped, the sequence's output is
 * unspecified, and ATTN_ERR_BAD_BLOCK_TABLE / ATTN_ERR_BAD_SEQLEN is recorded
 * for attn_device_status().
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE_TOO_SMALL, CUDA.
 */
ATTN_API int mla_decode(const void* q, const void* kv_cache, const int32_t* block_table,
               const int32_t* seqlens, void* o, float* lse, int B, int Hq,
               float scale, int max_blocks_per_seq, int num_blocks,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_split -- mla_decode with a fixed split length.
 *
 * Identical to mla_decode except that every sequence's pages are cut into
 * splits of `pages_per_split` 64-token pages along one flat page order
 * (0 = the automatic plan).  The results agree with mla_decode within
 * rounding; it exists to exercise the split/merge path at any split count.
 * The workspace must be sized by mla_decode_split_workspace_size with the
 * same pages_per_split.
 */
ATTN_API int mla_decode_split(const void* q, const void* kv_cache,
                     const int32_t* block_table, const int32_t* seqlens,
                     void* o, float* lse, int B, int Hq, float scale,
                     int max_blocks_per_seq, int num_blocks, void* workspace,
                     size_t workspace_bytes, int pages_per_split,
                     void* stream);

/*
 * mla_decode_noalloc -- mla_decode for callers that cannot allocate device
 * memory when they call.
 *
 * The pages this library follows have no counterpart to this entry point.
 * It exists for callers that are not allowed to allocate device memory at
 * call time: for example a host that hands all free device memory to its
 * own pool up front and forbids later cudaMalloc, or a caller on a path that
 * must not pay for the allocator (cudaMalloc / cudaFree can synchronise the
 * device).  Such callers cannot provide mla_decode's workspace.
 *
 * Arguments and results are those of mla_decode minus the workspace; the
 * automatic split plan is used.  The plan and the split partials live in
 * one fixed array inside libattn.so (a file-scope static __device__ array of
 * 21,218,048 bytes, about 20.2 MiB), which every GPU that loads the library
 * keeps until the process exits.
 *   Limits: B <= 8192 sequences and a device of at most 160 SMs; beyond
 *   them the call returns ATTN_ERR_UNSUPPORTED and launches nothing.
 *   Set-up: the first call on each device looks up the array's device
 *   address (cudaGetSymbolAddress, with that device current) and caches it;
 *   make that first call before any stream capture.
 *   Sharing: every call on a device uses the same array, and the array keeps
 *   the last call's contents (each call rewrites everything it reads).  Calls
 *   that can overlap on the GPU -- on unordered streams or from several host
 *   threads -- race on it; the caller must serialise them.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA.
 */
ATTN_API int mla_decode_noalloc(const void* q, const void* kv_cache,
                                const int32_t* block_table,
                                const int32_t* seqlens, void* o, float* lse,
                                int B, int Hq, float scale,
                                int max_blocks_per_seq, int num_blocks,
                                void* stream);

/*
 * mla_absorb_q -- the absorbed query that mla_decode takes ("MLA x
 * FlashAttention-3 fusion" article: the absorption identity
 * Q K^T = (Q W_UK) c^T + Q_R k_R^T, which folds W_UK into the query).
 *
 *   q_nope   : [B, Hq, d_nope] bf16, the non-rotary part of each head's query.
 *   q_rope   : [B, Hq, d_rope] bf16, the rotary part (passed through).
 *   w_uk     : [Hq, d_nope, d_latent] bf16, each head's key up-projection
 *              (key_nope_h = c W_UK_h^T for a latent row c).
 *   q_out    : [B, Hq, d_latent + d_rope] bf16 (written):
 *              [q_nope_h W_UK_h | q_rope_h]; mla_decode takes d_latent = 512,
 *              d_rope = 64.
 * One kernel on `stream`: per (head, 128 output columns, 64 tokens) a
 * tcgen05 product with fp32 accumulation and a bf16 result, plus the copy of
 * q_rope.  It is launched as a programmatic dependent of the previous kernel
 * on the stream and reads nothing before that kernel has completed.
 * Requirements: pointers non-null and 16-byte aligned; every width a
 * multiple of 8.  Built for d_nope a multiple of 64 up to 512 and d_latent a
 * multiple of 64 (else UNSUPPORTED).  Errors: INVALID_ARG, UNSUPPORTED,
 * MISALIGNED, CUDA.
 */
ATTN_API int mla_absorb_q(const void* q_nope, const void* q_rope, const void* w_uk,
                          void* q_out, int B, int Hq, int d_nope, int d_rope, int d_latent,
                          void* stream);

/*
 * mla_project_out -- each head's output from mla_decode's latent output:
 * out_h = o_latent_h W_UV_h (the value up-projection the article's fused
 * kernel applies after the latent attention).
 *
 *   o_latent : [B, Hq, d_latent] bf16 (mla_decode's o; d_latent = 512).
 *   w_uv     : [Hq, d_latent, d_v] bf16, each head's value up-projection.
 *   out      : [B, Hq, d_v] bf16 (written).
 * Same execution and errors as mla_absorb_q; built for d_latent a multiple of
 * 64 up to 512 and d_v a multiple of 64.
 */
ATTN_API int mla_project_out(const void* o_latent, const void* w_uv, void* out, int B, int Hq,
                             int d_latent, int d_v, void* stream);

/*
 * attn_device_status -- synchronise `stream`, then return and clear the
 * device error word of the current device (ATTN_OK if no kernel recorded an
 * error since the last call).  attn_last_error() then names the failing check.
 */
ATTN_API int attn_device_status(void* stream);

/* attn_last_error -- thread-local text for the last nonzero return. */
ATTN_API const char* attn_last_error(void);

/*
 * attn_fwd_test_skip_load -- TEST HOOK for the bounded-wait failure path.
 *
 * Same as attn_fwd with dtype = ATTN_DTYPE_BF16, except that the producer
 * warp of every CTA deliberately never issues K/V load number
 * `skip_load_index` (>= 1, counting K0, V0, K1, V1, ...); K_j and V_j share
 * one pipeline stage, so both loads of that block are skipped.  The consumers'
 * bounded waits then run out (about 2 s), the kernel records
 * ATTN_ERR_DEVICE_TIMEOUT, every CTA unwinds and frees its tensor memory, and
 * attn_device_status() returns the code.  Nothing hangs, faults or traps.
 * Output contents are unspecified.  Not for production use.
 */
ATTN_API int attn_fwd_test_skip_load(const void* q, const void* k, const void* v,
                            void* o, float* lse, int B, int H, int N, int D,
                            int causal, float scale, void* stream,
                            int skip_load_index);

/*
 * attn_fwd_f32_test_skip_load -- TEST HOOK for the bounded-wait failure path
 * of the fp32 CUDA-core kernel.
 *
 * Same as attn_fwd with dtype = ATTN_DTYPE_F32 (D = 64), except that no thread
 * of any CTA copies K/V block `skip_block` (>= 0, 64 keys each) or reports it
 * on the block's full mbarrier.  The CTA's bounded waits on that block (and,
 * for block 0, the second half's wait for the first half to start it) run out
 * after about 2 s, the kernel records ATTN_ERR_DEVICE_TIMEOUT, each thread
 * lets its own copies land and returns, and attn_device_status() returns the
 * code.  Nothing hangs, faults or traps.  Output contents are unspecified.
 * Not for production use.
 */
ATTN_API int attn_fwd_f32_test_skip_load(const float* q, const float* k, const float* v,
                                         float* o, float* lse, int B, int H, int N, int D,
                                         int causal, float scale, void* stream,
                                         int skip_block);

/*
 * attn_fwd_tf32x3_test_skip_load -- TEST HOOK for the bounded-wait failure
 * path of attn_fwd_tf32x3.
 *
 * Same as attn_fwd_tf32x3, except that the producer warp of every CTA never
 * issues the loads of K/V block `skip_block` (>= 0, 64 keys per block).  The
 * S issuer's bounded wait for that block runs out (about 2 s), the kernel
 * records ATTN_ERR_DEVICE_TIMEOUT, every role of the CTA unwinds (its issued
 * MMAs complete and its issued copies land before tensor memory is freed)
 * and attn_device_status() returns the code.  CTAs whose tile visits fewer
 * blocks finish normally.  Output contents are unspecified.  Not for
 * production use.
 */
ATTN_API int attn_fwd_tf32x3_test_skip_load(const float* q, const float* k, const float* v,
                                            float* o, float* lse, int B, int H, int N, int D,
                                            int causal, float scale, void* workspace,
                                            size_t workspace_bytes, void* stream,
                                            int skip_block);

/*
 * mla_decode_test_skip_load -- TEST HOOK for the bounded-wait failure path
 * of the two-CTA decode cluster.
 *
 * Same as mla_decode (automatic plan), except that in every cluster the
 * producer warp of CTA rank 1 never issues the loads of its pipeline step
 * `skip_step` (>= 0; one step = one 64-token page of the cluster's work, in
 * order).  Rank 1's bounded wait for that step runs out (about 2 s); rank 0,
 * which then never receives rank 1's partial scores for the step, runs out
 * in its own bounded wait; the kernel records ATTN_ERR_DEVICE_TIMEOUT; both
 * CTAs unwind, meet at the final cluster barrier (an aborted CTA waits 50 us
 * first, so that no partial-score store or P-row copy is in flight towards a
 * CTA that has left) and free their tensor memory.  attn_device_status()
 * returns the code.
 * Clusters with fewer steps finish normally.  Output contents are
 * unspecified.  Not for production use.
 */
ATTN_API int mla_decode_test_skip_load(const void* q, const void* kv_cache,
                                       const int32_t* block_table, const int32_t* seqlens,
                                       void* o, float* lse, int B, int Hq, float scale,
                                       int max_blocks_per_seq, int num_blocks,
                                       void* workspace, size_t workspace_bytes,
                                       void* stream, int skip_step);

/*
 * attn_kv_tiles -- host helper: number of KV tiles of width Bc that the Q
 * tile `q_tile` (rows [q_tile*Br, q_tile*Br + Br)) visits for sequence
 * length N.  Causal: kv_limit = min(q_start + Br, N), else N; the count is
 * ceil(kv_limit / Bc) (blog 3.4).  Returns -1 on invalid arguments.
 */
ATTN_API int attn_kv_tiles(int N, int Br, int Bc, int causal, int q_tile);

/*
 * attn_kernel_info -- host helper: tile shape and dynamic shared memory of
 * the prefill kernel that attn_fwd launches for (dtype, D): writes Br, Bc,
 * threads per CTA and shared bytes per CTA.  Returns ATTN_ERR_UNSUPPORTED
 * for a combination that is not built.
 */
ATTN_API int attn_kernel_info(int dtype, int D, int* Br, int* Bc, int* threads,
                     int* smem_bytes);

#ifdef __cplusplus
}
#endif
#endif /* GB300_ATTN_H_ */
