/*
 * libbiv -- batch-invariant verification step of deterministic LLM decoding,
 * hand-written CUDA for sm_103a (GB300).
 *
 * Sources (pages cited by title and paragraph / section):
 *   [DVR]      tgstat @ashnskt post 392: batch-invariant matmul / RMSNorm /
 *              attention (para 1); LLM-42 Decode-Verify-Rollback: a fixed-batch
 *              verifier anchored at the last correct token, rollback on
 *              divergence, fast-path KV rows overwritten by the verifier
 *              (para 3); W = N requests x K tokens in one verify batch (para 4).
 *   [GUIDE]    "NVIDIA publishes AI inference guide, 6x lossless speedup":
 *              speculative decoding (verify the drafts in one pass, restart at
 *              the break point); GQA tile rule G * (1 + D) <= 128.
 *   [COUPLING] tginsight AIexTime post 185 ("Coupling without Communication
 *              and Drafter-Invariant Speculative Decoding"): Gumbel-max
 *              sampling; the same noise for drafter and target, so the check
 *              compares two tokens and the output does not depend on the
 *              drafter.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees or keeps them past the call.  bf16 tensors are raw
 *     __nv_bfloat16 storage; every layout is dense row-major as stated.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work: they return before the GPU has run it.
 *   - Arguments are validated on the host before anything is enqueued; a
 *     rejected call returns a non-zero biv_status and launches nothing.  A
 *     zero-sized problem (rows == 0 etc.) returns BIV_OK and launches nothing.
 *   - Device-side checks (indices read from device memory: slots, positions,
 *     token ids; bounded waits inside kernels) cannot be seen by the host at
 *     call time.  They skip the offending row and set a bit in the library's
 *     device error word, read with biv_device_error().
 *   - Inputs are never modified, except the caches of biv_kv_overwrite and the
 *     caller-provided workspace of biv_decode_attn_fixedsplit.
 *   - Kernels launch with programmatic dependent launch: a kernel may start
 *     while the previous libbiv kernel on the same stream is finishing, and
 *     waits for it before reading that kernel's outputs.  A few inputs that
 *     are never a step's intermediate results are read before that wait:
 *     GEMM weights (B operands), the row_slot / row_pos arrays of attention
 *     and the cache rows of each attention row group below the group's
 *     smallest position (the requests' committed context).  They must not be
 *     written by the immediately preceding libbiv kernel on the stream
 *     (kernels of other libraries, and copies, are waited for in full).
 *   - No call allocates device memory.  The exceptions in kind are part of
 *     the loaded module and held until the process exits: the fixed scratch
 *     array behind biv_decode_attn_fixedsplit_noalloc
 *     (BIV_NOALLOC_SCRATCH_BYTES per GPU) and the 512-byte ring of row
 *     counters of the streaming selection (64 slots, each reset to zero by
 *     the call that used it).
 */
#ifndef BIV_H_
#define BIV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* biv_stream_t; /* identical to cudaStream_t */

typedef enum biv_status {
    BIV_OK = 0,
    BIV_ERR_NULL = 1,        /* a required pointer is NULL                          */
    BIV_ERR_SHAPE = 2,       /* a size is negative, inconsistent or out of range    */
    BIV_ERR_ALIGN = 3,       /* a pointer or leading dimension breaks 16-B alignment */
    BIV_ERR_VALUE = 4,       /* a scalar is out of its domain (eps, temperature, ...) */
    BIV_ERR_UNSUPPORTED = 5, /* valid, but not built (head dim != 128, split != 256)  */
    BIV_ERR_CUDA = 6,        /* a CUDA runtime call failed; see biv_last_cuda_error() */
    BIV_ERR_DEVICE = 7,      /* no usable sm_100-family device for this call          */
    BIV_ERR_SCRATCH = 8      /* the problem needs more than the fixed no-alloc scratch */
} biv_status;

typedef enum biv_dtype { BIV_BF16 = 0, BIV_F32 = 1 } biv_dtype;

/* Device error word bits (biv_device_error). */
#define BIV_DEVERR_TIMEOUT 1u /* a bounded wait inside a kernel ran out; the kernel returned */
#define BIV_DEVERR_INDEX 2u   /* a slot / position / token id read from device memory was out of range */
#define BIV_DEVERR_GROUP 4u   /* rows declared to share a cache slot did not */

/* Build constants. */
#define BIV_KV_SPLIT 256      /* fixed KV split of the decode attention ([DVR] para 1) */
#define BIV_HEAD_DIM 128      /* attention head dimension built */
#define BIV_ATTN_TILE 128     /* rows of one attention MMA tile ([GUIDE] GQA tile rule) */

/* ------------------------------------------------------------- status */
const char* biv_status_string(int status);           /* static string, never NULL */
int biv_last_cuda_error(void);                        /* thread-local cudaError_t of the last BIV_ERR_CUDA */
int biv_version(void);                                /* 100 * major + minor */

/* Synchronises the device, then returns (and clears) the OR of all device
 * error bits raised since the last call.  Returns BIV_ERR_CUDA if the
 * synchronisation failed.  Not for the hot path. */
int biv_device_error(uint32_t* bits_out);

/* Self-test of the device-side failure detection: launches one kernel in
 * which a thread waits, through the same bounded wait every pipeline of the
 * library uses, on a barrier that nothing completes.  After the wait's limit
 * (about 2 s) it gives up, raises BIV_DEVERR_TIMEOUT and returns; the next
 * biv_device_error() reports the bit and the context stays usable.  Nothing
 * traps, faults or spins without bound.  Not for the hot path. */
int biv_selftest_wait_timeout(biv_stream_t stream);

/* --------------------------------------------------------- RMSNorm
 * [DVR] para 1: RMSNorm with a fixed split over the hidden dimension that
 * does not depend on the batch or on how many SMs are busy.
 *   y[r][i] = bf16( x[r][i] * rsqrt(mean_i x[r][i]^2 + eps) * w[i] )
 * x, y: bf16 [rows, d]; w: bf16 [d].  fp32 accumulation in a fixed order
 * (each thread owns fixed 8-element chunks; a fixed xor-butterfly inside the
 * warp, then a fixed tree across warps), identical for every row count.
 * Requires d % 8 == 0, 8 <= d <= 16384, eps > 0 finite, 16-B aligned pointers.
 * y may alias x.                                                          */
int biv_rmsnorm(const void* x, const void* w, void* y, int rows, int d, float eps,
                biv_stream_t stream);

/* --------------------------------------------------- no-split-K GEMM
 * [DVR] para 1: a matmul that never splits K and always uses the same
 * data-parallel tiling.
 *   C[m][n] = sum_k A[m][k] * B[n][k]        (fp32 accumulation)
 * A: bf16 [M, K] row-major; B: bf16 [N, K] row-major (nn.Linear weight);
 * C: [M, N] row-major, bf16 (round-to-nearest-even) or fp32 per out_dtype.
 * tcgen05 tensor-core MMAs (M tile 128, K step 16) accumulate in TMEM; each
 * output tile's K loop runs in one CTA in increasing k, so every element's
 * accumulation order is fixed and independent of M, of the tile width and of
 * the row's position inside the tile (outputs are bitwise identical for any
 * M; tests check this).  Launched with programmatic dependent launch.
 * Requires M >= 0, N % 8 == 0, K % 8 == 0, K > 0, N > 0, 16-B aligned pointers.
 * C must not overlap A or B.                                              */
int biv_gemm_nosplitk(const void* A, const void* B, void* C, int out_dtype, int M, int N, int K,
                      biv_stream_t stream);

/* Same GEMM with the N-tile width forced (a multiple of 16 in [16, 256])
 * instead of chosen by biv_gemm_tile_n.  For tests of tile-width
 * independence and for tuning; results are bitwise identical to
 * biv_gemm_nosplitk's.                                                    */
int biv_gemm_nosplitk_bn(const void* A, const void* B, void* C, int out_dtype, int M, int N, int K,
                         int bn, biv_stream_t stream);

/* The N-tile width biv_gemm_nosplitk uses: with one row tile (M <= 128) the
 * widest tile that keeps the N tiles within one wave of 152 CTAs; otherwise
 * the width in [64, 256] that best fills whole waves (mildly preferring wide
 * tiles).  Only the work split depends on it, never an element's arithmetic. */
int biv_gemm_tile_n(int M, int N, int K);

/* ------------------------------------------- fixed-split decode attention
 * [DVR] para 1: attention with a fixed KV-split size that never adapts to the
 * sequence length or the GPU load.  [GUIDE] GQA tile rule: the G = Hq/Hkv
 * query heads sharing a KV head, times the verified rows of one request, are
 * packed into one 128-row MMA tile.
 * For each row w (cache slot s = row_slot[w], position p = row_pos[w]) and
 * query head h (KV head h / (Hq/Hkv)):
 *   o[w][h] = sum_{j<=p} softmax_j(q[w][h] . k[s][kvh][j] / sqrt(hd)) v[s][kvh][j]
 * Keys are split at absolute multiples of BIV_KV_SPLIT; each split yields a
 * partial (max, sum, unnormalised output) in fp32 and the splits of a row are
 * combined in increasing split order.  A row's result depends only on its own
 * q, its slot's cache and its position.
 * q, o: bf16 [W, Hq, hd]; k_cache, v_cache: bf16 [n_slots, Hkv, max_len, hd].
 * Rows [g*rows_per_group, (g+1)*rows_per_group) must share one cache slot (the
 * K rows of one request in a W = N*K window, [DVR] para 4); rows_per_group = 1
 * is always valid.  Positions must be < max_len and every cache row
 * j <= p must hold finite values.
 * workspace: device memory of at least biv_decode_attn_workspace_size(W, Hq,
 * max_len) bytes, 16-B aligned, contents ignored on entry.
 * Requires hd == 128, kv_split == 256, Hq % Hkv == 0, Hq/Hkv <= 128.        */
size_t biv_decode_attn_workspace_size(int W, int Hq, int max_len);
int biv_decode_attn_fixedsplit(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* row_slot, const int32_t* row_pos, void* o, int W,
                               int rows_per_group, int Hq, int Hkv, int hd, int n_slots,
                               int max_len, int kv_split, void* workspace, size_t ws_bytes,
                               biv_stream_t stream);

/* Largest number of drafts D with G * (1 + D) <= tile ([GUIDE] GQA tile rule:
 * D = tile / G - 1).  Returns -1 when G <= 0 or G > tile.                  */
int biv_gqa_max_drafts(int G, int tile);

/* Bytes of the scratch array that biv_decode_attn_fixedsplit_noalloc uses. */
#define BIV_NOALLOC_SCRATCH_BYTES (16u << 20)

/* The same attention as biv_decode_attn_fixedsplit, for callers that cannot
 * allocate device memory: code that runs where cudaMalloc is unavailable or
 * forbidden (inside a memory-pool-managed runtime that owns every device
 * allocation, a plugin with no allocator handle, or a step that must not
 * touch the allocator mid-run).  The pages have no counterpart; this is a
 * convenience of the library.
 * Instead of a caller workspace it uses one file-scope device array of
 * BIV_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU loading the library holds
 * until the process exits.  Problems whose workspace
 * (biv_decode_attn_workspace_size) exceeds that return BIV_ERR_SCRATCH and
 * launch nothing.  The first call on each device looks up the array's device
 * address (with that device current), so make that first call before any
 * stream capture.  The address is kept for the life of the process: it
 * assumes the device's primary context outlives every call (after a
 * cudaDeviceReset the kept address is stale; do not call this entry point
 * again in that process).  All calls share the one array and it keeps the last
 * call's contents (nothing in it has to start at zero: every partial is
 * written before it is read); calls whose kernels overlap on the GPU -- on
 * different streams, or from different threads -- race on it.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.  Other arguments and
 * results are exactly those of biv_decode_attn_fixedsplit.              */
int biv_decode_attn_fixedsplit_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* row_slot, const int32_t* row_pos, void* o,
                                       int W, int rows_per_group, int Hq, int Hkv, int hd,
                                       int n_slots, int max_len, int kv_split,
                                       biv_stream_t stream);

/* ------------------------------------------------------ KV overwrite
 * [DVR] para 3: at each verification the fast path's cache rows are
 * overwritten by the verifier's values.  Row w = r*K + j of the window writes
 * k_new[w] and v_new[w] (bf16 [Hkv, hd] each; consecutive rows k_stride and
 * v_stride elements apart) into its slot at position row_pos[w].  If
 * rows_keep (int32 [N], N = W / K) is not NULL, only rows j < rows_keep[r]
 * are written.  Rows with an out-of-range slot or position are skipped and
 * raise BIV_DEVERR_INDEX.
 * Requires hd % 8 == 0, strides % 8 == 0 and >= Hkv*hd, W % K == 0,
 * 16-B aligned pointers.                                                  */
int biv_kv_overwrite(void* k_cache, void* v_cache, const void* k_new, long long k_stride,
                     const void* v_new, long long v_stride, const int32_t* row_slot,
                     const int32_t* row_pos, const int32_t* rows_keep, int W, int K, int Hkv, int hd,
                     int n_slots, int max_len, biv_stream_t stream);

/* RoPE and KV overwrite in one pass: q heads of qkv (bf16 [W, (Hq + 2 Hkv) hd])
 * are rotated into q_out (bf16 [W, Hq, hd]); k heads are rotated and written,
 * with the v heads, into the caches at (row_slot[w], row_pos[w]).  Bitwise the
 * same as biv_rope_qk followed by biv_kv_overwrite (same rows_keep rule).
 * Requires hd % 8 == 0, hd <= 256, theta > 1, W % K == 0, aligned pointers. */
int biv_rope_kv_write(const void* qkv, void* q_out, void* k_cache, void* v_cache,
                      const int32_t* row_slot, const int32_t* row_pos, const int32_t* rows_keep, int W,
                      int K, int Hq, int Hkv, int hd, int n_slots, int max_len, float theta,
                      biv_stream_t stream);

/* QKV projection with RoPE and the KV overwrite in its epilogue: bitwise the
 * same as biv_gemm_nosplitk(A, W_qkv) into a bf16 buffer followed by
 * biv_rope_kv_write (same rows_keep rule, same index checks), without the
 * round trip of the projection through memory.  B_packed is W_qkv
 * ([(Hq + 2 Hkv) hd, d] nn.Linear layout) rearranged once by
 * biv_rope_pack_qkv_weights so that each 16 output columns of the q and k
 * part hold 8 rotation pairs of one head.  A: bf16 [W, d]; q_out: bf16 [W, Hq, hd]; caches:
 * bf16 [n_slots, Hkv, max_len, hd]; qkv_out: optional bf16 [W, (Hq+2Hkv) hd]
 * receiving the unrotated projection in the original column order (NULL to
 * skip).  Requires hd % 16 == 0, hd <= 256, d % 8 == 0, Hq % Hkv == 0,
 * W % K == 0, theta > 1 finite, 16-B aligned pointers.                    */
int biv_gemm_qkv_rope(const void* A, const void* B_packed, void* q_out, void* k_cache, void* v_cache,
                      void* qkv_out, const int32_t* row_slot, const int32_t* row_pos, const int32_t* rows_keep,
                      int W, int K, int d, int Hq, int Hkv, int hd, int n_slots, int max_len, float theta,
                      biv_stream_t stream);

/* Rearrange W_qkv (bf16 [(Hq + 2 Hkv) hd, K]) for biv_gemm_qkv_rope: the
 * q and k rows (heads h = 0 .. Hq + Hkv - 1, q heads first) are packed as
 * [g][h][16] for frequency groups g = 0 .. hd/16 - 1: packed rows e = 0..7 of
 * (g, h) are head h's dims 8 g + e, rows e = 8..15 its dims hd/2 + 8 g + e - 8;
 * v rows unchanged.  w_packed must not alias w_qkv.                       */
int biv_rope_pack_qkv_weights(const void* w_qkv, void* w_packed, int Hq, int Hkv, int hd, int K,
                              biv_stream_t stream);

/* ----------------------------------------------------- Gumbel-max select
 * [COUPLING]: adding Gumbel(0,1) noise to the logits and taking the argmax
 * samples from softmax(logits / T) without computing a softmax; the noise does
 * not depend on the logits.  Row r selects the token at position
 * row_pos[r] + 1 of request row_req[r]:
 *   w_v   = word (v & 3) of Philox4x32-10(counter = (v >> 2, row_pos[r] + 1,
 *           row_req[r], 0), key = (seed & 0xffffffff, seed >> 32))
 *   u_v   = (2 * (w_v >> 9) + 1) * 2^-24
 *   g_v   = -L(-L(u_v)), L = the library's fp32 log (IEEE +,-,*,/,fma only)
 *   key_v = fl(fl(logit_v * fl(1/T)) + g_v)
 *   tokens[r] = the v with the largest key; the lowest v among equal keys;
 *               a NaN key never beats a number.  T == 0 selects the largest
 *               logit (lowest index on ties).
 * The noise is a pure function of (seed, request, position, v), so the same
 * token is selected at any batch size, with or without a drafter.
 * logits: fp32 [R, ld] (first V columns used); row_req: uint32 [R];
 * row_pos: int32 [R]; tokens: int32 [R].  Requires V % 4 == 0, ld % 4 == 0,
 * ld >= V, 4 <= V <= 2^22 (BIV_ERR_UNSUPPORTED above), T >= 0 finite, 16-B
 * aligned logits.  Two or more rows per SM are streamed one row per CTA
 * (rows dealt out by a counter of the library's; up to 64 such calls may
 * run at the same time); fewer rows are shared by eight-CTA clusters; both
 * give the same tokens.  Allocates nothing.                              */
int biv_gumbel_argmax(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                      const int32_t* row_pos, uint64_t seed, float temperature, int32_t* tokens,
                      biv_stream_t stream);

/* biv_gumbel_argmax with a workspace: when rows are streamed and T > 0, rows
 * on which many entries can still win (flat rows: more than a quarter of
 * their 256-logit blocks can reach the first exact key; up to R/8 of them,
 * the rest as in biv_gumbel_argmax) are not finished by the CTA that
 * streamed them but handed, as one unit per 8192-logit chunk, to a second
 * kernel that runs over all SMs after the first.  Same tokens, bit for bit.
 * workspace: device memory of at least biv_gumbel_argmax_workspace_size(R,
 * V) bytes (R/8 * (2 ceil(V/256) + 16 ceil(V/8192) + 16) + 64, about), 16-B
 * aligned, owned by the caller, contents ignored on entry; one call at a
 * time per workspace.  Errors as biv_gumbel_argmax, plus BIV_ERR_NULL /
 * BIV_ERR_ALIGN / BIV_ERR_SHAPE for a missing, misaligned or short
 * workspace (R > 0).                                                     */
size_t biv_gumbel_argmax_workspace_size(int R, int V);
int biv_gumbel_argmax_ws(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                         const int32_t* row_pos, uint64_t seed, float temperature, int32_t* tokens,
                         void* workspace, size_t ws_bytes, biv_stream_t stream);

/* The noise g_v of biv_gumbel_argmax for v in [0, V) of each row (fp32
 * [R, V]); for tests of the noise itself.                                  */
int biv_gumbel_noise(uint64_t seed, const uint32_t* row_req, const int32_t* row_pos, int R, int V,
                     float* g, biv_stream_t stream);

/* g = -L(-L(u(w))) for raw 32-bit words w[0..n); for tests of L.           */
int biv_gumbel_from_words(const uint32_t* words, long long n, float* g, biv_stream_t stream);

/* The 256 per-bucket noise bounds biv_gumbel_argmax prunes with (host memory,
 * float[256]): every noise value whose word has top byte b is <= bounds[b].
 * For tests of the pruning bound.                                         */
int biv_gumbel_bucket_bounds(float* bounds_out);

/* LM head with the selection fused into its epilogue ([COUPLING]: the noise
 * does not depend on the logits, so it can be applied where the logits are
 * made).  tokens[r] is bit-identical to biv_gemm_nosplitk(A, B, C, BIV_F32,
 * M, N, K) followed by biv_gumbel_argmax(C, M, N, N, row_req, row_pos, seed,
 * temperature, tokens): the keys are formed from the same fp32 accumulators.
 * Each CTA selects the winner of every row of its output tile from TMEM and
 * writes it (a 64-bit packed key) to the workspace; a second kernel takes the
 * largest per row.  The fp32 logits are stored only if `logits` is non-NULL.
 *   A: bf16 [M, K] row-major; B: bf16 [N, K] row-major (nn.Linear weight);
 *   logits: fp32 [M, N] or NULL; row_req, row_pos, tokens: [M] as in
 *   biv_gumbel_argmax; workspace: device memory of at least
 *   biv_lm_head_gumbel_workspace_size(M, N, K) bytes, 16-B aligned, owned by
 *   the caller and overwritten.
 * Requires N % 8 == 0, K % 8 == 0, T >= 0 finite, 16-B aligned A, B, logits.
 * Errors: BIV_ERR_SHAPE (also for a workspace that is too small),
 * BIV_ERR_VALUE, BIV_ERR_NULL, BIV_ERR_ALIGN; nothing is launched then.   */
size_t biv_lm_head_gumbel_workspace_size(int M, int N, int K);
int biv_lm_head_gumbel(const void* A, const void* B, float* logits, int M, int N, int K,
                       const uint32_t* row_req, const int32_t* row_pos, uint64_t seed, float temperature,
                       int32_t* tokens, void* workspace, size_t ws_bytes, biv_stream_t stream);

/* biv_lm_head_gumbel followed by biv_verify_accept in one launch less: the
 * per-row winners and the coupled accept of each request are taken by one
 * small kernel.  M = n_req * rows_per_req rows, request r owning rows
 * [r*K, (r+1)*K) with K = rows_per_req; draft, p0, accept_len, new_len as in
 * biv_verify_accept.  tokens, accept_len and new_len are bit-identical to the
 * two calls.  Requires what both calls require.                           */
int biv_lm_head_gumbel_accept(const void* A, const void* B, float* logits, int M, int N, int K,
                              const uint32_t* row_req, const int32_t* row_pos, uint64_t seed, float temperature,
                              int32_t* tokens, const int32_t* draft, const int32_t* p0, int n_req,
                              int rows_per_req, int32_t* accept_len, int32_t* new_len, void* workspace,
                              size_t ws_bytes, biv_stream_t stream);

/* Gumbel top-k ([COUPLING]: the trick gives top-k sampling as it stands;
 * Kool, van Hoof & Welling, "Stochastic Beams and Where to Find Them"):
 * out[r * k + j] = the entry with the (j+1)-th largest key of row r, keys and
 * order exactly as biv_gumbel_argmax (so column 0 is its token); the k
 * entries are k draws without replacement from softmax(logits / T).
 * logits: fp32 [R, ld]; row_req, row_pos: [R]; out: int32 [R, k].
 * Requires 1 <= k <= min(64, V), V % 4 == 0, ld % 4 == 0, ld >= V,
 * T >= 0 finite, 16-B aligned logits; otherwise BIV_ERR_SHAPE /
 * BIV_ERR_VALUE / BIV_ERR_NULL / BIV_ERR_ALIGN and nothing is launched.   */
int biv_gumbel_topk(const float* logits, int R, int V, long long ld, const uint32_t* row_req,
                    const int32_t* row_pos, uint64_t seed, float temperature, int k, int32_t* out,
                    biv_stream_t stream);

/* ----------------------------------------------------- n-gram drafter
 * Training-free n-gram lookup drafter ([GUIDE]: a drafting method that finds
 * and copies repeated fragments of the earlier text).  For request r with
 * committed history hist[r * ld + 0 .. len[r]): the longest n in
 * [n_min, n_max] whose last-n-token suffix occurs earlier with at least one
 * token after it, at its most recent such occurrence p; the drafts copy the
 * tokens from s = p + n on, continuing from the drafts themselves once the
 * copy reaches the end of the history (LZ77-style), so periodic text is
 * continued exactly.  No match: all K drafts are the last token (0 for an
 * empty history).  draft_src[r] = s, or -1.
 * hist: int32 [N, ld]; len: int32 [N] (each in [0, ld], else the device error
 * word gets BIV_DEVERR_INDEX and the length is clamped); drafts: int32
 * [N, K]; draft_src: int32 [N].  Requires 1 <= n_min <= n_max <= 64,
 * 1 <= K <= 1024, ld >= 1.  The drafts never change what a coupled verify
 * step commits, only how many tokens it can accept.                      */
int biv_ngram_draft(const int32_t* hist, int N, long long ld, const int32_t* len, int n_max, int n_min,
                    int K, int32_t* drafts, int32_t* draft_src, biv_stream_t stream);

/* ----------------------------------------------------- coupled accept
 * [COUPLING] + [GUIDE] + [DVR] para 3: with shared noise the check compares
 * tokens only.  Row j of request r outputs target[r*K + j] = y_{j+1}, and
 * draft[r*K + j] = d_{j+1} is the draft it must match.
 *   accept_len[r] = (first j with y_{j+1} != d_{j+1}) + 1, or K if none
 *   new_len[r]    = p0[r] + accept_len[r]   (rollback point)
 * The emitted tokens are y_1 .. y_{accept_len}: always the target's own.
 * All arrays int32.  Requires N >= 0, K >= 1.                              */
int biv_verify_accept(const int32_t* target, const int32_t* draft, const int32_t* p0, int N, int K,
                      int32_t* accept_len, int32_t* new_len, biv_stream_t stream);

/* --------------------------------------- per-row glue of the decoder layer
 * The pages do not describe the verifier model; these are the standard
 * pre-norm Llama pieces needed to compose one (each row is independent).   */

/* Fused residual add + RMSNorm: x_out = bf16(x + r), y = RMSNorm(x_out) * w,
 * bit-identical to biv_residual_add followed by biv_rmsnorm.  x_out may alias
 * x.  Same requirements as biv_rmsnorm.                                    */
int biv_add_rmsnorm(const void* x, const void* r, const void* w, void* x_out, void* y, int rows, int d,
                    float eps, biv_stream_t stream);

/* Fused embedding gather + RMSNorm: x_out = table[tokens], y = RMSNorm(x_out) * w,
 * bit-identical to biv_embed followed by biv_rmsnorm.                      */
int biv_embed_rmsnorm(const void* table, const int32_t* tokens, const void* w, void* x_out, void* y,
                      int W, int d, int vocab, float eps, biv_stream_t stream);

/* out[w] = table[tokens[w]] ; table bf16 [vocab, d], out bf16 [W, d], d % 8 == 0. */
int biv_embed(const void* table, const int32_t* tokens, void* out, int W, int d, int vocab,
              biv_stream_t stream);

/* Rotate-half RoPE at the rows' positions.  qkv: bf16 [W, (Hq + 2 Hkv) * hd]
 * (q heads, then k heads, then v heads); q_out: bf16 [W, Hq, hd]; k_out:
 * bf16 [W, Hkv, hd].  Pair (i, i + hd/2) rotates by row_pos * theta^(-2i/hd).
 * Requires hd % 2 == 0, hd <= 256, theta > 1.                              */
int biv_rope_qk(const void* qkv, void* q_out, void* k_out, const int32_t* row_pos, int W, int Hq,
                int Hkv, int hd, float theta, biv_stream_t stream);

/* out[r][i] = bf16(silu(gu[r][i]) * gu[r][F + i]) ; gu bf16 [rows, 2F], F % 8 == 0. */

int biv_silu_mul(const void* gu, void* out, int rows, int F, biv_stream_t stream);

/* Gate/up GEMM with SwiGLU in the epilogue: act[m][i] = bf16(silu(bf16(g)) *
 * bf16(u)) with g = A[m]·Wg[i], u = A[m]·Wu[i]; bitwise the same as
 * biv_gemm_nosplitk (bf16 out) on the stacked weight followed by
 * biv_silu_mul.  B_packed is the [2F, K] weight rearranged by
 * biv_swiglu_pack_weights; act bf16 [M, F].  F % 16 == 0, K % 8 == 0.      */
int biv_gemm_swiglu(const void* A, const void* B_packed, void* act, int M, int F, int K,
                    biv_stream_t stream);

/* Rearrange a stacked gate/up weight ([2F, K], the F gate rows first) into the
 * layout biv_gemm_swiglu reads: blocks of 32 rows, 16 gate rows then the same
 * 16 up rows.  w_packed must not overlap w_gu.                             */
int biv_swiglu_pack_weights(const void* w_gu, void* w_packed, int F, int K, biv_stream_t stream);

/* out[i] = bf16(x[i] + y[i]) over n bf16 elements, n % 8 == 0; out may alias x. */
int biv_residual_add(const void* x, const void* y, void* out, long long n, biv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BIV_H_ */
