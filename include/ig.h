/*
 * ig.h — C ABI of the GB300 (sm_103a) InfiniGen decode hot path.
 *
 * InfiniGen ("InfiniGen: Efficient Generative Inference of Large Language Models with
 * Dynamic KV Cache Management", OSDI 2024) speculates, one layer ahead, which keys and
 * values the next attention layer needs, and fetches only those from a KV pool in host
 * memory.  Citations below name the paper-graph summary page of that paper and the part of
 * its section 3.4 ("Detailed, Sentence-Based Technical Breakdown") that defines each call.
 *
 * Conventions (every function):
 *   - Returns ig_status: IG_OK (0) or a negative error.  ig_last_error() gives a message
 *     for the calling thread.  Nothing aborts the process or traps the GPU.
 *   - "dev" pointers are device memory (or, where stated, host memory the GPU can map);
 *     "host" pointers are ordinary host memory.  The caller owns every buffer it passes.
 *     The library owns only the KV pool (ig_pool_create / ig_pool_destroy): its pinned host
 *     rows and, for a quantized pool, the device-memory array of the rows' scales.
 *   - Device calls are asynchronous on the caller's cudaStream_t, passed as void* (NULL =
 *     legacy default stream).  Argument and launch errors are returned at once; a guard
 *     that trips inside a kernel (an index out of range, a bounded wait that ran out) is
 *     recorded in a device error word that ig_check() reads and clears.
 *   - fp16 tensors are passed as uint16_t bit patterns; fp32 as float; indices as int32_t.
 *   - All multi-dimensional arrays are dense, row-major, in the order written ([B][H][k]
 *     means the last index is contiguous).
 *   - No CPU fallback: with no usable GPU, device calls return IG_ERR_CUDA.
 */
#ifndef IG_H_
#define IG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int ig_status;

#define IG_OK 0
#define IG_ERR_INVALID (-1)   /* bad argument: sizes, alignment, null pointer, alpha <= 0 ... */
#define IG_ERR_CUDA (-2)      /* a CUDA runtime call or a launch failed                       */
#define IG_ERR_OOM (-3)       /* pinned host allocation failed                                */
#define IG_ERR_NUMERIC (-4)   /* the offline SVD did not converge                              */
#define IG_ERR_TIMEOUT (-5)   /* a bounded in-kernel wait ran out (reported by ig_check)       */
#define IG_ERR_CAPACITY (-6)  /* workspace or pool too small for the request                   */

/* Selection policies for ig_select. */
#define IG_SEL_THRESHOLD 0    /* each head keeps {t : s_t > max(s) - alpha}                   */
#define IG_SEL_HEAD_AVG 1     /* each head keeps its top-cbar, cbar = mean count over heads    */
#define IG_SEL_NORMALIZED 2   /* each head keeps {t : max(s) - s_t < alpha * sigma} and the ties
                                 of the maximum; sigma = population std of the head's resident
                                 scores (the portable threshold alpha' = alpha / sigma proposed
                                 as follow-up work; ig_select only)                            */

/* Device error-word bits (ig_check maps them to a status). */
#define IG_DEVERR_INDEX 1     /* an index or count was out of range; the access was skipped  */
#define IG_DEVERR_TIMEOUT 2   /* a bounded wait on a copy ran out                              */

/* Last error message of the calling thread ("" if none). */
const char* ig_last_error(void);

/* ABI version (major * 100 + minor). */
int ig_version(void);

/* Waits for `stream`, then reads and clears the device error word of the current device.
 * Returns IG_OK, IG_ERR_INVALID (an index guard tripped), IG_ERR_TIMEOUT, or IG_ERR_CUDA. */
ig_status ig_check(void* stream);

/* Iteration limit of the score kernels' bounded waits for their staged copies (k2_scores,
 * k23_score_select) on the current device: a wait that runs out records IG_DEVERR_TIMEOUT,
 * the CTA then waits (with the fixed default limit) for its copies in flight to land and
 * leaves without scoring, and the next ig_check returns IG_ERR_TIMEOUT.  max_iters < 0
 * restores the default (2^22 probes, far more than a copy needs); 0 makes the first wait give
 * up at once, which is how tests exercise the timeout path without faulting anything.
 * Synchronous (a 4-byte copy to the device); not for use during stream capture.  No
 * counterpart in the paper. */
ig_status ig_set_wait_limit(int max_iters);

/* ------------------------------------------------------------------------------------
 * Offline skew and partial-column choice.
 * Section 3.4, "Skewed Partial Weights" (Q = U S V^T, A = V, W~_Q = W_Q A, W~_K = W_K A) and
 * "Prefill Stage", Step 2 (column score = column sums of |W~_Q| plus column sums of |K~|,
 * top-k).  Per head h: Q_h = X_s W_Q,h (rotated by RoPE at positions 0..Ns-1 when
 * rope_theta > 0), A_h = right singular vectors of Q_h in descending singular value
 * (one-sided Jacobi SVD in float64), each column's largest-magnitude entry made positive.
 * k = floor(ratio * d + 0.5).
 *
 *   Xs      host fp16 [Ns][D]            sample attention inputs
 *   Wq, Wk  host fp16 [D][H*d]           unskewed query / key weights (head h = columns h*d..)
 *   Kp      host fp16 [Nk][H][d] or NULL prompt keys in the unskewed basis (post-RoPE for
 *                                        RoPE models); they join the column score
 *   A       host fp32 [H][d][d]   out    skew matrices
 *   Wq_skew host fp16 [D][H*d]    out    W_Q A (rounded once to nearest even); may be NULL
 *   Wk_skew host fp16 [D][H*d]    out    W_K A; may be NULL
 *   Kp_skew host fp16 [Nk][H][d]  out    Kp A; may be NULL (ignored when Kp is NULL)
 *   cols    host int32 [H][k]     out    chosen columns per head, ascending
 *   k_out   host int              out    k
 * Host-only and synchronous; uses up to `threads` host threads (0 = all cores).
 * Errors: IG_ERR_INVALID (d odd with RoPE, ratio outside (0,1], null required pointer),
 *         IG_ERR_NUMERIC (Jacobi sweeps did not converge within 80 sweeps; tests force it
 *         with the environment variable IG_FAULT=svd_noconverge, which allows no sweeps). */
ig_status ig_skew_weights(int D, int H, int d, float ratio, float rope_theta,
                          const uint16_t* Xs, int Ns, const uint16_t* Wq, const uint16_t* Wk,
                          const uint16_t* Kp, int Nk, float* A, uint16_t* Wq_skew,
                          uint16_t* Wk_skew, uint16_t* Kp_skew, int32_t* cols, int* k_out,
                          int threads);

/* The singular values of each head's sample queries Q_h = X_s W_Q,h (RoPE-rotated when
 * rope_theta > 0), descending: sigma host fp32 [H][d] out.  The same SVD as ig_skew_weights
 * (whose A_h are the matching right singular vectors). */
ig_status ig_skew_spectrum(int D, int H, int d, float rope_theta, const uint16_t* Xs, int Ns,
                           const uint16_t* Wq, float* sigma, int threads);

/* A layer's partial width from that spectrum (the per-layer ratio proposed as follow-up work:
 * layers whose singular values decay faster need fewer columns): the smallest k in [1, d]
 * whose captured energy, the mean over heads of sum_{i<k} sigma_i^2 / sum_i sigma_i^2, reaches
 * `energy` (in (0, 1]); heads with no energy count as fully captured.  Host only. */
ig_status ig_ratio_from_spectrum(int H, int d, const float* sigma, float energy, int* k_out);

/* ------------------------------------------------------------------------------------
 * Speculation: partial query projection and speculated scores for layer i, from layer
 * i-1's attention input.  Section 3.4, "Decoding Stage", Step 1 (q~p = x_a^(i-1) W~_Q^p,(i))
 * and Step 2 (SpecScore = q~p (K~p)^T over the N+t resident tokens).
 *
 *   x        dev fp16 [B][D]          attention input of layer i-1
 *   Wq_part  dev fp16 [H*k][D]        partial query weight of layer i, stored transposed: row
 *                                     h*k + c holds the D weights of head h's component c
 *   Kpart    dev fp16 [B][H][k][Lcap] partial key cache of layer i, token index contiguous
 *                                     (16-byte aligned; Lcap a multiple of 8)
 *   L_valid  dev int32 [B]            resident slots per sequence (0 <= L_valid <= Lcap)
 *   scores   dev fp32 [B][H][Lcap] out s[b][h][t] = score_scale * sum_c q~p[c] K~p[c][t]
 *                                     for t < L_valid[b]; -inf for L_valid[b] <= t < Lcap
 *   q_part   dev fp32 [B][H][k] out   the partial query (unscaled), or NULL
 *   workspace dev, >= ig_speculate_workspace_bytes(B, D, H, k) bytes, 256-byte aligned
 * Partial query: fp16 x fp16 products on the tensor cores (tcgen05), fp32 accumulation; scores
 * in fp32.  D must be a multiple of 8; x and Wq_part 16-byte aligned. */
size_t ig_speculate_workspace_bytes(int B, int D, int H, int k);
ig_status ig_speculate(void* stream, int B, int D, int H, int k, int Lcap,
                       const uint16_t* x, const uint16_t* Wq_part, const uint16_t* Kpart,
                       const int32_t* L_valid, float score_scale, float* scores,
                       float* q_part, void* workspace, size_t workspace_bytes);

/* ig_speculate without a workspace argument, for callers that cannot allocate device memory
 * (the paper has no counterpart; this is an interface convenience).  Some embedders hand
 * all device memory to their own allocator up front, so a stray cudaMalloc either fails or
 * breaks their accounting, and some cannot afford the implicit synchronisation an allocation
 * may bring.  Here the projection's split partial sums live in a 4 MiB array inside the
 * library (a file-scope __device__ array, held on every GPU that loads the library until the
 * process exits); nothing is allocated, by this call or by anything it calls.
 *   - Limit: ig_speculate_workspace_bytes(B, D, H, k) must be <= 4 MiB (4194304 bytes), else
 *     IG_ERR_CAPACITY with a message; e.g. B = 16, D = 7168, H * k = 2128 needs 3.8 MB.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     and caches it; make that first call before any stream capture.
 *   - Every call on a device shares the one array and leaves its partial sums there (each call
 *     overwrites all it reads, so nothing needs clearing); calls whose work overlaps on the GPU
 *     (different streams, or other threads) race on it and must be serialised by the caller.
 * Arguments and results are those of ig_speculate. */
ig_status ig_speculate_static(void* stream, int B, int D, int H, int k, int Lcap,
                              const uint16_t* x, const uint16_t* Wq_part, const uint16_t* Kpart,
                              const int32_t* L_valid, float score_scale, float* scores,
                              float* q_part);

/* RoPE models (Llama-2): the skew has to follow the rotary embedding, so the partial query
 * is q~p_h = RoPE_p(x W_Q,h) A_h[:, S_h] (the full per-head query, rotated at the current
 * position, then projected on the chosen skewed columns).
 *   Wq       dev fp16 [H*d][D]   unskewed query weight of layer i, transposed (row h*d + j)
 *   A_cols   dev fp32 [H][d][k]  A_h[:, S_h]
 *   positions dev int32 [B]      position of the current token of each sequence
 * Other arguments as ig_speculate; workspace >= ig_speculate_rope_workspace_bytes(). */
size_t ig_speculate_rope_workspace_bytes(int B, int D, int H, int d, int k);
ig_status ig_speculate_rope(void* stream, int B, int D, int H, int d, int k, int Lcap,
                            const uint16_t* x, const uint16_t* Wq, const float* A_cols,
                            const int32_t* positions, float rope_theta,
                            const uint16_t* Kpart, const int32_t* L_valid, float score_scale,
                            float* scores, float* q_part, void* workspace,
                            size_t workspace_bytes);

/* ------------------------------------------------------------------------------------
 * Selection.  Section 3.4, "Decoding Stage", Step 3 ({t : s_t > max(s) - alpha}, evaluated
 * as max(s) - s_t < alpha in fp32 so the maximum is always kept), Step 4 (multi-head
 * averaging: cbar = max(1, round-half-up(mean_h count_h)), each head then keeps its cbar
 * best) and Step 5 (a head keeps at most round-half-up(cap_frac * L_valid) tokens, the best
 * by score then lower index; cap_frac >= 1 means no cap).  NaN scores are never chosen.
 * policy IG_SEL_NORMALIZED: the threshold is alpha times the head's score standard deviation
 * (computed in fp32 over the resident, non-NaN scores); the cap applies as for the threshold.
 *
 *   scores   dev fp32 [B][H][Lcap]
 *   L_valid  dev int32 [B]
 *   alpha    > 0 (may be +inf)
 *   idx      dev int32 [B][H][Lcap] out  chosen slots, ascending, in idx[b][h][0..cnt)
 *   cnt      dev int32 [B][H] out
 *   used     dev uint8 [B][Lcap] out     1 where any head of b chose slot t; may be NULL
 *   workspace dev, >= ig_select_workspace_bytes(B, H) bytes (HEAD_AVG only; else may be NULL) */
size_t ig_select_workspace_bytes(int B, int H);
ig_status ig_select(void* stream, int B, int H, int Lcap, const float* scores,
                    const int32_t* L_valid, float alpha, int policy, float cap_frac,
                    int32_t* idx, int32_t* cnt, uint8_t* used, void* workspace,
                    size_t workspace_bytes);

/* ------------------------------------------------------------------------------------
 * Fused speculation + threshold selection: ig_speculate followed by ig_select with
 * IG_SEL_THRESHOLD and no cap, with the scores kept on chip.  Section 3.4, "Decoding Stage",
 * Steps 1-3.  Persistent CTAs stream whole heads (two CTAs per SM at the OPT-30B shape): the
 * partial-key rows go through a two-stage ring of bulk copies that runs ahead into the next
 * head, the head's scores stay in shared memory, and each warp compacts a contiguous run of
 * tokens in order.  Identical results to the two calls (same fp32 operations).
 *   Wq        dev fp16 [H*k][D] (rope_theta == 0) or [H*d][D] (RoPE: then A_cols [H][d][k] and
 *             positions [B] are required, as in ig_speculate_rope)
 *   idx, cnt, used   as ig_select (used may be NULL)
 *   scores    dev fp32 [B][H][Lcap] or NULL: the scores, written only when asked for
 *   q_part    dev fp32 [B][H][k] or NULL
 *   workspace >= ig_speculate_select_workspace_bytes(B, D, H, d, k, rope != 0)
 * Lcap must be <= 8192 (the on-chip score row); else IG_ERR_INVALID. */
size_t ig_speculate_select_workspace_bytes(int B, int D, int H, int d, int k, int rope);
ig_status ig_speculate_select(void* stream, int B, int D, int H, int d, int k, int Lcap,
                              const uint16_t* x, const uint16_t* Wq, const float* A_cols,
                              const int32_t* positions, float rope_theta, const uint16_t* Kpart,
                              const int32_t* L_valid, float score_scale, float alpha,
                              int32_t* idx, int32_t* cnt, uint8_t* used, float* scores,
                              float* q_part, void* workspace, size_t workspace_bytes);

/* ------------------------------------------------------------------------------------
 * KV pool in pinned, mapped host memory: one pool per layer and sequence, `cap` slots, each
 * holding the full key and value row of every head (section 3.4, "KV Cache Pool Management
 * Under Memory Pressure").  Keys and values are in the skewed basis.  Layout per layer:
 * K[B][H][cap][d] and V[B][H][cap][d] fp16, 16-byte aligned rows.  Each slot has an 8-bit
 * access counter used by ig_pool_evict. */
typedef struct ig_pool ig_pool;

/* Victim policies (section 3.4, pool management, and the three policies of Table 2).
 * Ties always go to the oldest insertion, then the lowest slot.
 *   IG_POOL_COUNTER  smallest 8-bit use counter (the policy InfiniGen uses; the default)
 *   IG_POOL_FIFO     oldest insertion
 *   IG_POOL_LRU      oldest last use by any head; a new entry counts as used when it is
 *                    inserted, and each folded step advances the pool's time by one */
#define IG_POOL_COUNTER 0
#define IG_POOL_FIFO 1
#define IG_POOL_LRU 2
/* ig_pool_create_ex flags.  IG_POOL_NO_STORAGE: the slot manager alone (no pinned K/V rows,
 * H and d ignored; needs no GPU), for host-side simulation of a policy; the calls that move
 * rows (ig_pool_kv, ig_pool_write, ig_gather_kv, ig_gather_attend, ig_append_kv with this
 * pool) then return IG_ERR_INVALID. */
#define IG_POOL_NO_STORAGE 1
/* IG_POOL_FP8: each (token, head) row stored as one record of 2d bytes of codes in the pinned
 * pool, the key's d e4m3 codes then the value's d codes, and the row's two fp32 scales (key,
 * value) in a device-memory array the pool allocates on the device current at creation (the
 * combination of a quantized pool with selective prefetch proposed as follow-up work).  A
 * record is whole 128-byte lines (256 bytes at d = 128), so each fetched row is two full lines
 * over the host link; the 8 bytes of scales per row stay resident in HBM (0.7 GB at the
 * OPT-30B shape).  Each row is quantized on its way in (ig_pool_write, ig_append_kv): scale =
 * amax / 448, codes = round-to-nearest-even e4m3 of x * (448 / amax) in fp32, saturating; a
 * row of zeros has scale 0.  ig_gather_kv reads one record per selected row and its scales
 * and dequantizes (code value x scale, rounded to fp16) into the usual fp16 staging rows, so
 * the link carries 2d bytes per row instead of 4d; the partial key cache (speculation) stays
 * fp16.  d must be 64 or 128; the pool's kernels must run on the device that holds its scales
 * (else IG_ERR_INVALID); ig_pool_kv and the prefill refuse quantized pools (use ig_pool_kv8). */
#define IG_POOL_FP8 2
/* IG_POOL_INT4: the same split with signed 4-bit codes (the format the follow-up work names):
 * a record of d / 2 bytes of key codes then d / 2 of value codes (d bytes: one 128-byte line at
 * d = 128) in the pinned pool, the two fp32 scales in device memory.  scale = amax / 7, codes =
 * the nearest integer (ties to even) of x * (7 / amax) in fp32, in [-7, 7], two per byte with
 * element 2j in the low nibble of byte j (two's complement); a row of zeros has scale 0.  The
 * gather dequantizes as for IG_POOL_FP8; the link carries d bytes per row.  Excludes
 * IG_POOL_FP8; d must be 64 or 128. */
#define IG_POOL_INT4 4

ig_status ig_pool_create(int layers, int B, int H, int d, int cap, ig_pool** out);
/* ig_pool_create with a victim policy (IG_POOL_COUNTER/FIFO/LRU) and flags (0, IG_POOL_NO_STORAGE,
 * IG_POOL_FP8 or IG_POOL_INT4). */
ig_status ig_pool_create_ex(int layers, int B, int H, int d, int cap, int policy, int flags,
                            ig_pool** out);
ig_status ig_pool_destroy(ig_pool* pool);

/* Host pointers (also valid on the device) to one layer's K and V arrays. */
ig_status ig_pool_kv(const ig_pool* pool, int layer, uint16_t** K, uint16_t** V);

/* Quantized (fp8 or int4) pools: host pointer (also valid on the device) to one layer's code
 * records [B][H][cap][record_bytes] (layouts under IG_POOL_FP8 and IG_POOL_INT4), the record
 * size (2d or d), and (when scales is not NULL) the device pointer to that layer's scales
 * [B][H][cap][2] fp32 (key, value). */
ig_status ig_pool_kv8(const ig_pool* pool, int layer, uint8_t** records, int* record_bytes,
                      float** scales);
/* Copies one layer's scales of a quantized pool to host memory out [B][H][cap][2] fp32
 * (synchronous). */
ig_status ig_pool_read_scales(const ig_pool* pool, int layer, float* out);

/* Copies one layer's K and V ([B][H][cap][d] fp16 each, from device or host memory) into
 * the pool, asynchronously on `stream`.  A quantized pool quantizes them in a kernel, so for it
 * the source must be device memory or pinned host memory. */
ig_status ig_pool_write(ig_pool* pool, void* stream, int layer, const uint16_t* K,
                        const uint16_t* V);

/* Host-side pool manager for one (layer, sequence), run once per decode step.  Section 3.4,
 * pool management (counter policy of Table 2): every slot that any head chose this step
 * (used[slot] != 0) gains 1, saturating at 255; when a counter reaches 255 all counters of
 * that pool are halved; the slot's last-use time becomes the current step (for LRU).  Then
 * the new token gets a slot: the next free slot while the pool is not full, otherwise the
 * victim of the pool's policy (the smallest counter by default; see IG_POOL_*).  The new
 * slot's counter starts at 0.
 *   used      host uint8 [cap] or NULL (no use to record, e.g. during prefill)
 *   slot_out  host int32: the slot the new token must be written to (ig_append_kv)
 *   filled_out host int32 or NULL: resident slots after the insertion */
ig_status ig_pool_evict(ig_pool* pool, int layer, int b, const uint8_t* used,
                        int32_t* slot_out, int32_t* filled_out);

/* Reads one (layer, sequence)'s counters (host uint8 [cap]). */
ig_status ig_pool_counters(const ig_pool* pool, int layer, int b, uint8_t* out);

/* Which token each slot of one (layer, sequence) holds: out host int32 [cap], the token's
 * insertion number (prompt tokens 0..n-1 in prefill order, then one per decode step, so the
 * token's position when every step inserts one token), -1 for a free slot. */
ig_status ig_pool_slot_tokens(const ig_pool* pool, int layer, int b, int32_t* out);

/* Number of placements into a full (layer, sequence) pool so far (host int64). */
ig_status ig_pool_evictions(const ig_pool* pool, int layer, int b, int64_t* out);

/* ------------------------------------------------------------------------------------
 * Gather of the chosen full key/value rows from the host pool into HBM.  Section 3.4,
 * "Decoding Stage", Step 5 (fetch the selected tokens' full keys and values, all d columns,
 * asynchronously and overlapped with layer i-1's compute).  The kernel reads the mapped
 * pinned pool directly (16-byte zero-copy loads over the host link); issue it on a side
 * stream.  max_ctas bounds its grid (0 = library default: a quarter of the SMs, or two CTAs
 * per SM of the stream's own partition after ig_sm_split_create, twice that for a quantized
 * pool) so that it leaves SMs to the compute stream.  Quantized pools (IG_POOL_FP8,
 * IG_POOL_INT4) are dequantized to fp16 here (codes over the link, scales from HBM).
 *   idx, cnt  dev, from ig_select (slots must be < cap)
 *   Kg, Vg    dev fp16 [B][H][Lcap][d] out  rows j < cnt[b][h] = pool rows idx[b][h][j] */
ig_status ig_gather_kv(void* stream, const ig_pool* pool, int layer, int B, int H, int d,
                       int Lcap, const int32_t* idx, const int32_t* cnt, uint16_t* Kg,
                       uint16_t* Vg, int max_ctas);

/* ------------------------------------------------------------------------------------
 * Attention over the gathered rows.  Section 3.4, Inference Controller (softmax(q K^T) V over
 * the prefetched entries only).  o[b][h] = sum_j w_j V_j, w = softmax(scale * q . K_j) over
 * rows j < cnt[b][h] plus, when k_new is given, the current token's own key/value.  fp32
 * online softmax and accumulation.
 *   q            dev fp16 [B][H][d]        query of layer i (skewed basis)
 *   Kg, Vg       dev fp16 [B][H][Lcap][d]  (16-byte aligned)
 *   cnt          dev int32 [B][H]
 *   k_new, v_new dev fp16 [B][H][d] or NULL
 *   out          dev fp32 [B][H][d] out
 *   workspace    dev, >= ig_attend_workspace_bytes(B, H, d, Lcap) bytes, 256-byte aligned
 * d must be 64 or 128. */
size_t ig_attend_workspace_bytes(int B, int H, int d, int Lcap);
ig_status ig_sparse_attend(void* stream, int B, int H, int d, int Lcap, float scale,
                           const uint16_t* q, const uint16_t* Kg, const uint16_t* Vg,
                           const int32_t* cnt, const uint16_t* k_new, const uint16_t* v_new,
                           float* out, void* workspace, size_t workspace_bytes);

/* Layer 0 (speculation starts at layer 1; section 3.4, "Why InfiniGen starts speculation from
 * Layer 1"): dense attention over all L_valid[b] resident rows of an HBM-resident KV
 * K, V [B][H][Lcap][d].  Same kernel and arguments as ig_sparse_attend, with the row count
 * taken per sequence from L_valid [B]. */
ig_status ig_dense_attend(void* stream, int B, int H, int d, int Lcap, float scale,
                          const uint16_t* q, const uint16_t* K, const uint16_t* V,
                          const int32_t* L_valid, const uint16_t* k_new,
                          const uint16_t* v_new, float* out, void* workspace,
                          size_t workspace_bytes);

/* Fused fetch + attention.  The same result as ig_gather_kv followed by ig_sparse_attend,
 * up to fp32 summation order, without staging the rows in HBM: the kernel loads each selected
 * row straight from the pinned pool (16-byte zero-copy loads over the host link) through idx
 * and folds it into a per-head online softmax.  This is the prefetch of section 3.4
 * (Inference Controller) with the copy and the attention that consumes it in one pass; the
 * pages stage the rows in GPU memory first.  A quantized pool (IG_POOL_FP8, IG_POOL_INT4) is
 * read as its code records (each lane its 8 or 4 bytes of codes) with the rows' scales from
 * HBM, dequantized in registers as ig_gather_kv dequantizes them (code value x scale in fp32,
 * rounded to fp16).  Issue it on a side stream; max_ctas bounds the grid (0 = library default:
 * a quarter of the SMs, or two CTAs per SM of the stream's own partition after
 * ig_sm_split_create, twice that for a quantized pool; at most 256).
 *   pool, layer        as for ig_gather_kv (B, H, d must match the pool)
 *   q                  dev fp16 [B][H][d]
 *   idx, cnt           dev, from ig_select (slots must be < the pool's capacity; a slot
 *                      out of range is skipped and raises IG_DEVERR_INDEX)
 *   k_new, v_new       dev fp16 [B][H][d] or NULL (the current token, always attended)
 *   out                dev fp32 [B][H][d] out
 *   workspace          dev, >= ig_gather_attend_workspace_bytes(B, H, d, Lcap) bytes,
 *                      256-byte aligned (per-head partials of the kernel's lane groups)
 * d must be 64 or 128. */
size_t ig_gather_attend_workspace_bytes(int B, int H, int d, int Lcap);
ig_status ig_gather_attend(void* stream, const ig_pool* pool, int layer, int B, int H, int d,
                           int Lcap, float scale, const uint16_t* q, const int32_t* idx,
                           const int32_t* cnt, const uint16_t* k_new, const uint16_t* v_new,
                           float* out, void* workspace, size_t workspace_bytes, int max_ctas);

/* The appends of every layer's current token in one launch (the same rows as ig_append_kv
 * called per layer), for a step whose fetches are done.  Layer 0 goes to Kdense/Vdense when
 * they are given (an HBM-resident layer 0), else to the pool like the others.
 *   ks      host int [layers]: partial width of each layer (0 where Kpart[l] is NULL)
 *   slot    dev int32 [layers][B]: slot per (layer, sequence); negative: skip
 *   cols    host array [layers] of dev int32 [H][ks[l]] (entries may be NULL with Kpart[l])
 *   k_new, v_new  dev fp16 [layers][B][H][d]
 *   Kpart   host array [layers] of dev fp16 [B][H][ks[l]][Lcap] or NULL entries; may be NULL
 * At most 128 layers per call; quantized pools quantize the rows as ig_append_kv does. */
ig_status ig_append_kv_layers(void* stream, ig_pool* pool, int layers, int B, int H, int d,
                              const int* ks, int Lcap, const int32_t* slot,
                              const int32_t* const* cols, const uint16_t* k_new,
                              const uint16_t* v_new, uint16_t* const* Kpart, uint16_t* Kdense,
                              uint16_t* Vdense);

/* ------------------------------------------------------------------------------------
 * Append of the current token.  Section 3.4, "Partial Key Cache Updates During Decoding":
 * the new token's full key and value go to the host pool, its k chosen columns to the
 * partial key cache in HBM, at the slot given by ig_pool_evict.
 *   slot     dev int32 [B]      slot per sequence (negative: skip that sequence)
 *   cols     dev int32 [H][k]   chosen columns
 *   k_new, v_new dev fp16 [B][H][d]
 *   pool     written at (layer, b, h, slot) when not NULL
 *   Kpart    dev fp16 [B][H][k][Lcap] or NULL
 *   Kdense, Vdense dev fp16 [B][H][Lcap][d] or NULL (an HBM-resident KV, as for layer 0) */
ig_status ig_append_kv(void* stream, ig_pool* pool, int layer, int B, int H, int d, int k,
                       int Lcap, const int32_t* slot, const int32_t* cols,
                       const uint16_t* k_new, const uint16_t* v_new, uint16_t* Kpart,
                       uint16_t* Kdense, uint16_t* Vdense);

/* ------------------------------------------------------------------------------------
 * One decode step over every layer (native runtime of the calls above).  Section 3.2
 * (architecture) and section 3.4, "Decoding Stage", Step 5 with Fig 8: while layer i-1
 * attends, layer i is speculated from layer i-1's input and its rows are fetched on a side
 * stream; layer 0 attends over its full, HBM-resident KV.  Order per step, compute stream S,
 * fetch stream G:
 *   for l = 1..L-1:  S: speculate(l), select(l)  ->  G: gather(l) into buffer l % 2
 *                    S: (wait gather(l-1)) attention(l-1), append(l-1)   [l-1 = 0: dense]
 *   S: wait gather(L-1), attention(L-1), append(L-1); S finally waits for G.
 * All buffers belong to the caller; the decoder holds only events.  The per-layer pointer
 * arrays in ig_decoder_buffers are host arrays of device pointers, copied at creation. */
typedef struct {
  int layers, B, H, d, D, k, Lcap;
  int policy;          /* IG_SEL_THRESHOLD, IG_SEL_HEAD_AVG or IG_SEL_NORMALIZED */
  float alpha;         /* > 0 */
  float cap_frac;      /* >= 1: no cap */
  float score_scale;   /* logit scale, e.g. 1/sqrt(d) */
  float rope_theta;    /* 0: no RoPE (partial weight path); > 0: RoPE path */
  int gather_ctas;     /* grid of the fetch kernel; 0 = library default */
  int stage_timing;    /* 1: record timing events around each stage (ig_decoder_stage_ms) */
  int fused_select;    /* 1: use ig_speculate_select when policy = IG_SEL_THRESHOLD, cap_frac >= 1
                          and Lcap <= 8192 (scores stay on chip); 0: separate calls */
  int fused_fetch;     /* 1: layers 1.. attend straight from the pool on the fetch stream
                          (ig_gather_attend's partials; its combine runs on the compute stream),
                          no staging in HBM, Kg/Vg unused (may be NULL); 0: gather into Kg/Vg on
                          the fetch stream, attend on the compute stream */
  int batched_append;  /* 1: every layer's new token is appended in one launch at the end of the
                          step (ig_append_kv_layers), after the fetches; 0: each layer's append
                          follows its attention */
  int append_on_fetch; /* staged fetch, batched_append = 0: 1: layer l >= 1's append runs on the
                          fetch stream right after its gather (spares the compute stream where
                          that is the critical path); 0: on the compute stream after attention */
  int keep_indices;    /* 1: idx is [layers][B][H][Lcap] and every layer's index list outlives the
                          step (for inspection; the kernels and their grids are unchanged);
                          0: idx is [2][B][H][Lcap], reused by layer parity */
} ig_decoder_config;

typedef struct {
  const uint16_t* const* Wq_part;  /* [layers] -> dev fp16 [H*k][D]       (no RoPE)        */
  const uint16_t* const* Wq;       /* [layers] -> dev fp16 [H*d][D]       (RoPE)           */
  const float* const* A_cols;      /* [layers] -> dev fp32 [H][d][k]      (RoPE)           */
  uint16_t* const* Kpart;          /* [layers] -> dev fp16 [B][H][k][Lcap] (layer 0: may be NULL) */
  const int32_t* const* cols;      /* [layers] -> dev int32 [H][k]                          */
  uint16_t* K0;                    /* dev fp16 [B][H][Lcap][d]: layer 0's KV in HBM          */
  uint16_t* V0;
  float* scores;                   /* dev fp32 [B][H][Lcap]                                  */
  int32_t* idx;                    /* dev int32 [2][B][H][Lcap] ([layers][B][H][Lcap] with
                                      config keep_indices)                                   */
  int32_t* cnt;                    /* dev int32 [layers][B][H]                               */
  uint8_t* used;                   /* dev uint8 [layers][B][Lcap] or NULL                    */
  uint16_t* Kg;                    /* dev fp16 [2][B][H][Lcap][d] (16-byte aligned); NULL
                                      allowed with fused_fetch                                */
  uint16_t* Vg;
  void* workspace;                 /* dev, >= ig_decoder_workspace_bytes(), 256-byte aligned */
  size_t workspace_bytes;
  const int* ks;                   /* host int [layers]: each layer's partial width (1..config
                                      k; the arrays above sized with it), or NULL: config k for
                                      every layer (the per-layer ratio of ig_ratio_from_spectrum) */
} ig_decoder_buffers;

typedef struct {
  const uint16_t* x;        /* dev fp16 [layers][B][D]    attention input of every layer       */
  const uint16_t* q;        /* dev fp16 [layers][B][H][d] query of every layer (skewed basis)  */
  const uint16_t* k_new;    /* dev fp16 [layers][B][H][d] current token's key                  */
  const uint16_t* v_new;    /* dev fp16 [layers][B][H][d] current token's value                */
  const int32_t* L_valid;   /* dev int32 [B] resident slots before this step's append          */
  const int32_t* positions; /* dev int32 [B] current position (RoPE only)                     */
  const int32_t* slot;      /* dev int32 [layers][B] append slot per layer, or NULL: no append */
  float* out;               /* dev fp32 [layers][B][H][d] attention output of every layer     */
} ig_step_io;

typedef struct ig_decoder ig_decoder;

size_t ig_decoder_workspace_bytes(const ig_decoder_config* cfg);
ig_status ig_decoder_create(const ig_decoder_config* cfg, const ig_decoder_buffers* buffers,
                            ig_pool* pool, ig_decoder** out);
ig_status ig_decoder_destroy(ig_decoder* dec);
/* Enqueues one step on `stream` (compute) and `side_stream` (fetch); returns at once. */
ig_status ig_decode_step(ig_decoder* dec, const ig_step_io* io, void* stream, void* side_stream);

/* CUDA-graph form of ig_decode_step: captures the whole step (both streams, with the pointers
 * in `io`, which must stay valid and in place) into graphs, so later steps replay it with one
 * launch instead of a few hundred.  Capture once, then per step: update the contents of the io
 * buffers (inputs, L_valid, slots) on `stream`, then ig_decoder_graph_launch.  Capture runs
 * nothing on the GPU; call it after one eager ig_decode_step (which sets kernel attributes).
 * Two graphs are kept when stage timing is on (one per timing-event set).
 * ig_decoder_graph_launch counts the step's kernels in ig_launch_count. */
ig_status ig_decoder_graph_capture(ig_decoder* dec, const ig_step_io* io, void* stream,
                                   void* side_stream);
ig_status ig_decoder_graph_launch(ig_decoder* dec, void* stream);

/* Pool counters only: folds one step's use of (layer, b) into its counters, without placing a
 * token (ig_pool_evict does both).  While the pool is not full the two orders agree, so a
 * runtime may fold use in late, off the critical path. */
ig_status ig_pool_update(ig_pool* pool, int layer, int b, const uint8_t* used);

/* Prefill: inserts n_tokens prompt tokens into every (layer, sequence) pool exactly as
 * n_tokens calls of ig_pool_evict(used = NULL) would (the free slots in order, then, with all
 * counters at 0, the oldest slot first).  slots_out: host int32 [n_tokens] or NULL, the slot
 * of each prompt token (the same for every layer and sequence). */
ig_status ig_pool_prefill(ig_pool* pool, int n_tokens, int32_t* slots_out);

/* One decode step of the pool manager for every (layer, sequence) at once.
 *   used      host uint8 [layers][B][Lcap] (first `cap` entries of each row are read) or NULL
 *   slots_out host int32 [layers][B] or NULL
 * With `used`, folds that step's use into the counters (as ig_pool_update); with `slots_out`,
 * then places the next token (as ig_pool_evict(used = NULL)).  ig_pool_full() tells whether
 * any pool is full, i.e. whether placement depends on the counters. */
ig_status ig_pool_step(ig_pool* pool, const uint8_t* used, int Lcap, int32_t* slots_out);
ig_status ig_pool_full(const ig_pool* pool, int* any_full);

/* Diagnostic of a capacity-limited pool (not a step of the method; section 3.4, pool
 * management): how much of a selection falls on tokens the pool has evicted.  Selection runs
 * over every token seen so far, indexed by token number t (a partial key cache that keeps
 * every token, scored by ig_speculate and selected by ig_select); the pool's slot -> token
 * map (ig_pool_slot_tokens) gives `resident`.  Per (b, h):
 *   miss_cnt  = |{ j < cnt : resident[b][idx_j] == 0 }|
 *   miss_mass = sum over missed j of exp(s_j - m) / sum over all j < cnt of exp(s_j - m),
 *               m = the largest selected score (0 when nothing is selected)
 *   scores    dev fp32 [B][H][Lcap]  by token number
 *   idx, cnt  dev int32 [B][H][Lcap], [B][H]  (token numbers < Lcap; others raise
 *             IG_DEVERR_INDEX and are skipped)
 *   resident  dev uint8 [B][Lcap]
 *   miss_cnt  dev int32 [B][H] out;  miss_mass dev fp32 [B][H] out */
ig_status ig_eviction_misses(void* stream, int B, int H, int Lcap, const float* scores,
                             const int32_t* idx, const int32_t* cnt, const uint8_t* resident,
                             int32_t* miss_cnt, float* miss_mass);

/* Speculation fidelity (diagnostic, not a step of the method; section 3.4, "Decoding Stage",
 * and the skew ablation of Fig 13): how well a speculated set matches the real attention of
 * its layer.  Per (b, h), with the real logits z_t = scale q . K_t over the L_valid[b]
 * resident rows and c = cnt[b][h] speculated tokens idx[b][h][0..c):
 *   recall = |{ j < c : z_{idx_j} >= z_(c) }| / c, z_(c) the c-th largest real logit (ties at
 *            z_(c) count as hits; c is capped at L for the threshold);
 *   weight = sum_{j < c} exp(z_{idx_j} - M) / sum_{t < L} exp(z_t - M), M = max_t z_t
 *            (the share of the real softmax weight the speculated set holds);
 * both 0 when c = 0 or L = 0.
 *   q          dev fp16 [B][H][d]        the layer's real query (16-byte aligned)
 *   K          dev fp16 [B][H][Lcap][d]  its keys (16-byte aligned), HBM
 *   L_valid    dev int32 [B];  idx, cnt dev int32 [B][H][Lcap], [B][H] (from ig_select)
 *   recall, weight  dev fp32 [B][H] out
 * d must be 64 or 128; Lcap <= 16384. */
ig_status ig_attention_recall(void* stream, int B, int H, int d, int Lcap, float scale,
                              const uint16_t* q, const uint16_t* K, const int32_t* L_valid,
                              const int32_t* idx, const int32_t* cnt, float* recall,
                              float* weight);

/* Captured dot-product fraction of a column set (diagnostic; the skew's purpose in section
 * 3.4, "Skewed Partial Weights"): per (b, h),
 *   frac = sum_{t < L} sum_{c in cols[h]} |q_c K_tc| / sum_{t < L} sum_c |q_c K_tc|
 * for a query and keys in any basis (skewed, with the skewed columns, or unskewed, with
 * columns chosen there), so the two can be compared.
 *   q dev fp16 [B][H][d], K dev fp16 [B][H][Lcap][d] (16-byte aligned), L_valid dev int32 [B],
 *   cols dev int32 [H][k], frac dev fp32 [B][H] out.  d must be 64 or 128. */
ig_status ig_captured_fraction(void* stream, int B, int H, int d, int k, int Lcap,
                               const uint16_t* q, const uint16_t* K, const int32_t* L_valid,
                               const int32_t* cols, float* frac);

/* ------------------------------------------------------------------------------------
 * Prefill stage (section 3.4, "Prefill Stage: Partial Weight Index Generation", Steps 1-3;
 * models without RoPE; ig_prefill_layer_rope below for RoPE models).  For one layer and a prompt of N tokens per sequence:
 *   Step 1  K~ = X W~_K and V = X W_V on the tensor cores (fp16 in, fp32 accumulate, fp16
 *           out); the rows of the tokens the pool keeps go to it, token t at slot t mod cap
 *           (the pool's own prefill placement: call ig_pool_prefill(pool, N, ...) for the
 *           slot manager; with N > cap the first N - cap tokens are dropped);
 *   Step 2  cols[h] = the k columns of head h with the largest sum of |W~_Q| over its rows
 *           plus |K~| over every prompt token of every sequence (float64 sums in a fixed
 *           order; ties to the lower column), ascending;
 *   Step 3  Wq_part_t = those rows of W~_Q^T (the partial query weight as ig_speculate takes
 *           it) and Kpart = the chosen columns of the resident keys, at their slots.
 *   X             dev fp16 [B][N][D]         the layer's attention input for the prompt
 *   Wq_t, Wk_t    dev fp16 [H*d][D]          W~_Q^T and W~_K^T (skewed, transposed)
 *   Wv_t          dev fp16 [H*d][D]          W_V^T
 *   cols          dev int32 [H][k] out
 *   Wq_part_t     dev fp16 [H*k][D] out
 *   Kpart         dev fp16 [B][H][k][Lcap] out (resident slots written; others untouched)
 *   workspace     dev, >= ig_prefill_workspace_bytes(B, N, H, d), 256-byte aligned (holds
 *                 K~, 2 B N H d bytes, per-tile column sums and a RoPE table; V goes from the
 *                 GEMM straight to the pool)
 * The pool must have storage and fp16 rows; d must be 64 or 128; D a multiple of 8.
 * V is projected on an internal side stream of the device's primary context (one per device,
 * joined back into `stream` before the call's last work): it runs on the whole device even
 * when `stream` belongs to an SM partition (ig_sm_split_create), so the prefill is not
 * confined by such a stream.  Calls from several host threads are serialised internally. */
size_t ig_prefill_workspace_bytes(int B, int N, int H, int d);
ig_status ig_prefill_layer(void* stream, ig_pool* pool, int layer, int B, int N, int D, int H,
                           int d, int k, int Lcap, const uint16_t* X, const uint16_t* Wq_t,
                           const uint16_t* Wk_t, const uint16_t* Wv_t, int32_t* cols,
                           uint16_t* Wq_part_t, uint16_t* Kpart, void* workspace,
                           size_t workspace_bytes);

/* The prefill of a RoPE model's layer.  The keys are rotated before the skew, so the skew is
 * not in the key weight: K = X W_K (tensor cores, rounded to fp16), then each row of head h
 * becomes K~ = RoPE_t(K_h) A_h (token t of the prompt at position t; angles in float64, the
 * rest in fp32, rounded to fp16).  The columns, the pool rows and the partial key cache as in
 * ig_prefill_layer; instead of a partial weight the decode stage of a RoPE model takes
 * A_cols = A_h[:, cols[h]] (ig_speculate_rope).
 *   Wq_t   dev fp16 [H*d][D]  W~_Q^T = (W_Q A)^T (skewed; it enters the column score only)
 *   Wk_t   dev fp16 [H*d][D]  W_K^T (unskewed);  Wv_t dev fp16 [H*d][D]  W_V^T
 *   A      dev fp32 [H][d][d] the skew matrices (ig_skew_weights)
 *   A_cols dev fp32 [H][d][k] out
 * Workspace: ig_prefill_workspace_bytes(B, N, H, d) (the same query). */
ig_status ig_prefill_layer_rope(void* stream, ig_pool* pool, int layer, int B, int N, int D, int H,
                                int d, int k, int Lcap, float rope_theta, const uint16_t* X,
                                const uint16_t* Wq_t, const uint16_t* Wk_t, const uint16_t* Wv_t,
                                const float* A, int32_t* cols, float* A_cols, uint16_t* Kpart,
                                void* workspace, size_t workspace_bytes);

/* The prefill's tensor-core GEMM on its own: C[M][N] = A[M][K] Bt[N][K]^T, fp16 operands
 * (both K-major), fp32 accumulation, fp16 result (row-major).  With colpart (dev fp32
 * [ceil(M/128)][N]) it also writes, per 128-row tile, the column sums of |C| as stored (fp16).
 * N must be a multiple of 32, K of 8; A, Bt, C 16-byte aligned. */
ig_status ig_gemm_tn(void* stream, int M, int N, int K, const uint16_t* A, const uint16_t* Bt,
                     uint16_t* C, float* colpart);

/* A spatial split of one GPU between two streams: two green contexts over disjoint sets of
 * SMs, each with one stream.  The decode step's host-link fetch (whose loads wait microseconds
 * on the link) and its HBM-bound speculation and attention then never share an SM; sharing
 * them, compute CTAs beside fetch CTAs run slower and hold back kernels that split their work
 * evenly over their CTAs.  fetch_sms is rounded up to the device's partition granularity (8 on
 * sm_90 and later); the compute stream gets the remaining SMs.  On success *compute_stream and
 * *fetch_stream (cudaStream_t, owned by the split; the fetch stream at the highest priority)
 * take work like any stream of the device: pass them to ig_decode_step and the per-stage calls.
 * Kernels launched on them size their grids by their partition (the attention by its SM count;
 * the fetch kernels, by default, two CTAs per fetch SM).  *compute_sms and *fetch_sms_out (may
 * be NULL) receive the sizes.  IG_ERR_CUDA when the driver has no green contexts;
 * IG_ERR_INVALID when the split leaves no SM for the compute stream.  Not part of the method:
 * the InfiniGen paper-graph summary overlaps the prefetch with compute (section 3.2, Fig 8)
 * on a GPU whose copy engine does the transfer. */
typedef struct ig_sm_split ig_sm_split;
ig_status ig_sm_split_create(int device, int fetch_sms, ig_sm_split** out, void** compute_stream,
                             void** fetch_stream, int* compute_sms, int* fetch_sms_out);
/* Destroys the streams and green contexts (after all work on them has finished).  NULL is a no-op. */
ig_status ig_sm_split_destroy(ig_sm_split* split);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t ig_launch_count(void);

/* Stage timing of a recent ig_decode_step (steps_back = 0: the last one, 1: the one before),
 * when the decoder was created with config.stage_timing = 1: ms_out[0] = sum of gather kernel
 * times (fetch stream; with fused_fetch, of fetch + partial attention), ms_out[1] = speculate +
 * select, ms_out[2] = attention + append of layers 1.. (compute stream; with fused_fetch, the
 * combines of the partials and the appends), ms_out[3] = layer 0's dense attention + append; counts_out[0..3] = the
 * number of timed intervals of each (both arrays hold 4 entries).  Waits for that
 * step to finish; reading step t-1 while step t is queued keeps the GPU busy. */
ig_status ig_decoder_stage_ms(ig_decoder* dec, int steps_back, float* ms_out, int* counts_out);

/* The same step's stages as a timeline (a trace of the two streams): t_out (host float
 * [layers][6]) receives, per layer, the device times in ms of the start and end of its fetch
 * (fetch stream), of its speculation + selection and of its attention + append (compute
 * stream; the roles of ig_decoder_stage_ms's intervals), all relative to the start of the
 * step's first timed stage (layer 1's speculation; layer 0's attention when there is one
 * layer).  Layer 0 has no fetch or speculation: NaN there.  The InfiniGen paper-graph summary
 * draws this overlap of the prefetch with the previous layer's compute (section 3.2, Fig 8);
 * the timeline shows it.  Needs config.stage_timing = 1; waits for that step to finish. */
ig_status ig_decoder_timeline(ig_decoder* dec, int steps_back, float* t_out);

/* Host-link probes (measurement, not steps of the method).  The fetch of the selected rows
 * (ig_gather_kv) is bound by the link between host memory and the GPU; the summary's critique
 * (section 6.3) ties InfiniGen's gains to that link, so its speed is measured on the machine
 * rather than assumed.  Both read mapped, pinned host memory in place (zero-copy), 16 bytes
 * per load, many loads in flight; ctas = 0 picks 4 CTAs per SM.
 *   ig_link_read:   streams `bytes` (a positive multiple of 16) of src; nothing is written
 *                   (sink, dev 16 bytes, 16-byte aligned, receives a store only for a
 *                   checksum no real buffer produces).
 *   ig_link_gather: dst row j = src row idx[j] for j < n, rows of row_bytes (16 times a
 *                   divisor of 256: 16 .. 4096); src [rows][row_bytes] mapped pinned host,
 *                   idx dev int32 [n], dst dev [n][row_bytes]; an index outside [0, rows)
 *                   sets IG_DEVERR_INDEX and its row is skipped.
 * src, dst 16-byte aligned.  Asynchronous on `stream`.  No counterpart in the paper. */
ig_status ig_link_read(void* stream, const void* src, size_t bytes, void* sink, int ctas);
ig_status ig_link_gather(void* stream, const void* src, size_t rows, int row_bytes,
                         const int32_t* idx, size_t n, void* dst, int ctas);

#ifdef __cplusplus
}
#endif

#endif /* IG_H_ */
