/*
 * spec_verify.h — C ABI of the exact greedy speculative verify step on one GB300.
 *
 * What the step computes.  The target model runs ONE batched forward over
 * M = k+1 rows: row 0 is the carried frontier token, rows 1..k are the draft
 * proposals.  Each row's argmax is the target's own next-token choice; the
 * draft is accepted up to the first disagreement, the disagreeing position's
 * target token becomes the next carried frontier, and the KV rows of the
 * rejected suffix are rolled back.
 *   - batched verify of k+1 rows per weight read: Muser book Ch. 33
 *     ("Speculation: the local win and the distributed verdict") §33.1 and
 *     Ch. 8 ("The DFlash draft") §8.1;
 *   - the accept rule: Ch. 33 §33.2 (verify_full_speculative_mt_ordered);
 *     greedy acceptance is its one-hot (temperature 0) special case, see
 *     spec_accept below;
 *   - the carried frontier: Ch. 33 §33.7 (carried-frontier state machine);
 *   - verify lengths {3, 7, 15} and the 16-row block: Ch. 8 §8.6 item 3;
 *   - metadata-only KV rewind: Ch. 8 §8.6 item 4 (MetalSpeculativeCheckpoint);
 *   - k-quant weights consumed directly by the GPU: Ch. 8 §8.5;
 *   - integer-exact dot products as the anchor: Ch. 32 ("Precision across the
 *     handoff") §32.4 and §32.7;
 *   - batch-height-invariant arithmetic: "The Two-Fifteen That Wasn't"
 *     (sanctum.run), section "The stream that was load-bearing".
 *
 * Conventions for every entry point.
 *   - Device pointers are CUDA global-memory pointers of the current device;
 *     host pointers are plain process memory.  Nothing here takes ownership of
 *     a caller pointer: the caller allocates and frees every input, output,
 *     weight and KV buffer.  The library allocates only the workspace owned by
 *     a spec_ctx, once, in spec_verify_init, and frees it in
 *     spec_verify_destroy.  No entry point allocates after init.
 *   - Work is enqueued on the ctx's stream and is asynchronous unless stated.
 *     Host-side validation happens before anything is enqueued; a negative
 *     return code means nothing was enqueued.
 *   - Device-detected conditions (token out of range, non-finite value, page
 *     pool exhausted, bad rollback length) are OR-ed into a device status word
 *     (spec_result.status, or the ctx status word read by spec_last_status)
 *     and never trap the GPU.
 *   - All matrices are row-major.  "Q4_K" below means the superblock format
 *     defined next.
 *
 * Q4_K superblock (144 bytes, 256 weights).  A weight matrix W of N output
 * columns and K inputs (K a multiple of 256) is stored, in the CANONICAL
 * layout, as N x (K/256) superblocks, column n's superblock b at byte offset
 * (n*(K/256) + b)*144.  Superblock b of column n holds W[n][256b .. 256b+255]:
 *   bytes 0..1   d    (IEEE binary16, little endian)
 *   bytes 2..3   dmin (IEEE binary16, little endian)
 *   bytes 4..15  a 96-bit little-endian field F: sub-scale sc_j = bits
 *                [6j, 6j+6) of F and sub-min m_j = bits [48+6j, 48+6j+6),
 *                j = 0..7 (6-bit unsigned each)
 *   bytes 16..143  4-bit codes: element e (0..255), j = e/32, r = e%32, lives
 *                in byte 16 + 16j + (r%16), low nibble if r < 16, else high.
 * Dequantised weight: w_e = d * sc_j * q_e - dmin * m_j, q_e in 0..15.
 * The TILED layout produced by spec_weights_repack holds the same bytes
 * permuted for the tensor-core fragments; every GEMM entry point here takes
 * the TILED layout.  Its size is identical (N*(K/256)*144 bytes).
 *
 * Activation quantisation (per row, per 256-block b): d_a = amax/127 (IEEE
 * fp32 division), q = clamp(rint(x/d_a), -127, 127) with round-half-even,
 * d_a = 0 and q = 0 for an all-zero block.  Sub-block sums A_j = sum of the 32
 * q's of sub-block j.
 * Integer sums per (row m, column n, superblock b):
 *   S_j = sum_{i<32} q_w[32j+i] * q_a[256b+32j+i]            (exact)
 *   ISc = sum_j sc_j * S_j,  IMn = sum_j m_j * A_j            (exact, int32)
 * Per-superblock value, fp32, each operation rounded to nearest, no fusion:
 *   v_b = d_a * ((float)d * (float)ISc - (float)dmin * (float)IMn)
 * Output y[m][n] = sum_b v_b in fp32, in a fixed order that depends on N, K
 * and the SM count P only, never on M: the U = ceil(N/128) * (K/256) units
 * (128-column group, superblock), numbered group-major, are cut into G
 * contiguous ranges [floor(i*U/G), floor((i+1)*U/G)), where G is the largest
 * value <= min(P, U, 6*U/(K/256)) (at least 1) for which no group meets more
 * than 8 ranges.  Within a range the v_b of a column are added from +0 in
 * superblock order; the partials of the ranges that meet the column's group
 * are added in range order, starting from the first.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>
#include <stddef.h>

#if defined(__GNUC__)
#define SPEC_API __attribute__((visibility("default")))
#else
#define SPEC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- host return codes (0 = OK, negative = nothing was enqueued) -------- */
#define SPEC_OK              0
#define SPEC_EINVAL         -1  /* geometry or argument out of range            */
#define SPEC_EVERIFYLEN     -2  /* k not in {3, 7, 15} (Ch. 8 §8.6 item 3)       */
#define SPEC_ENULL          -3  /* a required pointer is NULL                    */
#define SPEC_EALIGN         -4  /* a pointer is not 16-byte aligned              */
#define SPEC_ENOMEM         -5  /* workspace allocation failed (init only)       */
#define SPEC_ECAPACITY      -6  /* request exceeds the ctx / KV capacity         */
#define SPEC_ECUDA          -7  /* a CUDA runtime call failed                    */
#define SPEC_ENODEV         -8  /* no sm_103 device current                      */

/* ---- device status bits (OR-ed; 0 = OK) ------------------------------ */
#define SPEC_ST_TOKEN_RANGE   0x1  /* a draft token is < 0 or >= vocab           */
#define SPEC_ST_NONFINITE     0x2  /* NaN/Inf in an activation or a logit       */
#define SPEC_ST_POOL_EMPTY    0x4  /* not enough free KV pages for the block     */
#define SPEC_ST_ROLLBACK      0x8  /* rollback length < 0 or > seq_len           */
#define SPEC_ST_CTX_FULL      0x10 /* seq_len + rows exceeds the page table or max_ctx */
#define SPEC_ST_DEVICE_WAIT   0x20 /* a bounded device wait (tensor core, bulk copy) gave up */
#define SPEC_ST_BAD_TREE      0x40 /* a token tree's parent list is not a tree in topological order */

/* Model geometry and workspace sizing.  H and ffn are multiples of 256; the
 * attention width Q = n_q_heads*head_dim is a multiple of 256 too (usually
 * Q = H; a draft block may differ, e.g. 48 query heads at H = 6656);
 * n_q_heads is a multiple of n_kv_heads, at most 13 query heads per KV head;
 * head_dim = 128; page_size = 16; max_rows <= 16 (k_max + 1).  max_ctx
 * bounds the attention workspace (positions per sequence). */
typedef struct spec_config {
    int32_t hidden;       /* H, e.g. 6656                                   */
    int32_t n_layers;     /* e.g. 52                                        */
    int32_t n_q_heads;    /* e.g. 52                                        */
    int32_t n_kv_heads;   /* e.g. 4  (query head h uses kv head h/(nq/nkv)) */
    int32_t head_dim;     /* 128                                            */
    int32_t ffn;          /* F, e.g. 17920                                  */
    int32_t vocab;        /* V, e.g. 131072 (multiple of 16)                */
    int32_t max_rows;     /* maximum k+1 per step, <= 16                    */
    int32_t page_size;    /* 16                                             */
    int32_t max_ctx;      /* maximum sequence length in positions           */
    float   rms_eps;      /* RMSNorm epsilon, e.g. 1e-6                     */
    /* Optional sliding-window layers (Ch. 8 §8.6 item 4, the window rings):
     * with swa_window W > 0, layer l is a sliding-window layer when
     * l % swa_period == swa_period - 1 (1 <= swa_period <= n_layers); its row
     * at position p sees positions p-W+1..p, and its K/V live in a ring of
     * SPEC_SWA_RING_ROWS(W) rows (spec_kv.swa_ring) instead of the paged
     * pool.  16 <= W <= max_ctx.  swa_window = 0: no such layers
     * (swa_period is ignored). */
    int32_t swa_window;
    int32_t swa_period;
    /* Optional rotary position embedding of q and k (Ch. 8 §8.2 lists RoPE
     * for the draft's attention): with rope_theta > 0, element pair
     * (i, i + head_dim/2) of every q and k head of the row at position p is
     * rotated by the angle p * rope_theta^(-i / (head_dim/2)), i < head_dim/2
     * ("rotate-half" pairing), after the optional QK-norm (spec_weights.q_norm,
     * k_norm).  The cos/sin table is computed on the host in double precision
     * at spec_verify_init for positions < max_ctx; a step that would place a
     * row at max_ctx or beyond is refused (SPEC_ST_CTX_FULL), whether or not
     * RoPE is on.  0 = no rotation.  Token trees (spec_verify_tree) refuse a
     * context with rope_theta > 0 (SPEC_EINVAL): their rows' positions are
     * their depths, which this table-per-row layout does not model. */
    float   rope_theta;
} spec_config;

/* Target weights.  Each `const void* const*` is a HOST array of n_layers
 * DEVICE pointers to TILED Q4_K matrices:
 *   w_qkv[l]     N = (n_q_heads + 2*n_kv_heads)*head_dim, K = H; output
 *                columns [0, nq*dh) are Q (head-major), then K, then V.
 *   w_o[l]       N = H, K = n_q_heads*head_dim
 *   w_gate_up[l] N = 2F, K = H; columns [0, F) gate, [F, 2F) up.
 *   w_down[l]    N = H, K = F
 *   w_head       N = V, K = H
 * Norm gains are device fp32 vectors of length H; a NULL entry means all ones
 * (norm vectors stay f32: Ch. 8 §8.5). */
typedef struct spec_weights {
    const void* const* w_qkv;
    const void* const* w_o;
    const void* const* w_gate_up;
    const void* const* w_down;
    const float* const* attn_norm;  /* host array of device pointers, or NULL */
    const float* const* ffn_norm;   /* host array of device pointers, or NULL */
    const float* final_norm;        /* device pointer or NULL                 */
    const void* w_head;
    /* Optional QK-norm (Ch. 8 §8.2): per-layer device fp32 gains of length
     * head_dim.  When q_norm (k_norm) is non-NULL and its entry for layer l is
     * non-NULL, every q (k) head of layer l's QKV output is RMS-normalised over
     * its head_dim elements, x * g / sqrt(mean(x^2) + rms_eps), before RoPE and
     * before the K row enters the cache.  NULL = no QK-norm for that side. */
    const float* const* q_norm;     /* host array of device pointers, or NULL */
    const float* const* k_norm;     /* host array of device pointers, or NULL */
} spec_weights;

/* Paged KV cache (all pointers DEVICE, caller-owned).
 *   pool        bf16 [num_pages][n_layers][2 (K,V)][n_kv_heads][page_size][head_dim]
 *   page_table  int32 [max_seq_pages]: logical page p (positions 16p..16p+15)
 *               -> physical page id, -1 when unmapped
 *   seq_len     int32 [1]: committed positions
 *   free_stack  int32 [num_pages] LIFO of free physical page ids
 *   free_top    int32 [1]: number of ids on free_stack
 * Committed state = (seq_len, page_table[0 .. ceil(seq_len/16)), free stack).
 * Bytes of positions >= seq_len are stale and carry no meaning.
 *
 * Sliding-window layers (spec_config.swa_window > 0; NULL pointers otherwise),
 * with n_swa = n_layers / swa_period such layers, s = l / swa_period:
 *   swa_ring   bf16 [n_swa][2 (K,V)][n_kv_heads][R][head_dim], R =
 *              SPEC_SWA_RING_ROWS(W): position t of layer s in slot t mod R
 *              (the caller lays down a prefilled context's last W positions
 *              there); 16-byte aligned
 *   swa_state  int32 [2]: {position of the last step's block (-1: none),
 *              rows in it}; set by spec_kv_reset, spec_kv_extend and the steps
 * The ring holds W rows rounded up to a multiple of 16, plus 16 spare rows:
 * a block of M <= 16 rows at positions n..n+M-1 overwrites only the slots of
 * positions n-R..n+M-1-R, which precede every window that a row at position
 * n or later sees.  So the rows that a rejected block would have displaced
 * are still in the ring, and every rollback to a length >= n (the step's own
 * accept, or spec_kv_rollback) is served by the metadata alone (Ch. 8 §8.6
 * item 4 keeps those rows in a checkpoint; here the spare slots are that
 * checkpoint).  A rollback below the last step's block, or after an extend,
 * is refused (SPEC_ST_ROLLBACK): the ring may no longer hold the rows a
 * window would need.  The paged pool's slices of sliding-window layers are
 * not used. */
#define SPEC_SWA_RING_ROWS(W) ((((W) + 15) / 16) * 16 + 16)

typedef struct spec_kv {
    void*    pool;
    int32_t  num_pages;
    int32_t  max_seq_pages;
    int32_t* page_table;
    int32_t* seq_len;
    int32_t* free_stack;
    int32_t* free_top;
    void*    swa_ring;
    int32_t* swa_state;
} spec_kv;

/* Step result, DEVICE memory written by the accept kernel at the end of the
 * step (Ch. 33 §33.2, SpeculativeDecision{accepted, next_token}). */
typedef struct spec_result {
    int32_t accepted_len;  /* L in [0, k]                                    */
    int32_t next_token;    /* argmax of row L: the new carried frontier      */
    int32_t status;        /* SPEC_ST_* bits; 0 = OK                         */
    int32_t seq_len;       /* committed KV length after the rollback         */
} spec_result;

/* Optional debug outputs of a step (all DEVICE, each may be NULL). */
typedef struct spec_taps {
    float*   resid;        /* fp32 [n_layers+1][rows][H]: residual stream at the
                              input of each layer, and after the last layer  */
    int32_t* argmax;       /* int32 [rows]: per-row argmax (lowest index wins) */
    float*   logits;       /* fp32 [rows][V]                                 */
} spec_taps;

typedef struct spec_ctx spec_ctx;

/* Create a context on the current device.  Allocates the workspace sized by
 * cfg and binds `cuda_stream` (a cudaStream_t; NULL = legacy default stream).
 * Returns SPEC_OK and *out, or a negative code and *out = NULL. */
SPEC_API int spec_verify_init(const spec_config* cfg, void* cuda_stream, spec_ctx** out);

/* Release the workspace.  Synchronises the ctx stream first.  NULL is a no-op. */
SPEC_API void spec_verify_destroy(spec_ctx* ctx);

/* Rebind the stream used by subsequent calls. */
SPEC_API int spec_set_stream(spec_ctx* ctx, void* cuda_stream);

/* Human-readable text for a return code. */
SPEC_API const char* spec_strerror(int code);

/* One exact greedy verify step (Ch. 33 §33.2 and §33.7; Ch. 8 §8.6).
 *   hidden  DEVICE fp32 [k+1][H]: residual-stream rows entering layer 0; row 0
 *           is the carried frontier, row i (1..k) the draft token draft[i-1].
 *   draft   DEVICE int32 [k]: proposed tokens.
 *   k       verify length, one of 3, 7, 15 (else SPEC_EVERIFYLEN before any
 *           GPU work: Ch. 8 §8.6 item 3); k+1 <= cfg.max_rows.
 *   res     DEVICE spec_result.
 * Enqueues: KV page reservation for positions seq_len..seq_len+k, the
 * 52-block batched forward (K/V rows appended as bf16), final norm, LM head
 * with fused per-row argmax, and one accept/rollback kernel that writes
 *   L = min{ i < k : draft[i] != argmax(row i) } (else k),
 *   next_token = argmax(row L),  seq_len := n_past + L + 1
 * and returns the pages wholly at or beyond the new seq_len to the free stack.
 * On a device error nothing is committed: seq_len, the page table and the free
 * stack are restored to their values before the step and res->status != 0.
 * No host synchronisation and no allocation happen inside. */
SPEC_API int spec_verify_step(spec_ctx* ctx, const spec_weights* w, spec_kv* kv,
                     const float* hidden, const int32_t* draft, int k,
                     spec_result* res);

/* spec_verify_step plus optional debug taps (taps may be NULL). */
SPEC_API int spec_verify_step_ex(spec_ctx* ctx, const spec_weights* w, spec_kv* kv,
                        const float* hidden, const int32_t* draft, int k,
                        spec_result* res, const spec_taps* taps);

/* The same step from HOST buffers: copies hidden [k+1][H] fp32 and draft [k]
 * int32 from host memory (pinned for overlap) to the ctx workspace, runs the
 * step, copies the spec_result back to *res_host, and synchronises the
 * stream before returning. */
SPEC_API int spec_verify_step_host(spec_ctx* ctx, const spec_weights* w, spec_kv* kv,
                          const float* hidden_host, const int32_t* draft_host,
                          int k, spec_result* res_host);

/* Number of kernels the last spec_verify_step enqueued (for accounting). */
SPEC_API int spec_last_step_launches(const spec_ctx* ctx);

/* Timing of the Q4_K GEMM launches of subsequent steps: with enable != 0 the
 * step records a CUDA event pair around each GEMM launch on the ctx stream
 * (events are created here, not in the step).  spec_profile_read synchronises
 * the stream and returns the summed GEMM time of the last step (ms) and the
 * number of GEMM launches it made. */
SPEC_API int spec_profile_gemms(spec_ctx* ctx, int enable);
SPEC_API int spec_profile_read(spec_ctx* ctx, float* gemm_ms, int* gemm_launches);

/* ---- KV cache management (Ch. 8 §8.6 item 4: metadata-only rewind) ------- */

/* Reset a KV cache to empty: seq_len = 0, page_table = -1, free_stack filled
 * descending (id num_pages-1 at the bottom) so that pops yield ids 0, 1, 2...
 * Requires num_pages <= 2^30. */
SPEC_API int spec_kv_reset(spec_ctx* ctx, spec_kv* kv);

/* Map pages for positions [seq_len, seq_len + n) and set seq_len += n.  Used to
 * lay down a prefilled context; the caller writes those rows' bytes.  Device
 * errors (pool empty, page table full) leave the state unchanged and set the
 * ctx status word. */
SPEC_API int spec_kv_extend(spec_ctx* ctx, spec_kv* kv, int32_t n);

/* Roll the committed length back to new_len (0 <= new_len <= seq_len, checked
 * on the device; violations set SPEC_ST_ROLLBACK in the ctx status word and
 * change nothing).  Logical pages p with 16p >= new_len are unmapped and their
 * ids pushed on the free stack from the highest p down, so re-extending maps
 * the same ids to the same pages again.  Retained rows are untouched. */
SPEC_API int spec_kv_rollback(spec_ctx* ctx, spec_kv* kv, int32_t new_len);

/* Read (synchronously) and clear the ctx status word set by the entry points
 * that have no spec_result.  Returns SPEC_ST_* bits, or a negative code. */
SPEC_API int spec_last_status(spec_ctx* ctx);

/* ---- building blocks, exposed for parity tests and benchmarks ------------ */

/* One-time weight repack: canonical Q4_K (DEVICE, N x K/256 superblocks) ->
 * TILED Q4_K (DEVICE, same size).  N % 16 == 0, K % 256 == 0.  src and dst
 * must not overlap.  Deterministic permutation of bytes, no arithmetic. */
SPEC_API int spec_weights_repack(spec_ctx* ctx, const void* src_canonical, void* dst_tiled,
                        int N, int K);

/* Activation quantisation of x (DEVICE fp32 [M][K]) exactly as described at
 * the top of this file, written in plain layout: q int8 [M][K], d_a fp32
 * [M][K/256], A int32 [M][K/32].  M <= 16, K % 256 == 0.  Non-finite input
 * sets SPEC_ST_NONFINITE in the ctx status word. */
SPEC_API int spec_quantize_q8(spec_ctx* ctx, const float* x, int M, int K,
                     int8_t* q, float* d_a, int32_t* A);

/* y = W x for M rows: quantise x (DEVICE fp32 [M][K]) per 256-block, run the
 * skinny Q4_K x Q8 tensor-core GEMM on the TILED weights, write y (DEVICE
 * fp32 [M][N]).  1 <= M <= 16, N % 16 == 0, K % 256 == 0, N*K within the
 * workspace built for cfg (largest of the model's matrices).  Row i of y is
 * bit-identical for every M >= i+1. */
SPEC_API int spec_gemm_q4k(spec_ctx* ctx, const void* w_tiled, int N, int K,
                  const float* x, int M, float* y);

/* The number G of contiguous unit ranges in the GEMM's fixed summation order
 * (stated at the top of this file) for an N x K matrix on a GPU of num_sms
 * SMs: the value every GEMM entry point here uses on such a GPU.  Host only:
 * touches no device and needs no ctx.  Returns G >= 1, or SPEC_EINVAL unless
 * N > 0, N % 16 == 0, K > 0, K % 256 == 0 and num_sms > 0. */
SPEC_API int spec_gemm_ranges(int N, int K, int num_sms);

/* Same GEMM, also writing the exact integer sums ISc and IMn (DEVICE int32
 * [M][N][K/256] each) of every (row, column, superblock). */
SPEC_API int spec_gemm_q4k_sums(spec_ctx* ctx, const void* w_tiled, int N, int K,
                       const float* x, int M, float* y,
                       int32_t* isc, int32_t* imn);

/* The same y = W x on CUDA cores: 4-way byte dot products (dp4a) instead of
 * tensor-core MMAs, for the comparison that chose the tensor cores for the
 * 16-row tile (the integer-dot anchor of Ch. 32 §32.7 on either unit).  The
 * integer sums and each superblock's value are the same exact quantities;
 * the sum over superblocks is split over CTAs and added with atomics, so y
 * agrees with spec_gemm_q4k within rounding and is not batch-height
 * invariant.  Not used by the verify step.  Arguments as spec_gemm_q4k
 * (K <= the largest K of the ctx's model, including 5*H). */
SPEC_API int spec_gemm_q4k_cudacore(spec_ctx* ctx, const void* w_tiled, int N, int K,
                                    const float* x, int M, float* y);

/* Self-test of the bounded device waits (failure detection without a GPU
 * fault): launches the GEMM kernel on w_tiled (N x K, as spec_gemm_q4k) with
 * its copy producer held back, so that no bulk copy or MMA is ever issued
 * and every consumer wait gives up after its limit (about 2 s).  The kernel
 * then unwinds and frees its tensor memory; the ctx status word holds
 * SPEC_ST_DEVICE_WAIT (spec_last_status) and the context stays usable.
 * Writes no output. */
SPEC_API int spec_gemm_wait_selftest(spec_ctx* ctx, const void* w_tiled, int N, int K);

/* The same GEMM for callers that must not allocate device memory (no ctx).
 * The pages have no counterpart; this exists for hosts where calling the CUDA
 * allocator is not allowed or not safe at the call site.  Scratch (activation
 * buffer and partial sums) lives in a fixed 8 MiB array that every device
 * loading the library holds until exit; requests that do not fit return
 * SPEC_ECAPACITY before anything is enqueued.  All calls on a device share
 * that array: calls that overlap on the GPU race, calls ordered on one stream
 * do not.  The first call on a device looks up the array's device address
 * (make it before capturing any stream).  Enqueued on cuda_stream (a
 * cudaStream_t, NULL = legacy default stream); y is DEVICE fp32 [M][N]. */
SPEC_API int spec_gemm_q4k_noalloc(const void* w_tiled, int N, int K, const float* x, int M,
                                   float* y, void* cuda_stream);

/* Device status of the last spec_gemm_q4k_noalloc call on the current device:
 * synchronises cuda_stream (the stream that call was enqueued on), then reads
 * the status word at the start of the fixed array without allocating.
 * Returns SPEC_ST_* bits (0 = OK; SPEC_ST_NONFINITE: a non-finite activation;
 * SPEC_ST_DEVICE_WAIT: a bounded device wait gave up and y is incomplete), or
 * a negative code.  Every call clears the word first, so it describes only the
 * latest call; calls that overlap on the GPU share it. */
SPEC_API int spec_gemm_q4k_noalloc_status(void* cuda_stream);

/* Final RMSNorm (gain final_norm, NULL = ones) + LM head (TILED Q4_K,
 * N = cfg.vocab, K = cfg.hidden) + per-row argmax, lowest index on ties.
 * x DEVICE fp32 [M][H]; idx DEVICE int32 [M]; logits DEVICE fp32 [M][V] or
 * NULL (the fused path writes no logits).  Non-finite logits set
 * SPEC_ST_NONFINITE in the ctx status word. */
SPEC_API int spec_lm_head_argmax(spec_ctx* ctx, const void* w_head_tiled,
                        const float* final_norm, const float* x, int M,
                        int32_t* idx, float* logits);

/* Verify attention of one layer: M query rows at positions seq_len-M ..
 * seq_len-1 (their K/V rows already in the cache) against all positions
 * 0..p_i of row i (a sliding-window layer: p_i-W+1..p_i, from its ring).
 * q DEVICE fp32 [M][n_q_heads][head_dim]; out DEVICE fp32
 * [M][n_q_heads*head_dim].  s = q.k/sqrt(head_dim), softmax over the visible
 * positions, o = sum p v; K and V read as bf16. */
SPEC_API int spec_attention(spec_ctx* ctx, const spec_kv* kv, int layer,
                   const float* q, int M, float* out);

/* Greedy accept + rollback alone (the last kernel of a step).
 *   idx    DEVICE int32 [k+1] per-row argmax of rows 0..k
 *   draft  DEVICE int32 [k]
 *   kv     if not NULL: its seq_len holds n_past + k + 1 (block appended) and
 *          is rolled back to n_past + L + 1.
 * Writes res (DEVICE).  Accept rule: Ch. 33 §33.2 with one-hot target and
 * draft distributions: p/q = 1 where draft == argmax (accept with certainty),
 * p = 0 elsewhere (reject), residual max(p - q, 0) one-hot at the argmax. */
SPEC_API int spec_accept(spec_ctx* ctx, const int32_t* idx, const int32_t* draft, int k,
                spec_kv* kv, spec_result* res);

/* ---- Token-tree verification (Ch. 33 §33.7: a tree spends the verify batch
 * on covering near-miss branches; the section names trees of 24, 32, 48 and
 * 64 nodes), up to 64 nodes.
 *
 * Node 0 is the carried frontier; node i >= 1 holds the draft token
 * tokens[i], proposed as the continuation of node parent[i] < i (parent[0] =
 * -1; tokens[0] is not read).  Node i's row is hidden[i]; it sees the
 * context and its ancestors and itself.  The root is accepted; node i is
 * accepted when its parent is and tokens[i] equals the parent's argmax.  The
 * deepest accepted node a (the lowest index among equals) ends the path root
 * -> a: accepted_len = depth(a), next_token = argmax of a.  The path's K/V
 * rows move to positions n_past .. n_past + depth(a), and the KV is rolled
 * back to n_past + depth(a) + 1.
 *   hidden   DEVICE fp32 [n][H]; tokens, parent DEVICE int32 [n]; 1 <= n <= 64
 *   path_out DEVICE int32 [max(16, n)] or NULL: the path's nodes, then -1
 *   taps     as in spec_verify_step_ex (argmax and logits = per node; the
 *            residual taps only for n <= max_rows, else SPEC_EINVAL)
 * Up to max_rows nodes run as one batched forward; a larger tree runs in
 * passes of max_rows rows (nodes 0..15, 16..31, ...), each a full forward of
 * its rows that streams the weights once, with every node's row seeing its
 * ancestors in earlier passes through the KV cache.  A parent list that is
 * not a tree in topological order sets SPEC_ST_BAD_TREE before any work; the
 * KV is left as it was.  A model with sliding-window layers is refused
 * (SPEC_EINVAL): the path's K/V moves are defined for the paged cache only. */
SPEC_API int spec_verify_tree(spec_ctx* ctx, const spec_weights* w, spec_kv* kv, const float* hidden,
                              const int32_t* tokens, const int32_t* parent, int n, spec_result* res,
                              int32_t* path_out, const spec_taps* taps);

/* ---- Hidden-state capture for a draft's front projection (Ch. 8: the
 * draft is fed the target's hidden states from five pinned target layers,
 * concatenated, through fc: 5 x 6,656 = 33,280 -> 6,656).
 *
 * From the next step on, the residual stream after block layer_ids[j] (the
 * block's output, fp32) of each of the M rows is written to
 * rows[m][j*H .. j*H + H), row stride n*H: the layout spec_gemm_q4k takes as
 * its input x for K = n*H.  n <= 8 distinct ids in [0, n_layers); n = 0 turns
 * the capture off.  rows: DEVICE fp32 [16][n*H], 16-byte aligned, owned by the
 * caller and kept alive while the capture is on.  The capture is part of the
 * residual kernel that produces the block output: no extra launch. */
SPEC_API int spec_set_capture(spec_ctx* ctx, const int32_t* layer_ids_host, int n, float* rows);

/* ---- Split submit (Ch. 33 §33.2, the Mirror-SD route of the paragraph
 * before Figure 33.1, and Figure 33.1): the target's graph is split at a
 * capture layer; the prefix through that layer runs first, and the draft's
 * work overlaps the target's remaining layers and LM head.
 *
 * From the next step on, every verify step (linear, tree or sampled) records
 * cuda_event (a cudaEvent_t created by the caller on this ctx's device) on
 * the ctx stream as soon as the output of block `layer` is written,
 * including its hidden-state capture rows (spec_set_capture).  A second
 * stream that waits on the event (cudaStreamWaitEvent) may read those rows
 * while the step's suffix runs, e.g. to run the draft's front projection.
 * The work on that stream must not use this ctx's workspace: give it a
 * spec_ctx of its own, or use spec_gemm_q4k_noalloc.  The step's result is
 * unchanged; its end is observed as before (the ctx stream).  A step that
 * is replayed as a recorded graph carries the event as an external event
 * record node, so a wait issued after the step was enqueued still refers to
 * that step's record.  layer = -1 turns the split off (cuda_event is
 * ignored); the event must stay valid while the split is on. */
SPEC_API int spec_set_split(spec_ctx* ctx, int layer, void* cuda_event);

/* ---- Stochastic exact acceptance (Ch. 33 §33.2; the rule of which
 * spec_accept is the one-hot case).
 *
 * For i < k: x = draft[i], p = p_i(x), q = q_i(x), a = 1 if q <= 0 else
 * min(p/q, 1); one uniform u; u <= a accepts and goes on.  On the first
 * rejection the next token is drawn from max(p_i - q_i, 0) renormalised (from
 * p_i itself when that is all zero); when all k are accepted, from p_k.
 * p_i = softmax of the target logits of row i (temperature 1).
 *
 * Uniforms come from a caller-owned MT19937 stream (Matsumoto & Nishimura
 * 1998), one per attempted draft, then one for the final draw, in that
 * order; uniform = (draw >> 8) * 2^-24.  A draw walks the tokens in index
 * order and returns the first whose running sum of the renormalised weights
 * exceeds u (the last token of positive weight if rounding leaves none).
 * On a device error (a draft token outside [0, V), non-finite logits) no
 * uniform is drawn; the result is as in spec_verify_step. */
#define SPEC_MT_WORDS 625   /* 624 state words + the index of the next word */

/* Seed an MT19937 state in HOST memory (state_host: SPEC_MT_WORDS words);
 * the caller copies it to the device once and keeps it there. */
SPEC_API int spec_mt_seed(uint32_t* state_host, uint32_t seed);

/* The decision alone, from logits that are already computed.
 *   logits DEVICE fp32 [k+1][V]   target logits of rows 0..k
 *   q      DEVICE fp32 [k][V]     the draft's distribution at positions 0..k-1
 *   draft  DEVICE int32 [k], 1 <= k <= 15
 *   mt     DEVICE uint32 [SPEC_MT_WORDS], advanced by the draws
 *   kv     as in spec_accept (NULL: no rollback)
 * Writes res (DEVICE); next_token is the drawn token. */
SPEC_API int spec_sample_accept(spec_ctx* ctx, const float* logits, const float* q,
                                const int32_t* draft, int k, uint32_t* mt, spec_kv* kv,
                                spec_result* res);

/* The verify step with the sampled decision: as spec_verify_step_ex, with
 * q (DEVICE fp32 [k][V]) and mt (DEVICE, SPEC_MT_WORDS words) as above.  The
 * step keeps the M rows' logits in its workspace (8 MB at V = 131072);
 * taps->logits and taps->argmax are filled when given. */
SPEC_API int spec_verify_step_sampled(spec_ctx* ctx, const spec_weights* w, spec_kv* kv,
                                      const float* hidden, const int32_t* draft, const float* q,
                                      int k, uint32_t* mt, spec_result* res,
                                      const spec_taps* taps);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
