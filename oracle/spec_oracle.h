/*
 * spec_oracle.h — plain single-threaded CPU oracle of the exact greedy verify
 * step.  TEST INFRASTRUCTURE ONLY: it exists to be compared against.  Only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg may load it;
 * the product library never links, calls or falls back to it.
 *
 * It shares no code, header, table or constant with the CUDA library.  Every
 * function computes the plain definition, scalar and in serial order, in the
 * precision stated beside it.  Sources (titles of the pages, and sections):
 *   [33]  Muser book Ch. 33 "Speculation: the local win and the distributed
 *         verdict"  (accept rule §33.2; carried frontier §33.7; batched verify
 *         §33.1)
 *   [8]   Muser book Ch. 8 "The DFlash draft"  (16-row block, verify lengths
 *         3/7/15 §8.6 item 3; metadata-only KV rewind §8.6 item 4; k-quant
 *         weights consumed directly and f32 norm vectors §8.5)
 *   [32]  Muser book Ch. 32 "Precision across the handoff"  (integer-dot anchor
 *         §32.7; one pinned reduction order and F32 residual, chapter intro and
 *         §32.4)
 *   [TF]  sanctum.run "The Two-Fifteen That Wasn't"  (temp-0 token-fidelity gate
 *         "Three phases, each behind the gate" / "Perfect, and slower";
 *         batch-height kernel flips "The stream that was load-bearing")
 * Where the pages leave a step open, the reading taken is stated at the
 * function (Q4_K byte layout, Q8 rounding, fp32 combination order, RMSNorm,
 * attention, SwiGLU, page allocation order).
 */
#ifndef SPEC_ORACLE_H
#define SPEC_ORACLE_H
#include <stdint.h>

typedef struct {
    int32_t hidden, n_layers, n_q_heads, n_kv_heads, head_dim, ffn, vocab, page_size;
    float rms_eps;
    /* sliding-window layers ([8] §8.6 item 4 names them "SWA rings"): layer l
     * is one when swa_window > 0, swa_period > 0 and l % swa_period ==
     * swa_period - 1; its row at position p sees positions p-swa_window+1..p */
    int32_t swa_window, swa_period;
    /* rotary position embedding of q and k ([8] §8.2 lists RoPE for the
     * draft's attention): 0 = none, else the base theta */
    float rope_theta;
} orc_cfg;

/* Host pointers to CANONICAL Q4_K matrices (see orc_q4k_* below). */
typedef struct {
    const uint8_t* const* w_qkv;
    const uint8_t* const* w_o;
    const uint8_t* const* w_gate_up;
    const uint8_t* const* w_down;
    const float* const* attn_norm;   /* NULL or entries NULL = ones */
    const float* const* ffn_norm;
    const float* final_norm;
    const uint8_t* w_head;
    /* per-head RMSNorm of q and of k before RoPE ([8] §8.2 "QK-norms"):
     * per-layer gains of head_dim floats; NULL = none */
    const float* const* q_norm;
    const float* const* k_norm;
} orc_weights;

/* Host paged KV model; same meaning as the library's cache. */
typedef struct {
    uint16_t* pool;       /* bf16 bits [num_pages][n_layers][2][n_kv][page][dh] */
    int32_t num_pages, max_seq_pages;
    int32_t* page_table;
    int32_t* seq_len;
    int32_t* free_stack;
    int32_t* free_top;
} orc_kv;

enum { ORC_ST_TOKEN_RANGE = 1, ORC_ST_NONFINITE = 2, ORC_ST_POOL_EMPTY = 4,
       ORC_ST_ROLLBACK = 8, ORC_ST_CTX_FULL = 16 };

/* number formats */
float    orc_half_to_float(uint16_t h);
float    orc_bf16_to_float(uint16_t b);
uint16_t orc_float_to_bf16(float f);

/* Q4_K superblock accessors (canonical layout) */
void orc_q4k_scale_min(const uint8_t* sb, int j, int* sc, int* m);
int  orc_q4k_code(const uint8_t* sb, int e);
void orc_q4k_dequant_f64(const uint8_t* W, int N, int K, double* out /* [N][K] */);

/* Q8 activation quantisation; returns ORC_ST_NONFINITE or 0 */
int orc_quantize_q8(const float* x, int M, int K, int8_t* q, float* d_a, int32_t* A);

/* integer-dot GEMM; isc/imn/vb may be NULL, else [M][N][K/256] */
void orc_gemm_q4k(const uint8_t* W, int N, int K, const int8_t* q, const float* d_a,
                  const int32_t* A, int M, float* y, int32_t* isc, int32_t* imn, float* vb);
/* quantise + GEMM; returns the quantiser status */
int orc_linear(const uint8_t* W, int N, int K, const float* x, int M, float* y);
/* the fixed fp32 summation order over superblocks (see spec_oracle.c) */
int  orc_split_ranges(int N, int K, int processors);
void orc_sum_split(const float* vb, int M, int N, int nb, int G, float* y);
/* dense fp64 reference: y = dequant(W) x, x given in fp64 */
void orc_dense_f64(const uint8_t* W, int N, int K, const double* x, int M, double* y);

void orc_rmsnorm(const float* x, const float* gamma, int M, int H, float eps, float* y);
void orc_silu_mul(const float* gate, const float* up, int n, float* h);
void orc_argmax(const float* logits, int M, int V, int32_t* idx, float* gap);
int  orc_accept(const int32_t* idx, const int32_t* draft, int k, int vocab,
                int32_t* accepted, int32_t* next);

/* KV metadata */
void orc_kv_reset(orc_kv* kv);
int  orc_kv_reserve(orc_kv* kv, int32_t upto);       /* map pages for positions < upto */
int  orc_kv_extend(orc_kv* kv, int32_t n);
int  orc_kv_rollback(orc_kv* kv, int32_t new_len);
void orc_kv_write_row(const orc_cfg* c, orc_kv* kv, int layer, int pos,
                      const float* k_row, const float* v_row);
void orc_attention(const orc_cfg* c, const orc_kv* kv, int layer, const float* q,
                   int M, int n_past, float* out);

/* one transformer block on M rows at positions n_past.. (K/V appended) */
int orc_block(const orc_cfg* c, const orc_weights* w, orc_kv* kv, int layer,
              const float* x_in, int M, int n_past, float* x_out);
/* token trees ([33] §33.7): node 0 = the carried frontier, parent[i] < i */
#define ORC_ST_BAD_TREE 0x40
#define ORC_TREE_MAX 64     /* nodes of a token tree ([33] §33.7 names 24 to 64) */
void orc_attention_tree(const orc_cfg* c, const orc_kv* kv, int layer, const float* q,
                        int M, int n_past, const uint64_t* mask, float* out);
int  orc_tree_masks(const int32_t* tokens, const int32_t* parent, int n, int vocab, uint64_t* mask);
void orc_tree_accept(const int32_t* idx, const int32_t* tokens, const int32_t* parent, int n,
                     int32_t* L, int32_t* next, int32_t* path);
void orc_kv_compact(const orc_cfg* c, orc_kv* kv, int n_past, const int32_t* path, int L);
int  orc_verify_tree(const orc_cfg* c, const orc_weights* w, orc_kv* kv, const float* hidden,
                     const int32_t* tokens, const int32_t* parent, int n, int32_t* res, int32_t* path,
                     int32_t* idx, float* logits);

/* QK-norm and RoPE of the M rows of a QKV projection output qkv [M][Nqkv]
 * (q heads, then k heads, then v heads) at positions n_past.., in place: the
 * q and k heads each normalised over head_dim (rms, eps, gain of the layer)
 * when the layer has gains, then rotated by RoPE when rope_theta > 0 */
void orc_qk_norm_rope(const orc_cfg* c, const orc_weights* w, int layer, float* qkv, int M, int n_past);

/* the window of layer l: swa_window for a sliding-window layer, 0 otherwise */
int orc_layer_window(const orc_cfg* c, int layer);

/* stochastic exact acceptance ([33] §33.2): MT19937 state of 625 words */
void     orc_mt_seed(uint32_t* st, uint32_t seed);
uint32_t orc_mt_next(uint32_t* st);
float    orc_uniform_f32(uint32_t* st);
void     orc_softmax_row(const float* l, int V, float* p);
/* one draw from the weights w [V] (a distribution): the first token in index
 * order whose running fp32 sum exceeds one uniform u (the last token of
 * positive weight if none does); *margin = distance of u from the nearest
 * running-sum boundary around the chosen token */
int32_t  orc_sample_ordered(const float* w, int V, uint32_t* mt, double* margin);
int      orc_sample_accept(const float* logits, const float* q, const int32_t* draft, int k, int V,
                           uint32_t* mt, int32_t* res, double* margin);
/* forward of M rows at positions seq_len..: reserves pages, appends K/V, sets
 * seq_len += M; writes argmax idx [M], logits [M][V] (nullable) and the
 * residual taps [(n_layers+1)][M][H] (nullable) */
int orc_forward(const orc_cfg* c, const orc_weights* w, orc_kv* kv, const float* hidden,
                int M, int32_t* idx, float* logits, float* resid);
/* the verify step: res = {accepted, next, status, seq_len} */
int orc_verify_step(const orc_cfg* c, const orc_weights* w, orc_kv* kv, const float* hidden,
                    const int32_t* draft, int k, int32_t* res, int32_t* idx, float* logits,
                    float* resid);
/* serial greedy decode of the same k+1 rows, one row per forward */
int orc_serial_greedy(const orc_cfg* c, const orc_weights* w, orc_kv* kv, const float* hidden,
                      int k, int32_t* tokens);
#endif
