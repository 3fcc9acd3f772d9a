// api.cu — the C ABI of include/spec_verify.h: context and workspace, host-side
// validation (everything is checked before anything is enqueued), and the
// orchestration of one verify step as a fixed sequence of kernel launches on
// one stream with programmatic dependent launch between them.
//
// Step (Muser book Ch. 33 §33.1-§33.2 and §33.7; Ch. 8 §8.6):
//   reserve pages for the k+1 block (validates the draft tokens first)
//   per layer: RMSNorm+Q8 -> QKV GEMM -> split Q / append K,V (bf16) ->
//              attention partials -> merge+Q8 -> O GEMM -> residual+RMSNorm+Q8
//              -> gate|up GEMM -> SwiGLU+Q8 -> down GEMM -> residual+RMSNorm+Q8
//   LM head GEMM -> per-row argmax -> accept + rollback
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <cmath>
#include <new>
#include <vector>

#include "../../include/spec_verify.h"
#include "common.cuh"
#include "internal.h"

using namespace spec;

struct spec_ctx {
  spec_config cfg;
  cudaStream_t stream = nullptr;
  int num_sms = 0;
  GemmPlan p_qkv, p_o, p_gu, p_down, p_head;
  AttnPlan attn;                 // paged layers: chunks over the whole context
  AttnPlan attn_swa;             // sliding-window layers: chunks over the window
  size_t act_bytes = 0, pieces_floats = 0;
  uint8_t* act = nullptr;
  float* pieces = nullptr;
  float* resid = nullptr;        // [16][H]
  float2* rope_cs = nullptr;     // [max_ctx][dh/2] (cos, sin) of the rotary angles
  int8_t* q8 = nullptr;          // plain int8 codes, d_a and sub-block sums of the
  float* da8 = nullptr;          // CUDA-core comparison GEMM
  int32_t* a8 = nullptr;
  int kmax = 0;
  uint8_t* qtile = nullptr;      // attention query tiles, 64 KB per (kv head, tile)
  float* attn_part = nullptr;
  float* head_val = nullptr;     // [nparts][16]
  int32_t* head_idx = nullptr;
  int head_parts = 0;
  int32_t* status = nullptr;     // device status word
  float* logits_ws = nullptr;    // [16][V] target logits of a sampled step
  float2* sstats = nullptr;      // [16] row max and sum of exp of a sampled step
  uint8_t* sscratch = nullptr;   // decision scratch of a sampled step
  uint64_t* tree_mask = nullptr; // [64] ancestor masks of a token-tree step
  uint8_t* tscratch = nullptr;   // decision scratch of a token-tree step
  // hidden-state capture: block outputs of cap_ids[j] -> cap_rows[m][j*H ..]
  int cap_n = 0;
  int cap_ids[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  float* cap_rows = nullptr;
  // split submit: an event recorded after block split_layer's output
  int split_layer = -1;
  cudaEvent_t split_ev = nullptr;
  int32_t* step_state = nullptr; // [2]
  int32_t* idx_buf = nullptr;    // [64] per-row (per tree node) argmax
  float* hidden_dev = nullptr;   // host-buffer entry point staging
  int32_t* draft_dev = nullptr;
  spec_result* res_dev = nullptr;
  int last_launches = 0;
  // optional GEMM timing
  bool profile = false;
  int prof_n = 0;
  cudaEvent_t* prof_ev = nullptr;   // 2 per GEMM launch
  int prof_cap = 0;
  // recorded steps: a step is replayed as a CUDA graph when every pointer and
  // size it bakes into its launches is unchanged
  struct GraphEntry {
    uint64_t key = 0;
    cudaGraphExec_t exec = nullptr;
    int launches = 0;
    uint64_t used = 0;
  };
  GraphEntry graphs[4];
  uint64_t graph_clock = 0;
  bool use_graphs = true;
};

namespace {

constexpr int kPreQkv = 3, kPreO = 3, kPreGu = 3, kPreDown = 3, kPreHead = 3;

constexpr int kAlign = 16;

bool aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) % kAlign) == 0; }

int cuda_code(cudaError_t e) { return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA; }

#define SPEC_TRY(expr)                         \
  do {                                         \
    cudaError_t _e = (expr);                   \
    if (_e != cudaSuccess) return SPEC_ECUDA;  \
  } while (0)

size_t pieces_need(const GemmPlan& p) { return (size_t)p.max_slots * 16 * p.N; }

KvView view_of(const spec_ctx* c, const spec_kv* kv) {
  KvView v;
  v.pool = static_cast<uint16_t*>(kv->pool);
  v.page_table = kv->page_table;
  v.seq_len = kv->seq_len;
  v.free_stack = kv->free_stack;
  v.free_top = kv->free_top;
  v.num_pages = kv->num_pages;
  v.max_seq_pages = kv->max_seq_pages;
  v.n_layers = c->cfg.n_layers;
  v.n_kv = c->cfg.n_kv_heads;
  v.head_dim = c->cfg.head_dim;
  v.page_size = c->cfg.page_size;
  v.swa_ring = static_cast<uint16_t*>(kv->swa_ring);
  v.swa_state = kv->swa_state;
  v.swa_window = c->cfg.swa_window;
  v.swa_period = c->cfg.swa_period;
  v.swa_rows = c->cfg.swa_window > 0 ? swa_ring_rows(c->cfg.swa_window) : 0;
  v.max_ctx = c->cfg.max_ctx;
  return v;
}

bool has_swa(const spec_config& c) { return c.swa_window > 0; }

// the sliding-window buffers a cache needs under this geometry
int check_kv_swa(const spec_ctx* c, const spec_kv* kv);

int check_kv(const spec_kv* kv) {
  if (!kv || !kv->pool || !kv->page_table || !kv->seq_len || !kv->free_stack || !kv->free_top)
    return SPEC_ENULL;
  if (kv->num_pages <= 0 || kv->max_seq_pages <= 0 || kv->num_pages > (1 << 30)) return SPEC_EINVAL;
  if (!aligned(kv->pool)) return SPEC_EALIGN;
  return SPEC_OK;
}

int check_kv_swa(const spec_ctx* c, const spec_kv* kv) {
  if (!has_swa(c->cfg)) return SPEC_OK;
  if (!kv->swa_ring || !kv->swa_state) return SPEC_ENULL;
  if (!aligned(kv->swa_ring)) return SPEC_EALIGN;
  return SPEC_OK;
}

int check_cfg(const spec_config* c) {
  if (!c) return SPEC_ENULL;
  if (c->hidden <= 0 || c->hidden % 256 || c->hidden / 256 > 64) return SPEC_EINVAL;
  if (c->ffn <= 0 || c->ffn % 256) return SPEC_EINVAL;
  if (c->head_dim != 128 || c->page_size != 16) return SPEC_EINVAL;
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_q_heads % c->n_kv_heads) return SPEC_EINVAL;
  if (c->n_q_heads / c->n_kv_heads > 13) return SPEC_EINVAL;
  // the attention output (n_q_heads * head_dim wide, the O projection's K)
  // is quantised in 256-blocks; it need not equal the hidden width
  if ((c->n_q_heads * c->head_dim) % 256 || c->n_q_heads * c->head_dim > 64 * 256) return SPEC_EINVAL;
  if (c->n_layers <= 0 || c->vocab <= 0 || c->vocab % 16) return SPEC_EINVAL;
  if (c->max_rows < 1 || c->max_rows > 16) return SPEC_EINVAL;
  if (c->max_ctx < c->max_rows) return SPEC_EINVAL;
  if (!(c->rms_eps >= 0.f)) return SPEC_EINVAL;
  if (c->swa_window < 0) return SPEC_EINVAL;
  if (c->swa_window > 0 &&
      (c->swa_window < 16 || c->swa_window > c->max_ctx || c->swa_period < 1 || c->swa_period > c->n_layers))
    return SPEC_EINVAL;
  if (!(c->rope_theta >= 0.f) || !(c->rope_theta < INFINITY)) return SPEC_EINVAL;
  return SPEC_OK;
}

template <class T>
int dalloc(T** p, size_t n) {
  if (n == 0) n = 1;
  return cudaMalloc(reinterpret_cast<void**>(p), n * sizeof(T)) == cudaSuccess ? SPEC_OK : SPEC_ENOMEM;
}

}  // namespace

extern "C" {

const char* spec_strerror(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_EINVAL: return "invalid argument or geometry";
    case SPEC_EVERIFYLEN: return "verify length k must be 3, 7 or 15";
    case SPEC_ENULL: return "required pointer is NULL";
    case SPEC_EALIGN: return "pointer not 16-byte aligned";
    case SPEC_ENOMEM: return "workspace allocation failed";
    case SPEC_ECAPACITY: return "request exceeds workspace or cache capacity";
    case SPEC_ECUDA: return "CUDA runtime error";
    case SPEC_ENODEV: return "no sm_103 device is current";
    default: return "unknown error";
  }
}

int spec_verify_init(const spec_config* cfg, void* cuda_stream, spec_ctx** out) {
  if (!out) return SPEC_ENULL;
  *out = nullptr;
  int rc = check_cfg(cfg);
  if (rc) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ENODEV;
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3) return SPEC_ENODEV;

  spec_ctx* c = new (std::nothrow) spec_ctx();
  if (!c) return SPEC_ENOMEM;
  c->cfg = *cfg;
  c->stream = static_cast<cudaStream_t>(cuda_stream);
  c->num_sms = sms;
  const int H = cfg->hidden, F = cfg->ffn, V = cfg->vocab;
  const int nqkv = (cfg->n_q_heads + 2 * cfg->n_kv_heads) * cfg->head_dim;
  c->p_qkv = make_gemm_plan(nqkv, H, sms);
  const int QW = cfg->n_q_heads * cfg->head_dim;   // attention output width
  c->p_o = make_gemm_plan(H, QW, sms);
  c->p_gu = make_gemm_plan(2 * F, H, sms);
  c->p_down = make_gemm_plan(H, F, sms);
  c->p_head = make_gemm_plan(V, H, sms);
  // Weight stages fetched before each GEMM's dependency wait, set per GEMM
  // by measuring the 2k verify step; the prefetch competes with the previous
  // kernel's L2 reads.  From all 3 (213.8 steps/s), one GEMM at a time:
  // QKV 1/6 gave 212.5/212.1, O 1/6 212.4/213.0, gate+up 1/6 212.7/211.7,
  // down 1/6 212.6/212.2, head 6 213.8.
  c->p_qkv.pre_stages = kPreQkv;
  c->p_o.pre_stages = kPreO;
  c->p_gu.pre_stages = kPreGu;
  c->p_down.pre_stages = kPreDown;
  c->p_head.pre_stages = kPreHead;
  c->attn = make_attn_plan(cfg->n_q_heads, cfg->n_kv_heads, cfg->head_dim, cfg->max_ctx);
  // a window layer's block sees at most W + 15 keys, from the page of its
  // first one: W + 32 covers them
  if (has_swa(*cfg))
    c->attn_swa = make_attn_plan(cfg->n_q_heads, cfg->n_kv_heads, cfg->head_dim, cfg->swa_window + 32);
  size_t pf = 0;
  for (const GemmPlan* p : {&c->p_qkv, &c->p_o, &c->p_gu, &c->p_down, &c->p_head})
    if (pieces_need(*p) > pf) pf = pieces_need(*p);
  c->pieces_floats = pf;
  int kmax = H > F ? H : F;
  if (QW > kmax) kmax = QW;
  if (5 * H > kmax) kmax = 5 * H;   // a draft front projection over 5 concatenated hidden rows
  c->act_bytes = (size_t)(kmax / 256) * kActSBBytes;
  c->kmax = kmax;
  c->head_parts = head_argmax_blocks(V);
  rc = SPEC_OK;
  rc |= dalloc(&c->act, c->act_bytes);
  rc |= dalloc(&c->pieces, c->pieces_floats);
  rc |= dalloc(&c->resid, (size_t)16 * H);
  rc |= dalloc(&c->q8, (size_t)16 * kmax);
  rc |= dalloc(&c->da8, (size_t)16 * (kmax / 256));
  rc |= dalloc(&c->a8, (size_t)16 * (kmax / 32));
  rc |= dalloc(&c->qtile, qtile_bytes(c->attn));
  {
    size_t parts = attn_partial_floats(c->attn, 16);
    if (has_swa(*cfg) && attn_partial_floats(c->attn_swa, 16) > parts) parts = attn_partial_floats(c->attn_swa, 16);
    rc |= dalloc(&c->attn_part, parts);
  }
  rc |= dalloc(&c->head_val, (size_t)c->head_parts * 16);
  rc |= dalloc(&c->head_idx, (size_t)c->head_parts * 16);
  rc |= dalloc(&c->status, 4);
  rc |= dalloc(&c->logits_ws, (size_t)16 * V);
  rc |= dalloc(&c->sstats, 16);
  rc |= dalloc(&c->sscratch, sample_scratch_bytes());
  rc |= dalloc(&c->tree_mask, kTreeMax);
  rc |= dalloc(&c->tscratch, tree_scratch_bytes());
  rc |= dalloc(&c->step_state, 4);
  rc |= dalloc(&c->idx_buf, kTreeMax);
  rc |= dalloc(&c->hidden_dev, (size_t)16 * H);
  rc |= dalloc(&c->draft_dev, 16);
  rc |= dalloc(&c->res_dev, 1);
  if (cfg->rope_theta > 0.f) rc |= dalloc(&c->rope_cs, (size_t)cfg->max_ctx * (cfg->head_dim / 2));
  if (rc != SPEC_OK) {
    spec_verify_destroy(c);
    return SPEC_ENOMEM;
  }
  if (gemm_init_attributes() != cudaSuccess) {
    spec_verify_destroy(c);
    return SPEC_ECUDA;
  }
  if (c->rope_cs) {
    // the rotary table: angle p * theta^(-i/h) and its cosine and sine in
    // double precision, rounded to float once
    const int h = cfg->head_dim / 2;
    std::vector<float2> cs((size_t)cfg->max_ctx * h);
    for (int i = 0; i < h; ++i) {
      const double f = std::pow((double)cfg->rope_theta, -(double)i / h);
      for (int p = 0; p < cfg->max_ctx; ++p) {
        const double a = (double)p * f;
        cs[(size_t)p * h + i] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
    }
    if (cudaMemcpy(c->rope_cs, cs.data(), sizeof(float2) * cs.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
      spec_verify_destroy(c);
      return SPEC_ECUDA;
    }
  }
  if (cudaMemsetAsync(c->status, 0, 16, c->stream) != cudaSuccess ||
      cudaMemsetAsync(c->act, 0, c->act_bytes, c->stream) != cudaSuccess ||
      cudaMemsetAsync(c->qtile, 0, qtile_bytes(c->attn), c->stream) != cudaSuccess ||
      cudaStreamSynchronize(c->stream) != cudaSuccess) {
    spec_verify_destroy(c);
    return SPEC_ECUDA;
  }
  *out = c;
  return SPEC_OK;
}

void spec_verify_destroy(spec_ctx* c) {
  if (!c) return;
  cudaStreamSynchronize(c->stream);
  for (int i = 0; i < c->prof_cap; ++i) cudaEventDestroy(c->prof_ev[i]);
  free(c->prof_ev);
  cudaFree(c->act);
  cudaFree(c->pieces);
  cudaFree(c->resid);
  cudaFree(c->q8);
  cudaFree(c->da8);
  cudaFree(c->a8);
  cudaFree(c->rope_cs);
  cudaFree(c->qtile);
  cudaFree(c->logits_ws);
  cudaFree(c->sstats);
  cudaFree(c->sscratch);
  cudaFree(c->tree_mask);
  cudaFree(c->tscratch);
  for (auto& gc : c->graphs)
    if (gc.exec) cudaGraphExecDestroy(gc.exec);
  cudaFree(c->attn_part);
  cudaFree(c->head_val);
  cudaFree(c->head_idx);
  cudaFree(c->status);
  cudaFree(c->step_state);
  cudaFree(c->idx_buf);
  cudaFree(c->hidden_dev);
  cudaFree(c->draft_dev);
  cudaFree(c->res_dev);
  delete c;
}

int spec_set_stream(spec_ctx* c, void* cuda_stream) {
  if (!c) return SPEC_ENULL;
  c->stream = static_cast<cudaStream_t>(cuda_stream);
  return SPEC_OK;
}

int spec_last_step_launches(const spec_ctx* c) { return c ? c->last_launches : SPEC_ENULL; }

int spec_profile_gemms(spec_ctx* c, int enable) {
  if (!c) return SPEC_ENULL;
  if (enable && !c->prof_ev) {
    const int cap = 2 * (4 * c->cfg.n_layers + 1);
    c->prof_ev = static_cast<cudaEvent_t*>(calloc(cap, sizeof(cudaEvent_t)));
    if (!c->prof_ev) return SPEC_ENOMEM;
    for (int i = 0; i < cap; ++i)
      if (cudaEventCreate(&c->prof_ev[i]) != cudaSuccess) return SPEC_ECUDA;
    c->prof_cap = cap;
  }
  c->profile = enable != 0;
  return SPEC_OK;
}

int spec_profile_read(spec_ctx* c, float* gemm_ms, int* gemm_launches) {
  if (!c || !gemm_ms || !gemm_launches) return SPEC_ENULL;
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return SPEC_ECUDA;
  float tot = 0.f;
  for (int i = 0; i < c->prof_n; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, c->prof_ev[2 * i], c->prof_ev[2 * i + 1]) != cudaSuccess)
      return SPEC_ECUDA;
    tot += ms;
  }
  *gemm_ms = tot;
  *gemm_launches = c->prof_n;
  return SPEC_OK;
}

int spec_last_status(spec_ctx* c) {
  if (!c) return SPEC_ENULL;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, c->status, 4, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess ||
      cudaStreamSynchronize(c->stream) != cudaSuccess)
    return SPEC_ECUDA;
  if (cudaMemsetAsync(c->status, 0, 4, c->stream) != cudaSuccess) return SPEC_ECUDA;
  return v;
}

// ---------------------------------------------------------------------------
// building blocks
// ---------------------------------------------------------------------------
int spec_weights_repack(spec_ctx* c, const void* src, void* dst, int N, int K) {
  if (!c || !src || !dst) return SPEC_ENULL;
  if (N <= 0 || K <= 0 || N % 16 || K % 256) return SPEC_EINVAL;
  const size_t bytes = (size_t)N * (K / 256) * 144;
  const uint8_t* s = static_cast<const uint8_t*>(src);
  const uint8_t* d = static_cast<const uint8_t*>(dst);
  if (!(s + bytes <= d || d + bytes <= s)) return SPEC_EINVAL;
  if (!aligned(src) || !aligned(dst)) return SPEC_EALIGN;
  return cuda_code(launch_repack(src, dst, N, K, c->stream));
}

int spec_quantize_q8(spec_ctx* c, const float* x, int M, int K, int8_t* q, float* d_a, int32_t* A) {
  if (!c || !x || !q || !d_a || !A) return SPEC_ENULL;
  if (M < 1 || M > 16 || K <= 0 || K % 256) return SPEC_EINVAL;
  if ((size_t)(K / 256) * kActSBBytes > c->act_bytes) return SPEC_ECAPACITY;
  if (!aligned(x)) return SPEC_EALIGN;
  return cuda_code(launch_quantize(x, M, K, c->act, q, d_a, A, c->status, c->stream, false));
}

static int gemm_common(spec_ctx* c, const void* w, int N, int K, const float* x, int M, float* y,
                       int32_t* isc, int32_t* imn) {
  if (!c || !w || !x || !y) return SPEC_ENULL;
  if (M < 1 || M > 16 || N <= 0 || K <= 0 || N % 16 || K % 256) return SPEC_EINVAL;
  if ((size_t)(K / 256) * kActSBBytes > c->act_bytes) return SPEC_ECAPACITY;
  const GemmPlan p = make_gemm_plan(N, K, c->num_sms);
  if (pieces_need(p) > c->pieces_floats) return SPEC_ECAPACITY;
  if (!aligned(w) || !aligned(x)) return SPEC_EALIGN;
  SPEC_TRY(launch_quantize(x, M, K, c->act, nullptr, nullptr, nullptr, c->status, c->stream, false));
  SPEC_TRY(launch_gemm(p, w, c->act, c->pieces, isc, imn, M, c->status, c->stream, true));
  SPEC_TRY(launch_sum_pieces(p, c->pieces, y, M, c->stream, true));
  return SPEC_OK;
}

int spec_gemm_q4k(spec_ctx* c, const void* w, int N, int K, const float* x, int M, float* y) {
  return gemm_common(c, w, N, K, x, M, y, nullptr, nullptr);
}

int spec_gemm_q4k_sums(spec_ctx* c, const void* w, int N, int K, const float* x, int M, float* y,
                       int32_t* isc, int32_t* imn) {
  if (!isc || !imn) return SPEC_ENULL;
  return gemm_common(c, w, N, K, x, M, y, isc, imn);
}

int spec_gemm_wait_selftest(spec_ctx* c, const void* w, int N, int K) {
  if (!c || !w) return SPEC_ENULL;
  if (N <= 0 || K <= 0 || N % 16 || K % 256 || K > c->kmax) return SPEC_EINVAL;
  if (!aligned(w)) return SPEC_EALIGN;
  const GemmPlan p = make_gemm_plan(N, K, c->num_sms);
  if (pieces_need(p) > c->pieces_floats) return SPEC_ECAPACITY;
  SPEC_TRY(cudaMemsetAsync(c->status, 0, 4, c->stream));
  return cuda_code(launch_gemm(p, w, c->act, c->pieces, nullptr, nullptr, 0, c->status, c->stream, false, true));
}

int spec_gemm_q4k_cudacore(spec_ctx* c, const void* w, int N, int K, const float* x, int M, float* y) {
  if (!c || !w || !x || !y) return SPEC_ENULL;
  if (M < 1 || M > 16 || N <= 0 || K <= 0 || N % 16 || K % 256 || K > c->kmax) return SPEC_EINVAL;
  if (!aligned(w) || !aligned(x) || !aligned(y)) return SPEC_EALIGN;
  SPEC_TRY(cudaMemsetAsync(c->status, 0, 4, c->stream));
  SPEC_TRY(launch_quantize(x, M, K, c->act, c->q8, c->da8, c->a8, c->status, c->stream, false));
  return cuda_code(launch_gemm_dp4a(w, c->q8, c->da8, c->a8, M, N, K, y, c->num_sms, c->stream));
}

int spec_lm_head_argmax(spec_ctx* c, const void* w_head, const float* final_norm, const float* x,
                        int M, int32_t* idx, float* logits) {
  if (!c || !w_head || !x || !idx) return SPEC_ENULL;
  if (M < 1 || M > 16) return SPEC_EINVAL;
  if (!aligned(w_head) || !aligned(x) || (final_norm && !aligned(final_norm))) return SPEC_EALIGN;
  const spec_config& g = c->cfg;
  SPEC_TRY(launch_resid_norm_quant(nullptr, nullptr, x, nullptr, final_norm, g.rms_eps, M, g.hidden,
                                   c->act, nullptr, c->status, c->stream, false));
  SPEC_TRY(launch_gemm(c->p_head, w_head, c->act, c->pieces, nullptr, nullptr, 0, c->status, c->stream, true));
  SPEC_TRY(launch_head_argmax(c->p_head, c->pieces, M, logits, c->head_val, c->head_idx, c->status,
                              c->stream, true));
  SPEC_TRY(launch_argmax_final(c->head_val, c->head_idx, c->head_parts, M, idx, c->stream, true));
  return SPEC_OK;
}

int spec_attention(spec_ctx* c, const spec_kv* kv, int layer, const float* q, int M, float* out) {
  if (!c || !q || !out) return SPEC_ENULL;
  int rc = check_kv(kv);
  if (rc) return rc;
  if (M < 1 || M > 16 || layer < 0 || layer >= c->cfg.n_layers) return SPEC_EINVAL;
  const bool ring = swa_index(view_of(c, kv), layer) >= 0;
  if (ring) {
    rc = check_kv_swa(c, kv);
    if (rc) return rc;
  } else if (kv->max_seq_pages * c->cfg.page_size > c->attn.max_chunks * c->attn.chunk) {
    return SPEC_ECAPACITY;   // attention workspace must cover every position the cache can hold
  }
  if (!aligned(q) || !aligned(out)) return SPEC_EALIGN;
  const AttnPlan& ap = ring ? c->attn_swa : c->attn;
  SPEC_TRY(cudaMemsetAsync(c->status, 0, 4, c->stream));
  SPEC_TRY(launch_q_to_tile(q, M, ap, c->qtile, c->stream, false));
  SPEC_TRY(launch_attention(ap, view_of(c, kv), layer, c->qtile, M, c->attn_part, out, nullptr,
                            c->status, c->stream, false));
  return SPEC_OK;
}

int spec_accept(spec_ctx* c, const int32_t* idx, const int32_t* draft, int k, spec_kv* kv,
                spec_result* res) {
  if (!c || !idx || !draft || !res) return SPEC_ENULL;
  if (k != 3 && k != 7 && k != 15) return SPEC_EVERIFYLEN;
  if (kv) {
    int rc = check_kv(kv);
    if (rc) return rc;
    rc = check_kv_swa(c, kv);
    if (rc) return rc;
  }
  KvView v;
  if (kv) v = view_of(c, kv);
  return cuda_code(launch_accept(idx, nullptr, nullptr, 0, draft, k, c->cfg.vocab, kv ? &v : nullptr, nullptr,
                                c->status, reinterpret_cast<int32_t*>(res), nullptr, c->stream, false));
}

int spec_kv_reset(spec_ctx* c, spec_kv* kv) {
  if (!c) return SPEC_ENULL;
  int rc = check_kv(kv);
  if (rc) return rc;
  rc = check_kv_swa(c, kv);
  if (rc) return rc;
  return cuda_code(launch_kv_reset(view_of(c, kv), c->stream));
}

int spec_kv_extend(spec_ctx* c, spec_kv* kv, int32_t n) {
  if (!c) return SPEC_ENULL;
  int rc = check_kv(kv);
  if (rc) return rc;
  rc = check_kv_swa(c, kv);
  if (rc) return rc;
  if (n < 0) return SPEC_EINVAL;
  return cuda_code(launch_kv_reserve(view_of(c, kv), n, 1, nullptr, 0, 0, c->status, nullptr,
                                     c->stream, false));
}

int spec_kv_rollback(spec_ctx* c, spec_kv* kv, int32_t new_len) {
  if (!c) return SPEC_ENULL;
  int rc = check_kv(kv);
  if (rc) return rc;
  if (new_len < 0) return SPEC_EINVAL;
  rc = check_kv_swa(c, kv);
  if (rc) return rc;
  return cuda_code(launch_kv_rollback(view_of(c, kv), new_len, c->status, c->stream));
}

// ---------------------------------------------------------------------------
// the verify step
// ---------------------------------------------------------------------------
static int check_weights(const spec_ctx* c, const spec_weights* w) {
  if (!w || !w->w_qkv || !w->w_o || !w->w_gate_up || !w->w_down || !w->w_head) return SPEC_ENULL;
  for (int l = 0; l < c->cfg.n_layers; ++l) {
    if (!w->w_qkv[l] || !w->w_o[l] || !w->w_gate_up[l] || !w->w_down[l]) return SPEC_ENULL;
    if (!aligned(w->w_qkv[l]) || !aligned(w->w_o[l]) || !aligned(w->w_gate_up[l]) ||
        !aligned(w->w_down[l]))
      return SPEC_EALIGN;
    if (w->attn_norm && w->attn_norm[l] && !aligned(w->attn_norm[l])) return SPEC_EALIGN;
    if (w->ffn_norm && w->ffn_norm[l] && !aligned(w->ffn_norm[l])) return SPEC_EALIGN;
    if (w->q_norm && w->q_norm[l] && !aligned(w->q_norm[l])) return SPEC_EALIGN;
    if (w->k_norm && w->k_norm[l] && !aligned(w->k_norm[l])) return SPEC_EALIGN;
  }
  if (!aligned(w->w_head) || (w->final_norm && !aligned(w->final_norm))) return SPEC_EALIGN;
  return SPEC_OK;
}

// the draft's distributions and the MT19937 state of a sampled step
struct SampleArgs {
  const float* q;
  uint32_t* mt;
};
// a token tree: node tokens (tokens[0], the carried frontier's, is unused),
// parents, and where to write the accepted path
struct TreeArgs {
  const int32_t* tokens;
  const int32_t* parent;
  int32_t* path_out;
};

static int enqueue_step(spec_ctx* c, const spec_weights* w, spec_kv* kv, const float* hidden,
                        const int32_t* draft, int k, spec_result* res, const spec_taps* taps,
                        const SampleArgs* sa, const TreeArgs* ta = nullptr) {
  const int M = k + 1;

  const spec_config& g = c->cfg;
  const int H = g.hidden, F = g.ffn;
  cudaStream_t st = c->stream;
  const KvView kvv = view_of(c, kv);
  int n = 0;
  c->prof_n = 0;
  auto gemm = [&](const GemmPlan& p, const void* wt) -> cudaError_t {
    const bool prof = c->profile && 2 * c->prof_n + 1 < c->prof_cap;
    if (prof) {
      cudaError_t e = cudaEventRecord(c->prof_ev[2 * c->prof_n], st);
      if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_gemm(p, wt, c->act, c->pieces, nullptr, nullptr, 0, c->status, st, !prof);
    if (e != cudaSuccess) return e;
    if (prof) {
      e = cudaEventRecord(c->prof_ev[2 * c->prof_n + 1], st);
      ++c->prof_n;
    }
    return e;
  };
  auto attn_gamma = [&](int l) -> const float* { return w->attn_norm ? w->attn_norm[l] : nullptr; };
  auto ffn_gamma = [&](int l) -> const float* { return w->ffn_norm ? w->ffn_norm[l] : nullptr; };
  auto qk_of = [&](int l) {
    QkTransform t;
    t.gq = w->q_norm ? w->q_norm[l] : nullptr;
    t.gk = w->k_norm ? w->k_norm[l] : nullptr;
    t.cs = c->rope_cs;
    t.cs_len = g.max_ctx;
    t.eps = g.rms_eps;
    return t;
  };
  float* tap_resid = taps ? taps->resid : nullptr;

  // A token tree of more than max_rows nodes runs in passes of up to
  // max_rows rows, each streaming the weights once; every other step is one
  // pass over its M rows.
  const int P = ta ? (M < g.max_rows ? M : g.max_rows) : M;
  const int npass = (M + P - 1) / P;
  SPEC_TRY(launch_kv_reserve(kvv, M, 0, ta ? ta->tokens + 1 : draft, k, g.vocab, c->status, c->step_state, st,
                             true, ta ? ta->parent : nullptr, ta ? c->tree_mask : nullptr)); ++n;
  for (int pass = 0; pass < npass; ++pass) {
    const int r0 = pass * P, Mp = (M - r0 < P) ? M - r0 : P;
    const size_t rows_bytes = sizeof(float) * (size_t)Mp * H;
    const float* hid = hidden + (size_t)r0 * H;
    const uint64_t* tmask = ta ? c->tree_mask + r0 : nullptr;
    if (npass > 1) {
      SPEC_TRY(launch_tree_pass(kvv, c->step_state, c->status, r0 + Mp, st, true)); ++n;
    }
    if (tap_resid) SPEC_TRY(cudaMemcpyAsync(tap_resid, hid, rows_bytes, cudaMemcpyDeviceToDevice, st));
    SPEC_TRY(launch_resid_norm_quant(nullptr, nullptr, hid, c->resid, attn_gamma(0), g.rms_eps, Mp, H,
                                     c->act, nullptr, c->status, st, true)); ++n;
    for (int l = 0; l < g.n_layers; ++l) {
      SPEC_TRY(gemm(c->p_qkv, w->w_qkv[l])); ++n;
      // a sliding-window layer: K/V into its ring, attention over the window
      const AttnPlan& ap = swa_index(kvv, l) >= 0 ? c->attn_swa : c->attn;
      SPEC_TRY(launch_qkv_post(c->p_qkv, c->pieces, Mp, g.n_q_heads, g.n_kv_heads, g.head_dim, kvv, l, c->qtile,
                                ap.tiles, c->status, st, true, ap.early, qk_of(l))); ++n;
      SPEC_TRY(launch_attention(ap, kvv, l, c->qtile, Mp, c->attn_part, nullptr, c->act, c->status, st, true,
                                tmask, ta ? c->step_state : nullptr)); n += 2;
      SPEC_TRY(gemm(c->p_o, w->w_o[l])); ++n;
      SPEC_TRY(launch_resid_norm_quant(&c->p_o, c->pieces, c->resid, c->resid, ffn_gamma(l), g.rms_eps,
                                       Mp, H, c->act, nullptr, c->status, st, true)); ++n;
      SPEC_TRY(gemm(c->p_gu, w->w_gate_up[l])); ++n;
      SPEC_TRY(launch_swiglu_quant(c->p_gu, c->pieces, Mp, F, c->act, c->status, st, true)); ++n;
      SPEC_TRY(gemm(c->p_down, w->w_down[l])); ++n;
      const float* next_gamma = (l + 1 < g.n_layers) ? attn_gamma(l + 1) : w->final_norm;
      float* cap = nullptr;
      if (pass == 0)                           // the capture holds the first pass's rows
        for (int j = 0; j < c->cap_n; ++j)
          if (c->cap_ids[j] == l) cap = c->cap_rows + (size_t)j * H;
      SPEC_TRY(launch_resid_norm_quant(&c->p_down, c->pieces, c->resid, c->resid, next_gamma, g.rms_eps,
                                       Mp, H, c->act, nullptr, c->status, st, true, cap, c->cap_n * H)); ++n;
      if (tap_resid)
        SPEC_TRY(cudaMemcpyAsync(tap_resid + (size_t)(l + 1) * Mp * H, c->resid, rows_bytes,
                                 cudaMemcpyDeviceToDevice, st));
      // the prefix through block l is done (its output and capture rows are
      // written): another stream that waits on this event overlaps the suffix
      if (l == c->split_layer && c->split_ev && pass == npass - 1) {
        // inside a recorded graph the record is an external event node, which
        // streams outside the graph can wait on
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        SPEC_TRY(cudaStreamIsCapturing(st, &cs));
        SPEC_TRY(cudaEventRecordWithFlags(c->split_ev, st,
                                          cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                              : cudaEventRecordDefault));
      }
    }
    SPEC_TRY(gemm(c->p_head, w->w_head)); ++n;
    if (ta) {
      // every node's argmax; the decision follows the last pass
      SPEC_TRY(launch_head_argmax(c->p_head, c->pieces, Mp,
                                  taps && taps->logits ? taps->logits + (size_t)r0 * g.vocab : nullptr,
                                  c->head_val, c->head_idx, c->status, st, true)); ++n;
      SPEC_TRY(launch_argmax_final(c->head_val, c->head_idx, c->head_parts, Mp, c->idx_buf + r0, st, true)); ++n;
    }
  }
  if (ta) {
    // token tree: the accepted path over all nodes, its K/V moves, the rollback
    if (npass > 1) {
      SPEC_TRY(launch_tree_pass(kvv, c->step_state, c->status, M, st, true)); ++n;
    }
    SPEC_TRY(launch_tree_accept(c->idx_buf, ta->tokens, ta->parent, M, g.vocab, kvv, c->step_state, c->tscratch,
                                c->status, reinterpret_cast<int32_t*>(res), ta->path_out,
                                taps ? taps->argmax : nullptr, st, true));
    n += 3;
  } else if (sa) {
    // sampled acceptance: the logits of every row, their normalizers, then
    // the decisions on the caller's MT19937 stream
    SPEC_TRY(launch_head_argmax(c->p_head, c->pieces, M, c->logits_ws, c->head_val, c->head_idx,
                                c->status, st, true)); ++n;
    if (taps && taps->argmax) {
      SPEC_TRY(launch_argmax_final(c->head_val, c->head_idx, c->head_parts, M, taps->argmax, st, true));
      ++n;
    }
    if (taps && taps->logits)
      SPEC_TRY(cudaMemcpyAsync(taps->logits, c->logits_ws, sizeof(float) * (size_t)M * g.vocab,
                               cudaMemcpyDeviceToDevice, st));
    SPEC_TRY(launch_sample_accept(c->logits_ws, sa->q, draft, k, g.vocab, c->sstats, c->sscratch, sa->mt,
                                  &kvv, c->step_state, c->status, reinterpret_cast<int32_t*>(res), st, true));
    n += 4;
  } else {
    SPEC_TRY(launch_head_argmax(c->p_head, c->pieces, M, taps ? taps->logits : nullptr, c->head_val,
                                c->head_idx, c->status, st, true)); ++n;
    SPEC_TRY(launch_accept(nullptr, c->head_val, c->head_idx, c->head_parts, draft, k, g.vocab, &kvv,
                           c->step_state, c->status, reinterpret_cast<int32_t*>(res),
                           taps ? taps->argmax : nullptr, st, true)); ++n;
  }
  c->last_launches = n;
  return SPEC_OK;
}

static uint64_t mix(uint64_t h, uint64_t v) {
  h ^= v + 0x9e3779b97f4a7c15ull + (h << 6) + (h >> 2);
  return h;
}

static uint64_t step_key(const spec_ctx* c, const spec_weights* w, const spec_kv* kv,
                         const float* hidden, const int32_t* draft, int k, const spec_result* res,
                         const SampleArgs* sa, const TreeArgs* ta) {
  uint64_t h = 0x1234567ull;
  auto P = [](const void* p) { return (uint64_t)(uintptr_t)p; };
  h = mix(h, sa ? 0x5a ^ P(sa->q) : 0x9e);
  h = mix(h, sa ? P(sa->mt) : 0);
  h = mix(h, P(c->cap_rows));
  h = mix(h, ta ? 0x7e ^ P(ta->tokens) : 0x31);
  h = mix(h, ta ? P(ta->parent) : 0);
  h = mix(h, ta ? P(ta->path_out) : 0);
  for (int j = 0; j < c->cap_n; ++j) h = mix(h, 0x100 + (uint64_t)c->cap_ids[j]);
  h = mix(h, 0x200 + (uint64_t)(c->split_layer + 1));
  h = mix(h, P(c->split_ev));
  h = mix(h, P(hidden));
  h = mix(h, P(draft));
  h = mix(h, P(res));
  h = mix(h, (uint64_t)k);
  h = mix(h, P(kv->pool));
  h = mix(h, P(kv->page_table));
  h = mix(h, P(kv->seq_len));
  h = mix(h, P(kv->free_stack));
  h = mix(h, P(kv->free_top));
  h = mix(h, (uint64_t)kv->num_pages);
  h = mix(h, (uint64_t)kv->max_seq_pages);
  h = mix(h, P(kv->swa_ring));
  h = mix(h, P(kv->swa_state));
  for (int l = 0; l < c->cfg.n_layers; ++l) {
    h = mix(h, P(w->w_qkv[l]));
    h = mix(h, P(w->w_o[l]));
    h = mix(h, P(w->w_gate_up[l]));
    h = mix(h, P(w->w_down[l]));
    h = mix(h, w->attn_norm ? P(w->attn_norm[l]) : 1);
    h = mix(h, w->ffn_norm ? P(w->ffn_norm[l]) : 2);
    h = mix(h, w->q_norm ? P(w->q_norm[l]) : 3);
    h = mix(h, w->k_norm ? P(w->k_norm[l]) : 4);
  }
  h = mix(h, P(w->final_norm));
  h = mix(h, P(w->w_head));
  return h | 1;
}

static int run_step(spec_ctx* c, const spec_weights* w, spec_kv* kv, const float* hidden,
                    const int32_t* draft, int k, spec_result* res, const spec_taps* taps,
                    const SampleArgs* sa, const TreeArgs* ta = nullptr) {
  if (!c || !hidden || !draft || !res) return SPEC_ENULL;
  if (ta ? (k < 0 || k > kTreeMax - 1) : (k != 3 && k != 7 && k != 15)) return SPEC_EVERIFYLEN;
  const int M = k + 1;
  // a tree larger than max_rows runs in passes; the residual taps hold one pass
  if (!ta && M > c->cfg.max_rows) return SPEC_ECAPACITY;
  if (ta && M > c->cfg.max_rows && taps && taps->resid) return SPEC_EINVAL;
  int rc = check_kv(kv);
  if (rc) return rc;
  rc = check_kv_swa(c, kv);
  if (rc) return rc;
  if (ta && has_swa(c->cfg)) return SPEC_EINVAL;   // K/V moves of a tree path: paged layers only
  if (ta && c->cfg.rope_theta > 0.f) return SPEC_EINVAL;   // a tree row's position is its depth
  rc = check_weights(c, w);
  if (rc) return rc;
  if (!aligned(hidden)) return SPEC_EALIGN;
  if (kv->max_seq_pages * c->cfg.page_size > c->attn.max_chunks * c->attn.chunk)
    return SPEC_ECAPACITY;   // attention workspace must cover every position the cache can hold

  // Steps with taps, with GEMM profiling, or on the legacy default stream
  // (which cannot be captured) are enqueued directly.
  if (taps || c->profile || !c->use_graphs || c->stream == nullptr)
    return enqueue_step(c, w, kv, hidden, draft, k, res, taps, sa, ta);

  const uint64_t key = step_key(c, w, kv, hidden, draft, k, res, sa, ta);
  spec_ctx::GraphEntry* hit = nullptr;
  for (auto& gc : c->graphs)
    if (gc.exec && gc.key == key) hit = &gc;
  if (!hit) {
    // record the step once: a one-time host-side graph build for this argument set
    spec_ctx::GraphEntry* victim = &c->graphs[0];
    for (auto& gc : c->graphs)
      if (!gc.exec || gc.used < victim->used) victim = &gc;
    if (victim->exec) {
      cudaGraphExecDestroy(victim->exec);
      victim->exec = nullptr;
    }
    cudaGraph_t graph = nullptr;
    SPEC_TRY(cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal));
    rc = enqueue_step(c, w, kv, hidden, draft, k, res, nullptr, sa, ta);
    cudaError_t e = cudaStreamEndCapture(c->stream, &graph);
    if (rc != SPEC_OK) {
      if (graph) cudaGraphDestroy(graph);
      return rc;
    }
    if (e != cudaSuccess) return SPEC_ECUDA;
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return SPEC_ECUDA;
    victim->exec = exec;
    victim->key = key;
    victim->launches = c->last_launches;
    hit = victim;
  }
  hit->used = ++c->graph_clock;
  c->last_launches = hit->launches;
  SPEC_TRY(cudaGraphLaunch(hit->exec, c->stream));
  return SPEC_OK;
}

int spec_verify_step_ex(spec_ctx* c, const spec_weights* w, spec_kv* kv, const float* hidden,
                        const int32_t* draft, int k, spec_result* res, const spec_taps* taps) {
  return run_step(c, w, kv, hidden, draft, k, res, taps, nullptr);
}

int spec_verify_step(spec_ctx* c, const spec_weights* w, spec_kv* kv, const float* hidden,
                     const int32_t* draft, int k, spec_result* res) {
  return run_step(c, w, kv, hidden, draft, k, res, nullptr, nullptr);
}

int spec_verify_tree(spec_ctx* c, const spec_weights* w, spec_kv* kv, const float* hidden,
                     const int32_t* tokens, const int32_t* parent, int n, spec_result* res,
                     int32_t* path_out, const spec_taps* taps) {
  if (!tokens || !parent) return SPEC_ENULL;
  if (n < 1 || n > kTreeMax) return SPEC_EVERIFYLEN;
  const TreeArgs ta{tokens, parent, path_out};
  return run_step(c, w, kv, hidden, tokens, n - 1, res, taps, nullptr, &ta);
}

int spec_verify_step_sampled(spec_ctx* c, const spec_weights* w, spec_kv* kv, const float* hidden,
                             const int32_t* draft, const float* q, int k, uint32_t* mt,
                             spec_result* res, const spec_taps* taps) {
  if (!q || !mt) return SPEC_ENULL;
  if (!aligned(q) || !aligned(mt)) return SPEC_EALIGN;
  const SampleArgs sa{q, mt};
  return run_step(c, w, kv, hidden, draft, k, res, taps, &sa);
}

int spec_set_capture(spec_ctx* c, const int32_t* layer_ids, int n, float* rows) {
  if (!c) return SPEC_ENULL;
  if (n < 0 || n > 8) return SPEC_EINVAL;
  if (n > 0 && (!layer_ids || !rows)) return SPEC_ENULL;
  if (n > 0 && !aligned(rows)) return SPEC_EALIGN;
  for (int j = 0; j < n; ++j) {
    if (layer_ids[j] < 0 || layer_ids[j] >= c->cfg.n_layers) return SPEC_EINVAL;
    for (int i = 0; i < j; ++i)
      if (layer_ids[i] == layer_ids[j]) return SPEC_EINVAL;
  }
  c->cap_n = n;
  for (int j = 0; j < n; ++j) c->cap_ids[j] = layer_ids[j];
  c->cap_rows = n > 0 ? rows : nullptr;
  return SPEC_OK;
}

int spec_set_split(spec_ctx* c, int layer, void* cuda_event) {
  if (!c) return SPEC_ENULL;
  if (layer < -1 || layer >= c->cfg.n_layers) return SPEC_EINVAL;
  if (layer >= 0 && !cuda_event) return SPEC_ENULL;
  c->split_layer = layer;
  c->split_ev = layer >= 0 ? static_cast<cudaEvent_t>(cuda_event) : nullptr;
  return SPEC_OK;
}

int spec_gemm_ranges(int N, int K, int num_sms) {
  if (N <= 0 || N % 16 != 0 || K <= 0 || K % 256 != 0 || num_sms <= 0) return SPEC_EINVAL;
  return make_gemm_plan(N, K, num_sms).G;
}

// MT19937 seeding (Matsumoto & Nishimura 1998): word 0 = seed, word i =
// 1812433253 * (w[i-1] ^ (w[i-1] >> 30)) + i; word 624 = 624 (regenerate first)
int spec_mt_seed(uint32_t* state_host, uint32_t seed) {
  if (!state_host) return SPEC_ENULL;
  state_host[0] = seed;
  for (uint32_t i = 1; i < 624; ++i)
    state_host[i] = 1812433253u * (state_host[i - 1] ^ (state_host[i - 1] >> 30)) + i;
  state_host[624] = 624;
  return SPEC_OK;
}

int spec_sample_accept(spec_ctx* c, const float* logits, const float* q, const int32_t* draft, int k,
                       uint32_t* mt, spec_kv* kv, spec_result* res) {
  if (!c || !logits || !q || !draft || !mt || !res) return SPEC_ENULL;
  if (k < 1 || k > 15) return SPEC_EVERIFYLEN;
  if (!aligned(logits) || !aligned(q) || !aligned(mt)) return SPEC_EALIGN;
  if (kv) {
    int rc = check_kv(kv);
    if (rc) return rc;
    rc = check_kv_swa(c, kv);
    if (rc) return rc;
  }
  KvView v;
  if (kv) v = view_of(c, kv);
  return cuda_code(launch_sample_accept(logits, q, draft, k, c->cfg.vocab, c->sstats, c->sscratch, mt,
                                       kv ? &v : nullptr, nullptr, c->status, reinterpret_cast<int32_t*>(res),
                                       c->stream, false));
}

int spec_verify_step_host(spec_ctx* c, const spec_weights* w, spec_kv* kv, const float* hidden_host,
                          const int32_t* draft_host, int k, spec_result* res_host) {
  if (!c || !hidden_host || !draft_host || !res_host) return SPEC_ENULL;
  if (k != 3 && k != 7 && k != 15) return SPEC_EVERIFYLEN;
  if (k + 1 > c->cfg.max_rows) return SPEC_ECAPACITY;
  const size_t hb = sizeof(float) * (size_t)(k + 1) * c->cfg.hidden;
  SPEC_TRY(cudaMemcpyAsync(c->hidden_dev, hidden_host, hb, cudaMemcpyHostToDevice, c->stream));
  SPEC_TRY(cudaMemcpyAsync(c->draft_dev, draft_host, sizeof(int32_t) * k, cudaMemcpyHostToDevice,
                           c->stream));
  int rc = spec_verify_step(c, w, kv, c->hidden_dev, c->draft_dev, k, c->res_dev);
  if (rc) return rc;
  SPEC_TRY(cudaMemcpyAsync(res_host, c->res_dev, sizeof(spec_result), cudaMemcpyDeviceToHost,
                           c->stream));
  SPEC_TRY(cudaStreamSynchronize(c->stream));
  return SPEC_OK;
}

}  // extern "C"
