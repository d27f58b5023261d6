// The C ABI (include/tv.h): host-side argument checks, the workspace layout and
// the launch sequence of each entry point.  Everything runs on the caller's
// stream; nothing here allocates device memory.
#include <cmath>
#include <cstring>

#include "tv_common.cuh"
#include "tv_gemm.cuh"
#include "tv_kernels.cuh"

namespace tv {
namespace {

constexpr int kMaxHeadGrid = 1024;   // top-2 partial rows reserved in the workspace

struct WsLayout {
  size_t rstats, meta, counter, h, q, part_qkv, attn_ml, attn_o, attn, part_o, hf, top2, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The residual walk's statistics come first, so that tv_accept_residual needs
// only the vocabulary to find them.
WsLayout ws_layout(const tv_dims& d) {
  WsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const size_t H = d.hidden, QD = (size_t)d.n_q_heads * d.head_dim;
  const size_t QKV = (size_t)(d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
  const GemmPlan pq = plan_gemm((int)QKV, (int)H, false);
  const GemmPlan po = plan_gemm((int)H, (int)QD, false);
  L.rstats = take((size_t)kMaxRows * n_vchunks(d.vocab) * sizeof(RowStat));
  L.meta = take(kMaxRows * sizeof(RowMeta));
  L.counter = take(256);
  L.h = take(kMaxRows * H * 2);
  L.q = take(kMaxRows * QD * 2);
  L.part_qkv = take((size_t)pq.splits * kMaxRows * QKV * 4);
  L.attn_ml = take((size_t)kMaxRows * d.n_q_heads * kChunkSlots * 2 * 4);
  L.attn_o = take((size_t)kMaxRows * d.n_q_heads * kChunkSlots * d.head_dim * 4);
  L.attn = take(kMaxRows * QD * 2);
  L.part_o = take((size_t)po.splits * kMaxRows * H * 4);
  L.hf = take(kMaxRows * H * 2);
  L.top2 = take((size_t)kMaxHeadGrid * 32 * sizeof(Top2));
  L.total = off;
  return L;
}

int check_dims(const tv_dims& d) {
  if (d.hidden <= 0 || d.n_q_heads <= 0 || d.n_kv_heads <= 0 || d.head_dim <= 0 || d.vocab < 2) return TV_E_ARG;
  if (!(d.rms_eps >= 0.f) || !(d.rope_theta > 0.f) || !std::isfinite(d.rope_theta)) return TV_E_ARG;
  if (d.head_dim != 64 && d.head_dim != 128) return TV_E_UNSUPPORTED;
  if (d.hidden % 64 != 0 || (d.n_q_heads * d.head_dim) % 64 != 0) return TV_E_UNSUPPORTED;
  if (d.n_q_heads % d.n_kv_heads != 0) return TV_E_UNSUPPORTED;
  return TV_OK;
}

int num_sms() {
  static std::atomic<int> cache[64];   // 0 = not read yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

// ---- optional stage timing (tv_profile_*) ----------------------------------
struct Profile {
  int cap = 0;       // calls that can be recorded
  int calls = 0;     // calls recorded so far
  cudaEvent_t* ev = nullptr;   // [cap][TV_PROFILE_STAGES + 1]
};
Profile g_prof;

struct StageMarks {
  cudaStream_t st;
  cudaEvent_t* ev = nullptr;
  explicit StageMarks(cudaStream_t s) : st(s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (g_prof.ev && g_prof.calls < g_prof.cap && cudaStreamIsCapturing(s, &cs) == cudaSuccess &&
        cs == cudaStreamCaptureStatusNone)
      ev = g_prof.ev + (size_t)(g_prof.calls++) * (TV_PROFILE_STAGES + 1);
  }
  void mark(int i) {
    if (ev) cudaEventRecord(ev[i], st);
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Fills the request table from host structs.  kv may be null (walks).
int build_table(ReqTable& t, const tv_tree* trees, const tv_kv* kv, int n_req, bool need_parent) {
  if (!trees || n_req < 1 || n_req > kMaxReq) return n_req < 1 || n_req > kMaxReq ? TV_E_ROWS : TV_E_ARG;
  memset(&t, 0, sizeof(t));
  t.n_req = n_req;
  int total = 0;
  for (int r = 0; r < n_req; ++r) {
    const int n = trees[r].n;
    if (n < 1 || n > kMaxRows) return TV_E_ROWS;
    t.row_off[r] = total;
    t.n[r] = n;
    total += n;
    if (total > kMaxRows) return TV_E_ROWS;
    if (need_parent && (!trees[r].parent || !trees[r].token)) return TV_E_ARG;
    t.parent[r] = trees[r].parent;
    t.token[r] = trees[r].token;
    if (kv) {
      if (!kv[r].k || !kv[r].v || !aligned16(kv[r].k) || !aligned16(kv[r].v)) return TV_E_ARG;
      if (kv[r].ctx_len < 0 || kv[r].capacity < 0) return TV_E_ARG;
      if ((long long)kv[r].ctx_len + n > (long long)kv[r].capacity) return TV_E_CAPACITY;
      t.ctx[r] = kv[r].ctx_len;
      t.capacity[r] = kv[r].capacity;
      t.k[r] = reinterpret_cast<__nv_bfloat16*>(kv[r].k);
      t.v[r] = reinterpret_cast<__nv_bfloat16*>(kv[r].v);
    }
  }
  t.row_off[n_req] = total;
  t.total_rows = total;
  return TV_OK;
}

}  // namespace tv

using namespace tv;

extern "C" {

int tv_workspace_size(const tv_dims* dims, int max_rows, int max_ctx, size_t* bytes) {
  if (!dims || !bytes || max_rows < 0 || max_ctx < 0) return TV_E_ARG;
  if (max_rows > kMaxRows) return TV_E_ROWS;
  const int rc = check_dims(*dims);
  if (rc) return rc;
  *bytes = ws_layout(*dims).total;
  return TV_OK;
}

int tv_verify_tree(const tv_model* model, const tv_kv* kv, const tv_tree* trees, int n_req, float* logits,
                   int32_t* argmax, float* top2_gap, tv_bf16* attn_out, void* workspace, size_t workspace_bytes,
                   int32_t* dev_status, void* stream) {
  if (!model || !kv || !trees || !logits || !argmax || !top2_gap || !dev_status) return TV_E_ARG;
  const tv_dims& d = model->dims;
  int rc = check_dims(d);
  if (rc) return rc;
  if (!model->embed || !model->ln1 || !model->wqkv || !model->wo || !model->ln_f || !model->lm_head)
    return TV_E_ARG;
  if (!aligned16(model->wqkv) || !aligned16(model->wo) || !aligned16(model->lm_head)) return TV_E_ARG;
  if (model->packed != 0 && model->packed != 1) return TV_E_ARG;
  ReqTable t;
  rc = build_table(t, trees, kv, n_req, true);
  if (rc) return rc;
  const int G = d.n_q_heads / d.n_kv_heads;
  for (int r = 0; r < n_req; ++r)
    if (G * t.n[r] > kMaxQueriesPerKvHead) return TV_E_UNSUPPORTED;
  const WsLayout L = ws_layout(d);
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return TV_E_WORKSPACE;
  if (attn_out && !aligned16(attn_out)) return TV_E_ARG;
  const int sms = num_sms();
  if (sms <= 0) return TV_E_CUDA;
  if (sms > kMaxHeadGrid) return TV_E_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  LayerBufs b;
  b.meta = reinterpret_cast<RowMeta*>(ws + L.meta);
  b.head_counter = reinterpret_cast<unsigned int*>(ws + L.counter);
  b.h = reinterpret_cast<__nv_bfloat16*>(ws + L.h);
  b.q = reinterpret_cast<__nv_bfloat16*>(ws + L.q);
  b.part_qkv = reinterpret_cast<float*>(ws + L.part_qkv);
  b.attn_ml = reinterpret_cast<float*>(ws + L.attn_ml);
  b.attn_o = reinterpret_cast<float*>(ws + L.attn_o);
  b.attn = attn_out ? reinterpret_cast<__nv_bfloat16*>(attn_out) : reinterpret_cast<__nv_bfloat16*>(ws + L.attn);
  b.part_o = reinterpret_cast<float*>(ws + L.part_o);
  b.hf = reinterpret_cast<__nv_bfloat16*>(ws + L.hf);

  const int H = d.hidden, QD = d.n_q_heads * d.head_dim;
  const int QKV = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
  const GemmPlan pq = plan_gemm(QKV, H, false);
  const GemmPlan po = plan_gemm(H, QD, false);
  const GemmPlan ph = plan_gemm(d.vocab, H, true);
  GemmParams gp;
  memset(&gp, 0, sizeof(gp));
  gp.status = dev_status;
  gp.packed = model->packed ? 1 : 0;

  StageMarks pm(st);
  pm.mark(0);
  if ((rc = launch_prologue_embed(t, d, model->embed, model->ln1, b, nullptr, dev_status, st))) return rc;
  pm.mark(1);
  gp.out = b.part_qkv;
  if ((rc = launch_gemm(GEMM_PARTIAL, model->wqkv, QKV, H, b.h, t.total_rows, pq, gp, sms, st))) return rc;
  pm.mark(2);
  if ((rc = launch_qkv_finalize(t, d, b, pq.splits, dev_status, st))) return rc;
  pm.mark(3);
  if ((rc = launch_attention(t, d, b, sms, dev_status, st))) return rc;
  pm.mark(4);
  gp.out = b.part_o;
  if ((rc = launch_gemm(GEMM_PARTIAL, model->wo, H, QD, b.attn, t.total_rows, po, gp, sms, st))) return rc;
  pm.mark(5);
  if ((rc = launch_o_finalize(t, *model, b, po.splits, dev_status, st))) return rc;
  pm.mark(6);
  gp.out = logits;
  gp.top2_part = reinterpret_cast<Top2*>(ws + L.top2);
  gp.done_counter = b.head_counter;
  gp.argmax = argmax;
  gp.gap = top2_gap;
  rc = launch_gemm(GEMM_HEAD, model->lm_head, d.vocab, H, b.hf, t.total_rows, ph, gp, sms, st);
  pm.mark(7);
  return rc;
}

int tv_accept_greedy(const tv_tree* trees, int n_req, const int32_t* argmax, int32_t* path, int32_t* accept_len,
                     int32_t* out_tokens, int32_t* dev_status, void* stream) {
  if (!argmax || !path || !accept_len || !out_tokens || !dev_status) return TV_E_ARG;
  ReqTable t;
  const int rc = build_table(t, trees, nullptr, n_req, true);
  if (rc) return rc;
  return launch_accept_greedy(t, argmax, path, accept_len, out_tokens, dev_status,
                              reinterpret_cast<cudaStream_t>(stream));
}

int tv_accept_residual(const tv_tree* trees, int n_req, const float* logits, int32_t vocab, float temperature,
                       const float* uniforms, int bonus_at_leaf, int32_t* path, int32_t* accept_len,
                       int32_t* out_tokens, int32_t* out_count, int32_t* dev_status, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!(std::isfinite(temperature) && temperature > 0.f)) return TV_E_TEMP;
  if (!logits || !uniforms || !path || !accept_len || !out_tokens || !out_count || !dev_status || vocab < 2)
    return TV_E_ARG;
  ReqTable t;
  const int rc = build_table(t, trees, nullptr, n_req, true);
  if (rc) return rc;
  const size_t need = align256((size_t)kMaxRows * n_vchunks(vocab) * sizeof(RowStat));
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return TV_E_WORKSPACE;
  return launch_accept_residual(t, logits, vocab, temperature, uniforms, bonus_at_leaf ? 1 : 0,
                                static_cast<RowStat*>(workspace), path, accept_len, out_tokens, out_count,
                                dev_status, reinterpret_cast<cudaStream_t>(stream));
}

// ---- sampled variants -------------------------------------------------------------
namespace {
struct SampleWs {   // byte offsets in the sampled entry points' workspace
  size_t stats, gumbel, rej, total;
};
SampleWs sample_ws(int vocab, int rows) {
  const size_t nvc = (size_t)n_vchunks(vocab);
  SampleWs w;
  w.stats = 0;
  w.gumbel = align256(w.stats + rows * nvc * sizeof(RowStat));
  w.rej = align256(w.gumbel + rows * nvc * sizeof(GumbelPart));
  w.total = align256(w.rej + rows * nvc * sizeof(RejStat));
  return w;
}
}  // namespace

int tv_sample_workspace_size(int32_t vocab, int max_rows, size_t* bytes) {
  if (!bytes || vocab < 2) return TV_E_ARG;
  if (max_rows < 1 || max_rows > kMaxRows) return TV_E_ROWS;
  *bytes = sample_ws(vocab, max_rows).total;
  return TV_OK;
}

int tv_sample_filter(const float* logits, float* filtered, int rows, int32_t vocab, float temperature, int32_t top_k,
                     float top_p, float min_p, int32_t* dev_status, void* stream) {
  if (!(std::isfinite(temperature) && temperature > 0.f)) return TV_E_TEMP;
  if (!logits || !filtered || logits == filtered || !dev_status || vocab < 2 || rows < 1 || rows > kMaxRows)
    return TV_E_ARG;
  if (top_k < 0 || !(top_p > 0.f && top_p <= 1.f) || !(min_p >= 0.f && min_p < 1.f)) return TV_E_ARG;
  return launch_filter(logits, filtered, rows, vocab, temperature, top_k, top_p, min_p, dev_status,
                       reinterpret_cast<cudaStream_t>(stream));
}

int tv_accept_single_draw(const tv_tree* trees, int n_req, const float* logits, int32_t vocab, float temperature,
                          const float* uniforms, int32_t* row_tokens, int32_t* path, int32_t* accept_len,
                          int32_t* out_tokens, int32_t* dev_status, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (!(std::isfinite(temperature) && temperature > 0.f)) return TV_E_TEMP;
  if (!logits || !uniforms || !row_tokens || !path || !accept_len || !out_tokens || !dev_status || vocab < 2)
    return TV_E_ARG;
  ReqTable t;
  int rc = build_table(t, trees, nullptr, n_req, true);
  if (rc) return rc;
  const SampleWs w = sample_ws(vocab, t.total_rows);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return TV_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  rc = launch_draw_rows(t, logits, vocab, temperature, uniforms, reinterpret_cast<RowStat*>(ws + w.stats), row_tokens,
                        dev_status, st);
  if (rc) return rc;
  return launch_accept_greedy(t, row_tokens, path, accept_len, out_tokens, dev_status, st);
}

int tv_accept_gumbel(const tv_tree* trees, int n_req, const float* logits, int32_t vocab, float temperature,
                     const uint64_t* seeds, const int32_t* positions, int32_t* row_tokens, int32_t* path,
                     int32_t* accept_len, int32_t* out_tokens, int32_t* dev_status, void* workspace,
                     size_t workspace_bytes, void* stream) {
  if (!(std::isfinite(temperature) && temperature > 0.f)) return TV_E_TEMP;
  if (!logits || !seeds || !positions || !row_tokens || !path || !accept_len || !out_tokens || !dev_status ||
      vocab < 2)
    return TV_E_ARG;
  ReqTable t;
  int rc = build_table(t, trees, nullptr, n_req, true);
  if (rc) return rc;
  SeedTable sd;
  memset(&sd, 0, sizeof(sd));
  for (int r = 0; r < n_req; ++r) {
    if (positions[r] < 0) return TV_E_ARG;
    sd.seed[r] = seeds[r];
    sd.pos[r] = positions[r];
  }
  const SampleWs w = sample_ws(vocab, t.total_rows);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return TV_E_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  rc = launch_gumbel_rows(t, logits, vocab, temperature, sd, reinterpret_cast<GumbelPart*>(ws + w.gumbel), row_tokens,
                          dev_status, st);
  if (rc) return rc;
  return launch_accept_greedy(t, row_tokens, path, accept_len, out_tokens, dev_status, st);
}

int tv_accept_rejection(const tv_tree* trees, int n_req, const float* logits, int32_t vocab, float temperature,
                        const float* proposals, const float* uniforms, int32_t* path, int32_t* accept_len,
                        int32_t* out_tokens, int32_t* out_count, int32_t* dev_status, void* workspace,
                        size_t workspace_bytes, void* stream) {
  if (!(std::isfinite(temperature) && temperature > 0.f)) return TV_E_TEMP;
  if (!logits || !proposals || !uniforms || !path || !accept_len || !out_tokens || !out_count || !dev_status ||
      vocab < 2)
    return TV_E_ARG;
  ReqTable t;
  const int rc = build_table(t, trees, nullptr, n_req, true);
  if (rc) return rc;
  const SampleWs w = sample_ws(vocab, t.total_rows);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return TV_E_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return launch_accept_rejection(t, logits, vocab, temperature, proposals, uniforms,
                                 reinterpret_cast<RowStat*>(ws + w.stats), reinterpret_cast<RejStat*>(ws + w.rej),
                                 path, accept_len, out_tokens, out_count, dev_status,
                                 reinterpret_cast<cudaStream_t>(stream));
}

// ---- Gated DeltaNet -----------------------------------------------------------------
namespace {
int dn_check(const tv_dn_dims* d) {
  if (!d) return TV_E_ARG;
  if (d->n_k_heads < 1 || d->n_v_heads < 1 || d->n_v_heads % d->n_k_heads != 0) return TV_E_UNSUPPORTED;
  auto ok = [](int x) { return x >= 32 && x <= kDnMaxDim && x % 32 == 0; };
  if (!ok(d->d_k) || !ok(d->d_v)) return TV_E_UNSUPPORTED;
  return TV_OK;
}
int dn_states(DnStates& st, float* const* states, int n_req) {
  if (!states) return TV_E_ARG;
  memset(&st, 0, sizeof(st));
  for (int r = 0; r < n_req; ++r) {
    if (!states[r] || !aligned16(states[r])) return TV_E_ARG;
    st.S[r] = states[r];
  }
  return TV_OK;
}
}  // namespace

int tv_dn_verify_tree(const tv_dn_dims* dims, const tv_tree* trees, int n_req, float* const* states, const float* q,
                      const float* k, const float* v, const float* beta, const float* g, float* o, float* u,
                      float* gc, int32_t* dev_status, void* stream) {
  int rc = dn_check(dims);
  if (rc) return rc;
  if (!q || !k || !v || !beta || !g || !o || !u || !gc || !dev_status) return TV_E_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return TV_E_ARG;
  ReqTable t;
  if ((rc = build_table(t, trees, nullptr, n_req, true))) return rc;
  DnStates st;
  if ((rc = dn_states(st, states, n_req))) return rc;
  return launch_dn_verify(t, st, dims->n_k_heads, dims->n_v_heads, dims->d_k, dims->d_v, q, k, v, beta, g, o, u, gc,
                          dev_status, reinterpret_cast<cudaStream_t>(stream));
}

int tv_dn_commit(const tv_dn_dims* dims, const tv_tree* trees, int n_req, int n_layers, float* const* states,
                 const float* k, const float* u, const float* gc, const int32_t* path, const int32_t* accept_len,
                 int32_t* dev_status, void* stream) {
  int rc = dn_check(dims);
  if (rc) return rc;
  if (n_layers < 1 || !k || !u || !gc || !path || !accept_len || !dev_status) return TV_E_ARG;
  if (!aligned16(k) || !aligned16(u)) return TV_E_ARG;
  ReqTable t;
  if ((rc = build_table(t, trees, nullptr, n_req, true))) return rc;
  DnStates st;
  if ((rc = dn_states(st, states, n_req))) return rc;
  return launch_dn_commit(t, st, dims->n_k_heads, dims->n_v_heads, dims->d_k, dims->d_v, n_layers, k, u, gc, path,
                          accept_len, dev_status, reinterpret_cast<cudaStream_t>(stream));
}

int tv_commit_kv(const tv_kv* kv, const tv_dims* dims, const tv_tree* trees, int n_req, const int32_t* path,
                 const int32_t* accept_len, int32_t* committed_src, int32_t* new_ctx, int32_t* dev_status,
                 void* stream) {
  if (!kv || !dims || !path || !accept_len || !committed_src || !new_ctx || !dev_status) return TV_E_ARG;
  if (dims->n_kv_heads <= 0 || (dims->head_dim != 64 && dims->head_dim != 128)) return TV_E_UNSUPPORTED;
  ReqTable t;
  const int rc = build_table(t, trees, kv, n_req, false);
  if (rc) return rc;
  return launch_commit(t, *dims, path, accept_len, committed_src, new_ctx, dev_status,
                       reinterpret_cast<cudaStream_t>(stream));
}

int tv_accept_greedy_commit(const tv_kv* kv, const tv_dims* dims, const tv_tree* trees, int n_req,
                            const int32_t* argmax, int32_t* path, int32_t* accept_len, int32_t* out_tokens,
                            int32_t* committed_src, int32_t* new_ctx, int32_t* dev_status, void* stream) {
  if (!kv || !dims || !argmax || !path || !accept_len || !out_tokens || !committed_src || !new_ctx || !dev_status)
    return TV_E_ARG;
  if (dims->n_kv_heads <= 0 || (dims->head_dim != 64 && dims->head_dim != 128)) return TV_E_UNSUPPORTED;
  ReqTable t;
  const int rc = build_table(t, trees, kv, n_req, true);
  if (rc) return rc;
  return launch_accept_greedy_commit(t, *dims, argmax, path, accept_len, out_tokens, committed_src, new_ctx,
                                     dev_status, reinterpret_cast<cudaStream_t>(stream));
}

int tv_profile_start(int max_calls) {
  if (max_calls < 1 || max_calls > (1 << 16)) return TV_E_ARG;
  if (g_prof.ev) return TV_E_ARG;   // already running
  const int n = max_calls * (TV_PROFILE_STAGES + 1);
  cudaEvent_t* ev = new cudaEvent_t[n];
  for (int i = 0; i < n; ++i) {
    if (cudaEventCreate(&ev[i]) != cudaSuccess) {
      for (int j = 0; j < i; ++j) cudaEventDestroy(ev[j]);
      delete[] ev;
      return TV_E_CUDA;
    }
  }
  g_prof.ev = ev;
  g_prof.cap = max_calls;
  g_prof.calls = 0;
  return TV_OK;
}

int tv_profile_stop(float* stage_ms, int max_stages, int* n_stages, int* n_calls) {
  if (!g_prof.ev) return TV_E_ARG;
  int rc = TV_OK;
  float sums[TV_PROFILE_STAGES] = {0};
  for (int c = 0; c < g_prof.calls && rc == TV_OK; ++c) {
    cudaEvent_t* e = g_prof.ev + (size_t)c * (TV_PROFILE_STAGES + 1);
    if (cudaEventSynchronize(e[TV_PROFILE_STAGES]) != cudaSuccess) rc = TV_E_CUDA;
    for (int s = 0; s < TV_PROFILE_STAGES && rc == TV_OK; ++s) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, e[s], e[s + 1]) != cudaSuccess) rc = TV_E_CUDA;
      sums[s] += ms;
    }
  }
  const int n = g_prof.cap * (TV_PROFILE_STAGES + 1);
  for (int i = 0; i < n; ++i) cudaEventDestroy(g_prof.ev[i]);
  delete[] g_prof.ev;
  if (n_calls) *n_calls = g_prof.calls;
  g_prof = Profile();
  if (n_stages) *n_stages = TV_PROFILE_STAGES;
  if (stage_ms)
    for (int s = 0; s < TV_PROFILE_STAGES && s < max_stages; ++s) stage_ms[s] = sums[s];
  return rc;
}

int tv_packed_weight_bytes(int32_t rows, int32_t cols, size_t* bytes) {
  if (!bytes || rows < 1 || cols < 64 || cols % 64 != 0) return TV_E_ARG;
  *bytes = (size_t)((rows + 127) / 128) * 128 * (size_t)cols * 2;
  return TV_OK;
}

int tv_pack_weight(const tv_bf16* w, int32_t rows, int32_t cols, tv_bf16* packed, void* stream) {
  if (!w || !packed || !aligned16(w) || !aligned16(packed) || rows < 1 || cols < 64 || cols % 64 != 0) return TV_E_ARG;
  return launch_pack_weight(w, rows, cols, packed, reinterpret_cast<cudaStream_t>(stream));
}

const char* tv_status_string(int code) {
  switch (code) {
    case TV_OK: return "ok";
    case TV_E_ARG: return "bad argument";
    case TV_E_ORDER: return "parent array not in parent-before-child order";
    case TV_E_DUP_SIBLING: return "duplicate sibling token";
    case TV_E_TOKEN: return "token id outside the vocabulary";
    case TV_E_CAPACITY: return "cache capacity below ctx_len + tree rows";
    case TV_E_ROWS: return "tree size outside 1..32 or more than 32 rows in one pass";
    case TV_E_UNIFORM: return "uniform not finite or not in [0, 1)";
    case TV_E_TEMP: return "temperature not finite or not above 0";
    case TV_E_WORKSPACE: return "workspace missing or too small";
    case TV_E_CUDA: return "CUDA runtime error";
    case TV_E_UNSUPPORTED: return "shape not supported by these kernels";
    case TV_E_TIMEOUT: return "a bounded device wait gave up";
    case TV_E_PATH: return "accept length or path entry out of range";
    case TV_E_CHAIN: return "single-path sampling needs a chain";
    case TV_E_PROPOSAL: return "proposal row not finite, negative, off unit mass or zero at its draft";
    default: return "unknown status";
  }
}

}  // extern "C"

// ---- the decoder-layer stack -----------------------------------------------------
namespace tv {
namespace {

struct StackLayout {
  size_t rstats, meta, counter, h, x, q, part, attn_ml, attn_o, attn, top2, dq, dv, dz, dbeta, dg, dout, act, dk_all,
      du_all, dgc_all, total;
  int n_attn, n_dn;
};

int stack_counts(const tv_stack& m, int& n_attn, int& n_dn) {
  n_attn = n_dn = 0;
  if (!m.layers || m.n_layers < 1) return TV_E_ARG;
  for (int l = 0; l < m.n_layers; ++l) {
    if (m.layers[l].kind == TV_LAYER_ATTN) ++n_attn;
    else if (m.layers[l].kind == TV_LAYER_DN) ++n_dn;
    else return TV_E_ARG;
  }
  return TV_OK;
}

size_t part_bytes(int M, int K) { return (size_t)plan_gemm(M, K, false).splits * kMaxRows * M * 4; }

StackLayout stack_layout(const tv_stack& m) {
  StackLayout L;
  stack_counts(m, L.n_attn, L.n_dn);
  const tv_dims& d = m.dims;
  const tv_dn_dims& dn = m.dn;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const int H = d.hidden, QD = d.n_q_heads * d.head_dim, QKV = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
  const int KD = dn.n_k_heads * dn.d_k, VD = dn.n_v_heads * dn.d_v, I = m.intermediate;
  const int DIN = 2 * KD + 2 * VD + 2 * dn.n_v_heads;
  size_t pb = 0;
  auto mx = [&](size_t b) { pb = b > pb ? b : pb; };
  if (L.n_attn) {
    mx(part_bytes(QKV, H));
    mx(part_bytes(H, QD));
  }
  if (L.n_dn) {
    mx(part_bytes(DIN, H));
    mx(part_bytes(H, VD));
  }
  mx(part_bytes(2 * I, H));
  mx(part_bytes(H, I));
  L.rstats = take((size_t)kMaxRows * n_vchunks(d.vocab) * sizeof(RowStat));
  L.meta = take(kMaxRows * sizeof(RowMeta));
  L.counter = take(256);
  L.h = take((size_t)kMaxRows * H * 2);
  L.x = take((size_t)kMaxRows * H * 2);
  L.q = take((size_t)kMaxRows * QD * 2);
  L.part = take(pb);
  L.attn_ml = take((size_t)kMaxRows * d.n_q_heads * kChunkSlots * 2 * 4);
  L.attn_o = take((size_t)kMaxRows * d.n_q_heads * kChunkSlots * d.head_dim * 4);
  L.attn = take((size_t)kMaxRows * QD * 2);
  L.top2 = take((size_t)kMaxHeadGrid * 32 * sizeof(Top2));
  L.dq = take((size_t)kMaxRows * KD * 4);
  L.dv = take((size_t)kMaxRows * VD * 4);
  L.dz = take((size_t)kMaxRows * VD * 4);
  L.dbeta = take((size_t)kMaxRows * dn.n_v_heads * 4);
  L.dg = take((size_t)kMaxRows * dn.n_v_heads * 4);
  L.dout = take((size_t)kMaxRows * VD * 4);
  L.act = take((size_t)kMaxRows * (I > VD ? I : VD) * 2);
  L.dk_all = take((size_t)L.n_dn * kMaxRows * KD * 4);
  L.du_all = take((size_t)L.n_dn * kMaxRows * VD * 4);
  L.dgc_all = take((size_t)L.n_dn * kMaxRows * dn.n_v_heads * 4);
  L.total = off;
  return L;
}

int stack_check(const tv_stack* m) {
  if (!m) return TV_E_ARG;
  int rc = check_dims(m->dims);
  if (rc) return rc;
  int na = 0, nd = 0;
  if ((rc = stack_counts(*m, na, nd))) return rc;
  if (nd > 0 && (rc = dn_check(&m->dn))) return rc;
  if (m->intermediate < 64 || m->intermediate % 64 != 0) return TV_E_UNSUPPORTED;
  if (m->dims.hidden > 16384 || m->intermediate > 65536) return TV_E_UNSUPPORTED;
  if (!m->embed || !m->ln_f || !m->lm_head || !aligned16(m->lm_head)) return TV_E_ARG;
  if (m->packed != 0 && m->packed != 1) return TV_E_ARG;
  for (int l = 0; l < m->n_layers; ++l) {
    const tv_layer& y = m->layers[l];
    if (!y.ln_mix || !y.ln_mlp || !y.w_mix_in || !y.w_mix_out || !y.w_gate_up || !y.w_down) return TV_E_ARG;
    if (y.kind == TV_LAYER_DN && !y.dn_norm) return TV_E_ARG;
    if (!aligned16(y.w_mix_in) || !aligned16(y.w_mix_out) || !aligned16(y.w_gate_up) || !aligned16(y.w_down))
      return TV_E_ARG;
  }
  return TV_OK;
}

// The request table of attention layer j: the trees and that layer's caches.
int stack_table(ReqTable& t, const tv_tree* trees, const tv_kv* kv, int n_req, int j) {
  return build_table(t, trees, kv + (size_t)j * n_req, n_req, true);
}

}  // namespace
}  // namespace tv

extern "C" {

int tv_stack_workspace_size(const tv_stack* model, size_t* bytes) {
  if (!bytes) return TV_E_ARG;
  const int rc = stack_check(model);
  if (rc) return rc;
  *bytes = stack_layout(*model).total;
  return TV_OK;
}

int tv_verify_stack(const tv_stack* model, const tv_kv* kv, float* const* dn_states, const tv_tree* trees, int n_req,
                    float* logits, int32_t* argmax, float* top2_gap, tv_bf16* x_taps, void* workspace,
                    size_t workspace_bytes, int32_t* dev_status, void* stream) {
  int rc = stack_check(model);
  if (rc) return rc;
  if (!trees || !logits || !argmax || !top2_gap || !dev_status) return TV_E_ARG;
  if (x_taps && !aligned16(x_taps)) return TV_E_ARG;
  const StackLayout L = stack_layout(*model);
  if ((L.n_attn > 0 && !kv) || (L.n_dn > 0 && !dn_states)) return TV_E_ARG;
  const tv_dims& d = model->dims;
  const tv_dn_dims& dn = model->dn;
  ReqTable t;
  if (L.n_attn > 0) {
    if ((rc = stack_table(t, trees, kv, n_req, 0))) return rc;
    for (int j = 1; j < L.n_attn; ++j) {
      ReqTable tj;
      if ((rc = stack_table(tj, trees, kv, n_req, j))) return rc;
      for (int r = 0; r < n_req; ++r)
        if (tj.ctx[r] != t.ctx[r]) return TV_E_ARG;
    }
    const int G = d.n_q_heads / d.n_kv_heads;
    for (int r = 0; r < n_req; ++r)
      if (G * t.n[r] > kMaxQueriesPerKvHead) return TV_E_UNSUPPORTED;
  } else if ((rc = build_table(t, trees, nullptr, n_req, true))) {
    return rc;
  }
  DnStates st;
  if (L.n_dn > 0 && (rc = ::dn_states(st, dn_states, n_req))) return rc;
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return TV_E_WORKSPACE;
  const int sms = num_sms();
  if (sms <= 0) return TV_E_CUDA;
  if (sms > kMaxHeadGrid) return TV_E_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto bf = [&](size_t o) { return reinterpret_cast<__nv_bfloat16*>(ws + o); };
  auto f32 = [&](size_t o) { return reinterpret_cast<float*>(ws + o); };
  LayerBufs b;
  b.meta = reinterpret_cast<RowMeta*>(ws + L.meta);
  b.head_counter = reinterpret_cast<unsigned int*>(ws + L.counter);
  b.h = bf(L.h);
  b.q = bf(L.q);
  b.part_qkv = f32(L.part);
  b.attn_ml = f32(L.attn_ml);
  b.attn_o = f32(L.attn_o);
  b.attn = bf(L.attn);
  b.part_o = f32(L.part);
  b.hf = bf(L.h);
  __nv_bfloat16* x = bf(L.x);
  __nv_bfloat16* act = bf(L.act);
  float* part = f32(L.part);
  const int rows = t.total_rows;
  const int H = d.hidden, QD = d.n_q_heads * d.head_dim, QKV = (d.n_q_heads + 2 * d.n_kv_heads) * d.head_dim;
  const int KD = dn.n_k_heads * dn.d_k, VD = dn.n_v_heads * dn.d_v, I = model->intermediate;
  const int DIN = 2 * KD + 2 * VD + 2 * dn.n_v_heads;
  GemmParams gp;
  memset(&gp, 0, sizeof(gp));
  gp.status = dev_status;
  gp.packed = model->packed ? 1 : 0;
  gp.out = part;
  auto gemm = [&](const void* W, int M, int K, const void* X, GemmPlan& pl) {
    pl = plan_gemm(M, K, false);
    return launch_gemm(GEMM_PARTIAL, W, M, K, X, rows, pl, gp, sms, s);
  };
  GemmPlan pl;
  int n_tap = 0;
  auto tap = [&]() {   // the residual stream into the next tap slot
    if (!x_taps) return TV_OK;
    const size_t bytes = (size_t)rows * H * sizeof(tv_bf16);
    return cudaMemcpyAsync(reinterpret_cast<uint8_t*>(x_taps) + (size_t)(n_tap++) * bytes, x, bytes,
                           cudaMemcpyDeviceToDevice, s) == cudaSuccess ? TV_OK : TV_E_CUDA;
  };
  if ((rc = launch_prologue_embed(t, d, model->embed, model->layers[0].ln_mix, b, x, dev_status, s))) return rc;
  if ((rc = tap())) return rc;
  int ja = 0, jd = 0;
  for (int l = 0; l < model->n_layers; ++l) {
    const tv_layer& y = model->layers[l];
    if (y.kind == TV_LAYER_ATTN) {
      ReqTable tl;
      if ((rc = stack_table(tl, trees, kv, n_req, ja))) return rc;
      if ((rc = gemm(y.w_mix_in, QKV, H, b.h, pl))) return rc;
      if ((rc = launch_qkv_finalize(tl, d, b, pl.splits, dev_status, s))) return rc;
      if ((rc = launch_attention(tl, d, b, sms, dev_status, s))) return rc;
      if ((rc = gemm(y.w_mix_out, H, QD, b.attn, pl))) return rc;
      ++ja;
    } else {
      float* kl = f32(L.dk_all) + (size_t)jd * rows * KD;
      float* ul = f32(L.du_all) + (size_t)jd * rows * VD;
      float* gcl = f32(L.dgc_all) + (size_t)jd * rows * dn.n_v_heads;
      DnStates sl;
      for (int r = 0; r < n_req; ++r) sl.S[r] = st.S[r] + (size_t)jd * dn.n_v_heads * dn.d_k * dn.d_v;
      if ((rc = gemm(y.w_mix_in, DIN, H, b.h, pl))) return rc;
      if ((rc = launch_dn_in(part, pl.splits, rows, dn.n_k_heads, dn.n_v_heads, dn.d_k, dn.d_v, f32(L.dq), kl,
                             f32(L.dv), f32(L.dz), f32(L.dbeta), f32(L.dg), dev_status, s)))
        return rc;
      if ((rc = launch_dn_verify(t, sl, dn.n_k_heads, dn.n_v_heads, dn.d_k, dn.d_v, f32(L.dq), kl, f32(L.dv),
                                 f32(L.dbeta), f32(L.dg), f32(L.dout), ul, gcl, dev_status, s, true)))
        return rc;
      if ((rc = launch_dn_out(f32(L.dout), f32(L.dz), y.dn_norm, rows, dn.n_v_heads, dn.d_v, d.rms_eps, act,
                              dev_status, s)))
        return rc;
      if ((rc = gemm(y.w_mix_out, H, VD, act, pl))) return rc;
      ++jd;
    }
    if ((rc = launch_resid(part, pl.splits, H, rows, x, y.ln_mlp, d.rms_eps, b.h, dev_status, s))) return rc;
    if ((rc = tap())) return rc;
    if ((rc = gemm(y.w_gate_up, 2 * I, H, b.h, pl))) return rc;
    if ((rc = launch_act(part, pl.splits, I, rows, act, dev_status, s))) return rc;
    if ((rc = gemm(y.w_down, H, I, act, pl))) return rc;
    const void* next = l + 1 < model->n_layers ? (const void*)model->layers[l + 1].ln_mix : (const void*)model->ln_f;
    if ((rc = launch_resid(part, pl.splits, H, rows, x, next, d.rms_eps, b.h, dev_status, s))) return rc;
    if ((rc = tap())) return rc;
  }
  gp.out = logits;
  gp.top2_part = reinterpret_cast<Top2*>(ws + L.top2);
  gp.done_counter = b.head_counter;
  gp.argmax = argmax;
  gp.gap = top2_gap;
  const GemmPlan ph = plan_gemm(d.vocab, H, true);
  return launch_gemm(GEMM_HEAD, model->lm_head, d.vocab, H, b.h, rows, ph, gp, sms, s);
}

int tv_commit_stack(const tv_stack* model, const tv_kv* kv, float* const* dn_states, const tv_tree* trees, int n_req,
                    const int32_t* path, const int32_t* accept_len, int32_t* committed_src, int32_t* new_ctx,
                    const void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  int rc = stack_check(model);
  if (rc) return rc;
  if (!trees || !path || !accept_len || !committed_src || !new_ctx || !dev_status) return TV_E_ARG;
  const StackLayout L = stack_layout(*model);
  if ((L.n_attn > 0 && !kv) || (L.n_dn > 0 && !dn_states)) return TV_E_ARG;
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return TV_E_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const tv_dn_dims& dn = model->dn;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  ReqTable t;
  for (int j = 0; j < L.n_attn; ++j) {
    if ((rc = stack_table(t, trees, kv, n_req, j))) return rc;
    if ((rc = launch_commit(t, model->dims, path, accept_len, committed_src, new_ctx, dev_status, s))) return rc;
  }
  if (L.n_dn > 0) {
    if ((rc = build_table(t, trees, nullptr, n_req, true))) return rc;
    DnStates st;
    if ((rc = ::dn_states(st, dn_states, n_req))) return rc;
    if ((rc = launch_dn_commit(t, st, dn.n_k_heads, dn.n_v_heads, dn.d_k, dn.d_v, L.n_dn,
                               reinterpret_cast<const float*>(ws + L.dk_all), reinterpret_cast<const float*>(ws + L.du_all),
                               reinterpret_cast<const float*>(ws + L.dgc_all), path, accept_len, dev_status, s)))
      return rc;
  }
  return TV_OK;
}

}  // extern "C"
