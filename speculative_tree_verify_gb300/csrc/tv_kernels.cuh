// Internal interface between the kernel translation units and the C ABI layer.
// Each .cu file launches its own kernels through the host functions declared
// here, so the library needs no relocatable device code.
#pragma once

#include "tv_common.cuh"

namespace tv {

// ---- attention chunking ------------------------------------------------------
// The cached keys of a request are cut into chunks of whole 128-key tiles.  The
// number of chunks aims at `target` = SMs / KV heads (at most kMaxChunks), so
// that one request's chunks x KV heads fill the GPU once; it depends on the
// context length, the model and the GPU only, never on the other rows or
// requests of the pass.  The tree keys get a chunk of their own while the
// cached tiles are fewer than the target (short contexts: one more CTA in the
// same wave), and otherwise join the last chunk.
constexpr int kMaxChunks = 32;
constexpr int kChunkSlots = kMaxChunks + 1;   // partial slots per (row, head) in the workspace

struct AttnPlan {
  int tiles_per_chunk;
  int n_chunks;    // chunks in all, the tree's own chunk included
  bool tree_own;   // the last chunk holds only the tree keys
};
__host__ __device__ inline AttnPlan attn_plan(int ctx, int target) {
  const int tiles = ctx > 0 ? (ctx + 127) / 128 : 0;
  target = target < 1 ? 1 : (target > kMaxChunks ? kMaxChunks : target);
  if (tiles < target) return AttnPlan{1, tiles + 1, true};
  const int per = (tiles + target - 1) / target;
  return AttnPlan{per, (tiles + per - 1) / per, false};
}
inline int attn_chunk_target(int sms, int n_kv_heads) { return n_kv_heads > 0 ? sms / n_kv_heads : 1; }

// ---- sampled walks: per-row statistics over vocabulary chunks ---------------
// A draw from a row searches its CDF in three steps, each one warp-wide:
// the row's chunks of 4096 tokens, the chunk's 32 segments of 128 tokens, the
// segment's 128 tokens (4 per lane).
constexpr int kVChunk = 4096;
constexpr int kVSeg = 128;
constexpr int kSegsPerChunk = kVChunk / kVSeg;   // 32: one per lane
struct RowStat {
  float m;                    // max logit of the chunk
  float s;                    // sum of seg[]
  float seg[kSegsPerChunk];   // per segment: sum of exp((logit - m) / T)
};
inline int n_vchunks(int vocab) { return (vocab + kVChunk - 1) / kVChunk; }

// ---- sampled walks ------------------------------------------------------------
// per request: the Gumbel seed and the sequence index of the root's token
struct SeedTable {
  unsigned long long seed[kMaxReq];
  int pos[kMaxReq];
};
struct GumbelPart {   // a vocabulary chunk's best x + G and its index
  float s;
  int idx;
};
struct RejStat {               // a vocabulary chunk of a draft's proposal row
  float seg[kSegsPerChunk];   // per segment: sum of max(p - q, 0), p the target row of the draft's parent
  float resid;                // sum of seg[]
  float qsum;                 // sum of q
  int bad;                    // a q entry not finite or negative
  int pad;
};

// ---- Gated DeltaNet --------------------------------------------------------------
constexpr int kDnMaxDim = 128;   // d_k, d_v: multiples of 32 up to this
struct DnStates {                // per request: the layer's state, [H_v][d_k][d_v] fp32 (per layer for the commit)
  float* S[kMaxReq];
};

// ---- block-uniform status check -------------------------------------------
__device__ __forceinline__ bool block_skip(const int32_t* status) {
  __shared__ int s_stat;
  if (threadIdx.x == 0) s_stat = status_get(status);
  __syncthreads();
  return s_stat != 0;
}

// ---- tree validation by one warp (lanes = nodes) ---------------------------
// Reports the first rule broken, in this order: parent order (parent[0] = -1,
// 0 <= parent[i] < i), token range (skipped when vocab <= 0), duplicate sibling
// tokens [Algorithm and correctness contract, §Target position and batching].
// par/tok receive this lane's parent and token.
// check_tree_warp takes the lane's parent and token already loaded (0 past n).
__device__ __forceinline__ int check_tree_warp(int par, int tok, int n, int vocab) {
  const int lane = threadIdx.x & 31;
  const bool bad_order = lane < n && (lane == 0 ? par != -1 : (par < 0 || par >= lane));
  const bool bad_token = lane < n && vocab > 0 && (tok < 0 || tok >= vocab);
  // a duplicate sibling: a lower lane with the same (parent, token); lanes
  // past n get keys no tree lane has (a parent of 0x80000000 + lane would be
  // out of order, which is reported first)
  const unsigned long long key =
      lane < n ? ((unsigned long long)(unsigned)par << 32) | (unsigned)tok
               : (unsigned long long)(0x80000000u + (unsigned)lane) << 32;
  const unsigned same = __match_any_sync(0xffffffffu, key);
  const bool dup = lane < n && (same & ((1u << lane) - 1u)) != 0u;
  if (__any_sync(0xffffffffu, bad_order)) return TV_E_ORDER;
  if (__any_sync(0xffffffffu, bad_token)) return TV_E_TOKEN;
  if (__any_sync(0xffffffffu, dup)) return TV_E_DUP_SIBLING;
  return TV_OK;
}
__device__ __forceinline__ int validate_tree_warp(const int32_t* parent, const int32_t* token, int n, int vocab,
                                                  int& par, int& tok) {
  const int lane = threadIdx.x & 31;
  par = lane < n ? parent[lane] : 0;
  tok = lane < n ? token[lane] : 0;
  return check_tree_warp(par, tok, n, vocab);
}

// ---- host argument checks (tv_api.cu) ------------------------------------------
// Fills the request table from the caller's host structs and checks them:
// TV_E_ROWS for a tree size outside 1..32 or more than 32 rows in all,
// TV_E_ARG for missing parent/token pointers (when need_parent) or bad caches,
// TV_E_CAPACITY when a cache cannot hold its tree.  kv may be null (walks).
int build_table(ReqTable& t, const tv_tree* trees, const tv_kv* kv, int n_req, bool need_parent);

// ---- launchers (host) -------------------------------------------------------
// RoPE frequencies theta^(-2d/D), computed in double on the host and split
// into hi + lo floats, and 2*pi split into two floats for the reduction.
struct RopeParams {
  float f_hi[64];
  float f_lo[64];
  float two_pi_hi, two_pi_lo, inv_two_pi;
};

constexpr int kMaxSplits = 16;   // split-K partials summed by the finalize kernels

struct LayerBufs {
  RowMeta* meta;
  unsigned int* head_counter;
  __nv_bfloat16* h;        // [32][H]
  __nv_bfloat16* q;        // [32][Hq][D]
  float* part_qkv;
  float* attn_ml;          // [32][Hq][kChunkSlots][2]: chunk max (log2 units), chunk sum
  float* attn_o;           // [32][Hq][kChunkSlots][D]: chunk output, not normalised
  __nv_bfloat16* attn;     // [rows][Hq D]
  float* part_o;
  __nv_bfloat16* hf;       // [32][H]
};

// the verify's first kernel: per request the tree prologue (validation, depth,
// position, ancestors), per row the embedding and first RMSNorm (h = bf16(
// RMSNorm(E[token]) gain)); x_out, when not null, receives E[token] itself
int launch_prologue_embed(const ReqTable& t, const tv_dims& d, const void* embed, const void* gain,
                          const LayerBufs& b, __nv_bfloat16* x_out, int32_t* status, cudaStream_t st);
int launch_qkv_finalize(const ReqTable& t, const tv_dims& d, const LayerBufs& b, int splits, int32_t* status,
                        cudaStream_t st);
int launch_attention(const ReqTable& t, const tv_dims& d, const LayerBufs& b, int sms, int32_t* status,
                     cudaStream_t st);
int launch_o_finalize(const ReqTable& t, const tv_model& m, const LayerBufs& b, int splits, int32_t* status,
                      cudaStream_t st);

// ---- the decoder-layer stack (tv_stack.cu) -------------------------------------
// x = bf16(x + sum of the split-K partials [splits][32][H]); h_out = bf16(
// RMSNorm(x) g).  A cluster of four CTAs per row.
int launch_resid(const float* part, int splits, int H, int rows, __nv_bfloat16* x, const void* g, float eps,
                 __nv_bfloat16* h_out, int32_t* status, cudaStream_t st);
// a = bf16(silu(gate) * up) from the partials of the [2 I] gate/up projection
int launch_act(const float* part, int splits, int I, int rows, __nv_bfloat16* a, int32_t* status, cudaStream_t st);
// Gated DeltaNet input stage: normalised q, k; v, z; beta = sigmoid(b), g = -softplus(a)
int launch_dn_in(const float* part, int splits, int rows, int Hk, int Hv, int dk, int dv, float* q, float* k,
                 float* v, float* z, float* beta, float* g, int32_t* status, cudaStream_t st);
// Gated DeltaNet output stage: y = bf16(RMSNorm(o) w silu(z)) per value head
int launch_dn_out(const float* o, const float* z, const void* w, int rows, int Hv, int dv, float eps,
                  __nv_bfloat16* y, int32_t* status, cudaStream_t st);

int launch_accept_greedy(const ReqTable& t, const int32_t* argmax, int32_t* path, int32_t* accept_len,
                         int32_t* out_tokens, int32_t* status, cudaStream_t st);
int launch_accept_residual(const ReqTable& t, const float* logits, int vocab, float temperature,
                           const float* uniforms, int bonus_at_leaf, RowStat* stats, int32_t* path,
                           int32_t* accept_len, int32_t* out_tokens, int32_t* out_count, int32_t* status,
                           cudaStream_t st);
int launch_accept_greedy_commit(const ReqTable& t, const tv_dims& d, const int32_t* argmax, int32_t* path,
                                int32_t* accept_len, int32_t* out_tokens, int32_t* committed_src, int32_t* new_ctx,
                                int32_t* status, cudaStream_t st);
int launch_commit(const ReqTable& t, const tv_dims& d, const int32_t* path, const int32_t* accept_len,
                  int32_t* committed_src, int32_t* new_ctx, int32_t* status, cudaStream_t st);

int launch_filter(const float* logits, float* out, int rows, int vocab, float temperature, int top_k, float top_p,
                  float min_p, int32_t* status, cudaStream_t st);
int launch_gumbel_rows(const ReqTable& t, const float* logits, int vocab, float temperature, const SeedTable& sd,
                       GumbelPart* part, int32_t* row_tokens, int32_t* status, cudaStream_t st);
int launch_draw_rows(const ReqTable& t, const float* logits, int vocab, float temperature, const float* uniforms,
                     RowStat* stats, int32_t* row_tokens, int32_t* status, cudaStream_t st);
// state_early: load each value head's state before the programmatic-launch
// wait; only for a caller whose preceding kernel triggers after its own wait
// and whose earlier kernels include every writer of the state (the layer
// stack: the DeltaNet input stage precedes it)
int launch_dn_verify(const ReqTable& t, const DnStates& st, int Hk, int Hv, int dk, int dv, const float* q,
                     const float* k, const float* v, const float* beta, const float* g, float* o, float* u, float* gc,
                     int32_t* status, cudaStream_t s, bool state_early = false);
int launch_dn_commit(const ReqTable& t, const DnStates& st, int Hk, int Hv, int dk, int dv, int n_layers,
                     const float* k, const float* u, const float* gc, const int32_t* path, const int32_t* accept_len,
                     int32_t* status, cudaStream_t s);
int launch_accept_rejection(const ReqTable& t, const float* logits, int vocab, float temperature,
                            const float* proposals, const float* uniforms, RowStat* stats, RejStat* rstats,
                            int32_t* path, int32_t* accept_len, int32_t* out_tokens, int32_t* out_count,
                            int32_t* status, cudaStream_t st);

}  // namespace tv
