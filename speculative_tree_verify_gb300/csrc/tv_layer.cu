// Per-row kernels of the verify pass: the tree prologue, embedding + RMSNorm,
// and the two finalizers that sum the projections' split-K partials in a fixed
// order (QKV + RoPE + tree K/V write; O + residual + final RMSNorm).
#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

// ---------------------------------------------------------------------------
// prologue: one warp per request.  Validates the tree, computes per row the
// depth, position ctx + depth and ancestor set (node i sees its ancestors and
// itself: "an attention mask of its ancestors and a position equal to its
// depth" [Drafters and tree verify, §Tree verify through recurrent layers]),
// and the RoPE rotation of each row's position (angles in fp64).
// ---------------------------------------------------------------------------
__global__ void prologue_kernel(ReqTable t, int vocab, int head_dim, float rope_theta, RowMeta* meta,
                                float2* rope_cs, unsigned int* head_counter, int32_t* status) {
  __shared__ int s_depth[32];
  __shared__ uint32_t s_anc[32];
  const int r = blockIdx.x;
  const int lane = threadIdx.x;
  if (status_get(status) != 0) return;
  if (r == 0 && lane == 0) *head_counter = 0u;
  const int n = t.n[r];
  int par, tok;
  const int err = validate_tree_warp(t.parent[r], t.token[r], n, vocab, par, tok);
  if (err != TV_OK) {
    if (lane == 0) status_set(status, err);
    return;
  }
  s_depth[lane] = 0;
  s_anc[lane] = 0;
  __syncwarp();
  // in node order: a parent precedes its child
  for (int i = 0; i < n; ++i) {
    const int pi = __shfl_sync(0xffffffffu, par, i);
    if (lane == 0) {
      s_depth[i] = i == 0 ? 0 : s_depth[pi] + 1;
      s_anc[i] = (i == 0 ? 0u : s_anc[pi]) | (1u << i);
    }
    __syncwarp();
  }
  const int row0 = t.row_off[r];
  const int ctx = t.ctx[r];
  if (lane < n) {
    RowMeta m;
    m.req = r;
    m.local = lane;
    m.token = tok;
    m.depth = s_depth[lane];
    m.pos = ctx + s_depth[lane];
    m.anc = s_anc[lane];
    meta[row0 + lane] = m;
  }
  const int half = head_dim / 2;
  for (int i = 0; i < n; ++i) {
    const double pos = (double)(ctx + s_depth[i]);
    for (int d = lane; d < half; d += 32) {
      const double inv_freq = pow((double)rope_theta, -2.0 * (double)d / (double)head_dim);
      double sn, cs;
      sincos(pos * inv_freq, &sn, &cs);
      rope_cs[(size_t)(row0 + i) * half + d] = make_float2((float)cs, (float)sn);
    }
  }
}

template <int NT>
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    float s = l < NT / 32 ? red[l] : 0.f;
    s = warp_sum(s);
    if (l == 0) red[NT / 32] = s;
  }
  __syncthreads();
  const float s = red[NT / 32];
  __syncthreads();
  return s;
}

// h = bf16( x / sqrt(mean(x^2) + eps) * g ), x = E[token]; one block per row
__global__ void __launch_bounds__(256) embed_norm_kernel(const RowMeta* meta, const __nv_bfloat16* embed,
                                                         const __nv_bfloat16* g, int H, float eps,
                                                         __nv_bfloat16* h, const int32_t* status) {
  __shared__ float red[16];
  if (block_skip(status)) return;
  const int row = blockIdx.x;
  const __nv_bfloat16* x = embed + (size_t)meta[row].token * H;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += 256) {
    const float v = bf2f(x[c]);
    ss += v * v;
  }
  ss = block_sum<256>(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)H + eps);
  for (int c = threadIdx.x; c < H; c += 256) h[(size_t)row * H + c] = f2bf(bf2f(x[c]) * inv * bf2f(g[c]));
}

// qkv: sum the split-K partials in split order, rotate q and k by RoPE
// (rotate-half pairs (d, d + D/2)), round to bf16; q goes to the q buffer, k and
// v to the request's cache at slot ctx + node ("the cache holds every node at
// its depth-first slot" [Drafters and tree verify, §Tree verify through
// recurrent layers]).  grid (rows, Hq + 2 Hkv), block D/2.
__global__ void qkv_finalize_kernel(ReqTable t, const RowMeta* meta, const float* part, int splits, int Hq, int Hkv,
                                    int D, const float2* rope_cs, __nv_bfloat16* q_out, const int32_t* status) {
  if (block_skip(status)) return;
  const int row = blockIdx.x, head = blockIdx.y, d = threadIdx.x;
  const int half = D / 2;
  const int M = (Hq + 2 * Hkv) * D;
  const int f1 = head * D + d, f2 = f1 + half;
  float x1 = 0.f, x2 = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float* ps = part + ((size_t)s * kMaxRows + row) * M;
    x1 += ps[f1];
    x2 += ps[f2];
  }
  float y1 = x1, y2 = x2;
  if (head < Hq + Hkv) {
    const float2 cs = rope_cs[(size_t)row * half + d];
    y1 = x1 * cs.x - x2 * cs.y;
    y2 = x2 * cs.x + x1 * cs.y;
  }
  const RowMeta m = meta[row];
  __nv_bfloat16* dst;
  if (head < Hq) {
    dst = q_out + ((size_t)row * Hq + head) * D;
  } else {
    const bool is_k = head < Hq + Hkv;
    const int g = is_k ? head - Hq : head - Hq - Hkv;
    __nv_bfloat16* base = is_k ? t.k[m.req] : t.v[m.req];
    dst = base + ((size_t)g * t.capacity[m.req] + t.ctx[m.req] + m.local) * D;
  }
  dst[d] = f2bf(y1);
  dst[d + half] = f2bf(y2);
}

// O projection finalize: r = bf16(x + sum_s partial_s), hf = bf16(RMSNorm(r) g_f);
// one block per row
__global__ void __launch_bounds__(256) o_finalize_kernel(const RowMeta* meta, const float* part, int splits, int H,
                                                         const __nv_bfloat16* embed, const __nv_bfloat16* g,
                                                         float eps, __nv_bfloat16* hf, const int32_t* status) {
  extern __shared__ float rbuf[];   // [H]
  __shared__ float red[16];
  if (block_skip(status)) return;
  const int row = blockIdx.x;
  const __nv_bfloat16* x = embed + (size_t)meta[row].token * H;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += 256) {
    float o = 0.f;
    for (int s = 0; s < splits; ++s) o += part[((size_t)s * kMaxRows + row) * H + c];
    const float r = bf2f(f2bf(bf2f(x[c]) + o));
    rbuf[c] = r;
    ss += r * r;
  }
  ss = block_sum<256>(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)H + eps);
  for (int c = threadIdx.x; c < H; c += 256) hf[(size_t)row * H + c] = f2bf(rbuf[c] * inv * bf2f(g[c]));
}

inline int last_error() { return cudaGetLastError() == cudaSuccess ? TV_OK : TV_E_CUDA; }

}  // namespace

int launch_prologue(const ReqTable& t, const tv_dims& d, const LayerBufs& b, int32_t* status, cudaStream_t st) {
  prologue_kernel<<<t.n_req, 32, 0, st>>>(t, d.vocab, d.head_dim, d.rope_theta, b.meta, b.rope, b.head_counter,
                                           status);
  return last_error();
}

int launch_embed_norm(const ReqTable& t, const tv_model& m, const LayerBufs& b, int32_t* status, cudaStream_t st) {
  embed_norm_kernel<<<t.total_rows, 256, 0, st>>>(b.meta, reinterpret_cast<const __nv_bfloat16*>(m.embed),
                                                   reinterpret_cast<const __nv_bfloat16*>(m.ln1), m.dims.hidden,
                                                   m.dims.rms_eps, b.h, status);
  return last_error();
}

int launch_qkv_finalize(const ReqTable& t, const tv_dims& d, const LayerBufs& b, int splits, int32_t* status,
                        cudaStream_t st) {
  dim3 grid(t.total_rows, d.n_q_heads + 2 * d.n_kv_heads);
  qkv_finalize_kernel<<<grid, d.head_dim / 2, 0, st>>>(t, b.meta, b.part_qkv, splits, d.n_q_heads, d.n_kv_heads,
                                                       d.head_dim, b.rope, b.q, status);
  return last_error();
}

int launch_o_finalize(const ReqTable& t, const tv_model& m, const LayerBufs& b, int splits, int32_t* status,
                      cudaStream_t st) {
  const size_t smem = (size_t)m.dims.hidden * sizeof(float);
  if (smem > 48 * 1024) {
    static bool attr = false;
    if (!attr) {
      if (cudaFuncSetAttribute(o_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
        return TV_E_CUDA;
      attr = true;
    }
  }
  o_finalize_kernel<<<t.total_rows, 256, smem, st>>>(b.meta, b.part_o, splits, m.dims.hidden,
                                                     reinterpret_cast<const __nv_bfloat16*>(m.embed),
                                                     reinterpret_cast<const __nv_bfloat16*>(m.ln_f),
                                                     m.dims.rms_eps, b.hf, status);
  return last_error();
}

}  // namespace tv
