// Per-row kernels of the verify pass: the tree prologue, embedding + RMSNorm,
// and the two finalizers that sum the projections' split-K partials in a fixed
// order (QKV + RoPE + tree K/V write; O + residual + final RMSNorm).
#include <cmath>

#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr int kRowThreads = 512;   // one block per row for the row-wise kernels
constexpr int kRowVecs = 4;        // uint4 (8 bf16) vectors per thread: hidden <= 16384

// ---------------------------------------------------------------------------
// prologue of request r, by one warp.  Validates the tree and computes per row
// the depth, position ctx + depth and ancestor set (node i sees its ancestors
// and itself: "an attention mask of its ancestors and a position equal to its
// depth" [Drafters and tree verify, §Tree verify through recurrent layers]).
// ---------------------------------------------------------------------------
__device__ void prologue_warp(const ReqTable& t, int r, int vocab, RowMeta* meta, int32_t* status) {
  __shared__ int s_depth[32];
  __shared__ uint32_t s_anc[32];
  const int lane = threadIdx.x & 31;
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
  if (lane < n) {
    RowMeta m;
    m.req = r;
    m.local = lane;
    m.token = tok;
    m.depth = s_depth[lane];
    m.pos = t.ctx[r] + s_depth[lane];
    m.anc = s_anc[lane];
    meta[t.row_off[r] + lane] = m;
  }
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    float s = l < (int)(blockDim.x >> 5) ? red[l] : 0.f;
    s = warp_sum(s);
    if (l == 0) red[32] = s;
  }
  __syncthreads();
  const float s = red[32];
  __syncthreads();
  return s;
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(p[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// The verify's first kernel.  Row blocks: h = bf16( x / sqrt(mean(x^2) + eps)
// * g ), x = E[token], each thread holding up to kRowVecs 8-element vectors of
// the row; x itself also goes to x_out when given (the residual stream of a
// layer stack).  The last n_req blocks: the prologue of each request (warp 0).
__global__ void __launch_bounds__(kRowThreads) prologue_embed_kernel(ReqTable t, int vocab, RowMeta* meta,
                                                                     unsigned int* head_counter,
                                                                     const __nv_bfloat16* embed,
                                                                     const __nv_bfloat16* g, int H, float eps,
                                                                     __nv_bfloat16* h, __nv_bfloat16* x_out,
                                                                     int32_t* status) {
  __shared__ float red[33];
  pdl_trigger();   // the QKV GEMM may start streaming its weights now
  // the norm's gain (a weight: no kernel writes it) before the wait
  const int nvec = H / 8;
  const uint4* gv = reinterpret_cast<const uint4*>(g);
  uint4 gvv[kRowVecs];
#pragma unroll
  for (int k = 0; k < kRowVecs; ++k) {
    const int vi = threadIdx.x + k * kRowThreads;
    gvv[k] = (int)blockIdx.x < t.total_rows && vi < nvec ? gv[vi] : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_wait();
  // no status check: nothing here indexes with data an earlier kernel wrote
  // (tokens are clamped), and the kernels after it check the status
  if ((int)blockIdx.x >= t.total_rows) {   // the last n_req blocks: the prologues
    if (threadIdx.x < 32) {
      const int r = blockIdx.x - t.total_rows;
      if (r == 0 && threadIdx.x == 0) *head_counter = 0u;
      prologue_warp(t, r, vocab, meta, status);
    }
    return;
  }
  // row blocks: the row's token straight from its tree (a token out of range,
  // which the prologue reports, reads row 0 here; the status stops the verify)
  const int row = blockIdx.x;
  int r = 0;
  while (r + 1 < t.n_req && t.row_off[r + 1] <= row) ++r;
  int token = t.token[r][row - t.row_off[r]];
  token = token < 0 || token >= vocab ? 0 : token;
  const uint4* x = reinterpret_cast<const uint4*>(embed + (size_t)token * H);
  float xf[kRowVecs][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kRowVecs; ++k) {
    const int vi = threadIdx.x + k * kRowThreads;
    if (vi < nvec) {
      unpack8(x[vi], xf[k]);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss += xf[k][e] * xf[k][e];
    }
  }
  ss = block_sum(ss, red);
  const float inv = 1.0f / sqrtf(ss / (float)H + eps);
  uint4* hv = reinterpret_cast<uint4*>(h + (size_t)row * H);
#pragma unroll
  for (int k = 0; k < kRowVecs; ++k) {
    const int vi = threadIdx.x + k * kRowThreads;
    if (vi < nvec) {
      float gf[8], y[8];
      unpack8(gvv[k], gf);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = xf[k][e] * inv * gf[e];
      hv[vi] = pack8(y);
      if (x_out) reinterpret_cast<uint4*>(x_out + (size_t)row * H)[vi] = x[vi];
    }
  }
}

// RoPE angle pos * f reduced to about [-pi, pi] in fp32 without fp64: f is
// carried as f_hi + f_lo; the product pos * f_hi is split into its rounded
// value and its exact rounding error (one fma); the multiple of 2 pi is taken
// off with a two-constant Cody-Waite reduction (2 pi = hi + lo), each step an
// fma with one rounding.  Error about 3e-7 rad for positions below 2^24.
__device__ __forceinline__ float rope_angle(int pos, float f_hi, float f_lo, const RopeParams& rp) {
  const float p = (float)pos;
  const float a = p * f_hi;
  const float a_err = fmaf(p, f_hi, -a);
  const float corr = fmaf(p, f_lo, a_err);
  const float k = rintf(a * rp.inv_two_pi);
  float r = fmaf(-k, rp.two_pi_hi, a);
  r = fmaf(-k, rp.two_pi_lo, r);
  return r + corr;
}

// qkv: sum the split-K partials in split order, rotate q and k by RoPE
// (rotate-half pairs (d, d + D/2)), round to bf16; q goes to the q buffer, k and
// v to the request's cache at slot ctx + node ("the cache holds every node at
// its depth-first slot" [Drafters and tree verify, §Tree verify through
// recurrent layers]).  grid (rows, Hq + 2 Hkv), block D/2.
__global__ void qkv_finalize_kernel(ReqTable t, const RowMeta* meta, const float* part, int splits, int Hq, int Hkv,
                                    int D, RopeParams rp, __nv_bfloat16* q_out, const int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, head = blockIdx.y, d = threadIdx.x;
  const int half = D / 2;
  const int M = (Hq + 2 * Hkv) * D;
  const int f1 = head * D + d, f2 = f1 + half;
  float p1[kMaxSplits], p2[kMaxSplits];
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s) {
    if (s < splits) {
      const float* ps = part + ((size_t)s * kMaxRows + row) * M;
      p1[s] = ps[f1];
      p2[s] = ps[f2];
    }
  }
  // the row's metadata and the status are read with the partials; the status
  // is checked before the metadata picks a cache address
  const RowMeta m = meta[row];
  const bool bad = status_get(status) != 0;
  float x1 = 0.f, x2 = 0.f;
#pragma unroll
  for (int s = 0; s < kMaxSplits; ++s) {
    if (s < splits) {
      x1 += p1[s];
      x2 += p2[s];
    }
  }
  if (bad) return;
  float y1 = x1, y2 = x2;
  if (head < Hq + Hkv) {
    float sn, cs;
    sincosf(rope_angle(m.pos, rp.f_hi[d], rp.f_lo[d], rp), &sn, &cs);
    y1 = x1 * cs - x2 * sn;
    y2 = x2 * cs + x1 * sn;
  }
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

// O projection finalize: r = bf16(x + sum_s partial_s) with the splits summed in
// order, hf = bf16(RMSNorm(r) g_f).  A cluster of kOCtas CTAs per row, each a
// contiguous slice of the row's 8-element vectors (VECS per thread, every split
// of a vector requested at once, up to eight), so that a row's partials stream
// into four SMs; the sum of squares is the four CTA sums added in rank order
// over distributed shared memory.
constexpr int kOCtas = 4;
constexpr int kOThreads = 160;
template <int VECS>
__global__ void __cluster_dims__(kOCtas, 1, 1) __launch_bounds__(kOThreads)
    o_finalize_kernel(ReqTable t, int vocab, const float* part, int splits, int H, const __nv_bfloat16* embed,
                      const __nv_bfloat16* g, float eps, __nv_bfloat16* hf, const int32_t* status) {
  __shared__ float red[33];
  __shared__ float s_ss;   // this CTA's sum of squares
  pdl_trigger();           // the head GEMM may start streaming its weights now
  const int row = blockIdx.x / kOCtas;
  const uint32_t rank = cluster_ctarank();
  const int nvec = H / 8;
  const int slice = (nvec + kOCtas - 1) / kOCtas;
  const int v0 = (int)rank * slice, v1 = min(nvec, v0 + slice);
  // Before the wait: the row's token straight from its tree (clamped like the
  // first kernel's) and its embedding row, the residual.  Neither is written
  // inside the round, and the tree is final: when this kernel starts, the
  // attention kernel has passed its wait, so the verify's first kernel, which
  // reads the tree after its own wait, has completed.
  int rq = 0;
  while (rq + 1 < t.n_req && t.row_off[rq + 1] <= row) ++rq;
  int token = t.token[rq][row - t.row_off[rq]];
  token = token < 0 || token >= vocab ? 0 : token;
  const uint4* x = reinterpret_cast<const uint4*>(embed + (size_t)token * H);
  const uint4* gv = reinterpret_cast<const uint4*>(g);
  uint4 xv[VECS], gvv[VECS];   // and the final norm's gain (a weight)
#pragma unroll
  for (int k = 0; k < VECS; ++k) {
    const int vi = v0 + threadIdx.x + k * kOThreads;
    xv[k] = vi < v1 ? x[vi] : make_uint4(0u, 0u, 0u, 0u);
    gvv[k] = vi < v1 ? gv[vi] : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_wait();
  const bool bad = status_get(status) != 0;   // nothing is written after an earlier error
  float r[VECS][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < VECS; ++k) {
    const int vi = v0 + threadIdx.x + k * kOThreads;
    if (vi < v1) {
      // partials summed in split order; loads issued eight splits at a time
      float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int s0 = 0; s0 < splits; s0 += 8) {
        float4 pv[8][2];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (s0 + j < splits) {
            const float4* ps =
                reinterpret_cast<const float4*>(part + ((size_t)(s0 + j) * kMaxRows + row) * H) + 2 * vi;
            pv[j][0] = ps[0];
            pv[j][1] = ps[1];
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (s0 + j < splits) {
            o[0] += pv[j][0].x; o[1] += pv[j][0].y; o[2] += pv[j][0].z; o[3] += pv[j][0].w;
            o[4] += pv[j][1].x; o[5] += pv[j][1].y; o[6] += pv[j][1].z; o[7] += pv[j][1].w;
          }
        }
      }
      float xf[8];
      unpack8(xv[k], xf);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        r[k][e] = bf2f(f2bf(xf[e] + o[e]));
        ss += r[k][e] * r[k][e];
      }
    }
  }
  ss = block_sum(ss, red);
  if (threadIdx.x == 0) s_ss = ss;
  cluster_sync_all();
  float tot = 0.f;
#pragma unroll
  for (int c = 0; c < kOCtas; ++c) tot += ld_dsmem_f32(dsmem_addr(&s_ss, (uint32_t)c));
  cluster_sync_all();   // every CTA has read the others' sums before any leaves
  if (bad) return;
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  uint4* hv = reinterpret_cast<uint4*>(hf + (size_t)row * H);
#pragma unroll
  for (int k = 0; k < VECS; ++k) {
    const int vi = v0 + threadIdx.x + k * kOThreads;
    if (vi < v1) {
      float gf[8], y[8];
      unpack8(gvv[k], gf);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = r[k][e] * inv * gf[e];
      hv[vi] = pack8(y);
    }
  }
}

RopeParams rope_params(int head_dim, float theta) {
  RopeParams rp;
  const double two_pi = 8.0 * std::atan(1.0);
  for (int d = 0; d < 64; ++d) {
    const double f = d < head_dim / 2 ? std::pow((double)theta, -2.0 * d / (double)head_dim) : 0.0;
    rp.f_hi[d] = (float)f;
    rp.f_lo[d] = (float)(f - (double)rp.f_hi[d]);
  }
  rp.two_pi_hi = (float)two_pi;
  rp.two_pi_lo = (float)(two_pi - (double)rp.two_pi_hi);
  rp.inv_two_pi = (float)(1.0 / two_pi);
  return rp;
}

}  // namespace

int launch_prologue_embed(const ReqTable& t, const tv_dims& d, const void* embed, const void* gain,
                          const LayerBufs& b, __nv_bfloat16* x_out, int32_t* status, cudaStream_t st) {
  if (d.hidden > kRowVecs * kRowThreads * 8) return TV_E_UNSUPPORTED;
  return launch_pdl(prologue_embed_kernel, dim3(t.total_rows + t.n_req), dim3(kRowThreads), 0, st, t, d.vocab,
                    b.meta, b.head_counter, reinterpret_cast<const __nv_bfloat16*>(embed),
                    reinterpret_cast<const __nv_bfloat16*>(gain), d.hidden, d.rms_eps, b.h, x_out, status);
}

int launch_qkv_finalize(const ReqTable& t, const tv_dims& d, const LayerBufs& b, int splits, int32_t* status,
                        cudaStream_t st) {
  thread_local RopeParams cached;   // per host thread: calls from several threads do not race
  thread_local int cached_dim = -1;
  thread_local float cached_theta = 0.f;
  if (cached_dim != d.head_dim || cached_theta != d.rope_theta) {
    cached = rope_params(d.head_dim, d.rope_theta);
    cached_dim = d.head_dim;
    cached_theta = d.rope_theta;
  }
  if (splits > kMaxSplits) return TV_E_UNSUPPORTED;
  dim3 grid(t.total_rows, d.n_q_heads + 2 * d.n_kv_heads);
  return launch_pdl(qkv_finalize_kernel, grid, dim3(d.head_dim / 2), 0, st, t, (const RowMeta*)b.meta,
                    (const float*)b.part_qkv, splits, d.n_q_heads, d.n_kv_heads, d.head_dim, cached, b.q,
                    (const int32_t*)status);
}

int launch_o_finalize(const ReqTable& t, const tv_model& m, const LayerBufs& b, int splits, int32_t* status,
                      cudaStream_t st) {
  const int nvec = m.dims.hidden / 8;
  const int slice = (nvec + kOCtas - 1) / kOCtas;
  if (slice > 4 * kOThreads || splits > kMaxSplits) return TV_E_UNSUPPORTED;
  auto go = [&](auto kern) {
    return launch_pdl(kern, dim3(t.total_rows * kOCtas), dim3(kOThreads), 0, st, t, m.dims.vocab,
                      (const float*)b.part_o, splits, m.dims.hidden, reinterpret_cast<const __nv_bfloat16*>(m.embed),
                      reinterpret_cast<const __nv_bfloat16*>(m.ln_f), m.dims.rms_eps, b.hf, (const int32_t*)status);
  };
  if (slice <= kOThreads) return go(o_finalize_kernel<1>);
  if (slice <= 2 * kOThreads) return go(o_finalize_kernel<2>);
  return go(o_finalize_kernel<4>);
}

}  // namespace tv
