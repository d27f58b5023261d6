// Per-row kernels of the verify through a decoder-layer stack (tv_verify_stack):
// the residual finalize between sublayers, the MLP activation, and the Gated
// DeltaNet layer's input and output stages around its recurrent core.
//
// One forward pass of the whole model over every tree row [Drafters and tree
// verify, §The round, step 2].  The layers are the reading of the pages that
// the stack entry point documents (include/tv.h): a pre-norm residual stack of
// Gated DeltaNet and attention layers, each followed by a SwiGLU MLP.  The
// projections run on the tcgen05 skinny GEMM (tv_gemm.cu) as split-K partials;
// the kernels here sum the partials of one row in split order, so a row's
// result never depends on the other rows of the pass.
#include <cmath>

#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

__device__ __forceinline__ void unpack8s(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 v = __bfloat1622float2(p[i]);
    f[2 * i] = v.x;
    f[2 * i + 1] = v.y;
  }
}

__device__ __forceinline__ uint4 pack8s(const float (&f)[8]) {
  uint4 u;
  __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

__device__ __forceinline__ float block_sum_s(float v, float* red) {
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

__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }

// ---------------------------------------------------------------------------
// Residual finalize: x = bf16(x + sum_s partial_s), splits in order; then
// h = bf16(RMSNorm(x) g) for the next sublayer (or hf for the head).  A
// cluster of kRCtas CTAs per row, each a contiguous slice of the row's
// 8-element vectors; the sum of squares is the CTAs' sums added in rank order
// over distributed shared memory.
// ---------------------------------------------------------------------------
constexpr int kRCtas = 4;
constexpr int kRThreads = 160;
template <int VECS>
__global__ void __cluster_dims__(kRCtas, 1, 1) __launch_bounds__(kRThreads)
    resid_kernel(const float* part, int splits, int H, __nv_bfloat16* x, const __nv_bfloat16* g, float eps,
                 __nv_bfloat16* h_out, const int32_t* status) {
  __shared__ float red[33];
  __shared__ float s_ss;
  pdl_trigger();   // the next GEMM may start streaming its weights now
  const int row = blockIdx.x / kRCtas;
  const uint32_t rank = cluster_ctarank();
  const int nvec = H / 8;
  const int slice = (nvec + kRCtas - 1) / kRCtas;
  const int v0 = (int)rank * slice, v1 = min(nvec, v0 + slice);
  const uint4* gv = reinterpret_cast<const uint4*>(g);
  uint4 gvv[VECS];   // the norm's gain (a weight) before the wait
#pragma unroll
  for (int k = 0; k < VECS; ++k) {
    const int vi = v0 + threadIdx.x + k * kRThreads;
    gvv[k] = vi < v1 ? gv[vi] : make_uint4(0u, 0u, 0u, 0u);
  }
  pdl_wait();
  const bool bad = status_get(status) != 0;   // nothing is written after an earlier error
  uint4* xv = reinterpret_cast<uint4*>(x + (size_t)row * H);
  float r[VECS][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < VECS; ++k) {
    const int vi = v0 + threadIdx.x + k * kRThreads;
    if (vi < v1) {
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
      unpack8s(xv[vi], xf);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        r[k][e] = bf2f(f2bf(xf[e] + o[e]));
        ss += r[k][e] * r[k][e];
      }
    }
  }
  ss = block_sum_s(ss, red);
  if (threadIdx.x == 0) s_ss = ss;
  cluster_sync_all();
  float tot = 0.f;
#pragma unroll
  for (int c = 0; c < kRCtas; ++c) tot += ld_dsmem_f32(dsmem_addr(&s_ss, (uint32_t)c));
  cluster_sync_all();   // every CTA has read the others' sums before any leaves
  if (bad) return;
  const float inv = 1.0f / sqrtf(tot / (float)H + eps);
  uint4* hv = reinterpret_cast<uint4*>(h_out + (size_t)row * H);
#pragma unroll
  for (int k = 0; k < VECS; ++k) {
    const int vi = v0 + threadIdx.x + k * kRThreads;
    if (vi < v1) {
      float gf[8], y[8];
      unpack8s(gvv[k], gf);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = r[k][e] * inv * gf[e];
      xv[vi] = pack8s(r[k]);
      hv[vi] = pack8s(y);
    }
  }
}

// ---------------------------------------------------------------------------
// SwiGLU activation: a = bf16( silu(gate) * up ), gate = partial sums of rows
// [0, I) of the gate/up projection, up = rows [I, 2I).  grid (rows, chunks of
// 4 x 256 columns).
// ---------------------------------------------------------------------------
constexpr int kActThreads = 256;
__global__ void __launch_bounds__(kActThreads) act_kernel(const float* part, int splits, int I,
                                                          __nv_bfloat16* a, const int32_t* status) {
  pdl_trigger();   // the down projection may start streaming its weights now
  pdl_wait();
  const int row = blockIdx.x;
  const int j = (blockIdx.y * kActThreads + threadIdx.x) * 4;
  if (j >= I || status_get(status) != 0) return;
  const size_t M = 2 * (size_t)I;
  float4 gs = make_float4(0.f, 0.f, 0.f, 0.f), us = gs;
  for (int s = 0; s < splits; ++s) {
    const float* ps = part + ((size_t)s * kMaxRows + row) * M;
    const float4 gp = *reinterpret_cast<const float4*>(ps + j);
    const float4 up = *reinterpret_cast<const float4*>(ps + I + j);
    gs.x += gp.x; gs.y += gp.y; gs.z += gp.z; gs.w += gp.w;
    us.x += up.x; us.y += up.y; us.z += up.z; us.w += up.w;
  }
  const __nv_bfloat162 lo = __floats2bfloat162_rn(silu(gs.x) * us.x, silu(gs.y) * us.y);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(silu(gs.z) * us.z, silu(gs.w) * us.w);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t*>(&lo);
  pk.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(a + (size_t)row * I + j) = pk;
}

// ---------------------------------------------------------------------------
// Gated DeltaNet input stage, from the partial sums of h W_in^T whose rows are
// [q: Hk dk][k: Hk dk][v: Hv dv][z: Hv dv][b: Hv][a: Hv].  grid (rows, Hk + Hv),
// one thread per element of a head (block = max(dk, dv)):
//   key head h:   q = q_raw / sqrt(|q_raw|^2 + 1e-6) / sqrt(dk),
//                 k = k_raw / sqrt(|k_raw|^2 + 1e-6)
//   value head h: v, z as summed; beta = sigmoid(b), g = -softplus(a)
// All fp32, [row][head][d]; k goes straight to the layer's slot of the
// commit's stacked keys.
// ---------------------------------------------------------------------------
__global__ void dn_in_kernel(const float* part, int splits, int Hk, int Hv, int dk, int dv, float* q, float* k,
                             float* v, float* z, float* beta, float* g, const int32_t* status) {
  __shared__ float red[33];
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x, hd = blockIdx.y, d = threadIdx.x;
  const size_t M = 2 * (size_t)Hk * dk + 2 * (size_t)Hv * dv + 2 * (size_t)Hv;
  auto sum = [&](size_t col) {
    float a = 0.f;
    for (int s = 0; s < splits; ++s) a += part[((size_t)s * kMaxRows + row) * M + col];
    return a;
  };
  const bool bad = status_get(status) != 0;
  if (hd < Hk) {
    const float qr = d < dk ? sum((size_t)hd * dk + d) : 0.f;
    const float kr = d < dk ? sum((size_t)(Hk + hd) * dk + d) : 0.f;
    const float sq = block_sum_s(qr * qr, red);
    const float sk = block_sum_s(kr * kr, red);
    if (bad || d >= dk) return;
    q[((size_t)row * Hk + hd) * dk + d] = qr / sqrtf(sq + 1e-6f) / sqrtf((float)dk);
    k[((size_t)row * Hk + hd) * dk + d] = kr / sqrtf(sk + 1e-6f);
  } else {
    const int h = hd - Hk;
    if (bad || d >= dv) return;
    const size_t vb = 2 * (size_t)Hk * dk;
    v[((size_t)row * Hv + h) * dv + d] = sum(vb + (size_t)h * dv + d);
    z[((size_t)row * Hv + h) * dv + d] = sum(vb + (size_t)Hv * dv + (size_t)h * dv + d);
    if (d == 0) {
      const size_t bb = vb + 2 * (size_t)Hv * dv;
      const float b = sum(bb + h), a = sum(bb + Hv + h);
      beta[(size_t)row * Hv + h] = 1.f / (1.f + expf(-b));
      g[(size_t)row * Hv + h] = -(a > 20.f ? a : log1pf(expf(a)));
    }
  }
}

// ---------------------------------------------------------------------------
// Gated DeltaNet output stage, per (row, value head): y = bf16( o /
// sqrt(mean(o^2) + eps) w silu(z) ), the input of the output projection.
// ---------------------------------------------------------------------------
__global__ void dn_out_kernel(const float* o, const float* z, const __nv_bfloat16* w, int Hv, int dv, float eps,
                              __nv_bfloat16* y, const int32_t* status) {
  __shared__ float red[33];
  pdl_trigger();   // the output projection may start streaming its weights now
  const int row = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const float wd = d < dv ? bf2f(w[d]) : 0.f;   // a weight: before the wait
  pdl_wait();
  const size_t i = ((size_t)row * Hv + h) * dv + d;
  const float ov = d < dv ? o[i] : 0.f;
  const float ms = block_sum_s(ov * ov, red) / (float)dv;
  if (d >= dv || status_get(status) != 0) return;
  y[i] = f2bf(ov / sqrtf(ms + eps) * wd * silu(z[i]));
}

}  // namespace

int launch_resid(const float* part, int splits, int H, int rows, __nv_bfloat16* x, const void* g, float eps,
                 __nv_bfloat16* h_out, int32_t* status, cudaStream_t st) {
  const int nvec = H / 8;
  const int slice = (nvec + kRCtas - 1) / kRCtas;
  if (H % 8 != 0 || slice > 4 * kRThreads || splits > kMaxSplits) return TV_E_UNSUPPORTED;
  auto go = [&](auto kern) {
    return launch_pdl(kern, dim3(rows * kRCtas), dim3(kRThreads), 0, st, part, splits, H, x,
                      reinterpret_cast<const __nv_bfloat16*>(g), eps, h_out, (const int32_t*)status);
  };
  if (slice <= kRThreads) return go(resid_kernel<1>);
  if (slice <= 2 * kRThreads) return go(resid_kernel<2>);
  return go(resid_kernel<4>);
}

int launch_act(const float* part, int splits, int I, int rows, __nv_bfloat16* a, int32_t* status, cudaStream_t st) {
  if (I % 4 != 0) return TV_E_UNSUPPORTED;
  const int per = kActThreads * 4;
  return launch_pdl(act_kernel, dim3(rows, (I + per - 1) / per), dim3(kActThreads), 0, st, part, splits, I, a,
                    (const int32_t*)status);
}

int launch_dn_in(const float* part, int splits, int rows, int Hk, int Hv, int dk, int dv, float* q, float* k,
                 float* v, float* z, float* beta, float* g, int32_t* status, cudaStream_t st) {
  const int threads = dk > dv ? dk : dv;
  return launch_pdl(dn_in_kernel, dim3(rows, Hk + Hv), dim3(threads), 0, st, part, splits, Hk, Hv, dk, dv, q, k, v,
                    z, beta, g, (const int32_t*)status);
}

int launch_dn_out(const float* o, const float* z, const void* w, int rows, int Hv, int dv, float eps,
                  __nv_bfloat16* y, int32_t* status, cudaStream_t st) {
  return launch_pdl(dn_out_kernel, dim3(rows, Hv), dim3(dv), 0, st, o, z, reinterpret_cast<const __nv_bfloat16*>(w),
                    Hv, dv, eps, y, (const int32_t*)status);
}

}  // namespace tv
