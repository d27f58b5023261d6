// Sampling filters and seeded Gumbel-max draws.
//
//  - filter: temperature, top_k, top_p and min_p through one function, one CTA
//    per row [Exactness, §Sampling, second paragraph].  The k-th largest
//    logit and the top-p boundary are found by radix selection on an
//    order-preserving integer key of the logit (four 8-bit passes each), with
//    integer histograms, so the result is exact and the same on every run.
//  - Gumbel: the token at sequence index t is argmax_i (x_i + G_i), G_i Gumbel
//    noise from Philox4x32-10 keyed by (seed, t) [Exactness, §Sampling, third
//    paragraph]; one pass of (vocab chunk, row) blocks and a per-row pick.
//    Philox4x32-10 follows Salmon, Moraes, Dror and Shaw, "Parallel random
//    numbers: as easy as 1, 2, 3" (SC 2011).
#include <climits>
#include <cmath>

#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kFilterThreads = 1024;

// order-preserving key: larger float -> larger unsigned (NaN sorts lowest)
__device__ __forceinline__ uint32_t fkey(float x) {
  if (x != x) return 0u;
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The radix selection shared by top_k (weights 1) and top_p (weights = the
// quantised probability): over the tokens with key >= floor_key, the largest
// key K such that the total weight of tokens with key >= K reaches `need`.
// Returns floor_key when the whole weight falls short of need.
template <typename Weight>
__device__ uint32_t radix_select(const float* lr, int V, uint32_t floor_key, unsigned long long need, Weight w,
                                 unsigned long long* hist, unsigned long long* s_scalar) {
  uint32_t prefix = 0u, mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0ull;
    __syncthreads();
    for (int y = threadIdx.x; y < V; y += blockDim.x) {
      const uint32_t k = fkey(lr[y]);
      if (k >= floor_key && (k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], w(y, lr[y]));
    }
    __syncthreads();
    if (threadIdx.x < 32) {   // one warp: the bin where the weight from the top reaches need
      const int lane = threadIdx.x;
      unsigned long long above = 0ull;
      int found = -1;
      unsigned long long above_found = 0ull;
      for (int b0 = 255; b0 >= 0 && found < 0; b0 -= 32) {
        const int b = b0 - lane;
        const unsigned long long h = b >= 0 ? hist[b] : 0ull;
        unsigned long long incl = h;   // inclusive scan from the top (lane 0 = highest bin)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long u = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += u;
        }
        const unsigned hit = __ballot_sync(FULL, b >= 0 && above + incl >= need);
        if (hit) {
          const int L = __ffs(hit) - 1;
          found = b0 - L;
          above_found = above + __shfl_sync(FULL, incl - h, L);
        }
        above += __shfl_sync(FULL, incl, 31);
      }
      if (lane == 0) {
        s_scalar[0] = found < 0 ? ~0ull : (unsigned long long)found;
        s_scalar[1] = above_found;
      }
    }
    __syncthreads();
    const unsigned long long f = s_scalar[0];
    const unsigned long long ab = s_scalar[1];
    __syncthreads();
    if (f == ~0ull) return floor_key;   // the weight falls short: keep every token
    prefix |= (uint32_t)f << shift;
    mask |= 255u << shift;
    need -= ab;
  }
  return prefix;
}

__device__ float block_max(float v, float* red) {
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  float m = red[0];
  for (int i = 1; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  return m;
}

__device__ double block_sum_d(double v, double* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  double s = 0.0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];   // fixed order
  __syncthreads();
  return s;
}

// One row per CTA.  out = x = logit / T where kept, -inf elsewhere; selection
// on the raw logits (the scale by 1/T keeps their order).
__global__ void __launch_bounds__(kFilterThreads) filter_kernel(const float* logits, float* out, int V, float inv_t,
                                                                int top_k, double top_p, float log_min_p,
                                                                const int32_t* status) {
  __shared__ unsigned long long hist[256];
  __shared__ unsigned long long s_scalar[2];
  __shared__ float redf[kFilterThreads / 32];
  __shared__ double redd[kFilterThreads / 32];
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const float* lr = logits + (size_t)blockIdx.x * V;
  float* orow = out + (size_t)blockIdx.x * V;
  float lmax = -INFINITY;
  for (int y = threadIdx.x; y < V; y += blockDim.x) lmax = fmaxf(lmax, lr[y]);
  lmax = block_max(lmax, redf);
  uint32_t kfloor = 1u;   // above every NaN key
  if (top_k > 0 && top_k < V)
    kfloor = radix_select(lr, V, kfloor, (unsigned long long)top_k, [](int, float) { return 1ull; }, hist,
                          s_scalar);
  if (top_p < 1.0) {
    // probabilities over the tokens kept so far, quantised to 2^-40 steps
    double z = 0.0;
    for (int y = threadIdx.x; y < V; y += blockDim.x)
      if (fkey(lr[y]) >= kfloor) z += (double)expf((lr[y] - lmax) * inv_t);
    z = block_sum_d(z, redd);
    const double scale = 1099511627776.0 / z;   // 2^40 / Z
    auto qmass = [&](int, float l) { return (unsigned long long)((double)expf((l - lmax) * inv_t) * scale + 0.5); };
    unsigned long long need = (unsigned long long)(top_p * 1099511627776.0);
    if (need == 0ull) need = 1ull;   // the largest token always stays
    kfloor = radix_select(lr, V, kfloor, need, qmass, hist, s_scalar);
  }
  // min_p: x >= x_max + log(min_p), i.e. (l - l_max) / T >= log(min_p)
  for (int y = threadIdx.x; y < V; y += blockDim.x) {
    const float l = lr[y];
    const bool keep = fkey(l) >= kfloor && (l - lmax) * inv_t >= log_min_p;
    orow[y] = keep ? l * inv_t : -INFINITY;
  }
}

// ---- Philox4x32-10 -------------------------------------------------------------
__device__ __forceinline__ uint32_t philox_w0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                              uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0), lo0 = 0xD2511F53u * c0;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2), lo1 = 0xCD9E8D57u * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return c0;
}

// G = -log(-log U), U = (w + 0.5) / 2^32, with -log U formed from whichever of
// U and 1 - U is small, so that it keeps its precision in fp32 at both ends
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
  float e;
  if (w < 0x80000000u) {
    e = -logf(((float)w + 0.5f) * 2.3283064365386963e-10f);
  } else {
    const float um = ((float)(0xFFFFFFFFu - w) + 0.5f) * 2.3283064365386963e-10f;   // 1 - U
    e = -log1pf(-um);
  }
  return -logf(e);
}

// per (vocab chunk, row): the largest x_i + G_i and its index (lowest on ties)
__global__ void __launch_bounds__(256) gumbel_partial_kernel(ReqTable t, const float* logits, int V, float inv_t,
                                                             SeedTable sd, int nvc, GumbelPart* part,
                                                             const int32_t* status) {
  __shared__ float sv[8];
  __shared__ int si[8];
  __shared__ uint32_t s_pos;
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int c = blockIdx.x, row = blockIdx.y;
  if (threadIdx.x == 0) {   // request of the row, and the sequence index of the token the row scores
    int r = 0;
    while (r + 1 < t.n_req && t.row_off[r + 1] <= row) ++r;
    // depth of the row's node (parents read as given; a malformed tree, which the
    // walk rejects, only stops the climb early)
    int i = row - t.row_off[r], d = 0;
    while (i > 0 && d < kMaxRows) {
      const int p = t.parent[r][i];
      if (p < 0 || p >= i) break;
      i = p;
      ++d;
    }
    s_pos = (uint32_t)(sd.pos[r] + d + 1);
    si[0] = r;
  }
  __syncthreads();
  const int r = si[0];
  const uint32_t tpos = s_pos;
  const uint32_t k0 = (uint32_t)(sd.seed[r] & 0xFFFFFFFFull), k1 = (uint32_t)(sd.seed[r] >> 32);
  __syncthreads();
  const float* lr = logits + (size_t)row * V;
  float best = -INFINITY;
  int bi = INT_MAX;
  for (int k = 0; k < kVChunk / 256; ++k) {
    const int y = c * kVChunk + k * 256 + threadIdx.x;
    if (y < V) {
      const float x = lr[y] * inv_t;
      if (x != -INFINITY) {
        const float s = x + gumbel_from_word(philox_w0((uint32_t)y, tpos, 0u, 0u, k0, k1));
        if (s > best || (s == best && y < bi)) {
          best = s;
          bi = y;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(FULL, best, o);
    const int oi = __shfl_xor_sync(FULL, bi, o);
    if (ob > best || (ob == best && oi < bi)) {
      best = ob;
      bi = oi;
    }
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    sv[w] = best;
    si[w] = bi;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 1; i < 8; ++i)
      if (sv[i] > best || (sv[i] == best && si[i] < bi)) {
        best = sv[i];
        bi = si[i];
      }
    part[(size_t)row * nvc + c] = GumbelPart{best, bi};
  }
}

// per row (one warp): the row's draw from its chunk partials
__global__ void gumbel_pick_kernel(const GumbelPart* part, int nvc, int32_t* row_tokens, const int32_t* status) {
  pdl_wait();
  pdl_trigger();
  if (status_get(status) != 0) return;
  const int row = blockIdx.x, lane = threadIdx.x;
  float best = -INFINITY;
  int bi = INT_MAX;
  for (int c = lane; c < nvc; c += 32) {
    const GumbelPart p = part[(size_t)row * nvc + c];
    if (p.s > best || (p.s == best && p.idx < bi)) {
      best = p.s;
      bi = p.idx;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(FULL, best, o);
    const int oi = __shfl_xor_sync(FULL, bi, o);
    if (ob > best || (ob == best && oi < bi)) {
      best = ob;
      bi = oi;
    }
  }
  if (lane == 0) row_tokens[row] = bi == INT_MAX ? 0 : bi;
}

}  // namespace

int launch_filter(const float* logits, float* out, int rows, int vocab, float temperature, int top_k, float top_p,
                  float min_p, int32_t* status, cudaStream_t st) {
  const float inv_t = (float)(1.0 / (double)temperature);
  const float log_min_p = min_p > 0.f ? (float)std::log((double)min_p) : -INFINITY;
  return launch_pdl(filter_kernel, dim3(rows), dim3(kFilterThreads), 0, st, logits, out, vocab, inv_t, top_k,
                    (double)top_p, log_min_p, (const int32_t*)status);
}

int launch_gumbel_rows(const ReqTable& t, const float* logits, int vocab, float temperature, const SeedTable& sd,
                       GumbelPart* part, int32_t* row_tokens, int32_t* status, cudaStream_t st) {
  const int nvc = n_vchunks(vocab);
  const float inv_t = (float)(1.0 / (double)temperature);
  int rc = launch_pdl(gumbel_partial_kernel, dim3(nvc, t.total_rows), dim3(256), 0, st, t, logits, vocab, inv_t, sd,
                      nvc, part, (const int32_t*)status);
  if (rc) return rc;
  return launch_pdl(gumbel_pick_kernel, dim3(t.total_rows), dim3(32), 0, st, (const GumbelPart*)part, nvc, row_tokens,
                    (const int32_t*)status);
}

}  // namespace tv
