// Sampling filters and seeded Gumbel-max draws.
//
//  - filter: temperature, top_k, top_p and min_p through one function
//    [Exactness, §Sampling, second paragraph].  One thread-block cluster of
//    8 CTAs per row; each CTA keeps a slice of the row in shared memory and
//    the cluster sums its histograms through distributed shared memory.  The
//    k-th largest logit and the top-p boundary are found in two levels: a
//    256-bin histogram of (l_max - l) / T, which places the boundary in one
//    bin, then an exact pass over an order-preserving integer key of the
//    logits in that bin (256 sub-bins, then ranking when the last bin is
//    small; else radix selection, four 8-bit passes).  Weights are integers
//    (counts, or exp((l - l_max) / T) in units of 2^-32), so the result is
//    exact and the same on every run.
//  - Gumbel: the token at sequence index t is argmax_i (x_i + G_i), G_i Gumbel
//    noise from Philox4x32-10 keyed by (seed, t) [Exactness, §Sampling, third
//    paragraph]; token i takes word i mod 4 of the generator block at counter
//    (i div 4, t, 0, 0).  One pass of (vocab chunk, row) blocks and a per-row
//    pick.  Philox4x32-10 follows Salmon, Moraes, Dror and Shaw, "Parallel
//    random numbers: as easy as 1, 2, 3" (SC 2011).
#include <climits>
#include <cmath>

#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr unsigned FULL = 0xffffffffu;

// ---- filter --------------------------------------------------------------------------
constexpr int kFCluster = 8;            // CTAs per row at most (6 or 8, chosen at launch)
constexpr int kFThreads = 512;
constexpr int kFWarps = kFThreads / 32;
constexpr int kFBins = 256;
constexpr float kFBinsPerUnit = 8.f;    // level-1 bin width: 1/8 of a unit of (l_max - l) / T
constexpr float kFSubBins = 256.f;      // level-2 bins per level-1 bin
constexpr int kFilterMaxVocab = 262144;
constexpr int kFPriv = 4;               // private level-1 histograms per CTA (warp w adds into w mod 4)
constexpr int kCandCap = 4096;          // tokens a CTA lists per level; past that it rescans its slice
constexpr int kGatherMax = 512;         // last bins this small (cluster-wide) are finished by ranking
constexpr int kFScratch = kFPriv * 2 * kFBins * 4;   // bytes: private histograms, or the gathered tokens
constexpr int kFRegF4 = 16;             // float4s of its slice a thread also keeps in registers (the fast cut's passes)
static_assert(kGatherMax * 12 <= kFScratch, "gathered keys and weights fit the scratch area");

// order-preserving key: larger float -> larger unsigned; -0 and +0 share a
// key (they compare equal), NaN sorts lowest
__device__ __forceinline__ uint32_t fkey(float x) {
  if (x != x) return 0u;
  const uint32_t u = x == 0.f ? 0u : __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct FilterShared {
  unsigned long long hist[2][kFBins];   // this CTA's histogram (two, used in turn); the cluster reads them
  unsigned long long tot[kFBins];       // the cluster's histogram
  unsigned long long res[3];            // selected bin, the weight before it, the weight needed
  float pub_max;                        // this CTA's slice maximum (read by the cluster)
  float redf[kFWarps];
  float M;
  int cnt1;                             // this CTA's level-1 boundary-bin tokens
  int cnt2[2];                          // its level-2 boundary-bin tokens, per selection (read by the cluster)
  int off[kFCluster + 1];               // the cluster's level-2 boundary-bin tokens, prefix by CTA
  uint32_t key_sel;
  unsigned long long totw[kFBins];      // the fast cut: the cluster's weight histogram
  unsigned long long wsum[kFWarps];     // and block scans' warp totals
  unsigned long long csum[kFWarps];
  float pub_top;                        // the fast top_k cut: this CTA's grid anchor (read by the cluster)
  float tops[kFCluster];                // every CTA's anchor
};

// The cluster's histogram tot[] from every CTA's hist[hb] (after a cluster barrier).
__device__ __forceinline__ void cluster_hist(FilterShared& sh, int hb) {
  if (threadIdx.x < kFBins) {
    unsigned long long s = 0ull;
#pragma unroll
    for (int r = 0; r < kFCluster; ++r)
      if (r < (int)cluster_nctarank()) s += ld_dsmem_u64(dsmem_addr(&sh.hist[hb][threadIdx.x], r));
    sh.tot[threadIdx.x] = s;
  }
  __syncthreads();
}

// One warp: the first bin, counted from bin 0 upward (descending = false) or
// from bin 255 downward, at which the running weight reaches need; with frac > 0
// need is first set to ceil(frac * the histogram's total), at least 1.
// res[0] = the bin (~0 when the total falls short), res[1] = the weight before
// it, res[2] = need.
__device__ __forceinline__ void find_bin(FilterShared& sh, unsigned long long need, double frac, bool descending) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  if (frac > 0.0) {
    unsigned long long s = 0ull;
#pragma unroll
    for (int k = 0; k < kFBins / 32; ++k) s += sh.tot[k * 32 + lane];
    s = warp_sum(s);
    const double want = ceil(frac * (double)s);
    need = want < 1.0 ? 1ull : (want >= (double)s ? s : (unsigned long long)want);
  }
  unsigned long long above = 0ull, before = 0ull;
  int found = -1;
  for (int b0 = 0; b0 < kFBins && found < 0; b0 += 32) {
    const int b = descending ? kFBins - 1 - (b0 + lane) : b0 + lane;
    const unsigned long long h = sh.tot[b];
    unsigned long long incl = h;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += u;
    }
    const unsigned hit = __ballot_sync(FULL, above + incl >= need);
    if (hit) {
      const int L = __ffs(hit) - 1;
      found = descending ? kFBins - 1 - (b0 + L) : b0 + L;
      before = above + __shfl_sync(FULL, incl - h, L);
    }
    above += __shfl_sync(FULL, incl, 31);
  }
  if (lane == 0) {
    sh.res[0] = found < 0 ? ~0ull : (unsigned long long)found;
    sh.res[1] = before;
    sh.res[2] = need;
  }
}

// hist[digit(x)] += wt(x) over the tokens list[0..n) of the slice (all tokens
// 0..n-1 when list is null) that pass keep; one atomic per warp where all of
// the warp's tokens share a digit.
template <typename Keep, typename Digit, typename Weight>
__device__ __forceinline__ void hist_pass(unsigned long long* hist, const float* xs, const uint16_t* list, int n,
                                          Keep keep, Digit digit, Weight wt) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int j0 = warp * 32; j0 < n; j0 += kFThreads) {
    const int j = j0 + lane;
    bool ok = false;
    float x = 0.f;
    if (j < n) {
      x = xs[list ? (int)list[j] : j];
      ok = keep(x);
    }
    const unsigned m = __ballot_sync(FULL, ok);
    if (m == 0u) continue;
    const int d = ok ? digit(x) : 0;
    const int d0 = __shfl_sync(FULL, d, __ffs(m) - 1);
    const unsigned long long w = ok ? wt(x) : 0ull;
    if (__all_sync(FULL, !ok || d == d0)) {
      const unsigned long long s = warp_sum(w);
      if (lane == 0) atomicAdd(&hist[d0], s);
    } else if (ok) {
      atomicAdd(&hist[d], w);
    }
  }
}

// out[...] = the slice indices among list[0..n) (all 0..n-1 when list is null)
// that pass keep, one slot allocation per warp; *count ends at the number found,
// which may pass kCandCap (entries past it are not written).
template <typename Keep>
__device__ __forceinline__ void list_pass(uint16_t* out, int* count, const float* xs, const uint16_t* list, int n,
                                          Keep keep) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int j0 = warp * 32; j0 < n; j0 += kFThreads) {
    const int j = j0 + lane;
    int i = 0;
    bool in = false;
    if (j < n) {
      i = list ? (int)list[j] : j;
      in = keep(xs[i]);
    }
    const unsigned m = __ballot_sync(FULL, in);
    if (m == 0u) continue;
    int base = 0;
    if (lane == 0) base = atomicAdd(count, __popc(m));
    base = __shfl_sync(FULL, base, 0);
    const int slot = base + __popc(m & ((1u << lane) - 1u));
    if (in && slot < kCandCap) out[slot] = (uint16_t)i;
  }
}

// Over the tokens with key >= floor: the largest key K such that the weight of
// the tokens with key >= K reaches need (need = ceil(frac * their total weight)
// when frac > 0); floor when the total falls short.
//  level 1: bins of d = (M - l) / T * 8, which falls as l rises, so every token
//           of a lower bin has a larger key than every token of a higher one;
//  level 2: 256 sub-bins of the level-1 boundary bin, by the same rule;
//  level 3: the keys of the level-2 boundary bin: when the cluster holds at
//           most kGatherMax of them every CTA gathers them all and ranks them;
//           otherwise radix selection, 8 bits at a time from the top.
template <typename Weight>
__device__ uint32_t select_key(FilterShared& sh, const float* xs, uint16_t* cand1, uint16_t* cand2,
                               unsigned char* scratch, int n_loc, float M, float inv_t, uint32_t floor_key,
                               unsigned long long need, double frac, Weight wt, int sel, int& hb) {
  const int warp = threadIdx.x >> 5;
  auto dval = [&](float x) { return (M - x) * inv_t * kFBinsPerUnit; };
  auto bin_of = [&](float x) { return (int)fminf(dval(x), (float)(kFBins - 1)); };

  // level 1, in private histograms of 32-bit parts, weight = hi * 2^16 + lo:
  // weights are at most 2^32 and a private histogram sees at most n_loc / 4
  // tokens, so a part sums below 2^30
  uint32_t* priv = reinterpret_cast<uint32_t*>(scratch);
  for (int b = threadIdx.x; b < kFPriv * 2 * kFBins; b += kFThreads) priv[b] = 0u;
  if (threadIdx.x == 0) {
    sh.cnt1 = 0;
    sh.cnt2[sel] = 0;
    sh.key_sel = floor_key;
  }
  __syncthreads();
  uint32_t* ph = priv + (warp & (kFPriv - 1)) * 2 * kFBins;
  for (int i = threadIdx.x; i < n_loc; i += kFThreads) {
    const float x = xs[i];
    if (fkey(x) >= floor_key) {
      const int b = bin_of(x);
      const unsigned long long w = wt(x);
      atomicAdd(&ph[b], (uint32_t)(w & 0xFFFFull));
      const uint32_t hi = (uint32_t)(w >> 16);
      if (hi != 0u) atomicAdd(&ph[kFBins + b], hi);
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kFBins; b += kFThreads) {
    unsigned long long s = 0ull;
#pragma unroll
    for (int g = 0; g < kFPriv; ++g)
      s += (unsigned long long)priv[g * 2 * kFBins + b] + ((unsigned long long)priv[g * 2 * kFBins + kFBins + b] << 16);
    sh.hist[hb][b] = s;
  }
  cluster_sync_all();
  cluster_hist(sh, hb);
  hb ^= 1;
  find_bin(sh, need, frac, false);
  __syncthreads();
  const unsigned long long B1 = sh.res[0];
  if (B1 == ~0ull) return floor_key;   // the weight falls short: no cut
  need = sh.res[2] - sh.res[1];
  auto in1 = [&](float x) { return fkey(x) >= floor_key && bin_of(x) == (int)B1; };

  // level 2
  list_pass(cand1, &sh.cnt1, xs, nullptr, n_loc, in1);
  for (int b = threadIdx.x; b < kFBins; b += kFThreads) sh.hist[hb][b] = 0ull;
  __syncthreads();
  const int c1 = sh.cnt1;
  const bool listed1 = c1 <= kCandCap;
  auto sub_of = [&](float x) { return (int)fminf((dval(x) - (float)B1) * kFSubBins, (float)(kFBins - 1)); };
  auto keep1 = [&](float x) { return listed1 || in1(x); };
  hist_pass(sh.hist[hb], xs, listed1 ? cand1 : nullptr, listed1 ? c1 : n_loc, keep1, sub_of, wt);
  cluster_sync_all();
  cluster_hist(sh, hb);
  hb ^= 1;
  find_bin(sh, need, 0.0, false);
  __syncthreads();
  const int B2 = (int)sh.res[0];   // found: bin B1 holds at least need
  need -= sh.res[1];
  auto keep2 = [&](float x) { return keep1(x) && sub_of(x) == B2; };

  // level 3
  list_pass(cand2, &sh.cnt2[sel], xs, listed1 ? cand1 : nullptr, listed1 ? c1 : n_loc, keep2);
  cluster_sync_all();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int ncl = (int)cluster_nctarank();
    int c = lane < ncl ? ld_dsmem_s32(dsmem_addr(&sh.cnt2[sel], lane)) : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(FULL, c, o);
      if (lane >= o) c += u;
    }
    if (lane < ncl) sh.off[lane + 1] = c;
    if (lane == 0) sh.off[0] = 0;
  }
  __syncthreads();
  const int total = sh.off[cluster_nctarank()];

  if (total <= kGatherMax) {   // every CTA ranks the whole bin (each listed all of its tokens)
    unsigned long long* gw = reinterpret_cast<unsigned long long*>(scratch);
    uint32_t* gk = reinterpret_cast<uint32_t*>(scratch + kGatherMax * sizeof(unsigned long long));
    for (int t = threadIdx.x; t < total; t += kFThreads) {
      int r = 0;
      while (t >= sh.off[r + 1]) ++r;
      const int ci = ld_dsmem_u16(dsmem_addr(&cand2[t - sh.off[r]], r));
      const float x = ld_dsmem_f32(dsmem_addr(&xs[ci], r));
      gk[t] = fkey(x);
      gw[t] = wt(x);
    }
    __syncthreads();
    for (int t = threadIdx.x; t < total; t += kFThreads) {
      const uint32_t k = gk[t];
      unsigned long long above = 0ull, eq = 0ull;
      for (int j = 0; j < total; ++j) {
        const uint32_t kj = gk[j];
        const unsigned long long wj = gw[j];
        above += kj > k ? wj : 0ull;
        eq += kj == k ? wj : 0ull;
      }
      if (above < need && need <= above + eq) sh.key_sel = k;   // one key; its ties write the same value
    }
    __syncthreads();
    return sh.key_sel;
  }

  const int c2 = sh.cnt2[sel];
  const bool listed2 = c2 <= kCandCap;
  uint32_t prefix = 0u, mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < kFBins; b += kFThreads) sh.hist[hb][b] = 0ull;
    __syncthreads();
    hist_pass(
        sh.hist[hb], xs, listed2 ? cand2 : nullptr, listed2 ? c2 : n_loc,
        [&](float x) { return (listed2 || keep2(x)) && (fkey(x) & mask) == prefix; },
        [&](float x) { return (int)((fkey(x) >> shift) & 255u); }, wt);
    cluster_sync_all();
    cluster_hist(sh, hb);
    hb ^= 1;
    find_bin(sh, need, 0.0, true);
    __syncthreads();
    const unsigned long long f = sh.res[0];
    if (f == ~0ull) return floor_key;   // not reached: the bin holds at least need
    prefix |= (uint32_t)f << shift;
    mask |= 255u << shift;
    need -= sh.res[1];
  }
  return prefix;
}

// The fast cut.  One level-1 pass over the slice counts the tokens (key >= 1:
// not NaN) per bin, and weighs them too when top_p is the only cut; the
// cluster's histogram places the boundary bin B of the first cut (the k-th
// largest, else the top_p boundary).  When B and the bins above it hold at
// most kFastCap tokens cluster-wide, every CTA lists its tokens of bins <= B,
// gathers the cluster's (a thread a candidate) and takes the cuts exactly,
// with the integer weights of select_key and no further cluster barrier, by
// counting: a candidate's key is the k-th largest when fewer than k keys are
// larger and at least k are at least as large, and the top_p key when the
// weight of the larger keys falls short of need and with its ties reaches it;
// kfloor = the top_k key, then the top_p key among the tokens at or above it.
// Returns false, having decided nothing, when the candidates are more (the
// caller then takes the general path after a cluster barrier).  `region`
// holds the private histograms, then the gathered keys, logits and weights.
constexpr int kFastCap = 256;

// Over a histogram h[256] (a thread a bin, threads 0..255): the first bin at
// which the running sum reaches need, the sum before it and the running
// count (c) through it; res = {bin or ~0, count through it}.  Block-wide scan.
__device__ __forceinline__ void boundary_bin(FilterShared& sh, const unsigned long long* h,
                                             const unsigned long long* c, unsigned long long need) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = 0ull, y = 0ull;
  if (threadIdx.x < kFBins) {
    x = h[threadIdx.x];
    y = c[threadIdx.x];
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long u = __shfl_up_sync(FULL, x, o), v = __shfl_up_sync(FULL, y, o);
    if (lane >= o) {
      x += u;
      y += v;
    }
  }
  if (lane == 31 && warp < kFBins / 32) {
    sh.wsum[warp] = x;
    sh.csum[warp] = y;
  }
  if (threadIdx.x == 0) sh.res[0] = ~0ull;
  __syncthreads();
  if (threadIdx.x < kFBins) {
    unsigned long long bx = 0ull, by = 0ull;
    for (int v = 0; v < warp; ++v) {
      bx += sh.wsum[v];
      by += sh.csum[v];
    }
    const unsigned long long incl = bx + x, excl = incl - h[threadIdx.x];
    if (incl >= need && excl < need) {   // the one bin where the running sum crosses need
      sh.res[0] = (unsigned long long)threadIdx.x;
      sh.res[1] = by + y;
    }
  }
  __syncthreads();
}

__device__ bool fast_cut(FilterShared& sh, const float* xs, const float4 (&xr)[kFRegF4], bool inreg,
                         uint16_t* cand, unsigned char* region, int n_loc, float& M, float m_loc, float inv_t,
                         int top_k, float top_p, bool by_k, float log_min_p, float* orow) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ncl = (int)cluster_nctarank();
  // top_p alone: bins of (M - x) / T * 8 under the cluster maximum M.  top_k:
  // bins on a fixed grid, g(x) = floor(x / T * 8), counted down from each CTA's
  // own anchor floor(m_loc / T * 8); the cluster's histogram shifts each CTA's
  // by its anchor's distance to the highest anchor, exact in bins 0..254 (bin
  // 255 lumps the rest), so no maximum needs exchanging first
  const bool anchored = by_k;
  const float s8 = inv_t * kFBinsPerUnit;
  const float top_loc = floorf(m_loc * s8);
  // the grid index g(x) = floor(x / T * 8) as an integer (saturating; every
  // anchor is below 2^23 in magnitude when the cut goes on, so a token at or
  // below the maximum never saturates upward and one saturated downward lands
  // in bin 255 / is never listed, as it would be in float)
  auto grid = [&](float x) { return __float2int_rd(x * s8); };
  const int top_loc_i = (fabsf(top_loc) < 8388608.f) ? (int)top_loc : 0;
  auto bin_of = [&](float x) { return (int)fminf((M - x) * inv_t * kFBinsPerUnit, (float)(kFBins - 1)); };
  auto lbin = [&](float x) {
    return anchored ? (int)min((uint32_t)top_loc_i - (uint32_t)grid(x), (uint32_t)(kFBins - 1)) : bin_of(x);
  };
  // the float4s of the slice: [0, kFThreads kFRegF4) from registers when inreg
  // (NaN past the slice), the rest from shared memory
  const int n4 = n_loc >> 2;
  const int j_smem = inreg ? kFThreads * kFRegF4 : 0;
  auto wt = [&](float x) { return (unsigned long long)__float2ull_rn(expf((x - M) * inv_t) * 4294967296.f); };
  // level 1 into private histograms: counts; weights as hi * 2^16 + lo
  uint32_t* pc = reinterpret_cast<uint32_t*>(region);            // [kFPriv][kFBins]
  uint32_t* pw = pc + kFPriv * kFBins;                            // [kFPriv][2][kFBins]
  for (int b = threadIdx.x; b < kFPriv * 3 * kFBins; b += kFThreads) pc[b] = 0u;
  if (threadIdx.x == 0) {
    sh.cnt1 = 0;
    sh.pub_top = top_loc;
  }
  __syncthreads();
  {
    uint32_t* myc = pc + (warp & (kFPriv - 1)) * kFBins;
    uint32_t* myw = pw + (warp & (kFPriv - 1)) * 2 * kFBins;
    auto one = [&](float x) {
      if (x == x) {   // NaN is never counted
        const int b = lbin(x);
        atomicAdd(&myc[b], 1u);
        if (!by_k) {
          const unsigned long long w = wt(x);
          atomicAdd(&myw[b], (uint32_t)(w & 0xFFFFull));
          const uint32_t hi = (uint32_t)(w >> 16);
          if (hi != 0u) atomicAdd(&myw[kFBins + b], hi);
        }
      }
    };
    if (inreg) {
#pragma unroll
      for (int r = 0; r < kFRegF4; ++r) {
        one(xr[r].x);
        one(xr[r].y);
        one(xr[r].z);
        one(xr[r].w);
      }
    }
    for (int j = j_smem + threadIdx.x; j < n4; j += kFThreads) {
      const float4 x4 = reinterpret_cast<const float4*>(xs)[j];
      one(x4.x);
      one(x4.y);
      one(x4.z);
      one(x4.w);
    }
    for (int i = 4 * n4 + threadIdx.x; i < n_loc; i += kFThreads) one(xs[i]);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < kFBins; b += kFThreads) {
    unsigned long long c = 0ull, w = 0ull;
#pragma unroll
    for (int g = 0; g < kFPriv; ++g) {
      c += pc[g * kFBins + b];
      w += (unsigned long long)pw[g * 2 * kFBins + b] + ((unsigned long long)pw[g * 2 * kFBins + kFBins + b] << 16);
    }
    sh.hist[0][b] = c;
    sh.hist[1][b] = w;
  }
  cluster_sync_all();
  float top = 0.f;   // anchored: the highest anchor
  if (anchored) {    // every CTA's anchor and maximum
    if (threadIdx.x < 32) {
      float t = -INFINITY, m = -INFINITY;
      if (lane < ncl) {
        t = ld_dsmem_f32(dsmem_addr(&sh.pub_top, lane));
        m = ld_dsmem_f32(dsmem_addr(&sh.pub_max, lane));
        sh.tops[lane] = t;
      }
      // anchors past 2^23 are not exact integers: no fast cut
      const bool bad = __any_sync(FULL, t != -INFINITY && fabsf(t) >= 8388608.f);
      t = warp_max(t);
      m = warp_max(m);
      if (lane == 0) {
        sh.M = m;
        sh.res[0] = bad ? 1ull : 0ull;
        sh.key_sel = __float_as_uint(t);
      }
    }
    __syncthreads();
    M = sh.M;
    top = __uint_as_float(sh.key_sel);
    if (M == -INFINITY || sh.res[0] != 0ull) return false;
  }
  unsigned long long wall = 0ull;   // this bin's cluster weight
  if (threadIdx.x < kFBins) {   // every remote load issued before the sums
    unsigned long long c[kFCluster], wv[kFCluster];
#pragma unroll
    for (int r = 0; r < kFCluster; ++r) {
      c[r] = 0ull;
      wv[r] = 0ull;
      if (r >= ncl) continue;
      int lb = threadIdx.x;
      if (anchored) {   // this CTA's bin at global bin threadIdx.x, or none
        const float d = top - sh.tops[r];
        lb = (threadIdx.x < kFBins - 1 && d <= (float)(kFBins - 2)) ? (int)threadIdx.x - (int)d : -1;
      }
      c[r] = lb >= 0 ? ld_dsmem_u64(dsmem_addr(&sh.hist[0][lb], r)) : 0ull;
      wv[r] = by_k ? 0ull : ld_dsmem_u64(dsmem_addr(&sh.hist[1][threadIdx.x], r));
    }
    unsigned long long cs = 0ull;
#pragma unroll
    for (int r = 0; r < kFCluster; ++r) {
      cs += c[r];
      wall += wv[r];
    }
    // anchored: the last bin lumps tokens of every depth; as the boundary it
    // holds too many candidates for the fast cut
    if (anchored && threadIdx.x == kFBins - 1) cs = 1ull << 40;
    sh.tot[threadIdx.x] = cs;
    sh.totw[threadIdx.x] = wall;
  }
  // the need of the first cut: k, else ceil(top_p x the row's weight)
  unsigned long long need = (unsigned long long)top_k;
  if (!by_k) {   // one thread evaluates the need (FP64 is slow here)
    const unsigned long long ws = warp_sum(wall);
    if (lane == 0 && warp < kFBins / 32) sh.csum[warp] = ws;
    __syncthreads();
    if (threadIdx.x == 0) {
      unsigned long long s = 0ull;
      for (int v = 0; v < kFBins / 32; ++v) s += sh.csum[v];
      const double want = ceil((double)top_p * (double)s);
      sh.res[2] = want < 1.0 ? 1ull : (want >= (double)s ? s : (unsigned long long)want);
    }
    __syncthreads();
    need = sh.res[2];
  }
  __syncthreads();
  boundary_bin(sh, by_k ? sh.tot : sh.totw, sh.tot, need);
  if (sh.res[0] == ~0ull || sh.res[1] > (unsigned long long)kFastCap) return false;
  const int B = (int)sh.res[0];
  const int C = (int)sh.res[1];
  
  // the candidates (key >= 1, bin <= B), listed by every CTA with their
  // logits; every output of the slice is written -inf on the way (the kept
  // candidates are written again at the end, after a CTA barrier)
  float* cx = reinterpret_cast<float*>(region + kFPriv * 3 * kFBins * sizeof(uint32_t));   // past the histograms
  {
    const int gmin = (int)top - B;   // anchored: bins <= B are g(x) >= top - B (top an integer below 2^23)
    auto in = [&](float x) { return x == x && (anchored ? grid(x) >= gmin : bin_of(x) <= B); };
    auto put = [&](bool ok, int i, float x) {
      const unsigned mk = __ballot_sync(FULL, ok);
      if (mk == 0u) return;
      int base = 0;
      if (lane == 0) base = atomicAdd(&sh.cnt1, __popc(mk));
      base = __shfl_sync(FULL, base, 0);
      if (ok) {   // at most C <= kFastCap a CTA
        const int slot = base + __popc(mk & ((1u << lane) - 1u));
        cand[slot] = (uint16_t)i;
        cx[slot] = x;
      }
    };
    const bool vec_out = (reinterpret_cast<uintptr_t>(orow) & 15u) == 0;
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    auto clear4 = [&](int j) {
      if (vec_out) {
        reinterpret_cast<float4*>(orow)[j] = ninf;
      } else {
        orow[4 * j] = -INFINITY;
        orow[4 * j + 1] = -INFINITY;
        orow[4 * j + 2] = -INFINITY;
        orow[4 * j + 3] = -INFINITY;
      }
    };
    if (inreg) {
#pragma unroll
      for (int r = 0; r < kFRegF4; ++r) {   // every lane of the warp takes every step
        const int j = (int)threadIdx.x + kFThreads * r;
        if (j < n4) clear4(j);
        const float4 x4 = xr[r];
        const bool a0 = in(x4.x), a1 = in(x4.y), a2 = in(x4.z), a3 = in(x4.w);
        if (__any_sync(FULL, a0 || a1 || a2 || a3)) {
          put(a0, 4 * j, x4.x);
          put(a1, 4 * j + 1, x4.y);
          put(a2, 4 * j + 2, x4.z);
          put(a3, 4 * j + 3, x4.w);
        }
      }
    }
    for (int j0 = j_smem + warp * 32; j0 < n4; j0 += kFThreads) {   // warp-uniform trip count
      const int j = j0 + lane;
      float4 x4 = make_float4(NAN, NAN, NAN, NAN);
      if (j < n4) {
        x4 = reinterpret_cast<const float4*>(xs)[j];
        clear4(j);
      }
      const bool a0 = in(x4.x), a1 = in(x4.y), a2 = in(x4.z), a3 = in(x4.w);
      if (__any_sync(FULL, a0 || a1 || a2 || a3)) {
        put(a0, 4 * j, x4.x);
        put(a1, 4 * j + 1, x4.y);
        put(a2, 4 * j + 2, x4.z);
        put(a3, 4 * j + 3, x4.w);
      }
    }
    if (warp == 0) {
      const int i = 4 * n4 + lane;
      const float x = i < n_loc ? xs[i] : NAN;
      if (i < n_loc) orow[i] = -INFINITY;
      put(in(x), i, x);
    }
  }
  cluster_sync_all();
  if (threadIdx.x < 32) {
    int c = lane < ncl ? ld_dsmem_s32(dsmem_addr(&sh.cnt1, lane)) : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(FULL, c, o);
      if (lane >= o) c += u;
    }
    if (lane < ncl) sh.off[lane + 1] = c;
    if (lane == 0) sh.off[0] = 0;
  }
  __syncthreads();
  // gathered: thread i < C holds candidate i; keys and weights shared
  uint32_t* gk = reinterpret_cast<uint32_t*>(region);
  unsigned long long* gw = reinterpret_cast<unsigned long long*>(region + kFastCap * sizeof(uint32_t));
  uint32_t key = 0u;
  unsigned long long w = 0ull;
  if ((int)threadIdx.x < C) {
    int r = 0;
    while ((int)threadIdx.x >= sh.off[r + 1]) ++r;
    const float x = ld_dsmem_f32(dsmem_addr(&cx[threadIdx.x - sh.off[r]], r));
    key = fkey(x);
    w = top_p < 1.f ? wt(x) : 0ull;
    gk[threadIdx.x] = key;
    gw[threadIdx.x] = w;
  }
  cluster_arrive();   // no more reads of other CTAs' shared memory
  if (threadIdx.x == 0) {
    sh.key_sel = 1u;   // above every NaN key
    sh.res[2] = 0ull;
  }
  __syncthreads();
  // one pass over the candidates: the count and the weight of the keys above
  // and at or above each candidate's own; G adjacent threads share a
  // candidate (each every G-th key), summed across them by shuffles
  int G = 1;
  while (G < 32 && G * 2 * C <= kFThreads) G <<= 1;
  const int ci = (int)threadIdx.x / G, part = (int)threadIdx.x % G;
  const uint32_t ki = ci < C ? gk[ci] : 0u;
  int above = 0, ge = 0;
  unsigned long long wabove = 0ull, wge = 0ull;
  if (ci < C) {
#pragma unroll 4
    for (int j = part; j < C; j += G) {
      const uint32_t kj = gk[j];
      const unsigned long long wj = gw[j];
      above += kj > ki;
      ge += kj >= ki;
      wabove += kj > ki ? wj : 0ull;
      wge += kj >= ki ? wj : 0ull;
    }
  }
  for (int o = 1; o < G; o <<= 1) {   // G divides 32: the group sits in one warp
    above += __shfl_xor_sync(FULL, above, o);
    ge += __shfl_xor_sync(FULL, ge, o);
    wabove += __shfl_xor_sync(FULL, wabove, o);
    wge += __shfl_xor_sync(FULL, wge, o);
  }
  // top_k: the k-th largest key, and top_p's need over the weight at or above
  // it, evaluated by the key's threads only (FP64 is slow here; a key's ties
  // write the same values)
  if (ci < C && part == 0 && by_k && above < top_k && ge >= top_k) {
    sh.key_sel = ki;
    if (top_p < 1.f) {
      const double want = ceil((double)top_p * (double)wge);
      sh.res[2] = want < 1.0 ? 1ull : (want >= (double)wge ? wge : (unsigned long long)want);
    }
  }
  __syncthreads();
  uint32_t kfloor = sh.key_sel;
  if (top_p < 1.f) {
    const unsigned long long nd = by_k ? sh.res[2] : need;
    __syncthreads();   // every thread has read the top_k key
    if (ci < C && part == 0 && ki >= kfloor && wabove < nd && wge >= nd) sh.key_sel = ki;
    __syncthreads();
    kfloor = sh.key_sel;
  }
  // the kept candidates' outputs: x = l / T when key >= kfloor and min_p holds
  for (int s2 = threadIdx.x; s2 < sh.cnt1; s2 += kFThreads) {
    const float l = cx[s2];
    if (fkey(l) >= kfloor && (l - M) * inv_t >= log_min_p) orow[cand[s2]] = l * inv_t;
  }
  cluster_wait();
  return true;
}

__device__ __forceinline__ float block_max(float v, float* red) {
  v = warp_max(v);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
  for (int i = 1; i < kFWarps; ++i) m = fmaxf(m, red[i]);
  return m;
}

// One cluster per row; CTA `rank` holds tokens [rank * slice, rank * slice + slice).
// out = x = logit / T where kept, -inf elsewhere; selection on the raw logits
// (the scale by 1/T keeps their order).  Dynamic shared memory: the slice, the
// level-1 and level-2 lists, the scratch area.
__global__ void __launch_bounds__(kFThreads)
    filter_kernel(const float* logits, float* out, int V, int slice, float inv_t, int top_k, float top_p,
                  float log_min_p, const int32_t* status) {
  __shared__ FilterShared sh;
  extern __shared__ __align__(16) unsigned char dyn[];
  float* xs = reinterpret_cast<float*>(dyn);
  uint16_t* cand1 = reinterpret_cast<uint16_t*>(dyn + (size_t)slice * sizeof(float));
  uint16_t* cand2 = cand1 + kCandCap;
  unsigned char* scratch = reinterpret_cast<unsigned char*>(cand2 + kCandCap);
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;   // the same status for every CTA of the cluster
  const uint32_t rank = cluster_ctarank();
  const int row = blockIdx.y;
  const int lo = (int)rank * slice;
  const int n_loc = max(0, min(V - lo, slice));
  const float* lr = logits + (size_t)row * V + lo;
  float* orow = out + (size_t)row * V + lo;

  float mx = -INFINITY;
  // float4 where the row slice is 16-byte aligned (the slice offset is a
  // multiple of 8 tokens), the tail one by one
  const bool vec_in = (reinterpret_cast<uintptr_t>(lr) & 15u) == 0;
  const int n4 = vec_in ? n_loc >> 2 : 0;
  // the first kFThreads kFRegF4 float4s are kept in registers too (NaN past
  // the slice), for the fast cut's passes
  float4 xr[kFRegF4];
#pragma unroll
  for (int r = 0; r < kFRegF4; ++r) {
    const int j = (int)threadIdx.x + kFThreads * r;
    xr[r] = make_float4(NAN, NAN, NAN, NAN);
    if (j < n4) {
      const float4 v = reinterpret_cast<const float4*>(lr)[j];
      xr[r] = v;
      reinterpret_cast<float4*>(xs)[j] = v;
      mx = fmaxf(fmaxf(mx, fmaxf(v.x, v.y)), fmaxf(v.z, v.w));
    }
  }
  for (int j = kFThreads * kFRegF4 + threadIdx.x; j < n4; j += kFThreads) {
    const float4 v = reinterpret_cast<const float4*>(lr)[j];
    reinterpret_cast<float4*>(xs)[j] = v;
    mx = fmaxf(fmaxf(mx, fmaxf(v.x, v.y)), fmaxf(v.z, v.w));
  }
  for (int i = 4 * n4 + threadIdx.x; i < n_loc; i += kFThreads) {
    const float v = lr[i];
    xs[i] = v;
    mx = fmaxf(mx, v);
  }
  mx = block_max(mx, sh.redf);
  if (threadIdx.x == 0) sh.pub_max = mx;
  int hb = 0;
  uint32_t kfloor = 1u;   // above every NaN key
  const bool by_k = top_k > 0 && top_k < V;
  float M = -INFINITY;
  unsigned char* region = reinterpret_cast<unsigned char*>(cand2);
  if (by_k) {   // the fast top_k cut reads the cluster maximum with its histograms
    if (fast_cut(sh, xs, xr, vec_in, cand1, region, n_loc, M, mx, inv_t, top_k, top_p, true, log_min_p, orow))
      return;   // outputs written, and the cluster's reads of this CTA done
    cluster_sync_all();   // every CTA has read the fast cut's shared memory
  } else {
    cluster_sync_all();
    if (threadIdx.x < 32) {
      float m = (int)threadIdx.x < (int)cluster_nctarank() ? ld_dsmem_f32(dsmem_addr(&sh.pub_max, threadIdx.x))
                                                             : -INFINITY;
      m = warp_max(m);
      if (threadIdx.x == 0) sh.M = m;
    }
    __syncthreads();
    M = sh.M;
    if (M != -INFINITY && top_p < 1.f) {
      if (fast_cut(sh, xs, xr, vec_in, cand1, region, n_loc, M, mx, inv_t, top_k, top_p, false, log_min_p, orow))
        return;
      cluster_sync_all();
    }
  }
  const bool done = M == -INFINITY || (!by_k && !(top_p < 1.f));
  if (!done) {
    if (top_k > 0 && top_k < V)
      kfloor = select_key(sh, xs, cand1, cand2, scratch, n_loc, M, inv_t, kfloor, (unsigned long long)top_k, 0.0,
                          [](float) { return 1ull; }, 0, hb);
    if (top_p < 1.f)   // weights: exp((l - l_max) / T) in units of 2^-32, at most 2^32
      kfloor = select_key(
          sh, xs, cand1, cand2, scratch, n_loc, M, inv_t, kfloor, 0ull, (double)top_p,
          [=](float x) { return (unsigned long long)__float2ull_rn(expf((x - M) * inv_t) * 4294967296.f); }, 1, hb);
  }
  // min_p: x >= x_max + log(min_p), i.e. (l - l_max) / T >= log(min_p)
  auto filt = [&](float l) {
    const bool keep = M != -INFINITY && fkey(l) >= kfloor && (l - M) * inv_t >= log_min_p;
    return keep ? l * inv_t : -INFINITY;
  };
  const int o4 = (reinterpret_cast<uintptr_t>(orow) & 15u) == 0 ? n_loc >> 2 : 0;
  for (int j = threadIdx.x; j < o4; j += kFThreads) {
    const float4 l = reinterpret_cast<const float4*>(xs)[j];
    reinterpret_cast<float4*>(orow)[j] = make_float4(filt(l.x), filt(l.y), filt(l.z), filt(l.w));
  }
  for (int i = 4 * o4 + threadIdx.x; i < n_loc; i += kFThreads) orow[i] = filt(xs[i]);
  cluster_sync_all();   // no CTA leaves while the cluster may still read its shared memory
}

// ---- Philox4x32-10 -------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
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
  return make_uint4(c0, c1, c2, c3);
}

// G = -log(E), E = -log U, U = (w + 0.5) / 2^32.  Near U = 1, E is formed
// from v = 1 - U = (2^32 - 1 - w + 0.5) / 2^32 by the series
// -log(1 - v) = v + v^2/2 + v^3/3 + ... (to v^5; the rest is below 2^-25 of
// E for v < 2^-5), so E keeps its relative precision at both ends.
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
  const float u = ((float)w + 0.5f) * 2.3283064365386963e-10f;
  const float v = ((float)(~w) + 0.5f) * 2.3283064365386963e-10f;
  const float e_series = v * (1.f + v * (0.5f + v * (0.33333334f + v * (0.25f + v * 0.2f))));
  const float e = v < 0.03125f ? e_series : -__logf(u);
  return -__logf(e);
}

// per (vocab chunk, row): the largest x_i + G_i and its index (lowest on ties)
__global__ void __launch_bounds__(256) gumbel_partial_kernel(ReqTable t, const float* logits, int V, float inv_t,
                                                             SeedTable sd, int nvc, int vec4, GumbelPart* part,
                                                             const int32_t* status) {
  __shared__ float sv[8];
  __shared__ int si[8];
  __shared__ int s_par[32];
  __shared__ uint32_t s_pos;
  __shared__ int s_req;
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int c = blockIdx.x, row = blockIdx.y;
  if (threadIdx.x < 32) {   // request of the row, and the sequence index of the token the row scores
    const int lane = threadIdx.x;
    int r = 0;
    while (r + 1 < t.n_req && t.row_off[r + 1] <= row) ++r;
    const int n = t.n[r];
    s_par[lane] = lane < n ? t.parent[r][lane] : -1;
    __syncwarp();
    if (lane == 0) {
      // depth of the row's node (a malformed tree, which the walk rejects, only
      // stops the climb early)
      int i = row - t.row_off[r], d = 0;
      while (i > 0 && d < kMaxRows) {
        const int p = s_par[i];
        if (p < 0 || p >= i) break;
        i = p;
        ++d;
      }
      s_pos = (uint32_t)(sd.pos[r] + d + 1);
      s_req = r;
    }
  }
  __syncthreads();
  const int r = s_req;
  const uint32_t tpos = s_pos;
  const uint32_t k0 = (uint32_t)(sd.seed[r] & 0xFFFFFFFFull), k1 = (uint32_t)(sd.seed[r] >> 32);
  const float* lr = logits + (size_t)row * V;
  float best = -INFINITY;
  int bi = INT_MAX;
#pragma unroll
  for (int k = 0; k < kVChunk / 1024; ++k) {
    const int g = c * (kVChunk / 4) + k * 256 + threadIdx.x;   // generator block: tokens 4g .. 4g + 3
    const int y0 = 4 * g;
    if (y0 >= V) continue;
    float l[4];
    if (vec4) {
      const float4 q = *reinterpret_cast<const float4*>(lr + y0);
      l[0] = q.x;
      l[1] = q.y;
      l[2] = q.z;
      l[3] = q.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) l[j] = y0 + j < V ? lr[y0 + j] : -INFINITY;
    }
    const uint4 w = philox4x32_10((uint32_t)g, tpos, 0u, 0u, k0, k1);
    const uint32_t wj[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float x = l[j] * inv_t;
      if (x != -INFINITY) {
        const float s = x + gumbel_from_word(wj[j]);
        if (s > best) {   // tokens in increasing order: the first of equal scores stays
          best = s;
          bi = y0 + j;
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

std::atomic<bool> g_filter_smem_set[64];

// tokens per CTA of a row's cluster (a multiple of 8, so the index array that
// follows the slice stays 16-byte aligned)
int filter_slice(int vocab, int ncl) { return ((vocab + ncl - 1) / ncl + 7) / 8 * 8; }
size_t filter_smem(int vocab, int ncl) {
  return (size_t)filter_slice(vocab, ncl) * sizeof(float) + 2 * kCandCap * sizeof(uint16_t) + kFScratch;
}
// dynamic shared memory that leaves room for one CTA an SM only
constexpr size_t kFOnePerSm = 110 * 1024;
std::atomic<int> g_filter_fit[64][2];   // clusters of 8 / of 6 active at once at one CTA an SM (0: unknown)

int filter_fit(int dev, int ncl) {
  std::atomic<int>& slot = g_filter_fit[dev][ncl == 8 ? 0 : 1];
  int n = slot.load(std::memory_order_relaxed);
  if (n > 0) return n;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = (unsigned)ncl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(ncl, 1, 1);
  cfg.blockDim = dim3(kFThreads, 1, 1);
  cfg.dynamicSmemBytes = kFOnePerSm;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, (void*)filter_kernel, &cfg) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    n = 1;
  }
  slot.store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace

// One cluster per row.  The rows' clusters run side by side when each CTA has
// an SM of its own: clusters of 8 when that many fit the GPU's partition into
// clusters, else of 6 (more clusters fit; a third more tokens a CTA), padding
// the shared memory to one CTA an SM; beyond that clusters of 8 share SMs.
int launch_filter(const float* logits, float* out, int rows, int vocab, float temperature, int top_k, float top_p,
                  float min_p, int32_t* status, cudaStream_t st) {
  if (vocab > kFilterMaxVocab) return TV_E_UNSUPPORTED;
  const float inv_t = (float)(1.0 / (double)temperature);
  const float log_min_p = min_p > 0.f ? (float)std::log((double)min_p) : -INFINITY;
  // the limit is raised once per device, to what the largest vocabulary needs
  const size_t max_smem = filter_smem(kFilterMaxVocab, 6);
  int rc = ensure_smem_limit(filter_kernel, max_smem, g_filter_smem_set);
  if (rc) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TV_E_CUDA;
  int ncl = kFCluster;
  size_t smem = filter_smem(vocab, kFCluster);
  if (rows <= filter_fit(dev, 8)) {
    smem = smem > kFOnePerSm ? smem : kFOnePerSm;
  } else if (rows <= filter_fit(dev, 6)) {
    ncl = 6;
    smem = filter_smem(vocab, 6);
    smem = smem > kFOnePerSm ? smem : kFOnePerSm;
  }
  const int slice = filter_slice(vocab, ncl);
  return launch_pdl_cluster(filter_kernel, dim3(ncl, rows), dim3(kFThreads), smem, st, ncl, logits, out, vocab, slice,
                            inv_t, top_k, top_p, log_min_p, (const int32_t*)status);
}

int launch_gumbel_rows(const ReqTable& t, const float* logits, int vocab, float temperature, const SeedTable& sd,
                       GumbelPart* part, int32_t* row_tokens, int32_t* status, cudaStream_t st) {
  const int nvc = n_vchunks(vocab);
  const float inv_t = (float)(1.0 / (double)temperature);
  const int vec4 = (vocab % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15u) == 0) ? 1 : 0;
  int rc = launch_pdl(gumbel_partial_kernel, dim3(nvc, t.total_rows), dim3(256), 0, st, t, logits, vocab, inv_t, sd,
                      nvc, vec4, part, (const int32_t*)status);
  if (rc) return rc;
  return launch_pdl(gumbel_pick_kernel, dim3(t.total_rows), dim3(32), 0, st, (const GumbelPart*)part, nvc, row_tokens,
                    (const int32_t*)status);
}

}  // namespace tv
