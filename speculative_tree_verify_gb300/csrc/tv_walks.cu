// Accept walks and the KV commit.
//
//  - greedy walk: one warp per request, lanes = tree nodes [Drafters and tree
//    verify, §The round, step 3];
//  - residual walk: a multi-CTA pass of per-chunk softmax statistics over the
//    logits, then one warp per request walks the tree [Algorithm and
//    correctness contract, §Deterministic tree candidates and residual
//    verification];
//  - commit: gathers the accepted rows down into place [Drafters and tree
//    verify, §Tree verify through recurrent layers, last paragraph].
#include <climits>

#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr unsigned FULL = 0xffffffffu;

// ---------------------------------------------------------------------------
// greedy: cur = root; repeat { t = argmax[cur]; the child of cur carrying t? }
// ---------------------------------------------------------------------------
__global__ void accept_greedy_kernel(ReqTable t, const int32_t* argmax, int32_t* path, int32_t* accept_len,
                                     int32_t* out_tokens, int32_t* status) {
  const int r = blockIdx.x, lane = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (status_get(status) != 0) return;
  const int n = t.n[r], row0 = t.row_off[r];
  int par, tok;
  const int err = validate_tree_warp(t.parent[r], t.token[r], n, 0, par, tok);
  if (err != TV_OK) {
    if (lane == 0) status_set(status, err);
    return;
  }
  int cur = 0, a = 0;
  if (lane == 0) path[row0] = 0;
  for (;;) {
    const int want = argmax[row0 + cur];
    const unsigned hit = __ballot_sync(FULL, lane > 0 && lane < n && par == cur && tok == want);
    if (hit == 0u) {
      if (lane == 0) out_tokens[row0 + a] = want;   // the model's token at the stopping node
      break;
    }
    const int c = __ffs(hit) - 1;
    const int ctok = __shfl_sync(FULL, tok, c);
    ++a;
    if (lane == 0) {
      path[row0 + a] = c;
      out_tokens[row0 + a - 1] = ctok;
    }
    cur = c;
  }
  if (lane == 0) accept_len[r] = a;
}

// ---------------------------------------------------------------------------
// residual walk, pass 1: per (row, vocab chunk) the chunk max m and
// s = sum exp((l - m) / T).  grid (chunks, rows), block 256.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) row_stats_kernel(const float* logits, int V, float inv_t, int nvc,
                                                        RowStat* stats, const int32_t* status) {
  __shared__ float red[8];
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int c = blockIdx.x, row = blockIdx.y;
  const float* lr = logits + (size_t)row * V;
  const int y0 = c * kVChunk;
  float v[kVChunk / 256];
  float mx = -INFINITY;
#pragma unroll
  for (int k = 0; k < kVChunk / 256; ++k) {
    const int y = y0 + k * 256 + threadIdx.x;
    v[k] = y < V ? lr[y] : -INFINITY;
    mx = fmaxf(mx, v[k]);
  }
  mx = warp_max(mx);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = mx;
  __syncthreads();
  mx = red[0];
  for (int i = 1; i < 8; ++i) mx = fmaxf(mx, red[i]);
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kVChunk / 256; ++k)
    if (v[k] != -INFINITY) s += expf((v[k] - mx) * inv_t);
  s = warp_sum(s);
  if (l == 0) red[w] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int i = 0; i < 8; ++i) tot += red[i];
    RowStat st;
    st.m = mx;
    st.s = tot;
    stats[(size_t)row * nvc + c] = st;
  }
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

__device__ __forceinline__ double warp_incl_scan_d(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double u = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

__device__ __forceinline__ bool is_rejected(int y, const int* rej, int nrej) {
  for (int k = 0; k < nrej; ++k)
    if (rej[k] == y) return true;
  return false;
}

// One draw y from r = p with the rejected tokens removed: the smallest y with
// sum_{j<=y} r~(j) > target, r~ the unnormalised residual; if rounding leaves
// none, the last y with r~(y) > 0.  Chunk masses first, then one chunk in
// lane-contiguous segments of 128 entries.
__device__ int residual_draw(const float* lr, int V, float M, float inv_t, const RowStat* st, int nvc,
                             const int* rej, int nrej, double target) {
  const int lane = threadIdx.x & 31;
  double base = 0.0, before = 0.0;
  int chunk = -1, last_pos = -1;
  for (int c0 = 0; c0 < nvc; c0 += 32) {
    const int c = c0 + lane;
    double w = 0.0;
    if (c < nvc) {
      w = (double)st[c].s * (double)expf((st[c].m - M) * inv_t);
      for (int k = 0; k < nrej; ++k)
        if (rej[k] / kVChunk == c) w -= (double)expf((lr[rej[k]] - M) * inv_t);
      if (w < 0.0) w = 0.0;
    }
    const int lp = __reduce_max_sync(FULL, (c < nvc && w > 0.0) ? c : -1);
    if (lp > last_pos) last_pos = lp;
    const double incl = warp_incl_scan_d(w);
    const unsigned hm = __ballot_sync(FULL, c < nvc && w > 0.0 && base + incl > target);
    if (hm != 0u) {
      const int L = __ffs(hm) - 1;
      chunk = c0 + L;
      before = base + __shfl_sync(FULL, incl - w, L);
      break;
    }
    base += __shfl_sync(FULL, incl, 31);
  }
  double t2 = target - before;
  if (chunk < 0) {   // rounding: fall back to the last entry with mass
    chunk = last_pos < 0 ? 0 : last_pos;
    t2 = INFINITY;
  }
  const int y0 = chunk * kVChunk + lane * (kVChunk / 32);
  double mine = 0.0;
  int last_valid = -1;
  for (int k = 0; k < kVChunk / 32; ++k) {
    const int y = y0 + k;
    if (y < V && !is_rejected(y, rej, nrej)) {
      const float e = expf((lr[y] - M) * inv_t);
      mine += (double)e;
      if (e > 0.f) last_valid = y;
    }
  }
  const double incl = warp_incl_scan_d(mine);
  const unsigned hm = __ballot_sync(FULL, mine > 0.0 && incl > t2);
  if (hm == 0u) {
    const int lv = __reduce_max_sync(FULL, last_valid);
    return lv < 0 ? chunk * kVChunk : lv;
  }
  const int L = __ffs(hm) - 1;
  int y_found = -1;
  if (lane == L) {
    double cum = incl - mine;
    for (int k = 0; k < kVChunk / 32; ++k) {
      const int y = y0 + k;
      if (y < V && !is_rejected(y, rej, nrej)) {
        const float e = expf((lr[y] - M) * inv_t);
        cum += (double)e;
        last_valid = e > 0.f ? y : last_valid;
        if (cum > t2) {
          y_found = y;
          break;
        }
      }
    }
    if (y_found < 0) y_found = last_valid;
  }
  return __shfl_sync(FULL, y_found, L);
}

// residual walk, pass 2: one warp per request
__global__ void accept_residual_kernel(ReqTable t, const float* logits, int V, float inv_t, const float* uniforms,
                                       int bonus_at_leaf, const RowStat* stats, int nvc, int32_t* path,
                                       int32_t* accept_len, int32_t* out_tokens, int32_t* out_count,
                                       int32_t* status) {
  __shared__ int s_rej[32];
  const int r = blockIdx.x, lane = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (status_get(status) != 0) return;
  const int n = t.n[r], row0 = t.row_off[r];
  int par, tok;
  const int err = validate_tree_warp(t.parent[r], t.token[r], n, V, par, tok);
  if (err != TV_OK) {
    if (lane == 0) status_set(status, err);
    return;
  }
  // every random input of the request must be finite and in [0, 1)
  // [Algorithm and correctness contract, §Single-path sampling]
  const float uu = lane < n ? uniforms[row0 + lane] : 0.f;
  if (__any_sync(FULL, lane < n && !(uu >= 0.f && uu < 1.f))) {
    if (lane == 0) status_set(status, TV_E_UNIFORM);
    return;
  }
  int cur = 0, a = 0, nout = 0, draw = 0;
  if (lane == 0) path[row0] = 0;
  for (;;) {
    const float* lr = logits + (size_t)(row0 + cur) * V;
    const RowStat* st = stats + (size_t)(row0 + cur) * nvc;
    float M = -INFINITY;
    for (int c = lane; c < nvc; c += 32) M = fmaxf(M, st[c].m);
    M = warp_max(M);
    double Z = 0.0;
    for (int c = lane; c < nvc; c += 32) Z += (double)st[c].s * (double)expf((st[c].m - M) * inv_t);
    Z = warp_sum_d(Z);

    // candidates: the children of cur, in increasing node index
    unsigned kids = __ballot_sync(FULL, lane > 0 && lane < n && par == cur);
    double R = 0.0;   // removed (rejected) mass
    int nrej = 0, acc = -1;
    while (kids != 0u) {
      const int c = __ffs(kids) - 1;
      kids &= kids - 1u;
      const int x = __shfl_sync(FULL, tok, c);
      const float u = __shfl_sync(FULL, uu, draw);
      ++draw;
      const double ex = (double)expf((lr[x] - M) * inv_t);
      if ((double)u < ex / (Z - R)) {   // accept x with probability r(x)
        acc = c;
        break;
      }
      R += ex;   // remove x and renormalise
      if (lane == 0) s_rej[nrej] = x;
      ++nrej;
      __syncwarp();
    }
    if (acc >= 0) {
      const int ctok = __shfl_sync(FULL, tok, acc);
      ++a;
      if (lane == 0) {
        path[row0 + a] = acc;
        out_tokens[row0 + nout] = ctok;
      }
      ++nout;
      cur = acc;
      continue;
    }
    if (nrej > 0 || bonus_at_leaf) {
      const float u = __shfl_sync(FULL, uu, draw);
      ++draw;
      const int y = residual_draw(lr, V, M, inv_t, st, nvc, s_rej, nrej, (double)u * (Z - R));
      if (lane == 0) out_tokens[row0 + nout] = y;
      ++nout;
    }
    break;
  }
  if (lane == 0) {
    accept_len[r] = a;
    out_count[r] = nout;
  }
}

// ---------------------------------------------------------------------------
// single-draw form [Exactness, §Sampling, first paragraph; Drafters and tree
// verify, §Sampling]: every row draws its own token from p = softmax(l / T)
// with its own uniform, by the inverse CDF; the greedy walk over these draws is
// the single-draw walk.  One warp per row.
// ---------------------------------------------------------------------------
__global__ void draw_rows_kernel(ReqTable t, const float* logits, int V, float inv_t, const float* uniforms,
                                 const RowStat* stats, int nvc, int32_t* row_tokens, int32_t* status) {
  const int row = blockIdx.x, lane = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (status_get(status) != 0) return;
  const float u = uniforms[row];
  if (!(u >= 0.f && u < 1.f)) {   // [Algorithm and correctness contract, §Single-path sampling]
    if (lane == 0) status_set(status, TV_E_UNIFORM);
    return;
  }
  const float* lr = logits + (size_t)row * V;
  const RowStat* st = stats + (size_t)row * nvc;
  float M = -INFINITY;
  for (int c = lane; c < nvc; c += 32) M = fmaxf(M, st[c].m);
  M = warp_max(M);
  double Z = 0.0;
  for (int c = lane; c < nvc; c += 32) Z += (double)st[c].s * (double)expf((st[c].m - M) * inv_t);
  Z = warp_sum_d(Z);
  const int y = residual_draw(lr, V, M, inv_t, st, nvc, nullptr, 0, (double)u * Z);
  if (lane == 0) row_tokens[row] = y;
}

// ---------------------------------------------------------------------------
// single-path rejection sampler [Algorithm and correctness contract,
// §Single-path sampling]: node i of a chain carries draft x_i drawn from the
// proposal row q_i; the target row of x_i is its parent's, p = softmax(l / T).
// Pass 1, per (vocab chunk, row i >= 1): sum max(p - q_i, 0), sum q_i, and a
// flag for q entries that are not finite or negative.  grid (chunks, rows).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rej_stats_kernel(ReqTable t, const float* logits, int V, float inv_t,
                                                        const float* proposals, const RowStat* stats, int nvc,
                                                        RejStat* rstats, const int32_t* status) {
  __shared__ double rd[8], qd[8];
  __shared__ int bd[8];
  __shared__ float s_M;
  __shared__ double s_Z;
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int c = blockIdx.x, row = blockIdx.y;
  int r = 0;
  while (r + 1 < t.n_req && t.row_off[r + 1] <= row) ++r;
  if (row == t.row_off[r]) return;   // the root carries no draft
  const int prow = row - 1;           // a chain: the parent's row is the previous row
  const RowStat* st = stats + (size_t)prow * nvc;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float M = -INFINITY;
    for (int k = lane; k < nvc; k += 32) M = fmaxf(M, st[k].m);
    M = warp_max(M);
    double Z = 0.0;
    for (int k = lane; k < nvc; k += 32) Z += (double)st[k].s * (double)expf((st[k].m - M) * inv_t);
    Z = warp_sum_d(Z);
    if (lane == 0) {
      s_M = M;
      s_Z = Z;
    }
  }
  __syncthreads();
  const float M = s_M;
  const double iz = 1.0 / s_Z;
  const float* lp = logits + (size_t)prow * V;
  const float* qr = proposals + (size_t)row * V;
  double resid = 0.0, qs = 0.0;
  int bad = 0;
  for (int k = 0; k < kVChunk / 256; ++k) {
    const int y = c * kVChunk + k * 256 + threadIdx.x;
    if (y < V) {
      const float q = qr[y];
      if (!(q >= 0.f) || isinf(q)) bad = 1;
      const double p = (double)expf((lp[y] - M) * inv_t) * iz;
      resid += fmax(p - (double)q, 0.0);
      qs += (double)q;
    }
  }
  resid = warp_sum_d(resid);
  qs = warp_sum_d(qs);
  bad = __any_sync(FULL, bad);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    rd[w] = resid;
    qd[w] = qs;
    bd[w] = bad;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    RejStat o;
    o.resid = 0.0;
    o.qsum = 0.0;
    o.bad = 0;
    o.pad = 0;
    for (int i = 0; i < 8; ++i) {
      o.resid += rd[i];
      o.qsum += qd[i];
      o.bad |= bd[i];
    }
    rstats[(size_t)row * nvc + c] = o;
  }
}

// One draw from r = max(p - q, 0): the smallest y with sum_{j<=y} r(j) >
// target (target = u * sum r), chunk masses first, then one chunk; if rounding
// leaves none, the last y with r(y) > 0.
__device__ int rejection_draw(const float* lp, const float* qr, int V, float M, double iz, float inv_t,
                              const RejStat* rs, int nvc, double target) {
  const int lane = threadIdx.x & 31;
  double base = 0.0, before = 0.0;
  int chunk = -1, last_pos = -1;
  for (int c0 = 0; c0 < nvc; c0 += 32) {
    const int c = c0 + lane;
    const double w = c < nvc ? rs[c].resid : 0.0;
    const int lp2 = __reduce_max_sync(FULL, (c < nvc && w > 0.0) ? c : -1);
    if (lp2 > last_pos) last_pos = lp2;
    const double incl = warp_incl_scan_d(w);
    const unsigned hm = __ballot_sync(FULL, c < nvc && w > 0.0 && base + incl > target);
    if (hm != 0u) {
      const int L = __ffs(hm) - 1;
      chunk = c0 + L;
      before = base + __shfl_sync(FULL, incl - w, L);
      break;
    }
    base += __shfl_sync(FULL, incl, 31);
  }
  double t2 = target - before;
  if (chunk < 0) {
    chunk = last_pos < 0 ? 0 : last_pos;
    t2 = INFINITY;
  }
  auto mass = [&](int y) { return fmax((double)expf((lp[y] - M) * inv_t) * iz - (double)qr[y], 0.0); };
  const int y0 = chunk * kVChunk + lane * (kVChunk / 32);
  double mine = 0.0;
  int last_valid = -1;
  for (int k = 0; k < kVChunk / 32; ++k) {
    const int y = y0 + k;
    if (y < V) {
      const double m = mass(y);
      mine += m;
      if (m > 0.0) last_valid = y;
    }
  }
  const double incl = warp_incl_scan_d(mine);
  const unsigned hm = __ballot_sync(FULL, mine > 0.0 && incl > t2);
  if (hm == 0u) {
    const int lv = __reduce_max_sync(FULL, last_valid);
    return lv < 0 ? chunk * kVChunk : lv;
  }
  const int L = __ffs(hm) - 1;
  int y_found = -1;
  if (lane == L) {
    double cum = incl - mine;
    for (int k = 0; k < kVChunk / 32; ++k) {
      const int y = y0 + k;
      if (y < V) {
        const double m = mass(y);
        cum += m;
        if (m > 0.0) last_valid = y;
        if (cum > t2) {
          y_found = y;
          break;
        }
      }
    }
    if (y_found < 0) y_found = last_valid;
  }
  return __shfl_sync(FULL, y_found, L);
}

// Pass 2, one warp per request: validate, then test the drafts in order.
__global__ void accept_rejection_kernel(ReqTable t, const float* logits, int V, float inv_t, const float* proposals,
                                        const float* uniforms, const RowStat* stats, const RejStat* rstats, int nvc,
                                        int32_t* path, int32_t* accept_len, int32_t* out_tokens,
                                        int32_t* out_count, int32_t* status) {
  const int r = blockIdx.x, lane = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (status_get(status) != 0) return;
  const int n = t.n[r], row0 = t.row_off[r];
  int par, tok;
  const int err = validate_tree_warp(t.parent[r], t.token[r], n, V, par, tok);
  if (err != TV_OK) {
    if (lane == 0) status_set(status, err);
    return;
  }
  if (__any_sync(FULL, lane < n && par != lane - 1)) {   // the single-path sampler verifies a path
    if (lane == 0) status_set(status, TV_E_CHAIN);
    return;
  }
  const float uu = lane < n ? uniforms[row0 + lane] : 0.f;
  if (__any_sync(FULL, lane < n && !(uu >= 0.f && uu < 1.f))) {
    if (lane == 0) status_set(status, TV_E_UNIFORM);
    return;
  }
  // proposal rows of nodes 1..n-1: finite, nonnegative, unit mass (|sum - 1| <= 1e-3),
  // and q(x) > 0 at the draft, which was drawn from q
  bool bad = false;
  for (int i = 1; i < n; ++i) {
    const RejStat* rs = rstats + (size_t)(row0 + i) * nvc;
    double qs = 0.0;
    int fl = 0;
    for (int c = lane; c < nvc; c += 32) {
      qs += rs[c].qsum;
      fl |= rs[c].bad;
    }
    qs = warp_sum_d(qs);
    fl = __any_sync(FULL, fl);
    const int x = __shfl_sync(FULL, tok, i);
    const float qx = proposals[(size_t)(row0 + i) * V + x];
    if (fl || fabs(qs - 1.0) > 1e-3 || !(qx > 0.f)) bad = true;
  }
  if (bad) {
    if (lane == 0) status_set(status, TV_E_PROPOSAL);
    return;
  }
  int a = 0, nout = 0;
  if (lane == 0) path[row0] = 0;
  for (int i = 1; i < n; ++i) {
    const int prow = row0 + i - 1;
    const RowStat* st = stats + (size_t)prow * nvc;
    float M = -INFINITY;
    for (int c = lane; c < nvc; c += 32) M = fmaxf(M, st[c].m);
    M = warp_max(M);
    double Z = 0.0;
    for (int c = lane; c < nvc; c += 32) Z += (double)st[c].s * (double)expf((st[c].m - M) * inv_t);
    Z = warp_sum_d(Z);
    const float* lp = logits + (size_t)prow * V;
    const float* qr = proposals + (size_t)(row0 + i) * V;
    const int x = __shfl_sync(FULL, tok, i);
    const double px = (double)expf((lp[x] - M) * inv_t) / Z;
    const double qx = (double)qr[x];
    const float u = __shfl_sync(FULL, uu, i);
    if ((double)u < px / qx) {   // accept with probability min(1, p/q)
      ++a;
      if (lane == 0) {
        path[row0 + a] = i;
        out_tokens[row0 + nout] = x;
      }
      ++nout;
      continue;
    }
    // the first rejection: one draw from normalize(max(p - q, 0)), then stop
    const RejStat* rs = rstats + (size_t)(row0 + i) * nvc;
    double R = 0.0;
    for (int c = lane; c < nvc; c += 32) R += rs[c].resid;
    R = warp_sum_d(R);
    const float u0 = __shfl_sync(FULL, uu, 0);
    const int y = rejection_draw(lp, qr, V, M, 1.0 / Z, inv_t, rs, nvc, (double)u0 * R);
    if (lane == 0) out_tokens[row0 + nout] = y;
    ++nout;
    break;
  }
  if (lane == 0) {
    accept_len[r] = a;
    out_count[r] = nout;
  }
}

// ---------------------------------------------------------------------------
// commit: slot ctx + path[d] -> slot ctx + d, d = 0..a; every source row is
// read into shared memory before any is written.  grid (Hkv, K|V, requests).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) commit_kernel(ReqTable t, int D, const int32_t* path, const int32_t* accept_len,
                                                     int32_t* committed_src, int32_t* new_ctx, int32_t* status) {
  __shared__ uint4 rows[kMaxRows * 128 * 2 / 16];
  __shared__ int s_src[kMaxRows];
  __shared__ int s_a;
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int g = blockIdx.x, which = blockIdx.y, r = blockIdx.z;
  const int n = t.n[r], row0 = t.row_off[r], ctx = t.ctx[r];
  if (threadIdx.x == 0) s_a = accept_len[r];
  __syncthreads();
  const int a = s_a;
  bool bad = a < 0 || a >= n;
  if (!bad && (int)threadIdx.x <= a) {
    const int p = path[row0 + threadIdx.x];
    s_src[threadIdx.x] = p;
    if (p < 0 || p >= n || (threadIdx.x == 0 && p != 0)) bad = true;
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) status_set(status, TV_E_PATH);
    return;
  }
  __nv_bfloat16* base = (which ? t.v[r] : t.k[r]) + (size_t)g * t.capacity[r] * D;
  const int vec_per_row = D / 8;
  const int total = (a + 1) * vec_per_row;
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int d = i / vec_per_row, c = i - d * vec_per_row;
    rows[i] = *reinterpret_cast<const uint4*>(base + (size_t)(ctx + s_src[d]) * D + c * 8);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int d = i / vec_per_row, c = i - d * vec_per_row;
    *reinterpret_cast<uint4*>(base + (size_t)(ctx + d) * D + c * 8) = rows[i];
  }
  if (g == 0 && which == 0) {
    if ((int)threadIdx.x <= a) committed_src[row0 + threadIdx.x] = ctx + s_src[threadIdx.x];
    if (threadIdx.x == 0) new_ctx[r] = ctx + a + 1;
  }
}

}  // namespace

int launch_accept_greedy(const ReqTable& t, const int32_t* argmax, int32_t* path, int32_t* accept_len,
                         int32_t* out_tokens, int32_t* status, cudaStream_t st) {
  return launch_pdl(accept_greedy_kernel, dim3(t.n_req), dim3(32), 0, st, t, argmax, path, accept_len, out_tokens,
                    status);
}

int launch_accept_residual(const ReqTable& t, const float* logits, int vocab, float temperature,
                           const float* uniforms, int bonus_at_leaf, RowStat* stats, int32_t* path,
                           int32_t* accept_len, int32_t* out_tokens, int32_t* out_count, int32_t* status,
                           cudaStream_t st) {
  const int nvc = n_vchunks(vocab);
  const float inv_t = (float)(1.0 / (double)temperature);
  const int rc = launch_pdl(row_stats_kernel, dim3(nvc, t.total_rows), dim3(256), 0, st, logits, vocab, inv_t, nvc,
                            stats, (const int32_t*)status);
  if (rc) return rc;
  return launch_pdl(accept_residual_kernel, dim3(t.n_req), dim3(32), 0, st, t, logits, vocab, inv_t, uniforms,
                    bonus_at_leaf, (const RowStat*)stats, nvc, path, accept_len, out_tokens, out_count, status);
}

int launch_draw_rows(const ReqTable& t, const float* logits, int vocab, float temperature, const float* uniforms,
                     RowStat* stats, int32_t* row_tokens, int32_t* status, cudaStream_t st) {
  const int nvc = n_vchunks(vocab);
  const float inv_t = (float)(1.0 / (double)temperature);
  const int rc = launch_pdl(row_stats_kernel, dim3(nvc, t.total_rows), dim3(256), 0, st, logits, vocab, inv_t, nvc,
                            stats, (const int32_t*)status);
  if (rc) return rc;
  return launch_pdl(draw_rows_kernel, dim3(t.total_rows), dim3(32), 0, st, t, logits, vocab, inv_t, uniforms,
                    (const RowStat*)stats, nvc, row_tokens, status);
}

int launch_accept_rejection(const ReqTable& t, const float* logits, int vocab, float temperature,
                            const float* proposals, const float* uniforms, RowStat* stats, RejStat* rstats,
                            int32_t* path, int32_t* accept_len, int32_t* out_tokens, int32_t* out_count,
                            int32_t* status, cudaStream_t st) {
  const int nvc = n_vchunks(vocab);
  const float inv_t = (float)(1.0 / (double)temperature);
  int rc = launch_pdl(row_stats_kernel, dim3(nvc, t.total_rows), dim3(256), 0, st, logits, vocab, inv_t, nvc, stats,
                      (const int32_t*)status);
  if (rc) return rc;
  rc = launch_pdl(rej_stats_kernel, dim3(nvc, t.total_rows), dim3(256), 0, st, t, logits, vocab, inv_t, proposals,
                  (const RowStat*)stats, nvc, rstats, (const int32_t*)status);
  if (rc) return rc;
  return launch_pdl(accept_rejection_kernel, dim3(t.n_req), dim3(32), 0, st, t, logits, vocab, inv_t, proposals,
                    uniforms, (const RowStat*)stats, (const RejStat*)rstats, nvc, path, accept_len, out_tokens,
                    out_count, status);
}

int launch_commit(const ReqTable& t, const tv_dims& d, const int32_t* path, const int32_t* accept_len,
                  int32_t* committed_src, int32_t* new_ctx, int32_t* status, cudaStream_t st) {
  return launch_pdl(commit_kernel, dim3(d.n_kv_heads, 2, t.n_req), dim3(128), 0, st, t, d.head_dim, path, accept_len,
                    committed_src, new_ctx, status);
}

}  // namespace tv
