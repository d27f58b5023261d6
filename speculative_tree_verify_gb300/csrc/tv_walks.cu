// Accept walks and the KV commit.
//
//  - greedy walk: one warp per request, lanes = tree nodes [Drafters and tree
//    verify, §The round, step 3];
//  - residual walk: a multi-CTA pass of per-chunk and per-segment softmax
//    statistics over the logits, then one warp per request walks the tree
//    [Algorithm and correctness contract, §Deterministic tree candidates and
//    residual verification];
//  - single-draw and single-path rejection walks on the same statistics;
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
  const int n = t.n[r], row0 = t.row_off[r];
  // every row's token, the status and the tree in one round trip (all reads
  // in bounds whatever an earlier kernel left); the walk shuffles
  const int am = lane < n ? argmax[row0 + lane] : 0;
  const bool prior = status_get(status) != 0;   // one load for the whole warp
  int par, tok;
  const int err = validate_tree_warp(t.parent[r], t.token[r], n, 0, par, tok);
  if (prior) return;
  if (err != TV_OK) {
    if (lane == 0) status_set(status, err);
    return;
  }
  int cur = 0, a = 0;
  if (lane == 0) path[row0] = 0;
  for (;;) {
    const int want = __shfl_sync(FULL, am, cur);
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
// greedy walk + commit in one launch.  grid (Hkv, K|V, requests), block 128:
// every block walks its request with one warp (a few hundred cycles: the
// tree and every row's token in one round trip), block (0, K) of the request
// writes the walk's outputs, and every block copies its (KV head, K|V) rows as
// commit_kernel does.  The path comes from the walk, so it is in range by
// construction.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) accept_greedy_commit_kernel(ReqTable t, int D, const int32_t* argmax,
                                                                   int32_t* path, int32_t* accept_len,
                                                                   int32_t* out_tokens, int32_t* committed_src,
                                                                   int32_t* new_ctx, int32_t* status) {
  __shared__ uint4 rows[kMaxRows * 128 * 2 / 16];
  __shared__ int s_src[kMaxRows], s_tok[kMaxRows];
  __shared__ int s_a;   // accepted count, -1: nothing to do
  pdl_wait();
  pdl_trigger();
  const int g = blockIdx.x, which = blockIdx.y, r = blockIdx.z;
  const int n = t.n[r], row0 = t.row_off[r], ctx = t.ctx[r];
  const bool lead = g == 0 && which == 0;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int am = lane < n ? argmax[row0 + lane] : 0;
    const bool prior = status_get(status) != 0;
    int par, tok;
    const int err = validate_tree_warp(t.parent[r], t.token[r], n, 0, par, tok);
    if (prior || err != TV_OK) {
      if (!prior && err != TV_OK && lead && lane == 0) status_set(status, err);
      if (lane == 0) s_a = -1;
    } else {
      int cur = 0, a = 0;
      if (lane == 0) s_src[0] = 0;
      for (;;) {
        const int want = __shfl_sync(FULL, am, cur);
        const unsigned hit = __ballot_sync(FULL, lane > 0 && lane < n && par == cur && tok == want);
        if (hit == 0u) {
          if (lane == 0) s_tok[a] = want;   // the model's token at the stopping node
          break;
        }
        const int c = __ffs(hit) - 1;
        const int ctok = __shfl_sync(FULL, tok, c);
        ++a;
        if (lane == 0) {
          s_src[a] = c;
          s_tok[a - 1] = ctok;
        }
        cur = c;
      }
      if (lane == 0) s_a = a;
    }
  }
  __syncthreads();
  const int a = s_a;
  if (a < 0) return;
  if (lead) {
    if ((int)threadIdx.x <= a) {
      path[row0 + threadIdx.x] = s_src[threadIdx.x];
      out_tokens[row0 + threadIdx.x] = s_tok[threadIdx.x];
      committed_src[row0 + threadIdx.x] = ctx + s_src[threadIdx.x];
    }
    if (threadIdx.x == 0) {
      accept_len[r] = a;
      new_ctx[r] = ctx + a + 1;
    }
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
}

// ---------------------------------------------------------------------------
// Pass 1 of every sampled walk: per (row, vocab chunk) the chunk max m and,
// per 128-token segment, sum exp((l - m) / T).  grid (chunks, rows), block
// 256: warp w reads the chunk's tokens 512w .. 512w + 511 (its segments
// 4w .. 4w + 3) in coalesced 128-byte rows.  fp32 throughout: the GPU's FP64
// rate is a small fraction of its FP32 rate, so FP64 appears below only where
// a handful of per-chunk values are combined.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float softmax_term(float l, float m, float inv_t) { return expf((l - m) * inv_t); }

// exp((m_c - M) / T): chunk units -> row units (0 for a chunk with no finite logit)
__device__ __forceinline__ float chunk_scale(float mc, float M, float inv_t) {
  return mc == -INFINITY ? 0.f : softmax_term(mc, M, inv_t);
}

__global__ void __launch_bounds__(256) row_stats_kernel(const float* logits, int V, float inv_t, int nvc,
                                                        RowStat* stats, const int32_t* status) {
  __shared__ float red[8];
  __shared__ float s_seg[kSegsPerChunk];
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int c = blockIdx.x, row = blockIdx.y;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* lr = logits + (size_t)row * V;
  const int yw = c * kVChunk + w * (4 * kVSeg);
  float v[16];
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int y = yw + j * 32 + lane;
    v[j] = y < V ? lr[y] : -INFINITY;
    mx = fmaxf(mx, v[j]);
  }
  mx = warp_max(mx);
  if (lane == 0) red[w] = mx;
  __syncthreads();
  mx = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) mx = fmaxf(mx, red[i]);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (mx != -INFINITY) {
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j >> 2] += softmax_term(v[j], mx, inv_t);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float sq = warp_sum(acc[q]);
    if (lane == 0) s_seg[w * 4 + q] = sq;
  }
  __syncthreads();
  if (w == 0) {
    const float sg = s_seg[lane];
    const float tot = warp_sum(sg);
    RowStat* o = stats + (size_t)row * nvc + c;
    o->seg[lane] = sg;
    if (lane == 0) {
      o->m = mx;
      o->s = tot;
    }
  }
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

template <typename T>
__device__ __forceinline__ T warp_incl_scan(T v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T u = __shfl_up_sync(FULL, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// The row max M and Z = sum over the row of exp((l - M) / T), from the row's
// chunk statistics.  One warp (lanes stride over the chunks, then a butterfly
// sum), explicit roundings: every kernel that needs a row's M and Z calls this
// with a whole warp and gets the same bits.
__device__ __forceinline__ void row_mz(const RowStat* st, int nvc, float inv_t, float& M, double& Z) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  for (int c = lane; c < nvc; c += 32) m = fmaxf(m, st[c].m);
  m = warp_max(m);
  double z = 0.0;
  for (int c = lane; c < nvc; c += 32) z = __dadd_rn(z, __dmul_rn((double)st[c].s, (double)chunk_scale(st[c].m, m, inv_t)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z = __dadd_rn(z, __shfl_xor_sync(FULL, z, o));
  M = m;
  Z = z;
}

// p = softmax(l / T) over a row with the tokens rej[0 .. nrej) removed
struct SoftmaxRow {
  const float* lr;
  const RowStat* st;
  const int* rej;
  int nrej, V;
  float M, inv_t;
  __device__ float scale(int c) const { return chunk_scale(st[c].m, M, inv_t); }
  __device__ double chunk_mass(int c) const {   // row units
    double w = (double)st[c].s * (double)scale(c);
    for (int k = 0; k < nrej; ++k)
      if (rej[k] / kVChunk == c) w -= (double)softmax_term(lr[rej[k]], M, inv_t);
    return w > 0.0 ? w : 0.0;
  }
  __device__ float seg_mass(int c, int s) const {   // chunk units
    float w = st[c].seg[s];
    const int g = c * kSegsPerChunk + s;
    for (int k = 0; k < nrej; ++k)
      if (rej[k] / kVSeg == g) w -= softmax_term(lr[rej[k]], st[c].m, inv_t);
    return fmaxf(w, 0.f);
  }
  __device__ float tok_mass(int c, int y) const {   // chunk units
    if (y >= V) return 0.f;
    for (int k = 0; k < nrej; ++k)
      if (rej[k] == y) return 0.f;
    const float m = st[c].m;
    return m == -INFINITY ? 0.f : softmax_term(lr[y], m, inv_t);
  }
};

// r = max(p - q, 0) of a draft: p = softmax(l / T) of its parent's row, q its
// proposal row; izf = 1 / Z of the parent's row, rounded to fp32 once
__device__ __forceinline__ float resid_term(float l, float q, float M, float inv_t, float izf) {
  return fmaxf(__fmaf_rn(softmax_term(l, M, inv_t), izf, -q), 0.f);
}

struct ResidRow {
  const float* lp;
  const float* qr;
  const RejStat* rs;
  int V;
  float M, inv_t, izf;
  __device__ float scale(int) const { return 1.f; }
  __device__ double chunk_mass(int c) const { return (double)rs[c].resid; }
  __device__ float seg_mass(int c, int s) const { return rs[c].seg[s]; }
  __device__ float tok_mass(int, int y) const { return y < V ? resid_term(lp[y], qr[y], M, inv_t, izf) : 0.f; }
};

// One draw by the inverse CDF: the smallest y whose cumulative mass exceeds
// target.  Searched chunk -> segment -> token, each step one warp-wide scan;
// where rounding leaves the target at or past a step's total, the last token
// with mass is taken.  Row supplies chunk_mass(c) in row units, scale(c) (row
// units per chunk unit), seg_mass(c, s) and tok_mass(c, y) in chunk units.
template <class Row>
__device__ int cdf_draw(const Row& R, int nvc, double target) {
  const int lane = threadIdx.x & 31;
  bool tail = false;
  double base = 0.0, before = 0.0;
  int chunk = -1, last_c = -1;
  for (int c0 = 0; c0 < nvc; c0 += 32) {
    const int c = c0 + lane;
    const double w = c < nvc ? R.chunk_mass(c) : 0.0;
    last_c = max(last_c, __reduce_max_sync(FULL, w > 0.0 ? c : -1));
    const double incl = warp_incl_scan(w);
    const unsigned hm = __ballot_sync(FULL, w > 0.0 && base + incl > target);
    if (hm != 0u) {
      const int L = __ffs(hm) - 1;
      chunk = c0 + L;
      before = base + __shfl_sync(FULL, incl - w, L);
      break;
    }
    base += __shfl_sync(FULL, incl, 31);
  }
  if (chunk < 0) {
    if (last_c < 0) return 0;   // no mass anywhere
    chunk = last_c;
    tail = true;
  }
  const double t2 = tail ? 0.0 : (target - before) / (double)R.scale(chunk);
  const float ws = R.seg_mass(chunk, lane);
  const double incl2 = warp_incl_scan((double)ws);
  const unsigned hm2 = __ballot_sync(FULL, !tail && ws > 0.f && incl2 > t2);
  int seg;
  double before2 = 0.0;
  if (hm2 != 0u) {
    seg = __ffs(hm2) - 1;
    before2 = __shfl_sync(FULL, incl2 - (double)ws, seg);
  } else {
    seg = __reduce_max_sync(FULL, ws > 0.f ? lane : -1);
    if (seg < 0) seg = kSegsPerChunk - 1;
    tail = true;
  }
  const float t3 = (float)(t2 - before2);
  for (int sg = seg; sg >= 0; --sg) {   // past `seg` only when rounding left a segment without mass
    const int yb = chunk * kVChunk + sg * kVSeg + lane * 4;
    float e[4], mine = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      e[j] = R.tok_mass(chunk, yb + j);
      mine += e[j];
    }
    if (!tail) {
      const float incl3 = warp_incl_scan(mine);
      const unsigned hm3 = __ballot_sync(FULL, mine > 0.f && incl3 > t3);
      if (hm3 != 0u) {
        const int L = __ffs(hm3) - 1;
        int yf = -1;
        if (lane == L) {
          float cum = incl3 - mine;
          int lastv = -1;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            cum += e[j];
            if (e[j] > 0.f) {
              lastv = yb + j;
              if (cum > t3 && yf < 0) yf = yb + j;
            }
          }
          if (yf < 0) yf = lastv;
        }
        return __shfl_sync(FULL, yf, L);
      }
    }
    int lv = -1;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (e[j] > 0.f) lv = yb + j;
    lv = __reduce_max_sync(FULL, lv);
    if (lv >= 0) return lv;
    tail = true;
  }
  return chunk * kVChunk;   // the chunk's statistics said mass, its tokens said none
}

// residual walk, pass 2: one CTA of 32 warps per request; warp w forms row w's
// M and Z, then warp 0 walks
__global__ void __launch_bounds__(1024) accept_residual_kernel(ReqTable t, const float* logits, int V, float inv_t,
                                                               const float* uniforms, int bonus_at_leaf,
                                                               const RowStat* stats, int nvc, int32_t* path,
                                                               int32_t* accept_len, int32_t* out_tokens,
                                                               int32_t* out_count, int32_t* status) {
  __shared__ int s_rej[32];
  __shared__ float s_M[32];
  __shared__ double s_Z[32];
  const int r = blockIdx.x, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  pdl_wait();
  pdl_trigger();
  if (status_get(status) != 0) return;
  const int n = t.n[r], row0 = t.row_off[r];
  if (wid < n) row_mz(stats + (size_t)(row0 + wid) * nvc, nvc, inv_t, s_M[wid], s_Z[wid]);
  __syncthreads();
  if (wid != 0) return;
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
    const float M = s_M[cur];
    const double Z = s_Z[cur];

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
      const double ex = (double)softmax_term(lr[x], M, inv_t);
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
      const SoftmaxRow row{lr, st, s_rej, nrej, V, M, inv_t};
      const int y = cdf_draw(row, nvc, (double)u * (Z - R));
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
  const RowStat* st = stats + (size_t)row * nvc;
  float M;
  double Z;
  row_mz(st, nvc, inv_t, M, Z);
  const SoftmaxRow R{logits + (size_t)row * V, st, nullptr, 0, V, M, inv_t};
  const int y = cdf_draw(R, nvc, (double)u * Z);
  if (lane == 0) row_tokens[row] = y;
}

// ---------------------------------------------------------------------------
// single-path rejection sampler [Algorithm and correctness contract,
// §Single-path sampling]: node i of a chain carries draft x_i drawn from the
// proposal row q_i; the target row of x_i is its parent's, p = softmax(l / T).
// Pass 2, per (vocab chunk, row i >= 1): per segment sum max(p - q_i, 0), sum
// q_i, and a flag for q entries that are not finite or negative.  grid
// (chunks, rows), block 256, the token layout of pass 1.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) rej_stats_kernel(ReqTable t, const float* logits, int V, float inv_t,
                                                        const float* proposals, const RowStat* stats, int nvc,
                                                        RejStat* rstats, const int32_t* status) {
  __shared__ float s_seg[kSegsPerChunk];
  __shared__ float s_q[8];
  __shared__ int s_bad[8];
  __shared__ float s_M, s_izf;
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int c = blockIdx.x, row = blockIdx.y;
  int r = 0;
  while (r + 1 < t.n_req && t.row_off[r + 1] <= row) ++r;
  if (row == t.row_off[r]) return;   // the root carries no draft
  const int prow = row - 1;           // a chain: the parent's row is the previous row
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* lp = logits + (size_t)prow * V;
  const float* qr = proposals + (size_t)row * V;
  const int yw = c * kVChunk + w * (4 * kVSeg);
  float lv[16], qv[16];   // loads in flight while warp 0 forms the row statistics
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int y = yw + j * 32 + lane;
    lv[j] = y < V ? lp[y] : -INFINITY;
    qv[j] = y < V ? qr[y] : 0.f;
  }
  if (w == 0) {
    float M;
    double Z;
    row_mz(stats + (size_t)prow * nvc, nvc, inv_t, M, Z);
    if (lane == 0) {
      s_M = M;
      s_izf = (float)(1.0 / Z);
    }
  }
  __syncthreads();
  const float M = s_M, izf = s_izf;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  float qs = 0.f;
  int bad = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float q = qv[j];
    if (!(q >= 0.f) || isinf(q)) bad = 1;
    acc[j >> 2] += resid_term(lv[j], q, M, inv_t, izf);
    qs += q;
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float sq = warp_sum(acc[q]);
    if (lane == 0) s_seg[w * 4 + q] = sq;
  }
  qs = warp_sum(qs);
  bad = __any_sync(FULL, bad);
  if (lane == 0) {
    s_q[w] = qs;
    s_bad[w] = bad;
  }
  __syncthreads();
  if (w == 0) {
    const float sg = s_seg[lane];
    const float tot = warp_sum(sg);
    const float qt = warp_sum(lane < 8 ? s_q[lane] : 0.f);
    const int bd = __any_sync(FULL, lane < 8 && s_bad[lane] != 0);
    RejStat* o = rstats + (size_t)row * nvc + c;
    o->seg[lane] = sg;
    if (lane == 0) {
      o->resid = tot;
      o->qsum = qt;
      o->bad = bd;
      o->pad = 0;
    }
  }
}

// Pass 3, one CTA of 32 warps per request: warp w forms row w's M and Z and
// checks node w's proposal row; warp 0 validates, then tests the drafts in order.
__global__ void __launch_bounds__(1024) accept_rejection_kernel(ReqTable t, const float* logits, int V, float inv_t,
                                                                const float* proposals, const float* uniforms,
                                                                const RowStat* stats, const RejStat* rstats, int nvc,
                                                                int32_t* path, int32_t* accept_len,
                                                                int32_t* out_tokens, int32_t* out_count,
                                                                int32_t* status) {
  __shared__ float s_M[32];
  __shared__ double s_Z[32];
  __shared__ int s_bad[32];
  const int r = blockIdx.x, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  pdl_wait();
  pdl_trigger();
  if (status_get(status) != 0) return;
  const int n = t.n[r], row0 = t.row_off[r];
  // proposal row of node w >= 1: finite, nonnegative, unit mass (|sum - 1| <=
  // 1e-3), and q(x) > 0 at the draft, which was drawn from q
  if (wid < n) {
    row_mz(stats + (size_t)(row0 + wid) * nvc, nvc, inv_t, s_M[wid], s_Z[wid]);
    int bad = 0;
    if (wid >= 1) {
      const RejStat* rs = rstats + (size_t)(row0 + wid) * nvc;
      double qs = 0.0;
      int fl = 0;
      for (int c = lane; c < nvc; c += 32) {
        qs += (double)rs[c].qsum;
        fl |= rs[c].bad;
      }
      qs = warp_sum_d(qs);
      fl = __any_sync(FULL, fl);
      int x = t.token[r][wid];
      x = x < 0 ? 0 : (x >= V ? V - 1 : x);   // a token out of range is reported by the tree check
      const float qx = proposals[(size_t)(row0 + wid) * V + x];
      bad = (fl || fabs(qs - 1.0) > 1e-3 || !(qx > 0.f)) ? 1 : 0;
    }
    if (lane == 0) s_bad[wid] = bad;
  }
  __syncthreads();
  if (wid != 0) return;
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
  if (__any_sync(FULL, lane < n && s_bad[lane] != 0)) {
    if (lane == 0) status_set(status, TV_E_PROPOSAL);
    return;
  }
  int a = 0, nout = 0;
  if (lane == 0) path[row0] = 0;
  for (int i = 1; i < n; ++i) {
    const int prow = row0 + i - 1;
    const float M = s_M[i - 1];
    const double Z = s_Z[i - 1];
    const float* lp = logits + (size_t)prow * V;
    const float* qr = proposals + (size_t)(row0 + i) * V;
    const int x = __shfl_sync(FULL, tok, i);
    const double px = (double)softmax_term(lp[x], M, inv_t) / Z;
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
    double Rm = 0.0;
    for (int c = lane; c < nvc; c += 32) Rm += (double)rs[c].resid;
    Rm = warp_sum_d(Rm);
    const float u0 = __shfl_sync(FULL, uu, 0);
    const ResidRow row{lp, qr, rs, V, M, inv_t, (float)(1.0 / Z)};
    const int y = cdf_draw(row, nvc, (double)u0 * Rm);
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
  pdl_wait();
  pdl_trigger();
  const int g = blockIdx.x, which = blockIdx.y, r = blockIdx.z;
  const int n = t.n[r], row0 = t.row_off[r], ctx = t.ctx[r];
  // the accepted length, the path entries and the status in one round trip
  // (every read in bounds whatever an earlier kernel left)
  const int a = accept_len[r];
  const int p = (int)threadIdx.x < n ? path[row0 + threadIdx.x] : 0;
  const int prior = threadIdx.x == 0 ? status_get(status) : 0;
  bool bad = a < 0 || a >= n;
  if (!bad && (int)threadIdx.x <= a) {
    s_src[threadIdx.x] = p;
    if (p < 0 || p >= n || (threadIdx.x == 0 && p != 0)) bad = true;
  }
  if (__syncthreads_or(prior != 0)) return;   // an earlier error: nothing is written
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
  return launch_pdl(accept_residual_kernel, dim3(t.n_req), dim3(1024), 0, st, t, logits, vocab, inv_t, uniforms,
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
  return launch_pdl(accept_rejection_kernel, dim3(t.n_req), dim3(1024), 0, st, t, logits, vocab, inv_t, proposals,
                    uniforms, (const RowStat*)stats, (const RejStat*)rstats, nvc, path, accept_len, out_tokens,
                    out_count, status);
}

int launch_accept_greedy_commit(const ReqTable& t, const tv_dims& d, const int32_t* argmax, int32_t* path,
                                int32_t* accept_len, int32_t* out_tokens, int32_t* committed_src, int32_t* new_ctx,
                                int32_t* status, cudaStream_t st) {
  return launch_pdl(accept_greedy_commit_kernel, dim3(d.n_kv_heads, 2, t.n_req), dim3(128), 0, st, t, d.head_dim,
                    argmax, path, accept_len, out_tokens, committed_src, new_ctx, status);
}

int launch_commit(const ReqTable& t, const tv_dims& d, const int32_t* path, const int32_t* accept_len,
                  int32_t* committed_src, int32_t* new_ctx, int32_t* status, cudaStream_t st) {
  return launch_pdl(commit_kernel, dim3(d.n_kv_heads, 2, t.n_req), dim3(128), 0, st, t, d.head_dim, path, accept_len,
                    committed_src, new_ctx, status);
}

}  // namespace tv
