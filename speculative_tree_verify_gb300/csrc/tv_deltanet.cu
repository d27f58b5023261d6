// Gated DeltaNet tree verify and the path-state commit
// [Drafters and tree verify, §Tree verify through recurrent layers].
//
// Per value head the state S is a d_k x d_v matrix; one step of the gated
// delta rule is S <- exp(g) (I - beta k k^T) S + beta k v^T and the output is
// S^T q.  On a tree the state after node t is the state after t's parent,
// updated by t.  Unrolled from the state before the round, S0, along t's root
// path P(t) (nodes in order, gc the cumulative gate along the path):
//
//   S_t = exp(gc_t) S0 + sum_{s in P(t)} exp(gc_t - gc_s) k_s u_s^T
//   u_t = beta_t (v_t - exp(gc_t) S0^T k_t)
//         - sum_{s in P(t), s != t} beta_t exp(gc_t - gc_s) (k_t . k_s) u_s
//   o_t = exp(gc_t) S0^T q_t + sum_{s in P(t)} exp(gc_t - gc_s) (q_t . k_s) u_s
//
// The system for the pseudo-values u is lower triangular with ancestor-masked
// off-diagonal terms, so u_t depends on t's own path only, and the state after
// any accepted root path is the first line with t = its last node: the commit
// reads the state once and adds one small product per layer, reading no
// weights.  A chain cut back to its first n nodes is the path of length n.
//
//  - dn_verify_kernel: one CTA per (value head, block of 32 value columns,
//    request); every product in fp32 from shared memory, the triangular solve
//    by forward substitution in node order (parents come first).
//  - dn_commit_kernel: one CTA per (value head, layer, request); the whole
//    d_k x d_v state is read, updated in place and written (HBM-bound: the
//    state is the only large operand).
#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kDnCols = 32;        // value columns per verify CTA
constexpr int kDnThreads = 256;    // verify CTA
constexpr int kDnCommitThreads = 512;
constexpr int kNodeStride = kMaxRows + 1;   // K^T / Q^T row stride: stores along d_k hit distinct banks

// dynamic shared memory of the verify CTA, in floats
struct DnVerifyLayout {
  int kt, qt, s0, vb, ks, qs, u, kk, qk, a, total;
};
__host__ __device__ inline DnVerifyLayout dn_verify_layout(int dk) {
  DnVerifyLayout L;
  int o = 0;
  L.kt = o; o += dk * kNodeStride;       // K^T of the key head: [d_k][32 nodes + 1]
  L.qt = o; o += dk * kNodeStride;       // Q^T
  L.s0 = o; o += dk * kDnCols;           // S0[:, column block]
  L.vb = o; o += kMaxRows * kDnCols;     // v[:, column block]
  L.ks = o; o += kMaxRows * kDnCols;     // K S0 (then the right-hand side)
  L.qs = o; o += kMaxRows * kDnCols;     // Q S0
  L.u = o; o += kMaxRows * kDnCols;      // pseudo-values
  L.kk = o; o += kMaxRows * kMaxRows;    // k_t . k_s
  L.qk = o; o += kMaxRows * kMaxRows;    // q_t . k_s
  L.a = o; o += kMaxRows * kMaxRows;     // beta_t exp(gc_t - gc_s) (k_t . k_s), s a strict ancestor of t
  L.total = o;
  return L;
}

__global__ void __launch_bounds__(kDnThreads) dn_verify_kernel(ReqTable t, DnStates st, int Hk, int Hv, int dk, int dv,
                                                               const float* q, const float* k, const float* v,
                                                               const float* beta, const float* g, float* o, float* u,
                                                               float* gc_out, int32_t* status) {
  extern __shared__ __align__(16) float dsm[];
  __shared__ float s_gc[kMaxRows], s_beta[kMaxRows];
  __shared__ unsigned s_anc[kMaxRows];   // bit s: s is on t's root path (t included)
  __shared__ int s_err;
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int h = blockIdx.x, cb = blockIdx.y, r = blockIdx.z;
  const int n = t.n[r], row0 = t.row_off[r];
  const int kh = h / (Hv / Hk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const DnVerifyLayout L = dn_verify_layout(dk);
  float *KT = dsm + L.kt, *QT = dsm + L.qt, *S0 = dsm + L.s0, *VB = dsm + L.vb, *KS = dsm + L.ks, *QS = dsm + L.qs,
        *U = dsm + L.u, *KK = dsm + L.kk, *QK = dsm + L.qk, *A = dsm + L.a;

  if (warp == 0) {   // the tree: parent order; then cumulative gates and root paths
    int par, tok;
    const int err = validate_tree_warp(t.parent[r], t.token[r], n, 0, par, tok);
    if (lane == 0) s_err = err;
    if (err == TV_OK) {
      const float gl = lane < n ? g[(size_t)(row0 + lane) * Hv + h] : 0.f;
      if (lane < n) s_beta[lane] = beta[(size_t)(row0 + lane) * Hv + h];
      // pointer doubling over the parent links: gc = sum of g over the root path
      float acc = gl;
      unsigned anc = lane < n ? (1u << lane) : 0u;
      int up = lane < n ? par : -1;
#pragma unroll
      for (int step = 0; step < 5; ++step) {
        const int src = up < 0 ? lane : up;
        const float a2 = __shfl_sync(FULL, acc, src);
        const unsigned m2 = __shfl_sync(FULL, anc, src);
        const int u2 = __shfl_sync(FULL, up, src);
        if (up >= 0) {
          acc += a2;
          anc |= m2;
          up = u2;
        }
      }
      if (lane < n) {
        s_gc[lane] = acc;
        s_anc[lane] = anc;
      }
    }
  }
  __syncthreads();
  if (s_err != TV_OK) {
    if (threadIdx.x == 0 && h == 0 && cb == 0) status_set(status, s_err);
    return;
  }
  // stage K^T, Q^T (key head kh), v and S0 column blocks
  const int c0 = cb * kDnCols;
  for (int idx = threadIdx.x; idx < kMaxRows * dk; idx += kDnThreads) {
    const int s = idx / dk, i = idx - s * dk;   // node s, coordinate i (coalesced along i)
    float kv = 0.f, qv = 0.f;
    if (s < n) {
      const size_t off = ((size_t)(row0 + s) * Hk + kh) * dk + i;
      kv = k[off];
      qv = q[off];
    }
    KT[i * kNodeStride + s] = kv;
    QT[i * kNodeStride + s] = qv;
  }
  const float* S0g = st.S[r] + (size_t)h * dk * dv;
  for (int idx = threadIdx.x; idx < dk * kDnCols; idx += kDnThreads) {
    const int i = idx / kDnCols, j = idx - i * kDnCols;
    S0[idx] = S0g[(size_t)i * dv + c0 + j];
  }
  for (int idx = threadIdx.x; idx < kMaxRows * kDnCols; idx += kDnThreads) {
    const int s = idx / kDnCols, j = idx - s * kDnCols;
    VB[idx] = s < n ? v[((size_t)(row0 + s) * Hv + h) * dv + c0 + j] : 0.f;
  }
  __syncthreads();
  // K S0, Q S0, K K^T, Q K^T: thread (rows warp + 8m, column lane)
  {
    float ks[4] = {0.f, 0.f, 0.f, 0.f}, qs[4] = {0.f, 0.f, 0.f, 0.f};
    float kk[4] = {0.f, 0.f, 0.f, 0.f}, qk[4] = {0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < dk; ++i) {
      const float sij = S0[i * kDnCols + lane];
      const float kis = KT[i * kNodeStride + lane];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int tt = warp + 8 * m;
        const float kti = KT[i * kNodeStride + tt], qti = QT[i * kNodeStride + tt];
        ks[m] = fmaf(kti, sij, ks[m]);
        qs[m] = fmaf(qti, sij, qs[m]);
        kk[m] = fmaf(kti, kis, kk[m]);
        qk[m] = fmaf(qti, kis, qk[m]);
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int tt = warp + 8 * m;
      KS[tt * kDnCols + lane] = ks[m];
      QS[tt * kDnCols + lane] = qs[m];
      KK[tt * kMaxRows + lane] = kk[m];
      QK[tt * kMaxRows + lane] = qk[m];
    }
  }
  __syncthreads();
  // right-hand side beta_t (v_t - exp(gc_t) S0^T k_t) in place of K S0, and the
  // ancestor-masked coefficients
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int tt = warp + 8 * m;
    if (tt < n) {
      KS[tt * kDnCols + lane] = s_beta[tt] * (VB[tt * kDnCols + lane] - expf(s_gc[tt]) * KS[tt * kDnCols + lane]);
      const int s = lane;
      const bool strict_anc = s < tt && ((s_anc[tt] >> s) & 1u);
      A[tt * kMaxRows + s] = strict_anc ? s_beta[tt] * expf(s_gc[tt] - s_gc[s]) * KK[tt * kMaxRows + s] : 0.f;
    }
  }
  __syncthreads();
  // forward substitution, one column per lane: u_t = rhs_t - sum_s A[t][s] u_s
  if (warp == 0) {
    for (int tt = 0; tt < n; ++tt) {
      float acc = KS[tt * kDnCols + lane];
      unsigned m = s_anc[tt] & ~(1u << tt);
      while (m != 0u) {
        const int s = __ffs(m) - 1;
        m &= m - 1u;
        acc = fmaf(-A[tt * kMaxRows + s], U[s * kDnCols + lane], acc);
      }
      U[tt * kDnCols + lane] = acc;
    }
  }
  __syncthreads();
  // outputs o_t = exp(gc_t) S0^T q_t + sum over the path of exp(gc_t - gc_s) (q_t . k_s) u_s
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int tt = warp + 8 * m;
    if (tt < n) {
      float acc = expf(s_gc[tt]) * QS[tt * kDnCols + lane];
      unsigned msk = s_anc[tt];
      while (msk != 0u) {
        const int s = __ffs(msk) - 1;
        msk &= msk - 1u;
        acc = fmaf(expf(s_gc[tt] - s_gc[s]) * QK[tt * kMaxRows + s], U[s * kDnCols + lane], acc);
      }
      const size_t off = ((size_t)(row0 + tt) * Hv + h) * dv + c0 + lane;
      o[off] = acc;
      u[off] = U[tt * kDnCols + lane];
    }
  }
  if (cb == 0 && threadIdx.x < n) gc_out[(size_t)(row0 + threadIdx.x) * Hv + h] = s_gc[threadIdx.x];
}

// S <- exp(gc_last) S + sum_{d <= a} exp(gc_last - gc_{p_d}) k_{p_d} u_{p_d}^T
// for the accepted path p_0 = 0, ..., p_a of each request, in every layer.
// The path is checked first: a in [0, n), p_0 = 0, parent(p_d) = p_{d-1}.
__global__ void __launch_bounds__(kDnCommitThreads) dn_commit_kernel(ReqTable t, DnStates st, int Hk, int Hv, int dk,
                                                                     int dv, int rows_per_layer, const float* k,
                                                                     const float* u, const float* gc,
                                                                     const int32_t* path, const int32_t* accept_len,
                                                                     int32_t* status) {
  extern __shared__ __align__(16) float dsm[];
  float* KP = dsm;                          // [32 path nodes][d_k]
  float* UP = dsm + kMaxRows * dk;          // [32][d_v], scaled by exp(gc_last - gc_p)
  __shared__ int s_p[kMaxRows];
  __shared__ int s_a;
  __shared__ float s_decay;
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int h = blockIdx.x, layer = blockIdx.y, r = blockIdx.z;
  const int n = t.n[r], row0 = t.row_off[r];
  const int kh = h / (Hv / Hk);
  if (threadIdx.x == 0) s_a = accept_len[r];
  __syncthreads();
  const int a = s_a;
  bool bad = a < 0 || a >= n;
  if (!bad && (int)threadIdx.x <= a) {
    const int p = path[row0 + threadIdx.x];
    s_p[threadIdx.x] = p;
    if (p < 0 || p >= n) {
      bad = true;
    } else if (threadIdx.x == 0) {
      bad = p != 0;
    } else {
      const int pp = path[row0 + threadIdx.x - 1];
      bad = t.parent[r][p] != pp;
    }
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && h == 0 && layer == 0) status_set(status, TV_E_PATH);
    return;
  }
  const size_t lrow = (size_t)layer * rows_per_layer;
  const float gl = gc[(lrow + row0 + s_p[a]) * Hv + h];
  if (threadIdx.x == 0) s_decay = expf(gl);
  for (int idx = threadIdx.x; idx < (a + 1) * dk; idx += kDnCommitThreads) {
    const int d = idx / dk, i = idx - d * dk;
    KP[d * dk + i] = k[((lrow + row0 + s_p[d]) * Hk + kh) * dk + i];
  }
  for (int idx = threadIdx.x; idx < (a + 1) * dv; idx += kDnCommitThreads) {
    const int d = idx / dv, j = idx - d * dv;
    const size_t pr = lrow + row0 + s_p[d];
    UP[d * dv + j] = expf(gl - gc[pr * Hv + h]) * u[(pr * Hv + h) * dv + j];
  }
  __syncthreads();
  float* S = st.S[r] + ((size_t)layer * Hv + h) * dk * dv;
  const float decay = s_decay;
  // thread: 4 consecutive value columns, rows i = tid / (dv / 4) + stride m
  const int cols4 = dv / 4;
  const int rows_per_pass = kDnCommitThreads / cols4;
  const int j4 = (threadIdx.x % cols4) * 4;
  for (int i = threadIdx.x / cols4; i < dk; i += rows_per_pass) {
    float4 s = *reinterpret_cast<const float4*>(S + (size_t)i * dv + j4);
    s.x *= decay;
    s.y *= decay;
    s.z *= decay;
    s.w *= decay;
    for (int d = 0; d <= a; ++d) {
      const float kdi = KP[d * dk + i];
      const float4 ud = *reinterpret_cast<const float4*>(UP + d * dv + j4);
      s.x = fmaf(kdi, ud.x, s.x);
      s.y = fmaf(kdi, ud.y, s.y);
      s.z = fmaf(kdi, ud.z, s.z);
      s.w = fmaf(kdi, ud.w, s.w);
    }
    *reinterpret_cast<float4*>(S + (size_t)i * dv + j4) = s;
  }
}

bool g_dn_verify_smem[64] = {false};
bool g_dn_commit_smem[64] = {false};

}  // namespace

size_t dn_verify_smem(int dk) { return (size_t)dn_verify_layout(dk).total * sizeof(float); }
size_t dn_commit_smem(int dk, int dv) { return (size_t)kMaxRows * (dk + dv) * sizeof(float); }

int launch_dn_verify(const ReqTable& t, const DnStates& st, int Hk, int Hv, int dk, int dv, const float* q,
                     const float* k, const float* v, const float* beta, const float* g, float* o, float* u, float* gc,
                     int32_t* status, cudaStream_t s) {
  int rc = ensure_smem_limit(dn_verify_kernel, dn_verify_smem(kDnMaxDim), g_dn_verify_smem);
  if (rc) return rc;
  return launch_pdl(dn_verify_kernel, dim3(Hv, dv / kDnCols, t.n_req), dim3(kDnThreads), dn_verify_smem(dk), s, t,
                    st, Hk, Hv, dk, dv, q, k, v, beta, g, o, u, gc, status);
}

int launch_dn_commit(const ReqTable& t, const DnStates& st, int Hk, int Hv, int dk, int dv, int n_layers,
                     const float* k, const float* u, const float* gc, const int32_t* path, const int32_t* accept_len,
                     int32_t* status, cudaStream_t s) {
  int rc = ensure_smem_limit(dn_commit_kernel, dn_commit_smem(kDnMaxDim, kDnMaxDim), g_dn_commit_smem);
  if (rc) return rc;
  return launch_pdl(dn_commit_kernel, dim3(Hv, n_layers, t.n_req), dim3(kDnCommitThreads), dn_commit_smem(dk, dv), s,
                    t, st, Hk, Hv, dk, dv, t.total_rows, k, u, gc, path, accept_len, status);
}

}  // namespace tv
