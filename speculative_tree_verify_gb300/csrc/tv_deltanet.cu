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
//  - dn_commit_kernel: persistent, one CTA per SM over the (request, layer,
//    value head) tiles, two in flight: each d_k x d_v state tile comes in by
//    one TMA bulk copy, is updated and written back in place (HBM-bound: the
//    state is the only large operand).
#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kDnCols = 32;        // value columns per verify CTA
constexpr int kDnThreads = 512;    // verify CTA
constexpr int kDnWarps = kDnThreads / 32;
constexpr int kDnCommitThreads = 512;
constexpr int kNodeStride = kMaxRows + 4;   // K^T / Q^T row stride: 16-byte aligned rows

// dynamic shared memory of the verify CTA, in floats
struct DnVerifyLayout {
  int kt, qt, s0, vb, ks, qs, u, kk, c, a, part, total;
};
__host__ __device__ inline DnVerifyLayout dn_verify_layout(int dk) {
  DnVerifyLayout L;
  int o = 0;
  L.kt = o; o += dk * kNodeStride;       // K^T of the key head: [d_k][32 nodes + 4]
  L.qt = o; o += dk * kNodeStride;       // Q^T
  L.s0 = o; o += dk * kDnCols;           // S0[:, column block]
  L.vb = o; o += kMaxRows * kDnCols;     // v[:, column block]
  L.ks = o; o += kMaxRows * kDnCols;     // K S0, then the right-hand side
  L.qs = o; o += kMaxRows * kDnCols;     // Q S0
  L.u = o; o += kMaxRows * kDnCols;      // pseudo-values (first: partial products)
  L.kk = o; o += kMaxRows * kMaxRows;    // k_t . k_s
  L.c = o; o += kMaxRows * kMaxRows;     // q_t . k_s, then exp(gc_t - gc_s) (q_t . k_s) on t's path
  L.a = o; o += kMaxRows * kMaxRows;     // beta_t exp(gc_t - gc_s) (k_t . k_s), s a strict ancestor
  L.part = o; o += 7 * 4 * 8 * 32;       // partial products of the d_k parts past the first
  L.total = o;
  return L;
}

__global__ void __launch_bounds__(kDnThreads) dn_verify_kernel(ReqTable t, DnStates st, int Hk, int Hv, int dk, int dv,
                                                               const float* q, const float* k, const float* v,
                                                               const float* beta, const float* g, float* o, float* u,
                                                               float* gc_out, int32_t* status, int state_early) {
  extern __shared__ __align__(16) float dsm[];
  __shared__ float s_gc[kMaxRows], s_beta[kMaxRows];
  __shared__ unsigned s_anc[kMaxRows];   // bit s: s is on t's root path (t included)
  __shared__ int s_err, s_stat;
  const int h = blockIdx.x, cb = blockIdx.y, r = blockIdx.z;
  // the state before the round: with state_early, loaded before the wait (the
  // caller guarantees that every writer of it has completed by then)
  const int c0 = cb * kDnCols;
  constexpr int kSB = kDnMaxDim * kDnCols / 4 / kDnThreads;    // float4 of S0 a thread
  float4 sreg[kSB];
  const float* S0g = st.S[r] + (size_t)h * dk * dv;
  auto load_state = [&]() {
#pragma unroll
    for (int m = 0; m < kSB; ++m) {
      const int idx = threadIdx.x + m * kDnThreads;
      const int i = idx / (kDnCols / 4), c = idx - i * (kDnCols / 4);
      sreg[m] = idx < dk * kDnCols / 4 ? *reinterpret_cast<const float4*>(S0g + (size_t)i * dv + c0 + 4 * c)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  if (state_early) load_state();
  pdl_wait();
  pdl_trigger();
  // every load below is in bounds whatever an earlier kernel left; the status
  // (an earlier error) is read with them and checked before anything is written
  if (threadIdx.x == 0) s_stat = status_get(status);
  const int n = t.n[r], row0 = t.row_off[r];
  const int kh = h / (Hv / Hk);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const DnVerifyLayout L = dn_verify_layout(dk);
  float *KT = dsm + L.kt, *QT = dsm + L.qt, *S0 = dsm + L.s0, *VB = dsm + L.vb, *KS = dsm + L.ks, *QS = dsm + L.qs,
        *U = dsm + L.u, *KK = dsm + L.kk, *C = dsm + L.c, *A = dsm + L.a;

  // the loads on the critical path first (warp 0: the tree and the node gates),
  // then every other load of the CTA, into registers
  int par = 0, tok = 0;
  float gl = 0.f, bl = 0.f;
  if (warp == 0 && lane < n) {
    par = t.parent[r][lane];
    tok = t.token[r][lane];
    gl = g[(size_t)(row0 + lane) * Hv + h];
    bl = beta[(size_t)(row0 + lane) * Hv + h];
  }
  constexpr int kKQ = kMaxRows * kDnMaxDim / 4 / kDnThreads;   // float4 of K and of Q a thread
  float4 kreg[kKQ], qreg[kKQ], vreg = make_float4(0.f, 0.f, 0.f, 0.f);
  const int k4 = dk / 4;
#pragma unroll
  for (int m = 0; m < kKQ; ++m) {
    const int idx = threadIdx.x + m * kDnThreads;
    // node s = the lane: the transposing stores below then hit 32 banks
    const int s = idx % kMaxRows, c = idx / kMaxRows;   // coordinates 4c .. 4c + 3
    kreg[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    qreg[m] = kreg[m];
    if (idx < kMaxRows * k4 && s < n) {
      const size_t off = ((size_t)(row0 + s) * Hk + kh) * dk + 4 * c;
      kreg[m] = *reinterpret_cast<const float4*>(k + off);
      qreg[m] = *reinterpret_cast<const float4*>(q + off);
    }
  }
  if (!state_early) load_state();
  if (threadIdx.x < kMaxRows * kDnCols / 4) {   // 256 = 32 nodes x 8 float4
    const int s = threadIdx.x / (kDnCols / 4), c = threadIdx.x - s * (kDnCols / 4);
    if (s < n) vreg = *reinterpret_cast<const float4*>(v + ((size_t)(row0 + s) * Hv + h) * dv + c0 + 4 * c);
  }

  if (warp == 0) {   // the tree: parent order; then cumulative gates and root paths
    const int err = check_tree_warp(par, tok, n, 0);
    if (lane == 0) s_err = err;
    if (err == TV_OK) {
      if (lane < n) s_beta[lane] = bl;
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
  // stage K^T, Q^T, S0 and v in shared memory
#pragma unroll
  for (int m = 0; m < kKQ; ++m) {
    const int idx = threadIdx.x + m * kDnThreads;
    if (idx < kMaxRows * k4) {
      const int s = idx % kMaxRows, c = idx / kMaxRows;
      const float kv[4] = {kreg[m].x, kreg[m].y, kreg[m].z, kreg[m].w};
      const float qv[4] = {qreg[m].x, qreg[m].y, qreg[m].z, qreg[m].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        KT[(4 * c + e) * kNodeStride + s] = kv[e];
        QT[(4 * c + e) * kNodeStride + s] = qv[e];
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kSB; ++m) {
    const int idx = threadIdx.x + m * kDnThreads;
    if (idx < dk * kDnCols / 4) reinterpret_cast<float4*>(S0)[idx] = sreg[m];
  }
  if (threadIdx.x < kMaxRows * kDnCols / 4) reinterpret_cast<float4*>(VB)[threadIdx.x] = vreg;
  __syncthreads();
  if (s_stat != 0) return;
  if (s_err != TV_OK) {
    if (threadIdx.x == 0 && h == 0 && cb == 0) status_set(status, s_err);
    return;
  }

  // K S0, Q S0, K K^T, Q K^T.  A warp takes 4 contiguous rows (one float4 of
  // K^T and of Q^T per coordinate) and the column lane; the row groups share
  // the 16 warps by cutting d_k into `split` parts, whose sums the first
  // part's warps add in part order.
  {
    float* PART = dsm + L.part;
    const int ng = (n + 3) / 4;                                // row groups of 4
    const int split = ng <= 2 ? 8 : (ng <= 4 ? 4 : 2);         // ng * split <= 16
    const int rg = warp % ng, part = warp / ng;
    const bool live = part < split;
    const int span = dk / split, i_lo = part * span, i_hi = i_lo + span;
    float ks[4] = {0.f, 0.f, 0.f, 0.f}, qs[4] = {0.f, 0.f, 0.f, 0.f};
    float kk[4] = {0.f, 0.f, 0.f, 0.f}, qk[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) {
      // rows in pairs through the paired fp32 FMA (each half a correctly
      // rounded fmaf, so the sums are those of scalar fmaf)
      float2 ks2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)}, qs2[2] = {ks2[0], ks2[1]};
      float2 kk2[2] = {ks2[0], ks2[1]}, qk2[2] = {ks2[0], ks2[1]};
#pragma unroll 4
      for (int i = i_lo; i < i_hi; ++i) {
        const float sij = S0[i * kDnCols + lane];
        const float kis = KT[i * kNodeStride + lane];
        const float4 kt4 = *reinterpret_cast<const float4*>(KT + i * kNodeStride + 4 * rg);
        const float4 qt4 = *reinterpret_cast<const float4*>(QT + i * kNodeStride + 4 * rg);
        const float2 kt2[2] = {make_float2(kt4.x, kt4.y), make_float2(kt4.z, kt4.w)};
        const float2 qt2[2] = {make_float2(qt4.x, qt4.y), make_float2(qt4.z, qt4.w)};
        const float2 s2 = make_float2(sij, sij), k2 = make_float2(kis, kis);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          ks2[m] = __ffma2_rn(kt2[m], s2, ks2[m]);
          qs2[m] = __ffma2_rn(qt2[m], s2, qs2[m]);
          kk2[m] = __ffma2_rn(kt2[m], k2, kk2[m]);
          qk2[m] = __ffma2_rn(qt2[m], k2, qk2[m]);
        }
      }
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        ks[2 * m] = ks2[m].x; ks[2 * m + 1] = ks2[m].y;
        qs[2 * m] = qs2[m].x; qs[2 * m + 1] = qs2[m].y;
        kk[2 * m] = kk2[m].x; kk[2 * m + 1] = kk2[m].y;
        qk[2 * m] = qk2[m].x; qk[2 * m + 1] = qk2[m].y;
      }
    }
    // PART[((part - 1) 4 + product) (4 ng 32) + row 32 + lane]
    const int pstride = 4 * ng * 32;
    if (live && part > 0) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int tt = 4 * rg + m;
        float* base = PART + (size_t)(part - 1) * 4 * pstride + tt * 32 + lane;
        base[0 * pstride] = ks[m];
        base[1 * pstride] = qs[m];
        base[2 * pstride] = kk[m];
        base[3 * pstride] = qk[m];
      }
    }
    __syncthreads();
    if (live && part == 0) {
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int tt = 4 * rg + m;
        for (int pp = 1; pp < split; ++pp) {
          const float* base = PART + (size_t)(pp - 1) * 4 * pstride + tt * 32 + lane;
          ks[m] += base[0 * pstride];
          qs[m] += base[1 * pstride];
          kk[m] += base[2 * pstride];
          qk[m] += base[3 * pstride];
        }
        KS[tt * kDnCols + lane] = ks[m];
        QS[tt * kDnCols + lane] = qs[m];
        KK[tt * kMaxRows + lane] = kk[m];
        C[tt * kMaxRows + lane] = qk[m];
      }
    }
  }
  __syncthreads();
  // right-hand side beta_t (v_t - exp(gc_t) S0^T k_t) in place of K S0; the
  // coefficients A (strict ancestors) and C (the path, t included)
  for (int idx = threadIdx.x; idx < n * kMaxRows; idx += kDnThreads) {
    const int tt = idx / kMaxRows, s = idx - tt * kMaxRows;
    KS[tt * kDnCols + s] = s_beta[tt] * (VB[tt * kDnCols + s] - expf(s_gc[tt]) * KS[tt * kDnCols + s]);
    const bool on_path = s < n && ((s_anc[tt] >> s) & 1u);
    const float decay = on_path ? expf(s_gc[tt] - s_gc[s]) : 0.f;
    A[tt * kMaxRows + s] = (on_path && s < tt) ? s_beta[tt] * decay * KK[tt * kMaxRows + s] : 0.f;
    C[tt * kMaxRows + s] = decay * C[tt * kMaxRows + s];
  }
  // rows past n of U meet zero coefficients in the outputs: clear them
  for (int idx = n * kDnCols + threadIdx.x; idx < kMaxRows * kDnCols; idx += kDnThreads) U[idx] = 0.f;
  __syncthreads();
  // forward substitution u_t = rhs_t - sum_{s < t} A[t][s] u_s, one column per
  // lane with the column in registers (A is zero off the path)
  if (warp == 0) {
    float ur[kMaxRows];
#pragma unroll
    for (int tt = 0; tt < kMaxRows; ++tt) {
      if (tt < n) {
        float a0 = KS[tt * kDnCols + lane], a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int s4 = 0; s4 < tt; s4 += 4) {
          const float4 c4 = *reinterpret_cast<const float4*>(A + tt * kMaxRows + s4);
          a0 = fmaf(-c4.x, ur[s4], a0);
          if (s4 + 1 < tt) a1 = fmaf(-c4.y, ur[s4 + 1], a1);
          if (s4 + 2 < tt) a2 = fmaf(-c4.z, ur[s4 + 2], a2);
          if (s4 + 3 < tt) a3 = fmaf(-c4.w, ur[s4 + 3], a3);
        }
        ur[tt] = (a0 + a1) + (a2 + a3);
        U[tt * kDnCols + lane] = ur[tt];
      }
    }
  }
  __syncthreads();
  // outputs o_t = exp(gc_t) S0^T q_t + sum_s C[t][s] u_s
#pragma unroll
  for (int m = 0; m < kMaxRows / kDnWarps; ++m) {
    const int tt = warp + kDnWarps * m;
    if (tt < n) {
      float a0 = expf(s_gc[tt]) * QS[tt * kDnCols + lane], a1 = 0.f;
      for (int s4 = 0; s4 <= tt; s4 += 4) {
        const float4 c4 = *reinterpret_cast<const float4*>(C + tt * kMaxRows + s4);
        a0 = fmaf(c4.x, U[s4 * kDnCols + lane], a0);
        a1 = fmaf(c4.y, U[(s4 + 1) * kDnCols + lane], a1);
        a0 = fmaf(c4.z, U[(s4 + 2) * kDnCols + lane], a0);
        a1 = fmaf(c4.w, U[(s4 + 3) * kDnCols + lane], a1);
      }
      const size_t off = ((size_t)(row0 + tt) * Hv + h) * dv + c0 + lane;
      o[off] = a0 + a1;
      u[off] = U[tt * kDnCols + lane];
    }
  }
  if (cb == 0 && threadIdx.x < n) gc_out[(size_t)(row0 + threadIdx.x) * Hv + h] = s_gc[threadIdx.x];
}

// Untiled TMA copy global -> shared, completing on an mbarrier (addresses
// 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// dynamic shared memory of the commit CTA, in floats: two slots of (state
// tile, the path's k rows, u rows, gates, weights)
struct DnCommitLayout {
  int st, kr, ur, gr, wr, slot, total;
};
__host__ __device__ inline DnCommitLayout dn_commit_layout(int dk, int dv) {
  DnCommitLayout L;
  int o = 0;
  L.st = o; o += dk * dv;
  L.kr = o; o += kMaxRows * dk;
  L.ur = o; o += kMaxRows * dv;
  L.gr = o; o += kMaxRows;
  L.wr = o; o += kMaxRows;
  L.slot = o;
  L.total = 2 * o;
  return L;
}

// S <- exp(gc_last) S + sum_{d <= a} exp(gc_last - gc_{p_d}) k_{p_d} u_{p_d}^T
// for the accepted path p_0 = 0, ..., p_a of each request, in every layer.
// Persistent: one CTA per SM walks the (request, layer, value head) tiles with
// a stride of the grid, two tiles in flight: the tile's state (d_k x d_v,
// contiguous) by one TMA bulk copy, the path's k rows, u rows and gates by
// asynchronous copies, while the previous tile is updated in 4 x 4 register
// blocks and written back.  Every CTA first checks every request's path
// (a in [0, n), p_0 = 0, parent(p_d) = p_{d-1}); with a bad path nothing is
// written anywhere.
__global__ void __launch_bounds__(kDnCommitThreads, 1) dn_commit_kernel(ReqTable t, DnStates st, int Hk, int Hv,
                                                                        int dk, int dv, int n_layers,
                                                                        int rows_per_layer, const float* k,
                                                                        const float* u, const float* gc,
                                                                        const int32_t* path, const int32_t* accept_len,
                                                                        int32_t* status) {
  extern __shared__ __align__(16) float dsm[];
  __shared__ __align__(8) uint64_t s_bar[2];
  __shared__ int s_p[kMaxReq][kMaxRows];
  __shared__ int s_a[kMaxReq];
  __shared__ int s_bad;
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const DnCommitLayout L = dn_commit_layout(dk, dv);
  if (threadIdx.x == 0) {
    s_bad = 0;
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  for (int r = warp; r < t.n_req; r += kDnCommitThreads / 32) {   // one warp per request
    const int n = t.n[r], row0 = t.row_off[r];
    const int a = accept_len[r];
    bool bad = a < 0 || a >= n;
    if (!bad && lane <= a) {
      const int p = path[row0 + lane];
      s_p[r][lane] = p;
      if (p < 0 || p >= n) bad = true;
      else if (lane == 0) bad = p != 0;
      else bad = t.parent[r][p] != path[row0 + lane - 1];
    }
    bad = __any_sync(FULL, bad);
    if (lane == 0) {
      s_a[r] = a;
      if (bad) s_bad = 1;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) status_set(status, TV_E_PATH);
    return;
  }

  const int per_req = n_layers * Hv;
  const int n_tiles = t.n_req * per_req;
  const uint32_t tile_bytes = (uint32_t)(dk * dv * sizeof(float));
  auto tile_state = [&](int tile) {
    const int r = tile / per_req, rem = tile - r * per_req;
    return st.S[r] + (size_t)rem * dk * dv;   // rem = layer * Hv + h
  };
  // start the copies of one tile into one slot (thread 0: the state; all: the rest)
  auto stage = [&](int tile, int slot) {
    float* base = dsm + slot * L.slot;
    const int r = tile / per_req, rem = tile - r * per_req;
    const int layer = rem / Hv, h = rem - layer * Hv, kh = h / (Hv / Hk);
    const int a = s_a[r], row0 = t.row_off[r];
    const size_t lrow = (size_t)layer * rows_per_layer + row0;
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&s_bar[slot], tile_bytes);
      bulk_g2s(base + L.st, tile_state(tile), tile_bytes, &s_bar[slot]);
    }
    const int k4 = dk / 4, v4 = dv / 4;
    for (int idx = threadIdx.x; idx < (a + 1) * (k4 + v4 + 1); idx += kDnCommitThreads) {
      const int d = idx / (k4 + v4 + 1), c = idx - d * (k4 + v4 + 1);
      const size_t pr = lrow + s_p[r][d];
      if (c < k4) cp_async16(base + L.kr + d * dk + 4 * c, k + (pr * Hk + kh) * dk + 4 * c);
      else if (c < k4 + v4) cp_async16(base + L.ur + d * dv + 4 * (c - k4), u + (pr * Hv + h) * dv + 4 * (c - k4));
      else cp_async4(base + L.gr + d, gc + pr * Hv + h);
    }
  };
  int tile = blockIdx.x;
  if (tile < n_tiles) stage(tile, 0);
  cp_async_commit();
  if (tile + (int)gridDim.x < n_tiles) stage(tile + gridDim.x, 1);
  cp_async_commit();
  bool timed_out = false;
  for (int j = 0; tile < n_tiles; ++j, tile += gridDim.x) {
    const int slot = j & 1;
    float* base = dsm + slot * L.slot;
    const float* ST = base + L.st;
    const float* KR = base + L.kr;
    const float* UR = base + L.ur;
    float* WR = base + L.wr;
    cp_async_wait_prev();   // this tile's group (the next tile's may still be in flight)
    if (!mbar_wait(&s_bar[slot], (uint32_t)((j >> 1) & 1))) {
      // report, then wait (bounded) once more for the copy in flight before leaving
      status_set(status, TV_E_TIMEOUT);
      mbar_wait(&s_bar[slot], (uint32_t)((j >> 1) & 1));
      timed_out = true;
    }
    timed_out = __syncthreads_or(timed_out);
    if (timed_out) {   // the other slot may hold a copy in flight too
      if (tile + (int)gridDim.x < n_tiles) mbar_wait(&s_bar[slot ^ 1], (uint32_t)(((j + 1) >> 1) & 1));
      break;
    }
    const int r = tile / per_req;
    const int a = s_a[r];
    const float gl = base[L.gr + a];
    if ((int)threadIdx.x <= a) WR[threadIdx.x] = expf(gl - base[L.gr + threadIdx.x]);
    __syncthreads();
    const float decay = expf(gl);
    float* S = tile_state(tile);
    const int cq_n = dv / 4, quads = (dk / 4) * cq_n;
    for (int pq = threadIdx.x; pq < quads; pq += kDnCommitThreads) {
      const int i4 = (pq / cq_n) * 4, j4 = (pq % cq_n) * 4;
      float4 x[4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        x[rr] = *reinterpret_cast<const float4*>(ST + (i4 + rr) * dv + j4);
        x[rr].x *= decay;
        x[rr].y *= decay;
        x[rr].z *= decay;
        x[rr].w *= decay;
      }
      for (int d = 0; d <= a; ++d) {
        const float w = WR[d];
        const float4 kd = *reinterpret_cast<const float4*>(KR + d * dk + i4);
        const float4 ud = *reinterpret_cast<const float4*>(UR + d * dv + j4);
        const float kr[4] = {kd.x * w, kd.y * w, kd.z * w, kd.w * w};
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
          x[rr].x = fmaf(kr[rr], ud.x, x[rr].x);
          x[rr].y = fmaf(kr[rr], ud.y, x[rr].y);
          x[rr].z = fmaf(kr[rr], ud.z, x[rr].z);
          x[rr].w = fmaf(kr[rr], ud.w, x[rr].w);
        }
      }
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) *reinterpret_cast<float4*>(S + (size_t)(i4 + rr) * dv + j4) = x[rr];
    }
    __syncthreads();   // the slot is free again
    if (tile + 2 * (int)gridDim.x < n_tiles) stage(tile + 2 * gridDim.x, slot);
    cp_async_commit();
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

std::atomic<bool> g_dn_verify_smem[64];
std::atomic<bool> g_dn_commit_smem[64];

}  // namespace

size_t dn_verify_smem(int dk) { return (size_t)dn_verify_layout(dk).total * sizeof(float); }
size_t dn_commit_smem(int dk, int dv) { return (size_t)dn_commit_layout(dk, dv).total * sizeof(float); }

int launch_dn_verify(const ReqTable& t, const DnStates& st, int Hk, int Hv, int dk, int dv, const float* q,
                     const float* k, const float* v, const float* beta, const float* g, float* o, float* u, float* gc,
                     int32_t* status, cudaStream_t s, bool state_early) {
  int rc = ensure_smem_limit(dn_verify_kernel, dn_verify_smem(kDnMaxDim), g_dn_verify_smem);
  if (rc) return rc;
  return launch_pdl(dn_verify_kernel, dim3(Hv, dv / kDnCols, t.n_req), dim3(kDnThreads), dn_verify_smem(dk), s, t,
                    st, Hk, Hv, dk, dv, q, k, v, beta, g, o, u, gc, status, state_early ? 1 : 0);
}

int launch_dn_commit(const ReqTable& t, const DnStates& st, int Hk, int Hv, int dk, int dv, int n_layers,
                     const float* k, const float* u, const float* gc, const int32_t* path, const int32_t* accept_len,
                     int32_t* status, cudaStream_t s) {
  int rc = ensure_smem_limit(dn_commit_kernel, dn_commit_smem(kDnMaxDim, kDnMaxDim), g_dn_commit_smem);
  if (rc) return rc;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return TV_E_CUDA;
  const int tiles = t.n_req * n_layers * Hv;
  const int grid = tiles < sms ? tiles : sms;
  return launch_pdl(dn_commit_kernel, dim3(grid), dim3(kDnCommitThreads), dn_commit_smem(dk, dv), s, t, st, Hk, Hv,
                    dk, dv, n_layers, t.total_rows, k, u, gc, path, accept_len, status);
}

}  // namespace tv
