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
//    request).  The dot products of the tree's keys and queries with S0's
//    columns and with each other (K S0, Q S0, K K^T, Q K^T) run as one
//    tcgen05 MMA chain over bf16 hi/lo splits of the fp32 operands, the four
//    hi/lo cross terms summed in fp32 (each product term within 2^-17 of the
//    fp32 product); the coefficients, the right-hand sides, the triangular
//    solve by forward substitution in node order (parents come first) and the
//    outputs follow in fp32 on the CUDA cores.
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

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Dynamic shared memory of the verify CTA (bytes from a 1024-byte aligned
// base).  The tensor-core operands are bf16, K-major, 128-byte swizzled slabs
// of 64 coordinates each (d_k padded to a multiple of 64 with zeros):
//   A: 128 rows = k_t hi (rows 0..31), q_t hi (32..63), k_t lo (64..95),
//      q_t lo (96..127), nodes past n zero;
//   B: 2 NB rows = S0's 32 block columns (S0^T) hi, the same lo, then the
//      tree's k rows (NK = 16 when n <= 16, else 32) hi, the same lo;
// hi = bf16(x), lo = bf16(x - hi).  D = A B^T (fp32, in TMEM): for a k or q
// row t the four (row, column) combinations t / t + 64 by the hi / lo column
// sum to (hi + lo)(hi + lo) over d_k, every product term within 2^-17 of the
// fp32 product.  Then fp32 matrices: the four sums of D ([128 rows][68]) and
// the solve's operands.
struct DnVerifyLayout {
  static constexpr int A_SLAB = 128 * 128;        // bytes per 64-coordinate slab of A
  static constexpr int B_SLAB = 128 * 128;        // of B (2 NB <= 128 rows)
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + 2 * A_SLAB;
  static constexpr int OFF_Y = 0;                                    // [128][68]: D, hi + lo columns added
  static constexpr int Y_F = 68;                                     // (over A and B, free once the MMAs are done)
  static constexpr int OFF_RHS = OFF_B + 2 * B_SLAB;                 // [32][36] beta_t (v_t - exp(gc_t) S0^T k_t)
  static constexpr int OFF_EQS = OFF_RHS + kMaxRows * 36 * 4;        // [32][36] exp(gc_t) S0^T q_t
  static constexpr int OFF_CA = OFF_EQS + kMaxRows * 36 * 4;         // [32][36] A: strict ancestors
  static constexpr int OFF_CC = OFF_CA + kMaxRows * 36 * 4;          // [32][36] C: the path, t included
  static constexpr int OFF_V = OFF_CC + kMaxRows * 36 * 4;           // [32][32] v[:, column block]
  static constexpr int OFF_U = OFF_V + kMaxRows * kDnCols * 4;       // [32][32] pseudo-values
  static constexpr int BYTES = OFF_U + kMaxRows * kDnCols * 4;
  static constexpr size_t ALLOC = 1024 + BYTES;
  static_assert(OFF_Y + 128 * Y_F * 4 <= OFF_RHS, "D's staging fits over the operands");
};
constexpr int kDnRowF = 36;
constexpr uint32_t kDnTmemCols = 128;
constexpr int kDnStageWarps = kDnWarps - 2;                 // warps 14, 15: the tree
constexpr int kDnStageThreads = 32 * kDnStageWarps;
constexpr int kDnTasks = 5;   // staging tasks a thread: 16-byte chunks of 8 coordinates (2048 at most)

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }

// 32 lanes x 16 consecutive 32-bit TMEM columns (this thread's lane)
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// y[0..16) = hi + lo of 16 columns
__device__ __forceinline__ void add16(float* y, const uint32_t (&a)[16], const uint32_t (&b)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    reinterpret_cast<float4*>(y)[j] =
        make_float4(__uint_as_float(a[4 * j]) + __uint_as_float(b[4 * j]),
                    __uint_as_float(a[4 * j + 1]) + __uint_as_float(b[4 * j + 1]),
                    __uint_as_float(a[4 * j + 2]) + __uint_as_float(b[4 * j + 2]),
                    __uint_as_float(a[4 * j + 3]) + __uint_as_float(b[4 * j + 3]));
}

// hi and lo bf16 planes of 8 consecutive coordinates
__device__ __forceinline__ void split8(const float (&x)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    const float2 hf = __bfloat1622float2(hv);
    h[e] = bf16x2_bits(hv);
    l[e] = bf16x2_bits(__floats2bfloat162_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// u_t = rhs_t - sum_{s < t} A[t][s] u_s by forward substitution in node order
// (parents come first), column c on lane c in registers.  All NMAX rows are
// computed (rows past n from whatever their shared-memory rows hold, and
// never used: row t depends on rows before it only), so the loop is straight
// code whose coefficient loads need not wait; rows below n are stored at the end.
template <int NMAX>
__device__ __forceinline__ void dn_substitute_warp(const float* RHS, const float* CA, float* U, float* u_out,
                                                   size_t row_stride, int n, int lane) {
  constexpr int NQ = NMAX / 4;
  float ur[NMAX];
  float4 cur[NQ], nxt[NQ];
  float rcur = RHS[lane], rnxt = 0.f;
#pragma unroll
  for (int tt = 0; tt < NMAX; ++tt) {
    // the next row's coefficients and right-hand side, asked for before this
    // row's FMAs (software pipelining: their latency hides behind them)
    if (tt + 1 < NMAX) {
#pragma unroll
      for (int q4 = 0; q4 < NQ; ++q4)
        if (4 * q4 < tt + 1) nxt[q4] = *reinterpret_cast<const float4*>(CA + (tt + 1) * kDnRowF + 4 * q4);
      rnxt = RHS[(tt + 1) * kDnRowF + lane];
    }
    float a0 = rcur, a1 = 0.f;
#pragma unroll
    for (int s4 = 0; s4 < tt; s4 += 4) {
      const float4 c4 = cur[s4 / 4];
      a0 = fmaf(-c4.x, ur[s4], a0);
      if (s4 + 1 < tt) a1 = fmaf(-c4.y, ur[s4 + 1], a1);
      if (s4 + 2 < tt) a0 = fmaf(-c4.z, ur[s4 + 2], a0);
      if (s4 + 3 < tt) a1 = fmaf(-c4.w, ur[s4 + 3], a1);
    }
    ur[tt] = a0 + a1;
#pragma unroll
    for (int q4 = 0; q4 < NQ; ++q4) cur[q4] = nxt[q4];
    rcur = rnxt;
  }
#pragma unroll
  for (int tt = 0; tt < NMAX; ++tt) {
    if (tt < n) {
      U[tt * kDnCols + lane] = ur[tt];
      u_out[tt * row_stride + lane] = ur[tt];
    }
  }
}

// o_t = exp(gc_t) S0^T q_t + sum_{s <= t} C[t][s] u_s for the rows t = warp,
// warp + 16, ... below n; the s loop unrolled to NMAX (C is zero off the path)
template <int NMAX>
__device__ __forceinline__ void dn_outputs(const float* EQS, const float* CC, const float* U, float* o_out,
                                           size_t row_stride, int n, int warp, int lane) {
  for (int r2 = warp; r2 < n; r2 += kDnWarps) {
    float a0 = EQS[r2 * kDnRowF + lane], a1 = 0.f;
#pragma unroll
    for (int s4 = 0; s4 < NMAX; s4 += 4) {
      if (s4 <= r2) {
        const float4 c4 = *reinterpret_cast<const float4*>(CC + r2 * kDnRowF + s4);
        a0 = fmaf(c4.x, U[s4 * kDnCols + lane], a0);
        if (s4 + 1 <= r2) a1 = fmaf(c4.y, U[(s4 + 1) * kDnCols + lane], a1);
        if (s4 + 2 <= r2) a0 = fmaf(c4.z, U[(s4 + 2) * kDnCols + lane], a0);
        if (s4 + 3 <= r2) a1 = fmaf(c4.w, U[(s4 + 3) * kDnCols + lane], a1);
      }
    }
    o_out[(size_t)r2 * row_stride + lane] = a0 + a1;
  }
}

// One CTA per (value head, block of 32 value columns, request), 512 threads.
// The dot products of the tree's keys and queries with S0's columns and with
// the tree's keys run on the tensor core (one M=128 MMA chain); the
// coefficients, the right-hand sides and the triangular solve follow in fp32
// on the CUDA cores.  Warps 0..13 stage the operands, warp 14 computes the
// cumulative gates and root paths, warp 15 checks the tree.
__global__ void __launch_bounds__(kDnThreads) dn_verify_kernel(ReqTable t, DnStates st, int Hk, int Hv, int dk, int dv,
                                                               const float* q, const float* k, const float* v,
                                                               const float* beta, const float* g, float* o, float* u,
                                                               float* gc_out, int32_t* status, int state_early) {
  using L = DnVerifyLayout;
  extern __shared__ __align__(16) uint8_t dn_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dn_smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t s_mma;
  __shared__ uint32_t s_tmem;
  __shared__ float s_gc[kMaxRows], s_beta[kMaxRows], s_eg[kMaxRows];
  __shared__ unsigned s_anc[kMaxRows];   // bit s: s is on t's root path (t included)
  __shared__ int s_err, s_stat, s_done;
  const int h = blockIdx.x, cb = blockIdx.y, r = blockIdx.z;
  const int c0 = cb * kDnCols;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int n = t.n[r], row0 = t.row_off[r];
  const int kh = h / (Hv / Hk);
  const int kcs = dk > 64 ? 4 : 3;              // log2 of the 16-byte chunks of a padded row
  const int KC = 1 << kcs;
  const int NK = n <= 16 ? 16 : 32;             // tree-node rows of B (each plane)
  const int NB = kDnCols + NK;                  // B rows a plane
  float* Y = reinterpret_cast<float*>(smem + L::OFF_Y);
  float* RHS = reinterpret_cast<float*>(smem + L::OFF_RHS);
  float* EQS = reinterpret_cast<float*>(smem + L::OFF_EQS);
  float* CA = reinterpret_cast<float*>(smem + L::OFF_CA);
  float* CC = reinterpret_cast<float*>(smem + L::OFF_CC);
  float* VB = reinterpret_cast<float*>(smem + L::OFF_V);
  float* U = reinterpret_cast<float*>(smem + L::OFF_U);
  if (warp == 0) {
    tmem_alloc(&s_tmem, kDnTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    mbar_init(&s_mma, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  // staging tasks of warps 0..13, task = threadIdx.x + 448 m: [0, 2 NK KC)
  // rows of A (NK k rows, then NK q rows), then 32 KC of S0's columns (lane =
  // column: coalesced), then NK KC tree-node k rows of B.  Rows of nodes past
  // NK are left as they are: they only meet D rows and columns never read.
  const int nks = n <= 16 ? 4 : 5;              // log2 NK
  const int nA = 2 * NK * KC, nS = kDnCols * KC, nT = nA + nS + NK * KC;
  const bool stager = warp < kDnStageWarps;
  const float* S0g = st.S[r] + (size_t)h * dk * dv + c0;
  float x[kDnTasks][8];
  auto load_task = [&](int m, bool state) {
    const int task = threadIdx.x + kDnStageThreads * m;
#pragma unroll
    for (int e = 0; e < 8; ++e) x[m][e] = 0.f;
    if (!stager || task >= nT) return;
    if (task >= nA && task < nA + nS) {
      if (!state) return;
      const int id = task - nA, c = id % kDnCols, j = id / kDnCols;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (8 * j + e < dk) x[m][e] = S0g[(size_t)(8 * j + e) * dv + c];
      return;
    }
    if (state) return;
    const bool a = task < nA;
    const int id = a ? task : task - nA - nS;
    const int row = id >> kcs, j = id & (KC - 1);
    const int node = row & (NK - 1);
    if (node >= n || 8 * j >= dk) return;
    const float* src = (a && row >= NK) ? q : k;
    const float4* p4 = reinterpret_cast<const float4*>(src + ((size_t)(row0 + node) * Hk + kh) * dk + 8 * j);
    const float4 lo4 = p4[0], hi4 = p4[1];
    x[m][0] = lo4.x; x[m][1] = lo4.y; x[m][2] = lo4.z; x[m][3] = lo4.w;
    x[m][4] = hi4.x; x[m][5] = hi4.y; x[m][6] = hi4.z; x[m][7] = hi4.w;
  };
  // the state before the round: with state_early loaded before the wait (the
  // caller guarantees that every writer of it has completed by then)
  if (state_early) {
#pragma unroll
    for (int m = 0; m < kDnTasks; ++m) load_task(m, true);
  } else if ((int)threadIdx.x < dk) {
    // otherwise the state's rows (128 bytes of this block's columns each) are
    // only asked into L2, which every write reaches: whatever writes them
    // before the wait, the loads after it read the written values
    asm volatile("prefetch.global.L2 [%0];" ::"l"(S0g + (size_t)threadIdx.x * dv) : "memory");
  }
  pdl_wait();
  pdl_trigger();
  // every load below is in bounds whatever an earlier kernel left; the status
  // (an earlier error) is read with them and checked before anything is written
  if (warp == kDnWarps - 2) {
    // cumulative gates and root paths by pointer doubling over the parent
    // links (gc = sum of g over the root path); the tree is checked by warp 15
    int up = -1;
    float acc = 0.f, bl = 0.f;
    if (lane < n) {
      up = t.parent[r][lane];
      acc = g[(size_t)(row0 + lane) * Hv + h];
      bl = beta[(size_t)(row0 + lane) * Hv + h];
    }
    up = (lane > 0 && up >= 0 && up < lane) ? up : -1;   // an out-of-order parent stops the walk (warp 15 reports it)
    unsigned anc = lane < n ? (1u << lane) : 0u;
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
      s_eg[lane] = expf(acc);
      s_anc[lane] = anc;
      s_beta[lane] = bl;
    }
  } else if (warp == kDnWarps - 1) {
    int par = 0, tok = 0;
    if (lane < n) {
      par = t.parent[r][lane];
      tok = t.token[r][lane];
    }
    const int err = check_tree_warp(par, tok, n, 0);
    if (lane == 0) {
      s_err = err;
      s_stat = status_get(status);
    }
  } else {
    float4 vreg = make_float4(0.f, 0.f, 0.f, 0.f);
    const int vs = threadIdx.x >> 3, vc = threadIdx.x & 7;   // v[:, column block]: 32 nodes x 8 float4
    if (threadIdx.x < kMaxRows * kDnCols / 4 && vs < n)
      vreg = *reinterpret_cast<const float4*>(v + ((size_t)(row0 + vs) * Hv + h) * dv + c0 + 4 * vc);
    // two waves of tasks (0..2, then the rest: only trees past 16 nodes have
    // them), each loaded, then split and stored
#pragma unroll
    for (int wv = 0; wv < 2; ++wv) {
      const int m0 = wv == 0 ? 0 : 3, m1 = wv == 0 ? 3 : kDnTasks;
#pragma unroll
      for (int m = m0; m < m1; ++m) {
        const int task = threadIdx.x + kDnStageThreads * m;
        const bool is_state = task >= nA && task < nA + nS;
        if (is_state) {
          if (!state_early) load_task(m, true);
        } else {
          load_task(m, false);
        }
      }
      // the operand planes (zeros for nodes past n and coordinates past d_k)
#pragma unroll
      for (int m = m0; m < m1; ++m) {
        const int task = threadIdx.x + kDnStageThreads * m;
        if (task >= nT) continue;
        uint4 hi, lo;
        split8(x[m], hi, lo);
        if (task < nA) {
          const int id = task >> kcs, j = task & (KC - 1);
          const int row = ((id >> nks) << 5) | (id & (NK - 1));   // k node rows 0.., q node rows 32..
          uint8_t* base = smem + L::OFF_A + (j >> 3) * L::A_SLAB;
          *reinterpret_cast<uint4*>(base + swz(row, j & 7)) = hi;
          *reinterpret_cast<uint4*>(base + swz(row + 64, j & 7)) = lo;
        } else {
          int row, row_lo, j;
          if (task < nA + nS) {   // S0^T: hi rows 0..31, lo rows 32..63
            const int id = task - nA;
            row = id % kDnCols;
            row_lo = kDnCols + row;
            j = id / kDnCols;
          } else {                // tree nodes: hi rows 64.., lo rows 64 + NK..
            const int id = task - nA - nS;
            row = 2 * kDnCols + (id >> kcs);
            row_lo = row + NK;
            j = id & (KC - 1);
          }
          uint8_t* base = smem + L::OFF_B + (j >> 3) * L::B_SLAB;
          *reinterpret_cast<uint4*>(base + swz(row, j & 7)) = hi;
          *reinterpret_cast<uint4*>(base + swz(row_lo, j & 7)) = lo;
        }
      }
    }
    if (threadIdx.x < kMaxRows * kDnCols / 4) reinterpret_cast<float4*>(VB)[threadIdx.x] = vreg;
    fence_async_smem();
  }
  __syncthreads();
  const bool go = s_stat == 0 && s_err == TV_OK;
  if (!go && s_stat == 0 && threadIdx.x == 0 && h == 0 && cb == 0) status_set(status, s_err);
  if (go) {
    // (1) D = A B^T: one thread issues and waits
    if (threadIdx.x == 0) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16_f32(128, 2 * NB);
      const uint32_t a0 = smem_u32(smem + L::OFF_A), b0 = smem_u32(smem + L::OFF_B);
      const int ksteps = KC / 2;   // 16 coordinates a step
#pragma unroll 1
      for (int ks = 0; ks < ksteps; ++ks) {
        const uint32_t aa = a0 + (uint32_t)((ks >> 2) * L::A_SLAB + (ks & 3) * 32);
        const uint32_t bb = b0 + (uint32_t)((ks >> 2) * L::B_SLAB + (ks & 3) * 32);
        umma_bf16(tmem, sdesc_sw128(aa, 16, 1024), sdesc_sw128(bb, 16, 1024), idesc, ks ? 1u : 0u);
      }
      umma_commit(&s_mma);
      int done = 1;
      if (!mbar_wait(&s_mma, 0)) {   // report, then wait (bounded) once more before TMEM is freed
        status_set(status, TV_E_TIMEOUT);
        mbar_wait(&s_mma, 0);
        done = 0;
      }
      s_done = done;
    }
    __syncthreads();
    if (s_done) {
      // (2) D to shared memory, hi and lo columns added: warp w reads TMEM
      //     lanes 32 (w & 3) .. (its subpartition); w < 4 the S0 columns, 4 <= w
      //     < 8 the tree-node columns
      if (warp < 8) {
        tc_fence_after();
        const int sp = warp & 3;
        const uint32_t ta = tmem + ((uint32_t)(32 * sp) << 16);
        float* yr = Y + (32 * sp + lane) * L::Y_F;
        uint32_t d0[16], d1[16];   // 16 columns a load (two CTAs share the SM's registers)
        if (warp < 4) {   // S0 columns: hi at 0.., lo at kDnCols..
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            tmem_ld_x16(ta + 16 * hf, d0);
            tmem_ld_x16(ta + kDnCols + 16 * hf, d1);
            tmem_ld_wait();
            add16(yr + 16 * hf, d0, d1);
          }
        } else {          // tree-node columns: hi at 0.., lo at NK..
          const uint32_t tn = ta + 2 * kDnCols;
          for (int hf = 0; hf < NK / 16; ++hf) {
            tmem_ld_x16(tn + 16 * hf, d0);
            tmem_ld_x16(tn + NK + 16 * hf, d1);
            tmem_ld_wait();
            add16(yr + kDnCols + 16 * hf, d0, d1);
          }
        }
      }
      __syncthreads();
      // (3) a warp per tree row t, the column on the lane: x = Y[t] + Y[64 + t]
      //     (k_t) and Y[32 + t] + Y[96 + t] (q_t); the right-hand side and A
      //     from k_t, exp(gc_t) S0^T q_t and C from q_t, zero off the path
      for (int tt = warp; tt < n; tt += kDnWarps) {
        const float* yk = Y + tt * L::Y_F;
        const float* yq = Y + (32 + tt) * L::Y_F;
        const float bt = s_beta[tt], et = s_eg[tt];
        const float pk = yk[lane] + yk[64 * L::Y_F + lane];
        const float pq = yq[lane] + yq[64 * L::Y_F + lane];
        RHS[tt * kDnRowF + lane] = bt * (VB[tt * kDnCols + lane] - et * pk);
        EQS[tt * kDnRowF + lane] = et * pq;
        if (lane < NK) {
          const int s = lane;
          const float kk = yk[kDnCols + s] + yk[64 * L::Y_F + kDnCols + s];
          const float qk = yq[kDnCols + s] + yq[64 * L::Y_F + kDnCols + s];
          const bool on = s < n && ((s_anc[tt] >> s) & 1u);
          const float decay = on ? expf(s_gc[tt] - s_gc[s]) : 0.f;
          CA[tt * kDnRowF + s] = (on && s != tt) ? bt * decay * kk : 0.f;
          CC[tt * kDnRowF + s] = on ? decay * qk : 0.f;
        }
      }
      __syncthreads();
      // (4) the pseudo-values, one warp
      if (warp == 0) {
        float* uo = u + ((size_t)row0 * Hv + h) * dv + c0;
        if (n <= 16) dn_substitute_warp<16>(RHS, CA, U, uo, (size_t)Hv * dv, n, lane);
        else dn_substitute_warp<kMaxRows>(RHS, CA, U, uo, (size_t)Hv * dv, n, lane);
      }
      __syncthreads();
      // (5) o_t = exp(gc_t) S0^T q_t + sum_{s <= t} C[t][s] u_s
      {
        float* oo = o + ((size_t)row0 * Hv + h) * dv + c0;
        if (n <= 16) dn_outputs<16>(EQS, CC, U, oo, (size_t)Hv * dv, n, warp, lane);
        else dn_outputs<kMaxRows>(EQS, CC, U, oo, (size_t)Hv * dv, n, warp, lane);
      }
      if (cb == 0 && threadIdx.x < n) gc_out[(size_t)(row0 + threadIdx.x) * Hv + h] = s_gc[threadIdx.x];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kDnTmemCols);
  }
}

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
  cp_async_wait_all();
}

std::atomic<bool> g_dn_verify_smem[64];
std::atomic<bool> g_dn_commit_smem[64];

}  // namespace

size_t dn_verify_smem(int) { return DnVerifyLayout::ALLOC; }
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
