// Tree-masked GQA attention over the cached context plus the tree rows, on the
// 5th-generation tensor cores.
//
// Row i, query head h attends to the cached slots [0, ctx) and to the tree
// slots ctx + a for every a in anc(i) (its ancestors and itself): each node is
// masked to its ancestors and placed at a position equal to its depth
// [Drafters and tree verify, §Tree verify through recurrent layers].  The
// positions were applied by RoPE before the keys were written.
//
// Split-context (flash-decoding) layout: one CTA per (request, KV head, context
// chunk).  It holds every query vector of its KV head at once: the request's
// rows x the GQA heads of the KV head, at most 160, so each K/V byte is read
// once.  The chunks are whole 128-key tiles, their count aimed at SMs / KV
// heads (one wave for one request); the tree tile has a chunk of its own in
// short contexts and otherwise goes first in the last chunk.
// The merge kernel combines the chunks' partials (offset, sum, unnormalised
// output) in chunk order, so a row's result does not depend on the other rows.
//
// Transposed products: the keys of a tile sit on the 128 TMEM lanes and the
// query vectors are the MMA's N dimension, so a KV head's queries need no
// padding to 128.  Per 128-key tile t:
//   S^T = K_t Q^T      tcgen05.mma M128 (keys) N (queries) K16, fp32 in TMEM;
//                      K by TMA (K-major A), Q once by a 3-D TMA box (K-major B)
//   softmax            16 warps: four per TMEM lane quarter, each thread one key
//                      x a quarter of the query columns.  Each query column
//                      has an offset m (log2 units) that moves only when a
//                      score passes m + 8: the warps of a column slice find
//                      out with one barrier reduction, and only then compute
//                      the tile's column maxima.  P = 2^(s log2(e)/sqrt(D) - m)
//                      (SFU ex2), masked, rounded to bf16, parked in TMEM
//                      until the previous O^T MMA has read P^T, then stored
//                      into swizzled smem
//   O^T += V_t^T P^T   tcgen05.mma M128 (dimensions) N (queries) K16, V straight
//                      from its TMA layout and P^T as MN-major operands
// O, the column sums and the offsets all carry the same offset, which cancels
// in O / sum, so the lazy offset is exact.
// A 17th warp issues the TMA loads (two K and two V stages) and the MMAs from
// an event loop; it issues the first two K tiles before the programmatic-launch
// wait and the queries and the first two V tiles right after it.  S^T is double-buffered in TMEM so that S^T of tile t+1
// overlaps the softmax of t, and O^T of tile t overlaps the next tile's
// softmax up to its P^T store.
#include <cmath>
#include <cstring>
#include <type_traits>

#include "tv_common.cuh"
#include "tv_gemm.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr int kSlices = 4;                         // softmax warps per TMEM lane quarter = query-column slices
constexpr int kAtSoftWarps = 4 * kSlices;          // 16
constexpr int kAtSoftThreads = kAtSoftWarps * 32;  // 512
constexpr int kWarpIssue = kAtSoftWarps;           // TMEM owner, TMA and MMA issue
constexpr int kAtThreads = kAtSoftThreads + 32;
constexpr int kNqMax = kMaxQueriesPerKvHead;       // query columns of one KV head
constexpr int kCps = kNqMax / 8 / kSlices;         // 8-column chunks per slice
constexpr int kColS0 = 0, kColS1 = kNqMax, kColO = 2 * kNqMax;   // TMEM columns: S^T double buffer, O^T
constexpr int kAtTmemCols = 512;
constexpr int kAtom = 128 * 128;                   // bytes of one 128-row x 128-byte swizzled slab
constexpr float kRescaleLog2 = 8.f;                // an offset moves when a score passes it by 2^8
static_assert(kNqMax % (8 * kSlices) == 0 && 3 * kNqMax <= kAtTmemCols && kCps == 5, "query columns must fit TMEM");

struct AttnMaps {
  CUtensorMap k[kMaxReq];   // per request: [Hkv * capacity][D] bf16, box 64 x 128, 128B swizzle
  CUtensorMap v[kMaxReq];
  CUtensorMap q[kMaxReq];   // per request: q as [rows][Hq][D], box 64 x G x n (one KV head's query columns)
};

template <int D>
struct AtSmem {
  static constexpr int QSLAB = kNqMax * 128;       // one 64-dimension slab of the queries
  static constexpr int Q_BYTES = (D / 64) * QSLAB;
  static constexpr int KV_BYTES = 2 * kAtom;       // 128 keys x 128 dimensions (D = 64: the V upper slab stays 0)
  static constexpr int P_BYTES = 3 * kAtom;        // P^T: 128 keys x 3 slabs of 64 query columns
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;    // K stage s at OFF_K + s KV_BYTES
  static constexpr int OFF_V = OFF_K + 2 * KV_BYTES;
  static constexpr int OFF_P = OFF_V + 2 * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr size_t BYTES = 1024 + OFF_BAR + 256;
  static_assert(OFF_K % 1024 == 0, "swizzled slabs start on 1024-byte boundaries");
};

// 2^x with the SFU's approximate base-2 exponential (PTX ex2.approx.ftz;
// about 2^-22 relative error, 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// the four warps of one query-column slice (named barriers 1..4)
__device__ __forceinline__ void slice_sync(int cs) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + cs), "n"(4 * 32) : "memory");
}
// true on every thread of the slice if v is true on any of them
__device__ __forceinline__ bool slice_any(bool v, int cs) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(1 + cs), "n"(4 * 32)
      : "memory");
  return out != 0;
}

// maximum over the warp's 32 lanes, on every lane (PTX redux.sync.max.f32;
// NaN inputs are ignored)
__device__ __forceinline__ float redux_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 5, %0;" ::"n"(kAtSoftThreads) : "memory"); }

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 8 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// grid (chunks, KV heads, requests); 16 softmax warps and one issue warp.
//
// Tiles of a chunk: (last chunk) the tree tile, then its cached-key tiles.
// The issue warp's lane 0 runs an event loop: an MMA or TMA instruction holds
// its thread for about as long as the unit takes to accept it, so one thread
// serves every ready event in priority order instead of waiting on one:
//   O^T += V_t^T P_t^T   once P^T(t) is stored and V_t has landed
//   S^T(t) = K_t Q^T     once K_t has landed and S^T[t % 2] was read (tile t-2)
//   TMA K_t              once S^T(t-2) is done (its K stage is free)
//   TMA V_t              once O^T(t-2) is done (its V stage is free)
// Softmax warps, per tile t: pass 1 (offset check), O^T rescale if an offset
// moved, pass 2 (P^T), each reading this thread's 40 scores from TMEM.
template <int D>
__global__ void __launch_bounds__(kAtThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnMaps maps, ReqTable t, const RowMeta* meta, const __nv_bfloat16* q,
                   int Hq, int Hkv, int chunk_target, float scale_log2, float* part_ml, float* part_o,
                   int32_t* status) {
  using L = AtSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);    // [2] K tile landed
  uint64_t* v_full = k_full + 2;                                          // [2] V tile landed
  uint64_t* v_free = v_full + 2;                                          // [2] O^T MMA of the V stage done
  uint64_t* s_full = v_free + 2;                                          // [2] S^T MMA done
  uint64_t* s_free = s_full + 2;                                          // [2] S^T buffer read (16 warps)
  uint64_t* p_full = s_free + 2;                                          // P^T stored (16 warps)
  uint64_t* o_done = p_full + 1;                                          // O^T MMA of a tile done
  uint64_t* q_full = o_done + 1;                                          // query padding zeroed (16 warps)
  uint64_t* q_land = q_full + 1;                                          // queries landed (TMA)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_land + 1);
  int* s_stat = reinterpret_cast<int*>(tmem_slot + 1);
  __shared__ uint32_t s_anc[32];
  __shared__ int s_qrow[kNqMax];                     // query column c: its row of q and of the partials, (row0 + c / G) Hq + g G + c % G
  __shared__ uint32_t s_canc[kNqMax];                // query column c: the ancestor set of its tree row c / G
  __shared__ float s_red[4][kNqMax];                 // per lane quarter: column maxima; column sums
  // column offsets, double-buffered: a move writes the other buffer, so the
  // old offsets stay readable until every thread of the slice has used them
  __shared__ __align__(16) float s_m[2][kNqMax];     // offset m (log2 units), -inf before any visible key
  __shared__ __align__(16) float s_negm[2][kNqMax];  // -m
  __shared__ __align__(16) float s_alpha[kNqMax];    // 2^(m_old - m_new) of the last move

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = blockIdx.x, g = blockIdx.y, r = blockIdx.z;
  const bool issuer = warp == kWarpIssue && lane == 0;

  // ---- structural early exit (kernel parameters only) -------------------------
  const int ctx = t.ctx[r], n = t.n[r], row0 = t.row_off[r], cap = t.capacity[r];
  const AttnPlan plan = attn_plan(ctx, chunk_target);
  if (chunk >= plan.n_chunks) {
    pdl_wait();
    pdl_trigger();
    return;
  }
  const int G = Hq / Hkv, nq = n * G;
  const int NQ = (nq + 15) & ~15;                    // MMA N: a multiple of 16
  const bool last = chunk == plan.n_chunks - 1;
  const int key0 = chunk * plan.tiles_per_chunk * 128;
  const int ncache = plan.tree_own && last ? 0 : max(0, min(ctx - key0, plan.tiles_per_chunk * 128));
  const int Tc = (ncache + 127) / 128;
  const bool has_tree = last;
  const int T = Tc + (has_tree ? 1 : 0);
  // tile j: the tree tile first (last chunk), then the cached-key tiles.  The
  // tree keys usually carry a tree row's largest scores; taking them first
  // gives those keys the exact offset (P = 1 rounds exactly to bf16)
  const int tc0 = has_tree ? 1 : 0;
  auto is_tree = [&](int j) { return has_tree && j == 0; };
  auto tile_row = [&](int j) { return g * cap + (is_tree(j) ? ctx : key0 + (j - tc0) * 128); };   // first K/V row
  auto tile_keys = [&](int j) { return is_tree(j) ? n : min(128, ncache - (j - tc0) * 128); };     // valid keys
  // whole tile of cached keys below ctx: readable before the wait
  auto pre_ok = [&](int j) { return !is_tree(j) && key0 + (j - tc0 + 1) * 128 <= ctx; };

  // ---- set-up --------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&k_full[b], 1);
      mbar_init(&v_full[b], 1);
      mbar_init(&v_free[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], kAtSoftWarps);
    }
    mbar_init(p_full, kAtSoftWarps);
    mbar_init(o_done, 1);
    mbar_init(q_full, kAtSoftWarps);
    mbar_init(q_land, 1);
    fence_mbar_init();
    prefetch_tmap(&maps.k[r]);
    prefetch_tmap(&maps.v[r]);
    prefetch_tmap(&maps.q[r]);
  }
  if (warp == kWarpIssue) {
    tmem_alloc(tmem_slot, kAtTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- TMA issue ------------------------------------------------------------------
  int kiss = 0, viss = 0;   // K / V tiles issued (in tile order)
  uint32_t pre = 0;         // bit j: K_j issued before the wait
  const uint64_t pol = policy_evict_first();
  auto issue = [&](bool is_v, int j) {
    const int st = j & 1;
    uint8_t* dst = smem + (is_v ? L::OFF_V : L::OFF_K) + st * L::KV_BYTES;
    uint64_t* bar = is_v ? &v_full[st] : &k_full[st];
    mbar_arrive_expect_tx(bar, (D / 64) * kAtom);
#pragma unroll
    for (int a = 0; a < D / 64; ++a)
      tma_load_2d(dst + a * kAtom, is_v ? &maps.v[r] : &maps.k[r], bar, a * 64, tile_row(j), pol);
  };
  if (issuer) {
    // Cached keys below ctx are final before this grid starts: it starts once
    // the previous kernel has passed its own wait, and every kernel waits for
    // its predecessor before it completes, so every earlier writer of the
    // cache is done.  The tree slots (written by the previous kernel) and the
    // queries are read after the wait.
    for (int j = 0; j < 2 && j < T; ++j)   // K only: the queries go ahead of the V tiles
      if (pre_ok(j)) {
        issue(false, j);
        pre |= 1u << j;
      }
  }

  pdl_wait();
  pdl_trigger();
  if (issuer) {
    // the KV head's query columns (rows row0 .. row0 + n - 1, heads g G .. g G + G - 1:
    // column c = row c / G, head c % G), then the first two V tiles
    mbar_arrive_expect_tx(q_land, (uint32_t)((D / 64) * nq * 128));
#pragma unroll
    for (int a = 0; a < D / 64; ++a) tma_load_3d(smem + L::OFF_Q + a * L::QSLAB, &maps.q[r], q_land, a * 64, g * G, row0);
    for (int j = 0; j < 2 && j < T; ++j) issue(true, j);
  }
  if (threadIdx.x == 0) *s_stat = status_get(status);
  if (threadIdx.x < 32) s_anc[threadIdx.x] = (int)threadIdx.x < n ? meta[row0 + threadIdx.x].anc : 0u;
  __syncthreads();
  const bool run = *s_stat == 0;

  if (warp == kWarpIssue) {
    // ---------------- event-loop issuer (one thread) ----------------
    if (issuer && run) {
      const uint32_t qaddr = smem_u32(smem + L::OFF_Q);
      const uint32_t paddr = smem_u32(smem + L::OFF_P);
      const uint32_t idesc_s = idesc_bf16_f32(128, NQ);
      const uint32_t idesc_o = idesc_bf16_f32(128, NQ) | (1u << 15) | (1u << 16);   // A = V^T, B = P^T: MN-major
      for (int j = 0; j < 2 && j < T; ++j)
        if (!((pre >> j) & 1u)) issue(false, j);
      kiss = T < 2 ? T : 2;
      viss = T < 2 ? T : 2;
      int ns = 0, no = 0;   // S^T / O^T MMAs issued
      bool qready = false, ok = true;
      unsigned long long t_last = globaltimer();
      uint32_t polls = 0;
      while (no < T) {
        bool progress = false;
        if (!qready) qready = mbar_test(q_land, 0) && mbar_test(q_full, 0);
        // O^T += V^T P^T of tile no
        if (qready && no < ns && mbar_test(p_full, (uint32_t)no & 1u) &&
            mbar_test(&v_full[no & 1], (uint32_t)(no >> 1) & 1u)) {
          tc_fence_after();
          const uint32_t vaddr = smem_u32(smem + L::OFF_V + (no & 1) * L::KV_BYTES);
#pragma unroll
          for (int k = 0; k < 8; ++k)   // 16 keys per step
            umma_bf16(tmem + kColO, sdesc_sw128(vaddr + k * 2048, kAtom, 1024),
                      sdesc_sw128(paddr + k * 2048, kAtom, 1024), idesc_o, (no > 0 || k > 0) ? 1u : 0u);
          umma_commit(&v_free[no & 1]);
          umma_commit(o_done);
          ++no;
          progress = true;
        }
        // S^T of tile ns, after O^T of tile ns-2: that MMA is on the softmax's
        // critical path, S^T(ns) is not needed before the softmax of tile ns
        if (qready && ns < T && ns - 2 < no && (ns < 2 || mbar_test(&s_free[ns & 1], (uint32_t)((ns - 2) >> 1) & 1u)) &&
            mbar_test(&k_full[ns & 1], (uint32_t)(ns >> 1) & 1u)) {
          tc_fence_after();
          const uint32_t kaddr = smem_u32(smem + L::OFF_K + (ns & 1) * L::KV_BYTES);
          const uint32_t dS = tmem + (uint32_t)((ns & 1) ? kColS1 : kColS0);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t ka = kaddr + (uint32_t)((k >> 2) * kAtom + (k & 3) * 32);
            const uint32_t qa = qaddr + (uint32_t)((k >> 2) * L::QSLAB + (k & 3) * 32);
            umma_bf16(dS, sdesc_sw128(ka, 16, 1024), sdesc_sw128(qa, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[ns & 1]);
          ++ns;
          progress = true;
        }
        // K of tile kiss: its stage held tile kiss-2, whose S^T is done (S^T
        // of tile kiss cannot have run yet, so the parity names tile kiss-2)
        if (kiss < T && kiss - 2 < ns && mbar_test(&s_full[kiss & 1], (uint32_t)((kiss - 2) >> 1) & 1u)) {
          issue(false, kiss);
          ++kiss;
          progress = true;
        }
        // V of tile viss: its stage held tile viss-2, whose O^T is done (O^T
        // of tile viss cannot have run yet, so the parity names tile viss-2)
        if (viss < T && viss - 2 < no && mbar_test(&v_free[viss & 1], (uint32_t)((viss - 2) >> 1) & 1u)) {
          issue(true, viss);
          ++viss;
          progress = true;
        }
        if (progress) {
          t_last = globaltimer();
          polls = 0;
        } else {
          __nanosleep(20);
          if ((++polls & 255u) == 0 && globaltimer() - t_last > kWaitLimitNs) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) status_set(status, TV_E_TIMEOUT);
      // loads still in flight land before the CTA leaves (every load issued is
      // waited for by an MMA, except after a timeout)
      for (int j = (ns > 0 ? ns : 0); j < kiss; ++j) mbar_wait(&k_full[j & 1], (uint32_t)(j >> 1) & 1u);
      for (int j = no; j < viss; ++j) mbar_wait(&v_full[j & 1], (uint32_t)(j >> 1) & 1u);
      if (!qready) mbar_wait(q_land, 0);
      // and every MMA issued is done before TMEM is released
      if (no > 0) mbar_wait(o_done, (uint32_t)(no - 1) & 1u);
      if (ns > 0) mbar_wait(&s_full[(ns - 1) & 1], (uint32_t)((ns - 1) >> 1) & 1u);
    } else if (issuer) {
      for (int j = 0; j < 2 && j < T; ++j) {   // loads already issued land before the CTA leaves
        if ((pre >> j) & 1u) mbar_wait(&k_full[j & 1], 0);
        mbar_wait(&v_full[j & 1], 0);
      }
      mbar_wait(q_land, 0);
    }
  } else if (run) {
    // ---------------- softmax / epilogue (warps 0-15) ----------------
    // warp (quarter qd, slice cs): TMEM lanes 32 qd .. 32 qd + 31, i.e. key kl
    // of each tile in S^T and dimension kl in O^T, and the 8-column query
    // chunks cs, cs + 4, cs + 8, ...
    const int qd = warp & 3, cs = warp >> 2;
    const int kl = qd * 32 + lane;
    const uint32_t lb = (uint32_t)(qd * 32) << 16;
    const int nu = ((NQ >> 3) - cs + kSlices - 1) / kSlices;   // chunks of this slice
    uint8_t* sQ = smem + L::OFF_Q;
    // query column c = local row c / G, head g G + c % G; zero past nq
    if (threadIdx.x < kNqMax) {
      const int c = threadIdx.x;
      s_qrow[c] = c < nq ? (row0 + c / G) * Hq + g * G + c % G : -1;
      s_canc[c] = c < nq ? s_anc[c / G] : 0u;
    }
    // query columns nq .. NQ-1 pad the MMA's N to a multiple of 16: zero (the
    // columns below nq arrive by TMA)
    for (int idx = threadIdx.x; idx < (NQ - nq) * (D / 8); idx += kAtSoftThreads) {
      const int c = nq + idx / (D / 8), e = idx % (D / 8);
      *reinterpret_cast<uint4*>(sQ + (e >> 3) * L::QSLAB + swz(c, e & 7)) = make_uint4(0u, 0u, 0u, 0u);
    }
    if constexpr (D == 64) {   // O^T is M = 128: dimensions 64..127 read a zero slab
      for (int idx = threadIdx.x; idx < 2 * kAtom / 16; idx += kAtSoftThreads) {
        const int st = idx / (kAtom / 16), e = idx % (kAtom / 16);
        reinterpret_cast<uint4*>(smem + L::OFF_V + st * L::KV_BYTES + kAtom)[e] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    for (int c = threadIdx.x; c < kNqMax; c += kAtSoftThreads) {
      s_m[0][c] = -INFINITY;
      s_negm[0][c] = INFINITY;
      s_alpha[c] = 1.f;
    }
    fence_async_smem();
    soft_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_full);

    // tree tile: bit 8u + j = key kl is an ancestor-or-self of column (cs + 4u) 8 + j's row
    uint64_t vis = 0;
    if (has_tree) {
      for (int u = 0; u < nu; ++u)
        for (int j = 0; j < 8; ++j) {
          const int c = (cs + kSlices * u) * 8 + j;
          if (kl < n && ((s_canc[c] >> kl) & 1u)) vis |= 1ull << (8 * u + j);
        }
    }

    float l[kCps][8];   // this key's share of each column sum, at the column's current offset
#pragma unroll
    for (int u = 0; u < kCps; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) l[u][j] = 0.f;
    const uint32_t tO = tmem + kColO + lb;
    int ver = 0;   // buffer of the current offsets (slice-uniform)
    bool ok = true;

    // One 128-key tile, compiled for this slice's chunk count NU and for
    // whether keys are masked (tree tile, ragged last tile), so that the
    // common tile carries no per-element mask or bound logic.
    auto tile = [&](auto nu_c, auto masked_c, int tl) {
      constexpr int NU = decltype(nu_c)::value;
      constexpr int NA = NU < 3 ? NU : 3;   // chunks of the first TMEM load wave
      constexpr bool MASKED = decltype(masked_c)::value;
      const int b = tl & 1;
      const bool tree_t = is_tree(tl);
      const int kvalid = tile_keys(tl);
      const bool kin = kl < kvalid;
      const uint32_t sb = tmem + (uint32_t)(b ? kColS1 : kColS0) + lb;
      // visible keys: bit j of chunk u's mask = column (cs + 4u) 8 + j sees key kl
      auto vis_mask = [&](int u) -> uint32_t {
        return tree_t ? (uint32_t)(vis >> (8 * u)) & 0xffu : (kin ? 0xffu : 0u);
      };
      // this thread's scores of chunks [U0, U0 + NW), one TMEM round trip, then
      // f(u, scores) for each chunk
      auto scores = [&](auto u0_c, auto nw_c, auto&& f) {
        constexpr int U0 = decltype(u0_c)::value, NW = decltype(nw_c)::value;
        if constexpr (NW > 0) {
          uint32_t sv[NW][8];
#pragma unroll
          for (int i = 0; i < NW; ++i) ld8(sb + (cs + kSlices * (U0 + i)) * 8, sv[i]);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < NW; ++i) f(U0 + i, sv[i]);
        }
      };
      auto all_scores = [&](auto&& f) {
        scores(std::integral_constant<int, 0>{}, std::integral_constant<int, NA>{}, f);
        scores(std::integral_constant<int, NA>{}, std::integral_constant<int, NU - NA>{}, f);
      };

      if (ok && !mbar_wait(&s_full[b], (uint32_t)(tl >> 1) & 1u)) ok = false;
      tc_fence_after();

      // Pass 1: the largest x = s scale - m of a visible key.  An offset must
      // move when an x passes 8 (on the first tile no offset is set): the
      // slice agrees on that with one barrier reduction, and only then are
      // the tile's column maxima taken.
      bool moved = tl == 0;
      if (!moved) {
        float xmax = -INFINITY;
        const float* negm = s_negm[ver];
        all_scores([&](int u, const uint32_t (&sv)[8]) {
          const int c0 = (cs + kSlices * u) * 8;
          const float4 m0 = *reinterpret_cast<const float4*>(&negm[c0]);
          const float4 m1 = *reinterpret_cast<const float4*>(&negm[c0 + 4]);
          const float nm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
          const uint32_t vm = MASKED ? vis_mask(u) : 0xffu;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float x = fmaf(__uint_as_float(sv[j]), scale_log2, nm[j]);
            if (!MASKED || ((vm >> j) & 1u)) xmax = fmaxf(xmax, x);
          }
        });
        moved = slice_any(xmax > kRescaleLog2, cs);
      }
      if (moved) {
        // the tile's column maxima over all 128 keys (raw scores)
        all_scores([&](int u, const uint32_t (&sv)[8]) {
          const uint32_t vm = MASKED ? vis_mask(u) : 0xffu;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float x = redux_max(((vm >> j) & 1u) ? __uint_as_float(sv[j]) : -INFINITY);
            if (lane == 0) s_red[qd][(cs + kSlices * u) * 8 + j] = x;
          }
        });
        slice_sync(cs);
        // one thread per column of the slice: its new offset and factor
        const int st = qd * 32 + lane;
        if (st < NU * 8) {
          const int c = (cs + kSlices * (st >> 3)) * 8 + (st & 7);
          const float cm = fmaxf(fmaxf(s_red[0][c], s_red[1][c]), fmaxf(s_red[2][c], s_red[3][c])) * scale_log2;
          const float mo = s_m[ver][c];
          const float mn = cm > mo + kRescaleLog2 ? cm : mo;
          s_m[ver ^ 1][c] = mn;
          s_negm[ver ^ 1][c] = -mn;
          s_alpha[c] = mn == mo ? 1.f : ex2(mo - mn);
        }
        slice_sync(cs);
        ver ^= 1;
        if (tl > 0) {   // the sums move to the new offsets
#pragma unroll
          for (int u = 0; u < NU; ++u) {
            const int c0 = (cs + kSlices * u) * 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) l[u][j] *= s_alpha[c0 + j];
          }
        }
      }

      // Pass 2: P = 2^(s scale - m) rounded to bf16, a chunk at a time (one
      // TMEM round trip each, which keeps the live scores to 8 registers);
      // the column sums add the rounded values, the weights O^T gets, so that
      // a key that dominates its column passes its V row through unchanged.
      // This pass overlaps O^T of the previous tile, which still reads P^T:
      // each chunk's P is parked in TMEM over the scores it came from (this
      // thread's lane, this slice's columns) until P^T is free.
      {
        const float* negm = s_negm[ver];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const int c0 = (cs + kSlices * u) * 8;
          uint32_t sv[8];
          ld8(sb + c0, sv);
          const float4 m0 = *reinterpret_cast<const float4*>(&negm[c0]);
          const float4 m1 = *reinterpret_cast<const float4*>(&negm[c0 + 4]);
          const float nm[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
          const uint32_t vm = MASKED ? vis_mask(u) : 0xffu;
          tmem_ld_wait();
          uint32_t pk[4];
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            float x0 = fmaf(__uint_as_float(sv[j]), scale_log2, nm[j]);
            float x1 = fmaf(__uint_as_float(sv[j + 1]), scale_log2, nm[j + 1]);
            if (MASKED && !((vm >> j) & 1u)) x0 = -INFINITY;
            if (MASKED && !((vm >> (j + 1)) & 1u)) x1 = -INFINITY;
            const __nv_bfloat162 pb = __floats2bfloat162_rn(ex2(x0), ex2(x1));
            pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
            l[u][j] += __uint_as_float(pk[j >> 1] << 16);
            l[u][j + 1] += __uint_as_float(pk[j >> 1] & 0xffff0000u);
          }
          st4(sb + c0, pk);
        }
        tmem_st_wait();
      }

      // keys past the tile's valid ones: zero their V rows so that 0 * V stays 0
      // whatever those slots hold (all softmax threads share the rows)
      if (MASKED && kvalid < 128) {
        if (ok && !mbar_wait(&v_full[b], (uint32_t)(tl >> 1) & 1u)) ok = false;
        uint8_t* vd = smem + L::OFF_V + b * L::KV_BYTES;
        const int per_row = (D / 64) * 8;
        for (int idx = threadIdx.x; idx < (128 - kvalid) * per_row; idx += kAtSoftThreads) {
          const int row = kvalid + idx / per_row, rem = idx % per_row;
          *reinterpret_cast<uint4*>(vd + (rem >> 3) * kAtom + row * 128 + (rem & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // P^T and O^T are free once O^T += V^T P^T of the previous tile is done
      if (tl > 0) {
        if (ok && !mbar_wait(o_done, (uint32_t)(tl - 1) & 1u)) ok = false;
        tc_fence_after();
        if (moved) {   // O^T columns (complete up to tile tl-1) move to the new offsets
#pragma unroll
          for (int u = 0; u < NU; ++u) {
            const int c0 = (cs + kSlices * u) * 8;
            uint32_t o[8];
            ld8(tO + c0, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * s_alpha[c0 + j]);
            st8(tO + c0, o);
          }
          tmem_st_wait();
        }
      }
      {   // the parked P into key kl's row of P^T (8 query columns = one 16-byte chunk)
        uint32_t pk[NU > 0 ? NU : 1][4];
#pragma unroll
        for (int u = 0; u < NU; ++u) ld4(sb + (cs + kSlices * u) * 8, pk[u]);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          const int k = cs + kSlices * u;
          *reinterpret_cast<uint4*>(smem + L::OFF_P + (k >> 3) * kAtom + swz(kl, k & 7)) =
              make_uint4(pk[u][0], pk[u][1], pk[u][2], pk[u][3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[b]);   // S^T[b] may take tile tl + 2
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    };
    using std::integral_constant;
    auto tile_nu = [&](auto nu_c, int tl) {
      const bool masked = is_tree(tl) || tile_keys(tl) < 128;
      if (masked) tile(nu_c, integral_constant<bool, true>{}, tl);
      else tile(nu_c, integral_constant<bool, false>{}, tl);
    };
    for (int tl = 0; tl < T; ++tl) {
      switch (nu) {   // slice-uniform
        case 5: tile_nu(integral_constant<int, 5>{}, tl); break;
        case 4: tile_nu(integral_constant<int, 4>{}, tl); break;
        case 3: tile_nu(integral_constant<int, 3>{}, tl); break;
        case 2: tile_nu(integral_constant<int, 2>{}, tl); break;
        case 1: tile_nu(integral_constant<int, 1>{}, tl); break;
        default: tile_nu(integral_constant<int, 0>{}, tl); break;
      }
    }

    // ---- epilogue: unnormalised O, offsets and sums of this chunk --------------
    // Column sums over the 128 keys while the last O^T MMA runs.  In each warp
    // a reduce-scatter over its 32 keys: the 40 sums of a lane are halved
    // three times (lane bits 4, 3, 2; the half a lane keeps follows its bit),
    // then the five left are summed over lane bits 1 and 0; so lane L ends with
    // the warp's sums of entries 20 b4 + 10 b3 + 5 b2 + k, k < 5, of its
    // [chunk u][column j] list.  The four lane quarters of a slice then meet
    // in s_red.
    {
      const uint32_t b4 = (lane >> 4) & 1u, b3 = (lane >> 3) & 1u, b2 = (lane >> 2) & 1u;
      float a20[20], a10[10], a5[5];
#pragma unroll
      for (int k = 0; k < 20; ++k) {
        const float lo = l[k / 8][k % 8], hi = l[(20 + k) / 8][(20 + k) % 8];
        a20[k] = (b4 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b4 ? lo : hi, 16);
      }
#pragma unroll
      for (int k = 0; k < 10; ++k)
        a10[k] = (b3 ? a20[10 + k] : a20[k]) + __shfl_xor_sync(0xffffffffu, b3 ? a20[k] : a20[10 + k], 8);
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        a5[k] = (b2 ? a10[5 + k] : a10[k]) + __shfl_xor_sync(0xffffffffu, b2 ? a10[k] : a10[5 + k], 4);
        a5[k] += __shfl_xor_sync(0xffffffffu, a5[k], 2);
        a5[k] += __shfl_xor_sync(0xffffffffu, a5[k], 1);
      }
      if ((lane & 3) == 0) {
#pragma unroll
        for (int k = 0; k < 5; ++k) {
          const int e = (int)(20 * b4 + 10 * b3 + 5 * b2) + k;   // entry: chunk e / 8, column e % 8
          if (e / 8 < nu) s_red[qd][(cs + kSlices * (e / 8)) * 8 + e % 8] = a5[k];
        }
      }
    }
    slice_sync(cs);
    // one thread per column of the slice: the column's sum over the four quarters
    const int own = qd * 32 + lane;
    const int c_own = own < nu * 8 ? (cs + kSlices * (own >> 3)) * 8 + (own & 7) : -1;
    const float l_own = c_own >= 0 ? (s_red[0][c_own] + s_red[1][c_own]) + (s_red[2][c_own] + s_red[3][c_own]) : 0.f;

    if (ok && !mbar_wait(o_done, (uint32_t)(T - 1) & 1u)) ok = false;
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
      // O^T row kl (dimension kl) of this thread's columns, stored straight from
      // the registers: for one column the warp writes 32 consecutive floats
      uint32_t o[kCps][8];
#pragma unroll
      for (int u = 0; u < kCps; ++u)
        if (u < nu) ld8(tO + (cs + kSlices * u) * 8, o[u]);
      tmem_ld_wait();
      if (kl < D) {
#pragma unroll
        for (int u = 0; u < kCps; ++u) {
          if (u < nu) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int qr = s_qrow[(cs + kSlices * u) * 8 + j];
              if (qr >= 0) part_o[((size_t)qr * kChunkSlots + chunk) * D + kl] = __uint_as_float(o[u][j]);
            }
          }
        }
      }
      if (c_own >= 0 && s_qrow[c_own] >= 0) {
        const size_t base = (size_t)s_qrow[c_own] * kChunkSlots + chunk;
        part_ml[base * 2] = s_m[ver][c_own];
        part_ml[base * 2 + 1] = l_own;
      }
    } else if (lane == 0) {
      status_set(status, TV_E_TIMEOUT);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpIssue) {
    tc_fence_after();
    tmem_dealloc(tmem, kAtTmemCols);
  }
}

// out[row][h*D + d] = bf16( sum_c o_c[d] 2^(m_c - M) / sum_c l_c 2^(m_c - M) ),
// chunks in order.  One warp per (row, query head), lane i holding dimensions
// 4i .. 4i + 3 (a chunk's partial is one 16-byte load per lane) and the offset
// and sum of chunks i and i + 32.  The row's chunk count follows from the
// kernel parameters, so the partials are requested right after the wait, up
// to kMergeBatch chunks at a time.
constexpr int kMergeWarps = 2;
constexpr int kMergeBatch = 20;
static_assert(kChunkSlots <= 64, "a lane holds at most two chunks' offsets");

__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(ReqTable t, int Hq, int D, int chunk_target,
                                                                      const float* part_ml, const float* part_o,
                                                                      __nv_bfloat16* out, const int32_t* status) {
  pdl_trigger();   // the O GEMM may start streaming its weights now
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x * kMergeWarps + warp;
  const int row = pair / Hq, hq = pair % Hq;
  if (row >= t.total_rows) {   // warp-uniform; the rest of the block does not synchronise
    pdl_wait();
    return;
  }
  int r = 0;
  while (r + 1 < t.n_req && t.row_off[r + 1] <= row) ++r;
  const int nch = attn_plan(t.ctx[r], chunk_target).n_chunks;
  const size_t base = ((size_t)row * Hq + hq) * kChunkSlots;
  const int nv = D / 4;   // 16-byte pieces of one chunk's partial
  const bool dl = lane < nv;
  pdl_wait();
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + base;
  float2 ml0 = make_float2(-INFINITY, 0.f), ml1 = make_float2(-INFINITY, 0.f);
  if (lane < nch) ml0 = __ldcg(ml + lane);
  if (lane + 32 < nch) ml1 = __ldcg(ml + lane + 32);
  const bool skip = status_get(status) != 0;
  const float4* po = reinterpret_cast<const float4*>(part_o + base * D) + lane;
  // the first batch of partials is requested with the offsets, before the
  // shuffles that need them
  float4 v[kMergeBatch];
#pragma unroll
  for (int i = 0; i < kMergeBatch; ++i)
    v[i] = dl && i < nch ? __ldcg(po + (size_t)i * nv) : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = fmaxf(ml0.x, ml1.x);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < nch; c0 += kMergeBatch) {   // a batch of loads in flight, then its terms in order
    if (c0 > 0) {
#pragma unroll
      for (int i = 0; i < kMergeBatch; ++i)
        v[i] = dl && c0 + i < nch ? __ldcg(po + (size_t)(c0 + i) * nv) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < kMergeBatch; ++i) {
      const int c = c0 + i;
      if (c < nch) {
        const float mc = __shfl_sync(0xffffffffu, c < 32 ? ml0.x : ml1.x, c & 31);
        const float lc = __shfl_sync(0xffffffffu, c < 32 ? ml0.y : ml1.y, c & 31);
        const float w = exp2f(mc - M);   // offsets are in log2 units
        L = fmaf(lc, w, L);
        O.x = fmaf(v[i].x, w, O.x);
        O.y = fmaf(v[i].y, w, O.y);
        O.z = fmaf(v[i].z, w, O.z);
        O.w = fmaf(v[i].w, w, O.w);
      }
    }
  }
  if (skip || !dl) return;
  __nv_bfloat162 lo = __floats2bfloat162_rn(O.x / L, O.y / L), hi = __floats2bfloat162_rn(O.z / L, O.w / L);
  uint2 pk;
  pk.x = *reinterpret_cast<const uint32_t*>(&lo);
  pk.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out + (size_t)row * Hq * D + (size_t)hq * D + 4 * lane) = pk;
}

template <int D>
int launch_attention_d(const ReqTable& t, const tv_dims& dm, const LayerBufs& b, int sms, int32_t* status,
                       cudaStream_t st) {
  AttnMaps maps;
  memset(&maps, 0, sizeof(maps));
  const int target = attn_chunk_target(sms, dm.n_kv_heads);
  int nch_max = 0;
  for (int r = 0; r < t.n_req; ++r) {
    const int rows = dm.n_kv_heads * t.capacity[r];
    int rc = make_tmap_bf16(&maps.k[r], t.k[r], D, rows, 64, 128);
    if (rc) return rc;
    rc = make_tmap_bf16(&maps.v[r], t.v[r], D, rows, 64, 128);
    if (rc) return rc;
    rc = make_tmap_bf16_3d(&maps.q[r], b.q, D, dm.n_q_heads, t.total_rows, 64, dm.n_q_heads / dm.n_kv_heads,
                           t.n[r]);
    if (rc) return rc;
    nch_max = max(nch_max, attn_plan(t.ctx[r], target).n_chunks);
  }
  const size_t smem = AtSmem<D>::BYTES;
  static std::atomic<bool> attr[64];
  if (ensure_smem_limit(attn_tc_kernel<D>, smem, attr)) return TV_E_CUDA;
  dim3 grid(nch_max, dm.n_kv_heads, t.n_req);
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));   // log2(e) / sqrt(D)
  int rc = launch_pdl(attn_tc_kernel<D>, grid, dim3(kAtThreads), smem, st, maps, t, (const RowMeta*)b.meta,
                      (const __nv_bfloat16*)b.q, dm.n_q_heads, dm.n_kv_heads, target, scale_log2, b.attn_ml,
                      b.attn_o, status);
  if (rc) return rc;
  const int pairs = t.total_rows * dm.n_q_heads;
  return launch_pdl(attn_merge_kernel, dim3((pairs + kMergeWarps - 1) / kMergeWarps), dim3(kMergeWarps * 32), 0, st, t,
                    dm.n_q_heads, D, target, (const float*)b.attn_ml, (const float*)b.attn_o, b.attn,
                    (const int32_t*)status);
}

}  // namespace

int launch_attention(const ReqTable& t, const tv_dims& d, const LayerBufs& b, int sms, int32_t* status,
                     cudaStream_t st) {
  if (d.head_dim == 128) return launch_attention_d<128>(t, d, b, sms, status, st);
  if (d.head_dim == 64) return launch_attention_d<64>(t, d, b, sms, status, st);
  return TV_E_UNSUPPORTED;
}

}  // namespace tv
