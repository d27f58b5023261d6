// Skinny GEMM on the 5th-generation tensor cores: out = W * X^T for a weight W
// [M][K] (bf16, K-major, streamed from HBM once) and at most 32 activation rows
// X [rows][K] (bf16).  Used for the LM head (fused fp32 logits + per-row
// argmax / top-2 gap) and for the QKV / O projections (split-K fp32 partials,
// summed in a fixed order by the finalize kernels).
//
// Reduction order.  "Every matrix-product kernel fixes its reduction order by
// the weight's shape and never by the row count" [Exactness, §The one
// exception: near ties]: the activation rows always fill a fixed MMA N of 32
// (missing rows read as zeros from the TMA's out-of-bounds fill), the K loop of
// every tile runs in increasing k, and the split-K partition is a function of
// (M, K) alone.  A row's outputs therefore do not depend on how many other rows
// share the pass [Exactness, §Parallel requests].
//
// Design (one CTA per SM, persistent over tiles):
//   - swap-AB: the weight is the MMA's A operand (M = 128 weight rows per tile
//     on the TMEM lanes), the activations are B (N = 32 columns), so the weight
//     stream needs no padding and the tiny operand is the one that is re-read
//     (from L2).
//   - warp 0 issues TMA loads of 128x64 weight tiles and 32x64 activation tiles
//     (128-byte swizzle) into an 8-stage shared-memory ring, weights with an
//     L2 evict-first hint;
//   - warp 1 owns the TMEM allocation and issues tcgen05.mma (M128 N32 K16,
//     bf16 in, fp32 accumulate in TMEM) from one thread; tcgen05.commit frees a
//     smem stage when its MMAs are done;
//   - warps 2-5 are the epilogue: each reads its 32 TMEM lanes with
//     tcgen05.ld while the MMA fills the other of two accumulators.
//   - LM head: the epilogue writes the fp32 logits and keeps a running per-row
//     top-2; the last CTA to finish (an atomic counter, no spin) merges the
//     per-CTA top-2 in CTA order and writes argmax and gap.
#include <climits>

#include "tv_common.cuh"
#include "tv_gemm.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr int BM = 128;
constexpr int BN = 32;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int THREADS = 192;
constexpr int TMEM_COLS = 64;
constexpr int EPI_STRIDE = 33;
constexpr int kPartialStages = 8;
constexpr size_t SMEM_BAR = 1024;
constexpr size_t SMEM_EPI = 4 * 32 * EPI_STRIDE * sizeof(float);
constexpr int kMergeWarpsHead = THREADS / 32;   // the last head CTA merges with all its warps
constexpr size_t SMEM_T2 = kMergeWarpsHead * 32 * sizeof(Top2);
// Ring depth and shared memory by mode.  The head streams 1.5 GB with eight
// 16 KB weight stages (six and ten were slower); the split-K GEMMs measured
// the same with eight and eleven; they need no top-2 tables.
template <int MODE>
struct GemmCfg {
  static constexpr int STAGES = MODE == GEMM_HEAD ? 8 : kPartialStages;
  static constexpr size_t TILES = (size_t)STAGES * (A_BYTES + B_BYTES);
  static constexpr size_t BYTES = 1024 + TILES + SMEM_BAR + (MODE == GEMM_HEAD ? SMEM_EPI + SMEM_T2 : 0);
};

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                       GemmParams p) {
  constexpr int STAGES = GemmCfg<MODE>::STAGES;
  constexpr size_t SMEM_TILES = GemmCfg<MODE>::TILES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + (size_t)STAGES * A_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + SMEM_TILES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* s_status = reinterpret_cast<int*>(tmem_slot + 1);
  float* epi = reinterpret_cast<float*>(smem + SMEM_TILES + SMEM_BAR);
  Top2* t2s = reinterpret_cast<Top2*>(epi + 4 * 32 * EPI_STRIDE);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- set-up: nothing here reads data written by an earlier kernel ----------
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    prefetch_tmap(&mapA);
    prefetch_tmap(&mapB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();

  const int KB = p.K / BK;
  // this CTA's work items in order: units blockIdx.x + i * gridDim.x, their k-blocks
  auto unit_kb = [&](int u, int& kb0, int& kb1) {
    kb0 = (u % p.splits) * p.kb_per_split;
    kb1 = min(KB, kb0 + p.kb_per_split);
  };

  // The producer starts streaming weights (never written by any kernel) into
  // the first stages before the previous kernel has finished.
  int pre = 0;
  int pre_u = blockIdx.x, pre_kb = 0, pre_kb1 = 0;
  uint64_t pol_w = 0, pol_x = 0;
  // weight tile (m-tile mt, k-block kb): a box of the row-major matrix, or
  // the tile's own contiguous 16 KB of the packed copy
  auto load_a = [&](uint8_t* dst, uint64_t* bar, int mt, int kb) {
    if (p.packed) tma_load_2d(dst, &mapA, bar, 0, (mt * KB + kb) * BM, pol_w);
    else tma_load_2d(dst, &mapA, bar, kb * BK, mt * BM, pol_w);
  };
  if (warp == 0 && lane == 0) {
    pol_w = policy_evict_first();
    pol_x = policy_evict_last();
    if (pre_u < p.n_units) unit_kb(pre_u, pre_kb, pre_kb1);
    int u = pre_u, kb = pre_kb, kb1 = pre_kb1;
    while (pre < STAGES && u < p.n_units) {
      mbar_expect_tx(&full[pre], A_BYTES);
      load_a(sA + (size_t)pre * A_BYTES, &full[pre], u / p.splits, kb);
      ++pre;
      if (++kb >= kb1) {
        u += gridDim.x;
        if (u < p.n_units) unit_kb(u, kb, kb1);
      }
    }
  }

  pdl_wait();
  if (threadIdx.x == 0) *s_status = status_get(p.status);
  __syncthreads();
  if (*s_status != 0) {
    if (warp == 0 && lane == 0) {   // let the weight loads already in flight land
      for (int s = 0; s < pre; ++s) {
        mbar_arrive(&full[s]);
        mbar_wait(&full[s], 0);
      }
    }
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, TMEM_COLS);
    }
    return;
  }

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t armed = 0;      // bit s: stage s was armed at least once
      uint32_t last_par = 0;   // bit s: parity of stage s's last armed phase
      // activations of the pre-issued stages
      int u = pre_u, kb = pre_kb, kb1 = pre_kb1;
      for (int s = 0; s < pre; ++s) {
        mbar_arrive_expect_tx(&full[s], B_BYTES);
        tma_load_2d(sB + (size_t)s * B_BYTES, &mapB, &full[s], kb * BK, 0, pol_x);
        armed |= 1u << s;
        if (++kb >= kb1) {
          u += gridDim.x;
          if (u < p.n_units) unit_kb(u, kb, kb1);
        }
      }
      int stage = pre % STAGES;
      uint32_t phase = pre == STAGES ? 1u : 0u;
      bool ok = true;
      while (u < p.n_units && ok) {
        if (!mbar_wait(&empty[stage], phase ^ 1u)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[stage], A_BYTES + B_BYTES);
        load_a(sA + (size_t)stage * A_BYTES, &full[stage], u / p.splits, kb);
        tma_load_2d(sB + (size_t)stage * B_BYTES, &mapB, &full[stage], kb * BK, 0, pol_x);
        armed |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
        if (++kb >= kb1) {
          u += gridDim.x;
          if (u < p.n_units) unit_kb(u, kb, kb1);
        }
      }
      if (!ok) status_set(p.status, TV_E_TIMEOUT);
      // every load this thread issued has landed before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if (armed & (1u << s)) mbar_wait(&full[s], (last_par >> s) & 1u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t aphase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.n_units && ok; u += gridDim.x) {
        const int sp = u % p.splits;
        const int kb0 = sp * p.kb_per_split;
        const int kb1 = min(KB, kb0 + p.kb_per_split);
        if (!mbar_wait(&tempty[acc], aphase ^ 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_k_sw128(smem_u32(sA + (size_t)stage * A_BYTES));
          const uint64_t bdesc = sdesc_k_sw128(smem_u32(sB + (size_t)stage * B_BYTES));
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)   // +32 bytes along K inside the swizzled row
            umma_bf16(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          aphase ^= 1u;
        }
      }
      if (!ok) status_set(p.status, TV_E_TIMEOUT);
      // all MMAs issued by this thread are complete before TMEM is released
      umma_commit(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;        // TMEM lane quarter this warp may access
    const int ew = warp - 2;
    float* mys = epi + ew * 32 * EPI_STRIDE;
    Top2 best;
    best.m1 = -INFINITY;
    best.i1 = INT_MAX;
    best.m2 = -INFINITY;
    best.pad = 0;
    int acc = 0;
    uint32_t aphase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.n_units; u += gridDim.x) {
      const int mt = u / p.splits, sp = u % p.splits;
      if (!mbar_wait(&tfull[acc], aphase)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r[32];
      tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN), r);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == 2) {
        acc = 0;
        aphase ^= 1u;
      }
      const int m0 = mt * BM + q * 32;
      const int m = m0 + lane;
      if (MODE == GEMM_PARTIAL) {
        if (m < p.M) {
          float* dst = p.out + (size_t)sp * kMaxRows * p.M + m;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < p.n_rows) dst[(size_t)j * p.M] = __uint_as_float(r[j]);
        }
      } else {
        if (m < p.M) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < p.n_rows) p.out[(size_t)j * p.M + m] = __uint_as_float(r[j]);
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) mys[lane * EPI_STRIDE + j] = m < p.M ? __uint_as_float(r[j]) : -INFINITY;
        __syncwarp();
        // lane j scans column j (activation row j) over this warp's 32 weight rows
        for (int l = 0; l < 32; ++l) top2_push(best, mys[l * EPI_STRIDE + lane], m0 + l);
        __syncwarp();
      }
    }
    if (!ok) status_set(p.status, TV_E_TIMEOUT);
    if (MODE == GEMM_HEAD) t2s[ew * 32 + lane] = best;
  }

  __syncthreads();

  if (MODE == GEMM_HEAD) {
    // this CTA's best per activation row goes out; the CTA that finishes last
    // merges every CTA's with all six of its warps (warp w: CTAs w, w + 6, ...,
    // every load in flight at once for a grid of up to 156), then warp 2
    // merges the six.
    // The merge keeps the largest value and the lowest index among equal
    // ones, so its order does not change the result.
    __shared__ int s_last;
    if (warp == 2) {
      Top2 b = t2s[lane];
      for (int e = 1; e < 4; ++e) top2_merge(b, t2s[e * 32 + lane]);
      p.top2_part[(size_t)blockIdx.x * 32 + lane] = b;
      __threadfence();
      unsigned prev = 0;
      if (lane == 0) prev = atomicAdd(p.done_counter, 1u);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (lane == 0) s_last = prev == gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      const unsigned ew = (unsigned)warp;
      Top2 g;
      g.m1 = -INFINITY;
      g.i1 = INT_MAX;
      g.m2 = -INFINITY;
      g.pad = 0;
      constexpr int kBatch = 26;
      for (unsigned c0 = ew; c0 < gridDim.x; c0 += kMergeWarpsHead * kBatch) {
        int4 raw[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const unsigned c = c0 + (unsigned)(kMergeWarpsHead * i);
          raw[i] = c < gridDim.x ? __ldcg(reinterpret_cast<const int4*>(p.top2_part + (size_t)c * 32 + lane))
                                 : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          if (c0 + (unsigned)(kMergeWarpsHead * i) < gridDim.x) {
            Top2 t;
            t.m1 = __int_as_float(raw[i].x);
            t.i1 = raw[i].y;
            t.m2 = __int_as_float(raw[i].z);
            t.pad = 0;
            top2_merge(g, t);
          }
        }
      }
      t2s[ew * 32 + lane] = g;
    }
    __syncthreads();
    if (s_last && warp == 2) {
      Top2 g = t2s[lane];
      for (int e = 1; e < kMergeWarpsHead; ++e) top2_merge(g, t2s[e * 32 + lane]);
      if (lane < p.n_rows) {
        p.argmax[lane] = g.i1;
        p.gap[lane] = g.m1 - g.m2;
      }
      if (lane == 0) *p.done_counter = 0u;
    }
  }

  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
GemmPlan plan_gemm(int M, int K, bool head) {
  GemmPlan pl;
  const int KB = K / BK;
  const int tiles = (M + BM - 1) / BM;
  if (head) {
    pl.splits = 1;
    pl.kb_per_split = KB;
  } else {
    // about two work units per SM of a 152-SM part; a constant, so the split
    // (and with it the summation order) depends on the weight shape only
    const int target_units = 304;
    int splits = target_units / tiles;
    if (splits < 1) splits = 1;
    if (splits > KB) splits = KB;
    if (splits > kMaxSplits) splits = kMaxSplits;
    pl.kb_per_split = (KB + splits - 1) / splits;
    pl.splits = (KB + pl.kb_per_split - 1) / pl.kb_per_split;
  }
  pl.n_units = tiles * pl.splits;
  return pl;
}

size_t gemm_smem_bytes() { return GemmCfg<GEMM_HEAD>::BYTES; }

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}
}  // namespace

int make_tmap_bf16(CUtensorMap* map, const void* base, int inner, int rows, int box_inner, int box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return TV_E_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (inner * 2) % 16 != 0) return TV_E_ARG;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TV_OK : TV_E_CUDA;
}

int make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d0, int d1, int d2, int b0, int b1, int b2) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return TV_E_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (d0 * 2) % 16 != 0) return TV_E_ARG;
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)d0 * 2, (cuuint64_t)d0 * d1 * 2};
  cuuint32_t box[3] = {(cuuint32_t)b0, (cuuint32_t)b1, (cuuint32_t)b2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? TV_OK : TV_E_CUDA;
}

int launch_gemm(int mode, const void* W, int M, int K, const void* X, int n_rows, const GemmPlan& pl,
                const GemmParams& base, int num_sms, cudaStream_t stream) {
  if (K % BK != 0 || n_rows < 1 || n_rows > kMaxRows) return TV_E_UNSUPPORTED;
  CUtensorMap mA, mB;
  const int m_tiles = (M + BM - 1) / BM;
  // packed: [m_tiles * (K / BK) * BM][BK], tile (mt, kb) at row (mt * K / BK + kb) * BM
  int rc = base.packed ? make_tmap_bf16(&mA, W, BK, m_tiles * (K / BK) * BM, BK, BM) : make_tmap_bf16(&mA, W, K, M, BK, BM);
  if (rc) return rc;
  rc = make_tmap_bf16(&mB, X, K, n_rows, BK, BN);
  if (rc) return rc;
  GemmParams p = base;
  p.M = M;
  p.K = K;
  p.n_rows = n_rows;
  p.splits = pl.splits;
  p.kb_per_split = pl.kb_per_split;
  p.n_units = pl.n_units;
  const int grid = pl.n_units < num_sms ? pl.n_units : num_sms;
  if (mode == GEMM_HEAD) {
    static std::atomic<bool> attr[64];
    constexpr size_t bytes = GemmCfg<GEMM_HEAD>::BYTES;
    if (ensure_smem_limit(gemm_skinny_kernel<GEMM_HEAD>, bytes, attr)) return TV_E_CUDA;
    return launch_pdl(gemm_skinny_kernel<GEMM_HEAD>, dim3(grid), dim3(THREADS), bytes, stream, mA, mB, p);
  } else {
    static std::atomic<bool> attr[64];
    constexpr size_t bytes = GemmCfg<GEMM_PARTIAL>::BYTES;
    if (ensure_smem_limit(gemm_skinny_kernel<GEMM_PARTIAL>, bytes, attr)) return TV_E_CUDA;
    return launch_pdl(gemm_skinny_kernel<GEMM_PARTIAL>, dim3(grid), dim3(THREADS), bytes, stream, mA, mB, p);
  }
}

// one thread per 16 bytes of the packed copy: tile t = mt * KB + kb, row r,
// 16-byte piece c of the tile's 128-byte row
__global__ void pack_weight_kernel(const uint4* __restrict__ w, int rows, int cols, uint4* __restrict__ packed,
                                   size_t total) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int c = (int)(i & 7);
  const size_t rt = i >> 3;          // row of the packed view
  const int r = (int)(rt % BM);
  const size_t tile = rt / BM;
  const int KB = cols / BK;
  const int kb = (int)(tile % KB);
  const size_t row = (tile / KB) * BM + r;
  packed[i] = row < (size_t)rows ? w[(row * cols + (size_t)kb * BK) / 8 + c] : make_uint4(0u, 0u, 0u, 0u);
}

int launch_pack_weight(const void* W, int rows, int cols, void* packed, cudaStream_t stream) {
  if (rows < 1 || cols < BK || cols % BK != 0) return TV_E_ARG;
  const size_t total = (size_t)((rows + BM - 1) / BM) * BM * cols / 8;
  const unsigned blocks = (unsigned)((total + 255) / 256);
  pack_weight_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const uint4*>(W), rows, cols,
                                                 reinterpret_cast<uint4*>(packed), total);
  return cudaGetLastError() == cudaSuccess ? TV_OK : TV_E_CUDA;
}

}  // namespace tv
