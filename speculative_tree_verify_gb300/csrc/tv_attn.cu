// Tree-masked GQA attention over the cached context plus the tree rows, on the
// 5th-generation tensor cores.
//
// Row i, query head h attends to the cached slots [0, ctx) and to the tree
// slots ctx + a for every a in anc(i) (its ancestors and itself): "give each
// node an attention mask of its ancestors and a position equal to its depth"
// [Drafters and tree verify, §Tree verify through recurrent layers].  The
// positions were applied by RoPE before the keys were written.
//
// Split-context (flash-decoding) layout: one CTA per (request, KV head, query
// tile, context chunk) plus one per (request, KV head, query tile) for the
// tree keys.  A query tile is 128 query vectors = the request's rows x the GQA
// heads of one KV head, so every K/V byte is read once per query tile.  The
// chunk length is a function of ctx only (a multiple of 128 keys, at most 32
// chunks), and the merge kernel combines the partials (max, sum, unnormalised
// output) in chunk order, then the tree slot: a row's result is the same
// whatever the other rows are.
//
// Per CTA, for each 128-key tile of its chunk:
//   S = Q K^T      tcgen05.mma M128 (queries) N128 (keys) K16, fp32 in TMEM;
//                  Q staged once into 128B-swizzled smem, K by TMA (K-major)
//   softmax        16 warps: four per TMEM lane quarter, each thread one query
//                  row x 32 keys; scores scaled by log2(e)/sqrt(D), masked
//                  (keys past the chunk; ancestors for the tree tile), row max
//                  exchanged in smem, online max / sum in fp32, P = 2^(x - m)
//                  (SFU ex2) rounded to bf16 into swizzled smem, O in TMEM rescaled when
//                  the max grows; quarters without a valid query row skip
//   O += P V       tcgen05.mma M128 N=D K16, V straight from its TMA layout as
//                  an MN-major operand
// K and V tiles each have a two-stage TMA ring, refilled two tiles ahead.
#include <cmath>
#include <cstring>

#include "tv_common.cuh"
#include "tv_gemm.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr int kSlices = 4;                          // softmax warps per TMEM lane quarter
constexpr int kKeysPer = 128 / kSlices;             // keys of a 128-key tile per softmax thread
constexpr int kAtSoftWarps = 4 * kSlices;           // 16
constexpr int kAtSoftThreads = kAtSoftWarps * 32;   // 512
constexpr int kAtThreads = kAtSoftThreads + 32;     // + one warp: TMEM owner, TMA and MMA issue
constexpr int kAtTmemCols = 512;  // S double buffer: columns [0, 128) and [128, 256); O: [256, 256 + D)
constexpr int kAtom = 128 * 128;  // bytes of one 128-row x 128-byte swizzled slab
constexpr float kRescaleLog2 = 8.f;   // O and l are rescaled only when the row max grows by more than 2^8

struct AttnMaps {
  CUtensorMap k[kMaxReq];   // per request: [Hkv * capacity][D] bf16, box 64 x 128, 128B swizzle
  CUtensorMap v[kMaxReq];
};

template <int D>
struct AtSmem {
  static constexpr int SLABS = D / 64;               // 64-element slabs along D
  static constexpr int Q_BYTES = SLABS * kAtom;      // 128 queries x D
  static constexpr int KV_BYTES = SLABS * kAtom;     // 128 keys x D
  static constexpr int P_BYTES = 2 * kAtom;          // 128 queries x 128 keys
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + Q_BYTES;     // K stage s at OFF_KV + s KV_BYTES, V stage s at OFF_KV + (2 + s) KV_BYTES
  static constexpr int OFF_P = OFF_KV + 4 * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr size_t BYTES = 1024 + OFF_BAR + 256;
};

// 128B-swizzle smem descriptor with explicit leading / stride byte offsets.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// byte offset of 16-byte chunk c of row r inside a 128-row x 128-byte slab
// stored with the 128-byte swizzle (chunk index XOR row mod 8)
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// 2^x with the SFU's approximate base-2 exponential (PTX ex2.approx.ftz;
// about 2^-22 relative error, 2^-inf = 0)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// the four warps of one TMEM lane quarter (named barriers 1..4)
__device__ __forceinline__ void quarter_barrier(int qd) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + qd), "n"(kSlices * 32) : "memory");
}
__device__ __forceinline__ void soft_barrier() { asm volatile("bar.sync 5, %0;" ::"n"(kAtSoftThreads) : "memory"); }

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Columns [OFF, OFF + 32) (or + 16) of a register array from / to 32 (16)
// consecutive TMEM columns of this thread's lane.  Constant indices keep the
// arrays in registers.
template <int OFF, int N>
__device__ __forceinline__ void ld32_at(uint32_t taddr, uint32_t (&r)[N]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]), "=r"(r[OFF + 4]), "=r"(r[OFF + 5]), "=r"(r[OFF + 6]), "=r"(r[OFF + 7]), "=r"(r[OFF + 8]), "=r"(r[OFF + 9]), "=r"(r[OFF + 10]), "=r"(r[OFF + 11]), "=r"(r[OFF + 12]), "=r"(r[OFF + 13]), "=r"(r[OFF + 14]), "=r"(r[OFF + 15]), "=r"(r[OFF + 16]), "=r"(r[OFF + 17]), "=r"(r[OFF + 18]), "=r"(r[OFF + 19]), "=r"(r[OFF + 20]), "=r"(r[OFF + 21]), "=r"(r[OFF + 22]), "=r"(r[OFF + 23]), "=r"(r[OFF + 24]), "=r"(r[OFF + 25]), "=r"(r[OFF + 26]), "=r"(r[OFF + 27]), "=r"(r[OFF + 28]), "=r"(r[OFF + 29]), "=r"(r[OFF + 30]), "=r"(r[OFF + 31])
               : "r"(taddr));
}
template <int OFF, int N>
__device__ __forceinline__ void ld16_at(uint32_t taddr, uint32_t (&r)[N]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
               : "=r"(r[OFF + 0]), "=r"(r[OFF + 1]), "=r"(r[OFF + 2]), "=r"(r[OFF + 3]), "=r"(r[OFF + 4]), "=r"(r[OFF + 5]), "=r"(r[OFF + 6]), "=r"(r[OFF + 7]), "=r"(r[OFF + 8]), "=r"(r[OFF + 9]), "=r"(r[OFF + 10]), "=r"(r[OFF + 11]), "=r"(r[OFF + 12]), "=r"(r[OFF + 13]), "=r"(r[OFF + 14]), "=r"(r[OFF + 15])
               : "r"(taddr));
}
template <int OFF, int N>
__device__ __forceinline__ void st32_at(uint32_t taddr, const uint32_t (&r)[N]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr), "r"(r[OFF + 0]), "r"(r[OFF + 1]), "r"(r[OFF + 2]), "r"(r[OFF + 3]), "r"(r[OFF + 4]), "r"(r[OFF + 5]), "r"(r[OFF + 6]), "r"(r[OFF + 7]), "r"(r[OFF + 8]), "r"(r[OFF + 9]), "r"(r[OFF + 10]), "r"(r[OFF + 11]), "r"(r[OFF + 12]), "r"(r[OFF + 13]), "r"(r[OFF + 14]), "r"(r[OFF + 15]), "r"(r[OFF + 16]), "r"(r[OFF + 17]), "r"(r[OFF + 18]), "r"(r[OFF + 19]), "r"(r[OFF + 20]), "r"(r[OFF + 21]), "r"(r[OFF + 22]), "r"(r[OFF + 23]), "r"(r[OFF + 24]), "r"(r[OFF + 25]), "r"(r[OFF + 26]), "r"(r[OFF + 27]), "r"(r[OFF + 28]), "r"(r[OFF + 29]), "r"(r[OFF + 30]), "r"(r[OFF + 31])
               : "memory");
}
template <int OFF, int N>
__device__ __forceinline__ void st16_at(uint32_t taddr, const uint32_t (&r)[N]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr), "r"(r[OFF + 0]), "r"(r[OFF + 1]), "r"(r[OFF + 2]), "r"(r[OFF + 3]), "r"(r[OFF + 4]), "r"(r[OFF + 5]), "r"(r[OFF + 6]), "r"(r[OFF + 7]), "r"(r[OFF + 8]), "r"(r[OFF + 9]), "r"(r[OFF + 10]), "r"(r[OFF + 11]), "r"(r[OFF + 12]), "r"(r[OFF + 13]), "r"(r[OFF + 14]), "r"(r[OFF + 15])
               : "memory");
}

// NC consecutive 32-bit TMEM columns of this thread's lane (NC = 16, 32 or 64)
template <int NC>
__device__ __forceinline__ void cols_ld(uint32_t taddr, uint32_t (&r)[NC]) {
  if constexpr (NC == 16) {
    ld16_at<0>(taddr, r);
  } else {
    ld32_at<0>(taddr, r);
    if constexpr (NC == 64) ld32_at<32>(taddr + 32, r);
  }
}
template <int NC>
__device__ __forceinline__ void cols_st(uint32_t taddr, const uint32_t (&r)[NC]) {
  if constexpr (NC == 16) {
    st16_at<0>(taddr, r);
  } else {
    st32_at<0>(taddr, r);
    if constexpr (NC == 64) st32_at<32>(taddr + 32, r);
  }
}

// grid (query tiles, chunks + 1, requests x KV heads); the query tiles of one
// chunk are neighbours in launch order, so their K/V tiles meet in L2.
//
// Pipeline over the chunk's 128-key tiles t (issuer = one thread of warp 16):
//   S[t % 2] = Q K_t^T            as soon as K_t has landed and S[t % 2] is free
//   softmax(t) by warps 0-15      P_t built in registers; stored to smem P once
//                                 O += P_{t-1} V_{t-1} is done; O rescaled if needed
//   O += P_t V_t                  after softmax(t); frees K/V stage t % 2
// so S(t+1) overlaps softmax(t), and the TMA of tile t+2 overlaps both.
template <int D>
__global__ void __launch_bounds__(kAtThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnMaps maps, ReqTable t, const RowMeta* meta, const __nv_bfloat16* q,
                   int Hq, int Hkv, float scale_log2, float* part_ml, float* part_o, int32_t* status) {
  using L = AtSmem<D>;
  constexpr int OC = D / kSlices;   // O columns per softmax thread
  static_assert(OC % 16 == 0 && kKeysPer % 32 == 0, "TMEM accesses come in 16- and 32-column pieces");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);    // [2] K tile landed
  uint64_t* k_free = k_full + 2;                                          // [2] S MMA of the K stage done
  uint64_t* v_full = k_free + 2;                                          // [2] V tile landed
  uint64_t* v_free = v_full + 2;                                          // [2] O MMA of the V stage done
  uint64_t* s_full = v_free + 2;                                          // [2] S MMA done
  uint64_t* p_full = s_full + 2;                                          // [2] softmax done (16 warps)
  uint64_t* o_ready = p_full + 2;                                         // O MMA of a tile done
  uint64_t* q_full = o_ready + 1;                                         // queries staged (16 warps)
  uint64_t* drain = q_full + 1;                                           // every MMA of the CTA done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* s_stat = reinterpret_cast<int*>(tmem_slot + 1);
  __shared__ uint32_t s_anc[32];
  __shared__ float s_red[2][kSlices][128];   // partial row maxima, double-buffered by tile parity
  __shared__ float s_l[kSlices][128];        // partial row sums

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, slot_x = blockIdx.y, g = blockIdx.z % Hkv, r = blockIdx.z / Hkv;

  // ---- structural early exits (kernel parameters only) ------------------------
  const int ctx = t.ctx[r], n = t.n[r], row0 = t.row_off[r], cap = t.capacity[r];
  const int nch = attn_n_chunks(ctx);
  const bool tree = slot_x == (int)gridDim.y - 1;
  const int G = Hq / Hkv;
  const int nq = n * G, q0 = qt * 128;
  if ((!tree && slot_x >= nch) || q0 >= nq) {
    pdl_wait();
    pdl_trigger();
    return;
  }
  const int slot = tree ? kTreeSlot : slot_x;
  int key0, nkeys;
  if (tree) {
    key0 = ctx;
    nkeys = n;
  } else {
    const int ch = attn_chunk_len(ctx);
    key0 = slot * ch;
    nkeys = min(ch, ctx - key0);
  }
  const int T = (nkeys + 127) / 128;

  // ---- set-up --------------------------------------------------------------------
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&k_full[b], 1);
      mbar_init(&k_free[b], 1);
      mbar_init(&v_full[b], 1);
      mbar_init(&v_free[b], 1);
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], kAtSoftWarps);
    }
    mbar_init(o_ready, 1);
    mbar_init(q_full, kAtSoftWarps);
    mbar_init(drain, 1);
    fence_mbar_init();
    prefetch_tmap(&maps.k[r]);
    prefetch_tmap(&maps.v[r]);
  }
  if (warp == kAtSoftWarps) {
    tmem_alloc(tmem_slot, kAtTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 256;

  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) *s_stat = status_get(status);
  if (threadIdx.x < 32) s_anc[threadIdx.x] = (int)threadIdx.x < n ? meta[row0 + threadIdx.x].anc : 0u;
  __syncthreads();

  if (*s_stat == 0) {
    uint8_t* sQ = smem + L::OFF_Q;
    if (warp == kAtSoftWarps) {
      // ---------------- issuer: TMA loads and MMAs (one thread) ----------------
      if (lane == 0) {
        const uint64_t pol = policy_evict_first();
        int k_iss[2] = {0, 0}, k_use[2] = {0, 0}, v_iss[2] = {0, 0}, v_use[2] = {0, 0};
        const int y0 = g * cap + key0;
        auto issue = [&](bool is_v, int tile) {   // one 128-key tile of K or V into its ring
          const int st = tile & 1;
          uint8_t* dst = smem + L::OFF_KV + ((is_v ? 2 : 0) + st) * L::KV_BYTES;
          uint64_t* bar = is_v ? &v_full[st] : &k_full[st];
          mbar_arrive_expect_tx(bar, L::KV_BYTES);
#pragma unroll
          for (int a = 0; a < L::SLABS; ++a)
            tma_load_2d(dst + a * kAtom, is_v ? &maps.v[r] : &maps.k[r], bar, a * 64, y0 + tile * 128, pol);
          if (is_v) ++v_iss[st]; else ++k_iss[st];
        };
        const uint32_t qaddr = smem_u32(sQ);
        const uint32_t idesc_s = idesc_bf16_f32(128, 128);
        const uint32_t idesc_o = idesc_bf16_f32(128, D) | (1u << 16);   // B (V) is MN-major
        auto mma_s = [&](int tile) -> bool {   // S[tile % 2] = Q K_tile^T
          const int st = tile & 1;
          if (!mbar_wait(&k_full[st], (uint32_t)(tile >> 1) & 1u)) return false;
          ++k_use[st];
          tc_fence_after();
          const uint32_t kaddr = smem_u32(smem + L::OFF_KV + st * L::KV_BYTES);
          const uint32_t tS = tmem + (uint32_t)(st * 128);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (uint32_t)((k >> 2) * kAtom + (k & 3) * 32);
            umma_bf16(tS, sdesc_sw128(qaddr + off, 16, 1024), sdesc_sw128(kaddr + off, 16, 1024), idesc_s,
                      k > 0 ? 1u : 0u);
          }
          umma_commit(&s_full[st]);
          umma_commit(&k_free[st]);
          return true;
        };
        auto mma_o = [&](int tile) -> bool {   // O += P_tile V_tile
          const int st = tile & 1;
          if (!mbar_wait(&v_full[st], (uint32_t)(tile >> 1) & 1u)) return false;
          ++v_use[st];
          tc_fence_after();
          const uint32_t vaddr = smem_u32(smem + L::OFF_KV + (2 + st) * L::KV_BYTES);
          const uint32_t paddr = smem_u32(smem + L::OFF_P);
#pragma unroll
          for (int k = 0; k < 8; ++k) {   // 16 keys per step
            const uint32_t aoff = (uint32_t)((k >> 2) * kAtom + (k & 3) * 32);
            umma_bf16(tO, sdesc_sw128(paddr + aoff, 16, 1024), sdesc_sw128(vaddr + k * 2048, kAtom, 1024),
                      idesc_o, (tile > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&v_free[st]);
          umma_commit(o_ready);
          return true;
        };
        // K tiles run two ahead of their S MMA (a K stage frees as soon as its
        // S MMA is done), V tiles two ahead of their O MMA
        issue(false, 0);
        issue(true, 0);
        if (T > 1) {
          issue(false, 1);
          issue(true, 1);
        }
        bool ok = mbar_wait(q_full, 0) && mma_s(0);
        if (ok && T > 2) {
          ok = mbar_wait(&k_free[0], 0);
          if (ok) issue(false, 2);
        }
        for (int tl = 0; tl < T && ok; ++tl) {
          if (tl + 1 < T) {   // S of the next tile, into the buffer softmax(tl - 1) released
            if (tl >= 1) ok = mbar_wait(&p_full[(tl + 1) & 1], (uint32_t)((tl - 1) >> 1) & 1u);
            if (ok) ok = mma_s(tl + 1);
            if (ok && tl + 3 < T) {
              ok = mbar_wait(&k_free[(tl + 1) & 1], (uint32_t)((tl + 1) >> 1) & 1u);
              if (ok) issue(false, tl + 3);
            }
            if (!ok) break;
          }
          ok = mbar_wait(&p_full[tl & 1], (uint32_t)(tl >> 1) & 1u);
          if (ok) {
            tc_fence_after();
            ok = mma_o(tl);
          }
          if (ok && tl + 2 < T) {   // V stage tl % 2 is free once this O MMA is done
            ok = mbar_wait(&v_free[tl & 1], (uint32_t)(tl >> 1) & 1u);
            if (ok) issue(true, tl + 2);
          }
        }
        if (!ok) status_set(status, TV_E_TIMEOUT);
        // loads still in flight land before the CTA leaves
        for (int st = 0; st < 2; ++st) {
          if (k_iss[st] > k_use[st]) mbar_wait(&k_full[st], (uint32_t)(k_iss[st] - 1) & 1u);
          if (v_iss[st] > v_use[st]) mbar_wait(&v_full[st], (uint32_t)(v_iss[st] - 1) & 1u);
        }
        umma_commit(drain);   // TMEM is released only after every MMA issued here is complete
        mbar_wait(drain, 0);
      }
    } else {
      // ---------------- softmax / epilogue ----------------
      // warp (quarter qd, slice cs): query rows 32 qd .. 32 qd + 31 of the tile
      // (its TMEM lanes), keys kKeysPer cs .. of every 128-key tile, and O
      // columns OC cs .. OC cs + OC - 1
      const int qd = warp & 3, cs = warp >> 2;
      const int i = qd * 32 + lane;
      const int qi = q0 + i;
      const bool valid_q = qi < nq;
      const bool active = q0 + qd * 32 < nq;   // warp-uniform: any valid row in this quarter
      const int local = valid_q ? qi / G : 0;
      const uint32_t anc = s_anc[local];
      for (int idx = threadIdx.x; idx < 128 * (D / 8); idx += kAtSoftThreads) {
        const int row = idx / (D / 8), c = idx % (D / 8);
        const int qr = q0 + row;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (qr < nq)
          v = reinterpret_cast<const uint4*>(q + ((size_t)(row0 + qr / G) * Hq + (size_t)(g * G + qr % G)) * D)[c];
        *reinterpret_cast<uint4*>(sQ + (c >> 3) * kAtom + swz(row, c & 7)) = v;
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);

      const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
      float m_use = -INFINITY, l_run = 0.f;   // m_use: the offset P and O are currently scaled by
      bool ok = true;
      for (int tl = 0; tl < T; ++tl) {
        const int b = tl & 1;
        if (ok) ok = mbar_wait(&s_full[b], (uint32_t)(tl >> 1) & 1u);
        tc_fence_after();
        const int kvalid = min(128, nkeys - tl * 128);
        const bool full = kvalid == 128 && !tree;
        const uint32_t s_addr = tmem + (uint32_t)(b * 128) + lane_base + cs * kKeysPer;
        float mx = -INFINITY;   // raw (unscaled) scores; the scale is positive
        if (active && ok) {   // pass 1: masked row maximum over this thread's keys, 32 at a time
#pragma unroll
          for (int h = 0; h < kKeysPer / 32; ++h) {
            uint32_t s[32];
            cols_ld<32>(s_addr + h * 32, s);
            tmem_ld_wait();
            if (full) {
#pragma unroll
              for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(s[j]));
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int key = cs * kKeysPer + h * 32 + j;
                if (key < kvalid && (!tree || ((anc >> key) & 1u))) mx = fmaxf(mx, __uint_as_float(s[j]));
              }
            }
          }
        }
        s_red[b][cs][i] = mx;
        // keys past the chunk: zero their V rows so that 0 * V stays 0 whatever
        // those slots hold (all softmax threads share the rows)
        if (kvalid < 128) {
          if (ok) ok = mbar_wait(&v_full[b], (uint32_t)(tl >> 1) & 1u);   // the V tile has landed
          uint8_t* vd = smem + L::OFF_KV + (2 + b) * L::KV_BYTES;
          const int nz = (128 - kvalid) * L::SLABS * 8;
          for (int idx = threadIdx.x; idx < nz; idx += kAtSoftThreads) {
            const int row = kvalid + idx / (L::SLABS * 8), rem = idx % (L::SLABS * 8);
            *reinterpret_cast<uint4*>(vd + (rem >> 3) * kAtom + row * 128 + (rem & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
        quarter_barrier(qd);
        float m_tile = s_red[b][0][i];
#pragma unroll
        for (int c = 1; c < kSlices; ++c) m_tile = fmaxf(m_tile, s_red[b][c][i]);
        m_tile *= scale_log2;   // to log2 units
        // new offset only when the max outgrows the current one by 2^8 (exact:
        // O and l carry the same offset, which cancels in O / l)
        const bool grow = m_tile > m_use + kRescaleLog2;
        const float m_new = grow ? m_tile : m_use;
        const float corr = (grow && m_use != -INFINITY) ? exp2f(m_use - m_new) : 1.f;
        if (active && ok) {
          // P = 2^(x - m) in bf16; the row sum adds the rounded values
          float lt = 0.f;
          uint32_t pk[kKeysPer / 2];
          const float neg_m = m_new == -INFINITY ? 0.f : -m_new;
#pragma unroll
          for (int h = 0; h < kKeysPer / 32; ++h) {   // pass 2: P = 2^(x - m), 32 keys at a time
            uint32_t s[32];
            cols_ld<32>(s_addr + h * 32, s);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              float p0 = ex2(fmaf(__uint_as_float(s[j]), scale_log2, neg_m));
              float p1 = ex2(fmaf(__uint_as_float(s[j + 1]), scale_log2, neg_m));
              if (!full) {
                const int key = cs * kKeysPer + h * 32 + j;
                if (!(key < kvalid && (!tree || ((anc >> key) & 1u)))) p0 = 0.f;
                if (!(key + 1 < kvalid && (!tree || ((anc >> (key + 1)) & 1u)))) p1 = 0.f;
              }
              lt += p0 + p1;
              const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
              pk[h * 16 + (j >> 1)] = *reinterpret_cast<const uint32_t*>(&pb);
            }
          }
          l_run = l_run * corr + lt;
          m_use = m_new;
          // the P buffer and O are free once O += P V of the previous tile is done
          if (tl > 0) {
            if (!mbar_wait(o_ready, (uint32_t)(tl - 1) & 1u)) ok = false;
            tc_fence_after();
          }
          // keys kKeysPer cs .. : 16-byte chunks (8 keys) of row i in the 64-key slabs
#pragma unroll
          for (int u = 0; u < kKeysPer / 8; ++u) {
            const int key8 = cs * kKeysPer + u * 8;
            *reinterpret_cast<uint4*>(smem + L::OFF_P + (key8 >> 6) * kAtom + swz(i, (key8 & 63) >> 3)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
          // a grown offset: O (complete up to tile tl-1) gets the same factor
          if (tl > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
            for (int h = 0; h < OC / 16; ++h) {
              uint32_t o[16];
              cols_ld<16>(tO + lane_base + cs * OC + h * 16, o);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 16; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * corr);
              cols_st<16>(tO + lane_base + cs * OC + h * 16, o);
            }
            tmem_st_wait();
          }
        } else if (tl > 0 && ok) {
          // an idle quarter still waits, so that no warp runs ahead of the O MMA
          if (!mbar_wait(o_ready, (uint32_t)(tl - 1) & 1u)) ok = false;
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[b]);
      }
      if (ok) ok = mbar_wait(o_ready, (uint32_t)(T - 1) & 1u);
      s_l[cs][i] = active ? l_run : 0.f;
      soft_barrier();
      if (!ok) {
        if (lane == 0) status_set(status, TV_E_TIMEOUT);
      } else if (active) {
        tc_fence_after();
        const int hq = g * G + (valid_q ? qi % G : 0);
        const size_t base = ((size_t)(row0 + local) * Hq + hq) * kChunkSlots + slot;
        float4* dst = reinterpret_cast<float4*>(part_o + base * D + cs * OC);
#pragma unroll
        for (int h = 0; h < OC / 16; ++h) {
          uint32_t o[16];
          cols_ld<16>(tO + lane_base + cs * OC + h * 16, o);
          tmem_ld_wait();
          if (valid_q) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[h * 4 + j] = make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                           __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
          }
        }
        if (valid_q) {
          if (cs == 0) {
            float l = s_l[0][i];
#pragma unroll
            for (int c = 1; c < kSlices; ++c) l += s_l[c][i];
            part_ml[base * 2] = m_use;
            part_ml[base * 2 + 1] = l;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kAtSoftWarps) {
    tc_fence_after();
    tmem_dealloc(tmem, kAtTmemCols);
  }
}

// out[row][h*D + d] = bf16( sum_c o_c[d] 2^(m_c - M) / sum_c l_c 2^(m_c - M) ),
// chunks in order 0..nch-1, then the tree slot.  grid (rows, Hq), block D.
__global__ void attn_merge_kernel(ReqTable t, const RowMeta* meta, int Hq, int D, const float* part_ml,
                                  const float* part_o, __nv_bfloat16* out, const int32_t* status) {
  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int row = blockIdx.x, hq = blockIdx.y, d = threadIdx.x;
  const int nch = attn_n_chunks(t.ctx[meta[row].req]);
  const size_t base = ((size_t)row * Hq + hq) * kChunkSlots;
  float M = part_ml[(base + kTreeSlot) * 2];
  for (int c = 0; c < nch; ++c) M = fmaxf(M, part_ml[(base + c) * 2]);
  float L = 0.f, O = 0.f;
  for (int k = 0; k <= nch; ++k) {
    const int c = k < nch ? k : kTreeSlot;
    const float w = exp2f(part_ml[(base + c) * 2] - M);   // maxima are in log2 units
    L = fmaf(part_ml[(base + c) * 2 + 1], w, L);
    O = fmaf(part_o[(base + c) * D + d], w, O);
  }
  out[(size_t)row * Hq * D + (size_t)hq * D + d] = f2bf(O / L);
}

template <int D>
int launch_attention_d(const ReqTable& t, const tv_dims& dm, const LayerBufs& b, int32_t* status,
                       cudaStream_t st) {
  AttnMaps maps;
  memset(&maps, 0, sizeof(maps));
  int nch_max = 0, nq_max = 0;
  const int G = dm.n_q_heads / dm.n_kv_heads;
  for (int r = 0; r < t.n_req; ++r) {
    const int rows = dm.n_kv_heads * t.capacity[r];
    int rc = make_tmap_bf16(&maps.k[r], t.k[r], D, rows, 64, 128);
    if (rc) return rc;
    rc = make_tmap_bf16(&maps.v[r], t.v[r], D, rows, 64, 128);
    if (rc) return rc;
    nch_max = max(nch_max, attn_n_chunks(t.ctx[r]));
    nq_max = max(nq_max, t.n[r] * G);
  }
  const int q_tiles = (nq_max + 127) / 128;
  const size_t smem = AtSmem<D>::BYTES;
  static bool attr[64] = {false};
  if (ensure_smem_limit(attn_tc_kernel<D>, smem, attr)) return TV_E_CUDA;
  dim3 grid(q_tiles, nch_max + 1, t.n_req * dm.n_kv_heads);
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));   // log2(e) / sqrt(D)
  int rc = launch_pdl(attn_tc_kernel<D>, grid, dim3(kAtThreads), smem, st, maps, t, (const RowMeta*)b.meta,
                      (const __nv_bfloat16*)b.q, dm.n_q_heads, dm.n_kv_heads, scale_log2, b.attn_ml, b.attn_o,
                      status);
  if (rc) return rc;
  return launch_pdl(attn_merge_kernel, dim3(t.total_rows, dm.n_q_heads), dim3(D), 0, st, t, (const RowMeta*)b.meta,
                    dm.n_q_heads, D, (const float*)b.attn_ml, (const float*)b.attn_o, b.attn, (const int32_t*)status);
}

}  // namespace

int launch_attention(const ReqTable& t, const tv_dims& d, const LayerBufs& b, int32_t* status, cudaStream_t st) {
  if (d.head_dim == 128) return launch_attention_d<128>(t, d, b, status, st);
  if (d.head_dim == 64) return launch_attention_d<64>(t, d, b, status, st);
  return TV_E_UNSUPPORTED;
}

}  // namespace tv
