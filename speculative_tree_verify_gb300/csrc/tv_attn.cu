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
//   softmax        one thread per query row (its TMEM lane): scale 1/sqrt(D),
//                  mask (keys past the chunk; ancestors for the tree tile),
//                  online max / sum in fp32, P = exp(s - m) rounded to bf16
//                  into swizzled smem, O in TMEM rescaled when the max grows
//   O += P V       tcgen05.mma M128 N=D K16, V straight from its TMA layout as
//                  an MN-major operand
// K/V tiles are double-buffered: TMA of tile t+1 overlaps tile t.
#include <cstring>

#include "tv_common.cuh"
#include "tv_gemm.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr int kAtThreads = 192;   // warps 0-3 softmax/epilogue, warp 4 TMA + MMA, warp 5 TMEM owner
constexpr int kAtTmemCols = 256;  // S: columns [0, 128), O: columns [128, 128 + D)
constexpr int kAtom = 128 * 128;  // bytes of one 128-row x 128-byte swizzled slab

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
  static constexpr int OFF_KV = OFF_Q + Q_BYTES;     // stage s: K at OFF_KV + 2 s KV_BYTES, V after it
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

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <int D>
__global__ void __launch_bounds__(kAtThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnMaps maps, ReqTable t, const RowMeta* meta, const __nv_bfloat16* q,
                   int Hq, int Hkv, float scale, int q_tiles, float* part_ml, float* part_o, int32_t* status) {
  using L = AtSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);   // [2]
  uint64_t* s_full = kv_full + 2;
  uint64_t* p_full = s_full + 1;
  uint64_t* o_done = p_full + 1;
  uint64_t* q_full = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 1);
  int* s_stat = reinterpret_cast<int*>(tmem_slot + 1);
  __shared__ uint32_t s_anc[32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot_x = blockIdx.x, g = blockIdx.y, r = blockIdx.z / q_tiles, qt = blockIdx.z % q_tiles;

  // ---- structural early exits (kernel parameters only) ------------------------
  const int ctx = t.ctx[r], n = t.n[r], row0 = t.row_off[r], cap = t.capacity[r];
  const int nch = attn_n_chunks(ctx);
  const bool tree = slot_x == (int)gridDim.x - 1;
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
    mbar_init(&kv_full[0], 1);
    mbar_init(&kv_full[1], 1);
    mbar_init(s_full, 1);
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(q_full, 4);
    fence_mbar_init();
    prefetch_tmap(&maps.k[r]);
    prefetch_tmap(&maps.v[r]);
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, kAtTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;

  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) *s_stat = status_get(status);
  if (threadIdx.x < 32) s_anc[threadIdx.x] = (int)threadIdx.x < n ? meta[row0 + threadIdx.x].anc : 0u;
  __syncthreads();

  if (*s_stat == 0) {
    uint8_t* sQ = smem + L::OFF_Q;
    uint8_t* sP = smem + L::OFF_P;
    if (warp == 4) {
      // ---------------- TMA + MMA (one thread) ----------------
      if (lane == 0) {
        const uint64_t pol = policy_evict_first();
        const CUtensorMap* km = &maps.k[r];
        const CUtensorMap* vm = &maps.v[r];
        int issued[2] = {0, 0}, used[2] = {0, 0};
        auto issue = [&](int tile) {
          const int st = tile & 1;
          uint8_t* kd = smem + L::OFF_KV + st * 2 * L::KV_BYTES;
          uint8_t* vd = kd + L::KV_BYTES;
          mbar_arrive_expect_tx(&kv_full[st], 2 * L::KV_BYTES);
          const int y = g * cap + key0 + tile * 128;
#pragma unroll
          for (int a = 0; a < L::SLABS; ++a) {
            tma_load_2d(kd + a * kAtom, km, &kv_full[st], a * 64, y, pol);
            tma_load_2d(vd + a * kAtom, vm, &kv_full[st], a * 64, y, pol);
          }
          ++issued[st];
        };
        issue(0);
        if (T > 1) issue(1);
        const uint32_t idesc_s = idesc_bf16_f32(128, 128);
        const uint32_t idesc_o = idesc_bf16_f32(128, D) | (1u << 16);   // B (V) is MN-major
        bool ok = mbar_wait(q_full, 0);
        for (int tl = 0; tl < T && ok; ++tl) {
          const int st = tl & 1;
          ok = mbar_wait(&kv_full[st], (uint32_t)(tl >> 1) & 1u);
          if (!ok) break;
          ++used[st];
          tc_fence_after();
          const uint32_t kaddr = smem_u32(smem + L::OFF_KV + st * 2 * L::KV_BYTES);
          const uint32_t vaddr = kaddr + L::KV_BYTES;
          const uint32_t qaddr = smem_u32(sQ);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {   // 16 elements of D per step
            const uint32_t off = (uint32_t)((k >> 2) * kAtom + (k & 3) * 32);
            umma_bf16(tS, sdesc_sw128(qaddr + off, 16, 1024), sdesc_sw128(kaddr + off, 16, 1024), idesc_s,
                      k > 0 ? 1u : 0u);
          }
          umma_commit(s_full);
          ok = mbar_wait(p_full, (uint32_t)tl & 1u);
          if (!ok) break;
          tc_fence_after();
          if (tl >= 1 && tl + 1 < T) issue(tl + 1);   // its stage held tile tl-1, whose MMAs are done
          const uint32_t paddr = smem_u32(sP);
#pragma unroll
          for (int k = 0; k < 8; ++k) {   // 16 keys per step
            const uint32_t aoff = (uint32_t)((k >> 2) * kAtom + (k & 3) * 32);
            umma_bf16(tO, sdesc_sw128(paddr + aoff, 16, 1024), sdesc_sw128(vaddr + k * 2048, kAtom, 1024),
                      idesc_o, (tl > 0 || k > 0) ? 1u : 0u);
          }
        }
        umma_commit(o_done);
        if (!ok) status_set(status, TV_E_TIMEOUT);
        // loads still in flight land before the CTA leaves
        for (int st = 0; st < 2; ++st)
          if (issued[st] > used[st]) mbar_wait(&kv_full[st], (uint32_t)(issued[st] - 1) & 1u);
      }
    } else if (warp < 4) {
      // ---------------- softmax / epilogue: thread i owns query row i ----------------
      const int i = threadIdx.x;
      const int qi = q0 + i;
      const bool valid_q = qi < nq;
      const int local = valid_q ? qi / G : 0;
      const uint32_t anc = s_anc[local];
      // this row's query vector (zeros past nq) into the swizzled tile
      {
        const uint4* src = reinterpret_cast<const uint4*>(
            q + ((size_t)(row0 + local) * Hq + (size_t)(g * G + (valid_q ? qi % G : 0))) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = valid_q ? src[c] : make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(sQ + (c >> 3) * kAtom + swz(i, c & 7)) = v;
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_full);

      const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int tl = 0; tl < T && ok; ++tl) {
        ok = mbar_wait(s_full, (uint32_t)tl & 1u);
        if (!ok) break;
        tc_fence_after();
        const int kvalid = min(128, nkeys - tl * 128);
        // pass 1: masked maximum of the scaled scores
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t s[32];
          tmem_ld_32x32b_x32(tS + lane_base + c * 32, s);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int key = c * 32 + j;
            const bool vis = key < kvalid && (!tree || ((anc >> key) & 1u));
            if (vis) mx = fmaxf(mx, __uint_as_float(s[j]) * scale);
          }
        }
        const float m_new = fmaxf(m_run, mx);
        const float corr = (m_run == -INFINITY || m_new == -INFINITY) ? 1.f : expf(m_run - m_new);
        // O += P V of the previous tile is complete (this tile's S commit follows
        // it): rescale O where the max grew
        if (tl > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO + lane_base + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * corr);
            tmem_st_32x32b_x32(tO + lane_base + c * 32, o);
          }
          tmem_st_wait();
        }
        // keys past the chunk: zero their V rows so that 0 * V stays 0 whatever
        // those slots hold
        if (kvalid < 128 && i >= kvalid) {
          uint8_t* vd = smem + L::OFF_KV + (tl & 1) * 2 * L::KV_BYTES + L::KV_BYTES;
#pragma unroll
          for (int a = 0; a < L::SLABS; ++a)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(vd + a * kAtom + i * 128 + c * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        // pass 2: P = exp(s - m) in bf16; the row sum adds the rounded values
        float lt = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t s[32];
          tmem_ld_32x32b_x32(tS + lane_base + c * 32, s);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float p2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int key = c * 32 + j + e;
              const bool vis = key < kvalid && (!tree || ((anc >> key) & 1u));
              p2[e] = (vis && m_new != -INFINITY) ? expf(__uint_as_float(s[j + e]) * scale - m_new) : 0.f;
            }
            const __nv_bfloat162 pb = __floats2bfloat162_rn(p2[0], p2[1]);
            const float2 pr = __bfloat1622float2(pb);
            lt += pr.x + pr.y;
            pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&pb);
          }
          // 32 keys = four 16-byte chunks of row i in key slab c / 2
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(sP + (c >> 1) * kAtom + swz(i, (c & 1) * 4 + u)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
        l_run = l_run * corr + lt;
        m_run = m_new;
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (ok) ok = mbar_wait(o_done, 0);
      if (!ok) {
        status_set(status, TV_E_TIMEOUT);
      } else {
        tc_fence_after();
        const int hq = g * G + (valid_q ? qi % G : 0);
        const size_t base = ((size_t)(row0 + local) * Hq + hq) * kChunkSlots + slot;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO + lane_base + c * 32, o);
          tmem_ld_wait();
          if (valid_q) {
            float4* dst = reinterpret_cast<float4*>(part_o + base * D + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(o[4 * j]), __uint_as_float(o[4 * j + 1]),
                                   __uint_as_float(o[4 * j + 2]), __uint_as_float(o[4 * j + 3]));
          }
        }
        if (valid_q) {
          part_ml[base * 2] = m_run;
          part_ml[base * 2 + 1] = l_run;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kAtTmemCols);
  }
}

// out[row][h*D + d] = bf16( sum_c o_c[d] e^(m_c - M) / sum_c l_c e^(m_c - M) ),
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
    const float w = expf(part_ml[(base + c) * 2] - M);
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
  dim3 grid(nch_max + 1, dm.n_kv_heads, t.n_req * q_tiles);
  int rc = launch_pdl(attn_tc_kernel<D>, grid, dim3(kAtThreads), smem, st, maps, t, (const RowMeta*)b.meta,
                      (const __nv_bfloat16*)b.q, dm.n_q_heads, dm.n_kv_heads, 1.0f / sqrtf((float)D), q_tiles,
                      b.attn_ml, b.attn_o, status);
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
