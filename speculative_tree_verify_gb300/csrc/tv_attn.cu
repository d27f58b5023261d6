// Tree-masked GQA attention over the cached context plus the tree rows.
//
// Row i, query head h attends to the cached slots [0, ctx) and to the tree
// slots ctx + a for every a in anc(i) (its ancestors and itself): "give each
// node an attention mask of its ancestors and a position equal to its depth"
// [Drafters and tree verify, §Tree verify through recurrent layers].  The
// positions were applied by RoPE before the keys were written.
//
// Split-context (flash-decoding) layout: one CTA per (request, KV head,
// context chunk) plus one CTA per (request, KV head) for the tree keys.  A CTA
// serves all GQA query heads of its KV head and all rows of its request, so
// each K/V byte is read once per CTA.  The chunk length is a function of ctx
// only, and the merge kernel combines the chunks' (max, sum, unnormalised
// output) partials in chunk order, then the tree slot, so every row's result
// is the same whatever the other rows are.
//
// Arithmetic: scores and softmax in fp32 (expf), K/V staged to shared memory
// as fp32.  Per query: s_j = (q . k_j) / sqrt(D); online softmax over 32-key
// tiles; the ancestor set comes from the prologue's bitmask (built from the
// parent array).
#include "tv_common.cuh"
#include "tv_kernels.cuh"

namespace tv {

namespace {

constexpr int kQPW = 5;                  // query vectors per warp
constexpr int kQPB = 8 * kQPW;           // query vectors per CTA (8 warps)
constexpr int kQSplits = (kMaxQueriesPerKvHead + kQPB - 1) / kQPB;   // CTAs per (request, KV head, chunk)

template <int D>
struct AttnSmem {
  static constexpr int DP = D + 4;   // fp32 row stride: 16-byte rows, conflict-free float4 reads
  static constexpr int NQ = 8 * kQPW;
  static constexpr size_t bytes = sizeof(float) * ((size_t)NQ * DP + 32 * DP + 32 * D + 8 * kQPW * 32);
};

template <int D>
__global__ void __launch_bounds__(256, 2)
    attn_partial_kernel(ReqTable t, const RowMeta* meta, const __nv_bfloat16* q, int Hq, int Hkv, float scale,
                        float* part_ml, float* part_o, const int32_t* status) {
  constexpr int DP = AttnSmem<D>::DP;
  constexpr int NQ = AttnSmem<D>::NQ;
  constexpr int DPL = D / 32;   // output dims per lane
  extern __shared__ float4 smem4[];
  float* Qs = reinterpret_cast<float*>(smem4);   // [NQ][DP]
  float* Ks = Qs + NQ * DP;                      // [32][DP]
  float* Vs = Ks + 32 * DP;                      // [32][D]
  float* Ps = Vs + 32 * D;                       // [8][kQPW][32]
  __shared__ uint32_t s_anc[32];

  pdl_wait();
  pdl_trigger();
  if (block_skip(status)) return;
  const int slot = blockIdx.x, g = blockIdx.y, r = blockIdx.z / kQSplits;
  const int q0 = (blockIdx.z % kQSplits) * kQPB;   // this CTA's first query vector
  const int ctx = t.ctx[r], n = t.n[r], row0 = t.row_off[r];
  const bool tree = slot == kTreeSlot;
  if (!tree && slot >= attn_n_chunks(ctx)) return;
  int key0, nkeys;
  if (tree) {
    key0 = ctx;
    nkeys = n;
  } else {
    const int ch = attn_chunk_len(ctx);
    key0 = slot * ch;
    nkeys = min(ch, ctx - key0);
  }
  const int G = Hq / Hkv;
  const int nq = n * G;
  if (q0 >= nq) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int nqw = 0;   // valid query vectors of this warp: qi = q0 + warp + 8 a
  for (int a = 0; a < kQPW; ++a)
    if (q0 + warp + 8 * a < nq) nqw = a + 1;

  for (int idx = threadIdx.x; idx < NQ * D; idx += 256) {
    const int qi = q0 + idx / D, d = idx - (idx / D) * D;
    float v = 0.f;
    if (qi < nq) {
      const int local = qi / G, hq = g * G + qi % G;
      v = bf2f(q[((size_t)(row0 + local) * Hq + hq) * D + d]);
    }
    Qs[(qi - q0) * DP + d] = v;
  }
  if (threadIdx.x < 32) s_anc[threadIdx.x] = (int)threadIdx.x < n ? meta[row0 + threadIdx.x].anc : 0u;

  const size_t head_off = (size_t)g * t.capacity[r] * D;
  const __nv_bfloat16* Kg = t.k[r] + head_off;
  const __nv_bfloat16* Vg = t.v[r] + head_off;

  float m[kQPW], l[kQPW], o[kQPW][DPL];
#pragma unroll
  for (int a = 0; a < kQPW; ++a) {
    m[a] = -INFINITY;
    l[a] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) o[a][e] = 0.f;
  }

  for (int kt = 0; kt < nkeys; kt += 32) {
    __syncthreads();   // queries staged / previous tile consumed
    for (int idx = threadIdx.x; idx < 32 * (D / 8); idx += 256) {
      const int j = idx / (D / 8), c8 = (idx - j * (D / 8)) * 8;
      float kf[8], vf[8];
      if (kt + j < nkeys) {
        const size_t off = (size_t)(key0 + kt + j) * D + c8;
        const uint4 kr = *reinterpret_cast<const uint4*>(Kg + off);
        const uint4 vr = *reinterpret_cast<const uint4*>(Vg + off);
        const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kr);
        const __nv_bfloat16* vb = reinterpret_cast<const __nv_bfloat16*>(&vr);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          kf[e] = bf2f(kb[e]);
          vf[e] = bf2f(vb[e]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) kf[e] = vf[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        Ks[j * DP + c8 + e] = kf[e];
        Vs[j * D + c8 + e] = vf[e];
      }
    }
    __syncthreads();

    const int j = lane;
    const bool kvalid = kt + j < nkeys;
    float s[kQPW];
#pragma unroll
    for (int a = 0; a < kQPW; ++a) s[a] = 0.f;
    const float4* k4 = reinterpret_cast<const float4*>(Ks + j * DP);
#pragma unroll 4
    for (int d4 = 0; d4 < D / 4; ++d4) {
      const float4 kk = k4[d4];
#pragma unroll
      for (int a = 0; a < kQPW; ++a) {
        if (a < nqw) {
          const float4 qq = *reinterpret_cast<const float4*>(Qs + (warp + 8 * a) * DP + 4 * d4);
          s[a] = fmaf(qq.x, kk.x, s[a]);
          s[a] = fmaf(qq.y, kk.y, s[a]);
          s[a] = fmaf(qq.z, kk.z, s[a]);
          s[a] = fmaf(qq.w, kk.w, s[a]);
        }
      }
    }
#pragma unroll
    for (int a = 0; a < kQPW; ++a) {
      if (a < nqw) {
        const int local = (q0 + warp + 8 * a) / G;
        const bool vis = kvalid && (!tree || ((s_anc[local] >> j) & 1u));
        const float sc = vis ? s[a] * scale : -INFINITY;
        const float mnew = fmaxf(m[a], warp_max(sc));
        const float corr = mnew == -INFINITY ? 1.f : expf(m[a] - mnew);
        const float p = mnew == -INFINITY ? 0.f : expf(sc - mnew);
        l[a] = l[a] * corr + p;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[a][e] *= corr;
        m[a] = mnew;
        Ps[(warp * kQPW + a) * 32 + j] = p;
      }
    }
    __syncwarp();
    for (int jj = 0; jj < 32; ++jj) {
      float v[DPL];
#pragma unroll
      for (int e = 0; e < DPL; ++e) v[e] = Vs[jj * D + lane * DPL + e];
#pragma unroll
      for (int a = 0; a < kQPW; ++a) {
        if (a < nqw) {
          const float p = Ps[(warp * kQPW + a) * 32 + jj];
#pragma unroll
          for (int e = 0; e < DPL; ++e) o[a][e] = fmaf(p, v[e], o[a][e]);
        }
      }
    }
  }

#pragma unroll
  for (int a = 0; a < kQPW; ++a) {
    if (a < nqw) {
      const int qi = q0 + warp + 8 * a;
      const float lt = warp_sum(l[a]);
      const int local = qi / G, hq = g * G + qi % G;
      const size_t base = ((size_t)(row0 + local) * Hq + hq) * kChunkSlots + slot;
      if (lane == 0) {
        part_ml[base * 2] = m[a];
        part_ml[base * 2 + 1] = lt;
      }
#pragma unroll
      for (int e = 0; e < DPL; ++e) part_o[base * D + lane * DPL + e] = o[a][e];
    }
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
  const size_t smem = AttnSmem<D>::bytes;
  static bool attr[64] = {false};
  if (ensure_smem_limit(attn_partial_kernel<D>, smem, attr)) return TV_E_CUDA;
  dim3 grid(kChunkSlots, dm.n_kv_heads, t.n_req * kQSplits);
  int rc = launch_pdl(attn_partial_kernel<D>, grid, dim3(256), smem, st, t, (const RowMeta*)b.meta,
                      (const __nv_bfloat16*)b.q, dm.n_q_heads, dm.n_kv_heads, 1.0f / sqrtf((float)D), b.attn_ml,
                      b.attn_o, (const int32_t*)status);
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
