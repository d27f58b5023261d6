// Host interface of the tcgen05 skinny GEMM (tv_gemm.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tv_common.cuh"

namespace tv {

enum GemmMode { GEMM_PARTIAL = 0, GEMM_HEAD = 1 };

struct GemmParams {
  int M, K;                  // weight [M][K]
  int n_rows;                // activation rows present (<= 32)
  int splits;                // split-K count (1 for the head)
  int kb_per_split;          // 64-wide k-blocks per split
  int n_units;               // ceil(M / 128) * splits
  float* out;                // PARTIAL: [splits][32][M] fp32; HEAD: logits [n_rows][M]
  Top2* top2_part;           // HEAD: [gridDim.x][32]
  unsigned int* done_counter;// HEAD: zero before the launch, left at zero
  int32_t* argmax;           // HEAD: [n_rows]
  float* gap;                // HEAD: [n_rows]
  int32_t* status;           // sticky status word
  int packed;                // weight in the tile-packed layout (tiles of BM x BK, row-major inside)
};

struct GemmPlan {
  int splits, kb_per_split, n_units;
};

// The split-K partition of a weight [M][K]: a function of (M, K) only.
GemmPlan plan_gemm(int M, int K, bool head);
size_t gemm_smem_bytes();
// 2-D bf16 tensor map over [rows][inner] with a box of box_rows x box_inner
// and the 128-byte swizzle; rows past `rows` read as zeros.
int make_tmap_bf16(CUtensorMap* map, const void* base, int inner, int rows, int box_inner, int box_rows);
// 3-D bf16 tensor map over [d2][d1][d0] (d0 contiguous) with a box of
// b2 x b1 x b0 and the 128-byte swizzle: a box lands as b2 * b1 rows of b0
// elements, row (z, y) at row index z * b1 + y.
int make_tmap_bf16_3d(CUtensorMap* map, const void* base, int d0, int d1, int d2, int b0, int b1, int b2);
int launch_gemm(int mode, const void* W, int M, int K, const void* X, int n_rows, const GemmPlan& pl,
                const GemmParams& base, int num_sms, cudaStream_t stream);
// W [rows][cols] row-major -> the tile-packed layout (128 x 64 tiles, rows
// padded with zeros to a multiple of 128)
int launch_pack_weight(const void* W, int rows, int cols, void* packed, cudaStream_t stream);

}  // namespace tv
