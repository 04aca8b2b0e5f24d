// Index branch of MSA prefill: scores of every visible key, causal block
// max-pool and top-k with the forced local block, fused so that neither the
// N x N scores nor (unless asked for) the block scores are written.
//
// Follows "MiniMax Sparse Attention (MSA): a Two-Branch Block-Sparse Attention
// Trained on a 109B-Parameter MoE With a 3T-Token Budget", section
// "两个分支如何工作" (how the two branches work): one index-query head per GQA
// group, one shared index-key head, visible keys scored and max-pooled to
// blocks, top-k per (query, group) with the query's own block always kept.
//
// Rows of the score matrix are the flattened (t, g) pairs of q_idx
// [N, n_g, d_idx]; columns are keys. Because the index key head is shared, one
// k_idx block serves all groups of a row tile.
//
// This version computes on CUDA cores: a CTA owns 64 rows and streams key
// blocks 0 .. loc_max; each key block becomes one fp32 max per row, which the
// row's owner thread feeds to its streaming top-k (RowTopK).
#include "msa_kernels.h"

namespace msa {
namespace {

constexpr int kRows = 64;    // rows (t, g) per CTA
constexpr int kBk = 128;     // keys per block
constexpr int kDc = 32;      // d_idx chunk staged per pass
constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads)
index_select_cc_kernel(const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx,
                       int64_t N, int n_g, int d_idx, int k, int32_t* __restrict__ block_ids,
                       float* __restrict__ block_scores, int64_t nb) {
  __shared__ float As[kRows][kDc + 1];
  __shared__ float Bs[kBk][kDc + 1];

  const int64_t n_rows = N * n_g;
  const int64_t n_tiles = (n_rows + kRows - 1) / kRows;
  const int64_t tile = n_tiles - 1 - blockIdx.x;  // heavy tiles first
  const int64_t row0 = tile * kRows;
  const int tid = threadIdx.x;
  const int rg = tid >> 4;   // rows rg*4 .. rg*4+3
  const int kg = tid & 15;   // keys kg + 16 i

  const int64_t last_row = min(row0 + kRows, n_rows) - 1;
  const int64_t loc_max = (last_row / n_g) / kBk;
  const int64_t b_end = block_scores ? loc_max + 1 : loc_max;  // local block only pooled on request

  // owner thread of row rg*4 + kg (kg < 4)
  const bool owner = kg < 4;
  const int64_t my_row = row0 + rg * 4 + kg;
  const bool my_valid = owner && my_row < n_rows;
  const int64_t my_t = my_valid ? my_row / n_g : 0;
  const int64_t my_loc = my_t / kBk;
  RowTopK top;
  top.init(k - 1);

  for (int64_t b = 0; b < b_end; ++b) {
    float acc[4][8];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[r][i] = 0.f;

    for (int c0 = 0; c0 < d_idx; c0 += kDc) {
      __syncthreads();
      for (int e = tid; e < kRows * kDc; e += kThreads) {
        int r = e / kDc, c = e % kDc;
        int64_t row = row0 + r;
        float x = 0.f;
        if (row < n_rows) x = __uint_as_float((uint32_t)q_idx[row * d_idx + c0 + c] << 16);
        As[r][c] = x;
      }
      for (int e = tid; e < kBk * kDc; e += kThreads) {
        int j = e / kDc, c = e % kDc;
        int64_t key = b * kBk + j;
        float x = 0.f;
        if (key < N) x = __uint_as_float((uint32_t)k_idx[key * d_idx + c0 + c] << 16);
        Bs[j][c] = x;
      }
      __syncthreads();
#pragma unroll 8
      for (int c = 0; c < kDc; ++c) {
        float a[4], bb[8];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = As[rg * 4 + r][c];
#pragma unroll
        for (int i = 0; i < 8; ++i) bb[i] = Bs[kg + 16 * i][c];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[r][i] = fmaf(a[r], bb[i], acc[r][i]);
      }
    }
    // causal mask and per-thread max over its 8 keys, then over the 16 lanes
    float mx[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      int64_t row = row0 + rg * 4 + r;
      int64_t t = row / n_g;
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        int64_t key = b * kBk + kg + 16 * i;
        if (key <= t) m = fmaxf(m, acc[r][i]);
      }
      mx[r] = m;
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1)
#pragma unroll
      for (int r = 0; r < 4; ++r) mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], off));
    if (my_valid && b <= my_loc) {
      float v = mx[0];
#pragma unroll
      for (int r = 1; r < 4; ++r)
        if (kg == r) v = mx[r];
      if (block_scores) block_scores[my_row * nb + b] = v;
      if (b < my_loc) {
        uint64_t key = rank_key(v, (uint32_t)b);
        if (top.wants(key)) top.offer(key);
      }
    }
  }
  if (my_valid) top.emit((int)my_loc, k, block_ids + my_row * k);
}

}  // namespace

cudaError_t launch_index_select(const void* q_idx, const void* k_idx, int64_t N, int n_g,
                                int d_idx, int k, int32_t* block_ids, float* block_scores,
                                int64_t nb, const Diag& dg, cudaStream_t st) {
  (void)dg;
  int64_t n_tiles = (N * n_g + kRows - 1) / kRows;
  if (n_tiles == 0) return cudaSuccess;
  note_launches(1);
  index_select_cc_kernel<<<(unsigned)n_tiles, kThreads, 0, st>>>(
      (const uint16_t*)q_idx, (const uint16_t*)k_idx, N, n_g, d_idx, k, block_ids,
      block_scores, nb);
  return cudaGetLastError();
}

}  // namespace msa
