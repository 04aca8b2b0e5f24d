// Host-side launchers of the MSA kernels (internal to libmsa).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "msa_common.cuh"

namespace msa {

// Counts every kernel launch / device memset enqueued by the library.
void note_launches(int n);

// Error word and wait limit of the current device, for entry points defined
// outside msa_abi.cu.
Diag current_diag();

// Index branch, prefill (msa_index.cu).
// e4m3: q_idx / k_idx hold E4M3 codes (d_idx = 128), and score_scale multiplies
// the reported block scores.
cudaError_t launch_index_select(const void* q_idx, const void* k_idx, int64_t N, int n_g,
                                int d_idx, int k, int32_t* block_ids, float* block_scores,
                                int64_t nb, const Diag& dg, cudaStream_t st, bool e4m3 = false,
                                float score_scale = 1.f);

// One launch per 128 non-empty sequences of a packed batch; cu_seqlens is a
// host array [B + 1] of token offsets (msa_index.cu).
cudaError_t launch_index_select_varlen(const void* q_idx, const void* k_idx,
                                       const int64_t* cu_seqlens, int B, int n_g, int d_idx,
                                       int k, int32_t* block_ids, const Diag& dg,
                                       cudaStream_t st);

// Exp-free top-k over block scores (msa_topk.cu).
cudaError_t launch_topk(const float* S, int64_t N, int n_g, int64_t nb, int Bk, int k,
                        int64_t q_offset, const int32_t* seq_lens, int32_t* ids, const Diag& dg,
                        cudaStream_t st);

// Main branch, prefill (msa_attn.cu).
struct AttnWs {
  int32_t* counts;    // [n_g * nb]
  int32_t* offsets;   // [n_g * nb + 1]
  int32_t* cursor;    // [n_g * nb]
  int32_t* tile_off;  // [n_g * nb + 1]
  int32_t* percta;    // [bucketing CTAs, n_g * nb] per-CTA counts, then first positions
  int32_t* entries;   // [chunk * n_g * k]
  int4* tinfo;        // per tile: block, first entry, queries | group << 8, end tile
  int32_t* rec_of;    // [chunk, n_g, k]: partial record of each (query, group, slot), or -1
  unsigned char* part;  // [tiles, qt] records of attn_rec_bytes(G, d) bytes, tile-major
};
// One partial record per (query, group, slot): the G heads' normalised O rows
// (bf16, d each), then their G LSEs (fp32), padded to a multiple of 16 bytes.
__host__ __device__ inline int attn_rec_bytes(int G, int d) { return G * d * 2 + (G + 3) / 4 * 16; }
size_t attn_ws_bytes(int64_t chunk, int64_t nb, int H_q, int H_kv, int d, int k);
AttnWs attn_ws_carve(void* ws, int64_t chunk, int64_t nb, int H_q, int H_kv, int d, int k);
cudaError_t launch_sparse_attn_chunk(const void* q, const void* kk, const void* v,
                                     const int32_t* ids, int64_t N, int64_t q0, int64_t q1,
                                     int H_q, int H_kv, int d, int k, float scale, void* out,
                                     float* lse, const AttnWs& ws, int64_t nb, const Diag& dg,
                                     cudaStream_t st);

// Decode (msa_decode.cu).
cudaError_t launch_decode_index(const void* q_idx, const void* k_idx_pages,
                                const int32_t* page_table, const int32_t* seq_lens, int B,
                                int max_pages, int n_g, int d_idx, float* scores,
                                const Diag& dg, cudaStream_t st);
size_t decode_ws_bytes(int B, int H_q, int d, int k);
cudaError_t launch_decode_attn(const void* q, const void* k_pages, const void* v_pages,
                               int kv_fp8, const float* k_scale, const float* v_scale,
                               const int32_t* page_table, const int32_t* seq_lens,
                               const int32_t* ids, int B, int max_pages, int H_q, int H_kv,
                               int d, int k, float scale, void* out, float* lse, void* ws,
                               const Diag& dg, cudaStream_t st);

}  // namespace msa
