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

// NVFP4 index operands (msa_index.cu): q_idx [N, n_g, d_idx] and k_idx
// [N, d_idx] as E2M1 codes (two per byte, the even dimension in the low
// nibble) with one E4M3 scale per 16 dimensions of a row, decoded exactly into
// bf16 rows in ws (q_idx first, its bytes rounded up to 256, then k_idx), then
// ranked by the bf16 kernel.
cudaError_t launch_index_select_nvfp4(const void* q_codes, const void* q_scales,
                                      const void* k_codes, const void* k_scales, int64_t N,
                                      int n_g, int d_idx, int k, int32_t* block_ids,
                                      float* block_scores, int64_t nb, void* ws, const Diag& dg,
                                      cudaStream_t st);

// One launch per 128 sequences of a packed batch; cu_seqlens is a host
// array [B + 1] of token offsets (msa_index.cu).
cudaError_t launch_index_select_varlen(const void* q_idx, const void* k_idx,
                                       const int64_t* cu_seqlens, int B, int n_g, int d_idx,
                                       int k, int32_t* block_ids, const Diag& dg,
                                       cudaStream_t st);
// Paged k_idx: pages [n_pages, 128, d_idx]; sequence b's queries are rows
// cu_q[b] .. cu_q[b + 1] - 1 of q_idx, its last tokens of kv_lens[b]; its key
// block j is page page_table[b * max_pages + j] (host arrays cu_q, kv_lens).
cudaError_t launch_index_select_paged(const void* q_idx, const void* k_idx_pages,
                                      int64_t n_pages, const int32_t* page_table, int max_pages,
                                      const int64_t* cu_q, const int64_t* kv_lens, int B, int n_g,
                                      int d_idx, int k, int32_t* block_ids, const Diag& dg,
                                      cudaStream_t st);

// Index-branch projections (msa_proj.cu): q_idx [N, n_g * d_idx] = x W_qidx^T,
// k_idx [N, d_idx] = x W_kidx^T; x [N, d_model], weights [out, d_model], bf16.
cudaError_t launch_index_project(const void* x, const void* w_qidx, const void* w_kidx,
                                 int64_t N, int d_model, int n_g, int d_idx, void* q_idx,
                                 void* k_idx, const Diag& dg, cudaStream_t st);

// Exp-free top-k over block scores (msa_topk.cu).
// ld: row stride of S in floats (0: nb); rows are read at S + r * ld.
cudaError_t launch_topk(const float* S, int64_t N, int n_g, int64_t nb, int Bk, int k,
                        int64_t q_offset, const int32_t* seq_lens, int32_t* ids, const Diag& dg,
                        cudaStream_t st, int64_t ld = 0);

// Main branch, prefill (msa_attn.cu).
struct AttnWs {
  int32_t* counts;    // [n_g * nb]
  int32_t* offsets;   // [n_g * nb + 1]
  int32_t* cursor;    // [n_g * nb]
  int32_t* tile_off;  // [n_g * nb + 1]
  int32_t* percta;    // [bucketing CTAs, n_g * nb] per-CTA counts, then first positions
  int32_t* entries;   // [chunk * n_g * k]
  int4* tinfo;        // per tile: K / V row, first entry, queries | group << 8, end tile
  int32_t* tbase;     // per tile: query row at the block's first key (paged batches only)
  int32_t* rec_of;    // [chunk, n_g, k]: partial record of each (query, group, slot), or -1
  unsigned char* part;  // [tiles, qt] records of attn_rec_bytes(G, d) bytes, tile-major,
                        // then (shared pass) one record per (query, group) of the chunk
  // shared-block pass (null when not carved): per (query, group) row of the
  // chunk, the slots it covers (bits 0-15) and the tile's shared blocks the
  // row selected (bits 16-31); per (query tile, group) its shared blocks
  int32_t* rowmask = nullptr;  // [chunk, n_g]
  int32_t* shlist = nullptr;   // [query tiles, n_g, 16], -1 padded
  int64_t shared_rec0 = 0;     // first shared record in part
};
// One partial record per (query, group, slot): the G heads' normalised O rows
// (bf16, d each), then their G LSEs (fp32), padded to a multiple of 16 bytes.
__host__ __device__ inline int attn_rec_bytes(int G, int d) { return G * d * 2 + (G + 3) / 4 * 16; }
// with_tbase: room for the per-tile query bases that paged K / V needs
// with_shared: room for the shared-block pass of single-sequence calls
size_t attn_ws_bytes(int64_t chunk, int64_t nb, int H_q, int H_kv, int d, int k,
                     bool with_tbase = false, bool with_shared = false);
AttnWs attn_ws_carve(void* ws, int64_t chunk, int64_t nb, int H_q, int H_kv, int d, int k,
                     bool with_tbase = false, bool with_shared = false);

// Geometry of a batch of sequences for the main branch. All null: one
// sequence whose query row t sits at position t and whose block b starts at
// K / V row 128 b. Otherwise blocks are numbered per batch ("virtual blocks",
// each sequence's blocks consecutive from its first virtual block) and
//   qinfo[t] = {first virtual block of query row t's sequence, t's position},
//   vinfo[v] = {K / V row of block v's first key,
//               query row that would sit at that key's position}.
// Packed sequences keep queries and keys in the same rows, so the two fields
// of vinfo agree; paged K / V (kv_rows rows of pages) is where they differ.
struct AttnBatch {
  const int2* qinfo = nullptr;
  const int2* vinfo = nullptr;
  int64_t kv_rows = 0;  // rows of the K / V tensors (0: as many as query rows)
  bool paged = false;
};
// Bucketing of query rows q0 .. q1 - 1 by (group, block): fills ws.counts ..
// ws.tinfo (and ws.tbase when paged) and ws.rec_of, the tile layout the tile
// kernels below read. A tile is one bucket's block against up to 128 / G of
// its queries; query i of tile T owns partial record T * (128 / G) + i.
cudaError_t launch_bucketing(const int32_t* ids, int64_t q0, int64_t q1, int H_q, int H_kv,
                             int k, const AttnWs& ws, int64_t nb, const Diag& dg, cudaStream_t st,
                             const AttnBatch& bt = AttnBatch());
cudaError_t launch_sparse_attn_chunk(const void* q, const void* kk, const void* v,
                                     const int32_t* ids, int64_t N, int64_t q0, int64_t q1,
                                     int H_q, int H_kv, int d, int k, float scale, void* out,
                                     float* lse, const AttnWs& ws, int64_t nb, const Diag& dg,
                                     cudaStream_t st, const AttnBatch& bt = AttnBatch());

// KL alignment signal (msa_kl.cu) for query rows q0 .. q1 - 1 of one
// sequence: bucketing as for the main branch, the KL tiles into ws.part (32
// bytes per record), the merge into kl[t * H_kv + g]. G = H_q / H_kv in
// {1, 2, 4, 8}.
cudaError_t launch_kl_chunk(const void* q, const void* kk, const void* q_idx, const void* k_idx,
                            const int32_t* ids, const float* lse, int64_t N, int64_t q0,
                            int64_t q1, int H_q, int H_kv, int d, int d_idx, int k, float scale,
                            float* kl, const AttnWs& ws, int64_t nb, const Diag& dg,
                            cudaStream_t st);

// Sequences of a batch for the main branch's geometry, at most kBatchSeqs
// per launch of launch_batch_info.
constexpr int kBatchSeqs = 128;
struct BatchSeqs {
  int B;
  int32_t q_start[kBatchSeqs];   // first query row
  int32_t q_len[kBatchSeqs];     // query rows
  int32_t q_off[kBatchSeqs];     // position of the first query (keys before it are cached)
  int32_t vb[kBatchSeqs];        // first virtual block
  int32_t n_blk[kBatchSeqs];     // blocks of the sequence's keys
  int32_t kv_start[kBatchSeqs];  // packed: first K / V row; paged: first page-table entry
};
// fills qinfo / vinfo (AttnBatch) for the sequences of tb; page_table null:
// packed K / V; else block j of a sequence starts at K / V row
// page_table[kv_start + j] * page_rows
cudaError_t launch_batch_info(const BatchSeqs& tb, const int32_t* page_table, int page_rows,
                              int2* qinfo, int2* vinfo, cudaStream_t st);

// Decode (msa_decode.cu).
// e4m3: q_idx and the k_idx pages hold E4M3 codes, and the block scores are
// written times score_scale. ss: row stride of scores in floats (0: max_pages).
cudaError_t launch_decode_index(const void* q_idx, const void* k_idx_pages,
                                const int32_t* page_table, const int32_t* seq_lens, int B,
                                int max_pages, int n_g, int d_idx, float* scores,
                                const Diag& dg, cudaStream_t st, bool e4m3 = false,
                                float score_scale = 1.f, int64_t ss = 0);
// NVFP4 k_idx cache: codes [P, 128, d_idx / 2] (two E2M1 per byte, even
// dimension low), kscales [P, 128, d_idx / 16] E4M3 micro-block scales;
// q_idx bf16. Scores written times score_scale.
cudaError_t launch_decode_index_fp4(const void* q_idx, const void* codes, const void* kscales,
                                    const int32_t* page_table, const int32_t* seq_lens, int B,
                                    int max_pages, int n_g, int d_idx, float score_scale,
                                    float* scores, const Diag& dg, cudaStream_t st,
                                    int64_t ss = 0);
size_t decode_ws_bytes(int B, int H_q, int d, int k);
cudaError_t launch_decode_attn(const void* q, const void* k_pages, const void* v_pages,
                               int kv_fp8, const float* k_scale, const float* v_scale,
                               const int32_t* page_table, const int32_t* seq_lens,
                               const int32_t* ids, int B, int max_pages, int H_q, int H_kv,
                               int d, int k, float scale, void* out, float* lse, void* ws,
                               const Diag& dg, cudaStream_t st);
// decode attention over NVFP4 K / V pages (E2M1 codes, one E4M3 scale per 16
// dimensions of a row), split-KV partials in ws and their merge
cudaError_t launch_decode_attn_fp4(const void* q, const void* k_codes, const void* k_scales,
                                   const void* v_codes, const void* v_scales,
                                   const int32_t* page_table, const int32_t* seq_lens,
                                   const int32_t* ids, int B, int max_pages, int H_q, int H_kv,
                                   int d, int k, float scale, void* out, float* lse, void* ws,
                                   const Diag& dg, cudaStream_t st);

}  // namespace msa
