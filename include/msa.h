/* msa.h - C ABI of the MiniMax Sparse Attention (MSA) forward path on GB300.
 *
 * The method, as defined by "MiniMax Sparse Attention (MSA): a Two-Branch
 * Block-Sparse Attention Trained on a 109B-Parameter MoE With a 3T-Token Budget"
 * (Chinese edition; sections "什么是 MSA" / what MSA is, "两个分支如何工作" /
 * how the two branches work, "内核协同设计" / kernel co-design, "运行 Kernel" /
 * running the kernel):
 *
 *  index branch  one index-query head per GQA group scores every causally
 *                visible key of one shared index-key head; the scores are
 *                max-pooled to blocks of Bk tokens; per (query, group) the k
 *                best blocks are kept, the query's own block always among them.
 *  main branch   every query head of the group runs exact scaled-dot-product
 *                softmax attention over the causally visible tokens of exactly
 *                those blocks.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, contiguous,
 *    row-major, 16-byte aligned. The library never allocates, frees or
 *    synchronises: it enqueues kernels on `stream` (a cudaStream_t passed as
 *    void*, NULL = legacy default stream) and returns.
 *  - bf16 tensors are passed as void* (IEEE bfloat16 bit patterns).
 *  - Head h of the main branch belongs to GQA group g = h / (H_q / H_kv); the
 *    index branch has one index-query head per group (n_groups = H_kv).
 *  - Block ids are int32, sorted ascending, padded with -1 at the end; the
 *    query's local block (position / Bk) is always present. Among candidate
 *    blocks of equal score the lower block id wins.
 *  - Scores are raw dot products of the index heads (no scale, no activation);
 *    they are accumulated in fp32. The main branch accumulates in fp32, feeds
 *    the tensor cores bf16 (or E4M3-dequantised) operands, and returns bf16
 *    outputs and fp32 natural-log LSE = log(sum_j exp(scale * q . k_j)).
 *  - Supported by the kernels: Bk = 128, 1 <= k <= 16, d and d_idx in {64, 128},
 *    H_q a multiple of H_kv with 128 % (H_q / H_kv) == 0. Other values return
 *    MSA_ERR_UNSUPPORTED. Inputs must be finite.
 *  - Errors are returned, never thrown; nothing is enqueued when an argument
 *    check fails. A kernel whose bounded wait expires records MSA_ERR_TIMEOUT
 *    in a device error word that msa_get_error() reads.
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = -1, /* null pointer, bad size, misalignment            */
  MSA_ERR_UNSUPPORTED = -2, /* valid for the method, not for these kernels      */
  MSA_ERR_WORKSPACE = -3,   /* workspace smaller than *_workspace_bytes()       */
  MSA_ERR_CUDA = -4,        /* a launch or runtime call failed                  */
  MSA_ERR_TIMEOUT = -5      /* a bounded device wait gave up (see msa_get_error) */
};

enum { MSA_KV_BF16 = 0, MSA_KV_E4M3 = 1 };

/* Human-readable name of a status code (static string). */
const char* msa_status_string(int status);

/* Library version, for load checks: 0xMMmmpp. */
int msa_version(void);

/* ---------------------------------------------------------------- prefill -- */

/* Workspace bytes msa_index_select needs (0 today; kept for ABI stability). */
size_t msa_index_select_workspace_bytes(int64_t N, int n_groups, int d_idx, int Bk, int k);

/* Index branch of prefill: block selection for every (query, group).
 *   q_idx        [N, n_groups, d_idx] bf16  index queries (one head per group)
 *   k_idx        [N, d_idx] bf16            shared index keys
 *   block_ids    [N, n_groups, k] int32     out: selected blocks (see above)
 *   block_scores [N, n_groups, nb] fp32     out, optional (NULL to skip),
 *                nb = ceil(N / Bk): S[t, g, b] = max over the visible keys of
 *                block b of q_idx[t, g] . k_idx[j] for b <= t / Bk; entries
 *                b > t / Bk are left untouched.
 * The N x N score matrix is never materialised: scores are pooled and ranked
 * as they come out of the tensor cores. */
int msa_index_select(const void* q_idx, const void* k_idx, int64_t N, int n_groups,
                     int d_idx, int Bk, int k, int32_t* block_ids, float* block_scores,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Index-branch projections: the two projection matrices the index branch adds
 * to a GQA layer ("MiniMax Sparse Attention (MSA) ...", section "两个分支如何工作":
 * one index-query head per group, one shared index-key head), read as plain
 * linear maps of the layer input (no bias, no activation):
 *   x       [N, d_model] bf16                  layer input
 *   w_qidx  [n_groups * d_idx, d_model] bf16   [out, in]; rows g*d_idx .. give group g
 *   w_kidx  [d_idx, d_model] bf16              [out, in]
 *   q_idx   [N, n_groups, d_idx] bf16 out      q_idx[t,g,c] = sum_m x[t,m] w_qidx[g*d_idx+c, m]
 *   k_idx   [N, d_idx] bf16 out                k_idx[t,c]   = sum_m x[t,m] w_kidx[c, m]
 * One tensor-core GEMM over both weight matrices, fp32 accumulation, each
 * output rounded once to bf16; the outputs feed msa_index_select directly.
 * d_model must be a multiple of 8 and d_idx in {64, 128} (MSA_ERR_UNSUPPORTED
 * otherwise); every tensor 16-byte aligned (MSA_ERR_INVALID_ARG otherwise). */
int msa_index_project(const void* x, const void* w_qidx, const void* w_kidx, int64_t N,
                      int d_model, int n_groups, int d_idx, void* q_idx, void* k_idx,
                      void* stream);

/* Index branch with FP8-E4M3 index operands (the kernel release lists FP8 among
 * its precisions: "MiniMax lança MSA ...", section "Kernel open source e
 * MiniMax-M3"):
 *   q_idx   [N, n_groups, 128] E4M3 codes, k_idx [N, 128] E4M3 codes
 *   (d_idx must be 128: MSA_ERR_UNSUPPORTED otherwise).
 * The scores are the dot products of the decoded codes, exact per product and
 * accumulated in fp32 on the tensor cores (kind::f8f6f4). A positive scale of
 * a whole q_idx row or of the whole k_idx tensor changes no ranking, so the
 * selection depends on the codes alone; score_scale (say, the product of the
 * two dequantisation scales) only multiplies the optional block_scores.
 * Selection rules, outputs and errors otherwise as msa_index_select. */
int msa_index_select_fp8(const void* q_idx, const void* k_idx, int64_t N, int n_groups,
                         int d_idx, int Bk, int k, int32_t* block_ids, float* block_scores,
                         float score_scale, void* stream);

/* Index branch with NVFP4 index operands (the kernel release lists NVFP4
 * among its precisions: "MiniMax lança MSA ...", section "Kernel open source e
 * MiniMax-M3"; "MiniMax Sparse Attention (MSA) ...", section "内核协同设计"):
 *   q_codes  [N, n_groups, d_idx / 2] uint8   E2M1 codes, two per byte, the
 *                                             even dimension in the low nibble
 *   q_scales [N, n_groups, d_idx / 16] uint8  E4M3 scale of each 16 dimensions
 *   k_codes  [N, d_idx / 2] uint8, k_scales [N, d_idx / 16] uint8, the same
 * A value is its E2M1 code's value times its 16 dimensions' scale (plain FP4,
 * E2M1 codes without block scaling, is every scale code 0x38 = 1.0). Such a
 * product has at most six significant bits and lies within bf16's range, so
 * the operands are decoded exactly into bf16 rows in the workspace (device,
 * caller-owned, msa_index_select_nvfp4_workspace_bytes() bytes, 16-byte
 * aligned; MSA_ERR_WORKSPACE when smaller) and ranked by the bf16 index
 * kernel: the result equals msa_index_select on the decoded values. The
 * tensor cores run bf16, not block-scaled FP4, MMAs. Selection rules,
 * block_scores, alignment and other errors as msa_index_select. */
size_t msa_index_select_nvfp4_workspace_bytes(int64_t N, int n_groups, int d_idx);
int msa_index_select_nvfp4(const void* q_codes, const void* q_scales, const void* k_codes,
                           const void* k_scales, int64_t N, int n_groups, int d_idx, int Bk,
                           int k, int32_t* block_ids, float* block_scores, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Exp-free top-k over given block scores ("内核协同设计": ranking raw scores
 * selects the same blocks as ranking their softmax).
 *   block_scores [n_rows / n_groups... ] laid out [N, n_groups, nb] fp32; row
 *                (t, g) is a query at position t + q_offset, or, when seq_lens
 *                is not NULL, at position seq_lens[t] - 1 (decode: one row
 *                per sequence t); only b <= position / Bk is read.
 *   block_ids    [N, n_groups, k] int32 out.
 * Requires position / Bk < nb for every row; N * n_groups above 2^31 - 1 rows
 * returns MSA_ERR_UNSUPPORTED. */
int msa_topk_blocks(const float* block_scores, int64_t N, int n_groups, int64_t nb, int Bk,
                    int k, int64_t q_offset, const int32_t* seq_lens, int32_t* block_ids,
                    void* stream);

/* Workspace bytes msa_sparse_attn needs to process up to `chunk_rows` query
 * positions per pass (chunk_rows = N: one pass). Larger workspaces let the
 * call take fewer, longer passes. */
size_t msa_sparse_attn_workspace_bytes(int64_t chunk_rows, int64_t N, int H_q, int H_kv, int d,
                                       int Bk, int k);

/* Main branch of prefill: exact softmax attention of every query head over
 * the causally visible tokens of its group's selected blocks.
 *   q          [N, H_q, d] bf16
 *   k, v       [N, H_kv, d] bf16
 *   block_ids  [N, H_kv, k] int32 (as produced by msa_index_select)
 *   scale      softmax scale (the method uses 1 / sqrt(d))
 *   out        [N, H_q, d] bf16 out
 *   lse        [N, H_q] fp32 out (may be NULL)
 *   workspace  at least msa_sparse_attn_workspace_bytes(c, ...) for some c >= 1;
 *              the call picks the largest chunk that fits.
 * Block ids must be valid for their row: -1 or 0 <= id <= t / Bk. */
int msa_sparse_attn(const void* q, const void* k, const void* v, const int32_t* block_ids,
                    int64_t N, int H_q, int H_kv, int d, int Bk, int topk, float scale,
                    void* out, float* lse, void* workspace, size_t workspace_bytes,
                    void* stream);

/* KL alignment signal of the index branch, forward only ("MiniMax Sparse
 * Attention (MSA) ...", section "MSA 如何训练"; "MiniMax lança MSA ...", section
 * "Treinamento com KL Divergence"): per (t, g), over the causally visible
 * tokens J of the group's selected blocks, the teacher is the main branch's
 * distribution averaged over the group's query heads,
 *   p_main(j) = (1/G) sum_h exp(scale q_h . k_j - lse_h),
 * and the student is the softmax of the raw index scores over the same tokens,
 *   p_idx(j) = exp(s_j) / sum_J exp(s_j),  s_j = q_idx[t, g] . k_idx[j].
 *   kl[t, g] = sum_J p_main(j) (log p_main(j) - log p_idx(j))   fp32 out [N, H_kv]
 *   lse          [N, H_q] fp32: the main branch's LSE on the same block ids
 *                (msa_sparse_attn)
 *   q, k, q_idx, k_idx, block_ids as in msa_sparse_attn / msa_index_select;
 *   d and d_idx in {64, 128}, G = H_q / H_kv in {1, 2, 4, 8}, else
 *   MSA_ERR_UNSUPPORTED.
 *   workspace    at least msa_kl_teacher_workspace_bytes(c, ...) for some c >= 1
 *                (the main branch's bucketing; the call takes the largest chunk
 *                of query rows that fits). */
size_t msa_kl_teacher_workspace_bytes(int64_t chunk_rows, int64_t N, int H_q, int H_kv, int d,
                                      int Bk, int k);
int msa_kl_teacher(const void* q, const void* k, const void* q_idx, const void* k_idx,
                   const int32_t* block_ids, const float* lse, int64_t N, int H_q, int H_kv,
                   int d, int d_idx, int Bk, int topk, float scale, float* kl, void* workspace,
                   size_t workspace_bytes, void* stream);

/* Varlen batched prefill: B sequences packed back to back, the serving form of
 * the two prefill entry points above (the usage listing of the MSA page,
 * "运行 Kernel", plans each call from per-sequence query and key lengths).
 * Sequence b holds rows cu_seqlens[b] .. cu_seqlens[b + 1] - 1 of every tensor;
 * its queries see only its own keys, and its block ids count blocks from its
 * own first token.
 *   cu_seqlens  host int64 [B + 1] with 0 = cu_seqlens[0] <= ... <= cu_seqlens[B]
 *               (MSA_ERR_INVALID_ARG otherwise)
 * Other tensors as in msa_index_select / msa_sparse_attn with N = cu_seqlens[B].
 * Index branch: one launch per 128 sequences; the row tiles of all of them
 * form one heaviest-first schedule over the SMs, so short sequences fill the
 * gaps that long ones leave. Main branch: one pass over the whole batch (its
 * buckets are the blocks of every sequence), in chunks of query rows when the
 * workspace is smaller than msa_sparse_attn_varlen_workspace_bytes.
 * Tensors must be 16-byte aligned (MSA_ERR_INVALID_ARG); N * n_groups must
 * stay below 2^31 (MSA_ERR_UNSUPPORTED). */
int msa_index_select_varlen(const void* q_idx, const void* k_idx, const int64_t* cu_seqlens,
                            int B, int n_groups, int d_idx, int Bk, int k, int32_t* block_ids,
                            void* stream);

/* Workspace for msa_sparse_attn_varlen to take the whole batch in one pass;
 * 0 when cu_seqlens is invalid or holds no token. A smaller workspace works in
 * chunks of query rows as long as it holds 16 bytes per token plus one
 * chunk's bucketing and partials (MSA_ERR_WORKSPACE otherwise). */
size_t msa_sparse_attn_varlen_workspace_bytes(const int64_t* cu_seqlens, int B, int H_q,
                                              int H_kv, int d, int Bk, int k);

int msa_sparse_attn_varlen(const void* q, const void* k, const void* v, const int32_t* block_ids,
                           const int64_t* cu_seqlens, int B, int H_q, int H_kv, int d, int Bk,
                           int topk, float scale, void* out, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------- paged prefill -- */

/* Prefill over paged caches (chunked prefill): sequence b holds kv_lens[b]
 * tokens, already written to the caches, of which the last
 * cu_q[b + 1] - cu_q[b] are its queries, packed back to back as rows cu_q[b] ..
 * cu_q[b + 1] - 1 of q_idx / q / out / lse / block_ids. Query i of sequence b
 * sits at position kv_lens[b] - (cu_q[b + 1] - cu_q[b]) + i and sees the keys
 * at positions 0 .. its own. Logical block j of sequence b is physical page
 * page_table[b * max_pages + j] (device int32 [B, max_pages]), the layout the
 * decode entry points below use ("运行 Kernel" of the MSA page plans its calls
 * from per-sequence query and key lengths over paged KV with page size = block
 * size). Block ids count from the sequence's first token, as in decode; with
 * kv_lens[b] equal to the query count every sequence is a plain varlen
 * sequence, and the results are those of msa_*_varlen.
 *   cu_q       host int64 [B + 1], 0 = cu_q[0] <= ... <= cu_q[B]
 *   kv_lens    host int64 [B], queries of b <= kv_lens[b] <= max_pages * Bk
 *              (MSA_ERR_INVALID_ARG otherwise)
 *   n_pages    pages P of the cache tensors; page ids outside 0 .. P - 1 read
 *              zeros (the caller keeps the table valid)
 * Sizes: cu_q[B] * n_groups and P * Bk (index), P * H_kv * Bk (main branch)
 * and B * max_pages below 2^31, else MSA_ERR_UNSUPPORTED. */

/* Index branch.
 *   q_idx        [cu_q[B], n_groups, d_idx] bf16
 *   k_idx_pages  [P, Bk, d_idx] bf16
 *   block_ids    [cu_q[B], n_groups, k] int32 out
 * One launch per 128 sequences; tiles are ordered by their row-tile index
 * within the sequence (the cached prefix adds the same key blocks to every
 * tile of a sequence). */
int msa_index_select_paged(const void* q_idx, const void* k_idx_pages, int64_t n_pages,
                           const int32_t* page_table, int max_pages, const int64_t* cu_q,
                           const int64_t* kv_lens, int B, int n_groups, int d_idx, int Bk, int k,
                           int32_t* block_ids, void* stream);

/* Workspace for msa_sparse_attn_paged in one pass; 0 on invalid lengths or
 * no query. Smaller workspaces work in chunks, as for varlen. */
size_t msa_sparse_attn_paged_workspace_bytes(const int64_t* cu_q, const int64_t* kv_lens, int B,
                                             int max_pages, int H_q, int H_kv, int d, int Bk,
                                             int k);

/* Main branch.
 *   q            [cu_q[B], H_q, d] bf16
 *   k_pages      [P, H_kv, Bk, d] bf16 (the decode layout)
 *   v_pages      same
 *   block_ids    [cu_q[B], H_kv, k] int32 (msa_index_select_paged)
 *   out, lse     [cu_q[B], H_q, d] bf16, [cu_q[B], H_q] fp32 (lse may be NULL)
 * Other arguments as in msa_sparse_attn. */
int msa_sparse_attn_paged(const void* q, const void* k_pages, const void* v_pages,
                          int64_t n_pages, const int32_t* page_table, int max_pages,
                          const int32_t* block_ids, const int64_t* cu_q, const int64_t* kv_lens,
                          int B, int H_q, int H_kv, int d, int Bk, int topk, float scale,
                          void* out, float* lse, void* workspace, size_t workspace_bytes,
                          void* stream);

/* ----------------------------------------------------------------- decode -- */

/* Paged caches ("运行 Kernel": page size = block size; the page tensor's second
 * dimension is the number of kv heads, so pages are head-major). Sequence s holds
 * seq_lens[s] tokens; its logical block b lives in physical page
 * page_table[s * max_pages + b]. The new token is the last one (position
 * seq_lens[s] - 1) and must already be written to the caches.
 * The decode entry points take no page count, so they cannot check page ids:
 * every entry page_table[s * max_pages + b] with b <= (seq_lens[s] - 1) / Bk
 * must name a page of the caches passed (0 <= id < P). A page id outside them
 * is read as an address, with undefined results. Sequence lengths and block
 * ids ARE checked on the device (see msa_get_error). */

/* Workspace bytes of the decode index branch: the block scores, B * n_groups
 * rows of max_pages fp32 each, every row padded to a multiple of 4 floats
 * (16-byte aligned rows, which the top-k reads as vectors). */
size_t msa_index_select_decode_workspace_bytes(int B, int max_pages, int n_groups);

/* Index branch of decode, one query per sequence.
 *   q_idx        [B, n_groups, d_idx] bf16
 *   k_idx_pages  [P, Bk, d_idx] bf16 paged shared index keys
 *   page_table   [B, max_pages] int32; seq_lens [B] int32 (>= 1)
 *   block_ids    [B, n_groups, k] int32 out
 *   block_scores [B, n_groups, max_pages] fp32 out, optional (NULL: kept in
 *                the workspace); visible entries b <= (seq_lens[s]-1) / Bk. */
int msa_index_select_decode(const void* q_idx, const void* k_idx_pages,
                            const int32_t* page_table, const int32_t* seq_lens, int B,
                            int max_pages, int n_groups, int d_idx, int Bk, int k,
                            int32_t* block_ids, float* block_scores, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Index branch of decode over an FP8-E4M3 k_idx cache: q_idx [B, n_groups,
 * d_idx] and k_idx_pages [P, Bk, d_idx] hold E4M3 codes (half the bytes of the
 * scan, which dominates a decode step). Scores are the dot products of the
 * decoded codes, exact per product and accumulated in fp32 (mma.m16n8k32 on
 * E4M3). A positive scale of all keys or of a query's row ranks the blocks
 * the same, so the selection depends on the codes alone; score_scale only
 * multiplies the optional block_scores. Everything else as
 * msa_index_select_decode. */
int msa_index_select_decode_fp8(const void* q_idx, const void* k_idx_pages,
                                const int32_t* page_table, const int32_t* seq_lens, int B,
                                int max_pages, int n_groups, int d_idx, int Bk, int k,
                                int32_t* block_ids, float* block_scores, float score_scale,
                                void* workspace, size_t workspace_bytes, void* stream);

/* Index branch of decode over an NVFP4 k_idx cache (the kernel release lists
 * NVFP4 and FP4 among its precisions: "MiniMax lança MSA ...", section "Kernel
 * open source e MiniMax-M3"; a quarter of the bf16 scan's bytes plus one scale
 * byte per 16 dimensions):
 *   k_idx_codes   [P, Bk, d_idx / 2] uint8: two OCP E2M1 codes per byte, the
 *                 even dimension in the low nibble
 *   k_idx_scales  [P, Bk, d_idx / 16] uint8: one E4M3 scale per 16 consecutive
 *                 dimensions of a key; key value = e2m1 * scale
 *   q_idx         [B, n_groups, d_idx] bf16, rounded to f16 for the products
 *                 (exact for |x| >= 2^-14 and below 65504 with 8 significant
 *                 bits, which every bf16 value in that range has)
 * A tensor-wide scale changes no ranking; score_scale only multiplies the
 * optional block_scores. Everything else as msa_index_select_decode. */
int msa_index_select_decode_nvfp4(const void* q_idx, const void* k_idx_codes,
                                  const void* k_idx_scales, const int32_t* page_table,
                                  const int32_t* seq_lens, int B, int max_pages, int n_groups,
                                  int d_idx, int Bk, int k, int32_t* block_ids,
                                  float* block_scores, float score_scale, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Workspace bytes of msa_decode (split-KV partials). */
size_t msa_decode_workspace_bytes(int B, int H_q, int d, int k);

/* Main branch of decode over a paged bf16 or FP8-E4M3 KV cache.
 *   q              [B, H_q, d] bf16
 *   k_pages        [P, H_kv, Bk, d] bf16 or E4M3 bytes (kv_dtype)
 *   v_pages        same layout and dtype
 *   k_scale        [H_kv] fp32 per-kv-head dequantisation scale (E4M3 only;
 *   v_scale        K or V value = code * scale); ignored for bf16
 *   block_ids      [B, H_kv, k] int32 (msa_index_select_decode)
 *   out            [B, H_q, d] bf16 out; lse [B, H_q] fp32 out (may be NULL) */
int msa_decode(const void* q, const void* k_pages, const void* v_pages, int kv_dtype,
               const float* k_scale, const float* v_scale, const int32_t* page_table,
               const int32_t* seq_lens, const int32_t* block_ids, int B, int max_pages,
               int H_q, int H_kv, int d, int Bk, int k, float scale, void* out, float* lse,
               void* workspace, size_t workspace_bytes, void* stream);

/* Main branch of decode over an NVFP4 KV cache (the kernel release lists NVFP4
 * and FP4 among its precisions: "MiniMax lança MSA ...", section "Kernel open
 * source e MiniMax-M3"; about a quarter of the bf16 cache's bytes plus one scale
 * byte per 16 elements):
 *   k_codes, v_codes    [P, H_kv, Bk, d / 2] uint8: two OCP E2M1 codes per byte,
 *                       the even dimension in the low nibble
 *   k_scales, v_scales  [P, H_kv, Bk, d / 16] uint8: one E4M3 scale per 16
 *                       consecutive dimensions of a row; value = e2m1 * scale
 *   q                   [B, H_q, d] bf16, rounded to f16 for q . K^T (exact for
 *                       |x| >= 2^-14 and below 65504, where every bf16 value
 *                       fits f16's 11 significant bits)
 * The attention itself is that of msa_decode on the decoded values (every
 * E2M1 code times an E4M3 scale is a bf16 value). Workspace:
 * msa_decode_workspace_bytes. Every device pointer is 16-byte aligned and owned
 * by the caller. Errors as msa_decode: MSA_ERR_INVALID_ARG for a null or
 * misaligned pointer or H_q not a multiple of H_kv, MSA_ERR_UNSUPPORTED for
 * Bk != 128, d not 64 or 128, k above the largest top-k or more than 8 query
 * heads per kv head, MSA_ERR_WORKSPACE for a missing or short workspace; block
 * ids and sequence lengths are checked on the device (skipped and reported
 * through msa_get_error). */
int msa_decode_nvfp4(const void* q, const void* k_codes, const void* k_scales,
                     const void* v_codes, const void* v_scales, const int32_t* page_table,
                     const int32_t* seq_lens, const int32_t* block_ids, int B, int max_pages,
                     int H_q, int H_kv, int d, int Bk, int k, float scale, void* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Decode index branch without any allocation (no counterpart in the pages):
 * same inputs, output and rules as msa_index_select_decode, but the per-page
 * block scores go to a fixed 4 MiB scratch array compiled into the library
 * instead of a caller workspace. For callers that may not allocate device
 * memory while running (engines that reserve all memory at start-up, code
 * where an allocation could stall or synchronise other device work).
 *   - B * n_groups * max_pages must not exceed
 *     msa_index_select_decode_noalloc_max_scores() (1 << 20); larger requests
 *     return MSA_ERR_WORKSPACE and enqueue nothing.
 *   - The first call on a device looks up the array's device address (a
 *     cudaGetSymbolAddress, no allocation); make that first call before any
 *     stream capture. With CUDA's default lazy module loading that first
 *     call is also when the driver loads this library's kernels and commits
 *     the 4 MiB array in device memory, which can fail (MSA_ERR_CUDA) once
 *     the caller has reserved all device memory. Make one warm-up call at
 *     start-up, before reserving memory, or load modules eagerly
 *     (CUDA_MODULE_LOADING=EAGER).
 *   - All calls share the array: calls whose executions overlap on the GPU
 *     (several streams or host threads) race and must be serialised.
 *   - Calls no cudaMalloc / cudaFree and no allocating library routine. */
int msa_index_select_decode_noalloc(const void* q_idx, const void* k_idx_pages,
                                    const int32_t* page_table, const int32_t* seq_lens, int B,
                                    int max_pages, int n_groups, int d_idx, int Bk, int k,
                                    int32_t* block_ids, void* stream);

/* Capacity of that scratch array, in block scores. */
int64_t msa_index_select_decode_noalloc_max_scores(void);

/* ------------------------------------------------------------ diagnostics -- */

/* Synchronises `stream`, then returns and clears the device error word:
 * MSA_OK; MSA_ERR_TIMEOUT if a bounded wait expired; MSA_ERR_INVALID_ARG if a
 * kernel met device-side data it cannot use (a block id outside 0..t/Bk, a
 * sequence length outside 1..max_pages*Bk) and skipped it. The first error
 * since the last call is kept. */
int msa_get_error(void* stream);

/* Number of kernel launches (and device memsets) this library has enqueued
 * since it was loaded, on all streams; for accounting in benchmarks. */
int64_t msa_launch_count(void);

/* Iteration limit of every bounded device wait (default 1 << 26 polls, or
 * the MSA_WAIT_LIMIT environment variable read when the library loads).
 * Lower values make waits give up sooner; for fault tests. Returns the
 * previous value. */
int64_t msa_set_wait_limit(int64_t polls);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
