// C ABI of libmsa (declared in include/msa.h): argument checks, workspace
// carving and kernel launches. No allocation, no synchronisation (except in
// msa_get_error), no exceptions.
#include <stdlib.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/msa.h"
#include "msa_kernels.h"

namespace msa {
static std::atomic<long long> g_launches{0};
void note_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace msa

namespace {

__device__ int g_msa_error = 0;

long long initial_wait_limit() {
  const char* e = getenv("MSA_WAIT_LIMIT");
  if (e && *e) {
    long long v = atoll(e);
    if (v >= 0) return v;
  }
  return 1ll << 26;
}
long long g_wait_limit = initial_wait_limit();
std::mutex g_mu;
int* g_err_ptr[64] = {nullptr};

// Device address of the error word on the current device (looked up once per
// device; the lookup is not a stream operation).
int* err_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_msa_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = (int*)p;
  }
  return g_err_ptr[dev];
}

msa::Diag diag() { return msa::Diag{err_ptr(), g_wait_limit}; }

}  // namespace

msa::Diag msa::current_diag() { return diag(); }

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int status_of(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA; }

bool supported_k(int k) { return k >= 1 && k <= msa::kMaxK; }
bool supported_d(int d) { return d == 64 || d == 128; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

const char* msa_status_string(int s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
    case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
    case MSA_ERR_TIMEOUT: return "MSA_ERR_TIMEOUT";
    default: return "MSA_ERR_UNKNOWN";
  }
}

int msa_version(void) { return 0x000100; }

size_t msa_index_select_workspace_bytes(int64_t, int, int, int, int) { return 0; }

int msa_index_select(const void* q_idx, const void* k_idx, int64_t N, int n_groups, int d_idx,
                     int Bk, int k, int32_t* block_ids, float* block_scores, void* workspace,
                     size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (N < 0 || n_groups < 1 || d_idx < 1 || Bk < 1 || k < 1) return MSA_ERR_INVALID_ARG;
  if (N == 0) return MSA_OK;
  if (!q_idx || !k_idx || !block_ids) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(block_ids) ||
      (block_scores && !aligned16(block_scores)))
    return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || !supported_k(k) || !supported_d(d_idx)) return MSA_ERR_UNSUPPORTED;
  if (N * n_groups >= (1ll << 31)) return MSA_ERR_UNSUPPORTED;
  int64_t nb = ceil_div(N, Bk);
  return status_of(msa::launch_index_select(q_idx, k_idx, N, n_groups, d_idx, k, block_ids,
                                            block_scores, nb, diag(), (cudaStream_t)stream));
}

int msa_index_project(const void* x, const void* w_qidx, const void* w_kidx, int64_t N,
                      int d_model, int n_groups, int d_idx, void* q_idx, void* k_idx,
                      void* stream) {
  if (N < 0 || d_model < 1 || n_groups < 1 || d_idx < 1) return MSA_ERR_INVALID_ARG;
  if (N == 0) return MSA_OK;
  if (!x || !w_qidx || !w_kidx || !q_idx || !k_idx) return MSA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_qidx) || !aligned16(w_kidx) || !aligned16(q_idx) ||
      !aligned16(k_idx))
    return MSA_ERR_INVALID_ARG;
  if (d_model % 8 != 0 || !supported_d(d_idx) || N >= (1ll << 31) ||
      (int64_t)n_groups * d_idx >= (1 << 20))
    return MSA_ERR_UNSUPPORTED;
  return status_of(msa::launch_index_project(x, w_qidx, w_kidx, N, d_model, n_groups, d_idx,
                                             q_idx, k_idx, diag(), (cudaStream_t)stream));
}

int msa_index_select_fp8(const void* q_idx, const void* k_idx, int64_t N, int n_groups,
                         int d_idx, int Bk, int k, int32_t* block_ids, float* block_scores,
                         float score_scale, void* stream) {
  if (N < 0 || n_groups < 1 || d_idx < 1 || Bk < 1 || k < 1) return MSA_ERR_INVALID_ARG;
  if (N == 0) return MSA_OK;
  if (!q_idx || !k_idx || !block_ids) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(block_ids) ||
      (block_scores && !aligned16(block_scores)))
    return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || !supported_k(k) || d_idx != 128) return MSA_ERR_UNSUPPORTED;
  if (N * n_groups >= (1ll << 31)) return MSA_ERR_UNSUPPORTED;
  int64_t nb = ceil_div(N, Bk);
  return status_of(msa::launch_index_select(q_idx, k_idx, N, n_groups, d_idx, k, block_ids,
                                            block_scores, nb, diag(), (cudaStream_t)stream,
                                            true, score_scale));
}

size_t msa_index_select_nvfp4_workspace_bytes(int64_t N, int n_groups, int d_idx) {
  if (N < 1 || n_groups < 1 || d_idx < 1) return 0;
  const size_t q = (size_t)N * n_groups * d_idx * 2, kb = (size_t)N * d_idx * 2;
  return ((q + 255) & ~(size_t)255) + ((kb + 255) & ~(size_t)255);
}

int msa_index_select_nvfp4(const void* q_codes, const void* q_scales, const void* k_codes,
                           const void* k_scales, int64_t N, int n_groups, int d_idx, int Bk,
                           int k, int32_t* block_ids, float* block_scores, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (N < 0 || n_groups < 1 || d_idx < 1 || Bk < 1 || k < 1) return MSA_ERR_INVALID_ARG;
  if (N == 0) return MSA_OK;
  if (!q_codes || !q_scales || !k_codes || !k_scales || !block_ids || !workspace)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_codes) || !aligned16(k_codes) || !aligned16(block_ids) ||
      !aligned16(workspace) || (block_scores && !aligned16(block_scores)))
    return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || !supported_k(k) || !supported_d(d_idx)) return MSA_ERR_UNSUPPORTED;
  if (N * n_groups >= (1ll << 31)) return MSA_ERR_UNSUPPORTED;
  if (workspace_bytes < msa_index_select_nvfp4_workspace_bytes(N, n_groups, d_idx))
    return MSA_ERR_WORKSPACE;
  int64_t nb = ceil_div(N, Bk);
  return status_of(msa::launch_index_select_nvfp4(q_codes, q_scales, k_codes, k_scales, N,
                                                  n_groups, d_idx, k, block_ids, block_scores,
                                                  nb, workspace, diag(), (cudaStream_t)stream));
}

int msa_topk_blocks(const float* block_scores, int64_t N, int n_groups, int64_t nb, int Bk,
                    int k, int64_t q_offset, const int32_t* seq_lens, int32_t* block_ids,
                    void* stream) {
  if (N < 0 || n_groups < 1 || nb < 1 || Bk < 1 || k < 1 || q_offset < 0)
    return MSA_ERR_INVALID_ARG;
  if (N == 0) return MSA_OK;
  if (!block_scores || !block_ids) return MSA_ERR_INVALID_ARG;
  if (!seq_lens && (N - 1 + q_offset) / Bk >= nb) return MSA_ERR_INVALID_ARG;
  if (!supported_k(k) || N * (int64_t)n_groups > INT32_MAX) return MSA_ERR_UNSUPPORTED;
  return status_of(msa::launch_topk(block_scores, N, n_groups, nb, Bk, k, q_offset, seq_lens,
                                    block_ids, diag(), (cudaStream_t)stream));
}

size_t msa_sparse_attn_workspace_bytes(int64_t chunk_rows, int64_t N, int H_q, int H_kv, int d,
                                       int Bk, int k) {
  if (chunk_rows < 1 || N < 1 || H_kv < 1 || Bk < 1 || k < 1) return 0;
  chunk_rows = std::min(chunk_rows, N);
  return msa::attn_ws_bytes(chunk_rows, ceil_div(N, Bk), H_q, H_kv, d, k, false, true);
}

int msa_sparse_attn(const void* q, const void* k, const void* v, const int32_t* block_ids,
                    int64_t N, int H_q, int H_kv, int d, int Bk, int topk, float scale, void* out,
                    float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (N < 0 || H_q < 1 || H_kv < 1 || d < 1 || Bk < 1 || topk < 1) return MSA_ERR_INVALID_ARG;
  if (N == 0) return MSA_OK;
  if (!q || !k || !v || !block_ids || !out || !workspace) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(workspace) || !aligned16(block_ids) || (lse && !aligned16(lse)))
    return MSA_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return MSA_ERR_INVALID_ARG;
  const int G = H_q / H_kv;
  if (Bk != 128 || !supported_k(topk) || !supported_d(d) || 128 % G != 0)
    return MSA_ERR_UNSUPPORTED;
  if (N >= (1ll << 27) || N * H_q * topk >= (1ll << 31)) return MSA_ERR_UNSUPPORTED;
  const int64_t nb = ceil_div(N, Bk);
  // largest chunk of query rows whose workspace fits
  int64_t lo = 0, hi = N;
  while (lo < hi) {
    int64_t mid = (lo + hi + 1) / 2;
    if (msa::attn_ws_bytes(mid, nb, H_q, H_kv, d, topk, false, true) <= workspace_bytes) lo = mid;
    else hi = mid - 1;
  }
  if (lo < 1) return MSA_ERR_WORKSPACE;
  const int64_t chunk = lo;
  msa::AttnWs ws = msa::attn_ws_carve(workspace, chunk, nb, H_q, H_kv, d, topk, false, true);
  msa::Diag dg = diag();
  for (int64_t q0 = 0; q0 < N; q0 += chunk) {
    int64_t q1 = std::min(N, q0 + chunk);
    cudaError_t e = msa::launch_sparse_attn_chunk(q, k, v, block_ids, N, q0, q1, H_q, H_kv, d,
                                                  topk, scale, out, lse, ws, nb, dg,
                                                  (cudaStream_t)stream);
    if (e != cudaSuccess) return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

// ------------------------------------------------------- KL alignment signal
size_t msa_kl_teacher_workspace_bytes(int64_t chunk_rows, int64_t N, int H_q, int H_kv, int d,
                                      int Bk, int k) {
  return msa_sparse_attn_workspace_bytes(chunk_rows, N, H_q, H_kv, d, Bk, k);
}

int msa_kl_teacher(const void* q, const void* k, const void* q_idx, const void* k_idx,
                   const int32_t* block_ids, const float* lse, int64_t N, int H_q, int H_kv,
                   int d, int d_idx, int Bk, int topk, float scale, float* kl, void* workspace,
                   size_t workspace_bytes, void* stream) {
  if (N < 0 || H_q < 1 || H_kv < 1 || d < 1 || d_idx < 1 || Bk < 1 || topk < 1)
    return MSA_ERR_INVALID_ARG;
  if (N == 0) return MSA_OK;
  if (!q || !k || !q_idx || !k_idx || !block_ids || !lse || !kl || !workspace)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(q_idx) || !aligned16(k_idx) ||
      !aligned16(block_ids) || !aligned16(lse) || !aligned16(kl) || !aligned16(workspace))
    return MSA_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return MSA_ERR_INVALID_ARG;
  const int G = H_q / H_kv;
  if (Bk != 128 || !supported_k(topk) || !supported_d(d) || !supported_d(d_idx) ||
      (G != 1 && G != 2 && G != 4 && G != 8))
    return MSA_ERR_UNSUPPORTED;
  if (N >= (1ll << 27) || N * H_q * topk >= (1ll << 31)) return MSA_ERR_UNSUPPORTED;
  const int64_t nb = ceil_div(N, Bk);
  int64_t lo = 0, hi = N;  // largest chunk of query rows whose workspace fits
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (msa::attn_ws_bytes(mid, nb, H_q, H_kv, d, topk) <= workspace_bytes) lo = mid;
    else hi = mid - 1;
  }
  if (lo < 1) return MSA_ERR_WORKSPACE;
  const int64_t chunk = lo;
  msa::AttnWs ws = msa::attn_ws_carve(workspace, chunk, nb, H_q, H_kv, d, topk);
  const msa::Diag dg = diag();
  for (int64_t q0 = 0; q0 < N; q0 += chunk) {
    const int64_t q1 = std::min(N, q0 + chunk);
    if (msa::launch_kl_chunk(q, k, q_idx, k_idx, block_ids, lse, N, q0, q1, H_q, H_kv, d, d_idx,
                             topk, scale, kl, ws, nb, dg, (cudaStream_t)stream) != cudaSuccess)
      return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

// --------------------------------------------------------------- varlen prefill
// cu_seqlens: host int64 [B + 1], 0 = cu[0] <= cu[1] <= ... <= cu[B]
static bool cu_ok(const int64_t* cu, int B) {
  if (B < 0 || (B > 0 && !cu) || (B > 0 && cu[0] != 0)) return false;
  for (int b = 0; b < B; ++b)
    if (cu[b + 1] < cu[b]) return false;
  return true;
}

}  // extern "C"

namespace {

// A batch for the main branch: queries packed by cu_q (host [B + 1]); keys
// packed the same way (kv_lens null) or paged, sequence b holding kv_lens[b]
// keys of which its queries are the last cu_q[b + 1] - cu_q[b].
struct BatchPlan {
  int64_t n_q = 0;   // query rows
  int64_t nbv = 0;   // virtual blocks: the blocks of every sequence with queries
  size_t fixed = 0;  // workspace bytes of qinfo and vinfo
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// false: bad lengths (a sequence with more queries than keys, or keys past
// its page-table row)
bool plan_batch(const int64_t* cu_q, const int64_t* kv_lens, int B, int max_pages,
                BatchPlan& p) {
  p = BatchPlan();
  for (int b = 0; b < B; ++b) {
    const int64_t nq = cu_q[b + 1] - cu_q[b];
    const int64_t nk = kv_lens ? kv_lens[b] : nq;
    if (nk < nq || (kv_lens && nk > (int64_t)max_pages * 128)) return false;
    if (nq > 0) p.nbv += ceil_div(nk, 128);
  }
  p.n_q = B > 0 ? cu_q[B] : 0;
  p.fixed = align256((size_t)p.n_q * 8) + align256((size_t)p.nbv * 8);
  return true;
}

size_t batch_ws_bytes(const BatchPlan& p, int64_t chunk, int H_q, int H_kv, int d, int k,
                      bool paged) {
  return p.fixed + msa::attn_ws_bytes(std::min(chunk, p.n_q), p.nbv, H_q, H_kv, d, k, paged);
}

int attn_batch(const void* q, const void* k, const void* v, const int32_t* block_ids,
               const int64_t* cu_q, const int64_t* kv_lens, const int32_t* page_table,
               int64_t n_pages, int max_pages, int B, int H_q, int H_kv, int d, int Bk,
               int topk, float scale, void* out, float* lse, void* workspace,
               size_t workspace_bytes, void* stream) {
  if (H_q < 1 || H_kv < 1 || d < 1 || Bk < 1 || topk < 1) return MSA_ERR_INVALID_ARG;
  BatchPlan p;
  if (!plan_batch(cu_q, kv_lens, B, max_pages, p)) return MSA_ERR_INVALID_ARG;
  if (p.n_q == 0) return MSA_OK;
  if (!q || !k || !v || !block_ids || !out || !workspace) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
      !aligned16(workspace) || !aligned16(block_ids) || (lse && !aligned16(lse)))
    return MSA_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return MSA_ERR_INVALID_ARG;
  const int G = H_q / H_kv;
  if (Bk != 128 || !supported_k(topk) || !supported_d(d) || 128 % G != 0)
    return MSA_ERR_UNSUPPORTED;
  const bool paged = page_table != nullptr;
  const int64_t kv_rows = paged ? n_pages * H_kv * 128 : p.n_q;
  if (p.n_q >= (1ll << 27) || p.n_q * H_q * topk >= (1ll << 31) || kv_rows >= (1ll << 31) ||
      p.nbv * H_kv >= (1ll << 31))
    return MSA_ERR_UNSUPPORTED;
  int64_t lo = 0, hi = p.n_q;  // largest chunk of query rows whose workspace fits
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (batch_ws_bytes(p, mid, H_q, H_kv, d, topk, paged) <= workspace_bytes) lo = mid;
    else hi = mid - 1;
  }
  if (lo < 1) return MSA_ERR_WORKSPACE;
  const int64_t chunk = lo;
  unsigned char* w = (unsigned char*)workspace;
  int2* qinfo = (int2*)w;
  int2* vinfo = (int2*)(w + align256((size_t)p.n_q * 8));
  msa::AttnWs ws = msa::attn_ws_carve(w + p.fixed, chunk, p.nbv, H_q, H_kv, d, topk, paged);
  const cudaStream_t st = (cudaStream_t)stream;
  // the batch's geometry, kBatchSeqs sequences per launch
  msa::BatchSeqs tb;
  tb.B = 0;
  int64_t vb = 0;
  for (int b = 0; b <= B; ++b) {
    if (tb.B == msa::kBatchSeqs || (b == B && tb.B > 0)) {
      if (msa::launch_batch_info(tb, page_table, paged ? H_kv * 128 : 0, qinfo, vinfo, st) !=
          cudaSuccess)
        return MSA_ERR_CUDA;
      tb.B = 0;
    }
    if (b == B) break;
    const int64_t nq = cu_q[b + 1] - cu_q[b];
    if (nq == 0) continue;
    const int64_t nk = kv_lens ? kv_lens[b] : nq;
    const int i = tb.B++;
    tb.q_start[i] = (int32_t)cu_q[b];
    tb.q_len[i] = (int32_t)nq;
    tb.q_off[i] = (int32_t)(nk - nq);
    tb.vb[i] = (int32_t)vb;
    tb.n_blk[i] = (int32_t)ceil_div(nk, 128);
    tb.kv_start[i] = (int32_t)(paged ? (int64_t)b * max_pages : cu_q[b]);
    vb += tb.n_blk[i];
  }
  msa::AttnBatch bt;
  bt.qinfo = qinfo;
  bt.vinfo = vinfo;
  bt.kv_rows = kv_rows;
  bt.paged = paged;
  const msa::Diag dg = diag();
  for (int64_t q0 = 0; q0 < p.n_q; q0 += chunk) {
    const int64_t q1 = std::min(p.n_q, q0 + chunk);
    if (msa::launch_sparse_attn_chunk(q, k, v, block_ids, p.n_q, q0, q1, H_q, H_kv, d, topk,
                                      scale, out, lse, ws, p.nbv, dg, st, bt) != cudaSuccess)
      return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

}  // namespace

extern "C" {

size_t msa_sparse_attn_varlen_workspace_bytes(const int64_t* cu_seqlens, int B, int H_q,
                                              int H_kv, int d, int Bk, int k) {
  BatchPlan p;
  if (!cu_ok(cu_seqlens, B) || H_q < 1 || H_kv < 1 || Bk < 1 || k < 1 ||
      !plan_batch(cu_seqlens, nullptr, B, 0, p) || p.n_q == 0)
    return 0;
  return batch_ws_bytes(p, p.n_q, H_q, H_kv, d, k, false);
}

int msa_index_select_varlen(const void* q_idx, const void* k_idx, const int64_t* cu_seqlens,
                            int B, int n_groups, int d_idx, int Bk, int k, int32_t* block_ids,
                            void* stream) {
  if (!cu_ok(cu_seqlens, B) || n_groups < 1 || d_idx < 1 || Bk < 1 || k < 1)
    return MSA_ERR_INVALID_ARG;
  if (B == 0 || cu_seqlens[B] == 0) return MSA_OK;
  if (!q_idx || !k_idx || !block_ids) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(block_ids)) return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || !supported_k(k) || !supported_d(d_idx)) return MSA_ERR_UNSUPPORTED;
  if (cu_seqlens[B] * n_groups >= (1ll << 31)) return MSA_ERR_UNSUPPORTED;
  // all sequences in one schedule (one launch per 128 non-empty sequences)
  return status_of(msa::launch_index_select_varlen(q_idx, k_idx, cu_seqlens, B, n_groups, d_idx,
                                                   k, block_ids, diag(), (cudaStream_t)stream));
}

int msa_sparse_attn_varlen(const void* q, const void* k, const void* v, const int32_t* block_ids,
                           const int64_t* cu_seqlens, int B, int H_q, int H_kv, int d, int Bk,
                           int topk, float scale, void* out, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (!cu_ok(cu_seqlens, B)) return MSA_ERR_INVALID_ARG;
  return attn_batch(q, k, v, block_ids, cu_seqlens, nullptr, nullptr, 0, 0, B, H_q, H_kv, d, Bk,
                    topk, scale, out, lse, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- paged prefill
// cu_q host [B + 1] query offsets; kv_lens host [B], kv_lens[b] >= queries of b
static bool paged_ok(const int64_t* cu_q, const int64_t* kv_lens, int B, int max_pages) {
  if (!cu_ok(cu_q, B) || max_pages < 1 || (B > 0 && !kv_lens)) return false;
  for (int b = 0; b < B; ++b)
    if (kv_lens[b] < cu_q[b + 1] - cu_q[b] || kv_lens[b] > (int64_t)max_pages * 128) return false;
  return true;
}

int msa_index_select_paged(const void* q_idx, const void* k_idx_pages, int64_t n_pages,
                           const int32_t* page_table, int max_pages, const int64_t* cu_q,
                           const int64_t* kv_lens, int B, int n_groups, int d_idx, int Bk, int k,
                           int32_t* block_ids, void* stream) {
  if (!paged_ok(cu_q, kv_lens, B, max_pages) || n_pages < 1 || n_groups < 1 || d_idx < 1 ||
      Bk < 1 || k < 1)
    return MSA_ERR_INVALID_ARG;
  if (B == 0 || cu_q[B] == 0) return MSA_OK;
  if (!q_idx || !k_idx_pages || !page_table || !block_ids) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx_pages) || !aligned16(block_ids))
    return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || !supported_k(k) || !supported_d(d_idx)) return MSA_ERR_UNSUPPORTED;
  if (cu_q[B] * n_groups >= (1ll << 31) || n_pages * 128 >= (1ll << 31) ||
      (int64_t)B * max_pages >= (1ll << 31))
    return MSA_ERR_UNSUPPORTED;
  return status_of(msa::launch_index_select_paged(q_idx, k_idx_pages, n_pages, page_table,
                                                  max_pages, cu_q, kv_lens, B, n_groups, d_idx,
                                                  k, block_ids, diag(), (cudaStream_t)stream));
}

size_t msa_sparse_attn_paged_workspace_bytes(const int64_t* cu_q, const int64_t* kv_lens, int B,
                                             int max_pages, int H_q, int H_kv, int d, int Bk,
                                             int k) {
  BatchPlan p;
  if (!paged_ok(cu_q, kv_lens, B, max_pages) || H_q < 1 || H_kv < 1 || Bk < 1 || k < 1 ||
      !plan_batch(cu_q, kv_lens, B, max_pages, p) || p.n_q == 0)
    return 0;
  return batch_ws_bytes(p, p.n_q, H_q, H_kv, d, k, true);
}

int msa_sparse_attn_paged(const void* q, const void* k_pages, const void* v_pages,
                          int64_t n_pages, const int32_t* page_table, int max_pages,
                          const int32_t* block_ids, const int64_t* cu_q, const int64_t* kv_lens,
                          int B, int H_q, int H_kv, int d, int Bk, int topk, float scale,
                          void* out, float* lse, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (!paged_ok(cu_q, kv_lens, B, max_pages) || n_pages < 1) return MSA_ERR_INVALID_ARG;
  if (B > 0 && cu_q[B] > 0 && !page_table) return MSA_ERR_INVALID_ARG;
  if ((int64_t)B * max_pages >= (1ll << 31)) return MSA_ERR_UNSUPPORTED;
  return attn_batch(q, k_pages, v_pages, block_ids, cu_q, kv_lens, page_table, n_pages,
                    max_pages, B, H_q, H_kv, d, Bk, topk, scale, out, lse, workspace,
                    workspace_bytes, stream);
}

// Rows of the decode block scores kept in the workspace start on 16-byte
// boundaries (a multiple of four floats), so the top-k reads them as vectors.
static int64_t decode_score_stride(int max_pages) { return ((int64_t)max_pages + 3) & ~(int64_t)3; }

size_t msa_index_select_decode_workspace_bytes(int B, int max_pages, int n_groups) {
  if (B < 0 || max_pages < 0 || n_groups < 0) return 0;
  return (size_t)B * decode_score_stride(max_pages) * n_groups * sizeof(float);
}

static int index_decode(const void* q_idx, const void* k_idx_pages, const int32_t* page_table,
                        const int32_t* seq_lens, int B, int max_pages, int n_groups, int d_idx,
                        int Bk, int k, int32_t* block_ids, float* block_scores, void* workspace,
                        size_t workspace_bytes, void* stream, bool e4m3, float score_scale) {
  if (B < 0 || max_pages < 1 || n_groups < 1 || d_idx < 1 || Bk < 1 || k < 1)
    return MSA_ERR_INVALID_ARG;
  if (B == 0) return MSA_OK;
  if (!q_idx || !k_idx_pages || !page_table || !seq_lens || !block_ids)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx_pages) || (block_scores && !aligned16(block_scores)))
    return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || !supported_k(k) || !supported_d(d_idx) || n_groups > 8)
    return MSA_ERR_UNSUPPORTED;
  float* scores = block_scores;
  int64_t ss = max_pages;  // caller's block_scores: [B, n_groups, max_pages]
  if (!scores) {
    if (!workspace || workspace_bytes < msa_index_select_decode_workspace_bytes(B, max_pages,
                                                                                n_groups))
      return MSA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MSA_ERR_INVALID_ARG;
    scores = (float*)workspace;
    ss = decode_score_stride(max_pages);
  }
  cudaStream_t st = (cudaStream_t)stream;
  msa::Diag dg = diag();
  cudaError_t e = msa::launch_decode_index(q_idx, k_idx_pages, page_table, seq_lens, B,
                                           max_pages, n_groups, d_idx, scores, dg, st, e4m3,
                                           score_scale, ss);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  e = msa::launch_topk(scores, B, n_groups, max_pages, Bk, k, 0, seq_lens, block_ids, dg, st,
                       ss);
  return status_of(e);
}

int msa_index_select_decode(const void* q_idx, const void* k_idx_pages,
                            const int32_t* page_table, const int32_t* seq_lens, int B,
                            int max_pages, int n_groups, int d_idx, int Bk, int k,
                            int32_t* block_ids, float* block_scores, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return index_decode(q_idx, k_idx_pages, page_table, seq_lens, B, max_pages, n_groups, d_idx,
                      Bk, k, block_ids, block_scores, workspace, workspace_bytes, stream, false,
                      1.f);
}

int msa_index_select_decode_fp8(const void* q_idx, const void* k_idx_pages,
                                const int32_t* page_table, const int32_t* seq_lens, int B,
                                int max_pages, int n_groups, int d_idx, int Bk, int k,
                                int32_t* block_ids, float* block_scores, float score_scale,
                                void* workspace, size_t workspace_bytes, void* stream) {
  return index_decode(q_idx, k_idx_pages, page_table, seq_lens, B, max_pages, n_groups, d_idx,
                      Bk, k, block_ids, block_scores, workspace, workspace_bytes, stream, true,
                      score_scale);
}

int msa_index_select_decode_nvfp4(const void* q_idx, const void* k_idx_codes,
                                  const void* k_idx_scales, const int32_t* page_table,
                                  const int32_t* seq_lens, int B, int max_pages, int n_groups,
                                  int d_idx, int Bk, int k, int32_t* block_ids,
                                  float* block_scores, float score_scale, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (B < 0 || max_pages < 1 || n_groups < 1 || d_idx < 1 || Bk < 1 || k < 1)
    return MSA_ERR_INVALID_ARG;
  if (B == 0) return MSA_OK;
  if (!q_idx || !k_idx_codes || !k_idx_scales || !page_table || !seq_lens || !block_ids)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx_codes) || !aligned16(k_idx_scales) ||
      (block_scores && !aligned16(block_scores)))
    return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || !supported_k(k) || !supported_d(d_idx) || n_groups > 8)
    return MSA_ERR_UNSUPPORTED;
  float* scores = block_scores;
  int64_t ss = max_pages;  // caller's block_scores: [B, n_groups, max_pages]
  if (!scores) {
    if (!workspace || workspace_bytes < msa_index_select_decode_workspace_bytes(B, max_pages,
                                                                                n_groups))
      return MSA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return MSA_ERR_INVALID_ARG;
    scores = (float*)workspace;
    ss = decode_score_stride(max_pages);
  }
  cudaStream_t st = (cudaStream_t)stream;
  msa::Diag dg = diag();
  cudaError_t e = msa::launch_decode_index_fp4(q_idx, k_idx_codes, k_idx_scales, page_table,
                                               seq_lens, B, max_pages, n_groups, d_idx,
                                               score_scale, scores, dg, st, ss);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  e = msa::launch_topk(scores, B, n_groups, max_pages, Bk, k, 0, seq_lens, block_ids, dg, st,
                       ss);
  return status_of(e);
}

size_t msa_decode_workspace_bytes(int B, int H_q, int d, int k) {
  if (B < 0 || H_q < 0 || d < 0 || k < 0) return 0;
  return msa::decode_ws_bytes(B, H_q, d, k);
}

int msa_decode(const void* q, const void* k_pages, const void* v_pages, int kv_dtype,
               const float* k_scale, const float* v_scale, const int32_t* page_table,
               const int32_t* seq_lens, const int32_t* block_ids, int B, int max_pages, int H_q,
               int H_kv, int d, int Bk, int k, float scale, void* out, float* lse,
               void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || max_pages < 1 || H_q < 1 || H_kv < 1 || d < 1 || Bk < 1 || k < 1)
    return MSA_ERR_INVALID_ARG;
  if (B == 0) return MSA_OK;
  if (kv_dtype != MSA_KV_BF16 && kv_dtype != MSA_KV_E4M3) return MSA_ERR_INVALID_ARG;
  if (!q || !k_pages || !v_pages || !page_table || !seq_lens || !block_ids || !out)
    return MSA_ERR_INVALID_ARG;
  if (kv_dtype == MSA_KV_E4M3 && (!k_scale || !v_scale)) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out))
    return MSA_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || !supported_k(k) || !supported_d(d) || H_q / H_kv > 8)
    return MSA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < msa_decode_workspace_bytes(B, H_q, d, k))
    return MSA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MSA_ERR_INVALID_ARG;
  return status_of(msa::launch_decode_attn(q, k_pages, v_pages, kv_dtype == MSA_KV_E4M3,
                                           k_scale, v_scale, page_table, seq_lens, block_ids,
                                           B, max_pages, H_q, H_kv, d, k, scale, out, lse,
                                           workspace, diag(), (cudaStream_t)stream));
}

int msa_decode_nvfp4(const void* q, const void* k_codes, const void* k_scales,
                     const void* v_codes, const void* v_scales, const int32_t* page_table,
                     const int32_t* seq_lens, const int32_t* block_ids, int B, int max_pages,
                     int H_q, int H_kv, int d, int Bk, int k, float scale, void* out, float* lse,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || max_pages < 1 || H_q < 1 || H_kv < 1 || d < 1 || Bk < 1 || k < 1)
    return MSA_ERR_INVALID_ARG;
  if (B == 0) return MSA_OK;
  if (!q || !k_codes || !k_scales || !v_codes || !v_scales || !page_table || !seq_lens ||
      !block_ids || !out)
    return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_codes) || !aligned16(k_scales) || !aligned16(v_codes) ||
      !aligned16(v_scales) || !aligned16(out))
    return MSA_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || !supported_k(k) || !supported_d(d) || H_q / H_kv > 8)
    return MSA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < msa_decode_workspace_bytes(B, H_q, d, k))
    return MSA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MSA_ERR_INVALID_ARG;
  return status_of(msa::launch_decode_attn_fp4(q, k_codes, k_scales, v_codes, v_scales,
                                               page_table, seq_lens, block_ids, B, max_pages,
                                               H_q, H_kv, d, k, scale, out, lse, workspace, diag(),
                                               (cudaStream_t)stream));
}

int msa_get_error(void* stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MSA_ERR_CUDA;
  int* p = err_ptr();
  if (!p) return MSA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MSA_ERR_CUDA;
  int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return MSA_ERR_CUDA;
  return v;
}

int64_t msa_launch_count(void) { return msa::g_launches.load(std::memory_order_relaxed); }

int64_t msa_set_wait_limit(int64_t polls) {
  std::lock_guard<std::mutex> lk(g_mu);
  int64_t old = g_wait_limit;
  if (polls >= 0) g_wait_limit = polls;
  return old;
}

}  // extern "C"
