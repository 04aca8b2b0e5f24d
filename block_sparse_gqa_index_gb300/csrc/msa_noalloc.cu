// Decode index branch for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or any allocating routine) once they
// are running: serving engines that reserve all device memory up front and
// forbid later allocations, code that runs where an allocation could block on
// or synchronise with other work on the device, or hosts whose memory
// manager owns every device byte. msa_index_select_decode needs a scratch
// buffer for the per-page block scores; this variant takes that scratch from a
// fixed array compiled into the library instead of a caller workspace.
//
// The array lives in every GPU that loads the library until the process exits
// (4 MiB). Every call shares it and it keeps the last call's contents; each
// call writes every score it later reads, so nothing needs clearing. Calls
// whose executions overlap on the GPU (different streams, or different host
// threads) race on the array and must be serialised by the caller.
#include <mutex>

#include "../../include/msa.h"
#include "msa_kernels.h"

namespace {

constexpr int64_t kScratchFloats = 1ll << 20;  // 4 MiB of fp32 block scores

static __device__ __align__(256) float g_decode_scores[kScratchFloats];

std::mutex g_mu;
float* g_scores_ptr[64] = {nullptr};

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
float* scratch_ptr(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *status = MSA_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scores_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scores);
    if (e != cudaSuccess || !p) {
      *status = MSA_ERR_CUDA;
      return nullptr;
    }
    g_scores_ptr[dev] = (float*)p;
  }
  *status = MSA_OK;
  return g_scores_ptr[dev];
}

}  // namespace

extern "C" {

int64_t msa_index_select_decode_noalloc_max_scores(void) { return kScratchFloats; }

int msa_index_select_decode_noalloc(const void* q_idx, const void* k_idx_pages,
                                    const int32_t* page_table, const int32_t* seq_lens, int B,
                                    int max_pages, int n_groups, int d_idx, int Bk, int k,
                                    int32_t* block_ids, void* stream) {
  if (B < 0 || max_pages < 1 || n_groups < 1 || d_idx < 1 || Bk < 1 || k < 1)
    return MSA_ERR_INVALID_ARG;
  if (B == 0) return MSA_OK;
  if (!q_idx || !k_idx_pages || !page_table || !seq_lens || !block_ids)
    return MSA_ERR_INVALID_ARG;
  if (((uintptr_t)q_idx & 15u) || ((uintptr_t)k_idx_pages & 15u)) return MSA_ERR_INVALID_ARG;
  if (Bk != 128 || k > msa::kMaxK || (d_idx != 64 && d_idx != 128) || n_groups > 8)
    return MSA_ERR_UNSUPPORTED;
  // the scores of B x n_groups x max_pages blocks must fit the fixed array
  if ((int64_t)B * n_groups * max_pages > kScratchFloats) return MSA_ERR_WORKSPACE;
  int status = MSA_OK;
  float* scores = scratch_ptr(&status);
  if (!scores) return status;
  cudaStream_t st = (cudaStream_t)stream;
  msa::Diag dg = msa::current_diag();
  cudaError_t e = msa::launch_decode_index(q_idx, k_idx_pages, page_table, seq_lens, B,
                                           max_pages, n_groups, d_idx, scores, dg, st);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  e = msa::launch_topk(scores, B, n_groups, max_pages, Bk, k, 0, seq_lens, block_ids, dg, st);
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // extern "C"
