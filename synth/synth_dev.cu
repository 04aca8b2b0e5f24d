/* Device fill of the synthetic MSA workloads (shared recipe: synth_recipe.h).
 * Element-wise, grid-stride; values are bit-identical to synth_host.c. */
#include <cuda_runtime.h>
#include <stdint.h>
#include "synth_recipe.h"

namespace {

__global__ void fill_bf16_kernel(SynthSpec sp, int tensor, uint64_t idx0, uint64_t count,
                                 uint16_t* __restrict__ out) {
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < count;
       i += (uint64_t)gridDim.x * blockDim.x)
    out[i] = synth_element(&sp, tensor, idx0 + i);
}

/* Paged cache [P, H, Bk, D] (head-major pages): logical element (s, t, h, c)
 * lives in physical page page_table[s * max_pages + t / Bk], head h, row t % Bk. */
template <typename T, bool FP8>
__global__ void fill_paged_kernel(SynthSpec sp, int tensor, int H, int D,
                                  const int32_t* __restrict__ page_table, int max_pages,
                                  T* __restrict__ out) {
  const uint64_t per_seq = (uint64_t)sp.L * H * D;
  const uint64_t total = per_seq * sp.B;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total;
       i += (uint64_t)gridDim.x * blockDim.x) {
    uint64_t s = i / per_seq;
    uint64_t rem = i % per_seq;
    uint64_t t = rem / ((uint64_t)H * D);
    uint64_t hc = rem % ((uint64_t)H * D);
    uint64_t h = hc / D, c = hc % D;
    int64_t page = page_table[s * max_pages + t / sp.Bk];
    uint64_t dst = (((uint64_t)page * H + h) * sp.Bk + t % sp.Bk) * D + c;
    if (FP8)
      out[dst] = (T)synth_element_e4m3(&sp, tensor, i);
    else
      out[dst] = (T)synth_element(&sp, tensor, i);
  }
}

int grid_for(uint64_t n) {
  uint64_t g = (n + 255) / 256;
  if (g > 152ull * 64ull) g = 152ull * 64ull;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

extern "C" {

/* out[i] = element idx0 + i (device buffer); planted must be a device pointer */
int synth_dev_fill_bf16(const SynthSpec* host_spec, int tensor, uint64_t idx0, uint64_t count,
                        void* out, void* stream) {
  if (count == 0) return 0;
  fill_bf16_kernel<<<grid_for(count), 256, 0, (cudaStream_t)stream>>>(
      *host_spec, tensor, idx0, count, (uint16_t*)out);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

int synth_dev_fill_paged(const SynthSpec* host_spec, int tensor, int H, int D, int fp8,
                         const int32_t* page_table, int max_pages, void* out, void* stream) {
  uint64_t total = (uint64_t)host_spec->L * H * D * host_spec->B;
  if (total == 0) return 0;
  if (fp8)
    fill_paged_kernel<uint8_t, true><<<grid_for(total), 256, 0, (cudaStream_t)stream>>>(
        *host_spec, tensor, H, D, page_table, max_pages, (uint8_t*)out);
  else
    fill_paged_kernel<uint16_t, false><<<grid_for(total), 256, 0, (cudaStream_t)stream>>>(
        *host_spec, tensor, H, D, page_table, max_pages, (uint16_t*)out);
  return cudaGetLastError() == cudaSuccess ? 0 : -1;
}

size_t synth_dev_spec_size(void) { return sizeof(SynthSpec); }

}  // extern "C"
