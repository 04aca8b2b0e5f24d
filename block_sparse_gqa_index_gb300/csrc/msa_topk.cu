// Exp-free top-k over MSA block scores.
//
// "MiniMax Sparse Attention (MSA): a Two-Branch Block-Sparse Attention Trained
// on a 109B-Parameter MoE With a 3T-Token Budget", section "内核协同设计"
// (kernel co-design): softmax preserves order, so the blocks are ranked on their
// raw max-pooled scores, with no max / exp / sum pass. Selection rule from
// "两个分支如何工作": the query's local block is always kept and the other k-1
// slots take the best earlier blocks; lower block id wins ties.
//
// One warp per (query, group) row. The row's candidates (blocks 0 .. loc-1) are
// streamed in chunks of 1024 scores, 32 per lane, read with 16-byte loads. Per
// chunk:
//   1. every lane takes the max ranking key of its 32 scores;
//   2. tau = max(15th largest lane max, worst key kept so far): at least k-1
//      keys are >= tau, so no key below tau can be in the answer;
//   3. the keys >= tau (typically a few dozen) are compacted into shared memory
//      and bitonic-sorted across the warp (64 keys, 2 per lane); the best k-1
//      are kept, one per lane. More than 64 survivors fall back to k-1 rounds of
//      warp arg-max.
// Finally the kept ids plus the local block are sorted ascending and written.
#include "msa_kernels.h"

namespace msa {
namespace {

constexpr int kWarps = 8;
constexpr int kChunk = 1024;
constexpr int kCap = 64;

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
  uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, m);
  uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), m);
  return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
  uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)v, src);
  uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(v >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// score of a ranking key (inverse of ord_f32 on the upper half)
__device__ __forceinline__ float key_value(uint64_t key) {
  uint32_t o = (uint32_t)(key >> 32);
  uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}

// bitonic sort of one key per lane, descending (lane 0 = largest)
__device__ __forceinline__ uint64_t sort32_desc(uint64_t a, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      uint64_t p = shfl_xor64(a, stride);
      bool up = (lane & size) == 0;
      bool lower = (lane & stride) == 0;
      uint64_t hi = a > p ? a : p, lo = a > p ? p : a;
      a = (lower == up) ? hi : lo;
    }
  return a;
}

// bitonic sort of 64 keys (element e = lane + 32 r held in a[r]), descending
__device__ __forceinline__ void sort64_desc(uint64_t& a0, uint64_t& a1, int lane) {
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride == 32) {
        uint64_t hi = a0 > a1 ? a0 : a1, lo = a0 > a1 ? a1 : a0;
        a0 = hi;
        a1 = lo;
      } else {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          uint64_t& a = r ? a1 : a0;
          int e = lane + 32 * r;
          uint64_t p = shfl_xor64(a, stride);
          bool up = (e & size) == 0;
          bool lower = (e & stride) == 0;
          uint64_t hi = a > p ? a : p, lo = a > p ? p : a;
          a = (lower == up) ? hi : lo;
        }
      }
    }
}

// bitonic sort of one int per lane, ascending
__device__ __forceinline__ int sort32_asc(int a, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      int p = __shfl_xor_sync(0xffffffffu, a, stride);
      bool up = (lane & size) == 0;
      bool lower = (lane & stride) == 0;
      a = (lower == up) ? min(a, p) : max(a, p);
    }
  return a;
}

// bitonic sort of one float per lane, descending
__device__ __forceinline__ float sort32_desc_f(float a, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      float p = __shfl_xor_sync(0xffffffffu, a, stride);
      bool up = (lane & size) == 0;
      bool lower = (lane & stride) == 0;
      a = (lower == up) ? fmaxf(a, p) : fminf(a, p);
    }
  return a;
}

// key of the j-th value held by a lane in chunk c0 (see the load pattern)
__device__ __forceinline__ int64_t elem_block(int64_t c0, int lane, int j) {
  return c0 + (j >> 2) * 128 + lane * 4 + (j & 3);
}

__global__ void __launch_bounds__(kWarps * 32)
topk_kernel(const float* __restrict__ S, int64_t n_rows, int n_g, int64_t nb, int Bk, int k,
            int64_t q_offset, const int32_t* __restrict__ seq_lens, int32_t* __restrict__ ids,
            Diag dg) {
  __shared__ uint64_t buf[kWarps][kCap];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int kfar = k - 1;
  const bool vec = (nb % 4) == 0 && ((uintptr_t)S % 16) == 0;

  for (int64_t r = (int64_t)blockIdx.x * kWarps + wid; r < n_rows;
       r += (int64_t)gridDim.x * kWarps) {
    const int64_t pos = seq_lens ? (int64_t)seq_lens[r / n_g] - 1 : r / n_g + q_offset;
    const int64_t loc = pos / Bk;
    const int64_t ncand = loc;  // candidate blocks 0 .. loc-1
    int32_t* out = ids + r * k;
    if (pos < 0 || loc >= nb) {  // position outside the score rows: flag, emit padding
      if (lane == 0) report(dg, kStatusBadIds);
      if (lane < k) out[lane] = -1;
      continue;
    }
    if (ncand <= kfar) {  // every visible block is kept
      if (lane < k) out[lane] = lane <= loc ? lane : -1;
      continue;
    }
    const float* row = S + r * nb;
    uint64_t best = 0;           // lane i < kfar: i-th best key so far (descending), else 0
    float best_min = -INFINITY;  // value of the kfar-th best so far (-inf before any chunk)
    for (int64_t c0 = 0; c0 < ncand; c0 += kChunk) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t b = c0 + i * 128 + lane * 4;
        float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (b < ncand) {
          if (vec) {
            x = __ldcs(reinterpret_cast<const float4*>(row + b));
            if (b + 3 >= ncand) {  // ragged end: mask the blocks past the candidates
              if (b + 1 >= ncand) x.y = -INFINITY;
              if (b + 2 >= ncand) x.z = -INFINITY;
              x.w = -INFINITY;
            }
          } else {
            x.x = row[b];
            if (b + 1 < ncand) x.y = row[b + 1];
            if (b + 2 < ncand) x.z = row[b + 2];
            if (b + 3 < ncand) x.w = row[b + 3];
          }
        }
        v[4 * i + 0] = x.x;
        v[4 * i + 1] = x.y;
        v[4 * i + 2] = x.z;
        v[4 * i + 3] = x.w;
      }
      // 1. lane max, 2. threshold: the kfar-th largest lane max (>= kfar values
      //    reach it) or the worst value kept so far, whichever is larger
      float lmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; j += 2) lmax = fmax3(lmax, v[j], v[j + 1]);
      const float srt = sort32_desc_f(lmax, lane);
      float tau = __shfl_sync(0xffffffffu, srt, kfar - 1);
      tau = fmaxf(tau, best_min);
      // 3. survivors (>= tau; ties at tau are kept and settled by the keys)
      uint32_t mask = 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) mask |= (v[j] >= tau && v[j] != -INFINITY) ? (1u << j) : 0u;
      const bool keep_old = lane < kfar && best != 0 && key_value(best) >= tau;
      const int cnt = __popc(mask) + (keep_old ? 1 : 0);
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      if (total <= kCap) {
        int p = incl - cnt;
        if (keep_old) buf[wid][p++] = best;
        while (mask) {
          const int j = __ffs(mask) - 1;
          mask &= mask - 1;
          float vj = v[0];
#pragma unroll
          for (int q = 1; q < 32; ++q)
            if (q == j) vj = v[q];
          buf[wid][p++] = rank_key(vj, (uint32_t)elem_block(c0, lane, j));
        }
        __syncwarp();
        uint64_t a0 = lane < total ? buf[wid][lane] : 0;
        if (total <= 32) {
          a0 = sort32_desc(a0, lane);
        } else {
          uint64_t a1 = lane + 32 < total ? buf[wid][lane + 32] : 0;
          sort64_desc(a0, a1, lane);
        }
        __syncwarp();
        best = lane < kfar ? a0 : 0;
      } else {
        // rare: too many survivors (heavy ties); extract the k-1 best one by one
        uint64_t nb_best = 0, prev = ~0ull;
        const uint64_t old = lane < kfar ? best : 0;
        for (int round = 0; round < kfar; ++round) {
          uint64_t m = old < prev ? old : 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (!((mask >> j) & 1u)) continue;
            uint64_t key = rank_key(v[j], (uint32_t)elem_block(c0, lane, j));
            if (key < prev && key > m) m = key;
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            uint64_t y = shfl_xor64(m, off);
            m = y > m ? y : m;
          }
          if (lane == round) nb_best = m;
          prev = m;
        }
        best = nb_best;
      }
      best_min = key_value(shfl64(best, kfar - 1));
    }
    int id = lane < kfar ? key_id(best) : (lane == kfar ? (int)loc : 0x7FFFFFFF);
    id = sort32_asc(id, lane);
    if (lane < k) out[lane] = id == 0x7FFFFFFF ? -1 : id;
  }
}

__global__ void topk_local_only_kernel(int64_t n_rows, int n_g, int Bk, int k, int64_t q_offset,
                                       const int32_t* __restrict__ seq_lens,
                                       int32_t* __restrict__ ids) {
  for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < n_rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    int64_t pos = seq_lens ? (int64_t)seq_lens[r / n_g] - 1 : r / n_g + q_offset;
    ids[r * k] = (int32_t)(pos / Bk);
  }
}

}  // namespace

cudaError_t launch_topk(const float* S, int64_t N, int n_g, int64_t nb, int Bk, int k,
                        int64_t q_offset, const int32_t* seq_lens, int32_t* ids, const Diag& dg,
                        cudaStream_t st) {
  int64_t n_rows = N * n_g;
  if (n_rows == 0) return cudaSuccess;
  note_launches(1);
  if (k == 1) {
    int64_t g = (n_rows + 255) / 256;
    topk_local_only_kernel<<<(unsigned)(g < 152 * 32 ? g : 152 * 32), 256, 0, st>>>(
        n_rows, n_g, Bk, k, q_offset, seq_lens, ids);
    return cudaGetLastError();
  }
  int64_t blocks = (n_rows + kWarps - 1) / kWarps;
  if (blocks > 152 * 64) blocks = 152 * 64;
  topk_kernel<<<(unsigned)blocks, kWarps * 32, 0, st>>>(S, n_rows, n_g, nb, Bk, k, q_offset,
                                                       seq_lens, ids, dg);
  return cudaGetLastError();
}

}  // namespace msa
