// Main branch of MSA prefill: exact softmax attention of every query head over
// the causally visible tokens of its group's selected blocks.
//
// "MiniMax Sparse Attention (MSA): a Two-Branch Block-Sparse Attention Trained
// on a 109B-Parameter MoE With a 3T-Token Budget", section "两个分支如何工作"
// (how the two branches work): the main branch gathers the causally visible
// tokens of the selected blocks and runs restricted scaled-dot-product softmax;
// each query head keeps its own projection and shares the group's block set.
//
// Work is organised KV-block-outer: every (group g, block b) pair is a bucket
// holding the queries that selected b. A tile is one bucket's 128-key block
// against up to 128 / G of its queries (all G heads of each: 128 score rows).
// Each tile yields, per (query, head), the block's softmax-normalised output in
// bf16 and its LSE; a merge pass combines the (at most k) partials of every
// (query, head) exactly:  lse = log sum_s exp(lse_s),
//                         o   = sum_s exp(lse_s - lse) * o_s.
// Queries are processed in chunks so that the partials fit the workspace.
#include "msa_kernels.h"

namespace msa {
namespace {

constexpr int kBk = 128;
constexpr int kTileRows = 128;
constexpr int kThreads = 256;

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// ------------------------------------------------------------ bucketing passes
// A block id is usable for row (t, g) iff 0 <= id <= t / 128; anything else
// (other than the -1 padding) is skipped and flagged in the error word.
__device__ __forceinline__ bool id_ok(int id, int64_t t, const Diag& dg) {
  if (id < 0) return false;
  if ((int64_t)id > t / kBk) {
    report(dg, kStatusBadIds);
    return false;
  }
  return true;
}

__global__ void bucket_count_kernel(const int32_t* __restrict__ ids, int64_t q0, int64_t q1,
                                    int n_g, int k, int64_t nb, int32_t* __restrict__ counts,
                                    Diag dg) {
  int64_t n = (q1 - q0) * n_g * k;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    int64_t row = q0 * n_g + e / k;  // (t, g) row
    int id = ids[row * k + e % k];
    if (id_ok(id, row / n_g, dg)) atomicAdd(&counts[(row % n_g) * nb + id], 1);
  }
}

// single CTA: exclusive scans of counts and of ceil(counts / qt) (tiles)
__global__ void bucket_scan_kernel(const int32_t* __restrict__ counts, int64_t n_b, int qt,
                                   int32_t* __restrict__ offsets, int32_t* __restrict__ tile_off,
                                   int32_t* __restrict__ cursor) {
  __shared__ int32_t s_a[1024], s_b[1024];
  const int tid = threadIdx.x;
  const int64_t per = (n_b + 1023) / 1024;
  const int64_t lo = min(n_b, tid * per), hi = min(n_b, lo + per);
  int32_t a = 0, b = 0;
  for (int64_t i = lo; i < hi; ++i) {
    a += counts[i];
    b += (counts[i] + qt - 1) / qt;
  }
  s_a[tid] = a;
  s_b[tid] = b;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive Hillis-Steele scan
    int32_t ya = tid >= off ? s_a[tid - off] : 0;
    int32_t yb = tid >= off ? s_b[tid - off] : 0;
    __syncthreads();
    s_a[tid] += ya;
    s_b[tid] += yb;
    __syncthreads();
  }
  a = s_a[tid] - a;
  b = s_b[tid] - b;
  for (int64_t i = lo; i < hi; ++i) {
    offsets[i] = a;
    tile_off[i] = b;
    cursor[i] = 0;
    a += counts[i];
    b += (counts[i] + qt - 1) / qt;
  }
  if (tid == 1023) {
    offsets[n_b] = s_a[1023];
    tile_off[n_b] = s_b[1023];
  }
}

__global__ void bucket_fill_kernel(const int32_t* __restrict__ ids, int64_t q0, int64_t q1,
                                   int n_g, int k, int64_t nb,
                                   const int32_t* __restrict__ offsets,
                                   int32_t* __restrict__ cursor, int32_t* __restrict__ entries) {
  const Diag none{nullptr, 0};
  int64_t n = (q1 - q0) * n_g * k;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    int64_t row = q0 * n_g + e / k;
    int slot = (int)(e % k);
    int id = ids[row * k + slot];
    if (!id_ok(id, row / n_g, none)) continue;
    int64_t bk = (row % n_g) * nb + id;
    int pos = offsets[bk] + atomicAdd(&cursor[bk], 1);
    entries[pos] = (int32_t)(((row / n_g - q0) << 4) | slot);
  }
}

// ------------------------------------------------------ tile kernel (CUDA cores)
template <int D>
__global__ void __launch_bounds__(kThreads)
attn_tile_cc_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ kk,
                    const uint16_t* __restrict__ v, int64_t N, int64_t q0, int H_q, int H_kv,
                    int k, float scale_log2, int64_t nb, const int32_t* __restrict__ entries,
                    const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_off,
                    int64_t n_b, uint16_t* __restrict__ part_o, float* __restrict__ part_lse) {
  constexpr int DP = D + 2;  // padded smem row (bf16 elements)
  extern __shared__ __align__(16) unsigned char smem[];
  uint16_t* Qs = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Ks = Qs + kTileRows * DP;
  uint16_t* Vs = Ks + kBk * DP;
  float* Ss = reinterpret_cast<float*>(Vs + kBk * DP);  // [128][129]
  float* row_m = Ss + kTileRows * 129;
  float* row_l = row_m + kTileRows;
  int* row_t = reinterpret_cast<int*>(row_l + kTileRows);
  int* row_dst = row_t + kTileRows;

  const int G = H_q / H_kv;
  const int qt = kTileRows / G;
  const int tid = threadIdx.x;
  const int total = tile_off[n_b];
  int64_t cur_bk = -1;

  for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
    // bucket of this tile: last bk with tile_off[bk] <= tile
    int64_t lo = 0, hi = n_b - 1;
    while (lo < hi) {
      int64_t mid = (lo + hi + 1) >> 1;
      if (tile_off[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    const int64_t bk = lo;
    const int g = (int)(bk / nb);
    const int64_t b = bk % nb;
    const int e0 = offsets[bk] + (tile - tile_off[bk]) * qt;
    const int e1 = min(e0 + qt, offsets[bk + 1]);
    const int nrows = (e1 - e0) * G;

    __syncthreads();
    if (bk != cur_bk) {  // K, V of block b, head g
      for (int e = tid; e < kBk * (D / 2); e += kThreads) {
        int j = e / (D / 2), c2 = e % (D / 2);
        int64_t key = b * kBk + j;
        uint32_t kw = 0, vw = 0;
        if (key < N) {
          size_t off = ((size_t)key * H_kv + g) * D + 2 * c2;
          kw = *reinterpret_cast<const uint32_t*>(kk + off);
          vw = *reinterpret_cast<const uint32_t*>(v + off);
        }
        *reinterpret_cast<uint32_t*>(Ks + j * DP + 2 * c2) = kw;
        *reinterpret_cast<uint32_t*>(Vs + j * DP + 2 * c2) = vw;
      }
      cur_bk = bk;
    }
    if (tid < kTileRows) {
      int r = tid;
      if (r < nrows) {
        int ent = entries[e0 + r / G];
        int64_t tl = ent >> 4;
        int slot = ent & 15;
        int h = g * G + r % G;
        row_t[r] = (int)(q0 + tl);
        row_dst[r] = (int)((tl * H_q + h) * k + slot);
      } else {
        row_t[r] = 0x7FFFFFFF;
        row_dst[r] = -1;
      }
    }
    __syncthreads();
    for (int e = tid; e < kTileRows * (D / 2); e += kThreads) {
      int r = e / (D / 2), c2 = e % (D / 2);
      uint32_t w = 0;
      if (r < nrows) {
        int64_t t = row_t[r];
        int h = g * G + r % G;
        w = *reinterpret_cast<const uint32_t*>(q + ((size_t)t * H_q + h) * D + 2 * c2);
      }
      *reinterpret_cast<uint32_t*>(Qs + r * DP + 2 * c2) = w;
    }
    __syncthreads();

    // S = Q K^T (rows rg*8.., keys kg + 16 i)
    const int rg = tid >> 4, kg = tid & 15;
    {
      float acc[8][8];
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[r][i] = 0.f;
#pragma unroll 4
      for (int c = 0; c < D; c += 2) {
        float qa[8], qb[8], ka[8], kb[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          uint32_t w = *reinterpret_cast<const uint32_t*>(Qs + (rg * 8 + r) * DP + c);
          qa[r] = bf16_lo(w);
          qb[r] = bf16_hi(w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t w = *reinterpret_cast<const uint32_t*>(Ks + (kg + 16 * i) * DP + c);
          ka[i] = bf16_lo(w);
          kb[i] = bf16_hi(w);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[r][i] = fmaf(qa[r], ka[i], fmaf(qb[r], kb[i], acc[r][i]));
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        int row = rg * 8 + r;
        int64_t t = row_t[row];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          int64_t key = b * kBk + kg + 16 * i;
          Ss[row * 129 + kg + 16 * i] = key <= t ? acc[r][i] * scale_log2 : -INFINITY;
        }
      }
    }
    __syncthreads();
    // softmax: two threads per row (64 keys each), base-2 domain
    {
      int row = tid >> 1, half = tid & 1;
      float* s = Ss + row * 129 + half * 64;
      float m = -INFINITY;
      for (int i = 0; i < 64; ++i) m = fmaxf(m, s[i]);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      float l = 0.f;
      for (int i = 0; i < 64; ++i) {
        float p = ex2_approx(s[i] - m);
        s[i] = p;
        l += p;
      }
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      if (half == 0) {
        row_m[row] = m;
        row_l[row] = l;
      }
    }
    __syncthreads();
    // O = P V (rows rg*8.., column pairs cg*2 + 32 i)
    {
      constexpr int NP = D / 32;  // column pairs per thread
      const int cg = tid & 15;
      float acc[8][2 * NP];
#pragma unroll
      for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int i = 0; i < 2 * NP; ++i) acc[r][i] = 0.f;
#pragma unroll 4
      for (int j = 0; j < kBk; ++j) {
        float p[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) p[r] = Ss[(rg * 8 + r) * 129 + j];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          uint32_t w = *reinterpret_cast<const uint32_t*>(Vs + j * DP + cg * 2 + 32 * i);
          float va = bf16_lo(w), vb = bf16_hi(w);
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            acc[r][2 * i] = fmaf(p[r], va, acc[r][2 * i]);
            acc[r][2 * i + 1] = fmaf(p[r], vb, acc[r][2 * i + 1]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        int row = rg * 8 + r;
        int dst = row_dst[row];
        if (dst < 0) continue;
        float inv = 1.f / row_l[row];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          uint32_t w = pack_bf16x2(acc[r][2 * i] * inv, acc[r][2 * i + 1] * inv);
          *reinterpret_cast<uint32_t*>(part_o + (size_t)dst * D + cg * 2 + 32 * i) = w;
        }
        if (cg == 0) part_lse[dst] = (row_m[row] + __log2f(row_l[row])) * 0.69314718055994531f;
      }
    }
  }
}

// ---------------------------------------------------------------------- merge
template <int D>
__global__ void attn_merge_kernel(const uint16_t* __restrict__ part_o,
                                  const float* __restrict__ part_lse,
                                  const int32_t* __restrict__ ids, int64_t q0, int64_t q1,
                                  int H_q, int H_kv, int k, uint16_t* __restrict__ out,
                                  float* __restrict__ lse) {
  constexpr int PER = D / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  const int G = H_q / H_kv;
  int64_t n = (q1 - q0) * H_q;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < n;
       w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    int64_t tl = w / H_q;
    int h = (int)(w % H_q);
    int64_t t = q0 + tl;
    const int32_t* id = ids + ((size_t)t * H_kv + h / G) * k;
    const float* pl = part_lse + (size_t)w * k;
    const Diag none{nullptr, 0};
    float M = -INFINITY;
    for (int s = 0; s < k; ++s)
      if (id_ok(id[s], t, none)) M = fmaxf(M, pl[s]);
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float L = 0.f;
    for (int s = 0; s < k; ++s) {
      if (!id_ok(id[s], t, none)) continue;
      float wgt = __expf(pl[s] - M);
      L += wgt;
      const uint16_t* po = part_o + ((size_t)w * k + s) * D + lane * PER;
      if (PER == 4) {
        uint2 u = *reinterpret_cast<const uint2*>(po);
        acc[0] = fmaf(wgt, bf16_lo(u.x), acc[0]);
        acc[1] = fmaf(wgt, bf16_hi(u.x), acc[1]);
        acc[2] = fmaf(wgt, bf16_lo(u.y), acc[2]);
        acc[3] = fmaf(wgt, bf16_hi(u.y), acc[3]);
      } else {
        uint32_t u = *reinterpret_cast<const uint32_t*>(po);
        acc[0] = fmaf(wgt, bf16_lo(u), acc[0]);
        acc[1] = fmaf(wgt, bf16_hi(u), acc[1]);
      }
    }
    float inv = 1.f / L;
    uint16_t* o = out + ((size_t)t * H_q + h) * D + lane * PER;
    if (PER == 4) {
      uint2 u;
      u.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      u.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(o) = u;
    } else {
      *reinterpret_cast<uint32_t*>(o) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
    if (lse && lane == 0) lse[(size_t)t * H_q + h] = M + logf(L);
  }
}

template <int D>
size_t tile_smem_bytes() {
  return (size_t)(kTileRows + 2 * kBk) * (D + 2) * 2 + kTileRows * 129 * 4 + kTileRows * 16;
}

}  // namespace

size_t attn_ws_bytes(int64_t chunk, int64_t nb, int H_q, int H_kv, int d, int k) {
  int64_t n_b = (int64_t)H_kv * nb;
  size_t s = 0;
  s += align256((size_t)n_b * 4);        // counts
  s += align256((size_t)(n_b + 1) * 4);  // offsets
  s += align256((size_t)n_b * 4);        // cursor
  s += align256((size_t)(n_b + 1) * 4);  // tile_off
  s += align256((size_t)chunk * H_kv * k * 4);
  s += align256((size_t)chunk * H_q * k * d * 2);
  s += align256((size_t)chunk * H_q * k * 4);
  return s;
}

AttnWs attn_ws_carve(void* ws, int64_t chunk, int64_t nb, int H_q, int H_kv, int d, int k) {
  int64_t n_b = (int64_t)H_kv * nb;
  unsigned char* p = (unsigned char*)ws;
  AttnWs w;
  w.counts = (int32_t*)p;   p += align256((size_t)n_b * 4);
  w.offsets = (int32_t*)p;  p += align256((size_t)(n_b + 1) * 4);
  w.cursor = (int32_t*)p;   p += align256((size_t)n_b * 4);
  w.tile_off = (int32_t*)p; p += align256((size_t)(n_b + 1) * 4);
  w.entries = (int32_t*)p;  p += align256((size_t)chunk * H_kv * k * 4);
  w.part_o = (uint16_t*)p;  p += align256((size_t)chunk * H_q * k * d * 2);
  w.part_lse = (float*)p;
  return w;
}

cudaError_t launch_sparse_attn_chunk(const void* q, const void* kk, const void* v,
                                     const int32_t* ids, int64_t N, int64_t q0, int64_t q1,
                                     int H_q, int H_kv, int d, int k, float scale, void* out,
                                     float* lse, const AttnWs& ws, int64_t nb, const Diag& dg,
                                     cudaStream_t st) {
  const int64_t n_b = (int64_t)H_kv * nb;
  const int G = H_q / H_kv;
  const int qt = kTileRows / G;
  note_launches(6);  // memset, count, scan, fill, tile, merge
  cudaError_t e = cudaMemsetAsync(ws.counts, 0, (size_t)n_b * 4, st);
  if (e != cudaSuccess) return e;
  int64_t n = (q1 - q0) * H_kv * k;
  unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 32);
  bucket_count_kernel<<<grid, 256, 0, st>>>(ids, q0, q1, H_kv, k, nb, ws.counts, dg);
  bucket_scan_kernel<<<1, 1024, 0, st>>>(ws.counts, n_b, qt, ws.offsets, ws.tile_off, ws.cursor);
  bucket_fill_kernel<<<grid, 256, 0, st>>>(ids, q0, q1, H_kv, k, nb, ws.offsets, ws.cursor,
                                           ws.entries);
  const float scale_log2 = scale * 1.4426950408889634f;
  if (d == 128) {
    size_t sm = tile_smem_bytes<128>();
    cudaFuncSetAttribute(attn_tile_cc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm);
    attn_tile_cc_kernel<128><<<152, kThreads, sm, st>>>(
        (const uint16_t*)q, (const uint16_t*)kk, (const uint16_t*)v, N, q0, H_q, H_kv, k,
        scale_log2, nb, ws.entries, ws.offsets, ws.tile_off, n_b, ws.part_o, ws.part_lse);
  } else {
    size_t sm = tile_smem_bytes<64>();
    cudaFuncSetAttribute(attn_tile_cc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm);
    attn_tile_cc_kernel<64><<<152, kThreads, sm, st>>>(
        (const uint16_t*)q, (const uint16_t*)kk, (const uint16_t*)v, N, q0, H_q, H_kv, k,
        scale_log2, nb, ws.entries, ws.offsets, ws.tile_off, n_b, ws.part_o, ws.part_lse);
  }
  int64_t nw = (q1 - q0) * H_q;
  unsigned mg = (unsigned)std::min<int64_t>((nw * 32 + 255) / 256, 152 * 64);
  if (d == 128)
    attn_merge_kernel<128><<<mg, 256, 0, st>>>(ws.part_o, ws.part_lse, ids, q0, q1, H_q, H_kv, k,
                                               (uint16_t*)out, lse);
  else
    attn_merge_kernel<64><<<mg, 256, 0, st>>>(ws.part_o, ws.part_lse, ids, q0, q1, H_q, H_kv, k,
                                              (uint16_t*)out, lse);
  return cudaGetLastError();
}

}  // namespace msa
