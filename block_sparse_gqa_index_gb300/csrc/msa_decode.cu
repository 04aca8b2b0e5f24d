// MSA decode: one new token per sequence against a paged KV cache whose page
// size equals the block size ("MiniMax Sparse Attention (MSA): a Two-Branch
// Block-Sparse Attention ...", section "运行 Kernel" / running the kernel: page
// size 128, top-k 16, block scores -> selected KV block indexes -> sparse
// attention), with bf16 or FP8-E4M3 K/V ("MiniMax lança MSA ...", section
// "Kernel open source e MiniMax-M3": BF16 and FP8 support).
//
// decode_index_kernel: streams each sequence's shared index-key cache once and
//   max-pools q_idx . k_idx per 128-key page for all groups at once. Keys are
//   the M dimension of mma.m16n8k16 and the (up to 8) groups its N dimension;
//   the d_idx reduction order is permuted identically in A and B so that each
//   thread reads 16 contiguous bytes per key row. HBM-bound.
// Caches: K / V pages are head-major [P, H_kv, 128, d] (the page tensor's second
// dimension is the kv-head count in the usage listing), so the block a group
// reads is one contiguous run; k_idx pages are [P, 128, d_idx].
// decode_attn_kernel: one CTA per (sequence, group, selected block): the G
//   query heads of the group against the block's visible tokens; writes the
//   block's normalised output and LSE (split-KV partials).
// decode_merge_kernel: combines the k partials of every (sequence, head).
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "msa_kernels.h"

namespace msa {
namespace {

constexpr int kBk = 128;

__device__ __forceinline__ void mma_bf16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int DI>
__global__ void __launch_bounds__(256)
decode_index_kernel(const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ kpages,
                    const int32_t* __restrict__ page_table, const int32_t* __restrict__ seq_lens,
                    int B, int max_pages, int n_g, float* __restrict__ scores, Diag dg) {
  constexpr int NC = DI / 32;  // 16-byte chunks per thread per key row
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, t4 = lane & 3;
  const int64_t n_tasks = (int64_t)B * max_pages;
  for (int64_t task = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; task < n_tasks;
       task += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int s = (int)(task / max_pages);
    const int b = (int)(task % max_pages);
    const int L = seq_lens[s];
    if (L < 1 || L > max_pages * kBk) {  // invalid length: flag once per sequence
      if (b == 0 && lane == 0) report(dg, kStatusBadIds);
      continue;
    }
    if ((int64_t)b * kBk >= L) continue;
    const int nvalid = min(kBk, L - b * kBk);
    uint4 bq[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) {
      bq[i] = make_uint4(0, 0, 0, 0);
      if (gq < n_g)
        bq[i] = *reinterpret_cast<const uint4*>(q_idx + ((size_t)s * n_g + gq) * DI +
                                                8 * (t4 + 4 * i));
    }
    const int64_t page = page_table[(size_t)s * max_pages + b];
    const uint16_t* base = kpages + (size_t)page * kBk * DI;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll 2
    for (int m = 0; m < kBk / 16; ++m) {
      const int key0 = m * 16 + gq, key1 = key0 + 8;
      uint4 a0[NC], a1[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        a0[i] = __ldg(reinterpret_cast<const uint4*>(base + (size_t)key0 * DI + 8 * (t4 + 4 * i)));
        a1[i] = __ldg(reinterpret_cast<const uint4*>(base + (size_t)key1 * DI + 8 * (t4 + 4 * i)));
      }
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        mma_bf16_16816(c, a0[i].x, a1[i].x, a0[i].y, a1[i].y, bq[i].x, bq[i].y);
        mma_bf16_16816(c, a0[i].z, a1[i].z, a0[i].w, a1[i].w, bq[i].z, bq[i].w);
      }
      if (key0 < nvalid) { mx0 = fmaxf(mx0, c[0]); mx1 = fmaxf(mx1, c[1]); }
      if (key1 < nvalid) { mx0 = fmaxf(mx0, c[2]); mx1 = fmaxf(mx1, c[3]); }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    if (gq == 0) {
      int g0 = 2 * t4, g1 = 2 * t4 + 1;
      if (g0 < n_g) scores[((size_t)s * n_g + g0) * max_pages + b] = mx0;
      if (g1 < n_g) scores[((size_t)s * n_g + g1) * max_pages + b] = mx1;
    }
  }
}

// 8 elements from a 16-byte (bf16) or 8-byte (FP8) vector
__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float* out) {
  out[0] = bf16_lo(u.x); out[1] = bf16_hi(u.x);
  out[2] = bf16_lo(u.y); out[3] = bf16_hi(u.y);
  out[4] = bf16_lo(u.z); out[5] = bf16_hi(u.z);
  out[6] = bf16_lo(u.w); out[7] = bf16_hi(u.w);
}
__device__ __forceinline__ void unpack_e4m3x8(const uint2& u, float* out) {
  const uint32_t w[2] = {u.x, u.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFF), __NV_E4M3);
    __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
    float2 a = __half22float2(*reinterpret_cast<__half2*>(&lo));
    float2 b = __half22float2(*reinterpret_cast<__half2*>(&hi));
    out[4 * i + 0] = a.x; out[4 * i + 1] = a.y; out[4 * i + 2] = b.x; out[4 * i + 3] = b.y;
  }
}

// One CTA (128 threads) per (sequence, group, selected page). Scores: thread j
// owns token j and issues all of its K-row loads before using them. P.V: the
// threads form 16 column groups (8 columns each) x 8 token groups (16 tokens
// each, strided so a warp reads whole token rows); partial sums over the token
// groups are added up in shared memory.
template <int D, bool FP8>
__global__ void __launch_bounds__(128)
decode_attn_kernel(const uint16_t* __restrict__ q, const void* __restrict__ kp,
                   const void* __restrict__ vp, const float* __restrict__ k_scale,
                   const float* __restrict__ v_scale, const int32_t* __restrict__ page_table,
                   const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ ids,
                   int max_pages, int H_q, int H_kv, int k, float scale_log2,
                   float* __restrict__ part_o, float* __restrict__ part_lse, Diag dg) {
  constexpr int GMAX = 8;
  constexpr int CG = D / 8;      // column groups
  constexpr int TG = 128 / CG;   // token groups
  constexpr int EB = FP8 ? 1 : 2;
  __shared__ float qs[GMAX][D];
  __shared__ float sc[GMAX][kBk];
  __shared__ float s_m[GMAX], s_l[GMAX];
  __shared__ float red[TG][GMAX][D];
  const int G = H_q / H_kv;
  const int tid = threadIdx.x;
  const int64_t task = blockIdx.x;  // (s * H_kv + g) * k + slot
  const int slot = (int)(task % k);
  const int64_t sg = task / k;
  const int g = (int)(sg % H_kv);
  const int s = (int)(sg / H_kv);
  const int id = ids[task];
  if (id < 0) return;
  const int L = seq_lens[s];
  if (L < 1 || L > max_pages * kBk || id > (L - 1) / kBk) {  // merge skips this slot
    if (tid == 0) report(dg, kStatusBadIds);
    return;
  }
  const int64_t page = page_table[(size_t)s * max_pages + id];
  const int nvalid = min(kBk, L - id * kBk);
  const float ks = FP8 ? k_scale[g] : 1.f;
  const float vs = FP8 ? v_scale[g] : 1.f;
  // pages are head-major [P, H_kv, Bk, D]: the (page, head g) block is contiguous
  const size_t row_stride = D;  // elements between tokens
  const size_t base = ((size_t)page * H_kv + g) * kBk * D;

  for (int e = tid; e < G * D; e += 128) {
    int h = e / D, c = e % D;
    qs[h][c] = __uint_as_float((uint32_t)q[((size_t)s * H_q + g * G + h) * D + c] << 16);
  }
  // K row of token tid, all loads in flight before use
  float acc[GMAX];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) acc[h] = 0.f;
  {
    const int j = tid;
    // raw K row (16-byte bf16 or 8-byte E4M3 vectors), unpacked in the FMA loop
    using Vec = typename std::conditional<FP8, uint2, uint4>::type;
    Vec u[D / 8];
    if (j < nvalid) {
      const Vec* kr = reinterpret_cast<const Vec*>((const unsigned char*)kp +
                                                   (base + j * row_stride) * EB);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) u[c] = __ldcs(kr + c);
    }
    __syncthreads();  // qs ready
    if (j < nvalid) {
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        float x[8];
        if constexpr (FP8) unpack_e4m3x8(u[c], x); else unpack_bf16x8(u[c], x);
#pragma unroll
        for (int h = 0; h < GMAX; ++h)
          if (h < G)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[h] = fmaf(qs[h][8 * c + i], x[i], acc[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h)
      if (h < G) sc[h][j] = j < nvalid ? acc[h] * ks * scale_log2 : -INFINITY;
  }
  __syncthreads();
  {
    const int w = tid >> 5, lane = tid & 31;
    for (int h = w; h < G; h += 4) {
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < kBk / 32; ++i) m = fmaxf(m, sc[h][lane + 32 * i]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float l = 0.f;
#pragma unroll
      for (int i = 0; i < kBk / 32; ++i) {
        float p = ex2_approx(sc[h][lane + 32 * i] - m);
        sc[h][lane + 32 * i] = p;
        l += p;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
      if (lane == 0) { s_m[h] = m; s_l[h] = l; }
    }
  }
  __syncthreads();
  {
    const int cg = tid % CG, tg = tid / CG;
    float o[GMAX][8];
#pragma unroll
    for (int h = 0; h < GMAX; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) o[h][i] = 0.f;
    constexpr int NT = kBk / TG;  // tokens per thread
    using Vec = typename std::conditional<FP8, uint2, uint4>::type;
    Vec vr[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int j = tg + n * TG;
      if (j < nvalid)
        vr[n] = __ldcs(reinterpret_cast<const Vec*>((const unsigned char*)vp +
                                                    (base + j * row_stride + cg * 8) * EB));
    }
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const int j = tg + n * TG;
      if (j >= nvalid) continue;
      float x[8];
      if constexpr (FP8) unpack_e4m3x8(vr[n], x); else unpack_bf16x8(vr[n], x);
#pragma unroll
      for (int h = 0; h < GMAX; ++h)
        if (h < G) {
          const float p = sc[h][j];
#pragma unroll
          for (int i = 0; i < 8; ++i) o[h][i] = fmaf(p, x[i], o[h][i]);
        }
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h)
      if (h < G)
#pragma unroll
        for (int i = 0; i < 8; ++i) red[tg][h][cg * 8 + i] = o[h][i];
  }
  __syncthreads();
  for (int e = tid; e < G * D; e += 128) {
    const int h = e / D, c = e % D;
    float sum = 0.f;
#pragma unroll
    for (int t = 0; t < TG; ++t) sum += red[t][h][c];
    const size_t dst = ((size_t)s * H_q + g * G + h) * k + slot;
    part_o[dst * D + c] = sum * vs / s_l[h];
    if (c == 0) part_lse[dst] = (s_m[h] + __log2f(s_l[h])) * 0.69314718055994531f;
  }
}

template <int D>
__global__ void decode_merge_kernel(const float* __restrict__ part_o,
                                    const float* __restrict__ part_lse,
                                    const int32_t* __restrict__ ids,
                                    const int32_t* __restrict__ seq_lens, int max_pages, int B,
                                    int H_q, int H_kv, int k, uint16_t* __restrict__ out,
                                    float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int G = H_q / H_kv;
  const int64_t n = (int64_t)B * H_q;
  for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < n;
       w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int s = (int)(w / H_q), h = (int)(w % H_q);
    const int32_t* id = ids + ((size_t)s * H_kv + h / G) * k;
    const float* pl = part_lse + (size_t)w * k;
    const int L = seq_lens[s];
    const int lim = (L < 1 || L > max_pages * kBk) ? -1 : (L - 1) / kBk;  // valid ids: 0..lim
    float M = -INFINITY;
    for (int i = 0; i < k; ++i)
      if (id[i] >= 0 && id[i] <= lim) M = fmaxf(M, pl[i]);
    float acc[D / 32];
#pragma unroll
    for (int i = 0; i < D / 32; ++i) acc[i] = 0.f;
    float Lsum = 0.f;
    for (int sl = 0; sl < k; ++sl) {
      if (id[sl] < 0 || id[sl] > lim) continue;
      float wgt = __expf(pl[sl] - M);
      Lsum += wgt;
      const float* po = part_o + ((size_t)w * k + sl) * D;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) acc[i] = fmaf(wgt, po[lane + 32 * i], acc[i]);
    }
    float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
      __nv_bfloat16 bv = __float2bfloat16_rn(acc[i] * inv);
      out[(size_t)w * D + lane + 32 * i] = *reinterpret_cast<uint16_t*>(&bv);
    }
    if (lse && lane == 0) lse[w] = M + logf(Lsum);
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

cudaError_t launch_decode_index(const void* q_idx, const void* k_idx_pages,
                                const int32_t* page_table, const int32_t* seq_lens, int B,
                                int max_pages, int n_g, int d_idx, float* scores,
                                const Diag& dg, cudaStream_t st) {
  int64_t warps = (int64_t)B * max_pages;
  if (warps == 0) return cudaSuccess;
  note_launches(1);
  unsigned grid = (unsigned)std::min<int64_t>((warps + 7) / 8, 152 * 16);
  if (d_idx == 128)
    decode_index_kernel<128><<<grid, 256, 0, st>>>((const uint16_t*)q_idx,
                                                   (const uint16_t*)k_idx_pages, page_table,
                                                   seq_lens, B, max_pages, n_g, scores, dg);
  else
    decode_index_kernel<64><<<grid, 256, 0, st>>>((const uint16_t*)q_idx,
                                                  (const uint16_t*)k_idx_pages, page_table,
                                                  seq_lens, B, max_pages, n_g, scores, dg);
  return cudaGetLastError();
}

size_t decode_ws_bytes(int B, int H_q, int d, int k) {
  return align256((size_t)B * H_q * k * d * 4) + align256((size_t)B * H_q * k * 4);
}

cudaError_t launch_decode_attn(const void* q, const void* k_pages, const void* v_pages,
                               int kv_fp8, const float* k_scale, const float* v_scale,
                               const int32_t* page_table, const int32_t* seq_lens,
                               const int32_t* ids, int B, int max_pages, int H_q, int H_kv,
                               int d, int k, float scale, void* out, float* lse, void* ws,
                               const Diag& dg, cudaStream_t st) {
  float* part_o = (float*)ws;
  float* part_lse = (float*)((unsigned char*)ws + align256((size_t)B * H_q * k * d * 4));
  const float sl2 = scale * 1.4426950408889634f;
  unsigned tasks = (unsigned)((int64_t)B * H_kv * k);
  if (tasks == 0) return cudaSuccess;
  note_launches(2);  // attention, merge
#define MSA_DEC(DD, F8)                                                                    \
  decode_attn_kernel<DD, F8><<<tasks, 128, 0, st>>>(                                       \
      (const uint16_t*)q, k_pages, v_pages, k_scale, v_scale, page_table, seq_lens, ids,   \
      max_pages, H_q, H_kv, k, sl2, part_o, part_lse, dg)
  if (d == 128) {
    if (kv_fp8) MSA_DEC(128, true); else MSA_DEC(128, false);
  } else {
    if (kv_fp8) MSA_DEC(64, true); else MSA_DEC(64, false);
  }
#undef MSA_DEC
  int64_t nw = (int64_t)B * H_q;
  unsigned mg = (unsigned)std::min<int64_t>((nw * 32 + 255) / 256, 152 * 32);
  if (d == 128)
    decode_merge_kernel<128><<<mg, 256, 0, st>>>(part_o, part_lse, ids, seq_lens, max_pages, B,
                                                 H_q, H_kv, k, (uint16_t*)out, lse);
  else
    decode_merge_kernel<64><<<mg, 256, 0, st>>>(part_o, part_lse, ids, seq_lens, max_pages, B,
                                                H_q, H_kv, k, (uint16_t*)out, lse);
  return cudaGetLastError();
}

}  // namespace msa
