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
#include "msa_sm100.cuh"

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

// Pipelined split-KV decode attention. One persistent CTA (256 threads) per SM
// walks the (sequence, group, selected page) tasks blockIdx.x, + gridDim.x, ...
// All tasks' validity and page numbers are looked up once up front; then thread
// 0 keeps two tasks ahead, bulk-copying each task's K block, V block (each one
// contiguous run of the head-major page) and the group's G query rows into a
// 3-stage shared-memory ring, so DRAM latency hides behind the current task.
//   scores  two threads per token (half of d each), reading their K row in a
//           rotated chunk order so the 8 lanes of a quarter warp hit distinct
//           banks;
//   softmax one warp per head;
//   P.V     warp w owns columns [w * D/8, (w+1) * D/8), lanes split the tokens
//           and combine by shuffles; writes the block's normalised output and
//           LSE (the split-KV partials that decode_merge_kernel combines).
constexpr int kDecThreads = 256;
constexpr int kDecStages = 3;
constexpr int kDecMaxTasks = 64;  // tasks per CTA (grid grows beyond the SM count if needed)

struct DecMeta {
  int32_t valid, nvalid, page, parity;
};

template <int D, bool FP8>
struct DecSmem {
  static constexpr int EB = FP8 ? 1 : 2;
  static constexpr int kKVBytes = kBk * D * EB;      // one K or V block
  static constexpr int kQBytes = 8 * D * 2;          // up to 8 query heads (bf16)
  static constexpr int kStageBytes = 2 * kKVBytes + kQBytes;
  static constexpr int kQsOff = kDecStages * kStageBytes;      // fp32 q [8][D]
  static constexpr int kScOff = kQsOff + 8 * D * 4;            // fp32 scores [8][128]
  static constexpr int kStatOff = kScOff + 8 * kBk * 4;        // m, l per head
  static constexpr int kMetaOff = kStatOff + 2 * 8 * 4;
  static constexpr int kBarOff = kMetaOff + kDecMaxTasks * (int)sizeof(DecMeta);
  static constexpr int kBytes = kBarOff + kDecStages * 8 + 16;
};

template <int D, bool FP8>
__global__ void __launch_bounds__(kDecThreads, 1)
decode_attn_kernel(const uint16_t* __restrict__ q, const void* __restrict__ kp,
                   const void* __restrict__ vp, const float* __restrict__ k_scale,
                   const float* __restrict__ v_scale, const int32_t* __restrict__ page_table,
                   const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ ids,
                   int max_pages, int H_q, int H_kv, int k, int64_t n_tasks, float scale_log2,
                   float* __restrict__ part_o, float* __restrict__ part_lse, Diag dg) {
  using namespace sm100;
  using S = DecSmem<D, FP8>;
  constexpr int EB = S::EB;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 127) & ~(uintptr_t)127);
  float* qs = reinterpret_cast<float*>(smem + S::kQsOff);
  float* sc = reinterpret_cast<float*>(smem + S::kScOff);
  float* s_m = reinterpret_cast<float*>(smem + S::kStatOff);
  float* s_l = s_m + 8;
  DecMeta* meta = reinterpret_cast<DecMeta*>(smem + S::kMetaOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + kDecStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = H_q / H_kv;
  const int64_t cnt64 = n_tasks > blockIdx.x ? (n_tasks - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int cnt = (int)(cnt64 < kDecMaxTasks ? cnt64 : kDecMaxTasks);
  auto task_of = [&](int n) -> int64_t { return blockIdx.x + (int64_t)n * gridDim.x; };

  if (tid == 0) {
    for (int s = 0; s < kDecStages; ++s) mbar_init(&full[s], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // look up every task's block, page and visible length in one parallel pass
  for (int n = tid; n < cnt; n += kDecThreads) {
    const int64_t task = task_of(n);
    const int64_t sg = task / k;
    const int s = (int)(sg / H_kv);
    const int id = ids[task];
    const int L = seq_lens[s];
    DecMeta m{0, 0, 0, 0};
    if (id >= 0) {
      if (L < 1 || L > max_pages * kBk || id > (L - 1) / kBk) {
        report(dg, kStatusBadIds);  // the merge skips this slot too
      } else {
        m.valid = 1;
        m.nvalid = min(kBk, L - id * kBk);
        m.page = page_table[(size_t)s * max_pages + id];
      }
    }
    meta[n] = m;
  }
  __syncthreads();
  // thread 0: parity bookkeeping and the bulk copies of task n into its stage
  int issued[kDecStages] = {0, 0, 0};
  auto issue = [&](int n) {
    DecMeta& m = meta[n];
    if (!m.valid) return;
    const int st = n % kDecStages;
    m.parity = issued[st] & 1;
    ++issued[st];
    const int64_t task = task_of(n);
    const int64_t sg = task / k;
    const int g = (int)(sg % H_kv);
    const int s = (int)(sg / H_kv);
    unsigned char* stage = smem + st * S::kStageBytes;
    const size_t blk = ((size_t)m.page * H_kv + g) * kBk * D * EB;  // byte offset of the block
    mbar_arrive_expect_tx(&full[st], 2 * S::kKVBytes + G * D * 2);
    bulk_load(stage, (const unsigned char*)kp + blk, S::kKVBytes, &full[st]);
    bulk_load(stage + S::kKVBytes, (const unsigned char*)vp + blk, S::kKVBytes, &full[st]);
    bulk_load(stage + 2 * S::kKVBytes, q + ((size_t)s * H_q + g * G) * D, G * D * 2, &full[st]);
  };
  if (tid == 0) {
    if (cnt > 0) issue(0);
    if (cnt > 1) issue(1);
  }
  __syncthreads();
  bool ok = true;
  for (int n = 0; n < cnt; ++n) {
    const int st = n % kDecStages;
    if (tid == 0 && n + 2 < cnt) issue(n + 2);  // its stage was released at the end of n-1
    const DecMeta m = meta[n];
    if (m.valid && ok) {
      const int64_t task = task_of(n);
      const int slot = (int)(task % k);
      const int64_t sg = task / k;
      const int g = (int)(sg % H_kv);
      const int s = (int)(sg / H_kv);
      const unsigned char* stage = smem + st * S::kStageBytes;
      int got = 0;
      if (lane == 0) got = mbar_wait(&full[st], (uint32_t)m.parity, abort_flag, dg) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (__syncthreads_and(got) == 0) {
        ok = false;
      } else {
        const float ks = FP8 ? k_scale[g] : 1.f;
        const float vs = FP8 ? v_scale[g] : 1.f;
        const uint16_t* qb = reinterpret_cast<const uint16_t*>(stage + 2 * S::kKVBytes);
        for (int e = tid; e < G * D; e += kDecThreads)
          qs[e] = __uint_as_float((uint32_t)qb[e] << 16);
        __syncthreads();
        // scores: token j = warp * 16 + (lane & 15), half of d = lane >> 4
        {
          constexpr int HALF = D / 2, NCH = HALF / 8;  // 8-element chunks per half
          const int j = warp * 16 + (lane & 15), hf = lane >> 4;
          float acc[8];
#pragma unroll
          for (int h = 0; h < 8; ++h) acc[h] = 0.f;
          const unsigned char* krow = stage + (size_t)j * D * EB + hf * HALF * EB;
#pragma unroll
          for (int c = 0; c < NCH; ++c) {
            const int ch = (c + j) % NCH;  // rotated: distinct banks within a quarter warp
            float x[8];
            if constexpr (FP8) unpack_e4m3x8(*reinterpret_cast<const uint2*>(krow + ch * 8), x);
            else unpack_bf16x8(*reinterpret_cast<const uint4*>(krow + ch * 16), x);
            const int col = hf * HALF + ch * 8;
#pragma unroll
            for (int h = 0; h < 8; ++h)
              if (h < G) {
                const float4 qa = *reinterpret_cast<const float4*>(qs + h * D + col);
                const float4 qc = *reinterpret_cast<const float4*>(qs + h * D + col + 4);
                acc[h] = fmaf(qa.x, x[0], fmaf(qa.y, x[1], fmaf(qa.z, x[2], fmaf(qa.w, x[3], acc[h]))));
                acc[h] = fmaf(qc.x, x[4], fmaf(qc.y, x[5], fmaf(qc.z, x[6], fmaf(qc.w, x[7], acc[h]))));
              }
          }
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            if (h >= G) break;
            float a = acc[h] + __shfl_xor_sync(0xffffffffu, acc[h], 16);
            if (hf == 0) sc[h * kBk + j] = j < m.nvalid ? a * ks * scale_log2 : -INFINITY;
          }
        }
        __syncthreads();
        if (warp < G) {  // softmax of head `warp` over the 128 tokens
          float* row = sc + warp * kBk;
          float mx = -INFINITY;
#pragma unroll
          for (int i = 0; i < kBk / 32; ++i) mx = fmaxf(mx, row[lane + 32 * i]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
          float l = 0.f;
#pragma unroll
          for (int i = 0; i < kBk / 32; ++i) {
            const float p = ex2_approx(row[lane + 32 * i] - mx);
            row[lane + 32 * i] = p;
            l += p;
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
          if (lane == 0) { s_m[warp] = mx; s_l[warp] = l; }
        }
        __syncthreads();
        // P.V: warp owns CPW columns; TQ lane groups split the tokens
        {
          constexpr int CPW = D / 8, TQ = 32 / CPW, TPG = kBk / TQ;
          const int col = warp * CPW + lane % CPW, tq = lane / CPW;
          float o[8];
#pragma unroll
          for (int h = 0; h < 8; ++h) o[h] = 0.f;
          const unsigned char* vblk = stage + S::kKVBytes;
          const int j0 = tq * TPG, j1 = min(j0 + TPG, m.nvalid);
          for (int j = j0; j < j1; ++j) {
            float x;
            if constexpr (FP8) {
              __half_raw hr = __nv_cvt_fp8_to_halfraw(vblk[(size_t)j * D + col], __NV_E4M3);
              x = __half2float(*reinterpret_cast<__half*>(&hr));
            } else {
              x = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(vblk)[(size_t)j * D + col] << 16);
            }
#pragma unroll
            for (int h = 0; h < 8; ++h)
              if (h < G) o[h] = fmaf(sc[h * kBk + j], x, o[h]);
          }
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            if (h >= G) break;
            float a = o[h];
#pragma unroll
            for (int off = CPW; off < 32; off <<= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
            if (tq == 0) {
              const size_t dst = ((size_t)s * H_q + g * G + h) * k + slot;
              part_o[dst * D + col] = a * vs / s_l[h];
              if (col == 0) part_lse[dst] = (s_m[h] + __log2f(s_l[h])) * 0.69314718055994531f;
            }
          }
        }
      }
    }
    __syncthreads();  // stage st, qs and sc are free again
  }
  if (tid == 0 && !ok) {  // let copies in flight land before shared memory goes away
    for (int n = 0; n < cnt; ++n)
      if (meta[n].valid && n < cnt) mbar_drain(&full[n % kDecStages], (uint32_t)meta[n].parity);
  }
  __syncthreads();
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
  const int64_t n_tasks = (int64_t)B * H_kv * k;
  if (n_tasks == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const unsigned grid = (unsigned)std::max<int64_t>(
      std::min<int64_t>(sms, n_tasks), (n_tasks + kDecMaxTasks - 1) / kDecMaxTasks);
  note_launches(2);  // attention, merge
#define MSA_DEC(DD, F8)                                                                    \
  do {                                                                                     \
    const int smem = DecSmem<DD, F8>::kBytes + 128;                                        \
    cudaError_t e = cudaFuncSetAttribute(decode_attn_kernel<DD, F8>,                       \
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem); \
    if (e != cudaSuccess) return e;                                                        \
    decode_attn_kernel<DD, F8><<<grid, kDecThreads, smem, st>>>(                           \
        (const uint16_t*)q, k_pages, v_pages, k_scale, v_scale, page_table, seq_lens, ids, \
        max_pages, H_q, H_kv, k, n_tasks, sl2, part_o, part_lse, dg);                     \
  } while (0)
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
