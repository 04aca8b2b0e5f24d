// MSA decode: one new token per sequence against a paged KV cache whose page
// size equals the block size ("MiniMax Sparse Attention (MSA): a Two-Branch
// Block-Sparse Attention ...", section "运行 Kernel" / running the kernel: page
// size 128, top-k 16, block scores -> selected KV block indexes -> sparse
// attention), with bf16 or FP8-E4M3 K/V ("MiniMax lança MSA ...", section
// "Kernel open source e MiniMax-M3": BF16 and FP8 support).
//
// decode_index_kernel: streams each sequence's shared index-key cache once and
//   max-pools q_idx . k_idx per 128-key page for all groups at once. Keys are
//   the M dimension of mma.m16n8k16 (bf16) or mma.m16n8k32 (E4M3 codes, half
//   the bytes) and the (up to 8) groups its N dimension; the d_idx reduction
//   order is permuted identically in A and B so that each thread reads 16
//   contiguous bytes per key row. HBM-bound.
// Caches: K / V pages are head-major [P, H_kv, 128, d] (the page tensor's second
// dimension is the kv-head count in the usage listing), so the block a group
// reads is one contiguous run; k_idx pages are [P, 128, d_idx].
// decode_attn_kernel: one CTA per (sequence, group, selected block): the G
//   query heads of the group against the block's visible tokens, with the
//   block's K and V bytes all in flight at once (two TMA copies, or 16-byte
//   cp.async for rows narrower than 128 bytes, into swizzled shared memory)
//   and both products on mma.m16n8k16. Each warp scores 32 of the block's
//   tokens; the block's softmax max and P pass through shared memory, and each
//   warp then forms P V for a quarter of the output columns over all 128
//   tokens, so it writes its columns of the block's normalised output (and the
//   LSE) straight from its accumulators (split-KV partials).
// decode_merge_kernel: combines the k partials of every (sequence, head), one
//   warp each, with all of its partial rows in flight at once.
#include <cuda.h>
#include <cudaTypedefs.h>
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

__device__ __forceinline__ void mma_e4m3_16832(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// F8: q_idx and the k_idx pages hold E4M3 codes; out_scale multiplies the
// block scores written (a positive scale of all keys or of a query's row
// ranks the blocks the same)
template <int DI, bool F8>
__global__ void __launch_bounds__(256)
decode_index_kernel(const unsigned char* __restrict__ q_idx,
                    const unsigned char* __restrict__ kpages,
                    const int32_t* __restrict__ page_table, const int32_t* __restrict__ seq_lens,
                    int B, int max_pages, int n_g, float out_scale, float* __restrict__ scores,
                    int64_t ss, Diag dg) {
  constexpr int RB = DI * (F8 ? 1 : 2);  // bytes of one key row
  constexpr int NC = RB / 64;            // 16-byte chunks per thread per key row
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
        bq[i] = *reinterpret_cast<const uint4*>(q_idx + ((size_t)s * n_g + gq) * RB +
                                                16 * (t4 + 4 * i));
    }
    const int64_t page = page_table[(size_t)s * max_pages + b];
    const unsigned char* base = kpages + (size_t)page * kBk * RB;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll (F8 ? 4 : 2)
    for (int m = 0; m < kBk / 16; ++m) {
      const int key0 = m * 16 + gq, key1 = key0 + 8;
      uint4 a0[NC], a1[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        a0[i] = __ldg(reinterpret_cast<const uint4*>(base + (size_t)key0 * RB + 16 * (t4 + 4 * i)));
        a1[i] = __ldg(reinterpret_cast<const uint4*>(base + (size_t)key1 * RB + 16 * (t4 + 4 * i)));
      }
      float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        if constexpr (F8) {
          mma_e4m3_16832(c, a0[i].x, a1[i].x, a0[i].y, a1[i].y, bq[i].x, bq[i].y);
          mma_e4m3_16832(c, a0[i].z, a1[i].z, a0[i].w, a1[i].w, bq[i].z, bq[i].w);
        } else {
          mma_bf16_16816(c, a0[i].x, a1[i].x, a0[i].y, a1[i].y, bq[i].x, bq[i].y);
          mma_bf16_16816(c, a0[i].z, a1[i].z, a0[i].w, a1[i].w, bq[i].z, bq[i].w);
        }
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
      if (g0 < n_g) scores[((size_t)s * n_g + g0) * ss + b] = F8 ? mx0 * out_scale : mx0;
      if (g1 < n_g) scores[((size_t)s * n_g + g1) * ss + b] = F8 ? mx1 * out_scale : mx1;
    }
  }
}

// ---- decode attention: one CTA (4 warps) per (sequence, group, selected block)
//
// The block's K and V rows (32 KB each in bf16, 16 KB in E4M3 at d = 128) are
// all put in flight at once by cp.async into shared memory, K in one group and
// V in a second, so a CTA keeps its whole block's bytes outstanding; rows past
// the sequence end are zero-filled by the copy itself. Shared rows are stored
// with their 16-byte chunks XOR-swizzled by (row mod 8), so the fragment loads
// below are free of bank conflicts.
//
// Warp w owns tokens 32w .. 32w+31 of the block. S = q K^T and O = P V run on
// mma.m16n8k16 (bf16 operands, fp32 accumulate): the G <= 8 query heads of the
// group are rows 0..G-1 of the 16-row A operand (the other rows are zero), so
// the S accumulators hand P to the P.V A operand without any data movement.
// E4M3 codes are widened to bf16 exactly (every E4M3 value is a bf16 value);
// the per-head scales multiply the scores and the output. Each warp keeps its
// own row max and sum; the four are combined in shared memory into the block's
// normalised output and LSE (split-KV partials, merged by decode_merge_kernel).
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ uint32_t lds_u16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];\n" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];\n" : "=h"(v) : "r"(a));
  return v;
}
// two E4M3 codes (first in the low byte) -> bf16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  return pack_bf16x2(f.x, f.y);
}
// byte offset of 16-byte chunk c of token row r in a swizzled K or V tile
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  constexpr int kCpr = ROWB / 16;
  constexpr int kMask = kCpr >= 8 ? 7 : kCpr - 1;
  return (uint32_t)(r * ROWB + ((c ^ (r & kMask)) << 4));
}

// ---- decode index scan over an NVFP4 k_idx cache
//
// Keys are E2M1 codes, two per byte (the even dimension in the low nibble),
// with one E4M3 scale per 16 consecutive dimensions of a key ("micro-block");
// a key's value in dimension c is e2m1 * scale[c / 16]. One warp per
// (sequence, page): it copies the page's codes and scales into its own shared
// buffer (cp.async: a whole page's bytes in flight per warp), then for every
// 16 keys runs one mma.m16n8k16 per micro-block (keys x the groups' q_idx, f16
// operands: every E2M1 value is an f16 value, and q_idx is rounded to f16) and
// adds the product times the keys' scales of that micro-block into fp32, so
// the scales never touch the operands. Within a micro-block the four lanes of
// a row take 4 contiguous dimensions each (one 16-bit read), and q_idx is
// permuted the same way.
__device__ __forceinline__ void mma_f16_16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)byte, __NV_E4M3);
  return __half2float(__ushort_as_half(h.x));
}

constexpr int kFp4Warps = 4;

template <int DI>
__global__ void __launch_bounds__(kFp4Warps * 32)
decode_index_fp4_kernel(const uint16_t* __restrict__ q_idx, const unsigned char* __restrict__ codes,
                        const unsigned char* __restrict__ kscales,
                        const int32_t* __restrict__ page_table,
                        const int32_t* __restrict__ seq_lens, int B, int max_pages, int n_g,
                        float out_scale, float* __restrict__ scores, int64_t srow, Diag dg) {
  constexpr int CB = DI / 2;    // code bytes per key
  constexpr int SB = DI / 16;   // scale bytes per key
  constexpr int KS = DI / 16;   // micro-blocks = k-steps
  static_assert(SB == 4 || SB == 8, "d_idx is 64 or 128");
  constexpr int WBYTES = kBk * (CB + SB);
  extern __shared__ __align__(128) unsigned char f4s[];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int gq = lane >> 2, t4 = lane & 3;
  unsigned char* sc = f4s + wi * WBYTES;  // codes [128][CB], then scales [128][SB]
  unsigned char* ss = sc + kBk * CB;
  const uint32_t sc_a = smem_addr(sc), ss_a = smem_addr(ss);
  const int64_t n_tasks = (int64_t)B * max_pages;
  for (int64_t task = (int64_t)blockIdx.x * kFp4Warps + wi; task < n_tasks;
       task += (int64_t)gridDim.x * kFp4Warps) {
    const int s = (int)(task / max_pages);
    const int b = (int)(task % max_pages);
    const int L = seq_lens[s];
    if (L < 1 || L > max_pages * kBk) {
      if (b == 0 && lane == 0) report(dg, kStatusBadIds);
      continue;
    }
    if ((int64_t)b * kBk >= L) continue;
    const int nvalid = min(kBk, L - b * kBk);
    const int64_t page = page_table[(size_t)s * max_pages + b];
    const unsigned char* gc = codes + (size_t)page * kBk * CB;
    const unsigned char* gs = kscales + (size_t)page * kBk * SB;
    __syncwarp();  // the previous task's reads of the buffer are done
    for (int e = lane; e < kBk * CB / 16; e += 32) cp_async16(sc_a + e * 16, gc + e * 16, 16u);
    for (int e = lane; e < kBk * SB / 16; e += 32) cp_async16(ss_a + e * 16, gs + e * 16, 16u);
    cp_async_commit();
    // B operand: group gq's q_idx in f16, dimensions 16 ks + 4 t4 + {0,1} | {2,3}
    uint32_t bq[KS][2];
    const uint16_t* qr = q_idx + ((size_t)s * n_g + (gq < n_g ? gq : 0)) * DI;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const uint2 w = gq < n_g ? *reinterpret_cast<const uint2*>(qr + 16 * ks + 4 * t4)
                               : make_uint2(0u, 0u);
      bq[ks][0] = f16x2_of(bf16_lo(w.x), bf16_hi(w.x));
      bq[ks][1] = f16x2_of(bf16_lo(w.y), bf16_hi(w.y));
    }
    cp_async_wait<0>();
    __syncwarp();
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll 2
    for (int m = 0; m < kBk / 16; ++m) {
      const int key0 = m * 16 + gq, key1 = key0 + 8;
      uint2 s0, s1;  // the keys' micro-block scales (E4M3 bytes)
      if constexpr (SB == 8) {
        s0 = *reinterpret_cast<const uint2*>(ss + key0 * SB);
        s1 = *reinterpret_cast<const uint2*>(ss + key1 * SB);
      } else {
        s0 = make_uint2(*reinterpret_cast<const uint32_t*>(ss + key0 * SB), 0u);
        s1 = make_uint2(*reinterpret_cast<const uint32_t*>(ss + key1 * SB), 0u);
      }
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const uint32_t c0 = lds_u16(sc_a + key0 * CB + 8 * ks + 2 * t4);
        const uint32_t c1 = lds_u16(sc_a + key1 * CB + 8 * ks + 2 * t4);
        float p[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16_16816(p, e2m1x2_to_f16x2(c0 & 0xFF), e2m1x2_to_f16x2(c1 & 0xFF),
                      e2m1x2_to_f16x2(c0 >> 8), e2m1x2_to_f16x2(c1 >> 8), bq[ks][0], bq[ks][1]);
        const uint32_t w0 = ks < 4 ? s0.x : s0.y, w1 = ks < 4 ? s1.x : s1.y;
        const float f0 = e4m3_to_float((w0 >> (8 * (ks & 3))) & 0xFF);
        const float f1 = e4m3_to_float((w1 >> (8 * (ks & 3))) & 0xFF);
        acc[0] = fmaf(p[0], f0, acc[0]);
        acc[1] = fmaf(p[1], f0, acc[1]);
        acc[2] = fmaf(p[2], f1, acc[2]);
        acc[3] = fmaf(p[3], f1, acc[3]);
      }
      if (key0 < nvalid) { mx0 = fmaxf(mx0, acc[0]); mx1 = fmaxf(mx1, acc[1]); }
      if (key1 < nvalid) { mx0 = fmaxf(mx0, acc[2]); mx1 = fmaxf(mx1, acc[3]); }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    if (gq == 0) {
      const int g0 = 2 * t4, g1 = 2 * t4 + 1;
      if (g0 < n_g) scores[((size_t)s * n_g + g0) * srow + b] = mx0 * out_scale;
      if (g1 < n_g) scores[((size_t)s * n_g + g1) * srow + b] = mx1 * out_scale;
    }
  }
}

// K / V rows of 128 bytes or a multiple of it arrive by TMA (one thread, two
// mbarriers, 128-byte swizzled boxes through a 3-D map over the pages; a whole
// block as 128-row boxes, the partial last block as the 16-row boxes that hold
// its tokens); narrower rows by 16-byte cp.async into the row-swizzled layout
template <int D, bool FP8>
__host__ __device__ constexpr bool dec_tma() {
  return (D * (FP8 ? 1 : 2)) % 128 == 0;
}
template <int D, bool FP8>
constexpr int dec_smem_bytes() {
  // K and V tiles, then the combine's m / l and (TMA) two mbarriers
  return 2 * kBk * D * (FP8 ? 1 : 2) + 2 * 32 * 4 + 16;
}

// byte offset of 16-byte unit c of row r in a tile that arrived as 128-byte
// swizzled boxes: chunk c / 8 of 128 bytes per row at (c / 8) * 16 KB, the
// units XOR-ed with r % 8
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return (uint32_t)((c >> 3) * (kBk * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D, bool FP8>
__global__ void __launch_bounds__(128, FP8 ? 6 : 3)
decode_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_k16,
                   const __grid_constant__ CUtensorMap tm_v16,
                   const uint16_t* __restrict__ q, const void* __restrict__ kp,
                   const void* __restrict__ vp, const float* __restrict__ k_scale,
                   const float* __restrict__ v_scale, const int32_t* __restrict__ page_table,
                   const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ ids,
                   int max_pages, int H_q, int H_kv, int k, float scale_log2,
                   float* __restrict__ part_o, float* __restrict__ part_lse, Diag dg) {
  constexpr int EB = FP8 ? 1 : 2;
  constexpr int ROWB = D * EB;      // bytes of one token row
  constexpr int CPR = ROWB / 16;    // 16-byte chunks per row
  constexpr int TILE = kBk * ROWB;  // bytes of one K or V block
  constexpr int KS = D / 16;        // k-steps of q K^T
  constexpr int NC = D / 8;         // 8-column tiles of P V
  constexpr bool TMA = dec_tma<D, FP8>();
  static_assert(8 * (kBk / 2 + 4) * 4 <= TILE, "P fits the K tile");
  extern __shared__ __align__(1024) unsigned char dsm[];
  // tile addressing: TMA boxes or the cp.async layout
  auto tile_off = [](int r, int c) -> uint32_t {
    if constexpr (TMA) return sw128(r, c);
    else return swz<ROWB>(r, c);
  };
  float(*s_m)[8] = reinterpret_cast<float(*)[8]>(dsm + 2 * TILE);
  float(*s_l)[8] = reinterpret_cast<float(*)[8]>(dsm + 2 * TILE + 128);
  uint64_t* kv_bar = reinterpret_cast<uint64_t*>(dsm + 2 * TILE + 256);  // K, V landed (TMA)

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int gq = lane >> 2, t4 = lane & 3;
  const int G = H_q / H_kv;
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
  // pages are head-major [P, H_kv, Bk, D]: the (page, head g) block is contiguous
  const size_t blk = ((size_t)page * H_kv + g) * TILE;
  const unsigned char* gk = (const unsigned char*)kp + blk;
  const unsigned char* gv = (const unsigned char*)vp + blk;
  const uint32_t sk = smem_addr(dsm), sv = sk + TILE;
  volatile int abort_flag = 0;  // this thread's waits only
  if constexpr (TMA) {
    if (sk & 1023) {
      if (tid == 0) report(dg, kStatusUnsupported);
      return;
    }
    if (tid == 0) {
      sm100::mbar_init(&kv_bar[0], 1);
      sm100::mbar_init(&kv_bar[1], 1);
      sm100::fence_barrier_init();
    }
    __syncthreads();
    if (tid == 0) {
      const int32_t z = (int32_t)(page * H_kv + g);
      if (nvalid == kBk) {  // a whole block: one 128-row box per 128-byte column chunk
        sm100::mbar_arrive_expect_tx(&kv_bar[0], TILE);
#pragma unroll
        for (int c = 0; c < ROWB / 128; ++c)
          sm100::tma_load_3d(dsm + c * kBk * 128, &tm_k, &kv_bar[0], c * (128 / EB), 0, z);
        sm100::mbar_arrive_expect_tx(&kv_bar[1], TILE);
#pragma unroll
        for (int c = 0; c < ROWB / 128; ++c)
          sm100::tma_load_3d(dsm + TILE + c * kBk * 128, &tm_v, &kv_bar[1], c * (128 / EB), 0,
                             z);
      } else {  // the partial last block: only its 16-row groups that hold tokens
        const int nbox = (nvalid + 15) >> 4;
        const uint32_t bytes = (uint32_t)(nbox * 16 * ROWB);
        sm100::mbar_arrive_expect_tx(&kv_bar[0], bytes);
        for (int c = 0; c < ROWB / 128; ++c)
          for (int b = 0; b < nbox; ++b)
            sm100::tma_load_3d(dsm + c * kBk * 128 + b * 16 * 128, &tm_k16, &kv_bar[0],
                               c * (128 / EB), 16 * b, z);
        sm100::mbar_arrive_expect_tx(&kv_bar[1], bytes);
        for (int c = 0; c < ROWB / 128; ++c)
          for (int b = 0; b < nbox; ++b)
            sm100::tma_load_3d(dsm + TILE + c * kBk * 128 + b * 16 * 128, &tm_v16, &kv_bar[1],
                               c * (128 / EB), 16 * b, z);
      }
    }
  } else {
#pragma unroll 4
    for (int e = tid; e < kBk * CPR; e += 128) {
      const int r = e / CPR;
      cp_async16(sk + swz<ROWB>(r, e % CPR), gk + (size_t)e * 16, r < nvalid ? 16u : 0u);
    }
    cp_async_commit();
#pragma unroll 4
    for (int e = tid; e < kBk * CPR; e += 128) {
      const int r = e / CPR;
      cp_async16(sv + swz<ROWB>(r, e % CPR), gv + (size_t)e * 16, r < nvalid ? 16u : 0u);
    }
    cp_async_commit();
  }

  // A operand rows: head gq of the group (rows >= G and the upper 8 rows are zero)
  uint32_t qa[KS][2];
  {
    const uint16_t* qr = q + ((size_t)s * H_q + (size_t)g * G + (gq < G ? gq : 0)) * D;
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      qa[i][0] = gq < G ? *reinterpret_cast<const uint32_t*>(qr + 16 * i + 2 * t4) : 0u;
      qa[i][1] = gq < G ? *reinterpret_cast<const uint32_t*>(qr + 16 * i + 8 + 2 * t4) : 0u;
    }
  }
  const float cs = scale_log2 * (FP8 ? k_scale[g] : 1.f);
  const float vs = FP8 ? v_scale[g] : 1.f;
  const int tok0 = 32 * w;

  if constexpr (TMA) {  // K has landed (a timed-out wait lets both copies land, then leaves)
    if (!sm100::mbar_wait(&kv_bar[0], 0, &abort_flag, dg)) {
      sm100::mbar_drain(&kv_bar[0], 0);
      sm100::mbar_drain(&kv_bar[1], 0);
      return;
    }
  } else {
    cp_async_wait<1>();  // this thread's K chunks have landed
    __syncthreads();     // everyone's have
  }
  float sacc[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.f;
  if constexpr (!FP8) {
#pragma unroll
    for (int p = 0; p < KS / 2; ++p)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sk + tile_off(tok0 + 8 * nt + (lane & 7), 4 * p + (lane >> 3)), b0, b1, b2, b3);
        mma_bf16_16816(sacc[nt], qa[2 * p][0], 0u, qa[2 * p][1], 0u, b0, b1);
        mma_bf16_16816(sacc[nt], qa[2 * p + 1][0], 0u, qa[2 * p + 1][1], 0u, b2, b3);
      }
  } else {
#pragma unroll
    for (int i = 0; i < KS; ++i)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const uint32_t a = sk + tile_off(tok0 + 8 * nt + gq, i);
        const uint32_t b0 = e4m3x2_to_bf16x2(lds_u16(a + 2 * t4));
        const uint32_t b1 = e4m3x2_to_bf16x2(lds_u16(a + 8 + 2 * t4));
        mma_bf16_16816(sacc[nt], qa[i][0], 0u, qa[i][1], 0u, b0, b1);
      }
  }

  // softmax of head gq over the block: each warp's max over its 32 tokens
  // (masked past nvalid), then the block max through shared memory
  float pr[4][2];
  float mw = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = tok0 + 8 * nt + 2 * t4 + i;
      pr[nt][i] = j < nvalid ? sacc[nt][i] * cs : -INFINITY;
      mw = fmaxf(mw, pr[nt][i]);
    }
  mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 1));
  mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 2));
  if (t4 == 0) s_m[w][gq] = mw;
  __syncthreads();  // every warp's max is in, and every warp is done with K
  // finite: token 0 is valid and belongs to warp 0
  const float M = fmaxf(fmaxf(s_m[0][gq], s_m[1][gq]), fmaxf(s_m[2][gq], s_m[3][gq]));
  // P (bf16 pairs, [8 heads][128 tokens], rows padded to PW words so that a
  // warp's fragment loads hit 32 banks) over the K tile
  constexpr int PW = kBk / 2 + 4;
  uint32_t* pw = reinterpret_cast<uint32_t*>(dsm) + gq * PW + t4;
  float lw = 0.f;
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const float p0 = ex2_approx(pr[nt][0] - M), p1 = ex2_approx(pr[nt][1] - M);
    lw += p0 + p1;
    pw[(tok0 + 8 * nt) / 2] = pack_bf16x2(p0, p1);
  }
  lw += __shfl_xor_sync(0xffffffffu, lw, 1);
  lw += __shfl_xor_sync(0xffffffffu, lw, 2);
  if (t4 == 0) s_l[w][gq] = lw;

  if constexpr (TMA) {
    if (!sm100::mbar_wait(&kv_bar[1], 0, &abort_flag, dg)) {  // V has landed
      sm100::mbar_drain(&kv_bar[1], 0);
      return;
    }
    // the block's rows past its last token hold other data: zero them (their P
    // is 0, and 0 times a NaN is not)
    for (int e = nvalid * CPR + tid; e < kBk * CPR; e += 128)
      sm100::st_shared_v4(sv + tile_off(e / CPR, e % CPR), 0u, 0u, 0u, 0u);
  } else {
    cp_async_wait<0>();  // V has landed
  }
  __syncthreads();  // P, the sums and V are complete

  // O[:, warp's quarter of the columns] = P V over the block's 128 tokens
  constexpr int NW = NC / 4;  // 8-column tiles per warp
  const int cb = w * NW;      // the warp's first 8-column tile
  float o[NW][4];
#pragma unroll
  for (int n = 0; n < NW; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
#pragma unroll
  for (int j = 0; j < kBk / 16; ++j) {  // 16 tokens per k-step
    const uint32_t a0 = pw[8 * j], a2 = pw[8 * j + 4];  // tokens 16 j + 2 t4 (+ 8)
    if constexpr (!FP8) {
      const int r = 16 * j + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int n = 0; n < NW; n += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sv + tile_off(r, cb + n + (lane >> 4)), b0, b1, b2, b3);
        mma_bf16_16816(o[n], a0, 0u, a2, 0u, b0, b1);
        mma_bf16_16816(o[n + 1], a0, 0u, a2, 0u, b2, b3);
      }
    } else {
      const int r = 16 * j + 2 * t4;
#pragma unroll
      for (int n = 0; n < NW; ++n) {
        const int col = 8 * (cb + n) + gq;
        const int ch = col >> 4, by = col & 15;
        const uint32_t v00 = lds_u8(sv + tile_off(r, ch) + by);
        const uint32_t v01 = lds_u8(sv + tile_off(r + 1, ch) + by);
        const uint32_t v10 = lds_u8(sv + tile_off(r + 8, ch) + by);
        const uint32_t v11 = lds_u8(sv + tile_off(r + 9, ch) + by);
        mma_bf16_16816(o[n], a0, 0u, a2, 0u, e4m3x2_to_bf16x2(v00 | (v01 << 8)),
                       e4m3x2_to_bf16x2(v10 | (v11 << 8)));
      }
    }
  }
  // the block's partial for head gq: its columns straight from the accumulators
  if (gq < G) {
    const float l = (s_l[0][gq] + s_l[1][gq]) + (s_l[2][gq] + s_l[3][gq]);
    const float f = vs / l;
    const size_t dst = ((size_t)s * H_q + (size_t)g * G + gq) * k + slot;
    float* po = part_o + dst * D + 8 * cb + 2 * t4;
#pragma unroll
    for (int n = 0; n < NW; ++n)
      *reinterpret_cast<float2*>(po + 8 * n) = make_float2(o[n][0] * f, o[n][1] * f);
    if (w == 0 && t4 == 0) part_lse[dst] = (M + __log2f(l)) * 0.69314718055994531f;
  }
}

// ---- decode attention over an NVFP4 K/V cache
//
// K and V pages hold E2M1 codes [P, H_kv, 128, D / 2] (two per byte, the even
// dimension in the low nibble) and one E4M3 scale per 16 dimensions of a row
// [P, H_kv, 128, D / 16]; a value is its code times its scale. One CTA per
// (sequence, group, selected block), as decode_attn_kernel: the block's codes
// and scales arrive by cp.async (rows past the sequence end zero-filled, so
// they decode to 0). q . K^T runs per 16-dimension micro-block on
// mma.m16n8k16 with f16 operands (every E2M1 value is an f16 value; q is
// rounded to f16), the key's scale multiplying each micro-block's product in
// fp32 (a key's scales read in one load and converted two at a time); within
// a micro-block the four lanes of a row take 4 contiguous dimensions each (one
// 16-bit read), and q is permuted the same way. V is widened once into an f16
// tile (a code times an E4M3 scale has at most 5 significant bits and lies in
// f16's normal range, so the widening is exact), and P . V runs on f16
// operands, reading V by ldmatrix.trans as the bf16 path does.
template <int D>
constexpr int dec_fp4_smem_bytes() {
  return 2 * kBk * (D / 2) + 2 * kBk * (D / 16) + kBk * D * 2 + 2 * 32 * 4;
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(a));
  return v;
}
// two E4M3 codes (first in the low byte) -> two floats, exact
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}
__device__ __forceinline__ uint2 lds_u64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

template <int D>
__global__ void __launch_bounds__(128, 4)
decode_attn_fp4_kernel(const uint16_t* __restrict__ q, const uint8_t* __restrict__ kc,
                       const uint8_t* __restrict__ ksc, const uint8_t* __restrict__ vc,
                       const uint8_t* __restrict__ vsc, const int32_t* __restrict__ page_table,
                       const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ ids,
                       int max_pages, int H_q, int H_kv, int k, float scale_log2,
                       float* __restrict__ part_o, float* __restrict__ part_lse, Diag dg) {
  constexpr int CB = D / 2;          // code bytes of a row
  constexpr int SB = D / 16;         // scale bytes of a row
  constexpr int CCH = CB / 16;       // 16-byte chunks of a code row
  constexpr int CTILE = kBk * CB;
  constexpr int STILE = kBk * SB;
  constexpr int VROWB = D * 2;       // bf16 row of the widened V tile
  constexpr int MB = D / 16;         // micro-blocks of a row
  constexpr int NC = D / 8;          // 8-column tiles of P V
  // (declared as in decode_attn_kernel, whose TMA boxes need 1024-byte alignment)
  extern __shared__ __align__(1024) unsigned char dsm[];
  const uint32_t s_kc = smem_addr(dsm), s_vc = s_kc + CTILE;
  const uint32_t s_ks = s_vc + CTILE, s_vs = s_ks + STILE;
  const uint32_t s_vb = s_vs + STILE;  // widened V (f16, row-swizzled)
  float(*s_m)[8] = reinterpret_cast<float(*)[8]>(dsm + 2 * CTILE + 2 * STILE + kBk * VROWB);
  float(*s_l)[8] = s_m + 4;

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int gq = lane >> 2, t4 = lane & 3;
  const int G = H_q / H_kv;
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
  const size_t blk = (size_t)page * H_kv + g;  // the (page, head g) block of codes / scales
  const unsigned char* gkc = kc + blk * CTILE;
  const unsigned char* gvc = vc + blk * CTILE;
  const unsigned char* gks = ksc + blk * STILE;
  const unsigned char* gvs = vsc + blk * STILE;
  // K codes and scales, then V codes and scales (rows past nvalid read as 0)
#pragma unroll
  for (int e = tid; e < kBk * CCH; e += 128) {
    const int r = e / CCH;
    cp_async16(s_kc + swz<CB>(r, e % CCH), gkc + (size_t)e * 16, r < nvalid ? 16u : 0u);
  }
#pragma unroll
  for (int e = tid; e < STILE / 16; e += 128) {
    const int r0 = e * 16 / SB;  // first row of the chunk
    const int nb = max(0, min(16, (nvalid - r0) * SB));
    cp_async16(s_ks + e * 16, gks + (size_t)e * 16, (uint32_t)nb);
  }
  cp_async_commit();
#pragma unroll
  for (int e = tid; e < kBk * CCH; e += 128) {
    const int r = e / CCH;
    cp_async16(s_vc + swz<CB>(r, e % CCH), gvc + (size_t)e * 16, r < nvalid ? 16u : 0u);
  }
#pragma unroll
  for (int e = tid; e < STILE / 16; e += 128) {
    const int r0 = e * 16 / SB;
    const int nb = max(0, min(16, (nvalid - r0) * SB));
    cp_async16(s_vs + e * 16, gvs + (size_t)e * 16, (uint32_t)nb);
  }
  cp_async_commit();

  // A operand: head gq of the group in f16, each micro-block's dimensions in
  // the lanes' order (lane t4 holds dims 4 t4 .. 4 t4 + 3)
  uint32_t qa[MB][2];
  {
    const uint16_t* qr = q + ((size_t)s * H_q + (size_t)g * G + (gq < G ? gq : 0)) * D;
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) {
      const uint2 v = *reinterpret_cast<const uint2*>(qr + mb * 16 + 4 * t4);
      const float x0 = __uint_as_float(v.x << 16), x1 = __uint_as_float(v.x & 0xFFFF0000u);
      const float x2 = __uint_as_float(v.y << 16), x3 = __uint_as_float(v.y & 0xFFFF0000u);
      qa[mb][0] = gq < G ? f16x2_of(x0, x1) : 0u;
      qa[mb][1] = gq < G ? f16x2_of(x2, x3) : 0u;
    }
  }
  const int tok0 = 32 * w;

  cp_async_wait<1>();  // this thread's K chunks have landed
  __syncthreads();     // everyone's have
  float sacc[4][2];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) sacc[nt][0] = sacc[nt][1] = 0.f;
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int kr = tok0 + 8 * nt + gq;           // the key of this lane's B fragment
    const int key0 = tok0 + 8 * nt + 2 * t4;     // the keys of this lane's accumulators
    // the two keys' scales (SB bytes each), as floats
    float sc0[MB], sc1[MB];
#pragma unroll
    for (int u = 0; u < SB / 4; ++u) {
      const uint32_t w0 = lds_u32(s_ks + key0 * SB + 4 * u);
      const uint32_t w1 = lds_u32(s_ks + (key0 + 1) * SB + 4 * u);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const float2 f0 = e4m3x2_to_float2((w0 >> (16 * hh)) & 0xFFFF);
        const float2 f1 = e4m3x2_to_float2((w1 >> (16 * hh)) & 0xFFFF);
        sc0[4 * u + 2 * hh] = f0.x;
        sc0[4 * u + 2 * hh + 1] = f0.y;
        sc1[4 * u + 2 * hh] = f1.x;
        sc1[4 * u + 2 * hh + 1] = f1.y;
      }
    }
#pragma unroll
    for (int mb = 0; mb < MB; ++mb) {
      const uint32_t c = lds_u16(s_kc + swz<CB>(kr, mb >> 1) + (mb & 1) * 8 + 2 * t4);
      float p[4] = {0.f, 0.f, 0.f, 0.f};
      mma_f16_16816(p, qa[mb][0], 0u, qa[mb][1], 0u, e2m1x2_to_f16x2(c & 0xFF),
                    e2m1x2_to_f16x2(c >> 8));
      sacc[nt][0] = fmaf(p[0], sc0[mb], sacc[nt][0]);
      sacc[nt][1] = fmaf(p[1], sc1[mb], sacc[nt][1]);
    }
  }

  // softmax of head gq over the block: each warp's max over its 32 tokens
  // (masked past nvalid), then the block max through shared memory
  float pr[4][2];
  float mw = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int j = tok0 + 8 * nt + 2 * t4 + i;
      pr[nt][i] = j < nvalid ? sacc[nt][i] * scale_log2 : -INFINITY;
      mw = fmaxf(mw, pr[nt][i]);
    }
  mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 1));
  mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 2));
  if (t4 == 0) s_m[w][gq] = mw;
  cp_async_wait<0>();  // this thread's V chunks have landed
  __syncthreads();     // every warp's max and V chunks are in, every warp is done with K
  // finite: token 0 is valid and belongs to warp 0
  const float M = fmaxf(fmaxf(s_m[0][gq], s_m[1][gq]), fmaxf(s_m[2][gq], s_m[3][gq]));
  // P (f16 pairs, [8 heads][128 tokens], rows padded to PW words so that a
  // warp's fragment loads hit 32 banks) over the K codes
  constexpr int PW = kBk / 2 + 4;
  static_assert(8 * PW * 4 <= CTILE, "P fits the K code tile");
  uint32_t* pw = reinterpret_cast<uint32_t*>(dsm) + gq * PW + t4;
  float lw = 0.f;
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const float p0 = ex2_approx(pr[nt][0] - M), p1 = ex2_approx(pr[nt][1] - M);
    lw += p0 + p1;
    pw[(tok0 + 8 * nt) / 2] = f16x2_of(p0, p1);
  }
  lw += __shfl_xor_sync(0xffffffffu, lw, 1);
  lw += __shfl_xor_sync(0xffffffffu, lw, 2);
  if (t4 == 0) s_l[w][gq] = lw;

  // V: widen codes times scales to f16 (exact), 16 dimensions (8 code bytes)
  // per job
#pragma unroll 2
  for (int e = tid; e < kBk * MB; e += 128) {
    const int r = e / MB, gi = e % MB;
    const uint2 c8 = lds_u64(s_vc + swz<CB>(r, gi >> 1) + (gi & 1) * 8);
    const __half_raw hs = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)lds_u8(s_vs + r * SB + gi),
                                                  __NV_E4M3);
    const __half2 sc2 = __halves2half2(__half(hs), __half(hs));
    uint32_t wv[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t byte = ((b < 4 ? c8.x : c8.y) >> (8 * (b & 3))) & 0xFF;
      const uint32_t h2 = e2m1x2_to_f16x2(byte);
      const __half2 v2 = __hmul2(*reinterpret_cast<const __half2*>(&h2), sc2);
      wv[b] = *reinterpret_cast<const uint32_t*>(&v2);
    }
    sm100::st_shared_v4(s_vb + swz<VROWB>(r, 2 * gi), wv[0], wv[1], wv[2], wv[3]);
    sm100::st_shared_v4(s_vb + swz<VROWB>(r, 2 * gi + 1), wv[4], wv[5], wv[6], wv[7]);
  }
  __syncthreads();  // P, the sums and the widened V are complete

  // O[:, warp's quarter of the columns] = P V over the block's 128 tokens
  constexpr int NW = NC / 4;  // 8-column tiles per warp
  const int cb = w * NW;      // the warp's first 8-column tile
  float o[NW][4];
#pragma unroll
  for (int n = 0; n < NW; ++n)
#pragma unroll
    for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
#pragma unroll
  for (int j = 0; j < kBk / 16; ++j) {  // 16 tokens per k-step
    const uint32_t a0 = pw[8 * j], a2 = pw[8 * j + 4];  // tokens 16 j + 2 t4 (+ 8)
    const int r = 16 * j + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int n = 0; n < NW; n += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(s_vb + swz<VROWB>(r, cb + n + (lane >> 4)), b0, b1, b2, b3);
      mma_f16_16816(o[n], a0, 0u, a2, 0u, b0, b1);
      mma_f16_16816(o[n + 1], a0, 0u, a2, 0u, b2, b3);
    }
  }
  // the block's partial for head gq: its columns straight from the accumulators
  if (gq < G) {
    const float l = (s_l[0][gq] + s_l[1][gq]) + (s_l[2][gq] + s_l[3][gq]);
    const float f = 1.f / l;
    const size_t dst = ((size_t)s * H_q + (size_t)g * G + gq) * k + slot;
    float* po = part_o + dst * D + 8 * cb + 2 * t4;
#pragma unroll
    for (int n = 0; n < NW; ++n)
      *reinterpret_cast<float2*>(po + 8 * n) = make_float2(o[n][0] * f, o[n][1] * f);
    if (w == 0 && t4 == 0) part_lse[dst] = (M + __log2f(l)) * 0.69314718055994531f;
  }
}

// One warp per (sequence, head). Lane i < k holds slot i: its block id, its
// LSE and (through the warp reductions) the slot's weight. Every lane owns D/32
// contiguous output columns, and the k partial rows of those columns are all
// requested before the first is used, so a warp waits on memory about twice
// (the ids and LSEs, then the rows) instead of once per slot. Slots whose block
// id is invalid get weight 0 and their rows, which the attention kernel may not
// have written, are never added.
template <int D>
__global__ void __launch_bounds__(256)
decode_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                    const int32_t* __restrict__ ids, const int32_t* __restrict__ seq_lens,
                    int max_pages, int B, int H_q, int H_kv, int k, uint16_t* __restrict__ out,
                    float* __restrict__ lse) {
  constexpr int PER = D / 32;
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int G = H_q / H_kv;
  const int64_t n = (int64_t)B * H_q;
  for (int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < n;
       w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int s = (int)(w / H_q), h = (int)(w % H_q);
    const float* po = part_o + (size_t)w * k * D + lane * PER;
    float x[kMaxK][PER];
#pragma unroll
    for (int sl = 0; sl < kMaxK; ++sl) {
      if (sl < k) {
        if constexpr (PER == 4) {
          const float4 t = __ldcs(reinterpret_cast<const float4*>(po + (size_t)sl * D));
          x[sl][0] = t.x; x[sl][1] = t.y; x[sl][2] = t.z; x[sl][3] = t.w;
        } else {
          const float2 t = __ldcs(reinterpret_cast<const float2*>(po + (size_t)sl * D));
          x[sl][0] = t.x; x[sl][1] = t.y;
        }
      }
    }
    const int L = seq_lens[s];
    const int lim = (L < 1 || L > max_pages * kBk) ? -1 : (L - 1) / kBk;  // valid ids: 0..lim
    bool valid = false;
    float li = -INFINITY;
    if (lane < k) {
      const int b = ids[((size_t)s * H_kv + h / G) * k + lane];
      const float l_raw = part_lse[(size_t)w * k + lane];
      valid = b >= 0 && b <= lim;
      li = valid ? l_raw : -INFINITY;
    }
    float M = li;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kAll, M, off));
    const float wgt = valid ? __expf(li - M) : 0.f;
    float Lsum = wgt;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) Lsum += __shfl_xor_sync(kAll, Lsum, off);
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
#pragma unroll
    for (int sl = 0; sl < kMaxK; ++sl) {
      const float ws = __shfl_sync(kAll, wgt, sl);
      if (sl < k && ws != 0.f) {
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = fmaf(ws, x[sl][i], acc[i]);
      }
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    uint16_t o16[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const __nv_bfloat16 bv = __float2bfloat16_rn(acc[i] * inv);
      o16[i] = *reinterpret_cast<const uint16_t*>(&bv);
    }
    uint16_t* op = out + (size_t)w * D + lane * PER;
    if constexpr (PER == 4) {
      *reinterpret_cast<uint2*>(op) = make_uint2(o16[0] | ((uint32_t)o16[1] << 16),
                                                 o16[2] | ((uint32_t)o16[3] << 16));
    } else {
      *reinterpret_cast<uint32_t*>(op) = o16[0] | ((uint32_t)o16[1] << 16);
    }
    if (lse && lane == 0) lse[w] = M + logf(Lsum);
  }
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// K or V pages [P, H_kv, 128, d] (bf16 or E4M3 bytes) seen as (columns, 128
// rows, block z = page * H_kv + head) with a box of one block's 128 rows by
// 128 bytes, 128-byte swizzle. The page count is not passed in; 2^25 blocks
// bound any pool that fits in device memory (a block is at least 8 KB), and a
// block past the bound would read as zeros instead of faulting.
bool make_map_dec_pages(CUtensorMap* m, const void* base, int D, bool fp8, int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess || qr != cudaDriverEntryPointSuccess)
      return false;
    fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  const int eb = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)kBk, (cuuint64_t)1 << 25};
  cuuint64_t strides[2] = {(cuuint64_t)D * eb, (cuuint64_t)kBk * D * eb};
  cuuint32_t box[3] = {(cuuint32_t)(128 / eb), (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_decode_index(const void* q_idx, const void* k_idx_pages,
                                const int32_t* page_table, const int32_t* seq_lens, int B,
                                int max_pages, int n_g, int d_idx, float* scores,
                                const Diag& dg, cudaStream_t st, bool e4m3, float score_scale,
                                int64_t ss) {
  if (ss <= 0) ss = max_pages;
  int64_t warps = (int64_t)B * max_pages;
  if (warps == 0) return cudaSuccess;
  note_launches(1);
  unsigned grid = (unsigned)std::min<int64_t>((warps + 7) / 8, 152 * 32);
  auto q = (const unsigned char*)q_idx;
  auto kp = (const unsigned char*)k_idx_pages;
#define MSA_DEC_INDEX(DI, F8)                                                                 \
  decode_index_kernel<DI, F8><<<grid, 256, 0, st>>>(q, kp, page_table, seq_lens, B, max_pages, \
                                                    n_g, score_scale, scores, ss, dg)
  if (e4m3) {
    if (d_idx == 128) MSA_DEC_INDEX(128, true);
    else MSA_DEC_INDEX(64, true);
  } else {
    if (d_idx == 128) MSA_DEC_INDEX(128, false);
    else MSA_DEC_INDEX(64, false);
  }
#undef MSA_DEC_INDEX
  return cudaGetLastError();
}

cudaError_t launch_decode_index_fp4(const void* q_idx, const void* codes, const void* kscales,
                                    const int32_t* page_table, const int32_t* seq_lens, int B,
                                    int max_pages, int n_g, int d_idx, float score_scale,
                                    float* scores, const Diag& dg, cudaStream_t st, int64_t ss) {
  if (ss <= 0) ss = max_pages;
  const int64_t tasks = (int64_t)B * max_pages;
  if (tasks == 0) return cudaSuccess;
  note_launches(1);
  const unsigned grid =
      (unsigned)std::min<int64_t>((tasks + kFp4Warps - 1) / kFp4Warps, 152 * 32);
  const int smem = kFp4Warps * kBk * (d_idx / 2 + d_idx / 16);
  auto q = (const uint16_t*)q_idx;
  auto c = (const unsigned char*)codes;
  auto sc = (const unsigned char*)kscales;
  cudaError_t e;
  if (d_idx == 128) {
    e = cudaFuncSetAttribute(decode_index_fp4_kernel<128>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    decode_index_fp4_kernel<128><<<grid, kFp4Warps * 32, smem, st>>>(
        q, c, sc, page_table, seq_lens, B, max_pages, n_g, score_scale, scores, ss, dg);
  } else {
    e = cudaFuncSetAttribute(decode_index_fp4_kernel<64>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    decode_index_fp4_kernel<64><<<grid, kFp4Warps * 32, smem, st>>>(
        q, c, sc, page_table, seq_lens, B, max_pages, n_g, score_scale, scores, ss, dg);
  }
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
  cudaError_t e = cudaSuccess;
#define MSA_DEC(DD, F8)                                                                    \
  do {                                                                                     \
    constexpr int sm = dec_smem_bytes<DD, F8>();                                           \
    CUtensorMap tk{}, tv{}, tk16{}, tv16{};                                                \
    if (dec_tma<DD, F8>() &&                                                               \
        (!make_map_dec_pages(&tk, k_pages, DD, F8, kBk) ||                                 \
         !make_map_dec_pages(&tv, v_pages, DD, F8, kBk) ||                                 \
         !make_map_dec_pages(&tk16, k_pages, DD, F8, 16) ||                                \
         !make_map_dec_pages(&tv16, v_pages, DD, F8, 16)))                                 \
      return cudaErrorInvalidValue;                                                        \
    e = cudaFuncSetAttribute(decode_attn_kernel<DD, F8>,                                   \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, sm);             \
    if (e != cudaSuccess) return e;                                                        \
    decode_attn_kernel<DD, F8><<<tasks, 128, sm, st>>>(                                    \
        tk, tv, tk16, tv16, (const uint16_t*)q, k_pages, v_pages, k_scale, v_scale, page_table, \
        seq_lens,                                                                          \
        ids, max_pages, H_q, H_kv, k, sl2, part_o, part_lse, dg);                          \
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

cudaError_t launch_decode_attn_fp4(const void* q, const void* k_codes, const void* k_scales,
                                   const void* v_codes, const void* v_scales,
                                   const int32_t* page_table, const int32_t* seq_lens,
                                   const int32_t* ids, int B, int max_pages, int H_q, int H_kv,
                                   int d, int k, float scale, void* out, float* lse, void* ws,
                                   const Diag& dg, cudaStream_t st) {
  float* part_o = (float*)ws;
  float* part_lse = (float*)((unsigned char*)ws + align256((size_t)B * H_q * k * d * 4));
  const float sl2 = scale * 1.4426950408889634f;
  const unsigned tasks = (unsigned)((int64_t)B * H_kv * k);
  if (tasks == 0) return cudaSuccess;
  note_launches(2);  // attention, merge
  cudaError_t e = cudaSuccess;
#define MSA_DEC_FP4(DD)                                                                       \
  do {                                                                                        \
    constexpr int sm = dec_fp4_smem_bytes<DD>();                                              \
    e = cudaFuncSetAttribute(decode_attn_fp4_kernel<DD>,                                      \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, sm);                \
    if (e != cudaSuccess) return e;                                                           \
    decode_attn_fp4_kernel<DD><<<tasks, 128, sm, st>>>(                                       \
        (const uint16_t*)q, (const uint8_t*)k_codes, (const uint8_t*)k_scales,                \
        (const uint8_t*)v_codes, (const uint8_t*)v_scales, page_table, seq_lens, ids,         \
        max_pages, H_q, H_kv, k, sl2, part_o, part_lse, dg);                                  \
  } while (0)
  if (d == 128) MSA_DEC_FP4(128);
  else MSA_DEC_FP4(64);
#undef MSA_DEC_FP4
  const int64_t nw = (int64_t)B * H_q;
  const unsigned mg = (unsigned)std::min<int64_t>((nw * 32 + 255) / 256, 152 * 32);
  if (d == 128)
    decode_merge_kernel<128><<<mg, 256, 0, st>>>(part_o, part_lse, ids, seq_lens, max_pages, B,
                                                 H_q, H_kv, k, (uint16_t*)out, lse);
  else
    decode_merge_kernel<64><<<mg, 256, 0, st>>>(part_o, part_lse, ids, seq_lens, max_pages, B,
                                                H_q, H_kv, k, (uint16_t*)out, lse);
  return cudaGetLastError();
}

}  // namespace msa
