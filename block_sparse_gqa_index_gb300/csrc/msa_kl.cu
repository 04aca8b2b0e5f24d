// KL alignment signal of the index branch, forward only.
//
// "MiniMax Sparse Attention (MSA): a Two-Branch Block-Sparse Attention Trained
// on a 109B-Parameter MoE With a 3T-Token Budget", section "MSA 如何训练" (how
// MSA is trained), and "MiniMax lança MSA ...", section "Treinamento com KL
// Divergence": the index branch learns from a KL loss whose teacher is the
// main branch's distribution over the selected tokens, averaged over the
// group's query heads. Per (t, g), with J the causally visible tokens of the
// group's selected blocks:
//   p_main(j) = (1/G) sum_h exp(scale q_h . k_j - lse_h)     (lse_h: main branch)
//   p_idx(j)  = exp(s_j - LSE),  s_j = q_idx[t,g] . k_idx[j], LSE = log sum_J exp(s_j)
//   KL        = sum_J p_main (log p_main - log p_idx).
//
// It runs on the main branch's bucketing: a tile is one (group, block) bucket
// against up to 128 / G of its queries, so the block's K and k_idx rows are
// staged once for all of them. 8 warps; warp w owns score rows 16w .. 16w+15,
// row r = (query r / G, head r % G). S = Q K^T and the index scores
// I = Q_idx K_idx^T run on mma.m16n8k16 with the same row layout: the A
// operand of I repeats each query's q_idx row G times, so a thread finds a
// query's teacher and student values for the same key in the same registers.
// The G rows of a query sit on lanes that differ only in their row bits, and a
// butterfly of shuffles sums the heads. Per (query, block) a thread keeps, over
// its columns, the running index max m, l = sum exp(s - m),
// D = sum p_main (s - m), C = sum p_main and A = sum p_main log p_main; the
// four lanes of a row combine them into the tile's 32-byte partial record.
// The merge pass then forms, per (t, g), LSE from the blocks' (m, l) and
//   KL = sum A - sum D - sum C (m - LSE),
// in which every term stays of the size of a log-probability (the raw index
// scores themselves never enter a difference of large numbers).
#include "msa_kernels.h"

namespace msa {
namespace {

constexpr int kKlThreads = 256;
constexpr int kKlRows = 128;  // score rows per tile
constexpr int kKlKeys = 128;  // keys per block
constexpr int kRecFloats = 8;  // {A, D, C, m, l, pad x 3}

__device__ __forceinline__ uint32_t smem_u32a(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_commit_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}
__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// byte offset of 16-byte chunk c of row r in a tile of ROWB-byte rows, chunks
// XOR-swizzled by (row mod 8) so that ldmatrix row reads hit 8 distinct banks
template <int ROWB>
__device__ __forceinline__ uint32_t swz16(int r, int c) {
  return (uint32_t)(r * ROWB + ((c ^ (r & 7)) << 4));
}

// running (m, l, D, C) of one row: fold in a new max
__device__ __forceinline__ void rebase(float& m, float& l, float& D, float C, float m_new) {
  if (m_new > m) {
    if (C > 0.f) D -= C * (m_new - m);
    l *= ex2_approx((m - m_new) * 1.4426950408889634f);
    m = m_new;
  }
}

template <int D, int DI, int G>
__global__ void __launch_bounds__(kKlThreads, 2)
kl_tile_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ kk,
               const uint16_t* __restrict__ q_idx, const uint16_t* __restrict__ k_idx,
               const float* __restrict__ lse, int64_t N, int64_t q0, int H_q, int H_kv,
               float scale_log2, const int32_t* __restrict__ entries,
               const int4* __restrict__ tinfo, const int32_t* __restrict__ n_tiles,
               float* __restrict__ part) {
  constexpr int QT = kKlRows / G;      // queries per tile
  constexpr int KB = D * 2, IB = DI * 2;  // row bytes of K and k_idx
  extern __shared__ __align__(128) unsigned char kl_smem[];
  unsigned char* sK = kl_smem;
  unsigned char* sI = kl_smem + kKlKeys * KB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;

  const int total = *n_tiles;
  const int t_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int t_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  int bucket_end = -1;
  for (int tile = t_begin; tile < t_end; ++tile) {
    const int4 inf = tinfo[tile];
    const int kv_row = inf.x, e0 = inf.y, cnt = inf.z & 0xFF, g = inf.z >> 8;
    if (tile >= bucket_end) {  // a new block: stage its K (head g) and k_idx rows
      bucket_end = inf.w;
      __syncthreads();          // every warp is done with the previous block
      for (int x = tid; x < kKlKeys * (KB / 16); x += kKlThreads) {
        const int r = x / (KB / 16), c = x % (KB / 16);
        const int64_t row = (int64_t)kv_row + r;
        const bool ok = row < N;
        cp16(smem_u32a(sK + swz16<KB>(r, c)),
             ok ? (const void*)(kk + (row * H_kv + g) * D + c * 8) : (const void*)kk, ok ? 16 : 0);
      }
      for (int x = tid; x < kKlKeys * (IB / 16); x += kKlThreads) {
        const int r = x / (IB / 16), c = x % (IB / 16);
        const int64_t row = (int64_t)kv_row + r;
        const bool ok = row < N;
        cp16(smem_u32a(sI + swz16<IB>(r, c)),
             ok ? (const void*)(k_idx + row * DI + c * 8) : (const void*)k_idx, ok ? 16 : 0);
      }
    }
    // this thread's two score rows: r = 16 warp + gid (+ 8)
    int64_t t[2];
    bool valid[2];
    float lse2[2];
    uint32_t aq[D / 16][4], ai[DI / 16][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = warp * 16 + gid + 8 * j;
      const int qi = r / G, h = r % G;
      valid[j] = qi < cnt;
      t[j] = valid[j] ? q0 + (entries[e0 + qi] >> 4) : 0;
      lse2[j] = valid[j] ? lse[t[j] * H_q + g * G + h] * 1.4426950408889634f : 0.f;
      const uint16_t* qr = q + (t[j] * H_q + g * G + h) * D;
      const uint16_t* ir = q_idx + (t[j] * H_kv + g) * DI;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        aq[ks][j] = valid[j] ? __ldg(reinterpret_cast<const uint32_t*>(qr + ks * 16 + tig * 2)) : 0u;
        aq[ks][2 + j] =
            valid[j] ? __ldg(reinterpret_cast<const uint32_t*>(qr + ks * 16 + 8 + tig * 2)) : 0u;
      }
#pragma unroll
      for (int ks = 0; ks < DI / 16; ++ks) {
        ai[ks][j] = valid[j] ? __ldg(reinterpret_cast<const uint32_t*>(ir + ks * 16 + tig * 2)) : 0u;
        ai[ks][2 + j] =
            valid[j] ? __ldg(reinterpret_cast<const uint32_t*>(ir + ks * 16 + 8 + tig * 2)) : 0u;
      }
    }
    cp_commit_wait_all();
    __syncthreads();  // the block's rows are in shared memory

    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f}, Dp[2] = {0.f, 0.f},
          C[2] = {0.f, 0.f}, A[2] = {0.f, 0.f};
    const uint32_t kbase = smem_u32a(sK), ibase = smem_u32a(sI);
    // ldmatrix x4 lane roles: matrix lane / 8 -> (key half, k half)
    const int lrow = (lane & 7) + ((lane >> 4) << 3), lk = (lane >> 3) & 1;
#pragma unroll 1
    for (int c = 0; c < kKlKeys / 32; ++c) {
      // index scores first: the chunk's index max rebases the running sums
      float iv[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) iv[nt][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < DI / 16; ++ks)
#pragma unroll
        for (int np = 0; np < 2; ++np) {  // key tiles 2np, 2np + 1
          uint32_t b[4];
          ldsm4(ibase + swz16<IB>(c * 32 + np * 16 + lrow, ks * 2 + lk), b);
          mma16816(iv[2 * np], ai[ks], b[0], b[1]);
          mma16816(iv[2 * np + 1], ai[ks], b[2], b[3]);
        }
      const int col0 = c * 32 + tig * 2;  // column of element (nt, e) = col0 + 8 nt + (e & 1)
      float cm[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = e >> 1;
          if (valid[j] && (int64_t)kv_row + col0 + nt * 8 + (e & 1) <= t[j])
            cm[j] = fmaxf(cm[j], iv[nt][e]);
        }
#pragma unroll
      for (int j = 0; j < 2; ++j) rebase(m[j], l[j], Dp[j], C[j], cm[j]);
      float s[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t b[4];
          ldsm4(kbase + swz16<KB>(c * 32 + np * 16 + lrow, ks * 2 + lk), b);
          mma16816(s[2 * np], aq[ks], b[0], b[1]);
          mma16816(s[2 * np + 1], aq[ks], b[2], b[3]);
        }
      // teacher probability of each element, summed over the query's G head
      // rows; the student's terms for the same key sit in iv
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = e >> 1;
          const bool v = valid[j] && (int64_t)kv_row + col0 + nt * 8 + (e & 1) <= t[j];
          float p = v ? ex2_approx(s[nt][e] * scale_log2 - lse2[j]) : 0.f;
#pragma unroll
          for (int off = 4; off < 4 * G; off <<= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
          p *= 1.f / G;
          if (v) {
            const float x = iv[nt][e];
            l[j] += ex2_approx((x - m[j]) * 1.4426950408889634f);
            Dp[j] += p * (x - m[j]);
            C[j] += p;
            if (p > 0.f) A[j] += p * __logf(p);
          }
        }
    }
    // combine the four lanes of each row, then the row's first lane writes
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m[j], off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l[j], off);
        const float D2 = __shfl_xor_sync(0xffffffffu, Dp[j], off);
        const float C2 = __shfl_xor_sync(0xffffffffu, C[j], off);
        const float A2 = __shfl_xor_sync(0xffffffffu, A[j], off);
        const float M = fmaxf(m[j], m2);
        float lm = 0.f, Dm = 0.f;
        if (M > -INFINITY) {
          lm = l[j] * ex2_approx((m[j] - M) * 1.4426950408889634f) +
               l2 * ex2_approx((m2 - M) * 1.4426950408889634f);
          Dm = (C[j] > 0.f ? Dp[j] + C[j] * (m[j] - M) : 0.f) + (C2 > 0.f ? D2 + C2 * (m2 - M) : 0.f);
        }
        m[j] = M;
        l[j] = lm;
        Dp[j] = Dm;
        C[j] += C2;
        A[j] += A2;
      }
      const int r = warp * 16 + gid + 8 * j;
      if (tig == 0 && r % G == 0 && valid[j]) {
        float* rec = part + ((size_t)tile * QT + r / G) * kRecFloats;
        *reinterpret_cast<float4*>(rec) = make_float4(A[j], Dp[j], C[j], m[j]);
        rec[4] = l[j];
      }
    }
  }
}

// one thread per (query, group): combine the k partial records
__global__ void kl_merge_kernel(const float* __restrict__ part, const int32_t* __restrict__ rec_of,
                                int64_t q0, int64_t q1, int n_g, int k, float* __restrict__ kl) {
  const int64_t n = (q1 - q0) * n_g;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < n;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int32_t* ro = rec_of + x * k;
    float M = -INFINITY;
    for (int s = 0; s < k; ++s)
      if (ro[s] >= 0) M = fmaxf(M, part[(size_t)ro[s] * kRecFloats + 3]);
    float L = 0.f, A = 0.f, Dsum = 0.f;
    for (int s = 0; s < k; ++s) {
      if (ro[s] < 0) continue;
      const float* rec = part + (size_t)ro[s] * kRecFloats;
      L += rec[4] * __expf(rec[3] - M);
    }
    const float LSE = M + __logf(L);
    for (int s = 0; s < k; ++s) {
      if (ro[s] < 0) continue;
      const float4 r = *reinterpret_cast<const float4*>(part + (size_t)ro[s] * kRecFloats);
      A += r.x;
      Dsum += r.y + r.z * (r.w - LSE);
    }
    kl[q0 * n_g + x] = M > -INFINITY ? A - Dsum : 0.f;
  }
}

int kl_sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int D, int DI, int G>
cudaError_t launch_kl_tiles(const void* q, const void* kk, const void* q_idx, const void* k_idx,
                            const float* lse, int64_t N, int64_t q0, int H_q, int H_kv,
                            float scale, const AttnWs& ws, int64_t n_b, cudaStream_t st) {
  const int smem = kKlKeys * (D + DI) * 2;
  cudaError_t e = cudaFuncSetAttribute(kl_tile_kernel<D, DI, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kl_tile_kernel<D, DI, G><<<kl_sm_count() * 2, kKlThreads, smem, st>>>(
      (const uint16_t*)q, (const uint16_t*)kk, (const uint16_t*)q_idx, (const uint16_t*)k_idx,
      lse, N, q0, H_q, H_kv, scale * 1.4426950408889634f, ws.entries, ws.tinfo,
      ws.tile_off + n_b, (float*)ws.part);
  return cudaGetLastError();
}

template <int D, int DI>
cudaError_t kl_tiles_g(int G, const void* q, const void* kk, const void* q_idx,
                       const void* k_idx, const float* lse, int64_t N, int64_t q0, int H_q,
                       int H_kv, float scale, const AttnWs& ws, int64_t n_b, cudaStream_t st) {
  switch (G) {
    case 1: return launch_kl_tiles<D, DI, 1>(q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, st);
    case 2: return launch_kl_tiles<D, DI, 2>(q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, st);
    case 4: return launch_kl_tiles<D, DI, 4>(q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, st);
    case 8: return launch_kl_tiles<D, DI, 8>(q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_kl_chunk(const void* q, const void* kk, const void* q_idx, const void* k_idx,
                            const int32_t* ids, const float* lse, int64_t N, int64_t q0,
                            int64_t q1, int H_q, int H_kv, int d, int d_idx, int k, float scale,
                            float* kl, const AttnWs& ws, int64_t nb, const Diag& dg,
                            cudaStream_t st) {
  cudaError_t e = launch_bucketing(ids, q0, q1, H_q, H_kv, k, ws, nb, dg, st);
  if (e != cudaSuccess) return e;
  note_launches(2);
  const int G = H_q / H_kv;
  const int64_t n_b = (int64_t)H_kv * nb;
  if (d == 128)
    e = d_idx == 128 ? kl_tiles_g<128, 128>(G, q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, st)
                     : kl_tiles_g<128, 64>(G, q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, st);
  else
    e = d_idx == 128 ? kl_tiles_g<64, 128>(G, q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, st)
                     : kl_tiles_g<64, 64>(G, q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, st);
  if (e != cudaSuccess) return e;
  const int64_t n = (q1 - q0) * H_kv;
  kl_merge_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 152 * 32), 256, 0, st>>>(
      (const float*)ws.part, ws.rec_of, q0, q1, H_kv, k, kl);
  return cudaGetLastError();
}

}  // namespace msa
