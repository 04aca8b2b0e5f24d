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
// against up to 128 / G of its queries, all G heads of each, 128 rows in all,
// query-major (row r = query r / G, head r % G). Per tile the tensor cores
// compute S = Q K^T and the index scores X = Q_idx K_idx^T into one of two
// TMEM stages (256 columns each), the A operand of X holding each query's q_idx
// row G times, so a row's teacher logit and index score for the same key sit
// in the same TMEM lane. One persistent CTA per SM, 12 warps:
//   warp 0      per block (bucket): K (head g) and k_idx rows by TMA, once the
//               bucket's last MMAs have completed; per tile the S and X MMAs
//               into the tile's stage once the KL warps two tiles back have
//               read it and the tile's query operands have landed;
//   warp 1      TMEM owner;
//   warps 2, 3  query producers, one per stage (alternate tiles): the G head
//               rows of each query by TMA row gathers (tile::gather4), and each
//               query's q_idx row, loaded by one lane (ahead of the stage's
//               release when it fits in registers) and stored G times into the
//               128B-swizzled operand layout;
//   warps 4-11  two KL groups of four warps, one per TMEM stage, one row per
//               thread. Per 32-key chunk a row turns its logits into teacher
//               probabilities exp2(s c - lse_h); a shuffle reduce-scatter over
//               the G lanes of a query sums the heads and leaves each lane 32/G
//               keys, for which it adds, against its running index max m,
//               l = sum exp(x - m), D = sum p (x - m), C = sum p and
//               A = sum p log p. The G lanes then combine their sums into the
//               tile's 32-byte record of the query.
// The merge pass forms, per (t, g), LSE from the blocks' (m, l) and
//   KL = sum A - sum D - sum C (m - LSE),
// in which every term stays of the size of a log-probability (the raw index
// scores themselves never enter a difference of large numbers).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "msa_kernels.h"
#include "msa_sm100.cuh"

namespace msa {
namespace {

using namespace sm100;

constexpr int kKlRows = 128;   // score rows per tile
constexpr int kKlKeys = 128;   // keys per block
constexpr int kRecFloats = 8;  // {A, D, C, m, l, pad x 3}
constexpr int kKlThreads = 384;  // 12 warps
constexpr int kKlQStages = 2;
constexpr int kKlProducers = kKlQStages;  // warps 2, 3: one per stage

template <int D, int DI>
struct KlSmem {
  static constexpr int kKBytes = kKlKeys * D * 2;
  static constexpr int kIBytes = kKlKeys * DI * 2;
  static constexpr int kQBytes = kKlRows * D * 2;
  static constexpr int kXBytes = kKlRows * DI * 2;
  static constexpr int kKOff = 0;
  static constexpr int kIOff = kKBytes;
  static constexpr int kQOff = kIOff + kIBytes;                    // Q stages
  static constexpr int kXOff = kQOff + kKlQStages * kQBytes;       // q_idx stages
  static constexpr int kBarOff = kXOff + kKlQStages * kXBytes;
  // k_full, k_empty, q_full[2], q_empty[2], s_full[2], t_empty[2], done
  static constexpr int kNumBars = 2 + 4 * kKlQStages + 1;
  static constexpr int kBytes = kBarOff + kNumBars * 8 + 32;
};
static_assert(KlSmem<128, 128>::kBytes <= 232448, "KL tile exceeds shared memory");

// running (m, l, D, C) of one lane: fold in a new max
__device__ __forceinline__ void rebase(float& m, float& l, float& D, float C, float m_new) {
  if (m_new > m) {
    if (C > 0.f) D -= C * (m_new - m);
    l *= ex2_approx((m - m_new) * 1.4426950408889634f);
    m = m_new;
  }
}

// byte offset of 16-byte chunk c (of DI * 2 / 16) of operand row r in the
// 128B-swizzled K-major layout: 128-byte column chunks of 128 rows each,
// 8-row atoms of 1024 bytes, chunks XOR-ed with the row within the atom
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  const int kc = c >> 3, s = c & 7;
  return (uint32_t)(kc * kKlRows * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((s ^ (r & 7)) << 4));
}

template <int D, int DI, int G>
__global__ void __launch_bounds__(kKlThreads, 1)
kl_tile_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_i,
                  const __grid_constant__ CUtensorMap tm_q, int64_t q_rows,
                  const uint16_t* __restrict__ q_idx, const float* __restrict__ lse, int64_t q0,
                  int H_q, int H_kv, float scale_log2, const int32_t* __restrict__ entries,
                  const int4* __restrict__ tinfo, const int32_t* __restrict__ n_tiles,
                  float* __restrict__ part, Diag dg) {
  using L = KlSmem<D, DI>;
  constexpr int QT = kKlRows / G;  // queries per tile
  constexpr int QS = kKlQStages;
  extern __shared__ __align__(1024) unsigned char smem[];
  if (smem_u32(smem) & 1023) {
    if (threadIdx.x == 0) report(dg, kStatusUnsupported);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* k_full = bars + 0;
  uint64_t* k_empty = bars + 1;
  uint64_t* q_full = bars + 2;
  uint64_t* q_empty = q_full + QS;
  uint64_t* s_full = q_empty + QS;
  uint64_t* t_empty = s_full + 2;
  uint64_t* done_bar = t_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + L::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    for (int s = 0; s < QS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&t_empty[s], 4);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_i);
    prefetch_tmap(&tm_q);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int64_t total = *n_tiles;
  const int t_begin = (int)(total * blockIdx.x / gridDim.x);
  const int t_end = (int)(total * (blockIdx.x + 1) / gridDim.x);
  const int n_local = t_end - t_begin;
  const int4 kNone = make_int4(0, 0, 0, 0);

  if (warp == 0) {
    // ------------------------------------------- K + k_idx per block; S and X MMAs
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kKlKeys);
      const uint32_t k_base = smem_u32(smem + L::kKOff), i_base = smem_u32(smem + L::kIOff);
      uint32_t epoch = 0;
      int last = -1;
      int4 inf = tinfo[t_begin];
      bool ok = true;
      for (int j = 0; j < n_local && ok; ++j) {
        if (j > last) {
          last = min(inf.w - t_begin, n_local) - 1;
          const int4 nxt = last + 1 < n_local ? tinfo[t_begin + last + 1] : kNone;
          if (!mbar_wait(k_empty, (epoch & 1) ^ 1, abort_flag, dg)) { ok = false; break; }
          mbar_arrive_expect_tx(k_full, L::kKBytes + L::kIBytes);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + L::kKOff + c * kKlKeys * 128, &tm_k, k_full, c * 64, inf.z >> 8,
                        inf.x);
          for (int c = 0; c < DI / 64; ++c)
            tma_load_2d(smem + L::kIOff + c * kKlKeys * 128, &tm_i, k_full, c * 64, inf.x);
          ++epoch;
          inf = nxt;
          if (!mbar_wait(k_full, (epoch - 1) & 1, abort_flag, dg)) { ok = false; break; }
        }
        const int st = j & 1, qs = j % QS;
        if ((j >= 2 && !mbar_wait(&t_empty[st], (uint32_t)(((j - 2) >> 1) & 1), abort_flag, dg)) ||
            !mbar_wait(&q_full[qs], (uint32_t)((j / QS) & 1), abort_flag, dg)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_s = tmem_base + (uint32_t)(st * 256);
        const uint32_t qa = smem_u32(smem + L::kQOff + qs * L::kQBytes);
        const uint32_t xa = smem_u32(smem + L::kXOff + qs * L::kXBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = kk / 4, off = (kk % 4) * 32;
          mma_bf16_ss(d_s, desc_kmajor_sw128(qa + c * kKlRows * 128 + off),
                      desc_kmajor_sw128(k_base + c * kKlKeys * 128 + off), idesc, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < DI / 16; ++kk) {
          const int c = kk / 4, off = (kk % 4) * 32;
          mma_bf16_ss(d_s + 128, desc_kmajor_sw128(xa + c * kKlRows * 128 + off),
                      desc_kmajor_sw128(i_base + c * kKlKeys * 128 + off), idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[st]);
        mma_commit(&q_empty[qs]);
        if (j == last) mma_commit(k_empty);
      }
      if (*abort_flag && epoch > 0) mbar_drain(k_full, (epoch - 1) & 1);
      mma_commit(done_bar);
      mbar_drain(done_bar, 0);
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------- query operands of every other tile
    // Q rows (query-major: row r = query r / G, head r % G) by TMA row gathers;
    // each query's q_idx row loaded by one lane (before the stage is free, when
    // the rows fit in registers) and stored G times
    // one producer per stage, so that a producer is never more than one phase of
    // its stage ahead (a parity wait cannot tell phase k from phase k + 2)
    const int p = warp - 2;
    constexpr int NJ = (QT + 31) / 32;  // queries per lane
    constexpr int NCH = D / 64;
    constexpr bool kEarly = NJ == 1;    // q_idx rows fetched ahead of the stage wait
    const int32_t oob_row = (int32_t)q_rows;  // past the q rows: zero fill
    uint32_t armed = 0, armed_par = 0;
    for (int i = p; i < n_local; i += kKlProducers) {
      const int4 inf = tinfo[t_begin + i];
      const int cnt = inf.z & 0xFF, g = inf.z >> 8;
      int32_t tq[NJ];  // this lane's queries' positions, or -1
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        const int qi = lane + 32 * jj;
        tq[jj] = qi < cnt ? (int32_t)(q0 + (entries[inf.y + qi] >> 4)) : -1;
      }
      uint4 v[kEarly ? DI / 8 : 1];
      if constexpr (kEarly) {
        if (tq[0] >= 0) {
          const uint4* src =
              reinterpret_cast<const uint4*>(q_idx + ((int64_t)tq[0] * H_kv + g) * DI);
#pragma unroll
          for (int c = 0; c < DI / 8; ++c) v[c] = __ldg(src + c);
        }
      }
      const int qs = i % QS;
      const uint32_t par = (uint32_t)((i / QS) & 1);
      int got = 0;
      if (lane == 0) got = mbar_wait(&q_empty[qs], par ^ 1, abort_flag, dg);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      unsigned char* qbuf = smem + L::kQOff + qs * L::kQBytes;
      unsigned char* xbuf = smem + L::kXOff + qs * L::kXBytes;
      // one tiled box per (query, 64-column chunk): a query's G head rows are
      // consecutive in q and in the tile (query-major rows); every lane runs the
      // same number of iterations (the shuffles need it)
      constexpr int kQJobs = QT * NCH;
      for (int jb = 0; jb < (kQJobs + 31) / 32; ++jb) {
        const int job = lane + 32 * jb;
        const int qi = (job / NCH) % QT, c = job % NCH;
        int32_t tv = -1;
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) {
          const int32_t x = __shfl_sync(0xffffffffu, tq[jj], qi & 31);
          if (jj == (qi >> 5)) tv = x;
        }
        const int32_t y = tv >= 0 ? (int32_t)((int64_t)tv * H_q + g * G) : oob_row;
        if (job < kQJobs)
          tma_load_2d(qbuf + c * kKlRows * 128 + qi * G * 128, &tm_q, &q_full[qs], c * 64, y);
      }
      // q_idx rows, G copies each, into the swizzled operand layout
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        const int qi = lane + 32 * jj;
        if (tq[jj] < 0) continue;
        if constexpr (!kEarly) {
          const uint4* src =
              reinterpret_cast<const uint4*>(q_idx + ((int64_t)tq[jj] * H_kv + g) * DI);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const int r = qi * G + h;
#pragma unroll
            for (int c = 0; c < DI / 8; ++c) {
              const uint4 w = __ldg(src + c);
              st_shared_v4(smem_u32(xbuf) + sw128_off(r, c), w.x, w.y, w.z, w.w);
            }
          }
        } else {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const int r = qi * G + h;
#pragma unroll
            for (int c = 0; c < DI / 8; ++c)
              st_shared_v4(smem_u32(xbuf) + sw128_off(r, c), v[c].x, v[c].y, v[c].z, v[c].w);
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&q_full[qs], L::kQBytes);
      armed |= 1u << qs;
      armed_par = (armed_par & ~(1u << qs)) | (par << qs);
      if (*abort_flag) break;
    }
    if (lane == 0 && *abort_flag) {  // let issued gathers land before shared memory goes
#pragma unroll
      for (int s = 0; s < QS; ++s)
        if ((armed >> s) & 1) mbar_drain(&q_full[s], (armed_par >> s) & 1);
    }
  } else if (warp >= 4) {
    // ------------------------------------------- KL rows
    const int wg = (warp - 4) >> 2;  // stage of this group: tiles i with i % 2 == wg
    const int qq = warp & 3;
    const int row = qq * 32 + lane;
    const int qi = row / G, hi = row % G;
    const uint32_t ts = tmem_base + ((uint32_t)(qq * 32) << 16) + (uint32_t)(wg * 256);
    const float l2e = 1.4426950408889634f;
    for (int i = wg; i < n_local; i += 2) {
      const int4 inf = tinfo[t_begin + i];
      const int cnt = inf.z & 0xFF, g = inf.z >> 8;
      const bool valid = qi < cnt;
      const int64_t t = valid ? q0 + (entries[inf.y + qi] >> 4) : 0;
      // keys of the block visible to this row: all, or up to t in the local block
      const int64_t vis = t - inf.x + 1;
      const int lim = valid ? (int)(vis < kKlKeys ? vis : kKlKeys) : 0;
      const float lse2 = valid ? lse[t * H_q + g * G + hi] * l2e : 0.f;
      int got = 0;
      if (lane == 0) got = mbar_wait(&s_full[wg], (uint32_t)((i >> 1) & 1), abort_flag, dg);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      tc_fence_after();
      float m = -INFINITY, l = 0.f, Dp = 0.f, C = 0.f, A = 0.f;
      const bool full = __all_sync(0xffffffffu, lim >= kKlKeys);
      // chunk ch + 1's columns load while chunk ch's sums are formed; the
      // stage is released as soon as the last chunk's columns have arrived
      uint32_t sr[32], xr[32];
      tmem_ld32(ts, sr);
      tmem_ld32(ts + 128, xr);
#pragma unroll 1
      for (int ch = 0; ch < kKlKeys / 32; ++ch) {
        tmem_ld_wait();
        float pv[32], xv[32];
        if (full) {  // no row of the warp masks a column of this block
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            pv[e] = ex2_approx(__uint_as_float(sr[e]) * scale_log2 - lse2);
            xv[e] = __uint_as_float(xr[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            pv[e] =
                ch * 32 + e < lim ? ex2_approx(__uint_as_float(sr[e]) * scale_log2 - lse2) : 0.f;
            xv[e] = __uint_as_float(xr[e]);
          }
        }
        if (ch + 1 < kKlKeys / 32) {
          tmem_ld32(ts + (ch + 1) * 32, sr);
          tmem_ld32(ts + 128 + (ch + 1) * 32, xr);
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&t_empty[wg]);  // the stage's columns are free again
        }
        // reduce-scatter over the G lanes of the query: after step s a lane
        // keeps the half of its keys that its lane bit s selects
        int col0 = ch * 32;
#pragma unroll
        for (int sh = 16, bit = 1; sh >= 32 / G; sh >>= 1, bit <<= 1) {
          const bool up = (lane & bit) != 0;
#pragma unroll
          for (int e = 0; e < sh; ++e) {
            const float send = up ? pv[e] : pv[e + sh];
            const float keep = up ? pv[e + sh] : pv[e];
            pv[e] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
            xv[e] = up ? xv[e + sh] : xv[e];
          }
          col0 += up ? sh : 0;
        }
        constexpr int OWN = 32 / G;
        float cm = -INFINITY;
#pragma unroll
        for (int e = 0; e < OWN; ++e)
          if (full || col0 + e < lim) cm = fmaxf(cm, xv[e]);
        rebase(m, l, Dp, C, cm);
#pragma unroll
        for (int e = 0; e < OWN; ++e) {
          if (full || col0 + e < lim) {
            const float pp = pv[e] * (1.f / G);
            const float dx = xv[e] - m;
            l += ex2_approx(dx * l2e);
            Dp += pp * dx;
            C += pp;
            if (pp > 0.f) A += pp * __logf(pp);
          }
        }
      }
      // combine the G lanes of the query
#pragma unroll
      for (int off = 1; off < G; off <<= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
        const float D2 = __shfl_xor_sync(0xffffffffu, Dp, off);
        const float C2 = __shfl_xor_sync(0xffffffffu, C, off);
        const float A2 = __shfl_xor_sync(0xffffffffu, A, off);
        const float M = fmaxf(m, m2);
        float lm = 0.f, Dm = 0.f;
        if (M > -INFINITY) {
          lm = l * ex2_approx((m - M) * l2e) + l2 * ex2_approx((m2 - M) * l2e);
          Dm = (C > 0.f ? Dp + C * (m - M) : 0.f) + (C2 > 0.f ? D2 + C2 * (m2 - M) : 0.f);
        }
        m = M;
        l = lm;
        Dp = Dm;
        C += C2;
        A += A2;
      }
      if (hi == 0 && valid) {
        float* rec = part + ((size_t)(t_begin + i) * QT + qi) * kRecFloats;
        *reinterpret_cast<float4*>(rec) = make_float4(A, Dp, C, m);
        rec[4] = l;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
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

PFN_cuTensorMapEncodeTiled_v12000 kl_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

// bf16 tensor of the given dims (innermost first) and row strides in bytes, box
// {64, box1[, box2]}, 128B swizzle; out-of-range elements read as zeros
bool kl_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = kl_encode_fn();
  if (!fn) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int DI, int G>
cudaError_t launch_kl_tiles(const void* q, const void* kk, const void* q_idx, const void* k_idx,
                            const float* lse, int64_t N, int64_t q0, int H_q, int H_kv,
                            float scale, const AttnWs& ws, int64_t n_b, const Diag& dg,
                            cudaStream_t st) {
  CUtensorMap tk, ti, tq;
  const cuuint64_t kd[3] = {(cuuint64_t)D, (cuuint64_t)H_kv, (cuuint64_t)N};
  const cuuint64_t ks[2] = {(cuuint64_t)D * 2, (cuuint64_t)H_kv * D * 2};
  const cuuint32_t kb[3] = {64, 1, (cuuint32_t)kKlKeys};
  const cuuint64_t id[2] = {(cuuint64_t)DI, (cuuint64_t)N};
  const cuuint64_t is[1] = {(cuuint64_t)DI * 2};
  const cuuint32_t ib[2] = {64, (cuuint32_t)kKlKeys};
  const cuuint64_t qd[2] = {(cuuint64_t)D, (cuuint64_t)(N * H_q)};
  const cuuint64_t qs[1] = {(cuuint64_t)D * 2};
  const cuuint32_t qb[2] = {64, (cuuint32_t)G};  // a query's G head rows
  if (!kl_map(&tk, kk, 3, kd, ks, kb) || !kl_map(&ti, k_idx, 2, id, is, ib) ||
      !kl_map(&tq, q, 2, qd, qs, qb))
    return cudaErrorInvalidValue;
  const int smem = KlSmem<D, DI>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(kl_tile_tc_kernel<D, DI, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kl_tile_tc_kernel<D, DI, G><<<kl_sm_count(), kKlThreads, smem, st>>>(
      tk, ti, tq, N * H_q, (const uint16_t*)q_idx, lse, q0, H_q, H_kv,
      scale * 1.4426950408889634f, ws.entries, ws.tinfo, ws.tile_off + n_b, (float*)ws.part, dg);
  return cudaGetLastError();
}

template <int D, int DI>
cudaError_t kl_tiles_g(int G, const void* q, const void* kk, const void* q_idx,
                       const void* k_idx, const float* lse, int64_t N, int64_t q0, int H_q,
                       int H_kv, float scale, const AttnWs& ws, int64_t n_b, const Diag& dg,
                       cudaStream_t st) {
  switch (G) {
    case 1: return launch_kl_tiles<D, DI, 1>(q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, dg, st);
    case 2: return launch_kl_tiles<D, DI, 2>(q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, dg, st);
    case 4: return launch_kl_tiles<D, DI, 4>(q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, dg, st);
    case 8: return launch_kl_tiles<D, DI, 8>(q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, dg, st);
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
    e = d_idx == 128 ? kl_tiles_g<128, 128>(G, q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, dg, st)
                     : kl_tiles_g<128, 64>(G, q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, dg, st);
  else
    e = d_idx == 128 ? kl_tiles_g<64, 128>(G, q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, dg, st)
                     : kl_tiles_g<64, 64>(G, q, kk, q_idx, k_idx, lse, N, q0, H_q, H_kv, scale, ws, n_b, dg, st);
  if (e != cudaSuccess) return e;
  const int64_t n = (q1 - q0) * H_kv;
  kl_merge_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 152 * 32), 256, 0, st>>>(
      (const float*)ws.part, ws.rec_of, q0, q1, H_kv, k, kl);
  return cudaGetLastError();
}

}  // namespace msa
