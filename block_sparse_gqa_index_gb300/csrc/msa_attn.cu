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
#include <cuda.h>
#include <cudaTypedefs.h>

#include "msa_kernels.h"
#include "msa_sm100.cuh"

namespace msa {
namespace {

constexpr int kBk = 128;
constexpr int kTileRows = 128;
constexpr int kThreads = 256;  // bucketing kernels

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

// ------------------------------------------------------- tile kernel (tcgen05)
// One persistent CTA per SM walks a contiguous range of tiles (consecutive
// tiles mostly share a bucket, so K / V of the bucket's block are loaded once):
//   warp 0     TMA: K and V of the bucket's block (128 keys, head g) when the
//              bucket changes (single buffer, released after the bucket's
//              last P.V MMA);
//   warp 1     TMEM owner and MMA issuer: S = Q K^T (128 x 128, A = Q tile,
//              B = K block, both K-major 128B-swizzled in shared memory), then,
//              once softmax wrote P, O = P V (A = P read from TMEM, B = V as an
//              MN-major operand). Two TMEM stages of 256 columns (S/P | O); the
//              S MMA of tile i+1 is issued before the P.V MMA of tile i;
//   warps 2-5  Q producers, one per Q stage (4 stages): gather the G head rows
//              of each of the tile's queries with 16-byte cp.async into the
//              128B-swizzled layout, record each row's query position and
//              partial slot, then publish the stage;
//   warps 6-9  softmax + epilogue, one score row per thread: masked row max,
//              exp2, row sum, P (bf16) back into TMEM over S; then O / l in
//              bf16 and the row's LSE to the partial buffers.
template <int D>
struct AttnSmem {
  static constexpr int kKVBytes = kBk * D * 2;            // one of K or V
  static constexpr int kQBytes = kTileRows * D * 2;       // one Q stage
  static constexpr int kQStages = 4;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKVBytes;
  static constexpr int kQOff = 2 * kKVBytes;
  static constexpr int kMetaOff = kQOff + kQStages * kQBytes;  // row_t, row_dst per stage
  static constexpr int kBarOff = kMetaOff + kQStages * kTileRows * 8;
  // kv_full, kv_empty, q_full[4], q_empty[4], s_full[2], p_full[2], o_full[2], t_empty[2], done
  static constexpr int kNumBars = 2 + 2 * kQStages + 8 + 1;
  static constexpr int kBytes = kBarOff + kNumBars * 8 + 16;
};

constexpr int kAttnThreads = 448;  // 14 warps

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ int64_t find_bucket(const int32_t* __restrict__ tile_off, int64_t n_b,
                                               int64_t tile) {
  int64_t lo = 0, hi = n_b - 1;
  while (lo < hi) {
    int64_t mid = (lo + hi + 1) >> 1;
    if (tile_off[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_tile_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_q, int64_t tm_rows,
                    int64_t q0, int H_q, int H_kv, int k,
                    float scale_log2, int64_t nb, const int32_t* __restrict__ entries,
                    const int32_t* __restrict__ offsets, const int32_t* __restrict__ tile_off,
                    int64_t n_b, uint16_t* __restrict__ part_o, float* __restrict__ part_lse,
                    Diag dg) {
  using namespace sm100;
  using S = AttnSmem<D>;
  constexpr int QS = S::kQStages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  int32_t* row_t_all = reinterpret_cast<int32_t*>(smem + S::kMetaOff);
  int32_t* row_dst_all = row_t_all + QS * kTileRows;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* kv_full = bars + 0;
  uint64_t* kv_empty = bars + 1;
  uint64_t* q_full = bars + 2;
  uint64_t* q_empty = q_full + QS;
  uint64_t* s_full = q_empty + QS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* t_empty = o_full + 2;
  uint64_t* done_bar = t_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + S::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = H_q / H_kv;
  const int qt = kTileRows / G;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < QS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1 + 4);  // S-MMA commit + the owning softmax group's 4 warps
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4);
      mbar_init(&o_full[s], 1);
      mbar_init(&t_empty[s], 4);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    prefetch_tmap(&tm_q);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // this CTA's contiguous range of tiles
  const int64_t total = tile_off[n_b];
  const int64_t t_begin = total * blockIdx.x / gridDim.x;
  const int64_t t_end = total * (blockIdx.x + 1) / gridDim.x;
  const long long n_local = t_end - t_begin;

  if (warp == 0) {
    // ---------------------------------------------------------- K / V loads
    if (lane == 0 && n_local > 0) {
      int64_t bk = find_bucket(tile_off, n_b, t_begin), prev = -1;
      uint32_t epoch = 0;
      bool ok = true;
      for (int64_t tile = t_begin; tile < t_end && ok; ++tile) {
        while (tile_off[bk + 1] <= tile) ++bk;
        if (bk == prev) continue;
        if (!mbar_wait(kv_empty, (epoch & 1) ^ 1, abort_flag, dg)) { ok = false; break; }
        const int g = (int)(bk / nb);
        const int32_t key0 = (int32_t)((bk % nb) * kBk);
        mbar_arrive_expect_tx(kv_full, 2 * S::kKVBytes);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(smem + S::kKOff + c * kBk * 128, &tm_k, kv_full, c * 64, g, key0);
          tma_load_3d(smem + S::kVOff + c * kBk * 128, &tm_v, kv_full, c * 64, g, key0);
        }
        prev = bk;
        ++epoch;
      }
      if (!ok && epoch > 0) mbar_drain(kv_full, (epoch - 1) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // Event loop: issue S(next) when its TMEM stage, Q stage and K/V are ready,
    // and P.V(pending) when its softmax has written P, whichever comes first.
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kBk);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      const uint32_t k_base = smem_u32(smem + S::kKOff), v_base = smem_u32(smem + S::kVOff);
      const uint32_t q_base = smem_u32(smem + S::kQOff);
      int64_t bk_s = find_bucket(tile_off, n_b, t_begin), bk_o = bk_s, cur = -1;
      uint32_t epoch = 0;
      long long si = 0, oi = 0, idle = 0;
      while (oi < n_local) {
        bool prog = false;
        if (si < n_local) {
          const int64_t tile = t_begin + si;
          while (tile_off[bk_s + 1] <= tile) ++bk_s;
          bool ready = true;
          if (bk_s != cur) {  // new K/V: every P.V of the old block must be issued first
            ready = oi == si && mbar_test(kv_full, epoch & 1);
            if (ready) { cur = bk_s; ++epoch; }
          }
          const int st = (int)(si & 1);
          const int qs = (int)(si % QS);
          if (ready && mbar_test(&t_empty[st], (uint32_t)(((si >> 1) & 1) ^ 1)) &&
              mbar_test(&q_full[qs], (uint32_t)((si / QS) & 1))) {
            tc_fence_after();
            const uint32_t d_s = tmem_base + (uint32_t)(st * 256);
            const uint32_t qa = q_base + qs * S::kQBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const int c = kk / 4, off = (kk % 4) * 32;
              mma_bf16_ss(d_s, desc_kmajor_sw128(qa + c * kTileRows * 128 + off),
                          desc_kmajor_sw128(k_base + c * kBk * 128 + off), idesc_s,
                          kk > 0 ? 1u : 0u);
            }
            mma_commit(&s_full[st]);
            mma_commit(&q_empty[qs]);
            ++si;
            prog = true;
          }
        }
        if (oi < si) {
          const int st = (int)(oi & 1);
          if (mbar_test(&p_full[st], (uint32_t)((oi >> 1) & 1))) {
            tc_fence_after();
            const uint32_t d_o = tmem_base + (uint32_t)(st * 256 + 128);
#pragma unroll
            for (int kk = 0; kk < kBk / 16; ++kk) {
              const uint32_t a_p = tmem_base + (uint32_t)(st * 256 + kk * 8);
              const uint64_t bd = desc_mnmajor_sw128(v_base + kk * 16 * 128, kBk * 128);
              mma_bf16_ts(d_o, a_p, bd, idesc_o, kk > 0 ? 1u : 0u);
            }
            mma_commit(&o_full[st]);
            const int64_t tile = t_begin + oi;
            while (tile_off[bk_o + 1] <= tile) ++bk_o;
            if (oi + 1 == n_local || tile_off[bk_o + 1] <= tile + 1) mma_commit(kv_empty);
            ++oi;
            prog = true;
          }
        }
        if (prog) {
          idle = 0;
        } else {
          if (*abort_flag) break;
          if (++idle > dg.wait_limit) {
            *abort_flag = 1;
            report(dg, kStatusTimeout);
            break;
          }
        }
      }
      mma_commit(done_bar);
      mbar_drain(done_bar, 0);
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------- Q producers
    // Tile rows are head-major: row r holds head i = r / qt of query r % qt, so
    // four consecutive rows are one head of four queries, fetched by one TMA
    // row gather (tile::gather4) per 64-column chunk. Rows past the tile's
    // queries use an out-of-range row and are zero-filled.
    const int my = warp - 2;  // Q stage owned by this warp
    unsigned char* qbuf = smem + S::kQOff + my * S::kQBytes;
    int32_t* row_t = row_t_all + my * kTileRows;
    int32_t* row_dst = row_dst_all + my * kTileRows;
    const int32_t oob_row = (int32_t)(tm_rows);  // first row past q: zero fill
    int64_t bk = n_local > 0 ? find_bucket(tile_off, n_b, t_begin) : 0;
    bool armed = false;
    uint32_t armed_par = 0;
    long long i = 0;
    for (int64_t tile = t_begin; tile < t_end; ++tile, ++i) {
      while (tile_off[bk + 1] <= tile) ++bk;
      if ((int)(i % QS) != my) continue;
      const uint32_t par = (uint32_t)((i / QS) & 1);
      int got = 0;
      if (lane == 0) got = mbar_wait(&q_empty[my], par ^ 1, abort_flag, dg);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      const int g = (int)(bk / nb);
      const int e0 = offsets[bk] + (int)(tile - tile_off[bk]) * qt;
      const int nq = min(qt, offsets[bk + 1] - e0);  // queries in this tile
      // row metadata for the softmax warps (row r: head r / qt, query r % qt)
      for (int r = lane; r < kTileRows; r += 32) {
        const int hi = r / qt, qi = r % qt;
        if (qi < nq) {
          const int ent = entries[e0 + qi];
          const int tl = ent >> 4, slot = ent & 15;
          row_t[r] = (int)(q0 + tl);
          row_dst[r] = (tl * k + slot) * H_q + g * G + hi;
        } else {
          row_t[r] = 0x7FFFFFFF;
          row_dst[r] = -1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&q_full[my], S::kQBytes);
      __syncwarp();
      // one gather4 per (group of 4 rows, 64-column chunk), spread over the lanes
      constexpr int NCH = D / 64;
      for (int job = lane; job < (kTileRows / 4) * NCH; job += 32) {
        const int r0 = (job / NCH) * 4, c = job % NCH;
        int32_t y[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = r0 + u, hi = r / qt, qi = r % qt;
          y[u] = qi < nq ? (int32_t)(((int64_t)row_t[r] * H_q + g * G + hi)) : oob_row;
        }
        tma_gather4(qbuf + c * kTileRows * 128 + r0 * 128, &tm_q, &q_full[my], c * 64, y[0],
                    y[1], y[2], y[3]);
      }
      armed = true;
      armed_par = par;
    }
    if (lane == 0 && armed && *abort_flag) mbar_drain(&q_full[my], armed_par);
  } else {
    // ---------------------------------------------------------- softmax + epilogue
    // two groups of 4 warps; group wg takes the tiles i with i % 2 == wg, which
    // use TMEM stage wg, so one group's softmax overlaps the other's epilogue
    const int wg = (warp - 6) >> 2;
    const int qq = warp & 3;
    const int row = qq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const int st = wg;
    const uint32_t ts = tmem_base + lane_off + (uint32_t)(st * 256);
    int64_t bk = n_local > 0 ? find_bucket(tile_off, n_b, t_begin) : 0;
    for (long long i = wg; i < n_local; i += 2) {
      const int64_t tile = t_begin + i;
      while (tile_off[bk + 1] <= tile) ++bk;
      const int64_t b = bk % nb;
      const uint32_t par = (uint32_t)((i >> 1) & 1);
      const int qs = (int)(i % QS);
      // q_full: acquire the producer's row metadata; s_full: scores are in TMEM
      int got = 0;
      if (lane == 0)
        got = mbar_wait(&q_full[qs], (uint32_t)((i / QS) & 1), abort_flag, dg) &&
              mbar_wait(&s_full[st], par, abort_flag, dg);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      const int64_t t = row_t_all[qs * kTileRows + row];
      const int dst = row_dst_all[qs * kTileRows + row];
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_empty[qs]);
      tc_fence_after();
      const int lim = (dst >= 0 && t / kBk == b) ? (int)(t - b * kBk) + 1 : kBk;
      // pass 1: row max
      float m = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; c += 2) {
        uint32_t r0[32], r1[32];
        tmem_ld32(ts + c * 32, r0);
        tmem_ld32(ts + c * 32 + 32, r1);
        tmem_ld_wait();
        if (lim >= kBk) {
#pragma unroll
          for (int j = 0; j < 32; j += 2)
            m = fmax3(m, fmaxf(__uint_as_float(r0[j]), __uint_as_float(r0[j + 1])),
                      fmaxf(__uint_as_float(r1[j]), __uint_as_float(r1[j + 1])));
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c * 32 + j < lim) m = fmaxf(m, __uint_as_float(r0[j]));
            if (c * 32 + 32 + j < lim) m = fmaxf(m, __uint_as_float(r1[j]));
          }
        }
      }
      const float mc = m * scale_log2;
      // pass 2: P = exp2(s * c - m * c) in bf16 over the first 64 columns, row sum
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32], pk[16];
        tmem_ld32(ts + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float p0 = c * 32 + j < lim ? ex2_approx(fmaf(__uint_as_float(r[j]), scale_log2, -mc)) : 0.f;
          float p1 = c * 32 + j + 1 < lim ? ex2_approx(fmaf(__uint_as_float(r[j + 1]), scale_log2, -mc)) : 0.f;
          l0 += p0;
          l1 += p1;
          pk[j >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st16(ts + c * 16, pk);
      }
      const float l = l0 + l1;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[st]);
      // O epilogue
      got = 0;
      if (lane == 0) got = mbar_wait(&o_full[st], par, abort_flag, dg);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      tc_fence_after();
      const float inv = 1.f / l;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(ts + 128 + c * 32, r);
        tmem_ld_wait();
        if (dst >= 0) {
          uint4* o = reinterpret_cast<uint4*>(part_o + (size_t)dst * D + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv, __uint_as_float(r[8 * v + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv, __uint_as_float(r[8 * v + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv, __uint_as_float(r[8 * v + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv, __uint_as_float(r[8 * v + 7]) * inv);
            __stcs(o + v, w);
          }
        }
      }
      if (dst >= 0) part_lse[dst] = (mc + __log2f(l)) * 0.69314718055994531f;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&t_empty[st]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// ---------------------------------------------------------------------- merge
// partials: part_o [rows, k, H_q, D] bf16, part_lse [rows, k, H_q]. Each half
// warp merges one (query, head): lane s < k holds slot s's LSE, max and sum come
// from shuffles within the half, and the k slot loads (16 bytes per lane for
// D = 128) are all issued before they are summed. The two halves take adjacent
// heads, so each slot read is one contiguous 2 * D * 2-byte run.
template <int D>
__global__ void __launch_bounds__(256)
attn_merge_kernel(const uint16_t* __restrict__ part_o, const float* __restrict__ part_lse,
                  const int32_t* __restrict__ ids, int64_t q0, int64_t q1, int H_q, int H_kv,
                  int k, uint16_t* __restrict__ out, float* __restrict__ lse) {
  constexpr int PER = D / 16;  // elements per lane (8 or 4)
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;          // lane within the half warp
  const int G = H_q / H_kv;
  const int64_t n = (q1 - q0) * H_q;
  const Diag none{nullptr, 0};
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; 2 * w < n; w += warps) {
    const int64_t task = 2 * w + (lane >> 4);
    const bool active = task < n;
    const int64_t tk = active ? task : n - 1;
    const int64_t tl = tk / H_q;
    const int h = (int)(tk % H_q);
    const int64_t t = q0 + tl;
    bool valid = false;
    float ls = -INFINITY;
    if (hl < k) {
      valid = id_ok(ids[((size_t)t * H_kv + h / G) * k + hl], t, none);
      if (valid) ls = part_lse[((size_t)tl * k + hl) * H_q + h];
    }
    float M = ls;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off, 16));
    const float wl = valid ? __expf(ls - M) : 0.f;
    float L = wl;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off, 16);
    const uint16_t* base = part_o + ((size_t)tl * k * H_q + h) * D + hl * PER;
    const size_t slot_stride = (size_t)H_q * D;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= k) break;
      const float wgt = __shfl_sync(0xffffffffu, wl, s, 16);
      if (wgt == 0.f) continue;  // invalid or padded slot
      const uint16_t* po = base + s * slot_stride;
      if (PER == 8) {
        uint4 u = __ldcs(reinterpret_cast<const uint4*>(po));
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = fmaf(wgt, bf16_lo(wd[i]), acc[2 * i]);
          acc[2 * i + 1] = fmaf(wgt, bf16_hi(wd[i]), acc[2 * i + 1]);
        }
      } else {
        uint2 u = __ldcs(reinterpret_cast<const uint2*>(po));
        acc[0] = fmaf(wgt, bf16_lo(u.x), acc[0]);
        acc[1] = fmaf(wgt, bf16_hi(u.x), acc[1]);
        acc[2] = fmaf(wgt, bf16_lo(u.y), acc[2]);
        acc[3] = fmaf(wgt, bf16_hi(u.y), acc[3]);
      }
    }
    if (!active) continue;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t* o = out + ((size_t)t * H_q + h) * D + hl * PER;
    if (PER == 8) {
      uint4 u;
      u.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      u.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      u.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      u.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(o) = u;
    } else {
      uint2 u;
      u.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      u.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(o) = u;
    }
    if (lse && hl == 0) lse[(size_t)t * H_q + h] = M + logf(L);
  }
}

// 3D bf16 tensor [N, H, D] viewed as (D, H, N); box {64, 1, 128}, 128B swizzle
bool make_map_kv(CUtensorMap* m, const void* base, int64_t N, int H, int D) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess || qr != cudaDriverEntryPointSuccess)
      return false;
    fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)N};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kBk};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D bf16 tensor [rows, D] with a one-row box of 64 columns, 128B swizzle (the
// layout tile::gather4 row gathers use)
bool make_map_rows(CUtensorMap* m, const void* base, int64_t rows, int D) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess || qr != cudaDriverEntryPointSuccess)
      return false;
    fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, 1};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int D>
cudaError_t launch_tiles(const void* q, const void* kk, const void* v, int64_t N, int64_t q0,
                         int H_q, int H_kv, int k, float scale_log2, int64_t nb, const AttnWs& ws,
                         int64_t n_b, const Diag& dg, cudaStream_t st) {
  CUtensorMap tk, tv;
  CUtensorMap tq;
  if (!make_map_kv(&tk, kk, N, H_kv, D) || !make_map_kv(&tv, v, N, H_kv, D) ||
      !make_map_rows(&tq, q, N * H_q, D))
    return cudaErrorInvalidValue;
  const int smem = AttnSmem<D>::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_tile_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_tile_tc_kernel<D><<<sm_count(), kAttnThreads, smem, st>>>(
      tk, tv, tq, N * H_q, q0, H_q, H_kv, k, scale_log2, nb, ws.entries, ws.offsets,
      ws.tile_off, n_b, ws.part_o, ws.part_lse, dg);
  return cudaGetLastError();
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
  e = d == 128 ? launch_tiles<128>(q, kk, v, N, q0, H_q, H_kv, k, scale_log2, nb, ws, n_b, dg, st)
               : launch_tiles<64>(q, kk, v, N, q0, H_q, H_kv, k, scale_log2, nb, ws, n_b, dg, st);
  if (e != cudaSuccess) return e;
  int64_t nw = (q1 - q0) * H_q;
  unsigned mg = (unsigned)std::min<int64_t>((nw * 16 + 255) / 256, 152 * 64);
  if (d == 128)
    attn_merge_kernel<128><<<mg, 256, 0, st>>>(ws.part_o, ws.part_lse, ids, q0, q1, H_q, H_kv, k,
                                               (uint16_t*)out, lse);
  else
    attn_merge_kernel<64><<<mg, 256, 0, st>>>(ws.part_o, ws.part_lse, ids, q0, q1, H_q, H_kv, k,
                                              (uint16_t*)out, lse);
  return cudaGetLastError();
}

}  // namespace msa
