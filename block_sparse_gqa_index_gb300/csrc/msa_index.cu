// Index branch of MSA prefill: scores of every visible key, causal block
// max-pool and top-k with the forced local block, fused so that neither the
// N x N scores nor (unless asked for) the block scores are written.
//
// Follows "MiniMax Sparse Attention (MSA): a Two-Branch Block-Sparse Attention
// Trained on a 109B-Parameter MoE With a 3T-Token Budget", section
// "两个分支如何工作" (how the two branches work): one index-query head per GQA
// group, one shared index-key head, visible keys scored and max-pooled to
// blocks, top-k per (query, group) with the query's own block always kept.
//
// Rows of the score matrix are the flattened (t, g) pairs of q_idx
// [N, n_g, d_idx]; columns are keys. Because the index key head is shared, one
// k_idx block serves every group of a row tile.
//
// GB300 design (one persistent CTA per SM, 11 warps):
//   warp 0      TMA producer: the CTA's 256 q_idx rows once per tile, then
//               k_idx blocks (128 keys x d_idx) through a 4-stage ring;
//   warp 1      TMEM owner and MMA issuer: per key block two 128x128xd_idx
//               tcgen05 MMAs (the two 128-row halves share the k_idx tile, so
//               every k_idx byte fetched from L2 feeds 256 rows) into one of
//               two TMEM accumulator stages (4 x 128 of the 512 columns);
//   warp 10     the second MMA issuer: warps 1 and 10 take alternate key
//               blocks, so the pipe is fed while the other waits;
//   warps 2-9   epilogue: each thread owns one row, reads its 128 scores of the
//               block from TMEM, applies the causal mask on the diagonal block,
//               max-pools them to the block score and feeds it to the row's
//               streaming top-k (RowTopK), overlapping the next block's MMAs.
// Tiles are visited heaviest-first in a boustrophedon order over the CTAs so
// the causal triangle balances; all CTAs sweep k_idx in the same order, which
// keeps the re-read k_idx stream in L2.
//
// One launch serves a packed batch of independent sequences (SeqTable): each
// sequence is cut into its own 256-row tiles, and the tiles of all sequences
// form one heaviest-first schedule. A tile's weight is its local index j (the
// number of key blocks its rows see), so the schedule walks j downwards and,
// at each j, round-robins over the sequences that have a tile j. A single
// sequence is the one-entry table.
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "msa_kernels.h"
#include "msa_sm100.cuh"

namespace msa {
namespace {

using namespace sm100;

constexpr int kRows = 256;     // rows (t, g) per tile: two M = 128 halves
constexpr int kKeys = 128;     // keys per block (= Bk)
constexpr int kStages = 4;     // k_idx ring depth
constexpr int kThreads = 352;  // 11 warps
constexpr int kIssuer2 = 10;   // the second MMA issuer
constexpr int kEpiWarps = 8;

// DI index dimensions of EB bytes each (bf16: 2, E4M3: 1)
template <int DI, int EB>
struct Smem {
  static constexpr int kChunks = DI * EB / 128;       // 128-byte K chunks
  static constexpr int kAChunk = kRows * 128;         // bytes of one A K-chunk
  static constexpr int kBChunk = kKeys * 128;         // bytes of one B K-chunk
  static constexpr int kABytes = kAChunk * kChunks;
  static constexpr int kBBytes = kBChunk * kChunks;
  static constexpr int kBarOff = kABytes + kStages * kBBytes;
  // barriers: a_full, a_empty, b_full[S], b_empty[S], t_full[2], t_empty[2], done
  static constexpr int kNumBars = 2 + 2 * kStages + 4 + 1;
  static constexpr int kBytes = kBarOff + kNumBars * 8 + 16;
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// max of 32 TMEM columns; columns >= lim are masked (lim >= 32: no mask)
__device__ __forceinline__ float max32(const uint32_t (&r)[32], int lim) {
  float m0 = -INFINITY, m1 = -INFINITY;
  if (lim >= 32) {
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      m0 = fmax3(m0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
      m1 = fmax3(m1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < lim) m0 = fmaxf(m0, __uint_as_float(r[i]));
  }
  return fmaxf(m0, m1);
}

// Sequences of one launch, sorted by tile count (non-increasing). The tile
// levels j in [tiles[s+1], tiles[s]) are shared by the first s+1 sequences;
// their (s+1) * (tiles[s] - tiles[s+1]) schedule ranks end at seg_end[s].
// A sequence's queries are its last len tokens: query i sits at position
// q_off + i and sees the keys at positions 0 .. q_off + i. Keys are packed
// (key position p at k_idx row key0 + p) or paged (at row 128 *
// page_table[pt_row + p / 128] + p % 128).
constexpr int kMaxSeq = 128;
struct SeqTable {
  int B;                     // sequences (1 .. kMaxSeq), none empty
  int n_tiles;               // sum of tiles[]
  int32_t start[kMaxSeq];    // first query row of the sequence (q_idx rows / n_g)
  int32_t len[kMaxSeq];      // queries
  int32_t q_off[kMaxSeq];    // position of the first query
  int32_t key0[kMaxSeq];     // packed: k_idx row of key position 0; paged: pt_row
  int32_t tiles[kMaxSeq];    // 256-row tiles of the sequence's (t, g) rows
  int32_t seg_end[kMaxSeq];  // exclusive end rank of level segment s
};

// one tile of the schedule
struct TileRef {
  int64_t row0;   // first (t, g) row of the tile in the packed batch
  int64_t lrow0;  // the same row counted from the sequence's first row
  int64_t rows;   // (t, g) rows of the sequence
  int64_t key0;   // packed: k_idx row of key position 0; paged: first page-table entry
  int64_t q_off;  // position of the sequence's first query
};

__device__ __forceinline__ bool tile_at(const SeqTable& tb, int i, int n_g, TileRef& tr) {
  if (i >= tb.n_tiles) return false;
  int lo = 0, hi = tb.B - 1;  // first segment whose ranks end after i
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (i < tb.seg_end[mid]) hi = mid;
    else lo = mid + 1;
  }
  const int o = i - (lo ? tb.seg_end[lo - 1] : 0);
  const int p = o % (lo + 1);
  const int j = tb.tiles[lo] - 1 - o / (lo + 1);
  tr.lrow0 = (int64_t)j * kRows;
  tr.row0 = (int64_t)tb.start[p] * n_g + tr.lrow0;
  tr.rows = (int64_t)tb.len[p] * n_g;
  tr.key0 = tb.key0[p];
  tr.q_off = tb.q_off[p];
  return true;
}

// F8: q_idx / k_idx are E4M3 codes (kind::f8f6f4 MMAs, 32 codes per 32-byte
// K step) and score_scale multiplies the reported block scores.
template <int DI, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
index_select_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ SeqTable tab,
                       const int32_t* __restrict__ page_table, int n_g, int k,
                       int32_t* __restrict__ block_ids, float* __restrict__ block_scores,
                       int64_t nb, float score_scale, Diag dg) {
  constexpr int EB = F8 ? 1 : 2;
  constexpr int kColsPerChunk = 128 / EB;  // elements in a 128-byte K chunk
  using S = Smem<DI, EB>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* sA = smem;
  unsigned char* sB = smem + S::kABytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* a_full = bars + 0;
  uint64_t* a_empty = bars + 1;
  uint64_t* b_full = bars + 2;
  uint64_t* b_empty = bars + 2 + kStages;
  uint64_t* t_full = bars + 2 + 2 * kStages;
  uint64_t* t_empty = t_full + 2;
  uint64_t* done_bar = t_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + S::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool want_scores = block_scores != nullptr;

  if (threadIdx.x == 0) {
    mbar_init(a_full, 1);
    mbar_init(a_empty, 2);  // one commit per MMA issuer
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&t_full[s], 1);
      mbar_init(&t_empty[s], kEpiWarps);
    }
    mbar_init(done_bar, 2);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  // tile schedule: heaviest first, boustrophedon over the CTAs
  const int G = gridDim.x;
  auto tile_of = [&](int round, TileRef& tr) -> bool {
    int i = round * G + ((round & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x);
    return tile_at(tab, i, n_g, tr);
  };
  auto key_blocks = [&](const TileRef& tr) -> int64_t {
    int64_t last = min(tr.lrow0 + kRows, tr.rows) - 1;
    int64_t loc_max = (tr.q_off + last / n_g) / kKeys;
    return want_scores ? loc_max + 1 : loc_max;
  };
  // k_idx row of key block b's first key
  auto key_row = [&](const TileRef& tr, int64_t b) -> int32_t {
    return page_table ? page_table[tr.key0 + b] * kKeys : (int32_t)(tr.key0 + b * kKeys);
  };
  const int rounds = (tab.n_tiles + G - 1) / G;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t a_par = 0;
      bool a_armed = false;
      uint32_t armed_par[kStages];
      bool armed[kStages];
      for (int s = 0; s < kStages; ++s) armed[s] = false;
      long long it = 0;
      bool ok = true;
      for (int rd = 0; rd < rounds && ok; ++rd) {
        TileRef tr;
        if (!tile_of(rd, tr)) continue;
        int64_t nkb = key_blocks(tr);
        if (nkb <= 0) continue;
        if (!mbar_wait(a_empty, a_par ^ 1, abort_flag, dg)) { ok = false; break; }
        mbar_arrive_expect_tx(a_full, S::kABytes);
        for (int c = 0; c < S::kChunks; ++c)
          tma_load_2d(sA + c * S::kAChunk, &tm_q, a_full, c * kColsPerChunk, (int32_t)tr.row0);
        a_armed = true;
        a_par ^= 1;
        int32_t row_next = key_row(tr, 0);  // paged: the page id is read a block ahead
        for (int64_t b = 0; b < nkb; ++b, ++it) {
          const int s = (int)(it % kStages);
          const uint32_t par = (uint32_t)((it / kStages) & 1);
          const int32_t krow = row_next;
          if (b + 1 < nkb) row_next = key_row(tr, b + 1);
          if (!mbar_wait(&b_empty[s], par ^ 1, abort_flag, dg)) { ok = false; break; }
          mbar_arrive_expect_tx(&b_full[s], S::kBBytes);
          for (int c = 0; c < S::kChunks; ++c)
            tma_load_2d(sB + s * S::kBBytes + c * S::kBChunk, &tm_k, &b_full[s], c * kColsPerChunk,
                        krow);
          armed[s] = true;
          armed_par[s] = par;
        }
      }
      // let every issued copy land before shared memory is released, also when
      // another role gave up after this one had issued all of its copies
      if (!ok || *abort_flag) {
        for (int s = 0; s < kStages; ++s)
          if (armed[s]) mbar_drain(&b_full[s], armed_par[s]);
        if (a_armed) mbar_drain(a_full, a_par ^ 1);
      }
    }
  } else if (warp == 1 || warp == kIssuer2) {
    // ------------------------------------------------------------ MMA issuers
    // Two threads issue the MMAs, warp 1 those of the even key blocks (of the
    // CTA's running count), warp 10 the odd ones: while one waits on its
    // barriers the other keeps the tensor pipe fed. Even and odd blocks use
    // disjoint accumulator and k_idx stages; both wait for every tile's q_idx
    // (so that each sees every phase of a_full) and both release it.
    if (lane == 0) {
      const int mine = warp == 1 ? 0 : 1;
      constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(128, kKeys) : idesc_bf16_f32(128, kKeys);
      const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
      uint32_t a_par = 0;
      long long it = 0;
      bool ok = true;
      for (int rd = 0; rd < rounds && ok; ++rd) {
        TileRef tr;
        if (!tile_of(rd, tr)) continue;
        int64_t nkb = key_blocks(tr);
        if (nkb <= 0) continue;
        if (!mbar_wait(a_full, a_par, abort_flag, dg)) { ok = false; break; }
        a_par ^= 1;
        for (int64_t b = 0; b < nkb; ++b, ++it) {
          if ((int)(it & 1) != mine) continue;
          const int s = (int)(it % kStages);
          const uint32_t bpar = (uint32_t)((it / kStages) & 1);
          const int acc = (int)(it & 1);
          const uint32_t tpar = (uint32_t)((it >> 1) & 1);
          if (!mbar_wait(&t_empty[acc], tpar ^ 1, abort_flag, dg)) { ok = false; break; }
          if (!mbar_wait(&b_full[s], bpar, abort_flag, dg)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 256 + h * 128);
#pragma unroll
            for (int kk = 0; kk < DI * EB / 32; ++kk) {  // 32-byte K steps
              const int c = kk / 4, off = (kk % 4) * 32;
              uint64_t ad = desc_kmajor_sw128(a_base + c * S::kAChunk + h * 128 * 128 + off);
              uint64_t bd = desc_kmajor_sw128(b_base + s * S::kBBytes + c * S::kBChunk + off);
              if constexpr (F8) mma_e4m3_ss(d_tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
              else mma_bf16_ss(d_tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
            }
          }
          mma_commit(&b_empty[s]);
          mma_commit(&t_full[acc]);
        }
        if (ok) mma_commit(a_empty);
      }
      // every MMA issued by this thread has completed once done_bar flips
      mma_commit(done_bar);
      mbar_drain(done_bar, 0);
    }
  } else if (warp < kIssuer2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;      // accumulator half (rows h*128 ..)
    const int row_in_tile = h * 128 + q * 32 + lane;
    uint32_t it = 0;  // key blocks of this CTA so far (all tiles)
    bool ok = true;
    for (int rd = 0; rd < rounds && ok; ++rd) {
      TileRef tr;
      if (!tile_of(rd, tr)) continue;
      // row and position indexes fit 32 bits (the host caps rows x groups below 2^31)
      const int nkb = (int)key_blocks(tr);
      const int lr = (int)(tr.lrow0 + row_in_tile);  // row within the sequence
      const int r = (int)(tr.row0 + row_in_tile);    // row within the packed batch
      const bool valid = lr < tr.rows;
      const int t = valid ? (int)tr.q_off + lr / n_g : 0;  // the query's position
      const int loc = t / kKeys;
      RowTopK top;
      top.init(k - 1);
      for (int b = 0; b < nkb; ++b, ++it) {
        const int acc = (int)(it & 1);
        const uint32_t tpar = (uint32_t)((it >> 1) & 1);
        // one lane waits, the warp follows (tcgen05.ld needs a converged warp)
        int got = 0;
        if (lane == 0) got = mbar_wait(&t_full[acc], tpar, abort_flag, dg) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) { ok = false; break; }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * 256 + h * 128);
        // visible columns of this row in block b: all, or up to t on the diagonal
        const int lim = (b < loc) ? 128 : (b == loc ? t - b * kKeys + 1 : 0);
        // with every column visible to every row of the warp the loads reduce
        // (sm_103 load-with-max); the diagonal block reduces in registers
        const bool full = __all_sync(0xffffffffu, lim >= kKeys);
        float m = -INFINITY;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r0[32], r1[32];
          float m0 = -INFINITY, m1 = -INFINITY;
          if (full) {
            tmem_ld32_max(taddr + half * 64, r0, m0);
            tmem_ld32_max(taddr + half * 64 + 32, r1, m1);
          } else {
            tmem_ld32(taddr + half * 64, r0);
            tmem_ld32(taddr + half * 64 + 32, r1);
          }
          tmem_ld_wait();
          if (!full) {
            m0 = max32(r0, lim - half * 64);
            m1 = max32(r1, lim - half * 64 - 32);
          }
          m = fmax3(m, m0, m1);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&t_empty[acc]);
        if (valid && b <= loc) {
          if (want_scores) block_scores[(int64_t)r * nb + b] = F8 ? m * score_scale : m;
          if (b < loc && top.wants(m)) top.offer(m, b);
        }
      }
      if (ok && valid) top.emit(loc, k, block_ids + (int64_t)r * k);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

// 2D tensor [rows, cols] of bf16 (eb = 2) or byte codes (eb = 1), cols
// contiguous, box {128 bytes of columns, box_rows}, 128B swizzle
bool make_map_2d(CUtensorMap* m, const void* base, int64_t rows, int cols, int box_rows,
                 int eb) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * eb};
  cuuint32_t box[2] = {(cuuint32_t)(128 / eb), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

// one sequence of a launch: queries start .. start + len - 1 at positions
// q_off .. q_off + len - 1, keys from key0 (packed row or page-table entry)
struct SeqIn {
  int64_t start, len, q_off, key0;
};

// fills tb from at most kMaxSeq non-empty sequences
void make_table(SeqTable& tb, const SeqIn* in, int B, int n_g) {
  int idx[kMaxSeq];
  for (int i = 0; i < B; ++i) idx[i] = i;
  auto tiles_of = [&](int i) { return (int32_t)((in[i].len * n_g + kRows - 1) / kRows); };
  std::stable_sort(idx, idx + B, [&](int a, int b) { return tiles_of(a) > tiles_of(b); });
  tb.B = B;
  for (int s = 0; s < B; ++s) {
    const SeqIn& x = in[idx[s]];
    tb.start[s] = (int32_t)x.start;
    tb.len[s] = (int32_t)x.len;
    tb.q_off[s] = (int32_t)x.q_off;
    tb.key0[s] = (int32_t)x.key0;
    tb.tiles[s] = tiles_of(idx[s]);
  }
  int64_t end = 0;
  for (int s = 0; s < B; ++s) {
    const int32_t below = s + 1 < B ? tb.tiles[s + 1] : 0;
    end += (int64_t)(s + 1) * (tb.tiles[s] - below);
    tb.seg_end[s] = (int32_t)end;
  }
  tb.n_tiles = (int)end;
}

// q_idx [n_q, n_g, DI] holds every query of tb; k_idx [n_keys, DI] its keys
// (packed, or pages of 128 rows when page_table is given)
template <int DI, bool F8>
cudaError_t launch_tc(const void* q_idx, const void* k_idx, int64_t n_q, int64_t n_keys,
                      const SeqTable& tb, const int32_t* page_table, int n_g, int k,
                      int32_t* block_ids, float* block_scores, int64_t nb, float score_scale,
                      const Diag& dg, cudaStream_t st) {
  constexpr int EB = F8 ? 1 : 2;
  CUtensorMap tq, tk;
  if (!make_map_2d(&tq, q_idx, n_q * n_g, DI, kRows, EB) ||
      !make_map_2d(&tk, k_idx, n_keys, DI, kKeys, EB))
    return cudaErrorInvalidValue;
  const int smem = Smem<DI, EB>::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(index_select_tc_kernel<DI, F8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = std::min(tb.n_tiles, num_sms());
  note_launches(1);
  index_select_tc_kernel<DI, F8><<<grid, kThreads, smem, st>>>(
      tq, tk, tb, page_table, n_g, k, block_ids, block_scores, nb, score_scale, dg);
  return cudaGetLastError();
}

// bf16 launches over a batch, kMaxSeq non-empty sequences at a time
cudaError_t launch_batch(const void* q_idx, const void* k_idx, int64_t n_q, int64_t n_keys,
                         const SeqIn* seqs, int B, const int32_t* page_table, int n_g, int d_idx,
                         int k, int32_t* block_ids, const Diag& dg, cudaStream_t st) {
  SeqIn part[kMaxSeq];
  int m = 0;
  for (int b = 0; b <= B; ++b) {
    if (m == kMaxSeq || (b == B && m > 0)) {
      SeqTable tb;
      make_table(tb, part, m, n_g);
      const cudaError_t e =
          d_idx == 128 ? launch_tc<128, false>(q_idx, k_idx, n_q, n_keys, tb, page_table, n_g, k,
                                               block_ids, nullptr, 0, 1.f, dg, st)
                       : launch_tc<64, false>(q_idx, k_idx, n_q, n_keys, tb, page_table, n_g, k,
                                              block_ids, nullptr, 0, 1.f, dg, st);
      if (e != cudaSuccess) return e;
      m = 0;
    }
    if (b == B) break;
    if (seqs[b].len > 0) part[m++] = seqs[b];
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_index_select(const void* q_idx, const void* k_idx, int64_t N, int n_g,
                                int d_idx, int k, int32_t* block_ids, float* block_scores,
                                int64_t nb, const Diag& dg, cudaStream_t st, bool e4m3,
                                float score_scale) {
  if (N * n_g == 0) return cudaSuccess;
  SeqTable tb;
  const SeqIn one{0, N, 0, 0};
  make_table(tb, &one, 1, n_g);
  if (e4m3)  // E4M3 codes: 128 dimensions fill one 128-byte swizzle row
    return launch_tc<128, true>(q_idx, k_idx, N, N, tb, nullptr, n_g, k, block_ids, block_scores,
                                nb, score_scale, dg, st);
  if (d_idx == 128)
    return launch_tc<128, false>(q_idx, k_idx, N, N, tb, nullptr, n_g, k, block_ids,
                                 block_scores, nb, 1.f, dg, st);
  return launch_tc<64, false>(q_idx, k_idx, N, N, tb, nullptr, n_g, k, block_ids, block_scores,
                              nb, 1.f, dg, st);
}

namespace {
// NVFP4 rows -> bf16 rows, one 16-value micro-block (8 code bytes, one E4M3
// scale) per thread and iteration. A value is an E2M1 value (at most two
// significant bits, |x| <= 6) times an E4M3 scale (at most four, 2^-9 .. 448):
// at most six significant bits within bf16's range, so the product in fp32 and
// its bf16 rounding are exact.
__global__ void nvfp4_to_bf16_kernel(const uint2* __restrict__ codes,
                                     const uint8_t* __restrict__ scales, int64_t n_mb,
                                     uint4* __restrict__ out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_mb;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint2 c = codes[i];
    const __half_raw hs = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)scales[i], __NV_E4M3);
    const float sc = __half2float(__half(hs));
    uint32_t w[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t h2 = e2m1x2_to_f16x2(((b < 4 ? c.x : c.y) >> (8 * (b & 3))) & 0xFF);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      w[b] = pack_bf16x2(f.x * sc, f.y * sc);
    }
    out[2 * i] = make_uint4(w[0], w[1], w[2], w[3]);
    out[2 * i + 1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

cudaError_t nvfp4_to_bf16(const void* codes, const void* scales, int64_t rows, int d, void* out,
                          cudaStream_t st) {
  const int64_t n_mb = rows * (d / 16);
  if (n_mb == 0) return cudaSuccess;
  const int64_t g = std::min<int64_t>((n_mb + 255) / 256, (int64_t)num_sms() * 16);
  nvfp4_to_bf16_kernel<<<(unsigned)g, 256, 0, st>>>((const uint2*)codes, (const uint8_t*)scales,
                                                   n_mb, (uint4*)out);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_index_select_nvfp4(const void* q_codes, const void* q_scales,
                                      const void* k_codes, const void* k_scales, int64_t N,
                                      int n_g, int d_idx, int k, int32_t* block_ids,
                                      float* block_scores, int64_t nb, void* ws, const Diag& dg,
                                      cudaStream_t st) {
  if (N * n_g == 0) return cudaSuccess;
  unsigned char* qb = (unsigned char*)ws;
  unsigned char* kb = qb + (((size_t)N * n_g * d_idx * 2 + 255) & ~(size_t)255);
  note_launches(2);
  cudaError_t e = nvfp4_to_bf16(q_codes, q_scales, N * n_g, d_idx, qb, st);
  if (e == cudaSuccess) e = nvfp4_to_bf16(k_codes, k_scales, N, d_idx, kb, st);
  if (e != cudaSuccess) return e;
  return launch_index_select(qb, kb, N, n_g, d_idx, k, block_ids, block_scores, nb, dg, st);
}

cudaError_t launch_index_select_varlen(const void* q_idx, const void* k_idx,
                                       const int64_t* cu_seqlens, int B, int n_g, int d_idx,
                                       int k, int32_t* block_ids, const Diag& dg,
                                       cudaStream_t st) {
  const int64_t n_tok = cu_seqlens[B];
  for (int b0 = 0; b0 < B; b0 += kMaxSeq) {  // the table is filled in slices of kMaxSeq
    SeqIn seqs[kMaxSeq];
    const int m = std::min(kMaxSeq, B - b0);
    for (int i = 0; i < m; ++i) {
      const int64_t t0 = cu_seqlens[b0 + i];
      seqs[i] = SeqIn{t0, cu_seqlens[b0 + i + 1] - t0, 0, t0};
    }
    const cudaError_t e = launch_batch(q_idx, k_idx, n_tok, n_tok, seqs, m, nullptr, n_g, d_idx,
                                       k, block_ids, dg, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_index_select_paged(const void* q_idx, const void* k_idx_pages,
                                      int64_t n_pages, const int32_t* page_table, int max_pages,
                                      const int64_t* cu_q, const int64_t* kv_lens, int B, int n_g,
                                      int d_idx, int k, int32_t* block_ids, const Diag& dg,
                                      cudaStream_t st) {
  const int64_t n_q = cu_q[B];
  for (int b0 = 0; b0 < B; b0 += kMaxSeq) {
    SeqIn seqs[kMaxSeq];
    const int m = std::min(kMaxSeq, B - b0);
    for (int i = 0; i < m; ++i) {
      const int b = b0 + i;
      const int64_t len = cu_q[b + 1] - cu_q[b];
      seqs[i] = SeqIn{cu_q[b], len, kv_lens[b] - len, (int64_t)b * max_pages};
    }
    const cudaError_t e = launch_batch(q_idx, k_idx_pages, n_q, n_pages * kKeys, seqs, m,
                                       page_table, n_g, d_idx, k, block_ids, dg, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace msa
