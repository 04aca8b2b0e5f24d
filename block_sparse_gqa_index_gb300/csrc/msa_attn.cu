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

#include <climits>

#include "msa_kernels.h"
#include "msa_sm100.cuh"

namespace msa {
namespace {

constexpr int kBk = 128;
constexpr int kTileRows = 128;

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// upper bound on the tiles of a chunk: sum over buckets of ceil(count / qt)
// <= entries / qt + buckets
inline int64_t max_tiles(int64_t chunk, int64_t n_b, int H_q, int H_kv, int k) {
  const int64_t qt = kTileRows / (H_q / H_kv);
  return (chunk * H_kv * k + qt - 1) / qt + n_b;
}

// ------------------------------------------------------------ shared blocks
// Query tiles of qt consecutive rows (at most 32 here, one per lane). A block
// that at least half of a full tile's queries selected in group g is "shared":
// its (query, slot) entries leave the block-outer tiles and go to the
// query-outer pass (attn_shared_tc_kernel), which runs the tile's queries
// against each of their shared blocks with the output accumulated across
// blocks, and writes one record per (query, group) for all of them. Candidates
// are the blocks of four probe queries of the tile (first, a third, two
// thirds, last); a block selected by at least half the queries is missed only
// if none of the four probes selected it, and then simply stays block-outer.
constexpr int kShMax = 16;  // shared blocks kept per (query tile, group)

__global__ void __launch_bounds__(256)
shared_sets_kernel(const int32_t* __restrict__ ids, int64_t q0, int64_t q1, int n_g, int k,
                   int qt, int64_t n_qt, int32_t* __restrict__ shlist,
                   int32_t* __restrict__ rowmask, int32_t* __restrict__ rec_of, int64_t rec0) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < n_qt * n_g;
       w += nw) {
    const int64_t u = w / n_g;
    const int g = (int)(w % n_g);
    const int64_t t0 = q0 + u * qt;
    const int64_t left = q1 - t0;
    const int nq = (int)(left < qt ? left : qt);
    const bool has_q = lane < nq;
    const int64_t t = t0 + lane;
    // this lane's query: its usable block ids (others -1)
    int id[kMaxK];
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      int v = -1;
      if (has_q && s < k) {
        v = ids[(t * n_g + g) * k + s];
        if (v < 0 || (int64_t)v > t / kBk) v = -1;
      }
      id[s] = v;
    }
    int my_entry = -1;  // lane j holds shared block j
    int n_sh = 0;
    if (2 * nq >= qt) {  // tiles with too few queries keep every block block-outer
      const int thr = (nq + 1) / 2;
#pragma unroll 1
      for (int pb = 0; pb < 4; ++pb) {
        const int pi = pb == 0 ? 0 : (pb == 3 ? nq - 1 : pb * nq / 3);
#pragma unroll
        for (int s = 0; s < kMaxK; ++s) {
          if (s >= k) break;
          const int c = __shfl_sync(0xffffffffu, id[s], pi);
          if (c < 0 || n_sh >= kShMax || __any_sync(0xffffffffu, my_entry == c)) continue;
          bool mine = false;
#pragma unroll
          for (int s2 = 0; s2 < kMaxK; ++s2) mine |= id[s2] == c;
          if (__popc(__ballot_sync(0xffffffffu, mine)) >= thr) {
            if (lane == n_sh) my_entry = c;
            ++n_sh;
          }
        }
      }
    }
    // shared blocks in ascending order (a canonical order of accumulation,
    // whichever probe found them): bitonic sort over the first 16 lanes
    {
      int v = lane < n_sh ? my_entry : INT_MAX;
#pragma unroll
      for (int size = 2; size <= 16; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          const int p = __shfl_xor_sync(0xffffffffu, v, stride);
          const bool up = (lane & size) == 0, lower = (lane & stride) == 0;
          v = (lower == up) ? min(v, p) : max(v, p);
        }
      my_entry = lane < n_sh ? v : -1;
    }
    // the slots of this lane's query that the shared blocks cover, and which of
    // the shared blocks it selected
    uint32_t slots = 0, sel = 0;
#pragma unroll 1
    for (int j = 0; j < n_sh; ++j) {
      const int c = __shfl_sync(0xffffffffu, my_entry, j);
#pragma unroll
      for (int s = 0; s < kMaxK; ++s)
        if (id[s] == c) {
          slots |= 1u << s;
          sel |= 1u << j;
        }
    }
    if (lane < kShMax) shlist[w * kShMax + lane] = my_entry;
    if (has_q) {
      const int64_t row = (t - q0) * n_g + g;
      rowmask[row] = (int32_t)(slots | (sel << 16));
      // the first covered slot points at the (query, group)'s shared record
      // (item-major: the records of item w are contiguous)
      bool first = true;
#pragma unroll
      for (int s = 0; s < kMaxK; ++s)
        if ((slots >> s) & 1u) {
          rec_of[row * k + s] = first ? (int32_t)(rec0 + w * qt + lane) : -1;
          first = false;
        }
    }
  }
}

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

// Bucket of entry (row, id), or -1 when the id is not usable. Without qinfo
// the query row t is its position and the bucket is (group, block id); with
// qinfo (packed or paged sequences) qinfo[t] = {the first virtual block of
// t's sequence, t's position in it}, and the bucket is (group, virtual block).
__device__ __forceinline__ int bucket_of(const int2* __restrict__ qinfo, int id, int row, int t,
                                         int n_g, int nb, const Diag& dg) {
  int pos = t, vb = 0;
  if (qinfo) {
    const int2 qi = qinfo[t];
    vb = qi.x;
    pos = qi.y;
  }
  if (!id_ok(id, pos, dg)) return -1;
  return (row - t * n_g) * nb + vb + id;
}

// Counts the queries of every bucket; a slot with no usable block gets no
// partial record (rec_of = -1). Lanes of a warp that hit the same bucket add
// their count with one atomic (popular blocks are selected by most queries).
// entries of the chunk that the shared-block pass covers (rowmask bits 0-15)
__device__ __forceinline__ bool is_shared(const int32_t* __restrict__ rowmask, int e, int k) {
  return rowmask && ((rowmask[e / k] >> (e % k)) & 1);
}

__global__ void bucket_count_kernel(const int32_t* __restrict__ ids, int64_t q0, int64_t q1,
                                    int n_g, int k, int64_t nb, const int2* __restrict__ qinfo,
                                    const int32_t* __restrict__ rowmask,
                                    int32_t* __restrict__ counts, int32_t* __restrict__ rec_of,
                                    Diag dg) {
  const int n = (int)((q1 - q0) * n_g * k);  // entries of the chunk (< 2^31)
  const int row0 = (int)(q0 * n_g);
  const int lane = threadIdx.x & 31;
  const int* __restrict__ cids = ids + (size_t)row0 * k;
  for (int base = blockIdx.x * blockDim.x; base < n; base += gridDim.x * blockDim.x) {
    const int e = base + threadIdx.x;
    int bk = -1;
    if (e < n && !is_shared(rowmask, e, k)) {
      const int row = row0 + e / k;
      bk = bucket_of(qinfo, cids[e], row, row / n_g, n_g, (int)nb, dg);
      if (bk < 0) rec_of[e] = -1;
    }
    const unsigned same = __match_any_sync(0xffffffffu, bk);
    if (bk >= 0 && lane == __ffs(same) - 1) atomicAdd(&counts[bk], __popc(same));
  }
}

// Shared-memory bucketing, used when a CTA's shared memory holds one counter
// per bucket. CTA c takes a contiguous slice of the chunk's entries. Popular
// blocks (picked by most queries) then cost shared-memory atomics instead of
// serialised global atomics on one address. Pass 1 counts per CTA; a scan over
// the CTAs turns the counts into each CTA's first position per bucket; pass 2
// places the entries from those positions.
constexpr int kBucketCtas = 296;
constexpr int kSmemBucketsMax = 48 * 1024 / 4;

__device__ __forceinline__ void slice_of(int n, int c, int& e0, int& e1) {
  e0 = (int)((int64_t)n * c / gridDim.x);
  e1 = (int)((int64_t)n * (c + 1) / gridDim.x);
}

__global__ void __launch_bounds__(1024)
bucket_count_smem_kernel(const int32_t* __restrict__ ids, int64_t q0, int64_t q1, int n_g, int k,
                         int64_t nb, const int2* __restrict__ qinfo,
                         const int32_t* __restrict__ rowmask, int32_t* __restrict__ counts,
                         int32_t* __restrict__ percta, int32_t* __restrict__ rec_of, Diag dg) {
  extern __shared__ int32_t hist[];
  const int n_b = (int)(n_g * nb);
  for (int i = threadIdx.x; i < n_b; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  const int n = (int)((q1 - q0) * n_g * k);
  const int row0 = (int)(q0 * n_g);
  const int* __restrict__ cids = ids + (size_t)row0 * k;
  int e0, e1;
  slice_of(n, blockIdx.x, e0, e1);
  for (int e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
    if (is_shared(rowmask, e, k)) continue;
    const int row = row0 + e / k;
    const int bk = bucket_of(qinfo, cids[e], row, row / n_g, n_g, (int)nb, dg);
    if (bk >= 0) atomicAdd(&hist[bk], 1);
    else rec_of[e] = -1;
  }
  __syncthreads();
  int32_t* mine = percta + (size_t)blockIdx.x * n_b;
  for (int i = threadIdx.x; i < n_b; i += blockDim.x) {
    const int c = hist[i];
    mine[i] = c;
    if (c) atomicAdd(&counts[i], c);
  }
}

// per bucket: percta[c][b] <- offsets[b] + (entries of b in CTAs before c)
// one warp per bucket: the CTAs' counts 32 at a time, an exclusive prefix sum
// over the lanes, so each warp has 32 counts in flight instead of one
__global__ void bucket_cta_base_kernel(const int32_t* __restrict__ offsets, int n_b, int ctas,
                                       int32_t* __restrict__ percta) {
  const int lane = threadIdx.x & 31;
  for (int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < n_b;
       b += (gridDim.x * blockDim.x) >> 5) {
    int run = offsets[b];
    for (int c0 = 0; c0 < ctas; c0 += 32) {
      const int c = c0 + lane;
      const int x = c < ctas ? percta[(size_t)c * n_b + b] : 0;
      int incl = x;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (c < ctas) percta[(size_t)c * n_b + b] = run + incl - x;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
}

__global__ void __launch_bounds__(1024)
bucket_fill_smem_kernel(const int32_t* __restrict__ ids, int64_t q0, int64_t q1, int n_g, int k,
                        int64_t nb, const int2* __restrict__ qinfo,
                        const int32_t* __restrict__ rowmask, int qt,
                        const int32_t* __restrict__ offsets,
                        const int32_t* __restrict__ tile_off, const int32_t* __restrict__ percta,
                        int32_t* __restrict__ entries, int32_t* __restrict__ rec_of) {
  extern __shared__ int32_t cur[];
  const Diag none{nullptr, 0};
  const int n_b = (int)(n_g * nb);
  const int32_t* mine = percta + (size_t)blockIdx.x * n_b;
  for (int i = threadIdx.x; i < n_b; i += blockDim.x) cur[i] = mine[i];
  __syncthreads();
  const int n = (int)((q1 - q0) * n_g * k);
  const int row0 = (int)(q0 * n_g);
  const int* __restrict__ cids = ids + (size_t)row0 * k;
  int e0, e1;
  slice_of(n, blockIdx.x, e0, e1);
  for (int e = e0 + threadIdx.x; e < e1; e += blockDim.x) {
    if (is_shared(rowmask, e, k)) continue;
    const int rl = e / k;
    const int row = row0 + rl;
    const int t = row / n_g;
    const int bk = bucket_of(qinfo, cids[e], row, t, n_g, (int)nb, none);
    if (bk < 0) continue;
    const int pos = atomicAdd(&cur[bk], 1);
    entries[pos] = ((t - (int)q0) << 4) | (e - rl * k);
    rec_of[e] = tile_off[bk] * qt + (pos - offsets[bk]);
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

// Places every (query, slot) of a bucket: its entry (query << 4 | slot) at the
// bucket's next position, and the index of its partial record, which is the
// tile-major position tile * qt + (query's place in its tile). Lanes of a warp
// that hit the same bucket take consecutive positions from one atomic.
__global__ void bucket_fill_kernel(const int32_t* __restrict__ ids, int64_t q0, int64_t q1,
                                   int n_g, int k, int64_t nb, const int2* __restrict__ qinfo,
                                   const int32_t* __restrict__ rowmask, int qt,
                                   const int32_t* __restrict__ offsets,
                                   const int32_t* __restrict__ tile_off,
                                   int32_t* __restrict__ cursor, int32_t* __restrict__ entries,
                                   int32_t* __restrict__ rec_of) {
  const Diag none{nullptr, 0};
  const int n = (int)((q1 - q0) * n_g * k);
  const int row0 = (int)(q0 * n_g);
  const int lane = threadIdx.x & 31;
  const int* __restrict__ cids = ids + (size_t)row0 * k;
  for (int base = blockIdx.x * blockDim.x; base < n; base += gridDim.x * blockDim.x) {
    const int e = base + threadIdx.x;
    int bk = -1, ent = 0;
    if (e < n && !is_shared(rowmask, e, k)) {
      const int rl = e / k;
      const int row = row0 + rl;
      const int t = row / n_g;
      bk = bucket_of(qinfo, cids[e], row, t, n_g, (int)nb, none);
      if (bk >= 0) ent = ((t - (int)q0) << 4) | (e - rl * k);
    }
    const unsigned same = __match_any_sync(0xffffffffu, bk);
    const int leader = __ffs(same) - 1;
    int c0 = 0;
    if (bk >= 0 && lane == leader) c0 = atomicAdd(&cursor[bk], __popc(same));
    c0 = __shfl_sync(0xffffffffu, c0, leader);
    if (bk >= 0) {
      const int c = c0 + __popc(same & ((1u << lane) - 1));
      entries[offsets[bk] + c] = ent;
      rec_of[e] = tile_off[bk] * qt + c;
    }
  }
}

// ------------------------------------------------------- tile kernel (tcgen05)
// One persistent CTA per SM walks a contiguous range of tiles (consecutive
// tiles mostly share a bucket, so K / V of the bucket's block are loaded once).
// Every role finds its tile through the tile's record (one 16-byte load,
// fetched ahead of use). Two TMEM stages of 256 columns (S/P | O) alternate
// between consecutive tiles.
//   warp 0     K by TMA when the bucket changes (128 keys of head g; single
//              buffer, reloaded once the bucket's last S has completed), then
//              S = Q K^T (128 x 128, A = Q tile, B = K block, both K-major and
//              128B-swizzled in shared memory) into the tile's S/P columns as
//              soon as the P.V that last read them has completed;
//   warp 1     TMEM owner; V by TMA when the bucket changes (reloaded once the
//              bucket's last P.V has completed), then O = P V (A = P read from
//              TMEM, B = V as an MN-major operand) once the softmax has written
//              P and the epilogue two tiles back has read the O columns.
//              Splitting the two MMA streams over two threads lets each block
//              on its own barriers;
//   warps 2, 3, 12, 13
//              Q producers: producer p fills the Q stage i % 4 of the tiles i
//              with i % 4 == p. It reads the tile's entries ahead of time, then
//              gathers the G head rows of each of the tile's queries with TMA
//              row gathers (tile::gather4) into the 128B-swizzled layout; a
//              stage is free again as soon as the S MMA that read it completed;
//   warps 4-11 softmax + epilogue, two groups of four warps (warpgroups 1 and
//              2, one per TMEM stage), one score row per thread: the row's
//              query and partial slot come straight from the tile's entries;
//              the whole row of S in registers (one TMEM load round trip),
//              masked row max, exp2, row sum, P (bf16) back into TMEM over S;
//              then the whole O row, O / l in bf16 and the row's LSE into the
//              tile's partial records in a shared-memory staging buffer;
//   warp 14    one bulk copy per tile of its records (tile-major, so a tile's
//              records are contiguous) from the staging buffer to the partial
//              buffer. Warp 15 only rounds out warpgroup 3.
// The softmax warpgroups hold 192 registers per thread and the other two 64
// (setmaxnreg at the top of each role's branch, so that the compiler allocates
// each branch with its own budget).
template <int D>
struct AttnSmem {
  static constexpr int kKVBytes = kBk * D * 2;            // one of K or V
  static constexpr int kQBytes = kTileRows * D * 2;       // one Q stage
  static constexpr int kQStages = 4;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKVBytes;
  static constexpr int kQOff = 2 * kKVBytes;
  static constexpr int kStgOff = kQOff + kQStages * kQBytes;
  static constexpr int kStgBytes = kTileRows * D * 2 + kTileRows * 16;  // a tile's records (G = 1)
  static constexpr int kBarOff = kStgOff + kStgBytes;
  // k_full, k_empty, v_full, v_empty, q_full[4], q_empty[4], s_full[2], p_full[2],
  // o_full[2], o_empty[2], done[2], stg_empty[2], stg_full
  static constexpr int kNumBars = 4 + 2 * kQStages + 8 + 2 + 3;
  static constexpr int kBytes = kBarOff + kNumBars * 8 + 32;
};
// the kernel needs its dynamic shared memory 1024-byte aligned (it checks)
static_assert(AttnSmem<128>::kBytes <= 232448, "attention tile exceeds shared memory");

constexpr int kProducers = 4;      // Q producer warps (2, 3, 12, 13)
constexpr int kStoreWarp = 14;     // bulk stores of the partial records
constexpr int kAttnThreads = 512;  // 16 warps: four warpgroups

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

// One record per tile, so that every role of the tile kernel finds its tile
// with one independent load: {row of the block's first key in K / V, first
// entry, queries | group g << 8, end tile of the bucket}. A single sequence's
// block b starts at row 128 b; with vinfo (packed or paged sequences) virtual
// block v starts at row vinfo[v].x, and tbase[tile] = vinfo[v].y is the query
// row that would sit at the block's first key position (the causal mask of
// the block is then key column c visible to query row t iff c <= t - base).
__global__ void tile_map_kernel(const int32_t* __restrict__ tile_off,
                                const int32_t* __restrict__ offsets, int64_t n_b, int64_t nb,
                                int qt, const int2* __restrict__ vinfo,
                                int32_t* __restrict__ tbase, int4* __restrict__ tinfo) {
  const int64_t total = tile_off[n_b];
  for (int64_t tile = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; tile < total;
       tile += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bk = find_bucket(tile_off, n_b, tile);
    const int e0 = offsets[bk] + (int)(tile - tile_off[bk]) * qt;
    const int v = (int)(bk % nb);
    int row = v * kBk;
    if (vinfo) {
      const int2 vi = vinfo[v];
      row = vi.x;
      if (tbase) tbase[tile] = vi.y;
    }
    tinfo[tile] = make_int4(row, e0, min(qt, offsets[bk + 1] - e0) | (int)(bk / nb) << 8,
                            tile_off[bk + 1]);
  }
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_tile_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_q, int64_t tm_rows,
                    int64_t q0, int H_q, int H_kv, int k,
                    float scale_log2, int64_t nb, const int32_t* __restrict__ entries,
                    const int4* __restrict__ tinfo, const int32_t* __restrict__ tbase,
                    const int32_t* __restrict__ n_tiles,
                    unsigned char* __restrict__ part, Diag dg) {
  using namespace sm100;
  using S = AttnSmem<D>;
  constexpr int QS = S::kQStages;
  extern __shared__ __align__(1024) unsigned char smem[];
  if (smem_u32(smem) & 1023) {  // the 128B-swizzled operands need 1024-byte alignment
    if (threadIdx.x == 0) report(dg, kStatusUnsupported);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* k_full = bars + 0;
  uint64_t* k_empty = bars + 1;
  uint64_t* v_full = bars + 2;
  uint64_t* v_empty = bars + 3;
  uint64_t* q_full = bars + 4;
  uint64_t* q_empty = q_full + QS;
  uint64_t* s_full = q_empty + QS;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = p_full + 2;
  uint64_t* o_empty = o_full + 2;
  uint64_t* done_bar = o_empty + 2;
  // stg_empty[i & 1] completes when tile i's records have been read out of the
  // staging buffer. Two barriers, because a group can reach tile i + 2 before
  // tile i's copy is done: a single barrier's parity would then be ambiguous.
  uint64_t* stg_empty = done_bar + 2;
  uint64_t* stg_full = stg_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + S::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = H_q / H_kv;
  const int qt = kTileRows / G;
  const int q0i = (int)q0;
  const int rec = attn_rec_bytes(G, D);

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    for (int s = 0; s < QS; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);  // the S-MMA commit
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4);
      mbar_init(&o_full[s], 1);
      mbar_init(&o_empty[s], 4);
    }
    mbar_init(&done_bar[0], 1);
    mbar_init(&done_bar[1], 1);
    mbar_init(&stg_empty[0], 1);
    mbar_init(&stg_empty[1], 1);
    mbar_init(stg_full, 4);
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
  // warpgroups 1 and 2 (warps 4-11) are the softmax groups: they take 192
  // registers per thread so that a thread holds a whole row; warpgroups 0 and
  // 3 (issuers, producers, store) drop to 64. 2 x 128 x 192 + 2 x 128 x 64
  // is the 65536 registers the 512 threads were launched with.

  // this CTA's contiguous range of tiles
  const int64_t total = *n_tiles;
  const int t_begin = (int)(total * blockIdx.x / gridDim.x);
  const int t_end = (int)(total * (blockIdx.x + 1) / gridDim.x);
  const int n_local = t_end - t_begin;
  const int4 kNone = make_int4(0, 0, 0, 0);

  const int wgid = warp >> 2;
  if (wgid == 0 || wgid == 3) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 64;\n" ::: "memory");
  if (warp == 0) {
    // ---------------------------------------------------------- K + S = Q K^T
    // Per K/V block (the next one starts at this block's end tile): once the
    // previous block's last S has completed, load K by TMA. Per tile j: S(j)
    // overwrites the S/P columns of TMEM stage j & 1, so it waits for
    // P.V(j - 2) to have completed, and for its Q stage.
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kBk);
      const uint32_t k_base = smem_u32(smem + S::kKOff);
      const uint32_t q_base = smem_u32(smem + S::kQOff);
      uint32_t epoch = 0;
      int s_last = -1;
      int4 inf = tinfo[t_begin];
      for (int j = 0; j < n_local; ++j) {
        if (j > s_last) {
          s_last = min(inf.w - t_begin, n_local) - 1;
          const int4 nxt = s_last + 1 < n_local ? tinfo[t_begin + s_last + 1] : kNone;
          if (!mbar_wait(k_empty, (epoch & 1) ^ 1, abort_flag, dg)) break;
          mbar_arrive_expect_tx(k_full, S::kKVBytes);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + S::kKOff + c * kBk * 128, &tm_k, k_full, c * 64, inf.z >> 8, inf.x);
          ++epoch;
          inf = nxt;
          if (!mbar_wait(k_full, (epoch - 1) & 1, abort_flag, dg)) break;
        }
        const int st = j & 1, qs = j % QS;
        if ((j >= 2 && !mbar_wait(&o_full[st], (uint32_t)(((j - 2) >> 1) & 1), abort_flag, dg)) ||
            !mbar_wait(&q_full[qs], (uint32_t)((j / QS) & 1), abort_flag, dg))
          break;
        tc_fence_after();
        const uint32_t d_s = tmem_base + (uint32_t)(st * 256);
        const uint32_t qa = q_base + qs * S::kQBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const int c = kk / 4, off = (kk % 4) * 32;
          mma_bf16_ss(d_s, desc_kmajor_sw128(qa + c * kTileRows * 128 + off),
                      desc_kmajor_sw128(k_base + c * kBk * 128 + off), idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[st]);
        mma_commit(&q_empty[qs]);
        if (j == s_last) mma_commit(k_empty);
      }
      if (*abort_flag && epoch > 0) mbar_drain(k_full, (epoch - 1) & 1);
      mma_commit(&done_bar[0]);
      mbar_drain(&done_bar[0], 0);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- V + O = P V
    // Per K/V block: once this thread's last P.V of the previous block has
    // completed, load V by TMA (meanwhile the block's first softmax runs). Per
    // tile j, once its softmax has written P: P.V(j) overwrites the O columns
    // of TMEM stage j & 1, so it waits for the epilogue of tile j - 2 to have
    // read them.
    if (lane == 0 && n_local > 0) {
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      const uint32_t v_base = smem_u32(smem + S::kVOff);
      uint32_t epoch = 0;
      int o_last = -1;
      int4 inf = tinfo[t_begin];
      for (int j = 0; j < n_local; ++j) {
        if (j > o_last) {
          o_last = min(inf.w - t_begin, n_local) - 1;
          const int4 nxt = o_last + 1 < n_local ? tinfo[t_begin + o_last + 1] : kNone;
          if (!mbar_wait(v_empty, (epoch & 1) ^ 1, abort_flag, dg)) break;
          mbar_arrive_expect_tx(v_full, S::kKVBytes);
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(smem + S::kVOff + c * kBk * 128, &tm_v, v_full, c * 64, inf.z >> 8, inf.x);
          ++epoch;
          inf = nxt;
          if (!mbar_wait(v_full, (epoch - 1) & 1, abort_flag, dg)) break;
        }
        const int st = j & 1;
        if (!mbar_wait(&p_full[st], (uint32_t)((j >> 1) & 1), abort_flag, dg) ||
            (j >= 2 && !mbar_wait(&o_empty[st], (uint32_t)(((j - 2) >> 1) & 1), abort_flag, dg)))
          break;
        tc_fence_after();
        const uint32_t d_o = tmem_base + (uint32_t)(st * 256 + 128);
#pragma unroll
        for (int kk = 0; kk < kBk / 16; ++kk) {
          const uint32_t a_p = tmem_base + (uint32_t)(st * 256 + kk * 8);
          const uint64_t bd = desc_mnmajor_sw128(v_base + kk * 16 * 128, kBk * 128);
          mma_bf16_ts(d_o, a_p, bd, idesc_o, kk > 0 ? 1u : 0u);
        }
        mma_commit(&o_full[st]);
        if (j == o_last) mma_commit(v_empty);
      }
      if (*abort_flag && epoch > 0) mbar_drain(v_full, (epoch - 1) & 1);
      mma_commit(&done_bar[1]);
      mbar_drain(&done_bar[1], 0);
    }
  } else if (warp == 2 || warp == 3 || warp == 12 || warp == 13) {
    // ---------------------------------------------------------- Q producers
    // Tile rows are head-major: row r holds head i = r / qt of query r % qt, so
    // four consecutive rows are one head of four queries, fetched by one TMA
    // row gather (tile::gather4) per 64-column chunk. Rows past the tile's
    // queries use an out-of-range row and are zero-filled. Lane l holds the
    // entries of queries l, l + 32, ... of the tile; the gathers pick up their
    // rows by shuffles. A tile's entries are loaded one iteration ahead and its
    // record two iterations ahead, so no global load is waited on here.
    const int p = warp < 4 ? warp - 2 : warp - 10;
    const int32_t oob_row = (int32_t)(tm_rows);  // first row past q: zero fill
    const int nj = (qt + 31) / 32;
    constexpr int NCH = D / 64;
    uint32_t armed = 0, armed_par = 0;  // per-stage bits: issued a copy, its parity
    int i = p;
    int4 inf_c = i < n_local ? tinfo[t_begin + i] : kNone;
    int ent_c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      ent_c[j] = (i < n_local && j < nj && lane + 32 * j < (inf_c.z & 0xFF))
                     ? entries[inf_c.y + lane + 32 * j] : -1;
    int4 inf_n = i + kProducers < n_local ? tinfo[t_begin + i + kProducers] : kNone;
    bool stop = false;
    for (; i < n_local && !stop; i += kProducers) {
      int ent_n[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ent_n[j] = (i + kProducers < n_local && j < nj && lane + 32 * j < (inf_n.z & 0xFF))
                       ? entries[inf_n.y + lane + 32 * j] : -1;
      const int4 inf_nn = i + 2 * kProducers < n_local ? tinfo[t_begin + i + 2 * kProducers] : kNone;
      const int gg = (inf_c.z >> 8) * G;
      int32_t qrow[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        qrow[j] = ent_c[j] >= 0 ? (int32_t)((q0 + (ent_c[j] >> 4)) * H_q + gg) : -1;
      const int qs = (int)(i % QS);
      const uint32_t par = (uint32_t)((i / QS) & 1);
      int got = 0;
      if (lane == 0) got = mbar_wait(&q_empty[qs], par ^ 1, abort_flag, dg);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      if (lane == 0) mbar_arrive_expect_tx(&q_full[qs], S::kQBytes);
      __syncwarp();
      unsigned char* qbuf = smem + S::kQOff + qs * S::kQBytes;
      // one gather4 per (group of 4 rows, 64-column chunk); 32 * NCH jobs, so
      // every lane runs the same number of iterations (the shuffles need it)
      for (int job = lane; job < (kTileRows / 4) * NCH; job += 32) {
        const int r0 = (job / NCH) * 4, c = job % NCH;
        const int hi = r0 / qt, qb = r0 % qt, jj = qb >> 5;
        int32_t y[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int src = (qb + u) & 31;
          int32_t v = -1;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (j < nj) {
              const int32_t x = __shfl_sync(0xffffffffu, qrow[j], src);
              if (j == jj) v = x;
            }
          }
          y[u] = v >= 0 ? v + hi : oob_row;
        }
        tma_gather4(qbuf + c * kTileRows * 128 + r0 * 128, &tm_q, &q_full[qs], c * 64, y[0],
                    y[1], y[2], y[3]);
      }
      armed |= 1u << qs;
      armed_par = (armed_par & ~(1u << qs)) | (par << qs);
      stop = *abort_flag != 0;
      inf_c = inf_n;
      inf_n = inf_nn;
#pragma unroll
      for (int j = 0; j < 4; ++j) ent_c[j] = ent_n[j];
    }
    // on abort, let every copy this warp issued land before shared memory goes
    if (lane == 0 && *abort_flag) {
#pragma unroll
      for (int s = 0; s < QS; ++s)
        if ((armed >> s) & 1) mbar_drain(&q_full[s], (armed_par >> s) & 1);
    }
  } else if (warp == kStoreWarp) {
    // ---------------------------------------------------------- partial records out
    // Tile i's records (its first nq queries, contiguous in the staging buffer)
    // go out in one bulk copy to their tile-major place once the four warps of
    // the tile's softmax group have written them; the buffer is free again once
    // the copy has read it.
    if (lane == 0 && n_local > 0) {
      int4 inf = tinfo[t_begin];
      for (int i = 0; i < n_local; ++i) {
        const int4 nxt = i + 1 < n_local ? tinfo[t_begin + i + 1] : kNone;
        if (!mbar_wait(stg_full, (uint32_t)(i & 1), abort_flag, dg)) break;
        bulk_store(part + (size_t)(t_begin + i) * qt * rec, smem + S::kStgOff,
                   (uint32_t)((inf.z & 0xFF) * rec));
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(&stg_empty[i & 1]);
        inf = nxt;
      }
    }
  }
  } else {
    // ---------------------------------------------------------- softmax + epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;\n" ::: "memory");
    // two groups of 4 warps; group wg takes the tiles i with i % 2 == wg, which
    // use TMEM stage wg, so one group's softmax overlaps the other's epilogue.
    // A row's entry is loaded one tile ahead, the tile record two tiles ahead.
    const int wg = (warp - 4) >> 2;
    const int qq = warp & 3;
    const int row = qq * 32 + lane;
    const int hi = row / qt, qi = row % qt;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const int st = wg;
    const uint32_t ts = tmem_base + lane_off + (uint32_t)(st * 256);
    const uint32_t stg_base = smem_u32(smem + S::kStgOff);
    int4 inf_c = wg < n_local ? tinfo[t_begin + wg] : kNone;
    int ent_c = (wg < n_local && qi < (inf_c.z & 0xFF)) ? entries[inf_c.y + qi] : -1;
    int4 inf_n = wg + 2 < n_local ? tinfo[t_begin + wg + 2] : kNone;
    for (int i = wg; i < n_local; i += 2) {
      const int ent_n = (i + 2 < n_local && qi < (inf_n.z & 0xFF)) ? entries[inf_n.y + qi] : -1;
      const int4 inf_nn = i + 4 < n_local ? tinfo[t_begin + i + 4] : kNone;
      const int base = tbase ? tbase[t_begin + i] : inf_c.x;  // query row at the block's key 0
      const uint32_t par = (uint32_t)((i >> 1) & 1);
      const int t = ent_c >= 0 ? q0i + (ent_c >> 4) : 0;
      int got = 0;
      if (lane == 0) got = mbar_wait(&s_full[st], par, abort_flag, dg);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      tc_fence_after();
      const int lim = (ent_c >= 0 && t - base < kBk) ? t - base + 1 : kBk;
      // the whole row in registers: one load round trip; with no masked column
      // in the warp the loads also reduce the row max (sm_103 load-with-max)
      const bool full = __all_sync(0xffffffffu, lim >= kBk);
      uint32_t r[128];
      float m;
      if (full) {
        float m0, m1, m2, m3;
        tmem_ld32_max(ts, *reinterpret_cast<uint32_t(*)[32]>(&r[0]), m0);
        tmem_ld32_max(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]), m1);
        tmem_ld32_max(ts + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]), m2);
        tmem_ld32_max(ts + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]), m3);
        tmem_ld_wait();
        m = fmaxf(fmax3(m0, m1, m2), m3);
      } else {
        tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_ld32(ts + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
        tmem_ld32(ts + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
        tmem_ld_wait();
        m = -INFINITY;
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j < lim) m = fmaxf(m, __uint_as_float(r[j]));
      }
      const float mc = m * scale_log2;
      // P = exp2(s * c - m * c), packed to bf16 pairs in place (r[j] holds
      // columns 2j, 2j + 1), row sum; rows of the local block mask the columns
      // past their query
      const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-mc, -mc);
      uint64_t l2 = f2_pack(0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        float p0, p1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), sc2,
                         nm2), p0, p1);
        p0 = ex2_approx(p0);
        p1 = ex2_approx(p1);
        if (!full) {
          p0 = 2 * j < lim ? p0 : 0.f;
          p1 = 2 * j + 1 < lim ? p1 : 0.f;
        }
        l2 = f2_add(l2, f2_pack(p0, p1));
        r[j] = pack_bf16x2(p0, p1);
      }
      tmem_st32(ts, *reinterpret_cast<const uint32_t(*)[32]>(&r[0]));
      tmem_st32(ts + 32, *reinterpret_cast<const uint32_t(*)[32]>(&r[32]));
      float l0, l1;
      f2_unpack(l2, l0, l1);
      const float l = l0 + l1;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[st]);
      // O epilogue: O / l in bf16 and the LSE into this tile's records in the
      // staging buffer (shared by both groups, taken in tile order), then one
      // bulk copy per query of its record to the partial buffer
      got = 0;
      if (lane == 0)
        got = mbar_wait(&o_full[st], par, abort_flag, dg) &&
              (i == 0 ||
               mbar_wait(&stg_empty[(i - 1) & 1], (uint32_t)(((i - 1) >> 1) & 1), abort_flag, dg));
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      tc_fence_after();
      const float inv = 1.f / l;
      const uint64_t inv2 = f2_pack(inv, inv);
      const uint32_t srow = stg_base + (uint32_t)(qi * rec + hi * D * 2);
      auto o_chunk = [&](const uint32_t(&r)[32], int c) {
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float x0, x1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(r[8 * v + 2 * u]),
                                     __uint_as_float(r[8 * v + 2 * u + 1])), inv2), x0, x1);
            w[u] = pack_bf16x2(x0, x1);
          }
          st_shared_v4(srow + c * 64 + v * 16, w[0], w[1], w[2], w[3]);
        }
      };
      {
        uint32_t ro[D];
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
          tmem_ld32(ts + 128 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&ro[32 * c]));
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) o_chunk(*reinterpret_cast<const uint32_t(*)[32]>(&ro[32 * c]), c);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_empty[st]);  // the O columns are free again
      *reinterpret_cast<float*>(smem + S::kStgOff + qi * rec + G * D * 2 + hi * 4) =
          (mc + __log2f(l)) * 0.69314718055994531f;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(stg_full);
      inf_c = inf_n;
      inf_n = inf_nn;
      ent_c = ent_n;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// ------------------------------------------------- shared blocks, query-outer
// One item = one (query tile, group) with its shared blocks (shared_sets_kernel):
// the tile's qt queries x G heads (128 rows, query-major: row r = query r / G,
// head r % G, loaded by one TMA box per 64-column chunk) against each shared
// block in turn, the output accumulated in TMEM across the blocks. A row whose
// query did not select a block, or whose local block masks it, takes P = 0
// there. Online softmax with a lazy rescale: a row keeps the running max it
// used for P unless a block's max exceeds it by more than 8 (a factor 2^8 in
// P, well within bf16 / fp32); only then does it rescale its O row in TMEM and
// its sum, and move its max. S(j + 1) is issued once P.V(j) has completed, so
// when the softmax sees S(j) its O holds every block before j. The item ends
// with its qt records (one per query, in the format of the block-outer
// partials, item-major so that they are contiguous), staged in the V buffer
// (free once the item's last P.V has completed) and written by one bulk copy;
// the merge combines them with the block-outer partials.
//
// Each CTA runs one item at a time, as a chain S -> softmax -> P.V -> S; two
// CTAs per SM (256 TMEM columns and about 100 KB of shared memory each) keep
// the tensor core busy with one while the other's softmax runs. 8 warps:
//   warp 0     TMA: each item's Q and each block's K (one buffer each);
//   warp 1     TMEM owner; MMA issuer;
//   warp 2     TMA: each block's V (one buffer, also the record staging);
//   warp 3     bulk copy of the staged records;
//   warps 4-7  softmax and epilogue, one row per thread.
template <int D>
struct ShSmem {
  static constexpr int kQBytes = kTileRows * D * 2;
  static constexpr int kKVBytes = kBk * D * 2;
  // an item's records: qt (G * D * 2 + G * 4) bytes = 128 (2 D + 4), any G
  static constexpr int kStgBytes = kTileRows * (2 * D + 4);
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQBytes;
  static constexpr int kVOff = kKOff + kKVBytes;
  static constexpr int kVBytes = kStgBytes > kKVBytes ? kStgBytes : kKVBytes;
  static constexpr int kBarOff = kVOff + kVBytes;
  // q_full, q_empty, k_full, k_empty, v_full, v_empty, s_full, p_full,
  // pv_done, o_full, o_free, stg_full, stg_free, done
  static constexpr int kNumBars = 14;
  static constexpr int kBytes = kBarOff + kNumBars * 8 + 32;
};
static_assert(2 * (ShSmem<128>::kBytes + 1024) <= 233472, "two shared-block CTAs per SM");
constexpr int kShThreads = 256;

// number of shared blocks of item w (its list is -1 past them)
__device__ __forceinline__ int sh_count(const int32_t* __restrict__ shlist, int64_t w) {
  const int4* p = reinterpret_cast<const int4*>(shlist + w * kShMax);
  int c = 0;
#pragma unroll
  for (int i = 0; i < kShMax / 4; ++i) {
    const int4 v = __ldg(p + i);
    c += (v.x >= 0) + (v.y >= 0) + (v.z >= 0) + (v.w >= 0);
  }
  return c;
}

template <int D>
__global__ void __launch_bounds__(kShThreads, 2)
attn_shared_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, int64_t q0, int64_t q1,
                      int H_q, int H_kv, float scale_log2, int64_t n_items,
                      const int32_t* __restrict__ shlist, const int32_t* __restrict__ rowmask,
                      int64_t rec0, unsigned char* __restrict__ part, Diag dg) {
  using namespace sm100;
  using S = ShSmem<D>;
  extern __shared__ __align__(1024) unsigned char smem[];
  if (smem_u32(smem) & 1023) {
    if (threadIdx.x == 0) report(dg, kStatusUnsupported);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = bars + 3;
  uint64_t* v_full = bars + 4;
  uint64_t* v_empty = bars + 5;
  uint64_t* s_full = bars + 6;
  uint64_t* p_full = bars + 7;
  uint64_t* pv_done = bars + 8;
  uint64_t* o_full = bars + 9;
  uint64_t* o_free = bars + 10;
  uint64_t* stg_full = bars + 11;
  uint64_t* stg_free = bars + 12;
  uint64_t* done_bar = bars + 13;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + S::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = H_q / H_kv;
  const int qt = kTileRows / G;
  const int n_g = H_kv;
  const int rec = attn_rec_bytes(G, D);
  if (threadIdx.x == 0) {
    for (int i = 0; i < S::kNumBars; ++i) mbar_init(&bars[i], 1);
    mbar_init(p_full, 4);
    mbar_init(o_free, 4);
    mbar_init(stg_full, 4);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // warpgroup 0 (TMA, MMA, store) runs on 48 registers per thread, the
  // softmax warpgroup on 208: 128 x 48 + 128 x 208 = 256 x 128, the launch's share
  if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 48;\n" ::: "memory");
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ TMA: Q, K
      uint32_t it = 0, e = 0;
      bool q_armed = false, k_armed = false;
      bool ok = true;
      for (int64_t w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int cnt = sh_count(shlist, w);
        if (cnt == 0) continue;
        const int g = (int)(w % n_g);
        if (!mbar_wait(q_empty, (it & 1) ^ 1, abort_flag, dg)) break;
        mbar_arrive_expect_tx(q_full, S::kQBytes);
        const int64_t t0 = q0 + (w / n_g) * qt;
        for (int ch = 0; ch < D / 64; ++ch)
          tma_load_3d(smem + S::kQOff + ch * kTileRows * 128, &tm_q, q_full, ch * 64, g * G,
                      (int32_t)t0);
        q_armed = true;
        for (int j = 0; j < cnt; ++j, ++e) {
          const int b = shlist[w * kShMax + j];
          if (!mbar_wait(k_empty, (e & 1) ^ 1, abort_flag, dg)) { ok = false; break; }
          mbar_arrive_expect_tx(k_full, S::kKVBytes);
          for (int ch = 0; ch < D / 64; ++ch)
            tma_load_3d(smem + S::kKOff + ch * kBk * 128, &tm_k, k_full, ch * 64, g, b * kBk);
          k_armed = true;
        }
        ++it;
      }
      if (*abort_flag) {  // let issued copies land before shared memory goes
        if (q_armed) mbar_drain(q_full, (it - (ok ? 1 : 0)) & 1);
        if (k_armed) mbar_drain(k_full, (e - 1) & 1);
      }
    } else if (warp == 2 && lane == 0) {
      // ------------------------------------------------------------ TMA: V
      // A new item's first V overwrites the staged records of the previous
      // item, so it waits for their bulk copy to have read them.
      uint32_t it = 0, e = 0;
      bool armed = false;
      bool ok = true;
      for (int64_t w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int cnt = sh_count(shlist, w);
        if (cnt == 0) continue;
        const int g = (int)(w % n_g);
        for (int j = 0; j < cnt; ++j, ++e) {
          const int b = shlist[w * kShMax + j];
          if (!mbar_wait(v_empty, (e & 1) ^ 1, abort_flag, dg) ||
              (j == 0 && it > 0 && !mbar_wait(stg_free, (it - 1) & 1, abort_flag, dg))) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(v_full, S::kKVBytes);
          for (int ch = 0; ch < D / 64; ++ch)
            tma_load_3d(smem + S::kVOff + ch * kBk * 128, &tm_v, v_full, ch * 64, g, b * kBk);
          armed = true;
        }
        ++it;
      }
      if (*abort_flag && armed) mbar_drain(v_full, (e - (ok ? 1 : 0)) & 1);
    } else if (warp == 3 && lane == 0) {
      // ------------------------------------------------------------ records out
      uint32_t it = 0;
      for (int64_t w = blockIdx.x; w < n_items; w += gridDim.x) {
        if (sh_count(shlist, w) == 0) continue;
        if (!mbar_wait(stg_full, it & 1, abort_flag, dg)) break;
        bulk_store(part + (size_t)(rec0 + w * qt) * rec, smem + S::kVOff, (uint32_t)(qt * rec));
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(stg_free);
        ++it;
      }
      bulk_wait_all();
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kBk);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, false, true);
      const uint32_t q_base = smem_u32(smem + S::kQOff);
      const uint32_t k_base = smem_u32(smem + S::kKOff), v_base = smem_u32(smem + S::kVOff);
      uint32_t it = 0, e = 0;
      bool ok = true;
      for (int64_t w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
        const int cnt = sh_count(shlist, w);
        if (cnt == 0) continue;
        for (int j = 0; j < cnt; ++j, ++e) {
          // S(j) = Q K(j)^T over the S / P columns, once K(j) has landed and
          // P.V(j - 1), which read them, has completed
          if ((j == 0 && !mbar_wait(q_full, it & 1, abort_flag, dg)) ||
              !mbar_wait(k_full, e & 1, abort_flag, dg) ||
              (e > 0 && !mbar_wait(pv_done, (e - 1) & 1, abort_flag, dg))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int c = kk / 4, off = (kk % 4) * 32;
            mma_bf16_ss(tmem_base, desc_kmajor_sw128(q_base + c * kTileRows * 128 + off),
                        desc_kmajor_sw128(k_base + c * kBk * 128 + off), idesc_s,
                        kk > 0 ? 1u : 0u);
          }
          mma_commit(s_full);
          mma_commit(k_empty);
          if (j + 1 == cnt) mma_commit(q_empty);
          // O += P(j) V(j), once the softmax has written P(j), V(j) has landed
          // and (first block) the previous item's epilogue has read O
          if (!mbar_wait(p_full, e & 1, abort_flag, dg) ||
              (j == 0 && it > 0 && !mbar_wait(o_free, (it - 1) & 1, abort_flag, dg)) ||
              !mbar_wait(v_full, e & 1, abort_flag, dg)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBk / 16; ++kk) {
            const uint64_t bd = desc_mnmajor_sw128(v_base + kk * 16 * 128, kBk * 128);
            mma_bf16_ts(tmem_base + 128, tmem_base + (uint32_t)(kk * 8), bd, idesc_o,
                        (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(v_empty);
          mma_commit(pv_done);
          if (j + 1 == cnt) mma_commit(o_full);
        }
        ++it;
      }
      // every MMA issued by this thread has completed once done_bar flips
      mma_commit(done_bar);
      mbar_drain(done_bar, 0);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 208;\n" ::: "memory");
    // ------------------------------------------------------------ softmax + epilogue
    const int qq = warp & 3;
    const int row = qq * 32 + lane;
    const int qi = row / G, hi = row % G;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const uint32_t ts = tmem_base + lane_off;
    const uint32_t srow = smem_u32(smem + S::kVOff) + (uint32_t)(qi * rec + hi * D * 2);
    uint32_t e = 0, it = 0;
    bool ok = true;
    for (int64_t w = blockIdx.x; w < n_items && ok; w += gridDim.x) {
      const int cnt = sh_count(shlist, w);
      if (cnt == 0) continue;
      const int g = (int)(w % n_g);
      const int64_t t = q0 + (w / n_g) * qt + qi;
      const bool valid = t < q1;
      const uint32_t sel = valid ? (uint32_t)rowmask[(t - q0) * n_g + g] >> 16 : 0u;
      const int64_t loc = t / kBk;
      float m = -INFINITY, l = 0.f;  // running max (log2 units) used for P, and sum
      for (int j = 0; j < cnt; ++j, ++e) {
        const int b = shlist[w * kShMax + j];
        const int lim = ((sel >> j) & 1) ? (b == loc ? (int)(t - (int64_t)b * kBk) + 1 : kBk) : 0;
        int got = 0;
        if (lane == 0) got = mbar_wait(s_full, e & 1, abort_flag, dg);
        if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
        tc_fence_after();
        // every row takes all of the block or none of it, unless it is the
        // rows' local block: then the row max comes with the loads
        const bool whole = !__any_sync(0xffffffffu, lim > 0 && lim < kBk);
        uint32_t r[128];
        float mx;
        if (whole) {
          float m0, m1, m2, m3;
          tmem_ld32_max(ts, *reinterpret_cast<uint32_t(*)[32]>(&r[0]), m0);
          tmem_ld32_max(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]), m1);
          tmem_ld32_max(ts + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]), m2);
          tmem_ld32_max(ts + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]), m3);
          tmem_ld_wait();
          mx = lim > 0 ? fmaxf(fmax3(m0, m1, m2), m3) : -INFINITY;
        } else {
          tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
          tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
          tmem_ld32(ts + 64, *reinterpret_cast<uint32_t(*)[32]>(&r[64]));
          tmem_ld32(ts + 96, *reinterpret_cast<uint32_t(*)[32]>(&r[96]));
          tmem_ld_wait();
          mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c < lim) mx = fmaxf(mx, __uint_as_float(r[c]));
        }
        const float mb = mx * scale_log2;  // -inf when the row takes nothing here
        const bool grow = lim > 0 && m > -INFINITY && mb > m + 8.f;
        if (__any_sync(0xffffffffu, grow)) {
          // rescale the O rows whose max grows by more than 8
          const float f = grow ? ex2_approx(m - mb) : 1.f;
          const uint64_t f2 = f2_pack(f, f);
#pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32(ts + 128 + c, o);
            tmem_ld_wait();
#pragma unroll
            for (int x = 0; x < 32; x += 2) {
              float x0, x1;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(o[x]), __uint_as_float(o[x + 1])), f2), x0,
                        x1);
              o[x] = __float_as_uint(x0);
              o[x + 1] = __float_as_uint(x1);
            }
            tmem_st32(ts + 128 + c, o);
          }
          tmem_st_wait();
          l *= f;
          if (grow) m = mb;
        }
        if (lim > 0 && m == -INFINITY) m = mb;  // the row's first block
        // P = exp2(s * c - m); a row that takes nothing here gets exp2(-inf) = 0
        const float nm = lim > 0 ? -m : -INFINITY;
        const uint64_t sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(nm, nm);
        uint64_t l2 = f2_pack(0.f, 0.f);
#pragma unroll
        for (int c2 = 0; c2 < 64; ++c2) {
          float p0, p1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(r[2 * c2]), __uint_as_float(r[2 * c2 + 1])), sc2,
                           nm2), p0, p1);
          p0 = ex2_approx(p0);
          p1 = ex2_approx(p1);
          if (!whole) {
            p0 = 2 * c2 < lim ? p0 : 0.f;
            p1 = 2 * c2 + 1 < lim ? p1 : 0.f;
          }
          l2 = f2_add(l2, f2_pack(p0, p1));
          r[c2] = pack_bf16x2(p0, p1);
        }
        float l0, l1;
        f2_unpack(l2, l0, l1);
        l += l0 + l1;
        tmem_st32(ts, *reinterpret_cast<const uint32_t(*)[32]>(&r[0]));
        tmem_st32(ts + 32, *reinterpret_cast<const uint32_t(*)[32]>(&r[32]));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok) break;
      // the item's records: O / l in bf16 and the LSE of this thread's (query,
      // head), staged in the V buffer (its last P.V has completed)
      int got = 0;
      if (lane == 0) got = mbar_wait(o_full, it & 1, abort_flag, dg);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      tc_fence_after();
      uint32_t o[D];
#pragma unroll
      for (int c = 0; c < D; c += 32)
        tmem_ld32(ts + 128 + c, *reinterpret_cast<uint32_t(*)[32]>(&o[c]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint64_t inv2 = f2_pack(inv, inv);
#pragma unroll
      for (int v = 0; v < D / 8; ++v) {
        uint32_t wv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float x0, x1;
          f2_unpack(f2_mul(f2_pack(__uint_as_float(o[8 * v + 2 * u]),
                                   __uint_as_float(o[8 * v + 2 * u + 1])), inv2), x0, x1);
          wv[u] = pack_bf16x2(x0, x1);
        }
        st_shared_v4(srow + v * 16, wv[0], wv[1], wv[2], wv[3]);
      }
      *reinterpret_cast<float*>(smem + S::kVOff + qi * rec + G * D * 2 + hi * 4) =
          (m + __log2f(l)) * 0.69314718055994531f;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(stg_full);
      ++it;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 256);
}

// ---------------------------------------------------------------------- merge
// partials: one record per (query, group, slot) holding the G heads' O rows
// (bf16) and then their LSEs, found through rec_of (-1: the slot has none).
// Each half warp merges one (query, head): lane s < k holds slot s's LSE, max
// and sum come from shuffles within the half, and the k slot loads (16 bytes
// per lane for D = 128) are all issued before they are summed. The two halves
// take adjacent heads, so with G > 1 each slot read is one contiguous
// 2 * D * 2-byte run.
template <int D>
__global__ void __launch_bounds__(256)
attn_merge_kernel(const unsigned char* __restrict__ part, const int32_t* __restrict__ rec_of,
                  int64_t q0, int64_t q1, int H_q, int H_kv, int k, uint16_t* __restrict__ out,
                  float* __restrict__ lse) {
  constexpr int PER = D / 16;  // elements per lane (8 or 4)
  const int lane = threadIdx.x & 31;
  const int hl = lane & 15;          // lane within the half warp
  const int G = H_q / H_kv;
  const int rec = attn_rec_bytes(G, D);
  const int64_t n = (q1 - q0) * H_q;
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; 2 * w < n; w += warps) {
    const int64_t task = 2 * w + (lane >> 4);
    const bool active = task < n;
    const int64_t tk = active ? task : n - 1;
    const int64_t tl = tk / H_q;
    const int h = (int)(tk % H_q);
    const int g = h / G, hi = h % G;
    const int64_t t = q0 + tl;
    const int ri = hl < k ? rec_of[((size_t)tl * H_kv + g) * k + hl] : -1;
    const bool valid = ri >= 0;
    const float ls =
        valid ? *reinterpret_cast<const float*>(part + (size_t)ri * rec + G * D * 2 + hi * 4)
              : -INFINITY;
    float M = ls;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off, 16));
    const float wl = valid ? __expf(ls - M) : 0.f;
    float L = wl;
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off, 16);
    const int col = (hi * D + hl * PER) * 2;  // this lane's bytes within a record
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= k) break;
      const float wgt = __shfl_sync(0xffffffffu, wl, s, 16);
      const int rs = __shfl_sync(0xffffffffu, ri, s, 16);
      if (wgt == 0.f) continue;  // invalid or padded slot
      const unsigned char* po = part + (size_t)rs * rec + col;
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

// Group merge: one warp per (query, group) reads each selected slot's whole
// record (the G heads' o/l rows are contiguous, so a slot is one G*D*2-byte
// run) and writes the group's G output rows, which are contiguous as well.
// Lane l covers the E = G*D/32 elements starting at l*E (head l*E/D). Lane
// s < k holds slot s's record index and LSEs; per head, max and sum come from
// shuffles over the slots. Used when G*D <= 1024.
// six CTAs per SM (40 registers, a few spilled): the merge waits on memory, and
// more warps per SM took the 128K main branch from 9.09 ms (four CTAs, 58
// registers) to 8.87 (five) and 8.77 (six); at seven or eight CTAs the kernel
// drops to 32 registers and spills ten times as much, so those were not timed
template <int D, int E>
__global__ void __launch_bounds__(256, 6)
attn_merge_group_kernel(const unsigned char* __restrict__ part,
                        const int32_t* __restrict__ rec_of, int64_t q0, int64_t q1, int H_q,
                        int H_kv, int k, uint16_t* __restrict__ out, float* __restrict__ lse) {
  constexpr int G = 32 * E / D;
  constexpr int kRec = G * D * 2 + (G + 3) / 4 * 16;
  static_assert(G >= 1 && 32 * E == G * D, "group merge needs G*D a multiple of 32");
  const int lane = threadIdx.x & 31;
  const int hi = lane * E / D;  // this lane's head within the group
  const int64_t n = (q1 - q0) * H_kv;
  const int64_t warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < n; w += warps) {
    const int64_t tl = w / H_kv;
    const int g = (int)(w % H_kv);
    const int ri = lane < k ? rec_of[((size_t)tl * H_kv + g) * k + lane] : -1;
    float wl[G], M[G], L[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float ls = ri >= 0 ? *reinterpret_cast<const float*>(part + (size_t)ri * kRec +
                                                                 G * D * 2 + h * 4)
                               : -INFINITY;
      float m = ls;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      const float e = ri >= 0 ? __expf(ls - m) : 0.f;
      float s = e;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      wl[h] = e;
      M[h] = m;
      L[h] = s;
    }
    float acc[E];
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxK; ++s) {
      if (s >= k) break;
      const int rs = __shfl_sync(0xffffffffu, ri, s);
      float wgt = 0.f;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float x = __shfl_sync(0xffffffffu, wl[h], s);
        if (h == hi) wgt = x;
      }
      if (rs < 0) continue;  // padded slot (the same for the whole warp)
      const uint32_t* po = reinterpret_cast<const uint32_t*>(part + (size_t)rs * kRec) + lane * E / 2;
#pragma unroll
      for (int v = 0; v < E / 2; v += (E >= 8 ? 4 : E / 2)) {
        uint32_t wd[4];
        if (E >= 8) {
          const uint4 u = __ldcs(reinterpret_cast<const uint4*>(po + v));
          wd[0] = u.x; wd[1] = u.y; wd[2] = u.z; wd[3] = u.w;
        } else if (E == 4) {
          const uint2 u = __ldcs(reinterpret_cast<const uint2*>(po + v));
          wd[0] = u.x; wd[1] = u.y;
        } else {
          wd[0] = __ldcs(po + v);
        }
#pragma unroll
        for (int j = 0; j < (E >= 8 ? 4 : E / 2); ++j) {
          acc[2 * (v + j)] = fmaf(wgt, bf16_lo(wd[j]), acc[2 * (v + j)]);
          acc[2 * (v + j) + 1] = fmaf(wgt, bf16_hi(wd[j]), acc[2 * (v + j) + 1]);
        }
      }
    }
    float Lh = 0.f, Mh = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h)
      if (h == hi) { Lh = L[h]; Mh = M[h]; }
    const float inv = Lh > 0.f ? 1.f / Lh : 0.f;
    const int64_t t = q0 + tl;
    uint32_t* o = reinterpret_cast<uint32_t*>(out + ((size_t)t * H_q + (size_t)g * G) * D) +
                  lane * E / 2;
#pragma unroll
    for (int v = 0; v < E / 2; v += (E >= 8 ? 4 : E / 2)) {
      if (E >= 8) {
        uint4 u;
        u.x = pack_bf16x2(acc[2 * v + 0] * inv, acc[2 * v + 1] * inv);
        u.y = pack_bf16x2(acc[2 * v + 2] * inv, acc[2 * v + 3] * inv);
        u.z = pack_bf16x2(acc[2 * v + 4] * inv, acc[2 * v + 5] * inv);
        u.w = pack_bf16x2(acc[2 * v + 6] * inv, acc[2 * v + 7] * inv);
        *reinterpret_cast<uint4*>(o + v) = u;
      } else if (E == 4) {
        uint2 u;
        u.x = pack_bf16x2(acc[2 * v + 0] * inv, acc[2 * v + 1] * inv);
        u.y = pack_bf16x2(acc[2 * v + 2] * inv, acc[2 * v + 3] * inv);
        *reinterpret_cast<uint2*>(o + v) = u;
      } else {
        o[v] = pack_bf16x2(acc[2 * v] * inv, acc[2 * v + 1] * inv);
      }
    }
    if (lse && (lane * E) % D == 0) lse[(size_t)t * H_q + g * G + hi] = Mh + logf(Lh);
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

// Pages [P, H, 128, D] bf16 seen through the same (D, H, rows) box as
// make_map_kv: coordinate (x, g, z) with z = page * H * 128 + r addresses row r
// of head g in the page (head stride 128 * D, row stride D elements), so a
// 128-row box at z = page * H * 128 is head g's whole page.
bool make_map_kv_pages(CUtensorMap* m, const void* base, int64_t pages, int H, int D) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess || qr != cudaDriverEntryPointSuccess)
      return false;
    fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)(pages * H * kBk)};
  cuuint64_t strides[2] = {(cuuint64_t)kBk * D * 2, (cuuint64_t)D * 2};
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
cudaError_t launch_tiles(const void* q, const void* kk, const void* v, int64_t N, int64_t kv_rows,
                         int64_t q0, int H_q, int H_kv, int k, float scale_log2, int64_t nb,
                         const AttnWs& ws, const int32_t* tbase, int64_t n_b, const Diag& dg,
                         cudaStream_t st) {
  CUtensorMap tk, tv;
  CUtensorMap tq;
  const bool paged = tbase != nullptr;  // kv_rows = pages * H_kv * 128
  const int64_t pages = kv_rows / ((int64_t)H_kv * kBk);
  if (!(paged ? make_map_kv_pages(&tk, kk, pages, H_kv, D) : make_map_kv(&tk, kk, kv_rows, H_kv, D)) ||
      !(paged ? make_map_kv_pages(&tv, v, pages, H_kv, D) : make_map_kv(&tv, v, kv_rows, H_kv, D)) ||
      !make_map_rows(&tq, q, N * H_q, D))
    return cudaErrorInvalidValue;
  const int smem = AttnSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(attn_tile_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_tile_tc_kernel<D><<<sm_count(), kAttnThreads, smem, st>>>(
      tk, tv, tq, N * H_q, q0, H_q, H_kv, k, scale_log2, nb, ws.entries, ws.tinfo, tbase,
      ws.tile_off + n_b, ws.part, dg);
  return cudaGetLastError();
}

// Q [N, H_q, D] seen as (D, H_q, N) with a box of all G heads of qt queries
bool make_map_q_tile(CUtensorMap* m, const void* base, int64_t N, int H_q, int D, int G, int qt) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess || qr != cudaDriverEntryPointSuccess)
      return false;
    fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H_q, (cuuint64_t)N};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H_q * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)qt};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_shared(const void* q, const void* kk, const void* v, int64_t N, int64_t q0,
                          int64_t q1, int H_q, int H_kv, float scale_log2, const AttnWs& ws,
                          const Diag& dg, cudaStream_t st) {
  const int G = H_q / H_kv, qt = kTileRows / G;
  CUtensorMap tq, tk, tv;
  if (!make_map_q_tile(&tq, q, N, H_q, D, G, qt) || !make_map_kv(&tk, kk, N, H_kv, D) ||
      !make_map_kv(&tv, v, N, H_kv, D))
    return cudaErrorInvalidValue;
  const int smem = ShSmem<D>::kBytes;
  cudaError_t e = cudaFuncSetAttribute(attn_shared_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t n_items = (q1 - q0 + qt - 1) / qt * H_kv;
  attn_shared_tc_kernel<D><<<2 * sm_count(), kShThreads, smem, st>>>(tq, tk, tv, q0, q1, H_q, H_kv,
                                                          scale_log2, n_items, ws.shlist,
                                                          ws.rowmask, ws.shared_rec0, ws.part, dg);
  return cudaGetLastError();
}

}  // namespace

// the shared-block pass needs query tiles of at most 32 queries (G >= 4)
inline bool shared_pass(bool with_shared, int H_q, int H_kv) {
  return with_shared && H_q / H_kv >= 4;
}

size_t attn_ws_bytes(int64_t chunk, int64_t nb, int H_q, int H_kv, int d, int k,
                     bool with_tbase, bool with_shared) {
  int64_t n_b = (int64_t)H_kv * nb;
  const int G = H_q / H_kv, qt = kTileRows / G;
  const bool sh = shared_pass(with_shared, H_q, H_kv);
  size_t s = 0;
  s += align256((size_t)n_b * 4);        // counts
  s += align256((size_t)(n_b + 1) * 4);  // offsets
  s += align256((size_t)n_b * 4);        // cursor
  s += align256((size_t)(n_b + 1) * 4);  // tile_off
  if (n_b <= kSmemBucketsMax) s += align256((size_t)kBucketCtas * n_b * 4);  // percta
  s += align256((size_t)chunk * H_kv * k * 4);
  s += align256((size_t)max_tiles(chunk, n_b, H_q, H_kv, k) * 16);
  if (with_tbase) s += align256((size_t)max_tiles(chunk, n_b, H_q, H_kv, k) * 4);
  s += align256((size_t)chunk * H_kv * k * 4);
  if (sh) {
    s += align256((size_t)chunk * H_kv * 4);                                // rowmask
    s += align256((size_t)((chunk + qt - 1) / qt) * H_kv * kShMax * 4);     // shlist
  }
  // block-outer partials, then the shared-block records (qt per item)
  const size_t sh_recs = sh ? (size_t)((chunk + qt - 1) / qt) * H_kv * qt : 0;
  s += align256(((size_t)max_tiles(chunk, n_b, H_q, H_kv, k) * qt + sh_recs) *
                attn_rec_bytes(G, d));
  return s;
}

AttnWs attn_ws_carve(void* ws, int64_t chunk, int64_t nb, int H_q, int H_kv, int d, int k,
                     bool with_tbase, bool with_shared) {
  int64_t n_b = (int64_t)H_kv * nb;
  const int G = H_q / H_kv, qt = kTileRows / G;
  const bool sh = shared_pass(with_shared, H_q, H_kv);
  unsigned char* p = (unsigned char*)ws;
  AttnWs w;
  w.counts = (int32_t*)p;   p += align256((size_t)n_b * 4);
  w.offsets = (int32_t*)p;  p += align256((size_t)(n_b + 1) * 4);
  w.cursor = (int32_t*)p;   p += align256((size_t)n_b * 4);
  w.tile_off = (int32_t*)p; p += align256((size_t)(n_b + 1) * 4);
  w.percta = nullptr;
  if (n_b <= kSmemBucketsMax) {
    w.percta = (int32_t*)p;
    p += align256((size_t)kBucketCtas * n_b * 4);
  }
  w.entries = (int32_t*)p;  p += align256((size_t)chunk * H_kv * k * 4);
  w.tinfo = (int4*)p;       p += align256((size_t)max_tiles(chunk, n_b, H_q, H_kv, k) * 16);
  w.tbase = nullptr;
  if (with_tbase) {
    w.tbase = (int32_t*)p;
    p += align256((size_t)max_tiles(chunk, n_b, H_q, H_kv, k) * 4);
  }
  w.rec_of = (int32_t*)p;   p += align256((size_t)chunk * H_kv * k * 4);
  if (sh) {
    w.rowmask = (int32_t*)p;  p += align256((size_t)chunk * H_kv * 4);
    w.shlist = (int32_t*)p;   p += align256((size_t)((chunk + qt - 1) / qt) * H_kv * kShMax * 4);
    w.shared_rec0 = max_tiles(chunk, n_b, H_q, H_kv, k) * qt;
  }
  w.part = p;
  return w;
}

cudaError_t launch_bucketing(const int32_t* ids, int64_t q0, int64_t q1, int H_q, int H_kv,
                             int k, const AttnWs& ws, int64_t nb, const Diag& dg, cudaStream_t st,
                             const AttnBatch& bt) {
  const int64_t n_b = (int64_t)H_kv * nb;
  const int32_t* tbase = bt.paged ? ws.tbase : nullptr;
  if (bt.paged && !tbase) return cudaErrorInvalidValue;
  const int G = H_q / H_kv;
  const int qt = kTileRows / G;
  note_launches(n_b <= kSmemBucketsMax ? 6 : 5);  // memset, count, scan, (base,) fill, map
  cudaError_t e = cudaMemsetAsync(ws.counts, 0, (size_t)n_b * 4, st);
  if (e != cudaSuccess) return e;
  if (ws.rowmask) {  // blocks shared by the query tiles leave the block-outer buckets
    note_launches(1);
    const int64_t n_qt = (q1 - q0 + qt - 1) / qt;
    const int64_t warps = n_qt * H_kv;
    shared_sets_kernel<<<(unsigned)std::min<int64_t>((warps * 32 + 255) / 256, 152 * 32), 256, 0,
                         st>>>(ids, q0, q1, H_kv, k, qt, n_qt, ws.shlist, ws.rowmask, ws.rec_of,
                               ws.shared_rec0);
  }
  int64_t n = (q1 - q0) * H_kv * k;
  const bool smem_buckets = n_b <= kSmemBucketsMax;
  unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 32);
  if (smem_buckets)
    bucket_count_smem_kernel<<<kBucketCtas, 1024, n_b * 4, st>>>(
        ids, q0, q1, H_kv, k, nb, bt.qinfo, ws.rowmask, ws.counts, ws.percta, ws.rec_of, dg);
  else
    bucket_count_kernel<<<grid, 256, 0, st>>>(ids, q0, q1, H_kv, k, nb, bt.qinfo, ws.rowmask,
                                              ws.counts, ws.rec_of, dg);
  bucket_scan_kernel<<<1, 1024, 0, st>>>(ws.counts, n_b, qt, ws.offsets, ws.tile_off, ws.cursor);
  if (smem_buckets) {
    bucket_cta_base_kernel<<<(unsigned)std::min<int64_t>((n_b * 32 + 255) / 256, 152 * 32),
                             256, 0, st>>>(ws.offsets, (int)n_b, kBucketCtas, ws.percta);
    bucket_fill_smem_kernel<<<kBucketCtas, 1024, n_b * 4, st>>>(
        ids, q0, q1, H_kv, k, nb, bt.qinfo, ws.rowmask, qt, ws.offsets, ws.tile_off, ws.percta,
        ws.entries, ws.rec_of);
  } else {
    bucket_fill_kernel<<<grid, 256, 0, st>>>(ids, q0, q1, H_kv, k, nb, bt.qinfo, ws.rowmask, qt,
                                             ws.offsets, ws.tile_off, ws.cursor, ws.entries,
                                             ws.rec_of);
  }
  const int64_t tiles_max = max_tiles(q1 - q0, n_b, H_q, H_kv, k);
  tile_map_kernel<<<(unsigned)std::min<int64_t>((tiles_max + 255) / 256, 152 * 16), 256, 0, st>>>(
      ws.tile_off, ws.offsets, n_b, nb, qt, bt.vinfo, const_cast<int32_t*>(tbase), ws.tinfo);
  return cudaGetLastError();
}

cudaError_t launch_sparse_attn_chunk(const void* q, const void* kk, const void* v,
                                     const int32_t* ids, int64_t N, int64_t q0, int64_t q1,
                                     int H_q, int H_kv, int d, int k, float scale, void* out,
                                     float* lse, const AttnWs& ws, int64_t nb, const Diag& dg,
                                     cudaStream_t st, const AttnBatch& bt) {
  const int64_t n_b = (int64_t)H_kv * nb;
  const int32_t* tbase = bt.paged ? ws.tbase : nullptr;
  const int G = H_q / H_kv;
  cudaError_t e = launch_bucketing(ids, q0, q1, H_q, H_kv, k, ws, nb, dg, st, bt);
  if (e != cudaSuccess) return e;
  note_launches(2);  // tile, merge
  const float scale_log2 = scale * 1.4426950408889634f;
  const int64_t kv_rows = bt.kv_rows > 0 ? bt.kv_rows : N;
  e = d == 128 ? launch_tiles<128>(q, kk, v, N, kv_rows, q0, H_q, H_kv, k, scale_log2, nb, ws,
                                   tbase, n_b, dg, st)
               : launch_tiles<64>(q, kk, v, N, kv_rows, q0, H_q, H_kv, k, scale_log2, nb, ws,
                                  tbase, n_b, dg, st);
  if (e != cudaSuccess) return e;
  if (ws.rowmask) {
    note_launches(1);
    e = d == 128 ? launch_shared<128>(q, kk, v, N, q0, q1, H_q, H_kv, scale_log2, ws, dg, st)
                 : launch_shared<64>(q, kk, v, N, q0, q1, H_q, H_kv, scale_log2, ws, dg, st);
    if (e != cudaSuccess) return e;
  }
  if (G * d <= 1024) {
    const int64_t nw = (q1 - q0) * H_kv;  // one warp per (query, group)
    const unsigned mg = (unsigned)std::min<int64_t>((nw * 32 + 255) / 256, 152 * 64);
    const int E = G * d / 32;
    auto* o16 = (uint16_t*)out;
#define MSA_MERGE_G(DD, EE)                                                                   \
  attn_merge_group_kernel<DD, EE><<<mg, 256, 0, st>>>(ws.part, ws.rec_of, q0, q1, H_q, H_kv, k, \
                                                      o16, lse)
    if (d == 128) {
      if (E == 4) MSA_MERGE_G(128, 4);
      else if (E == 8) MSA_MERGE_G(128, 8);
      else if (E == 16) MSA_MERGE_G(128, 16);
      else MSA_MERGE_G(128, 32);
    } else {
      if (E == 2) MSA_MERGE_G(64, 2);
      else if (E == 4) MSA_MERGE_G(64, 4);
      else if (E == 8) MSA_MERGE_G(64, 8);
      else if (E == 16) MSA_MERGE_G(64, 16);
      else MSA_MERGE_G(64, 32);
    }
#undef MSA_MERGE_G
  } else {
    int64_t nw = (q1 - q0) * H_q;
    unsigned mg = (unsigned)std::min<int64_t>((nw * 16 + 255) / 256, 152 * 64);
    if (d == 128)
      attn_merge_kernel<128><<<mg, 256, 0, st>>>(ws.part, ws.rec_of, q0, q1, H_q, H_kv, k,
                                                 (uint16_t*)out, lse);
    else
      attn_merge_kernel<64><<<mg, 256, 0, st>>>(ws.part, ws.rec_of, q0, q1, H_q, H_kv, k,
                                                (uint16_t*)out, lse);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------ batch geometry
// grid (sequences, slices): slice y of sequence s writes every gridDim.y-th
// query and block of s
__global__ void batch_info_kernel(const __grid_constant__ BatchSeqs tb,
                                  const int32_t* __restrict__ page_table, int page_rows,
                                  int2* __restrict__ qinfo, int2* __restrict__ vinfo) {
  const int s = blockIdx.x;
  const int step = gridDim.y * blockDim.x;
  const int first = blockIdx.y * blockDim.x + threadIdx.x;
  const int vb = tb.vb[s], q_start = tb.q_start[s], q_off = tb.q_off[s];
  for (int i = first; i < tb.q_len[s]; i += step) qinfo[q_start + i] = make_int2(vb, q_off + i);
  for (int b = first; b < tb.n_blk[s]; b += step) {
    const int row = page_table ? page_table[tb.kv_start[s] + b] * page_rows
                               : tb.kv_start[s] + b * kBk;
    vinfo[vb + b] = make_int2(row, q_start - q_off + b * kBk);
  }
}

cudaError_t launch_batch_info(const BatchSeqs& tb, const int32_t* page_table, int page_rows,
                              int2* qinfo, int2* vinfo, cudaStream_t st) {
  if (tb.B <= 0) return cudaSuccess;
  note_launches(1);
  batch_info_kernel<<<dim3((unsigned)tb.B, 16), 256, 0, st>>>(tb, page_table, page_rows, qinfo,
                                                              vinfo);
  return cudaGetLastError();
}

}  // namespace msa
