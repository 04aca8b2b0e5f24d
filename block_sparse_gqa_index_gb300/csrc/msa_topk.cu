// Exp-free top-k over MSA block scores.
//
// "MiniMax Sparse Attention (MSA): a Two-Branch Block-Sparse Attention Trained
// on a 109B-Parameter MoE With a 3T-Token Budget", section "内核协同设计"
// (kernel co-design): softmax preserves order, so the blocks are ranked on their
// raw max-pooled scores, with no max / exp / sum pass. Selection rule from
// "两个分支如何工作": the query's local block is always kept and the other k-1
// slots take the best earlier blocks; lower block id wins ties.
//
// Each 16-lane half of a warp ranks one (query, group) row, so every shuffle,
// compare and select of the sorting networks below serves two rows. A row's
// candidates (blocks 0 .. loc-1) are streamed in chunks of 512 scores, 32 per
// lane, read with 16-byte loads; the half's next chunk (of this row or of its
// next row) is already loading while the current one is ranked. Per chunk:
//   1. the values are staged in the half's shared buffer, and every lane takes
//      the max of its even and of its odd blocks (32 group maxima per row);
//   2. tau = max((k-1)-th largest group max, worst key kept so far): at least
//      k-1 keys are >= tau, so no key below tau can be in the answer. The group
//      maxima are taken as two lists of 16 (even, odd), each bitonic-sorted
//      across the half, and tau read off their merge. Once both rows of the
//      warp keep k-1 keys, the worst kept key alone is tried first, and the
//      group maxima are needed only when more than 32 values reach it;
//   3. the keys >= tau (typically 15-30) are compacted into shared memory (each
//      lane reads its survivors back from its staged values); every survivor
//      counts the survivors that beat it (on the fp32 scores when no two are
//      equal, else on the 64-bit keys), and the k-1 with the lowest counts are
//      kept, one per lane, in descending order. More than 32 survivors in
//      either half send both halves through k-1 rounds of arg-max instead.
// Finally the kept ids plus the local block are sorted ascending and written.
// Blocks past the candidates read as NaN, which no comparison keeps and which
// max.f32 ignores (inputs themselves must be finite).
#include <algorithm>
#include <climits>

#include "msa_kernels.h"

namespace msa {
namespace {

constexpr int kWarps = 4;
constexpr int kHalf = 512;  // candidates per half-warp chunk: 32 per lane
constexpr int kCap = 32;    // survivors of a row sorted in the fast path
constexpr unsigned kAll = 0xffffffffu;

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
  uint32_t lo = __shfl_xor_sync(kAll, (uint32_t)v, m);
  uint32_t hi = __shfl_xor_sync(kAll, (uint32_t)(v >> 32), m);
  return ((uint64_t)hi << 32) | lo;
}
// value of lane src of this lane's half
__device__ __forceinline__ uint64_t shfl64_h(uint64_t v, int src) {
  uint32_t lo = __shfl_sync(kAll, (uint32_t)v, src, 16);
  uint32_t hi = __shfl_sync(kAll, (uint32_t)(v >> 32), src, 16);
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

// The kfar-th largest (1 <= kfar <= 15) of the 32 floats a half holds 2 per
// lane. a (one per lane) is bitonic-sorted descending and b ascending across the
// half; the kfar-th largest of the union of two sorted lists is the largest,
// over the splits i + j = kfar, of min(i-th largest of a, j-th largest of b),
// with the 0-th largest read as +inf. Lane hl takes the split i = hl + 1 (and
// lane kfar the split i = 0), then a max over the half. Returned in every lane.
__device__ __forceinline__ float kth_largest32h(float a, float b, int kfar, int hl) {
#pragma unroll
  for (int size = 2; size <= 16; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const float pa = __shfl_xor_sync(kAll, a, stride);
      const float pb = __shfl_xor_sync(kAll, b, stride);
      const bool low_min = ((hl & stride) == 0) == ((hl & size) == 0);  // ascending: lower lane keeps the min
      a = low_min ? fmaxf(a, pa) : fminf(a, pa);
      b = low_min ? fminf(b, pb) : fmaxf(b, pb);
    }
  // b ascending: its j-th largest (1-based) sits in half-lane 16 - j
  const int src = hl <= kfar - 2 ? 17 - kfar + hl : 16 - kfar;
  const float bs = __shfl_sync(kAll, b, src, 16);
  float t = hl <= kfar - 2 ? fminf(a, bs) : hl == kfar - 1 ? a : hl == kfar ? bs : -INFINITY;
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) t = fmaxf(t, __shfl_xor_sync(kAll, t, off));
  return t;
}

// bitonic sort of one int per lane within each 16-lane half, ascending
__device__ __forceinline__ int sort16h_asc(int a, int hl) {
#pragma unroll
  for (int size = 2; size <= 16; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int p = __shfl_xor_sync(kAll, a, stride);
      const bool up = (hl & size) == 0;
      const bool lower = (hl & stride) == 0;
      a = (lower == up) ? min(a, p) : max(a, p);
    }
  return a;
}

// Loads a half's chunk (p = first candidate of the chunk, rem = candidates left
// in the row from there): lane value 4 i + e is candidate 64 i + 4 hl + e;
// candidates at or past rem read as NaN. VEC: p is 16-byte aligned.
template <bool VEC>
__device__ __forceinline__ void load_chunk(float (&v)[32], const float* __restrict__ p, int rem,
                                           int hl) {
  const float nan = __int_as_float(0x7fffffff);
  if (VEC && rem >= kHalf) {  // a whole chunk: no masking
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 x = __ldcs(reinterpret_cast<const float4*>(p + i * 64 + hl * 4));
      v[4 * i + 0] = x.x;
      v[4 * i + 1] = x.y;
      v[4 * i + 2] = x.z;
      v[4 * i + 3] = x.w;
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int o = i * 64 + hl * 4;
    float4 x = make_float4(nan, nan, nan, nan);
    if (o < rem) {
      if constexpr (VEC) {
        // the whole vector is in the row (rows hold a multiple of 4 scores);
        // the blocks past the candidates are masked by selects, not branches
        x = __ldcs(reinterpret_cast<const float4*>(p + o));
        const int nv = rem - o;
        x.y = nv > 1 ? x.y : nan;
        x.z = nv > 2 ? x.z : nan;
        x.w = nv > 3 ? x.w : nan;
      } else {
        x.x = p[o];
        if (o + 1 < rem) x.y = p[o + 1];
        if (o + 2 < rem) x.z = p[o + 2];
        if (o + 3 < rem) x.w = p[o + 3];
      }
    }
    v[4 * i + 0] = x.x;
    v[4 * i + 1] = x.y;
    v[4 * i + 2] = x.z;
    v[4 * i + 3] = x.w;
  }
}

// Row cursor of one half: row r = q * n_g + g walks by a fixed stride, and its
// query index q follows without a division per step.
struct RowCursor {
  uint32_t r;  // rows number at most INT_MAX, so r + stride stays below 2^32
  int q, rm;   // r / n_g, r % n_g
  __device__ __forceinline__ void step(uint32_t stride, int sq, int sr, int n_g) {
    r += stride;
    q += sq;
    rm += sr;
    if (rm >= n_g) {
      rm -= n_g;
      ++q;
    }
  }
};

// Local block of the cursor's row (its query's position / Bk), or -1 when that
// position lies outside the score rows.
__device__ __forceinline__ int row_loc(const RowCursor& c, int Bk, int bk_shift, int64_t nb,
                                       int64_t q_offset, const int32_t* __restrict__ seq_lens) {
  const int64_t pos = seq_lens ? (int64_t)seq_lens[c.q] - 1 : c.q + q_offset;
  if (pos < 0) return -1;
  const int64_t loc = bk_shift >= 0 ? pos >> bk_shift : pos / Bk;
  return loc < nb ? (int)loc : -1;
}

// Ranks each half's staged chunk (sv) into the kfar best keys the half kept so
// far (best: half-lane i < kfar holds the i-th best, descending). m0, m1: the
// lane's two group maxima.
// survivor mask of the lane's staged values (>= tau; ties at tau are kept and
// settled by the keys), the kept entries >= tau, and the half's prefix count
__device__ __forceinline__ void survivors(const float4* sv, float tau, int kfar, int hl,
                                          uint64_t best, uint32_t& mask, bool& keep_old,
                                          int& cnt, int& incl, int& total) {
  mask = 0;
#pragma unroll 2
  for (int i = 0; i < 8; ++i) {
    const float4 x = sv[i * 16 + hl];
    const uint32_t m4 = (x.x >= tau ? 1u : 0u) | (x.y >= tau ? 2u : 0u) |
                        (x.z >= tau ? 4u : 0u) | (x.w >= tau ? 8u : 0u);
    mask |= m4 << (4 * i);
  }
  keep_old = hl < kfar && best != 0 && key_value(best) >= tau;
  cnt = __popc(mask) + (keep_old ? 1 : 0);
  incl = cnt;
#pragma unroll
  for (int off = 1; off < 16; off <<= 1) {
    const int y = __shfl_up_sync(kAll, incl, off, 16);
    if (hl >= off) incl += y;
  }
  total = __shfl_sync(kAll, incl, 15, 16);
}

__device__ __forceinline__ void rank_chunk(const float4* sv, float m0, float m1, float* vb,
                                           int* ib, int c0, int kfar, int hl, uint64_t& best,
                                           float& best_min) {
  uint32_t mask;
  bool keep_old;
  int cnt, incl, total;
  // once both halves keep kfar entries, their worst kept score is a threshold
  // of its own (kfar values reach it); the group maxima below are needed only
  // when too many of the chunk's values reach it
  bool settled = false;
  if (__all_sync(kAll, best_min > -INFINITY)) {
    survivors(sv, best_min, kfar, hl, best, mask, keep_old, cnt, incl, total);
    settled = !__any_sync(kAll, total > kCap);
  }
  if (!settled) {
    // threshold: the kfar-th largest group max (>= kfar values reach it) or the
    // worst value kept so far, whichever is larger
    const float tau = fmaxf(kth_largest32h(m0, m1, kfar, hl), best_min);
    survivors(sv, tau, kfar, hl, best, mask, keep_old, cnt, incl, total);
  }
  const float* svf = reinterpret_cast<const float*>(sv);
  if (!__any_sync(kAll, total > kCap)) {
    const float nan = __int_as_float(0x7fffffff);
    int p = incl - cnt;
    if (keep_old) {
      vb[p] = key_value(best);
      ib[p++] = key_id(best);
    }
    while (mask) {  // this lane's survivors, read back from its own staged values
      const int j = __ffs(mask) - 1;
      mask &= mask - 1;
      const int e = (j >> 2) * 64 + hl * 4 + (j & 3);
      vb[p] = svf[e];
      ib[p++] = c0 + e;
    }
    if (hl < 4) vb[total + hl] = nan;  // pads the last vector of the loop below
    __syncwarp();
    const float f0 = hl < total ? vb[hl] : nan;
    const float f1 = hl + 16 < total ? vb[hl + 16] : nan;
    const int i0 = ib[hl], i1 = ib[hl + 16];  // read only where hl (+ 16) < total
    // rank of a survivor = how many survivors beat it (keys are distinct, so the
    // ranks are a permutation); the kfar best land in slots 0..kfar-1, descending.
    // Counted on the scores first: with no two equal scores among the survivors,
    // the survivors scoring >= a survivor are exactly those beating it plus
    // itself, and these counts sum to total (total + 1) / 2; equal scores make
    // the sum larger, and then the ranks are counted on the 64-bit keys.
    int r0 = 0, r1 = 0;
    const float4* vb4 = reinterpret_cast<const float4*>(vb);
    for (int j = 0; 4 * j < total; ++j) {
      const float4 y = vb4[j];
      r0 += (y.x >= f0) + (y.y >= f0) + (y.z >= f0) + (y.w >= f0);
      r1 += (y.x >= f1) + (y.y >= f1) + (y.z >= f1) + (y.w >= f1);
    }
    int sum = r0 + r1;  // NaN rows (past total) count 0
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(kAll, sum, off);
    if (__any_sync(kAll, sum != total * (total + 1) / 2)) {
      const uint64_t a0 = hl < total ? rank_key(f0, (uint32_t)i0) : 0;
      const uint64_t a1 = hl + 16 < total ? rank_key(f1, (uint32_t)i1) : 0;
      r0 = 0;
      r1 = 0;
      for (int j = 0; j < total; ++j) {
        const uint64_t y = rank_key(vb[j], (uint32_t)ib[j]);
        r0 += y > a0 ? 1 : 0;
        r1 += y > a1 ? 1 : 0;
      }
    } else {
      --r0;
      --r1;
    }
    __syncwarp();
    if (hl < total && r0 < kfar) {
      vb[r0] = f0;
      ib[r0] = i0;
    }
    if (hl + 16 < total && r1 < kfar) {
      vb[r1] = f1;
      ib[r1] = i1;
    }
    __syncwarp();
    // total >= kfar: tau leaves at least kfar survivors
    best = hl < kfar ? rank_key(vb[hl], (uint32_t)ib[hl]) : 0;
    best_min = vb[kfar - 1];
    __syncwarp();
  } else {
    // rare (heavy ties): extract the kfar best of each half one by one
    uint64_t nb_best = 0, prev = ~0ull;
    const uint64_t old = hl < kfar ? best : 0;
    for (int round = 0; round < kfar; ++round) {
      uint64_t m = old < prev ? old : 0;
      for (uint32_t mm = mask; mm; mm &= mm - 1) {
        const int j = __ffs(mm) - 1;
        const int e = (j >> 2) * 64 + hl * 4 + (j & 3);
        const uint64_t key = rank_key(svf[e], (uint32_t)(c0 + e));
        if (key < prev && key > m) m = key;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) {
        const uint64_t y = shfl_xor64(m, off);
        m = y > m ? y : m;
      }
      if (hl == round) nb_best = m;
      prev = m;
    }
    best = nb_best;
    best_min = key_value(shfl64_h(best, kfar - 1));
  }
}

template <bool VEC>
__global__ void __launch_bounds__(kWarps * 32, 6)
topk_kernel(const float* __restrict__ S, int64_t n_rows, int n_g, int64_t nb, int64_t ld, int Bk,
            int bk_shift, int k, int64_t q_offset, const int32_t* __restrict__ seq_lens,
            int32_t* __restrict__ ids, Diag dg) {
  __shared__ float4 vbuf[kWarps][2][kCap / 4 + 1];  // survivor scores, NaN-padded
  __shared__ int ibuf[kWarps][2][kCap + 1];         // their block ids
  __shared__ float4 sval[kWarps][2][8 * 16];
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int half = lane >> 4, hl = lane & 15;
  const int kfar = k - 1;
  const uint32_t stride = gridDim.x * kWarps * 2;  // rows per sweep (one per half)
  const uint32_t rows = (uint32_t)n_rows;           // at most INT_MAX (host check)
  const int sq = (int)(stride / n_g), sr = (int)(stride % n_g);
  float4* sv = sval[wid][half];
  float* vbf = reinterpret_cast<float*>(vbuf[wid][half]);
  int* ibf = ibuf[wid][half];

  // Moves the cursor to the first row at or after it that needs ranking; rows
  // that need none (position outside the score rows, or no more candidates than
  // far slots) are written on the way by this half. loc_out: that row's local
  // block. The cursor ends at n_rows or beyond when there is none.
  auto seek = [&](RowCursor& c, int& loc_out) {
    for (; c.r < rows; c.step(stride, sq, sr, n_g)) {
      const int loc = row_loc(c, Bk, bk_shift, nb, q_offset, seq_lens);
      int32_t* out = ids + (int64_t)c.r * k;
      if (loc < 0) {  // flag, emit padding
        if (hl == 0) report(dg, kStatusBadIds);
        if (hl < k) out[hl] = -1;
        continue;
      }
      if (loc <= kfar) {  // every visible block is kept
        if (hl < k) out[hl] = hl <= loc ? hl : -1;
        continue;
      }
      loc_out = loc;
      return;
    }
  };

  RowCursor cur;
  cur.r = (blockIdx.x * kWarps + wid) * 2 + half;
  cur.q = (int)(cur.r / n_g);
  cur.rm = (int)(cur.r % n_g);
  int loc = 0, c0 = 0;
  seek(cur, loc);
  float vn[32];
  load_chunk<VEC>(vn, S + (cur.r < rows ? (int64_t)cur.r * ld : 0),
                  cur.r < rows ? min(loc, kHalf) : 0, hl);
  uint64_t best = 0;           // half-lane i < kfar: i-th best key so far, else 0
  float best_min = -INFINITY;  // value of the kfar-th best so far (-inf before any chunk)
  while (__any_sync(kAll, cur.r < rows)) {
    const bool act = cur.r < rows;
    // stage the chunk; group maxima over the lane's even and odd blocks (so a
    // short row's few candidates still give two maxima per lane)
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      sv[i * 16 + hl] = make_float4(vn[4 * i], vn[4 * i + 1], vn[4 * i + 2], vn[4 * i + 3]);
      m0 = fmax3(m0, vn[4 * i], vn[4 * i + 2]);
      m1 = fmax3(m1, vn[4 * i + 1], vn[4 * i + 3]);
    }
    // the half's next work item: this row's next chunk, else its next row's first
    RowCursor nxt = cur;
    int c2 = c0 + kHalf, loc2 = loc;
    if (act && c2 >= loc) {
      nxt.step(stride, sq, sr, n_g);
      seek(nxt, loc2);
      c2 = 0;
    }
    const bool act2 = nxt.r < rows;
    load_chunk<VEC>(vn, S + (act2 ? (int64_t)nxt.r * ld + c2 : 0),
                    act2 ? min(loc2 - c2, kHalf) : 0, hl);
    rank_chunk(sv, m0, m1, vbf, ibf, c0, kfar, hl, best, best_min);
    const bool done = act && c0 + kHalf >= loc;
    if (__any_sync(kAll, done)) {  // kept ids plus the local block, ascending
      int id = hl < kfar ? (best ? key_id(best) : INT_MAX) : (hl == kfar ? loc : INT_MAX);
      id = sort16h_asc(id, hl);
      if (done) {
        if (hl < k) ids[(int64_t)cur.r * k + hl] = id == INT_MAX ? -1 : id;
        best = 0;
        best_min = -INFINITY;
      }
    }
    cur = nxt;
    c0 = c2;
    loc = loc2;
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
                        cudaStream_t st, int64_t ld) {
  if (ld <= 0) ld = nb;
  int64_t n_rows = N * n_g;
  if (n_rows == 0) return cudaSuccess;
  note_launches(1);
  if (k == 1) {
    int64_t g = (n_rows + 255) / 256;
    topk_local_only_kernel<<<(unsigned)(g < 152 * 32 ? g : 152 * 32), 256, 0, st>>>(
        n_rows, n_g, Bk, k, q_offset, seq_lens, ids);
    return cudaGetLastError();
  }
  // persistent: as many CTAs as fit on the device at once
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_kernel<true>, kWarps * 32, 0);
  if (e != cudaSuccess) return e;
  if (n_rows > INT_MAX) return cudaErrorInvalidValue;  // query indexes are 32-bit
  int64_t blocks = (n_rows + 2 * kWarps - 1) / (2 * kWarps);
  blocks = std::min<int64_t>(blocks, (int64_t)sms * std::max(per_sm, 1));
  const int bk_shift = (Bk & (Bk - 1)) == 0 ? __builtin_ctz((unsigned)Bk) : -1;
  const bool vec = (ld % 4) == 0 && ((uintptr_t)S % 16) == 0;
  if (vec)
    topk_kernel<true><<<(unsigned)blocks, kWarps * 32, 0, st>>>(S, n_rows, n_g, nb, ld, Bk,
                                                               bk_shift, k, q_offset, seq_lens,
                                                               ids, dg);
  else
    topk_kernel<false><<<(unsigned)blocks, kWarps * 32, 0, st>>>(S, n_rows, n_g, nb, ld, Bk,
                                                                bk_shift, k, q_offset, seq_lens,
                                                                ids, dg);
  return cudaGetLastError();
}

}  // namespace msa
