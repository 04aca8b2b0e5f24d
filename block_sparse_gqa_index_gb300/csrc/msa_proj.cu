// Index-branch projections of MSA: the two projection matrices the index branch
// adds to a GQA layer ("MiniMax Sparse Attention (MSA): a Two-Branch
// Block-Sparse Attention Trained on a 109B-Parameter MoE With a 3T-Token
// Budget", section "两个分支如何工作" / how the two branches work): one gives the
// index-query head of every GQA group, the other the single shared index-key
// head. Read as plain linear maps of the layer input:
//   q_idx[t, g, :] = x[t, :] . W_qidx[g * d_idx .. g * d_idx + d_idx - 1, :]^T
//   k_idx[t, :]    = x[t, :] . W_kidx^T
// with weights in [out, in] layout, bf16 operands, fp32 accumulation and bf16
// outputs (what the index branch consumes).
//
// One persistent tcgen05 GEMM over both weight matrices: tiles of 128 rows of x
// by 256 output columns, the column tiles of W_qidx first and then those of
// W_kidx, all column tiles of a row tile in a row so that the tile's x rows are
// reused from L2. Per CTA:
//   warp 0     TMA producer: per 64-deep K step the x chunk (128 x 64) and the
//              weight chunk (256 x 64, rows past the weight matrix read as
//              zeros) into a 4-stage ring, 128B-swizzled;
//   warp 1     TMEM owner (512 columns: two 256-column accumulators) and MMA
//              issuer: four 128 x 256 x 16 MMAs per K step;
//   warps 4-7  epilogue: each thread owns one row, reads its 256 accumulator
//              columns 32 at a time, rounds them to bf16 and stores the valid
//              ones with 16-byte stores, while the other accumulator fills.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "msa_kernels.h"
#include "msa_sm100.cuh"

namespace msa {
namespace {

using namespace sm100;

constexpr int kBM = 128;       // rows of x per tile
constexpr int kBN = 256;       // output columns per tile
constexpr int kBK = 64;        // K elements per step (one 128-byte swizzle row)
constexpr int kStagesP = 4;
constexpr int kThreadsP = 256;  // 8 warps: producer, MMA, (idle), (idle), epilogue x4

struct ProjSmem {
  static constexpr int kABytes = kBM * 128;  // one K step of x
  static constexpr int kBBytes = kBN * 128;  // one K step of weights
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kBarOff = kStagesP * kStageBytes;
  // full[S], empty[S], t_full[2], t_empty[2], done
  static constexpr int kNumBars = 2 * kStagesP + 5;
  static constexpr int kBytes = kBarOff + kNumBars * 8 + 16;
};

struct ProjShape {
  int64_t N;       // rows of x
  int d_model;     // K
  int n_q;         // columns of q_idx (n_groups * d_idx)
  int n_k;         // columns of k_idx (d_idx)
  int tq, tk;      // column tiles of each output
  int64_t tiles;   // row tiles * (tq + tk)
};

__global__ void __launch_bounds__(kThreadsP, 1)
index_project_kernel(const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_wq,
                     const __grid_constant__ CUtensorMap tm_wk, ProjShape sh,
                     uint16_t* __restrict__ q_out, uint16_t* __restrict__ k_out, Diag dg) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ProjSmem::kBarOff);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStagesP;
  uint64_t* t_full = bars + 2 * kStagesP;
  uint64_t* t_empty = t_full + 2;
  uint64_t* done_bar = t_empty + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + ProjSmem::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesP; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&t_full[s], 1);
      mbar_init(&t_empty[s], 4);  // the four epilogue warps
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_x);
    prefetch_tmap(&tm_wq);
    prefetch_tmap(&tm_wk);
  }
  if (warp == 1) tmem_alloc(tmem_holder, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  const int ct = sh.tq + sh.tk;                  // column tiles per row tile
  const int ksteps = (sh.d_model + kBK - 1) / kBK;
  // tile i: row tile i / ct, column tile i % ct (q tiles first)
  auto tile_cols = [&](int64_t i, int& c0, bool& is_q) {
    const int c = (int)(i % ct);
    is_q = c < sh.tq;
    c0 = (is_q ? c : c - sh.tq) * kBN;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      long long it = 0;
      bool armed[kStagesP];
      uint32_t armed_par[kStagesP];
      for (int s = 0; s < kStagesP; ++s) armed[s] = false;
      bool ok = true;
      for (int64_t i = blockIdx.x; i < sh.tiles && ok; i += gridDim.x) {
        int c0;
        bool is_q;
        tile_cols(i, c0, is_q);
        const int32_t r0 = (int32_t)((i / ct) * kBM);
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const int s = (int)(it % kStagesP);
          const uint32_t par = (uint32_t)((it / kStagesP) & 1);
          if (!mbar_wait(&empty[s], par ^ 1, abort_flag, dg)) { ok = false; break; }
          unsigned char* st = smem + s * ProjSmem::kStageBytes;
          mbar_arrive_expect_tx(&full[s], ProjSmem::kStageBytes);
          tma_load_2d(st, &tm_x, &full[s], ks * kBK, r0);
          tma_load_2d(st + ProjSmem::kABytes, is_q ? &tm_wq : &tm_wk, &full[s], ks * kBK, c0);
          armed[s] = true;
          armed_par[s] = par;
        }
      }
      if (!ok || *abort_flag)  // let issued copies land before shared memory goes
        for (int s = 0; s < kStagesP; ++s)
          if (armed[s]) mbar_drain(&full[s], armed_par[s]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      long long it = 0;
      int64_t n = 0;  // tiles of this CTA
      bool ok = true;
      for (int64_t i = blockIdx.x; i < sh.tiles && ok; i += gridDim.x, ++n) {
        const int acc = (int)(n & 1);
        if (!mbar_wait(&t_empty[acc], (uint32_t)(((n >> 1) & 1) ^ 1), abort_flag, dg)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        for (int ks = 0; ks < ksteps; ++ks, ++it) {
          const int s = (int)(it % kStagesP);
          if (!mbar_wait(&full[s], (uint32_t)((it / kStagesP) & 1), abort_flag, dg)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + s * ProjSmem::kStageBytes);
          const uint32_t b = a + ProjSmem::kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            mma_bf16_ss(d_tmem, desc_kmajor_sw128(a + kk * 32), desc_kmajor_sw128(b + kk * 32),
                        idesc, (ks > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&t_full[acc]);
      }
      // every MMA issued by this thread has completed once done flips
      mma_commit(done_bar);
      mbar_drain(done_bar, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter
    const int row = q * 32 + lane;
    int64_t n = 0;
    for (int64_t i = blockIdx.x; i < sh.tiles; i += gridDim.x, ++n) {
      const int acc = (int)(n & 1);
      int got = 0;
      if (lane == 0) got = mbar_wait(&t_full[acc], (uint32_t)((n >> 1) & 1), abort_flag, dg);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      tc_fence_after();
      int c0;
      bool is_q;
      tile_cols(i, c0, is_q);
      const int64_t r = (i / ct) * kBM + row;
      const int width = is_q ? sh.n_q : sh.n_k;
      uint16_t* dst = (is_q ? q_out : k_out) + r * width + c0;
      const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * kBN);
#pragma unroll 1
      for (int c = 0; c < kBN; c += 32) {
        uint32_t v[32];
        tmem_ld32(taddr + c, v);
        tmem_ld_wait();
        if (r < sh.N && c0 + c < width) {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            w[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
          uint4* o = reinterpret_cast<uint4*>(dst + c);
          // widths are multiples of 8 columns, so a 32-column chunk is whole
          // 16-byte vectors; the chunk is cut at the output's last column
          const int nv = min(4, (width - c0 - c) / 8);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (j < nv) o[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&t_empty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// 2D bf16 tensor [rows, cols] with box {64 columns, box_rows}, 128B swizzle;
// elements outside the tensor read as zeros
bool make_map_bf16(CUtensorMap* m, const void* base, int64_t rows, int cols, int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess || qr != cudaDriverEntryPointSuccess)
      return false;
    fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int proj_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

}  // namespace

cudaError_t launch_index_project(const void* x, const void* w_qidx, const void* w_kidx,
                                 int64_t N, int d_model, int n_g, int d_idx, void* q_idx,
                                 void* k_idx, const Diag& dg, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  ProjShape sh;
  sh.N = N;
  sh.d_model = d_model;
  sh.n_q = n_g * d_idx;
  sh.n_k = d_idx;
  sh.tq = (sh.n_q + kBN - 1) / kBN;
  sh.tk = (sh.n_k + kBN - 1) / kBN;
  sh.tiles = ((N + kBM - 1) / kBM) * (sh.tq + sh.tk);
  CUtensorMap tx, tq, tk;
  if (!make_map_bf16(&tx, x, N, d_model, kBM) || !make_map_bf16(&tq, w_qidx, sh.n_q, d_model, kBN) ||
      !make_map_bf16(&tk, w_kidx, sh.n_k, d_model, kBN))
    return cudaErrorInvalidValue;
  const int smem = ProjSmem::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(index_project_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<int64_t>(sh.tiles, proj_sms());
  note_launches(1);
  index_project_kernel<<<grid, kThreadsP, smem, st>>>(tx, tq, tk, sh, (uint16_t*)q_idx,
                                                      (uint16_t*)k_idx, dg);
  return cudaGetLastError();
}

}  // namespace msa
