// Device helpers shared by the MSA kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace msa {

constexpr int kStatusTimeout = -5;
constexpr int kStatusUnsupported = -2;  // a kernel could not run as launched (did nothing)
constexpr int kStatusBadIds = -1;  // invalid block ids / sequence lengths found on the device
constexpr int kMaxK = 16;        // largest k the kernels are built for
constexpr int kMaxFar = kMaxK - 1;

// Diagnostics every kernel receives: the device error word and the poll limit
// of bounded waits.
struct Diag {
  int* err;
  long long wait_limit;
};

__device__ __forceinline__ void report(const Diag& dg, int code) {
  if (dg.err) atomicCAS(dg.err, 0, code);
}

// ---------------------------------------------------------------- ranking keys
// A block is ranked by the 64-bit key (order-preserving bits of its fp32 score,
// ~block id): a larger key is a better block, and among equal scores the lower
// id has the larger key ("lower id wins"). -0 ranks as +0 (the two scores are
// equal), NaN maps below -inf. Key 0 means "empty slot" and is below every real
// key.
__device__ __forceinline__ uint32_t ord_f32(float f) {
  uint32_t b = __float_as_uint(f);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0u;  // NaN
  if (b == 0x80000000u) b = 0u;                     // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ uint64_t rank_key(float score, uint32_t id) {
  return ((uint64_t)ord_f32(score) << 32) | (uint64_t)(0xFFFFFFFFu - id);
}
__device__ __forceinline__ int key_id(uint64_t key) { return (int)(0xFFFFFFFFu - (uint32_t)key); }

// ------------------------------------------------------- per-row streaming top-k
// Keeps the `kfar` (<= 15) best blocks offered so far, in registers, sorted
// descending by score in the last kfar slots, so the worst kept score is always
// the last slot. The slots before them hold +inf, which nothing displaces, and
// a kept slot not yet filled holds -inf (id -1). An offered block is compared
// with every slot at once and the slots from its place on shift down by one,
// which keeps the dependent chain of an insertion a few instructions long.
// Blocks must be offered in increasing id order: the comparisons are strict,
// so of two equal scores the earlier (lower) id stays ahead, and a later block
// whose score equals the worst kept one does not enter.
struct RowTopK {
  float val[kMaxFar];
  int32_t id[kMaxFar];

  __device__ __forceinline__ void init(int kf) {
#pragma unroll
    for (int i = 0; i < kMaxFar; ++i) {
      val[i] = i < kMaxFar - kf ? INFINITY : -INFINITY;
      id[i] = -1;
    }
  }
  // Cheap pre-test for the hot loop: can this score enter at all?
  __device__ __forceinline__ bool wants(float v) const { return v > val[kMaxFar - 1]; }
  __device__ __forceinline__ void offer(float v, int32_t b) {
    bool gt[kMaxFar];
#pragma unroll
    for (int i = 0; i < kMaxFar; ++i) gt[i] = v > val[i];
#pragma unroll
    for (int i = kMaxFar - 1; i >= 0; --i) {  // slot i - 1 still holds its old entry here
      const bool from_prev = i > 0 && gt[i - 1];
      val[i] = gt[i] ? (from_prev ? val[i - 1] : v) : val[i];
      id[i] = gt[i] ? (from_prev ? id[i - 1] : b) : id[i];
    }
  }
  // Writes the kept blocks plus `local`, ascending, padded with -1, to out[0..k).
  __device__ __forceinline__ void emit(int local, int k, int32_t* out) const {
    int v[kMaxK];
#pragma unroll
    for (int i = 0; i < kMaxFar; ++i) v[i] = id[i] >= 0 ? id[i] : 0x7FFFFFFF;
    v[kMaxK - 1] = local;
    // odd-even transposition sort, fully unrolled (16 elements, 16 rounds)
#pragma unroll
    for (int r = 0; r < kMaxK; ++r) {
#pragma unroll
      for (int i = (r & 1); i + 1 < kMaxK; i += 2) {
        int a = v[i], b = v[i + 1];
        v[i] = min(a, b);
        v[i + 1] = max(a, b);
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxK; ++i)
      if (i < k) out[i] = v[i] == 0x7FFFFFFF ? -1 : v[i];
  }
};

// ------------------------------------------------------------------- misc math
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// two OCP FP4 E2M1 codes (the low nibble first) -> f16x2, exact
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n"
      : "=r"(r)
      : "r"(byte));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

}  // namespace msa
