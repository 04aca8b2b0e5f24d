/* Seeded synthetic inputs for the MiniMax Sparse Attention (MSA) workloads.
 *
 * This header is the ONLY code shared by the CPU oracle and the GPU path. It
 * holds no step of the method: it turns (seed, tensor id, element index) into
 * an input value, deterministically and bit-identically on host and device.
 *
 *  - counter-based generator: splitmix64 (Steele, Lea, Flood, "Fast splittable
 *    pseudorandom number generators", OOPSLA 2014), applied to a counter;
 *  - "N(0,1)" values: Irwin-Hall sum of 12 uniform 24-bit integers minus 6,
 *    exact in double (k * 2^-24), then one additive offset (a double add, one
 *    rounding) and one round-to-nearest-even to bf16 (or to FP8 E4M3);
 *  - integer values: uniform in {-4..4}, exact in bf16.
 *
 * Every float operation below is a single IEEE operation whose result does not
 * depend on contraction (no a*b+c patterns), so host and device agree bit for
 * bit. Compile host code with -ffp-contract=off all the same.
 */
#ifndef MSA_SYNTH_H
#define MSA_SYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_HD __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

/* tensor ids: each input tensor draws from its own counter stream */
enum {
  SYNTH_T_Q = 1,      /* main-branch queries        [N, H_q, d]     */
  SYNTH_T_K = 2,      /* main-branch keys           [N, H_kv, d]    */
  SYNTH_T_V = 3,      /* main-branch values         [N, H_kv, d]    */
  SYNTH_T_QIDX = 4,   /* index queries              [N, n_g, d_idx] */
  SYNTH_T_KIDX = 5,   /* shared index keys          [N, d_idx]      */
  SYNTH_T_DIR = 6,    /* shared planted sign direction s[c] in {-1,+1} */
  SYNTH_T_PLANT = 7,  /* planted-block draws                         */
  SYNTH_T_PERM = 8    /* page-table permutation draws               */
};

SYNTH_HD uint64_t synth_mix64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}

/* stream key of one tensor */
SYNTH_HD uint64_t synth_key(uint64_t seed, uint64_t tensor) {
  return synth_mix64(synth_mix64(seed) ^ (tensor * 0xD1B54A32D192ED03ull));
}

/* draw number j (0..7) of element idx */
SYNTH_HD uint64_t synth_draw(uint64_t key, uint64_t idx, uint32_t j) {
  return synth_mix64(key + idx * 8ull + (uint64_t)j);
}

/* Irwin-Hall(12) - 6 as an exact double: (sum of 12 u24) * 2^-24 - 6 */
SYNTH_HD double synth_gauss(uint64_t key, uint64_t idx) {
  int64_t s = 0;
  for (uint32_t j = 0; j < 6; ++j) {
    uint64_t u = synth_draw(key, idx, j);
    s += (int64_t)(u & 0xFFFFFFull);
    s += (int64_t)((u >> 24) & 0xFFFFFFull);
  }
  s -= 6ll * 16777216ll;
  return (double)s * (1.0 / 16777216.0); /* exact: |s| < 2^27 */
}

/* uniform integer in {-4, ..., 4} */
SYNTH_HD int synth_int9(uint64_t key, uint64_t idx) {
  return (int)(synth_draw(key, idx, 0) % 9ull) - 4;
}

/* shared direction sign s[c] in {-1, +1} */
SYNTH_HD int synth_dir_sign(uint64_t seed, uint64_t c) {
  return (synth_draw(synth_key(seed, SYNTH_T_DIR), c, 0) >> 63) ? -1 : 1;
}

SYNTH_HD uint64_t synth_f64_bits(double x) {
  union { double d; uint64_t u; } v;
  v.d = x;
  return v.u;
}

/* double -> bf16 bits, round to nearest even, straight from the double (no
 * double rounding through fp32). Inputs here are finite and either zero or of
 * magnitude in the bf16 normal range; anything below it flushes to +-0. */
SYNTH_HD uint16_t synth_bf16_rne(double x) {
  uint64_t b = synth_f64_bits(x);
  uint16_t sign = (uint16_t)((b >> 63) << 15);
  int e = (int)((b >> 52) & 0x7FF);
  uint64_t m = b & 0xFFFFFFFFFFFFFull;
  if (e == 0) return sign;
  int E = e - 1023 + 127;
  if (E <= 0) return sign;
  uint64_t full = (1ull << 52) | m;    /* 53 significant bits */
  uint64_t keep = full >> 45;          /* top 8 bits          */
  uint64_t rem = full & ((1ull << 45) - 1);
  const uint64_t half = 1ull << 44;
  if (rem > half || (rem == half && (keep & 1ull))) keep += 1;
  if (keep == 256ull) { keep = 128ull; E += 1; }
  if (E >= 255) return (uint16_t)(sign | 0x7F80u); /* never reached here */
  return (uint16_t)(sign | ((uint16_t)E << 7) | (uint16_t)(keep & 0x7Full));
}

/* double -> OCP FP8 E4M3 bits (bias 7, 3 mantissa bits, max 448, subnormal
 * step 2^-9), round to nearest even, saturating at +-448. */
SYNTH_HD uint8_t synth_e4m3_rne(double x) {
  uint64_t b = synth_f64_bits(x);
  uint8_t sign = (uint8_t)((b >> 63) << 7);
  int e = (int)((b >> 52) & 0x7FF);
  uint64_t m = b & 0xFFFFFFFFFFFFFull;
  if (e == 0) return sign;
  int ue = e - 1023;                   /* |x| = 1.m * 2^ue */
  uint64_t full = (1ull << 52) | m;
  /* quantum: 2^(ue-3) for normals (ue >= -6), 2^-9 for subnormals */
  int qexp = ue >= -6 ? ue - 3 : -9;
  int shift = 52 - (ue - qexp);        /* bits dropped from the 53-bit significand */
  uint64_t q;
  if (shift >= 64) {
    q = 0;
  } else {
    q = full >> shift;
    uint64_t rem = full & ((1ull << shift) - 1);
    uint64_t half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1ull))) q += 1;
  }
  /* q is the value in units of 2^qexp */
  if (ue < -6) {                       /* subnormal range (possibly rounded up to 2^-6) */
    if (q >= 8) return (uint8_t)(sign | 0x08u);
    return (uint8_t)(sign | (uint8_t)q);
  }
  int E = ue + 7;
  if (q == 16) { q = 8; E += 1; }
  if (E > 15 || (E == 15 && q > 14)) return (uint8_t)(sign | 0x7Eu); /* saturate to 448 */
  return (uint8_t)(sign | (uint8_t)(E << 3) | (uint8_t)(q - 8));
}

/* ---- workload element recipes (one per value distribution) ---------------- */

/* Gaussian element plus an additive planted offset (0.0 when unplanted). */
SYNTH_HD uint16_t synth_gauss_bf16(uint64_t key, uint64_t idx, double offset) {
  double z = synth_gauss(key, idx);
  return synth_bf16_rne(offset == 0.0 ? z : z + offset);
}

/* Gaussian element quantised to E4M3 at a fixed multiplier (one rounding for
 * the product, one for the E4M3 conversion). */
SYNTH_HD uint8_t synth_gauss_e4m3(uint64_t key, uint64_t idx, double mult) {
  double z = synth_gauss(key, idx);
  return synth_e4m3_rne(z * mult);
}

#endif /* MSA_SYNTH_H */
