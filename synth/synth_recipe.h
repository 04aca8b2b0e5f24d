/* Element recipes of the synthetic MSA workloads, shared by host and device.
 *
 * A workload is a batch of B sequences of L tokens each (prefill: B = 1,
 * L = N). Every tensor is addressed by its logical element index
 *     idx = ((s * L + t) * H + h) * D + c
 * (H = heads of that tensor, D = its head dim), so a value never depends on
 * where a paged cache stores it, and a decode query is row L-1 of the same
 * sequence's prefill query tensor.
 *
 * Structure of the index inputs (the rest is plain N(0,1)):
 *  - kind SYNTH_KIND_GAUSS: q_idx = bf16(z + s[c] * q_off), k_idx of a planted
 *    block = bf16(z + s[c] * plant_amp), other k_idx = bf16(z);
 *  - kind SYNTH_KIND_INT:   q_idx = clamp(u + s[c], -4, 4), k_idx of a planted
 *    block = plant_amp * s[c], other k_idx = u, with u uniform in {-4..4}.
 * s[c] in {-1,+1} is one shared direction per seed; planted[s * nb + b] marks
 * the planted blocks of sequence s.
 */
#ifndef MSA_SYNTH_RECIPE_H
#define MSA_SYNTH_RECIPE_H

#include "synth.h"

enum { SYNTH_KIND_GAUSS = 0, SYNTH_KIND_INT = 1 };

typedef struct {
  uint64_t seed;
  int32_t kind;
  int32_t B;          /* sequences                                   */
  int64_t L;          /* tokens per sequence                          */
  int32_t H_q, H_kv, d;
  int32_t n_g, d_idx;
  int32_t Bk;
  int32_t nb;         /* blocks per sequence = ceil(L / Bk)           */
  int32_t pad_;
  double q_off;       /* q_idx offset along s[] (gauss kind)          */
  double plant_amp;   /* planted k_idx amplitude along s[]            */
  double fp8_mult;    /* multiplier applied before E4M3 rounding      */
  const uint8_t* planted; /* [B * nb], pointer valid on the filling side */
} SynthSpec;

/* bf16 bits of element idx of tensor `tensor` (SYNTH_T_Q .. SYNTH_T_KIDX) */
SYNTH_HD uint16_t synth_element(const SynthSpec* sp, int tensor, uint64_t idx) {
  uint64_t key = synth_key(sp->seed, (uint64_t)tensor);
  if (tensor == SYNTH_T_Q || tensor == SYNTH_T_K || tensor == SYNTH_T_V)
    return synth_gauss_bf16(key, idx, 0.0);
  uint64_t D = (uint64_t)sp->d_idx;
  uint64_t c = idx % D;
  int sgn = synth_dir_sign(sp->seed, c);
  if (tensor == SYNTH_T_QIDX) {
    if (sp->kind == SYNTH_KIND_INT) {
      int v = synth_int9(key, idx) + sgn;
      v = v < -4 ? -4 : (v > 4 ? 4 : v);
      return synth_bf16_rne((double)v);
    }
    return synth_gauss_bf16(key, idx, sgn > 0 ? sp->q_off : -sp->q_off);
  }
  /* SYNTH_T_KIDX: row r = s * L + t */
  uint64_t r = idx / D;
  uint64_t s = r / (uint64_t)sp->L;
  uint64_t t = r % (uint64_t)sp->L;
  int planted = sp->planted ? sp->planted[s * (uint64_t)sp->nb + t / (uint64_t)sp->Bk] : 0;
  if (sp->kind == SYNTH_KIND_INT) {
    if (planted) return synth_bf16_rne(sgn > 0 ? sp->plant_amp : -sp->plant_amp);
    return synth_bf16_rne((double)synth_int9(key, idx));
  }
  double off = planted ? (sgn > 0 ? sp->plant_amp : -sp->plant_amp) : 0.0;
  return synth_gauss_bf16(key, idx, off);
}

/* E4M3 bits of element idx of SYNTH_T_K or SYNTH_T_V (same z as the bf16 run) */
SYNTH_HD uint8_t synth_element_e4m3(const SynthSpec* sp, int tensor, uint64_t idx) {
  return synth_gauss_e4m3(synth_key(sp->seed, (uint64_t)tensor), idx, sp->fp8_mult);
}

#endif /* MSA_SYNTH_RECIPE_H */
