/* Host fill of the synthetic MSA workloads (shared recipe: synth_recipe.h).
 * Built with -ffp-contract=off so the recipe's single IEEE operations round
 * exactly as on the device. */
#include <stddef.h>
#include "synth_recipe.h"

/* out[i] = bf16 bits of element idx0 + i, i < count */
void synth_host_fill_bf16(const SynthSpec* sp, int tensor, uint64_t idx0, uint64_t count,
                          uint16_t* out) {
  SynthSpec s = *sp;
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)count; ++i)
    out[i] = synth_element(&s, tensor, idx0 + (uint64_t)i);
}

/* out[i] = E4M3 bits of element idx0 + i of SYNTH_T_K / SYNTH_T_V */
void synth_host_fill_e4m3(const SynthSpec* sp, int tensor, uint64_t idx0, uint64_t count,
                          uint8_t* out) {
  SynthSpec s = *sp;
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)count; ++i)
    out[i] = synth_element_e4m3(&s, tensor, idx0 + (uint64_t)i);
}

/* scalar helpers, exposed so tests can check the conversions on their own */
uint16_t synth_host_bf16_rne(double x) { return synth_bf16_rne(x); }
uint8_t synth_host_e4m3_rne(double x) { return synth_e4m3_rne(x); }
double synth_host_gauss(uint64_t seed, int tensor, uint64_t idx) {
  return synth_gauss(synth_key(seed, (uint64_t)tensor), idx);
}
uint64_t synth_host_draw(uint64_t seed, int tensor, uint64_t idx, uint32_t j) {
  return synth_draw(synth_key(seed, (uint64_t)tensor), idx, j);
}
int synth_host_dir_sign(uint64_t seed, uint64_t c) { return synth_dir_sign(seed, c); }
size_t synth_host_spec_size(void) { return sizeof(SynthSpec); }
