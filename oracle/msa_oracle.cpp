// MSA (MiniMax Sparse Attention) forward path: plain CPU oracle.
//
// TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
// CPU-baseline leg load this library. It shares no code with the GPU path: it
// decodes its own inputs, accumulates in fp64 and runs the method's steps one
// after another, with the definitions of the article "MiniMax Sparse Attention
// (MSA): a Two-Branch Block-Sparse Attention Trained on a 109B-Parameter MoE
// With a 3T-Token Budget" (Chinese edition; cited below as [MSA-2B] with its
// section heading) and "MiniMax lança MSA: atenção esparsa treinada em modelo
// de 109B parâmetros com 3 trilhões de tokens" (cited as [MSA-PT]):
//
//   a1  index scores   s[t,g,j] = q_idx[t,g] . k_idx[j] for every visible key
//                      j <= t; one index-query head per GQA group g and one
//                      shared index-key head ([MSA-2B] "两个分支如何工作",
//                      how the two branches work).
//   a2  block max-pool S[t,g,b] = max of s[t,g,j] over the visible keys j of
//                      block b (same section); block size Bk = 128 and k = 16
//                      ([MSA-2B] "什么是 MSA", what MSA is).
//   a3  top-k          per (t, g): the block holding t is always kept; the
//                      other k-1 slots take the highest S among the earlier
//                      blocks ([MSA-2B] "两个分支如何工作"; the forced local
//                      block in "MSA 如何训练"; [MSA-PT] "Treinamento com KL
//                      Divergence", item 3). Raw scores are ranked directly,
//                      since softmax keeps their order ([MSA-2B] "内核协同设计",
//                      kernel co-design). Ties go to the lower block id.
//   a4  main branch    each query head h of group g attends, with exact
//                      scaled-dot-product softmax (scale 1/sqrt(d)), to the
//                      causally visible tokens of the group's selected blocks
//                      ([MSA-2B] "两个分支如何工作"; [MSA-PT] "Como funciona o
//                      MSA").
//   projections        q_idx = x W_qidx^T (n_g heads of d_idx), k_idx = x W_kidx^T
//                      (one shared head): the index branch's two projection
//                      matrices ([MSA-2B] "两个分支如何工作"), plain linear maps.
//   decode             the same steps for one new token at position L-1 of a
//                      paged KV cache whose page size is the block size
//                      ([MSA-2B] "运行 Kernel", the usage listing), with bf16 or
//                      FP8-E4M3 K/V dequantised as code * per-(K/V, kv head)
//                      scale ([MSA-PT] "Kernel open source e MiniMax-M3").
//
// Readings where the pages are silent (each is listed in the design notes):
// raw, unscaled index dot products (no ReLU, no weights); the local block
// takes one of the k slots and does not compete; when a query sees at most k
// blocks all of them are kept; block ids are returned in ascending order and
// padded with -1; LSE is the natural log of sum(exp(scale * q.k)).
//
// Pins (tests/test_oracle.py): dense causal GQA attention from torch's SDPA
// when k covers every visible block; an independently coded brute-force
// per-token index path; top-k order invariance under log-softmax; closed
// forms of attention (constant V, single key, equal keys, in-block permutation);
// exhaustive E4M3 and bf16 decodes against torch; integer fixtures in
// tests/golden worked out by hand.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

const double NEG_INF = -std::numeric_limits<double>::infinity();

// bf16 is the upper half of an IEEE binary32 word.
double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
// infinities, S.1111.111 is NaN, largest finite value 448.
double e4m3_to_double(uint8_t b) {
  int sign = b >> 7;
  int e = (b >> 3) & 0xF;
  int m = b & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
  if (e == 0)
    v = std::ldexp((double)m, -9);               // m/8 * 2^(1-7)
  else
    v = std::ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

// OCP FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no
// infinities or NaN; exponent 0 is subnormal (m * 0.5).
double e2m1_to_double(uint8_t c) {
  int sign = (c >> 3) & 1, e = (c >> 1) & 3, m = c & 1;
  double v = e == 0 ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -v : v;
}

// Key rows of one sequence. Unpaged tensors are [tokens, H, D]. Paged caches
// keep each page head-major, [pages, H, Bk, D] (the page tensor's second
// dimension is the number of kv heads in the pages' usage listing), with
// logical block b of the sequence in page pages[b].
struct Rows {
  const uint8_t* base = nullptr;   // element bytes
  int64_t H = 1, D = 0;            // heads and head dim of the tensor
  int elem_bytes = 2;
  const int32_t* pages = nullptr;  // page table of this sequence (nullptr: unpaged)
  int Bk = 128;
  // first element of (token j, head h)
  const uint8_t* at(int64_t j, int64_t h) const {
    int64_t e = pages ? (((int64_t)pages[j / Bk] * H + h) * Bk + j % Bk) * D : (j * H + h) * D;
    return base + (size_t)e * elem_bytes;
  }
};

double load(const uint8_t* p, int64_t i, int elem_bytes) {
  if (elem_bytes == 2) {
    uint16_t h;
    std::memcpy(&h, p + 2 * i, 2);
    return bf16_to_double(h);
  }
  return e4m3_to_double(p[i]);
}

// a1 + a2 for one (t, g): S[b] for b = 0 .. t/Bk (the visible blocks).
void block_scores(const double* qi, const Rows& kidx, int d_idx, int64_t t, int Bk,
                  std::vector<double>& S) {
  int64_t loc = t / Bk;
  S.assign((size_t)(loc + 1), NEG_INF);
  for (int64_t j = 0; j <= t; ++j) {
    const uint8_t* kr = kidx.at(j, 0);
    double s = 0.0;
    for (int c = 0; c < d_idx; ++c) s += qi[c] * load(kr, c, 2);
    int64_t b = j / Bk;
    if (s > S[(size_t)b]) S[(size_t)b] = s;
  }
}

// a3 for one (t, g): local block + top (k-1) earlier blocks, ascending, -1 pad.
void select_blocks(const std::vector<double>& S, int64_t loc, int k, int32_t* ids) {
  std::vector<int64_t> cand;
  for (int64_t b = 0; b < loc; ++b) cand.push_back(b);
  std::stable_sort(cand.begin(), cand.end(), [&](int64_t x, int64_t y) {
    if (S[(size_t)x] != S[(size_t)y]) return S[(size_t)x] > S[(size_t)y];
    return x < y;
  });
  int64_t take = std::min<int64_t>(k - 1, loc);
  std::vector<int64_t> sel(cand.begin(), cand.begin() + take);
  sel.push_back(loc);
  std::sort(sel.begin(), sel.end());
  for (int i = 0; i < k; ++i) ids[i] = i < (int)sel.size() ? (int32_t)sel[(size_t)i] : -1;
}

// a4 for one (t, h): softmax attention over the visible tokens of ids[0..k).
void attend(const double* q, const Rows& K, const Rows& V, int kvh, int d,
            const double* kscale, const double* vscale, const int32_t* ids, int k, int Bk,
            int64_t t, double scale, double* o, double* lse) {
  std::vector<int64_t> J;
  for (int i = 0; i < k; ++i) {
    if (ids[i] < 0) continue;
    int64_t b = ids[i];
    for (int64_t j = b * Bk; j < (b + 1) * Bk && j <= t; ++j) J.push_back(j);
  }
  std::sort(J.begin(), J.end());
  J.erase(std::unique(J.begin(), J.end()), J.end());
  std::vector<double> x(J.size());
  double m = NEG_INF;
  for (size_t n = 0; n < J.size(); ++n) {
    const uint8_t* kr = K.at(J[n], kvh);
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += q[c] * (load(kr, c, K.elem_bytes) * *kscale);
    x[n] = s * scale;
    m = std::max(m, x[n]);
  }
  double l = 0.0;
  std::vector<double> acc((size_t)d, 0.0);
  for (size_t n = 0; n < J.size(); ++n) {
    double p = std::exp(x[n] - m);
    l += p;
    const uint8_t* vr = V.at(J[n], kvh);
    for (int c = 0; c < d; ++c) acc[(size_t)c] += p * (load(vr, c, V.elem_bytes) * *vscale);
  }
  for (int c = 0; c < d; ++c) o[c] = J.empty() ? 0.0 : acc[(size_t)c] / l;
  *lse = J.empty() ? NEG_INF : m + std::log(l);
}

void decode_row(const uint16_t* src, int n, double* dst) {
  for (int i = 0; i < n; ++i) dst[i] = bf16_to_double(src[i]);
}

}  // namespace

extern "C" {

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

unsigned oracle_hardware_concurrency(void) { return std::thread::hardware_concurrency(); }

double oracle_bf16_to_f64(uint16_t h) { return bf16_to_double(h); }
double oracle_e4m3_to_f64(uint8_t b) { return e4m3_to_double(b); }
double oracle_e2m1_to_f64(uint8_t c) { return e2m1_to_double(c); }

// Prefill index branch (a1-a3) for n_rows query positions rows[i].
//   q_idx_rows [n_rows, n_g, d_idx] bf16 bits: the index queries of those rows
//   k_idx      [N, d_idx] bf16 bits (tokens 0 .. max(rows))
//   scores_out [n_rows, n_g, nb_out] fp64 or null: S, -inf beyond visibility
//   ids_out    [n_rows, n_g, k] int32
int oracle_index_select(const uint16_t* q_idx_rows, const int64_t* rows, int64_t n_rows,
                        const uint16_t* k_idx, int n_g, int d_idx, int Bk, int k,
                        int64_t nb_out, double* scores_out, int32_t* ids_out) {
  if (k < 1 || Bk < 1 || d_idx < 1 || n_g < 1) return -1;
  Rows kr;
  kr.base = (const uint8_t*)k_idx;
  kr.D = d_idx;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows * n_g; ++r) {
    int64_t t = rows[r / n_g];
    std::vector<double> qi((size_t)d_idx), S;
    decode_row(q_idx_rows + (size_t)r * d_idx, d_idx, qi.data());
    block_scores(qi.data(), kr, d_idx, t, Bk, S);
    if (scores_out)
      for (int64_t b = 0; b < nb_out; ++b)
        scores_out[(size_t)r * nb_out + b] = b < (int64_t)S.size() ? S[(size_t)b] : NEG_INF;
    select_blocks(S, t / Bk, k, ids_out + (size_t)r * k);
  }
  return 0;
}

// a3 alone on given fp32 block scores [n_rows, n_g, nb] of rows at positions
// rows[i] (entries beyond visibility are ignored).
int oracle_topk_blocks(const float* S_rows, const int64_t* rows, int64_t n_rows, int n_g,
                       int64_t nb, int Bk, int k, int32_t* ids_out) {
  if (k < 1 || Bk < 1) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n_rows * n_g; ++r) {
    int64_t t = rows[r / n_g];
    int64_t loc = t / Bk;
    if (loc >= nb) continue;
    std::vector<double> S((size_t)(loc + 1));
    for (int64_t b = 0; b <= loc; ++b) S[(size_t)b] = (double)S_rows[(size_t)r * nb + b];
    select_blocks(S, loc, k, ids_out + (size_t)r * k);
  }
  return 0;
}

// Prefill main branch (a4) for rows[i], on the given block ids.
//   q_rows [n_rows, H_q, d]; K, V [N, H_kv, d] bf16 bits; ids [n_rows, n_g, k]
//   o_out [n_rows, H_q, d] fp64; lse_out [n_rows, H_q] fp64
int oracle_sparse_attn(const uint16_t* q_rows, const int64_t* rows, int64_t n_rows,
                       const uint16_t* K, const uint16_t* V, const int32_t* ids, int H_q,
                       int H_kv, int d, int Bk, int k, double scale, double* o_out,
                       double* lse_out) {
  if (H_kv < 1 || H_q % H_kv != 0) return -1;
  int G = H_q / H_kv;
  Rows kr, vr;
  kr.base = (const uint8_t*)K;
  vr.base = (const uint8_t*)V;
  kr.H = vr.H = H_kv;
  kr.D = vr.D = d;
  const double one = 1.0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows * H_q; ++r) {
    int64_t i = r / H_q;
    int h = (int)(r % H_q);
    int g = h / G;
    std::vector<double> q((size_t)d);
    decode_row(q_rows + (size_t)r * d, d, q.data());
    attend(q.data(), kr, vr, g, d, &one, &one, ids + ((size_t)i * H_kv + g) * k, k, Bk, rows[i],
           scale, o_out + (size_t)r * d, lse_out + r);
  }
  return 0;
}

// KL alignment signal of the index branch ([MSA-2B] "MSA 如何训练", how MSA is
// trained; [MSA-PT] "Treinamento com KL Divergence"): the teacher is the main
// branch's distribution over the selected tokens J of (t, g), averaged over
// the group's G query heads,
//   p_main(j) = (1/G) sum_h exp(scale q_h . k_j - lse_h),  lse_h = log sum_J exp(scale q_h . k_j);
// the student is the index branch's distribution over the same tokens,
//   p_idx(j) = exp(s_j - LSE),  s_j = q_idx[t,g] . k_idx[j] (raw, as in a1),
//   LSE = log sum_J exp(s_j);
// and the signal is KL(p_main || p_idx) = sum_J p_main (log p_main - log p_idx),
// a term with p_main = 0 counting 0.
//   q_rows [n_rows, H_q, d], qi_rows [n_rows, n_g, d_idx], K [N, H_kv, d],
//   k_idx [N, d_idx] (bf16 bits), ids [n_rows, n_g, k]
//   kl_out [n_rows, n_g]; mag_out [n_rows, n_g] or null:
//   sum_J p_main (|log p_main| + |log p_idx|), the size of the terms that cancel
int oracle_kl_teacher(const uint16_t* q_rows, const uint16_t* qi_rows, const int64_t* rows,
                      int64_t n_rows, const uint16_t* K, const uint16_t* k_idx,
                      const int32_t* ids, int H_q, int H_kv, int d, int d_idx, int Bk, int k,
                      double scale, double* kl_out, double* mag_out) {
  if (H_kv < 1 || H_q % H_kv != 0 || Bk < 1 || k < 1) return -1;
  const int G = H_q / H_kv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows * H_kv; ++r) {
    const int64_t i = r / H_kv, t = rows[i];
    const int g = (int)(r % H_kv);
    const int32_t* sel = ids + (size_t)r * k;
    std::vector<int64_t> J;
    for (int u = 0; u < k; ++u) {
      if (sel[u] < 0) continue;
      for (int64_t j = (int64_t)sel[u] * Bk; j < ((int64_t)sel[u] + 1) * Bk && j <= t; ++j)
        J.push_back(j);
    }
    std::sort(J.begin(), J.end());
    J.erase(std::unique(J.begin(), J.end()), J.end());
    const size_t n = J.size();
    // teacher: the group's heads, each normalised over J, then averaged
    std::vector<double> pm(n, 0.0), x(n), q((size_t)d);
    for (int h = g * G; h < (g + 1) * G; ++h) {
      decode_row(q_rows + ((size_t)i * H_q + h) * d, d, q.data());
      double m = NEG_INF;
      for (size_t u = 0; u < n; ++u) {
        const uint16_t* kj = K + ((size_t)J[u] * H_kv + g) * d;
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += q[(size_t)c] * bf16_to_double(kj[c]);
        x[u] = s * scale;
        m = std::max(m, x[u]);
      }
      double l = 0.0;
      for (size_t u = 0; u < n; ++u) l += std::exp(x[u] - m);
      const double lse = m + std::log(l);
      for (size_t u = 0; u < n; ++u) pm[u] += std::exp(x[u] - lse) / G;
    }
    // student: softmax of the raw index scores over J
    std::vector<double> qi((size_t)d_idx), sidx(n);
    decode_row(qi_rows + (size_t)r * d_idx, d_idx, qi.data());
    double ms = NEG_INF;
    for (size_t u = 0; u < n; ++u) {
      const uint16_t* kj = k_idx + (size_t)J[u] * d_idx;
      double s = 0.0;
      for (int c = 0; c < d_idx; ++c) s += qi[(size_t)c] * bf16_to_double(kj[c]);
      sidx[u] = s;
      ms = std::max(ms, s);
    }
    double ls = 0.0;
    for (size_t u = 0; u < n; ++u) ls += std::exp(sidx[u] - ms);
    const double LSE = ms + std::log(ls);
    double kl = 0.0, mag = 0.0;
    for (size_t u = 0; u < n; ++u) {
      if (pm[u] <= 0.0) continue;
      const double lp = std::log(pm[u]), lq = sidx[u] - LSE;
      kl += pm[u] * (lp - lq);
      mag += pm[u] * (std::fabs(lp) + std::fabs(lq));
    }
    kl_out[r] = kl;
    if (mag_out) mag_out[r] = mag;
  }
  return 0;
}

// Index-branch projections ([MSA-2B] "两个分支如何工作": the index branch adds
// two projection matrices to the GQA layer, one giving the index-query head of
// every group, one giving the shared index-key head). Read as plain linear
// maps of the layer input, no bias and no activation:
//   q_idx[t, g, c] = sum_m x[t, m] * w_qidx[g * d_idx + c, m]
//   k_idx[t, c]    = sum_m x[t, m] * w_kidx[c, m]
//   x [n_rows, d_model], w_qidx [n_g * d_idx, d_model], w_kidx [d_idx, d_model]
//   (bf16 bits; weights in [out, in] layout); outputs fp64.
int oracle_index_project(const uint16_t* x, const uint16_t* w_qidx, const uint16_t* w_kidx,
                         int64_t n_rows, int d_model, int n_g, int d_idx, double* q_out,
                         double* k_out) {
  if (n_rows < 0 || d_model < 1 || n_g < 1 || d_idx < 1) return -1;
  const int n_out = n_g * d_idx + d_idx;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < n_rows; ++t) {
    std::vector<double> xr((size_t)d_model);
    decode_row(x + (size_t)t * d_model, d_model, xr.data());
    for (int o = 0; o < n_out; ++o) {
      const bool is_q = o < n_g * d_idx;
      const uint16_t* w = is_q ? w_qidx + (size_t)o * d_model
                               : w_kidx + (size_t)(o - n_g * d_idx) * d_model;
      double acc = 0.0;
      for (int m = 0; m < d_model; ++m) acc += xr[(size_t)m] * bf16_to_double(w[m]);
      if (is_q) q_out[(size_t)t * n_g * d_idx + o] = acc;
      else k_out[(size_t)t * d_idx + (o - n_g * d_idx)] = acc;
    }
  }
  return 0;
}

// Textbook dense causal GQA attention (every j <= t), used to pin a4.
int oracle_dense_gqa(const uint16_t* q_rows, const int64_t* rows, int64_t n_rows,
                     const uint16_t* K, const uint16_t* V, int H_q, int H_kv, int d,
                     double scale, double* o_out, double* lse_out) {
  if (H_kv < 1 || H_q % H_kv != 0) return -1;
  int G = H_q / H_kv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows * H_q; ++r) {
    int64_t t = rows[r / H_q];
    int g = (int)(r % H_q) / G;
    std::vector<double> q((size_t)d), x((size_t)(t + 1)), acc((size_t)d, 0.0);
    decode_row(q_rows + (size_t)r * d, d, q.data());
    double m = NEG_INF;
    for (int64_t j = 0; j <= t; ++j) {
      const uint16_t* kj = K + ((size_t)j * H_kv + g) * d;
      double s = 0.0;
      for (int c = 0; c < d; ++c) s += q[(size_t)c] * bf16_to_double(kj[c]);
      x[(size_t)j] = s * scale;
      m = std::max(m, x[(size_t)j]);
    }
    double l = 0.0;
    for (int64_t j = 0; j <= t; ++j) {
      double p = std::exp(x[(size_t)j] - m);
      l += p;
      const uint16_t* vj = V + ((size_t)j * H_kv + g) * d;
      for (int c = 0; c < d; ++c) acc[(size_t)c] += p * bf16_to_double(vj[c]);
    }
    for (int c = 0; c < d; ++c) o_out[(size_t)r * d + c] = acc[(size_t)c] / l;
    lse_out[r] = m + std::log(l);
  }
  return 0;
}

// Independent brute-force index path for tiny shapes: scores every (t, j) pair
// with an explicit causality test, pools each block by scanning the whole
// token range, orders ALL visible blocks by (score desc, id asc) with a plain
// insertion sort, then keeps the local block plus the first k-1 others.
int oracle_index_brute(const uint16_t* q_idx_rows, const int64_t* rows, int64_t n_rows,
                       const uint16_t* k_idx, int n_g, int d_idx, int Bk, int k,
                       int32_t* ids_out) {
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t t = rows[i];
    for (int g = 0; g < n_g; ++g) {
      int64_t nblk = t / Bk + 1;
      std::vector<double> best((size_t)nblk, NEG_INF);
      std::vector<int> seen((size_t)nblk, 0);
      for (int64_t j = 0; j < (t / Bk + 1) * (int64_t)Bk; ++j) {
        if (!(j <= t)) continue;
        double s = 0.0;
        for (int c = 0; c < d_idx; ++c)
          s += bf16_to_double(q_idx_rows[((size_t)i * n_g + g) * d_idx + c]) *
               bf16_to_double(k_idx[(size_t)j * d_idx + c]);
        int64_t b = j / Bk;
        if (!seen[(size_t)b] || s > best[(size_t)b]) best[(size_t)b] = s;
        seen[(size_t)b] = 1;
      }
      int64_t local = t / Bk;
      std::vector<int64_t> order;
      for (int64_t b = 0; b < nblk; ++b) {
        if (b == local) continue;
        size_t pos = order.size();
        order.push_back(b);
        while (pos > 0) {
          int64_t a = order[pos - 1], c = order[pos];
          bool swap = best[(size_t)c] > best[(size_t)a] ||
                      (best[(size_t)c] == best[(size_t)a] && c < a);
          if (!swap) break;
          std::swap(order[pos - 1], order[pos]);
          --pos;
        }
      }
      std::vector<int64_t> keep;
      keep.push_back(local);
      for (size_t n = 0; n < order.size() && (int)keep.size() < k; ++n) keep.push_back(order[n]);
      std::sort(keep.begin(), keep.end());
      int32_t* out = ids_out + ((size_t)i * n_g + g) * k;
      for (int n = 0; n < k; ++n) out[n] = n < (int)keep.size() ? (int32_t)keep[(size_t)n] : -1;
    }
  }
  return 0;
}

// Decode index branch: one query per sequence at t = seq_lens[s] - 1.
//   q_idx [B, n_g, d_idx]; k_idx_pages [P, Bk, d_idx]; page_table [B, max_pages]
//   scores_out [B, n_g, nb_out] fp64 or null; ids_out [B, n_g, k]
int oracle_decode_index_select(const uint16_t* q_idx, const uint16_t* k_idx_pages,
                               const int32_t* page_table, const int32_t* seq_lens, int B,
                               int max_pages, int n_g, int d_idx, int Bk, int k, int64_t nb_out,
                               double* scores_out, int32_t* ids_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < (int64_t)B * n_g; ++r) {
    int s = (int)(r / n_g);
    int64_t t = (int64_t)seq_lens[s] - 1;
    Rows kr;
    kr.base = (const uint8_t*)k_idx_pages;
    kr.D = d_idx;
    kr.pages = page_table + (size_t)s * max_pages;
    kr.Bk = Bk;
    std::vector<double> qi((size_t)d_idx), S;
    decode_row(q_idx + (size_t)r * d_idx, d_idx, qi.data());
    block_scores(qi.data(), kr, d_idx, t, Bk, S);
    if (scores_out)
      for (int64_t b = 0; b < nb_out; ++b)
        scores_out[(size_t)r * nb_out + b] = b < (int64_t)S.size() ? S[(size_t)b] : NEG_INF;
    select_blocks(S, t / Bk, k, ids_out + (size_t)r * k);
  }
  return 0;
}

// Decode main branch with a paged bf16 (kv_fp8 = 0) or E4M3 (kv_fp8 = 1) cache.
//   q [B, H_q, d] bf16; k_pages, v_pages [P, H_kv, Bk, d]; k_scale, v_scale
//   [H_kv] fp32 (used for E4M3 only); ids [B, n_g, k]
//   o_out [B, H_q, d] fp64; lse_out [B, H_q] fp64
int oracle_decode_attn(const uint16_t* q, const void* k_pages, const void* v_pages, int kv_fp8,
                       const float* k_scale, const float* v_scale, const int32_t* page_table,
                       const int32_t* seq_lens, const int32_t* ids, int B, int max_pages,
                       int H_q, int H_kv, int d, int Bk, int k, double scale, double* o_out,
                       double* lse_out) {
  if (H_kv < 1 || H_q % H_kv != 0) return -1;
  int G = H_q / H_kv;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < (int64_t)B * H_q; ++r) {
    int s = (int)(r / H_q);
    int h = (int)(r % H_q);
    int g = h / G;
    Rows kr, vr;
    kr.base = (const uint8_t*)k_pages;
    vr.base = (const uint8_t*)v_pages;
    kr.H = vr.H = H_kv;
    kr.D = vr.D = d;
    kr.elem_bytes = vr.elem_bytes = kv_fp8 ? 1 : 2;
    kr.pages = vr.pages = page_table + (size_t)s * max_pages;
    kr.Bk = vr.Bk = Bk;
    double ks = kv_fp8 ? (double)k_scale[g] : 1.0;
    double vs = kv_fp8 ? (double)v_scale[g] : 1.0;
    std::vector<double> qv((size_t)d);
    decode_row(q + (size_t)r * d, d, qv.data());
    attend(qv.data(), kr, vr, g, d, &ks, &vs, ids + ((size_t)s * H_kv + g) * k, k, Bk,
           (int64_t)seq_lens[s] - 1, scale, o_out + (size_t)r * d, lse_out + r);
  }
  return 0;
}

}  // extern "C"
