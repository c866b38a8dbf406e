/*
 * Float64 CPU oracle for decode attention over a paged KV cache, in plain C.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by tests/ and by the CPU-baseline leg of
 * bench.py (through ctypes); the CUDA library never links or calls it, and it
 * shares no code with the CUDA path.  It restates, loop by loop, what
 * oracle/paged_attention.py computes (ATOM model-operations guide,
 * "Multi-head attention" forward flow and "Attention dispatch"; configuration
 * guide, kv_cache_block_size and kv_cache_dtype), and its parity pin is that
 * Python oracle (tests/test_oracle_c.py), itself pinned against a library
 * attention routine, closed forms and invariants.
 *
 * For sequence i (L = seq_lens[i] cached tokens, which include its qn query
 * tokens), query row r (absolute position p = L - qn + r) and query head hq
 * (KV head hk = hq / (Hq / Hkv)):
 *   key j is visible when j <= p (and, with a sliding window W > 0, j > p - W);
 *   K_j, V_j = rows of page block_tables[i][j / 16], slot j % 16, head hk,
 *              decoded to double (bf16 exactly; e4m3fn code value times the
 *              fp32 tensor scale, times the row's fp32 scale when per-token
 *              scales are given);
 *   s_j = scale * <q, K_j>; an optional sink logit joins the softmax with a
 *   zero value row;
 *   lse = m + ln sum_j exp(s_j - m),  out = sum_j exp(s_j - lse) V_j.
 * Two plain passes per row (all scores, then the normaliser and the weighted
 * sum); OpenMP over (sequence, KV head) pairs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PA_PAGE 16

/* bf16 bit pattern -> double: the upper half of an IEEE binary32. */
static double bf16_value(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* OCP e4m3fn code -> double from its fields: sign (bit 7), exponent (bits
 * 6..3, bias 7), mantissa (bits 2..0); exponent 0 is subnormal; 0x7F / 0xFF
 * are NaN (no infinities). */
static double e4m3fn_value(uint8_t code) {
  const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* Cached element (page, slot, head, d) decoded to double. */
static double cached(const void* cache, int fp8, int64_t page, int slot, int h, int d, int Hkv, int D,
                     double tensor_scale, const float* tok, int64_t tok_page_stride) {
  const int64_t idx = ((page * PA_PAGE + slot) * (int64_t)Hkv + h) * D + d;
  if (!fp8) return bf16_value(((const uint16_t*)cache)[idx]);
  double v = e4m3fn_value(((const uint8_t*)cache)[idx]) * tensor_scale;
  if (tok) v *= (double)tok[page * tok_page_stride + (int64_t)h * PA_PAGE + slot];
  return v;
}

/*
 * q_bits    uint16 [T, Hq, D] (bf16 patterns)
 * k, v      [NB, 16, Hkv, D] contiguous: uint16 bf16 patterns (kv_fp8 = 0) or uint8 e4m3fn codes
 * block_tables int32 [B, bt_stride]; seq_lens int32 [B]; qsl int32 [B + 1] or NULL (one token each)
 * scale, k_scale, v_scale  taken as the fp32 numbers the kernel receives
 * k_tok, v_tok  float32 [NB, Hkv, 16] per-token scales or NULL (fp8 only)
 * window    > 0: sliding window of that many keys; sinks float32 [Hq] or NULL
 * out       double [T, Hq, D]; lse double [T, Hq]   (rows of sequences not in
 *           seq_mask, when given, are left untouched)
 * seq_mask  uint8 [B] or NULL: evaluate only sequences with a non-zero entry
 * threads   OpenMP threads (<= 0: the runtime's default)
 * Returns 0, or -1 on an invalid argument (the oracle only checks shapes it relies on).
 */
int pa_oracle_decode(const uint16_t* q_bits, const void* k, const void* v, int kv_fp8,
                     const int32_t* block_tables, int64_t bt_stride, const int32_t* seq_lens, const int32_t* qsl,
                     int B, int T, int Hq, int Hkv, int D, int64_t NB, float scale, float k_scale, float v_scale,
                     const float* k_tok, const float* v_tok, int window, const float* sinks, double* out,
                     double* lse, const uint8_t* seq_mask, int threads) {
  if (B < 0 || T < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return -1;
  const int G = Hq / Hkv;
  const double sc = (double)scale, ks = (double)k_scale, vs = (double)v_scale;
  const int64_t tok_stride = (int64_t)Hkv * PA_PAGE;
  int bad = 0;
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t task = 0; task < (int64_t)B * Hkv; ++task) {
    const int i = (int)(task / Hkv), hk = (int)(task % Hkv);
    if (seq_mask && !seq_mask[i]) continue;
    const int L = seq_lens[i];
    const int t0 = qsl ? qsl[i] : i;
    const int qn = qsl ? qsl[i + 1] - qsl[i] : 1;
    if (L < 1 || qn < 1 || qn > L || t0 < 0 || t0 + qn > T) {
      bad = 1;
      continue;
    }
    /* the sequence's K and V rows of head hk, gathered through the block table */
    double* K = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* V = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* s = (double*)malloc(sizeof(double) * (size_t)(L + 1));
    if (!K || !V || !s) {
      free(K);
      free(V);
      free(s);
      bad = 1;
      continue;
    }
    for (int j = 0; j < L; ++j) {
      const int64_t page = block_tables[(int64_t)i * bt_stride + j / PA_PAGE];
      if (page < 0 || page >= NB) {
        bad = 1;
        break;
      }
      for (int d = 0; d < D; ++d) {
        K[(size_t)j * D + d] = cached(k, kv_fp8, page, j % PA_PAGE, hk, d, Hkv, D, ks, kv_fp8 ? k_tok : NULL, tok_stride);
        V[(size_t)j * D + d] = cached(v, kv_fp8, page, j % PA_PAGE, hk, d, Hkv, D, vs, kv_fp8 ? v_tok : NULL, tok_stride);
      }
    }
    for (int r = 0; r < qn && !bad; ++r) {
      const int p = L - qn + r;
      for (int g = 0; g < G; ++g) {
        const int hq = hk * G + g;
        const uint16_t* qrow = q_bits + ((int64_t)(t0 + r) * Hq + hq) * D;
        /* pass 1: scores of the visible keys, and their maximum */
        double m = -INFINITY;
        for (int j = 0; j < L; ++j) {
          int visible = j <= p;
          if (window > 0) visible = visible && j > p - window;
          if (!visible) {
            s[j] = -INFINITY;
            continue;
          }
          double dot = 0.0;
          for (int d = 0; d < D; ++d) dot += bf16_value(qrow[d]) * K[(size_t)j * D + d];
          s[j] = sc * dot;
          if (s[j] > m) m = s[j];
        }
        const double sink = sinks ? (double)sinks[hq] : -INFINITY;
        if (sink > m) m = sink;
        /* pass 2: normaliser and weighted sum of the value rows */
        double sum = sinks ? exp(sink - m) : 0.0;
        for (int j = 0; j < L; ++j)
          if (s[j] != -INFINITY) sum += exp(s[j] - m);
        const double l = m + log(sum);
        double* orow = out + ((int64_t)(t0 + r) * Hq + hq) * D;
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        for (int j = 0; j < L; ++j) {
          if (s[j] == -INFINITY) continue;
          const double w = exp(s[j] - l);
          for (int d = 0; d < D; ++d) orow[d] += w * V[(size_t)j * D + d];
        }
        lse[(int64_t)(t0 + r) * Hq + hq] = l;
      }
    }
    free(K);
    free(V);
    free(s);
  }
  return bad ? -1 : 0;
}

/*
 * MLA decode over a paged latent cache (the NumPy oracle's oracle/mla.py,
 * restated loop by loop; ATOM model-operations guide, "Multi-head latent
 * attention"): every cached token is one row C_j of Dqk values (latent part
 * first, kv_lora_rank values, then the rotary part) shared by all query heads;
 * s_j = scale * <q[t, h], C_j> for j <= p, out = sum_j exp(s_j - lse) C_j[0:Dv].
 * Sequence by sequence: the rows are decoded once (OpenMP over rows), then
 * OpenMP over (query row, head) pairs.
 *
 * q_bits   uint16 [T, Hq, Dqk]; cache [NB, 16, Dqk] contiguous, uint16 bf16 patterns
 *          (kv_fp8 = 0) or uint8 e4m3fn codes (value = code * kv_scale)
 * out      double [T, Hq, Dv]; lse double [T, Hq]; other arguments as pa_oracle_decode.
 * Returns 0, or -1 on an invalid argument.
 */
int pa_oracle_mla_decode(const uint16_t* q_bits, const void* cache, int kv_fp8, const int32_t* block_tables,
                         int64_t bt_stride, const int32_t* seq_lens, const int32_t* qsl, int B, int T, int Hq,
                         int Dqk, int Dv, int64_t NB, float scale, float kv_scale, double* out, double* lse,
                         const uint8_t* seq_mask, int threads) {
  if (B < 0 || T < 0 || Hq <= 0 || Dqk <= 0 || Dv <= 0 || Dv > Dqk) return -1;
  const double sc = (double)scale, ks = (double)kv_scale;
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#else
  (void)threads;
#endif
  for (int i = 0; i < B; ++i) {
    if (seq_mask && !seq_mask[i]) continue;
    const int L = seq_lens[i];
    const int t0 = qsl ? qsl[i] : i;
    const int qn = qsl ? qsl[i + 1] - qsl[i] : 1;
    if (L < 1 || qn < 1 || qn > L || t0 < 0 || t0 + qn > T) return -1;
    for (int j = 0; j < L; j += PA_PAGE) {
      const int64_t page = block_tables[(int64_t)i * bt_stride + j / PA_PAGE];
      if (page < 0 || page >= NB) return -1;
    }
    /* the sequence's decoded rows, gathered through the block table (once for all heads) */
    double* C = (double*)malloc(sizeof(double) * (size_t)L * Dqk);
    if (!C) return -1;
#pragma omp parallel for schedule(static)
    for (int j = 0; j < L; ++j) {
      const int64_t page = block_tables[(int64_t)i * bt_stride + j / PA_PAGE];
      const int64_t row = (page * PA_PAGE + j % PA_PAGE) * (int64_t)Dqk;
      for (int d = 0; d < Dqk; ++d)
        C[(size_t)j * Dqk + d] = kv_fp8 ? e4m3fn_value(((const uint8_t*)cache)[row + d]) * ks
                                        : bf16_value(((const uint16_t*)cache)[row + d]);
    }
    int bad = 0;
    /* one task per (query row, head) */
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int rh = 0; rh < qn * Hq; ++rh) {
      const int r = rh / Hq, h = rh % Hq;
      const int p = L - qn + r;
      const uint16_t* qrow = q_bits + ((int64_t)(t0 + r) * Hq + h) * Dqk;
      double* s = (double*)malloc(sizeof(double) * (size_t)(p + 1));
      if (!s) {
        bad = 1;
        continue;
      }
      /* pass 1: scores of keys 0..p and their maximum */
      double m = -INFINITY;
      for (int j = 0; j <= p; ++j) {
        double dot = 0.0;
        for (int d = 0; d < Dqk; ++d) dot += bf16_value(qrow[d]) * C[(size_t)j * Dqk + d];
        s[j] = sc * dot;
        if (s[j] > m) m = s[j];
      }
      /* pass 2: normaliser and the weighted sum of the latent parts */
      double sum = 0.0;
      for (int j = 0; j <= p; ++j) sum += exp(s[j] - m);
      const double l = m + log(sum);
      double* orow = out + ((int64_t)(t0 + r) * Hq + h) * Dv;
      for (int d = 0; d < Dv; ++d) orow[d] = 0.0;
      for (int j = 0; j <= p; ++j) {
        const double w = exp(s[j] - l);
        for (int d = 0; d < Dv; ++d) orow[d] += w * C[(size_t)j * Dqk + d];
      }
      lse[(int64_t)(t0 + r) * Hq + h] = l;
      free(s);
    }
    free(C);
    if (bad) return -1;
  }
  return 0;
}

/* Threads OpenMP would use by default (1 without OpenMP). */
int pa_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
