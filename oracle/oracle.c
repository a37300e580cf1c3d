/*
 * oracle.c — plain, slow, fp64 CPU oracle of hybrid prefill+decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this code; the product path never does. It shares no source with the CUDA
 * library: no headers, no helpers, no constants.
 *
 * What it computes (each function cites the passage it follows):
 *   "Week 6: Beyond PyTorch: Custom Kernel과 vLLM" (core-sig.pytorch.kr)
 *     §"Attention에 적용하기"            out = softmax(q·Kᵀ / sqrt(d_k)) · V (scale passed in)
 *     §"Safe softmax (3-pass, 수치 안정성 확보)"   max pass, exp-sum pass, normalise pass
 *     §"Non-Causal vs. Causal Attention"  causal: a token sees itself and earlier tokens only;
 *                                         non-causal: a token sees every token of its sequence
 *     §"한 스텝에 여러 종류의 request 섞기"      extend: a chunk token sees the cached prefix and
 *                                         the earlier tokens of its own chunk; decode is an
 *                                         extend of one token
 *     §"PagedAttention"                   logical block -> physical block through a table
 *   "LLMSO - W4 - Optimization & Frameworks" (seojhoon.tistory.com)
 *     §"FlashDecoding — decode 단계의 병렬성 확보"  split the keys, keep each part's max and sum,
 *                                         merge exactly
 *     §"KV 헤드 줄이기 — MHA → GQA → MQA → MLA"   several query heads share one KV head
 *
 * Readings where the pages are silent:
 *   - causal alignment of a chunk with a prefix: local token i of a chunk of q_len tokens in a
 *     sequence of kv_len cached rows sits at absolute position p = kv_len - q_len + i and sees
 *     rows 0..p;
 *   - query head h reads kv-head h / (Hq / Hkv) (contiguous groups);
 *   - pool layout [num_blocks][Hkv][block_size][head_dim], K and V in separate pools.
 *
 * Inputs are bf16 bit patterns (uint16), widened exactly to double. All arithmetic is double.
 * Every pool index is range-checked; a bad block-table entry returns -1 instead of reading.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 -> double: a bf16 value is the upper half of an IEEE binary32. */
static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Address of row j of kv-head g of one sequence (PagedAttention: table lookup, then offset). */
static int64_t pool_row(const int32_t* bt_row, int64_t j, int g, int Hkv, int D, int BS,
                        int64_t num_blocks) {
  int64_t logical = j / BS;
  int64_t phys = bt_row[logical];
  if (phys < 0 || phys >= num_blocks) return -1;
  return ((phys * Hkv + g) * BS + (j % BS)) * (int64_t)D;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Partial attention of one query over the key range [j0, j1) of one sequence:
 *   m = max_j x_j,  l = sum_j exp(x_j - m),  o[c] = sum_j exp(x_j - m) v_j[c]   (unnormalised)
 * with x_j = scale * q·k_j. An empty range returns m = -inf, l = 0, o = 0.
 * This is the per-chunk state of the split-KV method ("FlashDecoding": each chunk's max and sum).
 * `x` is caller scratch of at least (j1 - j0) doubles. Returns 0, or -1 on a bad table entry.
 */
int oracle_attend_range(const uint16_t* q, const int32_t* bt_row, int64_t j0, int64_t j1, int g,
                        int Hkv, int D, int BS, const uint16_t* k_pool, const uint16_t* v_pool,
                        int64_t num_blocks, double scale, double* m_out, double* l_out,
                        double* o, double* x) {
  for (int c = 0; c < D; ++c) o[c] = 0.0;
  if (j1 <= j0) {
    *m_out = -INFINITY;
    *l_out = 0.0;
    return 0;
  }
  /* pass 1: scores and their maximum */
  double m = -INFINITY;
  for (int64_t j = j0; j < j1; ++j) {
    int64_t r = pool_row(bt_row, j, g, Hkv, D, BS, num_blocks);
    if (r < 0) return -1;
    double dot = 0.0;
    for (int c = 0; c < D; ++c) dot += widen_bf16(q[c]) * widen_bf16(k_pool[r + c]);
    x[j - j0] = scale * dot;
    if (x[j - j0] > m) m = x[j - j0];
  }
  /* pass 2: exponentials relative to the maximum, their sum, and the weighted V rows */
  double l = 0.0;
  for (int64_t j = j0; j < j1; ++j) {
    double w = exp(x[j - j0] - m);
    l += w;
    int64_t r = pool_row(bt_row, j, g, Hkv, D, BS, num_blocks);
    for (int c = 0; c < D; ++c) o[c] += w * widen_bf16(v_pool[r + c]);
  }
  *m_out = m;
  *l_out = l;
  return 0;
}

/*
 * Exact merge of n partial states (m_i, l_i, o_i) into the normalised output
 * ("FlashDecoding": rescale each chunk by its max, then combine):
 *   m* = max_i m_i,  out = sum_i exp(m_i - m*) o_i / sum_i exp(m_i - m*) l_i.
 * Partials with m_i = -inf (empty ranges) carry no weight. o is [n][D] row-major.
 */
void oracle_merge(int n, const double* m, const double* l, const double* o, int D, double* out) {
  double ms = -INFINITY;
  for (int i = 0; i < n; ++i)
    if (m[i] > ms) ms = m[i];
  double den = 0.0;
  for (int c = 0; c < D; ++c) out[c] = 0.0;
  for (int i = 0; i < n; ++i) {
    if (m[i] == -INFINITY) continue;
    double w = exp(m[i] - ms);
    den += w * l[i];
    for (int c = 0; c < D; ++c) out[c] += w * o[(int64_t)i * D + c];
  }
  for (int c = 0; c < D; ++c) out[c] /= den;
}

/*
 * One attention output row by the 3-pass safe softmax over rows [0, nvis) of one sequence:
 *   pass 1  m = max_j x_j
 *   pass 2  den = sum_j exp(x_j - m)
 *   pass 3  out[c] = sum_j exp(x_j - m) / den * v_j[c]
 * `x` is caller scratch of nvis doubles. Returns 0, -1 on a bad table entry, -2 if nvis < 1.
 */
int oracle_attend_row(const uint16_t* q, const int32_t* bt_row, int64_t nvis, int g, int Hkv,
                      int D, int BS, const uint16_t* k_pool, const uint16_t* v_pool,
                      int64_t num_blocks, double scale, double* out, double* x) {
  if (nvis < 1) return -2;
  double m = -INFINITY;
  for (int64_t j = 0; j < nvis; ++j) {
    int64_t r = pool_row(bt_row, j, g, Hkv, D, BS, num_blocks);
    if (r < 0) return -1;
    double dot = 0.0;
    for (int c = 0; c < D; ++c) dot += widen_bf16(q[c]) * widen_bf16(k_pool[r + c]);
    x[j] = scale * dot;
    if (x[j] > m) m = x[j];
  }
  double den = 0.0;
  for (int64_t j = 0; j < nvis; ++j) den += exp(x[j] - m);
  for (int c = 0; c < D; ++c) out[c] = 0.0;
  for (int64_t j = 0; j < nvis; ++j) {
    double p = exp(x[j] - m) / den;
    int64_t r = pool_row(bt_row, j, g, Hkv, D, BS, num_blocks);
    for (int c = 0; c < D; ++c) out[c] += p * widen_bf16(v_pool[r + c]);
  }
  return 0;
}

/* The query rows the oracle is asked for: (kind, index, head).
 * kind 0: prefill token `index` (global index into the concatenated chunks);
 * kind 1: decode sequence `index`. */
typedef struct {
  int Hq, Hkv, D, BS;
  int Np, Nd;
  int64_t num_blocks;
  int max_blocks_per_seq;
  double scale;
  const uint16_t *q_prefill, *q_decode, *k_pool, *v_pool;
  const int32_t *block_tables, *cu_seqlens_q, *kv_lens;
  int causal; /* nonzero: chunk tokens see rows 0..p; zero: all kv_len rows */
} oracle_batch;

/* Locate the sequence, visible row count and query vector of one requested row. */
static int resolve_row(const oracle_batch* b, int kind, int64_t index, int h, const uint16_t** q,
                       const int32_t** bt_row, int64_t* nvis) {
  if (h < 0 || h >= b->Hq) return -3;
  if (kind == 0) {
    if (index < 0 || b->Np < 1 || index >= b->cu_seqlens_q[b->Np]) return -3;
    int s = 0;
    while (!(index >= b->cu_seqlens_q[s] && index < b->cu_seqlens_q[s + 1])) ++s;
    int64_t qlen = b->cu_seqlens_q[s + 1] - b->cu_seqlens_q[s];
    int64_t i = index - b->cu_seqlens_q[s];
    int64_t prefix = (int64_t)b->kv_lens[s] - qlen;
    if (prefix < 0) return -3;
    *nvis = b->causal ? prefix + i + 1 : b->kv_lens[s]; /* rows 0..prefix+i, or all */
    *bt_row = b->block_tables + (int64_t)s * b->max_blocks_per_seq;
    *q = b->q_prefill + (index * b->Hq + h) * (int64_t)b->D;
  } else {
    if (index < 0 || index >= b->Nd) return -3;
    int s = b->Np + (int)index;
    *nvis = b->kv_lens[s]; /* the decode token sees every cached row */
    *bt_row = b->block_tables + (int64_t)s * b->max_blocks_per_seq;
    *q = b->q_decode + (index * b->Hq + h) * (int64_t)b->D;
  }
  if (*nvis > (int64_t)b->max_blocks_per_seq * b->BS) return -3;
  return 0;
}

/*
 * Output rows for an explicit list of n (kind, index, head) requests, out is [n][D].
 * OpenMP over requests. Returns 0, or the first nonzero per-row code.
 */
int oracle_rows(int Hq, int Hkv, int D, int BS, int Np, int Nd, int64_t num_blocks,
                int max_blocks_per_seq, double scale, const uint16_t* q_prefill,
                const uint16_t* q_decode, const uint16_t* k_pool, const uint16_t* v_pool,
                const int32_t* block_tables, const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                int64_t n, const int32_t* kinds, const int64_t* indices, const int32_t* heads,
                double* out, int causal) {
  if (Hkv < 1 || Hq % Hkv != 0) return -3;
  oracle_batch b = {Hq, Hkv, D, BS, Np, Nd, num_blocks, max_blocks_per_seq, scale,
                    q_prefill, q_decode, k_pool, v_pool, block_tables, cu_seqlens_q, kv_lens,
                    causal};
  int group = Hq / Hkv;
  int err = 0;
  int64_t max_rows = (int64_t)max_blocks_per_seq * BS;
#pragma omp parallel
  {
    double* x = (double*)malloc(sizeof(double) * (size_t)(max_rows > 0 ? max_rows : 1));
#pragma omp for schedule(dynamic, 4)
    for (int64_t t = 0; t < n; ++t) {
      const uint16_t* q;
      const int32_t* bt_row;
      int64_t nvis;
      int rc = resolve_row(&b, kinds[t], indices[t], heads[t], &q, &bt_row, &nvis);
      if (rc == 0)
        rc = oracle_attend_row(q, bt_row, nvis, heads[t] / group, Hkv, D, BS, k_pool, v_pool,
                               num_blocks, scale, out + t * (int64_t)D, x);
      if (rc != 0) {
#pragma omp critical
        if (err == 0) err = rc;
      }
    }
    free(x);
  }
  return err;
}

/*
 * The whole hybrid batch: every prefill token and every decode sequence, every query head.
 * o_prefill is [num_prefill_tokens][Hq][D], o_decode is [Nd][Hq][D], both double.
 */
int oracle_hybrid_attention(int Hq, int Hkv, int D, int BS, int Np, int Nd, int64_t num_blocks,
                            int max_blocks_per_seq, double scale, const uint16_t* q_prefill,
                            const uint16_t* q_decode, const uint16_t* k_pool,
                            const uint16_t* v_pool, const int32_t* block_tables,
                            const int32_t* cu_seqlens_q, const int32_t* kv_lens,
                            double* o_prefill, double* o_decode, int causal) {
  if (Hkv < 1 || Hq % Hkv != 0) return -3;
  oracle_batch b = {Hq, Hkv, D, BS, Np, Nd, num_blocks, max_blocks_per_seq, scale,
                    q_prefill, q_decode, k_pool, v_pool, block_tables, cu_seqlens_q, kv_lens,
                    causal};
  int64_t tp = Np > 0 ? cu_seqlens_q[Np] : 0;
  int64_t total = (tp + Nd) * Hq;
  int group = Hq / Hkv;
  int err = 0;
  int64_t max_rows = (int64_t)max_blocks_per_seq * BS;
#pragma omp parallel
  {
    double* x = (double*)malloc(sizeof(double) * (size_t)(max_rows > 0 ? max_rows : 1));
#pragma omp for schedule(dynamic, 4)
    for (int64_t t = 0; t < total; ++t) {
      int64_t row = t / Hq;
      int h = (int)(t % Hq);
      int kind = row < tp ? 0 : 1;
      int64_t index = row < tp ? row : row - tp;
      double* out = (kind == 0 ? o_prefill : o_decode) + (index * Hq + h) * (int64_t)D;
      const uint16_t* q;
      const int32_t* bt_row;
      int64_t nvis;
      int rc = resolve_row(&b, kind, index, h, &q, &bt_row, &nvis);
      if (rc == 0)
        rc = oracle_attend_row(q, bt_row, nvis, h / group, Hkv, D, BS, k_pool, v_pool,
                               num_blocks, scale, out, x);
      if (rc != 0) {
#pragma omp critical
        if (err == 0) err = rc;
      }
    }
    free(x);
  }
  return err;
}

/*
 * FP8 KV cache. Every decode step reads the whole cache ("Week 6: Beyond PyTorch: Custom
 * Kernel과 vLLM", §"KV Cache"), so fewer bytes per element mean a shorter step; "LLMSO - W4 -
 * Optimization & Frameworks", §"2-4. 고급 KV 캐싱 기법", scales K per channel (its outliers sit
 * in particular channels) and V per token.
 *
 * e4m3 (the 8-bit floating-point format with 4 exponent and 3 mantissa bits and no
 * infinities): bit 7 sign; bits 6..3 exponent E (bias 7); bits 2..0 mantissa M.
 *   E = 0:            (-1)^s * M/8 * 2^(1-7)      (subnormal, and zero)
 *   E = 15, M = 7:    NaN
 *   otherwise:        (-1)^s * (1 + M/8) * 2^(E-7)   (largest: 448)
 */
double oracle_e4m3_to_double(uint8_t bits) {
  int s = bits >> 7, e = (bits >> 3) & 15, m = bits & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, 1 - 7);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/*
 * e4m3 code of a float: the nearest e4m3 value, ties to the one with an even mantissa (round to
 * nearest even), magnitudes from 448 up saturating to +-448, the sign kept (a negative value
 * that rounds to zero is -0, 0x80), NaN to 0x7F. Written from the format's definition: the
 * candidates are the 127 finite magnitudes oracle_e4m3_to_double gives for codes 0x00..0x7E.
 */
uint8_t oracle_e4m3_from_float(float x) {
  if (x != x) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  int best = 0;
  double best_d = a;  /* distance to code 0 (value 0) */
  for (int c = 1; c <= 0x7E; ++c) {
    const double d = fabs(oracle_e4m3_to_double((uint8_t)c) - a);
    /* codes ascend with their values, so an equal distance is a tie between neighbours: keep
       the even mantissa */
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return sign | (uint8_t)best;
}

/*
 * Append of an iteration's new tokens to a bf16 cache ("Week 6: Beyond PyTorch: Custom Kernel과
 * vLLM", §"PagedAttention": the cache only grows by appended rows; §"한 스텝에 여러 종류의
 * request 섞기": an extend chunk follows its sequence's cached rows, a decode token is its
 * sequence's last row). New token t carries one K and one V row per kv-head (k_new / v_new are
 * bf16 [T_p + Nd][Hkv][D]; the prefill chunks' tokens first in order, then one token per decode
 * sequence). Chunk token i of prefill sequence s goes to position kv_len[s] - q_len(s) + i,
 * decode d's token to position kv_len[Np + d] - 1; position j of a sequence is row j % BS of
 * its physical block block_tables[seq][j / BS]. The rows are copied bit for bit into the pools
 * [num_blocks][Hkv][BS][D]. Returns 0, or -1 on a bad table entry (that row is not written).
 */
int oracle_append_bf16(int Hkv, int D, int BS, int Np, int Nd, int64_t num_blocks, int max_blocks,
                       const int32_t* cu_seqlens, const int32_t* kv_lens,
                       const int32_t* block_tables, const uint16_t* k_new, const uint16_t* v_new,
                       uint16_t* k_pool, uint16_t* v_pool) {
  int err = 0;
  int64_t t = 0;  /* index of the new token in k_new / v_new */
  for (int seq = 0; seq < Np + Nd; ++seq) {
    const int64_t q_len = seq < Np ? (int64_t)cu_seqlens[seq + 1] - cu_seqlens[seq] : 1;
    const int64_t first = (int64_t)kv_lens[seq] - q_len;
    for (int64_t i = 0; i < q_len; ++i, ++t) {
      const int64_t pos = first + i;
      const int32_t phys = block_tables[(int64_t)seq * max_blocks + pos / BS];
      if (phys < 0 || phys >= num_blocks) {
        err = -1;
        continue;
      }
      for (int g = 0; g < Hkv; ++g) {
        const int64_t dst = (((int64_t)phys * Hkv + g) * BS + pos % BS) * D;
        const int64_t src = (t * Hkv + g) * D;
        memcpy(k_pool + dst, k_new + src, (size_t)D * sizeof(uint16_t));
        memcpy(v_pool + dst, v_new + src, (size_t)D * sizeof(uint16_t));
      }
    }
  }
  return err;
}

/*
 * Append of one new token per decode sequence to an FP8 cache. The token's row goes to
 * position kv_len - 1 of its sequence, through the block table. K row, channel c:
 * e4m3((float)k / k_scale[g][c]); V row: scale = max_c |v| / 448 (1 when that max is 0), values
 * e4m3((float)v / scale), the scale stored in v_scale. Every division and the max are
 * binary32 (round to nearest), the precision the quantised codes are decided in. k_new / v_new
 * are bf16 [Nd][Hkv][D]. Returns 0, or -1 on a bad table entry (that row is not written).
 */
int oracle_append_fp8(int Hkv, int D, int BS, int Nd, int64_t num_blocks, int max_blocks,
                      const uint16_t* k_new, const uint16_t* v_new, const float* k_scale,
                      const int32_t* block_tables, const int32_t* kv_lens, uint8_t* k8,
                      uint8_t* v8, float* v_scale) {
  int err = 0;
  for (int d = 0; d < Nd; ++d) {
    const int pos = kv_lens[d] - 1;
    const int32_t phys = block_tables[(int64_t)d * max_blocks + pos / BS];
    if (phys < 0 || phys >= num_blocks) {
      err = -1;
      continue;
    }
    for (int g = 0; g < Hkv; ++g) {
      const int64_t row = ((int64_t)phys * Hkv + g) * BS + pos % BS;
      const uint16_t* kr = k_new + ((int64_t)d * Hkv + g) * D;
      const uint16_t* vr = v_new + ((int64_t)d * Hkv + g) * D;
      float amax = 0.f;
      for (int c = 0; c < D; ++c) {
        const float v = (float)widen_bf16(vr[c]);
        if (fabsf(v) > amax) amax = fabsf(v);
      }
      const float vs = amax > 0.f ? amax / 448.0f : 1.0f;
      for (int c = 0; c < D; ++c) {
        const float kq = (float)widen_bf16(kr[c]) / k_scale[g * D + c];
        const float vq = (float)widen_bf16(vr[c]) / vs;
        k8[row * D + c] = oracle_e4m3_from_float(kq);
        v8[row * D + c] = oracle_e4m3_from_float(vq);
      }
      v_scale[row] = vs;
    }
  }
  return err;
}

/*
 * Decode attention over an FP8 cache. K row j, channel c of kv-head g is
 * e4m3(k8[row j][c]) * k_scale[g][c] (one scale per kv-head and channel); V row j is
 * e4m3(v8[row j][c]) * v_scale[row j] (one scale per cached token and kv-head). Every decode
 * token attends to all kv_len rows of its sequence, as in oracle_attend_row. Pools are
 * [num_blocks][Hkv][BS][D] bytes, v_scale is [num_blocks][Hkv][BS], block_tables is
 * [Nd][max_blocks_per_seq]; o_decode is [Nd][Hq][D] doubles. OpenMP over (sequence, head).
 * Returns 0, -1 on a bad table entry, -3 on bad shapes.
 */
int oracle_decode_fp8(int Hq, int Hkv, int D, int BS, int Nd, int64_t num_blocks,
                      int max_blocks_per_seq, double scale, const uint16_t* q_decode,
                      const uint8_t* k8, const uint8_t* v8, const float* k_scale,
                      const float* v_scale, const int32_t* block_tables, const int32_t* kv_lens,
                      double* o_decode) {
  if (Hkv < 1 || Hq % Hkv != 0) return -3;
  int group = Hq / Hkv;
  int err = 0;
  int64_t max_rows = (int64_t)max_blocks_per_seq * BS;
#pragma omp parallel
  {
    double* x = (double*)malloc(sizeof(double) * (size_t)(max_rows > 0 ? max_rows : 1));
#pragma omp for schedule(dynamic, 4)
    for (int64_t t = 0; t < (int64_t)Nd * Hq; ++t) {
      int64_t d = t / Hq;
      int h = (int)(t % Hq), g = h / group;
      int64_t nvis = kv_lens[d];
      const int32_t* bt_row = block_tables + d * (int64_t)max_blocks_per_seq;
      const uint16_t* q = q_decode + (d * Hq + h) * (int64_t)D;
      double* out = o_decode + (d * Hq + h) * (int64_t)D;
      int rc = 0;
      if (nvis < 1 || nvis > max_rows) rc = -3;
      double m = -INFINITY;
      for (int64_t j = 0; rc == 0 && j < nvis; ++j) {
        int64_t r = pool_row(bt_row, j, g, Hkv, D, BS, num_blocks);
        if (r < 0) {
          rc = -1;
          break;
        }
        double dot = 0.0;
        for (int c = 0; c < D; ++c)
          dot += widen_bf16(q[c]) * (oracle_e4m3_to_double(k8[r + c]) * (double)k_scale[g * D + c]);
        x[j] = scale * dot;
        if (x[j] > m) m = x[j];
      }
      if (rc == 0) {
        double den = 0.0;
        for (int64_t j = 0; j < nvis; ++j) den += exp(x[j] - m);
        for (int c = 0; c < D; ++c) out[c] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
          double p = exp(x[j] - m) / den;
          int64_t r = pool_row(bt_row, j, g, Hkv, D, BS, num_blocks);
          double vs = (double)v_scale[r / D];
          for (int c = 0; c < D; ++c) out[c] += p * (oracle_e4m3_to_double(v8[r + c]) * vs);
        }
      }
      if (rc != 0) {
#pragma omp critical
        if (err == 0) err = rc;
      }
    }
    free(x);
  }
  return err;
}
