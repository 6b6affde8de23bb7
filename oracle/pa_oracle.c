/*
 * pa_oracle.c - plain CPU oracle for the paged KV-cache hot path (test infrastructure).
 *
 * This file is the checker, not the product: only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark load it. It shares no code, header, table or constant
 * with the CUDA library. Everything is written for a reader to check against the sources by
 * eye: straight loops, fp64 arithmetic, no blocking, no fusion, no reordering.
 *
 * Sources:
 *  [PA]   "Efficient Memory Management for Large Language Model Serving with PagedAttention"
 *         (paper summary page): paragraph on the PagedAttention kernel (block K_j holds the
 *         keys of tokens (j-1)B+1..jB; each block is fetched wherever it is stored; the result
 *         is identical to ordinary attention); paragraph on the block table (logical blocks
 *         filled left to right, filled-slot count); paragraph on copy-on-write sharing.
 *  [P1]   "When KV Capacity Runs Out: Pausing and Resuming Requests": Figures 1-2 (positions
 *         numbered from 0; the KV of position 8 goes into the first slot of a newly linked
 *         block) and Figure 4 (KV copied to CPU memory and restored into possibly different
 *         blocks).
 *  [CB]   "Continuous Batching and PagedAttention", section "The block table is a page table"
 *         (attention math unchanged; gather through the table).
 *  [PV]   "KV Cache Preemption in vLLM: Swap, Recompute and Behavior Under Memory Pressure",
 *         section "How much KV cache a token costs" (an FP8 cache holds one byte per element).
 *  Number formats (the pages name FP16 and FP8 but do not define them): IEEE 754 binary16,
 *  bfloat16 (binary32 with the low 16 fraction bits dropped) and OCP 8-bit floating point
 *  E4M3 (bias 7, no infinities, S.1111.111 = NaN).
 *
 * Readings where the pages are silent (each listed with the design notes):
 *  - positions are 0-indexed: position t lives in logical block t / B, slot t % B;
 *  - ctx_len counts every filled slot including the token written this step;
 *  - GQA groups are contiguous: query head h reads kv head h / (Hq / Hkv);
 *  - ctx_len == 0 gives an all-zero output row;
 *  - FP8 values are dequantised as (stored value) * per-tensor scale, and quantised on write as
 *    the nearest E4M3 code (ties to even, saturating at 448) of value * (1 / scale), both the
 *    reciprocal and the product rounded to binary32.
 *
 * Parity pins: every function here is pinned by tests against library decoders, a library
 * attention routine on the unpaged data, closed forms and the worked example of [P1].
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { PAO_F16 = 0, PAO_BF16 = 1, PAO_E4M3 = 2 };

/* ---------------------------------------------------------------- number formats */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double pao_f16_value(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 10) & 0x1f;
  int f = bits & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -24); /* subnormal: (f / 2^10) * 2^-14 */
  } else if (e == 31) {
    mag = f ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(1024 + f), e - 15 - 10); /* (1 + f / 2^10) * 2^(e - 15) */
  }
  return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double pao_bf16_value(uint16_t bits) {
  int sign = (bits >> 15) & 1;
  int e = (bits >> 7) & 0xff;
  int f = bits & 0x7f;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -126 - 7); /* subnormal: (f / 2^7) * 2^-126 */
  } else if (e == 255) {
    mag = f ? NAN : INFINITY;
  } else {
    mag = ldexp((double)(128 + f), e - 127 - 7); /* (1 + f / 2^7) * 2^(e - 127) */
  }
  return sign ? -mag : mag;
}

/* OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits. There are no
 * infinities; only S.1111.111 is NaN, so exponent 15 with fraction 0..6 is a normal number
 * (largest 448). */
double pao_e4m3_value(uint8_t bits) {
  int sign = (bits >> 7) & 1;
  int e = (bits >> 3) & 0xf;
  int f = bits & 0x7;
  double mag;
  if (e == 15 && f == 7) {
    mag = NAN;
  } else if (e == 0) {
    mag = ldexp((double)f, -6 - 3); /* subnormal: (f / 2^3) * 2^-6 */
  } else {
    mag = ldexp((double)(8 + f), e - 7 - 3); /* (1 + f / 2^3) * 2^(e - 7) */
  }
  return sign ? -mag : mag;
}

/* Round to the nearest integer, ties to the even one, of a value 0 <= m < 2^31. */
static uint32_t round_half_even(double m) {
  const double f = floor(m);
  const double r = m - f;
  uint32_t q = (uint32_t)f;
  if (r > 0.5 || (r == 0.5 && (q & 1u))) ++q;
  return q;
}

/* The E4M3 code nearest to x, ties to the code with an even fraction field; magnitudes at or
 * beyond the largest finite value 448 (infinities included) saturate to it, NaN gives the NaN
 * code 0x7F. Subnormal codes are the multiples of 2^-9 below 2^-6. */
uint8_t pao_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  const uint8_t sign = signbit(x) ? 0x80 : 0x00;
  const double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {
    /* q = 8 rounds up to 2^-6, whose code (exponent field 1, fraction 0) is also 8 */
    return sign | (uint8_t)round_half_even(ldexp(a, 9));
  }
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1), so a = (1 + m / 8) * 2^(e - 1) */
  int E = e - 1;
  uint32_t q = round_half_even((ldexp(a, -E) - 1.0) * 8.0);
  if (q == 8) { /* rounded up to the next power of two */
    q = 0;
    E += 1;
  }
  return sign | (uint8_t)(((E + 7) << 3) | q);
}

void pao_e4m3_encode_array(const float* x, uint8_t* out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = pao_e4m3_encode(x[i]);
}

/* Threads the OpenMP runtime would use (1 when built without OpenMP). */
int pao_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

static int elt_bytes(int dtype) { return dtype == PAO_E4M3 ? 1 : 2; }

/* Value of element `index` of a raw array holding `dtype` elements. */
static double element(const void* base, size_t index, int dtype) {
  if (dtype == PAO_E4M3) return pao_e4m3_value(((const uint8_t*)base)[index]);
  uint16_t bits;
  memcpy(&bits, (const uint8_t*)base + 2 * index, 2);
  return dtype == PAO_F16 ? pao_f16_value(bits) : pao_bf16_value(bits);
}

/* ---------------------------------------------------------------- decode attention */

/*
 * out[s][h][:] for every sequence s and query head h, in fp64 ([PA], [CB]):
 *   1. gather: for t < L, K^[t] = k_scale * k_pool[block_tables[s][t / B]][g][t % B][:],
 *      V^[t] likewise, with g = h / (Hq / Hkv);
 *   2. ordinary softmax attention on the gathered rows:
 *      s_t = scale * sum_d q[s][h][d] * K^[t][d];  p = softmax(s);  out = sum_t p_t V^[t].
 * Returns 0, or -1 if some ctx_len or block id lies outside the pool (those rows are zero).
 */
int pao_decode(const void* q, int q_dtype, const void* k_pool, const void* v_pool, int kv_dtype,
               const int32_t* block_tables, const int32_t* ctx_lens, int num_seqs,
               int num_q_heads, int num_kv_heads, int head_dim, int block_size, int num_blocks,
               int max_blocks_per_seq, double scale, double k_scale, double v_scale, double* out,
               int num_threads) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
  const int group = num_q_heads / num_kv_heads;
  int bad = 0;
  const int threads = num_threads > 0 ? num_threads : pao_max_threads();
  (void)threads;
#pragma omp parallel for collapse(2) schedule(dynamic) num_threads(threads) reduction(| : bad)
  for (int s = 0; s < num_seqs; ++s) {
    for (int h = 0; h < num_q_heads; ++h) {
      double* o = out + ((size_t)s * num_q_heads + h) * head_dim;
      for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
      const int L = ctx_lens[s];
      if (L == 0) continue;
      if (L < 0 || L > max_blocks_per_seq * block_size) {
        bad = 1;
        continue;
      }
      const int g = h / group;

      /* 1. gather the sequence's keys and values into contiguous rows */
      double* K = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
      double* V = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
      double* score = (double*)malloc(sizeof(double) * (size_t)L);
      int row_ok = 1;
      for (int t = 0; t < L && row_ok; ++t) {
        const int j = t / block_size;    /* logical block */
        const int slot = t % block_size; /* slot inside the block */
        const int phys = block_tables[(size_t)s * max_blocks_per_seq + j];
        if (phys < 0 || phys >= num_blocks) {
          row_ok = 0;
          break;
        }
        const size_t first = (((size_t)phys * num_kv_heads + g) * block_size + slot) * head_dim;
        for (int d = 0; d < head_dim; ++d) {
          K[(size_t)t * head_dim + d] = element(k_pool, first + d, kv_dtype) * k_scale;
          V[(size_t)t * head_dim + d] = element(v_pool, first + d, kv_dtype) * v_scale;
        }
      }
      if (!row_ok) {
        bad = 1;
        free(K);
        free(V);
        free(score);
        continue;
      }

      /* 2. ordinary softmax attention */
      const size_t qoff = ((size_t)s * num_q_heads + h) * head_dim;
      double max_score = -INFINITY;
      for (int t = 0; t < L; ++t) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
          dot += element(q, qoff + d, q_dtype) * K[(size_t)t * head_dim + d];
        score[t] = scale * dot;
        if (score[t] > max_score) max_score = score[t];
      }
      double denom = 0.0;
      for (int t = 0; t < L; ++t) {
        score[t] = exp(score[t] - max_score);
        denom += score[t];
      }
      for (int d = 0; d < head_dim; ++d) {
        double acc = 0.0;
        for (int t = 0; t < L; ++t) acc += score[t] * V[(size_t)t * head_dim + d];
        o[d] = acc / denom;
      }
      free(K);
      free(V);
      free(score);
    }
  }
  return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- prefill attention */

/*
 * Causal attention of a chunk of new tokens over the paged cache ([PA] prompt phase: all prompt
 * tokens processed at once, building their KV; [P1] Figure 3: a recomputed request processes
 * all its retained tokens together; [CB] chunked prefill). Sequence s holds L = ctx_lens[s]
 * positions (its chunk's K/V already written); its chunk has n = q_starts[s + 1] - q_starts[s]
 * query tokens, q rows q_starts[s] .. q_starts[s + 1] - 1, and query i stands at position
 * L - n + i. For each query head h (kv group g = h / (Hq / Hkv)):
 *   s_t = scale * sum_d q[h][d] * K^[t][d]  for t <= L - n + i;  out = sum_t softmax(s)_t V^[t],
 * with K^, V^ gathered through the block table as in pao_decode: for an FP8 cache ([PV]
 * section "How much KV cache a token costs") K^ = k_scale * the stored E4M3 value and
 * V^ = v_scale * the stored value, so a recomputed request can be prefilled over the same
 * one-byte cache its decode steps read. Returns 0, or -1 if some length or block id is invalid
 * (those rows are zero).
 */
int pao_prefill(const void* q, int q_dtype, const void* k_pool, const void* v_pool, int kv_dtype,
                const int32_t* block_tables, const int32_t* ctx_lens, const int32_t* q_starts,
                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                int num_blocks, int max_blocks_per_seq, double scale, double k_scale,
                double v_scale, double* out, int num_threads) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
  const int group = num_q_heads / num_kv_heads;
  int bad = 0;
  const int threads = num_threads > 0 ? num_threads : pao_max_threads();
  (void)threads;
#pragma omp parallel for collapse(2) schedule(dynamic) num_threads(threads) reduction(| : bad)
  for (int s = 0; s < num_seqs; ++s) {
    for (int h = 0; h < num_q_heads; ++h) {
      const int L = ctx_lens[s];
      const int n = q_starts[s + 1] - q_starts[s];
      for (int i = 0; i < n; ++i) {
        double* o = out + ((size_t)(q_starts[s] + i) * num_q_heads + h) * head_dim;
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
      }
      if (n <= 0) continue;
      if (n > L || L > max_blocks_per_seq * block_size) {
        bad = 1;
        continue;
      }
      const int g = h / group;

      /* 1. gather the sequence's keys and values into contiguous rows */
      double* K = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
      double* V = (double*)malloc(sizeof(double) * (size_t)L * head_dim);
      double* score = (double*)malloc(sizeof(double) * (size_t)L);
      int rows_ok = 1;
      for (int t = 0; t < L && rows_ok; ++t) {
        const int phys = block_tables[(size_t)s * max_blocks_per_seq + t / block_size];
        if (phys < 0 || phys >= num_blocks) {
          rows_ok = 0;
          break;
        }
        const size_t first =
            (((size_t)phys * num_kv_heads + g) * block_size + t % block_size) * head_dim;
        for (int d = 0; d < head_dim; ++d) {
          K[(size_t)t * head_dim + d] = k_scale * element(k_pool, first + d, kv_dtype);
          V[(size_t)t * head_dim + d] = v_scale * element(v_pool, first + d, kv_dtype);
        }
      }
      if (!rows_ok) {
        bad = 1;
        free(K);
        free(V);
        free(score);
        continue;
      }

      /* 2. each query: ordinary softmax attention over positions 0 .. its own */
      for (int i = 0; i < n; ++i) {
        const int last = L - n + i;
        const size_t qoff = ((size_t)(q_starts[s] + i) * num_q_heads + h) * head_dim;
        double max_score = -INFINITY;
        for (int t = 0; t <= last; ++t) {
          double dot = 0.0;
          for (int d = 0; d < head_dim; ++d)
            dot += element(q, qoff + d, q_dtype) * K[(size_t)t * head_dim + d];
          score[t] = scale * dot;
          if (score[t] > max_score) max_score = score[t];
        }
        double denom = 0.0;
        for (int t = 0; t <= last; ++t) {
          score[t] = exp(score[t] - max_score);
          denom += score[t];
        }
        double* o = out + ((size_t)(q_starts[s] + i) * num_q_heads + h) * head_dim;
        for (int d = 0; d < head_dim; ++d) {
          double acc = 0.0;
          for (int t = 0; t <= last; ++t) acc += score[t] * V[(size_t)t * head_dim + d];
          o[d] = acc / denom;
        }
      }
      free(K);
      free(V);
      free(score);
    }
  }
  return bad ? -1 : 0;
}

/* ---------------------------------------------------------------- block movers */

/*
 * Store each new token's K and V in its slot ([P1] Figure 2): for token t with
 * sigma = slot_mapping[t] >= 0, pool[sigma / B][h][sigma % B][:] = new[t][h][:] for all heads.
 * Negative slots are padding. Returns -1 if a slot lies outside the pool (that token is skipped).
 */
int pao_write_kv(const void* k, const void* v, void* k_pool, void* v_pool,
                 const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                 int block_size, int num_blocks, int kv_dtype) {
  const size_t row = (size_t)head_dim * elt_bytes(kv_dtype);
  int bad = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t sigma = slot_mapping[t];
    if (sigma < 0) continue;
    const int64_t blk = sigma / block_size;
    const int64_t slot = sigma % block_size;
    if (blk >= num_blocks) {
      bad = 1;
      continue;
    }
    for (int h = 0; h < num_kv_heads; ++h) {
      const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + slot) * row;
      const size_t src = ((size_t)t * num_kv_heads + h) * row;
      memcpy((uint8_t*)k_pool + dst, (const uint8_t*)k + src, row);
      memcpy((uint8_t*)v_pool + dst, (const uint8_t*)v + src, row);
    }
  }
  return bad ? -1 : 0;
}

/*
 * Quantise-on-write into an FP8 cache ([PV] section "How much KV cache a token costs": one byte
 * per element): each new K or V element x, given in f16 or bf16, is stored as the E4M3 code of
 * x * inv, with inv = 1 / scale rounded to binary32 (k_scale for K, v_scale for V), so that
 * code * scale recovers it; the product is rounded to binary32 first. The pages give no rounding
 * for this step; multiplying by the binary32 reciprocal is the usual form. In fp64 the product
 * of two binary32 values is exact, so rounding it once to float gives the binary32 product, and
 * rounding 1 / scale from fp64 to float gives the correctly rounded reciprocal. Slots as in
 * pao_write_kv. Returns -1 if a slot lies outside the pool (that token is skipped).
 */
int pao_write_kv_fp8(const void* k, const void* v, int src_dtype, void* k_pool, void* v_pool,
                     const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                     int block_size, int num_blocks, float k_scale, float v_scale) {
  const float k_inv = (float)(1.0 / (double)k_scale);
  const float v_inv = (float)(1.0 / (double)v_scale);
  int bad = 0;
  for (int t = 0; t < num_tokens; ++t) {
    const int64_t sigma = slot_mapping[t];
    if (sigma < 0) continue;
    const int64_t blk = sigma / block_size;
    const int64_t slot = sigma % block_size;
    if (blk >= num_blocks) {
      bad = 1;
      continue;
    }
    for (int h = 0; h < num_kv_heads; ++h) {
      const size_t dst = (((size_t)blk * num_kv_heads + h) * block_size + slot) * head_dim;
      const size_t src = ((size_t)t * num_kv_heads + h) * head_dim;
      for (int d = 0; d < head_dim; ++d) {
        const float qk = (float)(element(k, src + d, src_dtype) * (double)k_inv);
        const float qv = (float)(element(v, src + d, src_dtype) * (double)v_inv);
        ((uint8_t*)k_pool)[dst + d] = pao_e4m3_encode(qk);
        ((uint8_t*)v_pool)[dst + d] = pao_e4m3_encode(qv);
      }
    }
  }
  return bad ? -1 : 0;
}

/*
 * Copy-on-write ([PA] sharing paragraph): for every pair (src, dst), every layer and both
 * pools, block dst becomes a byte copy of block src. The pairs form one step: every source is
 * read before any destination is written. Returns -1 if an id lies outside the pool (that pair
 * is skipped).
 */
int pao_copy_blocks(void* const* k_pools, void* const* v_pools, int num_layers,
                    const int32_t* pairs, int num_pairs, int num_blocks, size_t block_bytes) {
  int bad = 0;
  uint8_t* snapshot = (uint8_t*)malloc(block_bytes * 2 * (size_t)num_layers * (num_pairs + 1));
  for (int p = 0; p < num_pairs; ++p) {
    const int src = pairs[2 * p];
    if (src < 0 || src >= num_blocks) continue;
    for (int l = 0; l < num_layers; ++l) {
      uint8_t* keep = snapshot + ((size_t)p * num_layers + l) * 2 * block_bytes;
      memcpy(keep, (const uint8_t*)k_pools[l] + (size_t)src * block_bytes, block_bytes);
      memcpy(keep + block_bytes, (const uint8_t*)v_pools[l] + (size_t)src * block_bytes,
             block_bytes);
    }
  }
  for (int p = 0; p < num_pairs; ++p) {
    const int src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      bad = 1;
      continue;
    }
    for (int l = 0; l < num_layers; ++l) {
      const uint8_t* keep = snapshot + ((size_t)p * num_layers + l) * 2 * block_bytes;
      memcpy((uint8_t*)k_pools[l] + (size_t)dst * block_bytes, keep, block_bytes);
      memcpy((uint8_t*)v_pools[l] + (size_t)dst * block_bytes, keep + block_bytes, block_bytes);
    }
  }
  free(snapshot);
  return bad ? -1 : 0;
}

/*
 * Swap ([P1] Figure 4): direction 0 copies blocks out,
 *   host[i][l][0] = k_pools[l][block_ids[i]],  host[i][l][1] = v_pools[l][block_ids[i]];
 * direction 1 performs the reverse assignment into the (possibly different) blocks listed.
 */
int pao_swap_blocks(void* const* k_pools, void* const* v_pools, int num_layers, void* host_buf,
                    const int32_t* block_ids, int n, int num_blocks, size_t block_bytes,
                    int direction) {
  for (int i = 0; i < n; ++i)
    if (block_ids[i] < 0 || block_ids[i] >= num_blocks) return -1;
  for (int i = 0; i < n; ++i) {
    for (int l = 0; l < num_layers; ++l) {
      uint8_t* host_k = (uint8_t*)host_buf + (((size_t)i * num_layers + l) * 2 + 0) * block_bytes;
      uint8_t* host_v = (uint8_t*)host_buf + (((size_t)i * num_layers + l) * 2 + 1) * block_bytes;
      uint8_t* dev_k = (uint8_t*)k_pools[l] + (size_t)block_ids[i] * block_bytes;
      uint8_t* dev_v = (uint8_t*)v_pools[l] + (size_t)block_ids[i] * block_bytes;
      if (direction == 0) {
        memcpy(host_k, dev_k, block_bytes);
        memcpy(host_v, dev_v, block_bytes);
      } else {
        memcpy(dev_k, host_k, block_bytes);
        memcpy(dev_v, host_v, block_bytes);
      }
    }
  }
  return 0;
}

