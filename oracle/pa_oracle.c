/*
 * pa_oracle.c -- plain fp64 CPU oracle for paged KV-cache attention (decode
 * and prefill).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test-suite, the smoke check and the CPU-baseline leg
 * of the benchmark use it.  It shares no code, header or constant with the
 * CUDA library; it decodes the stored half/bfloat16 bit patterns itself.
 *
 * What it computes (sources):
 *  - Block count / tail slots: lihaoran.work "auto-20261007-1900", section
 *    "末块会浪费多少空间？" (blocks = ceil(T/b), empty slots = blocks*b - T,
 *    T = 0 allocates nothing, invalid sizes are an error).
 *  - Address of token t: aiqz.cc "paged-attention-mechanism", section
 *    "块表映射机制" (pid = block_table[i], off = j mod B) and lihaoran.work,
 *    section "块表把逻辑顺序映射到物理位置" (logical block t // b, offset t % b).
 *  - Writing a new token into its slot and the copy-on-write block copy:
 *    aiqz.cc, section "前缀共享机制" (allocate, copy the old block, then write).
 *  - Decode attention: every new token attends to all cached history
 *    (aiqz.cc, section "显存痛点"; lihaoran.work: full causal attention still
 *    covers the visible history); the kernel reads K/V by first looking up the
 *    block table (cf-1.com news/5879632, section 5.1).  The formula itself,
 *    softmax(scale * q.K^T) V, and the grouped-query head mapping
 *    kv_head = h / (Hq/Hkv) are not printed on the pages; they are the plain
 *    textbook definition, evaluated here in double precision on the stored
 *    (already rounded) input values, in logical token order.
 *  - Prefill: the prompt's tokens are written into blocks taken as the
 *    request enters (cf-1.com news/5879632, section 3.2) and each attends to
 *    all history before it (aiqz.cc, section "显存痛点"); the causal mask
 *    (a prompt token sees the history and the prompt up to itself) is again
 *    the textbook definition.
 *
 * Layouts (all row-major):
 *   q, out        [S][Hq][D]
 *   k/v pools     [NB][Hkv][B][D]
 *   block_tables  int32 [S][max_blocks]
 *   context_lens  int32 [S]
 *   slot_mapping  int64 [T]          (slot < 0: token skipped)
 *   copy pairs    int64 [P][2]       (src, dst), applied in order
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

static size_t orc_elem_bytes(int dtype) { return dtype == ORC_F32 ? 4u : 2u; }

/* IEEE binary16 -> double, written from the format definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits). */
static double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int ex = (h >> 10) & 0x1f;
  int fr = h & 0x3ff;
  double v;
  if (ex == 0) {
    v = ldexp((double)fr, -24); /* subnormal: fr * 2^-14 * 2^-10 */
  } else if (ex == 31) {
    v = fr ? NAN : INFINITY;
  } else {
    v = ldexp(1.0 + (double)fr / 1024.0, ex - 15);
  }
  return sign ? -v : v;
}

/* bfloat16 is the top half of an IEEE binary32 pattern. */
static double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double orc_load(const void *base, size_t idx, int dtype) {
  if (dtype == ORC_F32) {
    float f;
    memcpy(&f, (const char *)base + idx * 4u, 4);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, (const char *)base + idx * 2u, 2);
  return dtype == ORC_F16 ? orc_half_to_double(h) : orc_bf16_to_double(h);
}

/* blocks = ceil(tokens / block_size), unused = blocks*block_size - tokens.
 * Returns 0, or -1 for tokens < 0 or block_size <= 0. */
int oracle_block_layout(int64_t tokens, int64_t block_size, int64_t *blocks,
                        int64_t *unused) {
  if (tokens < 0 || block_size <= 0) return -1;
  int64_t n = tokens / block_size + (tokens % block_size != 0);
  *blocks = n;
  *unused = n * block_size - tokens;
  return 0;
}

/* Token position t of a sequence -> (physical block, offset in block).
 * Returns 0, or -1 when t is negative or past the table's entries. */
int oracle_locate(const int32_t *table_row, int64_t entries, int64_t t,
                  int64_t block_size, int64_t *pid, int64_t *off) {
  if (t < 0 || block_size <= 0) return -1;
  int64_t logical = t / block_size;
  if (logical >= entries) return -1;
  *pid = table_row[logical];
  *off = t % block_size;
  return 0;
}

/* Slot of token position t: pid * B + off. */
int oracle_slot(const int32_t *table_row, int64_t entries, int64_t t,
                int64_t block_size, int64_t *slot) {
  int64_t pid, off;
  if (oracle_locate(table_row, entries, t, block_size, &pid, &off)) return -1;
  *slot = pid * block_size + off;
  return 0;
}

/* Byte offset of row (pid, head, off) inside a [NB][Hkv][B][D] pool. */
static size_t orc_row(int64_t pid, int64_t head, int64_t off, int Hkv, int B,
                      int D) {
  return (((size_t)pid * (size_t)Hkv + (size_t)head) * (size_t)B + (size_t)off) *
         (size_t)D;
}

/* Scatter each new token's K and V rows into its slot (bit copy).
 * key/value: [T][Hkv][D].  Tokens with slot < 0 are skipped.
 * Returns 0, or -1 if a slot lies outside the pool. */
int oracle_write_kv(const void *key, const void *value, void *k_cache,
                    void *v_cache, const int64_t *slot_mapping, int64_t T,
                    int Hkv, int D, int B, int64_t NB, int dtype) {
  size_t e = orc_elem_bytes(dtype);
  for (int64_t i = 0; i < T; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    if (slot >= NB * (int64_t)B) return -1;
    int64_t pid = slot / B, off = slot % B;
    for (int h = 0; h < Hkv; ++h) {
      size_t src = ((size_t)i * (size_t)Hkv + (size_t)h) * (size_t)D;
      size_t dst = orc_row(pid, h, off, Hkv, B, D);
      memcpy((char *)k_cache + dst * e, (const char *)key + src * e, (size_t)D * e);
      memcpy((char *)v_cache + dst * e, (const char *)value + src * e, (size_t)D * e);
    }
  }
  return 0;
}

/* Copy-on-write block copy: for each (src, dst) pair, in order, the whole
 * physical block (all heads, all slots) of K and of V is copied.
 * Returns 0, or -1 if an id lies outside the pool. */
int oracle_copy_blocks(void *k_cache, void *v_cache, const int64_t *pairs,
                       int64_t P, int Hkv, int D, int B, int64_t NB, int dtype) {
  size_t blk = (size_t)Hkv * (size_t)B * (size_t)D * orc_elem_bytes(dtype);
  for (int64_t p = 0; p < P; ++p) {
    int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= NB || dst < 0 || dst >= NB) return -1;
    if (src == dst) continue;
    memmove((char *)k_cache + (size_t)dst * blk, (char *)k_cache + (size_t)src * blk, blk);
    memmove((char *)v_cache + (size_t)dst * blk, (char *)v_cache + (size_t)src * blk, blk);
  }
  return 0;
}

/* Attention of one query row (element offset qrow in q, query head h) over
 * the first L tokens of a sequence, in logical order.  Returns 0 or -1. */
static int orc_attend_one(double *out_row, const void *q, size_t qrow, const void *k_cache,
                          const void *v_cache, const int32_t *table_row,
                          int64_t max_blocks, int64_t L, int h, int Hq,
                          int Hkv, int D, int B, int64_t NB, double scale,
                          int dtype, double *x) {
  for (int d = 0; d < D; ++d) out_row[d] = 0.0;
  if (L == 0) return 0; /* no cached tokens: nothing to attend to */
  int G = Hq / Hkv;
  int g = h / G; /* query heads are grouped contiguously per KV head */
  double m = -INFINITY;
  for (int64_t t = 0; t < L; ++t) {
    int64_t pid, off;
    if (oracle_locate(table_row, max_blocks, t, B, &pid, &off)) return -1;
    if (pid < 0 || pid >= NB) return -1;
    size_t krow = orc_row(pid, g, off, Hkv, B, D);
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += orc_load(q, qrow + (size_t)d, dtype) * orc_load(k_cache, krow + (size_t)d, dtype);
    x[t] = scale * dot;
    if (x[t] > m) m = x[t];
  }
  double den = 0.0;
  for (int64_t t = 0; t < L; ++t) {
    double w = exp(x[t] - m);
    den += w;
    int64_t pid, off;
    oracle_locate(table_row, max_blocks, t, B, &pid, &off);
    size_t vrow = orc_row(pid, g, off, Hkv, B, D);
    for (int d = 0; d < D; ++d) out_row[d] += w * orc_load(v_cache, vrow + (size_t)d, dtype);
  }
  for (int d = 0; d < D; ++d) out_row[d] /= den;
  return 0;
}

/* out (double) [S][Hq][D] = softmax(scale * q K^T) V per sequence and head,
 * K/V gathered through the block table in logical order.  nthreads <= 0 uses
 * the OpenMP default.  Returns 0, or -1 on an invalid argument or index. */
int oracle_decode(double *out, const void *q, const void *k_cache,
                  const void *v_cache, const int32_t *block_tables,
                  int64_t max_blocks, const int32_t *context_lens, int S, int Hq,
                  int Hkv, int D, int B, int64_t NB, double scale, int dtype,
                  int nthreads) {
  if (S < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || B <= 0) return -1;
  int64_t maxL = 0;
  for (int s = 0; s < S; ++s) {
    if (context_lens[s] < 0 || (int64_t)context_lens[s] > max_blocks * B) return -1;
    if (context_lens[s] > maxL) maxL = context_lens[s];
  }
  int err = 0;
  int64_t work = (int64_t)S * Hq;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel reduction(| : err)
#endif
  {
    double *x = (double *)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
    if (!x) err |= 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t w = 0; w < work; ++w) {
      if (!x) continue;
      int s = (int)(w / Hq), h = (int)(w % Hq);
      double *row = out + (size_t)w * (size_t)D;
      if (orc_attend_one(row, q, (size_t)w * (size_t)D, k_cache, v_cache,
                         block_tables + (size_t)s * (size_t)max_blocks, max_blocks, context_lens[s], h, Hq,
                         Hkv, D, B, NB, scale, dtype, x))
        err |= 1;
    }
    free(x);
  }
  (void)nthreads;
  return err ? -1 : 0;
}

/* Prefill (prompt) attention.  Sequence s owns the query rows
 * q_start[s] .. q_start[s+1]-1 of q / out ([T][Hq][D]); they are the last
 * n = q_start[s+1] - q_start[s] positions of its context, whose length
 * context_lens[s] counts them.  Row i (position p = L - n + i) attends over
 * tokens 0 .. p: the whole cached history, then the prompt up to itself
 * (causal).  Returns 0, or -1 on an invalid argument or index. */
int oracle_prefill(double *out, const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *block_tables, int64_t max_blocks, const int32_t *context_lens,
                   const int32_t *q_start, int S, int Hq, int Hkv, int D, int B, int64_t NB, double scale,
                   int dtype, int nthreads) {
  if (S < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || B <= 0) return -1;
  if (S > 0 && q_start[0] != 0) return -1;
  int64_t maxL = 0;
  for (int s = 0; s < S; ++s) {
    int64_t n = (int64_t)q_start[s + 1] - q_start[s];
    if (n < 0 || context_lens[s] < n || (int64_t)context_lens[s] > max_blocks * B) return -1;
    if (context_lens[s] > maxL) maxL = context_lens[s];
  }
  int64_t T = S > 0 ? q_start[S] : 0;
  int err = 0;
  int64_t work = T * Hq;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel reduction(| : err)
#endif
  {
    double *x = (double *)malloc(sizeof(double) * (size_t)(maxL > 0 ? maxL : 1));
    if (!x) err |= 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
    for (int64_t w = 0; w < work; ++w) {
      if (!x) continue;
      int64_t row = w / Hq;
      int h = (int)(w % Hq);
      int s = 0;
      while (s + 1 < S && q_start[s + 1] <= row) ++s; /* the sequence owning query row `row` */
      int64_t n = (int64_t)q_start[s + 1] - q_start[s];
      int64_t p = (int64_t)context_lens[s] - n + (row - q_start[s]);
      if (orc_attend_one(out + (size_t)w * (size_t)D, q, (size_t)w * (size_t)D, k_cache, v_cache,
                         block_tables + (size_t)s * (size_t)max_blocks, max_blocks, p + 1, h, Hq, Hkv, D, B,
                         NB, scale, dtype, x))
        err |= 1;
    }
    free(x);
  }
  (void)nthreads;
  return err ? -1 : 0;
}

/* Threads the OpenMP runtime would use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
