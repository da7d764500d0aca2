/*
 * cpmla_oracle.c -- plain fp64 CPU oracle for context-parallel (PCP) prefill
 * attention over MLA latent KV.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library under context_sparse_mla_gb300/csrc.
 *
 * What it follows (page titles and sections of the source pages):
 *   - "[Core] Add MRV2 virtual-batch PCP for MLA", section "DualChunkSwap
 *     partitioning" and its PCP=4 diagram: a request is cut into 2P contiguous
 *     chunks; shard r takes chunks r and 2P-1-r.
 *   - same page, section "PCP algorithm": every prefill is partitioned on its
 *     own; decode rows are replicated on every shard.
 *   - same page, "DualChunkSwap partitioning" (last paragraphs): the full
 *     latent KV is visible to every shard; outputs are restored to global
 *     token order.
 *   - "[DeepSeekV4][PCP] Enable context-parallel prefill for hybrid KV and
 *     MegaMoE", "Implementation summary" and "Main challenges": each shard
 *     computes a partial attention (output + log-sum-exp), the partials are
 *     merged globally by LSE and the attention sink is applied once, after
 *     the merge, never per shard.
 *
 * Readings taken where the pages are silent (labels used below):
 *   R1 sink = one extra logit per head, zero value vector, same units as the
 *      scaled scores: O_final = O * e^L / (e^L + e^sink).
 *   R3 returned LSE is natural-log and excludes the sink.
 *   R4 chunk sizes when S mod 2P != 0: base = S / 2P, the first S mod 2P
 *      chunks get one extra token.
 *   R5 row order inside a shard: requests in input order; inside a request the
 *      rows of chunk r then chunk 2P-1-r, ascending; a decode request's single
 *      row sits in its request slot in every shard and is owned by shard 0.
 *   R6 causal boundary inclusive: a token at position t sees keys 0..t.
 *   R8 fp8 latent is OCP E4M3 (bias 7, max 448, no infinities; S.1111.111 is
 *      NaN) times one fp32 scale per token per 128-channel group.
 *
 * Every floating-point step is done in double from the stored bf16 / fp8
 * values.  No blocking, fusion or reordering beyond the definitions below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_DQK 576 /* absorbed latent (512) + rope (64) */
#define ORC_DV 512  /* latent part, which is also the value */
#define ORC_DROPE 64
#define ORC_GROUP 128 /* fp8 scale group width along the latent */

/* ---------------------------------------------------------------- decoding */

/* bf16 -> double: the 16 stored bits are the high half of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* OCP 8-bit E4M3 -> double, from the format's bit fields (R8). */
double oracle_e4m3_to_double(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int e = (byte >> 3) & 0xF;
  int m = byte & 0x7;
  double v;
  if (e == 0xF && m == 0x7) return NAN; /* the only non-finite encodings */
  if (e == 0)
    v = ldexp((double)m / 8.0, 1 - 7); /* subnormal: 0.m * 2^(1-bias) */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* --------------------------------------------------------------- partition */

/* Start and length of chunk c of a request of S tokens cut into n chunks (R4). */
static void orc_chunk(int S, int n, int c, int *start, int *len) {
  int base = S / n, rem = S % n;
  *start = c * base + (c < rem ? c : rem);
  *len = base + (c < rem ? 1 : 0);
}

/*
 * Total number of shard rows the partition produces (decode rows counted once
 * per shard since they are replicated).
 */
long long oracle_partition_rows(int P, int B, const int32_t *cu_seqlens,
                                const uint8_t *is_decode) {
  long long n = 0;
  for (int b = 0; b < B; ++b) {
    int S = cu_seqlens[b + 1] - cu_seqlens[b];
    n += is_decode[b] ? (long long)P * S : S;
  }
  return n;
}

/*
 * DualChunkSwap partition of a global batch into P virtual shards.
 *   cu_seqlens[B+1]  global token offsets of each request's scheduled tokens
 *   q_start_pos[B]   position of each request's first scheduled token
 *   is_decode[B]     1 = decode request (replicated), 0 = prefill
 * Outputs (caller-owned):
 *   shard_offsets[P+1]          row ranges of each shard in the row arrays
 *   rows/pos/req[n_rows_total]  global token id, position, request of a row
 *   owner_shard/owner_row[T]    for each global token, the shard and the
 *                               index (into the concatenated row arrays) of
 *                               the one row whose result is kept.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_partition(int P, int B, const int32_t *cu_seqlens,
                     const int32_t *q_start_pos, const uint8_t *is_decode,
                     int32_t *shard_offsets, int32_t *rows, int32_t *pos,
                     int32_t *req, int32_t *owner_shard, int32_t *owner_row) {
  if (P < 1 || B < 0) return -1;
  int n = 0;
  for (int r = 0; r < P; ++r) {
    shard_offsets[r] = n;
    for (int b = 0; b < B; ++b) {
      int g0 = cu_seqlens[b];
      int S = cu_seqlens[b + 1] - g0;
      if (S < 0) return -1;
      if (is_decode[b]) {
        /* replicated rows (R5): every shard computes them, shard 0 owns them */
        for (int i = 0; i < S; ++i) {
          rows[n] = g0 + i;
          pos[n] = q_start_pos[b] + i;
          req[n] = b;
          if (r == 0) {
            owner_shard[g0 + i] = 0;
            owner_row[g0 + i] = n;
          }
          ++n;
        }
        continue;
      }
      int chunk_ids[2] = {r, 2 * P - 1 - r};
      for (int k = 0; k < 2; ++k) {
        int st, len;
        orc_chunk(S, 2 * P, chunk_ids[k], &st, &len);
        for (int i = st; i < st + len; ++i) {
          rows[n] = g0 + i;
          pos[n] = q_start_pos[b] + i;
          req[n] = b;
          owner_shard[g0 + i] = r;
          owner_row[g0 + i] = n;
          ++n;
        }
      }
    }
  }
  shard_offsets[P] = n;
  return 0;
}

/* -------------------------------------------------------------- attention */

/* Value of latent-KV element d of global KV row j, in double. */
static double orc_kv(int fmt, const uint16_t *kv_bf16, const uint8_t *kv_fp8,
                     const float *kv_scale, const uint16_t *kv_rope, long long j,
                     int d) {
  if (fmt == 0) return oracle_bf16_to_double(kv_bf16[j * ORC_DQK + d]);
  if (d < ORC_DV)
    return oracle_e4m3_to_double(kv_fp8[j * ORC_DV + d]) *
           (double)kv_scale[j * (ORC_DV / ORC_GROUP) + d / ORC_GROUP];
  return oracle_bf16_to_double(kv_rope[j * ORC_DROPE + (d - ORC_DV)]);
}

/*
 * Plain definition of attention for n query rows, all H heads each.
 *
 * For row i (request-local position t = pos[i], KV rows of its request start
 * at kv_start[i]) the key set J is
 *   dense  (topk == NULL): positions 0..t                          (R6)
 *   sparse (topk != NULL): the entries >= 0 of topk[i*k .. i*k+k-1]
 * intersected with [kv_lo[i], kv_hi[i]] when those arrays are given (they
 * restrict a row to part of its keys, which is how KV-split partials are made).
 * For head h:  s_j = scale * sum_{d<576} q[i,h,d] * kv[j,d]
 *              L   = ln sum_j exp(s_j)           (-inf when J is empty)
 *              O   = sum_j exp(s_j - L) * kv[j, 0:512]   (0 when J is empty)
 * If sink != NULL the sink of head h is applied to O (R1):
 *              O  *= 1 / (1 + exp(sink[h] - L))
 * and the LSE written out is still L (R3).
 *
 * q: bf16 bits [n, H, 576] (the n rows' queries, compact).
 * KV format fmt: 0 = bf16 [*, 576]; 1 = e4m3 latent [*, 512] + fp32 scale
 * [*, 4] + bf16 rope [*, 64].
 * Outputs: o [n, H, 512] and lse [n, H], double.
 * Returns 0, or -1 when an index points outside 0..t.
 */
int oracle_attention(int n, int H, const uint16_t *q, const int32_t *pos,
                     const long long *kv_start, int fmt, const uint16_t *kv_bf16,
                     const uint8_t *kv_fp8, const float *kv_scale,
                     const uint16_t *kv_rope, const int32_t *topk, int k,
                     const int32_t *kv_lo, const int32_t *kv_hi, double scale,
                     const float *sink, double *o, double *lse) {
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n; ++i) {
    int t = pos[i];
    int nkeys = topk ? k : t + 1;
    int lo = kv_lo ? kv_lo[i] : 0;
    int hi = kv_hi ? kv_hi[i] : t;
    size_t cap = (size_t)(nkeys > 0 ? nkeys : 1);
    int32_t *keys = (int32_t *)malloc(sizeof(int32_t) * cap);
    double *s = (double *)malloc(sizeof(double) * cap * (size_t)H);
    double *qd = (double *)malloc(sizeof(double) * (size_t)H * ORC_DQK);
    double *kvd = (double *)malloc(sizeof(double) * ORC_DQK);
    double *L = (double *)malloc(sizeof(double) * (size_t)H);
    /* key positions of this row */
    int m = 0;
    for (int e = 0; e < nkeys; ++e) {
      int p = topk ? topk[(long long)i * k + e] : e;
      if (p < 0) continue;
      if (p > t) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      if (p < lo || p > hi) continue;
      keys[m++] = p;
    }
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < ORC_DQK; ++d)
        qd[h * ORC_DQK + d] = oracle_bf16_to_double(q[((long long)i * H + h) * ORC_DQK + d]);
    /* scores s[h][e] = scale * q_h . kv_j */
    for (int e = 0; e < m; ++e) {
      long long j = kv_start[i] + keys[e];
      for (int d = 0; d < ORC_DQK; ++d)
        kvd[d] = orc_kv(fmt, kv_bf16, kv_fp8, kv_scale, kv_rope, j, d);
      for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int d = 0; d < ORC_DQK; ++d) acc += qd[h * ORC_DQK + d] * kvd[d];
        s[(size_t)h * cap + e] = scale * acc;
      }
    }
    /* L_h = ln sum_j exp(s_hj), computed as max + ln sum exp(s - max) */
    for (int h = 0; h < H; ++h) {
      if (m == 0) {
        L[h] = -INFINITY;
        continue;
      }
      double mx = -INFINITY;
      for (int e = 0; e < m; ++e)
        if (s[(size_t)h * cap + e] > mx) mx = s[(size_t)h * cap + e];
      double z = 0.0;
      for (int e = 0; e < m; ++e) z += exp(s[(size_t)h * cap + e] - mx);
      L[h] = mx + log(z);
    }
    /* O_h = sum_j exp(s_hj - L_h) * kv_j[0:512] */
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < ORC_DV; ++d) o[((long long)i * H + h) * ORC_DV + d] = 0.0;
    for (int e = 0; e < m; ++e) {
      long long j = kv_start[i] + keys[e];
      for (int d = 0; d < ORC_DV; ++d)
        kvd[d] = orc_kv(fmt, kv_bf16, kv_fp8, kv_scale, kv_rope, j, d);
      for (int h = 0; h < H; ++h) {
        double w = exp(s[(size_t)h * cap + e] - L[h]);
        double *oh = o + ((long long)i * H + h) * ORC_DV;
        for (int d = 0; d < ORC_DV; ++d) oh[d] += w * kvd[d];
      }
    }
    for (int h = 0; h < H; ++h) {
      if (sink && m > 0) {
        double f = 1.0 / (1.0 + exp((double)sink[h] - L[h]));
        double *oh = o + ((long long)i * H + h) * ORC_DV;
        for (int d = 0; d < ORC_DV; ++d) oh[d] *= f;
      }
      lse[(long long)i * H + h] = L[h];
    }
    free(keys);
    free(s);
    free(qd);
    free(kvd);
    free(L);
  }
  return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ merge */

/*
 * Global LSE merge of partial results, then the sink once, then restore to
 * global order.
 *   partial o [n_part, H, 512], lse [n_part, H] (double, sink NOT applied).
 *   For global row g the contributing partial rows are
 *   contrib_rows[contrib_off[g] .. contrib_off[g+1]-1].
 *   L   = ln sum_c exp(lse_c)             (-inf if every lse_c is -inf)
 *   O   = sum_c exp(lse_c - L) * o_c      (0 then)
 *   O  *= 1 / (1 + exp(sink[h] - L))      (if sink != NULL)
 * Outputs o_out [T, H, 512], lse_out [T, H] in global order.
 */
void oracle_merge(int T, int H, const double *o_part, const double *lse_part,
                  const int32_t *contrib_off, const int32_t *contrib_rows,
                  const float *sink, double *o_out, double *lse_out) {
#pragma omp parallel for schedule(static)
  for (int g = 0; g < T; ++g) {
    for (int h = 0; h < H; ++h) {
      double *og = o_out + ((long long)g * H + h) * ORC_DV;
      for (int d = 0; d < ORC_DV; ++d) og[d] = 0.0;
      double mx = -INFINITY;
      for (int c = contrib_off[g]; c < contrib_off[g + 1]; ++c) {
        double l = lse_part[(long long)contrib_rows[c] * H + h];
        if (l > mx) mx = l;
      }
      if (mx == -INFINITY) {
        lse_out[(long long)g * H + h] = -INFINITY;
        continue;
      }
      double z = 0.0;
      for (int c = contrib_off[g]; c < contrib_off[g + 1]; ++c)
        z += exp(lse_part[(long long)contrib_rows[c] * H + h] - mx);
      double L = mx + log(z);
      for (int c = contrib_off[g]; c < contrib_off[g + 1]; ++c) {
        long long r = contrib_rows[c];
        double w = exp(lse_part[r * H + h] - L);
        const double *oc = o_part + (r * H + h) * ORC_DV;
        for (int d = 0; d < ORC_DV; ++d) og[d] += w * oc[d];
      }
      if (sink) {
        double f = 1.0 / (1.0 + exp((double)sink[h] - L));
        for (int d = 0; d < ORC_DV; ++d) og[d] *= f;
      }
      lse_out[(long long)g * H + h] = L;
    }
  }
}

/* --------------------------------------------------------- cache insertion */
/*
 * "[Core] Add MRV2 virtual-batch PCP for MLA", Summary (sparse MLA cache
 * insertion) and "DualChunkSwap partitioning" (the all-gathered latent KV is
 * what the cache insertion writes); the "fp8_ds_mla" KV-cache dtype of
 * "[Feature][PCP] Add DeepSeek-V4.1-Flash support".  The pages fix neither
 * the fp8 layout nor the quantisation rule.  Readings (R13):
 *   token t with slot s >= 0 goes to cache row s; s = -1 skips the token;
 *   bf16 cache: the 576 values copied;
 *   fp8 cache (R8 layout): per 128-channel latent group, amax = max |x|,
 *   scale = amax / 448 in binary32 (1 when amax == 0), code = E4M3(x / scale)
 *   with the quotient in binary32 and E4M3 rounding to nearest, ties to even,
 *   saturating at +-448; the rope copied as bf16.
 * The codes are integers decided by binary32 arithmetic, so the oracle takes
 * those decisions in binary32 -- the precision the kernel takes them in.
 */

/* Round-half-to-even of a non-negative double to an integer value. */
static double orc_round_half_even(double q) {
  double fl = floor(q), d = q - fl;
  if (d > 0.5) return fl + 1.0;
  if (d < 0.5) return fl;
  return fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;
}

/* binary32 -> OCP E4M3 byte (R8 format: 3 fraction bits, exponent bias 7,
 * normal exponents -6..8, subnormals m * 2^-9): round to nearest, ties to
 * even; every finite value at or above 448 in magnitude (and infinity)
 * saturates to +-448; NaN gives 0x7F. */
uint8_t oracle_e4m3_encode(float f) {
  if (isnan(f)) return 0x7F;
  const uint8_t sign = signbit(f) ? 0x80 : 0x00;
  const double a = fabs((double)f);
  if (a >= 448.0) return sign | 0x7E; /* 448 is the largest finite value */
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);        /* a = frac * 2^e2, frac in [0.5, 1) */
  int ex = e2 - 1;      /* floor(log2 a) */
  if (ex < -6) ex = -6; /* below 2^-6 the subnormal step 2^-9 */
  const double quantum = ldexp(1.0, ex - 3);
  const double v = orc_round_half_even(a / quantum) * quantum; /* <= 448 */
  if (v == 0.0) return sign;
  int ev2;
  frexp(v, &ev2);
  const int ev = ev2 - 1;
  if (ev < -6) return sign | (uint8_t)(v / ldexp(1.0, -9)); /* subnormal m */
  const int m = (int)((v / ldexp(1.0, ev) - 1.0) * 8.0);
  return sign | (uint8_t)(((ev + 7) << 3) | m);
}

/* Insert n tokens' latent KV (bf16 [n, 576]) into the cache rows slot[t]
 * (R13).  fmt 0: cache_bf16 [s_cache, 576]; fmt 1: cache_fp8 [s_cache, 512],
 * cache_scale [s_cache, 4], cache_rope [s_cache, 64].  Returns -1 if a slot
 * lies outside [-1, s_cache). */
int oracle_kv_insert(int n, const uint16_t *kv, const int64_t *slot, int fmt, long long s_cache,
                     uint16_t *cache_bf16, uint8_t *cache_fp8, float *cache_scale,
                     uint16_t *cache_rope) {
  for (int t = 0; t < n; ++t)
    if (slot[t] < -1 || slot[t] >= s_cache) return -1;
  for (int t = 0; t < n; ++t) {
    const long long s = slot[t];
    if (s < 0) continue;
    const uint16_t *x = kv + (long long)t * ORC_DQK;
    if (fmt == 0) {
      memcpy(cache_bf16 + s * ORC_DQK, x, ORC_DQK * sizeof(uint16_t));
      continue;
    }
    for (int g = 0; g < ORC_DV / ORC_GROUP; ++g) {
      float amax = 0.0f;
      for (int d = 0; d < ORC_GROUP; ++d) {
        const float v = fabsf((float)oracle_bf16_to_double(x[g * ORC_GROUP + d]));
        if (v > amax) amax = v;
      }
      const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
      cache_scale[s * 4 + g] = scale;
      for (int d = 0; d < ORC_GROUP; ++d) {
        const float v = (float)oracle_bf16_to_double(x[g * ORC_GROUP + d]);
        cache_fp8[s * ORC_DV + g * ORC_GROUP + d] = oracle_e4m3_encode(v / scale);
      }
    }
    memcpy(cache_rope + s * ORC_DROPE, x + ORC_DV, ORC_DROPE * sizeof(uint16_t));
  }
  return 0;
}
