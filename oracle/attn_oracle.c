/*
 * FP64 CPU oracle for the tiled attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline leg use it.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes is the plain definition of attention, not the tiled
 * streaming algorithm:
 *   - "FlashAttention（V3）深度解析" (dtcms.com), section 2 "注意力机制基础":
 *       S = Q K^T, P = softmax(S), O = P V.
 *   - same page, section 11, function standard_attention: the scores are
 *       divided by sqrt(head_dim) before the softmax; here the factor is the
 *       caller's `scale` (1/sqrt(d) in every workload).
 *   - same page, section 11, FlashAttention3._apply_causal_mask: key j is
 *       kept for query i iff i >= j, with absolute indices from 0
 *       (top-left alignment, also when Nq != Nk).
 *   - the log-sum-exp is not defined on the pages; it is taken as
 *       LSE_i = ln sum_{j allowed} exp(scale * q_i . k_j)   (natural log).
 *   - grouped-query heads: the pages only name HEAD_NUM_KV (section 7.4,
 *       TransposeVLayout); query head h reads key/value head
 *       h / (Hq / Hkv) (contiguous groups).
 *
 * Two passes per row, in double precision: all allowed logits first, then
 * their maximum, then the exponentials, their sum and the weighted sum of V.
 * No online/streaming rescaling appears here, so the oracle does not share
 * the GPU kernel's arithmetic.
 *
 * Element types of the raw inputs: 0 = IEEE binary16, 1 = bfloat16,
 * 2 = binary32, 3 = binary64.  The 16-bit decoders are written out from the
 * formats' definitions below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1
#define ORACLE_F32 2
#define ORACLE_F64 3

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp(1.0 + (double)f / 1024.0, e - 15);
  }
  return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double decode_bf16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xff;
  int f = h & 0x7f;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -133); /* f * 2^-126 * 2^-7 */
  } else if (e == 255) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp(1.0 + (double)f / 128.0, e - 127);
  }
  return sign ? -v : v;
}

static double decode_one(const void* base, long long idx, int elem) {
  switch (elem) {
    case ORACLE_F16: return decode_f16(((const uint16_t*)base)[idx]);
    case ORACLE_BF16: return decode_bf16(((const uint16_t*)base)[idx]);
    case ORACLE_F32: return (double)((const float*)base)[idx];
    default: return ((const double*)base)[idx];
  }
}

/* Decode n raw elements to double (exported so tests can pin the decoders
 * against an independent library conversion). */
int oracle_decode(const void* in, int elem, long long n, double* out) {
  if (elem < 0 || elem > 3 || n < 0 || (n > 0 && (!in || !out))) return -1;
  for (long long i = 0; i < n; ++i) out[i] = decode_one(in, i, elem);
  return 0;
}

typedef struct {
  const void* q_rows;
  const double* k; /* decoded [B][Nk][Hkv][d] */
  const double* v;
  int elem;
  long long B, Hq, Hkv, Nk, d;
  int causal;
  double scale;
  const long long *row_b, *row_h, *row_i;
  long long r_begin, r_end;
  double* o_out;
  double* lse_out;
  int status;
} row_job;

static void* row_worker(void* arg) {
  row_job* J = (row_job*)arg;
  const long long d = J->d, Nk = J->Nk, Hkv = J->Hkv;
  const long long group = J->Hq / J->Hkv;
  double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double* q = (double*)malloc(sizeof(double) * (size_t)d);
  if (!s || !q) {
    free(s);
    free(q);
    J->status = -2;
    return NULL;
  }
  for (long long r = J->r_begin; r < J->r_end; ++r) {
    const long long b = J->row_b[r], h = J->row_h[r], i = J->row_i[r];
    const long long hk = h / group;
    for (long long c = 0; c < d; ++c) q[c] = decode_one(J->q_rows, r * d + c, J->elem);

    /* allowed keys: j < Nk, and j <= i under the causal rule */
    long long jn = Nk;
    if (J->causal && i + 1 < jn) jn = i + 1;

    /* pass 1: logits and their maximum */
    double m = -INFINITY;
    for (long long j = 0; j < jn; ++j) {
      const double* kr = J->k + ((b * Nk + j) * Hkv + hk) * d;
      double acc = 0.0;
      for (long long c = 0; c < d; ++c) acc += q[c] * kr[c];
      s[j] = J->scale * acc;
      if (s[j] > m) m = s[j];
    }
    /* pass 2: exponentials, their sum, and the weighted sum of V */
    double* o = J->o_out + r * d;
    for (long long c = 0; c < d; ++c) o[c] = 0.0;
    double z = 0.0;
    for (long long j = 0; j < jn; ++j) {
      const double e = exp(s[j] - m);
      z += e;
      const double* vr = J->v + ((b * Nk + j) * Hkv + hk) * d;
      for (long long c = 0; c < d; ++c) o[c] += e * vr[c];
    }
    for (long long c = 0; c < d; ++c) o[c] /= z;
    J->lse_out[r] = m + log(z);
  }
  free(s);
  free(q);
  return NULL;
}

typedef struct {
  const void* in;
  int elem;
  long long begin, end;
  double* out;
} decode_job;

static void* decode_worker(void* arg) {
  decode_job* J = (decode_job*)arg;
  for (long long i = J->begin; i < J->end; ++i) J->out[i] = decode_one(J->in, i, J->elem);
  return NULL;
}

static void parallel_decode(const void* in, int elem, long long n, double* out, int nthreads) {
  pthread_t th[256];
  decode_job jobs[256];
  const long long chunk = (n + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].in = in;
    jobs[t].elem = elem;
    jobs[t].begin = t * chunk < n ? t * chunk : n;
    jobs[t].end = (t + 1) * chunk < n ? (t + 1) * chunk : n;
    jobs[t].out = out;
    if (pthread_create(&th[started], NULL, decode_worker, &jobs[t]) == 0)
      ++started;
    else
      decode_worker(&jobs[t]); /* no thread available: do the chunk here */
  }
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

/*
 * Attention for R selected query rows.
 *   q_rows : [R][d] raw elements; row r is query (row_b[r], row_h[r], row_i[r])
 *   k, v   : [B][Nk][Hkv][d] raw elements (BSHD, d innermost)
 *   o_out  : [R][d] double;  lse_out : [R] double (natural log)
 * Returns 0, or -1 on a bad argument, -2 on allocation failure.
 */
int oracle_attention_rows(const void* q_rows, const void* k, const void* v, int elem, long long B,
                          long long Hq, long long Hkv, long long Nk, long long d, int causal,
                          double scale, const long long* row_b, const long long* row_h,
                          const long long* row_i, long long R, double* o_out, double* lse_out,
                          int nthreads) {
  if (elem < 0 || elem > 3 || B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Nk < 1 || d < 1 ||
      R < 0)
    return -1;
  if (R == 0) return 0;
  if (!q_rows || !k || !v || !row_b || !row_h || !row_i || !o_out || !lse_out) return -1;
  for (long long r = 0; r < R; ++r)
    if (row_b[r] < 0 || row_b[r] >= B || row_h[r] < 0 || row_h[r] >= Hq || row_i[r] < 0) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;

  const long long nkv = B * Nk * Hkv * d;
  double* kd = (double*)malloc(sizeof(double) * (size_t)nkv);
  double* vd = (double*)malloc(sizeof(double) * (size_t)nkv);
  if (!kd || !vd) {
    free(kd);
    free(vd);
    return -2;
  }
  parallel_decode(k, elem, nkv, kd, nthreads);
  parallel_decode(v, elem, nkv, vd, nthreads);

  if (nthreads > R) nthreads = (int)R;
  pthread_t th[256];
  row_job jobs[256];
  long long chunk = (R + nthreads - 1) / nthreads;
  int nstarted = 0;
  int ok = 0;
  for (int t = 0; t < nthreads; ++t) {
    row_job* J = &jobs[t];
    J->q_rows = q_rows;
    J->k = kd;
    J->v = vd;
    J->elem = elem;
    J->B = B;
    J->Hq = Hq;
    J->Hkv = Hkv;
    J->Nk = Nk;
    J->d = d;
    J->causal = causal;
    J->scale = scale;
    J->row_b = row_b;
    J->row_h = row_h;
    J->row_i = row_i;
    J->r_begin = t * chunk < R ? t * chunk : R;
    J->r_end = (t + 1) * chunk < R ? (t + 1) * chunk : R;
    J->o_out = o_out;
    J->lse_out = lse_out;
    J->status = 0;
  }
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[nstarted], NULL, row_worker, &jobs[t]) == 0)
      ++nstarted;
    else
      row_worker(&jobs[t]);
  }
  for (int t = 0; t < nstarted; ++t) pthread_join(th[t], NULL);
  for (int t = 0; t < nthreads; ++t)
    if (jobs[t].status != 0) ok = jobs[t].status;
  free(kd);
  free(vd);
  return ok;
}
