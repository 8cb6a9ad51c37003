/*
 * Plain C statement of the W4A16 layer, for timing the CPU baseline.
 *
 * TEST INFRASTRUCTURE ONLY, like the rest of this directory: nothing in the
 * product package links or calls it; bench.py's CPU-baseline legs and the tests
 * that pin it to the numpy oracle (w4_oracle.py) do. It shares no code with
 * the CUDA path.
 *
 * What it computes (vLLM API docs, inc.schemes.inc_w4a8_linear, class
 * docstring: the W4A16 path reads the GPTQ qweight; vllm-omni
 * quantization/cpu_int4.py, module docstring: w = (q - 8) * scale + zero):
 *
 *   r[m, n] = fp32( sum_k x[m, k] * ((q[k, n] - 8) * s[k / g, n] + z[k / g, n]) + bias[n] )
 *
 * with q the code of input column k, output n: nibble k % 8 (bits 4 (k % 8)
 * and up) of word [k / 8, n] of the GPTQ int32 qweight [K/8, N]. Every product
 * and sum is in double precision; the result is rounded once to float. x,
 * zeros and bias are bf16 bit patterns, the scales fp16 or bf16 bit patterns.
 *
 * Threads split the output columns; within a thread the loops run over k
 * (one weight row at a time, contiguous in n) and accumulate into a double
 * per (token, column).
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bits -> double: the top half of an IEEE binary32. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* IEEE binary16 bits -> double: 1 sign bit, 5 exponent bits (bias 15), 10
 * fraction bits; exponent 0 holds zero and the subnormals m * 2^-24. Infinity
 * and NaN are outside the layer's inputs and come out as large finite values. */
static double half_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = (double)m / 16777216.0; /* m * 2^-24 */
  } else {
    v = (1.0 + (double)m / 1024.0);
    int p = e - 15;
    while (p > 0) { v *= 2.0; --p; }
    while (p < 0) { v *= 0.5; ++p; }
  }
  return sign ? -v : v;
}

struct job {
  const uint16_t* x;
  const int32_t* qweight;
  const uint16_t* scale;
  const uint16_t* zeros;
  const uint16_t* bias;
  float* out;
  int64_t M, K, N, n0, n1;
  int64_t group;
  int scale_bf16;
  int status;
};

static void* run_block(void* arg) {
  struct job* j = (struct job*)arg;
  const int64_t w = j->n1 - j->n0;
  double* acc = (double*)calloc((size_t)(j->M * w), sizeof(double));
  double* wrow = (double*)malloc((size_t)w * sizeof(double));
  double* srow = (double*)malloc((size_t)w * sizeof(double));
  double* zrow = (double*)malloc((size_t)w * sizeof(double));
  if (acc == NULL || wrow == NULL || srow == NULL || zrow == NULL) {
    free(acc);
    free(wrow);
    free(srow);
    free(zrow);
    j->status = 1;
    return NULL;
  }
  for (int64_t k = 0; k < j->K; ++k) {
    const int64_t g = k / j->group;
    if (k % j->group == 0) {
      /* this group's scales and zeros for the thread's outputs */
      for (int64_t c = 0; c < w; ++c) {
        const int64_t n = j->n0 + c;
        const uint16_t sb = j->scale[g * j->N + n];
        srow[c] = j->scale_bf16 ? bf16_to_double(sb) : half_to_double(sb);
        zrow[c] = j->zeros ? bf16_to_double(j->zeros[g * j->N + n]) : 0.0;
      }
    }
    const int shift = (int)(4 * (k % 8));
    const int32_t* qrow = j->qweight + (k / 8) * j->N + j->n0;
    /* the dequantized weights of input column k for this thread's outputs */
    for (int64_t c = 0; c < w; ++c) {
      const int q = (int)(((uint32_t)qrow[c] >> shift) & 0xFu);
      wrow[c] = (double)(q - 8) * srow[c] + zrow[c];
    }
    for (int64_t m = 0; m < j->M; ++m) {
      const double xv = bf16_to_double(j->x[m * j->K + k]);
      double* a = acc + m * w;
      for (int64_t c = 0; c < w; ++c) a[c] += xv * wrow[c];
    }
  }
  for (int64_t m = 0; m < j->M; ++m)
    for (int64_t c = 0; c < w; ++c) {
      const int64_t n = j->n0 + c;
      const double b = j->bias ? bf16_to_double(j->bias[n]) : 0.0;
      j->out[m * j->N + n] = (float)(acc[m * w + c] + b);
    }
  free(acc);
  free(wrow);
  free(srow);
  free(zrow);
  j->status = 0;
  return NULL;
}

/* Returns 0 on success, nonzero on bad arguments or a failed allocation. */
int w4o_w4a16_linear(const uint16_t* x, int64_t M, int64_t K, const int32_t* qweight, int64_t N,
                     const uint16_t* scale, int scale_bf16, const uint16_t* zeros, int64_t group,
                     const uint16_t* bias, float* out, int nthreads) {
  if (M < 0 || K <= 0 || N <= 0 || K % 8 != 0) return 2;
  const int64_t g = group == -1 ? K : group;
  if (g <= 0 || K % g != 0) return 2;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > N) nthreads = (int)N;
  struct job* jobs = (struct job*)calloc((size_t)nthreads, sizeof(struct job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  char* started = (char*)calloc((size_t)nthreads, 1);
  if (jobs == NULL || tids == NULL || started == NULL) {
    free(jobs);
    free(tids);
    free(started);
    return 1;
  }
  int rc = 0;
  for (int t = 0; t < nthreads; ++t) {
    struct job* j = &jobs[t];
    j->x = x;
    j->qweight = qweight;
    j->scale = scale;
    j->zeros = zeros;
    j->bias = bias;
    j->out = out;
    j->M = M;
    j->K = K;
    j->N = N;
    j->n0 = N * t / nthreads;
    j->n1 = N * (t + 1) / nthreads;
    j->group = g;
    j->scale_bf16 = scale_bf16;
    j->status = 1;
    if (pthread_create(&tids[t], NULL, run_block, j) == 0)
      started[t] = 1;
    else
      run_block(j); /* no thread to spare: do this block here */
  }
  for (int t = 0; t < nthreads; ++t) {
    if (started[t]) pthread_join(tids[t], NULL);
    rc |= jobs[t].status;
  }
  free(jobs);
  free(tids);
  free(started);
  return rc;
}
