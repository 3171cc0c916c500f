/*
 * Plain CPU reference ("oracle") for the 2D convolution forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code with the CUDA library.
 *
 * Every routine is the textbook definition written out as loops, with no
 * blocking, fusion or reordering:
 *
 *  - oracle_conv2d_f64: the nested-loop direct convolution of the
 *    razer666.cn post "卷积总结", section "最原始的卷积实现" (six loops over
 *    filter, channel, output row, output column, kernel row, kernel column,
 *    seven with the batch), generalised by the stride, dilation and padding
 *    that the same section names as the parameters it leaves out.  The post's
 *    pseudocode indexes the output as [filter, channel, out_h, out_h]; the
 *    plain reading (and the only one consistent with its stated output shape
 *    [num_filters, output_height, output_width]) is [filter, out_h, out_w]
 *    with the channel index summed.  It is cross-correlation (no kernel flip):
 *    the same post's "稀疏连接" worked example gives s1 = a*k1+b*k2+e*k3+f*k4
 *    for the top-left window.  Arithmetic is IEEE fp64.
 *  - oracle_conv2d_i8: the same loops over int8 operands with an exact
 *    integer accumulator (the 96x.com.cn MegEngine Beta report, section
 *    "推理：高效原生 int8 实现"), followed by the requantisation this library
 *    defines (the pages give no formula): t = acc + bias (int32),
 *    q = clamp(round_half_even(fp32(t) * scale[k]), -128, 127), then ReLU.
 *    The fp32 steps are written with explicit float variables; this file is
 *    compiled with -ffp-contract=off and without fast-math.
 *  - oracle_round_bf16 / oracle_round_f16: round-to-nearest-even of an fp32
 *    value to bfloat16 / IEEE half, returned as a float, by the bit-level
 *    definition of the two formats.
 *  - oracle_maxpool2d / oracle_global_avgpool: the plain pooling definitions
 *    used by the ResNet-50 forward pass (max over a window with -inf outside
 *    the image; mean over all pixels).
 *
 * Layouts follow the post ("存储顺序和行主序"): row-major NCHW activations,
 * weights [K][C/groups][R][S].
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline int64_t out_dim(int64_t in, int k, int stride, int pad, int dil) {
  return (in + 2 * pad - (int64_t)dil * (k - 1) - 1) / stride + 1;
}

/* Output spatial size: floor((H + 2*pad - dil*(R-1) - 1)/stride) + 1. */
int64_t oracle_out_dim(int64_t in, int k, int stride, int pad, int dil) {
  return out_dim(in, k, stride, pad, dil);
}

static double apply_act(double v, int act) {
  if (act == 1) return v > 0.0 ? v : 0.0;
  if (act == 2) return v < 0.0 ? 0.0 : (v > 6.0 ? 6.0 : v);
  return v;
}

/* One output element of the direct convolution:
 *   y[n,k,oh,ow] = b[k] + sum_{c in group(k)} sum_r sum_s
 *                  w[k, c - g*Cg, r, s] * x[n, c, oh*st - pad + r*dil, ow*st - pad + s*dil]
 * with x = 0 outside the image, then + residual, then the activation. */
static double conv_point_f64(int C, int H, int W, int K, int R, int S, int stride, int pad,
                             int dil, int groups, const double* x, const double* w,
                             const double* b, const double* res, int act, int64_t OH,
                             int64_t OW, int64_t n, int64_t k, int64_t oh, int64_t ow) {
  const int Cg = C / groups;
  const int Kg = K / groups;
  const int64_t g = k / Kg;
  double acc = 0.0;
  for (int cc = 0; cc < Cg; ++cc) {
    const int64_t c = g * Cg + cc;
    for (int r = 0; r < R; ++r) {
      const int64_t ih = oh * stride - pad + (int64_t)r * dil;
      if (ih < 0 || ih >= H) continue;
      for (int s = 0; s < S; ++s) {
        const int64_t iw = ow * stride - pad + (int64_t)s * dil;
        if (iw < 0 || iw >= W) continue;
        acc += w[((k * Cg + cc) * R + r) * S + s] * x[((n * C + c) * H + ih) * W + iw];
      }
    }
  }
  double v = acc + (b ? b[k] : 0.0);
  if (res) v += res[((n * K + k) * OH + oh) * OW + ow];
  return apply_act(v, act);
}

int oracle_conv2d_f64(int N, int C, int H, int W, int K, int R, int S, int stride, int pad,
                      int dil, int groups, const double* x, const double* w, const double* b,
                      const double* res, int act, double* y) {
  if (groups <= 0 || C % groups || K % groups || stride <= 0 || dil <= 0 || pad < 0) return -1;
  const int64_t OH = out_dim(H, R, stride, pad, dil), OW = out_dim(W, S, stride, pad, dil);
  if (OH <= 0 || OW <= 0) return -1;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      for (int64_t oh = 0; oh < OH; ++oh)
        for (int64_t ow = 0; ow < OW; ++ow)
          y[((n * K + k) * OH + oh) * OW + ow] = conv_point_f64(
              C, H, W, K, R, S, stride, pad, dil, groups, x, w, b, res, act, OH, OW, n, k, oh, ow);
  return 0;
}

/* Selected outputs only: idx holds P quadruples (n, k, oh, ow). */
int oracle_conv2d_f64_points(int N, int C, int H, int W, int K, int R, int S, int stride,
                             int pad, int dil, int groups, const double* x, const double* w,
                             const double* b, const double* res, int act, const int64_t* idx,
                             int64_t P, double* out) {
  if (groups <= 0 || C % groups || K % groups || stride <= 0 || dil <= 0 || pad < 0) return -1;
  const int64_t OH = out_dim(H, R, stride, pad, dil), OW = out_dim(W, S, stride, pad, dil);
  for (int64_t p = 0; p < P; ++p) {
    const int64_t* q = idx + 4 * p;
    if (q[0] < 0 || q[0] >= N || q[1] < 0 || q[1] >= K || q[2] < 0 || q[2] >= OH || q[3] < 0 ||
        q[3] >= OW)
      return -2;
  }
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < P; ++p) {
    const int64_t* q = idx + 4 * p;
    out[p] = conv_point_f64(C, H, W, K, R, S, stride, pad, dil, groups, x, w, b, res, act, OH,
                            OW, q[0], q[1], q[2], q[3]);
  }
  return 0;
}

/* fp32 requantisation of one exact integer: round-to-nearest-even conversion
 * to fp32, one fp32 multiply, round half to even to an integer, clamp, ReLU. */
int oracle_requant_one(int64_t t, float scale, int relu) {
  volatile float tf = (float)t; /* int64 -> fp32, round to nearest even */
  volatile float p = tf * scale; /* single fp32 multiply, no contraction */
  float q = nearbyintf(p);       /* default rounding mode: half to even */
  if (q > 127.0f) q = 127.0f;
  if (q < -128.0f) q = -128.0f;
  int v = (int)q;
  if (relu && v < 0) v = 0;
  return v;
}

/* int8 convolution, exact accumulate.  Returns the number of outputs whose
 * accumulator (before the bias) does not fit in int32 (the library's
 * accumulator type), or -1 on bad parameters.  acc_out (optional) receives
 * acc + bias as int64. */
int64_t oracle_conv2d_i8(int N, int C, int H, int W, int K, int R, int S, int stride, int pad,
                         int dil, int groups, const int8_t* x, const int8_t* w,
                         const int32_t* bias, const float* scale, int relu, int8_t* y,
                         int64_t* acc_out) {
  if (groups <= 0 || C % groups || K % groups || stride <= 0 || dil <= 0 || pad < 0) return -1;
  const int64_t OH = out_dim(H, R, stride, pad, dil), OW = out_dim(W, S, stride, pad, dil);
  if (OH <= 0 || OW <= 0) return -1;
  const int Cg = C / groups, Kg = K / groups;
  int64_t overflow = 0;
#pragma omp parallel for collapse(2) schedule(dynamic) reduction(+ : overflow)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      const int64_t g = k / Kg;
      for (int64_t oh = 0; oh < OH; ++oh)
        for (int64_t ow = 0; ow < OW; ++ow) {
          int64_t acc = 0;
          for (int cc = 0; cc < Cg; ++cc) {
            const int64_t c = g * Cg + cc;
            for (int r = 0; r < R; ++r) {
              const int64_t ih = oh * stride - pad + (int64_t)r * dil;
              if (ih < 0 || ih >= H) continue;
              for (int s = 0; s < S; ++s) {
                const int64_t iw = ow * stride - pad + (int64_t)s * dil;
                if (iw < 0 || iw >= W) continue;
                acc += (int64_t)w[((k * Cg + cc) * R + r) * S + s] *
                       (int64_t)x[((n * C + c) * H + ih) * W + iw];
              }
            }
          }
          if (acc > INT32_MAX || acc < INT32_MIN) overflow += 1;
          const int64_t t = acc + (bias ? bias[k] : 0);
          const int64_t o = ((n * K + k) * OH + oh) * OW + ow;
          if (acc_out) acc_out[o] = t;
          y[o] = (int8_t)oracle_requant_one(t, scale[k], relu);
        }
    }
  return overflow;
}

/* fp32 -> bfloat16, round to nearest, ties to even; NaN stays NaN. */
float oracle_round_bf16(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) {
    u |= 0x00400000u;
  } else {
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
  }
  u &= 0xffff0000u;
  float r;
  memcpy(&r, &u, 4);
  return r;
}

void oracle_round_bf16_array(const float* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(in[i]);
}

/* fp32 -> IEEE binary16 value (as float), round to nearest even, with
 * overflow to infinity and gradual underflow. */
float oracle_round_f16(float v) {
  if (isnan(v) || isinf(v)) return v;
  const float a = fabsf(v);
  if (a >= 65520.0f) return v > 0 ? INFINITY : -INFINITY; /* past max + half ulp */
  int e;
  frexpf(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  /* half has 11 significant bits for normals (exponent >= -14, i.e. e >= -13);
   * subnormals are multiples of 2^-24. */
  int quantum_exp = (e - 11 > -24) ? e - 11 : -24;
  const float q = ldexpf(1.0f, quantum_exp);
  const float r = nearbyintf(a / q) * q; /* a/q exact: power-of-two scaling */
  return v < 0 ? -r : r;
}

void oracle_round_f16_array(const float* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_f16(in[i]);
}

/* Max pooling, NCHW, window R x S, positions outside the image ignored
 * (treated as -inf). */
int oracle_maxpool2d(int N, int C, int H, int W, int R, int S, int stride, int pad,
                     const double* x, double* y) {
  const int64_t OH = out_dim(H, R, stride, pad, 1), OW = out_dim(W, S, stride, pad, 1);
  if (OH <= 0 || OW <= 0) return -1;
#pragma omp parallel for collapse(2)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t c = 0; c < C; ++c)
      for (int64_t oh = 0; oh < OH; ++oh)
        for (int64_t ow = 0; ow < OW; ++ow) {
          double m = -INFINITY;
          for (int r = 0; r < R; ++r)
            for (int s = 0; s < S; ++s) {
              const int64_t ih = oh * stride - pad + r, iw = ow * stride - pad + s;
              if (ih < 0 || ih >= H || iw < 0 || iw >= W) continue;
              const double v = x[((n * C + c) * H + ih) * W + iw];
              if (v > m) m = v;
            }
          y[((n * C + c) * OH + oh) * OW + ow] = m;
        }
  return 0;
}

/* Global average pooling, NCHW -> [N][C]. */
int oracle_global_avgpool(int N, int C, int H, int W, const double* x, double* y) {
#pragma omp parallel for collapse(2)
  for (int64_t n = 0; n < N; ++n)
    for (int64_t c = 0; c < C; ++c) {
      double s = 0.0;
      for (int64_t i = 0; i < (int64_t)H * W; ++i) s += x[(n * C + c) * (int64_t)H * W + i];
      y[n * C + c] = s / ((double)H * W);
    }
  return 0;
}
