// Device helpers shared by the CUDA translation units of libakv.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "akv_internal.h"

namespace akv {

// cos/sin of pos * theta.  The angle is formed and reduced modulo 2*pi in
// double (one product, one fused multiply-add: exact enough for positions up
// to 2^31), then evaluated in float on an argument in [-pi, pi].
__device__ __forceinline__ void rope_cs(double theta, double pos, float *c, float *s) {
  const double two_pi = 6.283185307179586476925286766559;
  const double a = pos * theta;
  const double k = rint(a * (1.0 / two_pi));
  const float r = (float)fma(-k, two_pi, a);
  sincosf(r, s, c);
}

// cos/sin of pos * theta_i without fp64 arithmetic for |pos| <= 2^18.
// The product pos * (hi + lo) is kept as an unevaluated float sum (the
// rounding error of pos * hi recovered exactly with an FMA, Dekker), and it is
// reduced by 2*pi split into three floats, the first two with 8 significant
// bits so that k * C1 and k * C2 are exact for |k| < 2^16 (Cody-Waite).  The
// reduced angle is accurate to ~3e-7 rad.  Larger positions take the double
// path above.
// pos * theta reduced to about [-pi, pi]
__device__ __forceinline__ float rope_angle(float hi, float lo, int pos) {
  const float p = (float)pos;  // exact
  const float ah = p * hi;
  const float ae = fmaf(p, hi, -ah);  // exact error of the product
  const float al = fmaf(p, lo, ae);
  const float k = rintf(ah * 0.159154943091895336f);
  float r = fmaf(-k, 6.28125f, ah);            // 2*pi = 6.28125
  r = fmaf(-k, 1.93023681640625e-3f, r);       //      + 1.93023681640625e-3
  r = fmaf(-k, 5.0703633860393888e-6f, r);     //      + 5.07036338...e-6 (+ ~2e-13)
  return r + al;
}
__device__ __forceinline__ void rope_cs_pair(float hi, float lo, int pos, float *c, float *s) {
  sincosf(rope_angle(hi, lo, pos), s, c);
}
__device__ __forceinline__ void rope_cs(const RopeTheta &th, int f, int pos, float *c, float *s) {
  if (pos < -262144 || pos > 262144) {
    rope_cs(th.th[f], (double)pos, c, s);
    return;
  }
  rope_cs_pair(th.hi[f], th.lo[f], pos, c, s);
}

// cos/sin for a frequency index that differs across the lanes of a warp,
// read from the RopeTheta kernel parameter with warp-uniform indices (an
// unrolled select) instead of one divergent constant-bank load.
__device__ __forceinline__ void rope_cs_lane(const RopeTheta &th, int f, int pos, float *c,
                                             float *s) {
  const bool wide = pos < -262144 || pos > 262144;
  float hi = 0.f, lo = 0.f;
  double t = 0.0;
#pragma unroll
  for (int i = 0; i < kD / 2; ++i)
    if (i == f) {
      hi = th.hi[i];
      lo = th.lo[i];
      if (wide) t = th.th[i];
    }
  if (wide) rope_cs(t, (double)pos, c, s);
  else rope_cs_pair(hi, lo, pos, c, s);
}

// The frequencies in shared memory.  A RopeTheta kernel parameter sits in
// the constant bank, which serves loads whose index differs across the lanes
// of a warp one address at a time; kernels that build cos/sin tables over
// many (row, frequency) pairs copy the float pairs here once per CTA.
struct ThetaSmem {
  float hi[kD / 2], lo[kD / 2];
};
// Threads 0..D/2-1 copy; the caller synchronises before use.
__device__ __forceinline__ void stage_theta(const RopeTheta &th, ThetaSmem &ts) {
  if (threadIdx.x < kD / 2) {
    ts.hi[threadIdx.x] = th.hi[threadIdx.x];
    ts.lo[threadIdx.x] = th.lo[threadIdx.x];
  }
}
__device__ __forceinline__ void rope_cs(const RopeTheta &th, const ThetaSmem &ts, int f, int pos,
                                        float *c, float *s) {
  if (pos < -262144 || pos > 262144) {
    rope_cs(th.th[f], (double)pos, c, s);
    return;
  }
  rope_cs_pair(ts.hi[f], ts.lo[f], pos, c, s);
}

// 16-byte chunks of one head row (D = 64): a bf16 chunk holds 8 elements, an
// f32 chunk 4.  Pair (i, i + D/2) lives in chunks c and c + kHalfChunks.
template <typename T>
struct Chunk;
template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int kElems = 8;
};
template <>
struct Chunk<__half> {
  static constexpr int kElems = 8;
};
template <>
struct Chunk<float> {
  static constexpr int kElems = 4;
};

template <typename T>
__device__ __forceinline__ void chunk_to_f32(const uint4 &u, float *f);
template <>
__device__ __forceinline__ void chunk_to_f32<__nv_bfloat16>(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ void chunk_to_f32<float>(const uint4 &u, float *f) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}

template <typename T>
__device__ __forceinline__ uint4 f32_to_chunk(const float *f);
template <>
__device__ __forceinline__ uint4 f32_to_chunk<__nv_bfloat16>(const float *f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ uint4 f32_to_chunk<__half>(const float *f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ uint4 f32_to_chunk<float>(const float *f) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}

// Rotate chunk pair c / c + half of one head row: y = R(angle) x with
// per-frequency cos/sin cs[i], sn[i] (i = frequency index within the half).
// Tin is read, Tout written (same number of elements per 16-byte chunk).
// Returns true if an output does not fit an fp16 operand (|y| > 65504).
template <typename Tin, typename Tout = Tin>
__device__ __forceinline__ bool rotate_pair(const Tin *src, Tout *dst, int c, const float *cs,
                                            const float *sn) {
  constexpr int E = Chunk<Tin>::kElems;
  static_assert(E == Chunk<Tout>::kElems, "chunk shapes differ");
  constexpr int H = (kD / 2) / E;  // chunks per half row
  const uint4 a = __ldg(reinterpret_cast<const uint4 *>(src) + c);
  const uint4 b = __ldg(reinterpret_cast<const uint4 *>(src) + c + H);
  float x1[E], x2[E], y1[E], y2[E];
  chunk_to_f32<Tin>(a, x1);
  chunk_to_f32<Tin>(b, x2);
  float big = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float co = cs[c * E + e], si = sn[c * E + e];
    y1[e] = x1[e] * co - x2[e] * si;
    y2[e] = x1[e] * si + x2[e] * co;
    big = fmaxf(big, fmaxf(fabsf(y1[e]), fabsf(y2[e])));
  }
  reinterpret_cast<uint4 *>(dst)[c] = f32_to_chunk<Tout>(y1);
  reinterpret_cast<uint4 *>(dst)[c + H] = f32_to_chunk<Tout>(y2);
  return !(big <= 65504.f);
}

// Survivors of a boundary as runs of kept messages, small enough to travel
// in a kernel's parameters (__grid_constant__): t = kstart[nk] |
// kprefix[nk + 1] | kpos[nk] -- first row of each run, its first compacted
// index (exclusive prefix of run lengths, total appended), position of its
// first row before the boundary's repos.
constexpr int kInlineRuns = 256;
struct KeptRunTable {
  int nk;
  int32_t t[3 * kInlineRuns + 1];
  __device__ __forceinline__ int32_t kstart(int run) const { return t[run]; }
  __device__ __forceinline__ int32_t kpos(int run) const { return t[2 * nk + 1 + run]; }
  // run holding compacted index j (0 <= j < total) and j's offset in it
  __device__ __forceinline__ void find(int j, int *run, int *off) const {
    const int32_t *kprefix = t + nk;
    int lo = 0, hi = nk;  // kprefix[lo] <= j < kprefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (kprefix[mid] <= j) lo = mid; else hi = mid;
    }
    *run = lo;
    *off = j - kprefix[lo];
  }
};
// fills rt from the host run tables; false unless 1 <= nk <= kInlineRuns
bool fill_run_table(KeptRunTable *rt, int nk, const int32_t *kstart, const int32_t *kprefix,
                    const int32_t *kpos);

}  // namespace akv
