// Element-wise pieces of the decoder layers around the segment attention:
// RMSNorm (one warp per row, fp32 math) and SwiGLU (silu(g) * u).
#include "common.cuh"

namespace akv {
namespace {

constexpr int kNormWarps = 8;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kNormWarps * 32)
    rmsnorm_kernel(int rows, int d, float eps, const Tin *__restrict__ x,
                   const float *__restrict__ w, Tout *__restrict__ y) {
  const int row = blockIdx.x * kNormWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= rows) return;
  const Tin *xr = x + (int64_t)row * d;
  float ss = 0.f;
  for (int i = lane; i < d; i += 32) {
    const float v = (float)xr[i];
    ss = fmaf(v, v, ss);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / (float)d + eps);
  Tout *yr = y + (int64_t)row * d;
  for (int i = lane; i < d; i += 32) {
    const float v = (float)xr[i] * inv * (w ? w[i] : 1.f);
    if constexpr (sizeof(Tout) == 2) yr[i] = __float2bfloat16_rn(v);
    else yr[i] = v;
  }
}

__device__ __forceinline__ float silu_mul(float a, float b) { return a / (1.f + __expf(-a)) * b; }

// out may alias g (element-wise, read before write).  kVec: 8 elements per
// 16-byte load (g, u, out 16-byte aligned); the elements past the last full
// group of 8 are done one by one either way.
template <bool kVec>
__global__ void swiglu_kernel(int64_t n, const __nv_bfloat16 *g, const __nv_bfloat16 *u,
                              __nv_bfloat16 *out) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t done = 0;
  if (kVec) {
    const int64_t n8 = n / 8;
    for (int64_t i = tid; i < n8; i += stride) {
      const uint4 a = reinterpret_cast<const uint4 *>(g)[i];
      const uint4 b = reinterpret_cast<const uint4 *>(u)[i];
      const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a);
      const __nv_bfloat162 *b2 = reinterpret_cast<const __nv_bfloat162 *>(&b);
      uint4 r;
      __nv_bfloat162 *r2 = reinterpret_cast<__nv_bfloat162 *>(&r);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(a2[e]), y = __bfloat1622float2(b2[e]);
        r2[e] = __floats2bfloat162_rn(silu_mul(x.x, y.x), silu_mul(x.y, y.y));
      }
      reinterpret_cast<uint4 *>(out)[i] = r;
    }
    done = n8 * 8;
  }
  for (int64_t i = done + tid; i < n; i += stride)
    out[i] = __float2bfloat16_rn(silu_mul(__bfloat162float(g[i]), __bfloat162float(u[i])));
}

__global__ void widen_kernel(int64_t n, const __nv_bfloat16 *__restrict__ x, float *__restrict__ y) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    y[i] = __bfloat162float(x[i]);
}

unsigned grid_for(int64_t n) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (n + 255) / 256;
  return (unsigned)(want < (int64_t)sms * 16 ? want : (int64_t)sms * 16);
}

}  // namespace

cudaError_t launch_widen(int64_t n, const void *x, float *y, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  widen_kernel<<<grid_for(n), 256, 0, s>>>(n, (const __nv_bfloat16 *)x, y);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(int rows, int d, float eps, int in_f32, const void *x, const float *w,
                           int out_f32, void *y, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const unsigned nb = (unsigned)((rows + kNormWarps - 1) / kNormWarps);
  if (in_f32 && out_f32)
    rmsnorm_kernel<float, float><<<nb, kNormWarps * 32, 0, s>>>(rows, d, eps, (const float *)x, w, (float *)y);
  else if (in_f32)
    rmsnorm_kernel<float, __nv_bfloat16><<<nb, kNormWarps * 32, 0, s>>>(rows, d, eps, (const float *)x, w,
                                                                       (__nv_bfloat16 *)y);
  else if (out_f32)
    rmsnorm_kernel<__nv_bfloat16, float><<<nb, kNormWarps * 32, 0, s>>>(
        rows, d, eps, (const __nv_bfloat16 *)x, w, (float *)y);
  else
    rmsnorm_kernel<__nv_bfloat16, __nv_bfloat16><<<nb, kNormWarps * 32, 0, s>>>(
        rows, d, eps, (const __nv_bfloat16 *)x, w, (__nv_bfloat16 *)y);
  return cudaGetLastError();
}

cudaError_t launch_swiglu(int64_t n, const void *g, const void *u, void *out, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const bool vec = ((uintptr_t)g | (uintptr_t)u | (uintptr_t)out) % 16 == 0;
  if (vec)
    swiglu_kernel<true><<<grid_for((n + 7) / 8), 256, 0, s>>>(
        n, (const __nv_bfloat16 *)g, (const __nv_bfloat16 *)u, (__nv_bfloat16 *)out);
  else
    swiglu_kernel<false><<<grid_for(n), 256, 0, s>>>(n, (const __nv_bfloat16 *)g,
                                                     (const __nv_bfloat16 *)u, (__nv_bfloat16 *)out);
  return cudaGetLastError();
}

}  // namespace akv
