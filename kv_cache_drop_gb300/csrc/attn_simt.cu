// fp32 segment attention (SIMT FMA) and the visibility counter.
//
// Both walk exactly what the tensor-core kernel walks: the query tile's
// 128-key windows over the permuted key slots, with the in-tile predicate
//     visible(t, j) <=> slot_u[j] <= t  and  seg(t) < slot_dseg[j]
// (row t sees key u iff u <= t and u was not dropped before t's segment;
// paper review page section 4.2 / Appendix A.1.1).  The fp32 path exists for
// fp32 inputs, where a 10-bit-mantissa tensor format would not hold the
// accuracy; it is small and latency-bound.
#include "common.cuh"

namespace akv {
namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ bool visible(const PlanDev &p, int64_t t, int seg, int64_t j) {
  return (int64_t)__ldg(p.slot_u + j) <= t && seg < __ldg(p.slot_dseg + j);
}

// One warp per (row, head); lanes take keys, each lane keeps its own online
// softmax state, and the warp merges them at the end.
__global__ void __launch_bounds__(kWarps * 32) attn_simt_f32_kernel(PlanDev p, float *out) {
  const QTile qt = p.qtiles[blockIdx.x];
  const int h = blockIdx.y, g = h / (p.Hq / p.Hkv);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float *kr = reinterpret_cast<const float *>(p.kr) + ((int64_t)qt.ver * p.Hkv + g) * p.T * kD;
  const float *vp = reinterpret_cast<const float *>(p.vp) + (int64_t)g * p.T * kD;
  const float scale = 0.125f;  // 1/sqrt(64)
  for (int r = warp; r < qt.len; r += kWarps) {
    const int64_t t = qt.t0 + r;
    const int seg = p.tok_seg[t];
    const float *qrow = reinterpret_cast<const float *>(p.qr) + ((int64_t)h * p.T + t) * kD;
    float qv[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) qv[d] = __ldg(qrow + d);
    float m = -INFINITY, l = 0.f, acc[kD];
#pragma unroll
    for (int d = 0; d < kD; ++d) acc[d] = 0.f;
    for (int w = 0; w < qt.win_cnt; ++w) {
      const int64_t base = p.windows[qt.win_off + w] & ~kWinFull;
      for (int k0 = 0; k0 < kTileK; k0 += 32) {
        const int64_t j = base + k0 + lane;
        if (j >= p.T || !visible(p, t, seg, j)) continue;
        const float *krow = kr + j * kD;
        float s = 0.f;
#pragma unroll
        for (int d = 0; d < kD; ++d) s = fmaf(qv[d], __ldg(krow + d), s);
        s *= scale;
        const float mn = fmaxf(m, s);
        const float a = __expf(m - mn), e = __expf(s - mn);
        l = l * a + e;
        const float *vrow = vp + j * kD;
#pragma unroll
        for (int d = 0; d < kD; ++d) acc[d] = fmaf(acc[d], a, e * __ldg(vrow + d));
        m = mn;
      }
    }
    // merge the 32 lane states
    float M = m;
#pragma unroll
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f = (m == -INFINITY) ? 0.f : __expf(m - M);
    float L = l * f;
#pragma unroll
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float *orow = out + (t * p.Hq + h) * kD;
#pragma unroll
    for (int d = 0; d < kD; ++d) {
      float x = acc[d] * f;
#pragma unroll
      for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (lane == (d & 31)) orow[d] = x / L;
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32) visible_counts_kernel(PlanDev p, int32_t *counts) {
  const QTile qt = p.qtiles[blockIdx.x];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = warp; r < qt.len; r += kWarps) {
    const int64_t t = qt.t0 + r;
    const int seg = p.tok_seg[t];
    int n = 0;
    for (int w = 0; w < qt.win_cnt; ++w) {
      const uint32_t win = p.windows[qt.win_off + w];
      const int64_t base = win & ~kWinFull;
      for (int k0 = 0; k0 < kTileK; k0 += 32) {
        const int64_t j = base + k0 + lane;
        // a full window needs no predicate: every slot in it is visible
        if ((win & kWinFull) || (j < p.T && visible(p, t, seg, j))) ++n;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    if (lane == 0) counts[t] = n;
  }
}

}  // namespace

cudaError_t launch_attn_simt_f32(const PlanDev &p, void *out, cudaStream_t s) {
  if (p.n_qtiles == 0) return cudaSuccess;
  dim3 grid(p.n_qtiles, p.Hq);
  attn_simt_f32_kernel<<<grid, kWarps * 32, 0, s>>>(p, (float *)out);
  return cudaGetLastError();
}

cudaError_t launch_visible_counts(const PlanDev &p, int32_t *counts, cudaStream_t s) {
  if (p.n_qtiles == 0) return cudaSuccess;
  visible_counts_kernel<<<p.n_qtiles, kWarps * 32, 0, s>>>(p, counts);
  return cudaGetLastError();
}

}  // namespace akv
