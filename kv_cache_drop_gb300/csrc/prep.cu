// Restoration pre-pass (paper review page, Appendix A.1.1: "per-segment
// temporary KV versions made by key rotation and value copy").
//
//  * Qr[h][t]     = R(pos(t)) Q[t][h]            fp32 inputs: rows in logical
//                                                  order; bf16 inputs: only
//                                                  the cos/sin of each row's
//                                                  angles, the attention
//                                                  kernel rotates Q itself
//  * Kr[v][g][j]  = R(pos_v(src(j))) K[src(j)][g] one copy per key version,
//                                                  slots in the plan's order
//  * Vp[g][j]     = V[src(j)][g]                  values copied once, shared
//                                                  by every version
// For bf16 inputs all three copies are written as fp16: the rotation's output
// is not a bf16 value anyway, fp16 keeps 3 more mantissa bits for the score
// contraction at the same tensor-core rate, and fp16 V lets the softmax hand
// fp16 probabilities (packed fp16 exp) straight to the P x V product.  A
// value beyond the fp16 range sets status bit kStatusFp16Range.
// Outputs are head-major so that a 128-row tile of one head is 16 KiB of
// contiguous memory (one TMA box).  Each CTA takes 32 rows, computes their
// 32 x 32 cos/sin table once in shared memory, and streams 16-byte chunks.
#include "common.cuh"

#include <type_traits>

namespace akv {
namespace {

constexpr int kRows = 32;
constexpr int kThreads = 256;

template <typename T, typename TR>
__global__ void __launch_bounds__(kThreads) prep_q_kernel(PlanDev p, const T *__restrict__ q,
                                                          RopeTheta th) {
  constexpr int H = (kD / 2) / Chunk<T>::kElems;
  bool ovf = false;
  __shared__ float cs[kRows][kD / 2], sn[kRows][kD / 2];
  __shared__ ThetaSmem ts;
  stage_theta(th, ts);
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * kRows;
  for (int i = threadIdx.x; i < kRows * (kD / 2); i += kThreads) {
    const int r = i / (kD / 2), f = i % (kD / 2);
    if (t0 + r < p.T) rope_cs(th, ts, f, p.tok_qpos[t0 + r], &cs[r][f], &sn[r][f]);
  }
  __syncthreads();
  const int units = kRows * p.Hq * H;
  for (int u = threadIdx.x; u < units; u += kThreads) {
    const int c = u % H, r = (u / H) % kRows, h = u / (H * kRows);
    const int64_t t = t0 + r;
    if (t >= p.T) continue;
    const T *src = q + (t * p.Hq + h) * kD;
    TR *dst = reinterpret_cast<TR *>(p.qr) + ((int64_t)h * p.T + t) * kD;
    ovf |= rotate_pair<T, TR>(src, dst, c, cs[r], sn[r]);
  }
  if (sizeof(TR) == 2 && ovf) atomicOr(p.status, kStatusFp16Range);
}

// bf16: cos/sin(pos(t) theta_f) for every row and frequency (the same
// values prep_q_kernel uses); the attention kernel rotates each query row
// with them as it loads it.
__global__ void __launch_bounds__(kThreads) prep_qcs_kernel(PlanDev p, RopeTheta th) {
  __shared__ ThetaSmem ts;
  stage_theta(th, ts);
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * kRows;
  for (int i = threadIdx.x; i < kRows * (kD / 2); i += kThreads) {
    const int r = i / (kD / 2), f = i % (kD / 2);
    if (t0 + r < p.T) {
      float c, s;
      rope_cs(th, ts, f, p.tok_qpos[t0 + r], &c, &s);
      p.qcs[(t0 + r) * (kD / 2) + f] = make_float2(c, s);
    }
  }
}

template <typename T, typename TR>
__global__ void __launch_bounds__(kThreads) prep_kv_kernel(PlanDev p, const T *__restrict__ k,
                                                           const T *__restrict__ v,
                                                           RopeTheta th) {
  bool ovf = false;
  constexpr int E = Chunk<T>::kElems;
  constexpr int H = (kD / 2) / E;
  __shared__ float cs[kRows][kD / 2], sn[kRows][kD / 2];
  __shared__ int32_t src[kRows];
  const int plane = blockIdx.y;  // < max_ver: key version; == max_ver: values
  const int64_t j0 = (int64_t)blockIdx.x * kRows;
  __shared__ ThetaSmem ts;
  if (threadIdx.x < kRows && j0 + threadIdx.x < p.T) src[threadIdx.x] = p.slot_src[j0 + threadIdx.x];
  if (plane < p.max_ver) {
    stage_theta(th, ts);
    __syncthreads();
    for (int i = threadIdx.x; i < kRows * (kD / 2); i += kThreads) {
      const int r = i / (kD / 2), f = i % (kD / 2);
      if (j0 + r < p.T)
        rope_cs(th, ts, f, p.slot_pos[(int64_t)plane * p.T + j0 + r], &cs[r][f], &sn[r][f]);
    }
  }
  __syncthreads();
  if (plane < p.max_ver) {
    TR *kr = reinterpret_cast<TR *>(p.kr) + (int64_t)plane * p.Hkv * p.T * kD;
    const int units = kRows * p.Hkv * H;
    for (int u = threadIdx.x; u < units; u += kThreads) {
      const int c = u % H, r = (u / H) % kRows, g = u / (H * kRows);
      const int64_t j = j0 + r;
      if (j >= p.T) continue;
      ovf |= rotate_pair<T, TR>(k + ((int64_t)src[r] * p.Hkv + g) * kD,
                                kr + ((int64_t)g * p.T + j) * kD, c, cs[r], sn[r]);
    }
    if (sizeof(TR) == 2 && ovf) atomicOr(p.status, kStatusFp16Range);
  } else {
    constexpr int C = kD / E;  // chunks per row
    const int units = kRows * p.Hkv * C;
    for (int u = threadIdx.x; u < units; u += kThreads) {
      const int c = u % C, r = (u / C) % kRows, g = u / (C * kRows);
      const int64_t j = j0 + r;
      if (j >= p.T) continue;
      const uint4 x = __ldg(reinterpret_cast<const uint4 *>(v + ((int64_t)src[r] * p.Hkv + g) * kD) + c);
      uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<TR *>(p.vp) + ((int64_t)g * p.T + j) * kD) + c;
      if constexpr (sizeof(TR) == sizeof(T)) {
        if constexpr (std::is_same<TR, T>::value) {
          *dst = x;
        } else {  // bf16 -> fp16
          float f[E];
          chunk_to_f32<T>(x, f);
          float big = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) big = fmaxf(big, fabsf(f[e]));
          ovf |= !(big <= 65504.f);
          *dst = f32_to_chunk<TR>(f);
        }
      }
    }
    if (sizeof(TR) == 2 && ovf) atomicOr(p.status, kStatusFp16Range);
  }
}

template <typename T, typename TR>
cudaError_t prep(const PlanDev &p, const void *q, const void *k, const void *v,
                 const RopeTheta &th, cudaStream_t s) {
  const unsigned nb = (unsigned)((p.T + kRows - 1) / kRows);
  if constexpr (std::is_same<T, float>::value)
    prep_q_kernel<T, TR><<<nb, kThreads, 0, s>>>(p, (const T *)q, th);
  else
    prep_qcs_kernel<<<nb, kThreads, 0, s>>>(p, th);
  dim3 g2(nb, p.max_ver + 1);
  prep_kv_kernel<T, TR><<<g2, kThreads, 0, s>>>(p, (const T *)k, (const T *)v, th);
  return cudaGetLastError();
}

}  // namespace

namespace {
// Visibility bits of the windows that need an in-tile mask, once per plan
// (heads share them): CTA = one window, thread = one query row.
__global__ void __launch_bounds__(kTileQ) mask_kernel(PlanDev p) {
  __shared__ int32_t su[kTileK], sd[kTileK];
  const MaskWin mw = p.mwin[blockIdx.x];
  const int r = threadIdx.x;
  // slot tables are padded after T with never-visible entries
  su[r] = p.slot_u[mw.slot0 + r];
  sd[r] = p.slot_dseg[mw.slot0 + r];
  __syncthreads();
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if (r < mw.len) {
    const int t = mw.t0 + r;
    const int seg = p.tok_seg[t];
#pragma unroll 8
    for (int c = 0; c < kTileK; ++c)
      w[c >> 5] |= (uint32_t)(su[c] <= t && seg < sd[c]) << (c & 31);
  }
  p.mask[(int64_t)blockIdx.x * kTileQ + r] = make_uint4(w[0], w[1], w[2], w[3]);
}
}  // namespace

cudaError_t launch_masks(const PlanDev &p, cudaStream_t s) {
  if (p.n_mask == 0) return cudaSuccess;
  static_assert(kTileQ == kTileK, "one thread per row and per key");
  mask_kernel<<<(unsigned)p.n_mask, kTileQ, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prep(const PlanDev &p, const void *q, const void *k, const void *v,
                        const RopeTheta &th, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  return p.dtype == AKV_F32 ? prep<float, float>(p, q, k, v, th, s)
                            : prep<__nv_bfloat16, __half>(p, q, k, v, th, s);
}

}  // namespace akv
