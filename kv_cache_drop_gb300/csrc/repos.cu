// Repos rotate + compact and append (paper review page section 3.3: a cached
// key moves from position p to q by the rotation R(q - p), its value is left
// as it is; section 4.2 / Appendix A.1.2: a key cached at another position
// version is converted by key rotation).
//
// One streaming pass: every surviving row is read once (K and V, 16-byte
// vector loads) and written once to its compacted place.  A CTA takes 32
// rows; their 32 x 32 cos/sin table is built once in shared memory and shared
// by all KV heads.
#include "common.cuh"

namespace akv {
namespace {

constexpr int kRows = 32;
constexpr int kThreads = 256;

template <typename T, bool kScatter>
__global__ void __launch_bounds__(kThreads)
    move_rows_kernel(int Hkv, int n, const int32_t *__restrict__ src, const int32_t *__restrict__ pf,
                     const int32_t *__restrict__ pt, const T *__restrict__ kin,
                     const T *__restrict__ vin, T *__restrict__ kout, T *__restrict__ vout,
                     RopeTheta th) {
  constexpr int E = Chunk<T>::kElems;
  constexpr int H = (kD / 2) / E;  // chunk pairs per head row
  constexpr int C = kD / E;        // chunks per head row
  __shared__ float cs[kRows][kD / 2], sn[kRows][kD / 2];
  __shared__ int64_t in_row[kRows], out_row[kRows];
  const int j0 = blockIdx.x * kRows;
  if (threadIdx.x < kRows) {
    const int j = j0 + threadIdx.x;
    if (j < n) {
      // kScatter (append): row j of the inputs goes to pool slot src[j],
      // rotated to absolute position pf[j].  Otherwise (repos): pool row
      // src[j] goes to compact row j, rotated by pos_to - pos_from.
      in_row[threadIdx.x] = kScatter ? j : src[j];
      out_row[threadIdx.x] = kScatter ? src[j] : j;
    }
  }
  for (int i = threadIdx.x; i < kRows * (kD / 2); i += kThreads) {
    const int r = i / (kD / 2), f = i % (kD / 2);
    const int j = j0 + r;
    if (j < n) {
      const int delta = kScatter ? pf[j] : (pt ? pt[j] : j) - pf[j];
      rope_cs(th, f, delta, &cs[r][f], &sn[r][f]);
    }
  }
  __syncthreads();
  const int rows = min(kRows, n - j0);
  const int k_units = rows * Hkv * H;
  for (int u = threadIdx.x; u < k_units; u += kThreads) {
    const int c = u % H, r = (u / H) % rows, g = u / (H * rows);
    rotate_pair<T>(kin + (in_row[r] * Hkv + g) * kD, kout + (out_row[r] * Hkv + g) * kD, c, cs[r],
                   sn[r]);
  }
  const int v_units = rows * Hkv * C;
  for (int u = threadIdx.x; u < v_units; u += kThreads) {
    const int c = u % C, row = u / C;  // row = r * Hkv + g, consecutive in memory
    const int r = row / Hkv, g = row % Hkv;
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(vin + (in_row[r] * Hkv + g) * kD) + c);
    reinterpret_cast<uint4 *>(vout + (out_row[r] * Hkv + g) * kD)[c] = x;
  }
}

template <typename T, bool kScatter>
cudaError_t move_rows(int Hkv, int n, const int32_t *src, const int32_t *pf, const int32_t *pt,
                      const void *kin, const void *vin, void *kout, void *vout,
                      const RopeTheta &th, cudaStream_t s) {
  const unsigned nb = (unsigned)((n + kRows - 1) / kRows);
  move_rows_kernel<T, kScatter><<<nb, kThreads, 0, s>>>(Hkv, n, src, pf, pt, (const T *)kin,
                                                       (const T *)vin, (T *)kout, (T *)vout, th);
  return cudaGetLastError();
}

// Repos at a boundary in one pass: the survivors' source rows and current
// positions follow from per-kept-message tables (first row, first compacted
// index, position of the first row), found by binary search; no index list.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    repos_boundary_kernel(int Hkv, int r, int nk, const int32_t *__restrict__ kstart,
                          const int32_t *__restrict__ kprefix, const int32_t *__restrict__ kpos,
                          const T *__restrict__ kin, const T *__restrict__ vin,
                          T *__restrict__ kout, T *__restrict__ vout, RopeTheta th) {
  constexpr int E = Chunk<T>::kElems;
  constexpr int H = (kD / 2) / E;
  constexpr int C = kD / E;
  __shared__ float cs[kRows][kD / 2], sn[kRows][kD / 2];
  __shared__ int64_t in_row[kRows];
  __shared__ int32_t delta[kRows];
  const int j0 = blockIdx.x * kRows;
  const int rows = min(kRows, r - j0);
  if (threadIdx.x < rows) {
    const int j = j0 + threadIdx.x;
    int lo = 0, hi = nk;  // kprefix[lo] <= j < kprefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(kprefix + mid) <= j) lo = mid; else hi = mid;
    }
    const int off = j - __ldg(kprefix + lo);
    in_row[threadIdx.x] = __ldg(kstart + lo) + off;
    delta[threadIdx.x] = j - (__ldg(kpos + lo) + off);  // new position j - current position
  }
  __syncthreads();
  for (int i = threadIdx.x; i < rows * (kD / 2); i += kThreads) {
    const int rr = i / (kD / 2), f = i % (kD / 2);
    rope_cs(th, f, delta[rr], &cs[rr][f], &sn[rr][f]);
  }
  __syncthreads();
  const int k_units = rows * Hkv * H;
  for (int u = threadIdx.x; u < k_units; u += kThreads) {
    const int c = u % H, rr = (u / H) % rows, g = u / (H * rows);
    rotate_pair<T>(kin + (in_row[rr] * Hkv + g) * kD, kout + ((int64_t)(j0 + rr) * Hkv + g) * kD,
                   c, cs[rr], sn[rr]);
  }
  const int v_units = rows * Hkv * C;
  for (int u = threadIdx.x; u < v_units; u += kThreads) {
    const int c = u % C, row = u / C;
    const int rr = row / Hkv, g = row % Hkv;
    const uint4 x = __ldg(reinterpret_cast<const uint4 *>(vin + (in_row[rr] * Hkv + g) * kD) + c);
    reinterpret_cast<uint4 *>(vout + ((int64_t)(j0 + rr) * Hkv + g) * kD)[c] = x;
  }
}

}  // namespace

cudaError_t launch_repos(int dtype, int Hkv, int r, const int32_t *src, const int32_t *pf,
                         const int32_t *pt, const void *kin, const void *vin, void *kout,
                         void *vout, const RopeTheta &th, cudaStream_t s) {
  return dtype == AKV_F32
             ? move_rows<float, false>(Hkv, r, src, pf, pt, kin, vin, kout, vout, th, s)
             : move_rows<__nv_bfloat16, false>(Hkv, r, src, pf, pt, kin, vin, kout, vout, th, s);
}

cudaError_t launch_append(int dtype, int Hkv, int n, const void *kn, const void *vn,
                          const int32_t *pos, const int32_t *slot, void *kp, void *vp,
                          const RopeTheta &th, cudaStream_t s) {
  return dtype == AKV_F32
             ? move_rows<float, true>(Hkv, n, slot, pos, nullptr, kn, vn, kp, vp, th, s)
             : move_rows<__nv_bfloat16, true>(Hkv, n, slot, pos, nullptr, kn, vn, kp, vp, th, s);
}

}  // namespace akv

namespace akv {
cudaError_t launch_repos_boundary(int dtype, int Hkv, int r, int nk, const int32_t *kstart,
                                  const int32_t *kprefix, const int32_t *kpos, const void *kin,
                                  const void *vin, void *kout, void *vout, const RopeTheta &th,
                                  cudaStream_t s) {
  if (r == 0) return cudaSuccess;
  const unsigned nb = (unsigned)((r + kRows - 1) / kRows);
  if (dtype == AKV_F32)
    repos_boundary_kernel<float><<<nb, kThreads, 0, s>>>(Hkv, r, nk, kstart, kprefix, kpos,
                                                         (const float *)kin, (const float *)vin,
                                                         (float *)kout, (float *)vout, th);
  else
    repos_boundary_kernel<__nv_bfloat16><<<nb, kThreads, 0, s>>>(
        Hkv, r, nk, kstart, kprefix, kpos, (const __nv_bfloat16 *)kin, (const __nv_bfloat16 *)vin,
        (__nv_bfloat16 *)kout, (__nv_bfloat16 *)vout, th);
  return cudaGetLastError();
}
}  // namespace akv
