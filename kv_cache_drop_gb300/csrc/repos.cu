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
  __shared__ ThetaSmem ts;
  stage_theta(th, ts);
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
  __syncthreads();
  for (int i = threadIdx.x; i < kRows * (kD / 2); i += kThreads) {
    const int r = i / (kD / 2), f = i % (kD / 2);
    const int j = j0 + r;
    if (j < n) {
      const int delta = kScatter ? pf[j] : (pt ? pt[j] : j) - pf[j];
      rope_cs(th, ts, f, delta, &cs[r][f], &sn[r][f]);
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

// Repos as a stream (bf16 and fp32): CTA = kSRows output rows.  The row
// sources are resolved first (one thread per row), then every thread issues
// all of its loads -- one K chunk pair and two V chunks per round -- before
// the rows' cos/sin table is built, so the angle arithmetic overlaps the
// loads in flight.  Output rows j0.. are written densely.
constexpr int kSRows = 8;

// rows of akv_repos_rotate: explicit source row and position delta
struct ExplicitRows {
  const int32_t *src, *pf, *pt;
  __device__ __forceinline__ void get(int j, int64_t *in, int32_t *delta) const {
    *in = __ldg(src + j);
    *delta = (pt ? __ldg(pt + j) : j) - __ldg(pf + j);
  }
};
// rows of akv_repos_boundary: runs of kept messages (first row, first
// compacted index, current position of the first row), by binary search
struct KeptRuns {
  int nk;
  const int32_t *kstart, *kprefix, *kpos;
  __device__ __forceinline__ void get(int j, int64_t *in, int32_t *delta) const {
    int lo = 0, hi = nk;  // kprefix[lo] <= j < kprefix[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(kprefix + mid) <= j) lo = mid; else hi = mid;
    }
    const int off = j - __ldg(kprefix + lo);
    *in = __ldg(kstart + lo) + off;
    *delta = j - (__ldg(kpos + lo) + off);  // new position j - current position
  }
};

// rows of akv_repos_boundary with the run tables carried in the kernel's
// parameters (no upload)
struct KeptRunsInline {
  KeptRunTable tab;
  __device__ __forceinline__ void get(int j, int64_t *in, int32_t *delta) const {
    int run, off;
    tab.find(j, &run, &off);
    *in = tab.kstart(run) + off;
    *delta = j - (tab.kpos(run) + off);
  }
};

template <typename T, typename Rows>
__global__ void __launch_bounds__(kThreads)
    repos_stream_kernel(int Hkv, int n, const __grid_constant__ Rows rs, const T *__restrict__ kin,
                        const T *__restrict__ vin, T *__restrict__ kout, T *__restrict__ vout,
                        RopeTheta th) {
  constexpr int E = Chunk<T>::kElems;
  constexpr int H = (kD / 2) / E;  // chunk pairs per head row
  constexpr int C = kD / E;        // chunks per head row (= 2H)
  __shared__ float cs[kSRows][kD / 2], sn[kSRows][kD / 2];
  __shared__ int64_t in_row[kSRows];
  __shared__ int32_t dl[kSRows];
  __shared__ ThetaSmem ts;
  const int j0 = blockIdx.x * kSRows;
  const int rows = min(kSRows, n - j0);
  if (threadIdx.x < rows) rs.get(j0 + threadIdx.x, &in_row[threadIdx.x], &dl[threadIdx.x]);
  stage_theta(th, ts);
  __syncthreads();
  const int k_units = rows * Hkv * H;  // V units = 2 * k_units
  for (int base = 0; base < k_units; base += kThreads) {
    const int u = base + (int)threadIdx.x;
    const bool on = u < k_units;
    int rk = 0, ck = 0, rv0 = 0, cv0 = 0, rv1 = 0, cv1 = 0;
    int64_t ok = 0, ov0 = 0, ov1 = 0;  // head-row offsets (elements) within a row block
    uint4 a{}, b{}, v0{}, v1{};
    if (on) {
      // consecutive threads walk consecutive chunks of one row: coalesced
      ck = u % H;
      const int hk = u / H;  // = row * Hkv + head
      rk = hk / Hkv;
      ok = (int64_t)(hk % Hkv) * kD;
      const T *ks = kin + in_row[rk] * Hkv * kD + ok;
      a = __ldg(reinterpret_cast<const uint4 *>(ks) + ck);
      b = __ldg(reinterpret_cast<const uint4 *>(ks) + ck + H);
      const int w0 = 2 * u, w1 = 2 * u + 1;
      cv0 = w0 % C;
      rv0 = (w0 / C) / Hkv;
      ov0 = (int64_t)((w0 / C) % Hkv) * kD;
      cv1 = w1 % C;
      rv1 = (w1 / C) / Hkv;
      ov1 = (int64_t)((w1 / C) % Hkv) * kD;
      v0 = __ldg(reinterpret_cast<const uint4 *>(vin + in_row[rv0] * Hkv * kD + ov0) + cv0);
      v1 = __ldg(reinterpret_cast<const uint4 *>(vin + in_row[rv1] * Hkv * kD + ov1) + cv1);
    }
    if (base == 0) {  // the rows' angle table, while the loads are in flight
      for (int i = threadIdx.x; i < rows * (kD / 2); i += kThreads) {
        const int r = i / (kD / 2), f = i % (kD / 2);
        rope_cs(th, ts, f, dl[r], &cs[r][f], &sn[r][f]);
      }
      __syncthreads();
    }
    if (on) {
      float x1[E], x2[E], y1[E], y2[E];
      chunk_to_f32<T>(a, x1);
      chunk_to_f32<T>(b, x2);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float co = cs[rk][ck * E + e], si = sn[rk][ck * E + e];
        y1[e] = x1[e] * co - x2[e] * si;
        y2[e] = x1[e] * si + x2[e] * co;
      }
      uint4 *kd = reinterpret_cast<uint4 *>(kout + (int64_t)(j0 + rk) * Hkv * kD + ok);
      kd[ck] = f32_to_chunk<T>(y1);
      kd[ck + H] = f32_to_chunk<T>(y2);
      reinterpret_cast<uint4 *>(vout + (int64_t)(j0 + rv0) * Hkv * kD + ov0)[cv0] = v0;
      reinterpret_cast<uint4 *>(vout + (int64_t)(j0 + rv1) * Hkv * kD + ov1)[cv1] = v1;
    }
  }
}

template <typename T, typename Rows>
cudaError_t repos_stream(int Hkv, int n, const Rows &rs, const void *kin, const void *vin,
                         void *kout, void *vout, const RopeTheta &th, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const unsigned nb = (unsigned)((n + kSRows - 1) / kSRows);
  repos_stream_kernel<T, Rows><<<nb, kThreads, 0, s>>>(Hkv, n, rs, (const T *)kin,
                                                       (const T *)vin, (T *)kout, (T *)vout, th);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_repos(int dtype, int Hkv, int r, const int32_t *src, const int32_t *pf,
                         const int32_t *pt, const void *kin, const void *vin, void *kout,
                         void *vout, const RopeTheta &th, cudaStream_t s) {
  const ExplicitRows rs{src, pf, pt};
  return dtype == AKV_F32
             ? repos_stream<float>(Hkv, r, rs, kin, vin, kout, vout, th, s)
             : repos_stream<__nv_bfloat16>(Hkv, r, rs, kin, vin, kout, vout, th, s);
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
  const KeptRuns rs{nk, kstart, kprefix, kpos};
  if (dtype == AKV_F32) return repos_stream<float>(Hkv, r, rs, kin, vin, kout, vout, th, s);
  return repos_stream<__nv_bfloat16>(Hkv, r, rs, kin, vin, kout, vout, th, s);
}

int repos_inline_runs() { return kInlineRuns; }
bool fill_run_table(KeptRunTable *rt, int nk, const int32_t *kstart, const int32_t *kprefix,
                    const int32_t *kpos) {
  if (nk < 1 || nk > kInlineRuns) return false;
  rt->nk = nk;
  for (int i = 0; i < nk; ++i) {
    rt->t[i] = kstart[i];
    rt->t[2 * nk + 1 + i] = kpos[i];
  }
  for (int i = 0; i <= nk; ++i) rt->t[nk + i] = kprefix[i];
  return true;
}

cudaError_t launch_repos_boundary_inline(int dtype, int Hkv, int r, int nk, const int32_t *kstart,
                                         const int32_t *kprefix, const int32_t *kpos,
                                         const void *kin, const void *vin, void *kout, void *vout,
                                         const RopeTheta &th, cudaStream_t s) {
  KeptRunsInline rs;
  if (!fill_run_table(&rs.tab, nk, kstart, kprefix, kpos)) return cudaErrorInvalidValue;
  if (dtype == AKV_F32) return repos_stream<float>(Hkv, r, rs, kin, vin, kout, vout, th, s);
  return repos_stream<__nv_bfloat16>(Hkv, r, rs, kin, vin, kout, vout, th, s);
}
}  // namespace akv
