// Projection / FFN GEMM of the restoration prefill's decoder layers (paper
// review page section 4.2, Appendix A.1.1: attention is segmented, the FFN
// runs once over the whole sequence):  Y[M,N] (+)= X[M,K] * W[N,K]^T.
//
// tcgen05 GEMM over 128 x 256 output tiles, persistent (one CTA per SM):
// warp 0 streams 64-wide K blocks of X and W with TMA (128-byte swizzle)
// through a 4-stage ring, warp 1 allocates two 256-column TMEM accumulators
// and issues 128x256x16 MMAs from one thread, warps 2-5 (one TMEM lane
// quarter each) read an accumulator back and write bf16, fp32, add into an
// fp32 output (the residual stream) or apply SwiGLU, while the next tile
// accumulates into the other one.  Waits are bounded like the attention
// kernel's.
//
// CTAs run in clusters of two that work on vertically adjacent tiles (the
// same 256 W rows, M tiles 2i and 2i + 1): each CTA loads its own X block
// and one half of the W block, which TMA multicasts into both CTAs' shared
// memory, so a K block costs each SM 32 KB of L2 reads instead of 48.  At
// one CTA per SM the K-block ring bounds the bytes in flight, and without
// the multicast the L2-to-SM stream (about 27 TB/s of L2 reads at full
// tensor rate) held the tensor pipe near 65% busy.  A stage of a CTA is
// refilled only after both CTAs' MMAs have read it: each MMA commit
// arrives on the stage's "empty" barrier in both CTAs.
#include "common.cuh"
#include "tc_ptx.cuh"

#include <cuda.h>

namespace akv {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, kStages = 4;
constexpr int kThreads = 192;
constexpr int kCluster = 2;  // CTAs per cluster (two M tiles sharing each W block)
constexpr uint32_t kABytes = BM * BK * 2, kBBytes = BN * BK * 2;
constexpr uint32_t kBPartBytes = kBBytes / kCluster;  // the W rows one CTA loads
constexpr long long kWaitBudget = 1000000000LL;

struct __align__(1024) GemmSmem {
  uint8_t a[kStages][kABytes];
  uint8_t b[kStages][kBBytes];
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];  // accumulator b: MMAs done / drained by the epilogue
  uint32_t tmem_base;
};

__device__ __forceinline__ void wait_bar(uint64_t *bar, uint32_t parity, uint32_t *status) {
  ptx::mbar_wait_grid(bar, parity, status, kStatusWaitTimeout, kWaitBudget);
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// every thread of both CTAs: release this CTA's earlier writes (barrier
// initialisation) to the peer, and wait until the peer has arrived too
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// TMA 2D load whose box is written at the same shared-memory offset in
// every CTA of `mask`, each signalling its own mbarrier at `bar`'s offset
__device__ __forceinline__ void tma_load_2d_mc(void *dst, const CUtensorMap *m, uint64_t *bar,
                                               int x, int y, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".multicast::cluster [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(ptx::smem_addr(dst)),
      "l"((uint64_t)m), "r"(ptx::smem_addr(bar)), "r"(x), "r"(y), "h"(mask)
      : "memory");
}
// once the MMAs issued before it have completed, arrive on the mbarrier at
// `bar`'s offset in every CTA of `mask`
__device__ __forceinline__ void mma_commit_mc(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(ptx::smem_addr(bar)),
      "h"(mask)
      : "memory");
}

// Epilogue of one 128 x 256 tile: this thread's row of the accumulator at
// TMEM address tl (its lane, column 0) into Y.
// out_mode: 0 bf16 store, 1 fp32 store, 2 fp32 add into Y, 3 SwiGLU: W holds
// gate and up rows interleaved in blocks of 128 (launch_interleave_gu), so a
// tile's accumulator columns 0-127 are gate and 128-255 the matching up
// columns; Y [M][N/2] bf16 gets silu(gate) * up
__device__ __forceinline__ void store_tile(uint32_t tl, int m, int n0, int M, int N, void *Y,
                                           int out_mode) {
  if (out_mode == 3) {
    const int NO = N / 2;  // output columns
#pragma unroll 1
    for (int c0 = 0; c0 < BN / 2; c0 += 32) {
      uint32_t gr[32], ur[32];
      ptx::tmem_ld32(tl + c0, gr);
      ptx::tmem_ld32(tl + BN / 2 + c0, ur);
      ptx::tmem_wait_ld();
      ptx::reg_fence32(gr);
      ptx::reg_fence32(ur);
      const int n = n0 / 2 + c0;
      if (m >= M || n >= NO) continue;
      uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(Y) + (int64_t)m * NO + n);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 8 * q + 2 * e;
          const float g0 = __uint_as_float(gr[c]), g1 = __uint_as_float(gr[c + 1]);
          const float y0 = __fdividef(g0, 1.f + __expf(-g0)) * __uint_as_float(ur[c]);
          const float y1 = __fdividef(g1, 1.f + __expf(-g1)) * __uint_as_float(ur[c + 1]);
          __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
          w[e] = *reinterpret_cast<uint32_t *>(&h);
        }
        dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    return;
  }
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t r[32];
    ptx::tmem_ld32(tl + c0, r);
    ptx::tmem_wait_ld();
    ptx::reg_fence32(r);
    const int n = n0 + c0;
    if (m >= M || n >= N) continue;  // N is a multiple of 32
    if (out_mode == 0) {
      uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(Y) + (int64_t)m * N + n);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(r[8 * q + 2 * e]),
                                                   __uint_as_float(r[8 * q + 2 * e + 1]));
          w[e] = *reinterpret_cast<uint32_t *>(&h);
        }
        dst[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
      float4 *dst = reinterpret_cast<float4 *>(reinterpret_cast<float *>(Y) + (int64_t)m * N + n);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 v = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                               __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
        if (out_mode == 2) {
          const float4 o = dst[q];
          v.x += o.x;
          v.y += o.y;
          v.z += o.z;
          v.w += o.w;
        }
        dst[q] = v;
      }
    }
  }
}

// Persistent: cluster q takes tile pairs q, q + clusters, ... (row-major over
// the grid of (M tile pair, N tile), so consecutive pairs share their X
// rows); rank r of the cluster computes M tile 2i + r of pair (i, n).  A
// pair whose second M tile lies past M still runs in full (its X rows are
// read as zeros, its rows are not stored), so both CTAs issue the same
// loads.  The K-block ring runs on across tiles; TMEM holds two 256-column
// accumulators, so the epilogue warps drain tile j while the MMA thread
// computes tile j + 1.
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                int M, int N, int K, void *__restrict__ Y, int out_mode, uint32_t *status) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem &sm = *reinterpret_cast<GemmSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_rank();
  const int q0 = blockIdx.x / kCluster, nq = gridDim.x / kCluster;
  const int nk = (K + BK - 1) / BK;
  const int tiles_n = (N + BN - 1) / BN;
  const int n_tiles = tiles_n * ((M + kCluster * BM - 1) / (kCluster * BM));  // tile groups
  // tile pair t: rows of this CTA's M tile, first column of its N tile
  auto m0_of = [&](int t) { return ((t / tiles_n) * kCluster + rank) * BM; };
  auto n0_of = [&](int t) { return (t % tiles_n) * BN; };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&sm.full[s], 1);
      ptx::mbar_init(&sm.empty[s], kCluster);  // both CTAs' MMAs have read the stage
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&sm.acc_full[b], 1);
      ptx::mbar_init(&sm.acc_empty[b], 4);  // one arrival per epilogue warp
    }
    ptx::fence_barrier_init();
  }
  if (warp == 1) ptx::tmem_alloc(&sm.tmem_base, 2 * BN);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  cluster_sync();  // the peer's barriers exist before any multicast or remote arrive

  if (warp == 0) {
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tmA);
      ptx::tma_prefetch_desc(&tmB);
      int c = 0;  // K blocks loaded so far, over all tiles
      for (int t = q0; t < n_tiles; t += nq) {
        const int m0 = m0_of(t), n0 = n0_of(t);
        for (int kb = 0; kb < nk; ++kb, ++c) {
          const int s = c % kStages;
          if (c >= kStages) wait_bar(&sm.empty[s], ((c / kStages) - 1) & 1, status);
          // this CTA's X block, and its half of the W block into both CTAs
          ptx::mbar_expect_tx(&sm.full[s], kABytes + kBBytes);
          ptx::tma_load_2d(sm.a[s], &tmA, &sm.full[s], kb * BK, m0);
          tma_load_2d_mc(sm.b[s] + rank * kBPartBytes, &tmB, &sm.full[s], kb * BK,
                         n0 + rank * (BN / kCluster), (uint16_t)((1u << kCluster) - 1));
        }
      }
      // before the CTA exits: every copy into it has landed (its own and the
      // peer's multicasts), and both CTAs' last MMA commits have arrived here
      for (int c2 = c > kStages ? c - kStages : 0; c2 < c; ++c2) {
        wait_bar(&sm.full[c2 % kStages], (c2 / kStages) & 1, status);
        wait_bar(&sm.empty[c2 % kStages], (c2 / kStages) & 1, status);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t id = ptx::idesc_bf16(BM, BN, false);
      const uint64_t da = ptx::sdesc_sw128(ptx::smem_addr(sm.a[0]));
      const uint64_t db = ptx::sdesc_sw128(ptx::smem_addr(sm.b[0]));
      int c = 0;
      int j = 0;  // this CTA's tile count
      for (int t = q0; t < n_tiles; t += nq, ++j) {
        const int acc = j & 1;
        // accumulator acc was last used by tile j - 2: wait until drained
        if (j >= 2) wait_bar(&sm.acc_empty[acc], ((j >> 1) - 1) & 1, status);
        ptx::tc_fence_after();
        const uint32_t d = tmem + BN * acc;
        for (int kb = 0; kb < nk; ++kb, ++c) {
          const int s = c % kStages;
          wait_bar(&sm.full[s], (c / kStages) & 1, status);
          ptx::tc_fence_after();
          const uint64_t a0 = da + s * (kABytes >> 4), b0 = db + s * (kBBytes >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            ptx::mma_f16_ss(d, a0 + 2 * kk, b0 + 2 * kk, id, (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit_mc(&sm.empty[s], (uint16_t)((1u << kCluster) - 1));  // both CTAs' stage s
        }
        ptx::mma_commit(&sm.acc_full[acc]);
      }
    }
  } else {
    // epilogue: warp w owns TMEM lanes 32*(w%4) .. +31 = tile rows
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
    int j = 0;
    for (int t = q0; t < n_tiles; t += nq, ++j) {
      const int acc = j & 1;
      const int m0 = m0_of(t), n0 = n0_of(t);
      wait_bar(&sm.acc_full[acc], (j >> 1) & 1, status);
      ptx::tc_fence_after();
      store_tile(tmem + lanes + BN * acc, m0 + row, n0, M, N, Y, out_mode);
      // this warp's reads of the accumulator are complete (tmem_wait_ld in
      // store_tile): hand it back to the MMA thread
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sm.acc_empty[acc]);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA exits while the other may still write into it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 2 * BN);
  }
}

// wgu[256 j + c] = wg[128 j + c] (c < 128), wu[128 j + c - 128] (c >= 128):
// rows of K bf16, copied 16 bytes at a time
__global__ void interleave_gu_kernel(const uint4 *__restrict__ wg, const uint4 *__restrict__ wu,
                                     uint4 *__restrict__ wgu, int d_ff, int k16) {
  const int64_t total = (int64_t)2 * d_ff * k16;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / k16, c16 = i % k16;
    const int64_t j = r / 256, c = r % 256;
    const uint4 *src = c < 128 ? wg + (128 * j + c) * k16 : wu + (128 * j + c - 128) * k16;
    wgu[i] = src[c16];
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiled)f;
  }
  return fn;
}

// row-major [rows][K] bf16, box = box_rows x 64 (128-byte swizzle)
bool make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t K, int box_rows) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(int M, int N, int K, const void *x, const void *w, void *y, int out_mode,
                        uint32_t *status, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  CUtensorMap ma, mb;
  if (!make_map(&ma, x, M, K, BM) || !make_map(&mb, w, N, K, BN / kCluster))
    return cudaErrorInvalidValue;
  const int smem = (int)sizeof(GemmSmem) + 1024;
  // per device, so set on every launch (cheap)
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // one wave of clusters: as many as can be resident at once (one CTA per
  // SM; a GPC with an odd SM count leaves one SM out), at most one per pair
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCluster);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, gemm_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  const int64_t n_groups = (int64_t)((N + BN - 1) / BN) * ((M + kCluster * BM - 1) / (kCluster * BM));
  const unsigned grid = (unsigned)(kCluster * (n_groups < clusters ? n_groups : clusters));
  gemm_kernel<<<grid, kThreads, smem, s>>>(ma, mb, M, N, K, y, out_mode, status);
  return cudaGetLastError();
}

cudaError_t launch_interleave_gu(const void *wg, const void *wu, void *wgu, int d_ff, int K,
                                 cudaStream_t s) {
  if ((d_ff % 128) || (K % 8)) return cudaErrorInvalidValue;
  const int k16 = K / 8;
  interleave_gu_kernel<<<1216, 256, 0, s>>>((const uint4 *)wg, (const uint4 *)wu, (uint4 *)wgu,
                                            d_ff, k16);
  return cudaGetLastError();
}

}  // namespace akv
