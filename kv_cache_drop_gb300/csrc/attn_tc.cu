// bf16 segment-batch attention on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA loads), sm_103a.
//
// Operands: rotated Q and K are fp16 copies (see the pre-pass), P and V are
// bf16; both products accumulate in fp32.
//
// What it computes (paper review page section 4.2, Appendix A.1.1): for each
// query row t of a tile and each key slot j of the tile's 128-key windows,
//   S = Qr[t] . Kr_v[j] / sqrt(D),  visible(t, j) <=> u(j) <= t and seg(t) < dseg(j),
//   O[t] = sum_j softmax_j(S) V[j]   (online softmax over the windows).
//
// CTA = one 128-row query tile x two query heads of one KV group (the two
// heads share every K/V window: GQA).  Warp roles:
//   warps 0-3  softmax for head 0 (thread = query row = TMEM lane)
//   warps 4-7  softmax for head 1
//   warp 8     TMA producer: Q tiles once, then K and V windows through a
//              kStages-deep ring
//   warp 9     TMEM allocator + single-thread tcgen05.mma issuer
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,320) O1 [320,384).
// Per window n the issue order is S0(n) S1(n) | PV0(n) S0(n+1) PV1(n) S1(n+1):
// while one softmax group turns S into P the tensor core works for the other.
// P goes to shared memory as bf16 (128-byte swizzled, K-major); O stays in
// TMEM for the whole tile.  The running max is only raised (and O rescaled)
// when it grows by more than 2^8, so O is rarely touched.
// Every barrier wait is bounded; a timeout sets a bit in the workspace status
// word, after which all waits in the grid return at once so the launch ends.
#include "common.cuh"
#include "tc_ptx.cuh"

#include <cuda.h>

namespace akv {
namespace {

constexpr int kStages = 3;
constexpr int kThreads = 320;
constexpr int kProdWarp = 8, kMmaWarp = 9;
constexpr uint32_t kTileBytes = 128 * 64 * 2;  // 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitBudget = 1000000000LL;  // SM clocks (~0.5 s)
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)
constexpr float kRescaleThreshold = 8.0f;                 // log2 units

struct __align__(1024) Smem {
  uint8_t q[2][kTileBytes];
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint8_t p[2][2][kTileBytes];  // [head][key half]
  int32_t mask_u[2][2][128];    // [head][buffer][column]
  int32_t mask_d[2][2][128];
  uint64_t bar_q;
  uint64_t bar_k[kStages], bar_v[kStages], bar_empty[kStages];
  uint64_t bar_s[2], bar_p[2], bar_o[2], bar_done;
  uint32_t tmem_base;
};

// Bounded wait; on timeout flags the grid (status word) so every later wait
// returns immediately.  Control flow continues either way, so warp-collective
// instructions stay convergent.
__device__ __forceinline__ void wait_bar(uint64_t *bar, uint32_t parity, uint32_t *status) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  if (*(volatile uint32_t *)status) return;
  if (!ptx::mbar_wait(bar, parity, kWaitBudget)) atomicOr(status, kStatusWaitTimeout);
}

__device__ __forceinline__ uint64_t desc_k_major(uint32_t saddr) {
  return ptx::sdesc_sw128(saddr);
}
// MN-major operand (V: keys along K, head dim along N): 8-key groups 1024 B
// apart; the same value is written to both stride fields.
__device__ __forceinline__ uint64_t desc_mn_major(uint32_t saddr) {
  return ptx::sdesc_sw128(saddr, 1024);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, PlanDev p,
                   __nv_bfloat16 *__restrict__ out, int n_pairs) {
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qi = p.order[blockIdx.x / n_pairs], pair = blockIdx.x % n_pairs;
  const QTile qt = p.qtiles[qi];
  const int grp = p.Hq / p.Hkv;
  const int h0 = 2 * pair, g = h0 / grp;
  const int n_win = qt.win_cnt;
  const int T = (int)p.T;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&sm.bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&sm.bar_k[s], 1);
      ptx::mbar_init(&sm.bar_v[s], 1);
      ptx::mbar_init(&sm.bar_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&sm.bar_s[i], 1);
      ptx::mbar_init(&sm.bar_p[i], 128);
      ptx::mbar_init(&sm.bar_o[i], 1);
    }
    ptx::mbar_init(&sm.bar_done, 1);
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
  if (warp == kProdWarp && lane == 0) {
    ptx::tma_prefetch_desc(&tmQ);
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kProdWarp) {
    if (lane == 0) {
      ptx::mbar_expect_tx(&sm.bar_q, 2 * kTileBytes);
      ptx::tma_load_2d(sm.q[0], &tmQ, &sm.bar_q, 0, h0 * T + qt.t0);
      ptx::tma_load_2d(sm.q[1], &tmQ, &sm.bar_q, 0, (h0 + 1) * T + qt.t0);
      const int krow = (qt.ver * p.Hkv + g) * T, vrow = g * T;
      for (int n = 0; n < n_win; ++n) {
        const int st = n % kStages;
        if (n >= kStages) wait_bar(&sm.bar_empty[st], ((n / kStages) - 1) & 1, p.status);
        const int w = (int)(p.windows[qt.win_off + n] & ~kWinFull);
        ptx::mbar_expect_tx(&sm.bar_k[st], kTileBytes);
        ptx::tma_load_2d(sm.k[st], &tmK, &sm.bar_k[st], 0, krow + w);
        ptx::mbar_expect_tx(&sm.bar_v[st], kTileBytes);
        ptx::tma_load_2d(sm.v[st], &tmV, &sm.bar_v[st], 0, vrow + w);
      }
      // no copy may still be in flight when the CTA exits
      for (int n = n_win > kStages ? n_win - kStages : 0; n < n_win; ++n) {
        wait_bar(&sm.bar_k[n % kStages], (n / kStages) & 1, p.status);
        wait_bar(&sm.bar_v[n % kStages], (n / kStages) & 1, p.status);
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      constexpr uint32_t idS = ptx::idesc_f16(128, 128, false);   // fp16 Qr x fp16 Kr
      constexpr uint32_t idO = ptx::idesc_bf16(128, 64, true);   // bf16 P x bf16 V
      const uint32_t q_base = ptx::smem_addr(sm.q[0]);
      auto issue_s = [&](int i, int st) {
        const uint32_t kb = ptx::smem_addr(sm.k[st]), qb = q_base + i * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f16_ss(tmem + 128 * i, desc_k_major(qb + 32 * kk), desc_k_major(kb + 32 * kk),
                          idS, kk > 0);
        ptx::mma_commit(&sm.bar_s[i]);
      };
      auto issue_o = [&](int i, int st, bool acc) {
        const uint32_t vb = ptx::smem_addr(sm.v[st]);
        const uint32_t pb = ptx::smem_addr(sm.p[i][0]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_f16_ss(tmem + 256 + 64 * i,
                          desc_k_major(pb + (kk >> 2) * kTileBytes + 32 * (kk & 3)),
                          desc_mn_major(vb + 2048 * kk), idO, (acc || kk > 0) ? 1u : 0u);
        ptx::mma_commit(&sm.bar_o[i]);
      };
      wait_bar(&sm.bar_q, 0, p.status);
      wait_bar(&sm.bar_k[0], 0, p.status);
      ptx::tc_fence_after();
      issue_s(0, 0);
      issue_s(1, 0);
      for (int n = 0; n < n_win; ++n) {
        const int st = n % kStages;
        const int st1 = (n + 1) % kStages;
        wait_bar(&sm.bar_v[st], (n / kStages) & 1, p.status);
        wait_bar(&sm.bar_p[0], n & 1, p.status);
        ptx::tc_fence_after();
        issue_o(0, st, n > 0);
        if (n + 1 < n_win) {
          wait_bar(&sm.bar_k[st1], ((n + 1) / kStages) & 1, p.status);
          ptx::tc_fence_after();
          issue_s(0, st1);
        }
        wait_bar(&sm.bar_p[1], n & 1, p.status);
        ptx::tc_fence_after();
        issue_o(1, st, n > 0);
        if (n + 1 < n_win) issue_s(1, st1);
        ptx::mma_commit(&sm.bar_empty[st]);
      }
      ptx::mma_commit(&sm.bar_done);
      wait_bar(&sm.bar_done, 0, p.status);
    }
  } else {
    // softmax: i = head within the pair, row = query row = TMEM lane
    const int i = warp >> 2;
    const int row = threadIdx.x & 127;
    const bool valid = row < qt.len;
    const int t = qt.t0 + row;
    const int seg = p.tok_seg[valid ? t : qt.t0];
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + i * 128;
    const uint32_t tO = tmem + lane_base + 256 + i * 64;
    float m_run = -INFINITY, l_run = 0.f;
    int n_partial = 0;
    for (int n = 0; n < n_win; ++n) {
      const uint32_t win = p.windows[qt.win_off + n];
      const bool full = (win & kWinFull) != 0;
      // visibility bits of this row over the window's 128 keys
      uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
      if (!full) {  // uniform over the group: stage the window's key tags
        const int buf = n_partial & 1;
        ++n_partial;
        const int j = (int)(win & ~kWinFull) + row;
        sm.mask_u[i][buf][row] = __ldg(p.slot_u + j);
        sm.mask_d[i][buf][row] = __ldg(p.slot_dseg + j);
        ptx::named_bar_sync(1 + i, 128);
        const int32_t *mu = sm.mask_u[i][buf], *md = sm.mask_d[i][buf];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t bits = 0;
#pragma unroll 8
          for (int c = 0; c < 32; ++c)
            bits |= (uint32_t)(mu[32 * w + c] <= t && seg < md[32 * w + c]) << c;
          vis[w] = bits;
        }
      }
      wait_bar(&sm.bar_s[i], n & 1, p.status);
      ptx::tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + 32 * c, sr + 32 * c);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::reg_fence32(sr + 32 * c);
      if (!full) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (!((vis[c >> 5] >> (c & 31)) & 1u)) sr[c] = 0xff800000u;  // -inf
      }
      float mx = __uint_as_float(sr[0]);
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
      const float m_new = fmaxf(m_run, mx * kScaleLog2);
      const bool need = m_new > m_run + kRescaleThreshold;
      const bool any = __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (need) {
        alpha = ptx::ex2(m_run - m_new);  // 0 on the first raise from -inf
        m_run = m_new;
      }
      const float mref = m_run == -INFINITY ? 0.f : m_run;
      // P(n) overwrites P(n-1): PV(n-1) was issued before S(n), so it has
      // completed by now and this wait returns at once
      if (n > 0) wait_bar(&sm.bar_o[i], (n - 1) & 1, p.status);
      float ls = 0.f;
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ptx::ex2(fmaf(__uint_as_float(sr[8 * ch + 2 * e]), kScaleLog2, -mref));
          const float p1 =
              ptx::ex2(fmaf(__uint_as_float(sr[8 * ch + 2 * e + 1]), kScaleLog2, -mref));
          ls += p0 + p1;
          w4[e] = pack_bf16(p0, p1);
        }
        const int c = ch & 7;
        uint8_t *dst = sm.p[i][ch >> 3] + row * 128 + ((c ^ (row & 7)) << 4);
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      l_run = l_run * alpha + ls;
      if (n > 0 && any) {  // rare: the running max grew by more than 2^8
        ptx::tc_fence_after();
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + 32 * hlf, o);
          ptx::tmem_wait_ld();
          ptx::reg_fence32(o);
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          ptx::tmem_st32(tO + 32 * hlf, o);
        }
        ptx::tmem_wait_st();
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&sm.bar_p[i]);
    }
    wait_bar(&sm.bar_o[i], (n_win - 1) & 1, p.status);
    ptx::tc_fence_after();
    uint32_t o[64];
    ptx::tmem_ld32(tO, o);
    ptx::tmem_ld32(tO + 32, o + 32);
    ptx::tmem_wait_ld();
    ptx::reg_fence32(o);
    ptx::reg_fence32(o + 32);
    if (valid) {
      const float inv = 1.f / l_run;
      uint4 *dst = reinterpret_cast<uint4 *>(out + ((int64_t)t * p.Hq + h0 + i) * kD);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          w4[e] = pack_bf16(__uint_as_float(o[8 * c + 2 * e]) * inv,
                            __uint_as_float(o[8 * c + 2 * e + 1]) * inv);
        dst[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
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

// 2-D view [rows][64] bf16, box 128 rows x 64 columns, 128-byte swizzle
bool make_map(CUtensorMap *m, void *base, int64_t rows, CUtensorMapDataType dt) {
  EncodeTiled enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kD, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attn_tc_bf16(const PlanDev &p, void *out, cudaStream_t s) {
  if (p.n_qtiles == 0) return cudaSuccess;
  if ((p.Hq / p.Hkv) % 2) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, p.qr, (int64_t)p.Hq * p.T, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) ||
      !make_map(&mk, p.kr, (int64_t)p.max_ver * p.Hkv * p.T, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) ||
      !make_map(&mv, p.vp, (int64_t)p.Hkv * p.T, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16))
    return cudaErrorInvalidValue;
  const int smem = (int)sizeof(Smem) + 1024;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int n_pairs = p.Hq / 2;
  const int64_t grid = (int64_t)p.n_qtiles * n_pairs;
  attn_tc_kernel<<<(unsigned)grid, kThreads, smem, s>>>(mq, mk, mv, p, (__nv_bfloat16 *)out,
                                                        n_pairs);
  return cudaGetLastError();
}

}  // namespace akv
