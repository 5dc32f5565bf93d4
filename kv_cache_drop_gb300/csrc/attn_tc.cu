// bf16 segment-batch attention on the 5th-generation tensor cores (tcgen05,
// TMEM accumulators, TMA loads), sm_103a.
//
// Operands: rotated K and the permuted V are fp16 copies (see the
// pre-pass); each softmax thread rotates its own query row (raw bf16 row,
// cos/sin from the pre-pass's per-row table) to fp16 as it loads it; P is
// produced as fp16 by a packed fp16 exp; both products accumulate in fp32.  Row sums of P come from the tensor core too: the PV
// product runs with N = 80, its B operand being the V tile (columns 0-63)
// followed by a constant tile of ones (columns 64-79), so column 64 of the
// accumulator is the row sum and the softmax threads never add.
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
//   warp 8     TMA producer: K and V windows through a kStages-deep ring
//   warp 9     TMEM allocator + single-thread tcgen05.mma issuer
// TMEM columns: S0 [0,128) S1 [128,256) O0 [256,336) O1 [336,416)
// (O columns 64-79 hold the row sum), Q0 [416,448) Q1 [448,480).  Q is
// written into TMEM once per CTA by the softmax threads and is the A operand
// of the score product, so that product reads only K from shared memory
// (operands read from shared memory are limited to ~128 B/clk per SM, which
// two shared-memory operands per MMA saturate).  P_i (fp16, two per 32-bit column)
// overwrites the first 64 columns of S_i once S_i is in registers, and the
// PV product reads it from there (A operand in TMEM): P never touches shared
// memory, whose bandwidth the K=16 MMAs would otherwise saturate.  S_i(n+1)
// is issued after PV_i(n) by the same thread, and tcgen05.mma operations of
// one thread execute in issue order, so it cannot overwrite P_i(n) early.
// Per window n the issue order is S0(n) S1(n) | PV0(n) S0(n+1) PV1(n) S1(n+1):
// while one softmax group turns S into P the tensor core works for the other.
// O stays in TMEM for the whole tile.  The running max is only raised (and O rescaled)
// when it grows by more than 2^8, so O is rarely touched.
// Every barrier wait is bounded; a timeout sets a bit in the workspace status
// word, after which every blocked wait in the grid returns within a poll
// interval (about 4 us) so the launch ends.
#include "common.cuh"
#include "tc_ptx.cuh"

#include <cuda.h>

namespace akv {
namespace {

constexpr int kStages = 5;
constexpr int kThreads = 320;
constexpr int kProdWarp = 8, kMmaWarp = 9;
constexpr uint32_t kTileBytes = 128 * 64 * 2;  // 128 rows x 64 bf16
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitBudget = 1000000000LL;  // SM clocks (~0.5 s)
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)
constexpr float kRescaleThreshold = 8.0f;                 // log2 units
// 2^f on [-1/2, 1/2] as a cubic (least-squares fit with relative-error
// weights, max relative error 7.5e-5: below half an fp16 ulp)
constexpr float kE0 = 0.99992806f, kE1 = 0.69326097f, kE2 = 0.24261113f, kE3 = 0.05517167f;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23: x + it holds rint(x) in its low bits
// hardware named barriers (0 is __syncthreads)
// Named barrier kBarP + i, one generation per window n (plus one for the
// prologue): softmax group i syncs once P_i(n) is in TMEM (128 threads),
// the TMA producer syncs once window n+1 has landed (32), and the MMA warp
// syncs before issuing P_i.V(n) and S_i(n+1) (32).  Every role waits for
// each generation to complete, so the counts of two generations never mix.
constexpr int kBarP = 3;
constexpr int kBarPCount = 192;

struct __align__(1024) Smem {
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint8_t ones[kTileBytes];     // fp16 1.0, right after v: second MN atom of the PV B operand
  uint64_t bar_kv[kStages];
  uint64_t bar_s[2], bar_done;
  uint32_t tmem_base;
};

// Bounded wait; on timeout flags the grid (status word) so that every wait
// still blocked returns within a poll interval.  Control flow continues
// either way, so warp-collective instructions stay convergent.
__device__ __forceinline__ void wait_bar(uint64_t *bar, uint32_t parity, uint32_t *status) {
  ptx::mbar_wait_grid(bar, parity, status, kStatusWaitTimeout, kWaitBudget);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, PlanDev p,
                   __nv_bfloat16 *__restrict__ out, int n_pairs) {
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // head pair major: the CTAs in flight share one KV head's K/V windows,
  // which then stay in L2; query tiles by decreasing window count within it
  const int qi = p.order[blockIdx.x % p.n_qtiles], pair = blockIdx.x / p.n_qtiles;
  const QTile qt = p.qtiles[qi];
  const int grp = p.Hq / p.Hkv;
  const int h0 = 2 * pair, g = h0 / grp;
  const int n_win = qt.win_cnt;
  const int T = (int)p.T;

  // softmax threads: this row's raw query and cos/sin, loaded first so that
  // their memory latency overlaps the CTA's set-up below
  uint4 qraw[8];
  float4 qcs[16];
  if (warp < kProdWarp) {
    const int row = threadIdx.x & 127, t = qt.t0 + row;
    if (row < qt.len) {
      const uint4 *qrow = reinterpret_cast<const uint4 *>(
          static_cast<const __nv_bfloat16 *>(p.q) + ((int64_t)t * p.Hq + h0 + (warp >> 2)) * kD);
      const float4 *cs4 = reinterpret_cast<const float4 *>(p.qcs + (int64_t)t * (kD / 2));
#pragma unroll
      for (int c = 0; c < 8; ++c) qraw[c] = __ldg(qrow + c);
#pragma unroll
      for (int c = 0; c < 16; ++c) qcs[c] = __ldg(cs4 + c);
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(&sm.bar_kv[s], 1);
    for (int i = 0; i < 2; ++i) ptx::mbar_init(&sm.bar_s[i], 1);
    ptx::mbar_init(&sm.bar_done, 1);
    ptx::fence_barrier_init();
  }
  {
    uint4 *o = reinterpret_cast<uint4 *>(sm.ones);
    const uint4 one8 = make_uint4(0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u);
    for (int i = threadIdx.x; i < (int)(kTileBytes / 16); i += kThreads) o[i] = one8;
    ptx::fence_proxy_async_smem();  // visible to the tensor core
  }
  if (warp == kMmaWarp) ptx::tmem_alloc(&sm.tmem_base, kTmemCols);
  if (warp == kProdWarp && lane == 0) {
    ptx::tma_prefetch_desc(&tmK);
    ptx::tma_prefetch_desc(&tmV);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == kProdWarp) {
    // The whole warp runs the loop (named barriers count all 32 lanes);
    // lane 0 issues the copies.  The producer takes part in every
    // generation of both P barriers, so it cannot run ahead of them; it
    // refills the stage of window n-1 while window n is in flight.  That
    // stage is free without a wait: generation n+1 of P_1 completes only
    // after softmax group 1 has seen S_1(n) complete, and the commit that
    // signalled S_1(n) tracks every MMA issued before it, P_1.V(n-1) -- the
    // last reader of the stage -- included.
    const int krow = (qt.ver * p.Hkv + g) * T, vrow = g * T;
    auto load = [&](int n) {
      if (lane == 0) {
        const int st = n % kStages;
        const int w = (int)(p.windows[qt.win_off + n] & ~kWinFull);
        ptx::mbar_expect_tx(&sm.bar_kv[st], 2 * kTileBytes);
        ptx::tma_load_2d(sm.k[st], &tmK, &sm.bar_kv[st], 0, krow + w);
        ptx::tma_load_2d(sm.v[st], &tmV, &sm.bar_kv[st], 0, vrow + w);
      }
    };
    for (int n = 0; n < n_win && n < kStages; ++n) load(n);
    wait_bar(&sm.bar_kv[0], 0, p.status);
    ptx::named_bar_sync(kBarP + 0, kBarPCount);
    ptx::named_bar_sync(kBarP + 1, kBarPCount);
    for (int n = 0; n < n_win; ++n) {
      if (n + 1 < n_win)
        wait_bar(&sm.bar_kv[(n + 1) % kStages], ((n + 1) / kStages) & 1, p.status);
      ptx::named_bar_sync(kBarP + 0, kBarPCount);
      ptx::named_bar_sync(kBarP + 1, kBarPCount);
      const int m = n - 1 + kStages;  // refill the stage of window n-1
      if (n >= 1 && m < n_win) load(m);
    }
    // every copy was waited for above: none is in flight when the CTA exits
  } else if (warp == kMmaWarp) {
    // The whole warp follows the loop (named barriers); lane 0 issues.  It
    // never polls a shared-memory barrier between MMAs: each such poll costs
    // the issuing thread ~200 clocks, during which the tensor core's short
    // instruction queue runs dry.
    constexpr uint32_t idS = ptx::idesc_f16(128, 128, false);  // fp16 Qr x fp16 Kr
    constexpr uint32_t idO = ptx::idesc_f16(128, 80, true);    // fp16 P x [fp16 V | ones]
    // Descriptors are built once; per MMA only a small constant is added to
    // the address field (16-byte units): +2 per 16-element K step of a
    // K-major operand, +128 per 16-key step of the MN-major V operand, and
    // 1024 per 16 KiB tile.
    constexpr uint64_t kTileStep = kTileBytes >> 4;
    const uint64_t dk = ptx::sdesc_sw128(ptx::smem_addr(sm.k[0]));
    // V stage st: start address one tile per stage further on, and the
    // ones atom (kStages - st) tiles beyond it (leading-byte offset, bits 16-29)
    const uint64_t dv0 = ptx::sdesc_sw128(ptx::smem_addr(sm.v[0]), kStages * kTileBytes);
    const bool leader = lane == 0;
    auto issue_s = [&](int i, int st) {
      if (!leader) return;
      const uint64_t b0 = dk + st * kTileStep;
      // Q_i in TMEM: 64 dims as 32 packed columns, 8 per K step
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        ptx::mma_f16_ts(tmem + 128 * i, tmem + 416 + 32 * i + 8 * kk, b0 + 2 * kk, idS, kk > 0);
      ptx::mma_commit(&sm.bar_s[i]);
    };
    auto issue_o = [&](int i, int st, bool acc) {
      if (!leader) return;
      const uint64_t vd = dv0 + (uint64_t)st * kTileStep - (((uint64_t)st * kTileStep) << 16);
      // P_i: 128 keys as 64 packed columns at the start of S_i, 8 per K step
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        ptx::mma_f16_ts(tmem + 256 + 80 * i, tmem + 128 * i + 8 * kk, vd + 128 * kk, idO,
                        (acc || kk > 0) ? 1u : 0u);
    };
    ptx::named_bar_sync(kBarP + 0, kBarPCount);  // Q_0 in TMEM, window 0 landed
    ptx::named_bar_sync(kBarP + 1, kBarPCount);  // Q_1 in TMEM
    ptx::tc_fence_after();
    issue_s(0, 0);
    issue_s(1, 0);
    for (int n = 0; n < n_win; ++n) {
      const int st = n % kStages;
      const int st1 = (n + 1) % kStages;
      ptx::named_bar_sync(kBarP + 0, kBarPCount);  // P_0(n) in TMEM, window n+1 landed
      ptx::tc_fence_after();
      issue_o(0, st, n > 0);
      if (n + 1 < n_win) issue_s(0, st1);
      ptx::named_bar_sync(kBarP + 1, kBarPCount);
      ptx::tc_fence_after();
      issue_o(1, st, n > 0);
      if (n + 1 < n_win) issue_s(1, st1);
    }
    if (leader) ptx::mma_commit(&sm.bar_done);
    wait_bar(&sm.bar_done, 0, p.status);
  } else {
    // softmax: i = head within the pair, row = query row = TMEM lane
    const int i = warp >> 2;
    const int row = threadIdx.x & 127;
    const bool valid = row < qt.len;
    const int t = qt.t0 + row;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + i * 128;
    const uint32_t tO = tmem + lane_base + 256 + i * 80;
    const uint32_t tL = tO + 64;  // row sums
    {  // this row's query rotated at its position, as fp16 (64 dims = 32
       // packed words) into TMEM: the raw bf16 row and the row's cos/sin
       // from the pre-pass's table (loaded at the start); the pair
       // (d, d + 32) turns by angle d, in fp32 as the pre-pass rotates keys
      uint32_t qw[32];
      bool ovf = false;
      if (valid) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // dims 8c..8c+7 with 8c+32..8c+39
          float x1[8], x2[8], y1[8], y2[8];
          chunk_to_f32<__nv_bfloat16>(qraw[c], x1);
          chunk_to_f32<__nv_bfloat16>(qraw[c + 4], x2);
          float big = 0.f;
#pragma unroll
          for (int e2 = 0; e2 < 4; ++e2) {
            const float4 t4 = qcs[4 * c + e2];  // (cos, sin) of dims 8c+2e2, +1
            const float co[2] = {t4.x, t4.z}, si[2] = {t4.y, t4.w};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int e = 2 * e2 + h;
              y1[e] = x1[e] * co[h] - x2[e] * si[h];
              y2[e] = x1[e] * si[h] + x2[e] * co[h];
              big = fmaxf(big, fmaxf(fabsf(y1[e]), fabsf(y2[e])));
            }
          }
          ovf |= !(big <= 65504.f);
          const uint4 a = f32_to_chunk<__half>(y1), b = f32_to_chunk<__half>(y2);
          qw[4 * c] = a.x;
          qw[4 * c + 1] = a.y;
          qw[4 * c + 2] = a.z;
          qw[4 * c + 3] = a.w;
          qw[16 + 4 * c] = b.x;
          qw[16 + 4 * c + 1] = b.y;
          qw[16 + 4 * c + 2] = b.z;
          qw[16 + 4 * c + 3] = b.w;
        }
      } else {
#pragma unroll
        for (int w = 0; w < 32; ++w) qw[w] = 0u;
      }
      if (ovf) atomicOr(p.status, kStatusFp16Range);
      ptx::tmem_st32(tmem + lane_base + 416 + 32 * i, qw);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::named_bar_sync(kBarP + i, kBarPCount);
    }
    const float2 scale2 = make_float2(kScaleLog2, kScaleLog2);
    float m_run = -INFINITY;
    // this row's visibility bits for the tile's partial windows (precomputed
    // per plan), loaded one partial window ahead
    int n_partial = 0;
    const uint4 *mrow = p.mask + (int64_t)qt.pm_off * kTileQ + row;
    uint4 vis_next = qt.pm_cnt > 0 ? __ldg(mrow) : make_uint4(0u, 0u, 0u, 0u);
    // window list read two entries ahead, so no iteration waits on its load
    uint32_t win = p.windows[qt.win_off];
    uint32_t win_nx = n_win > 1 ? p.windows[qt.win_off + 1] : 0u;
    for (int n = 0; n < n_win; ++n) {
      const uint32_t win_next = win_nx;
      win_nx = n + 2 < n_win ? p.windows[qt.win_off + n + 2] : 0u;
      const bool full = (win & kWinFull) != 0;
      // visibility bits of this row over the window's 128 keys
      uint32_t vis[4] = {~0u, ~0u, ~0u, ~0u};
      if (!full) {
        vis[0] = vis_next.x;
        vis[1] = vis_next.y;
        vis[2] = vis_next.z;
        vis[3] = vis_next.w;
        if (++n_partial < qt.pm_cnt) vis_next = __ldg(mrow + (int64_t)n_partial * kTileQ);
      }
      win = win_next;
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
      // row max: eight independent 3-input chains over columns k8 + 8j
      // (j = 0-2, then pairs up to j = 14, then j = 15), then a short tree
      float mx8[8];
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8)
        mx8[k8] = ptx::max3(__uint_as_float(sr[k8]), __uint_as_float(sr[8 + k8]),
                            __uint_as_float(sr[16 + k8]));
#pragma unroll
      for (int c = 24; c + 16 <= 120; c += 16)
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8)
          mx8[k8] = ptx::max3(mx8[k8], __uint_as_float(sr[c + k8]), __uint_as_float(sr[c + 8 + k8]));
#pragma unroll
      for (int k8 = 0; k8 < 8; ++k8) mx8[k8] = fmaxf(mx8[k8], __uint_as_float(sr[120 + k8]));
      const float mx = fmaxf(ptx::max3(mx8[0], mx8[1], mx8[2]),
                             fmaxf(ptx::max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = fmaxf(m_run, mx * kScaleLog2);
      const bool need = m_new > m_run + kRescaleThreshold;
      const bool any = __any_sync(0xffffffffu, need);
      float alpha = 1.f;
      if (need) {
        alpha = ptx::ex2(m_run - m_new);  // 0 on the first raise from -inf
        m_run = m_new;
      }
      const float mref = m_run == -INFINITY ? 0.f : m_run;
      const float2 neg2 = make_float2(-mref, -mref);
      // p = 2^(s * scale - m): packed fp32 FMA, then a packed fp16 exp whose
      // result is already the fp16 A operand of the P x V product.  Word k of
      // the row holds keys 2k, 2k+1 and overwrites S column k (already read).
      // One pair in four takes 2^x on the FMA pipe instead (the exp unit is
      // the busiest one): x clamped at -100 (2^-100 is 0 in fp16), split
      // into n = rint(x) and f = x - n, 2^f by the cubic, n added to the
      // exponent field, then one conversion to fp16.
#pragma unroll
      for (int qtr = 0; qtr < 4; ++qtr) {  // quarters: fewer registers live at once
        uint32_t pw[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int k2 = 16 * qtr + k;
          const float2 sv = make_float2(__uint_as_float(sr[2 * k2]), __uint_as_float(sr[2 * k2 + 1]));
          const float2 x = __ffma2_rn(sv, scale2, neg2);
          if ((k2 & 3) == 3) {
            const float2 xc = make_float2(fmaxf(x.x, -100.f), fmaxf(x.y, -100.f));
            const float2 j = __fadd2_rn(xc, make_float2(kRoundMagic, kRoundMagic));
            const float2 nf = __fadd2_rn(j, make_float2(-kRoundMagic, -kRoundMagic));
            const float2 f = __ffma2_rn(nf, make_float2(-1.f, -1.f), xc);
            float2 q = __ffma2_rn(make_float2(kE3, kE3), f, make_float2(kE2, kE2));
            q = __ffma2_rn(q, f, make_float2(kE1, kE1));
            q = __ffma2_rn(q, f, make_float2(kE0, kE0));
            const float r0 = __uint_as_float(__float_as_uint(q.x) + (__float_as_uint(j.x) << 23));
            const float r1 = __uint_as_float(__float_as_uint(q.y) + (__float_as_uint(j.y) << 23));
            __half2 h = __floats2half2_rn(r0, r1);
            pw[k] = *reinterpret_cast<uint32_t *>(&h);
          } else {
            __half2 h = __floats2half2_rn(x.x, x.y);
            pw[k] = ptx::ex2_f16x2(*reinterpret_cast<uint32_t *>(&h));
          }
        }
        ptx::tmem_st16(tS + 16 * qtr, pw);
      }
      if (n > 0 && any) {  // rare: the running max grew by more than 2^8
        // O may be rescaled only once PV(n-1) has completed: it has, since
        // the commit that signalled S(n) tracks every MMA issued before it
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
        uint32_t lsum[16];
        ptx::tmem_ld16(tL, lsum);
        ptx::tmem_wait_ld();
        ptx::reg_fence16(lsum);
#pragma unroll
        for (int c = 0; c < 16; ++c) lsum[c] = __float_as_uint(__uint_as_float(lsum[c]) * alpha);
        ptx::tmem_st16(tL, lsum);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      // P_i (and a rescaled O_i) are in TMEM.  The softmax waits for the
      // generation to complete (its next S_i is issued after it anyway), so
      // no role can reach a later generation of this barrier before the
      // current one has all its arrivals, even after a timed-out wait
      ptx::named_bar_sync(kBarP + i, kBarPCount);
    }
    wait_bar(&sm.bar_done, 0, p.status);  // the last PV
    ptx::tc_fence_after();
    uint32_t o[64], lsum[16];
    ptx::tmem_ld32(tO, o);
    ptx::tmem_ld32(tO + 32, o + 32);
    ptx::tmem_ld16(tL, lsum);
    ptx::tmem_wait_ld();
    ptx::reg_fence32(o);
    ptx::reg_fence32(o + 32);
    ptx::reg_fence16(lsum);
    if (valid) {
      const float inv = 1.f / __uint_as_float(lsum[0]);
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
  CUtensorMap mk, mv;
  if (!make_map(&mk, p.kr, (int64_t)p.max_ver * p.Hkv * p.T, CU_TENSOR_MAP_DATA_TYPE_FLOAT16) ||
      !make_map(&mv, p.vp, (int64_t)p.Hkv * p.T, CU_TENSOR_MAP_DATA_TYPE_FLOAT16))
    return cudaErrorInvalidValue;
  const int smem = (int)sizeof(Smem) + 1024;
  // per device, so set on every launch (cheap)
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int n_pairs = p.Hq / 2;
  const int64_t grid = (int64_t)p.n_qtiles * n_pairs;
  attn_tc_kernel<<<(unsigned)grid, kThreads, smem, s>>>(mk, mv, p, (__nv_bfloat16 *)out,
                                                        n_pairs);
  return cudaGetLastError();
}

}  // namespace akv
