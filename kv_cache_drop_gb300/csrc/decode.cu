// Decode attention over the active cache in a page-size-1 pool (paper review
// page section 4 serving flow: decode reads only the active cache; system
// README: drop/repos work at page size 1).
//
// Split-KV: request b's index list is cut into chunks of `chunk` keys; one CTA
// takes (chunk, KV head g, request b) and produces a partial (row max m, row
// sum l, unnormalised output o) for the Hq/Hkv query heads of group g; the
// partials are merged by their log-sum-exp -- for bf16 inside the same
// launch, by the last CTA of each (request, KV head) to finish; for fp32 by
// a combine kernel.  bf16 with rotation on read and 4 or 8 KV heads takes
// all KV heads of a chunk per CTA (the rotation angles are shared) and
// merges in a second launch.
//
// bf16: the group's query heads form the rows of an m16n8k16 tensor-core tile
// (S = Q K^T with K rows as the B operand, then O += P V with P reused from
// the S accumulator registers); keys and values are gathered 16 rows at a
// time with 16-byte cp.async into an XOR-swizzled shared tile, several tiles
// in flight per warp.  The work is bound by the gather from HBM (2 x 128 B
// per key and head group); the tensor-core tile only keeps the arithmetic
// off the critical path.
// fp32: one thread per key, FMA dot products, block-level merge.
#include "common.cuh"

#include <algorithm>

namespace akv {
namespace {

constexpr int kChunk = 2048;     // keys per CTA of the fp32 kernel
constexpr int kMinChunk = 1024;  // bf16: chunk chosen per call in [kMinChunk, kMaxChunk]
constexpr int kMaxChunk = 4096;
constexpr int kMaxSplits = 1000;  // bf16: the in-kernel merge's weights fit shared memory
constexpr int kRChunk = 512;  // fp32 rotate-on-read: keys per CTA; bf16 all-heads: the least
constexpr int kWarps = 4;
constexpr int kTileKeys = 16;
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;

struct Partials {
  float *ml;  // [B][Hq][ns][2]  (m in log2 units, l)
  float *o;   // [B][Hq][ns][kD]
};

__host__ __device__ inline int n_splits(int max_kv, int chunk = kChunk) {
  return max_kv <= 0 ? 1 : (max_kv + chunk - 1) / chunk;
}

Partials partials(void *ws, int B, int Hq, int max_kv, int chunk = kChunk) {
  const int ns = n_splits(max_kv, chunk);
  Partials p;
  p.ml = (float *)ws;
  const size_t ml_bytes = ((size_t)B * Hq * ns * 2 * 4 + 255) / 256 * 256;
  p.o = (float *)((char *)ws + ml_bytes);
  return p;
}

int device_sms() {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 148;
  return sms;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 16 : 0;  // 0 source bytes: zero fill
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                        uint32_t &d) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c,
                                          uint32_t &d) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// byte offset of (row, 16-byte chunk) in a [16][64] bf16 tile, XOR swizzled
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Each CTA also counts itself done for its (request, KV head); the last one
// merges the group's split partials and writes the output (no separate
// combine launch).  With new_slot, the CTA that owns a request's last key
// first appends the step's token: K rotated at q_pos (the same rotation
// table as the query) and V, into pool slot new_slot[b].
//
// kRope (rotation on read): the pool holds keys before RoPE and kvpos gives
// each entry's position; a tile's 16 positions arrive with its K/V by
// cp.async, every lane forms cos/sin for the 16 (key, frequency) pairs of its
// K fragments (keys gid, gid + 8; the pair (d, d + 32) sits in k-steps ks and
// ks + 2 of the same lane), rotates them in fp32 registers and rounds the
// result to fp16 (11-bit significand); the query is split into fp16 hi + lo
// and S = qhi k + qlo k in fp16 MMAs.  Rotated keys must lie within the fp16
// range (|k| < 65504; a larger one gives inf).  The append is then a plain
// copy.
// The angles: a request's entries are in position order and mostly close
// together, so per tile lane f forms cos/sin(p0 theta_f) once for the tile's
// first position p0, and a key at p = p0 + delta, 0 <= delta < kDeltas,
// takes it rotated by delta theta_f (angle addition) from a per-CTA table
// of cos/sin(delta theta_f); other keys compute their angles directly.
constexpr int kStageBytes(bool rope) { return rope ? 4096 + 64 : 4096; }
constexpr int kDeltas = 64;
// table row: for frequency pair j = f / 2, float4 (cos f, sin f, cos f+1,
// sin f+1); rows padded to 20 float4 so that the two rows read by one
// 8-lane phase of a 16-byte load fall in different banks
constexpr int kDeltaRow = kD / 4 + 4;

// cos/sin of pos * theta by the fast sin/cos instructions (absolute error
// about 4e-7 on the reduced angle, |r| <= pi)
__device__ __forceinline__ void rope_cs_fast(float hi, float lo, int pos, float *c, float *s) {
  __sincosf(rope_angle(hi, lo, pos), s, c);
}

// cos/sin of pos * theta for frequencies f and f + 1 computed from the
// angle itself: keys kDeltas or more positions past their tile's first one,
// and positions beyond 2^18 (the double-precision path).  Rare, so kept out
// of line: the unrolled loop around its call stays small.
__device__ __noinline__ float4 rope_cs_direct2(const ThetaSmem &ts, const double *thd, int f,
                                               int pos) {
  float4 r;
  if (pos < -262144 || pos > 262144) {
    rope_cs(thd[f], (double)pos, &r.x, &r.y);
    rope_cs(thd[f + 1], (double)pos, &r.z, &r.w);
  } else {
    rope_cs_fast(ts.hi[f], ts.lo[f], pos, &r.x, &r.y);
    rope_cs_fast(ts.hi[f + 1], ts.lo[f + 1], pos, &r.z, &r.w);
  }
  return r;
}

template <bool kRope>
__global__ void __launch_bounds__(kWarps * 32, 4)
    decode_bf16_kernel(int Hq, int Hkv, const __nv_bfloat16 *__restrict__ q,
                       const int32_t *__restrict__ qpos, __nv_bfloat16 *kp, __nv_bfloat16 *vp,
                       const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                       Partials part, RopeTheta th, int *counters, __nv_bfloat16 *out,
                       const __nv_bfloat16 *k_new, const __nv_bfloat16 *v_new,
                       const int32_t *new_slot, int chunk, const int32_t *__restrict__ kvpos) {
  // dynamic smem: per warp kStages x (K tile 2 KiB + V tile 2 KiB [+ 16
  // positions]); reused for the merge of the warps' partials
  constexpr int kSB = kStageBytes(kRope);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float cs[kD / 2], sn[kD / 2];
  __shared__ ThetaSmem ts;
  __shared__ float4 dtab[kRope ? kDeltas * kDeltaRow : 1];
  __shared__ double thd[kRope ? kD / 2 : 1];
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int ns = gridDim.x;
  const int grp = Hq / Hkv;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int beg = indptr[b], n = indptr[b + 1] - beg;
  const int c0 = split * chunk, c1 = min(n, c0 + chunk);
  if (c0 >= n) {  // the merge reads only the splits that hold keys
    if (n <= 0 && split == 0)  // a request with no keys gets zeros
      for (int i = threadIdx.x; i < grp * kD; i += blockDim.x)
        out[((int64_t)b * Hq + g * grp) * kD + i] = __float2bfloat16_rn(0.f);
    return;
  }

  if (threadIdx.x < kD / 2) rope_cs_lane(th, threadIdx.x, qpos[b], &cs[threadIdx.x], &sn[threadIdx.x]);
  if (kRope) {
    stage_theta(th, ts);
    if (threadIdx.x < kD / 2) thd[threadIdx.x] = th.th[threadIdx.x];
    // delta table: thread = (frequency f, block of 16 deltas); the block's
    // first entry directly, then 15 steps of the delta = 1 rotation
    for (int u = threadIdx.x; u < (kD / 2) * (kDeltas / 16); u += blockDim.x) {
      const int f = u % (kD / 2), d0 = 16 * (u / (kD / 2));
      float c, sv, c1, s1;
      rope_cs_pair(th.hi[f], th.lo[f], d0, &c, &sv);
      rope_cs_pair(th.hi[f], th.lo[f], 1, &c1, &s1);
      float *row = reinterpret_cast<float *>(dtab) + 4 * (f >> 1) + 2 * (f & 1);
      for (int i = 0; i < 16; ++i) {
        row[(d0 + i) * 4 * kDeltaRow] = c;
        row[(d0 + i) * 4 * kDeltaRow + 1] = sv;
        const float cn = c * c1 - sv * s1;
        sv = sv * c1 + c * s1;
        c = cn;
      }
    }
  }
  __syncthreads();
  if (new_slot && c1 == n) {  // fused append of the step's token (head g)
    const int64_t src = ((int64_t)b * Hkv + g) * kD, dst = ((int64_t)new_slot[b] * Hkv + g) * kD;
    if (kRope) {  // the pool keeps keys before RoPE: a copy
      if (threadIdx.x < 2 * (kD / 8)) {
        const int c = threadIdx.x % (kD / 8);
        if (threadIdx.x < kD / 8)
          reinterpret_cast<uint4 *>(kp + dst)[c] = reinterpret_cast<const uint4 *>(k_new + src)[c];
        else
          reinterpret_cast<uint4 *>(vp + dst)[c] = reinterpret_cast<const uint4 *>(v_new + src)[c];
      }
    } else if (threadIdx.x < kD / 2) {
      const int f = threadIdx.x;
      const float x1 = __bfloat162float(k_new[src + f]), x2 = __bfloat162float(k_new[src + f + kD / 2]);
      kp[dst + f] = __float2bfloat16_rn(x1 * cs[f] - x2 * sn[f]);
      kp[dst + f + kD / 2] = __float2bfloat16_rn(x1 * sn[f] + x2 * cs[f]);
    } else if (threadIdx.x < kD / 2 + kD / 8) {
      const int c = threadIdx.x - kD / 2;
      reinterpret_cast<uint4 *>(vp + dst)[c] = reinterpret_cast<const uint4 *>(v_new + src)[c];
    }
    __syncthreads();  // the appended row is visible to this CTA's gathers
  }

  // Q fragments (A operand, rows = query heads of the group, 16 rows padded
  // with zeros), rotated at the query position; 1/sqrt(D) * log2(e) folded in.
  // The rotated query is not a bf16 value: it is split into hi + lo bf16
  // parts (hi = bf16(q), lo = bf16(q - hi)) and S = hi K^T + lo K^T, so the
  // scores carry ~16 mantissa bits of q at twice the (idle) MMA work.
  uint32_t qa[4][4], ql[4][4];
  {
    const float qs = 0.125f * kLog2e;
    float qv[2][16];  // [row half][element]: rows gid and gid+8
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = gid + 8 * hh;
      const bool ok = row < grp;
      const __nv_bfloat16 *qrow = q + ((int64_t)b * Hq + g * grp + (ok ? row : 0)) * kD;
      // elements held by this thread: ks*16 + {2tig, 2tig+1, 2tig+8, 2tig+9}
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = ks * 16 + 2 * tig + (e & 1) + (e >> 1) * 8;
          qv[hh][ks * 4 + e] = ok ? __bfloat162float(qrow[d]) : 0.f;
        }
    }
    // rotate: element d (< 32) pairs with d + 32, i.e. k-step ks with ks + 2
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = ks * 16 + 2 * tig + (e & 1) + (e >> 1) * 8;
          const float x1 = qv[hh][ks * 4 + e], x2 = qv[hh][(ks + 2) * 4 + e];
          qv[hh][ks * 4 + e] = (x1 * cs[d] - x2 * sn[d]) * qs;
          qv[hh][(ks + 2) * 4 + e] = (x1 * sn[d] + x2 * cs[d]) * qs;
        }
    // kRope: the score product runs in fp16 (the rotated keys are rounded
    // to fp16), so the query parts are fp16 too
    auto pk = [](float x, float y) { return kRope ? pack_f16(x, y) : pack_bf16(x, y); };
    auto lo = [](float x) {
      return kRope ? x - __half2float(__float2half_rn(x))
                   : x - __bfloat162float(__float2bfloat16_rn(x));
    };
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const float *a0 = &qv[0][ks * 4], *a1 = &qv[1][ks * 4];
      qa[ks][0] = pk(a0[0], a0[1]);
      qa[ks][1] = pk(a1[0], a1[1]);
      qa[ks][2] = pk(a0[2], a0[3]);
      qa[ks][3] = pk(a1[2], a1[3]);
      ql[ks][0] = pk(lo(a0[0]), lo(a0[1]));
      ql[ks][1] = pk(lo(a1[0]), lo(a1[1]));
      ql[ks][2] = pk(lo(a0[2]), lo(a0[3]));
      ql[ks][3] = pk(lo(a1[2]), lo(a1[3]));
    }
  }

  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

  uint8_t *wsm = smem + warp * kStages * kSB;
  const uint32_t wsm_u = smem_u32(wsm);
  const int n_tiles = c0 < c1 ? (c1 - c0 + kTileKeys - 1) / kTileKeys : 0;
  // tiles of this warp: warp, warp + kWarps, ...
  // pool slot of key `lane` of this warp's tile it (0 past the end); loaded
  // one tile ahead of its use, so the gather never waits on the index load
  auto load_slot = [&](int it) {
    const int k = c0 + (warp + it * kWarps) * kTileKeys + lane;
    return lane < kTileKeys && k < c1 ? __ldg(indices + beg + k) : 0;
  };
  auto issue = [&](int it, int slot) {
    const int tile = warp + it * kWarps;
    const int stage = it % kStages;
    if (tile < n_tiles) {
      const int k0 = c0 + tile * kTileKeys;
      const bool have = lane < kTileKeys && k0 + lane < c1;
      if (kRope && lane < kTileKeys)  // the tile's positions (0 past the end)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(
                         wsm_u + stage * kSB + 4096 + 4 * lane),
                     "l"(kvpos + beg + (have ? k0 + lane : 0)), "r"(have ? 4 : 0));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = lane + 32 * i;  // 128 chunks per tile: key = idx/8, chunk = idx%8
        const int key = idx >> 3, ch = idx & 7;
        const int s = __shfl_sync(0xffffffffu, slot, key);
        const bool valid = k0 + key < c1;
        const int64_t off = ((int64_t)s * Hkv + g) * kD + ch * 8;
        cp_async16(wsm_u + stage * kSB + swz(key, ch), kp + off, valid);
        cp_async16(wsm_u + stage * kSB + 2048 + swz(key, ch), vp + off, valid);
      }
    }
    asm volatile("cp.async.commit_group;\n" ::);
  };

  const int my_tiles = n_tiles > warp ? (n_tiles - warp + kWarps - 1) / kWarps : 0;
  int slot_nx = load_slot(0);
#pragma unroll
  for (int it = 0; it < kStages - 1; ++it) {
    const int sl = slot_nx;
    slot_nx = load_slot(it + 1);
    issue(it, sl);
  }
  for (int it = 0; it < my_tiles; ++it) {
    const int sl = slot_nx;
    slot_nx = load_slot(it + kStages);
    issue(it + kStages - 1, sl);
    asm volatile("cp.async.wait_group %0;\n" ::"n"(kStages - 1));
    __syncwarp();
    const uint32_t kt = wsm_u + (it % kStages) * kSB, vt = kt + 2048;
    const int k0 = c0 + (warp + it * kWarps) * kTileKeys;
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (kRope) {
      const int32_t *tpos = reinterpret_cast<const int32_t *>(wsm + (it % kStages) * kSB + 4096);
      const int pa = tpos[gid], pb = tpos[gid + 8];
      // cos/sin(p0 theta_lane) at the tile's first position
      const int p0 = tpos[0];
      float cb, sb;
      if (p0 < -262144 || p0 > 262144) rope_cs(th.th[lane], (double)p0, &cb, &sb);
      else rope_cs_fast(ts.hi[lane], ts.lo[lane], p0, &cb, &sb);
      // the base angles of this lane's frequencies f = 16ks + 8h + 2tig and f + 1
      float bc[2][2][2], bs[2][2][2];  // [ks][h][f or f + 1]
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int f = ks * 16 + 8 * h + 2 * tig + e;
            bc[ks][h][e] = __shfl_sync(0xffffffffu, cb, f);
            bs[ks][h][e] = __shfl_sync(0xffffffffu, sb, f);
          }
      uint32_t kb[4][4];
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int mi = lane >> 3;
        const int key = (mi >> 1) * 8 + (lane & 7);
        const int ch = ks * 2 + (mi & 1);
        ldsm_x4(kt + swz(key, ch), kb[ks][0], kb[ks][1], kb[ks][2], kb[ks][3]);
      }
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int r = 0; r < 4; ++r) {  // r: (key half, dim half) = (r >> 1, r & 1)
          const int pos = (r >> 1) ? pb : pa;
          const int f = ks * 16 + 8 * (r & 1) + 2 * tig;
          const float cb0 = bc[ks][r & 1][0], sb0 = bs[ks][r & 1][0];
          const float cb1 = bc[ks][r & 1][1], sb1 = bs[ks][r & 1][1];
          float c0f, s0f, c1f, s1f;
          const unsigned delta = (unsigned)pos - (unsigned)p0;  // wraps when pos < p0
          if (delta < (unsigned)kDeltas) {
            const float4 t = dtab[delta * kDeltaRow + (f >> 1)];
            c0f = cb0 * t.x - sb0 * t.y;
            s0f = sb0 * t.x + cb0 * t.y;
            c1f = cb1 * t.z - sb1 * t.w;
            s1f = sb1 * t.z + cb1 * t.w;
          } else {
            const float4 d = rope_cs_direct2(ts, thd, f, pos);
            c0f = d.x;
            s0f = d.y;
            c1f = d.z;
            s1f = d.w;
          }
          __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&kb[ks][r]);
          __nv_bfloat162 bq = *reinterpret_cast<__nv_bfloat162 *>(&kb[ks + 2][r]);
          const float x1a = __low2float(a), x1b = __high2float(a);
          const float x2a = __low2float(bq), x2b = __high2float(bq);
          const float y1a = x1a * c0f - x2a * s0f, y1b = x1b * c1f - x2b * s1f;
          const float y2a = x1a * s0f + x2a * c0f, y2b = x1b * s1f + x2b * c1f;
          kb[ks][r] = pack_f16(y1a, y1b);
          kb[ks + 2][r] = pack_f16(y2a, y2b);
        }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_f16(s[0], qa[ks], kb[ks][0], kb[ks][1]);
        mma_f16(s[1], qa[ks], kb[ks][2], kb[ks][3]);
        mma_f16(s[0], ql[ks], kb[ks][0], kb[ks][1]);
        mma_f16(s[1], ql[ks], kb[ks][2], kb[ks][3]);
      }
    }
    // S = Q K^T: two n-blocks of 8 keys
#pragma unroll
    for (int ks = 0; ks < 4 && !kRope; ++ks) {
      // matrices: (keys 0-7, d lo), (keys 0-7, d hi), (keys 8-15, d lo), (keys 8-15, d hi)
      const int mi = lane >> 3;
      const int key = (mi >> 1) * 8 + (lane & 7);
      const int ch = ks * 2 + (mi & 1);
      uint32_t b00, b01, b10, b11;
      ldsm_x4(kt + swz(key, ch), b00, b01, b10, b11);
      mma_bf16(s[0], qa[ks], b00, b01);
      mma_bf16(s[1], qa[ks], b10, b11);
      mma_bf16(s[0], ql[ks], b00, b01);
      mma_bf16(s[1], ql[ks], b10, b11);
    }
    // mask the ragged tail; online softmax in log2 units
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = k0 + nb * 8 + 2 * tig + (e & 1);
        if (key >= c1) s[nb][e] = -INFINITY;
        mx[e >> 1] = fmaxf(mx[e >> 1], s[nb][e]);
      }
    float alpha[2], mref[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mn = fmaxf(m[r], mx[r]);
      mref[r] = mn == -INFINITY ? 0.f : mn;
      alpha[r] = exp2f(m[r] - mref[r]);
      m[r] = mn;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[nb][e] = exp2f(s[nb][e] - mref[e >> 1]);
        rs[e >> 1] += s[nb][e];
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) l[r] = l[r] * alpha[r] + rs[r];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }
    // O += P V: P from the S accumulators (keys as k), V through ldmatrix.trans
    uint32_t pa[4];
    pa[0] = pack_bf16(s[0][0], s[0][1]);
    pa[1] = pack_bf16(s[0][2], s[0][3]);
    pa[2] = pack_bf16(s[1][0], s[1][1]);
    pa[3] = pack_bf16(s[1][2], s[1][3]);
#pragma unroll
    for (int nb2 = 0; nb2 < 4; ++nb2) {
      // matrices: (keys 0-7, d 16nb2..+7), (keys 8-15, same), (keys 0-7, d +8), (keys 8-15, d +8)
      const int mi = lane >> 3;
      const int key = (mi & 1) * 8 + (lane & 7);
      const int ch = nb2 * 2 + (mi >> 1);
      uint32_t v0, v1, v2, v3;
      ldsm_x4_t(vt + swz(key, ch), v0, v1, v2, v3);
      mma_bf16(o[2 * nb2], pa, v0, v1);
      mma_bf16(o[2 * nb2 + 1], pa, v2, v3);
    }
    __syncwarp();
  }
  asm volatile("cp.async.wait_group 0;\n" ::);
  __syncthreads();

  // row sums over the quad
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
  // merge the warps: smem [warp][16 rows][kD] + m, l
  float *mo = reinterpret_cast<float *>(smem);           // kWarps*16*64 floats = 16 KiB
  float *mm = mo + kWarps * 16 * kD;                      // kWarps*16
  float *ml = mm + kWarps * 16;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int row = gid + 8 * (e >> 1), col = i * 8 + 2 * tig + (e & 1);
      mo[(warp * 16 + row) * kD + col] = o[i][e];
    }
  if (tig == 0) {
    mm[warp * 16 + gid] = m[0];
    mm[warp * 16 + gid + 8] = m[1];
    ml[warp * 16 + gid] = l[0];
    ml[warp * 16 + gid + 8] = l[1];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < grp * kD; idx += kWarps * 32) {
    const int row = idx / kD, col = idx % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * 16 + row]);
    const float Mr = M == -INFINITY ? 0.f : M;
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = exp2f(mm[w * 16 + row] - Mr);
      L += ml[w * 16 + row] * f;
      acc += mo[(w * 16 + row) * kD + col] * f;
    }
    const int h = g * grp + row;
    const int64_t pi = ((int64_t)b * Hq + h) * ns + split;
    part.o[pi * kD + col] = acc;
    if (col == 0) {
      part.ml[2 * pi] = M;
      part.ml[2 * pi + 1] = L;
    }
  }
  // the last CTA of (request, KV head) to finish merges the splits
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  const int used = min(ns, (n + chunk - 1) / chunk);
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(counters + (int64_t)b * Hkv + g, 1);
    is_last = prev == used - 1;
    if (is_last) counters[(int64_t)b * Hkv + g] = 0;  // ready for the next call
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // merge: per query head (row) the split weights 2^(m_s - M) / L go to
  // shared memory (reusing the tile buffers), then every output element is
  // a weighted sum over the splits with all its loads in flight.
  float *wgt = reinterpret_cast<float *>(smem);  // [16 rows][used]
  float *rowl = wgt + 16 * used;                 // [16]
  for (int i = threadIdx.x; i < grp * used; i += kWarps * 32) {
    const int row = i / used, sp = i % used;
    wgt[row * used + sp] = __ldcg(part.ml + 2 * (((int64_t)b * Hq + g * grp + row) * ns + sp));
  }
  __syncthreads();
  if (threadIdx.x < grp) {
    const int row = threadIdx.x;
    float M = -INFINITY;
    for (int sp = 0; sp < used; ++sp) M = fmaxf(M, wgt[row * used + sp]);
    const float Mr = M == -INFINITY ? 0.f : M;
    float L = 0.f;
    for (int sp = 0; sp < used; ++sp) {
      const float f = exp2f(wgt[row * used + sp] - Mr);
      L += __ldcg(part.ml + 2 * (((int64_t)b * Hq + g * grp + row) * ns + sp) + 1) * f;
      wgt[row * used + sp] = f;
    }
    rowl[row] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < grp * kD; idx += kWarps * 32) {
    const int row = idx / kD, col = idx % kD;
    const float *po = part.o + ((int64_t)b * Hq + g * grp + row) * ns * kD + col;
    const float *w = wgt + row * used;
    float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
    int sp = 0;
    for (; sp + 4 <= used; sp += 4) {
      x0 += __ldcg(po + (int64_t)sp * kD) * w[sp];
      x1 += __ldcg(po + (int64_t)(sp + 1) * kD) * w[sp + 1];
      x2 += __ldcg(po + (int64_t)(sp + 2) * kD) * w[sp + 2];
      x3 += __ldcg(po + (int64_t)(sp + 3) * kD) * w[sp + 3];
    }
    for (; sp < used; ++sp) x0 += __ldcg(po + (int64_t)sp * kD) * w[sp];
    out[((int64_t)b * Hq + g * grp + row) * kD + col] =
        __float2bfloat16_rn(((x0 + x1) + (x2 + x3)) * rowl[row]);
  }
}

// ---------------------------------------------------------------------------
// bf16 decode, all KV heads of a key chunk in one CTA (2, 4, 8 or 16 KV
// heads; rotation on read with 4, 8 or 16).
// A CTA takes (key chunk, request) with one warp per KV head (kHkv warps),
// so the CTA reads a key's whole K and V rows.  Per head the work is the
// per-head kernel's: 16-key tiles gathered by cp.async, the query split
// into hi + lo parts, S in m16n8k16 MMAs, online softmax, P.V in bf16.
// kRope (rotation on read): a key's rotation needs cos/sin of (position x
// frequency), the same for every KV head, so the CTA fills, one tile ahead,
// a shared table of the 16 x 32 cos/sin pairs of each 16-key tile, which
// every head's warp then reads.  A thread's share of the next table is
// computed into registers in the middle of the current tile's arithmetic
// and stored after it, so the sin/cos latency overlaps that work; one
// barrier per tile publishes the table and frees the previous one.  Keys
// are rotated in fp32 (packed over frequency pairs) and rounded to fp16;
// the query parts and the score MMAs are fp16.  Without kRope (pre-rotated
// pool) the warps run independently: bf16 query parts and score MMAs, no
// table, no barrier in the loop.
// Each CTA leaves its chunk's partial (m, l, o) per query head and a
// second launch merges them (decode_merge_heads_kernel).  Merged in this
// kernel by the last CTA of a request, each request's merge (all its query
// heads over all its chunks) ran in one CTA at the end of the launch and
// made the rotate-on-read step 12 % slower.
// ---------------------------------------------------------------------------
// K/V tiles per warp (the one in use and those in flight): rotation on read
// (issue-bound; a third stage measured no faster) and pre-rotated pools
// (gather-bound; the third stage is 1.6 % faster)
constexpr int kHStages = 2;
constexpr int kHStagesPre = 3;
// table row of one key: 32 (cos, sin) pairs padded to 40 so that the two
// keys read by one 8-lane phase of a 16-byte load fall in different banks
constexpr int kTabRow = kD / 2 + 8;
constexpr int kTabBytes = kTileKeys * kTabRow * 8;  // one tile's cos/sin table
constexpr int kHeadsWaves = 8;  // CTA waves aimed for when choosing the chunk

// cos/sin of pos * theta_f beyond 2^18 (the double path); rare, so out of line
__device__ __noinline__ float2 rope_cs_wide(double theta, int pos) {
  float2 r;
  rope_cs(theta, (double)pos, &r.x, &r.y);
  return r;
}

template <int kHkv, bool kRope>
__global__ void __launch_bounds__(kHkv * 32, kHkv == 16 ? 1 : kHkv == 8 ? 2 : kHkv == 4 ? 3 : 8)
    decode_heads_kernel(int Hq, const __nv_bfloat16 *__restrict__ q,
                        const int32_t *__restrict__ qpos, __nv_bfloat16 *kp, __nv_bfloat16 *vp,
                        const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                        Partials part, RopeTheta th, __nv_bfloat16 *out,
                        const __nv_bfloat16 *k_new, const __nv_bfloat16 *v_new,
                        const int32_t *new_slot, int chunk, const int32_t *__restrict__ kvpos) {
  constexpr int kThreads = kHkv * 32;
  // the angle table is filled by the first kTabThreads threads (at most 256,
  // so that a thread computes at least two frequencies: one float4 entry)
  constexpr int kTabThreads = kThreads < 256 ? kThreads : 256;
  constexpr int kTpk = kTabThreads / kTileKeys;  // table: threads per key
  constexpr int kFpt = (kD / 2) / kTpk;          // table: frequencies per thread (2, 4 or 8)
  constexpr int kNc4 = kFpt / 2;                 // their float4 entries
  const bool tab_thread = threadIdx.x < kTabThreads;
  constexpr int kSt = kRope ? kHStages : kHStagesPre;
  constexpr int kSB = 4096;                   // one stage: K tile 2 KiB | V tile 2 KiB
  // dynamic smem: [warp][kSt][stage], then (kRope) two cos/sin tables
  // [16 keys][kTabRow] float2
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float cs[kD / 2], sn[kD / 2];
  __shared__ ThetaSmem ts;
  __shared__ double thd[kD / 2];
  const int split = blockIdx.x, b = blockIdx.y;
  const int ns = gridDim.x;
  const int grp = Hq / kHkv;
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;  // warp = KV head
  const int gid = lane >> 2, tig = lane & 3;
  // the merge launch may be placed once every CTA of this grid has started
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
  const int beg = indptr[b], n = indptr[b + 1] - beg;
  const int c0 = split * chunk, c1 = min(n, c0 + chunk);
  if (c0 >= n) {  // the merge reads only the splits that hold keys
    if (n <= 0 && split == 0)  // a request with no keys gets zeros
      for (int i = threadIdx.x; i < Hq * kD; i += kThreads)
        out[(int64_t)b * Hq * kD + i] = __float2bfloat16_rn(0.f);
    return;
  }
  float2 *tabs = reinterpret_cast<float2 *>(smem + kHkv * kSt * kSB);
  const int nk = c1 - c0;
  const int n_tiles = (nk + kTileKeys - 1) / kTileKeys;
  // this thread's table entries: key tkey of the tile, frequencies tf..tf+kFpt-1
  const int tkey = threadIdx.x / kTpk, tf = (threadIdx.x % kTpk) * kFpt;
  auto load_pos = [&](int t) {
    const int k = t * kTileKeys + tkey;
    return t < n_tiles && k < nk ? __ldg(kvpos + beg + c0 + k) : 0;
  };
  auto angles = [&](int pos, float4 *cs4) {
    const bool wide = pos < -262144 || pos > 262144;
#pragma unroll
    for (int j = 0; j < kFpt / 2; ++j) {
      const int f = tf + 2 * j;
      // (cos f, cos f+1, sin f, sin f+1): the rotation's packed operands
      if (wide) {
        const float2 a = rope_cs_wide(thd[f], pos), c = rope_cs_wide(thd[f + 1], pos);
        cs4[j] = make_float4(a.x, c.x, a.y, c.y);
      } else {
        rope_cs_fast(ts.hi[f], ts.lo[f], pos, &cs4[j].x, &cs4[j].z);
        rope_cs_fast(ts.hi[f + 1], ts.lo[f + 1], pos, &cs4[j].y, &cs4[j].w);
      }
    }
  };
  auto store_tab = [&](int t, const float4 *cs4) {
    float4 *row = reinterpret_cast<float4 *>(tabs + (t & 1) * (kTileKeys * kTabRow) +
                                             tkey * kTabRow + tf);
#pragma unroll
    for (int j = 0; j < kFpt / 2; ++j) row[j] = cs4[j];
  };
  // positions of the next tiles' table keys, loaded three tiles ahead
  int pos1 = 0, pos2 = 0, pos3 = 0, pos0 = 0;
  if (kRope) {
    pos1 = load_pos(1);
    pos2 = load_pos(2);
    pos3 = load_pos(3);
    pos0 = load_pos(0);
  }

  if (threadIdx.x < kD / 2) {
    rope_cs_lane(th, threadIdx.x, qpos[b], &cs[threadIdx.x], &sn[threadIdx.x]);
    if (kRope) thd[threadIdx.x] = th.th[threadIdx.x];
  }
  if (kRope) stage_theta(th, ts);
  if (new_slot && c1 == n) {  // fused append of the step's token
    const int64_t src = ((int64_t)b * kHkv + g) * kD, dst = ((int64_t)new_slot[b] * kHkv + g) * kD;
    if (kRope) {  // the pool keeps raw keys: a copy
      if (lane < kD / 8)
        reinterpret_cast<uint4 *>(kp + dst)[lane] = reinterpret_cast<const uint4 *>(k_new + src)[lane];
      else if (lane < kD / 4)
        reinterpret_cast<uint4 *>(vp + dst)[lane - kD / 8] =
            reinterpret_cast<const uint4 *>(v_new + src)[lane - kD / 8];
    } else {  // the key rotated at the query position (cos/sin above)
      __syncthreads();
      const int f = lane;
      const float x1 = __bfloat162float(k_new[src + f]), x2 = __bfloat162float(k_new[src + f + kD / 2]);
      kp[dst + f] = __float2bfloat16_rn(x1 * cs[f] - x2 * sn[f]);
      kp[dst + f + kD / 2] = __float2bfloat16_rn(x1 * sn[f] + x2 * cs[f]);
      if (lane < kD / 8)
        reinterpret_cast<uint4 *>(vp + dst)[lane] = reinterpret_cast<const uint4 *>(v_new + src)[lane];
    }
  }
  __syncthreads();  // frequencies staged, the appended row visible
  if (kRope) {
    float4 c4[kNc4];
    if (tab_thread) {
      angles(pos0, c4);
      store_tab(0, c4);
    }
  }

  uint8_t *wsm = smem + g * kSt * kSB;
  const uint32_t wsm_u = smem_u32(wsm);
  // pool slot of key `lane` of tile t (0 past the end), loaded one tile
  // ahead of its use
  auto load_slot = [&](int t) {
    const int k = t * kTileKeys + lane;
    return lane < kTileKeys && k < nk ? __ldg(indices + beg + c0 + k) : 0;
  };
  auto issue = [&](int t, int slot) {
    const int stage = t % kSt;
    if (t < n_tiles) {
      const int k0 = t * kTileKeys;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = lane + 32 * i;  // 128 chunks per tile: key = idx/8, chunk = idx%8
        const int key = idx >> 3, ch = idx & 7;
        const int sl = __shfl_sync(0xffffffffu, slot, key);
        const bool valid = k0 + key < nk;
        const int64_t off = ((int64_t)sl * kHkv + g) * kD + ch * 8;
        cp_async16(wsm_u + stage * kSB + swz(key, ch), kp + off, valid);
        cp_async16(wsm_u + stage * kSB + 2048 + swz(key, ch), vp + off, valid);
      }
    }
    asm volatile("cp.async.commit_group;\n" ::);
  };
  int slot_nx = load_slot(0);
#pragma unroll
  for (int t = 0; t < kSt - 1; ++t) {
    const int sl = slot_nx;
    slot_nx = load_slot(t + 1);
    issue(t, sl);
  }

  // Q fragments of this warp's head group (rows = its query heads, 16 rows
  // padded with zeros), rotated at the query position, 1/sqrt(D) * log2(e)
  // folded in, split into hi + lo parts: fp16 with rotation on read (the
  // score product takes fp16 keys), else bf16
  uint32_t qa[4][4], ql[4][4];
  {
    const float qsc = 0.125f * kLog2e;
    float qv[2][16];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = gid + 8 * hh;
      const bool ok = row < grp;
      const __nv_bfloat16 *qrow = q + ((int64_t)b * Hq + g * grp + (ok ? row : 0)) * kD;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = ks * 16 + 2 * tig + (e & 1) + (e >> 1) * 8;
          qv[hh][ks * 4 + e] = ok ? __bfloat162float(qrow[d]) : 0.f;
        }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = ks * 16 + 2 * tig + (e & 1) + (e >> 1) * 8;
          const float x1 = qv[hh][ks * 4 + e], x2 = qv[hh][(ks + 2) * 4 + e];
          qv[hh][ks * 4 + e] = (x1 * cs[d] - x2 * sn[d]) * qsc;
          qv[hh][(ks + 2) * 4 + e] = (x1 * sn[d] + x2 * cs[d]) * qsc;
        }
    auto pk = [](float x, float y) { return kRope ? pack_f16(x, y) : pack_bf16(x, y); };
    auto lo = [](float x) {
      return kRope ? x - __half2float(__float2half_rn(x))
                   : x - __bfloat162float(__float2bfloat16_rn(x));
    };
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const float *a0 = &qv[0][ks * 4], *a1 = &qv[1][ks * 4];
      qa[ks][0] = pk(a0[0], a0[1]);
      qa[ks][1] = pk(a1[0], a1[1]);
      qa[ks][2] = pk(a0[2], a0[3]);
      qa[ks][3] = pk(a1[2], a1[3]);
      ql[ks][0] = pk(lo(a0[0]), lo(a0[1]));
      ql[ks][1] = pk(lo(a1[0]), lo(a1[1]));
      ql[ks][2] = pk(lo(a0[2]), lo(a0[3]));
      ql[ks][3] = pk(lo(a1[2]), lo(a1[3]));
    }
  }

  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  if (kRope) __syncthreads();  // table 0 complete

  for (int it = 0; it < n_tiles; ++it) {
    const int sl = slot_nx;
    slot_nx = load_slot(it + kSt);
    issue(it + kSt - 1, sl);
    asm volatile("cp.async.wait_group %0;\n" ::"n"(kSt - 1));
    __syncwarp();
    const float2 *tab = tabs + (it & 1) * (kTileKeys * kTabRow);
    const uint32_t kt = wsm_u + (it % kSt) * kSB, vt = kt + 2048;
    const int k0 = it * kTileKeys;
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      uint32_t kb[4][4];
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const int mi = lane >> 3;
        const int key = (mi >> 1) * 8 + (lane & 7);
        const int ch = ks * 2 + (mi & 1);
        ldsm_x4(kt + swz(key, ch), kb[ks][0], kb[ks][1], kb[ks][2], kb[ks][3]);
      }
      // rotate: the pair (d, d + 32) of keys gid and gid + 8 sits in k-steps
      // ks and ks + 2 of this lane; frequencies f = 16ks + 8h + 2tig, f + 1
#pragma unroll
      for (int ks = 0; ks < 2 && kRope; ++ks)
#pragma unroll
        for (int r = 0; r < 4; ++r) {  // r: (key half, dim half) = (r >> 1, r & 1)
          const int key = gid + 8 * (r >> 1);
          const int f = ks * 16 + 8 * (r & 1) + 2 * tig;
          // packed over the pair (f, f + 1): y1 = x1 c - x2 s, y2 = x1 s + x2 c
          const float4 t = *reinterpret_cast<const float4 *>(tab + key * kTabRow + f);
          const float2 c = make_float2(t.x, t.y), sn2 = make_float2(t.z, t.w);
          const float2 nsn = make_float2(-t.z, -t.w);
          const uint32_t ua = kb[ks][r], ub = kb[ks + 2][r];  // bf16 pairs (f, f + 1)
          const float2 x1 = make_float2(__uint_as_float(ua << 16), __uint_as_float(ua & 0xffff0000u));
          const float2 x2 = make_float2(__uint_as_float(ub << 16), __uint_as_float(ub & 0xffff0000u));
          const float2 y1 = __ffma2_rn(x1, c, __fmul2_rn(x2, nsn));
          const float2 y2 = __ffma2_rn(x1, sn2, __fmul2_rn(x2, c));
          kb[ks][r] = pack_f16(y1.x, y1.y);
          kb[ks + 2][r] = pack_f16(y2.x, y2.y);
        }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        if (kRope) {
          mma_f16(s[0], qa[ks], kb[ks][0], kb[ks][1]);
          mma_f16(s[1], qa[ks], kb[ks][2], kb[ks][3]);
          mma_f16(s[0], ql[ks], kb[ks][0], kb[ks][1]);
          mma_f16(s[1], ql[ks], kb[ks][2], kb[ks][3]);
        } else {
          mma_bf16(s[0], qa[ks], kb[ks][0], kb[ks][1]);
          mma_bf16(s[1], qa[ks], kb[ks][2], kb[ks][3]);
          mma_bf16(s[0], ql[ks], kb[ks][0], kb[ks][1]);
          mma_bf16(s[1], ql[ks], kb[ks][2], kb[ks][3]);
        }
      }
    }
    // the next tile's angles (stored after this tile's arithmetic)
    float4 nxt[kNc4];
    if (kRope) {
      if (tab_thread) angles(pos1, nxt);
      pos1 = pos2;
      pos2 = pos3;
      pos3 = load_pos(it + 4);
    }
    // mask the ragged tail; online softmax in log2 units
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = k0 + nb * 8 + 2 * tig + (e & 1);
        if (key >= nk) s[nb][e] = -INFINITY;
        mx[e >> 1] = fmaxf(mx[e >> 1], s[nb][e]);
      }
    float alpha[2], mref[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mn = fmaxf(m[r], mx[r]);
      mref[r] = mn == -INFINITY ? 0.f : mn;
      alpha[r] = exp2f(m[r] - mref[r]);
      m[r] = mn;
    }
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int nb = 0; nb < 2; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[nb][e] = exp2f(s[nb][e] - mref[e >> 1]);
        rs[e >> 1] += s[nb][e];
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) l[r] = l[r] * alpha[r] + rs[r];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }
    // O += P V: P from the S accumulators (keys as k), V through ldmatrix.trans
    uint32_t pa[4];
    pa[0] = pack_bf16(s[0][0], s[0][1]);
    pa[1] = pack_bf16(s[0][2], s[0][3]);
    pa[2] = pack_bf16(s[1][0], s[1][1]);
    pa[3] = pack_bf16(s[1][2], s[1][3]);
#pragma unroll
    for (int nb2 = 0; nb2 < 4; ++nb2) {
      const int mi = lane >> 3;
      const int key = (mi & 1) * 8 + (lane & 7);
      const int ch = nb2 * 2 + (mi >> 1);
      uint32_t v0, v1, v2, v3;
      ldsm_x4_t(vt + swz(key, ch), v0, v1, v2, v3);
      mma_bf16(o[2 * nb2], pa, v0, v1);
      mma_bf16(o[2 * nb2 + 1], pa, v2, v3);
    }
    // publish the next table; every warp is done with this one (its buffer
    // is the one the following iteration fills)
    if (kRope) {
      if (tab_thread && it + 1 < n_tiles) store_tab(it + 1, nxt);
      __syncthreads();
    } else {
      __syncwarp();
    }
  }
  asm volatile("cp.async.wait_group 0;\n" ::);

  // this warp's split partial: rows gid and gid + 8 (query heads of its
  // group), columns 8i + 2tig (+1)
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
  }
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int row = gid + 8 * hh;
    if (row < grp) {
      const int64_t pi = ((int64_t)b * Hq + g * grp + row) * ns + split;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        *reinterpret_cast<float2 *>(part.o + pi * kD + i * 8 + 2 * tig) =
            make_float2(o[i][2 * hh], o[i][2 * hh + 1]);
      if (tig == 0) {
        part.ml[2 * pi] = m[hh];
        part.ml[2 * pi + 1] = l[hh];
      }
    }
  }
}

// Merge of the chunk partials of decode_heads_kernel: a CTA per (query
// head, request).  One warp folds the chunks' (m, l) pairs into (M, L) with
// a running maximum (each chunk's m kept in shared memory), then every
// thread turns the m into weights 2^(m_s - M), and 16 groups of 16 threads
// each sum every 16th chunk's output row (4 columns per thread); the
// groups' sums are added in shared memory.  A request with no keys gets
// zeros.  Launched as a programmatic dependent of the attention kernel: its
// CTAs are placed while the last attention CTAs run and wait (griddepcontrol
// .wait) until that grid has finished and its partials are visible.
__global__ void __launch_bounds__(256) decode_merge_heads_kernel(int Hq, int ns, int chunk,
                                                                 const int32_t *indptr,
                                                                 Partials part,
                                                                 __nv_bfloat16 *out) {
  const int h = blockIdx.x, b = blockIdx.y;
  const int n = indptr[b + 1] - indptr[b];
  const int used = n <= 0 ? 0 : min(ns, (n + chunk - 1) / chunk);
  const int64_t base = ((int64_t)b * Hq + h) * ns;
  __shared__ float wsm[kMaxSplits];
  __shared__ float4 red[16][kD / 4];
  __shared__ float mrow, rl;
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float M = -INFINITY, L = 0.f;
    for (int s = lane; s < used; s += 32) {
      const float2 ml = __ldcg(reinterpret_cast<const float2 *>(part.ml) + base + s);
      wsm[s] = ml.x;
      if (ml.x > M) {
        L = L * exp2f(M - ml.x) + ml.y;
        M = ml.x;
      } else if (ml.x > -INFINITY) {
        L += ml.y * exp2f(ml.x - M);
      }
    }
    for (int o = 16; o; o >>= 1) {
      const float M2 = __shfl_xor_sync(0xffffffffu, M, o), L2 = __shfl_xor_sync(0xffffffffu, L, o);
      const float Mn = fmaxf(M, M2);
      L = (M == -INFINITY ? 0.f : L * exp2f(M - Mn)) + (M2 == -INFINITY ? 0.f : L2 * exp2f(M2 - Mn));
      M = Mn;
    }
    if (lane == 0) {
      mrow = M == -INFINITY ? 0.f : M;
      rl = L > 0.f ? 1.f / L : 0.f;
    }
  }
  __syncthreads();
  for (int s = threadIdx.x; s < used; s += blockDim.x) wsm[s] = exp2f(wsm[s] - mrow);
  __syncthreads();
  const int cg = threadIdx.x & 15, sg = threadIdx.x >> 4;  // 4-column group, chunk group
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = sg; s < used; s += 16) {
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(part.o + (base + s) * kD) + cg);
    const float w = wsm[s];
    acc.x += v.x * w;
    acc.y += v.y * w;
    acc.z += v.z * w;
    acc.w += v.w * w;
  }
  red[sg][cg] = acc;
  __syncthreads();
  if (threadIdx.x < kD) {
    const int col = threadIdx.x;
    float x = 0.f;
    for (int j = 0; j < 16; ++j) x += reinterpret_cast<const float *>(&red[j][col >> 2])[col & 3];
    out[((int64_t)b * Hq + h) * kD + col] = __float2bfloat16_rn(x * rl);
  }
}

// fp32: thread per key, block of 128 threads per (split, query head, request)
__global__ void __launch_bounds__(128)
    decode_f32_kernel(int Hq, int Hkv, const float *__restrict__ q, const int32_t *__restrict__ qpos,
                      const float *__restrict__ kp, const float *__restrict__ vp,
                      const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                      Partials part, RopeTheta th) {
  __shared__ float qs[kD];
  __shared__ float red_m[4], red_l[4];
  __shared__ float red_o[4][kD];
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int ns = gridDim.x, g = h / (Hq / Hkv);
  const int beg = indptr[b], n = indptr[b + 1] - beg;
  const int c0 = split * kChunk, c1 = min(n, c0 + kChunk);
  if (c0 >= n) return;
  if (threadIdx.x < kD / 2) {
    float c, s;
    rope_cs_lane(th, threadIdx.x, qpos[b], &c, &s);
    const float *qr = q + ((int64_t)b * Hq + h) * kD;
    const float x1 = qr[threadIdx.x], x2 = qr[threadIdx.x + kD / 2];
    qs[threadIdx.x] = (x1 * c - x2 * s) * 0.125f * kLog2e;
    qs[threadIdx.x + kD / 2] = (x1 * s + x2 * c) * 0.125f * kLog2e;
  }
  __syncthreads();
  float m = -INFINITY, l = 0.f, acc[kD];
#pragma unroll
  for (int d = 0; d < kD; ++d) acc[d] = 0.f;
  for (int k = c0 + threadIdx.x; k < c1; k += 128) {
    const int64_t row = ((int64_t)__ldg(indices + beg + k) * Hkv + g) * kD;
    float sc = 0.f;
#pragma unroll
    for (int d = 0; d < kD; ++d) sc = fmaf(qs[d], __ldg(kp + row + d), sc);
    const float mn = fmaxf(m, sc);
    const float a = exp2f(m - mn), e = exp2f(sc - mn);
    l = l * a + e;
#pragma unroll
    for (int d = 0; d < kD; ++d) acc[d] = fmaf(acc[d], a, e * __ldg(vp + row + d));
    m = mn;
  }
  // block merge
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float M = m;
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float f = m == -INFINITY ? 0.f : exp2f(m - M);
  float L = l * f;
#pragma unroll
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
#pragma unroll
  for (int d = 0; d < kD; ++d) {
    float x = acc[d] * f;
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red_o[warp][d] = x;
  }
  if (lane == 0) {
    red_m[warp] = M;
    red_l[warp] = L;
  }
  __syncthreads();
  if (threadIdx.x < kD) {
    float MM = -INFINITY;
    for (int w = 0; w < 4; ++w) MM = fmaxf(MM, red_m[w]);
    const float Mr = MM == -INFINITY ? 0.f : MM;
    float LL = 0.f, x = 0.f;
    for (int w = 0; w < 4; ++w) {
      const float ff = exp2f(red_m[w] - Mr);
      LL += red_l[w] * ff;
      x += red_o[w][threadIdx.x] * ff;
    }
    const int64_t pi = ((int64_t)b * Hq + h) * ns + split;
    part.o[pi * kD + threadIdx.x] = x;
    if (threadIdx.x == 0) {
      part.ml[2 * pi] = MM;
      part.ml[2 * pi + 1] = LL;
    }
  }
}

// ---------------------------------------------------------------------------
// Decode with rotation on read.  The pool holds keys before RoPE and every
// index entry carries its position, so a repos only rewrites the positions
// (4 bytes per entry) instead of moving and re-rotating the keys.  The step's
// append is fused: the new raw K/V rows are copied into the pool before the
// keys are read.  bf16 runs decode_bf16_kernel<true> (above).
// ---------------------------------------------------------------------------
// fp32 with rotation on read: thread per key, block of 128 threads per
// (split, query head, request).  The new rows are appended by every CTA of
// the last split before it reads (identical values).
__global__ void __launch_bounds__(128)
    decode_rope_f32_kernel(int Hq, int Hkv, const float *__restrict__ q,
                           const int32_t *__restrict__ qpos, const float *k_new,
                           const float *v_new, const int32_t *new_slot, float *kp, float *vp,
                           const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                           const int32_t *__restrict__ kvpos, Partials part, RopeTheta th) {
  __shared__ float qs[kD];
  __shared__ float red_m[4], red_l[4];
  __shared__ float red_o[4][kD];
  __shared__ ThetaSmem ts;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int ns = gridDim.x, g = h / (Hq / Hkv);
  const int beg = indptr[b], n = indptr[b + 1] - beg;
  const int c0 = split * kRChunk, c1 = min(n, c0 + kRChunk);
  if (c0 >= n) return;
  stage_theta(th, ts);
  if (new_slot && c1 == n && threadIdx.x < kD) {
    const int64_t slot = new_slot[b];
    kp[(slot * Hkv + g) * kD + threadIdx.x] = k_new[((int64_t)b * Hkv + g) * kD + threadIdx.x];
    vp[(slot * Hkv + g) * kD + threadIdx.x] = v_new[((int64_t)b * Hkv + g) * kD + threadIdx.x];
  }
  __syncthreads();
  if (threadIdx.x < kD / 2) {
    float c, s;
    rope_cs(th, ts, threadIdx.x, qpos[b], &c, &s);
    const float *qr = q + ((int64_t)b * Hq + h) * kD;
    const float x1 = qr[threadIdx.x], x2 = qr[threadIdx.x + kD / 2];
    qs[threadIdx.x] = (x1 * c - x2 * s) * 0.125f * kLog2e;
    qs[threadIdx.x + kD / 2] = (x1 * s + x2 * c) * 0.125f * kLog2e;
  }
  __syncthreads();
  float m = -INFINITY, l = 0.f, acc[kD];
#pragma unroll
  for (int d = 0; d < kD; ++d) acc[d] = 0.f;
  for (int k = c0 + threadIdx.x; k < c1; k += 128) {
    const int64_t row = ((int64_t)indices[beg + k] * Hkv + g) * kD;
    const int pos = kvpos[beg + k];
    float sc = 0.f;
#pragma unroll 4
    for (int f = 0; f < kD / 2; ++f) {
      float c, sn;
      rope_cs(th, ts, f, pos, &c, &sn);
      const float x1 = kp[row + f], x2 = kp[row + f + kD / 2];
      sc = fmaf(qs[f], x1 * c - x2 * sn, sc);
      sc = fmaf(qs[f + kD / 2], x1 * sn + x2 * c, sc);
    }
    const float mn = fmaxf(m, sc);
    const float a = exp2f(m - mn), e = exp2f(sc - mn);
    l = l * a + e;
#pragma unroll
    for (int d = 0; d < kD; ++d) acc[d] = fmaf(acc[d], a, e * vp[row + d]);
    m = mn;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float M = m;
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float f = m == -INFINITY ? 0.f : exp2f(m - M);
  float L = l * f;
#pragma unroll
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
#pragma unroll
  for (int d = 0; d < kD; ++d) {
    float x = acc[d] * f;
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0) red_o[warp][d] = x;
  }
  if (lane == 0) {
    red_m[warp] = M;
    red_l[warp] = L;
  }
  __syncthreads();
  if (threadIdx.x < kD) {
    float MM = -INFINITY;
    for (int w = 0; w < 4; ++w) MM = fmaxf(MM, red_m[w]);
    const float Mr = MM == -INFINITY ? 0.f : MM;
    float LL = 0.f, x = 0.f;
    for (int w = 0; w < 4; ++w) {
      const float ff = exp2f(red_m[w] - Mr);
      LL += red_l[w] * ff;
      x += red_o[w][threadIdx.x] * ff;
    }
    const int64_t pi = ((int64_t)b * Hq + h) * ns + split;
    part.o[pi * kD + threadIdx.x] = x;
    if (threadIdx.x == 0) {
      part.ml[2 * pi] = MM;
      part.ml[2 * pi + 1] = LL;
    }
  }
}

template <typename T>
__global__ void __launch_bounds__(kD) decode_combine_kernel(int Hq, int ns, int chunk,
                                                            const int32_t *indptr, Partials part,
                                                            T *out) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int n = indptr[b + 1] - indptr[b];
  const int used = n <= 0 ? 0 : min(ns, (n + chunk - 1) / chunk);
  const int64_t base = ((int64_t)b * Hq + h) * ns;
  float M = -INFINITY;
  for (int s = 0; s < used; ++s) M = fmaxf(M, part.ml[2 * (base + s)]);
  const float Mr = M == -INFINITY ? 0.f : M;
  float L = 0.f, x = 0.f;
  for (int s = 0; s < used; ++s) {
    const float f = exp2f(part.ml[2 * (base + s)] - Mr);
    L += part.ml[2 * (base + s) + 1] * f;
    x += part.o[(base + s) * kD + d] * f;
  }
  const float y = L > 0.f ? x / L : 0.f;
  T *o = out + ((int64_t)b * Hq + h) * kD + d;
  if constexpr (sizeof(T) == 4) *o = y;
  else *o = __float2bfloat16_rn(y);
}

}  // namespace

size_t decode_partials_bytes(int B, int Hq, int max_kv, bool rope) {
  const int ns = n_splits(max_kv, rope ? kRChunk : kMinChunk);  // bf16: the most splits
  const size_t ml = ((size_t)B * Hq * ns * 2 * 4 + 255) / 256 * 256;
  const size_t o = ((size_t)B * Hq * ns * kD * 4 + 255) / 256 * 256;
  return ml + o;
}

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int max_kv) {
  return decode_partials_bytes(B, Hq, max_kv) + ((size_t)B * Hkv * 4 + 255) / 256 * 256;
}

size_t decode_rope_workspace_bytes(int dtype, int B, int Hq, int Hkv, int max_kv) {
  // partials for the most splits (chunks of kRChunk keys); bf16 adds the
  // merge counters of the per-head kernel
  if (dtype != AKV_BF16) return decode_partials_bytes(B, Hq, max_kv, true);
  return decode_partials_bytes(B, Hq, max_kv, true) + ((size_t)B * Hkv * 4 + 255) / 256 * 256;
}

namespace {
// bf16 decode over a workspace laid out as partials then merge counters
cudaError_t decode_bf16(int B, int Hq, int Hkv, const void *q, const int32_t *qpos, void *kp,
                        void *vp, const int32_t *indptr, const int32_t *indices, int max_kv,
                        void *out, void *ws, const RopeTheta &th, const void *k_new,
                        const void *v_new, const int32_t *new_slot, cudaStream_t s,
                        const int32_t *kvpos = nullptr) {
  const int sms = device_sms();
  const bool rope = kvpos != nullptr;
  // 4, 8 or 16 KV heads, and 2 over a pre-rotated pool (with rotation on
  // read a 2-warp CTA spreads each tile's angle table over too few threads:
  // 5% slower than the per-head kernel there, and 22% faster without it)
  if (Hkv == 4 || Hkv == 8 || Hkv == 16 || (Hkv == 2 && !rope)) {
    // all KV heads of a chunk in one CTA of Hkv warps (one CTA per SM for 16
    // heads, two for 8, three for 4: shared memory, eight for 2); the chunk
    // is the largest that still gives about kHeadsWaves waves of CTAs when
    // every request is max_kv long; then the merge launch
    const int per_sm = Hkv == 16 ? 1 : Hkv == 8 ? 2 : Hkv == 4 ? 3 : 8;
    int rc = kMaxChunk;
    const int floor = rope ? kRChunk : kMinChunk;  // the workspace holds that many splits
    while (rc > floor && (int64_t)B * n_splits(max_kv, rc) < (int64_t)kHeadsWaves * per_sm * sms)
      rc /= 2;
    while (n_splits(max_kv, rc) > kMaxSplits) rc *= 2;
    const int rns = n_splits(max_kv, rc);
    Partials rpart = partials(ws, B, Hq, max_kv, rc);
    const int rsmem = Hkv * (rope ? kHStages : kHStagesPre) * 4096 + (rope ? 2 * kTabBytes : 0);
    auto kern = rope ? (Hkv == 16  ? decode_heads_kernel<16, true>
                        : Hkv == 8 ? decode_heads_kernel<8, true>
                                   : decode_heads_kernel<4, true>)
                     : (Hkv == 16  ? decode_heads_kernel<16, false>
                        : Hkv == 8 ? decode_heads_kernel<8, false>
                        : Hkv == 4 ? decode_heads_kernel<4, false>
                                   : decode_heads_kernel<2, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, rsmem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(rns, B), Hkv * 32, rsmem, s>>>(
        Hq, (const __nv_bfloat16 *)q, qpos, (__nv_bfloat16 *)kp, (__nv_bfloat16 *)vp, indptr,
        indices, rpart, th, (__nv_bfloat16 *)out, (const __nv_bfloat16 *)k_new,
        (const __nv_bfloat16 *)v_new, new_slot, rc, kvpos);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the merge as a programmatic dependent launch (it waits for this grid)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(Hq, B);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_heads_kernel, Hq, rns, rc, indptr, rpart,
                              (__nv_bfloat16 *)out);
  }
  // other head counts: a CTA per (chunk, KV head, request); the chunk is the
  // largest of 4096, 2048, 1024 keys that still gives about two waves of
  // CTAs (4 per SM) when every request is max_kv long
  int chunk = kMaxChunk;
  while (chunk > kMinChunk && (int64_t)B * n_splits(max_kv, chunk) * Hkv < 2LL * 4 * sms) chunk /= 2;
  while (n_splits(max_kv, chunk) > kMaxSplits) chunk *= 2;
  const int ns = n_splits(max_kv, chunk);
  Partials part = partials(ws, B, Hq, max_kv, chunk);
  int *counters = reinterpret_cast<int *>(
      static_cast<char *>(ws) + decode_partials_bytes(B, Hq, max_kv, rope));
  // dynamic shared memory: the tile buffers, or the merge's per-split
  // weights ([16 rows][ns] floats and 16 row totals) when those are larger
  const int smem = std::max(kWarps * kStages * kStageBytes(rope), (16 * ns + 16) * 4);
  auto kern = rope ? decode_bf16_kernel<true> : decode_bf16_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // the merge counters start at zero (the kernel also leaves them at zero)
  e = cudaMemsetAsync(counters, 0, (size_t)B * Hkv * 4, s);
  if (e != cudaSuccess) return e;
  kern<<<dim3(ns, Hkv, B), kWarps * 32, smem, s>>>(
      Hq, Hkv, (const __nv_bfloat16 *)q, qpos, (__nv_bfloat16 *)kp, (__nv_bfloat16 *)vp, indptr,
      indices, part, th, counters, (__nv_bfloat16 *)out, (const __nv_bfloat16 *)k_new,
      (const __nv_bfloat16 *)v_new, new_slot, chunk, kvpos);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_decode_append(int dtype, int B, int Hq, int Hkv, const void *q,
                                 const int32_t *qpos, const void *k_new, const void *v_new,
                                 const int32_t *new_slot, void *kp, void *vp,
                                 const int32_t *indptr, const int32_t *indices, int max_kv,
                                 void *out, void *ws, const RopeTheta &th, cudaStream_t s) {
  if (dtype == AKV_BF16)
    return decode_bf16(B, Hq, Hkv, q, qpos, kp, vp, indptr, indices, max_kv, out, ws, th, k_new,
                       v_new, new_slot, s);
  cudaError_t e = launch_append(dtype, Hkv, B, k_new, v_new, qpos, new_slot, kp, vp, th, s);
  if (e != cudaSuccess) return e;
  return launch_decode(dtype, B, Hq, Hkv, q, qpos, kp, vp, indptr, indices, max_kv, out, ws, th,
                       s);
}

cudaError_t launch_decode(int dtype, int B, int Hq, int Hkv, const void *q, const int32_t *qpos,
                          const void *kp, const void *vp, const int32_t *indptr,
                          const int32_t *indices, int max_kv, void *out, void *ws,
                          const RopeTheta &th, cudaStream_t s) {
  const int ns = n_splits(max_kv);
  Partials part = partials(ws, B, Hq, max_kv);
  if (dtype == AKV_BF16) {
    return decode_bf16(B, Hq, Hkv, q, qpos, const_cast<void *>(kp), const_cast<void *>(vp),
                       indptr, indices, max_kv, out, ws, th, nullptr, nullptr, nullptr, s);
  } else {
    dim3 grid(ns, Hq, B);
    decode_f32_kernel<<<grid, 128, 0, s>>>(Hq, Hkv, (const float *)q, qpos, (const float *)kp,
                                          (const float *)vp, indptr, indices, part, th);
    decode_combine_kernel<float><<<dim3(Hq, B), kD, 0, s>>>(Hq, ns, kChunk, indptr, part, (float *)out);
  }
  return cudaGetLastError();
}

cudaError_t launch_decode_rope(int dtype, int B, int Hq, int Hkv, const void *q,
                               const int32_t *qpos, const void *k_new, const void *v_new,
                               const int32_t *new_slot, void *kp, void *vp, const int32_t *indptr,
                               const int32_t *indices, const int32_t *kvpos, int max_kv, void *out,
                               void *ws, const RopeTheta &th, cudaStream_t s) {
  const int ns = n_splits(max_kv, kRChunk);
  Partials part = partials(ws, B, Hq, max_kv, kRChunk);
  if (dtype == AKV_BF16)
    return decode_bf16(B, Hq, Hkv, q, qpos, kp, vp, indptr, indices, max_kv, out, ws, th, k_new,
                       v_new, new_slot, s, kvpos);
  decode_rope_f32_kernel<<<dim3(ns, Hq, B), 128, 0, s>>>(
      Hq, Hkv, (const float *)q, qpos, (const float *)k_new, (const float *)v_new, new_slot,
      (float *)kp, (float *)vp, indptr, indices, kvpos, part, th);
  decode_combine_kernel<float><<<dim3(Hq, B), kD, 0, s>>>(Hq, ns, kRChunk, indptr, part, (float *)out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Debug check of caller-provided decode index data, which the decode kernels
// trust (an out-of-range slot would be read).  Reads only kv_indptr and
// kv_indices; never touches a pool slot.
// ---------------------------------------------------------------------------
namespace {
__global__ void check_indices_kernel(int B, const int32_t *__restrict__ indptr,
                                     const int32_t *__restrict__ indices, int S, int max_kv,
                                     int64_t nnz_cap, uint32_t *status) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  uint32_t bad = 0;
  if (tid == 0 && indptr[0] != 0) bad |= kDecodeIndptr;
  for (int64_t b = tid; b < B; b += stride) {
    const int64_t len = (int64_t)indptr[b + 1] - indptr[b];
    if (len < 0 || len > max_kv) bad |= kDecodeIndptr;
  }
  // the entries actually listed (bounded by the caller's capacity)
  int64_t nnz = indptr[B];
  if (nnz < 0) nnz = 0;
  if (nnz > nnz_cap) {
    if (tid == 0) bad |= kDecodeIndptr;
    nnz = nnz_cap;
  }
  for (int64_t i = tid; i < nnz; i += stride) {
    const int32_t slot = indices[i];
    if (slot < 0 || slot >= S) bad |= kDecodeSlot;
  }
  if (bad) atomicOr(status, bad);
}
}  // namespace

cudaError_t launch_check_indices(int B, const int32_t *indptr, const int32_t *indices, int S,
                                 int max_kv, int64_t nnz_cap, uint32_t *status, cudaStream_t s) {
  const int64_t work = nnz_cap > B ? nnz_cap : B;
  const int64_t want = (work + 255) / 256;
  const unsigned grid = (unsigned)(want < 4096 ? (want > 0 ? want : 1) : 4096);
  check_indices_kernel<<<grid, 256, 0, s>>>(B, indptr, indices, S, max_kv, nnz_cap, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Decode without a caller workspace.  The split-KV partials and merge
// counters go to a fixed array in this module's device memory instead: every
// GPU on which the module is loaded keeps kStaticScratchBytes for it until the
// process exits (under lazy module loading the module, and so the array, is
// loaded with the first use of one of this file's kernels or symbols).  Host
// code cannot pass the array's name to a kernel (on the host it is only a
// stand-in, not a device address), so every call looks its address up with
// cudaGetSymbolAddress in the current context.  The address is not cached:
// it belongs to the context the module was loaded into, and a device reset
// or another context made current on the same device would leave a cached
// one pointing at memory that is no longer this array.
// ---------------------------------------------------------------------------
namespace {
__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];
}  // namespace

cudaError_t decode_static_scratch(void **ptr) {
  void *a = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&a, g_decode_scratch);
  if (e != cudaSuccess) return e;
  *ptr = a;
  return cudaSuccess;
}

cudaError_t launch_decode_static(int dtype, int B, int Hq, int Hkv, const void *q,
                                 const int32_t *qpos, const void *kp, const void *vp,
                                 const int32_t *indptr, const int32_t *indices, int max_kv,
                                 void *out, const RopeTheta &th, cudaStream_t s) {
  void *scratch = nullptr;
  const cudaError_t e = decode_static_scratch(&scratch);
  if (e != cudaSuccess) return e;
  return launch_decode(dtype, B, Hq, Hkv, q, qpos, kp, vp, indptr, indices, max_kv, out, scratch,
                       th, s);
}

}  // namespace akv
