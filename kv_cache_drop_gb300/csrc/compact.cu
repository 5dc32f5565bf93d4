// Compaction of the active cache (drop, paper review page section 3.3; the
// active cache vs the logical trajectory, explainer page section 1).
//
// The host reduces the op log to two flags per message (survives the drops
// up to the boundary; alive right after the last earlier repos).  On the
// device every token takes its message's flags, and two exclusive scans give
// each survivor its place in the compacted list and its position (rank among
// the survivors of the last repos, or r + offset for later appends).  Two
// launches: per-block counts, then per-block prefix (over the few preceding
// block counts) + block scan + scatter.  Bit-exact integer work.
//
// Since both flags are per message, the survivors are runs of whole kept
// messages whose positions are consecutive within a run; when there are few
// runs the host passes them in the kernel's parameters and one launch
// expands them, one thread per compacted index (compact_runs_kernel).
#include "common.cuh"

namespace akv {
namespace {

constexpr int kThreads = 256;
constexpr int kPer = 4;  // consecutive tokens per thread
constexpr int kBlock = kThreads * kPer;

constexpr int kSmemMsgs = 2048;  // per-message tables staged in shared memory up to this size

__device__ __forceinline__ int msg_of(const int32_t *ms, int n_msgs, int u) {
  int lo = 0, hi = n_msgs;  // ms[lo] <= u < ms[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (ms[mid] <= u) lo = mid; else hi = mid;
  }
  return lo;
}

// The message of a token is found by binary search in msg_start, a chain of
// dependent loads: the block first copies the per-message tables into
// shared memory (coalesced) and searches there.  Returns the view to use.
__device__ __forceinline__ CompactDev stage_tables(const CompactDev &c, int32_t *s_ms,
                                                   uint8_t *s_keep, uint8_t *s_alive) {
  if (c.n_msgs > kSmemMsgs) return c;
  for (int i = threadIdx.x; i <= c.n_msgs; i += blockDim.x) s_ms[i] = __ldg(c.msg_start + i);
  for (int i = threadIdx.x; i < c.n_msgs; i += blockDim.x) {
    s_keep[i] = __ldg(c.keep + i);
    s_alive[i] = __ldg(c.alive_br + i);
  }
  __syncthreads();
  CompactDev v = c;
  v.msg_start = s_ms;
  v.keep = s_keep;
  v.alive_br = s_alive;
  return v;
}

// flags of the kPer tokens of this thread: bit i of keep / alive
__device__ __forceinline__ void token_flags(const CompactDev &c, int u0, uint32_t *keep,
                                            uint32_t *alive) {
  *keep = 0;
  *alive = 0;
  if (u0 >= c.T) return;
  int m = msg_of(c.msg_start, c.n_msgs, u0);
  for (int i = 0; i < kPer; ++i) {
    const int u = u0 + i;
    if (u >= c.T) break;
    while (c.msg_start[m + 1] <= u) ++m;
    if (c.keep[m]) *keep |= 1u << i;
    if (c.has_br && u < c.br_end && c.alive_br[m]) *alive |= 1u << i;
  }
}

// exclusive block scan of two counters packed as (hi << 16) | lo
__device__ __forceinline__ uint32_t block_exscan(uint32_t x, uint32_t *total) {
  __shared__ uint32_t warp_sum[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_sum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = warp_sum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sum[lane] = w;  // inclusive
  }
  __syncthreads();
  const uint32_t before = (warp ? warp_sum[warp - 1] : 0u) + inc - x;
  *total = warp_sum[kThreads / 32 - 1];
  return before;
}

__global__ void __launch_bounds__(kThreads) compact_count_kernel(CompactDev cg) {
  __shared__ int32_t s_ms[kSmemMsgs + 1];
  __shared__ uint8_t s_keep[kSmemMsgs], s_alive[kSmemMsgs];
  const CompactDev c = stage_tables(cg, s_ms, s_keep, s_alive);
  uint32_t keep, alive;
  token_flags(c, blockIdx.x * kBlock + threadIdx.x * kPer, &keep, &alive);
  uint32_t total;
  block_exscan(((uint32_t)__popc(alive) << 16) | (uint32_t)__popc(keep), &total);
  if (threadIdx.x == 0) {
    c.block_cnt[2 * blockIdx.x] = (int32_t)(total & 0xffffu);
    c.block_cnt[2 * blockIdx.x + 1] = (int32_t)(total >> 16);
  }
}

__global__ void __launch_bounds__(kThreads) compact_write_kernel(CompactDev cg, int32_t *active_idx,
                                                                 int32_t *active_pos) {
  __shared__ int32_t s_ms[kSmemMsgs + 1];
  __shared__ uint8_t s_keep[kSmemMsgs], s_alive[kSmemMsgs];
  const CompactDev c = stage_tables(cg, s_ms, s_keep, s_alive);
  __shared__ int32_t base_keep, base_alive;
  if (threadIdx.x < 32) {
    int32_t a = 0, b = 0;
    for (int i = threadIdx.x; i < (int)blockIdx.x; i += 32) {
      a += c.block_cnt[2 * i];
      b += c.block_cnt[2 * i + 1];
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if (threadIdx.x == 0) {
      base_keep = a;
      base_alive = b;
    }
  }
  const int u0 = blockIdx.x * kBlock + threadIdx.x * kPer;
  uint32_t keep, alive;
  token_flags(c, u0, &keep, &alive);
  uint32_t total;
  const uint32_t ex = block_exscan(((uint32_t)__popc(alive) << 16) | (uint32_t)__popc(keep), &total);
  int32_t k_at = base_keep + (int32_t)(ex & 0xffffu);
  int32_t a_at = base_alive + (int32_t)(ex >> 16);
  for (int i = 0; i < kPer; ++i) {
    const int u = u0 + i;
    if (u >= c.T) break;
    int32_t pos;
    if (!c.has_br) pos = u;
    else if (u < c.br_end) pos = a_at;
    else pos = c.r + (u - c.br_end);
    if (alive >> i & 1u) ++a_at;
    if (keep >> i & 1u) {
      active_idx[k_at] = u;
      active_pos[k_at] = pos;
      ++k_at;
    }
  }
}

// thread = compacted index j: its run by binary search over the run table
// (lanes of a warp mostly share a run, so the parameter reads broadcast)
__global__ void __launch_bounds__(kThreads)
    compact_runs_kernel(int n, const __grid_constant__ KeptRunTable rt, int32_t *__restrict__ active_idx,
                        int32_t *__restrict__ active_pos) {
  const int64_t jj = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  if (jj >= n) return;
  const int j = (int)jj;
  int run, off;
  rt.find(j, &run, &off);
  active_idx[j] = rt.kstart(run) + off;
  active_pos[j] = rt.kpos(run) + off;
}

__global__ void __launch_bounds__(256) param_upload_kernel(const ParamBlob blob, char *dst) {
  for (int sg = 0; sg < blob.n_seg; ++sg) {
    const ParamSeg g = blob.seg[sg];
    for (uint32_t i = threadIdx.x; i < g.bytes; i += blockDim.x)
      dst[g.dst_off + i] = (char)blob.data[g.src_off + i];
  }
}

// grid-stride copy of segments from a device-visible host block; 16 bytes
// at a time where source, destination and length are 16-byte multiples
__global__ void __launch_bounds__(256) mapped_upload_kernel(const uint8_t *__restrict__ src,
                                                            char *__restrict__ dst,
                                                            const UploadSegs segs) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int sg = 0; sg < segs.n; ++sg) {
    const ParamSeg g = segs.seg[sg];
    const uint8_t *s = src + g.src_off;
    char *d = dst + g.dst_off;
    int64_t done = 0;
    if (((g.src_off | g.dst_off | (uintptr_t)src | (uintptr_t)dst) & 15) == 0) {
      const int64_t n16 = g.bytes / 16;
      for (int64_t i = tid; i < n16; i += stride)
        reinterpret_cast<uint4 *>(d)[i] = reinterpret_cast<const uint4 *>(s)[i];
      done = n16 * 16;
    }
    for (int64_t i = done + tid; i < (int64_t)g.bytes; i += stride) d[i] = (char)s[i];
  }
}

}  // namespace

int compact_blocks(int T) { return (T + kBlock - 1) / kBlock; }

cudaError_t launch_mapped_upload(const void *src_dev, char *dst, const UploadSegs &segs,
                                 cudaStream_t s) {
  int64_t total = 0;
  for (int i = 0; i < segs.n; ++i) total += segs.seg[i].bytes;
  if (total == 0) return cudaSuccess;
  const int64_t want = (total / 16 + 255) / 256;
  const unsigned grid = (unsigned)(want < 1024 ? (want > 0 ? want : 1) : 1024);
  mapped_upload_kernel<<<grid, 256, 0, s>>>((const uint8_t *)src_dev, dst, segs);
  return cudaGetLastError();
}

cudaError_t launch_param_upload(char *dst, const ParamBlob &blob, cudaStream_t s) {
  param_upload_kernel<<<1, 256, 0, s>>>(blob, dst);
  return cudaGetLastError();
}

cudaError_t launch_compact(const CompactDev &c, int32_t *active_idx, int32_t *active_pos,
                           cudaStream_t s) {
  const int nb = compact_blocks(c.T);
  compact_count_kernel<<<nb, kThreads, 0, s>>>(c);
  compact_write_kernel<<<nb, kThreads, 0, s>>>(c, active_idx, active_pos);
  return cudaGetLastError();
}

cudaError_t launch_compact_runs(int n, int nk, const int32_t *kstart, const int32_t *kprefix,
                                const int32_t *kpos, int32_t *active_idx, int32_t *active_pos,
                                cudaStream_t s) {
  KeptRunTable rt;
  if (n < 1 || !fill_run_table(&rt, nk, kstart, kprefix, kpos)) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)(((int64_t)n + kThreads - 1) / kThreads);
  compact_runs_kernel<<<grid, kThreads, 0, s>>>(n, rt, active_idx, active_pos);
  return cudaGetLastError();
}

}  // namespace akv
