// C ABI of libakv: argument validation, the host planner for segment-batch
// restoration, workspace layout, and kernel orchestration.
//
// The planner restates "Cache Engineering for Agents" (paper review page,
// section 3.3 cache operations, section 4 operate-after grammar / Figure 6,
// section 4.2 and Appendix A.1.1 segment-batch attention):
//  * a segment ends at every boundary that lists a drop or a repos;
//  * row t (segment seg(t)) sees key u iff u <= t and seg(t) < drop_seg(u),
//    where drop_seg(u) is the segment right after the boundary that first
//    drops u's message;
//  * every repos opens a new key version: the survivors are renumbered
//    0..r-1 in logical order and later appends continue from r; rows read
//    keys at the positions of their own version.
// Key slots are permuted once per request so that keys with the same drop
// segment are contiguous (never-dropped keys first, then by decreasing drop
// segment, logical order inside): the keys a query tile can see then form a
// few long runs instead of one run per surviving message, and the attention
// kernels cover them with 128-key windows.
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <numeric>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "akv_internal.h"

using namespace akv;

namespace {

thread_local std::string g_err;

akv_status fail(akv_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

akv_status cuda_fail(cudaError_t e, const char *what) {
  return fail(AKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// AKV_FAULT=invalid|cuda|workspace makes entry points fail before launching
// anything, so callers can exercise their error paths without a GPU fault.
akv_status injected_fault(const char *entry) {
  static const char *f = getenv("AKV_FAULT");
  if (!f || !*f) return AKV_OK;
  if (!strcmp(f, "invalid")) return fail(AKV_ERR_INVALID, "%s: injected fault", entry);
  if (!strcmp(f, "cuda")) return fail(AKV_ERR_CUDA, "%s: injected fault", entry);
  if (!strcmp(f, "workspace")) return fail(AKV_ERR_WORKSPACE, "%s: injected fault", entry);
  return AKV_OK;
}

// Every entry point opens an NVTX range named after it (visible to nsys and
// to ncu --nvtx; no cost without a tool attached), then applies AKV_FAULT.
struct NvtxRange {
  explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange &) = delete;
  NvtxRange &operator=(const NvtxRange &) = delete;
};
#define AKV_ENTRY(name)            \
  NvtxRange akv_nvtx_range_(name); \
  if (akv_status akv_fault_ = injected_fault(name)) return akv_fault_

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t esize(akv_dtype d) { return d == AKV_F32 ? 4 : 2; }

akv_status check_shape(const akv_shape *s) {
  if (!s) return fail(AKV_ERR_INVALID, "shape is NULL");
  if (s->Hq <= 0 || s->Hkv <= 0 || s->Hq % s->Hkv)
    return fail(AKV_ERR_INVALID, "need Hq %% Hkv == 0 (Hq=%d Hkv=%d)", s->Hq, s->Hkv);
  if (s->dtype != AKV_F32 && s->dtype != AKV_BF16)
    return fail(AKV_ERR_INVALID, "unknown dtype %d", (int)s->dtype);
  if (!(s->rope_base > 1.0f) || !std::isfinite(s->rope_base))
    return fail(AKV_ERR_INVALID, "rope_base must be finite and > 1");
  if (s->D != kD) return fail(AKV_ERR_UNSUPPORTED, "head dim %d (only %d)", s->D, kD);
  return AKV_OK;
}

// Validate one op log against the request's token count.
akv_status check_oplog(const akv_oplog *o, int64_t T, int req) {
  if (!o) return fail(AKV_ERR_INVALID, "request %d: op log is NULL", req);
  if (o->n_msgs < 0 || o->n_drops < 0 || o->n_repos < 0)
    return fail(AKV_ERR_INVALID, "request %d: negative count", req);
  if (!o->msg_start) return fail(AKV_ERR_INVALID, "request %d: msg_start is NULL", req);
  if (o->msg_start[0] != 0) return fail(AKV_ERR_INVALID, "request %d: msg_start[0] != 0", req);
  for (int m = 0; m < o->n_msgs; ++m)
    if (o->msg_start[m + 1] < o->msg_start[m])
      return fail(AKV_ERR_INVALID, "request %d: msg_start decreases at %d", req, m);
  if (T >= 0 && o->msg_start[o->n_msgs] != T)
    return fail(AKV_ERR_INVALID, "request %d: messages hold %d tokens, rows %lld", req,
                o->msg_start[o->n_msgs], (long long)T);
  if (o->n_drops && (!o->drop_after || !o->drop_target))
    return fail(AKV_ERR_INVALID, "request %d: drop arrays are NULL", req);
  if (o->n_repos && !o->repos_after)
    return fail(AKV_ERR_INVALID, "request %d: repos array is NULL", req);
  for (int i = 0; i < o->n_drops; ++i) {
    int a = o->drop_after[i], t = o->drop_target[i];
    if (a < 0 || a >= o->n_msgs)
      return fail(AKV_ERR_INVALID, "request %d: drop boundary %d out of range", req, a);
    if (t < 0 || t > a)
      return fail(AKV_ERR_INVALID,
                  "request %d: drop target %d must be an appended message (<= %d)", req, t, a);
  }
  for (int i = 0; i < o->n_repos; ++i) {
    int a = o->repos_after[i];
    if (a < 0 || a >= o->n_msgs)
      return fail(AKV_ERR_INVALID, "request %d: repos boundary %d out of range", req, a);
  }
  return AKV_OK;
}

}  // namespace

void akv::rope_theta(float base, RopeTheta *out) {
  for (int i = 0; i < kD / 2; ++i) {
    out->th[i] = std::pow((double)base, -2.0 * i / kD);
    out->hi[i] = (float)out->th[i];
    out->lo[i] = (float)(out->th[i] - (double)out->hi[i]);
  }
}

// ------------------------------------------------------------------------
// Plan
// ------------------------------------------------------------------------

struct WsLayout {
  size_t status, tok_qpos, tok_seg, slot_src, slot_u, slot_dseg, slot_pos, qtiles, windows, mwin, mask,
      order, qcs, qr, kr, vp, total;
};

struct akv_plan {
  akv_shape shape{};
  int n_req = 0;
  int64_t T = 0;
  int max_ver = 1;
  std::vector<int32_t> tok_pos, tok_seg, tok_ver, drop_seg;  // request-relative
  std::vector<int32_t> slot_src, slot_u, slot_dseg, slot_pos;
  std::vector<QTile> qtiles;
  std::vector<MaskWin> mwin;
  std::vector<uint32_t> windows;
  std::vector<int32_t> order;
  int64_t visible_pairs = 0, n_full = 0, n_segments = 0;
  WsLayout ws{};
};

namespace {

struct Group {  // run of permuted slots sharing one drop segment
  int32_t begin, end, dseg;
};

// Plan one request: tables for its stored rows and its query tiles.  The
// request's logical rows are 0..T-1; with a shared prefix of Ps rows (held
// by another request whose key slots start at owner_c0) only rows Ps..T-1
// are stored, at batch rows c0..c0+T-Ps-1, and its query tiles read the
// prefix keys through full windows over the owner's first slots.
void plan_request(akv_plan *P, int req, int64_t c0, const akv_oplog *o, int64_t Ps = 0,
                  int64_t owner_c0 = 0) {
  const int n = o->n_msgs;
  const int32_t *ms = o->msg_start;
  const int64_t T = ms[n];
  const int64_t Tst = T - Ps;  // stored rows
  std::vector<std::vector<int>> drops_at(n);
  std::vector<char> repos_at(n, 0);
  for (int i = 0; i < o->n_drops; ++i) drops_at[o->drop_after[i]].push_back(o->drop_target[i]);
  for (int i = 0; i < o->n_repos; ++i) repos_at[o->repos_after[i]] = 1;

  std::vector<int32_t> tpos_v(T), tseg_v(T), tver_v(T), dseg_v(T);
  int32_t *tpos = tpos_v.data(), *tseg = tseg_v.data(), *tver = tver_v.data(),
          *dseg = dseg_v.data();
  std::vector<char> alive(n, 0);
  std::vector<int32_t> msg_dseg(n, INT32_MAX);
  // positions per version: version 0 and every repos
  std::vector<std::vector<int32_t>> vpos(1, std::vector<int32_t>(T, -1));
  std::vector<int> ver_first_msg(1, 0);  // first message appended in each version
  int64_t next_pos = 0, n_active = 0;
  int seg = 0, ver = 0;
  for (int m = 0; m < n; ++m) {
    const int64_t a = ms[m], b = ms[m + 1];
    for (int64_t t = a; t < b; ++t) {
      tpos[t] = (int32_t)next_pos;
      vpos[ver][t] = (int32_t)next_pos;
      ++next_pos;
      tseg[t] = seg;
      tver[t] = ver;
      // row t sees the active cache at its start plus its own message prefix
      if (t >= Ps) P->visible_pairs += n_active + (t - a) + 1;
    }
    alive[m] = 1;
    n_active += b - a;
    bool op = false;
    for (int j : drops_at[m]) {
      op = true;
      if (alive[j]) {
        alive[j] = 0;
        msg_dseg[j] = seg + 1;
        n_active -= ms[j + 1] - ms[j];
      }
    }
    if (repos_at[m]) {
      op = true;
      ++ver;
      vpos.emplace_back(T, -1);
      ver_first_msg.push_back(m + 1);
      int32_t r = 0;
      for (int j = 0; j <= m; ++j)
        if (alive[j])
          for (int64_t u = ms[j]; u < ms[j + 1]; ++u) vpos[ver][u] = r++;
      next_pos = r;
    }
    if (op) ++seg;
  }
  const int n_seg = seg + 1, n_ver = ver + 1;
  P->n_segments += n_seg;
  for (int m = 0; m < n; ++m)
    for (int64_t u = ms[m]; u < ms[m + 1]; ++u) dseg[u] = msg_dseg[m];
  for (int64_t t = Ps; t < T; ++t) {  // stored rows
    P->tok_pos[c0 + t - Ps] = tpos[t];
    P->tok_seg[c0 + t - Ps] = tseg[t];
    P->tok_ver[c0 + t - Ps] = tver[t];
    P->drop_seg[c0 + t - Ps] = dseg[t];
  }

  // permuted slot order: messages by decreasing drop segment, then logical order
  std::vector<int> morder(n);
  std::iota(morder.begin(), morder.end(), 0);
  std::stable_sort(morder.begin(), morder.end(),
                   [&](int x, int y) { return msg_dseg[x] > msg_dseg[y]; });
  std::vector<Group> groups;
  std::vector<int32_t> u_of(Tst);  // local slot -> local (logical) row
  {
    int64_t j = 0;
    for (int m : morder) {
      if (ms[m + 1] == ms[m] || ms[m] < Ps) continue;  // empty, or in the shared prefix
      if (groups.empty() || groups.back().dseg != msg_dseg[m])
        groups.push_back({(int32_t)j, (int32_t)j, msg_dseg[m]});
      for (int64_t u = ms[m]; u < ms[m + 1]; ++u) u_of[j++] = (int32_t)u;
      groups.back().end = (int32_t)j;
    }
  }
  for (int64_t j = 0; j < Tst; ++j) {
    P->slot_src[c0 + j] = (int32_t)(c0 + u_of[j] - Ps);
    P->slot_u[c0 + j] = (int32_t)(c0 + u_of[j] - Ps);
    P->slot_dseg[c0 + j] = dseg[u_of[j]];
    for (int v = 0; v < P->max_ver; ++v) {
      int32_t p = v < n_ver ? vpos[v][u_of[j]] : -1;
      P->slot_pos[(size_t)v * P->T + c0 + j] = p < 0 ? 0 : p;
    }
  }

  // query tiles: per version, consecutive rows, 128 at a time
  for (int v = 0; v < n_ver; ++v) {
    int64_t r0 = std::max<int64_t>(Ps, ms[ver_first_msg[v]]);
    int64_t r1 = (v + 1 < n_ver) ? ms[ver_first_msg[v + 1]] : T;
    for (int64_t t0 = r0; t0 < r1; t0 += kTileQ) {
      const int64_t t1 = std::min<int64_t>(r1, t0 + kTileQ);
      QTile q{};
      q.t0 = (int32_t)(c0 + t0 - Ps);
      q.len = (int32_t)(t1 - t0);
      q.ver = v;
      q.req = req;
      q.win_off = (int32_t)P->windows.size();
      q.pm_off = (int32_t)P->mwin.size();
      q.seg_lo = tseg[t0];
      q.seg_hi = tseg[t1 - 1];
      // the shared prefix: never dropped, before every stored row, Ps a
      // multiple of 128 -> full windows over the owner's first slots
      for (int64_t a = 0; a < Ps; a += kTileK) {
        P->windows.push_back((uint32_t)(owner_c0 + a) | kWinFull);
        ++P->n_full;
      }
      // visible slot intervals, in slot order: groups with dseg > seg_lo, the
      // prefix of each with u <= t1-1
      int64_t cover_end = -1;
      for (const Group &g : groups) {
        if (g.dseg <= q.seg_lo) break;  // groups are by decreasing dseg
        if (u_of[g.begin] > t1 - 1) continue;
        const int32_t *e = std::upper_bound(u_of.data() + g.begin, u_of.data() + g.end,
                                            (int32_t)(t1 - 1));
        int64_t a = g.begin, b = e - u_of.data();
        if (a < cover_end) a = cover_end;
        while (a < b) {
          // full if every slot of [a, a+128) is in this request, in groups
          // that outlive the tile, and not after the tile's first row
          bool full = a + kTileK <= Tst;
          if (full) {
            int64_t s = a;
            const Group *gp = &g;
            while (full && s < a + kTileK) {
              while (!(gp->begin <= s && s < gp->end)) ++gp;
              int64_t last = std::min<int64_t>(gp->end, a + kTileK) - 1;
              if (gp->dseg <= q.seg_hi || u_of[last] > t0) full = false;
              s = last + 1;
            }
          }
          P->windows.push_back((uint32_t)(c0 + a) | (full ? kWinFull : 0u));
          if (full) ++P->n_full;
          else P->mwin.push_back({q.t0, q.len, (int32_t)(c0 + a), 0});
          cover_end = a + kTileK;
          a = cover_end;
        }
      }
      q.win_cnt = (int32_t)(P->windows.size() - q.win_off);
      q.pm_cnt = (int32_t)(P->mwin.size() - q.pm_off);
      P->qtiles.push_back(q);
    }
  }
}

void layout_workspace(akv_plan *P) {
  WsLayout &w = P->ws;
  const size_t T = (size_t)P->T, nt = P->qtiles.size(), nw = P->windows.size();
  const size_t es = esize(P->shape.dtype);
  size_t o = 0;
  auto take = [&](size_t bytes, size_t al) {
    o = align_up(o, al);
    size_t r = o;
    o += bytes;
    return r;
  };
  w.status = take(256, 256);
  w.tok_qpos = take(4 * T, 256);
  w.tok_seg = take(4 * T, 256);
  w.slot_src = take(4 * T, 256);
  w.slot_u = take(4 * (T + kSlotPad), 256);
  w.slot_dseg = take(4 * (T + kSlotPad), 256);
  w.slot_pos = take(4 * T * P->max_ver, 256);
  w.qtiles = take(sizeof(QTile) * nt, 256);
  w.windows = take(4 * nw, 256);
  w.mwin = take(sizeof(MaskWin) * P->mwin.size(), 256);
  w.mask = take((size_t)kTileQ * 16 * P->mwin.size(), 256);
  w.order = take(4 * nt, 256);
  // bf16: the attention kernel rotates each query row itself, from the raw
  // Q and a per-row cos/sin table; fp32: the pre-pass writes rotated queries
  const bool bf16 = P->shape.dtype == AKV_BF16;
  w.qcs = take(bf16 ? 8 * T * (kD / 2) : 0, 256);
  w.qr = take(bf16 ? 0 : es * T * P->shape.Hq * kD, 1024);
  w.kr = take(es * T * P->shape.Hkv * kD * P->max_ver, 1024);
  w.vp = take(es * T * P->shape.Hkv * kD, 1024);
  w.total = align_up(o, 1024);
}

PlanDev device_view(const akv_plan *P, void *ws) {
  char *b = (char *)ws;
  const WsLayout &w = P->ws;
  PlanDev d{};
  d.status = (uint32_t *)(b + w.status);
  d.tok_qpos = (const int32_t *)(b + w.tok_qpos);
  d.tok_seg = (const int32_t *)(b + w.tok_seg);
  d.slot_src = (const int32_t *)(b + w.slot_src);
  d.slot_u = (const int32_t *)(b + w.slot_u);
  d.slot_dseg = (const int32_t *)(b + w.slot_dseg);
  d.slot_pos = (const int32_t *)(b + w.slot_pos);
  d.qtiles = (const QTile *)(b + w.qtiles);
  d.windows = (const uint32_t *)(b + w.windows);
  d.mwin = (const MaskWin *)(b + w.mwin);
  d.mask = (uint4 *)(b + w.mask);
  d.n_mask = (int32_t)P->mwin.size();
  d.order = (const int32_t *)(b + w.order);
  d.qr = b + w.qr;
  d.qcs = (float2 *)(b + w.qcs);
  d.kr = b + w.kr;
  d.vp = b + w.vp;
  d.T = P->T;
  d.n_qtiles = (int32_t)P->qtiles.size();
  d.max_ver = P->max_ver;
  d.Hq = P->shape.Hq;
  d.Hkv = P->shape.Hkv;
  d.rope_base = P->shape.rope_base;
  d.dtype = (int32_t)P->shape.dtype;
  return d;
}

// Host-to-device uploads of tables built on the host.  A cudaMemcpyAsync
// from pageable memory returns only after the copy has run, i.e. after all
// earlier work on the stream, so every call would wait for the GPU.  The
// tables are instead packed into pinned host blocks owned by the library and
// copied from there asynchronously.  A block is handed out again only once
// every copy out of it has completed (one event per upload); blocks are
// kept for reuse and never freed before the process exits.
struct HostPart {
  size_t dst_off;  // byte offset from the destination base
  const void *src;
  size_t bytes;
};

class PinnedPool {
 public:
  struct Block {
    char *p = nullptr;
    size_t bytes = 0;
    std::vector<cudaEvent_t> pending;  // uploads from this block not yet known complete
  };
  // A block of at least `bytes` with no copy in flight; false if pinned
  // memory cannot be had.  At most kMaxBlocks blocks are allocated: beyond
  // that the caller waits for the copies out of a block that fits (the host
  // is then at most a few uploads ahead of the GPU), instead of pinning more
  // memory (pinning is slow and may synchronise the device).
  bool acquire(size_t bytes, Block *out) {
    std::unique_lock<std::mutex> lock(mu_);
    int best = -1, busy = -1;
    for (int i = 0; i < (int)free_.size(); ++i) {
      Block &b = free_[i];
      prune(&b);
      if (b.bytes < bytes) continue;
      if (b.pending.empty()) {
        if (best < 0 || b.bytes < free_[best].bytes) best = i;
      } else if (busy < 0) {
        busy = i;  // the oldest returned block that fits
      }
    }
    if (best < 0 && busy >= 0 && n_alloc_ >= kMaxBlocks) best = busy;
    if (best >= 0) {
      *out = std::move(free_[best]);
      free_.erase(free_.begin() + best);
      lock.unlock();
      for (cudaEvent_t e : out->pending) {
        (void)cudaEventSynchronize(e);
        cudaEventDestroy(e);
      }
      (void)cudaGetLastError();
      out->pending.clear();
      return true;
    }
    Block b;
    b.bytes = align_up(std::max<size_t>(bytes, 1), size_t(1) << 20);
    if (cudaHostAlloc((void **)&b.p, b.bytes, cudaHostAllocPortable | cudaHostAllocMapped) !=
        cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    ++n_alloc_;
    *out = std::move(b);
    return true;
  }
  void release(Block b) {
    std::lock_guard<std::mutex> lock(mu_);
    free_.push_back(std::move(b));
  }

 private:
  static void prune(Block *b) {
    std::vector<cudaEvent_t> keep;
    for (cudaEvent_t e : b->pending) {
      const cudaError_t q = cudaEventQuery(e);
      if (q == cudaErrorNotReady) {
        keep.push_back(e);
      } else {
        (void)cudaGetLastError();
        cudaEventDestroy(e);
      }
    }
    b->pending.swap(keep);
  }
  static constexpr int kMaxBlocks = 4;
  std::mutex mu_;
  std::vector<Block> free_;  // returned blocks, oldest first
  int n_alloc_ = 0;
};

PinnedPool &pinned_pool() {
  static PinnedPool *pool = new PinnedPool();  // never destroyed: blocks may be in use at exit
  return *pool;
}

// Copies the parts to dst + dst_off on stream s without waiting for the
// stream.  A few KB at most travel as the parameters of a copy kernel (no
// copy-engine start-up); larger uploads go through the pinned blocks, or
// plain (blocking) copies when no pinned memory can be had.
cudaError_t upload_async(char *dst, const HostPart *parts, int n, cudaStream_t s) {
  size_t total = 0;
  bool off32 = true;  // segment offsets fit the copy kernels' 32-bit fields
  for (int i = 0; i < n; ++i) {
    total += align_up(parts[i].bytes, 16);
    off32 = off32 && parts[i].dst_off + parts[i].bytes <= (size_t)UINT32_MAX;
  }
  off32 = off32 && total <= (size_t)UINT32_MAX;
  if (off32 && total <= (size_t)kParamBlobBytes && n <= kParamMaxSegs) {
    ParamBlob blob;
    blob.n_seg = 0;
    size_t o = 0;
    for (int i = 0; i < n; ++i) {
      if (!parts[i].bytes) continue;
      std::memcpy(blob.data + o, parts[i].src, parts[i].bytes);
      blob.seg[blob.n_seg++] = ParamSeg{(uint32_t)parts[i].dst_off, (uint32_t)o,
                                        (uint32_t)parts[i].bytes};
      o += align_up(parts[i].bytes, 16);
    }
    return launch_param_upload(dst, blob, s);
  }
  PinnedPool::Block blk;
  if (!pinned_pool().acquire(total, &blk)) {
    for (int i = 0; i < n; ++i) {
      if (!parts[i].bytes) continue;
      cudaError_t e = cudaMemcpyAsync(dst + parts[i].dst_off, parts[i].src, parts[i].bytes,
                                      cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  size_t o = 0;
  for (int i = 0; i < n; ++i) {
    if (parts[i].bytes) std::memcpy(blk.p + o, parts[i].src, parts[i].bytes);
    o += align_up(parts[i].bytes, 16);
  }
  // The block is mapped: a kernel on the stream reads it directly.  (A
  // cudaMemcpyAsync would queue on a copy engine behind whatever the caller
  // is transferring on other streams, e.g. the next step's inputs.)
  cudaError_t e = cudaSuccess;
  void *dsrc = nullptr;
  if (off32 && n <= kUploadMaxSegs && cudaHostGetDevicePointer(&dsrc, blk.p, 0) == cudaSuccess) {
    UploadSegs segs;
    segs.n = 0;
    o = 0;
    for (int i = 0; i < n; ++i) {
      if (parts[i].bytes)
        segs.seg[segs.n++] = ParamSeg{(uint32_t)parts[i].dst_off, (uint32_t)o,
                                      (uint32_t)parts[i].bytes};
      o += align_up(parts[i].bytes, 16);
    }
    e = launch_mapped_upload(dsrc, dst, segs, s);
  } else {
    (void)cudaGetLastError();
    o = 0;
    for (int i = 0; i < n && e == cudaSuccess; ++i) {
      if (parts[i].bytes)
        e = cudaMemcpyAsync(dst + parts[i].dst_off, blk.p + o, parts[i].bytes,
                            cudaMemcpyHostToDevice, s);
      o += align_up(parts[i].bytes, 16);
    }
  }
  cudaEvent_t ev = nullptr;
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventRecord(ev, s);
  if (e != cudaSuccess) {
    // copies may be in flight without an event to track them: the block is
    // not reused (it stays allocated)
    if (ev) cudaEventDestroy(ev);
    return e;
  }
  blk.pending.push_back(ev);
  pinned_pool().release(std::move(blk));
  return cudaSuccess;
}

akv_status upload_plan(const akv_plan *P, void *ws, cudaStream_t s) {
  char *b = (char *)ws;
  const WsLayout &w = P->ws;
  const HostPart parts[] = {
      {w.tok_qpos, P->tok_pos.data(), 4 * P->tok_pos.size()},
      {w.tok_seg, P->tok_seg.data(), 4 * P->tok_seg.size()},
      {w.slot_src, P->slot_src.data(), 4 * P->slot_src.size()},
      {w.slot_u, P->slot_u.data(), 4 * P->slot_u.size()},
      {w.slot_dseg, P->slot_dseg.data(), 4 * P->slot_dseg.size()},
      {w.slot_pos, P->slot_pos.data(), 4 * P->slot_pos.size()},
      {w.qtiles, P->qtiles.data(), sizeof(QTile) * P->qtiles.size()},
      {w.windows, P->windows.data(), 4 * P->windows.size()},
      {w.mwin, P->mwin.data(), sizeof(MaskWin) * P->mwin.size()},
      {w.order, P->order.data(), 4 * P->order.size()},
  };
  cudaError_t e = cudaMemsetAsync(b + w.status, 0, 256, s);
  if (e != cudaSuccess) return cuda_fail(e, "status reset");
  e = upload_async(b, parts, (int)(sizeof(parts) / sizeof(parts[0])), s);
  if (e != cudaSuccess) return cuda_fail(e, "plan upload");
  return AKV_OK;
}

akv_status check_ws(const akv_plan *P, void *ws, size_t bytes) {
  if (!ws && P->ws.total) return fail(AKV_ERR_WORKSPACE, "workspace is NULL");
  if ((uintptr_t)ws % 256) return fail(AKV_ERR_WORKSPACE, "workspace not 256-byte aligned");
  if (bytes < P->ws.total)
    return fail(AKV_ERR_WORKSPACE, "workspace %zu bytes, need %zu", bytes, P->ws.total);
  return AKV_OK;
}

}  // namespace

extern "C" {

const char *akv_last_error(void) { return g_err.c_str(); }

const char *akv_version(void) { return "akv-gb300 0.1 (sm_103a)"; }

}  // extern "C"

namespace akv {
akv_status report_error(akv_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  return fail(st, "%s", buf);
}
akv_status validate_oplog(const akv_oplog *o, int64_t T, int req) { return check_oplog(o, T, req); }
akv_status fault_point(const char *entry) { return injected_fault(entry); }
}  // namespace akv

namespace {
// Shared prefix of request b (0 if none): validated against its owner.
akv_status check_share(int32_t n_req, const int32_t *cu_seqlens, const akv_oplog *ops,
                       const int32_t *share_from, const int32_t *share_len, int b,
                       int64_t *Ps) {
  *Ps = 0;
  if (!share_from || share_from[b] < 0) return AKV_OK;
  const int a = share_from[b];
  const int64_t L = share_len ? share_len[b] : 0;
  if (a >= b) return fail(AKV_ERR_INVALID, "request %d shares from %d: must be an earlier request", b, a);
  if (share_from[a] >= 0)
    return fail(AKV_ERR_INVALID, "request %d shares from %d, which itself shares a prefix", b, a);
  if (L <= 0 || L % kTileK)
    return fail(AKV_ERR_UNSUPPORTED, "request %d: shared length %lld must be a positive multiple of %d",
                b, (long long)L, kTileK);
  const akv_oplog &ob = ops[b], &oa = ops[a];
  int m_end = -1;  // the shared prefix is messages 0..m_end-1 in both requests
  for (int m = 0; m <= ob.n_msgs && m <= oa.n_msgs; ++m) {
    if (ob.msg_start[m] != oa.msg_start[m]) break;
    if (ob.msg_start[m] == L) { m_end = m; break; }
  }
  if (m_end < 0)
    return fail(AKV_ERR_INVALID, "request %d: shared length %lld is not a common message boundary of requests %d and %d",
                b, (long long)L, b, a);
  for (const akv_oplog *o : {&ob, &oa})
    for (int i = 0; i < o->n_drops; ++i)
      if (o->drop_target[i] < m_end)
        return fail(AKV_ERR_INVALID, "request %d: a shared prefix message (%d) is dropped", b,
                    o->drop_target[i]);
  if (L > oa.msg_start[oa.n_msgs] || (int64_t)cu_seqlens[a + 1] - cu_seqlens[a] != oa.msg_start[oa.n_msgs])
    return fail(AKV_ERR_INVALID, "request %d: owner %d must store all its rows", b, a);
  *Ps = L;
  (void)n_req;
  return AKV_OK;
}

akv_status plan_create_impl(const akv_shape *shape, int32_t n_req, const int32_t *cu_seqlens,
                            const int32_t *logical_idx, const akv_oplog *ops,
                            const int32_t *share_from, const int32_t *share_len,
                            akv_plan **plan_out) {
  AKV_ENTRY("akv_plan_create");
  if (!plan_out) return fail(AKV_ERR_INVALID, "plan_out is NULL");
  *plan_out = nullptr;
  if (akv_status st = check_shape(shape)) return st;
  if (n_req < 0 || (n_req > 0 && (!cu_seqlens || !ops)))
    return fail(AKV_ERR_INVALID, "bad request batch");
  if (n_req > 0 && cu_seqlens[0] != 0) return fail(AKV_ERR_INVALID, "cu_seqlens[0] != 0");
  std::vector<int64_t> shared(n_req, 0);
  for (int b = 0; b < n_req; ++b) {
    if (cu_seqlens[b + 1] < cu_seqlens[b])
      return fail(AKV_ERR_INVALID, "cu_seqlens decreases at %d", b);
    if (akv_status st = check_oplog(&ops[b], -1, b)) return st;
    if (akv_status st = check_share(n_req, cu_seqlens, ops, share_from, share_len, b, &shared[b]))
      return st;
    const int64_t Tb = ops[b].msg_start[ops[b].n_msgs];
    if ((int64_t)cu_seqlens[b + 1] - cu_seqlens[b] != Tb - shared[b])
      return fail(AKV_ERR_INVALID, "request %d: messages hold %lld tokens, %lld shared, rows %lld",
                  b, (long long)Tb, (long long)shared[b],
                  (long long)(cu_seqlens[b + 1] - cu_seqlens[b]));
  }
  const int64_t T = n_req ? cu_seqlens[n_req] : 0;
  if (T >= (int64_t)INT32_MAX - kSlotPad) return fail(AKV_ERR_UNSUPPORTED, "too many rows");
  if (logical_idx)
    for (int b = 0; b < n_req; ++b)
      for (int64_t i = cu_seqlens[b]; i < cu_seqlens[b + 1]; ++i)
        if (logical_idx[i] != i - cu_seqlens[b] + shared[b])
          return fail(AKV_ERR_INVALID, "row %lld carries logical index %d, expected %lld",
                      (long long)i, logical_idx[i],
                      (long long)(i - cu_seqlens[b] + shared[b]));
  akv_plan *P = new (std::nothrow) akv_plan;
  if (!P) return fail(AKV_ERR_INVALID, "host allocation failed");
  P->shape = *shape;
  P->n_req = n_req;
  P->T = T;
  int max_ver = 1;
  for (int b = 0; b < n_req; ++b) {
    std::vector<int> rb(ops[b].repos_after, ops[b].repos_after + ops[b].n_repos);
    std::sort(rb.begin(), rb.end());
    max_ver = std::max<int>(max_ver, 1 + (int)(std::unique(rb.begin(), rb.end()) - rb.begin()));
  }
  P->max_ver = max_ver;
  // the attention kernel addresses rotated-key rows (version, KV head, slot)
  // with one 32-bit TMA coordinate
  if ((int64_t)max_ver * shape->Hkv * T >= (int64_t)INT32_MAX) {
    delete P;
    return fail(AKV_ERR_UNSUPPORTED, "key versions x KV heads x rows (%d x %d x %lld) exceed 2^31",
                max_ver, shape->Hkv, (long long)T);
  }
  try {
    P->tok_pos.assign(T, 0);
    P->tok_seg.assign(T, 0);
    P->tok_ver.assign(T, 0);
    P->drop_seg.assign(T, INT32_MAX);
    P->slot_src.assign(T, 0);
    P->slot_u.assign(T + kSlotPad, INT32_MAX);
    P->slot_dseg.assign(T + kSlotPad, INT32_MIN);
    P->slot_pos.assign((size_t)T * max_ver, 0);
    for (int b = 0; b < n_req; ++b)
      plan_request(P, b, cu_seqlens[b], &ops[b], shared[b],
                   shared[b] ? cu_seqlens[share_from[b]] : 0);
    // a shared prefix is never dropped and precedes every other token, so its
    // keys sit at positions 0..Ps-1 in every key version of every sharer
    for (int b = 0; b < n_req; ++b)
      if (shared[b])
        for (int v = 0; v < max_ver; ++v)
          for (int64_t j = 0; j < shared[b]; ++j)
            P->slot_pos[(size_t)v * T + cu_seqlens[share_from[b]] + j] = (int32_t)j;
    P->order.resize(P->qtiles.size());
    std::iota(P->order.begin(), P->order.end(), 0);
    std::stable_sort(P->order.begin(), P->order.end(), [&](int x, int y) {
      return P->qtiles[x].win_cnt > P->qtiles[y].win_cnt;
    });
  } catch (const std::bad_alloc &) {
    delete P;
    return fail(AKV_ERR_INVALID, "host allocation failed while planning");
  }
  layout_workspace(P);
  *plan_out = P;
  return AKV_OK;
}
}  // namespace

extern "C" {

akv_status akv_plan_create(const akv_shape *shape, int32_t n_req, const int32_t *cu_seqlens,
                           const int32_t *logical_idx, const akv_oplog *ops,
                           akv_plan **plan_out) {
  return plan_create_impl(shape, n_req, cu_seqlens, logical_idx, ops, nullptr, nullptr, plan_out);
}

akv_status akv_plan_create_shared(const akv_shape *shape, int32_t n_req,
                                  const int32_t *cu_seqlens, const akv_oplog *ops,
                                  const int32_t *share_from, const int32_t *share_len,
                                  akv_plan **plan_out) {
  if (!share_from || !share_len) return fail(AKV_ERR_INVALID, "share_from/share_len is NULL");
  return plan_create_impl(shape, n_req, cu_seqlens, nullptr, ops, share_from, share_len,
                          plan_out);
}

void akv_plan_destroy(akv_plan *plan) { delete plan; }

akv_status akv_plan_get_info(const akv_plan *P, akv_plan_info *info) {
  if (!P || !info) return fail(AKV_ERR_INVALID, "NULL argument");
  info->T = P->T;
  info->n_qtiles = (int64_t)P->qtiles.size();
  info->n_windows = (int64_t)P->windows.size();
  info->n_full_windows = P->n_full;
  info->visible_pairs = P->visible_pairs;
  info->n_segments = P->n_segments;
  info->max_versions = P->max_ver;
  info->reserved = 0;
  info->workspace_bytes = P->ws.total;
  return AKV_OK;
}

akv_status akv_plan_tables(const akv_plan *P, int32_t *tok_pos, int32_t *tok_seg,
                           int32_t *tok_ver, int32_t *drop_seg) {
  if (!P) return fail(AKV_ERR_INVALID, "plan is NULL");
  const size_t n = (size_t)P->T * 4;
  if (tok_pos) memcpy(tok_pos, P->tok_pos.data(), n);
  if (tok_seg) memcpy(tok_seg, P->tok_seg.data(), n);
  if (tok_ver) memcpy(tok_ver, P->tok_ver.data(), n);
  if (drop_seg) memcpy(drop_seg, P->drop_seg.data(), n);
  return AKV_OK;
}

namespace {
akv_status check_run(const akv_plan *P, void *workspace, size_t workspace_bytes) {
  if (!P) return fail(AKV_ERR_INVALID, "plan is NULL");
  if (P->shape.dtype == AKV_BF16 && (P->shape.Hq / P->shape.Hkv) % 2)
    return fail(AKV_ERR_UNSUPPORTED,
                "bf16 prefill needs an even number of query heads per KV head");
  return check_ws(P, workspace, workspace_bytes);
}
}  // namespace

akv_status akv_segment_prepare(const akv_plan *P, const void *q, const void *k, const void *v,
                               void *workspace, size_t workspace_bytes, akv_stream_t stream) {
  AKV_ENTRY("akv_segment_prepare");
  if (!P) return fail(AKV_ERR_INVALID, "plan is NULL");
  if (P->T == 0) return AKV_OK;
  if (!q || !k || !v) return fail(AKV_ERR_INVALID, "NULL tensor");
  if (akv_status st = check_run(P, workspace, workspace_bytes)) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (akv_status st = upload_plan(P, workspace, s)) return st;
  RopeTheta th;
  rope_theta(P->shape.rope_base, &th);
  const PlanDev d = device_view(P, workspace);
  cudaError_t e = launch_prep(d, q, k, v, th, s);
  if (e == cudaSuccess && P->shape.dtype == AKV_BF16) e = launch_masks(d, s);
  if (e != cudaSuccess) return cuda_fail(e, "rope/permute pre-pass");
  return AKV_OK;
}

akv_status akv_segment_attend(const akv_plan *P, const void *q, void *out, void *workspace,
                              size_t workspace_bytes, akv_stream_t stream) {
  AKV_ENTRY("akv_segment_attend");
  if (!P) return fail(AKV_ERR_INVALID, "plan is NULL");
  if (P->T == 0) return AKV_OK;
  if (!out) return fail(AKV_ERR_INVALID, "NULL output");
  if (P->shape.dtype == AKV_BF16 && !q) return fail(AKV_ERR_INVALID, "NULL queries");
  if (akv_status st = check_run(P, workspace, workspace_bytes)) return st;
  PlanDev d = device_view(P, workspace);
  d.q = q;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = P->shape.dtype == AKV_F32 ? launch_attn_simt_f32(d, out, s)
                                            : launch_attn_tc_bf16(d, out, s);
  if (e != cudaSuccess) return cuda_fail(e, "segment attention");
  return AKV_OK;
}

akv_status akv_segment_attention_run(const akv_plan *P, const void *q, const void *k,
                                     const void *v, void *out, void *workspace,
                                     size_t workspace_bytes, akv_stream_t stream) {
  AKV_ENTRY("akv_segment_attention_run");
  if (!P) return fail(AKV_ERR_INVALID, "plan is NULL");
  if (P->T == 0) return AKV_OK;
  if (!q || !k || !v || !out) return fail(AKV_ERR_INVALID, "NULL tensor");
  if (akv_status st = check_run(P, workspace, workspace_bytes)) return st;
  if (akv_status st = akv_segment_prepare(P, q, k, v, workspace, workspace_bytes, stream))
    return st;
  return akv_segment_attend(P, q, out, workspace, workspace_bytes, stream);
}

size_t akv_segment_attention_workspace(const akv_shape *shape, int32_t n_req,
                                       const int32_t *cu_seqlens, const akv_oplog *ops) {
  akv_plan *P = nullptr;
  if (akv_plan_create(shape, n_req, cu_seqlens, nullptr, ops, &P) != AKV_OK) return 0;
  size_t r = P->ws.total;
  akv_plan_destroy(P);
  return r;
}

akv_status akv_segment_attention(const akv_shape *shape, int32_t n_req, const int32_t *cu_seqlens,
                                 const int32_t *logical_idx, const akv_oplog *ops, const void *q,
                                 const void *k, const void *v, void *out, void *workspace,
                                 size_t workspace_bytes, akv_stream_t stream) {
  akv_plan *P = nullptr;
  akv_status st = akv_plan_create(shape, n_req, cu_seqlens, logical_idx, ops, &P);
  if (st != AKV_OK) return st;
  st = akv_segment_attention_run(P, q, k, v, out, workspace, workspace_bytes, stream);
  akv_plan_destroy(P);
  return st;
}

akv_status akv_segment_visible_counts(const akv_plan *P, int32_t *counts, void *workspace,
                                      size_t workspace_bytes, akv_stream_t stream) {
  if (!P || !counts) return fail(AKV_ERR_INVALID, "NULL argument");
  if (P->T == 0) return AKV_OK;
  if (akv_status st = check_ws(P, workspace, workspace_bytes)) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (akv_status st = upload_plan(P, workspace, s)) return st;
  cudaError_t e = launch_visible_counts(device_view(P, workspace), counts, s);
  if (e != cudaSuccess) return cuda_fail(e, "visible counts");
  return AKV_OK;
}

akv_status akv_workspace_status(void *workspace, akv_stream_t stream, uint32_t *code) {
  if (!workspace || !code) return fail(AKV_ERR_INVALID, "NULL argument");
  cudaStream_t s = (cudaStream_t)stream;
  uint32_t h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, workspace, 4, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, 4, s);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  *code = h;
  if (h) return fail(AKV_ERR_DEVICE, "kernel status word 0x%x", h);
  return AKV_OK;
}

// ------------------------------------------------------------------------
// Compaction
// ------------------------------------------------------------------------

namespace {
struct CompactHost {
  int32_t upto, n_msgs, T_upto, br_end, r, has_br;
  std::vector<uint8_t> keep, alive_br;
  int64_t n_active;
};

akv_status compact_host(const akv_oplog *o, int32_t upto, CompactHost *c) {
  const int n = o->n_msgs;
  if (upto < 0) upto = n - 1;
  if (n == 0) {
    c->upto = -1;
    c->n_msgs = 0;
    c->T_upto = 0;
    c->br_end = 0;
    c->r = 0;
    c->has_br = 0;
    c->n_active = 0;
    return AKV_OK;
  }
  if (upto >= n) return fail(AKV_ERR_INVALID, "boundary %d out of range", upto);
  c->upto = upto;
  c->n_msgs = upto + 1;
  c->T_upto = o->msg_start[upto + 1];
  // first drop boundary of each message, and repos boundaries before upto
  std::vector<int> first_drop(n, INT32_MAX);
  for (int i = 0; i < o->n_drops; ++i)
    first_drop[o->drop_target[i]] = std::min(first_drop[o->drop_target[i]], o->drop_after[i]);
  int br = -1;
  for (int i = 0; i < o->n_repos; ++i)
    if (o->repos_after[i] < upto) br = std::max(br, o->repos_after[i]);
  c->keep.assign(upto + 1, 0);
  c->alive_br.assign(upto + 1, 0);
  c->n_active = 0;
  c->r = 0;
  for (int m = 0; m <= upto; ++m) {
    c->keep[m] = first_drop[m] > upto;
    if (c->keep[m]) c->n_active += o->msg_start[m + 1] - o->msg_start[m];
    if (br >= 0 && m <= br) {
      c->alive_br[m] = first_drop[m] > br;
      if (c->alive_br[m]) c->r += o->msg_start[m + 1] - o->msg_start[m];
    }
  }
  c->has_br = br >= 0;
  c->br_end = br >= 0 ? o->msg_start[br + 1] : 0;
  return AKV_OK;
}

size_t compact_ws_bytes(int n_msgs, int T) {
  return align_up(4 * (size_t)(n_msgs + 1), 256) + 2 * align_up((size_t)n_msgs + 1, 256) +
         align_up(8 * (size_t)compact_blocks(T), 256);
}
}  // namespace

namespace {
// Survivors after the drops of boundary `upto`, as runs of kept messages:
// first row, first compacted index (exclusive prefix of kept lengths, with
// the total appended), position of the first row in the version current
// before any repos at `upto`.
void kept_runs(const akv_oplog *o, const CompactHost &c, std::vector<int32_t> *kstart,
               std::vector<int32_t> *kprefix, std::vector<int32_t> *kpos) {
  int32_t j = 0, alive_base = 0;
  for (int m = 0; m < c.n_msgs; ++m) {
    const int32_t a = o->msg_start[m], len = o->msg_start[m + 1] - a;
    int32_t pos0;
    if (!c.has_br) pos0 = a;
    else if (a < c.br_end) pos0 = alive_base;  // renumbered by the last earlier repos
    else pos0 = c.r + (a - c.br_end);
    if (c.has_br && a < c.br_end && c.alive_br[m]) alive_base += len;
    if (!c.keep[m] || len == 0) continue;
    kstart->push_back(a);
    kprefix->push_back(j);
    kpos->push_back(pos0);
    j += len;
  }
  kprefix->push_back(j);
}
}  // namespace

size_t akv_compact_workspace(const akv_oplog *ops, int32_t T) {
  if (!ops || ops->n_msgs < 0) return 0;
  return compact_ws_bytes(ops->n_msgs, T);
}

akv_status akv_compact(const akv_oplog *ops, int32_t T, int32_t upto, int32_t *active_idx,
                       int32_t *active_pos, int32_t *n_active, void *workspace,
                       size_t workspace_bytes, akv_stream_t stream) {
  AKV_ENTRY("akv_compact");
  if (akv_status st = check_oplog(ops, T, 0)) return st;
  if (!n_active || !active_idx || !active_pos) return fail(AKV_ERR_INVALID, "NULL output");
  CompactHost c;
  if (akv_status st = compact_host(ops, upto, &c)) return st;
  *n_active = (int32_t)c.n_active;
  if (c.T_upto == 0) return AKV_OK;
  const size_t need = compact_ws_bytes(ops->n_msgs, T);
  if (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < need)
    return fail(AKV_ERR_WORKSPACE, "compact workspace: need %zu aligned bytes", need);
  if (c.n_active == 0) return AKV_OK;
  cudaStream_t s = (cudaStream_t)stream;
  {
    std::vector<int32_t> kstart, kprefix, kpos;
    kept_runs(ops, c, &kstart, &kprefix, &kpos);
    const int nk = (int)kstart.size();
    if (nk <= repos_inline_runs()) {  // one launch, the run tables in its parameters
      cudaError_t e = launch_compact_runs((int)c.n_active, nk, kstart.data(), kprefix.data(),
                                          kpos.data(), active_idx, active_pos, s);
      if (e != cudaSuccess) return cuda_fail(e, "compact");
      return AKV_OK;
    }
  }
  char *b = (char *)workspace;
  size_t o0 = 0, o1 = align_up(4 * (size_t)(ops->n_msgs + 1), 256);
  size_t o2 = o1 + align_up((size_t)ops->n_msgs + 1, 256);
  size_t o3 = o2 + align_up((size_t)ops->n_msgs + 1, 256);
  const HostPart parts[] = {{o0, ops->msg_start, 4 * (size_t)(c.n_msgs + 1)},
                            {o1, c.keep.data(), (size_t)c.n_msgs},
                            {o2, c.alive_br.data(), (size_t)c.n_msgs}};
  cudaError_t e = upload_async(b, parts, 3, s);
  if (e != cudaSuccess) return cuda_fail(e, "compact upload");
  CompactDev d{};
  d.msg_start = (const int32_t *)(b + o0);
  d.keep = (const uint8_t *)(b + o1);
  d.alive_br = (const uint8_t *)(b + o2);
  d.block_cnt = (int32_t *)(b + o3);
  d.n_msgs = c.n_msgs;
  d.T = c.T_upto;
  d.br_end = c.br_end;
  d.r = c.r;
  d.has_br = c.has_br;
  e = launch_compact(d, active_idx, active_pos, s);
  if (e != cudaSuccess) return cuda_fail(e, "compact");
  return AKV_OK;
}


size_t akv_repos_boundary_workspace(const akv_oplog *ops, int32_t T) {
  if (!ops || ops->n_msgs < 0) return 0;
  (void)T;
  return align_up(4 * (3 * (size_t)ops->n_msgs + 1), 256);
}

akv_status akv_repos_boundary(const akv_shape *shape, const akv_oplog *ops, int32_t T,
                              int32_t upto, const void *k_in, const void *v_in, void *k_out,
                              void *v_out, int32_t *n_out, void *workspace,
                              size_t workspace_bytes, akv_stream_t stream) {
  AKV_ENTRY("akv_repos_boundary");
  if (akv_status st = check_shape(shape)) return st;
  if (akv_status st = check_oplog(ops, T, 0)) return st;
  if (!n_out) return fail(AKV_ERR_INVALID, "n_out is NULL");
  CompactHost c;
  if (akv_status st = compact_host(ops, upto, &c)) return st;
  *n_out = (int32_t)c.n_active;
  if (c.n_active == 0) return AKV_OK;
  if (!k_in || !v_in || !k_out || !v_out) return fail(AKV_ERR_INVALID, "NULL tensor");
  const size_t need = 4 * (3 * (size_t)ops->n_msgs + 1);
  if (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < need)
    return fail(AKV_ERR_WORKSPACE, "repos workspace: need %zu aligned bytes", need);
  std::vector<int32_t> kstart, kprefix, kpos;
  kept_runs(ops, c, &kstart, &kprefix, &kpos);
  const int nk = (int)kstart.size();
  if (nk >= 1 && nk <= repos_inline_runs()) {  // the tables travel with the launch
    RopeTheta th;
    rope_theta(shape->rope_base, &th);
    cudaError_t e = launch_repos_boundary_inline(shape->dtype, shape->Hkv, (int)c.n_active, nk,
                                                 kstart.data(), kprefix.data(), kpos.data(), k_in,
                                                 v_in, k_out, v_out, th, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "repos at boundary");
    return AKV_OK;
  }
  // one upload: [kstart | kprefix | kpos]
  std::vector<int32_t> packed;
  packed.reserve(3 * nk + 1);
  packed.insert(packed.end(), kstart.begin(), kstart.end());
  packed.insert(packed.end(), kprefix.begin(), kprefix.end());
  packed.insert(packed.end(), kpos.begin(), kpos.end());
  cudaStream_t s = (cudaStream_t)stream;
  int32_t *b = (int32_t *)workspace;
  const HostPart part{0, packed.data(), 4 * packed.size()};
  cudaError_t e = upload_async((char *)b, &part, 1, s);
  if (e != cudaSuccess) return cuda_fail(e, "repos tables upload");
  RopeTheta th;
  rope_theta(shape->rope_base, &th);
  e = launch_repos_boundary(shape->dtype, shape->Hkv, (int)c.n_active, nk, b, b + nk,
                            b + 2 * nk + 1, k_in, v_in, k_out, v_out, th, s);
  if (e != cudaSuccess) return cuda_fail(e, "repos at boundary");
  return AKV_OK;
}

// ------------------------------------------------------------------------
// Repos rotate, append, decode
// ------------------------------------------------------------------------

akv_status akv_repos_rotate(const akv_shape *shape, int32_t r, const int32_t *src_idx,
                            const int32_t *pos_from, const int32_t *pos_to, const void *k_in,
                            const void *v_in, void *k_out, void *v_out, akv_stream_t stream) {
  AKV_ENTRY("akv_repos_rotate");
  if (akv_status st = check_shape(shape)) return st;
  if (r < 0) return fail(AKV_ERR_INVALID, "r < 0");
  if (r == 0) return AKV_OK;
  if (!src_idx || !pos_from || !k_in || !v_in || !k_out || !v_out)
    return fail(AKV_ERR_INVALID, "NULL argument");
  RopeTheta th;
  rope_theta(shape->rope_base, &th);
  cudaError_t e = launch_repos(shape->dtype, shape->Hkv, r, src_idx, pos_from, pos_to, k_in, v_in,
                               k_out, v_out, th, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "repos rotate");
  return AKV_OK;
}

akv_status akv_append_kv(const akv_shape *shape, int32_t n, const void *k_new, const void *v_new,
                         const int32_t *pos, const int32_t *slot, void *k_pool, void *v_pool,
                         akv_stream_t stream) {
  AKV_ENTRY("akv_append_kv");
  if (akv_status st = check_shape(shape)) return st;
  if (n < 0) return fail(AKV_ERR_INVALID, "n < 0");
  if (n == 0) return AKV_OK;
  if (!k_new || !v_new || !pos || !slot || !k_pool || !v_pool)
    return fail(AKV_ERR_INVALID, "NULL argument");
  RopeTheta th;
  rope_theta(shape->rope_base, &th);
  cudaError_t e = launch_append(shape->dtype, shape->Hkv, n, k_new, v_new, pos, slot, k_pool,
                                v_pool, th, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "append");
  return AKV_OK;
}

size_t akv_decode_workspace(const akv_shape *shape, int32_t B, int32_t max_kv) {
  if (!shape || B < 0 || max_kv < 0 || shape->Hkv <= 0 || shape->Hq % shape->Hkv) return 0;
  return decode_workspace_bytes(B, shape->Hq, shape->Hkv, max_kv);
}

akv_status akv_decode_attention(const akv_shape *shape, int32_t B, const void *q,
                                const int32_t *q_pos, const void *k_pool, const void *v_pool,
                                const int32_t *kv_indptr, const int32_t *kv_indices,
                                int32_t max_kv, void *out, void *workspace, size_t workspace_bytes,
                                akv_stream_t stream) {
  AKV_ENTRY("akv_decode_attention");
  if (akv_status st = check_shape(shape)) return st;
  if (B < 0 || max_kv < 0) return fail(AKV_ERR_INVALID, "negative size");
  if (B > 65535) return fail(AKV_ERR_UNSUPPORTED, "decode supports B <= 65535");
  if (B == 0) return AKV_OK;
  if (!q || !q_pos || !k_pool || !v_pool || !kv_indptr || !out || (max_kv > 0 && !kv_indices))
    return fail(AKV_ERR_INVALID, "NULL argument");
  if (shape->dtype == AKV_BF16 && shape->Hq / shape->Hkv > 16)
    return fail(AKV_ERR_UNSUPPORTED, "bf16 decode supports up to 16 query heads per KV head");
  if (shape->dtype == AKV_BF16 && max_kv > kDecodeMaxKeys)
    return fail(AKV_ERR_UNSUPPORTED, "bf16 decode supports up to %d keys per request", kDecodeMaxKeys);
  const size_t need = decode_workspace_bytes(B, shape->Hq, shape->Hkv, max_kv);
  if (need && (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < need))
    return fail(AKV_ERR_WORKSPACE, "decode workspace: need %zu aligned bytes", need);
  RopeTheta th;
  rope_theta(shape->rope_base, &th);
  cudaError_t e = launch_decode(shape->dtype, B, shape->Hq, shape->Hkv, q, q_pos, k_pool, v_pool,
                                kv_indptr, kv_indices, max_kv, out, workspace, th,
                                (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode");
  return AKV_OK;
}

akv_status akv_decode_attention_append(const akv_shape *shape, int32_t B, const void *q,
                                       const int32_t *q_pos, const void *k_new,
                                       const void *v_new, const int32_t *new_slot, void *k_pool,
                                       void *v_pool, const int32_t *kv_indptr,
                                       const int32_t *kv_indices, int32_t max_kv, void *out,
                                       void *workspace, size_t workspace_bytes,
                                       akv_stream_t stream) {
  AKV_ENTRY("akv_decode_attention_append");
  if (akv_status st = check_shape(shape)) return st;
  if (B < 0 || max_kv < 0) return fail(AKV_ERR_INVALID, "negative size");
  if (B > 65535) return fail(AKV_ERR_UNSUPPORTED, "decode supports B <= 65535");
  if (B == 0) return AKV_OK;
  if (!q || !q_pos || !k_new || !v_new || !new_slot || !k_pool || !v_pool || !kv_indptr ||
      !out || (max_kv > 0 && !kv_indices))
    return fail(AKV_ERR_INVALID, "NULL argument");
  if (shape->dtype == AKV_BF16 && shape->Hq / shape->Hkv > 16)
    return fail(AKV_ERR_UNSUPPORTED, "bf16 decode supports up to 16 query heads per KV head");
  if (shape->dtype == AKV_BF16 && max_kv > kDecodeMaxKeys)
    return fail(AKV_ERR_UNSUPPORTED, "bf16 decode supports up to %d keys per request", kDecodeMaxKeys);
  const size_t need = decode_workspace_bytes(B, shape->Hq, shape->Hkv, max_kv);
  if (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < need)
    return fail(AKV_ERR_WORKSPACE, "decode workspace: need %zu aligned bytes", need);
  RopeTheta th;
  rope_theta(shape->rope_base, &th);
  cudaError_t e = launch_decode_append(shape->dtype, B, shape->Hq, shape->Hkv, q, q_pos, k_new,
                                       v_new, new_slot, k_pool, v_pool, kv_indptr, kv_indices,
                                       max_kv, out, workspace, th, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode with append");
  return AKV_OK;
}

size_t akv_decode_rope_workspace(const akv_shape *shape, int32_t B, int32_t max_kv) {
  if (!shape || B <= 0 || max_kv < 0) return 0;
  return decode_rope_workspace_bytes(shape->dtype, B, shape->Hq, shape->Hkv, max_kv);
}

akv_status akv_decode_attention_rope(const akv_shape *shape, int32_t B, const void *q,
                                     const int32_t *q_pos, const void *k_new, const void *v_new,
                                     const int32_t *new_slot, void *k_pool, void *v_pool,
                                     const int32_t *kv_indptr, const int32_t *kv_indices,
                                     const int32_t *kv_pos, int32_t max_kv, void *out,
                                     void *workspace, size_t workspace_bytes,
                                     akv_stream_t stream) {
  AKV_ENTRY("akv_decode_attention_rope");
  if (akv_status st = check_shape(shape)) return st;
  if (B < 0 || max_kv < 0) return fail(AKV_ERR_INVALID, "negative size");
  if (B > 65535) return fail(AKV_ERR_UNSUPPORTED, "decode supports B <= 65535");
  if (B == 0) return AKV_OK;
  if (!q || !q_pos || !k_pool || !v_pool || !kv_indptr || !out ||
      (max_kv > 0 && (!kv_indices || !kv_pos)))
    return fail(AKV_ERR_INVALID, "NULL argument");
  if ((new_slot == nullptr) != (k_new == nullptr) || (new_slot == nullptr) != (v_new == nullptr))
    return fail(AKV_ERR_INVALID, "k_new, v_new and new_slot are given together or not at all");
  if (shape->dtype == AKV_BF16 && shape->Hq / shape->Hkv > 16)
    return fail(AKV_ERR_UNSUPPORTED, "bf16 decode supports up to 16 query heads per KV head");
  if (shape->dtype == AKV_BF16 && max_kv > kDecodeMaxKeys)
    return fail(AKV_ERR_UNSUPPORTED, "bf16 decode supports up to %d keys per request", kDecodeMaxKeys);
  const size_t need = decode_rope_workspace_bytes(shape->dtype, B, shape->Hq, shape->Hkv, max_kv);
  if (need && (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < need))
    return fail(AKV_ERR_WORKSPACE, "decode (rotate on read) workspace: need %zu aligned bytes", need);
  RopeTheta th;
  rope_theta(shape->rope_base, &th);
  cudaError_t e = launch_decode_rope(shape->dtype, B, shape->Hq, shape->Hkv, q, q_pos, k_new,
                                     v_new, new_slot, k_pool, v_pool, kv_indptr, kv_indices,
                                     kv_pos, max_kv, out, workspace, th, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode (rotate on read)");
  return AKV_OK;
}

akv_status akv_decode_attention_static(const akv_shape *shape, int32_t B, const void *q,
                                       const int32_t *q_pos, const void *k_pool,
                                       const void *v_pool, const int32_t *kv_indptr,
                                       const int32_t *kv_indices, int32_t max_kv, void *out,
                                       akv_stream_t stream) {
  AKV_ENTRY("akv_decode_attention_static");
  if (akv_status st = check_shape(shape)) return st;
  if (B < 0 || max_kv < 0) return fail(AKV_ERR_INVALID, "negative size");
  if (B > 65535) return fail(AKV_ERR_UNSUPPORTED, "decode supports B <= 65535");
  if (B == 0) {  // set-up only: loads the module that holds the array
    void *scratch = nullptr;
    const cudaError_t e = decode_static_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail(e, "static decode scratch look-up");
    return AKV_OK;
  }
  if (!q || !q_pos || !k_pool || !v_pool || !kv_indptr || !out || (max_kv > 0 && !kv_indices))
    return fail(AKV_ERR_INVALID, "NULL argument");
  if (shape->dtype == AKV_BF16 && shape->Hq / shape->Hkv > 16)
    return fail(AKV_ERR_UNSUPPORTED, "bf16 decode supports up to 16 query heads per KV head");
  if (shape->dtype == AKV_BF16 && max_kv > kDecodeMaxKeys)
    return fail(AKV_ERR_UNSUPPORTED, "bf16 decode supports up to %d keys per request", kDecodeMaxKeys);
  const size_t need = decode_workspace_bytes(B, shape->Hq, shape->Hkv, max_kv);
  if (need > kStaticScratchBytes)
    return fail(AKV_ERR_UNSUPPORTED,
                "akv_decode_attention_static: B=%d, Hq=%d, max_kv=%d need %zu bytes of split-KV "
                "partials but the static scratch holds %zu; use akv_decode_attention with a "
                "workspace",
                B, shape->Hq, max_kv, need, kStaticScratchBytes);
  RopeTheta th;
  rope_theta(shape->rope_base, &th);
  cudaError_t e = launch_decode_static(shape->dtype, B, shape->Hq, shape->Hkv, q, q_pos, k_pool,
                                       v_pool, kv_indptr, kv_indices, max_kv, out, th,
                                       (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode (static scratch)");
  return AKV_OK;
}

size_t akv_decode_static_scratch_bytes(void) { return kStaticScratchBytes; }

akv_status akv_decode_check_indices(int32_t B, const int32_t *kv_indptr, const int32_t *kv_indices,
                                    int32_t n_indices, int32_t S, int32_t max_kv, uint32_t *status,
                                    akv_stream_t stream) {
  AKV_ENTRY("akv_decode_check_indices");
  if (B < 0 || n_indices < 0 || S < 0 || max_kv < 0) return fail(AKV_ERR_INVALID, "negative size");
  if (!kv_indptr || !status || (n_indices > 0 && !kv_indices))
    return fail(AKV_ERR_INVALID, "NULL argument");
  if (B == 0) return AKV_OK;
  cudaError_t e = launch_check_indices(B, kv_indptr, kv_indices, S, max_kv, n_indices, status,
                                       (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode index check");
  return AKV_OK;
}

// ------------------------------------------------------------------------
// Decoder layers around the segment attention
// ------------------------------------------------------------------------

akv_status akv_gemm_bf16(int32_t M, int32_t N, int32_t K, const void *x, const void *w, void *y,
                         int32_t out_mode, akv_stream_t stream) {
  AKV_ENTRY("akv_gemm_bf16");
  if (M < 0 || N < 0 || K <= 0 || out_mode < 0 || out_mode > 2)
    return fail(AKV_ERR_INVALID, "bad GEMM arguments");
  if (N % 32 || K % 8)
    return fail(AKV_ERR_UNSUPPORTED, "GEMM needs N %% 32 == 0 and K %% 8 == 0 (N=%d K=%d)", N, K);
  if ((int64_t)M * 1 >= (int64_t)1 << 31) return fail(AKV_ERR_UNSUPPORTED, "M too large");
  if (M == 0 || N == 0) return AKV_OK;
  if (!x || !w || !y) return fail(AKV_ERR_INVALID, "NULL argument");
  if ((uintptr_t)x % 16 || (uintptr_t)w % 16 || (uintptr_t)y % 16)
    return fail(AKV_ERR_INVALID, "GEMM operands must be 16-byte aligned");
  cudaError_t e = launch_gemm(M, N, K, x, w, y, out_mode, nullptr, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "gemm");
  return AKV_OK;
}

akv_status akv_rmsnorm(int32_t rows, int32_t d, float eps, akv_dtype in_dtype, const void *x,
                       const float *weight, akv_dtype out_dtype, void *y, akv_stream_t stream) {
  AKV_ENTRY("akv_rmsnorm");
  if (rows < 0 || d <= 0 || !(eps >= 0.f)) return fail(AKV_ERR_INVALID, "bad rmsnorm arguments");
  if (rows == 0) return AKV_OK;
  if (!x || !y) return fail(AKV_ERR_INVALID, "NULL argument");
  cudaError_t e = launch_rmsnorm(rows, d, eps, in_dtype == AKV_F32, x, weight, out_dtype == AKV_F32,
                                 y, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "rmsnorm");
  return AKV_OK;
}

akv_status akv_swiglu(int64_t n, const void *g, const void *u, void *out, akv_stream_t stream) {
  AKV_ENTRY("akv_swiglu");
  if (n < 0) return fail(AKV_ERR_INVALID, "n < 0");
  if (n == 0) return AKV_OK;
  if (!g || !u || !out) return fail(AKV_ERR_INVALID, "NULL argument");
  cudaError_t e = launch_swiglu(n, g, u, out, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "swiglu");
  return AKV_OK;
}

namespace {
struct DecoderLayout {
  size_t h, a, q, k, v, o, g, u, wgu, attn, total;
};
DecoderLayout decoder_layout(const akv_plan *P, int d_model, int d_ff) {
  DecoderLayout L{};
  const size_t T = (size_t)P->T;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    off = align_up(off, 1024);
    size_t r = off;
    off += bytes;
    return r;
  };
  L.attn = take(P->ws.total);  // first: its status word starts the workspace
  L.h = take(4 * T * d_model);
  L.a = take(2 * T * d_model);
  L.q = take(2 * T * P->shape.Hq * kD);
  L.k = take(2 * T * P->shape.Hkv * kD);
  L.v = take(2 * T * P->shape.Hkv * kD);
  L.o = take(2 * T * P->shape.Hq * kD);
  L.g = take(2 * T * d_ff);
  // d_ff a multiple of 128: gate and up run as one GEMM with a SwiGLU
  // epilogue over interleaved weights ([2 d_ff][d_model]); otherwise as two
  // GEMMs into g and u, then SwiGLU
  if (d_ff % 128 == 0) L.wgu = take(2 * 2 * (size_t)d_ff * d_model);
  else L.u = take(2 * T * d_ff);
  L.total = align_up(off, 1024);
  return L;
}
}  // namespace

size_t akv_decoder_workspace(const akv_plan *P, int32_t d_model, int32_t d_ff) {
  if (!P || d_model <= 0 || d_ff <= 0) return 0;
  return decoder_layout(P, d_model, d_ff).total;
}

akv_status akv_decoder_forward(const akv_plan *P, int32_t n_layers, const akv_layer_weights *layers,
                               int32_t d_model, int32_t d_ff, float eps, const void *x, float *out,
                               void *workspace, size_t workspace_bytes, akv_stream_t stream) {
  AKV_ENTRY("akv_decoder_forward");
  if (!P || n_layers < 0 || (n_layers > 0 && !layers) || d_model <= 0 || d_ff <= 0 || !x || !out)
    return fail(AKV_ERR_INVALID, "bad decoder arguments");
  if (P->shape.dtype != AKV_BF16) return fail(AKV_ERR_UNSUPPORTED, "decoder layers run in bf16");
  if (d_model % 32 || d_ff % 32)
    return fail(AKV_ERR_UNSUPPORTED, "d_model and d_ff must be multiples of 32");
  for (int l = 0; l < n_layers; ++l) {
    const akv_layer_weights &w = layers[l];
    if (!w.wq || !w.wk || !w.wv || !w.wo || !w.wg || !w.wu || !w.wd)
      return fail(AKV_ERR_INVALID, "layer %d: NULL weight", l);
  }
  const DecoderLayout L = decoder_layout(P, d_model, d_ff);
  if (!workspace || (uintptr_t)workspace % 256 || workspace_bytes < L.total)
    return fail(AKV_ERR_WORKSPACE, "decoder workspace: need %zu aligned bytes", L.total);
  if (P->T == 0) return AKV_OK;
  cudaStream_t s = (cudaStream_t)stream;
  char *b = (char *)workspace;
  float *h = (float *)(b + L.h);
  void *a = b + L.a, *q = b + L.q, *k = b + L.k, *v = b + L.v, *o = b + L.o, *g = b + L.g,
       *u = b + L.u, *wgu = b + L.wgu, *aws = b + L.attn;
  const bool fused_ffn = d_ff % 128 == 0;
  const int T = (int)P->T, dq = P->shape.Hq * kD, dkv = P->shape.Hkv * kD;
  uint32_t *status = (uint32_t *)((char *)aws + P->ws.status);
  // The kernels' bounded waits stop waiting once this word is nonzero (a
  // timeout elsewhere in the launch); a reused workspace may hold any value,
  // so clear it before the first GEMM reads it.
  cudaError_t e = cudaMemsetAsync(status, 0, 256, s);
  if (e == cudaSuccess) e = launch_widen((int64_t)T * d_model, x, h, s);
#define AKV_TRY(call, what)                       \
  do {                                            \
    if (e == cudaSuccess) e = (call);             \
    if (e != cudaSuccess) return cuda_fail(e, what); \
  } while (0)
  AKV_TRY(cudaSuccess, "widen");
  for (int l = 0; l < n_layers; ++l) {
    const akv_layer_weights &w = layers[l];
    AKV_TRY(launch_rmsnorm(T, d_model, eps, 1, h, nullptr, 0, a, s), "rmsnorm");
    AKV_TRY(launch_gemm(T, dq, d_model, a, w.wq, q, 0, status, s), "q projection");
    AKV_TRY(launch_gemm(T, dkv, d_model, a, w.wk, k, 0, status, s), "k projection");
    AKV_TRY(launch_gemm(T, dkv, d_model, a, w.wv, v, 0, status, s), "v projection");
    if (akv_status st = akv_segment_attention_run(P, q, k, v, o, aws, P->ws.total, stream))
      return st;
    AKV_TRY(launch_gemm(T, d_model, dq, o, w.wo, h, 2, status, s), "output projection");
    AKV_TRY(launch_rmsnorm(T, d_model, eps, 1, h, nullptr, 0, a, s), "rmsnorm");
    if (fused_ffn) {  // gate and up as one GEMM, SwiGLU in its epilogue
      AKV_TRY(launch_interleave_gu(w.wg, w.wu, wgu, d_ff, d_model, s), "gate/up interleave");
      AKV_TRY(launch_gemm(T, 2 * d_ff, d_model, a, wgu, g, 3, status, s), "gate/up projection");
    } else {
      AKV_TRY(launch_gemm(T, d_ff, d_model, a, w.wg, g, 0, status, s), "gate projection");
      AKV_TRY(launch_gemm(T, d_ff, d_model, a, w.wu, u, 0, status, s), "up projection");
      AKV_TRY(launch_swiglu((int64_t)T * d_ff, g, u, g, s), "swiglu");
    }
    AKV_TRY(launch_gemm(T, d_model, d_ff, g, w.wd, h, 2, status, s), "down projection");
  }
  AKV_TRY(launch_rmsnorm(T, d_model, eps, 1, h, nullptr, 1, out, s), "final rmsnorm");
#undef AKV_TRY
  return AKV_OK;
}

}  // extern "C"
