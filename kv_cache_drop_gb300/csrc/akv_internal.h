// Internal declarations shared by the host planner / C ABI and the CUDA
// launchers.  Nothing here is part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "akv.h"

namespace akv {

constexpr int kD = 64;          // head dim supported by every kernel
constexpr int kTileQ = 128;     // query rows per tile (tcgen05 M)
constexpr int kTileK = 128;     // keys per window (tcgen05 N of Q K^T)
constexpr int kSlotPad = 128;   // padding entries after the slot tables
constexpr uint32_t kWinFull = 0x80000000u;  // window flag: no in-tile mask needed
constexpr uint32_t kStatusWaitTimeout = 1u; // status bit: a barrier wait gave up
constexpr uint32_t kStatusFp16Range = 2u;   // status bit: a rotated Q/K value exceeded fp16

// One query tile: rows [t0, t0+len) of one request, all in one key version.
struct QTile {
  int32_t t0;       // first row (batch-global)
  int32_t len;      // 1..kTileQ
  int32_t ver;      // key version read by these rows
  int32_t req;      // request index
  int32_t win_off;  // first entry in the window array
  int32_t win_cnt;  // number of 128-key windows
  int32_t seg_lo;   // segment of row t0 (request-relative)
  int32_t seg_hi;   // segment of the last row
  int32_t pm_off;   // first visibility-mask block of the tile's partial windows
  int32_t pm_cnt;   // number of partial (masked) windows
  int32_t pad[2];
};
static_assert(sizeof(QTile) == 48, "QTile layout");

// A window that needs an in-tile mask: its rows' visibility bits are
// precomputed once per plan (they do not depend on the head) into a block of
// 128 rows x 128 bits, bit j of row r = key slot (slot0 + j) visible to row
// (t0 + r).
struct MaskWin {
  int32_t t0;     // first row of the query tile (batch-global)
  int32_t len;    // rows in the tile
  int32_t slot0;  // first key slot of the window
  int32_t pad;
};

// Device views of the plan tables and the rotated copies, all inside one
// caller workspace.
struct PlanDev {
  uint32_t *status;          // workspace status word
  const int32_t *tok_qpos;   // [T] query position (append position) of each row
  const int32_t *tok_seg;    // [T] segment of each row
  const int32_t *slot_src;   // [T] permuted key slot -> source row
  const int32_t *slot_u;     // [T+pad] permuted key slot -> batch-global logical row (pad INT_MAX)
  const int32_t *slot_dseg;  // [T+pad] first segment that no longer sees the slot (pad INT_MIN)
  const int32_t *slot_pos;   // [max_ver][T] position of the slot's key in each version
  const QTile *qtiles;       // [n_qtiles]
  const uint32_t *windows;   // [n_windows] slot start | kWinFull
  const MaskWin *mwin;       // [n_mask] partial windows, in tile then window order
  uint4 *mask;               // [n_mask][128 rows] visibility bits (words = keys 0-31, ..)
  const int32_t *order;      // [n_qtiles] tiles by decreasing window count
  void *qr;                  // fp32: [Hq][T][D] rotated queries, head-major (bf16: unused)
  float2 *qcs;               // bf16: [T][D/2] cos/sin of each row's query angles
  const void *q;             // bf16: the raw queries [T][Hq][D] (set for the attention)
  void *kr;                  // [max_ver][Hkv][T][D] rotated keys, permuted slots, head-major
                             // (fp16 for bf16 inputs)
  void *vp;                  // [Hkv][T][D] values, permuted slots, head-major
                             // (fp16 for bf16 inputs)
  int64_t T;
  int32_t n_qtiles;
  int32_t n_mask;
  int32_t max_ver;
  int32_t Hq, Hkv;
  float rope_base;
  int32_t dtype;             // akv_dtype
};

// RoPE frequencies theta_i = base^(-2i/D), computed in double on the host,
// also as an unevaluated float pair hi + lo (hi = fl(theta), lo = fl(theta - hi)).
struct RopeTheta {
  double th[kD / 2];
  float hi[kD / 2];
  float lo[kD / 2];
};

void rope_theta(float base, RopeTheta *out);

// ---- host helpers shared by the C-ABI translation units (api.cpp) ----
// Records the message returned by akv_last_error and returns st.
akv_status report_error(akv_status st, const char *fmt, ...);
// Validates an op log (msg_start CSR, drop/repos boundaries and targets);
// T < 0 skips the row-count check.
akv_status validate_oplog(const akv_oplog *o, int64_t T, int req);
// AKV_FAULT injection for host tests (AKV_OK when not injected).
akv_status fault_point(const char *entry);

// ---- launchers (defined in the .cu files) ----
cudaError_t launch_prep(const PlanDev &p, const void *q, const void *k, const void *v,
                        const RopeTheta &th, cudaStream_t s);
cudaError_t launch_attn_simt_f32(const PlanDev &p, void *out, cudaStream_t s);
cudaError_t launch_visible_counts(const PlanDev &p, int32_t *counts, cudaStream_t s);
cudaError_t launch_attn_tc_bf16(const PlanDev &p, void *out, cudaStream_t s);
cudaError_t launch_masks(const PlanDev &p, cudaStream_t s);
cudaError_t launch_repos(int dtype, int Hkv, int r, const int32_t *src, const int32_t *pf,
                         const int32_t *pt, const void *kin, const void *vin, void *kout,
                         void *vout, const RopeTheta &th, cudaStream_t s);
cudaError_t launch_append(int dtype, int Hkv, int n, const void *kn, const void *vn,
                          const int32_t *pos, const int32_t *slot, void *kp, void *vp,
                          const RopeTheta &th, cudaStream_t s);

cudaError_t launch_repos_boundary(int dtype, int Hkv, int r, int nk, const int32_t *kstart,
                                  const int32_t *kprefix, const int32_t *kpos, const void *kin,
                                  const void *vin, void *kout, void *vout, const RopeTheta &th,
                                  cudaStream_t s);
// the same with the run tables in the kernel's parameters (nk <= repos_inline_runs())
int repos_inline_runs();
cudaError_t launch_repos_boundary_inline(int dtype, int Hkv, int r, int nk, const int32_t *kstart,
                                         const int32_t *kprefix, const int32_t *kpos,
                                         const void *kin, const void *vin, void *kout, void *vout,
                                         const RopeTheta &th, cudaStream_t s);

struct CompactDev {
  const int32_t *msg_start;  // [n_msgs+1]
  const uint8_t *keep;       // [n_msgs] message survives the drops up to the boundary
  const uint8_t *alive_br;   // [n_msgs] message alive right after the last earlier repos
  int32_t *block_cnt;        // [2 * n_blocks] kept / alive counts per block
  int32_t n_msgs;
  int32_t T;                 // tokens in messages <= boundary
  int32_t br_end;            // first token after the last earlier repos (0 if none)
  int32_t r;                 // survivors at that repos
  int32_t has_br;
};
cudaError_t launch_compact(const CompactDev &c, int32_t *active_idx, int32_t *active_pos,
                           cudaStream_t s);
int compact_blocks(int T);
// the same from the kept runs (host tables, nk <= repos_inline_runs(), n >= 1
// compacted entries), one launch with the tables in its parameters
cudaError_t launch_compact_runs(int n, int nk, const int32_t *kstart, const int32_t *kprefix,
                                const int32_t *kpos, int32_t *active_idx, int32_t *active_pos,
                                cudaStream_t s);

// Small host tables delivered as the parameters of a copy kernel on the
// stream: a launch costs far less latency than starting the copy engine for
// a few hundred bytes.  Segment s copies seg[s].bytes bytes from
// data + seg[s].src_off to dst + seg[s].dst_off.
constexpr int kParamBlobBytes = 3840;
constexpr int kParamMaxSegs = 8;
struct ParamSeg {
  uint32_t dst_off, src_off, bytes;
};
struct ParamBlob {
  int32_t n_seg;
  ParamSeg seg[kParamMaxSegs];
  alignas(16) uint8_t data[kParamBlobBytes];
};
static_assert(sizeof(ParamBlob) + sizeof(void *) <= 4096, "kernel parameter space");
cudaError_t launch_param_upload(char *dst, const ParamBlob &blob, cudaStream_t s);

// Larger host tables staged in mapped pinned memory, copied by a kernel that
// reads the host block directly (the copy engine queues behind unrelated
// copies, e.g. a caller's input transfer on another stream).
constexpr int kUploadMaxSegs = 16;
struct UploadSegs {
  int32_t n;
  ParamSeg seg[kUploadMaxSegs];
};
cudaError_t launch_mapped_upload(const void *src_dev, char *dst, const UploadSegs &segs,
                                 cudaStream_t s);

size_t decode_partials_bytes(int B, int Hq, int max_kv, bool rope = false);
// partials + the per-(request, KV head) merge counters of the bf16 kernel
size_t decode_workspace_bytes(int B, int Hq, int Hkv, int max_kv);
size_t decode_rope_workspace_bytes(int dtype, int B, int Hq, int Hkv, int max_kv);
cudaError_t launch_decode_append(int dtype, int B, int Hq, int Hkv, const void *q,
                                 const int32_t *qpos, const void *k_new, const void *v_new,
                                 const int32_t *new_slot, void *kp, void *vp,
                                 const int32_t *indptr, const int32_t *indices, int max_kv,
                                 void *out, void *ws, const RopeTheta &th, cudaStream_t s);
cudaError_t launch_decode_rope(int dtype, int B, int Hq, int Hkv, const void *q,
                               const int32_t *qpos, const void *k_new, const void *v_new,
                               const int32_t *new_slot, void *kp, void *vp, const int32_t *indptr,
                               const int32_t *indices, const int32_t *kvpos, int max_kv, void *out,
                               void *ws, const RopeTheta &th, cudaStream_t s);
cudaError_t launch_decode(int dtype, int B, int Hq, int Hkv, const void *q, const int32_t *qpos,
                          const void *kp, const void *vp, const int32_t *indptr,
                          const int32_t *indices, int max_kv, void *out, void *ws,
                          const RopeTheta &th, cudaStream_t s);

// Decoder-layer pieces (GEMM: out_mode 0 bf16, 1 fp32, 2 fp32 +=)
cudaError_t launch_gemm(int M, int N, int K, const void *x, const void *w, void *y, int out_mode,
                        uint32_t *status, cudaStream_t s);
cudaError_t launch_rmsnorm(int rows, int d, float eps, int in_f32, const void *x, const float *w,
                           int out_f32, void *y, cudaStream_t s);
cudaError_t launch_swiglu(int64_t n, const void *g, const void *u, void *out, cudaStream_t s);
// gate [d_ff][K] and up [d_ff][K] into [2 d_ff][K] with 128-row blocks
// alternating, for the SwiGLU GEMM (out_mode 3); d_ff % 128 == 0, K % 8 == 0
cudaError_t launch_interleave_gu(const void *wg, const void *wu, void *wgu, int d_ff, int K,
                                 cudaStream_t s);
cudaError_t launch_widen(int64_t n, const void *x, float *y, cudaStream_t s);

// Decode with its split-KV partials in a static device array (no workspace).
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
// akv_decode_check_indices status bits
constexpr uint32_t kDecodeIndptr = 1u;  // indptr[0] != 0, a negative or > max_kv length, or too many entries
constexpr uint32_t kDecodeSlot = 2u;    // a slot outside [0, S)
cudaError_t launch_check_indices(int B, const int32_t *indptr, const int32_t *indices, int S,
                                 int max_kv, int64_t nnz_cap, uint32_t *status, cudaStream_t s);
// bf16 decode: the in-kernel split merge keeps one weight per split and query
// head of a group in shared memory (<= 1000 splits of 2048 keys)
constexpr int kDecodeMaxKeys = 1000 * 2048;
cudaError_t decode_static_scratch(void **ptr);
cudaError_t launch_decode_static(int dtype, int B, int Hq, int Hkv, const void *q,
                                 const int32_t *qpos, const void *kp, const void *vp,
                                 const int32_t *indptr, const int32_t *indices, int max_kv,
                                 void *out, const RopeTheta &th, cudaStream_t s);

}  // namespace akv
