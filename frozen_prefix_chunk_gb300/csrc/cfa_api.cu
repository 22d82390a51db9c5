// C-ABI boundary of the cfa library: argument validation, work planning,
// workspace carve-up, TMA descriptor encoding and kernel launches.  Nothing
// here allocates device memory or synchronises (except cfa_read_status).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "cfa.h"
#include "cfa_kernels.cuh"

using namespace cfa;

namespace {

constexpr size_t kWsHeader = 256;      // status word + padding
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// bf16 tensor [rows, heads, d] -> 3-D map with boxes of 64 columns x box_h
// heads x box_t rows, 128-byte swizzle (the UMMA K-major / MN-major canonical
// layout).  Rows beyond the tensor read as zero.
int make_map_bf16(CUtensorMap* m, const void* ptr, int d, int heads, long long rows, int box_h,
                  int box_t) {
  std::memset(m, 0, sizeof(*m));
  if (rows <= 0) return CFA_OK;  // never dereferenced
  EncodeTiledFn fn = encode_fn();
  if (!fn) return CFA_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
  cuuint32_t box[3] = {64u, (cuuint32_t)box_h, (cuuint32_t)box_t};
  cuuint32_t es[3] = {1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CFA_OK : CFA_ERR_INVALID_ARG;
}

int validate(const cfa_args* a) {
  if (!a) return CFA_ERR_INVALID_ARG;
  if (a->batch < 1 || a->batch > 65535) return CFA_ERR_INVALID_ARG;
  if (a->hq < 1 || a->hkv < 1 || a->hkv > 65535 || a->hq % a->hkv != 0) return CFA_ERR_INVALID_ARG;
  if (a->hq / a->hkv > 128 || a->hq > 65535) return CFA_ERR_UNSUPPORTED;
  if (a->head_dim != 64 && a->head_dim != 128) return CFA_ERR_UNSUPPORTED;
  if (a->prefix_dtype != CFA_PREFIX_BF16 && a->prefix_dtype != CFA_PREFIX_Q8_0 &&
      a->prefix_dtype != CFA_PREFIX_F16)
    return CFA_ERR_INVALID_ARG;
  if (a->max_lp < 0 || a->max_lc < 0 || a->total_lp < 0 || a->total_lc < 0)
    return CFA_ERR_INVALID_ARG;
  if (a->max_lp > a->total_lp || a->max_lc > a->total_lc) return CFA_ERR_INVALID_ARG;
  if (!(a->softmax_scale > 0.f) || !std::isfinite(a->softmax_scale)) return CFA_ERR_INVALID_ARG;
  if (!a->cu_seqlens_prefix || !a->cu_seqlens_chunk) return CFA_ERR_INVALID_ARG;
  if (a->total_lc > 0 && (!a->q || !a->k_chunk || !a->v_chunk)) return CFA_ERR_INVALID_ARG;
  if (a->total_lp > 0 && (!a->k_prefix || !a->v_prefix)) return CFA_ERR_INVALID_ARG;
  if (!aligned16(a->q) || !aligned16(a->k_chunk) || !aligned16(a->v_chunk))
    return CFA_ERR_INVALID_ARG;
  if (a->prefix_dtype == CFA_PREFIX_Q8_0) {
    // q8_0 blocks are 34 bytes: the fp16 scale needs 2-byte alignment
    if ((reinterpret_cast<uintptr_t>(a->k_prefix) | reinterpret_cast<uintptr_t>(a->v_prefix)) & 1u)
      return CFA_ERR_INVALID_ARG;
  } else if (!aligned16(a->k_prefix) || !aligned16(a->v_prefix)) {
    return CFA_ERR_INVALID_ARG;
  }
  if ((long long)a->total_lc * a->hq * a->head_dim >= (1ll << 40)) return CFA_ERR_UNSUPPORTED;
  return CFA_OK;
}

struct Plan {
  Tiling fwd, dq;
  int n_kc_max;        // 128-key chunk tiles per window, upper bound
  size_t off_wp_fwd, off_opart, off_lsepart, ws_fwd;
  size_t off_wp_bwd, off_dqpart, ws_bwd;
  size_t off_kp16;       // forward workspace: bf16 copies of a q8_0 prefix, K then V
  size_t off_kp16_bwd;   // the same copies in the backward workspace
};

int sm_count(int* n) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CFA_ERR_CUDA;
  if (cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return CFA_ERR_CUDA;
  return CFA_OK;
}

Tiling make_tiling(const cfa_args* a, int q_per_cta, int sms) {
  Tiling t;
  t.g = a->hq / a->hkv;
  t.tpt = kTileM / t.g;
  t.rows = t.tpt * t.g;
  t.q_per_cta = q_per_cta;
  t.grid = sms;  // persistent: one CTA per SM (each uses all of TMEM)
  // taking up a query block costs a CTA about two key tiles' time (measured:
  // CTAs whose range crosses a block start finished 2-3.5 us later)
  t.setup = 2;
  t.nrow = 1;
  return t;
}

// Row mode (Tiling::nrow, cfa_sched.cuh) pays when the heads' K/V is well
// beyond L2 (129 MB): then the query blocks of one (window, KV head), which
// read the same keys, must run in lockstep for a key tile to come from DRAM
// once.  It needs every window to have the same chunk length (the rows then
// have the same layout) and a grid that the rows divide.  Returns the number
// of rows for a grid of `grid` CTAs, or 1.
constexpr double kRowModeKvBytes = 96.0 * (1 << 20);

int row_mode_rows(const cfa_args* a, const Tiling& t, int grid) {
  const double kv_bytes = 4.0 * (double)a->total_lp * a->hkv * a->head_dim;  // bf16 K and V
  if (kv_bytes < kRowModeKvBytes) return 1;
  if ((long long)a->total_lc != (long long)a->batch * a->max_lc) return 1;  // lengths differ
  const int nb = blocks_of_window(t, a->max_lc);
  if (nb <= 1 || grid % nb != 0) return 1;
  return nb;
}

// Workspace layout (every region 256-byte aligned):
//   [0, 256)           status word
//   win_prefix         int64 [rows][batch + 1]  (stream-K plan, per schedule row)
//   partials           fp32, two slots per CTA: forward O [G, 2, 256, d] and
//                      LSE [G, 2, 256]; backward dQ [G, 2, 128, d]
//   bf16 prefix        K then V [total_lp, hkv, d], only for a q8_0 prefix
int make_plan(const cfa_args* a, Plan* p) {
  int sms = 0;
  int st = sm_count(&sms);
  if (st) return st;
  p->fwd = make_tiling(a, 2, sms);
  p->dq = make_tiling(a, 1, sms);
  p->fwd.nrow = row_mode_rows(a, p->fwd, sms);
  // the dQ grid is the GPU less the dK/dV kernel's SMs, fixed by the call;
  // its row count is settled there (dq_rows), the prefix arrays sized here
  const int dq_rows_max = blocks_of_window(p->dq, a->max_lc > 0 ? a->max_lc : 1);
  p->n_kc_max = ceil_div(a->max_lc > 0 ? a->max_lc : 1, kTileN);
  const size_t G = (size_t)sms;
  const size_t wp_rows = (size_t)(p->fwd.nrow > dq_rows_max ? p->fwd.nrow : dq_rows_max);
  const size_t wp = align256(wp_rows * (size_t)(a->batch + 1) * 8);
  const size_t kv16 = (a->prefix_dtype != CFA_PREFIX_BF16)
                          ? align256((size_t)a->total_lp * a->hkv * a->head_dim * 2)
                          : 0;
  size_t off = kWsHeader;
  p->off_wp_fwd = off;
  off += wp;
  p->off_opart = off;
  off = align256(off + G * 2 * 256 * a->head_dim * 4);
  p->off_lsepart = off;
  off = align256(off + G * 2 * 256 * 4);
  p->off_kp16 = kv16 ? off : 0;
  p->ws_fwd = off + 2 * kv16;
  off = kWsHeader;
  p->off_wp_bwd = off;
  off += wp;
  p->off_dqpart = off;
  off = align256(off + G * 2 * 128 * a->head_dim * 4);
  p->off_kp16_bwd = kv16 ? off : 0;
  p->ws_bwd = off + 2 * kv16;
  return CFA_OK;
}

unsigned long long wait_limit_ns() {
  const char* e = std::getenv("CFA_WAIT_LIMIT_NS");
  if (!e || !*e) return kDefaultWaitNs;
  char* end = nullptr;
  unsigned long long v = std::strtoull(e, &end, 10);
  return (end && *end == 0) ? v : kDefaultWaitNs;
}

// Test hook for the failure-detection tests: with CFA_DEBUG_WAIT_NEVER=1 the
// attention kernels' MMA thread first waits on a barrier that nothing arrives
// on, so the bounded wait runs out and the kernel reports
// CFA_ERR_DEVICE_TIMEOUT instead of computing.
int debug_wait_never() {
  const char* e = std::getenv("CFA_DEBUG_WAIT_NEVER");
  return (e && e[0] == '1') ? 1 : 0;
}

SeqLimits seq_limits(const cfa_args* a) {
  SeqLimits l;
  l.total_lp = a->total_lp;
  l.total_lc = a->total_lc;
  l.max_lp = a->max_lp;
  l.max_lc = a->max_lc;
  return l;
}

int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < need)
    return CFA_ERR_WORKSPACE;
  return CFA_OK;
}

// Chunk maps always; prefix maps over `kp16`/`vp16` (bf16 rows), or none
// when those are null (the dK/dV half never reads the prefix).
int encode_kv_maps(const cfa_args* a, const void* kp16, const void* vp16, Maps* m) {
  const int d = a->head_dim;
  const long long lp_rows = (kp16 && vp16) ? a->total_lp : 0;
  int st = make_map_bf16(&m->kc, a->k_chunk, d, a->hkv, a->total_lc, 1, kTileN);
  if (!st) st = make_map_bf16(&m->vc, a->v_chunk, d, a->hkv, a->total_lc, 1, kTileN);
  if (!st) st = make_map_bf16(&m->kp, kp16, d, a->hkv, lp_rows, 1, kTileN);
  if (!st) st = make_map_bf16(&m->vp, vp16, d, a->hkv, lp_rows, 1, kTileN);
  return st;
}

// The bf16 prefix rows the attention kernels read: the caller's tensors, or
// for a q8_0 / fp16 prefix the workspace copies, filled here (on the stream)
// by the dequant / conversion kernel.
int prefix_rows_bf16(const cfa_args* a, uint8_t* ws, size_t off_k, cudaStream_t s,
                     const void** kp16, const void** vp16) {
  if (a->total_lp == 0) {
    *kp16 = *vp16 = nullptr;
    return CFA_OK;
  }
  if (a->prefix_dtype == CFA_PREFIX_BF16) {
    *kp16 = a->k_prefix;
    *vp16 = a->v_prefix;
    return CFA_OK;
  }
  const size_t kv16 = align256((size_t)a->total_lp * a->hkv * a->head_dim * 2);
  __nv_bfloat16* k16 = reinterpret_cast<__nv_bfloat16*>(ws + off_k);
  __nv_bfloat16* v16 = reinterpret_cast<__nv_bfloat16*>(ws + off_k + kv16);
  cudaError_t e;
  if (a->prefix_dtype == CFA_PREFIX_F16) {
    e = launch_f16_to_bf16(static_cast<const __half*>(a->k_prefix),
                           static_cast<const __half*>(a->v_prefix),
                           (long long)a->total_lp * a->hkv * a->head_dim, k16, v16, s);
  } else {
    const long long nb = (long long)a->total_lp * a->hkv * (a->head_dim / 32);
    e = launch_dequant_prefix(static_cast<const uint8_t*>(a->k_prefix),
                              static_cast<const uint8_t*>(a->v_prefix), nb, k16, v16, s);
  }
  if (e != cudaSuccess) return CFA_ERR_LAUNCH;
  *kp16 = k16;
  *vp16 = v16;
  return CFA_OK;
}

}  // namespace

extern "C" {

int cfa_version(void) { return (1 << 16) | 0; }

const char* cfa_status_string(int s) {
  switch (s) {
    case CFA_OK: return "ok";
    case CFA_ERR_INVALID_ARG: return "invalid argument";
    case CFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case CFA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case CFA_ERR_LAUNCH: return "kernel launch failed";
    case CFA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case CFA_ERR_CUDA: return "CUDA error";
    case CFA_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of cfa_forward_noalloc";
    default: return "unknown status";
  }
}

size_t cfa_workspace_size(const cfa_args* a, int which) {
  if (validate(a) != CFA_OK) return 0;
  Plan p;
  if (make_plan(a, &p) != CFA_OK) return 0;
  if (which == CFA_WS_FORWARD) return p.ws_fwd;
  if (which == CFA_WS_BACKWARD) return p.ws_bwd;
  return 0;
}

int cfa_forward(const cfa_args* a, void* o, float* lse, void* ws, size_t ws_bytes, void* stream) {
  int st = validate(a);
  if (st) return st;
  if (a->total_lc > 0 && (!o || !lse || !aligned16(o))) return CFA_ERR_INVALID_ARG;
  Plan p;
  if ((st = make_plan(a, &p))) return st;
  if ((st = check_ws(ws, ws_bytes, p.ws_fwd))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a->total_lc == 0 || a->max_lc == 0)  // no kernel to clear the status word
    return cudaMemsetAsync(ws, 0, 4, s) == cudaSuccess ? CFA_OK : CFA_ERR_LAUNCH;

  Maps m;
  std::memset(&m, 0, sizeof(m));
  const Tiling& tl = p.fwd;
  if ((st = make_map_bf16(&m.q, a->q, a->head_dim, a->hq, a->total_lc, tl.g, tl.tpt))) return st;
  const void *kp16 = nullptr, *vp16 = nullptr;
  if ((st = prefix_rows_bf16(a, static_cast<uint8_t*>(ws), p.off_kp16, s, &kp16, &vp16)))
    return st;
  if ((st = encode_kv_maps(a, kp16, vp16, &m))) return st;

  uint8_t* w = static_cast<uint8_t*>(ws);
  FwdArgs fa;
  fa.cu_p = a->cu_seqlens_prefix;
  fa.cu_c = a->cu_seqlens_chunk;
  fa.win_prefix = reinterpret_cast<long long*>(w + p.off_wp_fwd);
  fa.batch = a->batch;
  fa.hq = a->hq;
  fa.hkv = a->hkv;
  fa.total_lc = a->total_lc;
  fa.lim = seq_limits(a);
  fa.tl = tl;
  fa.scale_log2 = a->softmax_scale * kLog2e;
  fa.o = static_cast<__nv_bfloat16*>(o);
  fa.lse = lse;
  fa.o_part = reinterpret_cast<float*>(w + p.off_opart);
  fa.lse_part = reinterpret_cast<float*>(w + p.off_lsepart);
  fa.status = reinterpret_cast<int*>(w);
  fa.clear_status = 1;
  fa.limit_ns = wait_limit_ns();
  fa.debug_wait_never = debug_wait_never();

  if (launch_fwd(m, fa, a->head_dim, 0, s) != cudaSuccess) return CFA_ERR_LAUNCH;
  if (launch_fwd_merge(fa, a->head_dim, a->max_lc, s) != cudaSuccess) return CFA_ERR_LAUNCH;
  return CFA_OK;
}

int cfa_backward_preprocess(const cfa_args* a, const void* o, const void* dout, float* delta,
                            void* stream) {
  int st = validate(a);
  if (st) return st;
  if (a->total_lc == 0) return CFA_OK;
  if (!o || !dout || !delta || !aligned16(o) || !aligned16(dout)) return CFA_ERR_INVALID_ARG;
  if (launch_delta(static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout),
                   delta, a->total_lc, a->hq, a->head_dim,
                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CFA_ERR_LAUNCH;
  return CFA_OK;
}

}  // extern "C"

namespace {

// Shared set-up of the backward halves: validation, plan, workspace check,
// status-word clear, TMA maps and the kernel argument block.  Returns a
// status; *skip is set when there is nothing to compute.
int prepare_backward(const cfa_args* a, const void* dout, const float* lse, const float* delta,
                     void* ws, size_t ws_bytes, bool need_partials, cudaStream_t s, Plan* p,
                     Maps* m, BwdArgs* ba, bool* skip) {
  *skip = false;
  int st = validate(a);
  if (st) return st;
  if (a->total_lc > 0 && (!dout || !lse || !delta || !aligned16(dout))) return CFA_ERR_INVALID_ARG;
  if ((st = make_plan(a, p))) return st;
  if ((st = check_ws(ws, ws_bytes, need_partials ? p->ws_bwd : kWsHeader))) return st;
  if (a->total_lc == 0 || a->max_lc == 0) {
    // no attention kernel runs to clear the status word
    if (cudaMemsetAsync(ws, 0, 4, s) != cudaSuccess) return CFA_ERR_LAUNCH;
    *skip = true;
    return CFA_OK;
  }
  std::memset(m, 0, sizeof(*m));
  const Tiling& tl = p->dq;
  if ((st = make_map_bf16(&m->q, a->q, a->head_dim, a->hq, a->total_lc, tl.g, tl.tpt))) return st;
  if ((st = make_map_bf16(&m->dout, dout, a->head_dim, a->hq, a->total_lc, tl.g, tl.tpt)))
    return st;
  const void *kp16 = nullptr, *vp16 = nullptr;
  if (need_partials &&
      (st = prefix_rows_bf16(a, static_cast<uint8_t*>(ws), p->off_kp16_bwd, s, &kp16, &vp16)))
    return st;
  if ((st = encode_kv_maps(a, kp16, vp16, m))) return st;
  ba->cu_p = a->cu_seqlens_prefix;
  ba->cu_c = a->cu_seqlens_chunk;
  ba->win_prefix = reinterpret_cast<long long*>(static_cast<uint8_t*>(ws) + p->off_wp_bwd);
  ba->batch = a->batch;
  ba->hq = a->hq;
  ba->hkv = a->hkv;
  ba->total_lc = a->total_lc;
  ba->lim = seq_limits(a);
  ba->tl = tl;
  ba->scale_log2 = a->softmax_scale * kLog2e;
  ba->scale = a->softmax_scale;
  ba->lse = lse;
  ba->delta = delta;
  ba->dq = ba->dk = ba->dv = nullptr;
  uint8_t* w = static_cast<uint8_t*>(ws);
  ba->dq_part = need_partials ? reinterpret_cast<float*>(w + p->off_dqpart) : nullptr;
  ba->dkv_tiles = p->n_kc_max;
  ba->horizon = 0;
  ba->pre_tiles = 0;
  ba->dk_p = ba->dv_p = nullptr;
  ba->status = reinterpret_cast<int*>(w);
  ba->clear_status = 1;  // the caller turns it off for a kernel that is not the first
  ba->limit_ns = wait_limit_ns();
  ba->debug_wait_never = debug_wait_never();
  return CFA_OK;
}

int run_dq(const cfa_args* a, const Plan& p, const Maps& m, const BwdArgs& ba, cudaStream_t s) {
  if (launch_bwd_dq(m, ba, a->head_dim, 0, s) != cudaSuccess) return CFA_ERR_LAUNCH;
  if (launch_bwd_dq_reduce(ba, a->head_dim, a->max_lc, s) != cudaSuccess) return CFA_ERR_LAUNCH;
  return CFA_OK;
}

// dK/dV work items (key tile slot x window x KV head, some empty).
long long dkdv_items(const cfa_args* a, const BwdArgs& ba) {
  return (long long)(ba.pre_tiles + ba.dkv_tiles) * a->batch * a->hkv;
}

int run_dkdv(const cfa_args* a, const Plan& p, const Maps& m, const BwdArgs& ba, int ctas,
             cudaStream_t s) {
  if (launch_bwd_dkdv(m, ba, a->head_dim, ctas, s) != cudaSuccess) return CFA_ERR_LAUNCH;
  return CFA_OK;
}

// SMs given to the dK/dV kernel when it runs beside the dQ kernel: its share
// of the work, estimated from window lengths averaged over the batch with the
// per-step times measured on GB300 (a dQ step -- query tile x key tile -- about
// 2100 cycles, a dK/dV step about 3000, plus about 4000 per dK/dV item for its
// K/V load and epilogue), rounded up and one more, since a dK/dV item cannot
// be split and a late dK/dV ends the backward.
int dkdv_share(const cfa_args* a, const Tiling& tl, int sms, long long items, int horizon) {
  const double B = a->batch;
  const double lc = (double)a->total_lc / B, lp = (double)a->total_lp / B;
  const double qt = std::ceil(lc / tl.tpt);
  const double nk = std::ceil(lc / kTileN);
  // chunk key tiles see the query tiles from their own on; horizon prefix
  // tiles see all of them
  const double nh = horizon > 0 ? std::ceil(std::min((double)horizon, lp) / kTileN) + 1 : 0;
  const double kv_steps = nk * qt - (double)kTileN / tl.tpt * nk * (nk - 1) / 2 + nh * qt;
  const double dq_steps = qt * (std::ceil(lp / kTileN) + (nk + 1) / 2 + tl.setup);
  const double w_kv = 3000 * kv_steps + 4000 * (nk + nh), w_dq = 2100 * dq_steps;
  long long k = (long long)std::ceil(sms * w_kv / (w_kv + w_dq)) + 1;
  if (k > sms / 2 && horizon == 0) k = sms / 2;
  if (k > sms - 8) k = sms - 8;
  if (k > items) k = items;
  return k < 1 ? 1 : (int)k;
}

// With equal chunk lengths and no horizon the dK/dV items' costs are known
// exactly (the same per-step costs as above; item j walks the query tiles from
// its key tile's on), so the share can shrink to the fewest CTAs whose
// busiest one (items c, c + k, ...) is no busier than with k: those SMs go to
// the dQ grid at no cost to the dK/dV kernel (qwen3_8b: 16 items, 5 -> 4).
int trim_dkdv_share(const cfa_args* a, const Tiling& tl, int k, long long items, int horizon) {
  if (horizon != 0 || k <= 1 || items > 65536 ||
      (long long)a->total_lc != (long long)a->batch * a->max_lc)
    return k;
  const long long per_slot = (long long)a->batch * a->hkv;
  const int qt = ceil_div(a->max_lc, tl.tpt);
  auto cost = [&](long long j) -> long long {
    const int key0 = (int)(j / per_slot) * kTileN;
    if (key0 >= a->max_lc) return 0;
    return 3000LL * (qt - key0 / tl.tpt) + 4000;
  };
  auto busiest = [&](int kk) {
    long long worst = 0;
    for (int c = 0; c < kk; ++c) {
      long long sum = 0;
      for (long long j = c; j < items; j += kk) sum += cost(j);
      worst = sum > worst ? sum : worst;
    }
    return worst;
  };
  const long long target = busiest(k);
  int best = k;
  for (int kk = k - 1; kk >= 1; --kk) {
    if (busiest(kk) > target) break;
    best = kk;
  }
  return best;
}

// The second stream and the fork / join events cfa_backward uses to run the
// dK/dV kernel beside the dQ kernel, one set per device, made on first use.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_side_mutex;
SideStream g_side[kMaxDevices];

int side_stream(SideStream** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CFA_ERR_CUDA;
  SideStream& ss = g_side[dev];
  if (!ss.stream) {
    if (cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess)
      return CFA_ERR_CUDA;
  }
  *out = &ss;
  return CFA_OK;
}

}  // namespace

extern "C" {

int cfa_backward(const cfa_args* a, const void* dout, const float* lse, const float* delta,
                 void* dq, void* dk_chunk, void* dv_chunk, void* ws, size_t ws_bytes,
                 void* stream) {
  return cfa_backward_horizon(a, 0, dout, lse, delta, dq, dk_chunk, dv_chunk, nullptr, nullptr,
                              ws, ws_bytes, stream);
}

int cfa_backward_horizon(const cfa_args* a, int horizon, const void* dout, const float* lse,
                         const float* delta, void* dq, void* dk_chunk, void* dv_chunk,
                         void* dk_prefix, void* dv_prefix, void* ws, size_t ws_bytes,
                         void* stream) {
  if (horizon < 0) return CFA_ERR_INVALID_ARG;
  if (a && a->total_lc > 0 && (!dq || !dk_chunk || !dv_chunk || !aligned16(dq) ||
                               !aligned16(dk_chunk) || !aligned16(dv_chunk)))
    return CFA_ERR_INVALID_ARG;
  const bool want_prefix = a && horizon > 0 && a->total_lp > 0;
  if (want_prefix &&
      (!dk_prefix || !dv_prefix || !aligned16(dk_prefix) || !aligned16(dv_prefix)))
    return CFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Plan p;
  Maps m;
  BwdArgs ba;
  bool skip;
  int st = prepare_backward(a, dout, lse, delta, ws, ws_bytes, true, s, &p, &m, &ba, &skip);
  if (st) return st;
  ba.dq = static_cast<__nv_bfloat16*>(dq);
  ba.dk = static_cast<__nv_bfloat16*>(dk_chunk);
  ba.dv = static_cast<__nv_bfloat16*>(dv_chunk);
  if (want_prefix) {
    // the last `horizon` prefix rows of a window span at most this many tiles
    const int h = horizon < a->max_lp ? horizon : a->max_lp;
    const int spans = ceil_div(h, kTileN) + 1, tiles = ceil_div(a->max_lp, kTileN);
    ba.horizon = horizon;
    ba.pre_tiles = spans < tiles ? spans : tiles;
    ba.dk_p = static_cast<__nv_bfloat16*>(dk_prefix);
    ba.dv_p = static_cast<__nv_bfloat16*>(dv_prefix);
  }
  if (skip) {
    // no chunk rows anywhere: nothing attends to the prefix, so the horizon
    // rows' gradients are zero
    if (want_prefix &&
        launch_zero_horizon(a->cu_seqlens_prefix, a->batch, a->hkv, a->head_dim, horizon,
                            seq_limits(a), ba.dk_p, ba.dv_p, static_cast<int*>(ws),
                            s) != cudaSuccess)
      return CFA_ERR_LAUNCH;
    return CFA_OK;
  }
  // The two halves share no outputs: the dK/dV kernel runs on a few SMs of
  // its own, on a second stream forked from and joined back into `s`, while
  // the dQ kernel's persistent grid takes the rest.
  const long long items = dkdv_items(a, ba);
  int k = trim_dkdv_share(a, p.dq, dkdv_share(a, p.dq, p.dq.grid, items, ba.horizon), items,
                          ba.horizon);
  // row mode for the dQ kernel: give the dK/dV kernel a few SMs more, if that
  // makes the rows divide the dQ grid
  for (int k2 = k; k2 <= k + 16 && k2 <= p.dq.grid / 2; ++k2) {
    const int rows = row_mode_rows(a, p.dq, p.dq.grid - k2);
    if (rows > 1) {
      k = k2;
      ba.tl.nrow = rows;
      break;
    }
  }
  ba.tl.grid = p.dq.grid - k;
  std::lock_guard<std::mutex> lock(g_side_mutex);
  SideStream* ss = nullptr;
  if ((st = side_stream(&ss))) return st;
  if (cudaEventRecord(ss->fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(ss->stream, ss->fork, 0) != cudaSuccess)
    return CFA_ERR_LAUNCH;
  // the dQ kernel clears the status word; the dK/dV kernel beside it must not
  BwdArgs ba_kv = ba;
  ba_kv.clear_status = 0;
  const int st_kv = run_dkdv(a, p, m, ba_kv, k, ss->stream);
  const int st_dq = run_dq(a, p, m, ba, s);
  // join even after a failed launch, so `s` never runs ahead of the side stream
  if (cudaEventRecord(ss->join, ss->stream) != cudaSuccess ||
      cudaStreamWaitEvent(s, ss->join, 0) != cudaSuccess)
    return CFA_ERR_LAUNCH;
  return st_kv ? st_kv : st_dq;
}

int cfa_backward_dq(const cfa_args* a, const void* dout, const float* lse, const float* delta,
                    void* dq, void* ws, size_t ws_bytes, void* stream) {
  if (a && a->total_lc > 0 && (!dq || !aligned16(dq))) return CFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Plan p;
  Maps m;
  BwdArgs ba;
  bool skip;
  int st = prepare_backward(a, dout, lse, delta, ws, ws_bytes, true, s, &p, &m, &ba, &skip);
  if (st || skip) return st;
  ba.dq = static_cast<__nv_bfloat16*>(dq);
  ba.tl.nrow = row_mode_rows(a, p.dq, ba.tl.grid);
  return run_dq(a, p, m, ba, s);
}

int cfa_backward_dkdv(const cfa_args* a, const void* dout, const float* lse, const float* delta,
                      void* dk_chunk, void* dv_chunk, void* ws, size_t ws_bytes, void* stream) {
  if (a && a->total_lc > 0 && (!dk_chunk || !dv_chunk || !aligned16(dk_chunk) ||
                               !aligned16(dv_chunk)))
    return CFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Plan p;
  Maps m;
  BwdArgs ba;
  bool skip;
  int st = prepare_backward(a, dout, lse, delta, ws, ws_bytes, false, s, &p, &m, &ba, &skip);
  if (st || skip) return st;
  ba.dk = static_cast<__nv_bfloat16*>(dk_chunk);
  ba.dv = static_cast<__nv_bfloat16*>(dv_chunk);
  const long long items = dkdv_items(a, ba);
  return run_dkdv(a, p, m, ba, (int)(items < p.dq.grid ? items : p.dq.grid), s);
}

int cfa_dequant_q8_0(const void* blocks, long long n_blocks, float* out_f32, void* out_bf16,
                     void* stream) {
  if (n_blocks < 0) return CFA_ERR_INVALID_ARG;
  if (n_blocks == 0) return CFA_OK;
  if (!blocks || (!out_f32 && !out_bf16)) return CFA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(blocks) & 1u) || (reinterpret_cast<uintptr_t>(out_f32) & 3u) ||
      (reinterpret_cast<uintptr_t>(out_bf16) & 1u))
    return CFA_ERR_INVALID_ARG;
  cudaError_t e;
  if (!out_f32 && (reinterpret_cast<uintptr_t>(out_bf16) & 15u) == 0)
    e = launch_dequant_prefix(static_cast<const uint8_t*>(blocks), nullptr, n_blocks,
                              static_cast<__nv_bfloat16*>(out_bf16), nullptr,
                              static_cast<cudaStream_t>(stream));
  else
    e = launch_dequant_q8_0(static_cast<const uint8_t*>(blocks), n_blocks, out_f32,
                            static_cast<__nv_bfloat16*>(out_bf16), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return CFA_ERR_LAUNCH;
  return CFA_OK;
}

int cfa_quantize_q8_0(const void* x_bf16, long long n_blocks, void* out_blocks, void* stream) {
  if (n_blocks < 0) return CFA_ERR_INVALID_ARG;
  if (n_blocks == 0) return CFA_OK;
  if (!x_bf16 || !out_blocks || !aligned16(x_bf16) ||
      (reinterpret_cast<uintptr_t>(out_blocks) & 1u))
    return CFA_ERR_INVALID_ARG;
  if (launch_quantize_q8_0(static_cast<const __nv_bfloat16*>(x_bf16), n_blocks,
                           static_cast<uint8_t*>(out_blocks),
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CFA_ERR_LAUNCH;
  return CFA_OK;
}

int cfa_read_status(const void* ws, void* stream) {
  if (!ws) return CFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return CFA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CFA_ERR_CUDA;
  return v;
}

}  // extern "C"

// ------------------------------------------- row-sparse projection backward --

#include "cfa_rowsparse.cuh"

namespace {

// Matrix [outer, inner] (row-major, bf16 or fp32) -> 2-D map, 128-byte
// swizzle, boxes of box_inner x box_outer elements.  Out-of-range elements
// read as zero; stores to them are dropped.
int make_map_2d(CUtensorMap* m, const void* ptr, long long inner, long long outer, int box_inner,
                int box_outer, bool f32 = false) {
  std::memset(m, 0, sizeof(*m));
  if (inner <= 0 || outer <= 0) return CFA_OK;  // never dereferenced
  EncodeTiledFn fn = encode_fn();
  if (!fn) return CFA_ERR_CUDA;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)inner * (f32 ? 4 : 2)};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer};
  cuuint32_t es[2] = {1u, 1u};
  CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(ptr), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? CFA_OK : CFA_ERR_INVALID_ARG;
}

int rs_validate(const cfa_rowsparse_args* r) {
  if (!r) return CFA_ERR_INVALID_ARG;
  if (r->n_keep < 0 || r->n_rows < 0 || r->in_features < 1 || r->out_features < 1)
    return CFA_ERR_INVALID_ARG;
  // 16-byte rows for TMA strides and the 16-byte gathers and stores
  if (r->in_features % 8 != 0 || r->out_features % 8 != 0) return CFA_ERR_INVALID_ARG;
  if (r->n_keep > 0 && (!r->dy || !aligned16(r->dy) || !r->keep_idx ||
                        (reinterpret_cast<uintptr_t>(r->keep_idx) & 3u)))
    return CFA_ERR_INVALID_ARG;
  if ((long long)r->n_rows * r->in_features >= (1ll << 40) ||
      (long long)r->out_features * r->in_features >= (1ll << 40) ||
      (long long)r->n_keep * r->out_features >= (1ll << 40))
    return CFA_ERR_UNSUPPORTED;
  return CFA_OK;
}

struct RsPlan {
  RsArgs a;
  int grid;
  size_t off_cnt, off_part, ws;
};

// Tiles of 128 x 256 outputs; K in 64-row stages, split when there are fewer
// tiles than SMs (each split keeps at least two stages).  The workspace holds
// the status word, the per-tile counters and the fp32 partial tiles.
int rs_plan(const cfa_rowsparse_args* r, int mode, RsPlan* p) {
  int sms = 0;
  int st = sm_count(&sms);
  if (st) return st;
  RsArgs& a = p->a;
  std::memset(&a, 0, sizeof(a));
  a.mode = mode;
  a.M = mode == 0 ? r->out_features : r->n_keep;
  a.N = r->in_features;
  a.K = mode == 0 ? r->n_keep : r->out_features;
  a.n_keep = r->n_keep;
  a.n_rows = r->n_rows;
  const int tiles_m = ceil_div(a.M, kRsTileM);
  a.tiles_n = ceil_div(a.N, kRsTileN);
  a.tiles = tiles_m * a.tiles_n;
  a.k_stages = ceil_div(a.K, kRsBK);
  int splits = 1;
  if (a.tiles > 0 && a.tiles < sms) {
    splits = sms / a.tiles;
    const int by_k = a.k_stages / 2 > 1 ? a.k_stages / 2 : 1;
    if (splits > by_k) splits = by_k;
    if (splits > kRsMaxSplits) splits = kRsMaxSplits;
    if (splits < 1) splits = 1;
  }
  a.splits = splits;
  a.units = (long long)a.tiles * splits;
  p->grid = (int)(a.units < sms ? a.units : sms);
  // dX split K: one cluster per tile when every tile's splits can be resident
  // together (they exchange their partials through L2 without counters)
  // (CFA_RS_CLUSTER=0 keeps the global-memory path: the tests compare the two)
  const char* env = std::getenv("CFA_RS_CLUSTER");
  const bool allow = !(env && env[0] == '0');
  a.cluster = (allow && mode == 1 && splits > 1 && a.units <= sms &&
               rowsparse_clusters_fit(splits, a.tiles))
                  ? 1
                  : 0;
  p->off_cnt = 16;
  const size_t hdr = align256(p->off_cnt + (size_t)a.tiles * 16);
  p->off_part = hdr;
  p->ws = hdr + (splits > 1 ? (size_t)a.tiles * splits * kRsTileM * kRsTileN * 4 : 0);
  if (p->ws < kWsHeader) p->ws = kWsHeader;
  a.limit_ns = wait_limit_ns();
  return CFA_OK;
}

int rs_run(const cfa_rowsparse_args* r, int mode, void* out, int out_f32, int accumulate,
           void* ws, size_t ws_bytes, cudaStream_t s) {
  RsPlan p;
  int st = rs_plan(r, mode, &p);
  if (st) return st;
  if ((st = check_ws(ws, ws_bytes, p.ws))) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  // status word and the (tile, lane quadrant) counters start at zero (the
  // cluster path has no counters, and its first CTA clears the status)
  if (!p.a.cluster && cudaMemsetAsync(ws, 0, p.off_cnt + (size_t)p.a.tiles * 16, s) != cudaSuccess)
    return CFA_ERR_LAUNCH;
  RsArgs& a = p.a;
  a.keep = r->keep_idx;
  a.x = static_cast<const __nv_bfloat16*>(r->x);
  a.out = out;
  a.out_f32 = out_f32;
  a.accumulate = accumulate;
  a.part = reinterpret_cast<float*>(w + p.off_part);
  a.counters = reinterpret_cast<unsigned*>(w + p.off_cnt);
  a.status = reinterpret_cast<int*>(w);
  if (a.units == 0) return CFA_OK;
  CUtensorMap ma, mb, mo, mp, mxt;
  std::memset(&mo, 0, sizeof(mo));
  std::memset(&mp, 0, sizeof(mp));
  std::memset(&mxt, 0, sizeof(mxt));
  if (mode == 0 && !accumulate &&
      (st = make_map_2d(&mo, out, r->in_features, r->out_features, out_f32 ? 32 : 64, 32,
                        out_f32 != 0)))
    return st;
  if (a.splits > 1 &&
      (st = make_map_2d(&mp, a.part, kRsTileN, (long long)a.tiles * a.splits * kRsTileM, 32, 32,
                        true)))
    return st;
  if (mode == 0) {
    if ((st = make_map_2d(&ma, r->dy, r->out_features, r->n_keep, 64, kRsBK))) return st;
    // X read by 4-row gathers (64-column x 1-row boxes), or by 64 x 64 tiles
    // where a stage's kept rows are consecutive
    if ((st = make_map_2d(&mb, r->x, r->in_features, r->n_rows, 64, 1))) return st;
    if ((st = make_map_2d(&mxt, r->x, r->in_features, r->n_rows, 64, kRsBK))) return st;
  } else {
    if ((st = make_map_2d(&ma, r->dy, r->out_features, r->n_keep, kRsBK, kRsTileM))) return st;
    if ((st = make_map_2d(&mb, r->w, r->in_features, r->out_features, 64, kRsBK))) return st;
  }
  if (launch_rowsparse(ma, mb, mo, mp, mxt, a, p.grid, s) != cudaSuccess) return CFA_ERR_LAUNCH;
  return CFA_OK;
}

}  // namespace

extern "C" {

size_t cfa_rowsparse_workspace_size(const cfa_rowsparse_args* a, int which) {
  if (rs_validate(a) != CFA_OK) return 0;
  if (which != CFA_RS_DW && which != CFA_RS_DX) return 0;
  RsPlan p;
  if (rs_plan(a, which == CFA_RS_DW ? 0 : 1, &p) != CFA_OK) return 0;
  return p.ws;
}

int cfa_rowsparse_dw(const cfa_rowsparse_args* a, void* dw, int dw_dtype, int accumulate,
                     void* ws, size_t ws_bytes, void* stream) {
  int st = rs_validate(a);
  if (st) return st;
  if (dw_dtype != CFA_GRAD_F32 && dw_dtype != CFA_GRAD_BF16) return CFA_ERR_INVALID_ARG;
  if (!dw || !aligned16(dw)) return CFA_ERR_INVALID_ARG;
  if (a->n_keep > 0 && (!a->x || !aligned16(a->x))) return CFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a->n_keep == 0) {
    // no kept rows: the gradient is zero (accumulating leaves dW as it is)
    RsPlan p;
    if ((st = rs_plan(a, 0, &p))) return st;
    if ((st = check_ws(ws, ws_bytes, p.ws))) return st;
    if (cudaMemsetAsync(ws, 0, 4, s) != cudaSuccess) return CFA_ERR_LAUNCH;
    if (!accumulate &&
        cudaMemsetAsync(dw, 0, (size_t)a->out_features * a->in_features *
                                   (dw_dtype == CFA_GRAD_F32 ? 4 : 2), s) != cudaSuccess)
      return CFA_ERR_LAUNCH;
    return CFA_OK;
  }
  return rs_run(a, 0, dw, dw_dtype == CFA_GRAD_F32, accumulate ? 1 : 0, ws, ws_bytes, s);
}

int cfa_rowsparse_dx(const cfa_rowsparse_args* a, void* dx, void* ws, size_t ws_bytes,
                     void* stream) {
  int st = rs_validate(a);
  if (st) return st;
  if (a->n_keep > 0 && (!dx || !aligned16(dx) || !a->w || !aligned16(a->w)))
    return CFA_ERR_INVALID_ARG;
  return rs_run(a, 1, dx, 0, 0, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

int cfa_keep_index_chunks(const int32_t* cu_seqlens_prefix, const int32_t* cu_seqlens_chunk,
                          int batch, int total_lc, int32_t* keep_idx, void* stream) {
  if (batch < 1 || total_lc < 0) return CFA_ERR_INVALID_ARG;
  if (total_lc == 0) return CFA_OK;
  if (!cu_seqlens_prefix || !cu_seqlens_chunk || !keep_idx) return CFA_ERR_INVALID_ARG;
  if (launch_keep_index_chunks(cu_seqlens_prefix, cu_seqlens_chunk, batch, total_lc, keep_idx,
                               static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CFA_ERR_LAUNCH;
  return CFA_OK;
}

}  // extern "C"
