/*
 * cfa -- frozen-prefix chunk attention for GB300 (sm_103a), C ABI.
 *
 * One trainable reply chunk of Lc query rows attends to a frozen KV prefix of
 * Lp cached rows plus its own causal keys.  The prefix is a constant: the
 * training walk of "train: walk the window" (llama.cpp fork PR #40, "What it
 * is") reads the cached prefix as constants, and its "Why it's a draft"
 * section states that cached prefixes are stop-gradient constants; the
 * two-phase step of "Context-Frozen Training" ("The Solution", Phase 2) runs
 * the decision tokens with gradients against the no-grad cache.  The backward
 * is the "query-split attention (grad for kept queries only)" that the
 * prime-rl POC "stop-gradient through context tokens" lists under "Known
 * gaps": it returns dQ for the chunk rows over all Lp + Lc keys and dK/dV for
 * the chunk's own keys, and never computes or writes a prefix gradient.
 *
 * Definitions (per window b, query head h, kv head h / (Hq/Hkv), chunk row t
 * at absolute position Lp + t, scale s):
 *   visible keys J_t = all Lp prefix keys and chunk keys j <= t
 *   S_tj = s * q_t . k_j,  LSE_t = ln sum_{J_t} exp S_tj,  P_tj = exp(S_tj - LSE_t)
 *   O_t = sum_{J_t} P_tj v_j
 *   for dO: delta_t = dO_t . O_t,  dS_tj = P_tj (dO_t . v_j - delta_t)
 *   dQ_t = s sum_{J_t} dS_tj k_j
 *   dK_chunk,j = s sum_{heads of the group} sum_{t >= j} dS_tj q_t
 *   dV_chunk,j =   sum_{heads of the group} sum_{t >= j} P_tj dO_t
 *
 * Layouts (packed varlen, "THD", head_dim innermost, row-major, contiguous):
 *   q, o, dout, dq            [total_lc, hq,  d]      bf16
 *   k_chunk, v_chunk, dk, dv  [total_lc, hkv, d]      bf16
 *   k_prefix, v_prefix        [total_lp, hkv, d]      bf16, or
 *                             [total_lp, hkv, d/32] q8_0 blocks of 34 bytes:
 *                             little-endian fp16 scale then 32 int8 codes
 *                             (the llama.cpp q8_0 cache type; V untransposed),
 *                             or [total_lp, hkv, d] fp16 (its F16 cache type)
 *   lse, delta                [hq, total_lc]          fp32 (natural log)
 *   cu_seqlens_prefix/chunk   [batch + 1]             int32, device memory,
 *                             non-decreasing, starting at 0
 * Window b owns prefix rows [cu_p[b], cu_p[b+1]) and chunk rows
 * [cu_c[b], cu_c[b+1]).  Empty windows and Lp = 0 are allowed.
 *
 * Ownership: every pointer is caller-owned device memory (the prefix may be an
 * imported cache); the library allocates no device memory at run time.  The
 * state it keeps across calls is a second stream and two events per device
 * (made by the first cfa_backward call there) and the fixed scratch array of
 * cfa_forward_noalloc (48 MiB, reserved when the module loads on a device;
 * see there).  `ws` is caller-provided scratch of at least
 * cfa_workspace_size() bytes, 256-byte aligned.
 *
 * Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 * legacy default stream).  Nothing synchronises the host or copies device
 * data to the host, except cfa_read_status().  Host-side sizes (batch,
 * max_*, total_*) must agree with the device cu_seqlens; they size the grids
 * and the TMA descriptors, so no device-to-host read is needed.
 *
 * CUDA graphs: cfa_forward, cfa_backward_preprocess, cfa_backward(_horizon),
 * and cfa_dequant_q8_0 can be captured into a CUDA graph
 * (stream capture on a non-default stream; the side stream of the backward
 * joins the capture through its fork / join events).  The TMA descriptors
 * are built at call time and captured as kernel parameters, so a replay
 * works on the buffers and sizes of the captured calls.  Make one call of
 * each kind before the capture: the first cfa_backward on a device creates
 * the library's second stream.  A replay gives bitwise the outputs of the
 * same calls launched one by one, and its status word reads as after them.
 *
 * Errors: every entry point returns CFA_OK (0) or a negative cfa_status and
 * never aborts.  Argument errors are found on the host before anything is
 * enqueued.  A device-side wait that does not finish in time (default 2 s;
 * the environment variable CFA_WAIT_LIMIT_NS overrides it) ends its kernel
 * early and records CFA_ERR_DEVICE_TIMEOUT in the status word at the start of
 * the workspace, readable with cfa_read_status().  Every call clears that
 * word before it computes: the call's first attention kernel does it as it
 * starts (stream-ordered after the previous work), or a 4-byte memset when
 * there is nothing to compute.
 *
 * Determinism: the same inputs give bitwise-identical outputs (fixed-order
 * reductions, no atomics on data); the forward does not depend on whether a
 * backward follows.
 */
#ifndef CFA_H
#define CFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cfa_status {
  CFA_OK = 0,
  CFA_ERR_INVALID_ARG = -1,     /* null/misaligned pointer, bad size or layout */
  CFA_ERR_UNSUPPORTED = -2,     /* valid but not implemented (e.g. head_dim not 64/128) */
  CFA_ERR_WORKSPACE = -3,       /* workspace missing, misaligned or too small */
  CFA_ERR_LAUNCH = -4,          /* a kernel launch or stream operation failed */
  CFA_ERR_DEVICE_TIMEOUT = -5,  /* a device-side wait ran out (see cfa_read_status) */
  CFA_ERR_CUDA = -6,            /* other CUDA runtime/driver error */
  CFA_ERR_SCRATCH_LIMIT = -7    /* request needs more than the fixed scratch of
                                   cfa_forward_noalloc */
} cfa_status;

enum { CFA_PREFIX_BF16 = 0, CFA_PREFIX_Q8_0 = 1, CFA_PREFIX_F16 = 2 };
enum { CFA_WS_FORWARD = 0, CFA_WS_BACKWARD = 1 };

typedef struct cfa_args {
  const void* q;                     /* [total_lc, hq, d] bf16 */
  const void* k_prefix;              /* see layouts; may be NULL iff total_lp == 0 */
  const void* v_prefix;
  const void* k_chunk;               /* [total_lc, hkv, d] bf16 */
  const void* v_chunk;
  const int32_t* cu_seqlens_prefix;  /* device [batch + 1] */
  const int32_t* cu_seqlens_chunk;   /* device [batch + 1] */
  int32_t batch;                     /* windows, >= 1 */
  int32_t max_lp;                    /* max over windows of Lp (host copy) */
  int32_t max_lc;                    /* max over windows of Lc (host copy) */
  int32_t total_lp;                  /* cu_seqlens_prefix[batch] (host copy) */
  int32_t total_lc;                  /* cu_seqlens_chunk[batch]  (host copy) */
  int32_t hq;                        /* query heads */
  int32_t hkv;                       /* kv heads; hq % hkv == 0, hq / hkv <= 128 */
  int32_t head_dim;                  /* 64 or 128 */
  int32_t prefix_dtype;              /* CFA_PREFIX_BF16, CFA_PREFIX_Q8_0 or CFA_PREFIX_F16 */
  float softmax_scale;               /* s > 0, applied to the fp32 logits */
} cfa_args;

/* Bytes of scratch that cfa_forward (which = CFA_WS_FORWARD) or cfa_backward
 * (which = CFA_WS_BACKWARD) needs for these arguments on the current device.
 * Returns 0 for invalid arguments. */
size_t cfa_workspace_size(const cfa_args* a, int which);

/* Forward: O (bf16, [total_lc, hq, d]) and LSE (fp32, [hq, total_lc]).
 * Attention over prefix + causal chunk keys with an online softmax, the
 * (query block, key tile) iterations split evenly over a persistent grid,
 * then a merge of the partials of query blocks that CTAs share.  The tensor
 * cores multiply bf16: a q8_0 prefix is dequantised (fp32(d) * q rounded to
 * bf16) and an fp16 prefix rounded to bf16 (nearest even) into the workspace
 * first. */
int cfa_forward(const cfa_args* a, void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

/* Backward preprocess: delta[h, t] = sum_c dO[t, h, c] * O[t, h, c] (fp32
 * accumulate of the bf16 inputs), the row term of dS. */
int cfa_backward_preprocess(const cfa_args* a, const void* o, const void* dout, float* delta,
                            void* stream);

/* Query-split backward: dq ([total_lc, hq, d]) over all prefix and causal
 * chunk keys; dk_chunk, dv_chunk ([total_lc, hkv, d]) for the chunk keys only,
 * summed over the query heads of each group.  No prefix gradient exists in
 * this interface.  Needs lse from cfa_forward and delta from
 * cfa_backward_preprocess.  The dK/dV half runs on a few SMs beside the dQ
 * half: on a second stream that the library owns (one per device), forked
 * from `stream` and joined back into it with events, so to the caller the
 * call is ordered on `stream` like any other.  Calls from several host
 * threads are serialised around that fork and join. */
int cfa_backward(const cfa_args* a, const void* dout, const float* lse, const float* delta,
                 void* dq, void* dk_chunk, void* dv_chunk, void* ws, size_t ws_bytes,
                 void* stream);

/* The backward with gradients for the frozen prefix's last rows: the "exact
 * reverse pass with horizon H" that "train: walk the window" ("Why it's a
 * draft") asks for, and the full k/v backward on context rows of the
 * prime-rl POC ("Mechanism") when the horizon covers the whole prefix.
 *   Everything cfa_backward writes, plus dk_prefix / dv_prefix
 *   ([total_lp, hkv, d] bf16, caller-owned, 16-byte aligned): for window b
 *   the rows [Lp_b - min(horizon, Lp_b), Lp_b) of its prefix get
 *   dK_p,j = s * sum dS_tj q_t and dV_p,j = sum P_tj dO_t over all chunk rows t
 *   (every one sees the prefix) and the group's query heads.  Other prefix
 *   rows are not written.  horizon = 0 is cfa_backward (the prefix pointers
 *   may then be NULL); horizon >= Lp_b gives every row of window b.  A q8_0
 *   prefix gets bf16 gradients of its dequantised values.  Same workspace as
 *   cfa_backward.  Errors: horizon < 0 or a NULL / misaligned prefix gradient
 *   pointer with horizon > 0 -> CFA_ERR_INVALID_ARG. */
int cfa_backward_horizon(const cfa_args* a, int horizon, const void* dout, const float* lse,
                         const float* delta, void* dq, void* dk_chunk, void* dv_chunk,
                         void* dk_prefix, void* dv_prefix, void* ws, size_t ws_bytes,
                         void* stream);

/* The two independent halves of cfa_backward, for callers that schedule them
 * separately (e.g. on two streams).  cfa_backward_dq writes dq (it needs the
 * cfa_workspace_size(CFA_WS_BACKWARD) workspace for its split partials);
 * cfa_backward_dkdv writes dk_chunk and dv_chunk and needs only the 256-byte
 * status header of a workspace.  Both clear the status word of the workspace
 * they are given, so concurrent halves need separate workspaces. */
int cfa_backward_dq(const cfa_args* a, const void* dout, const float* lse, const float* delta,
                    void* dq, void* ws, size_t ws_bytes, void* stream);
int cfa_backward_dkdv(const cfa_args* a, const void* dout, const float* lse, const float* delta,
                      void* dk_chunk, void* dv_chunk, void* ws, size_t ws_bytes, void* stream);

/* q8_0 dequantisation of n_blocks contiguous 34-byte blocks into 32*n_blocks
 * values: out_f32 = fp32(d) * q (exact), out_bf16 = that value rounded to
 * nearest-even bf16 -- the operand the attention kernels multiply with.
 * Either output may be NULL.  Device pointers; blocks need 2-byte alignment. */
int cfa_dequant_q8_0(const void* blocks, long long n_blocks, float* out_f32, void* out_bf16,
                     void* stream);

/* q8_0 quantisation of n_blocks blocks of 32 contiguous bf16 values into
 * 34-byte blocks: the cache write of the walk ("train: walk the window",
 * "What it is": a chunk's keys and values go into the q8_0 cache so that the
 * next chunk sees them).  Per block, in fp32: d = absmax / 127 (0 for an
 * all-zero block), code q_i = x_i / d rounded half away from zero and clamped
 * to [-127, 127]; the stored scale is fp16(d), nearest even (infinity when d
 * exceeds the fp16 range).  `out_blocks` may point anywhere into an existing
 * cache, e.g. at the first row after a window's prefix (an append).  Device
 * pointers; x 16-byte aligned, out 2-byte aligned; else CFA_ERR_INVALID_ARG. */
int cfa_quantize_q8_0(const void* x_bf16, long long n_blocks, void* out_blocks, void* stream);

/* Forward without a caller workspace, for callers that cannot allocate device
 * memory: a trainer sharing the GPU with an inference server that reserved
 * the memory up front, or a C program whose device memory comes only from
 * someone else's pool.  The pages have no counterpart to this entry point.
 * Same inputs and outputs as cfa_forward; the split partials live in a
 * fixed array of cfa_noalloc_scratch_bytes() bytes (48 MiB) inside the
 * library.  The array is reserved on a device when the library's module is
 * loaded there -- with lazy loading (the CUDA default) on the first call of
 * this entry point, with CUDA_MODULE_LOADING=EAGER on every device where the
 * process uses the library at all -- and held until the process exits.  The
 * first call on a device looks up that array's address (loading the module
 * if needed), so make it before any stream capture; a cudaDeviceReset makes
 * the looked-up address stale, so do not use this entry point across a
 * device reset.  Calls whose forward workspace would exceed the array return
 * CFA_ERR_SCRATCH_LIMIT, and invalid arguments the status cfa_forward gives
 * them, before anything is enqueued.  Nothing is allocated.  All calls share
 * the array: calls that overlap on the GPU (other streams or threads on the
 * same device) race and must be serialised by the caller.  The device status
 * word is the array's first word; read it with cfa_noalloc_read_status. */
int cfa_forward_noalloc(const cfa_args* a, void* o, float* lse, void* stream);

/* Size in bytes of the fixed scratch array used by cfa_forward_noalloc. */
size_t cfa_noalloc_scratch_bytes(void);

/* The device status word of the last cfa_forward_noalloc call on the current
 * device (CFA_OK, or CFA_ERR_DEVICE_TIMEOUT when a device-side wait ran out
 * and O / LSE were not computed), after waiting for `stream`; or a CUDA
 * error.  Allocates nothing. */
int cfa_noalloc_read_status(void* stream);

/* ---------------------------------------------------------------------------
 * Row-sparse projection backward ("POC: stop-gradient through context tokens",
 * prime-rl, "Mechanism": row_sparse_linear).  A linear layer Y = X W^T keeps
 * its full-row forward; when the gradient reaching Y is zero on every row but
 * the kept ones (the context rows of a frozen-prefix step), its backward is
 *   dW          = dY_keep^T X[keep]          [out, in]
 *   dX[keep[i]] = dY_keep[i] W                [in] per kept row
 * and dX is zero on every other row.  dY_keep is compact: row i is the
 * gradient of Y row keep_idx[i].  The query-split attention backward produces
 * exactly this for the q projection (cfa_backward's dQ, [total_lc, hq * d],
 * is dY_keep as it is, with keep_idx from cfa_keep_index_chunks).
 *
 * Layouts (row-major, contiguous, bf16 unless stated):
 *   dy        [n_keep, out_features]
 *   x         [n_rows, in_features]   (cfa_rowsparse_dw only)
 *   w         [out_features, in_features] (the nn.Linear weight; dx only)
 *   keep_idx  [n_keep] int32, device memory; distinct rows of x for dx
 *   dW        [out_features, in_features] fp32 or bf16
 *   dX        [n_rows, in_features]; only the kept rows are written
 * in_features and out_features are multiples of 8; dy, x, w, dW, dX 16-byte
 * aligned.  A keep index outside [0, n_rows) reads as a zero row of x (dw),
 * or its dX row is skipped (dx), and the status word at the start of the
 * workspace is set to CFA_ERR_INVALID_ARG (cfa_read_status).
 * Determinism: each output element is one fixed-order fp32 sum (split
 * contraction ranges are added in range order), so the same inputs give the
 * same bits. */
typedef struct cfa_rowsparse_args {
  const void* dy;
  const void* x;
  const void* w;
  const int32_t* keep_idx;
  int n_keep;        /* kept rows (rows of dy) */
  int n_rows;        /* rows of x and dX */
  int in_features;
  int out_features;
} cfa_rowsparse_args;

enum { CFA_RS_DW = 0, CFA_RS_DX = 1 };          /* workspace size selector */
enum { CFA_GRAD_F32 = 0, CFA_GRAD_BF16 = 1 };   /* dW element type */

/* Workspace bytes (256-byte aligned buffer) for cfa_rowsparse_dw (CFA_RS_DW)
 * or cfa_rowsparse_dx (CFA_RS_DX); 0 for invalid arguments. */
size_t cfa_rowsparse_workspace_size(const cfa_rowsparse_args* a, int which);

/* dW = dY_keep^T X[keep] (accumulate = 0) or dW += dY_keep^T X[keep]
 * (accumulate != 0, read and written in dw_dtype), fp32 accumulation on the
 * tensor cores.  With n_keep = 0, dW is zeroed (or left as it is when
 * accumulating).  x, dy, keep_idx, dw device pointers; w unused. */
int cfa_rowsparse_dw(const cfa_rowsparse_args* a, void* dw, int dw_dtype, int accumulate,
                     void* ws, size_t ws_bytes, void* stream);

/* dX[keep_idx[i]] = dY_keep[i] W (bf16, fp32 accumulation); rows of dX that
 * are not kept are not written (the caller zeroes them once).  dy, w,
 * keep_idx, dx device pointers; x unused. */
int cfa_rowsparse_dx(const cfa_rowsparse_args* a, void* dx, void* ws, size_t ws_bytes,
                     void* stream);

/* The kept rows of a frozen-prefix batch: chunk row j of window b (packed
 * windows of Lp_b prefix rows followed by Lc_b chunk rows, in window order)
 * sits at row cu_seqlens_prefix[b + 1] + j of the packed full sequence.
 * Writes keep_idx[0 .. total_lc) on the device; cu_seqlens as in cfa_args. */
int cfa_keep_index_chunks(const int32_t* cu_seqlens_prefix, const int32_t* cu_seqlens_chunk,
                          int batch, int total_lc, int32_t* keep_idx, void* stream);

/* Waits for `stream`, then returns the status word that the kernels of the
 * last call on this workspace left (CFA_OK, CFA_ERR_DEVICE_TIMEOUT, or for the
 * row-sparse calls CFA_ERR_INVALID_ARG for a keep index outside x), or a CUDA
 * error. */
int cfa_read_status(const void* ws, void* stream);

/* Short description of a status code (static string). */
const char* cfa_status_string(int status);

/* ABI version: (major << 16) | minor. */
int cfa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CFA_H */
