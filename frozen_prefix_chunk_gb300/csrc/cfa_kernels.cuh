// Kernel argument blocks and launchers shared between the host layer
// (cfa_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "cfa_sched.cuh"

namespace cfa {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kStatusInvalidArg = -1;  // CFA_ERR_INVALID_ARG, as the kernels record it

// Wall-clock limit of the bounded waits that unwind a CTA after it has
// already given up (draining copies and MMAs still in flight).
constexpr unsigned long long kDrainLimitNs = 200000000ull;  // 0.2 s

struct FwdArgs {
  const int32_t* cu_p;
  const int32_t* cu_c;
  long long* win_prefix;  // [rows][batch + 1], each row's by its first CTA, for the merge kernel
  int batch, hq, hkv, total_lc;
  SeqLimits lim;         // host sizes the device cu_seqlens must agree with
  Tiling tl;
  float scale_log2;      // softmax_scale * log2(e)
  __nv_bfloat16* o;      // [total_lc, hq, D]
  float* lse;            // [hq, total_lc]
  float* o_part;         // [grid, 2, rows per block, D]  partials of cut blocks
  float* lse_part;       // [grid, 2, rows per block]
  int* status;           // workspace status word
  int clear_status;      // CTA 0 zeroes *status as the kernel starts
  unsigned long long limit_ns;
  int debug_wait_never;  // test hook: the MMA thread waits on a barrier nobody sets
};

struct BwdArgs {
  const int32_t* cu_p;
  const int32_t* cu_c;
  long long* win_prefix;  // [rows][batch + 1], each row's by its first CTA, for the reduce kernel
  int batch, hq, hkv, total_lc;
  SeqLimits lim;         // host sizes the device cu_seqlens must agree with
  Tiling tl;             // dQ tiling (one query tile per block)
  float scale_log2;
  float scale;
  const float* lse;      // [hq, total_lc]
  const float* delta;    // [hq, total_lc]
  __nv_bfloat16* dq;     // [total_lc, hq, D]
  __nv_bfloat16* dk;     // [total_lc, hkv, D]
  __nv_bfloat16* dv;     // [total_lc, hkv, D]
  float* dq_part;        // [grid, 2, 128, D]  partials of cut query tiles
  int dkv_tiles;         // 128-key chunk tiles of the longest window (dK/dV items)
  int horizon;           // prefix rows per window (the last ones) that get dK/dV
  int pre_tiles;         // prefix key tiles a horizon can span (dK/dV items)
  __nv_bfloat16* dk_p;   // [total_lp, hkv, D]  prefix gradients in the horizon
  __nv_bfloat16* dv_p;
  int* status;
  int clear_status;      // CTA 0 zeroes *status as the kernel starts
  unsigned long long limit_ns;
  int debug_wait_never;  // test hook: the MMA thread waits on a barrier nobody sets
};

// The five TMA descriptors of one call.  Prefix maps describe bf16 K/V
// [total_lp, hkv, D] in 64-column boxes of 128 rows, or, for q8_0, the raw
// block bytes.
struct Maps {
  CUtensorMap q, dout, kp, vp, kc, vc;
};

// Launch `k` so that it may overlap the tail of the previous kernel in the
// stream (programmatic stream serialisation); the kernel itself waits for that
// kernel's completion in pdl_start() before touching memory.  Used for the
// persistent kernels (attention and row-sparse GEMM: one CTA per SM, placed
// as the previous grid's CTAs leave) and the delta kernel.  The split merge
// and the dQ reduce keep normal launches: launched this way the merge piled
// onto the first SMs to free up (~4 us slower), and the reduce's waiting CTAs
// held SMs that the dK/dV kernel beside the dQ kernel needed.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}

// Launchers (return a cudaError_t of the launch).
int fwd_smem_bytes(int d, int q8);
cudaError_t launch_fwd(const Maps& m, const FwdArgs& a, int d, int q8, cudaStream_t st);
cudaError_t launch_fwd_merge(const FwdArgs& a, int d, int max_lc, cudaStream_t st);

int bwd_dq_smem_bytes(int d, int q8);
int bwd_dkdv_smem_bytes(int d);
cudaError_t launch_bwd_dq(const Maps& m, const BwdArgs& a, int d, int q8, cudaStream_t st);
cudaError_t launch_bwd_dkdv(const Maps& m, const BwdArgs& a, int d, int ctas, cudaStream_t st);
cudaError_t launch_bwd_dq_reduce(const BwdArgs& a, int d, int max_lc, cudaStream_t st);
cudaError_t launch_delta(const __nv_bfloat16* o, const __nv_bfloat16* dout, float* delta,
                         int total_lc, int hq, int d, cudaStream_t st);
// q8_0 -> bf16 of one or two tensors of n_blocks blocks each (v_blocks may be
// null); outputs 16-byte aligned.
cudaError_t launch_dequant_prefix(const uint8_t* k_blocks, const uint8_t* v_blocks,
                                  long long n_blocks, __nv_bfloat16* k_out,
                                  __nv_bfloat16* v_out, cudaStream_t st);
// fp16 -> bf16 (round to nearest even) of two tensors of n values each.
cudaError_t launch_f16_to_bf16(const __half* k, const __half* v, long long n, __nv_bfloat16* k_out,
                               __nv_bfloat16* v_out, cudaStream_t st);
cudaError_t launch_quantize_q8_0(const __nv_bfloat16* x, long long n_blocks, uint8_t* out,
                                 cudaStream_t st);
cudaError_t launch_zero_horizon(const int32_t* cu_p, int batch, int hkv, int d, int horizon,
                                const SeqLimits& lim, __nv_bfloat16* dk_p, __nv_bfloat16* dv_p,
                                int* status, cudaStream_t st);
cudaError_t launch_dequant_q8_0(const uint8_t* blocks, long long n_blocks, float* out_f32,
                                __nv_bfloat16* out_bf16, cudaStream_t st);

}  // namespace cfa
