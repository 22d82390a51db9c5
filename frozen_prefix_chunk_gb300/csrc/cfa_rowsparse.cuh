// Row-sparse projection backward: argument block and launchers shared between
// the host layer (cfa_api.cu) and cfa_rowsparse.cu.
//
// "POC: stop-gradient through context tokens" (prime-rl), "Mechanism",
// row_sparse_linear: for Y = X W^T whose incoming gradient is zero on every
// row but the kept ones, the backward runs on the kept rows only:
//   dW = dY_keep^T X[keep]        (mode 0: M = out, N = in, K = n_keep)
//   dX[keep[i]] = dY_keep[i] W    (mode 1: M = n_keep, N = in, K = out)
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace cfa {

constexpr int kRsTileM = 128;      // output tile: 128 x 256 (one M=128, N=256 MMA shape)
constexpr int kRsTileN = 256;
constexpr int kRsBK = 64;          // contraction rows per pipeline stage
constexpr int kRsMaxSplits = 16;

struct RsArgs {
  int mode;                 // 0: dW, 1: dX
  int M, N, K;              // output M x N, contraction K
  int tiles_n, tiles;       // 128 x 256 output tiles (n fastest)
  int k_stages, splits;     // 64-row stages of K; K split into `splits` ranges
  long long units;          // tiles * splits work units, CTA c takes c, c + grid, ...
  const int32_t* keep;      // [n_keep] rows of X / dX
  int n_keep, n_rows;
  const __nv_bfloat16* x;   // mode 0: X [n_rows, N], gathered by `keep`
  void* out;                // mode 0: dW [M, N] (fp32 or bf16); mode 1: dX [n_rows, N] bf16
  int out_f32, accumulate;  // mode 0: output type, dW += instead of dW =
  float* part;              // splits > 1: fp32 partial tiles [tiles][splits][128][256]
  unsigned* counters;       // splits > 1: [tiles][4 lane quadrants], zero before the launch
  int* status;              // workspace status word
  unsigned long long limit_ns;
  int cluster;              // mode 1, splits > 1: the splits of a tile are one cluster of
                            // `splits` CTAs that exchange their partials through L2 and
                            // each sum a share of the rows (no counters); CTA 0 then
                            // clears the status word itself
};

int rowsparse_smem_bytes();
// map_a: mode 0 dY [n_keep, out] in 64 x 64 boxes (read MN-major), mode 1 dY
// in 64-column x 128-row boxes (K-major); map_b: mode 0 X [n_rows, in] in
// 64-column x 1-row boxes (4-row gathers), mode 1 W [out, in] in 64 x 64
// boxes (MN-major).  Grid: at most one CTA per SM.
// map_o: mode 0 dW [M, N] (fp32 or bf16) in 128-byte x 32-row boxes, used
// when dW is overwritten; map_p: the split partials [tiles * splits * 128,
// 256] fp32 in 32 x 32 boxes, used when splits > 1 (both 128-byte swizzled).
// map_xt: mode 0 X [n_rows, in] in 64 x 64 boxes (stages whose kept rows are
// one run of consecutive rows).
// Whether `clusters` clusters of `splits` CTAs of the mode-1 kernel can be
// resident at once on this device (the cluster path needs every split of
// every tile running together).
bool rowsparse_clusters_fit(int splits, int clusters);
cudaError_t launch_rowsparse(const CUtensorMap& map_a, const CUtensorMap& map_b,
                             const CUtensorMap& map_o, const CUtensorMap& map_p,
                             const CUtensorMap& map_xt, const RsArgs& a, int grid,
                             cudaStream_t st);
cudaError_t launch_keep_index_chunks(const int32_t* cu_p, const int32_t* cu_c, int batch,
                                     int total_lc, int32_t* keep, cudaStream_t st);

}  // namespace cfa
