// GPU check of ex2_poly_x2 (cfa_ptx.cuh), the forward's polynomial 2^x for a
// pair, against 2^x in double precision on the host and against the special
// function unit's ex2.approx on the same inputs.  Exits 0 when
//   * every x in [-125, 9] has relative error below 1e-4 (the polynomial's
//     fitted bound is 7.5e-5; fp32 evaluation adds a few ulps),
//   * every x below -125 (including -inf) gives a finite value in [0, 2^-124]
//     (the documented underflow tail: the argument is clamped at -126),
//   * the two halves of a pair are independent (pairs are checked with the
//     halves swapped).
#include <cmath>
#include <cstdio>
#include <vector>

#include "cfa_ptx.cuh"

__global__ void ex2_pairs(const float* x, float* y_poly, float* y_sfu, int n_pairs) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_pairs) return;
  const uint64_t v = cfa::f2(x[2 * i], x[2 * i + 1]);
  float a, b;
  cfa::f2_split(cfa::ex2_poly_x2(v), a, b);
  y_poly[2 * i] = a;
  y_poly[2 * i + 1] = b;
  cfa::f2_split(cfa::ex2_sfu_x2(v), a, b);
  y_sfu[2 * i] = a;
  y_sfu[2 * i + 1] = b;
}

int main() {
  std::vector<float> x;
  const int dense = 1 << 21;
  for (int i = 0; i < dense; ++i) x.push_back(-140.f + 149.f * (float)i / (float)(dense - 1));
  const float special[] = {-INFINITY, -1000.f, -200.f, -126.5f, -126.f, -125.5f, -125.f, -0.5f,
                           -0.49999997f, -1e-30f, 0.f, 1e-30f, 0.5f, 0.50000006f, 1.f, 7.5f,
                           8.f, 8.5f, 9.f};
  for (float s : special) x.push_back(s);
  // the same values with the halves of each pair swapped
  const size_t base = x.size();
  for (size_t i = 0; i + 1 < base; i += 2) {
    x.push_back(x[i + 1]);
    x.push_back(x[i]);
  }
  if (x.size() & 1) x.push_back(0.f);
  const int n = (int)x.size(), pairs = n / 2;
  float *dx, *dp, *ds;
  if (cudaMalloc(&dx, n * 4) || cudaMalloc(&dp, n * 4) || cudaMalloc(&ds, n * 4)) {
    std::printf("cudaMalloc failed\n");
    return 2;
  }
  cudaMemcpy(dx, x.data(), n * 4, cudaMemcpyHostToDevice);
  ex2_pairs<<<(pairs + 255) / 256, 256>>>(dx, dp, ds, pairs);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    std::printf("kernel failed\n");
    return 2;
  }
  std::vector<float> yp(n), ys(n);
  cudaMemcpy(yp.data(), dp, n * 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(ys.data(), ds, n * 4, cudaMemcpyDeviceToHost);
  double max_rel = 0.0, max_rel_sfu = 0.0, worst_x = 0.0;
  int bad = 0;
  for (int i = 0; i < n; ++i) {
    const double xi = x[i], p = yp[i];
    if (xi >= -125.0) {
      const double ref = std::exp2(xi);
      const double rel = std::fabs(p / ref - 1.0);
      if (rel > max_rel) {
        max_rel = rel;
        worst_x = xi;
      }
      if (ys[i] > 0.f) max_rel_sfu = std::fmax(max_rel_sfu, std::fabs(p / (double)ys[i] - 1.0));
      if (!(rel < 1e-4)) ++bad;
    } else if (!(p >= 0.0 && p <= std::ldexp(1.0, -124))) {
      ++bad;
    }
  }
  std::printf("values %d bad %d max_rel_err %.3e at x=%.6g max_rel_vs_sfu %.3e\n", n, bad, max_rel,
              worst_x, max_rel_sfu);
  return bad == 0 ? 0 : 1;
}
