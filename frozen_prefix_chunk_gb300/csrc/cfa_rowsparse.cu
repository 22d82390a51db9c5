// Row-sparse projection backward on the fifth-generation tensor cores.
//
// "POC: stop-gradient through context tokens" (prime-rl), "Mechanism": the
// q/o projections and the dense MLP keep a full-row forward, but their
// backward runs on the kept rows only -- dW = dY[keep]^T X[keep] and
// dX[keep] = dY[keep] W -- because the gradient reaching Y is exactly zero on
// every context row.  Here dY arrives compacted to the kept rows: it is what
// the query-split attention backward produces (dQ exists for the chunk rows
// only), so the q projection's backward reads that dQ as it is.
//
// One persistent kernel, two modes, 128 x 128 output tiles, K in 64-row
// stages:
//   mode 0, dW [out, in] = dY_keep^T X[keep]: A = dY_keep read MN-major by
//     TMA (64 x 64 boxes), B = the kept rows of X gathered with cp.async into
//     the same 128-byte-swizzled MN-major layout (each row of a stage comes
//     from another X row, which a tensor map cannot express);
//   mode 1, dX[keep[i]] = dY_keep[i] W: A = dY_keep K-major (TMA, 64-column x
//     128-row box), B = W [out, in] MN-major (TMA, 64 x 64 boxes); the
//     epilogue scatters each output row to its row of dX.
// Warp roles (256 threads): warps 0-1 load (mode 0: one 64-column slab of
// the gathered rows each, warp 0 lane 0 also the TMA of A; mode 1: warp 0
// lane 0 issues all TMA), warp 2 owns TMEM and issues tcgen05.mma
// (converged warp, elect.sync), warp 3 idles, warps 4-7 are the epilogue
// (TMEM lane quadrant = warp % 4).  Two 128-column fp32 accumulators in TMEM
// let the epilogue of one tile overlap the MMAs of the next.
//
// Split K (when there are fewer tiles than SMs): every split writes an fp32
// partial tile to the workspace.  Each epilogue warp owns 32 rows of the tile
// and a counter of its own per (tile, lane quadrant); the warp that finishes
// its rows last sums their partials in split order -- deterministic -- and
// writes them out.  No barrier spans more than one warp, so a warp that gives
// up on a timed-out wait cannot leave the others blocked.
#include "cfa_kernels.cuh"
#include "cfa_ptx.cuh"
#include "cfa_rowsparse.cuh"

namespace cfa {
namespace {

constexpr int kStages = 6;
constexpr int kStageBytes = 2 * kRsTile * kRsBK * 2;  // A 16 KB + B 16 KB
constexpr int kABytes = kRsTile * kRsBK * 2;
constexpr int kSlabBytes = kRsBK * 128;              // 64 rows x 64 bf16 (128 B)
constexpr int kGatherDepth = 4;                      // cp.async stages in flight per lane
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;
static_assert(kGatherDepth <= kStages, "gather depth within the ring");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ float4 ld_cg_f4(const float* p) {
  return __ldcg(reinterpret_cast<const float4*>(p));
}

struct Unit {
  int tm, tn, tile, split, kb, ke;  // k stages [kb, ke)
};

__device__ __forceinline__ Unit unit_of(const RsArgs& a, long long u) {
  Unit r;
  r.tile = (int)(u / a.splits);
  r.split = (int)(u % a.splits);
  r.tm = r.tile / a.tiles_n;
  r.tn = r.tile % a.tiles_n;
  r.kb = (int)((long long)r.split * a.k_stages / a.splits);
  r.ke = (int)((long long)(r.split + 1) * a.k_stages / a.splits);
  return r;
}

// Final store of one output row (128 fp32 values, columns tn*128 ...).
template <int MODE>
__device__ __forceinline__ void store_row(const RsArgs& a, const Unit& t, int row, const float* v) {
  const int n0 = t.tn * kRsTile;
  if (MODE == 0) {
    const int m = t.tm * kRsTile + row;
    if (m >= a.M) return;
    if (a.out_f32) {
      float* dst = static_cast<float*>(a.out) + (size_t)m * a.N + n0;
#pragma unroll
      for (int g = 0; g < 32; ++g) {
        if (n0 + 4 * g >= a.N) break;
        float4 w = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        if (a.accumulate) {
          const float4 o = *reinterpret_cast<const float4*>(dst + 4 * g);
          w.x += o.x;
          w.y += o.y;
          w.z += o.z;
          w.w += o.w;
        }
        *reinterpret_cast<float4*>(dst + 4 * g) = w;
      }
    } else {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + (size_t)m * a.N + n0;
#pragma unroll
      for (int g = 0; g < 16; ++g) {
        if (n0 + 8 * g >= a.N) break;
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = v[8 * g + e];
        if (a.accumulate) {
          const uint4 o = *reinterpret_cast<const uint4*>(dst + 8 * g);
          const __nv_bfloat162* ob = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 p = __bfloat1622float2(ob[e]);
            f[2 * e] += p.x;
            f[2 * e + 1] += p.y;
          }
        }
        uint4 w;
        w.x = pack_bf16x2(f[0], f[1]);
        w.y = pack_bf16x2(f[2], f[3]);
        w.z = pack_bf16x2(f[4], f[5]);
        w.w = pack_bf16x2(f[6], f[7]);
        *reinterpret_cast<uint4*>(dst + 8 * g) = w;
      }
    }
  } else {
    const int i = t.tm * kRsTile + row;
    if (i >= a.n_keep) return;
    const int r = a.keep[i];
    if (r < 0 || r >= a.n_rows) {
      atomicExch(a.status, -1 /* CFA_ERR_INVALID_ARG: a kept row outside X */);
      return;
    }
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + (size_t)r * a.N + n0;
#pragma unroll
    for (int g = 0; g < 16; ++g) {
      if (n0 + 8 * g >= a.N) break;
      uint4 w;
      w.x = pack_bf16x2(v[8 * g + 0], v[8 * g + 1]);
      w.y = pack_bf16x2(v[8 * g + 2], v[8 * g + 3]);
      w.z = pack_bf16x2(v[8 * g + 4], v[8 * g + 5]);
      w.w = pack_bf16x2(v[8 * g + 6], v[8 * g + 7]);
      *reinterpret_cast<uint4*>(dst + 8 * g) = w;
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(256, 1)
    rowsparse_kernel(const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_b, const RsArgs a) {
  pdl_start();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((long long)blockIdx.x >= a.units) return;

  const uint32_t bars = base + kBarOff;
  const uint32_t bar_full = bars;                    // [kStages]
  const uint32_t bar_empty = bars + 8 * kStages;     // [kStages]
  const uint32_t bar_tfull = bars + 16 * kStages;    // [2]
  const uint32_t bar_tempty = bar_tfull + 16;        // [2]
  const uint32_t bar_drain = bar_tempty + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kBarOff + 240);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kBarOff + 244);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // mode 0: the A copy's expect_tx arrive plus one arrive per gather warp
      mbar_init(bar_full + 8 * s, MODE == 0 ? 3 : 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 4);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{a.limit_ns, abort_flag, a.status};
  const long long u0 = blockIdx.x, ustep = gridDim.x;

  if (warp < 2) {
    // ---------------------------------------------------------- producers --
    if (MODE == 1 && warp == 1) {
      // mode 1 loads everything by TMA from warp 0
    } else {
      const bool tma_lane = warp == 0 && lane == 0;
      int it = 0, signalled = 0;
      bool ok = true;
      // mode 0 gather: this warp's slab (64 columns) of the stage's 64 rows;
      // lane l always moves 16-byte chunk c = l % 8 of rows l / 8 + 4 j
      const int c = lane & 7;
      auto signal = [&](int upto) {
        // the stages before `upto` have landed: make them visible to the
        // tensor core (async proxy) and report them
        fence_proxy_async_smem();
        __syncwarp();
        for (; signalled < upto; ++signalled)
          if (lane == 0) mbar_arrive(bar_full + 8 * (signalled % kStages));
      };
      for (long long u = u0; ok && u < a.units; u += ustep) {
        const Unit t = unit_of(a, u);
        for (int kk = t.kb; kk < t.ke; ++kk, ++it) {
          const int s = it % kStages;
          if (!(ok = warp_wait(W, bar_empty + 8 * s, ((uint32_t)(it / kStages) & 1u) ^ 1u))) break;
          const uint32_t st_a = base + s * kStageBytes, st_b = st_a + kABytes;
          if (MODE == 1) {
            if (tma_lane) {
              mbar_arrive_expect_tx(bar_full + 8 * s, kStageBytes);
              tma_load_2d(st_a, &map_a, bar_full + 8 * s, kk * kRsBK, t.tm * kRsTile);
              tma_load_2d(st_b, &map_b, bar_full + 8 * s, t.tn * kRsTile, kk * kRsBK);
              tma_load_2d(st_b + kSlabBytes, &map_b, bar_full + 8 * s, t.tn * kRsTile + 64,
                          kk * kRsBK);
            }
            __syncwarp();
          } else {
            if (tma_lane) {
              mbar_arrive_expect_tx(bar_full + 8 * s, kABytes);
              tma_load_2d(st_a, &map_a, bar_full + 8 * s, t.tm * kRsTile, kk * kRsBK);
              tma_load_2d(st_a + kSlabBytes, &map_a, bar_full + 8 * s, t.tm * kRsTile + 64,
                          kk * kRsBK);
            }
            const int k0 = kk * kRsBK;
            const int col = t.tn * kRsTile + warp * 64 + c * 8;
            const bool col_ok = col < a.N;
            int idx0 = -1, idx1 = -1;
            if (k0 + lane < a.n_keep) idx0 = a.keep[k0 + lane];
            if (k0 + 32 + lane < a.n_keep) idx1 = a.keep[k0 + 32 + lane];
            const uint32_t slab = st_b + warp * kSlabBytes;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int r = j * 4 + (lane >> 3);  // row of the stage
              const int idx = __shfl_sync(0xffffffffu, j < 8 ? idx0 : idx1, r & 31);
              const bool in_keep = k0 + r < a.n_keep;
              const bool row_ok = idx >= 0 && idx < a.n_rows;
              if (in_keep && !row_ok) atomicExch(a.status, -1 /* kept row outside X */);
              const bool take = in_keep && row_ok && col_ok;
              const __nv_bfloat16* src = take ? a.x + (size_t)idx * a.N + col : a.x;
              cp_async_16(slab + r * 128 + ((c ^ (r & 7)) << 4), src, take ? 16u : 0u);
            }
            cp_async_commit();
            if (it + 1 - signalled >= kGatherDepth) {
              cp_async_wait<kGatherDepth - 1>();
              signal(it + 2 - kGatherDepth);
            }
          }
        }
      }
      if (MODE == 0) {
        cp_async_wait<0>();
        signal(it);
      }
      // unwind: the TMA copies this lane issued have landed before exit
      if (tma_lane)
        for (int i = (it > kStages ? it - kStages : 0); i < it; ++i)
          mbar_wait_bounded(bar_full + 8 * (i % kStages), (uint32_t)(i / kStages) & 1u,
                            kDrainLimitNs);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- MMA --
    constexpr uint32_t idesc = idesc_bf16_f32(128, 128, MODE == 0 ? 1 : 0, 1);
    constexpr uint32_t hi = sw128_desc_hi(1024);
    int it = 0, tc = 0;
    bool ok = true;
    for (long long u = u0; ok && u < a.units; u += ustep, ++tc) {
      const Unit t = unit_of(a, u);
      const int buf = tc & 1;
      if (!(ok = warp_wait(W, bar_tempty + 8 * buf, ((uint32_t)(tc >> 1) & 1u) ^ 1u))) break;
      tc_fence_after_sync();
      const uint32_t d = tmem + (uint32_t)buf * 128u;
      for (int kk = t.kb; kk < t.ke; ++kk, ++it) {
        const int s = it % kStages;
        if (!(ok = warp_wait(W, bar_full + 8 * s, (uint32_t)(it / kStages) & 1u))) break;
        tc_fence_after_sync();
        const uint32_t st_a = base + s * kStageBytes, st_b = st_a + kABytes;
        const uint32_t a_lo = sw128_desc_lo(st_a, MODE == 0 ? kSlabBytes : 16);
        const uint32_t b_lo = sw128_desc_lo(st_b, kSlabBytes);
#pragma unroll
        for (int k = 0; k < kRsBK / 16; ++k) {
          // 16 contraction rows: +2048 B in an MN-major tile, +32 B in a K-major one
          const uint32_t a_off = MODE == 0 ? (uint32_t)k * (2048u >> 4) : (uint32_t)k * 2u;
          mma_ss_warp(d, a_lo + a_off, hi, b_lo + (uint32_t)k * (2048u >> 4), hi, idesc,
                      (kk > t.kb || k > 0) ? 1u : 0u);
        }
        tc_commit_warp(bar_empty + 8 * s);
      }
      if (!ok) break;
      tc_commit_warp(bar_tfull + 8 * buf);
    }
    tc_commit_warp(bar_drain);
    mbar_wait_bounded(bar_drain, 0, kDrainLimitNs);
  } else if (warp >= 4) {
    // ----------------------------------------------------------- epilogue --
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    int tc = 0;
    bool ok = true;
    for (long long u = u0; ok && u < a.units; u += ustep, ++tc) {
      const Unit t = unit_of(a, u);
      const int buf = tc & 1;
      if (!(ok = warp_wait(W, bar_tfull + 8 * buf, (uint32_t)(tc >> 1) & 1u))) break;
      tc_fence_after_sync();
      float v[128];
      {
        uint32_t r[128];
        tmem_ld_x128(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)buf * 128u, r);
#pragma unroll
        for (int e = 0; e < 128; ++e) v[e] = __uint_as_float(r[e]);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * buf);  // the accumulator may be reused
      if (a.splits == 1) {
        store_row<MODE>(a, t, row, v);
        continue;
      }
      // split K: publish this split's partial rows; the warp that adds the
      // last split of its 32 rows sums them
      float* mine = a.part + (((size_t)t.tile * a.splits + t.split) * kRsTile + row) * kRsTile;
#pragma unroll
      for (int g = 0; g < 32; ++g)
        __stcg(reinterpret_cast<float4*>(mine + 4 * g),
               make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
      __threadfence();
      __syncwarp();
      unsigned old = 0;
      if (lane == 0) old = atomicAdd(a.counters + 4 * t.tile + quad, 1u);
      old = __shfl_sync(0xffffffffu, old, 0);
      if (old != (unsigned)(a.splits - 1)) continue;
      __threadfence();
#pragma unroll
      for (int e = 0; e < 128; ++e) v[e] = 0.f;
      for (int sp = 0; sp < a.splits; ++sp) {
        const float* p = a.part + (((size_t)t.tile * a.splits + sp) * kRsTile + row) * kRsTile;
#pragma unroll
        for (int g = 0; g < 32; ++g) {
          const float4 q = ld_cg_f4(p + 4 * g);
          v[4 * g] += q.x;
          v[4 * g + 1] += q.y;
          v[4 * g + 2] += q.z;
          v[4 * g + 3] += q.w;
        }
      }
      store_row<MODE>(a, t, row, v);
      if (lane == 0) a.counters[4 * t.tile + quad] = 0u;  // ready for the next call
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 256);
  }
}

__global__ void keep_index_chunks_kernel(const int32_t* __restrict__ cu_p,
                                         const int32_t* __restrict__ cu_c, int batch,
                                         int total_lc, int32_t* __restrict__ keep) {
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < total_lc; j += gridDim.x * blockDim.x) {
    // window b: cu_c[b] <= j < cu_c[b + 1] (the last such b skips empty windows)
    int lo = 0, hi = batch;  // invariant: cu_c[lo] <= j < cu_c[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu_c[mid] <= j) lo = mid;
      else hi = mid;
    }
    // the packed window b starts at cu_p[b] + cu_c[b]; its chunk follows its
    // Lp_b prefix rows, so chunk row j sits at cu_p[b + 1] + j
    keep[j] = cu_p[lo + 1] + j;
  }
}

}  // namespace

int rowsparse_smem_bytes() { return kSmemBytes; }

cudaError_t launch_rowsparse(const CUtensorMap& map_a, const CUtensorMap& map_b, const RsArgs& a,
                             int grid, cudaStream_t st) {
  void (*k)(const CUtensorMap, const CUtensorMap, const RsArgs) =
      a.mode == 0 ? rowsparse_kernel<0> : rowsparse_kernel<1>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(grid), dim3(256), kSmemBytes, st, map_a, map_b, a);
}

cudaError_t launch_keep_index_chunks(const int32_t* cu_p, const int32_t* cu_c, int batch,
                                     int total_lc, int32_t* keep, cudaStream_t st) {
  if (total_lc <= 0) return cudaSuccess;
  const int threads = 256;
  int blocks = (total_lc + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  keep_index_chunks_kernel<<<blocks, threads, 0, st>>>(cu_p, cu_c, batch, total_lc, keep);
  return cudaGetLastError();
}

}  // namespace cfa
