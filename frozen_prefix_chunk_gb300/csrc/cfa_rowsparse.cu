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
// One persistent kernel, two modes, 128 x 256 output tiles, K in 64-row
// stages (48 KB each, four in flight):
//   mode 0, dW [out, in] = dY_keep^T X[keep]: A = dY_keep read MN-major by
//     TMA (64 x 64 boxes), B = the kept rows of X gathered with cp.async into
//     the same 128-byte-swizzled MN-major layout (each row of a stage comes
//     from another X row, which a tensor map cannot express);
//   mode 1, dX[keep[i]] = dY_keep[i] W: A = dY_keep K-major (TMA, 64-column x
//     128-row box), B = W [out, in] MN-major (TMA, 64 x 64 boxes); the
//     epilogue scatters each output row to its row of dX.
// Warp roles (288 threads): warps 0-3 load (mode 0: one 64-column slab of
// the gathered rows each, with the next stage's keep indices fetched a stage
// ahead so their latency stays off the copy path, and warp 0 lane 0 also the
// TMA of A; mode 1: lane 0 of warps 0-2 issues A and the two halves of B),
// warps 4-7 are the epilogue (TMEM lane quadrant = warp % 4), warp 8 owns
// TMEM and issues tcgen05.mma
// (converged warp, elect.sync).  Two 256-column fp32 accumulators in TMEM let
// the epilogue of one tile overlap the MMAs of the next.  The epilogue stages
// each 32 x 32 block of its rows through shared memory, so that every global
// store instruction writes four whole rows' 128-byte runs instead of 32
// scattered pieces.
//
// Split K, mode 1 (dX, whose kept rows make few tiles): the splits of a tile
// run as one thread-block cluster.  After its K range each CTA stores its fp32
// partial tile to the workspace (TMA tile stores), the CTAs signal one
// another through mbarriers (remote arrives, release / acquire at cluster
// scope), and CTA rank r of the cluster copies rows [r * 128 / splits,
// (r + 1) * 128 / splits) of every split's partial from L2 into its shared
// memory (bulk copies, all in flight at once), sums them in split order
// (deterministic, the same sums as the global-memory path below) and writes
// them out.  No per-tile counter, no memset.  Summing over distributed shared
// memory instead ran at about 12 bytes a cycle per SM, several times slower
// than these copies.  Every wait is bounded; a CTA whose wait for its peers
// runs out reads no partial.
//
// Split K otherwise (when there are fewer tiles than SMs): every split writes an fp32
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

constexpr int kStages = 4;
constexpr int kABytes = kRsTileM * kRsBK * 2;          // 16 KB
constexpr int kBBytes = kRsTileN * kRsBK * 2;          // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSlabBytes = kRsBK * 128;                // 64 rows x 64 bf16 (128 B)
constexpr int kStgStride = 36;                         // put4 staging row: 32 floats + 4 pad
constexpr int kStgBufBytes = 32 * 128;                 // TMA-store staging: 32 rows x 128 B
constexpr int kStgWarpBytes = 2 * kStgBufBytes;        // two buffers per epilogue warp
constexpr int kStgOff = kStages * kStageBytes;
constexpr int kBarOff = kStgOff + 4 * kStgWarpBytes;
static_assert(32 * kStgStride * 4 <= kStgWarpBytes, "put4 staging fits a warp's buffers");
constexpr int kSmemBytes = kBarOff + 256 + 1024;
constexpr int kThreads = 288;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// Four rows of a 2-D tensor, given by their row coordinates, each one box of
// 64 columns x 1 row, into 4 consecutive 128-byte rows of shared memory
// (swizzled by the tensor map's 128-byte mode like any tile).  Rows outside
// the tensor (a negative or too large coordinate) read as zero.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int col, int r0, int r1, int r2, int r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Tile store (or add) of a 128-byte-wide box from shared memory; completion
// tracked per thread with bulk groups.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int c0, int c1,
                                             uint32_t src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   map),
               "r"(c0), "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// ------------------------------------------------------------ cluster --
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this thread's
// (and, cumulatively, what it has observed of its CTA's) earlier writes.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n"
      ".reg .pred p;\n"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Bounded wait for an exchange among the cluster's CTAs (acquire at cluster
// scope, so the peers' shared-memory writes released by their arrivals are
// visible).  `drain`: ignore the CTA's abort flag (used while unwinding).
__device__ __forceinline__ bool cluster_wait(const Waiter& w, uint32_t bar, uint32_t parity,
                                             bool drain) {
  bool ok = mbar_try_wait_acq_cluster(bar, parity);
  if (!ok) {
    const uint64_t t0 = global_timer_ns();
    const uint64_t lim = drain ? kDrainLimitNs : w.limit_ns;
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait_acq_cluster(bar, parity)) {
        ok = true;
        break;
      }
      if ((it & 15u) == 0u) {
        if (!drain && *w.abort) break;
        if (global_timer_ns() - t0 > lim) {
          if (!drain) {
            *w.abort = 1;
            atomicExch(w.status, -5 /* CFA_ERR_DEVICE_TIMEOUT */);
          }
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}
// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory, completing on mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory to global memory, tracked by the thread's bulk
// groups.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}

// Cluster split K: this warp's rows of the CTA's share of the tile, summed
// over the SP partial rows staged at `base` (split k's row j at
// base + (k * R + j) * 1024, R = 128 / SP) in split order, written out as
// bf16.  Lane l takes columns 4l .. 4l + 3 and 128 + 4l .. 128 + 4l + 3, so
// that each shared-memory load reads 512 contiguous bytes (no bank conflict)
// and each store writes 256 contiguous bytes of the row.  Rows go in batches
// of 8 / SP, every load of a batch issued before any is added (16 in flight
// per lane; one row at a time, the loads' latency made a row about 600
// cycles).
template <int SP>
__device__ __forceinline__ void cluster_sum_rows(const RsArgs& a, int tm, int tn, uint32_t base,
                                                 uint32_t rank, int quad, int lane, int my_keep) {
  constexpr int R = kRsTileM / SP, RPW = R / 4;
  constexpr int RB = (8 / SP) < RPW ? 8 / SP : RPW;
  static_assert(RPW % RB == 0, "whole batches of rows");
  const int n0 = tn * kRsTileN + 4 * lane, n1 = n0 + 128;  // output columns
  const bool vec = n1 + 4 <= a.N && (a.N & 3) == 0 && (reinterpret_cast<uintptr_t>(a.out) & 7u) == 0;
  for (int rb = 0; rb < RPW; rb += RB) {
    float4 v[RB][SP][2];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const int j = quad * RPW + rb + r;  // row within the CTA's share
#pragma unroll
      for (int k = 0; k < SP; ++k) {
        const uint32_t src = base + (uint32_t)((k * R + j) * (kRsTileN * 4) + 16 * lane);
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v[r][k][0].x), "=f"(v[r][k][0].y), "=f"(v[r][k][0].z), "=f"(v[r][k][0].w)
                     : "r"(src));
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v[r][k][1].x), "=f"(v[r][k][1].y), "=f"(v[r][k][1].z), "=f"(v[r][k][1].w)
                     : "r"(src + 512u));
      }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < SP; ++k) {
        s[0] += v[r][k][0].x; s[1] += v[r][k][0].y; s[2] += v[r][k][0].z; s[3] += v[r][k][0].w;
        s[4] += v[r][k][1].x; s[5] += v[r][k][1].y; s[6] += v[r][k][1].z; s[7] += v[r][k][1].w;
      }
      const int j = quad * RPW + rb + r;
      if (quad == 0 && lane == 0) CFA_TRACE(5, 1 + rb + r, 0);
      const int i = tm * kRsTileM + (int)rank * R + j;  // kept-row index
      const int keep_r = __shfl_sync(0xffffffffu, my_keep, rb + r);  // fetched by lane rb + r
      if (i >= a.n_keep) continue;
      if (keep_r < 0 || keep_r >= a.n_rows) {
        if (lane == 0) atomicExch(a.status, -1 /* kept row outside X */);
        continue;
      }
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) + (size_t)keep_r * a.N;
      if (vec) {
        *reinterpret_cast<uint2*>(orow + n0) = make_uint2(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]));
        *reinterpret_cast<uint2*>(orow + n1) = make_uint2(pack_bf16x2(s[4], s[5]), pack_bf16x2(s[6], s[7]));
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (n0 + e < a.N) orow[n0 + e] = __float2bfloat16_rn(s[e]);
          if (n1 + e < a.N) orow[n1 + e] = __float2bfloat16_rn(s[4 + e]);
        }
      }
      if (quad == 0 && lane == 0) CFA_TRACE(5, 1 + rb + r, 1);
    }
  }
}
// Hardware barrier over every thread of the cluster: used once, right after
// the mbarriers are initialised and before any remote arrive, by all threads
// of all CTAs (no CTA can leave before it).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Barrier among the four epilogue warps (named barrier 1, 128 threads).
__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}
// The same barrier, returning whether `p` holds in all four warps.
__device__ __forceinline__ bool epilogue_all(bool p) {
  uint32_t r;
  asm volatile(
      "{\n"
      ".reg .pred a, b;\n"
      "setp.ne.u32 a, %1, 0;\n"
      "bar.red.and.pred b, 1, 128, a;\n"
      "selp.u32 %0, 1, 0, b;\n"
      "}\n"
      : "=r"(r)
      : "r"((uint32_t)p)
      : "memory");
  return r != 0;
}
// The cluster path: a CTA's partial staged in the freed pipeline stages at
// this row stride (256 floats + 16 bytes, so that the lanes' row-per-thread
// writes spread over the banks), and later the 128 partial rows it sums
// copied in at 1 KB each.
constexpr int kClRowBytes = 1040;
static_assert(kRsTileM * kClRowBytes <= kStages * kStageBytes, "staged partial fits the stages");
static_assert(kRsTileM * kRsTileN * 4 <= kStages * kStageBytes, "partial rows fit the stages");

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

// Walks a CTA's (unit, k stage) sequence: units c, c + grid, ... and the k
// stages of each.
struct StageIter {
  long long u;
  Unit t;
  int kk;
  bool valid;
  __device__ __forceinline__ void start(const RsArgs& a, long long u0) {
    u = u0;
    valid = u < a.units;
    if (valid) {
      t = unit_of(a, u);
      kk = t.kb;
    }
  }
  __device__ __forceinline__ void next(const RsArgs& a, long long ustep) {
    if (++kk < t.ke) return;
    u += ustep;
    valid = u < a.units;
    if (valid) {
      t = unit_of(a, u);
      kk = t.kb;
    }
  }
};

// Output of 4 consecutive columns (n, n+1, n+2, n+3) of one row at `dst`:
// fp32 or bf16, overwritten or accumulated.
__device__ __forceinline__ void put4(const RsArgs& a, void* dst, float4 q, bool f32) {
  if (f32) {
    float4* p = static_cast<float4*>(dst);
    if (a.accumulate) {
      const float4 o = *p;
      q.x += o.x;
      q.y += o.y;
      q.z += o.z;
      q.w += o.w;
    }
    *p = q;
  } else {
    uint2* p = static_cast<uint2*>(dst);
    if (a.accumulate) {
      const uint2 o = *p;
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o.y));
      q.x += lo.x;
      q.y += lo.y;
      q.z += hi.x;
      q.w += hi.y;
    }
    *p = make_uint2(pack_bf16x2(q.x, q.y), pack_bf16x2(q.z, q.w));
  }
}

// Where tile row `r` (0..127) of unit t goes, or null when it has no output
// row: mode 0 row tm*128 + r of dW; mode 1 row keep[tm*128 + r] of dX
// (`keep_r` = that index, fetched by the caller).
template <int MODE>
__device__ __forceinline__ uint8_t* out_row(const RsArgs& a, const Unit& t, int r, int keep_r) {
  const size_t esz = (MODE == 0 && a.out_f32) ? 4 : 2;
  if (MODE == 0) {
    const int m = t.tm * kRsTileM + r;
    if (m >= a.M) return nullptr;
    return static_cast<uint8_t*>(a.out) + (size_t)m * a.N * esz;
  }
  const int i = t.tm * kRsTileM + r;
  if (i >= a.n_keep || keep_r < 0 || keep_r >= a.n_rows) return nullptr;
  return static_cast<uint8_t*>(a.out) + (size_t)keep_r * a.N * esz;
}

template <int MODE, bool CL>
__global__ void __launch_bounds__(kThreads, 1)
    rowsparse_kernel(const __grid_constant__ CUtensorMap map_a,
                     const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_o,
                     const __grid_constant__ CUtensorMap map_p,
                     const __grid_constant__ CUtensorMap map_xt, const RsArgs a) {
  // map_b: mode 0 X [n_rows, in] in 64-column x 1-row boxes (gathered),
  //        mode 1 W [out, in] in 64 x 64 boxes
  // map_o: mode 0 dW in 128-byte x 32-row boxes (TMA stores); map_p: the
  //        split partials [tiles * splits * 128, 256] fp32 in 32 x 32 boxes
  // map_xt: mode 0 X in 64 x 64 boxes, for stages whose 64 kept rows are one
  //        run of consecutive rows (the chunk rows of a window): one tile
  //        copy per slab instead of 16 gathers, same shared-memory layout
  pdl_start();
  // cluster path: no memset before the launch; the first CTA clears the
  // status word (a device wait gives up only after its wall-clock limit,
  // long after this store, so no error of this launch is cleared)
  if (CL && blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // (the cluster path launches exactly one CTA per unit: no CTA returns here)
  if ((long long)blockIdx.x >= a.units) return;

  const uint32_t bars = base + kBarOff;
  const uint32_t bar_full = bars;                    // [kStages]
  const uint32_t bar_empty = bars + 8 * kStages;     // [kStages]
  const uint32_t bar_tfull = bars + 16 * kStages;    // [2]
  const uint32_t bar_tempty = bar_tfull + 16;        // [2]
  const uint32_t bar_drain = bar_tempty + 16;
  const uint32_t bar_staged = bar_drain + 8;  // cluster path: every split's partial stored
  const uint32_t bar_rows = bar_drain + 16;   // cluster path: this CTA's partial rows copied in
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + kBarOff + 240);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + kBarOff + 244);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // mode 0: one expect_tx arrive per gather warp (warp 0's covers A too);
      // mode 1: one per loading warp (A; B's first half; B's second half)
      mbar_init(bar_full + 8 * s, MODE == 0 ? 4 : 3);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, 4);
    }
    mbar_init(bar_drain, 1);
    if (CL) {
      mbar_init(bar_staged, (uint32_t)a.splits);
      mbar_init(bar_rows, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  // every CTA of the cluster has initialised its barriers before any remote
  // arrive
  if (CL) cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{a.limit_ns, abort_flag, a.status};
  const long long u0 = blockIdx.x, ustep = gridDim.x;

  if (warp < 4) {
    // ---------------------------------------------------------- producers --
    if (MODE == 1 && warp > 2) {
      // mode 1 loads by TMA from warps 0-2
    } else {
      const bool leader = lane == 0;
      int it = 0;
      bool ok = true;
      // Lane l < 16 gathers rows 4l .. 4l + 3 of a stage and holds their keep
      // indices.  Rows past n_keep gather row 0 (their dY rows are
      // zero-filled, so they add nothing); a kept index outside X gathers row
      // n_rows, past the end, which the copy fills with zeros.
      auto fetch_idx = [&](const StageIter& st, int (&r)[4]) {
        r[0] = r[1] = r[2] = r[3] = 0;
        if (MODE != 0 || !st.valid || lane >= 16) return;
        const int k0 = st.kk * kRsBK + 4 * lane;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (k0 + q < a.n_keep) r[q] = a.keep[k0 + q];
      };
      StageIter cur;
      cur.start(a, u0);
      int nidx[4];
      fetch_idx(cur, nidx);
      for (; ok && cur.valid; ++it) {
        const Unit t = cur.t;
        const int kk = cur.kk;
        int g[4] = {nidx[0], nidx[1], nidx[2], nidx[3]};
        StageIter nxt = cur;
        nxt.next(a, ustep);
        fetch_idx(nxt, nidx);  // a stage ahead: consumed next iteration
        if (MODE == 0) {
          // a kept row outside X reads as zero; report it
          bool bad = false;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (g[q] < 0 || g[q] >= a.n_rows) {
              g[q] = a.n_rows;
              bad = true;
            }
          if (warp == 0 && bad) atomicExch(a.status, -1 /* a kept row outside X */);
        }
        const int s = it % kStages;
        if (leader) CFA_TRACE(warp, it, 0);
        if (!(ok = warp_wait(W, bar_empty + 8 * s, ((uint32_t)(it / kStages) & 1u) ^ 1u))) break;
        if (leader) CFA_TRACE(warp, it, 1);
        const uint32_t st_a = base + s * kStageBytes, st_b = st_a + kABytes;
        if (MODE == 1) {
          // three warps issue a stage's copies side by side: warp 0 A, warps
          // 1 and 2 a half of B each (a warp issuing all five took about 400
          // cycles a stage, more than the stage's MMAs)
          if (leader && warp == 0) {
            mbar_arrive_expect_tx(bar_full + 8 * s, kABytes);
            tma_load_2d(st_a, &map_a, bar_full + 8 * s, kk * kRsBK, t.tm * kRsTileM);
          } else if (leader) {
            constexpr int kHalf = kRsTileN / 128;  // 64-column slabs per half of B
            mbar_arrive_expect_tx(bar_full + 8 * s, kBBytes / 2);
#pragma unroll
            for (int h = (warp - 1) * kHalf; h < warp * kHalf; ++h)
              tma_load_2d(st_b + h * kSlabBytes, &map_b, bar_full + 8 * s,
                          t.tn * kRsTileN + h * 64, kk * kRsBK);
          }
        } else {
          // warp w: its 64-column slab of the stage's 64 kept rows -- one tile
          // copy when they are 64 consecutive rows of X, else one 4-row
          // gather per lane 0..15; warp 0 also loads A.  The expected bytes
          // are posted before any of the warp's copies is issued.
          const int run0 = __shfl_sync(0xffffffffu, g[0], 0);
          const bool mine = lane >= 16 || (g[0] == run0 + 4 * lane && g[1] == g[0] + 1 &&
                                           g[2] == g[0] + 2 && g[3] == g[0] + 3);
          const bool run = __all_sync(0xffffffffu, mine) && (kk + 1) * kRsBK <= a.n_keep &&
                           run0 + kRsBK <= a.n_rows;
          if (leader)
            mbar_arrive_expect_tx(bar_full + 8 * s, (warp == 0 ? kABytes : 0) + kSlabBytes);
          __syncwarp();
          if (leader && warp == 0) {
            tma_load_2d(st_a, &map_a, bar_full + 8 * s, t.tm * kRsTileM, kk * kRsBK);
            tma_load_2d(st_a + kSlabBytes, &map_a, bar_full + 8 * s, t.tm * kRsTileM + 64,
                        kk * kRsBK);
          }
          if (run) {
            if (leader)
              tma_load_2d(st_b + warp * kSlabBytes, &map_xt, bar_full + 8 * s,
                          t.tn * kRsTileN + warp * 64, run0);
          } else if (lane < 16) {
            tma_gather4(st_b + warp * kSlabBytes + lane * 512, &map_b, bar_full + 8 * s,
                        t.tn * kRsTileN + warp * 64, g[0], g[1], g[2], g[3]);
          }
        }
        if (leader) CFA_TRACE(warp, it, 2);
        __syncwarp();
        cur = nxt;
      }
      // unwind: the copies this lane issued have landed before exit
      if (leader)
        for (int i = (it > kStages ? it - kStages : 0); i < it; ++i)
          mbar_wait_bounded(bar_full + 8 * (i % kStages), (uint32_t)(i / kStages) & 1u,
                            kDrainLimitNs);
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------------- MMA --
    constexpr uint32_t idesc = idesc_bf16_f32(kRsTileM, kRsTileN, MODE == 0 ? 1 : 0, 1);
    constexpr uint32_t hi = sw128_desc_hi(1024);
    int it = 0, tc = 0;
    bool ok = true;
    for (long long u = u0; ok && u < a.units; u += ustep, ++tc) {
      const Unit t = unit_of(a, u);
      const int buf = tc & 1;
      if (!(ok = warp_wait(W, bar_tempty + 8 * buf, ((uint32_t)(tc >> 1) & 1u) ^ 1u))) break;
      tc_fence_after_sync();
      const uint32_t d = tmem + (uint32_t)buf * kRsTileN;
      for (int kk = t.kb; kk < t.ke; ++kk, ++it) {
        const int s = it % kStages;
        CFA_TRACE(4, it, 0);
        if (!(ok = warp_wait(W, bar_full + 8 * s, (uint32_t)(it / kStages) & 1u))) break;
        CFA_TRACE(4, it, 1);
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
  } else if (CL) {
    // ------------------------------------------- epilogue, cluster split K --
    // One unit per CTA; its split is the CTA's rank in the cluster.
    const int quad = warp & 3;
    const Unit t = unit_of(a, u0);
    const int splits = a.splits;
    const uint32_t rank = cluster_ctarank();
    const int R = kRsTileM / splits;  // rows of the tile this CTA sums
    // lane j < R / 4 fetches the keep index of this warp's row j of the sum
    // now, so that its latency is off the reduction
    int my_keep = -1;
    {
      const int i = t.tm * kRsTileM + (int)rank * R + quad * (R / 4) + lane;
      if (lane < R / 4 && i < a.n_keep) my_keep = a.keep[i];
    }
    if (quad == 0 && lane == 0) CFA_TRACE(5, 0, 0);
    bool ok = warp_wait(W, bar_tfull, 0u);
    if (quad == 0 && lane == 0) CFA_TRACE(5, 0, 1);
    if (ok) {
      // this split's 128 x 256 fp32 partial to the workspace: each lane
      // stages its tile row in the freed pipeline stages and sends it with
      // one 1 KB bulk copy
      tc_fence_after_sync();
      const int row = quad * 32 + lane;
      const uint32_t srow = base + (uint32_t)(row * kClRowBytes);
#pragma unroll
      for (int h = 0; h < kRsTileN / 128; ++h) {
        uint32_t r[128];
        tmem_ld_x128(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(h * 128), r);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(srow + (uint32_t)(h * 512 + 16 * j)),
                       "r"(r[4 * j]), "r"(r[4 * j + 1]), "r"(r[4 * j + 2]), "r"(r[4 * j + 3])
                       : "memory");
      }
      fence_proxy_async_smem();
      bulk_store(a.part + ((size_t)(t.tile * splits + t.split) * kRsTileM + row) * kRsTileN, srow,
                 (uint32_t)(kRsTileN * 4));
      bulk_commit();
    }
    // the stores have completed, and are ordered before the release below
    bulk_wait<0>();
    fence_proxy_async_global();
    __syncwarp();
    ok = epilogue_all(ok);
    if (quad == 0 && lane == 0) CFA_TRACE(5, 0, 2);
    // one arrival per CTA on every CTA's `staged` barrier (this one's too)
    if (warp == 4 && lane < splits) {
      asm volatile("fence.acq_rel.cluster;" ::: "memory");
      mbar_arrive_remote(mapa_shared(bar_staged, (uint32_t)lane));
    }
    if (ok) ok = cluster_wait(W, bar_staged, 0u, false);
    ok = epilogue_all(ok);  // the same branch in all four warps
    if (quad == 0 && lane == 0) CFA_TRACE(5, 0, 3);
    if (ok) {
      // rows [rank * R, rank * R + R) of every split's partial into the freed
      // pipeline stages (split k's row j at base + (k * R + j) * 1 KB): one
      // 1 KB bulk copy per thread, all on one mbarrier
      fence_proxy_async_global();
      if (warp == 4 && lane == 0) mbar_arrive_expect_tx(bar_rows, (uint32_t)(kRsTileM * kRsTileN * 4));
      epilogue_sync();
      const int e = (int)threadIdx.x - 128;  // 0 .. 127 = k * R + j
      const int k = e / R, jr = e % R;
      const float* src = a.part + ((size_t)(t.tile * splits + k) * kRsTileM + (size_t)rank * R + jr) *
                                      kRsTileN;
      bulk_load(base + (uint32_t)(e * kRsTileN * 4), src, (uint32_t)(kRsTileN * 4), bar_rows);
      ok = warp_wait(W, bar_rows, 0u);
      if (quad == 0 && lane == 0) CFA_TRACE(5, 0, 4);
      if (ok) {
        if (splits == 2)
          cluster_sum_rows<2>(a, t.tm, t.tn, base, rank, quad, lane, my_keep);
        else if (splits == 4)
          cluster_sum_rows<4>(a, t.tm, t.tn, base, rank, quad, lane, my_keep);
        else
          cluster_sum_rows<8>(a, t.tm, t.tn, base, rank, quad, lane, my_keep);
      }
      if (!ok) mbar_wait_bounded(bar_rows, 0u, kDrainLimitNs);  // no copy left in flight
    }
    if (quad == 0 && lane == 0) CFA_TRACE(5, 0, 5);
  } else if (warp >= 4) {
    // ----------------------------------------------------------- epilogue --
    // Warp q owns tile rows 32q .. 32q + 31 (its TMEM lane quadrant).
    //  * dW overwritten, and split partials: each 32-row x 128-byte block is
    //    written (128-byte swizzled) into one of the warp's two staging
    //    buffers and sent by a TMA tile store;
    //  * dW accumulated and dX (rows scattered by the keep index): the block
    //    goes through padded staging rows and lanes read back 4 rows x 8
    //    column groups per instruction, so each global access covers whole
    //    128-byte row runs.
    const int quad = warp & 3;
    uint8_t* stg_g = gbase + kStgOff + quad * kStgWarpBytes;
    const uint32_t stg_s = base + kStgOff + quad * kStgWarpBytes;
    float* stg = reinterpret_cast<float*>(stg_g);
    const int rr0 = lane >> 3, cg = lane & 7;  // read-back: row rr0 + 4 i, columns 4 cg ..
    const bool f32 = MODE == 0 && a.out_f32;
    const bool tma_out = MODE == 0 && !a.accumulate;
    const size_t esz = f32 ? 4 : 2;
    int sb = 0;  // staging buffer for the next TMA store
    // one 128-byte row segment per lane (w: 32 words) -> TMA store at (c0, r0)
    auto stage_store = [&](const CUtensorMap* map, int c0, int r0, const uint32_t* w) {
      if (lane == 0) bulk_wait_read<1>();  // buffer sb no longer read by its last store
      __syncwarp();
      uint8_t* b = stg_g + sb * kStgBufBytes;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(b + lane * 128 + ((j ^ (lane & 7)) << 4)) =
            make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(map, c0, r0, stg_s + sb * kStgBufBytes);
        bulk_commit();
      }
      sb ^= 1;
    };
    int tc = 0;
    bool ok = true;
    for (long long u = u0; ok && u < a.units; u += ustep, ++tc) {
      const Unit t = unit_of(a, u);
      const int buf = tc & 1;
      int my_keep = -1;
      if (MODE == 1) {
        const int i = t.tm * kRsTileM + quad * 32 + lane;
        if (i < a.n_keep) {
          my_keep = a.keep[i];
          if (my_keep < 0 || my_keep >= a.n_rows) atomicExch(a.status, -1 /* kept row outside X */);
        }
      }
      if (quad == 0 && lane == 0) CFA_TRACE(5, tc, 0);
      if (!(ok = warp_wait(W, bar_tfull + 8 * buf, (uint32_t)(tc >> 1) & 1u))) break;
      if (quad == 0 && lane == 0) CFA_TRACE(5, tc, 1);
      tc_fence_after_sync();
      // output rows of the 8 read-back rows of this lane (put4 path)
      uint8_t* orow[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = rr0 + 4 * i;
        orow[i] = out_row<MODE>(a, t, quad * 32 + rr, __shfl_sync(0xffffffffu, my_keep, rr));
      }
      const bool split = a.splits > 1;
      const int prow0 = ((t.tile * a.splits + t.split) * kRsTileM) + quad * 32;
      if (!split && !tma_out) {
        if (lane == 0) bulk_wait_read<0>();  // the padded staging overlaps both buffers
        __syncwarp();
      }
      for (int h = 0; h < kRsTileN / 128; ++h) {
        uint32_t r[128];
        tmem_ld_x128(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)buf * kRsTileN + h * 128, r);
        if (quad == 0 && lane == 0) CFA_TRACE(5, tc, 2 + h);
        if (h == kRsTileN / 128 - 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_tempty + 8 * buf);  // the accumulator may be reused
        }
        if (split) {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) stage_store(&map_p, h * 128 + ch * 32, prow0, r + ch * 32);
        } else if (tma_out) {
          const int c0 = t.tn * kRsTileN + h * 128;
          const int r0 = t.tm * kRsTileM + quad * 32;
          if (f32) {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) stage_store(&map_o, c0 + ch * 32, r0, r + ch * 32);
          } else {
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
              uint32_t pk[32];
#pragma unroll
              for (int e = 0; e < 32; ++e)
                pk[e] = pack_bf16x2(__uint_as_float(r[ch * 64 + 2 * e]),
                                    __uint_as_float(r[ch * 64 + 2 * e + 1]));
              stage_store(&map_o, c0 + ch * 64, r0, pk);
            }
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            __syncwarp();  // the previous block has been read back
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(stg + lane * kStgStride + 4 * j) =
                  make_uint4(r[ch * 32 + 4 * j], r[ch * 32 + 4 * j + 1], r[ch * 32 + 4 * j + 2],
                             r[ch * 32 + 4 * j + 3]);
            __syncwarp();
            const int n = t.tn * kRsTileN + h * 128 + ch * 32 + 4 * cg;  // output column
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = rr0 + 4 * i;
              const float4 q = *reinterpret_cast<const float4*>(stg + rr * kStgStride + 4 * cg);
              if (orow[i] && n < a.N) put4(a, orow[i] + (size_t)n * esz, q, f32);
            }
          }
        }
      }
      if (quad == 0 && lane == 0) CFA_TRACE(5, tc, 4);
      if (!split) continue;
      // split K: the partial rows are in global memory (async proxy) before
      // the count; the warp that adds the last split of its 32 rows sums them
      if (lane == 0) {
        bulk_wait<0>();
        fence_proxy_async_global();
      }
      __threadfence();
      __syncwarp();
      unsigned old = 0;
      if (lane == 0) old = atomicAdd(a.counters + 4 * t.tile + quad, 1u);
      old = __shfl_sync(0xffffffffu, old, 0);
      if (quad == 0 && lane == 0) CFA_TRACE(5, tc, 5);
      if (old != (unsigned)(a.splits - 1)) continue;
      __threadfence();
      const float* p0 = a.part + (size_t)t.tile * a.splits * kRsTileM * kRsTileN +
                        (size_t)quad * 32 * kRsTileN;
      // 32 independent loads in flight per round (4 splits x 8 rows), added
      // in split order
      for (int nb = 0; nb < kRsTileN; nb += 32) {
        const int nt = nb + 4 * cg;
        const int n = t.tn * kRsTileN + nt;
        float4 acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp0 = 0; sp0 < a.splits; sp0 += 4) {
          float4 x[4][8];
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 8; ++i)
              x[q][i] = sp0 + q < a.splits
                            ? __ldcg(reinterpret_cast<const float4*>(
                                  p0 + (size_t)(sp0 + q) * kRsTileM * kRsTileN +
                                  (size_t)(rr0 + 4 * i) * kRsTileN + nt))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              acc[i].x += x[q][i].x;
              acc[i].y += x[q][i].y;
              acc[i].z += x[q][i].z;
              acc[i].w += x[q][i].w;
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (orow[i] && n < a.N) put4(a, orow[i] + (size_t)n * esz, acc[i], f32);
      }
      if (lane == 0) a.counters[4 * t.tile + quad] = 0u;  // ready for the next call
      if (quad == 0 && lane == 0) CFA_TRACE(5, tc, 6);
    }
    // every store this warp issued has completed (and left shared memory)
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
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

bool rowsparse_clusters_fit(int splits, int clusters) {
  if (splits < 2 || splits > 8 || (splits & (splits - 1)) != 0) return false;
  auto k = rowsparse_kernel<1, true>;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess)
    return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(splits * clusters));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return n >= clusters;
}

cudaError_t launch_rowsparse(const CUtensorMap& map_a, const CUtensorMap& map_b,
                             const CUtensorMap& map_o, const CUtensorMap& map_p,
                             const CUtensorMap& map_xt, const RsArgs& a, int grid,
                             cudaStream_t st) {
  void (*k)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
            const CUtensorMap, const RsArgs) =
      a.mode == 0 ? rowsparse_kernel<0, false>
                  : (a.cluster ? rowsparse_kernel<1, true> : rowsparse_kernel<1, false>);
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  if (!a.cluster)
    return launch_pdl(k, dim3(grid), dim3(kThreads), kSmemBytes, st, map_a, map_b, map_o, map_p,
                      map_xt, a);
  // one cluster per tile, its `splits` CTAs consecutive in x
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)a.splits;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, map_a, map_b, map_o, map_p, map_xt, a);
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

#ifdef CFA_TRACE_BUILD
extern "C" int cfa_trace_read_rs(long long* dst, int clear) {
  const size_t n = sizeof(long long) * cfa::kTraceRoles * cfa::kTraceIters * cfa::kTraceEvents;
  if (dst && cudaMemcpyFromSymbol(dst, cfa::cfa_trace_buf, n) != cudaSuccess) return -1;
  if (clear) {
    static long long zero[cfa::kTraceRoles * cfa::kTraceIters * cfa::kTraceEvents];
    if (cudaMemcpyToSymbol(cfa::cfa_trace_buf, zero, n) != cudaSuccess) return -1;
  }
  return 0;
}
#endif
