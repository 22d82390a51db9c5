// Query-split backward of frozen-prefix chunk attention on sm_103a.
//
// The prefix is a stop-gradient constant, so the backward needs
//   dQ_t  = s * sum_{visible j} dS_tj k_j        over prefix AND chunk keys
//   dK_j, dV_j                                    over the chunk's keys only
// with P_tj = exp(s q_t.k_j - LSE_t), dS_tj = P_tj (dO_t.v_j - delta_t).
//
// Two kernels split the work so that neither needs atomics:
//
// * bwd_dq_kernel -- query-major, persistent stream-K (cfa_sched.cuh): a
//   CTA walks an equal share of the (128-row query tile, key tile)
//   iterations and streams K/V through three MMAs per tile: S = Q K^T,
//   dP = dO V^T, dQ += dS K.  Prefix tiles never produce dK/dV.  Query tiles
//   cut by CTA boundaries leave fp32 partials that bwd_dq_reduce_kernel sums
//   in CTA order.
//     warps 0-7  elementwise (two warps per TMEM lane quadrant, each owning
//                64 of the 128 key columns): P, dS, bf16 dS into TMEM
//     warp  8    TMA producer      warp 9  TMEM owner + MMA issuer
//   TMEM: S0 [0,128) S1 [128,256) dP [256,384) dQ [384,384+D); dS overwrites
//   the S columns its own warp has read (keys 0-63 -> cols 0-31, keys
//   64-127 -> cols 64-95) and is the A operand of the dQ MMA.
//
// * bwd_dkdv_kernel -- key-major over the chunk keys.  A CTA owns one
//   128-key chunk tile and walks the query tiles that can see it:
//   S^T = K Q^T, dP^T = V dO^T, dV += P^T dO, dK += dS^T Q, with P^T and dS^T
//   staged bf16 in TMEM and handed over separately, so the MMAs of one query
//   tile overlap the elementwise work of the neighbouring one.
//   TMEM: S^T [0,128) dP^T [128,256) dV, dK.
#include "cfa_kernels.cuh"
#include "cfa_ptx.cuh"

namespace cfa {
namespace {

constexpr int kBoxBytes = 128 * 128;

// Column of the k-th 16-key slice of a bf16 operand staged in TMEM by the two
// half-warps (keys 0-63 at columns 0-31, keys 64-127 at columns 64-95).
__device__ __forceinline__ uint32_t staged_col(int k) {
  return (k < 4) ? (uint32_t)(k * 8) : (uint32_t)(64 + (k - 4) * 8);
}

// D = A B^T with A, B K-major 128B-swizzled tiles of 128 rows x D columns.
template <int D>
__device__ __forceinline__ void issue_nt(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
  constexpr uint32_t hi = sw128_desc_hi(1024);
  const uint32_t a_lo = sw128_desc_lo(a_addr, 16), b_lo = sw128_desc_lo(b_addr, 16);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t off = ((uint32_t)(k >> 2) * kBoxBytes + (uint32_t)(k & 3) * 32u) >> 4;
    mma_ss_warp(d_tmem, a_lo + off, hi, b_lo + off, hi, idesc, k > 0 ? 1u : 0u);
  }
}

// D (+)= A[tmem, staged] B with B a 128-row x D tile read MN-major.
template <int D>
__device__ __forceinline__ void issue_tn(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_addr,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
  constexpr uint32_t hi = sw128_desc_hi(1024);
  const uint32_t b_lo = sw128_desc_lo(b_addr, kBoxBytes);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    mma_ts_warp(d_tmem, a_tmem + staged_col(k), b_lo + (uint32_t)k * (2048u >> 4), hi, idesc,
                (accumulate || k > 0) ? 1u : 0u);
}

template <int D>
struct DqCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  // K(i) is read by S(i) and, late, by dQ(i); V(i) only by dP(i).  Separate
  // rings let V refill early and give K one extra stage of lead.
  static constexpr int kKStages = (D == 128) ? 3 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kDOOff = kTileBytes;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(8 * (2 + 2 * kKStages + 2 * kVStages + 8) <= 240, "barrier area");
};

template <int D, bool ROW>
__global__ void __launch_bounds__(320, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q,
                  const __grid_constant__ CUtensorMap map_do,
                  const __grid_constant__ CUtensorMap map_kp,
                  const __grid_constant__ CUtensorMap map_vp,
                  const __grid_constant__ CUtensorMap map_kc,
                  const __grid_constant__ CUtensorMap map_vc, const BwdArgs a) {
  CFA_TRACE_SPAN(2, 0);
  pdl_start();
  CFA_TRACE_SPAN(2, 1);
  // A call's first kernel clears the status word once the previous work in
  // the stream is done (no separate memset: one dependent launch less).  A
  // device wait gives up only after its wall-clock limit, long after CTA 0
  // has started, so no error of this launch is cleared.
  if (a.clear_status && blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0;
  CFA_TRACE_CTA(0);
  using C = DqCfg<D>;
  constexpr int SK = C::kKStages;
  constexpr int SV = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Tiling tl = a.tl;
  {
    // schedule prologue: shared scratch in the (not yet used) barrier area;
    // inconsistent cu_seqlens end the kernel before any load or store (see
    // the forward kernel)
    long long* sched = reinterpret_cast<long long*>(gbase + C::kBarOff);
    if (!plan_schedule<ROW>(a.cu_p, a.cu_c, a.batch, a.hkv, tl, a.lim, a.win_prefix, sched + 4,
                            sched, reinterpret_cast<int*>(sched + 1), sched + 2)) {
      if (threadIdx.x == 0) atomicExch(a.status, kStatusInvalidArg);
      return;
    }
  }
  SegmentWalkerT<ROW> walk;
  {
    const long long* sched = reinterpret_cast<const long long*>(gbase + C::kBarOff);
    walk.init(a.cu_p, a.cu_c, a.batch, a.hkv, tl, blockIdx.x, sched[0],
              *reinterpret_cast<const int*>(sched + 1), sched[2]);
  }
  __syncthreads();  // the barrier area is initialised below
  if (walk.cur >= walk.end) return;

  const uint32_t bars = base + C::kBarOff;
  const uint32_t bar_qdo = bars;
  const uint32_t bar_qempty = bars + 8;
  const uint32_t bar_kfull = bars + 16;               // [SK]
  const uint32_t bar_kempty = bar_kfull + 8 * SK;     // [SK]
  const uint32_t bar_vfull = bar_kempty + 8 * SK;     // [SV]
  const uint32_t bar_vempty = bar_vfull + 8 * SV;     // [SV]
  const uint32_t bar_sfull = bar_vempty + 8 * SV;     // [2]
  const uint32_t bar_dpfull = bar_sfull + 16;
  const uint32_t bar_dpfree = bar_dpfull + 8;
  const uint32_t bar_dsfull = bar_dpfree + 8;
  const uint32_t bar_dqfull = bar_dsfull + 8;
  const uint32_t bar_dqfree = bar_dqfull + 8;
  const uint32_t bar_drain = bar_dqfree + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kBarOff + 240);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBarOff + 244);

  if (threadIdx.x == 0) {
    mbar_init(bar_qdo, 1);
    mbar_init(bar_qempty, 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_vempty + 8 * s, 1);
    }
    mbar_init(bar_sfull, 1);
    mbar_init(bar_sfull + 8, 1);
    mbar_init(bar_dpfull, 1);
    mbar_init(bar_dsfull, 8);
    mbar_init(bar_dqfull, 1);
    mbar_init(bar_dqfree, 8);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{a.limit_ns, abort_flag, a.status};
  Segment sg;

  if (warp == 8) {
    // producer: the whole warp walks and waits (converged); lane 0 issues
    const bool leader = lane == 0;
    const uint32_t qbytes = (uint32_t)(C::kBoxes * 128 * tl.rows);
    int it = 0, seg = 0, issued_k = 0, issued_v = 0;
    bool ok = true;
    while (ok && walk.next(sg)) {
      // Q and dO are reused: the previous segment's S and dP must be done
      if (seg > 0 && !(ok = warp_wait(W, bar_qempty, (uint32_t)(seg - 1) & 1u))) break;
      const int tok = sg.c0 + sg.qb * tl.tpt;
      if (leader) {
        mbar_arrive_expect_tx(bar_qdo, 2 * qbytes);
        for (int kb = 0; kb < C::kBoxes; ++kb) {
          tma_load_3d(base + C::kQOff + kb * kBoxBytes, &map_q, bar_qdo, kb * 64, sg.hk * tl.g,
                      tok);
          tma_load_3d(base + C::kDOOff + kb * kBoxBytes, &map_do, bar_qdo, kb * 64, sg.hk * tl.g,
                      tok);
        }
      }
      __syncwarp();
      ++seg;
      const int np_t = ceil_div(sg.lp, kTileN);
      for (int kt = sg.t_begin; kt < sg.t_end; ++kt, ++it) {
        const CUtensorMap* mk = &map_kc;
        const CUtensorMap* mv = &map_vc;
        int row0 = sg.c0 + (kt - np_t) * kTileN;
        if (kt < np_t) {
          mk = &map_kp;
          mv = &map_vp;
          row0 = sg.p0 + kt * kTileN;
        }
        const int sk = it % SK, sv = it % SV;
        if (!(ok = warp_wait(W, bar_kempty + 8 * sk, ((uint32_t)(it / SK) & 1u) ^ 1u))) break;
        CFA_TRACE(3, it, 0);
        if (leader) {
          mbar_arrive_expect_tx(bar_kfull + 8 * sk, C::kTileBytes);
          for (int kb = 0; kb < C::kBoxes; ++kb)
            tma_load_3d(base + C::kKOff + sk * C::kTileBytes + kb * kBoxBytes, mk,
                        bar_kfull + 8 * sk, kb * 64, sg.hk, row0);
        }
        __syncwarp();
        issued_k = it + 1;
        if (!(ok = warp_wait(W, bar_vempty + 8 * sv, ((uint32_t)(it / SV) & 1u) ^ 1u))) break;
        CFA_TRACE(3, it, 1);
        if (leader) {
          mbar_arrive_expect_tx(bar_vfull + 8 * sv, C::kTileBytes);
          for (int kb = 0; kb < C::kBoxes; ++kb)
            tma_load_3d(base + C::kVOff + sv * C::kTileBytes + kb * kBoxBytes, mv,
                        bar_vfull + 8 * sv, kb * 64, sg.hk, row0);
        }
        __syncwarp();
        issued_v = it + 1;
      }
    }
    if (seg > 0) mbar_wait_bounded(bar_qdo, (uint32_t)(seg - 1) & 1u, kDrainLimitNs);
    for (int i = (issued_k > SK ? issued_k - SK : 0); i < issued_k; ++i)
      mbar_wait_bounded(bar_kfull + 8 * (i % SK), (uint32_t)(i / SK) & 1u, kDrainLimitNs);
    for (int i = (issued_v > SV ? issued_v - SV : 0); i < issued_v; ++i)
      mbar_wait_bounded(bar_vfull + 8 * (i % SV), (uint32_t)(i / SV) & 1u, kDrainLimitNs);
  } else if (warp == 9) {
    // Issue order: S runs one key tile ahead.  A segment starts with S(0),
    // dP(0), S(1); then for every later tile g, after the single wait for
    // dS(g-1):  dQ(g-1)  dP(g)  S(g+1).  S(g+1) goes to the S buffer that
    // dS(g-1) occupied, which dQ(g-1) has read by then (the pipe is in
    // order); so the elementwise warps find S(g) ready the moment they hand
    // over dS(g-1) and compute P(g) while dQ(g-1) and dP(g) run.  dQ(g-1)
    // goes first so that K(g-1)'s stage frees early: K(g+2) then has most of
    // two tiles' time to arrive.  This warp waits for K(g+1) itself, right
    // after queueing dP(g), so the tensor pipe still has work during the
    // check; V(g) is checked by an elementwise warp before it hands over
    // dS(g-1), at a point where it waits for dP(g-1) anyway.
    // The whole warp waits and issues (converged); elect.sync picks the lane
    // that issues the MMAs and commits.
    const uint32_t t_dq = tmem + 384;
    int it = 0, seg = 0;
    // test hook: see the forward kernel
    bool ok = !(a.debug_wait_never && !warp_wait(W, bar_drain, 0));
    auto issue_s = [&](int g) {
      issue_nt<D>(tmem + (uint32_t)(g & 1) * 128u, base + C::kQOff,
                  base + C::kKOff + (g % SK) * C::kTileBytes);
      tc_commit_warp(bar_sfull + 8 * (g & 1));
    };
    auto issue_dp = [&](int g, bool last) {
      issue_nt<D>(tmem + 256, base + C::kDOOff, base + C::kVOff + (g % SV) * C::kTileBytes);
      tc_commit_warp(bar_dpfull);
      tc_commit_warp(bar_vempty + 8 * (g % SV));
      if (last) tc_commit_warp(bar_qempty);  // the segment's last S and dP
    };
    auto issue_dq = [&](int g, bool accumulate) {
      issue_tn<D>(t_dq, tmem + (uint32_t)(g & 1) * 128u,
                  base + C::kKOff + (g % SK) * C::kTileBytes, accumulate);
      tc_commit_warp(bar_kempty + 8 * (g % SK));
    };
    while (ok && walk.next(sg)) {
      const int n = sg.t_end - sg.t_begin;
      if (!(ok = warp_wait(W, bar_qdo, (uint32_t)seg & 1u))) break;
      if (!(ok = warp_wait(W, bar_kfull + 8 * (it % SK), (uint32_t)(it / SK) & 1u))) break;
      if (!(ok = warp_wait(W, bar_vfull + 8 * (it % SV), (uint32_t)(it / SV) & 1u))) break;
      issue_s(it);
      issue_dp(it, n == 1);
      if (n > 1) {
        if (!(ok = warp_wait(W, bar_kfull + 8 * ((it + 1) % SK), (uint32_t)((it + 1) / SK) & 1u)))
          break;
        issue_s(it + 1);
      }
      for (int i = 1; i < n; ++i) {
        const int g = it + i;
        // the first dQ of a segment overwrites the accumulator: the previous
        // segment's epilogue must have read it
        if (i == 1 && seg > 0 && !(ok = warp_wait(W, bar_dqfree, (uint32_t)(seg - 1) & 1u))) break;
        CFA_TRACE(2, g, 0);
        if (!(ok = warp_wait(W, bar_dsfull, (uint32_t)(g - 1) & 1u))) break;
        CFA_TRACE(2, g, 1);
        tc_fence_after_sync();
        issue_dq(g - 1, i > 1);
        CFA_TRACE(2, g, 2);
        issue_dp(g, i == n - 1);  // V(g): checked by the elementwise warps
        CFA_TRACE(2, g, 3);
        if (i + 1 < n) {
          if (!(ok = warp_wait(W, bar_kfull + 8 * ((g + 1) % SK), (uint32_t)((g + 1) / SK) & 1u)))
            break;
          CFA_TRACE(2, g, 6);
          issue_s(g + 1);
        }
        CFA_TRACE(2, g, 4);
      }
      if (!ok) break;
      const int gl = it + n - 1;
      if (n == 1 && seg > 0 && !(ok = warp_wait(W, bar_dqfree, (uint32_t)(seg - 1) & 1u))) break;
      if (!(ok = warp_wait(W, bar_dsfull, (uint32_t)gl & 1u))) break;
      tc_fence_after_sync();
      issue_dq(gl, n > 1);
      tc_commit_warp(bar_dqfull);
      it += n;
      ++seg;
    }
    tc_commit_warp(bar_drain);
    mbar_wait_bounded(bar_drain, 0, kDrainLimitNs);
  } else {
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const float sl2 = a.scale_log2;
    int u = 0, seg = 0;  // tiles and segments processed
    bool ok = true;
    while (ok && walk.next(sg)) {
      const int n = sg.t_end - sg.t_begin;
      const int np_t = ceil_div(sg.lp, kTileN);
      const int token = sg.qb * tl.tpt + row / tl.g;
      const int head = sg.hk * tl.g + row % tl.g;
      const bool row_valid = row < tl.rows && token < sg.lc;
      const size_t grow = (size_t)(sg.c0 + (row_valid ? token : 0));
      const float lse2 = row_valid ? a.lse[(size_t)head * a.total_lc + grow] * kLog2e : 0.f;
      const float dl = row_valid ? a.delta[(size_t)head * a.total_lc + grow] : 0.f;
      for (int i = 0; i < n; ++i, ++u) {
        const uint32_t sb = (uint32_t)(u & 1) * 128u + (uint32_t)half * 64u;
        if (!(ok = warp_wait(W, bar_sfull + 8 * (u & 1), (uint32_t)(u >> 1) & 1u))) break;
        if (warp < 2 && lane == 0) CFA_TRACE(warp, u, 0);
        tc_fence_after_sync();
        const int kt = sg.t_begin + i;
        int lim = (kt < np_t) ? (sg.lp - kt * kTileN) : (token - (kt - np_t) * kTileN + 1);
        if (!row_valid) lim = 0;
        lim -= half * 64;  // visible columns [0, lim) of this warp's 64
        float p[64];
        {
          // two 32-column loads: the exponentials of the first half run while
          // the second half loads
          uint32_t r[64];
          tmem_ld_x32_async(t_lane + sb, r);
          tmem_wait_ld_x32(r);
          tmem_ld_x32_async(t_lane + sb + 32, r + 32);
          const uint64_t sl2x2 = f2(sl2, sl2), nl2 = f2(-lse2, -lse2);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j == 16) tmem_wait_ld_x32(r + 32);
            f2_split(ex2_sfu_x2(f2_fma(f2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])),
                                       sl2x2, nl2)),
                     p[2 * j], p[2 * j + 1]);
          }
          if (lim < 64) {  // edge tiles only: the prefix tail, the causal diagonal, padding rows
#pragma unroll
            for (int j = 0; j < 64; ++j) p[j] = (j < lim) ? p[j] : 0.f;
          }
        }
        if (warp < 2 && lane == 0) CFA_TRACE(warp, u, 1);
        if (warp == 0 && i + 1 < n) {
          // V(u+1) is in shared memory before dS(u) is handed over, so the
          // MMA warp need not wait for it before dP(u+1); checked here, where
          // this warp waits for dP(u) anyway
          const int v = u + 1;
          if (!(ok = warp_wait(W, bar_vfull + 8 * (v % SV), (uint32_t)(v / SV) & 1u))) break;
        }
        if (!(ok = warp_wait(W, bar_dpfull, (uint32_t)u & 1u))) break;
        if (warp < 2 && lane == 0) CFA_TRACE(warp, u, 2);
        tc_fence_after_sync();
        uint32_t pk[32];
        {
          // dP in two 32-column loads: dS of the first half is computed while
          // the second half loads
          uint32_t r[64];
          tmem_ld_x32_async(t_lane + 256 + half * 64, r);
          tmem_wait_ld_x32(r);
          tmem_ld_x32_async(t_lane + 256 + half * 64 + 32, r + 32);
          const uint64_t dl2 = f2(dl, dl);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j == 16) tmem_wait_ld_x32(r + 32);
            float d0, d1;
            f2_split(f2_mul(f2(p[2 * j], p[2 * j + 1]),
                            f2_sub(f2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), dl2)),
                     d0, d1);
            pk[j] = pack_bf16x2(d0, d1);
          }
        }
        tmem_st_x32(t_lane + sb, pk);
        tmem_st_wait();
        if (warp < 2 && lane == 0) CFA_TRACE(warp, u, 3);
        tc_fence_before_sync();
        __syncwarp();
        if (warp < 2 && lane == 0) CFA_TRACE(warp, u, 4);
        if (lane == 0) mbar_arrive(bar_dsfull);
      }
      if (!ok) break;
      if (!(ok = warp_wait(W, bar_dqfull, (uint32_t)seg & 1u))) break;
      tc_fence_after_sync();
      const bool final_out = !sg.head && !sg.tail;
      const int slot = sg.head ? 0 : 1;
      const size_t pslot = (size_t)blockIdx.x * 2 + slot;
      // this warp's half of the dQ row in one TMEM load, then the hand-off
      // (before the global stores, which the arrive would otherwise wait for)
      constexpr int HW = D / 2;
      uint32_t r[HW];
      if constexpr (HW == 64)
        tmem_ld_x64(t_lane + 384 + half * HW, r);
      else
        tmem_ld_x32(t_lane + 384 + half * HW, r);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dqfree);
#pragma unroll
      for (int c = 0; c < HW; c += 32) {
        const int cb = half * HW + c;
        if (row_valid) {
          if (final_out) {
            uint4* dst = reinterpret_cast<uint4*>(a.dq + (grow * a.hq + head) * D + cb);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 w;
              w.x = pack_bf16x2(__uint_as_float(r[c + 8 * v + 0]) * a.scale,
                                __uint_as_float(r[c + 8 * v + 1]) * a.scale);
              w.y = pack_bf16x2(__uint_as_float(r[c + 8 * v + 2]) * a.scale,
                                __uint_as_float(r[c + 8 * v + 3]) * a.scale);
              w.z = pack_bf16x2(__uint_as_float(r[c + 8 * v + 4]) * a.scale,
                                __uint_as_float(r[c + 8 * v + 5]) * a.scale);
              w.w = pack_bf16x2(__uint_as_float(r[c + 8 * v + 6]) * a.scale,
                                __uint_as_float(r[c + 8 * v + 7]) * a.scale);
              dst[v] = w;
            }
          } else {
            // feature-major partial [D/4][128][4]: a warp's store is one
            // contiguous 512-byte run
            float4* dst = reinterpret_cast<float4*>(a.dq_part) + pslot * (D / 4) * kTileM +
                          (size_t)(cb / 4) * kTileM + row;
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[(size_t)v * kTileM] = make_float4(__uint_as_float(r[c + 4 * v + 0]) * a.scale,
                                                    __uint_as_float(r[c + 4 * v + 1]) * a.scale,
                                                    __uint_as_float(r[c + 4 * v + 2]) * a.scale,
                                                    __uint_as_float(r[c + 4 * v + 3]) * a.scale);
          }
        }
      }
      ++seg;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  CFA_TRACE_CTA(1);
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
  CFA_TRACE_SPAN(2, 2);
}

template <int D>
struct DkvCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kStages = (D == 128) ? 2 : 4;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kTileBytes;
  static constexpr int kQOff = 2 * kTileBytes;           // stage s: Q at +2s*T, dO at +(2s+1)*T
  static constexpr int kRowOff = kQOff + 2 * kStages * kTileBytes;  // per-warp LSE/delta
  static constexpr int kBarOff = kRowOff + 8 * 128 * 4;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
};

// Work items of the dK/dV kernel: (key tile, window b, KV head hk), numbered
// tile-slot-major so that the longest items come first; CTA c takes items c,
// c + G, c + 2G, ...  The first a.pre_tiles slots are prefix key tiles of the
// horizon (the last a.horizon prefix rows of each window, whose gradient the
// caller asked for; every chunk row sees them), the next a.dkv_tiles slots
// the 128-key chunk tiles (chunk key j seen by chunk rows t >= j).
struct DkvItem {
  int b, hk;
  bool pre;          // a prefix key tile
  int c0, lc;        // the window's chunk rows
  int k0, krows;     // first row of the key tile in its tensor, and the keys there are
  int kmin;          // keys below this index in the tile get no gradient written
  int key0;          // key index of the tile's first key within the chunk (chunk tiles)
  int qi_lo, n;      // query tiles [qi_lo, qi_lo + n)
};

__device__ inline bool dkv_item(const BwdArgs& a, long long j, DkvItem& it) {
  it.hk = (int)(j % a.hkv);
  it.b = (int)((j / a.hkv) % a.batch);
  const int slot = (int)(j / ((long long)a.hkv * a.batch));
  it.c0 = a.cu_c[it.b];
  it.lc = a.cu_c[it.b + 1] - it.c0;
  it.pre = slot < a.pre_tiles;
  if (it.pre) {
    const int p0 = a.cu_p[it.b], lp = a.cu_p[it.b + 1] - p0;
    const int h = a.horizon < lp ? a.horizon : lp;
    const int first = lp - h;                       // first prefix row in the horizon
    const int kt = first / kTileN + slot;
    if (h == 0 || kt * kTileN >= lp) return false;
    it.k0 = p0 + kt * kTileN;
    it.krows = lp - kt * kTileN;
    it.kmin = first - kt * kTileN;
    it.key0 = 0;
    it.qi_lo = 0;
    it.n = ceil_div(it.lc, a.tl.tpt);               // every chunk row sees the prefix
    return true;
  }
  const int kt = slot - a.pre_tiles;
  it.key0 = kt * kTileN;
  if (it.key0 >= it.lc) return false;
  it.k0 = it.c0 + it.key0;
  it.krows = it.lc - it.key0;
  it.kmin = 0;
  it.qi_lo = it.key0 / a.tl.tpt;
  it.n = ceil_div(it.lc, a.tl.tpt) - it.qi_lo;
  return true;
}

template <int D>
__global__ void __launch_bounds__(320, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_do,
                    const __grid_constant__ CUtensorMap map_kc,
                    const __grid_constant__ CUtensorMap map_vc,
                    const __grid_constant__ CUtensorMap map_kp,
                    const __grid_constant__ CUtensorMap map_vp, const BwdArgs a) {
  CFA_TRACE_SPAN(5, 0);
  pdl_start();
  CFA_TRACE_SPAN(5, 1);
  // clears the status word when this kernel is its call's first (see the dQ kernel)
  if (a.clear_status && blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0;
  using C = DkvCfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Tiling tl = a.tl;
  const long long n_items = (long long)(a.pre_tiles + a.dkv_tiles) * a.batch * a.hkv;
  if ((long long)blockIdx.x >= n_items) return;
  const long long j0 = blockIdx.x, jstep = gridDim.x;
  {
    // the items' rows come from the device cu_seqlens: check them against the
    // host sizes first (every CTA, all windows; see the forward kernel)
    bool bad = false;
    for (int b = threadIdx.x; b < a.batch; b += blockDim.x)
      bad |= !window_valid(a.cu_p, a.cu_c, b, a.batch, a.lim);
    if (__syncthreads_or(bad)) {
      if (threadIdx.x == 0) atomicExch(a.status, kStatusInvalidArg);
      return;
    }
  }

  const uint32_t bars = base + C::kBarOff;
  const uint32_t bar_kv = bars;
  const uint32_t bar_qfull = bars + 8;               // [S]
  const uint32_t bar_qempty = bars + 8 * (1 + S);    // [S]
  const uint32_t bar_stfull = bars + 8 * (1 + 2 * S);
  const uint32_t bar_dptfull = bar_stfull + 8;
  const uint32_t bar_pfull = bar_dptfull + 8;
  const uint32_t bar_dsfull = bar_pfull + 8;
  const uint32_t bar_dkvfull = bar_dsfull + 8;
  const uint32_t bar_dkvfree = bar_dkvfull + 8;
  const uint32_t bar_kvfree = bar_dkvfree + 8;
  const uint32_t bar_drain = bar_kvfree + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kBarOff + 240);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBarOff + 244);

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_qfull + 8 * s, 1);
      mbar_init(bar_qempty + 8 * s, 1);
    }
    mbar_init(bar_stfull, 1);
    mbar_init(bar_dptfull, 1);
    mbar_init(bar_pfull, 8);
    mbar_init(bar_dsfull, 8);
    mbar_init(bar_dkvfull, 1);
    mbar_init(bar_dkvfree, 8);
    mbar_init(bar_kvfree, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{a.limit_ns, abort_flag, a.status};
  const uint32_t t_dv = tmem + 256, t_dk = tmem + 256 + D;
  DkvItem it;

  if (warp == 8) {
    // producer: the whole warp waits (converged); lane 0 issues.  K/V of an
    // item reuse one buffer: they load once the previous item's last S^T and
    // dP^T are done (kvfree), while its dV and dK still run.
    const bool leader = lane == 0;
    const uint32_t qbytes = (uint32_t)(C::kBoxes * 128 * tl.rows);
    int qn = 0, items = 0, issued = 0;
    bool ok = true;
    for (long long j = j0; ok && j < n_items; j += jstep) {
      if (!dkv_item(a, j, it) || it.n == 0) continue;
      if (items > 0 && !(ok = warp_wait(W, bar_kvfree, (uint32_t)(items - 1) & 1u))) break;
      if (leader) {
        mbar_arrive_expect_tx(bar_kv, 2 * C::kTileBytes);
        for (int kb = 0; kb < C::kBoxes; ++kb) {
          tma_load_3d(base + C::kKOff + kb * kBoxBytes, it.pre ? &map_kp : &map_kc, bar_kv,
                      kb * 64, it.hk, it.k0);
          tma_load_3d(base + C::kVOff + kb * kBoxBytes, it.pre ? &map_vp : &map_vc, bar_kv,
                      kb * 64, it.hk, it.k0);
        }
      }
      __syncwarp();
      ++items;
      for (int i = 0; i < it.n; ++i, ++qn) {
        const int s = qn % S;
        if (!(ok = warp_wait(W, bar_qempty + 8 * s, ((uint32_t)(qn / S) & 1u) ^ 1u))) break;
        const int tok = it.c0 + (it.qi_lo + i) * tl.tpt;
        if (leader) {
          mbar_arrive_expect_tx(bar_qfull + 8 * s, 2 * qbytes);
          for (int kb = 0; kb < C::kBoxes; ++kb) {
            tma_load_3d(base + C::kQOff + (2 * s) * C::kTileBytes + kb * kBoxBytes, &map_q,
                        bar_qfull + 8 * s, kb * 64, it.hk * tl.g, tok);
            tma_load_3d(base + C::kQOff + (2 * s + 1) * C::kTileBytes + kb * kBoxBytes, &map_do,
                        bar_qfull + 8 * s, kb * 64, it.hk * tl.g, tok);
          }
        }
        __syncwarp();
        issued = qn + 1;
      }
    }
    // Unwind: every copy this warp issued has landed before the CTA exits.
    if (items > 0) mbar_wait_bounded(bar_kv, (uint32_t)(items - 1) & 1u, kDrainLimitNs);
    for (int i = (issued > S ? issued - S : 0); i < issued; ++i)
      mbar_wait_bounded(bar_qfull + 8 * (i % S), (uint32_t)(i / S) & 1u, kDrainLimitNs);
  } else if (warp == 9) {
    // Issue order per item:  S^T(0) dP^T(0), then per query tile i:
    //   dV(i) [after P^T(i)]  S^T(i+1)  dK(i) [after dS^T(i)]  dP^T(i+1)
    // so dV(i) and S^T(i+1) run while dS^T(i) is computed and dK(i),
    // dP^T(i+1) while P^T(i+1) is.  S^T(i+1) reuses the columns of P^T(i)
    // and dP^T(i+1) those of dS^T(i), each consumed by the MMA issued just
    // before it (the MMA pipe is in order).  The first dV of an item
    // overwrites the accumulators, so it waits for the previous item's
    // epilogue (dkvfree).  Query-tile counters run across items.  The whole
    // warp waits and issues (converged); elect.sync picks the issuing lane.
    int qn = 0, items = 0;
    bool ok = !(a.debug_wait_never && !warp_wait(W, bar_drain, 0));
    for (long long j = j0; ok && j < n_items; j += jstep) {
      if (!dkv_item(a, j, it) || it.n == 0) continue;
      const int n = it.n;
      if (!(ok = warp_wait(W, bar_kv, (uint32_t)items & 1u))) break;
      if (!(ok = warp_wait(W, bar_qfull + 8 * (qn % S), (uint32_t)(qn / S) & 1u))) break;
      issue_nt<D>(tmem, base + C::kKOff, base + C::kQOff + (2 * (qn % S)) * C::kTileBytes);
      tc_commit_warp(bar_stfull);                                                 // S^T = K Q^T
      issue_nt<D>(tmem + 128, base + C::kVOff,
                  base + C::kQOff + (2 * (qn % S) + 1) * C::kTileBytes);          // dP^T = V dO^T
      tc_commit_warp(bar_dptfull);
      if (n == 1) tc_commit_warp(bar_kvfree);
      for (int i = 0; i < n; ++i) {
        const int t = qn + i;
        const int s = t % S, s1 = (t + 1) % S;
        const uint32_t q_addr = base + C::kQOff + (2 * s) * C::kTileBytes;
        const uint32_t do_addr = q_addr + C::kTileBytes;
        const uint32_t q1_addr = base + C::kQOff + (2 * s1) * C::kTileBytes;
        CFA_TRACE(2, t, 0);
        if (!(ok = warp_wait(W, bar_pfull, (uint32_t)t & 1u))) break;
        if (i == 0 && items > 0 &&
            !(ok = warp_wait(W, bar_dkvfree, (uint32_t)(items - 1) & 1u)))
          break;
        CFA_TRACE(2, t, 1);
        tc_fence_after_sync();
        issue_tn<D>(t_dv, tmem, do_addr, i > 0);                                  // dV += P^T dO
        if (i + 1 < n) {
          if (!(ok = warp_wait(W, bar_qfull + 8 * s1, (uint32_t)((t + 1) / S) & 1u))) break;
          issue_nt<D>(tmem, base + C::kKOff, q1_addr);                            // S^T(i+1)
          tc_commit_warp(bar_stfull);
        }
        CFA_TRACE(2, t, 2);
        if (!(ok = warp_wait(W, bar_dsfull, (uint32_t)t & 1u))) break;
        CFA_TRACE(2, t, 3);
        tc_fence_after_sync();
        issue_tn<D>(t_dk, tmem + 128, q_addr, i > 0);                             // dK += dS^T Q
        tc_commit_warp(bar_qempty + 8 * s);
        if (i + 1 < n) {
          issue_nt<D>(tmem + 128, base + C::kVOff, q1_addr + C::kTileBytes);      // dP^T(i+1)
          tc_commit_warp(bar_dptfull);
          if (i + 2 == n) tc_commit_warp(bar_kvfree);  // the item's last S^T and dP^T
        }
      }
      if (!ok) break;
      tc_commit_warp(bar_dkvfull);
      qn += n;
      ++items;
    }
    tc_commit_warp(bar_drain);
    mbar_wait_bounded(bar_drain, 0, kDrainLimitNs);
  } else {
    const int quad = warp & 3, half = warp >> 2;
    const int krow = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    float* my_lse = reinterpret_cast<float*>(gbase + C::kRowOff) + warp * 128;
    float* my_dl = my_lse + 64;
    const float sl2 = a.scale_log2;
    float lse_n[2], dl_n[2];
    // LSE and delta of this warp's 64 query rows of query tile qi, loaded
    // one tile ahead so the global-memory latency stays off the critical path
    auto fetch_rows = [&](int qi) {
      const int tok0 = qi * tl.tpt;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int r = half * 64 + u * 32 + lane;
        const int tok = tok0 + r / tl.g;
        const bool v = r < tl.rows && tok < it.lc;
        const size_t idx = (size_t)(it.hk * tl.g + r % tl.g) * a.total_lc + (size_t)(it.c0 + tok);
        lse_n[u] = v ? a.lse[idx] * kLog2e : 0.f;
        dl_n[u] = v ? a.delta[idx] : 0.f;
      }
    };
    int qn = 0, items = 0;
    bool ok = true;
    for (long long j = j0; ok && j < n_items; j += jstep) {
      if (!dkv_item(a, j, it)) continue;
      const int n = it.n;
      // this thread's key: row krow of the tile; its gradient is written when
      // it exists and lies in the horizon (prefix) / the chunk
      const bool key_valid = krow < it.krows;
      const bool key_out = key_valid && krow >= it.kmin;
      __nv_bfloat16* const dk_base = it.pre ? a.dk_p : a.dk;
      __nv_bfloat16* const dv_base = it.pre ? a.dv_p : a.dv;
      const size_t grow = (size_t)(it.k0 + krow) * a.hkv + it.hk;
      if (n == 0) {
        // a window without chunk rows: its horizon rows' gradient is zero
        if (key_out) {
          uint4* dv = reinterpret_cast<uint4*>(dv_base + grow * D + half * (D / 2));
          uint4* dk = reinterpret_cast<uint4*>(dk_base + grow * D + half * (D / 2));
#pragma unroll
          for (int v = 0; v < D / 16; ++v) dv[v] = dk[v] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const int key = it.key0 + krow;
      fetch_rows(it.qi_lo);
      for (int i = 0; i < n; ++i) {
        const int t = qn + i;
        const int tok0 = (it.qi_lo + i) * tl.tpt;
        // columns r of this warp are half*64 + j; row r is (token tok0 + r / g, head r % g)
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          my_lse[u * 32 + lane] = -lse_n[u];   // stored negated: p = 2^(s*scale_log2 + that)
          my_dl[u * 32 + lane] = dl_n[u];
        }
        __syncwarp();
        if (i + 1 < n) fetch_rows(it.qi_lo + i + 1);
        // visible columns: r_min <= r < r_max (chunk keys: key <= token;
        // token < Lc, r < rows)
        int r_lo = it.pre ? 0 : (key - tok0) * tl.g;
        r_lo = r_lo < 0 ? 0 : r_lo;
        int r_hi = (it.lc - tok0) * tl.g;
        r_hi = r_hi < tl.rows ? r_hi : tl.rows;
        if (!key_valid) r_hi = 0;
        r_lo -= half * 64;
        r_hi -= half * 64;
        if (warp == 0 && lane == 0) CFA_TRACE(0, t, 0);
        if (!(ok = warp_wait(W, bar_stfull, (uint32_t)t & 1u))) break;
        if (warp == 0 && lane == 0) CFA_TRACE(0, t, 1);
        tc_fence_after_sync();
        float p[64];
        {
          uint32_t r[64];
          tmem_ld_x64(t_lane + half * 64, r);
          uint32_t pk[32];
          const uint64_t* nlse2 = reinterpret_cast<const uint64_t*>(my_lse);
          if (__all_sync(0xffffffffu, r_lo <= 0 && r_hi >= 64)) {
            // every column visible (all tiles but the diagonal and the ragged
            // ends): packed scale-and-subtract, no mask
            const uint64_t sl2x2 = f2(sl2, sl2);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              f2_split(ex2_sfu_x2(f2_fma(f2(__uint_as_float(r[2 * jj]), __uint_as_float(r[2 * jj + 1])),
                                         sl2x2, nlse2[jj])),
                       p[2 * jj], p[2 * jj + 1]);
          } else {
#pragma unroll
            for (int jj = 0; jj < 64; ++jj)
              p[jj] = (jj >= r_lo && jj < r_hi)
                          ? ex2_approx(fmaf(__uint_as_float(r[jj]), sl2, my_lse[jj]))
                          : 0.f;
          }
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) pk[jj] = pack_bf16x2(p[2 * jj], p[2 * jj + 1]);
          tmem_st_x32(t_lane + half * 64, pk);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pfull);  // P^T(i) is in TMEM: dV(i) may start
        if (warp == 0 && lane == 0) CFA_TRACE(0, t, 2);
        if (!(ok = warp_wait(W, bar_dptfull, (uint32_t)t & 1u))) break;
        if (warp == 0 && lane == 0) CFA_TRACE(0, t, 3);
        tc_fence_after_sync();
        {
          uint32_t r[64];
          tmem_ld_x64(t_lane + 128 + half * 64, r);
          uint32_t pk[32];
          const uint64_t* dl2 = reinterpret_cast<const uint64_t*>(my_dl);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            float d0, d1;
            f2_split(f2_mul(f2(p[2 * jj], p[2 * jj + 1]),
                            f2_sub(f2(__uint_as_float(r[2 * jj]), __uint_as_float(r[2 * jj + 1])),
                                   dl2[jj])),
                     d0, d1);
            pk[jj] = pack_bf16x2(d0, d1);
          }
          tmem_st_x32(t_lane + 128 + half * 64, pk);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_dsfull);
        if (warp == 0 && lane == 0) CFA_TRACE(0, t, 4);
      }
      if (!ok) break;
      if (!(ok = warp_wait(W, bar_dkvfull, (uint32_t)items & 1u))) break;
      tc_fence_after_sync();
      // this warp's half of the dV and dK rows in two TMEM loads, then the
      // hand-off (before the global stores, which the arrive would wait for)
      constexpr int HW = D / 2;
      uint32_t rv[HW], rk[HW];
      const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
      if constexpr (HW == 64) {
        tmem_ld_x64(t_dv + lane_off + half * HW, rv);
        tmem_ld_x64(t_dk + lane_off + half * HW, rk);
      } else {
        tmem_ld_x32(t_dv + lane_off + half * HW, rv);
        tmem_ld_x32(t_dk + lane_off + half * HW, rk);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dkvfree);  // dK/dV read: the next item may overwrite
      if (key_out) {
        uint4* dv = reinterpret_cast<uint4*>(dv_base + grow * D + half * HW);
        uint4* dk = reinterpret_cast<uint4*>(dk_base + grow * D + half * HW);
#pragma unroll
        for (int v = 0; v < HW / 8; ++v) {
          uint4 u, w;
          u.x = pack_bf16x2(__uint_as_float(rv[8 * v + 0]), __uint_as_float(rv[8 * v + 1]));
          u.y = pack_bf16x2(__uint_as_float(rv[8 * v + 2]), __uint_as_float(rv[8 * v + 3]));
          u.z = pack_bf16x2(__uint_as_float(rv[8 * v + 4]), __uint_as_float(rv[8 * v + 5]));
          u.w = pack_bf16x2(__uint_as_float(rv[8 * v + 6]), __uint_as_float(rv[8 * v + 7]));
          w.x = pack_bf16x2(__uint_as_float(rk[8 * v + 0]) * a.scale,
                            __uint_as_float(rk[8 * v + 1]) * a.scale);
          w.y = pack_bf16x2(__uint_as_float(rk[8 * v + 2]) * a.scale,
                            __uint_as_float(rk[8 * v + 3]) * a.scale);
          w.z = pack_bf16x2(__uint_as_float(rk[8 * v + 4]) * a.scale,
                            __uint_as_float(rk[8 * v + 5]) * a.scale);
          w.w = pack_bf16x2(__uint_as_float(rk[8 * v + 6]) * a.scale,
                            __uint_as_float(rk[8 * v + 7]) * a.scale);
          dv[v] = u;
          dk[v] = w;
        }
      }
      qn += n;
      ++items;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
  CFA_TRACE_SPAN(5, 2);
}

// Sum the dQ partials of every query tile that CTA boundaries cut, in CTA
// order (deterministic), and round to bf16.  One CTA per (query tile, 32
// rows); every thread finds the tile's parts in closed form (part_count /
// part_cta); thread t takes row t % 32 of the chunk and column slice t / 32,
// so a warp reads consecutive rows of the feature-major partials (coalesced).
constexpr int kReduceRows = 32;

template <int D>
__global__ void __launch_bounds__(256) bwd_dq_reduce_kernel(const BwdArgs a) {
  CFA_TRACE_SPAN(3, 0);
  pdl_start();
  CFA_TRACE_SPAN(3, 1);
  constexpr int CW = D / 8;
  const Tiling tl = a.tl;
  const int chunks = kTileM / kReduceRows;
  const int b = blockIdx.z, hk = blockIdx.y;
  const int qb = blockIdx.x / chunks;
  const int row = (blockIdx.x % chunks) * kReduceRows + (threadIdx.x & 31);
  const int c0col = (threadIdx.x >> 5) * CW;
  // the block's schedule row: its prefix array and its first CTA.  The status
  // word and the index loads go out together (one round trip, not two); the
  // indices are in bounds whatever the status says.
  const int srow = row_of_block(tl, qb), rg = row_grid(tl);
  const long long* wp = a.win_prefix + (size_t)srow * (a.batch + 1);
  const int status = *reinterpret_cast<volatile int*>(a.status);
  const long long w0 = wp[b], total = wp[a.batch];
  const int p0 = a.cu_p[b], lp = a.cu_p[b + 1] - p0;
  const int c0 = a.cu_c[b], lc = a.cu_c[b + 1] - c0;
  // the dQ kernel found inconsistent cu_seqlens (or gave up on a wait): its
  // partials and prefix arrays were not written
  if (status != 0) return;
  if (qb >= blocks_of_window(tl, lc)) return;
  // the tile's parts (every thread finds them; no shared list, no barrier)
  long long bs, be;
  block_span(tl, w0, hk, qb, lp, lc, &bs, &be);
  const int np = part_count(bs, be, total, rg);
  if (np == 0) return;
  const int cf = srow * rg + cta_of(bs, total, rg);
  const bool dense = total >= rg;  // then the parts are CTAs cf, cf + 1, ...
  const int token = qb * tl.tpt + row / tl.g;
  if (row >= tl.rows || token >= lc) return;
  const int head = hk * tl.g + row % tl.g;
  float acc[CW];
#pragma unroll
  for (int e = 0; e < CW; ++e) acc[e] = 0.f;
  // the loads of kBatch parts are issued before any is used (latency-bound:
  // a handful of parts per row); parts are summed in CTA order
  constexpr int kBatch = 4;
  for (int j0 = 0; j0 < np; j0 += kBatch) {
    float4 v[kBatch][CW / 4];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = j0 + u;
      const int jj = j < np ? j : 0;
      const size_t slot = (size_t)(dense ? cf + jj : srow * rg + part_cta(bs, total, rg, jj)) * 2 + (j == 0);
      const float4* src = reinterpret_cast<const float4*>(a.dq_part) + slot * (D / 4) * kTileM;
#pragma unroll
      for (int e = 0; e < CW; e += 4)
        v[u][e / 4] = (j < np) ? src[(size_t)((c0col + e) >> 2) * kTileM + row]
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
#pragma unroll
      for (int e = 0; e < CW; e += 4) {
        acc[e] += v[u][e / 4].x;
        acc[e + 1] += v[u][e / 4].y;
        acc[e + 2] += v[u][e / 4].z;
        acc[e + 3] += v[u][e / 4].w;
      }
    }
  }
  const size_t grow = (size_t)(c0 + token);
  uint4* dst = reinterpret_cast<uint4*>(a.dq + (grow * a.hq + head) * D + c0col);
#pragma unroll
  for (int e = 0; e < CW; e += 8)
    dst[e / 8] = make_uint4(pack_bf16x2(acc[e], acc[e + 1]), pack_bf16x2(acc[e + 2], acc[e + 3]),
                            pack_bf16x2(acc[e + 4], acc[e + 5]),
                            pack_bf16x2(acc[e + 6], acc[e + 7]));
  CFA_TRACE_SPAN(3, 2);
}

// delta[h, t] = sum_c dO[t, h, c] * O[t, h, c].  A CTA takes kDeltaRows
// consecutive tokens of one head (blockIdx.y), so its delta writes are one
// contiguous run; D/8 threads share a row, each loading 16 bytes of O and of
// dO, with every load of the thread issued before the first use.
constexpr int kDeltaRows = 32;
template <int D>
__global__ void __launch_bounds__(256) delta_kernel(const __nv_bfloat16* __restrict__ o,
                                                    const __nv_bfloat16* __restrict__ dout,
                                                    float* __restrict__ delta, int total_lc,
                                                    int hq) {
  CFA_TRACE_SPAN(4, 0);
  pdl_start();
  CFA_TRACE_SPAN(4, 1);
  constexpr int TPR = D / 8;              // threads per row
  constexpr int RPP = 256 / TPR;          // rows per pass of the CTA
  constexpr int NP = kDeltaRows / RPP;    // passes
  const int h = blockIdx.y;
  const int sub = threadIdx.x / TPR, part = threadIdx.x % TPR;
  uint4 xo[NP], xd[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const long long t = (long long)blockIdx.x * kDeltaRows + p * RPP + sub;
    xo[p] = xd[p] = make_uint4(0u, 0u, 0u, 0u);
    if (t < total_lc) {
      const size_t off = ((size_t)t * hq + h) * D + part * 8;
      xo[p] = *reinterpret_cast<const uint4*>(o + off);
      xd[p] = *reinterpret_cast<const uint4*>(dout + off);
    }
  }
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&xo[p]);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&xd[p]);
    float sum = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fx = __bfloat1622float2(x[e]), fy = __bfloat1622float2(y[e]);
      sum = fmaf(fx.x, fy.x, sum);
      sum = fmaf(fx.y, fy.y, sum);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const long long t = (long long)blockIdx.x * kDeltaRows + p * RPP + sub;
    if (part == 0 && t < total_lc) delta[(size_t)h * total_lc + t] = sum;
  }
  CFA_TRACE_SPAN(4, 2);
}

// q8_0 -> fp32 (exact) and bf16 (round to nearest even), one thread per value.
__global__ void dequant_q8_0_kernel(const uint8_t* __restrict__ blocks, long long n_values,
                                    float* __restrict__ out_f32,
                                    __nv_bfloat16* __restrict__ out_bf16) {
  pdl_start();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_values) return;
  const uint8_t* blk = blocks + (idx >> 5) * 34;
  const uint16_t hbits = (uint16_t)blk[0] | ((uint16_t)blk[1] << 8);
  const float d = __half2float(__ushort_as_half(hbits));
  const float v = d * (float)(int8_t)blk[2 + (idx & 31)];
  if (out_f32) out_f32[idx] = v;
  if (out_bf16) out_bf16[idx] = __float2bfloat16_rn(v);
}

// q8_0 prefix -> bf16 rows for the attention kernels' TMA maps, K and V in
// one launch (blockIdx.y).  A warp takes chunks of 32 consecutive 34-byte
// blocks (1088 bytes in, 2048 bytes out), grid-stride.  A full chunk at a
// 16-byte aligned address comes in with three 16-byte loads per lane, issued
// one chunk ahead so that they are in flight while the previous chunk is
// expanded; a ragged or unaligned chunk comes in with 2-byte loads.  Each
// lane expands one block to 32 values, fp32(d) * q (exact) rounded to
// nearest-even bf16 -- the same operand the export kernel above produces --
// into shared memory, and the warp writes the chunk's 2048 bytes back with
// 16-byte stores, 512 contiguous bytes per instruction.  The staged output is
// 16 rows of eight 16-byte columns, column XOR (row & 7), so that both the
// per-lane writes and the coalesced read-back take four wavefronts.
constexpr int kDqWarps = 8;
#ifndef CFA_DQ_CTAS_PER_SM
#define CFA_DQ_CTAS_PER_SM 8
#endif
constexpr int kDqCtasPerSm = CFA_DQ_CTAS_PER_SM;  // resident CTAs per SM the grid aims for

__device__ __forceinline__ uint32_t dq_stage_slot(int chunk16) {
  const int row = chunk16 >> 3, col = chunk16 & 7;
  return (uint32_t)(row * 8 + (col ^ (row & 7)));
}

// Expand the `nb` blocks staged at `in` into the swizzled output stage; lane
// `lane` takes block `lane`.
__device__ __forceinline__ void dq_expand_block(const uint8_t* in, uint4* out, int lane, int nb) {
  if (lane >= nb) return;
  const uint16_t* p = reinterpret_cast<const uint16_t*>(in + lane * 34);
  const float d = __half2float(__ushort_as_half(p[0]));
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint16_t two = p[1 + i];
    w[i] = pack_bf16x2(d * (float)(int8_t)(two & 0xff), d * (float)(int8_t)(two >> 8));
  }
#pragma unroll
  for (int v = 0; v < 4; ++v)
    out[dq_stage_slot(lane * 4 + v)] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
}

__global__ void __launch_bounds__(kDqWarps * 32)
    dequant_prefix_kernel(const uint8_t* __restrict__ k_blocks, const uint8_t* __restrict__ v_blocks,
                          long long n_blocks, __nv_bfloat16* __restrict__ k_out,
                          __nv_bfloat16* __restrict__ v_out) {
  CFA_TRACE_SPAN(6, 0);
  pdl_start();
  CFA_TRACE_SPAN(6, 1);
  __shared__ uint4 in_st[kDqWarps][68];
  __shared__ uint4 out_st[kDqWarps][128];
  const uint8_t* src = blockIdx.y ? v_blocks : k_blocks;
  uint4* out = reinterpret_cast<uint4*>(blockIdx.y ? v_out : k_out);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long n_chunks = (n_blocks + 31) / 32;
  const long long full = ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) ? n_blocks / 32 : 0;
  const long long stride = (long long)gridDim.x * kDqWarps;
  uint8_t* in_b = reinterpret_cast<uint8_t*>(in_st[warp]);
  long long c = (long long)blockIdx.x * kDqWarps + warp;
  // full aligned chunks, loads one chunk ahead
  uint4 r0 = make_uint4(0, 0, 0, 0), r1 = r0, r2 = r0;
  if (c < full) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src + c * 1088);
    r0 = s4[lane];
    r1 = s4[lane + 32];
    if (lane < 4) r2 = s4[lane + 64];
  }
  for (; c < full; c += stride) {
    in_st[warp][lane] = r0;
    in_st[warp][lane + 32] = r1;
    if (lane < 4) in_st[warp][lane + 64] = r2;
    __syncwarp();
    if (c + stride < full) {
      const uint4* s4 = reinterpret_cast<const uint4*>(src + (c + stride) * 1088);
      r0 = s4[lane];
      r1 = s4[lane + 32];
      if (lane < 4) r2 = s4[lane + 64];
    }
    dq_expand_block(in_b, out_st[warp], lane, 32);
    __syncwarp();
    uint4* dst = out + c * 128;
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k * 32 + lane] = out_st[warp][dq_stage_slot(k * 32 + lane)];
    __syncwarp();
  }
  // the ragged last chunk, or every chunk of an unaligned source
  for (; c < n_chunks; c += stride) {
    const long long b0 = c * 32;
    const int nb = (n_blocks - b0 < 32) ? (int)(n_blocks - b0) : 32;
    const uint16_t* s2 = reinterpret_cast<const uint16_t*>(src + b0 * 34);
    for (int i = lane; i < nb * 17; i += 32) reinterpret_cast<uint16_t*>(in_b)[i] = s2[i];
    __syncwarp();
    dq_expand_block(in_b, out_st[warp], lane, nb);
    __syncwarp();
    uint4* dst = out + c * 128;
    for (int j = lane; j < nb * 4; j += 32) dst[j] = out_st[warp][dq_stage_slot(j)];
    __syncwarp();
  }
  CFA_TRACE_SPAN(6, 2);
}

// bf16 -> q8_0 (the cache write of the walk: the chunk's K/V appended to a
// q8_0 cache).  A warp takes 32 consecutive blocks: each lane encodes one
// block -- d = absmax / 127 in fp32, codes x / d rounded half away from zero
// and clamped to +-127, scale fp16(d) nearest even -- into shared memory, then
// the warp writes the 1088 bytes out with 16-byte stores when the
// destination allows it (2-byte stores otherwise: an append may start at any
// block).
__global__ void __launch_bounds__(kDqWarps * 32)
    quantize_q8_0_kernel(const __nv_bfloat16* __restrict__ x, long long n_blocks,
                         uint8_t* __restrict__ out) {
  pdl_start();
  __shared__ uint4 stage[kDqWarps][68];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long b0 = ((long long)blockIdx.x * kDqWarps + warp) * 32;
  if (b0 >= n_blocks) return;
  const int nb = (n_blocks - b0 < 32) ? (int)(n_blocks - b0) : 32;
  uint8_t* st = reinterpret_cast<uint8_t*>(stage[warp]);
  if (lane < nb) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (b0 + lane) * 32);
    float v[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 w = src[c];
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        v[8 * c + 2 * e] = f.x;
        v[8 * c + 2 * e + 1] = f.y;
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float d = __fdiv_rn(amax, 127.f);
    const uint16_t dh = __half_as_ushort(__float2half_rn(d));
    uint16_t* o16 = reinterpret_cast<uint16_t*>(st + lane * 34);
    o16[0] = dh;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      int q[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        int c = 0;
        if (d > 0.f) {
          c = (int)roundf(__fdiv_rn(v[2 * i + u], d));
          c = c > 127 ? 127 : (c < -127 ? -127 : c);
        }
        q[u] = c;
      }
      o16[1 + i] = (uint16_t)((q[0] & 0xff) | ((q[1] & 0xff) << 8));
    }
  }
  __syncwarp();
  uint8_t* dst = out + b0 * 34;
  if (nb == 32 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (int i = lane; i < 68; i += 32) d4[i] = stage[warp][i];
  } else {
    uint16_t* d2 = reinterpret_cast<uint16_t*>(dst);
    for (int i = lane; i < nb * 17; i += 32) d2[i] = reinterpret_cast<const uint16_t*>(st)[i];
  }
}

// fp16 prefix -> bf16 rows for the attention kernels' TMA maps, K and V in one
// launch (blockIdx.y): exact fp16 -> fp32, then round to nearest even.  Eight
// values (16 bytes) per thread; n is a multiple of 64 (head_dim).
__global__ void __launch_bounds__(256) f16_to_bf16_kernel(const __half* __restrict__ k,
                                                          const __half* __restrict__ v,
                                                          long long n8,
                                                          __nv_bfloat16* __restrict__ k_out,
                                                          __nv_bfloat16* __restrict__ v_out) {
  pdl_start();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const uint4 x = reinterpret_cast<const uint4*>(blockIdx.y ? v : k)[i];
  const __half2* h = reinterpret_cast<const __half2*>(&x);
  uint4 y;
  uint32_t* w = reinterpret_cast<uint32_t*>(&y);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __half22float2(h[e]);
    w[e] = pack_bf16x2(f.x, f.y);
  }
  reinterpret_cast<uint4*>(blockIdx.y ? v_out : k_out)[i] = y;
}

// Zero the horizon rows of the prefix gradients of every window (used when
// no window has chunk rows, so nothing attends to the prefix).  One CTA per
// window; the rows of a window are contiguous.  A window whose prefix rows
// fall outside [0, total_lp) or exceed max_lp records CFA_ERR_INVALID_ARG and
// writes nothing.
__global__ void __launch_bounds__(256) zero_horizon_kernel(const int32_t* __restrict__ cu_p,
                                                           int batch, int hkv, int d, int horizon,
                                                           SeqLimits lim,
                                                           __nv_bfloat16* __restrict__ dk_p,
                                                           __nv_bfloat16* __restrict__ dv_p,
                                                           int* status) {
  const int b = blockIdx.x;
  const long long p0l = cu_p[b], p1l = cu_p[b + 1];
  if (p0l < 0 || p1l < p0l || p1l > lim.total_lp || p1l - p0l > lim.max_lp ||
      (b == 0 && p0l != 0) || (b == batch - 1 && p1l != lim.total_lp)) {
    if (threadIdx.x == 0) atomicExch(status, kStatusInvalidArg);
    return;
  }
  const int p0 = (int)p0l, lp = (int)(p1l - p0l);
  const int h = horizon < lp ? horizon : lp;
  const size_t first = (size_t)(p0 + lp - h) * hkv * d / 8, count = (size_t)h * hkv * d / 8;
  uint4* k = reinterpret_cast<uint4*>(dk_p) + first;
  uint4* v = reinterpret_cast<uint4*>(dv_p) + first;
  for (size_t i = threadIdx.x; i < count; i += blockDim.x) k[i] = v[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

cudaError_t launch_dequant_prefix(const uint8_t* k_blocks, const uint8_t* v_blocks,
                                  long long n_blocks, __nv_bfloat16* k_out,
                                  __nv_bfloat16* v_out, cudaStream_t st) {
  if (n_blocks <= 0) return cudaSuccess;
  // grid-stride: enough CTAs to fill every SM several times over, no more
  // than the chunks need
  const long long chunks = (n_blocks + 31) / 32;
  const long long ctas_needed = (chunks + kDqWarps - 1) / kDqWarps;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorUnknown;
  const long long cap = (long long)sms * kDqCtasPerSm / (v_blocks ? 2 : 1);
  const dim3 grid((unsigned)(ctas_needed < cap ? ctas_needed : cap), v_blocks ? 2 : 1);
  dequant_prefix_kernel<<<grid, kDqWarps * 32, 0, st>>>(k_blocks, v_blocks, n_blocks, k_out,
                                                        v_out);
  return cudaGetLastError();
}

int bwd_dq_smem_bytes(int d, int q8) {
  (void)q8;
  return d == 128 ? DqCfg<128>::kSmemBytes : DqCfg<64>::kSmemBytes;
}
int bwd_dkdv_smem_bytes(int d) {
  return d == 128 ? DkvCfg<128>::kSmemBytes : DkvCfg<64>::kSmemBytes;
}

namespace {
template <int D, bool ROW>
cudaError_t launch_bwd_dq_t(const Maps& m, const BwdArgs& a, cudaStream_t st) {
  auto k = bwd_dq_kernel<D, ROW>;
  cudaError_t e =
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, DqCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3((unsigned)a.tl.grid), 320, DqCfg<D>::kSmemBytes, st, m.q, m.dout, m.kp,
                    m.vp, m.kc, m.vc, a);
}
}  // namespace

cudaError_t launch_bwd_dq(const Maps& m, const BwdArgs& a, int d, int q8, cudaStream_t st) {
  (void)q8;
  const bool row = a.tl.nrow > 1;
  if (d == 128)
    return row ? launch_bwd_dq_t<128, true>(m, a, st) : launch_bwd_dq_t<128, false>(m, a, st);
  return row ? launch_bwd_dq_t<64, true>(m, a, st) : launch_bwd_dq_t<64, false>(m, a, st);
}

cudaError_t launch_bwd_dkdv(const Maps& m, const BwdArgs& a, int d, int ctas, cudaStream_t st) {
  const dim3 grid((unsigned)ctas);
  if (d == 128) {
    auto k = bwd_dkdv_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DkvCfg<128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    k<<<grid, 320, DkvCfg<128>::kSmemBytes, st>>>(m.q, m.dout, m.kc, m.vc, m.kp, m.vp, a);
  } else {
    auto k = bwd_dkdv_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DkvCfg<64>::kSmemBytes);
    if (e != cudaSuccess) return e;
    k<<<grid, 320, DkvCfg<64>::kSmemBytes, st>>>(m.q, m.dout, m.kc, m.vc, m.kp, m.vp, a);
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq_reduce(const BwdArgs& a, int d, int max_lc, cudaStream_t st) {
  const int nblk = ceil_div(max_lc > 0 ? max_lc : 1, a.tl.tpt);
  dim3 grid((unsigned)(nblk * (kTileM / kReduceRows)), (unsigned)a.hkv, (unsigned)a.batch);
  // (a normal launch: with a programmatic one the reduce's waiting CTAs took
  // the SMs the dK/dV kernel beside the dQ kernel needed, and the backward got
  // 40-90 us slower)
  if (d == 128)
    bwd_dq_reduce_kernel<128><<<grid, 256, 0, st>>>(a);
  else
    bwd_dq_reduce_kernel<64><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_delta(const __nv_bfloat16* o, const __nv_bfloat16* dout, float* delta,
                         int total_lc, int hq, int d, cudaStream_t st) {
  const dim3 blocks((unsigned)((total_lc + kDeltaRows - 1) / kDeltaRows), (unsigned)hq);
  // A programmatic launch: its CTAs are placed while the previous kernel (the
  // forward's split merge, in a training step) runs and start the moment it
  // completes (delta_kernel waits for it in pdl_start before any access).
  // Measured in a step replayed as a CUDA graph: the 8B layer's step 4% faster
  // (the merge and the dQ reduce launched this way made their steps slower).
  if (d == 128)
    return launch_pdl(delta_kernel<128>, blocks, dim3(256), 0, st, o, dout, delta, total_lc, hq);
  return launch_pdl(delta_kernel<64>, blocks, dim3(256), 0, st, o, dout, delta, total_lc, hq);
}

cudaError_t launch_f16_to_bf16(const __half* k, const __half* v, long long n, __nv_bfloat16* k_out,
                               __nv_bfloat16* v_out, cudaStream_t st) {
  const long long n8 = n / 8;
  if (n8 <= 0) return cudaSuccess;
  const dim3 grid((unsigned)((n8 + 255) / 256), 2);
  f16_to_bf16_kernel<<<grid, 256, 0, st>>>(k, v, n8, k_out, v_out);
  return cudaGetLastError();
}

cudaError_t launch_quantize_q8_0(const __nv_bfloat16* x, long long n_blocks, uint8_t* out,
                                 cudaStream_t st) {
  if (n_blocks <= 0) return cudaSuccess;
  const long long per_cta = 32LL * kDqWarps;
  const unsigned grid = (unsigned)((n_blocks + per_cta - 1) / per_cta);
  quantize_q8_0_kernel<<<grid, kDqWarps * 32, 0, st>>>(x, n_blocks, out);
  return cudaGetLastError();
}

cudaError_t launch_zero_horizon(const int32_t* cu_p, int batch, int hkv, int d, int horizon,
                                const SeqLimits& lim, __nv_bfloat16* dk_p, __nv_bfloat16* dv_p,
                                int* status, cudaStream_t st) {
  zero_horizon_kernel<<<batch, 256, 0, st>>>(cu_p, batch, hkv, d, horizon, lim, dk_p, dv_p,
                                             status);
  return cudaGetLastError();
}

cudaError_t launch_dequant_q8_0(const uint8_t* blocks, long long n_blocks, float* out_f32,
                                __nv_bfloat16* out_bf16, cudaStream_t st) {
  const long long nv = n_blocks * 32;
  const unsigned grid = (unsigned)((nv + 255) / 256);
  dequant_q8_0_kernel<<<grid, 256, 0, st>>>(blocks, nv, out_f32, out_bf16);
  return cudaGetLastError();
}

}  // namespace cfa

#ifdef CFA_TRACE_BUILD
extern "C" int cfa_trace_read_cta_bwd(unsigned long long* dst) {
  return cudaMemcpyFromSymbol(dst, cfa::cfa_trace_cta, sizeof(unsigned long long) * 2048) ==
                 cudaSuccess ? 0 : -1;
}

extern "C" int cfa_trace_read_bwd(long long* dst, int clear) {
  const size_t n = sizeof(long long) * cfa::kTraceRoles * cfa::kTraceIters * cfa::kTraceEvents;
  if (dst && cudaMemcpyFromSymbol(dst, cfa::cfa_trace_buf, n) != cudaSuccess) return -1;
  if (clear) {
    static long long zero[cfa::kTraceRoles * cfa::kTraceIters * cfa::kTraceEvents];
    if (cudaMemcpyToSymbol(cfa::cfa_trace_buf, zero, n) != cudaSuccess) return -1;
  }
  return 0;
}
// Kernel spans of this translation unit's kernels; reset = 1 re-arms them.
extern "C" int cfa_trace_read_span_bwd(unsigned long long* dst, int reset) {
  if (dst && cudaMemcpyFromSymbol(dst, cfa::cfa_trace_span, sizeof(unsigned long long) * 24) !=
                 cudaSuccess)
    return -1;
  if (reset) {
    unsigned long long init[24];
    for (int i = 0; i < 24; ++i) init[i] = (i % 3 == 2) ? 0ull : ~0ull;
    if (cudaMemcpyToSymbol(cfa::cfa_trace_span, init, sizeof(init)) != cudaSuccess) return -1;
  }
  return 0;
}
#endif
