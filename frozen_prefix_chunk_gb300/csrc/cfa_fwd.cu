// Forward pass of frozen-prefix chunk attention on sm_103a.
//
// Persistent stream-K kernel: one CTA per SM takes an equal, contiguous range
// of (query block, key tile) iterations (see cfa_sched.cuh) and walks it as
// segments, one per query block.  A query block is two 128-row query tiles of
// one KV head, rows packed token-major over the g query heads of the group.
// Roles:
//
//   warps 0-3  softmax for query tile 0      (TMEM lanes 0-127, one row each)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q per segment, K and V tiles into two rings
//   warp  9    TMEM owner and single-thread tcgen05.mma issuer
//
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,...).
// The bf16 probabilities P_t overwrite the first 64 columns of S_t and feed
// the PV MMA straight from TMEM.  The MMA warp interleaves the two tiles so
// the tensor core computes S and PV of one tile while the other tile's
// softmax runs:  PV0(i-1) S0(i) PV1(i-1) S1(i).
//
// Softmax is online, in the log2 domain, with a lazy rescale: the running
// max is only moved (and O rescaled in TMEM) when a tile's max exceeds it by
// more than 8, so the un-normalised P stays below 2^8.  Masking: keys of the
// last prefix tile beyond Lp, and chunk keys j > t (row t sits at absolute
// position Lp + t, so it sees the whole prefix).
//
// A segment that covers its whole query block writes bf16 O and LSE; the
// pieces of a block cut by CTA boundaries write normalised fp32 O and LSE
// partials, which fwd_merge_kernel combines in CTA order:
// LSE = log sum_k exp(LSE_k),  O = sum_k exp(LSE_k - LSE) O_k.
#include "cfa_kernels.cuh"
#include "cfa_ptx.cuh"

namespace cfa {
namespace {

constexpr int kBoxBytes = 128 * 128;  // one TMA box: 128 rows x 64 bf16 (128 B), swizzled


template <int D>
struct FwdCfg {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  // K and V have rings of their own: K(i) is free once the last S MMA of
  // tile i is done, V(i) only after the last PV, so K can be refilled early.
  static constexpr int kKStages = (D == 128) ? 3 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  static constexpr int kSmemBytes = kBarOff + 256 + 1024;
  static constexpr int kThreads = 352;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(8 * (2 + 2 * kKStages + 2 * kVStages + 9) <= 240, "barrier area");
};

// S_t = Q_t K^T: A = Q tile, B = K tile, both K-major 128B-swizzled; one MMA
// per 16 columns of head_dim.  Inside a 64-column box the K offset advances
// the start address by 32 bytes; the next box starts 16 KB further.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
  constexpr uint32_t hi = sw128_desc_hi(1024);
  const uint32_t a_lo = sw128_desc_lo(a_addr, 16), b_lo = sw128_desc_lo(b_addr, 16);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t off = ((uint32_t)(k >> 2) * kBoxBytes + (uint32_t)(k & 3) * 32u) >> 4;
    mma_ss_warp(d_tmem, a_lo + off, hi, b_lo + off, hi, idesc, k > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t V: A = P from TMEM (64 columns of bf16 pairs, 8 per 16 keys),
// B = V tile read MN-major (head_dim contiguous): 16 keys = two 8-row groups
// of 1024 bytes; the next 64 head_dim columns sit one box (16 KB) further.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
  constexpr uint32_t hi = sw128_desc_hi(1024);
  const uint32_t b_lo = sw128_desc_lo(v_addr, kBoxBytes);
#pragma unroll
  for (int k = 0; k < 8; ++k)
    mma_ts_warp(d_tmem, p_tmem + (uint32_t)(k * 8), b_lo + (uint32_t)k * (2048u >> 4), hi, idesc,
                (accumulate || k > 0) ? 1u : 0u);
}

template <int D, bool ROW>
__global__ void __launch_bounds__(352, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kp,
               const __grid_constant__ CUtensorMap map_vp,
               const __grid_constant__ CUtensorMap map_kc,
               const __grid_constant__ CUtensorMap map_vc, const FwdArgs a) {
  using C = FwdCfg<D>;
  constexpr int SK = C::kKStages;
  constexpr int SV = C::kVStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_addr(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_base);

  CFA_TRACE_SPAN(0, 0);
  pdl_start();
  CFA_TRACE_SPAN(0, 1);
  // A call's first kernel clears the status word once the previous work in
  // the stream is done (no separate memset: one dependent launch less).  A
  // device wait gives up only after its wall-clock limit, long after CTA 0
  // has started, so no error of this launch is cleared.
  if (a.clear_status && blockIdx.x == 0 && threadIdx.x == 0) *a.status = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  CFA_TRACE_CTA(0);
  const Tiling tl = a.tl;
  const int tok_blk = tl.q_per_cta * tl.tpt;
  const int rows_blk = tl.q_per_cta * kTileM;
  {
    // schedule prologue: shared scratch in the (not yet used) barrier area.
    // Device cu_seqlens that disagree with the host sizes: record the error
    // and leave before any load or store (every CTA reaches this verdict;
    // CTA 0 records it after its clear above).
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
  const uint32_t bar_q = bars;
  const uint32_t bar_qempty = bars + 8;
  const uint32_t bar_kfull = bars + 16;                 // [SK]
  const uint32_t bar_kempty = bar_kfull + 8 * SK;       // [SK]
  const uint32_t bar_vfull = bar_kempty + 8 * SK;       // [SV]
  const uint32_t bar_vempty = bar_vfull + 8 * SV;       // [SV]
  const uint32_t bar_sfull = bar_vempty + 8 * SV;       // [2]
  const uint32_t bar_pfull = bar_sfull + 16;            // [2]
  const uint32_t bar_ofull = bar_pfull + 16;            // [2]
  const uint32_t bar_ofree = bar_ofull + 16;            // [2]
  const uint32_t bar_drain = bar_ofree + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kBarOff + 240);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBarOff + 244);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_qempty, 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(bar_kfull + 8 * s, 1);
      mbar_init(bar_kempty + 8 * s, 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(bar_vfull + 8 * s, 1);
      mbar_init(bar_vempty + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_sfull + 8 * t, 1);
      mbar_init(bar_pfull + 8 * t, 4);
      mbar_init(bar_ofull + 8 * t, 1);
      mbar_init(bar_ofree + 8 * t, 4);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_map(&map_q);
    tma_prefetch_map(&map_kc);
    tma_prefetch_map(&map_vc);
    tma_prefetch_map(&map_kp);
    tma_prefetch_map(&map_vp);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{a.limit_ns, abort_flag, a.status};
  Segment sg;

  if (warp == 8) {
    // ---------------------------------------------------- Q and K producer
    // The whole warp walks the schedule and waits (converged); lane 0 issues.
    // V has a warp of its own (below), so a V stage still held by a PV never
    // holds back the K load queued behind it: K(i+1) is needed one P
    // hand-off before V(i+1).
    const bool leader = lane == 0;
    int it = 0, seg = 0, issued_k = 0;
    bool ok = true;
    while (ok && walk.next(sg)) {
      // the Q tiles are reused: the previous segment's S MMAs must be done
      if (seg > 0 && !(ok = warp_wait(W, bar_qempty, (uint32_t)(seg - 1) & 1u))) break;
      CFA_TRACE(4, seg, 0);
      if (leader) {
        mbar_arrive_expect_tx(bar_q, (uint32_t)(sg.nq * C::kBoxes * 128 * tl.rows));
        for (int qt = 0; qt < sg.nq; ++qt)
          for (int kb = 0; kb < C::kBoxes; ++kb)
            tma_load_3d(base + C::kQOff + (qt * C::kBoxes + kb) * kBoxBytes, &map_q, bar_q,
                        kb * 64, sg.hk * tl.g, sg.c0 + sg.qb * tok_blk + qt * tl.tpt);
      }
      __syncwarp();
      ++seg;
      const int np_t = ceil_div(sg.lp, kTileN);
      for (int kt = sg.t_begin; kt < sg.t_end; ++kt, ++it) {
        const bool pre = kt < np_t;
        const int row0 = pre ? sg.p0 + kt * kTileN : sg.c0 + (kt - np_t) * kTileN;
        const int sk = it % SK;
        // One-row schedule: the CTA's K(1) and later wait until K(0) has
        // landed (V likewise below), so that every CTA's first tiles are not
        // queued behind its later ones when all CTAs load from DRAM at once
        // (the 8B layer's step 0.6 us faster; in row mode the blocks that
        // share K/V read it in lockstep, and waiting there made it slower).
        if (!ROW && it == 1 && !(ok = warp_wait(W, bar_kfull, 0u))) break;
        if (!(ok = warp_wait(W, bar_kempty + 8 * sk, ((uint32_t)(it / SK) & 1u) ^ 1u))) break;
        CFA_TRACE(3, it, 0);
        if (leader) {
          mbar_arrive_expect_tx(bar_kfull + 8 * sk, C::kTileBytes);
          for (int kb = 0; kb < C::kBoxes; ++kb)
            tma_load_3d(base + C::kKOff + sk * C::kTileBytes + kb * kBoxBytes,
                        pre ? &map_kp : &map_kc, bar_kfull + 8 * sk, kb * 64, sg.hk, row0);
        }
        __syncwarp();
        issued_k = it + 1;
      }
    }
    // Unwind: every copy this warp issued has landed before the CTA exits.
    if (seg > 0) mbar_wait_bounded(bar_q, (uint32_t)(seg - 1) & 1u, kDrainLimitNs);
    for (int i = (issued_k > SK ? issued_k - SK : 0); i < issued_k; ++i)
      mbar_wait_bounded(bar_kfull + 8 * (i % SK), (uint32_t)(i / SK) & 1u, kDrainLimitNs);
  } else if (warp == 10) {
    // ------------------------------------------------------------ V producer
    const bool leader = lane == 0;
    int it = 0, issued_v = 0;
    bool ok = true;
    while (ok && walk.next(sg)) {
      const int np_t = ceil_div(sg.lp, kTileN);
      for (int kt = sg.t_begin; kt < sg.t_end; ++kt, ++it) {
        const bool pre = kt < np_t;
        const int row0 = pre ? sg.p0 + kt * kTileN : sg.c0 + (kt - np_t) * kTileN;
        const int sv = it % SV;
        if (!ROW && it == 1 && !(ok = warp_wait(W, bar_vfull, 0u))) break;
        if (!(ok = warp_wait(W, bar_vempty + 8 * sv, ((uint32_t)(it / SV) & 1u) ^ 1u))) break;
        CFA_TRACE(3, it, 1);
        if (leader) {
          mbar_arrive_expect_tx(bar_vfull + 8 * sv, C::kTileBytes);
          for (int kb = 0; kb < C::kBoxes; ++kb)
            tma_load_3d(base + C::kVOff + sv * C::kTileBytes + kb * kBoxBytes,
                        pre ? &map_vp : &map_vc, bar_vfull + 8 * sv, kb * 64, sg.hk, row0);
        }
        __syncwarp();
        issued_v = it + 1;
      }
    }
    for (int i = (issued_v > SV ? issued_v - SV : 0); i < issued_v; ++i)
      mbar_wait_bounded(bar_vfull + 8 * (i % SV), (uint32_t)(i / SV) & 1u, kDrainLimitNs);
  } else if (warp == 9) {
    // ----------------------------------------------------------- MMA issue
    // Issue order per key tile i of a segment:  PV0(i-1) S0(i) PV1(i-1)
    // S1(i).  PV of the previous tile goes first (it does not need K(i));
    // S_t(i) reuses the TMEM columns of P_t(i-1), which the in-order MMA
    // pipe has consumed.  The tensor pipe holds about one MMA beyond the one
    // executing, so every wait here is a bubble: the softmax warps of query
    // tile 0 wait for K(i+1) and V(i) before they hand over P0(i), and this
    // warp waits only for the P hand-offs (and K at a segment's start).  The
    // whole warp waits and issues (converged); elect.sync picks the lane that
    // issues the MMAs and commits.
    int it = 0, seg = 0;
    int ut[2] = {0, 0}, us[2] = {0, 0};  // per query tile: tiles, segments done
    // test hook: wait on a barrier nothing arrives on before the end, so the
    // bounded wait runs out and the CTA unwinds
    bool ok = !(a.debug_wait_never && !warp_wait(W, bar_drain, 0));
    while (ok && walk.next(sg)) {
      const int n = sg.t_end - sg.t_begin, nq = sg.nq;
      CFA_TRACE(4, seg, 1);
      if (!(ok = warp_wait(W, bar_q, (uint32_t)seg & 1u))) break;
      CFA_TRACE(4, seg, 2);
      if (!(ok = warp_wait(W, bar_kfull + 8 * (it % SK), (uint32_t)(it / SK) & 1u))) break;
      CFA_TRACE(4, seg, 3);
      for (int i = 0; ok && i < n; ++i) {
        const int g = it + i;
        const int sk = g % SK, svp = (g + SV - 1) % SV;
#pragma unroll
        for (int qt = 0; qt < 2; ++qt) {
          if (qt >= nq) break;
          if (i > 0) {
            // the first PV of a segment overwrites O_t: the previous
            // segment's epilogue must have read it
            if (i == 1 && us[qt] > 0 &&
                !(ok = warp_wait(W, bar_ofree + 8 * qt, (uint32_t)(us[qt] - 1) & 1u)))
              break;
            CFA_TRACE(2, it + i, 5 + qt);
            if (!(ok = warp_wait(W, bar_pfull + 8 * qt, (uint32_t)(ut[qt] + i - 1) & 1u))) break;
            CFA_TRACE(2, it + i, 2 * qt);
            tc_fence_after_sync();
            issue_pv<D>(tmem + 256 + qt * D, tmem + qt * 128,
                        base + C::kVOff + svp * C::kTileBytes, i - 1 > 0);
            if (qt == nq - 1) tc_commit_warp(bar_vempty + 8 * svp);
          }
          issue_qk<D>(tmem + qt * 128, base + C::kQOff + qt * C::kTileBytes,
                      base + C::kKOff + sk * C::kTileBytes);
          tc_commit_warp(bar_sfull + 8 * qt);
          if (qt == nq - 1) tc_commit_warp(bar_kempty + 8 * sk);
          if (qt == nq - 1 && i == n - 1) tc_commit_warp(bar_qempty);  // segment's last S
          CFA_TRACE(2, it + i, 2 * qt + 1);
        }
        if (!ok) break;
        CFA_TRACE(2, g, 4);
      }
      if (!ok) break;
      const int gl = it + n - 1, svl = gl % SV;
#pragma unroll
      for (int qt = 0; qt < 2; ++qt) {
        if (!ok || qt >= nq) break;
        if (n == 1 && us[qt] > 0 &&
            !(ok = warp_wait(W, bar_ofree + 8 * qt, (uint32_t)(us[qt] - 1) & 1u)))
          break;
        if (!(ok = warp_wait(W, bar_pfull + 8 * qt, (uint32_t)(ut[qt] + n - 1) & 1u))) break;
        tc_fence_after_sync();
        issue_pv<D>(tmem + 256 + qt * D, tmem + qt * 128, base + C::kVOff + svl * C::kTileBytes,
                    n > 1);
        tc_commit_warp(bar_ofull + 8 * qt);
        CFA_TRACE(4, seg, 4 + qt);
      }
      if (!ok) break;
      tc_commit_warp(bar_vempty + 8 * svl);  // V of the segment's last tile
      it += n;
      ++seg;
#pragma unroll
      for (int qt = 0; qt < 2; ++qt) {
        if (qt < nq) {
          ut[qt] += n;
          ++us[qt];
        }
      }
    }
    // Unwind: all issued MMAs have completed before TMEM is released.
    tc_commit_warp(bar_drain);
    mbar_wait_bounded(bar_drain, 0, kDrainLimitNs);
  } else {
    // ------------------------------------------------------------- softmax
    const int qt = warp >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t s_col = (uint32_t)qt * 128u;
    const uint32_t o_col = 256u + (uint32_t)(qt * D);
    const float sl2 = a.scale_log2;
    // Every kPolyEvery-th exponential pair of a tile with no masked key runs
    // on the FMA pipe (ex2_poly_x2), which shortens the row's turn on the
    // special-function unit: the forward 2-3% faster in the row-mode
    // instantiation.  The one-row instantiation spills with it at this
    // kernel's 168 registers and keeps the SFU for every pair.
    constexpr int kPolyEvery = ROW ? 8 : 0;
    int u = 0, us = 0;  // tiles and segments this query tile has processed
    bool ok = true;
    while (ok && walk.next(sg)) {
      if (qt >= sg.nq) continue;
      const int n = sg.t_end - sg.t_begin;
      const int np_t = ceil_div(sg.lp, kTileN);
      const int token = sg.qb * tok_blk + qt * tl.tpt + row / tl.g;
      const int head = sg.hk * tl.g + row % tl.g;
      const bool row_valid = row < tl.rows && token < sg.lc;
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < n; ++i, ++u) {
        if (i == 0 && quad == 0 && lane == 0) CFA_TRACE(5, 10 + us, 4 * qt);
        if (qt == 0 && quad == 0) {
          // V(u) and K(u+1) are in shared memory before P0(u) is handed over,
          // so the MMA warp need not wait for them itself; checking here,
          // before S0(u) is ready, keeps the waits off the hand-off
          if (!(ok = warp_wait(W, bar_vfull + 8 * (u % SV), (uint32_t)(u / SV) & 1u))) break;
          if (i + 1 < n &&
              !(ok = warp_wait(W, bar_kfull + 8 * ((u + 1) % SK), (uint32_t)((u + 1) / SK) & 1u)))
            break;
        }
        if (i == 0 && quad == 0 && lane == 0) CFA_TRACE(5, 10 + us, 4 * qt + 1);
        if (!(ok = warp_wait(W, bar_sfull + 8 * qt, (uint32_t)u & 1u))) break;
        if (quad == 0 && lane == 0) CFA_TRACE(qt, u, 0);
        tc_fence_after_sync();
        uint32_t r[128];  // S row; reused in place for the packed P
        tmem_ld_x128(t_lane + s_col, r);
        const int kt = sg.t_begin + i;
        // keys [0, lim) of this tile are visible to this row
        const int lim =
            (kt < np_t) ? (sg.lp - kt * kTileN) : (token - (kt - np_t) * kTileN + 1);
        if (lim < 128) {
#pragma unroll
          for (int c = 0; c < 128; ++c) r[c] = (c < lim) ? r[c] : 0xff800000u;  // -inf
        }
        // row max: four independent chains of 3-input maxes
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 128; c += 8)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            mx4[j] = fmax3(mx4[j], __uint_as_float(r[c + 2 * j]), __uint_as_float(r[c + 2 * j + 1]));
        const float mx = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3])) * sl2;
        const float m_new = fmaxf(m, mx);
        const bool resc = m_new > m + 8.f;
        const float alpha = resc ? ex2_approx(m - m_new) : 1.f;
        if (resc) {
          l *= alpha;
          m = m_new;
        }
        const float mref = (m == -INFINITY) ? 0.f : m;
        // exponentials in pairs: the scale-and-subtract and the row sums run
        // as packed f32x2 instructions
        const uint64_t sl2x2 = f2(sl2, sl2), nmx2 = f2(-mref, -mref);
        uint64_t rs2[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
        if (kPolyEvery > 0 && __all_sync(0xffffffffu, lim >= 128)) {
          // no masked key in the warp's rows: every kPolyEvery-th pair on
          // the FMA pipe
          constexpr int P = kPolyEvery > 0 ? kPolyEvery : 1;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const uint64_t x =
                f2_fma(f2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])), sl2x2, nmx2);
            const uint64_t e = (c % P == P - 1) ? ex2_poly_x2(x) : ex2_sfu_x2(x);
            rs2[c & 1] = f2_add(rs2[c & 1], e);
            float e0, e1;
            f2_split(e, e0, e1);
            r[c] = pack_bf16x2(e0, e1);
          }
        } else
        {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const uint64_t e = ex2_sfu_x2(
                f2_fma(f2(__uint_as_float(r[2 * c]), __uint_as_float(r[2 * c + 1])), sl2x2, nmx2));
            rs2[c & 1] = f2_add(rs2[c & 1], e);
            float e0, e1;
            f2_split(e, e0, e1);
            r[c] = pack_bf16x2(e0, e1);  // r[2c], r[2c+1] are no longer needed
          }
        }
        float l0, l1, l2, l3;
        f2_split(rs2[0], l0, l1);
        f2_split(rs2[1], l2, l3);
        l += (l0 + l1) + (l2 + l3);
        if (quad == 0 && lane == 0) CFA_TRACE(qt, u, 1);
        tmem_st_x64(t_lane + s_col, reinterpret_cast<const uint32_t(&)[64]>(r));
        tmem_st_wait();
        if (quad == 0 && lane == 0) CFA_TRACE(qt, u, 2);  // P stored
        if (i > 0 && __any_sync(0xffffffffu, resc)) {
          // O is quiescent here (the commit behind S_t(i) also covers
          // PV_t(i-1)) and PV_t(i) waits for our arrival below.
#pragma unroll
          for (int cb = 0; cb < D; cb += 32) {
            uint32_t o[32];
            tmem_ld_x32(t_lane + o_col + cb, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st_x32(t_lane + o_col + cb, o);
          }
          tmem_st_wait();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) CFA_TRACE(qt, u, quad == 0 ? 3 : 4 + quad);  // hand-off
        if (lane == 0) mbar_arrive(bar_pfull + 8 * qt);
      }
      if (!ok) break;
      if (!(ok = warp_wait(W, bar_ofull + 8 * qt, (uint32_t)us & 1u))) break;
      if (quad == 0 && lane == 0) CFA_TRACE(5, us, 2 * qt);
      tc_fence_after_sync();
      const bool final_out = !sg.head && !sg.tail;
      const int slot = sg.head ? 0 : 1;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const float lse_v = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      const size_t grow = (size_t)(sg.c0 + token);
      const size_t pslot = (size_t)blockIdx.x * 2 + slot;
      const int prow_in = qt * kTileM + row;
      const size_t prow = pslot * rows_blk + prow_in;
      // The whole O row in one TMEM load; O_t may be overwritten by the next
      // segment's first PV as soon as it is in registers.  The hand-off goes
      // before the global stores: an mbarrier arrive releases the thread's
      // earlier writes, so after the stores it would wait for them to drain.
      uint32_t r[D];
      if constexpr (D == 128)
        tmem_ld_x128(t_lane + o_col, r);
      else
        tmem_ld_x64(t_lane + o_col, r);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ofree + 8 * qt);
      if (row_valid) {
        if (final_out) {
          uint4* dst = reinterpret_cast<uint4*>(a.o + (grow * a.hq + head) * D);
#pragma unroll
          for (int v = 0; v < D / 8; ++v) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv_l,
                              __uint_as_float(r[8 * v + 1]) * inv_l);
            w.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l,
                              __uint_as_float(r[8 * v + 3]) * inv_l);
            w.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l,
                              __uint_as_float(r[8 * v + 5]) * inv_l);
            w.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l,
                              __uint_as_float(r[8 * v + 7]) * inv_l);
            dst[v] = w;
          }
        } else {
          // feature-major partial [D/4][rows][4]: a warp's store is one
          // contiguous 512-byte run
          float4* dst =
              reinterpret_cast<float4*>(a.o_part) + pslot * (D / 4) * rows_blk + prow_in;
#pragma unroll
          for (int v = 0; v < D / 4; ++v)
            dst[(size_t)v * rows_blk] = make_float4(__uint_as_float(r[4 * v + 0]) * inv_l,
                                                    __uint_as_float(r[4 * v + 1]) * inv_l,
                                                    __uint_as_float(r[4 * v + 2]) * inv_l,
                                                    __uint_as_float(r[4 * v + 3]) * inv_l);
        }
      }
      if (row_valid) {
        if (final_out)
          a.lse[(size_t)head * a.total_lc + grow] = lse_v;
        else
          a.lse_part[prow] = lse_v;
      }
      if (quad == 0 && lane == 0) CFA_TRACE(5, us, 2 * qt + 1);
      ++us;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  CFA_TRACE_CTA(1);
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
  CFA_TRACE_SPAN(0, 2);
}

// Merge the partials of every query block that CTA boundaries cut.  One CTA
// per (query block, 32 packed rows); every thread finds the block's parts in
// closed form (part_count / part_cta: slot 1 of the first CTA, slot 0 of the
// others).  Thread t takes row r0 + t % 32 and the column slice t / 32 (of
// 8), so the lanes of a warp read consecutive rows of the feature-major
// partials (coalesced).
constexpr int kMergeRows = 32;

#ifdef CFA_TRACE_BUILD
static __device__ unsigned long long cfa_trace_merge[4 * 1024];
#define CFA_TRACE_MERGE(ev)                                                                  \
  do {                                                                                       \
    const int lin = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;         \
    if (threadIdx.x == 0 && lin < 1024) cfa_trace_merge[4 * lin + (ev)] = global_timer_ns_raw(); \
  } while (0)
#else
#define CFA_TRACE_MERGE(ev) \
  do {                      \
  } while (0)
#endif

template <int D>
__global__ void __launch_bounds__(256) fwd_merge_kernel(const FwdArgs a) {
  CFA_TRACE_SPAN(1, 0);
  pdl_start();
  CFA_TRACE_SPAN(1, 1);
  constexpr int CW = D / 8;  // columns per thread
  const Tiling tl = a.tl;
  const int tok_blk = tl.q_per_cta * tl.tpt;
  const int rows_blk = tl.q_per_cta * kTileM;
  const int chunks = rows_blk / kMergeRows;
  const int b = blockIdx.z, hk = blockIdx.y;
  const int qb = blockIdx.x / chunks;
  const int r = (blockIdx.x % chunks) * kMergeRows + (threadIdx.x & 31);
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
  // the forward kernel found inconsistent cu_seqlens (or gave up on a wait):
  // its partials and prefix arrays were not written
  if (status != 0) return;
  CFA_TRACE_MERGE(0);
  if (qb >= blocks_of_window(tl, lc)) return;
  CFA_TRACE_MERGE(1);
  // the block's parts (every thread finds them; no shared list, no barrier)
  long long bs, be;
  block_span(tl, w0, hk, qb, lp, lc, &bs, &be);
  const int np = part_count(bs, be, total, rg);
  CFA_TRACE_MERGE(2);
  if (np == 0) return;
  const int qt = r / kTileM, row = r % kTileM;
  const int token = qb * tok_blk + qt * tl.tpt + row / tl.g;
  if (row >= tl.rows || token >= lc) return;
  const int head = hk * tl.g + row % tl.g;
  // The merge is latency-bound (a handful of parts per row): loads are issued
  // kBatch parts at a time before any is used.  With at most kBatch parts (the
  // common case) the LSE and O loads go out together, one round trip; more
  // parts take an online max/sum pass over the LSEs, then the O pass.
  constexpr int kBatch = 4;
  const int cf = srow * rg + cta_of(bs, total, rg);
  const bool dense = total >= rg;  // then the parts are CTAs cf, cf + 1, ...
  auto slot_of = [&](int j) {
    const int jj = j < np ? j : 0;
    const int c = dense ? cf + jj : srow * rg + part_cta(bs, total, rg, jj);
    return (size_t)c * 2 + (j == 0);
  };
  const float4* o4 = reinterpret_cast<const float4*>(a.o_part);
  float acc[CW];
#pragma unroll
  for (int e = 0; e < CW; ++e) acc[e] = 0.f;
  float lse;
  auto accumulate = [&](int j0, const float (&ls)[kBatch], const float4 (&v)[kBatch][CW / 4]) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const float w = (j0 + u < np && ls[u] != -INFINITY) ? expf(ls[u] - lse) : 0.f;
#pragma unroll
      for (int e = 0; e < CW; e += 4) {
        acc[e] = fmaf(w, v[u][e / 4].x, acc[e]);
        acc[e + 1] = fmaf(w, v[u][e / 4].y, acc[e + 1]);
        acc[e + 2] = fmaf(w, v[u][e / 4].z, acc[e + 2]);
        acc[e + 3] = fmaf(w, v[u][e / 4].w, acc[e + 3]);
      }
    }
  };
  auto load_batch = [&](int j0, float (&ls)[kBatch], float4 (&v)[kBatch][CW / 4]) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int j = j0 + u;
      const size_t slot = slot_of(j);
      ls[u] = (j < np) ? a.lse_part[slot * rows_blk + r] : -INFINITY;
#pragma unroll
      for (int e = 0; e < CW; e += 4)
        v[u][e / 4] = (j < np) ? o4[slot * (D / 4) * rows_blk + (size_t)((c0col + e) >> 2) * rows_blk + r]
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  if (np <= kBatch) {
    float ls[kBatch];
    float4 v[kBatch][CW / 4];
    load_batch(0, ls, v);
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) mx = fmaxf(mx, ls[u]);
    float sum = 0.f;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) sum += (ls[u] == -INFINITY) ? 0.f : expf(ls[u] - mx);
    lse = mx + logf(sum);
    accumulate(0, ls, v);
  } else if (np <= 2 * kBatch) {
    // two rounds of loads: all LSEs with the first batch of O, then the rest
    float ls[kBatch], ls2[kBatch];
    float4 v[kBatch][CW / 4];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      ls2[u] = (kBatch + u < np) ? a.lse_part[slot_of(kBatch + u) * rows_blk + r] : -INFINITY;
    load_batch(0, ls, v);
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) mx = fmaxf(mx, fmaxf(ls[u], ls2[u]));
    float sum = 0.f;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      sum += (ls[u] == -INFINITY) ? 0.f : expf(ls[u] - mx);
      sum += (ls2[u] == -INFINITY) ? 0.f : expf(ls2[u] - mx);
    }
    lse = mx + logf(sum);
    accumulate(0, ls, v);
    load_batch(kBatch, ls, v);
    accumulate(kBatch, ls, v);
  } else {
    float mx = -INFINITY, sum = 0.f;
    for (int j0 = 0; j0 < np; j0 += kBatch) {
      float ls[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) ls[u] = (j0 + u < np) ? a.lse_part[slot_of(j0 + u) * rows_blk + r] : -INFINITY;
      float bm = mx;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) bm = fmaxf(bm, ls[u]);
      if (bm == -INFINITY) continue;
      sum = (mx == -INFINITY) ? 0.f : sum * expf(mx - bm);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) sum += (ls[u] == -INFINITY) ? 0.f : expf(ls[u] - bm);
      mx = bm;
    }
    lse = mx + logf(sum);
    for (int j0 = 0; j0 < np; j0 += kBatch) {
      float ls[kBatch];
      float4 v[kBatch][CW / 4];
      load_batch(j0, ls, v);
      accumulate(j0, ls, v);
    }
  }
  const size_t grow = (size_t)(c0 + token);
  uint4* dst = reinterpret_cast<uint4*>(a.o + (grow * a.hq + head) * D + c0col);
#pragma unroll
  for (int e = 0; e < CW; e += 8)
    dst[e / 8] = make_uint4(pack_bf16x2(acc[e], acc[e + 1]), pack_bf16x2(acc[e + 2], acc[e + 3]),
                            pack_bf16x2(acc[e + 4], acc[e + 5]),
                            pack_bf16x2(acc[e + 6], acc[e + 7]));
  if (threadIdx.x < 32) a.lse[(size_t)head * a.total_lc + grow] = lse;
  CFA_TRACE_MERGE(3);
  CFA_TRACE_SPAN(1, 2);
}

}  // namespace

int fwd_smem_bytes(int d, int q8) {
  (void)q8;
  return d == 128 ? FwdCfg<128>::kSmemBytes : FwdCfg<64>::kSmemBytes;
}

namespace {
template <int D, bool ROW>
cudaError_t launch_fwd_t(const Maps& m, const FwdArgs& a, cudaStream_t st) {
  auto k = fwd_kernel<D, ROW>;
  cudaError_t e =
      cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, FwdCfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3((unsigned)a.tl.grid), FwdCfg<D>::kThreads, FwdCfg<D>::kSmemBytes, st,
                    m.q, m.kp, m.vp, m.kc, m.vc, a);
}
}  // namespace

cudaError_t launch_fwd(const Maps& m, const FwdArgs& a, int d, int q8, cudaStream_t st) {
  (void)q8;
  const bool row = a.tl.nrow > 1;
  if (d == 128) return row ? launch_fwd_t<128, true>(m, a, st) : launch_fwd_t<128, false>(m, a, st);
  return row ? launch_fwd_t<64, true>(m, a, st) : launch_fwd_t<64, false>(m, a, st);
}

cudaError_t launch_fwd_merge(const FwdArgs& a, int d, int max_lc, cudaStream_t st) {
  const int rows_blk = a.tl.q_per_cta * kTileM;
  const int nblk = ceil_div(max_lc > 0 ? max_lc : 1, a.tl.q_per_cta * a.tl.tpt);
  dim3 grid((unsigned)(nblk * (rows_blk / kMergeRows)), (unsigned)a.hkv, (unsigned)a.batch);
  if (d == 128)
    fwd_merge_kernel<128><<<grid, 256, 0, st>>>(a);
  else
    fwd_merge_kernel<64><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace cfa

#ifdef CFA_TRACE_BUILD
extern "C" int cfa_trace_read_cta_fwd(unsigned long long* dst) {
  return cudaMemcpyFromSymbol(dst, cfa::cfa_trace_cta, sizeof(unsigned long long) * 2048) ==
                 cudaSuccess ? 0 : -1;
}

extern "C" int cfa_trace_read_merge(unsigned long long* dst) {
  return cudaMemcpyFromSymbol(dst, cfa::cfa_trace_merge, sizeof(unsigned long long) * 4096) ==
                 cudaSuccess ? 0 : -1;
}

extern "C" int cfa_trace_read_fwd(long long* dst, int clear) {
  const size_t n = sizeof(long long) * cfa::kTraceRoles * cfa::kTraceIters * cfa::kTraceEvents;
  if (dst && cudaMemcpyFromSymbol(dst, cfa::cfa_trace_buf, n) != cudaSuccess) return -1;
  if (clear) {
    static long long zero[cfa::kTraceRoles * cfa::kTraceIters * cfa::kTraceEvents];
    if (cudaMemcpyToSymbol(cfa::cfa_trace_buf, zero, n) != cudaSuccess) return -1;
  }
  return 0;
}
// Kernel spans of this translation unit's kernels; reset = 1 re-arms them.
extern "C" int cfa_trace_read_span_fwd(unsigned long long* dst, int reset) {
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
