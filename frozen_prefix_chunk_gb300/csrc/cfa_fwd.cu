// Forward pass of frozen-prefix chunk attention on sm_103a.
//
// One CTA takes a query block (two 128-row query tiles of one KV head, rows
// packed token-major over the g query heads of the group) and one split of
// its key-tile list (prefix tiles, then the visible chunk tiles).  Roles:
//
//   warps 0-3  softmax for query tile 0      (TMEM lanes 0-127, one row each)
//   warps 4-7  softmax for query tile 1
//   warp  8    TMA producer: Q once, then K and V tiles into a ring of stages
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
// A single-split block writes bf16 O and LSE directly; otherwise each split
// writes its normalised fp32 O and its LSE to the workspace and
// fwd_combine_kernel merges them:  LSE = log sum_k exp(LSE_k),
// O = sum_k exp(LSE_k - LSE) O_k.
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
  static constexpr int kThreads = 320;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(8 * (1 + 2 * kKStages + 2 * kVStages + 7) <= 240, "barrier area");
};

// S_t = Q_t K^T: A = Q tile, B = K tile, both K-major 128B-swizzled; one MMA
// per 16 columns of head_dim.  Inside a 64-column box the K offset advances
// the start address by 32 bytes; the next box starts 16 KB further.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t a_addr, uint32_t b_addr) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0, 0);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t off = (uint32_t)(k >> 2) * kBoxBytes + (uint32_t)(k & 3) * 32u;
    mma_bf16_ss(d_tmem, smem_desc_sw128(a_addr + off, 16, 1024),
                smem_desc_sw128(b_addr + off, 16, 1024), idesc, k > 0 ? 1u : 0u);
  }
}

// O_t (+)= P_t V: A = P from TMEM (64 columns of bf16 pairs, 8 per 16 keys),
// B = V tile read MN-major (head_dim contiguous): 16 keys = two 8-row groups
// of 1024 bytes; the next 64 head_dim columns sit one box (16 KB) further.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, 0, 1);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    mma_bf16_ts(d_tmem, p_tmem + (uint32_t)(k * 8),
                smem_desc_sw128(v_addr + (uint32_t)k * 2048u, kBoxBytes, 1024), idesc,
                (accumulate || k > 0) ? 1u : 0u);
  }
}

template <int D>
__global__ void __launch_bounds__(320, 1)
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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Tiling tl = a.tl;
  const int b = blockIdx.z, hk = blockIdx.y;
  const int qblk = blockIdx.x / tl.n_split_max, split = blockIdx.x % tl.n_split_max;
  const int p0 = a.cu_p[b], lp = a.cu_p[b + 1] - p0;
  const int c0 = a.cu_c[b], lc = a.cu_c[b + 1] - c0;
  const int tok_blk = tl.q_per_cta * tl.tpt;
  const int t0 = qblk * tok_blk;
  if (t0 >= lc) return;
  const int nq = min(tl.q_per_cta, ceil_div(lc - t0, tl.tpt));
  const int np_t = ceil_div(lp, kTileN);
  const int n_kt = block_key_tiles(lp, lc, t0, tok_blk);
  const int n_split = ceil_div(n_kt, tl.tiles_per_split);
  if (split >= n_split) return;
  const int kt0 = split * tl.tiles_per_split;
  const int n = min(tl.tiles_per_split, n_kt - kt0);

  const uint32_t bars = base + C::kBarOff;
  const uint32_t bar_q = bars;
  const uint32_t bar_kfull = bars + 8;                  // [SK]
  const uint32_t bar_kempty = bar_kfull + 8 * SK;       // [SK]
  const uint32_t bar_vfull = bar_kempty + 8 * SK;       // [SV]
  const uint32_t bar_vempty = bar_vfull + 8 * SV;       // [SV]
  const uint32_t bar_sfull = bar_vempty + 8 * SV;       // [2]
  const uint32_t bar_pfull = bar_sfull + 16;            // [2]
  const uint32_t bar_ofull = bar_pfull + 16;            // [2]
  const uint32_t bar_drain = bar_ofull + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kBarOff + 240);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kBarOff + 244);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
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
    if (np_t > 0) {
      tma_prefetch_map(&map_kp);
      tma_prefetch_map(&map_vp);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{a.limit_ns, abort_flag, a.status};

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, (uint32_t)(nq * C::kBoxes * 128 * tl.rows));
      for (int qt = 0; qt < nq; ++qt)
        for (int kb = 0; kb < C::kBoxes; ++kb)
          tma_load_3d(base + C::kQOff + (qt * C::kBoxes + kb) * kBoxBytes, &map_q, bar_q, kb * 64,
                      hk * tl.g, c0 + t0 + qt * tl.tpt);
      int issued_k = 0, issued_v = 0;
      for (int i = 0; i < n; ++i) {
        const int kt = kt0 + i;
        const CUtensorMap* mk = &map_kc;
        const CUtensorMap* mv = &map_vc;
        int row0 = c0 + (kt - np_t) * kTileN;
        if (kt < np_t) {
          mk = &map_kp;
          mv = &map_vp;
          row0 = p0 + kt * kTileN;
        }
        const int sk = i % SK, sv = i % SV;
        if (!mbar_wait(W, bar_kempty + 8 * sk, ((uint32_t)(i / SK) & 1u) ^ 1u)) break;
        mbar_arrive_expect_tx(bar_kfull + 8 * sk, C::kTileBytes);
        for (int kb = 0; kb < C::kBoxes; ++kb)
          tma_load_3d(base + C::kKOff + sk * C::kTileBytes + kb * kBoxBytes, mk,
                      bar_kfull + 8 * sk, kb * 64, hk, row0);
        issued_k = i + 1;
        if (!mbar_wait(W, bar_vempty + 8 * sv, ((uint32_t)(i / SV) & 1u) ^ 1u)) break;
        mbar_arrive_expect_tx(bar_vfull + 8 * sv, C::kTileBytes);
        for (int kb = 0; kb < C::kBoxes; ++kb)
          tma_load_3d(base + C::kVOff + sv * C::kTileBytes + kb * kBoxBytes, mv,
                      bar_vfull + 8 * sv, kb * 64, hk, row0);
        issued_v = i + 1;
      }
      // Unwind: every copy this thread issued has landed before the CTA exits.
      mbar_wait_bounded(bar_q, 0, kDrainLimitNs);
      for (int i = (issued_k > SK ? issued_k - SK : 0); i < issued_k; ++i)
        mbar_wait_bounded(bar_kfull + 8 * (i % SK), (uint32_t)(i / SK) & 1u, kDrainLimitNs);
      for (int i = (issued_v > SV ? issued_v - SV : 0); i < issued_v; ++i)
        mbar_wait_bounded(bar_vfull + 8 * (i % SV), (uint32_t)(i / SV) & 1u, kDrainLimitNs);
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0) {
      bool ok = mbar_wait(W, bar_q, 0) && mbar_wait(W, bar_kfull, 0);
      // Issue order per key tile i:  PV0(i-1) S0(i) PV1(i-1) S1(i).  PV of the
      // previous tile goes first (it does not need K(i)); S_t(i) reuses the
      // TMEM columns of P_t(i-1), which the in-order MMA pipe has consumed.
      // The K(i+1) / V(i) waits sit at the end of the iteration, where the
      // tensor pipe is still busy with the work just issued; only the P
      // hand-offs remain on the critical path.
      for (int i = 0; ok && i < n; ++i) {
        const int sk = i % SK, svp = (i + SV - 1) % SV;
        for (int qt = 0; qt < nq; ++qt) {
          if (i > 0) {
            if (!(ok = mbar_wait(W, bar_pfull + 8 * qt, (uint32_t)(i - 1) & 1u))) break;
            tc_fence_after_sync();
            issue_pv<D>(tmem + 256 + qt * D, tmem + qt * 128, base + C::kVOff + svp * C::kTileBytes,
                        i - 1 > 0);
            if (qt == nq - 1) tc_commit(bar_vempty + 8 * svp);
          }
          issue_qk<D>(tmem + qt * 128, base + C::kQOff + qt * C::kTileBytes,
                      base + C::kKOff + sk * C::kTileBytes);
          tc_commit(bar_sfull + 8 * qt);
          if (qt == nq - 1) tc_commit(bar_kempty + 8 * sk);
        }
        if (!ok) break;
        if (i + 1 < n &&
            !(ok = mbar_wait(W, bar_kfull + 8 * ((i + 1) % SK), (uint32_t)((i + 1) / SK) & 1u)))
          break;
        ok = mbar_wait(W, bar_vfull + 8 * (i % SV), (uint32_t)(i / SV) & 1u);
      }
      if (ok) {
        const int i = n - 1, sv = i % SV;
        for (int qt = 0; ok && qt < nq; ++qt) {
          if (!(ok = mbar_wait(W, bar_pfull + 8 * qt, (uint32_t)i & 1u))) break;
          tc_fence_after_sync();
          issue_pv<D>(tmem + 256 + qt * D, tmem + qt * 128, base + C::kVOff + sv * C::kTileBytes,
                      i > 0);
          tc_commit(bar_ofull + 8 * qt);
        }
      }
      // Unwind: all issued MMAs have completed before TMEM is released.
      tc_commit(bar_drain);
      mbar_wait_bounded(bar_drain, 0, kDrainLimitNs);
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int qt = warp >> 2;
    if (qt < nq) {
      const int quad = warp & 3;
      const int row = quad * 32 + lane;
      const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
      const uint32_t s_col = (uint32_t)qt * 128u;
      const uint32_t o_col = 256u + (uint32_t)(qt * D);
      const int tok_tile = t0 + qt * tl.tpt;
      const int token = tok_tile + row / tl.g;
      const int head = hk * tl.g + row % tl.g;
      const bool row_valid = row < tl.rows && token < lc;
      const float sl2 = a.scale_log2;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int i = 0; i < n; ++i) {
        if (!(ok = warp_wait(W, bar_sfull + 8 * qt, (uint32_t)i & 1u))) break;
        tc_fence_after_sync();
        float s[128];
        {
          uint32_t r[128];
          tmem_ld_x128(t_lane + s_col, r);
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(r[c]);
        }
        const int kt = kt0 + i;
        // keys [0, lim) of this tile are visible to this row
        const int lim = (kt < np_t) ? (lp - kt * kTileN) : (token - (kt - np_t) * kTileN + 1);
        if (lim < 128) {
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
        }
        // row max: four independent chains of 3-input maxes
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 128; c += 8)
#pragma unroll
          for (int j = 0; j < 4; ++j) mx4[j] = fmax3(mx4[j], s[c + 2 * j], s[c + 2 * j + 1]);
        float mx = fmax3(mx4[0], mx4[1], fmaxf(mx4[2], mx4[3]));
        mx *= sl2;
        const float m_new = fmaxf(m, mx);
        const bool resc = m_new > m + 8.f;
        if (i > 0 && __any_sync(0xffffffffu, resc)) {
          // O is quiescent here: the commit behind S_t(i) also covers PV_t(i-1).
          const float alpha = resc ? ex2_approx(m - m_new) : 1.f;
#pragma unroll
          for (int cb = 0; cb < D; cb += 32) {
            uint32_t r[32];
            tmem_ld_x32(t_lane + o_col + cb, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
            tmem_st_x32(t_lane + o_col + cb, r);
          }
          tmem_st_wait();
        }
        if (resc) {
          l *= ex2_approx(m - m_new);
          m = m_new;
        }
        const float mref = (m == -INFINITY) ? 0.f : m;
        float rs4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float e0 = ex2_approx(fmaf(s[2 * c], sl2, -mref));
          const float e1 = ex2_approx(fmaf(s[2 * c + 1], sl2, -mref));
          rs4[c & 3] += e0 + e1;
          pk[c] = pack_bf16x2(e0, e1);
        }
        const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
        l += rs;
        tmem_st_x64(t_lane + s_col, pk);
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pfull + 8 * qt);
      }
      if (ok) ok = warp_wait(W, bar_ofull + 8 * qt, 0);
      if (ok) {
        tc_fence_after_sync();
        const bool single = (n_split == 1);
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const float lse_v = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        const size_t grow = (size_t)(c0 + token);
#pragma unroll
        for (int cb = 0; cb < D; cb += 32) {
          uint32_t r[32];
          tmem_ld_x32(t_lane + o_col + cb, r);
          if (row_valid) {
            if (single) {
              uint4* dst = reinterpret_cast<uint4*>(a.o + (grow * a.hq + head) * D + cb);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 u;
                u.x = pack_bf16x2(__uint_as_float(r[8 * v + 0]) * inv_l,
                                  __uint_as_float(r[8 * v + 1]) * inv_l);
                u.y = pack_bf16x2(__uint_as_float(r[8 * v + 2]) * inv_l,
                                  __uint_as_float(r[8 * v + 3]) * inv_l);
                u.z = pack_bf16x2(__uint_as_float(r[8 * v + 4]) * inv_l,
                                  __uint_as_float(r[8 * v + 5]) * inv_l);
                u.w = pack_bf16x2(__uint_as_float(r[8 * v + 6]) * inv_l,
                                  __uint_as_float(r[8 * v + 7]) * inv_l);
                dst[v] = u;
              }
            } else {
              float4* dst = reinterpret_cast<float4*>(
                  a.o_part + (((size_t)split * a.total_lc + grow) * a.hq + head) * D + cb);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(r[4 * v + 0]) * inv_l,
                                     __uint_as_float(r[4 * v + 1]) * inv_l,
                                     __uint_as_float(r[4 * v + 2]) * inv_l,
                                     __uint_as_float(r[4 * v + 3]) * inv_l);
            }
          }
        }
        if (row_valid) {
          if (single)
            a.lse[(size_t)head * a.total_lc + grow] = lse_v;
          else
            a.lse_part[((size_t)split * a.hq + head) * a.total_lc + grow] = lse_v;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// Merge the split partials of every row whose query block was split.
// One warp per (token, head) row; each lane owns D/32 consecutive columns.
template <int D>
__global__ void __launch_bounds__(256) fwd_combine_kernel(const FwdArgs a) {
  constexpr int E = D / 32;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rid = blockIdx.x * 8 + warp;
  const int t = rid / a.hq, h = rid % a.hq;
  const int p0 = a.cu_p[b], lp = a.cu_p[b + 1] - p0;
  const int c0 = a.cu_c[b], lc = a.cu_c[b + 1] - c0;
  if (t >= lc) return;
  const int tok_blk = a.tl.q_per_cta * a.tl.tpt;
  const int ns = block_splits(a.tl, lp, lc, t / tok_blk);
  if (ns <= 1) return;
  const size_t grow = (size_t)(c0 + t);
  float mx = -INFINITY;
  for (int s = 0; s < ns; ++s)
    mx = fmaxf(mx, a.lse_part[((size_t)s * a.hq + h) * a.total_lc + grow]);
  float sum = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float ls = a.lse_part[((size_t)s * a.hq + h) * a.total_lc + grow];
    sum += (ls == -INFINITY) ? 0.f : expf(ls - mx);
  }
  const float lse = mx + logf(sum);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s = 0; s < ns; ++s) {
    const float ls = a.lse_part[((size_t)s * a.hq + h) * a.total_lc + grow];
    if (ls == -INFINITY) continue;
    const float w = expf(ls - lse);
    const float* src = a.o_part + (((size_t)s * a.total_lc + grow) * a.hq + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(w, src[e], acc[e]);
  }
  __nv_bfloat16* dst = a.o + (grow * a.hq + h) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) *reinterpret_cast<uint32_t*>(dst + e) = pack_bf16x2(acc[e], acc[e + 1]);
  if (lane == 0) a.lse[(size_t)h * a.total_lc + grow] = lse;
}

}  // namespace

int fwd_smem_bytes(int d, int q8) {
  (void)q8;
  return d == 128 ? FwdCfg<128>::kSmemBytes : FwdCfg<64>::kSmemBytes;
}

cudaError_t launch_fwd(const Maps& m, const FwdArgs& a, int d, int q8, dim3 grid,
                       cudaStream_t st) {
  (void)q8;
  if (d == 128) {
    auto k = fwd_kernel<128>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdCfg<128>::kSmemBytes);
    if (e != cudaSuccess) return e;
    k<<<grid, FwdCfg<128>::kThreads, FwdCfg<128>::kSmemBytes, st>>>(m.q, m.kp, m.vp, m.kc, m.vc, a);
  } else {
    auto k = fwd_kernel<64>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdCfg<64>::kSmemBytes);
    if (e != cudaSuccess) return e;
    k<<<grid, FwdCfg<64>::kThreads, FwdCfg<64>::kSmemBytes, st>>>(m.q, m.kp, m.vp, m.kc, m.vc, a);
  }
  return cudaGetLastError();
}

cudaError_t launch_fwd_combine(const FwdArgs& a, int d, int batch, int max_lc, cudaStream_t st) {
  const long long rows = (long long)max_lc * a.hq;
  dim3 grid((unsigned)((rows + 7) / 8), (unsigned)batch);
  if (d == 128)
    fwd_combine_kernel<128><<<grid, 256, 0, st>>>(a);
  else
    fwd_combine_kernel<64><<<grid, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace cfa
