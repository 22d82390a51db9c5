// Host-side check of the stream-K schedule in cfa_sched.cuh (the logic every
// persistent kernel runs on the device): for one configuration read from the
// command line it walks every CTA's iteration range and checks that
//   * every key tile of every query block is covered by exactly one segment,
//     in increasing order, and no segment is empty;
//   * a segment's head / tail flags say whether earlier / later key tiles of
//     its block belong to other CTAs;
//   * block_parts lists exactly the CTAs holding a segment of the block, in
//     CTA order, the one without `head` first;
//   * each CTA's iterations, virtual setup ones included, are within one of
//     the mean of its schedule row.
// With nrow > 1 (row mode) the grid is nrow independent schedules of G / nrow
// CTAs, row r holding query block r of every (window, KV head); every check
// then applies per row, with the row's own prefix array and iteration count.
// Prints "OK <total iterations> <segments>" or the first violation.
//
// Mode "seq" checks the kernels' cu_seqlens validation instead: given the
// host sizes and two raw cu_seqlens arrays (which need not be consistent), it
// prints VALID or INVALID as seqlens_valid decides, and checks that the
// per-window test window_valid, which the kernels run one window per thread,
// agrees with a direct statement of the rule.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <vector>

#include "cfa_sched.cuh"

using namespace cfa;

// The rule, stated directly: both arrays start at 0, never decrease, end at
// the host totals, and no window is longer than the host maxima.
static bool rule(const std::vector<long long>& p, const std::vector<long long>& c,
                 const SeqLimits& s) {
  const size_t n = p.size();
  if (n < 2 || p[0] != 0 || c[0] != 0) return false;
  if (p[n - 1] != s.total_lp || c[n - 1] != s.total_lc) return false;
  for (size_t i = 0; i + 1 < n; ++i) {
    if (p[i + 1] < p[i] || c[i + 1] < c[i]) return false;
    if (p[i + 1] - p[i] > s.max_lp || c[i + 1] - c[i] > s.max_lc) return false;
  }
  return true;
}

static int seq_mode(int argc, char** argv) {
  // args: seq total_lp total_lc max_lp max_lc batch cp_0 .. cp_batch cc_0 .. cc_batch
  if (argc < 7) return 2;
  SeqLimits s;
  s.total_lp = atoi(argv[2]);
  s.total_lc = atoi(argv[3]);
  s.max_lp = atoi(argv[4]);
  s.max_lc = atoi(argv[5]);
  const int batch = atoi(argv[6]);
  if (batch < 1 || argc != 7 + 2 * (batch + 1)) return 2;
  std::vector<int32_t> cp(batch + 1), cc(batch + 1);
  std::vector<long long> lp(batch + 1), lc(batch + 1);
  for (int i = 0; i <= batch; ++i) {
    lp[i] = strtoll(argv[7 + i], nullptr, 10);
    lc[i] = strtoll(argv[8 + batch + i], nullptr, 10);
    cp[i] = (int32_t)lp[i];
    cc[i] = (int32_t)lc[i];
  }
  const bool v = seqlens_valid(cp.data(), cc.data(), batch, s);
  if (v != rule(lp, lc, s)) {
    printf("FAIL seqlens_valid disagrees with the rule\n");
    return 1;
  }
  printf(v ? "VALID\n" : "INVALID\n");
  return 0;
}

int main(int argc, char** argv) {
  if (argc > 1 && std::strcmp(argv[1], "seq") == 0) return seq_mode(argc, argv);
  // args: G hkv g q_per_cta setup nrow batch lp_0 lc_0 lp_1 lc_1 ...
  if (argc < 8) return 2;
  const int G = atoi(argv[1]), hkv = atoi(argv[2]), g = atoi(argv[3]);
  const int qpc = atoi(argv[4]), setup = atoi(argv[5]), nrow = atoi(argv[6]);
  const int batch = atoi(argv[7]);
  if (argc != 8 + 2 * batch || nrow < 1 || G % nrow != 0) return 2;
  std::vector<int32_t> cu_p(batch + 1, 0), cu_c(batch + 1, 0);
  for (int b = 0; b < batch; ++b) {
    cu_p[b + 1] = cu_p[b] + atoi(argv[8 + 2 * b]);
    cu_c[b + 1] = cu_c[b] + atoi(argv[9 + 2 * b]);
  }
  Tiling tl;
  tl.g = g;
  tl.tpt = kTileM / g;
  tl.rows = tl.tpt * g;
  tl.q_per_cta = qpc;
  tl.grid = G;
  tl.setup = setup;
  tl.nrow = nrow;
  const int rg = row_grid(tl);
  // row mode: every window with chunk rows has exactly nrow query blocks
  for (int b = 0; b < batch && nrow > 1; ++b) {
    const int lc = cu_c[b + 1] - cu_c[b];
    if (lc > 0 && blocks_of_window(tl, lc) != nrow) return 2;
  }
  // window prefixes of every schedule row, as plan_schedule computes them
  std::vector<std::vector<long long>> wps(nrow, std::vector<long long>(batch + 1, 0));
  long long W = 0;
  for (int r = 0; r < nrow; ++r) {
    for (int b = 0; b < batch; ++b)
      wps[r][b + 1] = wps[r][b] + (long long)hkv * head_work_row(tl, cu_p[b + 1] - cu_p[b],
                                                                  cu_c[b + 1] - cu_c[b], r);
    W += wps[r][batch];
  }
  // (b, hk, qb) -> segments as (cta, t_begin, t_end, head, tail)
  struct Seg { int cta, tb, te; bool head, tail; };
  std::map<long long, std::vector<Seg>> by_block;
  long long n_seg = 0;
  for (int c = 0; c < G; ++c) {
    const int row = c / rg, j = c % rg;
    const std::vector<long long>& wp = wps[row];
    const long long Wr = wp[batch];
    const long long start = cta_begin(j, Wr, rg);
    if (start >= cta_begin(j + 1, Wr, rg)) continue;
    int b0 = -1;
    for (int b = 0; b < batch; ++b)
      if (wp[b + 1] > wp[b] && wp[b] <= start && start < wp[b + 1]) b0 = b;
    if (b0 < 0) { printf("FAIL cta %d: no window holds iteration %lld\n", c, start); return 1; }
    SegmentWalkerT<false> walk1;
    SegmentWalkerT<true> walkr;
    if (nrow > 1)
      walkr.init(cu_p.data(), cu_c.data(), batch, hkv, tl, c, Wr, b0, wp[b0]);
    else
      walk1.init(cu_p.data(), cu_c.data(), batch, hkv, tl, c, Wr, b0, wp[b0]);
    Segment sg;
    long long last_key = -1;
    while (nrow > 1 ? walkr.next(sg) : walk1.next(sg)) {
      ++n_seg;
      if (sg.t_end <= sg.t_begin) { printf("FAIL cta %d: empty segment\n", c); return 1; }
      const long long key = ((long long)sg.b * hkv + sg.hk) * 1000000 + sg.qb;
      if (key <= last_key) { printf("FAIL cta %d: blocks out of order\n", c); return 1; }
      last_key = key;
      by_block[key].push_back({c, sg.t_begin, sg.t_end, sg.head, sg.tail});
    }
  }
  long long n_blocks = 0;
  for (int b = 0; b < batch; ++b) {
    const int lp = cu_p[b + 1] - cu_p[b], lc = cu_c[b + 1] - cu_c[b];
    for (int hk = 0; hk < hkv; ++hk)
      for (int qb = 0, nb = blocks_of_window(tl, lc); qb < nb; ++qb) {
        ++n_blocks;
        const long long key = ((long long)b * hkv + hk) * 1000000 + qb;
        const int nk = block_iters(tl, lp, lc, qb) - setup;
        const auto& v = by_block[key];
        int next = 0;
        for (size_t i = 0; i < v.size(); ++i) {
          if (v[i].tb != next) { printf("FAIL block %lld: gap or overlap at tile %d\n", key, next); return 1; }
          if (v[i].head != (v[i].tb > 0) || v[i].tail != (v[i].te < nk)) {
            printf("FAIL block %lld: head/tail flags\n", key); return 1;
          }
          if (i > 0 && v[i].cta <= v[i - 1].cta) { printf("FAIL block %lld: CTA order\n", key); return 1; }
          next = v[i].te;
        }
        if (next != nk) { printf("FAIL block %lld: covers %d of %d tiles\n", key, next, nk); return 1; }
        if (nrow > 1 && qb >= nrow) { printf("FAIL block %lld: no schedule row\n", key); return 1; }
        const int row = row_of_block(tl, qb);
        const long long Wr = wps[row][batch];
        long long first, end;
        block_span(tl, wps[row][b], hk, qb, lp, lc, &first, &end);
        int parts[4096];
        const int np = block_parts(first, end, Wr, rg, parts, 4096);
        for (int i = 0; i < np; ++i) parts[i] += row * rg;
        if (v.size() == 1) {
          if (np != 0) { printf("FAIL block %lld: one holder but %d parts\n", key, np); return 1; }
        } else {
          if (np != (int)v.size()) { printf("FAIL block %lld: %d parts, %zu holders\n", key, np, v.size()); return 1; }
          for (int i = 0; i < np; ++i)
            if (parts[i] != v[i].cta) { printf("FAIL block %lld: part %d is CTA %d, holder %d\n", key, i, parts[i], v[i].cta); return 1; }
        }
        // the closed form the split kernels use agrees with the list
        if (part_count(first, end, Wr, rg) != np) { printf("FAIL block %lld: part_count\n", key); return 1; }
        for (int i = 0; i < np; ++i)
          if (row * rg + part_cta(first, Wr, rg, i) != parts[i]) { printf("FAIL block %lld: part_cta %d\n", key, i); return 1; }
      }
  }
  // balance: within a schedule row, iterations per CTA differ by at most one
  for (int r = 0; r < nrow; ++r) {
    const long long Wr = wps[r][batch];
    long long lo = Wr, hi = 0;
    for (int j = 0; j < rg; ++j) {
      const long long n = cta_begin(j + 1, Wr, rg) - cta_begin(j, Wr, rg);
      lo = n < lo ? n : lo;
      hi = n > hi ? n : hi;
    }
    if (hi - lo > 1) { printf("FAIL balance row %d: %lld..%lld\n", r, lo, hi); return 1; }
  }
  printf("OK %lld %lld %lld\n", W, n_seg, n_blocks);
  return 0;
}
