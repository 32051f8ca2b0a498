// selfcheck.cu -- host checks of arithmetic the kernels share with their
// host planning code (no device needed).
#include <utility>
#include <vector>

#include "tc.h"
#include "tcs_pieces.cuh"

namespace detffn {

// Host check of the piece machinery the kernels above share with their host
// planning code: for every tile of 2^E groups, E <= max_levels, (1) the
// closed-form pieces of every group range equal its greedy decomposition
// into maximal aligned blocks, and (2) for every split of the tile into three
// consecutive ranges, folding the ranges' pieces left to right with their
// fold codes pairs every right child with its own left sibling and ends in
// the root exactly once (nodes tracked as (level, index)).  Returns the
// number of failed cases.
unsigned long long tcs_selfcheck_pieces(int max_levels) {
  struct Node {
    int lv, idx;
  };
  unsigned long long bad = 0;
  std::vector<std::pair<int, int>> g, c;
  for (int E = 0; E <= max_levels && E <= kTcsMaxLv; ++E) {
    const int Q = 1 << E;
    auto pieces = [&](int x, int y, std::vector<std::pair<int, int>>& out) {  // (start, size), left to right
      out.clear();
      const PieceSplit p = piece_split(x, y);
      if (p.one) {
        out.push_back({x, y - x});
        return;
      }
      int at = x;
      for (unsigned rem = (unsigned)(p.z - x); rem;) {
        const unsigned bit = rem & (0u - rem);
        out.push_back({at, (int)bit});
        at += (int)bit;
        rem -= bit;
      }
      for (unsigned rem = (unsigned)(y - p.z); rem;) {
        const unsigned bit = 1u << hibit(rem);
        out.push_back({at, (int)bit});
        at += (int)bit;
        rem -= bit;
      }
    };
    for (int x = 0; x < Q; ++x)
      for (int y = x + 1; y <= Q; ++y) {
        g.clear();
        for (int cur = x; cur < y;) {
          int sz = cur ? (cur & -cur) : Q;
          while (cur + sz > y) sz >>= 1;
          g.push_back({cur, sz});
          cur += sz;
        }
        pieces(x, y, c);
        if (c != g || count_pieces(x, y) != (int)g.size()) ++bad;
      }
    for (int c1 = 0; c1 <= Q; ++c1)
      for (int c2 = c1; c2 <= Q; ++c2) {
        Node stk[kTcsMaxLv + 1];
        bool full[kTcsMaxLv + 1] = {};
        int roots = 0;
        bool ok = true;
        const int cuts[4] = {0, c1, c2, Q};
        for (int r = 0; r < 3 && ok; ++r) {
          if (cuts[r] == cuts[r + 1]) continue;
          pieces(cuts[r], cuts[r + 1], c);
          for (const auto& pc : c) {
            const int m = hibit((unsigned)pc.second);
            const int code = fold_code(pc.first, m, E);
            const int k = (code >> 8) & 0xFF;
            Node cur{m, pc.first >> m};
            if ((code & 0xFF) != m) ok = false;
            for (int i = 0; i < k && ok; ++i) {  // merge with the pending left sibling at level m + i
              const Node l = stk[m + i];
              if (!full[m + i] || l.lv != m + i || cur.lv != m + i || (l.idx & 1) || cur.idx != l.idx + 1) ok = false;
              full[m + i] = false;
              cur = Node{m + i + 1, l.idx >> 1};
            }
            if (code >> 16) {
              if (cur.lv != E || cur.idx != 0) ok = false;
              ++roots;
            } else {
              if (m + k >= E || full[m + k]) ok = false;
              else {
                stk[m + k] = cur;
                full[m + k] = true;
              }
            }
          }
        }
        for (int l = 0; l <= E; ++l)
          if (full[l]) ok = false;
        if (!ok || roots != 1) ++bad;
      }
  }
  return bad;
}

// Host check of the one-launch forward's schedule (see fwd_block_of): for
// every covered (H, I, SMs) of a grid of shapes, each down block runs on
// exactly one CTA, no CTA holds more than one tile or block, the tiles that
// count into a range are exactly those whose 64 columns of h make up the K
// range its blocks read, each range has one block per tree (so its waiters
// are two per tree), the trees' blocks tile their K axis, and the fold of a
// tree's pieces fits the pipeline stages.  Returns the failed cases.
unsigned long long tcs_selfcheck_fused_schedule(unsigned long long* cases) {
  static const long long dims[] = {256, 512, 768, 1024, 1536, 2048, 3072, 4096, 6144, 8192, 12288};
  static const int sms_list[] = {1, 2, 8, 16, 66, 76, 132, 148, 152, 160};
  unsigned long long bad = 0, n = 0;
  for (long long H : dims)
    for (long long I : dims)
      for (int sms : sms_list) {
        TcsFusedInfo f;
        if (!tcs_forward_fused_info(8, H, I, sms, &f)) continue;
        ++n;
        bool ok = f.nA * 64LL == I && f.fold_n >= 2 && f.fold_n * f.trees == f.nB && f.nA <= f.P && f.nB <= f.P &&
                  (long long)f.fold_n * f.bG * f.GB * 64 == I && ((long long)f.bG * f.fold_n == (1LL << f.EB)) &&
                  f.per_range == f.bG * f.GB && f.waiters == 2 * f.trees && f.GB >= 2 &&
                  f.fold_n * 128 * 32 * 2 <= f.nstage * (128 * 64 * 2 + 32 * 64 * 2) && f.smem <= 113 * 1024 &&
                  f.scratch >= (size_t)f.nB * 128 * 32 * 2;
        std::vector<int> blocks_seen(f.nB, 0), range_tiles(f.fold_n, 0), range_blocks(f.fold_n, 0);
        for (int b = 0; b < f.P && ok; ++b) {
          const int j = fwd_block_of(b, f.nA, f.P);
          if (j < f.nB) {
            ++blocks_seen[j];
            const int tree = fwd_tree_of(j, f.fold_n), range = fwd_range_of(j, f.fold_n);
            if (tree >= f.trees || range >= f.fold_n) ok = false;
            else ++range_blocks[range];
            // The block's K range of I, in 64-column leaves, and the tiles counted into its range.
            const long long k0 = (long long)range * f.bG * f.GB, k1 = k0 + (long long)f.bG * f.GB;
            for (int t = 0; t < f.nA && ok; ++t) {
              const bool counted = fwd_tile_range(t, f.per_range) == range, inside = t >= k0 && t < k1;
              if (counted != inside) ok = false;
            }
          }
        }
        for (int t = 0; t < f.nA && ok; ++t) {
          const int r = fwd_tile_range(t, f.per_range);
          if (r >= f.fold_n) ok = false;
          else ++range_tiles[r];
        }
        for (int j = 0; j < f.nB && ok; ++j) ok = blocks_seen[j] == 1;
        for (int r = 0; r < f.fold_n && ok; ++r) ok = range_tiles[r] == f.per_range && 2 * range_blocks[r] == f.waiters;
        if (!ok) ++bad;
      }
  if (cases) *cases = n;
  return bad;
}

}  // namespace detffn
