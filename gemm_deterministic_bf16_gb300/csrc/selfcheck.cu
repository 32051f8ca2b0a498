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

}  // namespace detffn
