// selfcheck.cu -- host checks of arithmetic the kernels share with their
// host planning code (no device needed).
#include <map>
#include <set>
#include <utility>
#include <vector>

#include "tc.h"
#include "tcs_pieces.cuh"

namespace detffn {

unsigned long long tcs_selfcheck_ranges(int max_levels);

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
  return bad + tcs_selfcheck_ranges(max_levels);
}

// Host check of the balanced ranges and the fold units of the few-token
// kernels, by simulating every CTA of a launch: the CTA that holds each group
// (cta_of), the pieces each CTA writes segment by segment in the order its
// epilogue writes them (a one-tree unit inside its range is stored directly;
// a fused unit always goes through pieces), the slot index of each segment's
// first piece (slot_base, pieces_of), the CTAs that arrive on each unit's
// ticket at the end of their ranges, and that their count is the one the
// kernel computes as the last arrival's target.  Returns the failed cases.
unsigned long long tcs_selfcheck_ranges(int max_levels) {
  unsigned long long bad = 0;
  for (int E = 0; E <= max_levels && E <= 6; ++E) {
    const int Q = 1 << E;
    for (int fused = 0; fused < 2; ++fused)
      for (int nseg_units = 1; nseg_units <= 9; ++nseg_units) {
        const int spu = fused ? 2 : 1, UG = spu * Q;
        const long long W = (long long)nseg_units * UG;
        for (long long P = 1; P <= W && P <= 40; ++P) {
          // cta_of against the ranges.
          for (long long b = 0; b < P; ++b)
            for (long long w = b * W / P; w < (b + 1) * W / P; ++w)
              if (cta_of(w, W, P) != b) ++bad;
          std::map<long long, std::set<long long>> arrivals;
          std::set<long long> stored;  // units whose roots a CTA stored directly
          for (long long b = 0; b < P; ++b) {
            const long long blo = b * W / P, bhi = (b + 1) * W / P;
            int j = 0;  // pieces written so far, in the epilogue's order
            for (long long s = blo / Q; s * Q < bhi; ++s) {
              const long long lo = blo > s * Q ? blo : s * Q, hi = bhi < (s + 1) * Q ? bhi : (s + 1) * Q;
              const long long u = s / spu;
              const bool inside = !fused && u * UG >= blo && (u + 1) * UG <= bhi;
              if (inside) {
                stored.insert(u);
                if (pieces_of(b, s, W, P, Q, UG) != 0) ++bad;
                continue;
              }
              if (slot_base(b, s, W, P, Q, UG) != j) ++bad;
              const int n = count_pieces((int)(lo - s * Q), (int)(hi - s * Q));
              if (pieces_of(b, s, W, P, Q, UG) != n) ++bad;
              j += n;
            }
            // Range end: the units the kernel visits.
            const long long ua = blo / UG, ub = (bhi - 1) / UG;
            const long long step = fused ? 1 : (ub > ua ? ub - ua : 1);
            for (long long u = ua; u <= ub; u += step) {
              if (!fused && u * UG >= blo && (u + 1) * UG <= bhi) continue;
              arrivals[u].insert(b);
            }
            if (slot_base(b, (bhi - 1) / Q + 1, W, P, Q, UG) != j) ++bad;  // the plan's per-CTA count
          }
          for (long long u = 0; u < W / UG; ++u) {
            const long long b0 = cta_of(u * UG, W, P), b1 = cta_of((u + 1) * UG - 1, W, P);
            const bool st = stored.count(u) != 0;
            const auto it = arrivals.find(u);
            if (st) {
              if (it != arrivals.end() || b0 != b1) ++bad;  // stored by its only CTA, no ticket
              continue;
            }
            if (it == arrivals.end()) {
              ++bad;
              continue;
            }
            std::set<long long> want;
            for (long long b = b0; b <= b1; ++b) want.insert(b);
            if (it->second != want) ++bad;
          }
        }
      }
  }
  return bad;
}

}  // namespace detffn
