// tcs_pieces.cuh -- the split of a tile's tree into pieces, shared by the
// few-token tensor kernels (k_tcs.cu), their host planning code and the
// host self-check (selfcheck.cu).
//
// A tile of 2^E bottom groups is the perfect binary tree above its groups
// (RL-Kernel PR #325, "Design": the canonical midpoint tree; every aligned
// block of 2^m groups is one of its subtrees).  A CTA whose balanced K range
// covers groups [x, y) of a tile folds them into the range's maximal aligned
// blocks ("pieces"); the top kernel folds the pieces of all ranges of the
// tile, left to right, into the root.
#pragma once

namespace detffn {

__host__ __device__ inline int hibit(unsigned v) {  // v > 0
#ifdef __CUDA_ARCH__
  return 31 - __clz(v);
#else
  return 31 - __builtin_clz(v);
#endif
}
__host__ __device__ inline int popc(unsigned v) {
#ifdef __CUDA_ARCH__
  return __popc(v);
#else
  return __builtin_popcount(v);
#endif
}

// The pieces of groups [x, y), 0 <= x < y <= 2^E, are its maximal aligned
// blocks.  Let h be the highest bit in which x and y - 1 differ and z the
// multiple of 2^h between them: left to right, the pieces have the sizes of
// the set bits of z - x (ascending) and then of y - z (descending) -- unless
// both halves are whole, when [x, y) is itself one aligned block.
struct PieceSplit {
  int x, z, y;
  bool one;  // [x, y) is one aligned block
};
__host__ __device__ inline PieceSplit piece_split(int x, int y) {
  PieceSplit p{x, y, y, true};
  if (y - x == 1) return p;
  const int h = hibit((unsigned)(x ^ (y - 1)));
  p.z = ((y - 1) >> h) << h;
  p.one = (p.z - x == (1 << h)) && (y - p.z == (1 << h));
  return p;
}
__host__ __device__ inline int count_pieces(int x, int y) {
  const PieceSplit p = piece_split(x, y);
  return p.one ? 1 : popc((unsigned)(p.z - x)) + popc((unsigned)(y - p.z));
}

// The fold step of a piece of level m starting at group `at`, for a tile of
// 2^E groups: it merges with the pending left siblings at levels m, m+1, ...
// while its subtree is a right child, then waits on the stack at the level
// reached or is the root.
__host__ __device__ inline int fold_code(int at, int m, int E) {
  int k = 0;
  while (m + k < E && ((at >> (m + k)) & 1)) ++k;
  return m | (k << 8) | ((m + k == E) ? (1 << 16) : 0);
}

// ---------------------------------------------------------------------------
// Balanced ranges and fold units.  The work of a launch is W bottom groups:
// segment s (one tree) is groups [s Q, (s+1) Q), Q = 2^E; a fold unit is UG
// groups (one segment, or -- gate and up fused -- two).  CTA b of P takes
// groups [floor(b W / P), floor((b+1) W / P)).
// ---------------------------------------------------------------------------

// First group of CTA b's range.  Direct mode deals whole fold units, so
// every unit's roots are formed in one CTA.
__host__ __device__ __forceinline__ long long range_lo(long long b, long long W, long long P, int UG, bool direct) {
  return direct ? (b * (W / UG) / P) * UG : b * W / P;
}

// The CTA whose (balanced, not direct) range holds group w: the largest b
// with floor(b W / P) <= w.
__host__ __device__ __forceinline__ long long cta_of(long long w, long long W, long long P) {
  return ((w + 1) * P + W - 1) / W - 1;
}

// Pieces CTA b writes for segment s: those of its part of the segment,
// unless the segment's (one-tree) fold unit lies inside its range: it then
// stores that root itself and writes no pieces.  (A fused unit -- gate and
// up of a tile -- always goes through pieces: h needs both roots.)
__host__ __device__ inline int pieces_of(long long b, long long s, long long W, long long P, int Q, int UG) {
  const long long blo = b * W / P, bhi = (b + 1) * W / P;
  const long long lo = blo > s * Q ? blo : s * Q, hi = bhi < (s + 1) * Q ? bhi : (s + 1) * Q;
  if (lo >= hi) return 0;
  const long long u = s * Q / UG;
  if (UG == Q && u * UG >= blo && (u + 1) * UG <= bhi) return 0;
  return count_pieces((int)(lo - s * Q), (int)(hi - s * Q));
}

// Index of CTA b's first piece of segment s among the pieces it writes (its
// slots are filled in segment order).  With one-tree units only the two
// units at the ends of its range can hold pieces.
__host__ __device__ inline int slot_base(long long b, long long s, long long W, long long P, int Q, int UG) {
  const long long blo = b * W / P, bhi = (b + 1) * W / P;
  const long long spu = UG / Q, sf = blo / Q;
  int j = 0;
  if (spu > 1) {
    for (long long sp = sf; sp < s; ++sp) j += pieces_of(b, sp, W, P, Q, UG);
    return j;
  }
  const long long ua = blo / UG, ub = (bhi - 1) / UG;
  if (ua < s) j += pieces_of(b, ua, W, P, Q, UG);
  if (ub != ua && ub < s) j += pieces_of(b, ub, W, P, Q, UG);
  return j;
}

}  // namespace detffn
