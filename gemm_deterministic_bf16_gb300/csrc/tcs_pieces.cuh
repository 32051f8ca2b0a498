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

}  // namespace detffn
