// tc.h -- launcher of the tensor-core (tcgen05) tree contraction.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace detffn {

// Bottom-group size G and number of upper levels E such that L = G * 2^E with
// G in {1, 2, 3}; false when the tensor-core kernel does not cover L leaves.
bool tc_tree_shape(long long L, int* G, int* E);

// Optional scratch for splitting K into aligned subtrees: block-root planes
// and one ticket per output tile (zero on entry; the kernel leaves them zero).
struct TcScratch {
  uint16_t* part = nullptr;
  size_t part_elems = 0;
  unsigned* cnt = nullptr;
  size_t cnt_elems = 0;
};

// One contraction of a (possibly two-problem) launch.
struct TcProblem {
  const uint16_t* A;
  long long lda;
  const uint16_t* B;
  long long ldb;
  uint16_t* out;
};

// Up to two same-shaped contractions in one launch (their units interleave);
// scratch must hold both problems' block-root planes and tickets.
cudaError_t launch_tc_gemms(const TcProblem* problems, int np, long long R, long long C, long long K,
                            long long ld_r, long long ld_c, int bn, const TcScratch& scratch, int* status,
                            long long spin_limit, int sm_count, cudaStream_t st);

// out[r*ld_r + c*ld_c] = T_K(A[r, :], B[c, :]) for r < R, c < C; A and B are
// K-contiguous BF16 with row strides lda, ldb (elements, multiples of 8) and
// 16-byte-aligned bases.  bn in {32, 64, 128} is the tile width over C.
// With scratch, K is split into up to 16 aligned subtrees when there are
// fewer output tiles than two per SM (the result is the same tree).
cudaError_t launch_tc_gemm(const uint16_t* A, long long lda, const uint16_t* B, long long ldb,
                           long long R, long long C, long long K, uint16_t* out, long long ld_r,
                           long long ld_c, int bn, const TcScratch& scratch, int* status,
                           long long spin_limit, int sm_count, cudaStream_t st);

}  // namespace detffn
