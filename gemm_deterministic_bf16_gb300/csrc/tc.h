// tc.h -- launcher of the tensor-core (tcgen05) tree contraction.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace detffn {

// Bottom-group size G and number of upper levels E such that L = G * 2^E with
// G in {1, 2, 3}; false when the tensor-core kernel does not cover L leaves.
bool tc_tree_shape(long long L, int* G, int* E);

// One contraction of a (possibly two-problem) launch.
struct TcProblem {
  const uint16_t* A;
  long long lda;
  const uint16_t* B;  // [C, K] (row stride ldb); with b_mn, [K, C] (C contiguous)
  long long ldb;
  uint16_t* out;
  bool b_mn = false;  // B read MN-major (no transposed copy needed)
  bool a_mn = false;  // A given as [K, R] (R contiguous, row stride lda), read MN-major
};

// A contraction whose K axis (the tokens, for the weight gradients) is given
// in chunks of one operand: chunk c holds tokens [sum of earlier chunks,
// + tokens[c]) at base[c] (same row stride as the operand, 16-byte aligned),
// read through a tensor map of its own -- one virtual K axis, no gather copy.
// Every chunk but the last holds a multiple of 64 tokens (a leaf never spans
// two chunks); op 1: operand A (read MN-major), op 2: operand B (MN-major).
constexpr int kMaxKChunks = 8;
struct TcKChunks {
  int op = 0;
  int n = 0;
  const uint16_t* base[kMaxKChunks] = {};
  long long tokens[kMaxKChunks] = {};
};

// Up to two same-shaped contractions in one launch (their tiles interleave).
cudaError_t launch_tc_gemms(const TcProblem* problems, int np, long long R, long long C, long long K,
                            long long ld_r, long long ld_c, const Waits& wt, int sm_count, cudaStream_t st,
                            float* dump = nullptr, const TcKChunks* kc = nullptr);

// out[r*ld_r + c*ld_c] = T_K(A[r, :], B[c, :]) for r < R, c < C; A and B are
// K-contiguous BF16 with row strides lda, ldb (elements, multiples of 8) and
// 16-byte-aligned bases; output tiles of 128 x 128, one CTA per SM.  With
// b_mn, B is given as [K, C] with C contiguous (row stride ldb), with a_mn, A
// as [K, R] with R contiguous (row stride lda); such operands are read
// MN-major by the tensor core.
cudaError_t launch_tc_gemm(const uint16_t* A, long long lda, const uint16_t* B, long long ldb,
                           long long R, long long C, long long K, uint16_t* out, long long ld_r,
                           long long ld_c, const Waits& wt, int sm_count, cudaStream_t st,
                           bool b_mn = false, bool a_mn = false, float* dump = nullptr);

// A 2-D BF16 tensor map over rows x K (row stride ld elements), 128-byte
// swizzle, boxes of 64 (K) x box_rows.
bool tc_make_map(CUtensorMap* m, const uint16_t* base, long long rows, long long K, long long ld, int box_rows);

// ---------------------------------------------------------------------------
// Few-token contractions (k_tcs.cu): out[r * ldo + c] = T_K(X[r, :], W[c, :])
// for r < R <= 32 tokens and c < C weight rows, the weights streamed once with
// the work split evenly over two CTAs per SM (balanced K ranges whose partial
// subtrees a second kernel folds into the canonical tree).
// ---------------------------------------------------------------------------
constexpr int kTcsMaxLv = 8;      // at most 2^8 bottom groups (K <= 3 * 256 * 64)
constexpr int kTcsMaxShards = 8;  // K shards per problem in one launch

struct TcsPlan {
  int R = 0, G = 0, E = 0, T = 0, np = 0, ns = 1, P = 0, cap = 0, nstage = 0, top_smem = 0;
  long long C = 0, K = 0, W = 0;    // K: the contraction length of one shard
  bool direct = false;  // whole tiles per CTA, roots stored directly (no scratch, no top kernel)
  size_t scratch = 0;   // bytes of piece slots the launch needs
  // Aligned ranges of at most kTcsFoldMax pieces per tree: each CTA's range is
  // one aligned block (one piece), fold_n of them per tree, and the last CTA
  // of a tree to finish folds them (no top kernel).  0: a top kernel folds.
  int fold_n = 0;
  // Kernels a launch takes: one, or the streaming kernel and its top kernel.
  int launches(bool plain) const { return direct || (plain && fold_n > 0) ? 1 : 2; }
};
constexpr int kTcsFoldMax = 8;    // pieces per tree the last CTA folds
constexpr int kTcsTickets = 1024; // tree tickets per handle (a fused launch has at most 2 x SMs trees)
constexpr int kTcsRanges = 64;    // fused decode forward: range counters per handle (two words each)

// Plans a launch on at most max_ctas CTAs (two per SM is the design point).
// False when the shape is not covered (R > 32, or K's leaf count not 1, 2^d or
// 3 * 2^d with at most 2^8 bottom groups).  The results never depend on the
// plan: only the split of each tree into pieces does.  With ns > 1, each
// problem is ns contractions over consecutive K ranges of K positions each
// (K a multiple of 64): shard q reads K positions [q K, (q+1) K) of the
// operands and writes its own output (out + q * oss), one tree each.
// Without direct, the CTAs take equal aligned blocks of 2^b groups, for the
// smallest 2^b that needs at most max_ctas CTAs; where a block holds whole
// trees (2^b >= a tree's groups) and whole_ok is set, the plan is direct with
// that many trees per CTA: balanced, and no pieces at all.
bool tcs_plan(long long R, long long C, long long K, int np, int max_ctas, bool direct, TcsPlan* plan,
              int ns = 1, bool whole_ok = true);

struct TcsProblem {
  const uint16_t* W;  // [C, K] weights, row stride ldw (multiple of 8), 16-byte aligned;
  long long ldw;      //   with w_mn, [K, C] (C contiguous), row stride ldw
  const uint16_t* X;  // [R, K] tokens, row stride ldx (multiple of 8), 16-byte aligned
  long long ldx;
  uint16_t* out;      // out[r * ldo + c]
  bool w_mn = false;  // weights read MN-major (no transposed copy needed)
};

// One or two same-shaped contractions (plan.np): two launches on `st`, or one
// in direct mode (scratch unused).
cudaError_t launch_tcs(const TcsPlan& plan, const TcsProblem* problems, long long ldo, void* scratch,
                       size_t scratch_bytes, const Waits& wt, cudaStream_t st, float* dump = nullptr,
                       long long oss = 0);

// Gate (problems[0]) and up (problems[1]) with the SiLU * up stage boundary
// fused into the top of the trees: h[r * ldo + c] = bf16(bf16(SiLU(gate)) * up);
// gate and up are stored only where problems[p].out is non-null.
cudaError_t launch_tcs_gateup(const TcsPlan& plan, const TcsProblem* problems, uint16_t* h, long long ldo,
                              const uint16_t* silu, void* scratch, size_t scratch_bytes, const Waits& wt,
                              cudaStream_t st);

// Gate and up of R <= 32 tokens with h = bf16(bf16(SiLU(gate)) * up) in one
// launch and no scratch: every CTA takes whole tiles of 64 rows of Wg over the
// same 64 rows of Wu (the MMA's 128 rows) and writes h, and gate and up where
// not null, itself.  C (rows of each weight) a multiple of 64.
cudaError_t launch_tcs_gateup_stacked(long long R, long long C, long long K, const uint16_t* Wg, const uint16_t* Wu,
                                      long long ldw, const uint16_t* X, long long ldx, uint16_t* gate, uint16_t* up,
                                      uint16_t* h, long long ldo, const uint16_t* silu, int sm_count, const Waits& wt,
                                      cudaStream_t st);

// The whole decode forward of R <= 32 tokens in one launch: x [R, H], Wg,
// Wu [I, H], Wd [H, I] (rows of H and I elements, 16-byte aligned), h [R, I]
// written (and gate, up where not null), out [R, H].  Stacked gate/up tiles
// and the down projection's folded trees, as launch_tcs_gateup_stacked and
// launch_tcs compute them (the same bits); a down block starts once the
// gate/up tiles of its K range are done.  Needs the tickets and range
// counters of `wt` and plan scratch bytes at `scratch`.  Returns
// cudaErrorNotSupported, launching nothing, for shapes it does not cover
// (tcs_forward_fused_covers false).
bool tcs_forward_fused_covers(long long R, long long H, long long I, int sm_count, size_t* scratch);

// The one-launch forward's unit schedule, shared by the kernel and the host
// check: CTA b of P takes gate/up tile b when b < nA, then down block
// j = fwd_block_of(b) when j < nB; block j is aligned block fwd_range_of(j)
// of down tree fwd_tree_of(j) (fold_n blocks per tree); gate/up tile t
// (64 columns of h) counts into range fwd_tile_range(t).
__host__ __device__ inline int fwd_block_of(int b, int nA, int P) {
  const int j = (b - nA) % P;
  return j < 0 ? j + P : j;
}
__host__ __device__ inline int fwd_tree_of(int j, int fold_n) { return j / fold_n; }
__host__ __device__ inline int fwd_range_of(int j, int fold_n) { return j % fold_n; }
__host__ __device__ inline int fwd_tile_range(int t, int per_range) { return t / per_range; }

// The one-launch forward's geometry for (R, H, I, SMs), for host checks.
struct TcsFusedInfo {
  int P, nA, nB, bG, GA, GB, EA, EB, fold_n, trees, per_range, waiters, nstage, smem;
  size_t scratch;
};
bool tcs_forward_fused_info(long long R, long long H, long long I, int sm_count, TcsFusedInfo* info);

// Host check of the one-launch forward's schedule over a set of shapes and
// SM counts (every down block on one CTA, each range counting exactly the
// gate/up tiles of its K range, waiter counts, shared-memory room); returns
// the failed cases and sets *cases to the shapes it covered.
unsigned long long tcs_selfcheck_fused_schedule(unsigned long long* cases);
cudaError_t launch_tcs_forward_fused(long long R, long long H, long long I, const uint16_t* x, const uint16_t* Wg,
                                     const uint16_t* Wu, const uint16_t* Wd, uint16_t* h, uint16_t* gate,
                                     uint16_t* up, uint16_t* out, const uint16_t* silu, void* scratch,
                                     size_t scratch_bytes, int sm_count, const Waits& wt, cudaStream_t st);

// Host check of the few-token kernels' piece decomposition and fold codes
// over every tile of up to 2^max_levels groups; returns the failed cases.
unsigned long long tcs_selfcheck_pieces(int max_levels);

}  // namespace detffn
