// k_exact.cu -- the exact CUDA-core tree contraction, any operand layout.
//
// out[r, c] = T_K(A[r, :], B[c, :]) with the canonical FP32-leaf / BF16-node
// midpoint tree (RL-Kernel PR #325, "Design").  Each leaf is computed in the
// LANE8x8 order: eight groups of eight contiguous K positions, each summed in
// ascending order with fused multiply-adds from +0, then
// ((s0+s1)+(s2+s3))+((s4+s5)+(s6+s7)) in FP32.  A bf16*bf16 product is exact
// in FP32, so this is the same value a CPU evaluation of that order gives.
//
// This is the general-layout path (transposed operands of the backward pass,
// odd shapes, tiny problems).  A 64x64 output tile per CTA; per leaf, both
// operand tiles are staged in shared memory as FP32 ([k][row], zero-filled
// outside the problem, which adds +0 to a group sum and changes nothing).
// Each thread owns a 4x4 block of outputs and a per-output stack of tree
// entries; the stack schedule (combines after each leaf) is uniform.
#include "common.cuh"

namespace detffn {
namespace {

constexpr int kT = 64;        // tile rows (A) and columns (B)
constexpr int kPad = kT + 4;  // shared row stride (keeps float4 alignment)
constexpr int kThreads = 256;
constexpr int kStack = 16;    // entries; enough for L < 2^15 leaves

__device__ __forceinline__ void load_tile(float (*sm)[kPad], const Strided& X, long long r0,
                                          long long R, long long k0, long long K) {
  const int tid = threadIdx.x;
  if (X.ks == 1) {  // K-contiguous rows: neighbouring threads read neighbouring k
    for (int i = tid; i < kT * kLeaf; i += kThreads) {
      const int k = i & (kLeaf - 1), r = i / kLeaf;
      const long long gr = r0 + r, gk = k0 + k;
      sm[k][r] = (gr < R && gk < K) ? bf2f(X.p[gr * X.rs + gk]) : 0.0f;
    }
  } else {  // otherwise neighbouring threads read neighbouring rows
    for (int i = tid; i < kT * kLeaf; i += kThreads) {
      const int r = i & (kT - 1), k = i / kT;
      const long long gr = r0 + r, gk = k0 + k;
      sm[k][r] = (gr < R && gk < K) ? bf2f(X.p[gr * X.rs + gk * X.ks]) : 0.0f;
    }
  }
}

__global__ void __launch_bounds__(kThreads) k_tree_gemm_exact(Strided A, Strided B, long long R,
                                                              long long C, long long K,
                                                              uint16_t* __restrict__ out,
                                                              long long o_rs) {
  __shared__ __align__(16) float As[kLeaf][kPad];
  __shared__ __align__(16) float Bs[kLeaf][kPad];
  const long long r0 = (long long)blockIdx.y * kT, c0 = (long long)blockIdx.x * kT;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int L = (int)n_leaves(K);

  float st[kStack][4][4];
  int sp = 0;

  for (int j = 0; j < L; ++j) {
    __syncthreads();
    load_tile(As, A, r0, R, (long long)j * kLeaf, K);
    load_tile(Bs, B, c0, C, (long long)j * kLeaf, K);
    __syncthreads();

    float even[4][4], half[4][4], q0[4][4], leaf[4][4];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      float s[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[i][c] = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int k = g * 8 + e;
        const float4 a = *reinterpret_cast<const float4*>(&As[k][ty * 4]);
        const float4 b = *reinterpret_cast<const float4*>(&Bs[k][tx * 4]);
        const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) s[i][c] = __fmaf_rn(av[i], bv[c], s[i][c]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if ((g & 1) == 0) {
            even[i][c] = s[i][c];
          } else {
            const float pair = __fadd_rn(even[i][c], s[i][c]);  // s_{g-1} + s_g
            if ((g & 2) == 0) {
              half[i][c] = pair;                                 // (s0+s1) or (s4+s5)
            } else {
              const float q = __fadd_rn(half[i][c], pair);       // q0 or q1
              if (g == 3) q0[i][c] = q;
              else leaf[i][c] = __fadd_rn(q0[i][c], q);         // q0 + q1
            }
          }
        }
    }

    // Push the leaf, then apply the combines that end at leaf j.
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) st[sp][i][c] = leaf[i][c];
    ++sp;
    for (int n = combines_after(j, L); n > 0; --n) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) st[sp - 2][i][c] = node(st[sp - 2][i][c], st[sp - 1][i][c]);
      --sp;
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long r = r0 + ty * 4 + i;
    if (r >= R) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const long long cc = c0 + tx * 4 + c;
      if (cc >= C) continue;
      out[r * o_rs + cc] = (L > 0) ? f2bf(st[0][i][c]) : (uint16_t)0;
    }
  }
}

}  // namespace

cudaError_t launch_tree_gemm_exact(Strided A, Strided B, long long R, long long C, long long K,
                                   uint16_t* out, long long o_rs, cudaStream_t st) {
  if (R <= 0 || C <= 0) return cudaSuccess;
  if (n_leaves(K) >= (1ll << (kStack - 1))) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)((C + kT - 1) / kT), (unsigned)((R + kT - 1) / kT));
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  k_tree_gemm_exact<<<grid, kThreads, 0, st>>>(A, B, R, C, K, out, o_rs);
  return cudaGetLastError();
}

}  // namespace detffn
