// common.cuh -- device helpers and internal launcher declarations of libdetffn.
//
// The canonical tree (RL-Kernel PR #325, "Design": FP32-leaf / BF16-node
// midpoint reduction tree): leaves of 64 contiguous K positions; internal
// node = rne_bf16(fp32(left) + fp32(right)); the left child of a node over n
// leaves takes floor(n/2) of them.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/detffn.h"

namespace detffn {

// Programmatic dependent launch.  grid_dep_wait blocks until the grid this
// one was launched after has completed and its memory is visible (it returns
// at once when there was no such launch); grid_dep_launch lets the next grid
// on the stream start launching (its CTAs then wait in grid_dep_wait).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// A launch that may begin while the previous kernel on the stream finishes
// (programmatic dependent launch); the kernel waits in grid_dep_wait before
// touching global memory, and lets its own successor launch with
// grid_dep_launch (which takes effect once every one of its CTAs has run it).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*k)(KArgs...), dim3 grid, int threads, int smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<Args&&>(args)...);
}

constexpr int kLeaf = 64;        // leaf width (K positions per FP32 leaf)
constexpr int kMaxDepth = 24;    // stack entries; enough for < 2^22 leaves
constexpr long long kMaxK = 1ll << 27;

// ---------------------------------------------------------------------------
// Element arithmetic
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
__device__ __forceinline__ uint16_t f2bf(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));  // cvt.rn.bf16.f32
}
// Tree node: one FP32 add (round to nearest even), then round to BF16.
__device__ __forceinline__ float node(float l, float r) { return bf2f(f2bf(__fadd_rn(l, r))); }

// The backward stages of one element, with BF16 at every stage boundary:
// dU = bf16(dh * SiLU(g)), dG = bf16(bf16(dh * u) * SiLU'(g)), and the
// forward's h = bf16(SiLU(g) * u) again, from the correctly rounded tables
// (SiLU in BF16, SiLU' in FP32, indexed by the bits of g).
struct SiluBwd1 {
  uint16_t dU, dG, h;
};
__device__ __forceinline__ SiluBwd1 silu_bwd1(uint16_t dh, uint16_t g, uint16_t u, const uint16_t* __restrict__ silu,
                                              const float* __restrict__ dsilu) {
  const float d = bf2f(dh), a = bf2f(__ldg(silu + g)), uu = bf2f(u);
  const float dA = bf2f(f2bf(__fmul_rn(d, uu)));
  return SiluBwd1{f2bf(__fmul_rn(d, a)), f2bf(__fmul_rn(dA, __ldg(dsilu + g))), f2bf(__fmul_rn(a, uu))};
}

// Number of internal nodes that end at leaf j in the midpoint tree over L
// leaves, i.e. how many combines follow the push of leaf j in a left-to-right
// post-order evaluation.
__host__ __device__ __forceinline__ int combines_after(int j, int L) {
  int lo = 0, hi = L, cnt = 0;
  while (hi - lo > 1) {
    if (hi - 1 == j) cnt++;
    int mid = lo + (hi - lo) / 2;
    if (j < mid) hi = mid; else lo = mid;
  }
  return cnt;
}

__host__ __device__ __forceinline__ long long n_leaves(long long K) { return (K + kLeaf - 1) / kLeaf; }

// ---------------------------------------------------------------------------
// Internal launchers (all asynchronous on `st`; they return cudaGetLastError)
// ---------------------------------------------------------------------------
// Bounded waits of a launch: where a timeout is recorded, the poll limit of
// the role loops' waits (0 = the default), and a test-only switch under which
// the kernels issue no copies, so that their first wait runs out.
struct Waits {
  int* status = nullptr;
  long long spin = 0;
  int stall = 0;
  // The handle's tree tickets (kTcsTickets words, zero between launches):
  // the few-token kernel's CTAs count their finished pieces of a tree there,
  // and the last one folds them.  Null: a separate top-of-tree kernel does.
  int* tickets = nullptr;
};

struct Strided {
  const uint16_t* p;
  long long rs, ks;  // element strides of a row and of a K position
};

// out[r*o_rs + c] = T_K(A[r,:], B[c,:]) on CUDA cores, LANE8x8 leaves.
cudaError_t launch_tree_gemm_exact(Strided A, Strided B, long long R, long long C, long long K,
                                   uint16_t* out, long long o_rs, cudaStream_t st);

// h = rne(silu[g] * u) on rows x cols elements at r*ld + c.
cudaError_t launch_silu_mul(const uint16_t* g, const uint16_t* u, uint16_t* h, long long rows,
                            long long cols, long long ld, const uint16_t* silu_tab,
                            cudaStream_t st);
// dU = rne(dh*a), dG = rne(rne_f32(rne(dh*u) * dsilu[g])), and, where hh is
// not null, hh = rne(a*u) (the forward's h, for the down projection's weight
// gradient).
cudaError_t launch_silu_bwd(const uint16_t* dh, const uint16_t* g, const uint16_t* u,
                            uint16_t* dU, uint16_t* dG, uint16_t* hh, long long n, const uint16_t* silu_tab,
                            const float* dsilu_tab, cudaStream_t st);
// out = rne_bf16(T(g[0..n)) + T(u[0..n))), T the BF16 rank tree (n in {2,4,8}).
cudaError_t launch_rank_tree_add_bf16(const void* const* g, const void* const* u, int n, void* out, long long count,
                                      int sm_count, cudaStream_t st);
// dst[0 .. bytes) = src[0 .. bytes) (bytes even) by a kernel of plain loads
// and stores: either side may be page-locked host memory (its device-visible
// address), which the GPU then reads or writes over the host link.
cudaError_t launch_copy(const void* src, void* dst, long long bytes, int sm_count, cudaStream_t st);
// out = rne(a + b).
cudaError_t launch_add_bf16(const uint16_t* a, const uint16_t* b, uint16_t* out, long long n,
                            cudaStream_t st);
// out[c*ld_out + r] = in[r*ld_in + c] (a copy).

// Self-check: counts pairs where add.rn.bf16x2 differs from the tree node.
cudaError_t launch_check_node_add(unsigned long long begin, unsigned long long end, unsigned long long* bad,
                                  int sm_count, cudaStream_t st);
// out[i] = rne_bf16(in[i]) with the kernels' own conversion (diagnostic).
cudaError_t launch_cvt_bf16(const float* in, uint16_t* out, long long n, int sm_count, cudaStream_t st);
// Balanced rank tree over n in {1,2,4,8} buffers.
cudaError_t launch_rank_tree(const void* const* in, int n, void* out, long long count, int dtype,
                             int sm_count, cudaStream_t st);

}  // namespace detffn
