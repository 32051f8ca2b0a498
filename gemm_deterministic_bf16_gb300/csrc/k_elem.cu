// k_elem.cu -- BF16 stage boundaries and the balanced rank-tree reduction.
//
// Stage boundaries (RL-Kernel PR #325, "Design": "preserve BF16 stage
// boundaries in forward and backward"):
//   h  = rne_bf16(silu_bf16(g) * u)
//   dU = rne_bf16(dh * a), dA = rne_bf16(dh * u), dG = rne_bf16(rne_f32(dA * silu'(g)))
//   dX = rne_bf16(cg + cu)        (gate contribution first; PR #325,
//                                  "Communication overlap assessment")
// Products of two BF16 values are exact in FP32, so h, dU and dA round once.
//
// Rank tree (PR #357, "Design"; PR #356, "Design"):
//   ((b0 + b1) + (b2 + b3)) + ((b4 + b5) + (b6 + b7)), every node an FP32 add
//   rounded to the buffers' dtype.  It streams n inputs and one output once:
//   16-byte vectors when every pointer is 16-byte aligned, two-element words
//   for 16-bit data on 4-byte-aligned pointers, scalars otherwise; the part of
//   the count that does not fill a vector is done by scalar lanes.
#include "common.cuh"

namespace detffn {
namespace {

constexpr int kThreads = 256;

// Rows x cols elements at r*ld + c in all three arrays.
__global__ void k_silu_mul(const uint16_t* __restrict__ g, const uint16_t* __restrict__ u,
                           uint16_t* __restrict__ h, long long rows, long long cols, long long ld,
                           const uint16_t* __restrict__ silu) {
  grid_dep_wait();  // the inputs may be the previous kernel's outputs
  grid_dep_launch();
  const long long n = rows * cols;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
       t += (long long)gridDim.x * blockDim.x) {
    const long long i = (t / cols) * ld + (t % cols);
    const float a = bf2f(__ldg(silu + g[i]));
    h[i] = f2bf(__fmul_rn(a, bf2f(u[i])));
  }
}

// The backward stages, and (hh not null) the forward's h again, which the
// weight gradient of the down projection reads.
__global__ void k_silu_bwd(const uint16_t* __restrict__ dh, const uint16_t* __restrict__ g,
                           const uint16_t* __restrict__ u, uint16_t* __restrict__ dU,
                           uint16_t* __restrict__ dG, uint16_t* __restrict__ hh, long long n,
                           const uint16_t* __restrict__ silu, const float* __restrict__ dsilu) {
  grid_dep_wait();  // the inputs may be the previous kernel's outputs
  grid_dep_launch();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const SiluBwd1 r = silu_bwd1(dh[i], g[i], u[i], silu, dsilu);
    dU[i] = r.dU;
    dG[i] = r.dG;
    if (hh) hh[i] = r.h;
  }
}

// The same two stages on eight elements per thread (16-byte loads and
// stores): rows x (cols / 8) vectors at row stride ld / 8 vectors.
__device__ __forceinline__ uint32_t silu_mul2(uint32_t g2, uint32_t u2, const uint16_t* __restrict__ silu) {
  const float a0 = bf2f(__ldg(silu + (g2 & 0xFFFFu))), a1 = bf2f(__ldg(silu + (g2 >> 16)));
  const uint32_t h0 = f2bf(__fmul_rn(a0, bf2f((uint16_t)(u2 & 0xFFFFu))));
  const uint32_t h1 = f2bf(__fmul_rn(a1, bf2f((uint16_t)(u2 >> 16))));
  return h0 | (h1 << 16);
}

__global__ void k_silu_mul_v8(const uint4* __restrict__ g, const uint4* __restrict__ u, uint4* __restrict__ h,
                              long long rows, long long cv, long long ldv, const uint16_t* __restrict__ silu) {
  grid_dep_wait();  // the inputs may be the previous kernel's outputs
  grid_dep_launch();
  const long long n = rows * cv;
  for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
       t += (long long)gridDim.x * blockDim.x) {
    const long long r = t / cv;
    const long long i = r * ldv + (t - r * cv);
    const uint4 gv = __ldg(g + i), uv = __ldg(u + i);
    h[i] = make_uint4(silu_mul2(gv.x, uv.x, silu), silu_mul2(gv.y, uv.y, silu), silu_mul2(gv.z, uv.z, silu),
                      silu_mul2(gv.w, uv.w, silu));
  }
}

__device__ __forceinline__ void silu_bwd2(uint32_t dh2, uint32_t g2, uint32_t u2, const uint16_t* __restrict__ silu,
                                          const float* __restrict__ dsilu, uint32_t& dU2, uint32_t& dG2) {
  const SiluBwd1 lo = silu_bwd1((uint16_t)dh2, (uint16_t)g2, (uint16_t)u2, silu, dsilu);
  const SiluBwd1 hi = silu_bwd1((uint16_t)(dh2 >> 16), (uint16_t)(g2 >> 16), (uint16_t)(u2 >> 16), silu, dsilu);
  dU2 = (uint32_t)lo.dU | ((uint32_t)hi.dU << 16);
  dG2 = (uint32_t)lo.dG | ((uint32_t)hi.dG << 16);
}

__global__ void k_silu_bwd_v8(const uint4* __restrict__ dh, const uint4* __restrict__ g, const uint4* __restrict__ u,
                              uint4* __restrict__ dU, uint4* __restrict__ dG, uint4* __restrict__ hh, long long nv,
                              const uint16_t* __restrict__ silu, const float* __restrict__ dsilu) {
  grid_dep_wait();  // the inputs may be the previous kernel's outputs
  grid_dep_launch();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < nv;
       i += (long long)gridDim.x * blockDim.x) {
    const uint4 dv = __ldg(dh + i), gv = __ldg(g + i), uv = __ldg(u + i);
    uint4 a, b;
    silu_bwd2(dv.x, gv.x, uv.x, silu, dsilu, a.x, b.x);
    silu_bwd2(dv.y, gv.y, uv.y, silu, dsilu, a.y, b.y);
    silu_bwd2(dv.z, gv.z, uv.z, silu, dsilu, a.z, b.z);
    silu_bwd2(dv.w, gv.w, uv.w, silu, dsilu, a.w, b.w);
    dU[i] = a;
    dG[i] = b;
    if (hh)
      hh[i] = make_uint4(silu_mul2(gv.x, uv.x, silu), silu_mul2(gv.y, uv.y, silu), silu_mul2(gv.z, uv.z, silu),
                         silu_mul2(gv.w, uv.w, silu));
  }
}

__global__ void k_add_bf16(const uint16_t* __restrict__ a, const uint16_t* __restrict__ b,
                           uint16_t* __restrict__ out, long long n) {
  grid_dep_wait();  // the inputs may be the previous kernel's outputs
  grid_dep_launch();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    out[i] = f2bf(__fadd_rn(bf2f(a[i]), bf2f(b[i])));
}

// Plain copy, 16 bytes (or 2 bytes) a thread per step: every thread's loads
// are independent, so a copy over the host link keeps as many requests in
// flight as it has threads.
template <class V>
__global__ void k_copy(const V* __restrict__ src, V* __restrict__ dst, long long n) {
  grid_dep_wait();  // the source may be the previous kernel's output
  grid_dep_launch();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// ----------------------------- rank tree ---------------------------------

struct Bufs {
  const unsigned char* in[8];
  unsigned char* out;
};

template <int DT> struct Elt;
template <> struct Elt<DETFFN_F32> {
  static constexpr int kBytes = 4;
  __device__ static float ld(const unsigned char* p, long long i) { return reinterpret_cast<const float*>(p)[i]; }
  __device__ static float rnd(float v) { return v; }
  __device__ static void st(unsigned char* p, long long i, float v) { reinterpret_cast<float*>(p)[i] = v; }
  __device__ static float from_bits(uint32_t b) { return __uint_as_float(b); }
  __device__ static uint32_t to_bits(float v) { return __float_as_uint(v); }
};
template <> struct Elt<DETFFN_F16> {
  static constexpr int kBytes = 2;
  __device__ static float from_bits(uint32_t b) { return __half2float(__ushort_as_half((unsigned short)b)); }
  __device__ static uint32_t to_bits(float v) { return __half_as_ushort(__float2half_rn(v)); }
  __device__ static float ld(const unsigned char* p, long long i) { return from_bits(reinterpret_cast<const uint16_t*>(p)[i]); }
  __device__ static float rnd(float v) { return from_bits(to_bits(v)); }
  __device__ static void st(unsigned char* p, long long i, float v) { reinterpret_cast<uint16_t*>(p)[i] = (uint16_t)to_bits(v); }
};
template <> struct Elt<DETFFN_BF16> {
  static constexpr int kBytes = 2;
  __device__ static float from_bits(uint32_t b) { return bf2f((uint16_t)b); }
  __device__ static uint32_t to_bits(float v) { return f2bf(v); }
  __device__ static float ld(const unsigned char* p, long long i) { return bf2f(reinterpret_cast<const uint16_t*>(p)[i]); }
  __device__ static float rnd(float v) { return bf2f(f2bf(v)); }
  __device__ static void st(unsigned char* p, long long i, float v) { reinterpret_cast<uint16_t*>(p)[i] = f2bf(v); }
};

// The balanced tree over v[0..N): N in {1,2,4,8}; each node rounded to DT.
template <int DT, int N>
__device__ __forceinline__ float rank_tree(const float* v) {
  if (N == 1) return v[0];
  const float a = Elt<DT>::rnd(__fadd_rn(v[0], v[1]));
  if (N == 2) return a;
  const float b = Elt<DT>::rnd(__fadd_rn(v[2], v[3]));
  const float ab = Elt<DT>::rnd(__fadd_rn(a, b));
  if (N == 4) return ab;
  const float c = Elt<DT>::rnd(__fadd_rn(v[4], v[5]));
  const float d = Elt<DT>::rnd(__fadd_rn(v[6], v[7]));
  const float cd = Elt<DT>::rnd(__fadd_rn(c, d));
  return Elt<DT>::rnd(__fadd_rn(ab, cd));
}

// VEC = bytes moved per input per step (16, 4 or the element size).
// Elements [0, head) are taken one at a time and the vector steps start at
// element head, through Bv (the buffers advanced by head elements: where
// every buffer sits the same number of bytes past a VEC-byte boundary, head
// elements bring them all onto the next one); the tail after the last whole
// vector, one at a time as well.
template <int DT, int N, int VEC>
__global__ void __launch_bounds__(kThreads) k_rank_tree(Bufs B, Bufs Bv, long long count, long long head) {
  grid_dep_wait();  // the inputs may be the previous kernel's outputs
  grid_dep_launch();
  constexpr int E = Elt<DT>::kBytes;
  constexpr int PER = VEC / E;  // elements per step
  constexpr bool kScalar = (VEC == E);
  const long long nvec = kScalar ? 0 : (count - head) / PER;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long t0 = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  for (long long v = t0; v < nvec; v += stride) {
    uint32_t w[N][VEC / 4 > 0 ? VEC / 4 : 1];
#pragma unroll
    for (int s = 0; s < N; ++s) {
      if (VEC == 16) {
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(Bv.in[s]) + v);
        w[s][0] = q.x; w[s][1] = q.y; w[s][2] = q.z; w[s][3] = q.w;
      } else {
        w[s][0] = reinterpret_cast<const uint32_t*>(Bv.in[s])[v];
      }
    }
    uint32_t o[VEC / 4 > 0 ? VEC / 4 : 1];
#pragma unroll
    for (int q = 0; q < (VEC / 4 > 0 ? VEC / 4 : 1); ++q) {
      if (E == 4) {
        float x[N];
#pragma unroll
        for (int s = 0; s < N; ++s) x[s] = Elt<DT>::from_bits(w[s][q]);
        o[q] = Elt<DT>::to_bits(rank_tree<DT, N>(x));
      } else {
        float lo[N], hi[N];
#pragma unroll
        for (int s = 0; s < N; ++s) {
          lo[s] = Elt<DT>::from_bits(w[s][q] & 0xFFFFu);
          hi[s] = Elt<DT>::from_bits(w[s][q] >> 16);
        }
        o[q] = (Elt<DT>::to_bits(rank_tree<DT, N>(lo)) & 0xFFFFu) |
               (Elt<DT>::to_bits(rank_tree<DT, N>(hi)) << 16);
      }
    }
    if (VEC == 16)
      reinterpret_cast<uint4*>(Bv.out)[v] = make_uint4(o[0], o[1], o[2], o[3]);
    else
      reinterpret_cast<uint32_t*>(Bv.out)[v] = o[0];
  }
  // Scalar head and tail (all of it when PER == 1).
  for (long long i = t0; i < head; i += stride) {
    float x[N];
#pragma unroll
    for (int s = 0; s < N; ++s) x[s] = Elt<DT>::ld(B.in[s], i);
    Elt<DT>::st(B.out, i, rank_tree<DT, N>(x));
  }
  for (long long i = head + nvec * PER + t0; i < count; i += stride) {
    float x[N];
#pragma unroll
    for (int s = 0; s < N; ++s) x[s] = Elt<DT>::ld(B.in[s], i);
    Elt<DT>::st(B.out, i, rank_tree<DT, N>(x));
  }
}

// dX = rne_bf16(T(g) + T(u)) where T is the rank tree over the shard
// partials of the gate contribution (g[0..N)) and of the up contribution
// (u[0..N)): both trees and the gate-then-up addition in one pass (the same
// arithmetic as two rank-tree passes and the addition).
struct Bufs2 {
  const unsigned char* g[8];
  const unsigned char* u[8];
  unsigned char* out;
};

template <int N, bool VEC16>
__global__ void __launch_bounds__(kThreads) k_rank_tree_add(Bufs2 B, long long count) {
  grid_dep_wait();  // the inputs may be the previous kernel's outputs
  grid_dep_launch();
  using EB = Elt<DETFFN_BF16>;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long t0 = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long nvec = VEC16 ? count / 8 : 0;
  for (long long v = t0; v < nvec; v += stride) {
    uint32_t wg[N][4], wu[N][4];
#pragma unroll
    for (int s = 0; s < N; ++s) {
      const uint4 a = __ldcs(reinterpret_cast<const uint4*>(B.g[s]) + v);
      const uint4 b = __ldcs(reinterpret_cast<const uint4*>(B.u[s]) + v);
      wg[s][0] = a.x; wg[s][1] = a.y; wg[s][2] = a.z; wg[s][3] = a.w;
      wu[s][0] = b.x; wu[s][1] = b.y; wu[s][2] = b.z; wu[s][3] = b.w;
    }
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t r = 0;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float xg[N], xu[N];
#pragma unroll
        for (int s = 0; s < N; ++s) {
          xg[s] = EB::from_bits((wg[s][q] >> (16 * hf)) & 0xFFFFu);
          xu[s] = EB::from_bits((wu[s][q] >> (16 * hf)) & 0xFFFFu);
        }
        const float sum = __fadd_rn(rank_tree<DETFFN_BF16, N>(xg), rank_tree<DETFFN_BF16, N>(xu));
        r |= (EB::to_bits(sum) & 0xFFFFu) << (16 * hf);
      }
      o[q] = r;
    }
    reinterpret_cast<uint4*>(B.out)[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  for (long long i = nvec * 8 + t0; i < count; i += stride) {
    float xg[N], xu[N];
#pragma unroll
    for (int s = 0; s < N; ++s) {
      xg[s] = EB::ld(B.g[s], i);
      xu[s] = EB::ld(B.u[s], i);
    }
    EB::st(B.out, i, __fadd_rn(rank_tree<DETFFN_BF16, N>(xg), rank_tree<DETFFN_BF16, N>(xu)));
  }
}

template <int N>
cudaError_t launch_rta_n(const Bufs2& B, long long count, bool v16, int sm_count, cudaStream_t st) {
  const long long work = v16 ? count / 8 + count % 8 : count;
  long long blocks = (work + kThreads - 1) / kThreads;
  const long long cap = (long long)sm_count * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (v16) return launch_dependent(k_rank_tree_add<N, true>, dim3((unsigned)blocks), kThreads, 0, st, B, count);
  return launch_dependent(k_rank_tree_add<N, false>, dim3((unsigned)blocks), kThreads, 0, st, B, count);
}

template <int DT, int N>
cudaError_t launch_rt_n(const Bufs& B, long long count, long long head, int align_all, int sm_count,
                        cudaStream_t st) {
  constexpr int E = Elt<DT>::kBytes;
  int vec = E;
  if (align_all % 16 == 0) vec = 16;
  else if (E == 2 && align_all % 4 == 0) vec = 4;
  const long long per = vec / E;
  long long work = count / per + (count % per);
  long long blocks = (work + kThreads - 1) / kThreads;
  const long long cap = (long long)sm_count * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  Bufs Bv = B;
  for (int s = 0; s < N; ++s) Bv.in[s] = B.in[s] + head * E;
  Bv.out = B.out + head * E;
  if (vec == 16) return launch_dependent(k_rank_tree<DT, N, 16>, dim3((unsigned)blocks), kThreads, 0, st, B, Bv, count, head);
  if (vec == 4) return launch_dependent(k_rank_tree<DT, N, 4>, dim3((unsigned)blocks), kThreads, 0, st, B, Bv, count, head);
  return launch_dependent(k_rank_tree<DT, N, E>, dim3((unsigned)blocks), kThreads, 0, st, B, B, count, 0ll);
}

template <int DT>
cudaError_t launch_rt_dt(const Bufs& B, int n, long long count, int sm_count, cudaStream_t st) {
  // Where every buffer sits the same number of bytes past a 16-byte
  // boundary, the first `head` elements bring them all onto the next one.
  constexpr int E = Elt<DT>::kBytes;
  const uintptr_t r = (uintptr_t)B.out & 15u;
  bool same = true;
  for (int s = 0; s < n; ++s) same = same && ((uintptr_t)B.in[s] & 15u) == r;
  long long head = 0;
  if (same && r != 0 && r % E == 0) {
    head = (long long)((16 - r) / E);
    if (head > count) head = count;
  }
  // Largest power of two (<= 16) dividing every address from element head on.
  uintptr_t acc = (uintptr_t)(B.out + head * E);
  for (int s = 0; s < n; ++s) acc |= (uintptr_t)(B.in[s] + head * E);
  int align_all = 16;
  while (align_all > 1 && (acc % (uintptr_t)align_all) != 0) align_all >>= 1;
  if (align_all < 4) head = 0;  // no common boundary: element by element from the start
  switch (n) {
    case 1: return launch_rt_n<DT, 1>(B, count, head, align_all, sm_count, st);
    case 2: return launch_rt_n<DT, 2>(B, count, head, align_all, sm_count, st);
    case 4: return launch_rt_n<DT, 4>(B, count, head, align_all, sm_count, st);
    case 8: return launch_rt_n<DT, 8>(B, count, head, align_all, sm_count, st);
    default: return cudaErrorInvalidValue;
  }
}

unsigned grid_for(long long n, int cap_blocks) {
  long long b = (n + kThreads - 1) / kThreads;
  if (b > cap_blocks) b = cap_blocks;
  return (unsigned)(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_rank_tree_add_bf16(const void* const* g, const void* const* u, int n, void* out, long long count,
                                      int sm_count, cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  if (!g || !u || !out || !(n == 2 || n == 4 || n == 8)) return cudaErrorInvalidValue;
  Bufs2 B{};
  uintptr_t al = (uintptr_t)out;
  for (int s = 0; s < n; ++s) {
    if (!g[s] || !u[s]) return cudaErrorInvalidValue;
    B.g[s] = static_cast<const unsigned char*>(g[s]);
    B.u[s] = static_cast<const unsigned char*>(u[s]);
    al |= (uintptr_t)g[s] | (uintptr_t)u[s];
  }
  B.out = static_cast<unsigned char*>(out);
  const bool v16 = (al & 15u) == 0;
  switch (n) {
    case 2: return launch_rta_n<2>(B, count, v16, sm_count, st);
    case 4: return launch_rta_n<4>(B, count, v16, sm_count, st);
    default: return launch_rta_n<8>(B, count, v16, sm_count, st);
  }
}

cudaError_t launch_silu_mul(const uint16_t* g, const uint16_t* u, uint16_t* h, long long rows,
                            long long cols, long long ld, const uint16_t* silu_tab,
                            cudaStream_t st) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const bool a16 = (((uintptr_t)g | (uintptr_t)u | (uintptr_t)h) & 15u) == 0;
  if (a16 && cols % 8 == 0 && ld % 8 == 0)
    return launch_dependent(k_silu_mul_v8, dim3(grid_for(rows * cols / 8, 4096)), kThreads, 0, st, (const uint4*)g,
                            (const uint4*)u, (uint4*)h, rows, cols / 8, ld / 8, silu_tab);
  return launch_dependent(k_silu_mul, dim3(grid_for(rows * cols, 4096)), kThreads, 0, st, g, u, h, rows, cols, ld,
                          silu_tab);
}

cudaError_t launch_silu_bwd(const uint16_t* dh, const uint16_t* g, const uint16_t* u,
                            uint16_t* dU, uint16_t* dG, uint16_t* hh, long long n, const uint16_t* silu_tab,
                            const float* dsilu_tab, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const bool a16 =
      (((uintptr_t)dh | (uintptr_t)g | (uintptr_t)u | (uintptr_t)dU | (uintptr_t)dG | (uintptr_t)hh) & 15u) == 0;
  if (a16 && n % 8 == 0)
    return launch_dependent(k_silu_bwd_v8, dim3(grid_for(n / 8, 4096)), kThreads, 0, st, (const uint4*)dh,
                            (const uint4*)g, (const uint4*)u, (uint4*)dU, (uint4*)dG, (uint4*)hh, n / 8, silu_tab,
                            dsilu_tab);
  return launch_dependent(k_silu_bwd, dim3(grid_for(n, 4096)), kThreads, 0, st, dh, g, u, dU, dG, hh, n, silu_tab,
                          dsilu_tab);
}

cudaError_t launch_add_bf16(const uint16_t* a, const uint16_t* b, uint16_t* out, long long n,
                            cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  return launch_dependent(k_add_bf16, dim3(grid_for(n, 4096)), kThreads, 0, st, a, b, out, n);
}

cudaError_t launch_copy(const void* src, void* dst, long long bytes, int sm_count, cudaStream_t st) {
  if (bytes <= 0) return cudaSuccess;
  if ((bytes & 1) != 0) return cudaErrorInvalidValue;
  const long long cap = 8ll * (sm_count > 0 ? sm_count : 1);  // blocks: one wave of small CTAs at most
  if ((((uintptr_t)src | (uintptr_t)dst | (uintptr_t)bytes) & 15u) == 0) {
    const long long n = bytes / 16;
    const long long g = (n + kThreads - 1) / kThreads;
    return launch_dependent(k_copy<uint4>, dim3((unsigned)(g < cap ? g : cap)), kThreads, 0, st,
                            static_cast<const uint4*>(src), static_cast<uint4*>(dst), n);
  }
  const long long n = bytes / 2;
  const long long g = (n + kThreads - 1) / kThreads;
  return launch_dependent(k_copy<uint16_t>, dim3((unsigned)(g < cap ? g : cap)), kThreads, 0, st,
                          static_cast<const uint16_t*>(src), static_cast<uint16_t*>(dst), n);
}

cudaError_t launch_rank_tree(const void* const* in, int n, void* out, long long count, int dtype,
                             int sm_count, cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  Bufs B{};
  for (int s = 0; s < n; ++s) B.in[s] = static_cast<const unsigned char*>(in[s]);
  B.out = static_cast<unsigned char*>(out);
  switch (dtype) {
    case DETFFN_F32: return launch_rt_dt<DETFFN_F32>(B, n, count, sm_count, st);
    case DETFFN_F16: return launch_rt_dt<DETFFN_F16>(B, n, count, sm_count, st);
    case DETFFN_BF16: return launch_rt_dt<DETFFN_BF16>(B, n, count, sm_count, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace detffn

// ------------------- self-check of the packed node add --------------------
// Counts BF16 pairs (a, b) for which add.rn.bf16x2 differs from the tree
// node rne_bf16(fp32(a) + fp32(b)); every NaN result counts as equal to every
// other NaN.  Pairs are a = i >> 16, b = i & 0xffff for i in [begin, end).
namespace detffn {
namespace {
__device__ __forceinline__ bool is_nan_bf16(uint32_t v) { return (v & 0x7F80u) == 0x7F80u && (v & 0x7Fu); }

__global__ void k_check_node_add(unsigned long long begin, unsigned long long end, unsigned long long* bad) {
  unsigned long long local = 0;
  for (unsigned long long i = begin + blockIdx.x * (unsigned long long)blockDim.x + threadIdx.x; i < end;
       i += (unsigned long long)gridDim.x * blockDim.x) {
    const uint32_t a = (uint32_t)(i >> 16) & 0xFFFFu, b = (uint32_t)i & 0xFFFFu;
    uint32_t packed;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(packed) : "r"(a | (b << 16)), "r"(b | (a << 16)));
    const uint32_t ref = f2bf(__fadd_rn(bf2f((uint16_t)a), bf2f((uint16_t)b)));
    const uint32_t lo = packed & 0xFFFFu, hi = packed >> 16;
    const bool ok_lo = (lo == ref) || (is_nan_bf16(lo) && is_nan_bf16(ref));
    const bool ok_hi = (hi == ref) || (is_nan_bf16(hi) && is_nan_bf16(ref));
    local += (!ok_lo) + (!ok_hi);
  }
  if (local) atomicAdd(bad, local);
}
}  // namespace

cudaError_t launch_check_node_add(unsigned long long begin, unsigned long long end, unsigned long long* bad,
                                  int sm_count, cudaStream_t st) {
  k_check_node_add<<<sm_count * 8, 256, 0, st>>>(begin, end, bad);
  return cudaGetLastError();
}

// ------------- the kernels' FP32 -> BF16 rounding, exposed for tests -------------
// out[i] = f2bf(in[i]): the conversion every kernel uses for leaves, nodes
// and stage boundaries (cvt.rn.bf16.f32), so that a test can compare it with
// an independent round-to-nearest-even rule on any set of bit patterns.
namespace {
__global__ void k_cvt_bf16(const float* in, uint16_t* out, long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    out[i] = f2bf(in[i]);
}
}  // namespace

cudaError_t launch_cvt_bf16(const float* in, uint16_t* out, long long n, int sm_count, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  k_cvt_bf16<<<sm_count * 8, 256, 0, st>>>(in, out, n);
  return cudaGetLastError();
}
}  // namespace detffn
