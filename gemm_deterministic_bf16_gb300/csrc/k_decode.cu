// k_decode.cu -- exact weight-streaming tree contraction for few tokens (M <= 8 per pass).
//
// Computes C[t, n] = T_K(X[t, :], W[n, :]) with the canonical FP32-leaf /
// BF16-node midpoint tree (RL-Kernel PR #325, "Design") and LANE8x8 leaves,
// bit-identical to the generic exact kernel and to a CPU evaluation.
//
// Work split.  The L = K/64 leaves form L = 2^d * b with b in {1, 3}; the
// midpoint tree is then a perfect binary tree over 2^d bottom subtrees of b
// leaves (b = 3 gives leaf0 + (leaf1 + leaf2)).  A CTA owns one aligned block
// of S = b * 2^s leaves (a subtree) and a tile of weight rows.  Per row:
//   * 8 lanes per leaf, each holding 8 contiguous K positions of x for all
//     tokens in registers (loaded once), multiply with the row's 16 bytes and
//     sum in ascending order (fused multiply-add from +0) -> group sums s_g;
//   * an 8-lane transpose-reduce (xor 1, 2, 4) forms
//     ((s0+s1)+(s2+s3))+((s4+s5)+(s6+s7)) while spreading tokens over lanes;
//   * after a batch of rows, each (row, token) block subtree root is formed
//     from the S leaves in shared memory and written (BF16) to a partial plane.
// The weight rows stream through a 3-stage ring of 1-D bulk (TMA) copies
// completing on mbarriers.  The last CTA of a row tile to finish (an atomic
// ticket; nothing waits on another CTA) applies the top of the tree over the
// block roots and the epilogue: a plain BF16 store, or for the gate/up pair
// the fused stage boundary h = bf16(bf16(SiLU(gate)) * up).
#include <mutex>

#include "common.cuh"
#include "decode.h"
#include "ptx.cuh"

namespace detffn {
namespace {

constexpr int kStages = 3;

template <int S> struct Geo {
  static constexpr int B = (S % 3 == 0) ? 3 : 1;  // bottom subtree size
  static constexpr int P = S / B;                 // bottom subtrees per block (power of 2)
  static constexpr int RB = (S <= 8) ? 4 : 2;     // rows per batch
  static constexpr int ROWB = S * 128;            // bytes of one row's block slice
  static constexpr int STAGEB = RB * ROWB;
  static constexpr int LVB = RB * 8 * (S + 1) * 4;
  static constexpr int SMEM = kStages * STAGEB + LVB + kStages * 8 + 16;
  static constexpr int THREADS = 8 * S;
};

// The 8-lane transpose-reduce.  Lane l (l = lane & 7) enters with its group
// sums s[j] for MT tokens held in the lane-dependent order j = token ^ (l % MT)
// and leaves with the leaf of token l % MT.  At the step with lane distance d
// (1, 2, 4) a lane keeps the tokens whose bit log2(d) equals its own, adds
// the partner's partial for the same token, and hands over the others; the
// permuted order makes "keep" and "send" fixed registers.  The pairs formed
// are ((s0+s1)+(s2+s3))+((s4+s5)+(s6+s7)) over the 8 lanes' group sums.
template <int MT>
__device__ __forceinline__ float reduce_leaf(const float (&s)[MT]) {
  constexpr int N1 = MT > 1 ? MT / 2 : 1;
  constexpr int N2 = N1 > 1 ? N1 / 2 : 1;
  float a[N1], b[N2];
  if constexpr (MT >= 2) {
#pragma unroll
    for (int j = 0; j < N1; ++j) a[j] = __fadd_rn(s[2 * j], __shfl_xor_sync(0xffffffffu, s[2 * j + 1], 1));
  } else {
    a[0] = __fadd_rn(s[0], __shfl_xor_sync(0xffffffffu, s[0], 1));
  }
  if constexpr (N1 >= 2) {
#pragma unroll
    for (int j = 0; j < N2; ++j) b[j] = __fadd_rn(a[2 * j], __shfl_xor_sync(0xffffffffu, a[2 * j + 1], 2));
  } else {
    b[0] = __fadd_rn(a[0], __shfl_xor_sync(0xffffffffu, a[0], 2));
  }
  if constexpr (N2 >= 2) {
    return __fadd_rn(b[0], __shfl_xor_sync(0xffffffffu, b[1], 4));
  } else {
    return __fadd_rn(b[0], __shfl_xor_sync(0xffffffffu, b[0], 4));
  }
}

// Root of the block subtree over S leaves (FP32 leaves -> BF16 node).
template <int S>
__device__ __forceinline__ float block_root(const float* lv) {
  constexpr int B = Geo<S>::B, P = Geo<S>::P;
  float v[P];
#pragma unroll
  for (int q = 0; q < P; ++q)
    v[q] = (B == 1) ? lv[q] : node(lv[3 * q], node(lv[3 * q + 1], lv[3 * q + 2]));
#pragma unroll
  for (int w = P; w > 1; w >>= 1)
#pragma unroll
    for (int q = 0; q < w / 2; ++q) v[q] = node(v[2 * q], v[2 * q + 1]);
  return v[0];
}

__device__ __forceinline__ void unpack8(const uint4 q, float (&w)[8]) {
  const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    w[2 * i] = __uint_as_float(u[i] << 16);
    w[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

// Top of the tree over the NB block roots of each (token, row) of a tile, and
// the epilogue.  Loads for CH items are issued before any of them is used.
template <int NB>
__device__ __forceinline__ float top_tree(const uint16_t (&v)[NB]) {
  float f[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) f[b] = bf2f(v[b]);
#pragma unroll
  for (int w = NB; w > 1; w >>= 1)
#pragma unroll
    for (int c = 0; c < w / 2; ++c) f[c] = node(f[2 * c], f[2 * c + 1]);
  return f[0];
}

template <int NB, int MT>
__device__ void fixup(const DecArgs& a, int tile, int nthreads) {
  constexpr int CH = 2;
  const bool gate_up = a.w1 != nullptr;
  const long long N = a.N;
  const long long rows_total = gate_up ? 2 * N : N;
  const long long r0 = (long long)tile * a.RT;
  const int rt_valid = (int)((N - r0) < a.RT ? (N - r0) : a.RT);
  const int items = a.M * rt_valid;
  for (int base = threadIdx.x; base < items; base += nthreads * CH) {
    uint16_t gv[CH][NB], uv[CH][NB];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int i = base + c * nthreads;
      if (i >= items) continue;
      const int t = i / rt_valid;
      const long long row = r0 + i % rt_valid;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const long long o = ((long long)b * MT + t) * rows_total + row;
        gv[c][b] = __ldcg(&a.part[o]);
        if (gate_up) uv[c][b] = __ldcg(&a.part[o + N]);
      }
    }
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int i = base + c * nthreads;
      if (i >= items) continue;
      const int t = i / rt_valid;
      const long long row = r0 + i % rt_valid;
      const uint16_t y = f2bf(top_tree<NB>(gv[c]));
      if (!gate_up) {
        a.out[t * a.ldo + row] = y;
        continue;
      }
      const uint16_t ub = f2bf(top_tree<NB>(uv[c]));
      a.out[t * a.ldo + row] = f2bf(__fmul_rn(bf2f(__ldg(a.silu + y)), bf2f(ub)));
      if (a.gsave) a.gsave[t * a.ldo + row] = y;
      if (a.usave) a.usave[t * a.ldo + row] = ub;
    }
  }
}

template <int MT, int S>
__global__ void __launch_bounds__(Geo<S>::THREADS) k_decode(DecArgs a) {
  using G = Geo<S>;
  constexpr int RB = G::RB, ROWB = G::ROWB, STAGEB = G::STAGEB, NT = G::THREADS;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* stage = smem;
  float* lv = reinterpret_cast<float*>(smem + kStages * STAGEB);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * STAGEB + G::LVB);
  int* last = reinterpret_cast<int*>(full + kStages);

  const int tid = threadIdx.x, g = tid >> 3, l = tid & 7;
  const int blk = blockIdx.x, tile = blockIdx.y;
  const long long k0 = (long long)blk * S * 64;
  const bool gate_up = a.w1 != nullptr;
  const long long N = a.N;
  const long long rows_total = gate_up ? 2 * N : N;
  const long long r0 = (long long)tile * a.RT;
  const int rt_valid = (int)((N - r0) < a.RT ? (N - r0) : a.RT);
  const int slots = gate_up ? 2 * a.RT : a.RT;
  const int nbatch = (slots + RB - 1) / RB;

  // Row slot -> weight row pointer (at this block's K start) and partial index.
  auto slot_row = [&](int sl, const uint16_t*& wrow, long long& pidx) -> bool {
    int m = 0, r = sl;
    if (gate_up && sl >= a.RT) { m = 1; r = sl - a.RT; }
    if (r >= rt_valid) return false;
    const long long i = r0 + r;
    wrow = (m ? a.w1 : a.w0) + i * a.ldw + k0;
    pidx = m ? N + i : i;
    return true;
  };
  auto issue = [&](int q) {  // one thread
    const int s = q % kStages;
    uint32_t bytes = 0;
    const uint16_t* wr;
    long long pi;
    for (int r = 0; r < RB; ++r)
      if (slot_row(q * RB + r, wr, pi)) bytes += ROWB;
    mbar_arrive_expect_tx(&full[s], bytes);
    for (int r = 0; r < RB; ++r)
      if (slot_row(q * RB + r, wr, pi)) bulk_g2s(stage + s * STAGEB + r * ROWB, wr, ROWB, &full[s]);
  };

  // A wait of an earlier launch ran out (the status word is set until the
  // caller reads it): its outputs, which may be this launch's inputs (h, the
  // tickets), are unfinished, so this launch does nothing.
  if (__syncthreads_or(a.status != nullptr && *(volatile int*)a.status != 0)) return;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  int issued = 0;  // batches whose copies thread 0 has issued
  if (tid == 0 && !a.stall)
    for (; issued < kStages && issued < nbatch; ++issued) issue(issued);

  // This lane's x slice: 8 contiguous K positions for every token, then
  // permuted so that slot j holds token j ^ (l % MT) (the order reduce_leaf
  // expects): one conditional swap per bit of l, once per CTA.
  float xr[MT][8];
  const long long kk = k0 + g * 64 + l * 8;
#pragma unroll
  for (int t = 0; t < MT; ++t) {
    if (t < a.M) {
      const uint4 q = *reinterpret_cast<const uint4*>(a.x + t * a.ldx + kk);
      unpack8(q, xr[t]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) xr[t][e] = 0.0f;
    }
  }
#pragma unroll
  for (int bit = 1; bit < MT; bit <<= 1) {
    const bool sw = (l & bit) != 0;
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      if (j & bit) continue;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float u = xr[j][e], v = xr[j | bit][e];
        xr[j][e] = sw ? v : u;
        xr[j | bit][e] = sw ? u : v;
      }
    }
  }

  const long long limit = a.spin_limit > 0 ? a.spin_limit : kDefaultSpin;
  int q = 0;
  for (; q < nbatch; ++q) {
    const int s = q % kStages;
    const bool ok = mbar_wait(&full[s], (uint32_t)((q / kStages) & 1), limit, a.status);
    if (__syncthreads_or(!ok)) break;
    const unsigned char* st = stage + s * STAGEB;
#pragma unroll 2
    for (int r = 0; r < RB; ++r) {
      float w[8];
      unpack8(*reinterpret_cast<const uint4*>(st + r * ROWB + g * 128 + l * 16), w);
      float sacc[MT];  // group sums in the permuted token order
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        float acc = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = __fmaf_rn(xr[j][e], w[e], acc);
        sacc[j] = acc;
      }
      const float leaf = reduce_leaf<MT>(sacc);
      if (l < MT) lv[(r * 8 + l) * (S + 1) + g] = leaf;
    }
    __syncthreads();
    if (tid == 0 && q + kStages < nbatch) {
      issue(q + kStages);
      issued = q + kStages + 1;
    }
    for (int i = tid; i < MT * RB; i += NT) {
      const int t = i / RB, r = i % RB;
      const uint16_t* wr;
      long long pidx;
      if (t < a.M && slot_row(q * RB + r, wr, pidx))
        a.part[((long long)blk * MT + t) * rows_total + pidx] = f2bf(block_root<S>(&lv[(r * 8 + t) * (S + 1)]));
    }
    __syncthreads();
  }
  if (q < nbatch) {
    // A wait ran out: drain the copies this CTA issued (on the long bound,
    // whatever the call's poll limit: it exits with no copy in flight), and
    // leave the tile unfinished.
    if (tid == 0)
      for (int p = q; p < issued; ++p)
        mbar_wait(&full[p % kStages], (uint32_t)((p / kStages) & 1), kDefaultSpin, nullptr);
    __syncthreads();
    return;
  }

  // Ticket: the last block of this row tile applies the top of the tree.
  __threadfence();
  __syncthreads();
  if (tid == 0) *last = (atomicAdd(&a.cnt[tile], 1u) == gridDim.x - 1);
  __syncthreads();
  if (!*last) return;
  __threadfence();
  switch (gridDim.x) {
    case 1: fixup<1, MT>(a, tile, NT); break;
    case 2: fixup<2, MT>(a, tile, NT); break;
    case 4: fixup<4, MT>(a, tile, NT); break;
    case 8: fixup<8, MT>(a, tile, NT); break;
    default: break;
  }
  if (tid == 0) a.cnt[tile] = 0u;
}

template <int MT, int S>
cudaError_t launch_ms(DecArgs a, int NB, int sm_count, cudaStream_t st) {
  using G = Geo<S>;
  // Resident CTAs per SM for this instance (registers, threads, smem), worked
  // out once; concurrent first calls (several host threads, the handle path
  // and the allocation-free entry point) all wait for the one set-up.
  static std::once_flag once;
  static cudaError_t setup_err = cudaSuccess;
  static int per_sm = 0;
  std::call_once(once, [] {
    setup_err = cudaFuncSetAttribute(k_decode<MT, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
    if (setup_err == cudaSuccess)
      setup_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode<MT, S>, G::THREADS, G::SMEM);
    if (per_sm < 1) per_sm = 1;
  });
  if (setup_err != cudaSuccess) return setup_err;
  // Rows per tile so that the grid is one wave of resident CTAs.
  long long tiles = ((long long)sm_count * per_sm) / NB;
  if (tiles < 1) tiles = 1;
  long long rt = (a.N + tiles - 1) / tiles;
  if (rt < 1) rt = 1;
  a.RT = (int)rt;
  tiles = (a.N + rt - 1) / rt;
  if (tiles > 65535) return cudaErrorInvalidValue;
  k_decode<MT, S><<<dim3((unsigned)NB, (unsigned)tiles), G::THREADS, G::SMEM, st>>>(a);
  return cudaGetLastError();
}

template <int S>
cudaError_t launch_s(const DecArgs& a, int NB, int sm_count, cudaStream_t st) {
  if (a.M <= 1) return launch_ms<1, S>(a, NB, sm_count, st);
  if (a.M <= 2) return launch_ms<2, S>(a, NB, sm_count, st);
  if (a.M <= 4) return launch_ms<4, S>(a, NB, sm_count, st);
  return launch_ms<8, S>(a, NB, sm_count, st);
}

}  // namespace

bool decode_geometry(long long K, int* S, int* NB) {
  if (K <= 0 || K % 64 != 0) return false;
  long long L = K / 64;
  int d = 0;
  while ((L & 1) == 0) { L >>= 1; ++d; }
  const long long b = L;  // odd part
  if (b != 1 && b != 3) return false;
  const int s = d < 3 ? d : 3;
  const int Sv = (int)(b << s);
  if (Sv % 4 != 0) return false;
  const long long nb = (K / 64) / Sv;
  if (nb > 8) return false;
  *S = Sv;
  *NB = (int)nb;
  return true;
}

size_t decode_part_elems(long long K, long long rows_total) {
  int S, NB;
  if (!decode_geometry(K, &S, &NB)) return 0;
  return (size_t)NB * 8 * (size_t)rows_total;
}

cudaError_t launch_decode_exact(DecArgs a, int sm_count, cudaStream_t st) {
  int S, NB;
  if (a.M < 1 || a.M > 8 || !decode_geometry(a.K, &S, &NB)) return cudaErrorInvalidValue;
  switch (S) {
    case 4: return launch_s<4>(a, NB, sm_count, st);
    case 8: return launch_s<8>(a, NB, sm_count, st);
    case 12: return launch_s<12>(a, NB, sm_count, st);
    case 24: return launch_s<24>(a, NB, sm_count, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace detffn
