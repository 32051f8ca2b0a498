// k_tc.cu -- tensor-core (tcgen05 / TMEM) tree contraction.
//
// out[r, c] = T_K(A[r, :], B[c, :]) for K-major BF16 A [R, K] and B [C, K],
// with the canonical FP32-leaf / BF16-node midpoint tree (RL-Kernel PR #325,
// "Design").  Each 64-wide leaf is one FP32 accumulation on the tensor core
// (4 MMAs of K = 16 into a fresh TMEM buffer; the hardware's in-leaf order),
// and the tree over the leaves is applied exactly by the epilogue warps.
//
// Tree shape.  The kernel covers L = 1, 2^d and 3 * 2^d leaves: the midpoint
// tree is then a perfect binary tree over Q = 2^E bottom groups of G leaves
// (G = 2: leaf pairs; G = 3: leaf0 + (leaf1 + leaf2); G = 1: a lone leaf).
//
// Used for many tokens (more than 32; fewer go to k_tcs.cu, which splits K
// evenly over the SMs).
//
// Roles (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: A and B tiles of one leaf per pipeline stage
//               (128-byte swizzle, K- or MN-major), a ring of up to 512/BN
//               stages on mbarriers (as many as fit beside the shared-memory
//               stack levels); a stage is reused once the leaf read from it
//               has been committed;
//   warps 1-3   MMA issuers (warp 1 also allocates TMEM: 512/BN leaf buffers
//               of BN columns); leaves are dealt round-robin over them, one
//               leaf per buffer, with one commit per leaf (the buffer's
//               "full" barrier, which the producer reads too);
//   warps 4-11  epilogue: each thread owns one row (TMEM lane) and BN/2
//               columns; it reads a group's leaves from TMEM, forms the
//               group roots, returns the buffers at once, and then folds the
//               roots into a binary-counter stack of BF16 nodes (low levels
//               in registers, high levels in shared memory); the last fold
//               is the output.
// Registers: warps 0-3 hand most of their share to the epilogue's two
// warpgroups (setmaxnreg), which hold a group's leaves in 32-column chunks.
// Every wait is bounded; on a timeout the CTA records DETFFN_ERR_TIMEOUT,
// stops, drains its own copies and MMAs (bounded) and frees its TMEM.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "tc.h"

namespace detffn {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kMaxAccBufs = 16;  // TMEM leaf buffers: 512 columns / BN (at most 16)
constexpr int kEpiWarp0 = 4;  // warps 0-3: TMA producers and MMA issuers, warps 4..11: epilogue
// Roles of warps 0-3.  Each leaf costs the threads that load it and issue
// its MMAs a few dependent barrier operations of a hundred-odd cycles of
// latency each, more than the 4 MMAs of a 128 x 128 leaf keep the tensor
// pipe busy, so the work is spread over several warps.  Every barrier is
// waited on by parity, which is only sound while no waiter can fall two
// phases behind; the two layouts below keep that true by construction:
//   paired (bottom groups of two leaves): leaves 4k, 4k+1 go to issuer 0
//     (warp 1) and leaves 4k+2, 4k+3 to issuer 1 (warp 2), one group at a
//     time, so that each TMEM buffer -- and with four stages each stage --
//     has one issuer; with an even number of stages the loads are split by
//     leaf parity between warp 0 and warp 3, each owning its stages (with
//     an odd number, warp 0 loads every leaf and warp 3 idles);
//   single (groups of one or three leaves): warp 0 loads every leaf, and
//   issuer q (warp 1 + q) takes leaves q, q + 3, ...
template <int GG> struct Roles {
  static constexpr bool PAIRED = GG == 2;
  static constexpr int ISSUERS = PAIRED ? 2 : 3;
  static constexpr int UNIT = PAIRED ? 2 : 1;  // consecutive leaves an issuer takes at a time
};
// Registers per thread: at launch (384 threads), and after the split between
// warpgroup 0 (producer and issuers) and the epilogue's two warpgroups.  The
// split hands over exactly what the launch holds; the host refuses to launch
// a build whose register count differs.
constexpr int kRegsLaunch = 168, kRegsLow = 56, kRegsHigh = 224;
static_assert(128 * kRegsLow + 256 * kRegsHigh == 384 * kRegsLaunch, "register split");
constexpr int kMaxLv = 6;  // up to Q = 64 bottom groups
constexpr int kLayRuntime = 4;  // operand layouts read at run time (leaf-dump instances)

// One CTA per SM, 8 epilogue warps (two per TMEM lane quarter, BN/2 columns
// each), 512/BN leaf buffers.
template <int BN> struct TcGeo {
  static constexpr int EPI_WARPS = 8;
  static constexpr int HALVES = EPI_WARPS / 4;            // epilogue warps per lane quarter
  static constexpr int THREADS = 32 * (kEpiWarp0 + EPI_WARPS);
  static_assert(THREADS == 384, "register split assumes 384 threads");
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int COLS = BN / HALVES;  // columns per epilogue thread
  static constexpr int WORDS = COLS / 2;    // packed BF16 pairs per stack level per thread
  static constexpr int REG_LV = 3;                        // stack levels kept in registers
  static constexpr int LV_BYTES = BM * BN * 2;            // one shared-memory stack level
  static constexpr int BAR_BYTES = 512;
  // Output staging for one-leaf trees (G = 1: the weight gradients over few
  // tokens, whose epilogue is nothing but stores; longer trees need the shared
  // memory for stack levels and stages): per epilogue warp two buffers of 32
  // rows x COLS columns in the 128-byte-swizzled layout of a TMA store box.
  static constexpr int STG_BUF = 32 * COLS * 2;  // bytes of one buffer (4 KB)
  static constexpr int STG_BYTES = EPI_WARPS * 2 * STG_BUF;
  static_assert(COLS * 2 == 128, "one 128-byte swizzle span per staged row");
  static __host__ __device__ int stg_for(int G) { return G == 1 ? STG_BYTES : 0; }
  static constexpr int MAX_SMEM = 227 * 1024;
  static constexpr int MAX_STAGES = 12;
  static constexpr int NBUF = (512 / BN) < kMaxAccBufs ? (512 / BN) : kMaxAccBufs;
  static constexpr int TMEM_COLS = NBUF * BN;
  // Stages that fit beside the shared-memory stack levels a tree of E levels needs.
  static __host__ __device__ int stages_for(int G, int E) {
    const int lv = E > REG_LV ? E - REG_LV : 0;
    int n = (MAX_SMEM - 1024 - BAR_BYTES - stg_for(G) - lv * LV_BYTES) / STAGE;
    return n > MAX_STAGES ? MAX_STAGES : n;
  }
  static __host__ __device__ int smem_for(int G, int E, int nstage) {
    const int lv = E > REG_LV ? E - REG_LV : 0;
    return 1024 + nstage * STAGE + lv * LV_BYTES + stg_for(G) + BAR_BYTES;
  }
};


// Tree node on packed pairs of BF16 nodes: rne_bf16(fp32(a) + fp32(b)) per
// half, which is the correctly rounded BF16 sum, i.e. add.rn.bf16x2 (checked
// on every one of the 2^32 operand pairs by detffn_selfcheck_node_add).
__device__ __forceinline__ uint32_t node2(uint32_t a, uint32_t b) { return add_bf16x2(a, b); }

struct Bars {  // must fit in TcGeo::BAR_BYTES
  uint64_t full[12], accf[kMaxAccBufs], acce[kMaxAccBufs], fin;  // up to 12 stages
  uint32_t tmem_slot;
  int abort;
};

// Bounded wait that also gives up when another role has aborted.
static_assert(sizeof(Bars) <= 512, "barrier block");

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, long long limit,
                                              volatile int* abort_flag, int* status) {
  for (long long i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 1023) == 1023 && *abort_flag) return false;
  }
  *abort_flag = 1;
  if (status) atomicExch(status, (int)DETFFN_ERR_TIMEOUT);
  return false;
}

}  // namespace
}  // namespace detffn

namespace detffn {
namespace {

struct TcArgs {
  int R, C;
  int L, G, E;      // leaves, bottom group size, levels above the groups
  int nstage;
  int num_m, num_n;
  int gm;           // tile order: blocks of gm row tiles, row tile fastest within a block
  int np;           // problems in this launch (1 or 2; the second uses tmA2/tmB2 and out2)
  int b_mn;         // B stored [K][C] (C contiguous): MN-major B tiles (BN = 128 only)
  int o_tma;        // row-major outputs may leave through TMA stores (maps tmO, tmO2)
  int a_mn;         // A stored [K][R] (R contiguous): MN-major A tiles
  uint16_t* out;
  uint16_t* out2;
  long long ld_r, ld_c;
  int* status;
  long long spin;
  int stall;        // test only: the producer issues no loads
  float* dump;      // leaf dump (DUMP instances): [np][R][C][L] FP32 leaves
  int kc_op;        // K axis in chunks (0: no; 1: operand A, 2: operand B), read through the chunk maps
  int kc_n;
  int kc_leaf[kMaxKChunks];  // first leaf of chunk c
};

// The tensor maps of a chunked operand, one per chunk.
struct KChunkMaps {
  CUtensorMap m[kMaxKChunks];
};

// Output tile of unit index t.  The tiles are taken in blocks of gm row
// tiles, row tile fastest within a block: the CTAs at work at one time then
// share a block of A rows (kept in L2 while the block sweeps the columns)
// and a few column tiles of B, so that neither operand is re-read from DRAM
// once per wave of tiles when A is larger than L2 can keep.
__device__ __forceinline__ void tile_of(int t, const TcArgs& a, int& tm, int& tn) {
  const int per = a.gm * a.num_n;
  const int mb = t / per, idx = t - mb * per;
  const int rows = min(a.gm, a.num_m - mb * a.gm);
  tm = mb * a.gm + idx % rows;
  tn = idx / rows;
}

// Writes the COLS columns of one row held as packed BF16 pairs: element i goes
// to base[row_off + (c0 + i) * ld_c] for c0 + i < C.
template <int WORDS>
__device__ __forceinline__ void store_cols(uint16_t* base, long long row_off, long long c0, long long ld_c,
                                           long long C, const uint32_t (&root)[WORDS]) {
  uint16_t* o = base + row_off + c0 * ld_c;
  if (ld_c == 1 && c0 + 2 * WORDS <= C && ((uintptr_t)o & 15u) == 0) {
#pragma unroll
    for (int v = 0; v < WORDS / 4; ++v)
      reinterpret_cast<uint4*>(o)[v] = make_uint4(root[4 * v], root[4 * v + 1], root[4 * v + 2], root[4 * v + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < 2 * WORDS; ++i)
      if (c0 + i < C) o[i * ld_c] = (uint16_t)(root[i >> 1] >> (16 * (i & 1)));
  }
}

// Stack level m >= REG_LV lives in shared memory as [level][epilogue
// warp][word][lane]: each warp's share of a level is its own 4 KB block
// (1024-byte aligned), which at the end of a tile doubles as the staging
// buffer of the warp's TMA output store.
template <int BN>
__device__ __forceinline__ uint32_t* stk_at(uint32_t* stk, int m, int ew, int w, int lane) {
  using T = TcGeo<BN>;
  return stk + (((m - T::REG_LV) * T::EPI_WARPS + ew) * T::WORDS + w) * 32 + lane;
}

// The epilogue's view of one CTA's pipeline.
struct EpiCtx {
  uint32_t tmem, lane_addr;
  int col0, lane;
  Bars* bars;
  long long limit;
  volatile int* abort_flag;
  uint32_t lc;  // leaves consumed (NBUF is a power of two)
  bool ok;
};

// Bottom group qg of tile (pb, tm, tn), whose leaves are the next GG in
// TMEM: wait for the commits of its leaves (of the second alone in the
// paired layout, where one issuer committed both), read them in column
// chunks, hand this thread's group root words to emit(w, word) as they are
// formed, and return the buffers to the MMA issuers.  False when a wait ran
// out.
template <int BN, int GG, bool DUMP, class Emit>
__device__ __forceinline__ bool group_root(EpiCtx& e, const TcArgs& a, Emit&& emit, int pb, long long r, int tn,
                                         int qg) {
  using T = TcGeo<BN>;
  if constexpr (GG == 2) {  // one issuer committed both leaves, the second last
    const uint32_t last = e.lc + 1;
    if (!wait_or_abort(&e.bars->accf[last % T::NBUF], (last / T::NBUF) & 1u, e.limit, e.abort_flag, a.status))
      e.ok = false;
  } else {
    // (Three-leaf groups: the first two slots here, the third further down.)
    for (int g = 0; g < (GG == 3 ? 2 : GG); ++g)
      if (!wait_or_abort(&e.bars->accf[(e.lc + g) % T::NBUF], ((e.lc + g) / T::NBUF) & 1u, e.limit, e.abort_flag,
                         a.status))
        e.ok = false;
  }
  if (__any_sync(0xffffffffu, !e.ok)) {
    e.ok = false;
    return false;
  }
  tc_fence_after();
  const uint32_t b0 = (uint32_t)((e.lc % T::NBUF) * BN), b1 = (uint32_t)(((e.lc + 1) % T::NBUF) * BN),
                 b2 = (uint32_t)(((e.lc + 2) % T::NBUF) * BN);
  constexpr int CW = 32;     // columns per chunk
  constexpr int WC = CW / 2;  // packed words per chunk
  if constexpr (GG == 1) {
    // A lone leaf (one-leaf trees: weight gradients over few tokens):
    // all columns read with one wait, each rounded once.
    static_assert(T::COLS % 32 == 0, "columns per thread");
#pragma unroll
    for (int c = 0; c < T::COLS / 32; c += 2) {
      uint32_t va[32], vb[32];
      tmem_ld32(e.tmem + e.lane_addr + b0 + (uint32_t)(e.col0 + 32 * c), va);
      if (c + 1 < T::COLS / 32) tmem_ld32(e.tmem + e.lane_addr + b0 + (uint32_t)(e.col0 + 32 * c + 32), vb);
      tmem_wait_ld();
      if constexpr (DUMP) {
        float* d = a.dump + (size_t)pb * a.R * a.C * a.L;
        const long long cc = (long long)tn * BN + e.col0 + 32 * c;
        dump_leaves(d, r, cc, a.R, a.C, a.L, qg, va);
        if (c + 1 < T::COLS / 32) dump_leaves(d, r, cc + 32, a.R, a.C, a.L, qg, vb);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) emit(16 * c + i, pack_bf16x2(__uint_as_float(va[2 * i]), __uint_as_float(va[2 * i + 1])));
      if (c + 1 < T::COLS / 32)
#pragma unroll
        for (int i = 0; i < 16; ++i)
          emit(16 * c + 16 + i, pack_bf16x2(__uint_as_float(vb[2 * i]), __uint_as_float(vb[2 * i + 1])));
    }
  } else if constexpr (GG == 2) {
#pragma unroll
    for (int c = 0; c < T::COLS / CW; ++c) {
      uint32_t v0[CW], v1[CW];
      const uint32_t col = (uint32_t)(e.col0 + CW * c);
      tmem_ld32(e.tmem + e.lane_addr + b0 + col, v0);
      tmem_ld32(e.tmem + e.lane_addr + b1 + col, v1);
      tmem_wait_ld();
      if constexpr (DUMP) {
        float* d = a.dump + (size_t)pb * a.R * a.C * a.L;
        const long long cc = (long long)tn * BN + col;
        dump_leaves(d, r, cc, a.R, a.C, a.L, qg * GG, v0);
        dump_leaves(d, r, cc, a.R, a.C, a.L, qg * GG + 1, v1);
      }
#pragma unroll
      for (int i = 0; i < WC; ++i)  // pairs of adjacent columns, added two at a time (add.rn.f32x2)
        emit(c * WC + i, pack_bf16x2_of(add_f32x2(f32x2(v0[2 * i], v0[2 * i + 1]), f32x2(v1[2 * i], v1[2 * i + 1]))));
    }
  } else {
    // Three leaves, loaded and issued in the order leaf 1, leaf 2, leaf 0
    // (slots 0, 1, 2): the node over leaves 1 and 2 is formed first and their
    // two buffers go back to the issuers before leaf 0 is read, so that the
    // next group's first two leaves can start while this one finishes.
    constexpr int CH = 16;  // columns per chunk in the first pass
    uint32_t n12[T::WORDS];
#pragma unroll
    for (int c = 0; c < T::COLS / CH; ++c) {
      uint32_t v1[CH], v2[CH];
      const uint32_t col = (uint32_t)(e.col0 + CH * c);
      tmem_ld16(e.tmem + e.lane_addr + b0 + col, v1);
      tmem_ld16(e.tmem + e.lane_addr + b1 + col, v2);
      tmem_wait_ld();
      if constexpr (DUMP) {
        float* d = a.dump + (size_t)pb * a.R * a.C * a.L;
        const long long cc = (long long)tn * BN + col;
        dump_leaves(d, r, cc, a.R, a.C, a.L, qg * GG + 1, v1);
        dump_leaves(d, r, cc, a.R, a.C, a.L, qg * GG + 2, v2);
      }
#pragma unroll
      for (int i = 0; i < CH / 2; ++i)
        n12[c * (CH / 2) + i] = pack_bf16x2_of(add_f32x2(f32x2(v1[2 * i], v1[2 * i + 1]), f32x2(v2[2 * i], v2[2 * i + 1])));
    }
    tc_fence_before();
    __syncwarp();
    if (e.lane == 0) {
      mbar_arrive(&e.bars->acce[e.lc % T::NBUF]);
      mbar_arrive(&e.bars->acce[(e.lc + 1) % T::NBUF]);
    }
    const uint32_t l0 = e.lc + 2;
    if (!wait_or_abort(&e.bars->accf[l0 % T::NBUF], (l0 / T::NBUF) & 1u, e.limit, e.abort_flag, a.status))
      e.ok = false;
    if (__any_sync(0xffffffffu, !e.ok)) {
      e.ok = false;
      return false;
    }
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < T::COLS / CH; ++c) {  // (chunks of 16 columns: the caller's nodes are live here)
      uint32_t v0[CH];
      const uint32_t col = (uint32_t)(e.col0 + CH * c);
      tmem_ld16(e.tmem + e.lane_addr + b2 + col, v0);
      tmem_wait_ld();
      if constexpr (DUMP) {
        float* d = a.dump + (size_t)pb * a.R * a.C * a.L;
        dump_leaves(d, r, (long long)tn * BN + col, a.R, a.C, a.L, qg * GG, v0);
      }
#pragma unroll
      for (int i = 0; i < CH / 2; ++i) {
        const uint32_t nn = n12[c * (CH / 2) + i];
        emit(c * (CH / 2) + i,
             pack_bf16x2_of(add_f32x2(f32x2(v0[2 * i], v0[2 * i + 1]), f32x2(nn << 16, nn & 0xFFFF0000u))));
      }
    }
  }
  // The leaves are in registers: return the TMEM buffers.
  tc_fence_before();
  __syncwarp();
  if (e.lane == 0)
    for (int g = (GG == 3 ? 2 : 0); g < GG; ++g) mbar_arrive(&e.bars->acce[(e.lc + g) % T::NBUF]);
  e.lc += GG;
  return true;
}

template <int BN, int GG, bool DUMP, bool KC, int LAY>
__global__ void __launch_bounds__(TcGeo<BN>::THREADS, 1)
    k_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
         const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
         const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmO2, const TcArgs a,
         const __grid_constant__ KChunkMaps kcm) {
  using T = TcGeo<BN>;
  // Operand layouts: fixed by the instance (LAY = a_mn + 2 b_mn) except in
  // the leaf-dump instances (LAY = kLayRuntime), which read them from a.
  const bool amn = LAY == kLayRuntime ? a.a_mn != 0 : (LAY & 1) != 0;
  const bool bmn = LAY == kLayRuntime ? a.b_mn != 0 : (LAY & 2) != 0;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int NS = a.nstage;
  const int slv = a.E > T::REG_LV ? a.E - T::REG_LV : 0;
  unsigned char* stages = smem;
  uint32_t* stk = reinterpret_cast<uint32_t*>(smem + NS * T::STAGE);
  unsigned char* stg_all = smem + NS * T::STAGE + slv * T::LV_BYTES;  // 1024-byte aligned
  Bars* bars = reinterpret_cast<Bars*>(smem + NS * T::STAGE + slv * T::LV_BYTES + T::stg_for(GG));
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = a.num_m * a.num_n;
  const int units = tiles * a.np;  // unit u: problem u % np, then tile
  const long long limit = a.spin > 0 ? a.spin : kDefaultSpin;
  // A wait of an earlier launch ran out (the status word is set until the
  // caller reads it): its outputs, which may be this launch's inputs, are
  // unfinished, so this launch does nothing.
  // Programmatic dependent launch: the previous kernel on the stream (whose
  // outputs may be this one's inputs, or whose inputs this one may
  // overwrite) has completed past this wait; the next may begin launching
  // (its CTAs cannot share an SM with this kernel's, and wait in turn).
  grid_dep_launch();
  grid_dep_wait();
  if (__syncthreads_or(a.status != nullptr && *(volatile int*)a.status != 0)) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->full[s], 1);
    }
    for (int b = 0; b < T::NBUF; ++b) {
      mbar_init(&bars->accf[b], 1);
      mbar_init(&bars->acce[b], T::EPI_WARPS);
    }
    mbar_init(&bars->fin, Roles<GG>::ISSUERS);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (a.np > 1) {
      prefetch_tmap(&tmA2);
      prefetch_tmap(&tmB2);
    }
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, T::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;

  using RL = Roles<GG>;
  const int nprod = (RL::PAIRED && NS % 2 == 0) ? 2 : 1;
  if (warp < kEpiWarp0) {
    // Warpgroup 0 hands most of its registers to the epilogue's two
    // warpgroups (the register budget of each role is set in its own
    // branch, so that the compiler allocates each role's code for it).
    regs_dec<kRegsLow>();
    if (warp == 0 || (RL::PAIRED && warp == 3)) {
      // ---------------- TMA producers (converged warps; one lane issues) ----------------
      // Producer p loads the leaves it with it % nprod == p.  Stage it % NS is
      // free once the MMAs of leaf it - NS (the same producer's) have
      // completed, which the leaf's own "full accumulator" barrier reports
      // (NS <= NBUF, and leaf it - NS + NBUF is not loaded before leaf it, so
      // that barrier cannot have moved on by a second phase).
      const int p = warp == 0 ? 0 : 1;
      long long it = 0;
      Ring rs;  // stage of load it
      Ring rv;  // TMEM buffer of leaf it - NS
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok && p < nprod; u += gridDim.x) {
        const int pb = u % a.np, v = u / a.np;
        const int t = v;
        int tm, tn;
        tile_of(t, a, tm, tn);
        const CUtensorMap* mA = pb ? &tmA2 : &tmA;
        const CUtensorMap* mB = pb ? &tmB2 : &tmB;
        int j3 = 0;  // j % 3
        for (int j = 0; j < a.L; ++j, ++it, rs.next(NS), j3 = (j3 == 2 ? 0 : j3 + 1)) {
          const int s = rs.slot;
          const bool own = (int)(it & (nprod - 1)) == p;
          if (it >= NS) {
            if (own) {
              const bool w = wait_or_abort(&bars->accf[rv.slot], rv.phase, limit, abort_flag, a.status);
              if (!__all_sync(0xffffffffu, w)) {
                ok = false;
                break;
              }
            }
            rv.next(T::NBUF);
          }
          if (own && !a.stall && elect_one()) {
            unsigned char* st = stages + s * T::STAGE;
            mbar_arrive_expect_tx(&bars->full[s], (uint32_t)T::STAGE);
            // Three-leaf groups are loaded leaf 1, leaf 2, leaf 0 (see the
            // epilogue): slot j3 = j % 3 of a group holds leaf (j3 + 1) % 3.
            const int x = (GG == 3 ? (j3 == 2 ? j - 2 : j + 1) : j) * BK;
            // A chunked K axis: the leaf's chunk (a leaf never spans two) and
            // the K coordinate within it.
            const CUtensorMap* lA = mA;
            const CUtensorMap* lB = mB;
            int xa = x, xb = x;
            if constexpr (KC) {  // (a separate instance: the branch costs the producer loop a few %)
              int c = 0;
              while (c + 1 < a.kc_n && a.kc_leaf[c + 1] * BK <= x) ++c;
              const int xc = x - a.kc_leaf[c] * BK;
              if (a.kc_op == 1) {
                lA = &kcm.m[c];
                xa = xc;
              } else {
                lB = &kcm.m[c];
                xb = xc;
              }
            }
            if (amn) {  // two boxes of 64 (R) x 64 (K)
              tma_load_2d(st, lA, tm * BM, xa, &bars->full[s]);
              tma_load_2d(st + T::A_BYTES / 2, lA, tm * BM + BM / 2, xa, &bars->full[s]);
            } else {
              tma_load_2d(st, lA, xa, tm * BM, &bars->full[s]);
            }
            if (bmn) {  // two boxes of 64 (C) x 64 (K)
              tma_load_2d(st + T::A_BYTES, lB, tn * BN, xb, &bars->full[s]);
              tma_load_2d(st + T::A_BYTES + T::B_BYTES / 2, lB, tn * BN + BN / 2, xb, &bars->full[s]);
            } else {
              tma_load_2d(st + T::A_BYTES, lB, xb, tn * BN, &bars->full[s]);
            }
          }
          __syncwarp();
        }
      }
      // Drain: the last loads issued into each stage have landed (on the long
      // bound, whatever the call's poll limit: no CTA exits with copies in
      // flight).
      if (lane == 0 && !a.stall)
        for (long long i = (it > NS ? it - NS : 0); i < it; ++i)
          if ((int)(i & (nprod - 1)) == p) mbar_wait(&bars->full[i % NS], (uint32_t)((i / NS) & 1), kDefaultSpin, nullptr);
    } else if (warp >= 1 && warp <= RL::ISSUERS) {
      const int q = warp - 1;  // issuer index
      // ---------------- MMA issuers (converged warps; one lane each issues) ----------------
      // Leaf n uses stage n % NS and TMEM buffer n % NBUF, with one commit per
      // leaf (its "full accumulator" barrier, which the producer reads).
      // Issuer q takes UNIT consecutive leaves at a time (units q, q + ISSUERS,
      // ...).  In the paired layout a unit is a bottom group, so the commit of
      // its second leaf also covers its first (a commit tracks all of its
      // thread's earlier MMAs) and the epilogue waits once per group.  Leaves
      // are independent accumulations, so the issuers' MMAs may reach the
      // tensor pipe in any order.
      static_assert(T::NBUF >= 3, "a group of up to 3 leaves in flight");
      const uint32_t idesc = idesc_bf16(BM, BN) | (bmn ? kIdescTransB : 0u) | (amn ? kIdescTransA : 0u);
      const uint32_t bstep = bmn ? 128u : 2u;  // K = 16 step in descriptor units
      const uint32_t astep = amn ? 128u : 2u;
      const int mine = blockIdx.x < units ? (units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
      const long long nunit = (long long)mine * (a.L / RL::UNIT);
      Ring rs, rb;  // pipeline stage; TMEM leaf buffer
      rs.adv(q * RL::UNIT, NS);
      rb.adv(q * RL::UNIT, T::NBUF);
      bool ok = true;
      for (long long gi = q; gi < nunit && ok; gi += RL::ISSUERS) {
       for (int gl = 0; gl < RL::UNIT; ++gl) {
        const int s = rs.slot, b = rb.slot;
        // The buffer must have been returned by the epilogue.  In the paired
        // layout the epilogue returns a pair's two buffers in order (each
        // warp arrives on the first, then the second), so the second one's
        // return, awaited before the first leaf, covers both.
        bool w = true;
        if (!RL::PAIRED || gl == 0)
          w = wait_or_abort(&bars->acce[RL::PAIRED ? b + 1 : b], rb.phase ^ 1u, limit, abort_flag, a.status);
        w = w && wait_or_abort(&bars->full[s], rs.phase, limit, abort_flag, a.status);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = amn ? smem_desc_sw128_mn(stages + s * T::STAGE) : smem_desc_sw128(stages + s * T::STAGE);
        const uint64_t db = bmn ? smem_desc_sw128_mn(stages + s * T::STAGE + T::A_BYTES)
                                   : smem_desc_sw128(stages + s * T::STAGE + T::A_BYTES);
        if (elect_one()) {
  #pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)  // a fresh FP32 accumulation per leaf
            tc_mma_bf16(tmem + (uint32_t)(b * BN), da + astep * kk, db + bstep * kk, idesc, kk > 0 ? 1u : 0u);
          tc_commit(&bars->accf[b]);
        }
        __syncwarp();
        rs.next(NS);
        rb.next(T::NBUF);
       }
       rs.adv((RL::ISSUERS - 1) * RL::UNIT, NS);
       rb.adv((RL::ISSUERS - 1) * RL::UNIT, T::NBUF);
      }
      if (elect_one()) tc_commit(&bars->fin);  // arrives when every MMA issued above has completed
      __syncwarp();
      // Every issuer's MMAs have completed before TMEM is freed (long bound).
      if (q == 0 && lane == 0) mbar_wait(&bars->fin, 0, kDefaultSpin, nullptr);
    }
  } else {
    regs_inc<kRegsHigh>();
    // ---------------- epilogue: leaves -> tree ----------------
    const int ew = warp - kEpiWarp0;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int half = ew >> 2;
    const int row = quarter * 32 + lane;
    const int col0 = half * T::COLS;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int Q = 1 << a.E;
    EpiCtx e{tmem, lane_addr, col0, lane, bars, limit, abort_flag, 0u, true};
    int stg_n = 0;  // tiles staged for a TMA store
    bool& ok = e.ok;


    if constexpr (GG >= 2) {
      // Blocks of four bottom groups (or the one or two groups of a shorter
      // tree), whose level-0 and level-1 nodes stay in fixed registers, as
      // does the pending level-2 node (n2); the binary counter above them
      // (levels >= 3) lives in shared memory, which leaves a 64-group tree
      // room for four pipeline stages.
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int pb = u % a.np, t = u / a.np;
        int tm, tn;
        tile_of(t, a, tm, tn);
        uint16_t* const outp = pb ? a.out2 : a.out;
        const long long r = (long long)tm * BM + row;
        uint32_t n2[T::WORDS];  // the pending level-2 node (left child over four groups)
        for (int q = 0; q < Q && ok; q += 4) {
          uint32_t n0[T::WORDS], n1[T::WORDS], cur[T::WORDS];
          // Two copies of the group reader, for the even and the odd group of
          // each pair, in a loop over the block's pairs; each hands its root
          // words straight to the node they enter: the even one's root goes
          // to n0, the odd one forms the pair's node in cur, which becomes n1
          // (first pair) or is folded with n1 into the node over the block
          // (second pair).  (Two copies run faster than one copy with a
          // per-group branch and node copies, and than four copies, whose
          // code no longer stays in the instruction cache.)
#pragma unroll 1
          for (int k = 0; k < 4 && k < Q; k += 2) {
            if (!group_root<BN, GG, DUMP>(e, a, [&](int w, uint32_t g) { n0[w] = g; }, pb, r, tn, q + k)) break;
            if (Q == 1) {
#pragma unroll
              for (int w = 0; w < T::WORDS; ++w) cur[w] = n0[w];
              break;
            }
            if (!group_root<BN, GG, DUMP>(e, a, [&](int w, uint32_t g) { cur[w] = node2(n0[w], g); }, pb, r, tn,
                                          q + k + 1))
              break;
            if (k == 2) {
#pragma unroll
              for (int w = 0; w < T::WORDS; ++w) cur[w] = node2(n1[w], cur[w]);
            } else if (Q >= 4) {
#pragma unroll
              for (int w = 0; w < T::WORDS; ++w) n1[w] = cur[w];
            }
          }
          if (!ok) break;
          const int qq = q + (Q < 4 ? Q : 4) - 1;  // the last group of this block
          // The binary counter above the block: fold the pending level-2 node
          // and then the stored nodes of levels 3, 4, ... while the group
          // index has those bits.
          int l = 2;
          if (a.E > 2 && ((qq >> 2) & 1)) {
#pragma unroll
            for (int w = 0; w < T::WORDS; ++w) cur[w] = node2(n2[w], cur[w]);
            l = 3;
#pragma unroll 1
            for (int m = 3; m < a.E && ((qq >> m) & 1); ++m) {
              const uint32_t* src = stk_at<BN>(stk, m, ew, 0, lane);
#pragma unroll
              for (int w = 0; w < T::WORDS; ++w) cur[w] = node2(src[w * 32], cur[w]);
              l = m + 1;
            }
          }
          if (qq != Q - 1) {
            if (l == 2) {
#pragma unroll
              for (int w = 0; w < T::WORDS; ++w) n2[w] = cur[w];
            } else {
              if (l == 3 && stg_n) {  // this warp's last output store has read its level-3 block
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
                stg_n = 0;
              }
              uint32_t* dst = stk_at<BN>(stk, l, ew, 0, lane);
#pragma unroll
              for (int w = 0; w < T::WORDS; ++w) dst[w * 32] = cur[w];
            }
          } else if (a.o_tma && a.E >= 4) {
            // Every stored level has just been folded: the warp's level-3
            // block stages its 32 rows x COLS columns in the swizzled layout
            // of a TMA box, which leaves as one bulk tensor store (clipped
            // at the output's edges) -- coalesced, where a row per thread is
            // not.
            unsigned char* buf = reinterpret_cast<unsigned char*>(stk_at<BN>(stk, 3, ew, 0, 0));
            __syncwarp();  // all lanes' reads of the level are done
#pragma unroll
            for (int v = 0; v < T::COLS / 8; ++v)  // 16-byte chunk v of row `lane` at chunk v ^ (lane % 8)
              *reinterpret_cast<uint4*>(buf + lane * 128 + ((v ^ (lane & 7)) << 4)) =
                  make_uint4(cur[4 * v], cur[4 * v + 1], cur[4 * v + 2], cur[4 * v + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            const int ox = tn * BN + col0, oy = tm * BM + quarter * 32;
            if (lane == 0 && ox < a.C && oy < a.R) {  // (a box wholly past the edge is skipped)
              tma_store_2d(pb ? &tmO2 : &tmO, buf, ox, oy);
              bulk_commit();
            }
            stg_n = 1;
          } else if (r < a.R) {
            store_cols(outp, r * a.ld_r, (long long)tn * BN + col0, a.ld_c, a.C, cur);
          }
        }
      }
    } else {
      // One-leaf trees (the weight gradients over at most 64 tokens): the
      // leaf, rounded once, is the output.
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int pb = u % a.np, t = u / a.np;
        int tm, tn;
        tile_of(t, a, tm, tn);
        uint16_t* const outp = pb ? a.out2 : a.out;
        const long long r = (long long)tm * BM + row;
        uint32_t root[T::WORDS];
        if (!group_root<BN, GG, DUMP>(e, a, [&](int w, uint32_t g) { root[w] = g; }, pb, r, tn, 0)) break;
        if (a.o_tma) {
          // Row-major output: this warp's 32 rows x COLS columns go to shared
          // memory in the swizzled layout of a TMA box and leave as one bulk
          // tensor store (clipped at the output's edges); two buffers per
          // warp, so that staging the next tile overlaps this store.
          unsigned char* buf = stg_all + (ew * 2 + (stg_n & 1)) * T::STG_BUF;
          if (lane == 0) bulk_wait_read<1>();  // the store that last used this buffer has read it
          __syncwarp();
#pragma unroll
          for (int v = 0; v < T::COLS / 8; ++v)  // 16-byte chunk v of row `lane` at chunk v ^ (lane % 8)
            *reinterpret_cast<uint4*>(buf + lane * 128 + ((v ^ (lane & 7)) << 4)) =
                make_uint4(root[4 * v], root[4 * v + 1], root[4 * v + 2], root[4 * v + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          const int ox = tn * BN + col0, oy = tm * BM + quarter * 32;
          if (lane == 0 && ox < a.C && oy < a.R) {  // (a box wholly past the edge is skipped)
            tma_store_2d(pb ? &tmO2 : &tmO, buf, ox, oy);
            bulk_commit();
          }
          ++stg_n;
        } else if (r < a.R) {
          store_cols(outp, r * a.ld_r, (long long)tn * BN + col0, a.ld_c, a.C, root);
        }
      }
    }
    if (lane == 0) bulk_wait<0>();  // this warp's output stores have completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool tc_make_map(CUtensorMap* m, const uint16_t* base, long long rows, long long K, long long ld, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int BN, int GG, bool DUMP, bool KC, int LAY>
cudaError_t launch_bng(const CUtensorMap* m, const TcArgs& a, const KChunkMaps& kcm, int sm_count, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t setup_err = cudaSuccess;
  std::call_once(once, [] {
    setup_err = cudaFuncSetAttribute(k_tc<BN, GG, DUMP, KC, LAY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     TcGeo<BN>::MAX_SMEM);
    if (setup_err != cudaSuccess) return;
    // The in-kernel register split (setmaxnreg) hands over exactly the
    // launch's registers; with any other count it could not complete.
    cudaFuncAttributes fa;
    setup_err = cudaFuncGetAttributes(&fa, k_tc<BN, GG, DUMP, KC, LAY>);
    if (setup_err == cudaSuccess && fa.numRegs != kRegsLaunch) setup_err = cudaErrorInvalidConfiguration;
  });
  if (setup_err != cudaSuccess) return setup_err;
  const int units = a.num_m * a.num_n * a.np;
  const int slots = sm_count;
  const int grid = units < slots ? units : slots;
  const int smem = TcGeo<BN>::smem_for(a.G, a.E, a.nstage);
  return launch_dependent(k_tc<BN, GG, DUMP, KC, LAY>, dim3(grid), TcGeo<BN>::THREADS, smem, st, m[0], m[1], m[2], m[3], m[4],
                          m[5], a, kcm);
}

template <int BN, int GG>
cudaError_t launch_lay(const CUtensorMap* m, const TcArgs& a, const KChunkMaps& kcm, int sm_count, cudaStream_t st) {
  if (a.kc_op) return launch_bng<BN, GG, false, true, 3>(m, a, kcm, sm_count, st);  // chunked: both MN-major
  switch (a.a_mn + 2 * a.b_mn) {
    case 0: return launch_bng<BN, GG, false, false, 0>(m, a, kcm, sm_count, st);
    case 1: return launch_bng<BN, GG, false, false, 1>(m, a, kcm, sm_count, st);
    case 2: return launch_bng<BN, GG, false, false, 2>(m, a, kcm, sm_count, st);
    default: return launch_bng<BN, GG, false, false, 3>(m, a, kcm, sm_count, st);
  }
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap* m, const TcArgs& a, const KChunkMaps& kcm, int sm_count, cudaStream_t st) {
  if (a.dump) {
    switch (a.G) {
      case 1: return launch_bng<BN, 1, true, false, kLayRuntime>(m, a, kcm, sm_count, st);
      case 2: return launch_bng<BN, 2, true, false, kLayRuntime>(m, a, kcm, sm_count, st);
      case 3: return launch_bng<BN, 3, true, false, kLayRuntime>(m, a, kcm, sm_count, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (a.G) {
    case 1: return launch_lay<BN, 1>(m, a, kcm, sm_count, st);
    case 2: return launch_lay<BN, 2>(m, a, kcm, sm_count, st);
    case 3: return launch_lay<BN, 3>(m, a, kcm, sm_count, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool tc_tree_shape(long long L, int* G, int* E) {
  if (L == 1) {
    *G = 1;
    *E = 0;
    return true;
  }
  long long q;
  int g;
  if ((L & (L - 1)) == 0) {
    g = 2;
    q = L / 2;
  } else if (L % 3 == 0 && ((L / 3) & (L / 3 - 1)) == 0) {
    g = 3;
    q = L / 3;
  } else {
    return false;
  }
  int e = 0;
  while ((1ll << e) < q) ++e;
  if (e > kMaxLv) return false;
  *G = g;
  *E = e;
  return true;
}

cudaError_t launch_tc_gemms(const TcProblem* pr, int np, long long R, long long C, long long K,
                            long long ld_r, long long ld_c, const Waits& wt, int sm_count, cudaStream_t st,
                            float* dump, const TcKChunks* kc) {
  constexpr int bn = 128;
  if (R <= 0 || C <= 0) return cudaSuccess;
  if (np < 1 || np > 2) return cudaErrorInvalidValue;
  const long long L = (K + BK - 1) / BK;
  int G, E;
  if (K <= 0 || !tc_tree_shape(L, &G, &E)) return cudaErrorInvalidValue;
  for (int p = 0; p < np; ++p)
    if ((pr[p].lda % 8) || (pr[p].ldb % 8) || ((uintptr_t)pr[p].A & 15u) || ((uintptr_t)pr[p].B & 15u))
      return cudaErrorInvalidValue;
  if (R > (1ll << 31) || C > (1ll << 31)) return cudaErrorInvalidValue;
  TcArgs a{};
  a.R = (int)R;
  a.C = (int)C;
  a.G = G;
  a.np = np;
  a.b_mn = pr[0].b_mn ? 1 : 0;
  a.a_mn = pr[0].a_mn ? 1 : 0;
  if (np > 1 && (pr[1].b_mn != pr[0].b_mn || pr[1].a_mn != pr[0].a_mn)) return cudaErrorInvalidValue;
  a.num_m = (int)((R + BM - 1) / BM);
  a.num_n = (int)((C + bn - 1) / bn);
  // Row blocks: all row tiles when A is small enough for L2 to keep whole
  // (then B is read once); otherwise as many row tiles as 48 MB of A holds.
  {
    const bool shared_a = np > 1 && pr[1].A == pr[0].A && pr[1].lda == pr[0].lda;
    const double row_bytes = (double)BM * (double)K * 2.0 * (shared_a ? 1 : np);
    const double keep = 48.0 * (1 << 20);
    int gm = a.num_m;
    if (row_bytes * a.num_m > keep) gm = (int)(keep / row_bytes);
    a.gm = gm < 1 ? 1 : (gm > a.num_m ? a.num_m : gm);
  }
  a.E = E;
  a.L = (int)L;
  a.out = pr[0].out;
  a.out2 = np > 1 ? pr[1].out : nullptr;
  a.ld_r = ld_r;
  a.ld_c = ld_c;
  a.status = wt.status;
  a.spin = wt.spin;
  a.stall = wt.stall;
  a.dump = dump;
  a.nstage = TcGeo<bn>::stages_for(a.G, a.E);
  if (a.nstage > TcGeo<bn>::NBUF) a.nstage = TcGeo<bn>::NBUF;  // stage reuse is read off the leaf barriers
  // At least three stages: with fewer, an issuer could wait on a stage barrier
  // two phases behind (every tree shape the kernel takes leaves room for three).
  if (a.nstage < 3) return cudaErrorInvalidValue;
  CUtensorMap m[6];
  // Row-major outputs store through TMA (one-leaf trees, and trees with a
  // shared-memory stack level): boxes of 32 rows x 64 columns (one epilogue
  // warp's share of a tile), 128-byte swizzle.
  a.o_tma = 0;
  if (ld_c == 1 && ld_r % 8 == 0) {
    bool okm = true;
    for (int p = 0; p < 2 && okm; ++p) {
      const uint16_t* o = pr[p < np ? p : 0].out;
      okm = ((uintptr_t)o & 15u) == 0 && tc_make_map(&m[4 + p], o, R, C, ld_r, 32);
    }
    a.o_tma = okm ? 1 : 0;
  }
  if (!a.o_tma) m[4] = m[5] = CUtensorMap{};
  for (int p = 0; p < 2; ++p) {
    const TcProblem& q = pr[p < np ? p : 0];
    const bool bmap = q.b_mn ? tc_make_map(&m[2 * p + 1], q.B, K, C, q.ldb, BK)
                             : tc_make_map(&m[2 * p + 1], q.B, C, K, q.ldb, bn);
    const bool amap = q.a_mn ? tc_make_map(&m[2 * p], q.A, K, R, q.lda, BK) : tc_make_map(&m[2 * p], q.A, R, K, q.lda, BM);
    if (!amap || !bmap)
      return cudaErrorInvalidValue;
  }
  // A chunked K axis: one map per chunk, each over the chunk's own tokens
  // (rows), so that TMA zero-fills the tail of the last leaf exactly as the
  // map of a gathered operand would.
  KChunkMaps kcm{};
  a.kc_op = 0;
  a.kc_n = 0;
  if (kc && kc->op) {
    // (The chunked instance reads both operands MN-major, as the weight
    // gradients give them.)
    if (kc->n < 1 || kc->n > kMaxKChunks || !a.a_mn || !a.b_mn ||
        (kc->op != 1 && kc->op != 2))
      return cudaErrorInvalidValue;
    const long long ld = kc->op == 1 ? pr[0].lda : pr[0].ldb;
    const long long inner = kc->op == 1 ? R : C;
    long long start = 0;
    for (int c = 0; c < kc->n; ++c) {
      const long long t = kc->tokens[c];
      if (t < 1 || ((uintptr_t)kc->base[c] & 15u) || (c + 1 < kc->n && t % BK)) return cudaErrorInvalidValue;
      a.kc_leaf[c] = (int)(start / BK);
      if (!tc_make_map(&kcm.m[c], kc->base[c], t, inner, ld, BK)) return cudaErrorInvalidValue;
      start += t;
    }
    if (start != K) return cudaErrorInvalidValue;
    a.kc_op = kc->op;
    a.kc_n = kc->n;
  }
  return launch_bn<bn>(m, a, kcm, sm_count, st);
}

cudaError_t launch_tc_gemm(const uint16_t* A, long long lda, const uint16_t* B, long long ldb,
                           long long R, long long C, long long K, uint16_t* out, long long ld_r,
                           long long ld_c, const Waits& wt, int sm_count, cudaStream_t st,
                           bool b_mn, bool a_mn, float* dump) {
  const TcProblem p{A, lda, B, ldb, out, b_mn, a_mn};
  return launch_tc_gemms(&p, 1, R, C, K, ld_r, ld_c, wt, sm_count, st, dump);
}

}  // namespace detffn
