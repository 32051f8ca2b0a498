// k_tcs.cu -- few-token tensor-core tree contraction over balanced K ranges.
//
// out[r * ldo + c] = T_K(X[r, :], W[c, :]) for r < R <= 32 tokens and c < C
// weight rows, with the canonical FP32-leaf / BF16-node midpoint tree
// (RL-Kernel PR #325, "Design").  This is the decode shape: the weights are
// read once, so streaming them from HBM is the whole cost.  The weights sit on
// the MMA's 128-row side and the tokens on its 32-column side (rows R..31 of
// the token tile are zero-filled by TMA and never stored).
//
// Balance.  The work is the sequence of bottom groups (G leaves each) of all
// output tiles, tile after tile (gate and up tiles of one row block next to
// each other).  CTA b of P takes the groups [b W / P, (b+1) W / P), so every
// CTA streams the same number of bytes to within one group.  Where a range
// covers only part of a tile, the CTA folds that part into its maximal
// aligned subtrees -- nodes of the canonical tree -- and writes them as
// "pieces".  The CTAs that share a tile take a ticket once their ranges are
// done; the last of them folds the tile's pieces, left to right, into the
// root (and, for gate and up, applies SiLU * up).  A tile that lies inside
// one CTA's range is finished by that CTA directly.  Nothing waits on
// another CTA.  Without scratch ("direct" mode) CTAs take whole tiles.
//
// Streaming.  Two CTAs per SM.  In each, two producer warps issue the TMA
// loads of alternate leaves, one warp issues the MMAs (4 x K=16 per 64-wide
// leaf into a fresh TMEM buffer, one commit per leaf), and four epilogue
// warps read the leaves from TMEM, form the group roots and fold them.  The
// producer and MMA warps run converged and issue from one elected lane.
//
// Every wait is bounded; on a timeout the CTA records DETFFN_ERR_TIMEOUT,
// stops, drains its own copies and MMAs (bounded) and frees its TMEM.
#include <cuda.h>

#include <atomic>
#include <chrono>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "ptx.cuh"
#include "tc.h"
#include "tcs_pieces.cuh"

namespace detffn {
namespace {

constexpr int BM = 128;           // weight rows per tile (MMA M)
constexpr int BK = 64;            // leaf width (MMA K = 4 x 16)
constexpr int BN = 32;            // token columns (MMA N)
constexpr int kProd = 2;          // producer warps 0, 1
constexpr int kMmaWarp = kProd;   // warp 2: TMEM allocation and MMA issue
constexpr int kEpi0 = kProd + 1;  // warps 3..6: epilogue
constexpr int kEpiWarps = 4;
constexpr int kThreads = 32 * (kEpi0 + kEpiWarps);
constexpr int kNBuf = 8;          // TMEM leaf buffers of BN columns (256 columns; two CTAs per SM)
constexpr int kTmemCols = kNBuf * BN;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int WORDS = BN / 2;     // packed BF16 pairs per epilogue thread (one row, all tokens)
constexpr int REG_LV = 3;         // pending stack levels kept in registers
constexpr int LV_BYTES = BM * WORDS * 4;
constexpr int BAR_BYTES = 512;
constexpr int MAX_SMEM = 113 * 1024;
constexpr int MAX_STAGES = 8;
constexpr int PIECE = BM * BN;    // elements of one piece: [row][token], 64 bytes per row
// The tile fold at the end of a CTA's range reuses the stage and stack-level
// shared memory (idle by then): a stack of E levels and a few staged pieces,
// each [4 quarters][128 rows] x 16 bytes, and the piece list (8 bytes per entry).
constexpr int kFoldRowBytes = BM * BN * 2;  // one level or one staged piece: 8 KB
constexpr int kPieceRefBytes = 8;           // sizeof(PieceRef), checked where it is defined
constexpr int kMaxFoldChunk = 8;

static_assert(kTcsMaxLv >= REG_LV, "stack levels");
static_assert(MAX_STAGES <= kNBuf, "stage reuse is read off the leaf barriers");

__host__ __device__ inline int stages_for(int E) {
  const int lv = E > REG_LV ? E - REG_LV : 0;
  int n = (MAX_SMEM - 1024 - BAR_BYTES - lv * LV_BYTES) / STAGE;
  if (n > MAX_STAGES) n = MAX_STAGES;
  return n & ~1;  // even: stage s is always filled by producer s % 2
}
__host__ __device__ inline int smem_for(int E, int ns) {
  const int lv = E > REG_LV ? E - REG_LV : 0;
  return 1024 + ns * STAGE + lv * LV_BYTES + BAR_BYTES;
}

struct Bars {
  uint64_t full[MAX_STAGES], accf[kNBuf], acce[kNBuf], fin;
  uint32_t tmem_slot;
  int abort;
  int fold_last;  // the tile fold: this CTA arrived last on the unit's ticket
  int fold_n;     // the tile fold: entries of the current piece list
};
static_assert(sizeof(Bars) <= BAR_BYTES, "barrier block");

struct TcsArgs {
  int R, C;         // tokens (<= 32), weight rows per problem
  int G, E;         // leaves per bottom group, levels above the groups (2^E groups per tile)
  int np, T;        // problems (1 or 2), 128-row tiles per problem
  int ns;           // K shards per problem (1..8): shard q contracts K positions [q*ksh, (q+1)*ksh)
  long long ksh;    // K positions per shard (a multiple of 64)
  long long oss;    // element offset between the outputs of consecutive shards
  long long W;      // groups in all: np * ns * T * 2^E
  int cap;          // piece slots per CTA
  int nstage;
  int w_mn;         // weights stored [K][C] (C contiguous): MN-major A tiles
  uint16_t* slots;  // [gridDim.x][cap][BM][BN]; null: direct mode
  unsigned long long* tick;  // per fold unit: (launch epoch << 32) | arrivals; 0 after the fold
  unsigned epoch;   // this launch's ticket epoch (stale tickets of an aborted launch read as 0)
  int fused;        // gate (problem 0) and up (problem 1) with h = bf16(bf16(SiLU(gate)) * up)
  int UG;           // groups per fold unit: 2^E (one tree), or 2^(E+1) when fused (gate and up of a tile)
  int fold_ch;      // pieces staged at a time by the tile fold
  uint16_t* out0;   // roots go to out_p[r * ldo + c] (+ shard * oss); fused: gate, or null
  uint16_t* out1;   // fused: up, or null
  uint16_t* h;      // fused: h[r * ldo + c]
  const uint16_t* silu;
  long long ldo;
  int* status;
  long long spin;
  int stall;        // test only: the producers issue no loads
  int L;            // leaves per tree (G * 2^E)
  float* dump;      // leaf dump (DUMP instances): [np][R][C][L] FP32 leaves
};

// What the tile fold needs from the launch's arguments, copied at the fold
// (taking the address of the kernel's parameter block would move it to local
// memory for the whole kernel, the streaming loops included).
struct FoldArgs {
  int R, C, E, np, ns, UG, cap, fold_ch, fused;
  long long W, oss, ldo;
  const uint16_t* slots;
  uint16_t *out0, *out1, *h;
  const uint16_t* silu;
};

// Segment s = one tree per (row tile t, K shard q, problem pb), in that
// nesting: s = (t * ns + q) * np + pb.
struct Seg {
  int t, q, pb;
};
__host__ __device__ __forceinline__ Seg seg_of(long long s, int np, int ns) {
  const long long per = (long long)np * ns;
  const int rem = (int)(s % per);
  return Seg{(int)(s / per), rem / np, rem % np};
}

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

// Leaf dump (diagnostic instances): weight row crow's leaves for tokens
// t0 .. t0 + 15, as leaf j of the [R][C][L] array (tokens are the rows).
__device__ __forceinline__ void dump_tokens(float* d, long long crow, int t0, int R, int C, int L, int j,
                                            const uint32_t (&v)[16]) {
  if (crow >= C) return;
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if (t0 + i < R) d[((size_t)(t0 + i) * (size_t)C + (size_t)crow) * (size_t)L + (size_t)j] = __uint_as_float(v[i]);
}

// The 4 epilogue warps' own barrier (the producers and the MMA warp do not
// take part).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory"); }
// True in every epilogue thread if p holds in any of them (the same barrier).
__device__ __forceinline__ bool epi_any(bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.or.pred po, 1, %2, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "n"(kEpiWarps * 32)
      : "memory");
  return r != 0;
}

// Token i of a row held as packed BF16 pairs (word i / 2, low half first) to
// o[i * ldo + c], for i < R and c < C.
__device__ __forceinline__ void store_words(const uint32_t (&v)[WORDS], uint16_t* o, long long ldo, int R, long long c,
                                            long long C) {
  if (c >= C) return;
#pragma unroll
  for (int i = 0; i < BN; ++i)
    if (i < R) o[i * ldo + c] = (uint16_t)(v[i >> 1] >> (16 * (i & 1)));
}

// The fused stage boundary of one row: h = bf16(bf16(SiLU(gate)) * up) for
// every token, plus gate and up where they are kept.
template <class Args>
__device__ __forceinline__ void store_fused(const uint32_t (&g)[WORDS], const uint32_t (&u)[WORDS], const Args& a,
                                           long long c) {
  if (c >= a.C) return;
#pragma unroll
  for (int i = 0; i < BN; ++i) {
    if (i < a.R) {
      const uint16_t gb = (uint16_t)(g[i >> 1] >> (16 * (i & 1))), ub = (uint16_t)(u[i >> 1] >> (16 * (i & 1)));
      a.h[i * a.ldo + c] = f2bf(__fmul_rn(bf2f(__ldg(a.silu + gb)), bf2f(ub)));
      if (a.out0) a.out0[i * a.ldo + c] = gb;
      if (a.out1) a.out1[i * a.ldo + c] = ub;
    }
  }
}

// Arrival of one CTA on a fold unit's ticket; true for the last of the `need`
// CTAs that share the unit (which then resets the ticket).  A ticket left by
// a launch that stopped early carries another epoch and counts as 0.
__device__ __forceinline__ bool arrive_unit(unsigned long long* t, unsigned epoch, unsigned need) {
  unsigned long long old = atomicAdd(t, 0ull);
  for (;;) {
    const unsigned cnt = ((unsigned)(old >> 32) == epoch) ? (unsigned)old : 0u;
    const unsigned long long nv = ((unsigned long long)epoch << 32) | (unsigned long long)(cnt + 1);
    const unsigned long long prev = atomicCAS(t, old, nv);
    if (prev == old) {
      if (cnt + 1 < need) return false;
      atomicExch(t, 0ull);
      return true;
    }
    old = prev;
  }
}

// Writes one row (all tokens) of the CTA's next piece: the row's 64 bytes
// at [row], so that the top kernel reads a quarter row with one 16-byte load.
__device__ __forceinline__ void emit_piece(uint16_t* slots, int& n, int cap, int row, const uint32_t (&v)[WORDS]) {
  if (n < cap) {
    uint4* o = reinterpret_cast<uint4*>(slots + (size_t)n * PIECE) + row * (WORDS / 4);
#pragma unroll
    for (int i = 0; i < WORDS / 4; ++i) o[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
  ++n;
}

}  // namespace
}  // namespace detffn

namespace detffn {
namespace {

// The weight tile of the leaf at K position k, row tile t: 128 rows x 64 K,
// K-major (one box) or, for weights stored [K][C], MN-major (two boxes of
// 64 rows x 64 K).
__device__ __forceinline__ void load_w(unsigned char* dst, const CUtensorMap* mW, int k, int t, uint64_t* bar,
                                       uint64_t pol, int mn) {
  if (mn) {
    tma_load_2d_hint(dst, mW, t * BM, k, bar, pol);
    tma_load_2d_hint(dst + A_BYTES / 2, mW, t * BM + BM / 2, k, bar, pol);
  } else {
    tma_load_2d_hint(dst, mW, k, t * BM, bar, pol);
  }
}

struct PieceRef {
  int slot;  // b * cap + j
  int at;    // level m (bits 0..7), left siblings it merges with (bits 8..15), and whether the
             // result is the root (bit 16): the fold, the same for every element, worked out once
};
static_assert(sizeof(PieceRef) == kPieceRefBytes, "piece list entries: shared-memory sizes assume 8 bytes");

// Lists, in order, the pieces of segment s that CTAs [b_base, min(b_base +
// 32, b_end)) wrote (P CTAs in all): one lane per CTA, placed by a warp
// scan.  Returns the count.
__device__ int list_pieces(const FoldArgs& a, long long s, long long b_base, long long b_end, long long P,
                           PieceRef* list, int lane) {
  const int Q = 1 << a.E;
  const long long ws = s * Q, we = ws + Q;
  const long long b = b_base + lane;
  int cnt = 0;
  long long lo = 0, hi = 0;
  if (b < b_end) {
    const long long blo = b * a.W / P, bhi = (b + 1) * a.W / P;
    lo = blo > ws ? blo : ws;
    hi = bhi < we ? bhi : we;
    if (lo < hi) cnt = count_pieces((int)(lo - ws), (int)(hi - ws));
  }
  int incl = cnt;
  for (int d = 1; d < 32; d <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += t;
  }
  if (cnt > 0) {
    int j = slot_base(b, s, a.W, P, Q, a.UG);
    int pos = incl - cnt;
    const PieceSplit p = piece_split((int)(lo - ws), (int)(hi - ws));
    if (p.one) {
      list[pos].slot = (int)(b * a.cap + j);
      list[pos].at = fold_code(p.x, hibit((unsigned)(p.y - p.x)), a.E);
    } else {
      int at = p.x;
#pragma unroll 1
      for (unsigned rem = (unsigned)(p.z - p.x); rem; ++pos, ++j) {  // ascending sizes
        const unsigned bit = rem & (0u - rem);
        list[pos].slot = (int)(b * a.cap + j);
        list[pos].at = fold_code(at, hibit(bit), a.E);
        at += (int)bit;
        rem -= bit;
      }
#pragma unroll 1
      for (unsigned rem = (unsigned)(p.y - p.z); rem; ++pos, ++j) {  // descending sizes
        const unsigned bit = 1u << hibit(rem);
        list[pos].slot = (int)(b * a.cap + j);
        list[pos].at = fold_code(at, hibit(bit), a.E);
        at += (int)bit;
        rem -= bit;
      }
    }
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}

__device__ __forceinline__ uint4 add4(uint4 l, uint4 r) {
  return make_uint4(add_bf16x2(l.x, r.x), add_bf16x2(l.y, r.y), add_bf16x2(l.z, r.z), add_bf16x2(l.w, r.w));
}

// Folds segment s's pieces (all CTAs that share it, in order) into this
// thread's row of the root: 32 tokens as 4 x 16 bytes.  Shared memory (the
// idle stage area): stack [E][4][BM] and staged pieces [fold_ch][4][BM]
// (16 bytes each, this thread's row only), then the list.
__device__ __noinline__ void fold_segment(const FoldArgs& a, long long s, unsigned char* fsm, Bars* bars, int row, int ew,
                             int lane, uint4 (&root)[4]) {
  const int Q = 1 << a.E;
  const long long P = gridDim.x;
  uint4* stk = reinterpret_cast<uint4*>(fsm);
  uint4* buf = stk + (size_t)a.E * 4 * BM;
  PieceRef* list = reinterpret_cast<PieceRef*>(buf + (size_t)a.fold_ch * 4 * BM);
  const long long b_last = cta_of((s + 1) * Q - 1, a.W, P);
#pragma unroll
  for (int i = 0; i < 4; ++i) root[i] = make_uint4(0, 0, 0, 0);
#pragma unroll 1
  for (long long b0 = cta_of(s * Q, a.W, P); b0 <= b_last; b0 += 32) {
    epi_sync();  // the previous batch's list is no longer read
    if (ew == 0) {
      const int n = list_pieces(a, s, b0, b_last + 1, P, list, lane);
      if (lane == 0) bars->fold_n = n;
    }
    epi_sync();
    const int n = bars->fold_n;
#pragma unroll 1
    for (int k0 = 0; k0 < n; k0 += a.fold_ch) {
      const int kend = n < k0 + a.fold_ch ? n : k0 + a.fold_ch;
#pragma unroll 1
      for (int k = k0; k < kend; ++k) {
        const uint16_t* src = a.slots + (size_t)list[k].slot * PIECE + (size_t)row * BN;
#pragma unroll
        for (int qd = 0; qd < 4; ++qd)
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(buf + ((k - k0) * 4 + qd) * BM + row)),
                       "l"(src + 8 * qd)
                       : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll 1
      for (int k = k0; k < kend; ++k) {
        const int code = list[k].at;
        const int m = code & 0xFF, kk = (code >> 8) & 0xFF;
        uint4 cur[4];
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) cur[qd] = buf[((k - k0) * 4 + qd) * BM + row];
#pragma unroll 1
        for (int i = 0; i < kk; ++i)
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) cur[qd] = add4(stk[((m + i) * 4 + qd) * BM + row], cur[qd]);
        if (code >> 16) {
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) root[qd] = cur[qd];
        } else {
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) stk[((m + kk) * 4 + qd) * BM + row] = cur[qd];
        }
      }
    }
  }
}

__device__ __forceinline__ void words_of(const uint4 (&r)[4], uint32_t (&v)[WORDS]) {
#pragma unroll
  for (int qd = 0; qd < 4; ++qd) {
    v[4 * qd] = r[qd].x;
    v[4 * qd + 1] = r[qd].y;
    v[4 * qd + 2] = r[qd].z;
    v[4 * qd + 3] = r[qd].w;
  }
}

// The last CTA to arrive on fold unit u: folds its segments' pieces and
// stores the result (the root, or h for gate and up).
__device__ __noinline__ void fold_unit(const FoldArgs& a, long long u, unsigned char* fsm, Bars* bars, int row, int ew, int lane) {
  const int spu = a.fused ? 2 : 1;
  uint4 r0[4];
  uint32_t v0[WORDS];
  fold_segment(a, u * spu, fsm, bars, row, ew, lane, r0);
  words_of(r0, v0);
  const Seg sg = seg_of(u * spu, a.np, a.ns);
  const long long c = (long long)sg.t * BM + row;
  if (!a.fused) {
    store_words(v0, (sg.pb ? a.out1 : a.out0) + sg.q * a.oss, a.ldo, a.R, c, a.C);
    return;
  }
  uint4 r1[4];
  uint32_t v1[WORDS];
  fold_segment(a, u * spu + 1, fsm, bars, row, ew, lane, r1);
  words_of(r1, v1);
  store_fused(v0, v1, a, c);
}

// The streaming kernel.  Each role walks the CTA's groups in the same order:
// segment (tile, problem) after segment, groups qa..qb-1 of each.
// 128 registers: registers are granted per 4 warps, so a CTA of 7 warps holds
// 8 x 32 x 128 = 32,768 and two CTAs fit one SM's 65,536.
template <int GG, bool DUMP>
__global__ void __maxnreg__(128)
    k_tcs(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
          const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmX2, const TcsArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int NS = a.nstage;
  const int slv = a.E > REG_LV ? a.E - REG_LV : 0;
  unsigned char* stages = smem;
  uint32_t* stk = reinterpret_cast<uint32_t*>(smem + NS * STAGE);
  Bars* bars = reinterpret_cast<Bars*>(smem + NS * STAGE + slv * LV_BYTES);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Q = 1 << a.E;
  const bool direct = a.slots == nullptr;
  const long long w0 = range_lo(blockIdx.x, a.W, gridDim.x, a.UG, direct);
  const long long w1 = range_lo(blockIdx.x + 1ll, a.W, gridDim.x, a.UG, direct);
  const long long limit = a.spin > 0 ? a.spin : kDefaultSpin;
  // A wait of an earlier launch ran out (the status word is set until the
  // caller reads it): its outputs, which may be this launch's inputs, are
  // unfinished, so this launch does nothing.
  if (__syncthreads_or(a.status != nullptr && *(volatile int*)a.status != 0)) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->full[s], 1);
    }
    for (int b = 0; b < kNBuf; ++b) {
      mbar_init(&bars->accf[b], 1);
      mbar_init(&bars->acce[b], kEpiWarps);
    }
    mbar_init(&bars->fin, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp < kProd && lane == 0) {
    prefetch_tmap(warp == 0 ? &tmW : &tmX);
    if (a.np > 1) prefetch_tmap(warp == 0 ? &tmW2 : &tmX2);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  // Programmatic dependent launch: the set-up above, and the weight tiles of
  // the first stages, overlap the previous kernel; nothing else touches
  // global memory before it has completed (grid_dep_wait).
  grid_dep_launch();

  if (warp < kProd) {
    // ---------------- TMA producers: leaf it goes to producer it % kProd ----------------
    // Converged warps; one lane issues.  Stage it % NS is free once leaf
    // it - NS has been committed, which its "full accumulator" barrier
    // reports (NS <= kNBuf, so that barrier cannot have moved on by a second
    // phase: the MMAs run in leaf order).
    // Weights are read once: evict them first, so that the pieces stay in L2.
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    // Before the previous kernel has finished: this producer's share of the
    // first NS stages, weight tiles only (no kernel here writes weights).
    if (!a.stall) {
      long long it = 0;
      for (long long w = w0; w < w1 && it < NS;) {
        const long long s = w / Q;
        const int qa = (int)(w - s * Q);
        const int qb = (int)((w1 - s * Q) < Q ? (w1 - s * Q) : Q);
        const Seg g = seg_of(s, a.np, a.ns);
        const int k0 = (int)(g.q * a.ksh);
        const CUtensorMap* mW = g.pb ? &tmW2 : &tmW;
        for (int j = qa * GG; j < qb * GG && it < NS; ++j, ++it) {
          if ((int)(it % kProd) != warp) continue;
          if (elect_one()) {
            mbar_arrive_expect_tx(&bars->full[it], (uint32_t)STAGE);
            load_w(stages + it * STAGE, mW, k0 + j * BK, g.t, &bars->full[it], pol, a.w_mn);
          }
          __syncwarp();
        }
        w = s * Q + qb;
      }
    }
    grid_dep_wait();  // the token tiles may be the previous kernel's output
    long long it = 0;
    Ring rs;  // stage of load it
    Ring rv;  // TMEM buffer of leaf it - NS
    bool ok = true;
    for (long long w = w0; w < w1 && ok;) {
      const long long s = w / Q;
      const int qa = (int)(w - s * Q);
      const int qb = (int)((w1 - s * Q) < Q ? (w1 - s * Q) : Q);
      const Seg g = seg_of(s, a.np, a.ns);
      const int k0 = (int)(g.q * a.ksh);
      const CUtensorMap* mW = g.pb ? &tmW2 : &tmW;
      const CUtensorMap* mX = g.pb ? &tmX2 : &tmX;
      for (int j = qa * GG; j < qb * GG; ++j, ++it, rs.next(NS)) {
        const bool reuse = it >= NS;  // (the first NS weight tiles are already on their way)
        const int vb = rv.slot;
        const uint32_t vph = rv.phase;
        if (reuse) rv.next(kNBuf);
        if ((int)(it % kProd) != warp) continue;
        const int st = rs.slot;
        unsigned char* dst = stages + st * STAGE;
        if (reuse) {
          const bool wok = wait_or_abort(&bars->accf[vb], vph, limit, abort_flag, a.status);
          if (!__all_sync(0xffffffffu, wok)) {
            ok = false;
            break;
          }
        }
        if (!a.stall && elect_one()) {
          if (reuse) {
            mbar_arrive_expect_tx(&bars->full[st], (uint32_t)STAGE);
            load_w(dst, mW, k0 + j * BK, g.t, &bars->full[st], pol, a.w_mn);
          }
          tma_load_2d(dst + A_BYTES, mX, k0 + j * BK, 0, &bars->full[st]);
        }
        __syncwarp();
      }
      w = s * Q + qb;
    }
    // Drain: this producer's last loads have landed (on the long bound,
    // whatever the call's poll limit: no CTA exits with copies in flight).
    if (lane == 0 && !a.stall)
      for (long long i = (it > NS ? it - NS : 0); i < it; ++i)
        if ((int)(i % kProd) == warp)
          mbar_wait(&bars->full[i % NS], (uint32_t)((i / NS) & 1), kDefaultSpin, nullptr);
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (converged warp; one lane issues) ----------------
    // Leaf n of this CTA's range uses stage n % NS and TMEM buffer n % kNBuf;
    // one commit per leaf (its "full accumulator" barrier, read by the
    // epilogue and the producers).
    const uint32_t idesc = idesc_bf16(BM, BN) | (a.w_mn ? kIdescTransA : 0u);
    const uint32_t astep = a.w_mn ? 128u : 2u;  // K = 16 step in descriptor units
    const long long nleaf = (w1 - w0) * GG;
    Ring rs, rb;  // pipeline stage; TMEM leaf buffer
    bool ok = true;
    for (long long n = 0; n < nleaf && ok; ++n, rs.next(NS), rb.next(kNBuf)) {
      const int st = rs.slot, b = rb.slot;
      const bool wok = wait_or_abort(&bars->acce[b], rb.phase ^ 1u, limit, abort_flag, a.status) &&
                       wait_or_abort(&bars->full[st], rs.phase, limit, abort_flag, a.status);
      if (!__all_sync(0xffffffffu, wok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t da = a.w_mn ? smem_desc_sw128_mn(stages + st * STAGE) : smem_desc_sw128(stages + st * STAGE);
      const uint64_t db = smem_desc_sw128(stages + st * STAGE + A_BYTES);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)  // a fresh FP32 accumulation per leaf
          tc_mma_bf16(tmem + (uint32_t)(b * BN), da + astep * kk, db + 2 * kk, idesc, kk > 0 ? 1u : 0u);
        tc_commit(&bars->accf[b]);
      }
      __syncwarp();
    }
    if (elect_one()) tc_commit(&bars->fin);  // arrives when every MMA issued above has completed
    __syncwarp();
    if (lane == 0) mbar_wait(&bars->fin, 0, kDefaultSpin, nullptr);  // before TMEM is freed (long bound)
  } else {
    // ---------------- epilogue: leaves -> group roots -> pieces ----------------
    grid_dep_wait();  // its stores may overwrite what the previous kernel reads
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    uint16_t* const myslots = direct ? nullptr : a.slots + (size_t)blockIdx.x * a.cap * PIECE;
    uint32_t lc = 0;  // leaves consumed (kNBuf is a power of two)
    int np_out = 0;  // pieces written
    bool ok = true;
    uint32_t reg_lv[REG_LV][WORDS];
    for (long long w = w0; w < w1 && ok;) {
      const long long s = w / Q;
      const int qa = (int)(w - s * Q);
      const int qb = (int)((w1 - s * Q) < Q ? (w1 - s * Q) : Q);
      unsigned pend = 0;  // levels holding a left child that waits for its right sibling
      for (int q = qa; q < qb; ++q) {
        for (int g = 0; g < GG; ++g)
          if (!wait_or_abort(&bars->accf[(lc + g) % kNBuf], (uint32_t)(((lc + g) / kNBuf) & 1), limit, abort_flag,
                             a.status))
            ok = false;
        if (__any_sync(0xffffffffu, !ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t b0 = (uint32_t)((lc % kNBuf) * BN), b1 = (uint32_t)(((lc + 1) % kNBuf) * BN),
                       b2 = (uint32_t)(((lc + 2) % kNBuf) * BN);
        // The group root: a lone leaf rounded once, l0 + l1, or l0 + (l1 + l2).
        uint32_t root[WORDS];
        // Leaf dump: this thread's weight row of the tile, tokens 16 c + i.
        const Seg sg = seg_of(s, a.np, a.ns);
        float* const dmp = DUMP ? a.dump + (size_t)sg.pb * a.R * a.C * a.L : nullptr;
        const long long crow = (long long)sg.t * BM + row;
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) {
          uint32_t v0[16];
          if constexpr (GG == 3) {
            uint32_t v1[16], v2[16], n12[8];
            tmem_ld16(tmem + lane_addr + b1 + 16 * c, v1);
            tmem_ld16(tmem + lane_addr + b2 + 16 * c, v2);
            tmem_wait_ld();
            if constexpr (DUMP) {
              dump_tokens(dmp, crow, 16 * c, a.R, a.C, a.L, q * GG + 1, v1);
              dump_tokens(dmp, crow, 16 * c, a.R, a.C, a.L, q * GG + 2, v2);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
              n12[i] = pack_bf16x2_of(add_f32x2(f32x2(v1[2 * i], v1[2 * i + 1]), f32x2(v2[2 * i], v2[2 * i + 1])));
            tmem_ld16(tmem + lane_addr + b0 + 16 * c, v0);
            tmem_wait_ld();
            if constexpr (DUMP) dump_tokens(dmp, crow, 16 * c, a.R, a.C, a.L, q * GG, v0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              root[8 * c + i] =
                  pack_bf16x2_of(add_f32x2(f32x2(v0[2 * i], v0[2 * i + 1]), f32x2(n12[i] << 16, n12[i] & 0xFFFF0000u)));
          } else if constexpr (GG == 2) {
            uint32_t v1[16];
            tmem_ld16(tmem + lane_addr + b0 + 16 * c, v0);
            tmem_ld16(tmem + lane_addr + b1 + 16 * c, v1);
            tmem_wait_ld();
            if constexpr (DUMP) {
              dump_tokens(dmp, crow, 16 * c, a.R, a.C, a.L, q * GG, v0);
              dump_tokens(dmp, crow, 16 * c, a.R, a.C, a.L, q * GG + 1, v1);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
              root[8 * c + i] = pack_bf16x2_of(add_f32x2(f32x2(v0[2 * i], v0[2 * i + 1]), f32x2(v1[2 * i], v1[2 * i + 1])));
          } else {
            tmem_ld16(tmem + lane_addr + b0 + 16 * c, v0);
            tmem_wait_ld();
            if constexpr (DUMP) dump_tokens(dmp, crow, 16 * c, a.R, a.C, a.L, q * GG, v0);
#pragma unroll
            for (int i = 0; i < 8; ++i) root[8 * c + i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
          }
        }
        // The leaves are in registers: return the TMEM buffers to the MMA warp.
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
          for (int g = 0; g < GG; ++g) mbar_arrive(&bars->acce[(lc + g) % kNBuf]);
        lc += GG;

        // Fold: merge with pending left siblings inside [qa, qb); a right
        // child whose left sibling lies before qa is a finished piece; a left
        // child waits on the stack for its right sibling.
        int at = q;
        bool live = true;
#pragma unroll
        for (int m = 0; m <= kTcsMaxLv; ++m) {
          if (live) {
            if (m == a.E) {  // the whole tile: its root
              const long long u = s * Q / a.UG;
              if (direct || (!a.fused && u * a.UG >= w0 && (u + 1) * a.UG <= w1)) {
                // A one-tree unit inside this range: store its root here.
                store_words(root, (sg.pb ? a.out1 : a.out0) + sg.q * a.oss, a.ldo, a.R, (long long)sg.t * BM + row,
                            a.C);
              } else {
                emit_piece(myslots, np_out, a.cap, row, root);
              }
              live = false;
            } else if (((at >> m) & 1) && at - (1 << m) >= qa) {
#pragma unroll
              for (int i = 0; i < WORDS; ++i) {
                const uint32_t left = m < REG_LV ? reg_lv[m < REG_LV ? m : 0][i]
                                                 : stk[((m - REG_LV) * WORDS + i) * BM + row];
                root[i] = add_bf16x2(left, root[i]);
              }
              pend &= ~(1u << m);
              at -= 1 << m;
            } else if ((at >> m) & 1) {
              emit_piece(myslots, np_out, a.cap, row, root);
              live = false;
            } else {
#pragma unroll
              for (int i = 0; i < WORDS; ++i) {
                if (m < REG_LV) reg_lv[m < REG_LV ? m : 0][i] = root[i];
                else stk[((m - REG_LV) * WORDS + i) * BM + row] = root[i];
              }
              pend |= 1u << m;
              live = false;
            }
          }
        }
      }
      if (!ok) break;
      // The segment ends: pending left children are finished pieces (left to right = high level first).
#pragma unroll
      for (int m = kTcsMaxLv - 1; m >= 0; --m)
        if ((pend >> m) & 1) {
          uint32_t v[WORDS];
#pragma unroll
          for (int i = 0; i < WORDS; ++i)
            v[i] = m < REG_LV ? reg_lv[m < REG_LV ? m : 0][i] : stk[((m - REG_LV) * WORDS + i) * BM + row];
          emit_piece(myslots, np_out, a.cap, row, v);
        }
      w = s * Q + qb;
    }
    // The fold units that hold pieces of this range (one-tree units at its
    // two ends that other CTAs share; every fused unit): arrive on their
    // tickets; the last CTA to arrive folds the unit's pieces.  (The stages
    // and stack levels are idle now: every leaf has been consumed.)  Every
    // epilogue warp gets here exactly once, also after a wait ran out, and
    // they decide together: a warp that stopped early must not leave the
    // others waiting at the fold's barriers.
    const bool all_ok = !epi_any(!ok);
    if (all_ok && !direct) {
      const long long ua = w0 / a.UG, ub = (w1 - 1) / a.UG;
      const long long step = a.fused ? 1 : (ub > ua ? ub - ua : 1);
      for (long long u = ua; u <= ub; u += step) {
        if (!a.fused && u * a.UG >= w0 && (u + 1) * a.UG <= w1) continue;  // stored directly
        __threadfence();  // this thread's pieces are visible before the ticket
        epi_sync();
        if (warp == kEpi0 && lane == 0) {
          const unsigned need =
              (unsigned)(cta_of((u + 1) * a.UG - 1, a.W, gridDim.x) - cta_of(u * a.UG, a.W, gridDim.x) + 1);
          bars->fold_last = arrive_unit(a.tick + u, a.epoch, need) ? 1 : 0;
        }
        epi_sync();
        if (bars->fold_last) {
          __threadfence();
          const FoldArgs fa{a.R,   a.C,   a.E,     a.np,  a.ns,  a.UG,   a.cap,  a.fold_ch, a.fused,
                            a.W,   a.oss, a.ldo,   a.slots, a.out0, a.out1, a.h, a.silu};
          fold_unit(fa, u, smem, bars, row, warp - kEpi0, lane);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace
}  // namespace detffn

namespace detffn {
namespace {

}  // namespace
}  // namespace detffn

namespace detffn {

bool tcs_plan(long long R, long long C, long long K, int np, int max_ctas, bool direct, TcsPlan* p, int ns,
              bool fused) {
  if (R < 1 || R > BN || C < 1 || K < 1 || np < 1 || np > 2 || max_ctas < 1) return false;
  if (ns < 1 || ns > kTcsMaxShards || (ns > 1 && K % BK != 0)) return false;
  if (fused && (np != 2 || ns != 1)) return false;
  const long long L = (K + BK - 1) / BK;
  int G;
  long long q;
  if (L == 1) {
    G = 1;
    q = 1;
  } else if ((L & (L - 1)) == 0) {
    G = 2;
    q = L / 2;
  } else if (L % 3 == 0 && ((L / 3) & (L / 3 - 1)) == 0) {
    G = 3;
    q = L / 3;
  } else {
    return false;
  }
  int E = 0;
  while ((1ll << E) < q) ++E;
  if (E > kTcsMaxLv || C > (1ll << 30)) return false;
  TcsPlan r;
  r.R = (int)R;
  r.C = C;
  r.K = K;
  r.G = G;
  r.E = E;
  r.np = np;
  r.ns = ns;
  r.fused = fused;
  r.T = (int)((C + BM - 1) / BM);
  const int Q = 1 << E;
  r.UG = fused ? 2 * Q : Q;
  r.W = (long long)np * ns * r.T * Q;
  r.direct = direct;
  const long long units = r.W / r.UG;
  r.P = (int)(max_ctas < (direct ? units : r.W) ? max_ctas : (direct ? units : r.W));
  r.nstage = stages_for(E);
  if (r.nstage < 2) return false;
  if (direct) {
    *p = r;
    return true;
  }
  // Piece slots per CTA: the most pieces any CTA writes (only the fold units
  // at the two ends of its range can be shared with other CTAs).
  int cap = 1;
  for (long long b = 0; b < r.P; ++b) {
    const long long bhi = (b + 1) * r.W / r.P;
    const int n = slot_base(b, (bhi - 1) / Q + 1, r.W, r.P, Q, r.UG);
    if (n > cap) cap = n;
  }
  r.cap = cap;
  // The tile fold reuses the stages and stack levels: the fold stack (E
  // levels), at least one staged piece and a list of up to 32 CTAs' pieces.
  const int lv = E > REG_LV ? E - REG_LV : 0;
  const long long avail = (long long)r.nstage * STAGE + (long long)lv * LV_BYTES;
  const long long list_bytes = (32ll * cap) * kPieceRefBytes;
  const long long ch = (avail - (long long)E * kFoldRowBytes - list_bytes) / kFoldRowBytes;
  if (ch < 1) return false;
  r.fold_ch = (int)(ch < kMaxFoldChunk ? ch : kMaxFoldChunk);
  const size_t slots = (size_t)r.P * cap * PIECE * 2;
  r.tick_off = (slots + 255) & ~(size_t)255;
  r.scratch = r.tick_off + (size_t)units * sizeof(unsigned long long);
  *p = r;
  return true;
}

namespace {

// A launch that may begin while the previous kernel on the stream finishes
// (programmatic dependent launch); the kernels wait in grid_dep_wait before
// touching global memory.
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
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

cudaError_t tcs_launch(const TcsPlan& plan, const TcsProblem* pr, long long ldo, uint16_t* h, const uint16_t* silu,
                       void* scratch, size_t scratch_bytes, const Waits& wt, cudaStream_t st, float* dump,
                       long long oss) {
  if (plan.ns > 1 && (h || dump)) return cudaErrorInvalidValue;
  if ((h != nullptr) != plan.fused || (h && !silu) || (plan.fused && plan.direct)) return cudaErrorInvalidValue;
  const long long Ktot = plan.K * plan.ns;  // the maps span every shard's K range
  if (!plan.direct && (!scratch || scratch_bytes < plan.scratch || ((uintptr_t)scratch & 255u)))
    return cudaErrorInvalidValue;
  for (int p = 0; p < plan.np; ++p)
    if ((pr[p].ldw % 8) || (pr[p].ldx % 8) || ((uintptr_t)pr[p].W & 15u) || ((uintptr_t)pr[p].X & 15u) ||
        pr[p].w_mn != pr[0].w_mn)
      return cudaErrorInvalidValue;
  CUtensorMap m[4];
  for (int p = 0; p < 2; ++p) {
    const TcsProblem& q = pr[p < plan.np ? p : 0];
    const bool wmap = q.w_mn ? tc_make_map(&m[2 * p], q.W, Ktot, plan.C, q.ldw, BK)
                             : tc_make_map(&m[2 * p], q.W, plan.C, Ktot, q.ldw, BM);
    if (!wmap ||
        !tc_make_map(&m[2 * p + 1], q.X, plan.R, Ktot, q.ldx, BN))
      return cudaErrorInvalidValue;
  }
  static std::once_flag once;
  static cudaError_t setup_err = cudaSuccess;
  std::call_once(once, [] {
    cudaError_t e = cudaSuccess;
    void (*ks[6])(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TcsArgs) = {
        k_tcs<1, false>, k_tcs<2, false>, k_tcs<3, false>, k_tcs<1, true>, k_tcs<2, true>, k_tcs<3, true>};
    for (auto k : ks) {
      // Two CTAs per SM: all of their shared memory, at most 113 KB each.
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_SMEM);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    }
    setup_err = e;
  });
  if (setup_err != cudaSuccess) return setup_err;
  TcsArgs a{};
  a.R = plan.R;
  a.C = (int)plan.C;
  a.G = plan.G;
  a.E = plan.E;
  a.np = plan.np;
  a.ns = plan.ns;
  a.ksh = plan.K;
  a.oss = oss;
  a.T = plan.T;
  a.W = plan.W;
  a.cap = plan.cap;
  a.nstage = plan.nstage;
  a.w_mn = pr[0].w_mn ? 1 : 0;
  a.slots = plan.direct ? nullptr : static_cast<uint16_t*>(scratch);
  a.tick = plan.direct ? nullptr
                       : reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(scratch) + plan.tick_off);
  // Launch epochs: consecutive per process from a start that varies between
  // processes; 0 is never used (a zeroed ticket is always read as empty).
  static std::atomic<unsigned> epochs{(unsigned)std::chrono::steady_clock::now().time_since_epoch().count() | 1u};
  unsigned ep = epochs.fetch_add(1u);
  if (ep == 0) ep = epochs.fetch_add(1u);
  a.epoch = ep;
  a.fused = plan.fused ? 1 : 0;
  a.UG = plan.UG;
  a.fold_ch = plan.fold_ch;
  a.h = h;
  a.silu = silu;
  a.out0 = pr[0].out;
  a.out1 = plan.np > 1 ? pr[1].out : nullptr;
  a.ldo = ldo;
  a.status = wt.status;
  a.spin = wt.spin;
  a.stall = wt.stall;
  a.L = plan.G << plan.E;
  a.dump = dump;
  const int smem = smem_for(plan.E, plan.nstage);
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TcsArgs) =
      dump ? (plan.G == 1 ? k_tcs<1, true> : plan.G == 2 ? k_tcs<2, true> : k_tcs<3, true>)
           : (plan.G == 1 ? k_tcs<1, false> : plan.G == 2 ? k_tcs<2, false> : k_tcs<3, false>);
  return launch_dependent(kern, dim3(plan.P), kThreads, smem, st, m[0], m[1], m[2], m[3], a);
}

}  // namespace

cudaError_t launch_tcs(const TcsPlan& plan, const TcsProblem* pr, long long ldo, void* scratch,
                       size_t scratch_bytes, const Waits& wt, cudaStream_t st, float* dump, long long oss) {
  for (int p = 0; p < plan.np; ++p)
    if (!pr[p].out) return cudaErrorInvalidValue;
  return tcs_launch(plan, pr, ldo, nullptr, nullptr, scratch, scratch_bytes, wt, st, dump, oss);
}

cudaError_t launch_tcs_gateup(const TcsPlan& plan, const TcsProblem* pr, uint16_t* h, long long ldo,
                              const uint16_t* silu, void* scratch, size_t scratch_bytes, const Waits& wt,
                              cudaStream_t st) {
  if (plan.np != 2 || !h || !silu) return cudaErrorInvalidValue;
  return tcs_launch(plan, pr, ldo, h, silu, scratch, scratch_bytes, wt, st, nullptr, 0);
}

}  // namespace detffn
