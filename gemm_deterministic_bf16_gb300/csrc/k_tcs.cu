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
// "pieces"; a second kernel folds each tile's pieces, left to right, into the
// root.  A whole tile is one piece, its root.  Where every range is one
// aligned block and a tile has at most 8 of them ("folded trees"), no second
// kernel runs: each CTA takes a ticket of its tile once its piece is
// written, and the tile's last CTA folds the pieces and stores the root.
// Nothing in the streaming kernel waits on another CTA.  Without scratch
// ("direct" mode) CTAs take whole tiles and store the roots themselves.
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
constexpr int kTopTok = 8;        // top kernel: tokens per CTA (one 16-byte quarter of a piece row; grid.y covers the rest)
constexpr int kTopThreads = BM;   // one thread per row
// Pieces per segment staged in shared memory at a time: fused gate/up CTAs
// (two segments, a few pieces each at decode sizes) and plain CTAs (one
// segment, up to a few dozen pieces).
__host__ __device__ constexpr int top_chunk(bool fused) { return fused ? 8 : 32; }
// Dynamic shared memory of a top CTA: staged pieces, the fold stacks (E
// levels), the output tiles and the piece lists (16 bytes per row and piece
// or level).
constexpr int kPieceRefBytes = 8;  // sizeof(PieceRef), checked where it is defined
__host__ __device__ inline int top_smem(bool fused, int E, int cap) {
  const int nseg = fused ? 2 : 1;
  return nseg * top_chunk(fused) * BM * 16 + nseg * E * BM * 16 + 3 * kTopTok * (BM + 8) * 2 +
         2 * (32 * cap + 1) * kPieceRefBytes;
}

static_assert(kTcsMaxLv >= REG_LV, "stack levels");
static_assert(MAX_STAGES <= kNBuf, "stage reuse is read off the leaf barriers");

// Stacked gate/up (see the streaming kernel): the up half of a tile's roots
// passes to the gate half through shared memory, 64 rows x WORDS words.
constexpr int XCH_BYTES = 64 * WORDS * 4;
__host__ __device__ inline int stages_for(int E, bool stacked = false) {
  const int lv = E > REG_LV ? E - REG_LV : 0;
  int n = (MAX_SMEM - 1024 - BAR_BYTES - lv * LV_BYTES - (stacked ? XCH_BYTES : 0)) / STAGE;
  if (n > MAX_STAGES) n = MAX_STAGES;
  return n & ~1;  // even: stage s is always filled by producer s % 2
}
__host__ __device__ inline int smem_for(int E, int ns, bool stacked = false) {
  const int lv = E > REG_LV ? E - REG_LV : 0;
  return 1024 + ns * STAGE + lv * LV_BYTES + BAR_BYTES + (stacked ? XCH_BYTES : 0);
}

struct Bars {
  uint64_t full[MAX_STAGES], accf[kNBuf], acce[kNBuf], fin;
  uint64_t xfull, xempty;  // stacked gate/up: the up half's roots are in the exchange buffer / have been read
  uint32_t tmem_slot;
  int abort;
  int last;  // folded trees: this CTA took its tree's last ticket
  int go;    // fused forward: the down block runs (nothing stopped before it)
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
  uint16_t* out0;   // direct mode: roots go to out_p[r * ldo + c]
  uint16_t* out1;
  long long ldo;
  int* status;
  long long spin;
  int stall;        // test only: the producers issue no loads
  int L;            // leaves per tree (G * 2^E)
  float* dump;      // leaf dump (DUMP instances): [np][R][C][L] FP32 leaves
  // Stacked gate/up (direct mode, one problem): a tile's 128 MMA rows are 64
  // rows of Wg (map tmW) over the same 64 rows of Wu (map tmW2), so that one
  // CTA holds both roots of every (row, token) of its tiles and writes
  // h = bf16(bf16(SiLU(gate)) * up) itself (gate and up too, to out0 / out1
  // where not null), with no pieces and no second kernel.  C counts the rows
  // of each weight; tiles are 64 rows.
  int stacked;
  uint16_t* hout;
  const uint16_t* silu;
  // Folded trees (aligned ranges, fold_n > 0): CTA b's range is one aligned
  // block of tree b / fold_n, its one piece in slot b * cap; the tree's last
  // CTA to finish (tickets[tree], counted up and reset to zero by that CTA)
  // folds the fold_n pieces into the root and stores it as in direct mode.
  int fold_n;
  int* tickets;
};

// First group of CTA b's range.  Direct mode deals whole tiles: segment
// boundaries only, so every tile's root is formed in one CTA.
__host__ __device__ __forceinline__ long long range_lo(long long b, long long W, long long P, int Q, bool direct) {
  return direct ? (b * (W / Q) / P) * Q : b * W / P;
}

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

// Barrier of the four epilogue warps alone (the other roles do not take part).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiWarps * 32) : "memory"); }

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
                                       uint64_t pol, int mn, const CUtensorMap* mW2 = nullptr) {
  if (mW2) {  // stacked: 64 rows of each weight (two boxes of 64 rows x 64 K)
    tma_load_2d_hint(dst, mW, k, t * (BM / 2), bar, pol);
    tma_load_2d_hint(dst + A_BYTES / 2, mW2, k, t * (BM / 2), bar, pol);
  } else if (mn) {
    tma_load_2d_hint(dst, mW, t * BM, k, bar, pol);
    tma_load_2d_hint(dst + A_BYTES / 2, mW, t * BM + BM / 2, k, bar, pol);
  } else {
    tma_load_2d_hint(dst, mW, k, t * BM, bar, pol);
  }
}

// The root of one bottom group, this thread's row and all tokens, from its
// GG leaves in TMEM buffers lc .. lc + GG - 1 of NB (taddr: the TMEM base
// plus the warp's lane quarter): a lone leaf rounded once, l0 + l1, or
// l0 + (l1 + l2).  DUMP: the leaves also go to the leaf dump, as leaves
// j0 .. j0 + GG - 1 of weight row crow.
template <int GG, bool DUMP, int NB = kNBuf>
__device__ __forceinline__ void group_root(uint32_t taddr, uint32_t lc, uint32_t (&root)[WORDS], float* dmp,
                                           long long crow, int R, int C, int L, int j0) {
  const uint32_t b0 = (uint32_t)((lc % NB) * BN), b1 = (uint32_t)(((lc + 1) % NB) * BN),
                 b2 = (uint32_t)(((lc + 2) % NB) * BN);
#pragma unroll
  for (int c = 0; c < BN / 16; ++c) {
    uint32_t v0[16];
    if constexpr (GG == 3) {
      uint32_t v1[16], v2[16], n12[8];
      tmem_ld16(taddr + b1 + 16 * c, v1);
      tmem_ld16(taddr + b2 + 16 * c, v2);
      tmem_wait_ld();
      if constexpr (DUMP) {
        dump_tokens(dmp, crow, 16 * c, R, C, L, j0 + 1, v1);
        dump_tokens(dmp, crow, 16 * c, R, C, L, j0 + 2, v2);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        n12[i] = pack_bf16x2_of(add_f32x2(f32x2(v1[2 * i], v1[2 * i + 1]), f32x2(v2[2 * i], v2[2 * i + 1])));
      tmem_ld16(taddr + b0 + 16 * c, v0);
      tmem_wait_ld();
      if constexpr (DUMP) dump_tokens(dmp, crow, 16 * c, R, C, L, j0, v0);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        root[8 * c + i] =
            pack_bf16x2_of(add_f32x2(f32x2(v0[2 * i], v0[2 * i + 1]), f32x2(n12[i] << 16, n12[i] & 0xFFFF0000u)));
    } else if constexpr (GG == 2) {
      uint32_t v1[16];
      tmem_ld16(taddr + b0 + 16 * c, v0);
      tmem_ld16(taddr + b1 + 16 * c, v1);
      tmem_wait_ld();
      if constexpr (DUMP) {
        dump_tokens(dmp, crow, 16 * c, R, C, L, j0, v0);
        dump_tokens(dmp, crow, 16 * c, R, C, L, j0 + 1, v1);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
        root[8 * c + i] = pack_bf16x2_of(add_f32x2(f32x2(v0[2 * i], v0[2 * i + 1]), f32x2(v1[2 * i], v1[2 * i + 1])));
    } else {
      tmem_ld16(taddr + b0 + 16 * c, v0);
      tmem_wait_ld();
      if constexpr (DUMP) dump_tokens(dmp, crow, 16 * c, R, C, L, j0, v0);
#pragma unroll
      for (int i = 0; i < 8; ++i) root[8 * c + i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
    }
  }
}

// Stacked gate/up, the tile's root (see TcsArgs): rows 0..63 hold gate,
// rows 64..127 up, of weight rows 64 t + (row mod 64).  The up half hands its
// roots over in shared memory (xch) and stores up where kept; the gate half
// forms h = bf16(bf16(SiLU(gate)) * up) and stores it, and gate where kept.
// xk counts the CTA's exchanges (the phase of xfull / xempty).  Every wait is
// bounded; false when one ran out.
__device__ __forceinline__ bool stacked_store(const TcsArgs& a, Bars* bars, uint32_t* xch, uint32_t xk, long long t,
                                              int row, int lane, const uint32_t (&root)[WORDS], long long limit,
                                              volatile int* abort_flag) {
  const long long c = t * (BM / 2) + (row & (BM / 2 - 1));
  const uint32_t ph = xk & 1u;
  bool ok = true;
  if (row >= BM / 2) {
    if (!wait_or_abort(&bars->xempty, ph ^ 1u, limit, abort_flag, a.status)) ok = false;
    if (ok) {
#pragma unroll
      for (int i = 0; i < WORDS; ++i) xch[i * (BM / 2) + (row - BM / 2)] = root[i];
      if (a.out1 && c < a.C)
#pragma unroll
        for (int i = 0; i < BN; ++i)
          if (i < a.R) a.out1[i * a.ldo + c] = (uint16_t)(root[i >> 1] >> (16 * (i & 1)));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->xfull);
  } else {
    if (!wait_or_abort(&bars->xfull, ph, limit, abort_flag, a.status)) ok = false;
    if (ok && c < a.C) {
#pragma unroll
      for (int i = 0; i < WORDS; ++i) {
        const uint32_t g2 = root[i], u2 = xch[i * (BM / 2) + row];
        const float h0 = __fmul_rn(bf2f(__ldg(a.silu + (g2 & 0xFFFFu))), __uint_as_float(u2 << 16));
        const float h1 = __fmul_rn(bf2f(__ldg(a.silu + (g2 >> 16))), __uint_as_float(u2 & 0xFFFF0000u));
        if (2 * i < a.R) a.hout[(2 * i) * a.ldo + c] = f2bf(h0);
        if (2 * i + 1 < a.R) a.hout[(2 * i + 1) * a.ldo + c] = f2bf(h1);
        if (a.out0) {
          if (2 * i < a.R) a.out0[(2 * i) * a.ldo + c] = (uint16_t)(g2 & 0xFFFFu);
          if (2 * i + 1 < a.R) a.out0[(2 * i + 1) * a.ldo + c] = (uint16_t)(g2 >> 16);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->xempty);
  }
  return ok;
}

// The fold of a tree's pieces by its last CTA.  src: the tree's first
// piece (n pieces, n a power of two, at most 8, pstride 16-byte units apart;
// the aligned blocks of the tree, left to right).  Each epilogue warp copies
// its 32 rows of every piece (2 KB per piece, contiguous) into shared memory
// at buf in one batch of copies, rows of 64 bytes whose four 16-byte
// quarters are rotated by bits 1-2 of the row, so that both the copies and
// the per-row reads below are free of bank conflicts.  Then each thread folds
// its row, a quarter at a time: the balanced tree over the n pieces.  Token
// i < R of the root goes to o[i * ldo]; o is null beyond the weight rows.
__device__ __forceinline__ void fold_pieces(const uint4* src, long long pstride, int n, unsigned char* buf, int ew,
                                            int lane, uint16_t* o, long long ldo, int R) {
  const int row = ew * 32 + lane;
  const uint32_t b0 = smem_u32(buf);
#pragma unroll 1
  for (int j = 0; j < n; ++j)
#pragma unroll
    for (int i = 0; i < WORDS / 4; ++i) {
      const int u = i * 32 + lane, r = ew * 32 + (u >> 2), q = u & 3;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                       b0 + (uint32_t)((j * BM + r) * 64 + ((q ^ ((r >> 1) & 3)) * 16))),
                   "l"(src + j * pstride + ew * 128 + u)
                   : "memory");
    }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
  __syncwarp();  // the warp's rows were copied by all its lanes
  uint32_t root[WORDS];
#pragma unroll
  for (int q = 0; q < WORDS / 4; ++q) {
    const unsigned char* at = buf + row * 64 + ((q ^ ((row >> 1) & 3)) * 16);
    uint4 v[kTcsFoldMax];
#pragma unroll
    for (int j = 0; j < kTcsFoldMax; ++j)
      if (j < n) v[j] = *reinterpret_cast<const uint4*>(at + j * BM * 64);
#pragma unroll
    for (int w = 2; w <= kTcsFoldMax; w *= 2)  // level by level: node j of the next level = v[2j] + v[2j+1]
#pragma unroll
      for (int j = 0; j < kTcsFoldMax / w; ++j)
        if (j < n / w)
          v[j] = make_uint4(add_bf16x2(v[2 * j].x, v[2 * j + 1].x), add_bf16x2(v[2 * j].y, v[2 * j + 1].y),
                            add_bf16x2(v[2 * j].z, v[2 * j + 1].z), add_bf16x2(v[2 * j].w, v[2 * j + 1].w));
    root[4 * q] = v[0].x;
    root[4 * q + 1] = v[0].y;
    root[4 * q + 2] = v[0].z;
    root[4 * q + 3] = v[0].w;
  }
  if (o)
#pragma unroll
    for (int i = 0; i < BN; ++i)
      if (i < R) o[i * ldo] = (uint16_t)(root[i >> 1] >> (16 * (i & 1)));
}

// Folded trees, after this CTA's piece of tree `tree` is written: the
// CTA takes the tree's ticket, and the last of its CTAs folds the tree's
// fold_n pieces (slots tree * fold_n .. tree * fold_n + fold_n - 1) into the
// root and stores it.  Every epilogue warp reaches the two barriers, whatever
// happened: a warp that stopped early has set the abort flag, and a CTA that
// stopped takes no ticket (its tree stays unfinished, which the status word
// reports).  One thread orders the CTA's piece rows (after the barrier)
// before its ticket, and the last CTA's reads after the tickets of the
// others, with device-scope fences.  The pipeline stages must be idle (every
// load landed and every MMA completed) and hold fold_n pieces.
__device__ __forceinline__ void finish_tree(const TcsArgs& a, int tree, unsigned char* stages, Bars* bars,
                                            volatile int* abort_flag, int quarter, int lane) {
  epi_sync();
  if (threadIdx.x == kEpi0 * 32) {
    int last = 0;
    if (!*abort_flag) {
      __threadfence();
      last = atomicAdd(a.tickets + tree, 1) == a.fold_n - 1;
      if (last) {
        a.tickets[tree] = 0;  // no other CTA of this launch takes it again
        __threadfence();
      }
    }
    bars->last = last;
  }
  epi_sync();
  if (bars->last) {
    const int row = quarter * 32 + lane;
    const int per = a.np * a.ns, rem = tree % per;
    const int c = (tree / per) * BM + row;
    fold_pieces(reinterpret_cast<const uint4*>(a.slots + (size_t)tree * a.fold_n * a.cap * PIECE),
                (long long)a.cap * (PIECE / 8), a.fold_n, stages, quarter, lane,
                c < a.C ? ((rem % a.np) ? a.out1 : a.out0) + (rem / a.np) * a.oss + c : nullptr, a.ldo, a.R);
  }
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
  uint32_t* xch = reinterpret_cast<uint32_t*>(smem + NS * STAGE + slv * LV_BYTES + BAR_BYTES);  // [word][64 rows]
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Q = 1 << a.E;
  const bool direct = a.slots == nullptr;
  const long long w0 = range_lo(blockIdx.x, a.W, gridDim.x, Q, direct);
  const long long w1 = range_lo(blockIdx.x + 1ll, a.W, gridDim.x, Q, direct);
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
    mbar_init(&bars->xfull, 2);   // the two warps of the up half (lanes 64..127)
    mbar_init(&bars->xempty, 2);  // the two warps of the gate half (lanes 0..63)
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
            load_w(stages + it * STAGE, mW, k0 + j * BK, g.t, &bars->full[it], pol, a.w_mn, a.stacked ? &tmW2 : nullptr);
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
            load_w(dst, mW, k0 + j * BK, g.t, &bars->full[st], pol, a.w_mn, a.stacked ? &tmW2 : nullptr);
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
    // epilogue and the producers).  No stage can fill before the previous
    // kernel has completed (the token tiles wait for it), so this warp waits
    // for it too, in the hardware, instead of polling barriers meanwhile:
    // the previous kernel's last CTAs may share this SM, and the polls would
    // take their shared-memory and issue bandwidth.
    grid_dep_wait();
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
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int row = quarter * 32 + lane;
    grid_dep_wait();  // its stores may overwrite what the previous kernel reads
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    uint16_t* const myslots = direct ? nullptr : a.slots + (size_t)blockIdx.x * a.cap * PIECE;
    uint32_t lc = 0;  // leaves consumed (kNBuf is a power of two)
    int np_out = 0;  // pieces written
    uint32_t xk = 0;  // stacked: tiles exchanged (the phase of xfull / xempty)
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
        // The group root; leaf dump: this thread's weight row of the tile.
        uint32_t root[WORDS];
        const Seg sg = seg_of(s, a.np, a.ns);
        group_root<GG, DUMP>(tmem + lane_addr, lc, root,
                             DUMP ? a.dump + (size_t)sg.pb * a.R * a.C * a.L : nullptr,
                             (long long)sg.t * BM + row, a.R, a.C, a.L, q * GG);
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
        bool tile_root = false;
#pragma unroll
        for (int m = 0; m <= kTcsMaxLv; ++m) {
          if (live) {
            if (m == a.E) {  // the whole tile: its root (stored below, outside the unrolled loop)
              if (direct) tile_root = true;
              else emit_piece(myslots, np_out, a.cap, row, root);
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
        if (tile_root) {
          if (a.stacked) {
            if (!stacked_store(a, bars, xch, xk, sg.t, row, lane, root, limit, abort_flag)) ok = false;
            ++xk;
          } else {
            const long long c = (long long)sg.t * BM + row;
            uint16_t* o = (sg.pb ? a.out1 : a.out0) + sg.q * a.oss;
            if (c < a.C)
#pragma unroll
              for (int i = 0; i < BN; ++i)
                if (i < a.R) o[i * a.ldo + c] = (uint16_t)(root[i >> 1] >> (16 * (i & 1)));
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
    // Folded trees: this CTA's piece is written; the tree's last CTA folds
    // all of them (every epilogue warp takes part, whatever happened).
    if (a.fold_n > 0) finish_tree(a, (int)(w0 / Q), stages, bars, abort_flag, quarter, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Fused decode forward: one launch for gate/up, SiLU * up and down.
// ---------------------------------------------------------------------------
// Unit A is one stacked gate/up tile (64 rows of Wg over the same 64 rows of
// Wu, the whole K = H; the gate half writes h, as in the stacked kernel),
// unit B one aligned block of groups of a down-projection tree (one piece;
// the tree's last CTA folds, as with folded trees).  CTA b takes tile b
// (b < nA) and then block (b - nA) mod P (when below nB).  A block's K range
// of I is h's columns of per_range consecutive tiles; before its first token
// tile each producer warp of the block waits until those tiles have been
// counted in ready[range] (each tile's gate half counts itself once its h is
// stored), and the last of the range's waiters resets both counters.  No unit
// A waits on a unit B, so every wait ends once the tiles it needs run.
// Pending levels of a unit's fold kept in registers: two, so that the
// epilogue fits its 128 registers.  The levels above them live in TMEM,
// 16 columns each, after kFwdNBuf leaf buffers (six, not eight: the room
// that the shared-memory stack would take goes to a fifth pipeline stage).
constexpr int kFwdRegLv = 2;
constexpr int kFwdNBuf = 6;
constexpr int kFwdStackCol = kFwdNBuf * BN;
constexpr int kFwdMaxLevels = (kTmemCols - kFwdStackCol) / WORDS + kFwdRegLv;  // deepest unit fold

struct FwdArgs {
  TcsArgs A, B;    // unit A geometry (stacked, direct), unit B geometry (folded trees)
  int nA, nB;      // gate/up tiles, down blocks
  int bG;          // groups per down block
  int per_range;   // gate/up tiles per down range (= bG * leaves per group)
  int waiters;     // producer warps that wait on one range (two per down tree)
  int* ready;      // [kTcsRanges] tiles counted, then [kTcsRanges] waiters passed
};

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Group root v (group q of a complete aligned block of 2^e groups, counted
// from the block's start) into the block's pending stack (levels below RL in
// registers, level m >= RL in TMEM columns tstk + WORDS (m - RL) of this
// thread's lane); true when v is then the block's root.
template <int RL>
__device__ __forceinline__ bool fold_push(uint32_t (&v)[WORDS], int q, int e, uint32_t (&reg_lv)[RL][WORDS],
                                          uint32_t tstk) {
  bool root = false, live = true;
#pragma unroll
  for (int m = 0; m <= kTcsMaxLv; ++m) {
    if (live) {
      if (m == e) {
        root = true;
        live = false;
      } else if ((q >> m) & 1) {
        if (m < RL) {
#pragma unroll
          for (int i = 0; i < WORDS; ++i) v[i] = add_bf16x2(reg_lv[m < RL ? m : 0][i], v[i]);
        } else {
          uint32_t left[WORDS];
          tmem_ld16(tstk + (uint32_t)(WORDS * (m - RL)), left);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < WORDS; ++i) v[i] = add_bf16x2(left[i], v[i]);
        }
      } else {
        if (m < RL) {
#pragma unroll
          for (int i = 0; i < WORDS; ++i) reg_lv[m < RL ? m : 0][i] = v[i];
        } else {
          tmem_st16(tstk + (uint32_t)(WORDS * (m - RL)), v);
          tmem_wait_st();
        }
        live = false;
      }
    }
  }
  return root;
}

// The epilogue's walk over one unit: 2^e groups of G leaves each (TMEM
// buffers from lc on), folded into the unit's root (root is the working
// value: each group's root, pushed or merged, and the unit's root at the
// end).  False when a wait ran out (root unfinished).
template <int G>
__device__ __forceinline__ bool unit_root(uint32_t taddr, uint32_t& lc, int e, uint32_t (&root)[WORDS], int lane,
                                          Bars* bars, long long limit, volatile int* abort_flag, int* status) {
  uint32_t reg_lv[kFwdRegLv][WORDS];
  bool ok = true;
#pragma unroll 1
  for (int q = 0; q < (1 << e); ++q) {
    for (int g = 0; g < G; ++g)
      if (!wait_or_abort(&bars->accf[(lc + g) % kFwdNBuf], (uint32_t)(((lc + g) / kFwdNBuf) & 1), limit, abort_flag,
                         status))
        ok = false;
    if (__any_sync(0xffffffffu, !ok)) return false;
    tc_fence_after();
    group_root<G, false, kFwdNBuf>(taddr, lc, root, nullptr, 0, 0, 0, 0, 0);
    tc_fence_before();
    __syncwarp();
    if (lane == 0)
      for (int g = 0; g < G; ++g) mbar_arrive(&bars->acce[(lc + g) % kFwdNBuf]);
    lc += G;
    // After the last group, root is the unit's root.
    fold_push<kFwdRegLv>(root, q, e, reg_lv, taddr + (uint32_t)kFwdStackCol);
  }
  return true;
}

template <int GA, int GB>
__global__ void __maxnreg__(128)
    k_tcs_fwd(const __grid_constant__ CUtensorMap tmWg, const __grid_constant__ CUtensorMap tmWu,
              const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmWd,
              const __grid_constant__ CUtensorMap tmH, const __grid_constant__ FwdArgs f) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const TcsArgs& A = f.A;
  const TcsArgs& B = f.B;
  const int NS = A.nstage;
  unsigned char* stages = smem;
  Bars* bars = reinterpret_cast<Bars*>(smem + NS * STAGE);
  uint32_t* xch = reinterpret_cast<uint32_t*>(smem + NS * STAGE + BAR_BYTES);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = (int)gridDim.x;
  const bool hasA = (int)blockIdx.x < f.nA;
  const int jB = fwd_block_of((int)blockIdx.x, f.nA, P);
  const bool hasB = jB < f.nB;
  const int nLA = hasA ? (GA << A.E) : 0;  // leaves of unit A (the whole K = H)
  const int nLB = hasB ? f.bG * GB : 0;     // leaves of unit B
  const int treeB = hasB ? fwd_tree_of(jB, B.fold_n) : 0, rangeB = hasB ? fwd_range_of(jB, B.fold_n) : 0;
  const int kB0 = rangeB * f.bG * GB;       // unit B's first leaf along K = I
  const long long limit = A.spin > 0 ? A.spin : kDefaultSpin;
  if (__syncthreads_or(A.status != nullptr && *(volatile int*)A.status != 0)) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bars->full[s], 1);
    for (int b = 0; b < kNBuf; ++b) {
      mbar_init(&bars->accf[b], 1);
      mbar_init(&bars->acce[b], kEpiWarps);
    }
    mbar_init(&bars->fin, 1);
    mbar_init(&bars->xfull, 2);
    mbar_init(&bars->xempty, 2);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp < kProd && lane == 0) {
    if (warp == 0) {
      prefetch_tmap(&tmWg);
      prefetch_tmap(&tmWu);
      prefetch_tmap(&tmWd);
    } else {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmH);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  grid_dep_launch();

  if (warp < kProd) {
    // ---------------- TMA producers: leaf it goes to producer it % kProd ----------------
    // Leaves 0 .. nLA-1 are unit A's (K positions 64 it of H), then unit B's
    // (K positions 64 (kB0 + it - nLA) of I).
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    const long long nL = nLA + nLB;
    auto load_weights = [&](long long it, unsigned char* dst, uint64_t* bar) {
      if (it < nLA) load_w(dst, &tmWg, (int)(it * BK), (int)blockIdx.x, bar, pol, 0, &tmWu);
      else load_w(dst, &tmWd, (int)((kB0 + it - nLA) * BK), treeB, bar, pol, 0);
    };
    // Before the previous kernel has finished: weight tiles of the first NS leaves.
    if (!A.stall)
      for (long long it = warp; it < nL && it < NS; it += kProd) {
        if (elect_one()) {
          mbar_arrive_expect_tx(&bars->full[it], (uint32_t)STAGE);
          load_weights(it, stages + it * STAGE, &bars->full[it]);
        }
        __syncwarp();
      }
    grid_dep_wait();
    // Leaf i uses stage i % NS, free once leaf i - NS has been committed.
    // This warp's leaves below wmax have their weight tiles issued, those
    // below xdone their token tiles too.
    bool ok = true;
    long long wmax = warp, xdone = warp;
    for (long long i = warp; i < nL && i < NS; i += kProd) wmax = i + kProd;  // the prefetch above
    auto stage_free = [&](long long i) -> bool {
      if (i < NS) return true;
      const long long v = i - NS;
      const bool wok =
          wait_or_abort(&bars->accf[v % kFwdNBuf], (uint32_t)((v / kFwdNBuf) & 1), limit, abort_flag, A.status);
      return __all_sync(0xffffffffu, wok) != 0;
    };
    auto issue_w = [&](long long i) {
      if (!A.stall && elect_one()) {
        mbar_arrive_expect_tx(&bars->full[i % NS], (uint32_t)STAGE);
        load_weights(i, stages + (i % NS) * STAGE, &bars->full[i % NS]);
      }
      __syncwarp();
      wmax = i + kProd;
    };
    auto issue_x = [&](long long i) {
      if (!A.stall && elect_one()) {
        unsigned char* dst = stages + (i % NS) * STAGE + A_BYTES;
        if (i < nLA) tma_load_2d(dst, &tmX, (int)(i * BK), 0, &bars->full[i % NS]);
        else tma_load_2d(dst, &tmH, (int)((kB0 + i - nLA) * BK), 0, &bars->full[i % NS]);
      }
      __syncwarp();
      xdone = i + kProd;
    };
    bool waited = false;
    for (long long it = warp; it < nL && ok; it += kProd) {
      if (it >= nLA && !waited) {
        // Unit B: first the weight tiles of its leaves within one ring of its
        // start (their stages free up as unit A drains), then the wait for
        // h's columns, which are per_range gate/up tiles of this launch.
        for (long long j = it; j < nL && j < nLA + NS && ok; j += kProd)
          if (j >= wmax) {
            if (stage_free(j)) issue_w(j);
            else ok = false;
          }
        if (!ok) break;
        bool rok = true;
        if (lane == 0) {
          long long i = 0;
          for (; i < limit; ++i) {
            if (ld_acquire(f.ready + rangeB) >= f.per_range) break;
            if ((i & 255) == 255 && *abort_flag) {
              i = limit;
              break;
            }
            __nanosleep(64);
          }
          if (i >= limit) {
            rok = false;
            *abort_flag = 1;
            if (A.status) atomicExch(A.status, (int)DETFFN_ERR_TIMEOUT);
          } else {
            fence_proxy_async_global();  // the TMA loads below read what generic stores wrote
            if (atomicAdd(f.ready + kTcsRanges + rangeB, 1) == f.waiters - 1) {
              f.ready[rangeB] = 0;  // every waiter of this launch has passed
              f.ready[kTcsRanges + rangeB] = 0;
            }
          }
        }
        waited = true;
        if (!__shfl_sync(0xffffffffu, rok, 0)) {
          ok = false;
          break;
        }
      }
      if (it >= wmax) {
        if (!stage_free(it)) {
          ok = false;
          break;
        }
        issue_w(it);
      }
      issue_x(it);
    }
    // After a stop, the stages whose weight tiles went out without their
    // token tiles get those too (in-bounds reads), so that each completes.
    // Then drain: this producer's loads have landed (long bound).
    if (!A.stall) {
      for (long long i = xdone; i < wmax; i += kProd) issue_x(i);
      if (lane == 0)
        for (long long i = (wmax > NS ? wmax - NS : 0); i < wmax; ++i)
          if ((int)(i % kProd) == warp) mbar_wait(&bars->full[i % NS], (uint32_t)((i / NS) & 1), kDefaultSpin, nullptr);
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer: every leaf of both units, in order ----------------
    grid_dep_wait();
    const uint32_t idesc = idesc_bf16(BM, BN);
    const long long nleaf = nLA + nLB;
    Ring rs, rb;
    bool ok = true;
    for (long long n = 0; n < nleaf && ok; ++n, rs.next(NS), rb.next(kFwdNBuf)) {
      const int st = rs.slot, b = rb.slot;
      const bool wok = wait_or_abort(&bars->acce[b], rb.phase ^ 1u, limit, abort_flag, A.status) &&
                       wait_or_abort(&bars->full[st], rs.phase, limit, abort_flag, A.status);
      if (!__all_sync(0xffffffffu, wok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t da = smem_desc_sw128(stages + st * STAGE);
      const uint64_t db = smem_desc_sw128(stages + st * STAGE + A_BYTES);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_bf16(tmem + (uint32_t)(b * BN), da + 2u * kk, db + 2 * kk, idesc, kk > 0 ? 1u : 0u);
        tc_commit(&bars->accf[b]);
      }
      __syncwarp();
    }
    if (elect_one()) tc_commit(&bars->fin);
    __syncwarp();
    if (lane == 0) mbar_wait(&bars->fin, 0, kDefaultSpin, nullptr);
  } else {
    // ---------------- epilogue ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    grid_dep_wait();
    const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
    uint32_t lc = 0;
    uint32_t root[WORDS];
    if (hasA) {
      // The tile's root, then h (and the saves) through the stacked exchange.
      bool ok = unit_root<GA>(taddr, lc, A.E, root, lane, bars, limit, abort_flag, A.status);
      if (ok) ok = stacked_store(A, bars, xch, 0, blockIdx.x, row, lane, root, limit, abort_flag);
      // The gate half (rows 0..63, two warps) stored h: count the tile in
      // its range once both warps are done (both always reach the barrier).
      if (row < BM / 2) {
        asm volatile("bar.sync 2, %0;" ::"n"(BM / 2) : "memory");
        if (row == 0 && !*abort_flag) {
          fence_proxy_async_global();
          __threadfence();
          atomicAdd(f.ready + fwd_tile_range((int)blockIdx.x, f.per_range), 1);
        }
      }
    }
    if (hasB) {
      // Unit B runs unless something stopped (one decision for all four warps).
      epi_sync();
      if (threadIdx.x == kEpi0 * 32) bars->go = !*abort_flag;
      epi_sync();
      if (bars->go &&
          unit_root<GB>(taddr, lc, B.E - hibit((unsigned)B.fold_n), root, lane, bars, limit, abort_flag, B.status)) {
        int n = 0;
        emit_piece(B.slots + (size_t)jB * B.cap * PIECE, n, B.cap, row, root);
      }
      finish_tree(B, treeB, stages, bars, abort_flag, quarter, lane);
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

struct TcsTopArgs {
  int R, C, E, np, ns;  // ns: K shards per problem (segments as in the streaming kernel)
  long long oss;        // element offset between consecutive shards' outputs
  long long W;
  int P, cap;
  const uint16_t* slots;
  uint16_t* out0;   // problem 0 result (gate when fused), or null when fused and not kept
  uint16_t* out1;   // problem 1 result (up when fused), or null
  long long ldo;    // row stride of out0, out1 and h (elements)
  uint16_t* h;      // fused: h = bf16(SiLU(gate)) * up, rounded to BF16; null: plain
  const uint16_t* silu;
  const int* status;
};

struct PieceRef {
  int slot;  // b * cap + j
  int at;    // level m (bits 0..7), left siblings it merges with (bits 8..15), and whether the
             // result is the root (bit 16): the fold, the same for every element, worked out once
};
static_assert(sizeof(PieceRef) == kPieceRefBytes, "piece list entries: shared-memory sizes assume 8 bytes");

// Lists, in order, the pieces of segment s that CTAs [b_base, b_base + 32)
// wrote: one lane per CTA, placed by a warp scan.  Returns the count.
__device__ int list_pieces(const TcsTopArgs& a, long long s, long long b_base, PieceRef* list, int lane) {
  const int Q = 1 << a.E;
  const long long ws = s * Q, we = ws + Q;
  const long long b = b_base + lane;
  int cnt = 0;
  long long lo = 0, hi = 0, blo = 0;
  if (b < a.P) {
    blo = b * a.W / a.P;
    const long long bhi = (b + 1) * a.W / a.P;
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
    // Pieces CTA b wrote for its earlier segments: its first (partial) one and whole ones.
    const long long s0 = blo / Q;
    int j = 0;
    if (s0 < s) j = count_pieces((int)(blo - s0 * Q), Q) + (int)(s - s0 - 1);
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

// Fold state of one segment for this thread's (row, 8 tokens): the pieces,
// left to right, meet their left siblings on a stack in this thread's column
// of shared memory.
struct Fold {
  uint4* stk;     // level l at stk[l * BM]
  uint4 root;
  long long b;    // first CTA of the current list batch
  int n;          // pieces in the current list batch
};

__device__ __forceinline__ uint4 add4(uint4 l, uint4 r) {
  return make_uint4(add_bf16x2(l.x, r.x), add_bf16x2(l.y, r.y), add_bf16x2(l.z, r.z), add_bf16x2(l.w, r.w));
}

// The first CTA whose range holds a group of segment s.
__device__ __forceinline__ long long first_cta(const TcsTopArgs& a, long long s) {
  const long long ws = s * (1ll << a.E);
  long long b = ws * a.P / a.W;
  if ((b + 1) * a.W / a.P <= ws) ++b;  // CTA b ends where segment s begins
  return b;
}
__device__ __forceinline__ bool more_ctas(const TcsTopArgs& a, long long s, long long b) {
  return b < a.P && b * a.W / a.P < (s + 1) * (1ll << a.E);
}

// Folds one piece (its fold code from the list) into the stack.
__device__ __forceinline__ void fold_piece(int code, uint4 cur, Fold& f) {
  const int m = code & 0xFF, k = (code >> 8) & 0xFF;
#pragma unroll 1
  for (int i = 0; i < k; ++i) cur = add4(f.stk[(m + i) * BM], cur);
  if (code >> 16) f.root = cur;
  else f.stk[(m + k) * BM] = cur;
}

// Copies (cp.async, 16 bytes per thread: 8 tokens of one row) this
// thread's part of pieces k0 .. min(k0 + CH, n) - 1 of the list into its
// column of buf.
template <int CH>
__device__ __forceinline__ void stage_pieces(const TcsTopArgs& a, const PieceRef* list, int k0, int n, int row,
                                             int quad, uint4* buf) {
  const int kend = n < k0 + CH ? n : k0 + CH;
#pragma unroll 1
  for (int k = k0; k < kend; ++k) {
    const uint16_t* src = a.slots + (size_t)list[k].slot * PIECE + row * BN + quad * kTopTok;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(buf + (k - k0) * BM + row)), "l"(src)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void staged_wait() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int CH>
__device__ __forceinline__ void fold_staged(const TcsTopArgs& a, const PieceRef* list, int k0, int n,
                                            const uint4* buf, Fold& f) {
  const int kend = n < k0 + CH ? n : k0 + CH;
#pragma unroll 1
  for (int k = k0; k < kend; ++k) fold_piece(list[k].at, buf[(k - k0) * BM + threadIdx.x], f);
}

// Everything of segment s after its first CH pieces (already staged and
// folded by the caller): the rest of that list, then further list batches.
template <int CH>
__device__ void fold_rest(const TcsTopArgs& a, long long s, PieceRef* list, int row, int quad, bool active,
                          uint4* buf, Fold& f) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 1
  for (int k0 = CH; k0 < f.n; k0 += CH) {
    if (active) {
      stage_pieces<CH>(a, list, k0, f.n, row, quad, buf);
      staged_wait();
      fold_staged<CH>(a, list, k0, f.n, buf, f);
    }
  }
#pragma unroll 1
  for (f.b += 32; more_ctas(a, s, f.b); f.b += 32) {
    __syncthreads();  // the previous batch's list is no longer read
    if (warp == 0) {
      const int n = list_pieces(a, s, f.b, list, lane);
      if (lane == 0) list[32 * a.cap].slot = n;
    }
    __syncthreads();
    f.n = list[32 * a.cap].slot;
#pragma unroll 1
    for (int k0 = 0; k0 < f.n; k0 += CH) {
      if (active) {
        stage_pieces<CH>(a, list, k0, f.n, row, quad, buf);
        staged_wait();
        fold_staged<CH>(a, list, k0, f.n, buf, f);
      }
    }
  }
}

// Writes a [kTopTok tokens][128 rows] tile held in shared memory to
// out[r * ldo + c] for r in [r0, min(r0 + kTopTok, R)), c in [c0, min(c0 + 128, C)).
__device__ __forceinline__ void store_tile(const uint16_t* tile, uint16_t* out, long long ldo, int R, int r0,
                                           long long c0, long long C) {
  static_assert(kTopTok * BM == 8 * kTopThreads, "one 16-byte store per thread");
  const int tok = threadIdx.x >> 4, c8 = (threadIdx.x & 15) * 8;
  if (r0 + tok >= R) return;
  const long long c = c0 + c8;
  uint16_t* o = out + (r0 + tok) * ldo + c;
  const uint16_t* src = tile + tok * (BM + 8) + c8;
  if (c + 8 <= C && ((uintptr_t)o & 15u) == 0) {
    *reinterpret_cast<uint4*>(o) = *reinterpret_cast<const uint4*>(src);
  } else {
    for (int i = 0; i < 8; ++i)
      if (c + i < C) o[i] = src[i];
  }
}

// Token t of this thread's 8 (word t / 2 of v, low half first) to tile[t][row].
__device__ __forceinline__ void put_tile(uint16_t* tile, int row, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    tile[(2 * i) * (BM + 8) + row] = (uint16_t)(w[i] & 0xFFFFu);
    tile[(2 * i + 1) * (BM + 8) + row] = (uint16_t)(w[i] >> 16);
  }
}

// Plain (FUSED false): CTA (s, y) folds segment s for tokens
// kTopTok * y .. kTopTok * y + kTopTok - 1.  Fused (np == 2): CTA (t, y) folds
// gate (segment 2t) and up (segment 2t+1) and forms h = bf16(SiLU(gate)) * up,
// rounded to BF16.  Each thread owns one row and 8 tokens (a 16-byte quarter
// of a piece row); the pieces are staged in shared memory (up to CH per
// segment in flight) and folded from there.  Launched as a programmatic
// dependent of the streaming kernel: the piece lists (arithmetic only) are
// built before waiting for its results.
template <bool FUSED>
__global__ void __launch_bounds__(kTopThreads) k_tcs_top(const TcsTopArgs a) {
  constexpr int NSEG = FUSED ? 2 : 1;
  constexpr int CH = top_chunk(FUSED);
  extern __shared__ __align__(16) unsigned char top_sm[];
  uint4* bufs = reinterpret_cast<uint4*>(top_sm);        // NSEG x [CH][BM]
  uint4* stacks = bufs + NSEG * CH * BM;                  // NSEG x [E][BM]
  uint16_t* tiles = reinterpret_cast<uint16_t*>(stacks + NSEG * a.E * BM);  // 3 x [kTopTok][BM + 8]
  PieceRef* lists = reinterpret_cast<PieceRef*>(tiles + 3 * kTopTok * (BM + 8));
  const int row = threadIdx.x, quad = blockIdx.y;
  const bool active = kTopTok * quad < a.R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long s0 = FUSED ? 2ll * blockIdx.x : (long long)blockIdx.x;
  const int stride = 32 * a.cap + 1;  // list entries per segment (the last holds the count)
  Fold f[NSEG];
  if (warp < NSEG) {
    PieceRef* list = lists + warp * stride;
    const int n = list_pieces(a, s0 + warp, first_cta(a, s0 + warp), list, lane);
    if (lane == 0) list[32 * a.cap].slot = n;
  }
  grid_dep_launch();
  __syncthreads();
  grid_dep_wait();  // the streaming kernel's pieces are complete and visible
  // A bounded wait of the streaming kernel (or of an earlier launch) ran out:
  // the pieces are unfinished, so nothing is folded or stored.
  if (__syncthreads_or(a.status != nullptr && *(volatile int*)a.status != 0)) return;
#pragma unroll
  for (int g = 0; g < NSEG; ++g) {
    f[g].b = first_cta(a, s0 + g);
    f[g].n = lists[g * stride + 32 * a.cap].slot;
    f[g].root = make_uint4(0, 0, 0, 0);
    f[g].stk = stacks + (g * a.E) * BM + row;
    if (active) stage_pieces<CH>(a, lists + g * stride, 0, f[g].n, row, quad, bufs + g * CH * BM);
  }
  staged_wait();
#pragma unroll
  for (int g = 0; g < NSEG; ++g) {
    if (active) fold_staged<CH>(a, lists + g * stride, 0, f[g].n, bufs + g * CH * BM, f[g]);
    fold_rest<CH>(a, s0 + g, lists + g * stride, row, quad, active, bufs + g * CH * BM, f[g]);
  }
  const int r0 = kTopTok * quad;
  if constexpr (!FUSED) {
    const Seg sg = seg_of(s0, a.np, a.ns);
    put_tile(tiles, row, f[0].root);
    __syncthreads();
    store_tile(tiles, (sg.pb ? a.out1 : a.out0) + sg.q * a.oss, a.ldo, a.R, r0, (long long)sg.t * BM, a.C);
  } else {
    const int t = blockIdx.x;
    const uint32_t gw[4] = {f[0].root.x, f[0].root.y, f[0].root.z, f[0].root.w};
    const uint32_t uw[4] = {f[1].root.x, f[1].root.y, f[1].root.z, f[1].root.w};
    uint32_t hw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float h0 = __fmul_rn(bf2f(__ldg(a.silu + (gw[i] & 0xFFFFu))), __uint_as_float(uw[i] << 16));
      const float h1 = __fmul_rn(bf2f(__ldg(a.silu + (gw[i] >> 16))), __uint_as_float(uw[i] & 0xFFFF0000u));
      hw[i] = (uint32_t)f2bf(h0) | ((uint32_t)f2bf(h1) << 16);
    }
    constexpr int TILE = kTopTok * (BM + 8);
    put_tile(tiles, row, make_uint4(hw[0], hw[1], hw[2], hw[3]));
    if (a.out0) put_tile(tiles + TILE, row, f[0].root);
    if (a.out1) put_tile(tiles + 2 * TILE, row, f[1].root);
    __syncthreads();
    store_tile(tiles, a.h, a.ldo, a.R, r0, (long long)t * BM, a.C);
    if (a.out0) store_tile(tiles + TILE, a.out0, a.ldo, a.R, r0, (long long)t * BM, a.C);
    if (a.out1) store_tile(tiles + 2 * TILE, a.out1, a.ldo, a.R, r0, (long long)t * BM, a.C);
  }
}

}  // namespace
}  // namespace detffn

namespace detffn {

bool tcs_plan(long long R, long long C, long long K, int np, int max_ctas, bool direct, TcsPlan* p, int ns,
              bool whole_ok) {
  if (R < 1 || R > BN || C < 1 || K < 1 || np < 1 || np > 2 || max_ctas < 1) return false;
  if (ns < 1 || ns > kTcsMaxShards || (ns > 1 && K % BK != 0)) return false;
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
  r.T = (int)((C + BM - 1) / BM);
  const int Q = 1 << E;
  r.W = (long long)np * ns * r.T * Q;
  const long long units = direct ? (long long)np * ns * r.T : r.W;
  r.P = (int)(max_ctas < units ? max_ctas : units);
  if (!direct) {
    // Equal, aligned ranges: the smallest power of two B of groups per CTA
    // with W / B <= max_ctas.  When B divides a tile's 2^E groups, every
    // range is one aligned block -- one piece, a node of the canonical tree
    // -- so a tile's fold takes 2^E / B pieces.  When B is a multiple of
    // 2^E, every range is B / 2^E whole tiles: direct, and balanced.
    long long B = 1;
    while (r.W / B > max_ctas) B <<= 1;
    if (B >= Q && whole_ok) {
      direct = true;
      r.P = (int)(r.W / B);
    } else if (B <= Q) {
      r.P = (int)(r.W / B);
      if (Q / B <= kTcsFoldMax && r.W / Q <= kTcsTickets) r.fold_n = (int)(Q / B);
    }
  }
  r.direct = direct;
  r.nstage = stages_for(E);
  if (r.nstage < 2) return false;
  if (r.fold_n * PIECE * 2 > r.nstage * STAGE) r.fold_n = 0;  // the last CTA stages the pieces there
  if (direct) {
    *p = r;
    return true;
  }
  // Piece slots per CTA: the most pieces any CTA's range produces.
  int cap = 1;
  for (long long b = 0; b < r.P; ++b) {
    const long long w0 = b * r.W / r.P, w1 = (b + 1) * r.W / r.P;
    int n = 0;
    for (long long w = w0; w < w1;) {
      const long long s = w / Q;
      const int qa = (int)(w - s * Q), qb = (int)((w1 - s * Q) < Q ? (w1 - s * Q) : Q);
      n += count_pieces(qa, qb);
      w = s * Q + qb;
    }
    if (n > cap) cap = n;
  }
  r.cap = cap;
  // Top kernel: staged pieces, output tiles, piece lists (the larger of its two modes).
  r.top_smem = top_smem(false, E, cap) > top_smem(true, E, cap) ? top_smem(false, E, cap) : top_smem(true, E, cap);
  if (r.top_smem > 200 * 1024) return false;
  r.scratch = (size_t)r.P * cap * PIECE * 2;
  *p = r;
  return true;
}

namespace {

// One-time kernel attributes (shared memory limits and carve-out).
cudaError_t tcs_setup() {
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
    void (*fws[4])(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, FwdArgs) = {
        k_tcs_fwd<2, 2>, k_tcs_fwd<2, 3>, k_tcs_fwd<3, 2>, k_tcs_fwd<3, 3>};
    for (auto k : fws) {
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, MAX_SMEM);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    }
    void (*tops[2])(TcsTopArgs) = {k_tcs_top<false>, k_tcs_top<true>};
    for (auto k : tops) {
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    }
    setup_err = e;
  });
  return setup_err;
}

cudaError_t tcs_launch(const TcsPlan& plan, const TcsProblem* pr, long long ldo, uint16_t* h, const uint16_t* silu,
                       void* scratch, size_t scratch_bytes, const Waits& wt, cudaStream_t st, float* dump,
                       long long oss) {
  if (plan.ns > 1 && (h || dump)) return cudaErrorInvalidValue;
  const long long Ktot = plan.K * plan.ns;  // the maps span every shard's K range
  if (!plan.direct && (!scratch || scratch_bytes < plan.scratch || ((uintptr_t)scratch & 15u)))
    return cudaErrorInvalidValue;
  if (plan.direct && h) return cudaErrorInvalidValue;
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
  const cudaError_t setup_err = tcs_setup();
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
  a.out0 = pr[0].out;
  a.out1 = plan.np > 1 ? pr[1].out : nullptr;
  a.ldo = ldo;
  a.status = wt.status;
  a.spin = wt.spin;
  a.stall = wt.stall;
  a.L = plan.G << plan.E;
  a.dump = dump;
  // Folded trees: the plain form (no h, no leaf dump) of aligned ranges, with
  // the handle's tickets.
  const bool fold = plan.fold_n > 0 && !h && !dump && wt.tickets;
  a.fold_n = fold ? plan.fold_n : 0;
  a.tickets = fold ? wt.tickets : nullptr;
  const int smem = smem_for(plan.E, plan.nstage);
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TcsArgs) =
      dump ? (plan.G == 1 ? k_tcs<1, true> : plan.G == 2 ? k_tcs<2, true> : k_tcs<3, true>)
           : (plan.G == 1 ? k_tcs<1, false> : plan.G == 2 ? k_tcs<2, false> : k_tcs<3, false>);
  cudaError_t e = launch_dependent(kern, dim3(plan.P), kThreads, smem, st, m[0], m[1], m[2], m[3], a);
  if (e != cudaSuccess || plan.direct || fold) return e;
  TcsTopArgs t{};
  t.R = plan.R;
  t.C = (int)plan.C;
  t.E = plan.E;
  t.np = plan.np;
  t.ns = plan.ns;
  t.oss = oss;
  t.W = plan.W;
  t.P = plan.P;
  t.cap = plan.cap;
  t.slots = static_cast<const uint16_t*>(scratch);
  t.out0 = pr[0].out;
  t.out1 = plan.np > 1 ? pr[1].out : nullptr;
  t.ldo = ldo;
  t.h = h;
  t.silu = silu;
  t.status = wt.status;
  const dim3 grid(h ? plan.T : plan.np * plan.ns * plan.T, (plan.R + kTopTok - 1) / kTopTok);
  const int smem_top = top_smem(h != nullptr, plan.E, plan.cap);
  return h ? launch_dependent(k_tcs_top<true>, grid, kTopThreads, smem_top, st, t)
           : launch_dependent(k_tcs_top<false>, grid, kTopThreads, smem_top, st, t);
}

}  // namespace

cudaError_t launch_tcs(const TcsPlan& plan, const TcsProblem* pr, long long ldo, void* scratch,
                       size_t scratch_bytes, const Waits& wt, cudaStream_t st, float* dump, long long oss) {
  for (int p = 0; p < plan.np; ++p)
    if (!pr[p].out) return cudaErrorInvalidValue;
  return tcs_launch(plan, pr, ldo, nullptr, nullptr, scratch, scratch_bytes, wt, st, dump, oss);
}

cudaError_t launch_tcs_gateup_stacked(long long R, long long C, long long K, const uint16_t* Wg, const uint16_t* Wu,
                                      long long ldw, const uint16_t* X, long long ldx, uint16_t* gate, uint16_t* up,
                                      uint16_t* h, long long ldo, const uint16_t* silu, int sm_count, const Waits& wt,
                                      cudaStream_t st) {
  if (R < 1 || R > BN || C < 1 || C % (BM / 2) || !h || !silu || (ldw % 8) || (ldx % 8) ||
      (((uintptr_t)Wg | (uintptr_t)Wu | (uintptr_t)X) & 15u))
    return cudaErrorInvalidValue;
  TcsPlan plan;
  // Tiles of 64 rows of each weight = 128 MMA rows: the plan of 2C rows.
  if (!tcs_plan(R, 2 * C, K, 1, 2 * sm_count, true, &plan, 1)) return cudaErrorInvalidValue;
  plan.nstage = stages_for(plan.E, true);
  if (plan.nstage < 2) return cudaErrorInvalidValue;
  CUtensorMap m[4];
  if (!tc_make_map(&m[0], Wg, C, K, ldw, BM / 2) || !tc_make_map(&m[2], Wu, C, K, ldw, BM / 2) ||
      !tc_make_map(&m[1], X, R, K, ldx, BN))
    return cudaErrorInvalidValue;
  m[3] = m[1];
  const cudaError_t setup_err = tcs_setup();
  if (setup_err != cudaSuccess) return setup_err;
  TcsArgs a{};
  a.R = (int)R;
  a.C = (int)C;
  a.G = plan.G;
  a.E = plan.E;
  a.np = 1;
  a.ns = 1;
  a.ksh = K;
  a.T = plan.T;
  a.W = plan.W;
  a.nstage = plan.nstage;
  a.out0 = gate;
  a.out1 = up;
  a.ldo = ldo;
  a.status = wt.status;
  a.spin = wt.spin;
  a.stall = wt.stall;
  a.L = plan.G << plan.E;
  a.stacked = 1;
  a.hout = h;
  a.silu = silu;
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, TcsArgs) =
      plan.G == 1 ? k_tcs<1, false> : plan.G == 2 ? k_tcs<2, false> : k_tcs<3, false>;
  return launch_dependent(kern, dim3(plan.P), kThreads, smem_for(plan.E, plan.nstage, true), st, m[0], m[1], m[2],
                          m[3], a);
}

namespace {

// The two plans of the fused forward and its launch geometry; false when the
// shape is not covered.
struct FusedPlan {
  TcsPlan a, b;
  int P, nA, nB, bG, nstage;
};
bool fused_plan_uncached(long long R, long long H, long long I, int sm_count, FusedPlan* fp) {
  if (R < 1 || R > BN || H < 1 || I < 1 || I % (BM / 2) || H % 8) return false;
  FusedPlan p;
  p.P = 2 * sm_count;
  // Unit A: stacked tiles (64 rows of each weight = 128 MMA rows) over K = H.
  if (!tcs_plan(R, 2 * I, H, 1, p.P, true, &p.a, 1)) return false;
  // Unit B: the down projection's aligned blocks, folded by the trees' last CTAs.
  if (!tcs_plan(R, H, I, 1, p.P, false, &p.b, 1, false) || p.b.fold_n < 2 || p.b.direct) return false;
  if (p.a.T > p.P || p.b.P > p.P || (p.a.G != 2 && p.a.G != 3) || (p.b.G != 2 && p.b.G != 3)) return false;
  p.nA = p.a.T;
  p.nB = p.b.P;
  p.bG = (int)(p.b.W / p.b.P);
  if (p.b.fold_n > kTcsRanges || p.b.cap != 1 || p.b.W / (1ll << p.b.E) > kTcsTickets) return false;
  // The down's K range of one block is bG * G leaves: that many 64-column tiles of h.
  if ((long long)p.bG * p.b.G * 64 * p.b.fold_n != I) return false;
  // The units' pending fold levels above the register ones live in TMEM.
  const int eB = p.b.E - hibit((unsigned)p.b.fold_n);
  if (p.a.E > kFwdMaxLevels || eB > kFwdMaxLevels) return false;
  // Stages: all the shared memory two CTAs per SM allow, at most one per
  // TMEM leaf buffer (a stage is reused once its leaf has been committed).
  p.nstage = (MAX_SMEM - 1024 - BAR_BYTES - XCH_BYTES) / STAGE;
  if (p.nstage > MAX_STAGES) p.nstage = MAX_STAGES;
  if (p.nstage > kFwdNBuf) p.nstage = kFwdNBuf;
  if (p.nstage < 2 || p.b.fold_n * PIECE * 2 > p.nstage * STAGE) return false;
  *fp = p;
  return true;
}

// The plan of a (R, H, I, SM count): worked out once (two few-token plans
// walk every CTA's range) and kept in a small table, as the call's other
// plans are.
bool fused_plan(long long R, long long H, long long I, int sm_count, FusedPlan* fp) {
  struct Entry {
    long long R, H, I;
    int sms;
    bool ok, used;
    FusedPlan plan;
  };
  constexpr int kEntries = 16;
  static Entry table[kEntries];
  static int next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : table)
      if (e.used && e.R == R && e.H == H && e.I == I && e.sms == sm_count) {
        if (e.ok) *fp = e.plan;
        return e.ok;
      }
  }
  FusedPlan p{};
  const bool ok = fused_plan_uncached(R, H, I, sm_count, &p);
  std::lock_guard<std::mutex> lock(mu);
  table[next] = Entry{R, H, I, sm_count, ok, true, p};
  next = (next + 1) % kEntries;
  if (ok) *fp = p;
  return ok;
}

}  // namespace

bool tcs_forward_fused_info(long long R, long long H, long long I, int sm_count, TcsFusedInfo* info) {
  FusedPlan p;
  if (!fused_plan(R, H, I, sm_count, &p)) return false;
  TcsFusedInfo r;
  r.P = p.P;
  r.nA = p.nA;
  r.nB = p.nB;
  r.bG = p.bG;
  r.GA = p.a.G;
  r.GB = p.b.G;
  r.EA = p.a.E;
  r.EB = p.b.E;
  r.fold_n = p.b.fold_n;
  r.trees = p.b.T;
  r.per_range = p.bG * p.b.G;
  r.waiters = 2 * p.b.T;
  r.nstage = p.nstage;
  r.smem = 1024 + p.nstage * STAGE + BAR_BYTES + XCH_BYTES;
  r.scratch = p.b.scratch;
  *info = r;
  return true;
}

bool tcs_forward_fused_covers(long long R, long long H, long long I, int sm_count, size_t* scratch) {
  FusedPlan p;
  if (!fused_plan(R, H, I, sm_count, &p)) return false;
  if (scratch) *scratch = p.b.scratch;
  return true;
}

cudaError_t launch_tcs_forward_fused(long long R, long long H, long long I, const uint16_t* x, const uint16_t* Wg,
                                     const uint16_t* Wu, const uint16_t* Wd, uint16_t* h, uint16_t* gate,
                                     uint16_t* up, uint16_t* out, const uint16_t* silu, void* scratch,
                                     size_t scratch_bytes, int sm_count, const Waits& wt, cudaStream_t st) {
  FusedPlan p;
  if (!fused_plan(R, H, I, sm_count, &p)) return cudaErrorNotSupported;
  if (!x || !Wg || !Wu || !Wd || !h || !out || !silu || !wt.tickets || !scratch || scratch_bytes < p.b.scratch ||
      (((uintptr_t)x | (uintptr_t)Wg | (uintptr_t)Wu | (uintptr_t)Wd | (uintptr_t)h | (uintptr_t)scratch) & 15u))
    return cudaErrorInvalidValue;
  CUtensorMap m[5];
  if (!tc_make_map(&m[0], Wg, I, H, H, BM / 2) || !tc_make_map(&m[1], Wu, I, H, H, BM / 2) ||
      !tc_make_map(&m[2], x, R, H, H, BN) || !tc_make_map(&m[3], Wd, H, I, I, BM) || !tc_make_map(&m[4], h, R, I, I, BN))
    return cudaErrorInvalidValue;
  const cudaError_t setup_err = tcs_setup();
  if (setup_err != cudaSuccess) return setup_err;
  FwdArgs f{};
  TcsArgs& A = f.A;
  A.R = (int)R;
  A.C = (int)I;
  A.G = p.a.G;
  A.E = p.a.E;
  A.np = 1;
  A.ns = 1;
  A.ksh = H;
  A.T = p.a.T;
  A.W = p.a.W;
  A.nstage = p.nstage;
  A.out0 = gate;
  A.out1 = up;
  A.ldo = I;
  A.status = wt.status;
  A.spin = wt.spin;
  A.stall = wt.stall;
  A.L = p.a.G << p.a.E;
  A.stacked = 1;
  A.hout = h;
  A.silu = silu;
  TcsArgs& B = f.B;
  B.R = (int)R;
  B.C = (int)H;
  B.G = p.b.G;
  B.E = p.b.E;
  B.np = 1;
  B.ns = 1;
  B.ksh = I;
  B.T = p.b.T;
  B.W = p.b.W;
  B.cap = p.b.cap;
  B.nstage = p.nstage;
  B.slots = static_cast<uint16_t*>(scratch);
  B.out0 = out;
  B.ldo = H;
  B.status = wt.status;
  B.spin = wt.spin;
  B.stall = wt.stall;
  B.L = p.b.G << p.b.E;
  B.fold_n = p.b.fold_n;
  B.tickets = wt.tickets;
  f.nA = p.nA;
  f.nB = p.nB;
  f.bG = p.bG;
  f.per_range = p.bG * p.b.G;
  f.waiters = 2 * p.b.T;
  f.ready = wt.tickets + kTcsTickets;
  const int smem = 1024 + p.nstage * STAGE + BAR_BYTES + XCH_BYTES;
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, FwdArgs) =
      p.a.G == 2 ? (p.b.G == 2 ? k_tcs_fwd<2, 2> : k_tcs_fwd<2, 3>) : (p.b.G == 2 ? k_tcs_fwd<3, 2> : k_tcs_fwd<3, 3>);
  return launch_dependent(kern, dim3(p.P), kThreads, smem, st, m[0], m[1], m[2], m[3], m[4], f);
}

cudaError_t launch_tcs_gateup(const TcsPlan& plan, const TcsProblem* pr, uint16_t* h, long long ldo,
                              const uint16_t* silu, void* scratch, size_t scratch_bytes, const Waits& wt,
                              cudaStream_t st) {
  if (plan.np != 2 || !h || !silu) return cudaErrorInvalidValue;
  return tcs_launch(plan, pr, ldo, h, silu, scratch, scratch_bytes, wt, st, nullptr, 0);
}

}  // namespace detffn
