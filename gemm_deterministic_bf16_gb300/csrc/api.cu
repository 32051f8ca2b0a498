// api.cu -- the C ABI of libdetffn: argument checks, scratch layout, dispatch.
//
// Every call validates its arguments on the host and returns an error before
// launching anything; every launch goes to the caller's stream.  Nothing here
// allocates device memory except detffn_create (tables and status word).
#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <initializer_list>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "decode.h"
#include "tc.h"

using namespace detffn;

constexpr int kTicketWords = kTcsTickets + 2 * kTcsRanges;

struct detffn_handle_s {
  int device = 0;
  int sm_count = 0;
  uint16_t* d_silu = nullptr;   // [65536] BF16 SiLU by gate bit pattern
  float* d_dsilu = nullptr;     // [65536] FP32 SiLU' by gate bit pattern
  int* d_status = nullptr;      // device status word (bounded waits)
  int* d_tickets = nullptr;     // tree tickets of the few-token kernels (kTcsTickets words) and the fused
                                // forward's range counters (2 x kTcsRanges words), zero between calls
  Waits wt;                     // the current call's wait settings (status word, poll limit, test stall)
  int flags = 0;                // the current call's option flags
  // A second stream and two events (made at creation) for the overlapped
  // dHidden reduction (DETFFN_FLAG_OVERLAP_DHIDDEN).
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  std::vector<uint16_t> h_silu;
  std::vector<float> h_dsilu;
  // Measurement: event pairs around launches while profiling is on.
  struct Rec {
    const char* name;
    cudaEvent_t a, b;
    double bytes, flops;
    int launches;
  };
  bool prof = false;
  std::vector<Rec> recs;
};

// ---------------------------------------------------------------------------
// SiLU tables, correctly rounded (the value of the real function rounded to
// FP32, and for SiLU then to BF16).  Method: binary64 evaluation; entries
// whose binary64 value lies within 2^-40 (relative) of an FP32 rounding
// boundary are re-evaluated in long double.  For |g| < 2^-10, SiLU'(g) is
// 1/2 + g/2 - g^3/12 + O(g^5): 1/2 + g/2 is exact in binary64 and the cubic
// term only decides an exact FP32 tie, toward the sign of -g.
// ---------------------------------------------------------------------------
namespace {

float widen_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

uint16_t bf16_rne_host(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
  const uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

// Distance from v to the nearest FP32 midpoint, relative to |v|.
double tie_gap(double v) {
  const float f = (float)v;
  const double d = v - (double)f;
  if (d == 0.0) return INFINITY;
  const float nb = nextafterf(f, d > 0 ? INFINITY : -INFINITY);
  const double mid = 0.5 * ((double)f + (double)nb);
  return fabs(v - mid) / fabs(v);
}

void silu_pair_ld(double g, float* y, float* d) {
  const long double G = (long double)g;
  const long double t = expl(-G);
  const long double s = 1.0L / (1.0L + t);
  const long double oms = t / (1.0L + t);
  *y = (float)(G * s);
  *d = (float)(s * (1.0L + G * oms));
}

void build_silu_tables(std::vector<uint16_t>& silu, std::vector<float>& dsilu) {
  silu.assign(65536, 0);
  dsilu.assign(65536, 0.0f);
  for (uint32_t i = 0; i < 65536u; ++i) {
    const float gf = widen_bf16((uint16_t)i);
    const double g = gf;
    float y, d;
    if (g != g) {
      silu[i] = bf16_rne_host(gf);
      dsilu[i] = gf;
      continue;
    }
    if (g > 200.0) {            // sigma(g) = 1 to far below FP32 resolution
      y = gf;
      d = 1.0f;
    } else if (g < -200.0) {    // both values are below 2^-150 in magnitude
      y = -0.0f;
      d = -0.0f;
    } else {
      const double t = exp(-g);
      const double s = 1.0 / (1.0 + t);
      const double oms = t / (1.0 + t);
      const double yd = g * s;
      const double dd = s * (1.0 + g * oms);
      y = (float)yd;
      d = (float)dd;
      if (fabs(g) < 0x1p-10) {
        const double lead = 0.5 + 0.5 * g;  // exact
        d = (float)lead;
        const double diff = lead - (double)d;
        if (diff != 0.0) {
          const float nb = nextafterf(d, diff > 0 ? INFINITY : -INFINITY);
          const double half = 0.5 * ((double)nb - (double)d);
          // At an exact tie the true value lies on the side of -g: take the
          // neighbour when that side is the neighbour's.
          if (diff == half && ((g < 0) == (diff > 0))) d = nb;
        }
        if (tie_gap(yd) < 0x1p-40) {
          float d_unused;
          silu_pair_ld(g, &y, &d_unused);
        }
      } else if (tie_gap(yd) < 0x1p-40 || tie_gap(dd) < 0x1p-40) {
        silu_pair_ld(g, &y, &d);
      }
    }
    silu[i] = bf16_rne_host(y);
    dsilu[i] = d;
  }
}

std::once_flag g_tab_once;
std::vector<uint16_t> g_silu;
std::vector<float> g_dsilu;

void host_tables() {
  std::call_once(g_tab_once, [] { build_silu_tables(g_silu, g_dsilu); });
}

}  // namespace

namespace detffn {
const uint16_t* host_silu_table() {
  host_tables();
  return g_silu.data();
}
}  // namespace detffn

// ---------------------------------------------------------------------------
// Argument checks and scratch layout
// ---------------------------------------------------------------------------
namespace {

struct Opts {
  int path = DETFFN_PATH_AUTO;
  int shards = 1;
  int flags = 0;
  long long spin_limit = 0;
};

// host_io_ok: the call takes DETFFN_FLAG_HOST_IO (the forward calls and
// their workspace sizes); elsewhere the flag is an invalid argument.
detffn_status read_opts(const detffn_options* o, Opts* out, bool host_io_ok = false) {
  Opts r;
  if (o) {
    if (o->leaf_width != 0 && o->leaf_width != kLeaf) return DETFFN_ERR_UNSUPPORTED;
    if (o->path < DETFFN_PATH_AUTO || o->path > DETFFN_PATH_TENSOR) return DETFFN_ERR_INVALID_ARG;
    if (!(o->shards == 0 || o->shards == 1 || o->shards == 2 || o->shards == 4 || o->shards == 8))
      return DETFFN_ERR_INVALID_ARG;
    if (o->spin_limit < 0) return DETFFN_ERR_INVALID_ARG;
    if (o->flags & ~(DETFFN_FLAG_TEST_STALL | DETFFN_FLAG_OVERLAP_DHIDDEN | DETFFN_FLAG_SPLIT_FORWARD |
                     DETFFN_FLAG_HOST_IO))
      return DETFFN_ERR_INVALID_ARG;
    if ((o->flags & DETFFN_FLAG_HOST_IO) && !host_io_ok) return DETFFN_ERR_INVALID_ARG;
    r.path = o->path;
    r.shards = o->shards ? o->shards : 1;
    r.flags = o->flags;
    r.spin_limit = o->spin_limit;
  }
  *out = r;
  return DETFFN_OK;
}

// The wait settings the launches of one call take from its options.
void set_waits(detffn_handle h, const Opts& o) {
  h->wt.status = h->d_status;
  h->wt.tickets = h->d_tickets;
  h->wt.spin = o.spin_limit;
  h->wt.stall = (o.flags & DETFFN_FLAG_TEST_STALL) ? 1 : 0;
  h->flags = o.flags;
}

// The kernel family a call uses.  EXACT: CUDA-core kernels with LANE8x8
// leaves (bit-identical to the oracle).  TENSOR: tcgen05 leaves.  AUTO takes
// TENSOR whenever the tensor kernels cover every contraction length of the
// call (H, I, I/k and M leaves of the form 1, 2^d or 3*2^d, and H, I
// multiples of 8), else EXACT.  A tensor-core leaf of an output element does
// not depend on the other rows or columns of its tile, nor on which operand
// sits on the MMA's 128-row side, so on the tensor family a token's result
// is the same for every token count (one token, a decode batch, a prefill);
// at one token the tensor family is also the faster one.  The choice never
// depends on the shard count or the chunking: a shard of I has the same
// leaf-count form as I.
enum Family { kExact = 0, kTensor = 1 };
constexpr long long kAutoExactMaxM = 0;

bool tc_len_ok(long long K) {
  int G, E;
  return K > 0 && tc_tree_shape((K + kLeaf - 1) / kLeaf, &G, &E);
}

bool tc_covers(long long M, long long H, long long I, bool backward) {
  if (H % 8 || I % 8) return false;
  if (!tc_len_ok(H) || !tc_len_ok(I)) return false;
  return !backward || tc_len_ok(M);
}

detffn_status pick_family(const Opts& o, long long M, long long H, long long I, bool backward, Family* f) {
  if (o.path == DETFFN_PATH_EXACT) {
    *f = kExact;
  } else if (o.path == DETFFN_PATH_TENSOR) {
    if (!tc_covers(M, H, I, backward)) return DETFFN_ERR_UNSUPPORTED;
    *f = kTensor;
  } else {
    *f = (M > kAutoExactMaxM && tc_covers(M, H, I, backward)) ? kTensor : kExact;
  }
  return DETFFN_OK;
}

struct Arena {
  char* base;
  size_t off = 0;
  explicit Arena(void* b) : base(static_cast<char*>(b)) {}
  template <class T>
  T* take(long long count) {
    off = (off + 255) & ~(size_t)255;
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += (size_t)count * sizeof(T);
    return p;
  }
};

// Piece slots of the few-token tensor contractions (R <= 32 tokens).
struct TcsScratch {
  void* p = nullptr;
  size_t bytes = 0;
};
constexpr int kSizingSms = 152;  // SM count a workspace is sized for when no handle is given

// Plans are validated and worked out once per signature (as the transport
// collectives do, RL-Kernel PR #356, "Design"): a plan depends only on
// (R, C, K, problems, CTAs, direct), and working it out walks every CTA's
// range, which costs microseconds of host time per call at decode sizes --
// comparable to the call's device time.  A small table keeps the recent ones.
bool tcs_plan_cached(long long R, long long C, long long K, int np, int ctas, bool direct, TcsPlan* p,
                     int ns = 1, bool whole_ok = true) {
  struct Entry {
    long long R, C, K;
    int np, ns, ctas;
    bool direct, whole_ok, ok, used;
    TcsPlan plan;
  };
  constexpr int kEntries = 32;
  static Entry table[kEntries];
  static int next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : table)
      if (e.used && e.R == R && e.C == C && e.K == K && e.np == np && e.ns == ns && e.ctas == ctas &&
          e.direct == direct && e.whole_ok == whole_ok) {
        if (e.ok) *p = e.plan;
        return e.ok;
      }
  }
  TcsPlan plan{};
  const bool ok = tcs_plan(R, C, K, np, ctas, direct, &plan, ns, whole_ok);
  std::lock_guard<std::mutex> lock(mu);
  table[next] = Entry{R, C, K, np, ns, ctas, direct, whole_ok, ok, true, plan};
  next = (next + 1) % kEntries;
  if (ok) *p = plan;
  return ok;
}

// Piece-slot bytes of a few-token contraction over C weight rows and K (ns
// shards of K each), two CTAs per SM.
size_t tcs_bytes(long long C, long long K, int np, int sms, int ns = 1) {
  TcsPlan p;  // sized for plans without whole-tile ranges (they need the most)
  return tcs_plan_cached(1, C, K, np, 2 * sms, false, &p, ns, false) ? p.scratch : 0;
}

// The plan for the scratch at hand: two CTAs per SM when the slots fit, fewer
// CTAs when they do not, whole tiles per CTA (no slots) as the last resort.
// The results are the same for every plan.
bool tcs_plan_fit(long long R, long long C, long long K, int np, int sms, const TcsScratch& sc, TcsPlan* p,
                  int ns = 1, bool whole_ok = true) {
  if (sc.p) {
    for (int ctas = 2 * sms; ctas >= 1; ctas = ctas * 3 / 4) {
      if (!tcs_plan_cached(R, C, K, np, ctas, false, p, ns, whole_ok)) return false;
      if (p->scratch <= sc.bytes) return true;
      if (ctas == 1) break;
    }
  }
  return tcs_plan_cached(R, C, K, np, 2 * sms, true, p, ns);
}

struct FwdWs {
  uint16_t *gate, *up, *h, *parts, *dec_part;
  uint16_t *x_stage, *out_stage;  // DETFFN_FLAG_HOST_IO: device copies of x and out
  unsigned* dec_cnt;
  TcsScratch tcs;
};
// Decode scratch: block-root planes (at most 8 blocks x 8 tokens x rows) and
// one ticket per row tile (at most one tile per row).
constexpr long long kDecPlanes = 64;
FwdWs plan_forward(Arena& a, long long M, long long H, long long I, int k, int sms, bool host_io = false) {
  FwdWs w;
  w.x_stage = host_io ? a.take<uint16_t>(M * H) : nullptr;
  w.out_stage = host_io ? a.take<uint16_t>(M * H) : nullptr;
  w.gate = a.take<uint16_t>(M * I);
  w.up = a.take<uint16_t>(M * I);
  w.h = a.take<uint16_t>(M * I);
  w.parts = k > 1 ? a.take<uint16_t>((long long)k * M * H) : nullptr;
  const long long rows = 2 * I > H ? 2 * I : H;
  w.dec_part = M <= 32 ? a.take<uint16_t>(kDecPlanes * rows) : nullptr;
  w.dec_cnt = M <= 32 ? a.take<unsigned>(rows + 1) : nullptr;
  // Tensor family with few tokens: piece slots for gate/up (all of I: the
  // shards' gate/up slices are computed by one launch) and for down.
  if (M >= 1 && M <= 32) {
    const long long sw = I / k;  // the down projection's k shards go in one launch
    const size_t gu = tcs_bytes(I, H, 2, sms), dn = tcs_bytes(H, sw, 1, sms, k);
    w.tcs.bytes = gu > dn ? gu : dn;
    w.tcs.p = a.take<unsigned char>((long long)w.tcs.bytes);
  }
  return w;
}

struct BwdWs {
  uint16_t *dh, *dU, *dG, *h, *cg, *cu, *cgs, *cus;
  TcsScratch tcs;  // tensor family, M <= 32
};
BwdWs plan_backward(Arena& a, long long M, long long H, long long I, int k, bool tensor, int sms) {
  BwdWs w{};
  w.dh = a.take<uint16_t>(M * I);
  w.dU = a.take<uint16_t>(M * I);
  w.dG = a.take<uint16_t>(M * I);
  w.h = a.take<uint16_t>(M * I);
  w.cg = a.take<uint16_t>(M * H);
  w.cu = a.take<uint16_t>(M * H);
  w.cgs = k > 1 ? a.take<uint16_t>((long long)k * M * H) : nullptr;
  w.cus = k > 1 ? a.take<uint16_t>((long long)k * M * H) : nullptr;
  if (tensor) {
    if (M >= 1 && M <= 32) {  // dh over K = H; cg and cu of all k shards (one launch) over K = I / k each
      const size_t d1 = tcs_bytes(I, H, 1, sms), d2 = tcs_bytes(H, I / k, 2, sms, k);
      w.tcs.bytes = d1 > d2 ? d1 : d2;
      w.tcs.p = a.take<unsigned char>((long long)w.tcs.bytes);
    }
  }
  return w;
}

struct ChunkWs {
  uint16_t *x, *dO, *g, *u, *dh, *dU, *dG, *h;
  TcsScratch tcs;  // tensor family: dh of chunks of <= 32 tokens
};
ChunkWs plan_chunked(Arena& a, long long M, long long H, long long I, bool tensor, int sms) {
  ChunkWs w{};
  w.x = a.take<uint16_t>(M * H);
  w.dO = a.take<uint16_t>(M * H);
  w.g = a.take<uint16_t>(M * I);
  w.u = a.take<uint16_t>(M * I);
  w.dh = a.take<uint16_t>(M * I);
  w.dU = a.take<uint16_t>(M * I);
  w.dG = a.take<uint16_t>(M * I);
  w.h = a.take<uint16_t>(M * I);
  if (tensor) {
    w.tcs.bytes = tcs_bytes(I, H, 1, sms);
    w.tcs.p = a.take<unsigned char>((long long)w.tcs.bytes);
  }
  return w;
}

size_t ws_bytes_for(int op, long long M, long long H, long long I, int k, bool tensor, int sms,
                    bool host_io = false) {
  Arena a(nullptr);
  switch (op) {
    case DETFFN_OP_FORWARD: plan_forward(a, M, H, I, 1, sms, host_io); break;
    case DETFFN_OP_FORWARD_SHARDED: plan_forward(a, M, H, I, k, sms, host_io); break;
    case DETFFN_OP_BACKWARD: plan_backward(a, M, H, I, k, tensor, sms); break;
    case DETFFN_OP_WGRAD_CHUNKED: plan_chunked(a, M, H, I, tensor, sms); break;
    default: return 0;
  }
  return (a.off + 255) & ~(size_t)255;
}

detffn_status check_ws(void* ws, size_t have, size_t need) {
  if (need == 0) return DETFFN_OK;
  if (!ws || ((uintptr_t)ws & 255u) != 0 || have < need) return DETFFN_ERR_WORKSPACE;
  return DETFFN_OK;
}

bool overlap(const void* a, long long na, const void* b, long long nb) {
  if (!a || !b || na <= 0 || nb <= 0) return false;
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

bool aligned2(const void* p) { return ((uintptr_t)p & 1u) == 0; }

detffn_status check_sizes(long long M, long long H, long long I) {
  if (M < 0 || H <= 0 || I <= 0) return DETFFN_ERR_SHAPE;
  if (H > kMaxK || I > kMaxK || M > kMaxK) return DETFFN_ERR_SHAPE;
  return DETFFN_OK;
}

thread_local cudaError_t g_last_cuda = cudaSuccess;

detffn_status cu(cudaError_t e) {
  if (e == cudaSuccess) return DETFFN_OK;
  g_last_cuda = e;
  return DETFFN_ERR_CUDA;
}

#define TRY(expr)                              \
  do {                                         \
    detffn_status _s = (expr);                 \
    if (_s != DETFFN_OK) return _s;            \
  } while (0)
#define TRYCU(expr) TRY(cu(expr))

// Runs `launch`; while profiling, brackets it with an event pair on `st`.
template <class F>
detffn_status timed(detffn_handle h, cudaStream_t st, const char* name, double bytes,
                    double flops, F&& launch, int launches = 1) {
  if (!h || !h->prof) return launch();
  detffn_handle_s::Rec r{name, nullptr, nullptr, bytes, flops, launches};
  if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return DETFFN_ERR_CUDA;
  cudaEventRecord(r.a, st);
  const detffn_status s = launch();
  cudaEventRecord(r.b, st);
  h->recs.push_back(r);
  return s;
}

// One tree contraction on the chosen family.
// Tensor family: A K-contiguous; B K-contiguous, or C-contiguous (weights in
// their stored [out, in] layout read along columns), which the tensor core
// then reads MN-major; 16-byte-aligned rows either way.  For R <= 32 (few
// tokens) the operands swap roles (weights fill the 128-row MMA side, tokens
// the 32-column side) and the result is stored transposed.
bool tc_operands_ok(const Strided& X) {
  return X.ks == 1 && (X.rs % 8) == 0 && (((uintptr_t)X.p) & 15u) == 0;
}
bool tc_mn_ok(const Strided& X) {
  return X.ks != 1 && X.rs == 1 && (X.ks % 8) == 0 && (((uintptr_t)X.p) & 15u) == 0;
}

detffn_status tree_gemm(detffn_handle h, Family f, Strided A, Strided B, long long R, long long C,
                        long long K, uint16_t* out, long long o_rs, cudaStream_t st,
                        const TcsScratch& sc = TcsScratch(), float* dump = nullptr) {
  const double bytes = 2.0 * ((double)R * K + (double)C * K + (double)R * C);
  if (f == kTensor) {
    const bool b_mn = tc_mn_ok(B), a_mn = tc_mn_ok(A);
    if (!(a_mn || tc_operands_ok(A)) || !(b_mn || tc_operands_ok(B))) return DETFFN_ERR_ALIGN;
    if (a_mn && R <= 32) return DETFFN_ERR_UNSUPPORTED;  // the few-token kernel takes K-major tokens
    const long long ldb = b_mn ? B.ks : B.rs;
    if (R <= 32) {  // few tokens: the weights (B) streamed on the MMA's 128-row side
      TcsPlan p;
      if (!tcs_plan_fit(R, C, K, 1, h->sm_count, sc, &p)) return DETFFN_ERR_SHAPE;
      const TcsProblem pr{B.p, ldb, A.p, A.rs, out, b_mn};
      return timed(h, st, "tcs_tree_gemm", bytes, 2.0 * R * C * K,
                   [&] { return cu(launch_tcs(p, &pr, o_rs, sc.p, sc.bytes, h->wt, st, dump)); },
                   p.launches(dump == nullptr));
    }
    return timed(h, st, "tc_tree_gemm", bytes, 2.0 * R * C * K, [&] {
      return cu(launch_tc_gemm(A.p, a_mn ? A.ks : A.rs, B.p, ldb, R, C, K, out, o_rs, 1, h->wt, h->sm_count, st,
                               b_mn, a_mn, dump));
    });
  }
  return timed(h, st, "tree_gemm_exact", bytes, 2.0 * R * C * K,
               [&] { return cu(launch_tree_gemm_exact(A, B, R, C, K, out, o_rs, st)); });
}

// Two same-shaped contractions: one launch of the tensor family (the two
// problems' tiles interleave over the SMs), two launches of the exact one.
detffn_status tree_gemm2(detffn_handle h, Family f, Strided A0, Strided B0, uint16_t* out0, Strided A1,
                         Strided B1, uint16_t* out1, long long R, long long C, long long K, long long o_rs,
                         cudaStream_t st, const TcsScratch& sc) {
  if (f != kTensor) {
    TRY(tree_gemm(h, f, A0, B0, R, C, K, out0, o_rs, st, sc));
    return tree_gemm(h, f, A1, B1, R, C, K, out1, o_rs, st, sc);
  }
  const double bytes = 4.0 * ((double)R * K + (double)C * K + (double)R * C);
  const bool b_mn = tc_mn_ok(B0), a_mn = tc_mn_ok(A0);
  if (tc_mn_ok(B1) != b_mn || tc_mn_ok(A1) != a_mn) return DETFFN_ERR_ALIGN;
  if (!(a_mn || (tc_operands_ok(A0) && tc_operands_ok(A1))) || !(b_mn || (tc_operands_ok(B0) && tc_operands_ok(B1))))
    return DETFFN_ERR_ALIGN;
  if (a_mn && R <= 32) return DETFFN_ERR_UNSUPPORTED;
  const long long ldb0 = b_mn ? B0.ks : B0.rs, ldb1 = b_mn ? B1.ks : B1.rs;
  if (R <= 32) {
    TcsPlan p;
    if (!tcs_plan_fit(R, C, K, 2, h->sm_count, sc, &p)) return DETFFN_ERR_SHAPE;
    const TcsProblem pr[2] = {{B0.p, ldb0, A0.p, A0.rs, out0, b_mn}, {B1.p, ldb1, A1.p, A1.rs, out1, b_mn}};
    return timed(h, st, "tcs_tree_gemm", bytes, 4.0 * R * C * K,
                 [&] { return cu(launch_tcs(p, pr, o_rs, sc.p, sc.bytes, h->wt, st)); }, p.launches(true));
  }
  return timed(h, st, "tc_tree_gemm", bytes, 4.0 * R * C * K, [&] {
    const TcProblem pr[2] = {{A0.p, a_mn ? A0.ks : A0.rs, B0.p, ldb0, out0, b_mn, a_mn},
                             {A1.p, a_mn ? A1.ks : A1.rs, B1.p, ldb1, out1, b_mn, a_mn}};
    return cu(launch_tc_gemms(pr, 2, R, C, K, o_rs, 1, h->wt, h->sm_count, st));
  });
}

// The K shard q of a strided operand: K positions [q * Ksh, (q + 1) * Ksh).
Strided kslice(const Strided& X, long long q, long long Ksh) { return Strided{X.p + q * Ksh * X.ks, X.rs, X.ks}; }

// k contractions over consecutive K shards of Ksh positions each (the
// tensor-parallel emulation): shard q's result goes to out + q * oss.  On the
// few-token tensor kernels all shards (and both problems of the two-problem
// form) are one launch; otherwise one launch per shard.
detffn_status tree_gemm_k(detffn_handle h, Family f, Strided A, Strided B, long long R, long long C,
                          long long Ksh, int k, uint16_t* out, long long o_rs, long long oss, cudaStream_t st,
                          const TcsScratch& sc) {
  if (f == kTensor && R <= 32 && k > 1) {
    const bool b_mn = tc_mn_ok(B);
    if (!tc_operands_ok(A) || !(b_mn || tc_operands_ok(B))) return DETFFN_ERR_ALIGN;
    TcsPlan p;
    if (!tcs_plan_fit(R, C, Ksh, 1, h->sm_count, sc, &p, k)) return DETFFN_ERR_SHAPE;
    const TcsProblem pr{B.p, b_mn ? B.ks : B.rs, A.p, A.rs, out, b_mn};
    const double bytes = 2.0 * ((double)R * Ksh * k + (double)C * Ksh * k + (double)R * C * k);
    return timed(h, st, "tcs_tree_gemm", bytes, 2.0 * R * C * Ksh * k, [&] {
      return cu(launch_tcs(p, &pr, o_rs, sc.p, sc.bytes, h->wt, st, nullptr, oss));
    }, p.launches(true));
  }
  for (int q = 0; q < k; ++q)
    TRY(tree_gemm(h, f, kslice(A, q, Ksh), kslice(B, q, Ksh), R, C, Ksh, out + q * oss, o_rs, st, sc));
  return DETFFN_OK;
}

detffn_status tree_gemm2_k(detffn_handle h, Family f, Strided A0, Strided B0, uint16_t* out0, Strided A1,
                           Strided B1, uint16_t* out1, long long R, long long C, long long Ksh, int k,
                           long long o_rs, long long oss, cudaStream_t st, const TcsScratch& sc) {
  if (f == kTensor && R <= 32 && k > 1) {
    const bool b_mn = tc_mn_ok(B0);
    if (tc_mn_ok(B1) != b_mn) return DETFFN_ERR_ALIGN;
    if (!tc_operands_ok(A0) || !tc_operands_ok(A1) || !(b_mn || (tc_operands_ok(B0) && tc_operands_ok(B1))))
      return DETFFN_ERR_ALIGN;
    TcsPlan p;
    if (!tcs_plan_fit(R, C, Ksh, 2, h->sm_count, sc, &p, k)) return DETFFN_ERR_SHAPE;
    const TcsProblem pr[2] = {{B0.p, b_mn ? B0.ks : B0.rs, A0.p, A0.rs, out0, b_mn},
                              {B1.p, b_mn ? B1.ks : B1.rs, A1.p, A1.rs, out1, b_mn}};
    const double bytes = 4.0 * ((double)R * Ksh * k + (double)C * Ksh * k + (double)R * C * k);
    return timed(h, st, "tcs_tree_gemm", bytes, 4.0 * R * C * Ksh * k, [&] {
      return cu(launch_tcs(p, pr, o_rs, sc.p, sc.bytes, h->wt, st, nullptr, oss));
    }, p.launches(true));
  }
  for (int q = 0; q < k; ++q)
    TRY(tree_gemm2(h, f, kslice(A0, q, Ksh), kslice(B0, q, Ksh), out0 + q * oss, kslice(A1, q, Ksh),
                   kslice(B1, q, Ksh), out1 + q * oss, R, C, Ksh, o_rs, st, sc));
  return DETFFN_OK;
}

detffn_status silu_mul(detffn_handle h, const uint16_t* g, const uint16_t* u, uint16_t* hh,
                       long long rows, long long cols, long long ld, cudaStream_t st) {
  return timed(h, st, "silu_mul", 6.0 * rows * cols, 0.0,
               [&] { return cu(launch_silu_mul(g, u, hh, rows, cols, ld, h->d_silu, st)); });
}

detffn_status silu_bwd(detffn_handle h, const uint16_t* dh, const uint16_t* g, const uint16_t* u,
                       uint16_t* dU, uint16_t* dG, uint16_t* hh, long long n, cudaStream_t st) {
  return timed(h, st, "silu_bwd", (hh ? 12.0 : 10.0) * n, 0.0, [&] {
    return cu(launch_silu_bwd(dh, g, u, dU, dG, hh, n, h->d_silu, h->d_dsilu, st));
  });
}

detffn_status add_bf16(detffn_handle h, const uint16_t* a, const uint16_t* b, uint16_t* out,
                       long long n, cudaStream_t st) {
  return timed(h, st, "add_bf16", 6.0 * n, 0.0, [&] { return cu(launch_add_bf16(a, b, out, n, st)); });
}

detffn_status rank_tree_bf16(detffn_handle h, const void* const* in, int k, void* out,
                             long long count, cudaStream_t st) {
  return timed(h, st, "rank_tree", 2.0 * (k + 1) * count, 0.0, [&] {
    return cu(launch_rank_tree(in, k, out, count, DETFFN_BF16, h->sm_count, st));
  });
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// True when the exact weight-streaming decode kernels cover a forward of M
// tokens with gate/up contraction length Kg over Ng rows and down contraction
// length Kd (same bits as the general exact kernel either way).
bool decode_covers(long long M, long long Kg, long long Kd, std::initializer_list<const void*> ptrs) {
  int S, NB;
  if (M < 1 || M > 32 || !decode_geometry(Kg, &S, &NB) || !decode_geometry(Kd, &S, &NB)) return false;
  for (const void* p : ptrs)
    if (!aligned16(p)) return false;
  return true;
}

// gate/up rows [0, N) of Wg/Wu (row stride ldw), K = Kg; h (and the optional
// saves) get columns [0, N) with row stride ldo.  Token passes of 8.
detffn_status decode_gateup(detffn_handle h, const uint16_t* x, long long ldx, const uint16_t* Wg,
                            const uint16_t* Wu, long long ldw, long long N, long long Kg,
                            long long M, uint16_t* hh, uint16_t* gsave, uint16_t* usave,
                            long long ldo, uint16_t* part, unsigned* cnt, cudaStream_t st) {
  const double bytes = 2.0 * (2.0 * N * Kg + (double)M * Kg + 3.0 * M * N);
  return timed(h, st, "decode_gateup", bytes, 4.0 * M * N * Kg, [&] {
    for (long long p = 0; p < M; p += 8) {
      DecArgs a{};
      a.x = x + p * ldx; a.ldx = ldx; a.w0 = Wg; a.w1 = Wu; a.ldw = ldw; a.N = N; a.K = Kg;
      a.M = (int)(M - p < 8 ? M - p : 8);
      a.part = part; a.cnt = cnt;
      a.out = hh + p * ldo; a.ldo = ldo;
      a.gsave = gsave ? gsave + p * ldo : nullptr;
      a.usave = usave ? usave + p * ldo : nullptr;
      a.silu = h->d_silu; a.status = h->wt.status; a.spin_limit = h->wt.spin; a.stall = h->wt.stall;
      const cudaError_t e = launch_decode_exact(a, h->sm_count, st);
      if (e != cudaSuccess) return DETFFN_ERR_CUDA;
    }
    return DETFFN_OK;
  }, (int)((M + 7) / 8));
}

// out[:, 0:N) = T_K(x, W rows) with W row stride ldw, x row stride ldx.
detffn_status decode_plain(detffn_handle h, const uint16_t* x, long long ldx, const uint16_t* W,
                           long long ldw, long long N, long long K, long long M, uint16_t* out,
                           long long ldo, uint16_t* part, unsigned* cnt, cudaStream_t st) {
  const double bytes = 2.0 * ((double)N * K + (double)M * K + (double)M * N);
  return timed(h, st, "decode_down", bytes, 2.0 * M * N * K, [&] {
    for (long long p = 0; p < M; p += 8) {
      DecArgs a{};
      a.x = x + p * ldx; a.ldx = ldx; a.w0 = W; a.w1 = nullptr; a.ldw = ldw; a.N = N; a.K = K;
      a.M = (int)(M - p < 8 ? M - p : 8);
      a.part = part; a.cnt = cnt;
      a.out = out + p * ldo; a.ldo = ldo;
      a.silu = h->d_silu; a.status = h->wt.status; a.spin_limit = h->wt.spin; a.stall = h->wt.stall;
      const cudaError_t e = launch_decode_exact(a, h->sm_count, st);
      if (e != cudaSuccess) return DETFFN_ERR_CUDA;
    }
    return DETFFN_OK;
  }, (int)((M + 7) / 8));
}

}  // namespace

// ---------------------------------------------------------------------------
// Exported calls
// ---------------------------------------------------------------------------
extern "C" {

const char* detffn_status_string(detffn_status s) {
  switch (s) {
    case DETFFN_OK: return "ok";
    case DETFFN_ERR_INVALID_ARG: return "invalid argument";
    case DETFFN_ERR_SHAPE: return "unsupported or inconsistent sizes";
    case DETFFN_ERR_ALIGN: return "misaligned pointer";
    case DETFFN_ERR_UNSUPPORTED: return "unsupported option";
    case DETFFN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DETFFN_ERR_CUDA: return "CUDA error";
    case DETFFN_ERR_TIMEOUT: return "bounded in-kernel wait timed out";
  }
  return "unknown status";
}

detffn_status detffn_create(detffn_handle* out, int device) {
  if (!out) return DETFFN_ERR_INVALID_ARG;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n) return DETFFN_ERR_INVALID_ARG;
  int prev = 0;
  TRYCU(cudaGetDevice(&prev));
  TRYCU(cudaSetDevice(device));
  host_tables();
  detffn_handle h = new detffn_handle_s();
  h->device = device;
  h->h_silu = g_silu;
  h->h_dsilu = g_dsilu;
  detffn_status st = DETFFN_OK;
  do {
    if (cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) { st = DETFFN_ERR_CUDA; break; }
    if (cudaMalloc(&h->d_silu, 65536 * sizeof(uint16_t)) != cudaSuccess) { st = DETFFN_ERR_CUDA; break; }
    if (cudaMalloc(&h->d_dsilu, 65536 * sizeof(float)) != cudaSuccess) { st = DETFFN_ERR_CUDA; break; }
    if (cudaMalloc(&h->d_status, sizeof(int)) != cudaSuccess) { st = DETFFN_ERR_CUDA; break; }
    if (cudaMalloc(&h->d_tickets, kTicketWords * sizeof(int)) != cudaSuccess) { st = DETFFN_ERR_CUDA; break; }
    if (cudaStreamCreateWithFlags(&h->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) != cudaSuccess) { st = DETFFN_ERR_CUDA; break; }
    if (cudaMemcpy(h->d_silu, h->h_silu.data(), 65536 * sizeof(uint16_t), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(h->d_dsilu, h->h_dsilu.data(), 65536 * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess ||
        cudaMemset(h->d_tickets, 0, kTicketWords * sizeof(int)) != cudaSuccess) { st = DETFFN_ERR_CUDA; break; }
  } while (0);
  cudaSetDevice(prev);
  if (st != DETFFN_OK) {
    detffn_destroy(h);
    return st;
  }
  *out = h;
  return DETFFN_OK;
}

detffn_status detffn_destroy(detffn_handle h) {
  if (!h) return DETFFN_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(h->device);
  if (h->d_silu) cudaFree(h->d_silu);
  if (h->d_dsilu) cudaFree(h->d_dsilu);
  if (h->d_status) cudaFree(h->d_status);
  if (h->d_tickets) cudaFree(h->d_tickets);
  if (h->ev_fork) cudaEventDestroy(h->ev_fork);
  if (h->ev_join) cudaEventDestroy(h->ev_join);
  if (h->side) cudaStreamDestroy(h->side);
  for (auto& r : h->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  cudaSetDevice(prev);
  delete h;
  return DETFFN_OK;
}

detffn_status detffn_workspace_size(detffn_handle h, int op, long long M, long long H, long long I,
                                    int k, const detffn_options* opts, size_t* bytes) {
  if (!bytes) return DETFFN_ERR_INVALID_ARG;
  Opts o;
  TRY(read_opts(opts, &o, true));
  TRY(check_sizes(M, H, I));
  if (op < DETFFN_OP_FORWARD || op > DETFFN_OP_WGRAD_CHUNKED) return DETFFN_ERR_INVALID_ARG;
  const bool host_io = (o.flags & DETFFN_FLAG_HOST_IO) != 0;
  if (host_io && op != DETFFN_OP_FORWARD && op != DETFFN_OP_FORWARD_SHARDED) return DETFFN_ERR_INVALID_ARG;
  if (op == DETFFN_OP_BACKWARD && k <= 1) k = o.shards;
  if (!(k == 1 || k == 2 || k == 4 || k == 8)) return DETFFN_ERR_INVALID_ARG;
  Family f;
  const bool bwd = op == DETFFN_OP_BACKWARD || op == DETFFN_OP_WGRAD_CHUNKED;
  TRY(pick_family(o, M, H, I, bwd, &f));
  *bytes = ws_bytes_for(op, M, H, I, k, f == kTensor, h ? h->sm_count : kSizingSms, host_io);
  return DETFFN_OK;
}

detffn_status detffn_silu_tables(detffn_handle h, unsigned short* silu_bf16, float* dsilu_f32) {
  const std::vector<uint16_t>* s;
  const std::vector<float>* d;
  if (h) {
    s = &h->h_silu;
    d = &h->h_dsilu;
  } else {
    host_tables();
    s = &g_silu;
    d = &g_dsilu;
  }
  if (silu_bf16) memcpy(silu_bf16, s->data(), 65536 * sizeof(uint16_t));
  if (dsilu_f32) memcpy(dsilu_f32, d->data(), 65536 * sizeof(float));
  return DETFFN_OK;
}

detffn_status detffn_get_status(detffn_handle h, void* stream) {
  if (!h) return DETFFN_ERR_INVALID_ARG;
  TRYCU(cudaStreamSynchronize((cudaStream_t)stream));
  int v = 0;
  TRYCU(cudaMemcpy(&v, h->d_status, sizeof(int), cudaMemcpyDeviceToHost));
  TRYCU(cudaMemset(h->d_status, 0, sizeof(int)));
  // A launch that stopped on a timeout may have left trees with some of
  // their tickets taken: start the next call from zero.
  if (v != 0) TRYCU(cudaMemset(h->d_tickets, 0, kTicketWords * sizeof(int)));
  return (detffn_status)v;
}

}  // extern "C"

namespace {

// The device-visible address of a page-locked host buffer of this process
// (DETFFN_FLAG_HOST_IO); anything else is an invalid argument.
detffn_status host_buffer(const void* p, void** dev) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // (clears the sticky-free error of the query)
    return DETFFN_ERR_INVALID_ARG;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return DETFFN_ERR_INVALID_ARG;
  *dev = at.devicePointer;
  return DETFFN_OK;
}

detffn_status check_ffn_ptrs(const void* x, const void* Wg, const void* Wu, const void* Wd) {
  if (!x || !Wg || !Wu || !Wd) return DETFFN_ERR_INVALID_ARG;
  if (!aligned2(x) || !aligned2(Wg) || !aligned2(Wu) || !aligned2(Wd)) return DETFFN_ERR_ALIGN;
  return DETFFN_OK;
}

// Forward of one shard (or of everything when w == I, s == 0): gate/up for
// rows [s*w, (s+1)*w) of Wg/Wu, then h on the same columns.
detffn_status gateup_slice(detffn_handle h, Family f, const uint16_t* x, const uint16_t* Wg,
                           const uint16_t* Wu, uint16_t* gate, uint16_t* up, bool keep, uint16_t* hh,
                           long long M, long long H, long long I, long long s, long long w,
                           cudaStream_t st, const TcsScratch& sc) {
  const Strided X{x, H, 1};
  if (f == kTensor) {
    // gate and up in one launch (their tiles interleave over the SMs).
    const Strided BG{Wg + s * w * H, H, 1}, BU{Wu + s * w * H, H, 1};
    if (!tc_operands_ok(X) || !tc_operands_ok(BG) || !tc_operands_ok(BU)) return DETFFN_ERR_ALIGN;
    if (M <= 32 && w % 64 == 0) {
      // Few tokens, whole tiles: 64 rows of Wg over the same 64 rows of Wu
      // per CTA, which forms both trees' roots and h itself (one launch, no
      // pieces); gate and up are stored only when the caller keeps them.
      const double bytes = 2.0 * (2.0 * w * H + (double)M * H + (keep ? 3.0 : 1.0) * M * w);
      return timed(h, st, "tcs_gateup", bytes, 4.0 * M * w * H, [&] {
        return cu(launch_tcs_gateup_stacked(M, w, H, BG.p, BU.p, H, x, H, keep ? gate + s * w : nullptr,
                                            keep ? up + s * w : nullptr, hh + s * w, I, h->d_silu, h->sm_count,
                                            h->wt, st));
      });
    }
    if (M <= 32) {
      // Few tokens: the top of both trees fused with SiLU * up; gate and up
      // are stored only when the caller keeps them.
      TcsPlan p;
      if (!tcs_plan_fit(M, w, H, 2, h->sm_count, sc, &p, 1, false) || p.direct) return DETFFN_ERR_WORKSPACE;
      const double bytes = 2.0 * (2.0 * w * H + (double)M * H + (keep ? 3.0 : 1.0) * M * w);
      const TcsProblem pr[2] = {{BG.p, H, x, H, keep ? gate + s * w : nullptr},
                                {BU.p, H, x, H, keep ? up + s * w : nullptr}};
      return timed(h, st, "tcs_gateup", bytes, 4.0 * M * w * H, [&] {
        return cu(launch_tcs_gateup(p, pr, hh + s * w, I, h->d_silu, sc.p, sc.bytes, h->wt, st));
      }, 2);
    }
    const double bytes = 2.0 * (2.0 * w * H + (double)M * H + 2.0 * M * w);
    TRY(timed(h, st, "tc_tree_gemm", bytes, 4.0 * M * w * H, [&] {
      const TcProblem pr[2] = {{x, H, BG.p, H, gate + s * w}, {x, H, BU.p, H, up + s * w}};
      return cu(launch_tc_gemms(pr, 2, M, w, H, I, 1, h->wt, h->sm_count, st));
    }));
  } else {
    TRY(tree_gemm(h, f, X, Strided{Wg + s * w * H, H, 1}, M, w, H, gate + s * w, I, st));
    TRY(tree_gemm(h, f, X, Strided{Wu + s * w * H, H, 1}, M, w, H, up + s * w, I, st));
  }
  return silu_mul(h, gate + s * w, up + s * w, hh + s * w, M, w, I, st);
}

detffn_status forward_impl(detffn_handle h, const void* x, const void* Wg, const void* Wu,
                           const void* Wd, void* out, void* gate_save, void* up_save, long long M,
                           long long H, long long I, int k, void* ws, size_t ws_bytes,
                           void* stream, const detffn_options* opts) {
  if (!h || !out) return DETFFN_ERR_INVALID_ARG;
  Opts o;
  TRY(read_opts(opts, &o, true));
  set_waits(h, o);
  TRY(check_sizes(M, H, I));
  TRY(check_ffn_ptrs(x, Wg, Wu, Wd));
  const bool host_io = (o.flags & DETFFN_FLAG_HOST_IO) != 0;
  if (!aligned2(out) || !aligned2(gate_save) || !aligned2(up_save)) return DETFFN_ERR_ALIGN;
  if ((gate_save == nullptr) != (up_save == nullptr)) return DETFFN_ERR_INVALID_ARG;
  if (!(k == 1 || k == 2 || k == 4 || k == 8)) return DETFFN_ERR_INVALID_ARG;
  if (k > 1 && (I % k != 0 || (I / k) % kLeaf != 0 || (I / k) / kLeaf < 2)) return DETFFN_ERR_SHAPE;
  const long long bx = 2 * M * H, bw = 2 * I * H, bmi = 2 * M * I;
  const void* ins[4] = {x, Wg, Wu, Wd};
  const long long nin[4] = {bx, bw, bw, bw};
  void* outs[3] = {out, gate_save, up_save};
  const long long nout[3] = {bx, bmi, bmi};
  for (int a = 0; a < 3; ++a) {
    for (int b = 0; b < 4; ++b)
      if (overlap(outs[a], nout[a], ins[b], nin[b])) return DETFFN_ERR_INVALID_ARG;
    for (int b = a + 1; b < 3; ++b)
      if (overlap(outs[a], nout[a], outs[b], nout[b])) return DETFFN_ERR_INVALID_ARG;
  }
  Family f;
  TRY(pick_family(o, M, H, I, false, &f));
  if (f == kTensor && ((!host_io && !aligned16(x)) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd))) {
    if (o.path == DETFFN_PATH_TENSOR) return DETFFN_ERR_ALIGN;
    f = kExact;
  }
  TRY(check_ws(ws, ws_bytes,
               ws_bytes_for(k > 1 ? DETFFN_OP_FORWARD_SHARDED : DETFFN_OP_FORWARD, M, H, I, k, false, h->sm_count,
                            host_io)));
  if (M == 0) return DETFFN_OK;
  TRYCU(cudaSetDevice(h->device));
  cudaStream_t st = (cudaStream_t)stream;
  Arena a(ws);
  FwdWs w = plan_forward(a, M, H, I, k, h->sm_count, host_io);
  void* out_host = nullptr;  // DETFFN_FLAG_HOST_IO: where out goes back to
  if (host_io) {
    // x comes in over the host link to its staged copy, which the kernels
    // read; out is formed in its staged copy and goes back at the end.
    void* x_host = nullptr;
    TRY(host_buffer(x, &x_host));
    TRY(host_buffer(out, &out_host));
    TRY(timed(h, st, "host_copy", 2.0 * M * H, 0.0, [&] {
      return cu(launch_copy(x_host, w.x_stage, 2 * M * H, h->sm_count, st));
    }));
    x = w.x_stage;
    out = w.out_stage;
  }
  uint16_t* gate = gate_save ? (uint16_t*)gate_save : w.gate;
  uint16_t* up = up_save ? (uint16_t*)up_save : w.up;
  const uint16_t* X = (const uint16_t*)x;
  const uint16_t* WG = (const uint16_t*)Wg;
  const uint16_t* WU = (const uint16_t*)Wu;
  const uint16_t* WD = (const uint16_t*)Wd;
  const long long sw = I / k;  // I-slice of one shard (all of I when k == 1)
  const bool dec = f == kExact &&
                   decode_covers(M, H, sw, {x, Wg, Wu, Wd, w.h, (const void*)(w.h + sw)});
  const bool saves = gate_save != nullptr;
  if (dec) TRYCU(cudaMemsetAsync(w.dec_cnt, 0, sizeof(unsigned) * (size_t)((2 * I > H ? 2 * I : H) + 1), st));
  const TcsScratch& sc = w.tcs;
  for (long long s = 0; s < k; ++s) {
    uint16_t* dst = k == 1 ? (uint16_t*)out : w.parts + s * M * H;
    if (dec) {
      TRY(decode_gateup(h, X, H, WG + s * sw * H, WU + s * sw * H, H, sw, H, M, w.h + s * sw,
                        saves ? gate + s * sw : nullptr, saves ? up + s * sw : nullptr, I,
                        w.dec_part, w.dec_cnt, st));
      TRY(decode_plain(h, w.h + s * sw, I, WD + s * sw, I, H, sw, M, dst, H, w.dec_part, w.dec_cnt, st));
    } else {
      // gate/up contract over H, which no shard splits: the shards' slices of
      // gate, up and h are the same bits whether computed slice by slice or
      // at once, so one launch computes all of them.  The down projection's
      // shards (consecutive K ranges of I) are one call as well.
      size_t need = 0;
      if (s == 0 && k == 1 && f == kTensor && !(o.flags & DETFFN_FLAG_SPLIT_FORWARD) && sc.p &&
          tcs_forward_fused_covers(M, H, I, h->sm_count, &need) && need <= sc.bytes) {
        // One launch: gate/up, SiLU * up and down (the same bits as below).
        const double bytes = 2.0 * (3.0 * I * H + (double)M * H * 2 + (saves ? 3.0 : 1.0) * M * I);
        TRY(timed(h, st, "tcs_forward", bytes, 6.0 * M * I * H, [&] {
          return cu(launch_tcs_forward_fused(M, H, I, X, WG, WU, WD, w.h, saves ? gate : nullptr,
                                             saves ? up : nullptr, dst, h->d_silu, sc.p, sc.bytes, h->sm_count,
                                             h->wt, st));
        }));
      } else if (s == 0) {
        TRY(gateup_slice(h, f, X, WG, WU, gate, up, saves, w.h, M, H, I, 0, I, st, sc));
        TRY(tree_gemm_k(h, f, Strided{w.h, I, 1}, Strided{WD, I, 1}, M, H, sw, k, dst, H, M * H, st, sc));
      }
    }
  }
  if (k > 1) {
    const void* parts[8];
    for (int s = 0; s < k; ++s) parts[s] = w.parts + (long long)s * M * H;
    TRY(rank_tree_bf16(h, parts, k, out, M * H, st));
  }
  if (!host_io) return DETFFN_OK;
  return timed(h, st, "host_copy", 2.0 * M * H, 0.0, [&] {
    return cu(launch_copy(out, out_host, 2 * M * H, h->sm_count, st));
  });
}

}  // namespace

extern "C" detffn_status detffn_forward(detffn_handle h, const void* x, const void* Wg,
                                        const void* Wu, const void* Wd, void* out,
                                        void* gate_save, void* up_save, long long M, long long H,
                                        long long I, void* ws, size_t ws_bytes, void* stream,
                                        const detffn_options* opts) {
  return forward_impl(h, x, Wg, Wu, Wd, out, gate_save, up_save, M, H, I, 1, ws, ws_bytes, stream, opts);
}

extern "C" detffn_status detffn_forward_sharded(detffn_handle h, const void* x, const void* Wg,
                                                const void* Wu, const void* Wd, void* out,
                                                void* gate_save, void* up_save, long long M,
                                                long long H, long long I, int k, void* ws,
                                                size_t ws_bytes, void* stream,
                                                const detffn_options* opts) {
  return forward_impl(h, x, Wg, Wu, Wd, out, gate_save, up_save, M, H, I, k, ws, ws_bytes, stream, opts);
}

namespace {

// Row-wise backward stages for rows [r0, r0+rows): dh, then dU and dG (and h
// again, for the down projection's weight gradient, in the same pass).
detffn_status rowwise_bwd(detffn_handle h, Family f, const uint16_t* dOut, const uint16_t* Wd,
                          const uint16_t* gate, const uint16_t* up,
                          uint16_t* dh, uint16_t* dU, uint16_t* dG, uint16_t* hh, long long rows, long long H,
                          long long I, cudaStream_t st, const TcsScratch& sc) {
  // dh[m, i] = T_{n<H}(dOut[m, n], Wd[n, i]): B row i is column i of Wd (K stride I),
  // (read MN-major by the tensor family).
  const Strided B{Wd, 1, I};
  TRY(tree_gemm(h, f, Strided{dOut, H, 1}, B, rows, I, H, dh, I, st, sc));
  return silu_bwd(h, dh, gate, up, dU, dG, hh, rows * I, st);
}

// Weight gradients over K = M tokens from row-major [M, .] stage tensors (the
// tensor family reads both operands MN-major: no transposed copies).
detffn_status wgrads(detffn_handle h, Family f, const uint16_t* x, const uint16_t* dOut,
                     const uint16_t* hh, const uint16_t* dU, const uint16_t* dG, uint16_t* dWg,
                     uint16_t* dWu, uint16_t* dWd, long long M, long long H, long long I,
                     cudaStream_t st) {
  // dWd[n, i] = T_m(dOut[m, n], h[m, i])
  TRY(tree_gemm(h, f, Strided{dOut, 1, H}, Strided{hh, 1, I}, H, I, M, dWd, I, st));
  // dWg[i, n] = T_m(dG[m, i], x[m, n]); dWu likewise with dU (one launch of
  // the tensor family for both).
  return tree_gemm2(h, f, Strided{dG, 1, I}, Strided{x, 1, H}, dWg, Strided{dU, 1, I}, Strided{x, 1, H}, dWu, I, H,
                    M, H, st, TcsScratch());
}

}  // namespace

extern "C" detffn_status detffn_backward(detffn_handle h, const void* x, const void* Wg,
                                         const void* Wu, const void* Wd, const void* gate,
                                         const void* up, const void* dOut, void* dX, void* dWg,
                                         void* dWu, void* dWd, void* dh_save, void* dU_save,
                                         void* dG_save, long long M, long long H, long long I,
                                         void* ws, size_t ws_bytes, void* stream,
                                         const detffn_options* opts) {
  if (!h || !gate || !up || !dOut || !dX || !dWg || !dWu || !dWd) return DETFFN_ERR_INVALID_ARG;
  Opts o;
  TRY(read_opts(opts, &o));
  set_waits(h, o);
  TRY(check_sizes(M, H, I));
  TRY(check_ffn_ptrs(x, Wg, Wu, Wd));
  const void* al[] = {gate, up, dOut, dX, dWg, dWu, dWd, dh_save, dU_save, dG_save};
  for (const void* p : al)
    if (!aligned2(p)) return DETFFN_ERR_ALIGN;
  const int k = o.shards;
  if (k > 1 && (I % k != 0 || (I / k) % kLeaf != 0 || (I / k) / kLeaf < 2)) return DETFFN_ERR_SHAPE;
  const long long bx = 2 * M * H, bw = 2 * I * H, bmi = 2 * M * I;
  const void* ins[7] = {x, Wg, Wu, Wd, gate, up, dOut};
  const long long nin[7] = {bx, bw, bw, bw, bmi, bmi, bx};
  void* outs[7] = {dX, dWg, dWu, dWd, dh_save, dU_save, dG_save};
  const long long nout[7] = {bx, bw, bw, bw, bmi, bmi, bmi};
  for (int a = 0; a < 7; ++a) {
    for (int b = 0; b < 7; ++b)
      if (overlap(outs[a], nout[a], ins[b], nin[b])) return DETFFN_ERR_INVALID_ARG;
    for (int b = a + 1; b < 7; ++b)
      if (overlap(outs[a], nout[a], outs[b], nout[b])) return DETFFN_ERR_INVALID_ARG;
  }
  Family f;
  TRY(pick_family(o, M, H, I, true, &f));
  if (f == kTensor) {
    const void* ps[] = {x, Wg, Wu, Wd, gate, up, dOut, dh_save, dU_save, dG_save};
    bool al = true;
    for (const void* p : ps) al = al && aligned16(p);
    if (!al) {
      if (o.path == DETFFN_PATH_TENSOR) return DETFFN_ERR_ALIGN;
      f = kExact;
    }
  }
  TRY(check_ws(ws, ws_bytes, ws_bytes_for(DETFFN_OP_BACKWARD, M, H, I, k, f == kTensor, h->sm_count)));
  if (M == 0) {
    // No tokens: the weight gradients are empty sums (+0); nothing else exists.
    TRYCU(cudaSetDevice(h->device));
    cudaStream_t st = (cudaStream_t)stream;
    TRYCU(cudaMemsetAsync(dWg, 0, (size_t)bw, st));
    TRYCU(cudaMemsetAsync(dWu, 0, (size_t)bw, st));
    return cu(cudaMemsetAsync(dWd, 0, (size_t)bw, st));
  }
  TRYCU(cudaSetDevice(h->device));
  cudaStream_t st = (cudaStream_t)stream;
  Arena a(ws);
  BwdWs w = plan_backward(a, M, H, I, k, f == kTensor, h->sm_count);
  uint16_t* dh = dh_save ? (uint16_t*)dh_save : w.dh;
  uint16_t* dU = dU_save ? (uint16_t*)dU_save : w.dU;
  uint16_t* dG = dG_save ? (uint16_t*)dG_save : w.dG;
  const uint16_t* G = (const uint16_t*)gate;
  const uint16_t* U = (const uint16_t*)up;
  const uint16_t* WG = (const uint16_t*)Wg;
  const uint16_t* WU = (const uint16_t*)Wu;
  TRY(rowwise_bwd(h, f, (const uint16_t*)dOut, (const uint16_t*)Wd, G, U, dh, dU, dG, w.h, M, H, I, st,
                  w.tcs));
  // dHidden: cg = T_i(dG[m, i], Wg[i, n]), cu = T_i(dU[m, i], Wu[i, n]); the two
  // trees stay separate until the final gate-then-up addition.  B row n is
  // column n of Wg (K stride H), read MN-major by the tensor family.
  auto wcol = [&](const uint16_t* W, long long s0) { return Strided{W + s0 * H, 1, H}; };
  const long long sw = I / k;
  if (k == 1) {
    TRY(tree_gemm2(h, f, Strided{dG, I, 1}, wcol(WG, 0), w.cg, Strided{dU, I, 1}, wcol(WU, 0), w.cu, M, H, I, H,
                   st, w.tcs));
  } else if (h->flags & DETFFN_FLAG_OVERLAP_DHIDDEN) {
    // Two streams (PR #325, "Communication overlap assessment"): the gate
    // contribution's shard roots, then their rank tree on the handle's second
    // stream while the up contribution's shards are computed here; the final
    // gate-then-up addition waits for both.  Same kernels, same trees, same
    // order of every addition: the same bits as one stream.
    const void *pg[8], *pu[8];
    for (int s = 0; s < k; ++s) {
      pg[s] = w.cgs + (long long)s * M * H;
      pu[s] = w.cus + (long long)s * M * H;
    }
    TRY(tree_gemm_k(h, f, Strided{dG, I, 1}, wcol(WG, 0), M, H, sw, k, w.cgs, H, M * H, st, w.tcs));
    TRYCU(cudaEventRecord(h->ev_fork, st));
    TRYCU(cudaStreamWaitEvent(h->side, h->ev_fork, 0));
    // Once forked, the side stream is joined back whatever fails in between,
    // so that nothing of this call is left running behind `stream`.
    detffn_status side_st = rank_tree_bf16(h, pg, k, w.cg, M * H, h->side);
    const detffn_status rec = cu(cudaEventRecord(h->ev_join, h->side));
    detffn_status main_st = tree_gemm_k(h, f, Strided{dU, I, 1}, wcol(WU, 0), M, H, sw, k, w.cus, H, M * H, st, w.tcs);
    if (main_st == DETFFN_OK) main_st = rank_tree_bf16(h, pu, k, w.cu, M * H, st);
    if (rec == DETFFN_OK) TRYCU(cudaStreamWaitEvent(st, h->ev_join, 0));
    else TRYCU(cudaStreamSynchronize(h->side));
    TRY(side_st);
    TRY(rec);
    TRY(main_st);
  } else {
    // Shard s contracts K positions [s sw, (s+1) sw) of I; all shards' cg and
    // cu subtree roots in one call.
    TRY(tree_gemm2_k(h, f, Strided{dG, I, 1}, wcol(WG, 0), w.cgs, Strided{dU, I, 1}, wcol(WU, 0), w.cus, M, H, sw,
                     k, H, M * H, st, w.tcs));
  }
  if (k > 1 && !(h->flags & DETFFN_FLAG_OVERLAP_DHIDDEN)) {
    const void *pg[8], *pu[8];
    for (int s = 0; s < k; ++s) {
      pg[s] = w.cgs + (long long)s * M * H;
      pu[s] = w.cus + (long long)s * M * H;
    }
    // Both rank trees and the gate-then-up addition in one pass (the same
    // arithmetic as the two trees and then the addition).
    TRY(timed(h, st, "rank_tree_add", 2.0 * (2 * k + 1) * M * H, 0.0, [&] {
      return cu(launch_rank_tree_add_bf16(pg, pu, k, dX, M * H, h->sm_count, st));
    }));
  } else {
    TRY(add_bf16(h, w.cg, w.cu, (uint16_t*)dX, M * H, st));
  }
  return wgrads(h, f, (const uint16_t*)x, (const uint16_t*)dOut, w.h, dU, dG, (uint16_t*)dWg,
                (uint16_t*)dWu, (uint16_t*)dWd, M, H, I, st);
}

extern "C" detffn_status detffn_wgrad_chunked(detffn_handle h, int n_chunks,
                                              const long long* chunk_tokens,
                                              const void* const* x_chunks,
                                              const void* const* gate_chunks,
                                              const void* const* up_chunks,
                                              const void* const* dOut_chunks, const void* Wd,
                                              void* dWg, void* dWu, void* dWd, long long H,
                                              long long I, void* ws, size_t ws_bytes,
                                              void* stream, const detffn_options* opts) {
  if (!h || n_chunks < 1 || !chunk_tokens || !x_chunks || !gate_chunks || !up_chunks ||
      !dOut_chunks || !Wd || !dWg || !dWu || !dWd)
    return DETFFN_ERR_INVALID_ARG;
  Opts o;
  TRY(read_opts(opts, &o));
  set_waits(h, o);
  long long M = 0;
  for (int c = 0; c < n_chunks; ++c) {
    if (chunk_tokens[c] < 0) return DETFFN_ERR_SHAPE;
    if (chunk_tokens[c] > 0 && (!x_chunks[c] || !gate_chunks[c] || !up_chunks[c] || !dOut_chunks[c]))
      return DETFFN_ERR_INVALID_ARG;
    if (!aligned2(x_chunks[c]) || !aligned2(gate_chunks[c]) || !aligned2(up_chunks[c]) ||
        !aligned2(dOut_chunks[c]))
      return DETFFN_ERR_ALIGN;
    M += chunk_tokens[c];
  }
  TRY(check_sizes(M, H, I));
  if (!aligned2(Wd) || !aligned2(dWg) || !aligned2(dWu) || !aligned2(dWd)) return DETFFN_ERR_ALIGN;
  const long long bw = 2 * I * H;
  if (overlap(dWg, bw, dWu, bw) || overlap(dWg, bw, dWd, bw) || overlap(dWu, bw, dWd, bw) ||
      overlap(dWg, bw, Wd, bw) || overlap(dWu, bw, Wd, bw) || overlap(dWd, bw, Wd, bw))
    return DETFFN_ERR_INVALID_ARG;
  Family f;
  TRY(pick_family(o, M, H, I, true, &f));  // by the total token count
  if (f == kTensor && !aligned16(Wd)) {
    if (o.path == DETFFN_PATH_TENSOR) return DETFFN_ERR_ALIGN;
    f = kExact;
  }
  TRY(check_ws(ws, ws_bytes, ws_bytes_for(DETFFN_OP_WGRAD_CHUNKED, M, H, I, 1, f == kTensor, h->sm_count)));
  TRYCU(cudaSetDevice(h->device));
  cudaStream_t st = (cudaStream_t)stream;
  if (M == 0) {
    TRYCU(cudaMemsetAsync(dWg, 0, (size_t)bw, st));
    TRYCU(cudaMemsetAsync(dWu, 0, (size_t)bw, st));
    return cu(cudaMemsetAsync(dWd, 0, (size_t)bw, st));
  }
  Arena a(ws);
  ChunkWs w = plan_chunked(a, M, H, I, f == kTensor, h->sm_count);
  // The row-wise stages (dh, dU, dG and h) run chunk by chunk on each
  // chunk's own rows, reading gate and up where the caller keeps them (a
  // copy first only where a chunk is not 16-byte aligned, which the tensor
  // kernels' TMA needs); x and dOut are gathered in logical token order for
  // the weight gradients, whose K axis is the tokens.
  // On the tensor family the weight gradients read x and dOut chunk by chunk
  // as one K axis (a tensor map per chunk), without gathering them, when
  // every chunk but the last holds a multiple of 64 tokens (no leaf spans
  // two chunks), there are at most 8 non-empty chunks and all are 16-byte
  // aligned; otherwise they are gathered in logical order first.
  TcKChunks kx, kd;
  bool virt = f == kTensor && H % 8 == 0 && M > 64;
  for (int c = 0; c < n_chunks && virt; ++c) {
    const long long t = chunk_tokens[c];
    if (t == 0) continue;
    if (kx.n == kMaxKChunks || !aligned16(x_chunks[c]) || !aligned16(dOut_chunks[c])) {
      virt = false;
      break;
    }
    kx.base[kx.n] = (const uint16_t*)x_chunks[c];
    kd.base[kd.n] = (const uint16_t*)dOut_chunks[c];
    kx.tokens[kx.n++] = t;
    kd.tokens[kd.n++] = t;
  }
  for (int c = 0; c + 1 < kx.n && virt; ++c)
    if (kx.tokens[c] % kLeaf) virt = false;
  long long r0 = 0;
  for (int c = 0; c < n_chunks; ++c) {
    const long long t = chunk_tokens[c];
    if (t == 0) continue;
    if (!virt) {
      TRYCU(cudaMemcpyAsync(w.x + r0 * H, x_chunks[c], (size_t)(2 * t * H), cudaMemcpyDeviceToDevice, st));
      TRYCU(cudaMemcpyAsync(w.dO + r0 * H, dOut_chunks[c], (size_t)(2 * t * H), cudaMemcpyDeviceToDevice, st));
    }
    const uint16_t* dOc = virt ? (const uint16_t*)dOut_chunks[c] : w.dO + r0 * H;
    const uint16_t* gc = (const uint16_t*)gate_chunks[c];
    const uint16_t* uc = (const uint16_t*)up_chunks[c];
    if (!aligned16(gc) || !aligned16(uc)) {
      TRYCU(cudaMemcpyAsync(w.g + r0 * I, gc, (size_t)(2 * t * I), cudaMemcpyDeviceToDevice, st));
      TRYCU(cudaMemcpyAsync(w.u + r0 * I, uc, (size_t)(2 * t * I), cudaMemcpyDeviceToDevice, st));
      gc = w.g + r0 * I;
      uc = w.u + r0 * I;
    }
    TRY(rowwise_bwd(h, f, dOc, (const uint16_t*)Wd, gc, uc, w.dh + r0 * I, w.dU + r0 * I,
                    w.dG + r0 * I, w.h + r0 * I, t, H, I, st, w.tcs));
    r0 += t;
  }
  if (!virt)
    return wgrads(h, f, w.x, w.dO, w.h, w.dU, w.dG, (uint16_t*)dWg, (uint16_t*)dWu, (uint16_t*)dWd, M, H, I,
                  st);
  // dWd[n, i] = T_m(dOut[m, n], h[m, i]): A = dOut, MN-major, in chunks.
  kd.op = 1;
  const double bd = 2.0 * ((double)H * M + (double)I * M + (double)H * I);
  TRY(timed(h, st, "tc_tree_gemm", bd, 2.0 * H * I * M, [&] {
    const TcProblem pd{kd.base[0], H, w.h, I, (uint16_t*)dWd, true, true};
    return cu(launch_tc_gemms(&pd, 1, H, I, M, I, 1, h->wt, h->sm_count, st, nullptr, &kd));
  }));
  // dWg[i, n] = T_m(dG[m, i], x[m, n]), dWu likewise: B = x, MN-major, in chunks.
  kx.op = 2;
  const double bg = 4.0 * ((double)I * M + (double)H * M + (double)I * H);
  return timed(h, st, "tc_tree_gemm", bg, 4.0 * I * H * M, [&] {
    const TcProblem pg[2] = {{w.dG, I, kx.base[0], H, (uint16_t*)dWg, true, true},
                             {w.dU, I, kx.base[0], H, (uint16_t*)dWu, true, true}};
    return cu(launch_tc_gemms(pg, 2, I, H, M, H, 1, h->wt, h->sm_count, st, nullptr, &kx));
  });
}

extern "C" detffn_status detffn_rank_tree_reduce(const void* const* inputs, int n, void* out,
                                                 long long count, int dtype, void* stream) {
  if (!inputs || count < 0) return DETFFN_ERR_INVALID_ARG;
  if (!(n == 1 || n == 2 || n == 4 || n == 8)) return DETFFN_ERR_INVALID_ARG;
  if (dtype < DETFFN_F32 || dtype > DETFFN_BF16) return DETFFN_ERR_INVALID_ARG;
  if (count == 0) return DETFFN_OK;  // empty buffers may have null addresses
  if (!out) return DETFFN_ERR_INVALID_ARG;
  const long long esz = dtype == DETFFN_F32 ? 4 : 2;
  if (((uintptr_t)out % (uintptr_t)esz) != 0) return DETFFN_ERR_ALIGN;
  for (int s = 0; s < n; ++s) {
    if (!inputs[s]) return DETFFN_ERR_INVALID_ARG;
    if (((uintptr_t)inputs[s] % (uintptr_t)esz) != 0) return DETFFN_ERR_ALIGN;
    // In place is allowed only at exactly the same address.
    if (inputs[s] != out && overlap(inputs[s], count * esz, out, count * esz)) return DETFFN_ERR_INVALID_ARG;
  }
  int dev = 0, sms = 0;
  TRYCU(cudaGetDevice(&dev));
  TRYCU(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  return cu(launch_rank_tree(inputs, n, out, count, dtype, sms, (cudaStream_t)stream));
}

extern "C" detffn_status detffn_tree_gemm(detffn_handle h, const void* A, long long a_rs,
                                          long long a_ks, const void* B, long long b_rs,
                                          long long b_ks, long long R, long long C, long long K,
                                          void* out, long long o_rs, void* stream,
                                          const detffn_options* opts) {
  if (!h || !out || R < 0 || C < 0 || K < 0 || K > kMaxK) return DETFFN_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B)) return DETFFN_ERR_INVALID_ARG;
  if (!aligned2(A) || !aligned2(B) || !aligned2(out)) return DETFFN_ERR_ALIGN;
  if (R > 1 && o_rs < C) return DETFFN_ERR_INVALID_ARG;
  Opts o;
  TRY(read_opts(opts, &o));
  set_waits(h, o);
  if (R == 0 || C == 0) return DETFFN_OK;
  Family f = kExact;
  const Strided SA{(const uint16_t*)A, a_rs, a_ks}, SB{(const uint16_t*)B, b_rs, b_ks};
  if (o.path == DETFFN_PATH_TENSOR || (o.path == DETFFN_PATH_AUTO && R > kAutoExactMaxM)) {
    const bool ok = tc_len_ok(K) && (tc_operands_ok(SA) || (tc_mn_ok(SA) && R > 32)) &&
                    (tc_operands_ok(SB) || tc_mn_ok(SB));
    if (ok) f = kTensor;
    else if (o.path == DETFFN_PATH_TENSOR) return DETFFN_ERR_UNSUPPORTED;
  }
  TRYCU(cudaSetDevice(h->device));
  return tree_gemm(h, f, Strided{(const uint16_t*)A, a_rs, a_ks}, Strided{(const uint16_t*)B, b_rs, b_ks},
                   R, C, K, (uint16_t*)out, o_rs, (cudaStream_t)stream);
}

extern "C" detffn_status detffn_tree_gemm_leaves(detffn_handle h, const void* A, long long a_rs,
                                                 long long a_ks, const void* B, long long b_rs,
                                                 long long b_ks, long long R, long long C, long long K,
                                                 void* out, long long o_rs, void* leaves, void* stream,
                                                 const detffn_options* opts) {
  if (!h || !out || !leaves || R < 0 || C < 0 || K <= 0 || K > kMaxK) return DETFFN_ERR_INVALID_ARG;
  if (!A || !B) return DETFFN_ERR_INVALID_ARG;
  if (!aligned2(A) || !aligned2(B) || !aligned2(out) || ((uintptr_t)leaves & 3u)) return DETFFN_ERR_ALIGN;
  if (R > 1 && o_rs < C) return DETFFN_ERR_INVALID_ARG;
  Opts o;
  TRY(read_opts(opts, &o));
  set_waits(h, o);
  if (o.path == DETFFN_PATH_EXACT) return DETFFN_ERR_UNSUPPORTED;  // its leaves are the oracle's order
  if (R == 0 || C == 0) return DETFFN_OK;
  const Strided SA{(const uint16_t*)A, a_rs, a_ks}, SB{(const uint16_t*)B, b_rs, b_ks};
  const bool ok = tc_len_ok(K) && (tc_operands_ok(SA) || (tc_mn_ok(SA) && R > 32)) &&
                  (tc_operands_ok(SB) || tc_mn_ok(SB));
  if (!ok) return DETFFN_ERR_UNSUPPORTED;
  TRYCU(cudaSetDevice(h->device));
  return tree_gemm(h, kTensor, SA, SB, R, C, K, (uint16_t*)out, o_rs, (cudaStream_t)stream, TcsScratch(),
                   (float*)leaves);
}

extern "C" detffn_status detffn_profiling(detffn_handle h, int enable) {
  if (!h) return DETFFN_ERR_INVALID_ARG;
  for (auto& r : h->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  h->recs.clear();
  h->prof = enable != 0;
  return DETFFN_OK;
}

extern "C" detffn_status detffn_profile_read(detffn_handle h, int max, detffn_kernel_time* out, int* n) {
  if (!h || !n || max < 0 || (max > 0 && !out)) return DETFFN_ERR_INVALID_ARG;
  TRYCU(cudaSetDevice(h->device));
  TRYCU(cudaDeviceSynchronize());
  std::vector<detffn_kernel_time> agg;
  for (auto& r : h->recs) {
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, r.a, r.b);
    size_t j = 0;
    while (j < agg.size() && strcmp(agg[j].name, r.name) != 0) ++j;
    if (j == agg.size()) {
      detffn_kernel_time t{};
      strncpy(t.name, r.name, sizeof(t.name) - 1);
      agg.push_back(t);
    }
    agg[j].launches += r.launches;
    agg[j].ms += ms;
    agg[j].bytes += r.bytes;
    agg[j].flops += r.flops;
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  h->recs.clear();
  *n = (int)(agg.size() < (size_t)max ? agg.size() : (size_t)max);
  for (int j = 0; j < *n; ++j) out[j] = agg[j];
  return DETFFN_OK;
}

extern "C" detffn_status detffn_selfcheck_fused_schedule(unsigned long long* cases, unsigned long long* failures) {
  if (!cases || !failures) return DETFFN_ERR_INVALID_ARG;
  *failures = tcs_selfcheck_fused_schedule(cases);
  return DETFFN_OK;
}

extern "C" detffn_status detffn_selfcheck_pieces(int max_levels, unsigned long long* failures) {
  if (!failures || max_levels < 0 || max_levels > kTcsMaxLv) return DETFFN_ERR_INVALID_ARG;
  *failures = tcs_selfcheck_pieces(max_levels);
  return DETFFN_OK;
}

extern "C" detffn_status detffn_cvt_f32_bf16(detffn_handle h, const void* in, void* out, long long n,
                                             void* stream) {
  if (!h || n < 0) return DETFFN_ERR_INVALID_ARG;
  if (n == 0) return DETFFN_OK;
  if (!in || !out) return DETFFN_ERR_INVALID_ARG;
  if (((uintptr_t)in & 3u) || ((uintptr_t)out & 1u)) return DETFFN_ERR_ALIGN;
  if (overlap(in, 4 * n, out, 2 * n)) return DETFFN_ERR_INVALID_ARG;
  TRYCU(cudaSetDevice(h->device));
  return cu(launch_cvt_bf16((const float*)in, (uint16_t*)out, n, h->sm_count, (cudaStream_t)stream));
}

extern "C" detffn_status detffn_selfcheck_node_add(detffn_handle h, unsigned long long* mismatches) {
  if (!h || !mismatches) return DETFFN_ERR_INVALID_ARG;
  TRYCU(cudaSetDevice(h->device));
  // A diagnostic call: an 8-byte device counter, one pass over all 2^32 pairs,
  // then a device synchronisation.
  unsigned long long* d = nullptr;
  TRYCU(cudaMalloc(&d, sizeof(unsigned long long)));
  detffn_status s = cu(cudaMemset(d, 0, sizeof(unsigned long long)));
  if (s == DETFFN_OK) s = cu(launch_check_node_add(0, 1ull << 32, d, h->sm_count, 0));
  if (s == DETFFN_OK) s = cu(cudaDeviceSynchronize());
  if (s == DETFFN_OK) s = cu(cudaMemcpy(mismatches, d, sizeof(unsigned long long), cudaMemcpyDeviceToHost));
  cudaFree(d);
  return s;
}

extern "C" const char* detffn_last_cuda_error(void) {
  const cudaError_t e = g_last_cuda;
  g_last_cuda = cudaSuccess;
  return e == cudaSuccess ? "no CUDA error recorded" : cudaGetErrorString(e);
}
