// noalloc.cu -- the decode forward for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: for example a process whose device
// memory is already held by a caching allocator (a framework's pool that
// owns nearly all of the GPU), or an embedded runtime that only hands out
// buffers it reserved up front.  detffn_forward needs a caller-provided
// workspace and detffn_create allocates its tables; this entry point needs
// neither.  Its scratch (the hidden activation h, the block-root planes and
// the tickets of the decode kernels) and its SiLU table live in file-scope
// __device__ arrays of fixed size, which every GPU that loads the library
// holds until the process exits.
//
// Host code may not use the arrays' names as device addresses (on the host
// they are stand-ins), so a one-time set-up per device looks up their device
// addresses with cudaGetSymbolAddress, with that device current.
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "decode.h"

namespace detffn {
namespace {

// Limits of this entry point: at most 8 tokens, and contraction lengths the
// weight-streaming decode kernel covers (decode_geometry: 4, 8, 16, 32 or 64
// leaves of 64, or 12, 24, 48, 96 or 192), i.e. 256 <= H, I <= 12288.
constexpr long long kNaMaxM = 8;
constexpr long long kNaMaxH = 12288;
constexpr long long kNaMaxI = 12288;
constexpr long long kNaRows = 2 * kNaMaxI > kNaMaxH ? 2 * kNaMaxI : kNaMaxH;

// Scratch layout (bytes): tickets | status word | block-root planes | h.
// The tickets and the status word are cleared together at the start of
// every call.
constexpr size_t kNaTicketBytes = (size_t)(kNaRows + 1) * sizeof(unsigned);
constexpr size_t kNaStatusOff = (kNaTicketBytes + 255) / 256 * 256;
constexpr size_t kNaPartOff = kNaStatusOff + 256;
constexpr size_t kNaPartBytes = (size_t)64 * kNaRows * sizeof(uint16_t);  // <= 8 blocks x 8 tokens
constexpr size_t kNaHOff = kNaPartOff + kNaPartBytes;
constexpr size_t kNaHBytes = (size_t)kNaMaxM * kNaMaxI * sizeof(uint16_t);
constexpr size_t kNaScratchBytes = kNaHOff + kNaHBytes;  // about 3.3 MiB

static __device__ __align__(256) unsigned char g_na_scratch[kNaScratchBytes];
static __device__ __align__(256) uint16_t g_na_silu[65536];

struct DevState {
  bool ready = false;
  unsigned char* scratch = nullptr;  // device address of g_na_scratch
  uint16_t* silu = nullptr;          // device address of g_na_silu
  int sm_count = 0;
};
constexpr int kNaMaxDevices = 64;
std::mutex g_na_mu;
// Test settings of the failure path (detffn_forward_decode_noalloc_test_waits):
// 0 and 0, the normal path, unless a test set them.
std::atomic<long long> g_na_test_spin{0};
std::atomic<int> g_na_test_stall{0};
DevState g_na_dev[kNaMaxDevices];

// Once per device, with that device current: resolve the arrays' device
// addresses and fill the SiLU table.
detffn_status na_setup(int dev, DevState** out) {
  if (dev < 0 || dev >= kNaMaxDevices) return DETFFN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_na_mu);
  DevState& d = g_na_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_na_scratch) != cudaSuccess || !p) return DETFFN_ERR_CUDA;
    d.scratch = static_cast<unsigned char*>(p);
    p = nullptr;
    if (cudaGetSymbolAddress(&p, g_na_silu) != cudaSuccess || !p) return DETFFN_ERR_CUDA;
    d.silu = static_cast<uint16_t*>(p);
    if (cudaMemcpy(d.silu, host_silu_table(), 65536 * sizeof(uint16_t), cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return DETFFN_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DETFFN_ERR_CUDA;
    d.ready = true;
  }
  *out = &d;
  return DETFFN_OK;
}

bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace detffn

using namespace detffn;

extern "C" detffn_status detffn_forward_decode_noalloc(const void* x, const void* Wg,
                                                       const void* Wu, const void* Wd, void* out,
                                                       long long M, long long H, long long I,
                                                       void* stream) {
  if (!x || !Wg || !Wu || !Wd || !out) return DETFFN_ERR_INVALID_ARG;
  if (M < 1 || M > kNaMaxM || H < 1 || H > kNaMaxH || I < 1 || I > kNaMaxI) return DETFFN_ERR_SHAPE;
  int S, NB;
  if (!decode_geometry(H, &S, &NB) || !decode_geometry(I, &S, &NB)) return DETFFN_ERR_SHAPE;
  if (!al16(x) || !al16(Wg) || !al16(Wu) || !al16(Wd) || ((uintptr_t)out & 1u)) return DETFFN_ERR_ALIGN;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DETFFN_ERR_CUDA;
  DevState* d = nullptr;
  const detffn_status s = na_setup(dev, &d);
  if (s != DETFFN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* tickets = reinterpret_cast<unsigned*>(d->scratch);
  int* status = reinterpret_cast<int*>(d->scratch + kNaStatusOff);
  uint16_t* part = reinterpret_cast<uint16_t*>(d->scratch + kNaPartOff);
  uint16_t* hh = reinterpret_cast<uint16_t*>(d->scratch + kNaHOff);
  // The tickets and the status word must start at zero; the shared array
  // keeps the last call's bytes.  (A wait that runs out in the gate/up launch
  // sets the status word, and the down launch then returns at entry instead
  // of folding unfinished block roots.)
  if (cudaMemsetAsync(tickets, 0, kNaStatusOff + sizeof(int), st) != cudaSuccess) return DETFFN_ERR_CUDA;

  DecArgs a{};
  a.x = static_cast<const uint16_t*>(x); a.ldx = H;
  a.w0 = static_cast<const uint16_t*>(Wg); a.w1 = static_cast<const uint16_t*>(Wu); a.ldw = H;
  a.N = I; a.K = H; a.M = (int)M;
  a.part = part; a.cnt = tickets;
  a.out = hh; a.ldo = I;
  a.silu = d->silu; a.status = status; a.spin_limit = g_na_test_spin.load(); a.stall = g_na_test_stall.load();
  if (launch_decode_exact(a, d->sm_count, st) != cudaSuccess) return DETFFN_ERR_CUDA;

  DecArgs b{};
  b.x = hh; b.ldx = I;
  b.w0 = static_cast<const uint16_t*>(Wd); b.w1 = nullptr; b.ldw = I;
  b.N = H; b.K = I; b.M = (int)M;
  b.part = part; b.cnt = tickets;
  b.out = static_cast<uint16_t*>(out); b.ldo = H;
  b.silu = d->silu; b.status = status; b.spin_limit = g_na_test_spin.load(); b.stall = g_na_test_stall.load();
  if (launch_decode_exact(b, d->sm_count, st) != cudaSuccess) return DETFFN_ERR_CUDA;
  return DETFFN_OK;
}

extern "C" detffn_status detffn_forward_decode_noalloc_status(void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DETFFN_ERR_CUDA;
  DevState* d = nullptr;
  const detffn_status s = na_setup(dev, &d);
  if (s != DETFFN_OK) return s;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DETFFN_ERR_CUDA;
  int* status = reinterpret_cast<int*>(d->scratch + kNaStatusOff);
  int v = 0;
  if (cudaMemcpy(&v, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DETFFN_ERR_CUDA;
  if (v != 0 && cudaMemset(status, 0, sizeof(int)) != cudaSuccess) return DETFFN_ERR_CUDA;
  return v == 0 ? DETFFN_OK : (detffn_status)v;
}

extern "C" detffn_status detffn_forward_decode_noalloc_test_waits(long long spin_limit, int stall) {
  if (spin_limit < 0 || (stall != 0 && stall != 1)) return DETFFN_ERR_INVALID_ARG;
  g_na_test_spin.store(spin_limit);
  g_na_test_stall.store(stall);
  return DETFFN_OK;
}
