// decode.h -- arguments of the exact weight-streaming decode contraction.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace detffn {

struct DecArgs {
  const uint16_t* x;   // [M, K] tokens, row stride ldx (elements)
  long long ldx;
  const uint16_t* w0;  // [N, K] weight rows, row stride ldw (the gate rows in gate/up mode)
  const uint16_t* w1;  // the up rows in gate/up mode, else nullptr
  long long ldw;
  long long N;         // rows per weight matrix
  long long K;         // contraction length, a multiple of 64
  int M;               // tokens in this pass (<= 8)
  int RT;              // rows per tile (per weight matrix)
  uint16_t* part;      // [NB][MT][rows_total] BF16 block roots (scratch)
  unsigned* cnt;       // [tiles] tickets (scratch, zero on entry, zero on exit)
  uint16_t* out;       // plain mode: C [M, ldo]; gate/up mode: h [M, ldo]
  long long ldo;
  uint16_t* gsave;     // gate/up mode, optional: gate [M, ldo]
  uint16_t* usave;     // gate/up mode, optional: up [M, ldo]
  const uint16_t* silu;
  int* status;
  long long spin_limit;
  int stall;           // test only: issue no copies, so the first wait runs out
};

// Leaf-block geometry for K: fills S (leaves per block), NB (blocks) and
// returns false when the decode kernel does not cover this K (the caller then
// uses the general exact kernel, which gives the same bits).
bool decode_geometry(long long K, int* S, int* NB);

// Elements of the block-root planes for one pass over rows_total rows.
size_t decode_part_elems(long long K, long long rows_total);

// Launches one pass (M <= 8 tokens).  Returns cudaErrorInvalidValue if the
// geometry is not covered.
cudaError_t launch_decode_exact(DecArgs a, int sm_count, cudaStream_t st);

// The library's host copy of the BF16 SiLU table (65536 entries, built once).
const uint16_t* host_silu_table();

}  // namespace detffn
