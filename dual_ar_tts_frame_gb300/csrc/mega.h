// Program and parameters of the persistent frame kernel (mega.cu).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"

namespace dualar {

enum MegaOpType : int {
  MOP_GEMV = 0,
  MOP_ATTN_PAGED = 1,
  MOP_ATTN_FAST = 2,
  MOP_SAMPLE_Q0 = 3,
  MOP_SAMPLE_FAST = 4,
  MOP_FUSION = 5,
};

// One op of the frame program (device memory, built once per batch size).
// Consumers copy the next op into shared memory in 16-byte pieces.
struct alignas(16) MegaOp {
  int type;
  int layer;
  int pos;     // fast attention: codebook position; fast sample: codebook k;
               // GEMV: 1 + layer of the paged attention that follows it (0: none)
  int in_src;  // attention, fast sample: index of the op that wrote the input
  const uint16_t* q_norm;
  const uint16_t* k_norm;
  GemvArgs g;  // MOP_GEMV
};

static_assert(sizeof(MegaOp) % 16 == 0, "copied in 16-byte pieces");

// What the producer needs of one GEMV of the program (GEMV ops only, in
// program order): the weight matrices and their shape.
struct ProdOp {
  const uint16_t* w0;
  const uint16_t* w1;
  int n0, n1, K, mode;
  int w4;   // packed 4-bit rows (gemv.cuh, "4-bit weights")
};

struct MegaParams {
  DevPtrs d;
  const MegaOp* ops;
  int n_ops;
  const ProdOp* prod;       // the GEMV ops of the program, for the producer
  int n_prod;
  int nrows;
  int units, chunk;         // paged-attention work list of this frame
  int kmax;                 // largest GEMV K (shared-memory x rows)
  SampIO io;
  const uint16_t* tok_emb;
  const uint16_t* fusion;
  uint32_t* bar;            // grid-barrier counter, zero at launch
  uint32_t bar_extra;       // test hook: arrivals a barrier waits for beyond the grid (0 normally)
  uint64_t* trace;          // optional: [n_sm][n_ops][4] global-timer stamps (op start, GEMV x staged, GEMV tiles consumed, op end)
  uint64_t prefetch_bytes;  // weight bytes per CTA kept in flight into L2 beyond the ring
  uint32_t epoch;           // launch epoch of the activation tags (1 .. 2^20 - 1)
  int w4;                   // some GEMV of the program reads packed 4-bit rows
};

// Launches the frame program as one cooperative kernel (grid = n_sm CTAs).
// *unsupported is set (and nothing launched) when the batch or head shape has
// no persistent instantiation or the shared-memory plan does not fit.
cudaError_t launch_mega(const MegaParams& p, int nb, int n_sm, cudaStream_t st, bool* unsupported);

}  // namespace dualar
