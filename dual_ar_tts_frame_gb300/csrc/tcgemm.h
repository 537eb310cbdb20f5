// Batched projections on the tensor cores (tcgemm.cu): host interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace dualar {

constexpr int kTcMinRows = 9;      // below this the weight-streaming GEMV (<= 8 rows per pass) is used
constexpr int kTcMaxRows = 128;    // activation rows per launch (the MMA's N <= 128)
constexpr int kTcMaxSlices = 16;   // split-K slices

// Work buffers of one handle.
struct TcBuffers {
  uint16_t* xh;          // [kTcMaxRows][ldx] bf16: high half of x'
  uint16_t* xl;          // [kTcMaxRows][ldx] bf16: low half
  int ldx;               // >= every projection's K
  float* part;           // split-K partial sums
  size_t part_floats;
};

// Whether the driver offers tensor-map encoding (checked once).
bool tc_available();
// Whether a projection can take the tensor-core path: 9..128 plain-buffer
// rows, K a multiple of 64 and <= ldx, segment boundaries on 128 rows.
bool tc_eligible(const GemvArgs& a, int ldx);
// Tensor map of a bf16 matrix [rows][K] (row stride ld elements), tiles of
// box_rows x 64 with 128-byte swizzle; built once per argument set and kept.
bool tc_bf16_map(CUtensorMap* out, const void* base, int K, int rows, int ld, int box_rows);
// A residual-add reduce that has not been queued yet: the split-K partial
// sums of the last projection, to be added to base and stored to out.
struct TcPending {
  bool on = false;
  int slices = 0, nb = 0, ldp = 0, n_out = 0;
  float* out = nullptr;
  int ldo = 0;
  const float* base = nullptr;
  int ldb = 0;
};

// Queues split (unless x_ready: the buffers already hold x's halves), GEMM
// and reduce kernels; split_out: the reduce also writes the output's halves
// (it is the next projection's input, without norm).  With defer (a
// residual-add projection whose output is one of the buffers' row blocks)
// the reduce is not queued but described in *defer: the caller queues it
// later, alone (launch_tc_pending) or fused with the next projection's
// norm and split (launch_tc_reduce_norm).  weights_pdl false: the GEMM is
// launched without programmatic dependent launch (it fetches its weights
// before waiting for the kernel before it, so weights written by that
// kernel need a plain launch).  w_hilo: the weights are [rows][2K], each
// weight's bf16 hi half in column k and lo half in K + k
// (launch_dequant_w4); the GEMM runs over 2K columns with x's column k mod
// K.  *launches += count.
cudaError_t launch_tc_gemm(const GemvArgs& a, const TcBuffers& b, int n_sm, cudaStream_t st, int* launches,
                           bool x_ready = false, bool split_out = false, TcPending* defer = nullptr,
                           bool weights_pdl = true, bool w_hilo = false);
// Whether a deferred reduce can be fused into the split of projection a
// (its input is the pending output, with a norm).
bool tc_can_fuse(const TcPending& p, const GemvArgs& a);
// The pending reduce on its own.
cudaError_t launch_tc_pending(const TcPending& p, const TcBuffers& b, int n_sm, cudaStream_t st);
// The pending reduce, then a's RMSNorm and bf16 halves (and save_x) in the
// same kernel, one CTA per row; a's GEMM then runs with x_ready.
cudaError_t launch_tc_reduce_norm(const TcPending& p, const GemvArgs& a, const TcBuffers& b, cudaStream_t st);

}  // namespace dualar
