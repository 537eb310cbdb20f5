// Internal declarations shared by the host runtime (api.cu) and the kernels
// (kernels.cu).  Not part of the public C ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace dualar {

// Launches kern with programmatic stream serialization: it may begin (its
// prologue, loads of constant data) while the previous kernel in the stream
// runs; the kernel calls pdl_wait() before anything that kernel produces.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

constexpr int kMaxRows = 128;        // rows per launch: decode batch or prefill chunk
constexpr int kMaxCodebooks = 16;
constexpr int kRasRing = 16;         // RAS history ring per slot (window <= 16)
constexpr int kMaxChunks = 64;       // split-KV chunks per (row, KV head)
constexpr int kMaxChunkPages = 64;   // pages per split-KV chunk
constexpr int kMaxGroup = 8;         // query heads per KV head
#ifndef DUALAR_GEMV_WARPS
#define DUALAR_GEMV_WARPS 16
#endif
constexpr int kGemvConsumerWarps = DUALAR_GEMV_WARPS;
constexpr int kGemvThreads = (kGemvConsumerWarps + 1) * 32;
constexpr int kSampThreads = 512;

// Device error word: bit flags OR-ed in by kernels, read by dualar_sync.
enum : uint32_t {
  DEV_ERR_MBAR_TIMEOUT = 1u << 0,   // an mbarrier wait gave up
  DEV_ERR_GRID_TIMEOUT = 1u << 1,   // a grid-wide barrier gave up
  DEV_ERR_BAD_INDEX = 1u << 2,      // an index failed its bounds check (access skipped)
  DEV_ERR_BAD_PAGE = 1u << 3,       // a page-table entry was out of range (access skipped)
  DEV_ERR_TC_WAIT = 1u << 4,        // with MBAR_TIMEOUT: in the tensor-core projection (tcgemm.cu)
  DEV_ERR_ATTN_WAIT = 1u << 5,      // with MBAR_TIMEOUT: in the tensor-core attention (attn_mma.cu)
};

// One row of a launch: a sequence (slot) writing one position.
struct RowInfo {
  int32_t slot;
  int32_t pos;
  int32_t active;    // 0: this row's KV writes and state commits are skipped
  int32_t unit0;     // first split-KV attention unit of this row
};

// Passed by value to the setup kernel at the start of every launch sequence.
struct LaunchSetup {
  int32_t n_rows;
  int32_t n_updates;                 // page-table updates
  int32_t commit_last_only;          // prefill: only the last row commits state
  int32_t embed;                     // prefill: gather tok_emb rows into xs
  RowInfo rows[kMaxRows];
  int32_t upd_slot[kMaxRows];
  int32_t upd_index[kMaxRows];
  int32_t upd_page[kMaxRows];
  int32_t tokens[kMaxRows];          // prefill ids (unused in decode)
};

// 4-bit weights: elements per scale group, and bytes of one packed row of K
// elements (K/2 code bytes, K/128 bf16 scales, zero padding to 16 bytes; the
// layout is described in gemv.cuh, "4-bit weights").
constexpr int kW4Group = 128;
__host__ __device__ inline int w4_row_bytes(int K) { return K / 2 + ((K / 64 + 15) & ~15); }

enum GemvMode : int { GEMV_STORE = 0, GEMV_ADD = 1, GEMV_SWIGLU = 2 };

struct GemvArgs {
  const uint16_t* w0;      // [n0][K] bf16 (segment 0, or the gate matrix)
  const uint16_t* w1;      // [n1][K] bf16 (segment 1, or the up matrix)
  int n0, n1;              // rows of the two segments (SWIGLU: n1 = n0)
  int K;
  int mode;
  int nb;                  // activation rows in this launch
  const float* x;          // [nb][ldx] input rows (fp32)
  int ldx;
  const uint16_t* norm_w;  // RMSNorm gain [K] (bf16) applied to x first, or null
  float eps;
  const float* base;       // GEMV_ADD: out = base + W x  (may alias out)
  int ldb;
  float* out;
  int ldo;
  const int32_t* out_map;  // optional: batch row b writes out row out_map[b] (< 0: skip)
  float* save_x;           // optional: CTA 0 stores the normalized x rows here
  const int32_t* save_map; // row map for save_x (< 0: skip)
  int lds;
  uint32_t* err;
  uint64_t wait_limit_ns;
  // Persistent frame kernel only: index of the op that wrote x / base, and of
  // this op (written into out); -1 means a plain fp32 buffer.  With an index
  // the pointer is a tagged 64-bit buffer (common.cuh, "tagged activations")
  // with the same element strides.
  int x_src, base_src, out_src;
  // 1: w0 / w1 hold 4-bit packed weights (gemv.cuh, "4-bit weights")
  // instead of bf16.
  int w4;
  // Persistent kernel, x_src >= 0: with x_scout > 0, warp 0 first waits for
  // the last word of every x_scout-word block of x (one word per lane) while
  // the other consumer warps wait at a barrier; only then do all threads read
  // x.  For inputs that every CTA waits on for a long time (the attention
  // output, written by a few CTAs): a whole CTA polling every word of x
  // crowds the lines that the writers are about to fill.
  int x_scout;
};

// Device buffers of one handle that kernels need (plain pointers).
struct DevPtrs {
  // shapes
  int D, Hq, Hkv, hd, F, n_sem, sem_begin, im_end, Cf, N, page_tokens, pages_per_seq, n_layer,
      fast_n_layer, max_pages, rope_len, max_seqs, qkv_dim, logit_ld;
  float eps;
  // tables and caches
  const uint16_t* rope_cos;   // [rope_len][hd/2] bf16
  const uint16_t* rope_sin;
  uint16_t* kv_pool;          // [max_pages][n_layer][2][Hkv][page_tokens][hd] bf16
  int32_t* page_table;        // [max_seqs][pages_per_seq]
  float* fast_kv;             // [kMaxRows][fast_n_layer][2][Hkv][N][hd] fp32
  // per-slot state
  float* h_last;              // [max_seqs][D]   final-normed hidden of the last position
  float* z_last;              // [max_seqs][n_sem+1] restricted logits
  int32_t* hist;              // [max_seqs][kRasRing]
  int32_t* hist_n;            // [max_seqs]
  int32_t* finished;          // [max_seqs]
  // per-launch rows
  RowInfo* rows;              // [kMaxRows]
  int32_t* commit_map;        // [kMaxRows] slot to commit state to, or -1
  // work buffers
  float* xs;                  // [kMaxRows][D] slow input (fusion / embedding)
  float* hs;                  // [kMaxRows][D] slow residual stream
  float* hf;                  // [kMaxRows][D] fast residual stream
  float* fin;                 // [2][kMaxRows][D] fast-pass inputs
  float* qkv;                 // [kMaxRows][qkv_dim]
  float* qrot;                // [kMaxRows][Hq][hd]
  float* attn;                // [kMaxRows][Hq*hd]
  float* act;                 // [kMaxRows][F]
  float* logits;              // [kMaxRows][logit_ld]
  float* part;                // split-KV partials [kMaxRows][Hkv][kMaxChunks][G][hd+2]
  uint32_t* arrive;           // [kMaxRows][Hkv] last-arriver counters
  uint32_t* sched;            // [n_layer] unit counters of the tensor-core attention (zeroed by setup)
  int32_t* codes_ws;          // [kMaxRows][kMaxCodebooks] codes of the current frame
  uint32_t* err;              // device error word
  uint64_t wait_limit_ns;
  // tagged copies of the work buffers, used by the persistent frame kernel
  // (kTaggedRows rows each, same strides as the fp32 buffers)
  uint64_t* qkv_t;            // [kTaggedRows][qkv_dim]
  uint64_t* attn_t;           // [kTaggedRows][Hq*hd]
  uint64_t* act_t;            // [kTaggedRows][F]
  uint64_t* hs_t;             // [kTaggedRows][D]
  uint64_t* hf_t;             // [kTaggedRows][D]
  uint64_t* xs_t;             // [kTaggedRows][D]
  uint64_t* fin_t;            // [kMaxCodebooks][kTaggedRows][D] input of fast pass p
  uint64_t* logits_t;         // [kTaggedRows][logit_ld]
  uint64_t* part_t;           // split-KV partials [kTaggedRows][Hkv][kMaxChunks][G][hd+2]
};
constexpr int kTaggedRows = 2;   // batch rows of the persistent frame kernel
constexpr int kTagOpBits = 12;   // low bits of an activation tag: index of the writing op

struct SamplingParams {
  float temperature, top_p;
  int32_t ras_win;
  float ras_temperature, ras_top_p;
  int32_t allow_eos;
};

// Per-call sampler arguments (device pointers).
struct SampIO {
  const float* uniforms;
  int ldu;
  SamplingParams sp;
  const int32_t* forced;
  int ldf;
  int32_t* codes_out;
  int32_t* status_out;
  float* slow_logits_out;
  float* fast_logits_out;
  int32_t* draws_out;
  const uint16_t* fast_emb;
};

// Per-op decode path: where the attention also writes the bf16 halves of its
// output for the o projection ([rows][ld]; xh null: nowhere).
struct AttnHalves {
  uint16_t* xh;
  uint16_t* xl;
  int ld;
};

// ---- launchers (kernels.cu) -------------------------------------------------
cudaError_t launch_setup(const LaunchSetup& s, const DevPtrs& d, const uint16_t* tok_emb,
                         cudaStream_t st);
cudaError_t launch_gemv(const GemvArgs& a, int n_sm, cudaStream_t st);
// Packs a bf16 matrix [n][K] (K % 128 == 0) into 4-bit records (gemv.cuh).
cudaError_t launch_quantize_w4(const uint16_t* w, int n, int K, unsigned char* out, cudaStream_t st);
// Packed 4-bit rows [n][record] -> bf16 [n][2K]: each weight q * s as hi in
// column k and lo in column K + k (hi + lo = q * s exactly), queued without
// programmatic dependent launch.
cudaError_t launch_dequant_w4(const void* packed, int n, int K, uint16_t* out, cudaStream_t st);
cudaError_t launch_append(const DevPtrs& d, int nrows, int layer, bool fast, int fast_pos,
                          const uint16_t* q_norm, const uint16_t* k_norm, cudaStream_t st);
cudaError_t launch_attn_paged(const DevPtrs& d, int nrows, int layer, int total_units,
                              int chunk_tokens, int n_sm, bool fuse_append, const uint16_t* q_norm,
                              const uint16_t* k_norm, cudaStream_t st, bool* mma_used = nullptr,
                              AttnHalves hv = AttnHalves{nullptr, nullptr, 0});
// Tensor-core variant for launches of >= kAttnMmaMinRows rows (attn_mma.cu);
// *used is false (nothing launched) when the shape or the driver rules it out.
constexpr int kAttnMmaMinRows = 3;
// Prefill (rows: consecutive positions of one sequence, K/V already
// appended): blocks of rows share every page read (attn_mma.cu).  *used is
// false when the shape or the driver rules it out.
cudaError_t launch_attn_prefill(const DevPtrs& d, int nrows, int layer, int total_units, int chunk_tokens, int n_sm,
                                cudaStream_t st, bool* used);
cudaError_t launch_attn_mma(const DevPtrs& d, int nrows, int layer, int total_units, int chunk_tokens, int n_sm,
                            bool fuse_append, const uint16_t* q_norm, const uint16_t* k_norm, cudaStream_t st,
                            bool* used,
                            AttnHalves hv = AttnHalves{nullptr, nullptr, 0});
cudaError_t launch_attn_fast(const DevPtrs& d, int nrows, int layer, int pos, const uint16_t* q_norm,
                             const uint16_t* k_norm, cudaStream_t st, AttnHalves hv = AttnHalves{nullptr, nullptr, 0});
cudaError_t launch_sample_q0(const DevPtrs& d, int nrows, const float* uniforms, int ldu,
                             const SamplingParams& sp, const int32_t* forced, int ldf,
                             int32_t* codes_out, int32_t* status_out, float* slow_logits_out,
                             int32_t* draws_out, const uint16_t* fast_emb, cudaStream_t st);
cudaError_t launch_sample_fast(const DevPtrs& d, int nrows, int k, const float* uniforms, int ldu,
                               const SamplingParams& sp, const int32_t* forced, int ldf,
                               int32_t* codes_out, float* fast_logits_out, int32_t* draws_out,
                               const uint16_t* fast_emb, cudaStream_t st);
cudaError_t launch_fusion(const DevPtrs& d, int nrows, const uint16_t* tok_emb,
                          const uint16_t* fusion, cudaStream_t st);
cudaError_t launch_synthetic_fill(const DevPtrs& d, int slot, int n_pages, uint32_t seed, int n_sm,
                                  cudaStream_t st);


}  // namespace dualar
