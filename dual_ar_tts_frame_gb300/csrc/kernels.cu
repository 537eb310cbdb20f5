// CUDA kernels of the Dual-AR frame decode (sm_103a).
//
// Kernels:
//   setup_kernel        row table, page-table updates, prompt embedding gather
//   gemv_kernel         weight-streaming GEMV: bulk copies (cp.async.bulk) of
//                       contiguous weight tiles into a shared-memory ring,
//                       fp32 dot products, RMSNorm prologue, store / residual /
//                       SwiGLU epilogues, two-segment rows (restricted head)
//   append_kernel       QK-norm + RoPE (bf16 tables) + KV append
//   attn_paged_kernel   split-KV GQA decode attention over 64-token pages,
//                       combined by the last CTA to finish a (row, KV head)
//   attn_fast_kernel    attention over the fast AR's per-frame cache
//   sample_q0_kernel    temperature / top-p draw of q0 + repetition-aware resample
//   sample_fast_kernel  temperature / top-p draw of q1..q(N-1)
//   fusion_kernel       multi-codebook gather-sum
//
// Pages cited (title, section):
//   [P1] "How the Dual-Autoregressive Architecture Works in Fish Speech S2: A Deep Dive"
//   [P2] "Fish Audio S2: a Qwen3-4B on the time axis, four layers on the codebook
//        axis, and tags that are only text"
#include <cfloat>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace dualar {

// ============================================================================
// setup: rows, page tables, prompt embeddings
// ============================================================================
__global__ void setup_kernel(const LaunchSetup s, DevPtrs d, const uint16_t* tok_emb) {
  const int r = blockIdx.x;
  if (r < s.n_rows && threadIdx.x == 0) {
    const RowInfo ri = s.rows[r];
    d.rows[r] = ri;
    const bool commit = ri.active && (!s.commit_last_only || r == s.n_rows - 1);
    d.commit_map[r] = commit ? ri.slot : -1;
  }
  if (r == 0) {
    for (int i = threadIdx.x; i < s.n_updates; i += blockDim.x) {
      const int sl = s.upd_slot[i], ix = s.upd_index[i], pg = s.upd_page[i];
      if (sl < 0 || sl >= d.max_seqs || ix < 0 || ix >= d.pages_per_seq || pg < 0 ||
          pg >= d.max_pages) {
        raise_error(d.err, DEV_ERR_BAD_PAGE);
        continue;
      }
      d.page_table[sl * d.pages_per_seq + ix] = pg;
    }
  }
  if (s.embed && r < s.n_rows) {
    // [P2] "Two autoregressions": prompt positions take the token's row of the
    // language model's embedding; fusion applies to generated frames only.
    const int tok = s.tokens[r];
    if (tok < 0) {
      raise_error(d.err, DEV_ERR_BAD_INDEX);
      return;
    }
    const uint16_t* src = tok_emb + static_cast<size_t>(tok) * d.D;
    for (int k = threadIdx.x; k < d.D; k += blockDim.x)
      d.xs[r * d.D + k] = bf16bits_to_f32(src[k]);
  }
}

cudaError_t launch_setup(const LaunchSetup& s, const DevPtrs& d, const uint16_t* tok_emb,
                         cudaStream_t st) {
  setup_kernel<<<s.n_rows > 0 ? s.n_rows : 1, 256, 0, st>>>(s, d, tok_emb);
  return cudaGetLastError();
}

// ============================================================================
// GEMV: y[b][n] = sum_k W[n][k] x'[b][k], x' = RMSNorm(x) (optional)
// ============================================================================
// Each CTA owns a contiguous range of output rows (balanced to +-1 row) and
// walks it in groups of 8 rows, one row per consumer warp.  K is cut into
// chunks of at most kChunk elements; a ring stage holds one (group, chunk)
// tile: up to 8 row-chunks per matrix (16 for the SwiGLU gate/up pair), each
// fetched by one bulk copy.  A warp accumulates its row over the chunks and
// reduces with shuffles only, so consumer warps never synchronise with each
// other; the producer thread runs ahead by the ring depth.
constexpr int kRowsPerGroup = kGemvConsumerWarps;   // 8
constexpr int kChunk = 2560;                        // elements per row-chunk (one matrix)
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 225 * 1024;             // dynamic shared memory per CTA

struct GemvPlan {
  int kc;          // chunk length (elements, multiple of 8)
  int n_chunks;
  int nmat;        // 1, or 2 for SwiGLU
  int tile_bytes;  // ring stage size
  int stages;
  int nbt;         // activation rows per launch (template)
  size_t smem;
};

// Shared-memory layout of gemv_kernel (offsets in bytes).
__host__ __device__ inline size_t gemv_misc_off() { return 256; }
__host__ __device__ inline size_t gemv_xs_off() { return 256 + 4 * 128; }
__host__ __device__ inline size_t gemv_ring_off(int nbt, int K) {
  return (gemv_xs_off() + sizeof(float) * size_t(nbt) * K + 127) & ~size_t(127);
}

template <int NB>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const GemvArgs a, const int kc, const int n_chunks, const int stages,
                const int tile_bytes) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  float* misc = reinterpret_cast<float*>(smem + gemv_misc_off());
  float* xs = reinterpret_cast<float*>(smem + gemv_xs_off());
  unsigned char* ring = smem + gemv_ring_off(NB, a.K);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int K = a.K;
  const bool swiglu = a.mode == GEMV_SWIGLU;
  const int nmat = swiglu ? 2 : 1;
  const int nv = swiglu ? a.n0 : a.n0 + a.n1;
  const int v_begin = static_cast<int>((static_cast<long long>(blockIdx.x) * nv) / gridDim.x);
  const int v_end = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * nv) / gridDim.x);
  const int n_groups = (v_end - v_begin + kRowsPerGroup - 1) / kRowsPerGroup;
  const int n_tiles = n_groups * n_chunks;
  const size_t slot_bytes = static_cast<size_t>(kc) * 2;   // one row-chunk in a stage

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGemvConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == kGemvConsumerWarps) {
    // ---------------- producer: one thread streams the CTA's weight rows ---
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    for (int t = 0; t < n_tiles; ++t) {
      const int s = t % stages;
      if (t >= stages) {
        if (!mbar_wait(&empty[s], ((t / stages) - 1) & 1, a.err, a.wait_limit_ns)) return;
      }
      const int g = t / n_chunks, c = t % n_chunks;
      const int v0 = v_begin + g * kRowsPerGroup;
      const int rows = min(kRowsPerGroup, v_end - v0);
      const int k0 = c * kc;
      const int len = min(kc, K - k0);
      const uint32_t bytes = static_cast<uint32_t>(len) * 2;
      mbar_arrive_expect_tx(&full[s], bytes * rows * nmat);
      unsigned char* st = ring + static_cast<size_t>(s) * tile_bytes;
      for (int m = 0; m < nmat; ++m) {
        for (int w = 0; w < rows; ++w) {
          const int v = v0 + w;
          const uint16_t* rowp;
          if (swiglu) rowp = (m ? a.w1 : a.w0) + static_cast<size_t>(v) * K;
          else rowp = v < a.n0 ? a.w0 + static_cast<size_t>(v) * K
                               : a.w1 + static_cast<size_t>(v - a.n0) * K;
          bulk_load_g2s(st + (m * kRowsPerGroup + w) * slot_bytes, rowp + k0, bytes, &full[s], pol);
        }
      }
    }
    return;
  }

  // ---------------- consumers ------------------------------------------------
  constexpr int NCT = kGemvConsumerWarps * 32;
  const int nb = a.nb;
  // Stage x (and its RMSNorm) in shared memory.
  float ss[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) ss[b] = 0.f;
  const int K4 = K >> 2;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (b < nb) {
      const float4* src = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(b) * a.ldx);
      float4* dst = reinterpret_cast<float4*>(xs + static_cast<size_t>(b) * K);
      for (int k = tid; k < K4; k += NCT) {
        const float4 v = src[k];
        dst[k] = v;
        ss[b] += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
    }
  }
  if (a.norm_w != nullptr) {
    // [P1] "Fast Transformer": RMSNorm(dim, eps=norm_eps), pre-norm blocks.
    float* red = misc + 8;   // [8 warps][NB]
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float w = warp_sum(ss[b]);
      if (lane == 0) red[warp * NB + b] = w;
    }
    named_barrier(1, NCT);
    if (tid < NB) {
      float t = 0.f;
      for (int w = 0; w < kGemvConsumerWarps; ++w) t += red[w * NB + tid];
      misc[tid] = 1.0f / sqrtf(t / static_cast<float>(K) + a.eps);
    }
    named_barrier(1, NCT);
    for (int b = 0; b < nb; ++b) {
      const float sc = misc[b];
      float* xb = xs + static_cast<size_t>(b) * K;
      for (int k = tid; k < K; k += NCT) xb[k] = (xb[k] * sc) * bf16bits_to_f32(a.norm_w[k]);
    }
  }
  named_barrier(1, NCT);
  if (a.save_x != nullptr && blockIdx.x == 0) {
    for (int b = 0; b < nb; ++b) {
      const int row = a.save_map ? a.save_map[b] : b;
      if (row < 0) continue;
      for (int k = tid; k < K; k += NCT)
        a.save_x[static_cast<size_t>(row) * a.lds + k] = xs[static_cast<size_t>(b) * K + k];
    }
  }

  const float4* xs4 = reinterpret_cast<const float4*>(xs);
  float acc[2][NB];
  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % stages;
    const int g = t / n_chunks, c = t % n_chunks;
    const int v0 = v_begin + g * kRowsPerGroup;
    const int rows = min(kRowsPerGroup, v_end - v0);
    if (c == 0) {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[m][b] = 0.f;
    }
    if (!mbar_wait(&full[s], (t / stages) & 1, a.err, a.wait_limit_ns)) return;
    if (warp < rows) {
      const int k0 = c * kc;
      const int nvec = min(kc, K - k0) >> 3;
      const unsigned char* st = ring + static_cast<size_t>(s) * tile_bytes;
      for (int m = 0; m < nmat; ++m) {
        const uint4* wr = reinterpret_cast<const uint4*>(st + (m * kRowsPerGroup + warp) * slot_bytes);
        float p0[NB], p1[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) p0[b] = p1[b] = 0.f;
        int j = lane;
#pragma unroll 2
        for (; j + 32 < nvec; j += 64) {
          const uint4 w0 = wr[j], w1 = wr[j + 32];
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const size_t xb = (static_cast<size_t>(b) * K + k0) >> 2;
            p0[b] = dot8(w0, xs4[xb + 2 * j], xs4[xb + 2 * j + 1], p0[b]);
            p1[b] = dot8(w1, xs4[xb + 2 * (j + 32)], xs4[xb + 2 * (j + 32) + 1], p1[b]);
          }
        }
        if (j < nvec) {
          const uint4 w0 = wr[j];
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const size_t xb = (static_cast<size_t>(b) * K + k0) >> 2;
            p0[b] = dot8(w0, xs4[xb + 2 * j], xs4[xb + 2 * j + 1], p0[b]);
          }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[m][b] += p0[b] + p1[b];
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (c == n_chunks - 1 && warp < rows) {
      const int n = v0 + warp;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        acc[0][b] = warp_sum(acc[0][b]);
        if (swiglu) acc[1][b] = warp_sum(acc[1][b]);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (lane == b && b < nb) {
          const int orow = a.out_map ? a.out_map[b] : b;
          if (orow >= 0) {
            float* o = a.out + static_cast<size_t>(orow) * a.ldo + n;
            if (a.mode == GEMV_STORE) *o = acc[0][b];
            else if (a.mode == GEMV_ADD) *o = a.base[static_cast<size_t>(orow) * a.ldb + n] + acc[0][b];
            // [P2] "The slow AR is Qwen3-4B": SwiGLU FFN, down(SiLU(gate) * up).
            else *o = silu(acc[0][b]) * acc[1][b];
          }
        }
      }
    }
  }
}

static GemvPlan plan_gemv(int K, int nb, int mode) {
  GemvPlan p;
  p.nmat = mode == GEMV_SWIGLU ? 2 : 1;
  const int kmax = kChunk / p.nmat;
  p.n_chunks = (K + kmax - 1) / kmax;
  p.kc = ((K + p.n_chunks - 1) / p.n_chunks + 7) & ~7;
  p.tile_bytes = (kRowsPerGroup * p.nmat * p.kc * 2 + 127) & ~127;
  int nbt = nb >= 8 ? 8 : nb >= 4 ? 4 : nb >= 2 ? 2 : 1;
  while (true) {
    const size_t ring = gemv_ring_off(nbt, K);
    const long long room = static_cast<long long>(kSmemBudget) - static_cast<long long>(ring);
    int st = room > 0 ? static_cast<int>(room / p.tile_bytes) : 0;
    if (st >= 2 || nbt == 1) {
      p.nbt = nbt;
      p.stages = st > kMaxStages ? kMaxStages : st;
      p.smem = ring + static_cast<size_t>(p.stages) * p.tile_bytes;
      return p;
    }
    nbt >>= 1;
  }
}

template <int NB>
static cudaError_t launch_gemv_nb(const GemvArgs& a, const GemvPlan& p, int grid, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBudget);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  gemv_kernel<NB><<<grid, kGemvThreads, p.smem, st>>>(a, p.kc, p.n_chunks, p.stages, p.tile_bytes);
  return cudaGetLastError();
}

cudaError_t launch_gemv(const GemvArgs& a, int n_sm, cudaStream_t st) {
  if (a.nb <= 0) return cudaSuccess;
  if (a.K % 8 != 0) return cudaErrorInvalidValue;
  const GemvPlan p = plan_gemv(a.K, a.nb, a.mode);
  if (p.stages < 1 || p.smem > static_cast<size_t>(kSmemBudget)) return cudaErrorInvalidValue;
  const int nv = (a.mode == GEMV_SWIGLU) ? a.n0 : a.n0 + a.n1;
  const int grid = nv < n_sm ? nv : n_sm;
  for (int g0 = 0; g0 < a.nb; g0 += p.nbt) {
    GemvArgs s = a;
    s.nb = (a.nb - g0) < p.nbt ? (a.nb - g0) : p.nbt;
    s.x = a.x + static_cast<size_t>(g0) * a.ldx;
    if (a.out_map) {
      s.out_map = a.out_map + g0;
    } else {
      s.out = a.out + static_cast<size_t>(g0) * a.ldo;
      if (a.base) s.base = a.base + static_cast<size_t>(g0) * a.ldb;
    }
    if (a.save_x) {
      if (a.save_map) s.save_map = a.save_map + g0;
      else s.save_x = a.save_x + static_cast<size_t>(g0) * a.lds;
    }
    cudaError_t e;
    switch (p.nbt) {
      case 8: e = launch_gemv_nb<8>(s, p, grid, st); break;
      case 4: e = launch_gemv_nb<4>(s, p, grid, st); break;
      case 2: e = launch_gemv_nb<2>(s, p, grid, st); break;
      default: e = launch_gemv_nb<1>(s, p, grid, st); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ============================================================================
// QK-norm + RoPE + KV append
// ============================================================================
// One warp per head vector.  [P2] "The slow AR is Qwen3-4B": qk-norm in the
// slow AR (not the fast one); "Streaming: whose numbers": bf16 RoPE tables.
// Pairs (2i, 2i+1) rotate by angle pos * base^(-2i/hd).
template <int EPL>
__global__ void append_kernel(DevPtrs d, int layer, int fast, int fast_pos, const uint16_t* q_norm,
                              const uint16_t* k_norm) {
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const RowInfo ri = d.rows[row];
  const int hd = d.hd, half = hd >> 1;
  const int pos = fast ? fast_pos : ri.pos;
  if (pos < 0 || pos >= d.rope_len) {
    if (threadIdx.x == 0) raise_error(d.err, DEV_ERR_BAD_INDEX);
    return;
  }
  const float* qkv = d.qkv + static_cast<size_t>(row) * d.qkv_dim;
  const int nheads = d.Hq + d.Hkv;
  for (int h = warp; h < nheads; h += blockDim.x >> 5) {
    const bool is_q = h < d.Hq;
    const int g = h - d.Hq;
    const float* src = is_q ? qkv + h * hd : qkv + d.Hq * hd + g * hd;
    const uint16_t* nw = is_q ? q_norm : k_norm;
    float v[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) v[j] = src[lane * EPL + j];
    if (nw != nullptr) {
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < EPL; ++j) s += v[j] * v[j];
      s = warp_sum(s);
      const float inv = 1.0f / sqrtf(s / static_cast<float>(hd) + d.eps);
#pragma unroll
      for (int j = 0; j < EPL; ++j) v[j] = (v[j] * inv) * bf16bits_to_f32(nw[lane * EPL + j]);
    }
#pragma unroll
    for (int pp = 0; pp < EPL / 2; ++pp) {
      const int i = (lane * EPL) / 2 + pp;
      const float c = bf16bits_to_f32(d.rope_cos[static_cast<size_t>(pos) * half + i]);
      const float sn = bf16bits_to_f32(d.rope_sin[static_cast<size_t>(pos) * half + i]);
      const float x0 = v[2 * pp], x1 = v[2 * pp + 1];
      v[2 * pp] = x0 * c - x1 * sn;
      v[2 * pp + 1] = x1 * c + x0 * sn;
    }
    if (is_q) {
      float* dst = d.qrot + (static_cast<size_t>(row) * d.Hq + h) * hd;
#pragma unroll
      for (int j = 0; j < EPL; ++j) dst[lane * EPL + j] = v[j];
      continue;
    }
    if (!ri.active) continue;
    const float* vsrc = qkv + d.Hq * hd + d.Hkv * hd + g * hd;
    if (fast) {
      float* kd = d.fast_kv +
                  ((((static_cast<size_t>(row) * d.fast_n_layer + layer) * 2 + 0) * d.Hkv + g) * d.N +
                   pos) * hd;
      float* vd = kd + static_cast<size_t>(d.Hkv) * d.N * hd;
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        kd[lane * EPL + j] = v[j];
        vd[lane * EPL + j] = vsrc[lane * EPL + j];
      }
    } else {
      const int pt = d.page_tokens;
      const int pidx = pos / pt;
      if (pidx >= d.pages_per_seq) {
        if (lane == 0) raise_error(d.err, DEV_ERR_BAD_INDEX);
        continue;
      }
      const int page = d.page_table[ri.slot * d.pages_per_seq + pidx];
      if (page < 0 || page >= d.max_pages) {
        if (lane == 0) raise_error(d.err, DEV_ERR_BAD_PAGE);
        continue;
      }
      uint16_t* kd = d.kv_pool +
                     (((static_cast<size_t>(page) * d.n_layer + layer) * 2 + 0) * d.Hkv + g) *
                         static_cast<size_t>(pt) * hd +
                     static_cast<size_t>(pos % pt) * hd;
      uint16_t* vd = kd + static_cast<size_t>(d.Hkv) * pt * hd;
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        kd[lane * EPL + j] = f32_to_bf16bits(v[j]);
        vd[lane * EPL + j] = f32_to_bf16bits(vsrc[lane * EPL + j]);
      }
    }
  }
}

cudaError_t launch_append(const DevPtrs& d, int nrows, int layer, bool fast, int fast_pos,
                          const uint16_t* q_norm, const uint16_t* k_norm, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  if (d.hd == 128)
    append_kernel<4><<<nrows, 256, 0, st>>>(d, layer, fast ? 1 : 0, fast_pos, q_norm, k_norm);
  else if (d.hd == 64)
    append_kernel<2><<<nrows, 256, 0, st>>>(d, layer, fast ? 1 : 0, fast_pos, q_norm, k_norm);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// ============================================================================
// Paged split-KV decode attention
// ============================================================================
// A unit is (row, KV head g, chunk c of chunk_tokens positions).  The unit
// computes softmax(q K^T / sqrt(hd)) V for the G query heads of g over its
// chunk with a running max; the last unit of (row, g) to finish merges the
// chunks in chunk order (deterministic).  [P2] fact table: 32 query heads
// over 8 KV heads.
constexpr int kAttnThreads = 256;
constexpr int kPageTokens = 64;

template <int HD, int G>
__global__ void __launch_bounds__(kAttnThreads)
    attn_paged_kernel(DevPtrs d, int nrows, int layer, int total_units, int chunk_tokens) {
  constexpr int QD = HD / 4;              // dims per thread in the score pass
  constexpr int PARTS = kAttnThreads / HD;  // token groups in the value pass
  constexpr int TPP = kPageTokens / PARTS;  // tokens per group
  __shared__ float qs[G][4][QD + 1];
  __shared__ float sc[G][kPageTokens];
  __shared__ float scl[G], msm[G], lsm[G];
  __shared__ float ored[PARTS][G][HD];
  __shared__ int s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hq = d.Hq, hkv = d.Hkv;
  const float qscale = 1.0f / sqrtf(static_cast<float>(HD));
  const size_t page_stride = static_cast<size_t>(kPageTokens) * HD;

  for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
    // row of this unit: rows are sorted by unit0
    int lo = 0, hi = nrows - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (d.rows[mid].unit0 <= u) lo = mid;
      else hi = mid - 1;
    }
    const int r = lo;
    const RowInfo ri = d.rows[r];
    const int L = ri.pos + 1;
    const int nch = (L + chunk_tokens - 1) / chunk_tokens;
    const int local = u - ri.unit0;
    const int g = local / nch, c = local % nch;
    if (!ri.active || g >= hkv) continue;
    const int t0 = c * chunk_tokens;
    const int t1 = min(L, t0 + chunk_tokens);

    for (int e = tid; e < G * HD; e += kAttnThreads) {
      const int h = e / HD, dd = e % HD;
      qs[h][dd / QD][dd % QD] = d.qrot[(static_cast<size_t>(r) * hq + g * G + h) * HD + dd] * qscale;
    }
    if (tid < G) {
      msm[tid] = -INFINITY;
      lsm[tid] = 0.f;
    }
    float o[G];
#pragma unroll
    for (int h = 0; h < G; ++h) o[h] = 0.f;
    __syncthreads();

    const int tok = tid >> 2, qd = tid & 3;
    const int vd = tid % HD, vpart = tid / HD;
    for (int ps = t0; ps < t1; ps += kPageTokens) {
      const int page = d.page_table[ri.slot * d.pages_per_seq + ps / kPageTokens];
      const bool page_ok = page >= 0 && page < d.max_pages;
      if (!page_ok && tid == 0) raise_error(d.err, DEV_ERR_BAD_PAGE);
      const int ntok = page_ok ? min(kPageTokens, t1 - ps) : 0;
      const uint16_t* kp =
          d.kv_pool + (((static_cast<size_t>(page_ok ? page : 0) * d.n_layer + layer) * 2 + 0) * hkv + g) *
                          page_stride;
      const uint16_t* vp = kp + static_cast<size_t>(hkv) * page_stride;
      // scores
      float s[G];
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = 0.f;
      if (tok < ntok) {
        const uint4* k4 = reinterpret_cast<const uint4*>(kp + static_cast<size_t>(tok) * HD + qd * QD);
#pragma unroll
        for (int v8 = 0; v8 < QD / 8; ++v8) {
          const uint4 w = k4[v8];
          const float kf[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                               bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int j = 0; j < 8; ++j) s[h] = fmaf(qs[h][qd][v8 * 8 + j], kf[j], s[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        s[h] += __shfl_xor_sync(0xFFFFFFFFu, s[h], 1);
        s[h] += __shfl_xor_sync(0xFFFFFFFFu, s[h], 2);
      }
      if (qd == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h][tok] = tok < ntok ? s[h] : -INFINITY;
      }
      __syncthreads();
      if (warp < G && ntok > 0) {
        const int h = warp;
        const float a0 = sc[h][lane], a1 = sc[h][lane + 32];
        const float mx = warp_max(fmaxf(a0, a1));
        const float mold = msm[h];
        const float mnew = fmaxf(mold, mx);
        const float p0 = lane < ntok ? expf(a0 - mnew) : 0.f;
        const float p1 = lane + 32 < ntok ? expf(a1 - mnew) : 0.f;
        sc[h][lane] = p0;
        sc[h][lane + 32] = p1;
        const float sum = warp_sum(p0 + p1);
        if (lane == 0) {
          const float f = expf(mold - mnew);   // 0 for the first page (mold = -inf)
          scl[h] = f;
          lsm[h] = lsm[h] * f + sum;
          msm[h] = mnew;
        }
      }
      __syncthreads();
      if (ntok > 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) o[h] *= scl[h];
        const int tb = vpart * TPP, te = min(ntok, tb + TPP);
        for (int t = tb; t < te; ++t) {
          const float v = bf16bits_to_f32(vp[static_cast<size_t>(t) * HD + vd]);
#pragma unroll
          for (int h = 0; h < G; ++h) o[h] = fmaf(sc[h][t], v, o[h]);
        }
      }
      __syncthreads();
    }
    // merge the token groups
#pragma unroll
    for (int h = 0; h < G; ++h) ored[vpart][h][vd] = o[h];
    __syncthreads();
    if (nch == 1) {
      for (int e = tid; e < G * HD; e += kAttnThreads) {
        const int h = e / HD, dd = e % HD;
        float t = 0.f;
#pragma unroll
        for (int p = 0; p < PARTS; ++p) t += ored[p][h][dd];
        d.attn[static_cast<size_t>(r) * hq * HD + (g * G + h) * HD + dd] = t / lsm[h];
      }
      __syncthreads();
      continue;
    }
    float* pw = d.part + ((static_cast<size_t>(r) * hkv + g) * kMaxChunks + c) * G * (HD + 2);
    for (int e = tid; e < G * HD; e += kAttnThreads) {
      const int h = e / HD, dd = e % HD;
      float t = 0.f;
#pragma unroll
      for (int p = 0; p < PARTS; ++p) t += ored[p][h][dd];
      pw[h * (HD + 2) + dd] = t;
    }
    if (tid < G) {
      pw[tid * (HD + 2) + HD] = msm[tid];
      pw[tid * (HD + 2) + HD + 1] = lsm[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const uint32_t old = atomic_add_acq_rel_gpu(&d.arrive[r * hkv + g], 1u);
      s_last = (old == static_cast<uint32_t>(nch - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (s_last) {
      __threadfence();
      const float* pb = d.part + (static_cast<size_t>(r) * hkv + g) * kMaxChunks * G * (HD + 2);
      for (int e = tid; e < G * HD; e += kAttnThreads) {
        const int h = e / HD, dd = e % HD;
        float M = -INFINITY;
        for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(pb + (cc * G + h) * (HD + 2) + HD));
        float Ls = 0.f, Os = 0.f;
        for (int cc = 0; cc < nch; ++cc) {
          const float* q = pb + (cc * G + h) * (HD + 2);
          const float f = expf(__ldcg(q + HD) - M);
          Ls += __ldcg(q + HD + 1) * f;
          Os += __ldcg(q + dd) * f;
        }
        d.attn[static_cast<size_t>(r) * hq * HD + (g * G + h) * HD + dd] = Os / Ls;
      }
      if (tid == 0) d.arrive[r * hkv + g] = 0u;
    }
    __syncthreads();
  }
}

template <int HD>
static cudaError_t attn_paged_hd(const DevPtrs& d, int nrows, int layer, int units, int chunk,
                                 int grid, cudaStream_t st) {
  const int G = d.Hq / d.Hkv;
  switch (G) {
    case 1: attn_paged_kernel<HD, 1><<<grid, kAttnThreads, 0, st>>>(d, nrows, layer, units, chunk); break;
    case 2: attn_paged_kernel<HD, 2><<<grid, kAttnThreads, 0, st>>>(d, nrows, layer, units, chunk); break;
    case 4: attn_paged_kernel<HD, 4><<<grid, kAttnThreads, 0, st>>>(d, nrows, layer, units, chunk); break;
    case 8: attn_paged_kernel<HD, 8><<<grid, kAttnThreads, 0, st>>>(d, nrows, layer, units, chunk); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_paged(const DevPtrs& d, int nrows, int layer, int total_units,
                              int chunk_tokens, int n_sm, cudaStream_t st) {
  if (nrows <= 0 || total_units <= 0) return cudaSuccess;
  if (d.page_tokens != kPageTokens || chunk_tokens % kPageTokens != 0) return cudaErrorInvalidValue;
  const int grid = total_units < 4 * n_sm ? total_units : 4 * n_sm;
  if (d.hd == 128) return attn_paged_hd<128>(d, nrows, layer, total_units, chunk_tokens, grid, st);
  if (d.hd == 64) return attn_paged_hd<64>(d, nrows, layer, total_units, chunk_tokens, grid, st);
  return cudaErrorInvalidValue;
}

// ============================================================================
// Fast-AR attention over the per-frame codebook cache (<= N positions)
// ============================================================================
// [P2] "Two autoregressions": the fast AR's KV cache is num_codebooks long
// and is overwritten every frame.
template <int EPL>
__global__ void attn_fast_kernel(DevPtrs d, int nrows, int layer, int npos) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x * (blockDim.x >> 5) + warp;
  const int hq = d.Hq, hd = d.hd;
  if (unit >= nrows * hq) return;
  const int r = unit / hq, h = unit % hq;
  const int g = h / (hq / d.Hkv);
  const float* q = d.qrot + (static_cast<size_t>(r) * hq + h) * hd;
  const float* kb = d.fast_kv +
                    (((static_cast<size_t>(r) * d.fast_n_layer + layer) * 2 + 0) * d.Hkv + g) * d.N * hd;
  const float* vb = kb + static_cast<size_t>(d.Hkv) * d.N * hd;
  float s = -INFINITY;
  if (lane < npos) {
    float t = 0.f;
    const float* kr = kb + static_cast<size_t>(lane) * hd;
    for (int e = 0; e < hd; ++e) t = fmaf(q[e], kr[e], t);
    s = t * (1.0f / sqrtf(static_cast<float>(hd)));
  }
  const float m = warp_max(s);
  const float p = lane < npos ? expf(s - m) : 0.f;
  const float l = warp_sum(p);
  float o[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) o[j] = 0.f;
  for (int t = 0; t < npos; ++t) {
    const float pt = __shfl_sync(0xFFFFFFFFu, p, t);
#pragma unroll
    for (int j = 0; j < EPL; ++j) o[j] = fmaf(pt, vb[static_cast<size_t>(t) * hd + lane * EPL + j], o[j]);
  }
  float* dst = d.attn + static_cast<size_t>(r) * hq * hd + h * hd;
#pragma unroll
  for (int j = 0; j < EPL; ++j) dst[lane * EPL + j] = o[j] / l;
}

cudaError_t launch_attn_fast(const DevPtrs& d, int nrows, int layer, int npos, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  const int units = nrows * d.Hq;
  const int grid = (units + 7) / 8;
  if (d.hd == 128) attn_fast_kernel<4><<<grid, 256, 0, st>>>(d, nrows, layer, npos);
  else if (d.hd == 64) attn_fast_kernel<2><<<grid, 256, 0, st>>>(d, nrows, layer, npos);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// ============================================================================
// Sampler: temperature + top-p on caller uniforms, one CTA per row
// ============================================================================
// Candidates are ordered by (logit descending, token id ascending), encoded
// as unique 64-bit keys.  Probability mass is integer fixed point
// (exp((z - zmax) / T) * 2^40, rounded), so every sum is exact and the
// result does not depend on the order of the atomics.  The top-p cut and the
// draw are both "first candidate in key order whose cumulative mass reaches
// a target", found by a radix descent over the key bytes with mass
// histograms.  [P2] "Two autoregressions": sample(biased_logits, ...) for
// q0, unmasked sample(logits, ...) for q1..q9.
constexpr int kSampWarps = kSampThreads / 32;

struct SampShared {
  unsigned long long hmass[256];
  unsigned int hcnt[256];
  unsigned long long red64[kSampWarps];
  float redf[kSampWarps];
  unsigned long long bc[6];
  int ibc[4];
};

struct Cands {
  int n;          // number of candidates
  int n_main;     // candidates 0..n_main-1 have ids id_base + i
  int id_base;
  int extra_id;   // candidate n_main (when n > n_main)
};

DEVI uint32_t ord_f32(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);   // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

DEVI int cand_id(const Cands& c, int i) { return i < c.n_main ? c.id_base + i : c.extra_id; }

DEVI int key_to_index(const Cands& c, unsigned long long key) {
  const int id = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
  if (c.n > c.n_main && id == c.extra_id) return c.n_main;
  return id - c.id_base;
}

DEVI float block_max_f(float v, SampShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  if (lane == 0) sh.redf[warp] = v;
  __syncthreads();
  float t = sh.redf[0];
  for (int w = 1; w < kSampWarps; ++w) t = fmaxf(t, sh.redf[w]);
  __syncthreads();
  return t;
}

DEVI unsigned long long block_sum_u64(unsigned long long v, SampShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (lane == 0) sh.red64[warp] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < kSampWarps; ++w) t += sh.red64[w];
  __syncthreads();
  return t;
}

DEVI unsigned long long block_max_u64(unsigned long long v, SampShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  if (lane == 0) sh.red64[warp] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < kSampWarps; ++w) t = sh.red64[w] > t ? sh.red64[w] : t;
  __syncthreads();
  return t;
}

// First key (descending) whose inclusive cumulative mass reaches target
// (1 <= target <= total).  Also returns the mass strictly before it and its
// own mass.
DEVI unsigned long long select_by_mass(const unsigned long long (&key)[kSampPerThread],
                                       const unsigned long long (&mass)[kSampPerThread], int n,
                                       unsigned long long target, SampShared& sh,
                                       unsigned long long* above_out,
                                       unsigned long long* mass_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long prefix = 0, above = 0, result = 0;
  for (int shift = 56;; shift -= 8) {
    for (int i = tid; i < 256; i += kSampThreads) {
      sh.hmass[i] = 0;
      sh.hcnt[i] = 0;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kSampPerThread; ++e) {
      const int i = tid + e * kSampThreads;
      if (i < n) {
        const unsigned long long k = key[e];
        if (shift == 56 || (k >> (shift + 8)) == prefix) {
          const int bin = static_cast<int>((k >> shift) & 255ull);
          atomicAdd(&sh.hmass[bin], mass[e]);
          atomicAdd(&sh.hcnt[bin], 1u);
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l (descending)
      unsigned long long m8[8];
      unsigned long long tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        m8[j] = sh.hmass[255 - 8 * lane - j];
        tot += m8[j];
      }
      unsigned long long incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned long long excl = incl - tot;
      const unsigned long long need = target - above;   // >= 1
      if (excl < need && need <= incl) {
        unsigned long long cc = excl;   // mass before bin jb
        int jb = 7;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cc + m8[j] >= need) {
            jb = j;
            break;
          }
          cc += m8[j];
        }
        const int bin = 255 - 8 * lane - jb;
        sh.ibc[0] = bin;
        sh.bc[0] = above + cc;
        sh.ibc[1] = static_cast<int>(sh.hcnt[bin]);
        sh.bc[1] = sh.hmass[bin];
      }
    }
    __syncthreads();
    const int bin = sh.ibc[0];
    const int cnt = sh.ibc[1];
    above = sh.bc[0];
    const unsigned long long mbin = sh.bc[1];
    prefix = (shift == 56) ? static_cast<unsigned long long>(bin)
                           : ((prefix << 8) | static_cast<unsigned long long>(bin));
    if (shift == 0) {
      result = prefix;
      *mass_out = mbin;
      break;
    }
    if (cnt == 1) {
#pragma unroll
      for (int e = 0; e < kSampPerThread; ++e) {
        const int i = tid + e * kSampThreads;
        if (i < n && (key[e] >> shift) == prefix) sh.bc[2] = key[e];
      }
      __syncthreads();
      result = sh.bc[2];
      *mass_out = mbin;
      break;
    }
    __syncthreads();
  }
  __syncthreads();
  *above_out = above;
  return result;
}

// One draw: returns the chosen candidate index.
DEVI int sample_draw(const float (&z)[kSampPerThread], const unsigned long long (&key)[kSampPerThread],
                     const Cands& c, float temperature, float top_p, float u, SampShared& sh) {
  const int tid = threadIdx.x;
  if (!(temperature > 0.f)) {
    unsigned long long best = 0;
#pragma unroll
    for (int e = 0; e < kSampPerThread; ++e)
      if (tid + e * kSampThreads < c.n && key[e] > best) best = key[e];
    return key_to_index(c, block_max_u64(best, sh));
  }
  float zmax = -INFINITY;
#pragma unroll
  for (int e = 0; e < kSampPerThread; ++e)
    if (tid + e * kSampThreads < c.n) zmax = fmaxf(zmax, z[e]);
  zmax = block_max_f(zmax, sh);
  unsigned long long mass[kSampPerThread];
  unsigned long long local = 0;
#pragma unroll
  for (int e = 0; e < kSampPerThread; ++e) {
    mass[e] = 0;
    if (tid + e * kSampThreads < c.n) {
      const float p = expf((z[e] - zmax) / temperature);
      mass[e] = __float2ull_rn(p * 1099511627776.0f);   // * 2^40
      local += mass[e];
    }
  }
  const unsigned long long Z = block_sum_u64(local, sh);
  unsigned long long tc = Z;
  if (top_p < 1.0f) {
    const double t = ceil(static_cast<double>(top_p) * static_cast<double>(Z));
    tc = t < 1.0 ? 1ull : static_cast<unsigned long long>(t);
    if (tc > Z) tc = Z;
  }
  unsigned long long above, mk;
  select_by_mass(key, mass, c.n, tc, sh, &above, &mk);
  const unsigned long long zk = above + mk;
  unsigned long long td = static_cast<unsigned long long>(floor(static_cast<double>(u) * static_cast<double>(zk))) + 1ull;
  if (td > zk) td = zk;
  if (td < 1ull) td = 1ull;
  const unsigned long long kd = select_by_mass(key, mass, c.n, td, sh, &above, &mk);
  return key_to_index(c, kd);
}

DEVI void load_candidates(const float* src, const Cands& c, float (&z)[kSampPerThread],
                          unsigned long long (&key)[kSampPerThread]) {
#pragma unroll
  for (int e = 0; e < kSampPerThread; ++e) {
    const int i = threadIdx.x + e * kSampThreads;
    z[e] = -INFINITY;
    key[e] = 0;
    if (i < c.n) {
      z[e] = src[i];
      key[e] = (static_cast<unsigned long long>(ord_f32(z[e])) << 32) |
               static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(cand_id(c, i)));
    }
  }
}

__global__ void __launch_bounds__(kSampThreads)
    sample_q0_kernel(DevPtrs d, const float* uniforms, int ldu, SamplingParams sp,
                     const int32_t* forced, int ldf, int32_t* codes_out, int32_t* status_out,
                     float* slow_logits_out, int32_t* draws_out, const uint16_t* fast_emb) {
  __shared__ SampShared sh;
  __shared__ int s_commit, s_active;
  const int row = blockIdx.x, tid = threadIdx.x;
  const RowInfo ri = d.rows[row];
  const int slot = ri.slot;
  const int ns = d.n_sem, N = d.N;
  const float* zsrc = d.z_last + static_cast<size_t>(slot) * (ns + 1);
  if (slow_logits_out)
    for (int i = tid; i < ns + 1; i += kSampThreads)
      slow_logits_out[static_cast<size_t>(row) * (ns + 1) + i] = zsrc[i];
  if (d.finished[slot]) {
    // a finished slot stays finished: no codes, no state change
    if (tid == 0) {
      status_out[row] = 2;
      d.rows[row].active = 0;
      d.commit_map[row] = -1;
    }
    for (int k = tid; k < N; k += kSampThreads) codes_out[row * N + k] = -1;
    return;
  }
  // [P2] "Two autoregressions": the bias keeps the semantic ids and <|im_end|>.
  Cands c{ns + (sp.allow_eos ? 1 : 0), ns, d.sem_begin, d.im_end};
  float z[kSampPerThread];
  unsigned long long key[kSampPerThread];
  load_candidates(zsrc, c, z, key);
  const float* u = uniforms + static_cast<size_t>(row) * ldu;
  const int normal = sample_draw(z, key, c, sp.temperature, sp.top_p, u[0], sh);
  // [P2] "Two autoregressions": a second draw at temperature 1.0, top-p 0.9,
  // used when the normal draw repeats a semantic token of the last 10 frames.
  const int ras = sample_draw(z, key, c, sp.ras_temperature, sp.ras_top_p, u[1], sh);
  if (tid == 0) {
    const int hn = d.hist_n[slot];
    const int w = min(sp.ras_win, hn);
    bool repeat = false;
    if (normal != ns)
      for (int j = 0; j < w; ++j)
        if (d.hist[slot * kRasRing + ((hn - 1 - j) % kRasRing)] == normal) repeat = true;
    const int chosen = (sp.ras_win > 0 && repeat) ? ras : normal;
    const int commit = forced ? forced[static_cast<size_t>(row) * ldf] : chosen;
    if (draws_out) {
      draws_out[row * (N + 2) + 0] = normal;
      draws_out[row * (N + 2) + 1] = ras;
      draws_out[row * (N + 2) + 2] = chosen;
    }
    int active = 1;
    if (commit == ns || commit < 0 || commit > ns) {
      if (commit != ns) raise_error(d.err, DEV_ERR_BAD_INDEX);
      status_out[row] = 1;
      d.finished[slot] = 1;
      d.rows[row].active = 0;
      d.commit_map[row] = -1;
      active = 0;
    } else {
      status_out[row] = 0;
      d.hist[slot * kRasRing + (hn % kRasRing)] = commit;
      d.hist_n[slot] = hn + 1;
      d.codes_ws[row * kMaxCodebooks] = commit;
    }
    s_commit = commit;
    s_active = active;
  }
  __syncthreads();
  if (!s_active) {
    for (int k = tid; k < N; k += kSampThreads) codes_out[row * N + k] = -1;
    return;
  }
  if (tid == 0) codes_out[row * N] = s_commit;
  // fast pass 0 reads the slow hidden state; pass 1 the embedding of q0
  // ([P2] "Two autoregressions", decode_one_token_ar).  q0 indexes the fast
  // embedding clamped to its rows (a no-op when n_sem == fast_vocab).
  const int D = d.D;
  const int e0 = min(s_commit, d.Cf - 1);
  float* f0 = d.fin + static_cast<size_t>(row) * D;
  float* f1 = d.fin + (static_cast<size_t>(kMaxRows) + row) * D;
  const float* hl = d.h_last + static_cast<size_t>(slot) * D;
  const uint16_t* er = fast_emb + static_cast<size_t>(e0) * D;
  for (int k = tid; k < D; k += kSampThreads) {
    f0[k] = hl[k];
    f1[k] = bf16bits_to_f32(er[k]);
  }
}

__global__ void __launch_bounds__(kSampThreads)
    sample_fast_kernel(DevPtrs d, int k, const float* uniforms, int ldu, SamplingParams sp,
                       const int32_t* forced, int ldf, int32_t* codes_out, float* fast_logits_out,
                       int32_t* draws_out, const uint16_t* fast_emb) {
  __shared__ SampShared sh;
  __shared__ int s_commit;
  const int row = blockIdx.x, tid = threadIdx.x;
  const int N = d.N, Cf = d.Cf;
  const float* zs = d.logits + static_cast<size_t>(row) * d.logit_ld;
  if (fast_logits_out)
    for (int i = tid; i < Cf; i += kSampThreads)
      fast_logits_out[(static_cast<size_t>(row) * (N - 1) + (k - 1)) * Cf + i] = zs[i];
  if (!d.rows[row].active) return;
  Cands c{Cf, Cf, 0, -1};
  float z[kSampPerThread];
  unsigned long long key[kSampPerThread];
  load_candidates(zs, c, z, key);
  const float* u = uniforms + static_cast<size_t>(row) * ldu;
  const int draw = sample_draw(z, key, c, sp.temperature, sp.top_p, u[k + 1], sh);
  if (tid == 0) {
    int commit = forced ? forced[static_cast<size_t>(row) * ldf + k] : draw;
    if (commit < 0 || commit >= Cf) {
      raise_error(d.err, DEV_ERR_BAD_INDEX);
      commit = 0;
    }
    if (draws_out) draws_out[row * (N + 2) + k + 2] = draw;
    d.codes_ws[row * kMaxCodebooks + k] = commit;
    codes_out[row * N + k] = commit;
    s_commit = commit;
  }
  __syncthreads();
  if (k + 1 < N) {
    const int D = d.D;
    float* f = d.fin + (static_cast<size_t>((k + 1) & 1) * kMaxRows + row) * D;
    const uint16_t* er = fast_emb + static_cast<size_t>(s_commit) * D;
    for (int j = tid; j < D; j += kSampThreads) f[j] = bf16bits_to_f32(er[j]);
  }
}

cudaError_t launch_sample_q0(const DevPtrs& d, int nrows, const float* uniforms, int ldu,
                             const SamplingParams& sp, const int32_t* forced, int ldf,
                             int32_t* codes_out, int32_t* status_out, float* slow_logits_out,
                             int32_t* draws_out, const uint16_t* fast_emb, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  sample_q0_kernel<<<nrows, kSampThreads, 0, st>>>(d, uniforms, ldu, sp, forced, ldf, codes_out,
                                                   status_out, slow_logits_out, draws_out, fast_emb);
  return cudaGetLastError();
}

cudaError_t launch_sample_fast(const DevPtrs& d, int nrows, int k, const float* uniforms, int ldu,
                               const SamplingParams& sp, const int32_t* forced, int ldf,
                               int32_t* codes_out, float* fast_logits_out, int32_t* draws_out,
                               const uint16_t* fast_emb, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  sample_fast_kernel<<<nrows, kSampThreads, 0, st>>>(d, k, uniforms, ldu, sp, forced, ldf, codes_out,
                                                     fast_logits_out, draws_out, fast_emb);
  return cudaGetLastError();
}

// ============================================================================
// Multi-codebook fusion
// ============================================================================
// [P2] "Two autoregressions", Eq. 1 and the code's scale:
//   x_{t+1} = (e_LM[q0] + sum_{k<N} E^(k)[q_k]) / sqrt(N+1)
// with E^(k) the block of the fusion table that starts at row
// n_sem + (k-1) * fast_vocab (row 0 for k = 0).
__global__ void fusion_kernel(DevPtrs d, const uint16_t* tok_emb, const uint16_t* fusion) {
  const int row = blockIdx.x;
  if (!d.rows[row].active) return;
  const int D = d.D, N = d.N;
  __shared__ const uint16_t* src[kMaxCodebooks + 1];
  __shared__ int bad;
  if (threadIdx.x == 0) {
    bad = 0;
    const int* q = d.codes_ws + row * kMaxCodebooks;
    if (q[0] < 0 || q[0] >= d.n_sem) bad = 1;
    src[0] = tok_emb + static_cast<size_t>(d.sem_begin + q[0]) * D;
    for (int k = 0; k < N; ++k) {
      const int lim = k == 0 ? d.n_sem : d.Cf;
      if (q[k] < 0 || q[k] >= lim) bad = 1;
      const int off = k == 0 ? 0 : d.n_sem + (k - 1) * d.Cf;
      src[k + 1] = fusion + static_cast<size_t>(off + q[k]) * D;
    }
    if (bad) raise_error(d.err, DEV_ERR_BAD_INDEX);
  }
  __syncthreads();
  if (bad) return;
  const float scale = 1.0f / sqrtf(static_cast<float>(N + 1));
  for (int j = threadIdx.x; j < D; j += blockDim.x) {
    float acc = 0.f;
    for (int k = 0; k <= N; ++k) acc += bf16bits_to_f32(src[k][j]);
    d.xs[static_cast<size_t>(row) * D + j] = acc * scale;
  }
}

cudaError_t launch_fusion(const DevPtrs& d, int nrows, const uint16_t* tok_emb,
                          const uint16_t* fusion, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  fusion_kernel<<<nrows, 256, 0, st>>>(d, tok_emb, fusion);
  return cudaGetLastError();
}

}  // namespace dualar
