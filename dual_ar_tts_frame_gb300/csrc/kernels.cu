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
#include "gemv.cuh"
#include "internal.h"
#include "ops.cuh"

namespace dualar {

// ============================================================================
// setup: rows, page tables, prompt embeddings
// ============================================================================
__global__ void setup_kernel(const LaunchSetup s, DevPtrs d, const uint16_t* tok_emb) {
  pdl_wait();
  pdl_launch();
  const int r = blockIdx.x;
  if (r < s.n_rows && threadIdx.x == 0) {
    const RowInfo ri = s.rows[r];
    d.rows[r] = ri;
    const bool commit = ri.active && (!s.commit_last_only || r == s.n_rows - 1);
    d.commit_map[r] = commit ? ri.slot : -1;
  }
  if (r == 0) {
    for (int i = threadIdx.x; i < d.n_layer; i += blockDim.x) d.sched[i] = 0;
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
  return launch_pdl(setup_kernel, dim3(s.n_rows > 0 ? s.n_rows : 1), dim3(256), 0, st, s, d, tok_emb);
}

// ============================================================================
// Synthetic context (benchmark / test hook)
// ============================================================================
// Fills the KV pages of a slot (all layers), its held hidden state and its
// held logits with seeded values in [-1, 1) (hidden) and [-3, 3) (logits),
// from a counter hash of (seed, element).  Not part of the decode path.
DEVI uint32_t synth_hash(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7FEB352Du;
  x ^= x >> 15;
  x *= 0x846CA68Bu;
  x ^= x >> 16;
  return x;
}
DEVI float synth_unit(uint32_t seed, uint64_t i) {
  const uint32_t h = synth_hash(synth_hash(static_cast<uint32_t>(i) ^ seed) + static_cast<uint32_t>(i >> 32));
  return static_cast<float>(h >> 8) * (2.0f / 16777216.0f) - 1.0f;
}
// grid: (x, n_pages); each thread writes 8 bf16 values per step
__global__ void synthetic_fill_kernel(DevPtrs d, int slot, uint32_t seed) {
  const size_t page_elems = static_cast<size_t>(d.n_layer) * 2 * d.Hkv * d.page_tokens * d.hd;
  const int p = blockIdx.y;
  const int pg = d.page_table[static_cast<size_t>(slot) * d.pages_per_seq + p];
  if (pg < 0 || pg >= d.max_pages) {
    if (threadIdx.x == 0) raise_error(d.err, DEV_ERR_BAD_PAGE);
    return;
  }
  const size_t base = static_cast<size_t>(pg) * page_elems;
  uint4* dst = reinterpret_cast<uint4*>(d.kv_pool + base);
  const size_t nv = page_elems / 8;
  for (size_t v = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; v < nv;
       v += static_cast<size_t>(gridDim.x) * blockDim.x) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint64_t e = base + 8 * v + 2 * q;
      w[q] = static_cast<uint32_t>(f32_to_bf16bits(synth_unit(seed, e))) |
             (static_cast<uint32_t>(f32_to_bf16bits(synth_unit(seed, e + 1))) << 16);
    }
    dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    for (int k = threadIdx.x; k < d.D; k += blockDim.x)
      d.h_last[static_cast<size_t>(slot) * d.D + k] = synth_unit(seed ^ 0x9E3779B9u, k);
    for (int k = threadIdx.x; k < d.n_sem + 1; k += blockDim.x)
      d.z_last[static_cast<size_t>(slot) * (d.n_sem + 1) + k] = 3.0f * synth_unit(seed ^ 0x85EBCA6Bu, k);
  }
}

cudaError_t launch_synthetic_fill(const DevPtrs& d, int slot, int n_pages, uint32_t seed, int n_sm,
                                  cudaStream_t st) {
  (void)n_sm;
  if (n_pages <= 0) return cudaSuccess;
  synthetic_fill_kernel<<<dim3(64, n_pages), 256, 0, st>>>(d, slot, seed);
  return cudaGetLastError();
}

// ============================================================================
// GEMV (standalone launch; device code in gemv.cuh)
// ============================================================================
constexpr int kMaxStages = kMaxStagesRing;
constexpr int kSmemBudget = 225 * 1024;   // dynamic shared memory per CTA

// Shared-memory layout of gemv_kernel (offsets in bytes): mbarriers, the
// consumers' scratch, x rows, then the ring.
__host__ __device__ inline size_t gemv_scratch_off() { return 256; }
__host__ __device__ inline size_t gemv_scratch_bytes(int nbt) {
  switch (nbt) {
    case 8: return sizeof(GemvScratch<8>);
    case 4: return sizeof(GemvScratch<4>);
    case 2: return sizeof(GemvScratch<2>);
    default: return sizeof(GemvScratch<1>);
  }
}
__host__ __device__ inline size_t gemv_pro_off(int nbt) {
  return (gemv_scratch_off() + gemv_scratch_bytes(nbt) + 15) & ~size_t(15);
}
__host__ __device__ inline size_t gemv_xs_off(int nbt) {
  return (gemv_pro_off(nbt) + sizeof(GemvPro<8>) + 127) & ~size_t(127);
}
// W4: the x rows are followed by the 32-element sums of x' ([nbt][K/32]).
__host__ __device__ inline size_t gemv_ring_off(int nbt, int K, bool w4 = false) {
  const size_t xf = size_t(nbt) * K + (w4 ? size_t(nbt) * (K / 32) : 0);
  return (gemv_xs_off(nbt) + sizeof(float) * xf + 127) & ~size_t(127);
}

template <int NB, bool W4>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_kernel(const GemvArgs a, const int stages) {
  extern __shared__ __align__(128) unsigned char smem[];
  GemvRing ring;
  ring.full = reinterpret_cast<uint64_t*>(smem);
  ring.empty = ring.full + kMaxStagesRing;
  ring.base = smem + gemv_ring_off(NB, a.K, W4);
  ring.stages = stages;
  GemvScratch<NB>& scr = *reinterpret_cast<GemvScratch<NB>*>(smem + gemv_scratch_off());
  GemvPro<NB>& pro = *reinterpret_cast<GemvPro<NB>*>(smem + gemv_pro_off(NB));
  float* xs = reinterpret_cast<float*>(smem + gemv_xs_off(NB));
  float* gsum = xs + static_cast<size_t>(NB) * a.K;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&ring.full[s], 1);
      mbar_init(&ring.empty[s], kGemvConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  const GemvGeo g = gemv_geo<W4>(a, blockIdx.x, gridDim.x);
  uint32_t t = 0;
  if (warp == kGemvConsumerWarps) {
    // the weights are constant: this CTA's rows are requested into L2 and
    // streamed into the ring while the previous kernel may still run (the
    // consumers wait for it before reading x)
    if (lane == 0) {
      gemv_prefetch_rows<W4>(a, g);
      gemv_produce<W4>(a, g, ring, t, policy_evict_first(), nullptr);
      gemv_drain(ring, t, a.wait_limit_ns);
    }
    pdl_wait();
    return;
  }
  pdl_wait();
  pdl_launch();
  if constexpr (W4) {
    gemv_stage_x<NB, true>(a, g, xs, pro, blockIdx.x, false, 0, gsum);
    gemv_consume_w4<NB>(a, g, ring, t, xs, gsum, scr, pro);
  } else {
    gemv_stage_x<NB>(a, g, xs, pro, blockIdx.x, false);
    gemv_consume<NB>(a, g, ring, t, xs, scr, pro);
  }
}

struct GemvPlan {
  int stages;
  int nbt;
  size_t smem;
};

static GemvPlan plan_gemv(int K, int nb, bool w4) {
  GemvPlan p;
  int nbt = nb >= 8 ? 8 : nb >= 4 ? 4 : nb >= 2 ? 2 : 1;
  while (true) {
    const size_t ring = gemv_ring_off(nbt, K, w4);
    const long long room = static_cast<long long>(kSmemBudget) - static_cast<long long>(ring);
    const int st = room > 0 ? static_cast<int>(room / kStageBytes) : 0;
    if (st >= 2 || nbt == 1) {
      p.nbt = nbt;
      p.stages = st > kMaxStages ? kMaxStages : st;
      p.smem = ring + static_cast<size_t>(p.stages) * kStageBytes;
      return p;
    }
    nbt >>= 1;
  }
}

template <int NB, bool W4>
static cudaError_t launch_gemv_nb(const GemvArgs& a, const GemvPlan& p, int grid, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NB, W4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBudget);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_pdl(gemv_kernel<NB, W4>, dim3(grid), dim3(kGemvThreads), p.smem, st, a, p.stages);
}

template <bool W4>
static cudaError_t launch_gemv_fmt(const GemvArgs& s, const GemvPlan& p, int grid, cudaStream_t st) {
  switch (p.nbt) {
    case 8: return launch_gemv_nb<8, W4>(s, p, grid, st);
    case 4: return launch_gemv_nb<4, W4>(s, p, grid, st);
    case 2: return launch_gemv_nb<2, W4>(s, p, grid, st);
    default: return launch_gemv_nb<1, W4>(s, p, grid, st);
  }
}

cudaError_t launch_gemv(const GemvArgs& a, int n_sm, cudaStream_t st) {
  if (a.nb <= 0) return cudaSuccess;
  const bool w4 = a.w4 != 0;
  if (w4) {
    // packed 4-bit rows: plain fp32 buffers, no saved x (gemv_stage_x<NB, true>)
    if (!w4_k_supported(a.K) || a.x_src >= 0 || a.base_src >= 0 || a.out_src >= 0 || a.save_x != nullptr)
      return cudaErrorInvalidValue;
  } else if (a.K % 8 != 0 || !gemv_k_supported(a.K)) {
    return cudaErrorInvalidValue;
  }
  const GemvPlan p = plan_gemv(a.K, a.nb, w4);
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
    const cudaError_t e = w4 ? launch_gemv_fmt<true>(s, p, grid, st) : launch_gemv_fmt<false>(s, p, grid, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ============================================================================
// 4-bit weight packing (w4a16; record layout in gemv.cuh, "4-bit weights")
// ============================================================================
// One warp per (row, group of 128 elements); lane l quantizes elements
// 4l .. 4l+3 of the group.  Symmetric absolute-maximum rule: m = max |w| over
// the group, scale s = bf16(m / 7) (fp32 division, round to nearest even),
// q = clamp(rint(w / s), -8, 7) (q = 0 when s = 0), stored as q + 8.
__global__ void quantize_w4_kernel(const uint16_t* w, int n, int K, unsigned char* out) {
  const int gpr = K / kW4Group;
  const long long wid = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= static_cast<long long>(n) * gpr) return;   // whole warps leave together
  const int row = static_cast<int>(wid / gpr), grp = static_cast<int>(wid % gpr);
  const uint2 raw =
      *reinterpret_cast<const uint2*>(w + static_cast<size_t>(row) * K + static_cast<size_t>(grp) * kW4Group + 4 * lane);
  const float v[4] = {bf16lo(raw.x), bf16hi(raw.x), bf16lo(raw.y), bf16hi(raw.y)};
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const uint16_t sbits = f32_to_bf16bits(m / 7.0f);
  const float sc = bf16bits_to_f32(sbits);
  uint32_t u[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float qf = sc > 0.f ? rintf(v[e] / sc) : 0.f;
    qf = fminf(fmaxf(qf, -8.f), 7.f);
    u[e] = static_cast<uint32_t>(static_cast<int>(qf) + 8);
  }
  const size_t rb = static_cast<size_t>(w4_row_bytes(K));
  unsigned char* rec = out + static_cast<size_t>(row) * rb;
  const uint16_t packed = static_cast<uint16_t>(u[0] | (u[1] << 4) | (u[2] << 8) | (u[3] << 12));
  *reinterpret_cast<uint16_t*>(rec + grp * (kW4Group / 2) + 2 * lane) = packed;
  if (lane == 0) *reinterpret_cast<uint16_t*>(rec + K / 2 + 2 * grp) = sbits;
  if (grp == 0) {
    const int pad0 = K / 2 + 2 * gpr;
    for (int i = pad0 + lane; i < static_cast<int>(rb); i += 32) rec[i] = 0;
  }
}

cudaError_t launch_quantize_w4(const uint16_t* w, int n, int K, unsigned char* out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (K <= 0 || K % kW4Group) return cudaErrorInvalidValue;
  const long long warps = static_cast<long long>(n) * (K / kW4Group);
  const long long blocks = (warps + 7) / 8;
  if (blocks > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  quantize_w4_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(w, n, K, out);
  return cudaGetLastError();
}

// Packed 4-bit rows back to bf16, for the tensor-core path: one thread per
// 32-element vector (16 code bytes, all in one scale group).  A weight q * s
// (exact in fp32: at most 4 + 8 significant bits) is written as two bf16
// values, hi = bf16(q s) and lo = bf16(q s - hi), which add up to it
// exactly: row r of out holds hi in columns [0, K) and lo in [K, 2K), so a
// product over the 2K columns with x repeated gives W x exactly.  Launched
// without programmatic dependent launch, so that it starts after everything
// before it (a projection may still read the previous contents) and the next
// kernel sees its writes.
__global__ void dequant_w4_kernel(const unsigned char* packed, int n, int K, uint16_t* out) {
  const int vpr = K / 32;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(n) * vpr) return;
  const int row = static_cast<int>(idx / vpr), v = static_cast<int>(idx % vpr);
  const unsigned char* rec = packed + static_cast<size_t>(row) * w4_row_bytes(K);
  const uint4 c = *reinterpret_cast<const uint4*>(rec + static_cast<size_t>(v) * 16);
  const float sc = bf16bits_to_f32(*reinterpret_cast<const uint16_t*>(rec + K / 2 + (v >> 2) * 2));
  const uint32_t wd[4] = {c.x, c.y, c.z, c.w};
  uint16_t* rowp = out + static_cast<size_t>(row) * 2 * K + static_cast<size_t>(v) * 32;
  uint4* dhi = reinterpret_cast<uint4*>(rowp);
  uint4* dlo = reinterpret_cast<uint4*>(rowp + K);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t oh[4], ol[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t byte = (wd[q] >> (8 * e)) & 0xFFu;   // elements 2e (low nibble) and 2e+1
      uint32_t h2 = 0, l2 = 0;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float w = static_cast<float>(static_cast<int>((byte >> (4 * half)) & 0xFu) - 8) * sc;
        const uint16_t hb = f32_to_bf16bits(w);
        const uint16_t lb = f32_to_bf16bits(w - bf16bits_to_f32(hb));
        h2 |= static_cast<uint32_t>(hb) << (16 * half);
        l2 |= static_cast<uint32_t>(lb) << (16 * half);
      }
      oh[e] = h2;
      ol[e] = l2;
    }
    dhi[q] = make_uint4(oh[0], oh[1], oh[2], oh[3]);
    dlo[q] = make_uint4(ol[0], ol[1], ol[2], ol[3]);
  }
}

cudaError_t launch_dequant_w4(const void* packed, int n, int K, uint16_t* out, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (K <= 0 || K % kW4Group) return cudaErrorInvalidValue;
  const long long threads = static_cast<long long>(n) * (K / 32);
  dequant_w4_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(
      static_cast<const unsigned char*>(packed), n, K, out);
  return cudaGetLastError();
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
  pdl_wait();
  pdl_launch();
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
  cudaError_t e;
  if (d.hd == 128)
    e = launch_pdl(append_kernel<4>, dim3(nrows), dim3(256), 0, st, d, layer, fast ? 1 : 0, fast_pos, q_norm, k_norm);
  else if (d.hd == 64)
    e = launch_pdl(append_kernel<2>, dim3(nrows), dim3(256), 0, st, d, layer, fast ? 1 : 0, fast_pos, q_norm, k_norm);
  else
    return cudaErrorInvalidValue;
  return e;
}

// ============================================================================
// Standalone launches of the ops in ops.cuh
// ============================================================================
constexpr int kAttnThreads = 512;   // same split as the persistent kernel (bit-identical paths)
constexpr int kAttnBufs = 2;        // pages in flight per CTA (measured: a third does not help)

template <int HD, int G>
__global__ void __launch_bounds__(kAttnThreads, 2)
    attn_paged_kernel(DevPtrs d, int nrows, int layer, int total_units, int chunk_tokens,
                      int fuse_append, const uint16_t* q_norm, const uint16_t* k_norm) {
  pdl_wait();
  pdl_launch();
  extern __shared__ __align__(128) unsigned char attn_smem_raw[];
  auto& sm = *reinterpret_cast<AttnSmem<HD, G, kAttnThreads, kAttnBufs>*>(attn_smem_raw);
  __shared__ uint64_t bars[kAttnBufs];
  if (threadIdx.x == 0) {
    for (int b = 0; b < kAttnBufs; ++b) mbar_init(&bars[b], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  uint32_t phase[kAttnBufs];
  for (int b = 0; b < kAttnBufs; ++b) phase[b] = 0u;
  attn_paged_units<HD, G, kAttnThreads, kAttnBufs>(d, nrows, layer, total_units, chunk_tokens, fuse_append != 0,
                                                   q_norm, k_norm, sm, bars, phase, blockIdx.x, gridDim.x);
}

template <int HD, int G>
static cudaError_t attn_paged_launch(const DevPtrs& d, int nrows, int layer, int units, int chunk,
                                     int grid, int fuse, const uint16_t* qn, const uint16_t* kn,
                                     cudaStream_t st) {
  static bool configured = false;
  const int smem = static_cast<int>(sizeof(AttnSmem<HD, G, kAttnThreads, kAttnBufs>));
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_paged_kernel<HD, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_pdl(attn_paged_kernel<HD, G>, dim3(grid), dim3(kAttnThreads), smem, st, d, nrows, layer, units,
                    chunk, fuse, qn, kn);
}

template <int HD>
static cudaError_t attn_paged_hd(const DevPtrs& d, int nrows, int layer, int units, int chunk,
                                 int grid, int fuse, const uint16_t* qn, const uint16_t* kn,
                                 cudaStream_t st) {
  switch (d.Hq / d.Hkv) {
    case 1: return attn_paged_launch<HD, 1>(d, nrows, layer, units, chunk, grid, fuse, qn, kn, st);
    case 2: return attn_paged_launch<HD, 2>(d, nrows, layer, units, chunk, grid, fuse, qn, kn, st);
    case 4: return attn_paged_launch<HD, 4>(d, nrows, layer, units, chunk, grid, fuse, qn, kn, st);
    case 8: return attn_paged_launch<HD, 8>(d, nrows, layer, units, chunk, grid, fuse, qn, kn, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_paged(const DevPtrs& d, int nrows, int layer, int total_units,
                              int chunk_tokens, int n_sm, bool fuse_append, const uint16_t* q_norm,
                              const uint16_t* k_norm, cudaStream_t st, bool* mma_used, AttnHalves hv) {
  if (mma_used) *mma_used = false;
  if (nrows <= 0 || total_units <= 0) return cudaSuccess;
  if (d.page_tokens != kPageTokens || chunk_tokens % kPageTokens != 0) return cudaErrorInvalidValue;
  if (!fuse_append) {
    // prefill: blocks of consecutive rows read each page once
    bool used = false;
    const cudaError_t e = launch_attn_prefill(d, nrows, layer, total_units, chunk_tokens, n_sm, st, &used);
    if (e != cudaSuccess || used) return e;
  }
  {
    // 3+ rows: the tensor-core variant; 1-2 rows keep this kernel, the same
    // device code as the persistent frame kernel (bit-identical paths)
    bool used = false;
    const cudaError_t e = launch_attn_mma(d, nrows, layer, total_units, chunk_tokens, n_sm, fuse_append, q_norm,
                                          k_norm, st, &used, hv);
    if (mma_used) *mma_used = used;
    if (e != cudaSuccess || used) return e;
  }
  const int grid = total_units < 4 * n_sm ? total_units : 4 * n_sm;
  const int f = fuse_append ? 1 : 0;
  if (d.hd == 128) return attn_paged_hd<128>(d, nrows, layer, total_units, chunk_tokens, grid, f, q_norm, k_norm, st);
  if (d.hd == 64) return attn_paged_hd<64>(d, nrows, layer, total_units, chunk_tokens, grid, f, q_norm, k_norm, st);
  return cudaErrorInvalidValue;
}

template <int EPL, int G>
__global__ void attn_fast_kernel(DevPtrs d, int layer, int pos, const uint16_t* q_norm,
                                 const uint16_t* k_norm, AttnHalves hv) {
  pdl_wait();
  pdl_launch();
  constexpr int NT = 32 * (G + 1 > 2 ? G + 1 : 2);
  __shared__ FastAttnSmem<EPL * 32> sm;
  attn_fast_unit<EPL, G, NT, true>(d, blockIdx.x, layer, pos, q_norm, k_norm, sm, OpTags{0u, 0u}, hv);
}

template <int EPL>
static cudaError_t attn_fast_epl(const DevPtrs& d, int nrows, int layer, int pos, const uint16_t* qn,
                                 const uint16_t* kn, cudaStream_t st, AttnHalves hv) {
  const int G = d.Hq / d.Hkv;
  const int grid = nrows * d.Hkv;
  switch (G) {
    case 1: return launch_pdl(attn_fast_kernel<EPL, 1>, dim3(grid), dim3(64), 0, st, d, layer, pos, qn, kn, hv);
    case 2: return launch_pdl(attn_fast_kernel<EPL, 2>, dim3(grid), dim3(96), 0, st, d, layer, pos, qn, kn, hv);
    case 4: return launch_pdl(attn_fast_kernel<EPL, 4>, dim3(grid), dim3(160), 0, st, d, layer, pos, qn, kn, hv);
    case 8: return launch_pdl(attn_fast_kernel<EPL, 8>, dim3(grid), dim3(288), 0, st, d, layer, pos, qn, kn, hv);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_fast(const DevPtrs& d, int nrows, int layer, int pos, const uint16_t* q_norm,
                             const uint16_t* k_norm, cudaStream_t st, AttnHalves hv) {
  if (nrows <= 0) return cudaSuccess;
  if (pos < 0 || pos >= d.N || pos >= d.rope_len) return cudaErrorInvalidValue;
  if (d.hd == 128) return attn_fast_epl<4>(d, nrows, layer, pos, q_norm, k_norm, st, hv);
  if (d.hd == 64) return attn_fast_epl<2>(d, nrows, layer, pos, q_norm, k_norm, st, hv);
  return cudaErrorInvalidValue;
}

__global__ void __launch_bounds__(kSampThreads) sample_q0_kernel(DevPtrs d, SampIO io) {
  pdl_wait();
  pdl_launch();
  __shared__ SampSmem<kSampThreads> sm;
  sample_q0_row<kSampThreads>(d, blockIdx.x, io, sm);
}

__global__ void __launch_bounds__(kSampThreads) sample_fast_kernel(DevPtrs d, int k, SampIO io) {
  pdl_wait();
  pdl_launch();
  __shared__ SampSmem<kSampThreads> sm;
  sample_fast_row<kSampThreads>(d, blockIdx.x, k, io, sm);
}

static SampIO make_io(const float* uniforms, int ldu, const SamplingParams& sp, const int32_t* forced,
                      int ldf, int32_t* codes_out, int32_t* status_out, float* slow_logits_out,
                      float* fast_logits_out, int32_t* draws_out, const uint16_t* fast_emb) {
  SampIO io;
  io.uniforms = uniforms;
  io.ldu = ldu;
  io.sp = sp;
  io.forced = forced;
  io.ldf = ldf;
  io.codes_out = codes_out;
  io.status_out = status_out;
  io.slow_logits_out = slow_logits_out;
  io.fast_logits_out = fast_logits_out;
  io.draws_out = draws_out;
  io.fast_emb = fast_emb;
  return io;
}

cudaError_t launch_sample_q0(const DevPtrs& d, int nrows, const float* uniforms, int ldu,
                             const SamplingParams& sp, const int32_t* forced, int ldf,
                             int32_t* codes_out, int32_t* status_out, float* slow_logits_out,
                             int32_t* draws_out, const uint16_t* fast_emb, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  return launch_pdl(sample_q0_kernel, dim3(nrows), dim3(kSampThreads), 0, st, d,
                    make_io(uniforms, ldu, sp, forced, ldf, codes_out, status_out, slow_logits_out, nullptr,
                            draws_out, fast_emb));
}

cudaError_t launch_sample_fast(const DevPtrs& d, int nrows, int k, const float* uniforms, int ldu,
                               const SamplingParams& sp, const int32_t* forced, int ldf,
                               int32_t* codes_out, float* fast_logits_out, int32_t* draws_out,
                               const uint16_t* fast_emb, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  return launch_pdl(sample_fast_kernel, dim3(nrows), dim3(kSampThreads), 0, st, d, k,
                    make_io(uniforms, ldu, sp, forced, ldf, codes_out, nullptr, nullptr, fast_logits_out,
                            draws_out, fast_emb));
}

__global__ void fusion_kernel(DevPtrs d, const uint16_t* tok_emb, const uint16_t* fusion) {
  pdl_wait();
  pdl_launch();
  fusion_row<256>(d, blockIdx.x, tok_emb, fusion);
}

cudaError_t launch_fusion(const DevPtrs& d, int nrows, const uint16_t* tok_emb,
                          const uint16_t* fusion, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  return launch_pdl(fusion_kernel, dim3(nrows), dim3(256), 0, st, d, tok_emb, fusion);
}

}  // namespace dualar
