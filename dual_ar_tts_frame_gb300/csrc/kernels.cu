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
// GEMV (standalone launch; device code in gemv.cuh)
// ============================================================================
constexpr int kMaxStages = kMaxStagesRing;
constexpr int kSmemBudget = 225 * 1024;   // dynamic shared memory per CTA

// Shared-memory layout of gemv_kernel (offsets in bytes): mbarriers, the
// consumers' scratch, x rows, then the ring.
__host__ __device__ inline size_t gemv_scratch_off() { return 256; }
__host__ __device__ inline size_t gemv_xs_off() {
  return (256 + sizeof(GemvScratch<8>) + sizeof(GemvPro<8>) + 127) & ~size_t(127);
}
__host__ __device__ inline size_t gemv_ring_off(int nbt, int K) {
  return (gemv_xs_off() + sizeof(float) * size_t(nbt) * K + 127) & ~size_t(127);
}

template <int NB>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_kernel(const GemvArgs a, const int stages) {
  extern __shared__ __align__(128) unsigned char smem[];
  GemvRing ring;
  ring.full = reinterpret_cast<uint64_t*>(smem);
  ring.empty = ring.full + kMaxStagesRing;
  ring.base = smem + gemv_ring_off(NB, a.K);
  ring.stages = stages;
  GemvScratch<NB>& scr = *reinterpret_cast<GemvScratch<NB>*>(smem + gemv_scratch_off());
  GemvPro<NB>& pro = *reinterpret_cast<GemvPro<NB>*>(smem + gemv_scratch_off() + sizeof(GemvScratch<8>));
  float* xs = reinterpret_cast<float*>(smem + gemv_xs_off());
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&ring.full[s], 1);
      mbar_init(&ring.empty[s], kGemvConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  for (int i = tid; i < kMaxStagesRing * kWarpsC; i += blockDim.x) (&scr.cnt[0][0])[i] = 0;
  __syncthreads();
  const GemvGeo g = gemv_geo(a, blockIdx.x, gridDim.x);
  uint32_t t = 0;
  if (warp == kGemvConsumerWarps) {
    if (lane == 0) {
      gemv_produce(a, g, ring, t, policy_evict_first(), nullptr);
      gemv_drain(ring, t, a.wait_limit_ns);
    }
    return;
  }
  gemv_stage_x<NB>(a, g, xs, pro, blockIdx.x, false);
  gemv_consume<NB>(a, g, ring, t, xs, scr, pro);
}

struct GemvPlan {
  int stages;
  int nbt;
  size_t smem;
};

static GemvPlan plan_gemv(int K, int nb) {
  GemvPlan p;
  int nbt = nb >= 8 ? 8 : nb >= 4 ? 4 : nb >= 2 ? 2 : 1;
  while (true) {
    const size_t ring = gemv_ring_off(nbt, K);
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

template <int NB>
static cudaError_t launch_gemv_nb(const GemvArgs& a, const GemvPlan& p, int grid, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBudget);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  gemv_kernel<NB><<<grid, kGemvThreads, p.smem, st>>>(a, p.stages);
  return cudaGetLastError();
}

cudaError_t launch_gemv(const GemvArgs& a, int n_sm, cudaStream_t st) {
  if (a.nb <= 0) return cudaSuccess;
  if (a.K % 8 != 0 || !gemv_k_supported(a.K)) return cudaErrorInvalidValue;
  const GemvPlan p = plan_gemv(a.K, a.nb);
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

// QK-norm (optional) + RoPE of one head vector held as EPL elements per lane.
template <int EPL>
DEVI void head_norm_rope(float (&v)[EPL], const uint16_t* nw, float eps, int pos, const DevPtrs& d,
                         int lane) {
  const int hd = EPL * 32, half = hd / 2;
  if (nw != nullptr) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < EPL; ++j) s += v[j] * v[j];
    s = warp_sum(s);
    const float inv = 1.0f / sqrtf(s / static_cast<float>(hd) + eps);
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
}

// ============================================================================
// Paged split-KV decode attention
// ============================================================================
// A unit is (row, KV head g, chunk c of chunk_tokens positions).  The unit
// computes softmax(q K^T / sqrt(hd)) V for the G query heads of g over its
// chunk with a running max; K and V pages (64 positions x hd, bf16) are
// staged in shared memory by double-buffered bulk copies.  The last unit of
// (row, g) to finish merges the chunks in chunk order (deterministic).
// With fuse_append (decode: one row per sequence) the unit applies QK-norm
// and RoPE to its query heads itself, and the unit holding the newest
// position also computes that position's K and V, writes them to the page
// and uses them directly.  [P2] fact table: 32 query heads over 8 KV heads.
constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kPageTokens = 64;

template <int HD, int G>
struct AttnSmem {
  uint16_t kv[2][2][kPageTokens * HD];   // [buffer][K/V][tok][dim]
  float qs[G][4][HD / 4 + 1];
  float sc[G][kPageTokens];
  float ored[kAttnThreads / HD][G][HD];
  float knew[HD], vnew[HD];
  float scl[G], msm[G], lsm[G];
  uint64_t bar[2];
  int s_last;
};

template <int HD, int G>
__global__ void __launch_bounds__(kAttnThreads)
    attn_paged_kernel(DevPtrs d, int nrows, int layer, int total_units, int chunk_tokens,
                      int fuse_append, const uint16_t* q_norm, const uint16_t* k_norm) {
  constexpr int EPL = HD / 32;
  constexpr int QD = HD / 4;                // dims per thread in the score pass
  constexpr int PARTS = kAttnThreads / HD;  // token groups in the value pass
  constexpr int TPP = kPageTokens / PARTS;  // tokens per group
  constexpr uint32_t kPageBytes = kPageTokens * HD * 2;
  extern __shared__ __align__(128) unsigned char attn_smem_raw[];
  AttnSmem<HD, G>& sm = *reinterpret_cast<AttnSmem<HD, G>*>(attn_smem_raw);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hq = d.Hq, hkv = d.Hkv;
  const float qscale = 1.0f / sqrtf(static_cast<float>(HD));
  const size_t page_stride = static_cast<size_t>(kPageTokens) * HD;
  if (tid == 0) {
    mbar_init(&sm.bar[0], 1);
    mbar_init(&sm.bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  uint32_t phase[2] = {0u, 0u};

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
    const int npages = (t1 - t0 + kPageTokens - 1) / kPageTokens;
    const bool newest = fuse_append && (c == nch - 1);

    // page table lookups (all threads agree); a bad entry skips the unit
    auto page_of = [&](int p) -> int {
      return d.page_table[ri.slot * d.pages_per_seq + (t0 / kPageTokens) + p];
    };
    bool ok = true;
    for (int p = 0; p < npages; ++p) {
      const int pg = page_of(p);
      if (pg < 0 || pg >= d.max_pages) ok = false;
    }
    if (!ok) {
      if (tid == 0) raise_error(d.err, DEV_ERR_BAD_PAGE);
      continue;
    }
    auto issue = [&](int p, int buf) {
      const uint16_t* kp = d.kv_pool +
          (((static_cast<size_t>(page_of(p)) * d.n_layer + layer) * 2 + 0) * hkv + g) * page_stride;
      const uint16_t* vp = kp + static_cast<size_t>(hkv) * page_stride;
      mbar_arrive_expect_tx(&sm.bar[buf], 2 * kPageBytes);
      bulk_load_g2s_plain(sm.kv[buf][0], kp, kPageBytes, &sm.bar[buf]);
      bulk_load_g2s_plain(sm.kv[buf][1], vp, kPageBytes, &sm.bar[buf]);
    };
    if (tid == 0) {
      issue(0, 0);
      if (npages > 1) issue(1, 1);
    }

    // query heads of g (norm + RoPE in place when fused)
    if (fuse_append) {
      if (warp < G) {
        const int h = g * G + warp;
        const float* src = d.qkv + static_cast<size_t>(r) * d.qkv_dim + h * HD;
        float v[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) v[j] = src[lane * EPL + j];
        head_norm_rope<EPL>(v, q_norm, d.eps, ri.pos, d, lane);
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
          const int dd = lane * EPL + j;
          sm.qs[warp][dd / QD][dd % QD] = v[j] * qscale;
        }
      }
      if (warp == (G % kAttnWarps) && newest) {
        const float* base = d.qkv + static_cast<size_t>(r) * d.qkv_dim;
        float kv[EPL], vv[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
          kv[j] = base[hq * HD + g * HD + lane * EPL + j];
          vv[j] = base[hq * HD + hkv * HD + g * HD + lane * EPL + j];
        }
        head_norm_rope<EPL>(kv, k_norm, d.eps, ri.pos, d, lane);
        const int pidx = ri.pos / kPageTokens;
        const int pg = d.page_table[ri.slot * d.pages_per_seq + pidx];
        uint16_t* kd = d.kv_pool + (((static_cast<size_t>(pg) * d.n_layer + layer) * 2 + 0) * hkv + g) *
                                       page_stride + static_cast<size_t>(ri.pos % kPageTokens) * HD;
        uint16_t* vd = kd + static_cast<size_t>(hkv) * page_stride;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
          const uint16_t kb = f32_to_bf16bits(kv[j]), vb = f32_to_bf16bits(vv[j]);
          kd[lane * EPL + j] = kb;
          vd[lane * EPL + j] = vb;
          sm.knew[lane * EPL + j] = bf16bits_to_f32(kb);
          sm.vnew[lane * EPL + j] = bf16bits_to_f32(vb);
        }
      }
    } else {
      for (int e = tid; e < G * HD; e += kAttnThreads) {
        const int h = e / HD, dd = e % HD;
        sm.qs[h][dd / QD][dd % QD] = d.qrot[(static_cast<size_t>(r) * hq + g * G + h) * HD + dd] * qscale;
      }
    }
    if (tid < G) {
      sm.msm[tid] = -INFINITY;
      sm.lsm[tid] = 0.f;
    }
    float o[G];
#pragma unroll
    for (int h = 0; h < G; ++h) o[h] = 0.f;
    __syncthreads();

    const int tok = tid >> 2, qd = tid & 3;
    const int vdim = tid % HD, vpart = tid / HD;
    for (int p = 0; p < npages; ++p) {
      const int buf = p & 1;
      const int ps = t0 + p * kPageTokens;
      const int ntok = min(kPageTokens, t1 - ps);
      if (!mbar_wait(&sm.bar[buf], phase[buf], d.err, d.wait_limit_ns)) return;
      phase[buf] ^= 1u;
      const uint16_t* ks = sm.kv[buf][0];
      const uint16_t* vs = sm.kv[buf][1];
      // scores
      float s[G];
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = 0.f;
      if (tok < ntok) {
        const bool isnew = newest && (ps + tok == ri.pos);
        if (isnew) {
#pragma unroll 4
          for (int j = 0; j < QD; ++j) {
            const float kf = sm.knew[qd * QD + j];
#pragma unroll
            for (int h = 0; h < G; ++h) s[h] = fmaf(sm.qs[h][qd][j], kf, s[h]);
          }
        } else {
          const uint4* k4 = reinterpret_cast<const uint4*>(ks + tok * HD + qd * QD);
#pragma unroll
          for (int v8 = 0; v8 < QD / 8; ++v8) {
            const uint4 w = k4[v8];
            const float kf[8] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y),
                                 bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w)};
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) s[h] = fmaf(sm.qs[h][qd][v8 * 8 + jj], kf[jj], s[h]);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        s[h] += __shfl_xor_sync(0xFFFFFFFFu, s[h], 1);
        s[h] += __shfl_xor_sync(0xFFFFFFFFu, s[h], 2);
      }
      if (qd == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) sm.sc[h][tok] = tok < ntok ? s[h] : -INFINITY;
      }
      __syncthreads();
      if (warp < G) {
        const int h = warp;
        const float a0 = sm.sc[h][lane], a1 = sm.sc[h][lane + 32];
        const float mx = warp_max(fmaxf(a0, a1));
        const float mold = sm.msm[h];
        const float mnew = fmaxf(mold, mx);
        const float p0 = lane < ntok ? expf(a0 - mnew) : 0.f;
        const float p1 = lane + 32 < ntok ? expf(a1 - mnew) : 0.f;
        sm.sc[h][lane] = p0;
        sm.sc[h][lane + 32] = p1;
        const float sum = warp_sum(p0 + p1);
        if (lane == 0) {
          const float f = expf(mold - mnew);   // 0 for the first page (mold = -inf)
          sm.scl[h] = f;
          sm.lsm[h] = sm.lsm[h] * f + sum;
          sm.msm[h] = mnew;
        }
      }
      __syncthreads();
#pragma unroll
      for (int h = 0; h < G; ++h) o[h] *= sm.scl[h];
      const int tb = vpart * TPP, te = min(ntok, tb + TPP);
      for (int t = tb; t < te; ++t) {
        const bool isnew = newest && (ps + t == ri.pos);
        const float v = isnew ? sm.vnew[vdim] : bf16bits_to_f32(vs[t * HD + vdim]);
#pragma unroll
        for (int h = 0; h < G; ++h) o[h] = fmaf(sm.sc[h][t], v, o[h]);
      }
      __syncthreads();   // buffer `buf` is free again
      if (tid == 0 && p + 2 < npages) issue(p + 2, buf);
    }
    // merge the token groups
#pragma unroll
    for (int h = 0; h < G; ++h) sm.ored[vpart][h][vdim] = o[h];
    __syncthreads();
    if (nch == 1) {
      for (int e = tid; e < G * HD; e += kAttnThreads) {
        const int h = e / HD, dd = e % HD;
        float t = 0.f;
#pragma unroll
        for (int p = 0; p < PARTS; ++p) t += sm.ored[p][h][dd];
        d.attn[static_cast<size_t>(r) * hq * HD + (g * G + h) * HD + dd] = t / sm.lsm[h];
      }
      __syncthreads();
      continue;
    }
    float* pw = d.part + ((static_cast<size_t>(r) * hkv + g) * kMaxChunks + c) * G * (HD + 2);
    for (int e = tid; e < G * HD; e += kAttnThreads) {
      const int h = e / HD, dd = e % HD;
      float t = 0.f;
#pragma unroll
      for (int p = 0; p < PARTS; ++p) t += sm.ored[p][h][dd];
      pw[h * (HD + 2) + dd] = t;
    }
    if (tid < G) {
      pw[tid * (HD + 2) + HD] = sm.msm[tid];
      pw[tid * (HD + 2) + HD + 1] = sm.lsm[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const uint32_t old = atomic_add_acq_rel_gpu(&d.arrive[r * hkv + g], 1u);
      sm.s_last = (old == static_cast<uint32_t>(nch - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (sm.s_last) {
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

template <int HD, int G>
static cudaError_t attn_paged_launch(const DevPtrs& d, int nrows, int layer, int units, int chunk,
                                     int grid, int fuse, const uint16_t* qn, const uint16_t* kn,
                                     cudaStream_t st) {
  static bool configured = false;
  const int smem = static_cast<int>(sizeof(AttnSmem<HD, G>));
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_paged_kernel<HD, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  attn_paged_kernel<HD, G><<<grid, kAttnThreads, smem, st>>>(d, nrows, layer, units, chunk, fuse, qn, kn);
  return cudaGetLastError();
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
                              const uint16_t* k_norm, cudaStream_t st) {
  if (nrows <= 0 || total_units <= 0) return cudaSuccess;
  if (d.page_tokens != kPageTokens || chunk_tokens % kPageTokens != 0) return cudaErrorInvalidValue;
  const int grid = total_units < 4 * n_sm ? total_units : 4 * n_sm;
  const int f = fuse_append ? 1 : 0;
  if (d.hd == 128) return attn_paged_hd<128>(d, nrows, layer, total_units, chunk_tokens, grid, f, q_norm, k_norm, st);
  if (d.hd == 64) return attn_paged_hd<64>(d, nrows, layer, total_units, chunk_tokens, grid, f, q_norm, k_norm, st);
  return cudaErrorInvalidValue;
}

// ============================================================================
// Fast-AR attention over the per-frame codebook cache (<= N positions)
// ============================================================================
// One CTA per (row, KV head g): warp 0 computes the new position's K (norm if
// configured, RoPE at the codebook index) and V and appends them; the K/V of
// earlier positions (written by earlier passes of this frame) are staged in
// shared memory; warp h < G then computes query head g*G+h.  [P2] "Two
// autoregressions": the fast AR's KV cache is num_codebooks long and is
// overwritten every frame.
template <int EPL, int G>
__global__ void attn_fast_kernel(DevPtrs d, int layer, int pos, const uint16_t* q_norm,
                                 const uint16_t* k_norm) {
  constexpr int HD = EPL * 32;
  __shared__ float ks[kMaxCodebooks][HD], vs[kMaxCodebooks][HD];
  const int r = blockIdx.x / d.Hkv, g = blockIdx.x % d.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = d.Hq, hkv = d.Hkv, N = d.N;
  const float* qkv = d.qkv + static_cast<size_t>(r) * d.qkv_dim;
  float* kb = d.fast_kv + (((static_cast<size_t>(r) * d.fast_n_layer + layer) * 2 + 0) * hkv + g) * N * HD;
  float* vb = kb + static_cast<size_t>(hkv) * N * HD;
  if (warp == 0) {
    float kv[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) kv[j] = qkv[hq * HD + g * HD + lane * EPL + j];
    head_norm_rope<EPL>(kv, k_norm, d.eps, pos, d, lane);
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      const float vv = qkv[hq * HD + hkv * HD + g * HD + lane * EPL + j];
      kb[static_cast<size_t>(pos) * HD + lane * EPL + j] = kv[j];
      vb[static_cast<size_t>(pos) * HD + lane * EPL + j] = vv;
      ks[pos][lane * EPL + j] = kv[j];
      vs[pos][lane * EPL + j] = vv;
    }
  } else {
    for (int e = threadIdx.x - 32; e < pos * HD; e += blockDim.x - 32) {
      ks[e / HD][e % HD] = kb[e];
      vs[e / HD][e % HD] = vb[e];
    }
  }
  __syncthreads();
  if (warp >= G) return;
  const int h = g * G + warp;
  float q[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) q[j] = qkv[h * HD + lane * EPL + j];
  head_norm_rope<EPL>(q, q_norm, d.eps, pos, d, lane);
  const float scale = 1.0f / sqrtf(static_cast<float>(HD));
  float s[kMaxCodebooks];
  float m = -INFINITY;
#pragma unroll
  for (int t = 0; t < kMaxCodebooks; ++t) {
    s[t] = -INFINITY;
    if (t <= pos) {
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < EPL; ++j) a = fmaf(q[j], ks[t][lane * EPL + j], a);
      s[t] = warp_sum(a) * scale;
      m = fmaxf(m, s[t]);
    }
  }
  float l = 0.f;
  float o[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) o[j] = 0.f;
#pragma unroll
  for (int t = 0; t < kMaxCodebooks; ++t) {
    if (t <= pos) {
      const float p = expf(s[t] - m);
      l += p;
#pragma unroll
      for (int j = 0; j < EPL; ++j) o[j] = fmaf(p, vs[t][lane * EPL + j], o[j]);
    }
  }
  float* dst = d.attn + static_cast<size_t>(r) * hq * HD + h * HD;
#pragma unroll
  for (int j = 0; j < EPL; ++j) dst[lane * EPL + j] = o[j] / l;
}

template <int EPL>
static cudaError_t attn_fast_epl(const DevPtrs& d, int nrows, int layer, int pos, const uint16_t* qn,
                                 const uint16_t* kn, cudaStream_t st) {
  const int G = d.Hq / d.Hkv;
  const int threads = 32 * (G > 1 ? G : 2);
  const int grid = nrows * d.Hkv;
  switch (G) {
    case 1: attn_fast_kernel<EPL, 1><<<grid, threads, 0, st>>>(d, layer, pos, qn, kn); break;
    case 2: attn_fast_kernel<EPL, 2><<<grid, threads, 0, st>>>(d, layer, pos, qn, kn); break;
    case 4: attn_fast_kernel<EPL, 4><<<grid, threads, 0, st>>>(d, layer, pos, qn, kn); break;
    case 8: attn_fast_kernel<EPL, 8><<<grid, threads, 0, st>>>(d, layer, pos, qn, kn); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_fast(const DevPtrs& d, int nrows, int layer, int pos, const uint16_t* q_norm,
                             const uint16_t* k_norm, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  if (pos < 0 || pos >= d.N || pos >= d.rope_len) return cudaErrorInvalidValue;
  if (d.hd == 128) return attn_fast_epl<4>(d, nrows, layer, pos, q_norm, k_norm, st);
  if (d.hd == 64) return attn_fast_epl<2>(d, nrows, layer, pos, q_norm, k_norm, st);
  return cudaErrorInvalidValue;
}

// ============================================================================
// Sampler: temperature + top-p on caller uniforms, one CTA per row
// ============================================================================
// Candidates are ordered by (logit descending, token id ascending): each gets
// a unique 64-bit key (order-preserving bits of the logit, then the inverted
// id).  Probability mass is integer fixed point, round(exp((z - zmax) / T) *
// 2^24), so every sum is exact and independent of thread order.  The top-p
// cut is the first candidate (in key order) whose inclusive cumulative mass
// reaches ceil(top_p * Z); the draw is the first kept candidate whose
// inclusive cumulative mass reaches floor(u * Zk) + 1, i.e. exceeds u * Zk.
// Both are found by a most-significant-byte-first radix descent over the
// keys with 256-bin mass histograms; lanes of a warp that hit the same bin
// are combined (match + reduce) before one shared-memory atomic.  [P2] "Two
// autoregressions": sample(biased_logits, ...) for q0, unmasked
// sample(logits, ...) for q1..q9.
constexpr int kMaxCands = 4097;

template <int NT>
struct SampSmem {
  static constexpr int NW = NT / 32;
  unsigned long long hmass[256];
  unsigned int hcnt[256];
  unsigned long long red64[NW];
  float redf[NW];
  unsigned long long bc[4];
  int ibc[4];
};

struct Cands {
  int n;          // candidates
  int n_main;     // candidates 0..n_main-1 have ids id_base + i
  int id_base;
  int extra_id;   // id of candidate n_main when n > n_main
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

template <int NT>
DEVI float samp_block_max(float v, SampSmem<NT>& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  if (lane == 0) sm.redf[warp] = v;
  __syncthreads();
  float t = sm.redf[0];
  for (int w = 1; w < SampSmem<NT>::NW; ++w) t = fmaxf(t, sm.redf[w]);
  __syncthreads();
  return t;
}

template <int NT>
DEVI unsigned long long samp_block_sum(unsigned long long v, SampSmem<NT>& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (lane == 0) sm.red64[warp] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < SampSmem<NT>::NW; ++w) t += sm.red64[w];
  __syncthreads();
  return t;
}

template <int NT>
DEVI unsigned long long samp_block_max_u64(unsigned long long v, SampSmem<NT>& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w > v ? w : v;
  }
  if (lane == 0) sm.red64[warp] = v;
  __syncthreads();
  unsigned long long t = 0;
  for (int w = 0; w < SampSmem<NT>::NW; ++w) t = sm.red64[w] > t ? sm.red64[w] : t;
  __syncthreads();
  return t;
}

// First key (descending) whose inclusive cumulative mass reaches target
// (1 <= target <= total).  *above_out: mass strictly before it; *mass_out:
// its own mass.
template <int NT, int EPT>
DEVI unsigned long long samp_select(const unsigned long long (&key)[EPT], const uint32_t (&mass)[EPT],
                                    int n, unsigned long long target, SampSmem<NT>& sm,
                                    unsigned long long* above_out, unsigned long long* mass_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long prefix = 0, above = 0, result = 0;
  for (int shift = 56;; shift -= 8) {
    for (int b = tid; b < 256; b += NT) {
      sm.hmass[b] = 0;
      sm.hcnt[b] = 0;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int i = tid + e * NT;
      const bool valid = i < n && (shift == 56 || (key[e] >> (shift + 8)) == prefix);
      const uint32_t bin = valid ? static_cast<uint32_t>((key[e] >> shift) & 255ull) : 256u;
      const uint32_t grp = __match_any_sync(0xFFFFFFFFu, bin);
      const uint32_t sum = __reduce_add_sync(grp, valid ? mass[e] : 0u);
      if (valid && (__ffs(grp) - 1) == lane) {
        atomicAdd(&sm.hmass[bin], static_cast<unsigned long long>(sum));
        atomicAdd(&sm.hcnt[bin], static_cast<unsigned int>(__popc(grp)));
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l (descending)
      unsigned long long m8[8];
      unsigned long long tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        m8[j] = sm.hmass[255 - 8 * lane - j];
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
        unsigned long long cc = excl;
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
        sm.ibc[0] = bin;
        sm.ibc[1] = static_cast<int>(sm.hcnt[bin]);
        sm.bc[0] = above + cc;
        sm.bc[1] = sm.hmass[bin];
      }
    }
    __syncthreads();
    const int bin = sm.ibc[0];
    const int cnt = sm.ibc[1];
    above = sm.bc[0];
    const unsigned long long mbin = sm.bc[1];
    prefix = (shift == 56) ? static_cast<unsigned long long>(bin)
                           : ((prefix << 8) | static_cast<unsigned long long>(bin));
    if (shift == 0) {
      result = prefix;
      *mass_out = mbin;
      break;
    }
    if (cnt == 1) {
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        const int i = tid + e * NT;
        if (i < n && (key[e] >> shift) == prefix) sm.bc[2] = key[e];
      }
      __syncthreads();
      result = sm.bc[2];
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
template <int NT, int EPT>
DEVI int samp_draw(const float (&z)[EPT], const unsigned long long (&key)[EPT], const Cands& c,
                   float zmax, float temperature, float top_p, float u, SampSmem<NT>& sm) {
  const int tid = threadIdx.x;
  if (!(temperature > 0.f)) {
    unsigned long long best = 0;
#pragma unroll
    for (int e = 0; e < EPT; ++e)
      if (tid + e * NT < c.n && key[e] > best) best = key[e];
    return key_to_index(c, samp_block_max_u64(best, sm));
  }
  const float inv_t = 1.0f / temperature;
  uint32_t mass[EPT];
  unsigned long long local = 0;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    mass[e] = 0;
    if (tid + e * NT < c.n) {
      mass[e] = __float2uint_rn(expf((z[e] - zmax) * inv_t) * 16777216.0f);   // * 2^24
      local += mass[e];
    }
  }
  const unsigned long long Z = samp_block_sum(local, sm);
  unsigned long long tc = Z;
  if (top_p < 1.0f) {
    const double t = ceil(static_cast<double>(top_p) * static_cast<double>(Z));
    tc = t < 1.0 ? 1ull : static_cast<unsigned long long>(t);
    if (tc > Z) tc = Z;
  }
  unsigned long long above, mk;
  samp_select<NT, EPT>(key, mass, c.n, tc, sm, &above, &mk);
  const unsigned long long zk = above + mk;
  unsigned long long td =
      static_cast<unsigned long long>(floor(static_cast<double>(u) * static_cast<double>(zk))) + 1ull;
  if (td > zk) td = zk;
  const unsigned long long kd = samp_select<NT, EPT>(key, mass, c.n, td, sm, &above, &mk);
  return key_to_index(c, kd);
}

// Loads the candidates' logits and keys into registers; returns zmax.
template <int NT, int EPT>
DEVI float samp_load(const float* src, const Cands& c, float (&z)[EPT], unsigned long long (&key)[EPT],
                     SampSmem<NT>& sm) {
  float zm = -INFINITY;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int i = threadIdx.x + e * NT;
    z[e] = -INFINITY;
    key[e] = 0;
    if (i < c.n) {
      z[e] = src[i];
      zm = fmaxf(zm, z[e]);
      key[e] = (static_cast<unsigned long long>(ord_f32(z[e])) << 32) |
               static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(cand_id(c, i)));
    }
  }
  return samp_block_max(zm, sm);
}

constexpr int kSampEPT = (kMaxCands + kSampThreads - 1) / kSampThreads;

__global__ void __launch_bounds__(kSampThreads)
    sample_q0_kernel(DevPtrs d, const float* uniforms, int ldu, SamplingParams sp,
                     const int32_t* forced, int ldf, int32_t* codes_out, int32_t* status_out,
                     float* slow_logits_out, int32_t* draws_out, const uint16_t* fast_emb) {
  __shared__ SampSmem<kSampThreads> sm;
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
  const Cands c{ns + (sp.allow_eos ? 1 : 0), ns, d.sem_begin, d.im_end};
  float z[kSampEPT];
  unsigned long long key[kSampEPT];
  const float zmax = samp_load<kSampThreads, kSampEPT>(zsrc, c, z, key, sm);
  const float* u = uniforms + static_cast<size_t>(row) * ldu;
  const int normal = samp_draw<kSampThreads, kSampEPT>(z, key, c, zmax, sp.temperature, sp.top_p, u[0], sm);
  // [P2] "Two autoregressions": a second draw at temperature 1.0, top-p 0.9,
  // used when the normal draw repeats a semantic token of the last 10 frames.
  const int ras = samp_draw<kSampThreads, kSampEPT>(z, key, c, zmax, sp.ras_temperature, sp.ras_top_p,
                                                   u[1], sm);
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
  __shared__ SampSmem<kSampThreads> sm;
  __shared__ int s_commit;
  const int row = blockIdx.x, tid = threadIdx.x;
  const int N = d.N, Cf = d.Cf;
  const float* zs = d.logits + static_cast<size_t>(row) * d.logit_ld;
  if (fast_logits_out)
    for (int i = tid; i < Cf; i += kSampThreads)
      fast_logits_out[(static_cast<size_t>(row) * (N - 1) + (k - 1)) * Cf + i] = zs[i];
  if (!d.rows[row].active) return;
  const Cands c{Cf, Cf, 0, -1};
  float z[kSampEPT];
  unsigned long long key[kSampEPT];
  const float zmax = samp_load<kSampThreads, kSampEPT>(zs, c, z, key, sm);
  const float* u = uniforms + static_cast<size_t>(row) * ldu;
  const int draw = samp_draw<kSampThreads, kSampEPT>(z, key, c, zmax, sp.temperature, sp.top_p, u[k + 1], sm);
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
  sample_q0_kernel<<<nrows, kSampThreads, 0, st>>>(
      d, uniforms, ldu, sp, forced, ldf, codes_out, status_out, slow_logits_out, draws_out, fast_emb);
  return cudaGetLastError();
}

cudaError_t launch_sample_fast(const DevPtrs& d, int nrows, int k, const float* uniforms, int ldu,
                               const SamplingParams& sp, const int32_t* forced, int ldf,
                               int32_t* codes_out, float* fast_logits_out, int32_t* draws_out,
                               const uint16_t* fast_emb, cudaStream_t st) {
  if (nrows <= 0) return cudaSuccess;
  sample_fast_kernel<<<nrows, kSampThreads, 0, st>>>(
      d, k, uniforms, ldu, sp, forced, ldf, codes_out, fast_logits_out, draws_out, fast_emb);
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
