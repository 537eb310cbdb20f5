// Weight-streaming GEMV device code, shared by the standalone GEMV kernel and
// the persistent frame kernel.
//
//   y[b][n] = sum_k W[n][k] x'[b][k],   x' = RMSNorm(x) * g   (optional)
//
// Each CTA owns a contiguous range of output rows (balanced to +-1 row) and
// walks it in groups of kRowsPerGroup rows, one row per consumer warp.  K is
// cut into chunks; a ring stage holds one (group, chunk) tile -- up to 16
// row-chunks per matrix (two matrices for the SwiGLU gate/up pair), each
// fetched by one bulk copy (cp.async.bulk) into shared memory.  A warp
// accumulates its row over the chunks and reduces with shuffles only, so
// consumer warps never synchronise with each other while streaming.  One
// producer thread runs ahead by the ring depth; in the persistent kernel it
// keeps streaming the next GEMV's weights while the consumers are still busy
// with other work, since weights never depend on activations.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace dualar {

constexpr int kRowsPerGroup = kGemvConsumerWarps;   // one row per consumer warp
constexpr int kStageBytes = 40960;                  // one ring stage
constexpr int kMaxVecPerLane = 5;                   // 16-byte weight vectors per lane per row-chunk

// Chunk length (elements) of one row-chunk: a tile of kRowsPerGroup rows x
// nmat matrices x kc elements fits one stage, and kc/8 vectors spread over
// 32 lanes give at most kMaxVecPerLane vectors per lane.
__host__ __device__ inline int gemv_kc(int K, int nmat, int* n_chunks) {
  const int kmax = kStageBytes / (kRowsPerGroup * nmat * 2);   // 1280 or 640
  const int n = (K + kmax - 1) / kmax;
  if (n_chunks) *n_chunks = n;
  return ((K + n - 1) / n + 7) & ~7;
}

struct GemvGeo {
  int v_begin, v_end;   // rows of this CTA
  int n_groups, n_chunks, kc, nmat, n_tiles;
};

DEVI GemvGeo gemv_geo(const GemvArgs& a, int cta, int ncta) {
  GemvGeo g;
  const bool swiglu = a.mode == GEMV_SWIGLU;
  g.nmat = swiglu ? 2 : 1;
  const int nv = swiglu ? a.n0 : a.n0 + a.n1;
  g.v_begin = static_cast<int>((static_cast<long long>(cta) * nv) / ncta);
  g.v_end = static_cast<int>((static_cast<long long>(cta + 1) * nv) / ncta);
  g.n_groups = (g.v_end - g.v_begin + kRowsPerGroup - 1) / kRowsPerGroup;
  g.kc = gemv_kc(a.K, g.nmat, &g.n_chunks);
  g.n_tiles = g.n_groups * g.n_chunks;
  return g;
}

struct GemvRing {
  uint64_t* full;
  uint64_t* empty;
  unsigned char* base;
  int stages;
};

// Producer side: issues the tiles of one GEMV for this CTA.  t is the ring's
// running tile counter (shared convention with the consumers).  Returns false
// if a wait gave up or the error word is set (then nothing more is issued).
DEVI bool gemv_produce(const GemvArgs& a, const GemvGeo& g, const GemvRing& ring, uint32_t& t,
                       uint64_t pol, const volatile uint32_t* abort_word) {
  const size_t slot_bytes = static_cast<size_t>(g.kc) * 2;
  for (int i = 0; i < g.n_tiles; ++i, ++t) {
    const int s = static_cast<int>(t % ring.stages);
    if (t >= static_cast<uint32_t>(ring.stages)) {
      const uint32_t parity = ((t / ring.stages) - 1) & 1;
      if (!mbar_try_wait(&ring.empty[s], parity)) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&ring.empty[s], parity)) {
          if ((abort_word && *abort_word) || global_timer_ns() - t0 > a.wait_limit_ns) {
            raise_error(a.err, DEV_ERR_MBAR_TIMEOUT);
            return false;
          }
        }
      }
    }
    const int grp = i / g.n_chunks, c = i % g.n_chunks;
    const int v0 = g.v_begin + grp * kRowsPerGroup;
    const int rows = min(kRowsPerGroup, g.v_end - v0);
    const int k0 = c * g.kc;
    const int len = min(g.kc, a.K - k0);
    const uint32_t bytes = static_cast<uint32_t>(len) * 2;
    mbar_arrive_expect_tx(&ring.full[s], bytes * rows * g.nmat);
    unsigned char* st = ring.base + static_cast<size_t>(s) * kStageBytes;
    for (int m = 0; m < g.nmat; ++m) {
      for (int w = 0; w < rows; ++w) {
        const int v = v0 + w;
        const uint16_t* rowp;
        if (g.nmat == 2) rowp = (m ? a.w1 : a.w0) + static_cast<size_t>(v) * a.K;
        else rowp = v < a.n0 ? a.w0 + static_cast<size_t>(v) * a.K
                             : a.w1 + static_cast<size_t>(v - a.n0) * a.K;
        bulk_load_g2s(st + (m * kRowsPerGroup + w) * slot_bytes, rowp + k0, bytes, &ring.full[s], pol);
      }
    }
  }
  return true;
}

// Waits (bounded) for every copy this producer may still have in flight, so
// the CTA never exits with bulk copies writing into its shared memory.
DEVI void gemv_drain(const GemvRing& ring, uint32_t t, uint64_t limit_ns) {
  const uint32_t n = t < static_cast<uint32_t>(ring.stages) ? t : ring.stages;
  for (uint32_t j = 1; j <= n; ++j) {
    const uint32_t tt = t - j;
    const int s = static_cast<int>(tt % ring.stages);
    const uint32_t parity = (tt / ring.stages) & 1;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(&ring.full[s], parity))
      if (global_timer_ns() - t0 > limit_ns) break;
  }
}

// Consumer prologue: x rows into shared memory in a split layout (xa holds
// elements 8j..8j+3, xb elements 8j+4..8j+7, so a warp's 16-byte reads are
// conflict-free), RMSNorm applied if requested.  Uses named barrier 1 over the
// consumer threads.  `red` needs 16 * NB floats, `scale` NB floats.
template <int NB>
DEVI void gemv_stage_x(const GemvArgs& a, float* xs, float* red, float* scale, int cta,
                       bool coherent) {
  constexpr int NCT = kGemvConsumerWarps * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, KV = K >> 3;
  float ss[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) ss[b] = 0.f;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if (b < a.nb) {
      const float4* src = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(b) * a.ldx);
      float4* xa = reinterpret_cast<float4*>(xs + static_cast<size_t>(b) * K);
      float4* xb = xa + KV;
      for (int j = tid; j < KV; j += NCT) {
        const float4 v0 = coherent ? __ldcg(src + 2 * j) : src[2 * j];
        const float4 v1 = coherent ? __ldcg(src + 2 * j + 1) : src[2 * j + 1];
        xa[j] = v0;
        xb[j] = v1;
        ss[b] += v0.x * v0.x + v0.y * v0.y + v0.z * v0.z + v0.w * v0.w + v1.x * v1.x + v1.y * v1.y +
                 v1.z * v1.z + v1.w * v1.w;
      }
    }
  }
  if (a.norm_w != nullptr) {
    // [P1] "Fast Transformer": RMSNorm(dim, eps=norm_eps), pre-norm blocks.
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float w = warp_sum(ss[b]);
      if (lane == 0) red[warp * NB + b] = w;
    }
    named_barrier(1, NCT);
    if (tid < NB) {
      float t = 0.f;
      for (int w = 0; w < kGemvConsumerWarps; ++w) t += red[w * NB + tid];
      scale[tid] = 1.0f / sqrtf(t / static_cast<float>(K) + a.eps);
    }
    named_barrier(1, NCT);
    for (int b = 0; b < a.nb; ++b) {
      const float sc = scale[b];
      float* xa = xs + static_cast<size_t>(b) * K;
      float* xb = xa + 4 * KV;
      for (int k = tid; k < K; k += NCT) {
        const int j = k >> 3, e = k & 7;
        float* p = e < 4 ? xa + 4 * j + e : xb + 4 * j + (e - 4);
        *p = (*p * sc) * bf16bits_to_f32(a.norm_w[k]);
      }
    }
  }
  named_barrier(1, NCT);
  if (a.save_x != nullptr && cta == 0) {
    for (int b = 0; b < a.nb; ++b) {
      const int row = a.save_map ? a.save_map[b] : b;
      if (row < 0) continue;
      const float* xa = xs + static_cast<size_t>(b) * K;
      const float* xb = xa + 4 * KV;
      for (int k = tid; k < K; k += NCT) {
        const int j = k >> 3, e = k & 7;
        a.save_x[static_cast<size_t>(row) * a.lds + k] = e < 4 ? xa[4 * j + e] : xb[4 * j + e - 4];
      }
    }
  }
}

// Consumer side: consumes the tiles of one GEMV, writes the epilogue.
// Returns false if a wait gave up.
template <int NB>
DEVI bool gemv_consume(const GemvArgs& a, const GemvGeo& g, const GemvRing& ring, uint32_t& t,
                       const float* xs) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K, KV = K >> 3;
  const size_t slot_bytes = static_cast<size_t>(g.kc) * 2;
  float acc[2][NB];
  for (int i = 0; i < g.n_tiles; ++i, ++t) {
    const int s = static_cast<int>(t % ring.stages);
    const int grp = i / g.n_chunks, c = i % g.n_chunks;
    const int v0 = g.v_begin + grp * kRowsPerGroup;
    const int rows = min(kRowsPerGroup, g.v_end - v0);
    if (c == 0) {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[m][b] = 0.f;
    }
    if (!mbar_wait(&ring.full[s], (t / ring.stages) & 1, a.err, a.wait_limit_ns)) return false;
    if (warp < rows) {
      const int j0 = (c * g.kc) >> 3;                 // first vector of this chunk
      const int nvec = min(g.kc, K - c * g.kc) >> 3;
      const unsigned char* st = ring.base + static_cast<size_t>(s) * kStageBytes;
      for (int m = 0; m < g.nmat; ++m) {
        const uint4* wr = reinterpret_cast<const uint4*>(st + (m * kRowsPerGroup + warp) * slot_bytes);
        uint4 w[kMaxVecPerLane];
#pragma unroll
        for (int q = 0; q < kMaxVecPerLane; ++q) {
          const int j = lane + 32 * q;
          if (j < nvec) w[q] = wr[j];
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const float4* xa = reinterpret_cast<const float4*>(xs + static_cast<size_t>(b) * K);
          const float4* xb = xa + KV;
          float p = 0.f;
#pragma unroll
          for (int q = 0; q < kMaxVecPerLane; ++q) {
            const int j = lane + 32 * q;
            if (j < nvec) p = dot8(w[q], xa[j0 + j], xb[j0 + j], p);
          }
          acc[m][b] += p;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ring.empty[s]);
    if (c == g.n_chunks - 1 && warp < rows) {
      const int n = v0 + warp;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        acc[0][b] = warp_sum(acc[0][b]);
        if (g.nmat == 2) acc[1][b] = warp_sum(acc[1][b]);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (lane == b && b < a.nb) {
          const int orow = a.out_map ? a.out_map[b] : b;
          if (orow >= 0) {
            float* o = a.out + static_cast<size_t>(orow) * a.ldo + n;
            if (a.mode == GEMV_STORE) *o = acc[0][b];
            else if (a.mode == GEMV_ADD) *o = __ldcg(a.base + static_cast<size_t>(orow) * a.ldb + n) + acc[0][b];
            // [P2] "The slow AR is Qwen3-4B": SwiGLU FFN, down(SiLU(gate) * up).
            else *o = silu(acc[0][b]) * acc[1][b];
          }
        }
      }
    }
  }
  return true;
}

}  // namespace dualar
