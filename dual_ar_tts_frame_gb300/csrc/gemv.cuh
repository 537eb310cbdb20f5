// Weight-streaming GEMV device code, shared by the standalone GEMV kernel and
// the persistent frame kernel.
//
//   y[b][n] = sum_k W[n][k] x'[b][k],   x' = RMSNorm(x) * g   (optional)
//
// Each CTA owns a contiguous range of output rows (balanced to +-1 row).  A
// ring stage holds one tile: R consecutive rows of one matrix, which are
// contiguous in memory, fetched by ONE bulk copy (cp.async.bulk) of up to
// 40 KB (R is a power of two with R*K*2 <= 40 KB).  The consumer warps split
// the tile: S = warps / R warps per row, each taking a contiguous segment of
// K, lane-strided 16-byte vectors.  A warp frees its ring stage as soon as its
// dot products have consumed the tile, then reduces its segment with shuffles
// and stores the partial in a per-tile buffer; no CTA-wide synchronisation
// while streaming.  When the buffer is full, and at the end of the GEMV, the
// consumers add each row's S partials in segment order (deterministic) and
// write the epilogue.  The SwiGLU gate and up rows are two consecutive
// tiles.  One producer thread runs ahead by the ring depth; in the persistent
// kernel it keeps streaming the next GEMV's weights while the consumers are
// still busy, since weights never depend on activations.
//
// Packed 4-bit rows ("4-bit weights" below) use the same ring, tiles and
// epilogue: a tile is R packed row records, a lane's 16-byte vector holds 32
// elements of one scale group (gemv_consume_w4).
#pragma once

#include "common.cuh"
#include "internal.h"

namespace dualar {

constexpr int kWarpsC = kGemvConsumerWarps;   // consumer warps (power of two)
constexpr int kStageBytes = 40960;            // one ring stage
constexpr int kMaxStagesRing = 8;
constexpr int kMaxVecPerLane = 5;             // 16-byte vectors per lane per tile (unrolled)

// Rows per tile for K (power of two, <= kWarpsC).
__host__ __device__ inline int gemv_rows_per_tile(int K) {
  int r = kWarpsC;
  while (r > 1 && r * K * 2 > kStageBytes) r >>= 1;
  return r;
}

// Whether a K fits the unrolled inner loop (vectors per lane per tile).
__host__ __device__ inline bool gemv_k_supported(int K) {
  const int R = gemv_rows_per_tile(K);
  if (R * K * 2 > kStageBytes) return false;
  const int S = kWarpsC / R;
  const int seg = (K / 8 + S - 1) / S;
  return (seg + 31) / 32 <= kMaxVecPerLane;
}

// ---- 4-bit weights (w4a16) ------------------------------------------------------
// A packed matrix [n][K] (K a multiple of 128) is one record per output row,
// records back to back:
//   bytes [0, K/2)          byte i holds the codes of elements 2i (low nibble)
//                           and 2i+1 (high nibble), each stored as u = q + 8
//                           (q in [-8, 7]);
//   bytes [K/2, K/2 + K/64) the bf16 scales of the K/128 groups of 128
//                           consecutive elements;
//   zero bytes up to a 16-byte multiple.
// Element k of the row is (u_k - 8) * scale[k / 128].  A tile is R whole
// records (one bulk copy); a lane reads 16-byte vectors of 32 elements, all
// in one group.
__host__ __device__ inline int w4_rows_per_tile(int K) {
  int r = kWarpsC;
  while (r > 1 && r * w4_row_bytes(K) > kStageBytes) r >>= 1;
  return r;
}

__host__ __device__ inline bool w4_k_supported(int K) {
  if (K <= 0 || K % kW4Group) return false;
  const int R = w4_rows_per_tile(K);
  if (R * w4_row_bytes(K) > kStageBytes) return false;
  const int S = kWarpsC / R;
  const int seg = (K / 32 + S - 1) / S;
  return (seg + 31) / 32 <= kMaxVecPerLane;
}

struct GemvGeo {
  int v_begin, v_end;   // rows of this CTA (virtual row space)
  int R, S, seg;        // rows per tile, warps per row, vectors per segment
  bool swiglu;
};

// seg: 16-byte vectors per warp segment (8 bf16 elements, or 32 packed
// 4-bit elements with W4).
template <bool W4 = false>
DEVI GemvGeo gemv_geo(const GemvArgs& a, int cta, int ncta) {
  GemvGeo g;
  g.swiglu = a.mode == GEMV_SWIGLU;
  const int nv = g.swiglu ? a.n0 : a.n0 + a.n1;
  g.v_begin = static_cast<int>((static_cast<long long>(cta) * nv) / ncta);
  g.v_end = static_cast<int>((static_cast<long long>(cta + 1) * nv) / ncta);
  g.R = W4 ? w4_rows_per_tile(a.K) : gemv_rows_per_tile(a.K);
  g.S = kWarpsC / g.R;
  g.seg = ((W4 ? a.K / 32 : a.K / 8) + g.S - 1) / g.S;
  return g;
}

// Tile sequence of one CTA: R-row tiles that never cross a segment boundary
// (restricted head: semantic block, then the <|im_end|> row); a SwiGLU tile
// is two loads (gate rows, then up rows).
struct TileIter {
  int v, v_end, n0, n1, R;
  bool swiglu;
  int sub;
  __device__ TileIter(const GemvArgs& a, const GemvGeo& g)
      : v(g.v_begin), v_end(g.v_end), n0(a.n0), n1(a.n1), R(g.R), swiglu(g.swiglu), sub(0) {}
  // row0, rows: rows of the tile; part: 0 gate / 1 up (SwiGLU)
  __device__ bool next(int& row0, int& rows, int& part) {
    if (v >= v_end) return false;
    if (swiglu) {
      rows = min(R, v_end - v);
      row0 = v;
      part = sub;
      if (sub == 1) v += rows;
      sub ^= 1;
      return true;
    }
    const int seg_end = v < n0 ? n0 : n0 + n1;
    rows = min(R, min(v_end, seg_end) - v);
    row0 = v;
    part = 0;
    v += rows;
    return true;
  }
};

DEVI const uint16_t* gemv_tile_src(const GemvArgs& a, int row0, int part) {
  if (a.mode == GEMV_SWIGLU) return (part ? a.w1 : a.w0) + static_cast<size_t>(row0) * a.K;
  return row0 < a.n0 ? a.w0 + static_cast<size_t>(row0) * a.K
                     : a.w1 + static_cast<size_t>(row0 - a.n0) * a.K;
}

// Bytes of one weight row, and where a tile starts (bf16 or packed 4-bit).
template <bool W4>
DEVI uint32_t gemv_row_bytes(int K) {
  return W4 ? static_cast<uint32_t>(w4_row_bytes(K)) : static_cast<uint32_t>(K) * 2u;
}
template <bool W4>
DEVI const void* gemv_tile_ptr(const GemvArgs& a, int row0, int part) {
  if (!W4) return gemv_tile_src(a, row0, part);
  const size_t rb = static_cast<size_t>(w4_row_bytes(a.K));
  const unsigned char* w0 = reinterpret_cast<const unsigned char*>(a.w0);
  const unsigned char* w1 = reinterpret_cast<const unsigned char*>(a.w1);
  if (a.mode == GEMV_SWIGLU) return (part ? w1 : w0) + static_cast<size_t>(row0) * rb;
  return row0 < a.n0 ? w0 + static_cast<size_t>(row0) * rb : w1 + static_cast<size_t>(row0 - a.n0) * rb;
}

struct GemvRing {
  uint64_t* full;
  uint64_t* empty;
  unsigned char* base;
  int stages;
};

// Shared scratch of the consumers: the per-warp partials of the last
// kPartTiles tiles and where each of those tiles starts.  A SwiGLU pair (gate
// tile, up tile) always sits in one window since kPartTiles is even.
template <int NB>
struct GemvScratch {
  static constexpr int kPartTiles = NB <= 2 ? 32 : 16;
  float part[kPartTiles][kWarpsC][NB];
  int2 tile[kPartTiles];   // first row, rows
};

// Producer side: issues the tiles of one GEMV for this CTA.  t is the ring's
// running tile counter (same convention as the consumers).  Returns false if
// a wait gave up or the abort word is set (then nothing more is issued).
template <bool W4 = false>
DEVI bool gemv_produce(const GemvArgs& a, const GemvGeo& g, const GemvRing& ring, uint32_t& t,
                       uint64_t pol, const volatile uint32_t* abort_word) {
  TileIter it(a, g);
  int row0, rows, part;
  while (it.next(row0, rows, part)) {
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
    const uint32_t bytes = static_cast<uint32_t>(rows) * gemv_row_bytes<W4>(a.K);
    mbar_arrive_expect_tx(&ring.full[s], bytes);
    bulk_load_g2s(ring.base + static_cast<size_t>(s) * kStageBytes, gemv_tile_ptr<W4>(a, row0, part), bytes,
                  &ring.full[s], pol);
    ++t;
  }
  return true;
}

// This CTA's weight rows (contiguous per segment) requested into L2, in 32 KB
// pieces (rows of 2 K bytes: 16-byte multiples).
template <bool W4 = false>
DEVI void gemv_prefetch_rows(const GemvArgs& a, const GemvGeo& g) {
  const size_t rb = gemv_row_bytes<W4>(a.K);
  auto range = [&](const uint16_t* base, int r0, int r1) {
    if (r1 <= r0) return;
    const unsigned char* p = reinterpret_cast<const unsigned char*>(base) + static_cast<size_t>(r0) * rb;
    const size_t bytes = static_cast<size_t>(r1 - r0) * rb;
    for (size_t o = 0; o < bytes; o += 32768) {
      const size_t n = bytes - o < 32768 ? bytes - o : 32768;
      bulk_prefetch_l2(p + o, static_cast<uint32_t>(n));
    }
  };
  if (g.swiglu) {
    range(a.w0, g.v_begin, g.v_end);
    range(a.w1, g.v_begin, g.v_end);
  } else {
    range(a.w0, g.v_begin, min(g.v_end, a.n0));
    range(a.w1, max(g.v_begin, a.n0) - a.n0, g.v_end - a.n0);
  }
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

// Consumer prologue.  Stages x' = x * g (g the RMSNorm gain, 1 without norm)
// in shared memory in a split layout (for each 8-element vector j, elements
// 0..3 at xa[j], 4..7 at xb[j], so a warp's 16-byte reads are
// conflict-free), and the RMSNorm scale s = 1/sqrt(mean(x^2) + eps) per row
// b, so that W (s x*g) = s (W x') is applied in the epilogue.  x and g are
// loaded in one pass (independent loads).  Also prefetches the residual base
// values of this CTA's rows and the output row map.  Uses named barrier 1
// over the consumer threads.  coherent: read x and base through L2 (data
// written by other CTAs of the same grid).
constexpr int kBaseRows = 64;   // residual rows prefetched per CTA

template <int NB>
struct GemvPro {
  float red[kWarpsC][NB];   // per-warp sums of x^2 (RMSNorm)
  int orow[NB];
  float base[kBaseRows][NB];
};

// RMSNorm scale of batch row b (1 without norm): 1/sqrt(mean(x^2) + eps).
template <int NB>
DEVI float gemv_scale(const GemvArgs& a, const GemvPro<NB>& pr, int b) {
  if (a.norm_w == nullptr) return 1.f;
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kWarpsC; ++w) t += pr.red[w][b];
  return 1.0f / sqrtf(t / static_cast<float>(a.K) + a.eps);
}

// W4: x' goes to a split-32 layout instead (float4 t, elements 4t..4t+3, of
// the 32-element vector v at float4 index t * (K/32) + v of the row), and
// gsum[b][v] receives the sum of vector v's 32 values of x'.
template <int NB, bool W4 = false>
DEVI void gemv_stage_x(const GemvArgs& a, const GemvGeo& g, float* xs, GemvPro<NB>& pr, int cta,
                       bool coherent, uint32_t epoch = 0, float* gsum = nullptr) {
  constexpr int NCT = kWarpsC * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, KV = K >> 3;
  const bool norm = a.norm_w != nullptr;
  // residual base of this CTA's rows (one value per thread at most): the load
  // is issued before the x loop and its result taken after it, so the two
  // round trips overlap
  const int nrows = g.v_end - g.v_begin;
  const bool pre_base = a.mode == GEMV_ADD && nrows <= kBaseRows;
  const int nbase = pre_base ? nrows * NB : 0;
  static_assert(kBaseRows * NB <= NCT, "one base value per thread");
  int my_rr = -1, my_b = 0;
  uint64_t wb = 0;
  float fb = 0.f;
  const uint64_t* pb = nullptr;
  if (tid < nbase) {
    my_rr = tid / NB;
    my_b = tid % NB;
    const int orow = my_b < a.nb ? (a.out_map ? __ldcg(a.out_map + my_b) : my_b) : -1;
    if (orow < 0) {
      my_rr = -1;
    } else {
      const size_t off = static_cast<size_t>(orow) * a.ldb + g.v_begin + my_rr;
      if (a.base_src >= 0) {
        pb = reinterpret_cast<const uint64_t*>(a.base) + off;
        wb = tag_load(pb);
      } else {
        fb = coherent ? __ldcg(a.base + off) : a.base[off];
      }
    }
  }
  float ss[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) ss[b] = 0.f;
  const uint32_t xtag = a.x_src >= 0 ? op_tag(epoch, a.x_src) : 0u;
  if (a.x_src >= 0 && a.x_scout > 0) {
    if (warp == 0) {
      const int nblk = K / a.x_scout;
      for (int b = 0; b < NB; ++b) {
        if (b >= a.nb) break;
        for (int blk = lane; blk < nblk; blk += 32)
          tag_wait1(reinterpret_cast<const uint64_t*>(a.x) + static_cast<size_t>(b) * a.ldx +
                        static_cast<size_t>(blk + 1) * a.x_scout - 1,
                    xtag, a.err, a.wait_limit_ns);
      }
    }
    named_barrier(1, NCT);
  }
  if constexpr (W4) {
    const int KV32 = K >> 5;
    for (int j0 = 0; j0 < KV; j0 += NCT) {   // uniform trip count: the quad shuffles below
      const int j = j0 + tid;
      const bool act = j < KV;
      float gw[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) gw[e] = 1.f;
      if (norm && act) {
        const uint4 gv = *reinterpret_cast<const uint4*>(a.norm_w + 8 * j);
        gw[0] = bf16lo(gv.x); gw[1] = bf16hi(gv.x); gw[2] = bf16lo(gv.y); gw[3] = bf16hi(gv.y);
        gw[4] = bf16lo(gv.z); gw[5] = bf16hi(gv.z); gw[6] = bf16lo(gv.w); gw[7] = bf16hi(gv.w);
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b >= a.nb) continue;   // uniform
        float part = 0.f;
        if (act) {
          float4 v0, v1;
          if (a.x_src >= 0) {
            float v[8];
            tag_wait<8>(reinterpret_cast<const uint64_t*>(a.x) + static_cast<size_t>(b) * a.ldx + 8 * j, xtag, v,
                        a.err, a.wait_limit_ns);
            v0 = make_float4(v[0], v[1], v[2], v[3]);
            v1 = make_float4(v[4], v[5], v[6], v[7]);
          } else {
            const float4* src = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(b) * a.ldx);
            v0 = coherent ? __ldcg(src + 2 * j) : src[2 * j];
            v1 = coherent ? __ldcg(src + 2 * j + 1) : src[2 * j + 1];
          }
          const float4 p0 = make_float4(v0.x * gw[0], v0.y * gw[1], v0.z * gw[2], v0.w * gw[3]);
          const float4 p1 = make_float4(v1.x * gw[4], v1.y * gw[5], v1.z * gw[6], v1.w * gw[7]);
          // 8-vector j is quarter (j & 3) of 32-vector j >> 2: float4s 2(j&3), 2(j&3)+1
          float4* x4 = reinterpret_cast<float4*>(xs + static_cast<size_t>(b) * K);
          const int t0 = 2 * (j & 3);
          x4[t0 * KV32 + (j >> 2)] = p0;
          x4[(t0 + 1) * KV32 + (j >> 2)] = p1;
          ss[b] += v0.x * v0.x + v0.y * v0.y + v0.z * v0.z + v0.w * v0.w + v1.x * v1.x + v1.y * v1.y +
                   v1.z * v1.z + v1.w * v1.w;
          part = ((p0.x + p0.y) + (p0.z + p0.w)) + ((p1.x + p1.y) + (p1.z + p1.w));
        }
        // the four 8-vectors of a 32-vector sit in lanes 4m .. 4m+3
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        if (act && (j & 3) == 0) gsum[b * KV32 + (j >> 2)] = part;
      }
    }
  } else {
    for (int j = tid; j < KV; j += NCT) {
      // the gain is loaded before x is polled: the two round trips overlap
      float gw[8];
      if (norm) {
        const uint4 gv = *reinterpret_cast<const uint4*>(a.norm_w + 8 * j);
        gw[0] = bf16lo(gv.x); gw[1] = bf16hi(gv.x); gw[2] = bf16lo(gv.y); gw[3] = bf16hi(gv.y);
        gw[4] = bf16lo(gv.z); gw[5] = bf16hi(gv.z); gw[6] = bf16lo(gv.w); gw[7] = bf16hi(gv.w);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) gw[e] = 1.f;
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (b < a.nb) {
          float v[8];
          if (a.x_src >= 0) {
            tag_wait<8>(reinterpret_cast<const uint64_t*>(a.x) + static_cast<size_t>(b) * a.ldx + 8 * j, xtag, v,
                        a.err, a.wait_limit_ns);
          } else {
            const float4* src = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(b) * a.ldx);
            const float4 v0 = coherent ? __ldcg(src + 2 * j) : src[2 * j];
            const float4 v1 = coherent ? __ldcg(src + 2 * j + 1) : src[2 * j + 1];
            v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
            v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
          }
          float4* xa = reinterpret_cast<float4*>(xs + static_cast<size_t>(b) * K);
          xa[j] = make_float4(v[0] * gw[0], v[1] * gw[1], v[2] * gw[2], v[3] * gw[3]);
          xa[KV + j] = make_float4(v[4] * gw[4], v[5] * gw[5], v[6] * gw[6], v[7] * gw[7]);
          ss[b] += v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3] + v[4] * v[4] + v[5] * v[5] +
                   v[6] * v[6] + v[7] * v[7];
        }
      }
    }
  }
  if (my_rr >= 0) {
    if (pb != nullptr) {
      const uint32_t btag = op_tag(epoch, a.base_src);
      fb = tag_of(wb) == btag ? tag_val(wb) : tag_wait1(pb, btag, a.err, a.wait_limit_ns);
    }
    pr.base[my_rr][my_b] = fb;
  }
  if (tid < NB) pr.orow[tid] = tid < a.nb ? (a.out_map ? __ldcg(a.out_map + tid) : tid) : -1;
  // RMSNorm partial sums per warp; the scale itself is finished where it is
  // used (epilogue), so the prologue needs a single barrier
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const float w = warp_sum(ss[b]);
    if (lane == 0) pr.red[warp][b] = w;
  }
  named_barrier(1, NCT);
  if (a.save_x != nullptr && cta == 0) {
    for (int b = 0; b < a.nb; ++b) {
      const int row = a.save_map ? __ldcg(a.save_map + b) : b;
      if (row < 0) continue;
      const float* xa = xs + static_cast<size_t>(b) * K;
      const float* xb = xa + 4 * KV;
      const float sc = gemv_scale(a, pr, b);
      for (int k = tid; k < K; k += NCT) {
        const int j = k >> 3, e = k & 7;
        a.save_x[static_cast<size_t>(row) * a.lds + k] = sc * (e < 4 ? xa[4 * j + e] : xb[4 * j + e - 4]);
      }
    }
  }
}

template <int NB>
DEVI void gemv_epilogue(const GemvArgs& a, const GemvGeo& g, const GemvPro<NB>& pr, int n, int b,
                        float y, float gate, uint32_t epoch) {
  if (b >= a.nb) return;
  const int orow = pr.orow[b];
  if (orow < 0) return;
  const size_t oi = static_cast<size_t>(orow) * a.ldo + n;
  const float sc = gemv_scale(a, pr, b);
  y *= sc;
  float r;
  if (a.mode == GEMV_STORE) {
    r = y;
  } else if (a.mode == GEMV_ADD) {
    const int rr = n - g.v_begin;
    float base;
    if (g.v_end - g.v_begin <= kBaseRows) {
      base = pr.base[rr][b];
    } else {
      const size_t bi = static_cast<size_t>(orow) * a.ldb + n;
      base = a.base_src >= 0
                 ? tag_wait1(reinterpret_cast<const uint64_t*>(a.base) + bi, op_tag(epoch, a.base_src), a.err,
                             a.wait_limit_ns)
                 : __ldcg(a.base + bi);
    }
    r = base + y;
  } else {
    // [P2] "The slow AR is Qwen3-4B": SwiGLU FFN, down(SiLU(gate) * up).
    r = silu(gate * sc) * y;
  }
  if (a.out_src >= 0) tag_store(reinterpret_cast<uint64_t*>(a.out) + oi, r, op_tag(epoch, a.out_src));
  else a.out[oi] = r;
}

// Consumer side: consumes the tiles of one GEMV and writes the epilogue.
// Combines the partials of the ntiles tiles in the window (S partials per
// row, added in segment order) and writes their epilogue.  Called by all
// consumer threads; named barrier 1 before (partials visible) and, when more
// tiles follow, after (window free again).
template <int NB>
DEVI void gemv_flush(const GemvArgs& a, const GemvGeo& g, GemvScratch<NB>& sc, const GemvPro<NB>& pr,
                     int ntiles, bool more, uint32_t epoch, uint64_t* stamp = nullptr) {
  constexpr int NCT = kWarpsC * 32;
  named_barrier(1, NCT);
  if (stamp && threadIdx.x == 0) *stamp = global_timer_ns();
  const int step = g.swiglu ? 2 : 1;   // SwiGLU: gate tile, then up tile
  const int per = g.R * NB;
  const int n = (ntiles / step) * per;
  for (int e = threadIdx.x; e < n; e += NCT) {
    const int tt = (e / per) * step, r = (e % per) / NB, b = e % NB;
    const int2 ti = sc.tile[tt];
    if (r >= ti.y) continue;
    float y = 0.f;
    for (int q = 0; q < g.S; ++q) y += sc.part[tt][r * g.S + q][b];
    float gate = 0.f;
    if (g.swiglu) {
      gate = y;
      y = 0.f;
      for (int q = 0; q < g.S; ++q) y += sc.part[tt + 1][r * g.S + q][b];
    }
    gemv_epilogue<NB>(a, g, pr, ti.x + r, b, y, gate, epoch);
  }
  if (more) named_barrier(1, NCT);
}

// Lane sums of a group of kGrp tiles' per-lane partials pg[u][b], stored as
// the warp's partials of window slots tw .. tw + ng - 1.  For kGrp = 8 one
// butterfly serves all tiles: the same pairwise sums, in the same order, as
// warp_sum per tile (so the same bits), with 9 shuffles instead of 5 per
// tile; lane 4u ends with tile u's sum.
template <int NB, int kGrp>
DEVI void gemv_group_sums(const float (&pg)[kGrp][NB], int ng, GemvScratch<NB>& sc, int tw, int warp, int lane) {
  static_assert(kGrp == 1 || kGrp == 8, "one tile, or eight in a butterfly");
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    if constexpr (kGrp == 1) {
      const float v = warp_sum(pg[0][b]);
      if (lane == 0) sc.part[tw][warp][b] = v;
    } else {
      const bool l4 = lane & 16, l3 = lane & 8, l2 = lane & 4;
      float h4[4], h3[2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float keep = l4 ? pg[i + 4][b] : pg[i][b], send = l4 ? pg[i][b] : pg[i + 4][b];
        h4[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float keep = l3 ? h4[i + 2] : h4[i], send = l3 ? h4[i] : h4[i + 2];
        h3[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
      }
      const float keep = l2 ? h3[1] : h3[0], send = l2 ? h3[0] : h3[1];
      float v = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 4);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 2);
      v += __shfl_xor_sync(0xFFFFFFFFu, v, 1);
      const int u = lane >> 2;
      if ((lane & 3) == 0 && u < ng) sc.part[tw + u][warp][b] = v;
    }
  }
}

// Consumer side: consumes the tiles of one GEMV and writes the epilogue.
// Returns false if a wait gave up.
template <int NB>
DEVI bool gemv_consume(const GemvArgs& a, const GemvGeo& g, const GemvRing& ring, uint32_t& t,
                       const float* xs, GemvScratch<NB>& sc, const GemvPro<NB>& pr, uint32_t epoch = 0,
                       uint64_t* stamp = nullptr) {
  constexpr int kWin = GemvScratch<NB>::kPartTiles;
  constexpr int kGrp = NB <= 2 ? 8 : 1;   // tiles per transposed reduction (registers: kGrp x NB)
  static_assert(kWin % kGrp == 0, "groups fill windows exactly");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K, KV = K >> 3;
  const int r = warp / g.S, sg = warp % g.S;
  const int j0 = sg * g.seg;
  const int nvec = max(0, min(g.seg, KV - j0));
  // Batch 1: this warp's x segment is the same for every row, so it is read
  // from shared memory once per op and kept in registers.
  constexpr int XR = NB == 1 ? kMaxVecPerLane : 1;
  float4 xra[XR], xrb[XR];
  if (NB == 1) {
    const float4* xa = reinterpret_cast<const float4*>(xs) + j0;
    const float4* xb = xa + KV;
#pragma unroll
    for (int q = 0; q < XR; ++q) {
      const int j = lane + 32 * q;
      xra[q] = j < nvec ? xa[j] : make_float4(0.f, 0.f, 0.f, 0.f);
      xrb[q] = j < nvec ? xb[j] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  TileIter it(a, g);
  int tw = 0;   // tiles in the current window
  bool more = true;
  while (more) {
    // kGrp tiles, then one transposed reduction for all of them
    float pg[kGrp][NB];
#pragma unroll
    for (int u = 0; u < kGrp; ++u)
#pragma unroll
      for (int b = 0; b < NB; ++b) pg[u][b] = 0.f;
    int ng = 0;
#pragma unroll
    for (int u = 0; u < kGrp; ++u) {
      int row0, rows, part;
      if (!it.next(row0, rows, part)) {
        more = false;
        break;
      }
      const int s = static_cast<int>(t % ring.stages);
      if (!mbar_wait(&ring.full[s], (t / ring.stages) & 1, a.err, a.wait_limit_ns)) return false;
      if (r < rows) {
        const uint4* wr = reinterpret_cast<const uint4*>(ring.base + static_cast<size_t>(s) * kStageBytes) +
                          static_cast<size_t>(r) * KV + j0;
        uint4 w[kMaxVecPerLane];
#pragma unroll
        for (int q = 0; q < kMaxVecPerLane; ++q) {
          const int j = lane + 32 * q;
          w[q] = j < nvec ? wr[j] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          // one accumulator per vector: independent FMA chains
          float acc[kMaxVecPerLane];
          if (NB == 1) {
#pragma unroll
            for (int q = 0; q < kMaxVecPerLane; ++q)
              acc[q] = dot8(w[q], xra[q < XR ? q : 0], xrb[q < XR ? q : 0], 0.f);
          } else {
            const float4* xa = reinterpret_cast<const float4*>(xs + static_cast<size_t>(b) * K) + j0;
            const float4* xb = xa + KV;
#pragma unroll
            for (int q = 0; q < kMaxVecPerLane; ++q) {
              const int j = lane + 32 * q;
              acc[q] = j < nvec ? dot8(w[q], xa[j], xb[j], 0.f) : 0.f;
            }
          }
          float sum = 0.f;
#pragma unroll
          for (int q = 0; q < kMaxVecPerLane; ++q) sum += acc[q];
          pg[u][b] = sum;
        }
      }
      // The stage is free once every lane's reads of it are done (the sums
      // above depend on them; the arrive is a release): the producer
      // refills it while this warp goes on.
      __syncwarp();
      if (lane == 0) mbar_arrive(&ring.empty[s]);
      ++t;
      if (threadIdx.x == 0) sc.tile[tw + u] = make_int2(row0, rows);
      ng = u + 1;
    }
    if (ng == 0) break;
    gemv_group_sums<NB, kGrp>(pg, ng, sc, tw, warp, lane);
    tw += ng;
    if (!more) break;
    if (tw == kWin) {
      gemv_flush<NB>(a, g, sc, pr, tw, true, epoch);
      tw = 0;
    }
  }
  if (tw > 0) gemv_flush<NB>(a, g, sc, pr, tw, false, epoch, stamp);
  else if (stamp && threadIdx.x == 0) *stamp = global_timer_ns();
  return true;
}

// ---- 4-bit consumer ------------------------------------------------------------
// Element of a packed row as the float 128 + u (u its stored nibble, 0..15):
// src holds one nibble per byte (the even or the odd elements of a word);
// byte I is moved to bits 16..23 under the exponent byte of 128.0f
// (0x43000000), so no integer-to-float conversion is needed.
template <int I>
DEVI float w4_val128(uint32_t src) {
  return __uint_as_float(__byte_perm(src, 0x43000000u, 0x7054u | (I << 8)));
}

// c.x += a0 * b0, c.y += a1 * b1 in one packed fp32 instruction (two
// independent round-to-nearest FMAs).
DEVI void ffma2(float2& c, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(c.x), "+f"(c.y)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// The 8 elements of one 32-bit word of codes (element e in bits 4e..4e+3)
// against x elements xa (0..3) and xb (4..7): c gets (128 + u_e) * x_e, even
// elements in c.x, odd ones in c.y.
DEVI float2 w4_word(uint32_t wd, const float4 xa, const float4 xb) {
  const uint32_t ev = wd & 0x0F0F0F0Fu, od = (wd >> 4) & 0x0F0F0F0Fu;
  float2 c = make_float2(w4_val128<0>(ev) * xa.x, w4_val128<0>(od) * xa.y);
  ffma2(c, w4_val128<1>(ev), w4_val128<1>(od), xa.z, xa.w);
  ffma2(c, w4_val128<2>(ev), w4_val128<2>(od), xb.x, xb.y);
  ffma2(c, w4_val128<3>(ev), w4_val128<3>(od), xb.z, xb.w);
  return c;
}

// Consumer side of a GEMV over packed 4-bit rows: like gemv_consume, with a
// lane's 16-byte vector holding 32 elements of one 128-element group.  For
// vector v of row n and batch row b,
//   sum_k (u_k - 8) s x'_k = s (sum_k (128 + u_k) x'_k - 136 gsum[b][v]),
// with the 32-term sum in fp32 (its terms are at most 143 |x'_k|, and the
// difference keeps about 2^-24 * 143 * 32 of relative error -- far below the
// bf16 rounding of the weights themselves).  x' in the split-32 layout of
// gemv_stage_x<NB, true>.
template <int NB>
DEVI bool gemv_consume_w4(const GemvArgs& a, const GemvGeo& g, const GemvRing& ring, uint32_t& t,
                          const float* xs, const float* gsum, GemvScratch<NB>& sc, const GemvPro<NB>& pr,
                          uint32_t epoch = 0, uint64_t* stamp = nullptr) {
  constexpr int kWin = GemvScratch<NB>::kPartTiles;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K, KV32 = K >> 5;
  const int rb = w4_row_bytes(K);
  const int r = warp / g.S, sg = warp % g.S;
  const int v0 = sg * g.seg;
  const int nvec = max(0, min(g.seg, KV32 - v0));
  TileIter it(a, g);
  int row0, rows, part;
  int tw = 0;
  while (it.next(row0, rows, part)) {
    const int s = static_cast<int>(t % ring.stages);
    if (!mbar_wait(&ring.full[s], (t / ring.stages) & 1, a.err, a.wait_limit_ns)) return false;
    const bool mine = r < rows;
    float p[NB];
    if (mine) {
      const unsigned char* rec = ring.base + static_cast<size_t>(s) * kStageBytes + static_cast<size_t>(r) * rb;
      const uint4* wr = reinterpret_cast<const uint4*>(rec) + v0;
      const uint16_t* scl = reinterpret_cast<const uint16_t*>(rec + K / 2);
      uint4 w[kMaxVecPerLane];
      float sv[kMaxVecPerLane];
#pragma unroll
      for (int q = 0; q < kMaxVecPerLane; ++q) {
        const int j = lane + 32 * q;
        w[q] = j < nvec ? wr[j] : make_uint4(0u, 0u, 0u, 0u);
        sv[q] = j < nvec ? bf16bits_to_f32(scl[(v0 + j) >> 2]) : 0.f;
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        p[b] = 0.f;
        if (b >= a.nb) continue;
        const float4* x4 = reinterpret_cast<const float4*>(xs + static_cast<size_t>(b) * K);
        const float* gs = gsum + static_cast<size_t>(b) * KV32;
#pragma unroll
        for (int q = 0; q < kMaxVecPerLane; ++q) {
          const int j = lane + 32 * q;
          if (j < nvec) {
            const int v = v0 + j;
            // four independent chains (one per word), then the group correction
            const float2 d0 = w4_word(w[q].x, x4[0 * KV32 + v], x4[1 * KV32 + v]);
            const float2 d1 = w4_word(w[q].y, x4[2 * KV32 + v], x4[3 * KV32 + v]);
            const float2 d2 = w4_word(w[q].z, x4[4 * KV32 + v], x4[5 * KV32 + v]);
            const float2 d3 = w4_word(w[q].w, x4[6 * KV32 + v], x4[7 * KV32 + v]);
            const float dv =
                fmaf(-136.f, gs[v], ((d0.x + d0.y) + (d1.x + d1.y)) + ((d2.x + d2.y) + (d3.x + d3.y)));
            p[b] = fmaf(sv[q], dv, p[b]);
          }
        }
      }
    }
    // the stage is free once every lane's reads of it are done
    __syncwarp();
    if (lane == 0) mbar_arrive(&ring.empty[s]);
    ++t;
    if (mine) {
#pragma unroll
      for (int b = 0; b < NB; ++b) p[b] = warp_sum(p[b]);
      if (lane < NB) {
        float y = p[0];
#pragma unroll
        for (int b = 1; b < NB; ++b)
          if (lane == b) y = p[b];
        sc.part[tw][warp][lane] = y;
      }
    }
    if (threadIdx.x == 0) sc.tile[tw] = make_int2(row0, rows);
    if (++tw == kWin) {
      gemv_flush<NB>(a, g, sc, pr, tw, true, epoch);
      tw = 0;
    }
  }
  if (tw > 0) gemv_flush<NB>(a, g, sc, pr, tw, false, epoch, stamp);
  else if (stamp && threadIdx.x == 0) *stamp = global_timer_ns();
  return true;
}

}  // namespace dualar
