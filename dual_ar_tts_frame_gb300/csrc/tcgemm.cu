// Batched projections on the tensor cores (tcgen05), for decode batches and
// prefill chunks of 9..128 rows:
//
//   y[m][n] = sum_k x'[m][k] W[n][k],   x' = RMSNorm(x) * g (optional)
//
// At these batch sizes a projection is still bound by the weight bytes (2*M
// FLOP per weight byte, below the ridge), but it is a dense contraction: the
// weights are read ONCE per launch instead of once per 8 rows.
//
// Three kernels per projection:
//  1. tc_split_kernel: x' per row (RMSNorm scale and gain applied), written as
//     two bf16 halves x' = hi + lo (lo = bf16(x' - hi)), so the bf16 tensor
//     cores see x' to ~16 significant bits;
//  2. tc_gemm_kernel: the weights are the MMA's M side (128 rows per
//     instruction, two instructions per CTA tile of 256 rows), the batch its N
//     side (padded to 16/32/64/128), K = 16 per instruction.  TMA copies
//     weight and activation tiles (64 K wide, 128-byte swizzle) into a ring of
//     shared-memory stages; one thread issues tcgen05.mma (hi and lo halves
//     into the same fp32 accumulator in tensor memory); four warps read the
//     accumulators back (tcgen05.ld) and store this CTA's split-K partial sums;
//  3. tc_reduce_kernel: adds the partial sums of the K slices in slice order
//     (deterministic) and applies the epilogue: store / residual add / SwiGLU,
//     with the optional output row map.
// A residual-add projection's reduce is usually fused with the next
// projection's split (tc_reduce_norm_kernel: the same sums and the same norm
// arithmetic, one CTA per row), since that projection reads the residual
// stream it writes.
// [P2] "The slow AR is Qwen3-4B" (the projections of a Qwen3 layer) and "Two
// autoregressions" (the fast AR's layers and head).
#include <cuda.h>

#include <cstdio>
#include <map>
#include <mutex>
#include <tuple>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tcgemm.h"

namespace dualar {

constexpr int kTcThreads = 192;     // warp 0: TMA, warp 1: MMA + TMEM, warps 2-5: read-back
constexpr int kTcWTile = 128 * 64 * 2;   // one 128-row x 64-K weight tile (bytes)
constexpr size_t kTcSmemBudget = 200 * 1024;
constexpr int kTcPrefetchChunks = 8;   // weight chunks (32 KB each) requested into L2 ahead of the ring

__host__ __device__ constexpr int tc_stage_bytes(int nbp) { return 2 * kTcWTile + 2 * nbp * 128; }
__host__ __device__ constexpr int tc_stages(int nbp) {
  return static_cast<int>(kTcSmemBudget / tc_stage_bytes(nbp)) > 6 ? 6
                                                                     : static_cast<int>(kTcSmemBudget / tc_stage_bytes(nbp));
}
__host__ __device__ constexpr size_t tc_smem_bytes(int nbp) {
  // stages, then full/empty/accumulator mbarriers and the TMEM address, plus
  // up to 1 KB to align the stages on 1024 bytes (128-byte swizzle atoms)
  return static_cast<size_t>(tc_stages(nbp)) * tc_stage_bytes(nbp) + 256 + 1024;
}

struct TcArgs {
  int n0, n1;          // weight rows of segment 0 (map 0) and segment 1 (map 1)
  int K;
  int nb;              // batch rows written back (<= NBP)
  int kc_per_slice;    // 64-wide K chunks per split-K slice
  float* part;         // [slices][nb][ldp] partial sums
  int ldp;             // n0 + n1
  int tma_store;       // the partial tile goes out through the tensor map tp (else plain stores)
  int kwrap;           // > 0: K runs over two weight halves; x's column is k mod kwrap (4-bit hi/lo)
  uint32_t* err;
  uint64_t wait_limit_ns;
};

template <int NBP>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tw0, const __grid_constant__ CUtensorMap tw1,
                   const __grid_constant__ CUtensorMap txh, const __grid_constant__ CUtensorMap txl,
                   const __grid_constant__ CUtensorMap tp, const TcArgs a) {
  constexpr int S = tc_stages(NBP);
  constexpr int SB = tc_stage_bytes(NBP);
  constexpr int XT = NBP * 128;                                   // one activation tile (bytes)
  constexpr uint32_t kCols = 2 * NBP < 32 ? 32u : static_cast<uint32_t>(2 * NBP);   // power of two
  static_assert(S >= 2, "at least two stages");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);   // 1024-byte aligned stages
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(accf + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, slice = blockIdx.y;
  const int kc_total = a.K / 64;
  const int c0 = slice * a.kc_per_slice;
  const int nch = min(kc_total, c0 + a.kc_per_slice) - c0;   // >= 1 (host)

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&accf[0], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    tmem_alloc(tslot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer.  The weights are constant: the first stages' weight
      // tiles are requested before waiting for the kernel that writes x.
      const uint64_t pol = policy_evict_first();
      auto load_w = [&](int i) {
        unsigned char* st = smem + (i % S) * SB;
        const int kx = (c0 + i) * 64;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int r0 = tile * 256 + t * 128;
          if (r0 < a.n0) tma_load_2d_hint(st + t * kTcWTile, &tw0, kx, r0, &full[i % S], pol);
          else tma_load_2d_hint(st + t * kTcWTile, &tw1, kx, r0 - a.n0, &full[i % S], pol);
        }
      };
      auto load_x = [&](int i) {
        unsigned char* st = smem + (i % S) * SB;
        int kx = (c0 + i) * 64;
        if (a.kwrap > 0 && kx >= a.kwrap) kx -= a.kwrap;
        tma_load_2d(st + 2 * kTcWTile, &txh, kx, 0, &full[i % S]);
        tma_load_2d(st + 2 * kTcWTile + XT, &txl, kx, 0, &full[i % S]);
      };
      const int pre = nch < S ? nch : S;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(&full[i], static_cast<uint32_t>(SB));
        load_w(i);
      }
      // and the next kTcPrefetchChunks chunks' weights into L2, so that the
      // memory keeps streaming while the kernels before this one finish
      for (int i = pre; i < nch && i < pre + kTcPrefetchChunks; ++i) {
        const int kx = (c0 + i) * 64;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int r0 = tile * 256 + t * 128;
          if (r0 < a.n0) tma_prefetch_l2_2d_hint(&tw0, kx, r0, pol);
          else tma_prefetch_l2_2d_hint(&tw1, kx, r0 - a.n0, pol);
        }
      }
      pdl_wait();
      pdl_launch();
      for (int i = 0; i < pre; ++i) load_x(i);
      int issued = pre;
      for (int i = pre; i < nch; ++i) {
        const int s = i % S;
        if (!mbar_wait(&empty[s], ((i / S) - 1) & 1, a.err, a.wait_limit_ns)) {
          raise_error(a.err, DEV_ERR_TC_WAIT);
          break;
        }
        mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(SB));
        load_w(i);
        load_x(i);
        ++issued;
      }
      // every copy issued here has landed before the CTA may exit (bounded)
      for (int i = issued > S ? issued - S : 0; i < issued; ++i) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&full[i % S], (i / S) & 1))
          if (global_timer_ns() - t0 > a.wait_limit_ns) break;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(128, NBP);
      for (int i = 0; i < nch; ++i) {
        const int s = i % S;
        if (!mbar_wait(&full[s], (i / S) & 1, a.err, a.wait_limit_ns)) {
          raise_error(a.err, DEV_ERR_TC_WAIT | (1u << 6));
          break;
        }
        tc_fence_after();
        unsigned char* st = smem + s * SB;
        const uint64_t dxh = smem_desc_sw128(st + 2 * kTcWTile);
        const uint64_t dxl = smem_desc_sw128(st + 2 * kTcWTile + XT);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint64_t dw = smem_desc_sw128(st + t * kTcWTile);
          const uint32_t dt = tbase + static_cast<uint32_t>(t * NBP);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ko = static_cast<uint64_t>(k * 32) >> 4;   // +32 bytes per 16-wide K step
            tc_mma_bf16(dt, dw + ko, dxh + ko, idesc, i > 0 || k > 0);
            tc_mma_bf16(dt, dw + ko, dxl + ko, idesc, true);
          }
        }
        tc_commit(&empty[s]);   // the stage is free once these MMAs have read it
      }
      tc_commit(&accf[0]);      // all MMAs above complete (also after an early stop)
    }
  } else {
    // ---- read-back: warp w may access TMEM lanes 32*(w%4) .. +31
    pdl_wait();   // (the partial sums' buffer is read by the previous reduce)
    const int q = warp & 3;
    const bool accd = mbar_wait(&accf[0], 0, a.err, a.wait_limit_ns);
    if (!accd && lane == 0) raise_error(a.err, DEV_ERR_TC_WAIT | (1u << 7));
    if (accd && a.tma_store) {
      // this warp's 32 weight rows of each 128-row half, for all NBP batch
      // rows, are staged in the (now idle) stage ring as [NBP][32] blocks
      // and leave in two tensor stores (no other warp involved)
      tc_fence_after();
      constexpr int CW = NBP < 64 ? NBP : 64;
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        float* blk = reinterpret_cast<float*>(smem) + ((warp - 2) * 2 + t) * (NBP * 32);
#pragma unroll 1
        for (int c0 = 0; c0 < NBP; c0 += CW) {
          uint32_t v[CW / 16][16];
#pragma unroll
          for (int c = 0; c < CW / 16; ++c)
            tmem_ld16_async(tbase + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(t * NBP + c0 + c * 16),
                            v[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < CW / 16; ++c)
#pragma unroll
            for (int j = 0; j < 16; ++j) blk[(c0 + c * 16 + j) * 32 + lane] = __uint_as_float(v[c][j]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        // (kept in L2 until the reduce reads them: the weight streams are evict-first)
        if (lane == 0) tma_store_3d_hint(&tp, blk, tile * 256 + t * 128 + q * 32, 0, slice, policy_evict_last());
      }
      if (lane == 0) {
        tma_store_commit();
        tma_store_wait();
      }
      __syncwarp();
    } else if (accd) {
      tc_fence_after();
      // up to 64 accumulator columns per round: their loads issued together,
      // one wait, then the stores (lane = weight row: 128-byte rows per store)
      constexpr int CW = NBP < 64 ? NBP : 64;
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {
        const int n = tile * 256 + t * 128 + q * 32 + lane;   // weight row of this lane
#pragma unroll 1
        for (int c0 = 0; c0 < NBP; c0 += CW) {
          uint32_t v[CW / 16][16];
#pragma unroll
          for (int c = 0; c < CW / 16; ++c)
            tmem_ld16_async(tbase + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(t * NBP + c0 + c * 16),
                            v[c]);
          tmem_wait_ld();
          if (n < a.ldp) {
            float* dst = a.part + (static_cast<size_t>(slice) * a.nb + c0) * a.ldp + n;
#pragma unroll
            for (int c = 0; c < CW / 16; ++c)
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + c * 16 + j < a.nb) dst[static_cast<size_t>(c * 16 + j) * a.ldp] = __uint_as_float(v[c][j]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kCols);
  }
}

// x' rows as bf16 hi/lo: one CTA of 1024 threads per row; the row is read
// once (float4, kept in registers: K <= 12288) and written as 4 bf16 per
// 8-byte store.
constexpr int kSplitThreads = 1024;
constexpr int kSplitVec = 3;   // float4 per thread

__global__ void __launch_bounds__(kSplitThreads, 1)
    tc_split_kernel(const float* x, int ldx, int K, const uint16_t* norm_w, float eps, uint16_t* xh, uint16_t* xl,
                    int ldxh, float* save_x, const int32_t* save_map, int lds) {
  pdl_launch();   // the next projection may start fetching its weights
  pdl_wait();
  const int m = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(m) * ldx);
  const int KV = K >> 2;
  __shared__ float red[32];
  float4 v[kSplitVec];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < kSplitVec; ++q) {
    const int j = threadIdx.x + q * kSplitThreads;
    v[q] = j < KV ? xr[j] : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += v[q].x * v[q].x + v[q].y * v[q].y + v[q].z * v[q].z + v[q].w * v[q].w;
  }
  float sc = 1.f;
  if (norm_w != nullptr) {
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float t = 0.f;
#pragma unroll 8
    for (int w = 0; w < kSplitThreads / 32; ++w) t += red[w];
    sc = 1.0f / sqrtf(t / static_cast<float>(K) + eps);
  }
  const int row = save_x ? (save_map ? save_map[m] : m) : -1;
#pragma unroll
  for (int q = 0; q < kSplitVec; ++q) {
    const int j = threadIdx.x + q * kSplitThreads;
    if (j >= KV) continue;
    float e[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
    if (norm_w != nullptr) {
      const uint2 gw = *reinterpret_cast<const uint2*>(norm_w + 4 * j);
      e[0] = (e[0] * bf16lo(gw.x)) * sc;
      e[1] = (e[1] * bf16hi(gw.x)) * sc;
      e[2] = (e[2] * bf16lo(gw.y)) * sc;
      e[3] = (e[3] * bf16hi(gw.y)) * sc;
    }
    uint32_t h[4], l[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint16_t hb = f32_to_bf16bits(e[c]);
      h[c] = hb;
      l[c] = f32_to_bf16bits(e[c] - bf16bits_to_f32(hb));
    }
    *reinterpret_cast<uint2*>(xh + static_cast<size_t>(m) * ldxh + 4 * j) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    *reinterpret_cast<uint2*>(xl + static_cast<size_t>(m) * ldxh + 4 * j) = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
    if (row >= 0)
      *reinterpret_cast<float4*>(save_x + static_cast<size_t>(row) * lds + 4 * j) = make_float4(e[0], e[1], e[2], e[3]);
  }
}

// Split-K sum at offset off of the partials: every slice's float4 in
// flight at once (slices <= MAXS), added in slice order.
template <int MAXS>
DEVI float4 tc_slice_sum(const float* part, int slices, size_t stride, size_t off) {
  float4 t[MAXS];
#pragma unroll
  for (int k = 0; k < MAXS; ++k)
    if (k < slices) t[k] = *reinterpret_cast<const float4*>(part + off + k * stride);
  float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < MAXS; ++k)
    if (k < slices) {
      y.x += t[k].x; y.y += t[k].y; y.z += t[k].z; y.w += t[k].w;
    }
  return y;
}

// Residual add of the K-slice partials (slice order, as tc_reduce_kernel),
// then the split of the result as tc_split_kernel does it (the same thread
// mapping, so the same sums): out = base + sum, x' = RMSNorm(out) * g.
__global__ void __launch_bounds__(kSplitThreads, 1)
    tc_reduce_norm_kernel(const float* part, int slices, int nb, int ldp, int K, const float* base, int ldb,
                          float* out, int ldo, const uint16_t* norm_w, float eps, uint16_t* xh, uint16_t* xl,
                          int ldxh, float* save_x, const int32_t* save_map, int lds) {
  pdl_launch();   // the next projection may start fetching its weights
  pdl_wait();
  const int m = blockIdx.x;
  const int KV = K >> 2;
  const size_t stride = static_cast<size_t>(nb) * ldp;
  __shared__ float red[32];
  float4 v[kSplitVec];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < kSplitVec; ++q) {
    const int j = threadIdx.x + q * kSplitThreads;
    v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < KV) {
      const float* p0 = part + static_cast<size_t>(m) * ldp + 4 * j;
      float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
      int sl = 0;
      for (; sl + 8 <= slices; sl += 8) {
        float4 t[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) t[k] = *reinterpret_cast<const float4*>(p0 + (sl + k) * stride);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          y.x += t[k].x; y.y += t[k].y; y.z += t[k].z; y.w += t[k].w;
        }
      }
      for (; sl < slices; ++sl) {
        const float4 t = *reinterpret_cast<const float4*>(p0 + sl * stride);
        y.x += t.x; y.y += t.y; y.z += t.z; y.w += t.w;
      }
      const float4 bb = *reinterpret_cast<const float4*>(base + static_cast<size_t>(m) * ldb + 4 * j);
      v[q] = make_float4(bb.x + y.x, bb.y + y.y, bb.z + y.z, bb.w + y.w);
      *reinterpret_cast<float4*>(out + static_cast<size_t>(m) * ldo + 4 * j) = v[q];
    }
    ss += v[q].x * v[q].x + v[q].y * v[q].y + v[q].z * v[q].z + v[q].w * v[q].w;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float t = 0.f;
#pragma unroll 8
  for (int w = 0; w < kSplitThreads / 32; ++w) t += red[w];
  const float sc = 1.0f / sqrtf(t / static_cast<float>(K) + eps);
  const int row = save_x ? (save_map ? save_map[m] : m) : -1;
#pragma unroll
  for (int q = 0; q < kSplitVec; ++q) {
    const int j = threadIdx.x + q * kSplitThreads;
    if (j >= KV) continue;
    const uint2 gw = *reinterpret_cast<const uint2*>(norm_w + 4 * j);
    float e[4] = {(v[q].x * bf16lo(gw.x)) * sc, (v[q].y * bf16hi(gw.x)) * sc, (v[q].z * bf16lo(gw.y)) * sc,
                  (v[q].w * bf16hi(gw.y)) * sc};
    uint32_t h[4], l[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint16_t hb = f32_to_bf16bits(e[c]);
      h[c] = hb;
      l[c] = f32_to_bf16bits(e[c] - bf16bits_to_f32(hb));
    }
    *reinterpret_cast<uint2*>(xh + static_cast<size_t>(m) * ldxh + 4 * j) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
    *reinterpret_cast<uint2*>(xl + static_cast<size_t>(m) * ldxh + 4 * j) = make_uint2(l[0] | (l[1] << 16), l[2] | (l[3] << 16));
    if (row >= 0)
      *reinterpret_cast<float4*>(save_x + static_cast<size_t>(row) * lds + 4 * j) = make_float4(e[0], e[1], e[2], e[3]);
  }
}

// Sum of the K-slice partials (slice order) and the epilogue, 4 columns per
// thread (all row strides multiples of 4 floats).
template <int MAXS>
__global__ void tc_reduce_kernel(const float* part, int slices, int nb, int ldp, int n_out, int mode, float* out,
                                 int ldo, const float* base, int ldb, const int32_t* out_map, int n0, uint16_t* xh,
                                 uint16_t* xl, int ldxh) {
  pdl_launch();   // the next projection may start fetching its weights
  pdl_wait();
  const int nq = n_out >> 2;   // n_out % 4 == 0 (host)
  const size_t total = static_cast<size_t>(nb) * nq;
  // the slices' partials, all loads in flight, added in slice order
  auto sum = [&](const float* p0, size_t stride) { return tc_slice_sum<MAXS>(p0, slices, stride, 0); };
  for (size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(e / nq), n = 4 * static_cast<int>(e % nq);
    const int orow = out_map ? out_map[m] : m;
    if (orow < 0) continue;
    const size_t stride = static_cast<size_t>(nb) * ldp;
    const float4 y = sum(part + static_cast<size_t>(m) * ldp + n, stride);
    float4 r;
    if (mode == GEMV_SWIGLU) {
      const float4 u = sum(part + static_cast<size_t>(m) * ldp + n0 + n, stride);
      // [P2] "The slow AR is Qwen3-4B": down(SiLU(gate) * up)
      r = make_float4(silu(y.x) * u.x, silu(y.y) * u.y, silu(y.z) * u.z, silu(y.w) * u.w);
    } else if (mode == GEMV_ADD) {
      const float4 b = *reinterpret_cast<const float4*>(base + static_cast<size_t>(orow) * ldb + n);
      r = make_float4(b.x + y.x, b.y + y.y, b.z + y.z, b.w + y.w);
    } else {
      r = y;
    }
    *reinterpret_cast<float4*>(out + static_cast<size_t>(orow) * ldo + n) = r;
    if (xh != nullptr) {
      // the output is the next projection's input (no norm): its bf16 halves
      const float e4[4] = {r.x, r.y, r.z, r.w};
      uint32_t hh[4], ll[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint16_t hb = f32_to_bf16bits(e4[c]);
        hh[c] = hb;
        ll[c] = f32_to_bf16bits(e4[c] - bf16bits_to_f32(hb));
      }
      *reinterpret_cast<uint2*>(xh + static_cast<size_t>(m) * ldxh + n) = make_uint2(hh[0] | (hh[1] << 16), hh[2] | (hh[3] << 16));
      *reinterpret_cast<uint2*>(xl + static_cast<size_t>(m) * ldxh + n) = make_uint2(ll[0] | (ll[1] << 16), ll[2] | (ll[3] << 16));
    }
  }
}

// The same, one column per thread (rows not 16-byte aligned: the head's 4,097).
__global__ void tc_reduce_scalar_kernel(const float* part, int slices, int nb, int ldp, int n_out, int mode,
                                        float* out, int ldo, const float* base, int ldb, const int32_t* out_map,
                                        int n0) {
  pdl_launch();   // the next projection may start fetching its weights
  pdl_wait();
  const size_t total = static_cast<size_t>(nb) * n_out;
  for (size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(e / n_out), n = static_cast<int>(e % n_out);
    const int orow = out_map ? out_map[m] : m;
    if (orow < 0) continue;
    float y = 0.f;
    for (int s = 0; s < slices; ++s) y += part[(static_cast<size_t>(s) * nb + m) * ldp + n];
    float r;
    if (mode == GEMV_SWIGLU) {
      float u = 0.f;
      for (int s = 0; s < slices; ++s) u += part[(static_cast<size_t>(s) * nb + m) * ldp + n0 + n];
      r = silu(y) * u;
    } else if (mode == GEMV_ADD) {
      r = base[static_cast<size_t>(orow) * ldb + n] + y;
    } else {
      r = y;
    }
    out[static_cast<size_t>(orow) * ldo + n] = r;
  }
}

// ---- host side ------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool tc_available() { return encode_fn() != nullptr; }

// bf16 matrix [rows][K] (row stride ld elements), tiles of box_rows x 64,
// 128-byte swizzle; rows beyond `rows` read as zeros.
static bool make_map(CUtensorMap* m, const void* base, int K, int rows, int ld, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t es[2] = {1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps are built once per (address, K, rows, box) and kept.
static bool cached_map(CUtensorMap* out, const void* base, int K, int rows, int ld, int box_rows) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, int, int>, CUtensorMap> cache;
  std::lock_guard<std::mutex> g(mu);
  const auto key = std::make_tuple(base, K, rows, ld, box_rows);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return true;
  }
  CUtensorMap m;
  if (!make_map(&m, base, K, rows, ld, box_rows)) return false;
  cache.emplace(key, m);
  *out = m;
  return true;
}

// fp32 [slices][nb][ldp] (rows of ldp floats), boxes of 32 x box_nb x 1;
// built once per argument set and kept.
static bool part_map(CUtensorMap* out, const float* base, int ldp, int nb, int slices, int box_nb) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, int, int>, CUtensorMap> cache;
  std::lock_guard<std::mutex> g(mu);
  const auto key = std::make_tuple(static_cast<const void*>(base), ldp, nb, slices, box_nb);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return true;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(ldp), static_cast<cuuint64_t>(nb),
                              static_cast<cuuint64_t>(slices)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ldp) * 4, static_cast<cuuint64_t>(ldp) * nb * 4};
  const cuuint32_t box[3] = {32u, static_cast<cuuint32_t>(box_nb), 1u};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  CUtensorMap m;
  if (fn(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  cache.emplace(key, m);
  *out = m;
  return true;
}

bool tc_bf16_map(CUtensorMap* out, const void* base, int K, int rows, int ld, int box_rows) {
  return cached_map(out, base, K, rows, ld, box_rows);
}

bool tc_eligible(const GemvArgs& a, int ldx) {
  if (!tc_available()) return false;
  if (a.nb < kTcMinRows || a.nb > kTcMaxRows || a.K % 64 != 0 || a.K > ldx) return false;
  if (a.K > 4 * kSplitThreads * kSplitVec) return false;          // one row in registers
  if (a.ldx % 4 != 0 || (a.save_x && a.lds % 4 != 0)) return false;   // float4 rows in the split
  if (a.x_src >= 0 || a.base_src >= 0 || a.out_src >= 0) return false;   // plain buffers only
  if (a.mode == GEMV_SWIGLU) return a.n0 % 128 == 0 && a.n1 == a.n0;
  return a.n1 == 0 || a.n0 % 128 == 0;
}

template <int NBP>
static cudaError_t launch_gemm_nbp(const CUtensorMap& w0, const CUtensorMap& w1, const CUtensorMap& xh,
                                   const CUtensorMap& xl, const CUtensorMap& tp, const TcArgs& t, dim3 grid,
                                   cudaStream_t st, bool pdl) {
  static bool configured = false;
  const size_t smem = tc_smem_bytes(NBP);
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<NBP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (!pdl) {
    tc_gemm_kernel<NBP><<<grid, kTcThreads, smem, st>>>(w0, w1, xh, xl, tp, t);
    return cudaGetLastError();
  }
  return launch_pdl(tc_gemm_kernel<NBP>, grid, dim3(kTcThreads), smem, st, w0, w1, xh, xl, tp, t);
}

cudaError_t launch_tc_gemm(const GemvArgs& a, const TcBuffers& b, int n_sm, cudaStream_t st, int* launches,
                           bool x_ready, bool split_out, TcPending* defer, bool weights_pdl, bool w_hilo) {
  const int nbp = a.nb <= 16 ? 16 : a.nb <= 32 ? 32 : a.nb <= 64 ? 64 : 128;
  const int n_rows = a.n0 + a.n1;   // virtual weight rows (SwiGLU: gate then up)
  const int tiles = (n_rows + 255) / 256;
  const int kw = w_hilo ? 2 * a.K : a.K;   // weight columns
  const int kc = kw / 64;
  int slices = (n_sm + tiles / 2) / tiles;
  slices = slices < 1 ? 1 : slices > kTcMaxSlices ? kTcMaxSlices : slices;
  if (slices > kc) slices = kc;
  const int kcps = (kc + slices - 1) / slices;
  slices = (kc + kcps - 1) / kcps;   // no empty slice
  if (static_cast<size_t>(slices) * a.nb * n_rows > b.part_floats) return cudaErrorInvalidValue;

  CUtensorMap m0, m1, mh, ml;
  const int seg1 = a.n1 > 0 ? a.n1 : 1;
  if (!cached_map(&m0, a.w0, kw, a.n0, kw, 128) ||
      !cached_map(&m1, a.n1 > 0 ? a.w1 : a.w0, kw, seg1, kw, 128) ||
      !cached_map(&mh, b.xh, a.K, kTcMaxRows, b.ldx, nbp) || !cached_map(&ml, b.xl, a.K, kTcMaxRows, b.ldx, nbp))
    return cudaErrorInvalidValue;

  cudaError_t e = cudaSuccess;
  if (!x_ready) {
    e = launch_pdl(tc_split_kernel, dim3(a.nb), dim3(kSplitThreads), 0, st, a.x, a.ldx, a.K, a.norm_w, a.eps, b.xh,
                   b.xl, b.ldx, a.save_x, a.save_map, a.lds);
    if (e != cudaSuccess) return e;
    if (launches) *launches += 1;
  }
  // the partial sums as a [slices][nb][ldp] fp32 tensor, boxes of 32 x NBP x 1
  CUtensorMap mp;
  const bool tstore = n_rows % 4 == 0 && part_map(&mp, b.part, n_rows, a.nb, slices, nbp);
  if (!tstore) mp = m0;   // unused
  TcArgs t{a.n0, a.n1, kw, a.nb, kcps, b.part, n_rows, tstore ? 1 : 0, w_hilo ? a.K : 0, a.err, a.wait_limit_ns};
  const dim3 grid(tiles, slices);
  switch (nbp) {
    case 16: e = launch_gemm_nbp<16>(m0, m1, mh, ml, mp, t, grid, st, weights_pdl); break;
    case 32: e = launch_gemm_nbp<32>(m0, m1, mh, ml, mp, t, grid, st, weights_pdl); break;
    case 64: e = launch_gemm_nbp<64>(m0, m1, mh, ml, mp, t, grid, st, weights_pdl); break;
    default: e = launch_gemm_nbp<128>(m0, m1, mh, ml, mp, t, grid, st, weights_pdl); break;
  }
  if (e != cudaSuccess) return e;
  const int n_out = a.mode == GEMV_SWIGLU ? a.n0 : n_rows;
  const bool vec = n_out % 4 == 0 && n_rows % 4 == 0 && a.ldo % 4 == 0 && (a.mode != GEMV_ADD || a.ldb % 4 == 0);
  if (split_out && (!vec || a.out_map != nullptr || n_out > b.ldx)) return cudaErrorInvalidValue;
  if (defer != nullptr && a.mode == GEMV_ADD && vec && a.out_map == nullptr && !split_out) {
    defer->on = true;
    defer->slices = slices;
    defer->nb = a.nb;
    defer->ldp = n_rows;
    defer->n_out = n_out;
    defer->out = a.out;
    defer->ldo = a.ldo;
    defer->base = a.base;
    defer->ldb = a.ldb;
    if (launches) *launches += 1;
    return cudaSuccess;
  }
  const size_t total = static_cast<size_t>(a.nb) * (vec ? n_out / 4 : n_out);
  int rgrid = static_cast<int>((total + 255) / 256);
  rgrid = rgrid > 8 * n_sm ? 8 * n_sm : rgrid;
  if (vec)
    e = launch_pdl(slices <= 4 ? tc_reduce_kernel<4> : slices <= 8 ? tc_reduce_kernel<8> : tc_reduce_kernel<16>, dim3(rgrid), dim3(256), 0, st, static_cast<const float*>(b.part), slices, a.nb,
                   n_rows, n_out, a.mode, a.out, a.ldo, a.base, a.ldb, a.out_map, a.n0,
                   split_out ? b.xh : static_cast<uint16_t*>(nullptr), split_out ? b.xl : static_cast<uint16_t*>(nullptr),
                   b.ldx);
  else
    e = launch_pdl(tc_reduce_scalar_kernel, dim3(rgrid), dim3(256), 0, st, static_cast<const float*>(b.part), slices,
                   a.nb, n_rows, n_out, a.mode, a.out, a.ldo, a.base, a.ldb, a.out_map, a.n0);
  if (launches) *launches += 2;
  return e;
}

bool tc_can_fuse(const TcPending& p, const GemvArgs& a) {
  return p.on && a.x == p.out && a.ldx == p.ldo && a.K == p.n_out && a.nb == p.nb && a.norm_w != nullptr &&
         a.K <= 4 * kSplitThreads * kSplitVec && (a.save_x == nullptr || a.lds % 4 == 0);
}

cudaError_t launch_tc_pending(const TcPending& p, const TcBuffers& b, int n_sm, cudaStream_t st) {
  const size_t total = static_cast<size_t>(p.nb) * (p.n_out / 4);
  int rgrid = static_cast<int>((total + 255) / 256);
  rgrid = rgrid > 8 * n_sm ? 8 * n_sm : rgrid;
  return launch_pdl(p.slices <= 4 ? tc_reduce_kernel<4> : p.slices <= 8 ? tc_reduce_kernel<8> : tc_reduce_kernel<16>, dim3(rgrid), dim3(256), 0, st, static_cast<const float*>(b.part), p.slices,
                    p.nb, p.ldp, p.n_out, static_cast<int>(GEMV_ADD), p.out, p.ldo, p.base, p.ldb,
                    static_cast<const int32_t*>(nullptr), 0, static_cast<uint16_t*>(nullptr),
                    static_cast<uint16_t*>(nullptr), b.ldx);
}

cudaError_t launch_tc_reduce_norm(const TcPending& p, const GemvArgs& a, const TcBuffers& b, cudaStream_t st) {
  return launch_pdl(tc_reduce_norm_kernel, dim3(p.nb), dim3(kSplitThreads), 0, st, static_cast<const float*>(b.part),
                    p.slices, p.nb, p.ldp, p.n_out, p.base, p.ldb, p.out, p.ldo, a.norm_w, a.eps, b.xh, b.xl, b.ldx,
                    a.save_x, a.save_map, a.lds);
}

}  // namespace dualar
