// Split-KV GQA attention over the paged cache on the tensor cores, for
// launches of 3 or more rows (decode batches, prefill chunks).
//
// Same work units as attn_paged_units (row, KV head, chunk of pages), the
// same partial-sum format and the same deterministic last-arriver combine.
// Inside a unit the G query heads of the KV head are the rows of warp-level
// MMAs (mma.sync m16n8k16, bf16 operands, fp32 accumulators; tcgen05's
// M >= 64 would waste far more):
//   S = Q K^T  (Q: the unit's query heads, 1/sqrt(hd) folded in, split into
//               bf16 hi + lo halves that sit in different rows of the same
//               MMA: rows h and h + 4 for G <= 4, rows h and h + 8 for G = 8;
//               the two row results are added afterwards),
//   online softmax over the page on the fragment rows,
//   O += P V   (P split into hi + lo rows the same way).
// A CTA has eight warps with fixed roles, chained by mbarriers:
//  * prep (warp 5) takes units from a per-layer counter shared by all CTAs
//    (a CTA that finishes early takes more): first every full chunk, row
//    by row, then every row's last (partial) chunk, rows ordered by that
//    chunk's page count, largest first.  For each it loads the page
//    indices, the query rows (QK-norm and RoPE when fused), and for the
//    unit holding the newest position that position's K/V, which it writes
//    to the cache; it publishes the unit in one of two shared-memory
//    descriptors;
//  * producer (warp 4, one lane) copies the units' K and V pages by TMA
//    (128-byte swizzle, so ldmatrix reads are conflict-free) into a ring of
//    page slots (K then V) that every compute warp reads in order (so an
//    mbarrier wait is never more than one phase ahead of its barrier: a
//    parity wait cannot tell phases two apart); the ring holds 160-192 KB
//    (five or six pages at hd 128), all lookahead for the four warps;
//  * compute warp w takes tokens 16 w .. 16 w + 15 of every page (a
//    function of the page alone, so the rounding does not depend on the
//    schedule), with its own running (m, l, O);
//  * compute warps hand their (m, l, O) to
//  * finalize (warps 6 and 7, alternate units), which merges the four in
//    warp order, writes the partial (or the output), and for the last chunk
//    of a (row, KV head) to arrive combines the chunks in chunk order.
// The compute warps thus never wait on global memory between units.  The
// page copy of the newest position may predate its cache write; the compute
// warp patches that row in shared memory from the descriptor.
// [P2] "The slow AR is Qwen3-4B" (GQA: 32 query heads over 8 KV heads,
// qk-norm, RoPE) and "Streaming: whose numbers" (bf16 RoPE tables).
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"
#include "ops.cuh"
#include "tc.cuh"
#include "tcgemm.h"

namespace dualar {

constexpr int kAmWarps = 4;                        // compute warps
constexpr int kAmProducer = kAmWarps;              // page copies
constexpr int kAmPrep = kAmWarps + 1;              // unit set-up
constexpr int kAmFinal = kAmWarps + 2;             // merge and combine: two warps, alternate units
constexpr int kAmFinalWarps = 2;
constexpr int kAmThreads = (kAmWarps + 2 + kAmFinalWarps) * 32;
constexpr int kAmBox = 64 * 64 * 2;                // one TMA box: 64 tokens x 64 dims (bf16)
constexpr uint32_t kAmUnitUsers = 1 + kAmWarps + 1;   // producer, compute warps, finalize

template <int HD, int G>
struct AmCfg {
  static constexpr int HALVES = HD / 64;                  // boxes per 64-token K (or V) block
  static constexpr int HALF = HALVES * kAmBox;            // the K (or the V) block of one page
  static constexpr int SLOT = 2 * HALF;                   // a slot: one page, K then V
  // pages in the ring: 192 KB, 160 KB where the merge buffers are largest
  static constexpr int NBUF = ((HD == 128 && G > 4 ? 160 : 192) * 1024) / SLOT;
};

// One unit as the prep warp publishes it.
template <int HD, int G>
struct AmUnitDesc {
  float q[G][HD];                         // query rows, 1/sqrt(hd) folded in
  uint32_t knew[HD / 2], vnew[HD / 2];    // newest position's K and V (bf16 pairs)
  int32_t pages[kMaxChunkPages];
  int32_t r, g, c, nch, t0, t1, npages, pos, newest, last;
};

// The launch's rows and the unit order built from them.
struct AmSmemRows {
  RowInfo rows[kMaxRows];    // read once at the start
  int32_t fpre[kMaxRows];    // full-chunk units before each row
  int32_t lorder[kMaxRows];  // active rows by last-chunk page count, largest first
  int32_t lcur[kMaxChunkPages + 1];
};
static_assert(kMaxRows == 4 * 32, "the prep warp's row scan: four rows per lane");

template <int HD, int G>
struct AmSmem {
  // after the ring
  AmUnitDesc<HD, G> unit[2];
  // the compute warps' states of units k (buffer k % 2), for finalize warp k % 2
  float co[2][kAmWarps][G][HD];
  float cm[2][kAmWarps][8], cl[2][kAmWarps][8];
  struct Fin {
    float fw[kAmWarps][8];              // merge weight of each warp's state, per head
    float m[8], ls[8];                  // merged max and sum, per head
    float fm[8][kMaxChunks], fl[8][kMaxChunks];   // chunk combine: max (then weight) and sum
  } fin[kAmFinalWarps];
  AmSmemRows t;
  uint64_t full[AmCfg<HD, G>::NBUF], empty[AmCfg<HD, G>::NBUF];
  uint64_t ufull[2], uempty[2], cfull[2], cempty[2];
  int abort_flag;
};

template <int HD, int G>
constexpr size_t am_smem_bytes() {
  return static_cast<size_t>(AmCfg<HD, G>::NBUF) * AmCfg<HD, G>::SLOT + sizeof(AmSmem<HD, G>) + 1024;
}

DEVI void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
DEVI void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
// C += A B: A 16x16 (a0/a2: row g, a1/a3: row g + 8 of the fragment layout),
// B 16x8, fp32 C (c0/c1: row g, c2/c3: row g + 8).
DEVI void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// (x, y) -> bf16x2 hi (x in the low half) and the residual lo = bf16x2(v - hi)
DEVI void split2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - __low2float(h), y - __high2float(h));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}
DEVI uint32_t pack_bf16(float x, float y) {
  return static_cast<uint32_t>(f32_to_bf16bits(x)) | (static_cast<uint32_t>(f32_to_bf16bits(y)) << 16);
}
// shared address of (token, dim) in a K or V block of 64 tokens stored as
// HD/64 swizzled boxes of [64 tokens][128 bytes]
DEVI uint32_t sw_addr(uint32_t block, int tok, int dim) {
  const int box = dim >> 6, chunk = (dim & 63) >> 3;
  return block + box * kAmBox + tok * 128 + ((chunk ^ (tok & 7)) << 4) + ((dim & 7) << 1);
}

DEVI bool am_wait(uint64_t* bar, uint32_t parity, const volatile int* abort_flag, const DevPtrs& d) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > d.wait_limit_ns) {
      raise_error(d.err, DEV_ERR_MBAR_TIMEOUT | DEV_ERR_ATTN_WAIT);
      return false;
    }
  }
  return true;
}

struct AmUnit {
  int r, g, c, nch, t0, t1, npages;
  RowInfo ri;
  const int32_t* ptab;
};

// Unit v of the launch's order (full chunks row by row, then the last
// chunks in lorder): its row, KV head and chunk.
DEVI void am_unit(const DevPtrs& d, const AmSmemRows& t, int nrows, int ftot, int v, int chunk_tokens, AmUnit& un) {
  if (v < ftot) {
    int lo = 0, hi = nrows - 1;   // the last row with fpre <= v
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (t.fpre[mid] <= v) lo = mid;
      else hi = mid - 1;
    }
    un.r = lo;
    un.ri = t.rows[lo];
    un.nch = (un.ri.pos + chunk_tokens) / chunk_tokens;
    const int local = v - t.fpre[lo];
    un.g = local / (un.nch - 1);
    un.c = local % (un.nch - 1);
  } else {
    const int w = v - ftot;
    un.r = t.lorder[w / d.Hkv];
    un.ri = t.rows[un.r];
    un.nch = (un.ri.pos + chunk_tokens) / chunk_tokens;
    un.g = w % d.Hkv;
    un.c = un.nch - 1;
  }
  const int L = un.ri.pos + 1;
  un.t0 = un.c * chunk_tokens;
  un.t1 = min(L, un.t0 + chunk_tokens);
  un.npages = (un.t1 - un.t0 + kPageTokens - 1) / kPageTokens;
  un.ptab = d.page_table + static_cast<size_t>(un.ri.slot) * d.pages_per_seq + un.t0 / kPageTokens;
}

// Whole warp: page p's index for p = lane + 32 * i in pg[i] (-1 beyond the
// unit); false if any index is out of range.  One round trip.
template <int NPG>
DEVI bool am_pages(const DevPtrs& d, const AmUnit& un, int lane, int (&pg)[NPG]) {
  bool ok = true;
#pragma unroll
  for (int i = 0; i < NPG; ++i) {
    const int p = lane + 32 * i;
    pg[i] = p < un.npages ? ldi(un.ptab + p) : -1;
    if (p < un.npages && (pg[i] < 0 || pg[i] >= d.max_pages)) ok = false;
  }
  return __all_sync(0xFFFFFFFFu, ok);
}
constexpr int kAmPageRegs = (kMaxChunkPages + 31) / 32;

// RMS norm over the head (gains nw, or none) then RoPE on adjacent pairs,
// with the position's cos/sin already loaded; lane holds dims lane*EPL ...
template <int EPL>
DEVI void am_norm_rope(float (&v)[EPL], const float (&nw)[EPL], bool norm, float eps, const float (&cs)[EPL / 2],
                       const float (&sn)[EPL / 2]) {
  if (norm) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < EPL; ++j) s += v[j] * v[j];
    s = warp_sum(s);
    const float inv = 1.0f / sqrtf(s / static_cast<float>(EPL * 32) + eps);
#pragma unroll
    for (int j = 0; j < EPL; ++j) v[j] = (v[j] * inv) * nw[j];
  }
#pragma unroll
  for (int pp = 0; pp < EPL / 2; ++pp) {
    const float x0 = v[2 * pp], x1 = v[2 * pp + 1];
    v[2 * pp] = x0 * cs[pp] - x1 * sn[pp];
    v[2 * pp + 1] = x1 * cs[pp] + x0 * sn[pp];
  }
}

template <int HD, int G>
__global__ void __launch_bounds__(kAmThreads, 1)
    attn_mma_kernel(const __grid_constant__ CUtensorMap tkv, const DevPtrs d, int nrows, int layer, int total_units,
                    int chunk_tokens, int fuse, const uint16_t* q_norm, const uint16_t* k_norm, const AttnHalves hv) {
  using C = AmCfg<HD, G>;
  using Desc = AmUnitDesc<HD, G>;
  constexpr int NB = C::NBUF;
  constexpr int EPL = HD / 32;
  constexpr bool ROWS8 = G > 4;   // lo halves in rows 8..15 (else rows 4..7)
  static_assert(G >= 1 && G <= 8, "query heads per KV head: the MMA rows 0..7");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  AmSmem<HD, G>& sm = *reinterpret_cast<AmSmem<HD, G>*>(ring + NB * C::SLOT);
  const uint32_t ring_s = smem_addr(ring);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hkv = d.Hkv, hq = d.Hq;
  if (tid == 0) {
    for (int b = 0; b < NB; ++b) {
      mbar_init(&sm.full[b], 1);
      mbar_init(&sm.empty[b], kAmWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.ufull[b], 1);
      mbar_init(&sm.uempty[b], kAmUnitUsers);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.cfull[b], kAmWarps);
      mbar_init(&sm.cempty[b], 1);
    }
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  pdl_launch();
  for (int i = tid; i < nrows; i += kAmThreads) sm.t.rows[i] = ld_row(&d.rows[i]);
  __syncthreads();
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == kAmPrep) {
    // ---- prep: publish the CTA's units in order, then an end marker
    const float qscale = 1.0f / sqrtf(static_cast<float>(HD));
    const bool qnorm = fuse && q_norm != nullptr, knorm = fuse && k_norm != nullptr;
    float qw[EPL], kw[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      qw[j] = qnorm ? bf16bits_to_f32(q_norm[lane * EPL + j]) : 1.f;
      kw[j] = knorm ? bf16bits_to_f32(k_norm[lane * EPL + j]) : 1.f;
    }
    // the unit order: per-row full-chunk counts (prefix sums), and the
    // active rows sorted by their last chunk's page count (counting sort)
    AmSmemRows& t = sm.t;
    for (int i = lane; i <= kMaxChunkPages; i += 32) t.lcur[i] = 0;
    __syncwarp();
    int fl[4], lp[4], fs = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = lane * 4 + i;
      fl[i] = lp[i] = 0;
      if (r < nrows && t.rows[r].active) {
        const int L = t.rows[r].pos + 1, nch = (L + chunk_tokens - 1) / chunk_tokens;
        fl[i] = (nch - 1) * hkv;
        lp[i] = (L - (nch - 1) * chunk_tokens + kPageTokens - 1) / kPageTokens;   // 1 .. chunk pages
        atomicAdd(&t.lcur[lp[i]], 1);
      }
      fs += fl[i];
    }
    int fx = fs;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, fx, o);
      if (lane >= o) fx += y;
    }
    const int ftot = __shfl_sync(0xFFFFFFFFu, fx, 31);
    {
      int fe = fx - fs;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        t.fpre[lane * 4 + i] = fe;
        fe += fl[i];
      }
    }
    __syncwarp();
    // bins in descending page count: lane takes counts 64 - 2 lane and 63 - 2 lane
    const int s0 = kMaxChunkPages - 2 * lane, s1 = s0 - 1;
    const int h0 = t.lcur[s0], h1 = s1 >= 1 ? t.lcur[s1] : 0;
    int hx = h0 + h1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, hx, o);
      if (lane >= o) hx += y;
    }
    const int nact = __shfl_sync(0xFFFFFFFFu, hx, 31);
    __syncwarp();
    t.lcur[s0] = hx - h0 - h1;
    if (s1 >= 1) t.lcur[s1] = hx - h1;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (lp[i] > 0) t.lorder[atomicAdd(&t.lcur[lp[i]], 1)] = lane * 4 + i;
    __syncwarp();
    const int total = ftot + nact * hkv;

    uint32_t k = 0;
    bool ok = true;
    uint32_t* counter = d.sched + layer;
    int next = 0;
    if (lane == 0) next = static_cast<int>(atomicAdd(counter, 1u));
    for (;;) {
      const int v = __shfl_sync(0xFFFFFFFFu, next, 0);
      if (v >= total) break;
      if (lane == 0) next = static_cast<int>(atomicAdd(counter, 1u));   // the one after (its latency overlaps)
      AmUnit un;
      am_unit(d, t, nrows, ftot, v, chunk_tokens, un);
      int pg[kAmPageRegs];
      if (!am_pages(d, un, lane, pg)) {
        if (lane == 0) raise_error(d.err, DEV_ERR_BAD_PAGE);
        continue;
      }
      const int r = un.r, pos = un.ri.pos;
      const bool newest = fuse && un.c == un.nch - 1;
      // loads first (they touch no shared memory)
      float qv[G][EPL];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float* src = fuse ? d.qkv + static_cast<size_t>(r) * d.qkv_dim + (un.g * G + h) * HD
                                : d.qrot + (static_cast<size_t>(r) * hq + un.g * G + h) * HD;
#pragma unroll
        for (int j = 0; j < EPL; ++j) qv[h][j] = ldf(src + lane * EPL + j);
      }
      float cs[EPL / 2], sn[EPL / 2];
      if (fuse) {
#pragma unroll
        for (int pp = 0; pp < EPL / 2; ++pp) {
          const size_t i = static_cast<size_t>(pos) * (HD / 2) + (lane * EPL) / 2 + pp;
          cs[pp] = bf16bits_to_f32(d.rope_cos[i]);
          sn[pp] = bf16bits_to_f32(d.rope_sin[i]);
        }
      }
      float kv[EPL], vv[EPL];
      if (newest) {
        const float* base = d.qkv + static_cast<size_t>(r) * d.qkv_dim + hq * HD + un.g * HD + lane * EPL;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
          kv[j] = ldf(base + j);
          vv[j] = ldf(base + hkv * HD + j);
        }
      }
      const int b = static_cast<int>(k & 1);
      if (k >= 2 && !am_wait(&sm.uempty[b], ((k >> 1) - 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        ok = false;
        break;
      }
      Desc& un_d = sm.unit[b];
#pragma unroll
      for (int i = 0; i < kAmPageRegs; ++i)
        if (lane + 32 * i < un.npages) un_d.pages[lane + 32 * i] = pg[i];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (fuse) am_norm_rope<EPL>(qv[h], qw, qnorm, d.eps, cs, sn);
#pragma unroll
        for (int j = 0; j < EPL; ++j) un_d.q[h][lane * EPL + j] = qv[h][j] * qscale;
      }
      if (newest) {
        am_norm_rope<EPL>(kv, kw, knorm, d.eps, cs, sn);
        // the newest position's page: the unit's page (pos - t0) / 64
        const int pl = (pos - un.t0) / kPageTokens;
        int pgn = 0;
#pragma unroll
        for (int i = 0; i < kAmPageRegs; ++i) {
          const int x = __shfl_sync(0xFFFFFFFFu, pg[i], pl & 31);
          if ((pl >> 5) == i) pgn = x;
        }
        const size_t page_stride = static_cast<size_t>(kPageTokens) * HD;
        uint16_t* kd = d.kv_pool + (((static_cast<size_t>(pgn) * d.n_layer + layer) * 2 + 0) * hkv + un.g) * page_stride +
                       static_cast<size_t>(pos % kPageTokens) * HD + lane * EPL;
        uint16_t* vd = kd + static_cast<size_t>(hkv) * page_stride;
#pragma unroll
        for (int j = 0; j < EPL; j += 2) {
          const uint32_t kp = pack_bf16(kv[j], kv[j + 1]), vp = pack_bf16(vv[j], vv[j + 1]);
          *reinterpret_cast<uint32_t*>(kd + j) = kp;
          *reinterpret_cast<uint32_t*>(vd + j) = vp;
          un_d.knew[(lane * EPL + j) / 2] = kp;
          un_d.vnew[(lane * EPL + j) / 2] = vp;
        }
      }
      if (lane == 0) {
        un_d.r = r;
        un_d.g = un.g;
        un_d.c = un.c;
        un_d.nch = un.nch;
        un_d.t0 = un.t0;
        un_d.t1 = un.t1;
        un_d.npages = un.npages;
        un_d.pos = pos;
        un_d.newest = newest ? 1 : 0;
        un_d.last = 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.ufull[b]);
      ++k;
    }
    // end markers: one for every reader, and one more for the finalize warp
    // that takes the next unit number
    for (int e = 0; ok && e < 2; ++e, ++k) {
      const int b = static_cast<int>(k & 1);
      if (k >= 2 && !am_wait(&sm.uempty[b], ((k >> 1) - 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        return;
      }
      if (lane == 0) {
        sm.unit[b].last = 1;
        mbar_arrive(&sm.ufull[b]);
      }
      __syncwarp();
    }
    return;
  }

  if (warp == kAmProducer) {
    // ---- producer (lane 0): the K/V pages of the published units, in order,
    // into a ring of page slots that every compute warp reads
    if (lane != 0) return;
    uint32_t gp = 0;   // pages issued
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
      const int b = static_cast<int>(k & 1);
      if (!am_wait(&sm.ufull[b], (k >> 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        break;
      }
      const Desc& un_d = sm.unit[b];
      if (un_d.last) break;
      const int npages = un_d.npages, g = un_d.g;
      for (int p = 0; p < npages; ++p, ++gp) {
        const int pgp = un_d.pages[p];
        const int s = static_cast<int>(gp % NB);
        if (gp >= static_cast<uint32_t>(NB) && !am_wait(&sm.empty[s], ((gp / NB) - 1) & 1, abort_flag, d)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        const int rowk = static_cast<int>(((static_cast<long long>(pgp) * d.n_layer + layer) * 2 * hkv + g) * 64);
        mbar_arrive_expect_tx(&sm.full[s], static_cast<uint32_t>(C::SLOT));
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
          for (int hh = 0; hh < C::HALVES; ++hh)
            tma_load_2d(ring + s * C::SLOT + kv * C::HALF + hh * kAmBox, &tkv, hh * 64, rowk + kv * hkv * 64,
                        &sm.full[s]);
      }
      if (ok) mbar_arrive(&sm.uempty[b]);
    }
    // every copy issued here lands before the CTA exits (bounded)
    for (uint32_t j = gp > static_cast<uint32_t>(NB) ? gp - NB : 0; j < gp; ++j) {
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&sm.full[j % NB], (j / NB) & 1))
        if (global_timer_ns() - t0 > d.wait_limit_ns) break;
    }
    return;
  }

  if (warp >= kAmFinal) {
    // ---- finalize warp fi: units fi, fi + 2, ... (descriptor and state
    // buffers fi); merge the compute warps' states, write, combine chunks
    constexpr int EPLF = HD / 32;
    const int fi = warp - kAmFinal;
    auto& fz = sm.fin[fi];
    for (uint32_t k = static_cast<uint32_t>(fi);; k += 2) {
      const int b = fi;
      if (!am_wait(&sm.ufull[b], (k >> 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        return;
      }
      const Desc& un_d = sm.unit[b];
      if (un_d.last) return;
      if (!am_wait(&sm.cfull[b], (k >> 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        return;
      }
      const int r = un_d.r, g = un_d.g, c = un_d.c, nch = un_d.nch;
      const size_t attn_off = static_cast<size_t>(r) * hq * HD + g * G * HD;
      float* pw = d.part + ((static_cast<size_t>(r) * hkv + g) * kMaxChunks + c) * G * (HD + 2);
      if (lane < G) {
        const int h = lane;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kAmWarps; ++w) M = fmaxf(M, sm.cm[b][w][h]);
        float Ls = 0.f;
#pragma unroll
        for (int w = 0; w < kAmWarps; ++w) {
          const float fw = sm.cm[b][w][h] == -INFINITY ? 0.f : expf(sm.cm[b][w][h] - M);
          fz.fw[w][h] = fw;
          Ls += sm.cl[b][w][h] * fw;
        }
        fz.m[h] = M;
        fz.ls[h] = Ls;
      }
      __syncwarp();
      for (int e = lane; e < G * HD; e += 32) {
        const int h = e / HD, dd = e % HD;
        float Os = 0.f;
#pragma unroll
        for (int w = 0; w < kAmWarps; ++w) Os += sm.co[b][w][h][dd] * fz.fw[w][h];
        if (nch == 1) {
          const float o1[1] = {Os / fz.ls[h]};
          d.attn[attn_off + h * HD + dd] = o1[0];
          if (hv.xh != nullptr) attn_halves<1>(hv, r, (g * G + h) * HD + dd, o1);
        } else {
          pw[h * (HD + 2) + dd] = Os;
          if (dd == 0) {
            pw[h * (HD + 2) + HD] = fz.m[h];
            pw[h * (HD + 2) + HD + 1] = fz.ls[h];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.cempty[b]);
      if (nch > 1) {
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          const uint32_t old = atomic_add_acq_rel_gpu(&d.arrive[r * hkv + g], 1u);
          if (old == static_cast<uint32_t>(nch - 1)) {
            // reset before any output of this (row, head) is written
            atomicExch(&d.arrive[r * hkv + g], 0u);
            last = 1;
          }
        }
        if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
          // the chunks in chunk order: every chunk's (m, l) first (one
          // round of loads), the weights per head, then O with all heads'
          // loads of a chunk in flight together
          __threadfence();
          const float* pb = d.part + (static_cast<size_t>(r) * hkv + g) * kMaxChunks * G * (HD + 2);
          for (int i = lane; i < nch * G; i += 32) {
            const int cc = i / G, h = i % G;
            const float* q = pb + (cc * G + h) * (HD + 2);
            fz.fm[h][cc] = ldf(q + HD);
            fz.fl[h][cc] = ldf(q + HD + 1);
          }
          __syncwarp();
          if (lane < G) {
            const int h = lane;
            float M = -INFINITY;
            for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, fz.fm[h][cc]);
            float Ls = 0.f;
            for (int cc = 0; cc < nch; ++cc) {
              const float f = expf(fz.fm[h][cc] - M);
              fz.fm[h][cc] = f;
              Ls += fz.fl[h][cc] * f;
            }
            fz.ls[h] = Ls;
          }
          __syncwarp();
          float os[G][EPLF];
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int j = 0; j < EPLF; ++j) os[h][j] = 0.f;
#pragma unroll 2
          for (int cc = 0; cc < nch; ++cc) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float* q = pb + (cc * G + h) * (HD + 2) + lane * EPLF;
              const float f = fz.fm[h][cc];
#pragma unroll
              for (int j = 0; j < EPLF; ++j) os[h][j] += ldf(q + j) * f;
            }
          }
#pragma unroll
          for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int j = 0; j < EPLF; ++j) {
              os[h][j] = os[h][j] / fz.ls[h];
              d.attn[attn_off + h * HD + lane * EPLF + j] = os[h][j];
            }
            if (hv.xh != nullptr) attn_halves<EPLF>(hv, r, (g * G + h) * HD + lane * EPLF, os[h]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.uempty[b]);
    }
  }

  // ---- compute warps
  const int gr = lane >> 2, tq = lane & 3;          // fragment row and column pair
  const int head = ROWS8 ? gr : (gr & 3);           // the query head of this lane's rows
  const bool lo_row = !ROWS8 && gr >= 4;            // rows 4..7 carry the lo halves (G <= 4)
  const bool writer = (ROWS8 || gr < 4) && head < G;
  uint32_t gp = 0;   // pages taken so far (the ring position)
  for (uint32_t k = 0;; ++k) {
    const int b = static_cast<int>(k & 1);
    if (!am_wait(&sm.ufull[b], (k >> 1) & 1, abort_flag, d)) {
      *abort_flag = 1;
      return;
    }
    const Desc& un_d = sm.unit[b];
    if (un_d.last) return;
    const int t0 = un_d.t0, t1 = un_d.t1, npages = un_d.npages, pos = un_d.pos;
    const bool newest = un_d.newest != 0;
    // Q fragments: row gr holds the hi half of head gr; the lo half sits in
    // row gr + 4 (G <= 4: another lane) or row gr + 8 (G = 8: a1/a3)
    uint32_t qa[HD / 16][2], qb[HD / 16][2];
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int dd = ks * 16 + half * 8 + 2 * tq;
        const float x = head < G ? un_d.q[head][dd] : 0.f, y = head < G ? un_d.q[head][dd + 1] : 0.f;
        uint32_t hi, lo;
        split2(x, y, hi, lo);
        qa[ks][half] = lo_row ? lo : hi;
        qb[ks][half] = ROWS8 ? lo : 0u;
      }
    }
    float m_run = -INFINITY, l_run = 0.f;
    float o[HD / 8][4];
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    // every page of the unit; this warp takes its tokens 16 warp .. +15
    const int tw = 16 * warp;
    for (int p = 0; p < npages; ++p, ++gp) {
      const int s = static_cast<int>(gp % NB);
      if (!am_wait(&sm.full[s], (gp / NB) & 1, abort_flag, d)) {
        *abort_flag = 1;
        return;
      }
      const int ps = t0 + p * kPageTokens;
      const int ntok = min(kPageTokens, t1 - ps);
      const uint32_t kb = ring_s + s * C::SLOT, vb = kb + C::HALF;
      if (newest && ps + tw <= pos && pos < ps + tw + 16) {
        // the newest row (its copy may predate the cache write)
        const int rr = pos - ps;
        if (lane < HD / 8) {
          const uint32_t ak = sw_addr(kb, rr, lane * 8), av = sw_addr(vb, rr, lane * 8);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ak), "r"(un_d.knew[lane * 4]),
                       "r"(un_d.knew[lane * 4 + 1]), "r"(un_d.knew[lane * 4 + 2]), "r"(un_d.knew[lane * 4 + 3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(av), "r"(un_d.vnew[lane * 4]),
                       "r"(un_d.vnew[lane * 4 + 1]), "r"(un_d.vnew[lane * 4 + 2]), "r"(un_d.vnew[lane * 4 + 3])
                       : "memory");
        }
        // (the slot is refilled by TMA later: order these writes before it)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      if (tw < ntok) {
        // S = Q K^T over the warp's 16 tokens: 2 tiles of 8
        float sc[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
          uint32_t bb[4];
          const int tok = tw + (lane >> 4) * 8 + (lane & 7);
          const int dim = ks * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x4(bb, sw_addr(kb, tok, dim));
          mma16816(sc[0], qa[ks][0], qb[ks][0], qa[ks][1], qb[ks][1], bb[0], bb[1]);
          mma16816(sc[1], qa[ks][0], qb[ks][0], qa[ks][1], qb[ks][1], bb[2], bb[3]);
        }
        // hi + lo rows -> the head's scores (tokens tw + 8j + 2tq, +1)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (ROWS8) {
            sc[j][0] += sc[j][2];
            sc[j][1] += sc[j][3];
          } else {
            sc[j][0] += __shfl_xor_sync(0xFFFFFFFFu, sc[j][0], 16);
            sc[j][1] += __shfl_xor_sync(0xFFFFFFFFu, sc[j][1], 16);
          }
        }
        // online softmax on the head's row
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int t = tw + 8 * j + 2 * tq;
          if (t >= ntok) sc[j][0] = -INFINITY;
          if (t + 1 >= ntok) sc[j][1] = -INFINITY;
          mx = fmaxf(mx, fmaxf(sc[j][0], sc[j][1]));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const float m_new = fmaxf(m_run, mx);   // finite: token tw is valid
        const float f = expf(m_run - m_new);     // 0 while m_run = -inf
        float ps_sum = 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          sc[j][0] = expf(sc[j][0] - m_new);
          sc[j][1] = expf(sc[j][1] - m_new);
          ps_sum += sc[j][0] + sc[j][1];
        }
        ps_sum += __shfl_xor_sync(0xFFFFFFFFu, ps_sum, 1);
        ps_sum += __shfl_xor_sync(0xFFFFFFFFu, ps_sum, 2);
        l_run = l_run * f + ps_sum;
        m_run = m_new;
#pragma unroll
        for (int n = 0; n < HD / 8; ++n) {
          o[n][0] *= f;
          o[n][1] *= f;
          if (ROWS8) {
            o[n][2] *= f;
            o[n][3] *= f;
          }
        }
        // O += P V over the 16 tokens
        uint32_t ph0, pl0, ph2, pl2;
        split2(sc[0][0], sc[0][1], ph0, pl0);
        split2(sc[1][0], sc[1][1], ph2, pl2);
        const uint32_t a0 = lo_row ? pl0 : ph0, a2 = lo_row ? pl2 : ph2;
        const uint32_t a1 = ROWS8 ? pl0 : 0u, a3 = ROWS8 ? pl2 : 0u;
#pragma unroll
        for (int np = 0; np < HD / 16; ++np) {
          uint32_t bb[4];
          const int tok = tw + ((lane >> 3) & 1) * 8 + (lane & 7);
          const int dim = np * 16 + (lane >> 4) * 8;
          ldsm_x4_t(bb, sw_addr(vb, tok, dim));
          mma16816(o[2 * np], a0, a1, a2, a3, bb[0], bb[1]);
          mma16816(o[2 * np + 1], a0, a1, a2, a3, bb[2], bb[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);   // this warp's reads of the slot are done
    }

    // hand (m, l, O) to the finalize warp
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      if (ROWS8) {
        o[n][0] += o[n][2];
        o[n][1] += o[n][3];
      } else {
        o[n][0] += __shfl_xor_sync(0xFFFFFFFFu, o[n][0], 16);
        o[n][1] += __shfl_xor_sync(0xFFFFFFFFu, o[n][1], 16);
      }
    }
    // (state buffer b was last used by unit k - 2)
    if (k >= 2 && !am_wait(&sm.cempty[b], ((k >> 1) - 1) & 1, abort_flag, d)) {
      *abort_flag = 1;
      return;
    }
    if (writer) {
      if (tq == 0) {
        sm.cm[b][warp][head] = m_run;
        sm.cl[b][warp][head] = l_run;
      }
#pragma unroll
      for (int n = 0; n < HD / 8; ++n) {
        sm.co[b][warp][head][8 * n + 2 * tq] = o[n][0];
        sm.co[b][warp][head][8 * n + 2 * tq + 1] = o[n][1];
      }
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&sm.cfull[b]);
      mbar_arrive(&sm.uempty[b]);
    }
  }
}

// ============================================================================
// Prefill: query blocks
// ============================================================================
// A prefill launch holds consecutive positions of one sequence, whose K/V
// the append kernel has already written.  Here a unit is (a block of
// QB = 32 / G consecutive rows, KV head g, chunk c of the block's last row),
// so every page is read once for QB rows instead of once per row.  Compute
// warp w owns rows w RW .. w RW + RW - 1 (RW = 8 / G) over all 64 tokens of
// every page: its 8 (row, head) pairs are MMA rows 0..7 with the bf16 hi
// halves of Q and P and rows 8..15 with the lo halves, and each row masks
// the positions after its own.  No merge between warps (each owns whole
// rows); the finalize warps write every row's partial (or output) and
// combine a row's chunks, in chunk order, when its last chunk arrives.  The
// prep, producer and finalize roles, the page ring and the dynamic schedule
// are those of the decode kernel above.
template <int HD, int G>
struct ApCfg {
  static constexpr int RW = 8 / G;                        // rows per compute warp
  static constexpr int QB = kAmWarps * RW;                // rows per unit
  static constexpr int SLOT = AmCfg<HD, G>::SLOT;
  static constexpr int NBUF = ((HD == 128 ? 160 : 192) * 1024) / SLOT;
};

struct ApDesc {
  int32_t pages[kMaxChunkPages];
  int32_t r0, nr, g, c, nch, t0, t1, npages, last;
};

template <int HD, int G>
struct ApSmem {
  ApDesc unit[2];
  float co[2][kAmWarps][8][HD];           // each warp's 8 (row, head) states of unit k (buffer k % 2)
  float cm[2][kAmWarps][8], cl[2][kAmWarps][8];
  struct Fin {
    float fm[8][kMaxChunks], fl[8][kMaxChunks];
  } fin[kAmFinalWarps];
  RowInfo rows[kMaxRows];
  int32_t bpre[kMaxRows + 1];             // units before each block
  uint64_t full[ApCfg<HD, G>::NBUF], empty[ApCfg<HD, G>::NBUF];
  uint64_t ufull[2], uempty[2], cfull[2], cempty[2];
  int abort_flag;
};

template <int HD, int G>
constexpr size_t ap_smem_bytes() {
  return static_cast<size_t>(ApCfg<HD, G>::NBUF) * ApCfg<HD, G>::SLOT + sizeof(ApSmem<HD, G>) + 1024;
}

template <int HD, int G>
__global__ void __launch_bounds__(kAmThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tkv, const DevPtrs d, int nrows, int layer,
                        int chunk_tokens) {
  using C = ApCfg<HD, G>;
  constexpr int NB = C::NBUF, RW = C::RW, QB = C::QB;
  constexpr int HALF = AmCfg<HD, G>::HALF, HALVES = AmCfg<HD, G>::HALVES;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  ApSmem<HD, G>& sm = *reinterpret_cast<ApSmem<HD, G>*>(ring + NB * C::SLOT);
  const uint32_t ring_s = smem_addr(ring);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hkv = d.Hkv, hq = d.Hq;
  if (tid == 0) {
    for (int b = 0; b < NB; ++b) {
      mbar_init(&sm.full[b], 1);
      mbar_init(&sm.empty[b], kAmWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sm.ufull[b], 1);
      mbar_init(&sm.uempty[b], kAmUnitUsers);
      mbar_init(&sm.cfull[b], kAmWarps);
      mbar_init(&sm.cempty[b], 1);
    }
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();
  pdl_launch();
  for (int i = tid; i < nrows; i += kAmThreads) sm.rows[i] = ld_row(&d.rows[i]);
  __syncthreads();
  volatile int* abort_flag = &sm.abort_flag;
  const int nblk = (nrows + QB - 1) / QB;

  if (warp == kAmPrep) {
    // ---- prep: units from the shared counter; pages and row range per unit
    if (lane == 0) {
      int acc = 0;
      for (int b = 0; b < nblk; ++b) {
        sm.bpre[b] = acc;
        const int rl = min(nrows, (b + 1) * QB) - 1;
        acc += hkv * ((sm.rows[rl].pos + chunk_tokens) / chunk_tokens);
      }
      sm.bpre[nblk] = acc;
    }
    __syncwarp();
    const int total = sm.bpre[nblk];
    uint32_t k = 0;
    bool ok = true;
    uint32_t* counter = d.sched + layer;
    int next = 0;
    if (lane == 0) next = static_cast<int>(atomicAdd(counter, 1u));
    for (;;) {
      const int v = __shfl_sync(0xFFFFFFFFu, next, 0);
      if (v >= total) break;
      if (lane == 0) next = static_cast<int>(atomicAdd(counter, 1u));
      int b = 0;
      while (b + 1 < nblk && sm.bpre[b + 1] <= v) ++b;
      const int r0 = b * QB, nr = min(nrows, r0 + QB) - r0;
      const RowInfo first = sm.rows[r0], lastr = sm.rows[r0 + nr - 1];
      // the block's rows must be consecutive positions of one sequence
      bool rows_ok = lane >= nr || (sm.rows[r0 + lane].slot == first.slot && sm.rows[r0 + lane].pos == first.pos + lane &&
                                    sm.rows[r0 + lane].active);
      if (!__all_sync(0xFFFFFFFFu, rows_ok)) {
        if (lane == 0) raise_error(d.err, DEV_ERR_BAD_INDEX);
        continue;
      }
      const int L = lastr.pos + 1;
      AmUnit un;
      un.nch = (L + chunk_tokens - 1) / chunk_tokens;
      const int local = v - sm.bpre[b];
      un.g = local / un.nch;
      un.c = local % un.nch;
      un.t0 = un.c * chunk_tokens;
      un.t1 = min(L, un.t0 + chunk_tokens);
      un.npages = (un.t1 - un.t0 + kPageTokens - 1) / kPageTokens;
      un.ptab = d.page_table + static_cast<size_t>(first.slot) * d.pages_per_seq + un.t0 / kPageTokens;
      int pg[kAmPageRegs];
      if (!am_pages(d, un, lane, pg)) {
        if (lane == 0) raise_error(d.err, DEV_ERR_BAD_PAGE);
        continue;
      }
      const int bb = static_cast<int>(k & 1);
      if (k >= 2 && !am_wait(&sm.uempty[bb], ((k >> 1) - 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        ok = false;
        break;
      }
      ApDesc& ud = sm.unit[bb];
#pragma unroll
      for (int i = 0; i < kAmPageRegs; ++i)
        if (lane + 32 * i < un.npages) ud.pages[lane + 32 * i] = pg[i];
      if (lane == 0) {
        ud.r0 = r0;
        ud.nr = nr;
        ud.g = un.g;
        ud.c = un.c;
        ud.nch = un.nch;
        ud.t0 = un.t0;
        ud.t1 = un.t1;
        ud.npages = un.npages;
        ud.last = 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.ufull[bb]);
      ++k;
    }
    for (int e = 0; ok && e < 2; ++e, ++k) {
      const int bb = static_cast<int>(k & 1);
      if (k >= 2 && !am_wait(&sm.uempty[bb], ((k >> 1) - 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        return;
      }
      if (lane == 0) {
        sm.unit[bb].last = 1;
        mbar_arrive(&sm.ufull[bb]);
      }
      __syncwarp();
    }
    return;
  }

  if (warp == kAmProducer) {
    // ---- producer (lane 0): every unit's pages into the ring
    if (lane != 0) return;
    uint32_t gp = 0;
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
      const int b = static_cast<int>(k & 1);
      if (!am_wait(&sm.ufull[b], (k >> 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        break;
      }
      const ApDesc& ud = sm.unit[b];
      if (ud.last) break;
      for (int p = 0; p < ud.npages; ++p, ++gp) {
        const int pgp = ud.pages[p];
        const int s = static_cast<int>(gp % NB);
        if (gp >= static_cast<uint32_t>(NB) && !am_wait(&sm.empty[s], ((gp / NB) - 1) & 1, abort_flag, d)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        const int rowk = static_cast<int>(((static_cast<long long>(pgp) * d.n_layer + layer) * 2 * hkv + ud.g) * 64);
        mbar_arrive_expect_tx(&sm.full[s], static_cast<uint32_t>(C::SLOT));
#pragma unroll
        for (int kv = 0; kv < 2; ++kv)
#pragma unroll
          for (int hh = 0; hh < HALVES; ++hh)
            tma_load_2d(ring + s * C::SLOT + kv * HALF + hh * kAmBox, &tkv, hh * 64, rowk + kv * hkv * 64,
                        &sm.full[s]);
      }
      if (ok) mbar_arrive(&sm.uempty[b]);
    }
    for (uint32_t j = gp > static_cast<uint32_t>(NB) ? gp - NB : 0; j < gp; ++j) {
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try_wait(&sm.full[j % NB], (j / NB) & 1))
        if (global_timer_ns() - t0 > d.wait_limit_ns) break;
    }
    return;
  }

  if (warp >= kAmFinal) {
    // ---- finalize warp fi: units fi, fi + 2, ...
    constexpr int EPLF = HD / 32;
    const int fi = warp - kAmFinal;
    auto& fz = sm.fin[fi];
    for (uint32_t k = static_cast<uint32_t>(fi);; k += 2) {
      const int b = fi;
      if (!am_wait(&sm.ufull[b], (k >> 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        return;
      }
      const ApDesc& ud = sm.unit[b];
      if (ud.last) return;
      if (!am_wait(&sm.cfull[b], (k >> 1) & 1, abort_flag, d)) {
        *abort_flag = 1;
        return;
      }
      const int r0 = ud.r0, nr = ud.nr, g = ud.g, c = ud.c, nch = ud.nch;
      // every (warp, pair) -> (row, head): output, or this chunk's partial
      for (int e = lane; e < kAmWarps * 8 * HD; e += 32) {
        const int w = e / (8 * HD), vv = (e / HD) % 8, dd = e % HD;
        const int jr = w * RW + vv / G, h = vv % G;
        if (jr >= nr) continue;
        const int r = r0 + jr;
        const float O = sm.co[b][w][vv][dd];
        if (nch == 1) {
          d.attn[static_cast<size_t>(r) * hq * HD + (g * G + h) * HD + dd] = O / sm.cl[b][w][vv];
        } else {
          float* pw = d.part + ((static_cast<size_t>(r) * hkv + g) * kMaxChunks + c) * G * (HD + 2) + h * (HD + 2);
          pw[dd] = O;
          if (dd == 0) {
            pw[HD] = sm.cm[b][w][vv];
            pw[HD + 1] = sm.cl[b][w][vv];
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.cempty[b]);
      if (nch > 1) {
        __threadfence();
        __syncwarp();
        // every row's arrival at once (lane = row), then the rows this unit completes
        int last = 0;
        if (lane < nr) {
          const int r = r0 + lane;
          const uint32_t old = atomic_add_acq_rel_gpu(&d.arrive[r * hkv + g], 1u);
          if (old == static_cast<uint32_t>(nch - 1)) {
            atomicExch(&d.arrive[r * hkv + g], 0u);
            last = 1;
          }
        }
        const uint32_t lastmask = __ballot_sync(0xFFFFFFFFu, last);
        for (int jr = 0; jr < nr; ++jr) {
          const int r = r0 + jr;
          if (!((lastmask >> jr) & 1u)) continue;
          // row r's chunks in chunk order
          __threadfence();
          const float* pb = d.part + (static_cast<size_t>(r) * hkv + g) * kMaxChunks * G * (HD + 2);
          for (int i = lane; i < nch * G; i += 32) {
            const int cc = i / G, h = i % G;
            const float* q = pb + (cc * G + h) * (HD + 2);
            fz.fm[h][cc] = ldf(q + HD);
            fz.fl[h][cc] = ldf(q + HD + 1);
          }
          __syncwarp();
          if (lane < G) {
            const int h = lane;
            float M = -INFINITY;
            for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, fz.fm[h][cc]);
            float Ls = 0.f;
            for (int cc = 0; cc < nch; ++cc) {
              const float f = fz.fm[h][cc] == -INFINITY ? 0.f : expf(fz.fm[h][cc] - M);
              fz.fm[h][cc] = f;
              Ls += fz.fl[h][cc] * f;
            }
            fz.fl[h][0] = Ls;   // (fl is not read again for this row)
          }
          __syncwarp();
          float os[G][EPLF];
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int j = 0; j < EPLF; ++j) os[h][j] = 0.f;
#pragma unroll 2
          for (int cc = 0; cc < nch; ++cc) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
              const float* q = pb + (cc * G + h) * (HD + 2) + lane * EPLF;
              const float f = fz.fm[h][cc];
#pragma unroll
              for (int j = 0; j < EPLF; ++j) os[h][j] += ldf(q + j) * f;
            }
          }
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int j = 0; j < EPLF; ++j)
              d.attn[static_cast<size_t>(r) * hq * HD + (g * G + h) * HD + lane * EPLF + j] = os[h][j] / fz.fl[h][0];
          __syncwarp();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.uempty[b]);
    }
  }

  // ---- compute warps
  const int gr = lane >> 2, tq = lane & 3;
  const float qscale = 1.0f / sqrtf(static_cast<float>(HD));
  uint32_t gp = 0;
  for (uint32_t k = 0;; ++k) {
    const int b = static_cast<int>(k & 1);
    if (!am_wait(&sm.ufull[b], (k >> 1) & 1, abort_flag, d)) {
      *abort_flag = 1;
      return;
    }
    const ApDesc& ud = sm.unit[b];
    if (ud.last) return;
    const int t0 = ud.t0, t1 = ud.t1, npages = ud.npages, g = ud.g;
    // this lane's (row, head): row rw0 + gr / G, head gr % G
    const int jr = warp * RW + gr / G, h = gr % G;
    const bool valid = jr < ud.nr;
    const int r = ud.r0 + (valid ? jr : 0);
    const int plim = valid ? sm.rows[r].pos : -1;   // the last position this row sees
    uint32_t qa[HD / 16][2], qb[HD / 16][2];
    const float* qsrc = d.qrot + (static_cast<size_t>(r) * hq + g * G + h) * HD;
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int dd = ks * 16 + half * 8 + 2 * tq;
        const float x = valid ? ldf(qsrc + dd) * qscale : 0.f, y = valid ? ldf(qsrc + dd + 1) * qscale : 0.f;
        split2(x, y, qa[ks][half], qb[ks][half]);
      }
    }
    float m_run = -INFINITY, l_run = 0.f;
    float o[HD / 8][4];
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    for (int p = 0; p < npages; ++p, ++gp) {
      const int s = static_cast<int>(gp % NB);
      if (!am_wait(&sm.full[s], (gp / NB) & 1, abort_flag, d)) {
        *abort_flag = 1;
        return;
      }
      const int ps = t0 + p * kPageTokens;
      const uint32_t kb = ring_s + s * C::SLOT, vb = kb + HALF;
      float sc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          uint32_t bb[4];
          const int tok = jp * 16 + (lane >> 4) * 8 + (lane & 7);
          const int dim = ks * 16 + ((lane >> 3) & 1) * 8;
          ldsm_x4(bb, sw_addr(kb, tok, dim));
          mma16816(sc[2 * jp], qa[ks][0], qb[ks][0], qa[ks][1], qb[ks][1], bb[0], bb[1]);
          mma16816(sc[2 * jp + 1], qa[ks][0], qb[ks][0], qa[ks][1], qb[ks][1], bb[2], bb[3]);
        }
      }
      // hi + lo rows -> scores; positions after the row's own, or past the chunk, masked
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        sc[j][0] += sc[j][2];
        sc[j][1] += sc[j][3];
        const int t = ps + 8 * j + 2 * tq;
        if (t > plim || t >= t1) sc[j][0] = -INFINITY;
        if (t + 1 > plim || t + 1 >= t1) sc[j][1] = -INFINITY;
        mx = fmaxf(mx, fmaxf(sc[j][0], sc[j][1]));
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const bool none = m_new == -INFINITY;   // nothing visible to this row yet
      const float f = none ? 1.f : expf(m_run - m_new);
      float ps_sum = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        sc[j][0] = none ? 0.f : expf(sc[j][0] - m_new);
        sc[j][1] = none ? 0.f : expf(sc[j][1] - m_new);
        ps_sum += sc[j][0] + sc[j][1];
      }
      ps_sum += __shfl_xor_sync(0xFFFFFFFFu, ps_sum, 1);
      ps_sum += __shfl_xor_sync(0xFFFFFFFFu, ps_sum, 2);
      l_run = l_run * f + ps_sum;
      m_run = m_new;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n) {
        o[n][0] *= f;
        o[n][1] *= f;
        o[n][2] *= f;
        o[n][3] *= f;
      }
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        uint32_t ph0, pl0, ph2, pl2;
        split2(sc[2 * kt][0], sc[2 * kt][1], ph0, pl0);
        split2(sc[2 * kt + 1][0], sc[2 * kt + 1][1], ph2, pl2);
#pragma unroll
        for (int np = 0; np < HD / 16; ++np) {
          uint32_t bb[4];
          const int tok = kt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
          const int dim = np * 16 + (lane >> 4) * 8;
          ldsm_x4_t(bb, sw_addr(vb, tok, dim));
          mma16816(o[2 * np], ph0, pl0, ph2, pl2, bb[0], bb[1]);
          mma16816(o[2 * np + 1], ph0, pl0, ph2, pl2, bb[2], bb[3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
    }
    // hand the rows' (m, l, O) to the finalize warp
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      o[n][0] += o[n][2];
      o[n][1] += o[n][3];
    }
    if (k >= 2 && !am_wait(&sm.cempty[b], ((k >> 1) - 1) & 1, abort_flag, d)) {
      *abort_flag = 1;
      return;
    }
    if (tq == 0) {
      sm.cm[b][warp][gr] = m_run;
      sm.cl[b][warp][gr] = l_run;
    }
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      sm.co[b][warp][gr][8 * n + 2 * tq] = o[n][0];
      sm.co[b][warp][gr][8 * n + 2 * tq + 1] = o[n][1];
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&sm.cfull[b]);
      mbar_arrive(&sm.uempty[b]);
    }
  }
}

template <int HD, int G>
static cudaError_t ap_launch(const CUtensorMap& m, const DevPtrs& d, int nrows, int layer, int chunk, int grid,
                             cudaStream_t st) {
  static bool configured = false;
  const size_t smem = ap_smem_bytes<HD, G>();
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_pdl(attn_prefill_kernel<HD, G>, dim3(grid), dim3(kAmThreads), smem, st, m, d, nrows, layer, chunk);
}

template <int HD>
static cudaError_t ap_hd(const CUtensorMap& m, const DevPtrs& d, int nrows, int layer, int chunk, int grid,
                         cudaStream_t st) {
  switch (d.Hq / d.Hkv) {
    case 1: return ap_launch<HD, 1>(m, d, nrows, layer, chunk, grid, st);
    case 2: return ap_launch<HD, 2>(m, d, nrows, layer, chunk, grid, st);
    case 4: return ap_launch<HD, 4>(m, d, nrows, layer, chunk, grid, st);
    case 8: return ap_launch<HD, 8>(m, d, nrows, layer, chunk, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_prefill(const DevPtrs& d, int nrows, int layer, int total_units, int chunk_tokens, int n_sm,
                                cudaStream_t st, bool* used) {
  *used = false;
  if (nrows < 2 || total_units <= 0 || !tc_available()) return cudaSuccess;
  if ((d.hd != 64 && d.hd != 128) || d.page_tokens != kPageTokens || chunk_tokens % kPageTokens != 0 ||
      chunk_tokens / kPageTokens > kMaxChunkPages || nrows > kMaxRows)
    return cudaSuccess;
  const long long rows = static_cast<long long>(d.max_pages) * d.n_layer * 2 * d.Hkv * kPageTokens;
  if (rows >= (1LL << 31)) return cudaSuccess;
  CUtensorMap m;
  if (!tc_bf16_map(&m, d.kv_pool, d.hd, static_cast<int>(rows), d.hd, 64)) return cudaSuccess;
  // chunks as long as a block of rows makes the units fewer: the split that
  // suits one row per unit, times the rows of a block (at most kMaxChunkPages)
  const int qb = 32 / (d.Hq / d.Hkv);
  int cp = chunk_tokens / kPageTokens * qb;
  cp = cp > kMaxChunkPages ? kMaxChunkPages : cp;
  chunk_tokens = cp * kPageTokens;
  const int grid = total_units < n_sm ? total_units : n_sm;
  cudaError_t e = d.hd == 128 ? ap_hd<128>(m, d, nrows, layer, chunk_tokens, grid, st)
                              : ap_hd<64>(m, d, nrows, layer, chunk_tokens, grid, st);
  if (e == cudaSuccess) *used = true;
  return e;
}

template <int HD, int G>
static cudaError_t am_launch(const CUtensorMap& m, const DevPtrs& d, int nrows, int layer, int units, int chunk,
                             int grid, int fuse, const uint16_t* qn, const uint16_t* kn, cudaStream_t st,
                             AttnHalves hv) {
  static bool configured = false;
  const size_t smem = am_smem_bytes<HD, G>();
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_mma_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_pdl(attn_mma_kernel<HD, G>, dim3(grid), dim3(kAmThreads), smem, st, m, d, nrows, layer, units, chunk,
                    fuse, qn, kn, hv);
}

template <int HD>
static cudaError_t am_hd(const CUtensorMap& m, const DevPtrs& d, int nrows, int layer, int units, int chunk, int grid,
                         int fuse, const uint16_t* qn, const uint16_t* kn, cudaStream_t st, AttnHalves hv) {
  switch (d.Hq / d.Hkv) {
    case 1: return am_launch<HD, 1>(m, d, nrows, layer, units, chunk, grid, fuse, qn, kn, st, hv);
    case 2: return am_launch<HD, 2>(m, d, nrows, layer, units, chunk, grid, fuse, qn, kn, st, hv);
    case 4: return am_launch<HD, 4>(m, d, nrows, layer, units, chunk, grid, fuse, qn, kn, st, hv);
    case 8: return am_launch<HD, 8>(m, d, nrows, layer, units, chunk, grid, fuse, qn, kn, st, hv);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_mma(const DevPtrs& d, int nrows, int layer, int total_units, int chunk_tokens, int n_sm,
                            bool fuse_append, const uint16_t* q_norm, const uint16_t* k_norm, cudaStream_t st,
                            bool* used, AttnHalves hv) {
  *used = false;
  if (nrows < kAttnMmaMinRows || total_units <= 0 || !tc_available()) return cudaSuccess;
  if ((d.hd != 64 && d.hd != 128) || d.page_tokens != kPageTokens || chunk_tokens % kPageTokens != 0 ||
      chunk_tokens / kPageTokens > kMaxChunkPages || nrows > kMaxRows)
    return cudaSuccess;
  const long long rows = static_cast<long long>(d.max_pages) * d.n_layer * 2 * d.Hkv * kPageTokens;
  if (rows >= (1LL << 31)) return cudaSuccess;
  CUtensorMap m;
  if (!tc_bf16_map(&m, d.kv_pool, d.hd, static_cast<int>(rows), d.hd, 64)) return cudaSuccess;
  const int grid = total_units < n_sm ? total_units : n_sm;
  const int f = fuse_append ? 1 : 0;
  cudaError_t e = d.hd == 128 ? am_hd<128>(m, d, nrows, layer, total_units, chunk_tokens, grid, f, q_norm, k_norm, st, hv)
                              : am_hd<64>(m, d, nrows, layer, total_units, chunk_tokens, grid, f, q_norm, k_norm, st, hv);
  if (e == cudaSuccess) *used = true;
  return e;
}

}  // namespace dualar
