// Split-KV GQA attention over the paged cache on the tensor cores, for
// launches of 3 or more rows (decode batches, prefill chunks).
//
// Same work units as attn_paged_units (row, KV head, chunk of pages), the
// same partial-sum format and the same deterministic last-arriver combine.
// Inside a unit the G query heads of the KV head are the rows of warp-level
// MMAs (mma.sync m16n8k16, bf16 operands, fp32 accumulators; G <= 8 of the 16
// rows are real -- tcgen05's M >= 64 would waste far more):
//   S = Q K^T  (Q: the unit's query heads, 1/sqrt(hd) folded in, as bf16
//               hi + lo halves; K: a 64-token page),
//   online softmax over the page on the fragment rows,
//   O += P V   (P as bf16 hi + lo halves built from the S fragments).
// Pages arrive by TMA (128-byte swizzle, so ldmatrix reads are conflict-free)
// from a producer warp that walks the CTA's pages across units.  Page number
// n (counted over the CTA's whole launch) belongs to compute warp n % 4, which
// owns a small ring of slots (each the K or the V block of a page) and takes
// them in order: every slot has a single consumer, so an mbarrier wait is
// never more than one phase ahead of its barrier (a parity wait cannot tell
// phases two apart).  The warps merge their (m, l, O) in warp order.  Decode (fuse): the
// unit holding the newest position computes its K/V (QK-norm, RoPE), writes
// them to the cache and patches the page's row in shared memory, since the
// page copy may predate the write.
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
constexpr int kAmThreads = (kAmWarps + 1) * 32;    // + the producer warp
constexpr int kAmBox = 64 * 64 * 2;                // one TMA box: 64 tokens x 64 dims (bf16)

template <int HD>
struct AmCfg {
  static constexpr int HALVES = HD / 64;                  // boxes per 64-token K (or V) block
  static constexpr int SLOT = HALVES * kAmBox;            // a slot: the K or the V block of one page
  static constexpr int SLOTS = HD == 128 ? 3 : 4;         // slots of each compute warp
  static constexpr int NBUF = kAmWarps * SLOTS;
};

template <int HD, int G>
struct AmSmem {
  // after the ring (offsets in floats / elements from the end of the ring)
  float qs[G][HD];
  float cm[kAmWarps][8], cl[kAmWarps][8];
  float co[kAmWarps][G][HD];
  float knew[HD], vnew[HD];
  RowInfo rows[kMaxRows];   // the launch's rows (read once)
  uint64_t full[AmCfg<HD>::NBUF], empty[AmCfg<HD>::NBUF];
  int abort_flag, s_last, unit_ok;
};

template <int HD, int G>
constexpr size_t am_smem_bytes() {
  return static_cast<size_t>(AmCfg<HD>::NBUF) * AmCfg<HD>::SLOT + sizeof(AmSmem<HD, G>) + 1024;
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
// C += A B: A 16x16 (rows g, g+8 of the fragment layout), B 16x8, fp32 C.
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

// Unit u's row and chunk (from the launch's rows in shared memory); false for
// an inactive row.
DEVI bool am_unit(const DevPtrs& d, const RowInfo* rows, int nrows, int u, int chunk_tokens, AmUnit& un) {
  int lo = 0, hi = nrows - 1;   // rows are sorted by unit0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (rows[mid].unit0 <= u) lo = mid;
    else hi = mid - 1;
  }
  un.r = lo;
  un.ri = rows[lo];
  const int L = un.ri.pos + 1;
  un.nch = (L + chunk_tokens - 1) / chunk_tokens;
  const int local = u - un.ri.unit0;
  un.g = local / un.nch;
  un.c = local % un.nch;
  if (!un.ri.active || un.g >= d.Hkv) return false;
  un.t0 = un.c * chunk_tokens;
  un.t1 = min(L, un.t0 + chunk_tokens);
  un.npages = (un.t1 - un.t0 + kPageTokens - 1) / kPageTokens;
  un.ptab = d.page_table + static_cast<size_t>(un.ri.slot) * d.pages_per_seq + un.t0 / kPageTokens;
  return true;
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

template <int HD, int G>
__global__ void __launch_bounds__(kAmThreads, 1)
    attn_mma_kernel(const __grid_constant__ CUtensorMap tkv, const DevPtrs d, int nrows, int layer, int total_units,
                    int chunk_tokens, int fuse, const uint16_t* q_norm, const uint16_t* k_norm) {
  using C = AmCfg<HD>;
  constexpr int NB = C::NBUF;
  constexpr int EPL = HD / 32;
  static_assert(G >= 1 && G <= 8, "query heads per KV head: the MMA rows 0..7");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  AmSmem<HD, G>& sm = *reinterpret_cast<AmSmem<HD, G>*>(ring + NB * C::SLOT);
  const uint32_t ring_s = smem_addr(ring);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hkv = d.Hkv, hq = d.Hq;
  const size_t page_stride = static_cast<size_t>(kPageTokens) * HD;
  if (tid == 0) {
    for (int b = 0; b < NB; ++b) {
      mbar_init(&sm.full[b], 1);
      mbar_init(&sm.empty[b], 1);
    }
    sm.abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = tid; i < nrows; i += kAmThreads) sm.rows[i] = ld_row(&d.rows[i]);
  __syncthreads();
  const volatile int* abort_flag = &sm.abort_flag;

  if (warp == kAmWarps) {
    // ---- producer (the whole warp; lane 0 issues): the K/V pages of this
    // CTA's units, in order
    uint32_t gs = 0;
    uint32_t cnt[kAmWarps];   // slot fills given to each compute warp so far
    uint32_t iss[kAmWarps];   // ... and actually issued (lane 0)
#pragma unroll
    for (int w = 0; w < kAmWarps; ++w) cnt[w] = iss[w] = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      AmUnit un;
      if (!am_unit(d, sm.rows, nrows, u, chunk_tokens, un)) continue;
      int pg[kAmPageRegs];
      if (!am_pages(d, un, lane, pg)) continue;
      for (int p = 0; p < un.npages; ++p) {
        int pgp = 0;
#pragma unroll
        for (int i = 0; i < kAmPageRegs; ++i) {
          const int v = __shfl_sync(0xFFFFFFFFu, pg[i], p & 31);
          if ((p >> 5) == i) pgp = v;
        }
        const int w = static_cast<int>(gs % kAmWarps);
        const int rowk = static_cast<int>(((static_cast<long long>(pgp) * d.n_layer + layer) * 2 * hkv + un.g) * 64);
#pragma unroll
        for (int kv = 0; kv < 2; ++kv) {
          uint32_t j = 0;
#pragma unroll
          for (int ww = 0; ww < kAmWarps; ++ww)
            if (ww == w) j = cnt[ww]++;
          const int s = w * C::SLOTS + static_cast<int>(j % C::SLOTS);
          if (lane == 0 && ok) {
            if (j >= static_cast<uint32_t>(C::SLOTS) &&
                !am_wait(&sm.empty[s], ((j / C::SLOTS) - 1) & 1, abort_flag, d)) {
              sm.abort_flag = 1;
              ok = false;
            } else {
              mbar_arrive_expect_tx(&sm.full[s], static_cast<uint32_t>(C::SLOT));
#pragma unroll
              for (int hh = 0; hh < C::HALVES; ++hh)
                tma_load_2d(ring + s * C::SLOT + hh * kAmBox, &tkv, hh * 64, rowk + kv * hkv * 64, &sm.full[s]);
#pragma unroll
              for (int ww = 0; ww < kAmWarps; ++ww)
                if (ww == w) ++iss[ww];
            }
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok) break;
        ++gs;
      }
    }
    if (lane == 0) {
      // every copy issued here lands before the CTA exits (bounded)
      for (int w = 0; w < kAmWarps; ++w)
        for (uint32_t j = iss[w] > static_cast<uint32_t>(C::SLOTS) ? iss[w] - C::SLOTS : 0; j < iss[w]; ++j) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try_wait(&sm.full[w * C::SLOTS + j % C::SLOTS], (j / C::SLOTS) & 1))
            if (global_timer_ns() - t0 > d.wait_limit_ns) break;
        }
    }
    return;
  }

  // ---- compute warps
  const float qscale = 1.0f / sqrtf(static_cast<float>(HD));
  const int gr = lane >> 2, tq = lane & 3;   // fragment row (head) and column pair
  uint32_t gs_base = 0;
  uint32_t mine = 0;   // pages this warp has taken so far (its slot sequence)
  for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
    AmUnit un;
    if (!am_unit(d, sm.rows, nrows, u, chunk_tokens, un)) continue;
    if (warp == 0) {
      int pg[kAmPageRegs];
      const bool pages_ok = am_pages(d, un, lane, pg);
      if (lane == 0) {
        sm.unit_ok = pages_ok ? 1 : 0;
        if (!pages_ok) raise_error(d.err, DEV_ERR_BAD_PAGE);
      }
    }
    const int r = un.r;
    const bool newest = fuse && un.c == un.nch - 1;
    // query heads of this unit (and the newest position's K/V)
    for (int h = warp; h < G; h += kAmWarps) {
      float v[EPL];
      if (fuse) {
        const float* src = d.qkv + static_cast<size_t>(r) * d.qkv_dim + (un.g * G + h) * HD;
#pragma unroll
        for (int j = 0; j < EPL; ++j) v[j] = ldf(src + lane * EPL + j);
        head_norm_rope<EPL>(v, q_norm, d.eps, un.ri.pos, d, lane);
      } else {
        const float* src = d.qrot + (static_cast<size_t>(r) * hq + un.g * G + h) * HD;
#pragma unroll
        for (int j = 0; j < EPL; ++j) v[j] = ldf(src + lane * EPL + j);
      }
#pragma unroll
      for (int j = 0; j < EPL; ++j) sm.qs[h][lane * EPL + j] = v[j] * qscale;
    }
    if (newest && warp == kAmWarps - 1) {
      const float* base = d.qkv + static_cast<size_t>(r) * d.qkv_dim;
      float kv[EPL], vv[EPL];
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        kv[j] = ldf(base + hq * HD + un.g * HD + lane * EPL + j);
        vv[j] = ldf(base + hq * HD + hkv * HD + un.g * HD + lane * EPL + j);
      }
      head_norm_rope<EPL>(kv, k_norm, d.eps, un.ri.pos, d, lane);
      const int pg = ldi(d.page_table + static_cast<size_t>(un.ri.slot) * d.pages_per_seq + un.ri.pos / kPageTokens);
      uint16_t* kd = d.kv_pool + (((static_cast<size_t>(pg) * d.n_layer + layer) * 2 + 0) * hkv + un.g) * page_stride +
                     static_cast<size_t>(un.ri.pos % kPageTokens) * HD;
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
    named_barrier(1, kAmWarps * 32);
    if (!sm.unit_ok) {
      named_barrier(1, kAmWarps * 32);   // (the producer skipped it too)
      continue;
    }
    // Q fragments (rows gr < G real; rows gr + 8 are zero)
    uint32_t qh[HD / 16][2], ql[HD / 16][2];
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int dd = ks * 16 + half * 8 + 2 * tq;
        const float x = gr < G ? sm.qs[gr][dd] : 0.f, y = gr < G ? sm.qs[gr][dd + 1] : 0.f;
        split2(x, y, qh[ks][half], ql[ks][half]);
      }
    }
    float m_run = -INFINITY, l_run = 0.f;
    float o[HD / 8][4];
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

    const int p0 = static_cast<int>((warp - static_cast<int>(gs_base % kAmWarps) + kAmWarps) % kAmWarps);
    for (int p = p0; p < un.npages; p += kAmWarps) {
      const uint32_t jk = mine++, jv = mine++;
      const int sk = warp * C::SLOTS + static_cast<int>(jk % C::SLOTS);
      const int sv = warp * C::SLOTS + static_cast<int>(jv % C::SLOTS);
      bool got = am_wait(&sm.full[sk], (jk / C::SLOTS) & 1, abort_flag, d);
      got = am_wait(&sm.full[sv], (jv / C::SLOTS) & 1, abort_flag, d) && got;
      if (!got) sm.abort_flag = 1;   // the others stop waiting too
      const int ps = un.t0 + p * kPageTokens;
      const int ntok = min(kPageTokens, un.t1 - ps);
      const uint32_t kb = ring_s + sk * C::SLOT, vb = ring_s + sv * C::SLOT;
      if (got && newest && ps <= un.ri.pos && un.ri.pos < ps + kPageTokens) {
        // the newest row (its copy may predate the cache write)
        const int rr = un.ri.pos - ps;
        if (lane < HD / 8) {
          uint32_t wk[4], wv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            wk[e] = static_cast<uint32_t>(f32_to_bf16bits(sm.knew[lane * 8 + 2 * e])) |
                    (static_cast<uint32_t>(f32_to_bf16bits(sm.knew[lane * 8 + 2 * e + 1])) << 16);
            wv[e] = static_cast<uint32_t>(f32_to_bf16bits(sm.vnew[lane * 8 + 2 * e])) |
                    (static_cast<uint32_t>(f32_to_bf16bits(sm.vnew[lane * 8 + 2 * e + 1])) << 16);
          }
          const uint32_t ak = sw_addr(kb, rr, lane * 8), av = sw_addr(vb, rr, lane * 8);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(ak), "r"(wk[0]), "r"(wk[1]), "r"(wk[2]),
                       "r"(wk[3])
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(av), "r"(wv[0]), "r"(wv[1]), "r"(wv[2]),
                       "r"(wv[3])
                       : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      if (got) {
        // S = Q K^T over the page: 8 tiles of 8 tokens
        float sc[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
          for (int jp = 0; jp < 4; ++jp) {
            uint32_t b[4];
            const int tok = jp * 16 + (lane >> 4) * 8 + (lane & 7);
            const int dim = ks * 16 + ((lane >> 3) & 1) * 8;
            ldsm_x4(b, sw_addr(kb, tok, dim));
            mma16816(sc[2 * jp], qh[ks][0], 0u, qh[ks][1], 0u, b[0], b[1]);
            mma16816(sc[2 * jp], ql[ks][0], 0u, ql[ks][1], 0u, b[0], b[1]);
            mma16816(sc[2 * jp + 1], qh[ks][0], 0u, qh[ks][1], 0u, b[2], b[3]);
            mma16816(sc[2 * jp + 1], ql[ks][0], 0u, ql[ks][1], 0u, b[2], b[3]);
          }
        }
        // online softmax on row gr (tokens 8j + 2tq, +1)
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int t = 8 * j + 2 * tq;
          if (t >= ntok) sc[j][0] = -INFINITY;
          if (t + 1 >= ntok) sc[j][1] = -INFINITY;
          mx = fmaxf(mx, fmaxf(sc[j][0], sc[j][1]));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float f = expf(m_run - m_new);   // 0 on the first page (m_run = -inf)
        float ps_sum = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
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
        }
        // O += P V: 4 steps of 16 tokens
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
          uint32_t ph0, pl0, ph2, pl2;
          split2(sc[2 * kt][0], sc[2 * kt][1], ph0, pl0);
          split2(sc[2 * kt + 1][0], sc[2 * kt + 1][1], ph2, pl2);
#pragma unroll
          for (int np = 0; np < HD / 16; ++np) {
            uint32_t b[4];
            const int tok = kt * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
            const int dim = np * 16 + (lane >> 4) * 8;
            ldsm_x4_t(b, sw_addr(vb, tok, dim));
            mma16816(o[2 * np], ph0, 0u, ph2, 0u, b[0], b[1]);
            mma16816(o[2 * np], pl0, 0u, pl2, 0u, b[0], b[1]);
            mma16816(o[2 * np + 1], ph0, 0u, ph2, 0u, b[2], b[3]);
            mma16816(o[2 * np + 1], pl0, 0u, pl2, 0u, b[2], b[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) {   // both slots are free (reads done: their values were used above)
        mbar_arrive(&sm.empty[sk]);
        mbar_arrive(&sm.empty[sv]);
      }
    }
    gs_base += un.npages;

    // merge the warps' (m, l, O) (warp order: deterministic)
    if (gr < G) {
      if (tq == 0) {
        sm.cm[warp][gr] = m_run;
        sm.cl[warp][gr] = l_run;
      }
#pragma unroll
      for (int n = 0; n < HD / 8; ++n) {
        sm.co[warp][gr][8 * n + 2 * tq] = o[n][0];
        sm.co[warp][gr][8 * n + 2 * tq + 1] = o[n][1];
      }
    }
    named_barrier(1, kAmWarps * 32);
    const size_t attn_off = static_cast<size_t>(r) * hq * HD + un.g * G * HD;
    float* pw = d.part + ((static_cast<size_t>(r) * hkv + un.g) * kMaxChunks + un.c) * G * (HD + 2);
    for (int e = tid; e < G * HD; e += kAmWarps * 32) {
      const int h = e / HD, dd = e % HD;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kAmWarps; ++w) M = fmaxf(M, sm.cm[w][h]);
      float Ls = 0.f, Os = 0.f;
#pragma unroll
      for (int w = 0; w < kAmWarps; ++w) {
        const float fw = sm.cm[w][h] == -INFINITY ? 0.f : expf(sm.cm[w][h] - M);
        Ls += sm.cl[w][h] * fw;
        Os += sm.co[w][h][dd] * fw;
      }
      if (un.nch == 1) {
        d.attn[attn_off + h * HD + dd] = Os / Ls;
      } else {
        pw[h * (HD + 2) + dd] = Os;
        if (dd == 0) {
          pw[h * (HD + 2) + HD] = M;
          pw[h * (HD + 2) + HD + 1] = Ls;
        }
      }
    }
    if (un.nch > 1) {
      __threadfence();
      named_barrier(1, kAmWarps * 32);
      if (tid == 0) {
        const uint32_t old = atomic_add_acq_rel_gpu(&d.arrive[r * hkv + un.g], 1u);
        int last = 0;
        if (old == static_cast<uint32_t>(un.nch - 1)) {
          const uint32_t prev = atomicExch(&d.arrive[r * hkv + un.g], 0u);
          last = prev == 0xFFFFFFFFu ? 2 : 1;
        }
        sm.s_last = last;
      }
      named_barrier(1, kAmWarps * 32);
      if (sm.s_last) {
        __threadfence();
        const float* pb = d.part + (static_cast<size_t>(r) * hkv + un.g) * kMaxChunks * G * (HD + 2);
        for (int e = tid; e < G * HD; e += kAmWarps * 32) {
          const int h = e / HD, dd = e % HD;
          float M = -INFINITY;
          for (int cc = 0; cc < un.nch; ++cc) M = fmaxf(M, ldf(pb + (cc * G + h) * (HD + 2) + HD));
          float Ls = 0.f, Os = 0.f;
          for (int cc = 0; cc < un.nch; ++cc) {
            const float* q = pb + (cc * G + h) * (HD + 2);
            const float fc = expf(ldf(q + HD) - M);
            Ls += ldf(q + HD + 1) * fc;
            Os += ldf(q + dd) * fc;
          }
          d.attn[attn_off + h * HD + dd] = Os / Ls;
        }
      }
    }
    named_barrier(1, kAmWarps * 32);   // shared buffers are reused by the next unit
  }
}

template <int HD, int G>
static cudaError_t am_launch(const CUtensorMap& m, const DevPtrs& d, int nrows, int layer, int units, int chunk,
                             int grid, int fuse, const uint16_t* qn, const uint16_t* kn, cudaStream_t st) {
  static bool configured = false;
  const size_t smem = am_smem_bytes<HD, G>();
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_mma_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  attn_mma_kernel<HD, G><<<grid, kAmThreads, smem, st>>>(m, d, nrows, layer, units, chunk, fuse, qn, kn);
  return cudaGetLastError();
}

template <int HD>
static cudaError_t am_hd(const CUtensorMap& m, const DevPtrs& d, int nrows, int layer, int units, int chunk, int grid,
                         int fuse, const uint16_t* qn, const uint16_t* kn, cudaStream_t st) {
  switch (d.Hq / d.Hkv) {
    case 1: return am_launch<HD, 1>(m, d, nrows, layer, units, chunk, grid, fuse, qn, kn, st);
    case 2: return am_launch<HD, 2>(m, d, nrows, layer, units, chunk, grid, fuse, qn, kn, st);
    case 4: return am_launch<HD, 4>(m, d, nrows, layer, units, chunk, grid, fuse, qn, kn, st);
    case 8: return am_launch<HD, 8>(m, d, nrows, layer, units, chunk, grid, fuse, qn, kn, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_mma(const DevPtrs& d, int nrows, int layer, int total_units, int chunk_tokens, int n_sm,
                            bool fuse_append, const uint16_t* q_norm, const uint16_t* k_norm, cudaStream_t st,
                            bool* used) {
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
  cudaError_t e = d.hd == 128 ? am_hd<128>(m, d, nrows, layer, total_units, chunk_tokens, grid, f, q_norm, k_norm, st)
                              : am_hd<64>(m, d, nrows, layer, total_units, chunk_tokens, grid, f, q_norm, k_norm, st);
  if (e == cudaSuccess) *used = true;
  return e;
}

}  // namespace dualar
