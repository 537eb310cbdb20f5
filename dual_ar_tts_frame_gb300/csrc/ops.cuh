// Device-side ops of the Dual-AR frame other than the GEMV: QK-norm/RoPE,
// paged split-KV attention (slow AR), attention over the per-frame codebook
// cache (fast AR), the sampler, and the multi-codebook fusion.
//
// Every op is a device function over NT participating threads that
// synchronise with named barrier 2 (never __syncthreads), so the same code
// runs as a standalone kernel (NT = blockDim) and inside the persistent frame
// kernel (NT = the consumer warps, while a producer warp streams weights).
// Activations are read through L2 (ld.global.cg): inside the persistent
// kernel they are rewritten by other CTAs between ops and L1 is not coherent.
//
// Pages cited (title, section):
//   [P1] "How the Dual-Autoregressive Architecture Works in Fish Speech S2: A Deep Dive"
//   [P2] "Fish Audio S2: a Qwen3-4B on the time axis, four layers on the codebook
//        axis, and tags that are only text"
#pragma once

#include <cfloat>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace dualar {

template <int NT>
DEVI void csync() {
  named_barrier(2, NT);
}

DEVI float ldf(const float* p) { return __ldcg(p); }
DEVI int ldi(const int32_t* p) { return __ldcg(p); }
DEVI RowInfo ld_row(const RowInfo* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  return RowInfo{v.x, v.y, v.z, v.w};
}

// Tags of an op's activation input and output inside the persistent frame
// kernel (common.cuh, "tagged activations"); 0 selects the plain fp32
// buffers (standalone kernels).
struct OpTags {
  uint32_t in, out;
};

// EPL consecutive activation values at element offset off.
template <int EPL>
DEVI void act_load(const float* plain, const uint64_t* tagged, size_t off, uint32_t tag, float (&v)[EPL],
                   const DevPtrs& d) {
  if (tag != 0u) {
    tag_wait<EPL>(tagged + off, tag, v, d.err, d.wait_limit_ns);
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j) v[j] = ldf(plain + off + j);
  }
}
// The bf16 halves (hi, lo = bf16(v - hi)) of EPL attention-output values at
// row r, column col, for the o projection (per-op path).
template <int EPL>
DEVI void attn_halves(const AttnHalves& hv, int r, int col, const float (&v)[EPL]) {
  uint16_t h[EPL], l[EPL];
#pragma unroll
  for (int j = 0; j < EPL; ++j) {
    h[j] = f32_to_bf16bits(v[j]);
    l[j] = f32_to_bf16bits(v[j] - bf16bits_to_f32(h[j]));
  }
  const size_t o = static_cast<size_t>(r) * hv.ld + col;
  if constexpr (EPL % 2 == 0) {
    // pairs in 32-bit words (col and ld even)
#pragma unroll
    for (int j = 0; j < EPL; j += 2) {
      *reinterpret_cast<uint32_t*>(hv.xh + o + j) = static_cast<uint32_t>(h[j]) | (static_cast<uint32_t>(h[j + 1]) << 16);
      *reinterpret_cast<uint32_t*>(hv.xl + o + j) = static_cast<uint32_t>(l[j]) | (static_cast<uint32_t>(l[j + 1]) << 16);
    }
  } else {
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      hv.xh[o + j] = h[j];
      hv.xl[o + j] = l[j];
    }
  }
}

DEVI void act_store(float* plain, uint64_t* tagged, size_t off, uint32_t tag, float v) {
  if (tag != 0u) tag_store(tagged + off, v, tag);
  else plain[off] = v;
}

// QK-norm (optional) + RoPE of one head vector held as EPL elements per lane.
// [P2] "The slow AR is Qwen3-4B": qk-norm (slow AR only), rope_base 1e6;
// "Streaming: whose numbers": bf16 tables.  Pairs (2i, 2i+1) rotate by
// pos * base^(-2i/hd).  The gain and the table entries do not depend on the
// activation, so callers load them (head_nr_load) before waiting for it.
template <int EPL>
struct HeadNR {
  float w[EPL];                 // norm gain of this lane's elements
  float c[EPL / 2], s[EPL / 2]; // cos, sin of this lane's pairs
};

template <int EPL>
DEVI HeadNR<EPL> head_nr_load(const uint16_t* nw, int pos, const DevPtrs& d, int lane) {
  constexpr int half = EPL * 16;
  HeadNR<EPL> t;
#pragma unroll
  for (int j = 0; j < EPL; ++j) t.w[j] = nw != nullptr ? bf16bits_to_f32(nw[lane * EPL + j]) : 1.f;
#pragma unroll
  for (int pp = 0; pp < EPL / 2; ++pp) {
    const int i = (lane * EPL) / 2 + pp;
    t.c[pp] = bf16bits_to_f32(d.rope_cos[static_cast<size_t>(pos) * half + i]);
    t.s[pp] = bf16bits_to_f32(d.rope_sin[static_cast<size_t>(pos) * half + i]);
  }
  return t;
}

template <int EPL>
DEVI void head_nr_apply(float (&v)[EPL], const HeadNR<EPL>& t, bool norm, float eps) {
  constexpr int hd = EPL * 32;
  if (norm) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < EPL; ++j) s += v[j] * v[j];
    s = warp_sum(s);
    const float inv = 1.0f / sqrtf(s / static_cast<float>(hd) + eps);
#pragma unroll
    for (int j = 0; j < EPL; ++j) v[j] = (v[j] * inv) * t.w[j];
  }
#pragma unroll
  for (int pp = 0; pp < EPL / 2; ++pp) {
    const float x0 = v[2 * pp], x1 = v[2 * pp + 1];
    v[2 * pp] = x0 * t.c[pp] - x1 * t.s[pp];
    v[2 * pp + 1] = x1 * t.c[pp] + x0 * t.s[pp];
  }
}

// ============================================================================
// Paged split-KV decode attention (slow AR)
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
constexpr int kPageTokens = 64;

template <int HD, int G, int NT>
struct AttnSmall {
  static constexpr int TPT = NT / kPageTokens;   // threads per token (score pass)
  static constexpr int QD = HD / TPT;            // dims per thread (score pass)
  static constexpr int PARTS = NT / HD;          // token groups (value pass)
  float qs[G][TPT][QD + 4];   // rows 16-byte aligned, 80 B apart: conflict-free float4 reads
  float sc[G][kPageTokens];
  float ored[PARTS][G][HD];
  float knew[HD], vnew[HD];
  float scl[G], msm[G], lsm[G];
  float cm[kMaxChunks][G], cl[kMaxChunks][G];   // tagged combine: (m, l) of every chunk
  int s_last;
};

template <int HD, int G, int NT, int NBUF = 2>
struct AttnSmem : AttnSmall<HD, G, NT> {
  static constexpr int BUFS = NBUF;              // page buffers (a ring of NBUF pages in flight)
  static constexpr size_t kSmall = sizeof(AttnSmall<HD, G, NT>);
  static constexpr size_t kKvAt = ((kSmall + 1 + 127) / 128) * 128;   // page buffers 128-byte aligned
  unsigned char pad_[kKvAt - kSmall];
  uint16_t kv[NBUF][2][kPageTokens * HD];        // [buffer][K/V][tok][dim]
};

template <int HD, int G, int NT, int NBUF>
DEVI void attn_paged_units(const DevPtrs& d, int nrows, int layer, int total_units, int chunk_tokens,
                           bool fuse_append, const uint16_t* q_norm, const uint16_t* k_norm,
                           AttnSmem<HD, G, NT, NBUF>& sm, uint64_t* bars, uint32_t* phase, int cta,
                           int ncta, OpTags tg = OpTags{0u, 0u}) {
  using S = AttnSmem<HD, G, NT, NBUF>;
  constexpr int EPL = HD / 32;
  constexpr int TPT = S::TPT, QD = S::QD, PARTS = S::PARTS;
  constexpr int TPP = kPageTokens / PARTS;
  constexpr int NW = NT / 32;
  constexpr uint32_t kPageBytes = kPageTokens * HD * 2;
  static_assert(QD % 8 == 0, "score pass reads 16-byte vectors");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hq = d.Hq, hkv = d.Hkv;
  const float qscale = 1.0f / sqrtf(static_cast<float>(HD));
  const size_t page_stride = static_cast<size_t>(kPageTokens) * HD;

  for (int u = cta; u < total_units; u += ncta) {
    int lo = 0, hi = nrows - 1;   // rows are sorted by unit0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (ldi(&d.rows[mid].unit0) <= u) lo = mid;
      else hi = mid - 1;
    }
    const int r = lo;
    const RowInfo ri = ld_row(&d.rows[r]);
    const int L = ri.pos + 1;
    const int nch = (L + chunk_tokens - 1) / chunk_tokens;
    const int local = u - ri.unit0;
    const int g = local / nch, c = local % nch;
    if (!ri.active || g >= hkv) {
      // tagged output: the readers wait for every row, so an inactive row
      // still writes (zeros) once per KV head
      if (tg.out != 0u && c == 0 && g < hkv)
        for (int e = tid; e < G * HD; e += NT)
          tag_store(d.attn_t + static_cast<size_t>(r) * hq * HD + g * G * HD + e, 0.f, tg.out);
      continue;
    }
    const int t0 = c * chunk_tokens;
    const int t1 = min(L, t0 + chunk_tokens);
    const int npages = (t1 - t0 + kPageTokens - 1) / kPageTokens;
    const bool newest = fuse_append && (c == nch - 1);
    const int32_t* ptab = d.page_table + static_cast<size_t>(ri.slot) * d.pages_per_seq + t0 / kPageTokens;
    bool ok = true;
    for (int p = 0; p < npages; ++p) {
      const int pg = ldi(ptab + p);
      if (pg < 0 || pg >= d.max_pages) ok = false;
    }
    if (!ok) {
      if (tid == 0) raise_error(d.err, DEV_ERR_BAD_PAGE);
      continue;
    }
    auto issue = [&](int p, int buf) {
      const uint16_t* kp = d.kv_pool +
          (((static_cast<size_t>(ldi(ptab + p)) * d.n_layer + layer) * 2 + 0) * hkv + g) * page_stride;
      const uint16_t* vp = kp + static_cast<size_t>(hkv) * page_stride;
      mbar_arrive_expect_tx(&bars[buf], 2 * kPageBytes);
      bulk_load_g2s_plain(sm.kv[buf][0], kp, kPageBytes, &bars[buf]);
      bulk_load_g2s_plain(sm.kv[buf][1], vp, kPageBytes, &bars[buf]);
    };
    if (tid == 0) {
      for (int p = 0; p < NBUF && p < npages; ++p) issue(p, p);
    }

    if (fuse_append) {
      if (warp < G) {
        const int h = g * G + warp;
        const HeadNR<EPL> nr = head_nr_load<EPL>(q_norm, ri.pos, d, lane);
        float v[EPL];
        act_load<EPL>(d.qkv, d.qkv_t, static_cast<size_t>(r) * d.qkv_dim + h * HD + lane * EPL, tg.in, v, d);
        head_nr_apply<EPL>(v, nr, q_norm != nullptr, d.eps);
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
          const int dd = lane * EPL + j;
          sm.qs[warp][dd / QD][dd % QD] = v[j] * qscale;
        }
      }
      if (warp == (G % NW) && newest) {
        const size_t base = static_cast<size_t>(r) * d.qkv_dim;
        const HeadNR<EPL> nr = head_nr_load<EPL>(k_norm, ri.pos, d, lane);
        const int pg = ldi(d.page_table + static_cast<size_t>(ri.slot) * d.pages_per_seq + ri.pos / kPageTokens);
        float kv[EPL], vv[EPL];
        act_load<EPL>(d.qkv, d.qkv_t, base + hq * HD + g * HD + lane * EPL, tg.in, kv, d);
        act_load<EPL>(d.qkv, d.qkv_t, base + hq * HD + hkv * HD + g * HD + lane * EPL, tg.in, vv, d);
        head_nr_apply<EPL>(kv, nr, k_norm != nullptr, d.eps);
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
      for (int e = tid; e < G * HD; e += NT) {
        const int h = e / HD, dd = e % HD;
        sm.qs[h][dd / QD][dd % QD] = ldf(d.qrot + (static_cast<size_t>(r) * hq + g * G + h) * HD + dd) * qscale;
      }
    }
    if (tid < G) {
      sm.msm[tid] = -INFINITY;
      sm.lsm[tid] = 0.f;
    }
    float o[G];
#pragma unroll
    for (int h = 0; h < G; ++h) o[h] = 0.f;
    csync<NT>();

    const int tok = tid / TPT, qd = tid % TPT;
    const int vdim = tid % HD, vpart = tid / HD;
    for (int p = 0; p < npages; ++p) {
      const int buf = p % NBUF;
      const int ps = t0 + p * kPageTokens;
      const int ntok = min(kPageTokens, t1 - ps);
      if (!mbar_wait(&bars[buf], phase[buf], d.err, d.wait_limit_ns)) return;
      phase[buf] ^= 1u;
      const uint16_t* ks = sm.kv[buf][0];
      const uint16_t* vs = sm.kv[buf][1];
      float s[G];
#pragma unroll
      for (int h = 0; h < G; ++h) s[h] = 0.f;
      if (tok < ntok) {
        if (newest && ps + tok == ri.pos) {
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
            for (int h = 0; h < G; ++h) {
              const float4* q4 = reinterpret_cast<const float4*>(&sm.qs[h][qd][v8 * 8]);
              const float4 qa = q4[0], qb = q4[1];
              const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) s[h] = fmaf(qv[jj], kf[jj], s[h]);
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int o2 = 1; o2 < TPT; o2 <<= 1) s[h] += __shfl_xor_sync(0xFFFFFFFFu, s[h], o2);
      if (qd == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) sm.sc[h][tok] = tok < ntok ? s[h] : -INFINITY;
      }
      csync<NT>();
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
      csync<NT>();
#pragma unroll
      for (int h = 0; h < G; ++h) o[h] *= sm.scl[h];
      const int tb = vpart * TPP, te = min(ntok, tb + TPP);
      if (te - tb == TPP && !(newest && ri.pos >= ps + tb && ri.pos < ps + te)) {
        // a full run of cached tokens: every V load in flight before the FMAs
        float vv[TPP];
#pragma unroll
        for (int k = 0; k < TPP; ++k) vv[k] = bf16bits_to_f32(vs[(tb + k) * HD + vdim]);
#pragma unroll
        for (int k = 0; k < TPP; ++k)
#pragma unroll
          for (int h = 0; h < G; ++h) o[h] = fmaf(sm.sc[h][tb + k], vv[k], o[h]);
      } else {
        for (int t = tb; t < te; ++t) {
          const float v = (newest && ps + t == ri.pos) ? sm.vnew[vdim] : bf16bits_to_f32(vs[t * HD + vdim]);
#pragma unroll
          for (int h = 0; h < G; ++h) o[h] = fmaf(sm.sc[h][t], v, o[h]);
        }
      }
      csync<NT>();   // buffer `buf` is free again
      if (tid == 0 && p + NBUF < npages) issue(p + NBUF, buf);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) sm.ored[vpart][h][vdim] = o[h];
    csync<NT>();
    const size_t attn_off = static_cast<size_t>(r) * hq * HD + g * G * HD;
    if (nch == 1) {
      for (int e = tid; e < G * HD; e += NT) {
        const int h = e / HD, dd = e % HD;
        float t = 0.f;
#pragma unroll
        for (int p = 0; p < PARTS; ++p) t += sm.ored[p][h][dd];
        act_store(d.attn, d.attn_t, attn_off + h * HD + dd, tg.out, t / sm.lsm[h]);
      }
      csync<NT>();
      continue;
    }
    if (tg.out != 0u) {
      // Tagged partials: the unit of the last chunk combines them.  It waits
      // only for units with smaller indices, and every CTA runs its units in
      // increasing order, so the waits always end.
      const size_t pbase = (static_cast<size_t>(r) * hkv + g) * kMaxChunks * G * (HD + 2);
      uint64_t* pt = d.part_t + pbase + static_cast<size_t>(c) * G * (HD + 2);
      for (int e = tid; e < G * HD; e += NT) {
        const int h = e / HD, dd = e % HD;
        float t = 0.f;
#pragma unroll
        for (int p = 0; p < PARTS; ++p) t += sm.ored[p][h][dd];
        tag_store(pt + h * (HD + 2) + dd, t, tg.out);
      }
      if (tid < G) {
        tag_store(pt + tid * (HD + 2) + HD, sm.msm[tid], tg.out);
        tag_store(pt + tid * (HD + 2) + HD + 1, sm.lsm[tid], tg.out);
      }
      csync<NT>();
      if (c != nch - 1) continue;
      const uint64_t* pb = d.part_t + pbase;
      for (int idx = tid; idx < nch * G; idx += NT) {
        const int cc = idx / G, h = idx % G;
        float ml[2];
        tag_wait<2>(pb + static_cast<size_t>(cc * G + h) * (HD + 2) + HD, tg.out, ml, d.err, d.wait_limit_ns);
        sm.cm[cc][h] = ml[0];
        sm.cl[cc][h] = ml[1];
      }
      csync<NT>();
      // same arithmetic and order as the last-arriver combine below
      for (int e = tid; e < G * HD; e += NT) {
        const int h = e / HD, dd = e % HD;
        float M = -INFINITY;
        for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, sm.cm[cc][h]);
        float Ls = 0.f, Os = 0.f;
        for (int c0 = 0; c0 < nch; c0 += 8) {
          uint64_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            w[k] = c0 + k < nch ? tag_load(pb + static_cast<size_t>((c0 + k) * G + h) * (HD + 2) + dd) : 0ull;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int cc = c0 + k;
            if (cc < nch) {
              const float o = tag_of(w[k]) == tg.out
                                  ? tag_val(w[k])
                                  : tag_wait1(pb + static_cast<size_t>(cc * G + h) * (HD + 2) + dd, tg.out, d.err,
                                              d.wait_limit_ns);
              const float f = expf(sm.cm[cc][h] - M);
              Ls += sm.cl[cc][h] * f;
              Os += o * f;
            }
          }
        }
        tag_store(d.attn_t + attn_off + h * HD + dd, Os / Ls, tg.out);
      }
      csync<NT>();
      continue;
    }
    float* pw = d.part + ((static_cast<size_t>(r) * hkv + g) * kMaxChunks + c) * G * (HD + 2);
    for (int e = tid; e < G * HD; e += NT) {
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
    csync<NT>();
    if (tid == 0) {
      const uint32_t old = atomic_add_acq_rel_gpu(&d.arrive[r * hkv + g], 1u);
      int last = 0;
      if (old == static_cast<uint32_t>(nch - 1)) {
        // the counter is reset before any output of this (row, head) is
        // written: whoever uses it next (the next layer) reads that output
        // first, directly or through later ops
        const uint32_t prev = atomicExch(&d.arrive[r * hkv + g], 0u);
        last = prev == 0xFFFFFFFFu ? 2 : 1;
      }
      sm.s_last = last;
    }
    csync<NT>();
    if (sm.s_last) {
      __threadfence();
      const float* pb = d.part + (static_cast<size_t>(r) * hkv + g) * kMaxChunks * G * (HD + 2);
      for (int e = tid; e < G * HD; e += NT) {
        const int h = e / HD, dd = e % HD;
        float M = -INFINITY;
        for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, ldf(pb + (cc * G + h) * (HD + 2) + HD));
        float Ls = 0.f, Os = 0.f;
        for (int cc = 0; cc < nch; ++cc) {
          const float* q = pb + (cc * G + h) * (HD + 2);
          const float f = expf(ldf(q + HD) - M);
          Ls += ldf(q + HD + 1) * f;
          Os += ldf(q + dd) * f;
        }
        act_store(d.attn, d.attn_t, attn_off + h * HD + dd, tg.out, Os / Ls);
      }
    }
    csync<NT>();
  }
}

// ============================================================================
// Fast-AR attention over the per-frame codebook cache (<= N positions)
// ============================================================================
// One unit per (row, KV head g): warp G computes the new position's K (norm
// if configured, RoPE at the codebook index) and V and appends them, while
// warp h < G loads query head g*G+h; the K/V of earlier positions (written by
// earlier passes of this frame to the global fast cache) are staged in shared
// memory first.  [P2] "Two
// autoregressions": the fast AR's KV cache is num_codebooks long and is
// overwritten every frame.
template <int HD>
struct FastAttnSmem {
  float ks[kMaxCodebooks][HD], vs[kMaxCodebooks][HD];
};

// HALVES (per-op path): also the bf16 halves of the output into hv.
template <int EPL, int G, int NT, bool HALVES = false>
DEVI void attn_fast_unit(const DevPtrs& d, int unit, int layer, int pos, const uint16_t* q_norm,
                         const uint16_t* k_norm, FastAttnSmem<EPL * 32>& sm, OpTags tg = OpTags{0u, 0u},
                         AttnHalves hv = AttnHalves{nullptr, nullptr, 0}) {
  constexpr int HD = EPL * 32;
  static_assert(G + 1 <= NT / 32, "one warp per query head plus a K/V warp");
  const int r = unit / d.Hkv, g = unit % d.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = d.Hq, hkv = d.Hkv, N = d.N;
  const size_t qkv = static_cast<size_t>(r) * d.qkv_dim;
  float* kb = d.fast_kv + (((static_cast<size_t>(r) * d.fast_n_layer + layer) * 2 + 0) * hkv + g) * N * HD;
  float* vb = kb + static_cast<size_t>(hkv) * N * HD;
  float (*ks)[HD] = sm.ks;
  float (*vs)[HD] = sm.vs;
  {
    // every load of the earlier positions in flight before the first store
    constexpr int kIt = (kMaxCodebooks * HD + NT - 1) / NT;
    float kt[kIt], vt[kIt];
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int e = threadIdx.x + it * NT;
      if (e < pos * HD) {
        kt[it] = ldf(kb + e);
        vt[it] = ldf(vb + e);
      }
    }
#pragma unroll
    for (int it = 0; it < kIt; ++it) {
      const int e = threadIdx.x + it * NT;
      if (e < pos * HD) {
        ks[e / HD][e % HD] = kt[it];
        vs[e / HD][e % HD] = vt[it];
      }
    }
  }
  float q[EPL];
  if (warp < G) {
    const HeadNR<EPL> nr = head_nr_load<EPL>(q_norm, pos, d, lane);
    act_load<EPL>(d.qkv, d.qkv_t, qkv + (g * G + warp) * HD + lane * EPL, tg.in, q, d);
    head_nr_apply<EPL>(q, nr, q_norm != nullptr, d.eps);
  } else if (warp == G) {
    const HeadNR<EPL> nr = head_nr_load<EPL>(k_norm, pos, d, lane);
    float kv[EPL], vv[EPL];
    act_load<EPL>(d.qkv, d.qkv_t, qkv + hq * HD + g * HD + lane * EPL, tg.in, kv, d);
    act_load<EPL>(d.qkv, d.qkv_t, qkv + hq * HD + hkv * HD + g * HD + lane * EPL, tg.in, vv, d);
    head_nr_apply<EPL>(kv, nr, k_norm != nullptr, d.eps);
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      kb[static_cast<size_t>(pos) * HD + lane * EPL + j] = kv[j];
      vb[static_cast<size_t>(pos) * HD + lane * EPL + j] = vv[j];
      ks[pos][lane * EPL + j] = kv[j];
      vs[pos][lane * EPL + j] = vv[j];
    }
  }
  csync<NT>();
  if (warp < G) {
    const int h = g * G + warp;
    const float scale = 1.0f / sqrtf(static_cast<float>(HD));
    float s[kMaxCodebooks];
#pragma unroll
    for (int t = 0; t < kMaxCodebooks; ++t) {
      float a = 0.f;
      if (t <= pos) {
#pragma unroll
        for (int j = 0; j < EPL; ++j) a = fmaf(q[j], ks[t][lane * EPL + j], a);
      }
      s[t] = a;
    }
    // lane sums of every position's dot product with their shuffles
    // interleaved (the butterfly of warp_sum, position by position)
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1)
#pragma unroll
      for (int t = 0; t < kMaxCodebooks; ++t) s[t] += __shfl_xor_sync(0xFFFFFFFFu, s[t], sh);
    float m = -INFINITY;
#pragma unroll
    for (int t = 0; t < kMaxCodebooks; ++t) {
      if (t <= pos) {
        s[t] *= scale;
        m = fmaxf(m, s[t]);
      } else {
        s[t] = -INFINITY;
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
    const size_t dst = static_cast<size_t>(r) * hq * HD + h * HD;
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
      o[j] = o[j] / l;
      act_store(d.attn, d.attn_t, dst + lane * EPL + j, tg.out, o[j]);
    }
    if (HALVES && hv.xh != nullptr) attn_halves<EPL>(hv, r, h * HD + lane * EPL, o);
  }
  csync<NT>();   // shared buffers are reused by the next unit
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
// Both are found from one histogram of mass over kSampBins bins of
// (zmax - z) / T (a bin index never increases with the key, so the bins
// partition the key order): an inclusive scan over the bins locates the bin
// holding a target, and only the candidates of that bin are ranked by key.
// A bin with more than kBinCap candidates (near-equal logits) falls back to a
// most-significant-byte-first radix descent over the keys.  [P2] "Two
// autoregressions": sample(biased_logits, ...) for q0, unmasked
// sample(logits, ...) for q1..q9.
constexpr int kMaxCands = 4097;

constexpr int kSampBins = 2048;
constexpr int kBinCap = 512;
// Candidates with (zmax - z) / T above ln(2^25) have zero mass and are never
// selected; the bins cover [0, 17.5) of that distance.
constexpr float kBinScale = static_cast<float>(kSampBins) / 17.5f;

template <int NT>
struct SampSmem {
  static constexpr int NW = NT / 32;
  unsigned long long hmass[kSampBins];   // per-bin mass, then its inclusive scan
  unsigned int hcnt[kSampBins];
  unsigned int hhi[kSampBins];           // samp_hist: per-bin sum of mass >> 8
  unsigned long long lkey[kBinCap];      // candidates of the target bin
  unsigned int lmass[kBinCap];
  int nlist;
  unsigned long long red64[NW];
  float redf[NW];
  unsigned long long bc[4];
  int ibc[4];
  int hist[kRasRing];   // q0: the slot's RAS history ring
  int s_commit, s_active;
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
  csync<NT>();
  float t = sm.redf[0];
  for (int w = 1; w < SampSmem<NT>::NW; ++w) t = fmaxf(t, sm.redf[w]);
  csync<NT>();
  return t;
}

template <int NT>
DEVI unsigned long long samp_block_sum(unsigned long long v, SampSmem<NT>& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  if (lane == 0) sm.red64[warp] = v;
  csync<NT>();
  unsigned long long t = 0;
  for (int w = 0; w < SampSmem<NT>::NW; ++w) t += sm.red64[w];
  csync<NT>();
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
  csync<NT>();
  unsigned long long t = 0;
  for (int w = 0; w < SampSmem<NT>::NW; ++w) t = sm.red64[w] > t ? sm.red64[w] : t;
  csync<NT>();
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
    csync<NT>();
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
    csync<NT>();
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
    csync<NT>();
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
      csync<NT>();
      result = sm.bc[2];
      *mass_out = mbin;
      break;
    }
    csync<NT>();
  }
  csync<NT>();
  *above_out = above;
  return result;
}

// Bin of a candidate with positive mass (monotone: never increases with z).
DEVI int samp_bin(float z, float zmax, float inv_t) {
  const float t = (zmax - z) * inv_t * kBinScale;
  return t < static_cast<float>(kSampBins - 1) ? static_cast<int>(t) : kSampBins - 1;
}

// Histogram of mass per bin, then its inclusive scan (hmass[b] = mass of
// bins 0..b).  hcnt keeps the per-bin counts.
template <int NT, int EPT>
DEVI void samp_hist(const float (&z)[EPT], const uint32_t (&mass)[EPT], int n, float zmax, float inv_t,
                    SampSmem<NT>& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int BPT = kSampBins / NT;   // bins per thread (contiguous)
  static_assert(kSampBins % NT == 0 && BPT >= 1, "bins split evenly over the threads");
  // A bin's mass is accumulated as two 32-bit sums, of mass & 255 (at most
  // 4,097 x 255) and of mass >> 8 (at most 4,097 x 2^16): exact, and 32-bit
  // shared-memory atomics.  The low sums live in the first half of hmass
  // until the scan (read by every thread before the barrier that precedes
  // the scan's writes).
  unsigned int* hlo = reinterpret_cast<unsigned int*>(sm.hmass);
  for (int b = tid; b < kSampBins; b += NT) {
    hlo[b] = 0u;
    sm.hhi[b] = 0u;
    sm.hcnt[b] = 0u;
  }
  csync<NT>();
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int i = tid + e * NT;
    if (i < n && mass[e] != 0u) {
      const int b = samp_bin(z[e], zmax, inv_t);
      atomicAdd(&hlo[b], mass[e] & 255u);
      atomicAdd(&sm.hhi[b], mass[e] >> 8);
      atomicAdd(&sm.hcnt[b], 1u);
    }
  }
  csync<NT>();
  unsigned long long c[BPT];
  unsigned long long run = 0;
#pragma unroll
  for (int j = 0; j < BPT; ++j) {
    const int b = tid * BPT + j;
    run += (static_cast<unsigned long long>(sm.hhi[b]) << 8) + hlo[b];
    c[j] = run;
  }
  unsigned long long incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sm.red64[warp] = incl;
  csync<NT>();
  unsigned long long off = incl - run;
  for (int w = 0; w < warp; ++w) off += sm.red64[w];
#pragma unroll
  for (int j = 0; j < BPT; ++j) sm.hmass[tid * BPT + j] = off + c[j];
  csync<NT>();
}

// First key (descending) whose inclusive cumulative mass reaches target
// (1 <= target <= total), using the scanned histogram; *incl_out is that
// inclusive cumulative mass.
template <int NT, int EPT>
DEVI unsigned long long samp_resolve(const float (&z)[EPT], const unsigned long long (&key)[EPT],
                                     const uint32_t (&mass)[EPT], int n, float zmax, float inv_t,
                                     unsigned long long target, SampSmem<NT>& sm,
                                     unsigned long long* incl_out, bool* radix) {
  const int tid = threadIdx.x;
  // the bin holding the target: excl(b) < target <= incl(b) (exactly one)
  for (int b = tid; b < kSampBins; b += NT) {
    const unsigned long long hi = sm.hmass[b];
    const unsigned long long lo = b == 0 ? 0ull : sm.hmass[b - 1];
    if (lo < target && target <= hi) {
      sm.ibc[0] = b;
      sm.bc[0] = lo;
    }
  }
  if (tid == 0) sm.nlist = 0;
  csync<NT>();
  const int bin = sm.ibc[0];
  const unsigned long long above = sm.bc[0];
  const int cnt = static_cast<int>(sm.hcnt[bin]);
  if (cnt > kBinCap) {
    // near-equal logits crowd one bin: radix descent over all keys
    unsigned long long ab, mk;
    const unsigned long long k = samp_select<NT, EPT>(key, mass, n, target, sm, &ab, &mk);
    *incl_out = ab + mk;
    *radix = true;   // the descent reused the bin arrays
    return k;
  }
  *radix = false;
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int i = tid + e * NT;
    if (i < n && mass[e] != 0u && samp_bin(z[e], zmax, inv_t) == bin) {
      const int slot = atomicAdd(&sm.nlist, 1);
      sm.lkey[slot] = key[e];
      sm.lmass[slot] = mass[e];
    }
  }
  csync<NT>();
  for (int i = tid; i < cnt; i += NT) {
    const unsigned long long ki = sm.lkey[i];
    unsigned long long cum = above;
    for (int j = 0; j < cnt; ++j)
      if (sm.lkey[j] >= ki) cum += sm.lmass[j];
    if (cum >= target && cum - sm.lmass[i] < target) {
      sm.bc[1] = ki;
      sm.bc[2] = cum;
    }
  }
  csync<NT>();
  *incl_out = sm.bc[2];
  const unsigned long long k = sm.bc[1];
  csync<NT>();
  return k;
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
  if (Z == 0ull) {
    // no finite mass (non-finite logits): take the largest key
    unsigned long long best = 0;
#pragma unroll
    for (int e = 0; e < EPT; ++e)
      if (tid + e * NT < c.n && key[e] > best) best = key[e];
    return key_to_index(c, samp_block_max_u64(best, sm));
  }
  unsigned long long tc = Z;
  if (top_p < 1.0f) {
    const double t = ceil(static_cast<double>(top_p) * static_cast<double>(Z));
    tc = t < 1.0 ? 1ull : static_cast<unsigned long long>(t);
    if (tc > Z) tc = Z;
  }
  samp_hist<NT, EPT>(z, mass, c.n, zmax, inv_t, sm);
  unsigned long long zk, zd;
  bool radix = false;
  samp_resolve<NT, EPT>(z, key, mass, c.n, zmax, inv_t, tc, sm, &zk, &radix);
  unsigned long long td =
      static_cast<unsigned long long>(floor(static_cast<double>(u) * static_cast<double>(zk))) + 1ull;
  if (td > zk) td = zk;
  if (radix) samp_hist<NT, EPT>(z, mass, c.n, zmax, inv_t, sm);
  const unsigned long long kd = samp_resolve<NT, EPT>(z, key, mass, c.n, zmax, inv_t, td, sm, &zd, &radix);
  return key_to_index(c, kd);
}

// Loads the candidates' logits and keys into registers; returns zmax.
// With tag != 0 the logits are tagged words at tsrc (all loads are issued
// before the first tag is checked).
template <int NT, int EPT>
DEVI float samp_load(const float* src, const Cands& c, float (&z)[EPT], unsigned long long (&key)[EPT],
                     SampSmem<NT>& sm, const uint64_t* tsrc = nullptr, uint32_t tag = 0u,
                     const DevPtrs* d = nullptr) {
  static_assert(EPT <= 32, "one bit per candidate slot");
  float zm = -INFINITY;
  uint32_t late = 0;   // tagged: words that did not carry the tag yet
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int i = threadIdx.x + e * NT;
    z[e] = -INFINITY;
    if (i < c.n) {
      if (tag != 0u) {
        const uint64_t w = tag_load(tsrc + i);
        z[e] = tag_val(w);
        late |= (tag_of(w) != tag ? 1u : 0u) << e;
      } else {
        z[e] = ldf(src + i);
      }
    }
  }
  if (late != 0u) {
#pragma unroll
    for (int e = 0; e < EPT; ++e)
      if ((late >> e) & 1u) z[e] = tag_wait1(tsrc + threadIdx.x + e * NT, tag, d->err, d->wait_limit_ns);
  }
#pragma unroll
  for (int e = 0; e < EPT; ++e) {
    const int i = threadIdx.x + e * NT;
    key[e] = 0;
    if (i < c.n) {
      zm = fmaxf(zm, z[e]);
      key[e] = (static_cast<unsigned long long>(ord_f32(z[e])) << 32) |
               static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(cand_id(c, i)));
    }
  }
  return samp_block_max(zm, sm);
}

// q0 of one row: normal draw, repetition-aware resample, commit, and the
// inputs of fast passes 0 and 1.
// Fast-pass inputs written by the samplers: pass p of batch row `row`.
DEVI size_t fin_plain_off(int p, int row, int D) {
  return (static_cast<size_t>(p & 1) * kMaxRows + row) * D;
}
DEVI size_t fin_tagged_off(int p, int row, int D) {
  return (static_cast<size_t>(p) * kTaggedRows + row) * D;
}
template <int NT>
DEVI void fin_zero(const DevPtrs& d, int p, int row, uint32_t tag) {
  if (tag == 0u) return;   // plain buffers: nothing waits for an inactive row
  uint64_t* f = d.fin_t + fin_tagged_off(p, row, d.D);
  for (int k = threadIdx.x; k < d.D; k += NT) tag_store(f + k, 0.f, tag);
}

template <int NT>
DEVI void sample_q0_row(const DevPtrs& d, int row, const SampIO& io, SampSmem<NT>& sm,
                        OpTags tg = OpTags{0u, 0u}) {
  constexpr int EPT = (kMaxCands + NT - 1) / NT;
  const int tid = threadIdx.x;
  const RowInfo ri = ld_row(&d.rows[row]);
  const int slot = ri.slot;
  const int ns = d.n_sem, N = d.N;
  // the slot's state, loaded once and in parallel: finished flag, RAS
  // history length and ring
  if (tid == 0) {
    sm.ibc[2] = ldi(d.finished + slot);
    sm.ibc[3] = ldi(d.hist_n + slot);
  } else if (tid >= 32 && tid < 32 + kRasRing) {
    sm.hist[tid - 32] = ldi(d.hist + slot * kRasRing + (tid - 32));
  }
  // the draw's uniforms and the forced code are requested before the logits
  // are waited on, so their round trips overlap
  const float* u = io.uniforms + static_cast<size_t>(row) * io.ldu;
  const float u_normal = u[0], u_ras = u[1];
  const int forced0 = (io.forced && tid == 0) ? io.forced[static_cast<size_t>(row) * io.ldf] : 0;
  const float* zsrc = d.z_last + static_cast<size_t>(slot) * (ns + 1);
  // [P2] "Two autoregressions": the bias keeps the semantic ids and <|im_end|>.
  const Cands c{ns + (io.sp.allow_eos ? 1 : 0), ns, d.sem_begin, d.im_end};
  float z[EPT];
  unsigned long long key[EPT];
  const float zmax = samp_load<NT, EPT>(zsrc, c, z, key, sm);   // (its block reduction orders the state loads)
  if (io.slow_logits_out) {
    float* so = io.slow_logits_out + static_cast<size_t>(row) * (ns + 1);
#pragma unroll
    for (int e = 0; e < EPT; ++e)
      if (tid + e * NT < c.n) so[tid + e * NT] = z[e];
    if (c.n < ns + 1 && tid == 0) so[ns] = ldf(zsrc + ns);
  }
  if (sm.ibc[2]) {
    // a finished slot stays finished: no codes, no state change
    if (tid == 0) {
      io.status_out[row] = 2;
      d.rows[row].active = 0;
      d.commit_map[row] = -1;
    }
    for (int k = tid; k < N; k += NT) io.codes_out[row * N + k] = -1;
    fin_zero<NT>(d, 0, row, tg.out);
    fin_zero<NT>(d, 1, row, tg.out);
    csync<NT>();
    return;
  }
  const int normal = samp_draw<NT, EPT>(z, key, c, zmax, io.sp.temperature, io.sp.top_p, u_normal, sm);
  // [P2] "Two autoregressions": a second draw at temperature 1.0, top-p 0.9,
  // used when the normal draw repeats a semantic token of the last 10 frames.
  // Every thread sees the same history, so the decision is uniform; the
  // second draw runs only when it is used or the caller records both draws.
  const int hn = sm.ibc[3];
  bool repeat = false;
  if (normal != ns) {
    const int w = min(io.sp.ras_win, hn);
    for (int j = 0; j < w; ++j)
      if (sm.hist[(hn - 1 - j) % kRasRing] == normal) repeat = true;
  }
  const bool use_ras = io.sp.ras_win > 0 && repeat;
  const int ras = (use_ras || io.draws_out)
                      ? samp_draw<NT, EPT>(z, key, c, zmax, io.sp.ras_temperature, io.sp.ras_top_p, u_ras, sm)
                      : -1;
  if (tid == 0) {
    const int chosen = use_ras ? ras : normal;
    const int commit = io.forced ? forced0 : chosen;
    if (io.draws_out) {
      io.draws_out[row * (N + 2) + 0] = normal;
      io.draws_out[row * (N + 2) + 1] = ras;
      io.draws_out[row * (N + 2) + 2] = chosen;
    }
    int active = 1;
    if (commit == ns || commit < 0 || commit > ns) {
      if (commit != ns) raise_error(d.err, DEV_ERR_BAD_INDEX);
      io.status_out[row] = 1;
      d.finished[slot] = 1;
      d.rows[row].active = 0;
      d.commit_map[row] = -1;
      active = 0;
    } else {
      io.status_out[row] = 0;
      d.hist[slot * kRasRing + (hn % kRasRing)] = commit;
      d.hist_n[slot] = hn + 1;
      d.codes_ws[row * kMaxCodebooks] = commit;
    }
    sm.s_commit = commit;
    sm.s_active = active;
  }
  csync<NT>();
  const int commit = sm.s_commit;
  if (!sm.s_active) {
    for (int k = tid; k < N; k += NT) io.codes_out[row * N + k] = -1;
    fin_zero<NT>(d, 0, row, tg.out);
    fin_zero<NT>(d, 1, row, tg.out);
    csync<NT>();
    return;
  }
  if (tid == 0) io.codes_out[row * N] = commit;
  // fast pass 0 reads the slow hidden state; pass 1 the embedding of q0
  // ([P2] "Two autoregressions", decode_one_token_ar).  q0 indexes the fast
  // embedding clamped to its rows (a no-op when n_sem == fast_vocab).
  const int D = d.D;
  const int e0 = min(commit, d.Cf - 1);
  const float* hl = d.h_last + static_cast<size_t>(slot) * D;
  const uint16_t* er = io.fast_emb + static_cast<size_t>(e0) * D;
  for (int k = tid; k < D; k += NT) {
    act_store(d.fin, d.fin_t, (tg.out ? fin_tagged_off(0, row, D) : fin_plain_off(0, row, D)) + k, tg.out,
              ldf(hl + k));
    act_store(d.fin, d.fin_t, (tg.out ? fin_tagged_off(1, row, D) : fin_plain_off(1, row, D)) + k, tg.out,
              bf16bits_to_f32(er[k]));
  }
  csync<NT>();
}

// q_k (k >= 1) of one row from the fast head's logits, and the input of pass k+1.
template <int NT>
DEVI void sample_fast_row(const DevPtrs& d, int row, int k, const SampIO& io, SampSmem<NT>& sm,
                          OpTags tg = OpTags{0u, 0u}) {
  constexpr int EPT = (kMaxCands + NT - 1) / NT;
  const int tid = threadIdx.x;
  const int N = d.N, Cf = d.Cf;
  const size_t zoff = static_cast<size_t>(row) * d.logit_ld;
  const Cands c{Cf, Cf, 0, -1};
  // the draw's uniform and the forced code are requested before the logits
  // are waited on, so their round trips overlap
  const float uk = io.uniforms[static_cast<size_t>(row) * io.ldu + k + 1];
  const int forced_k = (io.forced && tid == 0) ? io.forced[static_cast<size_t>(row) * io.ldf + k] : 0;
  const int active = ldi(&d.rows[row].active);   // settled by the q0 draw
  float z[EPT];
  unsigned long long key[EPT];
  const float zmax = samp_load<NT, EPT>(d.logits + zoff, c, z, key, sm, d.logits_t + zoff, tg.in, &d);
  if (io.fast_logits_out) {
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      const int i = tid + e * NT;
      if (i < Cf) io.fast_logits_out[(static_cast<size_t>(row) * (N - 1) + (k - 1)) * Cf + i] = z[e];
    }
  }
  if (!active) {
    if (k + 1 < N) fin_zero<NT>(d, k + 1, row, tg.out);
    csync<NT>();
    return;
  }
  const int draw = samp_draw<NT, EPT>(z, key, c, zmax, io.sp.temperature, io.sp.top_p, uk, sm);
  if (tid == 0) {
    int commit = io.forced ? forced_k : draw;
    if (commit < 0 || commit >= Cf) {
      raise_error(d.err, DEV_ERR_BAD_INDEX);
      commit = 0;
    }
    if (io.draws_out) io.draws_out[row * (N + 2) + k + 2] = draw;
    d.codes_ws[row * kMaxCodebooks + k] = commit;
    io.codes_out[row * N + k] = commit;
    sm.s_commit = commit;
  }
  csync<NT>();
  if (k + 1 < N) {
    const int D = d.D;
    const size_t f = tg.out ? fin_tagged_off(k + 1, row, D) : fin_plain_off(k + 1, row, D);
    const uint16_t* er = io.fast_emb + static_cast<size_t>(sm.s_commit) * D;
    for (int j = tid; j < D; j += NT) act_store(d.fin, d.fin_t, f + j, tg.out, bf16bits_to_f32(er[j]));
  }
  csync<NT>();
}

// ============================================================================
// Multi-codebook fusion
// ============================================================================
// [P2] "Two autoregressions", Eq. 1 and the code's scale:
//   x_{t+1} = (e_LM[q0] + sum_{k<N} E^(k)[q_k]) / sqrt(N+1)
// with E^(k) the block of the fusion table that starts at row
// n_sem + (k-1) * fast_vocab (row 0 for k = 0).
template <int NT>
DEVI void fusion_row(const DevPtrs& d, int row, const uint16_t* tok_emb, const uint16_t* fusion,
                     OpTags tg = OpTags{0u, 0u}) {
  const int D = d.D, N = d.N;
  if (!ldi(&d.rows[row].active)) {
    if (tg.out != 0u)
      for (int k = threadIdx.x; k < D; k += NT) tag_store(d.xs_t + static_cast<size_t>(row) * D + k, 0.f, tg.out);
    return;
  }
  int q[kMaxCodebooks];
  bool bad = false;
  for (int k = 0; k < N; ++k) {
    q[k] = ldi(d.codes_ws + row * kMaxCodebooks + k);
    const int lim = k == 0 ? d.n_sem : d.Cf;
    if (q[k] < 0 || q[k] >= lim) bad = true;
  }
  if (bad) {
    if (threadIdx.x == 0) raise_error(d.err, DEV_ERR_BAD_INDEX);
    if (tg.out != 0u)
      for (int k = threadIdx.x; k < D; k += NT) tag_store(d.xs_t + static_cast<size_t>(row) * D + k, 0.f, tg.out);
    return;
  }
  const float scale = 1.0f / sqrtf(static_cast<float>(N + 1));
  // one 8-element vector per thread; the row reads are independent and the
  // compiler keeps a few of them in flight (few live registers: this code is
  // inlined into the persistent kernel)
  const int DV = D >> 3;
  for (int j = threadIdx.x; j < DV; j += NT) {
    float acc[8];
    {
      const uint4 v = *reinterpret_cast<const uint4*>(tok_emb + static_cast<size_t>(d.sem_begin + q[0]) * D + 8 * j);
      acc[0] = bf16lo(v.x); acc[1] = bf16hi(v.x); acc[2] = bf16lo(v.y); acc[3] = bf16hi(v.y);
      acc[4] = bf16lo(v.z); acc[5] = bf16hi(v.z); acc[6] = bf16lo(v.w); acc[7] = bf16hi(v.w);
    }
#pragma unroll 4
    for (int k = 0; k < N; ++k) {
      const int off = k == 0 ? 0 : d.n_sem + (k - 1) * d.Cf;
      const uint4 w = *reinterpret_cast<const uint4*>(fusion + static_cast<size_t>(off + q[k]) * D + 8 * j);
      acc[0] += bf16lo(w.x); acc[1] += bf16hi(w.x); acc[2] += bf16lo(w.y); acc[3] += bf16hi(w.y);
      acc[4] += bf16lo(w.z); acc[5] += bf16hi(w.z); acc[6] += bf16lo(w.w); acc[7] += bf16hi(w.w);
    }
    if (tg.out != 0u) {
      uint64_t* dst = d.xs_t + static_cast<size_t>(row) * D + 8 * j;
#pragma unroll
      for (int e = 0; e < 8; e += 2) tag_store2(dst + e, acc[e] * scale, acc[e + 1] * scale, tg.out);
    } else {
      float4* dst = reinterpret_cast<float4*>(d.xs + static_cast<size_t>(row) * D + 8 * j);
      dst[0] = make_float4(acc[0] * scale, acc[1] * scale, acc[2] * scale, acc[3] * scale);
      dst[1] = make_float4(acc[4] * scale, acc[5] * scale, acc[6] * scale, acc[7] * scale);
    }
  }
}

}  // namespace dualar
