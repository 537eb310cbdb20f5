// Persistent frame kernel: one cooperative launch runs a whole Dual-AR frame
// for a batch of 1-2 sequences -- q0 draw, the N fast-AR passes (all
// codebooks, without returning to the host), fusion, the slow-AR position and
// the restricted head.
//
// One CTA per SM: 16 consumer warps execute the ops of a fixed program in
// order, separated by grid-wide barriers; one producer warp walks the same
// program and streams the weight tiles of every GEMV into a shared-memory ring
// with bulk copies.  Weights never depend on activations, so the producer
// runs ahead across op boundaries (bounded by the ring depth) and HBM keeps
// streaming while the consumers wait at a barrier, sample or attend.
//
// Ops hand activations to each other as tagged words (common.cuh): a reader
// spins on the words it needs until they carry the tag of the op that writes
// them, so consecutive ops need no grid-wide barrier -- a CTA moves on as soon
// as its own inputs are there.  Every activation buffer is rewritten in place
// only by an op that (directly or through earlier ops) has read outputs of
// every reader of the previous contents, so a word is never overwritten while
// someone still waits for its old tag.  One grid barrier remains, after the
// q0 draw, which may deactivate a row (read by attention units anywhere).
//
// Every wait is bounded: a wait that does not complete within the handle's
// wait limit raises DEV_ERR_GRID_TIMEOUT, and once the error word is set the
// remaining waits give up quickly, so the kernel always finishes.
//
// [P2] "Two autoregressions" (decode_one_token_ar order, fast KV cache of
// num_codebooks positions, Eq. 1 fusion); "The slow AR is Qwen3-4B".
#include "common.cuh"
#include "gemv.cuh"
#include "internal.h"
#include "mega.h"
#include "ops.cuh"

namespace dualar {

constexpr int kMegaNCT = kWarpsC * 32;   // consumer threads
constexpr int kMegaMaxStages = 4;   // measured: 4 stages beat 3 with the fast K/V resident in shared memory
constexpr size_t kMegaSmemLimit = 227 * 1024;
// producer timing, in SM cycles (about 2 GHz)
constexpr long long kIdleCycles = 3000;        // a wait this long: the consumers are not streaming
constexpr long long kTileCycles = 1600;        // one 40 KB tile per SM at its share of HBM bandwidth
constexpr long long kAbortCheckCycles = 20000; // how often a long wait looks at the error word
constexpr uint64_t kIdlePrefetchBytes = 512 * 1024;   // prefetch window growth while the consumers idle

// W4: the program has packed 4-bit GEMVs, whose x rows are followed by
// their 32-element sums (gemv_stage_x<NB, true>).
template <int NB, int HD, int G, bool W4>
struct MegaLayout {
  // fixed area (offsets from the dynamic shared memory base)
  static constexpr size_t bars = 0;   // full[8], empty[8], attn[2]
  static constexpr size_t scratch = 256;
  static constexpr size_t pro = (scratch + sizeof(GemvScratch<NB>) + 15) & ~size_t(15);
  static constexpr size_t opbuf = (pro + sizeof(GemvPro<NB>) + 15) & ~size_t(15);   // MegaOp[2]
  static constexpr size_t uni = (opbuf + 2 * sizeof(MegaOp) + 127) & ~size_t(127);
  // union region: GEMV x rows | paged attention | fast attention | sampler
  __host__ __device__ static size_t union_bytes(int kmax) {
    size_t u = sizeof(float) * size_t(NB) * (kmax + (W4 ? kmax / 32 : 0));
    u = u > sizeof(AttnSmem<HD, G, kMegaNCT, 1>) ? u : sizeof(AttnSmem<HD, G, kMegaNCT, 1>);
    u = u > sizeof(FastAttnSmem<HD>) ? u : sizeof(FastAttnSmem<HD>);
    u = u > sizeof(SampSmem<kMegaNCT>) ? u : sizeof(SampSmem<kMegaNCT>);
    return u;
  }
  __host__ __device__ static size_t ring(int kmax) { return (uni + union_bytes(kmax) + 127) & ~size_t(127); }
  // as many 40 KB ring stages as fit next to the fixed area and the union
  __host__ __device__ static int stages(int kmax) {
    const size_t r = ring(kmax);
    const size_t room = kMegaSmemLimit > r ? kMegaSmemLimit - r : 0;
    const int s = static_cast<int>(room / kStageBytes);
    return s > kMegaMaxStages ? kMegaMaxStages : s;
  }
  __host__ __device__ static size_t total(int kmax) {
    return ring(kmax) + size_t(stages(kmax)) * kStageBytes;
  }
};

DEVI void grid_barrier(uint32_t* counter, uint32_t target, uint32_t* err, uint64_t limit_ns) {
  named_barrier(1, kMegaNCT);
  if (threadIdx.x == 0) {
    // release: every write of this CTA's consumers (ordered before this
    // thread by the CTA barrier) is visible before the arrival counts
    red_release_gpu_add(counter, 1u);
    const volatile uint32_t* ev = err;
    if (ld_acquire_gpu(counter) < target) {
      const uint64_t t0 = global_timer_ns();
      uint64_t next_chk = kAbortCheckNs;
      while (ld_acquire_gpu(counter) < target) {
        const uint64_t dt = global_timer_ns() - t0;
        if (dt > next_chk) {
          next_chk = dt + kAbortCheckNs;
          if (*ev & (DEV_ERR_GRID_TIMEOUT | DEV_ERR_MBAR_TIMEOUT)) break;   // another CTA gave up
        }
        if (dt > limit_ns) {
          raise_error(err, DEV_ERR_GRID_TIMEOUT);
          break;
        }
      }
    }
  }
  named_barrier(1, kMegaNCT);
}

// Position in the sequence of weight tiles of the frame program (all GEMV
// ops, in order) for one CTA.  The descriptor of the next GEMV is loaded one
// op ahead, so moving to it costs no memory round trip.
template <bool W4>
struct TileCursor {
  const ProdOp* prod;
  int n, cta, ncta;
  int j;
  ProdOp nxt;
  GemvArgs a;
  GemvGeo g;
  TileIter it;
  __device__ static GemvArgs args_of(const ProdOp& q) {
    GemvArgs a{};
    a.w0 = q.w0;
    a.w1 = q.w1;
    a.n0 = q.n0;
    a.n1 = q.n1;
    a.K = q.K;
    a.mode = q.mode;
    a.w4 = W4 ? q.w4 : 0;
    return a;
  }
  __device__ GemvGeo geo(const GemvArgs& x) const {
    if constexpr (W4) {
      if (x.w4) return gemv_geo<true>(x, cta, ncta);
    }
    return gemv_geo(x, cta, ncta);
  }
  __device__ TileCursor(const ProdOp* pr, int np, int c, int nc)
      : prod(pr), n(np), cta(c), ncta(nc), j(0), nxt(), a(), g(), it(a, g) {
    if (n > 0) {
      a = args_of(prod[0]);
      g = geo(a);
      it = TileIter(a, g);
    }
    if (n > 1) nxt = prod[1];
  }
  __device__ bool next(const uint16_t*& src, uint32_t& bytes) {
    while (j < n) {
      int row0, rows, part;
      if (it.next(row0, rows, part)) {
        if constexpr (W4) {
          if (a.w4) {
            src = static_cast<const uint16_t*>(gemv_tile_ptr<true>(a, row0, part));
            bytes = static_cast<uint32_t>(rows) * gemv_row_bytes<true>(a.K);
            return true;
          }
        }
        src = gemv_tile_src(a, row0, part);
        bytes = static_cast<uint32_t>(rows) * a.K * 2;
        return true;
      }
      if (++j >= n) break;
      a = args_of(nxt);
      g = geo(a);
      it = TileIter(a, g);
      if (j + 1 < n) nxt = prod[j + 1];
    }
    return false;
  }
};

template <int NB, int HD, int G, bool W4>
__global__ void __launch_bounds__(kGemvThreads, 1) mega_kernel(const MegaParams p) {
  using Lay = MegaLayout<NB, HD, G, W4>;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::bars);
  GemvRing ring;
  ring.full = bars;
  ring.empty = bars + kMaxStagesRing;
  ring.base = smem + Lay::ring(p.kmax);
  ring.stages = Lay::stages(p.kmax);
  uint64_t* abars = bars + 2 * kMaxStagesRing;
  GemvScratch<NB>& scr = *reinterpret_cast<GemvScratch<NB>*>(smem + Lay::scratch);
  GemvPro<NB>& pro = *reinterpret_cast<GemvPro<NB>*>(smem + Lay::pro);
  unsigned char* uni = smem + Lay::uni;
  MegaOp* opb = reinterpret_cast<MegaOp*>(smem + Lay::opbuf);   // ops i and i+1 (slot i & 1)
  constexpr int kOpChunks = static_cast<int>(sizeof(MegaOp) / 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, ncta = gridDim.x;
  const DevPtrs& d = p.d;

  if (tid == 0) {
    for (int s = 0; s < ring.stages; ++s) {
      mbar_init(&ring.full[s], 1);
      mbar_init(&ring.empty[s], kWarpsC);
    }
    mbar_init(&abars[0], 1);
    mbar_init(&abars[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (tid < kOpChunks && p.n_ops > 0)
    reinterpret_cast<uint4*>(opb)[tid] = reinterpret_cast<const uint4*>(p.ops)[tid];
  __syncthreads();

  if (warp == kWarpsC) {
    // ---------------- producer: weights of every GEMV of the program -------
    // Tiles go into the ring in program order; a second cursor keeps the next
    // p.prefetch_bytes of tiles beyond the ring in flight into L2, so HBM
    // keeps streaming while the consumers wait at a barrier, sample or attend.
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      TileCursor<W4> lc(p.prod, p.n_prod, cta, ncta), pc(p.prod, p.n_prod, cta, ncta);
      uint64_t loaded = 0, prefetched = 0;
      const uint32_t* errp = d.err;
      uint32_t t = 0;
      const uint16_t* src;
      uint32_t bytes;
      bool ok = true;
      while (ok && lc.next(src, bytes)) {
        const int s = static_cast<int>(t % ring.stages);
        if (t >= static_cast<uint32_t>(ring.stages)) {
          const uint32_t parity = ((t / ring.stages) - 1) & 1;
          if (!mbar_try_wait(&ring.empty[s], parity)) {
            // Ring full: keep the next p.prefetch_bytes of tiles beyond the
            // ring in flight into L2.  A wait longer than a tile interval
            // means the consumers are not streaming (they wait for
            // activations, attend or sample): the window then grows by one
            // tile per tile interval, up to kIdlePrefetchBytes more, so HBM
            // keeps working.
            {
              const uint16_t* ps;
              uint32_t pb;
              while (prefetched < loaded + p.prefetch_bytes && pc.next(ps, pb)) {
                if (prefetched + pb > loaded + bytes) bulk_prefetch_l2(ps, pb);
                prefetched += pb;
              }
            }
            const long long c0 = clock64();
            long long next_pf = c0 + kIdleCycles, next_chk = c0 + kAbortCheckCycles;
            const uint64_t g0 = global_timer_ns();
            while (!mbar_try_wait(&ring.empty[s], parity)) {
              const long long now = clock64();
              if (now >= next_pf) {
                next_pf = now + kTileCycles;
                const uint16_t* ps;
                uint32_t pb;
                bool issued = false;
                while (!issued && prefetched < loaded + p.prefetch_bytes + kIdlePrefetchBytes && pc.next(ps, pb)) {
                  if (prefetched + pb > loaded + bytes) {
                    bulk_prefetch_l2(ps, pb);
                    issued = true;
                  }
                  prefetched += pb;
                }
              }
              if (now >= next_chk) {
                next_chk = now + kAbortCheckCycles;
                const uint64_t dt = global_timer_ns() - g0;
                if (*reinterpret_cast<const volatile uint32_t*>(errp) || dt > d.wait_limit_ns) {
                  raise_error(d.err, DEV_ERR_MBAR_TIMEOUT);
                  ok = false;
                  break;
                }
              }
            }
            if (!ok) break;
          }
        }
        mbar_arrive_expect_tx(&ring.full[s], bytes);
        bulk_load_g2s(ring.base + static_cast<size_t>(s) * kStageBytes, src, bytes, &ring.full[s], pol);
        loaded += bytes;
        ++t;
        // the prefetch cursor never falls behind the ring: otherwise the next
        // ring-full wait would first walk every tile it missed, with the
        // stage it waits for possibly long free
        {
          const uint16_t* ps;
          uint32_t pb;
          while (prefetched < loaded && pc.next(ps, pb)) prefetched += pb;
        }
      }
      gemv_drain(ring, t, d.wait_limit_ns);
    }
    return;
  }

  // ---------------- consumers ------------------------------------------------
  uint32_t t = 0;
  uint32_t aphase[2] = {0u, 0u};
  const uint32_t ep = p.epoch;
  // (thread 0) this CTA's first paged-attention unit, found at the first QKV
  // projection of the slow AR (after the q0 draw has settled the rows)
  const int hkv = d.Hkv;
  for (int i = 0; i < p.n_ops; ++i) {
    const MegaOp& op = opb[i & 1];
    // the next op's descriptor arrives while this op runs
    const bool fetch = i + 1 < p.n_ops && tid < kOpChunks;
    if (fetch) {
      cp_async16(reinterpret_cast<uint4*>(&opb[(i + 1) & 1]) + tid, reinterpret_cast<const uint4*>(p.ops + i + 1) + tid);
      cp_async_commit();
    }
    uint64_t* tr = p.trace ? p.trace + (static_cast<size_t>(cta) * p.n_ops + i) * 4 : nullptr;
    if (tr && tid == 0) {
      tr[0] = global_timer_ns();
      tr[1] = tr[2] = 0;
    }
    switch (op.type) {
      case MOP_GEMV: {
        const bool w4op = W4 && op.g.w4;
        const GemvGeo g = w4op ? gemv_geo<true>(op.g, cta, ncta) : gemv_geo(op.g, cta, ncta);
        float* xs = reinterpret_cast<float*>(uni);
        float* gsum = xs + static_cast<size_t>(NB) * op.g.K;   // packed rows: the 32-element sums of x
        bool ok;
        if constexpr (W4) {
          if (w4op) {
            gemv_stage_x<NB, true>(op.g, g, xs, pro, cta, true, ep, gsum);
            if (tr && tid == 0) tr[1] = global_timer_ns();
            ok = gemv_consume_w4<NB>(op.g, g, ring, t, xs, gsum, scr, pro, ep, tr ? tr + 2 : nullptr);
          } else {
            gemv_stage_x<NB>(op.g, g, xs, pro, cta, true, ep);
            if (tr && tid == 0) tr[1] = global_timer_ns();
            ok = gemv_consume<NB>(op.g, g, ring, t, xs, scr, pro, ep, tr ? tr + 2 : nullptr);
          }
        } else {
          gemv_stage_x<NB>(op.g, g, xs, pro, cta, true, ep);
          if (tr && tid == 0) tr[1] = global_timer_ns();
          ok = gemv_consume<NB>(op.g, g, ring, t, xs, scr, pro, ep, tr ? tr + 2 : nullptr);
        }
        if (!ok) {
          // the ring protocol is broken: stop streaming (the error word is set)
          if (fetch) cp_async_wait_all();
          return;
        }
        break;
      }
      case MOP_ATTN_PAGED:
        attn_paged_units<HD, G, kMegaNCT, 1>(d, p.nrows, op.layer, p.units, p.chunk, true, op.q_norm,
                                          op.k_norm, *reinterpret_cast<AttnSmem<HD, G, kMegaNCT, 1>*>(uni),
                                          abars, aphase, cta, ncta, OpTags{op_tag(ep, op.in_src), op_tag(ep, i)});
        break;
      case MOP_ATTN_FAST:
        // unit u always runs on CTA u % ncta, so the fast K/V that one pass
        // writes to the global fast cache is read back by the same CTA in
        // later passes
        for (int u = cta; u < p.nrows * hkv; u += ncta)
          attn_fast_unit<HD / 32, G, kMegaNCT>(d, u, op.layer, op.pos, op.q_norm, op.k_norm,
                                               *reinterpret_cast<FastAttnSmem<HD>*>(uni),
                                               OpTags{op_tag(ep, op.in_src), op_tag(ep, i)});
        break;
      case MOP_SAMPLE_Q0:
        for (int r = cta; r < p.nrows; r += ncta)
          sample_q0_row<kMegaNCT>(d, r, p.io, *reinterpret_cast<SampSmem<kMegaNCT>*>(uni),
                                  OpTags{0u, op_tag(ep, i)});
        break;
      case MOP_SAMPLE_FAST:
        // row r always runs on CTA r: the codes of the frame (codes_ws) are
        // written and read (fusion) by one CTA
        for (int r = cta; r < p.nrows; r += ncta)
          sample_fast_row<kMegaNCT>(d, r, op.pos, p.io, *reinterpret_cast<SampSmem<kMegaNCT>*>(uni),
                                    OpTags{op_tag(ep, op.in_src), op_tag(ep, i)});
        break;
      case MOP_FUSION:
        for (int r = cta; r < p.nrows; r += ncta)
          fusion_row<kMegaNCT>(d, r, p.tok_emb, p.fusion, OpTags{0u, op_tag(ep, i)});
        break;
      default:
        break;
    }
    if (tr && tid == 0) tr[3] = global_timer_ns();
    if (fetch) cp_async_wait_all();
    if (i + 1 < p.n_ops) {
      if (i == 0) grid_barrier(p.bar, static_cast<uint32_t>(ncta) + p.bar_extra, d.err, d.wait_limit_ns);
      else named_barrier(1, kMegaNCT);   // shared memory is reused by the next op
    }
  }
}

template <int NB, int HD, int G, bool W4>
static cudaError_t mega_launch_t(const MegaParams& p, int n_sm, cudaStream_t st, bool* unsupported) {
  using Lay = MegaLayout<NB, HD, G, W4>;
  const size_t smem = Lay::total(p.kmax);
  if (Lay::stages(p.kmax) < 2 || smem > kMegaSmemLimit) {
    *unsupported = true;
    return cudaSuccess;
  }
  static int configured = 0;
  if (configured != static_cast<int>(smem)) {
    cudaError_t e = cudaFuncSetAttribute(mega_kernel<NB, HD, G, W4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mega_kernel<NB, HD, G, W4>, kGemvThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) {
      *unsupported = true;
      return cudaSuccess;
    }
    configured = static_cast<int>(smem);
  }
  MegaParams q = p;
  void* args[] = {&q};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(mega_kernel<NB, HD, G, W4>), dim3(n_sm),
                                     dim3(kGemvThreads), args, smem, st);
}

cudaError_t launch_mega(const MegaParams& p, int nb, int n_sm, cudaStream_t st, bool* unsupported) {
  *unsupported = false;
  const int hd = p.d.hd, G = p.d.Hq / p.d.Hkv;
  if (p.w4) {
    if (nb == 1 && hd == 128 && G == 4) return mega_launch_t<1, 128, 4, true>(p, n_sm, st, unsupported);
    if (nb == 2 && hd == 128 && G == 4) return mega_launch_t<2, 128, 4, true>(p, n_sm, st, unsupported);
    if (nb == 1 && hd == 64 && G == 2) return mega_launch_t<1, 64, 2, true>(p, n_sm, st, unsupported);
    if (nb == 2 && hd == 64 && G == 2) return mega_launch_t<2, 64, 2, true>(p, n_sm, st, unsupported);
    *unsupported = true;
    return cudaSuccess;
  }
  if (nb == 1 && hd == 128 && G == 4) return mega_launch_t<1, 128, 4, false>(p, n_sm, st, unsupported);
  if (nb == 2 && hd == 128 && G == 4) return mega_launch_t<2, 128, 4, false>(p, n_sm, st, unsupported);
  if (nb == 1 && hd == 64 && G == 2) return mega_launch_t<1, 64, 2, false>(p, n_sm, st, unsupported);
  if (nb == 2 && hd == 64 && G == 2) return mega_launch_t<2, 64, 2, false>(p, n_sm, st, unsupported);
  *unsupported = true;
  return cudaSuccess;
}

}  // namespace dualar
