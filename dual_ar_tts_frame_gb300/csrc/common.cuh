// Device-side helpers shared by the Dual-AR kernels (sm_103a).
//
// PTX wrappers for mbarriers and the bulk-copy engine (cp.async.bulk), bf16
// unpacking, warp/block reductions and bounded waits.  Every wait in this
// library gives up after a time limit, records an error code in the device
// error word and returns, so a missed arrival never hangs the GPU.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

#define DEVI __device__ __forceinline__

namespace dualar {

DEVI void raise_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

DEVI uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- tagged activations ----------------------------------------------------
// Inside the persistent frame kernel an activation value travels with the tag
// of the op that wrote it: one 64-bit word, the float in the low half and the
// tag in the high half, written and read as a single 8-byte access (so value
// and tag are seen together).  A reader spins on its own words until they
// carry the tag it expects; no grid-wide barrier and no fence is needed
// between the writer and the reader.  A tag is (launch epoch << 12) | index
// of the writing op, never 0.
constexpr uint64_t kAbortCheckNs = 10000;   // how often a long wait looks at the error word

DEVI uint32_t op_tag(uint32_t epoch, int op) { return (epoch << kTagOpBits) | static_cast<uint32_t>(op); }
DEVI uint64_t tag_pack(float v, uint32_t tag) {
  return (static_cast<uint64_t>(tag) << 32) | static_cast<uint64_t>(__float_as_uint(v));
}
DEVI uint32_t tag_of(uint64_t w) { return static_cast<uint32_t>(w >> 32); }
DEVI float tag_val(uint64_t w) { return __uint_as_float(static_cast<uint32_t>(w)); }

DEVI void tag_store(uint64_t* p, float v, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(tag_pack(v, tag)) : "memory");
}
// two consecutive words (16-byte aligned)
DEVI void tag_store2(uint64_t* p, float a, float b, uint32_t tag) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(tag_pack(a, tag)),
               "l"(tag_pack(b, tag))
               : "memory");
}
DEVI uint64_t tag_load(const uint64_t* p) {
  uint64_t w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
// two consecutive words (16-byte aligned); each word is read as one access
DEVI void tag_load2(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

// Bounded wait on n <= 8 tagged words: returns their values once every word
// carries `tag`.  Gives up (zeros, false) when the error word shows that
// another wait gave up, or after limit_ns, raising DEV_ERR_GRID_TIMEOUT.
template <int n>
DEVI bool tag_wait(const uint64_t* p, uint32_t tag, float (&v)[n], uint32_t* err, uint64_t limit_ns) {
  static_assert(n >= 1 && n <= 8, "tag_wait reads at most 8 words");
  uint64_t w[n];
  if (n % 2 == 0 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0) {
#pragma unroll
    for (int q = 0; q < n / 2; ++q) tag_load2(p + 2 * q, w[2 * q], w[2 * q + 1]);
  } else {
#pragma unroll
    for (int q = 0; q < n; ++q) w[q] = tag_load(p + q);
  }
  bool ok = true;
#pragma unroll
  for (int q = 0; q < n; ++q) ok = ok && tag_of(w[q]) == tag;
  if (!ok) {
    const uint64_t t0 = global_timer_ns();
    uint64_t next_chk = kAbortCheckNs;
    while (true) {
      ok = true;
#pragma unroll
      for (int q = 0; q < n; ++q) {
        if (tag_of(w[q]) != tag) w[q] = tag_load(p + q);
        ok = ok && tag_of(w[q]) == tag;
      }
      if (ok) break;
      const uint64_t dt = global_timer_ns() - t0;
      if (dt > next_chk) {
        // another wait gave up: give up too (looked at every kAbortCheckNs)
        next_chk = dt + kAbortCheckNs;
        if (*reinterpret_cast<const volatile uint32_t*>(err) & (DEV_ERR_GRID_TIMEOUT | DEV_ERR_MBAR_TIMEOUT)) break;
      }
      if (dt > limit_ns) {
        raise_error(err, DEV_ERR_GRID_TIMEOUT);
        break;
      }
    }
    if (!ok) {
#pragma unroll
      for (int q = 0; q < n; ++q) v[q] = 0.f;
      return false;
    }
  }
#pragma unroll
  for (int q = 0; q < n; ++q) v[q] = tag_val(w[q]);
  return true;
}

DEVI float tag_wait1(const uint64_t* p, uint32_t tag, uint32_t* err, uint64_t limit_ns) {
  float v[1];
  tag_wait<1>(p, tag, v, err, limit_ns);
  return v[0];
}

// ---- shared-memory addresses and mbarriers ---------------------------------
DEVI uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared (through L2), completed by
// cp_async_wait_all in the issuing thread
DEVI void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}
DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
DEVI void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization (launch_pdl) may start while the kernel before it in the
// stream still runs: pdl_wait() blocks until that kernel has completed and
// its writes are visible (a no-op after a normal launch), so every kernel
// calls it before touching memory that an earlier kernel writes or reads,
// and every CTA calls it before it exits (so that a kernel's completion
// implies its predecessor's).  pdl_launch() lets the next kernel start.
DEVI void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DEVI void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

DEVI void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

DEVI void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

DEVI void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

DEVI bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; gives up after
// limit_ns, raising DEV_ERR_MBAR_TIMEOUT.  Returns false on timeout.
DEVI bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* err, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      raise_error(err, DEV_ERR_MBAR_TIMEOUT);
      return false;
    }
  }
}

// One bulk copy global -> shared (no tensor map), completing on an mbarrier
// with a transaction count.  dst/src 16-byte aligned, bytes a multiple of 16.
// The L2 policy marks the source lines evict-first: weights are streamed
// once per use and should not push activations or KV out of L2.
DEVI void bulk_load_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                        uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Same without an L2 policy (data that is worth keeping in L2).
DEVI void bulk_load_g2s_plain(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

DEVI uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
DEVI uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Named barrier over a subset of the block's warps (the consumer warps).
DEVI void named_barrier(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

DEVI uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Release-ordered add at GPU scope (cumulative: writes this thread observed
// before it, e.g. through a CTA barrier, are ordered before the add).
DEVI void red_release_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Prefetch [src, src+bytes) into L2 (bulk, asynchronous, no completion
// tracking).  src 16-byte aligned, bytes a multiple of 16.
DEVI void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

DEVI uint32_t atomic_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// ---- bf16 ------------------------------------------------------------------
// Two bf16 packed in a 32-bit word -> two floats (exact widening).
DEVI float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
DEVI float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
DEVI float bf16bits_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
DEVI uint16_t f32_to_bf16bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// 8 bf16 (one 16-byte vector) dotted with 8 floats.
DEVI float dot8(const uint4 w, const float4 a, const float4 b, float acc) {
  acc = fmaf(bf16lo(w.x), a.x, acc);
  acc = fmaf(bf16hi(w.x), a.y, acc);
  acc = fmaf(bf16lo(w.y), a.z, acc);
  acc = fmaf(bf16hi(w.y), a.w, acc);
  acc = fmaf(bf16lo(w.z), b.x, acc);
  acc = fmaf(bf16hi(w.z), b.y, acc);
  acc = fmaf(bf16lo(w.w), b.z, acc);
  acc = fmaf(bf16hi(w.w), b.w, acc);
  return acc;
}

// ---- reductions --------------------------------------------------------------
DEVI float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

DEVI float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

DEVI float silu(float g) { return g / (1.0f + expf(-g)); }

}  // namespace dualar
