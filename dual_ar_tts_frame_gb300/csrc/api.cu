// Host runtime of libdualar.so: the C ABI declared in include/dualar.h.
//
// Owns the KV page pool and per-slot state, allocates pages on the host
// (lowest free page first), and queues the kernels of a prefill or a frame
// on the handle's stream.  Kernels are in kernels.cu.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <set>
#include <string>
#include <vector>

#include "dualar.h"
#include "internal.h"
#include "mega.h"
#include "tcgemm.h"

using namespace dualar;

struct dualar_handle {
  dualar_config cfg{};
  dualar_weights w{};
  std::vector<dualar_layer_weights> slow, fast;
  cudaStream_t stream = nullptr;
  int device = 0;
  int n_sm = 0;
  DevPtrs d{};
  std::vector<void*> allocs;
  // host mirrors
  std::vector<int> length;               // next position per slot, -1 = empty
  std::vector<std::vector<int>> pages;   // pages per slot
  std::set<int> free_pages;
  std::vector<int> page_refs;            // slots whose page table holds each page (shared prefixes)
  LaunchSetup setup{};                   // the setup kernel's argument, filled per launch sequence
  std::vector<char> prefix_only;         // slot holds a shared prefix without its prompt's end
  std::string err;
  int launches = 0;
  // GEMV timing (dualar_profile)
  bool profiling = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  std::vector<double> prof_bytes;
  // persistent frame kernel
  bool use_mega = true;
  bool use_tc = true;            // dualar_set_tensor_cores
  TcBuffers tc{};                // tensor-core projection buffers
  const float* tc_ready_x = nullptr;   // the tc buffers hold the halves of this [nb][K] input
  int tc_ready_k = 0, tc_ready_nb = 0;
  TcPending tc_pend;             // a residual-add reduce not yet queued (see run_gemv)
  uint32_t bar_extra = 0;
  uint32_t* bar_counter = nullptr;
  uint64_t* tagged = nullptr;    // the tagged work buffers (one region)
  size_t tagged_words = 0;
  uint32_t epoch = 0;            // tag epoch of the last persistent launch
  uint64_t prefetch_bytes = 65536;   // dualar_set_prefetch
  uint64_t* trace = nullptr;     // dualar_set_trace
  int64_t trace_bytes = 0;
  MegaOp* mega_ops[3] = {nullptr, nullptr, nullptr};
  ProdOp* mega_prod[3] = {nullptr, nullptr, nullptr};   // GEMV ops of each program, for the producer
  int mega_nprod[3] = {0, 0, 0};   // programs for batch 1, 2
  int mega_nops[3] = {0, 0, 0};
  bool mega_unsupported[3] = {false, false, false};
  // packed 4-bit projections (dualar_set_w4a16); empty: all bf16
  std::vector<dualar_w4a16_layer> slow_q, fast_q;
  bool any_w4 = false;
  // bf16 copy of one packed projection (a SwiGLU pair: both) for the
  // tensor-core path at 9+ rows; sized for the largest packed projection
  uint16_t* w4_bf16 = nullptr;
  size_t w4_bf16_elems = 0;
};

namespace {

void set_err(dualar_handle* h, const char* fmt, ...) {
  if (!h) return;
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  h->err = buf;
}

// The lowest free page, now held by one slot.
int take_page(dualar_handle* h) {
  const int pg = *h->free_pages.begin();
  h->free_pages.erase(h->free_pages.begin());
  h->page_refs[pg] = 1;
  return pg;
}

// One slot fewer holds the page; the last one returns it to the pool.
void drop_page(dualar_handle* h, int pg) {
  if (--h->page_refs[pg] == 0) h->free_pages.insert(pg);
}

// Queues the deferred residual-add reduce, if any.
int flush_tc(dualar_handle* h) {
  if (!h->tc_pend.on) return DUALAR_OK;
  h->tc_pend.on = false;
  ++h->launches;
  const cudaError_t e = launch_tc_pending(h->tc_pend, h->tc, h->n_sm, h->stream);
  if (e != cudaSuccess) {
    set_err(h, "tensor-core reduce failed: %s", cudaGetErrorString(e));
    return DUALAR_ERR_CUDA;
  }
  return DUALAR_OK;
}

// Every stream operation first queues a deferred reduce (flush_tc), so that
// nothing can read the residual stream before it is written.
#define CUDA_TRY(h, call)                                                               \
  do {                                                                                  \
    if (const int frc_ = flush_tc(h)) return frc_;                                      \
    cudaError_t e_ = (call);                                                            \
    if (e_ != cudaSuccess) {                                                            \
      set_err(h, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
      return DUALAR_ERR_CUDA;                                                           \
    }                                                                                   \
  } while (0)

#define LAUNCH(h, call)                                                                 \
  do {                                                                                  \
    if (const int frc_ = flush_tc(h)) return frc_;                                      \
    cudaError_t e_ = (call);                                                            \
    ++(h)->launches;                                                                    \
    if (e_ != cudaSuccess) {                                                            \
      set_err(h, "launch %s failed: %s", #call, cudaGetErrorString(e_));                \
      return DUALAR_ERR_CUDA;                                                           \
    }                                                                                   \
  } while (0)

template <typename T>
int dev_alloc(dualar_handle* h, T** p, size_t count) {
  void* q = nullptr;
  const size_t bytes = std::max<size_t>(count * sizeof(T), 256);
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) {
    set_err(h, "cudaMalloc(%zu bytes) failed: %s", bytes, cudaGetErrorString(e));
    return DUALAR_ERR_CUDA;
  }
  h->allocs.push_back(q);
  e = cudaMemsetAsync(q, 0, bytes, h->stream);
  if (e != cudaSuccess) {
    set_err(h, "cudaMemsetAsync failed: %s", cudaGetErrorString(e));
    return DUALAR_ERR_CUDA;
  }
  *p = static_cast<T*>(q);
  return DUALAR_OK;
}

// float -> bf16 bits, round to nearest even (host).
uint16_t host_f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return static_cast<uint16_t>(u >> 16);  // inf / nan
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_layer(dualar_handle* h, const dualar_layer_weights& l, bool qk, const char* which, int i) {
  const void* ptrs[] = {l.attn_norm, l.wqkv, l.wo, l.ffn_norm, l.w_gate, l.w_up, l.w_down};
  for (const void* p : ptrs) {
    if (!p || !aligned16(p)) {
      set_err(h, "%s layer %d: a weight pointer is NULL or not 16-byte aligned", which, i);
      return DUALAR_ERR_INVALID_ARG;
    }
  }
  if (qk && (!l.q_norm || !l.k_norm)) {
    set_err(h, "%s layer %d: qk-norm enabled but q_norm/k_norm missing", which, i);
    return DUALAR_ERR_INVALID_ARG;
  }
  return DUALAR_OK;
}

int validate_config(dualar_handle* h, const dualar_config& c) {
  auto bad = [&](const char* what) {
    set_err(h, "invalid config: %s", what);
    return DUALAR_ERR_INVALID_ARG;
  };
  if (c.dim <= 0 || c.dim % 8) return bad("dim must be a positive multiple of 8");
  if (c.ffn <= 0 || c.ffn % 8) return bad("ffn must be a positive multiple of 8");
  if (c.head_dim != 64 && c.head_dim != 128) return bad("head_dim must be 64 or 128");
  if (c.n_head <= 0 || c.n_kv_head <= 0 || c.n_head % c.n_kv_head) return bad("heads");
  const int g = c.n_head / c.n_kv_head;
  if (g != 1 && g != 2 && g != 4 && g != 8) return bad("n_head / n_kv_head must be 1, 2, 4 or 8");
  if (c.n_layer <= 0 || c.fast_n_layer <= 0) return bad("layer counts");
  if (c.page_tokens != 64) return bad("page_tokens must be 64");
  if (c.n_codebooks < 2 || c.n_codebooks > kMaxCodebooks) return bad("n_codebooks in [2, 16]");
  if (c.n_sem <= 0 || c.n_sem > 4096) return bad("n_sem in [1, 4096]");
  if (c.fast_vocab <= 0 || c.fast_vocab > 4096) return bad("fast_vocab in [1, 4096]");
  if (c.sem_begin < 0 || c.sem_begin + c.n_sem > c.vocab) return bad("semantic id range");
  if (c.im_end_id < 0 || c.im_end_id >= c.vocab ||
      (c.im_end_id >= c.sem_begin && c.im_end_id < c.sem_begin + c.n_sem))
    return bad("im_end_id must be a non-semantic id");
  if (c.max_seqs <= 0 || c.max_seqs > kMaxRows) return bad("max_seqs in [1, 128]");
  if (c.max_pages <= 0) return bad("max_pages");
  if (c.max_ctx <= 0 || (c.max_ctx + 63) / 64 > kMaxChunks * 1024) return bad("max_ctx");
  if (!(c.norm_eps > 0.f) || !(c.rope_base > 1.f)) return bad("norm_eps / rope_base");
  if ((c.n_head * c.head_dim) % 8) return bad("n_head * head_dim");
  return DUALAR_OK;
}

// ---- launch helpers --------------------------------------------------------
GemvArgs gemv_base(dualar_handle* h) {
  GemvArgs a{};
  a.eps = h->cfg.norm_eps;
  a.err = h->d.err;
  a.wait_limit_ns = h->d.wait_limit_ns;
  a.x_src = a.base_src = a.out_src = -1;
  return a;
}

double gemv_bytes(const GemvArgs& a) {
  const double rows = (a.mode == GEMV_SWIGLU) ? 2.0 * a.n0 : static_cast<double>(a.n0 + a.n1);
  const double out_rows = (a.mode == GEMV_SWIGLU) ? a.n0 : a.n0 + a.n1;
  double b = rows * (a.w4 ? static_cast<double>(w4_row_bytes(a.K)) : a.K * 2.0);   // weights
  b += static_cast<double>(a.nb) * a.K * 4.0;        // x
  if (a.norm_w) b += a.K * 2.0;                      // norm gain
  b += static_cast<double>(a.nb) * out_rows * 4.0;   // y
  if (a.mode == GEMV_ADD) b += static_cast<double>(a.nb) * out_rows * 4.0;   // residual base
  return b;
}

cudaEvent_t next_event(dualar_handle* h) {
  if (h->ev_used == h->ev_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    h->ev_pool.push_back(e);
  }
  return h->ev_pool[h->ev_used++];
}

int run_gemv(dualar_handle* h, GemvArgs a) {
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (h->profiling) {
    e0 = next_event(h);
    e1 = next_event(h);
    if (!e0 || !e1) {
      set_err(h, "cudaEventCreate failed");
      return DUALAR_ERR_CUDA;
    }
    CUDA_TRY(h, cudaEventRecord(e0, h->stream));
  }
  // packed 4-bit weights at 9+ rows: expanded to exact bf16 hi/lo pairs
  // (one pass over the packed bytes, launched plainly after everything
  // before it) and multiplied on the tensor cores over 2K columns, instead
  // of GEMV passes of 8 rows; that GEMM is launched plainly too, since it
  // fetches weights before waiting for its predecessor
  bool weights_pdl = true, w_hilo = false;
  if (a.w4 && h->use_tc && h->w4_bf16 && a.nb >= kTcMinRows && a.nb <= kTcMaxRows) {
    GemvArgs t = a;
    t.w4 = 0;
    t.w0 = h->w4_bf16;
    t.w1 = a.n1 > 0 ? h->w4_bf16 + static_cast<size_t>(a.n0) * 2 * a.K : nullptr;
    if (static_cast<size_t>(a.n0 + a.n1) * 2 * a.K <= h->w4_bf16_elems && tc_eligible(t, h->tc.ldx)) {
      LAUNCH(h, launch_dequant_w4(a.w0, a.n0, a.K, h->w4_bf16, h->stream));
      if (a.n1 > 0) LAUNCH(h, launch_dequant_w4(a.w1, a.n1, a.K, const_cast<uint16_t*>(t.w1), h->stream));
      a = t;
      weights_pdl = false;
      w_hilo = true;
    }
  }
  if (!a.w4 && h->use_tc && tc_eligible(a, h->tc.ldx)) {
    // 9..128 rows: one pass over the weights on the tensor cores.  The
    // SwiGLU output feeds the down projection without norm: its reduce
    // writes the halves the next GEMM reads, and that split is skipped.
    // A residual-add projection's reduce waits for the next projection: if
    // that one normalises the residual stream, reduce, norm and split run
    // as one kernel.
    int n = 0;
    bool fused = false;
    if (h->tc_pend.on && tc_can_fuse(h->tc_pend, a)) {
      h->tc_pend.on = false;
      ++n;
      const cudaError_t ef = launch_tc_reduce_norm(h->tc_pend, a, h->tc, h->stream);
      if (ef != cudaSuccess) {
        set_err(h, "tensor-core reduce failed: %s", cudaGetErrorString(ef));
        return DUALAR_ERR_CUDA;
      }
      fused = true;
    } else if (const int frc = flush_tc(h)) {
      return frc;
    }
    const bool ready = fused || (h->tc_ready_x == a.x && h->tc_ready_k == a.K && h->tc_ready_nb == a.nb &&
                                 a.ldx == a.K && a.norm_w == nullptr && a.save_x == nullptr);
    const bool split_out = a.mode == GEMV_SWIGLU && a.out_map == nullptr && a.ldo == a.n0;
    h->tc_ready_x = nullptr;
    const cudaError_t e =
        launch_tc_gemm(a, h->tc, h->n_sm, h->stream, &n, ready, split_out, &h->tc_pend, weights_pdl, w_hilo);
    if (e == cudaSuccess && split_out) {
      h->tc_ready_x = a.out;
      h->tc_ready_k = a.n0;
      h->tc_ready_nb = a.nb;
    }
    h->launches += n;
    if (e != cudaSuccess) {
      set_err(h, "tensor-core projection failed: %s", cudaGetErrorString(e));
      return DUALAR_ERR_CUDA;
    }
  } else {
    h->tc_ready_x = nullptr;
    LAUNCH(h, launch_gemv(a, h->n_sm, h->stream));
  }
  if (h->profiling) {
    CUDA_TRY(h, cudaEventRecord(e1, h->stream));
    h->prof_bytes.push_back(gemv_bytes(a));
  }
  return DUALAR_OK;
}

#define TRY(x)                    \
  do {                            \
    int rc_ = (x);                \
    if (rc_ != DUALAR_OK) return rc_; \
  } while (0)

const uint16_t* U16(const void* p) { return static_cast<const uint16_t*>(p); }

// GEMV arguments of the four projections of a block and of the heads.
GemvArgs args_qkv(dualar_handle* h, const dualar_layer_weights& lw, int nrows, const float* xin) {
  GemvArgs a = gemv_base(h);
  a.w0 = U16(lw.wqkv);
  a.n0 = h->d.qkv_dim;
  a.K = h->cfg.dim;
  a.mode = GEMV_STORE;
  a.nb = nrows;
  a.x = xin;
  a.ldx = h->cfg.dim;
  a.norm_w = U16(lw.attn_norm);
  a.out = h->d.qkv;
  a.ldo = h->d.qkv_dim;
  return a;
}

GemvArgs args_o(dualar_handle* h, const dualar_layer_weights& lw, int nrows, const float* base, float* out) {
  const int qd = h->cfg.n_head * h->cfg.head_dim;
  GemvArgs a = gemv_base(h);
  a.w0 = U16(lw.wo);
  a.n0 = h->cfg.dim;
  a.K = qd;
  a.mode = GEMV_ADD;
  a.nb = nrows;
  a.x = h->d.attn;
  a.ldx = qd;
  a.base = base;
  a.ldb = h->cfg.dim;
  a.out = out;
  a.ldo = h->cfg.dim;
  return a;
}

GemvArgs args_gateup(dualar_handle* h, const dualar_layer_weights& lw, int nrows, const float* hres) {
  GemvArgs a = gemv_base(h);
  a.w0 = U16(lw.w_gate);
  a.w1 = U16(lw.w_up);
  a.n0 = h->cfg.ffn;
  a.n1 = h->cfg.ffn;
  a.K = h->cfg.dim;
  a.mode = GEMV_SWIGLU;
  a.nb = nrows;
  a.x = hres;
  a.ldx = h->cfg.dim;
  a.norm_w = U16(lw.ffn_norm);
  a.out = h->d.act;
  a.ldo = h->cfg.ffn;
  return a;
}

GemvArgs args_down(dualar_handle* h, const dualar_layer_weights& lw, int nrows, float* hres) {
  GemvArgs a = gemv_base(h);
  a.w0 = U16(lw.w_down);
  a.n0 = h->cfg.dim;
  a.K = h->cfg.ffn;
  a.mode = GEMV_ADD;
  a.nb = nrows;
  a.x = h->d.act;
  a.ldx = h->cfg.ffn;
  a.base = hres;
  a.ldb = h->cfg.dim;
  a.out = hres;
  a.ldo = h->cfg.dim;
  return a;
}

GemvArgs args_fast_head(dualar_handle* h, int nrows) {
  GemvArgs a = gemv_base(h);
  a.w0 = U16(h->w.fast_out);
  a.n0 = h->cfg.fast_vocab;
  a.K = h->cfg.dim;
  a.mode = GEMV_STORE;
  a.nb = nrows;
  a.x = h->d.hf;
  a.ldx = h->cfg.dim;
  a.norm_w = U16(h->w.fast_norm);
  a.out = h->d.logits;
  a.ldo = h->d.logit_ld;
  return a;
}

// Final RMSNorm + restricted head for rows [r0, r0 + n): commits the normed
// hidden state and the logits of rows whose commit_map entry is a slot.
// [P2] "Two autoregressions" (bias keeps semantic ids + <|im_end|>) and "The
// slow AR is Qwen3-4B" (tied head): only those 4,097 rows are computed.
GemvArgs args_head(dualar_handle* h, int r0, int n) {
  const dualar_config& c = h->cfg;
  GemvArgs a = gemv_base(h);
  a.w0 = U16(h->w.tok_emb) + static_cast<size_t>(c.sem_begin) * c.dim;
  a.n0 = c.n_sem;
  a.w1 = U16(h->w.tok_emb) + static_cast<size_t>(c.im_end_id) * c.dim;
  a.n1 = 1;
  a.K = c.dim;
  a.mode = GEMV_STORE;
  a.nb = n;
  a.x = h->d.hs + static_cast<size_t>(r0) * c.dim;
  a.ldx = c.dim;
  a.norm_w = U16(h->w.final_norm);
  a.out = h->d.z_last;
  a.ldo = c.n_sem + 1;
  a.out_map = h->d.commit_map + r0;
  a.save_x = h->d.h_last;
  a.save_map = h->d.commit_map + r0;
  a.lds = c.dim;
  return a;
}

// One transformer block over nrows rows.  Slow blocks attend over the paged
// cache; fast blocks over the per-frame codebook cache.
// The packed 4-bit form of a projection, when dualar_set_w4a16 gave one.
GemvArgs packed(GemvArgs a, const void* q0, const void* q1 = nullptr) {
  if (q0 != nullptr) {
    a.w0 = U16(q0);
    if (q1 != nullptr) a.w1 = U16(q1);
    a.w4 = 1;
  }
  return a;
}

// The packed projections of a block (all NULL when none were given).
const dualar_w4a16_layer& packed_or_none(const dualar_handle* h, bool fast, int layer) {
  static const dualar_w4a16_layer kNone{};
  const std::vector<dualar_w4a16_layer>& v = fast ? h->fast_q : h->slow_q;
  return v.empty() ? kNone : v[layer];
}

int block(dualar_handle* h, const dualar_layer_weights& lw, int layer, bool fast, int nrows,
          const float* xin, float* hres, int fast_pos, int units, int chunk, bool fuse_append) {
  const dualar_config& c = h->cfg;
  const DevPtrs& d = h->d;
  const dualar_w4a16_layer& lq = packed_or_none(h, fast, layer);
  // decode: the attention writes the bf16 halves of its output for the o
  // projection (no split kernel between them)
  TRY(run_gemv(h, packed(args_qkv(h, lw, nrows, xin), lq.wqkv)));
  AttnHalves hv{nullptr, nullptr, 0};
  const GemvArgs ao = packed(args_o(h, lw, nrows, xin, hres), lq.wo);
  const bool o_halves =
      (fast || fuse_append) && h->use_tc && !h->profiling && !ao.w4 && tc_eligible(ao, h->tc.ldx);
  if (o_halves) hv = AttnHalves{h->tc.xh, h->tc.xl, h->tc.ldx};
  bool halves_written = false;
  const bool qk = fast ? c.fast_qk_norm : c.slow_qk_norm;
  const uint16_t* qn = qk ? U16(lw.q_norm) : nullptr;
  const uint16_t* kn = qk ? U16(lw.k_norm) : nullptr;
  if (fast) {
    LAUNCH(h, launch_attn_fast(d, nrows, layer, fast_pos, qn, kn, h->stream, hv));
    halves_written = o_halves;
  } else if (fuse_append) {
    bool mma = false;
    LAUNCH(h, launch_attn_paged(d, nrows, layer, units, chunk, h->n_sm, true, qn, kn, h->stream, &mma, hv));
    halves_written = o_halves && mma;   // (the SIMT kernel writes no halves)
  } else {
    LAUNCH(h, launch_append(d, nrows, layer, false, 0, qn, kn, h->stream));
    LAUNCH(h, launch_attn_paged(d, nrows, layer, units, chunk, h->n_sm, false, nullptr, nullptr, h->stream));
  }
  if (halves_written) {
    h->tc_ready_x = ao.x;
    h->tc_ready_k = ao.K;
    h->tc_ready_nb = ao.nb;
  }
  TRY(run_gemv(h, ao));
  TRY(run_gemv(h, packed(args_gateup(h, lw, nrows, hres), lq.w_gate, lq.w_up)));
  return run_gemv(h, packed(args_down(h, lw, nrows, hres), lq.w_down));
}

// The frame program of the persistent kernel for batch nb (same op order as
// the per-op path in decode_impl).  Activations go through the tagged
// buffers; each read names the op that wrote the version it needs.
int build_mega_program(dualar_handle* h, int nb) {
  const dualar_config& c = h->cfg;
  const DevPtrs& d = h->d;
  std::vector<MegaOp> ops;
  auto F = [](uint64_t* p) { return reinterpret_cast<float*>(p); };
  auto op = [&](int type, int layer, int pos, int in_src) {
    MegaOp o{};
    o.type = type;
    o.layer = layer;
    o.pos = pos;
    o.in_src = in_src;
    return o;
  };
  // appends op o and returns its index (the tag its outputs carry)
  auto push = [&](const MegaOp& o) {
    ops.push_back(o);
    return static_cast<int>(ops.size()) - 1;
  };
  auto gemv = [&](GemvArgs a, float* x, int x_src, float* base, int base_src, float* out, bool tagged_out) {
    a.x = x;
    a.x_src = x_src;
    if (a.mode == GEMV_ADD) {
      a.base = base;
      a.base_src = base_src;
    }
    const int idx = static_cast<int>(ops.size());
    if (tagged_out) {
      a.out = out;
      a.out_src = idx;
    }
    MegaOp o = op(MOP_GEMV, 0, 0, -1);
    o.g = a;
    return push(o);
  };
  auto attn_op = [&](int type, int layer, int pos, int qkv_src, bool qk, const dualar_layer_weights& lw) {
    MegaOp a = op(type, layer, pos, qkv_src);
    a.q_norm = qk ? U16(lw.q_norm) : nullptr;
    a.k_norm = qk ? U16(lw.k_norm) : nullptr;
    return push(a);
  };
  const size_t D = c.dim;
  int fin_src[kMaxCodebooks];
  fin_src[0] = fin_src[1] = push(op(MOP_SAMPLE_Q0, 0, 0, -1));   // writes the inputs of passes 0 and 1
  int hf_src = -1;
  for (int p = 0; p < c.n_codebooks; ++p) {
    float* xin = F(d.fin_t + static_cast<size_t>(p) * kTaggedRows * D);
    for (int l = 0; l < c.fast_n_layer; ++l) {
      const dualar_layer_weights& lw = h->fast[l];
      const dualar_w4a16_layer& lq = packed_or_none(h, true, l);
      float* x = l == 0 ? xin : F(d.hf_t);
      const int x_src = l == 0 ? fin_src[p] : hf_src;
      const int qkv = gemv(packed(args_qkv(h, lw, nb, nullptr), lq.wqkv), x, x_src, nullptr, -1, F(d.qkv_t), true);
      const int at = attn_op(MOP_ATTN_FAST, l, p, qkv, c.fast_qk_norm, lw);
      hf_src = gemv(packed(args_o(h, lw, nb, nullptr, nullptr), lq.wo), F(d.attn_t), at, x, x_src, F(d.hf_t), true);
      ops[hf_src].g.x_scout = c.head_dim;   // one sentinel per query head
      const int act = gemv(packed(args_gateup(h, lw, nb, nullptr), lq.w_gate, lq.w_up), F(d.hf_t), hf_src,
                           nullptr, -1, F(d.act_t), true);
      hf_src = gemv(packed(args_down(h, lw, nb, nullptr), lq.w_down), F(d.act_t), act, F(d.hf_t), hf_src,
                    F(d.hf_t), true);
    }
    if (p == 0) continue;
    const int head = gemv(args_fast_head(h, nb), F(d.hf_t), hf_src, nullptr, -1, F(d.logits_t), true);
    const int smp = push(op(MOP_SAMPLE_FAST, 0, p, head));
    if (p + 1 < c.n_codebooks) fin_src[p + 1] = smp;
  }
  int hs_src = push(op(MOP_FUSION, 0, 0, -1));
  for (int l = 0; l < c.n_layer; ++l) {
    const dualar_layer_weights& lw = h->slow[l];
    const dualar_w4a16_layer& lq = packed_or_none(h, false, l);
    float* x = l == 0 ? F(d.xs_t) : F(d.hs_t);
    const int x_src = hs_src;
    const int qkv = gemv(packed(args_qkv(h, lw, nb, nullptr), lq.wqkv), x, x_src, nullptr, -1, F(d.qkv_t), true);
    const int at = attn_op(MOP_ATTN_PAGED, l, 0, qkv, c.slow_qk_norm, lw);
    hs_src = gemv(packed(args_o(h, lw, nb, nullptr, nullptr), lq.wo), F(d.attn_t), at, x, x_src, F(d.hs_t), true);
    ops[hs_src].g.x_scout = c.head_dim;
    const int act = gemv(packed(args_gateup(h, lw, nb, nullptr), lq.w_gate, lq.w_up), F(d.hs_t), hs_src, nullptr,
                         -1, F(d.act_t), true);
    hs_src = gemv(packed(args_down(h, lw, nb, nullptr), lq.w_down), F(d.act_t), act, F(d.hs_t), hs_src, F(d.hs_t),
                  true);
  }
  // the head writes the held state (plain buffers, read by the host and the
  // next launch)
  gemv(args_head(h, 0, nb), F(d.hs_t), hs_src, nullptr, -1, nullptr, false);
  if (ops.size() >= (1u << kTagOpBits)) {
    h->mega_unsupported[nb] = true;   // op indices do not fit the tag
    return DUALAR_OK;
  }
  std::vector<ProdOp> prod;
  for (const MegaOp& o : ops)
    if (o.type == MOP_GEMV) prod.push_back(ProdOp{o.g.w0, o.g.w1, o.g.n0, o.g.n1, o.g.K, o.g.mode, o.g.w4});
  MegaOp* dev = nullptr;
  CUDA_TRY(h, cudaMalloc(&dev, ops.size() * sizeof(MegaOp)));
  h->allocs.push_back(dev);
  CUDA_TRY(h, cudaMemcpy(dev, ops.data(), ops.size() * sizeof(MegaOp), cudaMemcpyHostToDevice));
  ProdOp* pdev = nullptr;
  CUDA_TRY(h, cudaMalloc(&pdev, std::max<size_t>(prod.size(), 1) * sizeof(ProdOp)));
  h->allocs.push_back(pdev);
  CUDA_TRY(h, cudaMemcpy(pdev, prod.data(), prod.size() * sizeof(ProdOp), cudaMemcpyHostToDevice));
  h->mega_ops[nb] = dev;
  h->mega_nops[nb] = static_cast<int>(ops.size());
  h->mega_prod[nb] = pdev;
  h->mega_nprod[nb] = static_cast<int>(prod.size());
  return DUALAR_OK;
}

// Split-KV work list: chunk size and per-row first unit.
// Chunks are as short as possible (one page) while the batch's (row, KV
// head, page) count is small -- a decode step of one or two sequences needs
// every unit it can get -- and grow once there are more pages than about
// eight units per SM, so that a unit streams several pages (double-buffered)
// instead of paying a page's latency per unit.
void plan_attention(dualar_handle* h, LaunchSetup& s, int* units, int* chunk) {
  int max_len = 0;
  long long page_units = 0;
  const int pt = h->cfg.page_tokens;
  for (int r = 0; r < s.n_rows; ++r) {
    max_len = std::max(max_len, s.rows[r].pos + 1);
    page_units += static_cast<long long>(h->cfg.n_kv_head) * ((s.rows[r].pos + 1 + pt - 1) / pt);
  }
  const int pages = (max_len + pt - 1) / pt;
  const long long target = 8LL * h->n_sm;
  const int ppc = std::max(std::max(1, (pages + kMaxChunks - 1) / kMaxChunks),
                           std::min(kMaxChunkPages, static_cast<int>(page_units / target)));
  *chunk = ppc * pt;
  int u = 0;
  for (int r = 0; r < s.n_rows; ++r) {
    s.rows[r].unit0 = u;
    u += h->cfg.n_kv_head * ((s.rows[r].pos + 1 + *chunk - 1) / *chunk);
  }
  *units = u;
}

// Decode rows are distinct sequences, so the KV append fuses into attention;
// prefill rows of one sequence must see each other's KV (separate append).
int slow_stack(dualar_handle* h, int nrows, int units, int chunk, bool decode) {
  for (int l = 0; l < h->cfg.n_layer; ++l)
    TRY(block(h, h->slow[l], l, false, nrows, l == 0 ? h->d.xs : h->d.hs, h->d.hs, 0, units, chunk,
              decode));
  return DUALAR_OK;
}

int decode_impl(dualar_handle* h, int32_t batch, const int32_t* slots, const float* uniforms,
                const dualar_sampling* smp, const int32_t* forced, int32_t* codes, int32_t* status,
                float* slow_logits, float* fast_logits, int32_t* draws, bool per_op_only = false) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  const dualar_config& c = h->cfg;
  if (batch < 1 || batch > c.max_seqs) {
    set_err(h, "batch %d outside [1, %d]", batch, c.max_seqs);
    return DUALAR_ERR_INVALID_ARG;
  }
  if (!slots || !uniforms || !smp || !codes || !status) {
    set_err(h, "decode: NULL argument");
    return DUALAR_ERR_INVALID_ARG;
  }
  if (!(smp->temperature >= 0.f) || !(smp->top_p > 0.f && smp->top_p <= 1.f) || smp->ras_win < 0 ||
      smp->ras_win > kRasRing || !(smp->ras_temperature >= 0.f) ||
      !(smp->ras_top_p > 0.f && smp->ras_top_p <= 1.f)) {
    set_err(h, "decode: invalid sampling parameters");
    return DUALAR_ERR_INVALID_ARG;
  }
  std::vector<char> seen(c.max_seqs, 0);
  int need = 0;
  for (int r = 0; r < batch; ++r) {
    const int s = slots[r];
    if (s < 0 || s >= c.max_seqs || seen[s]) {
      set_err(h, "decode: slot %d invalid or repeated", s);
      return DUALAR_ERR_INVALID_ARG;
    }
    seen[s] = 1;
    if (h->length[s] < 0) {
      set_err(h, "decode: slot %d is empty", s);
      return DUALAR_ERR_SLOT_EMPTY;
    }
    if (h->prefix_only[s]) {
      set_err(h, "decode: slot %d holds a shared prefix; append the rest of its prompt first", s);
      return DUALAR_ERR_INVALID_ARG;
    }
    if (h->length[s] >= c.max_ctx) {
      set_err(h, "decode: slot %d reached max_ctx %d", s, c.max_ctx);
      return DUALAR_ERR_CONTEXT_FULL;
    }
    if (h->length[s] % c.page_tokens == 0) ++need;
  }
  if (need > static_cast<int>(h->free_pages.size())) {
    set_err(h, "decode: %d pages needed, %zu free", need, h->free_pages.size());
    return DUALAR_ERR_OOM_PAGES;
  }
  LaunchSetup& s = h->setup;   // large; filled per call, copied into the launch
  std::memset(&s, 0, sizeof(s));
  s.n_rows = batch;
  s.commit_last_only = 0;
  s.embed = 0;
  for (int r = 0; r < batch; ++r) {
    const int sl = slots[r];
    const int pos = h->length[sl];
    s.rows[r] = RowInfo{sl, pos, 1, 0};
    if (pos % c.page_tokens == 0) {
      const int pg = take_page(h);
      h->pages[sl].push_back(pg);
      s.upd_slot[s.n_updates] = sl;
      s.upd_index[s.n_updates] = pos / c.page_tokens;
      s.upd_page[s.n_updates] = pg;
      ++s.n_updates;
    }
  }
  int units = 0, chunk = 0;
  plan_attention(h, s, &units, &chunk);
  h->launches = 0;
  const DevPtrs& d = h->d;
  SamplingParams sp{smp->temperature, smp->top_p, smp->ras_win, smp->ras_temperature,
                    smp->ras_top_p, smp->allow_eos};
  const int N = c.n_codebooks;
  LAUNCH(h, launch_setup(s, d, U16(h->w.tok_emb), h->stream));
  if (!per_op_only && h->use_mega && batch <= kTaggedRows && !h->mega_unsupported[batch] && !h->mega_ops[batch])
    TRY(build_mega_program(h, batch));
  if (!per_op_only && h->use_mega && batch <= kTaggedRows && !h->mega_unsupported[batch]) {
    // a new tag epoch per launch; when it would no longer fit its bits the
    // tagged buffers are cleared and the count starts again
    if (h->epoch + 1 >= (1u << (32 - kTagOpBits))) {
      CUDA_TRY(h, cudaMemsetAsync(h->tagged, 0, h->tagged_words * sizeof(uint64_t), h->stream));
      h->epoch = 0;
    }
    h->epoch += 1;
    MegaParams mp{};
    mp.epoch = h->epoch;
    mp.d = d;
    mp.ops = h->mega_ops[batch];
    mp.n_ops = h->mega_nops[batch];
    mp.prod = h->mega_prod[batch];
    mp.n_prod = h->mega_nprod[batch];
    mp.nrows = batch;
    mp.units = units;
    mp.chunk = chunk;
    mp.kmax = std::max(std::max(c.dim, c.n_head * c.head_dim), c.ffn);
    mp.io = SampIO{uniforms, N + 1, sp, forced, N, codes, status, slow_logits, fast_logits, draws,
                   U16(h->w.fast_emb)};
    mp.tok_emb = U16(h->w.tok_emb);
    mp.fusion = U16(h->w.fusion);
    mp.bar = h->bar_counter;
    mp.bar_extra = h->bar_extra;
    const int64_t need = static_cast<int64_t>(h->n_sm) * mp.n_ops * 4 * 8;
    mp.trace = (h->trace && h->trace_bytes >= need) ? h->trace : nullptr;
    mp.prefetch_bytes = h->prefetch_bytes;
    mp.w4 = h->any_w4 ? 1 : 0;
    CUDA_TRY(h, cudaMemsetAsync(h->bar_counter, 0, 4, h->stream));
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (h->profiling) {
      e0 = next_event(h);
      e1 = next_event(h);
      CUDA_TRY(h, cudaEventRecord(e0, h->stream));
    }
    bool unsupported = false;
    LAUNCH(h, launch_mega(mp, batch, h->n_sm, h->stream, &unsupported));
    if (!unsupported) {
      if (h->profiling) {
        CUDA_TRY(h, cudaEventRecord(e1, h->stream));
        h->prof_bytes.push_back(0.0);
      }
      for (int r = 0; r < batch; ++r) h->length[slots[r]] += 1;
      return DUALAR_OK;
    }
    if (h->profiling) h->ev_used -= 2;
    --h->launches;
    h->mega_unsupported[batch] = true;   // fall through to the per-op path
  }
  // 1. q0 from the held restricted logits (+ repetition-aware resample)
  LAUNCH(h, launch_sample_q0(d, batch, uniforms, N + 1, sp, forced, N, codes, status, slow_logits,
                             draws, U16(h->w.fast_emb), h->stream));
  // 2. fast AR: pass 0 stores the slow hidden state; passes 1..N-1 draw q_k
  for (int p = 0; p < N; ++p) {
    const float* xin = d.fin + static_cast<size_t>(p & 1) * kMaxRows * c.dim;
    for (int l = 0; l < c.fast_n_layer; ++l)
      TRY(block(h, h->fast[l], l, true, batch, l == 0 ? xin : d.hf, d.hf, p, 0, 0, false));
    if (p == 0) continue;
    GemvArgs a = gemv_base(h);
    a.w0 = U16(h->w.fast_out);
    a.n0 = c.fast_vocab;
    a.K = c.dim;
    a.mode = GEMV_STORE;
    a.nb = batch;
    a.x = d.hf;
    a.ldx = c.dim;
    a.norm_w = U16(h->w.fast_norm);
    a.out = d.logits;
    a.ldo = d.logit_ld;
    TRY(run_gemv(h, a));
    LAUNCH(h, launch_sample_fast(d, batch, p, uniforms, N + 1, sp, forced, N, codes, fast_logits,
                                 draws, U16(h->w.fast_emb), h->stream));
  }
  // 3. fusion -> next slow input; 4. one slow position; restricted head
  LAUNCH(h, launch_fusion(d, batch, U16(h->w.tok_emb), U16(h->w.fusion), h->stream));
  TRY(slow_stack(h, batch, units, chunk, true));
  TRY(run_gemv(h, args_head(h, 0, batch)));
  TRY(flush_tc(h));
  for (int r = 0; r < batch; ++r) h->length[slots[r]] += 1;
  return DUALAR_OK;
}

// ---- decode without allocating ------------------------------------------------
// dualar_decode_frame_noalloc keeps the split-KV attention's scratch (arrival
// counters, then partial results) in this fixed array instead of the handle's
// workspace.  It lives in every GPU that loads the library, until exit.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB
constexpr int kNoAllocMaxDevices = 64;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
static void* g_noalloc_addr[kNoAllocMaxDevices] = {};   // device address of the array, per device
static std::mutex g_noalloc_mutex;

// Device address of the fixed scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int noalloc_scratch(dualar_handle* h, int dev, void** out) {
  if (dev < 0 || dev >= kNoAllocMaxDevices) {
    set_err(h, "decode_frame_noalloc: device %d beyond the %d supported", dev, kNoAllocMaxDevices);
    return DUALAR_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_err(h, "cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(e));
      return DUALAR_ERR_CUDA;
    }
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return DUALAR_OK;
}

}  // namespace

// ============================================================================
// C ABI
// ============================================================================
extern "C" {

int dualar_create(const dualar_config* cfg, const dualar_weights* w, void* cuda_stream,
                  dualar_handle** out) {
  if (!out) return DUALAR_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w) return DUALAR_ERR_INVALID_ARG;
  dualar_handle* h = new dualar_handle();
  h->cfg = *cfg;
  h->stream = static_cast<cudaStream_t>(cuda_stream);
  auto fail = [&](int rc) {
    // keep the message readable by printing it: the handle is not returned
    fprintf(stderr, "dualar_create: %s\n", h->err.c_str());
    dualar_destroy(h);
    return rc;
  };
  int rc = validate_config(h, *cfg);
  if (rc != DUALAR_OK) return fail(rc);
  const dualar_config& c = h->cfg;
  const void* top[] = {w->tok_emb, w->final_norm, w->fast_emb, w->fast_norm, w->fast_out, w->fusion};
  for (const void* p : top)
    if (!p || !aligned16(p)) {
      set_err(h, "a weight pointer is NULL or not 16-byte aligned");
      return fail(DUALAR_ERR_INVALID_ARG);
    }
  if (!w->slow || !w->fast) {
    set_err(h, "per-layer weight arrays missing");
    return fail(DUALAR_ERR_INVALID_ARG);
  }
  h->w = *w;
  h->slow.assign(w->slow, w->slow + c.n_layer);
  h->fast.assign(w->fast, w->fast + c.fast_n_layer);
  for (int i = 0; i < c.n_layer; ++i)
    if ((rc = check_layer(h, h->slow[i], c.slow_qk_norm, "slow", i)) != DUALAR_OK) return fail(rc);
  for (int i = 0; i < c.fast_n_layer; ++i)
    if ((rc = check_layer(h, h->fast[i], c.fast_qk_norm, "fast", i)) != DUALAR_OK) return fail(rc);
  h->w.slow = nullptr;
  h->w.fast = nullptr;

  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    set_err(h, "no CUDA device");
    return fail(DUALAR_ERR_CUDA);
  }

  DevPtrs& d = h->d;
  d.D = c.dim;
  d.Hq = c.n_head;
  d.Hkv = c.n_kv_head;
  d.hd = c.head_dim;
  d.F = c.ffn;
  d.n_sem = c.n_sem;
  d.sem_begin = c.sem_begin;
  d.im_end = c.im_end_id;
  d.Cf = c.fast_vocab;
  d.N = c.n_codebooks;
  d.page_tokens = c.page_tokens;
  d.pages_per_seq = (c.max_ctx + c.page_tokens - 1) / c.page_tokens;
  d.n_layer = c.n_layer;
  d.fast_n_layer = c.fast_n_layer;
  d.max_pages = c.max_pages;
  d.rope_len = std::max(c.max_ctx, c.n_codebooks) + 1;
  d.max_seqs = c.max_seqs;
  d.qkv_dim = (c.n_head + 2 * c.n_kv_head) * c.head_dim;
  d.logit_ld = ((std::max(c.n_sem + 1, c.fast_vocab) + 3) / 4) * 4;
  d.eps = c.norm_eps;
  d.wait_limit_ns = 2000000000ull;

  const size_t R = kMaxRows;
  const int half = c.head_dim / 2;
  const int G = c.n_head / c.n_kv_head;
  uint16_t *rc_cos = nullptr, *rc_sin = nullptr;
  const size_t kv_elems = static_cast<size_t>(c.max_pages) * c.n_layer * 2 * c.n_kv_head *
                          c.page_tokens * c.head_dim;
#define ALLOC(p, n)                                   \
  do {                                                \
    if ((rc = dev_alloc(h, &(p), (n))) != DUALAR_OK) return fail(rc); \
  } while (0)
  ALLOC(rc_cos, static_cast<size_t>(d.rope_len) * half);
  ALLOC(rc_sin, static_cast<size_t>(d.rope_len) * half);
  d.rope_cos = rc_cos;
  d.rope_sin = rc_sin;
  ALLOC(d.kv_pool, kv_elems);
  ALLOC(d.page_table, static_cast<size_t>(c.max_seqs) * d.pages_per_seq);
  ALLOC(d.fast_kv, R * c.fast_n_layer * 2 * c.n_kv_head * c.n_codebooks * c.head_dim);
  ALLOC(d.h_last, static_cast<size_t>(c.max_seqs) * c.dim);
  ALLOC(d.z_last, static_cast<size_t>(c.max_seqs) * (c.n_sem + 1));
  ALLOC(d.hist, static_cast<size_t>(c.max_seqs) * kRasRing);
  ALLOC(d.hist_n, c.max_seqs);
  ALLOC(d.finished, c.max_seqs);
  ALLOC(d.rows, R);
  ALLOC(d.commit_map, R);
  ALLOC(d.xs, R * c.dim);
  ALLOC(d.hs, R * c.dim);
  ALLOC(d.hf, R * c.dim);
  ALLOC(d.fin, 2 * R * c.dim);
  ALLOC(d.qkv, R * d.qkv_dim);
  ALLOC(d.qrot, R * c.n_head * c.head_dim);
  ALLOC(d.attn, R * c.n_head * c.head_dim);
  ALLOC(d.act, R * c.ffn);
  ALLOC(d.logits, R * d.logit_ld);
  ALLOC(d.part, R * c.n_kv_head * kMaxChunks * G * (c.head_dim + 2));
  ALLOC(d.arrive, R * c.n_kv_head);
  ALLOC(d.sched, c.n_layer);
  ALLOC(d.codes_ws, R * kMaxCodebooks);
  ALLOC(d.err, 1);
  ALLOC(h->bar_counter, 1);
  {
    // tensor-core projections: x' halves for up to 128 rows and the split-K
    // partial sums
    const int kmax = std::max(std::max(c.dim, c.n_head * c.head_dim), c.ffn);
    const int nmax = std::max(std::max(d.qkv_dim, 2 * c.ffn), std::max(c.n_sem + 1, std::max(c.fast_vocab, c.dim)));
    h->tc.ldx = kmax;
    h->tc.part_floats = static_cast<size_t>(kTcMaxSlices) * kTcMaxRows * nmax;
    ALLOC(h->tc.xh, static_cast<size_t>(kTcMaxRows) * kmax);
    ALLOC(h->tc.xl, static_cast<size_t>(kTcMaxRows) * kmax);
    ALLOC(h->tc.part, h->tc.part_floats);
  }
  {
    // tagged work buffers of the persistent frame kernel, one region (cleared
    // together when the tag epoch wraps); every buffer starts on 64 bytes
    const size_t TR = kTaggedRows;
    const size_t sizes[9] = {TR * d.qkv_dim, TR * c.n_head * c.head_dim, TR * c.ffn, TR * c.dim,
                             TR * c.dim, TR * c.dim, kMaxCodebooks * TR * c.dim, TR * d.logit_ld,
                             TR * c.n_kv_head * kMaxChunks * G * (c.head_dim + 2)};
    size_t offs[9], total = 0;
    for (int i = 0; i < 9; ++i) {
      offs[i] = total;
      total += (sizes[i] + 7) / 8 * 8;
    }
    ALLOC(h->tagged, total);
    h->tagged_words = total;
    d.qkv_t = h->tagged + offs[0];
    d.attn_t = h->tagged + offs[1];
    d.act_t = h->tagged + offs[2];
    d.hs_t = h->tagged + offs[3];
    d.hf_t = h->tagged + offs[4];
    d.xs_t = h->tagged + offs[5];
    d.fin_t = h->tagged + offs[6];
    d.logits_t = h->tagged + offs[7];
    d.part_t = h->tagged + offs[8];
  }
#undef ALLOC

  // RoPE tables: angle = pos * base^(-2i/head_dim) in double, cos/sin rounded
  // once to bf16.  [P2] "Streaming: whose numbers": bf16 tables; "The slow AR
  // is Qwen3-4B": rope_base 1e6.
  {
    std::vector<uint16_t> hc(static_cast<size_t>(d.rope_len) * half), hs(hc.size());
    for (int p = 0; p < d.rope_len; ++p)
      for (int i = 0; i < half; ++i) {
        const double inv = std::pow(static_cast<double>(c.rope_base), -(2.0 * i) / c.head_dim);
        const double ang = static_cast<double>(p) * inv;
        hc[static_cast<size_t>(p) * half + i] = host_f32_to_bf16(static_cast<float>(std::cos(ang)));
        hs[static_cast<size_t>(p) * half + i] = host_f32_to_bf16(static_cast<float>(std::sin(ang)));
      }
    cudaError_t e = cudaMemcpy(rc_cos, hc.data(), hc.size() * 2, cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(rc_sin, hs.data(), hs.size() * 2, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      set_err(h, "rope upload: %s", cudaGetErrorString(e));
      return fail(DUALAR_ERR_CUDA);
    }
  }
  // page table entries start at -1 (no page)
  {
    std::vector<int32_t> neg(static_cast<size_t>(c.max_seqs) * d.pages_per_seq, -1);
    if (cudaMemcpy(d.page_table, neg.data(), neg.size() * 4, cudaMemcpyHostToDevice) != cudaSuccess) {
      set_err(h, "page table init failed");
      return fail(DUALAR_ERR_CUDA);
    }
  }
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) {
    set_err(h, "stream sync failed after allocation");
    return fail(DUALAR_ERR_CUDA);
  }
  h->length.assign(c.max_seqs, -1);
  h->pages.assign(c.max_seqs, {});
  h->page_refs.assign(c.max_pages, 0);
  h->prefix_only.assign(c.max_seqs, 0);
  for (int p = 0; p < c.max_pages; ++p) h->free_pages.insert(p);
  *out = h;
  return DUALAR_OK;
}

namespace {

// Prompt positions [p0, p0 + n_tokens) of a slot: p0 = 0 starts a sequence in
// an empty slot; p0 > 0 continues one (after a shared prefix).
int prefill_impl(dualar_handle* h, int32_t slot, const int32_t* tokens, int32_t n_tokens, bool append) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  const dualar_config& c = h->cfg;
  if (slot < 0 || slot >= c.max_seqs || !tokens || n_tokens <= 0) {
    set_err(h, "prefill: bad slot or tokens");
    return DUALAR_ERR_INVALID_ARG;
  }
  if (!append && h->length[slot] >= 0) {
    set_err(h, "prefill: slot %d holds a sequence", slot);
    return DUALAR_ERR_SLOT_BUSY;
  }
  if (append && h->length[slot] < 0) {
    set_err(h, "prefill: slot %d is empty", slot);
    return DUALAR_ERR_SLOT_EMPTY;
  }
  const int p0 = append ? h->length[slot] : 0;
  if (p0 + n_tokens > c.max_ctx) {
    set_err(h, "prefill: %d tokens exceed max_ctx %d", p0 + n_tokens, c.max_ctx);
    return DUALAR_ERR_CONTEXT_FULL;
  }
  for (int i = 0; i < n_tokens; ++i)
    if (tokens[i] < 0 || tokens[i] >= c.vocab) {
      set_err(h, "prefill: token %d out of range", tokens[i]);
      return DUALAR_ERR_INVALID_ARG;
    }
  const int need = (p0 + n_tokens + c.page_tokens - 1) / c.page_tokens - (p0 + c.page_tokens - 1) / c.page_tokens;
  if (need > static_cast<int>(h->free_pages.size())) {
    set_err(h, "prefill: %d pages needed, %zu free", need, h->free_pages.size());
    return DUALAR_ERR_OOM_PAGES;
  }
  const DevPtrs& d = h->d;
  if (!append) {
    CUDA_TRY(h, cudaMemsetAsync(d.hist_n + slot, 0, 4, h->stream));
    CUDA_TRY(h, cudaMemsetAsync(d.finished + slot, 0, 4, h->stream));
    h->length[slot] = 0;
  }
  h->launches = 0;
  LaunchSetup& s = h->setup;
  for (int c0 = 0; c0 < n_tokens; c0 += kMaxRows) {
    const int m = std::min(kMaxRows, n_tokens - c0);
    std::memset(&s, 0, sizeof(s));
    s.n_rows = m;
    s.commit_last_only = 1;
    s.embed = 1;
    for (int r = 0; r < m; ++r) {
      const int pos = p0 + c0 + r;
      s.rows[r] = RowInfo{slot, pos, 1, 0};
      s.tokens[r] = tokens[c0 + r];
      if (pos % c.page_tokens == 0) {
        const int pg = take_page(h);
        h->pages[slot].push_back(pg);
        s.upd_slot[s.n_updates] = slot;
        s.upd_index[s.n_updates] = pos / c.page_tokens;
        s.upd_page[s.n_updates] = pg;
        ++s.n_updates;
      }
    }
    int units = 0, chunk = 0;
    plan_attention(h, s, &units, &chunk);
    LAUNCH(h, launch_setup(s, d, U16(h->w.tok_emb), h->stream));
    TRY(slow_stack(h, m, units, chunk, false));
    if (c0 + m == n_tokens) TRY(run_gemv(h, args_head(h, m - 1, 1)));
  }
  TRY(flush_tc(h));
  h->length[slot] = p0 + n_tokens;
  h->prefix_only[slot] = 0;
  return DUALAR_OK;
}

}  // namespace

int dualar_prefill(dualar_handle* h, int32_t slot, const int32_t* tokens, int32_t n_tokens) {
  return prefill_impl(h, slot, tokens, n_tokens, false);
}

int dualar_prefill_append(dualar_handle* h, int32_t slot, const int32_t* tokens, int32_t n_tokens) {
  return prefill_impl(h, slot, tokens, n_tokens, true);
}

int dualar_share_prefix(dualar_handle* h, int32_t src, int32_t dst, int32_t n_tokens) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  const dualar_config& c = h->cfg;
  if (src < 0 || src >= c.max_seqs || dst < 0 || dst >= c.max_seqs || src == dst || n_tokens <= 0) {
    set_err(h, "share_prefix: bad slots or length");
    return DUALAR_ERR_INVALID_ARG;
  }
  if (h->length[src] < 0) {
    set_err(h, "share_prefix: slot %d is empty", src);
    return DUALAR_ERR_SLOT_EMPTY;
  }
  if (h->length[dst] >= 0) {
    set_err(h, "share_prefix: slot %d holds a sequence", dst);
    return DUALAR_ERR_SLOT_BUSY;
  }
  if (n_tokens > h->length[src]) {
    set_err(h, "share_prefix: %d tokens exceed slot %d's %d", n_tokens, src, h->length[src]);
    return DUALAR_ERR_INVALID_ARG;
  }
  const int pt = c.page_tokens;
  const int nfull = n_tokens / pt;
  const bool partial = n_tokens % pt != 0;
  if (partial && h->free_pages.empty()) {
    set_err(h, "share_prefix: no free page for the partly filled last page");
    return DUALAR_ERR_OOM_PAGES;
  }
  const DevPtrs& d = h->d;
  h->launches = 0;
  // full pages by reference; the partly filled one as a copy (both sequences
  // will write its remaining rows)
  for (int i = 0; i < nfull; ++i) {
    const int pg = h->pages[src][i];
    ++h->page_refs[pg];
    h->pages[dst].push_back(pg);
  }
  if (partial) {
    const int from = h->pages[src][nfull];
    const int pg = take_page(h);
    h->pages[dst].push_back(pg);
    const size_t page_elems = static_cast<size_t>(d.n_layer) * 2 * d.Hkv * pt * d.hd;
    CUDA_TRY(h, cudaMemcpyAsync(d.kv_pool + static_cast<size_t>(pg) * page_elems,
                                d.kv_pool + static_cast<size_t>(from) * page_elems, page_elems * 2,
                                cudaMemcpyDeviceToDevice, h->stream));
  }
  LaunchSetup& s = h->setup;
  const int np = static_cast<int>(h->pages[dst].size());
  for (int p0 = 0; p0 < np; p0 += kMaxRows) {
    std::memset(&s, 0, sizeof(s));
    for (int p = p0; p < std::min(np, p0 + kMaxRows); ++p) {
      s.upd_slot[s.n_updates] = dst;
      s.upd_index[s.n_updates] = p;
      s.upd_page[s.n_updates] = h->pages[dst][p];
      ++s.n_updates;
    }
    LAUNCH(h, launch_setup(s, d, U16(h->w.tok_emb), h->stream));
  }
  if (n_tokens == h->length[src]) {
    // the whole sequence: its held state too (the next frame starts from it)
    CUDA_TRY(h, cudaMemcpyAsync(d.h_last + static_cast<size_t>(dst) * d.D, d.h_last + static_cast<size_t>(src) * d.D,
                                sizeof(float) * d.D, cudaMemcpyDeviceToDevice, h->stream));
    CUDA_TRY(h, cudaMemcpyAsync(d.z_last + static_cast<size_t>(dst) * (d.n_sem + 1),
                                d.z_last + static_cast<size_t>(src) * (d.n_sem + 1), sizeof(float) * (d.n_sem + 1),
                                cudaMemcpyDeviceToDevice, h->stream));
    CUDA_TRY(h, cudaMemcpyAsync(d.hist + static_cast<size_t>(dst) * kRasRing, d.hist + static_cast<size_t>(src) * kRasRing,
                                sizeof(int32_t) * kRasRing, cudaMemcpyDeviceToDevice, h->stream));
    CUDA_TRY(h, cudaMemcpyAsync(d.hist_n + dst, d.hist_n + src, 4, cudaMemcpyDeviceToDevice, h->stream));
    CUDA_TRY(h, cudaMemcpyAsync(d.finished + dst, d.finished + src, 4, cudaMemcpyDeviceToDevice, h->stream));
    h->prefix_only[dst] = h->prefix_only[src];
  } else {
    CUDA_TRY(h, cudaMemsetAsync(d.hist_n + dst, 0, 4, h->stream));
    CUDA_TRY(h, cudaMemsetAsync(d.finished + dst, 0, 4, h->stream));
    h->prefix_only[dst] = 1;
  }
  h->length[dst] = n_tokens;
  return DUALAR_OK;
}

int dualar_debug_synthetic_context(dualar_handle* h, int32_t slot, int32_t n_tokens, uint32_t seed) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  const dualar_config& c = h->cfg;
  if (slot < 0 || slot >= c.max_seqs || n_tokens <= 0) {
    set_err(h, "synthetic context: bad slot or length");
    return DUALAR_ERR_INVALID_ARG;
  }
  if (h->length[slot] >= 0) {
    set_err(h, "synthetic context: slot %d holds a sequence", slot);
    return DUALAR_ERR_SLOT_BUSY;
  }
  if (n_tokens > c.max_ctx) {
    set_err(h, "synthetic context: %d tokens exceed max_ctx %d", n_tokens, c.max_ctx);
    return DUALAR_ERR_CONTEXT_FULL;
  }
  const int need = (n_tokens + c.page_tokens - 1) / c.page_tokens;
  if (need > static_cast<int>(h->free_pages.size())) {
    set_err(h, "synthetic context: %d pages needed, %zu free", need, h->free_pages.size());
    return DUALAR_ERR_OOM_PAGES;
  }
  const DevPtrs& d = h->d;
  CUDA_TRY(h, cudaMemsetAsync(d.hist_n + slot, 0, 4, h->stream));
  CUDA_TRY(h, cudaMemsetAsync(d.finished + slot, 0, 4, h->stream));
  h->launches = 0;
  LaunchSetup& s = h->setup;
  // pages in the order prefill takes them (lowest free first)
  for (int p0 = 0; p0 < need; p0 += kMaxRows) {
    std::memset(&s, 0, sizeof(s));
    for (int p = p0; p < std::min(need, p0 + kMaxRows); ++p) {
      const int pg = take_page(h);
      h->pages[slot].push_back(pg);
      s.upd_slot[s.n_updates] = slot;
      s.upd_index[s.n_updates] = p;
      s.upd_page[s.n_updates] = pg;
      ++s.n_updates;
    }
    LAUNCH(h, launch_setup(s, d, U16(h->w.tok_emb), h->stream));
  }
  LAUNCH(h, launch_synthetic_fill(d, slot, need, seed, h->n_sm, h->stream));
  h->length[slot] = n_tokens;
  return DUALAR_OK;
}

int dualar_decode_frame(dualar_handle* h, int32_t batch, const int32_t* slots,
                        const float* uniforms, const dualar_sampling* sampling, int32_t* codes,
                        int32_t* status) {
  return decode_impl(h, batch, slots, uniforms, sampling, nullptr, codes, status, nullptr, nullptr,
                     nullptr);
}

int dualar_decode_frame_forced(dualar_handle* h, int32_t batch, const int32_t* slots,
                               const float* uniforms, const dualar_sampling* sampling,
                               const int32_t* forced_codes, int32_t* codes, int32_t* status,
                               float* slow_logits, float* fast_logits, int32_t* draws) {
  return decode_impl(h, batch, slots, uniforms, sampling, forced_codes, codes, status, slow_logits,
                     fast_logits, draws);
}

int dualar_decode_frame_noalloc(dualar_handle* h, int32_t batch, const int32_t* slots,
                                const float* uniforms, const dualar_sampling* sampling,
                                int32_t* codes, int32_t* status) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  const dualar_config& c = h->cfg;
  const size_t G = static_cast<size_t>(c.n_head / c.n_kv_head);
  const size_t cnt_bytes =
      (static_cast<size_t>(batch > 0 ? batch : 0) * c.n_kv_head * sizeof(uint32_t) + 255) & ~size_t(255);
  const size_t part_bytes = static_cast<size_t>(batch > 0 ? batch : 0) * c.n_kv_head * kMaxChunks * G *
                            (c.head_dim + 2) * sizeof(float);
  if (batch < 1 || cnt_bytes + part_bytes > kNoAllocScratchBytes) {
    const size_t per_seq = 256 + static_cast<size_t>(c.n_kv_head) * kMaxChunks * G * (c.head_dim + 2) * 4;
    set_err(h, "decode_frame_noalloc: batch %d needs %zu bytes of attention scratch; the fixed array holds "
               "%zu bytes (at most %zu sequences per call for this model)",
            batch, cnt_bytes + part_bytes, kNoAllocScratchBytes, kNoAllocScratchBytes / per_seq);
    return DUALAR_ERR_INVALID_ARG;
  }
  int dev = -1;
  CUDA_TRY(h, cudaGetDevice(&dev));
  if (dev != h->device) {
    set_err(h, "decode_frame_noalloc: device %d is current, the handle lives on device %d", dev, h->device);
    return DUALAR_ERR_INVALID_ARG;
  }
  void* base = nullptr;
  int rc = noalloc_scratch(h, dev, &base);
  if (rc != DUALAR_OK) return rc;
  uint32_t* cnt = static_cast<uint32_t*>(base);
  float* part = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + cnt_bytes);
  // the last call's counters may be anything: they must start at zero
  CUDA_TRY(h, cudaMemsetAsync(cnt, 0, cnt_bytes, h->stream));
  uint32_t* saved_arrive = h->d.arrive;
  float* saved_part = h->d.part;
  const bool saved_prof = h->profiling;
  h->d.arrive = cnt;
  h->d.part = part;
  h->profiling = false;   // timing events would be created on demand
  rc = decode_impl(h, batch, slots, uniforms, sampling, nullptr, codes, status, nullptr, nullptr, nullptr,
                   /*per_op_only=*/true);
  h->d.arrive = saved_arrive;
  h->d.part = saved_part;
  h->profiling = saved_prof;
  return rc;
}

int dualar_release(dualar_handle* h, int32_t slot) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  if (slot < 0 || slot >= h->cfg.max_seqs) {
    set_err(h, "release: bad slot %d", slot);
    return DUALAR_ERR_INVALID_ARG;
  }
  for (int p : h->pages[slot]) drop_page(h, p);
  h->pages[slot].clear();
  h->length[slot] = -1;
  h->prefix_only[slot] = 0;
  return DUALAR_OK;
}

int dualar_sync(dualar_handle* h) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  uint32_t e = 0;
  CUDA_TRY(h, cudaMemcpy(&e, h->d.err, 4, cudaMemcpyDeviceToHost));
  if (e) {
    CUDA_TRY(h, cudaMemset(h->d.err, 0, 4));
    if (e & (DEV_ERR_MBAR_TIMEOUT | DEV_ERR_GRID_TIMEOUT)) {
      set_err(h, "a device-side wait timed out (error word 0x%x)", e);
      return DUALAR_ERR_TIMEOUT;
    }
    set_err(h, "a device-side bounds check failed (error word 0x%x)", e);
    return DUALAR_ERR_DEVICE;
  }
  return DUALAR_OK;
}

int dualar_get_error(const dualar_handle* h, char* buf, size_t len) {
  if (!h || !buf || len == 0) return DUALAR_ERR_INVALID_ARG;
  std::snprintf(buf, len, "%s", h->err.c_str());
  return DUALAR_OK;
}

void dualar_destroy(dualar_handle* h) {
  if (!h) return;
  if (!h->allocs.empty()) cudaStreamSynchronize(h->stream);
  for (void* p : h->allocs) cudaFree(p);
  for (cudaEvent_t e : h->ev_pool) cudaEventDestroy(e);
  delete h;
}

int dualar_get_page_table(const dualar_handle* h, int32_t slot, int32_t* pages,
                          int32_t max_entries, int32_t* n_pages) {
  if (!h || slot < 0 || slot >= h->cfg.max_seqs || !n_pages) return DUALAR_ERR_INVALID_ARG;
  const auto& v = h->pages[slot];
  *n_pages = static_cast<int32_t>(v.size());
  if (pages) {
    // read the device table (what the kernels use)
    std::vector<int32_t> dev(h->d.pages_per_seq);
    if (cudaMemcpy(dev.data(), h->d.page_table + static_cast<size_t>(slot) * h->d.pages_per_seq,
                   dev.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
      return DUALAR_ERR_CUDA;
    for (int i = 0; i < std::min<int>(max_entries, static_cast<int>(v.size())); ++i) pages[i] = dev[i];
  }
  return DUALAR_OK;
}

int dualar_get_rope_table(dualar_handle* h, int32_t n_pos, uint16_t* cos_bits, uint16_t* sin_bits) {
  if (!h || n_pos <= 0 || n_pos > h->d.rope_len || !cos_bits || !sin_bits)
    return DUALAR_ERR_INVALID_ARG;
  const size_t n = static_cast<size_t>(n_pos) * (h->cfg.head_dim / 2);
  CUDA_TRY(h, cudaMemcpy(cos_bits, h->d.rope_cos, n * 2, cudaMemcpyDeviceToHost));
  CUDA_TRY(h, cudaMemcpy(sin_bits, h->d.rope_sin, n * 2, cudaMemcpyDeviceToHost));
  return DUALAR_OK;
}

int dualar_read_state(dualar_handle* h, int32_t slot, float* hidden, float* logits) {
  if (!h || slot < 0 || slot >= h->cfg.max_seqs) return DUALAR_ERR_INVALID_ARG;
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  if (hidden)
    CUDA_TRY(h, cudaMemcpy(hidden, h->d.h_last + static_cast<size_t>(slot) * h->cfg.dim,
                           sizeof(float) * h->cfg.dim, cudaMemcpyDeviceToHost));
  if (logits)
    CUDA_TRY(h, cudaMemcpy(logits, h->d.z_last + static_cast<size_t>(slot) * (h->cfg.n_sem + 1),
                           sizeof(float) * (h->cfg.n_sem + 1), cudaMemcpyDeviceToHost));
  return DUALAR_OK;
}

int32_t dualar_slot_length(const dualar_handle* h, int32_t slot) {
  if (!h || slot < 0 || slot >= h->cfg.max_seqs) return -1;
  return h->length[slot];
}

int dualar_set_wait_limit(dualar_handle* h, uint64_t nanoseconds) {
  if (!h || nanoseconds == 0) return DUALAR_ERR_INVALID_ARG;
  h->d.wait_limit_ns = nanoseconds;
  return DUALAR_OK;
}

int32_t dualar_last_launch_count(const dualar_handle* h) { return h ? h->launches : -1; }

int dualar_set_persistent(dualar_handle* h, int32_t enable) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  h->use_mega = enable != 0;
  return DUALAR_OK;
}

int64_t dualar_w4a16_bytes(int32_t n, int32_t k) {
  if (n < 0 || k <= 0 || k % kW4Group) return -1;
  return static_cast<int64_t>(n) * w4_row_bytes(k);
}

int dualar_quantize_w4a16(const void* w, int32_t n, int32_t k, void* out, void* cuda_stream) {
  if (n < 0 || k <= 0 || k % kW4Group || (n > 0 && (!w || !out || !aligned16(w) || !aligned16(out))))
    return DUALAR_ERR_INVALID_ARG;
  const cudaError_t e = launch_quantize_w4(static_cast<const uint16_t*>(w), n, k, static_cast<unsigned char*>(out),
                                           static_cast<cudaStream_t>(cuda_stream));
  return e == cudaSuccess ? DUALAR_OK : DUALAR_ERR_CUDA;
}

int dualar_set_w4a16(dualar_handle* h, const dualar_w4a16_layer* slow, const dualar_w4a16_layer* fast) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  const dualar_config& c = h->cfg;
  const int qd = c.n_head * c.head_dim;
  auto check = [&](const dualar_w4a16_layer* v, int n, const char* which) {
    for (int i = 0; v && i < n; ++i) {
      const dualar_w4a16_layer& l = v[i];
      const void* ptrs[] = {l.wqkv, l.wo, l.w_gate, l.w_up, l.w_down};
      for (const void* p : ptrs)
        if (p && !aligned16(p)) {
          set_err(h, "%s layer %d: a packed weight pointer is not 16-byte aligned", which, i);
          return DUALAR_ERR_INVALID_ARG;
        }
      if ((l.w_gate == nullptr) != (l.w_up == nullptr)) {
        set_err(h, "%s layer %d: w_gate and w_up must be packed together", which, i);
        return DUALAR_ERR_INVALID_ARG;
      }
      const bool in_dim_ok = ((l.wqkv || l.w_gate) ? c.dim % kW4Group == 0 : true) &&
                             (l.wo ? qd % kW4Group == 0 : true) && (l.w_down ? c.ffn % kW4Group == 0 : true);
      if (!in_dim_ok) {
        set_err(h, "%s layer %d: a packed projection's in-dimension is not a multiple of %d", which, i, kW4Group);
        return DUALAR_ERR_INVALID_ARG;
      }
    }
    return DUALAR_OK;
  };
  if (int rc = check(slow, c.n_layer, "slow")) return rc;
  if (int rc = check(fast, c.fast_n_layer, "fast")) return rc;
  if (const int frc = flush_tc(h)) return frc;
  // the persistent kernel's programs name the old weights: built again on use
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) {
    set_err(h, "stream synchronisation failed");
    return DUALAR_ERR_CUDA;
  }
  for (int b = 0; b < 3; ++b) {
    for (void* p : {static_cast<void*>(h->mega_ops[b]), static_cast<void*>(h->mega_prod[b])}) {
      if (!p) continue;
      h->allocs.erase(std::remove(h->allocs.begin(), h->allocs.end(), p), h->allocs.end());
      cudaFree(p);
    }
    h->mega_ops[b] = nullptr;
    h->mega_prod[b] = nullptr;
    h->mega_nops[b] = h->mega_nprod[b] = 0;
    h->mega_unsupported[b] = false;
  }
  h->slow_q.clear();
  h->fast_q.clear();
  if (slow) h->slow_q.assign(slow, slow + c.n_layer);
  if (fast) h->fast_q.assign(fast, fast + c.fast_n_layer);
  h->any_w4 = false;
  size_t need = 0;   // 2 x the elements of the largest packed projection (SwiGLU: gate and up)
  const size_t D = c.dim, F = c.ffn;
  for (const auto* v : {&h->slow_q, &h->fast_q})
    for (const dualar_w4a16_layer& l : *v) {
      if (l.wqkv || l.wo || l.w_gate || l.w_down) h->any_w4 = true;
      if (l.wqkv) need = std::max(need, static_cast<size_t>(c.n_head + 2 * c.n_kv_head) * c.head_dim * D);
      if (l.wo) need = std::max(need, D * qd);
      if (l.w_gate) need = std::max(need, 2 * F * D);
      if (l.w_down) need = std::max(need, D * F);
    }
  need *= 2;   // hi and lo halves
  if (h->w4_bf16 && need != h->w4_bf16_elems) {
    h->allocs.erase(std::remove(h->allocs.begin(), h->allocs.end(), static_cast<void*>(h->w4_bf16)), h->allocs.end());
    cudaFree(h->w4_bf16);
    h->w4_bf16 = nullptr;
    h->w4_bf16_elems = 0;
  }
  if (need > 0 && !h->w4_bf16) {
    void* p = nullptr;
    if (cudaMalloc(&p, need * sizeof(uint16_t)) != cudaSuccess) {
      set_err(h, "cudaMalloc of the 4-bit projections' bf16 scratch failed");
      return DUALAR_ERR_CUDA;
    }
    h->allocs.push_back(p);
    h->w4_bf16 = static_cast<uint16_t*>(p);
    h->w4_bf16_elems = need;
  }
  return DUALAR_OK;
}

int dualar_set_tensor_cores(dualar_handle* h, int32_t enable) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  h->use_tc = enable != 0;
  return DUALAR_OK;
}

int dualar_set_trace(dualar_handle* h, void* device_buffer, int64_t bytes, int32_t* n_ops,
                     int32_t* n_ctas) {
  if (!h || bytes < 0) return DUALAR_ERR_INVALID_ARG;
  h->trace = static_cast<uint64_t*>(device_buffer);
  h->trace_bytes = device_buffer ? bytes : 0;
  if (n_ctas) *n_ctas = h->n_sm;
  if (n_ops) {
    // ops of the batch-1 program (built on demand)
    if (!h->mega_ops[1]) {
      const int rc = build_mega_program(h, 1);
      if (rc != DUALAR_OK) return rc;
    }
    *n_ops = h->mega_nops[1];
  }
  return DUALAR_OK;
}

int dualar_set_prefetch(dualar_handle* h, uint64_t bytes_per_sm) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  h->prefetch_bytes = bytes_per_sm;
  return DUALAR_OK;
}

int dualar_debug_barrier_extra(dualar_handle* h, uint32_t extra) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  h->bar_extra = extra;
  return DUALAR_OK;
}

int dualar_profile(dualar_handle* h, int32_t enable) {
  if (!h) return DUALAR_ERR_INVALID_ARG;
  h->profiling = enable != 0;
  return DUALAR_OK;
}

int dualar_profile_read(dualar_handle* h, int64_t* launches, double* total_ms, double* total_bytes,
                        double* max_ms) {
  if (!h || !launches || !total_ms || !total_bytes || !max_ms) return DUALAR_ERR_INVALID_ARG;
  CUDA_TRY(h, cudaStreamSynchronize(h->stream));
  const size_t n = h->prof_bytes.size();
  double t = 0.0, b = 0.0, mx = 0.0;
  for (size_t i = 0; i < n; ++i) {
    float ms = 0.f;
    CUDA_TRY(h, cudaEventElapsedTime(&ms, h->ev_pool[2 * i], h->ev_pool[2 * i + 1]));
    t += ms;
    mx = std::max(mx, static_cast<double>(ms));
    b += h->prof_bytes[i];
  }
  *launches = static_cast<int64_t>(n);
  *total_ms = t;
  *total_bytes = b;
  *max_ms = mx;
  h->prof_bytes.clear();
  h->ev_used = 0;
  return DUALAR_OK;
}

}  // extern "C"
