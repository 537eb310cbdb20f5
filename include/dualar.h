/* dualar.h -- C ABI of the GB300 Dual-AR frame decoder (libdualar.so).
 *
 * One call of dualar_decode_frame runs, for every sequence of a batch, the
 * per-frame Dual-Autoregressive decode step of a Fish-Speech-S2-shaped model:
 *
 *   1. draw q0 from the restricted slow-AR logits held since the last slow step
 *      (temperature / top-p, with the repetition-aware resample);
 *   2. N fast-AR passes along the codebook axis, drawing q1 .. q(N-1);
 *   3. multi-codebook fusion of the N codes into the next slow-AR input;
 *   4. one slow-AR decode position on that input over the paged KV cache,
 *      ending in the restricted head (semantic ids + <|im_end|>).
 *
 * Pages the operations follow (title, section):
 *   [P1] "How the Dual-Autoregressive Architecture Works in Fish Speech S2:
 *        A Deep Dive" -- Core Components (slow BaseTransformer, fast
 *        sub-network, DualARModelArgs), Inference Pipeline
 *        (decode_one_token_ar, generate).
 *   [P2] "Fish Audio S2: a Qwen3-4B on the time axis, four layers on the
 *        codebook axis, and tags that are only text" -- fact table (shapes),
 *        "Two autoregressions" (per-frame order, semantic logit bias,
 *        repetition-aware sampling, fast KV cache, Eq. 1 fusion with the
 *        1/sqrt(N+1) scale), "The slow AR is Qwen3-4B" (Qwen3 layer,
 *        qk-norm, rope_base, tied head, semantic id range), "Streaming"
 *        (bf16 RoPE tables).
 *   [P3] "s2-pro-w4a16-late12attn" (model card) -- its opening line: the
 *        4-bit-weight variant that keeps the late 12 attention layers bf16.
 *
 * Conventions for every call:
 *   - Return value: DUALAR_OK (0) or a negative DUALAR_ERR_* code.  Nothing
 *     aborts the process; dualar_get_error returns the last message.
 *   - All GPU work is queued on the CUDA stream given to dualar_create and is
 *     asynchronous: outputs and device-side errors become visible after the
 *     stream is synchronised (dualar_sync does that and reports device-side
 *     errors such as a wait that timed out).
 *   - "device" pointers are CUDA device memory, "host" pointers CPU memory.
 *   - The caller owns the weights, uniforms and output buffers; the library
 *     owns the KV page pool, per-sequence state and work buffers, all
 *     allocated by dualar_create and freed by dualar_destroy.
 *   - One handle is not thread-safe; calls on it must be serialised.
 */
#ifndef DUALAR_H
#define DUALAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  DUALAR_OK = 0,
  DUALAR_ERR_INVALID_ARG = -1,   /* bad pointer, size, slot or config field */
  DUALAR_ERR_OOM_PAGES = -2,     /* the KV page pool has no free page left */
  DUALAR_ERR_SLOT_BUSY = -3,     /* prefill on a slot that holds a sequence */
  DUALAR_ERR_SLOT_EMPTY = -4,    /* decode on a slot that was never prefilled */
  DUALAR_ERR_CUDA = -5,          /* a CUDA runtime call failed */
  DUALAR_ERR_TIMEOUT = -6,       /* a device-side wait gave up (see dualar_sync) */
  DUALAR_ERR_DEVICE = -7,        /* a device-side bounds check failed (see dualar_sync) */
  DUALAR_ERR_CONTEXT_FULL = -8   /* the sequence reached max_ctx positions */
};

/* Model shapes and runtime limits.  [P1] DualARModelArgs: the fast AR has
 * the slow AR's width and heads (fast_dim = dim; no fast_project_in).
 * Requirements: dim % 8 == 0, ffn % 8 == 0, head_dim in {64, 128},
 * n_head % n_kv_head == 0 with n_head / n_kv_head in {1, 2, 4, 8},
 * page_tokens == 64, n_codebooks in [2, 16], n_sem <= 4096,
 * fast_vocab <= 4096, im_end_id outside [sem_begin, sem_begin + n_sem). */
typedef struct dualar_config {
  int32_t dim;           /* model width D */
  int32_t n_layer;       /* slow-AR layers */
  int32_t n_head;        /* query heads */
  int32_t n_kv_head;     /* key/value heads */
  int32_t head_dim;
  int32_t ffn;           /* SwiGLU intermediate size */
  int32_t vocab;         /* slow vocabulary (tied embedding rows) */
  int32_t sem_begin;     /* first <|semantic:i|> id */
  int32_t n_sem;         /* number of semantic ids S */
  int32_t im_end_id;     /* <|im_end|> id */
  int32_t fast_n_layer;  /* fast-AR layers */
  int32_t fast_vocab;    /* fast embedding / head rows (codebook_size) */
  int32_t n_codebooks;   /* N codes per frame */
  int32_t slow_qk_norm;  /* 1: per-head RMSNorm on q, k in the slow AR */
  int32_t fast_qk_norm;  /* 1: same in the fast AR (0 for S2) */
  int32_t page_tokens;   /* positions per KV page (64) */
  int32_t max_pages;     /* KV pages in the pool */
  int32_t max_seqs;      /* slots; also the largest decode batch (<= 128) */
  int32_t max_ctx;       /* positions per sequence */
  float rope_base;       /* 1e6 for S2 */
  float norm_eps;        /* RMSNorm epsilon */
} dualar_config;

/* One transformer block's weights: device pointers to bf16 row-major
 * matrices [out][in], 16-byte aligned.  q_norm / k_norm may be NULL when the
 * block has no QK-norm. */
typedef struct dualar_layer_weights {
  const void* attn_norm;  /* [dim] */
  const void* wqkv;       /* [(n_head + 2 n_kv_head) head_dim][dim]: q rows, then k, then v */
  const void* q_norm;     /* [head_dim] */
  const void* k_norm;     /* [head_dim] */
  const void* wo;         /* [dim][n_head head_dim] */
  const void* ffn_norm;   /* [dim] */
  const void* w_gate;     /* [ffn][dim] */
  const void* w_up;       /* [ffn][dim] */
  const void* w_down;     /* [dim][ffn] */
} dualar_layer_weights;

/* All weights (device pointers, bf16, 16-byte aligned; they must stay valid
 * for the handle's lifetime).  slow and fast are HOST arrays of per-layer
 * structs, copied by dualar_create. */
typedef struct dualar_weights {
  const void* tok_emb;                 /* [vocab][dim]; also the tied slow head */
  const void* final_norm;              /* [dim] */
  const dualar_layer_weights* slow;    /* host array [n_layer] */
  const void* fast_emb;                /* [fast_vocab][dim] */
  const dualar_layer_weights* fast;    /* host array [fast_n_layer] */
  const void* fast_norm;               /* [dim] */
  const void* fast_out;                /* [fast_vocab][dim] (untied) */
  const void* fusion;                  /* [n_sem + (n_codebooks-1) fast_vocab][dim]:
                                          codebook 0 rows, then codebooks 1..N-1 */
} dualar_weights;

/* Sampling parameters of a decode call.  [P2] "Two autoregressions": the
 * repetition-aware resample draws at ras_temperature 1.0 / ras_top_p 0.9 and
 * replaces q0 when q0 repeats a semantic code among the last ras_win
 * (<= 16; 0 disables) committed q0 of the sequence.  temperature 0 is greedy
 * (largest logit, lowest id on ties).  allow_eos = 0 removes <|im_end|> from
 * the q0 candidates. */
typedef struct dualar_sampling {
  float temperature;
  float top_p;
  int32_t ras_win;
  float ras_temperature;
  float ras_top_p;
  int32_t allow_eos;
} dualar_sampling;

typedef struct dualar_handle dualar_handle;

/* Library plumbing: the pages define no such call (they describe a Python
 * engine); it sets up what the decode step below needs.
 * Creates a decoder on the current CUDA device.  cfg, w: host structs (read
 * during the call).  cuda_stream: a cudaStream_t (NULL = legacy default
 * stream) on which all later work is queued.  Allocates the KV pool
 * (max_pages x n_layer x 2 x n_kv_head x page_tokens x head_dim bf16), the
 * per-slot state and the work buffers.  On failure *out is NULL. */
int dualar_create(const dualar_config* cfg, const dualar_weights* w, void* cuda_stream,
                  dualar_handle** out);

/* Runs the slow AR over a prompt and starts a sequence in an empty slot.
 * [P2] "Two autoregressions" / "Speakers and turns": prompt ids are embedded
 * with the slow embedding (no fusion).  tokens: host int32[n_tokens], ids in
 * [0, vocab).  Leaves the slot holding the final-normed hidden state and the
 * restricted logits of the last prompt position, from which the first
 * decode_frame draws q0.  Errors: INVALID_ARG, SLOT_BUSY, OOM_PAGES,
 * CONTEXT_FULL, CUDA. */
int dualar_prefill(dualar_handle* h, int32_t slot, const int32_t* tokens, int32_t n_tokens);

/* Decodes one frame for `batch` sequences.  [P1] "decode_one_token_ar";
 * [P2] "Two autoregressions".
 *   slots:    host int32[batch], distinct prefilled slots
 *   uniforms: device float[batch][n_codebooks + 1] in [0, 1):
 *             u[0] normal q0 draw, u[1] resample draw, u[k+1] draw of q_k
 *   codes:    device int32[batch][n_codebooks] out: q0 as a semantic index in
 *             [0, n_sem), q1..q(N-1) in [0, fast_vocab); -1 for a row that ended
 *   status:   device int32[batch] out: 0 ok, 1 q0 was <|im_end|> (the sequence
 *             ends; release the slot), 2 the slot had already ended
 * Host-side page allocation happens before any GPU work; on OOM_PAGES or
 * CONTEXT_FULL nothing is queued.  Errors: INVALID_ARG, SLOT_EMPTY,
 * OOM_PAGES, CONTEXT_FULL, CUDA. */
int dualar_decode_frame(dualar_handle* h, int32_t batch, const int32_t* slots,
                        const float* uniforms, const dualar_sampling* sampling, int32_t* codes,
                        int32_t* status);

/* Teacher-forced / instrumented variant of dualar_decode_frame.  The draws are
 * made exactly as in dualar_decode_frame, but when forced_codes is not NULL the
 * codes committed (fed to the fast AR, fusion and history) are forced_codes
 * (device int32[batch][n_codebooks], same layout as codes).  Optional device
 * outputs (NULL to skip):
 *   slow_logits: float[batch][n_sem + 1] restricted logits q0 was drawn from
 *                (semantic ids in order, <|im_end|> last)
 *   fast_logits: float[batch][n_codebooks - 1][fast_vocab] fast-head logits of
 *                passes 1..N-1
 *   draws:       int32[batch][n_codebooks + 2]: normal q0 draw, resample draw,
 *                chosen q0 (before forcing), then the draws of q1..q(N-1) */
int dualar_decode_frame_forced(dualar_handle* h, int32_t batch, const int32_t* slots,
                               const float* uniforms, const dualar_sampling* sampling,
                               const int32_t* forced_codes, int32_t* codes, int32_t* status,
                               float* slow_logits, float* fast_logits, int32_t* draws);

/* Decodes one frame like dualar_decode_frame, but allocates nothing during the
 * call.  The pages have no counterpart of this call; it exists for callers
 * that cannot allocate device memory once they are running -- for example a
 * host that hands the library a fixed device budget at start-up and owns
 * every remaining byte through its own arena, or a process where another
 * framework has already reserved the rest of the GPU.  dualar_decode_frame
 * may allocate on the first call with a new batch size (it uploads the
 * persistent kernel's op program then) and while timing is on (events); this
 * call never does: it runs one kernel per op, and the split-KV attention
 * keeps its scratch (arrival counters and partial results) in a fixed 4 MiB
 * array compiled into the library instead of the handle's workspace.
 *   - Limit: batch * n_kv_head * 64 * (n_head/n_kv_head) * (head_dim+2) * 4
 *     bytes of partials plus counters must fit in 4 MiB -- at most 3
 *     sequences per call for the S2-Pro shape; larger batches return
 *     DUALAR_ERR_INVALID_ARG with the sizes in the error message.
 *   - Every GPU that loads the library holds the array until the process
 *     exits.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  The handle's device must be
 *     current.
 *   - All calls share the one array.  Each call clears the counters first;
 *     calls whose GPU work overlaps (other streams, other handles on the same
 *     device) race on the array and must not overlap.
 * Arguments, outputs and errors as dualar_decode_frame. */
int dualar_decode_frame_noalloc(dualar_handle* h, int32_t batch, const int32_t* slots,
                                const float* uniforms, const dualar_sampling* sampling,
                                int32_t* codes, int32_t* status);

/* Library plumbing with no passage of its own: the end of a sequence whose
 * q0 was <|im_end|> ([P2] "Two autoregressions"), or its replacement by a
 * queued request, frees its slot here.
 * Ends the sequence in a slot and returns its KV pages to the pool (lowest
 * page numbers are handed out first); a page shared with other slots
 * (dualar_share_prefix) returns only when the last of them releases it.
 * Queues nothing on the GPU. */
int dualar_release(dualar_handle* h, int32_t slot);

/* Starts a sequence in the empty slot dst from the first n_tokens positions
 * of slot src: a common prompt prefix such as a reference voice, which
 * [P2] "Tags are text" places in the system prompt so that requests with the
 * same voice share it, and whose cache hits [P2] "Streaming: whose numbers"
 * reports.  dst's page table takes src's full pages of those positions by
 * reference (each page counts the slots holding it); a partly filled last
 * page is copied (one page of every layer's K/V), so neither sequence ever
 * writes a shared page.  With n_tokens equal to src's length dst also takes
 * src's held state (final hidden, restricted logits, resample history) and
 * can decode at once; with fewer, dst holds only the prefix and must be
 * continued with dualar_prefill_append before decoding (decode rejects it).
 * 1 <= n_tokens <= src's length.  Errors: INVALID_ARG, SLOT_EMPTY (src),
 * SLOT_BUSY (dst), OOM_PAGES, CUDA. */
int dualar_share_prefix(dualar_handle* h, int32_t src, int32_t dst, int32_t n_tokens);

/* Continues the prompt of a slot that holds a sequence (typically a shared
 * prefix): positions length .. length + n_tokens - 1, exactly as
 * dualar_prefill computes a prompt, and the slot then holds the state of the
 * last of them.  tokens: host int32[n_tokens].  Errors: INVALID_ARG,
 * SLOT_EMPTY, OOM_PAGES, CONTEXT_FULL, CUDA. */
int dualar_prefill_append(dualar_handle* h, int32_t slot, const int32_t* tokens, int32_t n_tokens);

/* ---- 4-bit weights (w4a16) --------------------------------------------
 * [P3] "s2-pro-w4a16-late12attn" (model card): the S2-Pro checkpoint with
 * 4-bit weights and 16-bit activations, keeping the attention of the late 12
 * slow layers in bf16.  The card gives no packing format; this library's:
 * a matrix [n][k] (k a positive multiple of 128) becomes n records, one per
 * output row, of k/2 + roundup(k/64, 16) bytes:
 *   bytes [0, k/2)            byte i holds the codes of elements 2i (low
 *                             nibble) and 2i+1 (high nibble), each stored as
 *                             u = q + 8 with q in [-8, 7];
 *   bytes [k/2, k/2 + k/64)   the bf16 scale of each group of 128 consecutive
 *                             elements (little-endian);
 *   the rest                  zero.
 * Element j of a row stands for (u_j - 8) * scale[j / 128].  Activations
 * stay fp32 (at least the 16 bits the name asks for). */

/* Bytes of the packed form of a [n][k] matrix; -1 if n < 0 or k is not a
 * positive multiple of 128. */
int64_t dualar_w4a16_bytes(int32_t n, int32_t k);

/* Packs a bf16 matrix into the format above, on cuda_stream (a cudaStream_t,
 * NULL = legacy default stream), asynchronously.  Each group of 128 takes
 * scale s = bf16(m / 7) with m its largest |w| (fp32 division, round to
 * nearest even) and q = clamp(rint(w / s), -8, 7) (0 when s = 0).
 *   w:   device bf16 [n][k], 16-byte aligned
 *   out: device, dualar_w4a16_bytes(n, k) bytes, 16-byte aligned
 * Finite weights only.  Errors: INVALID_ARG (sizes, NULL or unaligned
 * pointers), CUDA. */
int dualar_quantize_w4a16(const void* w, int32_t n, int32_t k, void* out, void* cuda_stream);

/* Packed projections of one transformer block (device pointers from
 * dualar_quantize_w4a16 of the bf16 matrix of the same name, which keeps its
 * shape [out][in]); NULL keeps that projection in bf16.  w_gate and w_up are
 * both packed or both NULL. */
typedef struct dualar_w4a16_layer {
  const void* wqkv;
  const void* wo;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
} dualar_w4a16_layer;

/* Makes the decoder read the given projections from their packed form from
 * the next call on (the caller keeps them valid until they are replaced or
 * the handle is destroyed).  slow: host array [n_layer] or NULL (all bf16);
 * fast: host array [fast_n_layer] or NULL.  Embeddings, norms and both heads
 * stay bf16.  Up to 8 rows a packed projection runs in the weight-streaming
 * GEMV on the packed bytes (exact products q * s * x): inside the persistent
 * frame kernel for batches of 1-2 (dualar_set_persistent), otherwise one
 * launch per projection in passes of at most 8 rows.  From 9 rows (decode
 * batches, prefill chunks) it is first expanded, in a scratch buffer the
 * handle allocates here (twice the largest packed projection's elements,
 * gate and up together), into two bf16 matrices whose sum is exactly q * s,
 * and multiplied on the tensor cores over both.  The call synchronises the handle's stream and drops the
 * persistent kernel's cached frame programs, which are built again for the
 * new weights on the next decode.  Both arrays NULL restores the all-bf16
 * decoder and frees the scratch.  Errors: INVALID_ARG (an unaligned pointer,
 * a gate without its up matrix, an in-dimension that is not a multiple of
 * 128), CUDA (also when the scratch cannot be allocated). */
int dualar_set_w4a16(dualar_handle* h, const dualar_w4a16_layer* slow, const dualar_w4a16_layer* fast);

/* Library plumbing (no counterpart on the pages).
 * Synchronises the handle's stream and reports device-side errors:
 * DUALAR_ERR_TIMEOUT if a bounded wait gave up, DUALAR_ERR_DEVICE if a bounds
 * check skipped an access.  Clears the device error word. */
int dualar_sync(dualar_handle* h);

/* Library plumbing (no counterpart on the pages).
 * Copies the last error message (NUL-terminated, truncated to len). */
int dualar_get_error(const dualar_handle* h, char* buf, size_t len);

/* Library plumbing (no counterpart on the pages).
 * Frees everything the handle allocated (after synchronising its stream). */
void dualar_destroy(dualar_handle* h);

/* ---- inspection (tests) ------------------------------------------------ */

/* Host copy of a slot's page-table entries: pages[0 .. *n_pages-1]. */
int dualar_get_page_table(const dualar_handle* h, int32_t slot, int32_t* pages,
                          int32_t max_entries, int32_t* n_pages);

/* Host copy of the bf16 RoPE tables (bits), [n_pos][head_dim / 2] each. */
int dualar_get_rope_table(dualar_handle* h, int32_t n_pos, uint16_t* cos_bits,
                          uint16_t* sin_bits);

/* Synchronous host copy of a slot's held state: hidden [dim] (final-normed)
 * and restricted logits [n_sem + 1]; either pointer may be NULL. */
int dualar_read_state(dualar_handle* h, int32_t slot, float* hidden, float* logits);

/* Next position of a slot (prompt length + frames decoded); -1 if empty. */
int32_t dualar_slot_length(const dualar_handle* h, int32_t slot);

/* Time limit of every device-side wait, in nanoseconds (default 2 s). */
int dualar_set_wait_limit(dualar_handle* h, uint64_t nanoseconds);

/* Number of kernel launches queued by the last decode call. */
int32_t dualar_last_launch_count(const dualar_handle* h);

/* Decode path for batches of 1-2 sequences: 1 (default) runs the whole frame
 * as one persistent cooperative kernel (one CTA per SM; the N fast-AR passes
 * and the slow step never return to the host); 0 queues one kernel per op.
 * Both paths compute the same values. */
int dualar_set_persistent(dualar_handle* h, int32_t enable);

/* Projections of 9..128 rows (decode batches above 8 sequences, prefill
 * chunks) run on the tensor cores: 1 (default) one tcgen05 GEMM per
 * projection that reads the weights once (activations as two bf16 halves,
 * fp32 accumulation, split-K partials added in a fixed order); 0 the
 * weight-streaming GEMV in passes of <= 8 rows.  Both compute the same
 * projection to fp32 rounding (not bit-identically).  Errors: INVALID_ARG. */
int dualar_set_tensor_cores(dualar_handle* h, int32_t enable);

/* Persistent frame kernel: weight bytes per SM that its producer keeps in
 * flight into L2 ahead of the shared-memory ring while the ring is full
 * (default 65536; on GB300 64 KiB hides part of the refill at op boundaries,
 * 128 KiB and more cost more than they hide; 0 turns it off).  A tuning knob;
 * results do not depend on it. */
int dualar_set_prefetch(dualar_handle* h, uint64_t bytes_per_sm);

/* Test hook for the failure path of the persistent kernel's grid barrier:
 * every barrier waits for `extra` arrivals beyond the grid, which never come,
 * so each wait runs into the handle's wait limit (dualar_set_wait_limit), the
 * kernel finishes with garbage outputs, and dualar_sync returns
 * DUALAR_ERR_TIMEOUT.  0 (default) restores normal operation. */
int dualar_debug_barrier_extra(dualar_handle* h, uint32_t extra);

/* Benchmark and test hook (no counterpart on the pages): gives a free slot a
 * context of n_tokens positions without running the model.  Pages are taken
 * exactly as dualar_prefill takes them (lowest free first); every K/V value of
 * those pages (all layers) is set to a seeded value in [-1, 1) (bf16), the
 * held hidden state to seeded values in [-1, 1) and the held restricted
 * logits to seeded values in [-3, 3); the resample history is empty.  The
 * slot then decodes like a prefilled one.  Used to set up long batched
 * contexts (e.g. 64 sequences of 1-4K tokens) whose prefill would dominate a
 * decode benchmark.  Errors: INVALID_ARG (slot or length), SLOT_BUSY,
 * CONTEXT_FULL, OOM_PAGES, CUDA.  Asynchronous on the handle's stream. */
int dualar_debug_synthetic_context(dualar_handle* h, int32_t slot, int32_t n_tokens, uint32_t seed);

/* Per-op timeline of the persistent frame kernel.  device_buffer: device
 * memory of `bytes` bytes (NULL stops tracing).  While set, every persistent
 * launch whose program fits writes, per CTA and op, four global-timer stamps
 * (ns): the op's start; for a GEMV, when its input is staged and when all of
 * its weight tiles are consumed (0 for other ops); the op's end before the
 * grid barrier: uint64 [n_ctas][n_ops][4].  *n_ops / *n_ctas (optional) receive the sizes
 * for a batch of 1 (n_ops builds that program if needed). */
int dualar_set_trace(dualar_handle* h, void* device_buffer, int64_t bytes, int32_t* n_ops,
                     int32_t* n_ctas);

/* Kernel timing: with enable = 1, every weight-streaming GEMV launch and
 * every persistent frame-kernel launch queued from now on is bracketed by
 * CUDA events on the handle's stream; for GEMV launches the algorithmic bytes
 * (weights read + activations read and written) are recorded as well (0 for
 * the frame kernel).  enable = 0 stops recording. */
int dualar_profile(dualar_handle* h, int32_t enable);

/* Synchronises the stream, then reports the recorded GEMV launches: their
 * count, summed device time (ms), summed algorithmic bytes, and the longest
 * single launch (ms).  Clears the record. */
int dualar_profile_read(dualar_handle* h, int64_t* launches, double* total_ms, double* total_bytes,
                        double* max_ms);

#ifdef __cplusplus
}
#endif

#endif /* DUALAR_H */
