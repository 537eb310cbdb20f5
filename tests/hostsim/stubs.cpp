// Kernel launchers of the host-runtime stand-in (see cuda_runtime.h here):
// nothing runs, except that the setup launch applies its page-table updates
// to the "device" table, as the setup kernel does, so the library's page
// tables can be read back and compared with the page oracle.
#include "internal.h"
#include "mega.h"
#include "tcgemm.h"

namespace dualar {

cudaError_t launch_setup(const LaunchSetup& s, const DevPtrs& d, const uint16_t*, cudaStream_t) {
  for (int i = 0; i < s.n_updates; ++i) {
    const int sl = s.upd_slot[i], ix = s.upd_index[i], pg = s.upd_page[i];
    if (sl < 0 || sl >= d.max_seqs || ix < 0 || ix >= d.pages_per_seq || pg < 0 || pg >= d.max_pages) {
      *d.err |= DEV_ERR_BAD_PAGE;
      continue;
    }
    d.page_table[sl * d.pages_per_seq + ix] = pg;
  }
  return cudaSuccess;
}
cudaError_t launch_gemv(const GemvArgs&, int, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_quantize_w4(const uint16_t*, int, int, unsigned char*, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_append(const DevPtrs&, int, int, bool, int, const uint16_t*, const uint16_t*, cudaStream_t) {
  return cudaSuccess;
}
cudaError_t launch_attn_paged(const DevPtrs&, int, int, int, int, int, bool, const uint16_t*, const uint16_t*,
                              cudaStream_t, bool* mma_used, AttnHalves) {
  if (mma_used) *mma_used = false;
  return cudaSuccess;
}
cudaError_t launch_attn_fast(const DevPtrs&, int, int, int, const uint16_t*, const uint16_t*, cudaStream_t,
                             AttnHalves) {
  return cudaSuccess;
}
cudaError_t launch_sample_q0(const DevPtrs&, int, const float*, int, const SamplingParams&, const int32_t*, int,
                             int32_t*, int32_t*, float*, int32_t*, const uint16_t*, cudaStream_t) {
  return cudaSuccess;
}
cudaError_t launch_sample_fast(const DevPtrs&, int, int, const float*, int, const SamplingParams&, const int32_t*,
                               int, int32_t*, float*, int32_t*, const uint16_t*, cudaStream_t) {
  return cudaSuccess;
}
cudaError_t launch_fusion(const DevPtrs&, int, const uint16_t*, const uint16_t*, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_synthetic_fill(const DevPtrs&, int, int, uint32_t, int, cudaStream_t) { return cudaSuccess; }
bool tc_available() { return false; }
bool tc_eligible(const GemvArgs&, int) { return false; }
bool tc_bf16_map(CUtensorMap*, const void*, int, int, int, int) { return false; }
cudaError_t launch_tc_gemm(const GemvArgs&, const TcBuffers&, int, cudaStream_t, int*, bool, bool, TcPending*,
                           bool, bool) {
  return cudaSuccess;
}
cudaError_t launch_dequant_w4(const void*, int, int, uint16_t*, cudaStream_t) { return cudaSuccess; }
bool tc_can_fuse(const TcPending&, const GemvArgs&) { return false; }
cudaError_t launch_tc_pending(const TcPending&, const TcBuffers&, int, cudaStream_t) { return cudaSuccess; }
cudaError_t launch_tc_reduce_norm(const TcPending&, const GemvArgs&, const TcBuffers&, cudaStream_t) {
  return cudaSuccess;
}
cudaError_t launch_mega(const MegaParams&, int, int, cudaStream_t, bool* unsupported) {
  *unsupported = false;
  return cudaSuccess;
}

}  // namespace dualar
