// mk_moe.cu -- MoE Dispatch + grouped GEMM (not built yet).
#include "mk_internal.h"

extern "C" {

size_t mk_moe_workspace_size(int R, int E_loc, int topk, long long T, long long H, long long N,
                             long long cap_rows, const mk_config* cfg) {
  (void)R; (void)E_loc; (void)topk; (void)T; (void)H; (void)N; (void)cap_rows; (void)cfg;
  return 0;
}

mk_status mk_moe_dispatch_gemm(const void* const* x, const float* const* logits, const void* const* w,
                               int R, int E_loc, int topk, long long T, long long H, long long N,
                               long long cap_rows, int* topk_idx, int* counts, int* const* recv_src,
                               int* recv_counts, void* const* recv_x, void* const* y, void* workspace,
                               size_t ws_bytes, const mk_config* cfg, mk_stream_t stream) {
  (void)x; (void)logits; (void)w; (void)R; (void)E_loc; (void)topk; (void)T; (void)H; (void)N;
  (void)cap_rows; (void)topk_idx; (void)counts; (void)recv_src; (void)recv_counts; (void)recv_x;
  (void)y; (void)workspace; (void)ws_bytes; (void)cfg; (void)stream;
  return MK_ERR_UNSUPPORTED;
}

}  // extern "C"
