// mk_noalloc.cu -- mk_ag_gemm_noalloc: AllGather + GEMM for callers that
// cannot allocate device memory.
//
// The fused AllGather+GEMM kernel needs a small scratch area (a header with the
// CTA ticket counter, the abort word and the device status, plus one ready
// flag per copied sub-chunk of A).  mk_ag_gemm takes it from the caller as a
// workspace buffer.  This entry point instead keeps it in a fixed array of
// MK_NOALLOC_SCRATCH_BYTES in the library's own device memory, so its caller
// passes only the inputs and outputs and no allocation happens on the way.
#include <mutex>

#include "mk_internal.h"

namespace {

// The scratch array.  Every GPU that loads the library holds one copy of it
// until the process exits.  In host code this name is only a stand-in for the
// device symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MK_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The first call
// on a device looks the address up and zero-fills the array on `s`.
mk_status scratch_on_current_device(cudaStream_t s, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MK_ERR_UNSUPPORTED;
  if (dev < 0 || dev >= kMaxDevices) return MK_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return MK_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, MK_NOALLOC_SCRATCH_BYTES, s) != cudaSuccess) return MK_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MK_OK;
}

}  // namespace

extern "C" mk_status mk_ag_gemm_noalloc(const void* const* a_shards, const void* b, void* a_gathered,
                                        void* c, mk_dtype c_dtype, int R, int local_rank, long long m_r,
                                        long long n, long long k, int* device_status,
                                        const mk_config* cfg, mk_stream_t stream) {
  // The in-kernel trace would land in the library's own array, where the
  // caller cannot read it: rejected.
  if (cfg && cfg->trace != 0) return MK_ERR_INVALID;
  // Size check first: it needs no GPU and rejects shapes whose scratch would
  // not fit in the fixed array.
  const size_t need = mk_workspace_size(MK_OP_AG_GEMM, R, m_r, n, k, cfg);
  if (need == 0 || need > MK_NOALLOC_SCRATCH_BYTES) return MK_ERR_INVALID;
  if (device_status && (reinterpret_cast<uintptr_t>(device_status) & 3u)) return MK_ERR_INVALID;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  mk_status st = scratch_on_current_device(s, &scratch);
  if (st != MK_OK) return st;
  // The array keeps the previous call's contents.  The ready flags carry a
  // per-call tag and need no clearing; the header (ticket counter, abort word,
  // status, detail) must start at zero.
  if (cudaMemsetAsync(scratch, 0, 4 * sizeof(uint32_t), s) != cudaSuccess) return MK_ERR_CUDA;
  st = mk_ag_gemm(a_shards, b, a_gathered, c, c_dtype, R, local_rank, m_r, n, k, scratch,
                  MK_NOALLOC_SCRATCH_BYTES, cfg, stream);
  if (st != MK_OK) return st;
  if (device_status) {
    const uint8_t* status_word = static_cast<const uint8_t*>(scratch) + 4 * mk::HDR_STATUS;
    if (cudaMemcpyAsync(device_status, status_word, sizeof(int), cudaMemcpyDeviceToDevice, s) !=
        cudaSuccess)
      return MK_ERR_CUDA;
  }
  return MK_OK;
}
