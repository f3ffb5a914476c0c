// mla_verify_attention_noalloc: the absorbed verify call for callers that
// cannot provide device scratch memory.
//
// Some callers have no way to allocate device memory for a workspace: plugin
// hosts and serving engines that own every device allocation through their
// own fixed pool and give their attention back-ends no allocator, and
// latency-critical loops where a cudaMalloc (which can synchronise the whole
// device) is not acceptable.  This entry point runs the same absorbed-branch
// kernels as mla_verify_attention, but their scratch lives in one
// file-scope __device__ array of kStaticScratchBytes, which every GPU that
// loads this library keeps reserved until the process exits.
//
// The array's name, used in host code, is only a host-side stand-in for the
// device symbol: its device address is looked up with cudaGetSymbolAddress
// once per device, with that device current, the first time this entry point
// runs on it.  That first call on each device should therefore come before
// any stream capture begins.
//
// Every call shares the one array and it keeps whatever the previous call
// left in it.  The absorbed launch path writes every scratch value before it
// reads it, so nothing has to start at zero; calls that overlap on the GPU
// (concurrent streams, or other threads) race on the array and must not be
// issued.

#include <mutex>

#include "mla_internal.h"

namespace mla {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) char g_static_scratch[kStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up once).
cudaError_t static_scratch(void** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_verify_attention_noalloc(
    const mla_geometry_t* g, const void* q_nope, const void* q_rope, const void* c_kv,
    const void* k_rope, int64_t c_kv_row_stride, int64_t k_rope_row_stride,
    int64_t seq_stride_rows, const void* W_UK, const void* W_UV, const int32_t* lens_dev,
    const int32_t* lens_host, int32_t batch, int32_t L, const int32_t* page_table,
    int32_t page_size, int32_t max_pages_per_seq, int32_t num_pages, void* out, void* stream,
    int32_t* branch_taken) {
  size_t need = 0;
  mla_status_t st = mla_workspace_bytes(g, batch, L, lens_host, MLA_MODE_ABSORBED, &need);
  if (st != MLA_OK) return st;
  if (need > kStaticScratchBytes) {
    set_error("this call needs %zu bytes of scratch; the static scratch of "
              "mla_verify_attention_noalloc holds %zu (use mla_verify_attention with a "
              "workspace)",
              need, kStaticScratchBytes);
    return MLA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const cudaError_t e = static_scratch(&scratch);
  if (e != cudaSuccess) {
    set_error("cudaGetSymbolAddress of the static scratch failed: %s", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return mla_verify_attention(g, q_nope, q_rope, c_kv, k_rope, c_kv_row_stride,
                              k_rope_row_stride, seq_stride_rows, W_UK, W_UV, lens_dev,
                              lens_host, batch, L, page_table, page_size, max_pages_per_seq,
                              num_pages, MLA_MODE_ABSORBED, out, scratch, kStaticScratchBytes,
                              stream, branch_taken);
}
