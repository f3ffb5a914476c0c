// mla_verify_attention_noalloc: the absorbed verify call for callers that
// cannot provide device scratch memory.
//
// Some callers have no way to allocate device memory for a workspace: plugin
// hosts and serving engines that own every device allocation through their
// own fixed pool and give their attention back-ends no allocator, and
// latency-critical loops where a cudaMalloc (which can synchronise the whole
// device) is not acceptable.  This entry point runs the same absorbed-branch
// kernels as mla_verify_attention, but their scratch lives in one
// file-scope __device__ array of kStaticScratchBytes.
//
// This file is its own CUDA module, and CUDA loads modules lazily: the array
// is reserved on a device when the module is first loaded there, which is the
// first call of this entry point on that device (its cudaGetSymbolAddress),
// not when the library is loaded.  From then on the device keeps the 32 MiB
// until the process exits.  The first call on each device should therefore
// come early, as a warm-up: before a host pool claims the device's memory
// (or the load fails for lack of memory, reported as MLA_ERR_WORKSPACE) and
// before any stream capture begins.
//
// The array's name, used in host code, is only a host-side stand-in for the
// device symbol.  Its device address is looked up with cudaGetSymbolAddress
// on every call, with the call's device current (the stream must belong to
// it), so a call made in another context or after a device reset gets that
// context's address, never a stale one.
//
// Every call shares the one array and it keeps whatever the previous call
// left in it.  The absorbed launch path writes every scratch value it later
// uses, so nothing has to start at zero; calls that overlap on the GPU
// (concurrent streams, or other threads) race on the array and must not be
// issued.

#include "mla_internal.h"

namespace mla {

constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) char g_static_scratch[kStaticScratchBytes];

namespace {

// Device address of g_static_scratch in the current context, after checking
// that `stream` belongs to the current device.
mla_status_t static_scratch(cudaStream_t stream, void** addr) {
  int dev = -1, sdev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaStreamGetDevice(stream, &sdev);
  if (e != cudaSuccess) {
    set_error("could not query the current device or the stream's device: %s",
              cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  if (sdev != dev) {
    set_error("the stream belongs to device %d but device %d is current", sdev, dev);
    return MLA_ERR_INVALID_ARG;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e == cudaErrorMemoryAllocation) {
    cudaGetLastError();
    set_error("device %d has no room left for the %zu-byte static scratch, which is reserved "
              "by the first mla_verify_attention_noalloc call on a device: make that call "
              "before the host's memory pool claims the device",
              dev, kStaticScratchBytes);
    return MLA_ERR_WORKSPACE;
  }
  if (e != cudaSuccess) {
    set_error("cudaGetSymbolAddress of the static scratch failed: %s", cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  *addr = p;
  return MLA_OK;
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
  st = static_scratch((cudaStream_t)stream, &scratch);
  if (st != MLA_OK) return st;
  return mla_verify_attention(g, q_nope, q_rope, c_kv, k_rope, c_kv_row_stride,
                              k_rope_row_stride, seq_stride_rows, W_UK, W_UV, lens_dev,
                              lens_host, batch, L, page_table, page_size, max_pages_per_seq,
                              num_pages, MLA_MODE_ABSORBED, out, scratch, kStaticScratchBytes,
                              stream, branch_taken);
}
