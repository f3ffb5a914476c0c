// Internal interfaces of libmla.so: the per-call plan that the host code builds
// from the C-ABI arguments, and the kernel launchers that consume it.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/mla.h"

namespace mla {

// Split-KV layout and workspace carve-up of one kernel family.
struct SplitPlan {
  int chunk = 0;    // KV rows per piece (multiple of 64)
  int splits = 0;   // largest number of pieces of any sequence
  size_t off_qlat = 0, off_opart = 0, off_ml = 0, off_exp = 0, off_olat = 0;
  size_t bytes = 0;
};

// Launch plan of one verify call.  Built on the host from the arguments and
// the host copy of the cache lengths, before anything is launched.
struct Plan {
  // geometry
  int B = 0, L = 0, H = 0, r = 0, n = 0, v = 0, rope = 0;
  float scale = 0.f;
  int dtype = MLA_DTYPE_BF16;
  int branch = MLA_BRANCH_ABSORBED;
  // cache lengths
  int Tmax = 0;
  int64_t sumT = 0;
  // split-KV: sequence b is cut into ceil(T_b / chunk) pieces of `chunk` rows;
  // `splits` is the largest such count over the batch
  int chunk = 0;
  int splits = 0;
  // the two kernel families' layouts; the workspace covers the larger
  SplitPlan generic;   // CUDA-core kernels, any geometry and paging
  SplitPlan fast;      // tcgen05/TMA kernels of the chosen branch
  bool fast_ok = false;
  size_t ws_bytes = 0;
  // the layout of the family that runs (copied from generic or fast)
  size_t off_qlat = 0, off_opart = 0, off_ml = 0, off_exp = 0, off_olat = 0;
  void use(const SplitPlan& sp) {
    chunk = sp.chunk;
    splits = sp.splits;
    off_qlat = sp.off_qlat;
    off_opart = sp.off_opart;
    off_ml = sp.off_ml;
    off_exp = sp.off_exp;
    off_olat = sp.off_olat;
  }
};



// Device-side view of the cache addressing shared by all kernels.
struct CacheView {
  const void* c_kv;
  const void* k_rope;
  int64_t ckv_stride;      // elements between consecutive rows of c_kv
  int64_t kr_stride;       // elements between consecutive rows of k_rope
  int64_t seq_stride;      // rows between sequences (contiguous cache)
  const int32_t* page_table;  // NULL: contiguous
  int32_t page_size;
  int32_t max_pages;
  int32_t num_pages;
};

// Status-word code a kernel records when a page-table entry it needs lies
// outside [0, num_pages): no address is formed from it, and the positions of
// that page read as zeros.  Codes below it are bounded waits that ran out.
constexpr int kBadPageSite = 300;

// Global row index of cached position t of sequence b, or -1 when the page
// id that holds it is outside [0, num_pages) (nothing may be read then).
__host__ __device__ inline int64_t cache_row(const CacheView& c, int b, int t) {
  if (c.page_table == nullptr) return (int64_t)b * c.seq_stride + t;
  const int32_t page = c.page_table[(int64_t)b * c.max_pages + t / c.page_size];
  if (page < 0 || page >= c.num_pages) return -1;
  return (int64_t)page * c.page_size + (t % c.page_size);
}

struct Args {
  const void* q_nope;
  const void* q_rope;
  CacheView cache;
  const void* W_UK;
  const void* W_UV;
  const int32_t* lens;      // device
  // sparse (top-k) calls: [B, L, topk_k] device positions per verify row;
  // NULL for the dense call
  const int32_t* topk = nullptr;
  int topk_k = 0;
  void* out;
  char* ws;                 // device workspace base
  cudaStream_t stream;
};

// Generic kernels: CUDA-core arithmetic for any geometry, fp32 or bf16.
cudaError_t launch_generic_absorbed(const Plan& p, const Args& a);
cudaError_t launch_generic_materialised(const Plan& p, const Args& a);
// Status word of the generic kernels (kBadPageSite or 0); synchronises.
int generic_device_status(bool clear);

// Streaming multiprocessors of the current device (152 on GB300; 152 also
// when no device can be queried, so host-only planning stays defined).
int device_sm_count();

// Tensor-core kernels for the absorbed branch (bf16, r = 512, rope = 64,
// n a multiple of 64 up to 256, v a multiple of 128 up to 512).
bool fast_absorbed_supported(const Plan& p);
cudaError_t launch_fast_absorbed(const Plan& p, const Args& a);
// Two-CTA clusters of the absorbed attention that fit on the current device
// at once (device_sm_count() / 2 when it cannot be queried).
int absorbed_cluster_slots();
// Status word of the tensor-core kernels (0 = no wait ran out); synchronises.
int absorbed_device_status(bool clear);
// The status-word site the bounded-wait self-test records.
constexpr int kSelftestSite = 99;
// One CTA whose bounded wait runs out on purpose (no fault, no hang: the wait
// gives up after its limit and records kSelftestSite).
cudaError_t launch_wait_selftest(cudaStream_t stream);
int selftest_device_status(bool clear);

// Tensor-core kernels for the materialised branch (bf16, r = 512, rope = 64,
// n and v multiples of 64 up to 256): a tcgen05 expansion GEMM into a
// [B*H, Tmax, n+v] workspace, then flash attention over it.
bool fast_materialised_supported(const Plan& p);
size_t fast_materialised_workspace(const Plan& p);
cudaError_t launch_fast_materialised(const Plan& p, const Args& a);
int materialised_device_status(bool clear);

// Status word of the indexer kernels (0 = no wait ran out); synchronises.
int indexer_device_status(bool clear);

// Records a one-line failure description for mla_last_error().
void set_error(const char* fmt, ...);

// Kernel timing instrumentation (mla_kernel_timing_*): while enabled, a
// KernelTimer brackets one launch with a pair of CUDA events on its stream.
bool timing_enabled();
class KernelTimer {
 public:
  KernelTimer(const char* name, cudaStream_t stream);
  ~KernelTimer();
  KernelTimer(const KernelTimer&) = delete;
  KernelTimer& operator=(const KernelTimer&) = delete;

 private:
  int id_ = -1;
  cudaStream_t stream_;
  cudaEvent_t start_ = nullptr;
};

}  // namespace mla
