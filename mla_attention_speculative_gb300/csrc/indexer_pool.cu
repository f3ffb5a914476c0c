// Indexer key pooling with an incremental tail, and the top-k window
// selection it feeds.
//
// "One guard, 110x off the verify step", section "The same bug, one layer
// over": the sparse model's indexer pools the cached keys into windows of
// four before scoring them; completed windows are kept and only the tail is
// recomputed, for any number S of new tokens in a step, as long as the cache
// has a pool, there is no padding, the batch shape matches and the cache is
// exactly as long as the pool remembers (a speculative rejection that trimmed
// the cache fails the last guard).  Section "The sparse model is different":
// the indexer's top 2048 positions are what the sparse attention reads.
//
// Window w covers positions 4w..4w+3; its pooled key is the mean of the keys
// it holds (a partial last window holds fewer than four).  Every window is
// computed by the same code whichever path asks for it, so a wide step pools
// bit for bit as the same tokens fed one at a time.
//
// Three kernels, all bound by memory or latency:
//   pool_windows   one warp per window: four key rows read once (as vectors),
//                  summed in a fixed order, scaled by 1/count, stored as fp32
//   score_windows  one thread per window: the window's pooled key read once
//                  and dotted with every new token's query (in shared memory)
//   select_topk    one CTA per new token: an 8-bit radix select of the k-th
//                  largest score over the windows the token may see, then the
//                  chosen windows in ascending order and their positions

#include <cuda_bf16.h>

#include <algorithm>
#include <cfloat>
#include <mutex>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kWindow = 4;
constexpr int kMaxDim = 512;
constexpr int kMaxNewTokens = 32;

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// pooled[b, w, :] for w in [w0, w1): one warp per window; lane j owns
// columns [j * dim/32, (j + 1) * dim/32), read as whole vectors when that run
// is a multiple of four elements.
template <typename T>
__device__ __forceinline__ void load4(const T* p, float (&f)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&f)[4]) {
  const float4 v = *(const float4*)p;
  f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&f)[4]) {
  const uint2 v = *(const uint2*)p;
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xffff0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xffff0000u);
}

template <typename T>
__global__ void __launch_bounds__(256) pool_windows(const T* __restrict__ keys, long long row_stride,
                                                    long long seq_stride, int dim, long long len,
                                                    long long w0, long long w1,
                                                    float* __restrict__ pooled, long long cap) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long w = w0 + (long long)blockIdx.x * 8 + warp;
  const int b = blockIdx.y;
  if (w >= w1) return;
  const long long t0 = kWindow * w;
  const int cnt = (int)min((long long)kWindow, len - t0);
  const T* base = keys + (long long)b * seq_stride * row_stride + t0 * row_stride;
  float* out = pooled + ((long long)b * cap + w) * dim;
  const int cpl = dim / 32;
  if (cpl % 4 == 0) {
    for (int c = lane * cpl; c < (lane + 1) * cpl; c += 4) {
      float rows[kWindow][4];
#pragma unroll
      for (int i = 0; i < kWindow; ++i) {
        if (i < cnt) load4(base + i * row_stride + c, rows[i]);
        else rows[i][0] = rows[i][1] = rows[i][2] = rows[i][3] = 0.f;
      }
      float ov[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float s = rows[0][e];
#pragma unroll
        for (int i = 1; i < kWindow; ++i)
          if (i < cnt) s += rows[i][e];
        ov[e] = cnt == kWindow ? s * 0.25f : s / (float)cnt;
      }
      *(float4*)(out + c) = make_float4(ov[0], ov[1], ov[2], ov[3]);
    }
  } else {
    for (int c = lane; c < dim; c += 32) {
      float s = ld_f(base + c);
      for (int i = 1; i < cnt; ++i) s += ld_f(base + i * row_stride + c);
      out[c] = cnt == kWindow ? s * 0.25f : s / (float)cnt;
    }
  }
}

// scores[b, s, w] = q[b, s, :] . pooled[b, w, :] for w < nwin.  One thread
// per window: it reads the window's pooled key once, 16 bytes at a time, and
// dots it with up to eight queries per pass; the queries sit in shared memory
// and every thread of a warp reads the same query element at once.
constexpr int kScoreGroup = 8;
__global__ void __launch_bounds__(256) score_windows(const float* __restrict__ q,
                                                     const float* __restrict__ pooled,
                                                     long long cap, int dim, int S,
                                                     long long nwin, float* __restrict__ scores) {
  extern __shared__ float sq[];  // [S][dim]
  const int b = blockIdx.y;
  for (int i = threadIdx.x; i < S * dim; i += blockDim.x) sq[i] = q[(long long)b * S * dim + i];
  __syncthreads();
  const long long w = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (w >= nwin) return;
  const float4* pk = (const float4*)(pooled + ((long long)b * cap + w) * dim);
  for (int s0 = 0; s0 < S; s0 += kScoreGroup) {
    float acc[kScoreGroup];
#pragma unroll
    for (int j = 0; j < kScoreGroup; ++j) acc[j] = 0.f;
    for (int c = 0; c < dim / 4; ++c) {
      const float4 kv = pk[c];
#pragma unroll
      for (int j = 0; j < kScoreGroup; ++j) {
        if (s0 + j < S) {
          const float4 qv = *(const float4*)(sq + (s0 + j) * dim + 4 * c);
          acc[j] = fmaf(qv.x, kv.x, acc[j]);
          acc[j] = fmaf(qv.y, kv.y, acc[j]);
          acc[j] = fmaf(qv.z, kv.z, acc[j]);
          acc[j] = fmaf(qv.w, kv.w, acc[j]);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kScoreGroup; ++j)
      if (s0 + j < S) scores[((long long)b * S + s0 + j) * nwin + w] = acc[j];
  }
}

// Order-preserving map of a float onto uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kSelThreads = 1024;
constexpr int kSelPerThread = 4;                       // consecutive windows per thread and round
constexpr int kSelRound = kSelThreads * kSelPerThread;
constexpr int kSelSmemWindows = 48 * 1024;            // scores staged in shared memory up to this

// Exclusive prefix sum of one value per thread over the CTA; *total receives the sum.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int t = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_sums[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

// Row (b, s): the k best of the windows w <= p/4 (p = len - S + s), ties to
// the lower window; windows listed ascending, then their positions <= p.
// The row's scores are staged in shared memory when they fit; the k-th
// largest is found by an 8-bit radix select over order-preserving keys, and
// the chosen windows are written in order, 4096 windows per round.
__global__ void __launch_bounds__(kSelThreads) select_topk(const float* __restrict__ scores,
                                                          long long nwin, int S, long long len,
                                                          int k, int32_t* __restrict__ win_out,
                                                          int32_t* __restrict__ pos_out) {
  extern __shared__ float ssc[];
  __shared__ int hist[256];
  __shared__ int warp_sums[32];
  __shared__ int sel[2];  // chosen digit, remaining count
  const int b = blockIdx.y, s = blockIdx.x;
  const long long p = len - S + s;
  const long long vis = p / kWindow + 1;
  const int keff = (int)min((long long)k, vis);
  const long long row = (long long)b * S + s;
  const float* src = scores + row * nwin;
  if (vis <= kSelSmemWindows) {
    for (long long w = threadIdx.x; w < vis; w += kSelThreads) ssc[w] = src[w];
    __syncthreads();
    src = ssc;
  }

  uint32_t prefix = 0, mask = 0;
  int remaining = keff;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (long long w = threadIdx.x; w < vis; w += kSelThreads) {
      const uint32_t key = order_key(src[w]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int cum = 0, d = 255;
      for (; d > 0; --d) {
        if (cum + hist[d] >= remaining) break;
        cum += hist[d];
      }
      sel[0] = d;
      sel[1] = remaining - cum;
    }
    __syncthreads();
    prefix |= (uint32_t)sel[0] << shift;
    mask |= 255u << shift;
    remaining = sel[1];
    __syncthreads();
  }
  // prefix is now the k-th largest key; `remaining` of the windows equal to
  // it are taken, lowest windows first.  Rounds of 4096 windows in order.
  int taken_before = 0, eq_before_round = 0;
  for (long long r0 = 0; r0 < vis; r0 += kSelRound) {
    const long long w0 = r0 + (long long)threadIdx.x * kSelPerThread;
    uint32_t keys[kSelPerThread];
    int gt = 0, eq = 0;
#pragma unroll
    for (int e = 0; e < kSelPerThread; ++e) {
      keys[e] = w0 + e < vis ? order_key(src[w0 + e]) : 0u;
      gt += w0 + e < vis && keys[e] > prefix;
      eq += w0 + e < vis && keys[e] == prefix;
    }
    int eq_total, take_total;
    const int eq_rank = eq_before_round + block_exclusive_scan(eq, warp_sums, &eq_total);
    const int eq_take = max(0, min(eq, remaining - eq_rank));
    const int take = keff > 0 ? gt + eq_take : 0;
    int o = taken_before + block_exclusive_scan(take, warp_sums, &take_total);
    int eq_seen = 0;
#pragma unroll
    for (int e = 0; e < kSelPerThread; ++e) {
      if (w0 + e >= vis || take == 0) continue;
      bool t = keys[e] > prefix;
      if (keys[e] == prefix) t = eq_seen++ < eq_take;
      if (!t) continue;
      const long long w = w0 + e;
      if (win_out) win_out[row * k + o] = (int32_t)w;
#pragma unroll
      for (int i = 0; i < kWindow; ++i) {
        const long long tpos = kWindow * w + i;
        pos_out[row * (long long)kWindow * k + (long long)kWindow * o + i] =
            tpos <= p ? (int32_t)tpos : -1;
      }
      ++o;
    }
    taken_before += take_total;
    eq_before_round += eq_total;
  }
  // padding past the chosen windows
  for (int j = taken_before + threadIdx.x; j < k; j += kSelThreads) {
    if (win_out) win_out[row * k + j] = -1;
#pragma unroll
    for (int i = 0; i < kWindow; ++i) pos_out[row * (long long)kWindow * k + kWindow * j + i] = -1;
  }
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_indexer_pool_update(const void* keys, int32_t dtype,
                                                int64_t key_row_stride, int64_t seq_stride_rows,
                                                int32_t batch, int32_t dim, int64_t cache_len,
                                                int32_t new_tokens, int32_t padded, float* pooled,
                                                int64_t pooled_windows_cap,
                                                mla_indexer_pool_state_t* state,
                                                int32_t* incremental_out, void* stream) {
  if (keys == nullptr || pooled == nullptr || state == nullptr) {
    set_error("keys, pooled and state must not be NULL");
    return MLA_ERR_INVALID_ARG;
  }
  if (dtype != MLA_DTYPE_BF16 && dtype != MLA_DTYPE_FP32) {
    set_error("unknown dtype %d", dtype);
    return MLA_ERR_INVALID_ARG;
  }
  if (batch < 1 || batch > 65535 || dim < 32 || dim > kMaxDim || dim % 32 != 0) {
    set_error("batch %d must be in [1, 65535] and dim %d a multiple of 32 in [32, %d]", batch,
              dim, kMaxDim);
    return MLA_ERR_INVALID_ARG;
  }
  if (new_tokens < 1 || cache_len < new_tokens) {
    set_error("need 1 <= new_tokens (%d) <= cache_len (%lld)", new_tokens, (long long)cache_len);
    return MLA_ERR_INVALID_ARG;
  }
  const long long nwin = (cache_len + kWindow - 1) / kWindow;
  if (pooled_windows_cap < nwin) {
    set_error("the pool holds %lld windows; a cache of %lld tokens fills %lld",
              (long long)pooled_windows_cap, (long long)cache_len, nwin);
    return MLA_ERR_INVALID_ARG;
  }
  if (key_row_stride < dim || (batch > 1 && seq_stride_rows < cache_len)) {
    set_error("key_row_stride %lld < dim, or seq_stride_rows %lld < cache_len",
              (long long)key_row_stride, (long long)seq_stride_rows);
    return MLA_ERR_INVALID_ARG;
  }
  // the guards of the incremental path
  const bool incremental = state->length >= 0 && padded == 0 && state->batch == batch &&
                           state->dim == dim && state->length == cache_len - new_tokens;
  const long long w0 = incremental ? state->length / kWindow : 0;
  const long long nw = nwin - w0;
  cudaError_t e = cudaSuccess;
  if (nw > 0) {
    const dim3 grid((unsigned)((nw + 7) / 8), batch);
    cudaStream_t st = (cudaStream_t)stream;
    KernelTimer kt("indexer_pool_windows", st);
    if (dtype == MLA_DTYPE_BF16)
      pool_windows<__nv_bfloat16><<<grid, 256, 0, st>>>(
          (const __nv_bfloat16*)keys, key_row_stride, seq_stride_rows, dim, cache_len, w0, nwin,
          pooled, pooled_windows_cap);
    else
      pool_windows<float><<<grid, 256, 0, st>>>((const float*)keys, key_row_stride,
                                                 seq_stride_rows, dim, cache_len, w0, nwin,
                                                 pooled, pooled_windows_cap);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) {
    set_error("CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  state->length = cache_len;
  state->batch = batch;
  state->dim = dim;
  if (incremental_out) *incremental_out = incremental ? 1 : 0;
  return MLA_OK;
}

extern "C" mla_status_t mla_indexer_select_workspace_bytes(int32_t batch, int32_t new_tokens,
                                                           int64_t cache_len, size_t* bytes) {
  if (bytes == nullptr || batch < 1 || new_tokens < 1 || cache_len < new_tokens) {
    set_error("bad arguments (batch %d, new_tokens %d, cache_len %lld)", batch, new_tokens,
              (long long)cache_len);
    return MLA_ERR_INVALID_ARG;
  }
  const long long nwin = (cache_len + kWindow - 1) / kWindow;
  *bytes = (size_t)batch * new_tokens * nwin * sizeof(float);
  return MLA_OK;
}

extern "C" mla_status_t mla_indexer_select(const float* q, const float* pooled,
                                           int64_t pooled_windows_cap, int32_t batch,
                                           int32_t dim, int64_t cache_len, int32_t new_tokens,
                                           int32_t k_windows, int32_t* windows_out,
                                           int32_t* positions_out, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  if (q == nullptr || pooled == nullptr || positions_out == nullptr) {
    set_error("q, pooled and positions_out must not be NULL");
    return MLA_ERR_INVALID_ARG;
  }
  if (batch < 1 || batch > 65535 || dim < 32 || dim > kMaxDim || dim % 32 != 0 ||
      new_tokens < 1 ||
      new_tokens > kMaxNewTokens || cache_len < new_tokens || k_windows < 1) {
    set_error("bad arguments (batch %d, dim %d, new_tokens %d (<= %d), cache_len %lld, k %d)",
              batch, dim, new_tokens, kMaxNewTokens, (long long)cache_len, k_windows);
    return MLA_ERR_INVALID_ARG;
  }
  const long long nwin = (cache_len + kWindow - 1) / kWindow;
  if (pooled_windows_cap < nwin) {
    set_error("the pool holds %lld windows; a cache of %lld tokens fills %lld",
              (long long)pooled_windows_cap, (long long)cache_len, nwin);
    return MLA_ERR_INVALID_ARG;
  }
  if ((size_t)new_tokens * dim * sizeof(float) > 48 * 1024) {
    set_error("new_tokens x dim = %d x %d queries exceed the 48 KB the scoring kernel stages",
              new_tokens, dim);
    return MLA_ERR_INVALID_ARG;
  }
  size_t need = 0;
  mla_indexer_select_workspace_bytes(batch, new_tokens, cache_len, &need);
  if (workspace == nullptr || workspace_bytes < need) {
    set_error("workspace of %zu bytes is smaller than the %zu this call needs", workspace_bytes,
              need);
    return MLA_ERR_WORKSPACE;
  }
  cudaStream_t st = (cudaStream_t)stream;
  float* scores = (float*)workspace;
  {
    KernelTimer kt("indexer_score_windows", st);
    score_windows<<<dim3((unsigned)((nwin + 255) / 256), batch), 256,
                    (size_t)new_tokens * dim * sizeof(float), st>>>(
        q, pooled, pooled_windows_cap, dim, new_tokens, nwin, scores);
  }
  {
    KernelTimer kt("indexer_select_topk", st);
    const long long vis_max = (cache_len - 1) / kWindow + 1;
    const size_t sel_smem = vis_max <= kSelSmemWindows ? (size_t)vis_max * sizeof(float) : 0;
    if (sel_smem > 48 * 1024) {
      static std::once_flag once;
      static cudaError_t attr_err = cudaSuccess;
      std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(select_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kSelSmemWindows * (int)sizeof(float));
      });
      if (attr_err != cudaSuccess) {
        set_error("CUDA error %d (%s)", (int)attr_err, cudaGetErrorString(attr_err));
        return MLA_ERR_CUDA;
      }
    }
    select_topk<<<dim3(new_tokens, batch), kSelThreads, sel_smem, st>>>(
        scores, nwin, new_tokens, cache_len, k_windows, windows_out, positions_out);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}
