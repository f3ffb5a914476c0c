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
// Three steps, all bound by memory or latency:
//   pool_windows        one warp per window: four key rows read once (as
//                       vectors), summed in a fixed order, scaled by 1/count,
//                       stored as fp32
//   score_windows_d128  each window's pooled key read once (TMA tensor copies
//                       of 64 windows, 128-byte swizzle) and dotted with every
//                       new token's query, one lane per window
//                       (score_windows: eight lanes per window, for dims
//                       other than 128)
//   select_topk_cluster a row (one new token) spread over a cluster of eight
//                       CTAs: a radix select (a 10-bit digit summed over the
//                       cluster, then the chosen bucket's keys gathered into
//                       every CTA for two 11-bit digits) of the k-th largest
//                       score over the windows the token may see, then the
//                       chosen windows in ascending order and their positions
//                       (select_topk: one CTA per row and 12, 10, 10-bit
//                       digits, for rows too long for the cluster's shared
//                       memory)

#include <cuda_bf16.h>

#include <mutex>

#include "mla_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace mla {
using namespace sm103;
namespace {

constexpr int kWindow = 4;
constexpr int kMaxDim = 512;
constexpr int kMaxNewTokens = 32;

__device__ __forceinline__ float ld_f(const float* p) { return *p; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// pooled[b, w, :] for w in [w0, w1): one warp per window; lane j owns
// columns [j * dim/32, (j + 1) * dim/32), read as whole vectors (vec) when
// that run is a multiple of four elements and the rows are aligned for it.
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
                                                    float* __restrict__ pooled, long long cap,
                                                    bool vec) {
  // the scoring may be placed at once; it waits for this grid before it reads
  pdl_launch_dependents();
  pdl_wait();  // the keys may come from the preceding kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long w = w0 + (long long)blockIdx.x * 8 + warp;
  const int b = blockIdx.y;
  if (w >= w1) return;
  const long long t0 = kWindow * w;
  const int cnt = (int)min((long long)kWindow, len - t0);
  const T* base = keys + (long long)b * seq_stride * row_stride + t0 * row_stride;
  float* out = pooled + ((long long)b * cap + w) * dim;
  const int cpl = dim / 32;
  if (vec) {
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

// scores[b, s, w] = q[b, s, :] . pooled[b, w, :] for w < nwin.
//
// dim = 128 (score_windows_d128): a CTA of eight warps per 64 windows.  Four
// TMA tensor copies, one per 32 dims (128 bytes of each window), bring the 64
// pooled keys into shared memory with the 128-byte swizzle, each completing
// on its own mbarrier.  Warp (x, half) takes box x of windows
// [32 half, 32 half + 32), one lane per window, and starts as soon as its box
// lands: each lane accumulates its window's partial dot products over those
// 32 dims with eight queries at a time in registers, dims in order, with no
// exchange between lanes.  The queries sit in shared memory (padded with zeros
// to a multiple of eight) and are read as broadcasts; boxes 1..3 leave their
// partial sums in shared memory and the box-0 warps add them, in box order,
// and write each query's 32 scores as one coalesced row.  The swizzle puts
// 16-byte piece c of window row r at piece c ^ (r & 7) of its 128-byte row,
// so the eight lanes of each shared-memory phase read eight different bank
// groups.
//
// Other dims (score_windows): eight lanes per window, lane g holding the
// 16-byte pieces g, g + 8, ... of the key; the queries are staged in shared
// memory, and the eight partial sums are folded over the eight lanes by a
// reduce-scatter (exchanges at distance 4, 2, 1).
constexpr int kD128CtaWindows = 64;
constexpr int kD128Boxes = 4;  // 32 dims (128 bytes) each
constexpr int kD128Threads = kD128Boxes * kD128CtaWindows;  // one warp per (box, 32 windows)
constexpr int kD128BoxBytes = kD128CtaWindows * 128;
constexpr int kD128RedBytes = (kD128Boxes - 1) * 8 * kD128CtaWindows * 4;
constexpr int kScoreThreads = 256;
constexpr int kIndexerWaitSite = 70;

__device__ int g_indexer_status = 0;

// Shared memory of score_windows_d128 for S new tokens: the key boxes
// (1024-byte aligned for the swizzle), the partial sums of boxes 1..3, then
// the queries padded to eight.
__host__ __device__ constexpr int d128_smem_bytes(int S) {
  return 1024 + kD128Boxes * kD128BoxBytes + kD128RedBytes + ((S + 7) / 8) * 8 * 512;
}

__global__ void __launch_bounds__(kD128Threads) score_windows_d128(
    const __grid_constant__ CUtensorMap tm_keys, const float* __restrict__ q, int S,
    long long nwin, float* __restrict__ scores) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // offsets from the shared array itself keep every access a shared-memory one
  uint8_t* keys = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  float* red = (float*)(keys + kD128Boxes * kD128BoxBytes);      // [box - 1][8][64]
  float4* sq = (float4*)(keys + kD128Boxes * kD128BoxBytes + kD128RedBytes);  // [S8][32]
  __shared__ __align__(8) uint64_t full[kD128Boxes];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int x = warp >> 1;                   // this warp's box (dims 32x .. 32x + 31)
  const int r = (warp & 1) * 32 + lane;      // this lane's window row in the tile
  const int b = blockIdx.y;
  const long long c0 = (long long)blockIdx.x * kD128CtaWindows;
  const long long w = c0 + r;
  const int S8 = (S + 7) & ~7;
  pdl_wait();  // the pooled keys and the queries may come from the preceding kernel
  if (threadIdx.x == 0) {
    for (int i = 0; i < kD128Boxes; ++i) mbar_init(smem_u32(&full[i]), 1);
    fence_mbar_init();
    for (int i = 0; i < kD128Boxes; ++i) {
      const uint32_t bar = smem_u32(&full[i]);
      mbar_arrive_expect_tx(bar, kD128BoxBytes);
      // rows past the pool's capacity come back as zeros; rows past nwin are
      // scored but not stored
      tma_load_3d(smem_u32(keys + i * kD128BoxBytes), &tm_keys, bar, 32 * i, (int)c0, b);
    }
  }
  // the queries of this sequence, staged while the keys arrive
  const float4* qb = (const float4*)(q + (long long)b * S * 128);
  for (int i = threadIdx.x; i < S8 * 32; i += kD128Threads)
    sq[i] = i < S * 32 ? __ldg(qb + i) : make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();  // the barriers are initialised and the queries staged
  // the selection may be placed now; it waits for this grid before it reads
  pdl_launch_dependents();
  if (!mbar_wait(smem_u32(&full[x]), 0)) {
    // the copy is still owed: record it (the call's scores are then not to be
    // used, and the status word says so) and give it one more bounded wait, as
    // the tile must outlive it; the warp still takes part in the barriers below
    if (lane == 0) atomicCAS(&g_indexer_status, 0, kIndexerWaitSite);
    mbar_wait(smem_u32(&full[x]), 0);
  }
  const uint8_t* row = keys + x * kD128BoxBytes + r * 128;
  for (int s0 = 0; s0 < S; s0 += 8) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.f;
    const float4* qx = sq + s0 * 32 + x * 8;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 kv = *(const float4*)(row + ((c ^ (r & 7)) << 4));
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 qv = qx[j * 32 + c];
        acc[j] = fmaf(kv.x, qv.x, acc[j]);
        acc[j] = fmaf(kv.y, qv.y, acc[j]);
        acc[j] = fmaf(kv.z, qv.z, acc[j]);
        acc[j] = fmaf(kv.w, qv.w, acc[j]);
      }
    }
    if (x > 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) red[((x - 1) * 8 + j) * kD128CtaWindows + r] = acc[j];
    }
    __syncthreads();  // the partial sums of boxes 1..3 are in shared memory
    if (x == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float t = acc[j];
#pragma unroll
        for (int xx = 0; xx < kD128Boxes - 1; ++xx) t += red[(xx * 8 + j) * kD128CtaWindows + r];
        acc[j] = t;
      }
      if (w < nwin) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j < S) scores[((long long)b * S + s0 + j) * nwin + w] = acc[j];
      }
    }
    __syncthreads();  // the partial sums are read before the next group writes them
  }
}

constexpr int kScoreLanes = 8;
constexpr int kScoreWinPerCta = kScoreThreads / kScoreLanes;
constexpr int kScoreMaxVec = kMaxDim / (4 * kScoreLanes);

__global__ void __launch_bounds__(kScoreThreads) score_windows(const float* __restrict__ q,
                                                               const float* __restrict__ pooled,
                                                               long long cap, int dim, int S,
                                                               long long nwin,
                                                               float* __restrict__ scores) {
  extern __shared__ float4 sq4[];  // [S][dim / 4]
  const int b = blockIdx.y;
  const int g = threadIdx.x & (kScoreLanes - 1);
  const long long w = (long long)blockIdx.x * kScoreWinPerCta + (threadIdx.x / kScoreLanes);
  const int nv = dim / (4 * kScoreLanes);
  const bool live = w < nwin;
  pdl_wait();  // the pooled keys and the queries may come from the preceding kernel
  // the key first: its loads are in flight while the queries are staged
  const float4* pk = (const float4*)(pooled + ((long long)b * cap + (live ? w : 0)) * dim) + g;
  float4 kv[kScoreMaxVec];
#pragma unroll
  for (int i = 0; i < kScoreMaxVec; ++i)
    kv[i] = (live && i < nv) ? __ldg(pk + kScoreLanes * i) : make_float4(0.f, 0.f, 0.f, 0.f);
  const int d4 = dim / 4;
  const float4* qb = (const float4*)(q + (long long)b * S * dim);
  for (int i = threadIdx.x; i < S * d4; i += kScoreThreads) sq4[i] = qb[i];
  __syncthreads();
  pdl_launch_dependents();
  const bool h4 = g & 4, h2 = g & 2, h1 = g & 1;
  for (int s0 = 0; s0 < S; s0 += 8) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc[j] = 0.f;
      if (s0 + j < S) {
        const float4* qs = sq4 + (s0 + j) * d4 + g;
#pragma unroll
        for (int i = 0; i < kScoreMaxVec; ++i) {
          if (i < nv) {
            const float4 qv = qs[kScoreLanes * i];
            acc[j] = fmaf(qv.x, kv[i].x, acc[j]);
            acc[j] = fmaf(qv.y, kv[i].y, acc[j]);
            acc[j] = fmaf(qv.z, kv[i].z, acc[j]);
            acc[j] = fmaf(qv.w, kv[i].w, acc[j]);
          }
        }
      }
    }
    float r4[4], r2[2];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float send = h4 ? acc[t] : acc[t + 4];
      r4[t] = (h4 ? acc[t + 4] : acc[t]) + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const float send = h2 ? r4[t] : r4[t + 2];
      r2[t] = (h2 ? r4[t + 2] : r4[t]) + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const float send = h1 ? r2[0] : r2[1];
    const float sc = (h1 ? r2[1] : r2[0]) + __shfl_xor_sync(0xffffffffu, send, 1);
    if (live && s0 + g < S) scores[((long long)b * S + s0 + g) * nwin + w] = sc;
  }
}

// Order-preserving map of a float onto uint32 (larger float, larger key).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kSelThreads = 1024;
constexpr int kSelRun = 32;                        // consecutive windows per thread and round
constexpr int kSelRound = kSelThreads * kSelRun;
constexpr int kSelSmemWindows = 48 * 1024;        // scores staged in shared memory up to this
constexpr int kSelTopBits = 12;                    // first digit: sign, exponent, 3 mantissa bits
constexpr int kSelLowBits = 10;                    // second and third digits
constexpr int kSelCand = 2048;                     // first-digit bucket kept as a list up to this

// Exclusive prefix sum of one value per thread over the CTA; *total receives the sum.
__device__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t t = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_sums[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before = (warp > 0 ? warp_sums[warp - 1] : 0u) + x - v;
  *total = warp_sums[31];
  __syncthreads();
  return before;
}

// The bin holding the `remaining`-th largest key of an nbins-bin histogram,
// counting from the top bin down.  Thread t brings the counts c[0..per) of
// the per = nbins/1024 bins top - 0, ..., top - (per - 1), top = nbins - 1 -
// t * per; one CTA-wide scan of their sums finds the thread whose run crosses
// `remaining`.  Every thread then reads out[0] = that bin, out[1] = how many
// of its keys are still to take, out[1] <= out[2] = its count.
__device__ void find_bucket_counts(const int (&c)[4], int per, int nbins, int remaining,
                                   uint32_t* warp_sums, int* out) {
  const int top = nbins - 1 - (int)threadIdx.x * per;
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) sum += i < per ? c[i] : 0;
  uint32_t total;
  const int excl = (int)block_exclusive_scan((uint32_t)sum, warp_sums, &total);
  if (excl < remaining && excl + sum >= remaining) {
    int cum = excl, pick = 0, cnt = 0;
    bool found = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // constant indices keep c[] in registers
      if (!found && i < per && cum + c[i] >= remaining) {
        found = true;
        pick = i;
        cnt = c[i];
      } else if (!found) {
        cum += i < per ? c[i] : 0;
      }
    }
    out[0] = top - pick;
    out[1] = remaining - cum;
    out[2] = cnt;
  }
  __syncthreads();
}

// The same over a histogram in this CTA's shared memory.
__device__ void find_bucket(const int* hist, int nbins, int remaining, uint32_t* warp_sums,
                            int* out) {
  const int per = nbins / kSelThreads;  // 1 or 4
  const int top = nbins - 1 - (int)threadIdx.x * per;
  int c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = i < per ? hist[top - i] : 0;
  find_bucket_counts(c, per, nbins, remaining, warp_sums, out);
}

// Appends up to four keys per lane to the candidate list: one shared atomic
// per warp, each lane's keys placed after those of the lanes below it.
__device__ __forceinline__ void append_keys(const uint32_t (&key)[4], const bool (&in)[4],
                                            uint32_t* cand, int* ncand) {
  const int lane = threadIdx.x & 31;
  const int c = (int)in[0] + (int)in[1] + (int)in[2] + (int)in[3];
  if (!__any_sync(0xffffffffu, c > 0)) return;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  int base = 0;
  if (lane == 31) base = atomicAdd(ncand, incl);
  base = __shfl_sync(0xffffffffu, base, 31) + incl - c;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (in[e]) cand[base++] = key[e];
}

// Row (b, s): the k best of the windows w <= p/4 (p = len - S + s), ties to
// the lower window; windows listed ascending, then their positions <= p.
// The row's scores are staged in shared memory when they fit (and then read
// four at a time).  The k-th largest is found by a radix select over
// order-preserving keys with digits of 12, 10 and 10 bits.  The first digit
// (sign, exponent and three mantissa bits) spreads the keys over enough bins
// that the shared atomics of one warp seldom collide.  The second pass
// histograms only the keys of the chosen first-digit bucket and, when that
// bucket holds at most 2048 keys, keeps them as a list, so the third pass
// reads the list instead of the row.  Once a chosen bucket is taken whole the
// later digits do not matter and the passes stop.  The output pass gives each
// thread 32 consecutive windows: it marks the keys above and at the
// threshold in two bit masks, one CTA-wide scan of both counts places its
// windows, and it writes them in ascending order.
__global__ void __launch_bounds__(kSelThreads) select_topk(const float* __restrict__ scores,
                                                          long long nwin, int S, long long len,
                                                          int k, int32_t* __restrict__ win_out,
                                                          int32_t* __restrict__ pos_out) {
  extern __shared__ float4 ssc4[];
  __shared__ int hist[1 << kSelTopBits];
  __shared__ uint32_t cand[kSelCand];
  __shared__ uint32_t warp_sums[32];
  __shared__ int sel[3];
  __shared__ int ncand;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.y, s = blockIdx.x;
  const long long p = len - S + s;
  const int vis = (int)(p / kWindow + 1);  // the host keeps windows below 2^31
  const int keff = min(k, vis);
  const long long row = (long long)b * S + s;
  const float* src = scores + row * nwin;
  const bool staged = vis <= kSelSmemWindows;
  pdl_wait();  // the scores come from the preceding kernel
  if (staged) {
    float* ssc = (float*)ssc4;
    int w = threadIdx.x;
    if (((uintptr_t)src & 15) == 0) {
      const float4* s4 = (const float4*)src;
#pragma unroll 4
      for (int i = threadIdx.x; i < vis / 4; i += kSelThreads) ssc4[i] = s4[i];
      w = (vis / 4) * 4 + threadIdx.x;
    }
#pragma unroll 8
    for (; w < vis; w += kSelThreads) ssc[w] = src[w];
    __syncthreads();
    src = ssc;
  }
  // a following call may start its independent loads; it waits for this grid
  pdl_launch_dependents();
  // staged rows are read as float4 up to n4, the rest one key at a time
  const int n4 = staged ? vis / 4 : 0;
  const int tail = 4 * n4;

  // first digit: bits 31..20 of every key
  for (int i = threadIdx.x; i < (1 << kSelTopBits); i += kSelThreads) hist[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n4; i += kSelThreads) {
    const float4 v = ssc4[i];
    atomicAdd(&hist[order_key(v.x) >> (32 - kSelTopBits)], 1);
    atomicAdd(&hist[order_key(v.y) >> (32 - kSelTopBits)], 1);
    atomicAdd(&hist[order_key(v.z) >> (32 - kSelTopBits)], 1);
    atomicAdd(&hist[order_key(v.w) >> (32 - kSelTopBits)], 1);
  }
  for (int w = tail + threadIdx.x; w < vis; w += kSelThreads)
    atomicAdd(&hist[order_key(src[w]) >> (32 - kSelTopBits)], 1);
  __syncthreads();
  find_bucket(hist, 1 << kSelTopBits, keff, warp_sums, sel);
  constexpr int kShift2 = 32 - kSelTopBits - kSelLowBits;
  constexpr uint32_t kLowMask = (1u << kSelLowBits) - 1;
  uint32_t prefix = (uint32_t)sel[0] << (32 - kSelTopBits);
  uint32_t mask = ~0u << (32 - kSelTopBits);
  int remaining = sel[1];
  bool whole = sel[2] == remaining;
  const bool use_list = sel[2] <= kSelCand;

  // second digit: bits 19..10 of the keys in the chosen bucket
  if (!whole) {
    hist[threadIdx.x] = 0;  // 1024 bins, one per thread
    if (threadIdx.x == 0) ncand = 0;
    __syncthreads();
    // warp-uniform loops, so that a warp appends its keys together
    for (int i0 = threadIdx.x - lane; i0 < n4; i0 += kSelThreads) {
      const int i = i0 + lane;
      uint32_t key[4] = {0u, 0u, 0u, 0u};
      bool in[4] = {false, false, false, false};
      if (i < n4) {
        const float4 v = ssc4[i];
        key[0] = order_key(v.x);
        key[1] = order_key(v.y);
        key[2] = order_key(v.z);
        key[3] = order_key(v.w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          in[e] = (key[e] & mask) == prefix;
          if (in[e]) atomicAdd(&hist[(key[e] >> kShift2) & kLowMask], 1);
        }
      }
      if (use_list) append_keys(key, in, cand, &ncand);
    }
    for (int w0 = tail + threadIdx.x - lane; w0 < vis; w0 += kSelThreads) {
      const int w = w0 + lane;
      uint32_t key[4] = {0u, 0u, 0u, 0u};
      bool in[4] = {false, false, false, false};
      if (w < vis) {
        key[0] = order_key(src[w]);
        in[0] = (key[0] & mask) == prefix;
        if (in[0]) atomicAdd(&hist[(key[0] >> kShift2) & kLowMask], 1);
      }
      if (use_list) append_keys(key, in, cand, &ncand);
    }
    __syncthreads();
    find_bucket(hist, 1 << kSelLowBits, remaining, warp_sums, sel);
    prefix |= (uint32_t)sel[0] << kShift2;
    mask |= kLowMask << kShift2;
    remaining = sel[1];
    whole = sel[2] == remaining;
  }

  // third digit: bits 9..0
  if (!whole) {
    hist[threadIdx.x] = 0;
    __syncthreads();
    if (use_list) {
      const int nc = ncand;
      for (int i = threadIdx.x; i < nc; i += kSelThreads) {
        const uint32_t key = cand[i];
        if ((key & mask) == prefix) atomicAdd(&hist[key & kLowMask], 1);
      }
    } else {
      for (int w = threadIdx.x; w < vis; w += kSelThreads) {
        const uint32_t key = order_key(src[w]);
        if ((key & mask) == prefix) atomicAdd(&hist[key & kLowMask], 1);
      }
    }
    __syncthreads();
    find_bucket(hist, 1 << kSelLowBits, remaining, warp_sums, sel);
    prefix |= (uint32_t)sel[0];
    mask = ~0u;
    remaining = sel[1];
  }

  // Keys whose digits under `mask` exceed `prefix` are taken; of those equal to
  // it, the first `remaining` (lowest windows first).
  const bool vec_pos = ((uintptr_t)pos_out & 15) == 0;
  int taken_before = 0, eq_before = 0;
  for (int r0 = 0; r0 < vis; r0 += kSelRound) {
    const int w0 = r0 + (int)threadIdx.x * kSelRun;
    uint32_t gtm = 0, eqm = 0;
    if (staged && w0 + kSelRun <= vis) {
#pragma unroll
      for (int e = 0; e < kSelRun / 4; ++e) {
        const int j = (e + lane) & (kSelRun / 4 - 1);  // rotated: eight lanes hit 32 banks
        const float4 v = ssc4[w0 / 4 + j];
        const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t key = order_key(f[c]) & mask;
          gtm |= (uint32_t)(key > prefix) << (4 * j + c);
          eqm |= (uint32_t)(key == prefix) << (4 * j + c);
        }
      }
    } else {
#pragma unroll 8
      for (int e = 0; e < kSelRun; ++e) {
        const int j = (e + lane) & (kSelRun - 1);  // rotated, so a warp's reads hit 32 banks
        if (w0 + j < vis) {
          const uint32_t key = order_key(src[w0 + j]) & mask;
          gtm |= (uint32_t)(key > prefix) << j;
          eqm |= (uint32_t)(key == prefix) << j;
        }
      }
    }
    const int gt = __popc(gtm), eq = __popc(eqm);
    uint32_t tot;
    const uint32_t pre = block_exclusive_scan(((uint32_t)gt << 16) | (uint32_t)eq, warp_sums, &tot);
    const int gt_pre = (int)(pre >> 16), eq_pre = (int)(pre & 0xffffu);
    const int rem_eq = max(0, remaining - eq_before);
    const int eq_take = max(0, min(eq, rem_eq - eq_pre));
    int o = taken_before + gt_pre + min(eq_pre, rem_eq);
    uint32_t takem = gtm;
    for (uint32_t m = eqm, n = 0; n < (uint32_t)eq_take; ++n) {
      takem |= m & (0u - m);  // lowest remaining equal key
      m &= m - 1;
    }
    while (takem) {
      const int j = __ffs(takem) - 1;
      takem &= takem - 1;
      const long long w = w0 + j;
      if (win_out) win_out[row * k + o] = (int32_t)w;
      int32_t pv[kWindow];
#pragma unroll
      for (int i = 0; i < kWindow; ++i) {
        const long long tpos = kWindow * w + i;
        pv[i] = tpos <= p ? (int32_t)tpos : -1;
      }
      int32_t* dst = pos_out + row * (long long)kWindow * k + (long long)kWindow * o;
      if (vec_pos) {
        *(int4*)dst = make_int4(pv[0], pv[1], pv[2], pv[3]);
      } else {
#pragma unroll
        for (int i = 0; i < kWindow; ++i) dst[i] = pv[i];
      }
      ++o;
    }
    taken_before += (int)(tot >> 16) + min((int)(tot & 0xffffu), rem_eq);
    eq_before += (int)(tot & 0xffffu);
  }
  // padding past the chosen windows
  for (int j = taken_before + threadIdx.x; j < k; j += kSelThreads) {
    if (win_out) win_out[row * k + j] = -1;
#pragma unroll
    for (int i = 0; i < kWindow; ++i) pos_out[row * (long long)kWindow * k + kWindow * j + i] = -1;
  }
}

// The same selection with a row spread over a cluster of eight CTAs: CTA r
// stages and scans windows [r * slice, (r + 1) * slice) of the row.  The
// first digit (10 bits) is histogrammed in every CTA's shared memory for its
// own slice; after a cluster barrier every CTA sums the eight histograms bin
// by bin through distributed shared memory, so all eight take the same
// decision.  Each CTA then compacts its slice's keys of the chosen bucket,
// and after one more barrier every CTA gathers all eight lists (at most 2048
// keys) and takes the last two digits (11 bits each) locally.  A bucket too
// large to gather has those digits summed over the cluster like the first.
// In the output pass a CTA's windows are placed after those its lower-ranked
// peers take, from the peers' totals (one more exchange).
constexpr int kSelCluster = 8;
constexpr int kSelClusterSlice = kSelThreads * 32;  // windows a CTA stages, at most
constexpr int kClD1 = 10;                           // digits of the cluster form: 10, 11, 11 bits
constexpr int kClD2 = 11;
constexpr int kClCand = 2048;                       // a chosen bucket gathered whole up to this

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint2 ld_cluster_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// This thread's top-down bin counts (as find_bucket_counts takes them),
// summed over the histograms at the same address in every CTA of the cluster.
__device__ __forceinline__ void cluster_counts(const int* hist, int nbins, int (&c)[4]) {
  const int per = nbins / kSelThreads;
  const int top = nbins - 1 - (int)threadIdx.x * per;
  c[0] = c[1] = c[2] = c[3] = 0;
  // every load is issued before the first sum, so the eight remote reads overlap
  if (per == 4) {
    const uint32_t a = smem_u32(hist + top - 3);  // bins top-3 .. top, 16-byte aligned
    uint4 v[kSelCluster];
#pragma unroll
    for (int r = 0; r < kSelCluster; ++r) v[r] = ld_cluster_v4(mapa(a, r));
#pragma unroll
    for (int r = 0; r < kSelCluster; ++r) {
      c[0] += (int)v[r].w;
      c[1] += (int)v[r].z;
      c[2] += (int)v[r].y;
      c[3] += (int)v[r].x;
    }
  } else if (per == 2) {
    const uint32_t a = smem_u32(hist + top - 1);  // bins top-1, top, 8-byte aligned
    uint2 v[kSelCluster];
#pragma unroll
    for (int r = 0; r < kSelCluster; ++r) v[r] = ld_cluster_v2(mapa(a, r));
#pragma unroll
    for (int r = 0; r < kSelCluster; ++r) {
      c[0] += (int)v[r].y;
      c[1] += (int)v[r].x;
    }
  } else {
    const uint32_t a = smem_u32(hist + top);
    uint32_t v[kSelCluster];
#pragma unroll
    for (int r = 0; r < kSelCluster; ++r) v[r] = ld_cluster_u32(mapa(a, r));
#pragma unroll
    for (int r = 0; r < kSelCluster; ++r) c[0] += (int)v[r];
  }
}

// One CTA per SM (the bound lets the registers grow from 32 to 47): two of
// these 1024-thread CTAs on one SM, from different clusters, had made the
// scoring-then-selection call 20 instead of 16.5 µs.
__global__ void __launch_bounds__(kSelThreads, 1) select_topk_cluster(
    const float* __restrict__ scores, long long nwin, int S, long long len, int k,
    int32_t* __restrict__ win_out, int32_t* __restrict__ pos_out) {
  extern __shared__ float4 ssc4[];  // this CTA's slice of the row
  __shared__ __align__(16) int hist_a[1 << kClD2];
  __shared__ __align__(16) int hist_b[1 << kClD2];
  __shared__ uint32_t cand[kClCand];      // this slice's keys of the chosen bucket
  __shared__ uint32_t all_cand[kClCand];  // every slice's, gathered
  __shared__ uint32_t warp_sums[32];
  __shared__ int sel[3];
  __shared__ int ncand;
  __shared__ int cta_tot[2];
  const int lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();
  const int s = blockIdx.y, b = blockIdx.z;
  const long long p = len - S + s;
  const int vis = (int)(p / kWindow + 1);
  const int keff = min(k, vis);
  const long long row = (long long)b * S + s;
  const int slice = ((vis + kSelCluster - 1) / kSelCluster + 3) & ~3;
  const int lo = min(vis, rank * slice);
  const int nloc = min(vis, lo + slice) - lo;
  float* ssc = (float*)ssc4;
  const float* src = scores + row * nwin + lo;
  pdl_wait();  // the scores come from the preceding kernel
#pragma unroll 4
  for (int i = threadIdx.x; i < nloc; i += kSelThreads) ssc[i] = src[i];
  for (int i = threadIdx.x; i < (1 << kClD1); i += kSelThreads) hist_a[i] = 0;
  __syncthreads();
  // a following call may start its independent loads; it waits for this grid
  pdl_launch_dependents();
  const int n4 = nloc / 4, tail = 4 * n4;

  // first digit: bits 31..22 (sign, exponent, one mantissa bit), summed over
  // the cluster: 1024 bins, so each CTA reads 32 KB of its peers' counts
  for (int i = threadIdx.x; i < n4; i += kSelThreads) {
    const float4 v = ssc4[i];
    atomicAdd(&hist_a[order_key(v.x) >> (32 - kClD1)], 1);
    atomicAdd(&hist_a[order_key(v.y) >> (32 - kClD1)], 1);
    atomicAdd(&hist_a[order_key(v.z) >> (32 - kClD1)], 1);
    atomicAdd(&hist_a[order_key(v.w) >> (32 - kClD1)], 1);
  }
  for (int w = tail + threadIdx.x; w < nloc; w += kSelThreads)
    atomicAdd(&hist_a[order_key(ssc[w]) >> (32 - kClD1)], 1);
  cluster_sync();  // every slice's histogram is complete
  int c[4];
  cluster_counts(hist_a, 1 << kClD1, c);
  find_bucket_counts(c, 1, 1 << kClD1, keff, warp_sums, sel);
  constexpr int kShift2 = 32 - kClD1 - kClD2;
  constexpr uint32_t kLowMask = (1u << kClD2) - 1;
  uint32_t prefix = (uint32_t)sel[0] << (32 - kClD1);
  uint32_t mask = ~0u << (32 - kClD1);
  int remaining = sel[1];
  bool whole = sel[2] == remaining;
  const bool gather = sel[2] <= kClCand;  // the same decision in every CTA

  if (!whole && gather) {
    // The bucket's keys of every slice, gathered into each CTA: the last two
    // digits are then taken locally, with no more cluster barriers.
    hist_b[threadIdx.x] = 0;
    hist_b[threadIdx.x + kSelThreads] = 0;
    if (threadIdx.x == 0) ncand = 0;
    __syncthreads();
    for (int i0 = threadIdx.x - lane; i0 < n4; i0 += kSelThreads) {
      const int i = i0 + lane;
      uint32_t key[4] = {0u, 0u, 0u, 0u};
      bool in[4] = {false, false, false, false};
      if (i < n4) {
        const float4 v = ssc4[i];
        key[0] = order_key(v.x);
        key[1] = order_key(v.y);
        key[2] = order_key(v.z);
        key[3] = order_key(v.w);
#pragma unroll
        for (int e = 0; e < 4; ++e) in[e] = (key[e] & mask) == prefix;
      }
      append_keys(key, in, cand, &ncand);
    }
    for (int w0 = tail + threadIdx.x - lane; w0 < nloc; w0 += kSelThreads) {
      const int w = w0 + lane;
      uint32_t key[4] = {0u, 0u, 0u, 0u};
      bool in[4] = {false, false, false, false};
      if (w < nloc) {
        key[0] = order_key(ssc[w]);
        in[0] = (key[0] & mask) == prefix;
      }
      append_keys(key, in, cand, &ncand);
    }
    cluster_sync();  // every slice's list is complete
    // lane r of each warp reads slice r's count; its list starts at the
    // exclusive prefix of the counts
    const int cnt = lane < kSelCluster ? (int)ld_cluster_u32(mapa(smem_u32(&ncand), lane)) : 0;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < kSelCluster; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int n_all = __shfl_sync(0xffffffffu, incl, kSelCluster - 1);
    int offs[kSelCluster];
#pragma unroll
    for (int r = 0; r < kSelCluster; ++r) offs[r] = __shfl_sync(0xffffffffu, incl - cnt, r);
    // at most two keys per thread; both loads are issued before either store
    uint32_t got[kClCand / kSelThreads];
#pragma unroll
    for (int u = 0; u < kClCand / kSelThreads; ++u) {
      const int j = threadIdx.x + u * kSelThreads;
      got[u] = 0u;
      if (j < n_all) {
        int rr = 0, base = 0;  // the last list starting at or before j
#pragma unroll
        for (int r = 1; r < kSelCluster; ++r) {
          if (j >= offs[r]) {
            rr = r;
            base = offs[r];
          }
        }
        got[u] = ld_cluster_u32(mapa(smem_u32(cand + (j - base)), rr));
      }
    }
#pragma unroll
    for (int u = 0; u < kClCand / kSelThreads; ++u) {
      const int j = threadIdx.x + u * kSelThreads;
      if (j < n_all) all_cand[j] = got[u];
    }
    __syncthreads();
    // second digit: bits 21..11 of the gathered keys
    for (int i = threadIdx.x; i < n_all; i += kSelThreads)
      atomicAdd(&hist_b[(all_cand[i] >> kShift2) & kLowMask], 1);
    __syncthreads();
    find_bucket(hist_b, 1 << kClD2, remaining, warp_sums, sel);
    prefix |= (uint32_t)sel[0] << kShift2;
    mask |= kLowMask << kShift2;
    remaining = sel[1];
    whole = sel[2] == remaining;
    if (!whole) {
      // third digit: bits 10..0
      hist_a[threadIdx.x] = 0;
      hist_a[threadIdx.x + kSelThreads] = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < n_all; i += kSelThreads) {
        const uint32_t key = all_cand[i];
        if ((key & mask) == prefix) atomicAdd(&hist_a[key & kLowMask], 1);
      }
      __syncthreads();
      find_bucket(hist_a, 1 << kClD2, remaining, warp_sums, sel);
      prefix |= (uint32_t)sel[0];
      mask = ~0u;
      remaining = sel[1];
    }
  } else if (!whole) {
    // A bucket too large to gather: the last two digits are summed over the
    // cluster like the first (2048 bins each).
    hist_b[threadIdx.x] = 0;
    hist_b[threadIdx.x + kSelThreads] = 0;
    __syncthreads();
    for (int w = threadIdx.x; w < nloc; w += kSelThreads) {
      const uint32_t key = order_key(ssc[w]);
      if ((key & mask) == prefix) atomicAdd(&hist_b[(key >> kShift2) & kLowMask], 1);
    }
    cluster_sync();
    cluster_counts(hist_b, 1 << kClD2, c);
    find_bucket_counts(c, 2, 1 << kClD2, remaining, warp_sums, sel);
    prefix |= (uint32_t)sel[0] << kShift2;
    mask |= kLowMask << kShift2;
    remaining = sel[1];
    whole = sel[2] == remaining;
    if (!whole) {
      // in the bins of hist_a: every peer read them before it arrived on
      // the barrier that ended the second digit
      hist_a[threadIdx.x] = 0;
      hist_a[threadIdx.x + kSelThreads] = 0;
      __syncthreads();
      for (int w = threadIdx.x; w < nloc; w += kSelThreads) {
        const uint32_t key = order_key(ssc[w]);
        if ((key & mask) == prefix) atomicAdd(&hist_a[key & kLowMask], 1);
      }
      cluster_sync();
      cluster_counts(hist_a, 1 << kClD2, c);
      find_bucket_counts(c, 2, 1 << kClD2, remaining, warp_sums, sel);
      prefix |= (uint32_t)sel[0];
      mask = ~0u;
      remaining = sel[1];
    }
  }

  // output: thread t marks windows [t * run, (t + 1) * run) of the slice
  const int run = 4 * ((nloc + 4 * kSelThreads - 1) / (4 * kSelThreads));  // <= 32
  const int t0 = (int)threadIdx.x * run;
  uint32_t gtm = 0, eqm = 0;
  if (run > 0 && t0 + run <= nloc) {
    const int q4 = run / 4;
    for (int e = 0; e < q4; ++e) {
      const int j = (e + lane) % q4;  // rotated across the lanes
      const float4 v = ssc4[t0 / 4 + j];
      const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const uint32_t key = order_key(f[cc]) & mask;
        gtm |= (uint32_t)(key > prefix) << (4 * j + cc);
        eqm |= (uint32_t)(key == prefix) << (4 * j + cc);
      }
    }
  } else {
    for (int j = 0; j < run && t0 + j < nloc; ++j) {
      const uint32_t key = order_key(ssc[t0 + j]) & mask;
      gtm |= (uint32_t)(key > prefix) << j;
      eqm |= (uint32_t)(key == prefix) << j;
    }
  }
  const int gt = __popc(gtm), eq = __popc(eqm);
  uint32_t tot;
  const uint32_t pre = block_exclusive_scan(((uint32_t)gt << 16) | (uint32_t)eq, warp_sums, &tot);
  if (threadIdx.x == 0) {
    cta_tot[0] = (int)(tot >> 16);
    cta_tot[1] = (int)(tot & 0xffffu);
  }
  cluster_sync();  // every CTA's totals are published
  // lane r < rank reads peer r's totals; a warp sum gives every lane the lot
  int gt_before = 0, eq_before = 0;
  if (lane < rank) {
    gt_before = (int)ld_cluster_u32(mapa(smem_u32(&cta_tot[0]), lane));
    eq_before = (int)ld_cluster_u32(mapa(smem_u32(&cta_tot[1]), lane));
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    gt_before += __shfl_xor_sync(0xffffffffu, gt_before, o);
    eq_before += __shfl_xor_sync(0xffffffffu, eq_before, o);
  }
  cluster_arrive();  // done with the peers' shared memory; wait for theirs at the end
  const int gt_pre = (int)(pre >> 16), eq_pre = (int)(pre & 0xffffu);
  const int rem_eq = max(0, remaining - eq_before);
  const int eq_take = max(0, min(eq, rem_eq - eq_pre));
  int o = gt_before + min(eq_before, remaining) + gt_pre + min(eq_pre, rem_eq);
  uint32_t takem = gtm;
  for (uint32_t m = eqm, n = 0; n < (uint32_t)eq_take; ++n) {
    takem |= m & (0u - m);
    m &= m - 1;
  }
  const bool vec_pos = ((uintptr_t)pos_out & 15) == 0;
  while (takem) {
    const int j = __ffs(takem) - 1;
    takem &= takem - 1;
    const long long w = (long long)lo + t0 + j;
    if (win_out) win_out[row * k + o] = (int32_t)w;
    int32_t pv[kWindow];
#pragma unroll
    for (int i = 0; i < kWindow; ++i) {
      const long long tpos = kWindow * w + i;
      pv[i] = tpos <= p ? (int32_t)tpos : -1;
    }
    int32_t* dst = pos_out + row * (long long)kWindow * k + (long long)kWindow * o;
    if (vec_pos) {
      *(int4*)dst = make_int4(pv[0], pv[1], pv[2], pv[3]);
    } else {
#pragma unroll
      for (int i = 0; i < kWindow; ++i) dst[i] = pv[i];
    }
    ++o;
  }
  // padding past the keff chosen windows
  if (rank == kSelCluster - 1) {
    for (int j = keff + threadIdx.x; j < k; j += kSelThreads) {
      if (win_out) win_out[row * k + j] = -1;
#pragma unroll
      for (int i = 0; i < kWindow; ++i) pos_out[row * (long long)kWindow * k + kWindow * j + i] = -1;
    }
  }
  cluster_wait();
}

// Per-device launch setup of the scoring and selection kernels (the opt-ins
// to more than 48 KB of shared memory, and whether a cluster of eight 1024-thread
// CTAs fits the device), made once per device; calls may come from several
// threads.
struct SelectSetup {
  cudaError_t err = cudaSuccess;
  bool cluster_ok = false;
};
SelectSetup select_setup() {
  static std::mutex mu;
  static bool done[64] = {};
  static SelectSetup setups[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    SelectSetup bad;
    bad.err = cudaErrorInvalidDevice;
    return bad;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    SelectSetup su;
    su.err = cudaFuncSetAttribute(select_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSelSmemWindows * (int)sizeof(float));
    if (su.err == cudaSuccess)
      su.err = cudaFuncSetAttribute(score_windows_d128, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    d128_smem_bytes(kMaxNewTokens));
    if (su.err == cudaSuccess &&
        cudaFuncSetAttribute(select_topk_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSelClusterSlice * (int)sizeof(float)) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kSelCluster;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(kSelCluster, 1, 1);
      cfg.blockDim = dim3(kSelThreads, 1, 1);
      cfg.dynamicSmemBytes = kSelClusterSlice * sizeof(float);
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      su.cluster_ok =
          cudaOccupancyMaxActiveClusters(&n, select_topk_cluster, &cfg) == cudaSuccess && n > 0;
    }
    cudaGetLastError();  // a device without room for the cluster is not an error
    setups[dev] = su;
    done[dev] = true;
  }
  return setups[dev];
}

}  // namespace

int indexer_device_status(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_indexer_status, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v != 0) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_indexer_status, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

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
    const size_t esz = dtype == MLA_DTYPE_BF16 ? 2 : 4;
    const bool vec = (dim / 32) % 4 == 0 && key_row_stride % 4 == 0 &&
                     (uintptr_t)keys % (4 * esz) == 0 && (uintptr_t)pooled % 16 == 0;
    KernelTimer kt("indexer_pool_windows", st);
    // chained to the preceding kernel (programmatic dependent launch)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const long long len = cache_len, first = w0, last = nwin, cap = pooled_windows_cap;
    if (dtype == MLA_DTYPE_BF16)
      e = cudaLaunchKernelEx(&cfg, pool_windows<__nv_bfloat16>, (const __nv_bfloat16*)keys,
                             (long long)key_row_stride, (long long)seq_stride_rows, (int)dim, len,
                             first, last, pooled, cap, vec);
    else
      e = cudaLaunchKernelEx(&cfg, pool_windows<float>, (const float*)keys,
                             (long long)key_row_stride, (long long)seq_stride_rows, (int)dim, len,
                             first, last, pooled, cap, vec);
    if (e == cudaSuccess) e = cudaGetLastError();
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
  if (nwin > (1LL << 30)) {
    set_error("a cache of %lld tokens has more than 2^30 windows", (long long)cache_len);
    return MLA_ERR_INVALID_ARG;
  }
  if (pooled_windows_cap < nwin) {
    set_error("the pool holds %lld windows; a cache of %lld tokens fills %lld",
              (long long)pooled_windows_cap, (long long)cache_len, nwin);
    return MLA_ERR_INVALID_ARG;
  }
  if (((uintptr_t)q | (uintptr_t)pooled) & 15) {
    set_error("q and pooled must be 16-byte aligned (the scoring kernel reads them as float4)");
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
  const SelectSetup setup = select_setup();
  if (setup.err != cudaSuccess) {
    set_error("CUDA error %d (%s)", (int)setup.err, cudaGetErrorString(setup.err));
    return MLA_ERR_CUDA;
  }
  CUtensorMap tm_keys;
  if (dim == 128 &&
      !make_tmap_f32_3d(&tm_keys, pooled, 128, (uint64_t)pooled_windows_cap, (uint64_t)batch, 512,
                        (uint64_t)pooled_windows_cap * 512, 32, kD128CtaWindows)) {
    set_error("the pooled keys' tensor map could not be encoded");
    return MLA_ERR_CUDA;
  }
  {
    KernelTimer kt("indexer_score_windows", st);
    // chained to the preceding kernel (programmatic dependent launch)
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dim == 128) {
      cfg.gridDim = dim3((unsigned)((nwin + kD128CtaWindows - 1) / kD128CtaWindows), batch);
      cfg.blockDim = dim3(kD128Threads);
      cfg.dynamicSmemBytes = d128_smem_bytes(new_tokens);
      cudaLaunchKernelEx(&cfg, score_windows_d128, tm_keys, q, (int)new_tokens, (long long)nwin,
                         scores);
    } else {
      cfg.gridDim = dim3((unsigned)((nwin + kScoreWinPerCta - 1) / kScoreWinPerCta), batch);
      cfg.blockDim = dim3(kScoreThreads);
      cfg.dynamicSmemBytes = (size_t)new_tokens * dim * sizeof(float);
      cudaLaunchKernelEx(&cfg, score_windows, q, pooled, (long long)pooled_windows_cap,
                         (int)dim, (int)new_tokens, (long long)nwin, scores);
    }
  }
  {
    KernelTimer kt("indexer_select_topk", st);
    const long long vis_max = (cache_len - 1) / kWindow + 1;
    const size_t sel_smem = vis_max <= kSelSmemWindows ? (size_t)vis_max * sizeof(float) : 0;
    // a cluster of eight CTAs per row when its slices fit and the device
    // can hold such a cluster; otherwise one CTA per row
    const bool cluster_ok = setup.cluster_ok;
    const long long slice_max = ((vis_max + kSelCluster - 1) / kSelCluster + 3) & ~3LL;
    if (cluster_ok && slice_max <= kSelClusterSlice) {
      // chained to the scoring kernel (programmatic dependent launch)
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kSelCluster;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.gridDim = dim3(kSelCluster, new_tokens, batch);
      cfg.blockDim = dim3(kSelThreads, 1, 1);
      cfg.dynamicSmemBytes = (size_t)slice_max * sizeof(float);
      cfg.stream = st;
      cfg.attrs = attr;
      cfg.numAttrs = 2;
      cudaLaunchKernelEx(&cfg, select_topk_cluster, (const float*)scores, (long long)nwin,
                         (int)new_tokens, (long long)cache_len, (int)k_windows, windows_out,
                         positions_out);
    } else {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.gridDim = dim3(new_tokens, batch, 1);
      cfg.blockDim = dim3(kSelThreads, 1, 1);
      cfg.dynamicSmemBytes = sel_smem;
      cfg.stream = st;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      cudaLaunchKernelEx(&cfg, select_topk, (const float*)scores, (long long)nwin,
                         (int)new_tokens, (long long)cache_len, (int)k_windows, windows_out,
                         positions_out);
    }
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}
