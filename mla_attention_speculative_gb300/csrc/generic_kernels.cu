// Generic MLA verify kernels on CUDA cores, for any geometry, fp32 or bf16
// inputs, fp32 arithmetic.  They are the fp32 path (tensor cores have no
// full-precision fp32 mode) and the path for geometries the tensor-core
// kernels do not cover.
//
// Both branches follow "One guard, 110x off the verify step", section "The
// defect": absorbed = fold W_UK into the query, attend against the latent,
// unembed with W_UV; materialised = expand the latent to per-head K and V,
// then attend.  Row l of a sequence of T cached positions sees t <= T-L+l.
//
// Layout of the split-KV partials (fp32, in the caller's workspace):
//   O_part [B, splits, L*H, Dv]   un-normalised sum of exp(s - m) * value
//   ml     [B, splits, L*H, 2]    (m, l): running max and sum of exp(s - m)
// Sequence b uses ceil(T_b / chunk) pieces; pieces past that are never read.
//
// Sparse (top-k) calls ("One guard, 110x off the verify step", section "The
// sparse model is different": attention runs over the positions an indexer
// selected) replace the position range of a row by its index list: verify
// row l of sequence b reads topk[b, l, 0..k), an entry used when
// 0 <= t <= T_b - L + l; pieces split the list, ceil(k / chunk) of them.

#include <cuda_bf16.h>

#include <cfloat>

#include "mla_internal.h"

namespace mla {

static __device__ int g_generic_status;

namespace {

__device__ __forceinline__ void report_bad_page() { atomicCAS(&g_generic_status, 0, kBadPageSite); }

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float* p, float x) { *p = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

constexpr int kMaxPerLane = 16;   // 512 / 32: widest dot or value row per warp lane
constexpr int kMaxRopeLane = 4;   // 128 / 32

// ---------------------------------------------------------------------------
// Fold: q_lat[row, h, :] = q_nope[row, h, :] . W_UK[h]      (n -> r), row = b*L + l
// ---------------------------------------------------------------------------
template <typename T, int ROWS>
__global__ void fold_kernel(const T* __restrict__ q_nope, const T* __restrict__ W_UK,
                            float* __restrict__ q_lat, int BL, int H, int n, int r) {
  extern __shared__ float sq[];  // [ROWS][n]
  const int h = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  const int row0 = blockIdx.z * ROWS;
  const int nrows = min(ROWS, BL - row0);
  for (int idx = threadIdx.x; idx < ROWS * n; idx += blockDim.x) {
    const int rr = idx / n, i = idx - rr * n;
    sq[idx] = rr < nrows ? to_f(q_nope[((size_t)(row0 + rr) * H + h) * n + i]) : 0.f;
  }
  __syncthreads();
  if (j >= r) return;
  float acc[ROWS];
#pragma unroll
  for (int rr = 0; rr < ROWS; ++rr) acc[rr] = 0.f;
  const T* w = W_UK + (size_t)h * n * r + j;
  for (int i = 0; i < n; ++i) {
    const float wi = to_f(w[(size_t)i * r]);
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) acc[rr] = fmaf(sq[rr * n + i], wi, acc[rr]);
  }
  for (int rr = 0; rr < nrows; ++rr) q_lat[((size_t)(row0 + rr) * H + h) * r + j] = acc[rr];
}

// ---------------------------------------------------------------------------
// Row-wise split-KV attention with an online softmax, one warp per query row.
//   absorbed:     key = [c_kv[t] || k_rope[t]], value = c_kv[t], query = [q_lat || q_rope]
//   materialised: key = [K_nope[t,h] || k_rope[t]], value = V[t,h], query = [q_nope || q_rope]
// ---------------------------------------------------------------------------
struct AttnParams {
  const void* q_main;       // absorbed: float q_lat [B*L*H, r]; materialised: T q_nope [B,L,H,n]
  const void* q_rope;       // T [B,L,H,rope]
  CacheView cache;
  const void* kexp;         // materialised: T [B, Tmax, H, n+v]
  const int32_t* lens;
  const int32_t* topk;      // sparse: [B, L, topk_k] positions, else NULL
  int topk_k;
  int L, H, Dm, rope, Dv, n_plus_v, Tmax;
  float scale;
  int chunk, splits;
  float* o_part;
  float* ml;
};

template <typename T, bool ABSORBED>
__global__ void __launch_bounds__(128) attn_rows_kernel(AttnParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, s = blockIdx.y;
  const int LH = p.L * p.H;
  const int row = blockIdx.x * 4 + warp;
  const int Tb = p.lens[b];
  const int klen = p.topk ? p.topk_k : Tb;  // positions (or list entries) to split
  const int nsplit = (klen + p.chunk - 1) / p.chunk;
  if (s >= nsplit || row >= LH) return;
  const int l = row / p.H, h = row - l * p.H;
  const int last = Tb - p.L + l;  // last visible position of this row
  const int t0 = s * p.chunk;
  const int t1 = p.topk ? min(t0 + p.chunk, klen) : min(min(t0 + p.chunk, Tb), last + 1);
  const int32_t* list = p.topk ? p.topk + ((size_t)b * p.L + l) * p.topk_k : nullptr;

  const int km = p.Dm / 32, kr = p.rope / 32, kv = p.Dv / 32;
  const int rm = p.Dm - km * 32, rr = p.rope - kr * 32, rvv = p.Dv - kv * 32;  // ragged tails
  float qm[kMaxPerLane + 1], qr[kMaxRopeLane + 1], o[kMaxPerLane + 1];
  const size_t qrow = (size_t)b * LH + row;
#pragma unroll
  for (int k = 0; k <= kMaxPerLane; ++k) {
    qm[k] = 0.f;
    o[k] = 0.f;
    const int d = lane + 32 * k;
    if (k < km || (k == km && lane < rm)) {
      if (ABSORBED) qm[k] = ((const float*)p.q_main)[qrow * p.Dm + d];
      else qm[k] = to_f(((const T*)p.q_main)[qrow * p.Dm + d]);
    }
  }
#pragma unroll
  for (int k = 0; k <= kMaxRopeLane; ++k) {
    qr[k] = 0.f;
    const int d = lane + 32 * k;
    if (k < kr || (k == kr && lane < rr)) qr[k] = to_f(((const T*)p.q_rope)[qrow * p.rope + d]);
  }

  float m = -FLT_MAX, lsum = 0.f;
  const T* ckv = (const T*)p.cache.c_kv;
  const T* krp = (const T*)p.cache.k_rope;
  bool any = false;
  for (int j = t0; j < t1; ++j) {
    int t = j;
    if (list) {
      t = list[j];
      if (t < 0 || t > last) continue;  // padding, or past the row's causal limit
    }
    any = true;
    const int64_t crow = cache_row(p.cache, b, t);
    if (crow < 0) {  // page id out of range: the position is left out
      if (lane == 0) report_bad_page();
      continue;
    }
    const T* kmain;
    const T* vrow;
    if (ABSORBED) {
      kmain = ckv + crow * p.cache.ckv_stride;
      vrow = kmain;
    } else {
      kmain = (const T*)p.kexp + (((size_t)b * p.Tmax + t) * p.H + h) * p.n_plus_v;
      vrow = kmain + p.Dm;
    }
    const T* krow = krp + crow * p.cache.kr_stride;
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k <= kMaxPerLane; ++k) {
      const int d = lane + 32 * k;
      if (k < km || (k == km && lane < rm)) dot = fmaf(qm[k], to_f(kmain[d]), dot);
    }
#pragma unroll
    for (int k = 0; k <= kMaxRopeLane; ++k) {
      const int d = lane + 32 * k;
      if (k < kr || (k == kr && lane < rr)) dot = fmaf(qr[k], to_f(krow[d]), dot);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    const float sc = dot * p.scale;
    const float mn = fmaxf(m, sc);
    const float corr = __expf(m - mn);
    const float pe = __expf(sc - mn);
    lsum = lsum * corr + pe;
#pragma unroll
    for (int k = 0; k <= kMaxPerLane; ++k) {
      const int d = lane + 32 * k;
      if (k < kv || (k == kv && lane < rvv)) o[k] = fmaf(pe, to_f(vrow[d]), o[k] * corr);
    }
    m = mn;
  }
  const size_t prow = ((size_t)b * p.splits + s) * LH + row;
  float* op = p.o_part + prow * p.Dv;
#pragma unroll
  for (int k = 0; k <= kMaxPerLane; ++k) {
    const int d = lane + 32 * k;
    if (k < kv || (k == kv && lane < rvv)) op[d] = o[k];
  }
  if (lane == 0) {
    p.ml[prow * 2 + 0] = any ? m : -FLT_MAX;
    p.ml[prow * 2 + 1] = lsum;
  }
}

// Log-sum-exp merge weights of the pieces of one query row: returns 1/sum_s w_s l_s
// and leaves M (the largest piece max) in *M_out.
__device__ __forceinline__ float merge_norm(const float* ml, size_t stride_rows, int nsplit,
                                            float* M_out) {
  float M = -FLT_MAX;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ml[s * stride_rows * 2]);
  float den = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ls = ml[s * stride_rows * 2 + 1];
    if (ls > 0.f) den += __expf(ml[s * stride_rows * 2] - M) * ls;
  }
  *M_out = M;
  return 1.f / den;
}

// ---------------------------------------------------------------------------
// Absorbed epilogue: merge the pieces, then out[b,l,h,:] = o_lat . W_UV[h]  (r -> v)
// One block per (group of ROWS (b,l) rows, head h); thread k owns output column k.
// ---------------------------------------------------------------------------
template <typename T, int ROWS>
__global__ void combine_unembed_kernel(const float* __restrict__ o_part,
                                       const float* __restrict__ ml, const T* __restrict__ W_UV,
                                       const int32_t* __restrict__ lens, T* __restrict__ out,
                                       int B, int L, int H, int r, int v, int chunk,
                                       int splits, int fixed_len) {
  extern __shared__ float so[];  // [ROWS][r]
  const int h = blockIdx.y;
  const int g0 = blockIdx.x * ROWS;  // first (b*L + l)
  const int LH = L * H;
  const int nrows = min(ROWS, B * L - g0);
  for (int rr = 0; rr < nrows; ++rr) {
    const int bl = g0 + rr;
    const int b = bl / L, l = bl - b * L;
    // pieces of this sequence: its cache length, or the index-list length
    const int nsplit = ((fixed_len > 0 ? fixed_len : lens[b]) + chunk - 1) / chunk;
    const size_t row = (size_t)l * H + h;
    const float* mlr = ml + (((size_t)b * splits) * LH + row) * 2;
    float M;
    const float inv = merge_norm(mlr, LH, nsplit, &M);
    for (int j = threadIdx.x; j < r; j += blockDim.x) {
      float acc = 0.f;
      for (int s = 0; s < nsplit; ++s) {
        const float ls = mlr[(size_t)s * LH * 2 + 1];
        if (ls > 0.f)
          acc += __expf(mlr[(size_t)s * LH * 2] - M) *
                 o_part[(((size_t)b * splits + s) * LH + row) * r + j];
      }
      so[rr * r + j] = acc * inv;
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < v; k += blockDim.x) {
    float acc[ROWS];
#pragma unroll
    for (int rr = 0; rr < ROWS; ++rr) acc[rr] = 0.f;
    const T* w = W_UV + (size_t)h * r * v + k;
    for (int j = 0; j < r; ++j) {
      const float wj = to_f(w[(size_t)j * v]);
#pragma unroll
      for (int rr = 0; rr < ROWS; ++rr) acc[rr] = fmaf(so[rr * r + j], wj, acc[rr]);
    }
    for (int rr = 0; rr < nrows; ++rr) {
      const int bl = g0 + rr;
      from_f(out + ((size_t)bl * H + h) * v + k, acc[rr]);
    }
  }
}

// Materialised epilogue: merge the pieces into out[b,l,h,:].
template <typename T>
__global__ void combine_kernel(const float* __restrict__ o_part, const float* __restrict__ ml,
                               const int32_t* __restrict__ lens, T* __restrict__ out, int L,
                               int H, int v, int chunk, int splits) {
  const int LH = L * H;
  const int row = blockIdx.x;  // l*H + h
  const int b = blockIdx.y;
  const int nsplit = (lens[b] + chunk - 1) / chunk;
  const float* mlr = ml + (((size_t)b * splits) * LH + row) * 2;
  float M;
  const float inv = merge_norm(mlr, LH, nsplit, &M);
  for (int k = threadIdx.x; k < v; k += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float ls = mlr[(size_t)s * LH * 2 + 1];
      if (ls > 0.f)
        acc += __expf(mlr[(size_t)s * LH * 2] - M) *
               o_part[(((size_t)b * splits + s) * LH + row) * v + k];
    }
    from_f(out + ((size_t)b * LH + row) * v + k, acc * inv);
  }
}

// ---------------------------------------------------------------------------
// Expansion: kexp[b, t, h, c] = c_kv[b,t] . W_UK[h, c, :]        for c <  n
//                             = c_kv[b,t] . W_UV[h, :, c - n]    for c >= n
// A 64x64-tile shared-memory GEMM over rows (b, t < T_b) and columns (h, c).
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) expand_kernel(CacheView cache, const T* __restrict__ W_UK,
                                                     const T* __restrict__ W_UV,
                                                     const int32_t* __restrict__ lens,
                                                     T* __restrict__ kexp, int Tmax, int H,
                                                     int r, int n, int v) {
  constexpr int BM = 64, BN = 64, BK = 16;
  __shared__ float sa[BK][BM + 4];
  __shared__ float sb[BK][BN + 4];
  const int b = blockIdx.z;
  const int Tb = lens[b];
  const int t0 = blockIdx.x * BM;
  if (t0 >= Tb) return;
  const int d = n + v;
  const int ncol = H * d;
  const int c0 = blockIdx.y * BN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  const T* ckv = (const T*)cache.c_kv;
  for (int k0 = 0; k0 < r; k0 += BK) {
    for (int idx = threadIdx.x; idx < BK * BM; idx += 256) {
      const int mm = idx / BK, kk = idx - mm * BK;
      const int t = t0 + mm;
      float x = 0.f;
      if (t < Tb && k0 + kk < r) {
        const int64_t crow = cache_row(cache, b, t);
        if (crow >= 0) x = to_f(ckv[crow * cache.ckv_stride + k0 + kk]);
        else if (kk == 0) report_bad_page();
      }
      sa[kk][mm] = x;
    }
    for (int idx = threadIdx.x; idx < BK * BN; idx += 256) {
      const int nn = idx / BK, kk = idx - nn * BK;
      const int col = c0 + nn, j = k0 + kk;
      float x = 0.f;
      if (col < ncol && j < r) {
        const int h = col / d, c = col - h * d;
        x = c < n ? to_f(W_UK[((size_t)h * n + c) * r + j])
                  : to_f(W_UV[((size_t)h * r + j) * v + (c - n)]);
      }
      sb[kk][nn] = x;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = sa[kk][ty * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i) bv[i] = sb[kk][tx * 4 + i];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(av[i], bv[jj], acc[i][jj]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= Tb) continue;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int col = c0 + tx * 4 + jj;
      if (col < ncol) from_f(kexp + ((size_t)b * Tmax + t) * ncol + col, acc[i][jj]);
    }
  }
}

template <typename T>
cudaError_t run_absorbed(const Plan& p, const Args& a) {
  constexpr int ROWS_FOLD = 16, ROWS_UNEMBED = 8;
  float* q_lat = (float*)(a.ws + p.off_qlat);
  float* o_part = (float*)(a.ws + p.off_opart);
  float* ml = (float*)(a.ws + p.off_ml);
  const int BL = p.B * p.L;
  {
    dim3 grid((p.r + 127) / 128, p.H, (BL + ROWS_FOLD - 1) / ROWS_FOLD);
    KernelTimer kt("generic_fold", a.stream);
    fold_kernel<T, ROWS_FOLD><<<grid, 128, ROWS_FOLD * p.n * sizeof(float), a.stream>>>(
        (const T*)a.q_nope, (const T*)a.W_UK, q_lat, BL, p.H, p.n, p.r);
  }
  {
    AttnParams ap;
    ap.q_main = q_lat;
    ap.q_rope = a.q_rope;
    ap.cache = a.cache;
    ap.kexp = nullptr;
    ap.lens = a.lens;
    ap.topk = a.topk;
    ap.topk_k = a.topk_k;
    ap.L = p.L; ap.H = p.H; ap.Dm = p.r; ap.rope = p.rope; ap.Dv = p.r; ap.n_plus_v = 0;
    ap.Tmax = p.Tmax; ap.scale = p.scale; ap.chunk = p.chunk; ap.splits = p.splits;
    ap.o_part = o_part; ap.ml = ml;
    dim3 grid((p.L * p.H + 3) / 4, p.splits, p.B);
    KernelTimer kt("generic_absorbed_attention", a.stream);
    attn_rows_kernel<T, true><<<grid, 128, 0, a.stream>>>(ap);
  }
  {
    dim3 grid((BL + ROWS_UNEMBED - 1) / ROWS_UNEMBED, p.H);
    const int threads = p.v >= 256 ? 256 : 128;
    KernelTimer kt("generic_combine_unembed", a.stream);
    combine_unembed_kernel<T, ROWS_UNEMBED>
        <<<grid, threads, ROWS_UNEMBED * p.r * sizeof(float), a.stream>>>(
            o_part, ml, (const T*)a.W_UV, a.lens, (T*)a.out, p.B, p.L, p.H, p.r, p.v, p.chunk,
            p.splits, a.topk ? a.topk_k : 0);
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t run_materialised(const Plan& p, const Args& a) {
  T* kexp = (T*)(a.ws + p.off_exp);
  float* o_part = (float*)(a.ws + p.off_opart);
  float* ml = (float*)(a.ws + p.off_ml);
  {
    dim3 grid((p.Tmax + 63) / 64, (p.H * (p.n + p.v) + 63) / 64, p.B);
    KernelTimer kt("generic_expand", a.stream);
    expand_kernel<T><<<grid, 256, 0, a.stream>>>(a.cache, (const T*)a.W_UK, (const T*)a.W_UV,
                                                  a.lens, kexp, p.Tmax, p.H, p.r, p.n, p.v);
  }
  {
    AttnParams ap;
    ap.q_main = a.q_nope;
    ap.q_rope = a.q_rope;
    ap.cache = a.cache;
    ap.kexp = kexp;
    ap.lens = a.lens;
    ap.topk = nullptr;
    ap.topk_k = 0;
    ap.L = p.L; ap.H = p.H; ap.Dm = p.n; ap.rope = p.rope; ap.Dv = p.v;
    ap.n_plus_v = p.n + p.v;
    ap.Tmax = p.Tmax; ap.scale = p.scale; ap.chunk = p.chunk; ap.splits = p.splits;
    ap.o_part = o_part; ap.ml = ml;
    dim3 grid((p.L * p.H + 3) / 4, p.splits, p.B);
    KernelTimer kt("generic_materialised_attention", a.stream);
    attn_rows_kernel<T, false><<<grid, 128, 0, a.stream>>>(ap);
  }
  {
    dim3 grid(p.L * p.H, p.B);
    KernelTimer kt("generic_combine", a.stream);
    combine_kernel<T><<<grid, 128, 0, a.stream>>>(o_part, ml, a.lens, (T*)a.out, p.L, p.H, p.v,
                                                  p.chunk, p.splits);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_generic_absorbed(const Plan& p, const Args& a) {
  return p.dtype == MLA_DTYPE_FP32 ? run_absorbed<float>(p, a) : run_absorbed<__nv_bfloat16>(p, a);
}

cudaError_t launch_generic_materialised(const Plan& p, const Args& a) {
  return p.dtype == MLA_DTYPE_FP32 ? run_materialised<float>(p, a)
                                   : run_materialised<__nv_bfloat16>(p, a);
}

int generic_device_status(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_generic_status, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v != 0) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_generic_status, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace mla
