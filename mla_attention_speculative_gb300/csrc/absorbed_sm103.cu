// Absorbed-branch MLA verify on GB300 tensor cores (tcgen05 + TMEM + TMA).
//
// "One guard, 110x off the verify step", section "The defect": fold the key
// up-projection into the query, attend against the compressed latent, then
// apply the value up-projection.  Three kernels, all bf16 operands with fp32
// accumulation in tensor memory:
//
//  fold_sm103      q_lat[row, h, :] = q_nope[row, h, :] . W_UK[h]  (n -> 512).
//                  Swap-AB GEMM per head: D[512 x rows] = W_UK[h]^T x q_nope^T,
//                  so the weight is the 128-row operand read once for all
//                  B*L rows (the pages' "small-M verify" idea, "Draft caps and
//                  calibration", section "Small-M verify kernel").
//  absorbed_attn   split-KV attention of the L*H query rows of a sequence
//                  against [c_kv || k_rope] (576 wide), online softmax, causal
//                  verify mask, o_lat = P . c_kv accumulated in the latent space.
//                  Each latent tile is read once for all 128 rows of a tile
//                  ("Multi-row attention kernel" on the same page).  A cluster
//                  of two CTAs shares one 128-row tile: CTA j holds latent
//                  columns [256j, 256j+256) (CTA 0 also the 64 RoPE columns),
//                  computes its partial scores over its columns, swaps them
//                  with the peer through distributed shared memory, and both
//                  accumulate their half of o_lat (128 x 256 fp32 in TMEM).
//  unembed_sm103   merges the split-KV pieces (log-sum-exp) and applies W_UV:
//                  D[v x rows] = W_UV[h]^T x o_lat^T (swap-AB, weight read once).
//
// Every wait is bounded; a wait that runs out sets the status word and the
// kernel finishes without waiting further (results are then undefined and
// mla_device_status reports MLA_ERR_TIMEOUT).

#include <cuda_bf16.h>

#include <cfloat>
#include <cmath>

#include "mla_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace mla {
using namespace sm103;

static __device__ int g_absorbed_status;

namespace {

constexpr int kLat = 512;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return (uint8_t*)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

__device__ __forceinline__ void report_timeout(int code) { atomicCAS(&g_absorbed_status, 0, code); }

// Wait unless an earlier wait of this thread already failed.
__device__ __forceinline__ void wait_or_fail(bool& ok, uint32_t bar, uint32_t parity, int code) {
  if (!ok) return;
  if (!mbar_wait(bar, parity)) {
    ok = false;
    report_timeout(code);
  }
}
__device__ __forceinline__ void wait_cluster_or_fail(bool& ok, uint32_t bar, uint32_t parity,
                                                     int code) {
  if (!ok) return;
  if (!mbar_wait_cluster(bar, parity)) {
    ok = false;
    report_timeout(code);
  }
}

__host__ __device__ constexpr uint32_t tmem_cols_for(int n) {
  return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : n <= 256 ? 256u : 512u;
}

// =========================================================================
// fold
// =========================================================================
struct FoldParams {
  __nv_bfloat16* q_lat;  // [B*L*H, 512]
  int BL, H, n, NB;      // NB: rows per CTA (multiple of 16, <= 256)
};

__global__ void __launch_bounds__(128) fold_sm103(const __grid_constant__ CUtensorMap tm_wuk,
                                                  const __grid_constant__ CUtensorMap tm_qn,
                                                  FoldParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int mt = blockIdx.x, h = blockIdx.y, row0 = blockIdx.z * p.NB;
  const int n = p.n, nk = n / 64, NB = p.NB;
  uint8_t* sA = smem;                   // W_UK[h][:, mt*128 +: 128], MN-major: 2 atoms x n rows
  uint8_t* sB = smem + 2 * n * 128;     // q_nope rows, K-major: nk chunks x NB rows
  uint64_t* bars = (uint64_t*)(sB + nk * NB * 128);
  uint32_t* slot = (uint32_t*)(bars + 2);
  volatile int* fail = (volatile int*)(bars + 3);
  const uint32_t bar_load = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ncols = tmem_cols_for(NB);

  if (threadIdx.x == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    *fail = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(slot), ncols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;

  if (threadIdx.x == 0) {
    bool ok = true;
    mbar_arrive_expect_tx(bar_load, 2 * n * 128 + nk * NB * 128);
    for (int j = 0; j < 2; ++j)
      for (int kc = 0; kc < nk; ++kc)
        tma_load_2d(smem_u32(sA + j * n * 128 + kc * 8192), &tm_wuk, bar_load, mt * 128 + 64 * j,
                    h * n + 64 * kc);
    for (int kc = 0; kc < nk; ++kc)
      tma_load_2d(smem_u32(sB + kc * NB * 128), &tm_qn, bar_load, h * n + 64 * kc, row0);
    wait_or_fail(ok, bar_load, 0, 1);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, NB, 1, 0);
      for (int kk = 0; kk < n / 16; ++kk) {
        const uint64_t a = sdesc_sw128(smem_u32(sA) + kk * 2048, n * 128, 1024);
        const uint64_t b =
            sdesc_sw128(smem_u32(sB) + (kk >> 2) * NB * 128 + (kk & 3) * 32, 16, 1024);
        mma_bf16(tmem, a, b, idesc, kk > 0);
      }
      mma_commit(bar_mma);
      wait_or_fail(ok, bar_mma, 0, 2);
    }
    if (!ok) *fail = 1;
  }
  __syncthreads();
  tc_fence_after();
  if (!*fail) {
    const int r = mt * 128 + warp * 32 + lane;
    for (int c0 = 0; c0 < NB; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int row = row0 + c0 + i;
        if (row < p.BL)
          p.q_lat[((size_t)row * p.H + h) * kLat + r] = __float2bfloat16_rn(__uint_as_float(v[i]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

// =========================================================================
// latent attention (2-CTA cluster per 128-row tile)
// =========================================================================
constexpr int BM = 128;                 // query rows per tile
constexpr int BN = 64;                  // cached positions per KV tile
constexpr int STAGES = 2;
constexpr int Q_CHUNK = BM * 128;       // one 64-column bf16 chunk of the Q tile
constexpr int KV_CHUNK = BN * 128;      // one 64-column bf16 chunk of a KV tile
constexpr int MAX_CH = 5;               // 4 latent chunks (+ RoPE on CTA 0)
constexpr int OFF_Q = 0;
constexpr int OFF_KV = OFF_Q + MAX_CH * Q_CHUNK;
constexpr int KV_STAGE = MAX_CH * KV_CHUNK;
constexpr int OFF_P = OFF_KV + STAGES * KV_STAGE;
constexpr int OFF_X = OFF_P + BM * 128;          // peer partial scores, fp32 [128][64]
constexpr int OFF_BAR = OFF_X + BM * BN * 4;
constexpr int ATTN_SMEM = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
constexpr uint32_t TM_O = 0;                     // O half: columns [0, 256)
constexpr uint32_t TM_S = 256;                   // S buffers: 256 + 64*sb

struct AttnParams {
  const int32_t* lens;
  const int32_t* page_table;
  int page_size, max_pages;
  long long seq_stride;
  int L, H, R;        // R = L*H query rows per sequence
  int chunk, splits;  // KV rows per split (multiple of 64), splits per sequence (max)
  float sl2;          // softmax scale * log2(e)
  float* o_part;      // [B, splits, R, 512]
  float* ml;          // [B, splits, R, 2]
};

enum {
  B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = 3, B_SFULL = 5, B_SFREE = 7, B_PFULL = 9,
  B_ODONE = 10, B_XFULL = 11, B_XFREE = 12, B_COUNT = 13
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    absorbed_attn_sm103(const __grid_constant__ CUtensorMap tm_ql,
                        const __grid_constant__ CUtensorMap tm_qr,
                        const __grid_constant__ CUtensorMap tm_ckv,
                        const __grid_constant__ CUtensorMap tm_kr, AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int tile = blockIdx.x >> 1, split = blockIdx.y, b = blockIdx.z;
  const int T = p.lens[b];
  const int nsplit = (T + p.chunk - 1) / p.chunk;
  if (split >= nsplit) return;  // both CTAs of the cluster leave together

  const int row0 = tile * BM;
  const int l_last = min(p.R - 1, row0 + BM - 1) / p.H;
  const int vis_end = T - p.L + l_last + 1;
  const int kv0 = split * p.chunk;
  const int kv1 = min(min(kv0 + p.chunk, T), vis_end);
  const int ntiles = kv1 > kv0 ? (kv1 - kv0 + BN - 1) / BN : 0;
  const int nch = rank == 0 ? 5 : 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = (uint64_t*)(smem + OFF_BAR);
  uint32_t* slot = (uint32_t*)(bars + 16);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ = smem_u32(smem + OFF_Q), sKV = smem_u32(smem + OFF_KV);
  const uint32_t sP = smem_u32(smem + OFF_P), sX = smem_u32(smem + OFF_X);

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(B_KVFULL + s), 1);
      mbar_init(bar(B_KVEMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SFREE + s), 128);
    }
    mbar_init(bar(B_PFULL), 128);
    mbar_init(bar(B_ODONE), 1);
    mbar_init(bar(B_XFULL), 128);
    mbar_init(bar(B_XFREE), 128);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote arrive
  const uint32_t tmem = *slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      bool ok = true;
      prefetch_tmap(&tm_ql);
      prefetch_tmap(&tm_ckv);
      const int qrow = b * p.R + row0;
      mbar_arrive_expect_tx(bar(B_QFULL), nch * Q_CHUNK);
      for (int c = 0; c < 4; ++c)
        tma_load_2d(sQ + c * Q_CHUNK, &tm_ql, bar(B_QFULL), (int)(4 * rank + c) * 64, qrow);
      if (rank == 0) tma_load_2d(sQ + 4 * Q_CHUNK, &tm_qr, bar(B_QFULL), 0, qrow);
      for (int i = 0; i < ntiles; ++i) {
        const int s = i % STAGES;
        if (i >= STAGES) wait_or_fail(ok, bar(B_KVEMPTY + s), ((i / STAGES) - 1) & 1, 10);
        if (!ok) break;
        const int t0 = kv0 + i * BN;
        const long long y =
            p.page_table ? (long long)p.page_table[(long long)b * p.max_pages + t0 / p.page_size] *
                                   p.page_size + (t0 % p.page_size)
                         : (long long)b * p.seq_stride + t0;
        const uint32_t st = sKV + s * KV_STAGE;
        mbar_arrive_expect_tx(bar(B_KVFULL + s), nch * KV_CHUNK);
        for (int c = 0; c < 4; ++c)
          tma_load_2d(st + c * KV_CHUNK, &tm_ckv, bar(B_KVFULL + s), (int)(4 * rank + c) * 64,
                      (int)y);
        if (rank == 0) tma_load_2d(st + 4 * KV_CHUNK, &tm_kr, bar(B_KVFULL + s), 0, (int)y);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && ntiles > 0) {
      bool ok = true;
      wait_or_fail(ok, bar(B_QFULL), 0, 11);
      const uint32_t id_s = idesc_bf16(BM, BN, 0, 0);
      const uint32_t id_o = idesc_bf16(BM, 256, 0, 1);
      for (int i = 0; i <= ntiles && ok; ++i) {
        if (i < ntiles) {
          const int s = i % STAGES, sb = i & 1;
          wait_or_fail(ok, bar(B_KVFULL + s), (i / STAGES) & 1, 12);
          if (i >= 2) wait_or_fail(ok, bar(B_SFREE + sb), ((i - 2) >> 1) & 1, 13);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = sKV + s * KV_STAGE;
          for (int c = 0; c < nch; ++c)
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16(tmem + TM_S + sb * BN, sdesc_sw128(sQ + c * Q_CHUNK + ks * 32, 16, 1024),
                       sdesc_sw128(st + c * KV_CHUNK + ks * 32, 16, 1024), id_s, (c | ks) != 0);
          mma_commit(bar(B_SFULL + sb));
        }
        if (i >= 1) {
          const int j = i - 1, sj = j % STAGES;
          wait_or_fail(ok, bar(B_PFULL), j & 1, 14);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = sKV + sj * KV_STAGE;
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + TM_O, sdesc_sw128(sP + ks * 32, 16, 1024),
                     sdesc_sw128(st + ks * 2048, KV_CHUNK, 1024), id_o, (j > 0 || ks > 0));
          mma_commit(bar(B_ODONE));
          mma_commit(bar(B_KVEMPTY + sj));
        }
      }
    }
  } else {
    // ------------------------------------------------- softmax warpgroup
    const int q = (warp & 3) * 32 + lane;  // tile row == TMEM lane
    const int row = row0 + q;
    const int l = min(row, p.R - 1) / p.H;
    const int last_t = T - p.L + l;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t peer_x = mapa(sX, peer);
    const uint32_t peer_xfull = mapa(bar(B_XFULL), peer);
    const uint32_t peer_xfree = mapa(bar(B_XFREE), peer);
    bool ok = true;
    float m_run = -INFINITY, l_run = 0.f;
    for (int i = 0; i < ntiles; ++i) {
      const int sb = i & 1;
      wait_or_fail(ok, bar(B_SFULL + sb), (i >> 1) & 1, 20);
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int k = 0; k < BN / 16; ++k) {
        uint32_t v[16];
        tmem_ld16(tmem + lane_base + TM_S + sb * BN + 16 * k, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) s[16 * k + e] = __uint_as_float(v[e]);
      }
      tc_fence_before();
      mbar_arrive(bar(B_SFREE + sb));
      // swap partial scores with the peer CTA
      if (i > 0) wait_cluster_or_fail(ok, bar(B_XFREE), (i - 1) & 1, 21);
#pragma unroll
      for (int c = 0; c < 16; ++c)
        st_cluster_v4(peer_x + q * 256 + ((c ^ (q & 15)) << 4), s[4 * c], s[4 * c + 1],
                      s[4 * c + 2], s[4 * c + 3]);
      mbar_arrive_remote(peer_xfull);
      wait_cluster_or_fail(ok, bar(B_XFULL), i & 1, 22);
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        float4 x;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                     : "r"(sX + q * 256 + ((c ^ (q & 15)) << 4)));
        s[4 * c] += x.x;
        s[4 * c + 1] += x.y;
        s[4 * c + 2] += x.z;
        s[4 * c + 3] += x.w;
      }
      mbar_arrive_remote(peer_xfree);
      // causal verify mask, log2-domain scores, tile maximum
      const int t0 = kv0 + i * BN;
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        s[j] = (t0 + j <= last_t) ? s[j] * p.sl2 : -INFINITY;
        mt = fmaxf(mt, s[j]);
      }
      // O (and the P buffer) are free once the previous P.V finished
      if (i > 0) wait_or_fail(ok, bar(B_ODONE), (i - 1) & 1, 23);
      tc_fence_after();
      // lazy rescale: move the running max only when it grows by more than 2^8
      const bool need = mt > m_run + 8.f;
      const float m_new = need ? mt : m_run;
      const float factor = need ? exp2f(m_run - m_new) : 1.f;
      if (i > 0 && __any_sync(0xffffffffu, need)) {
        for (int c = 0; c < 256; c += 16) {
          uint32_t v[16];
          tmem_ld16(tmem + lane_base + TM_O + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * factor);
          tmem_st16(tmem + lane_base + TM_O + c, v);
        }
        tmem_wait_st();
      }
      l_run *= factor;
      m_run = m_new;
      // P = 2^(s - m) in bf16, K-major 128-byte-swizzled rows of 64 positions
      float rs = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int j = 0; j < BN; j += 2) {
        const float a = m_run == -INFINITY ? 0.f : exp2f(s[j] - m_run);
        const float c = m_run == -INFINITY ? 0.f : exp2f(s[j + 1] - m_run);
        rs += a + c;
        pk[j / 2] = pack_bf16(a, c);
      }
      l_run += rs;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t addr = sP + q * 128 + (((c ^ q) & 7) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * c]),
                     "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      }
      // positions at or past T in the last tile: zero their value rows (they may hold
      // anything, and 0 * NaN would poison the accumulator)
      if (t0 + BN > T) {
        const int z0 = max(T - t0, 0);
        const uint32_t st = sKV + (i % STAGES) * KV_STAGE;
        const int units = (BN - z0) * 8;  // 16-byte units per 128-byte row
        for (int u = q; u < 4 * units; u += 128) {
          const int c = u / units, w = u - c * units;
          const uint32_t addr = st + c * KV_CHUNK + (z0 + w / 8) * 128 + (w & 7) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u)
                       : "memory");
        }
      }
      fence_async_shared();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL));
    }
    // ---------------------------------------------------------------- epilogue
    if (ntiles > 0) wait_or_fail(ok, bar(B_ODONE), (ntiles - 1) & 1, 24);
    tc_fence_after();
    const bool live = row < p.R;
    float* op = p.o_part + (((size_t)b * p.splits + split) * p.R + (live ? row : 0)) * kLat +
                rank * 256;
    for (int c = 0; c < 256; c += 16) {
      uint32_t v[16];
      if (ntiles > 0) {
        tmem_ld16(tmem + lane_base + TM_O + c, v);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = 0u;
      }
      if (live) {
#pragma unroll
        for (int e = 0; e < 16; e += 4)
          *(float4*)(op + c + e) =
              make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                          __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
      }
    }
    if (live && rank == 0) {
      float* mlp = p.ml + (((size_t)b * p.splits + split) * p.R + row) * 2;
      mlp[0] = m_run == -INFINITY ? -FLT_MAX : m_run;
      mlp[1] = l_run;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
  cluster_sync();  // no peer access may outlive this CTA
}

// =========================================================================
// merge + unembed
// =========================================================================
struct UnembedParams {
  const float* o_part;
  const float* ml;
  const int32_t* lens;
  __nv_bfloat16* out;  // [B, L, H, v]
  int BL, L, H, v, R, chunk, splits;
};

constexpr int UN_ROWS = 64;

__global__ void __launch_bounds__(128) unembed_sm103(const __grid_constant__ CUtensorMap tm_wuv,
                                                     UnembedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int vt = blockIdx.x, h = blockIdx.y, rt = blockIdx.z;
  uint8_t* sW = smem;                     // W_UV[h][:, vt*128 +: 128], MN-major: 2 atoms x 512
  uint8_t* sO = smem + 2 * 65536;         // merged o_lat rows, K-major: 8 chunks x NRpad rows
  uint64_t* bars = (uint64_t*)(sO + 8 * UN_ROWS * 128);
  uint32_t* slot = (uint32_t*)(bars + 2);
  volatile int* fail = (volatile int*)(bars + 3);
  const uint32_t bar_w = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[1]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int NR = min(UN_ROWS, p.BL - rt * UN_ROWS);
  const int NRpad = (NR + 15) & ~15;

  if (tid == 0) {
    mbar_init(bar_w, 1);
    mbar_init(bar_mma, 1);
    *fail = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_u32(slot), 64);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_w, 2 * 65536);
    for (int j = 0; j < 2; ++j)
      for (int kb = 0; kb < 4; ++kb)
        tma_load_2d(smem_u32(sW + j * 65536 + kb * 16384), &tm_wuv, bar_w, vt * 128 + 64 * j,
                    h * kLat + 128 * kb);
  }
  // merge the split-KV pieces of each row (thread owns latent columns 4*tid .. 4*tid+3)
  for (int nn = 0; nn < NRpad; ++nn) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (nn < NR) {
      const int bl = rt * UN_ROWS + nn;
      const int bb = bl / p.L, ll = bl - bb * p.L;
      const int row = ll * p.H + h;
      const int nsplit = (p.lens[bb] + p.chunk - 1) / p.chunk;
      const size_t base = (size_t)bb * p.splits * p.R + row;
      float M = -FLT_MAX;
      for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p.ml[(base + (size_t)s * p.R) * 2]);
      float den = 0.f;
      for (int s = 0; s < nsplit; ++s) {
        const float* mls = p.ml + (base + (size_t)s * p.R) * 2;
        if (mls[1] > 0.f) {
          const float w = exp2f(mls[0] - M);
          den += w * mls[1];
          const float4 o = *(const float4*)(p.o_part + (base + (size_t)s * p.R) * kLat + 4 * tid);
          acc.x += w * o.x;
          acc.y += w * o.y;
          acc.z += w * o.z;
          acc.w += w * o.w;
        }
      }
      const float inv = 1.f / den;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
    const int k = 4 * tid, c = k >> 6, col = k & 63;
    const uint32_t addr = smem_u32(sO) + c * NRpad * 128 + sw128_offset(nn, col);
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(pack_bf16(acc.x, acc.y)),
                 "r"(pack_bf16(acc.z, acc.w))
                 : "memory");
  }
  fence_async_shared();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    bool ok = true;
    wait_or_fail(ok, bar_w, 0, 30);
    if (ok) {
      tc_fence_after();
      const uint32_t idesc = idesc_bf16(128, NRpad, 1, 0);
      for (int kk = 0; kk < kLat / 16; ++kk)
        mma_bf16(tmem, sdesc_sw128(smem_u32(sW) + kk * 2048, 65536, 1024),
                 sdesc_sw128(smem_u32(sO) + (kk >> 2) * NRpad * 128 + (kk & 3) * 32, 16, 1024),
                 idesc, kk > 0);
      mma_commit(bar_mma);
      wait_or_fail(ok, bar_mma, 0, 31);
    }
    if (!ok) *fail = 1;
  }
  __syncthreads();
  tc_fence_after();
  if (!*fail) {
    const int vcol = vt * 128 + warp * 32 + lane;
    for (int c0 = 0; c0 < NRpad; c0 += 16) {
      uint32_t v[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int nn = c0 + i;
        if (nn < NR) {
          const int bl = rt * UN_ROWS + nn;
          p.out[((size_t)bl * p.H + h) * p.v + vcol] = __float2bfloat16_rn(__uint_as_float(v[i]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

bool fast_absorbed_supported(const Plan& p) {
  return p.dtype == MLA_DTYPE_BF16 && p.r == kLat && p.rope == 64 && p.n % 64 == 0 &&
         p.n >= 64 && p.n <= 256 && p.v % 128 == 0 && p.v <= 512;
}

int fast_fold_rows(int BL) {
  const int nb = ((BL + 15) / 16) * 16;
  return nb > 256 ? 256 : nb;
}

cudaError_t launch_fast_absorbed(const Plan& p, const Args& a) {
  const int BL = p.B * p.L;
  const int R = p.L * p.H;
  __nv_bfloat16* q_lat = (__nv_bfloat16*)(a.ws + p.off_qlat);
  float* o_part = (float*)(a.ws + p.off_opart);
  float* ml = (float*)(a.ws + p.off_ml);
  const CacheView& c = a.cache;
  const long long cache_rows =
      c.page_table ? (long long)c.num_pages * c.page_size
                   : (long long)(p.B - 1) * c.seq_stride + p.Tmax;

  CUtensorMap tm_wuk, tm_qn, tm_ql, tm_qr, tm_ckv, tm_kr, tm_wuv;
  const int NB = fast_fold_rows(BL);
  bool ok = make_tmap_bf16_2d(&tm_wuk, a.W_UK, kLat, (uint64_t)p.H * p.n, kLat * 2, 64, 64, true);
  ok = ok && make_tmap_bf16_2d(&tm_qn, a.q_nope, (uint64_t)p.H * p.n, BL, (uint64_t)p.H * p.n * 2,
                               64, NB, true);
  ok = ok && make_tmap_bf16_2d(&tm_ql, q_lat, kLat, (uint64_t)p.B * R, kLat * 2, 64, BM, true);
  ok = ok && make_tmap_bf16_2d(&tm_qr, a.q_rope, 64, (uint64_t)p.B * R, 128, 64, BM, true);
  ok = ok && make_tmap_bf16_2d(&tm_ckv, c.c_kv, kLat, cache_rows, c.ckv_stride * 2, 64, BN, true);
  ok = ok && make_tmap_bf16_2d(&tm_kr, c.k_rope, 64, cache_rows, c.kr_stride * 2, 64, BN, true);
  ok = ok && make_tmap_bf16_2d(&tm_wuv, a.W_UV, p.v, (uint64_t)p.H * kLat, (uint64_t)p.v * 2, 64,
                               128, true);
  if (!ok) return cudaErrorInvalidValue;

  static bool attrs = false;
  const int fold_smem = 2 * p.n * 128 + (p.n / 64) * NB * 128 + 1024 + 64;
  const int un_smem = 2 * 65536 + 8 * UN_ROWS * 128 + 1024 + 64;
  if (!attrs) {
    cudaError_t e = set_smem(fold_sm103, 2 * 256 * 128 + 4 * 256 * 128 + 1024 + 64);
    if (e == cudaSuccess) e = set_smem(absorbed_attn_sm103, ATTN_SMEM);
    if (e == cudaSuccess) e = set_smem(unembed_sm103, un_smem);
    if (e != cudaSuccess) return e;
    attrs = true;
  }
  {
    FoldParams fp{q_lat, BL, p.H, p.n, NB};
    dim3 grid(kLat / 128, p.H, (BL + NB - 1) / NB);
    KernelTimer kt("fold_sm103", a.stream);
    fold_sm103<<<grid, 128, fold_smem, a.stream>>>(tm_wuk, tm_qn, fp);
  }
  {
    AttnParams ap;
    ap.lens = a.lens;
    ap.page_table = c.page_table;
    ap.page_size = c.page_size;
    ap.max_pages = c.max_pages;
    ap.seq_stride = c.seq_stride;
    ap.L = p.L;
    ap.H = p.H;
    ap.R = R;
    ap.chunk = p.chunk;
    ap.splits = p.splits;
    ap.sl2 = p.scale * 1.4426950408889634f;
    ap.o_part = o_part;
    ap.ml = ml;
    dim3 grid(2 * ((R + BM - 1) / BM), p.splits, p.B);
    KernelTimer kt("absorbed_attn_sm103", a.stream);
    absorbed_attn_sm103<<<grid, 192, ATTN_SMEM, a.stream>>>(tm_ql, tm_qr, tm_ckv, tm_kr, ap);
  }
  {
    UnembedParams up{o_part, ml, a.lens, (__nv_bfloat16*)a.out, BL, p.L, p.H, p.v, R,
                     p.chunk, p.splits};
    dim3 grid(p.v / 128, p.H, (BL + UN_ROWS - 1) / UN_ROWS);
    KernelTimer kt("unembed_sm103", a.stream);
    unembed_sm103<<<grid, 128, un_smem, a.stream>>>(tm_wuv, up);
  }
  return cudaGetLastError();
}

int absorbed_device_status(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_absorbed_status, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v != 0) {
    const int z = 0;
    cudaMemcpyToSymbol(g_absorbed_status, &z, sizeof(int));
  }
  return v;
}

}  // namespace mla
