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
#include <cuda_fp16.h>

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
constexpr int STAGES = 3;
constexpr int Q_CHUNK = BM * 128;       // one 64-column bf16 chunk of the Q tile (128-B swizzle)
constexpr int Q_ROPE = BM * 64;         // the 32 RoPE columns of this CTA (64-B swizzle)
constexpr int KV_CHUNK = BN * 128;      // one 64-column bf16 chunk of a KV tile
constexpr int KV_ROPE = BN * 64;        // 32 RoPE columns of a KV tile
constexpr int X_BYTES = BM * BN * 2;    // the peer's partial scores, fp16 [128][64]
constexpr int OFF_Q = 0;
constexpr int OFF_QR = OFF_Q + 4 * Q_CHUNK;
constexpr int OFF_KV = OFF_QR + Q_ROPE;
constexpr int KV_STAGE = 4 * KV_CHUNK + KV_ROPE;
constexpr int OFF_X = OFF_KV + STAGES * KV_STAGE;
constexpr int OFF_BAR = OFF_X + X_BYTES;
constexpr int ATTN_SMEM = OFF_BAR + 256 + 1024;     // + barriers + alignment slack
constexpr uint32_t TM_O = 0;                        // O half: columns [0, 256)
constexpr uint32_t TM_S = 256;                      // S / P buffers: 256 + 64*sb
constexpr int SBUF = 4;                             // S / P buffers (TMEM columns 256..511)
static_assert(OFF_KV % 1024 == 0 && KV_STAGE % 1024 == 0, "swizzle atoms need 1 KiB alignment");
static_assert(ATTN_SMEM <= 232448, "shared memory per CTA");

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

// Barrier slots.  Every barrier that is waited on by parity alone has enough
// copies that it cannot complete twice before its waiter looks: P-full and
// O-done alternate by tile parity, S buffers by tile % 4.
enum {
  B_QFULL = 0, B_KVFULL = 1, B_KVEMPTY = 4, B_SFULL = 7, B_SFREE = 11, B_PFULL = 15,
  B_ODONE = 17, B_XFULL = 19, B_XFREE = 20, B_COUNT = 21
};

// This CTA's partial scores of tile j from TMEM, scaled to log2-softmax units.
__device__ __forceinline__ void load_partial(bool& ok, uint32_t tmem, uint32_t lane_base, int j,
                                             uint32_t bar_sfull0, uint32_t bar_sfree0,
                                             float sl2, float (&s)[BN]) {
  const int sb = j & (SBUF - 1);
  wait_or_fail(ok, bar_sfull0 + 8 * sb, (j / SBUF) & 1, 20);
  tc_fence_after();
  uint32_t v[BN];
#pragma unroll
  for (int k = 0; k < BN / 16; ++k)
    tmem_ld16(tmem + lane_base + TM_S + sb * BN + 16 * k, *(uint32_t(*)[16])(v + 16 * k));
  tmem_wait_ld();
#pragma unroll
  for (int e = 0; e < BN; ++e) s[e] = __uint_as_float(v[e]) * sl2;
  tc_fence_before();
  mbar_arrive(bar_sfree0 + 8 * sb);
}

// Round this row's partial scores to fp16 (both CTAs add the same two rounded
// partials, so their sums agree bit for bit) and send them into the peer's
// exchange buffer; each 16-byte store counts itself off the peer's barrier.
__device__ __forceinline__ void send_partial(uint32_t peer_x, uint32_t peer_xfull, int q,
                                             float (&s)[BN]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint32_t h[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 v = __floats2half2_rn(s[8 * c + 2 * e], s[8 * c + 2 * e + 1]);
      h[e] = *reinterpret_cast<const uint32_t*>(&v);
      const float2 back = __half22float2(v);
      s[8 * c + 2 * e] = back.x;
      s[8 * c + 2 * e + 1] = back.y;
    }
    st_async_v4(peer_x + q * 128 + ((c ^ (q & 7)) << 4), h[0], h[1], h[2], h[3], peer_xfull);
  }
}

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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  uint64_t* bars = (uint64_t*)(smem + OFF_BAR);
  uint32_t* slot = (uint32_t*)(bars + 24);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const uint32_t sQ = smem_u32(smem + OFF_Q), sQR = smem_u32(smem + OFF_QR);
  const uint32_t sKV = smem_u32(smem + OFF_KV), sX = smem_u32(smem + OFF_X);

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(B_KVFULL + s), 1);
      mbar_init(bar(B_KVEMPTY + s), 1);
    }
    for (int s = 0; s < SBUF; ++s) {
      mbar_init(bar(B_SFULL + s), 1);
      mbar_init(bar(B_SFREE + s), 128);
    }
    for (int s = 0; s < 2; ++s) mbar_init(bar(B_ODONE + s), 1);
    for (int s = 0; s < 2; ++s) mbar_init(bar(B_PFULL + s), 128);
    mbar_init(bar(B_XFULL), 1);
    mbar_init(bar(B_XFREE), 1);
    fence_mbar_init();
    // arm the exchange barrier for tile 0 (the peer's stores count it down)
    if (ntiles > 0) mbar_arrive_expect_tx(bar(B_XFULL), X_BYTES);
  }
  if (warp == 1) tmem_alloc(smem_u32(slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist (and are armed) before any remote access
  const uint32_t tmem = *slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && ntiles > 0) {
      bool ok = true;
      prefetch_tmap(&tm_ql);
      prefetch_tmap(&tm_ckv);
      const int qrow = b * p.R + row0;
      mbar_arrive_expect_tx(bar(B_QFULL), 4 * Q_CHUNK + Q_ROPE);
      for (int c = 0; c < 4; ++c)
        tma_load_2d(sQ + c * Q_CHUNK, &tm_ql, bar(B_QFULL), (int)(4 * rank + c) * 64, qrow);
      tma_load_2d(sQR, &tm_qr, bar(B_QFULL), (int)rank * 32, qrow);
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
        mbar_arrive_expect_tx(bar(B_KVFULL + s), KV_STAGE);
        for (int c = 0; c < 4; ++c)
          tma_load_2d(st + c * KV_CHUNK, &tm_ckv, bar(B_KVFULL + s), (int)(4 * rank + c) * 64,
                      (int)y);
        tma_load_2d(st + 4 * KV_CHUNK, &tm_kr, bar(B_KVFULL + s), (int)rank * 32, (int)y);
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
          // S(i) = Q . K(i)^T over this CTA's 256 latent + 32 RoPE columns
          const int s = i % STAGES, sb = i & (SBUF - 1);
          wait_or_fail(ok, bar(B_KVFULL + s), (i / STAGES) & 1, 12);
          if (i >= SBUF) wait_or_fail(ok, bar(B_SFREE + sb), ((i - SBUF) / SBUF) & 1, 13);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = sKV + s * KV_STAGE;
          const uint32_t d = tmem + TM_S + sb * BN;
          for (int c = 0; c < 4; ++c)
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16(d, sdesc_sw128(sQ + c * Q_CHUNK + ks * 32, 16, 1024),
                       sdesc_sw128(st + c * KV_CHUNK + ks * 32, 16, 1024), id_s, (c | ks) != 0);
          for (int ks = 0; ks < 2; ++ks)
            mma_bf16(d, sdesc_sw64(sQR + ks * 32, 512), sdesc_sw64(st + 4 * KV_CHUNK + ks * 32, 512),
                     id_s, 1);
          mma_commit(bar(B_SFULL + sb));
        }
        if (i >= 1) {
          // O += P(j) . V(j): P from TMEM (bf16 pairs over S buffer j%4), V = this
          // CTA's 256 latent columns of the KV tile
          const int j = i - 1, sj = j % STAGES, pb = j & (SBUF - 1);
          wait_or_fail(ok, bar(B_PFULL + (j & 1)), (j >> 1) & 1, 14);
          if (!ok) break;
          tc_fence_after();
          const uint32_t st = sKV + sj * KV_STAGE;
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16_tmem_a(tmem + TM_O, tmem + TM_S + pb * BN + ks * 8,
                            sdesc_sw128(st + ks * 2048, KV_CHUNK, 1024), id_o, (j > 0 || ks > 0));
          mma_commit(bar(B_ODONE + (j & 1)));
          mma_commit(bar(B_KVEMPTY + sj));
        }
      }
    }
  } else {
    // ------------------------------------------------- softmax warpgroup
    // Tile i's scores are finished (own + peer partial) while tile i+1's
    // partial is already on its way to the peer.  P(i) goes back into the TMEM
    // columns S(i) came from; S(i+4) reuses them, long after P.V(i) has run.
    const int q = (warp & 3) * 32 + lane;  // tile row == TMEM lane
    const int sm_tid = threadIdx.x - 64;
    const int row = row0 + q;
    const int l = min(row, p.R - 1) / p.H;
    const int last_t = T - p.L + l;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t peer_x = mapa(sX, peer);
    const uint32_t peer_xfull = mapa(bar(B_XFULL), peer);
    const uint32_t peer_xfree = mapa(bar(B_XFREE), peer);
    bool ok = true;
    float m_run = -INFINITY, l_run = 0.f;
    float s[BN];
    if (ntiles > 0) {
      load_partial(ok, tmem, lane_base, 0, bar(B_SFULL), bar(B_SFREE), p.sl2, s);
      send_partial(peer_x, peer_xfull, q, s);
    }
    for (int i = 0; i < ntiles; ++i) {
      // finish tile i's scores with the peer's partial
      wait_cluster_or_fail(ok, bar(B_XFULL), i & 1, 22);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t h[4];
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
                     : "r"(sX + q * 128 + ((c ^ (q & 7)) << 4)));
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
          s[8 * c + 2 * e] += f.x;
          s[8 * c + 2 * e + 1] += f.y;
        }
      }
      named_bar_sync(1, 128);  // every row has read the exchange buffer
      if (sm_tid == 0) {
        if (i + 1 < ntiles) mbar_arrive_expect_tx(bar(B_XFULL), X_BYTES);  // arm tile i+1
        mbar_arrive_remote(peer_xfree);  // the peer may now send tile i+1
      }
      // start tile i+1's exchange
      float sn[BN];
      if (i + 1 < ntiles) {
        load_partial(ok, tmem, lane_base, i + 1, bar(B_SFULL), bar(B_SFREE), p.sl2, sn);
        wait_cluster_or_fail(ok, bar(B_XFREE), i & 1, 21);  // the peer has read my tile i
        send_partial(peer_x, peer_xfull, q, sn);
      }
      // causal verify mask and tile maximum (scores are in log2 units already)
      const int t0 = kv0 + i * BN;
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        s[j] = (t0 + j <= last_t) ? s[j] : -INFINITY;
        mt = fmaxf(mt, s[j]);
      }
      // lazy rescale: move the running max only when it grows by more than 2^8;
      // O must then hold every earlier P.V
      const bool need = mt > m_run + 8.f;
      const float m_new = need ? mt : m_run;
      const float factor = need ? ex2(m_run - m_new) : 1.f;
      if (i > 0 && __any_sync(0xffffffffu, need)) {
        wait_or_fail(ok, bar(B_ODONE + ((i - 1) & 1)), ((i - 1) >> 1) & 1, 23);
        tc_fence_after();
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
      // P = 2^(s - m) as bf16 pairs into the first 32 columns of S buffer i%4
      const float m_use = m_run == -INFINITY ? 0.f : m_run;
      float rs = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int e = 0; e < BN / 2; ++e) {
        const float a = ex2(s[2 * e] - m_use);
        const float d = ex2(s[2 * e + 1] - m_use);
        rs += a + d;
        pk[e] = pack_bf16(a, d);
      }
      l_run += rs;
      tmem_st32(tmem + lane_base + TM_S + (i & (SBUF - 1)) * BN, pk);
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
        fence_async_shared();
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(B_PFULL + (i & 1)));
#pragma unroll
      for (int e = 0; e < BN; ++e) s[e] = sn[e];
    }
    // ---------------------------------------------------------------- epilogue
    if (ntiles > 0) wait_or_fail(ok, bar(B_ODONE + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, 25);
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
  bool ok = make_tmap_bf16_2d(&tm_wuk, a.W_UK, kLat, (uint64_t)p.H * p.n, kLat * 2, 64, 64, 128);
  ok = ok && make_tmap_bf16_2d(&tm_qn, a.q_nope, (uint64_t)p.H * p.n, BL, (uint64_t)p.H * p.n * 2,
                               64, NB, 128);
  ok = ok && make_tmap_bf16_2d(&tm_ql, q_lat, kLat, (uint64_t)p.B * R, kLat * 2, 64, BM, 128);
  ok = ok && make_tmap_bf16_2d(&tm_qr, a.q_rope, 64, (uint64_t)p.B * R, 128, 32, BM, 64);
  ok = ok && make_tmap_bf16_2d(&tm_ckv, c.c_kv, kLat, cache_rows, c.ckv_stride * 2, 64, BN, 128);
  ok = ok && make_tmap_bf16_2d(&tm_kr, c.k_rope, 64, cache_rows, c.kr_stride * 2, 32, BN, 64);
  ok = ok && make_tmap_bf16_2d(&tm_wuv, a.W_UV, p.v, (uint64_t)p.H * kLat, (uint64_t)p.v * 2, 64,
                               128, 128);
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
